// Device kernels of libpa.so (sm_103a): load-time validation, the event-count
// work partitioner, the fused dynamic + leakage power kernel and the final
// reduction. The computation is the power step of "GPU-Accelerated Gate-Level
// Time-Based Power Analysis via Event-Density-Aware Partitioning and Kernel
// Fusion" (Sections 2.4.1-2.4.2, Eqs. 1-4, Figs. 2, 3 and 7); the mapping onto
// the GPU is this library's own:
//
//  * Work is cut by event count. Runs of consecutive light gates form tiles of
//    about `tile_target` events (one contiguous slice of the CSR arrays);
//    every gate with more than `heavy_thresh` events is streamed by one CTA in
//    time windows of at most kTileCap events, sized in proportion to each pin's
//    remaining events (the role of the paper's event-density-aware per-gate
//    cycle partitioning, Figs. 5, 19 and 20, without a fixed cycles-per-thread).
//  * One thread per event inside a staged tile. The gate state before the
//    event's timestamp (the "preceding gate state" of Section 2.4.1 and the
//    per-timestamp state S of Fig. 7) is rebuilt from parities: an input pin's
//    value before time t is its initial value flipped once per earlier event,
//    and the number of earlier events on another pin is a binary search of t
//    in that pin's sorted, staged segment. Ties see the pre-timestamp state.
//  * Glitch counter (Fig. 7, GlitchDetectUpdate): an event is a glitch iff the
//    previous event of the same pin lies in the same cycle, which is the
//    adjacent CSR element -- no counter state is carried.
//  * Leakage (Section 2.4.2, Eq. 4) without per-cycle work: a gate's leakage
//    power is piecewise constant and changes only at input events. Each input
//    event contributes its step dP = p(S_after) - p(S_before), taken in (time,
//    pin) order so simultaneous events telescope to the group's total. The
//    part of the step inside the event's own cycle goes to the cycle's energy
//    bin, the step itself to a per-cycle step array whose prefix sum (final
//    reduction) carries it to every later cycle, and dP * (t_max - t) to the
//    leakage total. This equals the interval-by-overlap split exactly in real
//    arithmetic, at O(events + cycles) instead of O(gates * cycles).
#include <cfloat>
#include <cstdint>

#include "pa_internal.cuh"

namespace pa {

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ void dev_err(unsigned long long* err, uint64_t idx, uint32_t code) {
  atomicMin(err, (unsigned long long)((idx << 8) | code));
}

__device__ __forceinline__ unsigned warp_max_u32(unsigned v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum_f32(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Inclusive warp scan of a u32.
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Block-wide exclusive scan of two u32 values (blockDim.x == 256).
__device__ __forceinline__ void block_excl_scan2(uint32_t a, uint32_t b, uint32_t& ea, uint32_t& eb,
                                                 uint32_t& ta, uint32_t& tb) {
  __shared__ uint32_t wa[8], wb[8];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t ia = warp_incl_scan(a, lane), ib = warp_incl_scan(b, lane);
  if (lane == 31) { wa[w] = ia; wb[w] = ib; }
  __syncthreads();
  uint32_t oa = 0, ob = 0, sa = 0, sb = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (i < w) { oa += wa[i]; ob += wb[i]; }
    sa += wa[i]; sb += wb[i];
  }
  ea = oa + ia - a;
  eb = ob + ib - b;
  ta = sa;
  tb = sb;
  __syncthreads();
}

// ------------------------------------------------------------------ validation

__global__ void k_check_pin_off(const uint64_t* __restrict__ off, uint64_t n_pins, uint64_t n_events,
                                unsigned long long* err) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t p = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; p <= n_pins; p += stride) {
    const uint64_t a = off[p];
    bool bad = a > n_events;
    if (p == 0 && a != 0) bad = true;
    if (p == n_pins && a != n_events) bad = true;
    if (p < n_pins && off[p + 1] < a) bad = true;
    if (bad) dev_err(err, p, kErrPinOff);
  }
}

cudaError_t launch_check_pin_off(const uint64_t* pin_off, uint64_t n_pins, uint64_t n_events,
                                 unsigned long long* err, cudaStream_t st) {
  const uint64_t n = n_pins + 1;
  const int grid = (int)std::min<uint64_t>((n + 255) / 256, 65535ull * 8);
  k_check_pin_off<<<grid, 256, 0, st>>>(pin_off, n_pins, n_events, err);
  return cudaGetLastError();
}

// Event checks in two flat passes, so that no gate's length sets the time:
// one thread per gate marks the first event of each of its non-empty pins in
// a bitmap, checks that event's value against the pin's initial value and
// writes gate_off; then one thread per event checks its time and slew ranges
// and, unless it starts a pin, its order and toggle against the event before
// it (the pin's previous event). Pin offsets are clamped to [0, n_events], so
// offsets that k_check_pin_off rejects cannot take a read out of bounds.
__global__ void __launch_bounds__(256) k_validate_gates(const ValidateArgs a) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  const uint64_t E = a.n_events;
  for (uint64_t g = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; g < a.n_gates; g += stride) {
    const GateRec r = a.gates[g];
    const int k = (int)((r.init >> 16) & 0xff);
    const uint64_t pb = r.pin_base;
    a.gate_off[g] = a.pin_off[pb];
    for (int p = 0; p <= k; ++p) {
      const uint64_t lo = min(a.pin_off[pb + p], E), hi = min(a.pin_off[pb + p + 1], E);
      if (lo >= hi) continue;
      atomicOr(a.starts + (lo >> 5), 1u << (lo & 31u));
      if (a.value) {
        const uint32_t init = p < k ? (r.init >> p) & 1u : (r.init >> 8) & 1u;
        const uint32_t v = a.value[lo];
        if (v > 1u) dev_err(a.err, lo, kErrValue);
        else if (v == init) dev_err(a.err, lo, kErrToggle);
      }
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) a.gate_off[a.n_gates] = E;
}

__global__ void __launch_bounds__(256) k_validate_events(const ValidateArgs a) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  unsigned tmax = 0;
  for (uint64_t e = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; e < a.n_events; e += stride) {
    const float t = a.t[e], s = a.s[e];
    if (!(t >= 0.f) || !(t <= FLT_MAX)) {
      dev_err(a.err, e, kErrRangeT);
    } else {
      tmax = max(tmax, t == 0.f ? 0u : __float_as_uint(t));
    }
    if (!(s > 0.f) || !(s <= FLT_MAX)) dev_err(a.err, e, kErrRangeSlew);
    const bool first = ((a.starts[e >> 5] >> (e & 31u)) & 1u) != 0u;
    if (!first && e > 0 && !(t > a.t[e - 1])) dev_err(a.err, e, kErrUnsorted);
    if (a.value) {
      const uint32_t v = a.value[e];
      if (v > 1u) dev_err(a.err, e, kErrValue);
      else if (!first && e > 0 && v == (uint32_t)a.value[e - 1]) dev_err(a.err, e, kErrToggle);
    }
  }
  tmax = warp_max_u32(tmax);
  __shared__ unsigned s_max[8];
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = tmax;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned m = 0;
    for (int i = 0; i < 8; ++i) m = max(m, s_max[i]);
    if (m) atomicMax(a.t_max_bits, m);
  }
}

cudaError_t launch_validate_events(const ValidateArgs& a, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(a.starts, 0, ((a.n_events + 31) / 32 + 1) * sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  const int gg = (int)std::min<uint64_t>(((uint64_t)a.n_gates + 255) / 256, 152ull * 16);
  k_validate_gates<<<gg > 0 ? gg : 1, 256, 0, st>>>(a);
  if (a.n_events) {
    const int ge = (int)std::min<uint64_t>((a.n_events + 255) / 256, 152ull * 32);
    k_validate_events<<<ge, 256, 0, st>>>(a);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------ partition
//
// A gate is heavy if it has more than heavy_thresh events. Light gates are
// grouped into tiles of consecutive gates: a tile starts at a light gate whose
// first event offset falls in a different tile_target-sized bucket than its
// predecessor's, after a heavy gate, at every kGateCap-th gate, and at gate 0.
// Every gate of a tile then starts in one bucket, so a tile holds fewer than
// tile_target + heavy_thresh events and at most kGateCap gates.

__device__ __forceinline__ bool is_heavy(const RunArgs& a, uint32_t g) {
  return a.gate_off[g + 1] - a.gate_off[g] > (uint64_t)a.heavy_thresh;
}

__device__ __forceinline__ bool is_head(const RunArgs& a, uint32_t g) {
  if (is_heavy(a, g)) return false;
  if (g == 0 || g % kGateCap == 0) return true;
  if (is_heavy(a, g - 1)) return true;
  return a.gate_off[g] / a.tile_target != a.gate_off[g - 1] / a.tile_target;
}

__global__ void __launch_bounds__(256) k_part_count(const RunArgs a) {
  const uint32_t g = blockIdx.x * 256u + threadIdx.x;
  uint32_t h = 0, hv = 0;
  double p0 = 0.0;
  if (g < a.n_gates) {
    hv = is_heavy(a, g);
    h = is_head(a, g);
    const GateRec r = a.gates[g];
    const CellDesc& cd = a.cells[r.cell];
    const uint32_t s0 = r.init & ((1u << cd.k) - 1u);
    p0 = (double)a.leak[cd.leak_off + s0];
  }
  uint32_t ea, eb, ta, tb;
  block_excl_scan2(h, hv, ea, eb, ta, tb);
  if (threadIdx.x == 0) {
    a.part_blk[2 * blockIdx.x] = ta;
    a.part_blk[2 * blockIdx.x + 1] = tb;
  }
  __shared__ double sp[8];
  p0 = warp_sum_f64(p0);
  if ((threadIdx.x & 31) == 0) sp[threadIdx.x >> 5] = p0;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0;
    for (int i = 0; i < 8; ++i) s += sp[i];
    atomicAdd(a.p0, s);
  }
}

// Single block: exclusive scan of the per-block (heads, heavies) counts.
__global__ void __launch_bounds__(1024) k_part_scan(const RunArgs a, uint32_t n_blocks) {
  __shared__ uint32_t sa[32], sb[32];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const uint32_t chunk = (n_blocks + 1023) / 1024;
  const uint32_t b0 = min(n_blocks, tid * chunk), b1 = min(n_blocks, b0 + chunk);
  uint32_t la = 0, lb = 0;
  for (uint32_t b = b0; b < b1; ++b) { la += a.part_blk[2 * b]; lb += a.part_blk[2 * b + 1]; }
  const uint32_t ia = warp_incl_scan(la, lane), ib = warp_incl_scan(lb, lane);
  if (lane == 31) { sa[w] = ia; sb[w] = ib; }
  __syncthreads();
  if (w == 0) {
    const uint32_t xa = warp_incl_scan(sa[lane], lane), xb = warp_incl_scan(sb[lane], lane);
    sa[lane] = xa;
    sb[lane] = xb;
  }
  __syncthreads();
  uint32_t oa = (w ? sa[w - 1] : 0) + ia - la, ob = (w ? sb[w - 1] : 0) + ib - lb;
  for (uint32_t b = b0; b < b1; ++b) {
    const uint32_t ca = a.part_blk[2 * b], cb = a.part_blk[2 * b + 1];
    a.part_blk[2 * b] = oa;
    a.part_blk[2 * b + 1] = ob;
    oa += ca;
    ob += cb;
  }
  if (tid == 1023) {
    a.part_counts[0] = oa;  // tiles
    a.part_counts[1] = ob;  // heavy gates
    a.part_counts[2] = 0;   // work-item counter of the fused kernel
  }
}

__global__ void __launch_bounds__(256) k_part_emit(const RunArgs a) {
  const uint32_t g = blockIdx.x * 256u + threadIdx.x;
  uint32_t h = 0, hv = 0, tail = 0;
  if (g < a.n_gates) {
    hv = is_heavy(a, g);
    h = is_head(a, g);
    if (!hv) tail = (g + 1 == a.n_gates) || is_heavy(a, g + 1) || is_head(a, g + 1);
  }
  uint32_t ea, eb, ta, tb;
  block_excl_scan2(h, hv, ea, eb, ta, tb);
  const uint32_t th = a.part_blk[2 * blockIdx.x] + ea;  // heads before g
  const uint32_t tv = a.part_blk[2 * blockIdx.x + 1] + eb;
  if (g < a.n_gates) {
    if (h) a.tiles[th].gb = g;
    if (tail) a.tiles[th + h - 1].ge = g + 1;
    if (hv) a.heavy[tv] = g;
  }
}

uint32_t partition_blocks(uint32_t n_gates) { return (n_gates + 255) / 256; }

cudaError_t launch_part_scan(const RunArgs& a, uint32_t n_blocks, cudaStream_t st) {
  k_part_scan<<<1, 1024, 0, st>>>(a, n_blocks);
  return cudaGetLastError();
}

cudaError_t launch_partition(const RunArgs& a, uint32_t n_blocks, cudaStream_t st) {
  if (n_blocks == 0) return cudaSuccess;
  k_part_count<<<n_blocks, 256, 0, st>>>(a);
  k_part_scan<<<1, 1024, 0, st>>>(a, n_blocks);
  k_part_emit<<<n_blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ fused kernel

// Per-gate slot of a staged work item.
struct __align__(16) Slot {
  uint16_t st[kMaxK + 2];  // staged start of pins 0..k; st[k+1] = end
  uint16_t np[kMaxK + 1];  // events of each pin to process in this step
  uint8_t k, init, j, pre; // inputs, initial input bits, load-axis interval, parity of earlier events per pin
  uint32_t cell;
  float v, esw;            // load-axis fraction; switching energy C V^2 / 2 (fJ)
  uint32_t gate;           // gate index (per-gate outputs)
  uint32_t pad;
};
static_assert(sizeof(Slot) == 48, "slot size");

struct HeavyState {
  uint64_t cur[kMaxK + 1], end[kMaxK + 1];
  float prev_t[kMaxK + 1], prev_s[kMaxK + 1];
  float bound[kMaxK + 1];
  uint8_t has_prev[kMaxK + 1];
  int done;
};

constexpr size_t kSmemT = sizeof(float) * kTileCap;
constexpr size_t kSmemTag = sizeof(uint16_t) * kTileCap;
constexpr size_t kSmemSlots = sizeof(Slot) * kGateCap;
constexpr size_t kSmemCellsB = sizeof(CellDesc) * kSmemCells;
constexpr size_t kSmemTotal = 2 * kSmemT + kSmemTag + kSmemSlots + kSmemCellsB;

size_t fused_smem_bytes() { return kSmemTotal; }

template <bool kPow2>
__device__ __forceinline__ uint32_t cycle_of(float t, float T, float inv_T) {
  // floor(fl32(t / T)) for t >= 0; with T a power of two t * (1/T) is the
  // same correctly rounded quotient.
  if (kPow2) return (uint32_t)(t * inv_T);
  return (uint32_t)__fdiv_rn(t, T);
}

// Number of elements of sorted a[0, n) strictly below x.
__device__ __forceinline__ int lower_bound_f(const float* a, int n, float x) {
  int lo = 0;
  while (n > 0) {
    const int half = n >> 1;
    if (a[lo + half] < x) {
      lo += half + 1;
      n -= half + 1;
    } else {
      n = half;
    }
  }
  return lo;
}

// Input state of a gate just before time t (all inputs, pre-timestamp), for
// the debug output of output-pin events.
__device__ __forceinline__ uint32_t state_before(const float* ts, const Slot& S, float t) {
  uint32_t st = S.init;
  for (int q = 0; q < S.k; ++q) {
    const int r = lower_bound_f(ts + S.st[q], S.st[q + 1] - S.st[q], t);
    st ^= (((uint32_t)S.pre >> q) ^ (uint32_t)r) & 1u ? (1u << q) : 0u;
  }
  return st;
}

// A thread's running sums of its events' totals; the leakage term dP (t_max -
// t) is large and of either sign (a gate's steps almost cancel), so its sum is
// compensated (Kahan, c_lk) and the warp sums are taken in fp64.
struct Acc {
  float e_int, e_sw, e_gl, e_lk, c_lk;
};

__device__ __forceinline__ void kahan_add(float& sum, float& comp, float x) {
  const float y = x - comp;
  const float t = sum + y;
  comp = (t - sum) - y;
  sum = t;
}

template <bool kPow2, bool kDebug, bool kExact>
__device__ __forceinline__ void do_event(const RunArgs& a, const float* __restrict__ ts,
                                         const float* __restrict__ ss, const Slot& S, int p, int e,
                                         const CellDesc* cells, bool have_prev0, float prev_t0,
                                         float prev_s0, uint64_t gidx, Acc& acc) {
  const int idx = e - (int)S.st[p];
  if (idx >= (int)S.np[p]) return;
  const float t = ts[e], s = ss[e];
  const uint32_t c = cycle_of<kPow2>(t, a.t_clk, a.inv_t_clk);
  bool has_prev = have_prev0;
  float tp = prev_t0, sp = prev_s0;
  if (idx > 0) {
    has_prev = true;
    tp = ts[e - 1];
    sp = ss[e - 1];
  }
  bool glitch = has_prev && cycle_of<kPow2>(tp, a.t_clk, a.inv_t_clk) == c;
  bool fwd = false;  // glitch-all reading: the first event of a pin-cycle takes the pulse to the next
  if (kDebug && a.glitch_all && !glitch) {  // the alternative readings run in the per-event path
    const GateRec gr = a.gates[S.gate];
    if (gidx + 1 < a.pin_off[(uint64_t)gr.pin_base + p + 1]) {
      const float tn = a.t[gidx + 1];
      if (cycle_of<kPow2>(tn, a.t_clk, a.inv_t_clk) == c) {
        glitch = fwd = true;
        tp = tn;
        sp = a.s[gidx + 1];
      }
    }
  }
  const int k = S.k;
  float e_int = 0.f, e_sw = 0.f, dp = 0.f;
  uint32_t s_pre = 0;
  int li = 0;
  if (p == k) {
    e_sw = S.esw;
    if (kDebug && a.esw_rise) {  // C V^2 on a rise: the output's new value from its initial one and its rank
      const GateRec gr = a.gates[S.gate];
      const uint64_t rank = gidx - a.pin_off[(uint64_t)gr.pin_base + k];
      e_sw = ((((gr.init >> 8) & 1u) ^ (uint32_t)((rank + 1) & 1u)) != 0u) ? 2.f * S.esw : 0.f;
    }
    if (kDebug) s_pre = state_before(ts, S, t);
  } else {
    const CellDesc& cd = cells[S.cell];
    // own pin: value before this event = initial value flipped per earlier event
    s_pre = (uint32_t)S.init ^ (((((uint32_t)S.pre >> p) ^ (uint32_t)idx) & 1u) << p);
    uint32_t s_b = s_pre;  // state just before this event in (time, pin) order
    for (int q = 0; q < k; ++q) {
      if (q == p) continue;
      const int qa = S.st[q], qn = (int)S.st[q + 1] - qa;
      const int r = lower_bound_f(ts + qa, qn, t);
      const bool eq = r < qn && ts[qa + r] == t;
      const uint32_t par = (((uint32_t)S.pre >> q) ^ (uint32_t)r) & 1u;
      s_pre ^= par << q;
      s_b ^= ((par ^ (uint32_t)(q < p && eq)) & 1u) << q;
    }
    // state-selected table, bilinear on (slew, load)
    const int ns = cd.ns, nl = cd.nl;
    for (int m = 1; m <= ns - 2; ++m) li += (s >= cd.sax[m]) ? 1 : 0;
    const float u = (s - cd.sax[li]) * cd.isax[li];
    const float* L = a.lut + cd.lut_off + ((int)s_pre * ns + li) * nl + S.j;
    const float l00 = __ldg(L), l01 = __ldg(L + 1), l10 = __ldg(L + nl), l11 = __ldg(L + nl + 1);
    const float r0 = fmaf(S.v, l01 - l00, l00), r1 = fmaf(S.v, l11 - l10, l10);
    e_int = fmaf(u, r1 - r0, r0);
    const float* lk = a.leak + cd.leak_off;
    dp = __ldg(lk + (s_b ^ (1u << p))) - __ldg(lk + s_b);
  }
  const float e_dyn = e_int + e_sw;
  float e_w;
  if (glitch) {
    const float r = fminf(1.f, 2000.f * (fwd ? tp - t : t - tp) / (s + sp));
    e_w = r * e_dyn;
    acc.e_gl += e_w;
  } else {
    acc.e_int += e_int;
    acc.e_sw += e_sw;
    e_w = e_dyn;
  }
  const float e_dyn_w = e_w;  // the event's dynamic (or glitch) energy
  if (p < k) {
    const float rem = fmaf(-(float)c, a.t_clk, t);  // t - c T
    e_w = fmaf(dp, a.t_clk - rem, e_w);
    kahan_add(acc.e_lk, acc.c_lk, dp * (a.t_max_f - t));
  }
  if (kExact) {
    // dense cycles: fp64 energy and step sums, integer counts
    double* bin = reinterpret_cast<double*>(a.bins + c);
    atomicAdd(bin, (double)e_w);
    if (p < k) atomicAdd(bin + 1, (double)dp);
    atomicAdd(a.cnt_ev + c, 1u);
    if (glitch) atomicAdd(a.cnt_gl + c, 1u);
  } else {
    float* bin = reinterpret_cast<float*>(a.bins + c);
    // one 16-byte reduction per event: energy, leakage step, event and glitch counts
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(bin), "f"(e_w), "f"(dp), "f"(1.0f),
                 "f"(glitch ? 1.0f : 0.0f)
                 : "memory");
  }
  if (kDebug) {
    if (a.dbg_state) a.dbg_state[gidx] = (uint8_t)s_pre;
    if (a.dbg_lut) a.dbg_lut[gidx] = p < k ? (uint8_t)((li << 4) | S.j) : (uint8_t)0xFF;
    if (a.dbg_glitch) a.dbg_glitch[gidx] = (uint8_t)glitch;
    if (a.gate_e) {  // this event's share of its gate's energies
      double* ge = a.gate_e + (size_t)S.gate * 4;
      if (glitch) {
        atomicAdd(ge + 2, (double)e_dyn_w);
      } else if (p < k) {
        atomicAdd(ge + 0, (double)e_int);
      } else {
        atomicAdd(ge + 1, (double)e_sw);
      }
      if (p < k) atomicAdd(ge + 3, (double)(dp * (a.t_max_f - t)));
    }
  }
}

__device__ __forceinline__ void fill_slot(const RunArgs& a, const CellDesc* cells, Slot& S, uint32_t g,
                                          uint64_t ea) {
  const GateRec r = a.gates[g];
  const int k = (int)((r.init >> 16) & 0xff);
  const CellDesc& cd = cells[r.cell];
  for (int p = 0; p <= k + 1; ++p) S.st[p] = (uint16_t)(a.pin_off[r.pin_base + p] - ea);
  for (int p = 0; p <= k; ++p) S.np[p] = (uint16_t)(S.st[p + 1] - S.st[p]);
  S.k = (uint8_t)k;
  S.init = (uint8_t)(r.init & 0xffu);
  S.pre = 0;
  S.cell = r.cell;
  const float C = r.load;
  int j = 0;
  for (int m = 1; m <= cd.nl - 2; ++m) j += (C >= cd.lax[m]) ? 1 : 0;
  S.j = (uint8_t)j;
  S.v = (C - cd.lax[j]) * cd.ilax[j];
  S.esw = a.half_vdd2 * C;
  S.gate = g;
}

__device__ __forceinline__ void flush_acc(Acc& acc, double* s_tot) {
  const double v0 = warp_sum_f64(acc.e_int), v1 = warp_sum_f64(acc.e_sw);
  const double v2 = warp_sum_f64(acc.e_gl), v3 = warp_sum_f64((double)acc.e_lk - (double)acc.c_lk);
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(s_tot + 0, v0);
    atomicAdd(s_tot + 1, v1);
    atomicAdd(s_tot + 2, v2);
    atomicAdd(s_tot + 3, v3);
  }
  acc = Acc{0.f, 0.f, 0.f, 0.f, 0.f};
}

template <bool kPow2, bool kDebug, bool kExact>
__global__ void __launch_bounds__(kThreads) k_fused(const RunArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* ts = reinterpret_cast<float*>(smem);
  float* ss = ts + kTileCap;
  uint16_t* tag = reinterpret_cast<uint16_t*>(ss + kTileCap);
  Slot* slots = reinterpret_cast<Slot*>(smem + 2 * kSmemT + kSmemTag);
  CellDesc* cells_s = reinterpret_cast<CellDesc*>(smem + 2 * kSmemT + kSmemTag + kSmemSlots);
  __shared__ HeavyState hs;
  __shared__ uint32_t s_item;
  __shared__ double s_tot[4];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kThreads / 32;
  if (tid < 4) s_tot[tid] = 0.0;
  const bool cells_in_smem = a.n_cells <= (uint32_t)kSmemCells;
  if (cells_in_smem) {
    const int words = (int)(a.n_cells * sizeof(CellDesc) / 4);
    const uint32_t* src = reinterpret_cast<const uint32_t*>(a.cells);
    uint32_t* dst = reinterpret_cast<uint32_t*>(cells_s);
    for (int i = tid; i < words; i += kThreads) dst[i] = src[i];
  }
  const CellDesc* cells = cells_in_smem ? cells_s : a.cells;
  const uint32_t n_tiles = a.part_counts[0], n_heavy = a.part_counts[1];
  const uint32_t n_items = n_tiles + n_heavy;
  Acc acc{0.f, 0.f, 0.f, 0.f, 0.f};
  __syncthreads();

  for (;;) {
    if (tid == 0) s_item = atomicAdd(a.part_counts + 2, 1u);
    __syncthreads();
    const uint32_t item = s_item;
    if (item >= n_items) break;

    if (item < n_heavy) {
      // ---------------- heavy gate: stream in event-count windows
      const uint32_t g = a.heavy[item];
      Slot& S = slots[0];
      if (tid == 0) {
        fill_slot(a, cells, S, g, 0);  // st/np overwritten per step below
        const GateRec r = a.gates[g];
        for (int p = 0; p <= S.k; ++p) {
          hs.cur[p] = a.pin_off[r.pin_base + p];
          hs.end[p] = a.pin_off[r.pin_base + p + 1];
          hs.has_prev[p] = 0;
          hs.prev_t[p] = 0.f;
          hs.prev_s[p] = 0.f;
        }
        hs.done = 0;
      }
      __syncthreads();
      const int k = S.k;
      for (;;) {
        if (tid == 0) {
          uint64_t R = 0;
          for (int p = 0; p <= k; ++p) R += hs.end[p] - hs.cur[p];
          if (R == 0) {
            hs.done = 1;
          } else {
            const uint64_t budget = (uint64_t)(kTileCap - (k + 1));
            uint32_t pos = 0;
            for (int p = 0; p <= k; ++p) {
              const uint64_t r = hs.end[p] - hs.cur[p];
              uint64_t ap = 0;
              if (r > 0) {
                const uint64_t share = budget * r / R;
                ap = share < 1 ? 1 : share;
                if (ap > r) ap = r;
              }
              S.st[p] = (uint16_t)pos;
              pos += (uint32_t)ap;
            }
            S.st[k + 1] = (uint16_t)pos;
          }
        }
        __syncthreads();
        if (hs.done) break;
        if (tid <= k) {  // first event past each pin's chunk bounds the window
          const uint64_t nx = hs.cur[tid] + (uint64_t)(S.st[tid + 1] - S.st[tid]);
          hs.bound[tid] = nx < hs.end[tid] ? a.t[nx] : FLT_MAX;
        }
        const int n = S.st[k + 1];
        for (int i = tid; i < n; i += kThreads) {
          int p = 0;
          for (int q = 1; q <= k; ++q) p += (i >= (int)S.st[q]) ? 1 : 0;
          const uint64_t ge = hs.cur[p] + (uint64_t)(i - (int)S.st[p]);
          ts[i] = a.t[ge];
          ss[i] = a.s[ge];
          tag[i] = (uint16_t)p;
        }
        __syncthreads();
        if (tid <= k) {
          float tau = FLT_MAX;
          for (int q = 0; q <= k; ++q) tau = fminf(tau, hs.bound[q]);
          const int len = (int)S.st[tid + 1] - (int)S.st[tid];
          // events at or after the horizon wait for the next window (a
          // timestamp group is never split); with no horizon take all
          S.np[tid] = (uint16_t)(tau == FLT_MAX ? len : lower_bound_f(ts + S.st[tid], len, tau));
        }
        __syncthreads();
        for (int i = tid; i < n; i += kThreads) {
          const int p = tag[i];
          do_event<kPow2, kDebug, kExact>(a, ts, ss, S, p, i, cells, hs.has_prev[p] != 0, hs.prev_t[p],
                                  hs.prev_s[p], hs.cur[p] + (uint64_t)(i - (int)S.st[p]), acc);
        }
        flush_acc(acc, s_tot);
        __syncthreads();
        if (tid == 0) {
          uint32_t moved = 0;
          for (int p = 0; p <= k; ++p) {
            const uint32_t m = S.np[p];
            if (m > 0) {
              hs.prev_t[p] = ts[S.st[p] + m - 1];
              hs.prev_s[p] = ss[S.st[p] + m - 1];
              hs.has_prev[p] = 1;
              hs.cur[p] += m;
              S.pre ^= (uint8_t)((m & 1u) << p);
              moved += m;
            }
          }
          if (moved == 0) {  // cannot happen for valid input; never spin
            dev_err(a.err, g, kErrTileOverflow);
            hs.done = 1;
          }
        }
        __syncthreads();
        if (hs.done) break;
      }
      __syncthreads();
    } else {
      // ---------------- light tile: consecutive whole gates
      const Tile tl = a.tiles[item - n_heavy];
      const uint64_t ea = a.gate_off[tl.gb], eb = a.gate_off[tl.ge];
      const uint64_t n64 = eb - ea;
      const uint32_t ng = tl.ge - tl.gb;
      if (n64 > (uint64_t)kTileCap || ng > (uint32_t)kGateCap || tl.ge <= tl.gb) {
        if (tid == 0) dev_err(a.err, tl.gb, kErrTileOverflow);
        __syncthreads();
        continue;
      }
      const int n = (int)n64;
      if (n == 0) {
        __syncthreads();
        continue;
      }
      for (int i = tid; i < n; i += kThreads) {
        ts[i] = a.t[ea + i];
        ss[i] = a.s[ea + i];
      }
      for (uint32_t gi = tid; gi < ng; gi += kThreads) fill_slot(a, cells, slots[gi], tl.gb + gi, ea);
      __syncthreads();
      for (uint32_t gi = warp; gi < ng; gi += kWarps) {
        const Slot& S = slots[gi];
        const int k = S.k;
        for (int e = (int)S.st[0] + lane; e < (int)S.st[k + 1]; e += 32) {
          int p = 0;
          for (int q = 1; q <= k; ++q) p += (e >= (int)S.st[q]) ? 1 : 0;
          tag[e] = (uint16_t)((gi << 3) | (uint32_t)p);
        }
      }
      __syncthreads();
      for (int e = tid; e < n; e += kThreads) {
        const uint32_t tg = tag[e];
        do_event<kPow2, kDebug, kExact>(a, ts, ss, slots[tg >> 3], (int)(tg & 7u), e, cells, false, 0.f, 0.f,
                                ea + (uint64_t)e, acc);
      }
      flush_acc(acc, s_tot);
      __syncthreads();
    }
  }
  __syncthreads();
  if (tid < 4) atomicAdd(a.totals + tid, s_tot[tid]);
}

template <bool P, bool D, bool X>
static void set_fused_attrs() {
  static bool done = false;
  if (!done) {
    cudaFuncSetAttribute(k_fused<P, D, X>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemTotal);
    done = true;
  }
}

template <bool P, bool D, bool X>
static int occupancy_of() {
  set_fused_attrs<P, D, X>();
  int n = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_fused<P, D, X>, kThreads, kSmemTotal);
  return n;
}

template <bool P, bool D, bool X>
static void launch_of(const RunArgs& a, int grid, cudaStream_t st) {
  set_fused_attrs<P, D, X>();
  k_fused<P, D, X><<<grid, kThreads, kSmemTotal, st>>>(a);
}

int fused_blocks_per_sm(bool pow2, bool debug, bool exact) {
  const int sel = (pow2 ? 4 : 0) | (debug ? 2 : 0) | (exact ? 1 : 0);
  int n = 0;
  switch (sel) {
    case 0: n = occupancy_of<false, false, false>(); break;
    case 1: n = occupancy_of<false, false, true>(); break;
    case 2: n = occupancy_of<false, true, false>(); break;
    case 3: n = occupancy_of<false, true, true>(); break;
    case 4: n = occupancy_of<true, false, false>(); break;
    case 5: n = occupancy_of<true, false, true>(); break;
    case 6: n = occupancy_of<true, true, false>(); break;
    default: n = occupancy_of<true, true, true>(); break;
  }
  return n > 0 ? n : 1;
}

cudaError_t launch_fused(const RunArgs& a, int grid, bool pow2, bool debug, bool exact, cudaStream_t st) {
  const int sel = (pow2 ? 4 : 0) | (debug ? 2 : 0) | (exact ? 1 : 0);
  switch (sel) {
    case 0: launch_of<false, false, false>(a, grid, st); break;
    case 1: launch_of<false, false, true>(a, grid, st); break;
    case 2: launch_of<false, true, false>(a, grid, st); break;
    case 3: launch_of<false, true, true>(a, grid, st); break;
    case 4: launch_of<true, false, false>(a, grid, st); break;
    case 5: launch_of<true, false, true>(a, grid, st); break;
    case 6: launch_of<true, true, false>(a, grid, st); break;
    default: launch_of<true, true, true>(a, grid, st); break;
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------ final reduction
//
// Prefix-sums the per-cycle leakage steps in fp64 and adds the leakage power
// held over each cycle, (P0 + steps of earlier cycles) * the cycle's length
// inside [0, t_max), to the cycle's energy bin; converts bins to W (energy /
// t_clk). Totals: P_x = E_x / t_max (Eq. 3), with E_leak = P0 t_max + sum over
// input events of dP (t_max - t). Two kernels over chunks of kReduceChunk
// cycles: step sums per chunk, then a block scan per chunk on top of the sum of
// the chunks before it.

constexpr int kRedThreads = 256;
constexpr int kRedPer = (int)kReduceChunk / kRedThreads;  // cycles per thread

// Energy W and step D of cycle c: f32 {W, D, ev, gl} bins (the sum of their
// copies), or fp64 {W, D} bins (same 16 bytes) when counts are taken exactly.
template <bool kExact>
__device__ __forceinline__ double2 bin_wd(const RunArgs& a, uint32_t c) {
  if (kExact) return reinterpret_cast<const double2*>(a.bins)[c];
  double2 r = make_double2(0.0, 0.0);
#pragma unroll
  for (uint32_t k = 0; k < kBinCopies; ++k) {  // (all copies' loads in flight at once)
    if (k == 0 || k < a.n_rep) {
      const float4 v = a.bins[(size_t)k * a.n_cycles + c];
      r.x += (double)v.x;
      r.y += (double)v.y;
    }
  }
  return r;
}

template <bool kExact>
__global__ void __launch_bounds__(kRedThreads) k_reduce_chunks(const RunArgs a) {
  const uint32_t c0 = blockIdx.x * kReduceChunk;
  double s = 0.0;
  for (uint32_t i = threadIdx.x; i < kReduceChunk; i += kRedThreads) {
    const uint32_t c = c0 + i;
    if (c < a.n_cycles) s += bin_wd<kExact>(a, c).y;
  }
  __shared__ double ws[kRedThreads / 32];
  s = warp_sum_f64(s);
  if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int i = 0; i < kRedThreads / 32; ++i) t += ws[i];
    a.chunk_sums[blockIdx.x] = t;
  }
}

template <bool kExact>
__global__ void __launch_bounds__(kRedThreads) k_reduce_apply(const RunArgs a, double T, double t_max, float* wave,
                                                            double* p_out) {
  __shared__ double wsum[kRedThreads / 32];
  __shared__ double s_base;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (w == 0) {  // P0 + the step sums of the chunks before this one (the first warp's lanes in parallel)
    double b = 0.0;
    for (uint32_t j = (uint32_t)lane; j < blockIdx.x; j += 32) b += a.chunk_sums[j];
    b = warp_sum_f64(b);
    if (lane == 0) s_base = *a.p0 + b;
  }
  const uint32_t c0 = blockIdx.x * kReduceChunk + (uint32_t)tid * kRedPer;
  double2 v[kRedPer];
  double local = 0.0;
#pragma unroll
  for (int i = 0; i < kRedPer; ++i) {
    const uint32_t c = c0 + i;
    v[i] = c < a.n_cycles ? bin_wd<kExact>(a, c) : make_double2(0.0, 0.0);
    local += v[i].y;
  }
  double incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  double pre = s_base + incl - local;
  for (int i = 0; i < w; ++i) pre += wsum[i];
  bool overflow = false;
#pragma unroll
  for (int i = 0; i < kRedPer; ++i) {
    const uint32_t c = c0 + i;
    if (c >= a.n_cycles) break;
    const double lo = (double)c * T, hi = lo + T;
    const double len = t_max >= hi ? T : (t_max > lo ? t_max - lo : 0.0);
    const double d = v[i].y;
    double e = v[i].x + pre * len;
    if (t_max > lo && t_max < hi) e -= d * (hi - t_max);
    if (wave) wave[c] = (float)(e / T * 1e-6);
    if (!kExact) {
      // f32 counts are exact integers while below 2^24: a cycle with 2^24
      // events or more in all repeats the pass with integer counts
      uint32_t ne = 0, ng = 0;
#pragma unroll
      for (uint32_t k = 0; k < kBinCopies; ++k) {
        if (k > 0 && k >= a.n_rep) continue;
        const float4 f = a.bins[(size_t)k * a.n_cycles + c];
        if (f.z >= 16777216.0f) overflow = true;
        ne += (uint32_t)f.z;
        ng += (uint32_t)f.w;
      }
      if (ne >= (1u << 24)) overflow = true;
      if (a.cnt_ev) a.cnt_ev[c] = ne;
      if (a.cnt_gl) a.cnt_gl[c] = ng;
    }
    pre += d;
  }
  if (overflow) dev_err(a.err, 0, kErrCountOverflow);
  if (blockIdx.x == 0 && tid == 0) {
    const double e_leak = *a.p0 * t_max + a.totals[3];
    p_out[0] = a.totals[0] / t_max * 1e-6;
    p_out[1] = a.totals[1] / t_max * 1e-6;
    p_out[2] = a.totals[2] / t_max * 1e-6;
    p_out[3] = e_leak / t_max * 1e-6;
  }
}

cudaError_t launch_final_reduce(const RunArgs& a, double t_clk, double t_max, float* wave_out,
                                double* p_out, bool exact, cudaStream_t st) {
  const uint32_t nc = reduce_chunks(a.n_cycles);
  if (exact) k_reduce_chunks<true><<<nc, kRedThreads, 0, st>>>(a);
  else k_reduce_chunks<false><<<nc, kRedThreads, 0, st>>>(a);
  if (exact) k_reduce_apply<true><<<nc, kRedThreads, 0, st>>>(a, t_clk, t_max, wave_out, p_out);
  else k_reduce_apply<false><<<nc, kRedThreads, 0, st>>>(a, t_clk, t_max, wave_out, p_out);
  return cudaGetLastError();
}

}  // namespace pa

// ------------------------------------------------------------------ per-gate power

namespace pa {

namespace {

// Gate g's energies (fJ) -> power (W): E / t_max, and for leakage the initial
// state's leakage held over the whole window plus the gate's power steps
// carried to t_max, E_leak = leak(S0) t_max + sum dP (t_max - t).
__global__ void __launch_bounds__(256) k_gate_power(const RunArgs a, double t_max) {
  const uint64_t g = (uint64_t)blockIdx.x * 256u + threadIdx.x;
  if (g >= a.n_gates) return;
  const GateRec r = a.gates[g];
  const CellDesc& cd = a.cells[r.cell];
  const double p0 = (double)a.leak[cd.leak_off + (r.init & ((1u << cd.k) - 1u))];  // uW
  double* ge = a.gate_e + g * 4;
  const double f = 1e-6 / t_max;  // fJ / ns = uW -> W
  ge[0] *= f;
  ge[1] *= f;
  ge[2] *= f;
  ge[3] = (p0 * t_max + ge[3]) * f;
  if (a.cell_p) {
    double* cp = a.cell_p + (size_t)r.cell * 4;
#pragma unroll
    for (int m = 0; m < 4; ++m) atomicAdd(cp + m, ge[m]);
  }
}

}  // namespace

cudaError_t launch_gate_power(const RunArgs& a, double t_max, cudaStream_t st) {
  if (a.n_gates && a.gate_e) k_gate_power<<<(a.n_gates + 255) / 256, 256, 0, st>>>(a, t_max);
  return cudaGetLastError();
}

}  // namespace pa

// ------------------------------------------------------------------ chunk rebasing (pa_run_stream)

namespace pa {

namespace {

__global__ void __launch_bounds__(256) k_rebase_pin_off(uint64_t* p, uint64_t n, uint64_t base) {
  const uint64_t i = (uint64_t)blockIdx.x * 256u + threadIdx.x;
  if (i < n) p[i] -= base;
}

__global__ void __launch_bounds__(256) k_rebase_gates(const GateRec* __restrict__ src, GateRec* dst, uint32_t n,
                                                      uint32_t pin0) {
  const uint32_t g = blockIdx.x * 256u + threadIdx.x;
  if (g < n) {
    GateRec r = src[g];
    r.pin_base -= pin0;
    dst[g] = r;
  }
}

}  // namespace

cudaError_t launch_rebase_chunk(uint64_t* pin_off, uint64_t n_pins, uint64_t ev0, const GateRec* gates_src,
                                GateRec* gates_dst, uint32_t n_gates, uint32_t pin0, cudaStream_t st) {
  if (n_pins + 1) k_rebase_pin_off<<<(unsigned)((n_pins + 1 + 255) / 256), 256, 0, st>>>(pin_off, n_pins + 1, ev0);
  if (n_gates) k_rebase_gates<<<(n_gates + 255) / 256, 256, 0, st>>>(gates_src, gates_dst, n_gates, pin0);
  return cudaGetLastError();
}

}  // namespace pa
