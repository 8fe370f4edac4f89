// The fused dynamic + leakage power kernel on the loaded per-pin (CSR)
// layout, one warp per work item, with its partition. The computation is the
// power step of "GPU-Accelerated Gate-Level Time-Based Power Analysis via
// Event-Density-Aware Partitioning and Kernel Fusion" (Sections 2.4.1-2.4.2,
// Eqs. 1-4, Figs. 2, 3 and 7), the same per-event arithmetic as the CTA kernel
// of pa_kernels.cu (k_fused); the mapping onto the GPU differs:
//
//  * Partition (inside the run, every pass). Gates with at most heavy_thresh
//    events are grouped into light tiles of consecutive whole gates (a tile
//    starts where a gate's first event enters a new tile_target-sized bucket,
//    after a heavy gate, and every kCsrGates gates), so a tile holds fewer
//    than tile_target + heavy_thresh events. A heavy gate with n_g events is
//    cut into ceil(n_g / kCsrPiece) pieces at times taken from its densest
//    pin (whose events are split evenly); every pin is split at its first
//    event at or after each such time. A piece thus holds all of the gate's
//    events in a time interval: the dense gates get short time windows and
//    the sparse ones whole timelines, the role of the event-density-aware
//    per-gate partitioning of Figs. 5, 19 and 20, cut by event count.
//  * One warp per item, no CTA-wide barrier in the item loop. A light tile's
//    times and slews are one contiguous range, staged with 16-byte loads; a
//    lane per gate fills the gate's slot (pin starts, cell, load-axis
//    interval and fraction, switching energy). A piece is staged in windows of
//    at most kCsrWin events shared among its pins in proportion to their
//    remaining events; the events before the earliest first unstaged event of
//    any pin are taken, so every pin's events earlier than a taken event are
//    either staged or counted in the pin's parity.
//  * One lane per event. The gate state before the event's timestamp: each
//    input pin's initial value flipped once per earlier event, the count on
//    another pin being a binary search of t in that pin's staged events (ties
//    see the pre-timestamp state; the leakage step is taken in (time, pin)
//    order, so simultaneous steps telescope). The slew interval by a
//    three-step search over the cell's axis in shared memory, the state's four
//    LUT corners in one 16-byte load, the leakage per state in shared memory.
//    Glitch: the previous event of the same pin in the same cycle (the CSR
//    neighbour). Each event adds {energy, leakage step, 1, glitch} to its
//    cycle's bin with one red.global.add.v4.f32; per-lane totals (the
//    leakage term compensated) are reduced in fp64.
#include <cfloat>
#include <cstdint>

#include "pa_internal.cuh"

namespace pa {

namespace {

constexpr int kCW = 32;               // warps per CTA
constexpr int kCT = kCW * 32;
constexpr int kStCap = 528;           // staged events per warp: 512 + 16-byte alignment slack
constexpr int kAx = 9;                // slew axis stride of the cell table (odd: lanes of different cells spread)
constexpr int kLk = 17;               // leakage stride of the cell table
constexpr int kTotEvery = 16;         // items between flushes of a warp's per-lane totals

// Cell tables in shared memory (libraries of at most kSmemCells cells): per
// cell the slew axis points 0..8 (+inf past ns - 2), an info word (ns - 1 |
// (nl - 1) << 8 | patch offset << 16), per slew interval {axis point, 1 /
// width}, and the leakage per state (uW).
constexpr size_t kCellsB =
    (size_t)kSmemCells * kAx * 4 + (size_t)kSmemCells * 4 + (size_t)kSmemCells * 8 * 8 + (size_t)kSmemCells * kLk * 4;

// Per gate of the warp's current item.
struct __align__(16) CSlot {
  uint16_t st[kMaxK + 2];    // staged start of pins 0..k; st[k + 1] = end
  uint8_t k, init, j, pre;   // inputs, initial input bits, load-axis interval, parity of earlier events per pin
  uint16_t cell, pad;
  float v, esw;              // load-axis fraction; switching energy C V^2 / 2 (fJ)
};
static_assert(sizeof(CSlot) == 32, "slot size");

// Per pin of a piece's current window.
struct HWin {
  uint16_t np[kMaxK + 1];    // events of the pin taken in this window
  uint8_t hp[kMaxK + 1];     // the pin has an event before the window
  float pt[kMaxK + 1], ps[kMaxK + 1];  // that event's time and slew
  uint64_t src[kMaxK + 1];   // global index of the window's first staged event of the pin
};

constexpr size_t kWarpB = (size_t)kStCap * 4 * 2 + kStCap + sizeof(CSlot) * kCsrGates + 128;
static_assert(sizeof(HWin) <= 128, "window record");
static_assert(kWarpB % 16 == 0 && kCellsB % 16 == 0, "alignment");
constexpr size_t kSmemB = kCellsB + (size_t)kCW * kWarpB;
static_assert(kSmemB + 1024 <= 227 * 1024, "shared memory budget");

struct CTab {
  const float* sax;
  const uint32_t* info;
  const float2* sxp;
  const float* leak;
};

struct Acc {
  float e_int, e_sw, e_gl, e_lk, c_lk;
};

__device__ __forceinline__ void kahan_add(float& sum, float& comp, float x) {
  const float y = x - comp;
  const float t = sum + y;
  comp = (t - sum) - y;
  sum = t;
}

__device__ __forceinline__ void flush_acc(Acc& acc, double* s_tot) {
  double v[4] = {acc.e_int, acc.e_sw, acc.e_gl, (double)acc.e_lk - (double)acc.c_lk};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
  }
  if ((threadIdx.x & 31) == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) atomicAdd(s_tot + i, v[i]);
  }
  acc = Acc{0.f, 0.f, 0.f, 0.f, 0.f};
}

__device__ __forceinline__ void dev_err(unsigned long long* err, uint64_t idx, uint32_t code) {
  atomicMin(err, (unsigned long long)((idx << 8) | code));
}

template <bool kPow2>
__device__ __forceinline__ uint32_t cyc(float t, float T, float inv_T) {
  // floor(fl32(t / T)) for t >= 0; with T a power of two t * (1/T) is the
  // same correctly rounded quotient
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

// Gate g's slot: cell, inputs, initial bits, load-axis interval and
// fraction, switching energy; pin starts relative to `base` (light tiles).
__device__ __forceinline__ void fill_slot(const RunArgs& a, CSlot& S, uint32_t g, uint64_t base, bool starts) {
  const GateRec r = a.gates[g];
  const int k = (int)((r.init >> 16) & 0xff);
  const CellDesc& cd = a.cells[r.cell];
  if (starts)
    for (int p = 0; p <= k + 1; ++p) S.st[p] = (uint16_t)(a.pin_off[r.pin_base + p] - base);
  S.k = (uint8_t)k;
  S.init = (uint8_t)(r.init & 0xffu);
  S.pre = 0;
  S.cell = (uint16_t)r.cell;
  const float C = r.load;
  int j = 0;
  for (int m = 1; m <= cd.nl - 2; ++m) j += (C >= cd.lax[m]) ? 1 : 0;
  S.j = (uint8_t)j;
  S.v = (C - cd.lax[j]) * cd.ilax[j];
  S.esw = a.half_vdd2 * C;
}

// One event: staged index i of pin p of slot S; (has_prev, tp, *spp) the
// pin's previous event (time; slew, read only for a glitch).
template <bool kPow2>
__device__ __forceinline__ void csr_event(const RunArgs& a, const CTab& CT, const float* ts, const float* ss,
                                          const CSlot& S, int p, int i, bool has_prev, float tp, const float* spp,
                                          Acc& acc) {
  const float t = ts[i], s = ss[i];
  const float T = a.t_clk;
  const uint32_t c = cyc<kPow2>(t, T, a.inv_t_clk);
  const bool glitch = has_prev && cyc<kPow2>(tp, T, a.inv_t_clk) == c;
  const int k = S.k;
  float e_int = 0.f, e_sw = 0.f, dp = 0.f;
  if (p == k) {
    e_sw = S.esw;
  } else {
    // own pin: value before this event = initial value flipped per earlier event
    const int idx = i - (int)S.st[p];
    uint32_t s_pre = (uint32_t)S.init ^ (((((uint32_t)S.pre >> p) ^ (uint32_t)idx) & 1u) << p);
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
    const uint32_t cell = S.cell;
    const uint32_t info = CT.info[cell];  // ns - 1 | (nl - 1) << 8 | patch offset << 16
    // slew interval: the number of axis points 1 .. ns - 2 that are <= s
    const float* axs = CT.sax + cell * kAx;
    int lis = s >= axs[4] ? 4 : 0;
    lis += s >= axs[lis + 2] ? 2 : 0;
    lis += s >= axs[lis + 1] ? 1 : 0;
    const float2 ax = CT.sxp[cell * 8 + lis];
    const float u = (s - ax.x) * ax.y;
    // corners {L[i][j], L[i][j+1], L[i+1][j], L[i+1][j+1]} of the state's table
    const float4 P = __ldg(a.patch + (info >> 16) +
                           ((int)s_pre * (int)(info & 0xFFu) + lis) * (int)((info >> 8) & 0xFFu) + S.j);
    const float r0 = fmaf(S.v, P.y - P.x, P.x), r1 = fmaf(S.v, P.w - P.z, P.z);
    e_int = fmaf(u, r1 - r0, r0);
    const float* lk = CT.leak + cell * kLk;
    dp = lk[s_b ^ (1u << p)] - lk[s_b];
  }
  const float e_dyn = e_int + e_sw;
  float e_w;
  if (glitch) {
    // r_gl = min(1, x / y), IEEE division; x >= y gives 1 without dividing
    const float x = 2000.f * (t - tp), y = s + *spp;
    const float r = x < y ? __fdiv_rn(x, y) : 1.f;
    e_w = r * e_dyn;
    acc.e_gl += e_w;
  } else {
    acc.e_int += e_int;
    acc.e_sw += e_sw;
    e_w = e_dyn;
  }
  if (p < k) {
    const float rem = fmaf(-(float)c, T, t);  // t - c T: the step's part inside its own cycle
    e_w = fmaf(dp, T - rem, e_w);
    kahan_add(acc.e_lk, acc.c_lk, dp * (a.t_max_f - t));
  }
  float* bin = reinterpret_cast<float*>(a.bins + c);
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(bin), "f"(e_w), "f"(dp), "f"(1.0f),
               "f"(glitch ? 1.0f : 0.0f)
               : "memory");
}

// A light tile: consecutive whole gates, staged whole.
template <bool kPow2>
__device__ __forceinline__ void csr_tile(const RunArgs& a, const CTab& CT, uint32_t ti, float* ts0, float* ss0,
                                         uint8_t* tg, CSlot* slots, Acc& acc) {
  const int lane = threadIdx.x & 31;
  const Tile tl = a.tiles[ti];
  const uint32_t ng = tl.ge - tl.gb;
  if (tl.ge <= tl.gb || ng > kCsrGates) {
    if (lane == 0) dev_err(a.err, tl.gb, kErrTileOverflow);
    return;
  }
  const uint64_t ea = a.gate_off[tl.gb], eb = a.gate_off[tl.ge];
  if (eb < ea || eb - ea > (uint64_t)(kStCap - 4)) {
    if (lane == 0) dev_err(a.err, tl.gb, kErrTileOverflow);
    return;
  }
  const int n = (int)(eb - ea);
  if (n == 0) return;
  // times and slews [ea, eb) with 16-byte loads from ea rounded down (the
  // event arrays are padded past their end)
  const uint64_t e4 = ea & ~3ull;
  const int off = (int)(ea - e4), nv = (off + n + 3) >> 2;
  const float4* t4 = reinterpret_cast<const float4*>(a.t + e4);
  const float4* s4 = reinterpret_cast<const float4*>(a.s + e4);
  for (int v = lane; v < nv; v += 32) {
    reinterpret_cast<float4*>(ts0)[v] = __ldg(t4 + v);
    reinterpret_cast<float4*>(ss0)[v] = __ldg(s4 + v);
  }
  if (lane < (int)ng) fill_slot(a, slots[lane], tl.gb + (uint32_t)lane, ea, true);
  __syncwarp();
  const float* ts = ts0 + off;
  const float* ss = ss0 + off;
  // tags: slot << 3 | pin
  for (uint32_t gi = 0; gi < ng; ++gi) {
    const CSlot& S = slots[gi];
    const int k = S.k;
    for (int e = (int)S.st[0] + lane; e < (int)S.st[k + 1]; e += 32) {
      int p = 0;
      for (int q = 1; q <= k; ++q) p += (e >= (int)S.st[q]) ? 1 : 0;
      tg[e] = (uint8_t)((gi << 3) | (uint32_t)p);
    }
  }
  __syncwarp();
  for (int e = lane; e < n; e += 32) {
    const uint32_t w = tg[e];
    const CSlot& S = slots[w >> 3];
    const int p = (int)(w & 7u);
    const bool hp = e > (int)S.st[p];  // light gates are whole: the pin's previous event is staged
    csr_event<kPow2>(a, CT, ts, ss, S, p, e, hp, hp ? ts[e - 1] : 0.f, ss + e - 1, acc);
  }
  __syncwarp();  // the stage is read before the next item overwrites it
}

// A piece of a heavy gate, in windows of at most kCsrWin events.
template <bool kPow2>
__device__ __forceinline__ void csr_piece(const RunArgs& a, const CTab& CT, uint32_t pi, float* ts, float* ss,
                                          uint8_t* tg, CSlot& S, HWin& hw, Acc& acc) {
  const int lane = threadIdx.x & 31;
  const Piece& P = a.pieces[pi];
  const uint32_t g = P.gate, pidx = P.idx;
  const GateRec r = a.gates[g];
  const int k = (int)((r.init >> 16) & 0xff);
  const uint64_t n_g = a.gate_off[g + 1] - a.gate_off[g];
  const uint32_t m = (uint32_t)((n_g + kCsrPiece - 1) / kCsrPiece);
  const bool last = pidx + 1 >= m;
  const bool mine = lane <= k;  // lane p holds pin p
  uint64_t pst = 0;
  uint32_t cur = 0, hi = 0;
  bool hp = false;
  float ptv = 0.f, psv = 0.f;
  if (mine) {
    pst = a.pin_off[(uint64_t)r.pin_base + lane];
    const uint64_t pe = a.pin_off[(uint64_t)r.pin_base + lane + 1];
    cur = P.lo[lane];
    hi = last ? (uint32_t)(pe - pst) : a.pieces[pi + 1].lo[lane];
    if (hi < cur) hi = cur;  // (never for a consistent partition)
    if (cur > 0) {  // the pin's event before the piece
      hp = true;
      ptv = a.t[pst + cur - 1];
      psv = a.s[pst + cur - 1];
    }
  }
  if (lane == 0) fill_slot(a, S, g, 0, false);
  for (int guard = 0;; ++guard) {
    const uint32_t rem = mine ? hi - cur : 0u;
    const uint32_t R = __reduce_add_sync(0xffffffffu, rem);
    if (R == 0) break;
    uint32_t share = 0;
    if (rem) {
      const uint64_t sh = (uint64_t)kCsrWin * rem / R;
      share = sh < 1 ? 1u : (sh > rem ? rem : (uint32_t)sh);
    }
    uint32_t incl = share;  // prefix over lanes 0..k
#pragma unroll
    for (int d = 1; d <= 4; d <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += y;
    }
    const uint32_t st = incl - share;
    const int nw = (int)__shfl_sync(0xffffffffu, incl, k);
    // the first unstaged event of each pin bounds the window (+inf: none left)
    float bound = FLT_MAX;
    if (mine && cur + share < hi) bound = a.t[pst + cur + share];
    const bool bounded = __any_sync(0xffffffffu, mine && cur + share < hi);
    const float hz = __uint_as_float(__reduce_min_sync(0xffffffffu, __float_as_uint(bound)));  // t >= 0
    if (mine) {
      S.st[lane] = (uint16_t)st;
      hw.src[lane] = pst + cur;
      hw.hp[lane] = (uint8_t)hp;
      hw.pt[lane] = ptv;
      hw.ps[lane] = psv;
    }
    if (lane == 0) S.st[k + 1] = (uint16_t)nw;
    const uint32_t pre = __ballot_sync(0xffffffffu, mine && (cur & 1u)) & 31u;
    if (lane == 0) S.pre = (uint8_t)pre;
    __syncwarp();
    for (int i = lane; i < nw; i += 32) {
      int p = 0;
      for (int q = 1; q <= k; ++q) p += (i >= (int)S.st[q]) ? 1 : 0;
      const uint64_t src = hw.src[p] + (uint64_t)(i - (int)S.st[p]);
      ts[i] = a.t[src];
      ss[i] = a.s[src];
      tg[i] = (uint8_t)p;
    }
    __syncwarp();
    // the events before the horizon are taken (a timestamp group is never split)
    uint32_t take = share;
    if (mine && share > 0 && bounded) take = (uint32_t)lower_bound_f(ts + st, (int)share, hz);
    if (mine) hw.np[lane] = (uint16_t)take;
    __syncwarp();
    for (int i = lane; i < nw; i += 32) {
      const int p = tg[i];
      const int idx = i - (int)S.st[p];
      if (idx >= (int)hw.np[p]) continue;
      const bool has_prev = idx > 0 || hw.hp[p] != 0;
      const float tp = idx > 0 ? ts[i - 1] : hw.pt[p];
      const float* spp = idx > 0 ? ss + i - 1 : &hw.ps[p];
      csr_event<kPow2>(a, CT, ts, ss, S, p, i, has_prev, tp, spp, acc);
    }
    __syncwarp();
    if (mine && take > 0) {
      hp = true;
      ptv = ts[st + take - 1];
      psv = ss[st + take - 1];
      cur += take;
    }
    const uint32_t moved = __reduce_add_sync(0xffffffffu, mine ? take : 0u);
    __syncwarp();
    if (moved == 0 || guard > (1 << 24)) {  // cannot happen for valid input; never spin
      if (lane == 0) dev_err(a.err, g, kErrTileOverflow);
      break;
    }
  }
}

template <bool kPow2>
__global__ void __launch_bounds__(kCT, 1) k_csr(const RunArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ double s_tot[4];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float* sax = reinterpret_cast<float*>(smem);
  uint32_t* info = reinterpret_cast<uint32_t*>(sax + kSmemCells * kAx);
  float2* sxp = reinterpret_cast<float2*>(info + kSmemCells);
  float* lk = reinterpret_cast<float*>(sxp + kSmemCells * 8);
  uint8_t* wb = smem + kCellsB + (size_t)warp * kWarpB;
  float* ts = reinterpret_cast<float*>(wb);
  float* ss = ts + kStCap;
  uint8_t* tg = reinterpret_cast<uint8_t*>(ss + kStCap);
  CSlot* slots = reinterpret_cast<CSlot*>(tg + kStCap);
  HWin* hw = reinterpret_cast<HWin*>(slots + kCsrGates);
  if (tid < 4) s_tot[tid] = 0.0;
  {  // cell tables (the kernel runs for libraries of at most kSmemCells cells)
    const uint32_t nc = min(a.n_cells, (uint32_t)kSmemCells);
    for (uint32_t i = tid; i < nc * (uint32_t)kAx; i += kCT) {
      const uint32_t ci = i / kAx, m = i % kAx;
      const CellDesc& cd = a.cells[ci];
      if (m == 0) info[ci] = (uint32_t)(cd.ns - 1) | ((uint32_t)(cd.nl - 1) << 8) | (cd.patch_off << 16);
      sax[i] = m == 0 ? cd.sax[0] : ((int)m <= (int)cd.ns - 2 ? cd.sax[m] : __int_as_float(0x7f800000));
      if (m < 8) sxp[ci * 8 + m] = make_float2(cd.sax[m], cd.isax[m]);
    }
    for (uint32_t i = tid; i < nc * (uint32_t)kLk; i += kCT) {
      const uint32_t ci = i / kLk, st = i % kLk;
      const CellDesc& cd = a.cells[ci];
      lk[i] = st < (1u << cd.k) ? a.leak[cd.leak_off + st] : 0.f;
    }
  }
  __syncthreads();
  const CTab CT{sax, info, sxp, lk};
  const uint32_t n_tiles = a.part_counts[0], n_pieces = a.part_counts[1];
  const uint32_t n_items = n_tiles + n_pieces;
  Acc acc{0.f, 0.f, 0.f, 0.f, 0.f};
  int since = 0;
  for (;;) {
    uint32_t item = 0;
    if (lane == 0) item = atomicAdd(a.part_counts + 2, 1u);
    item = __shfl_sync(0xffffffffu, item, 0);
    if (item >= n_items) break;
    if (item < n_pieces)  // the heavy gates' pieces first: the longest items
      csr_piece<kPow2>(a, CT, item, ts, ss, tg, slots[0], *hw, acc);
    else
      csr_tile<kPow2>(a, CT, item - n_pieces, ts, ss, tg, slots, acc);
    if (++since == kTotEvery) {
      flush_acc(acc, s_tot);
      since = 0;
    }
  }
  flush_acc(acc, s_tot);
  __syncthreads();
  if (tid < 4) atomicAdd(a.totals + tid, s_tot[tid]);
}

// ------------------------------------------------------------------ partition

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Block-wide exclusive scan of two u32 values (256 threads).
__device__ __forceinline__ void scan2(uint32_t a, uint32_t b, uint32_t& ea, uint32_t& eb, uint32_t& ta,
                                      uint32_t& tb) {
  __shared__ uint32_t wa[8], wb[8];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t ia = warp_incl_scan(a, lane), ib = warp_incl_scan(b, lane);
  if (lane == 31) {
    wa[w] = ia;
    wb[w] = ib;
  }
  __syncthreads();
  uint32_t oa = 0, ob = 0, sa = 0, sb = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (i < w) {
      oa += wa[i];
      ob += wb[i];
    }
    sa += wa[i];
    sb += wb[i];
  }
  ea = oa + ia - a;
  eb = ob + ib - b;
  ta = sa;
  tb = sb;
  __syncthreads();
}

__device__ __forceinline__ uint64_t gate_events(const RunArgs& a, uint32_t g) {
  return a.gate_off[g + 1] - a.gate_off[g];
}

__device__ __forceinline__ bool heavy_gate(const RunArgs& a, uint32_t g) {
  return gate_events(a, g) > (uint64_t)a.heavy_thresh;
}

__device__ __forceinline__ uint32_t n_pieces_of(const RunArgs& a, uint32_t g) {
  const uint64_t n = gate_events(a, g);
  return n > (uint64_t)a.heavy_thresh ? (uint32_t)((n + kCsrPiece - 1) / kCsrPiece) : 0u;
}

__device__ __forceinline__ bool tile_head(const RunArgs& a, uint32_t g) {
  if (heavy_gate(a, g)) return false;
  if (g == 0 || g % kCsrGates == 0) return true;
  if (heavy_gate(a, g - 1)) return true;
  return a.gate_off[g] / a.tile_target != a.gate_off[g - 1] / a.tile_target;
}

__global__ void __launch_bounds__(256) k_cp_count(const RunArgs a) {
  const uint32_t g = blockIdx.x * 256u + threadIdx.x;
  uint32_t h = 0, pc = 0;
  double p0 = 0.0;
  if (g < a.n_gates) {
    pc = n_pieces_of(a, g);
    h = tile_head(a, g);
    const GateRec r = a.gates[g];
    const CellDesc& cd = a.cells[r.cell];
    p0 = (double)a.leak[cd.leak_off + (r.init & ((1u << cd.k) - 1u))];
  }
  uint32_t ea, eb, ta, tb;
  scan2(h, pc, ea, eb, ta, tb);
  if (threadIdx.x == 0) {
    a.part_blk[2 * blockIdx.x] = ta;
    a.part_blk[2 * blockIdx.x + 1] = tb;
  }
  __shared__ double sp[8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) p0 += __shfl_xor_sync(0xffffffffu, p0, o);
  if ((threadIdx.x & 31) == 0) sp[threadIdx.x >> 5] = p0;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0;
    for (int i = 0; i < 8; ++i) s += sp[i];
    atomicAdd(a.p0, s);
  }
}

__global__ void __launch_bounds__(256) k_cp_emit(const RunArgs a) {
  const uint32_t g = blockIdx.x * 256u + threadIdx.x;
  uint32_t h = 0, pc = 0, tail = 0;
  if (g < a.n_gates) {
    pc = n_pieces_of(a, g);
    h = tile_head(a, g);
    if (pc == 0) tail = (g + 1 == a.n_gates) || heavy_gate(a, g + 1) || tile_head(a, g + 1);
  }
  uint32_t ea, eb, ta, tb;
  scan2(h, pc, ea, eb, ta, tb);
  const uint32_t th = a.part_blk[2 * blockIdx.x] + ea;
  const uint32_t tv = a.part_blk[2 * blockIdx.x + 1] + eb;
  if (g < a.n_gates) {
    if (h) a.tiles[th].gb = g;
    if (tail) a.tiles[th + h - 1].ge = g + 1;
    for (uint32_t i = 0; i < pc; ++i) {
      a.pieces[tv + i].gate = g;
      a.pieces[tv + i].idx = i;
    }
  }
}

// Cut points of every piece: piece i > 0 of gate g starts, on each pin, at
// the first event at or after time tau_i, the time of event floor(i c / m)
// of the gate's densest pin (c events, m pieces).
__global__ void __launch_bounds__(256) k_cp_bounds(const RunArgs a) {
  const uint32_t n = a.part_counts[1];
  for (uint32_t pi = blockIdx.x * 256u + threadIdx.x; pi < n; pi += gridDim.x * 256u) {
    Piece& P = a.pieces[pi];
    const uint32_t g = P.gate, i = P.idx;
    const GateRec r = a.gates[g];
    const int k = (int)((r.init >> 16) & 0xff);
    uint32_t lo[kMaxK + 1] = {0, 0, 0, 0, 0};
    if (i > 0) {
      const uint64_t pb = r.pin_base;
      uint64_t cmax = 0;
      int pmax = 0;
      for (int p = 0; p <= k; ++p) {
        const uint64_t c = a.pin_off[pb + p + 1] - a.pin_off[pb + p];
        if (c > cmax) {
          cmax = c;
          pmax = p;
        }
      }
      const uint64_t m = (gate_events(a, g) + kCsrPiece - 1) / kCsrPiece;
      const float tau = a.t[a.pin_off[pb + pmax] + (uint64_t)i * cmax / m];
      for (int p = 0; p <= k; ++p) {
        const uint64_t b = a.pin_off[pb + p];
        uint64_t l = 0, len = a.pin_off[pb + p + 1] - b;
        while (len > 0) {  // first event at or after tau
          const uint64_t half = len >> 1;
          if (a.t[b + l + half] < tau) {
            l += half + 1;
            len -= half + 1;
          } else {
            len = half;
          }
        }
        lo[p] = (uint32_t)l;
      }
    }
#pragma unroll
    for (int p = 0; p <= kMaxK; ++p) P.lo[p] = lo[p];
  }
}

template <bool P>
void csr_attr() {
  static bool done = false;
  if (!done) {
    cudaFuncSetAttribute(k_csr<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemB);
    done = true;
  }
}

}  // namespace

uint64_t csr_max_pieces(uint64_t n_events, uint32_t n_gates, uint32_t heavy_thresh) {
  const uint64_t heavy = std::min<uint64_t>(n_gates, n_events / ((uint64_t)heavy_thresh + 1));
  return n_events / kCsrPiece + heavy + 1;
}

bool csr_eligible(uint32_t n_cells, uint32_t tile_target, uint32_t heavy_thresh) {
  return n_cells <= (uint32_t)kSmemCells && tile_target >= 1 && heavy_thresh >= 1 &&
         (uint64_t)tile_target + heavy_thresh <= kCsrMaxTileHeavy;
}

cudaError_t launch_csr_partition(const RunArgs& a, uint32_t n_blocks, uint64_t max_pieces, cudaStream_t st) {
  if (n_blocks == 0) return cudaSuccess;
  k_cp_count<<<n_blocks, 256, 0, st>>>(a);
  cudaError_t e = launch_part_scan(a, n_blocks, st);
  if (e != cudaSuccess) return e;
  k_cp_emit<<<n_blocks, 256, 0, st>>>(a);
  const uint64_t nb = std::max<uint64_t>(1, std::min<uint64_t>((max_pieces + 255) / 256, 152ull * 8));
  k_cp_bounds<<<(unsigned)nb, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_csr(const RunArgs& a, int sm_count, bool pow2, cudaStream_t st) {
  if (pow2) {
    csr_attr<true>();
    k_csr<true><<<sm_count, kCT, kSmemB, st>>>(a);
  } else {
    csr_attr<false>();
    k_csr<false><<<sm_count, kCT, kSmemB, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace pa
