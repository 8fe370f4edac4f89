// Cycle-banded event layout and the banded fused power kernel (sm_103a).
//
// The power step of "GPU-Accelerated Gate-Level Time-Based Power Analysis via
// Event-Density-Aware Partitioning and Kernel Fusion" (Sections 2.4.1-2.4.2,
// Eqs. 1-4, Figs. 2, 3 and 7) adds every event's energy to the waveform bin of
// its clock cycle (Fig. 7's atomicAdd into w). With one global atomic per event
// a billion events are bound by the L2 atomic units. Here the events are first
// regrouped (a load-time layout for one clock period) into units: one gate's
// events inside one window of whole cycles of a band, cut greedily so that no
// pin has more than 7 events in a window (15 in a window of one cycle) -- the
// role of the paper's event-density-aware cycle partitioning, Figs. 5, 19 and
// 20: dense gates get narrow windows, sparse gates one window per band. Units
// are stored band by band, so a CTA keeps the band's cycle bins in shared
// memory and adds them to global memory once per band with a TMA bulk
// reduction. Inside a unit the input events are stored merged in (time, pin)
// order, so the gate state before an event is the unit's start state flipped
// by the pin bits of the unit's earlier events: a warp prefix XOR at run time.
#include <cfloat>
#include <cstdint>

#include "pa_internal.cuh"

namespace pa {

namespace {

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ void berr(unsigned long long* err, uint64_t idx, uint32_t code) {
  atomicMin(err, (unsigned long long)((idx << 8) | code));
}

template <bool kPow2>
__device__ __forceinline__ uint32_t cyc(float t, float T, float inv_T) {
  if (kPow2) return (uint32_t)(t * inv_T);
  return (uint32_t)__fdiv_rn(t, T);
}

__device__ __forceinline__ uint64_t wscan_incl_u64(uint64_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Block (256 threads) exclusive scan of a u64; returns the block total in tot.
__device__ __forceinline__ uint64_t bscan_excl_u64(uint64_t v, uint64_t& tot) {
  __shared__ uint64_t ws[8];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint64_t inc = wscan_incl_u64(v, lane);
  if (lane == 31) ws[w] = inc;
  __syncthreads();
  uint64_t off = 0, t = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (i < w) off += ws[i];
    t += ws[i];
  }
  tot = t;
  __syncthreads();
  return off + inc - v;
}

constexpr int kScanPer = 4;                 // elements per thread
constexpr int kScanBlock = 256 * kScanPer;  // elements per block

// ---- generic u32 -> u64 exclusive scan: block sums, one-block scan, apply
__global__ void __launch_bounds__(256) k_scan_sum(const uint32_t* __restrict__ in, uint64_t n, uint64_t* blk) {
  const uint64_t i0 = (uint64_t)blockIdx.x * kScanBlock + (uint64_t)threadIdx.x * kScanPer;
  uint64_t s = 0;
#pragma unroll
  for (int i = 0; i < kScanPer; ++i)
    if (i0 + i < n) s += in[i0 + i];
  uint64_t tot;
  bscan_excl_u64(s, tot);
  if (threadIdx.x == 0) blk[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(1024) k_scan_blocks(uint64_t* blk, uint32_t nb) {
  __shared__ uint64_t ws[32];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const uint32_t chunk = (nb + 1023) / 1024;
  const uint32_t b0 = min(nb, tid * chunk), b1 = min(nb, b0 + chunk);
  uint64_t loc = 0;
  for (uint32_t b = b0; b < b1; ++b) loc += blk[b];
  const uint64_t inc = wscan_incl_u64(loc, lane);
  if (lane == 31) ws[w] = inc;
  __syncthreads();
  if (w == 0) ws[lane] = wscan_incl_u64(ws[lane], lane);
  __syncthreads();
  uint64_t off = (w ? ws[w - 1] : 0) + inc - loc;
  for (uint32_t b = b0; b < b1; ++b) {
    const uint64_t c = blk[b];
    blk[b] = off;
    off += c;
  }
  if (tid == 1023) blk[nb] = off;
}

__global__ void __launch_bounds__(256) k_scan_apply(const uint32_t* __restrict__ in, uint64_t n,
                                                    const uint64_t* __restrict__ blk, uint64_t* out) {
  const uint64_t i0 = (uint64_t)blockIdx.x * kScanBlock + (uint64_t)threadIdx.x * kScanPer;
  uint32_t v[kScanPer];
  uint64_t s = 0;
#pragma unroll
  for (int i = 0; i < kScanPer; ++i) {
    v[i] = i0 + i < n ? in[i0 + i] : 0u;
    s += v[i];
  }
  uint64_t tot;
  uint64_t off = blk[blockIdx.x] + bscan_excl_u64(s, tot);
#pragma unroll
  for (int i = 0; i < kScanPer; ++i) {
    if (i0 + i < n) out[i0 + i] = off;
    off += v[i];
  }
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) out[n] = blk[gridDim.x];
}

}  // namespace

cudaError_t scan_u32_to_u64(const uint32_t* in, uint64_t n, uint64_t* blk, uint64_t* out, cudaStream_t st) {
  const uint32_t nb = (uint32_t)((n + kScanBlock - 1) / kScanBlock);
  if (nb == 0) return cudaMemsetAsync(out, 0, sizeof(uint64_t), st);
  k_scan_sum<<<nb, 256, 0, st>>>(in, n, blk);
  k_scan_blocks<<<1, 1024, 0, st>>>(blk, nb);
  k_scan_apply<<<nb, 256, 0, st>>>(in, n, blk, out);
  return cudaGetLastError();
}

uint32_t band_scan_blocks(uint64_t n) { return (uint32_t)((n + kScanBlock - 1) / kScanBlock) + 1; }

// ------------------------------------------------------------------ layout build (load time)
//
// One warp per gate walks the gate's cycles in order (a merge of its pins'
// cycle streams; a pin's events are time-sorted, so its cycles are
// non-decreasing) and cuts windows greedily: the current window closes at a
// band boundary, or before a cycle whose events would take one of the pins
// past kUnitPinSoft in the window; a first cycle that alone takes a pin past
// kUnitPinSoft is a window by itself (past kUnitPinMax: the gate is left to
// the unbanded kernel). Counting pass: units and events per
// (band, gate). Writing pass: the same walk writes each unit's record and
// copies its events, pin by pin, to the unit's place in the banded arrays.
// Items: a unit starts an item at a band start, where its event offset enters
// a new bucket of the band (kItemEvents - 1 - the largest unit's events), or
// every kItemUnits units.

namespace {

__device__ __forceinline__ uint32_t bcyc(const BandBuildArgs& a, float t) {
  return a.pow2 ? (uint32_t)(t * a.inv_t_clk) : (uint32_t)__fdiv_rn(t, a.t_clk);
}

constexpr uint32_t kNoCycle = 0xFFFFFFFFu;
// Gates with more events than this are walked by warps, the others by a thread.
constexpr uint64_t kDenseGate = 256;
constexpr int kWalkSegs = 64;  // band segments per dense gate walked in parallel

// Dense gates (more than kDenseGate events) are walked one warp per (gate,
// segment of consecutive bands), up to kWalkSegs segments per gate: windows
// never cross a band boundary, and the input state and output value at a
// segment's start are the parities of each pin's earlier events, so the
// segments of one gate are independent (a Zipf-hot gate's bands no longer
// run one after another). kWrite false: units / events per (band, gate), big
// gates flagged (cleared and listed by k_bw_dense_fix); true:
// records, unit offsets and the event copy. Each pin keeps a chunk of 32
// consecutive events' cycles in the warp's lanes, refilled (one coalesced
// load) before its lookahead of 16 events would leave the chunk. One window
// per step: it starts at the earliest next cycle of the pins and ends at the
// band end or at the cycle of some pin's (kUnitPinSoft + 1)-th event from its
// cursor, whichever is first; each pin's count in the window is one ballot.
// This gives the same windows as walking the gate's cycles one by one.
template <bool kWrite>
__global__ void __launch_bounds__(256) k_bw_walk(const BandBuildArgs a) {
  constexpr int P = kMaxK + 1;
  const int lane = threadIdx.x & 31;
  const uint64_t warp = (blockIdx.x * (uint64_t)blockDim.x + threadIdx.x) >> 5;
  const uint64_t n_warps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
  const uint64_t G = a.n_gates;
  const uint64_t NB = a.n_bands;
  const uint64_t NS = NB < (uint64_t)kWalkSegs ? NB : (uint64_t)kWalkSegs;  // segments per gate
  const uint64_t SB = (NB + NS - 1) / NS;                                       // bands per segment
  const uint64_t n_work = (uint64_t)a.counters[3] * NS;
  for (uint64_t w = warp; w < n_work; w += n_warps) {
    const uint64_t g = a.dense[w / NS];
    const uint64_t b0 = (w % NS) * SB, b1 = b0 + SB < NB ? b0 + SB : NB;
    if (b0 >= b1) continue;
    if (kWrite && a.bigf[g]) continue;
    const GateRec r = a.gates[g];
    const int k = (int)((r.init >> 16) & 0xff);
    const uint64_t gr = a.grank[g];  // the gate's place in the layout's gate order
    const uint32_t c_lo = (uint32_t)(b0 << a.mb);
    const uint64_t se = b1 << a.mb;
    const uint32_t c_seg_end = se > 0xFFFFFFFFull ? 0xFFFFFFFFu : (uint32_t)se;
    // lane p <= k: its pin's events of this segment, [first with cycle >= c_lo, first with cycle >= its end)
    uint64_t my_lo = 0;
    uint32_t my_j = 0, my_hi = 0;
    if (lane <= k) {
      my_lo = a.pin_off[(uint64_t)r.pin_base + lane];
      const uint32_t n = (uint32_t)(a.pin_off[(uint64_t)r.pin_base + lane + 1] - my_lo);
      uint32_t l = 0, m = n;
      while (m > 0) {
        const uint32_t h = m >> 1;
        if (bcyc(a, a.t[my_lo + l + h]) < c_lo) {
          l += h + 1;
          m -= h + 1;
        } else {
          m = h;
        }
      }
      my_j = l;
      m = n - l;
      while (m > 0) {
        const uint32_t h = m >> 1;
        if (bcyc(a, a.t[my_lo + l + h]) < c_seg_end) {
          l += h + 1;
          m -= h + 1;
        } else {
          m = h;
        }
      }
      my_hi = l;
    }
    uint64_t lo[P];
    uint32_t hi[P], j[P], cb[P], cy[P];  // segment end, cursor, chunk base (relative to lo), lane's chunk cycle
    bool any = false;
#pragma unroll
    for (int p = 0; p < P; ++p) {
      lo[p] = __shfl_sync(0xffffffffu, my_lo, p);
      j[p] = __shfl_sync(0xffffffffu, my_j, p);
      hi[p] = __shfl_sync(0xffffffffu, my_hi, p);
      cb[p] = j[p];
      any |= j[p] < hi[p];
      cy[p] = j[p] + (uint32_t)lane < hi[p] ? bcyc(a, a.t[lo[p] + j[p] + lane]) : kNoCycle;
    }
    if (!any) continue;  // no event of this gate in this segment
    uint32_t state = r.init & ((1u << k) - 1u);  // input state at the segment start
#pragma unroll
    for (int p = 0; p < kMaxK; ++p)
      if (p < k) state ^= (j[p] & 1u) << p;
    uint32_t oval = ((r.init >> 8) & 1u) ^ (j[k] & 1u);  // output value at the segment start
    uint32_t band = kNoCycle, units = 0, events = 0, max_unit = 0;
    uint64_t u = 0, dst = 0;  // next unit / banded event of this (band, gate)
    bool big = false, split = false;
    for (;;) {
      uint32_t c_start = kNoCycle;
#pragma unroll
      for (int p = 0; p < P; ++p) {
        const uint32_t c = __shfl_sync(0xffffffffu, cy[p], (int)(j[p] - cb[p]) & 31);
        if (j[p] < hi[p]) c_start = min(c_start, c);
      }
      if (c_start == kNoCycle) break;
      const uint32_t b = c_start >> a.mb;
      if (b != band) {
        if (!kWrite && band != kNoCycle && lane == 0) {
          a.cnt_gb[(uint64_t)band * G + gr] = units;
          a.evc_gb[(uint64_t)band * G + gr] = events;
        }
        band = b;
        units = 0;
        events = 0;
        if (kWrite) {
          u = a.ubase[(uint64_t)b * G + gr];
          dst = a.ebase[(uint64_t)b * G + gr];
        }
      }
      const uint64_t bend = ((uint64_t)b + 1) << a.mb;
      const uint32_t c_band_end = bend > 0xFFFFFFFFull ? 0xFFFFFFFFu : (uint32_t)bend;
      uint32_t c_end = c_band_end, c_hard = c_band_end;
#pragma unroll
      for (int p = 0; p < P; ++p) {
        const uint32_t cs = __shfl_sync(0xffffffffu, cy[p], (int)(j[p] + kUnitPinSoft - cb[p]) & 31);
        if (j[p] + kUnitPinSoft < hi[p]) c_end = min(c_end, cs);
        const uint32_t ch = __shfl_sync(0xffffffffu, cy[p], (int)(j[p] + kUnitPinMax - cb[p]) & 31);
        if (j[p] + kUnitPinMax < hi[p]) c_hard = min(c_hard, ch);
      }
      if (c_end <= c_start) {  // the first cycle alone gives a pin more than kUnitPinSoft events
        if (c_hard <= c_start) {  // more than kUnitPinMax
          big = true;
          break;
        }
        c_end = c_start + 1;
      }
      if (c_end < c_band_end) split = true;
      uint32_t n[P], size = 0;
#pragma unroll
      for (int p = 0; p < P; ++p) {
        const int l0 = (int)(j[p] - cb[p]);
        const bool in = lane >= l0 && lane < l0 + 16 && cy[p] < c_end;
        n[p] = (uint32_t)__popc(__ballot_sync(0xffffffffu, in));
        size += n[p];
      }
      if (!kWrite) max_unit = max(max_unit, size);
      if (kWrite) {
        if (u < (uint64_t)a.L.n_units && dst + size <= a.L.n_ev) {
          if (lane == 0) {
            uint32_t x = 0;
#pragma unroll
            for (int p = 0; p < P; ++p) x |= n[p] << (4 * p);
            x |= state << 20;
            x |= (r.cell & 63u) << 24;
            x |= oval << 30;
            a.urec2[u] = make_uint2(x, __float_as_uint(r.load));
            a.L.ugate[u] = (uint32_t)g;
            a.uband[u] = band;
            a.uoff[u] = dst;
          }
          uint64_t d = dst;
#pragma unroll
          for (int p = 0; p < P; ++p) {
            if ((uint32_t)lane < n[p]) {
              const uint64_t src = lo[p] + j[p] + lane;
              a.L.bt[d + lane] = a.t[src];
              a.L.bs[d + lane] = a.s[src];
            }
            d += n[p];
          }
        } else if (lane == 0) {
          atomicMin(a.err, (unsigned long long)((g << 8) | kErrTileOverflow));
        }
        ++u;
        dst += size;
      }
#pragma unroll
      for (int p = 0; p < P; ++p) {
        if (p < k) state ^= (n[p] & 1u) << p;
        if (p == k) oval ^= n[p] & 1u;
        j[p] += n[p];
        if (j[p] - cb[p] > 16u && j[p] < hi[p]) {  // keep 16 events of lookahead inside the chunk
          cb[p] = j[p];
          cy[p] = j[p] + (uint32_t)lane < hi[p] ? bcyc(a, a.t[lo[p] + j[p] + lane]) : kNoCycle;
        }
      }
      ++units;
      events += size;
    }
    if (!kWrite && lane == 0) {
      if (big) {
        a.bigf[g] = 1;  // k_bw_dense_fix clears the gate's bands and lists it
      } else {
        if (band != kNoCycle) {
          a.cnt_gb[(uint64_t)band * G + gr] = units;
          a.evc_gb[(uint64_t)band * G + gr] = events;
        }
        if (split) a.gflag[g] = 1;
        if (max_unit) atomicMax(a.counters + 2, max_unit);
      }
    }
  }
}

int walk_grid(uint64_t n_gates) {
  return (int)std::min<uint64_t>((n_gates * 32 + 255) / 256 + 1, 152ull * 64);
}

// The dense-gate list (counters[3] entries, any order); their flags cleared.
__global__ void __launch_bounds__(256) k_bw_dense_list(const BandBuildArgs a) {
  const uint64_t g = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= a.n_gates) return;
  const GateRec r = a.gates[g];
  const uint32_t k = (r.init >> 16) & 0xffu;
  if (a.pin_off[(uint64_t)r.pin_base + k + 1] - a.pin_off[r.pin_base] <= kDenseGate) return;
  a.bigf[g] = 0;
  a.gflag[g] = 0;
  a.dense[atomicAdd(a.counters + 3, 1u)] = (uint32_t)g;
}

// After the dense counting walk: a dense gate with a too-dense cycle in any
// band has none of its units kept (its bands cleared) and joins the list of
// gates the unbanded kernel streams; the others with a window narrower than a
// band are counted.
__global__ void __launch_bounds__(256) k_bw_dense_fix(const BandBuildArgs a) {
  const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.counters[3]) return;
  const uint32_t g = a.dense[i];
  if (a.bigf[g]) {
    const uint64_t gr = a.grank[g], G = a.n_gates;
    for (uint32_t bb = 0; bb < a.n_bands; ++bb) {
      a.cnt_gb[(uint64_t)bb * G + gr] = 0;
      a.evc_gb[(uint64_t)bb * G + gr] = 0;
    }
    a.L.big[atomicAdd(a.counters, 1u)] = g;
  } else if (a.gflag[g]) {
    atomicAdd(a.counters + 1, 1u);
  }
}

// The same walk for one sparse gate (at most kDenseGate events) by one thread:
// each window's bounds and per-pin counts read the gate's few events directly
// (they stay in L1 across its windows) instead of a warp's shuffles and
// ballots, which for a handful of events per window idle most of the warp.
// Produces exactly the windows, records and copies of k_bw_walk.

template <bool kWrite>
__global__ void __launch_bounds__(256) k_bw_walk_sparse(const BandBuildArgs a) {
  constexpr int P = kMaxK + 1;
  const uint64_t G = a.n_gates;
  for (uint64_t g = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; g < G; g += (uint64_t)gridDim.x * blockDim.x) {
    const GateRec r = a.gates[g];
    const int k = (int)((r.init >> 16) & 0xff);
    const uint64_t g_lo = a.pin_off[r.pin_base], g_hi = a.pin_off[(uint64_t)r.pin_base + k + 1];
    if (g_hi - g_lo > kDenseGate) continue;  // dense gates: the warp walk
    if (kWrite && a.bigf[g]) continue;
    const uint64_t gr = a.grank[g];
    uint64_t lo[P];
    uint32_t hi[P], j[P];
#pragma unroll
    for (int p = 0; p < P; ++p) {
      lo[p] = 0;
      hi[p] = 0;
      j[p] = 0;
      if (p <= k) {
        lo[p] = a.pin_off[(uint64_t)r.pin_base + p];
        hi[p] = (uint32_t)(a.pin_off[(uint64_t)r.pin_base + p + 1] - lo[p]);
      }
    }
    uint32_t state = r.init & ((1u << k) - 1u);
    uint32_t oval = (r.init >> 8) & 1u;
    uint32_t band = kNoCycle, units = 0, events = 0, max_unit = 0;
    uint64_t u = 0, dst = 0;
    bool big = false, split = false;
    for (;;) {
      uint32_t c_start = kNoCycle;
#pragma unroll
      for (int p = 0; p < P; ++p)
        if (j[p] < hi[p]) c_start = min(c_start, bcyc(a, a.t[lo[p] + j[p]]));
      if (c_start == kNoCycle) break;
      const uint32_t b = c_start >> a.mb;
      if (b != band) {
        if (!kWrite && band != kNoCycle) {
          a.cnt_gb[(uint64_t)band * G + gr] = units;
          a.evc_gb[(uint64_t)band * G + gr] = events;
        }
        band = b;
        units = 0;
        events = 0;
        if (kWrite) {
          u = a.ubase[(uint64_t)b * G + gr];
          dst = a.ebase[(uint64_t)b * G + gr];
        }
      }
      const uint64_t be = ((uint64_t)b + 1) << a.mb;
      const uint32_t c_band_end = be > 0xFFFFFFFFull ? 0xFFFFFFFFu : (uint32_t)be;
      uint32_t c_end = c_band_end, c_hard = c_band_end;
#pragma unroll
      for (int p = 0; p < P; ++p) {
        if (j[p] + kUnitPinSoft < hi[p]) c_end = min(c_end, bcyc(a, a.t[lo[p] + j[p] + kUnitPinSoft]));
        if (j[p] + kUnitPinMax < hi[p]) c_hard = min(c_hard, bcyc(a, a.t[lo[p] + j[p] + kUnitPinMax]));
      }
      if (c_end <= c_start) {
        if (c_hard <= c_start) {
          big = true;
          break;
        }
        c_end = c_start + 1;
      }
      if (c_end < c_band_end) split = true;
      uint32_t n[P], size = 0;
#pragma unroll
      for (int p = 0; p < P; ++p) {
        uint32_t m = j[p];
        while (m < hi[p] && m < j[p] + (uint32_t)kUnitPinMax + 1u && bcyc(a, a.t[lo[p] + m]) < c_end) ++m;
        n[p] = m - j[p];
        size += n[p];
      }
      if (!kWrite) max_unit = max(max_unit, size);
      if (kWrite) {
        if (u < (uint64_t)a.L.n_units && dst + size <= a.L.n_ev) {
          uint32_t x = 0;
#pragma unroll
          for (int p = 0; p < P; ++p) x |= n[p] << (4 * p);
          x |= state << 20;
          x |= (r.cell & 63u) << 24;
          x |= oval << 30;
          a.urec2[u] = make_uint2(x, __float_as_uint(r.load));
          a.L.ugate[u] = (uint32_t)g;
          a.uband[u] = band;
          a.uoff[u] = dst;
          uint64_t d = dst;
#pragma unroll
          for (int p = 0; p < P; ++p) {
            for (uint32_t m = 0; m < n[p]; ++m) {
              const uint64_t src = lo[p] + j[p] + m;
              a.L.bt[d + m] = a.t[src];
              a.L.bs[d + m] = a.s[src];
            }
            d += n[p];
          }
        } else {
          atomicMin(a.err, (unsigned long long)((g << 8) | kErrTileOverflow));
        }
        ++u;
        dst += size;
      }
#pragma unroll
      for (int p = 0; p < P; ++p) {
        if (p < k) state ^= (n[p] & 1u) << p;
        if (p == k) oval ^= n[p] & 1u;
        j[p] += n[p];
      }
      ++units;
      events += size;
    }
    if (!kWrite) {
      if (big) {
        for (uint32_t bb = 0; bb < a.n_bands; ++bb) {
          a.cnt_gb[(uint64_t)bb * G + gr] = 0;
          a.evc_gb[(uint64_t)bb * G + gr] = 0;
        }
        a.L.big[atomicAdd(a.counters, 1u)] = (uint32_t)g;
        a.bigf[g] = 1;
      } else {
        a.bigf[g] = 0;
        if (band != kNoCycle) {
          a.cnt_gb[(uint64_t)band * G + gr] = units;
          a.evc_gb[(uint64_t)band * G + gr] = events;
        }
        if (split) atomicAdd(a.counters + 1, 1u);
        if (max_unit) atomicMax(a.counters + 2, max_unit);
      }
    }
  }
}

int walk_grid_sparse(uint64_t n_gates) {
  return (int)std::min<uint64_t>((n_gates + 255) / 256 + 1, 152ull * 16);
}

// Layout gate order: gates grouped by class (k, and whether the gate has more
// than kDenseGate events), gate order kept inside a class. Units of a band
// follow this order, so the lanes of a warp mostly see cells with the same
// number of inputs and pin segments of similar length.
constexpr int kGateClasses = 2 * (kMaxK + 1);

__device__ __forceinline__ uint32_t gate_class(const BandBuildArgs& a, uint32_t g) {
  const GateRec r = a.gates[g];
  const uint32_t k = (r.init >> 16) & 0xffu;
  const uint64_t n = a.pin_off[(uint64_t)r.pin_base + k + 1] - a.pin_off[r.pin_base];
  return 2u * k + (n > kDenseGate ? 1u : 0u);
}

__global__ void __launch_bounds__(256) k_bw_class_flags(const BandBuildArgs a, uint32_t cls) {
  const uint32_t g = blockIdx.x * 256u + threadIdx.x;
  if (g < a.n_gates) a.flags[g] = gate_class(a, g) == cls ? 1u : 0u;
}

// grank[g] = base + (exclusive scan of the class flags) for the gates of class cls.
__global__ void __launch_bounds__(256) k_bw_class_rank(const BandBuildArgs a, uint32_t cls, const uint64_t* pos,
                                                       const uint64_t* base) {
  const uint32_t g = blockIdx.x * 256u + threadIdx.x;
  if (g < a.n_gates && a.flags[g]) a.grank[g] = (uint32_t)(*base + pos[g]);
}

__global__ void k_bw_class_base(uint64_t* base, const uint64_t* pos, uint32_t n_gates) {
  if (threadIdx.x == 0 && blockIdx.x == 0) *base += pos[n_gates];
}

// Item heads over the units.
__global__ void __launch_bounds__(256) k_bw_item_flags(const BandBuildArgs a, uint32_t n_units) {
  const uint32_t u = blockIdx.x * 256u + threadIdx.x;
  if (u >= n_units) return;
  const uint32_t b = a.uband[u];
  const uint32_t bu0 = (uint32_t)a.ubase[(uint64_t)b * a.n_gates];
  const uint64_t be = a.uoff[bu0];
  bool head = u == bu0;
  if (!head) {
    head = (a.uoff[u] - be) / a.item_bucket != (a.uoff[u - 1] - be) / a.item_bucket ||
           (u - bu0) / (uint32_t)kItemUnits != (u - 1 - bu0) / (uint32_t)kItemUnits;
  }
  a.flags[u] = head ? 1u : 0u;
}

__global__ void __launch_bounds__(256) k_bw_item_emit(const BandBuildArgs a, uint32_t n_units, uint32_t n_items) {
  const uint32_t u = blockIdx.x * 256u + threadIdx.x;
  if (u < n_units && a.flags[u]) {
    BandItem it;
    it.e0 = a.uoff[u];
    it.u0 = u;
    it.bw = a.uband[u];  // the finalize pass adds the input-event count
    a.L.items[a.ipos[u]] = it;
  }
  if (u == 0) {
    BandItem s;
    s.e0 = a.L.n_ev;
    s.u0 = n_units;
    s.bw = a.n_bands;
    a.L.items[n_items] = s;
  }
}

// Finalize pass, one warp per item: the item's events are moved into an
// input region (every unit's input-pin events, unit by unit, each unit's in
// (time, pin) order: the merge of its pins' time-ordered runs) followed by an
// output region (every unit's output-pin events, unit by unit, in time
// order), each event gets its tag word, and each unit its 16-byte record. The
// merge is the order of the layout, fixed once like the regions; the gate
// states along it are left to the run, as is everything that depends on the
// events' arithmetic. The load-axis interval and fraction of the unit's gate
// are fixed here (the library and the netlist do not change while the layout
// lives).
constexpr int kFinWarps = 6;

__global__ void __launch_bounds__(kFinWarps * 32) k_bw_finalize(const BandBuildArgs a) {
  __shared__ float tb[kFinWarps][kItemEvents];
  __shared__ float sb[kFinWarps][kItemEvents];
  __shared__ uint16_t gb[kFinWarps][kItemEvents];  // tag words, in region order
  __shared__ uint16_t dd[kFinWarps][kItemEvents];  // region index of each event, in the walk's order
  __shared__ uint32_t ust[kFinWarps][kItemUnits];  // unit starts in the walk's order, item-relative
  __shared__ uint32_t udst[kFinWarps][kItemUnits]; // input offset | output offset (in the region) << 9 | inputs << 18
  __shared__ uint32_t ups[kFinWarps][kItemUnits];  // ends of input pins 0..3 in the walk's order, one byte each
  __shared__ uint32_t upin[kFinWarps][kItemUnits]; // record word y
  __shared__ uint32_t utie[kFinWarps][kItemUnits / 32];  // units with events at one time on two input pins
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint64_t n_warps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
  const BandLayout& L = a.L;
  for (uint64_t it = warp; it < L.n_items; it += n_warps) {
    const uint64_t e0 = L.items[it].e0, e1 = L.items[it + 1].e0;
    const uint32_t u0 = L.items[it].u0, u1 = L.items[it + 1].u0;
    if (e1 <= e0 || e1 - e0 >= (uint64_t)kItemEvents || u1 <= u0 || u1 - u0 > (uint32_t)kItemUnits) {
      if (lane == 0) atomicMin(a.err, (unsigned long long)((it << 8) | kErrLayout));
      continue;
    }
    const int n = (int)(e1 - e0), nu = (int)(u1 - u0);
    // units: sizes, the two regions' offsets, pin runs
    uint32_t carry = 0;
    for (int r = 0; r < 2; ++r) {
      const int uu = lane + 32 * r;
      uint32_t pk = 0, n_in = 0, x = 0, ends = 0;
      if (uu < nu) {
        x = a.urec2[u0 + uu].x;
        const uint32_t k = a.cells[(x >> 24) & 63u].k;
        uint32_t s = 0;
#pragma unroll
        for (int p = 0; p < kMaxK; ++p) {
          if ((uint32_t)p < k) s += (x >> (4 * p)) & 15u;
          ends |= s << (8 * p);
        }
        n_in = s;
        const uint32_t n_out = (x >> (4 * k)) & 15u;
        pk = (n_in + n_out) | (n_in << 10) | (n_out << 20);
        // record word y: the unit's input events | output value at the window start << 6 | (k - 1) << 30
        upin[wl][uu] = n_in | (((x >> 30) & 1u) << 6) | ((k - 1u) << 30);
        ups[wl][uu] = ends;
      }
      uint32_t inc = pk;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      const uint32_t ex = carry + inc - pk;
      carry += __shfl_sync(0xffffffffu, inc, 31);
      if (uu < nu) {
        ust[wl][uu] = ex & 1023u;
        udst[wl][uu] = ((ex >> 10) & 1023u) | (((ex >> 20) & 1023u) << 9) | (n_in << 18);
      }
    }
    __syncwarp();
    const uint32_t n_in_all = (carry >> 10) & 1023u;
    if ((carry & 1023u) != (uint32_t)n || n_in_all + ((carry >> 20) & 1023u) != (uint32_t)n) {
      if (lane == 0) atomicMin(a.err, (unsigned long long)((it << 8) | kErrLayout));
      continue;
    }
    for (int i = lane; i < n; i += 32) sb[wl][i] = L.bt[e0 + i];  // times in the walk's order
    __syncwarp();
    // each event's place: an input event at its rank in its unit's (time,
    // pin) order -- its index in its pin's run plus, for every other input
    // pin, the events earlier than it (at an equal time: on a lower pin)
    for (int i = lane; i < n; i += 32) {
      int u = 0;
#pragma unroll
      for (int h = kItemUnits / 2; h > 0; h >>= 1)
        if (u + h < nu && ust[wl][u + h] <= (uint32_t)i) u += h;
      const int ub = (int)ust[wl][u], li = i - ub;
      const uint32_t d = udst[wl][u], ends = ups[wl][u];
      const int n_in = (int)(d >> 18);
      const int k = (int)(upin[wl][u] >> 30) + 1;
      int dst;
      uint32_t tag = (uint32_t)u;
      if (li < n_in) {
        int p = 0;
        while (p < k - 1 && li >= (int)((ends >> (8 * p)) & 255u)) ++p;
        const int ps = p == 0 ? 0 : (int)((ends >> (8 * (p - 1))) & 255u);
        const float t = sb[wl][i];
        int rank = li - ps;
        for (int q = 0; q < k; ++q) {
          if (q == p) continue;
          const int qa = q == 0 ? 0 : (int)((ends >> (8 * (q - 1))) & 255u);
          const int qb = (int)((ends >> (8 * q)) & 255u);
          for (int m = ub + qa; m < ub + qb; ++m) {
            const float tq = sb[wl][m];
            rank += (tq < t || (tq == t && q < p)) ? 1 : 0;
          }
        }
        dst = (int)(d & 511u) + rank;
        tag |= (uint32_t)p << 6;
      } else {
        dst = (int)n_in_all + (int)((d >> 9) & 511u) + (li - n_in);
        if (li > n_in) tag |= 1u << 8;  // the output's previous event is the one just before
      }
      dd[wl][i] = (uint16_t)dst;
      gb[wl][dst] = (uint16_t)tag;
      tb[wl][dst] = sb[wl][i];
    }
    __syncwarp();
    // distance back to the pin's previous event in the unit (input events; 0
    // for a unit's first event of a pin): in the walk's order that event is
    // the one just before, when it lies in the same pin run
    for (int i = lane; i < n; i += 32) {
      const int dst = dd[wl][i];
      if (dst < (int)n_in_all) {
        int u = 0;
#pragma unroll
        for (int h = kItemUnits / 2; h > 0; h >>= 1)
          if (u + h < nu && ust[wl][u + h] <= (uint32_t)i) u += h;
        const int li = i - (int)ust[wl][u];
        const uint32_t ends = ups[wl][u];
        const int p = (int)((gb[wl][dst] >> 6) & 3u);
        const int ps = p == 0 ? 0 : (int)((ends >> (8 * (p - 1))) & 255u);
        if (li > ps) gb[wl][dst] |= (uint16_t)((dst - (int)dd[wl][i - 1]) << 8);
      }
    }
    if (lane < kItemUnits / 32) utie[wl][lane] = 0u;
    __syncwarp();
    // ties: in (time, pin) order two input events of a unit at one time are neighbours
    for (int i = lane + 1; i < (int)n_in_all; i += 32) {
      const uint32_t u = gb[wl][i] & 63u;
      if ((gb[wl][i - 1] & 63u) == u && tb[wl][i - 1] == tb[wl][i]) atomicOr(&utie[wl][u >> 5], 1u << (u & 31u));
    }
    __syncwarp();
    for (int i = lane; i < n; i += 32) sb[wl][dd[wl][i]] = L.bs[e0 + i];  // the walk-order times are no longer read
    for (int r = 0; r < 2; ++r) {
      const int uu = lane + 32 * r;
      if (uu < nu) {
        const uint2 w = a.urec2[u0 + uu];
        const uint32_t cell = (w.x >> 24) & 63u;
        const CellDesc& cd = a.cells[cell];
        const float C = __uint_as_float(w.y);
        int j = 0;
        for (int m = 1; m <= (int)cd.nl - 2; ++m) j += (C >= cd.lax[m]) ? 1 : 0;
        const float v = (C - cd.lax[j]) * cd.ilax[j];
        const uint32_t d = udst[wl][uu];
        const uint32_t x = (d & 511u) | ((n_in_all + ((d >> 9) & 511u)) << 9) | (cell << 18) |
                           (((w.x >> 20) & 15u) << 24) | ((uint32_t)j << 28) |
                           (((utie[wl][uu >> 5] >> (uu & 31)) & 1u) << 31);
        L.urec[u0 + uu] = make_uint4(x, __float_as_uint(v), w.y, upin[wl][uu]);
      }
    }
    __syncwarp();
    for (int i = lane; i < n; i += 32) {
      L.bt[e0 + i] = tb[wl][i];
      L.bs[e0 + i] = sb[wl][i];
      L.btag[e0 + i] = gb[wl][i];
    }
    // events sharing the cycle of the event stored before them (same region)
    uint32_t cont = 0;
    for (int i = lane + 1; i < n; i += 32)
      cont += (i != (int)n_in_all && bcyc(a, tb[wl][i]) == bcyc(a, tb[wl][i - 1])) ? 1u : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cont += __shfl_xor_sync(0xffffffffu, cont, o);
    if (lane == 0)
      L.items[it].bw = (L.items[it].bw & kItemBandMask) | (n_in_all << kItemBandBits) |
                       (3u * cont >= 2u * (uint32_t)n ? kItemRunsBit : 0u);
    __syncwarp();
  }
}

}  // namespace

cudaError_t band_build_count(BandBuildArgs& a, cudaStream_t st) {
  const uint64_t n = (uint64_t)a.n_bands * a.n_gates;
  // gate order: one stable pass per class (flags, scan, ranks after the earlier classes)
  cudaError_t e = cudaMemsetAsync(a.ipos + a.n_gates + 1, 0, sizeof(uint64_t), st);  // running class base
  if (e != cudaSuccess) return e;
  const uint32_t gb = (a.n_gates + 255) / 256;
  for (uint32_t cls = 0; cls < (uint32_t)kGateClasses && a.n_gates; ++cls) {
    k_bw_class_flags<<<gb, 256, 0, st>>>(a, cls);
    e = scan_u32_to_u64(a.flags, a.n_gates, a.scan_blk, a.ipos, st);
    if (e != cudaSuccess) return e;
    k_bw_class_rank<<<gb, 256, 0, st>>>(a, cls, a.ipos, a.ipos + a.n_gates + 1);
    k_bw_class_base<<<1, 32, 0, st>>>(a.ipos + a.n_gates + 1, a.ipos, a.n_gates);
  }
  e = cudaMemsetAsync(a.counters, 0, 4 * sizeof(uint32_t), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(a.cnt_gb, 0, (n + 1) * sizeof(uint32_t), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(a.evc_gb, 0, (n + 1) * sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  if (a.n_gates) {
    k_bw_dense_list<<<(a.n_gates + 255) / 256, 256, 0, st>>>(a);
    k_bw_walk_sparse<false><<<walk_grid_sparse(a.n_gates), 256, 0, st>>>(a);
    k_bw_walk<false><<<walk_grid(a.n_gates), 256, 0, st>>>(a);
    k_bw_dense_fix<<<(a.n_gates + 255) / 256, 256, 0, st>>>(a);
  }
  e = scan_u32_to_u64(a.cnt_gb, n, a.scan_blk, a.ubase, st);
  if (e == cudaSuccess) e = scan_u32_to_u64(a.evc_gb, n, a.scan_blk, a.ebase, st);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t band_build_write(BandBuildArgs& a, cudaStream_t st) {
  if (a.n_gates) {
    k_bw_walk_sparse<true><<<walk_grid_sparse(a.n_gates), 256, 0, st>>>(a);
    k_bw_walk<true><<<walk_grid(a.n_gates), 256, 0, st>>>(a);
  }
  const uint32_t nu = a.L.n_units;
  cudaError_t e = cudaMemcpyAsync(a.uoff + nu, &a.L.n_ev, sizeof(uint64_t), cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return e;
  if (nu) k_bw_item_flags<<<(nu + 255) / 256, 256, 0, st>>>(a, nu);
  e = scan_u32_to_u64(a.flags, nu, a.scan_blk, a.ipos, st);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t band_build_items(BandBuildArgs& a, cudaStream_t st) {
  const uint32_t nu = a.L.n_units;
  k_bw_item_emit<<<nu ? (nu + 255) / 256 : 1, 256, 0, st>>>(a, nu, a.L.n_items);
  if (a.L.n_items) {
    const uint64_t blocks = ((uint64_t)a.L.n_items + kFinWarps - 1) / kFinWarps;
    k_bw_finalize<<<(int)std::min<uint64_t>(blocks, 152ull * 16), kFinWarps * 32, 0, st>>>(a);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------ P0 of a run

namespace {

__global__ void __launch_bounds__(256) k_band_p0(const RunArgs a) {
  const uint32_t g = blockIdx.x * 256u + threadIdx.x;
  double p0 = 0.0;
  if (g < a.n_gates) {
    const GateRec r = a.gates[g];
    const CellDesc& cd = a.cells[r.cell];
    p0 = (double)a.leak[cd.leak_off + (r.init & ((1u << cd.k) - 1u))];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) p0 += __shfl_xor_sync(0xffffffffu, p0, o);
  __shared__ double ws[8];
  if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = p0;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int i = 0; i < 8; ++i) s += ws[i];
    if (s != 0.0) atomicAdd(a.p0, s);
  }
}

}  // namespace

cudaError_t band_p0(const RunArgs& r, cudaStream_t st) {
  if (r.n_gates) k_band_p0<<<(r.n_gates + 255) / 256, 256, 0, st>>>(r);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ banded fused kernel
//
// One CTA of 32 warps per SM takes chunks of items from a global counter and
// works through each chunk band by band. Inside a band the warps take items
// from a shared counter and work independently: lane 0 starts the TMA bulk
// copies of the item's times, event tags and unit records into the warp's
// stage (completing on the warp's mbarrier), with the record of the warp's
// next item loaded ahead. Then one lane per event: first the item's input
// region (gate state from the unit's start state and the parities of the
// other input pins' earlier events, LUT energy from one corner-patch load,
// glitch and leakage step), then its output region (switching energy); the
// sums go into the band's cycle bins in shared memory. When the band's items
// are done the CTA adds the bins to global memory with one TMA bulk reduction.

namespace {

constexpr int kBW = 32;
constexpr int kBT = kBW * 32;
constexpr int kStEv = kItemEvents + 8;                     // staged times (16-byte rounding)
constexpr size_t kStTagOff = (size_t)kStEv * 4;            // staged event tag words
constexpr size_t kStRecOff = kStTagOff + (size_t)kStEv * 2; // staged unit records
constexpr size_t kWarpB = kStRecOff + (size_t)kItemUnits * 16;
constexpr size_t kHist = (size_t)kBandMaxCycles * 16;
// Cell table in shared memory: per cell the slew axis points 0..8 at a
// stride of 9 words (an odd stride, so that lanes of different cells spread
// over the banks; points 1..8 past ns - 2 read +inf), then one info word per
// cell (ns - 1 | (nl - 1) << 8 | patch offset << 16; a library of at most 64
// cells with axes of at most 8 points has fewer than 2^16 corner patches),
// then per cell and slew interval i the pair {axis point i, 1 / interval
// width} (one 8-byte load per event), then per cell its leakage per state
// (uW, at a stride of 17 words: the step of an event is the difference of
// two of them, the same f32 subtraction as the unbanded kernel's).
constexpr int kAxStride = 9;
constexpr int kLeakStride = 17;
constexpr size_t kCellsB = (size_t)kSmemCells * kAxStride * 4 + (size_t)kSmemCells * 4 + (size_t)kSmemCells * 8 * 8 +
                           (size_t)kSmemCells * kLeakStride * 4;
// Item records of the CTA's current and next chunk (the next one's copy in
// flight while the current one is worked on), one more for the end.
constexpr uint32_t kChunkMaxItems = 680;
constexpr size_t kChunkRecB = (size_t)(kChunkMaxItems + 1) * sizeof(BandItem);
constexpr size_t kSmemB = kHist + kCellsB + kBW * kWarpB + 2 * kChunkRecB;
static_assert(kStTagOff % 16 == 0 && kStRecOff % 16 == 0 && kWarpB % 16 == 0 && kHist % 16 == 0 &&
                  kCellsB % 16 == 0 && kChunkRecB % 16 == 0,
              "alignment");
static_assert(kBW * kWarpB >= kHist, "a band's rows fit the warp buffers");
static_assert(kSmemB + 1024 <= 227 * 1024, "shared memory budget");
constexpr int kTotEvery = 16;              // items between flushes of a warp's per-lane totals
// Items a CTA takes from the global counter at a time: about 16 chunks per
// CTA, within [kChunkMin, kChunkMax] (big chunks mean fewer CTA-wide syncs,
// small ones a shorter tail; item costs vary with the gate class, so chunks
// that shrink over the run would leave the early, big ones unbalanced).
constexpr uint32_t kChunkMin = 64, kChunkMax = kChunkMaxItems;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_arrive(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// One bounded wait on the barrier's phase: the thread may be suspended for up
// to about 0.1 ms (the suspend-time hint) before it reports "not yet".
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(100000u)
      : "memory");
  return ok != 0;
}

// Bulk copy global -> shared, completing on the mbarrier (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bulk f32 add of shared memory into global memory (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_red_add_f32(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// A lane's running sums of its events' totals. The leakage term dP (t_max -
// t) of an event is large (t_max - t up to the whole window) and of either
// sign, and the terms of a gate's rising and falling steps almost cancel, so
// its f32 sum is compensated (Kahan: c_lk holds the low-order part lost so
// far) and the warp sums are taken in fp64.
struct BAcc {
  float e_int, e_sw, e_gl, e_lk, c_lk;
};

__device__ __forceinline__ void kahan_add(float& sum, float& comp, float x) {
  const float y = x - comp;
  const float t = sum + y;
  comp = (t - sum) - y;
  sum = t;
}

__device__ __forceinline__ void bflush_acc(BAcc& acc, double* s_tot) {
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
  acc = BAcc{0.f, 0.f, 0.f, 0.f, 0.f};
}

// The band's bins in shared memory: four arrays of kBandMaxCycles words,
// W and D (f32) then ev and gl (u32), so one field of 32 different cycles falls
// in 32 different banks.
constexpr uint32_t kHW = 0, kHD = kBandMaxCycles, kHE = 2 * kBandMaxCycles, kHG = 3 * kBandMaxCycles;

// Add the band's shared-memory bins to the global bins and clear them. Fast
// mode: the rows {W, D, ev, gl} (counts as f32) are written to `rows` (free
// shared memory while no warp holds an item), then one bulk reduction. Exact
// mode adds per event to global memory; nothing to flush.
template <bool kExact>
__device__ void bflush_band(const BandRunArgs& A, float* hist, float4* rows, uint32_t band) {
  const uint32_t cb = A.L.band_cycles, N = A.r.n_cycles;
  const uint32_t c0 = band * cb;
  const uint32_t nb = c0 < N ? min(cb, N - c0) : 0u;
  const uint32_t* hu = reinterpret_cast<const uint32_t*>(hist);
  if (!kExact) {
    for (uint32_t i = threadIdx.x; i < nb; i += kBT)
      rows[i] = make_float4(hist[kHW + i], hist[kHD + i], (float)hu[kHE + i], (float)hu[kHG + i]);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (threadIdx.x == 0 && nb) bulk_red_add_f32(A.r.bins + c0, rows, nb * 16u);
    __syncthreads();
  }
  for (uint32_t i = threadIdx.x; i < 4 * cb; i += kBT) {
    const uint32_t f = i / cb, c = i - f * cb;
    hist[f * kBandMaxCycles + c] = 0.f;
  }
}

__device__ __forceinline__ uint32_t item_band(const BandItem& it) { return it.bw & kItemBandMask; }

// Thread 0 of a CTA: the next chunk [x, y) of items, y == x when none is left.
// The last twentieth of the items goes out in quarter-size chunks from a
// second counter (ctr[1]), so the CTAs finish closer together; big chunks for
// the rest keep the band flushes few.
__device__ __forceinline__ uint2 take_chunk(uint32_t* ctr, uint32_t n, uint32_t chunk) {
  const uint32_t n_main = n - n / 20;
  const uint32_t x = atomicAdd(ctr, chunk);
  if (x < n_main) return make_uint2(x, x + min(chunk, n_main - x));
  const uint32_t small = max(kChunkMin / 2, chunk / 4);
  const uint32_t y = n_main + atomicAdd(ctr + 1, small);
  return y >= n ? make_uint2(n, n) : make_uint2(y, y + min(small, n - y));
}

// First item in [lo, hi) whose band differs from `band` (items are band-sorted;
// it[] holds the records of the chunk from item lo on).
__device__ uint32_t band_end(const BandItem* it, uint32_t lo, uint32_t hi, uint32_t band) {
  const uint32_t base = lo;
  uint32_t n = hi - lo;
  while (n > 0) {
    const uint32_t half = n >> 1;
    if ((it[lo + half - base].bw & kItemBandMask) <= band) {
      lo += half + 1;
      n -= half + 1;
    } else {
      n = half;
    }
  }
  return lo;
}

// Staging geometry of an item: events [e0, e0 + n) (the first n_in of them
// input-pin events) and units [u0, u0 + nu), rounded out to 16-byte copies.
// ok is false for an item that cannot be staged (never for a consistent
// layout).
struct ItemGeo {
  uint64_t e0, ea;
  uint32_t u0, n, nu, n_in, ev_off, tag_off, ev_bytes, tag_bytes;
  bool runs;  // the item's events come in runs of one cycle (merge their bin updates)
  bool ok;
};

__device__ __forceinline__ ItemGeo item_geo(const BandItem& a, const BandItem& b) {
  ItemGeo g;
  g.e0 = a.e0;
  g.u0 = a.u0;
  g.ea = a.e0 & ~3ull;
  g.ev_off = (uint32_t)(a.e0 - g.ea);
  g.tag_off = (uint32_t)(a.e0 & 7ull);  // tag words: 16-byte copies of 8
  g.n_in = (a.bw >> kItemBandBits) & 511u;  // bits 20..28
  g.runs = (a.bw & kItemRunsBit) != 0u;
  g.ok = b.e0 > a.e0 && b.u0 > a.u0 && b.e0 - a.e0 < (uint64_t)kItemEvents && b.u0 - a.u0 <= (uint32_t)kItemUnits &&
         (uint64_t)g.n_in <= b.e0 - a.e0;
  g.n = g.ok ? (uint32_t)(b.e0 - a.e0) : 0u;
  g.nu = g.ok ? b.u0 - a.u0 : 0u;
  g.ev_bytes = ((g.ev_off + g.n + 3u) & ~3u) * 4u;
  g.tag_bytes = ((g.tag_off + g.n + 7u) & ~7u) * 2u;
  return g;
}

// Lane 0: start the copies of an item into a stage (an empty arrival for an
// item that cannot be staged, so the wait still completes).
__device__ __forceinline__ void stage_item(const BandLayout& L, const ItemGeo& g, uint8_t* stage, uint64_t* bar) {
  if (!g.ok) {
    mbar_expect_arrive(bar, 0);
    return;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_arrive(bar, g.ev_bytes + g.tag_bytes + g.nu * 16u);
  bulk_g2s(stage, L.bt + g.ea, g.ev_bytes, bar);
  bulk_g2s(stage + kStTagOff, L.btag + (g.e0 - g.tag_off), g.tag_bytes, bar);
  bulk_g2s(stage + kStRecOff, L.urec + g.u0, g.nu * 16u, bar);
}

// Lane 0: bring an item that this warp will stage next into L2 (its times,
// tags, unit records and slews), so that its stage copy does not wait on HBM.
__device__ __forceinline__ void prefetch_item(const BandLayout& L, const ItemGeo& g) {
  if (!g.ok) return;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(L.bt + g.ea), "r"(g.ev_bytes) : "memory");
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(L.bs + g.ea), "r"(g.ev_bytes) : "memory");
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(L.btag + (g.e0 - g.tag_off)), "r"(g.tag_bytes)
               : "memory");
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(L.urec + g.u0), "r"(g.nu * 16u) : "memory");
}

// Gate states of one round of 32 input events (lane l: staged index base +
// l). A unit's input events are contiguous and in (time, pin) order, so the
// input values just before an event in that order are the unit's start state
// flipped by the pin bits x of the unit's earlier events: a prefix XOR over
// the round, restarted at the unit's first event (lane in_off - base), plus
// `carry`, the XOR of the round's first unit's bits in earlier rounds
// (warp-uniform, advanced to the next round here). Lanes past the item's
// input events pass x = 0 and come after every valid lane.
__device__ __forceinline__ uint32_t round_state(uint32_t x, int in_off, int base, uint32_t start, uint32_t& carry,
                                                int lane) {
  uint32_t v = x;  // inclusive prefix XOR over the round
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v ^= y;
  }
  const uint32_t ex = v ^ x;
  const int ss = in_off > base ? in_off - base : 0;  // the unit's first lane in this round
  const uint32_t ex_ss = __shfl_sync(0xffffffffu, ex, ss);
  const uint32_t before = ex_ss ^ (in_off < base ? carry : 0u);  // bits of the unit's events before lane ss
  carry = __shfl_sync(0xffffffffu, v ^ before, 31);
  return start ^ ex ^ before;
}

// The same for two rounds at once (staged indices base + l and base + 32 +
// l): their pin bits travel through one scan in one word (the first round's
// in bits 0..3, the second's in bits 8..11).
__device__ __forceinline__ void pair_state(uint32_t xa, int offa, uint32_t sta, uint32_t xb, int offb, uint32_t stb,
                                           int base, uint32_t& carry, int lane, uint32_t& sa, uint32_t& sb) {
  const uint32_t x = xa | (xb << 8);
  uint32_t v = x;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v ^= y;
  }
  const uint32_t ex = v ^ x;
  const int ssa = offa > base ? offa - base : 0;
  const int ssb = offb > base + 32 ? offb - base - 32 : 0;
  const uint32_t befa = (__shfl_sync(0xffffffffu, ex, ssa) & 15u) ^ (offa < base ? carry : 0u);
  sa = sta ^ (ex & 15u) ^ befa;
  const uint32_t ca = __shfl_sync(0xffffffffu, (v & 15u) ^ befa, 31);  // into the second round
  const uint32_t befb = ((__shfl_sync(0xffffffffu, ex, ssb) >> 8) & 15u) ^ (offb < base + 32 ? ca : 0u);
  sb = stb ^ ((ex >> 8) & 15u) ^ befb;
  carry = __shfl_sync(0xffffffffu, ((v >> 8) & 15u) ^ befb, 31);
}

struct CellTab {
  const float* sax;       // [kSmemCells * kAxStride] slew axes, +inf past ns - 2
  const uint32_t* info;   // [kSmemCells] ns - 1 | (nl - 1) << 8 | patch offset << 16
  const float2* sxp;      // [kSmemCells * 8] {slew axis point i, 1 / (ax[i + 1] - ax[i])}
  const float* leak;      // [kSmemCells * kLeakStride] leakage per state, uW
};

// One event's result before any shared or global memory is written: its
// cycle, the energy for the cycle's bin, the leakage step and its kind. The
// per-event work is split in compute (loads and arithmetic only, so that the
// compiler may interleave two events of a lane) and commit (the bins).
struct EvOut {
  uint32_t c;
  float e_w, dp;
  uint32_t flags;  // 1: input-pin event (carries a leakage step), 2: glitch
};

// Debug values of an event (only with kDebug): what the per-event outputs
// need, and the event's share of its gate's energies.
struct EvDbg {
  uint32_t s_pre, lut_ij, unit;
  int p;
  float t;
  bool glitch;
  float g_int, g_sw, g_gl, g_lk;  // fJ
};

// Glitch test against the pin's previous event (staged index ep, if has_prev)
// and scaling of the dynamic energy; the one branch is the division of a
// narrow glitch pulse (predicated lanes). en: the pin's next event in the unit (staged
// index, -1 if none; only asked for in the glitch-all reading, where the
// first event of a multi-event pin-cycle takes the pulse to that next event).
template <bool kPow2, bool kDebug>
__device__ __forceinline__ float glitch_scale(const RunArgs& a, const float* ts, const float* gs, int ep,
                                              bool has_prev, int en, float t, float s, uint32_t c, float e_dyn,
                                              bool& glitch) {
  float tp = ts[ep];
  glitch = has_prev && cyc<kPow2>(tp, a.t_clk, a.inv_t_clk) == c;
  // the previous edge's slew only for glitches (a predicated load: only those lanes touch L1)
  float sp = s;
  if (glitch) sp = __ldg(gs + ep);
  float pw = t - tp;
  if (kDebug && a.glitch_all && !glitch && en >= 0) {  // the reading runs in the per-event path
    const float tn = ts[en];
    if (cyc<kPow2>(tn, a.t_clk, a.inv_t_clk) == c) {
      glitch = true;
      pw = tn - t;
      sp = __ldg(gs + en);
    }
  }
  // r_gl = min(1, x / y) with IEEE division, as in the unbanded kernel, so
  // both kernels give one event the same value; x >= y gives 1 (the rounded
  // quotient of x >= y is >= 1), so only glitch lanes with a narrow pulse divide
  const float x = 2000.f * pw, y = s + sp;
  float r = 1.f;
  if (glitch && x < y) r = __fdiv_rn(x, y);
  return glitch ? r * e_dyn : e_dyn;
}

// Input-pin event at staged index i (tag word w, unit record R): its state
// s_b (input values just before it in (time, pin) order, from round_state),
// LUT energy, leakage step, glitch, totals. `valid` false: computed for a
// padding lane, not counted.
template <bool kPow2, bool kDebug>
__device__ __forceinline__ EvOut ev_input(const RunArgs& a, const CellTab& CT, const float* ts, const uint16_t* tg,
                                          const uint4* rec, const float* gs, int i, uint32_t w, const uint2& R,
                                          uint32_t s_b, bool valid, BAcc& acc, EvDbg& dbg) {
  const float t = ts[i];
  const float s = __ldg(gs + i);
  const int p = (int)((w >> 6) & 3u);
  const int d = (int)(w >> 8);  // back to the pin's previous event in the unit (0: none)
  // the LUT's state is the state before the whole timestamp: at a time two
  // input pins share (flagged units only), the lower pins' events at t, just
  // before this one in (time, pin) order, are taken back out
  uint32_t s_pre = s_b;
  if ((R.x >> 31) != 0u) {
    const int in_off = (int)(R.x & 511u);
    for (int j = i - 1; j >= in_off && ts[j] == t; --j) s_pre ^= 1u << ((tg[j] >> 6) & 3u);
  }
  const uint32_t cell = (R.x >> 18) & 63u;
  const uint32_t info = CT.info[cell];  // ns - 1 | (nl - 1) << 8 | patch offset << 16
  // slew interval: the number of axis points 1 .. ns - 2 that are <= s, by a
  // three-step binary search over points 1..7 (sorted, +inf past ns - 2)
  const float* axs = CT.sax + cell * kAxStride;
  int lis = s >= axs[4] ? 4 : 0;
  lis += s >= axs[lis + 2] ? 2 : 0;
  lis += s >= axs[lis + 1] ? 1 : 0;
  const float2 ax = CT.sxp[cell * 8 + lis];
  const float uu2 = (s - ax.x) * ax.y;
  const int j = (int)((R.x >> 28) & 7u);
  // corners {L[i][j], L[i][j+1], L[i+1][j], L[i+1][j+1]} of the state's table
  const float4 P =
      __ldg(a.patch + (info >> 16) + ((int)s_pre * (int)(info & 0xFFu) + lis) * (int)((info >> 8) & 0xFFu) + j);
  const float vv = __uint_as_float(R.y);
  const float r0 = fmaf(vv, P.y - P.x, P.x), r1 = fmaf(vv, P.w - P.z, P.z);
  const float e_int = fmaf(uu2, r1 - r0, r0);
  const float* lk = CT.leak + cell * kLeakStride;
  const float dp = lk[s_b ^ (1u << p)] - lk[s_b];
  const float T = a.t_clk;
  const uint32_t c = cyc<kPow2>(t, T, a.inv_t_clk);
  int en = -1;
  if (kDebug && a.glitch_all) {  // the pin's next event in the unit
    const int end = (int)(R.x & 511u) + (int)(rec[w & 63u].w & 63u);
    for (int m = i + 1; m < end; ++m)
      if ((int)((tg[m] >> 6) & 3u) == p) {
        en = m;
        break;
      }
  }
  bool glitch;
  float e_w = glitch_scale<kPow2, kDebug>(a, ts, gs, i - d, d > 0, en, t, s, c, e_int, glitch);
  if (valid) {
    acc.e_gl += glitch ? e_w : 0.f;
    acc.e_int += glitch ? 0.f : e_int;
    kahan_add(acc.e_lk, acc.c_lk, dp * (a.t_max_f - t));
  }
  if (kDebug)
    dbg = EvDbg{s_pre, (uint32_t)((lis << 4) | j), w & 63u, p, t, glitch, glitch ? 0.f : e_int, 0.f,
                glitch ? e_w : 0.f, dp * (a.t_max_f - t)};
  const float rem = fmaf(-(float)c, T, t);  // t - c T: the step's part inside its own cycle
  e_w = fmaf(dp, T - rem, e_w);
  return EvOut{c, e_w, dp, 1u | (glitch ? 2u : 0u)};
}

// Output-pin event at staged index i: switching energy, glitch, totals.
template <bool kPow2, bool kDebug>
__device__ __forceinline__ EvOut ev_output(const RunArgs& a, const float* ts, const uint16_t* tg, const uint4* rec,
                                           const float* gs, int i, int n, bool valid, BAcc& acc, EvDbg& dbg) {
  const uint32_t w = tg[i];
  const float t = ts[i];
  const bool has_prev = (w >> 8) != 0u;  // the unit's previous output event is the one just before
  // the slew only enters a glitch ratio: loaded for lanes whose previous event
  // is on the pin (or, in the glitch-all reading, for every lane)
  float s = 0.f;
  if (has_prev || (kDebug && a.glitch_all)) s = __ldg(gs + i);
  float e_sw = a.half_vdd2 * __uint_as_float(reinterpret_cast<const uint32_t*>(rec)[(w & 63u) * 4u + 2u]);
  uint4 R = make_uint4(0u, 0u, 0u, 0u);
  if (kDebug) R = rec[w & 63u];
  if (kDebug && a.esw_rise) {  // C V^2 on a rise: the output's value at the window start, flipped per earlier event
    const int idx = i - (int)((R.x >> 9) & 511u);
    e_sw = ((((R.w >> 6) & 1u) ^ ((uint32_t)(idx + 1) & 1u)) != 0u) ? 2.f * e_sw : 0.f;
  }
  const uint32_t c = cyc<kPow2>(t, a.t_clk, a.inv_t_clk);
  const int en = (kDebug && a.glitch_all && i + 1 < n && (tg[i + 1] & 63u) == (w & 63u)) ? i + 1 : -1;
  bool glitch;
  const float e_w = glitch_scale<kPow2, kDebug>(a, ts, gs, has_prev ? i - 1 : i, has_prev, en, t, s, c, e_sw, glitch);
  if (valid) {
    acc.e_gl += glitch ? e_w : 0.f;
    acc.e_sw += glitch ? 0.f : e_sw;
  }
  if (kDebug) {
    // input values before t: the unit's start state flipped by its input
    // events earlier than t (in time order)
    uint32_t s_pre = (R.x >> 24) & 15u;
    const int in_off = (int)(R.x & 511u), in_end = in_off + (int)(R.w & 63u);
    for (int m = in_off; m < in_end && ts[m] < t; ++m) s_pre ^= 1u << ((tg[m] >> 6) & 3u);
    dbg = EvDbg{s_pre, 0xFFu, w & 63u, (int)(R.w >> 30) + 1, t, glitch, 0.f, glitch ? 0.f : e_sw,
                glitch ? e_w : 0.f, 0.f};
  }
  return EvOut{c, e_w, 0.f, glitch ? 2u : 0u};
}

// The bins of one event: the band's shared-memory bins, or (exact mode) the
// global fp64 bins and integer counts.
template <bool kExact>
__device__ __forceinline__ void ev_commit(const BandRunArgs& A, float* hist, const EvOut& o, uint32_t item,
                                          uint32_t c0) {
  const RunArgs& a = A.r;
  const uint32_t lc = o.c - c0;
  if (lc >= A.L.band_cycles) {  // an event outside its band: layout inconsistency
    berr(a.err, item, kErrLayout);
    return;
  }
  const bool input = (o.flags & 1u) != 0u, glitch = (o.flags & 2u) != 0u;
  if (kExact) {
    double* bin = reinterpret_cast<double*>(a.bins + o.c);
    atomicAdd(bin, (double)o.e_w);
    if (input) atomicAdd(bin + 1, (double)o.dp);
    atomicAdd(a.cnt_ev + o.c, 1u);
    if (glitch) atomicAdd(a.cnt_gl + o.c, 1u);
  } else {
    float* h = hist + lc;
    atomicAdd(h + kHW, o.e_w);
    if (input) atomicAdd(h + kHD, o.dp);
    atomicAdd(reinterpret_cast<uint32_t*>(h + kHE), 1u);
    if (glitch) atomicAdd(reinterpret_cast<uint32_t*>(h + kHG), 1u);
  }
}

// The bins of one round of 32 events whose equal cycles come in runs of
// neighbouring lanes (items flagged by the layout): a segmented sum over each
// run of equal cycles, then one set of shared-memory atomics per run, by its
// last lane, instead of one per event -- lanes of a run would otherwise hit
// the same words and serialise. Called by all 32 lanes; `valid` false for
// lanes without an event.
__device__ __forceinline__ void ev_commit_runs(const BandRunArgs& A, float* hist, const EvOut& o, bool valid,
                                               uint32_t item, uint32_t c0, int lane) {
  uint32_t lc = o.c - c0;
  if (valid && lc >= A.L.band_cycles) {  // an event outside its band: layout inconsistency
    berr(A.r.err, item, kErrLayout);
    valid = false;
  }
  if (!valid) lc = 0xFFFFFFFFu;  // lanes without an event come last and form runs of their own
  const uint32_t lc_up = __shfl_up_sync(0xffffffffu, lc, 1);
  bool f = lane == 0 || lc_up != lc;  // the lane starts a run
  float w = o.e_w, d = (o.flags & 1u) ? o.dp : 0.f;
  uint32_t nc = valid ? (1u | ((o.flags & 2u) ? 1u << 16 : 0u)) : 0u;  // events | glitches << 16
#pragma unroll
  for (int sh = 1; sh < 32; sh <<= 1) {
    const float w2 = __shfl_up_sync(0xffffffffu, w, sh), d2 = __shfl_up_sync(0xffffffffu, d, sh);
    const uint32_t n2 = __shfl_up_sync(0xffffffffu, nc, sh);
    const bool f2 = __shfl_up_sync(0xffffffffu, (int)f, sh) != 0;
    if (lane >= sh) {
      if (!f) {
        w += w2;
        d += d2;
        nc += n2;
      }
      f = f || f2;
    }
  }
  const uint32_t lc_dn = __shfl_down_sync(0xffffffffu, lc, 1);
  if (valid && (lane == 31 || lc_dn != lc)) {  // the run's last lane holds its sums
    float* h = hist + lc;
    atomicAdd(h + kHW, w);
    if (d != 0.f) atomicAdd(h + kHD, d);
    atomicAdd(reinterpret_cast<uint32_t*>(h + kHE), nc & 0xFFFFu);
    if (nc >> 16) atomicAdd(reinterpret_cast<uint32_t*>(h + kHG), nc >> 16);
  }
}

// Debug outputs of one event: its CSR index is found by its time among its
// pin's events.
__device__ void event_debug(const RunArgs& a, uint32_t gate, int p, float t, uint32_t s_pre, int lut_ij,
                            bool glitch, uint32_t item) {
  const GateRec gr = a.gates[gate];
  const uint64_t pin = (uint64_t)gr.pin_base + p;
  const uint64_t hi = a.pin_off[pin + 1];
  uint64_t l = a.pin_off[pin], cnt = hi - l;
  while (cnt > 0) {
    const uint64_t half = cnt >> 1;
    if (a.t[l + half] < t) {
      l += half + 1;
      cnt -= half + 1;
    } else {
      cnt = half;
    }
  }
  if (l < hi && a.t[l] == t) {
    if (a.dbg_state) a.dbg_state[l] = (uint8_t)s_pre;
    if (a.dbg_lut) a.dbg_lut[l] = (uint8_t)lut_ij;
    if (a.dbg_glitch) a.dbg_glitch[l] = (uint8_t)glitch;
  } else {
    berr(a.err, item, kErrLayout);
  }
}

// One staged item on one warp: one lane per event, the input region first,
// then the output region. Input events take their states from a scan over
// each round of 32; where a region has events left for a second round, each
// lane computes two events before committing either.
template <bool kPow2, bool kDebug, bool kExact, bool kRuns>
__device__ __forceinline__ void band_item(const BandRunArgs& A, const CellTab& CT, float* hist,
                                          const uint8_t* stage, uint32_t item, const ItemGeo& g, uint32_t c0,
                                          BAcc& acc) {
  const RunArgs& a = A.r;
  const int lane = threadIdx.x & 31;
  if (!g.ok) {
    if (lane == 0) berr(a.err, item, kErrLayout);
    return;
  }
  const float* ts = reinterpret_cast<const float*>(stage) + g.ev_off;
  const uint16_t* tg = reinterpret_cast<const uint16_t*>(stage + kStTagOff) + g.tag_off;
  const uint4* rec = reinterpret_cast<const uint4*>(stage + kStRecOff);
  const uint2* rec2 = reinterpret_cast<const uint2*>(stage + kStRecOff);  // {x, v} of unit u at 2 u
  const float* gs = A.L.bs + g.e0;  // slews: read once, from HBM (prefetched into L2 ahead of the item)
  // and into L1: one 128-byte line per lane
  if ((uint32_t)lane * 32u < g.ev_off + g.n)
    asm volatile("prefetch.global.L1 [%0];" ::"l"(A.L.bs + g.ea + 32u * (uint32_t)lane) : "memory");
  const int n = (int)g.n, n_in = (int)g.n_in;
  EvDbg d0{}, d1{};
  uint32_t carry = 0;  // state scan across rounds
  if (kDebug) {
    for (int base = 0; base < n; base += 32) {
      const int i = base + lane;
      EvOut o;
      bool valid = i < n;
      if (base < n_in) {  // an input round (warp-uniform)
        const bool v = i < n_in;
        const int jj = v ? i : n_in - 1;
        const uint32_t w = tg[jj];
        const uint2 R = rec2[(w & 63u) * 2u];
        const uint32_t sb = round_state(v ? 1u << ((w >> 6) & 3u) : 0u, (int)(R.x & 511u), base,
                                        (R.x >> 24) & 15u, carry, lane);
        if (v) o = ev_input<kPow2, true>(a, CT, ts, tg, rec, gs, i, w, R, sb, true, acc, d0);
        else if (valid) o = ev_output<kPow2, true>(a, ts, tg, rec, gs, i, n, true, acc, d0);
      } else if (valid) {
        o = ev_output<kPow2, true>(a, ts, tg, rec, gs, i, n, true, acc, d0);
      }
      if (!valid) continue;
      ev_commit<kExact>(A, hist, o, item, c0);
      const uint32_t gate = A.L.ugate[g.u0 + d0.unit];
      if (a.gate_e) {  // this event's share of its gate's energies
        double* ge = a.gate_e + (size_t)gate * 4;
        if (d0.glitch) atomicAdd(ge + 2, (double)d0.g_gl);
        else if (i < n_in) atomicAdd(ge + 0, (double)d0.g_int);
        else atomicAdd(ge + 1, (double)d0.g_sw);
        if (i < n_in) atomicAdd(ge + 3, (double)d0.g_lk);
      }
      if (a.dbg_state || a.dbg_lut || a.dbg_glitch)
        event_debug(a, gate, d0.p, d0.t, d0.s_pre, (int)d0.lut_ij, d0.glitch, item);
    }
  } else if (kRuns) {
    // the same rounds, every lane computing (padding lanes on a clamped
    // index, not counted) so that the merged commit has all 32 lanes
    for (int base = 0; base < n_in; base += 64) {
      const int i0 = base + lane, i1 = i0 + 32;
      const bool v0 = i0 < n_in, v1 = i1 < n_in;
      const int j0 = min(i0, n_in - 1), j1 = min(i1, n_in - 1);
      const uint32_t w0 = tg[j0], w1 = tg[j1];
      const uint2 R0 = rec2[(w0 & 63u) * 2u], R1 = rec2[(w1 & 63u) * 2u];
      if (base + 32 < n_in) {
        uint32_t s0, s1;
        pair_state(1u << ((w0 >> 6) & 3u), (int)(R0.x & 511u), (R0.x >> 24) & 15u, v1 ? 1u << ((w1 >> 6) & 3u) : 0u,
                   (int)(R1.x & 511u), (R1.x >> 24) & 15u, base, carry, lane, s0, s1);
        const EvOut o0 = ev_input<kPow2, false>(a, CT, ts, tg, rec, gs, j0, w0, R0, s0, true, acc, d0);
        const EvOut o1 = ev_input<kPow2, false>(a, CT, ts, tg, rec, gs, j1, w1, R1, s1, v1, acc, d1);
        ev_commit_runs(A, hist, o0, true, item, c0, lane);
        ev_commit_runs(A, hist, o1, v1, item, c0, lane);
      } else {
        const uint32_t s0 = round_state(v0 ? 1u << ((w0 >> 6) & 3u) : 0u, (int)(R0.x & 511u), base,
                                        (R0.x >> 24) & 15u, carry, lane);
        const EvOut o0 = ev_input<kPow2, false>(a, CT, ts, tg, rec, gs, j0, w0, R0, s0, v0, acc, d0);
        ev_commit_runs(A, hist, o0, v0, item, c0, lane);
      }
    }
    for (int base = n_in; base < n; base += 32) {
      const int i0 = base + lane;
      const EvOut o0 = ev_output<kPow2, false>(a, ts, tg, rec, gs, min(i0, n - 1), n, i0 < n, acc, d0);
      ev_commit_runs(A, hist, o0, i0 < n, item, c0, lane);
    }
  } else {
    for (int base = 0; base < n_in; base += 64) {
      const int i0 = base + lane, i1 = i0 + 32;
      const bool v1 = i1 < n_in;
      const uint32_t w0 = tg[min(i0, n_in - 1)], w1 = tg[min(i1, n_in - 1)];
      const uint2 R0 = rec2[(w0 & 63u) * 2u], R1 = rec2[(w1 & 63u) * 2u];
      if (base + 32 < n_in) {  // every lane has a first event; some a second
        uint32_t s0, s1;
        pair_state(1u << ((w0 >> 6) & 3u), (int)(R0.x & 511u), (R0.x >> 24) & 15u, v1 ? 1u << ((w1 >> 6) & 3u) : 0u,
                   (int)(R1.x & 511u), (R1.x >> 24) & 15u, base, carry, lane, s0, s1);
        const EvOut o0 = ev_input<kPow2, false>(a, CT, ts, tg, rec, gs, i0, w0, R0, s0, true, acc, d0);
        const EvOut o1 = ev_input<kPow2, false>(a, CT, ts, tg, rec, gs, min(i1, n_in - 1), w1, R1, s1, v1, acc, d1);
        ev_commit<kExact>(A, hist, o0, item, c0);
        if (v1) ev_commit<kExact>(A, hist, o1, item, c0);
      } else {
        const uint32_t s0 = round_state(i0 < n_in ? 1u << ((w0 >> 6) & 3u) : 0u, (int)(R0.x & 511u), base,
                                        (R0.x >> 24) & 15u, carry, lane);
        if (i0 < n_in)
          ev_commit<kExact>(A, hist, ev_input<kPow2, false>(a, CT, ts, tg, rec, gs, i0, w0, R0, s0, true, acc, d0),
                            item, c0);
      }
    }
    for (int base = n_in; base < n; base += 64) {
      const int i0 = base + lane;
      if (base + 32 < n) {
        const int i1 = i0 + 32;
        const EvOut o0 = ev_output<kPow2, false>(a, ts, tg, rec, gs, i0, n, true, acc, d0);
        const EvOut o1 = ev_output<kPow2, false>(a, ts, tg, rec, gs, min(i1, n - 1), n, i1 < n, acc, d1);
        ev_commit<kExact>(A, hist, o0, item, c0);
        if (i1 < n) ev_commit<kExact>(A, hist, o1, item, c0);
      } else if (i0 < n) {
        ev_commit<kExact>(A, hist, ev_output<kPow2, false>(a, ts, tg, rec, gs, i0, n, true, acc, d0), item, c0);
      }
    }
  }
  __syncwarp();
}

template <bool kPow2, bool kDebug, bool kExact>
__global__ void __launch_bounds__(kBT, 1) k_band(const BandRunArgs A) {
  extern __shared__ __align__(128) uint8_t smem[];
  float* hist = reinterpret_cast<float*>(smem);
  float4* rows = reinterpret_cast<float4*>(smem + kHist + kCellsB);  // the warp buffers, during a flush
  uint32_t* cells_s = reinterpret_cast<uint32_t*>(smem + kHist);
  BandItem* s_items = reinterpret_cast<BandItem*>(smem + kHist + kCellsB + kBW * kWarpB);  // [2][kChunkMaxItems + 1]
  __shared__ __align__(8) uint64_t s_bar[kBW];
  __shared__ __align__(8) uint64_t s_ibar[2];
  __shared__ uint32_t s_chunk_lo, s_chunk_hi, s_seg_end, s_band, s_abort;
  __shared__ unsigned int s_next;
  __shared__ double s_tot[4];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RunArgs& a = A.r;
  const BandLayout& L = A.L;
  const uint32_t cb = L.band_cycles;
  const uint32_t n_items = L.n_items;
  uint8_t* wbuf = smem + kHist + kCellsB + (size_t)warp * kWarpB;
  uint64_t* bar = &s_bar[warp];

  if (tid < 4) s_tot[tid] = 0.0;
  for (uint32_t i = tid; i < 4 * kBandMaxCycles; i += kBT) hist[i] = 0.f;
  CellTab CT;
  {  // the layout is only built for libraries of at most kSmemCells cells
    float* sax = reinterpret_cast<float*>(cells_s);
    uint32_t* info = cells_s + kSmemCells * kAxStride;
    float2* sxp = reinterpret_cast<float2*>(info + kSmemCells);
    const uint32_t nc = min(a.n_cells, (uint32_t)kSmemCells);
    for (uint32_t i = tid; i < nc * (uint32_t)kAxStride; i += kBT) {
      const uint32_t ci = i / kAxStride, m = i % kAxStride;
      const CellDesc& cd = a.cells[ci];
      if (m == 0) info[ci] = (uint32_t)(cd.ns - 1) | ((uint32_t)(cd.nl - 1) << 8) | (cd.patch_off << 16);
      sax[i] = m == 0 ? cd.sax[0] : ((int)m <= (int)cd.ns - 2 ? cd.sax[m] : __int_as_float(0x7f800000));
      if (m < 8) sxp[ci * 8 + m] = make_float2(cd.sax[m], cd.isax[m]);
    }
    float* lk = reinterpret_cast<float*>(sxp + kSmemCells * 8);
    for (uint32_t i = tid; i < nc * (uint32_t)kLeakStride; i += kBT) {
      const uint32_t ci = i / kLeakStride, st = i % kLeakStride;
      const CellDesc& cd = a.cells[ci];
      lk[i] = st < (1u << cd.k) ? a.leak[cd.leak_off + st] : 0.f;
    }
    CT.sax = sax;
    CT.leak = lk;
    CT.info = info;
    CT.sxp = sxp;
  }
  if (lane == 0) {
    mbar_init(bar, 1);
    if (tid == 0) {
      mbar_init(&s_ibar[0], 1);
      mbar_init(&s_ibar[1], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  BAcc acc{0.f, 0.f, 0.f, 0.f, 0.f};
  int since = 0;
  uint32_t phase = 0;  // parity of the stage barrier's next completion
  bool bad = false;    // a stage copy never landed: this warp stops working
  // CTAs take chunks of A.chunk items from a global counter; thread 0 takes
  // the next chunk one chunk ahead and copies its item records into the other
  // half of s_items. The band bins stay in shared memory until a chunk brings
  // a new band.
  uint2 pref = make_uint2(0, 0);
  uint32_t ibuf = 0, iphase = 0;  // records buffer of the current chunk, parity bits of both buffers
  if (tid == 0) {
    const uint2 c = take_chunk(A.item_ctr, n_items, A.chunk);
    s_chunk_lo = c.x;
    s_chunk_hi = c.y;
    if (c.x < c.y) {
      mbar_expect_arrive(&s_ibar[0], (c.y - c.x + 1) * 16u);
      bulk_g2s(s_items, L.items + c.x, (c.y - c.x + 1) * 16u, &s_ibar[0]);
    }
    pref = take_chunk(A.item_ctr, n_items, A.chunk);
    if (pref.x < pref.y) {
      mbar_expect_arrive(&s_ibar[1], (pref.y - pref.x + 1) * 16u);
      bulk_g2s(s_items + (kChunkMaxItems + 1), L.items + pref.x, (pref.y - pref.x + 1) * 16u, &s_ibar[1]);
    }
    s_band = 0xFFFFFFFFu;
    s_abort = 0;
  }
  __syncthreads();
  for (;;) {
    const uint32_t c_lo = s_chunk_lo, c_hi = s_chunk_hi;
    if (c_lo >= c_hi) break;
    const BandItem* it = s_items + ibuf * (kChunkMaxItems + 1);  // records of items c_lo .. c_hi
    if (tid == 0) {
      bool ok = false;
      for (uint32_t w = 0; w < A.wait_limit && !ok; ++w) ok = mbar_try_wait(&s_ibar[ibuf], (iphase >> ibuf) & 1u);
      if (ok) {
        iphase ^= 1u << ibuf;
      } else {
        berr(a.err, c_lo, kErrStageTimeout);
        s_abort = 1;
      }
    }
    __syncthreads();  // the chunk's records are in
    if (s_abort) break;
    for (uint32_t cur = c_lo; cur < c_hi;) {
      const uint32_t old_band = s_band;
      __syncthreads();  // everyone has read s_band
      if (tid == 0) {
        const uint32_t b = item_band(it[cur - c_lo]);
        s_band = b;
        s_seg_end = band_end(it + (cur - c_lo), cur, c_hi, b);
        s_next = 0;
      }
      __syncthreads();
      const uint32_t band = s_band, seg_end = s_seg_end;
      if (band != old_band && old_band != 0xFFFFFFFFu) {
        bflush_band<kExact>(A, hist, rows, old_band);
        __syncthreads();
      }
      const uint32_t c0 = band * cb;
      uint32_t my = seg_end;
      if (lane == 0 && !bad) my = cur + atomicAdd(&s_next, 1u);
      my = __shfl_sync(0xffffffffu, my, 0);
      while (my < seg_end) {
        uint32_t nx = seg_end;
        ItemGeo gl{};
        if (lane == 0) {
          gl = item_geo(it[my - c_lo], it[my + 1 - c_lo]);
          // (test hook: the skipped item gets neither an arrival nor a copy,
          // so its bounded wait below runs out)
          if (my != A.skip_item) stage_item(L, gl, wbuf, bar);
          // take the next item now and start bringing its data into L2
          nx = cur + atomicAdd(&s_next, 1u);
          if (nx < seg_end) prefetch_item(L, item_geo(it[nx - c_lo], it[nx + 1 - c_lo]));
        }
        ItemGeo gcur;
        gcur.e0 = __shfl_sync(0xffffffffu, gl.e0, 0);
        gcur.ea = __shfl_sync(0xffffffffu, gl.ea, 0);
        gcur.u0 = __shfl_sync(0xffffffffu, gl.u0, 0);
        gcur.n = __shfl_sync(0xffffffffu, gl.n, 0);
        gcur.nu = __shfl_sync(0xffffffffu, gl.nu, 0);
        gcur.n_in = __shfl_sync(0xffffffffu, gl.n_in, 0);
        gcur.ev_off = __shfl_sync(0xffffffffu, gl.ev_off, 0);
        gcur.tag_off = __shfl_sync(0xffffffffu, gl.tag_off, 0);
        gcur.ev_bytes = gcur.tag_bytes = 0;
        gcur.ok = __shfl_sync(0xffffffffu, (int)gl.ok, 0) != 0;
        gcur.runs = __shfl_sync(0xffffffffu, (int)gl.runs, 0) != 0;
        bool ok = false;
        for (uint32_t w = 0; w < A.wait_limit && !ok; ++w) ok = mbar_try_wait(bar, phase);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) {
            berr(a.err, my, kErrStageTimeout);
            // keep waiting (bounded) for the copy in flight: the warp buffers
            // are reused as flush rows once the band's items are done
            bool done = false;
            for (uint32_t w = 0; w < A.wait_limit && !done; ++w) done = mbar_try_wait(bar, phase);
          }
          __syncwarp();
          bad = true;
          break;
        }
        phase ^= 1u;
        if (!kDebug && !kExact && gcur.runs)  // warp-uniform
          band_item<kPow2, kDebug, kExact, true>(A, CT, hist, wbuf, my, gcur, c0, acc);
        else
          band_item<kPow2, kDebug, kExact, false>(A, CT, hist, wbuf, my, gcur, c0, acc);
        if (++since == kTotEvery) {
          bflush_acc(acc, s_tot);
          since = 0;
        }
        my = __shfl_sync(0xffffffffu, nx, 0);
      }
      cur = seg_end;
    }
    __syncthreads();  // the chunk's items are done and its records no longer read
    if (tid == 0) {
      s_chunk_lo = pref.x;
      s_chunk_hi = pref.y;
      pref = take_chunk(A.item_ctr, n_items, A.chunk);
      if (pref.x < pref.y) {  // into the buffer just freed
        mbar_expect_arrive(&s_ibar[ibuf], (pref.y - pref.x + 1) * 16u);
        bulk_g2s(s_items + ibuf * (kChunkMaxItems + 1), L.items + pref.x, (pref.y - pref.x + 1) * 16u,
                 &s_ibar[ibuf]);
      }
    }
    ibuf ^= 1u;
    __syncthreads();
  }
  __syncthreads();
  if (s_band != 0xFFFFFFFFu) bflush_band<kExact>(A, hist, rows, s_band);
  bflush_acc(acc, s_tot);
  __syncthreads();
  if (tid < 4) atomicAdd(a.totals + tid, s_tot[tid]);
  if (s_abort && tid == 0) {
    // a records copy never landed: wait (bounded) for the copies that may
    // still be in flight before the CTA's shared memory is released
    for (int bsel = 0; bsel < 2; ++bsel) {
      bool done = false;
      for (uint32_t w = 0; w < A.wait_limit && !done; ++w) done = mbar_try_wait(&s_ibar[bsel], (iphase >> bsel) & 1u);
    }
  }
}

template <bool P, bool D, bool X>
void band_attr() {
  static bool done = false;
  if (!done) {
    cudaFuncSetAttribute(k_band<P, D, X>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemB);
    done = true;
  }
}

template <bool P, bool D, bool X>
int band_occ() {
  band_attr<P, D, X>();
  int n = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_band<P, D, X>, kBT, kSmemB);
  return n > 0 ? n : 1;
}

template <bool P, bool D, bool X>
void band_launch(const BandRunArgs& A, int grid, cudaStream_t st) {
  band_attr<P, D, X>();
  k_band<P, D, X><<<grid, kBT, kSmemB, st>>>(A);
}

}  // namespace

int band_blocks_per_sm(bool pow2, bool debug, bool exact) {
  const int sel = (pow2 ? 4 : 0) | (debug ? 2 : 0) | (exact ? 1 : 0);
  switch (sel) {
    case 0: return band_occ<false, false, false>();
    case 1: return band_occ<false, false, true>();
    case 2: return band_occ<false, true, false>();
    case 3: return band_occ<false, true, true>();
    case 4: return band_occ<true, false, false>();
    case 5: return band_occ<true, false, true>();
    case 6: return band_occ<true, true, false>();
    default: return band_occ<true, true, true>();
  }
}

cudaError_t band_fused(const BandRunArgs& A0, int sm_count, bool debug, bool exact, cudaStream_t st) {
  if (A0.L.n_items == 0) return cudaSuccess;
  const bool pow2 = A0.r.inv_t_clk != 0.f;
  const int grid = sm_count * band_blocks_per_sm(pow2, debug, exact);
  BandRunArgs A = A0;
  A.chunk = std::min(kChunkMax, std::max(kChunkMin, A.L.n_items / (16u * (uint32_t)grid)));
  const int sel = (pow2 ? 4 : 0) | (debug ? 2 : 0) | (exact ? 1 : 0);
  switch (sel) {
    case 0: band_launch<false, false, false>(A, grid, st); break;
    case 1: band_launch<false, false, true>(A, grid, st); break;
    case 2: band_launch<false, true, false>(A, grid, st); break;
    case 3: band_launch<false, true, true>(A, grid, st); break;
    case 4: band_launch<true, false, false>(A, grid, st); break;
    case 5: band_launch<true, false, true>(A, grid, st); break;
    case 6: band_launch<true, true, false>(A, grid, st); break;
    default: band_launch<true, true, true>(A, grid, st); break;
  }
  return cudaGetLastError();
}

}  // namespace pa
