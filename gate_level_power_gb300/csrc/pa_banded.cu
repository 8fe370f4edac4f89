// Cycle-banded event layout and the banded fused power kernel (sm_103a).
//
// The power step of "GPU-Accelerated Gate-Level Time-Based Power Analysis via
// Event-Density-Aware Partitioning and Kernel Fusion" (Sections 2.4.1-2.4.2,
// Eqs. 1-4, Figs. 2, 3 and 7) adds every event's energy to the waveform bin of
// its clock cycle (Fig. 7's atomicAdd into w). Done with one global atomic per
// event, a billion events are bound by the L2 atomic units. Here the events are
// first regrouped into bands of consecutive cycles (a load-time layout for one
// clock period): work items never leave their band, so each CTA keeps the
// band's cycle bins in shared memory and flushes them to global memory once per
// band it touches. Within a band the per-pin CSR order is kept, so the gate
// state and glitch rules are the ones of the unbanded kernel; the state at the
// band start travels in the per-(band, gate) record.
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

__device__ __forceinline__ uint32_t wscan_incl_u32(uint32_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
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

cudaError_t scan_u32_to_u64(const uint32_t* in, uint64_t n, uint64_t* blk, uint64_t* out, cudaStream_t st) {
  const uint32_t nb = (uint32_t)((n + kScanBlock - 1) / kScanBlock);
  if (nb == 0) return cudaMemsetAsync(out, 0, sizeof(uint64_t), st);
  k_scan_sum<<<nb, 256, 0, st>>>(in, n, blk);
  k_scan_blocks<<<1, 1024, 0, st>>>(blk, nb);
  k_scan_apply<<<nb, 256, 0, st>>>(in, n, blk, out);
  return cudaGetLastError();
}

}  // namespace

uint32_t band_scan_blocks(uint64_t n) { return (uint32_t)((n + kScanBlock - 1) / kScanBlock) + 1; }

// ------------------------------------------------------------------ layout build (load time)

namespace {

// Events per (pin, band): one warp per gate; the band of consecutive events of
// a pin is non-decreasing, so a warp adds each band's share with one atomic.
template <bool kPow2>
__global__ void __launch_bounds__(256) k_bb_count(const BandBuildArgs a) {
  const int lane = threadIdx.x & 31;
  const uint64_t warp = (blockIdx.x * (uint64_t)blockDim.x + threadIdx.x) >> 5;
  const uint64_t n_warps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
  const uint32_t nb = a.n_bands;
  for (uint64_t g = warp; g < a.n_gates; g += n_warps) {
    const GateRec r = a.gates[g];
    const int k = (int)((r.init >> 16) & 0xff);
    for (int p = 0; p <= k; ++p) {
      const uint64_t pin = (uint64_t)r.pin_base + p;
      const uint64_t lo = a.pin_off[pin], hi = a.pin_off[pin + 1];
      for (uint64_t e0 = lo; e0 < hi; e0 += 32) {
        const uint64_t e = e0 + lane;
        const bool act = e < hi;
        const uint32_t b = act ? cyc<kPow2>(a.t[e], a.t_clk, a.inv_t_clk) / a.band_cycles : 0xFFFFFFFFu;
        const unsigned grp = __match_any_sync(0xffffffffu, b);
        if (act && lane == __ffs(grp) - 1) atomicAdd(a.cnt + pin * nb + b, (uint32_t)__popc(grp));
      }
    }
  }
}

// Heavy if some pin has more than kLightPinMax events in some band.
__global__ void __launch_bounds__(256) k_bb_classify(const BandBuildArgs a) {
  const uint32_t g = blockIdx.x * 256u + threadIdx.x;
  if (g >= a.n_gates) return;
  const GateRec r = a.gates[g];
  const int k = (int)((r.init >> 16) & 0xff);
  const uint32_t nb = a.n_bands;
  bool heavy = false;
  for (int p = 0; p <= k && !heavy; ++p) {
    const uint32_t* c = a.cnt + ((uint64_t)r.pin_base + p) * nb;
    for (uint32_t b = 0; b < nb; ++b) heavy |= c[b] > (uint32_t)kLightPinMax;
  }
  a.heavy[g] = heavy ? 1 : 0;
}

// Light / heavy ranks: scan of (light ? 1 : 2^32) over gates.
__global__ void __launch_bounds__(256) k_bb_flag_sum(const BandBuildArgs a, uint64_t* blk) {
  const uint64_t i0 = (uint64_t)blockIdx.x * kScanBlock + (uint64_t)threadIdx.x * kScanPer;
  uint64_t s = 0;
#pragma unroll
  for (int i = 0; i < kScanPer; ++i)
    if (i0 + i < a.n_gates) s += a.heavy[i0 + i] ? (1ull << 32) : 1ull;
  uint64_t tot;
  bscan_excl_u64(s, tot);
  if (threadIdx.x == 0) blk[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(256) k_bb_flag_apply(const BandBuildArgs a, const uint64_t* blk) {
  const uint64_t i0 = (uint64_t)blockIdx.x * kScanBlock + (uint64_t)threadIdx.x * kScanPer;
  uint64_t v[kScanPer];
  uint64_t s = 0;
#pragma unroll
  for (int i = 0; i < kScanPer; ++i) {
    v[i] = i0 + i < a.n_gates ? (a.heavy[i0 + i] ? (1ull << 32) : 1ull) : 0ull;
    s += v[i];
  }
  uint64_t tot;
  uint64_t off = blk[blockIdx.x] + bscan_excl_u64(s, tot);
#pragma unroll
  for (int i = 0; i < kScanPer; ++i) {
    const uint64_t g = i0 + i;
    if (g < a.n_gates) {
      const uint32_t lr = (uint32_t)off, hr = (uint32_t)(off >> 32);
      if (a.heavy[g]) {
        a.rank[g] = hr;
        a.L.hgate[hr] = (uint32_t)g;
      } else {
        a.rank[g] = lr;
        a.L.lgate[lr] = (uint32_t)g;
      }
    }
    off += v[i];
  }
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) {
    const uint64_t t = blk[gridDim.x];
    a.totals[0] = (uint32_t)t;
    a.totals[1] = (uint32_t)(t >> 32);
  }
}

// Unit of (band b, gate g): position b * G + (light ? lr : n_light + hr).
__device__ __forceinline__ uint64_t unit_pos(const BandBuildArgs& a, uint32_t g) {
  return a.heavy[g] ? (uint64_t)a.L.n_light + a.rank[g] : (uint64_t)a.rank[g];
}

__global__ void __launch_bounds__(256) k_bb_unitsize(const BandBuildArgs a) {
  const uint32_t g = blockIdx.x * 256u + threadIdx.x;
  if (g >= a.n_gates) return;
  const GateRec r = a.gates[g];
  const int k = (int)((r.init >> 16) & 0xff);
  const uint32_t nb = a.n_bands;
  const uint64_t pos = unit_pos(a, g);
  const uint32_t* c = a.cnt + (uint64_t)r.pin_base * nb;
  for (uint32_t b = 0; b < nb; ++b) {
    uint32_t sz = 0;
    for (int p = 0; p <= k; ++p) sz += c[(uint64_t)p * nb + b];
    a.unit_size[(uint64_t)b * a.n_gates + pos] = sz;
  }
}

// Scatter: one warp per gate; lane b (and b + 32) holds band b's running
// offset, count and count-before for the current pin.
template <bool kPow2>
__global__ void __launch_bounds__(256) k_bb_scatter(const BandBuildArgs a) {
  const int lane = threadIdx.x & 31;
  const uint64_t warp = (blockIdx.x * (uint64_t)blockDim.x + threadIdx.x) >> 5;
  const uint64_t n_warps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
  const uint32_t nb = a.n_bands, G = a.n_gates;
  const uint32_t b0 = (uint32_t)lane, b1 = (uint32_t)lane + 32;
  for (uint64_t g = warp; g < G; g += n_warps) {
    const GateRec r = a.gates[g];
    const int k = (int)((r.init >> 16) & 0xff);
    const bool heavy = a.heavy[g] != 0;
    const uint64_t pos = unit_pos(a, (uint32_t)g);
    uint64_t off0 = b0 < nb ? a.unit_off[(uint64_t)b0 * G + pos] : 0;
    uint64_t off1 = b1 < nb ? a.unit_off[(uint64_t)b1 * G + pos] : 0;
    const uint64_t base0 = off0, base1 = off1;
    const uint32_t init = r.init & 0xffu;
    uint32_t st0 = init, st1 = init, rec0 = 0, rec1 = 0;
    for (int p = 0; p <= k; ++p) {
      const uint64_t pin = (uint64_t)r.pin_base + p;
      const uint32_t c0 = b0 < nb ? a.cnt[pin * nb + b0] : 0u;
      const uint32_t c1 = b1 < nb ? a.cnt[pin * nb + b1] : 0u;
      const uint32_t inc0 = wscan_incl_u32(c0, lane);
      const uint32_t tot0 = __shfl_sync(0xffffffffu, inc0, 31);
      const uint32_t inc1 = wscan_incl_u32(c1, lane) + tot0;
      const uint32_t cum0 = inc0 - c0, cum1 = inc1 - c1;  // events of the pin in earlier bands
      if (p < k) {
        st0 ^= (cum0 & 1u) << p;
        st1 ^= (cum1 & 1u) << p;
      }
      rec0 |= (c0 & 31u) << (5 * p);
      rec1 |= (c1 & 31u) << (5 * p);
      if (heavy) {
        if (b0 < nb) a.L.hrec[(uint64_t)b0 * a.L.n_heavy + a.rank[g]].cnt[p] = c0;
        if (b1 < nb) a.L.hrec[(uint64_t)b1 * a.L.n_heavy + a.rank[g]].cnt[p] = c1;
      }
      const uint64_t lo = a.pin_off[pin], hi = a.pin_off[pin + 1];
      for (uint64_t e0 = lo; e0 < hi; e0 += 32) {
        const uint64_t e = e0 + lane;
        const bool act = e < hi;
        const float t = act ? a.t[e] : 0.f;
        const uint32_t b = act ? cyc<kPow2>(t, a.t_clk, a.inv_t_clk) / a.band_cycles : 0u;
        const int src = (int)(b & 31u);
        const uint32_t cum_a = __shfl_sync(0xffffffffu, cum0, src);
        const uint32_t cum_b = __shfl_sync(0xffffffffu, cum1, src);
        const uint64_t off_a = __shfl_sync(0xffffffffu, off0, src);
        const uint64_t off_b = __shfl_sync(0xffffffffu, off1, src);
        if (act) {
          const bool hi_band = b >= 32;
          const uint64_t rank = (e - lo) - (hi_band ? cum_b : cum_a);
          const uint64_t dest = (hi_band ? off_b : off_a) + rank;
          a.L.bt[dest] = t;
          a.L.bs[dest] = a.s[e];
        }
      }
      off0 += c0;
      off1 += c1;
    }
    if (!heavy) {
      if (b0 < nb) a.L.lrec[(uint64_t)b0 * a.L.n_light + a.rank[g]] = rec0 | (st0 << 25);
      if (b1 < nb) a.L.lrec[(uint64_t)b1 * a.L.n_light + a.rank[g]] = rec1 | (st1 << 25);
    } else {
      if (b0 < nb) {
        HeavyRec& h = a.L.hrec[(uint64_t)b0 * a.L.n_heavy + a.rank[g]];
        h.base = base0;
        h.state = st0;
        for (int p = k + 1; p < 5; ++p) h.cnt[p] = 0;
      }
      if (b1 < nb) {
        HeavyRec& h = a.L.hrec[(uint64_t)b1 * a.L.n_heavy + a.rank[g]];
        h.base = base1;
        h.state = st1;
        for (int p = k + 1; p < 5; ++p) h.cnt[p] = 0;
      }
    }
  }
}

__global__ void __launch_bounds__(256) k_bb_lblk(const BandBuildArgs a) {
  const uint32_t nlb = a.L.n_lblk;
  const uint64_t i = blockIdx.x * (uint64_t)256 + threadIdx.x;
  if (i >= (uint64_t)a.n_bands * (nlb + 1)) return;
  const uint32_t b = (uint32_t)(i / (nlb + 1)), j = (uint32_t)(i % (nlb + 1));
  const uint32_t lr = min(j * (uint32_t)kLightBlock, a.L.n_light);
  a.L.lblk[i] = a.unit_off[(uint64_t)b * a.n_gates + lr];
}

int warp_grid(uint64_t n_gates) {
  return (int)std::min<uint64_t>((n_gates * 32 + 255) / 256 + 1, 152ull * 64);
}

}  // namespace

cudaError_t band_build_phase1(BandBuildArgs& a, cudaStream_t st) {
  const uint64_t ncnt = a.n_pins * (uint64_t)a.n_bands;
  cudaError_t e = cudaMemsetAsync(a.cnt, 0, ncnt * sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  if (a.pow2) k_bb_count<true><<<warp_grid(a.n_gates), 256, 0, st>>>(a);
  else k_bb_count<false><<<warp_grid(a.n_gates), 256, 0, st>>>(a);
  const uint32_t gb = (a.n_gates + 255) / 256;
  if (gb) k_bb_classify<<<gb, 256, 0, st>>>(a);
  const uint32_t nb = (uint32_t)((a.n_gates + kScanBlock - 1) / kScanBlock);
  if (nb) {
    k_bb_flag_sum<<<nb, 256, 0, st>>>(a, a.scan_blk);
    k_scan_blocks<<<1, 1024, 0, st>>>(a.scan_blk, nb);
    k_bb_flag_apply<<<nb, 256, 0, st>>>(a, a.scan_blk);
  } else {
    e = cudaMemsetAsync(a.totals, 0, 2 * sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t band_build_phase2(BandBuildArgs& a, cudaStream_t st) {
  const uint32_t gb = (a.n_gates + 255) / 256;
  const uint64_t nu = (uint64_t)a.n_bands * a.n_gates;
  if (gb) k_bb_unitsize<<<gb, 256, 0, st>>>(a);
  cudaError_t e = scan_u32_to_u64(a.unit_size, nu, a.scan_blk, a.unit_off, st);
  if (e != cudaSuccess) return e;
  if (a.pow2) k_bb_scatter<true><<<warp_grid(a.n_gates), 256, 0, st>>>(a);
  else k_bb_scatter<false><<<warp_grid(a.n_gates), 256, 0, st>>>(a);
  const uint64_t nl = (uint64_t)a.n_bands * (a.L.n_lblk + 1);
  k_bb_lblk<<<(uint32_t)((nl + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ banded partition (per run)
//
// Work items in band-major order: light tiles (runs of light blocks of one band
// whose first event offsets share a kBTileTarget bucket; at most kBGateCap
// gates), then heavy items (runs of small heavy units sharing a bucket, or one
// unit alone when it has more than kBUnitSmall events; units above kBTileCap
// events are streamed). The CTAs of the fused kernel take contiguous runs of
// this list holding equal shares of the events, so each touches few bands.

namespace {

__device__ __forceinline__ uint64_t lblk_at(const BandLayout& L, uint32_t b, uint32_t j) {
  return L.lblk[(uint64_t)b * (L.n_lblk + 1) + j];
}

__device__ __forceinline__ uint32_t hunit_n(const HeavyRec& h) {
  return h.cnt[0] + h.cnt[1] + h.cnt[2] + h.cnt[3] + h.cnt[4];
}

__device__ bool light_head(const BandLayout& L, uint32_t b, uint32_t j) {
  if (j == 0 || j % (uint32_t)(kBGateCap / kLightBlock) == 0) return true;
  const uint64_t base = lblk_at(L, b, 0);
  return (lblk_at(L, b, j) - base) / kBTileTarget != (lblk_at(L, b, j - 1) - base) / kBTileTarget;
}

__device__ bool heavy_big(const BandLayout& L, uint32_t b, uint32_t h) {
  return hunit_n(L.hrec[(uint64_t)b * L.n_heavy + h]) > kBUnitSmall;
}

__device__ bool heavy_head(const BandLayout& L, uint32_t b, uint32_t h) {
  if (h == 0 || h % (uint32_t)kBGateCap == 0) return true;
  if (heavy_big(L, b, h) || heavy_big(L, b, h - 1)) return true;
  const uint64_t base = L.hrec[(uint64_t)b * L.n_heavy].base;
  return (L.hrec[(uint64_t)b * L.n_heavy + h].base - base) / kBTileTarget !=
         (L.hrec[(uint64_t)b * L.n_heavy + h - 1].base - base) / kBTileTarget;
}

// flags[i] = 1 where a light (kind 0) or heavy (kind 1) item starts.
__global__ void __launch_bounds__(256) k_bp_flags(const BandLayout L, uint32_t kind, uint32_t* flags) {
  const uint64_t per = kind == 0 ? L.n_lblk : L.n_heavy;
  const uint64_t i = blockIdx.x * (uint64_t)256 + threadIdx.x;
  if (i >= (uint64_t)L.n_bands * per) return;
  const uint32_t b = (uint32_t)(i / per), j = (uint32_t)(i % per);
  flags[i] = kind == 0 ? (uint32_t)light_head(L, b, j) : (uint32_t)heavy_head(L, b, j);
}

// Items of one kind at item_base + (exclusive scan of the flags); events per item.
__global__ void __launch_bounds__(256) k_bp_emit(const BandLayout L, uint32_t kind, const uint32_t* flags,
                                                 const uint64_t* pos, uint32_t item_base, BandItem* items,
                                                 uint32_t* item_n) {
  const uint64_t per = kind == 0 ? L.n_lblk : L.n_heavy;
  const uint64_t n = (uint64_t)L.n_bands * per;
  const uint64_t i = blockIdx.x * (uint64_t)256 + threadIdx.x;
  if (i >= n || !flags[i]) return;
  const uint32_t b = (uint32_t)(i / per), j = (uint32_t)(i % per);
  // the item ends before the next head of the same band
  uint32_t e = j + 1;
  while (e < per && !flags[(uint64_t)b * per + e]) ++e;
  BandItem it;
  it.band = b;
  it.first = j;
  it.last = e;
  uint64_t ev;
  if (kind == 0) {
    it.kind = 0;
    ev = lblk_at(L, b, e) - lblk_at(L, b, j);
  } else {
    const HeavyRec& h0 = L.hrec[(uint64_t)b * L.n_heavy + j];
    const HeavyRec& h1 = L.hrec[(uint64_t)b * L.n_heavy + e - 1];
    ev = h1.base + hunit_n(h1) - h0.base;
    it.kind = (e == j + 1 && ev > (uint64_t)kBTileCap) ? 2u : 1u;
  }
  it.e0 = kind == 0 ? lblk_at(L, b, j) : L.hrec[(uint64_t)b * L.n_heavy + j].base;
  it.n = (uint32_t)ev;
  it.pad = 0;
  const uint32_t k = item_base + (uint32_t)pos[i];
  items[k] = it;
  item_n[k] = (uint32_t)ev;
}

}  // namespace

uint32_t band_max_items(const BandLayout& L) {
  return L.n_bands * (L.n_lblk + L.n_heavy) + 1;
}

// Build the item list; host_items[0..1] = light and heavy item counts.
cudaError_t band_partition(BandRunArgs& A, uint32_t* flags, uint64_t* pos, uint64_t* scan_blk,
                           uint32_t* item_n, uint32_t* host_items, cudaStream_t st) {
  const BandLayout& L = A.L;
  uint32_t base = 0;
  for (uint32_t kind = 0; kind < 2; ++kind) {
    const uint64_t n = (uint64_t)L.n_bands * (kind == 0 ? L.n_lblk : L.n_heavy);
    host_items[kind] = 0;
    if (n == 0) continue;
    const uint32_t g = (uint32_t)((n + 255) / 256);
    k_bp_flags<<<g, 256, 0, st>>>(L, kind, flags);
    cudaError_t e = scan_u32_to_u64(flags, n, scan_blk, pos, st);
    if (e != cudaSuccess) return e;
    uint64_t cnt = 0;
    e = cudaMemcpyAsync(&cnt, pos + n, sizeof(cnt), cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return e;
    k_bp_emit<<<g, 256, 0, st>>>(L, kind, flags, pos, base, A.items, item_n);
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    host_items[kind] = (uint32_t)cnt;
    base += (uint32_t)cnt;
  }
  // event prefix of the items
  return scan_u32_to_u64(item_n, base, scan_blk, A.item_ev, st);
}

// ------------------------------------------------------------------ per-run gate records

namespace {

__global__ void __launch_bounds__(256) k_bg_gaterun(const BandRunArgs A) {
  const uint64_t i = blockIdx.x * (uint64_t)256 + threadIdx.x;
  const uint64_t nl = A.L.n_light, nh = A.L.n_heavy;
  double p0 = 0.0;
  if (i < nl + nh) {
    const bool light = i < nl;
    const uint32_t g = light ? A.L.lgate[i] : A.L.hgate[i - nl];
    const GateRec r = A.r.gates[g];
    const CellDesc& cd = A.r.cells[r.cell];
    const float C = r.load;
    int j = 0;
    for (int m = 1; m <= cd.nl - 2; ++m) j += (C >= cd.lax[m]) ? 1 : 0;
    GateRun gr;
    gr.packed = (r.cell & 0xffffu) | ((uint32_t)cd.k << 16) | ((uint32_t)j << 20);
    gr.v = (C - cd.lax[j]) * cd.ilax[j];
    gr.esw = A.r.half_vdd2 * C;
    gr.gate = g;
    if (light) A.grun_l[i] = gr;
    else A.grun_h[i - nl] = gr;
    // P0: leakage of every gate's initial input state
    p0 = (double)A.r.leak[cd.leak_off + (r.init & ((1u << cd.k) - 1u))];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) p0 += __shfl_xor_sync(0xffffffffu, p0, o);
  if ((threadIdx.x & 31) == 0 && p0 != 0.0) atomicAdd(A.r.p0, p0);
}

}  // namespace

cudaError_t band_gate_run(BandRunArgs& A, cudaStream_t st) {
  const uint64_t n = (uint64_t)A.L.n_light + A.L.n_heavy;
  if (n) k_bg_gaterun<<<(uint32_t)((n + 255) / 256), 256, 0, st>>>(A);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ banded fused kernel
//
// One CTA per SM takes a contiguous, event-balanced run of band-major items.
// Thread 0 prefetches item i+1 with TMA bulk copies (events, unit records,
// per-run gate records) into the spare one of two shared-memory stages while
// the CTA works on item i; an mbarrier per stage signals completion. Events
// add into the band's cycle bins in shared memory; a band change flushes them.

namespace {

constexpr int kBThreads = 512;
constexpr int kBWarps = kBThreads / 32;
static_assert(kBGateCap == kBThreads, "one unit per thread in tile setup");

struct __align__(16) BSlot {
  uint16_t st[5];   // staged start of each pin's segment
  uint16_t len[5];  // events of each pin to process
  uint8_t kj;       // k (bits 0..3), load-axis interval j (bits 4..7)
  uint8_t state;    // input state before the segments (band start, or stream window start)
  uint16_t cell;
  float v, esw;
};
static_assert(sizeof(BSlot) == 32, "slot size");

struct BStream {
  uint64_t cur[5], end[5];
  float prev_t[5], prev_s[5], bound[5];
  uint8_t has_prev[5];
  uint8_t pre;  // parity of the events already processed, per pin
  int done;
};

struct BAcc {
  float e_int, e_sw, e_gl, e_lk;
};

struct StageMeta {
  BandItem it;
  uint32_t ev_off, rec_off;
};

constexpr int kStEv = kBTileCap + 8;  // staged floats per array (16-byte rounding slack)
constexpr size_t kStTs = (size_t)kStEv * 4;
constexpr size_t kStRec = (size_t)kBGateCap * sizeof(HeavyRec) + 16;
constexpr size_t kStGrun = (size_t)kBGateCap * sizeof(GateRun);
constexpr size_t kStage = 2 * kStTs + kStRec + kStGrun;
static_assert(kStage % 16 == 0, "stage alignment");

constexpr size_t kBHist = (size_t)kBandMaxCycles * 16;
constexpr size_t kBSlots = (size_t)kBGateCap * sizeof(BSlot);
constexpr size_t kBTag = (size_t)kBTileCap * 2;
constexpr size_t kBGates = (size_t)kBGateCap * 4;
constexpr size_t kBCells = (size_t)kSmemCells * sizeof(CellDesc);
constexpr size_t kBSmem = kBHist + 2 * kStage + kBSlots + kBTag + kBGates + kBCells;
static_assert(kBSmem <= 227 * 1024, "shared memory budget");

constexpr uint32_t kWaitLimit = 1u << 24;  // mbarrier polls before giving up

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

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
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

__device__ __forceinline__ int lb_f(const float* a, int n, float x) {
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

struct BCtx {
  float* W;
  float* D;
  uint32_t* EV;
  uint32_t* GL;
  uint16_t* tag;
  BSlot* slots;
  uint32_t* sgate;  // gate id per slot (debug outputs)
  const CellDesc* cells;
  uint32_t c0;      // first cycle of the current band
};

// One event of a staged segment (gate state, LUT, switching, glitch, leakage)
// into the shared-memory band histogram.
template <bool kPow2, bool kDebug>
__device__ __forceinline__ void bevent(const BandRunArgs& A, const BCtx& X, const float* __restrict__ ts,
                                       const float* __restrict__ ss, int si, int p, int e, bool hp0, float pt0,
                                       float ps0, BAcc& acc) {
  const RunArgs& a = A.r;
  const BSlot& S = X.slots[si];
  const int a0 = S.st[p];
  const int idx = e - a0;
  if (idx >= (int)S.len[p]) return;
  const float t = ts[e], s = ss[e];
  const uint32_t c = cyc<kPow2>(t, a.t_clk, a.inv_t_clk);
  bool has_prev = hp0;
  float tp = pt0, sp = ps0;
  if (idx > 0) {
    has_prev = true;
    tp = ts[e - 1];
    sp = ss[e - 1];
  }
  const bool glitch = has_prev && cyc<kPow2>(tp, a.t_clk, a.inv_t_clk) == c;
  const uint32_t kj = S.kj;
  const int k = (int)(kj & 15u);
  float e_int = 0.f, e_sw = 0.f, dp = 0.f;
  uint32_t s_pre = S.state;
  int li = 0;
  if (p == k) {
    e_sw = S.esw;
    if (kDebug) {
      for (int q = 0; q < k; ++q) s_pre ^= ((uint32_t)lb_f(ts + S.st[q], S.len[q], t) & 1u) << q;
    }
  } else {
    const CellDesc& cd = X.cells[S.cell];
    s_pre ^= ((uint32_t)idx & 1u) << p;
    uint32_t s_b = s_pre;
    for (int q = 0; q < k; ++q) {
      if (q == p) continue;
      const int qa = S.st[q], qn = S.len[q];
      const int r = lb_f(ts + qa, qn, t);
      const uint32_t par = (uint32_t)r & 1u;
      s_pre ^= par << q;
      const bool eq = q < p && r < qn && ts[qa + r] == t;
      s_b ^= (par ^ (uint32_t)eq) << q;
    }
    // slew interval: largest i <= ns - 2 with axis[i] <= s (axes have <= 8 points)
    const int ns = cd.ns, nl = cd.nl;
    {
      const int hi = ns - 2;
      int w = 4;
      while (w > 0) {
        const int cand = li + w;
        if (cand <= hi && s >= cd.sax[cand]) li = cand;
        w >>= 1;
      }
    }
    const float u = (s - cd.sax[li]) * cd.isax[li];
    const float* L = a.lut + cd.lut_off + ((int)s_pre * ns + li) * nl + (int)(kj >> 4);
    const float l00 = __ldg(L), l01 = __ldg(L + 1), l10 = __ldg(L + nl), l11 = __ldg(L + nl + 1);
    const float v = S.v;
    const float r0 = fmaf(v, l01 - l00, l00), r1 = fmaf(v, l11 - l10, l10);
    e_int = fmaf(u, r1 - r0, r0);
    const float* lk = a.leak + cd.leak_off;
    dp = __ldg(lk + (s_b ^ (1u << p))) - __ldg(lk + s_b);
  }
  const float e_dyn = e_int + e_sw;
  float e_w;
  if (glitch) {
    const float r = fminf(1.f, 2000.f * (t - tp) / (s + sp));
    e_w = r * e_dyn;
    acc.e_gl += e_w;
  } else {
    acc.e_int += e_int;
    acc.e_sw += e_sw;
    e_w = e_dyn;
  }
  const uint32_t lc = c - X.c0;
  if (lc >= A.L.band_cycles) {  // an event outside its band: layout inconsistency
    berr(a.err, e, kErrTileOverflow);
    return;
  }
  if (p < k) {
    const float rem = fmaf(-(float)c, a.t_clk, t);  // t - c T
    e_w = fmaf(dp, a.t_clk - rem, e_w);
    acc.e_lk = fmaf(dp, a.t_max_f - t, acc.e_lk);
    atomicAdd(X.D + lc, dp);
  }
  atomicAdd(X.W + lc, e_w);
  atomicAdd(X.EV + lc, 1u);
  if (glitch) atomicAdd(X.GL + lc, 1u);
  if (kDebug) {
    // original (CSR) index of this event: its rank among the pin's events
    const GateRec r = a.gates[X.sgate[si]];
    const uint64_t pin = (uint64_t)r.pin_base + p;
    const uint64_t lo = a.pin_off[pin], hi = a.pin_off[pin + 1];
    uint64_t l = lo, n = hi - lo;
    while (n > 0) {
      const uint64_t half = n >> 1;
      if (a.t[l + half] < t) {
        l += half + 1;
        n -= half + 1;
      } else {
        n = half;
      }
    }
    a.dbg_state[l] = (uint8_t)s_pre;
    a.dbg_lut[l] = p < k ? (uint8_t)((li << 4) | (int)(kj >> 4)) : (uint8_t)0xFF;
    a.dbg_glitch[l] = (uint8_t)glitch;
  }
}

__device__ __forceinline__ void bflush_acc(BAcc& acc, double* s_tot) {
  float v[4] = {acc.e_int, acc.e_sw, acc.e_gl, acc.e_lk};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
  }
  if ((threadIdx.x & 31) == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) atomicAdd(s_tot + i, (double)v[i]);
  }
  acc = BAcc{0.f, 0.f, 0.f, 0.f};
}

// Add the band's shared-memory bins to the global fp64 / u32 bins and clear them.
__device__ void bflush_band(const BandRunArgs& A, const BCtx& X, uint32_t band) {
  const uint32_t cb = A.L.band_cycles, N = A.r.n_cycles;
  double* bins = reinterpret_cast<double*>(A.r.bins);
  for (uint32_t lc = threadIdx.x; lc < cb; lc += kBThreads) {
    const uint32_t c = band * cb + lc;
    const float w = X.W[lc], d = X.D[lc];
    const uint32_t ev = X.EV[lc], gl = X.GL[lc];
    if (c < N) {
      if (w != 0.f) atomicAdd(bins + 2 * (uint64_t)c, (double)w);
      if (d != 0.f) atomicAdd(bins + 2 * (uint64_t)c + 1, (double)d);
      if (ev) atomicAdd(A.r.cnt_ev + c, ev);
      if (gl) atomicAdd(A.r.cnt_gl + c, gl);
    }
    X.W[lc] = 0.f;
    X.D[lc] = 0.f;
    X.EV[lc] = 0u;
    X.GL[lc] = 0u;
  }
}

__device__ __forceinline__ void bslot_from(BSlot& S, const GateRun& gr, uint32_t state) {
  S.kj = (uint8_t)(((gr.packed >> 16) & 15u) | (((gr.packed >> 20) & 15u) << 4));
  S.state = (uint8_t)state;
  S.cell = (uint16_t)(gr.packed & 0xffffu);
  S.v = gr.v;
  S.esw = gr.esw;
}

// Thread 0: stage item `i` into stage buffer `stage` (TMA bulk copies).
__device__ void bprefetch(const BandRunArgs& A, uint32_t i, uint8_t* stage, StageMeta& meta, uint64_t* bar) {
  const BandItem it = A.items[i];
  meta.it = it;
  meta.ev_off = 0;
  meta.rec_off = 0;
  if (it.kind == 2) {  // streamed: nothing staged
    mbar_expect_arrive(bar, 0);
    return;
  }
  float* ts = reinterpret_cast<float*>(stage);
  float* ss = reinterpret_cast<float*>(stage + kStTs);
  uint8_t* rec = stage + 2 * kStTs;
  uint8_t* grun = rec + kStRec;
  const bool light = it.kind == 0;
  const uint32_t u0 = light ? it.first * kLightBlock : it.first;
  const uint32_t u1 = light ? min(it.last * (uint32_t)kLightBlock, A.L.n_light) : it.last;
  const uint32_t nu = u1 - u0;
  if (it.n > (uint32_t)kBTileCap || nu > (uint32_t)kBGateCap || u1 < u0) {  // never stage past a buffer
    meta.it.kind = 3;
    mbar_expect_arrive(bar, 0);
    return;
  }
  const uint64_t ea = it.e0 & ~3ull;
  const uint32_t ev_off = (uint32_t)(it.e0 - ea);
  const uint32_t ev_bytes = it.n ? ((ev_off + it.n + 3u) & ~3u) * 4u : 0u;
  uint32_t rec_bytes = 0, rec_off = 0;
  const void* rec_src = nullptr;
  if (light) {
    const uint64_t rb = (uint64_t)it.band * A.L.n_light + u0;
    const uint64_t ra = rb & ~3ull;
    rec_off = (uint32_t)(rb - ra);
    rec_bytes = nu ? ((rec_off + nu + 3u) & ~3u) * 4u : 0u;
    rec_src = A.L.lrec + ra;
  } else {
    rec_bytes = nu * (uint32_t)sizeof(HeavyRec);
    rec_src = A.L.hrec + (uint64_t)it.band * A.L.n_heavy + u0;
  }
  const uint32_t g_bytes = nu * (uint32_t)sizeof(GateRun);
  const void* g_src = (light ? A.grun_l : A.grun_h) + u0;
  meta.ev_off = ev_off;
  meta.rec_off = rec_off;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_arrive(bar, 2 * ev_bytes + rec_bytes + g_bytes);
  if (ev_bytes) {
    bulk_g2s(ts, A.L.bt + ea, ev_bytes, bar);
    bulk_g2s(ss, A.L.bs + ea, ev_bytes, bar);
  }
  if (rec_bytes) bulk_g2s(rec, rec_src, rec_bytes, bar);
  if (g_bytes) bulk_g2s(grun, g_src, g_bytes, bar);
}

}  // namespace

namespace {

template <bool kPow2, bool kDebug>
__global__ void __launch_bounds__(kBThreads, 1) k_banded(const BandRunArgs A, uint32_t n_items) {
  extern __shared__ __align__(128) uint8_t smem[];
  BCtx X;
  const uint32_t cb = A.L.band_cycles;
  X.W = reinterpret_cast<float*>(smem);
  X.D = X.W + kBandMaxCycles;
  X.EV = reinterpret_cast<uint32_t*>(X.D + kBandMaxCycles);
  X.GL = X.EV + kBandMaxCycles;
  uint8_t* stages = smem + kBHist;
  X.slots = reinterpret_cast<BSlot*>(stages + 2 * kStage);
  X.tag = reinterpret_cast<uint16_t*>(stages + 2 * kStage + kBSlots);
  X.sgate = reinterpret_cast<uint32_t*>(stages + 2 * kStage + kBSlots + kBTag);
  CellDesc* cells_s = reinterpret_cast<CellDesc*>(stages + 2 * kStage + kBSlots + kBTag + kBGates);
  __shared__ __align__(8) uint64_t s_bar[2];
  __shared__ StageMeta s_meta[2];
  __shared__ BStream hs;
  __shared__ double s_tot[4];
  __shared__ uint32_t s_range[2];
  __shared__ uint32_t s_wsum[kBWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RunArgs& a = A.r;

  if (tid < 4) s_tot[tid] = 0.0;
  const bool cells_in_smem = a.n_cells <= (uint32_t)kSmemCells;
  if (cells_in_smem) {
    const int words = (int)(a.n_cells * sizeof(CellDesc) / 4);
    const uint32_t* src = reinterpret_cast<const uint32_t*>(a.cells);
    uint32_t* dst = reinterpret_cast<uint32_t*>(cells_s);
    for (int i = tid; i < words; i += kBThreads) dst[i] = src[i];
  }
  X.cells = cells_in_smem ? cells_s : a.cells;
  for (uint32_t i = tid; i < cb; i += kBThreads) {
    X.W[i] = 0.f;
    X.D[i] = 0.f;
    X.EV[i] = 0u;
    X.GL[i] = 0u;
  }
  if (tid < 2) {
    // items whose first event falls in this CTA's share of all events
    const uint64_t total = A.item_ev[n_items];
    const uint64_t want = total * (uint64_t)(blockIdx.x + tid) / gridDim.x;
    uint32_t lo = 0, n = n_items;
    while (n > 0) {
      const uint32_t half = n >> 1;
      if (A.item_ev[lo + half] < want) {
        lo += half + 1;
        n -= half + 1;
      } else {
        n = half;
      }
    }
    s_range[tid] = (blockIdx.x + tid == gridDim.x) ? n_items : lo;
  }
  if (tid == 0) {
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const uint32_t i0 = s_range[0], i1 = s_range[1];
  if (tid == 0 && i0 < i1) bprefetch(A, i0, stages, s_meta[0], &s_bar[0]);
  uint32_t band = 0xFFFFFFFFu;
  BAcc acc{0.f, 0.f, 0.f, 0.f};
  int since_flush = 0;

  for (uint32_t item = i0; item < i1; ++item) {
    const uint32_t q = item - i0, st = q & 1u;
    if (tid == 0 && item + 1 < i1)  // the other stage was released by the barrier ending item - 1
      bprefetch(A, item + 1, stages + (st ^ 1u) * kStage, s_meta[st ^ 1u], &s_bar[st ^ 1u]);
    bool ok = false;
    for (uint32_t it = 0; it < kWaitLimit && !ok; ++it) ok = mbar_try_wait(&s_bar[st], (q >> 1) & 1u);
    if (__syncthreads_or(!ok)) {  // a staged copy never landed: report and stop this CTA
      if (tid == 0) {
        berr(a.err, item, kErrTileOverflow);
        if (item + 1 < i1) {  // let our own prefetch of the next item land (bounded) before leaving
          bool done = false;
          for (uint32_t it = 0; it < kWaitLimit && !done; ++it)
            done = mbar_try_wait(&s_bar[st ^ 1u], ((q + 1) >> 1) & 1u);
        }
      }
      return;
    }
    const StageMeta M = s_meta[st];
    const BandItem it = M.it;
    uint8_t* stage = stages + st * kStage;
    const float* ts = reinterpret_cast<const float*>(stage) + M.ev_off;
    const float* ss = reinterpret_cast<const float*>(stage + kStTs) + M.ev_off;
    if (it.band != band) {
      if (band != 0xFFFFFFFFu) bflush_band(A, X, band);
      band = it.band;
      X.c0 = band * cb;
      __syncthreads();
    }
    if (it.kind == 3) {  // refused by the prefetch bounds check
      if (tid == 0) berr(a.err, item, kErrTileOverflow);
      __syncthreads();
      continue;
    }
    if (it.kind == 0 || it.kind == 1) {
      // ---------------- a tile of whole units (light gates or small heavy units)
      const bool light = it.kind == 0;
      const uint32_t u0 = light ? it.first * kLightBlock : it.first;
      const uint32_t u1 = light ? min(it.last * (uint32_t)kLightBlock, A.L.n_light) : it.last;
      const uint32_t ng = u1 - u0;
      const uint32_t n = it.n;
      if (n > (uint32_t)kBTileCap || ng > (uint32_t)kBGateCap) {
        if (tid == 0) berr(a.err, item, kErrTileOverflow);
        __syncthreads();
        continue;
      }
      const uint8_t* rec = stage + 2 * kStTs;
      const GateRun* grun = reinterpret_cast<const GateRun*>(rec + kStRec);
      uint32_t c5 = 0, state = 0, tot = 0;
      uint32_t hc[5] = {0, 0, 0, 0, 0};  // events of each pin of this thread's unit
      if ((uint32_t)tid < ng) {
        if (light) {
          c5 = reinterpret_cast<const uint32_t*>(rec)[M.rec_off + tid];
          state = c5 >> 25;
#pragma unroll
          for (int p = 0; p < 5; ++p) hc[p] = (c5 >> (5 * p)) & 31u;
        } else {
          const HeavyRec& hr = reinterpret_cast<const HeavyRec*>(rec)[tid];
#pragma unroll
          for (int p = 0; p < 5; ++p) hc[p] = hr.cnt[p];
          state = hr.state;
        }
#pragma unroll
        for (int p = 0; p < 5; ++p) tot += hc[p];
      }
      uint32_t inc = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t nn = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += nn;
      }
      if (lane == 31) s_wsum[warp] = inc;
      __syncthreads();
      uint32_t off = inc - tot;
      for (int w = 0; w < warp; ++w) off += s_wsum[w];
      if ((uint32_t)tid < ng) {
        const GateRun gr = grun[tid];
        BSlot S;
        bslot_from(S, gr, state);
        uint32_t pos = off;
#pragma unroll
        for (int p = 0; p < 5; ++p) {
          S.st[p] = (uint16_t)pos;
          S.len[p] = (uint16_t)hc[p];
          pos += hc[p];
        }
        X.slots[tid] = S;
        X.sgate[tid] = gr.gate;
      }
      __syncthreads();
      for (uint32_t gi = warp; gi < ng; gi += kBWarps) {
        const BSlot& S = X.slots[gi];
        const int k = S.kj & 15;
        const int b0 = S.st[0], b1 = S.st[k] + S.len[k];
        for (int e = b0 + lane; e < b1; e += 32) {
          int p = 0;
          for (int qq = 1; qq <= k; ++qq) p += (e >= (int)S.st[qq]) ? 1 : 0;
          X.tag[e] = (uint16_t)((gi << 3) | (uint32_t)p);
        }
      }
      __syncthreads();
      for (uint32_t e = tid; e < n; e += kBThreads) {
        const uint32_t tg = X.tag[e];
        bevent<kPow2, kDebug>(A, X, ts, ss, (int)(tg >> 3), (int)(tg & 7u), (int)e, false, 0.f, 0.f, acc);
      }
      __syncthreads();
    } else {
      // ---------------- one big heavy unit: stream it in event-count windows
      float* wts = reinterpret_cast<float*>(stage);
      float* wss = reinterpret_cast<float*>(stage + kStTs);
      const HeavyRec hr = A.L.hrec[(uint64_t)band * A.L.n_heavy + it.first];
      const GateRun gr = A.grun_h[it.first];
      const int k = (int)((gr.packed >> 16) & 15u);
      if (tid == 0) {
        bslot_from(X.slots[0], gr, hr.state);
        X.sgate[0] = gr.gate;
        uint64_t pos = hr.base;
        for (int p = 0; p <= k; ++p) {
          hs.cur[p] = pos;
          hs.end[p] = pos + hr.cnt[p];
          pos += hr.cnt[p];
          hs.has_prev[p] = 0;
          hs.prev_t[p] = 0.f;
          hs.prev_s[p] = 0.f;
        }
        hs.pre = 0;
        hs.done = 0;
      }
      __syncthreads();
      for (;;) {
        BSlot& S = X.slots[0];
        if (tid == 0) {
          uint64_t R = 0;
          for (int p = 0; p <= k; ++p) R += hs.end[p] - hs.cur[p];
          if (R == 0) {
            hs.done = 1;
          } else {
            const uint64_t budget = (uint64_t)(kBTileCap - (k + 1));
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
              S.len[p] = (uint16_t)ap;
              pos += (uint32_t)ap;
            }
            for (int p = k + 1; p < 5; ++p) {
              S.st[p] = (uint16_t)pos;
              S.len[p] = 0;
            }
            // the window's state: band-start state flipped per event already processed
            S.state = (uint8_t)((hr.state ^ hs.pre) & ((1u << k) - 1u));  // input pins only
          }
        }
        __syncthreads();
        if (hs.done) break;
        if (tid <= k) {
          const uint64_t nx = hs.cur[tid] + S.len[tid];
          hs.bound[tid] = nx < hs.end[tid] ? A.L.bt[nx] : FLT_MAX;
        }
        const int nw = S.st[k] + S.len[k];
        for (int i = tid; i < nw; i += kBThreads) {
          int p = 0;
          for (int qq = 1; qq <= k; ++qq) p += (i >= (int)S.st[qq]) ? 1 : 0;
          const uint64_t ge = hs.cur[p] + (uint64_t)(i - (int)S.st[p]);
          wts[i] = A.L.bt[ge];
          wss[i] = A.L.bs[ge];
          X.tag[i] = (uint16_t)p;
        }
        __syncthreads();
        if (tid <= k) {
          float tau = FLT_MAX;
          for (int qq = 0; qq <= k; ++qq) tau = fminf(tau, hs.bound[qq]);
          // events at or after the horizon wait for the next window; a
          // timestamp group is never split
          if (tau != FLT_MAX) S.len[tid] = (uint16_t)lb_f(wts + S.st[tid], S.len[tid], tau);
        }
        __syncthreads();
        for (int i = tid; i < nw; i += kBThreads) {
          const int p = X.tag[i];
          bevent<kPow2, kDebug>(A, X, wts, wss, 0, p, i, hs.has_prev[p] != 0, hs.prev_t[p], hs.prev_s[p], acc);
        }
        __syncthreads();
        if (tid == 0) {
          uint32_t moved = 0;
          for (int p = 0; p <= k; ++p) {
            const uint32_t m = S.len[p];
            if (m > 0) {
              hs.prev_t[p] = wts[S.st[p] + m - 1];
              hs.prev_s[p] = wss[S.st[p] + m - 1];
              hs.has_prev[p] = 1;
              hs.cur[p] += m;
              hs.pre ^= (uint8_t)((m & 1u) << p);
              moved += m;
            }
          }
          if (moved == 0) {  // cannot happen for valid input; never spin
            berr(a.err, item, kErrTileOverflow);
            hs.done = 1;
          }
        }
        __syncthreads();
        if (hs.done) break;
      }
      __syncthreads();
    }
    if (++since_flush >= 16) {
      bflush_acc(acc, s_tot);
      since_flush = 0;
    }
  }
  bflush_acc(acc, s_tot);
  __syncthreads();
  if (band != 0xFFFFFFFFu) bflush_band(A, X, band);
  __syncthreads();
  if (tid < 4) atomicAdd(a.totals + tid, s_tot[tid]);
}

template <bool P, bool D>
void launch_banded(const BandRunArgs& A, uint32_t n_items, int grid, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(k_banded<P, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBSmem);
    attr = true;
  }
  k_banded<P, D><<<grid, kBThreads, kBSmem, st>>>(A, n_items);
}

}  // namespace

cudaError_t band_fused(BandRunArgs& A, uint32_t n_items, int sm_count, bool debug, cudaStream_t st) {
  if (n_items == 0) return cudaSuccess;
  const bool pow2 = A.r.inv_t_clk != 0.f;
  const int grid = sm_count;
  if (pow2 && debug) launch_banded<true, true>(A, n_items, grid, st);
  else if (pow2) launch_banded<true, false>(A, n_items, grid, st);
  else if (debug) launch_banded<false, true>(A, n_items, grid, st);
  else launch_banded<false, false>(A, n_items, grid, st);
  return cudaGetLastError();
}

}  // namespace pa
