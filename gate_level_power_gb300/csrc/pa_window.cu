// The paper's own work decomposition as a selectable partition of libpa.so
// (sm_103a): one thread per (gate g, window of n_cyc^(g) whole cycles), as in
// the event-density-aware per-gate cycle partitioning of "GPU-Accelerated
// Gate-Level Time-Based Power Analysis via Event-Density-Aware Partitioning and
// Kernel Fusion" (Fig. 5) and the globally fixed partition it is compared with
// (Figs. 19 and 20). It computes the same results as the other two kernels; it
// exists to time the two partitions against each other on this GPU and to
// report their thread statistics (thread count, events per thread).
//
//  * Plan (one thread per gate): rho = N_evt / N_cyc, n_cyc,floor =
//    ceil(N_cyc / N_thr,floor), rho_floor = n_evt,tgt / n_cyc,floor, n_cyc =
//    floor(n_evt,tgt / (rho + rho_floor) + 1/2) clamped to [1, N_cyc], all in
//    fp64 (the additive effective density of the text); or n_cyc = n_cyc^fix
//    for every gate. Threads per gate ceil(N_cyc / n_cyc), scanned into the
//    first thread of each gate.
//  * Window kernel: CTAs (as many as fit the GPU) take chunks of 256 thread
//    ids in grid-stride order; a chunk's ids map to (gate, window) with one
//    32-way search of the scanned offsets and a search in shared memory. Each
//    thread finds, per pin, the events whose cycle floor(fl32(t / T)) lies in
//    its window, then walks them in (time, pin) order: a serial k-way merge
//    that carries the gate state (the state before a timestamp selects the LUT;
//    leakage steps are taken event by event in (time, pin) order, so a
//    timestamp group telescopes), the glitch test against the pin's previous
//    event (windows start on cycle boundaries, so a window's first event on a
//    pin never is a glitch), and one 16-byte global reduction per event into
//    the cycle bins {W, D, ev, gl} -- the per-event atomic of the paper's
//    kernel. Leakage uses the same per-event step formulation as the other
//    kernels (no per-cycle loop).

#include "pa_internal.cuh"

namespace pa {

namespace {

constexpr int kWT = 256;           // threads per CTA of the window kernel
constexpr int kWinHistSmem = 256;  // events-per-thread histogram bins kept in shared memory
constexpr int kWinFold = 32;       // events between folds of a thread's f32 sums into fp64

template <bool kPow2>
__device__ __forceinline__ uint32_t wcyc(float t, float T, float inv_T) {
  // floor(fl32(t / T)) for t >= 0; with T a power of two t * (1/T) is the
  // same correctly rounded quotient
  if (kPow2) return (uint32_t)(t * inv_T);
  return (uint32_t)__fdiv_rn(t, T);
}

// First index in [lo, hi) of a pin's time-ordered events whose cycle is >= c.
template <bool kPow2>
__device__ __forceinline__ uint64_t first_in_cycle(const float* __restrict__ t, uint64_t lo, uint64_t hi, uint32_t c,
                                                   float T, float inv_T) {
  uint64_t n = hi - lo;
  while (n > 0) {
    const uint64_t h = n >> 1;
    if (wcyc<kPow2>(__ldg(t + lo + h), T, inv_T) < c) {
      lo += h + 1;
      n -= h + 1;
    } else {
      n = h;
    }
  }
  return lo;
}

// The same from a start known to be at or before the answer, by galloping
// (a window holds few events, so its end is near its start).
template <bool kPow2>
__device__ __forceinline__ uint64_t first_in_cycle_from(const float* __restrict__ t, uint64_t lo, uint64_t hi,
                                                        uint32_t c, float T, float inv_T) {
  uint64_t step = 1, prev = lo;
  while (lo < hi && wcyc<kPow2>(__ldg(t + lo), T, inv_T) < c) {
    prev = lo + 1;
    lo = (hi - lo > step) ? lo + step : hi;
    step <<= 1;
  }
  return first_in_cycle<kPow2>(t, prev, lo, c, T, inv_T);
}

__global__ void __launch_bounds__(256) k_win_plan(const RunArgs a, const WinArgs w) {
  const uint32_t g = blockIdx.x * 256u + threadIdx.x;
  if (g >= a.n_gates) return;
  const uint32_t N = a.n_cycles;
  const uint64_t n_evt = a.gate_off[g + 1] - a.gate_off[g];
  // a thread's per-pin cursors are 32-bit offsets into its gate's events
  if (n_evt >> 32) atomicMin(a.err, (unsigned long long)(((uint64_t)g << 8) | kErrTileOverflow));
  uint64_t n;
  if (w.mode == PA_PART_FIXED) {
    n = w.n_cyc_fix;
  } else {
    const uint64_t n_floor = ((uint64_t)N + w.n_thr_floor - 1) / w.n_thr_floor;
    const double rho = (double)n_evt / (double)N;
    const double rho_floor = (double)w.n_evt_tgt / (double)n_floor;
    const double x = (double)w.n_evt_tgt / (rho + rho_floor);
    const double r = floor(x + 0.5);
    n = r >= (double)N ? (uint64_t)N : (uint64_t)r;
  }
  if (n < 1) n = 1;
  if (n > N) n = N;
  w.ncyc[g] = (uint32_t)n;
  w.nthr[g] = (uint32_t)(((uint64_t)N + n - 1) / n);
}

struct WAcc {
  float f[4];   // E_int, E_sw, E_gl, sum dP (t_max - t): the current run of events
  float c3;     // Kahan compensation of f[3] (large terms of either sign that nearly cancel)
  double d[4];  // folded sums
  __device__ __forceinline__ void add_lk(float x) {
    const float y = x - c3;
    const float t = f[3] + y;
    c3 = (t - f[3]) - y;
    f[3] = t;
  }
  __device__ __forceinline__ void fold() {
#pragma unroll
    for (int m = 0; m < 4; ++m) d[m] += (double)f[m];
    d[3] -= (double)c3;
#pragma unroll
    for (int m = 0; m < 4; ++m) f[m] = 0.f;
    c3 = 0.f;
  }
};

// One (gate, window) thread: returns the number of its events.
template <bool kPow2, bool kDebug, bool kExact>
__device__ __forceinline__ uint32_t win_thread(const RunArgs& a, const WinArgs& w, const CellDesc* cells, uint32_t g,
                                               uint32_t tau, WAcc& acc) {
  const GateRec gr = a.gates[g];
  const int k = (int)((gr.init >> 16) & 0xffu);
  const uint32_t N = a.n_cycles;
  const uint32_t n = w.ncyc[g];
  const uint64_t c_lo64 = (uint64_t)tau * n, c_hi64 = c_lo64 + n;
  const uint32_t c_lo = (uint32_t)c_lo64, c_hi = c_hi64 >= N ? N : (uint32_t)c_hi64;
  const float T = a.t_clk, iT = a.inv_t_clk;
  const float* __restrict__ tt = a.t;
  const uint64_t pb = gr.pin_base;
  const uint64_t ebase = a.pin_off[pb];
  // per pin (0..k-1 inputs, k the output): cursor and end, relative to ebase;
  // head time; cycle of the pin's previous event in the window (none: ~0)
  uint32_t cur[kMaxK + 1], end[kMaxK + 1], pcy[kMaxK + 1];
  float ht[kMaxK + 1];
  uint32_t S = gr.init & 0xffu;  // input values: the running state in (time, pin) order
  uint32_t n_ev = 0;
#pragma unroll
  for (int p = 0; p <= kMaxK; ++p) {
    cur[p] = end[p] = 0;
    pcy[p] = 0xffffffffu;
    ht[p] = __int_as_float(0x7f800000);  // +inf: no event
    if (p <= k) {
      const uint64_t a0 = a.pin_off[pb + p], a1 = a.pin_off[pb + p + 1];
      const uint64_t lo = c_lo == 0 ? a0 : first_in_cycle<kPow2>(tt, a0, a1, c_lo, T, iT);
      const uint64_t hi = c_hi == N ? a1 : first_in_cycle_from<kPow2>(tt, lo, a1, c_hi, T, iT);
      cur[p] = (uint32_t)(lo - ebase);
      end[p] = (uint32_t)(hi - ebase);
      if (lo < hi) ht[p] = __ldg(tt + lo);
      if (p < k) S ^= (uint32_t)((lo - a0) & 1u) << p;  // parity of the pin's earlier events
      n_ev += (uint32_t)(hi - lo);
    }
  }
  if (n_ev == 0) return 0;
  const CellDesc& cd = cells[gr.cell];
  const float C = gr.load;
  int j = 0;
  for (int m = 1; m <= cd.nl - 2; ++m) j += (C >= cd.lax[m]) ? 1 : 0;
  const float v = (C - cd.lax[j]) * cd.ilax[j];
  const float esw = a.half_vdd2 * C;
  const float* lk = a.leak + cd.leak_off;
  const float4* patch = a.patch + cd.patch_off;
  const int ns = cd.ns, nl = cd.nl;
  double ge[4] = {0.0, 0.0, 0.0, 0.0};  // this thread's share of its gate's energies (kDebug)
  float t_grp = -1.f;
  uint32_t S_grp = S;
  for (uint32_t done = 0; done < n_ev; ++done) {
    // next event in (time, pin) order: the lowest pin among the earliest heads
    int p = 0;
    float t = ht[0];
#pragma unroll
    for (int q = 1; q <= kMaxK; ++q) {
      if (ht[q] < t) {
        t = ht[q];
        p = q;
      }
    }
    uint32_t ce = 0, ee = 0, pc = 0;
#pragma unroll
    for (int q = 0; q <= kMaxK; ++q) {
      if (q == p) {
        ce = cur[q];
        ee = end[q];
        pc = pcy[q];
      }
    }
    const uint64_t e = ebase + ce;
    if (t != t_grp) {  // a new timestamp: the LUT state is the state before it
      t_grp = t;
      S_grp = S;
    }
    const float s = __ldg(a.s + e);
    const uint32_t c = wcyc<kPow2>(t, T, iT);
    bool glitch = pc == c;
    bool fwd = false;
    float tp = 0.f, sp = 0.f;
    if (glitch) {
      tp = __ldg(tt + e - 1);
      sp = __ldg(a.s + e - 1);
    }
    // the pin's next event in the window (its cycle is in the window)
    const bool has_next = ce + 1 < ee;
    const float tn = has_next ? __ldg(tt + e + 1) : __int_as_float(0x7f800000);
    if (kDebug && a.glitch_all && !glitch && has_next && wcyc<kPow2>(tn, T, iT) == c) {
      glitch = fwd = true;  // glitch-all reading: the first event of the pin-cycle takes the pulse to the next
      tp = tn;
      sp = __ldg(a.s + e + 1);
    }
    float e_int = 0.f, e_sw = 0.f, dp = 0.f;
    int li = 0;
    if (p == k) {
      e_sw = esw;
      if (kDebug && a.esw_rise) {  // C V^2 on a rise: the output's new value from its initial one and its rank
        const uint64_t rank = e - a.pin_off[pb + k];
        e_sw = ((((gr.init >> 8) & 1u) ^ (uint32_t)((rank + 1) & 1u)) != 0u) ? 2.f * esw : 0.f;
      }
    } else {
      for (int m = 1; m <= ns - 2; ++m) li += (s >= cd.sax[m]) ? 1 : 0;
      const float u = (s - cd.sax[li]) * cd.isax[li];
      const float4 P = __ldg(patch + ((int)S_grp * (ns - 1) + li) * (nl - 1) + j);
      const float r0 = fmaf(v, P.y - P.x, P.x), r1 = fmaf(v, P.w - P.z, P.z);
      e_int = fmaf(u, r1 - r0, r0);
      const uint32_t bit = 1u << p;
      dp = __ldg(lk + (S ^ bit)) - __ldg(lk + S);
      S ^= bit;
    }
    const float e_dyn = e_int + e_sw;
    float e_w;
    if (glitch) {
      const float r = fminf(1.f, 2000.f * (fwd ? tp - t : t - tp) / (s + sp));
      e_w = r * e_dyn;
      acc.f[2] += e_w;
      if (kDebug) ge[2] += (double)e_w;
    } else {
      acc.f[0] += e_int;
      acc.f[1] += e_sw;
      e_w = e_dyn;
      if (kDebug) {
        ge[0] += (double)e_int;
        ge[1] += (double)e_sw;
      }
    }
    if (p < k) {
      const float rem = fmaf(-(float)c, T, t);  // t - c T: the step's part inside its own cycle
      e_w = fmaf(dp, T - rem, e_w);
      acc.add_lk(dp * (a.t_max_f - t));
      if (kDebug) ge[3] += (double)(dp * (a.t_max_f - t));
    }
    if (kExact) {
      double* bin = reinterpret_cast<double*>(a.bins + c);
      atomicAdd(bin, (double)e_w);
      if (p < k) atomicAdd(bin + 1, (double)dp);
      atomicAdd(a.cnt_ev + c, 1u);
      if (glitch) atomicAdd(a.cnt_gl + c, 1u);
    } else {
      float* bin = reinterpret_cast<float*>(a.bins + c);
      asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(bin), "f"(e_w), "f"(dp), "f"(1.0f),
                   "f"(glitch ? 1.0f : 0.0f)
                   : "memory");
    }
    if (kDebug) {
      if (a.dbg_state) a.dbg_state[e] = (uint8_t)S_grp;
      if (a.dbg_lut) a.dbg_lut[e] = p < k ? (uint8_t)((li << 4) | j) : (uint8_t)0xFF;
      if (a.dbg_glitch) a.dbg_glitch[e] = (uint8_t)glitch;
    }
    // advance pin p
#pragma unroll
    for (int q = 0; q <= kMaxK; ++q) {
      if (q == p) {
        cur[q] = ce + 1;
        pcy[q] = c;
        ht[q] = tn;
      }
    }
    if ((done & (kWinFold - 1)) == kWinFold - 1) acc.fold();
  }
  if (kDebug && a.gate_e) {
    double* gp = a.gate_e + (size_t)g * 4;
#pragma unroll
    for (int m = 0; m < 4; ++m)
      if (ge[m] != 0.0) atomicAdd(gp + m, ge[m]);
  }
  return n_ev;
}

template <bool kPow2, bool kDebug, bool kExact>
__global__ void __launch_bounds__(kWT, 3) k_window(const RunArgs a, const WinArgs w) {
  __shared__ CellDesc cells_s[kSmemCells];
  __shared__ uint64_t s_off[kWT + 1];
  __shared__ uint32_t s_g0;
  __shared__ double s_tot[4];
  __shared__ uint32_t s_hist[kWinHistSmem];
  const int tid = threadIdx.x, lane = tid & 31;
  const bool cells_in_smem = a.n_cells <= (uint32_t)kSmemCells;
  if (cells_in_smem) {
    for (uint32_t i = tid; i < a.n_cells; i += kWT) cells_s[i] = a.cells[i];
  }
  const CellDesc* cells = cells_in_smem ? cells_s : a.cells;
  const uint32_t G = a.n_gates;
  const uint64_t total = w.thr_off[G];
  const uint64_t n_chunks = (total + kWT - 1) / kWT;  // CTAs take chunks of kWT thread ids, grid-strided
  WAcc acc;
  acc.c3 = 0.f;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    acc.f[m] = 0.f;
    acc.d[m] = 0.0;
  }
  if (tid < 4) s_tot[tid] = 0.0;
  for (uint64_t chunk = blockIdx.x; chunk < n_chunks; chunk += gridDim.x) {
    const uint64_t base = chunk * kWT;
    if (w.hist) {
      for (int i = tid; i < kWinHistSmem; i += kWT) s_hist[i] = 0u;
    }
    if (tid < 32) {
      // the gate of thread `base`: largest g with thr_off[g] <= base, by a
      // 32-way search (thr_off is strictly increasing: every gate has a thread)
      uint32_t lo = 0, hi = G;  // thr_off[lo] <= base < thr_off[hi]
      while (hi - lo > 1) {
        const uint32_t step = (hi - lo + 31u) / 32u;
        const uint64_t pos = (uint64_t)lo + (uint64_t)(lane + 1) * step;
        const bool le = pos < hi && w.thr_off[pos] <= base;
        const uint32_t cnt = __popc(__ballot_sync(0xffffffffu, le));
        const uint32_t nlo = lo + cnt * step;
        const uint64_t nhi = (uint64_t)lo + (uint64_t)(cnt + 1) * step;
        lo = nlo;
        hi = nhi < hi ? (uint32_t)nhi : hi;
      }
      if (lane == 0) s_g0 = lo;
    }
    __syncthreads();
    const uint32_t g0 = s_g0;
    for (int i = tid; i <= kWT; i += kWT) {
      const uint64_t gi = (uint64_t)g0 + i;
      s_off[i] = w.thr_off[gi < G ? gi : G];
    }
    __syncthreads();
    const uint64_t id = base + tid;
    uint32_t ne = 0;
    if (id < total) {
      // largest i with s_off[i] <= id (the CTA's 256 ids span at most 256 gates)
      int lo = 0, n = kWT + 1;
      while (n > 1) {
        const int h = n >> 1;
        if (s_off[lo + h] <= id) {
          lo += h;
          n -= h;
        } else {
          n = h;
        }
      }
      const uint32_t g = g0 + (uint32_t)lo;
      const uint32_t tau = (uint32_t)(id - s_off[lo]);
      ne = win_thread<kPow2, kDebug, kExact>(a, w, cells, g, tau, acc);
    }
    if (w.hist) {  // thread statistics: events per thread
      if (id < total) {
        if (ne < (uint32_t)kWinHistSmem) {
          atomicAdd(&s_hist[ne], 1u);
        } else {
          atomicAdd(w.hist + (ne < kWinHistBins ? ne : kWinHistBins - 1u), 1ull);
        }
      }
      const uint32_t mx = __reduce_max_sync(0xffffffffu, ne);
      if (lane == 0 && mx) atomicMax(w.ev_max, mx);
      __syncthreads();
      for (int i = tid; i < kWinHistSmem; i += kWT)
        if (s_hist[i]) atomicAdd(w.hist + i, (unsigned long long)s_hist[i]);
    }
    __syncthreads();  // s_g0 / s_off / s_hist are rewritten by the next chunk
  }
  acc.fold();
  double v[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    v[m] = acc.d[m];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[m] += __shfl_xor_sync(0xffffffffu, v[m], o);
  }
  if (lane == 0) {
#pragma unroll
    for (int m = 0; m < 4; ++m)
      if (v[m] != 0.0) atomicAdd(&s_tot[m], v[m]);
  }
  __syncthreads();
  if (tid < 4 && s_tot[tid] != 0.0) atomicAdd(w.tot_slots + (blockIdx.x % kWinTotSlots) * 4 + tid, s_tot[tid]);
}

// Folds the window kernel's total slots into the run's totals.
__global__ void __launch_bounds__(kWinTotSlots) k_win_totals(const RunArgs a, const WinArgs w) {
  __shared__ double s[4][kWinTotSlots];
  const int i = threadIdx.x;
#pragma unroll
  for (int m = 0; m < 4; ++m) s[m][i] = w.tot_slots[i * 4 + m];
  __syncthreads();
  for (int h = kWinTotSlots / 2; h > 0; h >>= 1) {
    if (i < h) {
#pragma unroll
      for (int m = 0; m < 4; ++m) s[m][i] += s[m][i + h];
    }
    __syncthreads();
  }
  if (i < 4) a.totals[i] += s[i][0];
}

template <bool P, bool D, bool X>
void launch_window_of(const RunArgs& a, const WinArgs& w, int grid, cudaStream_t st) {
  k_window<P, D, X><<<grid, kWT, 0, st>>>(a, w);
}

template <bool P, bool D, bool X>
int window_occupancy_of() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_window<P, D, X>, kWT, 0) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

}  // namespace

int window_blocks_per_sm(bool pow2, bool debug, bool exact) {
  const int sel = (pow2 ? 4 : 0) | (debug ? 2 : 0) | (exact ? 1 : 0);
  switch (sel) {
    case 0: return window_occupancy_of<false, false, false>();
    case 1: return window_occupancy_of<false, false, true>();
    case 2: return window_occupancy_of<false, true, false>();
    case 3: return window_occupancy_of<false, true, true>();
    case 4: return window_occupancy_of<true, false, false>();
    case 5: return window_occupancy_of<true, false, true>();
    case 6: return window_occupancy_of<true, true, false>();
    default: return window_occupancy_of<true, true, true>();
  }
}

cudaError_t launch_window_plan(const RunArgs& a, const WinArgs& w, cudaStream_t st) {
  if (a.n_gates) {
    k_win_plan<<<(a.n_gates + 255) / 256, 256, 0, st>>>(a, w);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return scan_u32_to_u64(w.nthr, a.n_gates, w.scan_blk, w.thr_off, st);
}

cudaError_t launch_window(const RunArgs& a, const WinArgs& w, int grid, bool pow2, bool debug, bool exact,
                          cudaStream_t st) {
  const int sel = (pow2 ? 4 : 0) | (debug ? 2 : 0) | (exact ? 1 : 0);
  switch (sel) {
    case 0: launch_window_of<false, false, false>(a, w, grid, st); break;
    case 1: launch_window_of<false, false, true>(a, w, grid, st); break;
    case 2: launch_window_of<false, true, false>(a, w, grid, st); break;
    case 3: launch_window_of<false, true, true>(a, w, grid, st); break;
    case 4: launch_window_of<true, false, false>(a, w, grid, st); break;
    case 5: launch_window_of<true, false, true>(a, w, grid, st); break;
    case 6: launch_window_of<true, true, false>(a, w, grid, st); break;
    default: launch_window_of<true, true, true>(a, w, grid, st); break;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_win_totals<<<1, kWinTotSlots, 0, st>>>(a, w);
  return cudaGetLastError();
}

}  // namespace pa
