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
//    per-gate partitioning of Figs. 5, 19 and 20, cut by event count. The
//    partition also writes what a warp needs to start an item: per light gate
//    its slot (pin starts, cell, load-axis interval and fraction, switching
//    energy), per piece its record (the same gate fields, the pins' starts,
//    the cut points), so an item starts from one coalesced read.
//  * One warp per item, no CTA-wide barrier in the item loop. A light tile's
//    times and slews are one contiguous range, staged with 16-byte copies
//    while a lane per gate loads the gate's slot. A piece is staged in windows of
//    at most kCsrWin events shared among its pins in proportion to their
//    remaining events (16-byte copies per pin run); the events before the
//    earliest first unstaged event of any pin are taken, so every pin's
//    events earlier than a taken event are either staged or counted in the
//    pin's parity.
//  * The gate state before an event's timestamp (ties see the pre-timestamp
//    state; the leakage step is taken in (time, pin) order, so simultaneous
//    steps telescope): in a light tile, one lane per event, each input pin's
//    initial value flipped once per earlier event, the count on another pin
//    being a binary search of t in that pin's staged events. In a piece's
//    window, the input events are walked in (time, pin) order, each lane an
//    even share of the merge of the pins' runs, the state following from the
//    parities of the events taken so far on each pin. The slew interval by a
//    three-step search over the cell's axis in shared memory, the state's four
//    LUT corners in one 16-byte load (a piece: from its gate's slice of the
//    table, copied into shared memory once), the leakage per state in shared
//    memory.
//    Glitch: the previous event of the same pin in the same cycle (the CSR
//    neighbour). Each event adds {energy, leakage step, 1, glitch} to its
//    cycle's bin with one red.global.add.v4.f32, in its warp's copy of the
//    bins (the final reduction adds the copies); per-lane totals (the leakage
//    term compensated) are reduced in fp64.
#include <cfloat>
#include <cstddef>
#include <cstdint>

#include "pa_internal.cuh"

namespace pa {

namespace {

constexpr int kCW = 32;               // warps per CTA (their stages fill the shared memory)
constexpr int kCT = kCW * 32;
constexpr int kStCap = 496;           // staged events per warp: a window, its bounds, the pins' previous events and 16-byte alignment slack
constexpr int kAx = 9;                // slew axis stride of the cell table (odd: lanes of different cells spread)
constexpr int kLk = 17;               // leakage stride of the cell table
constexpr int kTotEvery = 16;         // items between flushes of a warp's per-lane totals
constexpr uint32_t kChunk = 4;        // items a warp takes from the global counter at a time

// Cell tables in shared memory (libraries of at most kSmemCells cells): per
// cell the slew axis points 0..8 (+inf past ns - 2), an info word (ns - 1 |
// (nl - 1) << 8 | patch offset << 16), per slew interval {axis point, 1 /
// width}, and the leakage per state (uW).
constexpr size_t kCellsB =
    (size_t)kSmemCells * kAx * 4 + (size_t)kSmemCells * 4 + (size_t)kSmemCells * 8 * 8 + (size_t)kSmemCells * kLk * 4;

// Per gate of the warp's current item (read by an event as two 16-byte words).
struct __align__(16) CSlot {
  uint16_t st[kMaxK + 2];    // staged start of pins 0..k; st[k + 1] = end
  uint8_t k, init, j, pre;   // inputs, initial input bits, load-axis interval, parity of earlier events per pin
  uint16_t cell, pad;
  float v, esw;              // load-axis fraction; switching energy C V^2 / 2 (fJ)
};
static_assert(sizeof(CSlot) == 32, "slot size");

// Per pin of a piece's current window: the events taken in this window (a
// prefix of the pin's staged run).
struct HWin {
  uint16_t take[kMaxK + 1];
};

// A light tile's map from staged event to (slot, pin): a bit per event that
// starts a pin's run, and per run (the tile's non-empty pins in order) its
// slot << 3 | pin.
constexpr int kSegWords = (kStCap + 31) / 32;
constexpr int kSegMax = kCsrGates * (kMaxK + 1);
struct TSeg {
  uint32_t bits[kSegWords];
  uint8_t run[kSegMax];
};

// A window's pairwise merges of two input pins' runs: per entry the staged
// index, whether the event is on the upper pin of the pair, and the parities
// of both pins' events up to and including it.
constexpr uint32_t kIdxMask = 0x3FFu;
constexpr int kSelShift = 10, kParShift = 11;

// A piece's gate: its LUT corner patches for its load-axis interval, per
// state and slew interval ([2^k][ns - 1] of the cell's [2^k][ns - 1][nl - 1]).
constexpr int kSliceMax = (1 << kMaxK) * (PA_MAX_AXIS - 1);

// One warp's shared memory. A light tile uses all the slots and the run map;
// a piece uses slot 0 and its gate's patch slice in their place.
struct TileMem {
  CSlot slot[kCsrGates];
  TSeg seg;
};
struct PieceMem {
  CSlot slot0;
  float4 slice[kSliceMax];
};
struct __align__(16) WarpBuf {
  float ts[kStCap], ss[kStCap];   // staged times (ns) and slews (ps)
  uint16_t mg[kStCap];            // a window's pairwise merges
  HWin hw;
  union {
    TileMem t;
    PieceMem p;
  } u;
};
static_assert(kCellsB % 16 == 0 && sizeof(WarpBuf) % 16 == 0 && kStCap % 4 == 0 && offsetof(WarpBuf, u) % 16 == 0,
              "alignment");
// a window: shares of at most kCsrWin + one per pin; per pin a bound event
// and at most 7 slots for its previous event (or the late time) and 16-byte
// alignment
static_assert(kCsrWin + 9 * (kMaxK + 1) <= (uint32_t)kStCap && kCsrMaxTileHeavy + 4 <= (uint32_t)kStCap, "stage");
static_assert(kStCap <= (int)kIdxMask + 1, "merge entry index");
constexpr size_t kSmemB = kCellsB + (size_t)kCW * sizeof(WarpBuf);
static_assert(kSmemB + 1024 <= 227 * 1024, "shared memory budget");

struct CTab {
  const float* sax;
  const uint32_t* info;
  const float2* sxp;
  const float* leak;
};

// A lane's totals, and the first bin of its warp's copy of the bins.
struct Acc {
  float e_int, e_sw, e_gl, e_lk, c_lk;
  uint32_t bin0;
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
  acc = Acc{0.f, 0.f, 0.f, 0.f, 0.f, acc.bin0};
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

// Asynchronous global -> shared copies (cp.async: no register round trip, so
// a lane's copies are all in flight at once); each lane waits for its own
// before the warp syncs.
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void copy16_async(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void copies_wait() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Staged start of pin q (0..k + 1) from the slot's first 16 bytes.
__device__ __forceinline__ int st_of(const uint4& A, int q) {
  const uint32_t w = q < 2 ? A.x : (q < 4 ? A.y : A.z);
  return (int)((w >> ((q & 1) * 16)) & 0xFFFFu);
}


// One 16-byte reduction per event into its cycle's bin, in the warp's copy
// of the bins: energy, leakage step, event and glitch counts.
__device__ __forceinline__ void commit(const RunArgs& a, const Acc& acc, uint32_t c, float e_w, float dp,
                                       bool glitch) {
  float* bin = reinterpret_cast<float*>(a.bins + acc.bin0 + c);
  // (nothing in the kernel reads the bins: no memory clobber, so shared
  // memory values need not be reloaded after it)
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(bin), "f"(e_w), "f"(dp), "f"(1.0f),
               "f"(glitch ? 1.0f : 0.0f));
}

// The glitch ratio of an event at t (slew s) whose previous event on the pin
// is at tp (slew sp): r_gl = min(1, x / y), IEEE division; x >= y gives 1
// without dividing.
__device__ __forceinline__ float glitch_ratio(float t, float s, float tp, float sp) {
  const float x = 2000.f * (t - tp), y = s + sp;
  return x < y ? __fdiv_rn(x, y) : 1.f;
}

// An output-pin event at staged index i (has_prev: the pin's previous event
// is at tp, slew *spp).
template <bool kPow2>
__device__ __forceinline__ void out_event(const RunArgs& a, const float* ts, const float* ss, const uint4& B, int i,
                                          bool has_prev, float tp, const float* spp, Acc& acc) {
  const float t = ts[i];
  const float T = a.t_clk;
  const uint32_t c = cyc<kPow2>(t, T, a.inv_t_clk);
  const bool glitch = has_prev && cyc<kPow2>(tp, T, a.inv_t_clk) == c;
  const float e_sw = __uint_as_float(B.z);
  float e_w = e_sw;
  if (glitch) {
    e_w = glitch_ratio(t, ss[i], tp, *spp) * e_sw;
    acc.e_gl += e_w;
  } else {
    acc.e_sw += e_sw;
  }
  commit(a, acc, c, e_w, 0.f, glitch);
}

// An input-pin event at staged index i (time t, held by the caller) of pin p, with its states: s_pre
// before its timestamp (selects the table), s_b just before it in (time, pin)
// order (the leakage step's base).
// The corners come from the gate's patch slice in shared memory in a piece,
// from the global patch table in a light tile.
template <bool kPow2, bool kPiece>
__device__ __forceinline__ void in_event(const RunArgs& a, const CTab& CT, const float4* slice, const float* ss,
                                         const uint4& A, const uint4& B, int i, float t, int p, uint32_t s_pre,
                                         uint32_t s_b, bool has_prev, float tp, const float* spp, Acc& acc) {
  const float s = ss[i];
  const float T = a.t_clk;
  const uint32_t c = cyc<kPow2>(t, T, a.inv_t_clk);
  const bool glitch = has_prev && cyc<kPow2>(tp, T, a.inv_t_clk) == c;
  const uint32_t cell = B.x & 0xFFFFu;
  const uint32_t info = CT.info[cell];  // ns - 1 | (nl - 1) << 8 | patch offset << 16
  // slew interval: the number of axis points 1 .. ns - 2 that are <= s
  const float* axs = CT.sax + cell * kAx;
  int lis = s >= axs[4] ? 4 : 0;
  lis += s >= axs[lis + 2] ? 2 : 0;
  lis += s >= axs[lis + 1] ? 1 : 0;
  const float2 ax = CT.sxp[cell * 8 + lis];
  const float u = (s - ax.x) * ax.y;
  // corners {L[i][j], L[i][j+1], L[i+1][j], L[i+1][j+1]} of the state's table
  const int x = (int)s_pre * (int)(info & 0xFFu) + lis;
  const float4 P = kPiece ? slice[x]
                          : __ldg(a.patch + (info >> 16) + x * (int)((info >> 8) & 0xFFu) + (int)((A.w >> 16) & 0xFFu));
  const float v = __uint_as_float(B.y);
  const float r0 = fmaf(v, P.y - P.x, P.x), r1 = fmaf(v, P.w - P.z, P.z);
  const float e_int = fmaf(u, r1 - r0, r0);
  const float* lk = CT.leak + cell * kLk;
  const float dp = lk[s_b ^ (1u << p)] - lk[s_b];
  float e_w = e_int;
  if (glitch) {
    e_w = glitch_ratio(t, s, tp, *spp) * e_int;
    acc.e_gl += e_w;
  } else {
    acc.e_int += e_int;
  }
  const float rem = fmaf(-(float)c, T, t);  // t - c T: the step's part inside its own cycle
  e_w = fmaf(dp, T - rem, e_w);
  kahan_add(acc.e_lk, acc.c_lk, dp * (a.t_max_f - t));
  commit(a, acc, c, e_w, dp, glitch);
}

// A piece's window stages each pin's run after the pin's previous event, or,
// where the pin has none, after a time so late that its cycle (the largest
// 32-bit index, as the conversion saturates) never equals an event's: the
// glitch test needs no flag.
constexpr float kNoPrev = 3.0e38f;

__device__ __forceinline__ float f_inf() { return __int_as_float(0x7f800000); }

// The pairwise merge of two input pins' runs (staged a0 .. a0 + na - 1 of the
// lower pin, b0 .. b0 + nb - 1 of the upper; a tie in time takes the lower
// pin first) by the 2^lg lanes of a group, this lane being number `sub`:
// merge path, each lane writing an even share of the outputs from the cut a
// binary search along its first diagonal finds.
__device__ __forceinline__ void merge_pair(const float* ts, int a0, int na, int b0, int nb, uint16_t* out, int sub,
                                           int lg) {
  const int n = na + nb;
  const int per = (n + (1 << lg) - 1) >> lg;
  const int d0 = min(n, sub * per), d1 = min(n, d0 + per);
  int lo = max(0, d0 - nb), hi = min(d0, na);
  while (lo < hi) {  // the number of lower-pin events among the first d0 outputs
    const int mid = (lo + hi) >> 1;
    if (ts[a0 + mid] <= ts[b0 + d0 - mid - 1]) lo = mid + 1;
    else hi = mid;
  }
  int i = lo, j = d0 - lo;
  float ta = i < na ? ts[a0 + i] : f_inf(), tb = j < nb ? ts[b0 + j] : f_inf();
  for (int d = d0; d < d1; ++d) {
    const bool take_a = ta <= tb;
    const int m = (take_a ? i : j) + 1;  // the taken run's next element
    const int x = (take_a ? a0 : b0) + m;
    const float nt = m < (take_a ? na : nb) ? ts[x] : f_inf();
    i = take_a ? m : i;
    j = take_a ? j : m;
    ta = take_a ? nt : ta;
    tb = take_a ? tb : nt;
    out[d] = (uint16_t)((uint32_t)(x - 1) | (take_a ? 0u : 1u << kSelShift) |
                        (((uint32_t)i & 1u) | ((uint32_t)j & 1u) << 1) << kParShift);
  }
}

// A merged run of n elements: with e, the entries mg[x0 ..] of a pairwise
// merge of pins q and q + 1; without, pin q's staged run from x0.
struct MRun {
  int x0, n, q;
  bool e;
};

// Element m of a run: staged index and pin.
__device__ __forceinline__ void run_at(const uint16_t* mg, const MRun& r, int m, int& idx, int& p) {
  const uint32_t w = r.e ? (uint32_t)mg[r.x0 + m] : (uint32_t)(r.x0 + m);
  idx = (int)(w & kIdxMask);
  p = r.q + (int)((w >> kSelShift) & 1u);
}

// The run's pins' parity bits (at the pins' positions) over its first m elements.
__device__ __forceinline__ uint32_t run_par(const uint16_t* mg, const MRun& r, int m) {
  if (r.e) return m > 0 ? (((uint32_t)mg[r.x0 + m - 1] >> kParShift) & 3u) << r.q : 0u;
  return ((uint32_t)m & 1u) << r.q;
}

// A window's input events in (time, pin) order, computed while merging the
// two runs A (pins below those of B) that hold them: lane l takes an even
// share of the merged order from the cut a binary search finds and walks it.
// The state just before an event in that order is the window's start state
// flipped by the parities of the events taken so far on each pin (known at
// the cut from the runs' counts or the entries' parities); the state before
// its timestamp is the one before the first event of its timestamp group.
template <bool kPow2>
__device__ __forceinline__ void walk_inputs(const RunArgs& a, const CTab& CT, const WarpBuf& W, const uint4& SA,
                                            const uint4& SB, const MRun& RA, const MRun& RB, uint32_t start, Acc& acc) {
  const int lane = threadIdx.x & 31;
  const float* ts = W.ts;
  const float* ss = W.ss;
  const uint16_t* mg = W.mg;
  const int na = RA.n, nb = RB.n;
  const int n = na + nb;
  const int per = (n + 31) >> 5;
  const int d0 = min(n, lane * per), d1 = min(n, d0 + per);
  if (d0 >= d1) return;
  int lo = max(0, d0 - nb), hi = min(d0, na);
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    int ia, ib, px;
    run_at(mg, RA, mid, ia, px);
    run_at(mg, RB, d0 - mid - 1, ib, px);
    if (ts[ia] <= ts[ib]) lo = mid + 1;
    else hi = mid;
  }
  int i = lo, j = d0 - lo;
  uint32_t s = start ^ run_par(mg, RA, i) ^ run_par(mg, RB, j);
  int ia = 0, pa = RA.q, ib = 0, pb = RB.q;
  float ta = f_inf(), tb = f_inf();
  if (i < na) {
    run_at(mg, RA, i, ia, pa);
    ta = ts[ia];
  }
  if (j < nb) {
    run_at(mg, RB, j, ib, pb);
    tb = ts[ib];
  }
  // a timestamp group that began before this lane's share: its state is the
  // cut's with the group's earlier events (the ends of both prefixes) taken out
  float t_prev = -1.f;  // times are >= 0
  uint32_t g = 0;
  if (d0 > 0) {
    int x, px;
    float tla = -1.f, tlb = -1.f;
    if (i > 0) {
      run_at(mg, RA, i - 1, x, px);
      tla = ts[x];
    }
    if (j > 0) {
      run_at(mg, RB, j - 1, x, px);
      tlb = ts[x];
    }
    t_prev = fmaxf(tla, tlb);
    const float t0 = fminf(ta, tb);
    if (t0 == t_prev) {
      g = s;
      for (int m = i - 1; m >= 0; --m) {
        run_at(mg, RA, m, x, px);
        if (ts[x] != t0) break;
        g ^= 1u << px;
      }
      for (int m = j - 1; m >= 0; --m) {
        run_at(mg, RB, m, x, px);
        if (ts[x] != t0) break;
        g ^= 1u << px;
      }
    }
  }
  for (int d = d0; d < d1; ++d) {
    const bool take_a = ta <= tb;
    const int idx = take_a ? ia : ib, p = take_a ? pa : pb;
    const float t = take_a ? ta : tb;
    {  // the next head of the run the event came from
      const int m = (take_a ? i : j) + 1;
      const MRun R{take_a ? RA.x0 : RB.x0, take_a ? na : nb, take_a ? RA.q : RB.q, take_a ? RA.e : RB.e};
      int nidx = 0, np = 0;
      float nt = f_inf();
      if (m < R.n) {
        run_at(mg, R, m, nidx, np);
        nt = ts[nidx];
      }
      if (take_a) {
        i = m;
        ia = nidx;
        pa = np;
        ta = nt;
      } else {
        j = m;
        ib = nidx;
        pb = np;
        tb = nt;
      }
    }
    const uint32_t s_b = s;
    s ^= 1u << p;
    if (t != t_prev) g = s_b;
    t_prev = t;
    in_event<kPow2, true>(a, CT, W.u.p.slice, ss, SA, SB, idx, t, p, g, s_b, true, ts[idx - 1], ss + idx - 1, acc);
  }
}

// A piece's window step (gate slot 0, the taken events of each pin a prefix
// of its staged run): output events one lane each; input events in (time,
// pin) order: one pin's run as it is, two pins' runs merged as they are
// walked, three or four pins by pairwise merges first (pins 0 + 1, and 2 + 3
// on the other half-warp) whose results are merged as they are walked.
template <bool kPow2>
__device__ __forceinline__ void window_step(const RunArgs& a, const CTab& CT, WarpBuf& W, Acc& acc) {
  const int lane = threadIdx.x & 31;
  const float* ts = W.ts;
  const float* ss = W.ss;
  const uint4 A = reinterpret_cast<const uint4*>(&W.u.p.slot0)[0];
  const uint4 B = reinterpret_cast<const uint4*>(&W.u.p.slot0)[1];
  const int k = (int)(A.w & 0xFFu);
  // output events
  {
    const int o0 = st_of(A, k), on = W.hw.take[k];
    for (int x = lane; x < on; x += 32) {
      const int i = o0 + x;
      out_event<kPow2>(a, ts, ss, B, i, true, ts[i - 1], ss + i - 1, acc);
    }
  }
  const int n0 = W.hw.take[0], n1 = k > 1 ? W.hw.take[1] : 0, n2 = k > 2 ? W.hw.take[2] : 0,
            n3 = k > 3 ? W.hw.take[3] : 0;
  const int s0 = st_of(A, 0), s1 = st_of(A, 1), s2 = st_of(A, 2), s3 = st_of(A, 3);
  const uint32_t kmask = (1u << k) - 1u;
  const uint32_t start = (((A.w >> 8) & 0xFFu) ^ (A.w >> 24)) & kmask;  // initial bits ^ parities before the window
  if (k >= 3) {  // pins 0 + 1 (the whole warp, or its lower half while the upper merges 2 + 3)
    const bool up = k == 4 && lane >= 16;
    merge_pair(ts, up ? s2 : s0, up ? n2 : n0, up ? s3 : s1, up ? n3 : n1, W.mg + (up ? n0 + n1 : 0),
               lane & (k == 4 ? 15 : 31), k == 4 ? 4 : 5);
    __syncwarp();
  }
  const MRun RA = k >= 3 ? MRun{0, n0 + n1, 0, true} : MRun{s0, n0, 0, false};
  const MRun RB = k == 4 ? MRun{n0 + n1, n2 + n3, 2, true} : (k == 3 ? MRun{s2, n2, 2, false} : MRun{s1, n1, 1, false});
  walk_inputs<kPow2>(a, CT, W, A, B, RA, RB, start, acc);
  __syncwarp();  // the stage is read before it is refilled
}

// A light tile's event at staged index e (slot S, pin p): the input state
// before the event's timestamp from the parities of each input pin's earlier
// events (the count on another pin a binary search of t in its staged run;
// simultaneous events on lower pins are taken back out for the leakage base).
template <bool kPow2>
__device__ __forceinline__ void tile_event(const RunArgs& a, const CTab& CT, const float* ts, const float* ss,
                                           const CSlot& S, int p, int e, Acc& acc) {
  const uint4 A = reinterpret_cast<const uint4*>(&S)[0];
  const uint4 B = reinterpret_cast<const uint4*>(&S)[1];
  const int k = (int)(A.w & 0xFFu);
  const int idx = e - st_of(A, p);
  const bool hp = idx > 0;  // light gates are staged whole: the pin's previous event is staged
  const float tp = hp ? ts[e - 1] : 0.f;
  if (p == k) {
    out_event<kPow2>(a, ts, ss, B, e, hp, tp, ss + e - 1, acc);
    return;
  }
  const uint32_t init = (A.w >> 8) & 0xFFu;
  uint32_t s_pre = init ^ (((uint32_t)idx & 1u) << p);
  uint32_t s_b = s_pre;  // state just before this event in (time, pin) order
  const float t = ts[e];
  for (int q = 0; q < k; ++q) {
    if (q == p) continue;
    const int qa = st_of(A, q), qn = st_of(A, q + 1) - qa;
    const int r = lower_bound_f(ts + qa, qn, t);
    const bool eq = r < qn && ts[qa + r] == t;
    const uint32_t par = (uint32_t)r & 1u;
    s_pre ^= par << q;
    s_b ^= ((par ^ (uint32_t)(q < p && eq)) & 1u) << q;
  }
  in_event<kPow2, false>(a, CT, nullptr, ss, A, B, e, t, p, s_pre, s_b, hp, tp, ss + e - 1, acc);
}

// A light tile: consecutive whole gates, staged whole.
template <bool kPow2>
__device__ __forceinline__ void csr_tile(const RunArgs& a, const CTab& CT, uint32_t ti, WarpBuf& W, Acc& acc) {
  const int lane = threadIdx.x & 31;
  const Tile tl = a.tiles[ti];
  const uint32_t ng = tl.ge - tl.gb;
  if (tl.ge <= tl.gb || ng > kCsrGates) {
    if (lane == 0) dev_err(a.err, tl.gb, kErrTileOverflow);
    return;
  }
  const uint64_t ea = a.tile_ev[2 * ti], eb = a.tile_ev[2 * ti + 1];  // its events, from the partition
  if (eb < ea || eb - ea > (uint64_t)(kStCap - 4)) {
    if (lane == 0) dev_err(a.err, tl.gb, kErrTileOverflow);
    return;
  }
  const int n = (int)(eb - ea);
  if (n == 0) return;
  // times and slews [ea, eb) with 16-byte loads from ea rounded down (the
  // event arrays are padded past their end): staged event i is at W.ts[off + i]
  const uint64_t e4 = ea & ~3ull;
  const int off = (int)(ea - e4), nv = (off + n + 3) >> 2;
  const float4* t4 = reinterpret_cast<const float4*>(a.t + e4);
  const float4* s4 = reinterpret_cast<const float4*>(a.s + e4);
  for (int v = lane; v < nv; v += 32) {  // in flight while the gates' slots are filled
    copy16_async(reinterpret_cast<float4*>(W.ts) + v, t4 + v);
    copy16_async(reinterpret_cast<float4*>(W.ss) + v, s4 + v);
  }
  if (lane < kSegWords) W.u.t.seg.bits[lane] = 0u;
  // a lane per gate: its slot (from the partition's record, pin starts moved
  // by the gate's first event in the tile: the events of the lanes below),
  // then its non-empty pins' runs
  uint4 SA = make_uint4(0u, 0u, 0u, 0u), SB = SA;
  if (lane < (int)ng) {
    SA = a.gslot[2 * (size_t)(tl.gb + (uint32_t)lane)];
    SB = a.gslot[2 * (size_t)(tl.gb + (uint32_t)lane) + 1];
  }
  const int gk = (int)(SA.w & 0xFFu);
  const uint32_t gn = lane < (int)ng ? (uint32_t)st_of(SA, gk + 1) : 0u;
  uint32_t gbase = gn;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, gbase, d);
    if (lane >= d) gbase += y;
  }
  gbase -= gn;
  uint32_t runs = 0, nonempty = 0;
  if (lane < (int)ng) {
    const uint32_t add = gbase | gbase << 16;  // each field stays below 2^16
    SA.x += add;
    SA.y += add;
    SA.z += add;
    reinterpret_cast<uint4*>(&W.u.t.slot[lane])[0] = SA;
    reinterpret_cast<uint4*>(&W.u.t.slot[lane])[1] = SB;
    for (int p = 0; p <= gk; ++p)
      if (st_of(SA, p + 1) > st_of(SA, p)) {
        nonempty |= 1u << p;
        ++runs;
      }
  }
  uint32_t rbase = runs;  // exclusive scan of the gates' run counts
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, rbase, d);
    if (lane >= d) rbase += y;
  }
  rbase -= runs;
  __syncwarp();  // bits cleared
  if (lane < (int)ng) {
    for (int p = 0; p <= gk; ++p)
      if ((nonempty >> p) & 1u) {
        const int e = st_of(SA, p);
        atomicOr(&W.u.t.seg.bits[e >> 5], 1u << (e & 31));
        W.u.t.seg.run[rbase++] = (uint8_t)((lane << 3) | p);
      }
  }
  __syncwarp();
  copies_wait();
  __syncwarp();
  // one lane per event; the event's run is the number of run starts at or
  // before it, minus one
  const float* ts = W.ts + off;  // staged event i: time ts[i], slew ss[i]
  const float* ss = W.ss + off;
  int carry = 0;
  const uint32_t le = 0xFFFFFFFFu >> (31 - lane);  // lanes <= this one
  for (int e0 = 0; e0 < n; e0 += 32) {
    const uint32_t word = W.u.t.seg.bits[e0 >> 5];
    const int e = e0 + lane;
    if (e < n) {
      const uint32_t w = W.u.t.seg.run[carry + __popc(word & le) - 1];
      tile_event<kPow2>(a, CT, ts, ss, W.u.t.slot[w >> 3], (int)(w & 7u), e, acc);
    }
    carry += __popc(word);
  }
  __syncwarp();  // the stage is read before the next item overwrites it
}

// A piece of a heavy gate, in windows of at most kCsrWin events.
template <bool kPow2>
__device__ __forceinline__ void csr_piece(const RunArgs& a, const CTab& CT, uint32_t pi, WarpBuf& W, Acc& acc) {
  const int lane = threadIdx.x & 31;
  const Piece& P = a.pieces[pi];
  const uint32_t g = P.gate, pinfo = P.info;
  const int k = (int)(pinfo & 7u);
  const uint32_t cell = (pinfo >> 12) & 0xFFFu, j = (pinfo >> 8) & 0xFu;
  const bool last = (pinfo >> 31) != 0u;
  const bool mine = lane <= k;  // lane p holds pin p
  uint64_t pst = 0;
  uint32_t cur = 0, hi = 0;
  if (mine) {
    const uint32_t p0 = P.pin[lane], p1 = lane < k ? P.pin[lane + 1] : P.gend;
    pst = P.pin0 + p0;
    cur = P.lo[lane];
    hi = last ? p1 - p0 : a.pieces[pi + 1].lo[lane];
    if (hi < cur) hi = cur;  // (never for a consistent partition)
  }
  CSlot& S = W.u.p.slot0;
  if (lane == 0) {
    S.k = (uint8_t)k;
    S.init = (uint8_t)((pinfo >> 4) & 0xFu);
    S.j = (uint8_t)j;
    S.pre = 0;
    S.cell = (uint16_t)cell;
    S.v = P.v;
    S.esw = P.esw;
  }
  {  // the gate's patch slice (in flight with the first window's copies)
    const uint32_t info = CT.info[cell];
    const int ns1 = (int)(info & 0xFFu), nl1 = (int)((info >> 8) & 0xFFu);
    const float4* src = a.patch + (info >> 16) + j;
    for (int x = lane; x < (ns1 << k); x += 32) copy16_async(&W.u.p.slice[x], src + x * nl1);
  }
  for (int guard = 0;; ++guard) {
    const uint32_t rem = mine ? hi - cur : 0u;
    const uint32_t R = __reduce_add_sync(0xffffffffu, rem);
    if (R == 0) break;
    // the pins' shares of the window, in proportion to their remaining
    // events (rounded down throughout, so they add up to at most kCsrWin,
    // plus one for each pin whose share rounds to nothing)
    uint32_t share = 0;
    if (rem) {
      const float f = __fmul_rd(__uint2float_rd(rem), __fmul_rd((float)kCsrWin, __frcp_rd(__uint2float_ru(R))));
      share = min(rem, max(1u, __float2uint_rd(f)));
    }
    // a pin's share is staged after the pin's previous event (if any) and
    // before its next one after the share, whose time bounds the window; each
    // pin's run is copied in 16-byte vectors from its first event rounded
    // down to a multiple of 4, into 16-byte aligned slots (the pin's events
    // at st .. st + share, then that event)
    const bool more = mine && cur + share < hi;
    const uint32_t before = mine && cur > 0 ? 1u : 0u;
    const uint32_t ns_ = before + share + (more ? 1u : 0u);
    const uint64_t src = pst + cur - before;
    const uint32_t h = ns_ ? (uint32_t)(src & 3u) : 0u;
    // a pin without a previous event whose run would start a vector gets an
    // empty leading vector, which holds the late time in its place
    const uint32_t lead = mine && !before && h == 0u ? 1u : 0u;
    const uint32_t nv = ((h + ns_ + 3u) >> 2) + lead;
    uint32_t vin = nv;  // inclusive prefix of the vectors over lanes 0..k
#pragma unroll
    for (int d = 1; d <= 4; d <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, vin, d);
      if (lane >= d) vin += y;
    }
    const uint32_t vex = vin - nv;
    const uint32_t v0q = vex + lead;  // the pin's first copied vector
    const uint32_t st = 4u * v0q + h + before;
    const uint32_t NV = __shfl_sync(0xffffffffu, vin, k);
    const bool bounded = __any_sync(0xffffffffu, more);
    if (mine) S.st[lane] = (uint16_t)st;
    if (lane == 0) S.st[k + 1] = (uint16_t)(4u * NV);
    const uint32_t pre = __ballot_sync(0xffffffffu, mine && (cur & 1u)) & 31u;
    if (lane == 0) S.pre = (uint8_t)pre;
    // bring the pin's next window into L2 while this one is worked on (about
    // the same share: the bytes from the pin's first unstaged event on)
    if (mine && cur + share < hi) {
      const uint64_t e = pst + cur + share;
      const uint32_t nb = min(hi - (cur + share), share);
      const uint64_t a0 = e & ~3ull;
      const uint32_t bytes = (uint32_t)(((e + nb + 3) & ~3ull) - a0) * 4u;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.t + a0), "r"(bytes));
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.s + a0), "r"(bytes));
    }
    // the vectors of all pins, a lane each (vector v belongs to the pin
    // whose prefix range holds it; the event arrays are padded past their end)
    {
      uint32_t vend[kMaxK];
#pragma unroll
      for (int x = 0; x < kMaxK; ++x) vend[x] = __shfl_sync(0xffffffffu, vin, x);
      const uint64_t src4 = src >> 2;
      for (uint32_t v0 = 0; v0 < NV; v0 += 32) {
        const uint32_t v = v0 + (uint32_t)lane;
        int q = 0;
#pragma unroll
        for (int x = 0; x < kMaxK; ++x) q += (x < k && v >= vend[x]) ? 1 : 0;
        const uint64_t g4 = __shfl_sync(0xffffffffu, src4, q);
        const uint32_t vq = __shfl_sync(0xffffffffu, v0q, q);
        if (v < NV && v >= vq) {
          copy16_async(reinterpret_cast<float4*>(W.ts) + v, reinterpret_cast<const float4*>(a.t) + g4 + (v - vq));
          copy16_async(reinterpret_cast<float4*>(W.ss) + v, reinterpret_cast<const float4*>(a.s) + g4 + (v - vq));
        }
      }
    }
    copies_wait();
    __syncwarp();
    if (mine && !before) W.ts[st - 1] = kNoPrev;  // (in the pin's own vectors, after all copies landed)
    __syncwarp();
    // the first unstaged event of each pin bounds the window
    const float bound = more ? W.ts[st + share] : FLT_MAX;
    const float hz = __uint_as_float(__reduce_min_sync(0xffffffffu, __float_as_uint(bound)));  // t >= 0
    // the events before the horizon are taken (a timestamp group is never split)
    uint32_t take = share;
    if (mine && share > 0 && bounded) take = (uint32_t)lower_bound_f(W.ts + st, (int)share, hz);
    if (mine) W.hw.take[lane] = (uint16_t)take;
    __syncwarp();
    window_step<kPow2>(a, CT, W, acc);
    cur += take;
    const uint32_t moved = __reduce_add_sync(0xffffffffu, mine ? take : 0u);
    __syncwarp();
    if (moved == 0 || guard > (1 << 24)) {  // cannot happen for valid input; never spin
      if (lane == 0) dev_err(a.err, g, kErrTileOverflow);
      break;
    }
  }
  copies_wait();  // (the slice's copies, for a piece without events)
  __syncwarp();
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
  WarpBuf& W = reinterpret_cast<WarpBuf*>(smem + kCellsB)[warp];
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
  // the warps spread their reductions over n_rep (a power of two) copies of the bins
  Acc acc{0.f, 0.f, 0.f, 0.f, 0.f, ((blockIdx.x * (uint32_t)kCW + (uint32_t)warp) & (a.n_rep - 1u)) * a.n_cycles};
  int since = 0;
  // a warp takes kChunk items at a time (the heavy gates' pieces come first:
  // the longest items); the next chunk is asked for as soon as one begins
  uint32_t base = 0;
  if (lane == 0) base = atomicAdd(a.part_counts + 2, kChunk);
  base = __shfl_sync(0xffffffffu, base, 0);
  while (base < n_items) {
    uint32_t nbase = 0;
    if (lane == 0) nbase = atomicAdd(a.part_counts + 2, kChunk);
    for (uint32_t j = 0; j < kChunk && base + j < n_items; ++j) {
      const uint32_t item = base + j;
      if (item < n_pieces)
        csr_piece<kPow2>(a, CT, item, W, acc);
      else
        csr_tile<kPow2>(a, CT, item - n_pieces, W, acc);
      if (++since == kTotEvery) {
        flush_acc(acc, s_tot);
        since = 0;
      }
    }
    base = __shfl_sync(0xffffffffu, nbase, 0);
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
    if (h) {
      a.tiles[th].gb = g;
      a.tile_ev[2 * th] = a.gate_off[g];
    }
    if (tail) {
      a.tiles[th + h - 1].ge = g + 1;
      a.tile_ev[2 * (th + h - 1) + 1] = a.gate_off[g + 1];
    }
    if (pc) {  // a heavy gate: what its pieces share, in its slot entry (k_cp_bounds builds their records)
      const GateRec r = a.gates[g];
      const int k = (int)((r.init >> 16) & 0xff);
      const uint64_t* po = a.pin_off + r.pin_base;
      const uint64_t b0 = po[0];
      const CellDesc& cd = a.cells[r.cell];
      const float C = r.load;
      const int nl = cd.nl;
      int j = 0;
#pragma unroll
      for (int q = 1; q <= PA_MAX_AXIS - 2; ++q) j += (q <= nl - 2 && C >= cd.lax[q]) ? 1 : 0;
      const uint32_t info = (uint32_t)k | ((r.init & 0xFu) << 4) | ((uint32_t)j << 8) | (r.cell << 12);
      const float v = (C - cd.lax[j]) * cd.ilax[j], esw = a.half_vdd2 * C;
      a.gslot[2 * (size_t)g] = make_uint4(info, __float_as_uint(v), __float_as_uint(esw), (uint32_t)(po[k + 1] - b0));
      a.gslot[2 * (size_t)g + 1] = make_uint4((uint32_t)b0, (uint32_t)(b0 >> 32), r.pin_base, 0u);
      for (uint32_t i = 0; i < pc; ++i) {
        a.pieces[tv + i].gate = g;
        a.pieces[tv + i].idx = i;
      }
    } else {  // a light gate: its slot, pin starts from its first event
      const GateRec r = a.gates[g];
      const int k = (int)((r.init >> 16) & 0xff);
      const uint64_t* po = a.pin_off + r.pin_base;
      uint32_t st[kMaxK + 2];
#pragma unroll
      for (int p = 0; p <= kMaxK + 1; ++p) st[p] = p <= k + 1 ? (uint32_t)(po[p] - po[0]) : 0u;
      const CellDesc& cd = a.cells[r.cell];
      const float C = r.load;
      const int nl = cd.nl;
      int j = 0;
#pragma unroll
      for (int q = 1; q <= PA_MAX_AXIS - 2; ++q) j += (q <= nl - 2 && C >= cd.lax[q]) ? 1 : 0;
      const float v = (C - cd.lax[j]) * cd.ilax[j], esw = a.half_vdd2 * C;
      a.gslot[2 * (size_t)g] = make_uint4(st[0] | st[1] << 16, st[2] | st[3] << 16, st[4] | st[5] << 16,
                                         (uint32_t)k | (r.init & 0xFFu) << 8 | (uint32_t)j << 16);
      a.gslot[2 * (size_t)g + 1] = make_uint4(r.cell, __float_as_uint(v), __float_as_uint(esw), 0u);
    }
  }
}

// Every piece's record, from its gate's slot entry (k_cp_emit) and pin
// offsets, with its cut points: piece i > 0 of gate g starts, on each pin, at
// the first event at or after time tau_i, the time of event floor(i c / m) of
// the gate's densest pin (c events, m pieces).
__global__ void __launch_bounds__(256) k_cp_bounds(const RunArgs a) {
  const uint32_t n = a.part_counts[1];
  for (uint32_t pi = blockIdx.x * 256u + threadIdx.x; pi < n; pi += gridDim.x * 256u) {
    Piece& P = a.pieces[pi];
    const uint32_t g = P.gate, i = P.idx;
    const uint4 G0 = a.gslot[2 * (size_t)g], G1 = a.gslot[2 * (size_t)g + 1];
    const int k = (int)(G0.x & 7u);
    const uint32_t gend = G0.w;
    const uint64_t b0 = (uint64_t)G1.x | (uint64_t)G1.y << 32;
    const uint64_t* po = a.pin_off + G1.z;
    const uint64_t m = ((uint64_t)gend + kCsrPiece - 1) / kCsrPiece;
    uint32_t cmax = 0, smax = 0;
    for (int p = 0; p <= k; ++p) {
      const uint32_t s0 = (uint32_t)(po[p] - b0), s1 = p < k ? (uint32_t)(po[p + 1] - b0) : gend;
      P.pin[p] = s0;
      if (s1 - s0 > cmax) {
        cmax = s1 - s0;
        smax = s0;
      }
    }
    P.info = G0.x | (i + 1 >= m ? 1u << 31 : 0u);
    P.v = __uint_as_float(G0.y);
    P.esw = __uint_as_float(G0.z);
    P.gend = gend;
    P.pin0 = b0;
    if (i == 0) {
      for (int p = 0; p <= k; ++p) P.lo[p] = 0;
      continue;
    }
    const float tau = a.t[b0 + smax + (uint64_t)i * cmax / m];
    for (int p = 0; p <= k; ++p) {
      const uint64_t b = po[p];
      uint32_t l = 0, len = (uint32_t)((p < k ? po[p + 1] : b0 + gend) - b);
      while (len > 0) {  // first event at or after tau
        const uint32_t half = len >> 1;
        if (a.t[b + l + half] < tau) {
          l += half + 1;
          len -= half + 1;
        } else {
          len = half;
        }
      }
      P.lo[p] = l;
    }
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
