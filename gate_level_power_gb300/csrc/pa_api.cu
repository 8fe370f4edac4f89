// Host side of libpa.so: the C ABI declared in include/pa.h.
//
// Owns the device copies of the library, netlist and events, validates input
// (library and netlist on the host, events on the device), and runs
// partition -> fused power kernel -> final reduction on the context's stream.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "pa_internal.cuh"

using namespace pa;

namespace {

struct DevBuf {
  void* p = nullptr;
  size_t bytes = 0;
};

}  // namespace

struct pa_ctx {
  int device = 0;
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  int sm_count = 0;
  std::string err;
  long alloc_fail_at = -1;  // test hook: the n-th device allocation fails (PA_TEST_FAIL_ALLOC)
  // test hook (PA_TEST_STAGE_TIMEOUT=i): the banded kernel never starts the
  // stage copy of item i and its bounded waits give up after a few ms
  uint32_t test_skip_item = kNoItem;
  long alloc_count = 0;
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};

  // library
  bool has_lib = false;
  uint32_t n_cells = 0;
  std::vector<CellDesc> h_cells;
  DevBuf cells, lut, leak, patch;

  // netlist
  bool has_net = false;
  uint32_t n_gates = 0;
  uint64_t n_pins = 0;
  DevBuf gates;
  std::vector<GateRec> h_gates;  // host copy (pa_run_stream cuts the netlist into chunks with it)

  // events
  bool has_ev = false;
  uint64_t n_events = 0;
  float t_last = 0.f;  // latest event time
  DevBuf pin_off, gate_off, t, s;

  // scratch
  DevBuf value_tmp, err_word, tmax_bits, val_starts;
  DevBuf bins, part_blk, part_counts, tiles, heavy, pieces, tile_ev, gslot, p0_tot, p_out;
  DevBuf dbg[3], wave_tmp, cnt_tmp, chunk_sums, gate_tmp, cell_tmp;
  // the paper's (gate, window) partition: per-gate plan, thread offsets, scan
  // scratch, total slots (+ the largest events per thread), histogram
  DevBuf w_ncyc, w_nthr, w_off, w_blk, w_tot, w_hist;

  // banded layout (pa_build_bands): persistent parts, build temporaries, run scratch
  BandLayout band;
  uint32_t band_windowed = 0;  // gates cut into windows narrower than a band
  DevBuf b_bt, b_bs, b_btag, b_urec, b_ugate, b_items, b_big;
  DevBuf b_bigf, b_grank, b_cnt, b_evc, b_ubase, b_ebase, b_uband, b_uoff, b_flags, b_ipos, b_scan, b_counters,
      b_urec2, b_dense, b_gflag;
  DevBuf b_part;
  DevBuf scratch_small;

  // pa_run_noalloc's scratch: the device address of the library's file-scope
  // array on this ctx's device, looked up by pa_create (null if that failed,
  // with the reason kept for pa_run_noalloc to report)
  unsigned char* noalloc_base = nullptr;
  std::string noalloc_err;

  // pa_run_stream: two staging slots per chunk array, a copy stream and its events
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t st_copied[2] = {nullptr, nullptr}, st_free[2] = {nullptr, nullptr};
  DevBuf st_t[2], st_s[2], st_v[2], st_pin[2], st_gates[2], st_goff[2];
};

namespace {

int fail(pa_ctx* c, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (c) c->err = buf;
  return code;
}

#define CUDA_TRY(ctx, call)                                                                   \
  do {                                                                                        \
    cudaError_t e_ = (call);                                                                  \
    if (e_ != cudaSuccess)                                                                    \
      return fail((ctx), e_ == cudaErrorMemoryAllocation ? PA_ERR_OOM : PA_ERR_CUDA,          \
                  "%s: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, __LINE__);       \
  } while (0)

void dfree(DevBuf& b) {
  if (b.p) cudaFree(b.p);
  b.p = nullptr;
  b.bytes = 0;
}

// Ensure `b` holds at least `bytes` (contents not preserved).
int dreserve(pa_ctx* c, DevBuf& b, size_t bytes) {
  if (bytes == 0) bytes = 16;
  if (b.p && b.bytes >= bytes) return PA_OK;
  dfree(b);
  ++c->alloc_count;
  if (c->alloc_fail_at >= 0 && c->alloc_count == c->alloc_fail_at)
    return fail(c, PA_ERR_OOM, "device allocation of %zu bytes failed (injected)", bytes);
  cudaError_t e = cudaMalloc(&b.p, bytes);
  if (e != cudaSuccess) {
    b.p = nullptr;
    cudaGetLastError();
    return fail(c, e == cudaErrorMemoryAllocation ? PA_ERR_OOM : PA_ERR_CUDA,
                "cudaMalloc(%zu): %s", bytes, cudaGetErrorString(e));
  }
  b.bytes = bytes;
  return PA_OK;
}

#define PA_TRY(x)                 \
  do {                            \
    int r_ = (x);                 \
    if (r_ != PA_OK) return r_;   \
  } while (0)

bool is_finite_f(float x) { return std::isfinite(x); }

void drop_events(pa_ctx* c) {
  c->has_ev = false;
  c->n_events = 0;
  c->band.built = false;
}

void drop_netlist(pa_ctx* c) {
  drop_events(c);
  c->has_net = false;
  c->n_gates = 0;
  c->n_pins = 0;
}

const char* err_code_name(uint32_t code) {
  switch (code) {
    case kErrPinOff: return "pin_off not monotone / not ending at n_events";
    case kErrUnsorted: return "event times not strictly increasing on a pin";
    case kErrRangeT: return "event time negative or not finite";
    case kErrRangeSlew: return "slew not finite or <= 0";
    case kErrToggle: return "event value equals the pin's previous value";
    case kErrValue: return "event value not 0/1";
    case kErrTileOverflow: return "work item exceeds its shared-memory tile";
    case kErrLayout: return "banded layout inconsistent";
    case kErrStageTimeout: return "stage wait timed out (a bounded wait for a shared-memory stage copy gave up)";
    default: return "unknown";
  }
}

int map_dev_err(pa_ctx* c, unsigned long long key, const char* what) {
  const uint32_t code = (uint32_t)(key & 0xff);
  const unsigned long long idx = key >> 8;
  int rc = PA_ERR_INTERNAL;
  switch (code) {
    case kErrPinOff: rc = PA_ERR_ARG; break;
    case kErrUnsorted: rc = PA_ERR_UNSORTED; break;
    case kErrRangeT:
    case kErrRangeSlew: rc = PA_ERR_RANGE; break;
    case kErrToggle:
    case kErrValue: rc = PA_ERR_TOGGLE; break;
    default: rc = PA_ERR_INTERNAL; break;
  }
  const char* unit = code == kErrPinOff            ? "pin"
                     : code == kErrTileOverflow     ? "gate"
                     : code == kErrLayout || code == kErrStageTimeout ? "item"
                                                    : "event";
  return fail(c, rc, "%s: %s (first at %s %llu)", what, err_code_name(code), unit, idx);
}

bool is_pow2(float x) {
  int e;
  const float m = std::frexp(x, &e);
  return x > 0.f && m == 0.5f;
}

// Validated parameters of one run.
struct RunPlan {
  float T = 0.f;
  double Td = 0.0, t_max = 0.0;
  uint32_t tile = 0, heavy = 0, N = 0, G = 0, nblk = 0;
  // the warp kernel's tile knobs (the user's, else its defaults) and whether
  // it runs the fast pass (no per-event outputs; cells and knobs within its limits)
  uint32_t csr_tile = 0, csr_heavy = 0;
  bool csr = false;
  bool pow2 = false, debug = false, timing = false, gate = false, glitch_all = false, esw_rise = false;
  double vdd = 0.0;
  // partition: PA_PART_*, with the paper's knobs
  uint32_t part_mode = PA_PART_EVENTS, n_evt_tgt = 8, n_thr_floor = 1, n_cyc_fix = 1;
  bool part_stats = false;
};

// Device buffers of one run (owned by the ctx or by the no-alloc scratch).
struct PassBufs {
  float4* bins = nullptr;
  uint32_t n_rep = 1;        // copies of the f32 bins the buffer holds (the warp kernel's pass)
  uint32_t* part_blk = nullptr;
  uint32_t* part_counts = nullptr;
  Tile* tiles = nullptr;
  uint32_t* heavy = nullptr;
  Piece* pieces = nullptr;   // the warp kernel's heavy-gate pieces (null: the CTA kernel runs)
  uint64_t max_pieces = 0;
  uint64_t* tile_ev = nullptr;  // the warp kernel's per-tile event ranges
  uint4* gslot = nullptr;       // the warp kernel's light-gate slots
  double* p0_tot = nullptr;
  double* p_out = nullptr;
  double* chunk_sums = nullptr;
  float* wave = nullptr;
  uint32_t* cnt_ev = nullptr;
  uint32_t* cnt_gl = nullptr;
  uint8_t* dbg[3] = {nullptr, nullptr, nullptr};
  double* gate_e = nullptr;  // per-gate accumulators (fJ), converted to W in place
  double* cell_p = nullptr;  // per-cell sums (W)
};

// stream: the events come with the call (pa_run_stream), so none need be
// loaded and their range is checked chunk by chunk.
int check_run(pa_ctx* c, const pa_run_params* prm, const pa_result* out, const char* who, RunPlan* plan,
              bool stream = false) {
  if (!c) return PA_ERR_ARG;
  if (stream ? !c->has_net : !c->has_ev)
    return fail(c, PA_ERR_ORDER, stream ? "%s: no netlist loaded" : "%s: events not loaded", who);
  if (!prm || !out) return fail(c, PA_ERR_ARG, "%s: null params or result", who);
  if (!(prm->t_clk_ns > 0.f) || !is_finite_f(prm->t_clk_ns)) return fail(c, PA_ERR_ARG, "%s: t_clk_ns must be > 0", who);
  if (prm->n_cycles == 0) return fail(c, PA_ERR_ARG, "%s: n_cycles must be > 0", who);
  if (!std::isfinite(prm->vdd)) return fail(c, PA_ERR_ARG, "%s: vdd not finite", who);
  if (out->out_mem != PA_MEM_HOST && out->out_mem != PA_MEM_DEVICE) return fail(c, PA_ERR_ARG, "%s: bad out_mem", who);
  plan->tile = prm->tile_events ? prm->tile_events : kDefaultTile;
  plan->heavy = prm->heavy_events ? prm->heavy_events : kDefaultHeavy;
  if ((uint64_t)plan->tile + plan->heavy > (uint64_t)kTileCap)
    return fail(c, PA_ERR_ARG, "%s: tile_events + heavy_events = %u exceeds %d", who, plan->tile + plan->heavy, kTileCap);
  plan->T = prm->t_clk_ns;
  plan->Td = (double)plan->T;
  plan->t_max = prm->t_max_ns > 0 ? prm->t_max_ns : (double)prm->n_cycles * plan->Td;
  if (!std::isfinite(plan->t_max)) return fail(c, PA_ERR_ARG, "%s: t_max not finite", who);
  if (!stream && c->n_events) {
    const float cyc = std::floor(c->t_last / plan->T);  // fp32 division, as the kernels take it
    if (!(cyc < (float)prm->n_cycles))
      return fail(c, PA_ERR_RANGE, "%s: latest event t = %.9g ns lies in cycle %.0f >= n_cycles %u", who,
                  (double)c->t_last, (double)cyc, prm->n_cycles);
    if ((double)c->t_last > plan->t_max)
      return fail(c, PA_ERR_RANGE, "%s: t_max %.9g ns is earlier than the latest event %.9g ns", who, plan->t_max,
                  (double)c->t_last);
  }
  plan->N = prm->n_cycles;
  plan->G = c->n_gates;
  plan->nblk = partition_blocks(plan->G);
  plan->gate = out->gate_power_w != nullptr || out->cell_power_w != nullptr;
  plan->debug = out->state_pre || out->lut_ij || out->is_glitch || plan->gate;
  plan->timing = (prm->flags & PA_RUN_TIMING) != 0;
  plan->glitch_all = (prm->flags & PA_RUN_GLITCH_ALL) != 0;
  plan->esw_rise = (prm->flags & PA_RUN_ESW_RISE) != 0;
  // the alternative readings are ablations: they run in the per-event path
  if (plan->glitch_all || plan->esw_rise) plan->debug = true;
  if (prm->flags & ~(PA_RUN_TIMING | PA_RUN_GLITCH_ALL | PA_RUN_ESW_RISE | PA_RUN_PART_STATS))
    return fail(c, PA_ERR_ARG, "%s: unknown flags 0x%x", who, prm->flags);
  if (prm->part_mode > PA_PART_FIXED) return fail(c, PA_ERR_ARG, "%s: unknown part_mode %u", who, prm->part_mode);
  if (stream && prm->part_mode != PA_PART_EVENTS)
    return fail(c, PA_ERR_ARG, "%s: part_mode must be PA_PART_EVENTS on a streamed run", who);
  plan->part_mode = prm->part_mode;
  plan->n_evt_tgt = prm->n_evt_tgt ? prm->n_evt_tgt : 8u;
  plan->n_thr_floor = prm->n_thr_floor ? prm->n_thr_floor : 1u;
  plan->n_cyc_fix = prm->n_cyc_fix ? prm->n_cyc_fix : 1u;
  plan->part_stats = (prm->flags & PA_RUN_PART_STATS) != 0 && plan->part_mode != PA_PART_EVENTS;
  plan->pow2 = is_pow2(plan->T);
  plan->vdd = prm->vdd;
  plan->csr_tile = prm->tile_events ? prm->tile_events : kCsrDefaultTile;
  plan->csr_heavy = prm->heavy_events ? prm->heavy_events : kCsrDefaultHeavy;
  plan->csr = !plan->debug && plan->part_mode == PA_PART_EVENTS && csr_eligible(c->n_cells, plan->csr_tile, plan->csr_heavy);
  return PA_OK;
}

// One run: unbanded (partition -> fused kernel -> final reduction) or, with a
// banded layout, P0 -> banded kernel (+ the unbanded kernel streaming the big
// gates) -> final reduction. Counts are taken in f32 and the pass is repeated
// with integer counts and fp64 bins if a cycle reached 2^24 events. Copies
// outputs on success.
// Per-gate and per-cell accumulators of a run that asks for them: the caller's
// device arrays, else the context's temporaries (copied out at the end).
int setup_gate_bufs(pa_ctx* c, const RunPlan& plan, const pa_result* out, PassBufs& B) {
  if (!plan.gate) return PA_OK;
  const bool dev = out->out_mem == PA_MEM_DEVICE;
  if (out->gate_power_w && dev) {
    B.gate_e = out->gate_power_w;
  } else {
    PA_TRY(dreserve(c, c->gate_tmp, ((size_t)plan.G + 1) * 4 * sizeof(double)));
    B.gate_e = (double*)c->gate_tmp.p;
  }
  if (out->cell_power_w) {
    if (dev) {
      B.cell_p = out->cell_power_w;
    } else {
      PA_TRY(dreserve(c, c->cell_tmp, ((size_t)c->n_cells + 1) * 4 * sizeof(double)));
      B.cell_p = (double*)c->cell_tmp.p;
    }
  }
  return PA_OK;
}

// Run arguments of a pass over the loaded data (a streamed chunk replaces the
// netlist and event pointers).
RunArgs make_run_args(pa_ctx* c, const RunPlan& plan, const PassBufs& B) {
  const uint32_t N = plan.N;
  RunArgs a;
  std::memset(&a, 0, sizeof(a));
  a.cells = (const CellDesc*)c->cells.p;
  a.n_cells = c->n_cells;
  a.lut = (const float*)c->lut.p;
  a.leak = (const float*)c->leak.p;
  a.patch = (const float4*)c->patch.p;
  a.gates = (const GateRec*)c->gates.p;
  a.n_gates = plan.G;
  a.pin_off = (const uint64_t*)c->pin_off.p;
  a.gate_off = (const uint64_t*)c->gate_off.p;
  a.t = (const float*)c->t.p;
  a.s = (const float*)c->s.p;
  a.t_clk = plan.T;
  a.inv_t_clk = plan.pow2 ? 1.0f / plan.T : 0.f;
  a.t_max_f = (float)plan.t_max;
  a.half_vdd2 = (float)(0.5 * plan.vdd * plan.vdd);
  a.glitch_all = plan.glitch_all ? 1u : 0u;
  a.esw_rise = plan.esw_rise ? 1u : 0u;
  a.n_cycles = N;
  a.tile_target = plan.tile;
  a.heavy_thresh = plan.heavy;
  a.part_blk = B.part_blk;
  a.part_counts = B.part_counts;
  a.tiles = B.tiles;
  a.heavy = B.heavy;
  a.p0 = B.p0_tot;
  a.totals = B.p0_tot + 4;
  a.bins = B.bins;
  a.n_rep = 1;
  a.cnt_ev = B.cnt_ev;
  a.cnt_gl = B.cnt_gl;
  a.chunk_sums = B.chunk_sums;
  a.err = (unsigned long long*)c->err_word.p;
  a.dbg_state = B.dbg[0];
  a.dbg_lut = B.dbg[1];
  a.dbg_glitch = B.dbg[2];
  a.gate_e = B.gate_e;
  a.cell_p = B.cell_p;
  return a;
}

// Nearest-rank percentile q of a histogram of n counts (bins[i]: counts equal
// to i; the last bin holds the rest): the smallest x with at least
// ceil(q n / 100) counts <= x.
uint32_t hist_rank(const std::vector<unsigned long long>& bins, uint64_t n, uint32_t q) {
  if (n == 0) return 0;
  const uint64_t r = (q * n + 99) / 100;
  uint64_t cum = 0;
  for (size_t i = 0; i < bins.size(); ++i) {
    cum += bins[i];
    if (cum >= r) return (uint32_t)i;
  }
  return (uint32_t)(bins.size() - 1);
}

int run_pass(pa_ctx* c, const RunPlan& plan, const PassBufs& B, pa_result* out, const char* who,
             const BandLayout* band, const WinArgs* win = nullptr) {
  const uint32_t N = plan.N;
  RunArgs a = make_run_args(c, plan, B);
  if (band) a.heavy = band->big;  // the unbanded kernel streams the gates the layout left out
  // the warp kernel runs the fast pass when the run has room for its pieces
  // (the exact-count retry and the per-event outputs take the CTA kernel)
  const bool csr = plan.csr && B.pieces != nullptr && !band && !win;
  if (csr) {
    a.tile_target = plan.csr_tile;
    a.heavy_thresh = plan.csr_heavy;
    a.pieces = B.pieces;
    a.tile_ev = B.tile_ev;
    a.gslot = B.gslot;
  }
  BandRunArgs A;
  if (band) {
    A.r = a;
    A.L = *band;
    A.item_ctr = B.part_counts + 4;  // part_counts[2] is the unbanded kernel's item counter
    A.skip_item = c->test_skip_item;
    A.wait_limit = c->test_skip_item == kNoItem ? kBandWaitLimit : kBandTestWaitLimit;
  }
  cudaStream_t st = c->stream;
  uint32_t launches = 0;
  double p[4];
  unsigned long long key = kNoErr;
  uint32_t counts[4] = {0, 0, 0, 0};
  bool ran_csr = false;
  for (int exact = 0; exact < 2; ++exact) {
    launches = 0;
    ran_csr = csr && !exact;
    a.n_rep = ran_csr ? B.n_rep : 1u;
    if (plan.timing) CUDA_TRY(c, cudaEventRecord(c->ev[0], st));
    CUDA_TRY(c, cudaMemsetAsync(B.bins, 0, (size_t)N * a.n_rep * sizeof(float4), st));
    if (exact) CUDA_TRY(c, cudaMemsetAsync(B.cnt_ev, 0, (size_t)N * sizeof(uint32_t), st));
    if (exact) CUDA_TRY(c, cudaMemsetAsync(B.cnt_gl, 0, (size_t)N * sizeof(uint32_t), st));
    CUDA_TRY(c, cudaMemsetAsync(B.p0_tot, 0, 8 * sizeof(double), st));
    CUDA_TRY(c, cudaMemsetAsync(c->err_word.p, 0xff, sizeof(unsigned long long), st));
    if (B.gate_e) CUDA_TRY(c, cudaMemsetAsync(B.gate_e, 0, (size_t)plan.G * 4 * sizeof(double), st));
    if (B.cell_p) CUDA_TRY(c, cudaMemsetAsync(B.cell_p, 0, (size_t)c->n_cells * 4 * sizeof(double), st));
    if (win) {
      // the paper's partition: cycles and threads per gate, then P0
      CUDA_TRY(c, cudaMemsetAsync(win->tot_slots, 0, (size_t)kWinTotSlots * 4 * sizeof(double), st));
      if (win->hist) {
        CUDA_TRY(c, cudaMemsetAsync(win->hist, 0, (size_t)kWinHistBins * sizeof(unsigned long long), st));
        CUDA_TRY(c, cudaMemsetAsync(win->ev_max, 0, sizeof(unsigned int), st));
      }
      CUDA_TRY(c, launch_window_plan(a, *win, st));
      CUDA_TRY(c, band_p0(a, st));
      launches += plan.G ? 5 : 0;
    } else if (band) {
      // the unbanded kernel's work list: no tiles, the big gates as heavy gates
      const uint32_t part[8] = {0, band->n_big, 0, 0, 0, 0, 0, 0};
      CUDA_TRY(c, cudaMemcpyAsync(B.part_counts, part, sizeof(part), cudaMemcpyHostToDevice, st));
      CUDA_TRY(c, band_p0(a, st));
      launches += plan.G ? 1 : 0;
    } else if (csr && !exact) {
      // the warp kernel's partition: light tiles and heavy-gate pieces
      CUDA_TRY(c, cudaMemsetAsync(B.part_counts, 0, 4 * sizeof(uint32_t), st));
      CUDA_TRY(c, launch_csr_partition(a, plan.nblk, B.max_pieces, st));
      launches += plan.nblk ? 4 : 0;
    } else {
      a.tile_target = plan.tile;
      a.heavy_thresh = plan.heavy;
      CUDA_TRY(c, cudaMemsetAsync(B.part_counts, 0, 4 * sizeof(uint32_t), st));
      CUDA_TRY(c, launch_partition(a, plan.nblk, st));
      launches += plan.nblk ? 3 : 0;
    }
    if (plan.timing) CUDA_TRY(c, cudaEventRecord(c->ev[1], st));
    if (win) {
      const int grid = c->sm_count * window_blocks_per_sm(plan.pow2, plan.debug, exact != 0);
      CUDA_TRY(c, launch_window(a, *win, grid, plan.pow2, plan.debug, exact != 0, st));
      launches += 2;
    }
    if (band) {
      CUDA_TRY(c, band_fused(A, c->sm_count, plan.debug, exact != 0, st));
      launches += band->n_items ? 1 : 0;
    }
    if (!win && (!band || band->n_big)) {
      if (csr && !exact && !band) {
        CUDA_TRY(c, launch_csr(a, c->sm_count, plan.pow2, st));
      } else {
        const int grid = c->sm_count * fused_blocks_per_sm(plan.pow2, plan.debug, exact != 0);
        CUDA_TRY(c, launch_fused(a, grid, plan.pow2, plan.debug, exact != 0, st));
      }
      launches += 1;
    }
    if (plan.timing) CUDA_TRY(c, cudaEventRecord(c->ev[2], st));
    CUDA_TRY(c, launch_final_reduce(a, plan.Td, plan.t_max, B.wave, B.p_out, exact != 0, st));
    launches += 2;
    if (B.gate_e && plan.G) {
      CUDA_TRY(c, launch_gate_power(a, plan.t_max, st));
      launches += 1;
    }
    if (plan.timing) CUDA_TRY(c, cudaEventRecord(c->ev[3], st));
    CUDA_TRY(c, cudaMemcpyAsync(p, B.p_out, sizeof(p), cudaMemcpyDeviceToHost, st));
    CUDA_TRY(c, cudaMemcpyAsync(&key, c->err_word.p, sizeof(key), cudaMemcpyDeviceToHost, st));
    if (!win) CUDA_TRY(c, cudaMemcpyAsync(counts, B.part_counts, sizeof(counts), cudaMemcpyDeviceToHost, st));
    CUDA_TRY(c, cudaStreamSynchronize(st));
    if (key == kNoErr) break;
    if ((key & 0xff) != kErrCountOverflow || exact) return map_dev_err(c, key, who);
  }
  const cudaMemcpyKind dk = out->out_mem == PA_MEM_HOST ? cudaMemcpyDeviceToHost : cudaMemcpyDeviceToDevice;
  if (out->waveform_w) CUDA_TRY(c, cudaMemcpyAsync(out->waveform_w, B.wave, (size_t)N * sizeof(float), dk, st));
  if (out->event_count) CUDA_TRY(c, cudaMemcpyAsync(out->event_count, B.cnt_ev, (size_t)N * 4, dk, st));
  if (out->glitch_count) CUDA_TRY(c, cudaMemcpyAsync(out->glitch_count, B.cnt_gl, (size_t)N * 4, dk, st));
  if (out->gate_power_w && out->gate_power_w != B.gate_e && plan.G)
    CUDA_TRY(c, cudaMemcpyAsync(out->gate_power_w, B.gate_e, (size_t)plan.G * 4 * sizeof(double), dk, st));
  if (out->cell_power_w && out->cell_power_w != B.cell_p)
    CUDA_TRY(c, cudaMemcpyAsync(out->cell_power_w, B.cell_p, (size_t)c->n_cells * 4 * sizeof(double), dk, st));
  if (plan.debug && c->n_events) {
    uint8_t* dst[3] = {out->state_pre, out->lut_ij, out->is_glitch};
    for (int i = 0; i < 3; ++i)
      if (dst[i] && dst[i] != B.dbg[i]) CUDA_TRY(c, cudaMemcpyAsync(dst[i], B.dbg[i], c->n_events, dk, st));
  }
  CUDA_TRY(c, cudaStreamSynchronize(st));
  out->p_int_w = p[0];
  out->p_sw_w = p[1];
  out->p_gl_w = p[2];
  out->p_leak_w = p[3];
  out->t_max_ns = plan.t_max;
  out->part_threads = 0;
  out->part_evt_p50 = out->part_evt_p90 = out->part_evt_p99 = out->part_evt_max = 0;
  if (win) {
    out->n_tiles = 0;
    out->n_heavy = 0;
    uint64_t n_thr = 0;
    CUDA_TRY(c, cudaMemcpy(&n_thr, win->thr_off + plan.G, sizeof(n_thr), cudaMemcpyDeviceToHost));
    out->part_threads = n_thr;
    if (win->hist) {
      std::vector<unsigned long long> h(kWinHistBins);
      unsigned int mx = 0;
      CUDA_TRY(c, cudaMemcpy(h.data(), win->hist, h.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost));
      CUDA_TRY(c, cudaMemcpy(&mx, win->ev_max, sizeof(mx), cudaMemcpyDeviceToHost));
      out->part_evt_p50 = hist_rank(h, n_thr, 50);
      out->part_evt_p90 = hist_rank(h, n_thr, 90);
      out->part_evt_p99 = hist_rank(h, n_thr, 99);
      out->part_evt_max = mx;
    }
  } else if (band) {
    out->n_tiles = band->n_items;
    out->n_heavy = c->band_windowed + band->n_big;
  } else {
    out->n_tiles = counts[0];
    out->n_heavy = counts[1];
  }
  out->kernel_launches = launches;
  out->path = win ? PA_PATH_WINDOWS : band ? PA_PATH_BANDED : ran_csr ? PA_PATH_WARP : PA_PATH_UNBANDED;
  if (plan.timing) {
    cudaEventElapsedTime(&out->ms_partition, c->ev[0], c->ev[1]);
    cudaEventElapsedTime(&out->ms_fused, c->ev[1], c->ev[2]);
    cudaEventElapsedTime(&out->ms_reduce, c->ev[2], c->ev[3]);
    cudaEventElapsedTime(&out->ms_total, c->ev[0], c->ev[3]);
  }
  return PA_OK;
}

// ----------------------------------------------------------------- streamed run
//
// pa_run_stream: the events stay in host memory and pass through the device
// in chunks of whole gates (about `target` events each). Chunk i + 1 is copied
// on the copy stream while chunk i is validated and computed on the context's
// stream, each chunk by partition -> unbanded fused kernel into the same cycle
// bins and totals; one final reduction at the end. Two staging slots: the copy
// into a slot waits for the compute of the chunk that used it last.

struct StreamChunk {
  uint32_t g0, g1;     // gates
  uint64_t pin0, pin1; // pins
  uint64_t e0, e1;     // events
};

int stream_copy(pa_ctx* c, const pa_events* ev, const StreamChunk& k, int slot, bool wait_free) {
  cudaStream_t cs = c->copy_stream;
  if (wait_free) CUDA_TRY(c, cudaStreamWaitEvent(cs, c->st_free[slot], 0));
  const uint64_t ne = k.e1 - k.e0;
  CUDA_TRY(c, cudaMemcpyAsync(c->st_pin[slot].p, ev->pin_off + k.pin0, (k.pin1 - k.pin0 + 1) * sizeof(uint64_t),
                              cudaMemcpyHostToDevice, cs));
  if (ne) {
    CUDA_TRY(c, cudaMemcpyAsync(c->st_t[slot].p, ev->t_ns + k.e0, ne * sizeof(float), cudaMemcpyHostToDevice, cs));
    CUDA_TRY(c, cudaMemcpyAsync(c->st_s[slot].p, ev->slew_ps + k.e0, ne * sizeof(float), cudaMemcpyHostToDevice, cs));
    if (ev->value) CUDA_TRY(c, cudaMemcpyAsync(c->st_v[slot].p, ev->value + k.e0, ne, cudaMemcpyHostToDevice, cs));
  }
  CUDA_TRY(c, cudaEventRecord(c->st_copied[slot], cs));
  return PA_OK;
}

int run_stream(pa_ctx* c, const RunPlan& plan, const pa_events* ev, uint64_t target, pa_result* out) {
  const char* who = "pa_run_stream";
  const uint32_t G = c->n_gates, N = plan.N;
  const uint64_t P = ev->n_pins, E = ev->n_events;
  const uint64_t* hpo = ev->pin_off;
  if (hpo[0] != 0 || hpo[P] != E) return fail(c, PA_ERR_ARG, "%s: pin_off must start at 0 and end at n_events", who);
  // Chunks of whole gates, each the longest run of gates from its first one
  // that holds at most `target` events (at least one gate), found by binary
  // search over the gates' first event offsets: a few reads of the host pin
  // offsets per chunk, none per pin. The offsets are checked where they cut
  // the trace (here: chunk boundaries in order, so every copy stays inside
  // the caller's arrays) and inside each chunk on the device before the chunk
  // reaches the bins (monotone, ending at the chunk's event count), which
  // together check the whole array.
  auto gate_pin = [&](uint32_t g) -> uint64_t { return g < G ? (uint64_t)c->h_gates[g].pin_base : P; };
  std::vector<StreamChunk> ch;
  uint64_t max_ev = 0, max_pins = 0;
  uint32_t max_g = 0;
  for (uint32_t g0 = 0; g0 < G || ch.empty();) {
    StreamChunk k{g0, 0, 0, 0, 0, 0};
    k.pin0 = gate_pin(g0);
    k.e0 = hpo[k.pin0];
    const uint64_t lim = k.e0 + target;
    uint32_t lo = g0 + 1, hi = G;  // the last g in [g0 + 1, G] whose first event offset is <= lim
    if (g0 < G && hpo[gate_pin(lo)] <= lim) {
      while (lo < hi) {
        const uint32_t mid = lo + (hi - lo + 1) / 2;
        if (hpo[gate_pin(mid)] <= lim) lo = mid;
        else hi = mid - 1;
      }
    }
    k.g1 = g0 < G ? lo : G;
    k.pin1 = gate_pin(k.g1);
    k.e1 = hpo[k.pin1];
    if (k.e1 < k.e0 || k.e1 > E)
      return fail(c, PA_ERR_ARG, "%s: pin_off not monotone (at pin %llu)", who, (unsigned long long)k.pin1);
    max_ev = std::max(max_ev, k.e1 - k.e0);
    max_pins = std::max(max_pins, k.pin1 - k.pin0);
    max_g = std::max(max_g, k.g1 - k.g0);
    ch.push_back(k);
    if (k.g1 == g0) break;  // no gates
    g0 = k.g1;
  }
  // staging slots and run scratch
  if (!c->copy_stream) {
    CUDA_TRY(c, cudaStreamCreateWithFlags(&c->copy_stream, cudaStreamNonBlocking));
    for (int i = 0; i < 2; ++i) {
      CUDA_TRY(c, cudaEventCreateWithFlags(&c->st_copied[i], cudaEventDisableTiming));
      CUDA_TRY(c, cudaEventCreateWithFlags(&c->st_free[i], cudaEventDisableTiming));
    }
  }
  const size_t ev_bytes = ((max_ev + 64) & ~(size_t)15) * sizeof(float);
  for (int i = 0; i < 2; ++i) {
    PA_TRY(dreserve(c, c->st_t[i], ev_bytes));
    PA_TRY(dreserve(c, c->st_s[i], ev_bytes));
    if (ev->value) PA_TRY(dreserve(c, c->st_v[i], max_ev + 16));
    PA_TRY(dreserve(c, c->st_pin[i], (max_pins + 1) * sizeof(uint64_t)));
    PA_TRY(dreserve(c, c->st_gates[i], ((size_t)max_g + 1) * sizeof(GateRec)));
    PA_TRY(dreserve(c, c->st_goff[i], ((size_t)max_g + 1) * sizeof(uint64_t)));
  }
  const uint32_t nblk = partition_blocks(max_g);
  PassBufs B;
  B.n_rep = plan.csr ? bin_copies(N) : 1u;
  PA_TRY(dreserve(c, c->bins, (size_t)N * B.n_rep * sizeof(float4)));
  PA_TRY(dreserve(c, c->part_blk, (size_t)(nblk + 1) * 2 * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->part_counts, 8 * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->tiles, ((size_t)max_g + 1) * sizeof(Tile)));
  PA_TRY(dreserve(c, c->heavy, ((size_t)max_g + 1) * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->p0_tot, 8 * sizeof(double)));
  PA_TRY(dreserve(c, c->p_out, 4 * sizeof(double)));
  PA_TRY(dreserve(c, c->chunk_sums, (size_t)reduce_chunks(N) * sizeof(double)));
  PA_TRY(dreserve(c, c->wave_tmp, (size_t)N * sizeof(float)));
  PA_TRY(dreserve(c, c->cnt_tmp, (size_t)N * 2 * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->err_word, sizeof(unsigned long long)));
  PA_TRY(dreserve(c, c->tmax_bits, sizeof(unsigned int)));
  PA_TRY(dreserve(c, c->val_starts, ((max_ev + 31) / 32 + 1) * sizeof(uint32_t)));
  B.bins = (float4*)c->bins.p;
  B.part_blk = (uint32_t*)c->part_blk.p;
  B.part_counts = (uint32_t*)c->part_counts.p;
  B.tiles = (Tile*)c->tiles.p;
  B.heavy = (uint32_t*)c->heavy.p;
  B.p0_tot = (double*)c->p0_tot.p;
  B.p_out = (double*)c->p_out.p;
  B.chunk_sums = (double*)c->chunk_sums.p;
  B.wave = (float*)c->wave_tmp.p;
  B.cnt_ev = (uint32_t*)c->cnt_tmp.p;
  B.cnt_gl = (uint32_t*)c->cnt_tmp.p + N;
  if (plan.csr) {
    B.max_pieces = csr_max_pieces(max_ev, max_g, plan.csr_heavy);
    PA_TRY(dreserve(c, c->pieces, (size_t)B.max_pieces * sizeof(Piece)));
    PA_TRY(dreserve(c, c->tile_ev, ((size_t)max_g + 1) * 2 * sizeof(uint64_t)));
    PA_TRY(dreserve(c, c->gslot, ((size_t)max_g + 1) * 2 * sizeof(uint4)));
    B.gslot = (uint4*)c->gslot.p;
    B.pieces = (Piece*)c->pieces.p;
    B.tile_ev = (uint64_t*)c->tile_ev.p;
  }
  PA_TRY(setup_gate_bufs(c, plan, out, B));
  cudaStream_t st = c->stream;
  const int nc = (int)ch.size();
  double p[4];
  unsigned long long key = kNoErr;
  uint32_t launches = 0;
  bool stream_csr = false;
  for (int exact = 0; exact < 2; ++exact) {
    launches = 0;
    stream_csr = B.pieces && !exact;
    const uint32_t n_rep = stream_csr ? B.n_rep : 1u;
    if (plan.timing) CUDA_TRY(c, cudaEventRecord(c->ev[0], st));
    CUDA_TRY(c, cudaMemsetAsync(B.bins, 0, (size_t)N * n_rep * sizeof(float4), st));
    if (exact) CUDA_TRY(c, cudaMemsetAsync(B.cnt_ev, 0, (size_t)N * 2 * sizeof(uint32_t), st));
    CUDA_TRY(c, cudaMemsetAsync(B.p0_tot, 0, 8 * sizeof(double), st));
    CUDA_TRY(c, cudaMemsetAsync(c->err_word.p, 0xff, sizeof(unsigned long long), st));
    CUDA_TRY(c, cudaMemsetAsync(c->tmax_bits.p, 0, sizeof(unsigned int), st));
    if (B.gate_e) CUDA_TRY(c, cudaMemsetAsync(B.gate_e, 0, (size_t)G * 4 * sizeof(double), st));
    if (B.cell_p) CUDA_TRY(c, cudaMemsetAsync(B.cell_p, 0, (size_t)c->n_cells * 4 * sizeof(double), st));
    CUDA_TRY(c, cudaStreamSynchronize(st));  // the slots are free and the accumulators clear
    PA_TRY(stream_copy(c, ev, ch[0], 0, false));
    for (int i = 0; i < nc; ++i) {
      const StreamChunk& k = ch[i];
      const int slot = i & 1;
      if (i + 1 < nc) PA_TRY(stream_copy(c, ev, ch[i + 1], (i + 1) & 1, i + 1 >= 2));
      CUDA_TRY(c, cudaStreamWaitEvent(st, c->st_copied[slot], 0));
      const uint32_t gk = k.g1 - k.g0;
      const uint64_t pk = k.pin1 - k.pin0, ek = k.e1 - k.e0;
      uint64_t* pin = (uint64_t*)c->st_pin[slot].p;
      GateRec* gates = (GateRec*)c->st_gates[slot].p;
      CUDA_TRY(c, launch_rebase_chunk(pin, pk, k.e0, (const GateRec*)c->gates.p + k.g0, gates, gk,
                                      (uint32_t)k.pin0, st));
      CUDA_TRY(c, launch_check_pin_off(pin, pk, ek, (unsigned long long*)c->err_word.p, st));
      ValidateArgs va;
      va.gates = gates;
      va.n_gates = gk;
      va.n_pins = pk;
      va.n_events = ek;
      va.pin_off = pin;
      va.t = (const float*)c->st_t[slot].p;
      va.s = (const float*)c->st_s[slot].p;
      va.value = ev->value ? (const uint8_t*)c->st_v[slot].p : nullptr;
      va.gate_off = (uint64_t*)c->st_goff[slot].p;
      va.err = (unsigned long long*)c->err_word.p;
      va.t_max_bits = (unsigned int*)c->tmax_bits.p;
      va.starts = (uint32_t*)c->val_starts.p;
      CUDA_TRY(c, launch_validate_events(va, st));
      launches += 1 + (gk ? 1 : 0) + 1 + 1 + (ek ? 1 : 0);  // rebase (pins, gates), check, validate (gates, events)
      // the chunk must be valid, and its events inside the window, before it touches the bins
      unsigned int tbits = 0;
      CUDA_TRY(c, cudaMemcpyAsync(&key, c->err_word.p, sizeof(key), cudaMemcpyDeviceToHost, st));
      CUDA_TRY(c, cudaMemcpyAsync(&tbits, c->tmax_bits.p, sizeof(tbits), cudaMemcpyDeviceToHost, st));
      CUDA_TRY(c, cudaStreamSynchronize(st));
      if (key != kNoErr) {
        const uint32_t code = (uint32_t)(key & 0xff);
        const uint64_t base = code == kErrPinOff ? k.pin0 : (code == kErrTileOverflow ? k.g0 : k.e0);
        CUDA_TRY(c, cudaStreamSynchronize(c->copy_stream));
        return map_dev_err(c, (((key >> 8) + base) << 8) | code, who);
      }
      float t_last;
      std::memcpy(&t_last, &tbits, sizeof(float));
      if (ek) {
        const float cyc = std::floor(t_last / plan.T);
        if (!(cyc < (float)N) || (double)t_last > plan.t_max) {
          CUDA_TRY(c, cudaStreamSynchronize(c->copy_stream));
          return fail(c, PA_ERR_RANGE, "%s: an event at t = %.9g ns lies outside the window (%u cycles, t_max %.9g)",
                      who, (double)t_last, N, plan.t_max);
        }
      }
      RunArgs a = make_run_args(c, plan, B);
      a.n_rep = n_rep;
      a.gates = gates;
      a.n_gates = gk;
      a.pin_off = pin;
      a.gate_off = (const uint64_t*)c->st_goff[slot].p;
      a.t = (const float*)c->st_t[slot].p;
      a.s = (const float*)c->st_s[slot].p;
      a.gate_e = B.gate_e ? B.gate_e + (size_t)k.g0 * 4 : nullptr;
      CUDA_TRY(c, cudaMemsetAsync(B.part_counts, 0, 4 * sizeof(uint32_t), st));
      if (B.pieces && !exact) {  // the warp kernel (fast pass)
        a.tile_target = plan.csr_tile;
        a.heavy_thresh = plan.csr_heavy;
        a.pieces = B.pieces;
        a.tile_ev = B.tile_ev;
        a.gslot = B.gslot;
        CUDA_TRY(c, launch_csr_partition(a, partition_blocks(gk), B.max_pieces, st));
        CUDA_TRY(c, launch_csr(a, c->sm_count, plan.pow2, st));
        launches += (gk ? 4 : 0) + 1;
      } else {
        CUDA_TRY(c, launch_partition(a, partition_blocks(gk), st));
        const int grid = c->sm_count * fused_blocks_per_sm(plan.pow2, plan.debug, exact != 0);
        CUDA_TRY(c, launch_fused(a, grid, plan.pow2, plan.debug, exact != 0, st));
        launches += (gk ? 3 : 0) + 1;
      }
      CUDA_TRY(c, cudaEventRecord(c->st_free[slot], st));
    }
    RunArgs a = make_run_args(c, plan, B);
    a.n_rep = n_rep;
    a.n_gates = G;
    a.gates = (const GateRec*)c->gates.p;
    CUDA_TRY(c, launch_final_reduce(a, plan.Td, plan.t_max, B.wave, B.p_out, exact != 0, st));
    launches += 2;
    if (B.gate_e && G) {
      CUDA_TRY(c, launch_gate_power(a, plan.t_max, st));
      launches += 1;
    }
    if (plan.timing) CUDA_TRY(c, cudaEventRecord(c->ev[3], st));
    CUDA_TRY(c, cudaMemcpyAsync(p, B.p_out, sizeof(p), cudaMemcpyDeviceToHost, st));
    CUDA_TRY(c, cudaMemcpyAsync(&key, c->err_word.p, sizeof(key), cudaMemcpyDeviceToHost, st));
    CUDA_TRY(c, cudaStreamSynchronize(st));
    if (key == kNoErr) break;
    if ((key & 0xff) != kErrCountOverflow || exact) return map_dev_err(c, key, who);
  }
  const cudaMemcpyKind dk = out->out_mem == PA_MEM_HOST ? cudaMemcpyDeviceToHost : cudaMemcpyDeviceToDevice;
  if (out->waveform_w) CUDA_TRY(c, cudaMemcpyAsync(out->waveform_w, B.wave, (size_t)N * sizeof(float), dk, st));
  if (out->event_count) CUDA_TRY(c, cudaMemcpyAsync(out->event_count, B.cnt_ev, (size_t)N * 4, dk, st));
  if (out->glitch_count) CUDA_TRY(c, cudaMemcpyAsync(out->glitch_count, B.cnt_gl, (size_t)N * 4, dk, st));
  if (out->gate_power_w && out->gate_power_w != B.gate_e && G)
    CUDA_TRY(c, cudaMemcpyAsync(out->gate_power_w, B.gate_e, (size_t)G * 4 * sizeof(double), dk, st));
  if (out->cell_power_w && out->cell_power_w != B.cell_p)
    CUDA_TRY(c, cudaMemcpyAsync(out->cell_power_w, B.cell_p, (size_t)c->n_cells * 4 * sizeof(double), dk, st));
  CUDA_TRY(c, cudaStreamSynchronize(st));
  out->p_int_w = p[0];
  out->p_sw_w = p[1];
  out->p_gl_w = p[2];
  out->p_leak_w = p[3];
  out->t_max_ns = plan.t_max;
  out->n_tiles = (uint32_t)nc;  // chunks
  out->n_heavy = 0;
  out->kernel_launches = launches;
  out->path = stream_csr ? PA_PATH_WARP : PA_PATH_UNBANDED;
  out->ms_partition = out->ms_fused = out->ms_reduce = out->ms_total = 0.f;
  if (plan.timing) cudaEventElapsedTime(&out->ms_total, c->ev[0], c->ev[3]);
  return PA_OK;
}

bool same_bits(float a, float b) { return std::memcmp(&a, &b, sizeof(float)) == 0; }

// Looks up the device address of pa_run_noalloc's scratch array on the
// current device (defined with the array, below).
void noalloc_lookup(pa_ctx* c);

}  // namespace

extern "C" {

int pa_version(void) { return PA_VERSION; }

void pa_default_params(pa_run_params* p) {
  if (!p) return;
  std::memset(p, 0, sizeof(*p));
  p->vdd = 0.9;
  p->t_clk_ns = 1.0f;
  p->n_cycles = 1;
}

const char* pa_last_error(const pa_ctx* ctx) { return ctx ? ctx->err.c_str() : "null context"; }

int pa_create(pa_ctx** out, int cuda_device, void* cuda_stream) {
  if (!out) return PA_ERR_ARG;
  *out = nullptr;
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n == 0) {
    cudaGetLastError();
    return PA_ERR_CUDA;
  }
  if (cuda_device < 0 || cuda_device >= n) return PA_ERR_ARG;
  pa_ctx* c = new (std::nothrow) pa_ctx();
  if (!c) return PA_ERR_OOM;
  c->device = cuda_device;
  if (const char* f = std::getenv("PA_TEST_FAIL_ALLOC")) c->alloc_fail_at = std::atol(f);
  if (const char* f = std::getenv("PA_TEST_STAGE_TIMEOUT")) c->test_skip_item = (uint32_t)std::strtoul(f, nullptr, 10);
  if (cudaSetDevice(cuda_device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, cuda_device) != cudaSuccess) {
    cudaGetLastError();
    delete c;
    return PA_ERR_CUDA;
  }
  if (cuda_stream) {
    c->stream = (cudaStream_t)cuda_stream;
  } else {
    if (cudaStreamCreateWithFlags(&c->stream, cudaStreamNonBlocking) != cudaSuccess) {
      cudaGetLastError();
      delete c;
      return PA_ERR_CUDA;
    }
    c->own_stream = true;
  }
  for (auto& e : c->ev) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      cudaGetLastError();
      pa_destroy(c);
      return PA_ERR_CUDA;
    }
  }
  noalloc_lookup(c);
  *out = c;
  return PA_OK;
}

void pa_destroy(pa_ctx* c) {
  if (!c) return;
  cudaSetDevice(c->device);
  if (c->stream) cudaStreamSynchronize(c->stream);
  DevBuf* all[] = {&c->cells, &c->lut, &c->leak, &c->patch, &c->gates, &c->pin_off, &c->gate_off, &c->t, &c->s,
                   &c->value_tmp, &c->err_word, &c->tmax_bits, &c->val_starts, &c->bins, &c->part_blk,
                   &c->part_counts, &c->tiles, &c->heavy, &c->pieces, &c->tile_ev, &c->gslot, &c->p0_tot, &c->p_out, &c->dbg[0],
                   &c->dbg[1], &c->dbg[2], &c->wave_tmp, &c->cnt_tmp, &c->gate_tmp, &c->cell_tmp, &c->scratch_small,
                   &c->chunk_sums, &c->b_bt, &c->b_bs, &c->b_btag, &c->b_urec, &c->b_ugate, &c->b_items,
                   &c->b_big, &c->b_bigf, &c->b_grank, &c->b_cnt, &c->b_evc, &c->b_ubase, &c->b_ebase,
                   &c->b_uband, &c->b_uoff, &c->b_flags, &c->b_ipos, &c->b_scan, &c->b_counters,
                   &c->b_urec2, &c->b_dense, &c->b_gflag, &c->b_part, &c->w_ncyc, &c->w_nthr, &c->w_off,
                   &c->w_blk, &c->w_tot, &c->w_hist};
  for (DevBuf* b : all) dfree(*b);
  for (int i = 0; i < 2; ++i) {
    DevBuf* st[] = {&c->st_t[i], &c->st_s[i], &c->st_v[i], &c->st_pin[i], &c->st_gates[i], &c->st_goff[i]};
    for (DevBuf* b : st) dfree(*b);
    if (c->st_copied[i]) cudaEventDestroy(c->st_copied[i]);
    if (c->st_free[i]) cudaEventDestroy(c->st_free[i]);
  }
  if (c->copy_stream) cudaStreamDestroy(c->copy_stream);
  for (auto& e : c->ev)
    if (e) cudaEventDestroy(e);
  if (c->own_stream && c->stream) cudaStreamDestroy(c->stream);
  delete c;
}

int pa_load_library(pa_ctx* c, const pa_library* L) {
  if (!c) return PA_ERR_ARG;
  if (!L || !L->n_inputs || !L->n_slew || !L->n_load || !L->slew_axis || !L->load_axis || !L->lut_off ||
      !L->lut || !L->leak_off || !L->leak || L->n_cells == 0)
    return fail(c, PA_ERR_ARG, "pa_load_library: null pointer or zero cells");
  cudaSetDevice(c->device);
  c->has_lib = false;
  drop_netlist(c);
  std::vector<CellDesc> cells(L->n_cells);
  for (uint32_t ci = 0; ci < L->n_cells; ++ci) {
    CellDesc& d = cells[ci];
    std::memset(&d, 0, sizeof(d));
    const int k = L->n_inputs[ci], ns = L->n_slew[ci], nl = L->n_load[ci];
    if (k < 1 || k > PA_MAX_INPUTS)
      return fail(c, PA_ERR_ARG, "cell %u: n_inputs %d outside [1, %d]", ci, k, PA_MAX_INPUTS);
    if (ns < 2 || ns > PA_MAX_AXIS || nl < 2 || nl > PA_MAX_AXIS)
      return fail(c, PA_ERR_ARG, "cell %u: axis lengths %d x %d outside [2, 8]", ci, ns, nl);
    const float* sa = L->slew_axis + (size_t)ci * 8;
    const float* la = L->load_axis + (size_t)ci * 8;
    for (int i = 0; i < ns; ++i) {
      if (!is_finite_f(sa[i]) || (i > 0 && !(sa[i] > sa[i - 1])))
        return fail(c, PA_ERR_ARG, "cell %u: slew axis not finite and strictly increasing", ci);
      d.sax[i] = sa[i];
    }
    for (int i = 0; i < nl; ++i) {
      if (!is_finite_f(la[i]) || (i > 0 && !(la[i] > la[i - 1])))
        return fail(c, PA_ERR_ARG, "cell %u: load axis not finite and strictly increasing", ci);
      d.lax[i] = la[i];
    }
    for (int i = 0; i + 1 < ns; ++i) d.isax[i] = 1.0f / (sa[i + 1] - sa[i]);
    for (int i = 0; i + 1 < nl; ++i) d.ilax[i] = 1.0f / (la[i + 1] - la[i]);
    const uint64_t lut_n = (uint64_t)(1u << k) * ns * nl;
    if ((uint64_t)L->lut_off[ci] + lut_n > L->lut_len)
      return fail(c, PA_ERR_ARG, "cell %u: LUT offset %u + %llu beyond lut_len %llu", ci, L->lut_off[ci],
                  (unsigned long long)lut_n, (unsigned long long)L->lut_len);
    if ((uint64_t)L->leak_off[ci] + (1u << k) > L->leak_len)
      return fail(c, PA_ERR_ARG, "cell %u: leakage offset beyond leak_len", ci);
    d.k = (uint8_t)k;
    d.ns = (uint8_t)ns;
    d.nl = (uint8_t)nl;
    d.lut_off = L->lut_off[ci];
    d.leak_off = L->leak_off[ci];
  }
  for (uint64_t i = 0; i < L->lut_len; ++i)
    if (!is_finite_f(L->lut[i])) return fail(c, PA_ERR_ARG, "LUT value %llu not finite", (unsigned long long)i);
  std::vector<float> leak_uw(L->leak_len);
  for (uint64_t i = 0; i < L->leak_len; ++i) {
    if (!is_finite_f(L->leak[i])) return fail(c, PA_ERR_ARG, "leakage value %llu not finite", (unsigned long long)i);
    leak_uw[i] = (float)((double)L->leak[i] * 1e-3);  // nW -> uW (= fJ / ns)
  }
  // derived table: LUT corner patches
  std::vector<float> patch;
  for (uint32_t ci = 0; ci < L->n_cells; ++ci) {
    CellDesc& d = cells[ci];
    d.patch_off = (uint32_t)(patch.size() / 4);
    const int k = d.k, ns = d.ns, nl = d.nl;
    for (int st = 0; st < (1 << k); ++st) {
      const float* T = L->lut + d.lut_off + (size_t)st * ns * nl;
      for (int i = 0; i + 1 < ns; ++i)
        for (int j = 0; j + 1 < nl; ++j) {
          patch.push_back(T[i * nl + j]);
          patch.push_back(T[i * nl + j + 1]);
          patch.push_back(T[(i + 1) * nl + j]);
          patch.push_back(T[(i + 1) * nl + j + 1]);
        }
    }
  }
  PA_TRY(dreserve(c, c->patch, patch.size() * sizeof(float)));
  CUDA_TRY(c, cudaMemcpyAsync(c->patch.p, patch.data(), patch.size() * sizeof(float), cudaMemcpyHostToDevice, c->stream));
  PA_TRY(dreserve(c, c->cells, cells.size() * sizeof(CellDesc)));
  PA_TRY(dreserve(c, c->lut, L->lut_len * sizeof(float)));
  PA_TRY(dreserve(c, c->leak, L->leak_len * sizeof(float)));
  CUDA_TRY(c, cudaMemcpyAsync(c->cells.p, cells.data(), cells.size() * sizeof(CellDesc), cudaMemcpyHostToDevice, c->stream));
  CUDA_TRY(c, cudaMemcpyAsync(c->lut.p, L->lut, L->lut_len * sizeof(float), cudaMemcpyHostToDevice, c->stream));
  CUDA_TRY(c, cudaMemcpyAsync(c->leak.p, leak_uw.data(), L->leak_len * sizeof(float), cudaMemcpyHostToDevice, c->stream));
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  c->h_cells = std::move(cells);
  c->n_cells = L->n_cells;
  c->has_lib = true;
  return PA_OK;
}

int pa_load_netlist(pa_ctx* c, const pa_netlist* N) {
  if (!c) return PA_ERR_ARG;
  if (!c->has_lib) return fail(c, PA_ERR_ORDER, "pa_load_netlist: no library loaded");
  if (!N || (N->n_gates && (!N->cell_id || !N->load_ff || !N->init_in || !N->init_out)))
    return fail(c, PA_ERR_ARG, "pa_load_netlist: null pointer");
  cudaSetDevice(c->device);
  drop_netlist(c);
  const uint32_t G = N->n_gates;
  std::vector<GateRec> recs(G);
  uint64_t pb = 0;
  for (uint32_t g = 0; g < G; ++g) {
    const uint32_t ci = N->cell_id[g];
    if (ci >= c->n_cells) return fail(c, PA_ERR_RANGE, "gate %u: cell id %u >= n_cells %u", g, ci, c->n_cells);
    const int k = c->h_cells[ci].k;
    const float C = N->load_ff[g];
    if (!is_finite_f(C) || C < 0.f) return fail(c, PA_ERR_RANGE, "gate %u: load %g not finite or < 0", g, (double)C);
    if (N->init_in[g] >> k) return fail(c, PA_ERR_RANGE, "gate %u: init_in has bits beyond k = %d", g, k);
    if (N->init_out[g] > 1) return fail(c, PA_ERR_RANGE, "gate %u: init_out not 0/1", g);
    if (pb > 0xFFFFFFFFull - 8) return fail(c, PA_ERR_ARG, "netlist has too many pins (>= 2^32)");
    recs[g].pin_base = (uint32_t)pb;
    recs[g].cell = ci;
    recs[g].load = C;
    recs[g].init = (uint32_t)N->init_in[g] | ((uint32_t)N->init_out[g] << 8) | ((uint32_t)k << 16);
    pb += (uint64_t)k + 1;
  }
  PA_TRY(dreserve(c, c->gates, (size_t)G * sizeof(GateRec)));
  if (G) CUDA_TRY(c, cudaMemcpyAsync(c->gates.p, recs.data(), (size_t)G * sizeof(GateRec), cudaMemcpyHostToDevice, c->stream));
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  c->h_gates = std::move(recs);
  c->n_gates = G;
  c->n_pins = pb;
  c->has_net = true;
  return PA_OK;
}

int pa_load_events(pa_ctx* c, const pa_events* ev) {
  if (!c) return PA_ERR_ARG;
  if (!c->has_net) return fail(c, PA_ERR_ORDER, "pa_load_events: no netlist loaded");
  if (!ev || !ev->pin_off || (ev->n_events && (!ev->t_ns || !ev->slew_ps)))
    return fail(c, PA_ERR_ARG, "pa_load_events: null pointer");
  if (ev->mem != PA_MEM_HOST && ev->mem != PA_MEM_DEVICE) return fail(c, PA_ERR_ARG, "pa_load_events: bad mem");
  if (ev->n_pins != c->n_pins)
    return fail(c, PA_ERR_ARG, "pa_load_events: n_pins %llu != netlist pins %llu",
                (unsigned long long)ev->n_pins, (unsigned long long)c->n_pins);
  cudaSetDevice(c->device);
  drop_events(c);
  const uint64_t E = ev->n_events, P = ev->n_pins;
  const cudaMemcpyKind kind = ev->mem == PA_MEM_HOST ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice;
  // Owned, padded copies (16-byte multiple plus slack for vector loads).
  const size_t ev_bytes = ((E + 64) & ~(size_t)15) * sizeof(float);
  PA_TRY(dreserve(c, c->pin_off, (P + 1) * sizeof(uint64_t)));
  PA_TRY(dreserve(c, c->gate_off, ((size_t)c->n_gates + 1) * sizeof(uint64_t)));
  PA_TRY(dreserve(c, c->t, ev_bytes));
  PA_TRY(dreserve(c, c->s, ev_bytes));
  PA_TRY(dreserve(c, c->err_word, sizeof(unsigned long long)));
  PA_TRY(dreserve(c, c->tmax_bits, sizeof(unsigned int)));
  CUDA_TRY(c, cudaMemcpyAsync(c->pin_off.p, ev->pin_off, (P + 1) * sizeof(uint64_t), kind, c->stream));
  CUDA_TRY(c, cudaMemsetAsync(c->err_word.p, 0xff, sizeof(unsigned long long), c->stream));
  CUDA_TRY(c, cudaMemsetAsync(c->tmax_bits.p, 0, sizeof(unsigned int), c->stream));
  CUDA_TRY(c, launch_check_pin_off((const uint64_t*)c->pin_off.p, P, E, (unsigned long long*)c->err_word.p, c->stream));
  unsigned long long key = kNoErr;
  CUDA_TRY(c, cudaMemcpyAsync(&key, c->err_word.p, sizeof(key), cudaMemcpyDeviceToHost, c->stream));
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  if (key != kNoErr) return map_dev_err(c, key, "pa_load_events");
  if (E) {
    CUDA_TRY(c, cudaMemcpyAsync(c->t.p, ev->t_ns, E * sizeof(float), kind, c->stream));
    CUDA_TRY(c, cudaMemcpyAsync(c->s.p, ev->slew_ps, E * sizeof(float), kind, c->stream));
  }
  const uint8_t* dval = nullptr;
  if (ev->value && E) {
    if (ev->mem == PA_MEM_HOST) {
      PA_TRY(dreserve(c, c->value_tmp, E));
      CUDA_TRY(c, cudaMemcpyAsync(c->value_tmp.p, ev->value, E, cudaMemcpyHostToDevice, c->stream));
      dval = (const uint8_t*)c->value_tmp.p;
    } else {
      dval = ev->value;
    }
  }
  ValidateArgs va;
  va.gates = (const GateRec*)c->gates.p;
  va.n_gates = c->n_gates;
  va.n_pins = P;
  va.n_events = E;
  va.pin_off = (const uint64_t*)c->pin_off.p;
  va.t = (const float*)c->t.p;
  va.s = (const float*)c->s.p;
  va.value = dval;
  va.gate_off = (uint64_t*)c->gate_off.p;
  va.err = (unsigned long long*)c->err_word.p;
  va.t_max_bits = (unsigned int*)c->tmax_bits.p;
  PA_TRY(dreserve(c, c->val_starts, ((E + 31) / 32 + 1) * sizeof(uint32_t)));
  va.starts = (uint32_t*)c->val_starts.p;
  CUDA_TRY(c, launch_validate_events(va, c->stream));
  unsigned int tbits = 0;
  CUDA_TRY(c, cudaMemcpyAsync(&key, c->err_word.p, sizeof(key), cudaMemcpyDeviceToHost, c->stream));
  CUDA_TRY(c, cudaMemcpyAsync(&tbits, c->tmax_bits.p, sizeof(tbits), cudaMemcpyDeviceToHost, c->stream));
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  if (key != kNoErr) return map_dev_err(c, key, "pa_load_events");
  std::memcpy(&c->t_last, &tbits, sizeof(float));
  c->n_events = E;
  c->has_ev = true;
  return PA_OK;
}

int pa_run(pa_ctx* c, const pa_run_params* prm, pa_result* out) {
  RunPlan plan;
  PA_TRY(check_run(c, prm, out, "pa_run", &plan));
  CUDA_TRY(c, cudaSetDevice(c->device));
  const bool banded = c->band.built && same_bits(c->band.t_clk, plan.T);
  const uint32_t N = plan.N, G = plan.G;
  PassBufs B;
  B.n_rep = plan.csr && !banded ? bin_copies(N) : 1u;
  PA_TRY(dreserve(c, c->bins, (size_t)N * B.n_rep * sizeof(float4)));
  PA_TRY(dreserve(c, c->part_blk, (size_t)(plan.nblk + 1) * 2 * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->part_counts, 8 * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->tiles, ((size_t)G + 1) * sizeof(Tile)));
  PA_TRY(dreserve(c, c->heavy, ((size_t)G + 1) * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->p0_tot, 8 * sizeof(double)));
  PA_TRY(dreserve(c, c->p_out, 4 * sizeof(double)));
  PA_TRY(dreserve(c, c->chunk_sums, (size_t)reduce_chunks(N) * sizeof(double)));
  PA_TRY(dreserve(c, c->wave_tmp, (size_t)N * sizeof(float)));
  PA_TRY(dreserve(c, c->cnt_tmp, (size_t)N * 2 * sizeof(uint32_t)));
  const bool dbg_arrays = out->state_pre || out->lut_ij || out->is_glitch;
  if (dbg_arrays) {
    for (int i = 0; i < 3; ++i) PA_TRY(dreserve(c, c->dbg[i], c->n_events));
  }
  B.bins = (float4*)c->bins.p;
  B.part_blk = (uint32_t*)c->part_blk.p;
  B.part_counts = (uint32_t*)c->part_counts.p;
  B.tiles = (Tile*)c->tiles.p;
  B.heavy = (uint32_t*)c->heavy.p;
  B.p0_tot = (double*)c->p0_tot.p;
  B.p_out = (double*)c->p_out.p;
  B.chunk_sums = (double*)c->chunk_sums.p;
  B.wave = (float*)c->wave_tmp.p;
  B.cnt_ev = (uint32_t*)c->cnt_tmp.p;
  B.cnt_gl = (uint32_t*)c->cnt_tmp.p + N;
  for (int i = 0; i < 3; ++i) B.dbg[i] = dbg_arrays ? (uint8_t*)c->dbg[i].p : nullptr;
  if (plan.csr && !banded) {
    B.max_pieces = csr_max_pieces(c->n_events, G, plan.csr_heavy);
    PA_TRY(dreserve(c, c->pieces, (size_t)B.max_pieces * sizeof(Piece)));
    PA_TRY(dreserve(c, c->tile_ev, ((size_t)G + 1) * 2 * sizeof(uint64_t)));
    PA_TRY(dreserve(c, c->gslot, ((size_t)G + 1) * 2 * sizeof(uint4)));
    B.gslot = (uint4*)c->gslot.p;
    B.pieces = (Piece*)c->pieces.p;
    B.tile_ev = (uint64_t*)c->tile_ev.p;
  }
  PA_TRY(setup_gate_bufs(c, plan, out, B));
  if (plan.part_mode != PA_PART_EVENTS) {
    // the paper's (gate, window) thread partition
    PA_TRY(dreserve(c, c->w_ncyc, ((size_t)G + 1) * sizeof(uint32_t)));
    PA_TRY(dreserve(c, c->w_nthr, ((size_t)G + 1) * sizeof(uint32_t)));
    PA_TRY(dreserve(c, c->w_off, ((size_t)G + 1) * sizeof(uint64_t)));
    PA_TRY(dreserve(c, c->w_blk, ((size_t)band_scan_blocks(G) + 1) * sizeof(uint64_t)));
    PA_TRY(dreserve(c, c->w_tot, (size_t)kWinTotSlots * 4 * sizeof(double) + 256));
    if (plan.part_stats) PA_TRY(dreserve(c, c->w_hist, (size_t)kWinHistBins * sizeof(unsigned long long)));
    WinArgs w;
    w.mode = plan.part_mode;
    w.n_evt_tgt = plan.n_evt_tgt;
    w.n_thr_floor = plan.n_thr_floor;
    w.n_cyc_fix = plan.n_cyc_fix;
    w.ncyc = (uint32_t*)c->w_ncyc.p;
    w.nthr = (uint32_t*)c->w_nthr.p;
    w.thr_off = (uint64_t*)c->w_off.p;
    w.scan_blk = (uint64_t*)c->w_blk.p;
    w.tot_slots = (double*)c->w_tot.p;
    w.ev_max = (unsigned int*)((char*)c->w_tot.p + (size_t)kWinTotSlots * 4 * sizeof(double));
    w.hist = plan.part_stats ? (unsigned long long*)c->w_hist.p : nullptr;
    return run_pass(c, plan, B, out, "pa_run", nullptr, &w);
  }
  return run_pass(c, plan, B, out, "pa_run", banded ? &c->band : nullptr);
}

int pa_run_stream(pa_ctx* c, const pa_run_params* prm, const pa_events* ev, uint64_t chunk_events,
                  pa_result* out) {
  RunPlan plan;
  PA_TRY(check_run(c, prm, out, "pa_run_stream", &plan, true));
  if (!ev || !ev->pin_off || (ev->n_events && (!ev->t_ns || !ev->slew_ps)))
    return fail(c, PA_ERR_ARG, "pa_run_stream: null event pointer");
  if (ev->mem != PA_MEM_HOST) return fail(c, PA_ERR_ARG, "pa_run_stream: events must be host memory (PA_MEM_HOST)");
  if (ev->n_pins != c->n_pins)
    return fail(c, PA_ERR_ARG, "pa_run_stream: n_pins %llu != netlist pins %llu", (unsigned long long)ev->n_pins,
                (unsigned long long)c->n_pins);
  if (out->state_pre || out->lut_ij || out->is_glitch)
    return fail(c, PA_ERR_ARG, "pa_run_stream: per-event debug arrays are not available on a streamed run");
  CUDA_TRY(c, cudaSetDevice(c->device));
  return run_stream(c, plan, ev, chunk_events ? chunk_events : PA_STREAM_DEFAULT_CHUNK, out);
}

}  // extern "C"

// ----------------------------------------------------------------- pa_run_noalloc
//
// The per-run scratch of pa_run_noalloc: one file-scope device array, so the
// entry point never allocates. Its name is only meaningful in device code; the
// host takes its device address once per device with cudaGetSymbolAddress.
// Layout (each part 256-byte aligned): cycle bins {W, D, ev, gl} (float4) x
// PA_NOALLOC_MAX_CYCLES, per-block partition counts, the four partition
// counters, tiles and heavy-gate lists for PA_NOALLOC_MAX_GATES gates, P0 and
// totals (8 doubles), the four result powers, the final reduction's chunk
// sums, and staging for the waveform and the two count arrays.
// pa_create resolves the array's address (noalloc_lookup) and keeps it in the
// context; pa_run_noalloc only reads it.

namespace {

constexpr size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
constexpr size_t kNaMaxC = PA_NOALLOC_MAX_CYCLES, kNaMaxG = PA_NOALLOC_MAX_GATES;
constexpr size_t kNaBins = 0;
constexpr size_t kNaPartBlk = align256(kNaBins + kNaMaxC * sizeof(float4));
constexpr size_t kNaPartCounts = align256(kNaPartBlk + (kNaMaxG / 256 + 2) * 2 * sizeof(uint32_t));
constexpr size_t kNaTiles = align256(kNaPartCounts + 8 * sizeof(uint32_t));
constexpr size_t kNaHeavy = align256(kNaTiles + (kNaMaxG + 1) * sizeof(Tile));
constexpr size_t kNaP0Tot = align256(kNaHeavy + (kNaMaxG + 1) * sizeof(uint32_t));
constexpr size_t kNaPOut = align256(kNaP0Tot + 8 * sizeof(double));
constexpr size_t kNaChunks = align256(kNaPOut + 4 * sizeof(double));
constexpr size_t kNaWave = align256(kNaChunks + (kNaMaxC / kReduceChunk + 1) * sizeof(double));
constexpr size_t kNaCounts = align256(kNaWave + kNaMaxC * sizeof(float));
constexpr size_t kNaEnd = align256(kNaCounts + 2 * kNaMaxC * sizeof(uint32_t));
static_assert(kNaEnd <= (size_t)PA_NOALLOC_SCRATCH_BYTES, "no-alloc scratch layout exceeds its array");

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

namespace {

// The array's device address on the current device. Under lazy module loading
// this lookup is what loads the module holding the array, so the 5 MiB are
// committed here, once per context at pa_create, and never inside
// pa_run_noalloc. A failure is kept and reported by pa_run_noalloc: the
// other entry points do not need the array.
void noalloc_lookup(pa_ctx* c) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p) {
    cudaGetLastError();
    c->noalloc_base = nullptr;
    c->noalloc_err = std::string("cudaGetSymbolAddress of the scratch array at pa_create: ") +
                     (e != cudaSuccess ? cudaGetErrorString(e) : "null address");
    return;
  }
  c->noalloc_base = (unsigned char*)p;
}

}  // namespace

extern "C" int pa_run_noalloc(pa_ctx* c, const pa_run_params* prm, pa_result* out) {
  RunPlan plan;
  PA_TRY(check_run(c, prm, out, "pa_run_noalloc", &plan));
  if (plan.part_mode != PA_PART_EVENTS)
    return fail(c, PA_ERR_ARG, "pa_run_noalloc: part_mode must be PA_PART_EVENTS (the window partition allocates)");
  if (prm->n_cycles > PA_NOALLOC_MAX_CYCLES)
    return fail(c, PA_ERR_ARG, "pa_run_noalloc: n_cycles %u exceeds PA_NOALLOC_MAX_CYCLES (%u)", prm->n_cycles,
                PA_NOALLOC_MAX_CYCLES);
  if (c->n_gates > PA_NOALLOC_MAX_GATES)
    return fail(c, PA_ERR_ARG, "pa_run_noalloc: %u gates exceed PA_NOALLOC_MAX_GATES (%u)", c->n_gates,
                PA_NOALLOC_MAX_GATES);
  const bool any_array = out->waveform_w || out->event_count || out->glitch_count || out->state_pre ||
                         out->lut_ij || out->is_glitch || out->gate_power_w || out->cell_power_w;
  if (any_array && out->out_mem != PA_MEM_DEVICE)
    return fail(c, PA_ERR_ARG, "pa_run_noalloc: output arrays must be device memory (out_mem = PA_MEM_DEVICE)");
  if (out->cell_power_w && !out->gate_power_w)
    return fail(c, PA_ERR_ARG, "pa_run_noalloc: cell_power_w needs gate_power_w (the per-gate accumulators)");
  unsigned char* base = c->noalloc_base;
  if (!base) return fail(c, PA_ERR_CUDA, "pa_run_noalloc: %s", c->noalloc_err.c_str());
  CUDA_TRY(c, cudaSetDevice(c->device));
  PassBufs B;
  B.bins = (float4*)(base + kNaBins);
  B.part_blk = (uint32_t*)(base + kNaPartBlk);
  B.part_counts = (uint32_t*)(base + kNaPartCounts);
  B.tiles = (Tile*)(base + kNaTiles);
  B.heavy = (uint32_t*)(base + kNaHeavy);
  B.p0_tot = (double*)(base + kNaP0Tot);
  B.p_out = (double*)(base + kNaPOut);
  B.chunk_sums = (double*)(base + kNaChunks);
  B.wave = (float*)(base + kNaWave);
  B.cnt_ev = (uint32_t*)(base + kNaCounts);
  B.cnt_gl = (uint32_t*)(base + kNaCounts) + plan.N;
  // per-event debug outputs go straight to the caller's device arrays
  B.dbg[0] = out->state_pre;
  B.dbg[1] = out->lut_ij;
  B.dbg[2] = out->is_glitch;
  B.gate_e = out->gate_power_w;  // accumulated in place
  B.cell_p = out->cell_power_w;
  return run_pass(c, plan, B, out, "pa_run_noalloc", nullptr);
}

// ----------------------------------------------------------------- pa_build_bands

namespace {

// Read one device word back (after the stream's earlier work).
template <typename T>
int read_back(pa_ctx* c, const void* src, T* dst) {
  CUDA_TRY(c, cudaMemcpyAsync(dst, src, sizeof(T), cudaMemcpyDeviceToHost, c->stream));
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  return PA_OK;
}

int check_build_err(pa_ctx* c) {
  unsigned long long key = kNoErr;
  PA_TRY(read_back(c, c->err_word.p, &key));
  if (key != kNoErr) return map_dev_err(c, key, "pa_build_bands");
  return PA_OK;
}

void free_build_temps(pa_ctx* c) {
  DevBuf* tmp[] = {&c->b_bigf, &c->b_grank, &c->b_cnt, &c->b_evc, &c->b_ubase, &c->b_ebase, &c->b_uband,
                   &c->b_uoff, &c->b_flags, &c->b_ipos, &c->b_scan, &c->b_counters, &c->b_urec2,
                   &c->b_dense, &c->b_gflag};
  for (DevBuf* b : tmp) dfree(*b);
}

int build_bands(pa_ctx* c, float t_clk, uint32_t cb) {
  const uint64_t E = c->n_events;
  const uint32_t G = c->n_gates;
  const float c_last = E ? std::floor(c->t_last / t_clk) : 0.f;  // fp32 division, as the kernels take it
  if (!(c_last < 4294967040.f)) return fail(c, PA_ERR_ARG, "pa_build_bands: events span too many cycles");
  const uint32_t nb = (uint32_t)c_last / cb + 1;
  if (nb > kBandMaxBands)
    return fail(c, PA_ERR_ARG, "pa_build_bands: events span %u bands of %u cycles; at most %u", nb, cb, kBandMaxBands);
  uint32_t mb = 0;
  while ((1u << mb) < cb) ++mb;
  const uint64_t nbg = (uint64_t)nb * G;
  BandBuildArgs a;
  std::memset(&a, 0, sizeof(a));
  a.gates = (const GateRec*)c->gates.p;
  a.n_gates = G;
  a.n_events = E;
  a.pin_off = (const uint64_t*)c->pin_off.p;
  a.t = (const float*)c->t.p;
  a.s = (const float*)c->s.p;
  a.t_clk = t_clk;
  a.pow2 = is_pow2(t_clk);
  a.inv_t_clk = a.pow2 ? 1.0f / t_clk : 0.f;
  a.mb = mb;
  a.n_bands = nb;
  a.err = (unsigned long long*)c->err_word.p;
  a.cells = (const CellDesc*)c->cells.p;
  BandLayout& L = a.L;
  L.t_clk = t_clk;
  L.band_cycles = cb;
  L.mb = mb;
  L.n_bands = nb;
  // count: units and events per (band, gate), big gates
  PA_TRY(dreserve(c, c->b_big, ((size_t)G + 1) * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->b_counters, 4 * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->b_bigf, (size_t)G + 1));
  PA_TRY(dreserve(c, c->b_dense, ((size_t)G + 1) * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->b_gflag, (size_t)G + 1));
  PA_TRY(dreserve(c, c->b_grank, ((size_t)G + 1) * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->b_flags, ((size_t)G + 1) * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->b_ipos, ((size_t)G + 2) * sizeof(uint64_t)));
  PA_TRY(dreserve(c, c->b_cnt, (nbg + 1) * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->b_evc, (nbg + 1) * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->b_ubase, (nbg + 1) * sizeof(uint64_t)));
  PA_TRY(dreserve(c, c->b_ebase, (nbg + 1) * sizeof(uint64_t)));
  PA_TRY(dreserve(c, c->b_scan, ((size_t)band_scan_blocks(nbg) + 1) * sizeof(uint64_t)));
  L.big = (uint32_t*)c->b_big.p;
  a.counters = (uint32_t*)c->b_counters.p;
  a.bigf = (uint8_t*)c->b_bigf.p;
  a.dense = (uint32_t*)c->b_dense.p;
  a.gflag = (uint8_t*)c->b_gflag.p;
  a.grank = (uint32_t*)c->b_grank.p;
  a.flags = (uint32_t*)c->b_flags.p;
  a.ipos = (uint64_t*)c->b_ipos.p;
  a.cnt_gb = (uint32_t*)c->b_cnt.p;
  a.evc_gb = (uint32_t*)c->b_evc.p;
  a.ubase = (uint64_t*)c->b_ubase.p;
  a.ebase = (uint64_t*)c->b_ebase.p;
  a.scan_blk = (uint64_t*)c->b_scan.p;
  CUDA_TRY(c, cudaMemsetAsync(c->err_word.p, 0xff, sizeof(unsigned long long), c->stream));
  CUDA_TRY(c, band_build_count(a, c->stream));
  uint64_t n_units = 0, n_ev = 0;
  uint32_t counters[4] = {0, 0, 0, 0};
  CUDA_TRY(c, cudaMemcpyAsync(&n_units, a.ubase + nbg, sizeof(n_units), cudaMemcpyDeviceToHost, c->stream));
  CUDA_TRY(c, cudaMemcpyAsync(&n_ev, a.ebase + nbg, sizeof(n_ev), cudaMemcpyDeviceToHost, c->stream));
  CUDA_TRY(c, cudaMemcpyAsync(counters, a.counters, sizeof(counters), cudaMemcpyDeviceToHost, c->stream));
  CUDA_TRY(c, cudaStreamSynchronize(c->stream));
  PA_TRY(check_build_err(c));
  if (n_units >= 0xFFFFFFF0ull) return fail(c, PA_ERR_ARG, "pa_build_bands: too many units (%llu)", (unsigned long long)n_units);
  L.n_units = (uint32_t)n_units;
  L.n_ev = n_ev;
  L.n_big = counters[0];
  // units hold at most 5 * kUnitPinMax events; the bucket leaves room for the largest one
  if (counters[2] > (uint32_t)kUnitMaxEvents) return fail(c, PA_ERR_INTERNAL, "pa_build_bands: unit of %u events", counters[2]);
  a.item_bucket = (uint32_t)kItemEvents - 1u - std::max<uint32_t>(counters[2], 1u);
  // write: records, event copy, item heads
  const size_t nu = (size_t)n_units;
  const size_t ev_bytes = ((n_ev + 64) & ~(size_t)15) * sizeof(float);
  PA_TRY(dreserve(c, c->b_urec2, (nu + 1) * sizeof(uint2)));
  PA_TRY(dreserve(c, c->b_urec, (nu + 1) * sizeof(uint4)));
  PA_TRY(dreserve(c, c->b_btag, ((size_t)n_ev + 64) * sizeof(uint16_t)));
  PA_TRY(dreserve(c, c->b_ugate, (nu + 1) * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->b_uband, (nu + 1) * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->b_uoff, (nu + 1) * sizeof(uint64_t)));
  PA_TRY(dreserve(c, c->b_flags, (std::max<size_t>(nu, G) + 1) * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->b_ipos, (std::max<size_t>(nu + 1, (size_t)G + 2) + 1) * sizeof(uint64_t)));
  PA_TRY(dreserve(c, c->b_bt, ev_bytes));
  PA_TRY(dreserve(c, c->b_bs, ev_bytes));
  PA_TRY(dreserve(c, c->b_scan, ((size_t)band_scan_blocks(std::max<uint64_t>(nbg, nu)) + 1) * sizeof(uint64_t)));
  L.urec = (uint4*)c->b_urec.p;
  L.btag = (uint16_t*)c->b_btag.p;
  a.urec2 = (uint2*)c->b_urec2.p;
  L.ugate = (uint32_t*)c->b_ugate.p;
  L.bt = (float*)c->b_bt.p;
  L.bs = (float*)c->b_bs.p;
  a.uband = (uint32_t*)c->b_uband.p;
  a.uoff = (uint64_t*)c->b_uoff.p;
  a.flags = (uint32_t*)c->b_flags.p;
  a.ipos = (uint64_t*)c->b_ipos.p;
  a.scan_blk = (uint64_t*)c->b_scan.p;
  CUDA_TRY(c, band_build_write(a, c->stream));
  uint64_t n_items = 0;
  PA_TRY(read_back(c, a.ipos + nu, &n_items));
  PA_TRY(check_build_err(c));
  L.n_items = (uint32_t)n_items;
  // items
  PA_TRY(dreserve(c, c->b_items, ((size_t)n_items + 1) * sizeof(BandItem)));
  L.items = (BandItem*)c->b_items.p;
  CUDA_TRY(c, band_build_items(a, c->stream));
  PA_TRY(check_build_err(c));
  L.built = true;
  c->band = L;
  c->band_windowed = counters[1];
  return PA_OK;
}

}  // namespace

extern "C" int pa_build_bands(pa_ctx* c, float t_clk, uint32_t band_cycles) {
  if (!c) return PA_ERR_ARG;
  if (!c->has_ev) return fail(c, PA_ERR_ORDER, "pa_build_bands: events not loaded");
  if (!(t_clk > 0.f) || !is_finite_f(t_clk)) return fail(c, PA_ERR_ARG, "pa_build_bands: t_clk_ns must be > 0");
  const uint32_t cb = band_cycles ? band_cycles : kBandDefaultCycles;
  if (cb > kBandMaxCycles || (cb & (cb - 1)) != 0)
    return fail(c, PA_ERR_ARG, "pa_build_bands: band_cycles %u is not a power of two <= %u", cb, kBandMaxCycles);
  CUDA_TRY(c, cudaSetDevice(c->device));
  c->band.built = false;
  // The banded kernel stages the cell tables of at most kSmemCells cells in
  // shared memory; with a larger library no layout is built and runs at this
  // clock take the unbanded path (pa_result.path says which ran).
  if (c->n_cells > (uint32_t)kSmemCells) return PA_OK;
  const int rc = build_bands(c, t_clk, cb);
  free_build_temps(c);
  return rc;
}
