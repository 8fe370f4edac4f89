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
#include <mutex>
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
  long alloc_count = 0;
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};

  // library
  bool has_lib = false;
  uint32_t n_cells = 0;
  std::vector<CellDesc> h_cells;
  DevBuf cells, lut, leak;

  // netlist
  bool has_net = false;
  uint32_t n_gates = 0;
  uint64_t n_pins = 0;
  DevBuf gates;

  // events
  bool has_ev = false;
  uint64_t n_events = 0;
  float t_last = 0.f;  // latest event time
  DevBuf pin_off, gate_off, t, s;

  // scratch
  DevBuf value_tmp, err_word, tmax_bits;
  DevBuf bins, part_blk, part_counts, tiles, heavy, p0_tot, p_out;
  DevBuf dbg[3], wave_tmp, cnt_tmp;
  DevBuf scratch_small;
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
  const char* unit = code == kErrPinOff ? "pin" : (code == kErrTileOverflow ? "gate" : "event");
  return fail(c, rc, "%s: %s (first at %s %llu)", what, err_code_name(code), unit, idx);
}

bool is_pow2(float x) {
  int e;
  const float m = std::frexp(x, &e);
  return x > 0.f && m == 0.5f;
}

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
  *out = c;
  return PA_OK;
}

void pa_destroy(pa_ctx* c) {
  if (!c) return;
  cudaSetDevice(c->device);
  if (c->stream) cudaStreamSynchronize(c->stream);
  DevBuf* all[] = {&c->cells, &c->lut, &c->leak, &c->gates, &c->pin_off, &c->gate_off, &c->t, &c->s,
                   &c->value_tmp, &c->err_word, &c->tmax_bits, &c->bins, &c->part_blk,
                   &c->part_counts, &c->tiles, &c->heavy, &c->p0_tot, &c->p_out, &c->dbg[0],
                   &c->dbg[1], &c->dbg[2], &c->wave_tmp, &c->cnt_tmp, &c->scratch_small};
  for (DevBuf* b : all) dfree(*b);
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
  if (!c) return PA_ERR_ARG;
  if (!c->has_ev) return fail(c, PA_ERR_ORDER, "pa_run: events not loaded");
  if (!prm || !out) return fail(c, PA_ERR_ARG, "pa_run: null params or result");
  if (!(prm->t_clk_ns > 0.f) || !is_finite_f(prm->t_clk_ns)) return fail(c, PA_ERR_ARG, "pa_run: t_clk_ns must be > 0");
  if (prm->n_cycles == 0) return fail(c, PA_ERR_ARG, "pa_run: n_cycles must be > 0");
  if (!std::isfinite(prm->vdd)) return fail(c, PA_ERR_ARG, "pa_run: vdd not finite");
  if (out->out_mem != PA_MEM_HOST && out->out_mem != PA_MEM_DEVICE) return fail(c, PA_ERR_ARG, "pa_run: bad out_mem");
  const uint32_t tile = prm->tile_events ? prm->tile_events : kDefaultTile;
  const uint32_t heavy = prm->heavy_events ? prm->heavy_events : kDefaultHeavy;
  if ((uint64_t)tile + heavy > (uint64_t)kTileCap)
    return fail(c, PA_ERR_ARG, "pa_run: tile_events + heavy_events = %u exceeds %d", tile + heavy, kTileCap);
  const float T = prm->t_clk_ns;
  const double Td = (double)T;
  const double t_max = prm->t_max_ns > 0 ? prm->t_max_ns : (double)prm->n_cycles * Td;
  if (!std::isfinite(t_max)) return fail(c, PA_ERR_ARG, "pa_run: t_max not finite");
  if (c->n_events) {
    const float cyc = std::floor(c->t_last / T);  // fp32 division, as the kernels take it
    if (!(cyc < (float)prm->n_cycles))
      return fail(c, PA_ERR_RANGE, "pa_run: latest event t = %.9g ns lies in cycle %.0f >= n_cycles %u",
                  (double)c->t_last, (double)cyc, prm->n_cycles);
    if ((double)c->t_last > t_max)
      return fail(c, PA_ERR_RANGE, "pa_run: t_max %.9g ns is earlier than the latest event %.9g ns", t_max,
                  (double)c->t_last);
  }
  cudaSetDevice(c->device);
  const uint32_t N = prm->n_cycles;
  const uint32_t G = c->n_gates;
  const uint32_t nblk = partition_blocks(G);
  const bool debug = out->state_pre || out->lut_ij || out->is_glitch;
  const bool timing = (prm->flags & PA_RUN_TIMING) != 0;
  const bool pow2 = is_pow2(T);

  // scratch: bins [W f32 | D f32 | ev u32 | gl u32] x N
  PA_TRY(dreserve(c, c->bins, (size_t)N * 16));
  PA_TRY(dreserve(c, c->part_blk, (size_t)(nblk + 1) * 2 * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->part_counts, 4 * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->tiles, ((size_t)G + 1) * sizeof(Tile)));
  PA_TRY(dreserve(c, c->heavy, ((size_t)G + 1) * sizeof(uint32_t)));
  PA_TRY(dreserve(c, c->p0_tot, 8 * sizeof(double)));
  PA_TRY(dreserve(c, c->p_out, 4 * sizeof(double)));
  if (debug) {
    for (int i = 0; i < 3; ++i) PA_TRY(dreserve(c, c->dbg[i], c->n_events));
  }
  float* wave_dev = nullptr;
  if (out->waveform_w) {
    if (out->out_mem == PA_MEM_DEVICE) {
      wave_dev = out->waveform_w;
    } else {
      PA_TRY(dreserve(c, c->wave_tmp, (size_t)N * sizeof(float)));
      wave_dev = (float*)c->wave_tmp.p;
    }
  }
  uint8_t* bins = (uint8_t*)c->bins.p;
  RunArgs a;
  std::memset(&a, 0, sizeof(a));
  a.cells = (const CellDesc*)c->cells.p;
  a.n_cells = c->n_cells;
  a.lut = (const float*)c->lut.p;
  a.leak = (const float*)c->leak.p;
  a.gates = (const GateRec*)c->gates.p;
  a.n_gates = G;
  a.pin_off = (const uint64_t*)c->pin_off.p;
  a.gate_off = (const uint64_t*)c->gate_off.p;
  a.t = (const float*)c->t.p;
  a.s = (const float*)c->s.p;
  a.t_clk = T;
  a.inv_t_clk = pow2 ? 1.0f / T : 0.f;
  a.t_max_f = (float)t_max;
  a.half_vdd2 = (float)(0.5 * prm->vdd * prm->vdd);
  a.n_cycles = N;
  a.tile_target = tile;
  a.heavy_thresh = heavy;
  a.part_blk = (uint32_t*)c->part_blk.p;
  a.part_counts = (uint32_t*)c->part_counts.p;
  a.tiles = (Tile*)c->tiles.p;
  a.heavy = (uint32_t*)c->heavy.p;
  a.p0 = (double*)c->p0_tot.p;
  a.totals = (double*)c->p0_tot.p + 4;
  a.bin_w = (float*)bins;
  a.bin_d = (float*)(bins + (size_t)N * 4);
  a.bin_ev = (uint32_t*)(bins + (size_t)N * 8);
  a.bin_gl = (uint32_t*)(bins + (size_t)N * 12);
  a.err = (unsigned long long*)c->err_word.p;
  if (debug) {
    a.dbg_state = (uint8_t*)c->dbg[0].p;
    a.dbg_lut = (uint8_t*)c->dbg[1].p;
    a.dbg_glitch = (uint8_t*)c->dbg[2].p;
  }
  cudaStream_t st = c->stream;
  uint32_t launches = 0;
  if (timing) CUDA_TRY(c, cudaEventRecord(c->ev[0], st));
  CUDA_TRY(c, cudaMemsetAsync(c->bins.p, 0, (size_t)N * 16, st));
  CUDA_TRY(c, cudaMemsetAsync(c->p0_tot.p, 0, 8 * sizeof(double), st));
  CUDA_TRY(c, cudaMemsetAsync(c->part_counts.p, 0, 4 * sizeof(uint32_t), st));
  CUDA_TRY(c, cudaMemsetAsync(c->err_word.p, 0xff, sizeof(unsigned long long), st));
  CUDA_TRY(c, launch_partition(a, nblk, st));
  launches += nblk ? 3 : 0;
  if (timing) CUDA_TRY(c, cudaEventRecord(c->ev[1], st));
  const int grid = c->sm_count * fused_blocks_per_sm(pow2, debug);
  CUDA_TRY(c, launch_fused(a, grid, pow2, debug, st));
  launches += 1;
  if (timing) CUDA_TRY(c, cudaEventRecord(c->ev[2], st));
  CUDA_TRY(c, launch_final_reduce(a, Td, t_max, wave_dev, (double*)c->p_out.p, st));
  launches += 1;
  if (timing) CUDA_TRY(c, cudaEventRecord(c->ev[3], st));
  // outputs
  double p[4];
  unsigned long long key = kNoErr;
  uint32_t counts[4] = {0, 0, 0, 0};
  CUDA_TRY(c, cudaMemcpyAsync(p, c->p_out.p, sizeof(p), cudaMemcpyDeviceToHost, st));
  CUDA_TRY(c, cudaMemcpyAsync(&key, c->err_word.p, sizeof(key), cudaMemcpyDeviceToHost, st));
  CUDA_TRY(c, cudaMemcpyAsync(counts, c->part_counts.p, sizeof(counts), cudaMemcpyDeviceToHost, st));
  const cudaMemcpyKind dk = out->out_mem == PA_MEM_HOST ? cudaMemcpyDeviceToHost : cudaMemcpyDeviceToDevice;
  if (out->waveform_w && out->out_mem == PA_MEM_HOST)
    CUDA_TRY(c, cudaMemcpyAsync(out->waveform_w, wave_dev, (size_t)N * sizeof(float), dk, st));
  if (out->event_count) CUDA_TRY(c, cudaMemcpyAsync(out->event_count, a.bin_ev, (size_t)N * 4, dk, st));
  if (out->glitch_count) CUDA_TRY(c, cudaMemcpyAsync(out->glitch_count, a.bin_gl, (size_t)N * 4, dk, st));
  if (debug && c->n_events) {
    if (out->state_pre) CUDA_TRY(c, cudaMemcpyAsync(out->state_pre, c->dbg[0].p, c->n_events, dk, st));
    if (out->lut_ij) CUDA_TRY(c, cudaMemcpyAsync(out->lut_ij, c->dbg[1].p, c->n_events, dk, st));
    if (out->is_glitch) CUDA_TRY(c, cudaMemcpyAsync(out->is_glitch, c->dbg[2].p, c->n_events, dk, st));
  }
  CUDA_TRY(c, cudaStreamSynchronize(st));
  if (key != kNoErr) return map_dev_err(c, key, "pa_run");
  out->p_int_w = p[0];
  out->p_sw_w = p[1];
  out->p_gl_w = p[2];
  out->p_leak_w = p[3];
  out->t_max_ns = t_max;
  out->n_tiles = counts[0];
  out->n_heavy = counts[1];
  out->kernel_launches = launches;
  if (timing) {
    cudaEventElapsedTime(&out->ms_partition, c->ev[0], c->ev[1]);
    cudaEventElapsedTime(&out->ms_fused, c->ev[1], c->ev[2]);
    cudaEventElapsedTime(&out->ms_reduce, c->ev[2], c->ev[3]);
    cudaEventElapsedTime(&out->ms_total, c->ev[0], c->ev[3]);
  }
  return PA_OK;
}

}  // extern "C"

// ----------------------------------------------------------------- pa_run_noalloc
//
// The per-run scratch of pa_run_noalloc: one file-scope device array, so the
// entry point never allocates. Its name is only meaningful in device code; the
// host takes its device address once per device with cudaGetSymbolAddress.
// Layout (each part 256-byte aligned): cycle bins [W f32 | D f32 | ev u32 |
// gl u32] x PA_NOALLOC_MAX_CYCLES, per-block partition counts, the four
// partition counters, tiles and heavy-gate lists for PA_NOALLOC_MAX_GATES
// gates, P0 and totals (8 doubles) and the four result powers.

namespace {

constexpr size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
constexpr size_t kNaBins = 0;
constexpr size_t kNaPartBlk = align256(kNaBins + (size_t)PA_NOALLOC_MAX_CYCLES * 16);
constexpr size_t kNaPartCounts =
    align256(kNaPartBlk + ((size_t)PA_NOALLOC_MAX_GATES / 256 + 2) * 2 * sizeof(uint32_t));
constexpr size_t kNaTiles = align256(kNaPartCounts + 4 * sizeof(uint32_t));
constexpr size_t kNaHeavy = align256(kNaTiles + ((size_t)PA_NOALLOC_MAX_GATES + 1) * sizeof(Tile));
constexpr size_t kNaP0Tot = align256(kNaHeavy + ((size_t)PA_NOALLOC_MAX_GATES + 1) * sizeof(uint32_t));
constexpr size_t kNaPOut = align256(kNaP0Tot + 8 * sizeof(double));
constexpr size_t kNaEnd = align256(kNaPOut + 4 * sizeof(double));
static_assert(kNaEnd <= (size_t)PA_NOALLOC_SCRATCH_BYTES, "no-alloc scratch layout exceeds its array");

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kNaMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNaMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device `dev` (looked up
// once per device).
int noalloc_scratch(pa_ctx* c, int dev, unsigned char** out) {
  if (dev < 0 || dev >= kNaMaxDevices) return fail(c, PA_ERR_ARG, "pa_run_noalloc: device ordinal %d too large", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return fail(c, PA_ERR_CUDA, "pa_run_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = (unsigned char*)g_noalloc_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" int pa_run_noalloc(pa_ctx* c, const pa_run_params* prm, pa_result* out) {
  if (!c) return PA_ERR_ARG;
  if (!c->has_ev) return fail(c, PA_ERR_ORDER, "pa_run_noalloc: events not loaded");
  if (!prm || !out) return fail(c, PA_ERR_ARG, "pa_run_noalloc: null params or result");
  if (!(prm->t_clk_ns > 0.f) || !is_finite_f(prm->t_clk_ns))
    return fail(c, PA_ERR_ARG, "pa_run_noalloc: t_clk_ns must be > 0");
  if (prm->n_cycles == 0) return fail(c, PA_ERR_ARG, "pa_run_noalloc: n_cycles must be > 0");
  if (prm->n_cycles > PA_NOALLOC_MAX_CYCLES)
    return fail(c, PA_ERR_ARG, "pa_run_noalloc: n_cycles %u exceeds PA_NOALLOC_MAX_CYCLES (%u)", prm->n_cycles,
                PA_NOALLOC_MAX_CYCLES);
  if (c->n_gates > PA_NOALLOC_MAX_GATES)
    return fail(c, PA_ERR_ARG, "pa_run_noalloc: %u gates exceed PA_NOALLOC_MAX_GATES (%u)", c->n_gates,
                PA_NOALLOC_MAX_GATES);
  if (!std::isfinite(prm->vdd)) return fail(c, PA_ERR_ARG, "pa_run_noalloc: vdd not finite");
  const bool any_array = out->waveform_w || out->event_count || out->glitch_count || out->state_pre ||
                         out->lut_ij || out->is_glitch;
  if (any_array && out->out_mem != PA_MEM_DEVICE)
    return fail(c, PA_ERR_ARG, "pa_run_noalloc: output arrays must be device memory (out_mem = PA_MEM_DEVICE)");
  const uint32_t tile = prm->tile_events ? prm->tile_events : kDefaultTile;
  const uint32_t heavy = prm->heavy_events ? prm->heavy_events : kDefaultHeavy;
  if ((uint64_t)tile + heavy > (uint64_t)kTileCap)
    return fail(c, PA_ERR_ARG, "pa_run_noalloc: tile_events + heavy_events = %u exceeds %d", tile + heavy, kTileCap);
  const float T = prm->t_clk_ns;
  const double Td = (double)T;
  const double t_max = prm->t_max_ns > 0 ? prm->t_max_ns : (double)prm->n_cycles * Td;
  if (!std::isfinite(t_max)) return fail(c, PA_ERR_ARG, "pa_run_noalloc: t_max not finite");
  if (c->n_events) {
    const float cyc = std::floor(c->t_last / T);
    if (!(cyc < (float)prm->n_cycles))
      return fail(c, PA_ERR_RANGE, "pa_run_noalloc: latest event t = %.9g ns lies in cycle %.0f >= n_cycles %u",
                  (double)c->t_last, (double)cyc, prm->n_cycles);
    if ((double)c->t_last > t_max)
      return fail(c, PA_ERR_RANGE, "pa_run_noalloc: t_max %.9g ns is earlier than the latest event %.9g ns",
                  t_max, (double)c->t_last);
  }
  CUDA_TRY(c, cudaSetDevice(c->device));
  unsigned char* base = nullptr;
  PA_TRY(noalloc_scratch(c, c->device, &base));
  const uint32_t N = prm->n_cycles;
  const uint32_t G = c->n_gates;
  const uint32_t nblk = partition_blocks(G);
  const bool debug = out->state_pre || out->lut_ij || out->is_glitch;
  const bool timing = (prm->flags & PA_RUN_TIMING) != 0;
  const bool pow2 = is_pow2(T);
  RunArgs a;
  std::memset(&a, 0, sizeof(a));
  a.cells = (const CellDesc*)c->cells.p;
  a.n_cells = c->n_cells;
  a.lut = (const float*)c->lut.p;
  a.leak = (const float*)c->leak.p;
  a.gates = (const GateRec*)c->gates.p;
  a.n_gates = G;
  a.pin_off = (const uint64_t*)c->pin_off.p;
  a.gate_off = (const uint64_t*)c->gate_off.p;
  a.t = (const float*)c->t.p;
  a.s = (const float*)c->s.p;
  a.t_clk = T;
  a.inv_t_clk = pow2 ? 1.0f / T : 0.f;
  a.t_max_f = (float)t_max;
  a.half_vdd2 = (float)(0.5 * prm->vdd * prm->vdd);
  a.n_cycles = N;
  a.tile_target = tile;
  a.heavy_thresh = heavy;
  a.part_blk = (uint32_t*)(base + kNaPartBlk);
  a.part_counts = (uint32_t*)(base + kNaPartCounts);
  a.tiles = (Tile*)(base + kNaTiles);
  a.heavy = (uint32_t*)(base + kNaHeavy);
  a.p0 = (double*)(base + kNaP0Tot);
  a.totals = (double*)(base + kNaP0Tot) + 4;
  a.bin_w = (float*)(base + kNaBins);
  a.bin_d = (float*)(base + kNaBins + (size_t)N * 4);
  a.bin_ev = (uint32_t*)(base + kNaBins + (size_t)N * 8);
  a.bin_gl = (uint32_t*)(base + kNaBins + (size_t)N * 12);
  a.err = (unsigned long long*)c->err_word.p;
  if (debug) {
    a.dbg_state = out->state_pre;
    a.dbg_lut = out->lut_ij;
    a.dbg_glitch = out->is_glitch;
  }
  double* p_dev = (double*)(base + kNaPOut);
  cudaStream_t st = c->stream;
  uint32_t launches = 0;
  if (timing) CUDA_TRY(c, cudaEventRecord(c->ev[0], st));
  CUDA_TRY(c, cudaMemsetAsync(base + kNaBins, 0, (size_t)N * 16, st));
  CUDA_TRY(c, cudaMemsetAsync(base + kNaP0Tot, 0, 8 * sizeof(double), st));
  CUDA_TRY(c, cudaMemsetAsync(base + kNaPartCounts, 0, 4 * sizeof(uint32_t), st));
  CUDA_TRY(c, cudaMemsetAsync(c->err_word.p, 0xff, sizeof(unsigned long long), st));
  CUDA_TRY(c, launch_partition(a, nblk, st));
  launches += nblk ? 3 : 0;
  if (timing) CUDA_TRY(c, cudaEventRecord(c->ev[1], st));
  const int grid = c->sm_count * fused_blocks_per_sm(pow2, debug);
  CUDA_TRY(c, launch_fused(a, grid, pow2, debug, st));
  launches += 1;
  if (timing) CUDA_TRY(c, cudaEventRecord(c->ev[2], st));
  CUDA_TRY(c, launch_final_reduce(a, Td, t_max, out->waveform_w, p_dev, st));
  launches += 1;
  if (timing) CUDA_TRY(c, cudaEventRecord(c->ev[3], st));
  double p[4];
  unsigned long long key = kNoErr;
  uint32_t counts[4] = {0, 0, 0, 0};
  CUDA_TRY(c, cudaMemcpyAsync(p, p_dev, sizeof(p), cudaMemcpyDeviceToHost, st));
  CUDA_TRY(c, cudaMemcpyAsync(&key, c->err_word.p, sizeof(key), cudaMemcpyDeviceToHost, st));
  CUDA_TRY(c, cudaMemcpyAsync(counts, a.part_counts, sizeof(counts), cudaMemcpyDeviceToHost, st));
  if (out->event_count)
    CUDA_TRY(c, cudaMemcpyAsync(out->event_count, a.bin_ev, (size_t)N * 4, cudaMemcpyDeviceToDevice, st));
  if (out->glitch_count)
    CUDA_TRY(c, cudaMemcpyAsync(out->glitch_count, a.bin_gl, (size_t)N * 4, cudaMemcpyDeviceToDevice, st));
  CUDA_TRY(c, cudaStreamSynchronize(st));
  if (key != kNoErr) return map_dev_err(c, key, "pa_run_noalloc");
  out->p_int_w = p[0];
  out->p_sw_w = p[1];
  out->p_gl_w = p[2];
  out->p_leak_w = p[3];
  out->t_max_ns = t_max;
  out->n_tiles = counts[0];
  out->n_heavy = counts[1];
  out->kernel_launches = launches;
  if (timing) {
    cudaEventElapsedTime(&out->ms_partition, c->ev[0], c->ev[1]);
    cudaEventElapsedTime(&out->ms_fused, c->ev[1], c->ev[2]);
    cudaEventElapsedTime(&out->ms_reduce, c->ev[2], c->ev[3]);
    cudaEventElapsedTime(&out->ms_total, c->ev[0], c->ev[3]);
  }
  return PA_OK;
}
