/*
 * fp64 CPU oracle for gate-level time-based power analysis.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this. The product path never calls it and shares no
 * code or headers with it.
 *
 * What it computes follows "GPU-Accelerated Gate-Level Time-Based Power
 * Analysis via Event-Density-Aware Partitioning and Kernel Fusion":
 *   - Section 2.4.1 (Naive-D): per event, the preceding gate state selects the
 *     state-dependent NLDM internal-power LUT (Fig. 2), which is interpolated on
 *     input slew and output load; switching energy of an output transition
 *     (Eq. 1); clock-cycle glitch detection by counting events per pin and cycle,
 *     with the glitch energy scaled by r_gl (Eq. 2); contributions p = E / t_max
 *     (Eq. 3) and per-cycle waveform accumulation.
 *   - Section 2.4.2 (Naive-L): per gate, a k-way merge of the per-pin event
 *     streams; at each timestamp the state-indexed leakage (Fig. 3) holds over
 *     the preceding inter-event interval, E_leak = p_leak(S) * dt (Eq. 4); each
 *     interval is split at clock-cycle boundaries and added to every overlapped
 *     cycle bin in proportion to the overlap; after a timestamp, all events at
 *     that timestamp are applied to the state.
 *   - The fused kernel's per-timestamp loop (Fig. 7): every pin with an event at
 *     t_cur is processed against the same state S, and GlitchDetectUpdate keeps a
 *     per-pin event counter per clock cycle.
 *   - Per-gate power (the spatial comparison of the accuracy evaluation, which
 *     ranks gates by their power, Fig. 10): each gate's internal, switching,
 *     glitch and leakage energies summed on their own, over t_max.
 *
 * The extracted text of that paper lost its display equations. The readings
 * used where it is silent or stripped (each restated in the repository's design
 * notes):
 *   Eq. 1:   E_sw = 1/2 * C * V^2 per output transition, either direction.
 *   Eq. 2:   r_gl = min(1, pulse_width / ((rSlew + fSlew) / 2)), pulse width =
 *            time since the previous event on the same pin (ns -> ps), slews of
 *            the two edges of the pulse.
 *   Glitch:  counter reading -- the first event of a pin in a cycle is regular,
 *            the second and later are glitches; a glitch contributes only
 *            r_gl * (E_int + E_sw), to the glitch total and to its cycle bin.
 *            Alternative (glitch_mode 1, the other reading of the per-cycle
 *            glitch definition): every event of a pin-cycle holding two or
 *            more events is a glitch; the first one's pulse is the one it
 *            opens (width and slew of the next event on the pin).
 *   Eq. 1 alternative (esw_mode 1): C * V^2 on a rising output transition,
 *            nothing on a falling one (the supply charges the load once per
 *            rise; the same total over a rise/fall pair).
 *   Events:  input-pin events carry E_int only, output-pin events E_sw only;
 *            the gate state is the vector of input-pin values.
 *   Cycle:   c = floor(fl32(t / T)) with IEEE fp32 round-to-nearest division.
 *   Leakage: integrated over [0, t_max) including the intervals before the
 *            first and after the last event; t_max defaults to n_cycles * T.
 *   LUT:     interval index = largest axis index <= x, clamped to [0, n - 2];
 *            linear extrapolation outside the axes.
 *
 * Units: t in ns, slew in ps, load in fF, V in volts, LUT in fJ, leakage in nW.
 * Energies are accumulated in fJ (1 nW * 1 ns = 1e-3 fJ); powers are returned
 * in W (1 fJ / 1 ns = 1e-6 W).
 *
 * Everything is fp64 except the cycle-index division, which is fp32 by the
 * reading above. Gates are walked serially; with threads > 1 the gate range is
 * cut into contiguous blocks whose partial sums are added in block order.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int bad;            /* an event fell outside [0, n_cycles) */
  double e_int, e_sw, e_gl, e_leak;
  double *wave;       /* [n_bins] fJ */
  uint64_t *evc, *glc; /* [n_cycles] */
} acc_t;

typedef struct {
  const or_lib *lib;
  const or_net *net;
  const or_ev *ev;
  const or_par *par;
  or_out *out;
  const uint64_t *pin_base; /* [gate_end - gate_begin + 1] */
  const int32_t *bin_of;    /* [n_cycles] sample index or -1; NULL in full mode */
  const uint32_t *sorted;   /* sampled cycles, ascending and distinct (sample mode) */
  uint32_t n_sorted;
  uint32_t n_bins;
  double T;                 /* (double) t_clk */
  double t_max;
} ctx_t;

/* Bilinear interpolation of one state's table (Section 2.4.1, Fig. 2). */
static double bilerp(const float *tab, int ns, int nl, const float *sax, const float *lax, float s,
                     float l, int *oi, int *oj) {
  int i = 0, j = 0;
  for (int m = 1; m <= ns - 2; ++m)
    if (s >= sax[m]) i = m;
  for (int m = 1; m <= nl - 2; ++m)
    if (l >= lax[m]) j = m;
  const double u = ((double)s - (double)sax[i]) / ((double)sax[i + 1] - (double)sax[i]);
  const double v = ((double)l - (double)lax[j]) / ((double)lax[j + 1] - (double)lax[j]);
  const double q00 = tab[i * nl + j], q10 = tab[(i + 1) * nl + j];
  const double q01 = tab[i * nl + j + 1], q11 = tab[(i + 1) * nl + j + 1];
  *oi = i;
  *oj = j;
  return (1.0 - u) * (1.0 - v) * q00 + u * (1.0 - v) * q10 + (1.0 - u) * v * q01 + u * v * q11;
}

/* Leakage of one inter-event interval [a, b) at constant power p_nw (Eq. 4),
 * split at cycle boundaries into the bins it overlaps (Section 2.4.2). */
static void leak_interval(const ctx_t *X, acc_t *A, double p_nw, double a, double b) {
  if (!(b > a)) return;
  A->e_leak += p_nw * (b - a) * 1e-3;
  if (X->par->wave_mode == OR_WAVE_NONE) return;
  const double T = X->T;
  const int64_t n_cyc = (int64_t)X->par->n_cycles;
  int64_t c0 = (int64_t)floor(a / T);
  if (c0 < 0) c0 = 0;
  if (X->bin_of) {
    /* only the sampled cycles: first sampled cycle >= c0, then walk */
    uint32_t lo_i = 0, hi_i = X->n_sorted;
    while (lo_i < hi_i) {
      const uint32_t mid = (lo_i + hi_i) / 2;
      if ((int64_t)X->sorted[mid] < c0) lo_i = mid + 1; else hi_i = mid;
    }
    for (uint32_t i = lo_i; i < X->n_sorted; ++i) {
      const int64_t c = X->sorted[i];
      const double lo = (double)c * T, hi = (double)(c + 1) * T;
      if (lo >= b) break;
      const double ov = (b < hi ? b : hi) - (a > lo ? a : lo);
      if (ov > 0) A->wave[X->bin_of[c]] += p_nw * ov * 1e-3;
    }
    return;
  }
  for (int64_t c = c0; c < n_cyc; ++c) {
    const double lo = (double)c * T, hi = (double)(c + 1) * T;
    if (lo >= b) break;
    const double ov = (b < hi ? b : hi) - (a > lo ? a : lo);
    if (ov <= 0) continue;
    A->wave[c] += p_nw * ov * 1e-3;
  }
}

static void add_bin(const ctx_t *X, acc_t *A, int64_t c, double e) {
  if (X->par->wave_mode == OR_WAVE_NONE) return;
  if (X->bin_of) {
    const int32_t k = X->bin_of[c];
    if (k >= 0) A->wave[k] += e;
  } else {
    A->wave[c] += e;
  }
}

#define MAXP 9 /* up to 8 inputs + output */

static void run_gate1(const ctx_t *X, acc_t *A, uint64_t g);

/* One gate, its energies summed on their own first (they are the gate's
 * contribution to each total and, divided by t_max, its per-gate power). */
static void run_gate(const ctx_t *X, acc_t *A, uint64_t g) {
  acc_t G = *A;
  G.e_int = G.e_sw = G.e_gl = G.e_leak = 0.0;
  run_gate1(X, &G, g);
  A->bad |= G.bad;
  A->e_int += G.e_int;
  A->e_sw += G.e_sw;
  A->e_gl += G.e_gl;
  A->e_leak += G.e_leak;
  if (X->out->gate_power) {
    double *P = X->out->gate_power + (g - X->par->gate_begin) * 4;
    const double f = 1e-6 / X->t_max; /* fJ / ns -> W */
    P[0] = G.e_int * f;
    P[1] = G.e_sw * f;
    P[2] = G.e_gl * f;
    P[3] = G.e_leak * f;
  }
}

static void run_gate1(const ctx_t *X, acc_t *A, uint64_t g) {
  const or_lib *L = X->lib;
  const or_net *N = X->net;
  const or_ev *E = X->ev;
  const uint32_t cell = N->cell[g];
  const int k = L->k[cell];
  const int ns = L->ns[cell], nl = L->nl[cell];
  const float *sax = L->sax + (size_t)cell * 8, *lax = L->lax + (size_t)cell * 8;
  const float *lut = L->lut + L->lut_off[cell];
  const float *leak = L->leak + L->leak_off[cell];
  const float C = N->load[g];
  const double vdd = X->par->vdd;
  const float Tf = X->par->t_clk;
  const uint64_t pb = X->pin_base[g - X->par->gate_begin];

  unsigned S = (unsigned)N->init_in[g] & ((1u << k) - 1u);
  uint64_t cur[MAXP], end[MAXP], cnt[MAXP];
  int64_t cyc[MAXP];
  double last_t[MAXP];
  float last_s[MAXP];
  for (int p = 0; p <= k; ++p) {
    cur[p] = E->pin_off[pb + p];
    end[p] = E->pin_off[pb + p + 1];
    cyc[p] = -1;
    cnt[p] = 0;
    last_t[p] = 0.0;
    last_s[p] = 0.0f;
  }
  double t_prev = 0.0;
  for (;;) {
    /* next timestamp of the k-way merge */
    int any = 0;
    float tmin = 0.0f;
    for (int p = 0; p <= k; ++p)
      if (cur[p] < end[p] && (!any || E->t[cur[p]] < tmin)) {
        tmin = E->t[cur[p]];
        any = 1;
      }
    if (!any) break;
    const double t = (double)tmin;
    /* leakage of the interval that ends here, at the state before this timestamp */
    leak_interval(X, A, (double)leak[S], t_prev, t);
    /* every pin with an event at this timestamp, ascending pin index, same S */
    for (int p = 0; p <= k; ++p) {
      if (!(cur[p] < end[p] && E->t[cur[p]] == tmin)) continue;
      const uint64_t e = cur[p];
      const float s = E->slew[e];
      const int64_t ce = (int64_t)floorf(tmin / Tf);
      if (ce < 0 || ce >= (int64_t)X->par->n_cycles) {
        A->bad = 1;
        return;
      }
      if (ce != cyc[p]) {
        cyc[p] = ce;
        cnt[p] = 0;
      }
      cnt[p] += 1;
      A->evc[ce] += 1;
      double e_int = 0.0, e_sw = 0.0;
      int li = 0, lj = 0;
      if (p < k) {
        e_int = bilerp(lut + (size_t)S * ns * nl, ns, nl, sax, lax, s, C, &li, &lj);
      } else if (X->par->esw_mode == 0) {
        e_sw = 0.5 * (double)C * vdd * vdd;
      } else {
        /* new value of the output: given, else toggling from its initial value */
        const unsigned v = E->value ? (unsigned)(E->value[e] & 1)
                                    : ((unsigned)N->init_out[g] ^ (unsigned)((e - E->pin_off[pb + p] + 1) & 1));
        e_sw = v ? (double)C * vdd * vdd : 0.0;
      }
      const double e_dyn = e_int + e_sw;
      /* the pin's next event, if it lies in the same cycle (glitch_mode 1) */
      const int next_same = X->par->glitch_mode == 1 && e + 1 < end[p] &&
                            (int64_t)floorf(E->t[e + 1] / Tf) == ce;
      const int glitch = cnt[p] > 1 || (cnt[p] == 1 && next_same);
      if (glitch) {
        /* the pulse: the previous edge on the pin in this cycle, else the next */
        const int prev = cnt[p] > 1;
        const double t_o = prev ? last_t[p] : (double)E->t[e + 1];
        const float s_o = prev ? last_s[p] : E->slew[e + 1];
        const double pw_ps = (prev ? t - t_o : t_o - t) * 1000.0;
        const double avg_slew = ((double)s + (double)s_o) * 0.5;
        double r = pw_ps / avg_slew;
        if (r > 1.0) r = 1.0;
        A->e_gl += r * e_dyn;
        add_bin(X, A, ce, r * e_dyn);
        A->glc[ce] += 1;
      } else {
        A->e_int += e_int;
        A->e_sw += e_sw;
        add_bin(X, A, ce, e_dyn);
      }
      last_t[p] = t;
      last_s[p] = s;
      if (X->out->state_pre) X->out->state_pre[e] = (uint8_t)S;
      if (X->out->lut_ij) X->out->lut_ij[e] = p < k ? (uint8_t)((li << 4) | lj) : (uint8_t)0xFF;
      if (X->out->is_glitch) X->out->is_glitch[e] = (uint8_t)glitch;
    }
    /* apply all events of this timestamp to the state */
    for (int p = 0; p <= k; ++p) {
      if (!(cur[p] < end[p] && E->t[cur[p]] == tmin)) continue;
      if (p < k) {
        if (E->value)
          S = (S & ~(1u << p)) | ((unsigned)(E->value[cur[p]] & 1) << p);
        else
          S ^= 1u << p;
      }
      cur[p] += 1;
    }
    t_prev = t;
  }
  leak_interval(X, A, (double)leak[S], t_prev, X->t_max);
}

typedef struct {
  const ctx_t *X;
  acc_t acc;
  uint64_t g0, g1;
} job_t;

static void *run_block(void *arg) {
  job_t *J = (job_t *)arg;
  for (uint64_t g = J->g0; g < J->g1; ++g) run_gate(J->X, &J->acc, g);
  return NULL;
}

static int acc_init(acc_t *A, uint32_t n_bins, uint32_t n_cycles) {
  memset(A, 0, sizeof(*A));
  A->wave = (double *)calloc(n_bins ? n_bins : 1, sizeof(double));
  A->evc = (uint64_t *)calloc(n_cycles ? n_cycles : 1, sizeof(uint64_t));
  A->glc = (uint64_t *)calloc(n_cycles ? n_cycles : 1, sizeof(uint64_t));
  return A->wave && A->evc && A->glc ? 0 : -1;
}

static void acc_free(acc_t *A) {
  free(A->wave);
  free(A->evc);
  free(A->glc);
}

int or_run(const or_lib *lib, const or_net *net, const or_ev *ev, const or_par *par, or_out *out) {
  if (!lib || !net || !ev || !par || !out) return -1;
  if (par->gate_end < par->gate_begin || par->gate_end > net->n_gates) return -1;
  if (!(par->t_clk > 0.0f) || par->n_cycles == 0) return -1;
  ctx_t X;
  memset(&X, 0, sizeof(X));
  X.lib = lib;
  X.net = net;
  X.ev = ev;
  X.par = par;
  X.out = out;
  X.T = (double)par->t_clk;
  X.t_max = par->t_max > 0.0 ? par->t_max : (double)par->n_cycles * X.T;
  const uint64_t gb = par->gate_begin, ge = par->gate_end, ng = ge - gb;

  /* pin bases: gate g owns pins base .. base + k, inputs first, output last */
  uint64_t *pin_base = (uint64_t *)malloc((ng + 1) * sizeof(uint64_t));
  if (!pin_base) return -2;
  uint64_t p = 0;
  for (uint64_t g = 0; g < gb; ++g) p += (uint64_t)lib->k[net->cell[g]] + 1;
  for (uint64_t g = gb; g < ge; ++g) {
    pin_base[g - gb] = p;
    p += (uint64_t)lib->k[net->cell[g]] + 1;
  }
  pin_base[ng] = p;
  X.pin_base = pin_base;

  int32_t *bin_of = NULL;
  uint32_t *sorted = NULL;
  X.n_bins = par->n_cycles;
  if (par->wave_mode == OR_WAVE_SAMPLE) {
    bin_of = (int32_t *)malloc((size_t)par->n_cycles * sizeof(int32_t));
    sorted = (uint32_t *)malloc(((size_t)par->n_sample + 1) * sizeof(uint32_t));
    if (!bin_of || !sorted) {
      free(bin_of);
      free(sorted);
      free(pin_base);
      return -2;
    }
    for (uint32_t c = 0; c < par->n_cycles; ++c) bin_of[c] = -1;
    for (uint32_t i = 0; i < par->n_sample; ++i) {
      if (par->sample_cycles[i] >= par->n_cycles || bin_of[par->sample_cycles[i]] >= 0) {
        free(bin_of);
        free(sorted);
        free(pin_base);
        return -1; /* sampled cycles must be distinct and in range */
      }
      bin_of[par->sample_cycles[i]] = (int32_t)i;
    }
    uint32_t n = 0;
    for (uint32_t c = 0; c < par->n_cycles; ++c)
      if (bin_of[c] >= 0) sorted[n++] = c;
    X.bin_of = bin_of;
    X.sorted = sorted;
    X.n_sorted = n;
    X.n_bins = par->n_sample;
  }

  int nt = par->threads > 0 ? par->threads : 1;
  if ((uint64_t)nt > ng && ng > 0) nt = (int)ng;
  if (nt < 1) nt = 1;
  job_t *jobs = (job_t *)calloc((size_t)nt, sizeof(job_t));
  pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
  int rc = 0;
  for (int i = 0; i < nt; ++i) {
    jobs[i].X = &X;
    jobs[i].g0 = gb + ng * (uint64_t)i / (uint64_t)nt;
    jobs[i].g1 = gb + ng * (uint64_t)(i + 1) / (uint64_t)nt;
    if (acc_init(&jobs[i].acc, X.n_bins, par->n_cycles)) rc = -2;
  }
  if (rc == 0) {
    for (int i = 1; i < nt; ++i) pthread_create(&th[i], NULL, run_block, &jobs[i]);
    run_block(&jobs[0]);
    for (int i = 1; i < nt; ++i) pthread_join(th[i], NULL);
    /* reduce in block order */
    double e_int = 0, e_sw = 0, e_gl = 0, e_leak = 0;
    for (int i = 0; i < nt; ++i)
      if (jobs[i].acc.bad) rc = -3;
    for (int i = 0; i < nt; ++i) {
      e_int += jobs[i].acc.e_int;
      e_sw += jobs[i].acc.e_sw;
      e_gl += jobs[i].acc.e_gl;
      e_leak += jobs[i].acc.e_leak;
    }
    out->e_int = e_int;
    out->e_sw = e_sw;
    out->e_gl = e_gl;
    out->e_leak = e_leak;
    /* Eq. 3: p = E / t_max ; fJ / ns = 1e-6 W */
    out->p_int = e_int / X.t_max * 1e-6;
    out->p_sw = e_sw / X.t_max * 1e-6;
    out->p_gl = e_gl / X.t_max * 1e-6;
    out->p_leak = e_leak / X.t_max * 1e-6;
    out->t_max = X.t_max;
    if (out->wave_energy || out->waveform) {
      for (uint32_t b = 0; b < X.n_bins; ++b) {
        double w = 0;
        for (int i = 0; i < nt; ++i) w += jobs[i].acc.wave[b];
        if (out->wave_energy) out->wave_energy[b] = w;
        if (out->waveform) out->waveform[b] = w / X.T * 1e-6;
      }
    }
    if (out->evcount || out->glcount) {
      for (uint32_t c = 0; c < par->n_cycles; ++c) {
        uint64_t a = 0, b = 0;
        for (int i = 0; i < nt; ++i) {
          a += jobs[i].acc.evc[c];
          b += jobs[i].acc.glc[c];
        }
        if (out->evcount) out->evcount[c] = a;
        if (out->glcount) out->glcount[c] = b;
      }
    }
  }
  for (int i = 0; i < nt; ++i) acc_free(&jobs[i].acc);
  free(jobs);
  free(th);
  free(bin_of);
  free(sorted);
  free(pin_base);
  return rc;
}
