// Seeded synthetic workload generator for gate-level time-based power analysis.
//
// This module only draws inputs: a cell library (NLDM-style internal-energy
// tables per gate state, leakage per state), a netlist (cell, output load,
// initial pin values) and per-pin event streams (sorted f32 timestamps in ns,
// slews in ps, toggling values) in the CSR-per-pin layout the power path takes.
// It holds none of the power arithmetic. Both the fp64 oracle and the CUDA path
// consume what it writes.
//
// Randomness: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC'11), implemented here from that definition.
// Every draw is keyed by (seed, config) and addressed by a counter built from
// (stream, gate, pin, index), so any gate block can be regenerated alone and
// the output does not depend on the thread count.
//
// The workload shapes follow the five configurations of the GPU time-based
// power analysis paper's evaluation scale (gates, cell mix, LUT size, cycles,
// events, activity skew, glitch share, bursts); the paper's real designs and
// activity files are not available, so these seeded inputs stand in for them.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------- Philox4x32-10
struct Ctr { uint32_t v[4]; };

inline void philox_round(uint32_t c[4], const uint32_t k[2]) {
  const uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
  const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
  const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
  const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
  const uint32_t n0 = hi1 ^ c[1] ^ k[0];
  const uint32_t n2 = hi0 ^ c[3] ^ k[1];
  c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
}

inline Ctr philox(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint64_t key64) {
  uint32_t c[4] = {c0, c1, c2, c3};
  uint32_t k[2] = {(uint32_t)key64, (uint32_t)(key64 >> 32)};
  for (int r = 0; r < 10; ++r) {
    philox_round(c, k);
    k[0] += 0x9E3779B9u;
    k[1] += 0xBB67AE85u;
  }
  return Ctr{{c[0], c[1], c[2], c[3]}};
}

inline double u01(uint32_t x) { return ((double)x + 0.5) * (1.0 / 4294967296.0); }

// Sequential stream of uniforms for one (stream, a, b) address.
struct Stream {
  uint64_t key; uint32_t s, a, b, i = 0; Ctr buf{}; int used = 4;
  Stream(uint64_t key_, uint32_t s_, uint32_t a_, uint32_t b_) : key(key_), s(s_), a(a_), b(b_) {}
  uint32_t next_u32() {
    if (used == 4) { buf = philox(s, a, b, i++, key); used = 0; }
    return buf.v[used++];
  }
  double uniform() { return u01(next_u32()); }
  double normal() {  // Box-Muller
    const double u1 = uniform(), u2 = uniform();
    return std::sqrt(-2.0 * std::log(u1)) * std::cos(6.283185307179586 * u2);
  }
};

enum : uint32_t {
  S_LIB = 1, S_GATE = 2, S_PERM = 3, S_PIN = 4, S_BURST = 5, S_GCYC = 6, S_RATE = 7
};

}  // namespace

extern "C" {

// Generation knobs. `config` 1..5 preloads the five standard workloads; fields
// set to a non-negative override value after synth_default() replace them.
typedef struct synth_cfg {
  int32_t  config;        // 1..5 standard workloads, 0 = fully custom
  uint64_t seed;
  int64_t  n_gates;
  int32_t  n_cells;
  int32_t  k_mode;        // 0: INV/NAND2/NOR2/XOR2 (k = 1,2,2,2); 1: k = 1 + c%4; 2: all k = 4
  int32_t  n_slew, n_load;
  int32_t  n_cycles;
  float    t_clk_ns;
  int64_t  n_events;
  int32_t  activity;      // 0: per-gate rate U[0.01, 0.2]; 1: Zipf-Mandelbrot (rank+q)^-s
  double   zipf_s;
  double   zipf_q;        // < 0: solve so the top 1% of gates carry `top1_share`
  double   top1_share;
  int32_t  slew_dist;     // 0: U[10, 200] ps; 1: lognormal, median 40 ps, sigma 0.5
  int32_t  load_dist;     // 0: U[1, 20] fF; 1: lognormal(mu = ln 5 fF, sigma = 0.6)
  double   pair_frac;     // share of events that are the second edge of a pulse pair
  double   pair_cycle_frac;  // > 0: pulse pairs only in this random share of cycles
  double   pair_w_lo_ns, pair_w_hi_ns;
  double   burst_frac;    // share of events drawn inside bursts
  int32_t  burst_width;   // cycles per burst
  double   burst_cover;   // share of cycles covered by bursts
  double   quantum_ns;    // > 0: snap times to multiples of this (forces cross-pin ties)
  double   vdd;
  int32_t  threads;       // 0 = hardware concurrency
  int32_t  toggles;       // > 0: every pin toggles exactly this many times in every cycle
                          // (high-activity stress waveforms; n_events follows from the netlist)
} synth_cfg;

typedef struct synth_stats {
  uint64_t n_pins, n_events;
  uint64_t max_gate_events, max_pin_events;
  double   top1_share;
  double   zipf_q;
  uint64_t glitch_events;     // events whose predecessor on the same pin is in the same cycle
  uint64_t max_pin_cycle_events;
  uint64_t heavy_events_over_2048;
} synth_stats;

}  // extern "C"

namespace {

struct Synth {
  synth_cfg cfg;
  uint64_t key;
  // library
  std::vector<uint8_t> k, ns, nl;
  std::vector<float> sax, lax;  // [n_cells * 8]
  std::vector<uint32_t> lut_off, leak_off;
  std::vector<float> lut, leak;
  // netlist
  std::vector<uint32_t> cell;
  std::vector<float> load;
  std::vector<uint8_t> init_in, init_out;
  std::vector<uint64_t> pin_base;  // [G + 1]
  // events
  std::vector<uint64_t> gate_n;    // per-gate event counts
  std::vector<uint64_t> pin_off;   // [P + 1]
  std::vector<uint32_t> burst_start, glitch_cycles;
  float limit = 0.f;               // smallest f32 whose cycle index is n_cycles
  synth_stats stats{};
};

int hw_threads(int req) {
  if (req > 0) return req;
  unsigned h = std::thread::hardware_concurrency();
  return h ? (int)h : 4;
}

template <class F>
void parallel_blocks(int64_t n, int64_t block, int threads, F f) {
  std::atomic<int64_t> next{0};
  auto worker = [&]() {
    for (;;) {
      const int64_t b = next.fetch_add(1);
      const int64_t lo = b * block;
      if (lo >= n) return;
      f(lo, std::min(n, lo + block));
    }
  };
  std::vector<std::thread> ts;
  for (int i = 1; i < threads; ++i) ts.emplace_back(worker);
  worker();
  for (auto& t : ts) t.join();
}

void set_defaults(synth_cfg* c, int config) {
  std::memset(c, 0, sizeof(*c));
  c->config = config;
  c->seed = 0;
  c->k_mode = 1; c->n_slew = 7; c->n_load = 7; c->t_clk_ns = 1.0f;
  c->activity = 0; c->zipf_s = 1.0; c->zipf_q = -1.0; c->top1_share = 0.5;
  c->slew_dist = 0; c->load_dist = 0;
  c->pair_frac = 0.0; c->pair_cycle_frac = 0.0; c->pair_w_lo_ns = 0.020; c->pair_w_hi_ns = 0.300;
  c->burst_frac = 0.0; c->burst_width = 20; c->burst_cover = 0.05;
  c->quantum_ns = 0.0; c->vdd = 0.9; c->threads = 0;
  switch (config) {
    case 1:  // tiny
      c->n_gates = 1000; c->n_cells = 4; c->k_mode = 0; c->n_cycles = 100; c->n_events = 10000;
      break;
    case 2:  // mid, uniform density, glitch pulses in ~5% of cycles
      c->n_gates = 100000; c->n_cells = 32; c->n_cycles = 1000; c->n_events = 10000000;
      c->pair_frac = 0.05; c->pair_cycle_frac = 0.05;
      break;
    case 3:  // large, skewed
      c->n_gates = 1000000; c->n_cells = 32; c->n_cycles = 10000; c->t_clk_ns = 0.8f;
      c->n_events = 200000000; c->activity = 1; c->zipf_s = 1.2; c->pair_frac = 0.15;
      c->load_dist = 1;
      break;
    case 4:  // very large, skewed
      c->n_gates = 5000000; c->n_cells = 64; c->n_slew = 8; c->n_load = 8; c->n_cycles = 100000;
      c->n_events = 1000000000; c->activity = 1; c->zipf_s = 1.1; c->slew_dist = 1; c->load_dist = 1;
      break;
    case 5:  // bursty stress
      c->n_gates = 10000000; c->n_cells = 64; c->k_mode = 2; c->n_slew = 8; c->n_load = 8;
      c->n_cycles = 50000; c->n_events = 2000000000; c->activity = 1; c->zipf_s = 1.3;
      c->slew_dist = 1; c->load_dist = 1; c->burst_frac = 0.8;
      break;
    case 6:  // waveform-bin stress: 100k cycles, every pin toggling 1, 2, 4 or 8 times per cycle
      c->n_gates = 1000; c->n_cells = 32; c->n_cycles = 100000; c->toggles = 4;
      break;
    default:  // custom: a small valid default
      c->n_gates = 16; c->n_cells = 4; c->n_cycles = 16; c->n_events = 200;
      break;
  }
}

inline int cell_k(const synth_cfg& c, int cell) {
  if (c.k_mode == 0) return cell % 4 == 0 ? 1 : 2;
  if (c.k_mode == 2) return 4;
  return 1 + cell % 4;
}

// Smallest f32 t >= 0 with floor(fl32(t / T)) >= n_cycles.
float cycle_limit(float T, int n_cycles) {
  float x = (float)((double)n_cycles * (double)T);
  auto cyc = [&](float t) { return (double)std::floor(t / T); };
  while (x > 0.f && cyc(std::nextafter(x, 0.f)) >= n_cycles) x = std::nextafter(x, 0.f);
  while (cyc(x) < n_cycles) x = std::nextafter(x, INFINITY);
  return x;
}

void build_library(Synth& S) {
  const synth_cfg& c = S.cfg;
  const int nc = c.n_cells;
  S.k.resize(nc); S.ns.resize(nc); S.nl.resize(nc);
  S.sax.assign((size_t)nc * 8, 0.f); S.lax.assign((size_t)nc * 8, 0.f);
  S.lut_off.resize(nc); S.leak_off.resize(nc);
  uint32_t lo = 0, ko = 0;
  for (int ci = 0; ci < nc; ++ci) {
    S.k[ci] = (uint8_t)cell_k(c, ci);
    S.ns[ci] = (uint8_t)c.n_slew; S.nl[ci] = (uint8_t)c.n_load;
    S.lut_off[ci] = lo; S.leak_off[ci] = ko;
    lo += (1u << S.k[ci]) * c.n_slew * c.n_load;
    ko += (1u << S.k[ci]);
  }
  S.lut.resize(lo); S.leak.resize(ko);
  for (int ci = 0; ci < nc; ++ci) {
    Stream r(S.key, S_LIB, (uint32_t)ci, 0);
    // Geometric axes, slew 5..500 ps and load 1..100 fF, with a small per-cell jitter
    // of the inner points so cells do not share identical axes.
    for (int a = 0; a < c.n_slew; ++a) {
      double f = (double)a / (c.n_slew - 1);
      if (a > 0 && a < c.n_slew - 1) f += (r.uniform() - 0.5) * 0.3 / (c.n_slew - 1);
      S.sax[ci * 8 + a] = (float)(5.0 * std::pow(100.0, f));
    }
    for (int a = 0; a < c.n_load; ++a) {
      double f = (double)a / (c.n_load - 1);
      if (a > 0 && a < c.n_load - 1) f += (r.uniform() - 0.5) * 0.3 / (c.n_load - 1);
      S.lax[ci * 8 + a] = (float)(1.0 * std::pow(100.0, f));
    }
    const double cs = 0.6 + 0.3 * r.uniform(), cl = 1.0 - cs;
    const double curv = 0.5 + r.uniform();
    const int nst = 1 << S.k[ci];
    for (int st = 0; st < nst; ++st) {
      const double scale = 0.7 + 0.6 * r.uniform();
      for (int i = 0; i < c.n_slew; ++i)
        for (int j = 0; j < c.n_load; ++j) {
          const double xs = std::log(S.sax[ci * 8 + i] / 5.0) / std::log(100.0);
          const double xl = std::log(S.lax[ci * 8 + j] / 1.0) / std::log(100.0);
          double v = 0.5 + 19.5 * (cs * std::pow(xs, curv) + cl * xl * (0.7 + 0.3 * xs));
          v *= scale;
          v = std::min(20.0, std::max(0.5, v));
          S.lut[S.lut_off[ci] + ((size_t)st * c.n_slew + i) * c.n_load + j] = (float)v;
        }
      S.leak[S.leak_off[ci] + st] = (float)(1.0 + 49.0 * r.uniform());
    }
  }
}

double zipf_sum(double a, double b, double s, double q) {
  // sum of (r + q)^-s for integer r in [a, b]: exact for the first ranks, midpoint integral after
  double tot = 0;
  double r = a;
  for (; r <= b && r < a + 20000; r += 1.0) tot += std::pow(r + q, -s);
  if (r <= b) {
    const double lo = r - 0.5 + q, hi = b + 0.5 + q;
    tot += (std::pow(lo, 1.0 - s) - std::pow(hi, 1.0 - s)) / (s - 1.0);
  }
  return tot;
}

double zipf_top1(int64_t G, double s, double q) {
  // fraction of weight on the top 1% of ranks for weights (r + q)^-s, r = 1..G
  const int64_t top = std::max<int64_t>(1, G / 100);
  const double a = zipf_sum(1.0, (double)top, s, q);
  return a / (a + zipf_sum((double)top + 1.0, (double)G, s, q));
}

double solve_q(int64_t G, double s, double share) {
  if (zipf_top1(G, s, 0.0) <= share) return 0.0;
  double lo = 0.0, hi = 1.0;
  while (zipf_top1(G, s, hi) > share) hi *= 2.0;
  for (int it = 0; it < 50; ++it) {
    const double mid = 0.5 * (lo + hi);
    if (zipf_top1(G, s, mid) > share) lo = mid; else hi = mid;
  }
  return 0.5 * (lo + hi);
}

void build_netlist_and_counts(Synth& S) {
  synth_cfg& c = S.cfg;
  const int64_t G = c.n_gates;
  const int threads = hw_threads(c.threads);
  S.cell.resize(G); S.load.resize(G); S.init_in.resize(G); S.init_out.resize(G);
  std::vector<double> w(G);
  parallel_blocks(G, 1 << 16, threads, [&](int64_t lo, int64_t hi) {
    for (int64_t g = lo; g < hi; ++g) {
      Stream r(S.key, S_GATE, (uint32_t)g, (uint32_t)(g >> 32));
      const uint32_t ci = r.next_u32() % (uint32_t)c.n_cells;
      S.cell[g] = ci;
      double L;
      if (c.load_dist == 0) L = 1.0 + 19.0 * r.uniform();
      else L = 5.0 * std::exp(0.6 * r.normal());
      S.load[g] = (float)L;
      const uint32_t bits = r.next_u32();
      S.init_in[g] = (uint8_t)(bits & ((1u << cell_k(c, (int)ci)) - 1));
      S.init_out[g] = (uint8_t)((bits >> 8) & 1);
      Stream rr(S.key, S_RATE, (uint32_t)g, (uint32_t)(g >> 32));
      w[g] = 0.01 + 0.19 * rr.uniform();
    }
  });
  if (c.activity == 1) {
    if (c.zipf_q < 0) c.zipf_q = solve_q(G, c.zipf_s, c.top1_share);
    // Random rank per gate: Fisher-Yates with counter-based draws.
    std::vector<uint32_t> rank(G);
    for (int64_t g = 0; g < G; ++g) rank[g] = (uint32_t)g;
    for (int64_t i = G - 1; i > 0; --i) {
      const Ctr x = philox(S_PERM, (uint32_t)i, (uint32_t)(i >> 32), 0, S.key);
      const uint64_t r64 = ((uint64_t)x.v[0] << 32) | x.v[1];
      const int64_t j = (int64_t)(r64 % (uint64_t)(i + 1));
      std::swap(rank[i], rank[j]);
    }
    for (int64_t g = 0; g < G; ++g) w[g] = std::pow((double)rank[g] + 1.0 + c.zipf_q, -c.zipf_s);
  }
  if (c.toggles > 0) {  // every pin: toggles events in each cycle
    int64_t tot_ev = 0;
    for (int64_t g = 0; g < G; ++g) tot_ev += (int64_t)(S.k[S.cell[g]] + 1) * c.toggles * (int64_t)c.n_cycles;
    c.n_events = tot_ev;
    S.cfg.n_events = tot_ev;
    for (int64_t g = 0; g < G; ++g) w[g] = (double)(S.k[S.cell[g]] + 1);
  }
  // Exact total: per-gate counts are differences of the rounded cumulative share.
  double tot = 0;
  for (int64_t g = 0; g < G; ++g) tot += w[g];
  S.gate_n.resize(G);
  double cum = 0;
  uint64_t prev = 0;
  for (int64_t g = 0; g < G; ++g) {
    cum += w[g];
    const uint64_t cur = (g == G - 1) ? (uint64_t)c.n_events
                                      : (uint64_t)std::llround((double)c.n_events * (cum / tot));
    S.gate_n[g] = cur - prev;
    prev = cur;
  }
  // Pin bases and per-pin counts.
  S.pin_base.resize(G + 1);
  uint64_t p = 0;
  for (int64_t g = 0; g < G; ++g) { S.pin_base[g] = p; p += (uint64_t)S.k[S.cell[g]] + 1; }
  S.pin_base[G] = p;
  S.pin_off.assign(p + 1, 0);
  parallel_blocks(G, 1 << 16, threads, [&](int64_t lo, int64_t hi) {
    for (int64_t g = lo; g < hi; ++g) {
      const int np = S.k[S.cell[g]] + 1;
      const uint64_t n = S.gate_n[g];
      const uint64_t base = n / np, rem = n % np;
      Stream r(S.key, S_PIN, (uint32_t)g, 0xFFFFFFFFu);
      const uint32_t start = r.next_u32() % (uint32_t)np;
      for (int q = 0; q < np; ++q) {
        const uint32_t d = ((uint32_t)q + (uint32_t)np - start) % (uint32_t)np;
        S.pin_off[S.pin_base[g] + q + 1] = base + (d < rem ? 1 : 0);
      }
    }
  });
  for (uint64_t i = 0; i < p; ++i) S.pin_off[i + 1] += S.pin_off[i];
  // Burst positions and glitch-carrying cycles.
  if (c.burst_frac > 0) {
    const int nb = std::max(1, (int)std::llround(c.burst_cover * c.n_cycles / c.burst_width));
    S.burst_start.resize(nb);
    for (int b = 0; b < nb; ++b) {
      const Ctr x = philox(S_BURST, (uint32_t)b, 0, 0, S.key);
      S.burst_start[b] = x.v[0] % (uint32_t)std::max(1, c.n_cycles - c.burst_width + 1);
    }
  }
  if (c.pair_cycle_frac > 0) {
    for (int cy = 0; cy < c.n_cycles; ++cy) {
      const Ctr x = philox(S_GCYC, (uint32_t)cy, 0, 0, S.key);
      if (u01(x.v[0]) < c.pair_cycle_frac) S.glitch_cycles.push_back((uint32_t)cy);
    }
    if (S.glitch_cycles.empty()) S.glitch_cycles.push_back(0);
  }
  S.limit = cycle_limit(c.t_clk_ns, c.n_cycles);
  // stats
  S.stats.n_pins = p; S.stats.n_events = (uint64_t)c.n_events; S.stats.zipf_q = c.zipf_q;
  std::vector<uint64_t> sorted(S.gate_n);
  std::sort(sorted.begin(), sorted.end(), std::greater<uint64_t>());
  const int64_t top = std::max<int64_t>(1, G / 100);
  uint64_t a = 0;
  for (int64_t i = 0; i < top; ++i) a += sorted[i];
  S.stats.top1_share = c.n_events ? (double)a / (double)c.n_events : 0.0;
  S.stats.max_gate_events = G ? sorted[0] : 0;
  uint64_t mp = 0, heavy = 0;
  for (uint64_t i = 0; i < p; ++i) mp = std::max(mp, S.pin_off[i + 1] - S.pin_off[i]);
  for (int64_t g = 0; g < G; ++g) if (S.gate_n[g] > 2048) heavy += S.gate_n[g];
  S.stats.max_pin_events = mp;
  S.stats.heavy_events_over_2048 = heavy;
}

struct Ev { double t; float s; };

// Fill the events of gates [g0, g1). Outputs are indexed by absolute event
// index minus `ev_base`.
void fill_gates(Synth& S, int64_t g0, int64_t g1, uint64_t ev_base, float* t_out, float* s_out,
                uint8_t* v_out, uint64_t* glitch_ctr, uint64_t* max_pc) {
  const synth_cfg& c = S.cfg;
  const double T = (double)c.t_clk_ns;
  const double window = (double)c.n_cycles * T;
  const float lim = S.limit;
  std::vector<Ev> buf;
  std::vector<float> tf;
  uint64_t glitches = 0, mpc = 0;
  for (int64_t g = g0; g < g1; ++g) {
    const int kk = S.k[S.cell[g]];
    for (int q = 0; q <= kk; ++q) {
      const uint64_t pin = S.pin_base[g] + q;
      const uint64_t a = S.pin_off[pin], n = S.pin_off[pin + 1] - a;
      if (n == 0) continue;
      Stream r(S.key, S_PIN, (uint32_t)g, (uint32_t)(q + 1) | ((uint32_t)(g >> 32) << 8));
      uint64_t pairs = 0;
      if (c.pair_frac > 0) {
        pairs = (uint64_t)std::floor(c.pair_frac * (double)n / 1.0 + r.uniform());
        pairs = std::min<uint64_t>(pairs, n / 2);
      }
      buf.clear();
      auto slew = [&]() -> float {
        if (c.slew_dist == 0) return (float)(10.0 + 190.0 * r.uniform());
        return (float)(40.0 * std::exp(0.5 * r.normal()));
      };
      auto draw_t = [&]() -> double {
        if (c.burst_frac > 0 && r.uniform() < c.burst_frac) {
          const uint32_t b = r.next_u32() % (uint32_t)S.burst_start.size();
          return ((double)S.burst_start[b] + r.uniform() * c.burst_width) * T;
        }
        return r.uniform() * window;
      };
      if (c.toggles > 0) {  // stress waveform: toggles events in every cycle, jittered
        pairs = 0;
        for (int64_t cy = 0; cy < c.n_cycles; ++cy)
          for (int j = 0; j < c.toggles; ++j)
            buf.push_back({((double)cy + ((double)j + 0.1 + 0.8 * r.uniform()) / c.toggles) * T, slew()});
      }
      for (uint64_t i = 0; c.toggles <= 0 && i < n - 2 * pairs; ++i) buf.push_back({draw_t(), slew()});
      for (uint64_t i = 0; i < pairs; ++i) {
        double t0;
        if (!S.glitch_cycles.empty()) {
          const uint32_t gc = S.glitch_cycles[r.next_u32() % (uint32_t)S.glitch_cycles.size()];
          t0 = ((double)gc + r.uniform()) * T;
        } else {
          t0 = draw_t();
        }
        const double w = c.pair_w_lo_ns + (c.pair_w_hi_ns - c.pair_w_lo_ns) * r.uniform();
        double t1 = t0 + w;
        if (t1 >= window) { t1 = t0; t0 = std::max(0.0, t0 - w); }
        buf.push_back({t0, slew()});
        buf.push_back({t1, slew()});
      }
      std::sort(buf.begin(), buf.end(), [](const Ev& x, const Ev& y) { return x.t < y.t; });
      // f32 (or quantum) rounding, then strictly increasing and below the window end.
      tf.resize(n);
      const double qn = c.quantum_ns;
      for (uint64_t i = 0; i < n; ++i) {
        double tt = buf[i].t;
        if (qn > 0) tt = std::floor(tt / qn) * qn;
        float f = (float)tt;
        if (i > 0 && !(f > tf[i - 1])) {
          if (qn > 0) {
            const double nx = std::floor((double)tf[i - 1] / qn + 1.5) * qn;
            f = (float)nx;
            if (!(f > tf[i - 1])) f = std::nextafter(tf[i - 1], INFINITY);
          } else {
            f = std::nextafter(tf[i - 1], INFINITY);
          }
        }
        tf[i] = f;
      }
      if (!(tf[n - 1] < lim)) {  // pull the tail back below the window end
        float hi = lim;
        for (int64_t i = (int64_t)n - 1; i >= 0; --i) {
          if (tf[i] < hi) break;
          tf[i] = std::nextafter(hi, 0.f);
          hi = tf[i];
        }
      }
      const uint8_t init = (q < kk) ? (uint8_t)((S.init_in[g] >> q) & 1) : S.init_out[g];
      int64_t prev_c = -1; uint64_t run = 0;
      for (uint64_t i = 0; i < n; ++i) {
        const uint64_t o = a + i - ev_base;
        t_out[o] = tf[i];
        s_out[o] = buf[i].s;
        if (v_out) v_out[o] = (uint8_t)(init ^ ((i + 1) & 1));
        const int64_t cy = (int64_t)std::floor(tf[i] / c.t_clk_ns);
        if (cy == prev_c) { ++glitches; ++run; } else { run = 1; prev_c = cy; }
        mpc = std::max<uint64_t>(mpc, run);
      }
    }
  }
  *glitch_ctr = glitches;
  *max_pc = mpc;
}

}  // namespace

extern "C" {

void synth_default(synth_cfg* c, int32_t config) { set_defaults(c, config); }

void* synth_create(const synth_cfg* cfg) {
  Synth* S = new Synth();
  S->cfg = *cfg;
  S->key = cfg->seed * 0x9E3779B97F4A7C15ull + (uint64_t)(cfg->config + 1) * 0xD1B54A32D192ED03ull;
  build_library(*S);
  build_netlist_and_counts(*S);
  return S;
}

void synth_destroy(void* h) { delete (Synth*)h; }

void synth_get_cfg(void* h, synth_cfg* out) { *out = ((Synth*)h)->cfg; }

void synth_sizes(void* h, uint32_t* n_cells, uint64_t* lut_len, uint64_t* leak_len, uint64_t* n_gates,
                 uint64_t* n_pins, uint64_t* n_events) {
  Synth* S = (Synth*)h;
  *n_cells = (uint32_t)S->cfg.n_cells;
  *lut_len = S->lut.size();
  *leak_len = S->leak.size();
  *n_gates = (uint64_t)S->cfg.n_gates;
  *n_pins = S->pin_base.back();
  *n_events = (uint64_t)S->cfg.n_events;
}

void synth_fill_library(void* h, uint8_t* k, uint8_t* ns, uint8_t* nl, float* sax, float* lax,
                        uint32_t* lut_off, float* lut, uint32_t* leak_off, float* leak) {
  Synth* S = (Synth*)h;
  std::memcpy(k, S->k.data(), S->k.size());
  std::memcpy(ns, S->ns.data(), S->ns.size());
  std::memcpy(nl, S->nl.data(), S->nl.size());
  std::memcpy(sax, S->sax.data(), S->sax.size() * 4);
  std::memcpy(lax, S->lax.data(), S->lax.size() * 4);
  std::memcpy(lut_off, S->lut_off.data(), S->lut_off.size() * 4);
  std::memcpy(lut, S->lut.data(), S->lut.size() * 4);
  std::memcpy(leak_off, S->leak_off.data(), S->leak_off.size() * 4);
  std::memcpy(leak, S->leak.data(), S->leak.size() * 4);
}

void synth_fill_netlist(void* h, uint32_t* cell, float* load, uint8_t* init_in, uint8_t* init_out) {
  Synth* S = (Synth*)h;
  const size_t G = S->cell.size();
  std::memcpy(cell, S->cell.data(), G * 4);
  std::memcpy(load, S->load.data(), G * 4);
  std::memcpy(init_in, S->init_in.data(), G);
  std::memcpy(init_out, S->init_out.data(), G);
}

// Fill pin offsets [P+1] and all events. value may be NULL.
void synth_fill_events(void* h, uint64_t* pin_off, float* t, float* slew, uint8_t* value,
                       synth_stats* stats) {
  Synth* S = (Synth*)h;
  const int64_t G = S->cfg.n_gates;
  std::memcpy(pin_off, S->pin_off.data(), S->pin_off.size() * 8);
  std::atomic<uint64_t> gl{0}, mpc{0};
  parallel_blocks(G, 4096, hw_threads(S->cfg.threads), [&](int64_t lo, int64_t hi) {
    uint64_t a = 0, m = 0;
    fill_gates(*S, lo, hi, 0, t, slew, value, &a, &m);
    gl += a;
    uint64_t cur = mpc.load();
    while (m > cur && !mpc.compare_exchange_weak(cur, m)) {}
  });
  S->stats.glitch_events = gl.load();
  S->stats.max_pin_cycle_events = mpc.load();
  if (stats) *stats = S->stats;
}

void synth_get_stats(void* h, synth_stats* stats) { *stats = ((Synth*)h)->stats; }

// Pin and event ranges of gates [g0, g1).
void synth_range(void* h, int64_t g0, int64_t g1, uint64_t* pin_lo, uint64_t* pin_hi, uint64_t* ev_lo,
                 uint64_t* ev_hi) {
  Synth* S = (Synth*)h;
  *pin_lo = S->pin_base[g0];
  *pin_hi = S->pin_base[g1];
  *ev_lo = S->pin_off[*pin_lo];
  *ev_hi = S->pin_off[*pin_hi];
}

// Events of gates [g0, g1) only, rebased: pin_off[0] = 0. Bit-identical to
// the same slice of synth_fill_events.
void synth_fill_range(void* h, int64_t g0, int64_t g1, uint64_t* pin_off, float* t, float* slew,
                      uint8_t* value) {
  Synth* S = (Synth*)h;
  const uint64_t p0 = S->pin_base[g0], p1 = S->pin_base[g1];
  const uint64_t e0 = S->pin_off[p0];
  for (uint64_t p = p0; p <= p1; ++p) pin_off[p - p0] = S->pin_off[p] - e0;
  parallel_blocks(g1 - g0, 1024, hw_threads(S->cfg.threads), [&](int64_t lo, int64_t hi) {
    uint64_t a = 0, m = 0;
    fill_gates(*S, g0 + lo, g0 + hi, e0, t, slew, value, &a, &m);
  });
}

}  // extern "C"
