/*
 * fp64 CPU oracle for gate-level time-based power analysis.
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path. It shares no code
 * or headers with the CUDA library.
 */
#ifndef GLP_ORACLE_H
#define GLP_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct or_lib {
  uint32_t n_cells;
  const uint8_t *k, *ns, *nl;  /* inputs, slew points, load points per cell */
  const float *sax, *lax;      /* [n_cells * 8] axes (ps, fF) */
  const uint32_t *lut_off;     /* cell table: [2^k][ns][nl] fJ */
  const float *lut;
  const uint32_t *leak_off;    /* cell leakage: [2^k] nW */
  const float *leak;
} or_lib;

typedef struct or_net {
  uint64_t n_gates;
  const uint32_t *cell;
  const float *load;
  const uint8_t *init_in, *init_out;
} or_net;

typedef struct or_ev {
  uint64_t n_pins;
  const uint64_t *pin_off; /* [n_pins + 1] */
  const float *t;          /* ns */
  const float *slew;       /* ps */
  const uint8_t *value;    /* new value per event, or NULL (toggle) */
} or_ev;

enum { OR_WAVE_FULL = 0, OR_WAVE_NONE = 1, OR_WAVE_SAMPLE = 2 };

typedef struct or_par {
  double vdd;
  float t_clk;
  uint32_t n_cycles;
  double t_max;                  /* 0 -> n_cycles * t_clk */
  int32_t wave_mode;             /* OR_WAVE_* */
  const uint32_t *sample_cycles; /* OR_WAVE_SAMPLE: bins to compute */
  uint32_t n_sample;
  uint64_t gate_begin, gate_end; /* gates to walk */
  int32_t threads;
  int32_t glitch_mode;           /* 0: counter reading (2nd and later events of a pin in a
                                    cycle); 1: every event of a pin-cycle with 2+ events */
  int32_t esw_mode;              /* 0: C V^2 / 2 per output transition; 1: C V^2 on a rising
                                    output transition, 0 on a falling one */
} or_par;

typedef struct or_out {
  double e_int, e_sw, e_gl, e_leak; /* fJ */
  double p_int, p_sw, p_gl, p_leak; /* W */
  double t_max;                     /* ns */
  double *wave_energy;              /* [bins] fJ or NULL */
  double *waveform;                 /* [bins] W or NULL */
  uint64_t *evcount, *glcount;      /* [n_cycles] or NULL */
  uint8_t *state_pre;               /* [E] input state before the event's timestamp */
  uint8_t *lut_ij;                  /* [E] (i << 4) | j for input events, 0xFF for output */
  uint8_t *is_glitch;               /* [E] */
  double *gate_power;               /* [(gate_end - gate_begin) * 4] W per gate: int, sw, gl, leak; or NULL */
} or_out;

int or_run(const or_lib *lib, const or_net *net, const or_ev *ev, const or_par *par, or_out *out);

#ifdef __cplusplus
}
#endif
#endif
