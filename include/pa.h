/*
 * pa.h -- gate-level time-based power analysis on one GB300 (sm_103a).
 *
 * C ABI of libpa.so. The operation is the power-computation step of "GPU-
 * Accelerated Gate-Level Time-Based Power Analysis via Event-Density-Aware
 * Partitioning and Kernel Fusion":
 *   - per-event dynamic power (Section 2.4.1, Fig. 2): the gate state before
 *     the event's timestamp selects the state-dependent NLDM internal-power
 *     table, which is bilinearly interpolated on input slew and output load;
 *     switching energy of an output transition from load and supply (Eq. 1);
 *     clock-cycle glitch detection (more than one event on a pin within a
 *     cycle) with the glitch energy scaled by r_gl (Eq. 2); each contribution
 *     p = E / t_max (Eq. 3) goes to the design-level internal, switching and
 *     glitch totals and to the per-cycle power waveform;
 *   - per-gate leakage (Section 2.4.2, Fig. 3): k-way merge of the per-pin
 *     event streams, state-indexed leakage held over each inter-event interval
 *     (Eq. 4), each interval split across cycle bins in proportion to overlap;
 *   - fused into one pass as in the fused kernel of Fig. 7 (all pins with an
 *     event at t_cur see the same state S; per-pin event counter per cycle).
 *
 * Readings where the extracted text of the paper lost its equations:
 *   E_sw = 1/2 * C * V^2 per output transition (rise or fall);
 *   r_gl = min(1, pulse_width / ((rSlew + fSlew) / 2)), pulse width = time since
 *     the previous event on the same pin, slews of the pulse's two edges;
 *   the first event of a pin in a cycle is regular, the 2nd and later in that
 *     cycle are glitches and contribute only r_gl * (E_int + E_sw);
 *   input-pin events carry E_int, output-pin events E_sw; the gate state is
 *     the vector of input-pin values (bit j = input j);
 *   cycle of an event c = floor(fl32(t / t_clk)), IEEE fp32 division;
 *   leakage is integrated over [0, t_max) including the intervals before the
 *     first and after the last event; t_max defaults to n_cycles * t_clk.
 *
 * Units: time ns, slew ps, load fF, vdd V, internal energy fJ, leakage nW;
 * results in W.
 *
 * Threading: a pa_ctx is used by one host thread at a time. Every call is
 * synchronous with respect to the host: when it returns, its device work on
 * the context's stream has completed.
 *
 * Errors: every int-returning call returns PA_OK (0) or a negative PA_ERR_*.
 * No C++ exception crosses the ABI. pa_last_error() describes the most recent
 * failure (first offending pin/event for validation errors). Outputs are
 * written only on PA_OK.
 */
#ifndef PA_H
#define PA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_VERSION 3

#define PA_OK 0
#define PA_ERR_ARG (-1)      /* null pointer, bad size, bad axis, bad parameter      */
#define PA_ERR_ORDER (-2)    /* library -> netlist -> events -> run order violated    */
#define PA_ERR_UNSORTED (-3) /* a pin's event times are not strictly increasing       */
#define PA_ERR_RANGE (-4)    /* t < 0, t not finite, slew <= 0, cell id out of range,
                                event cycle >= n_cycles, t_max earlier than an event  */
#define PA_ERR_TOGGLE (-5)   /* an event's value equals the pin's previous value      */
#define PA_ERR_OOM (-6)      /* device or host allocation failed                     */
#define PA_ERR_CUDA (-7)     /* a CUDA runtime call failed                           */
#define PA_ERR_INTERNAL (-8) /* a device-side consistency check failed, or a bounded
                                device-side wait gave up (pa_last_error says which)  */

#define PA_MEM_HOST 0   /* pointers are host memory (pageable or pinned)   */
#define PA_MEM_DEVICE 1 /* pointers are device memory on the ctx's device  */

#define PA_MAX_INPUTS 4 /* k, inputs per cell: 1..4 (2^k gate states)       */
#define PA_MAX_AXIS 8   /* LUT axis points per dimension: 2..8              */

typedef struct pa_ctx pa_ctx;

/*
 * Cell library (Section 2.4.1 Fig. 2; Section 2.4.2 Fig. 3). Host memory,
 * copied by pa_load_library; the caller keeps ownership.
 *   n_inputs[c]          k in [1, 4]; cell c has 2^k states, state bit j = input j
 *   n_slew[c], n_load[c] axis lengths in [2, 8]
 *   slew_axis[c*8 + i]   ps, strictly increasing over i < n_slew[c]
 *   load_axis[c*8 + j]   fF, strictly increasing over j < n_load[c]
 *   lut[lut_off[c] + (S*n_slew[c] + i)*n_load[c] + j]   fJ, internal energy
 *                        of an input transition in state S at (slew_i, load_j)
 *   leak[leak_off[c] + S]  nW, leakage power in state S
 * Interpolation: interval index = largest axis index <= x clamped to
 * [0, n - 2]; linear extrapolation outside the axes.
 */
typedef struct pa_library {
  uint32_t n_cells;
  const uint8_t *n_inputs;
  const uint8_t *n_slew;
  const uint8_t *n_load;
  const float *slew_axis;
  const float *load_axis;
  const uint32_t *lut_off;
  const float *lut;
  uint64_t lut_len;
  const uint32_t *leak_off;
  const float *leak;
  uint64_t leak_len;
} pa_library;

/*
 * Netlist. Host memory, copied by pa_load_netlist (requires a library).
 * Gate g is an instance of cell_id[g] with k = n_inputs[cell_id[g]] inputs; it
 * owns pins pin_base(g) .. pin_base(g) + k where pin_base(g) = sum over g' < g
 * of (k(g') + 1): inputs 0..k-1 first, the output pin last.
 *   load_ff[g]   total output load capacitance (load pins + interconnect), fF
 *   init_in[g]   initial input values, bit j = input j
 *   init_out[g]  initial output value, 0 or 1
 */
typedef struct pa_netlist {
  uint32_t n_gates;
  const uint32_t *cell_id;
  const float *load_ff;
  const uint8_t *init_in;
  const uint8_t *init_out;
} pa_netlist;

/*
 * Per-pin event streams in CSR form (requires a netlist).
 *   pin_off[n_pins + 1]  events of pin p are [pin_off[p], pin_off[p+1]);
 *                        pin_off[0] = 0, pin_off[n_pins] = n_events;
 *                        n_pins must equal the netlist's pin count
 *   t_ns[e]              event time, finite, >= 0, strictly increasing per pin
 *   slew_ps[e]           transition time, finite, > 0
 *   value[e]             new logic value (0/1), must differ from the pin's
 *                        previous value; NULL means every event toggles
 * mem = PA_MEM_HOST: host arrays, copied. PA_MEM_DEVICE: device arrays on the
 * ctx's device; copied on the device, so the caller may free them after the
 * call. Device arrays must be complete when the call is made: the ctx's
 * stream does not wait on other streams. Either way the library keeps its own padded copy of pin_off, t_ns and
 * slew_ps until the next pa_load_events or pa_destroy.
 */
typedef struct pa_events {
  uint64_t n_pins;
  uint64_t n_events;
  const uint64_t *pin_off;
  const float *t_ns;
  const float *slew_ps;
  const uint8_t *value;
  int32_t mem;
} pa_events;

#define PA_RUN_TIMING 1u /* record per-kernel CUDA-event times in pa_result */
/* Alternative readings of the paper's stripped definitions (ablations; the
 * defaults are the readings listed at the top of this header):
 *   PA_RUN_GLITCH_ALL  every event of a pin-cycle holding two or more events
 *                      is a glitch; the first one takes the pulse it opens
 *                      (width and slew of the pin's next event);
 *   PA_RUN_ESW_RISE    switching energy C * V^2 on a rising output transition
 *                      and none on a falling one (Eq. 1 read per charge).
 * Either flag selects the slower per-event path (as debug outputs do). */
#define PA_RUN_GLITCH_ALL 2u
#define PA_RUN_ESW_RISE 4u
/* With part_mode PA_PART_DENSITY or PA_PART_FIXED: count the events of every
 * (gate, window) thread and report their quantiles in pa_result (a slower
 * run; leave it off when timing the partition). */
#define PA_RUN_PART_STATS 8u

/* Work partitions (pa_run_params.part_mode). The results do not depend on the
 * partition beyond floating-point summation order; the paper's two partitions
 * are there to compare them (Figs. 5, 19 and 20: event-density-aware per-gate
 * cycle windows against one globally fixed window length), on one kernel that
 * runs one thread per (gate, window) and adds every event to the cycle bins
 * with a global atomic, as the paper's fused kernel does.
 *   PA_PART_EVENTS   the library's own event-count partition (default): the
 *                    banded layout if one is built for this clock, else
 *                    event-count tiles of the CSR arrays;
 *   PA_PART_DENSITY  per gate g: rho = N_evt^(g) / n_cycles, n_cyc,floor =
 *                    ceil(n_cycles / n_thr_floor), rho_floor = n_evt_tgt /
 *                    n_cyc,floor, n_cyc^(g) = floor(n_evt_tgt / (rho +
 *                    rho_floor) + 1/2) clamped to [1, n_cycles] (fp64);
 *   PA_PART_FIXED    n_cyc^(g) = min(n_cyc_fix, n_cycles) for every gate.
 * Thread tau of gate g takes the events whose cycle floor(fl32(t / t_clk))
 * lies in [tau n_cyc^(g), (tau + 1) n_cyc^(g)); a gate has
 * ceil(n_cycles / n_cyc^(g)) threads, gates without events included. */
#define PA_PART_EVENTS 0u
#define PA_PART_DENSITY 1u
#define PA_PART_FIXED 2u

/*
 * Run parameters. pa_default_params() fills the defaults.
 *   vdd            supply voltage, V
 *   t_clk_ns       clock period, ns (> 0)
 *   n_cycles       cycle bins (> 0); every event needs floor(fl32(t/t_clk)) < n_cycles
 *   t_max_ns       analysis window end for Eq. 3 and leakage; 0 -> n_cycles * t_clk;
 *                  otherwise it must be >= the latest event time
 *   tile_events    work partition: target events per light tile (0 = default:
 *                  320 for the warp kernel, 2048 for the CTA kernel)
 *   heavy_events   gates with more events than this are heavy (0 = default: 64
 *                  / 2048): cut into time pieces of about 2048 events, each
 *                  worked through by one warp in windows (warp kernel), or
 *                  streamed in event-count windows by one CTA (CTA kernel);
 *                  tile_events + heavy_events must not exceed 4096. The run on
 *                  the per-pin layout takes the warp kernel when it asks for
 *                  no per-event output (state_pre, lut_ij, is_glitch,
 *                  gate_power_w, cell_power_w, the alternative readings),
 *                  the library has at most 64 cells and tile_events +
 *                  heavy_events (defaults resolved) is at most 448; else the
 *                  CTA kernel. pa_run_noalloc always takes the CTA kernel.
 *   flags          PA_RUN_* bits
 *   part_mode      PA_PART_* (pa_run only; the other entry points take
 *                  PA_PART_EVENTS)
 *   n_evt_tgt      PA_PART_DENSITY: target events per thread (0 = 8, the paper's)
 *   n_thr_floor    PA_PART_DENSITY: parallelism floor N_thr,floor (0 = 1)
 *   n_cyc_fix      PA_PART_FIXED: cycles per thread (0 = 1)
 * The partition knobs change only how work is cut, never the results beyond
 * floating-point summation order.
 */
typedef struct pa_run_params {
  double vdd;
  float t_clk_ns;
  uint32_t n_cycles;
  double t_max_ns;
  uint32_t tile_events;
  uint32_t heavy_events;
  uint32_t flags;
  uint32_t part_mode;
  uint32_t n_evt_tgt;
  uint32_t n_thr_floor;
  uint32_t n_cyc_fix;
} pa_run_params;

/*
 * Results. Scalars are outputs; array pointers are caller-owned inputs (NULL =
 * not wanted), host or device memory per out_mem.
 *   waveform_w[n_cycles]    per-cycle power, W (energy in the cycle / t_clk)
 *   event_count[n_cycles]   events per cycle
 *   glitch_count[n_cycles]  glitch events per cycle
 *   state_pre[n_events]     per event: input state before its timestamp (debug)
 *   lut_ij[n_events]        per input event: (i << 4) | j of the LUT interval;
 *                           0xFF for output events (debug)
 *   is_glitch[n_events]     per event: 1 if a glitch (debug)
 *   gate_power_w[n_gates * 4]  per gate g at [4g .. 4g + 3]: its internal,
 *                           switching, glitch and leakage power, W (double); over
 *                           all gates the four sum to p_int_w .. p_leak_w. This
 *                           is the per-gate view the paper's accuracy study ranks
 *                           gates by (Kendall's Tau of gate power, Fig. 10). With
 *                           out_mem = PA_MEM_DEVICE the array itself accumulates
 *                           the gate energies, so after an error it may hold
 *                           partial values.
 *   cell_power_w[n_cells * 4]  per library cell c at [4c .. 4c + 3]: the sum of
 *                           gate_power over the gates that instantiate it (W,
 *                           double); may be asked for with or without
 *                           gate_power_w.
 * The per-event debug arrays, gate_power_w and cell_power_w take a slower per-event path
 * (one event per lane, extra global writes); ask for them only when needed.
 * With PA_RUN_TIMING, ms_* hold CUDA-event times of the partition, fused and
 * reduction kernels and of the whole device pass. n_tiles / n_heavy count the
 * work items (light tiles / heavy items: heavy gates for the CTA kernel, heavy
 * gates' pieces for the warp kernel); path says which kernel ran.
 * With part_mode PA_PART_DENSITY or PA_PART_FIXED, part_threads is the number
 * of (gate, window) threads, and with PA_RUN_PART_STATS the part_evt_* hold
 * the nearest-rank 50th, 90th and 99th percentiles and the maximum of the
 * events per thread (the smallest x with at least ceil(q n / 100) of the n
 * threads at or below x; percentiles of 65535 or more read 65535).
 */
typedef struct pa_result {
  double p_int_w, p_sw_w, p_gl_w, p_leak_w;
  double t_max_ns;
  int32_t out_mem;
  float *waveform_w;
  uint32_t *event_count;
  uint32_t *glitch_count;
  uint8_t *state_pre;
  uint8_t *lut_ij;
  uint8_t *is_glitch;
  float ms_partition, ms_fused, ms_reduce, ms_total;
  uint32_t n_tiles, n_heavy;
  uint32_t kernel_launches;
  uint32_t path;  /* out: PA_PATH_* of the kernel that ran */
  double *gate_power_w;
  double *cell_power_w;
  uint64_t part_threads;
  uint32_t part_evt_p50, part_evt_p90, part_evt_p99, part_evt_max;
} pa_result;

#define PA_PATH_UNBANDED 0u /* the per-pin layout, the CTA kernel (per-event outputs, exact counts) */
#define PA_PATH_BANDED 1u
#define PA_PATH_WINDOWS 2u /* the paper's (gate, window) thread partition */
#define PA_PATH_WARP 3u    /* the per-pin layout, the warp kernel (the pass without per-event outputs) */

/* Create a context on CUDA device `cuda_device`. `cuda_stream` is a
 * cudaStream_t to run on (borrowed, must outlive the ctx) or NULL for a stream
 * the ctx creates. Errors: PA_ERR_ARG, PA_ERR_CUDA, PA_ERR_OOM. */
int pa_create(pa_ctx **out, int cuda_device, void *cuda_stream);

/* Free every device and host buffer the ctx owns. NULL is a no-op. */
void pa_destroy(pa_ctx *ctx);

/* Load (replace) the cell library. Replacing it drops the netlist and events.
 * Errors: PA_ERR_ARG (k, axis length, non-increasing axis, offsets out of
 * range, non-finite values), PA_ERR_OOM, PA_ERR_CUDA. */
int pa_load_library(pa_ctx *ctx, const pa_library *lib);

/* Load (replace) the netlist; requires a library. Drops loaded events.
 * Errors: PA_ERR_ORDER, PA_ERR_ARG, PA_ERR_RANGE (cell id >= n_cells, load
 * not finite or < 0, init bits beyond k), PA_ERR_OOM, PA_ERR_CUDA. */
int pa_load_netlist(pa_ctx *ctx, const pa_netlist *nl);

/* Load (replace) the events; requires a netlist. Validates them on the device.
 * Errors: PA_ERR_ORDER, PA_ERR_ARG (pin count, pin_off not monotone or not
 * ending at n_events), PA_ERR_UNSORTED, PA_ERR_RANGE, PA_ERR_TOGGLE,
 * PA_ERR_OOM, PA_ERR_CUDA. On error no events are loaded. */
int pa_load_events(pa_ctx *ctx, const pa_events *ev);

/*
 * pa_build_bands -- regroup the loaded events by clock bands (load-time layout).
 * Call after pa_load_events, with the clock period the runs will use. Each
 * gate's timeline (cycle = floor(fl32(t / t_clk_ns))) is cut, in cycle order,
 * into windows of whole cycles inside bands of band_cycles cycles: a window
 * closes at a band boundary or before a cycle that would give one of the
 * gate's pins more than 7 events in it; a single cycle that alone gives a pin
 * 8 to 15 events is a window of its own. Every non-empty (gate, window) is a
 * unit; units are ordered band by band and grouped into work items of at
 * most 511 events, and inside an item the events are copied into an input
 * region (each unit's input-pin events merged in (time, pin) order) followed
 * by an output region. Dense gates thus get narrow
 * cycle windows and sparse gates wide ones, as in the event-density-aware
 * per-gate cycle partitioning (Figs. 5, 19 and 20), fixed here at load time by
 * a per-pin event bound instead of a per-thread event target. Every pa_run whose t_clk_ns equals this
 * t_clk_ns bit for bit then uses the banded kernel, which keeps a band's cycle
 * bins in shared memory instead of adding every event to global memory; other
 * clocks use the unbanded kernel. Gates with more than 15 events of one pin in
 * a single cycle stay out of the layout and are streamed by the unbanded kernel
 * within the same run. Results agree with the unbanded path to floating-point
 * summation order.
 *   band_cycles  cycles per band: a power of two <= 4096; 0 = 4096
 * Memory: a second copy of the times and slews plus a two-byte tag word (10
 * bytes per event), 20 bytes per unit and 16 bytes per work item; the build also
 * takes temporary space of about 24 bytes per (band, gate) and 32 bytes per
 * unit.
 * A library of more than 64 cells gets no layout (the banded kernel stages
 * at most 64 cells' tables in shared memory): the call succeeds and runs take
 * the unbanded path (pa_result.path = PA_PATH_UNBANDED).
 * Errors: PA_ERR_ORDER (no events loaded), PA_ERR_ARG (t_clk_ns not > 0,
 * band_cycles not a power of two <= 4096, events spanning more than 2^20
 * bands), PA_ERR_OOM, PA_ERR_CUDA. Loading a new library, netlist or events
 * drops the bands.
 */
int pa_build_bands(pa_ctx *ctx, float t_clk_ns, uint32_t band_cycles);

/* Run partition -> fused power kernel -> final reduction on the loaded data.
 * May be called repeatedly with different parameters. Errors: PA_ERR_ORDER,
 * PA_ERR_ARG, PA_ERR_RANGE (an event's cycle >= n_cycles, t_max too early),
 * PA_ERR_OOM, PA_ERR_CUDA, PA_ERR_INTERNAL. */
int pa_run(pa_ctx *ctx, const pa_run_params *params, pa_result *out);

/*
 * pa_run_noalloc -- pa_run for callers that must not allocate device memory
 * at run time. (The paper has no counterpart: this is an integration entry
 * point of this library.)
 *
 * Who needs it: code that owns the GPU's memory budget outright (a framework
 * whose caching allocator has already reserved the device), loops that may
 * not stall the device (cudaMalloc/cudaFree synchronise it), and processes
 * that forbid allocation after start-up. pa_run may grow its scratch buffers
 * on the first call or when n_cycles or the gate count grows; this entry point
 * never does: its per-run scratch (cycle bins, work lists, totals) lives in
 * one file-scope device array of PA_NOALLOC_SCRATCH_BYTES (5 MiB).
 *
 * When the array is committed: pa_create looks up the array's device address
 * on the context's device (with that device current) and keeps it in the
 * context; under CUDA's lazy module loading that lookup is what loads the
 * library's module holding the array, so the 5 MiB are taken at the first
 * pa_create on a device and held until the process exits. pa_run_noalloc
 * itself only reads the kept address. If the lookup failed at pa_create
 * (e.g. the device had no memory left), pa_create still succeeds and
 * pa_run_noalloc returns PA_ERR_CUDA with that reason.
 *
 * Same arguments, computation and results as pa_run on the data loaded into
 * ctx (loading itself still allocates; do it beforehand), with these limits:
 *   n_cycles <= PA_NOALLOC_MAX_CYCLES, netlist gates <= PA_NOALLOC_MAX_GATES,
 *   out->out_mem == PA_MEM_DEVICE for every non-NULL array in out,
 *   part_mode == PA_PART_EVENTS, and cell_power_w only together with
 *   gate_power_w (the per-gate sums are accumulated in gate_power_w).
 * Beyond them it returns PA_ERR_ARG and says which limit was hit.
 * All calls share the one array and it keeps the last call's contents (each
 * call clears what it needs zeroed): calls whose device work overlaps -- from
 * several threads, contexts or streams at once -- race and must be
 * serialised by the caller. Per-event debug arrays and gate_power_w are
 * written in place and may hold partial data after an error; the other
 * outputs are written only on PA_OK.
 */
#define PA_NOALLOC_MAX_CYCLES 65536u
#define PA_NOALLOC_MAX_GATES 262144u
#define PA_NOALLOC_SCRATCH_BYTES (5u << 20)
int pa_run_noalloc(pa_ctx *ctx, const pa_run_params *params, pa_result *out);

/*
 * pa_run_stream -- the run of pa_run on a trace that stays in host memory,
 * for traces larger than the device's memory or runs made once per trace.
 * The paper's flow overlaps the host's event packing with the GPU work; here
 * the events pass through the device in chunks of whole gates (about
 * chunk_events events each; 0 = PA_STREAM_DEFAULT_CHUNK), the copy of the next
 * chunk overlapping the validation and computation of the current one (pinned
 * host memory gives the overlap). Each chunk is checked as pa_load_events
 * checks a trace and computed by the unbanded kernel into the same cycle bins
 * and totals; results equal pa_run's on the loaded trace to floating-point
 * summation order.
 *   ev   host arrays (mem = PA_MEM_HOST) in pa_load_events' form; not retained
 * Requires a netlist; does not use or change the loaded events or bands. Device
 * memory: two staging slots of about 9 bytes per event of the largest chunk,
 * plus pa_run's scratch. The host reads pin_off only where chunks are cut
 * (a binary search per chunk); the offsets inside a chunk are checked on the
 * device before the chunk is computed. Outputs as pa_run, without the per-event debug arrays
 * (PA_ERR_ARG); n_tiles returns the number of chunks. Errors as pa_load_events
 * and pa_run (indices of the offending pin / event / gate in the whole trace).
 */
#define PA_STREAM_DEFAULT_CHUNK (1ull << 26)
int pa_run_stream(pa_ctx *ctx, const pa_run_params *params, const pa_events *ev, uint64_t chunk_events,
                  pa_result *out);

/* Defaults: vdd 0.9 V, t_clk 1 ns, n_cycles 1, t_max 0, partition knobs 0. */
void pa_default_params(pa_run_params *params);

/* Text of the most recent error on ctx; valid until the next call on ctx. */
const char *pa_last_error(const pa_ctx *ctx);

/* PA_VERSION of the library. */
int pa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PA_H */
