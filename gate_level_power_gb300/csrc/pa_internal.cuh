// Internal declarations shared by the host API (pa_api.cu) and the kernels
// (pa_kernels.cu) of libpa.so. Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "pa.h"

namespace pa {

constexpr int kMaxK = PA_MAX_INPUTS;   // inputs per cell
constexpr int kTileCap = 4096;         // events staged in shared memory per work item
constexpr int kGateCap = 256;          // gates per light tile
constexpr int kThreads = 256;          // threads per CTA of the fused kernel
constexpr int kSmemCells = 64;         // cell descriptors staged in shared memory
constexpr uint32_t kDefaultTile = 2048;
constexpr uint32_t kDefaultHeavy = 2048;
constexpr uint32_t kReduceChunk = 2048;  // cycles per CTA of the final reduction

// Per-cell descriptor: axes, reciprocal interval widths and table offsets.
struct __align__(16) CellDesc {
  uint8_t k, ns, nl, pad0;
  uint32_t lut_off;   // floats into the LUT array: [2^k][ns][nl]
  uint32_t leak_off;  // floats into the leakage array: [2^k], in uW (fJ/ns)
  uint32_t patch_off; // float4s into the patch table: [2^k][ns - 1][nl - 1]
  float sax[8], lax[8];    // slew (ps) / load (fF) axes
  float isax[8], ilax[8];  // 1 / (ax[i+1] - ax[i])
};

// Derived table built with the library (used by the banded kernel): for each
// state and interpolation cell (i, j) of a LUT the four corners {L[i][j],
// L[i][j+1], L[i+1][j], L[i+1][j+1]} as one float4.

// Per-gate record (16 B): pin base, cell, load, initial values and k.
struct __align__(16) GateRec {
  uint32_t pin_base;
  uint32_t cell;
  float load;
  uint32_t init;  // bits 0..7 initial input values, bit 8 initial output, bits 16..23 k
};

// A light tile: contiguous gates [gb, ge) whose events fit one shared-memory tile.
struct Tile {
  uint32_t gb, ge;
};

// Device-side error word: (index << 8) | code, smallest wins.
// At one event the lowest code wins: a time that is out of range is reported
// as such, not as the order violation it also causes.
enum DevErrCode : uint32_t {
  kErrNone = 0,
  kErrPinOff = 1,
  kErrRangeT = 2,
  kErrRangeSlew = 3,
  kErrUnsorted = 4,
  kErrValue = 5,
  kErrToggle = 6,
  kErrTileOverflow = 7,
  kErrCountOverflow = 8,  // a cycle reached 2^24 events: counts must be accumulated exactly
  kErrLayout = 9,         // a work item of the banded layout is inconsistent (index: item)
  kErrStageTimeout = 10,  // a bounded wait for a shared-memory stage copy gave up (index: item)
};
constexpr unsigned long long kNoErr = ~0ull;

struct ValidateArgs {
  const GateRec* gates;
  uint32_t n_gates;
  uint64_t n_pins, n_events;
  const uint64_t* pin_off;
  const float* t;
  const float* s;
  const uint8_t* value;   // may be null
  uint64_t* gate_off;     // out [G + 1]
  unsigned long long* err;
  unsigned int* t_max_bits;  // out: max event time as ordered bits
  uint32_t* starts;       // scratch [(n_events + 31) / 32 + 1]: bit e set if event e starts a pin
};

struct Piece;  // a piece of a heavy gate (warp kernel, below)

struct RunArgs {
  // inputs
  const CellDesc* cells;
  uint32_t n_cells;
  const float* lut;
  const float* leak;       // uW
  const float4* patch;     // LUT corner patches
  const GateRec* gates;
  uint32_t n_gates;
  const uint64_t* pin_off;
  const uint64_t* gate_off;
  const float* t;
  const float* s;
  // parameters
  float t_clk, inv_t_clk;
  float t_max_f;           // window end as f32 (for per-event leakage spans)
  float half_vdd2;         // 0.5 * V^2
  uint32_t glitch_all;     // PA_RUN_GLITCH_ALL: every event of a multi-event pin-cycle is a glitch
  uint32_t esw_rise;       // PA_RUN_ESW_RISE: C V^2 on a rising output edge, 0 on a falling one
  uint32_t n_cycles;
  uint32_t tile_target, heavy_thresh;
  // partition
  uint32_t* part_blk;      // [2 * n_blocks] heads / heavies per block, then scanned
  uint32_t* part_counts;   // [4]: n_tiles, n_heavy (n_pieces for the warp kernel), item counter, pad
  Tile* tiles;
  uint32_t* heavy;
  Piece* pieces;           // heavy-gate pieces of the warp kernel (pa_csr.cu)
  uint64_t* tile_ev;       // per light tile of the warp kernel: its first event and its end
  uint4* gslot;            // per light gate of the warp kernel: its slot (two uint4), pin starts from its first event
  double* p0;              // sum of leakage of initial states, uW
  // accumulators: per cycle {W, D, ev, gl}
  //   W  energy in the cycle: dynamic + in-cycle leakage parts (fJ)
  //   D  leakage power steps taking effect after the cycle (uW)
  //   ev, gl event / glitch counts as f32 (exact below 2^24 per cycle). In
  //   exact mode (a cycle reached 2^24 events) the same 16 bytes hold {W, D} as
  //   fp64 -- f32 sums of that many terms are too coarse -- and the counts go
  //   to cnt_ev / cnt_gl as integers.
  float4* bins;            // [n_rep][n_cycles]
  uint32_t n_rep;          // copies of the f32 bins (a power of two; the warp kernel's pass spreads its
                           // reductions over them, the final reduction adds them up), else 1
  uint32_t* cnt_ev;        // [n_cycles] exact counts (exact mode) / count output (fast mode), may be null
  uint32_t* cnt_gl;
  double* chunk_sums;      // [ceil(n_cycles / kReduceChunk)] final-reduction partial sums
  double* totals;          // [4]: E_int, E_sw, E_gl (fJ), sum dP * (t_max - t) (fJ)
  unsigned long long* err;
  // debug outputs (device, each may be null)
  uint8_t* dbg_state;
  uint8_t* dbg_lut;
  uint8_t* dbg_glitch;
  // per-gate energies {E_int, E_sw, E_gl, sum dP (t_max - t)} (fJ, zeroed), or null
  double* gate_e;
  double* cell_p;          // [n_cells * 4] per-cell sums of the per-gate power (W, zeroed), or null
};

// ------------------------------------------------------------------ banded layout
//
// A copy of the events regrouped by clock bands of band_cycles = 2^mb cycles,
// for one clock period fixed when the layout is built. Every gate's timeline is
// cut greedily, in cycle order, into windows of whole cycles: a window closes
// at a band boundary or before a cycle that would give one of its pins more
// than kUnitPinSoft events; a single cycle that alone gives a pin more than
// kUnitPinSoft (but at most kUnitPinMax) events is a window of its own. A
// unit is one non-empty (gate, window). Units are
// ordered band by band, gate by gate; work items are runs of whole units of
// one band. Inside an item the events are stored in two regions: first the
// input-pin events of all its units (unit by unit, each unit's events merged
// in (time, pin) order), then the output-pin events (unit by unit, in time
// order). Each event carries a two-byte tag word (unit within the item, input
// pin, distance back to the pin's previous event in the unit), each unit a
// 16-byte record (region offsets, input count, window start state, cell,
// load-axis interval and fraction, load). Windows start on
// cycle boundaries, so the event before a unit's first event on a pin lies in
// an earlier cycle: glitches never straddle units. Gates with more than
// kUnitPinMax events of one pin in a single cycle ("big" gates) stay out of
// the layout and are streamed by the unbanded kernel.

constexpr int kUnitPinMax = 15;                  // events per pin per unit (a unit of one cycle)
constexpr int kUnitPinSoft = 7;                  // events per pin per unit of several cycles
constexpr int kUnitMaxEvents = 5 * kUnitPinMax;  // events per unit
constexpr uint32_t kBandDefaultCycles = 4096;
constexpr uint32_t kBandMaxCycles = 4096;        // shared-memory histogram capacity (cycles)
constexpr uint32_t kBandMaxBands = (1u << 20) - 1;  // the item word's band field also holds the sentinel
constexpr int kItemEvents = 512;                 // events per item (cap): one warp's work item
constexpr int kItemUnits = 64;                   // units per item (cap): 6-bit unit tags
// A new item starts where a unit's event offset enters a new bucket of
// kItemEvents - 1 - (the layout's largest unit) events (or a new band, or
// every kItemUnits units), so an item holds fewer than kItemEvents events.

// Item word `bw`: band (bits 0..19; items[n_items] is a sentinel with band =
// n_bands) | input events of the item (bits 20..28) | bit 29: the item's
// events come in runs of one cycle (at least two thirds of them share the
// cycle of the event stored before them: runs of three or more on average),
// so the run merges the bin updates of each run of equal cycles in a warp
// before its shared-memory atomics.
constexpr uint32_t kItemBandBits = 20;
constexpr uint32_t kItemBandMask = (1u << kItemBandBits) - 1u;
constexpr uint32_t kItemRunsBit = 1u << 29;

// Unit record (uint4), written by the finalize pass:
//   x: input offset in the item (bits 0..8) | output offset in the item (9..17)
//      | cell (18..23) | input state at the window start (24..27)
//      | load-axis interval j (28..30)
//      | the unit has input events at one time on two pins (31)
//   y: load-axis fraction v (f32), z: load C (f32, fF)
//   w: the unit's input events (bits 0..5) | the output pin's value at the
//      window start (6) | (k - 1) << 30
// (an input event reads {x, y}, an output event z)
// A unit's input events are stored in (time, pin) order (the merge of its
// pins' time-ordered runs), its output events in time order.
// Unit record of the walk (uint2, a build temporary): x = counts of pins 0..4
// (4 bits each) | start state << 20 | cell << 24 (6 bits) | output value at
// the window start << 30, y = load (f32 bits).
// Event tag word (u16): unit within the item (bits 0..5) | input pin (bits
// 6..7) | for an input event, the distance back (in the unit's (time, pin)
// order) to the previous event of its pin in the unit, 0 if none; for an
// output event 1 if the unit has an earlier output event (bits 8..15).
struct BandItem {
  uint64_t e0;    // first event in the banded arrays
  uint32_t u0;    // first unit
  uint32_t bw;    // band | input-event count << kItemBandBits
};

struct BandLayout {
  bool built = false;
  float t_clk = 0.f;
  uint32_t band_cycles = 0, mb = 0, n_bands = 0;
  uint64_t n_ev = 0;          // events in the banded arrays
  uint32_t n_units = 0, n_items = 0, n_big = 0;
  float* bt = nullptr;        // [n_ev + pad] banded times
  float* bs = nullptr;        // [n_ev + pad] banded slews
  uint16_t* btag = nullptr;   // [n_ev + pad] event tag words
  uint4* urec = nullptr;      // [n_units] unit records
  uint32_t* ugate = nullptr;  // [n_units] gate of each unit
  BandItem* items = nullptr;  // [n_items + 1]
  uint32_t* big = nullptr;    // [n_big] gates streamed by the unbanded kernel
};

struct BandBuildArgs {
  const GateRec* gates;
  uint32_t n_gates;
  uint64_t n_events;
  const uint64_t* pin_off;
  const float* t;
  const float* s;
  float t_clk, inv_t_clk;
  bool pow2;
  uint32_t mb, n_bands;
  uint8_t* bigf;         // [G] 1 for a big gate -- temporary
  uint32_t* grank;       // [G] place of each gate in the layout's gate order -- temporary
  uint32_t* cnt_gb;      // [n_bands * G] units per (band, gate) -- temporary
  uint32_t* evc_gb;      // [n_bands * G] events per (band, gate) -- temporary
  uint64_t* ubase;       // [n_bands * G + 1] first unit of each (band, gate) -- temporary
  uint64_t* ebase;       // [n_bands * G + 1] first banded event of each (band, gate) -- temporary
  uint32_t* uband;       // [n_units] -- temporary
  uint64_t* uoff;        // [n_units + 1] -- temporary
  uint32_t* flags;       // [max(G, n_units)] class flags, then item heads -- temporary
  uint64_t* ipos;        // [max(G + 2, n_units + 1)] scans -- temporary
  uint64_t* scan_blk;    // scan scratch -- temporary
  uint32_t* counters;    // [4]: big gates, gates with windows narrower than a band, largest unit,
                         //      dense gates -- temporary
  uint32_t* dense;       // [G] gates walked one warp per (gate, band) -- temporary
  uint8_t* gflag;        // [G] a dense gate has a window narrower than a band -- temporary
  uint32_t item_bucket;  // events per item bucket (set after the counting pass)
  uint2* urec2;          // [n_units] unit records of the walk -- temporary
  const CellDesc* cells; // library (load axes for the unit records)
  BandLayout L;
  unsigned long long* err;
};

// Bounded waits of the banded kernel on its TMA stage copies: tries of
// mbarrier.try_wait (each suspends the thread for at most about 0.1 ms)
// before the wait gives up, records kErrStageTimeout and the warp stops.
constexpr uint32_t kBandWaitLimit = 1u << 16;
// The same limit under the test hook that leaves one item's stage unstarted
// (PA_TEST_STAGE_TIMEOUT): a few milliseconds.
constexpr uint32_t kBandTestWaitLimit = 64;
constexpr uint32_t kNoItem = 0xFFFFFFFFu;

struct BandRunArgs {
  RunArgs r;             // cells, lut, leak, gates, params, bins, totals, err, debug
  BandLayout L;
  uint32_t* item_ctr;    // [2] items handed out so far, of the main part and of the tail (zero before the launch)
  uint32_t chunk;        // items a CTA takes at a time (set by band_fused)
  uint32_t wait_limit;   // tries per bounded stage wait (kBandWaitLimit)
  uint32_t skip_item;    // test hook: the item whose stage copy is never started (kNoItem: none)
};

// ------------------------------------------------------------------ warp kernel on the per-pin layout
//
// The fused kernel of the run on the loaded (CSR) layout (pa_csr.cu), one
// warp per work item. Work items: light tiles, runs of consecutive whole
// gates of at most kCsrGates gates whose events fit one warp's stage (the
// event-count rule of the CTA kernel's tiles, with a target of tile_target
// events and gates of at most heavy_thresh events), and pieces of the heavy
// gates: gate g with n_g events is cut into ceil(n_g / kCsrPiece) pieces at
// times taken from its densest pin (that pin's events split evenly), each pin
// split at the first event at or after that time, so a piece holds every
// event of the gate in a time interval. A warp works through a piece in
// windows of at most kCsrWin events.
constexpr uint32_t kCsrDefaultTile = 320;
constexpr uint32_t kCsrDefaultHeavy = 64;
constexpr uint32_t kCsrMaxTileHeavy = 448;  // tile_target + heavy_thresh a warp's stage holds
constexpr uint32_t kCsrGates = 32;          // gates per light tile (one lane per gate)
constexpr uint32_t kCsrPiece = 2048;        // target events per piece of a heavy gate
constexpr uint32_t kCsrWin = 448;           // events per window of a piece

// A piece of a heavy gate, with what the warp kernel needs to start it
// without further dependent loads (filled by the partition).
struct __align__(16) Piece {
  uint32_t gate, idx;          // the gate; the piece's index among the gate's pieces
  uint32_t info;               // k | initial input bits << 4 | load-axis interval j << 8 | cell << 12 | last piece << 31
  float v, esw;                // load-axis fraction; switching energy C V^2 / 2 (fJ)
  uint32_t gend;               // the gate's events, from its first one
  uint64_t pin0;               // the gate's first event (its first pin's start)
  uint32_t lo[kMaxK + 1];      // per pin, the piece's first event as an index into the pin's events
  uint32_t pin[kMaxK + 1];     // per pin, its first event from the gate's first event
  uint32_t pad[2];
};
static_assert(sizeof(Piece) == 80, "piece record size");

// Upper bound of the pieces of a run over n_events events of n_gates gates
// (gates with more than heavy_thresh events).
uint64_t csr_max_pieces(uint64_t n_events, uint32_t n_gates, uint32_t heavy_thresh);
// The warp kernel runs a pass (no per-event outputs, f32 bins) when the
// library fits its shared-memory cell tables and the tile knobs fit its stage.
bool csr_eligible(uint32_t n_cells, uint32_t tile_target, uint32_t heavy_thresh);
// Partition (tiles, pieces and their cut points; P0) into a.tiles / a.pieces /
// a.part_counts, then the kernel.
cudaError_t launch_csr_partition(const RunArgs& a, uint32_t n_blocks, uint64_t max_pieces, cudaStream_t st);
cudaError_t launch_csr(const RunArgs& a, int sm_count, bool pow2, cudaStream_t st);

// kernels (pa_kernels.cu)
// Exclusive scan of the per-block (heads, heavies) pairs of a partition
// (single block), totals into part_counts[0..1], part_counts[2] = 0.
cudaError_t launch_part_scan(const RunArgs& a, uint32_t n_blocks, cudaStream_t st);
cudaError_t launch_check_pin_off(const uint64_t* pin_off, uint64_t n_pins, uint64_t n_events,
                                 unsigned long long* err, cudaStream_t st);
cudaError_t launch_validate_events(const ValidateArgs& a, cudaStream_t st);
cudaError_t launch_partition(const RunArgs& a, uint32_t n_blocks, cudaStream_t st);
uint32_t partition_blocks(uint32_t n_gates);
cudaError_t launch_fused(const RunArgs& a, int grid, bool pow2, bool debug, bool exact, cudaStream_t st);
int fused_blocks_per_sm(bool pow2, bool debug, bool exact);
size_t fused_smem_bytes();
// Two kernels: per-chunk step sums, then the scan/apply pass. In fast mode it
// writes u32 counts to cnt_ev / cnt_gl (if set) and flags kErrCountOverflow
// when a cycle's f32 count may be inexact.
// banded layout (pa_banded.cu), built in steps with host reads in between:
// count  windows per gate: units and events per (band, gate), their scans
//        (ubase / ebase, totals at index n_bands * G), big gates (counters[0]);
// write  unit records and the event scatter, item heads and their scan
//        (ipos[n_units] = n_items), after the layout arrays are allocated;
// items  the item list (after it is allocated), then the finalize pass:
//        per item, the input / output regions, event tags and unit records.
cudaError_t band_build_count(BandBuildArgs& a, cudaStream_t st);
cudaError_t band_build_write(BandBuildArgs& a, cudaStream_t st);
cudaError_t band_build_items(BandBuildArgs& a, cudaStream_t st);
uint32_t band_scan_blocks(uint64_t n);
// Exclusive scan of u32 into u64 (out[n] = total); blk holds band_scan_blocks(n) entries.
cudaError_t scan_u32_to_u64(const uint32_t* in, uint64_t n, uint64_t* blk, uint64_t* out, cudaStream_t st);
// P0 of a run: leakage of every gate's initial input state, added to *r.p0.
cudaError_t band_p0(const RunArgs& r, cudaStream_t st);
// The banded fused kernel over the layout's items.
cudaError_t band_fused(const BandRunArgs& A, int sm_count, bool debug, bool exact, cudaStream_t st);
int band_blocks_per_sm(bool pow2, bool debug, bool exact);

// The paper's (gate, window) thread partition (pa_window.cu): plan, then the
// window kernel, whose per-thread sums go through kWinTotSlots slots into
// RunArgs::totals.
constexpr uint32_t kWinHistBins = 65536;  // events-per-thread histogram (the last bin: 65535 or more)
constexpr int kWinTotSlots = 256;         // total accumulator slots (spread the CTAs' fp64 atomics)

struct WinArgs {
  uint32_t mode;          // PA_PART_DENSITY or PA_PART_FIXED
  uint32_t n_evt_tgt, n_thr_floor, n_cyc_fix;
  uint32_t* ncyc;         // [G] cycles per thread of each gate
  uint32_t* nthr;         // [G] threads of each gate
  uint64_t* thr_off;      // [G + 1] first thread of each gate; [G] = threads in all
  uint64_t* scan_blk;     // scan scratch (band_scan_blocks(G) entries)
  double* tot_slots;      // [kWinTotSlots * 4] zeroed before the window kernel
  unsigned long long* hist;  // [kWinHistBins] events per thread (zeroed), or null: no statistics
  unsigned int* ev_max;   // largest events per thread (zeroed; with hist)
};

// Plan: cycles and threads per gate, and their scan (thr_off[G] = threads).
cudaError_t launch_window_plan(const RunArgs& a, const WinArgs& w, cudaStream_t st);
// The window kernel over the planned (gate, window) threads (grid-stride over
// chunks of thread ids, the count read on the device), then the totals fold.
cudaError_t launch_window(const RunArgs& a, const WinArgs& w, int grid, bool pow2, bool debug, bool exact,
                          cudaStream_t st);
int window_blocks_per_sm(bool pow2, bool debug, bool exact);

cudaError_t launch_final_reduce(const RunArgs& a, double t_clk, double t_max, float* wave_out,
                                double* p_out, bool exact, cudaStream_t st);
// Per-gate power in place: a.gate_e (fJ) -> W, with each gate's initial-state
// leakage held to t_max added to its leakage; with a.cell_p, each gate's power
// is also added to its cell's.
cudaError_t launch_gate_power(const RunArgs& a, double t_max, cudaStream_t st);
// A chunk of pa_run_stream: its pin offsets (n_pins + 1, in place) made relative
// to its first event ev0, and its gate records copied with pin bases relative
// to its first pin pin0.
cudaError_t launch_rebase_chunk(uint64_t* pin_off, uint64_t n_pins, uint64_t ev0, const GateRec* gates_src,
                                GateRec* gates_dst, uint32_t n_gates, uint32_t pin0, cudaStream_t st);
inline uint32_t reduce_chunks(uint32_t n_cycles) { return (n_cycles + kReduceChunk - 1) / kReduceChunk; }

// Copies of the f32 bins for the warp kernel's pass: up to kBinCopies, within
// kBinCopyBytes in all. Reductions of many events into one cycle's bin
// serialise at its L2 slice; spread over copies, bursts of activity in a few
// cycles cost less.
constexpr uint32_t kBinCopies = 8;
constexpr size_t kBinCopyBytes = (size_t)64 << 20;
inline uint32_t bin_copies(uint32_t n_cycles) {
  uint32_t r = kBinCopies;
  while (r > 1 && (size_t)r * n_cycles * 16 > kBinCopyBytes) r >>= 1;
  return r;
}

}  // namespace pa
