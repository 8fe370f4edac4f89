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
  uint32_t pad1;
  float sax[8], lax[8];    // slew (ps) / load (fF) axes
  float isax[8], ilax[8];  // 1 / (ax[i+1] - ax[i])
};

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
};

struct RunArgs {
  // inputs
  const CellDesc* cells;
  uint32_t n_cells;
  const float* lut;
  const float* leak;       // uW
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
  uint32_t n_cycles;
  uint32_t tile_target, heavy_thresh;
  // partition
  uint32_t* part_blk;      // [2 * n_blocks] heads / heavies per block, then scanned
  uint32_t* part_counts;   // [4]: n_tiles, n_heavy, item counter, pad
  Tile* tiles;
  uint32_t* heavy;
  double* p0;              // sum of leakage of initial states, uW
  // accumulators: per cycle {W, D, ev, gl}
  //   W  energy in the cycle: dynamic + in-cycle leakage parts (fJ)
  //   D  leakage power steps taking effect after the cycle (uW)
  //   ev, gl event / glitch counts as f32 (exact below 2^24 per cycle). In
  //   exact mode (a cycle reached 2^24 events) the same 16 bytes hold {W, D} as
  //   fp64 -- f32 sums of that many terms are too coarse -- and the counts go
  //   to cnt_ev / cnt_gl as integers.
  float4* bins;            // [n_cycles]
  uint32_t* cnt_ev;        // [n_cycles] exact counts (exact mode) / count output (fast mode), may be null
  uint32_t* cnt_gl;
  double* chunk_sums;      // [ceil(n_cycles / kReduceChunk)] final-reduction partial sums
  double* totals;          // [4]: E_int, E_sw, E_gl (fJ), sum dP * (t_max - t) (fJ)
  unsigned long long* err;
  // debug outputs (device, may be null)
  uint8_t* dbg_state;
  uint8_t* dbg_lut;
  uint8_t* dbg_glitch;
};

// ------------------------------------------------------------------ banded layout
//
// A copy of the events regrouped by clock bands of band_cycles cycles (for one
// clock period fixed when the layout is built). Inside a band, events keep the
// per-pin CSR order; the band holds first the light gates (every pin has at
// most kLightPinMax events in every band), in gate order, then the heavy
// gates. Per (band, light gate) one packed u32 record: 5-bit event count of
// each pin (pins 0..4) and, in bits 25..28, the input state at the band start;
// per (band, heavy gate) an explicit record. Bands start on cycle boundaries,
// so the first event of a pin in a band is never a glitch of an earlier one.

constexpr int kLightPinMax = 31;       // per-pin events per band of a light gate
constexpr int kLightBlock = 8;         // light gates per partition block
constexpr int kBandMaxBands = 64;
constexpr uint32_t kBandDefaultCycles = 4096;
constexpr uint32_t kBandMaxCycles = 4096;  // shared-memory histogram capacity (cycles)
constexpr int kBTileCap = 4096;        // events per banded tile
constexpr int kBGateCap = 512;         // gates per banded tile (multiple of kLightBlock)
constexpr uint32_t kBTileTarget = 2560;  // bucket size; + one light block (<= 8 * 155) stays <= kBTileCap
constexpr uint32_t kBUnitSmall = kBTileCap - kBTileTarget;  // heavy units up to this share tiles

struct __align__(16) HeavyRec {
  uint64_t base;           // offset of the unit's first event in the banded arrays
  uint32_t cnt[5];         // events per pin in the band
  uint32_t state;          // input state at the band start
};

// Per-run gate record (light and heavy orders): cell (bits 0..15), k (16..19),
// load-axis interval j (20..23), initial... ; load-axis fraction; switching energy.
struct __align__(16) GateRun {
  uint32_t packed;
  float v;
  float esw;
  uint32_t gate;
};

struct __align__(16) BandItem {
  uint32_t band;
  uint32_t kind;   // 0 light tile, 1 heavy tile, 2 streamed heavy unit
  uint32_t first;  // light block / heavy rank
  uint32_t last;   // exclusive
  uint64_t e0;     // first event in the banded arrays
  uint32_t n;      // events
  uint32_t pad;
};

struct BandLayout {
  bool built = false;
  float t_clk = 0.f;
  uint32_t band_cycles = 0, n_bands = 0;
  uint32_t n_light = 0, n_heavy = 0, n_lblk = 0;
  float* bt = nullptr;        // [E] banded times
  float* bs = nullptr;        // [E] banded slews
  uint32_t* lrec = nullptr;   // [n_bands * n_light]
  HeavyRec* hrec = nullptr;   // [n_bands * n_heavy]
  uint64_t* lblk = nullptr;   // [n_bands * (n_lblk + 1)] offset of each light block; last = light region end
  uint32_t* lgate = nullptr;  // [n_light] gate id of each light rank
  uint32_t* hgate = nullptr;  // [n_heavy]
};

struct BandBuildArgs {
  const GateRec* gates;
  uint32_t n_gates;
  uint64_t n_pins, n_events;
  const uint64_t* pin_off;
  const float* t;
  const float* s;
  float t_clk, inv_t_clk;
  bool pow2;
  uint32_t band_cycles, n_bands;
  uint32_t* cnt;         // [n_pins * n_bands] events per (pin, band) -- temporary
  uint8_t* heavy;        // [n_gates] -- temporary
  uint32_t* rank;        // [n_gates] light or heavy rank -- temporary
  uint32_t* blk;         // scan scratch -- temporary
  uint32_t* totals;      // [4] n_light, n_heavy -- temporary
  uint32_t* unit_size;   // [n_bands * n_gates] -- temporary
  uint64_t* unit_off;    // [n_bands * n_gates + 1] -- temporary
  uint64_t* scan_blk;    // scan scratch -- temporary
  BandLayout L;
  unsigned long long* err;
};

struct BandRunArgs {
  RunArgs r;             // cells, lut, leak, gates, params, totals, err, debug, bins (fp64 layout)
  BandLayout L;
  GateRun* grun_l;       // [n_light]
  GateRun* grun_h;       // [n_heavy]
  BandItem* items;
  uint64_t* item_ev;     // [n_items + 1] event prefix of the items
  uint32_t* item_counts; // [4]: light items, heavy items
  uint32_t* blk;         // scan scratch
  uint32_t max_items;
};

// kernels (pa_kernels.cu)
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
// banded layout (pa_banded.cu)
// phase 1: counts per (pin, band), light/heavy ranks, totals[0..1] = n_light,
// n_heavy; phase 2 (after L.lrec/hrec/lblk are allocated): offsets, scatter.
cudaError_t band_build_phase1(BandBuildArgs& a, cudaStream_t st);
cudaError_t band_build_phase2(BandBuildArgs& a, cudaStream_t st);
uint32_t band_scan_blocks(uint64_t n);
uint32_t band_max_items(const BandLayout& L);
// Item list of a run: flags / pos / scan_blk / item_n are scratch sized for
// band_max_items(); host_items[0..1] = light and heavy item counts.
cudaError_t band_partition(BandRunArgs& A, uint32_t* flags, uint64_t* pos, uint64_t* scan_blk, uint32_t* item_n,
                           uint32_t* host_items, cudaStream_t st);
// Per-run gate records, then the banded fused kernel over n_items items.
cudaError_t band_gate_run(BandRunArgs& A, cudaStream_t st);
cudaError_t band_fused(BandRunArgs& A, uint32_t n_items, int sm_count, bool debug, cudaStream_t st);

cudaError_t launch_final_reduce(const RunArgs& a, double t_clk, double t_max, float* wave_out,
                                double* p_out, bool exact, cudaStream_t st);
inline uint32_t reduce_chunks(uint32_t n_cycles) { return (n_cycles + kReduceChunk - 1) / kReduceChunk; }

}  // namespace pa
