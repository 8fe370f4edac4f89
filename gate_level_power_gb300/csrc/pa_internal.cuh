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
  // accumulators
  float* bin_w;            // [n_cycles] energy: dynamic + in-cycle leakage parts, fJ
  float* bin_d;            // [n_cycles] leakage power steps taking effect after the cycle, uW
  uint32_t* bin_ev;        // [n_cycles]
  uint32_t* bin_gl;        // [n_cycles]
  double* totals;          // [4]: E_int, E_sw, E_gl (fJ), sum dP * (t_max - t) (fJ)
  unsigned long long* err;
  // debug outputs (device, may be null)
  uint8_t* dbg_state;
  uint8_t* dbg_lut;
  uint8_t* dbg_glitch;
};

// kernels (pa_kernels.cu)
cudaError_t launch_check_pin_off(const uint64_t* pin_off, uint64_t n_pins, uint64_t n_events,
                                 unsigned long long* err, cudaStream_t st);
cudaError_t launch_validate_events(const ValidateArgs& a, cudaStream_t st);
cudaError_t launch_partition(const RunArgs& a, uint32_t n_blocks, cudaStream_t st);
uint32_t partition_blocks(uint32_t n_gates);
cudaError_t launch_fused(const RunArgs& a, int grid, bool pow2, bool debug, cudaStream_t st);
int fused_blocks_per_sm(bool pow2, bool debug);
size_t fused_smem_bytes();
cudaError_t launch_final_reduce(const RunArgs& a, double t_clk, double t_max, float* wave_out,
                                double* p_out, cudaStream_t st);

}  // namespace pa
