// Internal launch interfaces between the host orchestration (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace df2 {

constexpr int kMaxSeg = 4;

// What happens to a finished 16-row tile of a GEMV segment.
enum GemvEpilogue : int {
  kEpiStore = 0,    // out[n][m] = y (fp32)
  kEpiSwiglu = 1,   // tile = 8 gate rows + the same 8 up rows: act[n][f] = silu(g) * u
  kEpiConvOut = 2,  // y = sublayer output channel: x += conv_out(y); act = x * w_next; ss partials
};

// One weight-streaming GEMV segment: y[n][m] = sum_k W[m][k] * X[n][k] for n < 8 * n_tiles.
struct GemvSeg {
  const void* w;          // bf16 [M][K] or int8 codes [M][K]
  const uint16_t* scale;  // Q8: bf16 [M][K/64]
  const uint16_t* bias;
  const void* w2;         // kEpiSwiglu: the up matrix (rows 8..15 of every tile), same layout as w
  const uint16_t* scale2;
  const uint16_t* bias2;
  const void* x;          // activations: bf16 (BF16 weights) or fp16 (Q8 weights), [n_rows][ldx]
  size_t xlo_off;         // elements from x to its low-order plane (x = hi + lo), 0 = hi only
  int ldx, K, n_tiles;
  int tiles;              // 16-row tiles of this segment
  int splits;             // K splits (K / splits is a multiple of 128)
  int epi;
  // kEpiStore
  float* out;             // [n_rows][ldo]
  int ldo;
  // kEpiSwiglu / kEpiConvOut: activation output of the next projection
  void* act;              // [n_rows][ld_act], bf16 or fp16 (act_fmt), plus its low plane at act + act_lo
  size_t act_lo;
  int ld_act, act_fmt;
  void* act2;             // kEpiConvOut: optional second activation copy (bf16, LM-head input), or null
  size_t act2_lo;
  // kEpiConvOut
  float* xres;            // residual stream [n_rows][H]
  const float* delta;     // [n_rows][4G]: dynamic coefficients (io 1 = conv after the sublayer)
  const uint16_t* base;   // [4][H]
  const uint16_t* norm_w; // norm weight of the next sublayer
  float* ss;              // [n_rows][H/16] sums of squares of the updated x, per tile
  int G;
  // schedule (filled by the launcher)
  int unit_begin;         // first global work unit (tile, split) of this segment
  int tile_begin;         // first global tile of this segment
};

struct GemvArgs {
  GemvSeg seg[kMaxSeg];
  int nseg;
  int total_units;
  int max_splits;         // partial slots per tile
  float* part;            // [total tiles][max_splits][NT][32 lanes][4]
  int* counters;          // [total tiles], zero between launches
};

// fmt: 0 = BF16 weights, 1 = Q8G64 weights.  max_tiles: largest n_tiles over segments.
// pdl: launch with programmatic stream serialisation.
cudaError_t launch_gemv(GemvArgs& a, int fmt, int max_tiles, int num_sms, bool pdl, cudaStream_t st);

// Chooses the K split of every segment (cost model: whole-grid rounds of units,
// per-unit and per-partial overheads), fills the schedule, and returns the scratch
// the launch needs (floats of partials, tile counters).
void gemv_plan(GemvArgs& a, int fmt, int num_sms, size_t* part_floats, int* n_counters);

// Launch helper: cudaLaunchKernelEx with the programmatic stream serialisation
// attribute when pdl is set.
template <typename Kern, typename... Args>
cudaError_t launch_ex(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace df2
