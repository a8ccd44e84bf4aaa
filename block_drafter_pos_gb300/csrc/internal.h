// Internal launch interfaces between the host orchestration (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace df2 {

constexpr int kMaxSeg = 4;

// K elements of one pipeline stage of the weight-streaming GEMV (64 weight rows).
constexpr int kGemvStageK = 128;

// One weight-streaming GEMV segment: for every K split s,
//   out[s][n][m] = sum_{k in split s} W[m][k] * X[n][k],  n < 8 * n_tiles, m < M.
// The consumer adds the split planes in split order.
struct GemvSeg {
  CUtensorMap wmap;       // W [M][K]: bf16 boxes 32 K x 64 rows or int8 boxes 64 K x 64 rows, 64-byte swizzle
  CUtensorMap xmap;       // X planes [2][rows][K] (hi rows, then lo rows): boxes of 8 rows (gemv_encode_xmap)
  const uint16_t* scale;  // Q8: bf16 [M][K/64]
  const uint16_t* bias;
  int x_lo_row;           // first row of the low-order plane in xmap
  int M, K, n_tiles;
  int splits;             // K splits (K / splits is a multiple of kGemvStageK)
  float* out;             // [splits][n_tiles * 8][M]
  int unit_begin;         // first global work unit (64-row block, split) of this segment (set by the launcher)
};

struct GemvArgs {
  GemvSeg seg[kMaxSeg];
  int nseg;
  int total_units;
  int* err;               // set nonzero if a pipeline wait gave up (never in a correct run), or null
};

// Encodes the tensor map of one weight matrix [M][K] (bf16 when fmt == 0, int8
// codes when fmt == 1).  Returns false if the driver rejects it.
bool gemv_encode_wmap(CUtensorMap* map, const void* w, int M, int K, int fmt);

// Encodes the tensor map of an activation buffer of `rows` rows of width K per
// plane, hi plane then lo plane (bf16 when fmt == 0, fp16 when fmt == 1).
bool gemv_encode_xmap(CUtensorMap* map, const void* x, int rows, int K, int fmt);

// fmt: 0 = BF16 weights, 1 = Q8G64 weights.  max_tiles: largest n_tiles over segments.
// pdl: launch with programmatic stream serialisation.
cudaError_t launch_gemv(GemvArgs& a, int fmt, int max_tiles, int num_sms, bool pdl, cudaStream_t st);

// K split for a launch over `blocks` 64-row weight blocks of depth K whose one
// output plane is `plane_bytes`: minimises whole-grid rounds of (block, split)
// units times their length in pipeline stages, plus the consumer's cost of
// adding planes.
int gemv_choose_splits(int blocks, int K, double plane_bytes, int num_sms, int fmt);

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
