// Internal launch interfaces between the host orchestration (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace df2 {

constexpr int kMaxSeg = 4;

// One weight-streaming GEMV segment: for every K split s,
//   out[s][n][m] = sum_{k in split s} W[m][k] * X[n][k],  n < 8 * n_tiles, m < M.
// The consumer adds the split planes in split order.
struct GemvSeg {
  const void* w;          // bf16 [M][K] or int8 codes [M][K]
  const uint16_t* scale;  // Q8: bf16 [M][K/64]
  const uint16_t* bias;
  const void* x;          // activations: bf16 (BF16 weights) or fp16 (Q8 weights), [n_rows][ldx]
  size_t xlo_off;         // elements from x to its low-order plane (x = hi + lo), 0 = hi only
  int ldx, M, K, n_tiles;
  int splits;             // K splits (K / splits is a multiple of 128)
  float* out;             // [splits][n_tiles * 8][M]
  int unit_begin;         // first global work unit (tile, split) of this segment (set by the launcher)
};

struct GemvArgs {
  GemvSeg seg[kMaxSeg];
  int nseg;
  int total_units;
};

// fmt: 0 = BF16 weights, 1 = Q8G64 weights.  max_tiles: largest n_tiles over segments.
// pdl: launch with programmatic stream serialisation.
cudaError_t launch_gemv(GemvArgs& a, int fmt, int max_tiles, int num_sms, bool pdl, cudaStream_t st);

// K split for a launch over `tiles` 16-row tiles of depth K: minimises whole-grid
// rounds of (tile, split) units times their length in 128-wide batches, plus one
// batch of pipeline start per unit and the consumer's cost of adding planes.
int gemv_choose_splits(int tiles, int K, int num_sms);

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
