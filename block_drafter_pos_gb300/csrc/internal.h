// Internal launch interfaces between the host orchestration (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace df2 {

constexpr int kMaxSeg = 4;

// One weight-streaming GEMV segment: out[s][n][m] = sum_{k in split s} W[m][k] * X[n][k].
struct GemvSeg {
  const void* w;          // bf16 [M][K] or int8 codes [M][K]
  const uint16_t* scale;  // Q8: bf16 [M][K/64]
  const uint16_t* bias;   // Q8: bf16 [M][K/64]
  const void* x;          // activations: bf16 (BF16 weights) or fp16 (Q8 weights), [n_rows][ldx]
  const float* xsum;      // Q8: per-64-group sums of x, [n_rows][K/64]
  float* out;             // [splits][n_rows][M] fp32
  int M, K, ldx;
  int n_tiles;            // n_rows / 8
  int splits;             // K split count (K/splits is a multiple of 128)
  int unit_begin;         // first global work unit of this segment
};

struct GemvArgs {
  GemvSeg seg[kMaxSeg];
  int nseg;
  int total_units;
};

// fmt: 0 = BF16 weights, 1 = Q8G64 weights.  max_tiles: largest n_tiles over segments.
cudaError_t launch_gemv(const GemvArgs& a, int fmt, int max_tiles, int num_sms, cudaStream_t st);

}  // namespace df2
