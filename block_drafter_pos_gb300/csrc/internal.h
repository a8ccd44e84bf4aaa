// Internal launch interfaces between the host orchestration (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace df2 {

constexpr int kMaxSeg = 4;

// K elements of one pipeline stage of the weight-streaming GEMV (64 weight rows).
constexpr int kGemvStageK = 128;

#ifdef __CUDACC__
#define DF2_HD __host__ __device__
#else
#define DF2_HD
#endif

// One weight-streaming GEMV segment (a matrix and its activations) of a launch.
// A launch's work is the sequence of (64-row weight block, kGemvStageK of K)
// stages of its segments, in order; CTA c of C takes stages
// [floor(c T / C), floor((c + 1) T / C)) of the T in total (stream-K: balanced to
// one stage whatever the shapes).  A block's K sum is split among the CTAs that
// share its stages; each writes its part to plane (c - first CTA of the block):
//   out[p][n][m] = sum over CTA p's stages of block m/64 of W[m][k] * X[n][k].
// The consumer adds planes 0 .. plane_count - 1 in order (GemvPlanes).
struct GemvSeg {
  CUtensorMap wmap;       // W [M][K]: bf16 boxes 64 K x 64 rows (128-byte swizzle) or int8 64 K x 64 rows (64-byte)
  CUtensorMap xmap;       // X planes [2][rows][K] (hi rows, then lo rows): boxes of 8 rows (gemv_encode_xmap)
  const uint16_t* scale;  // Q8: bf16 [M][K/64]
  const uint16_t* bias;
  int x_lo_row;           // first row of the low-order plane in xmap
  int M, K, n_tiles;
  float* out;             // [planes][n_tiles * 8][M]
  long long stage_begin;  // first stage of this segment in the launch (set by gemv_plan)
  const void* xt;         // tensor-core GEMM: X in its operand layout (slices of xt_rows rows), or null (xmap)
  int xt_rows;
};

struct GemvArgs {
  GemvSeg seg[kMaxSeg];
  int nseg;
  long long total_stages;  // T (set by gemv_plan)
  int stage_k;             // K per stage: 128 (bf16) or 256 (int8) (set by gemv_plan)
  int* err;                // set nonzero if a pipeline wait gave up (never in a correct run), or null
};

// Where the partial planes of one segment's output channel m are: planes
// 0 .. count(m) - 1, with count from the block's first and last stage.
struct GemvPlanes {
  long long T, base;  // launch stages; the segment's first stage
  int C, kst;         // launch CTAs; stages per weight block
  int bshift;         // log2 of the rows of one weight block (64 for the GEMV, 128 for the GEMM)
};

// (the element-wise kernels evaluate this per thread: in 32-bit arithmetic whenever
// the product fits, since a 64-bit division costs several times as many instructions)
// Context chunks per attention part (host planning).  A part's CTA streams its chunks
// one after the other; each part costs a fixed latency (queries, first copy, merge,
// partial stores) and a partial for the combine.  Parts are at most 8 per (request,
// KV head), and longer while the grid exceeds 1.3 waves of two CTAs per SM; at most
// 16 chunks a part.  Measured (ms per step): 1 request, context 1024: 1 chunk 1.181,
// 2: 1.168, 4: 1.172; context 2048: 1: 1.032, 2: 1.022, 4: 1.016; 4 requests,
// context 8192: 2: 1.341, 4: 1.311, 8: 1.342; 16 requests: 4: 2.010, 8: 1.977,
// 16: 1.948, 32: 2.104.
inline int attn_chunks_per_part(int n_req, int nkv, int n_ctx_chunks, int num_sms) {
  int c = 1;
  while (c < 16 && (n_ctx_chunks + c - 1) / c > 8) c *= 2;
  while (c < 16 && 10LL * n_req * nkv * ((n_ctx_chunks + c - 1) / c + 1) > 26LL * num_sms) c *= 2;
  return c;
}

DF2_HD inline int gemv_cta_of_stage(long long t, int C, long long T) {
  const unsigned long long num = static_cast<unsigned long long>(t + 1) * static_cast<unsigned long long>(C) - 1ull;
  if (num <= 0xFFFFFFFFull && T <= 0xFFFFFFFFll)
    return static_cast<int>(static_cast<unsigned int>(num) / static_cast<unsigned int>(T));
  return static_cast<int>(num / static_cast<unsigned long long>(T));
}

DF2_HD inline int gemv_plane_count(const GemvPlanes& p, int m) {
  const long long b0 = p.base + static_cast<long long>(m >> p.bshift) * p.kst;
  return gemv_cta_of_stage(b0 + p.kst - 1, p.C, p.T) - gemv_cta_of_stage(b0, p.C, p.T) + 1;
}

// Fills stage_begin, total_stages and stage_k for the weight format; returns the
// CTA count of the launch.
int gemv_plan(GemvArgs& a, int num_sms, int fmt);
// Plane map of segment i of a planned launch with C CTAs, and its largest plane count.
GemvPlanes gemv_planes(const GemvArgs& a, int i, int C);
int gemv_max_planes(const GemvArgs& a, int i, int C);

// Encodes the tensor map of one weight matrix [M][K] (bf16 when fmt == 0, int8
// codes when fmt == 1).  Returns false if the driver rejects it.
bool gemv_encode_wmap(CUtensorMap* map, const void* w, int M, int K, int fmt);

// Encodes the tensor map of an activation buffer of `rows` rows of width K per
// plane, hi plane then lo plane (bf16 when fmt == 0, fp16 when fmt == 1).
bool gemv_encode_xmap(CUtensorMap* map, const void* x, int rows, int K, int fmt);

// Two-dimensional bulk-copy descriptor of a row-major [rows][inner] array of esz-byte
// elements, boxes of box_rows x box_inner; rows past the end read as zero.
bool tma_encode_2d(CUtensorMap* map, CUtensorMapDataType dt, int esz, const void* p, int inner, int rows,
                   int box_inner, int box_rows, CUtensorMapSwizzle swz);

// ---------------------------------------------------------------- tensor-core GEMM
// The same segments, stage order, stream-K split and partial planes as the GEMV,
// for calls with many activation rows (8 * n_tiles <= 256): weight blocks of 128
// rows, stages of 64 K (bf16) or 128 K (int8), activations one 16-bit plane, read
// from the operand layout the element-wise kernels write (xt) or through xmap.
// Fills stage_begin, total_stages and stage_k; returns the CTA count (two per SM for
// bf16, one for int8).
// nmax: the launch's largest activation-row count rounded up to 16, 128 or 256 (the
// int8 stage length depends on it; wide_nmax gives the launch's).
int wide_plan(GemvArgs& a, int num_sms, int fmt, int nmax);
int wide_nmax(const GemvArgs& a);
GemvPlanes wide_planes(const GemvArgs& a, int i, int C);
int wide_max_planes(const GemvArgs& a, int i, int C);
// Weight map: bf16 boxes 64 K x 128 rows or int8 boxes 128 K x 128 rows (128-byte rows, 128-byte swizzle).
bool wide_encode_wmap(CUtensorMap* map, const void* w, int M, int K, int fmt);
// Activation map of `rows` rows of width K: boxes 64 K x round_up(rows, 16) rows (128-byte swizzle).
bool wide_encode_xmap(CUtensorMap* map, const void* x, int rows, int K, int fmt);
cudaError_t launch_wide(GemvArgs& a, int fmt, int num_sms, bool pdl, cudaStream_t st);

// fmt: 0 = BF16 weights, 1 = Q8G64 weights.  max_tiles: largest n_tiles over segments.
// pdl: launch with programmatic stream serialisation.
cudaError_t launch_gemv(GemvArgs& a, int fmt, int max_tiles, int num_sms, bool pdl, cudaStream_t st);

// Raises a kernel's dynamic shared-memory limit on the current device, once per
// (call site, device): the attribute belongs to a device, so a process driving
// several GPUs sets it on each.  `done` is the call site's set of devices (bit d).
template <typename Kern>
cudaError_t set_smem_once(Kern kern, int smem, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (bit != 0ull && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && bit != 0ull) done.fetch_or(bit, std::memory_order_release);
  return e;
}

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
