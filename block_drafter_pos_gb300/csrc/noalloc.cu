// LM head + top-16 for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all.  Examples: a serving runtime whose
// allocator owns every byte of HBM, or a plug-in that runs inside another
// framework's memory pool.  Others cannot afford an allocation on their path: a
// first-use cudaMalloc can synchronise the device or fail with out-of-memory in
// the middle of a step.  The handle-based entry points reserve their scratch at
// dflash2_create time; this one needs no handle.  The per-CTA candidate lists of
// the LM-head kernel live in one fixed device array of this library.  The array
// is loaded with the library and held on every GPU that uses it until the
// process exits.
#include <atomic>
#include <mutex>

#include "../../include/dflash2.h"
#include "glue.h"

using namespace df2;

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kKeys = static_cast<size_t>(DFLASH2_NOALLOC_MAX_ROWS) * DFLASH2_NOALLOC_MAX_CTAS * 16;

// [rows][CTAs][16] candidate keys (value bits + vocabulary id), 1.25 MiB.
static __device__ __align__(256) unsigned long long g_noalloc_keys[kKeys];
// Set by the LM-head kernel when one of its bounded pipeline waits gives up; the
// merge then writes the sentinel instead of candidates.  Cleared by every call.
static __device__ __align__(16) int g_noalloc_err;

struct DeviceSlot {
  unsigned long long* keys;  // device address of g_noalloc_keys on this device
  int* err;                  // device address of g_noalloc_err on this device
  int n_cta;
};

std::mutex g_mu;
DeviceSlot g_slots[kMaxDevices];
bool g_ready[kMaxDevices];
std::atomic<int> g_inject_error{0};

// CTAs of one call: two per SM like the handle's LM head, so every SM streams the
// same share of the vocabulary; where that exceeds the array's CTA bound, one per SM
// (or the bound itself on a GPU with more SMs than it).
int noalloc_ctas(int sms) {
  const int two = lmhead_ctas(sms);
  if (two <= DFLASH2_NOALLOC_MAX_CTAS) return two;
  return sms <= DFLASH2_NOALLOC_MAX_CTAS ? sms : DFLASH2_NOALLOC_MAX_CTAS;
}

// Looks up the arrays' device addresses and the SM count once per device, with
// that device current.  The names g_noalloc_keys and g_noalloc_err are only
// host-side stand-ins in host code; the kernels must get these addresses instead.
cudaError_t device_slot(DeviceSlot* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ready[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_keys);
    if (e != cudaSuccess) return e;
    void* pe = nullptr;
    e = cudaGetSymbolAddress(&pe, g_noalloc_err);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_slots[dev].keys = static_cast<unsigned long long*>(p);
    g_slots[dev].err = static_cast<int*>(pe);
    g_slots[dev].n_cta = noalloc_ctas(sms);
    g_ready[dev] = true;
  }
  *out = g_slots[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" dflash2_status dflash2_debug_noalloc_inject_error(int32_t on) {
  if (on != 0 && on != 1) return DFLASH2_E_INVAL;
  g_inject_error.store(on, std::memory_order_relaxed);
  return DFLASH2_OK;
}

extern "C" dflash2_status dflash2_head_topk_noalloc(const void* lm_head, int32_t vocab, int32_t hidden_dim,
                                                    int32_t n_rows, const void* hidden, int32_t* cand_ids,
                                                    float* cand_logits, float* logits_out, void* stream) {
  if (!lm_head || !hidden || !cand_ids || !cand_logits) return DFLASH2_E_INVAL;
  if ((reinterpret_cast<uintptr_t>(lm_head) & 15u) || (reinterpret_cast<uintptr_t>(hidden) & 15u))
    return DFLASH2_E_INVAL;
  if (vocab < 16 || hidden_dim < 128 || n_rows < 8 || n_rows % 8) return DFLASH2_E_INVAL;
  // sizes the fixed scratch or the kernel's instantiations do not cover
  if (n_rows > DFLASH2_NOALLOC_MAX_ROWS || vocab % 16 || hidden_dim % 128) return DFLASH2_E_UNSUPPORTED;
  DeviceSlot slot;
  if (device_slot(&slot) != cudaSuccess) return DFLASH2_E_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The error word starts clear (set, under the test hook, as a pipeline wait that
  // gave up would set it).  A memset of a device symbol allocates nothing.
  if (cudaMemsetAsync(slot.err, g_inject_error.load(std::memory_order_relaxed) ? 1 : 0, sizeof(int), st) !=
      cudaSuccess)
    return DFLASH2_E_CUDA;
  // Every (row, CTA) list the merge reads is rewritten by the LM-head launch
  // first, so nothing left in the array by an earlier call is ever read.
  LmHeadArgs a;
  // bulk-copy descriptors live in the kernel's parameters: encoding them allocates nothing
  if (!lm_encode_map(&a.wmap, lm_head, hidden_dim, vocab, 64) || !lm_encode_map(&a.xmap, hidden, hidden_dim, n_rows, 8))
    return DFLASH2_E_CUDA;
  a.x_lo_row = -1;
  a.ss = nullptr;
  a.logits_out = logits_out;
  a.part_keys = slot.keys;
  a.V = vocab;
  a.H = hidden_dim;
  a.n_rows = n_rows;
  a.B = 8;  // rows are (request, block position) of blocks of 8
  a.nch = hidden_dim / 32;
  a.n_cta = slot.n_cta;
  a.eps = 0.f;
  a.err = slot.err;
  if (launch_lmhead(a, false, st) != cudaSuccess) return DFLASH2_E_CUDA;
  TopkMergeArgs m = {};
  m.part_keys = slot.keys;
  m.sel = nullptr;
  m.ss = nullptr;
  m.cand_ids = cand_ids;
  m.cand_logits = cand_logits;
  m.gate = nullptr;
  m.n_rows = n_rows;
  m.B = 8;
  m.n_cta = slot.n_cta;
  m.rank = 0;
  m.nch = hidden_dim / 128;
  m.H = hidden_dim;
  m.eps = 0.f;
  m.err = slot.err;
  if (launch_topk_merge(m, false, st) != cudaSuccess) return DFLASH2_E_CUDA;
  return DFLASH2_OK;
}
