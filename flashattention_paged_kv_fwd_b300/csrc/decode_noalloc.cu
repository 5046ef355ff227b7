// pa_attn_decode_paged_noalloc: the paged decode for callers that cannot
// allocate device memory on the call path.
//
// The regular entry point asks the caller for a workspace that holds the
// split-KV partial outputs. Some callers cannot provide one: a serving process
// that reserves its whole memory budget at start-up and must not allocate
// afterwards (cudaMalloc can synchronise the device, and can fail once memory
// is fragmented), or a plugin that only receives tensors from a host framework
// that owns every device allocation. This variant keeps the partials in one
// fixed array compiled into the library instead, and otherwise runs exactly
// the same kernels as pa_attn_decode_paged.
//
// The array is a file-scope __device__ variable of PA_NOALLOC_SCRATCH_BYTES:
// every GPU that loads the library holds it until the process exits. From host
// code its name is only a host-side stand-in, so its device address is looked
// up with cudaGetSymbolAddress on the first call in a context and cached per
// device together with that context's unique id. A call from another context
// of the device, or from the context that replaced a reset one (the module and
// its array are loaded anew there, possibly at another address), finds a
// different id and looks the address up again.
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>

#include "../../include/pagedattn.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct ScratchEntry {
  unsigned long long ctx_id;  // unique id of the context the lookup was made in (0 = none)
  void* addr;
};
std::mutex g_scratch_mu;
ScratchEntry g_scratch[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(p);
  return nullptr;
}

// Unique id of the calling thread's current context (ids are never reused
// within a process), or 0 when it cannot be read.
unsigned long long current_context_id() {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_decode_scratch in the current context of the current
// device, or nullptr if the lookup failed.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  const unsigned long long id = current_context_id();  // 0 before the thread has a context
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchEntry& e = g_scratch[dev];
  if (id != 0 && e.ctx_id == id && e.addr != nullptr) return e.addr;
  void* p = nullptr;
  // (this also makes the device's primary context current if none was)
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();  // leave no sticky error from a failed lookup behind
    return nullptr;
  }
  const unsigned long long now = id != 0 ? id : current_context_id();
  // without a context id nothing is cached: every call looks the address up
  e.ctx_id = now;
  e.addr = now != 0 ? p : nullptr;
  return p;
}

}  // namespace

extern "C" int pa_attn_decode_paged_noalloc(const void* q, const void* k_cache,
                                            const void* v_cache, const int32_t* block_table,
                                            int max_blocks_per_seq, const int32_t* seq_lens,
                                            void* o, float* lse, int B, int Hq, int Hkv, int d,
                                            int block_size, int num_blocks, int window,
                                            float scale, int num_splits, pa_dtype dtype,
                                            int32_t* err_flag, void* stream) {
  // The partials this call needs (0 when every sequence fits one range, or
  // when the arguments are invalid -- the delegate below then rejects them).
  const size_t need = pa_decode_workspace_bytes(B, Hq, Hkv, d, max_blocks_per_seq, block_size,
                                                window, num_splits);
  if (need > static_cast<size_t>(PA_NOALLOC_SCRATCH_BYTES)) return PA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = scratch_address();
    if (scratch == nullptr) return PA_ERR_CUDA;
  }
  // Nothing in the scratch has to start at zero: every partial is written by
  // its range's CTA before the merge kernel of the same call reads it.
  return pa_attn_decode_paged(q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, o,
                              lse, B, Hq, Hkv, d, block_size, num_blocks, window, scale,
                              num_splits, scratch, need > 0 ? PA_NOALLOC_SCRATCH_BYTES : 0, dtype,
                              err_flag, stream);
}
