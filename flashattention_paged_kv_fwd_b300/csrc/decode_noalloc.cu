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
// code its name is only a host-side stand-in, so the device address is looked
// up once per device with cudaGetSymbolAddress and cached.
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/pagedattn.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of g_decode_scratch on the current device (looked up on the
// first call for that device), or nullptr if the lookup failed.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // leave no sticky error from a failed lookup behind
      return nullptr;
    }
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
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
