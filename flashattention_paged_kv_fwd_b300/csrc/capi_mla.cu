// C ABI of multi-head latent attention (declared in include/pagedattn.h):
// host-side checks, TMA descriptor encoding and dispatch. Every check that can
// fail runs before any CUDA call.
#include <cmath>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "host_util.h"
#include "mla_kernels.h"
#include "pa_kernels.h"

using namespace pa::host;

namespace {

// MLA latent pool [num_blocks, 16, 576] bf16 described as (64 elements,
// token, 64-element panel, block): one box per block lands as 9 panels of
// 16 rows x 128 bytes, 128-byte swizzled.
bool encode_mla_pool(CUtensorMap* m, const void* ptr, int num_blocks) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t row = pa::kMlaRow * 2;
  const cuuint64_t dims[4] = {64, 16, static_cast<cuuint64_t>(pa::kMlaRow / 64),
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[3] = {row, 128, 16 * row};
  const cuuint32_t box[4] = {64, 16, static_cast<cuuint32_t>(pa::kMlaRow / 64), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

int pa_mla_append_paged(const void* rows_new, void* cache, const int32_t* block_table,
                        int max_blocks_per_seq, const int32_t* seq_lens, const int32_t* cu_new,
                        int num_new_tokens, int B, int row_elems, int block_size, int num_blocks,
                        pa_dtype dtype, int32_t* err_flag, void* stream) {
  if (!valid_dtype(dtype)) return PA_ERR_INVALID_ARG;
  if (B <= 0 || row_elems <= 0 || block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_new_tokens < 0 || (!cu_new && num_new_tokens != B)) return PA_ERR_INVALID_ARG;
  if (!rows_new || !cache || !block_table || !seq_lens) return PA_ERR_INVALID_ARG;
  if (!aligned(rows_new, 16) || !aligned(cache, 16) || !aligned(block_table, 4) ||
      !aligned(seq_lens, 4) || (cu_new && !aligned(cu_new, 4)) ||
      (err_flag && !aligned(err_flag, 4)))
    return PA_ERR_INVALID_ARG;
  const long long row_bytes = static_cast<long long>(row_elems) * elem_size(dtype);
  if (row_bytes % 16 != 0 || row_bytes > 0x7FFFFFFFLL) return PA_ERR_INVALID_ARG;
  const cudaError_t e = pa::launch_kv_append(
      rows_new, nullptr, cache, nullptr, block_table, max_blocks_per_seq, seq_lens, cu_new,
      num_new_tokens, B, static_cast<int>(row_bytes), block_size, num_blocks, err_flag,
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_mla_decode_workspace_bytes(int B, int H, int d_c, int d_rope, int max_blocks_per_seq,
                                     int block_size, int num_splits) {
  if (B <= 0 || H <= 0 || d_c != pa::kMlaDc || d_rope != pa::kMlaDr || block_size != 16 ||
      max_blocks_per_seq <= 0 || num_splits < 0)
    return 0;
  return pa::plan_mla_decode(B, H, max_blocks_per_seq, num_splits,
                             num_splits > 0 ? 0 : sm_count()).workspace;
}

int pa_mla_decode_paged(const void* q, const void* cache, const int32_t* block_table,
                        int max_blocks_per_seq, const int32_t* seq_lens, void* o, float* lse,
                        int B, int H, int d_c, int d_rope, int block_size, int num_blocks,
                        float scale, int num_splits, void* workspace, size_t workspace_bytes,
                        pa_dtype dtype, int32_t* err_flag, void* stream) {
  if (!valid_dtype(dtype)) return PA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || num_splits < 0 ||
      d_c <= 0 || d_rope < 0 || !(scale > 0.f) || !std::isfinite(scale))
    return PA_ERR_INVALID_ARG;
  if (dtype != PA_BF16 || d_c != pa::kMlaDc || d_rope != pa::kMlaDr || block_size != 16)
    return PA_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_blocks_per_seq) * block_size > 0x7FFFFFFFLL)
    return PA_ERR_INVALID_ARG;
  if (!q || !cache || !block_table || !seq_lens || !o) return PA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(cache, 16) || !aligned(o, 16) || !aligned(block_table, 4) ||
      !aligned(seq_lens, 4) || (lse && !aligned(lse, 4)) || (err_flag && !aligned(err_flag, 4)))
    return PA_ERR_INVALID_ARG;
  if (workspace && !aligned(workspace, 256)) return PA_ERR_INVALID_ARG;
  const pa::MlaPlan p = pa::plan_mla_decode(B, H, max_blocks_per_seq, num_splits,
                                            num_splits > 0 ? 0 : sm_count());
  if (p.workspace > 0 && (!workspace || workspace_bytes < p.workspace)) return PA_ERR_WORKSPACE;
  pa::MlaArgs a{};
  a.q = q; a.o = o; a.lse = lse; a.table = block_table; a.seq_lens = seq_lens; a.err = err_flag;
  if (p.workspace > 0) {
    const size_t n = static_cast<size_t>(B) * H * p.num_splits;
    a.ws_o = static_cast<float*>(workspace);
    a.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        (n * pa::kMlaDc * 4 + 255) / 256 * 256);
  }
  a.max_blocks = max_blocks_per_seq; a.num_blocks = num_blocks; a.B = B; a.H = H;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  a.wait_ns = pa::role_wait_limit_ns();
  CUtensorMap cm;
  if (!encode_mla_pool(&cm, cache, num_blocks)) return PA_ERR_CUDA;
  const cudaError_t e = pa::launch_mla_decode_bf16(a, p, cm, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"
