// C ABI of libpagedattn.so (declared in include/pagedattn.h): host-side
// argument checks, TMA descriptor encoding and kernel dispatch.
//
// Every check that can fail runs before any CUDA call, so an invalid call
// returns an error without touching the device. The library keeps no state
// besides the cached driver entry point for cuTensorMapEncodeTiled, the SM
// count per device and the per-kernel shared-memory attribute flags.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pagedattn.h"
#include "bwd_kernels.h"
#include "mla_kernels.h"
#include "pa_kernels.h"

namespace {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  }
  return fn;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t elem_size(pa_dtype dt) { return dt == PA_F32 ? 4 : 2; }

bool valid_dtype(pa_dtype dt) { return dt == PA_BF16 || dt == PA_F32; }

// bf16 tensor map over a token-major [rows, heads, d] tensor (3D) or a
// pool [num_blocks, block_size, heads, d] (4D), 64-element x 128-byte-swizzled
// boxes.
bool encode_3d(CUtensorMap* m, const void* ptr, int d, int heads, long long rows, int box_rows) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(heads) * d * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 tensor map over a token-major [rows, heads, d] buffer: boxes of 32
// elements (128 bytes) x 1 head x 32 rows, 128-byte swizzled.
bool encode_3d_f32_rows32(CUtensorMap* m, const void* ptr, int d, int heads, long long rows) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                                 static_cast<cuuint64_t>(heads) * d * 4};
  const cuuint32_t box[3] = {32, 1, 32};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

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

// Pool [num_blocks, block_size, heads, d] described with the dimensions in
// the order (d, token, head, block): one box of 64 elements x block_size
// tokens x `box_heads` heads lands in shared memory as `box_heads` head tiles
// of block_size x 128 bytes, each 128-byte swizzled exactly like a one-head
// box, so a whole page of a CTA's heads is one copy per 64-column panel.
bool encode_pool(CUtensorMap* m, const void* ptr, int d, int heads, int block_size,
                 int num_blocks, int box_heads) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(block_size),
                              static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(heads) * d * 2,
                                 static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(block_size) * heads * d * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(block_size),
                             static_cast<cuuint32_t>(box_heads), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

double softmax_scale(float scale, int d) {
  return scale > 0.f ? static_cast<double>(scale) : 1.0 / std::sqrt(static_cast<double>(d));
}

float scale_log2(float scale, int d) {
  return static_cast<float>(softmax_scale(scale, d) * 1.4426950408889634074);  // * log2(e)
}

}  // namespace

extern "C" {

const char* pa_status_str(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int pa_attn_prefill(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int Hq, int Hkv, int N, int d, const int32_t* cu_seqlens, int max_seqlen,
                    int causal, int window, float scale, pa_dtype dtype, int32_t* err_flag,
                    void* stream) {
  if (!valid_dtype(dtype)) return PA_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || N < 0 || Hq % Hkv != 0) return PA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o) return PA_ERR_INVALID_ARG;
  // the bf16 epilogue writes O in 32-byte pieces
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(o, dtype == PA_BF16 ? 32 : 16))
    return PA_ERR_INVALID_ARG;
  if (lse && !aligned(lse, 4)) return PA_ERR_INVALID_ARG;
  if (err_flag && !aligned(err_flag, 4)) return PA_ERR_INVALID_ARG;
  if (window > 0 && !causal) return PA_ERR_UNSUPPORTED;
  if (cu_seqlens && (max_seqlen < 0 || !aligned(cu_seqlens, 4))) return PA_ERR_INVALID_ARG;
  const long long T = cu_seqlens ? static_cast<long long>(N) : static_cast<long long>(B) * N;
  if (T > 0x7FFFFFFFLL) return PA_ERR_INVALID_ARG;
  const int msl = cu_seqlens ? max_seqlen : N;
  if (T == 0 || msl == 0) return PA_OK;

  pa::PrefillArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse; a.cu_seqlens = cu_seqlens; a.err = err_flag;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.N = N; a.T = static_cast<int>(T); a.d = d;
  a.max_seqlen = msl; a.causal = causal ? 1 : 0; a.window = window > 0 ? window : 0;
  a.scale_log2 = scale_log2(scale, d);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (dtype == PA_F32) {
    e = pa::launch_prefill_f32(a, s);
  } else {
    CUtensorMap qm, km, vm;
    if (!encode_3d(&qm, q, d, Hq, T, 128) || !encode_3d(&km, k, d, Hkv, T, 128) ||
        !encode_3d(&vm, v, d, Hkv, T, 128))
      return PA_ERR_CUDA;
    e = pa::launch_prefill_bf16(a, qm, km, vm, sm_count(), s);
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_attn_prefill_paged(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_table, int max_blocks_per_seq,
                          const int32_t* seq_lens, const int32_t* cu_seqlens_q, int total_q,
                          int max_seqlen_q, void* o, float* lse, int B, int Hq, int Hkv, int d,
                          int block_size, int num_blocks, int causal, int window, float scale,
                          pa_dtype dtype, int32_t* err_flag, void* stream) {
  if (!valid_dtype(dtype)) return PA_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || total_q < 0 || max_seqlen_q < 0 ||
      num_blocks <= 0 || max_blocks_per_seq <= 0)
    return PA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PA_ERR_INVALID_ARG;
  if (dtype != PA_BF16 || block_size != 16) return PA_ERR_UNSUPPORTED;
  if (window > 0 && !causal) return PA_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_blocks_per_seq) * block_size > 0x7FFFFFFFLL)
    return PA_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !cu_seqlens_q || !o)
    return PA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 32) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(cu_seqlens_q, 4) ||
      (lse && !aligned(lse, 4)) || (err_flag && !aligned(err_flag, 4)))
    return PA_ERR_INVALID_ARG;
  if (total_q == 0 || max_seqlen_q == 0) return PA_OK;

  pa::PrefillArgs a{};
  a.q = q; a.k = k_cache; a.v = v_cache; a.o = o; a.lse = lse; a.cu_seqlens = cu_seqlens_q;
  a.err = err_flag;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.N = total_q; a.T = total_q; a.d = d;
  a.max_seqlen = max_seqlen_q; a.causal = causal ? 1 : 0; a.window = window > 0 ? window : 0;
  a.scale_log2 = scale_log2(scale, d);
  a.table = block_table; a.seq_lens_k = seq_lens;
  a.max_blocks = max_blocks_per_seq; a.num_blocks = num_blocks;
  CUtensorMap qm, km, vm;
  if (!encode_3d(&qm, q, d, Hq, total_q, 128) ||
      !encode_pool(&km, k_cache, d, Hkv, block_size, num_blocks, 1) ||
      !encode_pool(&vm, v_cache, d, Hkv, block_size, num_blocks, 1))
    return PA_ERR_CUDA;
  const cudaError_t e =
      pa::launch_prefill_bf16(a, qm, km, vm, sm_count(), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_attn_prefill_backward_workspace_bytes(int total_tokens, int Hq, int d) {
  if (total_tokens < 0 || Hq <= 0 || (d != 64 && d != 128)) return 0;
  return pa::backward_workspace_bytes(total_tokens, Hq, d);
}

int pa_attn_prefill_backward(const void* q, const void* k, const void* v, const void* o,
                             const void* dout, const float* lse, void* dq, void* dk, void* dv,
                             int B, int Hq, int Hkv, int N, int d, const int32_t* cu_seqlens,
                             int max_seqlen, int causal, int window, float scale,
                             void* workspace, size_t workspace_bytes, pa_dtype dtype,
                             int32_t* err_flag, void* stream) {
  if (!valid_dtype(dtype)) return PA_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || N < 0 || Hq % Hkv != 0) return PA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PA_ERR_INVALID_ARG;
  if (dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (window > 0 && !causal) return PA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return PA_ERR_INVALID_ARG;
  // dK / dV rows are written in 32-byte pieces, dQ in 16-byte pieces
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(dout, 16) || !aligned(lse, 4) || !aligned(dq, 16) || !aligned(dk, 32) ||
      !aligned(dv, 32) || (err_flag && !aligned(err_flag, 4)))
    return PA_ERR_INVALID_ARG;
  if (cu_seqlens && (max_seqlen < 0 || !aligned(cu_seqlens, 4))) return PA_ERR_INVALID_ARG;
  const long long T = cu_seqlens ? static_cast<long long>(N) : static_cast<long long>(B) * N;
  if (T > 0x7FFFFFFFLL) return PA_ERR_INVALID_ARG;
  const int msl = cu_seqlens ? max_seqlen : N;
  if (T == 0 || msl == 0) return PA_OK;
  const size_t need = pa::backward_workspace_bytes(T, Hq, d);
  if (!workspace || workspace_bytes < need) return PA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PA_ERR_INVALID_ARG;

  pa::BackwardArgs a{};
  a.q = q; a.k = k; a.v = v; a.o = o; a.dout = dout; a.lse = lse;
  a.dq = dq; a.dk = dk; a.dv = dv;
  a.dq_acc = static_cast<float*>(workspace);
  a.dvec = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                    (static_cast<size_t>(T) * Hq * d * 4 + 255) / 256 * 256);
  a.cu_seqlens = cu_seqlens; a.err = err_flag;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.N = N; a.T = static_cast<int>(T); a.d = d;
  a.max_seqlen = msl; a.causal = causal ? 1 : 0; a.window = window > 0 ? window : 0;
  a.scale_log2 = scale_log2(scale, d);
  a.scale = static_cast<float>(softmax_scale(scale, d));
  CUtensorMap qm, km, vm, dom, dqm;
  if (!encode_3d(&qm, q, d, Hq, T, 128) || !encode_3d(&km, k, d, Hkv, T, 128) ||
      !encode_3d(&vm, v, d, Hkv, T, 128) || !encode_3d(&dom, dout, d, Hq, T, 128) ||
      !encode_3d_f32_rows32(&dqm, a.dq_acc, d, Hq, T))
    return PA_ERR_CUDA;
  const cudaError_t e = pa::launch_prefill_backward_bf16(a, qm, km, vm, dom, dqm, sm_count(),
                                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

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
  CUtensorMap cm;
  if (!encode_mla_pool(&cm, cache, num_blocks)) return PA_ERR_CUDA;
  const cudaError_t e = pa::launch_mla_decode_bf16(a, p, cm, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_kv_append_paged(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                       const int32_t* block_table, int max_blocks_per_seq,
                       const int32_t* seq_lens, const int32_t* cu_new, int num_new_tokens,
                       int B, int Hkv, int d, int block_size, int num_blocks, pa_dtype dtype,
                       int32_t* err_flag, void* stream) {
  if (!valid_dtype(dtype)) return PA_ERR_INVALID_ARG;
  if (B <= 0 || Hkv <= 0 || block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0)
    return PA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PA_ERR_INVALID_ARG;
  if (num_new_tokens < 0 || (!cu_new && num_new_tokens != B)) return PA_ERR_INVALID_ARG;
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !seq_lens)
    return PA_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      (cu_new && !aligned(cu_new, 4)) || (err_flag && !aligned(err_flag, 4)))
    return PA_ERR_INVALID_ARG;
  const long long row_bytes = static_cast<long long>(Hkv) * d * elem_size(dtype);
  if (row_bytes % 16 != 0 || row_bytes > 0x7FFFFFFFLL) return PA_ERR_INVALID_ARG;
  const cudaError_t e = pa::launch_kv_append(
      k_new, v_new, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, cu_new,
      num_new_tokens, B, static_cast<int>(row_bytes), block_size, num_blocks, err_flag,
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* src_blocks,
                   const int32_t* dst_blocks, int num_pairs, int block_size, int Hkv, int d,
                   int num_blocks, pa_dtype dtype, int32_t* err_flag, void* stream) {
  if (!valid_dtype(dtype)) return PA_ERR_INVALID_ARG;
  if (num_pairs < 0 || block_size <= 0 || Hkv <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !src_blocks || !dst_blocks) return PA_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(src_blocks, 4) ||
      !aligned(dst_blocks, 4) || (err_flag && !aligned(err_flag, 4)))
    return PA_ERR_INVALID_ARG;
  const long long block_bytes =
      static_cast<long long>(block_size) * Hkv * d * static_cast<long long>(elem_size(dtype));
  if (block_bytes % 16 != 0 || block_bytes / 16 > 0x7FFFFFFFLL) return PA_ERR_INVALID_ARG;
  const cudaError_t e = pa::launch_copy_blocks(k_cache, v_cache, src_blocks, dst_blocks,
                                               num_pairs, block_bytes, num_blocks, err_flag,
                                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_decode_workspace_bytes(int B, int Hq, int Hkv, int d, int max_blocks_per_seq,
                                 int block_size, int window, int num_splits) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || (d != 64 && d != 128) ||
      max_blocks_per_seq <= 0 || block_size != 16 || num_splits < 0)
    return 0;
  const pa::DecodePlan p = pa::plan_decode(B, Hq, Hkv, d, max_blocks_per_seq, block_size, window,
                                           num_splits, num_splits > 0 ? 0 : sm_count(), false);
  const pa::DecodePlan pf = pa::plan_decode(B, Hq, Hkv, d, max_blocks_per_seq, block_size, window,
                                            num_splits, num_splits > 0 ? 0 : sm_count(), true);
  return p.workspace > pf.workspace ? p.workspace : pf.workspace;
}

int pa_attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_table, int max_blocks_per_seq,
                         const int32_t* seq_lens, void* o, float* lse, int B, int Hq, int Hkv,
                         int d, int block_size, int num_blocks, int window, float scale,
                         int num_splits, void* workspace, size_t workspace_bytes,
                         pa_dtype dtype, int32_t* err_flag, void* stream) {
  if (!valid_dtype(dtype)) return PA_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || num_blocks <= 0 ||
      max_blocks_per_seq <= 0 || num_splits < 0)
    return PA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PA_ERR_INVALID_ARG;
  if (block_size != 16) return PA_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_blocks_per_seq) * block_size > 0x7FFFFFFFLL)
    return PA_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o) return PA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || (lse && !aligned(lse, 4)) ||
      (err_flag && !aligned(err_flag, 4)))
    return PA_ERR_INVALID_ARG;
  if (workspace && !aligned(workspace, 256)) return PA_ERR_INVALID_ARG;

  const bool f32 = dtype == PA_F32;
  // bf16: the G query heads of a KV head are packed 16 per warp, at most
  // 8 (d = 128) or 12 (d = 64) warps per KV head.
  if (!f32 && (Hq / Hkv + 15) / 16 > (d == 128 ? 8 : 12)) return PA_ERR_UNSUPPORTED;
  const pa::DecodePlan p = pa::plan_decode(B, Hq, Hkv, d, max_blocks_per_seq, block_size, window,
                                           num_splits, num_splits > 0 ? 0 : sm_count(), f32);
  if (p.workspace > 0 && (!workspace || workspace_bytes < p.workspace)) return PA_ERR_WORKSPACE;

  pa::DecodeArgs a{};
  a.q = q; a.o = o; a.lse = lse; a.k_cache = k_cache; a.v_cache = v_cache;
  a.table = block_table; a.seq_lens = seq_lens; a.err = err_flag;
  if (p.workspace > 0) {
    const size_t n = static_cast<size_t>(B) * Hq * p.num_splits;
    a.ws_o = static_cast<float*>(workspace);
    a.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        (n * d * 4 + 255) / 256 * 256);
  }
  a.max_blocks = max_blocks_per_seq; a.num_blocks = num_blocks; a.B = B; a.Hq = Hq;
  a.Hkv = Hkv; a.d = d; a.window = window > 0 ? window : 0;
  a.scale_log2 = scale_log2(scale, d);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (f32) {
    e = pa::launch_decode_f32(a, p, s);
  } else {
    CUtensorMap km, vm;
    if (!encode_pool(&km, k_cache, d, Hkv, block_size, num_blocks, p.hg) ||
        !encode_pool(&vm, v_cache, d, Hkv, block_size, num_blocks, p.hg))
      return PA_ERR_CUDA;
    e = pa::launch_decode_bf16(a, p, km, vm, s);
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"
