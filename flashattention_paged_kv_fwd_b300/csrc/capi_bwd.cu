// C ABI of the attention backward pass (declared in include/pagedattn.h):
// host-side checks, TMA descriptor encoding and dispatch. Every check that can
// fail runs before any CUDA call.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "bwd_kernels.h"
#include "host_util.h"

using namespace pa::host;

namespace {

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

}  // namespace

extern "C" {

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
  a.wait_ns = pa::role_wait_limit_ns();
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

}  // extern "C"
