// C ABI of libpagedattn.so (declared in include/pagedattn.h): host-side
// argument checks, TMA descriptor encoding and kernel dispatch.
//
// Every check that can fail runs before any CUDA call, so an invalid call
// returns an error without touching the device. The library keeps no state
// besides the cached driver entry point for cuTensorMapEncodeTiled, the SM
// count per device and the per-kernel shared-memory attribute flags.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pagedattn.h"
#include "../../include/pagedattn_testing.h"
#include "host_util.h"
#include "pa_kernels.h"

using namespace pa::host;

namespace pa {
namespace {
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitNs};
}  // namespace

unsigned long long role_wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
}  // namespace pa

extern "C" {

unsigned long long pa_testing_set_wait_limit_ns(unsigned long long ns) {
  const unsigned long long v = (ns == 0 || ns > pa::kDefaultWaitNs) ? pa::kDefaultWaitNs : ns;
  return pa::g_wait_limit_ns.exchange(v, std::memory_order_relaxed);
}

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
  a.wait_ns = pa::role_wait_limit_ns();
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
  a.wait_ns = pa::role_wait_limit_ns();
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
  const pa::DecodePlan p8 = pa::plan_decode(B, Hq, Hkv, d, max_blocks_per_seq, block_size, window,
                                            num_splits, num_splits > 0 ? 0 : sm_count(), false,
                                            true);
  size_t w = p.workspace > pf.workspace ? p.workspace : pf.workspace;
  return w > p8.workspace ? w : p8.workspace;
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
  if (!f32 && Hq / Hkv > pa::decode_max_group(d, false)) return PA_ERR_UNSUPPORTED;
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
  a.wait_ns = pa::role_wait_limit_ns();
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

int pa_kv_append_paged_fp8(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                           const float* k_scale, const float* v_scale, const int32_t* block_table,
                           int max_blocks_per_seq, const int32_t* seq_lens, const int32_t* cu_new,
                           int num_new_tokens, int B, int Hkv, int d, int block_size,
                           int num_blocks, int32_t* err_flag, void* stream) {
  if (B <= 0 || Hkv <= 0 || num_new_tokens < 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 ||
      block_size <= 0)
    return PA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PA_ERR_INVALID_ARG;
  if (!k_new || !v_new || !k_cache || !v_cache || !k_scale || !v_scale || !block_table ||
      !seq_lens)
    return PA_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 8) || !aligned(v_cache, 8) ||
      !aligned(k_scale, 4) || !aligned(v_scale, 4) || !aligned(block_table, 4) ||
      !aligned(seq_lens, 4) || (cu_new && !aligned(cu_new, 4)) ||
      (err_flag && !aligned(err_flag, 4)))
    return PA_ERR_INVALID_ARG;
  if (!cu_new && num_new_tokens != B) return PA_ERR_INVALID_ARG;
  const cudaError_t e = pa::launch_kv_append_fp8(
      k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_table, max_blocks_per_seq, seq_lens,
      cu_new, num_new_tokens, B, Hkv, d, block_size, num_blocks, err_flag,
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_attn_decode_paged_fp8(const void* q, const void* k_cache, const void* v_cache,
                             const float* k_scale, const float* v_scale,
                             const int32_t* block_table, int max_blocks_per_seq,
                             const int32_t* seq_lens, void* o, float* lse, int B, int Hq, int Hkv,
                             int d, int block_size, int num_blocks, int window, float scale,
                             int num_splits, void* workspace, size_t workspace_bytes,
                             int32_t* err_flag, void* stream) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || num_blocks <= 0 ||
      max_blocks_per_seq <= 0 || num_splits < 0)
    return PA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return PA_ERR_INVALID_ARG;
  if (block_size != 16) return PA_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_blocks_per_seq) * block_size > 0x7FFFFFFFLL)
    return PA_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !k_scale || !v_scale || !block_table || !seq_lens || !o)
    return PA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(k_scale, 4) || !aligned(v_scale, 4) || !aligned(block_table, 4) ||
      !aligned(seq_lens, 4) || (lse && !aligned(lse, 4)) || (err_flag && !aligned(err_flag, 4)))
    return PA_ERR_INVALID_ARG;
  if (workspace && !aligned(workspace, 256)) return PA_ERR_INVALID_ARG;
  if (Hq / Hkv > pa::decode_max_group(d, true)) return PA_ERR_UNSUPPORTED;
  const pa::DecodePlan p = pa::plan_decode(B, Hq, Hkv, d, max_blocks_per_seq, block_size, window,
                                           num_splits, num_splits > 0 ? 0 : sm_count(), false,
                                           true);
  if (p.smem > 227 * 1024) return PA_ERR_UNSUPPORTED;
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
  a.wait_ns = pa::role_wait_limit_ns();
  CUtensorMap km, vm;
  if (!encode_pool_u8(&km, k_cache, d, Hkv, block_size, num_blocks, p.hg) ||
      !encode_pool_u8(&vm, v_cache, d, Hkv, block_size, num_blocks, p.hg))
    return PA_ERR_CUDA;
  const cudaError_t e = pa::launch_decode_fp8(a, p, km, vm, k_scale, v_scale,
                                              static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"
