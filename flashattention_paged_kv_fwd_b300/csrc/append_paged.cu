// kv_append_paged: scatter new tokens' K/V rows into the paged pools.
//
// "Module 09: Efficient Attention", section "Code: A Paged KV Cache from
// Scratch": the token at logical position t of a sequence is stored at
// (block_table[t // block_size], t % block_size) of a pool shaped
// (num_blocks, block_size, num_kv_heads, head_dim). One token's row for all
// KV heads is contiguous both in the input ([T_new, Hkv, d]) and in the pool,
// so each token is one contiguous copy of Hkv*d*elem bytes, moved as 16-byte
// vectors by one warp. Bit-exact by construction (no arithmetic on values).
// With no value tensor (v_new == nullptr) it appends the rows of a single
// pool, such as the latent rows of an MLA cache.
#include <cstdint>
#include <cuda_runtime.h>

#include "pa_ptx.cuh"
#include "pa_kernels.h"

namespace pa {

namespace {

constexpr int kAppendWarps = 8;       // tokens per CTA
constexpr int kMaxCuInSmem = 4096;    // sequences whose offsets are staged in smem
constexpr int kUnroll = 4;            // 16-byte vectors in flight per lane per tensor

__device__ __forceinline__ int find_sequence(const int32_t* cu, int n_seq, int t) {
  // largest b with cu[b] <= t (cu is non-decreasing; empty sequences skipped)
  int lo = 0, hi = n_seq - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kAppendWarps * 32)
kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                 uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                 const int32_t* __restrict__ table, int max_blocks,
                 const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_new,
                 int n_seq, int n_tok, int row_vecs, int block_size, int num_blocks,
                 int32_t* err) {
  __shared__ int32_t cu_s[kMaxCuInSmem + 1];
  const bool staged = cu_new != nullptr && n_seq <= kMaxCuInSmem;
  if (staged) {
    for (int i = threadIdx.x; i <= n_seq; i += blockDim.x) cu_s[i] = cu_new[i];
    __syncthreads();
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kAppendWarps + warp;
  if (t >= n_tok) return;

  int b, first;
  if (cu_new == nullptr) {
    b = t;
    first = t;
  } else {
    const int32_t* cu = staged ? cu_s : cu_new;
    // a token outside [cu[0], cu[n_seq]) belongs to no sequence: the offsets
    // disagree with the token count, and guessing a sequence would overwrite
    // another token's slot
    if (t < cu[0] || t >= cu[n_seq]) {
      if (lane == 0) raise_err(err, kDevErrBadPosition);
      return;
    }
    b = find_sequence(cu, n_seq, t);
    first = cu[b];
  }
  const int pos = seq_lens[b] + (t - first);
  const int lblk = pos / block_size;
  if (pos < 0 || lblk >= max_blocks) {
    if (lane == 0) raise_err(err, kDevErrBadPosition);
    return;
  }
  const int blk = table[static_cast<int64_t>(b) * max_blocks + lblk];
  if (blk < 0 || blk >= num_blocks) {
    if (lane == 0) raise_err(err, kDevErrBadBlock);
    return;
  }
  const int64_t src = static_cast<int64_t>(t) * row_vecs;
  const int64_t dst = (static_cast<int64_t>(blk) * block_size + pos % block_size) * row_vecs;
  for (int i0 = 0; i0 < row_vecs; i0 += 32 * kUnroll) {
    uint4 kv[kUnroll], vv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u * 32 + lane;
      if (i < row_vecs) {
        kv[u] = __ldg(k_new + src + i);
        if (v_new) vv[u] = __ldg(v_new + src + i);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u * 32 + lane;
      if (i < row_vecs) {
        k_cache[dst + i] = kv[u];
        if (v_new) v_cache[dst + i] = vv[u];
      }
    }
  }
}

// FP8 cache: each new bf16 row is quantised on the way in. Element e of the
// row belongs to KV head e / d; y = x / scale[head] with IEEE division, then
// the nearest E4M3 code (ties to even, saturating to +-448). One warp per
// token; a lane handles 8 elements (16 bytes in, 8 bytes out) at a time.
__global__ void __launch_bounds__(kAppendWarps * 32)
kv_append_fp8_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     uint2* __restrict__ k_cache, uint2* __restrict__ v_cache,
                     const float* __restrict__ k_scale, const float* __restrict__ v_scale,
                     const int32_t* __restrict__ table, int max_blocks,
                     const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_new,
                     int n_seq, int n_tok, int row_vecs, int d, int block_size, int num_blocks,
                     int32_t* err) {
  __shared__ int32_t cu_s[kMaxCuInSmem + 1];
  const bool staged = cu_new != nullptr && n_seq <= kMaxCuInSmem;
  if (staged) {
    for (int i = threadIdx.x; i <= n_seq; i += blockDim.x) cu_s[i] = cu_new[i];
    __syncthreads();
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kAppendWarps + warp;
  if (t >= n_tok) return;
  int b, first;
  if (cu_new == nullptr) {
    b = t;
    first = t;
  } else {
    const int32_t* cu = staged ? cu_s : cu_new;
    if (t < cu[0] || t >= cu[n_seq]) {
      if (lane == 0) raise_err(err, kDevErrBadPosition);
      return;
    }
    b = find_sequence(cu, n_seq, t);
    first = cu[b];
  }
  const int pos = seq_lens[b] + (t - first);
  const int lblk = pos / block_size;
  if (pos < 0 || lblk >= max_blocks) {
    if (lane == 0) raise_err(err, kDevErrBadPosition);
    return;
  }
  const int blk = table[static_cast<int64_t>(b) * max_blocks + lblk];
  if (blk < 0 || blk >= num_blocks) {
    if (lane == 0) raise_err(err, kDevErrBadBlock);
    return;
  }
  const int64_t src = static_cast<int64_t>(t) * row_vecs;
  const int64_t dst = (static_cast<int64_t>(blk) * block_size + pos % block_size) * row_vecs;
  auto quant = [&](const uint4& x, float sc) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t out[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float y0 = __fdiv_rn(__uint_as_float(w[2 * e] << 16), sc);
      const float y1 = __fdiv_rn(__uint_as_float(w[2 * e] & 0xFFFF0000u), sc);
      const float y2 = __fdiv_rn(__uint_as_float(w[2 * e + 1] << 16), sc);
      const float y3 = __fdiv_rn(__uint_as_float(w[2 * e + 1] & 0xFFFF0000u), sc);
      out[e] = static_cast<uint32_t>(f32x2_to_e4m3x2(y0, y1)) |
               (static_cast<uint32_t>(f32x2_to_e4m3x2(y2, y3)) << 16);
    }
    return make_uint2(out[0], out[1]);
  };
  for (int i = lane; i < row_vecs; i += 32) {
    const int head = (i * 8) / d;
    const uint4 kx = __ldg(k_new + src + i);
    const uint4 vx = __ldg(v_new + src + i);
    k_cache[dst + i] = quant(kx, k_scale[head]);
    v_cache[dst + i] = quant(vx, v_scale[head]);
  }
}

}  // namespace

cudaError_t launch_kv_append_fp8(const void* k_new, const void* v_new, void* k_cache,
                                 void* v_cache, const float* k_scale, const float* v_scale,
                                 const int32_t* table, int max_blocks, const int32_t* seq_lens,
                                 const int32_t* cu_new, int n_tok, int n_seq, int Hkv, int d,
                                 int block_size, int num_blocks, int32_t* err, cudaStream_t s) {
  if (n_tok == 0) return cudaSuccess;
  const int grid = (n_tok + kAppendWarps - 1) / kAppendWarps;
  kv_append_fp8_kernel<<<grid, kAppendWarps * 32, 0, s>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      static_cast<uint2*>(k_cache), static_cast<uint2*>(v_cache), k_scale, v_scale, table,
      max_blocks, seq_lens, cu_new, n_seq, n_tok, Hkv * d / 8, d, block_size, num_blocks, err);
  return cudaGetLastError();
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int32_t* table, int max_blocks, const int32_t* seq_lens,
                             const int32_t* cu_new, int n_tok, int n_seq, int row_bytes,
                             int block_size, int num_blocks, int32_t* err, cudaStream_t s) {
  if (n_tok == 0) return cudaSuccess;
  const int grid = (n_tok + kAppendWarps - 1) / kAppendWarps;
  kv_append_kernel<<<grid, kAppendWarps * 32, 0, s>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), table, max_blocks, seq_lens,
      cu_new, n_seq, n_tok, row_bytes / 16, block_size, num_blocks, err);
  return cudaGetLastError();
}

}  // namespace pa
