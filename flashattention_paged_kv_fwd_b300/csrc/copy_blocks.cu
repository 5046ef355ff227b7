// copy_blocks: whole-block copies inside the paged pools, for copy-on-write.
//
// "Module 09: Efficient Attention", section "Sharing Blocks: Copy-on-Write":
// sequences that share a prefix point at the same physical blocks, a
// per-block reference count tracks the sharers, and a sharer that is about
// to write into a shared block first gets its own copy of that one block.
// The bookkeeping is host-side; this kernel does the copies of a whole batch
// of (source, destination) block pairs in one launch. A block of a pool is
// block_size * Hkv * d * elem contiguous bytes, moved as 16-byte vectors with
// several in flight per thread. Bit-exact (no arithmetic on values).
#include <cstdint>
#include <cuda_runtime.h>

#include "pa_kernels.h"
#include "pa_ptx.cuh"

namespace pa {

namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;  // 16-byte vectors in flight per thread per pool

__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                   const int32_t* __restrict__ src, const int32_t* __restrict__ dst, int n_pairs,
                   int block_vecs, int num_blocks, int32_t* err) {
  // CTA (x, y): pair y (+ a grid-stride over pairs), slice x of the block
  const int slice = kCopyThreads * kCopyUnroll;
  for (int p = blockIdx.y; p < n_pairs; p += gridDim.y) {
    const int s = src[p], d = dst[p];
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
      if (threadIdx.x == 0 && blockIdx.x == 0) raise_err(err, kDevErrBadBlock);
      continue;
    }
    if (s == d) continue;
    const int64_t so = static_cast<int64_t>(s) * block_vecs;
    const int64_t dof = static_cast<int64_t>(d) * block_vecs;
    for (int i0 = blockIdx.x * slice; i0 < block_vecs; i0 += gridDim.x * slice) {
      uint4 kv[kCopyUnroll], vv[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int i = i0 + u * kCopyThreads + threadIdx.x;
        if (i < block_vecs) {
          kv[u] = __ldg(k_cache + so + i);
          vv[u] = __ldg(v_cache + so + i);
        }
      }
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int i = i0 + u * kCopyThreads + threadIdx.x;
        if (i < block_vecs) {
          k_cache[dof + i] = kv[u];
          v_cache[dof + i] = vv[u];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* src,
                               const int32_t* dst, int n_pairs, long long block_bytes,
                               int num_blocks, int32_t* err, cudaStream_t s) {
  if (n_pairs == 0) return cudaSuccess;
  const long long vecs = block_bytes / 16;
  const long long slice = kCopyThreads * kCopyUnroll;
  const unsigned gx = static_cast<unsigned>((vecs + slice - 1) / slice);
  const unsigned gy = static_cast<unsigned>(n_pairs < 65535 ? n_pairs : 65535);
  copy_blocks_kernel<<<dim3(gx, gy), kCopyThreads, 0, s>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), src, dst, n_pairs,
      static_cast<int>(vecs), num_blocks, err);
  return cudaGetLastError();
}

}  // namespace pa
