// Host-side helpers shared by the C ABI translation units: argument checks,
// TMA descriptor encoding (through the driver entry point, so the library
// links only the CUDA runtime) and the SM count.
#pragma once

#include <cmath>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pagedattn.h"

namespace pa {
namespace host {
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

// FP8 pool [num_blocks, block_size, heads, d] of 1-byte codes, dimensions in
// the order (d, token, head, block), boxes of d x block_size x box_heads x 1
// landing as [box_heads][block_size][d] bytes with the 16-byte pieces of each
// row swizzled: the 128-byte pattern for d = 128 (piece p of row r at p ^ (r % 8)),
// the 64-byte one for d = 64 (at p ^ ((r / 2) % 4)).
bool encode_pool_u8(CUtensorMap* m, const void* ptr, int d, int heads, int block_size,
                    int num_blocks, int box_heads) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(block_size),
                              static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(heads) * d,
                                 static_cast<cuuint64_t>(d),
                                 static_cast<cuuint64_t>(block_size) * heads * d};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(d), static_cast<cuuint32_t>(block_size),
                             static_cast<cuuint32_t>(box_heads), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

double softmax_scale(float scale, int d) {
  return scale > 0.f ? static_cast<double>(scale) : 1.0 / std::sqrt(static_cast<double>(d));
}

float scale_log2(float scale, int d) {
  return static_cast<float>(softmax_scale(scale, d) * 1.4426950408889634074);  // * log2(e)
}

}  // namespace
}  // namespace host
}  // namespace pa
