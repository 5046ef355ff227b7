// Internal launcher interface of multi-head latent attention (MLA) decode
// (capi.cu -> mla_decode.cu).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pa {

// Latent rows: d_c = 512 latent numbers followed by d_R = 64 rope numbers.
constexpr int kMlaDc = 512;
constexpr int kMlaDr = 64;
constexpr int kMlaRow = kMlaDc + kMlaDr;

// How one MLA decode call is cut into CTAs: CTA (s, hc, b) attends query
// heads [hc * 16 * ng, ...) of sequence b over blocks [s * chunk, ...) of its
// visible range. Sequences with more than one range write normalised
// partials (o_s, lse_s) to the workspace and a merge kernel combines them.
struct MlaPlan {
  int ng;           // groups of 16 query heads per CTA (1 or 2)
  int head_chunks;  // ceil(H / (16 * ng)) (grid.y)
  int chunk;        // blocks per range
  int num_splits;   // ranges per sequence at most (grid.x)
  int stages;       // two-block steps in flight per CTA
  int threads;
  size_t smem;
  size_t workspace;  // bytes of partial outputs, 0 when num_splits == 1
};

MlaPlan plan_mla_decode(int B, int H, int max_blocks, int num_splits_req, int sm_count);

struct MlaArgs {
  const void* q;      // [B, H, 576] bf16: absorbed content query, then the rope query
  void* o;            // [B, H, 512] bf16: sum_j p_ij c_j
  float* lse;         // [H, B] or nullptr
  const int32_t* table;
  const int32_t* seq_lens;
  float* ws_o;        // [B, H, num_splits, 512]
  float* ws_lse;      // [B, H, num_splits]
  int32_t* err;
  int max_blocks, num_blocks, B, H;
  float scale_log2;
  unsigned long long wait_ns;  // give-up limit of the pipeline waits (role_wait_limit_ns())
};

// Give-up limit of the kernels' pipeline waits (2 s unless a test shortened it).
unsigned long long role_wait_limit_ns();

// `cmap`: the pool [num_blocks, 16, 576] described as (64 elements, 16
// tokens, 9 panels, blocks), one 128-byte-swizzled box per block.
cudaError_t launch_mla_decode_bf16(const MlaArgs& a, const MlaPlan& p, const CUtensorMap& cmap,
                                   cudaStream_t s);

}  // namespace pa
