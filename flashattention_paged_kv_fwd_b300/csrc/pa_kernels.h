// Internal launcher interface between the C ABI (capi.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pa {

// Give-up limit (ns) of the waits between the roles of the prefill and decode
// kernels: 2 s, unless a test shortened it (pa_testing_set_wait_limit_ns).
// Waits for copies and MMAs already in flight keep their own limits.
unsigned long long role_wait_limit_ns();

// ------------------------------------------------------------------ append
cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int32_t* table, int max_blocks, const int32_t* seq_lens,
                             const int32_t* cu_new, int n_tok, int n_seq, int row_bytes,
                             int block_size, int num_blocks, int32_t* err, cudaStream_t s);

// ------------------------------------------------------------- block copy
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* src,
                               const int32_t* dst, int n_pairs, long long block_bytes,
                               int num_blocks, int32_t* err, cudaStream_t s);

// ------------------------------------------------------------------ decode
// How one decode call is cut into CTAs. Each sequence's visible blocks
// [first, last] are cut into ranges of `chunk` blocks; range s of sequence b
// is one CTA (for each group of `hg` KV heads). Sequences with more than one
// range write normalised partials (o_s, lse_s) to the workspace and a merge
// kernel combines them.
struct DecodePlan {
  int chunk;       // blocks per range
  int num_splits;  // ranges per sequence at most (grid.x)
  int hg;          // KV heads per CTA
  int head_chunks; // Hkv / hg (grid.y)
  int mt;          // 16-row MMA tiles per KV head (ceil(G / 16))
  int stages;      // pipeline depth (pages in flight per CTA)
  int threads;
  size_t smem;
  size_t workspace;  // bytes of partial outputs, 0 when num_splits == 1
};

DecodePlan plan_decode(int B, int Hq, int Hkv, int d, int max_blocks, int block_size, int window,
                       int num_splits_req, int sm_count, bool f32, bool fp8 = false);

// Largest Hq / Hkv the bf16 (or FP8) decode kernel serves: its consumer warps
// per CTA times the query heads one warp takes (16 as MMA rows for bf16, 8 as
// MMA columns for FP8).
int decode_max_group(int d, bool fp8);

struct DecodeArgs {
  const void* q;
  void* o;
  float* lse;
  const void* k_cache;
  const void* v_cache;
  const int32_t* table;
  const int32_t* seq_lens;
  float* ws_o;    // [B, Hq, num_splits, d]
  float* ws_lse;  // [B, Hq, num_splits]
  int32_t* err;
  int max_blocks, num_blocks, B, Hq, Hkv, d, window;
  float scale_log2;
  unsigned long long wait_ns;  // give-up limit of the pipeline waits (role_wait_limit_ns())
};

cudaError_t launch_decode_bf16(const DecodeArgs& a, const DecodePlan& p, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, cudaStream_t s);
cudaError_t launch_decode_f32(const DecodeArgs& a, const DecodePlan& p, cudaStream_t s);
// FP8 (E4M3) pools [num_blocks, 16, Hkv, d] of codes; kmap / vmap are uint8
// maps ordered (d, token, head, block) with d x 16 x hg x 1 boxes.
cudaError_t launch_decode_fp8(const DecodeArgs& a, const DecodePlan& p, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, const float* k_scale,
                              const float* v_scale, cudaStream_t s);
// Quantise new bf16 rows with their heads' scales into FP8 pools.
cudaError_t launch_kv_append_fp8(const void* k_new, const void* v_new, void* k_cache,
                                 void* v_cache, const float* k_scale, const float* v_scale,
                                 const int32_t* table, int max_blocks, const int32_t* seq_lens,
                                 const int32_t* cu_new, int n_tok, int n_seq, int Hkv, int d,
                                 int block_size, int num_blocks, int32_t* err, cudaStream_t s);

// ----------------------------------------------------------------- prefill
struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  const int32_t* cu_seqlens;  // nullptr => fixed length N
  int32_t* err;
  int B, Hq, Hkv, N, T, d, max_seqlen, causal, window;
  float scale_log2;
  int pair_heads;  // bf16 path: a work unit pairs two query heads (else two row tiles)
  int n_units;     // bf16 path: work units in the launch
  int compact;     // bf16 path: build the sorted on-chip work list (packed sequences)
  // paged keys (prefill into a non-empty cache): keys and values of sequence b
  // are its first seq_lens_k[b] tokens in the pools [num_blocks, 16, Hkv, d]
  // addressed through table[b][*]; query row i of its Lq rows sits at
  // position seq_lens_k[b] - Lq + i. k / v above are then the pools.
  const int32_t* table;       // nullptr => contiguous keys (rows of k / v)
  const int32_t* seq_lens_k;
  int max_blocks, num_blocks;
  unsigned long long wait_ns;  // give-up limit of the pipeline waits (role_wait_limit_ns())
};

// Work units of the bf16 prefill (two 128-row query tiles each).
long long prefill_units(int B, int Hq, int Hkv, int max_seqlen, bool* pair_heads);

// kmap / vmap: 3-D maps over [T, Hkv, d] rows, or -- with a.table -- 4-D maps
// over the pools ordered (d, token, head, block) with 64 x 16 x 1 x 1 boxes.
cudaError_t launch_prefill_bf16(const PrefillArgs& a, const CUtensorMap& qmap,
                                const CUtensorMap& kmap, const CUtensorMap& vmap, int num_sms,
                                cudaStream_t s);
cudaError_t launch_prefill_f32(const PrefillArgs& a, cudaStream_t s);

size_t prefill_bf16_smem(int d);

}  // namespace pa
