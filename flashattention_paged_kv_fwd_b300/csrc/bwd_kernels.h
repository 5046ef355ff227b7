// Internal launcher interface of the attention backward pass (capi_bwd.cu ->
// prefill_bwd.cu).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pa {

struct BackwardArgs {
  const void* q;     // [T, Hq, d] bf16
  const void* k;     // [T, Hkv, d]
  const void* v;     // [T, Hkv, d]
  const void* o;     // [T, Hq, d]   forward output
  const void* dout;  // [T, Hq, d]   dL/dO
  const float* lse;  // [Hq, T]      forward log-sum-exp (natural log)
  void* dq;          // [T, Hq, d]
  void* dk;          // [T, Hkv, d]
  void* dv;          // [T, Hkv, d]
  float* dq_acc;     // workspace [T, Hq, d] fp32, zeroed before the main kernel
  float* dvec;       // workspace [Hq, T]: D_i = sum_c dO_ic O_ic
  const int32_t* cu_seqlens;  // nullptr => fixed length N
  int32_t* err;
  int B, Hq, Hkv, N, T, d, max_seqlen, causal, window;
  float scale;       // softmax scale (natural units)
  float scale_log2;  // scale * log2(e)
  int n_units;       // key tiles x KV heads x sequences enumerated by the main kernel
  unsigned long long wait_ns;  // give-up limit of the pipeline waits (role_wait_limit_ns())
};

// Give-up limit of the kernels' pipeline waits (2 s unless a test shortened it).
unsigned long long role_wait_limit_ns();

// Bytes of workspace the backward pass needs for T packed tokens.
size_t backward_workspace_bytes(long long T, int Hq, int d);

// D = rowsum(dO * O), dQ accumulation (tensor cores), dQ conversion. qmap,
// kmap, vmap, domap: 64-element x 128-row, 128-byte-swizzled bf16 boxes over
// q, k, v, dout; dqmap: 32-element (fp32) x 1-head x 32-row, 128-byte-swizzled
// boxes over the fp32 buffer [T, Hq, d] (the reduce-add target).
cudaError_t launch_prefill_backward_bf16(const BackwardArgs& a, const CUtensorMap& qmap,
                                         const CUtensorMap& kmap, const CUtensorMap& vmap,
                                         const CUtensorMap& domap, const CUtensorMap& dqmap,
                                         int num_sms, cudaStream_t s);

}  // namespace pa
