/*
 * pagedattn.h -- C ABI of libpagedattn.so: exact scaled-dot-product attention
 * computed FlashAttention-style on one B300 (sm_103a), over contiguous
 * (prefill) and paged (decode) key/value storage.
 *
 * The operation. For query row i of a sequence with Lq queries and Lk keys,
 * and query head h:
 *
 *   o[i,h,:] = sum_j softmax_j( scale * q[i,h,:] . k[j,g,:] ) v[j,g,:]
 *   lse[h,i] = ln sum_j exp( scale * q[i,h,:] . k[j,g,:] )
 *
 * over the visible keys j, with g = floor(h / (Hq / Hkv)) and scale defaulting
 * to 1/sqrt(d). Sources: "Module 09: Efficient Attention" (learnllm notebook),
 * section "The Math: Sharing Keys and Values" (the formula, n_rep and the
 * query-to-KV-head mapping; MHA, GQA and MQA are Hkv = Hq, 1 < Hkv < Hq and
 * Hkv = 1). The score matrix is never written to memory: keys are streamed in
 * tiles with a running (max, sum) that is rescaled whenever the max grows
 * ("Cache KV, atención flash y optimización de la inferencia", section "La
 * atención de flash el truco de la balsa"; "Ли Хунъи, «Машинное обучение»
 * 2026 ...", lecture "Ускоряем генерацию, часть 1: FlashAttention").
 *
 * Visibility. Query row i sits at absolute position p_i = Lk - Lq + i (the
 * causal mask is aligned to the bottom-right corner: "Генерация и KV-кэш",
 * section "Три ловушки, на которых спотыкаются все", trap 2). Causal: j <= p_i.
 * Sliding window W > 0 (causal only): additionally j > p_i - W, so the
 * diagonal counts toward W ("Module 09: Efficient Attention", section
 * "Attention Mask Gallery", sliding_window_mask(6, window=3)).
 *
 * LSE is the natural logarithm of the softmax denominator (not given on the
 * pages; see the design notes). A query with no visible key gets o = 0 and
 * lse = -inf.
 *
 * Conventions shared by every call:
 *  - All pointers are DEVICE pointers except where stated; all tensors are
 *    dense and row-major in the index order given; the caller owns every
 *    buffer. The library never allocates device memory. Its state between
 *    calls is host-side caches (driver entry points, the SM count, kernel
 *    attribute flags) plus one device-side array: the fixed scratch of
 *    pa_attn_decode_paged_noalloc (PA_NOALLOC_SCRATCH_BYTES per GPU, part of
 *    the loaded module), which only that entry point uses.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy stream).
 *  - Return value: PA_OK, or a host-detected error (nothing is launched).
 *  - err_flag (optional, may be NULL): an int32 in device memory that kernels
 *    OR PA_DEV_* bits into when they meet bad data (a block id outside the
 *    pool, a position beyond a block table, a bounded wait that gave up).
 *    Outputs are undefined where a bit was raised. Kernels never trap; the
 *    caller reads the flag after synchronising. The library never clears it.
 *  - dtype PA_BF16: bf16 inputs and outputs, fp32 accumulation. PA_F32: fp32
 *    inputs and outputs (a CUDA-core correctness path), fp32 accumulation.
 *  - Head dimension d must be 64 or 128 (MLA: latent rows of d_c = 512 plus
 *    d_rope = 64).
 *
 * Beyond the forward pass the library has the backward pass of the prefill
 * (pa_attn_prefill_backward), chunked prefill into a paged cache
 * (pa_attn_prefill_paged), block copies for copy-on-write (pa_copy_blocks)
 * and multi-head latent attention decode over a paged latent cache
 * (pa_mla_decode_paged, pa_mla_append_paged).
 */
#ifndef PAGEDATTN_H_
#define PAGEDATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PA_BF16 = 0, PA_F32 = 1 } pa_dtype;

enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, Hkv not dividing Hq */
  PA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. window without causal) */
  PA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (launch, encode) */
  PA_ERR_WORKSPACE = 4    /* workspace missing or smaller than required */
};

enum {
  PA_DEV_BAD_BLOCK = 1,    /* a block-table entry outside [0, num_blocks) */
  PA_DEV_BAD_POSITION = 2, /* a token position beyond the sequence's table */
  PA_DEV_TIMEOUT = 4,      /* a bounded wait gave up */
  PA_DEV_INTERNAL = 8      /* a kernel found its launch state unusable (e.g. a misaligned
                              shared-memory base); it computed nothing */
};

/* Short description of a status code (static string). */
PA_API const char* pa_status_str(int status);

/*
 * attn_prefill -- causal / sliding-window / full attention of each sequence's
 * queries over its own keys (Lq = Lk per sequence), GQA through Hkv.
 * "Cache KV, atención flash ...", section "La atención de flash el truco de la
 * balsa" (tile loop over K/V with the output written once per query tile);
 * "Генерация и KV-кэш", section "Две фазы генерации: prefill и decode".
 *
 *  q    [T, Hq, d]   queries, token-major (T = total tokens of the batch)
 *  k, v [T, Hkv, d]  keys / values, token-major
 *  o    [T, Hq, d]   output (same dtype as q); must not alias q, k or v
 *  lse  [Hq, T]      float32 natural-log LSE per (head, token); may be NULL
 *  B    number of sequences
 *  N    tokens per sequence when cu_seqlens is NULL (then T = B*N); when
 *       cu_seqlens is given, N is the total packed token count T
 *  cu_seqlens  NULL, or int32[B+1] device array of packed sequence offsets
 *       (cu_seqlens[0] = 0, non-decreasing, cu_seqlens[B] = T); zero-length
 *       sequences are allowed
 *  max_seqlen  with cu_seqlens: an upper bound on every sequence's length
 *  causal      1 = causal, 0 = every query sees every key of its sequence
 *  window      <= 0: none; > 0: sliding window W (requires causal)
 *  scale       <= 0: 1/sqrt(d)
 * Alignment: q, k, v 16-byte aligned; o 32-byte aligned for bf16 (16 for
 * f32); lse 4-byte aligned.
 */
PA_API int pa_attn_prefill(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int Hq, int Hkv, int N, int d, const int32_t* cu_seqlens, int max_seqlen,
                    int causal, int window, float scale, pa_dtype dtype, int32_t* err_flag,
                    void* stream);

/*
 * attn_prefill_paged -- a chunk of new queries per sequence attending to the
 * sequence's whole paged cache: chunked prefill, or a prompt whose prefix is
 * already cached. "Генерация и KV-кэш", section "Три ловушки, на которых
 * спотыкаются все", trap 2 (queries that continue a cache are aligned to the
 * bottom-right corner of the score matrix); "Module 09: Efficient Attention",
 * sections "Code: A Paged KV Cache from Scratch" and "The Block Table" (key
 * t of a sequence is (block_table[t / 16], t % 16) of the pools).
 * Sequence b holds seq_lens[b] keys in the cache; its Lq_b =
 * cu_seqlens_q[b+1] - cu_seqlens_q[b] queries are the LAST Lq_b of those
 * positions (append the chunk's keys and values with pa_kv_append_paged
 * first), so query row i sits at position p_i = seq_lens[b] - Lq_b + i and
 * the visibility rules of attn_prefill apply with that p_i.
 *
 *  q     [total_q, Hq, d]   packed queries (bf16), token-major
 *  k_cache, v_cache [num_blocks, 16, Hkv, d] pools (bf16), read only
 *  block_table int32 [B, max_blocks_per_seq]; entries past a sequence's
 *        last block are never read (any value)
 *  seq_lens   int32 [B]: keys of each sequence, the chunk's own included
 *        (>= its Lq; <= max_blocks_per_seq * 16)
 *  cu_seqlens_q int32 [B+1]: packed offsets of the queries; total_q =
 *        cu_seqlens_q[B]; max_seqlen_q bounds every Lq_b
 *  o     [total_q, Hq, d] output (bf16); lse [Hq, total_q] float32 or NULL
 *  block_size must be 16; dtype must be PA_BF16 (PA_ERR_UNSUPPORTED
 *  otherwise). causal / window / scale as in attn_prefill.
 * Slots of a block past a sequence's keys may hold anything (even NaN): they
 * are never used. A block id outside [0, num_blocks) raises PA_DEV_BAD_BLOCK
 * and that block is skipped. Alignment: q, pools 16-byte aligned; o 32-byte
 * aligned; int32 arrays and lse 4-byte aligned.
 */
PA_API int pa_attn_prefill_paged(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_table, int max_blocks_per_seq,
                                 const int32_t* seq_lens, const int32_t* cu_seqlens_q,
                                 int total_q, int max_seqlen_q, void* o, float* lse, int B,
                                 int Hq, int Hkv, int d, int block_size, int num_blocks,
                                 int causal, int window, float scale, pa_dtype dtype,
                                 int32_t* err_flag, void* stream);

/*
 * attn_prefill_backward -- gradients of attn_prefill's output: given dO =
 * dL/dO, returns dQ, dK, dV. "Cache KV, atención flash y optimización de la
 * inferencia", section "La atención de flash el truco de la balsa": the
 * backward pass recomputes the forward values (the scores and P) from Q, K
 * and the saved per-row LSE instead of storing the attention matrix. The
 * gradients are the chain rule through O = softmax(S) V, S = scale Q K^T:
 *   P = exp(S - lse), dV = P^T dO, dP = dO V^T, D_i = sum_c dO_ic O_ic,
 *   dS = P (dP - D), dQ = scale dS K, dK = scale dS^T Q,
 * with masked (invisible) pairs contributing nothing; dK and dV of a KV head
 * are summed over the query heads that read it.
 *
 *  q, o, dout [T, Hq, d] bf16: the forward call's queries and output, and
 *             the upstream gradient
 *  k, v       [T, Hkv, d] bf16
 *  lse        [Hq, T] float32: the forward call's LSE (natural log)
 *  dq [T, Hq, d], dk, dv [T, Hkv, d] bf16 outputs (must not alias inputs).
 *             Rows of dq outside every sequence are set to zero; such rows
 *             of dk / dv are not written.
 *  B, N, cu_seqlens, max_seqlen, causal, window, scale: as in attn_prefill,
 *             and the same values the forward call used
 *  workspace  device buffer of >= pa_attn_prefill_backward_workspace_bytes
 *             bytes, 256-byte aligned, owned by the caller, unused after the
 *             stream reaches the end of this call (fp32 dQ accumulator and
 *             the D vector)
 * dtype must be PA_BF16 (PA_ERR_UNSUPPORTED otherwise); d is 64 or 128.
 * Alignment: q, k, v, o, dout, dq 16-byte aligned; dk, dv 32-byte aligned;
 * lse 4-byte aligned. Errors: PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED /
 * PA_ERR_WORKSPACE before any CUDA call; PA_DEV_TIMEOUT in err_flag if a
 * bounded wait of the main kernel gave up.
 */
PA_API size_t pa_attn_prefill_backward_workspace_bytes(int total_tokens, int Hq, int d);

PA_API int pa_attn_prefill_backward(const void* q, const void* k, const void* v, const void* o,
                                    const void* dout, const float* lse, void* dq, void* dk,
                                    void* dv, int B, int Hq, int Hkv, int N, int d,
                                    const int32_t* cu_seqlens, int max_seqlen, int causal,
                                    int window, float scale, void* workspace,
                                    size_t workspace_bytes, pa_dtype dtype, int32_t* err_flag,
                                    void* stream);

/*
 * mla_decode_paged -- multi-head latent attention decode: one query per
 * sequence attends, in every head, to the sequence's cached latent rows.
 * "Module 09: Efficient Attention", section "Multi-head Latent Attention: A
 * Different Lever": the cache keeps per token one latent c_j (d_c numbers)
 * and one shared rope key kR_j (d_R numbers), no head axis; head i's key is
 * [W^UK_i c_j ; kR_j] and its value W^UV_i c_j; by absorption ("Why RoPE Has
 * To Be Decoupled") the query attends the latent directly and the weighted
 * sum is formed in the latent space ("Ли Хунъи ... 2026", KV-compression
 * lever 2). With the absorbed query q_i = [W^UK_i^T q^C_i ; q^R_i] supplied
 * by the caller, this computes
 *   s_ij = scale * q_i . r_j,   o_i = sum_j softmax_j(s)_ij r_j[0:d_c],
 * where r_j = [c_j ; kR_j] is cached row j; the caller up-projects o_i with
 * W^UV_i.
 *
 *  q      [B, H, d_c + d_rope] bf16: absorbed content query, then rope query
 *  cache  [num_blocks, block_size, d_c + d_rope] bf16 rows [c_j ; kR_j], read
 *         only; token t of sequence b at (block_table[b][t / 16], t % 16)
 *  block_table int32 [B, max_blocks_per_seq]; seq_lens int32 [B] (keys per
 *         sequence, the new token's own row included)
 *  o      [B, H, d_c] bf16 output; lse [H, B] float32 (natural log) or NULL
 *  scale  > 0 (1/sqrt(d_head + d_rope) for the model's head dim), required
 *  num_splits 0 = automatic; workspace as in attn_decode_paged, sized by
 *         pa_mla_decode_workspace_bytes (0 = none needed)
 * Supported: bf16, d_c = 512, d_rope = 64, block_size 16 (PA_ERR_UNSUPPORTED
 * otherwise); any H >= 1. A block id outside [0, num_blocks) raises
 * PA_DEV_BAD_BLOCK and its tokens are skipped; a sequence with no key gets
 * o = 0 and lse = -inf. Alignment: q, cache, o 16-byte aligned; int32 arrays
 * and lse 4-byte aligned; workspace 256-byte aligned.
 */
PA_API size_t pa_mla_decode_workspace_bytes(int B, int H, int d_c, int d_rope,
                                            int max_blocks_per_seq, int block_size,
                                            int num_splits);

PA_API int pa_mla_decode_paged(const void* q, const void* cache, const int32_t* block_table,
                               int max_blocks_per_seq, const int32_t* seq_lens, void* o,
                               float* lse, int B, int H, int d_c, int d_rope, int block_size,
                               int num_blocks, float scale, int num_splits, void* workspace,
                               size_t workspace_bytes, pa_dtype dtype, int32_t* err_flag,
                               void* stream);

/*
 * mla_append_paged -- write new tokens' latent rows ([c ; kR], row_elems
 * numbers each) into an MLA cache [num_blocks, block_size, row_elems]: the
 * single-pool form of kv_append_paged (same table, seq_lens, cu_new and
 * error semantics; a byte copy). row_elems * element size must be a
 * multiple of 16; pointers 16-byte aligned, int32 arrays 4-byte aligned.
 */
PA_API int pa_mla_append_paged(const void* rows_new, void* cache, const int32_t* block_table,
                               int max_blocks_per_seq, const int32_t* seq_lens,
                               const int32_t* cu_new, int num_new_tokens, int B, int row_elems,
                               int block_size, int num_blocks, pa_dtype dtype,
                               int32_t* err_flag, void* stream);

/*
 * kv_append_paged -- write new tokens' keys and values into the paged pools.
 * "Module 09: Efficient Attention", section "Code: A Paged KV Cache from
 * Scratch": token t of a sequence lives at (block_table[t / block_size],
 * t % block_size) of a pool shaped (num_blocks, block_size, Hkv, d).
 * A pure copy: the pools receive the new rows bit for bit.
 *
 *  k_new, v_new  [T_new, Hkv, d]  rows to append, token-major
 *  k_cache, v_cache [num_blocks, block_size, Hkv, d]  pools, written in place
 *  block_table   int32 [B, max_blocks_per_seq]; entries past a sequence's
 *                last block are never read (any value)
 *  seq_lens      int32 [B]: tokens each sequence holds BEFORE this append;
 *                the library never modifies it (the caller advances it)
 *  cu_new        NULL (one new token per sequence, T_new = B) or int32[B+1]
 *                offsets of each sequence's new rows in k_new / v_new
 *  num_new_tokens  T_new (must equal cu_new[B] when cu_new is given)
 * The blocks a write lands in must already be claimed by the caller's
 * allocator; an entry outside [0, num_blocks) or a position beyond the table
 * raises a PA_DEV_* bit and that row is skipped.
 * Alignment: every pointer 16-byte aligned; Hkv*d*elem_size a multiple of 16.
 */
PA_API int pa_kv_append_paged(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                       const int32_t* block_table, int max_blocks_per_seq,
                       const int32_t* seq_lens, const int32_t* cu_new, int num_new_tokens,
                       int B, int Hkv, int d, int block_size, int num_blocks, pa_dtype dtype,
                       int32_t* err_flag, void* stream);

/*
 * copy_blocks -- copy whole blocks of both pools (keys and values), for
 * copy-on-write of shared prefix blocks. "Module 09: Efficient Attention",
 * section "Sharing Blocks: Copy-on-Write": sequences sharing a prefix point
 * at the same physical blocks, with a per-block reference count; before a
 * sharer writes into a shared block, that one block is copied and the
 * sharer's table is pointed at the copy. The reference counting and table
 * updates are the caller's (host) work; this call does the copies.
 *
 *  k_cache, v_cache [num_blocks, block_size, Hkv, d] pools, written in place
 *  src_blocks, dst_blocks int32 [num_pairs] (device): block src_blocks[i] is
 *        copied over block dst_blocks[i] in both pools, bit for bit
 * Destinations must be distinct and no destination may be the source of
 * another pair in the same call (the copies run concurrently). A pair with
 * an id outside [0, num_blocks) raises PA_DEV_BAD_BLOCK and is skipped; a
 * pair with src == dst is a no-op. Alignment: pools 16-byte aligned, the id
 * arrays 4-byte aligned.
 */
PA_API int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* src_blocks,
                          const int32_t* dst_blocks, int num_pairs, int block_size, int Hkv,
                          int d, int num_blocks, pa_dtype dtype, int32_t* err_flag,
                          void* stream);

/*
 * attn_decode_paged -- one query per sequence, attending over every cached
 * key of that sequence through its block table (the query's own key
 * included; no causal mask is needed), optionally limited to the last
 * `window` keys. "Генерация и KV-кэш", section "KV-кэш для одной головы на
 * NumPy" (decode_step); "Module 09: Efficient Attention", section "The Block
 * Table" (gather by walking the table).
 *
 * Long contexts are split into ranges of blocks processed in parallel; each
 * range yields a normalised partial output and its LSE, and a merge computes
 * lse = ln sum_s e^{lse_s}, o = sum_s e^{lse_s - lse} o_s.
 *
 *  q          [B, Hq, d]
 *  k_cache, v_cache [num_blocks, block_size, Hkv, d]
 *  block_table int32 [B, max_blocks_per_seq]
 *  seq_lens   int32 [B]: keys visible to each query (the current token's own
 *             key included, so it must already be appended); 0 is allowed
 *  o          [B, Hq, d] (same dtype as q)
 *  lse        float32 [Hq, B] natural-log LSE; may be NULL
 *  window     <= 0: all keys; > 0: only the last `window` keys
 *  scale      <= 0: 1/sqrt(d)
 *  num_splits 0: chosen by the library from B, the table width and the SM
 *             count; > 0: the maximum number of ranges per sequence
 *  workspace  device scratch of at least pa_decode_workspace_bytes(...)
 *             bytes for the same arguments (may be NULL when that is 0)
 * block_size must be 16, and for bf16 Hq / Hkv at most 128 (d = 128) or 192
 * (d = 64); otherwise PA_ERR_UNSUPPORTED. Alignment: q, o, pools 16-byte
 * aligned; workspace 256-byte aligned.
 */
PA_API int pa_attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_table, int max_blocks_per_seq,
                         const int32_t* seq_lens, void* o, float* lse, int B, int Hq, int Hkv,
                         int d, int block_size, int num_blocks, int window, float scale,
                         int num_splits, void* workspace, size_t workspace_bytes,
                         pa_dtype dtype, int32_t* err_flag, void* stream);

/*
 * Workspace bytes attn_decode_paged (or attn_decode_paged_fp8) needs for these
 * arguments (0 when every sequence fits one range). Host-only arithmetic
 * except that num_splits = 0
 * reads the current device's SM count and the decode kernel's register count
 * (both cached per device). Returns 0 on invalid arguments too.
 */
PA_API size_t pa_decode_workspace_bytes(int B, int Hq, int Hkv, int d, int max_blocks_per_seq,
                                 int block_size, int window, int num_splits);

/*
 * FP8 key/value cache. "Генерация и KV-кэш", section "Сколько весит KV-кэш"
 * (one byte per cached number in FP8 instead of two in BF16) and section "Как
 * уменьшить кэш" (the byte lever); "Cache KV, atención flash ..." (a serving
 * engine started with an FP8 KV cache). The pages fix neither the format nor
 * the scaling; this library reads them as:
 *  - codes: E4M3 (OCP 8-bit floating point: sign, 4 exponent bits with bias 7,
 *    3 mantissa bits, no infinities, largest finite value 448), one byte per
 *    element, pools [num_blocks, block_size, Hkv, d] of uint8 like the bf16
 *    pools;
 *  - scales: k_scale[Hkv] and v_scale[Hkv], float32 device arrays; a code q of
 *    KV head h stands for value(q) * scale[h]. Scales must be finite and > 0:
 *    they live on the device, so the host cannot check them, and the decode
 *    folds the key scale into the softmax scale (a scale <= 0 would turn the
 *    running max into a running min: the result is then unspecified).
 */

/*
 * kv_append_paged_fp8 -- kv_append_paged into FP8 pools: each new bf16 row
 * element x of KV head h is stored as the E4M3 code nearest to
 * float32(x) / scale[h] (IEEE division; ties to the even mantissa; beyond
 * +-448 it saturates to +-448; NaN stays NaN). Placement, arguments and
 * error reporting as kv_append_paged (k_new / v_new bf16 [num_new_tokens,
 * Hkv, d]; pools uint8). Alignment: k_new, v_new 16 bytes; pools 8 bytes.
 */
PA_API int pa_kv_append_paged_fp8(const void* k_new, const void* v_new, void* k_cache,
                                  void* v_cache, const float* k_scale, const float* v_scale,
                                  const int32_t* block_table, int max_blocks_per_seq,
                                  const int32_t* seq_lens, const int32_t* cu_new,
                                  int num_new_tokens, int B, int Hkv, int d, int block_size,
                                  int num_blocks, int32_t* err_flag, void* stream);

/*
 * attn_decode_paged_fp8 -- attn_decode_paged over FP8 pools: the attention of
 * each query over the dequantised keys and values value(q) * scale[h]. q and o
 * are bf16; the keys and values are converted exactly to fp16 on chip, the
 * query is rounded to fp16 (exact for bf16 values of magnitude 2^-14 .. 65504)
 * and the probabilities to fp16 for the warp MMAs; the key scale is folded
 * into the head's softmax scale and the value scale into its output; fp32
 * accumulation. Arguments, workspace
 * (size it with pa_decode_workspace_bytes) and errors as attn_decode_paged;
 * block_size must be 16 and Hq / Hkv at most 64 (PA_ERR_UNSUPPORTED
 * otherwise). Alignment: q, o, pools 16 bytes; workspace 256.
 */
PA_API int pa_attn_decode_paged_fp8(const void* q, const void* k_cache, const void* v_cache,
                                    const float* k_scale, const float* v_scale,
                                    const int32_t* block_table, int max_blocks_per_seq,
                                    const int32_t* seq_lens, void* o, float* lse, int B, int Hq,
                                    int Hkv, int d, int block_size, int num_blocks, int window,
                                    float scale, int num_splits, void* workspace,
                                    size_t workspace_bytes, int32_t* err_flag, void* stream);

/* Bytes of the library's built-in decode scratch (see below): 32 MiB. */
#define PA_NOALLOC_SCRATCH_BYTES (32 * 1024 * 1024)

/*
 * attn_decode_paged_noalloc -- the same paged decode as attn_decode_paged
 * (same arguments, same kernels, same results) without the workspace
 * arguments. The pages have no counterpart: this entry point exists for
 * callers that cannot allocate device memory when they call it, such as a
 * serving process that reserves its whole memory budget at start-up and must
 * not allocate afterwards, or a plugin that only receives buffers from a host
 * framework that owns all device allocations.
 *
 * The split-KV partial outputs go to a scratch array compiled into the
 * library: PA_NOALLOC_SCRATCH_BYTES per GPU, held by every GPU that loads the
 * library until the process exits. The call allocates nothing.
 *  - A call whose partials need more than PA_NOALLOC_SCRATCH_BYTES
 *    (pa_decode_workspace_bytes for the same arguments) returns
 *    PA_ERR_WORKSPACE and launches nothing; pass a smaller num_splits (1 needs
 *    no scratch at all).
 *  - The first call on a device looks up the scratch's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture. PA_ERR_CUDA if the lookup fails. The address
 *    is cached per device with the unique id of the context it was looked up
 *    in; the first call from another context of the device, or after
 *    cudaDeviceReset replaced the context, looks it up again (so that call,
 *    too, belongs before any capture).
 *  - All calls on a device share the one array, which keeps whatever the last
 *    call left there (nothing in it needs to start at zero). Calls that can
 *    overlap on the GPU -- on different streams, or from different host
 *    threads -- race on it; order them on one stream.
 */
PA_API int pa_attn_decode_paged_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_table, int max_blocks_per_seq,
                                        const int32_t* seq_lens, void* o, float* lse, int B,
                                        int Hq, int Hkv, int d, int block_size, int num_blocks,
                                        int window, float scale, int num_splits, pa_dtype dtype,
                                        int32_t* err_flag, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H_ */
