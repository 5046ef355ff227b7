// attn_decode_paged: one query per sequence over its paged KV cache, with
// split-KV ranges merged through their log-sum-exp.
//
// Sources: the decode step ("Генерация и KV-кэш", section "KV-кэш для одной
// головы на NumPy": the new token's query against every cached key, stable
// softmax), the gather through the block table ("Module 09: Efficient
// Attention", section "The Block Table"), the query-to-KV-head mapping (same
// notebook, section "The Math: Sharing Keys and Values"), and the online
// recurrence with rescaling by e^{m_old - m_new} ("Ли Хунъи ... 2026", lecture
// "Ускоряем генерацию, часть 1: FlashAttention"). Merging two ranges is the
// same recurrence applied to their (max, sum) pairs, written with
// lse = m + ln(l).
//
// bf16 design (memory-bound, ~1-8 FLOP per byte read):
//  * CTA = (sequence, group of `hg` KV heads, range of `chunk` blocks).
//  * One producer thread walks the range's slice of the block table (staged
//    in shared memory) and issues TMA copies of each block's K and V rows for
//    the CTA's heads into a ring of `stages` shared-memory buffers. One copy
//    per 64-element panel brings the page's rows of all the CTA's heads
//    (16 tokens x hg heads x 128 B, up to 24 KB): the pool's tensor map lists
//    its dimensions as (d, token, head, block), so the box lands as hg head
//    tiles of 16 tokens x 128 B, each 128-byte swizzled so that the ldmatrix
//    reads below are bank-conflict free. (Per-head 2 KB copies cap an SM near
//    40 GB/s: copies, not bytes, were the limit.)
//  * One consumer warp per (KV head, 16 query heads): the G = Hq/Hkv query
//    heads that share the KV head are packed as the 16 rows of an m16n8k16
//    warp MMA (rows past G are zero), so K and V are read from shared memory
//    once per group. S = Q K^T and O += P V run on the tensor cores with fp32
//    accumulators; the running (max, sum) lives in registers and is reduced
//    across the 4 threads that share a row with warp shuffles.
//  * Scores of tokens outside [first visible, seq_len) are set to -inf and
//    their V rows zeroed, so unused slots of a block may hold anything.
#include <cmath>
#include <cstdint>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pa_kernels.h"
#include "pa_ptx.cuh"

namespace pa {

namespace {

constexpr int kBlk = 16;              // tokens per block (page)
constexpr int kBox = kBlk * 128;      // bytes of one (head, panel) box
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kNegInf = -INFINITY;

struct SeqRange {
  int len;      // visible keys end (exclusive), clamped to the table
  int t_begin;  // first visible key
  int p_begin;  // first block touched
  int n_pages;  // blocks touched
  int n_split;  // ranges
};

__device__ __forceinline__ SeqRange seq_range(int len, int max_blocks, int window, int chunk,
                                              int32_t* err, bool report) {
  SeqRange r;
  if (len < 0 || len > max_blocks * kBlk) {
    if (report) raise_err(err, kDevErrBadPosition);
    len = len < 0 ? 0 : max_blocks * kBlk;
  }
  r.len = len;
  r.t_begin = (window > 0 && len > window) ? len - window : 0;
  r.p_begin = r.t_begin / kBlk;
  r.n_pages = len > 0 ? (len + kBlk - 1) / kBlk - r.p_begin : 0;
  r.n_split = (r.n_pages + chunk - 1) / chunk;
  return r;
}

// ---------------------------------------------------------------- bf16 path
// Consumer warps per CTA at most (plus one producer warp), chosen so the
// accumulators (d/8 x 4 fp32) and Q fragments stay in registers.
template <int D>
constexpr int kMaxConsumerWarps = D == 128 ? 8 : 12;
constexpr int kSmemPerSm = 228 * 1024;  // shared memory per SM (planner input)

// One page (16 tokens) of one KV head for the 16 query-head rows of a
// consumer warp: S = Q K^T on the tensor cores, the mask of tokens outside
// [first visible, seq_len), the online softmax update (log2 domain) and
// O += P V. kb / vb: the page's K / V tile of this head in shared memory
// (64-column panel p at + p * hg * kBox), 128-byte swizzled.
template <int D>
__device__ __forceinline__ void consume_page(const uint32_t (&qa)[D / 16][4], uint32_t kb,
                                             uint32_t vb, int hg, int tok0, const SeqRange& r,
                                             float sl2, int mi, int tq, int ktok, int vtok,
                                             float& m0, float& m1, float& l0, float& l1,
                                             float (&acc)[D / 8][4]) {
  float sc[2][4];
#pragma unroll
  for (int t = 0; t < 2; ++t) sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int c = kk * 2 + (mi & 1);
    const uint32_t addr = kb + (c >> 3) * hg * kBox + ktok * 128 + (((c & 7) ^ (ktok & 7)) << 4);
    uint32_t b0, b1, b2, b3;
    ldsm_x4(addr, b0, b1, b2, b3);
    mma_bf16_16816(sc[0], qa[kk], b0, b1);
    mma_bf16_16816(sc[1], qa[kk], b2, b3);
  }

  const bool edge = (tok0 + kBlk > r.len) || (tok0 < r.t_begin);
  uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
  if (edge) {
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = tok0 + 8 * t + 2 * tq + (e & 1);
        if (tok >= r.len || tok < r.t_begin) sc[t][e] = kNegInf;
      }
    auto ok = [&](int tok) { return tok < r.len && tok >= r.t_begin; };
    const int ta = tok0 + 2 * tq, tb = tok0 + 8 + 2 * tq;
    mlo = (ok(ta) ? 0x0000FFFFu : 0u) | (ok(ta + 1) ? 0xFFFF0000u : 0u);
    mhi = (ok(tb) ? 0x0000FFFFu : 0u) | (ok(tb + 1) ? 0xFFFF0000u : 0u);
  }

  // online softmax (log2 domain), rows gr (e = 0,1) and gr + 8 (e = 2,3)
  float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1])) * sl2;
  float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3])) * sl2;
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 2));
  const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
  const float mu0 = mn0 == kNegInf ? 0.f : mn0;
  const float mu1 = mn1 == kNegInf ? 0.f : mn1;
  const float al0 = ex2(m0 - mu0), al1 = ex2(m1 - mu1);
  m0 = mn0;
  m1 = mn1;
  float ps[2][4];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    ps[t][0] = ex2(fmaf(sc[t][0], sl2, -mu0));
    ps[t][1] = ex2(fmaf(sc[t][1], sl2, -mu0));
    ps[t][2] = ex2(fmaf(sc[t][2], sl2, -mu1));
    ps[t][3] = ex2(fmaf(sc[t][3], sl2, -mu1));
  }
  l0 = l0 * al0 + (ps[0][0] + ps[0][1] + ps[1][0] + ps[1][1]);
  l1 = l1 * al1 + (ps[0][2] + ps[0][3] + ps[1][2] + ps[1][3]);
#pragma unroll
  for (int j = 0; j < D / 8; ++j) {
    acc[j][0] *= al0;
    acc[j][1] *= al0;
    acc[j][2] *= al1;
    acc[j][3] *= al1;
  }
  const uint32_t pa[4] = {pack_bf16(ps[0][0], ps[0][1]), pack_bf16(ps[0][2], ps[0][3]),
                          pack_bf16(ps[1][0], ps[1][1]), pack_bf16(ps[1][2], ps[1][3])};
#pragma unroll
  for (int jj = 0; jj < D / 16; ++jj) {
    const int c = jj * 2 + (mi >> 1);
    const uint32_t addr = vb + (c >> 3) * hg * kBox + vtok * 128 + (((c & 7) ^ (vtok & 7)) << 4);
    uint32_t v0, v1, v2, v3;
    ldsm_x4_t(addr, v0, v1, v2, v3);
    mma_bf16_16816(acc[2 * jj], pa, v0 & mlo, v1 & mhi);
    mma_bf16_16816(acc[2 * jj + 1], pa, v2 & mlo, v3 & mhi);
  }
}

template <int D>
__global__ void __launch_bounds__((kMaxConsumerWarps<D> + 1) * 32, 1)
decode_bf16_kernel(const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const DecodeArgs a, const int chunk,
                   const int num_splits, const int hg, const int mt, const int ns) {
  constexpr int P = D / 64;  // 128-byte panels per token row
  const int G = a.Hq / a.Hkv;
  const int b = blockIdx.z, hc = blockIdx.y, s = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = hg * mt;  // consumer warps

  const SeqRange r = seq_range(a.seq_lens[b], a.max_blocks, a.window, chunk, a.err,
                               s == 0 && hc == 0 && threadIdx.x == 0);
  if (s >= (r.n_split > 0 ? r.n_split : 1)) return;

  if (r.n_pages == 0) {  // no visible key: o = 0, lse = -inf
    const int h0 = hc * hg * G, nh = hg * G;
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.o);
    for (int i = threadIdx.x; i < nh * D; i += blockDim.x)
      o[(static_cast<int64_t>(b) * a.Hq + h0) * D + i] = __float2bfloat16_rn(0.f);
    if (a.lse)
      for (int i = threadIdx.x; i < nh; i += blockDim.x) a.lse[(h0 + i) * a.B + b] = kNegInf;
    return;
  }
  const int pstart = r.p_begin + s * chunk;
  const int npg = min(chunk, r.n_pages - s * chunk);
  const bool single = r.n_split == 1;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t stage_bytes = 2u * hg * P * kBox;
  const uint32_t bars = base + ns * stage_bytes;  // full[ns], empty[ns]
  int32_t* phys_s = reinterpret_cast<int32_t*>(gbase + ns * stage_bytes + 16 * ns);
  int32_t* tab_s = phys_s + ns;
  volatile int32_t* abort_s = tab_s + chunk;
  auto full = [&](int i) { return bars + 8u * i; };
  auto empty = [&](int i) { return bars + 8u * (ns + i); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), nw);
    }
    *abort_s = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < npg; i += blockDim.x)
    tab_s[i] = a.table[static_cast<int64_t>(b) * a.max_blocks + pstart + i];
  __syncthreads();

  if (warp == nw) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
      int issued = 0;
      uint32_t valid_mask = 0;  // validity of the last `ns` issued blocks (bit per stage)
      for (int i = 0; i < npg; ++i) {
        const int st = i % ns, u = i / ns;
        if (u > 0 && !mbar_wait(empty(st), (u - 1) & 1, a.wait_ns)) {
          raise_err(a.err, kDevErrTimeout);
          *abort_s = 1;
          break;
        }
        if (*abort_s) break;
        const int phys = tab_s[i];
        const bool ok = phys >= 0 && phys < a.num_blocks;
        if (!ok) raise_err(a.err, kDevErrBadBlock);
        phys_s[st] = ok ? phys : -1;
        if (ok) {
          mbar_arrive_expect_tx(full(st), stage_bytes);
          const uint32_t sb = base + st * stage_bytes;
          // one copy per 64-column panel brings the page's rows of all hg
          // heads: tiles [panel][head] of 16 tokens x 128 B, K then V
#pragma unroll
          for (int p = 0; p < P; ++p) {
            tma_load_4d(sb + p * hg * kBox, &kmap, full(st), p * 64, 0, hc * hg, phys);
            tma_load_4d(sb + (P + p) * hg * kBox, &vmap, full(st), p * 64, 0, hc * hg, phys);
          }
          valid_mask |= 1u << st;
        } else {
          valid_mask &= ~(1u << st);
          mbar_arrive(full(st));
        }
        issued = i + 1;
      }
      // Let no copy land after the CTA exits: wait for the last use of each
      // stage (already complete unless the loop was abandoned).
      for (int i = issued - ns > 0 ? issued - ns : 0; i < issued; ++i) {
        const int st = i % ns;
        if (valid_mask & (1u << st)) mbar_wait(full(st), (i / ns) & 1, 100000000ull);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = warp / mt, mti = warp % mt;
  const int kvh = hc * hg + g;
  const int qh0 = kvh * G + mti * 16;
  const int nrows = min(16, G - mti * 16);
  const int gr = lane >> 2, tq = lane & 3;
  const float sl2 = a.scale_log2;

  uint32_t qa[D / 16][4];
  {
    const uint32_t* q32 = static_cast<const uint32_t*>(a.q);
    const int64_t ra = (static_cast<int64_t>(b) * a.Hq + qh0 + gr) * (D / 2);
    const int64_t rb = ra + 8 * (D / 2);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][0] = gr < nrows ? q32[ra + kk * 8 + tq] : 0u;
      qa[kk][1] = gr + 8 < nrows ? q32[rb + kk * 8 + tq] : 0u;
      qa[kk][2] = gr < nrows ? q32[ra + kk * 8 + 4 + tq] : 0u;
      qa[kk][3] = gr + 8 < nrows ? q32[rb + kk * 8 + 4 + tq] : 0u;
    }
  }

  float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;
  float acc[D / 8][4];
#pragma unroll
  for (int j = 0; j < D / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  const int mi = lane >> 3, rr = lane & 7;
  const int ktok = ((mi >> 1) << 3) + rr;  // token row this lane addresses for K
  const int vtok = ((mi & 1) << 3) + rr;   // ... and for V (transposed load)

  for (int i = 0; i < npg; ++i) {
    const int st = i % ns;
    // warp-uniform outcome: the ldmatrix / mma.sync below need all 32 lanes
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(full(st), (i / ns) & 1, a.wait_ns))) {
      if (lane == 0) raise_err(a.err, kDevErrTimeout);
      *abort_s = 1;
      break;
    }
    const int phys = phys_s[st];
    if (phys >= 0)
      consume_page<D>(qa, base + st * stage_bytes + g * kBox,
                             base + st * stage_bytes + (P * hg + g) * kBox, hg,
                             (pstart + i) * kBlk, r, sl2, mi, tq, ktok, vtok, m0, m1, l0, l1, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(st));
  }

  // ------------------------------------------------------------- epilogue
  l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
  l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
  l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
  l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int row = gr + 8 * half;
    if (row >= nrows) continue;
    const int h = qh0 + row;
    const float l = half ? l1 : l0;
    const float m = half ? m1 : m0;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse_v = l > 0.f ? (m + log2f(l)) * kLn2 : kNegInf;
    const int64_t bh = static_cast<int64_t>(b) * a.Hq + h;
    if (single) {
      uint32_t* o32 = static_cast<uint32_t*>(a.o) + bh * (D / 2);
#pragma unroll
      for (int j = 0; j < D / 8; ++j)
        o32[j * 4 + tq] = pack_bf16(acc[j][2 * half] * inv, acc[j][2 * half + 1] * inv);
      if (tq == 0 && a.lse) a.lse[h * a.B + b] = lse_v;
    } else {
      float2* w = reinterpret_cast<float2*>(a.ws_o + (bh * num_splits + s) * D);
#pragma unroll
      for (int j = 0; j < D / 8; ++j)
        w[j * 4 + tq] = make_float2(acc[j][2 * half] * inv, acc[j][2 * half + 1] * inv);
      if (tq == 0) a.ws_lse[bh * num_splits + s] = lse_v;
    }
  }
}

// ------------------------------------------------------- FP8 (E4M3) cache path
// The same decode over pools of E4M3 codes with one fp32 scale per KV head for
// keys and one for values (a code q stands for value(q) * scale). A page's
// codes arrive by TMA: one box of d bytes x 16 tokens x hg heads for K and one
// for V (half the bytes of the bf16 path), swizzled in 16-byte pieces (the
// 128-byte pattern for d = 128, the 64-byte one for d = 64). A consumer warp
// serves up to 8 query heads of one KV head and builds its MMA operands
// straight from the codes in registers: every E4M3 value is an fp16 value, so
// one conversion per pair of codes gives one fp16 pair, and no fp16 copy of a
// page is written to shared memory (that copy cost five bytes of shared-memory
// traffic per byte of cache). The products are transposed so that the page's
// 16 keys, not the query heads, are the 16 rows of an m16n8k16 MMA and the
// heads its 8 columns: no padding rows for Hq / Hkv <= 8, half the MMAs and
// half the accumulator registers of a heads-as-rows layout.
//  * S^T = K Q^T. A = the K codes (rows = keys), contracted over the head
//    dims. A dot product does not depend on the order of its terms, so a lane
//    reads 16 whole bytes of each of its two key rows with one 128-bit load
//    and feeds 4 of them to each of four k-steps; the query (the B operand) is
//    loaded once in that same dim order.
//  * P^T (keys x heads, fp16) is the S^T accumulator tile as it stands, moved
//    into B-operand layout by two 8x8 register transposes.
//  * O^T += V^T P^T. A = V^T (rows = head dims, k = keys): an MMA register
//    pairs two keys of one dim, so a lane loads 8 bytes (8 dims) of each of its
//    4 key rows and interleaves two rows' bytes with byte permutes. Row r of
//    output tile 4u + t is dim 64u + 8 (r % 8) + 4 (r / 8) + t, so a lane ends
//    with 8 consecutive dims of each of its two heads.
//  * Row r < 8 of the score tile is page row fp8_key_row(r), row 8 + r is
//    page row 8 + fp8_key_row(r): with this order and the swizzle neither
//    load has a bank conflict (checked for both head dims).
// The query is rounded to fp16 once (exact for bf16 values of magnitude
// 2^-14 .. 65504). The key scale is folded into the softmax scale of the head
// and the value scale into its output, so no element is rescaled.

constexpr int kFp8ConsumerWarps = 8;  // per CTA at most; two CTAs fit on an SM

// Page row of score-tile row n < 8: 0, 7, 3, 4, 5, 2, 6, 1. The K loads of a
// quarter warp read rows fp8_key_row(2m), fp8_key_row(2m + 1), which differ in
// bits 0 and 2; the V loads read the rows of even n, or of odd n, across a
// warp, which differ in bits 1-2 and in bits 0 and 2: with the swizzle below
// every 16-byte piece a quarter (K) or half (V) warp reads lies in distinct
// banks.
__device__ __forceinline__ int fp8_key_row(int n) { return (0x16254370u >> (4 * n)) & 0xFu; }

// XOR pattern of the tensor copy's swizzle for byte offsets in page row `row`
// of a head tile of 16 rows x D bytes (tile base aligned to the pattern's
// period): 16-byte piece p of the row sits at piece p ^ pattern.
template <int D>
__device__ __forceinline__ uint32_t fp8_row_swz(int row) {
  if constexpr (D == 128)
    return static_cast<uint32_t>(row & 7) << 4;
  else
    return static_cast<uint32_t>((row >> 1) & 3) << 4;
}

__device__ __forceinline__ uint32_t e4m3_lo(uint32_t w) {
  return e4m3x2_to_f16x2(static_cast<uint16_t>(w));
}
__device__ __forceinline__ uint32_t e4m3_hi(uint32_t w) {
  return e4m3x2_to_f16x2(static_cast<uint16_t>(w >> 16));
}

// One page (16 tokens) of one KV head for the up to 8 query heads of a
// consumer warp, over the page's code tiles kt / vt (shared addresses). Lane
// (gr, tq) holds the scores of page rows fp8_key_row(gr) and 8 +
// fp8_key_row(gr) for the warp's heads 2 tq and 2 tq + 1; m[i] and l[i] are
// the running max (log2 domain) and sum of head 2 tq + i, l over this lane's
// keys only (summed across the lanes of a head at the end).
template <int D>
__device__ __forceinline__ void consume_page_fp8(const uint32_t (&qb)[D / 16][2], uint32_t kt,
                                                 uint32_t vt, int tok0, const SeqRange& r,
                                                 float sl2, int gr, int tq, float (&m)[2],
                                                 float (&l)[2], float (&acc)[D / 16][4]) {
  const int k0 = fp8_key_row(gr), k1 = 8 + k0;  // this lane's score rows
  const int ra = fp8_key_row(2 * tq), rb = fp8_key_row(2 * tq + 1);  // its V rows (and + 8)

  // S^T, even and odd k-steps in two accumulators (two MMA chains)
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const uint32_t a0 = kt + k0 * D + ((16u * tq) ^ fp8_row_swz<D>(k0));
    const uint32_t a1 = kt + k1 * D + ((16u * tq) ^ fp8_row_swz<D>(k1));
#pragma unroll
    for (int qc = 0; qc < D / 64; ++qc) {
      // qc > 0 only for D = 128, whose rows are 128-byte aligned: bit 6 of the
      // address is bit 6 of the in-row offset, and XOR commutes with the swizzle
      uint32_t w0[4], w1[4];
      lds_v4(a0 ^ (64u * qc), w0);
      lds_v4(a1 ^ (64u * qc), w1);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t a[4] = {e4m3_lo(w0[j]), e4m3_lo(w1[j]), e4m3_hi(w0[j]), e4m3_hi(w1[j])};
        if (j & 1)
          mma_f16_16816(s1, a, qb[4 * qc + j][0], qb[4 * qc + j][1]);
        else
          mma_f16_16816(s0, a, qb[4 * qc + j][0], qb[4 * qc + j][1]);
      }
    }
  }
  // V once the score MMAs are issued: the loads do not depend on the scores,
  // so their latency hides behind the MMAs and the softmax, and they hold no
  // registers across the K reads. vw[u][i]: 8 bytes (dims 64u + 8 gr .. + 7)
  // of row ra, rb, 8 + ra, 8 + rb. 64u sets bit 6 of the in-row offset, 8 gr
  // bits 3-5: the swizzle XORs bits 4-6 and the row bases keep bit 6 clear,
  // so the group offset is applied with XOR too.
  uint32_t vw[D / 64][4][2];
  {
    const int rows[4] = {ra, rb, 8 + ra, 8 + rb};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t a = vt + rows[i] * D + ((8u * gr) ^ fp8_row_swz<D>(rows[i]));
#pragma unroll
      for (int u = 0; u < D / 64; ++u) lds_v2(a ^ (64u * u), vw[u][i][0], vw[u][i][1]);
    }
  }

  // sc[0] / sc[1]: row k0, heads 2 tq / 2 tq + 1; sc[2] / sc[3]: row k1
  float sc[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) sc[e] = s0[e] + s1[e];

  const bool edge = (tok0 + kBlk > r.len) || (tok0 < r.t_begin);
  uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
  if (edge) {
    auto ok = [&](int tok) { return tok < r.len && tok >= r.t_begin; };
    if (!ok(tok0 + k0)) sc[0] = sc[1] = kNegInf;
    if (!ok(tok0 + k1)) sc[2] = sc[3] = kNegInf;
    mlo = (ok(tok0 + ra) ? 0x0000FFFFu : 0u) | (ok(tok0 + rb) ? 0xFFFF0000u : 0u);
    mhi = (ok(tok0 + 8 + ra) ? 0x0000FFFFu : 0u) | (ok(tok0 + 8 + rb) ? 0xFFFF0000u : 0u);
  }

  // online softmax per head (log2 domain): max over the page's 16 keys, i.e.
  // this lane's two rows and the lanes of other gr
  float mx0 = fmaxf(sc[0], sc[2]) * sl2, mx1 = fmaxf(sc[1], sc[3]) * sl2;
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, o));
  }
  const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
  const float mu0 = mn0 == kNegInf ? 0.f : mn0;
  const float mu1 = mn1 == kNegInf ? 0.f : mn1;
  const float al0 = ex2(m[0] - mu0), al1 = ex2(m[1] - mu1);
  m[0] = mn0;
  m[1] = mn1;
  const float p0 = ex2(fmaf(sc[0], sl2, -mu0)), p1 = ex2(fmaf(sc[1], sl2, -mu1));
  const float p2 = ex2(fmaf(sc[2], sl2, -mu0)), p3 = ex2(fmaf(sc[3], sl2, -mu1));
  l[0] = l[0] * al0 + (p0 + p2);
  l[1] = l[1] * al1 + (p1 + p3);
  // the factors are exactly 1 unless a head's max moved, which gets rare as
  // keys accumulate: skip the multiplies when no head of the warp needs them
  if (__any_sync(0xFFFFFFFFu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
    for (int t = 0; t < D / 16; ++t) {
      acc[t][0] *= al0;
      acc[t][1] *= al1;
      acc[t][2] *= al0;
      acc[t][3] *= al1;
    }
  }
  // P^T as the B operand: head gr, score rows 2 tq, 2 tq + 1 (pb0) and
  // 8 + 2 tq, 8 + 2 tq + 1 (pb1)
  const uint32_t pb0 = movmatrix_trans(pack_f16(p0, p1));
  const uint32_t pb1 = movmatrix_trans(pack_f16(p2, p3));

  // O^T += V^T P^T. A registers of tile 4u + t: rows (ra, rb) of dim
  // 64u + 8 gr + t, the same rows of dim + 4, then rows (8 + ra, 8 + rb) of
  // both dims. Edge pages zero the V values of masked keys (P = 0 times a NaN
  // code is NaN); the others skip the masking.
  auto pv = [&](auto masked) {
    auto mk = [&](uint32_t h, uint32_t msk) { return decltype(masked)::value ? h & msk : h; };
#pragma unroll
    for (int u = 0; u < D / 64; ++u) {
      const uint32_t x01 = __byte_perm(vw[u][0][0], vw[u][1][0], 0x5140);
      const uint32_t x23 = __byte_perm(vw[u][0][0], vw[u][1][0], 0x7362);
      const uint32_t y01 = __byte_perm(vw[u][0][1], vw[u][1][1], 0x5140);
      const uint32_t y23 = __byte_perm(vw[u][0][1], vw[u][1][1], 0x7362);
      const uint32_t z01 = __byte_perm(vw[u][2][0], vw[u][3][0], 0x5140);
      const uint32_t z23 = __byte_perm(vw[u][2][0], vw[u][3][0], 0x7362);
      const uint32_t w01 = __byte_perm(vw[u][2][1], vw[u][3][1], 0x5140);
      const uint32_t w23 = __byte_perm(vw[u][2][1], vw[u][3][1], 0x7362);
      const uint32_t a0[4] = {mk(e4m3_lo(x01), mlo), mk(e4m3_lo(y01), mlo),
                              mk(e4m3_lo(z01), mhi), mk(e4m3_lo(w01), mhi)};
      mma_f16_16816(acc[4 * u + 0], a0, pb0, pb1);
      const uint32_t a1[4] = {mk(e4m3_hi(x01), mlo), mk(e4m3_hi(y01), mlo),
                              mk(e4m3_hi(z01), mhi), mk(e4m3_hi(w01), mhi)};
      mma_f16_16816(acc[4 * u + 1], a1, pb0, pb1);
      const uint32_t a2[4] = {mk(e4m3_lo(x23), mlo), mk(e4m3_lo(y23), mlo),
                              mk(e4m3_lo(z23), mhi), mk(e4m3_lo(w23), mhi)};
      mma_f16_16816(acc[4 * u + 2], a2, pb0, pb1);
      const uint32_t a3[4] = {mk(e4m3_hi(x23), mlo), mk(e4m3_hi(y23), mlo),
                              mk(e4m3_hi(z23), mhi), mk(e4m3_hi(w23), mhi)};
      mma_f16_16816(acc[4 * u + 3], a3, pb0, pb1);
    }
  };
  if (edge)
    pv(std::true_type{});
  else
    pv(std::false_type{});
}

template <int D>
__global__ void __launch_bounds__((kFp8ConsumerWarps + 1) * 32, 2)
decode_fp8_kernel(const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const DecodeArgs a,
                  const float* __restrict__ k_scale, const float* __restrict__ v_scale,
                  const int chunk, const int num_splits, const int hg, const int mt,
                  const int ns) {
  const int G = a.Hq / a.Hkv;
  const int b = blockIdx.z, hc = blockIdx.y, s = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = hg * mt;  // consumer warps

  const SeqRange r = seq_range(a.seq_lens[b], a.max_blocks, a.window, chunk, a.err,
                               s == 0 && hc == 0 && threadIdx.x == 0);
  if (s >= (r.n_split > 0 ? r.n_split : 1)) return;

  if (r.n_pages == 0) {  // no visible key: o = 0, lse = -inf
    const int h0 = hc * hg * G, nh = hg * G;
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.o);
    for (int i = threadIdx.x; i < nh * D; i += blockDim.x)
      o[(static_cast<int64_t>(b) * a.Hq + h0) * D + i] = __float2bfloat16_rn(0.f);
    if (a.lse)
      for (int i = threadIdx.x; i < nh; i += blockDim.x) a.lse[(h0 + i) * a.B + b] = kNegInf;
    return;
  }
  const int pstart = r.p_begin + s * chunk;
  const int npg = min(chunk, r.n_pages - s * chunk);
  const bool single = r.n_split == 1;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  // K codes [hg][16][D], then V codes: head tiles of 1 or 2 KB on 1024-byte
  // boundaries, as the swizzle pattern needs
  const uint32_t stage_bytes = 2u * hg * kBlk * D;
  const uint32_t bars = base + ns * stage_bytes;  // full[ns], empty[ns]
  int32_t* phys_s = reinterpret_cast<int32_t*>(gbase + ns * stage_bytes + 16 * ns);
  int32_t* tab_s = phys_s + ns;
  volatile int32_t* abort_s = tab_s + chunk;
  auto full = [&](int i) { return bars + 8u * i; };
  auto empty = [&](int i) { return bars + 8u * (ns + i); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), nw);
    }
    *abort_s = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < npg; i += blockDim.x)
    tab_s[i] = a.table[static_cast<int64_t>(b) * a.max_blocks + pstart + i];
  __syncthreads();

  if (warp == nw) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
      int issued = 0;
      uint32_t valid_mask = 0;  // validity of the last `ns` issued blocks (bit per stage)
      for (int i = 0; i < npg; ++i) {
        const int st = i % ns, u = i / ns;
        if (u > 0 && !mbar_wait(empty(st), (u - 1) & 1, a.wait_ns)) {
          raise_err(a.err, kDevErrTimeout);
          *abort_s = 1;
          break;
        }
        if (*abort_s) break;
        const int phys = tab_s[i];
        const bool ok = phys >= 0 && phys < a.num_blocks;
        if (!ok) raise_err(a.err, kDevErrBadBlock);
        phys_s[st] = ok ? phys : -1;
        if (ok) {
          mbar_arrive_expect_tx(full(st), stage_bytes);
          const uint32_t sb = base + st * stage_bytes;
          tma_load_4d(sb, &kmap, full(st), 0, 0, hc * hg, phys);
          tma_load_4d(sb + stage_bytes / 2, &vmap, full(st), 0, 0, hc * hg, phys);
          valid_mask |= 1u << st;
        } else {
          valid_mask &= ~(1u << st);
          mbar_arrive(full(st));
        }
        issued = i + 1;
      }
      for (int i = issued - ns > 0 ? issued - ns : 0; i < issued; ++i) {
        const int st = i % ns;
        if (valid_mask & (1u << st)) mbar_wait(full(st), (i / ns) & 1, 100000000ull);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = warp / mt, mti = warp % mt;
  const int kvh = hc * hg + g;
  const int qh0 = kvh * G + mti * 8;  // the warp's heads: columns 0 .. nh - 1
  const int nh = min(8, G - mti * 8);
  const int gr = lane >> 2, tq = lane & 3;
  const float sl2 = a.scale_log2 * k_scale[kvh];
  const float vsc = v_scale[kvh];

  // query of head gr (the B operand's column), rounded to fp16, in the dim
  // order of the K reads: k-step 4 qc + j takes dims 64 qc + 16 tq + 4 j +
  // {0, 1} (k = 2 tq, 2 tq + 1) and + {2, 3} (k = 2 tq + 8, 2 tq + 9)
  uint32_t qb[D / 16][2];
  {
    const uint32_t* q32 = static_cast<const uint32_t*>(a.q);
    const int64_t rq = (static_cast<int64_t>(b) * a.Hq + qh0 + gr) * (D / 2);
    auto h2 = [](uint32_t w) {
      return pack_f16(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    };
#pragma unroll
    for (int qc = 0; qc < D / 64; ++qc)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int w = 32 * qc + 8 * tq + 2 * j;  // word w holds dims 2w, 2w + 1
        qb[4 * qc + j][0] = gr < nh ? h2(q32[rq + w]) : 0u;
        qb[4 * qc + j][1] = gr < nh ? h2(q32[rq + w + 1]) : 0u;
      }
  }

  float m[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f};
  float acc[D / 16][4];
#pragma unroll
  for (int t = 0; t < D / 16; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

  for (int i = 0; i < npg; ++i) {
    const int st = i % ns;
    // warp-uniform outcome: the mma.sync below need all 32 lanes
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(full(st), (i / ns) & 1, a.wait_ns))) {
      if (lane == 0) raise_err(a.err, kDevErrTimeout);
      *abort_s = 1;
      break;
    }
    const int phys = phys_s[st];
    if (phys >= 0) {
      const uint32_t kt = base + st * stage_bytes + static_cast<uint32_t>(g * kBlk * D);
      consume_page_fp8<D>(qb, kt, kt + stage_bytes / 2, (pstart + i) * kBlk, r, sl2, gr, tq, m,
                          l, acc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(st));
  }

  // ------------------------------------------------------------- epilogue
  // head 2 tq + i: dim 64u + 8 gr + t is acc[4u + t][i], dim 64u + 8 gr + 4 + t
  // is acc[4u + t][2 + i]: 8 consecutive dims per lane, head and group
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) l[i] += __shfl_xor_sync(0xFFFFFFFFu, l[i], o);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int n = 2 * tq + i;
    if (n >= nh) continue;
    const int h = qh0 + n;
    const float inv = l[i] > 0.f ? vsc / l[i] : 0.f;
    const float lse_v = l[i] > 0.f ? (m[i] + log2f(l[i])) * kLn2 : kNegInf;
    const int64_t bh = static_cast<int64_t>(b) * a.Hq + h;
    if (single) {
      uint4* o4 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o) + bh * D);
#pragma unroll
      for (int u = 0; u < D / 64; ++u)
        o4[8 * u + gr] =
            make_uint4(pack_bf16(acc[4 * u][i] * inv, acc[4 * u + 1][i] * inv),
                       pack_bf16(acc[4 * u + 2][i] * inv, acc[4 * u + 3][i] * inv),
                       pack_bf16(acc[4 * u][2 + i] * inv, acc[4 * u + 1][2 + i] * inv),
                       pack_bf16(acc[4 * u + 2][2 + i] * inv, acc[4 * u + 3][2 + i] * inv));
      if (gr == 0 && a.lse) a.lse[h * a.B + b] = lse_v;
    } else {
      float4* w = reinterpret_cast<float4*>(a.ws_o + (bh * num_splits + s) * D);
#pragma unroll
      for (int u = 0; u < D / 64; ++u) {
        w[16 * u + 2 * gr] = make_float4(acc[4 * u][i] * inv, acc[4 * u + 1][i] * inv,
                                         acc[4 * u + 2][i] * inv, acc[4 * u + 3][i] * inv);
        w[16 * u + 2 * gr + 1] =
            make_float4(acc[4 * u][2 + i] * inv, acc[4 * u + 1][2 + i] * inv,
                        acc[4 * u + 2][2 + i] * inv, acc[4 * u + 3][2 + i] * inv);
      }
      if (gr == 0) a.ws_lse[bh * num_splits + s] = lse_v;
    }
  }
}

// --------------------------------------------------------------- fp32 path
// CUDA-core reference-speed path for fp32 caches: one warp per (sequence,
// query head, range); each lane owns d/32 columns; dot products are reduced
// with warp shuffles.
template <int D>
__global__ void __launch_bounds__(128)
decode_f32_kernel(const DecodeArgs a, const int chunk, const int num_splits) {
  const int b = blockIdx.z, s = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * 4 + warp;
  if (h >= a.Hq) return;
  const int G = a.Hq / a.Hkv, g = h / G;
  const SeqRange r = seq_range(a.seq_lens[b], a.max_blocks, a.window, chunk, a.err,
                               s == 0 && h == 0 && lane == 0);
  if (s >= (r.n_split > 0 ? r.n_split : 1)) return;
  const int64_t bh = static_cast<int64_t>(b) * a.Hq + h;
  float* o = static_cast<float*>(a.o);
  if (r.n_pages == 0) {
    for (int c = lane; c < D; c += 32) o[bh * D + c] = 0.f;
    if (lane == 0 && a.lse) a.lse[h * a.B + b] = kNegInf;
    return;
  }
  const float* qf = static_cast<const float*>(a.q) + bh * D;
  const float* kc = static_cast<const float*>(a.k_cache);
  const float* vc = static_cast<const float*>(a.v_cache);
  float qv[D / 32], acc[D / 32];
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    qv[i] = qf[lane + 32 * i];
    acc[i] = 0.f;
  }
  float m = kNegInf, l = 0.f;
  const int pstart = r.p_begin + s * chunk;
  const int npg = min(chunk, r.n_pages - s * chunk);
  for (int i = 0; i < npg; ++i) {
    const int page = pstart + i;
    const int phys = a.table[static_cast<int64_t>(b) * a.max_blocks + page];
    if (phys < 0 || phys >= a.num_blocks) {
      if (lane == 0) raise_err(a.err, kDevErrBadBlock);
      continue;
    }
    for (int t = 0; t < kBlk; ++t) {
      const int tok = page * kBlk + t;
      if (tok < r.t_begin || tok >= r.len) continue;
      const int64_t row = ((static_cast<int64_t>(phys) * kBlk + t) * a.Hkv + g) * D;
      float dot = 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) dot = fmaf(qv[c], kc[row + lane + 32 * c], dot);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, off);
      const float s2 = dot * a.scale_log2;
      const float mn = fmaxf(m, s2);
      const float al = ex2(m - mn);
      const float p = ex2(s2 - mn);
      l = l * al + p;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) acc[c] = fmaf(p, vc[row + lane + 32 * c], acc[c] * al);
      m = mn;
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const float lse_v = l > 0.f ? (m + log2f(l)) * kLn2 : kNegInf;
  if (r.n_split == 1) {
#pragma unroll
    for (int c = 0; c < D / 32; ++c) o[bh * D + lane + 32 * c] = acc[c] * inv;
    if (lane == 0 && a.lse) a.lse[h * a.B + b] = lse_v;
  } else {
#pragma unroll
    for (int c = 0; c < D / 32; ++c) a.ws_o[(bh * num_splits + s) * D + lane + 32 * c] = acc[c] * inv;
    if (lane == 0) a.ws_lse[bh * num_splits + s] = lse_v;
  }
}

// ------------------------------------------------------------------ merge
// lse = ln sum_s e^{lse_s}; o = sum_s e^{lse_s - lse} o_s. One warp per
// (sequence, query head); sequences that used a single range were finished
// by the decode kernel and are skipped here.
template <typename OutT, int D>
__global__ void __launch_bounds__(256)
decode_merge_kernel(const DecodeArgs a, const int chunk, const int num_splits) {
  // launched as a programmatic dependent of the decode kernel: its CTAs may
  // start while the decode's last CTAs finish, and wait here until that grid
  // has completed and its partials are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int idx = blockIdx.x * 8 + warp;
  if (idx >= a.B * a.Hq) return;
  const int b = idx / a.Hq, h = idx % a.Hq;
  const SeqRange r = seq_range(a.seq_lens[b], a.max_blocks, a.window, chunk, a.err, false);
  if (r.n_split <= 1) return;
  const float* ls = a.ws_lse + static_cast<int64_t>(idx) * num_splits;
  float mx = kNegInf;
  for (int i = lane; i < r.n_split; i += 32) mx = fmaxf(mx, ls[i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  // each lane owns D/32 consecutive columns; four ranges are loaded before
  // any is used, so their latencies overlap
  constexpr int V = D / 32;
  float acc[V];
#pragma unroll
  for (int c = 0; c < V; ++c) acc[c] = 0.f;
  float total = 0.f;
  const float* wo = a.ws_o + static_cast<int64_t>(idx) * num_splits * D + lane * V;
  auto load_row = [&](int i, float (&v)[V]) {
    if constexpr (V == 4) {
      const float4 t = *reinterpret_cast<const float4*>(wo + static_cast<int64_t>(i) * D);
      v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
      const float2 t = *reinterpret_cast<const float2*>(wo + static_cast<int64_t>(i) * D);
      v[0] = t.x; v[1] = t.y;
    }
  };
  int i = 0;
  for (; i + 4 <= r.n_split; i += 4) {
    float v[4][V], lw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      lw[u] = ls[i + u];
      load_row(i + u, v[u]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = expf(lw[u] - mx);
      total += w;
#pragma unroll
      for (int c = 0; c < V; ++c) acc[c] = fmaf(w, v[u][c], acc[c]);
    }
  }
  for (; i < r.n_split; ++i) {
    float v[V];
    load_row(i, v);
    const float w = expf(ls[i] - mx);
    total += w;
#pragma unroll
    for (int c = 0; c < V; ++c) acc[c] = fmaf(w, v[c], acc[c]);
  }
  const float inv = 1.f / total;
  OutT* o = static_cast<OutT*>(a.o) + static_cast<int64_t>(idx) * D + lane * V;
#pragma unroll
  for (int c = 0; c < V; ++c) {
    if constexpr (sizeof(OutT) == 2)
      o[c] = __float2bfloat16_rn(acc[c] * inv);
    else
      o[c] = acc[c] * inv;
  }
  if (lane == 0 && a.lse) a.lse[h * a.B + b] = mx + logf(total);
}

int g_attr_done[2][64];

template <int D>
void ensure_smem_attr(size_t bytes) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (g_attr_done[D == 128][dev] < static_cast<int>(bytes)) {
    cudaFuncSetAttribute(decode_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(bytes));
    g_attr_done[D == 128][dev] = static_cast<int>(bytes);
  }
}

// Registers per thread of the bf16 (or FP8) decode kernel as compiled (read
// once per device), rounded up to the allocation step of 8: the planner's
// count of CTAs that fit on an SM follows the build instead of a number
// written down.
int decode_regs(int d, bool fp8) {
  static int cached[2][2][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int& c = cached[fp8][d == 128][dev];
  if (!c) {
    cudaFuncAttributes fa{};
    cudaError_t e;
    if (fp8)
      e = d == 128 ? cudaFuncGetAttributes(&fa, decode_fp8_kernel<128>)
                   : cudaFuncGetAttributes(&fa, decode_fp8_kernel<64>);
    else
      e = d == 128 ? cudaFuncGetAttributes(&fa, decode_bf16_kernel<128>)
                   : cudaFuncGetAttributes(&fa, decode_bf16_kernel<64>);
    if (e != cudaSuccess || fa.numRegs <= 0) {
      cudaGetLastError();
      return 255;  // unknown: plan as if one CTA per SM
    }
    c = (fa.numRegs + 7) / 8 * 8;
  }
  return c;
}

int g_attr8_done[2][64];

template <int D>
void ensure_smem_attr_fp8(size_t bytes) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (g_attr8_done[D == 128][dev] < static_cast<int>(bytes)) {
    cudaFuncSetAttribute(decode_fp8_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(bytes));
    g_attr8_done[D == 128][dev] = static_cast<int>(bytes);
  }
}

}  // namespace

int decode_max_group(int d, bool fp8) {
  if (fp8) return 8 * kFp8ConsumerWarps;
  return 16 * (d == 128 ? kMaxConsumerWarps<128> : kMaxConsumerWarps<64>);
}

DecodePlan plan_decode(int B, int Hq, int Hkv, int d, int max_blocks, int block_size, int window,
                       int num_splits_req, int sm_count, bool f32, bool fp8) {
  DecodePlan p{};
  const int G = Hq / Hkv;
  const int sms = sm_count > 0 ? sm_count : 148;
  int eff = max_blocks;  // blocks one sequence can touch
  if (window > 0) {
    const int wb = (window + block_size - 2) / block_size + 1;
    eff = wb < max_blocks ? wb : max_blocks;
  }
  if (eff < 1) eff = 1;
  if (f32) {
    p.hg = 1;
    p.head_chunks = 1;
    p.mt = 1;
    p.stages = 0;
    p.threads = 128;
  } else {
    const int P = d / 64;
    // a bf16 consumer warp serves 16 query heads (MMA rows), an FP8 one 8
    // (MMA columns of the transposed products)
    const int max_warps =
        fp8 ? kFp8ConsumerWarps : (d == 128 ? kMaxConsumerWarps<128> : kMaxConsumerWarps<64>);
    p.mt = fp8 ? (G + 7) / 8 : (G + 15) / 16;
    int hg = 1;
    for (int c = 1; c <= Hkv; ++c)
      if (Hkv % c == 0 && c * p.mt <= max_warps && 2 * c * P * kBox <= 64 * 1024) hg = c;
    p.hg = hg;
    p.head_chunks = Hkv / hg;
    // FP8 pages are half the bytes, and two FP8 CTAs share an SM (its
    // registers allow it), each with half the ring
    const int stage = fp8 ? hg * P * kBox : 2 * hg * P * kBox;
    int ns = (fp8 ? 100 : 200) * 1024 / stage;
    p.stages = ns < 2 ? 2 : (ns > 8 ? 8 : ns);
    p.threads = (hg * p.mt + 1) * 32;
  }
  int chunk;
  if (num_splits_req > 0) {
    chunk = (eff + num_splits_req - 1) / num_splits_req;
  } else {
    // Ranges of 4-64 blocks, about two CTAs per SM: fine enough to even out
    // sequences of very different lengths.
    const long long units = static_cast<long long>(B) * p.head_chunks;
    const long long target = 2LL * sms;
    long long c = (units * eff + target - 1) / target;
    c = c < 4 ? 4 : (c > 64 ? 64 : c);
    chunk = static_cast<int>(c);
    // A small call that this cut would spread over a few waves (a ring CTA
    // holds most of an SM's shared memory and registers) runs in one wave
    // instead: the largest range count per sequence that still fits.
    if (!f32) {
      const int regs = decode_regs(d, fp8);
      const int P = d / 64;
      const long long smem = 1024 + p.stages * ((fp8 ? 1LL : 2LL) * p.hg * P * kBox) + 64;
      long long cps = kSmemPerSm / (smem + 1024);
      const long long cps_regs = 65536 / (static_cast<long long>(p.threads) * regs);
      cps = cps < cps_regs ? cps : cps_regs;
      if (cps < 1) cps = 1;
      const long long slots = cps * sms;
      const long long ctas = units * ((eff + chunk - 1) / chunk);
      if (ctas > slots && ctas <= 3 * slots && units <= slots) {
        const long long splits = slots / units;
        chunk = static_cast<int>((eff + splits - 1) / splits);
      }
    }
  }
  if (chunk > eff) chunk = eff;
  if (chunk < 1) chunk = 1;
  p.chunk = chunk;
  p.num_splits = (eff + chunk - 1) / chunk;
  if (!f32) {
    const int P = d / 64;
    const size_t stage = (fp8 ? 1ull : 2ull) * p.hg * P * kBox;
    p.smem = 1024 + p.stages * stage + 16ull * p.stages + 4ull * p.stages + 4ull * chunk + 16;
  }
  if (p.num_splits > 1) {
    const size_t n = static_cast<size_t>(B) * Hq * p.num_splits;
    const size_t o_bytes = (n * d * 4 + 255) / 256 * 256;
    p.workspace = o_bytes + (n * 4 + 255) / 256 * 256;
  } else {
    p.workspace = 0;
  }
  return p;
}

// The merge kernel follows the decode kernel on the same stream as a
// programmatic dependent launch, which hides its launch latency behind the
// decode's tail.
template <typename K>
cudaError_t launch_merge(K kernel, const DecodeArgs& a, const DecodePlan& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.B * a.Hq + 7) / 8);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a, p.chunk, p.num_splits);
}

cudaError_t launch_decode_bf16(const DecodeArgs& a, const DecodePlan& p, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, cudaStream_t s) {
  const dim3 grid(p.num_splits, p.head_chunks, a.B);
  if (a.d == 128) {
    ensure_smem_attr<128>(p.smem);
    decode_bf16_kernel<128><<<grid, p.threads, p.smem, s>>>(kmap, vmap, a, p.chunk, p.num_splits,
                                                            p.hg, p.mt, p.stages);
  } else {
    ensure_smem_attr<64>(p.smem);
    decode_bf16_kernel<64><<<grid, p.threads, p.smem, s>>>(kmap, vmap, a, p.chunk, p.num_splits,
                                                           p.hg, p.mt, p.stages);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.num_splits <= 1) return e;
  if (a.d == 128) return launch_merge(decode_merge_kernel<__nv_bfloat16, 128>, a, p, s);
  return launch_merge(decode_merge_kernel<__nv_bfloat16, 64>, a, p, s);
}

cudaError_t launch_decode_fp8(const DecodeArgs& a, const DecodePlan& p, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, const float* k_scale,
                              const float* v_scale, cudaStream_t s) {
  const dim3 grid(p.num_splits, p.head_chunks, a.B);
  if (a.d == 128) {
    ensure_smem_attr_fp8<128>(p.smem);
    decode_fp8_kernel<128><<<grid, p.threads, p.smem, s>>>(kmap, vmap, a, k_scale, v_scale,
                                                           p.chunk, p.num_splits, p.hg, p.mt,
                                                           p.stages);
  } else {
    ensure_smem_attr_fp8<64>(p.smem);
    decode_fp8_kernel<64><<<grid, p.threads, p.smem, s>>>(kmap, vmap, a, k_scale, v_scale,
                                                          p.chunk, p.num_splits, p.hg, p.mt,
                                                          p.stages);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.num_splits <= 1) return e;
  if (a.d == 128) return launch_merge(decode_merge_kernel<__nv_bfloat16, 128>, a, p, s);
  return launch_merge(decode_merge_kernel<__nv_bfloat16, 64>, a, p, s);
}

cudaError_t launch_decode_f32(const DecodeArgs& a, const DecodePlan& p, cudaStream_t s) {
  const dim3 grid(p.num_splits, (a.Hq + 3) / 4, a.B);
  if (a.d == 128)
    decode_f32_kernel<128><<<grid, 128, 0, s>>>(a, p.chunk, p.num_splits);
  else
    decode_f32_kernel<64><<<grid, 128, 0, s>>>(a, p.chunk, p.num_splits);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.num_splits <= 1) return e;
  if (a.d == 128) return launch_merge(decode_merge_kernel<float, 128>, a, p, s);
  return launch_merge(decode_merge_kernel<float, 64>, a, p, s);
}

}  // namespace pa
