// attn_mla_decode_paged: multi-head latent attention, one query per sequence
// over a paged cache of latent rows, split-KV ranges merged through their
// log-sum-exp.
//
// Sources: the latent cache (one latent c_j of d_c = 512 numbers and one
// decoupled rope key of d_R = 64 per token, no head axis), the per-head
// reconstruction k_{j,i} = [W^UK_i c_j ; kR_j], v_{j,i} = W^UV_i c_j, and the
// absorption that lets the query attend the latent directly ("Module 09:
// Efficient Attention", section "Multi-head Latent Attention: A Different
// Lever", subsections "The Math: Compress, Reconstruct, Decouple" and "Why
// RoPE Has To Be Decoupled"); the weighted sum formed in the latent space and
// decompressed once at the end ("Ли Хунъи ... 2026", the KV-compression
// levers, item 2). With the absorbed query q_i = [W^UK_i^T q^C_i ; q^R_i]
// this kernel computes, per head i,
//     s_ij = scale * q_i . r_j,  o_lat_i = sum_j softmax_j(s)_ij r_j[:512],
// where r_j = [c_j ; kR_j] is the cached row; the caller up-projects o_lat.
// Paging, online softmax and the split-KV merge are those of the paged GQA
// decode.
//
// sm_103a design. Every query head reads the same latent rows, so MLA decode
// is multi-query attention with a 576-wide key and a 512-wide value that is
// the key's first 512 numbers. A CTA takes one sequence, 16 or 32 query
// heads and a range of blocks:
//  * one producer thread copies two blocks per step (32 rows x 1152 bytes)
//    with one TMA per block: the pool's tensor map lists the dimensions as
//    (64 elements, token, 64-element panel, block), so a block lands as 9
//    panels of 16 rows x 128 bytes, 128-byte swizzled;
//  * four consumer warps per 16 heads. S = Q R^T is split over the 576-wide
//    dot product (warp w takes dims 144w..144w+143, nine m16n8k16 steps); the
//    four partial score tiles are summed through shared memory (a bounded
//    mbarrier exchange, double-buffered), every warp then holds the same
//    scores, runs the same online softmax, and multiplies P into its own 128
//    latent dims (O += P C with the value tile read transposed from the same
//    rows). K and V are one tile: each row is read from HBM once for all
//    heads.
//  * The queries of the CTA's heads sit in shared memory in the same
//    swizzled panel layout and are read as A fragments with ldmatrix.
// Tokens past the sequence end, and blocks whose id is out of range, get
// -inf scores and zeroed value fragments, so unused slots may hold anything.
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mla_kernels.h"
#include "pa_ptx.cuh"

namespace pa {

namespace {

constexpr int kBlk = 16;                       // tokens per block
constexpr int kPanels = kMlaRow / 64;          // 64-element panels per row (9)
constexpr int kPanelBytes = kBlk * 128;        // one panel of a block: 16 rows x 128 B
constexpr int kPage = kPanels * kPanelBytes;   // one block of rows (18 KB)
constexpr int kStep = 2 * kPage;               // two blocks per consumer step
constexpr int kQTile = kPanels * 16 * 128;     // 16 query rows in the same layout (18 KB)
constexpr int kRedBytes = 4 * 4 * 32 * 16;     // partial scores of one group: 4 warps x 16 x 32 fp32
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kNegInf = -INFINITY;

struct MlaRange {
  int len;      // keys, clamped to the table
  int n_pages;  // blocks holding them
  int n_split;  // ranges
};

__device__ __forceinline__ MlaRange mla_range(int len, int max_blocks, int chunk, int32_t* err,
                                              bool report) {
  MlaRange r;
  if (len < 0 || len > max_blocks * kBlk) {
    if (report) raise_err(err, kDevErrBadPosition);
    len = len < 0 ? 0 : max_blocks * kBlk;
  }
  r.len = len;
  r.n_pages = (len + kBlk - 1) / kBlk;
  r.n_split = (r.n_pages + chunk - 1) / chunk;
  return r;
}

// shared-memory address of 16-byte chunk c (of 72 along a 576-wide row) of
// row `row` in a tile stored as 64-element panels of `rows` x 128 bytes
__device__ __forceinline__ uint32_t swz_addr(uint32_t tile, int panel_bytes, int row, int c) {
  return tile + (c >> 3) * panel_bytes + row * 128 + (((c & 7) ^ (row & 7)) << 4);
}

template <int NG>
__global__ void __launch_bounds__((4 * NG + 1) * 32, NG == 1 ? 2 : 1)
mla_decode_kernel(const __grid_constant__ CUtensorMap cmap, const MlaArgs a, const int chunk,
                  const int num_splits, const int ns) {
  constexpr int NW = 4 * NG;  // consumer warps
  const int b = blockIdx.z, hc = blockIdx.y, s = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h0 = hc * 16 * NG;

  const MlaRange r = mla_range(a.seq_lens[b], a.max_blocks, chunk, a.err,
                               s == 0 && hc == 0 && threadIdx.x == 0);
  if (s >= (r.n_split > 0 ? r.n_split : 1)) return;
  const int nh = min(16 * NG, a.H - h0);  // heads of this CTA
  if (r.n_pages == 0) {  // no key: o = 0, lse = -inf
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.o);
    for (int i = threadIdx.x; i < nh * kMlaDc; i += blockDim.x)
      o[(static_cast<int64_t>(b) * a.H + h0) * kMlaDc + i] = __float2bfloat16_rn(0.f);
    if (a.lse)
      for (int i = threadIdx.x; i < nh; i += blockDim.x) a.lse[(h0 + i) * a.B + b] = kNegInf;
    return;
  }
  const int pstart = s * chunk;
  const int npg = min(chunk, r.n_pages - pstart);
  const int nsteps = (npg + 1) / 2;
  const bool single = r.n_split == 1;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t qs = base + ns * kStep;
  const uint32_t red_off = ns * kStep + NG * kQTile;
  const uint32_t bars = base + red_off + 2 * NG * kRedBytes;
  auto full = [&](int i) { return bars + 8u * i; };
  auto empty = [&](int i) { return bars + 8u * (ns + i); };
  auto xchg = [&](int g, int k) { return bars + 8u * (2 * ns + 2 * g + k); };
  int32_t* phys_s = reinterpret_cast<int32_t*>(gbase + red_off + 2 * NG * kRedBytes +
                                               8 * (2 * ns + 2 * NG));
  int32_t* tab_s = phys_s + 2 * ns;
  volatile int32_t* abort_s = tab_s + chunk;

  if (threadIdx.x == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), NW);
    }
    for (int i = 0; i < 2 * NG; ++i) mbar_init(bars + 8u * (2 * ns + i), 128);
    *abort_s = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < npg; i += blockDim.x)
    tab_s[i] = a.table[static_cast<int64_t>(b) * a.max_blocks + pstart + i];
  // the CTA's query rows (absent heads are zero rows), swizzled like the cache
  {
    const uint4* q = static_cast<const uint4*>(a.q);
    for (int i = threadIdx.x; i < 16 * NG * (kMlaRow / 8); i += blockDim.x) {
      const int row = i / (kMlaRow / 8), c = i % (kMlaRow / 8);
      const int h = h0 + row;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (h < a.H) v = q[(static_cast<int64_t>(b) * a.H + h) * (kMlaRow / 8) + c];
      *reinterpret_cast<uint4*>(gbase + (swz_addr(qs + (row >> 4) * kQTile, 16 * 128, row & 15, c) -
                                         base)) = v;
    }
  }
  __syncthreads();

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&cmap);
      int issued = 0;
      uint32_t loaded = 0;  // stages whose last fill had copies in flight
      for (int i = 0; i < nsteps; ++i) {
        const int st = i % ns, u = i / ns;
        if (u > 0 && !mbar_wait(empty(st), (u - 1) & 1, a.wait_ns)) {
          raise_err(a.err, kDevErrTimeout);
          *abort_s = 1;
          break;
        }
        if (*abort_s) break;
        int ph[2];
        uint32_t bytes = 0;
#pragma unroll
        for (int pg = 0; pg < 2; ++pg) {
          ph[pg] = -1;
          const int idx = 2 * i + pg;
          if (idx < npg) {
            const int phys = tab_s[idx];
            if (phys >= 0 && phys < a.num_blocks) {
              ph[pg] = phys;
              bytes += kPage;
            } else {
              raise_err(a.err, kDevErrBadBlock);
            }
          }
          phys_s[2 * st + pg] = ph[pg];
        }
        if (bytes) {
          mbar_arrive_expect_tx(full(st), bytes);
          const uint32_t sb = base + st * kStep;
#pragma unroll
          for (int pg = 0; pg < 2; ++pg)
            if (ph[pg] >= 0) tma_load_4d(sb + pg * kPage, &cmap, full(st), 0, 0, 0, ph[pg]);
          loaded |= 1u << st;
        } else {
          loaded &= ~(1u << st);
          mbar_arrive(full(st));
        }
        issued = i + 1;
      }
      // no copy may land after the CTA exits
      for (int i = issued - ns > 0 ? issued - ns : 0; i < issued; ++i) {
        const int st = i % ns;
        if (loaded & (1u << st)) mbar_wait(full(st), (i / ns) & 1, 100000000ull);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = warp >> 2, wk = warp & 3;
  const int nrows = min(16, a.H - (h0 + 16 * g));
  const int gr = lane >> 2, tq = lane & 3;
  const int mi = lane >> 3, rr = lane & 7;
  const int arow = rr + ((mi & 1) << 3);        // query row this lane addresses
  const int ktok = ((mi >> 1) << 3) + rr;       // key row for the score fragments
  const int vtok = ((mi & 1) << 3) + rr;        // key row for the (transposed) value fragments
  const uint32_t qg = qs + g * kQTile;
  const float sl2 = a.scale_log2;
  float* red = reinterpret_cast<float*>(gbase + red_off);

  float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;
  float acc[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  for (int i = 0; i < nsteps; ++i) {
    const int st = i % ns;
    // warp-uniform: the ldmatrix / mma.sync below need all 32 lanes
    const bool got = __all_sync(0xFFFFFFFFu, mbar_wait(full(st), (i / ns) & 1, a.wait_ns));
    if (!got && lane == 0) {
      raise_err(a.err, kDevErrTimeout);
      *abort_s = 1;
    }
    const int ph0 = got ? phys_s[2 * st] : -1, ph1 = got ? phys_s[2 * st + 1] : -1;
    const uint32_t sb = base + st * kStep;

    // partial scores over this warp's 144 of the 576 dims
    float sc[4][4];
#pragma unroll
    for (int t = 0; t < 4; ++t) sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
    if (got) {
#pragma unroll
      for (int kk = 0; kk < 9; ++kk) {
        const int kg = 9 * wk + kk;
        uint32_t qa[4];
        ldsm_x4(swz_addr(qg, 16 * 128, arow, 2 * kg + (mi >> 1)), qa[0], qa[1], qa[2], qa[3]);
#pragma unroll
        for (int pg = 0; pg < 2; ++pg) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(swz_addr(sb + pg * kPage, kPanelBytes, ktok, 2 * kg + (mi & 1)), b0, b1, b2,
                  b3);
          mma_bf16_16816(sc[2 * pg], qa, b0, b1);
          mma_bf16_16816(sc[2 * pg + 1], qa, b2, b3);
        }
      }
    }
    // sum the group's four partials (fixed order: every warp gets the same
    // bits) through a double-buffered exchange with a bounded wait
    const int buf = i & 1;
    float* rb = red + (buf * NG + g) * (kRedBytes / 4);
#pragma unroll
    for (int t = 0; t < 4; ++t)
      *reinterpret_cast<float4*>(rb + ((wk * 4 + t) * 32 + lane) * 4) =
          make_float4(sc[t][0], sc[t][1], sc[t][2], sc[t][3]);
    mbar_arrive(xchg(g, buf));
    const bool synced = mbar_wait(xchg(g, buf), (i >> 1) & 1, a.wait_ns);
    if (!synced && lane == 0) {
      raise_err(a.err, kDevErrTimeout);
      *abort_s = 1;
    }
    if (!__all_sync(0xFFFFFFFFu, got && synced)) break;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      float4 v = *reinterpret_cast<const float4*>(rb + ((0 * 4 + t) * 32 + lane) * 4);
#pragma unroll
      for (int w = 1; w < 4; ++w) {
        const float4 x = *reinterpret_cast<const float4*>(rb + ((w * 4 + t) * 32 + lane) * 4);
        v.x += x.x;
        v.y += x.y;
        v.z += x.z;
        v.w += x.w;
      }
      sc[t][0] = v.x;
      sc[t][1] = v.y;
      sc[t][2] = v.z;
      sc[t][3] = v.w;
    }

    // keys outside the sequence or in a skipped block
    const int tok0 = (pstart + 2 * i) * kBlk;
    uint32_t mlo[2] = {0xFFFFFFFFu, 0xFFFFFFFFu}, mhi[2] = {0xFFFFFFFFu, 0xFFFFFFFFu};
    if (tok0 + 2 * kBlk > r.len || ph0 < 0 || ph1 < 0) {
      auto ok = [&](int tok) {
        return tok < r.len && (tok - tok0 < kBlk ? ph0 >= 0 : ph1 >= 0);
      };
#pragma unroll
      for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (!ok(tok0 + 8 * t + 2 * tq + (e & 1))) sc[t][e] = kNegInf;
#pragma unroll
      for (int pg = 0; pg < 2; ++pg) {
        const int ta = tok0 + kBlk * pg + 2 * tq, tb = ta + 8;
        mlo[pg] = (ok(ta) ? 0x0000FFFFu : 0u) | (ok(ta + 1) ? 0xFFFF0000u : 0u);
        mhi[pg] = (ok(tb) ? 0x0000FFFFu : 0u) | (ok(tb + 1) ? 0xFFFF0000u : 0u);
      }
    }

    // online softmax (log2 domain), rows gr (e = 0,1) and gr + 8 (e = 2,3)
    float mx0 = kNegInf, mx1 = kNegInf;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      mx0 = fmaxf(mx0, fmaxf(sc[t][0], sc[t][1]));
      mx1 = fmaxf(mx1, fmaxf(sc[t][2], sc[t][3]));
    }
    mx0 *= sl2;
    mx1 *= sl2;
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
    float ps[4][4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      ps[t][0] = ex2(fmaf(sc[t][0], sl2, -mu0));
      ps[t][1] = ex2(fmaf(sc[t][1], sl2, -mu0));
      ps[t][2] = ex2(fmaf(sc[t][2], sl2, -mu1));
      ps[t][3] = ex2(fmaf(sc[t][3], sl2, -mu1));
    }
    l0 = l0 * al0 + ((ps[0][0] + ps[0][1]) + (ps[1][0] + ps[1][1])) +
         ((ps[2][0] + ps[2][1]) + (ps[3][0] + ps[3][1]));
    l1 = l1 * al1 + ((ps[0][2] + ps[0][3]) + (ps[1][2] + ps[1][3])) +
         ((ps[2][2] + ps[2][3]) + (ps[3][2] + ps[3][3]));
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      acc[j][0] *= al0;
      acc[j][1] *= al0;
      acc[j][2] *= al1;
      acc[j][3] *= al1;
    }

    // O += P C over this warp's latent dims 128*wk.., block by block
#pragma unroll
    for (int pg = 0; pg < 2; ++pg) {
      if ((pg ? ph1 : ph0) < 0) continue;
      const uint32_t pa[4] = {pack_bf16(ps[2 * pg][0], ps[2 * pg][1]),
                              pack_bf16(ps[2 * pg][2], ps[2 * pg][3]),
                              pack_bf16(ps[2 * pg + 1][0], ps[2 * pg + 1][1]),
                              pack_bf16(ps[2 * pg + 1][2], ps[2 * pg + 1][3])};
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(swz_addr(sb + pg * kPage, kPanelBytes, vtok, 16 * wk + 2 * jj + (mi >> 1)), v0,
                  v1, v2, v3);
        mma_bf16_16816(acc[2 * jj], pa, v0 & mlo[pg], v1 & mhi[pg]);
        mma_bf16_16816(acc[2 * jj + 1], pa, v2 & mlo[pg], v3 & mhi[pg]);
      }
    }
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
    const int h = h0 + 16 * g + row;
    const float l = half ? l1 : l0;
    const float m = half ? m1 : m0;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse_v = l > 0.f ? (m + log2f(l)) * kLn2 : kNegInf;
    const int64_t bh = static_cast<int64_t>(b) * a.H + h;
    if (single) {
      uint32_t* o32 = static_cast<uint32_t*>(a.o) + bh * (kMlaDc / 2) + 64 * wk;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        o32[j * 4 + tq] = pack_bf16(acc[j][2 * half] * inv, acc[j][2 * half + 1] * inv);
      if (wk == 0 && tq == 0 && a.lse) a.lse[h * a.B + b] = lse_v;
    } else {
      float2* w = reinterpret_cast<float2*>(a.ws_o + (bh * num_splits + s) * kMlaDc + 128 * wk);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        w[j * 4 + tq] = make_float2(acc[j][2 * half] * inv, acc[j][2 * half + 1] * inv);
      if (wk == 0 && tq == 0) a.ws_lse[bh * num_splits + s] = lse_v;
    }
  }
}

// ------------------------------------------------------------------ merge
// lse = ln sum_s e^{lse_s}; o = sum_s e^{lse_s - lse} o_s. One warp per
// (sequence, head), 16 latent dims per lane; single-range sequences were
// finished by the decode kernel.
__global__ void __launch_bounds__(256) mla_merge_kernel(const MlaArgs a, const int chunk,
                                                        const int num_splits) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int idx = blockIdx.x * 8 + warp;
  if (idx >= a.B * a.H) return;
  const int b = idx / a.H, h = idx % a.H;
  const MlaRange r = mla_range(a.seq_lens[b], a.max_blocks, chunk, a.err, false);
  if (r.n_split <= 1) return;
  const float* ls = a.ws_lse + static_cast<int64_t>(idx) * num_splits;
  float mx = kNegInf;
  for (int i = lane; i < r.n_split; i += 32) mx = fmaxf(mx, ls[i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  float acc[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) acc[c] = 0.f;
  float total = 0.f;
  // lane owns dims 4*lane + 128*k (k = 0..3): each float4 load of the warp is 512 contiguous bytes
  const float* wo = a.ws_o + static_cast<int64_t>(idx) * num_splits * kMlaDc + 4 * lane;
  for (int i = 0; i < r.n_split; ++i) {
    float4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      v[k] = *reinterpret_cast<const float4*>(wo + static_cast<int64_t>(i) * kMlaDc + 128 * k);
    const float w = expf(ls[i] - mx);
    total += w;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc[4 * k] = fmaf(w, v[k].x, acc[4 * k]);
      acc[4 * k + 1] = fmaf(w, v[k].y, acc[4 * k + 1]);
      acc[4 * k + 2] = fmaf(w, v[k].z, acc[4 * k + 2]);
      acc[4 * k + 3] = fmaf(w, v[k].w, acc[4 * k + 3]);
    }
  }
  const float inv = 1.f / total;
  uint2* o = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.o) +
                                      static_cast<int64_t>(idx) * kMlaDc + 4 * lane);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    o[32 * k] = make_uint2(pack_bf16(acc[4 * k] * inv, acc[4 * k + 1] * inv),
                           pack_bf16(acc[4 * k + 2] * inv, acc[4 * k + 3] * inv));
  if (lane == 0 && a.lse) a.lse[h * a.B + b] = mx + logf(total);
}

int g_mla_attr[2][64];

template <int NG>
void ensure_mla_attr(size_t bytes) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (g_mla_attr[NG - 1][dev] < static_cast<int>(bytes)) {
    cudaFuncSetAttribute(mla_decode_kernel<NG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(bytes));
    g_mla_attr[NG - 1][dev] = static_cast<int>(bytes);
  }
}

}  // namespace

MlaPlan plan_mla_decode(int B, int H, int max_blocks, int num_splits_req, int sm_count) {
  MlaPlan p{};
  const int sms = sm_count > 0 ? sm_count : 148;
  p.ng = H <= 16 ? 1 : 2;
  p.head_chunks = (H + 16 * p.ng - 1) / (16 * p.ng);
  p.stages = 2;
  p.threads = (4 * p.ng + 1) * 32;
  const int eff = max_blocks < 1 ? 1 : max_blocks;
  int chunk;
  if (num_splits_req > 0) {
    chunk = (eff + num_splits_req - 1) / num_splits_req;
  } else {
    // ranges sized so that, were every sequence as long as the table, the
    // call would fill the CTA slots (two per SM for 16 heads, one for 32)
    // about 3.5 times: sequences of mixed lengths then leave about two
    // waves, short enough a tail; at least 8 blocks per range
    const long long units = static_cast<long long>(B) * p.head_chunks;
    const long long slots = static_cast<long long>(sms) * (p.ng == 1 ? 2 : 1);
    long long c = (units * eff * 2 + 7 * slots - 1) / (7 * slots);
    if (c < 8) c = 8;
    chunk = static_cast<int>(c);
  }
  if (chunk > eff) chunk = eff;
  if (chunk < 1) chunk = 1;
  p.chunk = chunk;
  p.num_splits = (eff + chunk - 1) / chunk;
  p.smem = 1024 + static_cast<size_t>(p.stages) * kStep + static_cast<size_t>(p.ng) * kQTile +
           2ull * p.ng * kRedBytes + 8ull * (2 * p.stages + 2 * p.ng) + 4ull * 2 * p.stages +
           4ull * chunk + 16;
  if (p.num_splits > 1) {
    const size_t n = static_cast<size_t>(B) * H * p.num_splits;
    p.workspace = (n * kMlaDc * 4 + 255) / 256 * 256 + (n * 4 + 255) / 256 * 256;
  } else {
    p.workspace = 0;
  }
  return p;
}

cudaError_t launch_mla_decode_bf16(const MlaArgs& a, const MlaPlan& p, const CUtensorMap& cmap,
                                   cudaStream_t s) {
  const dim3 grid(p.num_splits, p.head_chunks, a.B);
  if (p.ng == 1) {
    ensure_mla_attr<1>(p.smem);
    mla_decode_kernel<1><<<grid, p.threads, p.smem, s>>>(cmap, a, p.chunk, p.num_splits,
                                                         p.stages);
  } else {
    ensure_mla_attr<2>(p.smem);
    mla_decode_kernel<2><<<grid, p.threads, p.smem, s>>>(cmap, a, p.chunk, p.num_splits,
                                                         p.stages);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.num_splits <= 1) return e;
  // programmatic dependent launch: the merge's launch overlaps the decode's tail
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.B * a.H + 7) / 8);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_merge_kernel, a, p.chunk, p.num_splits);
}

}  // namespace pa
