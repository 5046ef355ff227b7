// attn_prefill: exact causal / sliding-window / full attention of packed
// sequences, computed tile by tile so the score matrix never leaves the SM.
//
// Sources: the tiled loop -- for each query tile, stream K/V tiles, compute
// S = Q K^T, fold it into a running softmax, accumulate into the output tile,
// write the output once ("Cache KV, atención flash y optimización de la
// inferencia", section "La atención de flash el truco de la balsa"); the
// running (max, sum) with rescaling by e^{m_old - m_new} ("Ли Хунъи ... 2026",
// lecture "Ускоряем генерацию, часть 1: FlashAttention", and "Module 09:
// Efficient Attention", section "FlashAttention: The Compute Wall"); masks as
// in "Генерация и KV-кэш" (np.tril, causal) and "Module 09: Efficient
// Attention", section "Attention Mask Gallery" (sliding window, diagonal
// included); GQA head mapping as in the notebook's section "The Math: Sharing
// Keys and Values".
//
// sm_103a design (one 128-row query tile of one head per CTA):
//  * warp 0, one thread: TMA producer. Q tile once; K and V tiles of 128 keys
//    through a `NS`-deep ring. Every tile is stored as 64-element (128-byte)
//    panels, 128-byte swizzled, which is the K-major / MN-major operand layout
//    the tensor cores read directly.
//  * warp 1, one thread: tcgen05.mma issuer. S_j = Q K_j^T (M=128, N=128,
//    bf16 x bf16 -> fp32) into one of two TMEM score buffers, then
//    O += P_{j-1} V_{j-1} (M=128, N=d) into a TMEM accumulator, so the tensor
//    cores compute the next scores while the softmax works on the current ones.
//    Completion is signalled with tcgen05.commit on mbarriers.
//  * warps 2-5 (128 threads, one query row each): load the row's scores from
//    TMEM, mask only on tiles that straddle the diagonal, the window edge or
//    the sequence end, update the running max in the log2 domain with
//    scale*log2(e) folded into one FMA, exponentiate with ex2, write P (bf16)
//    to shared memory in the swizzled A-operand layout, and at the end read O
//    back from TMEM, divide by the running sum and store O and the LSE.
//  * The max is rescaled lazily: O and the sum are only rescaled when the max
//    grows by more than 2^8, otherwise the stale max is kept. The final O / sum
//    is unchanged (both carry the same factor), P stays <= 256, and TMEM
//    round trips of O become rare.
//  * Tiles above the diagonal or left of the window are never loaded; CTAs
//    are launched heaviest query tile first to even out the causal triangle.
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pa_kernels.h"
#include "pa_ptx.cuh"

namespace pa {

namespace {

constexpr int BM = 128;  // query rows per tile (= TMEM lanes)
constexpr int BN = 128;  // keys per tile
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kNegInf = -INFINITY;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows > 256x

template <int D>
struct PfCfg {
  static constexpr int P = D / 64;                   // 128-byte panels per row
  static constexpr int NS = (D == 128) ? 2 : 4;      // K/V ring depth
  static constexpr int QB = BM * D * 2;              // Q tile bytes
  static constexpr int KB = BN * D * 2;              // one K (or V) tile
  static constexpr int PB = BM * BN * 2;             // P tile (bf16)
  static constexpr int QPANEL = BM * 128;            // bytes per Q / P panel
  static constexpr int KPANEL = BN * 128;            // bytes per K / V panel
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QB;
  static constexpr int OFF_V = OFF_K + NS * KB;
  static constexpr int OFF_P = OFF_V + NS * KB;
  static constexpr int OFF_BAR = OFF_P + PB;
  // barriers
  static constexpr int B_QFULL = 0;
  static constexpr int B_KFULL = 1;                  // + stage
  static constexpr int B_KEMPTY = 1 + NS;
  static constexpr int B_VFULL = 1 + 2 * NS;
  static constexpr int B_VEMPTY = 1 + 3 * NS;
  static constexpr int B_SFULL = 1 + 4 * NS;         // + buffer (2)
  static constexpr int B_SFREE = 3 + 4 * NS;         // + buffer (2)
  static constexpr int B_PFULL = 5 + 4 * NS;
  static constexpr int B_ODONE = 6 + 4 * NS;
  static constexpr int B_DRAIN = 7 + 4 * NS;
  static constexpr int NBAR = 8 + 4 * NS;
  static constexpr int SMEM = 1024 + OFF_BAR + NBAR * 8 + 16;
  static constexpr uint32_t TMEM_COLS = 512;         // S0 | S1 | O
  static constexpr uint32_t TM_S0 = 0, TM_S1 = BN, TM_O = 2 * BN;
};

template <int D>
__global__ void __launch_bounds__(192, 1)
prefill_bf16_kernel(const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  using C = PfCfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ------------------------------------------------------- tile -> work item
  const int n_qt = (a.max_seqlen + BM - 1) / BM;
  const int per = a.Hq * a.B;
  const int qt_r = blockIdx.x / per, hb = blockIdx.x % per;
  const int h = hb % a.Hq, b = hb / a.Hq;
  const int qt = a.causal ? (n_qt - 1 - qt_r) : qt_r;  // heaviest tiles first
  int start, len;
  if (a.cu_seqlens) {
    start = a.cu_seqlens[b];
    len = a.cu_seqlens[b + 1] - start;
  } else {
    start = b * a.N;
    len = a.N;
  }
  const int q0 = qt * BM;
  if (q0 >= len) return;
  const int rows = min(BM, len - q0);
  const int q_last = q0 + rows - 1;
  const int kv_end = a.causal ? q_last + 1 : len;
  const int kv_begin = a.window > 0 ? max(0, q0 - a.window + 1) : 0;
  const int t_begin = kv_begin / BN;
  const int n_tiles = (kv_end + BN - 1) / BN - t_begin;
  const int kvh = h / (a.Hq / a.Hkv);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  const uint32_t sQ = base + C::OFF_Q, sK = base + C::OFF_K, sV = base + C::OFF_V,
                 sP = base + C::OFF_P;
  const uint32_t bar0 = base + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (warp == 1) {
    if (lane == 0) {
      mbar_init(bar(C::B_QFULL), 1);
      for (int i = 0; i < C::NS; ++i) {
        mbar_init(bar(C::B_KFULL + i), 1);
        mbar_init(bar(C::B_KEMPTY + i), 1);
        mbar_init(bar(C::B_VFULL + i), 1);
        mbar_init(bar(C::B_VEMPTY + i), 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(bar(C::B_SFULL + i), 1);
        mbar_init(bar(C::B_SFREE + i), 128);
      }
      mbar_init(bar(C::B_PFULL), 128);
      mbar_init(bar(C::B_ODONE), 1);
      mbar_init(bar(C::B_DRAIN), 1);
      *abort_flag = 0;
      fence_mbar_init();
    }
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&qmap);
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
      mbar_arrive_expect_tx(bar(C::B_QFULL), C::QB);
#pragma unroll
      for (int p = 0; p < C::P; ++p)
        tma_load_3d(sQ + p * C::QPANEL, &qmap, bar(C::B_QFULL), p * 64, h, start + q0);
      int issued = 0;
      for (int it = 0; it < n_tiles; ++it) {
        const int st = it % C::NS, u = it / C::NS;
        const int krow = start + (t_begin + it) * BN;
        if (u > 0 && !mbar_wait(bar(C::B_KEMPTY + st), (u - 1) & 1)) break;
        mbar_arrive_expect_tx(bar(C::B_KFULL + st), C::KB);
#pragma unroll
        for (int p = 0; p < C::P; ++p)
          tma_load_3d(sK + st * C::KB + p * C::KPANEL, &kmap, bar(C::B_KFULL + st), p * 64, kvh,
                      krow);
        if (u > 0 && !mbar_wait(bar(C::B_VEMPTY + st), (u - 1) & 1)) {
          issued = -(it + 1);  // K of this tile issued, V not
          break;
        }
        mbar_arrive_expect_tx(bar(C::B_VFULL + st), C::KB);
#pragma unroll
        for (int p = 0; p < C::P; ++p)
          tma_load_3d(sV + st * C::KB + p * C::KPANEL, &vmap, bar(C::B_VFULL + st), p * 64, kvh,
                      krow);
        issued = it + 1;
        if (*abort_flag) break;
      }
      if (issued < n_tiles) {
        // abandoned: record it and let every copy in flight land before exit
        raise_err(a.err, kDevErrTimeout);
        *abort_flag = 1;
        const int nk = issued < 0 ? -issued : issued;
        const int nv = issued < 0 ? nk - 1 : issued;
        mbar_wait(bar(C::B_QFULL), 0, 100000000ull);
        for (int i = nk - C::NS > 0 ? nk - C::NS : 0; i < nk; ++i)
          mbar_wait(bar(C::B_KFULL + i % C::NS), (i / C::NS) & 1, 100000000ull);
        for (int i = nv - C::NS > 0 ? nv - C::NS : 0; i < nv; ++i)
          mbar_wait(bar(C::B_VFULL + i % C::NS), (i / C::NS) & 1, 100000000ull);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc_bf16_f32(BM, BN, 0, 0);
      constexpr uint32_t idesc_pv = umma_idesc_bf16_f32(BM, D, 0, 1);
      auto issue_pv = [&](int j) -> bool {
        const int st = j % C::NS, u = j / C::NS;
        if (!mbar_wait(bar(C::B_PFULL), j & 1)) return false;
        if (!mbar_wait(bar(C::B_VFULL + st), u & 1)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // A = P tile, K-major: 16 keys = 32 bytes inside a 128-byte panel row.
          const uint64_t ad =
              umma_smem_desc_sw128(sP + (kk >> 2) * C::QPANEL + (kk & 3) * 32, 16, 1024);
          // B = V tile, MN-major (d contiguous): 16 keys = 16 rows of 128 bytes;
          // panels of 64 d-columns are KPANEL bytes apart.
          const uint64_t bd =
              umma_smem_desc_sw128(sV + st * C::KB + kk * 16 * 128, C::KPANEL, 1024);
          umma_ss(tmem + C::TM_O, ad, bd, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(C::B_VEMPTY + st));
        umma_commit(bar(C::B_ODONE));
        return true;
      };
      bool ok = mbar_wait(bar(C::B_QFULL), 0);
      tc_fence_after();
      for (int it = 0; ok && it < n_tiles; ++it) {
        const int st = it % C::NS, u = it / C::NS, sb = it & 1;
        if (!mbar_wait(bar(C::B_KFULL + st), u & 1)) { ok = false; break; }
        if (it >= 2 && !mbar_wait(bar(C::B_SFREE + sb), ((it >> 1) - 1) & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off_q = (kk >> 2) * C::QPANEL + (kk & 3) * 32;
          const uint32_t off_k = (kk >> 2) * C::KPANEL + (kk & 3) * 32;
          const uint64_t ad = umma_smem_desc_sw128(sQ + off_q, 16, 1024);
          const uint64_t bd = umma_smem_desc_sw128(sK + st * C::KB + off_k, 16, 1024);
          umma_ss(tmem + (sb ? C::TM_S1 : C::TM_S0), ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(C::B_KEMPTY + st));
        umma_commit(bar(C::B_SFULL + sb));
        if (it >= 1) ok = issue_pv(it - 1);
      }
      if (ok) ok = issue_pv(n_tiles - 1);
      if (!ok) {
        raise_err(a.err, kDevErrTimeout);
        *abort_flag = 1;
      }
      // every MMA issued above has finished once this commit arrives
      umma_commit(bar(C::B_DRAIN));
      mbar_wait(bar(C::B_DRAIN), 0, 100000000ull);
    }
  } else {
    // ------------------------------------------------ softmax / epilogue
    const int wq = warp & 3;               // TMEM lane quarter of this warp
    const int r = wq * 32 + lane;          // row of the query tile
    const int i_abs = q0 + r;              // query position in its sequence
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = a.scale_log2;
    float m = kNegInf, l = 0.f;
    bool ok = true;
    for (int it = 0; it < n_tiles; ++it) {
      const int sb = it & 1;
      const int kt0 = (t_begin + it) * BN;
      if (!mbar_wait(bar(C::B_SFULL + sb), (it >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
        tmem_ld32(tmem + lane_off + (sb ? C::TM_S1 : C::TM_S0) + 32 * c,
                  *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(C::B_SFREE + sb));

      const bool need_mask = (kt0 + BN > len) || (a.causal && kt0 + BN - 1 > q0) ||
                             (a.window > 0 && kt0 <= q_last - a.window);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const int j = kt0 + c;
          const bool vis = j < len && (!a.causal || j <= i_abs) &&
                           (a.window <= 0 || j > i_abs - a.window);
          if (!vis) sr[c] = __float_as_uint(kNegInf);
        }
      }
      float mx = kNegInf;
#pragma unroll
      for (int c = 0; c < BN; ++c) mx = fmaxf(mx, __uint_as_float(sr[c]));
      const float m_new = fmaxf(m, mx * sl2);
      const bool resc = m_new > m + kRescaleThreshold;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2(m - m_new);  // 0 when m = -inf
        m = m_new;
      }
      if (it > 0) {
        // PV of the previous tile must be done before O is touched or P reused
        if (!mbar_wait(bar(C::B_ODONE), (it - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xFFFFFFFFu, resc)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + C::TM_O + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tmem + lane_off + C::TM_O + 32 * c, o);
          }
          tmem_wait_st();
        }
      }
      l *= alpha;
      const float m_use = m == kNegInf ? 0.f : m;
      float lsum = 0.f;
#pragma unroll
      for (int c = 0; c < BN / 8; ++c) {
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          p[e] = ex2(fmaf(__uint_as_float(sr[8 * c + e]), sl2, -m_use));
          lsum += p[e];
        }
        const uint32_t addr = sP + (c >> 3) * C::QPANEL + r * 128 + (((c & 7) ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                     "r"(pack_bf16(p[0], p[1])), "r"(pack_bf16(p[2], p[3])),
                     "r"(pack_bf16(p[4], p[5])), "r"(pack_bf16(p[6], p[7]))
                     : "memory");
      }
      l += lsum;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::B_PFULL));
    }
    if (ok && mbar_wait(bar(C::B_ODONE), (n_tiles - 1) & 1)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.o) +
                            (static_cast<int64_t>(start + i_abs) * a.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + C::TM_O + 32 * c, o);
        tmem_wait_ld();
        if (r < rows) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
            dst[v] = w;
          }
        }
      }
      if (a.lse && r < rows)
        a.lse[static_cast<int64_t>(h) * a.T + start + i_abs] =
            l > 0.f ? (m + log2f(l)) * kLn2 : kNegInf;
    } else {
      raise_err(a.err, kDevErrTimeout);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// --------------------------------------------------------------- fp32 path
// CUDA-core path for fp32 inputs: one warp per (token, query head); keys are
// visited one at a time with the same running (max, sum) recurrence.
template <int D>
__global__ void __launch_bounds__(128) prefill_f32_kernel(const PrefillArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * 4 + warp;
  if (idx >= static_cast<int64_t>(a.T) * a.Hq) return;
  const int tok = static_cast<int>(idx / a.Hq), h = static_cast<int>(idx % a.Hq);
  int start, len;
  if (a.cu_seqlens) {
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.cu_seqlens[mid] <= tok) lo = mid; else hi = mid - 1;
    }
    start = a.cu_seqlens[lo];
    len = a.cu_seqlens[lo + 1] - start;
  } else {
    start = (tok / a.N) * a.N;
    len = a.N;
  }
  const int i = tok - start;
  const int j_end = a.causal ? i + 1 : len;
  const int j_begin = a.window > 0 ? max(0, i - a.window + 1) : 0;
  const int g = h / (a.Hq / a.Hkv);
  const float* q = static_cast<const float*>(a.q) + (static_cast<int64_t>(tok) * a.Hq + h) * D;
  const float* k = static_cast<const float*>(a.k);
  const float* v = static_cast<const float*>(a.v);
  float qv[D / 32], acc[D / 32];
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    qv[c] = q[lane + 32 * c];
    acc[c] = 0.f;
  }
  float m = kNegInf, l = 0.f;
  for (int j = j_begin; j < j_end; ++j) {
    const int64_t row = (static_cast<int64_t>(start + j) * a.Hkv + g) * D;
    float dot = 0.f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) dot = fmaf(qv[c], k[row + lane + 32 * c], dot);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, off);
    const float s2 = dot * a.scale_log2;
    const float mn = fmaxf(m, s2);
    const float al = ex2(m - mn);
    const float p = ex2(s2 - mn);
    l = l * al + p;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) acc[c] = fmaf(p, v[row + lane + 32 * c], acc[c] * al);
    m = mn;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  float* o = static_cast<float*>(a.o) + (static_cast<int64_t>(tok) * a.Hq + h) * D;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) o[lane + 32 * c] = acc[c] * inv;
  if (lane == 0 && a.lse)
    a.lse[static_cast<int64_t>(h) * a.T + tok] = l > 0.f ? (m + log2f(l)) * kLn2 : kNegInf;
}

int g_pf_attr[2][64];

template <int D>
void ensure_pf_attr() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!g_pf_attr[D == 128][dev]) {
    cudaFuncSetAttribute(prefill_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         PfCfg<D>::SMEM);
    g_pf_attr[D == 128][dev] = 1;
  }
}

}  // namespace

size_t prefill_bf16_smem(int d) { return d == 128 ? PfCfg<128>::SMEM : PfCfg<64>::SMEM; }

cudaError_t launch_prefill_bf16(const PrefillArgs& a, const CUtensorMap& qmap,
                                const CUtensorMap& kmap, const CUtensorMap& vmap,
                                cudaStream_t s) {
  const int n_qt = (a.max_seqlen + BM - 1) / BM;
  const long long grid = static_cast<long long>(n_qt) * a.Hq * a.B;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  if (a.d == 128) {
    ensure_pf_attr<128>();
    prefill_bf16_kernel<128><<<static_cast<unsigned>(grid), 192, PfCfg<128>::SMEM, s>>>(qmap, kmap, vmap, a);
  } else {
    ensure_pf_attr<64>();
    prefill_bf16_kernel<64><<<static_cast<unsigned>(grid), 192, PfCfg<64>::SMEM, s>>>(qmap, kmap, vmap, a);
  }
  return cudaGetLastError();
}

cudaError_t launch_prefill_f32(const PrefillArgs& a, cudaStream_t s) {
  const long long warps = static_cast<long long>(a.T) * a.Hq;
  if (warps == 0) return cudaSuccess;
  const long long blocks = (warps + 3) / 4;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  if (a.d == 128)
    prefill_f32_kernel<128><<<static_cast<unsigned>(blocks), 128, 0, s>>>(a);
  else
    prefill_f32_kernel<64><<<static_cast<unsigned>(blocks), 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace pa
