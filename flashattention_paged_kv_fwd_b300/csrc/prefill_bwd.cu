// attn_prefill_backward: gradients dQ, dK, dV of exact attention of packed
// sequences (causal / sliding-window / full, GQA), recomputing the scores
// from Q, K and the forward pass's per-row log-sum-exp instead of storing the
// attention matrix.
//
// Sources: the backward pass recomputes forward values rather than storing
// them ("Cache KV, atención flash y optimización de la inferencia", section
// "La atención de flash el truco de la balsa"); the gradients themselves are
// the chain rule through O = softmax(S) V, S = scale * Q K^T:
//     P = exp(S - lse),  dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,
//     dS = P * (dP - D),  dQ = scale * dS K,  dK = scale * dS^T Q;
// masks and GQA mapping as in the forward pass.
//
// sm_103a design. Three kernels and a memset:
//  1. D = rowsum(dO * O) per (token, query head) (one warp each).
//  2. The main kernel, a persistent grid of one CTA per SM over work units
//     (key tile of 128 keys, KV head, sequence), key tiles nearest the start
//     first (under a causal mask they see the most query tiles). A unit keeps
//     its K and V tile in shared memory and its dK, dV accumulators in TMEM,
//     and streams the query tiles (128 rows) of every query head of the KV
//     group that can see its keys. Per query tile, five tcgen05 MMAs:
//        S^T  = K Q^T            M=128 keys, N=128 queries, K=d   (SS)
//        dP^T = V dO^T           same shape                       (SS)
//        dV  += P^T dO           A = P^T read from TMEM           (TS)
//        dK  += dS^T Q           A = dS^T from shared memory      (SS)
//        dQ   = dS K             M=128 queries, A = dS^T read MN-major
//     Everything is kept transposed (keys on TMEM lanes) so dV and dK
//     accumulate in place; dQ of the tile is added into an fp32 buffer
//     [T, Hq, d] by bulk tensor reduce-adds (performed in L2).
//      * warp 8 (TMA producer): K, V once per unit; Q, dO and the rows'
//        -lse*log2(e) and -D through two stages.
//      * warp 9 (tcgen05 issuer): per tile dP (once the previous tile's dQ
//        has left the TMEM columns it reuses), dV (two halves, as the halves
//        of P arrive), S of the next tile (when its Q has landed), then dK
//        and dQ once dS is in shared memory.
//      * warps 0-7 (warp (wq, ch): key rows 32*wq.. = its TMEM lane quarter,
//        query columns 64*ch..), per tile s:
//          P(s) = 2^(S*scale*log2 e - lse*log2 e), written as bf16 into the S
//            columns it came from (the A operand of dV);
//          the read-out of dQ(s-1): TMEM -> registers (freeing the columns
//            dP(s) needs) -> this warp's rows of the dS^T tile, 128-byte
//            swizzled -> bulk tensor reduce-add;
//          dS(s) = P (dP - D), written as bf16 into the 128-byte-swizzled dS^T
//            tile, the operand layout of both the dK and the dQ MMA, once the
//            copies of the staged dQ have read it.
//        At the end of a unit they write dK (times scale) and dV as bf16.
//     TMEM (512 columns): S^T / P at 0, dP^T at 128 (dQ reuses these columns
//     once dS has been formed), dV at 256, dK at 256 + d.
//  3. dQ = scale * buffer, converted to bf16.
// All waits are bounded; a wait that gives up raises PA_DEV_TIMEOUT and every
// role winds down, waiting for its copies and MMAs in flight before TMEM is
// freed.
#include <climits>
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bwd_kernels.h"
#include "pa_ptx.cuh"

namespace pa {

namespace {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per tile (TMEM lanes of S^T, dP^T, dV, dK)
constexpr float kLog2e = 1.4426950408889634074f;

constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;  // 8 softmax / gradient warps, producer, MMA issuer

constexpr uint64_t kDrainLimitNs = 100000000ull;  // 0.1 s for copies / MMAs already in flight

template <int D>
struct BwCfg {
  static constexpr int TB = 128 * D * 2;    // one 128-row tile of Q, K, V or dO
  static constexpr int PANEL = 128 * 128;   // one 64-column panel of a 128-row tile
  static constexpr int DSB = BN * BM * 2;   // dS^T: 128 keys x 128 queries, bf16
  static constexpr int NST = 2;             // Q / dO stages
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TB;
  static constexpr int OFF_DS = 2 * TB;
  static constexpr int OFF_ST = 2 * TB + DSB;            // stage s: Q, then dO
  static constexpr int OFF_ROW = OFF_ST + NST * 2 * TB;  // stage s: -lse*log2(e) [128], -D [128]
  static constexpr int OFF_BAR = OFF_ROW + NST * 2 * BM * 4;
  static constexpr int B_KVFULL = 0;
  static constexpr int B_KVFREE = 1;
  static constexpr int B_STFULL = 2;         // + stage
  static constexpr int B_STFREE = 2 + NST;   // + stage
  static constexpr int B_SFULL = 2 + 2 * NST;
  static constexpr int B_DPFULL = B_SFULL + 1;
  static constexpr int B_PRDY = B_SFULL + 2;  // + column half
  static constexpr int B_DSRDY = B_SFULL + 4;
  static constexpr int B_DQFULL = B_SFULL + 5;
  static constexpr int B_DQFREE = B_SFULL + 6;
  static constexpr int B_ACCFULL = B_SFULL + 7;
  static constexpr int B_ACCFREE = B_SFULL + 8;
  static constexpr int B_DRAIN = B_SFULL + 9;
  static constexpr int NBAR = B_SFULL + 10;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16;  // + TMEM slot and abort flag
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D;
  static constexpr uint32_t TMEM_COLS = 512;
};
static_assert(BwCfg<128>::SMEM <= 227 * 1024, "backward d=128 shared memory");
static_assert(BwCfg<64>::SMEM <= 227 * 1024, "backward d=64 shared memory");
static_assert(BwCfg<128>::TM_DK + 128 <= BwCfg<128>::TMEM_COLS, "backward TMEM columns");

// One work unit: a key tile of one KV head of one sequence, and the query
// tiles (of every query head of the group) that can see any of its keys.
struct BUnit {
  int start, len;  // packed row offset and length of the sequence
  int kvh;
  int k0;          // first key of the tile
  int mt0, n_mt;   // first query tile and query tiles per head
  int n_steps;     // n_mt * (Hq / Hkv)
};

// Units are numbered key-tile-major: index u -> (key tile u / (Hkv*B),
// then KV head, then sequence), so the tiles nearest the sequence start,
// which under a causal mask have the most work, come first.
__device__ __forceinline__ bool decode_bunit(const BackwardArgs& a, int u, BUnit& w) {
  const int per = a.Hkv * a.B;
  const int nt = u / per, rem = u - nt * per;
  w.kvh = rem % a.Hkv;
  const int b = rem / a.Hkv;
  if (a.cu_seqlens) {
    w.start = __ldg(a.cu_seqlens + b);
    w.len = min(__ldg(a.cu_seqlens + b + 1) - w.start, a.max_seqlen);
  } else {
    w.start = b * a.N;
    w.len = a.N;
  }
  w.k0 = nt * BN;
  if (w.k0 >= w.len) return false;
  const int nqt = (w.len + BM - 1) / BM;
  w.mt0 = a.causal ? w.k0 / BM : 0;
  int mt_end = nqt;
  // query i sees key j only if i < j + window: the last query that sees the tile
  if (a.window > 0) mt_end = min(nqt, (w.k0 + BN - 1 + a.window - 1) / BM + 1);
  w.n_mt = mt_end - w.mt0;
  w.n_steps = w.n_mt * (a.Hq / a.Hkv);
  return w.n_steps > 0;
}

// Unit of the k-th round of CTA c, alternating direction every round.
__device__ __forceinline__ int unit_of(int k, int c, int G) {
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// Bounded wait that also gives up as soon as another role has aborted. The
// give-up limit sits in shared memory in the word after the abort flag and is
// read only once the first poll has failed. Short limits (set only by tests
// of the give-up path) poll without suspending, as mbar_wait does.
__device__ __forceinline__ bool bw_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint32_t limit_ns = static_cast<uint32_t>(abort_flag[1]);
  const bool quick = limit_ns < kQuickPollBelowNs;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < (quick ? 4 : 64); ++i)
      if (mbar_poll(bar, parity, quick)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      return false;
    }
  }
}

// Warp-uniform outcome: a give-up seen by one lane ends the loops of all 32.
__device__ __forceinline__ bool wwait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = bw_wait(bar, parity, abort_flag);
  return __all_sync(0xFFFFFFFFu, ok);
}

// 32 lanes x 16 consecutive 32-bit TMEM columns from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// Expect `bytes` more transaction bytes on an mbarrier without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// dst[tensor box at (x, y, z)] += smem tile (fp32 add, performed in L2).
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* m, uint32_t src, int x, int y,
                                                  int z) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], "
      "[%1];" ::"l"(m), "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N committed bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t x, uint32_t y, uint32_t z,
                                             uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z),
               "r"(w)
               : "memory");
}

// ----------------------------------------------------------------- kernel 1
// D[h][t] = sum_c dO[t][h][c] * O[t][h][c], one warp per (token, head).
template <int D>
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const BackwardArgs a) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (idx >= static_cast<int64_t>(a.T) * a.Hq) return;
  const int t = static_cast<int>(idx / a.Hq), h = static_cast<int>(idx % a.Hq);
  constexpr int E = D / 32;  // elements per lane
  const int64_t off = idx * D + lane * E;
  const __nv_bfloat16* o = static_cast<const __nv_bfloat16*>(a.o) + off;
  const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(a.dout) + off;
  float s = 0.f;
  if constexpr (E == 4) {
    const uint2 ov = *reinterpret_cast<const uint2*>(o);
    const uint2 gv = *reinterpret_cast<const uint2*>(g);
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float2 of = __bfloat1622float2(o2[e]), gf = __bfloat1622float2(g2[e]);
      s = fmaf(of.x, gf.x, s);
      s = fmaf(of.y, gf.y, s);
    }
  } else {
    const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(o));
    const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(g));
    s = fmaf(of.x, gf.x, of.y * gf.y);
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, m);
  if (lane == 0) a.dvec[static_cast<int64_t>(h) * a.T + t] = s;
}

// ----------------------------------------------------------------- kernel 2
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap vmap,
                const __grid_constant__ CUtensorMap domap,
                const __grid_constant__ CUtensorMap dqmap, const BackwardArgs a) {
  using C = BwCfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {
    if (threadIdx.x == 0) raise_err(a.err, kDevErrInternal);
    return;
  }
  const uint32_t sK = base + C::OFF_K, sV = base + C::OFF_V, sDS = base + C::OFF_DS;
  const uint32_t sST = base + C::OFF_ST;
  float* rows = reinterpret_cast<float*>(smem_raw + C::OFF_ROW);
  const uint32_t bar0 = base + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int Gq = a.Hq / a.Hkv;
  const int n_units = a.n_units;

  if (warp == kMmaWarp) {
    if (lane == 0) {
      mbar_init(bar(C::B_KVFULL), 1);
      mbar_init(bar(C::B_KVFREE), 1);
      for (int s = 0; s < C::NST; ++s) {
        mbar_init(bar(C::B_STFULL + s), 1);
        mbar_init(bar(C::B_STFREE + s), 1);
      }
      mbar_init(bar(C::B_SFULL), 1);
      mbar_init(bar(C::B_DPFULL), 1);
      mbar_init(bar(C::B_PRDY + 0), 128);
      mbar_init(bar(C::B_PRDY + 1), 128);
      mbar_init(bar(C::B_DSRDY), 256);
      mbar_init(bar(C::B_DQFULL), 1);
      mbar_init(bar(C::B_DQFREE), 256);
      mbar_init(bar(C::B_ACCFULL), 1);
      mbar_init(bar(C::B_ACCFREE), 256);
      mbar_init(bar(C::B_DRAIN), 1);
      *abort_flag = 0;
      abort_flag[1] = static_cast<int>(a.wait_ns);  // <= 2 s: fits in 32 bits
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

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    const bool leader = lane == 0;
    if (leader) {
      prefetch_tmap(&qmap);
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
      prefetch_tmap(&domap);
    }
    int gstep = 0, uc = 0;
    bool ok = true;
    for (int kr = 0; ok && kr * G < n_units; ++kr) {
      const int u = unit_of(kr, cta, G);
      BUnit w;
      if (u >= n_units || !decode_bunit(a, u, w)) continue;
      // the previous unit's last MMAs have read K and V
      if (uc > 0 && !(ok = wwait(bar(C::B_KVFREE), (uc - 1) & 1, abort_flag))) break;
      if (leader) {
        const uint32_t fb = bar(C::B_KVFULL);
        mbar_arrive_expect_tx(fb, 2 * C::TB);
#pragma unroll
        for (int p = 0; p < D / 64; ++p) {
          tma_load_3d(sK + p * C::PANEL, &kmap, fb, p * 64, w.kvh, w.start + w.k0);
          tma_load_3d(sV + p * C::PANEL, &vmap, fb, p * 64, w.kvh, w.start + w.k0);
        }
      }
      __syncwarp();
      ++uc;
      for (int s = 0; s < w.n_steps; ++s, ++gstep) {
        const int st = gstep % C::NST, use = gstep / C::NST;
        const int g = s / w.n_mt, q0 = (w.mt0 + s % w.n_mt) * BM;
        const int h = w.kvh * Gq + g;
        // the rows' statistics, negated (the softmax warps only add them);
        // fetched before the wait below so that their latency overlaps it
        float l2[BM / 32], dd[BM / 32];
#pragma unroll
        for (int t = 0; t < BM / 32; ++t) {
          const int i = lane + 32 * t;
          l2[t] = 0.f;
          dd[t] = 0.f;
          if (q0 + i < w.len) {
            const int64_t ix = static_cast<int64_t>(h) * a.T + w.start + q0 + i;
            l2[t] = -__ldg(a.lse + ix) * kLog2e;
            dd[t] = -a.dvec[ix];
          }
        }
        // stage free: its MMAs finished, and with them (they waited for dS)
        // the softmax warps' reads of its row statistics
        if (use > 0 && !(ok = wwait(bar(C::B_STFREE + st), (use - 1) & 1, abort_flag))) break;
        const uint32_t fb = bar(C::B_STFULL + st);
        if (leader) {
          // the copies go out first; the barrier completes once they have
          // landed and the leader has arrived after the row statistics
          const uint32_t sq = sST + st * 2 * C::TB;
          mbar_expect_tx(fb, 2 * C::TB);
#pragma unroll
          for (int p = 0; p < D / 64; ++p) {
            tma_load_3d(sq + p * C::PANEL, &qmap, fb, p * 64, h, w.start + q0);
            tma_load_3d(sq + C::TB + p * C::PANEL, &domap, fb, p * 64, h, w.start + q0);
          }
        }
        float* rl = rows + st * 2 * BM;
#pragma unroll
        for (int t = 0; t < BM / 32; ++t) {
          rl[lane + 32 * t] = l2[t];
          rl[BM + lane + 32 * t] = dd[t];
        }
        __syncwarp();  // the lanes' stores are ordered before the leader's arrive
        if (leader) mbar_arrive(fb);
        __syncwarp();
      }
    }
    // every copy issued must land before the CTA exits
    if (leader) {
      const int last = gstep < C::NST ? gstep : C::NST;
      for (int t = 1; t <= last; ++t) {
        const int gs = gstep - t;
        mbar_wait(bar(C::B_STFULL + gs % C::NST), (gs / C::NST) & 1, kDrainLimitNs);
      }
      if (uc > 0) mbar_wait(bar(C::B_KVFULL), (uc - 1) & 1, kDrainLimitNs);
      if (!ok) raise_err(a.err, kDevErrTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // Lane 0 issues and commits; the whole warp takes part in every wait.
    // Order within a tile: dP (once the previous tile's dQ has left the
    // columns it reuses), dV (as the halves of P arrive), S of the next tile
    // (if its Q has landed), then dK and dQ once dS is in shared memory.
    constexpr uint32_t idesc_s = umma_idesc_bf16_f32(BN, BM, 0, 0);  // S^T, dP^T
    constexpr uint32_t idesc_kv = umma_idesc_bf16_f32(BN, D, 0, 1);  // dV, dK (B: dO, Q MN-major)
    constexpr uint32_t idesc_q = umma_idesc_bf16_f32(BM, D, 1, 1);   // dQ (A: dS, B: K MN-major)
    const uint64_t k_kmaj = umma_smem_desc_sw128(sK, 16, 1024);
    const uint64_t v_kmaj = umma_smem_desc_sw128(sV, 16, 1024);
    const uint64_t k_mn = umma_smem_desc_sw128(sK, C::PANEL, 1024);
    const uint64_t ds_kmaj = umma_smem_desc_sw128(sDS, 16, 1024);
    const uint64_t ds_mn = umma_smem_desc_sw128(sDS, C::PANEL, 1024);
    // descriptor offset (16-byte units) of k-step kk (16 elements):
    // K-major: 32 bytes along a 128-byte panel row, panels 16 KB apart;
    // MN-major: 16 rows of 128 bytes
    auto kmaj = [](int kk) -> uint64_t { return 2u * (kk & 3) + 1024u * (kk >> 2); };
    auto mnmaj = [](int kk) -> uint64_t { return 128u * kk; };
    const bool issuer = lane == 0;
    // S^T = K Q^T of step g (stage g % NST) into the S columns. Those held P
    // of the previous tile, read by its dV MMAs, which this thread issued
    // earlier (the tensor core runs one thread's MMAs in issue order).
    auto issue_s = [&](int g) -> bool {
      const int st = g % C::NST;
      if (!wwait(bar(C::B_STFULL + st), (g / C::NST) & 1, abort_flag)) return false;
      tc_fence_after();
      const uint64_t q_kmaj = umma_smem_desc_sw128(sST + st * 2 * C::TB, 16, 1024);
      if (issuer) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + C::TM_S, k_kmaj + kmaj(kk), q_kmaj + kmaj(kk), idesc_s, kk > 0);
        umma_commit(bar(C::B_SFULL));
      }
      __syncwarp();
      return true;
    };
    int gstep = 0, uc = 0;
    bool ok = true;
    bool s_early = false;  // S of the current step already issued
    for (int kr = 0; ok && kr * G < n_units; ++kr) {
      const int u = unit_of(kr, cta, G);
      BUnit w;
      if (u >= n_units || !decode_bunit(a, u, w)) continue;
      if (!(ok = wwait(bar(C::B_KVFULL), uc & 1, abort_flag))) break;
      for (int s = 0; s < w.n_steps; ++s, ++gstep) {
        const int st = gstep % C::NST;
        const uint32_t sq = sST + st * 2 * C::TB, sdo = sq + C::TB;
        const bool first = s == 0;
        if (!s_early && !(ok = issue_s(gstep))) break;
        const uint64_t do_kmaj = umma_smem_desc_sw128(sdo, 16, 1024);
        const uint64_t q_mn = umma_smem_desc_sw128(sq, C::PANEL, 1024);
        const uint64_t do_mn = umma_smem_desc_sw128(sdo, C::PANEL, 1024);
        // dP^T = V dO^T first (dS waits for it; dV does not), into the
        // columns of the previous tile's dQ once that has been read out
        if (gstep > 0 && !(ok = wwait(bar(C::B_DQFREE), (gstep - 1) & 1, abort_flag))) break;
        tc_fence_after();
        if (issuer) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(tmem + C::TM_DP, v_kmaj + kmaj(kk), do_kmaj + kmaj(kk), idesc_s, kk > 0);
          umma_commit(bar(C::B_DPFULL));
        }
        __syncwarp();
        // dV += P^T dO: the previous unit's dK / dV must have been read out
        if (first && uc > 0 && !(ok = wwait(bar(C::B_ACCFREE), (uc - 1) & 1, abort_flag))) break;
        if (!(ok = wwait(bar(C::B_PRDY + 0), gstep & 1, abort_flag))) break;
        tc_fence_after();
        if (issuer) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ts(tmem + C::TM_DV, tmem + C::TM_S + 8 * kk, do_mn + mnmaj(kk), idesc_kv,
                    (!first || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
        if (!(ok = wwait(bar(C::B_PRDY + 1), gstep & 1, abort_flag))) break;
        tc_fence_after();
        if (issuer) {
#pragma unroll
          for (int kk = 4; kk < 8; ++kk)
            umma_ts(tmem + C::TM_DV, tmem + C::TM_S + 64 + 8 * (kk - 4), do_mn + mnmaj(kk),
                    idesc_kv, 1u);
        }
        __syncwarp();
        // S of the next tile (same unit: same K) if its Q has landed; it
        // runs while the softmax warps form this tile's dS
        s_early = false;
        if (s + 1 < w.n_steps) {
          const int g1 = gstep + 1;
          const bool ready = __all_sync(
              0xFFFFFFFFu, mbar_try_wait(bar(C::B_STFULL + g1 % C::NST), (g1 / C::NST) & 1));
          if (ready) {
            if (!(ok = issue_s(g1))) break;
            s_early = true;
          }
        }
        // dK += dS^T Q and dQ = dS K, both reading the dS^T tile
        if (!(ok = wwait(bar(C::B_DSRDY), gstep & 1, abort_flag))) break;
        tc_fence_after();
        if (issuer) {
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            umma_ss(tmem + C::TM_DK, ds_kmaj + kmaj(kk), q_mn + mnmaj(kk), idesc_kv,
                    (!first || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            umma_ss(tmem + C::TM_DP, ds_mn + mnmaj(kk), k_mn + mnmaj(kk), idesc_q, kk > 0);
          umma_commit(bar(C::B_DQFULL));
          umma_commit(bar(C::B_STFREE + st));
          if (s == w.n_steps - 1) {
            umma_commit(bar(C::B_KVFREE));
            umma_commit(bar(C::B_ACCFULL));
          }
        }
        __syncwarp();
      }
      if (!ok) break;
      ++uc;
    }
    // every MMA issued above has finished once this commit arrives
    if (issuer) umma_commit(bar(C::B_DRAIN));
    __syncwarp();
    mbar_wait(bar(C::B_DRAIN), 0, kDrainLimitNs);
    if (!ok && issuer) raise_err(a.err, kDevErrTimeout);
  } else {
    // --------------------------------- P, dS, dQ read-out, dK / dV (warps 0-7)
    // Warp (wq, ch): key rows 32*wq.. (its TMEM lane quarter) and query
    // columns 64*ch.. of S^T / dP^T; the same lanes and d columns (d/2)*ch..
    // of dQ, dK and dV. Per tile s the order is
    //   P(s), read-out of dQ(s-1), dS(s),
    // so P(s) runs while the tensor core computes dK / dQ of the previous
    // tile, and the read-out frees the columns dP(s) needs right after.
    const int wq = warp & 3, ch = warp >> 2;
    const int r = wq * 32 + lane;  // key row of the tile; query row of dQ
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::TM_S + 64 * ch;  // S^T columns of this half
    const uint32_t tDP = tmem + lane_off + C::TM_DP + 64 * ch;
    const uint32_t tDQ = tmem + lane_off + C::TM_DP + (D / 2) * ch;  // d columns (d/2)*ch..
    // this warp's rows of the dS^T tile (32 rows x 128 bytes of panel ch);
    // between the dQ MMA and the next dS they stage this warp's dQ columns
    const uint32_t my_ds = sDS + ch * C::PANEL + wq * 32 * 128;
    const uint32_t ds_row = my_ds + lane * 128;
    const uint32_t swz = static_cast<uint32_t>(lane & 7);  // = row & 7
    const uint64_t sl2x2 = f2(a.scale_log2, a.scale_log2);

    // dQ of step gs (query head h, first row q0 of a sequence starting at
    // `start`, `len` rows): TMEM -> registers (the columns are then free)
    // -> 128-byte-swizzled staging in this warp's dS^T rows -> bulk tensor
    // reduce-add into the fp32 buffer [T, Hq, d], performed in L2. Rows past
    // the sequence hold dQ = 0 exactly (their P and dS are 0), so whole
    // boxes are added; boxes wholly past it are skipped.
    auto readout = [&](int gs, int h, int q0, int start, int len) -> bool {
      if (!wwait(bar(C::B_DQFULL), gs & 1, abort_flag)) return false;
      tc_fence_after();
      uint32_t x[D / 2];
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tmem_ld32(tDQ + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&x[32 * c]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(C::B_DQFREE));
      const bool any_live = q0 + wq * 32 < len;
      const int row0 = start + q0 + wq * 32;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        if (c > 0) {
          if (lane == 0) bulk_wait_read<0>();  // the previous chunk's copy has read the staging
          __syncwarp();
        }
#pragma unroll
        for (int m = 0; m < 8; ++m)
          st_shared_v4(ds_row + ((static_cast<uint32_t>(m) ^ swz) << 4), x[32 * c + 4 * m],
                       x[32 * c + 4 * m + 1], x[32 * c + 4 * m + 2], x[32 * c + 4 * m + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && any_live) {
          tma_reduce_add_3d(&dqmap, my_ds, (D / 2) * ch + 32 * c, h, row0);
          bulk_commit();
        }
      }
      return true;
    };

    int gstep = 0, uc = 0;
    bool ok = true;
    for (int kr = 0; ok && kr * G < n_units; ++kr) {
      const int u = unit_of(kr, cta, G);
      BUnit w;
      if (u >= n_units || !decode_bunit(a, u, w)) continue;
      const int j = w.k0 + r;  // key position
      int prev_h = 0, prev_q0 = 0;
      for (int s = 0; s < w.n_steps; ++s, ++gstep) {
        const int st = gstep % C::NST, use = gstep / C::NST;
        const int g = s / w.n_mt, q0 = (w.mt0 + s % w.n_mt) * BM;
        const int h = w.kvh * Gq + g;
        const int qc = q0 + 64 * ch;  // query of this half's first column
        // the stage's row statistics (generic stores released by the
        // producer's arrive) and S^T
        if (!(ok = wwait(bar(C::B_STFULL + st), use & 1, abort_flag))) break;
        if (!(ok = wwait(bar(C::B_SFULL), gstep & 1, abort_flag))) break;
        tc_fence_after();
        const float4* nl4 = reinterpret_cast<const float4*>(rows + st * 2 * BM + 64 * ch);
        const float4* nd4 = nl4 + BM / 4;
        const bool need_mask = (q0 + BM > w.len) || (w.k0 + BN > w.len) ||
                               (a.causal && w.k0 + BN - 1 > q0) ||
                               (a.window > 0 && w.k0 <= q0 + BM - 1 - a.window);
        // P = 2^(S*scale*log2 e - lse*log2 e) for this half's 64 queries,
        // kept in fp32 (for dS) and stored as bf16 pairs into the first 32 of
        // the half's S columns (all 64 were read first)
        uint32_t p[64];
        tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&p[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&p[32]));
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float4 l = nl4[e];
          float x0, x1, x2, x3;
          unf2(ffma2(f2(__uint_as_float(p[4 * e]), __uint_as_float(p[4 * e + 1])), sl2x2,
                     f2(l.x, l.y)), x0, x1);
          unf2(ffma2(f2(__uint_as_float(p[4 * e + 2]), __uint_as_float(p[4 * e + 3])), sl2x2,
                     f2(l.z, l.w)), x2, x3);
          p[4 * e] = __float_as_uint(ex2(x0));
          p[4 * e + 1] = __float_as_uint(ex2(x1));
          p[4 * e + 2] = __float_as_uint(ex2(x2));
          p[4 * e + 3] = __float_as_uint(ex2(x3));
        }
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int i = qc + c;
            const bool vis = i < w.len && j < w.len && (!a.causal || j <= i) &&
                             (a.window <= 0 || j > i - a.window);
            if (!vis) p[c] = 0u;
          }
        }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16(__uint_as_float(p[32 * hf + 2 * e]),
                              __uint_as_float(p[32 * hf + 2 * e + 1]));
          tmem_st16(tS + 16 * hf, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(C::B_PRDY + ch));
        // the previous tile's dQ, which frees the columns of this tile's dP
        if (s > 0 && !(ok = readout(gstep - 1, prev_h, prev_q0, w.start, w.len))) break;
        // dP^T; this warp's dS^T rows are free once the copies of the dQ
        // staged there have read them (the dK / dQ MMAs that read the
        // previous dS finished before that dQ was read out)
        if (!(ok = wwait(bar(C::B_DPFULL), gstep & 1, abort_flag))) break;
        tc_fence_after();
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t dp[32];
          tmem_ld32(tDP + 32 * cc, dp);
          tmem_wait_ld();
          uint32_t dsk[16];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 nd = nd4[8 * cc + e];
            const int c = 32 * cc + 4 * e;
            float d0, d1, d2, d3;
            unf2(fmul2(fadd2(f2(__uint_as_float(dp[4 * e]), __uint_as_float(dp[4 * e + 1])),
                             f2(nd.x, nd.y)),
                       f2(__uint_as_float(p[c]), __uint_as_float(p[c + 1]))), d0, d1);
            unf2(fmul2(fadd2(f2(__uint_as_float(dp[4 * e + 2]), __uint_as_float(dp[4 * e + 3])),
                             f2(nd.z, nd.w)),
                       f2(__uint_as_float(p[c + 2]), __uint_as_float(p[c + 3]))), d2, d3);
            dsk[2 * e] = pack_bf16(d0, d1);
            dsk[2 * e + 1] = pack_bf16(d2, d3);
          }
          // 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r & 7)
#pragma unroll
          for (int m = 0; m < 4; ++m)
            st_shared_v4(ds_row + ((static_cast<uint32_t>(4 * cc + m) ^ swz) << 4), dsk[4 * m],
                         dsk[4 * m + 1], dsk[4 * m + 2], dsk[4 * m + 3]);
        }
        fence_proxy_async_smem();  // generic stores -> tensor-core reads
        mbar_arrive(bar(C::B_DSRDY));
        prev_h = h;
        prev_q0 = q0;
      }
      if (!ok) break;
      // the unit's last dQ, then its dK (times scale) and dV
      if (!(ok = readout(gstep - 1, prev_h, prev_q0, w.start, w.len))) break;
      if (!(ok = wwait(bar(C::B_ACCFULL), uc & 1, abort_flag))) break;
      tc_fence_after();
      const bool klive = j < w.len;
      const int64_t row = (static_cast<int64_t>(w.start + j) * a.Hkv + w.kvh) * D + (D / 2) * ch;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t t0 = tmem + lane_off + (which ? C::TM_DK : C::TM_DV) + (D / 2) * ch;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(which ? a.dk : a.dv) + row;
        const float sc = which ? a.scale : 1.f;
        const uint64_t sc2 = f2(sc, sc);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t x[32];
          tmem_ld32(t0 + 32 * c, x);
          tmem_wait_ld();
          if (klive) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float lo, hi;
              unf2(fmul2(f2(__uint_as_float(x[2 * e]), __uint_as_float(x[2 * e + 1])), sc2), lo,
                   hi);
              pk[e] = pack_bf16(lo, hi);
            }
            st_global_v8(out + 32 * c, pk);
            st_global_v8(out + 32 * c + 16, pk + 8);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_ACCFREE));
      ++uc;
    }
    if (lane == 0) {
      bulk_wait<0>();  // every reduction issued has completed
      if (!ok) raise_err(a.err, kDevErrTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ----------------------------------------------------------------- kernel 3
// dq = bf16(scale * acc), both [T, Hq, d]; 8 elements per thread.
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const BackwardArgs a, int64_t n8) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  if (i >= n8) return;
  const float4 lo = reinterpret_cast<const float4*>(a.dq_acc)[2 * i];
  const float4 hi = reinterpret_cast<const float4*>(a.dq_acc)[2 * i + 1];
  uint4 out;
  out.x = pack_bf16(lo.x * a.scale, lo.y * a.scale);
  out.y = pack_bf16(lo.z * a.scale, lo.w * a.scale);
  out.z = pack_bf16(hi.x * a.scale, hi.y * a.scale);
  out.w = pack_bf16(hi.z * a.scale, hi.w * a.scale);
  reinterpret_cast<uint4*>(a.dq)[i] = out;
}

int g_bw_attr[2][64];

template <int D>
cudaError_t launch_all(const BackwardArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                       const CUtensorMap& vmap, const CUtensorMap& domap,
                       const CUtensorMap& dqmap, int num_sms, cudaStream_t s) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!g_bw_attr[D == 128][dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, BwCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    g_bw_attr[D == 128][dev] = 1;
  }
  cudaError_t e = cudaMemsetAsync(a.dq_acc, 0, static_cast<size_t>(a.T) * a.Hq * D * 4, s);
  if (e != cudaSuccess) return e;
  const long long warps = static_cast<long long>(a.T) * a.Hq;
  bwd_rowdot_kernel<D><<<static_cast<unsigned>((warps + 7) / 8), 256, 0, s>>>(a);
  const unsigned grid = static_cast<unsigned>(a.n_units < num_sms ? a.n_units : num_sms);
  attn_bwd_kernel<D><<<grid, kThreads, BwCfg<D>::SMEM, s>>>(qmap, kmap, vmap, domap, dqmap, a);
  const int64_t n8 = static_cast<int64_t>(a.T) * a.Hq * D / 8;
  bwd_dq_convert_kernel<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, s>>>(a, n8);
  return cudaGetLastError();
}

}  // namespace

size_t backward_workspace_bytes(long long T, int Hq, int d) {
  const size_t acc = static_cast<size_t>(T) * Hq * d * 4;
  const size_t dv = static_cast<size_t>(T) * Hq * 4;
  return ((acc + 255) & ~static_cast<size_t>(255)) + ((dv + 255) & ~static_cast<size_t>(255));
}

cudaError_t launch_prefill_backward_bf16(const BackwardArgs& a0, const CUtensorMap& qmap,
                                         const CUtensorMap& kmap, const CUtensorMap& vmap,
                                         const CUtensorMap& domap, const CUtensorMap& dqmap,
                                         int num_sms, cudaStream_t s) {
  BackwardArgs a = a0;
  const long long n_kt = (a.max_seqlen + BN - 1) / BN;
  const long long units = n_kt * a.Hkv * a.B;
  if (units == 0) return cudaSuccess;
  if (units > INT_MAX || static_cast<long long>(a.T) * a.Hq * a.d / 8 / 256 + 1 > INT_MAX)
    return cudaErrorInvalidConfiguration;
  a.n_units = static_cast<int>(units);
  return a.d == 128 ? launch_all<128>(a, qmap, kmap, vmap, domap, dqmap, num_sms, s)
                    : launch_all<64>(a, qmap, kmap, vmap, domap, dqmap, num_sms, s);
}

}  // namespace pa
