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
// sm_103a design. A persistent grid of one CTA per SM walks a static list of
// work units, heaviest first. A unit is two 128-row query tiles that read the
// same K/V stream: the same rows of two query heads of one KV group when
// Hq/Hkv is even, otherwise two consecutive row tiles of one head (their key
// ranges are merged; keys a tile may not see are masked).
//  * warp 16 (K/V producer): K and V tiles of 128 keys in turn through a
//    ring of 32 KB slots (d = 128). Every tile is stored as 64-element
//    (128-byte) panels, 128-byte swizzled: the K-major / MN-major operand
//    layouts the tensor cores read directly.
//  * warp 18 (Q producer): the unit's two Q tiles, each as soon as the last
//    QK^T of the previous unit on that tile has been issued. Apart from the
//    K/V producer, so that the ring keeps filling across unit boundaries.
//  * warp 17 (tcgen05 issuer): MMAs in the steady order
//      ... QK_0(j), PV_1(j-1), QK_1(j), PV_0(j), QK_0(j+1), PV_1(j), ...
//    S_i = Q_i K^T (M=128, N=128, both operands in shared memory) into TMEM,
//    and O_i += P_i V (A = P_i read from TMEM, B = V in shared memory). Each
//    softmax therefore has two other MMAs (about 1000 cycles) to run in, and
//    the two softmax groups take turns on the SFU. Descriptors are formed
//    once; the per-MMA issue work is one add, which keeps the MMA pipe full.
//  * warps 0-7 / 8-15 (softmax of query tile 0 / 1): each warp owns 16 rows
//    through the 16-lane TMEM access shapes, four threads per row. Per key
//    tile and per half of 64 keys: read the scores from TMEM, mask only on
//    tiles that straddle the diagonal, the window edge or the sequence end,
//    reduce the rows' max over the quad with shuffles, update the running
//    max in the log2 domain with scale*log2(e) folded into one FMA,
//    exponentiate with ex2, write P as bf16 pairs back into the score
//    buffer's first 64 columns, where the PV MMA reads it, and hand that
//    half over. At the end of a unit they read O from TMEM, divide by the
//    running sum and store O and the LSE.
//  * The max is rescaled lazily: O and the sum are only rescaled when the max
//    grows by more than 2^8; otherwise the stale max is kept. O / sum is
//    unchanged (both carry the same factor), P stays <= 256, and TMEM round
//    trips of O become rare. Before a tile's first hand-over O is idle (the
//    commit that signalled S_i(j) also covers PV_i(j-1)); before the second,
//    the rescale waits for the commit that follows the first PV half.
//  * S_i(j+1) overwrites the TMEM columns that hold P_i(j). The MMA that
//    reads P_i(j) is issued before the MMA that overwrites it, by the same
//    thread, and the SM's tensor core executes one thread's MMAs in issue
//    order.
//  * Tiles above the diagonal or left of the window are never loaded. All
//    waits are bounded; a wait that gives up raises PA_DEV_TIMEOUT, and every
//    role then winds down: copies and MMAs in flight are waited for before
//    TMEM is freed.
#include <climits>
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

constexpr int kMaxSchedSeqs = 512;  // packed sequences the on-chip work list can sort

constexpr int kSoftmaxWarps = 16;  // 8 per query tile
constexpr int kLoadWarp = 16;      // K / V producer
constexpr int kMmaWarp = 17;       // tcgen05 issuer
constexpr int kQWarp = 18;         // Q producer
constexpr int kThreads = 19 * 32;

template <int D>
struct PfCfg {
  static constexpr int QB = BM * D * 2;        // one Q tile (bytes)
  static constexpr int TB = BN * D * 2;        // one K or V tile
  static constexpr int PANEL_Q = BM * 128;     // bytes per 64-column panel of a Q tile
  static constexpr int PANEL_T = BN * 128;     // of a K / V tile
  static constexpr int NSLOT = D == 128 ? 5 : 10;  // K/V ring slots
  static constexpr int OFF_Q = 0;              // Q tile 0, Q tile 1
  static constexpr int OFF_RING = 2 * QB;
  static constexpr int OFF_BAR = OFF_RING + NSLOT * TB;
  // mbarriers
  static constexpr int B_QFULL = 0;            // + query tile
  static constexpr int B_QFREE = 2;            // + query tile
  static constexpr int B_FULL = 4;             // + ring slot
  static constexpr int B_EMPTY = 4 + NSLOT;    // + ring slot
  static constexpr int B_SFULL = 4 + 2 * NSLOT;   // + query tile
  static constexpr int B_PRDY = 6 + 2 * NSLOT;    // + 2 * query tile + half (keys 0-63 / 64-127)
  static constexpr int B_OFULL = 10 + 2 * NSLOT;  // + query tile
  static constexpr int B_DRAIN = 12 + 2 * NSLOT;
  static constexpr int B_PVH0 = 13 + 2 * NSLOT;   // + query tile: PV over keys 0-63 done
  static constexpr int B_EPI = 15 + 2 * NSLOT;    // + 4 * query tile + lane quarter
  static constexpr int NBAR = 23 + 2 * NSLOT;
  static constexpr int OFF_SCHED = OFF_BAR + NBAR * 8 + 16;  // after the TMEM slot + abort flag
  static constexpr int SMEM = OFF_SCHED + 2 * kMaxSchedSeqs * 2 + 16;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TM_O = 2 * BN;     // S_i at i*BN, O_i at TM_O + i*D
};
static_assert(PfCfg<128>::SMEM <= 227 * 1024, "prefill d=128 shared memory");
static_assert(PfCfg<128>::PANEL_Q == PfCfg<128>::PANEL_T, "Q and K panels share descriptor offsets");
static_assert(PfCfg<64>::SMEM <= 227 * 1024, "prefill d=64 shared memory");

// One work unit: two query tiles sharing a KV head and a key range.
struct Unit {
  int start, len;  // packed row offset and number of query rows of the sequence
  int lk;          // keys of the sequence (= len unless the keys are paged)
  int qoff;        // position of query row 0 among the keys (lk - len when paged)
  int b;           // sequence
  int q0[2];       // first row (within the sequence) of each query tile
  int h[2];        // query head of each tile
  int kvh;
  int t_begin;     // first key tile
  int n_tiles;     // key tiles streamed
};

// Work list. Level L of a sequence is its L-th 128-row query tile (two-head
// units) or its L-th pair of query tiles (two-tile units); under a causal mask
// a higher level has a longer key range. Units are ordered by level, highest
// first, then by `pair` (head pair, or head) and sequence.
__device__ __forceinline__ bool decode_unit(const PrefillArgs& a, int level, int b, int pair,
                                            Unit& w) {
  int qt0, qt1;
  if (a.pair_heads) {
    qt0 = qt1 = level;
    w.h[0] = 2 * pair;
    w.h[1] = 2 * pair + 1;
  } else {
    qt0 = 2 * level;
    qt1 = qt0 + 1;
    w.h[0] = w.h[1] = pair;
  }
  if (a.cu_seqlens) {
    w.start = a.cu_seqlens[b];
    w.len = min(a.cu_seqlens[b + 1] - w.start, a.max_seqlen);
  } else {
    w.start = b * a.N;
    w.len = a.N;
  }
  w.b = b;
  w.lk = w.len;
  w.qoff = 0;
  if (a.table) {
    // keys from the paged cache: the last len of them are this chunk's own
    w.lk = min(max(a.seq_lens_k[b], 0), a.max_blocks * 16);
    w.qoff = w.lk - w.len;  // < 0 only on bad input (raised by the caller check)
  }
  w.q0[0] = qt0 * BM;
  w.q0[1] = qt1 * BM;
  if (w.q0[0] >= w.len) return false;
  const int q_last = min(w.len, w.q0[1] + BM) - 1;  // last row of either tile
  int kv_end = a.causal ? min(w.lk, w.qoff + q_last + 1) : w.lk;
  int kv_begin = a.window > 0 ? max(0, w.qoff + w.q0[0] - a.window + 1) : 0;
  kv_end = max(kv_end, 1);  // at least one (possibly fully masked) key tile
  kv_begin = min(kv_begin, kv_end - 1);
  w.t_begin = kv_begin / BN;
  w.n_tiles = (kv_end + BN - 1) / BN - w.t_begin;
  w.kvh = w.h[0] / (a.Hq / a.Hkv);
  return true;
}

// Index -> (level, sequence, pair) over the work list. Without a compact
// list (fixed-length batches, or more packed sequences than the on-chip
// table holds) every (level, pair, sequence) of the longest sequence is an
// index and indices past a shorter sequence's end are skipped. With it
// (packed batches), sequences are sorted by their level count, longest first,
// and only existing units get an index, so consecutive indices -- handed out
// round-robin to the CTAs -- are all real work.
struct Sched {
  const uint16_t* order;  // sequence of each rank
  const uint16_t* nl;     // levels of each rank (non-increasing unless seq_major)
  int nseq, npairs, nlev;
  bool compact;
  bool seq_major;         // paged keys: rank by rank (longest cache first), not level by level
  int L, cum, cnt;        // compact walk: current level (seq_major: rank), indices below it, ...

  __device__ __forceinline__ int count_gt(int lv) const {  // ranks with more than lv levels
    int lo = 0, hi = nseq;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (nl[mid] > lv) lo = mid + 1; else hi = mid;
    }
    return lo;
  }
  __device__ __forceinline__ void start() {
    if (compact && seq_major) {
      L = 0;  // rank
      cum = 0;
    } else if (compact) {
      L = static_cast<int>(nl[0]) - 1;
      cum = 0;
      cnt = L >= 0 ? count_gt(L) : 0;
    }
  }
  // indices must be visited in increasing order
  __device__ __forceinline__ void map(int v, int& level, int& b, int& pair) {
    if (compact && seq_major) {
      // a sequence's units (its levels, highest first, times the pairs) are
      // consecutive, so the units in flight share one or two sequences' keys
      while (v >= cum + static_cast<int>(nl[L]) * npairs) {
        cum += static_cast<int>(nl[L]) * npairs;
        ++L;
      }
      const int j = v - cum;
      b = order[L];
      level = static_cast<int>(nl[L]) - 1 - j / npairs;
      pair = j % npairs;
    } else if (compact) {
      while (v >= cum + cnt * npairs) {
        cum += cnt * npairs;
        --L;
        cnt = count_gt(L);
      }
      const int j = v - cum;
      b = order[j % cnt];
      pair = j / cnt;
      level = L;
    } else {
      const int per = npairs * nseq;
      const int lvl = v / per, rem = v - lvl * per;
      b = rem % nseq;
      pair = rem / nseq;
      level = nlev - 1 - lvl;
    }
  }
};

// Unit of the k-th round of CTA c: rounds alternate direction ("snake"), so
// with units sorted heaviest first every CTA gets a similar total.
__device__ __forceinline__ int unit_of(int k, int c, int G) {
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// Bounded wait (limit_ns of wall time) that also gives up as soon as another
// role has aborted.
__device__ __forceinline__ bool pf_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                        uint64_t limit_ns) {
  const bool quick = limit_ns < kQuickPollBelowNs;  // a test's short limit
  const int spins = quick ? 4 : 64;                  // polls between clock reads
  if (mbar_poll(bar, parity, quick)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < spins; ++i)
      if (mbar_poll(bar, parity, quick)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      return false;
    }
  }
}

// Every lane of the warp waits; the outcome is made warp-uniform so that a
// give-up seen by one lane ends the loops of all 32 together (the warp-wide
// tcgen05 and shuffle instructions that follow need every lane).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity,
                                          volatile int* abort_flag, uint64_t limit_ns) {
  const bool ok = pf_wait(bar, parity, abort_flag, limit_ns);
  return __all_sync(0xFFFFFFFFu, ok);
}

constexpr uint64_t kDrainLimitNs = 100000000ull;  // 0.1 s for copies / MMAs already in flight

template <int D, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1)
prefill_bf16_kernel(const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  using C = PfCfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;

  // 1024-byte alignment is what the 128-byte swizzle expects of every tile
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {
    if (threadIdx.x == 0) raise_err(a.err, kDevErrInternal);
    return;
  }
  uint8_t* gb = smem_raw;
  const uint32_t sQ = base + C::OFF_Q, sRing = base + C::OFF_RING;
  const uint32_t bar0 = base + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // ---- work list (all threads): sort packed sequences by level count
  uint16_t* s_order = reinterpret_cast<uint16_t*>(gb + C::OFF_SCHED);
  uint16_t* s_nl = s_order + kMaxSchedSeqs;
  int* s_total = reinterpret_cast<int*>(s_nl + kMaxSchedSeqs);
  const int npairs = a.pair_heads ? (a.Hq >> 1) : a.Hq;
  if (a.compact) {
    uint16_t* tmp = reinterpret_cast<uint16_t*>(gb + C::OFF_RING);  // the ring is still unused
    if (threadIdx.x == 0) *s_total = 0;
    // levels of sequence b; the sort key is the level count, or with paged
    // keys the cache length in blocks (the work grows with the cached prefix)
    auto levels = [&](int b) {
      const int len = max(0, min(a.cu_seqlens[b + 1] - a.cu_seqlens[b], a.max_seqlen));
      const int nqt = (len + BM - 1) / BM;
      return a.pair_heads ? nqt : (nqt + 1) >> 1;
    };
    for (int b = threadIdx.x; b < a.B; b += kThreads) {
      int key = levels(b);
      if (a.table) key = min(65535, (min(max(a.seq_lens_k[b], 0), a.max_blocks * 16) + 15) / 16);
      tmp[b] = static_cast<uint16_t>(key);
    }
    __syncthreads();
    int part = 0;
    for (int b = threadIdx.x; b < a.B; b += kThreads) {
      const int n = tmp[b];
      int rank = 0;
      for (int b2 = 0; b2 < a.B; ++b2) {
        const int n2 = tmp[b2];
        rank += (n2 > n) || (n2 == n && b2 < b);
      }
      const int nl = levels(b);
      s_order[rank] = static_cast<uint16_t>(b);
      s_nl[rank] = static_cast<uint16_t>(nl);
      part += nl;
    }
    __syncthreads();  // *s_total zeroed and every rank of tmp read
    if (part) atomicAdd(s_total, part * npairs);
    fence_proxy_async_smem();  // the ring's generic writes before TMA reuses it
  }

  if (warp == kMmaWarp) {
    if (lane == 0) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(bar(C::B_QFULL + i), 1);
        mbar_init(bar(C::B_QFREE + i), 1);
        mbar_init(bar(C::B_SFULL + i), 1);
        mbar_init(bar(C::B_PRDY + 2 * i), kSoftmaxWarps / 2 * 32);
        mbar_init(bar(C::B_PRDY + 2 * i + 1), kSoftmaxWarps / 2 * 32);
        mbar_init(bar(C::B_OFULL + i), 1);
        mbar_init(bar(C::B_PVH0 + i), 1);
        for (int q = 0; q < 4; ++q) mbar_init(bar(C::B_EPI + 4 * i + q), 64);
      }
      for (int s = 0; s < C::NSLOT; ++s) {
        mbar_init(bar(C::B_FULL + s), 1);
        mbar_init(bar(C::B_EMPTY + s), 1);
      }
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
  Sched sched;
  sched.order = s_order;
  sched.nl = s_nl;
  sched.nseq = a.B;
  sched.npairs = npairs;
  sched.nlev = a.pair_heads ? (a.max_seqlen + BM - 1) / BM : ((a.max_seqlen + BM - 1) / BM + 1) / 2;
  sched.compact = a.compact != 0;
  sched.seq_major = a.table != nullptr;
  sched.start();
  const int n_units = a.compact ? *s_total : a.n_units;

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    const bool leader = lane == 0;
    if (leader) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
    }
    uint32_t slot = 0, phase = 0;
    int issued = 0;             // K/V tiles issued into the ring
    bool ok = true;
    auto load_tile = [&](const CUtensorMap* m, int row, int head) -> bool {
      if (issued >= C::NSLOT && !warp_wait(bar(C::B_EMPTY + slot), phase ^ 1u, abort_flag, a.wait_ns))
        return false;
      if (leader) {
        const uint32_t fb = bar(C::B_FULL + slot);
        mbar_arrive_expect_tx(fb, C::TB);
#pragma unroll
        for (int p = 0; p < D / 64; ++p)
          tma_load_3d(sRing + slot * C::TB + p * C::PANEL_T, m, fb, p * 64, head, row);
      }
      __syncwarp();
      ++issued;
      if (++slot == C::NSLOT) {
        slot = 0;
        phase ^= 1u;
      }
      return true;
    };
    // Paged keys: a tile of 128 keys is 8 blocks of 16; lane t < 8 copies
    // block t (one 16-row box per 64-column panel) straight to its rows of
    // the slot. Blocks past the sequence's keys are not loaded.
    auto load_tile_paged = [&](const CUtensorMap* m, int key0, const Unit& w) -> bool {
      if (issued >= C::NSLOT && !warp_wait(bar(C::B_EMPTY + slot), phase ^ 1u, abort_flag, a.wait_ns))
        return false;
      const int pg = key0 / 16 + lane;
      bool have = lane < BN / 16 && pg * 16 < w.lk;
      int blk = -1;
      if (have) {
        blk = a.table[static_cast<int64_t>(w.b) * a.max_blocks + pg];
        if (blk < 0 || blk >= a.num_blocks) {
          raise_err(a.err, kDevErrBadBlock);
          have = false;
        }
      }
      const unsigned n = __popc(__ballot_sync(0xFFFFFFFFu, have));
      const uint32_t fb = bar(C::B_FULL + slot);
      if (leader) mbar_arrive_expect_tx(fb, n * (D / 64) * 16 * 128);
      __syncwarp();
      if (have) {
#pragma unroll
        for (int p = 0; p < D / 64; ++p)
          tma_load_4d(sRing + slot * C::TB + p * C::PANEL_T + lane * 16 * 128, m, fb, p * 64, 0,
                      w.kvh, blk);
      }
      __syncwarp();
      ++issued;
      if (++slot == C::NSLOT) {
        slot = 0;
        phase ^= 1u;
      }
      return true;
    };
    for (int k = 0; ok && k * G < n_units; ++k) {
      const int u = unit_of(k, cta, G);
      Unit w;
      int lv, sb, pr;
      if (u >= n_units) continue;
      sched.map(u, lv, sb, pr);
      if (!decode_unit(a, lv, sb, pr, w)) continue;
      for (int j = 0; ok && j < w.n_tiles; ++j) {
        const int key0 = (w.t_begin + j) * BN;
        if constexpr (PAGED)
          ok = load_tile_paged(&kmap, key0, w) && load_tile_paged(&vmap, key0, w);
        else
          ok = load_tile(&kmap, w.start + key0, w.kvh) && load_tile(&vmap, w.start + key0, w.kvh);
      }
    }
    // every copy issued must land before the CTA exits
    if (leader) {
      const int nring = issued < C::NSLOT ? issued : C::NSLOT;
      for (int t = 1; t <= nring; ++t) {
        const int p = issued - t;
        mbar_wait(bar(C::B_FULL + p % C::NSLOT), (p / C::NSLOT) & 1, kDrainLimitNs);
      }
      if (!ok) raise_err(a.err, kDevErrTimeout);
    }
  } else if (warp == kQWarp) {
    // ---------------------------------------------------------- Q producer
    // The two query tiles of each unit, each as soon as the MMA warp has
    // issued the last QK^T of the previous unit on that tile. Kept apart
    // from the K / V producer so that its ring runs on into the next unit
    // while these wait.
    const bool leader = lane == 0;
    if (leader) prefetch_tmap(&qmap);
    int q_loads = 0;  // units whose Q tiles were issued
    int half = 0;     // tiles of the current unit issued (an abort may leave 1)
    bool ok = true;
    for (int k = 0; ok && k * G < n_units; ++k) {
      const int u = unit_of(k, cta, G);
      Unit w;
      int lv, sb, pr;
      if (u >= n_units) continue;
      sched.map(u, lv, sb, pr);
      if (!decode_unit(a, lv, sb, pr, w)) continue;
      for (half = 0; half < 2; ++half) {
        if (q_loads > 0 &&
            !warp_wait(bar(C::B_QFREE + half), (q_loads - 1) & 1, abort_flag, a.wait_ns)) {
          ok = false;
          break;
        }
        if (leader) {
          const uint32_t qb = bar(C::B_QFULL + half);
          mbar_arrive_expect_tx(qb, C::QB);
#pragma unroll
          for (int p = 0; p < D / 64; ++p)
            tma_load_3d(sQ + half * C::QB + p * C::PANEL_Q, &qmap, qb, p * 64, w.h[half],
                        w.start + w.q0[half]);
        }
        __syncwarp();
      }
      if (ok) ++q_loads;
    }
    // every Q copy issued must land before the CTA exits
    if (leader) {
      if (!ok && half > 0) mbar_wait(bar(C::B_QFULL + 0), q_loads & 1, kDrainLimitNs);
      if (q_loads > 0) {
        mbar_wait(bar(C::B_QFULL + 0), (q_loads - 1) & 1, kDrainLimitNs);
        mbar_wait(bar(C::B_QFULL + 1), (q_loads - 1) & 1, kDrainLimitNs);
      }
      if (!ok) raise_err(a.err, kDevErrTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs this loop; tcgen05 instructions are issued by one
    // elected lane inside each asm block (the same lane every time).
    constexpr uint32_t idesc_qk = umma_idesc_bf16_f32(BM, BN, 0, 0);
    constexpr uint32_t idesc_pv = umma_idesc_bf16_f32(BM, D, 0, 1);
    const uint64_t dq0 = umma_smem_desc_sw128(sQ, 16, 1024);
    const uint64_t dq1 = umma_smem_desc_sw128(sQ + C::QB, 16, 1024);
    const uint64_t dk = umma_smem_desc_sw128(sRing, 16, 1024);         // K: K-major
    const uint64_t dv = umma_smem_desc_sw128(sRing, C::PANEL_T, 1024);  // V: MN-major
    uint32_t fslot = 0, fphase = 0;  // next ring slot to consume
    uint32_t rslot = 0;              // next ring slot to release
    int uc = 0, tc = 0;
    bool ok = true;
    auto wait_full = [&](uint32_t& s) -> bool {
      if (!warp_wait(bar(C::B_FULL + fslot), fphase, abort_flag, a.wait_ns)) return false;
      s = fslot;
      if (++fslot == C::NSLOT) {
        fslot = 0;
        fphase ^= 1u;
      }
      return true;
    };
    auto release = [&]() {
      umma_commit_elect(bar(C::B_EMPTY + rslot));
      if (++rslot == C::NSLOT) rslot = 0;
    };
    auto commit = [&](int b) { umma_commit_elect(bar(b)); };
    // S_i = Q_i K^T over d
    auto qk = [&](int i, uint32_t ks) {
      const uint64_t kd = dk + ((ks * C::TB) >> 4);
      const uint32_t d_tm = tmem + static_cast<uint32_t>(i * BN);
      if constexpr (D == 128)
        umma_ss_k128_elect(d_tm, i ? dq1 : dq0, kd, idesc_qk);
      else
        umma_ss_k64_elect(d_tm, i ? dq1 : dq0, kd, idesc_qk);
      commit(C::B_SFULL + i);
    };
    // O_i (+)= P_i V over the tile's 128 keys, in two halves of 64 keys: each
    // half is issued as soon as the softmax has handed over its part of P
    auto pv = [&](int i, uint32_t vs, uint32_t acc) -> bool {
      const uint32_t o_tm = tmem + C::TM_O + static_cast<uint32_t>(i * D);
      const uint32_t p_tm = tmem + static_cast<uint32_t>(i * BN);
      const uint64_t vd = dv + ((vs * C::TB) >> 4);
      if (!warp_wait(bar(C::B_PRDY + 2 * i), tc & 1, abort_flag, a.wait_ns)) return false;
      tc_fence_after();
      umma_ts_k64keys_elect(o_tm, p_tm, vd, idesc_pv, acc);
      commit(C::B_PVH0 + i);  // a softmax that must rescale O before the second half waits for it
      if (!warp_wait(bar(C::B_PRDY + 2 * i + 1), tc & 1, abort_flag, a.wait_ns)) return false;
      tc_fence_after();
      umma_ts_k64keys_elect(o_tm, p_tm + 32, vd + 512, idesc_pv, 1u);
      return true;
    };
    for (int k = 0; ok && k * G < n_units; ++k) {
      const int u = unit_of(k, cta, G);
      Unit w;
      int lv, sb, pr;
      if (u >= n_units) continue;
      sched.map(u, lv, sb, pr);
      if (!decode_unit(a, lv, sb, pr, w)) continue;
      const int n = w.n_tiles;
      uint32_t ks = 0, vs = 0;
      if (!(ok = warp_wait(bar(C::B_QFULL + 0), uc & 1, abort_flag, a.wait_ns) && wait_full(ks))) break;
      tc_fence_after();
      qk(0, ks);
      if (n == 1) commit(C::B_QFREE + 0);
      if (!(ok = warp_wait(bar(C::B_QFULL + 1), uc & 1, abort_flag, a.wait_ns))) break;
      tc_fence_after();
      qk(1, ks);
      release();  // K(0)
      if (n == 1) commit(C::B_QFREE + 1);
      for (int j = 0; j < n; ++j, ++tc) {
        if (!(ok = wait_full(vs))) break;
        if constexpr (PAGED) {
          // slots past the sequence's keys may hold anything (even NaN): P is
          // 0 there, but 0 * NaN is not, so those V rows are cleared first
          const int valid = w.lk - (w.t_begin + j) * BN;
          if (valid < BN) {
            const int r0 = valid > 0 ? valid : 0;
            uint8_t* vt = gb + C::OFF_RING + vs * C::TB;
            for (int e = r0 * 8 + lane; e < BN * 8; e += 32)  // 16-byte pieces of 128-byte rows
#pragma unroll
              for (int p = 0; p < D / 64; ++p)
                *reinterpret_cast<uint4*>(vt + p * C::PANEL_T + e * 16) = make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
            __syncwarp();
          }
        }
        if (!(ok = pv(0, vs, j > 0 ? 1u : 0u))) break;
        if (j == n - 1) commit(C::B_OFULL + 0);
        if (j + 1 < n) {
          if (!(ok = wait_full(ks))) break;
          tc_fence_after();
          qk(0, ks);
          if (j + 1 == n - 1) commit(C::B_QFREE + 0);
        }
        if (!(ok = pv(1, vs, j > 0 ? 1u : 0u))) break;
        release();  // V(j)
        if (j == n - 1) commit(C::B_OFULL + 1);
        if (j + 1 < n) {
          qk(1, ks);
          release();  // K(j+1)
          if (j + 1 == n - 1) commit(C::B_QFREE + 1);
        }
      }
      if (!ok) break;
      ++uc;
    }
    // every MMA issued above has finished once this commit arrives
    commit(C::B_DRAIN);
    __syncwarp();
    mbar_wait(bar(C::B_DRAIN), 0, kDrainLimitNs);
    if (!ok && lane == 0) raise_err(a.err, kDevErrTimeout);
  } else {
    // ------------------------------------------------ softmax / epilogue
    // Eight warps per query tile. Warp (ti, q4, hh) owns the 16 rows q4*32 +
    // hh*16 .. +15 of tile ti (TMEM lanes of its quarter q4) and reaches them
    // with the 16-lane access shapes: thread t holds rows ra = t/4 and ra + 8
    // of those, key columns 8r + 2(t%4) + {0, 1} for r = 0..15. The four
    // threads of a quad share two rows; row max and sum are reduced with two
    // shuffles. P for keys (8r + 2(t%4), +1) is one bf16 pair, which belongs
    // in TMEM column 4r + t%4: exactly where the .16x128b store puts this
    // thread's register, so every warp reads S and writes P in its own 16
    // lanes only.
    const int ti = warp >> 3;                         // query tile of this warp
    const int q4 = warp & 3, hh = (warp >> 2) & 1;    // lane quarter, half of it
    const int jq = lane & 3;                          // thread within the quad
    const int ra = q4 * 32 + hh * 16 + (lane >> 2);   // row a of the tile; row b = ra + 8
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32 + hh * 16) << 16;
    const uint32_t tS = tmem + lane_off + static_cast<uint32_t>(ti * BN);
    const uint32_t tO = tmem + lane_off + C::TM_O + static_cast<uint32_t>(ti * D);
    const float sl2 = a.scale_log2;
    int uc = 0, tc = 0;
    bool ok = true;
    for (int k = 0; ok && k * G < n_units; ++k) {
      const int u = unit_of(k, cta, G);
      Unit w;
      int lv, sb, pr;
      if (u >= n_units) continue;
      sched.map(u, lv, sb, pr);
      if (!decode_unit(a, lv, sb, pr, w)) continue;
      const int q0 = w.q0[ti];
      const int qa = q0 + ra, qb = qa + 8;   // query rows within the sequence
      const int ia = w.qoff + qa;            // their positions among the keys (ib = ia + 8)
      const int p0 = w.qoff + q0;            // position of the tile's first row
      float ma = kNegInf, mb = kNegInf, la = 0.f, lb = 0.f;
      for (int j = 0; j < w.n_tiles; ++j, ++tc) {
        if (!(ok = warp_wait(bar(C::B_SFULL + ti), tc & 1, abort_flag, a.wait_ns))) break;
        tc_fence_after();
        const int kt0 = (w.t_begin + j) * BN;
        const bool need_mask = (kt0 + BN > w.lk) || (a.causal && kt0 + BN - 1 > p0) ||
                               (a.window > 0 && kt0 <= p0 + BM - 1 - a.window);
        // key column 8r + e + 2*jq of the tile is visible to a row iff
        // lo <= 8r + e < hi (bounds shifted by this thread's 2*jq)
        const int sh = kt0 + 2 * jq;
        const int lim = w.lk - sh;
        const int hia = a.causal ? min(lim, ia + 1 - sh) : lim;
        const int hib = a.causal ? min(lim, ia + 9 - sh) : lim;
        const int loa = a.window > 0 ? ia + 1 - a.window - sh : -BN;
        const int lob = loa + 8;
        const uint64_t sl2x2 = f2(sl2, sl2);
        uint64_t sa[2] = {0ull, 0ull}, sb2[2] = {0ull, 0ull};
        // Keys in two halves of 64. Each half: load its scores, take the
        // rows' max over the quad, move the running max if it grew by more
        // than 2^8 (lazy rescale, log2 domain), exponentiate, write P to TMEM
        // and hand it to the MMA warp, so PV of the first half runs while the
        // second is computed.
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t sr[32];
          tmem_ld16x256_x8(tS + 64 * hf, sr);
          tmem_wait_ld();
          if (need_mask) {
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int c = 64 * hf + 8 * r + e;
                if (c >= hia || c < loa) sr[4 * r + e] = __float_as_uint(kNegInf);
                if (c >= hib || c < lob) sr[4 * r + 2 + e] = __float_as_uint(kNegInf);
              }
          }
          float xa0 = fmaxf(__uint_as_float(sr[0]), __uint_as_float(sr[1]));
          float xa1 = fmaxf(__uint_as_float(sr[4]), __uint_as_float(sr[5]));
          float xb0 = fmaxf(__uint_as_float(sr[2]), __uint_as_float(sr[3]));
          float xb1 = fmaxf(__uint_as_float(sr[6]), __uint_as_float(sr[7]));
#pragma unroll
          for (int r = 2; r < 8; r += 2) {
            xa0 = fmax3(xa0, __uint_as_float(sr[4 * r]), __uint_as_float(sr[4 * r + 1]));
            xa1 = fmax3(xa1, __uint_as_float(sr[4 * r + 4]), __uint_as_float(sr[4 * r + 5]));
            xb0 = fmax3(xb0, __uint_as_float(sr[4 * r + 2]), __uint_as_float(sr[4 * r + 3]));
            xb1 = fmax3(xb1, __uint_as_float(sr[4 * r + 6]), __uint_as_float(sr[4 * r + 7]));
          }
          float mxa = fmaxf(xa0, xa1), mxb = fmaxf(xb0, xb1);
          mxa = fmaxf(mxa, __shfl_xor_sync(0xFFFFFFFFu, mxa, 1));
          mxb = fmaxf(mxb, __shfl_xor_sync(0xFFFFFFFFu, mxb, 1));
          mxa = fmaxf(mxa, __shfl_xor_sync(0xFFFFFFFFu, mxa, 2));
          mxb = fmaxf(mxb, __shfl_xor_sync(0xFFFFFFFFu, mxb, 2));
          const float mna = fmaxf(ma, mxa * sl2), mnb = fmaxf(mb, mxb * sl2);
          const bool rsa = mna > ma + kRescaleThreshold, rsb = mnb > mb + kRescaleThreshold;
          float ala = 1.f, alb = 1.f;
          if (rsa) {
            ala = ex2(ma - mna);  // 0 when ma = -inf
            ma = mna;
          }
          if (rsb) {
            alb = ex2(mb - mnb);
            mb = mnb;
          }
          la *= ala;
          lb *= alb;
          if (hf == 1) {
            // the first half's sums were taken with the old max
            sa[0] = fmul2(sa[0], f2(ala, ala));
            sa[1] = fmul2(sa[1], f2(ala, ala));
            sb2[0] = fmul2(sb2[0], f2(alb, alb));
            sb2[1] = fmul2(sb2[1], f2(alb, alb));
          }
          // O carries the same factor. Before the first hand-over of a tile
          // O is idle (PV of the previous tile finished before S was
          // signalled); before the second, PV of the first half may still
          // run, so its completion is waited for. On a tile's first half of
          // a unit's first tile O is about to be overwritten: nothing to do.
          if ((hf == 1 || j > 0) && __any_sync(0xFFFFFFFFu, rsa || rsb)) {
            if (hf == 1 && !(ok = warp_wait(bar(C::B_PVH0 + ti), tc & 1, abort_flag, a.wait_ns)))
              break;
            tc_fence_after();
            const uint64_t a2 = f2(ala, ala), b2 = f2(alb, alb);
#pragma unroll 1
            for (int c = 0; c < D / 16; ++c) {
              uint32_t o[8];
              tmem_ld16x256_x2(tO + 16 * c, o);
              tmem_wait_ld();
#pragma unroll
              for (int r = 0; r < 2; ++r) {
                float x0, x1;
                unf2(fmul2(f2(__uint_as_float(o[4 * r]), __uint_as_float(o[4 * r + 1])), a2), x0,
                     x1);
                o[4 * r] = __float_as_uint(x0);
                o[4 * r + 1] = __float_as_uint(x1);
                unf2(fmul2(f2(__uint_as_float(o[4 * r + 2]), __uint_as_float(o[4 * r + 3])), b2),
                     x0, x1);
                o[4 * r + 2] = __float_as_uint(x0);
                o[4 * r + 3] = __float_as_uint(x1);
              }
              tmem_st16x256_x2(tO + 16 * c, o);
            }
          }
          // p = 2^(s*scale*log2(e) - m) on pairs of scores
          const float mua = ma == kNegInf ? 0.f : ma, mub = mb == kNegInf ? 0.f : mb;
          const uint64_t nma = f2(-mua, -mua), nmb = f2(-mub, -mub);
          uint32_t pk[16];
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            float p0a, p1a, p0b, p1b;
            unf2(ffma2(f2(__uint_as_float(sr[4 * r]), __uint_as_float(sr[4 * r + 1])), sl2x2, nma),
                 p0a, p1a);
            unf2(ffma2(f2(__uint_as_float(sr[4 * r + 2]), __uint_as_float(sr[4 * r + 3])), sl2x2,
                       nmb),
                 p0b, p1b);
            p0a = ex2(p0a);
            p1a = ex2(p1a);
            p0b = ex2(p0b);
            p1b = ex2(p1b);
            sa[r & 1] = fadd2(sa[r & 1], f2(p0a, p1a));
            sb2[r & 1] = fadd2(sb2[r & 1], f2(p0b, p1b));
            pk[2 * r] = pack_bf16(p0a, p1a);
            pk[2 * r + 1] = pack_bf16(p0b, p1b);
          }
          tmem_st16x128_x8(tS + 32 * hf, pk);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(C::B_PRDY + 2 * ti + hf));
        }
        if (!ok) break;
        float u0, u1, v0, v1;
        unf2(fadd2(sa[0], sa[1]), u0, u1);
        unf2(fadd2(sb2[0], sb2[1]), v0, v1);
        la += u0 + u1;
        lb += v0 + v1;
      }
      if (!ok) break;
      if (!(ok = warp_wait(bar(C::B_OFULL + ti), uc & 1, abort_flag, a.wait_ns))) break;
      tc_fence_after();
      // the rows' sums over the whole quad
      la += __shfl_xor_sync(0xFFFFFFFFu, la, 1);
      lb += __shfl_xor_sync(0xFFFFFFFFu, lb, 1);
      la += __shfl_xor_sync(0xFFFFFFFFu, la, 2);
      lb += __shfl_xor_sync(0xFFFFFFFFu, lb, 2);
      const float inva = la > 0.f ? 1.f / la : 0.f, invb = lb > 0.f ? 1.f / lb : 0.f;
      const int h = w.h[ti];
      if (a.lse && jq == 0) {
        if (qa < w.len)
          a.lse[static_cast<int64_t>(h) * a.T + w.start + qa] =
              la > 0.f ? (ma + log2f(la)) * kLn2 : kNegInf;
        if (qb < w.len)
          a.lse[static_cast<int64_t>(h) * a.T + w.start + qb] =
              lb > 0.f ? (mb + log2f(lb)) * kLn2 : kNegInf;
      }
      // O / l in place for this warp's 16 rows ...
      const uint64_t ia2 = f2(inva, inva), ib2 = f2(invb, invb);
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[16];
        tmem_ld16x256_x4(tO + 32 * c, o);
        tmem_wait_ld();
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          float x0, x1;
          unf2(fmul2(f2(__uint_as_float(o[4 * r]), __uint_as_float(o[4 * r + 1])), ia2), x0, x1);
          o[4 * r] = __float_as_uint(x0);
          o[4 * r + 1] = __float_as_uint(x1);
          unf2(fmul2(f2(__uint_as_float(o[4 * r + 2]), __uint_as_float(o[4 * r + 3])), ib2), x0,
               x1);
          o[4 * r + 2] = __float_as_uint(x0);
          o[4 * r + 3] = __float_as_uint(x1);
        }
        tmem_st16x256_x4(tO + 32 * c, o);
      }
      tmem_wait_st();
      // ... then, once the other warp of this lane quarter has done the same,
      // this warp stores half of the columns of all 32 rows of the quarter:
      // the 32x32b shape gives each thread one row's consecutive columns, so
      // every store is a whole 32-byte sector
      tc_fence_before();
      mbar_arrive(bar(C::B_EPI + 4 * ti + q4));
      if (!(ok = warp_wait(bar(C::B_EPI + 4 * ti + q4), uc & 1, abort_flag, a.wait_ns))) break;
      tc_fence_after();
      const int row = q0 + q4 * 32 + lane;  // query row within the sequence
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.o) +
                            (static_cast<int64_t>(w.start + row) * a.Hq + h) * D + hh * (D / 2);
      const uint32_t tq = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + C::TM_O +
                          static_cast<uint32_t>(ti * D + hh * (D / 2));
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t o[32];
        tmem_ld32(tq + 32 * c, o);
        tmem_wait_ld();
        if (row < w.len) {
          uint32_t wv[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            wv[e] = pack_bf16(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1]));
          st_global_v8(orow + 32 * c, wv);
          st_global_v8(orow + 32 * c + 16, wv + 8);
        }
      }
      ++uc;
    }
    if (!ok && lane == 0) raise_err(a.err, kDevErrTimeout);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
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

int g_pf_attr[4][64];

template <int D, bool PAGED>
void ensure_pf_attr() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  const int v = (D == 128) + 2 * PAGED;
  if (!g_pf_attr[v][dev]) {
    cudaFuncSetAttribute(prefill_bf16_kernel<D, PAGED>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, PfCfg<D>::SMEM);
    g_pf_attr[v][dev] = 1;
  }
}

template <int D, bool PAGED>
void launch_pf(unsigned grid, const CUtensorMap& qmap, const CUtensorMap& kmap,
               const CUtensorMap& vmap, const PrefillArgs& a, cudaStream_t s) {
  ensure_pf_attr<D, PAGED>();
  prefill_bf16_kernel<D, PAGED><<<grid, kThreads, PfCfg<D>::SMEM, s>>>(qmap, kmap, vmap, a);
}

}  // namespace

size_t prefill_bf16_smem(int d) { return d == 128 ? PfCfg<128>::SMEM : PfCfg<64>::SMEM; }

long long prefill_units(int B, int Hq, int Hkv, int max_seqlen, bool* pair_heads) {
  const long long n_qt = (max_seqlen + BM - 1) / BM;
  const bool pair = ((Hq / Hkv) % 2) == 0;
  if (pair_heads) *pair_heads = pair;
  return pair ? n_qt * (Hq / 2) * B : ((n_qt + 1) / 2) * Hq * static_cast<long long>(B);
}

cudaError_t launch_prefill_bf16(const PrefillArgs& a0, const CUtensorMap& qmap,
                                const CUtensorMap& kmap, const CUtensorMap& vmap, int num_sms,
                                cudaStream_t s) {
  PrefillArgs a = a0;
  bool pair = false;
  const long long units = prefill_units(a.B, a.Hq, a.Hkv, a.max_seqlen, &pair);
  if (units == 0) return cudaSuccess;
  if (units > INT_MAX) return cudaErrorInvalidConfiguration;
  a.pair_heads = pair ? 1 : 0;
  a.n_units = static_cast<int>(units);
  a.compact = (a.cu_seqlens && a.B <= kMaxSchedSeqs && (a.max_seqlen + BM - 1) / BM <= 65535) ? 1 : 0;
  const unsigned grid = static_cast<unsigned>(units < num_sms ? units : num_sms);
  const bool paged = a.table != nullptr;
  if (a.d == 128) {
    if (paged) launch_pf<128, true>(grid, qmap, kmap, vmap, a, s);
    else launch_pf<128, false>(grid, qmap, kmap, vmap, a, s);
  } else {
    if (paged) launch_pf<64, true>(grid, qmap, kmap, vmap, a, s);
    else launch_pf<64, false>(grid, qmap, kmap, vmap, a, s);
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
