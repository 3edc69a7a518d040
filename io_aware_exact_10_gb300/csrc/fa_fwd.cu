// fa_fwd.cu -- exact softmax attention forward for sm_103a.
//
// Computes O = softmax(scale * Q K^T [causal]) V and the per-row natural-log
// log-sum-exp, tiled so the Nq x Nk score matrix never leaves the SM
// (FlashAttention: exact attention made fast by counting memory traffic,
// "The method"; Flash Attention (ostralyan.com), "Block-Wise Attention
// Computation" and "Core Flash Attention Algorithm").
//
// One CTA owns two 128-row query tiles of one (batch, head) and streams the
// head's 128-key K/V tiles through a TMA ring.  Roles (320 threads):
//   warps 0-3  softmax for query tile 0 (thread = query row = TMEM lane)
//   warps 4-7  softmax for query tile 1
//   warp  8    TMA producer (Q tiles once, then K_0, V_0, K_1, V_1, ...)
//   warp  9    tcgen05 MMA issuer (one thread) and TMEM owner
// Tensor memory (512 columns) at d = 128: S_0 | S_1 | O_0 | O_1.  The softmax
// writes P as bf16 pairs into the first 64 columns of its S region and the
// MMA reads it from there as the A operand of O += P V.  The two query tiles
// alternate on the tensor core: while one tile's softmax runs, the other
// tile's O += P V and S = Q K^T run.
// At d = 64: S_0 | S_1 | P_0 | P_1 | O_0 | O_1.  With P in columns of its own,
// the softmax takes its whole S row into registers and releases S at once,
// so S_t(j+1) is computed while the softmax of step j runs; "P_t free"
// (PV_t(j-1) complete) guards the P store and the rare rescale of O.
//
// Online softmax in base 2 with the scale folded into one FMA: the running
// max m and normaliser l of each row follow the recurrence of Flash Attention,
// "Online Softmax Algorithm"; O stays unnormalised and is divided by l once at
// the end, and one log-sum-exp per row is written (FlashAttention and
// IO-aware exact attention, "Core ideas").  The max is updated lazily: a new
// max within TAU (log2 units) of the current one is not adopted, which keeps
// P <= 2^TAU and skips the rescale of O in TMEM; the result is the same in
// exact arithmetic because l and O always share one reference max.
#include <cuda_bf16.h>

#include "fa_kernels.h"

namespace fa {
namespace {

constexpr float kTau = 8.0f;
constexpr int kSplit = 1;  // softmax warpgroups per query tile (2 measured no faster)
constexpr float kLn2 = 0.6931471805599453f;

template <int HD, int NH, int BN_ = 128, bool STG = false>
struct FwdCfg {
  static constexpr int BM = 128;                  // query rows per tile
  static constexpr int BN = BN_;                  // keys per K/V tile (128, or 64)
  static constexpr int KB = HD / 64;              // 64-column (128-byte) blocks per row
  static constexpr int QTILE = BM * HD * 2;       // bytes of one Q tile
  static constexpr int KVTILE = BN * HD * 2;      // bytes of one K or V tile
  // the ring holds 128 KB of K/V tiles whatever their size
  static constexpr int STAGES = (HD == 128 ? 4 : 8) * (128 / BN);
  // Q buffers per query tile: two in the staged kernels (d = 64, persistent
  // launches), so that the next item's Q loads while the current item's S
  // still read theirs and the epilogue can stage O in the finished one (at
  // d = 128 the ring leaves no room for a second pair)
  static constexpr int QBUF = STG ? 2 : 1;
  static constexpr int SMEM = 2 * QBUF * QTILE + STAGES * KVTILE + 1024;
  // NH warpgroups share each query tile's softmax, each taking 128 / NH of
  // the key columns; then come the TMA warp and the MMA warp.
  static constexpr int WS = 8 * NH;               // softmax warps
  static constexpr int W_LOAD = WS, W_MMA = WS + 1;
  static constexpr int THREADS = (WS + 2) * 32;
  static constexpr int CPT = BN / NH;             // key columns per softmax thread
  static constexpr int OCPT = HD / NH;            // O columns per softmax thread
  static constexpr uint32_t TMEM_COLS = 512;
  // P in columns of its own (d = 64 only: with 128-key tiles, S, P and O of
  // two tiles fill the 512)
  static constexpr bool SEPP = HD == 64 && NH == 1;
  static constexpr uint32_t colS(int t) { return (uint32_t)t * BN; }
  static constexpr uint32_t colP(int t) {
    return SEPP ? 2 * BN + (uint32_t)t * (BN / 2) : (uint32_t)t * BN;
  }
  static constexpr uint32_t colO(int t) {
    return SEPP ? 3 * BN + (uint32_t)t * HD : 2 * BN + (uint32_t)t * HD;
  }
  static_assert(BN == 128 || (BN == 64 && NH == 1), "64-key tiles: one softmax warpgroup per tile");
  static_assert(colO(1) + HD <= TMEM_COLS, "tensor memory plan");
};

struct FwdParams {
  __nv_bfloat16* o;
  float* lse;
  int Nq, Nk;    // query rows and keys per head
  int nq, nkv, npairs, BH, group;
  int kv_group;  // query heads per key/value head (1: multi-head)
  int coff;      // causal offset Nk - Nq: query i sees keys j <= i + coff
  const uint8_t* bmask;  // block mask [nq][nkv] (block-sparse kernels only)
  float scale2;  // scale * log2(e)
  KernelCtl ctl;
};

// Warp-uniform bounded wait: every lane polls, all agree on the outcome.
template <bool TEST_FIRST = true>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const KernelCtl& ctl,
                                          volatile int* abort, uint32_t site) {
  const bool ok = mbar_wait<TEST_FIRST>(bar, parity, ctl, abort, site);
  return __all_sync(0xffffffffu, ok);
}

// Phases of up to three barriers tested in one shared-memory round trip: the
// tests are issued back to back and combined before the result is read
// (a completed phase costs ~250 cycles of round trip inside the busy kernel;
// three separate tests pay it three times).
__device__ __forceinline__ bool mbar_test3(uint32_t b0, uint32_t p0, uint32_t b1, uint32_t p1, uint32_t b2,
                                           uint32_t p2) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred q0, q1, q2;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q0, [%1], %2;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q1, [%3], %4;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q2, [%5], %6;\n\t"
      "and.pred q0, q0, q1;\n\t"
      "and.pred q0, q0, q2;\n\t"
      "selp.u32 %0, 1, 0, q0;\n\t}"
      : "=r"(ok)
      : "r"(b0), "r"(p0), "r"(b1), "r"(p1), "r"(b2), "r"(p2)
      : "memory");
  return ok != 0;
}

// TMEM column (relative to S_t) of the bf16 pairs of P for K-step k (16 keys
// of the P V contraction).  Each softmax warpgroup packs its keys into the
// first half of its own, already read, column range.
template <int NH>
__device__ __forceinline__ uint32_t p_col(int k) {
  return NH == 1 ? (uint32_t)(k * 8) : (uint32_t)(k * 8 + (k >= 4 ? 32 : 0));
}

template <int HD, bool CAUSAL, int NH, bool SPARSE, int BN = 128, bool STG = false>
__global__ void __launch_bounds__((8 * NH + 2) * 32, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                  const FwdParams p) {
  using C = FwdCfg<HD, NH, BN, STG>;
  static_assert(!STG || (HD == 64 && !SPARSE), "staged kernels: dense d = 64");
  // First poll of every wait a non-blocking test at d = 64 (measured 4-5 % faster there);
  // at d = 128 the plain suspending wait (the test measured 1-2 % slower).
  constexpr bool TF = HD == 64;
  // The d = 64 MMA loop's waits: 0 = each barrier tested on its own; 2 = a
  // tile's K or V landing tested with its S read (or P stored) in one round
  // trip; 3 = both tiles' barriers and the K or V landing in one.  Chosen per
  // kernel by measurement (alternating runs on one GPU): 3 on one-item and
  // long-item launches (+2-3 % at N = 4096-16384 causal, +20 % with 64-key
  // tiles), 2 on the staged kernel with 64-key tiles (+17 %), 0 on the staged
  // kernel with 128-key tiles (1-2 % ahead of both).
  constexpr int BATCH = STG ? (BN == 64 ? 2 : 0) : 3;
  static_assert(BN == 128 || !SPARSE, "block masks are over 128 x 128 blocks");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);

  // Q buffer b of tile t: index 2 b + t.  It is free again once the last S of
  // its item has completed (one Q buffer per tile), or, with two, once the
  // item's epilogue has staged O in it and the TMA store has read it.
  __shared__ __align__(8) uint64_t bar_q[2 * C::QBUF];
  __shared__ __align__(8) uint64_t bar_qe[2 * C::QBUF];
  __shared__ __align__(8) uint64_t bar_full[C::STAGES];
  __shared__ __align__(8) uint64_t bar_empty[C::STAGES];
  __shared__ __align__(8) uint64_t bar_s[2];
  __shared__ __align__(8) uint64_t bar_p[2];
  __shared__ __align__(8) uint64_t bar_o[2];
  __shared__ __align__(8) uint64_t bar_of[2];  // O_t free: read by the previous item's epilogue
  __shared__ __align__(8) uint64_t bar_sf[2];  // S_t read by its softmax (P in own columns)
  __shared__ __align__(8) uint64_t bar_pf[2];  // PV_t complete (P in own columns)
  __shared__ __align__(8) uint64_t bar_drain;
  __shared__ __align__(8) uint64_t bar_x[2][4];  // partner-warp exchange (NH == 2)
  __shared__ float xch[2][2][2][128];             // [tile][parity][half][row]
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  volatile int* abort = &abort_sh;
  // block-sparse: the key tiles query tile 0 keeps, tile 1 keeps, and their
  // union (the tiles the pair streams); mcount holds their sizes
  __shared__ uint32_t mbits[SPARSE ? 3 * kMaskWords : 1];
  __shared__ int mcount[3];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work items are the query-tile pairs of every head, in a one-dimensional
  // order over (head group, pair rank, head): the pairs that share a head's
  // K and V run together and find them in L2, and within a group the
  // heaviest (causal) pairs come first.  Persistent launches (see
  // persistent_launch) have one CTA per SM (G CTAs), and CTA b takes items b,
  // 2G-1-b, 2G+b, 4G-1-b, ...: each pass over G items runs the other way, so
  // causal CTAs pair heavy items with light ones, and the next item's Q and
  // K/V loads and first S overlap the current item's last steps and
  // epilogue.  Other launches have one CTA per item.  Every role walks the
  // same items; the ring index and the barrier phases run on across items.
  const int n_items = p.npairs * p.BH;
  const int L0 = (int)blockIdx.x, LS = (int)gridDim.x;
  // k-th item (k >= 1); a block-sparse CTA has one item, which the compiler
  // then knows: its item loops run once
  auto item_at = [&](int k) { return SPARSE ? n_items : k * LS + ((k & 1) ? LS - 1 - L0 : L0); };
  struct Item {
    int bh, bhkv, qt0;
    bool valid[2];
    int nkv_t[2];  // causal: key tiles up to the one its last row's last key is in
    int ntile[2];  // key tiles query tile t visits
    int nu;        // key tiles the pair streams
  };
  auto item_info = [&](int L) {
    Item I;
    const GridPos gp = decode_grid(L, p.BH, p.npairs, p.group);
    I.bh = gp.bh;
    I.bhkv = gp.bh / p.kv_group;  // key/value head of this query head
    I.qt0 = 2 * (p.npairs - 1 - gp.rank);
    #pragma unroll
    for (int t = 0; t < 2; ++t) {
      I.valid[t] = I.qt0 + t < p.nq;
      I.nkv_t[t] = !I.valid[t] ? 0
                   : (CAUSAL ? min(((I.qt0 + t) * C::BM + C::BM - 1 + p.coff) / C::BN + 1, p.nkv)
                             : p.nkv);
      I.ntile[t] = I.nkv_t[t];
    }
    I.nu = max(I.nkv_t[0], I.nkv_t[1]);
    return I;
  };
  // Key tiles each query tile visits and the tiles the pair streams: dense,
  // tiles 0 .. nkv_t-1 and 0 .. max(nkv_t)-1; block-sparse, the tiles the
  // mask keeps within those bounds, in ascending order.  The TMA warp builds
  // the bitsets of the CTA's one item; the other warps read the counts after
  // the CTA-wide sync.
  Item I0 = item_info(L0);
  const int nw = (p.nkv + 31) >> 5;
  uint32_t* const ubits = mbits + (SPARSE ? 2 * kMaskWords : 0);
  if constexpr (SPARSE) {
    if (warp == C::W_LOAD) {
      #pragma unroll
      for (int t = 0; t < 2; ++t)
        mask_bits_warp(p.bmask + (I0.valid[t] ? (size_t)(I0.qt0 + t) * p.nkv : 0), 1, 0,
                       I0.valid[t] ? I0.nkv_t[t] : 0, nw, mbits + t * kMaskWords, lane);
      __syncwarp();
      for (int w = lane; w < nw; w += 32) ubits[w] = mbits[w] | mbits[kMaskWords + w];
      __syncwarp();
      I0.ntile[0] = mask_popc_warp(mbits, nw, lane);
      I0.ntile[1] = mask_popc_warp(mbits + kMaskWords, nw, lane);
      I0.nu = mask_popc_warp(ubits, nw, lane);
      if (lane == 0) {
        mcount[0] = I0.ntile[0];
        mcount[1] = I0.ntile[1];
        mcount[2] = I0.nu;
      }
    }
  }

  const uint32_t sQ = smem_u32(smem);
  const uint32_t sRing = sQ + 2 * C::QBUF * C::QTILE;

  // The TMA thread initialises the barriers and issues the copies that need
  // no wait (the Q tiles and the first ring slots) before the CTA-wide sync,
  // so their latency overlaps the rest of the set-up.  Ring index it holds
  // K_j (it even) or V_j (it odd) of the pair's (it/2)-th key tile j.
  auto issue_kv = [&](int it, int j, int bhkv) {
    const int slot = it % C::STAGES;
    const uint32_t bar = smem_u32(&bar_full[slot]);
    mbar_arrive_expect_tx(bar, C::KVTILE);
    const uint32_t dst = sRing + slot * C::KVTILE;
    for (int b = 0; b < C::KB; ++b)
      tma_load_3d(dst + b * C::BN * 128, (it & 1) ? &tv : &tk, bar, b * 64, j * C::BN, bhkv);
  };
  auto issue_q = [&](int t, const Item& I, int qb) {
    const int qi = 2 * qb + t;
    const uint32_t bar = smem_u32(&bar_q[qi]);
    mbar_arrive_expect_tx(bar, C::QTILE);
    for (int b = 0; b < C::KB; ++b)
      tma_load_3d(sQ + qi * C::QTILE + b * C::BM * 128, &tq, bar, b * 64, (I.qt0 + t) * C::BM, I.bh);
  };
  auto live = [](const Item& I, int t) { return I.valid[t] && I.ntile[t] > 0; };
  const int pre_it = 2 * I0.nu < C::STAGES ? 2 * I0.nu : C::STAGES;  // issued before the sync
  int jw = 0;  // the TMA thread's key tile (of ring index it; block-sparse)
  if (warp == C::W_LOAD && lane == 0) {
    abort_sh = 0;
    #pragma unroll
    for (int t = 0; t < 2; ++t) {
      for (int qb = 0; qb < C::QBUF; ++qb) {
        mbar_init(smem_u32(&bar_q[2 * qb + t]), 1);
        mbar_init(smem_u32(&bar_qe[2 * qb + t]), C::QBUF == 2 ? 4 : 1);
      }
      mbar_init(smem_u32(&bar_s[t]), 1);
      mbar_init(smem_u32(&bar_p[t]), 4 * NH);
      for (int sp = 0; sp < 4; ++sp) mbar_init(smem_u32(&bar_x[t][sp]), 64);
      mbar_init(smem_u32(&bar_o[t]), 1);
      mbar_init(smem_u32(&bar_of[t]), 4 * NH);
      mbar_init(smem_u32(&bar_sf[t]), 4 * NH);
      mbar_init(smem_u32(&bar_pf[t]), 1);
    }
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&bar_full[s]), 1);
      mbar_init(smem_u32(&bar_empty[s]), 1);
    }
    mbar_init(smem_u32(&bar_drain), 1);
    fence_barrier_init();
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    if (C::QBUF == 2) tma_prefetch_desc(&to);
    #pragma unroll
    for (int t = 0; t < 2; ++t)
      if (live(I0, t)) issue_q(t, I0, 0);
    if constexpr (SPARSE) jw = next_bit(ubits, nw, -1);
    for (int it = 0; it < pre_it; ++it) {
      issue_kv(it, SPARSE ? jw : it >> 1, I0.bhkv);
      if (SPARSE && (it & 1)) jw = next_bit(ubits, nw, jw);
    }
  }
  if (warp == C::W_MMA) {
    tmem_alloc(smem_u32(&tmem_base_sh), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  if constexpr (SPARSE) {
    I0.ntile[0] = mcount[0];
    I0.ntile[1] = mcount[1];
    I0.nu = mcount[2];
  }
  if (warp == C::W_LOAD) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      int it = pre_it;  // ring index, across items
      int nql[2] = {live(I0, 0) ? 1 : 0, live(I0, 1) ? 1 : 0};  // Q_t loads issued
      bool ok = true;
      Item I = I0;
      int i = pre_it;  // ring use within the item
      for (int L = L0, kk = 0;;) {
        for (; i < 2 * I.nu; ++i, ++it) {
          const int slot = it % C::STAGES, use = it / C::STAGES;
          if (use > 0 && !mbar_wait<TF>(smem_u32(&bar_empty[slot]), (use - 1) & 1, p.ctl, abort, 10)) {
            ok = false;
            break;
          }
          issue_kv(it, SPARSE ? jw : i >> 1, I.bhkv);
          if (SPARSE && (i & 1)) jw = next_bit(ubits, nw, jw);
        }
        if (!ok) break;
        L = item_at(++kk);
        if (L >= n_items) break;
        I = item_info(L);
        // the next item's Q_t, once the MMA no longer reads the previous one
        #pragma unroll
        for (int t = 0; t < 2 && ok; ++t) {
          if (!live(I, t)) continue;
          const int qb = nql[t] % C::QBUF;
          if (nql[t] >= C::QBUF &&
              !mbar_wait<TF>(smem_u32(&bar_qe[2 * qb + t]), ((nql[t] - C::QBUF) / C::QBUF) & 1, p.ctl, abort, 11)) {
            ok = false;
            break;
          }
          issue_q(t, I, qb);
          ++nql[t];
        }
        if (!ok) break;
        i = 0;
      }
      if (!ok) {
        // Abort: let the copies already issued land before the CTA exits.
        for (int s = 0; s < C::STAGES && s < it; ++s)
          mbar_wait_quiet(smem_u32(&bar_full[s]), ((it - 1 - s) / C::STAGES) & 1, 200000000ull);
        #pragma unroll
        for (int t = 0; t < 2; ++t)
          for (int n = nql[t] > C::QBUF ? nql[t] - C::QBUF : 0; n < nql[t]; ++n)
            mbar_wait_quiet(smem_u32(&bar_q[2 * (n % C::QBUF) + t]), (n / C::QBUF) & 1, 200000000ull);
      }
    }
  } else if (warp == C::W_MMA) {
    // ------------------------------------------------------------------ MMA
    // The whole warp runs the issue loop (control flow and descriptors stay
    // warp-uniform); one elected lane issues.
    {
      const uint32_t lead = elect_one();
      constexpr uint32_t kIdS = idesc_bf16(128, C::BN, false, false);
      constexpr uint32_t kIdPV = idesc_bf16(128, HD, false, true);
      // descriptor halves (sdesc_lo / sdesc_hi) of Q tile 0 and ring slot 0
      constexpr uint32_t HI = sdesc_hi(1024);
      // 64-column blocks of a Q tile (128 rows) and of a K tile (BN rows), in 16-byte units
      constexpr uint32_t QT16 = C::QTILE >> 4, KV16 = C::KVTILE >> 4, QBLK16 = (C::BM * 128) >> 4,
                         KBLK16 = (C::BN * 128) >> 4;
      const uint32_t qK = sdesc_lo(sQ, 16), rK = sdesc_lo(sRing, 16), rMN = sdesc_lo(sRing, C::BN * 128);
      // S_t = Q_t K^T for the K tile in ring slot `slot`.
      int qb[2] = {0, 0};  // the item's Q buffer of each tile
      auto issue_s = [&](int t, int slot) {
        const uint32_t a0 = qK + (uint32_t)(2 * qb[t] + t) * QT16, b0 = rK + (uint32_t)slot * KV16;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t koff = (uint32_t)(k % 4) * 2;
          mma_ss_e(lead, tmem + C::colS(t), a0 + (uint32_t)(k / 4) * QBLK16 + koff, HI,
                   b0 + (uint32_t)(k / 4) * KBLK16 + koff, HI, kIdS, k > 0);
        }
        mma_commit_e(lead, smem_u32(&bar_s[t]));
      };
      // O_t (+)= P_t V for the V tile in ring slot `slot`.
      auto issue_pv = [&](int t, int slot, bool acc) {
        const uint32_t b0 = rMN + (uint32_t)slot * KV16;
#pragma unroll
        for (int k = 0; k < C::BN / 16; ++k)
          mma_ts_e(lead, tmem + C::colO(t), tmem + C::colP(t) + p_col<NH>(k), b0 + 128 * k, HI, kIdPV,
                   (acc || k > 0) ? 1u : 0u);
      };

      // Per query tile, across items: S issued, O += P V issued (barrier
      // phases follow them), Q_t waits, and items whose O_t was committed.
      int cs[2] = {0, 0}, cp[2] = {0, 0}, nqw[2] = {0, 0}, no[2] = {0, 0};
      int it0 = 0;  // ring index of the item's first K
      bool ok = true;
      for (int L = L0, kk = 0; L < n_items && ok; L = item_at(++kk)) {
        const Item I = L == L0 ? I0 : item_info(L);
        #pragma unroll
        for (int t = 0; t < 2 && ok; ++t)
          if (live(I, t)) {
            qb[t] = nqw[t] % C::QBUF;
            ok = warp_wait<TF>(smem_u32(&bar_q[2 * qb[t] + t]), (nqw[t] / C::QBUF) & 1, p.ctl, abort, 20);
            ++nqw[t];
          }
        if (!ok) break;
        // Does query tile t use key tile j?  The next key tile of the pair.
        auto active = [&](int t, int j) -> bool {
          if constexpr (SPARSE)
            return ((mbits[t * kMaskWords + (j >> 5)] >> (j & 31)) & 1u) != 0;
          else
            return I.valid[t] && j < I.nkv_t[t];
        };
        auto next_j = [&](int j) -> int {
          if constexpr (SPARSE)
            return next_bit(ubits, nw, j);
          else
            return j + 1;
        };
        int ls[2] = {0, 0}, lp[2] = {0, 0};  // S and O += P V issued in this item
        // S_t for the K tile in ring slot ks, with the item's Q_t released
        // after its last S_t.
        auto s_step = [&](int t, int ks) {
          issue_s(t, ks);
          ++cs[t];
          if (++ls[t] == I.ntile[t] && C::QBUF == 1) mma_commit_e(lead, smem_u32(&bar_qe[t]));
        };
        // O_t (+)= P_t V for the V tile in ring slot vs.  The item's first one
        // overwrites O_t: the previous item's epilogue must have read it.
        auto pv_step = [&](int t, int vs) -> bool {
          if (lp[t] == 0 && no[t] > 0 &&
              !warp_wait<TF>(smem_u32(&bar_of[t]), (no[t] - 1) & 1, p.ctl, abort, 27))
            return false;
          if (!warp_wait<TF>(smem_u32(&bar_p[t]), cp[t] & 1, p.ctl, abort, 23)) return false;
          tc_fence_after();
          issue_pv(t, vs, lp[t] > 0);
          if constexpr (C::SEPP) mma_commit_e(lead, smem_u32(&bar_pf[t]));
          ++cp[t];
          if (++lp[t] == I.ntile[t]) {
            mma_commit_e(lead, smem_u32(&bar_o[t]));
            ++no[t];
          }
          return true;
        };

        if constexpr (C::SEPP) {
          // The pair's q-th key tile u_q has K at ring index it0 + 2q, V at
          // it0 + 2q + 1.  Per q, with j = u_q and jn = u_{q+1}:
          //   [S_t read] S_t(jn);  [P_t ready] O_t += P_t V_j
          // S_t overwrites S_t only after the softmax has read it (also the
          // last S_t of the previous item).
          int j = SPARSE ? next_bit(ubits, nw, -1) : 0;
          if constexpr (BATCH >= 2) {
          // S_0(jn), S_1(jn) once K(jn) has landed and both S have been read:
          // one round trip tests all three.
          auto s_pair = [&](int ks, uint32_t kpar, bool a0, bool a1) -> bool {
            const uint32_t kb = smem_u32(&bar_full[ks]);
            const bool w0 = a0 && cs[0] > 0, w1 = a1 && cs[1] > 0;
            const uint32_t f0 = smem_u32(&bar_sf[0]), f1 = smem_u32(&bar_sf[1]);
            const uint32_t q0 = (uint32_t)(cs[0] - 1) & 1u, q1 = (uint32_t)(cs[1] - 1) & 1u;
            if (!__all_sync(0xffffffffu, mbar_test3(kb, kpar, w0 ? f0 : kb, w0 ? q0 : kpar, w1 ? f1 : kb,
                                                     w1 ? q1 : kpar))) {
              if (!warp_wait<TF>(kb, kpar, p.ctl, abort, 24)) return false;
              if (w0 && !warp_wait<TF>(f0, q0, p.ctl, abort, 26)) return false;
              if (w1 && !warp_wait<TF>(f1, q1, p.ctl, abort, 26)) return false;
            }
            tc_fence_after();
            if (a0) s_step(0, ks);
            if (a1) s_step(1, ks);
            return true;
          };
          // O_0 += P_0 V_j, O_1 += P_1 V_j once V_j has landed and both P are
          // stored (the item's first P V also waits for the epilogue to free O_t).
          auto pv_pair = [&](int vs, uint32_t vpar, bool a0, bool a1) -> bool {
            #pragma unroll
            for (int t = 0; t < 2; ++t)
              if ((t ? a1 : a0) && lp[t] == 0 && no[t] > 0 &&
                  !warp_wait<TF>(smem_u32(&bar_of[t]), (no[t] - 1) & 1, p.ctl, abort, 27))
                return false;
            const uint32_t vb = smem_u32(&bar_full[vs]);
            const uint32_t g0 = smem_u32(&bar_p[0]), g1 = smem_u32(&bar_p[1]);
            const uint32_t q0 = (uint32_t)cp[0] & 1u, q1 = (uint32_t)cp[1] & 1u;
            if (!__all_sync(0xffffffffu, mbar_test3(vb, vpar, a0 ? g0 : vb, a0 ? q0 : vpar, a1 ? g1 : vb,
                                                     a1 ? q1 : vpar))) {
              if (!warp_wait<TF>(vb, vpar, p.ctl, abort, 22)) return false;
              if (a0 && !warp_wait<TF>(g0, q0, p.ctl, abort, 23)) return false;
              if (a1 && !warp_wait<TF>(g1, q1, p.ctl, abort, 23)) return false;
            }
            tc_fence_after();
            #pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (!(t ? a1 : a0)) continue;
              issue_pv(t, vs, lp[t] > 0);
              mma_commit_e(lead, smem_u32(&bar_pf[t]));
              ++cp[t];
              if (++lp[t] == I.ntile[t]) {
                mma_commit_e(lead, smem_u32(&bar_o[t]));
                ++no[t];
              }
            }
            return true;
          };
          // both tiles behind one test, or each tile behind its own
          auto s_all = [&](int ks, uint32_t kpar, bool a0, bool a1) -> bool {
            if (BATCH == 3) return s_pair(ks, kpar, a0, a1);
            return (!a0 || s_pair(ks, kpar, true, false)) && (!a1 || s_pair(ks, kpar, false, true));
          };
          auto pv_all = [&](int vs, uint32_t vpar, bool a0, bool a1) -> bool {
            if (BATCH == 3) return pv_pair(vs, vpar, a0, a1);
            return (!a0 || pv_pair(vs, vpar, true, false)) && (!a1 || pv_pair(vs, vpar, false, true));
          };
          if (I.nu > 0) {
            const int ks = it0 % C::STAGES;
            ok = s_all(ks, (uint32_t)(it0 / C::STAGES) & 1u, active(0, j), active(1, j));
            if (ok) mma_commit_e(lead, smem_u32(&bar_empty[ks]));
          }
          for (int q = 0; q < I.nu && ok; ++q) {
            const int jn = q + 1 < I.nu ? next_j(j) : -1;
            if (q + 1 < I.nu) {
              const int ik = it0 + 2 * (q + 1), ks = ik % C::STAGES;
              if (!(ok = s_all(ks, (uint32_t)(ik / C::STAGES) & 1u, active(0, jn), active(1, jn)))) break;
              mma_commit_e(lead, smem_u32(&bar_empty[ks]));
            }
            const int iv = it0 + 2 * q + 1, vs = iv % C::STAGES;
            if (!(ok = pv_all(vs, (uint32_t)(iv / C::STAGES) & 1u, active(0, j), active(1, j)))) break;
            mma_commit_e(lead, smem_u32(&bar_empty[vs]));
            j = jn;
          }
          } else {
          auto s_after_read = [&](int t, int ks) -> bool {
            if (cs[t] > 0 && !warp_wait<TF>(smem_u32(&bar_sf[t]), (cs[t] - 1) & 1, p.ctl, abort, 26))
              return false;
            tc_fence_after();
            s_step(t, ks);
            return true;
          };
          if (I.nu > 0) {
            const int ks = it0 % C::STAGES;
            ok = warp_wait<TF>(smem_u32(&bar_full[ks]), (it0 / C::STAGES) & 1, p.ctl, abort, 21);
            if (ok) {
              tc_fence_after();
              #pragma unroll
              for (int t = 0; t < 2 && ok; ++t)
                if (active(t, j)) ok = s_after_read(t, ks);
              if (ok) mma_commit_e(lead, smem_u32(&bar_empty[ks]));
            }
          }
          for (int q = 0; q < I.nu && ok; ++q) {
            const int jn = q + 1 < I.nu ? next_j(j) : -1;
            if (q + 1 < I.nu) {
              const int ik = it0 + 2 * (q + 1), ks = ik % C::STAGES;
              if (!(ok = warp_wait<TF>(smem_u32(&bar_full[ks]), (ik / C::STAGES) & 1, p.ctl, abort, 24))) break;
              #pragma unroll
              for (int t = 0; t < 2 && ok; ++t)
                if (active(t, jn)) ok = s_after_read(t, ks);
              if (!ok) break;
              mma_commit_e(lead, smem_u32(&bar_empty[ks]));
            }
            const int iv = it0 + 2 * q + 1, vs = iv % C::STAGES;
            if (!(ok = warp_wait<TF>(smem_u32(&bar_full[vs]), (iv / C::STAGES) & 1, p.ctl, abort, 22))) break;
            #pragma unroll
            for (int t = 0; t < 2 && ok; ++t)
              if (active(t, j)) ok = pv_step(t, vs);
            if (!ok) break;
            mma_commit_e(lead, smem_u32(&bar_empty[vs]));
            j = jn;
          }
          }
        } else {
          // Iteration q takes V of the pair's key tile j = u_{q-1}, then K of
          // jn = u_q.  S_t(jn) overwrites the columns that O_t += P_t V read,
          // so it is issued after tile t's last O += P V, which comes earlier
          // in the same iteration or in an earlier one (or item).
          int it = it0;
          int j = SPARSE ? next_bit(ubits, nw, -1) : 0;
          if (I.nu > 0) {
            ok = warp_wait<TF>(smem_u32(&bar_full[it % C::STAGES]), (it / C::STAGES) & 1, p.ctl, abort, 21);
            if (ok) {
              tc_fence_after();
              #pragma unroll
              for (int t = 0; t < 2; ++t)
                if (active(t, j)) s_step(t, it % C::STAGES);
              mma_commit_e(lead, smem_u32(&bar_empty[it % C::STAGES]));
              ++it;
            }
          }
          for (int q = 1; q <= I.nu && ok; ++q) {
            const int vslot = it % C::STAGES;
            ok = warp_wait<TF>(smem_u32(&bar_full[vslot]), (it / C::STAGES) & 1, p.ctl, abort, 22);
            ++it;
            if (!ok) break;
            tc_fence_after();
            const bool have_k = q < I.nu;
            const int jn = have_k ? next_j(j) : -1;
            const int kslot = it % C::STAGES, kpar = (it / C::STAGES) & 1;
            if (have_k) ++it;
            bool k_ready = false;
            #pragma unroll
            for (int t = 0; t < 2 && ok; ++t) {
              if (active(t, j) && !(ok = pv_step(t, vslot))) break;
              if (have_k && active(t, jn)) {
                if (!k_ready) {
                  ok = warp_wait<TF>(smem_u32(&bar_full[kslot]), kpar, p.ctl, abort, 24);
                  if (!ok) break;
                  tc_fence_after();
                  k_ready = true;
                }
                s_step(t, kslot);
              }
            }
            if (!ok) break;
            mma_commit_e(lead, smem_u32(&bar_empty[vslot]));
            if (have_k) {
              if (!k_ready) {
                ok = warp_wait<TF>(smem_u32(&bar_full[kslot]), kpar, p.ctl, abort, 25);
                if (!ok) break;
              }
              mma_commit_e(lead, smem_u32(&bar_empty[kslot]));
            }
            j = jn;
          }
        }
        it0 += 2 * I.nu;
      }
      // Drain: every MMA issued above completes before TMEM is released.
      if (cs[0] + cs[1] > 0) {
        mma_commit_e(lead, smem_u32(&bar_drain));
        mbar_wait_quiet(smem_u32(&bar_drain), 0, 200000000ull);
      }
    }
  } else if (warp < C::WS) {
    // -------------------------------------------------------------- softmax
    // Thread = (query row r, column half h): warps [4*NH*t, 4*NH*(t+1)) serve
    // query tile t; warp w covers TMEM lanes 32*(w % 4) and key columns
    // [h*CPT, (h+1)*CPT) of the tile.
    const int t = warp / (4 * NH);
    const int h = (warp % (4 * NH)) / 4;
    const int sp = warp & 3;
    const int r = sp * 32 + lane;
    const int cb = h * C::CPT;          // first key column of this thread
    const int ob = h * C::OCPT;         // first O column of this thread
    {
      const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
      const uint32_t tS = tmem + lane_off + C::colS(t);
      const uint32_t tO = tmem + lane_off + C::colO(t);
      const float scale2 = p.scale2;
      const bool tail = (p.Nk % C::BN) != 0;
      const uint32_t xbar = smem_u32(&bar_x[t][sp]);
      int xph = 0;
      // Exchange one value per row with the partner warp (the other column
      // half of the same rows); bounded like every other wait.  Slots
      // alternate with every exchange: a value is overwritten only after the
      // partner has arrived at the next exchange, i.e. after it read it.
      auto exchange = [&](float v) -> float {
        const int slot = xph & 1;
        xch[t][slot][h][r] = v;
        mbar_arrive(xbar);  // every lane: releases its own write
        const bool okx = warp_wait<TF>(xbar, xph & 1, p.ctl, abort, 32);
        ++xph;
        return okx ? xch[t][slot][h ^ 1][r] : NAN;
      };
      // l: sum of the fp32 P values (gives the LSE).  lr normalises O: l plus,
      // for each tile, the bf16 rounding error of the row's largest P (the
      // value O += P V multiplied), so a row dominated by one key gets that
      // key's V row exactly.  With NH = 2 each half keeps partial sums,
      // combined once at the end.
      // Step lstep of an item handles key tile j: j = lstep when dense, the
      // lstep-th kept tile when block-sparse; gstep counts steps across
      // items (barrier phases).  Under a block mask a row may have seen no
      // key yet (m = -inf); its exponentials then use 0 in place of m, which
      // gives P = 0 for masked keys instead of -inf - -inf.
      const uint32_t* tbits = mbits + t * (SPARSE ? kMaskWords : 0);
      auto m_ref = [](float mv) { return (SPARSE && mv == -INFINITY) ? 0.f : mv; };
      int gstep = 0, nio = 0;  // steps and epilogues of this tile so far
      int nlq = 0;             // live items of this tile so far
      bool ok = true;
      for (int L = L0, kk = 0; L < n_items && ok; L = item_at(++kk)) {
      const Item I = L == L0 ? I0 : item_info(L);
      // this tile's flags as scalars (a runtime index into the item's
      // arrays would put them in local memory)
      const bool valid_t = t ? I.valid[1] : I.valid[0];
      const int ntile_t = t ? I.ntile[1] : I.ntile[0];
      if (!valid_t) continue;
      // this item's Q buffer (the loads count the tile's live items too)
      const int qbi = nlq % C::QBUF;
      if (ntile_t > 0) ++nlq;
      const int bh = I.bh;
      const int row = (I.qt0 + t) * C::BM + r;
      float m = -INFINITY, l = 0.f, lr = 0.f;
      if constexpr (C::SEPP) {
        const uint32_t tP = tmem + lane_off + C::colP(t);
        int j = SPARSE ? next_bit(tbits, nw, -1) : 0;
        for (int lstep = 0; lstep < ntile_t; ++lstep, ++gstep) {
          if (!warp_wait<TF>(smem_u32(&bar_s[t]), gstep & 1, p.ctl, abort, 30)) {
            ok = false;
            break;
          }
          tc_fence_after();
          int lim = C::BN;
          if (CAUSAL) lim = min(lim, row + p.coff + 1 - j * C::BN);
          if (!CAUSAL && tail && j == p.nkv - 1) lim = p.Nk - j * C::BN;
          // The whole row of S into registers; S_t may then be overwritten.
          float sv[C::BN];
#pragma unroll
          for (int c = 0; c < C::BN; c += 32) tmem_ld32(tS + c, *reinterpret_cast<uint32_t(*)[32]>(sv + c));
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bar_sf[t]));
          if (lim < C::BN) {
#pragma unroll
            for (int c = 0; c < C::BN; ++c)
              if (c >= lim) sv[c] = -INFINITY;
          }
          float mc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < C::BN; c += 8) {
#pragma unroll
            for (int e = 0; e < 4; ++e) mc[e] = fmax3(mc[e], sv[c + 2 * e], sv[c + 2 * e + 1]);
          }
          const float mx = fmax3(mc[0], mc[1], fmaxf(mc[2], mc[3]));
          const float m_new = fmaxf(m, mx * scale2);
          const bool need = m_new > m + kTau;
          const bool any_need = __any_sync(0xffffffffu, need);
          const float alpha = need ? ex2(m - m_new) : 1.0f;
          if (need) m = m_new;
          l *= alpha;
          lr *= alpha;
          const float mr = m_ref(m);
          {
            const float pmax = ex2(fmaf(mx, scale2, -mr));
            lr += __uint_as_float(pack_bf16(pmax, 0.f) << 16) - pmax;
          }
          // P = exp2(scale2 * s - m) as bf16 pairs in registers: this runs
          // while O_t += P_t V of the previous step may still read P_t
          const uint64_t sc2 = f2_pack(scale2, scale2), nm2 = f2_pack(-mr, -mr);
          uint64_t l2 = f2_pack(0.f, 0.f);
          uint32_t pk[C::BN / 2];
#pragma unroll
          for (int i = 0; i < C::BN / 2; ++i) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(sv[2 * i], sv[2 * i + 1]), sc2, nm2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            pk[i] = pack_bf16(p0, p1);
            l2 = f2_add(l2, f2_pack(p0, p1));
          }
          {
            float a0, a1;
            f2_unpack(l2, a0, a1);
            l += a0 + a1;
            lr += a0 + a1;
          }
          // P_t and O_t: the previous O_t += P_t V (also of the previous
          // item) must have completed
          if (gstep > 0 && !warp_wait<TF>(smem_u32(&bar_pf[t]), (gstep - 1) & 1, p.ctl, abort, 33)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < C::BN / 2; c0 += 16)
            tmem_st16(tP + c0, *reinterpret_cast<uint32_t(*)[16]>(pk + c0));
          if (any_need && lstep > 0) {
#pragma unroll 1
            for (int c0 = 0; c0 < HD; c0 += 32) {
              uint32_t ov[32];
              tmem_ld32(tO + c0, ov);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
              tmem_st32(tO + c0, ov);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bar_p[t]));
          if constexpr (SPARSE)
            j = next_bit(tbits, nw, j);
          else
            j = lstep + 1;
        }
      } else {
      int j = SPARSE ? next_bit(tbits, nw, -1) : 0;
      for (int lstep = 0; lstep < ntile_t; ++lstep, ++gstep) {
        if (!warp_wait<TF>(smem_u32(&bar_s[t]), gstep & 1, p.ctl, abort, 30)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // Keys c >= lim of this row are masked in this tile (the causal
        // boundary, key index <= row + coff; or the ragged last tile).  lim
        // may be <= 0: a tile past the row's last key.  Without a block mask
        // key 0 is in every row's first tile, so the running max is finite
        // from there on.
        int lim = C::BN;
        if (CAUSAL) lim = min(lim, row + p.coff + 1 - j * C::BN);
        if (!CAUSAL && tail && j == p.nkv - 1) lim = p.Nk - j * C::BN;
        // Pass 1: max over this thread's columns, 64 at a time (pass 2 reads
        // them again chunk by chunk).
        float mc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c64 = 0; c64 < C::CPT; c64 += 64) {
          float sv[64];
          tmem_ld32(tS + cb + c64, *reinterpret_cast<uint32_t(*)[32]>(sv));
          tmem_ld32(tS + cb + c64 + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
          tmem_wait_ld();
          if (lim < C::BN) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (cb + c64 + c >= lim) sv[c] = -INFINITY;
          }
#pragma unroll
          for (int c = 0; c < 64; c += 8) {
#pragma unroll
            for (int e = 0; e < 4; ++e) mc[e] = fmax3(mc[e], sv[c + 2 * e], sv[c + 2 * e + 1]);
          }
        }
        float mx = fmax3(mc[0], mc[1], fmaxf(mc[2], mc[3]));
        const float mxh = mx;  // max over this thread's own columns
        if (NH == 2) {
          mx = fmaxf(mx, exchange(mx));
          if (__any_sync(0xffffffffu, mx != mx)) {  // the exchange gave up
            ok = false;
            break;
          }
        }
        const float m_new = fmaxf(m, mx * scale2);
        const bool need = m_new > m + kTau;
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2(m - m_new) : 1.0f;
          if (need) m = m_new;
          l *= alpha;
          lr *= alpha;
          if (lstep > 0) {
            // O_t is complete here: S_t of this step was issued after the
            // previous O_t += P_t V and its commit covers every earlier MMA
            // of the issuing thread.
#pragma unroll 1
            for (int c0 = 0; c0 < C::OCPT; c0 += 32) {
              uint32_t ov[32];
              tmem_ld32(tO + ob + c0, ov);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
              tmem_st32(tO + ob + c0, ov);
            }
          }
        }
        // Rounding error of this tile's largest P (mx is the max over this
        // thread's columns, which holds the row's maximum in one half).
        const float mr = m_ref(m);
        {
          const float pmax = ex2(fmaf(mxh, scale2, -mr));
          lr += __uint_as_float(pack_bf16(pmax, 0.f) << 16) - pmax;
        }
        // Pass 2: P = exp2(scale2 * s - m), two elements per paired FMA and
        // add, 32 columns at a time with the next chunk's load in flight.  P
        // of chunk c lands in columns [cb + c/2, cb + c/2 + 16), all already
        // read by this thread.
        const uint64_t sc2 = f2_pack(scale2, scale2), nm2 = f2_pack(-mr, -mr);
        uint64_t l2 = f2_pack(0.f, 0.f);
        float sbuf[2][32];
        tmem_ld32(tS + cb, *reinterpret_cast<uint32_t(*)[32]>(sbuf[0]));
        tmem_wait_ld();
#pragma unroll
        for (int c0 = 0; c0 < C::CPT; c0 += 32) {
          float* sv = sbuf[(c0 / 32) & 1];
          if (c0 + 32 < C::CPT)
            tmem_ld32(tS + cb + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(sbuf[((c0 / 32) + 1) & 1]));
          if (lim < C::BN) {
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (cb + c0 + c >= lim) sv[c] = -INFINITY;
          }
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(sv[2 * i], sv[2 * i + 1]), sc2, nm2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            pk[i] = pack_bf16(p0, p1);
            l2 = f2_add(l2, f2_pack(p0, p1));
          }
          tmem_st16(tS + cb + c0 / 2, pk);
          if (c0 + 32 < C::CPT) tmem_wait_ld();
        }
        {
          float a0, a1;
          f2_unpack(l2, a0, a1);
          l += a0 + a1;
          lr += a0 + a1;
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar_p[t]));
        if constexpr (SPARSE)
          j = next_bit(tbits, nw, j);
        else
          j = lstep + 1;
      }
      }
      // Epilogue: O / lr -> bf16, and LSE = ln 2 * (m + log2 l).
      if (ok && NH == 2) {
        // the two halves' partial sums (one exchange slot each)
        const float lo = exchange(l);
        const float lro = exchange(lr);
        if (__any_sync(0xffffffffu, lo != lo || lro != lro)) ok = false;
        l += lo;
        lr += lro;
      }
      if (!ok) break;
      if (SPARSE && ntile_t == 0) {
        // no kept block: every row of the tile sees no key (o = 0, lse = -inf)
        if (row < p.Nq) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + ((size_t)bh * p.Nq + row) * HD + ob);
#pragma unroll
          for (int i = 0; i < C::OCPT / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
          if (h == 0) p.lse[(size_t)bh * p.Nq + row] = -INFINITY;
        }
      } else {
        if (!(ok = warp_wait<TF>(smem_u32(&bar_o[t]), (nio++) & 1, p.ctl, abort, 31))) break;
        tc_fence_after();
        // a row that saw no key (block-sparse only) has lr = 0 and o = 0
        const float inv_l = (SPARSE && !(lr > 0.f)) ? 0.f : 1.0f / lr;
        // O through shared memory when another item follows on this CTA:
        // each warp stages its 32 rows (128-byte swizzled, the TMA store's
        // layout) in this item's Q buffer, which the item's last S has
        // finished reading (bar_o follows it), and one TMA store writes them
        // as whole lines.  Per-thread row stores touch 32 lines per
        // instruction and hold the shared-memory pipe while the next item's
        // first S needs it; a CTA's last item (every item of a one-item
        // launch) keeps them, which measured faster there.
        if (C::QBUF == 2 && item_at(kk + 1) < n_items) {
          uint8_t* stg = smem + (size_t)(2 * qbi + t) * C::QTILE + (size_t)sp * 4096 + (size_t)lane * 128;
#pragma unroll
          for (int c0 = 0; c0 < HD; c0 += 32) {
            uint32_t ov[32];
            tmem_ld32(tO + c0, ov);
            tmem_wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              *reinterpret_cast<uint4*>(stg + (((c0 / 8 + i) ^ (lane & 7)) * 16)) =
                  make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
          if (row < p.Nq) p.lse[(size_t)bh * p.Nq + row] = (m + __log2f(l)) * kLn2;
          // O_t has been read: the next item's first O_t += P_t V may overwrite it
          tc_fence_before();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_u32(&bar_of[t]));
            const int row0 = (I.qt0 + t) * C::BM + sp * 32;
            if (row0 < p.Nq) {
              tma_store_3d(&to, smem_u32(stg), 0, row0, bh);
              bulk_commit_group();
              bulk_wait_group_read<0>();
            }
            mbar_arrive(smem_u32(&bar_qe[2 * qbi + t]));  // the Q buffer is free again
          }
          __syncwarp();
          continue;
        }
        __nv_bfloat16* orow = p.o + ((size_t)bh * p.Nq + row) * HD;
#pragma unroll 1
        for (int c0 = 0; c0 < C::OCPT; c0 += 32) {
          uint32_t ov[32];
          tmem_ld32(tO + ob + c0, ov);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
          if (row < p.Nq) {
            if constexpr (STG) {  // the staged-store kernel measured faster with 16-byte stores here
              uint4* dst = reinterpret_cast<uint4*>(orow + ob + c0);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            } else {
              st_global_64B(orow + ob + c0, pk);
            }
          }
        }
        if (h == 0 && row < p.Nq) p.lse[(size_t)bh * p.Nq + row] = (m + __log2f(l)) * kLn2;
        // O_t has been read: the next item's first O_t += P_t V may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&bar_of[t]));
          if (C::QBUF == 2) mbar_arrive(smem_u32(&bar_qe[2 * qbi + t]));  // the Q buffer is free again
        }
      }
      }  // items
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::W_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int HD, bool CAUSAL, bool SPARSE, int BN, bool STG>
cudaError_t launch_fwd_k(const FwdParams& p, const FwdLaunch& a, long ctas, cudaStream_t stream) {
  using C = FwdCfg<HD, kSplit, BN, STG>;
  auto kern = fa_fwd_kernel<HD, CAUSAL, kSplit, SPARSE, BN, STG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)ctas);
  kern<<<grid, C::THREADS, C::SMEM, stream>>>(a.tq, a.tk, a.tv, a.to, p);
  return cudaGetLastError();
}

template <int HD, bool CAUSAL, bool SPARSE, int BN = 128>
cudaError_t launch_fwd_t(const FwdLaunch& a, cudaStream_t stream) {
  using C = FwdCfg<HD, kSplit, BN>;
  FwdParams p;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.coff = a.Nk - a.Nq;
  p.nq = (a.Nq + C::BM - 1) / C::BM;
  p.nkv = (a.Nk + C::BN - 1) / C::BN;
  p.npairs = (p.nq + 1) / 2;
  p.BH = a.BH;
  p.group = head_group(a.BH, p.npairs, a.num_sms);
  p.kv_group = a.group;
  p.bmask = a.bmask;
  p.scale2 = a.scale * 1.4426950408889634f;
  p.ctl = a.ctl;
  // one persistent CTA per SM walks the pairs, or one CTA per pair
  // (block-sparse: each builds the bitsets of its own mask rows)
  const long n_items = (long)p.npairs * a.BH;
  const bool persistent = persistent_launch(CAUSAL, SPARSE, p.npairs) && n_items > a.num_sms;
  const long ctas = persistent ? a.num_sms : n_items;
  // d = 64 persistent launches of short items (at most 16 key tiles) stage O
  // through shared memory: there the epilogue is a large share of an item.
  // The staged kernel's step loop measured 2 % slower at 32 key tiles and
  // 5 % on one-item launches, which keep the other instantiation.
  if constexpr (HD == 64 && !SPARSE)
    if (persistent && p.nkv * BN <= 2048) return launch_fwd_k<HD, CAUSAL, SPARSE, BN, true>(p, a, ctas, stream);
  return launch_fwd_k<HD, CAUSAL, SPARSE, BN, false>(p, a, ctas, stream);
}

}  // namespace

cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream) {
  if (a.key_tile == 64) {  // dense only (the caller checks)
    if (a.d == 128)
      return a.causal ? launch_fwd_t<128, true, false, 64>(a, stream)
                      : launch_fwd_t<128, false, false, 64>(a, stream);
    return a.causal ? launch_fwd_t<64, true, false, 64>(a, stream)
                    : launch_fwd_t<64, false, false, 64>(a, stream);
  }
  if (a.bmask) {
    if (a.d == 128)
      return a.causal ? launch_fwd_t<128, true, true>(a, stream) : launch_fwd_t<128, false, true>(a, stream);
    return a.causal ? launch_fwd_t<64, true, true>(a, stream) : launch_fwd_t<64, false, true>(a, stream);
  }
  if (a.d == 128)
    return a.causal ? launch_fwd_t<128, true, false>(a, stream) : launch_fwd_t<128, false, false>(a, stream);
  return a.causal ? launch_fwd_t<64, true, false>(a, stream) : launch_fwd_t<64, false, false>(a, stream);
}

}  // namespace fa
