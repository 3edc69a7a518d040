// fa_bwd_d64.cu -- main attention backward kernel for head dimension 64.
//
// Same arithmetic as the general backward kernel (FlashAttention: exact
// attention made fast by counting memory traffic, "The method"; FlashAttention
// and IO-aware exact attention, "Backward by recomputation"): one CTA per
// 128-key tile of one head, looping over the 128-query tiles that see it,
//   S^T = K Q_i^T,  P^T = exp2(scale2 S^T - LSE2_i),
//   dP^T = V dO_i^T,  dS^T = P^T o (dP^T - D_i),
//   dV += P^T dO_i,  dK += dS^T Q_i,  dQ_i = dS K  (added into dQacc).
//
// At d = 64 the operands are small enough to software-pipeline the loop:
// tensor memory holds S^T (then P^T as bf16 pairs), dP^T (then dS^T pairs),
// dV, dK, dQ, and K and V themselves in separate columns.  Per query tile u
// the MMA warp issues
//   [P(u) ready]   dV(u) (A = P^T pairs), S^T(u+1) (A = K)
//   [dS(u) ready]  dK(u) (A = dS^T pairs), dP^T(u+1) (A = V), dQ(u)
// so the next tile's S^T and dP^T are computed while the P/dS warps work on
// the current one, and the P/dS warps run P(u), dS(u), P(u+1), ... with two
// waits per tile.  The hand-offs rely on a tcgen05.commit tracking every
// MMA issued before it: "S^T(u+1) done" also says that dV(u) has read the
// P^T pairs, and "dP^T(u) done" that dK(u-1) has read the dS^T pairs and
// dQ(u-2) the dS buffer the P/dS warps are about to overwrite.  dQ takes dS
// from shared memory (query-major), double-buffered.  Q goes through a
// 3-slot ring, dO through a 2-slot ring, and the dQ drain stages its
// reductions in a buffer of its own.  The row statistics of each query tile
// (-LSE log2 e and -D, written by the preprocess kernel) come with its Q
// tile.
//
// Dense launches run one CTA per SM over many key tiles (work items), with
// the ring positions and barrier phases running on across items; the next
// item's K is loaded early into the V buffer (free once V is in tensor
// memory), and copied into tensor memory by the drain warps once the item's
// last S^T has completed.  Block-sparse launches run one CTA per key tile.
//
// Roles (448 threads):
//   warps 0-7   P / dS: thread = key row = TMEM lane (warp w takes lanes
//               32 (w % 4) ...); warp w takes query columns [64 g, 64 g + 64)
//               of the tile, g = w / 4
//   warps 8-11  K and V into tensor memory, dQ drain (thread = query row),
//               then the dK epilogue
//   warp  12    TMA producer
//   warp  13    tcgen05 MMA issuer and TMEM owner
#include <cuda_bf16.h>

#include "fa_kernels.h"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct Cfg64 {
  static constexpr int HD = 64;
  static constexpr int BQ = 128;              // queries per iteration
  static constexpr int BK = 128;              // keys per CTA
  static constexpr int TILE = 128 * HD * 2;   // one 128-row bf16 tile: 16 KB
  static constexpr int DS_BYTES = BQ * BK * 2;
  static constexpr int QSLOTS = 3, DOSLOTS = 2;
  // dynamic shared memory layout (offsets from a 1024-byte aligned base)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_Q = OFF_V + TILE;
  static constexpr int OFF_DO = OFF_Q + QSLOTS * TILE;
  static constexpr int OFF_DS = OFF_DO + DOSLOTS * TILE;     // 2 buffers
  static constexpr int OFF_STAGE = OFF_DS + 2 * DS_BYTES;    // dQ boxes, 8 KB per drain warp
  // P/dS warps: NG column groups per TMEM lane quarter, CW query columns each
  static constexpr int NG = 2;
  static constexpr int NPW = 4 * NG;
  static constexpr int CW = BQ / NG;
  // row statistics of the tile in each Q slot: 128 x -LSE log2 e, 128 x -D
  static constexpr int OFF_STATS = OFF_STAGE + BQ * HD * 4;
  static constexpr int STATS_SLOT = 2 * BQ * 4;
  static constexpr int OFF_BAR = OFF_STATS + QSLOTS * STATS_SLOT;
  static constexpr int NBAR = 32;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16;
  // roles: P/dS warps, 4 dQ drain warps, the TMA warp, the MMA warp
  static constexpr int W_LOAD = NPW + 4, W_MMA = NPW + 5;  // drain: warps NPW ... NPW + 3
  static constexpr int THREADS = (NPW + 6) * 32;
  static constexpr uint32_t TMEM_COLS = 512;
  // S^T (then P^T bf16 pairs) | dP^T (then dS^T pairs) | dV | dK | dQ | K | V
  static constexpr uint32_t COL_ST = 0, COL_DPT = 128, COL_DV = 256, COL_DK = 320, COL_DQ = 384,
                            COL_KT = 448, COL_VT = 480;
  // Column, relative to S^T (or dP^T), of the bf16 pairs of P^T (or dS^T) for
  // MMA K-step k (16 queries): each P/dS warp packs its CW queries into the
  // first CW/2 of its own, already read, columns.
  static constexpr uint32_t pcol(int k) { return (uint32_t)((k / (CW / 16)) * CW + (k % (CW / 16)) * 8); }
};
static_assert(Cfg64::SMEM <= 232448, "shared memory budget");
static_assert(Cfg64::SMEM % 16 == 0 && Cfg64::SMEM + kMaskWords * 4 + 16 <= 232448,
              "shared memory budget with a block-mask column");
static_assert(Cfg64::QSLOTS >= 2 && Cfg64::QSLOTS <= 3 && Cfg64::DOSLOTS == 2, "ring sizes");
static_assert(Cfg64::NG == 2 || Cfg64::NG == 4, "32 or 64 query columns per P/dS warp");

// barrier indices
enum : int {
  B_K = 0, B_V, B_QF0, B_QF1, B_QF2, B_QE0, B_QE1, B_QE2, B_DOF0, B_DOF1, B_DOE0, B_DOE1,
  B_ST, B_P, B_DPT, B_DS, B_DQF, B_DQE, B_FIN, B_DRAIN, B_KT, B_VT, B_DKR, B_COUNT
};
static_assert(B_COUNT <= Cfg64::NBAR, "barrier area");
// arrival counts: TMA and tcgen05.commit barriers take one arrival; P and DS
// one per P/dS warp; DQE, KT, VT and DKR one per drain warp.
__device__ __constant__ const uint32_t kBarCount64[B_COUNT] = {
    1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1,           // K, V, QF*, QE*, DOF*, DOE*
    1, Cfg64::NPW, 1, Cfg64::NPW, 1, 4, 1, 1,     // ST, P, DPT, DS, DQF, DQE, FIN, DRAIN
    4, 4, 4};  // KT, VT (K, V copied to tensor memory), DKR (dK read out by the drain)

struct BwdParams64 {
  const float* stats;  // per tile: -LSE log2 e (128), -D (128)
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int Nq, Nk;    // query rows and keys per head
  int nq, nkv, BHkv, group;
  int coff;      // causal offset Nk - Nq: query i sees keys j <= i + coff
  int kv_group;  // query heads per key/value head (1: multi-head)
  const uint8_t* bmask;  // block mask [nq][nkv] (block-sparse kernels only)
  float scale, scale2;
  KernelCtl ctl;
};

template <bool TEST_FIRST = true>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const KernelCtl& ctl,
                                          volatile int* abort, uint32_t site) {
  const bool ok = mbar_wait<TEST_FIRST>(bar, parity, ctl, abort, site);
  return __all_sync(0xffffffffu, ok);
}

// XV (persistent launches): the drain copies the next item's V into tensor
// memory before its dK epilogue, and the MMA warp's first dK of an item waits
// for that epilogue's reads (DKR) instead of following the V copy.
template <bool CAUSAL, bool SPARSE, bool XV = false, bool PAIRS = false>
__global__ void __launch_bounds__(Cfg64::THREADS, 1)
    fa_bwd_d64_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                      const __grid_constant__ CUtensorMap tdq, const __grid_constant__ CUtensorMap tdk,
                      const BwdParams64 p) {
  using C = Cfg64;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) record_error(p.ctl, kErrSmemAlign, 2);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::NBAR * 8 + 4);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work items are (key/value head, key tile) pairs in the grid order of
  // decode_grid.  An item loops over the query tiles i0 ... nq-1 of each of
  // the kv_group query heads that share the key/value head, in that order;
  // each role follows the (tile, head) pair of its own position in the loop
  // with a TileWalk.  Persistent launches (see persistent_launch) have one
  // CTA per SM (G CTAs), and CTA b takes items b, 2G-1-b, 2G+b, 4G-1-b, ...:
  // every pass over G items visits them in the other direction, so with
  // causal masking (items heaviest first within a head group) each CTA pairs
  // heavy items with light ones.  Long square causal launches (PAIRS) walk
  // units of two key tiles of equal total work instead (see decode_pair).
  // An item's set-up then overlaps the previous item's last tiles instead of
  // costing a CTA launch.  Other launches have one CTA per item, which the
  // hardware scheduler balances.  The ring positions and the per-tile
  // barrier phases run on across items (global tile index U); K, V, their
  // copy into tensor memory and FIN have one phase per item.
  const int n_items = p.BHkv * p.nkv;
  const int B0 = (int)blockIdx.x, LS = (int)gridDim.x;
  // k-th item of this CTA (n_items or more: none); a block-sparse CTA has
  // one item, which the compiler then knows: its item loops run once
  auto item_at = [&](int k) {
    if (SPARSE) return k == 0 ? B0 : n_items;
    if (PAIRS) return 2 * (B0 + (k >> 1) * LS) + (k & 1);
    return k * LS + ((k & 1) ? LS - 1 - B0 : B0);
  };
  const int L0 = item_at(0);
  struct Item {
    int bk, kt, i0;
  };
  auto item_info = [&](int L) {
    const GridPos gp = PAIRS ? decode_pair(L, p.nkv) : decode_grid(L, p.BHkv, p.nkv, p.group);
    Item I;
    I.bk = gp.bh;
    I.kt = gp.rank;
    I.i0 = CAUSAL ? first_query_tile(I.kt, p.coff) : 0;  // first query tile that sees this key tile
    return I;
  };
  const Item I0 = item_info(L0);
  const int bk = I0.bk, kt = I0.kt, i0 = I0.i0;
  // Block-sparse (one item per CTA): the TMA warp turns this key tile's mask
  // column (query tiles i0 .. nq-1) into a bitset after the statistics; with
  // no kept tile the CTA only zeroes its dK, dV rows.
  QuerySeq<SPARSE> qseq{reinterpret_cast<const uint32_t*>(smem + C::SMEM), (p.nq + 31) >> 5, i0, p.nq};
  int nqt = p.nq - i0;  // query tiles per query head
  if constexpr (SPARSE) {
    uint32_t* qbits = reinterpret_cast<uint32_t*>(smem + C::SMEM);
    int* qcount = reinterpret_cast<int*>(smem + C::SMEM + kMaskWords * 4);
    if (warp == C::W_LOAD) {
      mask_bits_warp(p.bmask + kt, p.nkv, i0, p.nq, qseq.nw, qbits, lane);
      __syncwarp();
      const int n = mask_popc_warp(qbits, qseq.nw, lane);
      if (lane == 0) *qcount = n;
    }
    __syncthreads();
    nqt = *qcount;
    if (nqt == 0) {
      zero_key_tile<C::HD>(p.dk, p.dv, bk, kt, p.Nk);
      return;
    }
    qseq.first = next_bit(qbits, qseq.nw, -1);
  }
  const int nit = nqt * p.kv_group;                // query tiles of the first item
  const TileWalk walk0{qseq.first, bk * p.kv_group};
  // per item (dense items after the first): query tiles, first position,
  // and the query-tile sequence
  auto item_nit = [&](const Item& I) { return (p.nq - I.i0) * p.kv_group; };
  auto item_seq = [&](const Item& I) {
    QuerySeq<SPARSE> s = qseq;
    if constexpr (!SPARSE) s.first = I.i0;
    return s;
  };

  const uint32_t s0 = smem_u32(smem);
  const uint32_t sK = s0 + C::OFF_K, sV = s0 + C::OFF_V, sQ = s0 + C::OFF_Q,
                 sDO = s0 + C::OFF_DO, sDS = s0 + C::OFF_DS;
  // K and V of item k: the two key-tile buffers swap every item.  V reaches
  // tensor memory early in its item, after which no one reads its buffer:
  // the next item's K is loaded there at once, and the next V goes into
  // this item's K buffer once the last dQ (B = K) has completed.
  auto k_buf = [&](int k) { return (k & 1) ? sV : sK; };
  auto v_buf = [&](int k) { return (k & 1) ? sK : sV; };

  // The TMA thread initialises the barriers and issues the copies that need
  // no wait (K, V, and Q with its statistics and dO of the first two query
  // tiles) before the CTA-wide sync, so their latency overlaps the set-up.
  int nq_issued = 0, ndo_issued = 0;
  TileWalk lw = walk0;  // the TMA thread's position
  QuerySeq<SPARSE> lseq = qseq;  // and its item's query-tile sequence
  auto issue_q = [&](int u) {
    const int qs = u % C::QSLOTS;
    mbar_arrive_expect_tx(bar(B_QF0 + qs), C::TILE + C::STATS_SLOT);
    tma_load_3d(sQ + qs * C::TILE, &tq, bar(B_QF0 + qs), 0, lw.qt * C::BQ, lw.qh);
    bulk_load(s0 + C::OFF_STATS + qs * C::STATS_SLOT, p.stats + ((size_t)lw.qh * p.nq + lw.qt) * 256,
              C::STATS_SLOT, bar(B_QF0 + qs));
    ++nq_issued;
  };
  auto issue_do = [&](int u) {  // after issue_q(u); moves to the next tile
    const int ds = u % C::DOSLOTS;
    mbar_arrive_expect_tx(bar(B_DOF0 + ds), C::TILE);
    tma_load_3d(sDO + ds * C::TILE, &tdo, bar(B_DOF0 + ds), 0, lw.qt * C::BQ, lw.qh);
    ++ndo_issued;
    lseq.next(lw);
  };
  const int pre = nit < C::DOSLOTS ? nit : C::DOSLOTS;   // tiles issued before the sync
  if (warp == C::W_LOAD && lane == 0) {
    *abort = 0;
    for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), kBarCount64[i]);
    fence_barrier_init();
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    tma_prefetch_desc(&tdo);
    tma_prefetch_desc(&tdq);
    tma_prefetch_desc(&tdk);
    // K and Q_0 first: S^T of the first tile needs only those two
    mbar_arrive_expect_tx(bar(B_K), C::TILE);
    tma_load_3d(sK, &tk, bar(B_K), 0, kt * C::BK, bk);
    for (int u = 0; u < pre; ++u) {
      issue_q(u);
      if (u == 0) {
        mbar_arrive_expect_tx(bar(B_V), C::TILE);
        tma_load_3d(sV, &tv, bar(B_V), 0, kt * C::BK, bk);
      }
      issue_do(u);
    }
  }
  if (warp == C::W_MMA) {
    tmem_alloc(smem_u32(tmem_base_sh), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_sh;

  if (warp == C::W_LOAD) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      bool ok = true;
      int nkv_issued = 1;  // items whose V has been issued (K: nk_issued)
      int nk_issued = 1;
      // Q_u (with its statistics) and dO_u of global tile u, once their ring
      // slots are free
      auto ring = [&](int u) -> bool {
        const int qs = u % C::QSLOTS, qn = u / C::QSLOTS;
        if (qn > 0 && !mbar_wait(bar(B_QE0 + qs), (qn - 1) & 1, p.ctl, abort, 50)) return false;
        issue_q(u);
        const int ds = u % C::DOSLOTS, dn = u / C::DOSLOTS;
        if (dn > 0 && !mbar_wait(bar(B_DOE0 + ds), (dn - 1) & 1, p.ctl, abort, 51)) return false;
        issue_do(u);
        return true;
      };
      int u = pre, uend = nit;  // global tile index; end of the current item
      for (int L = L0, kk = 0;;) {
        while (u < uend && (ok = ring(u))) ++u;  // a failed tile is not counted
        if (!ok) break;
        L = item_at(++kk);
        if (L >= n_items) break;
        // the next item (index nkv_issued): its K once the previous V is in
        // tensor memory, its first tiles as soon as their slots are free,
        // then its V once every MMA of the previous item has completed
        const Item I = item_info(L);
        const int kn = nkv_issued;
        if (!(ok = mbar_wait(bar(B_VT), (kn - 1) & 1, p.ctl, abort, 53))) break;
        mbar_arrive_expect_tx(bar(B_K), C::TILE);
        tma_load_3d(k_buf(kn), &tk, bar(B_K), 0, I.kt * C::BK, I.bk);
        ++nk_issued;
        lw = TileWalk{I.i0, I.bk * p.kv_group};
        lseq = item_seq(I);
        uend = u + item_nit(I);
        const int upre = min(uend, u + C::DOSLOTS);
        while (u < upre && (ok = ring(u))) ++u;
        if (!ok || !(ok = mbar_wait(bar(B_FIN), (kn - 1) & 1, p.ctl, abort, 52))) break;
        mbar_arrive_expect_tx(bar(B_V), C::TILE);
        tma_load_3d(v_buf(kn), &tv, bar(B_V), 0, I.kt * C::BK, I.bk);
        ++nkv_issued;
      }
      if (!ok) {
        // Abort: let every copy already issued land before the CTA exits.
        mbar_wait_quiet(bar(B_K), (nk_issued - 1) & 1, 200000000ull);
        mbar_wait_quiet(bar(B_V), (nkv_issued - 1) & 1, 200000000ull);
        for (int v = (nq_issued > C::QSLOTS ? nq_issued - C::QSLOTS : 0); v < nq_issued; ++v)
          mbar_wait_quiet(bar(B_QF0 + v % C::QSLOTS), (v / C::QSLOTS) & 1, 200000000ull);
        for (int v = (ndo_issued > C::DOSLOTS ? ndo_issued - C::DOSLOTS : 0); v < ndo_issued; ++v)
          mbar_wait_quiet(bar(B_DOF0 + v % C::DOSLOTS), (v / C::DOSLOTS) & 1, 200000000ull);
      }
    }
  } else if (warp == C::W_MMA) {
    // ------------------------------------------------------------------ MMA
    // The whole warp runs the issue loop; one elected lane issues.
    {
      const uint32_t lead = elect_one();
      constexpr uint32_t kIdS = idesc_bf16(128, C::BQ, false, false);  // S^T, dP^T
      constexpr uint32_t kIdG = idesc_bf16(128, C::HD, false, true);   // dV, dK
      constexpr uint32_t kIdQ = idesc_bf16(128, C::HD, true, true);    // dQ = dS K
      const uint32_t tST = tmem + C::COL_ST, tDPT = tmem + C::COL_DPT, tDV = tmem + C::COL_DV,
                     tDK = tmem + C::COL_DK, tDQ = tmem + C::COL_DQ, tKT = tmem + C::COL_KT,
                     tVT = tmem + C::COL_VT;
      // Descriptor low halves of every operand tile (sdesc_lo): K-major
      // operands with lbo 16, M/N-major ones with lbo 16384 (the distance
      // between 64-element blocks); the high half is the same for all.
      constexpr uint32_t HI = sdesc_hi(1024);
      constexpr uint32_t TILE16 = C::TILE >> 4, DS16 = C::DS_BYTES >> 4;
      uint32_t kMN = sdesc_lo(sK, 16384);  // K of the current item (B of dQ)
      const uint32_t qK = sdesc_lo(sQ, 16), qMN = sdesc_lo(sQ, 16384);
      const uint32_t doK = sdesc_lo(sDO, 16), doMN = sdesc_lo(sDO, 16384);
      const uint32_t dsMN = sdesc_lo(sDS, 16384);
      // S^T = K Q_v^T   (M = keys, N = queries, K = d; A = K in tensor memory)
      auto issue_st = [&](uint32_t qo) {
#pragma unroll
        for (int k = 0; k < C::HD / 16; ++k)
          mma_ts_e(lead, tST, tKT + 8 * k, qK + qo + 2 * k, HI, kIdS, k > 0);
        mma_commit_e(lead, bar(B_ST));
      };
      // dP^T = V dO_v^T   (A = V in tensor memory)
      auto issue_dpt = [&](uint32_t dof) {
#pragma unroll
        for (int k = 0; k < C::HD / 16; ++k)
          mma_ts_e(lead, tDPT, tVT + 8 * k, doK + dof + 2 * k, HI, kIdS, k > 0);
        mma_commit_e(lead, bar(B_DPT));
      };
      // dQ_w = dS K   (A = dS buffer w&1 read query-major, B = K key-major),
      // once the drain has taken dQ_{w-1} out of tensor memory; issued after
      // dP^T(w+1), whose completion then covers dQ(w-1)
      auto issue_dq = [&](int w) -> bool {
        if (w > 0 && !warp_wait(bar(B_DQE), (w - 1) & 1, p.ctl, abort, 70)) return false;
        tc_fence_after();
        const uint32_t dsw = (uint32_t)(w & 1) * DS16;
#pragma unroll
        for (int k = 0; k < C::BK / 16; ++k)
          mma_ss_e(lead, tDQ, dsMN + dsw + 128 * k, HI, kMN + 128 * k, HI, kIdQ, k > 0);
        mma_commit_e(lead, bar(B_DQF));
        return true;
      };
      // Q slot offset of global tile v and the phase of its fill
      auto q_off = [](int v) { return (uint32_t)(v % C::QSLOTS) * TILE16; };
      auto q_ph = [](int v) { return (uint32_t)(v / C::QSLOTS) & 1u; };
      bool ok = true;
      int U0 = 0;  // global index of the item's first tile
      for (int L = L0, k = 0; L < n_items && ok; L = item_at(++k)) {
        const int nit_i = L == L0 ? nit : item_nit(item_info(L));
        const uint32_t kp = (uint32_t)k & 1u;
        kMN = sdesc_lo(k_buf(k), 16384);
        // K and V in tensor memory (the drain waited for their loads)
        ok = warp_wait(bar(B_KT), kp, p.ctl, abort, 59) &&
             warp_wait(bar(B_QF0 + U0 % C::QSLOTS), q_ph(U0), p.ctl, abort, 61);
        if (ok) {
          tc_fence_after();
          issue_st(q_off(U0));
          ok = warp_wait(bar(B_VT), kp, p.ctl, abort, 62) &&
               warp_wait(bar(B_DOF0 + (U0 & 1)), (uint32_t)(U0 >> 1) & 1u, p.ctl, abort, 63);
        }
        if (ok) {
          tc_fence_after();
          issue_dpt((uint32_t)(U0 & 1) * TILE16);
        }
        // Q ring of tiles u and u + 1, advanced per tile: slot offset of u,
        // slot and fill phase of u + 1
        uint32_t qo_u = q_off(U0);
        int qs_v = (U0 + 1) % C::QSLOTS;
        uint32_t qph_v = q_ph(U0 + 1);
        for (int u = 0; u < nit_i && ok; ++u) {
          const int U = U0 + u, Vn = U + 1;
          const uint32_t qo_v = (uint32_t)qs_v * TILE16;
          const uint32_t dof_u = (uint32_t)(U & 1) * TILE16, dof_v = (uint32_t)(Vn & 1) * TILE16;
          const uint32_t acc0 = u > 0 ? 1u : 0u;
          const bool more = u + 1 < nit_i;
          // dV += P^T dO_u   (A = P^T bf16 in TMEM, B = dO_u query-major)
          if (!(ok = warp_wait(bar(B_P), U & 1, p.ctl, abort, 66))) break;
          tc_fence_after();
#pragma unroll
          for (int k2 = 0; k2 < C::BQ / 16; ++k2)
            mma_ts_e(lead, tDV, tST + C::pcol(k2), doMN + dof_u + 128 * k2, HI, kIdG, k2 > 0 ? 1u : acc0);
          mma_commit_e(lead, bar(B_DOE0 + (U & 1)));       // dO_u slot free
          // S^T of the next tile overwrites the P^T pairs only after dV(u) has
          // read them (tcgen05.mma runs in issue order)
          if (more) {
            if (!(ok = warp_wait(bar(B_QF0 + qs_v), qph_v, p.ctl, abort, 64))) break;
            tc_fence_after();
            issue_st(qo_v);
          }
          // dS(u) is in shared memory, its transpose in the dP^T columns
          if (!(ok = warp_wait(bar(B_DS), U & 1, p.ctl, abort, 69))) break;
          tc_fence_after();
          // the item's first dK overwrites the previous item's: the drain has
          // read that out (it copies the next V before its dK epilogue)
          if (XV && u == 0 && k > 0 && !(ok = warp_wait(bar(B_DKR), (uint32_t)(k - 1) & 1u, p.ctl, abort, 68)))
            break;
          // dK += dS^T Q_u   (A = dS^T bf16 pairs in TMEM, B = Q_u query-major)
#pragma unroll
          for (int k2 = 0; k2 < C::BQ / 16; ++k2)
            mma_ts_e(lead, tDK, tDPT + C::pcol(k2), qMN + qo_u + 128 * k2, HI, kIdG, k2 > 0 ? 1u : acc0);
          mma_commit_e(lead, bar(B_QE0 + (int)(qo_u / TILE16)));  // Q_u slot free
          // dP^T of the next tile overwrites the dS^T pairs only after dK(u)
          // has read them; its completion covers dK(u), dQ(u-1) and every
          // earlier MMA
          if (more) {
            if (!(ok = warp_wait(bar(B_DOF0 + (Vn & 1)), (uint32_t)(Vn >> 1) & 1u, p.ctl, abort, 67))) break;
            tc_fence_after();
            issue_dpt(dof_v);
          }
          if (!(ok = issue_dq(U))) break;
          qo_u = qo_v;
          if (++qs_v == C::QSLOTS) {
            qs_v = 0;
            qph_v ^= 1u;
          }
        }
        // every MMA of the item: dK, dV final, K and V free for the next item
        if (ok) mma_commit_e(lead, bar(B_FIN));
        U0 += nit_i;
      }
      mma_commit_e(lead, bar(B_DRAIN));
      mbar_wait_quiet(bar(B_DRAIN), 0, 200000000ull);
    }
  } else if (warp < C::NPW) {
    // ------------------------------------------------------------- P / dS
    constexpr int CW = C::CW;                       // query columns of this warp
    const int g = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int cb = CW * g;                          // first query column of this thread
    const uint32_t tST = tmem + lane_off + C::COL_ST + cb, tDPT = tmem + lane_off + C::COL_DPT + cb;
    const uint64_t sc2 = f2_pack(p.scale2, p.scale2);
    // statistics of the tile in Q slot s: 128 x -LSE log2 e, 128 x -D,
    // loaded with the Q tile (same barrier)
    const float* stats = reinterpret_cast<const float*>(smem + C::OFF_STATS);
    int qs_u = 0;
    uint32_t qph_u = 0;
    bool ok = true;
    const uint32_t sw = (uint32_t)(r & 7);
    // this thread's 16-byte chunks of a dS key row: 64-query block cb / 64,
    // chunks (cb % 64) / 8 ... of 8 queries each
    const uint32_t ds_row = (uint32_t)(cb >> 6) * 16384u + (uint32_t)r * 128u;
    const uint32_t ds_c0 = (uint32_t)((cb & 63) >> 3);
    int U0 = 0;  // global index of the item's first tile
    for (int L = L0, k = 0; L < n_items && ok; L = item_at(++k)) {
    const Item I = L == L0 ? I0 : item_info(L);
    const int kt = I.kt;
    const int nit_i = L == L0 ? nit : item_nit(I);
    const QuerySeq<SPARSE> seq = L == L0 ? qseq : item_seq(I);
    const size_t rowbase = (size_t)I.bk * p.Nk;      // key rows (dK, dV)
    TileWalk w = L == L0 ? walk0 : TileWalk{seq.first, I.bk * p.kv_group};
    for (int u = 0; u < nit_i && ok; ++u, seq.next(w)) {
      const int U = U0 + u;
      const int qt = w.qt;
      const float* lse_u = stats + qs_u * 256 + cb;
      const float* d_u = lse_u + 128;
      if (!(ok = warp_wait(bar(B_QF0 + qs_u), qph_u, p.ctl, abort, 80))) break;
      if (++qs_u == C::QSLOTS) {
        qs_u = 0;
        qph_u ^= 1u;
      }
      // ---- P^T[r][q] = exp2(scale2 * S^T - LSE2_q); causal: zero where query < key
      // (S^T(u) was issued after dV(u-1): the P^T pairs of the last tile are
      // consumed.  This thread's pairs go into the first CW/2 of its own
      // S^T columns once it has read them.)
      if (!(ok = warp_wait(bar(B_ST), U & 1, p.ctl, abort, 81))) break;
      tc_fence_after();
      uint32_t pk[CW / 2];
      {
        float pr[CW];
#pragma unroll
        for (int c = 0; c < CW; c += 32) tmem_ld32(tST + c, *reinterpret_cast<uint32_t(*)[32]>(pr + c));
        tmem_wait_ld();
        // causal: zero where query qt*128 + q does not see key kt*128 + r,
        // i.e. q < r + (kt - qt)*128 - coff; the tile needs it when that
        // bound is positive for the last key
        const int qdelta = (kt - qt) * C::BK - p.coff;
        const bool diag = CAUSAL && qdelta > 1 - C::BK;
        const int rlim = r + qdelta;
        // statistics four at a time (one 16-byte broadcast load per two pairs)
        uint64_t nlp[CW / 2];
#pragma unroll
        for (int i = 0; i < CW / 4; ++i) {
          const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(lse_u + 4 * i);
          nlp[2 * i] = v.x;
          nlp[2 * i + 1] = v.y;
        }
#pragma unroll
        for (int i = 0; i < CW / 2; ++i) {
          const int q = 2 * i;
          const uint64_t nl2 = nlp[i];
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(pr[q], pr[q + 1]), sc2, nl2), x0, x1);
          float p0 = ex2(x0), p1 = ex2(x1);
          if (diag && cb + q < rlim) p0 = 0.f;
          if (diag && cb + q + 1 < rlim) p1 = 0.f;
          pk[i] = pack_bf16(p0, p1);
        }
      }
#pragma unroll
      for (int c = 0; c < CW / 2; c += 16) tmem_st16(tST + c, *reinterpret_cast<const uint32_t(*)[16]>(pk + c));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_P));
      // ---- dS = P o (dP - D), with P the bf16 values dV multiplied
      // (dP^T(u) was issued after dK(u-1) and dQ(u-2): the dS^T pairs of the
      // last tile and dS buffer u&1 are consumed.)
      if (!(ok = warp_wait(bar(B_DPT), U & 1, p.ctl, abort, 83))) break;
      tc_fence_after();
      uint32_t dp[CW];
#pragma unroll
      for (int c = 0; c < CW; c += 32) tmem_ld32(tDPT + c, *reinterpret_cast<uint32_t(*)[32]>(dp + c));
      tmem_wait_ld();
      uint64_t ndp[CW / 2];
#pragma unroll
      for (int i = 0; i < CW / 4; ++i) {
        const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(d_u + 4 * i);
        ndp[2 * i] = v.x;
        ndp[2 * i + 1] = v.y;
      }
#pragma unroll
      for (int i = 0; i < CW / 2; ++i) {
        const uint64_t nd2 = ndp[i];
        const uint32_t w = pk[i];
        const uint64_t pv = f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
        float a, b;
        f2_unpack(f2_mul(f2_add(f2_pack(__uint_as_float(dp[2 * i]), __uint_as_float(dp[2 * i + 1])), nd2), pv), a, b);
        pk[i] = pack_bf16(a, b);
      }
      // dS^T pairs for dK into the first CW/2 of this thread's dP^T columns
#pragma unroll
      for (int c = 0; c < CW / 2; c += 16) tmem_st16(tDPT + c, *reinterpret_cast<const uint32_t(*)[16]>(pk + c));
      // key row r of dS buffer u&1, 128-byte swizzled (A operand of dQ)
      const uint32_t srow = sDS + (uint32_t)(U & 1) * C::DS_BYTES + ds_row;
#pragma unroll
      for (int c = 0; c < CW / 8; ++c)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(srow + (((ds_c0 + (uint32_t)c) ^ sw) << 4)),
                     "r"(pk[4 * c]), "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                     : "memory");
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DS));         // also: dP^T(u) has been read
    }
    // epilogue: dV rows of this key tile, columns [DVC g, DVC g + DVC); the
    // next item's first dV (computed after this warp's next P) overwrites them
    constexpr int DVC = C::HD / C::NG;
    static_assert(DVC % 32 == 0, "whole 64-byte pieces of a dV row per thread");
    if (ok && (ok = warp_wait(bar(B_FIN), (uint32_t)k & 1u, p.ctl, abort, 86))) {
      tc_fence_after();
      const int key = kt * C::BK + r;
      uint32_t v[32];
      if constexpr (DVC == 32) {
        tmem_ld32(tmem + lane_off + C::COL_DV + DVC * g, v);
      } else {
        tmem_ld16(tmem + lane_off + C::COL_DV + DVC * g, *reinterpret_cast<uint32_t(*)[16]>(v));
      }
      tmem_wait_ld();
      uint32_t pkv[DVC / 2];
#pragma unroll
      for (int i = 0; i < DVC / 2; ++i) pkv[i] = pack_bf16(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
      if (key < p.Nk) {
        uint4* d4 = reinterpret_cast<uint4*>(p.dv + (rowbase + key) * C::HD + DVC * g);
#pragma unroll
        for (int i = 0; i < DVC / 32; ++i) st_global_64B(d4 + 4 * i, pkv + 16 * i);
      }
    }
    U0 += nit_i;
    }  // items
  } else {
    // ---------------------------------------------------------- dQ drain
    // dQ_u (128 query rows x 64, fp32) leaves TMEM once per tile and is added
    // into dQacc by TMA bulk reductions of two 32-row x 32-column boxes per
    // warp, staged (128-byte swizzled) in this warp's 8 KB of the staging area.
    const int sp = warp & 3;
    const int r = sp * 32 + lane;
    const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
    const uint32_t sw = (uint32_t)(lane & 7);
    const uint32_t stage = s0 + C::OFF_STAGE + (uint32_t)sp * 8192u;
    // This warp's 32 key rows of a K or V tile into tensor memory (the A
    // operands of S^T and dP^T): 128 bytes of a 128-byte-swizzled row are 32
    // words, element 2c in the low half of word c.  The K copy of an item
    // comes right after the previous item's FIN (its MMAs are complete), the
    // V copy after this warp's dK epilogue of the previous item.
    auto to_tmem = [&](uint32_t buf, uint32_t col, int done) {
      const uint32_t src = buf + (uint32_t)r * 128u;
      uint32_t w[32];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[4 * c]), "=r"(w[4 * c + 1]), "=r"(w[4 * c + 2]), "=r"(w[4 * c + 3])
                     : "r"(src + (((uint32_t)c ^ sw) << 4))
                     : "memory");
      tmem_st32(tmem + lane_off + col, w);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(done));
    };
    bool ok = warp_wait(bar(B_K), 0, p.ctl, abort, 92);
    if (ok) to_tmem(k_buf(0), C::COL_KT, B_KT);
    int U0 = 0;  // global index of the item's first tile
    for (int L = L0, k = 0; L < n_items && ok; L = item_at(++k)) {
    const Item I = L == L0 ? I0 : item_info(L);
    const int kt = I.kt;
    const int nit_i = L == L0 ? nit : item_nit(I);
    const QuerySeq<SPARSE> seq = L == L0 ? qseq : item_seq(I);
    if (!XV || k == 0) {  // with XV later items' V is copied at the end of the item before
      if (!(ok = warp_wait(bar(B_V), (uint32_t)k & 1u, p.ctl, abort, 93))) break;
      to_tmem(v_buf(k), C::COL_VT, B_VT);
    }
    TileWalk w = L == L0 ? walk0 : TileWalk{seq.first, I.bk * p.kv_group};
    const bool has_next = item_at(k + 1) < n_items;
    for (int u = 0; u < nit_i && ok; ++u, seq.next(w)) {
      // The next item's K goes into tensor memory as soon as the item's last
      // S^T (the last MMA that reads the K columns) has completed and that K
      // has landed, so the next item's first S^T need not wait for this
      // item's last dQ, its drain and the dK epilogue.  Nothing issues the
      // next S^T before this copy, so the S^T barrier cannot run past it.
      if (has_next && u + 1 == nit_i) {
        if (!(ok = warp_wait(bar(B_ST), (uint32_t)(U0 + u) & 1u, p.ctl, abort, 95) &&
                   warp_wait(bar(B_K), (uint32_t)(k + 1) & 1u, p.ctl, abort, 94)))
          break;
        tc_fence_after();
        to_tmem(k_buf(k + 1), C::COL_KT, B_KT);
      }
      if (!(ok = warp_wait(bar(B_DQF), (U0 + u) & 1, p.ctl, abort, 90))) break;
      tc_fence_after();
      uint32_t v[64];
      tmem_ld32(tmem + lane_off + C::COL_DQ, *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld32(tmem + lane_off + C::COL_DQ + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(B_DQE));                   // dQ's TMEM columns are free again
        bulk_wait_group_read<0>();                 // the previous boxes have left the staging area
      }
      __syncwarp();
      const int y = w.qt * C::BQ + sp * 32, zq = w.qh;
      // columns [32 bb, 32 bb + 32) -> box bb
#pragma unroll
      for (int bb = 0; bb < 2; ++bb) {
        const uint32_t row = stage + (uint32_t)bb * 4096u + (uint32_t)lane * 128u;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (((uint32_t)c ^ sw) << 4)),
                       "r"(v[32 * bb + 4 * c]), "r"(v[32 * bb + 4 * c + 1]), "r"(v[32 * bb + 4 * c + 2]),
                       "r"(v[32 * bb + 4 * c + 3])
                       : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_reduce_add_3d(&tdq, stage, 0, y, zq);
        tma_reduce_add_3d(&tdq, stage + 4096u, 32, y, zq);
        bulk_commit_group();
      }
    }
    // epilogue: the next item's V into tensor memory first (its first dP^T
    // waits for it), then the dK rows of this key tile (scaled); the next
    // item's first dK waits for DKR, which follows their reads
    if (ok && (ok = warp_wait(bar(B_FIN), (uint32_t)k & 1u, p.ctl, abort, 91))) {
      tc_fence_after();
      if (XV && has_next) {
        if (!(ok = warp_wait(bar(B_V), (uint32_t)(k + 1) & 1u, p.ctl, abort, 93))) break;
        to_tmem(v_buf(k + 1), C::COL_VT, B_VT);
      }
      // The warp's 32 rows go out through its staging area (128-byte
      // swizzled, as the TMA store reads them) in one store of whole lines,
      // once the area's last dQ boxes have been read; per-thread row stores
      // would touch 32 lines per instruction.
      const float scale = p.scale;
      if (lane == 0) bulk_wait_group_read<0>();
      __syncwarp();
#pragma unroll 1
      for (int c0 = 0; c0 < C::HD; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + C::COL_DK + c0, v);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16(__uint_as_float(v[2 * i]) * scale, __uint_as_float(v[2 * i + 1]) * scale);
        const uint32_t row = stage + (uint32_t)lane * 128u;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((((uint32_t)(c0 / 8 + i)) ^ sw) << 4)),
                       "r"(pk[4 * i]), "r"(pk[4 * i + 1]), "r"(pk[4 * i + 2]), "r"(pk[4 * i + 3])
                       : "memory");
      }
      // dK has been read out of tensor memory: the next item's first dK may overwrite it
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (XV && lane == 0) mbar_arrive(bar(B_DKR));
      const int key0 = kt * C::BK + sp * 32;
      if (lane == 0 && key0 < p.Nk) {
        tma_store_3d(&tdk, stage, 0, key0, I.bk);
        bulk_commit_group();
      }
    }
    U0 += nit_i;
    }  // items
    // every reduction has landed before the CTA exits
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::W_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <bool CAUSAL, bool SPARSE, bool XV, bool PAIRS = false>
cudaError_t launch_k(const BwdLaunch& a, const BwdParams64& p, long ctas, cudaStream_t stream) {
  using C = Cfg64;
  auto kern = fa_bwd_d64_kernel<CAUSAL, SPARSE, XV, PAIRS>;
  // block-sparse: the mask column's bitset and its count follow the layout
  const int smem_bytes = C::SMEM + (SPARSE ? kMaskWords * 4 + 16 : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)ctas);
  kern<<<grid, C::THREADS, smem_bytes, stream>>>(a.tq, a.tk, a.tv, a.tdo, a.tdq, a.tdk, p);
  return cudaGetLastError();
}

template <bool CAUSAL, bool SPARSE>
cudaError_t launch_t(const BwdLaunch& a, cudaStream_t stream) {
  using C = Cfg64;
  BwdParams64 p;
  p.stats = a.stats;
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.coff = a.Nk - a.Nq;
  p.nq = (a.Nq + C::BQ - 1) / C::BQ;
  p.nkv = (a.Nk + C::BK - 1) / C::BK;
  p.BHkv = a.BH / a.group;
  p.kv_group = a.group;
  p.bmask = a.bmask;
  p.group = head_group(p.BHkv, p.nkv, a.num_sms);
  p.scale = a.scale;
  p.scale2 = a.scale * kLog2e;
  p.ctl = a.ctl;
  // one persistent CTA per SM walks the items, or one CTA per item; long
  // square causal launches in units of two key tiles (pair_launch; measured
  // +9 % at 32 key tiles per head, +4 % at 64, +2 % at 128)
  const long n_items = (long)p.nkv * p.BHkv;
  const bool pairs = pair_launch(CAUSAL, SPARSE, a.Nq == a.Nk, p.nkv, n_items, a.num_sms, 128);
  const bool persistent = pairs || (persistent_launch(CAUSAL, SPARSE, p.nkv) && n_items > a.num_sms);
  const long ctas = persistent ? a.num_sms : n_items;
  // the cross-item V copy pays where CTAs run several items (+6 % on the
  // GPT-2 backward); one-item launches keep the other instantiation, which
  // measured 1-2 % faster for them
  if constexpr (CAUSAL && !SPARSE)
    if (pairs) return launch_k<CAUSAL, SPARSE, true, true>(a, p, ctas, stream);
  if constexpr (!SPARSE)
    if (persistent) return launch_k<CAUSAL, SPARSE, true>(a, p, ctas, stream);
  return launch_k<CAUSAL, SPARSE, false>(a, p, ctas, stream);
}

}  // namespace

cudaError_t launch_bwd_main_d64(const BwdLaunch& a, cudaStream_t stream) {
  if (a.bmask) return a.causal ? launch_t<true, true>(a, stream) : launch_t<false, true>(a, stream);
  return a.causal ? launch_t<true, false>(a, stream) : launch_t<false, false>(a, stream);
}

}  // namespace fa
