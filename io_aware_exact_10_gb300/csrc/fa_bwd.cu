// fa_bwd.cu -- exact softmax attention backward for sm_103a.
//
// The backward recomputes P block by block from Q, K and the saved per-row
// log-sum-exp instead of storing it (FlashAttention: exact attention made fast
// by counting memory traffic, "The method"; FlashAttention and IO-aware exact
// attention, "Backward by recomputation").  The pages print no gradient
// formulas; the ones used are the chain rule through S = scale Q K^T,
// P = softmax(S), O = P V:
//   D_i   = sum_c dO_ic O_ic
//   dP    = dO V^T,   dS = P o (dP - D)
//   dV    = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K
//
// Three kernels, all on the caller's stream:
//   fa_bwd_pre_kernel   D = rowsum(dO o O) and dQacc = 0      (memory bound)
//   fa_bwd_kernel       one CTA per 128-key tile of one head; loops over the
//                       128-query tiles that see it; dK, dV accumulate in
//                       TMEM; dQ contributions are added into dQacc (fp32).
//                       d = 128 uses the kernel below; d = 64 a software-
//                       pipelined variant (fa_bwd_d64.cu) that the smaller
//                       operands leave room for
//   fa_bwd_dq_kernel    dq = bf16(scale * dQacc)                (memory bound)
//
// fa_bwd_kernel roles (448 threads):
//   warps 0-7   P / dS: thread = key row = TMEM lane; warps 0-3 take query
//               columns 0-63 of the tile, warps 4-7 columns 64-127
//   warps 8-11  dQ drain (thread = query row = TMEM lane), then dK epilogue
//   warp  12    TMA producer (K, V once; then Q_i, dO_i through rings of two
//               slots each, or of three for Q and one for dO)
//   warp  13    tcgen05 MMA issuer and TMEM owner
// Tensor memory (512 columns): ST (S^T, then P^T bf16) | DPT (dP^T, then dS^T
// bf16, then dQ) | dV | dK.  The bf16 pairs of P^T and dS^T for queries 0-63
// sit in columns 0-31 of their region and those for queries 64-127 in
// columns 64-95, inside the fp32 columns of the warpgroup that wrote them.  Per query tile the MMA thread issues, in order:
//   S^T = K Q_i^T -> ST;  dP^T = V dO_i^T -> DPT;  dV += P^T dO_i;
//   dK += dS^T Q_i;  dQ_i = dS K -> DPT.
// dS is also written to shared memory (query-major) as the A operand of dQ;
// dQ is staged for its bulk reductions in ring slots of Q_u (and dO_u).
#include <cuda_bf16.h>

#include "fa_kernels.h"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// preprocess: for every row q of every head, D = rowsum(dO * O) and the
// row's statistics for the main kernels, -LSE log2 e and -D (-inf and 0 for
// the pad rows q >= N of a head's last tile; N = query rows); and dQacc = 0.  Statistics
// layout: per head and 128-query tile, 128 values of -LSE log2 e then 128 of
// -D.  A thread takes 8 elements (16 bytes) of a row, a group of HD / 8
// lanes one row; blockIdx.x = head * (blocks per tile * nq) + block.
// ---------------------------------------------------------------------------
template <int HD>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         const float* __restrict__ lse,
                                                         float* __restrict__ stats,
                                                         float* __restrict__ dq_acc, int N, int nq) {
  constexpr int TPR = HD / 8;                  // threads per row
  constexpr int ROWS = 256 / TPR;              // rows per block
  constexpr int BLOCKS_PER_TILE = 128 / ROWS;
  const unsigned blocks_per_head = (unsigned)nq * BLOCKS_PER_TILE;
  const unsigned hb = blockIdx.x / blocks_per_head;
  const int qp = (int)((blockIdx.x - hb * blocks_per_head) * ROWS + threadIdx.x / TPR);  // padded row
  const int part = threadIdx.x % TPR;
  float* st = stats + ((size_t)hb * nq + (qp >> 7)) * 256 + (qp & 127);
  // pad rows take no loads but stay in the warp for the shuffles below
  const bool valid = qp < N;
  const size_t row = (size_t)hb * N + (valid ? qp : 0);
  const float l = valid && part == 0 ? lse[row] : 0.f;
  const size_t base = row * HD + part * 8;
  uint4 a = make_uint4(0u, 0u, 0u, 0u), b = make_uint4(0u, 0u, 0u, 0u);
  if (valid) {
    a = *reinterpret_cast<const uint4*>(o + base);
    b = *reinterpret_cast<const uint4*>(dO + base);
    float4* z = reinterpret_cast<float4*>(dq_acc + base);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fa2 = __bfloat1622float2(a2[i]), fb2 = __bfloat1622float2(b2[i]);
    acc = fmaf(fa2.x, fb2.x, acc);
    acc = fmaf(fa2.y, fb2.y, acc);
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (part == 0) {
    // -inf also for a row that sees no key (lse = -inf under a block mask)
    st[0] = valid && l != -INFINITY ? -l * kLog2e : -INFINITY;
    st[128] = valid ? -acc : 0.f;
  }
}

// ---------------------------------------------------------------------------
// dq = bf16(scale * dQacc).  8 elements per thread.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const float* __restrict__ dq_acc,
                                                        __nv_bfloat16* __restrict__ dq,
                                                        long n8, float scale) {
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(dq_acc)[2 * i + 1];
  uint4 out;
  out.x = pack_bf16(a.x * scale, a.y * scale);
  out.y = pack_bf16(a.z * scale, a.w * scale);
  out.z = pack_bf16(b.x * scale, b.y * scale);
  out.w = pack_bf16(b.z * scale, b.w * scale);
  reinterpret_cast<uint4*>(dq)[i] = out;
}

// ---------------------------------------------------------------------------
// main backward kernel
// ---------------------------------------------------------------------------
template <int HD>
struct BwdCfg {
  static constexpr int BQ = 128;              // queries per iteration
  static constexpr int BK = 128;              // keys per CTA
  static constexpr int KB = HD / 64;          // 64-column blocks per row
  static constexpr int TILE = 128 * HD * 2;   // bytes of one 128-row bf16 tile
  static constexpr int DS_BYTES = BQ * BK * 2;
  // dynamic shared memory layout (offsets from a 1024-byte aligned base)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  // four ring slots for Q and dO: two each, or (persistent launches) three
  // for Q and one for dO
  static constexpr int OFF_Q = OFF_V + TILE;
  static constexpr int OFF_DS = OFF_Q + 4 * TILE;
  static constexpr int OFF_LSE = OFF_DS + DS_BYTES; // 2 x 128 floats (-LSE * log2 e)
  static constexpr int OFF_D = OFF_LSE + 2 * BQ * 4;  // 2 x 128 floats (-D)
  static constexpr int OFF_BAR = OFF_D + 2 * BQ * 4;
  static constexpr int NBAR = 24;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16;
  static constexpr int THREADS = 448;
  static constexpr int W_LOAD = 12, W_MMA = 13;  // warps 0-7: P / dS; 8-11: dQ drain
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_ST = 0, COL_DPT = 128, COL_DV = 256, COL_DK = 256 + HD;
};
static_assert(BwdCfg<128>::SMEM % 16 == 0 && BwdCfg<128>::SMEM + kMaskWords * 4 + 16 <= 232448,
              "shared memory budget with a block-mask column");

// barrier indices
enum : int {
  B_KV = 0, B_QF0 = 1, B_DOF0 = 4, B_QE0 = 6, B_DOE0 = 9,  // up to 3 Q, 2 dO slots
  B_ST = 11, B_DPT = 12, B_P = 13, B_DS = 14, B_DQF = 15, B_DQE = 16, B_FIN = 17,
  B_DRAIN = 18, B_WG = 19, B_DKF = 20, B_DS0 = 21, B_COUNT = 22
};
// arrival counts: TMA / commit barriers take one arrival; B_P, B_DS0 (the
// first half of each warp's dS^T in TMEM) and B_DS one per P/dS warp; B_QE*,
// B_DOE* and B_DQE one per drain warp (the drain frees the slots it stages
// dQ in), except that with one dO slot B_DOE0 is the commit after dV (the
// last MMA that reads dO); B_WG every P/dS thread; B_DKF (dK read out, the
// next item may overwrite it) one per drain warp.
static_assert(B_COUNT <= BwdCfg<128>::NBAR, "barrier slots");
__device__ __constant__ const uint32_t kBarCount[B_COUNT] = {1, 1, 1, 1, 1, 1, 4, 4, 4, 4, 4,
                                                             1, 1, 8, 8, 1, 4, 1, 1, 256, 4, 8};

struct BwdParams {
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

// TMEM column, relative to the S^T (or dP^T) region, of the packed bf16 pairs
// of P^T (or dS^T) for MMA K-step k (16 queries).  Each P/dS warpgroup packs
// its 64 queries into the first 32 columns of its own 64-column half, which it
// has already read: queries 0-63 -> columns 0-31, queries 64-127 -> 64-95.
__device__ __forceinline__ uint32_t pcol(int k) { return (uint32_t)((k >> 2) * 64 + (k & 3) * 8); }

template <bool TEST_FIRST = true>
__device__ __forceinline__ bool warp_wait_b(uint32_t bar, uint32_t parity, const KernelCtl& ctl,
                                            volatile int* abort, uint32_t site) {
  const bool ok = mbar_wait<TEST_FIRST>(bar, parity, ctl, abort, site);
  return __all_sync(0xffffffffu, ok);
}

// SCHED 0: one CTA per item, two Q and two dO slots, dQ staged in the Q and
// dO slots of its tile.  SCHED 1 and 2: persistent CTAs (2: causal, in units
// of two key tiles) with three Q slots and one dO slot, the dO slot refilled
// once dV has read it and dQ staged in two halves in the Q slot.
template <int HD, bool CAUSAL, bool SPARSE, int SCHED = 0>
__global__ void __launch_bounds__(448, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const __grid_constant__ CUtensorMap tdq, const BwdParams p) {
  using C = BwdCfg<HD>;
  extern __shared__ __align__(1024) uint8_t smem[];
  // The swizzled tiles need a 1024-byte aligned base; with no static shared
  // memory the dynamic window starts aligned.  Check rather than assume.
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) record_error(p.ctl, kErrSmemAlign, 1);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + C::NBAR * 8 + 4);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  constexpr bool R3 = SCHED >= 1, PAIRS = SCHED == 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work items are (key/value head, key tile) pairs in a one-dimensional
  // order over (head group, key tile, head): the items of a group's heads run
  // together, share their Q, dO in L2 and add into the same dQ rows (which
  // then stay in L2); key tile 0 (the most work when causal) of every head in
  // the group comes first.  An item loops over the query tiles i0 ... nq-1 of
  // each of the kv_group query heads that share the key/value head, in that
  // order; each role follows the (tile, head) pair of its own position in the
  // loop with a TileWalk.  Persistent launches (see persistent_launch) have
  // one CTA per SM (G CTAs), and CTA b takes items b, 2G-1-b, 2G+b, ...:
  // each pass over G items runs the other way, pairing heavy causal items
  // with light ones.  Persistent causal launches over square heads with many
  // key tiles (SCHED 2) instead walk units of two key tiles of one head, j
  // and nkv-1-j, which see nq + 1 query tiles together whatever j (see
  // decode_pair).  Other launches have one CTA per item.  The ring positions, the per-tile
  // barrier phases and the statistics buffers run on across items (global
  // tile index U); K, V, FIN and "dK read out" have one phase per item.
  const int n_items = p.BHkv * p.nkv;
  const int B0 = (int)blockIdx.x, LS = (int)gridDim.x;
  // k-th item of this CTA (n_items or more: none); a block-sparse CTA has one
  // item, which the compiler then knows: its item loops run once
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
  // column (query tiles i0 .. nq-1) into a bitset after the barrier area;
  // with no kept tile the CTA only zeroes its dK, dV rows.
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
      zero_key_tile<HD>(p.dk, p.dv, bk, kt, p.Nk);
      return;
    }
    qseq.first = next_bit(qbits, qseq.nw, -1);
  }
  const int nit = nqt * p.kv_group;                // query tiles of the first item
  const TileWalk walk0{qseq.first, bk * p.kv_group};
  // per item (dense items after the first): query tiles and query-tile sequence
  auto item_nit = [&](const Item& I) { return (p.nq - I.i0) * p.kv_group; };
  auto item_seq = [&](const Item& I) {
    QuerySeq<SPARSE> s = qseq;
    if constexpr (!SPARSE) s.first = I.i0;
    return s;
  };

  constexpr int QSLOTS = R3 ? 3 : 2;
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sK = s0 + C::OFF_K, sV = s0 + C::OFF_V, sQ = s0 + C::OFF_Q,
                 sDO = sQ + QSLOTS * C::TILE, sDS = s0 + C::OFF_DS;
  // ring slots and barrier phases of global tile u
  // (u >= 0)
  auto qslot = [](int u) { return R3 ? (int)((uint32_t)u % 3u) : (u & 1); };
  auto qphase = [](int u) { return (R3 ? (uint32_t)u / 3u : (uint32_t)u >> 1) & 1u; };
  auto doslot = [](int u) { return R3 ? 0 : (u & 1); };
  auto dophase = [](int u) { return (uint32_t)(R3 ? u : (u >> 1)) & 1u; };
  float* lse_sh = reinterpret_cast<float*>(smem + C::OFF_LSE);
  float* d_sh = reinterpret_cast<float*>(smem + C::OFF_D);

  // The TMA thread initialises the barriers and issues the copies that need
  // no wait (K, V, and Q and dO of the first query tiles) before the
  // CTA-wide sync, so their latency overlaps the rest of the set-up.
  TileWalk lw = walk0;  // the TMA thread's position
  QuerySeq<SPARSE> lseq = qseq;  // and its item's query-tile sequence
  auto issue_q = [&](int u) {
    const int st = qslot(u);
    mbar_arrive_expect_tx(bar(B_QF0 + st), C::TILE);
    for (int b = 0; b < C::KB; ++b)
      tma_load_3d(sQ + st * C::TILE + b * 16384, &tq, bar(B_QF0 + st), b * 64, lw.qt * C::BQ, lw.qh);
  };
  auto issue_do = [&](int u) {  // then moves to the next tile
    const int st = doslot(u);
    mbar_arrive_expect_tx(bar(B_DOF0 + st), C::TILE);
    for (int b = 0; b < C::KB; ++b)
      tma_load_3d(sDO + st * C::TILE + b * 16384, &tdo, bar(B_DOF0 + st), b * 64, lw.qt * C::BQ, lw.qh);
    lseq.next(lw);
  };
  // tiles issued before the sync; with one dO slot the second tile's dO
  // waits for the first tile's dV
  constexpr int PRE = R3 ? 1 : 2;
  const int pre = nit < PRE ? nit : PRE;
  if (warp == C::W_LOAD && lane == 0) {
    *abort = 0;
    for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), R3 && i == B_DOE0 ? 1u : kBarCount[i]);
    fence_barrier_init();
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    tma_prefetch_desc(&tdo);
    tma_prefetch_desc(&tdq);
    mbar_arrive_expect_tx(bar(B_KV), 2 * C::TILE);
    for (int b = 0; b < C::KB; ++b) {
      tma_load_3d(sK + b * 16384, &tk, bar(B_KV), b * 64, kt * C::BK, bk);
      tma_load_3d(sV + b * 16384, &tv, bar(B_KV), b * 64, kt * C::BK, bk);
    }
    for (int u = 0; u < pre; ++u) {
      issue_q(u);
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
      int nkv_issued = 1;  // items whose K, V have been issued
      // Q_u and dO_u of global tile u, once their ring slots are free: a
      // slot's previous tile (u - QSLOTS for Q, u - 1 or u - 2 for dO) has
      // released it (phase of that tile on the slot's barrier)
      auto ring = [&](int u) -> bool {
        const int qs = qslot(u), ds = doslot(u);
        if (u >= QSLOTS && !mbar_wait(bar(B_QE0 + qs), qphase(u) ^ 1u, p.ctl, abort, 10)) return false;
        issue_q(u);
        const int ud = u - (R3 ? 1 : 2);  // the dO slot's previous tile
        if (ud >= 0 && !mbar_wait(bar(B_DOE0 + ds), dophase(ud), p.ctl, abort, 11)) {
          // the Q load above is in flight; wait for it here
          mbar_wait_quiet(bar(B_QF0 + qs), qphase(u), 200000000ull);
          return false;
        }
        issue_do(u);
        return true;
      };
      int u = pre, uend = nit;  // global tile index; end of the current item
      for (int L = L0, kk = 0;;) {
        while (u < uend && (ok = ring(u))) ++u;  // a failed tile is not counted
        if (!ok) break;
        L = item_at(++kk);
        if (L >= n_items) break;
        // the next item: its first tiles (as many as there are dO slots: a
        // later dO waits for a dV of the new item) as soon as their slots
        // are free, then K and V once every MMA of the previous item has
        // completed
        const Item I = item_info(L);
        lw = TileWalk{I.i0, I.bk * p.kv_group};
        lseq = item_seq(I);
        uend = u + item_nit(I);
        const int upre = min(uend, u + PRE);
        while (u < upre && (ok = ring(u))) ++u;
        if (!ok || !(ok = mbar_wait(bar(B_FIN), (nkv_issued - 1) & 1, p.ctl, abort, 12))) break;
        mbar_arrive_expect_tx(bar(B_KV), 2 * C::TILE);
        for (int b = 0; b < C::KB; ++b) {
          tma_load_3d(sK + b * 16384, &tk, bar(B_KV), b * 64, I.kt * C::BK, I.bk);
          tma_load_3d(sV + b * 16384, &tv, bar(B_KV), b * 64, I.kt * C::BK, I.bk);
        }
        ++nkv_issued;
      }
      if (!ok) {
        // Abort: let every copy already issued land before the CTA exits.
        mbar_wait_quiet(bar(B_KV), (nkv_issued - 1) & 1, 200000000ull);
        // (a slot's earlier loads completed before it was refilled)
        for (int v = (u >= QSLOTS ? u - QSLOTS : 0); v < u; ++v)
          mbar_wait_quiet(bar(B_QF0 + qslot(v)), qphase(v), 200000000ull);
        for (int v = (u >= PRE ? u - PRE : 0); v < u; ++v)
          mbar_wait_quiet(bar(B_DOF0 + doslot(v)), dophase(v), 200000000ull);
      }
    }
  } else if (warp == C::W_MMA) {
    // ------------------------------------------------------------------ MMA
    // The whole warp runs the issue loop (control flow and descriptors stay
    // warp-uniform); one elected lane issues.
    {
      const uint32_t lead = elect_one();
      constexpr uint32_t kIdS = idesc_bf16(128, C::BQ, false, false);  // S^T, dP^T
      constexpr uint32_t kIdG = idesc_bf16(128, HD, false, true);      // dV, dK (A in TMEM)
      constexpr uint32_t kIdQ = idesc_bf16(128, HD, true, true);       // dQ = dS K
      const uint32_t tST = tmem + C::COL_ST, tDPT = tmem + C::COL_DPT, tDV = tmem + C::COL_DV,
                     tDK = tmem + C::COL_DK;
      // descriptor halves (sdesc_lo / sdesc_hi): K-major operands with lbo
      // 16, M/N-major ones with lbo 16384; ring slot 0 of Q and dO
      constexpr uint32_t HI = sdesc_hi(1024);
      constexpr uint32_t TILE16 = C::TILE >> 4;
      const uint32_t kK = sdesc_lo(sK, 16), kMN = sdesc_lo(sK, 16384), vK = sdesc_lo(sV, 16);
      const uint32_t qK = sdesc_lo(sQ, 16), qMN = sdesc_lo(sQ, 16384);
      const uint32_t doK = sdesc_lo(sDO, 16), doMN = sdesc_lo(sDO, 16384), dsMN = sdesc_lo(sDS, 16384);
      bool ok = true;
      int U0 = 0;  // global index of the item's first tile
      for (int L = L0, ki = 0; L < n_items && ok; L = item_at(++ki)) {
      const int nit_i = L == L0 ? nit : item_nit(item_info(L));
      if (!(ok = warp_wait_b(bar(B_KV), (uint32_t)ki & 1u, p.ctl, abort, 20))) break;
      for (int u = 0; u < nit_i && ok; ++u) {
        const int U = U0 + u;
        const uint32_t so = (uint32_t)qslot(U) * TILE16, sd = (uint32_t)doslot(U) * TILE16;
        const uint32_t acc0 = u > 0 ? 1u : 0u;
        if (!(ok = warp_wait_b(bar(B_QF0 + qslot(U)), qphase(U), p.ctl, abort, 21))) break;
        tc_fence_after();
        // S^T = K Q_i^T   (M = keys, N = queries, K = d; both K-major)
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t off = (uint32_t)(k / 4) * 1024 + (uint32_t)(k % 4) * 2;
          mma_ss_e(lead, tST, kK + off, HI, qK + so + off, HI, kIdS, k > 0);
        }
        mma_commit_e(lead, bar(B_ST));
        if (!(ok = warp_wait_b(bar(B_DOF0 + doslot(U)), dophase(U), p.ctl, abort, 22))) break;
        if (U > 0 && !(ok = warp_wait_b(bar(B_DQE), (U - 1) & 1, p.ctl, abort, 23))) break;
        tc_fence_after();
        // dP^T = V dO_i^T
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t off = (uint32_t)(k / 4) * 1024 + (uint32_t)(k % 4) * 2;
          mma_ss_e(lead, tDPT, vK + off, HI, doK + sd + off, HI, kIdS, k > 0);
        }
        mma_commit_e(lead, bar(B_DPT));
        // dV += P^T dO_i   (A = P^T bf16 in TMEM, B = dO_i query-major)
        if (!(ok = warp_wait_b(bar(B_P), U & 1, p.ctl, abort, 24))) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < C::BQ / 16; ++k)
          mma_ts_e(lead, tDV, tST + pcol(k), doMN + sd + 128 * k, HI, kIdG, k > 0 ? 1u : acc0);
        if (R3) mma_commit_e(lead, bar(B_DOE0));  // dO_i read: the next dO may load
        // dK += dS^T Q_i   (A = dS^T bf16 in TMEM), in two halves: the
        // K-steps of the queries whose dS^T the P/dS warps write first (0-31
        // and 64-95: steps 0, 1, 4, 5) run while the warps compute the rest
        if (!(ok = warp_wait_b(bar(B_DS0), U & 1, p.ctl, abort, 27))) break;
        // the item's first dK overwrites the previous item's, once the drain
        // has read it out
        if (u == 0 && ki > 0 && !(ok = warp_wait_b(bar(B_DKF), (uint32_t)(ki - 1) & 1u, p.ctl, abort, 26)))
          break;
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int k = (j >> 1) * 4 + (j & 1);
          mma_ts_e(lead, tDK, tDPT + pcol(k), qMN + so + 128 * k, HI, kIdG, k > 0 ? 1u : acc0);
        }
        if (!(ok = warp_wait_b(bar(B_DS), U & 1, p.ctl, abort, 25))) break;
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int k = (j >> 1) * 4 + (j & 1) + 2;
          mma_ts_e(lead, tDK, tDPT + pcol(k), qMN + so + 128 * k, HI, kIdG, 1u);
        }
        // dQ_i = dS K   (M = queries, N = d, K = keys; A = dS smem query-major, B = K key-major)
#pragma unroll
        for (int k = 0; k < C::BK / 16; ++k)
          mma_ss_e(lead, tDPT, dsMN + 128 * k, HI, kMN + 128 * k, HI, kIdQ, k > 0);
        mma_commit_e(lead, bar(B_DQF));
      }
      // every MMA of the item: dK, dV final, K and V free for the next item
      if (ok) mma_commit_e(lead, bar(B_FIN));
      U0 += nit_i;
      }  // items
      mma_commit_e(lead, bar(B_DRAIN));
      mbar_wait_quiet(bar(B_DRAIN), 0, 200000000ull);
    }
  } else if (warp < 8) {
    // --------------------------------------------- P / dS warpgroups (x2)
    // Thread = key row r (TMEM lane); warpgroup h takes query columns
    // [64h, 64h + 64) of the tile.
    const int h = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tST = tmem + lane_off + C::COL_ST, tDPT = tmem + lane_off + C::COL_DPT;
    const int cb = 64 * h;                          // first query column of this thread
    const float scale2 = p.scale2;
    const uint64_t sc2 = f2_pack(scale2, scale2);
    // warpgroup 0 stages the negated log2-scaled LSE and negated D of the
    // first query tile
    if (h == 0) {
      const float* st = p.stats + ((size_t)walk0.qh * p.nq + walk0.qt) * 256;
      lse_sh[r] = st[r];
      d_sh[r] = st[128 + r];
    }
    // Both warpgroups synchronise on an mbarrier (256 arrivals per phase) so
    // that the wait stays bounded if another warp gives up.
    mbar_arrive(bar(B_WG));
    bool ok = warp_wait_b(bar(B_WG), 0, p.ctl, abort, 34);
    int U0 = 0;  // global index of the item's first tile
    for (int L = L0, ki = 0; L < n_items && ok; L = item_at(++ki)) {
    const Item I = L == L0 ? I0 : item_info(L);
    const int kt = I.kt;
    const int nit_i = L == L0 ? nit : item_nit(I);
    const QuerySeq<SPARSE> seq = L == L0 ? qseq : item_seq(I);
    const size_t rowbase = (size_t)I.bk * p.Nk;      // key rows (dK, dV)
    // the next item's first tile, whose statistics this item's last tile fetches
    const int Ln = item_at(ki + 1);
    const bool has_next = Ln < n_items;
    TileWalk wn{0, 0};
    if (has_next) {
      const Item In = item_info(Ln);
      wn = TileWalk{item_seq(In).first, In.bk * p.kv_group};
    }
    TileWalk w = L == L0 ? walk0 : TileWalk{seq.first, I.bk * p.kv_group};
    for (int u = 0; u < nit_i && ok; ++u) {
      const int U = U0 + u;
      const int qt = w.qt;
      seq.next(w);  // w now names tile u + 1 ...
      if (u + 1 == nit_i) w = wn;  // ... or the next item's first
      const float* lse_u = lse_sh + (U & 1) * C::BQ + cb;
      const float* d_u = d_sh + (U & 1) * C::BQ + cb;
      // next tile's statistics, copied asynchronously so that no warp
      // stalls on the global loads; waited for at the end of the iteration
      float* lse_n = lse_sh + ((U + 1) & 1) * C::BQ + r;
      float* d_n = d_sh + ((U + 1) & 1) * C::BQ + r;
      const bool fetch = h == 0 && (u + 1 < nit_i || has_next);
      if (fetch) {
        const float* st = p.stats + ((size_t)w.qh * p.nq + w.qt) * 256;
        cp_async_4(smem_u32(lse_n), st + r, 4u);
        cp_async_4(smem_u32(d_n), st + 128 + r, 4u);
        cp_async_commit();
      }
      if (!(ok = warp_wait_b(bar(B_ST), U & 1, p.ctl, abort, 30))) break;
      tc_fence_after();
      // statistics four at a time (one 16-byte broadcast load per two pairs),
      // the first chunk's while the TMEM loads are in flight
      auto load_stats = [](const float* src, uint64_t (&dst)[16]) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(src + 4 * i);
          dst[2 * i] = v.x;
          dst[2 * i + 1] = v.y;
        }
      };
      float pr[64];
      tmem_ld32(tST + cb, *reinterpret_cast<uint32_t(*)[32]>(pr));
      tmem_ld32(tST + cb + 32, *reinterpret_cast<uint32_t(*)[32]>(pr + 32));
      uint64_t nlp[16];
      load_stats(lse_u, nlp);
      tmem_wait_ld();
      // P^T[r][q] = exp2(scale2 * S^T - LSE2_q); causal: zero where query
      // qt*128 + q does not see key kt*128 + r, i.e. q < r + (kt - qt)*128 - coff.
      // The tile needs it when that bound is positive for the last key.
      const int qdelta = (kt - qt) * C::BK - p.coff;
      const bool diag = CAUSAL && qdelta > 1 - C::BK;
      const int rlim = r + qdelta;
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t pk[16];
        if (c0 > 0) load_stats(lse_u + c0, nlp);
        // two queries per paired FMA: scale2 * s - LSE2 (the shared copy holds
        // -LSE2).  Persistent launches branch (warp-uniformly) to a loop
        // without the mask's compares and selects on the tiles that need no
        // mask: +1-1.5 % there; one-CTA-per-item launches keep one loop,
        // whose registers the second would push into spills.
        if (SCHED == 0 || diag) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int q = c0 + 2 * i;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(pr[q], pr[q + 1]), sc2, nlp[i]), x0, x1);
            float p0 = ex2(x0), p1 = ex2(x1);
            if (diag && cb + q < rlim) p0 = 0.f;
            if (diag && cb + q + 1 < rlim) p1 = 0.f;
            pk[i] = pack_bf16(p0, p1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int q = c0 + 2 * i;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(pr[q], pr[q + 1]), sc2, nlp[i]), x0, x1);
            pk[i] = pack_bf16(ex2(x0), ex2(x1));
          }
        }
        tmem_st16(tST + cb + c0 / 2, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_P));
      // dS^T = P^T o (dP^T - D), with P^T the bf16 values dV multiplied
      // The dS buffer is the A operand of dQ_{U-1}, which has completed
      // when dP^T_U has: the MMA warp issues dP^T_U after it, and the commit
      // behind B_DPT covers every MMA issued before.
      if (!(ok = warp_wait_b(bar(B_DPT), U & 1, p.ctl, abort, 31))) break;
      tc_fence_after();
      const uint32_t srow = sDS + (uint32_t)h * 16384u + (uint32_t)r * 128u;
      const uint32_t sw = (uint32_t)(r & 7);
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        // dP^T of 32 queries, and the bf16 pairs of P^T that dV used for them
        uint32_t dp[32], pp[16];
        tmem_ld32(tDPT + cb + c0, dp);
        tmem_ld16(tST + cb + c0 / 2, pp);
        uint64_t ndp[16];
        load_stats(d_u + c0, ndp);  // while the TMEM loads are in flight
        tmem_wait_ld();
        uint32_t pk[16];
        // two queries per paired add and multiply: (dP - D) * P (the shared
        // copy holds -D)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint64_t nd2 = ndp[i];
          const uint32_t w = pp[i];
          const uint64_t pv = f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
          float a, b;
          f2_unpack(f2_mul(f2_add(f2_pack(__uint_as_float(dp[2 * i]), __uint_as_float(dp[2 * i + 1])), nd2), pv), a, b);
          pk[i] = pack_bf16(a, b);
        }
        tmem_st16(tDPT + cb + c0 / 2, pk);
        // shared copy, query-major 128-byte swizzled: block h, chunks of 8 queries
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint32_t chunk = (uint32_t)(c0 / 8 + cc);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(srow + ((chunk ^ sw) << 4)),
                       "r"(pk[4 * cc]), "r"(pk[4 * cc + 1]), "r"(pk[4 * cc + 2]), "r"(pk[4 * cc + 3])
                       : "memory");
        }
        if (c0 == 0) {  // the first 32 queries' dS^T is in TMEM: dK may take them
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_DS0));
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DS));
      // publish the next tile's statistics
      if (fetch) cp_async_wait_all();
      mbar_arrive(bar(B_WG));
      if (!(ok = warp_wait_b(bar(B_WG), (U + 1) & 1, p.ctl, abort, 35))) break;
    }
    cp_async_wait_all();  // none in flight when a wait above gave up
    // epilogue: dV rows of this key tile, columns [h*HD/2, (h+1)*HD/2); the
    // next item's first dV (after this warp's next P) overwrites them
    if (ok && (ok = warp_wait_b(bar(B_FIN), (uint32_t)ki & 1u, p.ctl, abort, 33))) {
      tc_fence_after();
      const int key = kt * C::BK + r;
      __nv_bfloat16* dst = p.dv + (rowbase + key) * HD;
#pragma unroll 1
      for (int c0 = h * (HD / 2); c0 < (h + 1) * (HD / 2); c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + C::COL_DV + c0, v);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        if (key < p.Nk) {
          st_global_64B(dst + c0, pk);
        }
      }
    }
    U0 += nit_i;
    }  // items
  } else {
    // ---------------------------------------------------------- dQ drain
    // dQ_u (128 query rows x d, fp32) leaves TMEM 64 columns at a time and is
    // added into dQacc by TMA bulk reductions of 32-row x 32-column boxes
    // (128-byte swizzled), staged in ring slots that no MMA reads once dQ_u
    // is complete.  Each warp's quarter of a slot holds two boxes (64
    // columns of its rows).  Two dO slots: the first half goes to the Q_u
    // slot, which is released as soon as the reductions have read it (the
    // next S^T needs it before the next dP^T needs a dO slot), the second to
    // the dO_u slot.  One dO slot: both halves go to the Q_u slot, the second
    // once the first has been read; both leave TMEM before that wait, so the
    // columns are free as early.
    const int sp = warp & 3;
    const int r = sp * 32 + lane;  // query row within the tile (dQ) / key row (dK)
    const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
    const uint32_t sw = (uint32_t)(lane & 7);
    static_assert(HD / 64 == 2, "two 64-column halves, one bulk group each");
    bool ok = true;
    int U0 = 0;  // global index of the item's first tile
    for (int L = L0, ki = 0; L < n_items && ok; L = item_at(++ki)) {
    const Item I = L == L0 ? I0 : item_info(L);
    const int kt = I.kt;
    const int nit_i = L == L0 ? nit : item_nit(I);
    const QuerySeq<SPARSE> seq = L == L0 ? qseq : item_seq(I);
    const size_t rowbase = (size_t)I.bk * p.Nk;      // key rows (dK, dV)
    TileWalk w = L == L0 ? walk0 : TileWalk{seq.first, I.bk * p.kv_group};
    for (int u = 0; u < nit_i; ++u, seq.next(w)) {
      const int U = U0 + u;
      if (!(ok = warp_wait_b(bar(B_DQF), U & 1, p.ctl, abort, 40))) break;
      tc_fence_after();
      const uint32_t quarter = (uint32_t)sp * (uint32_t)(C::TILE / 4);  // 8 KB
      const uint32_t stage_q = sQ + qslot(U) * C::TILE + quarter;
      const uint32_t stage_2 = R3 ? stage_q : sDO + doslot(U) * C::TILE + quarter;
      const int y = w.qt * C::BQ + sp * 32, zq = w.qh;
#pragma unroll
      for (int hh = 0; hh < HD / 64; ++hh) {
        uint32_t v[64];
        tmem_ld32(tmem + lane_off + C::COL_DPT + hh * 64, *reinterpret_cast<uint32_t(*)[32]>(v));
        tmem_ld32(tmem + lane_off + C::COL_DPT + hh * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
        tmem_wait_ld();
        if (hh == HD / 64 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_DQE));  // dQ's TMEM columns are free again
        }
        if (R3 && hh > 0) {  // the first half's boxes must have been read
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
        }
        const uint32_t stage = hh == 0 ? stage_q : stage_2;
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          // box 2 hh + bb: columns [64 hh + 32 bb, 64 hh + 32 bb + 32)
          const uint32_t row = stage + (uint32_t)bb * 4096u + (uint32_t)lane * 128u;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int col = bb * 32 + c * 4;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (((uint32_t)c ^ sw) << 4)),
                         "r"(v[col]), "r"(v[col + 1]), "r"(v[col + 2]), "r"(v[col + 3])
                         : "memory");
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int bb = 0; bb < 2; ++bb)
            tma_reduce_add_3d(&tdq, stage + (uint32_t)bb * 4096u, (2 * hh + bb) * 32, y, zq);
          bulk_commit_group();
        }
      }
      // once their boxes have been read, the slots may be refilled
      if (lane == 0) {
        if constexpr (R3) {
          bulk_wait_group_read<0>();
          mbar_arrive(bar(B_QE0 + qslot(U)));
        } else {
          bulk_wait_group_read<1>();
          mbar_arrive(bar(B_QE0 + qslot(U)));
          bulk_wait_group_read<0>();
          mbar_arrive(bar(B_DOE0 + doslot(U)));
        }
      }
      __syncwarp();
    }
    // epilogue: dK rows of this key tile (scaled); then "dK read out" lets
    // the next item's first dK overwrite them
    if (ok && (ok = warp_wait_b(bar(B_FIN), (uint32_t)ki & 1u, p.ctl, abort, 41))) {
      tc_fence_after();
      const int key = kt * C::BK + r;
      __nv_bfloat16* dst = p.dk + (rowbase + key) * HD;
      const float scale = p.scale;
#pragma unroll 1
      for (int c0 = 0; c0 < HD; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + C::COL_DK + c0, v);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16(__uint_as_float(v[2 * i]) * scale, __uint_as_float(v[2 * i + 1]) * scale);
        if (key < p.Nk) {
          st_global_64B(dst + c0, pk);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DKF));
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

template <int HD, bool CAUSAL, bool SPARSE>
cudaError_t launch_bwd_main(const BwdLaunch& a, cudaStream_t stream) {
  using C = BwdCfg<HD>;
  BwdParams p;
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
  // one persistent CTA per SM walks the items (with the three-Q-slot ring,
  // measured faster there), or one CTA per item; long square causal
  // launches in units of two key tiles (pair_launch; measured +4 % at 32 key
  // tiles per head, +1.5 % at 64, +1.3 % at 128, -0.9 % at 256)
  const long n_items = (long)p.nkv * p.BHkv;
  const bool pairs = pair_launch(CAUSAL, SPARSE, a.Nq == a.Nk, p.nkv, n_items, a.num_sms, 128);
  const bool pers = pairs || (persistent_launch(CAUSAL, SPARSE, p.nkv) && n_items > a.num_sms);
  const long ctas = pers ? a.num_sms : n_items;
  auto kern = fa_bwd_kernel<HD, CAUSAL, SPARSE, 0>;
  if constexpr (!SPARSE) {
    if (pers) kern = fa_bwd_kernel<HD, CAUSAL, SPARSE, 1>;
    if constexpr (CAUSAL)
      if (pairs) kern = fa_bwd_kernel<HD, CAUSAL, SPARSE, 2>;
  }
  // block-sparse: the mask column's bitset and its count follow the layout
  const int smem_bytes = C::SMEM + (SPARSE ? kMaskWords * 4 + 16 : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)ctas);
  kern<<<grid, C::THREADS, smem_bytes, stream>>>(a.tq, a.tk, a.tv, a.tdo, a.tdq, p);
  return cudaGetLastError();
}

template <int HD>
cudaError_t launch_bwd_t(const BwdLaunch& a, cudaStream_t stream) {
  const long rows = (long)a.BH * a.Nq;
  const int nq = (a.Nq + 127) / 128;
  fa_bwd_pre_kernel<HD><<<(unsigned)((long)a.BH * nq * (128 / (256 / (HD / 8)))), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dO), a.lse, a.stats,
      a.dq_acc, a.Nq, nq);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if constexpr (HD == 64)
    e = launch_bwd_main_d64(a, stream);
  else
    e = a.bmask ? (a.causal ? launch_bwd_main<HD, true, true>(a, stream)
                            : launch_bwd_main<HD, false, true>(a, stream))
                : (a.causal ? launch_bwd_main<HD, true, false>(a, stream)
                            : launch_bwd_main<HD, false, false>(a, stream));
  if (e != cudaSuccess) return e;
  const long n8 = rows * HD / 8;
  fa_bwd_dq_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, stream>>>(
      a.dq_acc, static_cast<__nv_bfloat16*>(a.dq), n8, a.scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdLaunch& a, cudaStream_t stream) {
  return a.d == 128 ? launch_bwd_t<128>(a, stream) : launch_bwd_t<64>(a, stream);
}

}  // namespace fa
