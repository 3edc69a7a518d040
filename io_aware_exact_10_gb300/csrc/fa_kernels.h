// fa_kernels.h -- host-side launch interface between the C-ABI layer and the
// kernel translation units.  Not part of the public header.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "sm103_ptx.cuh"

namespace fa {

// Everything a forward launch needs; tensor maps are encoded by the caller.
struct FwdLaunch {
  CUtensorMap tq;               // bf16 [BH][Nq][d], box {64, 128, 1}, 128-byte swizzle
  CUtensorMap tk, tv;           // bf16 [BH / group][Nk][d], box {64, key_tile, 1}
  CUtensorMap to;               // bf16 [BH][Nq][d] output, box {64, 32, 1} (d = 64 stores)
  void* o;                      // bf16 [BH][Nq][d]
  float* lse;                   // fp32 [BH][Nq]
  int BH, Nq, Nk, d;            // causal requires Nk >= Nq (bottom-right aligned)
  int group;                    // query heads per key/value head (1: multi-head)
  int num_sms;                  // multiprocessors of the device (grid ordering)
  float scale;
  int causal;
  const uint8_t* bmask;         // block mask [ceil(Nq/128)][ceil(Nk/128)], or null (dense)
  int key_tile = 128;           // keys per K/V tile: 128, or 64 (dense only)
  KernelCtl ctl;
};

// Everything a backward launch needs.
struct BwdLaunch {
  CUtensorMap tq, tdo;          // bf16 [BH][Nq][d], box {64, 128, 1}, 128-byte swizzle
  CUtensorMap tk, tv;           // bf16 [BH / group][Nk][d], same box
  CUtensorMap tdq;              // fp32 dQacc [BH][Nq][d], box {32, 32, 1}, 128-byte swizzle
  CUtensorMap tdk;              // bf16 dk [BH / group][Nk][d], box {64, 32, 1} (d = 64 stores)
  const void* o;                // bf16 [BH][Nq][d]
  const void* dO;               // bf16 [BH][Nq][d]
  const float* lse;             // fp32 [BH][Nq]
  float* stats;                 // fp32 [BH][nq][2][128] workspace: per 128-query tile,
                                // -LSE log2 e then -D of its rows (-inf, 0 past Nq)
  float* dq_acc;                // fp32 [BH][Nq][d] workspace
  void* dq;                     // bf16 [BH][Nq][d]
  void* dk;                     // bf16 [BH / group][Nk][d]
  void* dv;                     // bf16 [BH / group][Nk][d]
  int BH, Nq, Nk, d;            // causal requires Nk >= Nq (bottom-right aligned)
  int group;                    // query heads per key/value head (1: multi-head)
  int num_sms;                  // multiprocessors of the device (grid ordering)
  float scale;
  int causal;
  const uint8_t* bmask;         // block mask as for the forward, or null (dense)
  KernelCtl ctl;
};

// First query tile whose rows see any key of key tile kt (tiles of 128):
// query i sees key j iff j <= i + coff, so the tile holding row kt*128 - coff.
__host__ __device__ inline int first_query_tile(int kt, int coff) {
  const int r = kt * 128 - coff;
  return r > 0 ? r / 128 : 0;
}

// Block-sparse attention: a block mask holds one byte per 128 x 128 block of
// (query rows, keys), row-major [ceil(Nq/128)][ceil(Nk/128)], shared by all
// heads; nonzero keeps the block.  A CTA turns the rows (forward) or the
// column (backward) it needs into bitsets in shared memory.
constexpr int kMaskMaxTiles = 4096;  // tiles per side a block mask may have
constexpr int kMaskWords = kMaskMaxTiles / 32;

// One warp: bit i of words[i / 32] = (base[i * stride] != 0) for i in
// [lo, hi), 0 elsewhere, for words 0 .. nw-1.  Eight loads per lane are in
// flight before the first ballot.
__device__ __forceinline__ void mask_bits_warp(const uint8_t* __restrict__ base, long stride,
                                               int lo, int hi, int nw, uint32_t* words, int lane) {
  for (int w0 = 0; w0 < nw; w0 += 8) {
    bool b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = (w0 + i) * 32 + lane;
      b[i] = w0 + i < nw && j >= lo && j < hi && base[(long)j * stride] != 0;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t bits = __ballot_sync(0xffffffffu, b[i]);
      if (lane == 0 && w0 + i < nw) words[w0 + i] = bits;
    }
  }
}

// One warp: number of set bits in words 0 .. nw-1 (every lane gets it).
__device__ __forceinline__ int mask_popc_warp(const uint32_t* words, int nw, int lane) {
  int c = 0;
  for (int w = lane; w < nw; w += 32) c += __popc(words[w]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  return c;
}

// Smallest set bit index greater than `after` in words 0 .. nw-1, or -1.
__device__ __forceinline__ int next_bit(const uint32_t* words, int nw, int after) {
  const int j = after + 1;
  int w = j >> 5;
  if (w >= nw) return -1;
  uint32_t x = words[w] & (0xffffffffu << (j & 31));
  while (x == 0) {
    if (++w >= nw) return -1;
    x = words[w];
  }
  return (w << 5) + __ffs(x) - 1;
}

// Position in a backward CTA's loop over (query head, query tile): tiles
// first .. nq-1 of one query head, then of the next head of the group.
struct TileWalk {
  int qt, qh;
  __host__ __device__ void next(int first, int nq) {
    if (++qt == nq) {
      qt = first;
      ++qh;
    }
  }
};

// The query tiles a backward CTA visits for its key tile, per query head of
// the group: first .. nq-1 (dense), or the tiles whose bit is set in the
// CTA's bitset of its block-mask column (block-sparse; `first` is the lowest).
template <bool SPARSE>
struct QuerySeq {
  const uint32_t* bits;
  int nw, first, nq;
  __device__ __forceinline__ void next(TileWalk& w) const {
    if constexpr (SPARSE) {
      const int n = next_bit(bits, nw, w.qt);
      if (n < 0) {
        w.qt = first;
        ++w.qh;
      } else {
        w.qt = n;
      }
    } else {
      w.next(first, nq);
    }
  }
};

// Zero dK and dV of key rows [kt*128, kt*128 + 128) of key/value head bk
// (cut at Nk): a key tile that no kept block reaches has zero gradients.
template <int HD>
__device__ __forceinline__ void zero_key_tile(__nv_bfloat16* dk, __nv_bfloat16* dv, int bk, int kt,
                                              int Nk) {
  const int rows = min(128, Nk - kt * 128);
  const size_t base = ((size_t)bk * Nk + (size_t)kt * 128) * HD;
  uint4* zk = reinterpret_cast<uint4*>(dk + base);
  uint4* zv = reinterpret_cast<uint4*>(dv + base);
  for (int i = threadIdx.x; i < rows * (HD / 8); i += blockDim.x) {
    zk[i] = make_uint4(0u, 0u, 0u, 0u);
    zv[i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Persistent CTAs (one per SM walking the work items in snake order) or one
// CTA per item, which the hardware schedules dynamically.  Persistent saves
// each item's launch gap and set-up (a few microseconds); the static snake
// order balances items of equal work, and causal items as long as a head has
// few tiles: with tiles_per_head = 32 or more the busiest CTA measured (in a
// simulation of the orders) 8-16 % above the mean, against about 1 % for the
// dynamic order.  Block-sparse items are uneven in no set order.
inline bool persistent_launch(bool causal, bool sparse, int tiles_per_head) {
  return !sparse && (!causal || tiles_per_head <= 16);
}

// Heads per scheduling group: enough tiles for about two waves of CTAs, so a
// group's heads stay resident in L2 while its heaviest tiles start first.
inline int head_group(int BH, int tiles_per_head, int num_sms) {
  int g = (2 * num_sms + tiles_per_head - 1) / tiles_per_head;
  return g < 1 ? 1 : (g > BH ? BH : g);
}

// Decode a one-dimensional grid index into (head, tile rank): heads come in
// groups of `group`; inside a group the tile rank varies slowest, so rank 0
// (the heaviest tile when causal) of every head in the group comes first.
struct GridPos {
  int bh, rank;
};
__host__ __device__ inline GridPos decode_grid(int L, int BH, int tiles, int group) {
  const int per_group = group * tiles;
  const int g = L / per_group;
  const int idx = L - g * per_group;
  const int gh = (BH - g * group) < group ? (BH - g * group) : group;
  GridPos r;
  r.rank = idx / gh;
  r.bh = g * group + (idx - r.rank * gh);
  return r;
}

// Persistent causal launches over square heads (query and key tiles alike)
// may instead walk units of two tiles of one head, j and tiles-1-j, whose
// causal work sums to the same for every j: unit u is (head u / (tiles/2),
// j = u mod tiles/2), and item 2u + s its tile j (s = 0, the heavier) or
// tiles-1-j (s = 1).  CTA b of G takes units b, b + G, b + 2G, ...
__host__ __device__ inline GridPos decode_pair(int L, int tiles) {
  const int hk = tiles >> 1, unit = L >> 1, h = unit / hk, j = unit - h * hk;
  GridPos r;
  r.bh = h;
  r.rank = (L & 1) ? tiles - 1 - j : j;
  return r;
}

// Whether a launch takes the paired schedule: causal, dense, square, an even
// number of tiles per head between persistent_launch's limit and max_tiles
// (the kernel's measured break-even), and units that fill the last wave of
// CTAs to 95 % or more.
inline bool pair_launch(bool causal, bool sparse, bool square, int tiles_per_head, long items,
                        int num_sms, int max_tiles) {
  if (!causal || sparse || !square || tiles_per_head % 2 != 0 || tiles_per_head > max_tiles ||
      persistent_launch(causal, sparse, tiles_per_head))
    return false;
  const long units = items / 2, waves = (units + num_sms - 1) / num_sms;
  return units >= num_sms && units * 20 >= waves * num_sms * 19;
}

// Each returns cudaSuccess or the launch error; nothing is synchronised.
cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream);
cudaError_t launch_bwd(const BwdLaunch& a, cudaStream_t stream);
// main backward kernel for d = 64 (the D preprocess and dQ convert stay in launch_bwd)
cudaError_t launch_bwd_main_d64(const BwdLaunch& a, cudaStream_t stream);

}  // namespace fa
