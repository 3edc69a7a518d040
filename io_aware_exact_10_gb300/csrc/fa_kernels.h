// fa_kernels.h -- host-side launch interface between the C-ABI layer and the
// kernel translation units.  Not part of the public header.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"

namespace fa {

// Everything a forward launch needs; tensor maps are encoded by the caller.
struct FwdLaunch {
  CUtensorMap tq;               // bf16 [BH][Nq][d], box {64, 128, 1}, 128-byte swizzle
  CUtensorMap tk, tv;           // bf16 [BH / group][Nk][d], same box
  void* o;                      // bf16 [BH][Nq][d]
  float* lse;                   // fp32 [BH][Nq]
  int BH, Nq, Nk, d;            // causal requires Nk >= Nq (bottom-right aligned)
  int group;                    // query heads per key/value head (1: multi-head)
  int num_sms;                  // multiprocessors of the device (grid ordering)
  float scale;
  int causal;
  KernelCtl ctl;
};

// Everything a backward launch needs.
struct BwdLaunch {
  CUtensorMap tq, tdo;          // bf16 [BH][Nq][d], box {64, 128, 1}, 128-byte swizzle
  CUtensorMap tk, tv;           // bf16 [BH / group][Nk][d], same box
  CUtensorMap tdq;              // fp32 dQacc [BH][Nq][d], box {32, 32, 1}, 128-byte swizzle
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
  KernelCtl ctl;
};

// First query tile whose rows see any key of key tile kt (tiles of 128):
// query i sees key j iff j <= i + coff, so the tile holding row kt*128 - coff.
__host__ __device__ inline int first_query_tile(int kt, int coff) {
  const int r = kt * 128 - coff;
  return r > 0 ? r / 128 : 0;
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

// Each returns cudaSuccess or the launch error; nothing is synchronised.
cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream);
cudaError_t launch_bwd(const BwdLaunch& a, cudaStream_t stream);
// main backward kernel for d = 64 (the D preprocess and dQ convert stay in launch_bwd)
cudaError_t launch_bwd_main_d64(const BwdLaunch& a, cudaStream_t stream);

}  // namespace fa
