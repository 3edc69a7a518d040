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
  CUtensorMap tq, tk, tv;       // bf16 [BH][N][d], box {64, 128, 1}, 128-byte swizzle
  void* o;                      // bf16 [BH][N][d]
  float* lse;                   // fp32 [BH][N]
  int BH, N, d;
  float scale;
  int causal;
  KernelCtl ctl;
};

// Everything a backward launch needs.
struct BwdLaunch {
  CUtensorMap tq, tk, tv, tdo;  // bf16 [BH][N][d], box {64, 128, 1}, 128-byte swizzle
  CUtensorMap tdq;              // fp32 dQacc [BH][N][d], box {32, 32, 1}, 128-byte swizzle
  const void* o;                // bf16 [BH][N][d]
  const void* dO;               // bf16 [BH][N][d]
  const float* lse;             // fp32 [BH][N]
  float* D;                     // fp32 [BH][N] workspace
  float* dq_acc;                // fp32 [BH][N][d] workspace
  void* dq;                     // bf16 [BH][N][d]
  void* dk;                     // bf16 [BH][N][d]
  void* dv;                     // bf16 [BH][N][d]
  int BH, N, d;
  float scale;
  int causal;
  KernelCtl ctl;
};

// Each returns cudaSuccess or the launch error; nothing is synchronised.
cudaError_t launch_fwd(const FwdLaunch& a, cudaStream_t stream);
cudaError_t launch_bwd(const BwdLaunch& a, cudaStream_t stream);

}  // namespace fa
