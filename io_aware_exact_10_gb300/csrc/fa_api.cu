// fa_api.cu -- the C ABI declared in include/fa.h: argument validation,
// tensor-map encoding, per-device state and kernel launches.  No device
// memory is allocated here; the only device-resident state is one error word
// per device (a file-scope __device__ variable).
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/fa.h"
#include "fa_kernels.h"

namespace {

__device__ unsigned long long g_fa_error_word;

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;

struct DeviceState {
  std::once_flag once;
  bool supported = false;
  int num_sms = 0;
  unsigned long long* err = nullptr;  // device address of g_fa_error_word
  cudaError_t init_error = cudaSuccess;
};
DeviceState g_dev[kMaxDevices];

std::atomic<unsigned long long> g_timeout_ns{0};
std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

unsigned long long timeout_ns() {
  unsigned long long t = g_timeout_ns.load(std::memory_order_relaxed);
  if (t) return t;
  static const unsigned long long env = [] {
    const char* s = std::getenv("FA_WAIT_TIMEOUT_MS");
    if (!s) return 0ull;
    const double ms = std::atof(s);
    return ms > 0 ? (unsigned long long)(ms * 1e6) : 0ull;
  }();
  return env ? env : kDefaultTimeoutNs;
}

// Resolve the current device: sm_103 check and the error word's address.
fa_status current_device(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return FA_ERR_NO_DEVICE;
  }
  if (dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  DeviceState& st = g_dev[dev];
  std::call_once(st.once, [&st, dev] {
    cudaDeviceProp prop;
    if ((st.init_error = cudaGetDeviceProperties(&prop, dev)) != cudaSuccess) return;
    st.supported = prop.major == 10 && prop.minor == 3;
    st.num_sms = prop.multiProcessorCount;
    void* p = nullptr;
    if ((st.init_error = cudaGetSymbolAddress(&p, g_fa_error_word)) != cudaSuccess) return;
    st.err = static_cast<unsigned long long*>(p);
  });
  if (st.init_error != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  if (!st.supported) return FA_ERR_UNSUPPORTED;
  *out = &st;
  return FA_OK;
}

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      cudaGetLastError();
  });
  return g_encode != nullptr;
}

// bf16 [BH][N][d] viewed as a 3-D tensor (d, N, BH); box of 64 columns x
// `rows` rows (128; 64 for 64-key tiles; 32 for one warp's rows of O),
// 128-byte swizzle (the layout the tcgen05 descriptors expect).
bool encode_bf16_3d(CUtensorMap* m, const void* ptr, int BH, int N, int d, int rows = 128) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [BH][N][d] dQ accumulator; box of 32 columns x 32 rows, 128-byte
// swizzle (one warp's slice of a tile, the unit of the bulk reductions).
bool encode_f32_3d(CUtensorMap* m, const void* ptr, int BH, int N, int d) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)N * d * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxRows = 1 << 30;  // per head, query rows and keys

// Shared validation of sizes and scalars.  *empty is set for a problem with
// no query rows (B, H or Nq zero); nothing is computed for it.
fa_status check_common(int B, int H, int H_kv, int Nq, int Nk, int d, float scale, int causal,
                       bool* empty) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || Nq > kMaxRows || Nk > kMaxRows)
    return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  *empty = (B == 0 || H == 0 || Nq == 0);
  if (B > 0 && H > 0 && (H_kv < 1 || H_kv > H || H % H_kv != 0)) return FA_ERR_INVALID_ARG;
  if (*empty) return FA_OK;
  // every query row needs a key; causal masking aligns the last query with
  // the last key, so it needs at least as many keys as queries
  if (Nk == 0 || (causal && Nk < Nq)) return FA_ERR_INVALID_ARG;
  // one-dimensional grids of (query-tile pairs or key tiles) x heads, and
  // the backward preprocess's 16 blocks per 128-row tile
  const long long BH = (long long)B * H;
  if (BH * ((Nq + 127) / 128) * 16 > 0x7FFFFFFFLL) return FA_ERR_INVALID_ARG;
  if (BH * ((Nk + 127) / 128) > 0x7FFFFFFFLL) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }
// a block mask has at most kMaskMaxTiles tiles per side (the kernels keep a
// row or column of it as a bitset in shared memory)
bool mask_fits(int Nq, int Nk) {
  return (Nq + 127) / 128 <= fa::kMaskMaxTiles && (Nk + 127) / 128 <= fa::kMaskMaxTiles;
}
// floats of the backward's row statistics: two per row, each head padded to
// whole 128-row tiles
size_t stats_floats(int BH, int N) { return (size_t)BH * (size_t)((N + 127) / 128) * 256; }

// The forward behind fa_fwd_sparse (128-key tiles, optional block mask)
// and fa_fwd_tiled (dense, 64- or 128-key tiles).
fa_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int H_kv, int N_q, int N_k, int d, float scale, int causal,
                   const unsigned char* block_mask, int key_tile, struct CUstream_st* stream);

}  // namespace

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, struct CUstream_st* stream) {
  return fa_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, scale, causal, stream);
}

fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int H_kv, int N, int d, float scale, int causal,
                     struct CUstream_st* stream) {
  return fa_fwd_ex(q, k, v, o, lse, B, H, H_kv, N, N, d, scale, causal, stream);
}

fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int H, int H_kv, int N_q, int N_k, int d, float scale, int causal,
                    struct CUstream_st* stream) {
  return fa_fwd_sparse(q, k, v, o, lse, B, H, H_kv, N_q, N_k, d, scale, causal, nullptr, stream);
}

fa_status fa_fwd_sparse(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int H_kv, int N_q, int N_k, int d, float scale, int causal,
                        const unsigned char* block_mask, struct CUstream_st* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, H_kv, N_q, N_k, d, scale, causal, block_mask, 128, stream);
}

fa_status fa_fwd_tiled(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int H_kv, int N_q, int N_k, int d, float scale, int causal,
                       int key_tile, struct CUstream_st* stream) {
  if (key_tile != 64 && key_tile != 128) return FA_ERR_UNSUPPORTED;
  return fwd_impl(q, k, v, o, lse, B, H, H_kv, N_q, N_k, d, scale, causal, nullptr, key_tile,
                  stream);
}

}  // extern "C"

namespace {

fa_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int H_kv, int N_q, int N_k, int d, float scale, int causal,
                   const unsigned char* block_mask, int key_tile, struct CUstream_st* stream) {
  bool empty = false;
  fa_status s = check_common(B, H, H_kv, N_q, N_k, d, scale, causal, &empty);
  if (s != FA_OK || empty) return s;
  if (block_mask && !mask_fits(N_q, N_k)) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  DeviceState* dev = nullptr;
  if ((s = current_device(&dev)) != FA_OK) return s;
  if (!get_encoder()) return FA_ERR_LAUNCH;
  fa::FwdLaunch a;
  const int BH = B * H, BHkv = B * H_kv;
  if (!encode_bf16_3d(&a.tq, q, BH, N_q, d) || !encode_bf16_3d(&a.tk, k, BHkv, N_k, d, key_tile) ||
      !encode_bf16_3d(&a.tv, v, BHkv, N_k, d, key_tile) || !encode_bf16_3d(&a.to, o, BH, N_q, d, 32))
    return FA_ERR_INVALID_ARG;
  a.key_tile = key_tile;
  a.o = o;
  a.lse = lse;
  a.BH = BH;
  a.group = H / H_kv;
  a.Nq = N_q;
  a.Nk = N_k;
  a.d = d;
  a.scale = scale;
  a.causal = causal;
  a.bmask = block_mask;
  a.num_sms = dev->num_sms;
  a.ctl.err = dev->err;
  a.ctl.timeout_ns = timeout_ns();
  if (fa::launch_fwd(a, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  bool empty = false;
  if (check_common(B, H, H, N, N, d, 1.0f, 0, &empty) != FA_OK || empty) return 0;
  const size_t rows = (size_t)B * H * N;
  return round256(stats_floats(B * H, N) * sizeof(float)) + round256(rows * d * sizeof(float));
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 float scale, int causal, void* workspace, size_t workspace_bytes,
                 struct CUstream_st* stream) {
  return fa_bwd_gqa(q, k, v, o, lse, dO, dq, dk, dv, B, H, H, N, d, scale, causal, workspace,
                    workspace_bytes, stream);
}

fa_status fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dO, void* dq, void* dk, void* dv, int B, int H,
                     int H_kv, int N, int d, float scale, int causal, void* workspace,
                     size_t workspace_bytes, struct CUstream_st* stream) {
  return fa_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, B, H, H_kv, N, N, d, scale, causal, workspace,
                   workspace_bytes, stream);
}

fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, int B, int H, int H_kv, int N_q,
                    int N_k, int d, float scale, int causal, void* workspace,
                    size_t workspace_bytes, struct CUstream_st* stream) {
  return fa_bwd_sparse(q, k, v, o, lse, dO, dq, dk, dv, B, H, H_kv, N_q, N_k, d, scale, causal,
                       nullptr, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_sparse(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                        int H, int H_kv, int N_q, int N_k, int d, float scale, int causal,
                        const unsigned char* block_mask, void* workspace,
                        size_t workspace_bytes, struct CUstream_st* stream) {
  bool empty = false;
  fa_status s = check_common(B, H, H_kv, N_q, N_k, d, scale, causal, &empty);
  if (s != FA_OK) return s;
  if (!empty && block_mask && !mask_fits(N_q, N_k)) return FA_ERR_INVALID_ARG;
  if (empty) {
    // No query rows: dk and dv are sums over nothing, i.e. zero.
    if (B == 0 || H == 0 || N_k == 0) return FA_OK;
    if (!aligned16(dk) || !aligned16(dv)) return FA_ERR_INVALID_ARG;
    DeviceState* dev = nullptr;
    if ((s = current_device(&dev)) != FA_OK) return s;
    const size_t bytes = (size_t)B * H_kv * N_k * d * 2;  // bf16 +0.0 is all zero bits
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(dk, 0, bytes, st) != cudaSuccess || cudaMemsetAsync(dv, 0, bytes, st) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_LAUNCH;
    }
    return FA_OK;
  }
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < fa_bwd_workspace_size(B, H, N_q, d))
    return FA_ERR_INVALID_ARG;
  DeviceState* dev = nullptr;
  if ((s = current_device(&dev)) != FA_OK) return s;
  if (!get_encoder()) return FA_ERR_LAUNCH;
  fa::BwdLaunch a;
  const int BH = B * H, BHkv = B * H_kv;
  if (!encode_bf16_3d(&a.tq, q, BH, N_q, d) || !encode_bf16_3d(&a.tk, k, BHkv, N_k, d) ||
      !encode_bf16_3d(&a.tv, v, BHkv, N_k, d) || !encode_bf16_3d(&a.tdo, dO, BH, N_q, d))
    return FA_ERR_INVALID_ARG;
  a.o = o;
  a.dO = dO;
  a.lse = lse;
  a.stats = static_cast<float*>(workspace);
  a.dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                      round256(stats_floats(BH, N_q) * sizeof(float)));
  if (!encode_f32_3d(&a.tdq, a.dq_acc, BH, N_q, d) || !encode_bf16_3d(&a.tdk, dk, BHkv, N_k, d, 32))
    return FA_ERR_INVALID_ARG;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.BH = BH;
  a.group = H / H_kv;
  a.Nq = N_q;
  a.Nk = N_k;
  a.d = d;
  a.scale = scale;
  a.causal = causal;
  a.bmask = block_mask;
  a.num_sms = dev->num_sms;
  a.ctl.err = dev->err;
  a.ctl.timeout_ns = timeout_ns();
  if (fa::launch_bwd(a, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

unsigned long long fa_device_error_word(struct CUstream_st* stream) {
  DeviceState* dev = nullptr;
  if (current_device(&dev) != FA_OK) return 0;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  unsigned long long w = 0;
  if (cudaMemcpy(&w, dev->err, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return w;
}

fa_status fa_last_device_error(struct CUstream_st* stream) {
  DeviceState* dev = nullptr;
  fa_status s = current_device(&dev);
  if (s != FA_OK) return s;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_DEVICE;
  }
  unsigned long long w = 0;
  if (cudaMemcpy(&w, dev->err, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_DEVICE;
  }
  if (w == 0) return FA_OK;
  const unsigned long long zero = 0;
  if (cudaMemcpy(dev->err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_DEVICE;
  }
  switch (w & 0xFF) {
    case fa::kErrTimeout: return FA_ERR_TIMEOUT;
    default: return FA_ERR_DEVICE;
  }
}

void fa_set_wait_timeout_ns(unsigned long long ns) {
  g_timeout_ns.store(ns, std::memory_order_relaxed);
}

const char* fa_strerror(int status) {
  switch (status) {
    case FA_OK: return "success";
    case FA_ERR_INVALID_ARG: return "invalid argument (pointer, alignment, size, scale, flag or workspace)";
    case FA_ERR_UNSUPPORTED: return "unsupported (head dimension must be 64 or 128; device must be sm_103)";
    case FA_ERR_LAUNCH: return "CUDA runtime call or kernel launch failed";
    case FA_ERR_TIMEOUT: return "a kernel gave up on an internal pipeline wait";
    case FA_ERR_NO_DEVICE: return "no CUDA device is current";
    case FA_ERR_DEVICE: return "asynchronous CUDA error reported by the stream or device";
    default: return "unknown status";
  }
}

const char* fa_version(void) { return "io_aware_exact_10_gb300 0.1.0 (sm_103a)"; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward without a caller-provided workspace.
//
// Some callers cannot hand the library a workspace: a plugin running inside a
// host framework that owns all device memory and gives the plugin none, or a
// latency-critical loop that must never call cudaMalloc (which may
// synchronise the device and takes unbounded time).  For them the backward's
// scratch (D and the fp32 dQ accumulator) lives in one file-scope device array
// that every GPU loading the library holds until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kStaticScratchBytes = 64ull << 20;  // 64 MiB per device
static __device__ __align__(256) unsigned char g_fa_bwd_static_scratch[kStaticScratchBytes];

struct StaticScratch {
  std::once_flag once;
  void* ptr = nullptr;  // device address of g_fa_bwd_static_scratch on this device
  cudaError_t err = cudaSuccess;
};
StaticScratch g_static_scratch[kMaxDevices];

}  // namespace

extern "C" {

fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, float scale, int causal,
                         struct CUstream_st* stream) {
  bool empty = false;
  fa_status s = check_common(B, H, H, N, N, d, scale, causal, &empty);
  if (s != FA_OK || empty) return s;
  // Problems whose D + dQ accumulator exceed the static array are refused.
  if (fa_bwd_workspace_size(B, H, N, d) > kStaticScratchBytes) return FA_ERR_INVALID_ARG;
  DeviceState* dev = nullptr;
  if ((s = current_device(&dev)) != FA_OK) return s;
  int id = -1;
  if (cudaGetDevice(&id) != cudaSuccess || id < 0 || id >= kMaxDevices) {
    cudaGetLastError();
    return FA_ERR_NO_DEVICE;
  }
  // Once per device, with that device current: the host-side name of the
  // array is not a device address, so ask the runtime for the real one.
  StaticScratch& sc = g_static_scratch[id];
  std::call_once(sc.once, [&sc] {
    void* p = nullptr;
    sc.err = cudaGetSymbolAddress(&p, g_fa_bwd_static_scratch);
    if (sc.err == cudaSuccess) sc.ptr = p;
  });
  if (sc.err != cudaSuccess || !sc.ptr) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  // The preprocess kernel of fa_bwd rewrites D and zeroes the dQ accumulator
  // on every call, so nothing left in the array by an earlier call leaks in.
  return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, sc.ptr,
                kStaticScratchBytes, stream);
}

}  // extern "C"
