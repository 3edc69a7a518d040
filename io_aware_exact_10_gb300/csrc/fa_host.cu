// fa_host.cu -- entry points for inputs and outputs in host memory: the
// heads are cut into groups, and each group's copies to the device, its
// kernels and its copies back run on three streams, so the copies of one
// group overlap the kernels and copies of its neighbours.  The kernels are
// the ones fa_fwd_sparse / fa_bwd_sparse launch (with a NULL mask, those of
// fa_fwd_ex / fa_bwd_ex); nothing here computes.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 64;
constexpr int kDefaultChunks = 8;

// Per device: the two copy streams and the events that order them against
// the caller's stream.  Created on first use and kept for the process; one
// call at a time enqueues on them (the mutex), so calls from several host
// threads are ordered by the order in which they take it.
struct Pipe {
  std::once_flag once;
  std::mutex mu;
  cudaError_t err = cudaSuccess;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t in_ev[kMaxChunks], fwd_ev[kMaxChunks], bwd_ev[kMaxChunks];
};
Pipe g_pipe[kMaxDevices];

fa_status device_pipe(Pipe** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return FA_ERR_NO_DEVICE;
  }
  if (dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  Pipe& p = g_pipe[dev];
  std::call_once(p.once, [&p] {
    auto ev = [&p](cudaEvent_t* e) {
      if (p.err == cudaSuccess) p.err = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
    };
    p.err = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking);
    if (p.err == cudaSuccess) p.err = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking);
    ev(&p.start);
    ev(&p.done);
    for (int c = 0; c < kMaxChunks; ++c) {
      ev(&p.in_ev[c]);
      ev(&p.fwd_ev[c]);
      ev(&p.bwd_ev[c]);
    }
  });
  if (p.err != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  *out = &p;
  return FA_OK;
}

size_t r256(size_t x) { return (x + 255) & ~(size_t)255; }

// Sizes shared by the entry points (the limits of fa_fwd_ex, restated so
// that a bad argument is refused before anything is enqueued).
bool sizes_ok(int B, int H, int H_kv, int N_q, int N_k, int d) {
  if (B < 0 || H < 0 || N_q < 0 || N_k < 0 || N_q > (1 << 30) || N_k > (1 << 30)) return false;
  if (d != 64 && d != 128) return false;
  if (B > 0 && H > 0 && (H_kv < 1 || H_kv > H || H % H_kv != 0)) return false;
  return true;
}
bool args_ok(int B, int H, int H_kv, int N_q, int N_k, int d, float scale, int causal,
             const unsigned char* block_mask) {
  if (!sizes_ok(B, H, H_kv, N_q, N_k, d)) return false;
  // a block mask has at most 4096 blocks per side (as for fa_fwd_sparse)
  if (block_mask && ((N_q + 127) / 128 > 4096 || (N_k + 127) / 128 > 4096)) return false;
  if (causal != 0 && causal != 1) return false;
  if (!(std::isfinite(scale) && scale > 0.f)) return false;
  if (B > 0 && H > 0 && N_q > 0 && (N_k == 0 || (causal && N_k < N_q))) return false;
  return true;
}

// Layout of the device staging area: every region 256-byte aligned.
struct Layout {
  size_t q, k, v, dO, o, lse, dq, dk, dv, ws, total;
};
Layout layout(int B, int H, int H_kv, int N_q, int N_k, int d, bool backward, int chunk_kv) {
  const size_t BH = (size_t)B * H, BHkv = (size_t)B * H_kv;
  const size_t qb = BH * N_q * d * 2, kb = BHkv * N_k * d * 2, lb = BH * N_q * 4;
  Layout L{};
  size_t at = 0;
  auto take = [&at](size_t bytes) {
    const size_t off = at;
    at += r256(bytes);
    return off;
  };
  L.q = take(qb);
  L.k = take(kb);
  L.v = take(kb);
  L.o = take(qb);
  // each group's lse starts 16-byte aligned (groups of odd row counts)
  L.lse = take(lb + 16 * (size_t)kMaxChunks);
  if (backward) {
    L.dO = take(qb);
    L.dq = take(qb);
    L.dk = take(kb);
    L.dv = take(kb);
    // one workspace reused by every group (their kernels run in stream order)
    const int G = H_kv > 0 ? H / H_kv : 1;
    L.ws = take(fa_bwd_workspace_size(1, chunk_kv * G, N_q, d));
  }
  L.total = at;
  return L;
}

int pick_chunks(int chunks, long long n_kv) {
  long long c = chunks > 0 ? chunks : kDefaultChunks;
  if (c > kMaxChunks) c = kMaxChunks;
  if (c > n_kv) c = n_kv;
  return (int)(c < 1 ? 1 : c);
}

// Key/value heads of group c of n: [lo, hi), as even as possible.
void group_range(long long n_kv, int n, int c, long long* lo, long long* hi) {
  *lo = n_kv * c / n;
  *hi = n_kv * (c + 1) / n;
}

fa_status run(const void* q, const void* k, const void* v, const void* dO, void* o, float* lse,
              void* dq, void* dk, void* dv, int B, int H, int H_kv, int N_q, int N_k, int d,
              float scale, int causal, const unsigned char* block_mask, void* dev,
              size_t dev_bytes, int chunks, cudaStream_t stream, bool backward) {
  if (!args_ok(B, H, H_kv, N_q, N_k, d, scale, causal, block_mask)) return FA_ERR_INVALID_ARG;
  if (B == 0 || H == 0) return FA_OK;
  const long long n_kv = (long long)B * H_kv;
  const int G = H / H_kv;
  const int n = pick_chunks(chunks, n_kv);
  const long long chunk_kv = (n_kv + n - 1) / n;
  if (chunk_kv * G > 0x7FFFFFFFLL) return FA_ERR_INVALID_ARG;
  const Layout L = layout(B, H, H_kv, N_q, N_k, d, backward, (int)chunk_kv);
  const bool need_q = N_q > 0, need_k = N_k > 0;
  if (need_q && (!q || !o || !lse || (backward && (!dO || !dq)))) return FA_ERR_INVALID_ARG;
  if (need_k && (!k || !v || (backward && (!dk || !dv)))) return FA_ERR_INVALID_ARG;
  if (!dev || (reinterpret_cast<uintptr_t>(dev) & 255u) != 0 || dev_bytes < L.total)
    return FA_ERR_INVALID_ARG;
  Pipe* P = nullptr;
  if (const fa_status s = device_pipe(&P); s != FA_OK) return s;

  char* base = static_cast<char*>(dev);
  const size_t qrow = (size_t)N_q * d * 2, krow = (size_t)N_k * d * 2;  // bytes per head
  std::lock_guard<std::mutex> lock(P->mu);
  bool ok = true;
  auto ck = [&ok](cudaError_t e) {
    if (e != cudaSuccess) ok = false;
  };
  auto h2d = [&](size_t dst_off, const void* src, size_t off, size_t bytes) {
    if (ok && bytes)
      ck(cudaMemcpyAsync(base + dst_off + off, static_cast<const char*>(src) + off, bytes,
                         cudaMemcpyHostToDevice, P->in));
  };
  auto d2h = [&](void* dst, size_t src_off, size_t off, size_t bytes) {
    if (ok && bytes)
      ck(cudaMemcpyAsync(static_cast<char*>(dst) + off, base + src_off + off, bytes,
                         cudaMemcpyDeviceToHost, P->out));
  };
  // Nothing is overwritten on the device before the caller's earlier work
  // on `stream` (which may still read the staging area) has finished.
  ck(cudaEventRecord(P->start, stream));
  if (ok) ck(cudaStreamWaitEvent(P->in, P->start, 0));
  if (ok) ck(cudaStreamWaitEvent(P->out, P->start, 0));
  fa_status st = FA_OK;
  size_t ldev = L.lse;  // device offset of the group's lse
  for (int c = 0; c < n && ok && st == FA_OK; ++c) {
    long long lo, hi;
    group_range(n_kv, n, c, &lo, &hi);
    const int nk = (int)(hi - lo), nh = nk * G;
    const size_t qo = (size_t)lo * G * qrow, qn = (size_t)nh * qrow;
    const size_t ko = (size_t)lo * krow, kn = (size_t)nk * krow;
    const size_t lo4 = (size_t)lo * G * N_q * 4, ln4 = (size_t)nh * N_q * 4;
    // inputs of group c
    h2d(L.q, q, qo, qn);
    h2d(L.k, k, ko, kn);
    h2d(L.v, v, ko, kn);
    if (backward) h2d(L.dO, dO, qo, qn);
    if (ok) ck(cudaEventRecord(P->in_ev[c], P->in));
    if (ok) ck(cudaStreamWaitEvent(stream, P->in_ev[c], 0));
    if (!ok) break;
    // its kernels, on the caller's stream (the block mask, shared by every
    // head, applies to each group as it is; NULL is the dense computation)
    st = fa_fwd_sparse(base + L.q + qo, base + L.k + ko, base + L.v + ko, base + L.o + qo,
                       reinterpret_cast<float*>(base + ldev), 1, nh, nk, N_q, N_k, d, scale,
                       causal, block_mask, stream);
    if (st != FA_OK) break;
    ck(cudaEventRecord(P->fwd_ev[c], stream));
    if (backward && ok) {
      st = fa_bwd_sparse(base + L.q + qo, base + L.k + ko, base + L.v + ko, base + L.o + qo,
                         reinterpret_cast<const float*>(base + ldev), base + L.dO + qo,
                         base + L.dq + qo, base + L.dk + ko, base + L.dv + ko, 1, nh, nk, N_q,
                         N_k, d, scale, causal, block_mask, base + L.ws,
                         fa_bwd_workspace_size(1, nh, N_q, d), stream);
      if (st != FA_OK) break;
      ck(cudaEventRecord(P->bwd_ev[c], stream));
    }
    // its outputs: o and lse once the forward is done, the gradients after
    // the backward
    if (ok) ck(cudaStreamWaitEvent(P->out, P->fwd_ev[c], 0));
    d2h(o, L.o, qo, qn);
    if (ok && ln4)
      ck(cudaMemcpyAsync(reinterpret_cast<char*>(lse) + lo4, base + ldev, ln4, cudaMemcpyDeviceToHost,
                         P->out));
    ldev += (ln4 + 15) & ~(size_t)15;
    if (backward) {
      if (ok) ck(cudaStreamWaitEvent(P->out, P->bwd_ev[c], 0));
      d2h(dq, L.dq, qo, qn);
      d2h(dk, L.dk, ko, kn);
      d2h(dv, L.dv, ko, kn);
    }
  }
  // The caller's stream passes this call only when both copy streams have
  // drained: synchronising it makes the host outputs readable.  Joined even
  // after a failure part way, so that no copy enqueued above can still touch
  // the staging area when later work on `stream` writes it.  (A wait takes
  // the event as last recorded, so one event serves both joins.)
  const bool joined = cudaEventRecord(P->done, P->out) == cudaSuccess &&
                      cudaStreamWaitEvent(stream, P->done, 0) == cudaSuccess &&
                      cudaEventRecord(P->done, P->in) == cudaSuccess &&
                      cudaStreamWaitEvent(stream, P->done, 0) == cudaSuccess;
  if (!ok || !joined) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return st;
}

}  // namespace

extern "C" {

size_t fa_fwd_host_device_bytes(int B, int H, int H_kv, int N_q, int N_k, int d) {
  if (!sizes_ok(B, H, H_kv, N_q, N_k, d) || B == 0 || H == 0) return 0;
  return layout(B, H, H_kv, N_q, N_k, d, false, 0).total;
}

size_t fa_fwd_bwd_host_device_bytes(int B, int H, int H_kv, int N_q, int N_k, int d,
                                    int chunks) {
  if (!sizes_ok(B, H, H_kv, N_q, N_k, d) || B == 0 || H == 0) return 0;
  const long long n_kv = (long long)B * H_kv;
  const int n = pick_chunks(chunks, n_kv);
  const long long chunk_kv = (n_kv + n - 1) / n;
  if (chunk_kv * (H / H_kv) > 0x7FFFFFFFLL) return 0;
  return layout(B, H, H_kv, N_q, N_k, d, true, (int)chunk_kv).total;
}

fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int H_kv, int N_q, int N_k, int d, float scale, int causal,
                      const unsigned char* block_mask, void* dev, size_t dev_bytes, int chunks,
                      struct CUstream_st* stream) {
  return run(q, k, v, nullptr, o, lse, nullptr, nullptr, nullptr, B, H, H_kv, N_q, N_k, d, scale,
             causal, block_mask, dev, dev_bytes, chunks, reinterpret_cast<cudaStream_t>(stream),
             false);
}

fa_status fa_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dO, void* o,
                          float* lse, void* dq, void* dk, void* dv, int B, int H, int H_kv,
                          int N_q, int N_k, int d, float scale, int causal,
                          const unsigned char* block_mask, void* dev, size_t dev_bytes,
                          int chunks, struct CUstream_st* stream) {
  return run(q, k, v, dO, o, lse, dq, dk, dv, B, H, H_kv, N_q, N_k, d, scale, causal, block_mask,
             dev, dev_bytes, chunks, reinterpret_cast<cudaStream_t>(stream), true);
}

}  // extern "C"
