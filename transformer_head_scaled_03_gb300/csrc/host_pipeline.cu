// host_pipeline.cu -- scaled dot-product attention from host buffers.
//
// The call copies Q, K, V (and the key lengths) in, attends and copies O
// out.  The problem is cut into about sixteen chunks of (b, h) heads.  Each
// chunk's inputs go over on a copy-in stream, its attention runs on the
// caller's stream as soon as they have landed, and its output returns on a
// copy-out stream as soon as it is written.  So the transfers of one chunk
// overlap the attention of others, and only the first chunk's copy-in and
// the last chunk's copy-out stay exposed.  Chunks alternate between the
// caller's stream and a second compute stream, so one chunk's grid can
// start while the previous one drains.  Attention of every head is
// independent ("How Transformers Work" (worksonmygpu.com), "Multi-head
// attention"), so chunking changes no arithmetic.
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "internal.h"

namespace mha {
namespace {

constexpr int kMaxDev = 16;
constexpr int kTargetChunks = 16;  // measured best of 4, 8, 16, 32 on the long-context shape

// Per device: the two copy streams and a pool of events, created on first
// use and kept; `lock` serialises calls that enqueue on one device.
struct HostCtx {
  std::mutex lock;
  cudaStream_t h2d = nullptr;
  cudaStream_t d2h = nullptr;
  cudaStream_t comp = nullptr;
  std::vector<cudaEvent_t> events;
};
HostCtx g_host[kMaxDev];

bool ensure_events(HostCtx& c, size_t n) {
  while (c.events.size() < n) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
    c.events.push_back(e);
  }
  return true;
}

size_t round256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }
size_t elem_bytes(int t) { return t == MHA_BF16 ? 2 : 4; }

// Device workspace: Q, K, V, O and the key lengths, each 256-byte aligned.
struct Layout {
  size_t q, k, v, o, len, total;
};

Layout layout_of(int B, int H, int Lq, int Lk, int d, int in_dt, int out_dt) {
  const size_t qn = static_cast<size_t>(B) * H * Lq * d;
  const size_t kn = static_cast<size_t>(B) * H * Lk * d;
  Layout L{};
  L.q = 0;
  L.k = L.q + round256(qn * elem_bytes(in_dt));
  L.v = L.k + round256(kn * elem_bytes(in_dt));
  L.o = L.v + round256(kn * elem_bytes(in_dt));
  L.len = L.o + round256(qn * elem_bytes(out_dt));
  L.total = L.len + round256(static_cast<size_t>(B) * sizeof(int32_t));
  return L;
}

}  // namespace
}  // namespace mha

using namespace mha;

extern "C" {

size_t sdpa_forward_host_workspace_bytes(int B, int H, int Lq, int Lk, int d, mha_dtype in_dtype,
                                         mha_dtype out_dtype) {
  if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || d < 1) return 0;
  if ((in_dtype != MHA_BF16 && in_dtype != MHA_F32) ||
      (out_dtype != MHA_BF16 && out_dtype != MHA_F32))
    return 0;
  return layout_of(B, H, Lq, Lk, d, in_dtype, out_dtype).total;
}

mha_status sdpa_forward_host(const void* Qh, const void* Kh, const void* Vh, void* Oh, int B,
                             int H, int Lq, int Lk, int d, float scale, int mask_kind,
                             const int32_t* key_lengths_h, mha_dtype in_dtype,
                             mha_dtype out_dtype, void* workspace, size_t workspace_bytes,
                             mha_stream stream) {
  const mha_status st = validate_sdpa(Qh, Kh, Vh, Oh, B, H, Lq, Lk, d, scale, mask_kind,
                                      key_lengths_h, in_dtype, out_dtype);
  if (st != MHA_OK) return st;
  if (static_cast<long long>(B) * H * Lq == 0) return MHA_OK;
  const Layout L = layout_of(B, H, Lq, Lk, d, in_dtype, out_dtype);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < L.total)
    return MHA_ERR_INVALID_ARG;
  DeviceCtl ctl;
  if (!device_ctl(&ctl)) return MHA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return MHA_ERR_CUDA;
  HostCtx& c = g_host[dev];
  std::lock_guard<std::mutex> guard(c.lock);
  if (!c.h2d && cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking) != cudaSuccess) {
    c.h2d = nullptr;
    return MHA_ERR_CUDA;
  }
  if (!c.d2h && cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking) != cudaSuccess) {
    c.d2h = nullptr;
    return MHA_ERR_CUDA;
  }
  if (!c.comp && cudaStreamCreateWithFlags(&c.comp, cudaStreamNonBlocking) != cudaSuccess) {
    c.comp = nullptr;
    return MHA_ERR_CUDA;
  }

  // chunks: whole batch items when there are enough of them, else a run of
  // heads of one item; either is one contiguous slice of [B, H, L, d]
  const int nb = B >= kTargetChunks ? (B + kTargetChunks - 1) / kTargetChunks : 1;
  const int hg = B >= kTargetChunks
                     ? H
                     : std::min(H, std::max(1, (B * H + kTargetChunks - 1) / kTargetChunks));
  const int n_chunks = ((B + nb - 1) / nb) * ((H + hg - 1) / hg);
  if (!ensure_events(c, 2 * static_cast<size_t>(n_chunks) + 2)) return MHA_ERR_CUDA;

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t comp[2] = {cs, c.comp};
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* Qd = ws + L.q;
  uint8_t* Kd = ws + L.k;
  uint8_t* Vd = ws + L.v;
  uint8_t* Od = ws + L.o;
  int32_t* lend = key_lengths_h ? reinterpret_cast<int32_t*>(ws + L.len) : nullptr;
  const size_t ies = elem_bytes(in_dtype), oes = elem_bytes(out_dtype);
  const float sc = scale == 0.f ? static_cast<float>(1.0 / sqrt(static_cast<double>(d))) : scale;

  cudaError_t e = cudaSuccess;
  auto ok = [&](cudaError_t r) {
    if (e == cudaSuccess) e = r;
    return e == cudaSuccess;
  };
  // after everything already queued on the caller's stream (a previous call
  // may still be reading this workspace)
  cudaEvent_t start = c.events[0], done = c.events[1];
  if (!ok(cudaEventRecord(start, cs)) || !ok(cudaStreamWaitEvent(c.h2d, start, 0)) ||
      !ok(cudaStreamWaitEvent(c.d2h, start, 0)) || !ok(cudaStreamWaitEvent(c.comp, start, 0)))
    return MHA_ERR_CUDA;
  if (lend && !ok(cudaMemcpyAsync(lend, key_lengths_h, static_cast<size_t>(B) * sizeof(int32_t),
                                  cudaMemcpyHostToDevice, c.h2d)))
    return MHA_ERR_CUDA;

  int ci = 0;
  for (int b0 = 0; b0 < B; b0 += nb) {
    const int nbc = std::min(nb, B - b0);
    for (int h0 = 0; h0 < H; h0 += hg, ++ci) {
      const int hc = std::min(hg, H - h0);
      const size_t head0 = static_cast<size_t>(b0) * H + h0;
      const size_t heads = static_cast<size_t>(nbc) * hc;
      const size_t qo = head0 * Lq * d, qn = heads * Lq * d;
      const size_t ko = head0 * Lk * d, kn = heads * Lk * d;
      cudaEvent_t in = c.events[2 + 2 * ci], out = c.events[3 + 2 * ci];
      ok(cudaMemcpyAsync(Qd + qo * ies, static_cast<const uint8_t*>(Qh) + qo * ies, qn * ies,
                         cudaMemcpyHostToDevice, c.h2d));
      ok(cudaMemcpyAsync(Kd + ko * ies, static_cast<const uint8_t*>(Kh) + ko * ies, kn * ies,
                         cudaMemcpyHostToDevice, c.h2d));
      ok(cudaMemcpyAsync(Vd + ko * ies, static_cast<const uint8_t*>(Vh) + ko * ies, kn * ies,
                         cudaMemcpyHostToDevice, c.h2d));
      cudaStream_t ks = comp[ci & 1];
      ok(cudaEventRecord(in, c.h2d));
      ok(cudaStreamWaitEvent(ks, in, 0));
      if (e != cudaSuccess) return MHA_ERR_CUDA;
      SdpaArgs a{Qd + qo * ies, Kd + ko * ies, Vd + ko * ies, Od + qo * oes, nbc, hc, Lq, Lk, d,
                 sc, mask_kind, lend ? lend + b0 : nullptr, in_dtype, out_dtype, false, ks};
      if (!ok(in_dtype == MHA_BF16 ? launch_sdpa_bf16(a, ctl) : launch_sdpa_f32(a, ctl)))
        return MHA_ERR_CUDA;
      ok(cudaEventRecord(out, ks));
      ok(cudaStreamWaitEvent(c.d2h, out, 0));
      ok(cudaMemcpyAsync(static_cast<uint8_t*>(Oh) + qo * oes, Od + qo * oes, qn * oes,
                         cudaMemcpyDeviceToHost, c.d2h));
      if (e != cudaSuccess) return MHA_ERR_CUDA;
    }
  }
  // the caller's stream covers the whole call, copies out included
  if (!ok(cudaEventRecord(done, c.d2h)) || !ok(cudaStreamWaitEvent(cs, done, 0)))
    return MHA_ERR_CUDA;
  return MHA_OK;
}

}  // extern "C"
