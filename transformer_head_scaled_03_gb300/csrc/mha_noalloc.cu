// mha_noalloc.cu -- mha_forward_noalloc: the multi-head attention layer
// forward for callers that cannot allocate device memory.
//
// mha_forward keeps its intermediate tensors (projected Q, K, V and the
// concatenated-heads context) in workspace that mha_create obtains with
// cudaMalloc.  Some callers cannot do that: a host program that hands all
// device memory to its own pool and forbids other allocations, a plugin
// whose execution step is not allowed to allocate, or a latency-critical
// loop that cannot afford cudaMalloc's implicit device synchronisation.
// This entry point runs the same kernels with the intermediates placed in
// one fixed-size device array declared below, so it allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU on which this
// library is loaded holds MHA_NOALLOC_SCRATCH_BYTES of it until the process
// exits.  All calls on a device share it and each call leaves its own
// intermediates behind; nothing in it needs to start at zero, because every
// call writes each intermediate element before reading it.  Two calls whose
// executions overlap on the GPU (different streams, no ordering between
// them) race on the array.
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"

namespace mha {
namespace {

constexpr size_t kScratchBytes = MHA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The intermediates' storage.  In host code this name is only a host-side
// stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress, once per device.
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// The current device's address of g_noalloc_scratch, resolved on the first
// call made with that device current.
bool scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return false;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return true;
}

size_t round256(size_t n) { return (n + 255u) & ~static_cast<size_t>(255u); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every launch step reports through this one mapping.  The entry point
// allocates nothing, so any CUDA failure of a step -- whatever its code --
// is reported as MHA_ERR_CUDA, the status the header lists.
mha_status step_status(cudaError_t e) { return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA; }

}  // namespace
}  // namespace mha

using namespace mha;

extern "C" mha_status mha_forward_noalloc(int d_model, mha_dtype dtype, const void* x_q,
                                          const void* x_kv, const void* Wq, const void* Wk,
                                          const void* Wv, const void* Wo, int B, int Lq, int Lk,
                                          int heads, int mask_kind, const int32_t* key_lengths,
                                          void* out, mha_stream stream) {
  const int D = d_model;
  if (D < 1 || (dtype != MHA_BF16 && dtype != MHA_F32)) return MHA_ERR_INVALID_ARG;
  if (heads < 1 || D % heads != 0) return MHA_ERR_INVALID_ARG;
  if (B < 0 || Lq < 0 || Lk < 1) return MHA_ERR_INVALID_ARG;
  const int d = D / heads;
  const bool empty = static_cast<long long>(B) * Lq == 0;
  if (!empty) {
    const void* ptrs[7] = {x_q, x_kv, Wq, Wk, Wv, Wo, out};
    for (const void* p : ptrs)
      if (!p || !aligned16(p)) return MHA_ERR_INVALID_ARG;
    if (out == x_q || out == x_kv) return MHA_ERR_INVALID_ARG;
  }
  // the intermediates must fit the fixed array
  const size_t es = dtype == MHA_BF16 ? 2 : 4;
  const size_t nq = round256(static_cast<size_t>(B) * Lq * D * es);
  const size_t nk = round256(static_cast<size_t>(B) * Lk * D * es);
  if (2 * nq + 2 * nk > kScratchBytes) return MHA_ERR_INVALID_ARG;
  // the attention step's own checks (placeholder non-null pointers: the real
  // ones are inside the array and 256-byte aligned)
  const void* aligned_stub = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
  mha_status st = validate_sdpa(aligned_stub, aligned_stub, aligned_stub, aligned_stub, B, heads,
                                Lq, Lk, d, 0.f, mask_kind, key_lengths, dtype, dtype);
  if (st != MHA_OK) return st;
  if (dtype == MHA_BF16 && D % 64 != 0) return MHA_ERR_UNSUPPORTED;
  if (empty) return MHA_OK;

  void* base = nullptr;
  if (!scratch_address(&base)) return MHA_ERR_CUDA;
  DeviceCtl ctl;
  if (!device_ctl(&ctl)) return MHA_ERR_CUDA;
  unsigned char* s = static_cast<unsigned char*>(base);
  void* q = s;
  void* k = s + nq;
  void* v = s + nq + nk;
  void* ctx = s + nq + 2 * nk;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  auto gemm = dtype == MHA_BF16 ? launch_gemm_bf16 : launch_gemm_f32;

  // projections, head split in the store layout
  cudaError_t e;
  if (x_kv == x_q && Lk == Lq) {
    GemmArgs g{};
    g.prob[0] = {x_q, Wq, q, GemmStore::kHeadSplit, Lq, d};
    g.prob[1] = {x_q, Wk, k, GemmStore::kHeadSplit, Lk, d};
    g.prob[2] = {x_q, Wv, v, GemmStore::kHeadSplit, Lk, d};
    g.count = 3;
    g.M = B * Lq;
    g.N = D;
    g.K = D;
    g.dtype = dtype;
    g.stream = cs;
    e = gemm(g, ctl);
  } else {
    GemmArgs g{};
    g.prob[0] = {x_q, Wq, q, GemmStore::kHeadSplit, Lq, d};
    g.count = 1;
    g.M = B * Lq;
    g.N = D;
    g.K = D;
    g.dtype = dtype;
    g.stream = cs;
    e = gemm(g, ctl);
    if (e == cudaSuccess) {
      GemmArgs g2{};
      g2.prob[0] = {x_kv, Wk, k, GemmStore::kHeadSplit, Lk, d};
      g2.prob[1] = {x_kv, Wv, v, GemmStore::kHeadSplit, Lk, d};
      g2.count = 2;
      g2.M = B * Lk;
      g2.N = D;
      g2.K = D;
      g2.dtype = dtype;
      g2.stream = cs;
      e = gemm(g2, ctl);
    }
  }
  if (e != cudaSuccess) return step_status(e);
  // attention per head, stored as the concatenated heads
  SdpaArgs a{q, k, v, ctx, B, heads, Lq, Lk, d,
             static_cast<float>(1.0 / sqrt(static_cast<double>(d))), mask_kind, key_lengths,
             dtype, dtype, true, cs};
  e = dtype == MHA_BF16 ? launch_sdpa_bf16(a, ctl) : launch_sdpa_f32(a, ctl);
  if (e != cudaSuccess) return step_status(e);
  // output projection
  GemmArgs go{};
  go.prob[0] = {ctx, Wo, out, GemmStore::kRowMajor, Lq, d};
  go.count = 1;
  go.M = B * Lq;
  go.N = D;
  go.K = D;
  go.dtype = dtype;
  go.stream = cs;
  return step_status(gemm(go, ctl));
}
