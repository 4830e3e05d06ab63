// mha_api.cu -- the C ABI declared in include/mha.h: argument validation,
// TMA descriptor encoding, workspace ownership and kernel launch order.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <new>

#include "internal.h"
#include "ptx.cuh"

namespace mha {

// Per-device error word: kernels OR error bits into it, mha_check reads and
// clears it.
__device__ unsigned g_device_error;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_wait_limit_ms = 2000;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
bool g_encode_tried = false;

bool get_device_ctl(DeviceCtl* ctl) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess || !p) return false;
    g_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  ctl->err = g_err_ptr[dev];
  ctl->limit_ns = static_cast<uint64_t>(g_wait_limit_ms) * 1000000ull;
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elem_size(mha_dtype t) { return t == MHA_BF16 ? 2 : 4; }

bool valid_dtype(int t) { return t == MHA_F32 || t == MHA_BF16; }

mha_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return MHA_OK;
  if (e == cudaErrorMemoryAllocation) return MHA_ERR_OOM;
  return MHA_ERR_CUDA;
}

}  // namespace

bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swizzle) {
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode_tried) {
      g_encode_tried = true;
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) == cudaSuccess &&
          q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  if (!g_encode) return false;
  cuuint64_t gdim[5], gstr[4];
  cuuint32_t bdim[5], estr[5];
  for (uint32_t i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estr[i] = 1;
    if (i + 1 < rank) gstr[i] = strides_bytes[i];
  }
  return g_encode(map, dtype, rank, base, gdim, gstr, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// Self-test of the bounded pipeline wait: one warp waits on an mbarrier that
// nothing ever arrives on, with the same helper the attention and GEMM
// kernels use.  The wait must give up after the limit, raise the abort flag
// and set the timeout bit in the device error word, and the kernel returns.
__global__ void wait_selftest_kernel(unsigned* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl ctl{&abort_flag, err, limit_ns};
  mbar_wait_warp(smem_u32(&bar), 0, ctl);
}

}  // namespace

}  // namespace mha

using namespace mha;

struct mha_ctx {
  int device;
  int d_model;
  mha_dtype dtype;
  int max_batch, max_lq, max_lk;
  void* q;    // [B, H, Lq, d]
  void* k;    // [B, H, Lk, d]
  void* v;    // [B, H, Lk, d]
  void* ctx;  // [B, Lq, D]
};

namespace {

// Shared validation of a scaled dot-product attention request.
mha_status check_sdpa(const void* Q, const void* K, const void* V, const void* O, int B, int H,
                      int Lq, int Lk, int d, float scale, int mask_kind,
                      const int32_t* key_lengths, int in_dtype, int out_dtype) {
  if (B < 0 || H < 0 || Lq < 0 || Lk < 1 || d < 1) return MHA_ERR_INVALID_ARG;
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return MHA_ERR_INVALID_ARG;
  if (!(scale >= 0.f) || isinf(scale)) return MHA_ERR_INVALID_ARG;
  if (mask_kind < 0 || mask_kind > (MHA_MASK_CAUSAL | MHA_MASK_KEY_PADDING))
    return MHA_ERR_INVALID_ARG;
  if ((mask_kind & MHA_MASK_CAUSAL) && Lq != Lk) return MHA_ERR_INVALID_ARG;
  if ((mask_kind & MHA_MASK_KEY_PADDING) && !key_lengths) return MHA_ERR_INVALID_ARG;
  if (key_lengths && (reinterpret_cast<uintptr_t>(key_lengths) & 3u)) return MHA_ERR_INVALID_ARG;
  const bool empty = (static_cast<long long>(B) * H * Lq) == 0;
  if (!empty) {
    if (!Q || !K || !V || !O) return MHA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O))
      return MHA_ERR_INVALID_ARG;
  }
  if (in_dtype == MHA_BF16) {
    if (d != 64 && d != 128) return MHA_ERR_UNSUPPORTED;
  } else {
    if (d > 128 || out_dtype != MHA_F32) return MHA_ERR_UNSUPPORTED;
  }
  // element counts stay far inside the kernels' 64-bit index range; the grid
  // (query blocks x B x H) must fit a 31-bit blockIdx.x
  if (static_cast<long long>((Lq + 127) / 128) * B * H > 0x7fffffffLL) return MHA_ERR_UNSUPPORTED;
  return MHA_OK;
}

}  // namespace

extern "C" {

const char* mha_status_string(mha_status s) {
  switch (s) {
    case MHA_OK: return "MHA_OK";
    case MHA_ERR_INVALID_ARG: return "MHA_ERR_INVALID_ARG";
    case MHA_ERR_UNSUPPORTED: return "MHA_ERR_UNSUPPORTED";
    case MHA_ERR_CUDA: return "MHA_ERR_CUDA";
    case MHA_ERR_OOM: return "MHA_ERR_OOM";
    case MHA_ERR_TIMEOUT: return "MHA_ERR_TIMEOUT";
    case MHA_ERR_DEVICE: return "MHA_ERR_DEVICE";
  }
  return "MHA_ERR_UNKNOWN";
}

int mha_set_wait_limit_ms(int ms) {
  std::lock_guard<std::mutex> lock(g_mutex);
  const int prev = g_wait_limit_ms;
  if (ms > 0) g_wait_limit_ms = ms;
  return prev;
}

mha_status sdpa_forward(const void* Q, const void* K, const void* V, void* O, int B, int H, int Lq,
                        int Lk, int d, float scale, int mask_kind, const int32_t* key_lengths,
                        mha_dtype in_dtype, mha_dtype out_dtype, mha_stream stream) {
  const mha_status st = check_sdpa(Q, K, V, O, B, H, Lq, Lk, d, scale, mask_kind, key_lengths,
                                   in_dtype, out_dtype);
  if (st != MHA_OK) return st;
  if (static_cast<long long>(B) * H * Lq == 0) return MHA_OK;
  DeviceCtl ctl;
  if (!get_device_ctl(&ctl)) return MHA_ERR_CUDA;
  SdpaArgs a{Q, K, V, O, B, H, Lq, Lk, d,
             scale == 0.f ? static_cast<float>(1.0 / sqrt(static_cast<double>(d))) : scale,
             mask_kind, key_lengths, in_dtype, out_dtype, false,
             reinterpret_cast<cudaStream_t>(stream)};
  const cudaError_t e = in_dtype == MHA_BF16 ? launch_sdpa_bf16(a, ctl) : launch_sdpa_f32(a, ctl);
  return from_cuda(e);
}

mha_status sdpa_forward_float_mask(const void* Q, const void* K, const void* V, void* O, int B,
                                   int H, int Lq, int Lk, int d, float scale, int mask_kind,
                                   const int32_t* key_lengths, const float* add_mask,
                                   int64_t mask_stride_b, int64_t mask_stride_h,
                                   mha_dtype in_dtype, mha_dtype out_dtype, mha_stream stream) {
  const mha_status st = check_sdpa(Q, K, V, O, B, H, Lq, Lk, d, scale, mask_kind, key_lengths,
                                   in_dtype, out_dtype);
  if (st != MHA_OK) return st;
  if (mask_stride_b < 0 || mask_stride_h < 0) return MHA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * Lq == 0) return MHA_OK;
  if (!add_mask || (reinterpret_cast<uintptr_t>(add_mask) & 3u)) return MHA_ERR_INVALID_ARG;
  DeviceCtl ctl;
  if (!get_device_ctl(&ctl)) return MHA_ERR_CUDA;
  SdpaArgs a{Q, K, V, O, B, H, Lq, Lk, d,
             scale == 0.f ? static_cast<float>(1.0 / sqrt(static_cast<double>(d))) : scale,
             mask_kind, key_lengths, in_dtype, out_dtype, false,
             reinterpret_cast<cudaStream_t>(stream), add_mask, mask_stride_b, mask_stride_h};
  const cudaError_t e = in_dtype == MHA_BF16 ? launch_sdpa_bf16(a, ctl) : launch_sdpa_f32(a, ctl);
  return from_cuda(e);
}

mha_status mha_create(mha_handle* out, int d_model, mha_dtype dtype, int max_batch, int max_lq,
                      int max_lk) {
  if (!out) return MHA_ERR_INVALID_ARG;
  *out = nullptr;
  if (d_model < 1 || !valid_dtype(dtype) || max_batch < 1 || max_lq < 1 || max_lk < 1)
    return MHA_ERR_INVALID_ARG;
  mha_ctx* h = new (std::nothrow) mha_ctx();
  if (!h) return MHA_ERR_OOM;
  if (cudaGetDevice(&h->device) != cudaSuccess) {
    delete h;
    return MHA_ERR_CUDA;
  }
  h->d_model = d_model;
  h->dtype = dtype;
  h->max_batch = max_batch;
  h->max_lq = max_lq;
  h->max_lk = max_lk;
  const size_t es = elem_size(dtype);
  const size_t nq = static_cast<size_t>(max_batch) * max_lq * d_model * es;
  const size_t nk = static_cast<size_t>(max_batch) * max_lk * d_model * es;
  cudaError_t e = cudaMalloc(&h->q, nq);
  if (e == cudaSuccess) e = cudaMalloc(&h->k, nk);
  if (e == cudaSuccess) e = cudaMalloc(&h->v, nk);
  if (e == cudaSuccess) e = cudaMalloc(&h->ctx, nq);
  if (e != cudaSuccess) {
    cudaFree(h->q);
    cudaFree(h->k);
    cudaFree(h->v);
    cudaFree(h->ctx);
    delete h;
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? MHA_ERR_OOM : MHA_ERR_CUDA;
  }
  *out = h;
  return MHA_OK;
}

mha_status mha_forward(mha_handle h, const void* x_q, const void* x_kv, const void* Wq,
                       const void* Wk, const void* Wv, const void* Wo, int B, int Lq, int Lk,
                       int heads, int mask_kind, const int32_t* key_lengths, void* out,
                       mha_stream stream) {
  if (!h) return MHA_ERR_INVALID_ARG;
  const int D = h->d_model;
  if (heads < 1 || D % heads != 0) return MHA_ERR_INVALID_ARG;
  if (B < 0 || Lq < 0 || Lk < 1) return MHA_ERR_INVALID_ARG;
  if (B > h->max_batch || Lq > h->max_lq || Lk > h->max_lk) return MHA_ERR_INVALID_ARG;
  const int d = D / heads;
  const bool empty = static_cast<long long>(B) * Lq == 0;
  if (!empty) {
    const void* ptrs[7] = {x_q, x_kv, Wq, Wk, Wv, Wo, out};
    for (const void* p : ptrs)
      if (!p || !aligned16(p)) return MHA_ERR_INVALID_ARG;
    if (out == x_q || out == x_kv) return MHA_ERR_INVALID_ARG;
  }
  // the attention step sees Q [B,H,Lq,d], K/V [B,H,Lk,d] in the workspace
  mha_status st = check_sdpa(h->q, h->k, h->v, h->ctx, B, heads, Lq, Lk, d, 0.f, mask_kind,
                             key_lengths, h->dtype, h->dtype);
  if (st != MHA_OK) return st;
  if (h->dtype == MHA_BF16 && D % 64 != 0) return MHA_ERR_UNSUPPORTED;
  if (empty) return MHA_OK;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device) return MHA_ERR_INVALID_ARG;
  DeviceCtl ctl;
  if (!get_device_ctl(&ctl)) return MHA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto gemm = h->dtype == MHA_BF16 ? launch_gemm_bf16 : launch_gemm_f32;

  // a1, a2: projections with the head split in the store layout
  cudaError_t e;
  if (x_kv == x_q && Lk == Lq) {
    GemmArgs g{};
    g.prob[0] = {x_q, Wq, h->q, GemmStore::kHeadSplit, Lq, d};
    g.prob[1] = {x_q, Wk, h->k, GemmStore::kHeadSplit, Lk, d};
    g.prob[2] = {x_q, Wv, h->v, GemmStore::kHeadSplit, Lk, d};
    g.count = 3;
    g.M = B * Lq;
    g.N = D;
    g.K = D;
    g.dtype = h->dtype;
    g.stream = s;
    e = gemm(g, ctl);
  } else {
    GemmArgs g{};
    g.prob[0] = {x_q, Wq, h->q, GemmStore::kHeadSplit, Lq, d};
    g.count = 1;
    g.M = B * Lq;
    g.N = D;
    g.K = D;
    g.dtype = h->dtype;
    g.stream = s;
    e = gemm(g, ctl);
    if (e == cudaSuccess) {
      GemmArgs g2{};
      g2.prob[0] = {x_kv, Wk, h->k, GemmStore::kHeadSplit, Lk, d};
      g2.prob[1] = {x_kv, Wv, h->v, GemmStore::kHeadSplit, Lk, d};
      g2.count = 2;
      g2.M = B * Lk;
      g2.N = D;
      g2.K = D;
      g2.dtype = h->dtype;
      g2.stream = s;
      e = gemm(g2, ctl);
    }
  }
  if (e != cudaSuccess) return from_cuda(e);
  // a3-a7: attention per head, stored as the concatenated heads [B, Lq, D]
  SdpaArgs a{h->q, h->k, h->v, h->ctx, B, heads, Lq, Lk, d,
             static_cast<float>(1.0 / sqrt(static_cast<double>(d))), mask_kind, key_lengths,
             h->dtype, h->dtype, true, s};
  e = h->dtype == MHA_BF16 ? launch_sdpa_bf16(a, ctl) : launch_sdpa_f32(a, ctl);
  if (e != cudaSuccess) return from_cuda(e);
  // a8: output projection
  GemmArgs go{};
  go.prob[0] = {h->ctx, Wo, out, GemmStore::kRowMajor, Lq, d};
  go.count = 1;
  go.M = B * Lq;
  go.N = D;
  go.K = D;
  go.dtype = h->dtype;
  go.stream = s;
  return from_cuda(gemm(go, ctl));
}

mha_status mha_selftest_wait_timeout(int limit_ms, mha_stream stream) {
  if (limit_ms < 1 || limit_ms > 10000) return MHA_ERR_INVALID_ARG;
  DeviceCtl ctl;
  if (!get_device_ctl(&ctl)) return MHA_ERR_CUDA;
  wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      ctl.err, static_cast<uint64_t>(limit_ms) * 1000000ull);
  return from_cuda(cudaGetLastError());
}

mha_status mha_check(mha_handle) {
  if (cudaDeviceSynchronize() != cudaSuccess) return MHA_ERR_CUDA;
  DeviceCtl ctl;
  if (!get_device_ctl(&ctl)) return MHA_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, ctl.err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MHA_ERR_CUDA;
  if (word) {
    const unsigned zero = 0;
    if (cudaMemcpy(ctl.err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return MHA_ERR_CUDA;
  }
  if (word & kErrTimeout) return MHA_ERR_TIMEOUT;
  if (word) return MHA_ERR_DEVICE;  // key length, token id, shared-memory layout
  return MHA_OK;
}

mha_status mha_destroy(mha_handle h) {
  if (!h) return MHA_OK;
  cudaDeviceSynchronize();
  cudaFree(h->q);
  cudaFree(h->k);
  cudaFree(h->v);
  cudaFree(h->ctx);
  delete h;
  return cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // extern "C"

// Accessors for other translation units of the library.
namespace mha {

bool device_ctl(DeviceCtl* ctl) { return get_device_ctl(ctl); }

mha_status validate_sdpa(const void* Q, const void* K, const void* V, const void* O, int B,
                         int H, int Lq, int Lk, int d, float scale, int mask_kind,
                         const int32_t* key_lengths, int in_dtype, int out_dtype) {
  return check_sdpa(Q, K, V, O, B, H, Lq, Lk, d, scale, mask_kind, key_lengths, in_dtype,
                    out_dtype);
}

}  // namespace mha
