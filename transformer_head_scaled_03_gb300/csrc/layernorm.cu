// layernorm.cu -- residual add + LayerNorm, the sublayer wrapper of the
// post-norm encoder layer: out = LayerNorm(a + b) * gamma + beta per row
// ("The Transformer" (hoshank.vercel.app), "The Mathematics": output =
// LayerNorm(x + Sublayer(x)); "The Transformer" (rayaq.ca), "Residuals and
// LayerNorm": each position rescaled to mean 0 and variance 1, then a
// learned scale and shift).  Memory-bound: one warp per row, the row held
// in registers, fp32 statistics with the centred two-pass variance
// (population variance, divisor D).
#include <cuda_bf16.h>

#include "internal.h"

namespace mha {
namespace {

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float lane_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr int kRowsPerBlock = 4;

// VPL: values per lane held in registers (D <= 32 * VPL); TO: output type
template <typename T, int VPL, typename TO = T>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
    add_layernorm_kernel(const T* __restrict__ a, const T* __restrict__ b,
                         const T* __restrict__ gamma, const T* __restrict__ beta, float eps,
                         TO* __restrict__ out, long M, int D) {
  const int lane = threadIdx.x & 31;
  const long row = static_cast<long>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  if (row >= M) return;  // whole warp leaves together
  const T* ar = a + row * D;
  const T* br = b + row * D;
  float v[VPL];
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int c = lane + 32 * i;
    v[i] = c < D ? to_f(ar[c]) + to_f(br[c]) : 0.f;
    sum += v[i];
  }
  const float mean = lane_sum(sum) / static_cast<float>(D);
  float sq = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int c = lane + 32 * i;
    const float dv = c < D ? v[i] - mean : 0.f;
    sq = fmaf(dv, dv, sq);
  }
  const float var = lane_sum(sq) / static_cast<float>(D);
  const float inv = 1.f / sqrtf(var + eps);
  TO* orow = out + row * D;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int c = lane + 32 * i;
    if (c < D) orow[c] = from_f<TO>((v[i] - mean) * inv * to_f(gamma[c]) + to_f(beta[c]));
  }
}

// The same with 16-byte loads and stores: lane l of the warp owns the
// 16-byte pieces l, l + 32, ... of the row (NCH pieces, E = 16 / sizeof(T)
// values each), so a warp instruction moves 512 contiguous bytes.  Used when
// D is a multiple of 32 * E and every row starts 16-byte aligned.
template <typename T, int NCH>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
    add_layernorm_vec_kernel(const T* __restrict__ a, const T* __restrict__ b,
                             const T* __restrict__ gamma, const T* __restrict__ beta, float eps,
                             T* __restrict__ out, long M, int D) {
  constexpr int E = 16 / static_cast<int>(sizeof(T));
  const int lane = threadIdx.x & 31;
  const long row = static_cast<long>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  if (row >= M) return;  // whole warp leaves together
  const uint4* ar = reinterpret_cast<const uint4*>(a + row * D);
  const uint4* br = reinterpret_cast<const uint4*>(b + row * D);
  float v[NCH][E];
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const uint4 ua = __ldg(ar + lane + 32 * i), ub = __ldg(br + lane + 32 * i);
    const T* ta = reinterpret_cast<const T*>(&ua);
    const T* tb = reinterpret_cast<const T*>(&ub);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      v[i][e] = to_f(ta[e]) + to_f(tb[e]);
      sum += v[i][e];
    }
  }
  const float mean = lane_sum(sum) / static_cast<float>(D);
  float sq = 0.f;
#pragma unroll
  for (int i = 0; i < NCH; ++i)
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float dv = v[i][e] - mean;
      sq = fmaf(dv, dv, sq);
    }
  const float var = lane_sum(sq) / static_cast<float>(D);
  const float inv = 1.f / sqrtf(var + eps);
  const uint4* gr = reinterpret_cast<const uint4*>(gamma);
  const uint4* be = reinterpret_cast<const uint4*>(beta);
  uint4* orow = reinterpret_cast<uint4*>(out + row * D);
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const uint4 ug = __ldg(gr + lane + 32 * i), ube = __ldg(be + lane + 32 * i);
    const T* tg = reinterpret_cast<const T*>(&ug);
    const T* tbe = reinterpret_cast<const T*>(&ube);
    uint4 uo;
    T* to = reinterpret_cast<T*>(&uo);
#pragma unroll
    for (int e = 0; e < E; ++e) to[e] = from_f<T>((v[i][e] - mean) * inv * to_f(tg[e]) + to_f(tbe[e]));
    orow[lane + 32 * i] = uo;
  }
}

template <typename T>
cudaError_t launch_typed(const void* a, const void* b, const void* g, const void* be, float eps,
                         void* out, long M, int D, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((M + kRowsPerBlock - 1) / kRowsPerBlock));
  const dim3 block(32 * kRowsPerBlock);
  auto args = [&](auto kern) {
    kern<<<grid, block, 0, s>>>(static_cast<const T*>(a), static_cast<const T*>(b),
                                static_cast<const T*>(g), static_cast<const T*>(be), eps,
                                static_cast<T*>(out), M, D);
  };
  constexpr int E = 16 / static_cast<int>(sizeof(T));
  bool vec = D % (32 * E) == 0 && D <= 32 * E * 16 &&
                   ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
                     reinterpret_cast<uintptr_t>(g) | reinterpret_cast<uintptr_t>(be) |
                     reinterpret_cast<uintptr_t>(out)) & 15u) == 0;
  if (vec) {
    const int nch = D / (32 * E);
    if (nch == 1) args(add_layernorm_vec_kernel<T, 1>);
    else if (nch == 2) args(add_layernorm_vec_kernel<T, 2>);
    else if (nch == 4) args(add_layernorm_vec_kernel<T, 4>);
    else if (nch == 8) args(add_layernorm_vec_kernel<T, 8>);
    else if (nch == 16) args(add_layernorm_vec_kernel<T, 16>);
    else vec = false;
    if (vec) return cudaGetLastError();
  }
  if (D <= 32 * 16) args(add_layernorm_kernel<T, 16>);
  else if (D <= 32 * 32) args(add_layernorm_kernel<T, 32>);
  else if (D <= 32 * 128) args(add_layernorm_kernel<T, 128>);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

// bf16 inputs, fp32 output (row by row; the layer's last LayerNorm only)
cudaError_t launch_bf16_to_f32(const void* a, const void* b, const void* g, const void* be,
                               float eps, void* out, long M, int D, cudaStream_t s) {
  using T = __nv_bfloat16;
  const dim3 grid(static_cast<unsigned>((M + kRowsPerBlock - 1) / kRowsPerBlock));
  const dim3 block(32 * kRowsPerBlock);
  auto args = [&](auto kern) {
    kern<<<grid, block, 0, s>>>(static_cast<const T*>(a), static_cast<const T*>(b),
                                static_cast<const T*>(g), static_cast<const T*>(be), eps,
                                static_cast<float*>(out), M, D);
  };
  if (D <= 32 * 16) args(add_layernorm_kernel<T, 16, float>);
  else if (D <= 32 * 32) args(add_layernorm_kernel<T, 32, float>);
  else if (D <= 32 * 128) args(add_layernorm_kernel<T, 128, float>);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_add_layernorm(const void* a, const void* b, const void* gamma,
                                 const void* beta, float eps, void* out, long M, int D,
                                 mha_dtype dt, mha_dtype out_dt, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  if (dt == MHA_BF16 && out_dt == MHA_F32)
    return launch_bf16_to_f32(a, b, gamma, beta, eps, out, M, D, stream);
  if (out_dt != dt) return cudaErrorInvalidValue;
  return dt == MHA_BF16 ? launch_typed<__nv_bfloat16>(a, b, gamma, beta, eps, out, M, D, stream)
                        : launch_typed<float>(a, b, gamma, beta, eps, out, M, D, stream);
}

}  // namespace mha
