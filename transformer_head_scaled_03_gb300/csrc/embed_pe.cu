// embed_pe.cu -- the input of the first layer: token embedding scaled by
// sqrt(d_model) plus the sinusoidal positional encoding, in one pass.
//
//   PE(pos, 2i)   = sin(pos / 10000^(2i / D))
//   PE(pos, 2i+1) = cos(pos / 10000^(2i / D))
//   x[b, l, :]    = table[ids[b, l], :] * sqrt(D) + PE(pos_offset + l, :)
// ("How Transformers Work" (worksonmygpu.com), "Positional encoding"; "The
// Transformer" (hoshank.vercel.app), "The Mathematics"; "The Transformer"
// (rayaq.ca), "Embeddings and positions" and the encode step of
// "Implementation".)
//
// The PE table is built once per length (fp64 sine and cosine of the fp64
// angle, stored fp32) and is shared by every batch item, so it stays in L2
// while the embedding pass streams: the pass reads each token's table row
// and writes its x row once, 16-byte vectors, one warp per row.
#include <math.h>
#include <stdint.h>

#include <cuda_bf16.h>

#include "internal.h"

namespace mha {
namespace {

constexpr int kRowsPerBlock = 8;  // one warp per row

__global__ void sinusoidal_pe_kernel(float* __restrict__ pe, int first_pos, int n_pos, int D) {
  const long long total = static_cast<long long>(n_pos) * D;
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(e / D);
    const int c = static_cast<int>(e - static_cast<long long>(r) * D);
    const int i = c >> 1;
    const double angle = static_cast<double>(first_pos + r) / pow(10000.0, (2.0 * i) / D);
    pe[e] = static_cast<float>((c & 1) ? cos(angle) : sin(angle));
  }
}

__device__ __forceinline__ void fma8(const uint4& t, const float4& p0, const float4& p1,
                                     float scale, float (&o)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&t);
  const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
  const float2 c = __bfloat1622float2(h[2]), d = __bfloat1622float2(h[3]);
  o[0] = fmaf(a.x, scale, p0.x);
  o[1] = fmaf(a.y, scale, p0.y);
  o[2] = fmaf(b.x, scale, p0.z);
  o[3] = fmaf(b.y, scale, p0.w);
  o[4] = fmaf(c.x, scale, p1.x);
  o[5] = fmaf(c.y, scale, p1.y);
  o[6] = fmaf(d.x, scale, p1.z);
  o[7] = fmaf(d.y, scale, p1.w);
}

// bf16 table and x, D % 8 == 0: lane j handles 8-column groups j, j+32, ...
__global__ void __launch_bounds__(32 * kRowsPerBlock)
    embed_pe_bf16_kernel(const int32_t* __restrict__ ids, const __nv_bfloat16* __restrict__ table,
                         int vocab, const float* __restrict__ pe, __nv_bfloat16* __restrict__ x,
                         long long rows, int L, int D, int pos_offset, float scale,
                         unsigned* err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int groups = D >> 3;
  for (long long row = static_cast<long long>(blockIdx.x) * kRowsPerBlock + warp; row < rows;
       row += static_cast<long long>(gridDim.x) * kRowsPerBlock) {
    const int id = __ldg(ids + row);
    const int l = static_cast<int>(row % L);
    uint4* xr = reinterpret_cast<uint4*>(x + row * D);
    if (id < 0 || id >= vocab) {
      if (lane == 0) atomicOr(err, kErrTokenId);
      for (int g = lane; g < groups; g += 32) xr[g] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const uint4* tr = reinterpret_cast<const uint4*>(table + static_cast<long long>(id) * D);
    const float4* pr = reinterpret_cast<const float4*>(pe + static_cast<long long>(pos_offset + l) * D);
    for (int g = lane; g < groups; g += 32) {
      const uint4 t = __ldg(tr + g);
      const float4 p0 = __ldg(pr + 2 * g), p1 = __ldg(pr + 2 * g + 1);
      float o[8];
      fma8(t, p0, p1, scale, o);
      uint4 w;
      __nv_bfloat162 q0 = __floats2bfloat162_rn(o[0], o[1]);
      __nv_bfloat162 q1 = __floats2bfloat162_rn(o[2], o[3]);
      __nv_bfloat162 q2 = __floats2bfloat162_rn(o[4], o[5]);
      __nv_bfloat162 q3 = __floats2bfloat162_rn(o[6], o[7]);
      w.x = *reinterpret_cast<uint32_t*>(&q0);
      w.y = *reinterpret_cast<uint32_t*>(&q1);
      w.z = *reinterpret_cast<uint32_t*>(&q2);
      w.w = *reinterpret_cast<uint32_t*>(&q3);
      xr[g] = w;
    }
  }
}

// Element-wise form for fp32, or bf16 rows that are not a multiple of 8.
template <typename T>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
    embed_pe_scalar_kernel(const int32_t* __restrict__ ids, const T* __restrict__ table, int vocab,
                           const float* __restrict__ pe, T* __restrict__ x, long long rows, int L,
                           int D, int pos_offset, float scale, unsigned* err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (long long row = static_cast<long long>(blockIdx.x) * kRowsPerBlock + warp; row < rows;
       row += static_cast<long long>(gridDim.x) * kRowsPerBlock) {
    const int id = __ldg(ids + row);
    const int l = static_cast<int>(row % L);
    T* xr = x + row * D;
    if (id < 0 || id >= vocab) {
      if (lane == 0) atomicOr(err, kErrTokenId);
      for (int c = lane; c < D; c += 32) xr[c] = static_cast<T>(0.f);
      continue;
    }
    const T* tr = table + static_cast<long long>(id) * D;
    const float* pr = pe + static_cast<long long>(pos_offset + l) * D;
    for (int c = lane; c < D; c += 32)
      xr[c] = static_cast<T>(fmaf(static_cast<float>(tr[c]), scale, __ldg(pr + c)));
  }
}

// SMs of the current device, asked at every launch (the runtime answers from
// its cached device properties), so that each device gets its own count; 1
// if the query fails, which only shrinks the grid.
int num_sms() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
    return v;
  return 1;
}

}  // namespace

cudaError_t launch_sinusoidal_pe(float* pe, int first_pos, int n_pos, int D, cudaStream_t s) {
  const long long total = static_cast<long long>(n_pos) * D;
  if (total == 0) return cudaSuccess;
  const long long want = (total + 255) / 256;
  const int blocks = static_cast<int>(want < 16LL * num_sms() ? want : 16LL * num_sms());
  sinusoidal_pe_kernel<<<blocks, 256, 0, s>>>(pe, first_pos, n_pos, D);
  return cudaGetLastError();
}

cudaError_t launch_embed_pe(const int32_t* ids, const void* table, int vocab, const float* pe,
                            void* x, long long rows, int L, int D, int pos_offset, float scale,
                            mha_dtype dt, unsigned* err, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  // enough warps in flight to cover HBM latency: 16 blocks of 8 rows per SM
  const long long want = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  const int blocks = static_cast<int>(want < 16LL * num_sms() ? want : 16LL * num_sms());
  const dim3 block(32 * kRowsPerBlock);
  if (dt == MHA_BF16 && D % 8 == 0) {
    embed_pe_bf16_kernel<<<blocks, block, 0, s>>>(
        ids, static_cast<const __nv_bfloat16*>(table), vocab, pe,
        static_cast<__nv_bfloat16*>(x), rows, L, D, pos_offset, scale, err);
  } else if (dt == MHA_BF16) {
    embed_pe_scalar_kernel<__nv_bfloat16><<<blocks, block, 0, s>>>(
        ids, static_cast<const __nv_bfloat16*>(table), vocab, pe,
        static_cast<__nv_bfloat16*>(x), rows, L, D, pos_offset, scale, err);
  } else {
    embed_pe_scalar_kernel<float><<<blocks, block, 0, s>>>(
        ids, static_cast<const float*>(table), vocab, pe, static_cast<float*>(x), rows, L, D,
        pos_offset, scale, err);
  }
  return cudaGetLastError();
}

}  // namespace mha

using namespace mha;

extern "C" {

mha_status sinusoidal_pe(float* pe, int first_pos, int n_pos, int d_model, mha_stream stream) {
  if (first_pos < 0 || n_pos < 0 || d_model < 1) return MHA_ERR_INVALID_ARG;
  if (static_cast<long long>(first_pos) + n_pos > 0x7fffffffLL) return MHA_ERR_INVALID_ARG;
  if (n_pos == 0) return MHA_OK;
  if (!pe || (reinterpret_cast<uintptr_t>(pe) & 3u)) return MHA_ERR_INVALID_ARG;
  const cudaError_t e =
      launch_sinusoidal_pe(pe, first_pos, n_pos, d_model, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

mha_status embed_pe_forward(const int32_t* ids, const void* table, int vocab, const float* pe,
                            int pe_rows, void* x, int B, int L, int d_model, int pos_offset,
                            float scale, mha_dtype dtype, mha_stream stream) {
  if (B < 0 || L < 0 || d_model < 1 || vocab < 1 || pos_offset < 0 || pe_rows < 0)
    return MHA_ERR_INVALID_ARG;
  if (dtype != MHA_BF16 && dtype != MHA_F32) return MHA_ERR_INVALID_ARG;
  if (!(scale >= 0.f) || isinf(scale)) return MHA_ERR_INVALID_ARG;
  if (static_cast<long long>(pos_offset) + L > pe_rows) return MHA_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * L;
  if (rows == 0) return MHA_OK;
  if (!ids || !table || !pe || !x) return MHA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ids) & 3u) || (reinterpret_cast<uintptr_t>(pe) & 15u) ||
      (reinterpret_cast<uintptr_t>(table) & 15u) || (reinterpret_cast<uintptr_t>(x) & 15u))
    return MHA_ERR_INVALID_ARG;
  DeviceCtl ctl;
  if (!device_ctl(&ctl)) return MHA_ERR_CUDA;
  const float sc = scale == 0.f ? static_cast<float>(sqrt(static_cast<double>(d_model))) : scale;
  const cudaError_t e = launch_embed_pe(ids, table, vocab, pe, x, rows, L, d_model, pos_offset,
                                        sc, dtype, ctl.err, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // extern "C"
