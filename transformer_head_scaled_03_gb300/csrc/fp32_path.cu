// fp32_path.cu -- fp32 CUDA-core kernels for callers that need fp32
// accuracy (max |err| ~1e-6 against an fp64 reference, where bf16 or TF32
// tensor-core inputs would not do):
//   * scaled dot-product attention, one warp per query row at a time, lane j
//     scoring key j of a 32-key chunk held in shared memory, the row max and
//     row sum reduced with warp shuffles, online over the chunks;
//   * a 64x64-tiled GEMM C = A @ W with the head-split or row-major store.
// Formulas as in sdpa_bf16.cu: "How Transformers Work" (worksonmygpu.com),
// "Scaled dot-product attention"; "The Transformer" (rayaq.ca), "Masks: who
// may look at whom"; projections y = x @ W as in "32 Transformer"
// (ml-canon-en), "PyTorch Implementation".
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kKeys = 32;  // keys per shared-memory chunk (one per lane)

struct SdpaF32Params {
  const float* Q;
  const float* K;
  const float* V;
  float* O;
  const int32_t* key_lengths;
  unsigned* err;
  int B, H, Lq, Lk, d;
  int mask_kind;
  float scale;
  int ctx_layout;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// DP: head dim bound (d <= DP, DP in {32, 64, 128}); RPW: query rows per warp.
template <int DP, int RPW>
__global__ void __launch_bounds__(128) sdpa_f32_kernel(const SdpaF32Params p) {
  constexpr int CPL = DP / 32;  // output columns per lane
  constexpr int kRows = 4 * RPW;
  __shared__ float sQ[kRows][DP];
  __shared__ float sK[kKeys][DP + 1];  // +1: lane j reads row j without bank conflicts
  __shared__ float sV[kKeys][DP];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * kRows;
  const int h = blockIdx.y, b = blockIdx.z;
  const int d = p.d;
  const size_t bh = static_cast<size_t>(b) * p.H + h;
  const bool causal = (p.mask_kind & MHA_MASK_CAUSAL) != 0;
  int key_end = p.Lk;
  bool bad_len = false;
  if (p.mask_kind & MHA_MASK_KEY_PADDING) {
    const int L = p.key_lengths[b];
    if (L < 1 || L > p.Lk) bad_len = true;
    else key_end = L;
  }
  if (bad_len && threadIdx.x == 0 && blockIdx.x == 0 && h == 0) atomicOr(p.err, kErrKeyLength);
  int kv_stop = bad_len ? 0 : key_end;
  if (causal) kv_stop = min(kv_stop, row0 + kRows);

  for (int idx = threadIdx.x; idx < kRows * DP; idx += blockDim.x) {
    const int r = idx / DP, c = idx % DP;
    const int q = row0 + r;
    sQ[r][c] = (q < p.Lq && c < d) ? p.Q[(bh * p.Lq + q) * d + c] : 0.f;
  }
  float m[RPW], l[RPW], o[RPW][CPL];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int cc = 0; cc < CPL; ++cc) o[i][cc] = 0.f;
  }
  for (int k0 = 0; k0 < kv_stop; k0 += kKeys) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kKeys * DP; idx += blockDim.x) {
      const int j = idx / DP, c = idx % DP;
      const int key = k0 + j;
      const bool in = key < p.Lk && c < d;
      sK[j][c] = in ? p.K[(bh * p.Lk + key) * d + c] : 0.f;
      sV[j][c] = in ? p.V[(bh * p.Lk + key) * d + c] : 0.f;
    }
    __syncthreads();
    const int key = k0 + lane;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const int r = warp * RPW + i;
      const int q_row = row0 + r;
      float s = 0.f;
#pragma unroll 8
      for (int c = 0; c < DP; ++c) s = fmaf(sQ[r][c], sK[lane][c], s);
      s *= p.scale;
      const bool valid = key < key_end && (!causal || key <= q_row);
      s = valid ? s : -INFINITY;
      const float m_new = fmaxf(m[i], warp_max(s));
      if (m_new == -INFINITY) continue;  // nothing visible to this row yet
      const float alpha = expf(m[i] - m_new);
      const float pj = valid ? expf(s - m_new) : 0.f;
      l[i] = l[i] * alpha + warp_sum(pj);
#pragma unroll
      for (int cc = 0; cc < CPL; ++cc) o[i][cc] *= alpha;
#pragma unroll 8
      for (int jj = 0; jj < kKeys; ++jj) {
        const float pjj = __shfl_sync(0xffffffffu, pj, jj);
#pragma unroll
        for (int cc = 0; cc < CPL; ++cc) o[i][cc] = fmaf(pjj, sV[jj][lane + 32 * cc], o[i][cc]);
      }
      m[i] = m_new;
    }
  }
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const int q_row = row0 + warp * RPW + i;
    if (q_row >= p.Lq) continue;
    const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
    const size_t row_idx = p.ctx_layout ? (static_cast<size_t>(b) * p.Lq + q_row) * p.H + h
                                        : bh * p.Lq + q_row;
#pragma unroll
    for (int cc = 0; cc < CPL; ++cc) {
      const int c = lane + 32 * cc;
      if (c < d) p.O[row_idx * d + c] = o[i][cc] * inv;
    }
  }
}

// ------------------------------------------------------------------ GEMM

struct GemmF32Params {
  const float* A[3];
  const float* W[3];
  float* C[3];
  int store[3];
  int L[3];
  int dh[3];
  int M, N, K;
};

constexpr int kT = 64;   // output tile
constexpr int kTK = 16;  // k step

__global__ void __launch_bounds__(256) gemm_f32_kernel(const GemmF32Params p) {
  __shared__ float As[kTK][kT + 4];
  __shared__ float Ws[kTK][kT];
  const int z = blockIdx.z;
  const float* __restrict__ A = p.A[z];
  const float* __restrict__ W = p.W[z];
  const int m0 = blockIdx.y * kT, n0 = blockIdx.x * kT;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int M = p.M, N = p.N, K = p.K;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kTK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = threadIdx.x + 256 * i;
      const int r = idx / kTK, kk = idx % kTK;
      const int gm = m0 + r, gk = k0 + kk;
      As[kk][r] = (gm < M && gk < K) ? A[static_cast<size_t>(gm) * K + gk] : 0.f;
      const int kk2 = idx / kT, c = idx % kT;
      const int gk2 = k0 + kk2, gn = n0 + c;
      Ws[kk2][c] = (gk2 < K && gn < N) ? W[static_cast<size_t>(gk2) * N + gn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kTK; ++kk) {
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = Ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* C = p.C[z];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      size_t off;
      if (p.store[z] == static_cast<int>(GemmStore::kHeadSplit)) {
        const int L = p.L[z], dh = p.dh[z];
        const int bb = m / L, l = m - bb * L, hh = n / dh, c = n - hh * dh;
        off = ((static_cast<size_t>(bb) * (N / dh) + hh) * L + l) * dh + c;
      } else {
        off = static_cast<size_t>(m) * N + n;
      }
      C[off] = acc[i][j];
    }
  }
}

}  // namespace

cudaError_t launch_sdpa_f32(const SdpaArgs& a, const DeviceCtl& ctl) {
  SdpaF32Params p{};
  p.Q = static_cast<const float*>(a.Q);
  p.K = static_cast<const float*>(a.K);
  p.V = static_cast<const float*>(a.V);
  p.O = static_cast<float*>(a.O);
  p.key_lengths = a.key_lengths;
  p.err = ctl.err;
  p.B = a.B;
  p.H = a.H;
  p.Lq = a.Lq;
  p.Lk = a.Lk;
  p.d = a.d;
  p.mask_kind = a.mask_kind;
  p.scale = a.scale;
  p.ctx_layout = a.ctx_layout ? 1 : 0;
  if (a.Lq == 0 || a.H == 0 || a.B == 0) return cudaSuccess;
  // 32 query rows per CTA (16 for d > 64, to stay within 48 KB of shared memory)
  if (a.d <= 32) {
    sdpa_f32_kernel<32, 8><<<dim3((a.Lq + 31) / 32, a.H, a.B), 128, 0, a.stream>>>(p);
  } else if (a.d <= 64) {
    sdpa_f32_kernel<64, 8><<<dim3((a.Lq + 31) / 32, a.H, a.B), 128, 0, a.stream>>>(p);
  } else {
    sdpa_f32_kernel<128, 4><<<dim3((a.Lq + 15) / 16, a.H, a.B), 128, 0, a.stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_gemm_f32(const GemmArgs& g, const DeviceCtl&) {
  GemmF32Params p{};
  for (int i = 0; i < g.count; ++i) {
    p.A[i] = static_cast<const float*>(g.prob[i].A);
    p.W[i] = static_cast<const float*>(g.prob[i].W);
    p.C[i] = static_cast<float*>(g.prob[i].C);
    p.store[i] = static_cast<int>(g.prob[i].store);
    p.L[i] = g.prob[i].L;
    p.dh[i] = g.prob[i].dh;
  }
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  const dim3 grid((g.N + kT - 1) / kT, (g.M + kT - 1) / kT, g.count);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  gemm_f32_kernel<<<grid, 256, 0, g.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mha
