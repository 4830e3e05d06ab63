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

constexpr int kKeys = 64;   // keys per shared-memory chunk (two per lane)
constexpr int kRowsW = 4;   // query rows per warp, processed together
constexpr int kWarps = 4;   // warps per CTA
constexpr int kRowsC = kRowsW * kWarps;

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
  const float* add_mask;  // optional additive float mask (scaled-score units)
  int64_t mask_sb, mask_sh;
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

// One CTA = 16 query rows of one (b, h); warp w owns rows 4w..4w+3 and
// scores them together against each 64-key chunk (lane j: keys j and j+32),
// so every K and V element read from shared memory serves four rows.
// DP: head-dim bound (d <= DP, DP in {32, 64, 128}).
template <int DP>
__global__ void __launch_bounds__(kWarps * 32) sdpa_f32_kernel(const SdpaF32Params p) {
  constexpr int CPL = DP / 32;  // output columns per lane
  extern __shared__ __align__(16) float fsm[];
  float* sQ = fsm;                              // [kRowsC][DP]
  float* sK = sQ + kRowsC * DP;                 // [kKeys][DP + 1]
  float* sV = sK + kKeys * (DP + 1);            // [kKeys][DP]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * kRowsC;
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
  if (causal) kv_stop = min(kv_stop, row0 + kRowsC);

  for (int idx = threadIdx.x; idx < kRowsC * DP; idx += blockDim.x) {
    const int r = idx / DP, c = idx % DP;
    const int q = row0 + r;
    sQ[idx] = (q < p.Lq && c < d) ? p.Q[(bh * p.Lq + q) * d + c] * p.scale : 0.f;
  }
  float m[kRowsW], l[kRowsW], o[kRowsW][CPL];
#pragma unroll
  for (int i = 0; i < kRowsW; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int cc = 0; cc < CPL; ++cc) o[i][cc] = 0.f;
  }
  const float* q_rows = sQ + warp * kRowsW * DP;
  for (int k0 = 0; k0 < kv_stop; k0 += kKeys) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kKeys * DP; idx += blockDim.x) {
      const int j = idx / DP, c = idx % DP;
      const int key = k0 + j;
      const bool in = key < p.Lk && c < d;
      sK[j * (DP + 1) + c] = in ? p.K[(bh * p.Lk + key) * d + c] : 0.f;
      sV[j * DP + c] = in ? p.V[(bh * p.Lk + key) * d + c] : 0.f;
    }
    __syncthreads();
    // scores s[i][t] of row i against key k0 + lane + 32 t (Q pre-scaled)
    float s[kRowsW][2];
#pragma unroll
    for (int i = 0; i < kRowsW; ++i) s[i][0] = s[i][1] = 0.f;
    const float* k_a = sK + lane * (DP + 1);
    const float* k_b = sK + (lane + 32) * (DP + 1);
#pragma unroll 8
    for (int c = 0; c < DP; ++c) {
      const float ka = k_a[c], kb = k_b[c];
#pragma unroll
      for (int i = 0; i < kRowsW; ++i) {
        const float qv = q_rows[i * DP + c];
        s[i][0] = fmaf(qv, ka, s[i][0]);
        s[i][1] = fmaf(qv, kb, s[i][1]);
      }
    }
    float pj[kRowsW][2];
#pragma unroll
    for (int i = 0; i < kRowsW; ++i) {
      const int q_row = row0 + warp * kRowsW + i;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int key = k0 + lane + 32 * t;
        const bool valid = key < key_end && (!causal || key <= q_row);
        s[i][t] = valid ? s[i][t] : -INFINITY;
        if (p.add_mask && valid && q_row < p.Lq)
          s[i][t] += __ldg(p.add_mask + static_cast<int64_t>(b) * p.mask_sb +
                           static_cast<int64_t>(h) * p.mask_sh +
                           static_cast<int64_t>(q_row) * p.Lk + key);
      }
      const float m_new = fmaxf(m[i], warp_max(fmaxf(s[i][0], s[i][1])));
      if (m_new == -INFINITY) {  // nothing visible to this row yet (uniform in the warp)
        pj[i][0] = pj[i][1] = 0.f;
        continue;
      }
      const float alpha = expf(m[i] - m_new);
      pj[i][0] = s[i][0] == -INFINITY ? 0.f : expf(s[i][0] - m_new);
      pj[i][1] = s[i][1] == -INFINITY ? 0.f : expf(s[i][1] - m_new);
      l[i] = l[i] * alpha + warp_sum(pj[i][0] + pj[i][1]);
#pragma unroll
      for (int cc = 0; cc < CPL; ++cc) o[i][cc] *= alpha;
      m[i] = m_new;
    }
    // o[i][c] += sum_j p_ij V[j][c]; lane owns columns lane + 32 cc
#pragma unroll 4
    for (int jj = 0; jj < 32; ++jj) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        float vv[CPL];
#pragma unroll
        for (int cc = 0; cc < CPL; ++cc) vv[cc] = sV[(jj + 32 * t) * DP + lane + 32 * cc];
#pragma unroll
        for (int i = 0; i < kRowsW; ++i) {
          const float pv = __shfl_sync(0xffffffffu, pj[i][t], jj);
#pragma unroll
          for (int cc = 0; cc < CPL; ++cc) o[i][cc] = fmaf(pv, vv[cc], o[i][cc]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kRowsW; ++i) {
    const int q_row = row0 + warp * kRowsW + i;
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
//
// C = A[M,K] @ W[K,N] in fp32 FFMA.  CTA tile 32 x 64, k-step 32, 256
// threads, each owning 2 rows x 4 columns; both operand tiles are staged in
// shared memory by cp.async through a two-stage ring so the next k-step's
// loads are in flight while the current one is multiplied.  When K or N is
// not a multiple of 4 (no 16-byte chunks), the tiles are filled by plain
// loads instead.

struct GemmF32Params {
  const float* A[3];
  const float* W[3];
  float* C[3];
  const float* bias[3];
  int relu[3];
  int store[3];
  int L[3];
  int dh[3];
  int M, N, K;
};

constexpr int kBM = 32, kBN = 64, kBK = 32;
constexpr int kApad = kBK + 4;  // A rows of 36 floats: 16-byte aligned, conflict-free column reads

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <bool kVec>
__global__ void __launch_bounds__(256) gemm_f32_kernel(const GemmF32Params p) {
  __shared__ __align__(16) float As[2][kBM][kApad];
  __shared__ __align__(16) float Ws[2][kBK][kBN];
  const int z = blockIdx.z;
  const float* __restrict__ A = p.A[z];
  const float* __restrict__ W = p.W[z];
  const int M = p.M, N = p.N, K = p.K;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;  // columns 4*tx.., rows 2*ty..
  const int num_k = (K + kBK - 1) / kBK;

  auto load_tile = [&](int kt, int buf) {
    const int k0 = kt * kBK;
    if constexpr (kVec) {
      {  // A: 32 rows x 8 chunks of 4 floats, one chunk per thread
        const int r = tid >> 3, c4 = (tid & 7) * 4;
        const int gm = m0 + r, gk = k0 + c4;
        const bool in = gm < M && gk < K;
        cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(&As[buf][r][c4])),
                   in ? A + static_cast<size_t>(gm) * K + gk : A, in ? 16u : 0u);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {  // W: 32 rows x 16 chunks, two per thread
        const int idx = tid + 256 * i;
        const int r = idx >> 4, c4 = (idx & 15) * 4;
        const int gk = k0 + r, gn = n0 + c4;
        const bool in = gk < K && gn < N;
        cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(&Ws[buf][r][c4])),
                   in ? W + static_cast<size_t>(gk) * N + gn : W, in ? 16u : 0u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int idx = tid + 256 * i;
        const int r = idx >> 5, c = idx & 31;
        const int gm = m0 + r, gk = k0 + c;
        As[buf][r][c] = (gm < M && gk < K) ? A[static_cast<size_t>(gm) * K + gk] : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int idx = tid + 256 * i;
        const int r = idx >> 6, c = idx & 63;
        const int gk = k0 + r, gn = n0 + c;
        Ws[buf][r][c] = (gk < K && gn < N) ? W[static_cast<size_t>(gk) * N + gn] : 0.f;
      }
    }
  };

  float acc[2][4] = {};
  load_tile(0, 0);
  if constexpr (kVec) cp_async_commit();
  for (int kt = 0; kt < num_k; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < num_k) {
      load_tile(kt + 1, buf ^ 1);
      if constexpr (kVec) {
        cp_async_commit();
        cp_async_wait<1>();  // tile kt has landed; kt+1 may still be in flight
      }
    } else if constexpr (kVec) {
      cp_async_wait<0>();
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      const float a0 = As[buf][2 * ty][kk], a1 = As[buf][2 * ty + 1][kk];
      const float4 w = *reinterpret_cast<const float4*>(&Ws[buf][kk][4 * tx]);
      acc[0][0] = fmaf(a0, w.x, acc[0][0]);
      acc[0][1] = fmaf(a0, w.y, acc[0][1]);
      acc[0][2] = fmaf(a0, w.z, acc[0][2]);
      acc[0][3] = fmaf(a0, w.w, acc[0][3]);
      acc[1][0] = fmaf(a1, w.x, acc[1][0]);
      acc[1][1] = fmaf(a1, w.y, acc[1][1]);
      acc[1][2] = fmaf(a1, w.z, acc[1][2]);
      acc[1][3] = fmaf(a1, w.w, acc[1][3]);
    }
    __syncthreads();  // the buffer is refilled two k-steps later
  }
  float* C = p.C[z];
  const bool split = p.store[z] == static_cast<int>(GemmStore::kHeadSplit);
  const float* bias = p.bias[z];
  const bool relu = p.relu[z] != 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int m = m0 + 2 * ty + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + 4 * tx + j;
      if (n >= N) continue;
      size_t off;
      if (split) {
        const int L = p.L[z], dh = p.dh[z];
        const int bb = m / L, l = m - bb * L, hh = n / dh, c = n - hh * dh;
        off = ((static_cast<size_t>(bb) * (N / dh) + hh) * L + l) * dh + c;
      } else {
        off = static_cast<size_t>(m) * N + n;
      }
      float v = acc[i][j];
      if (bias) v += bias[n];
      if (relu) v = fmaxf(v, 0.f);
      C[off] = v;
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
  p.add_mask = a.add_mask;
  p.mask_sb = a.mask_sb;
  p.mask_sh = a.mask_sh;
  if (a.Lq == 0 || a.H == 0 || a.B == 0) return cudaSuccess;
  const dim3 grid((a.Lq + kRowsC - 1) / kRowsC, a.H, a.B);
  auto smem = [](int DP) { return (kRowsC * DP + kKeys * (DP + 1) + kKeys * DP) * 4; };
  if (a.d <= 32) {
    sdpa_f32_kernel<32><<<grid, kWarps * 32, smem(32), a.stream>>>(p);
  } else if (a.d <= 64) {
    sdpa_f32_kernel<64><<<grid, kWarps * 32, smem(64), a.stream>>>(p);
  } else {
    cudaError_t e = cudaFuncSetAttribute(sdpa_f32_kernel<128>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem(128));
    if (e != cudaSuccess) return e;
    sdpa_f32_kernel<128><<<grid, kWarps * 32, smem(128), a.stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_gemm_f32(const GemmArgs& g, const DeviceCtl&) {
  GemmF32Params p{};
  for (int i = 0; i < g.count; ++i) {
    p.A[i] = static_cast<const float*>(g.prob[i].A);
    p.W[i] = static_cast<const float*>(g.prob[i].W);
    p.C[i] = static_cast<float*>(g.prob[i].C);
    p.bias[i] = static_cast<const float*>(g.prob[i].bias);
    p.relu[i] = g.prob[i].relu;
    p.store[i] = static_cast<int>(g.prob[i].store);
    p.L[i] = g.prob[i].L;
    p.dh[i] = g.prob[i].dh;
  }
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  const dim3 grid((g.N + kBN - 1) / kBN, (g.M + kBM - 1) / kBM, g.count);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  bool vec = g.K % 4 == 0 && g.N % 4 == 0;
  for (int i = 0; i < g.count; ++i)
    vec = vec && (reinterpret_cast<uintptr_t>(p.A[i]) & 15u) == 0 &&
          (reinterpret_cast<uintptr_t>(p.W[i]) & 15u) == 0;
  if (vec) gemm_f32_kernel<true><<<grid, 256, 0, g.stream>>>(p);
  else gemm_f32_kernel<false><<<grid, 256, 0, g.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mha
