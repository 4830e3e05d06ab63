// fp32_path.cu -- fp32 CUDA-core kernels for callers that need fp32
// accuracy (max |err| ~1e-6 against an fp64 reference, where bf16 or TF32
// tensor-core inputs would not do):
//   * scaled dot-product attention, one warp per two query rows against
//     64-key chunks held in shared memory (lane j scoring keys j and j + 32,
//     or, for short layers, two key groups of warps with lane j scoring key
//     32g + j and a final merge), the row max and row sum reduced with warp
//     shuffles, online over the chunks;
//   * a tiled GEMM C = A @ W with the head-split or row-major store (32 x 64
//     tiles, or 16 x 32 tiles with the k-steps split inside the CTA for
//     problems too small to fill the GPU).
// Formulas as in sdpa_bf16.cu: "How Transformers Work" (worksonmygpu.com),
// "Scaled dot-product attention"; "The Transformer" (rayaq.ca), "Masks: who
// may look at whom"; projections y = x @ W as in "32 Transformer"
// (ml-canon-en), "PyTorch Implementation".
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kKeys = 64;   // keys per shared-memory chunk
constexpr int kRowsW = 2;   // query rows per warp, processed together
constexpr int kWarps = 8;   // warps per CTA
// query rows per CTA with KG key groups (the warps of a group share rows)
__host__ __device__ constexpr int rows_per_cta(int KG) { return kRowsW * kWarps / KG; }

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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}

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

// One CTA = eight warps in KG key groups over 16 / KG query rows of one
// (b, h).  Warp w of group g owns rows 2w, 2w+1 and scores them together
// against its keys of each 64-key chunk (KG = 1: lane j takes keys j and
// j + 32; KG = 2: group g takes keys 32g..32g+31, lane j key 32g + j), so
// every K and V element read from shared memory serves two rows.  With two
// groups each keeps its own running max, sum and output and the two are
// merged at the end: twice the CTAs for a short layer whose 16-row grid
// would leave SMs idle.  The chunks stream through two shared-memory stages
// by cp.async: chunk c + 1 is in flight while chunk c is scored, and the
// first two are requested before Q is read, so the load latencies of a short
// key range overlap.
// DP: head-dim bound (d <= DP, DP in {32, 64, 128}).
template <int DP, int KG>
__global__ void __launch_bounds__(kWarps * 32) sdpa_f32_kernel(const SdpaF32Params p) {
  constexpr int CPL = DP / 32;             // output columns per lane
  constexpr int KPL = kKeys / 32 / KG;     // keys per lane per chunk
  constexpr int kGroupWarps = kWarps / KG;
  constexpr int kRowsC = rows_per_cta(KG);
  extern __shared__ __align__(16) float fsm[];
  float* sQ = fsm;                              // [kRowsC][DP]
  float* sK0 = sQ + kRowsC * DP;                // two stages of [kKeys][DP + 1]
  float* sV0 = sK0 + 2 * kKeys * (DP + 1);      // two stages of [kKeys][DP]
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

  // key chunk c (keys c*kKeys ..) -> stage c & 1; rows past Lk and columns
  // past d are zero-filled.  V goes in 16-byte pieces when its rows allow
  // (d a multiple of 4, 16-byte aligned base).
  const bool v_vec = (d % 4 == 0) && (reinterpret_cast<uintptr_t>(p.V) & 15u) == 0;
  auto load_chunk = [&](int chunk) {
    float* sK = sK0 + (chunk & 1) * kKeys * (DP + 1);
    float* sV = sV0 + (chunk & 1) * kKeys * DP;
    const int k0 = chunk * kKeys;
    for (int idx = threadIdx.x; idx < kKeys * DP; idx += blockDim.x) {
      const int j = idx / DP, c = idx % DP;
      const int key = k0 + j;
      const bool in = key < p.Lk && c < d;
      const size_t g = in ? (bh * p.Lk + key) * d + c : 0;
      // K rows are padded to DP + 1 floats (conflict-free column reads), so
      // they go element by element
      cp_async4(static_cast<uint32_t>(__cvta_generic_to_shared(sK + j * (DP + 1) + c)), p.K + g,
                in ? 4u : 0u);
    }
    if (v_vec) {  // V rows: 16-byte pieces
      for (int idx = threadIdx.x; idx < kKeys * DP / 4; idx += blockDim.x) {
        const int j = idx / (DP / 4), c = (idx % (DP / 4)) * 4;
        const int key = k0 + j;
        const bool in = key < p.Lk && c < d;
        const size_t g = in ? (bh * p.Lk + key) * d + c : 0;
        cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(sV + j * DP + c)), p.V + g,
                   in ? 16u : 0u);
      }
    } else {
      for (int idx = threadIdx.x; idx < kKeys * DP; idx += blockDim.x) {
        const int j = idx / DP, c = idx % DP;
        const int key = k0 + j;
        const bool in = key < p.Lk && c < d;
        const size_t g = in ? (bh * p.Lk + key) * d + c : 0;
        cp_async4(static_cast<uint32_t>(__cvta_generic_to_shared(sV + j * DP + c)), p.V + g,
                  in ? 4u : 0u);
      }
    }
  };
  const int n_chunks = (kv_stop + kKeys - 1) / kKeys;
  // the Q rows are requested first, so that their loads are not queued behind
  // the two chunks' copies; they are scaled and stored once those are issued
  constexpr int kQPerThread = kRowsC * DP / (kWarps * 32);
  static_assert(kQPerThread * kWarps * 32 == kRowsC * DP, "Q tile split over the threads");
  float qv[kQPerThread];
#pragma unroll
  for (int i = 0; i < kQPerThread; ++i) {
    const int idx = threadIdx.x + kWarps * 32 * i;
    const int r = idx / DP, c = idx % DP;
    const int q = row0 + r;
    qv[i] = (q < p.Lq && c < d) ? __ldg(p.Q + (bh * p.Lq + q) * d + c) : 0.f;
  }
  if (n_chunks > 0) load_chunk(0);
  cp_async_commit();
  if (n_chunks > 1) load_chunk(1);
  cp_async_commit();
#pragma unroll
  for (int i = 0; i < kQPerThread; ++i) sQ[threadIdx.x + kWarps * 32 * i] = qv[i] * p.scale;
  const int grp = warp / kGroupWarps, wg = warp % kGroupWarps;
  // this lane's keys within a chunk: 32 (grp KPL + t) + lane, t < KPL
  auto key_of = [&](int t) { return 32 * (grp * KPL + t) + lane; };
  float m[kRowsW], l[kRowsW], o[kRowsW][CPL];
#pragma unroll
  for (int i = 0; i < kRowsW; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int cc = 0; cc < CPL; ++cc) o[i][cc] = 0.f;
  }
  const float* q_rows = sQ + wg * kRowsW * DP;
  for (int chunk = 0; chunk < n_chunks; ++chunk) {
    const int k0 = chunk * kKeys;
    const float* sK = sK0 + (chunk & 1) * kKeys * (DP + 1);
    const float* sV = sV0 + (chunk & 1) * kKeys * DP;
    cp_async_wait<1>();  // this chunk has landed (the next may be in flight)
    __syncthreads();
    // scores s[i][t] of row i against key k0 + key_of(t) (Q pre-scaled)
    float s[kRowsW][KPL];
#pragma unroll
    for (int i = 0; i < kRowsW; ++i)
#pragma unroll
      for (int t = 0; t < KPL; ++t) s[i][t] = 0.f;
#pragma unroll 8
    for (int c = 0; c < DP; ++c) {
      float kv[KPL];
#pragma unroll
      for (int t = 0; t < KPL; ++t) kv[t] = sK[key_of(t) * (DP + 1) + c];
#pragma unroll
      for (int i = 0; i < kRowsW; ++i) {
        const float qv = q_rows[i * DP + c];
#pragma unroll
        for (int t = 0; t < KPL; ++t) s[i][t] = fmaf(qv, kv[t], s[i][t]);
      }
    }
    float pj[kRowsW][KPL];
#pragma unroll
    for (int i = 0; i < kRowsW; ++i) {
      const int q_row = row0 + wg * kRowsW + i;
      float mx = -INFINITY;
#pragma unroll
      for (int t = 0; t < KPL; ++t) {
        const int key = k0 + key_of(t);
        const bool valid = key < key_end && (!causal || key <= q_row);
        s[i][t] = valid ? s[i][t] : -INFINITY;
        if (p.add_mask && valid && q_row < p.Lq)
          s[i][t] += __ldg(p.add_mask + static_cast<int64_t>(b) * p.mask_sb +
                           static_cast<int64_t>(h) * p.mask_sh +
                           static_cast<int64_t>(q_row) * p.Lk + key);
        mx = fmaxf(mx, s[i][t]);
      }
      const float m_new = fmaxf(m[i], warp_max(mx));
      if (m_new == -INFINITY) {  // nothing visible to this row yet (uniform in the warp)
#pragma unroll
        for (int t = 0; t < KPL; ++t) pj[i][t] = 0.f;
        continue;
      }
      const float alpha = expf(m[i] - m_new);
      float ps = 0.f;
#pragma unroll
      for (int t = 0; t < KPL; ++t) {
        pj[i][t] = s[i][t] == -INFINITY ? 0.f : expf(s[i][t] - m_new);
        ps += pj[i][t];
      }
      l[i] = l[i] * alpha + warp_sum(ps);
#pragma unroll
      for (int cc = 0; cc < CPL; ++cc) o[i][cc] *= alpha;
      m[i] = m_new;
    }
    // o[i][c] += sum_j p_ij V[j][c] over this group's keys; lane owns
    // columns lane + 32 cc
#pragma unroll 4
    for (int jj = 0; jj < 32; ++jj) {
#pragma unroll
      for (int t = 0; t < KPL; ++t) {
        float vv[CPL];
#pragma unroll
        for (int cc = 0; cc < CPL; ++cc)
          vv[cc] = sV[(32 * (grp * KPL + t) + jj) * DP + lane + 32 * cc];
#pragma unroll
        for (int i = 0; i < kRowsW; ++i) {
          const float pv = __shfl_sync(0xffffffffu, pj[i][t], jj);
#pragma unroll
          for (int cc = 0; cc < CPL; ++cc) o[i][cc] = fmaf(pv, vv[cc], o[i][cc]);
        }
      }
    }
    __syncthreads();  // every warp is done with this stage before it is refilled
    if (chunk + 2 < n_chunks) load_chunk(chunk + 2);
    cp_async_commit();
  }
  cp_async_wait<0>();
  float* mrg = sK0;  // [kRowsC][DP + 2]: group 1's max, sum and output rows
  if constexpr (KG == 2) {
    // merge the two key groups' partial softmax states through the (now
    // idle) first K stage
    __syncthreads();
    if (grp == 1) {
#pragma unroll
      for (int i = 0; i < kRowsW; ++i) {
        float* row = mrg + (wg * kRowsW + i) * (DP + 2);
        if (lane == 0) {
          row[0] = m[i];
          row[1] = l[i];
        }
#pragma unroll
        for (int cc = 0; cc < CPL; ++cc) row[2 + lane + 32 * cc] = o[i][cc];
      }
    }
    __syncthreads();
    if (grp != 0) return;
  }
#pragma unroll
  for (int i = 0; i < kRowsW; ++i) {
    const int q_row = row0 + wg * kRowsW + i;
    if (q_row >= p.Lq) continue;
    float a0 = 1.f, a1 = 0.f, lsum = l[i];
    const float* row = mrg + (wg * kRowsW + i) * (DP + 2);
    if constexpr (KG == 2) {
      const float m1 = row[0];
      const float mm = fmaxf(m[i], m1);
      a0 = m[i] == -INFINITY ? 0.f : expf(m[i] - mm);
      a1 = m1 == -INFINITY ? 0.f : expf(m1 - mm);
      lsum = l[i] * a0 + row[1] * a1;
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const size_t row_idx = p.ctx_layout ? (static_cast<size_t>(b) * p.Lq + q_row) * p.H + h
                                        : bh * p.Lq + q_row;
#pragma unroll
    for (int cc = 0; cc < CPL; ++cc) {
      const int c = lane + 32 * cc;
      if (c >= d) continue;
      float v = o[i][cc] * a0;
      if constexpr (KG == 2) v += row[2 + c] * a1;
      p.O[row_idx * d + c] = v * inv;
    }
  }
}

// ------------------------------------------------------------------ GEMM
//
// C = A[M,K] @ W[K,N] in fp32 FFMA.  CTA tile 32 x 64, k-step 32, 256
// threads, each owning 2 rows x 4 columns (the small-M form below serves
// problems that would leave SMs idle).  Both operand tiles are staged in
// shared memory by cp.async through a ring of kStages k-steps, so that
// kStages - 1 k-steps of loads are in flight while one is multiplied: with
// K = 512 a k-step is a few hundred cycles of arithmetic, well under the
// latency of an L2 or HBM load.  When K or N is not a multiple of 4 (no
// 16-byte chunks), the tiles are filled by plain loads instead.

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

constexpr int kBM = 32, kBK = 32;
constexpr int kApad = kBK + 4;  // A rows of 36 floats: 16-byte aligned, conflict-free column reads
constexpr int kStages = 4;
constexpr int kSplitBM = 16;  // rows of the small-M form's tiles


template <int BN>
constexpr int gemm_f32_smem() {
  return kStages * (kBM * kApad + kBK * BN) * 4;
}

template <bool kVec, int BN>
__global__ void __launch_bounds__(256) gemm_f32_kernel(const GemmF32Params p) {
  constexpr int TX = BN / 4;         // threads across the columns (4 columns each)
  constexpr int TY = 256 / TX;       // threads down the rows
  constexpr int RM = kBM / TY;       // rows per thread
  static_assert(RM * TY == kBM && TX * TY == 256, "thread layout");
  extern __shared__ __align__(16) float gsm[];
  float (*As)[kBM][kApad] = reinterpret_cast<float (*)[kBM][kApad]>(gsm);
  float (*Ws)[kBK][BN] = reinterpret_cast<float (*)[kBK][BN]>(gsm + kStages * kBM * kApad);
  const int z = blockIdx.z;
  const float* __restrict__ A = p.A[z];
  const float* __restrict__ W = p.W[z];
  const int M = p.M, N = p.N, K = p.K;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * BN;
  const int tid = threadIdx.x;
  const int tx = tid % TX, ty = tid / TX;  // columns 4*tx.., rows RM*ty..
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
      for (int i = 0; i < BN / 32; ++i) {  // W: 32 rows x BN/4 chunks
        const int idx = tid + 256 * i;
        const int r = idx / TX, c4 = (idx % TX) * 4;
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
      for (int i = 0; i < BN / 8; ++i) {
        const int idx = tid + 256 * i;
        const int r = idx / BN, c = idx % BN;
        const int gk = k0 + r, gn = n0 + c;
        Ws[buf][r][c] = (gk < K && gn < N) ? W[static_cast<size_t>(gk) * N + gn] : 0.f;
      }
    }
  };

  float acc[RM][4] = {};
  // prologue: the first kStages - 1 k-steps in flight (empty groups keep the
  // group count in step when K is short)
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < num_k) load_tile(s, s);
    if constexpr (kVec) cp_async_commit();
  }
  for (int kt = 0; kt < num_k; ++kt) {
    const int buf = kt % kStages;
    if constexpr (kVec) cp_async_wait<kStages - 2>();  // k-step kt has landed
    __syncthreads();  // ... for every thread; and the buffer refilled below is free
    {
      const int kn = kt + kStages - 1;
      if (kn < num_k) load_tile(kn, kn % kStages);
      if constexpr (kVec) cp_async_commit();
    }
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      const float4 w = *reinterpret_cast<const float4*>(&Ws[buf][kk][4 * tx]);
#pragma unroll
      for (int i = 0; i < RM; ++i) {
        const float a = As[buf][RM * ty + i][kk];
        acc[i][0] = fmaf(a, w.x, acc[i][0]);
        acc[i][1] = fmaf(a, w.y, acc[i][1]);
        acc[i][2] = fmaf(a, w.z, acc[i][2]);
        acc[i][3] = fmaf(a, w.w, acc[i][3]);
      }
    }
  }
  float* C = p.C[z];
  const bool split = p.store[z] == static_cast<int>(GemmStore::kHeadSplit);
  const float* bias = p.bias[z];
  const bool relu = p.relu[z] != 0;
#pragma unroll
  for (int i = 0; i < RM; ++i) {
    const int m = m0 + RM * ty + i;
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

// Small-M form: 16 x 32 CTA tiles with the k-step split eight ways inside the
// CTA.  Warp g multiplies k-columns 4g..4g+3 of every staged k-step, each
// lane a 4 x 4 block of the tile (rows ty + 4i, columns 4tx..4tx+3): one
// 16-byte load brings a row's four k values of A, one a k row's four columns
// of W, so 8 shared-memory loads feed 64 FMAs (both conflict-free).  The
// eight partial tiles are summed through shared memory at the end, in a fixed
// order.  It puts eight warps on each output tile, for problems too small to
// fill the GPU with CTAs (a 128-row layer).
template <bool kVec, int BM, int NS, int CNT>
__global__ void __launch_bounds__(256) gemm_f32_splitk_kernel(const GemmF32Params p) {
  // CNT problems per CTA (1, or 3 when the three share A: the same tile of
  // Q, K and V from one staged tile of x)
  constexpr int BN = 32;
  static_assert(BM == 16, "a warp covers 16 rows x 32 columns in 4 x 4 blocks");
  extern __shared__ __align__(16) float gsm[];
  float (*As)[BM][kApad] = reinterpret_cast<float (*)[BM][kApad]>(gsm);
  float (*Ws)[CNT][kBK][BN] = reinterpret_cast<float (*)[CNT][kBK][BN]>(gsm + NS * BM * kApad);
  const int z0 = blockIdx.z * CNT;
  const float* __restrict__ A = p.A[z0];
  const int M = p.M, N = p.N, K = p.K;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int tid = threadIdx.x;
  const int grp = tid >> 5, lane = tid & 31;
  const int ty = lane >> 3, tx = lane & 7;  // rows ty + 4i, columns 4tx..4tx+3
  const int num_k = (K + kBK - 1) / kBK;

  auto load_tile = [&](int kt, int buf) {
    const int k0 = kt * kBK;
    if constexpr (kVec) {
      if (tid < BM * 8) {  // A: BM rows x 8 chunks of 4 floats
        const int r = tid >> 3, c4 = (tid & 7) * 4;
        const int gm = m0 + r, gk = k0 + c4;
        const bool in = gm < M && gk < K;
        cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(&As[buf][r][c4])),
                   in ? A + static_cast<size_t>(gm) * K + gk : A, in ? 16u : 0u);
      }
#pragma unroll
      for (int zz = 0; zz < CNT; ++zz) {  // W: 32 rows x 8 chunks per problem
        const float* __restrict__ W = p.W[z0 + zz];
        const int r = tid >> 3, c4 = (tid & 7) * 4;
        const int gk = k0 + r, gn = n0 + c4;
        const bool in = gk < K && gn < N;
        cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(&Ws[buf][zz][r][c4])),
                   in ? W + static_cast<size_t>(gk) * N + gn : W, in ? 16u : 0u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int idx = tid + 256 * i;
        const int r = idx >> 5, c = idx & 31;
        if (r < BM) {
          const int gm = m0 + r, gk = k0 + c;
          As[buf][r][c] = (gm < M && gk < K) ? A[static_cast<size_t>(gm) * K + gk] : 0.f;
        }
        const int gk2 = k0 + r, gn = n0 + c;
#pragma unroll
        for (int zz = 0; zz < CNT; ++zz)
          Ws[buf][zz][r][c] =
              (gk2 < K && gn < N) ? p.W[z0 + zz][static_cast<size_t>(gk2) * N + gn] : 0.f;
      }
    }
  };

  float acc[CNT][4][4] = {};
#pragma unroll
  for (int st = 0; st < NS - 1; ++st) {
    if (st < num_k) load_tile(st, st);
    if constexpr (kVec) cp_async_commit();
  }
  for (int kt = 0; kt < num_k; ++kt) {
    const int buf = kt % NS;
    if constexpr (kVec) cp_async_wait<NS - 2>();
    __syncthreads();
    {
      const int kn = kt + NS - 1;
      if (kn < num_k) load_tile(kn, kn % NS);
      if constexpr (kVec) cp_async_commit();
    }
    float4 a4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a4[i] = *reinterpret_cast<const float4*>(&As[buf][ty + 4 * i][4 * grp]);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int zz = 0; zz < CNT; ++zz) {
        const float4 w = *reinterpret_cast<const float4*>(&Ws[buf][zz][4 * grp + kk][4 * tx]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float a = kk == 0 ? a4[i].x : kk == 1 ? a4[i].y : kk == 2 ? a4[i].z : a4[i].w;
          acc[zz][i][0] = fmaf(a, w.x, acc[zz][i][0]);
          acc[zz][i][1] = fmaf(a, w.y, acc[zz][i][1]);
          acc[zz][i][2] = fmaf(a, w.z, acc[zz][i][2]);
          acc[zz][i][3] = fmaf(a, w.w, acc[zz][i][3]);
        }
      }
    }
  }
  if constexpr (kVec) cp_async_wait<0>();
  __syncthreads();  // the stages are free: reuse them for the eight partial tiles
  float (*red)[8][BM][BN + 1] = reinterpret_cast<float (*)[8][BM][BN + 1]>(gsm);
#pragma unroll
  for (int zz = 0; zz < CNT; ++zz)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) red[zz][grp][ty + 4 * i][4 * tx + j] = acc[zz][i][j];
  __syncthreads();
#pragma unroll
  for (int zz = 0; zz < CNT; ++zz) {
    const int z = z0 + zz;
    float* C = p.C[z];
    const bool split = p.store[z] == static_cast<int>(GemmStore::kHeadSplit);
    const float* bias = p.bias[z];
    const bool relu = p.relu[z] != 0;
#pragma unroll
    for (int e = 0; e < BM / 8; ++e) {
      const int o = tid + 256 * e;
      const int r = o >> 5, c = o & 31;
      const int m = m0 + r, n = n0 + c;
      if (m >= M || n >= N) continue;
      float v = ((red[zz][0][r][c] + red[zz][1][r][c]) + (red[zz][2][r][c] + red[zz][3][r][c])) +
                ((red[zz][4][r][c] + red[zz][5][r][c]) + (red[zz][6][r][c] + red[zz][7][r][c]));
      size_t off;
      if (split) {
        const int L = p.L[z], dh = p.dh[z];
        const int bb = m / L, l = m - bb * L, hh = n / dh, cc = n - hh * dh;
        off = ((static_cast<size_t>(bb) * (N / dh) + hh) * L + l) * dh + cc;
      } else {
        off = static_cast<size_t>(m) * N + n;
      }
      if (bias) v += bias[n];
      if (relu) v = fmaxf(v, 0.f);
      C[off] = v;
    }
  }
}

template <bool kVec, int NS, int CNT>
cudaError_t launch_splitk_ns(const GemmF32Params& p, int count, cudaStream_t s) {
  constexpr int BM = kSplitBM;
  const dim3 grid((p.N + 31) / 32, (p.M + BM - 1) / BM, count / CNT);
  auto kern = gemm_f32_splitk_kernel<kVec, BM, NS, CNT>;
  constexpr int smem = NS * (BM * kApad + CNT * kBK * 32) * 4;
  static_assert(smem >= CNT * 8 * BM * 33 * 4, "partial tiles fit in the stages");
  static_assert(smem <= 232448, "shared memory");
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, 256, smem, s>>>(p);
  return cudaGetLastError();
}

// The ring is as deep as residency allows: a 128-row layer's GEMM is a chain
// of k-steps waiting on L2, so more k-steps in flight shorten it, as long as
// the grid still fits on the GPU at once (a stage is 6.4 KB: 16 stages keep two
// CTAs per SM, 8 keep four).  Three problems that share A (the Q, K and V
// projections of self-attention) run as one CTA per tile position when that
// fits on the GPU in one CTA per SM: x's tile is staged once for all three,
// and each warp keeps three independent accumulator sets.
template <bool kVec>
cudaError_t launch_gemm_f32_splitk(const GemmF32Params& p, int count, cudaStream_t s, int sms) {
  const long long pos = static_cast<long long>((p.N + 31) / 32) * ((p.M + kSplitBM - 1) / kSplitBM);
  if (count == 3 && p.A[0] == p.A[1] && p.A[0] == p.A[2] && pos <= sms)
    return launch_splitk_ns<kVec, 12, 3>(p, count, s);
  const long long ctas = pos * count;
  if (ctas <= 2LL * sms) return launch_splitk_ns<kVec, 16, 1>(p, count, s);
  if (ctas <= 4LL * sms) return launch_splitk_ns<kVec, 8, 1>(p, count, s);
  return launch_splitk_ns<kVec, 4, 1>(p, count, s);
}

template <bool kVec, int BN>
cudaError_t launch_gemm_f32_tiles(const GemmF32Params& p, int count, cudaStream_t s) {
  const dim3 grid((p.N + BN - 1) / BN, (p.M + kBM - 1) / kBM, count);
  auto kern = gemm_f32_kernel<kVec, BN>;
  constexpr int smem = gemm_f32_smem<BN>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, 256, smem, s>>>(p);
  return cudaGetLastError();
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
  auto smem = [](int DP, int KG) {
    return (rows_per_cta(KG) * DP + 2 * kKeys * (DP + 1) + 2 * kKeys * DP) * 4;
  };
  auto run = [&](auto kern, int DP, int KG) -> cudaError_t {
    const int rows = rows_per_cta(KG);
    const dim3 grid((a.Lq + rows - 1) / rows, a.H, a.B);
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem(DP, KG));
    if (e != cudaSuccess) return e;
    kern<<<grid, kWarps * 32, smem(DP, KG), a.stream>>>(p);
    return cudaGetLastError();
  };
  // two key groups (8-row CTAs) when 16-row CTAs would not give every SM one
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  const long long ctas16 =
      static_cast<long long>((a.Lq + rows_per_cta(1) - 1) / rows_per_cta(1)) * a.H * a.B;
  const bool split = ctas16 < sms;
  if (a.d <= 32) return split ? run(sdpa_f32_kernel<32, 2>, 32, 2) : run(sdpa_f32_kernel<32, 1>, 32, 1);
  if (a.d <= 64) return split ? run(sdpa_f32_kernel<64, 2>, 64, 2) : run(sdpa_f32_kernel<64, 1>, 64, 1);
  return split ? run(sdpa_f32_kernel<128, 2>, 128, 2) : run(sdpa_f32_kernel<128, 1>, 128, 1);
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
  if (g.N <= 0 || g.M <= 0 || g.count <= 0) return cudaSuccess;
  bool vec = g.K % 4 == 0 && g.N % 4 == 0;
  for (int i = 0; i < g.count; ++i)
    vec = vec && (reinterpret_cast<uintptr_t>(p.A[i]) & 15u) == 0 &&
          (reinterpret_cast<uintptr_t>(p.W[i]) & 15u) == 0;
  // the split-k form when 32 x 64 tiles would not give every SM a CTA
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  const long long wide = static_cast<long long>((g.N + 63) / 64) * ((g.M + kBM - 1) / kBM) * g.count;
  if (wide < sms)
    return vec ? launch_gemm_f32_splitk<true>(p, g.count, g.stream, sms)
               : launch_gemm_f32_splitk<false>(p, g.count, g.stream, sms);
  return vec ? launch_gemm_f32_tiles<true, 64>(p, g.count, g.stream)
             : launch_gemm_f32_tiles<false, 64>(p, g.count, g.stream);
}

}  // namespace mha
