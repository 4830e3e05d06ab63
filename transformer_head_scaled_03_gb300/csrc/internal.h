// internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mha.h"

namespace mha {

// One scaled dot-product attention launch.
struct SdpaArgs {
  const void* Q;  // [B, H, Lq, d]
  const void* K;  // [B, H, Lk, d]
  const void* V;  // [B, H, Lk, d]
  void* O;        // [B, H, Lq, d], or [B, Lq, H*d] when ctx_layout
  int B, H, Lq, Lk, d;
  float scale;  // resolved (> 0)
  int mask_kind;
  const int32_t* key_lengths;  // device, or nullptr
  mha_dtype in_dtype, out_dtype;
  bool ctx_layout;
  cudaStream_t stream;
  // optional additive float mask: element (b, h, i, j) at
  // add_mask[b*mask_sb + h*mask_sh + i*Lk + j]; nullptr when absent
  const float* add_mask;
  int64_t mask_sb, mask_sh;
  // optional: per query row the base-2 log-sum-exp of the scaled scores,
  // [B, H, Lq] fp32 (bf16 path only); nullptr when not wanted
  float* lse = nullptr;
};

// Row-major GEMM C = A[M,K] @ W[K,N] with a choice of store layout.
enum class GemmStore : int {
  kRowMajor = 0,   // C[m, n] at m*N + n
  kHeadSplit = 1,  // m = b*L + l, n = h*dh + c  ->  C[b, h, l, c]
};

struct GemmProblem {
  const void* A;  // [M, K]
  const void* W;  // [K, N]
  void* C;
  GemmStore store;
  int L;   // rows per batch item (head split)
  int dh;  // head width (head split)
  const void* bias = nullptr;  // [N], same element type, added in the epilogue
  int relu = 0;                // max(0, .) after the bias
};

struct GemmArgs {
  GemmProblem prob[3];  // up to three problems with one shape, one launch
  int count;
  int M, N, K;
  mha_dtype dtype;
  cudaStream_t stream;
};

struct DeviceCtl {
  unsigned* err;       // device error word
  uint64_t limit_ns;   // wait limit for pipelined kernels
};

// out[m, :] = LayerNorm(a[m, :] + b[m, :]) * gamma + beta over rows of width D
// (population variance, eps), fp32 statistics; element type `dt` for a, b,
// gamma and beta, `out_dt` for out (F32 out of a BF16 layer keeps the last
// LayerNorm's output unrounded).
cudaError_t launch_add_layernorm(const void* a, const void* b, const void* gamma,
                                 const void* beta, float eps, void* out, long M, int D,
                                 mha_dtype dt, mha_dtype out_dt, cudaStream_t stream);

// C[M, N] = LayerNorm(resid + A[M, K] @ W[K, N] + bias) * gamma + beta, the
// residual add and LayerNorm in the GEMM epilogue (bf16 operands, fp32
// accumulator and statistics, population variance); N = 64..512 in steps of
// 64 so that one CTA holds whole rows.  C is bf16, or fp32 when out_dtype is
// MHA_F32.
struct GemmLnArgs {
  const void* A;      // [M, K] bf16
  const void* W;      // [K, N] bf16
  const void* bias;   // [N] bf16
  const void* resid;  // [M, N] bf16
  const void* gamma;  // [N] bf16
  const void* beta;   // [N] bf16
  float eps;
  void* C;
  mha_dtype out_dtype;
  int M, N, K;
  cudaStream_t stream;
};

bool gemm_ln_bf16_supported(int N);
cudaError_t launch_gemm_ln_bf16(const GemmLnArgs& g, const DeviceCtl& ctl);

// Device error bits of the embedding pass and the backward pass (ptx.cuh
// holds the others).
constexpr unsigned kErrTokenId = 4u;     // a token id outside [0, vocab)
constexpr unsigned kErrSmemLayout = 8u;  // dynamic shared memory too misaligned for the layout

cudaError_t launch_sinusoidal_pe(float* pe, int first_pos, int n_pos, int D, cudaStream_t s);
cudaError_t launch_embed_pe(const int32_t* ids, const void* table, int vocab, const float* pe,
                            void* x, long long rows, int L, int D, int pos_offset, float scale,
                            mha_dtype dt, unsigned* err, cudaStream_t s);

// One decode-shape attention launch (bf16 cache).
struct DecodeArgs {
  const void* Q;  // [B, H, Lq, d]
  const void* K;  // [B, H, Lk, d] cache
  const void* V;
  void* O;        // [B, H, Lq, d]
  int B, H, Lq, Lk, d;
  float scale;    // resolved (> 0)
  bool causal;    // bottom-right
  const int32_t* kv_len;  // device [B] or nullptr
  mha_dtype out_dtype;
  int splits;
  cudaStream_t stream;
};

cudaError_t launch_sdpa_decode_bf16(const DecodeArgs& a, const DeviceCtl& ctl);
int decode_default_splits(int B, int H, int Lk, int d);

cudaError_t launch_sdpa_bf16(const SdpaArgs& a, const DeviceCtl& ctl);
cudaError_t launch_sdpa_f32(const SdpaArgs& a, const DeviceCtl& ctl);
cudaError_t launch_gemm_bf16(const GemmArgs& g, const DeviceCtl& ctl);
cudaError_t launch_gemm_f32(const GemmArgs& g, const DeviceCtl& ctl);

// cuTensorMapEncodeTiled through the runtime's driver entry point.
// Returns false when the entry point is unavailable or encoding failed.
bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank,
                       void* base, const uint64_t* dims, const uint64_t* strides_bytes,
                       const uint32_t* box, CUtensorMapSwizzle swizzle);

}  // namespace mha

namespace mha {

// The current device's error word and wait limit (false if CUDA fails).
bool device_ctl(DeviceCtl* ctl);

// The argument checks sdpa_forward applies, for other entry points.
mha_status validate_sdpa(const void* Q, const void* K, const void* V, const void* O, int B,
                         int H, int Lq, int Lk, int d, float scale, int mask_kind,
                         const int32_t* key_lengths, int in_dtype, int out_dtype);

}  // namespace mha
