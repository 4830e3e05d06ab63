// encoder_api.cu -- encoder_create / encoder_forward / encoder_destroy: one
// post-norm Transformer encoder layer on the library's kernels.
//
//   a   = MultiHead(x, x, x) with biases      (GEMM with bias epilogue and
//                                               head-split store, attention
//                                               with concat store, GEMM + bo)
//   x1  = LayerNorm1(x + a)
//   f   = max(0, x1 W1 + b1) W2 + b2          (GEMM bias+ReLU, GEMM bias)
//   out = LayerNorm2(x1 + f)
// ("The Transformer" (hoshank.vercel.app), "The Mathematics"; "The
// Transformer" (rayaq.ca), "The feed-forward block", "Residuals and
// LayerNorm", "The encoder stack".)
// bf16 layers with d_model <= 512 run five launches: the residual add and
// LayerNorm are the epilogues of the W^O and W2 GEMMs (gemm_ln_bf16), so a
// and f stay in fp32 and never reach memory.  Other layers run seven: each
// GEMM stores its output and add_layernorm reads it back.
#include <math.h>
#include <stdint.h>

#include <new>

#include "internal.h"

using namespace mha;

struct mha_encoder_ctx {
  int device;
  int D, H, F;
  mha_dtype dtype;
  int max_batch, max_len;
  void* q;    // [B, H, L, d]
  void* k;
  void* v;
  void* ctx;  // [B, L, D]
  void* tmp;  // [B, L, D]: attention output, then FFN output
  void* x1;   // [B, L, D]
  void* hid;  // [B, L, F]
};

namespace {

bool al16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mha_status status_of(cudaError_t e) {
  if (e == cudaSuccess) return MHA_OK;
  return e == cudaErrorMemoryAllocation ? MHA_ERR_OOM : MHA_ERR_CUDA;
}

void free_all(mha_encoder_ctx* c) {
  cudaFree(c->q);
  cudaFree(c->k);
  cudaFree(c->v);
  cudaFree(c->ctx);
  cudaFree(c->tmp);
  cudaFree(c->x1);
  cudaFree(c->hid);
}

}  // namespace

extern "C" {

mha_status encoder_create(mha_encoder* out, int d_model, int heads, int d_ff, mha_dtype dtype,
                          int max_batch, int max_len) {
  if (!out) return MHA_ERR_INVALID_ARG;
  *out = nullptr;
  if (d_model < 1 || heads < 1 || d_model % heads != 0 || d_ff < 1 || max_batch < 1 ||
      max_len < 1 || (dtype != MHA_BF16 && dtype != MHA_F32))
    return MHA_ERR_INVALID_ARG;
  const int d = d_model / heads;
  if (d_model > 4096) return MHA_ERR_UNSUPPORTED;
  if (dtype == MHA_BF16 && (!(d == 64 || d == 128) || d_model % 64 || d_ff % 64))
    return MHA_ERR_UNSUPPORTED;
  if (dtype == MHA_F32 && d > 128) return MHA_ERR_UNSUPPORTED;
  mha_encoder_ctx* c = new (std::nothrow) mha_encoder_ctx();
  if (!c) return MHA_ERR_OOM;
  if (cudaGetDevice(&c->device) != cudaSuccess) {
    delete c;
    return MHA_ERR_CUDA;
  }
  c->D = d_model;
  c->H = heads;
  c->F = d_ff;
  c->dtype = dtype;
  c->max_batch = max_batch;
  c->max_len = max_len;
  const size_t es = dtype == MHA_BF16 ? 2 : 4;
  const size_t nd = static_cast<size_t>(max_batch) * max_len * d_model * es;
  const size_t nf = static_cast<size_t>(max_batch) * max_len * d_ff * es;
  void** bufs[6] = {&c->q, &c->k, &c->v, &c->ctx, &c->tmp, &c->x1};
  cudaError_t e = cudaSuccess;
  for (void** b : bufs)
    if (e == cudaSuccess) e = cudaMalloc(b, nd);
  if (e == cudaSuccess) e = cudaMalloc(&c->hid, nf);
  if (e != cudaSuccess) {
    free_all(c);
    delete c;
    cudaGetLastError();
    return status_of(e);
  }
  *out = c;
  return MHA_OK;
}

mha_status encoder_forward(mha_encoder c, const void* x, const mha_encoder_params* w, int B,
                           int L, int mask_kind, const int32_t* key_lengths, float ln_eps,
                           void* out, mha_dtype out_dtype, mha_stream stream) {
  if (!c || !w) return MHA_ERR_INVALID_ARG;
  if (out_dtype != c->dtype && !(c->dtype == MHA_BF16 && out_dtype == MHA_F32))
    return MHA_ERR_INVALID_ARG;
  if (B < 0 || L < 1 || B > c->max_batch || L > c->max_len) return MHA_ERR_INVALID_ARG;
  if (!(ln_eps >= 0.f) || isinf(ln_eps)) return MHA_ERR_INVALID_ARG;
  if (mask_kind < 0 || mask_kind > (MHA_MASK_CAUSAL | MHA_MASK_KEY_PADDING))
    return MHA_ERR_INVALID_ARG;
  if ((mask_kind & MHA_MASK_KEY_PADDING) && !key_lengths) return MHA_ERR_INVALID_ARG;
  if (B == 0) return MHA_OK;
  const void* ptrs[] = {x,          out,         w->Wq,  w->Wk,  w->Wv, w->Wo,
                        w->bq,      w->bk,       w->bv,  w->bo,  w->W1, w->b1,
                        w->W2,      w->b2,       w->ln1_gamma, w->ln1_beta,
                        w->ln2_gamma, w->ln2_beta};
  for (const void* p : ptrs)
    if (!al16(p)) return MHA_ERR_INVALID_ARG;
  if (out == x) return MHA_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != c->device) return MHA_ERR_INVALID_ARG;
  DeviceCtl ctl;
  if (!device_ctl(&ctl)) return MHA_ERR_CUDA;
  const int D = c->D, H = c->H, F = c->F, d = D / H;
  const int M = B * L;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto gemm = c->dtype == MHA_BF16 ? launch_gemm_bf16 : launch_gemm_f32;
  auto gemm1 = [&](const void* A, const void* W, void* C, const void* bias, int relu, int N,
                   int K) {
    GemmArgs g{};
    g.prob[0] = {A, W, C, GemmStore::kRowMajor, L, d, bias, relu};
    g.count = 1;
    g.M = M;
    g.N = N;
    g.K = K;
    g.dtype = c->dtype;
    g.stream = s;
    return gemm(g, ctl);
  };
  // projections with biases, head split in the store
  GemmArgs g{};
  g.prob[0] = {x, w->Wq, c->q, GemmStore::kHeadSplit, L, d, w->bq, 0};
  g.prob[1] = {x, w->Wk, c->k, GemmStore::kHeadSplit, L, d, w->bk, 0};
  g.prob[2] = {x, w->Wv, c->v, GemmStore::kHeadSplit, L, d, w->bv, 0};
  g.count = 3;
  g.M = M;
  g.N = D;
  g.K = D;
  g.dtype = c->dtype;
  g.stream = s;
  cudaError_t e = gemm(g, ctl);
  if (e != cudaSuccess) return status_of(e);
  // attention, concatenated heads
  SdpaArgs a{c->q, c->k, c->v, c->ctx, B, H, L, L, d,
             static_cast<float>(1.0 / sqrt(static_cast<double>(d))), mask_kind, key_lengths,
             c->dtype, c->dtype, true, s, nullptr, 0, 0};
  e = c->dtype == MHA_BF16 ? launch_sdpa_bf16(a, ctl) : launch_sdpa_f32(a, ctl);
  if (e != cudaSuccess) return status_of(e);
  if (c->dtype == MHA_BF16 && gemm_ln_bf16_supported(D)) {
    // x1 = LN1(x + ctx Wo + bo); hid = relu(x1 W1 + b1); out = LN2(x1 + hid W2 + b2)
    auto gemm_ln = [&](const void* A, const void* W, const void* bias, const void* resid,
                       const void* gamma, const void* beta, void* C, mha_dtype odt, int K) {
      GemmLnArgs g{A, W, bias, resid, gamma, beta, ln_eps, C, odt, M, D, K, s};
      return launch_gemm_ln_bf16(g, ctl);
    };
    if ((e = gemm_ln(c->ctx, w->Wo, w->bo, x, w->ln1_gamma, w->ln1_beta, c->x1, MHA_BF16, D)) !=
        cudaSuccess)
      return status_of(e);
    if ((e = gemm1(c->x1, w->W1, c->hid, w->b1, 1, F, D)) != cudaSuccess) return status_of(e);
    return status_of(gemm_ln(c->hid, w->W2, w->b2, c->x1, w->ln2_gamma, w->ln2_beta, out,
                             out_dtype, F));
  }
  if ((e = gemm1(c->ctx, w->Wo, c->tmp, w->bo, 0, D, D)) != cudaSuccess) return status_of(e);
  if ((e = launch_add_layernorm(x, c->tmp, w->ln1_gamma, w->ln1_beta, ln_eps, c->x1, M, D,
                                c->dtype, c->dtype, s)) != cudaSuccess)
    return status_of(e);
  if ((e = gemm1(c->x1, w->W1, c->hid, w->b1, 1, F, D)) != cudaSuccess) return status_of(e);
  if ((e = gemm1(c->hid, w->W2, c->tmp, w->b2, 0, D, F)) != cudaSuccess) return status_of(e);
  return status_of(launch_add_layernorm(c->x1, c->tmp, w->ln2_gamma, w->ln2_beta, ln_eps, out, M,
                                        D, c->dtype, out_dtype, s));
}

mha_status encoder_destroy(mha_encoder c) {
  if (!c) return MHA_OK;
  cudaDeviceSynchronize();
  free_all(c);
  delete c;
  return cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // extern "C"
