/*
 * mha.h -- C ABI of the GB300 (sm_103a) multi-head scaled dot-product
 * attention library (libmha_gb300.so).
 *
 * What the library computes
 *   Attention(Q, K, V) = softmax(Q K^T * scale + M) V  per (batch, head),
 *   with scale = 1/sqrt(d_k) by default and M an additive 0/-inf mask
 *     -- "How Transformers Work" (worksonmygpu.com), "Scaled dot-product
 *        attention"; "The Transformer" (hoshank.vercel.app), "The
 *        Mathematics"; masks: "The Transformer" (rayaq.ca), "Masks: who may
 *        look at whom".
 *   MultiHead(x_q, x_kv) = Concat(head_1..head_h) W^O,
 *   head_i = Attention(x_q W^Q_i, x_kv W^K_i, x_kv W^V_i)
 *     -- hoshank.vercel.app, "The Mathematics" (multi-head equation);
 *        "32 Transformer" (ml-canon-en), "PyTorch Implementation": y = x @ W,
 *        head i = column block i of the projection, heads concatenated in
 *        order before W^O.  No bias terms.
 *
 * Conventions shared by every entry point
 *   - Tensors are dense, row-major (C order), in device memory unless stated
 *     otherwise, and owned by the caller.  Every tensor pointer must be
 *     16-byte aligned (TMA requirement); pointers to distinct tensors must
 *     not overlap, except x_kv == x_q (self-attention).
 *   - Element type: MHA_BF16 = bfloat16 (uint16 bit pattern), MHA_F32 = IEEE
 *     float.  bf16 work accumulates in fp32.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Arguments are validated on the host before anything
 *     is launched; a call that returns an error has launched nothing.
 *   - Errors are returned, never printed; the library never aborts.
 *   - Device-side conditions (a key length outside [1, Lk], a pipeline wait
 *     that exceeded its time limit) set a per-device error word that
 *     mha_check() reads.  The affected rows are written as zeros.
 *   - Masks: mask_kind is a bit set of MHA_MASK_CAUSAL (key j blocked for
 *     query i when j > i; requires Lq == Lk) and MHA_MASK_KEY_PADDING (key j
 *     blocked for batch item b when j >= key_lengths[b]).  There are no
 *     boolean mask tensors, so no mask polarity to get wrong.
 */
#ifndef GB300_MHA_H
#define GB300_MHA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MHA_OK = 0,
    MHA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, bad mask */
    MHA_ERR_UNSUPPORTED = 2, /* valid request outside what is implemented */
    MHA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
    MHA_ERR_OOM = 4,         /* device allocation failed (mha_create) */
    MHA_ERR_TIMEOUT = 5,     /* a kernel pipeline wait gave up (mha_check) */
    MHA_ERR_DEVICE = 6       /* device-side argument error, e.g. a key
                                length outside [1, Lk] (mha_check) */
} mha_status;

typedef enum { MHA_F32 = 0, MHA_BF16 = 1 } mha_dtype;

enum {
    MHA_MASK_NONE = 0,
    MHA_MASK_CAUSAL = 1,
    MHA_MASK_KEY_PADDING = 2,
    /* sdpa_decode only: query i of Lq sees keys j <= len_b - Lq + i */
    MHA_MASK_CAUSAL_BOTTOM_RIGHT = 4
};

/* Largest number of new queries per (batch item, head) sdpa_decode takes. */
#define MHA_DECODE_MAX_QUERIES 16

/* Same type as cudaStream_t, declared here so the header needs no CUDA
 * include. */
typedef struct CUstream_st *mha_stream;

/* Opaque layer handle: owns the Q/K/V/context workspace for one d_model and
 * element type. */
typedef struct mha_ctx *mha_handle;

/*
 * sdpa_forward -- scaled dot-product attention for B*H independent heads.
 *   Q [B, H, Lq, d], K [B, H, Lk, d], V [B, H, Lk, d]  (in_dtype)
 *   O [B, H, Lq, d]                                    (out_dtype)
 *   scale       : multiplier of Q K^T; 0 selects 1/sqrt(d); must be finite
 *                 and >= 0.
 *   mask_kind   : bit set of MHA_MASK_*; CAUSAL requires Lq == Lk.
 *   key_lengths : device int32[B], required iff KEY_PADDING is set; each
 *                 value must lie in [1, Lk] (checked on the device).
 * Supported: in_dtype BF16 with d in {64, 128} (tcgen05 tensor-core path,
 * out_dtype BF16 or F32); in_dtype F32 with 1 <= d <= 128 (fp32 CUDA-core
 * path, out_dtype F32).  B, H, Lq may be 0 (nothing is launched); Lk >= 1.
 * Returns MHA_OK, MHA_ERR_INVALID_ARG, MHA_ERR_UNSUPPORTED or MHA_ERR_CUDA.
 */
mha_status sdpa_forward(const void *Q, const void *K, const void *V, void *O,
                        int B, int H, int Lq, int Lk, int d, float scale,
                        int mask_kind, const int32_t *key_lengths,
                        mha_dtype in_dtype, mha_dtype out_dtype,
                        mha_stream stream);

/*
 * sdpa_forward_host -- sdpa_forward on host buffers: Q, K, V (and the key
 * lengths) are copied in, attended and O is copied out, in about sixteen
 * chunks of (b, h) heads whose copies overlap the attention of other chunks
 * (every head is independent: "How Transformers Work" (worksonmygpu.com),
 * "Multi-head attention").
 *   Qh, Kh, Vh, Oh : host, same shapes and types as sdpa_forward; pinned
 *             (page-locked) memory lets the copies run asynchronously.
 *   key_lengths_h : host int32[B] or NULL, as sdpa_forward's key_lengths.
 *   workspace : device, 256-byte aligned, at least
 *             sdpa_forward_host_workspace_bytes(...) bytes; the call keeps
 *             device copies of Q, K, V, O and the lengths there.
 *   stream    : the call is ordered after work already queued on `stream`,
 *             and `stream` covers it: Oh is complete once `stream` has been
 *             synchronised.  Two internal copy streams and a second compute
 *             stream carry the overlap.
 * Same dtypes, head sizes and checks as sdpa_forward.  The call allocates
 * nothing on the device; it creates its internal streams and events once per
 * device.  Calls on one device are serialised on the host while they
 * enqueue.
 * Returns MHA_OK, MHA_ERR_INVALID_ARG, MHA_ERR_UNSUPPORTED or MHA_ERR_CUDA.
 */
mha_status sdpa_forward_host(const void *Qh, const void *Kh, const void *Vh, void *Oh,
                             int B, int H, int Lq, int Lk, int d, float scale,
                             int mask_kind, const int32_t *key_lengths_h,
                             mha_dtype in_dtype, mha_dtype out_dtype,
                             void *workspace, size_t workspace_bytes, mha_stream stream);

/* Device workspace sdpa_forward_host needs, in bytes (0 for bad arguments). */
size_t sdpa_forward_host_workspace_bytes(int B, int H, int Lq, int Lk, int d,
                                         mha_dtype in_dtype, mha_dtype out_dtype);

/*
 * sdpa_forward_float_mask -- sdpa_forward with an additive float mask added
 * to the scaled scores, the optional mask of the reference SDPA that "The
 * Transformer" (rayaq.ca) describes in "Attention, by hand" (with -inf
 * giving weight exactly 0, "Masks: who may look at whom").
 *   add_mask : device float32; element (b, h, i, j) at
 *              add_mask[b*mask_stride_b + h*mask_stride_h + i*Lk + j]
 *              (strides in elements, >= 0; 0 broadcasts over that axis;
 *              rows of Lk contiguous values).  Entries must be finite or
 *              -inf.  4-byte aligned.
 *   Other arguments, layouts and support as for sdpa_forward; mask_kind and
 *   key_lengths still apply on top.  A query row whose keys are all blocked
 *   has no defined softmax and is written as zeros.
 * Returns MHA_OK, MHA_ERR_INVALID_ARG, MHA_ERR_UNSUPPORTED or MHA_ERR_CUDA.
 */
mha_status sdpa_forward_float_mask(const void *Q, const void *K, const void *V,
                                   void *O, int B, int H, int Lq, int Lk,
                                   int d, float scale, int mask_kind,
                                   const int32_t *key_lengths,
                                   const float *add_mask,
                                   int64_t mask_stride_b,
                                   int64_t mask_stride_h, mha_dtype in_dtype,
                                   mha_dtype out_dtype, mha_stream stream);

/*
 * sdpa_decode -- attention of Lq <= 16 new queries per (batch item, head)
 * against a key/value cache: the decoder's masked self-attention while it
 * generates left to right, reusing the keys and values it has stored ("How
 * Transformers Work" (worksonmygpu.com), "What changed since 2017"; "The
 * Transformer" (hoshank.vercel.app), "The Breakthrough"; "The Transformer"
 * (rayaq.ca), "The decoder stack").
 *   Q       [B, H, Lq, d] bf16: the queries of the newest Lq positions.
 *   K_cache [B, H, Lk, d] bf16, V_cache [B, H, Lk, d] bf16: a cache of
 *           capacity Lk; batch item b holds len_b tokens in rows
 *           [0, len_b), the newest Lq of them being the queries' own.
 *   O       [B, H, Lq, d], out_dtype BF16 or F32.
 *   scale   : as for sdpa_forward (0 selects 1/sqrt(d)).
 *   mask_kind : bit set of MHA_MASK_KEY_PADDING (len_b = kv_lengths[b]; else
 *           every item holds Lk tokens) and MHA_MASK_CAUSAL_BOTTOM_RIGHT
 *           (query i sees keys j <= len_b - Lq + i; without it every query
 *           sees all len_b keys, as cross-attention to an encoder memory).
 *           MHA_MASK_CAUSAL is not accepted here.
 *   kv_lengths : device int32[B], given iff KEY_PADDING is set; each value
 *           must lie in [1, Lk], and in [Lq, Lk] with the causal bit
 *           (checked on the device: MHA_ERR_DEVICE from mha_check, rows
 *           written as zeros).
 *   num_splits : CTAs that share one (b, h)'s keys, 1..16, merged exactly
 *           through one thread-block cluster; 0 picks a default
 *           (sdpa_decode_splits).
 * d must be 64 or 128; Q, K_cache, V_cache and O 16-byte aligned.  B or H
 * may be 0 (nothing is launched).  The call allocates nothing.
 * Returns MHA_OK, MHA_ERR_INVALID_ARG, MHA_ERR_UNSUPPORTED (Lq > 16, other
 * d) or MHA_ERR_CUDA.
 */
mha_status sdpa_decode(const void *Q, const void *K_cache, const void *V_cache,
                       void *O, int B, int H, int Lq, int Lk, int d,
                       float scale, int mask_kind, const int32_t *kv_lengths,
                       mha_dtype out_dtype, int num_splits,
                       mha_stream stream);

/* The split count sdpa_decode uses for num_splits = 0 (0 for bad sizes). */
int sdpa_decode_splits(int B, int H, int Lk, int d);

/*
 * sdpa_forward_lse -- sdpa_forward (bf16 inputs) that also writes, per query
 * row, the base-2 log-sum-exp of the scaled scores, which the backward pass
 * needs to recompute the attention weights:
 *   lse[b, h, i] = log2( sum_j 2^((scale * <Q_i, K_j> + M_ij) * log2(e)) )
 * (+inf for a row with no visible key).
 *   lse : device fp32 [B, H, Lq], 4-byte aligned, caller-owned.
 * Other arguments, layouts, support and errors as for sdpa_forward with
 * in_dtype = MHA_BF16.
 */
mha_status sdpa_forward_lse(const void *Q, const void *K, const void *V, void *O,
                            float *lse, int B, int H, int Lq, int Lk, int d,
                            float scale, int mask_kind,
                            const int32_t *key_lengths, mha_dtype out_dtype,
                            mha_stream stream);

/* Workspace sdpa_backward needs, in bytes (one fp32 per query row). */
size_t sdpa_backward_workspace_bytes(int B, int H, int Lq);

/*
 * sdpa_backward -- gradients of scaled dot-product attention (the training
 * step through the attention formula of "How Transformers Work"
 * (worksonmygpu.com), "Scaled dot-product attention"): given dO = dL/dO for
 * O = sdpa_forward(Q, K, V),
 *   dV = P^T dO,  dS = P * (dO V^T - rowsum(dO * O)),
 *   dQ = scale * dS K,  dK = scale * dS^T Q.
 *   Q, O, dO [B, H, Lq, d] bf16; K, V [B, H, Lk, d] bf16 (as in the forward).
 *   lse     : fp32 [B, H, Lq] from sdpa_forward_lse on the same inputs.
 *   dQ      : fp32 [B, H, Lq, d], written once (its sum over keys stays on
 *             the chip; nothing is accumulated in global memory).
 *   dK, dV  : [B, H, Lk, d] of grad_dtype (MHA_BF16 or MHA_F32).
 *   scale, mask_kind, key_lengths : as in the forward (CAUSAL and
 *             KEY_PADDING; no float mask).
 *   workspace : device, >= sdpa_backward_workspace_bytes(B, H, Lq) bytes.
 * d must be 64 or 128; all pointers 16-byte aligned.  Blocked keys receive
 * zero gradient; a query row with no visible key gets dQ = 0.  The call
 * allocates nothing.  Two kernels run on `stream`: dK and dV (a CTA per key
 * tile) and dQ (a CTA per query tile), after the row dot products D.
 * Returns MHA_OK, MHA_ERR_INVALID_ARG, MHA_ERR_UNSUPPORTED or MHA_ERR_CUDA.
 */
mha_status sdpa_backward(const void *Q, const void *K, const void *V,
                         const void *O, const void *dO, const float *lse,
                         float *dQ, void *dK, void *dV, int B, int H, int Lq,
                         int Lk, int d, float scale, int mask_kind,
                         const int32_t *key_lengths, mha_dtype grad_dtype,
                         void *workspace, size_t workspace_bytes,
                         mha_stream stream);

/*
 * sinusoidal_pe -- the positional-encoding table, fp32 [n_pos, d_model]:
 * row r holds PE(first_pos + r, :) with PE(pos, 2i) = sin(pos / 10000^(2i/D))
 * and PE(pos, 2i+1) = cos(pos / 10000^(2i/D)) ("How Transformers Work"
 * (worksonmygpu.com), "Positional encoding"; "The Transformer"
 * (hoshank.vercel.app), "The Mathematics").  Each value is the fp64 sine or
 * cosine of the fp64 angle, rounded to fp32.  pe: device, 4-byte aligned,
 * caller-owned.  Built once per length and reused.
 * Returns MHA_OK, MHA_ERR_INVALID_ARG or MHA_ERR_CUDA.
 */
mha_status sinusoidal_pe(float *pe, int first_pos, int n_pos, int d_model,
                         mha_stream stream);

/*
 * embed_pe_forward -- the first layer's input in one pass:
 *   x[b, l, :] = table[ids[b, l], :] * scale + pe[pos_offset + l, :]
 * the token embedding scaled by sqrt(d_model) plus the positional encoding
 * ("The Transformer" (rayaq.ca), "Embeddings and positions" and the encode
 * step of "Implementation").
 *   ids   : device int32 [B, L]; each must lie in [0, vocab) (checked on the
 *           device: MHA_ERR_DEVICE from mha_check, the row written as zeros).
 *   table : device [vocab, d_model] of dtype (BF16 or F32), 16-byte aligned.
 *   pe    : device fp32 [pe_rows, d_model] from sinusoidal_pe (first_pos 0),
 *           16-byte aligned; pos_offset + L <= pe_rows.
 *   x     : device [B, L, d_model] of dtype, 16-byte aligned; the sum is
 *           taken in fp32 and rounded once.
 *   scale : 0 selects sqrt(d_model); otherwise finite and >= 0.
 * Returns MHA_OK, MHA_ERR_INVALID_ARG or MHA_ERR_CUDA.
 */
mha_status embed_pe_forward(const int32_t *ids, const void *table, int vocab,
                            const float *pe, int pe_rows, void *x, int B,
                            int L, int d_model, int pos_offset, float scale,
                            mha_dtype dtype, mha_stream stream);

/*
 * mha_create -- allocate a multi-head attention layer handle.
 *   d_model   : model width D.
 *   dtype     : element type of x, W and out (MHA_BF16 or MHA_F32).
 *   max_batch, max_lq, max_lk : the largest B, Lq, Lk later calls may use;
 *               they size the device workspace the handle owns
 *               (Q [B,H,Lq,d], K and V [B,H,Lk,d], context [B,Lq,D]).
 * The handle allocates that workspace with cudaMalloc on the current device
 * and frees it in mha_destroy.  *out is set to NULL on failure.
 * Returns MHA_OK, MHA_ERR_INVALID_ARG, MHA_ERR_OOM or MHA_ERR_CUDA.
 */
mha_status mha_create(mha_handle *out, int d_model, mha_dtype dtype,
                      int max_batch, int max_lq, int max_lk);

/*
 * mha_forward -- one multi-head attention layer forward.
 *   x_q  [B, Lq, D], x_kv [B, Lk, D] (x_kv may equal x_q: self-attention;
 *        a different tensor: cross-attention, keys/values from x_kv)
 *   Wq, Wk, Wv, Wo [D, D] row-major, applied as y = x @ W
 *   h    : number of heads; D % h must be 0; d = D / h.
 *   mask_kind, key_lengths : as for sdpa_forward.
 *   out  [B, Lq, D]
 * The projections write Q, K, V in [B, h, L, d] (the head split is the
 * store layout); attention writes the context in [B, Lq, D] (the concat is
 * the store layout); the output projection reads it.  Four launches on
 * `stream`.  Supported: BF16 with d in {64, 128}; F32 with d <= 128.
 * Returns MHA_OK, MHA_ERR_INVALID_ARG (incl. B/Lq/Lk above the handle's
 * maxima), MHA_ERR_UNSUPPORTED or MHA_ERR_CUDA.
 */
mha_status mha_forward(mha_handle handle, const void *x_q, const void *x_kv,
                       const void *Wq, const void *Wk, const void *Wv,
                       const void *Wo, int B, int Lq, int Lk, int h,
                       int mask_kind, const int32_t *key_lengths, void *out,
                       mha_stream stream);

/*
 * mha_forward_noalloc -- mha_forward for callers that cannot allocate device
 * memory.  (This entry point has no counterpart in the pages that define
 * the method; it is a property of this library's interface.)
 *
 * mha_forward keeps the projected Q, K, V and the concatenated-heads context
 * in workspace that mha_create allocates with cudaMalloc.  Callers that must
 * not call cudaMalloc -- a host program that gives all device memory to its
 * own pool, a plugin whose execution step may not allocate, a latency-bound
 * loop that cannot take cudaMalloc's implicit synchronisation -- call this
 * instead: the same four launches, with those intermediates in a fixed
 * device array inside the library.  It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *   d_model, dtype : as for mha_create; the other arguments as for
 *                    mha_forward.
 * Limit: the intermediates need 2*B*Lq*D + 2*B*Lk*D elements (each tensor
 * rounded up to 256 bytes); a call needing more than
 * MHA_NOALLOC_SCRATCH_BYTES returns MHA_ERR_INVALID_ARG and launches
 * nothing.
 * The array is held on every GPU that loads the library until the process
 * exits.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture on the device.  All calls on a device share the
 * array and leave their intermediates in it; calls whose executions overlap
 * on the GPU (different streams without ordering) race on it.
 * Returns MHA_OK, MHA_ERR_INVALID_ARG, MHA_ERR_UNSUPPORTED or MHA_ERR_CUDA.
 */
#define MHA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
mha_status mha_forward_noalloc(int d_model, mha_dtype dtype, const void *x_q,
                               const void *x_kv, const void *Wq,
                               const void *Wk, const void *Wv, const void *Wo,
                               int B, int Lq, int Lk, int h, int mask_kind,
                               const int32_t *key_lengths, void *out,
                               mha_stream stream);

/*
 * One post-norm Transformer encoder layer (next to the attention layer it
 * contains):
 *   a   = MultiHead(x, x, x) with biases (as mha_forward, plus bq, bk, bv
 *         added to the projections and bo to the output projection)
 *   x1  = LayerNorm(x + a) * ln1_gamma + ln1_beta
 *   f   = max(0, x1 W1 + b1) W2 + b2
 *   out = LayerNorm(x1 + f) * ln2_gamma + ln2_beta
 * LayerNorm over each position's D values, population variance, ln_eps
 * added to the variance (PyTorch's default is 1e-5).
 *   -- "The Transformer" (hoshank.vercel.app), "The Mathematics" (FFN and
 *      output = LayerNorm(x + Sublayer(x))); "The Transformer" (rayaq.ca),
 *      "The feed-forward block", "Residuals and LayerNorm", "The encoder
 *      stack" and the EncoderLayer of "Implementation".
 * All parameters have the layer's element type and are device pointers,
 * 16-byte aligned; matrices are row-major [d_in, d_out] applied as y = x@W.
 */
typedef struct {
    const void *Wq, *Wk, *Wv, *Wo;     /* [D, D] */
    const void *bq, *bk, *bv, *bo;     /* [D] */
    const void *ln1_gamma, *ln1_beta;  /* [D] */
    const void *W1;                    /* [D, F] */
    const void *b1;                    /* [F] */
    const void *W2;                    /* [F, D] */
    const void *b2;                    /* [D] */
    const void *ln2_gamma, *ln2_beta;  /* [D] */
} mha_encoder_params;

typedef struct mha_encoder_ctx *mha_encoder;

/* encoder_create -- a layer handle for d_model D, `heads`, FFN width d_ff,
 * element type `dtype`, up to max_batch x max_len tokens; owns cudaMalloc'd
 * workspace (Q, K, V, context, two [B,L,D] temporaries, x1, the [B,L,F]
 * hidden activation).  Supported: BF16 with D/heads in {64, 128} and D, d_ff
 * multiples of 64; F32 with D/heads <= 128; D <= 4096.  Returns MHA_OK,
 * MHA_ERR_INVALID_ARG, MHA_ERR_UNSUPPORTED, MHA_ERR_OOM or MHA_ERR_CUDA. */
mha_status encoder_create(mha_encoder *out, int d_model, int heads, int d_ff,
                          mha_dtype dtype, int max_batch, int max_len);

/* encoder_forward -- out [B, L, D] = layer(x [B, L, D]); mask_kind and
 * key_lengths as for mha_forward (self-attention, Lq = Lk = L).
 * out_dtype is the element type of `out`: the layer's type, or MHA_F32 for
 * a BF16 layer (the final LayerNorm's output stored unrounded).  BF16
 * layers with D <= 512 take five launches on `stream` (the residual add and
 * LayerNorm run in the epilogues of the W^O and W2 GEMMs, so the sublayer
 * outputs stay fp32 and are never stored); other layers take seven.  The
 * hidden activation and x1 are stored in the layer's type.  out must not
 * alias x.  Returns MHA_OK, MHA_ERR_INVALID_ARG or MHA_ERR_CUDA. */
mha_status encoder_forward(mha_encoder enc, const void *x,
                           const mha_encoder_params *params, int B, int L,
                           int mask_kind, const int32_t *key_lengths,
                           float ln_eps, void *out, mha_dtype out_dtype,
                           mha_stream stream);

/* encoder_destroy -- free the handle (synchronises the device).  NULL is
 * accepted. */
mha_status encoder_destroy(mha_encoder enc);

/*
 * mha_check -- synchronise the current device and report (then clear) its
 * device-side error word.  `handle` may be NULL.  Returns MHA_OK,
 * MHA_ERR_TIMEOUT, MHA_ERR_DEVICE or MHA_ERR_CUDA.
 */
mha_status mha_check(mha_handle handle);

/*
 * mha_selftest_wait_timeout -- exercise the failure path of the kernels'
 * bounded waits: launches one warp that waits on a shared-memory mbarrier
 * nothing arrives on, using the same wait routine as the attention and GEMM
 * pipelines, with a limit of `limit_ms` (1..10000).  The wait gives up, the
 * kernel sets MHA_ERR_TIMEOUT in the device error word and returns; a later
 * mha_check() reports (and clears) it and the context stays usable.  (A
 * property of this library's interface; the pages have no counterpart.)
 * Returns MHA_OK (launched), MHA_ERR_INVALID_ARG or MHA_ERR_CUDA.
 */
mha_status mha_selftest_wait_timeout(int limit_ms, mha_stream stream);

/* mha_destroy -- free the handle and its workspace (synchronises the
 * device first).  NULL is accepted. */
mha_status mha_destroy(mha_handle handle);

/* Static, NUL-terminated name of a status code. */
const char *mha_status_string(mha_status status);

/* Set the time limit, in milliseconds, after which a kernel pipeline wait
 * gives up and reports MHA_ERR_TIMEOUT (default 2000; applies to later
 * launches).  Returns the previous value. */
int mha_set_wait_limit_ms(int ms);

#ifdef __cplusplus
}
#endif

#endif /* GB300_MHA_H */
