// sdpa_bf16.cu -- fused scaled dot-product attention forward, bf16 in, fp32
// accumulate, for sm_103a (tcgen05 tensor cores, tensor memory, TMA).
//
// Computes, per (batch b, head h) and query row i,
//     O[i] = sum_j softmax_j(scale * <Q[i], K[j]> + M[i][j]) V[j]
// ("How Transformers Work" (worksonmygpu.com), "Scaled dot-product
// attention"; masks as in "The Transformer" (rayaq.ca), "Masks: who may look
// at whom") without ever writing the Lq x Lk score matrix to memory: keys
// are visited in 128-key tiles and the softmax is accumulated online (a
// running row maximum m and row sum l in fp32; when m grows the partial
// output is rescaled by 2^((m_old - m_new) * scale * log2 e)).  This is the
// exact-attention-by-tiling idea the pages credit to FlashAttention
// ("32 Transformer" (ml-canon-en), "Connections"), laid out for tcgen05.
//
// CTA = NQT query tiles of 128 rows of one (b, h).  Warp roles:
//   warps 0 .. 4*NQT-1 : one softmax warpgroup per query tile; thread r of
//                        the group owns query row r (TMEM lane r), so the
//                        row max and row sum are thread-local.
//   warp 4*NQT         : TMA producer (Q once, then a ring of NST K and V
//                        stages, 128-byte swizzled).
//   warp 4*NQT+1       : MMA issuer (one thread) and TMEM owner.
// Per key tile j (BN = 128 or 64 keys) and query tile t:
//   S_t  = Q_t K_j^T           tcgen05.mma, A and B from shared memory,
//                              fp32 accumulator in TMEM (BN columns)
//   P_t  = 2^(S_t*c - m*c)     softmax warps: tcgen05.ld of S, mask, online
//                              max/sum, P packed to bf16 and tcgen05.st back
//                              into the first BN/2 columns of S_t
//   O_t += P_t V_j             tcgen05.mma with A = P_t from TMEM and
//                              B = V_j (MN-major) from shared memory
// Under the causal mask each query tile stops at its own diagonal.
// The epilogue divides O_t by l and stores bf16 or fp32, either as
// [B,H,Lq,d] or directly in the concatenated-heads layout [B,Lq,H*d].
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kBlockM = 128;      // query rows per tile = TMEM lanes
constexpr int kSub = 128 * 128;   // bytes of a 128-row x 64-column bf16 block

struct SdpaParams {
  void* O;
  const int32_t* key_lengths;
  unsigned* err;
  uint64_t limit_ns;
  int B, H, Lq, Lk;
  int num_q_blocks;
  int mask_kind;
  float scale_log2;  // scale * log2(e)
  int out_f32;
  int ctx_layout;
  const float* add_mask;  // additive float mask (kernels instantiated with kAddMask)
  int64_t mask_sb, mask_sh;
  float inv_scale;        // the mask is added to raw scores as M / scale
  int mask_vec;           // rows are 16-byte aligned: load the mask as float4
  float* lse;             // optional [B, H, Lq]: log2 of sum_j 2^(s_ij * scale_log2)
};

// BN = keys per K/V tile (128, or 64 to fit more query tiles in tensor
// memory: each query tile holds BN columns of S and D columns of O).
template <int D, int NQT, int NST, int BN = 128>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(BN == 64 || BN == 128, "key tile");
  static constexpr int KB = D / 64;                 // 64-column (128-byte) blocks per row
  static constexpr int kQTileBytes = KB * kSub;     // one 128-row tile of Q
  static constexpr int kKVBlock = BN * 128;         // one BN-row x 64-column block of K or V
  static constexpr int kKVTileBytes = KB * kKVBlock;
  static constexpr int kSoftmaxWarps = 4 * NQT;
  static constexpr int kTmaWarp = kSoftmaxWarps;
  static constexpr int kMmaWarp = kSoftmaxWarps + 1;
  static constexpr int kThreads = 32 * (kSoftmaxWarps + 2);
  static constexpr int kTmemNeed = NQT * (BN + D);
  static constexpr uint32_t kTmemCols = kTmemNeed <= 128 ? 128u : kTmemNeed <= 256 ? 256u : 512u;
  static_assert(kTmemNeed <= 512, "TMEM budget");
  // CTAs meant to share an SM: as many as tensor memory allows for the
  // short-sequence d = 64 forms (their shared memory and registers are
  // sized for it), one otherwise
  static constexpr int kMinBlocks =
      (D == 64 && NST == 2 && NQT == 1) ? static_cast<int>(512u / kTmemCols)
      : (D == 64 && BN == 64) ? 2 : 1;
  // tensor-memory columns
  __host__ __device__ static constexpr uint32_t tS(int t) { return static_cast<uint32_t>(t * BN); }
  __host__ __device__ static constexpr uint32_t tO(int t) { return static_cast<uint32_t>(NQT * BN + t * D); }
  // barrier indices
  static constexpr int bQ = 0;
  __host__ __device__ static constexpr int bKF(int s) { return 1 + s; }
  __host__ __device__ static constexpr int bKE(int s) { return 1 + NST + s; }
  __host__ __device__ static constexpr int bVF(int s) { return 1 + 2 * NST + s; }
  __host__ __device__ static constexpr int bVE(int s) { return 1 + 3 * NST + s; }
  __host__ __device__ static constexpr int bS(int t) { return 1 + 4 * NST + t; }
  __host__ __device__ static constexpr int bP(int t) { return 1 + 4 * NST + NQT + t; }
  __host__ __device__ static constexpr int bO(int t) { return 1 + 4 * NST + 2 * NQT + t; }
  static constexpr int bDrain = 1 + 4 * NST + 3 * NQT;
  static constexpr int kNumBars = bDrain + 1;
  // shared-memory layout from a 1024-byte aligned base
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + NQT * kQTileBytes;
  static constexpr int kOffV = kOffK + NST * kKVTileBytes;
  static constexpr int kOffBar = kOffV + NST * kKVTileBytes;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory");
};

// Bounded wait that ignores the abort flag: used to let copies and MMAs that
// are already in flight land before the CTA releases its memory.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return;
  }
}

template <int D, int NQT, int NST, int BN, bool kAddMask, bool kLse>
__global__ void __launch_bounds__(Cfg<D, NQT, NST, BN>::kThreads, Cfg<D, NQT, NST, BN>::kMinBlocks)
    sdpa_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const SdpaParams p) {
  using C = Cfg<D, NQT, NST, BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffMisc + 4);
  auto bar = [base](int i) -> uint32_t { return base + C::kOffBar + 8u * i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtl ctl{abort_flag, p.err, p.limit_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(C::bQ), 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar(C::bKF(s)), 1);
      mbar_init(bar(C::bKE(s)), 1);
      mbar_init(bar(C::bVF(s)), 1);
      mbar_init(bar(C::bVE(s)), 1);
    }
    for (int t = 0; t < NQT; ++t) {
      mbar_init(bar(C::bS(t)), 1);
      mbar_init(bar(C::bP(t)), kBlockM);
      mbar_init(bar(C::bO(t)), 1);
    }
    mbar_init(bar(C::bDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc<C::kTmemCols>(smem_u32(tmem_slot));
    tmem_relinquish();
  }
  if (warp == C::kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  // ---- which (b, h, query block) this CTA computes.  Head-major order:
  // consecutive CTAs take the query blocks of one head, so the CTAs resident
  // at any moment share one or two heads' K/V in L2 instead of streaming
  // every head's K/V from HBM.  Causal blocks of a head go longest-first so
  // the short ones fill the tail of the grid.
  const bool causal = (p.mask_kind & MHA_MASK_CAUSAL) != 0;
  const bool padded = (p.mask_kind & MHA_MASK_KEY_PADDING) != 0;
  const int bh = static_cast<int>(blockIdx.x) / p.num_q_blocks;
  const int blk = static_cast<int>(blockIdx.x) - bh * p.num_q_blocks;
  const int qb = causal ? (p.num_q_blocks - 1 - blk) : blk;
  const int b = bh / p.H;
  const int h = bh - b * p.H;
  const int q0 = qb * (NQT * kBlockM);
  int key_end = p.Lk;  // keys [0, key_end) pass the padding rule
  bool bad_len = false;
  if (padded) {
    const int L = __ldg(p.key_lengths + b);
    if (L < 1 || L > p.Lk) bad_len = true;
    else key_end = L;
  }
  // key tiles that query tile t walks: up to its own diagonal when causal
  auto n_kv_of = [&](int t) -> int {
    int stop = bad_len ? 0 : key_end;
    if (causal) stop = min(stop, q0 + (t + 1) * kBlockM);
    return (stop + BN - 1) / BN;
  };
  const int n_kv = n_kv_of(NQT - 1);  // the most any tile of this CTA needs
  if (bad_len && threadIdx.x == 0) atomicOr(p.err, kErrKeyLength);

  if (warp == C::kTmaWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_kv > 0) {
      mbar_expect_tx(bar(C::bQ), NQT * C::kQTileBytes);
      for (int t = 0; t < NQT; ++t)
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(base + C::kOffQ + (t * C::KB + kb) * kSub, &tmQ, bar(C::bQ), kb * 64,
                      q0 + t * kBlockM, bh);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % NST;
        const uint32_t ph = (j / NST) & 1;
        if (!mbar_wait(bar(C::bKE(st)), ph ^ 1u, ctl)) break;
        mbar_expect_tx(bar(C::bKF(st)), C::kKVTileBytes);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(base + C::kOffK + (st * C::KB + kb) * C::kKVBlock, &tmK, bar(C::bKF(st)),
                      kb * 64, j * BN, bh);
        k_issued = j + 1;
        if (!mbar_wait(bar(C::bVE(st)), ph ^ 1u, ctl)) break;
        mbar_expect_tx(bar(C::bVF(st)), C::kKVTileBytes);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(base + C::kOffV + (st * C::KB + kb) * C::kKVBlock, &tmV, bar(C::bVF(st)),
                      kb * 64, j * BN, bh);
        v_issued = j + 1;
      }
      // let every issued copy land before the CTA can exit
      wait_drain(bar(C::bQ), 0, p.limit_ns);
      for (int j = max(0, k_issued - NST); j < k_issued; ++j)
        wait_drain(bar(C::bKF(j % NST)), (j / NST) & 1, p.limit_ns);
      for (int j = max(0, v_issued - NST); j < v_issued; ++j)
        wait_drain(bar(C::bVF(j % NST)), (j / NST) & 1, p.limit_ns);
    }
  } else if (warp == C::kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // Issue order per key tile j: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1).
    // S_t(j+1) overwrites the TMEM columns that P_t(j) occupies; it is
    // issued after PV_t(j) by the same thread, and tcgen05 MMAs of one CTA
    // execute in issue order, so PV_t(j) has read P_t(j) before S_t(j+1)
    // writes.  Each softmax warpgroup thus has two MMAs' time (the other
    // tile's PV and S) between S_t(j+1) landing and P_t(j+1) being needed.
    if (lane == 0 && n_kv > 0) {
      constexpr uint32_t kIdescQK = idesc_bf16_f32(kBlockM, BN, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(kBlockM, D, false, true);
      // Descriptors are built once; per MMA only a compile-time offset (in
      // 16-byte units, the descriptor's address granule) is added, which
      // keeps the single issuing thread off long integer chains.
      const uint64_t q_desc = sdesc_sw128(base + C::kOffQ, 16, 1024);
      const uint64_t k_desc = sdesc_sw128(base + C::kOffK, 16, 1024);
      const uint64_t v_desc = sdesc_sw128(base + C::kOffV, C::kKVBlock, 1024);
      auto issue_qk = [&](int t, int st) {
        const uint64_t qd = q_desc + static_cast<uint64_t>((t * C::kQTileBytes) >> 4);
        const uint64_t kd = k_desc + static_cast<uint64_t>((st * C::kKVTileBytes) >> 4);
        const uint32_t d_tmem = tmem + C::tS(t);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          // 16 elements = 32 bytes inside a 128-byte row; the 64-column blocks
          // are kSub apart in Q and kKVBlock apart in K
          const uint64_t qoff = static_cast<uint64_t>(((ks >> 2) * kSub + (ks & 3) * 32) >> 4);
          const uint64_t koff =
              static_cast<uint64_t>(((ks >> 2) * C::kKVBlock + (ks & 3) * 32) >> 4);
          umma_ss(d_tmem, qd + qoff, kd + koff, kIdescQK, ks > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int st, uint32_t accumulate) {
        const uint64_t vd = v_desc + static_cast<uint64_t>((st * C::kKVTileBytes) >> 4);
        const uint32_t d_tmem = tmem + C::tO(t);
        const uint32_t a_tmem = tmem + C::tS(t);
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          // 16 keys of V = 16 rows of 128 bytes; P: 16 bf16 = 8 TMEM columns
          umma_ts(d_tmem, a_tmem + ks * 8, vd + static_cast<uint64_t>((ks * 16 * 128) >> 4),
                  kIdescPV, ks > 0 ? 1u : accumulate);
        }
      };
      bool ok = mbar_wait(bar(C::bQ), 0, ctl) && mbar_wait(bar(C::bKF(0)), 0, ctl);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < NQT; ++t) {
          issue_qk(t, 0);
          umma_commit(bar(C::bS(t)));
        }
        umma_commit(bar(C::bKE(0)));
      }
      // A query tile whose last key tile is j gets no S(j + 1); its output
      // is complete after PV(j) and its epilogue runs while the other tile
      // of the CTA (causal: the one further down) walks on.
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j % NST;
        const uint32_t ph = (j / NST) & 1;
        const bool more = j + 1 < n_kv;
        const int st1 = (j + 1) % NST;
        const uint32_t ph1 = ((j + 1) / NST) & 1;
        if (!(ok = mbar_wait(bar(C::bVF(st)), ph, ctl))) break;
        bool k_ready = false;
        for (int t = 0; t < NQT && ok; ++t) {
          const int n_t = n_kv_of(t);
          if (j >= n_t) continue;
          if (!(ok = mbar_wait(bar(C::bP(t)), j & 1, ctl))) break;
          tc_fence_after();
          issue_pv(t, st, j > 0 ? 1u : 0u);
          if (j + 1 >= n_t) {
            umma_commit(bar(C::bO(t)));
            continue;
          }
          if (!k_ready && !(ok = mbar_wait(bar(C::bKF(st1)), ph1, ctl))) break;
          k_ready = true;
          issue_qk(t, st1);
          umma_commit(bar(C::bS(t)));
        }
        if (!ok) break;
        if (more) umma_commit(bar(C::bKE(st1)));
        umma_commit(bar(C::bVE(st)));
      }
      // every issued MMA completes before tensor memory is released
      umma_commit(bar(C::bDrain));
      wait_drain(bar(C::bDrain), 0, p.limit_ns);
    }
  } else {
    // --------------------------------------------------- softmax warpgroup
    const int t = warp >> 2;
    const int quarter = warp & 3;  // this warp may touch TMEM lanes [32q, 32q+32)
    const int r = quarter * 32 + lane;
    const int q_row = q0 + t * kBlockM + r;
    const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_bits + C::tS(t);
    const uint32_t tO = tmem + lane_bits + C::tO(t);
    const float sl2 = p.scale_log2;
    // m_ref: the reference maximum (raw score units) that p = 2^((s - m_ref)
    // * sl2) is taken against.  It is raised only when a tile's maximum
    // exceeds it by more than kRescaleLog2 (in log2 units); below that the
    // stale reference is kept and p may reach 2^kRescaleLog2.  O and l share
    // the reference, so O / l is unchanged.
    constexpr float kRescaleLog2 = 8.f;
    float m_ref = -INFINITY;
    float l = 0.f;
    bool ok = true;
    const int n_t = n_kv_of(t);
    for (int j = 0; j < n_t; ++j) {
      if (!(ok = mbar_wait_warp(bar(C::bS(t)), j & 1, ctl))) break;
      tc_fence_after();
      const int k0 = j * BN;
      const bool edge = (k0 + BN > key_end) || (causal && k0 + BN - 1 > q0 + t * kBlockM);
      // visible keys of this row in this tile: columns c <= last
      int last = key_end - 1 - k0;
      if (causal) last = min(last, q_row - k0);
      // S row -> registers (masked)
      auto load_scores = [&](float (&x)[BN]) {
        uint32_t s[BN];
#pragma unroll
        for (int c = 0; c < BN; c += 32)
          tmem_ld32(tS + c, *reinterpret_cast<uint32_t(*)[32]>(&s[c]));
        tmem_ld_wait(s);
#pragma unroll
        for (int c = 0; c < BN; ++c) x[c] = __uint_as_float(s[c]);
        if (edge) {
#pragma unroll
          for (int c = 0; c < BN; ++c) x[c] = c <= last ? x[c] : -INFINITY;
        }
        if constexpr (kAddMask) {
          // additive float mask, in raw-score units (M / scale); -inf blocks
          if (q_row < p.Lq) {
            const float* mrow = p.add_mask + static_cast<int64_t>(b) * p.mask_sb +
                                static_cast<int64_t>(h) * p.mask_sh +
                                static_cast<int64_t>(q_row) * p.Lk + k0;
            const int nvalid = min(BN, p.Lk - k0);
            if (p.mask_vec && nvalid == BN) {
#pragma unroll
              for (int c = 0; c < BN; c += 4) {
                const float4 mv = __ldg(reinterpret_cast<const float4*>(mrow + c));
                x[c] = fmaf(mv.x, p.inv_scale, x[c]);
                x[c + 1] = fmaf(mv.y, p.inv_scale, x[c + 1]);
                x[c + 2] = fmaf(mv.z, p.inv_scale, x[c + 2]);
                x[c + 3] = fmaf(mv.w, p.inv_scale, x[c + 3]);
              }
            } else {
#pragma unroll
              for (int c = 0; c < BN; ++c)
                if (c < nvalid) x[c] = fmaf(__ldg(mrow + c), p.inv_scale, x[c]);
            }
          }
        }
      };
      // tile maximum: eight independent 3-input max chains, then combine
      auto tile_max = [&](const float (&x)[BN]) -> float {
        float m8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmax3(x[i], x[8 + i], x[16 + i]);
#pragma unroll
        for (int c = 24; c < BN - 8; c += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = fmax3(m8[i], x[c + i], x[c + 8 + i]);
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], x[BN - 8 + i]);
        return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]),
                     fmaxf(m8[6], m8[7]));
      };
      // p = 2^(s*sl2 - mb), two at a time with four independent partial sums
      auto exps = [&](const float (&x)[BN], float mb, float2 (&acc)[4], uint32_t (&pk)[BN / 2]) {
        const float2 scale2 = make_float2(sl2, sl2);
        const float2 shift2 = make_float2(-mb, -mb);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < BN / 2; ++c) {
          const float2 e = ffma2(make_float2(x[2 * c], x[2 * c + 1]), scale2, shift2);
          const float2 pp = make_float2(ex2_approx(e.x), ex2_approx(e.y));
          acc[c & 3] = fadd2(acc[c & 3], pp);
          pk[c] = pack_bf16x2(pp.x, pp.y);
        }
      };
      float x[BN];
      float2 acc[4];
      uint32_t pk[BN / 2];
      float alpha = 1.f;
      load_scores(x);
      const float mt = tile_max(x);
      if (mt > m_ref && (m_ref == -INFINITY || (mt - m_ref) * sl2 > kRescaleLog2)) {
        alpha = ex2_approx((m_ref - mt) * sl2);  // 0 when m_ref = -inf
        m_ref = mt;
        l *= alpha;
      }
      exps(x, m_ref == -INFINITY ? 0.f : m_ref * sl2, acc, pk);
      const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
      const float2 a = fadd2(a01, a23);
      l += a.x + a.y;
#pragma unroll
      for (int c = 0; c < BN / 2; c += 32)
        tmem_st32(tS + c, *reinterpret_cast<const uint32_t(*)[32]>(&pk[c]));
      // Rescale the partial output when the reference max moved.  P.V of the
      // previous tile is complete: it was issued before this tile's S, whose
      // commit covers it.  Done after P is stored, when the score registers
      // are free again.
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t o[32];
          tmem_ld32(tO + cb * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tO + cb * 32, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::bP(t)));
    }
    // ------------------------------------------------------------ epilogue
    bool have = ok && n_t > 0;
    if (have) {
      have = mbar_wait_warp(bar(C::bO(t)), 0, ctl);
      tc_fence_after();
    }
    const float inv_l = (have && l > 0.f) ? 1.f / l : 0.f;
    // The backward pass recomputes P = 2^(s * scale_log2 - lse) from this:
    // with p = 2^((s - m_ref) * scale_log2) summing to l, the row's
    // log-sum-exp (base 2) is m_ref * scale_log2 + log2(l); +inf for a row
    // with no visible key, so that its P is 0.
    if constexpr (kLse) {
      if (q_row < p.Lq)
        p.lse[static_cast<size_t>(bh) * p.Lq + q_row] =
            (have && l > 0.f) ? fmaf(m_ref, sl2, log2f(l)) : INFINITY;
    }
    const size_t row_idx = p.ctx_layout
                               ? (static_cast<size_t>(b) * p.Lq + q_row) * p.H + h
                               : static_cast<size_t>(bh) * p.Lq + q_row;
    bool stored = false;
    if constexpr (D == 64) {
      if (!p.out_f32) {
        // A bf16 row of d = 64 is 128 bytes.  The warp's 32 rows go through
        // shared memory (this tile's Q block, free once bO covered its last
        // Q K^T product) so that each store writes four whole rows: 16-byte
        // piece q of row r at slot q ^ (r & 7).
        uint32_t o[64];
        if (have) {
          tmem_ld32(tO, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
          tmem_ld32(tO + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
          tmem_ld_wait(o);
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) o[i] = 0u;
        }
        uint4* stg = reinterpret_cast<uint4*>(gbase + C::kOffQ + t * C::kQTileBytes +
                                              quarter * (32 * 128));
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv_l,
                            __uint_as_float(o[8 * q + 1]) * inv_l);
          v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv_l,
                            __uint_as_float(o[8 * q + 3]) * inv_l);
          v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv_l,
                            __uint_as_float(o[8 * q + 5]) * inv_l);
          v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv_l,
                            __uint_as_float(o[8 * q + 7]) * inv_l);
          stg[lane * 8 + (q ^ (lane & 7))] = v;
        }
        __syncwarp();
        const int q = lane & 7;
#pragma unroll
        for (int g4 = 0; g4 < 8; ++g4) {
          const int rr = 4 * g4 + (lane >> 3);  // the warp's row rr, lane rr's own row
          const uint4 w = stg[rr * 8 + (q ^ (rr & 7))];
          const unsigned long long ri = __shfl_sync(0xffffffffu, static_cast<unsigned long long>(row_idx), rr);
          if (q0 + t * kBlockM + quarter * 32 + rr < p.Lq)
            reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.O) + ri * D)[q] = w;
        }
        stored = true;
      }
    }
#pragma unroll
    for (int cb = 0; cb < D / 32 && !stored; ++cb) {
      uint32_t o[32];
      if (have) {
        tmem_ld32(tO + cb * 32, o);
        tmem_ld_wait(o);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;
      }
      if (q_row < p.Lq) {
        if (p.out_f32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.O) + row_idx * D + cb * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv_l,
                                 __uint_as_float(o[4 * i + 1]) * inv_l,
                                 __uint_as_float(o[4 * i + 2]) * inv_l,
                                 __uint_as_float(o[4 * i + 3]) * inv_l);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.O) + row_idx * D +
                                                cb * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * i + 0]) * inv_l,
                              __uint_as_float(o[8 * i + 1]) * inv_l);
            v.y = pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv_l,
                              __uint_as_float(o[8 * i + 3]) * inv_l);
            v.z = pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv_l,
                              __uint_as_float(o[8 * i + 5]) * inv_l);
            v.w = pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv_l,
                              __uint_as_float(o[8 * i + 7]) * inv_l);
            dst[i] = v;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::kMmaWarp) tmem_dealloc<C::kTmemCols>(tmem);
}

template <int D, int NQT, int NST, bool kAddMask, bool kLse = false, int BN = 128>
cudaError_t launch_impl(const SdpaArgs& a, const DeviceCtl& ctl) {
  using C = Cfg<D, NQT, NST, BN>;
  CUtensorMap maps[3];
  const void* ptrs[3] = {a.Q, a.K, a.V};
  const int lens[3] = {a.Lq, a.Lk, a.Lk};
  for (int i = 0; i < 3; ++i) {
    const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(lens[i]),
                              static_cast<uint64_t>(a.B) * a.H};
    const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2,
                                 static_cast<uint64_t>(lens[i]) * D * 2};
    const uint32_t box[3] = {64, i == 0 ? 128u : static_cast<uint32_t>(BN), 1};
    if (!encode_tensor_map(&maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                           const_cast<void*>(ptrs[i]), dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  SdpaParams p{};
  p.O = a.O;
  p.key_lengths = a.key_lengths;
  p.err = ctl.err;
  p.limit_ns = ctl.limit_ns;
  p.B = a.B;
  p.H = a.H;
  p.Lq = a.Lq;
  p.Lk = a.Lk;
  p.num_q_blocks = (a.Lq + NQT * kBlockM - 1) / (NQT * kBlockM);
  p.mask_kind = a.mask_kind;
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.out_f32 = a.out_dtype == MHA_F32 ? 1 : 0;
  p.ctx_layout = a.ctx_layout ? 1 : 0;
  p.add_mask = a.add_mask;
  p.mask_sb = a.mask_sb;
  p.mask_sh = a.mask_sh;
  p.inv_scale = 1.f / a.scale;
  p.lse = a.lse;
  p.mask_vec = a.add_mask && (reinterpret_cast<uintptr_t>(a.add_mask) & 15u) == 0 &&
               a.Lk % 4 == 0 && a.mask_sb % 4 == 0 && a.mask_sh % 4 == 0;
  const long long grid = static_cast<long long>(p.num_q_blocks) * a.B * a.H;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  auto kern = sdpa_fwd_bf16_kernel<D, NQT, NST, BN, kAddMask, kLse>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;

  kern<<<static_cast<unsigned>(grid), C::kThreads, C::kSmemBytes, a.stream>>>(maps[0], maps[1],
                                                                              maps[2], p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sdpa_bf16(const SdpaArgs& a, const DeviceCtl& ctl) {
  // Two query tiles per CTA share every K/V tile (half the K/V traffic per
  // query row); a single tile when there are too few rows to fill two.  At
  // d = 64 every two-tile form (plain, additive mask, row log-sum-exp) uses
  // 64-key tiles, so the three give bit-identical outputs.
  const bool two = a.Lq > kBlockM;
  if (a.add_mask) {
    if (a.d == 64)
      return two ? launch_impl<64, 2, 3, true, false, 64>(a, ctl)
                 : launch_impl<64, 1, 3, true>(a, ctl);
    if (a.d == 128)
      return two ? launch_impl<128, 2, 2, true>(a, ctl) : launch_impl<128, 1, 2, true>(a, ctl);
    return cudaErrorInvalidValue;
  }
  // the row log-sum-exp store is a separate instantiation, so the plain
  // forward's code is unchanged by it
  if (a.lse != nullptr) {
    if (a.d == 64)
      return two ? launch_impl<64, 2, 3, false, true, 64>(a, ctl)
                 : launch_impl<64, 1, 3, false, true>(a, ctl);
    if (a.d == 128)
      return two ? launch_impl<128, 2, 2, false, true>(a, ctl)
                 : launch_impl<128, 1, 2, false, true>(a, ctl);
    return cudaErrorInvalidValue;
  }
  // d = 64: two query tiles per CTA on 64-key tiles, so that a query tile
  // needs 128 TMEM columns and two CTAs share an SM: four query tiles (four
  // softmax/MMA chains) per SM instead of two.  A lone query tile keeps the
  // 128-key form, two CTAs per SM (measured faster for Lq <= 128).
  if (a.d == 64 && two) return launch_impl<64, 2, 3, false, false, 64>(a, ctl);
  if (a.d == 64 && a.Lk <= 2048) return launch_impl<64, 1, 2, false>(a, ctl);
  if (a.d == 64) return launch_impl<64, 1, 3, false>(a, ctl);
  if (a.d == 128)
    return two ? launch_impl<128, 2, 2, false>(a, ctl) : launch_impl<128, 1, 2, false>(a, ctl);
  return cudaErrorInvalidValue;
}

}  // namespace mha
