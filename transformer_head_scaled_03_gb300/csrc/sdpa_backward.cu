// sdpa_backward.cu -- the backward pass of scaled dot-product attention
// (training), bf16 in, fp32 accumulate, on sm_103a tcgen05 tensor cores.
//
// Given dO = dL/dO for O = softmax(S) V, S = scale Q K^T + M, and the row
// log-sum-exp of the forward pass (lse, base 2):
//   P    = 2^(S log2(e) - lse)               recomputed per tile
//   dV   = P^T dO
//   dP   = dO V^T
//   dS   = P (dP - D),  D_i = <dO_i, O_i>    (= sum_j P_ij dP_ij)
//   dK   = scale dS^T Q
//   dQ   = scale dS K
// (the chain rule through the attention formula of "How Transformers Work"
// (worksonmygpu.com), "Scaled dot-product attention"; the softmax gradient
// "32 Transformer" (ml-canon-en), "Why we divide by sqrt(dk)", discusses).
//
// dK and dV sum over queries, dQ over keys.  Two kernels each keep their sum
// in tensor memory, so no gradient is ever accumulated in global memory:
//
// sdpa_bwd_dkdv_kernel: CTA = 128 keys of one (b, h), walking the query
// tiles that can see them; keys on the TMEM lanes.
//   S^T  = K Q^T, dP^T = V dO^T    M 128 keys, N 128 queries, K = d
//   P^T  -> bf16 pairs: queries 0-63 in S^T cols 0-31, 64-127 in cols 64-95
//   dS^T -> bf16 pairs in the same places of dP^T
//   dV  += P^T dO, dK += dS^T Q   A from TMEM, B MN-major
//
// sdpa_bwd_dq_kernel: CTA = 128 queries of one (b, h), walking the key tiles
// they can see; queries on the TMEM lanes (the forward's orientation).
//   S    = Q K^T, dP = dO V^T     M 128 queries, N 128 keys, K = d
//   dS   -> bf16 pairs over the S tile it came from (double-buffered S)
//   dQ  += dS K                   A = dS from TMEM, B = K (MN-major)
//
// In both, warps 0-7 compute P and dS: warp w takes TMEM lanes
// 32 (w % 4) .. +31 and one 64-column half (w / 4) of the tile, two such
// warps per SM sub-partition, each writing only inside the columns it alone
// reads.  Warp 8 loads (TMA), warp 9 issues the MMAs.  P and dS cost a
// second pass over the exponentials (7 products in all instead of 5), which
// buys away the fp32 reductions of a dQ summed across CTAs in global memory.
// Every wait is bounded; waiting threads sleep on the barrier.
#include <math.h>
#include <stdint.h>

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "ptx_cluster.cuh"

namespace mha {
namespace {

constexpr int kTile = 128;       // keys or queries per tile
constexpr int kSub = 16384;      // one 128-row x 64-column bf16 box
constexpr int kCompWarps = 8;    // warps 0-7
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxSmem = 232448;  // per-CTA opt-in limit

// ---------------------------------------------------------------- dK, dV
template <int D>
struct CfgKV {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int KB = D / 64;
  static constexpr int kTileBytes = KB * kSub;   // a 128-row tile of K, V, Q or dO
  static constexpr int NST = D == 128 ? 2 : 4;    // Q/dO stages
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;                 // NST stages
  static constexpr int kOffDO = kOffQ + NST * kTileBytes;          // NST stages
  static constexpr int kOffRow = kOffDO + NST * kTileBytes;        // NST x {-lse[128], -D[128]}
  static constexpr int kOffBar = kOffRow + NST * 1024;
  static constexpr int bKV = 0;
  __host__ __device__ static constexpr int bFull(int s) { return 1 + s; }
  __host__ __device__ static constexpr int bEmpty(int s) { return 1 + NST + s; }
  static constexpr int bS = 1 + 2 * NST;   // S^T(j) complete
  static constexpr int bDP = bS + 1;       // dP^T(j) complete
  static constexpr int bP0 = bS + 2;       // P^T(j) queries 0-63 in TMEM
  static constexpr int bP1 = bS + 3;       // P^T(j) queries 64-127 in TMEM
  static constexpr int bDS = bS + 4;       // dS^T(j) in TMEM
  static constexpr int bFinal = bS + 5;
  static constexpr int bDrain = bS + 6;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kUsed = kOffMisc + 16;
  static_assert(kUsed <= kMaxSmem, "shared memory");
  static constexpr int kSmemBytes = kUsed + 1024 <= kMaxSmem ? kUsed + 1024 : kMaxSmem;
  static constexpr uint32_t tS = 0, tDP = 128, tDV = 256, tDK = 256 + D;
};

// ---------------------------------------------------------------- dQ
template <int D>
struct CfgQ {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int KB = D / 64;
  static constexpr int kTileBytes = KB * kSub;
  static constexpr int NK = D == 128 ? 3 : 4;     // K stages (read by S and by dQ)
  static constexpr int NV = D == 128 ? 2 : 3;     // V stages (read by dP)
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kOffQ + kTileBytes;
  static constexpr int kOffK = kOffDO + kTileBytes;                // NK stages
  static constexpr int kOffV = kOffK + NK * kTileBytes;            // NV stages
  static constexpr int kOffBar = kOffV + NV * kTileBytes;
  static constexpr int bQ = 0;                                     // Q, dO loaded
  __host__ __device__ static constexpr int bKFull(int s) { return 1 + s; }
  __host__ __device__ static constexpr int bKEmpty(int s) { return 1 + NK + s; }
  __host__ __device__ static constexpr int bVFull(int s) { return 1 + 2 * NK + s; }
  __host__ __device__ static constexpr int bVEmpty(int s) { return 1 + 2 * NK + NV + s; }
  static constexpr int bS0 = 1 + 2 * NK + 2 * NV;   // S(i) complete in buffer i % 2: bS0 + i % 2
  static constexpr int bDP = bS0 + 2;               // dP(i) complete
  static constexpr int bDPR = bS0 + 3;              // dP(i) read out of TMEM
  static constexpr int bDS0 = bS0 + 4;              // dS(i) in TMEM: bDS0 + i % 2
  static constexpr int bFinal = bS0 + 6;
  static constexpr int bDrain = bS0 + 7;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kUsed = kOffMisc + 16;
  static_assert(kUsed <= kMaxSmem, "shared memory");
  static constexpr int kSmemBytes = kUsed + 1024 <= kMaxSmem ? kUsed + 1024 : kMaxSmem;
  static constexpr uint32_t tS0 = 0, tDP = 256, tDQ = 384;   // S buffers at 0 and 128
};

struct BwdParams {
  const float* lse;     // [B, H, Lq], base 2
  const float* dsum;    // [B, H, Lq], D_i = <dO_i, O_i>
  float* dq;            // [B, H, Lq, d] fp32
  void* dk;             // [B, H, Lk, d]
  void* dv;
  int B, H, Lq, Lk;
  int num_k_tiles, num_q_tiles;
  int mask_kind;
  const int32_t* key_lengths;
  float scale;
  float scale_log2;
  int out_f32;
  unsigned* err;
  uint64_t limit_ns;
};

__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return;
  }
}

// try_wait with a suspend-time hint: a thread whose phase is not complete
// sleeps on the barrier (up to 20 us) instead of re-polling.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(20000u)
      : "memory");
  return done != 0;
}

// Bounded wait that sleeps between polls: false when the CTA is aborting or
// the wait ran past its limit (then the abort flag and the timeout bit are
// set), as mbar_wait.
__device__ __forceinline__ bool mbar_wait_s(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (*ctl.abort_flag) return false;
    if (global_timer_ns() - t0 > ctl.limit_ns) {
      *ctl.abort_flag = 1;
      atomicOr(ctl.err, kErrTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait_s_warp(uint32_t bar, uint32_t parity,
                                                 const WaitCtl& ctl) {
  const bool ok = mbar_wait_s(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}

// 4 consecutive values of a per-row array from row q on, negated; `fill`
// past Lq.  One float4 only when every head's row starts 16-byte aligned
// (Lq % 4 == 0).
__device__ __forceinline__ float4 load_row4_neg(const float* row, int q, int Lq, float fill) {
  if ((Lq & 3) == 0 && q + 3 < Lq) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(row + q));
    return make_float4(-v.x, -v.y, -v.z, -v.w);
  }
  return make_float4(q < Lq ? -__ldg(row + q) : fill, q + 1 < Lq ? -__ldg(row + q + 1) : fill,
                     q + 2 < Lq ? -__ldg(row + q + 2) : fill,
                     q + 3 < Lq ? -__ldg(row + q + 3) : fill);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// NCB x 32 fp32 columns from TMEM (whole warp; zeros when `have` is false),
// times `mul`, stored at out + row for a live row.
template <int NCB>
__device__ __forceinline__ void store_row(uint32_t taddr, bool have, float mul, void* out,
                                          size_t row, bool live, bool f32) {
#pragma unroll
  for (int cb = 0; cb < NCB; ++cb) {
    uint32_t g[32];
    if (have) {
      tmem_ld32(taddr + cb * 32, g);
      tmem_ld_wait(g);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) g[i] = 0u;
    }
    if (!live) continue;
    if (f32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + row + cb * 32);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dst[i] = make_float4(__uint_as_float(g[4 * i]) * mul, __uint_as_float(g[4 * i + 1]) * mul,
                             __uint_as_float(g[4 * i + 2]) * mul,
                             __uint_as_float(g[4 * i + 3]) * mul);
    } else {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + row + cb * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        dst[i] = make_uint4(
            pack_bf16x2(__uint_as_float(g[8 * i]) * mul, __uint_as_float(g[8 * i + 1]) * mul),
            pack_bf16x2(__uint_as_float(g[8 * i + 2]) * mul, __uint_as_float(g[8 * i + 3]) * mul),
            pack_bf16x2(__uint_as_float(g[8 * i + 4]) * mul, __uint_as_float(g[8 * i + 5]) * mul),
            pack_bf16x2(__uint_as_float(g[8 * i + 6]) * mul, __uint_as_float(g[8 * i + 7]) * mul));
    }
  }
}

// 2^(s sl2 + nl) for 64 scores, as 32 bf16 pairs; columns c >= lim are
// blocked (p = 0): lim >= 64 takes no mask at all.  nl is the negated
// log-sum-exp, per column (`nl_col`) or one value (`nl_row`).
template <bool kPerColumn>
__device__ __forceinline__ void exp_tile64(const uint32_t (&s)[64], float2 sl2,
                                           const float* nl_col, float nl_row, int lim,
                                           uint32_t (&pk)[32]) {
  if (lim >= 64) {
#pragma unroll
    for (int c = 0; c < 64; c += 4) {
      float2 n01, n23;
      if constexpr (kPerColumn) {
        const float4 nl = *reinterpret_cast<const float4*>(nl_col + c);
        n01 = make_float2(nl.x, nl.y);
        n23 = make_float2(nl.z, nl.w);
      } else {
        n01 = n23 = make_float2(nl_row, nl_row);
      }
      const float2 x01 =
          ffma2(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2, n01);
      const float2 x23 =
          ffma2(make_float2(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3])), sl2, n23);
      pk[c / 2] = pack_bf16x2(ex2_approx(x01.x), ex2_approx(x01.y));
      pk[c / 2 + 1] = pack_bf16x2(ex2_approx(x23.x), ex2_approx(x23.y));
    }
  } else if (lim <= 0) {
#pragma unroll
    for (int c = 0; c < 32; ++c) pk[c] = 0u;
  } else {
#pragma unroll
    for (int c = 0; c < 64; c += 2) {
      float2 n01;
      if constexpr (kPerColumn) {
        n01 = *reinterpret_cast<const float2*>(nl_col + c);
      } else {
        n01 = make_float2(nl_row, nl_row);
      }
      const float2 x =
          ffma2(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2, n01);
      pk[c / 2] = pack_bf16x2(c < lim ? ex2_approx(x.x) : 0.f, c + 1 < lim ? ex2_approx(x.y) : 0.f);
    }
  }
}

// dS = P (dP + nd) for 32 columns from column c0 of the half: dp holds the
// 32 dP values, pk the half's P pairs; nd per column or one value.
template <bool kPerColumn>
__device__ __forceinline__ void ds_tile32(const uint32_t (&dp)[32], const uint32_t (&pk)[32],
                                          int c0, const float* nd_col, float nd_row,
                                          uint32_t (&dsk)[16]) {
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    float2 n01, n23;
    if constexpr (kPerColumn) {
      const float4 nd = *reinterpret_cast<const float4*>(nd_col + c0 + i);
      n01 = make_float2(nd.x, nd.y);
      n23 = make_float2(nd.z, nd.w);
    } else {
      n01 = n23 = make_float2(nd_row, nd_row);
    }
    const float2 d01 = fadd2(make_float2(__uint_as_float(dp[i]), __uint_as_float(dp[i + 1])), n01);
    const float2 d23 =
        fadd2(make_float2(__uint_as_float(dp[i + 2]), __uint_as_float(dp[i + 3])), n23);
    const float2 s01 = fmul2(unpack_bf16x2(pk[(c0 + i) / 2]), d01);
    const float2 s23 = fmul2(unpack_bf16x2(pk[(c0 + i) / 2 + 1]), d23);
    dsk[i / 2] = pack_bf16x2(s01.x, s01.y);
    dsk[i / 2 + 1] = pack_bf16x2(s23.x, s23.y);
  }
}

// ============================================================ dK, dV kernel
// 10 warps: three on two of the sub-partitions (16K registers each), so at
// most 168 registers per thread.
template <int D>
__global__ void __maxnreg__(168)
    sdpa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmDO, const BwdParams p) {
  using C = CfgKV<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  if (base - raw + C::kUsed > static_cast<uint32_t>(C::kSmemBytes)) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemLayout);
    return;
  }
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffMisc + 4);
  auto bar = [base](int i) -> uint32_t { return base + C::kOffBar + 8u * i; };
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtl ctl{abort_flag, p.err, p.limit_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(C::bKV), 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar(C::bFull(s)), 1);
      mbar_init(bar(C::bEmpty(s)), 1);
    }
    mbar_init(bar(C::bS), 1);
    mbar_init(bar(C::bDP), 1);
    mbar_init(bar(C::bP0), 128);
    mbar_init(bar(C::bP1), 128);
    mbar_init(bar(C::bDS), 32 * kCompWarps);
    mbar_init(bar(C::bFinal), 1);
    mbar_init(bar(C::bDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc<kTmemCols>(smem_u32(tmem_slot));
    tmem_relinquish();
  }
  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  // this CTA's (b, h) and key tile: head-major, so the CTAs resident at once
  // share a head's Q and dO in L2; causal key tiles go from the first (which
  // sees the most query tiles) to the last
  const bool causal = (p.mask_kind & MHA_MASK_CAUSAL) != 0;
  const bool padded = (p.mask_kind & MHA_MASK_KEY_PADDING) != 0;
  const int bh = static_cast<int>(blockIdx.x) / p.num_k_tiles;
  const int kt = static_cast<int>(blockIdx.x) - bh * p.num_k_tiles;
  const int b = bh / p.H;
  const int k0 = kt * kTile;
  int len = p.Lk;
  bool bad_len = false;
  if (padded) {
    len = __ldg(p.key_lengths + b);
    if (len < 1 || len > p.Lk) bad_len = true;
  }
  if (bad_len && kt == 0 && threadIdx.x == 0) atomicOr(p.err, kErrKeyLength);
  const int qt_begin = causal ? k0 / kTile : 0;
  const int n_qt = (bad_len || k0 >= len) ? 0 : max(0, p.num_q_tiles - qt_begin);

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (n_qt > 0) {
      if (lane == 0) {
        mbar_expect_tx(bar(C::bKV), 2 * C::kTileBytes);
        for (int kb = 0; kb < C::KB; ++kb) {
          tma_load_3d(base + C::kOffK + kb * kSub, &tmK, bar(C::bKV), kb * 64, k0, bh);
          tma_load_3d(base + C::kOffV + kb * kSub, &tmV, bar(C::bKV), kb * 64, k0, bh);
        }
      }
      const float* lse_h = p.lse + static_cast<size_t>(bh) * p.Lq;
      const float* dsum_h = p.dsum + static_cast<size_t>(bh) * p.Lq;
      int issued = 0;
      for (int j = 0; j < n_qt; ++j) {
        const int st = j % C::NST;
        const uint32_t ph = (j / C::NST) & 1;
        if (!mbar_wait_s_warp(bar(C::bEmpty(st)), ph ^ 1u, ctl)) break;
        const int q0 = (qt_begin + j) * kTile;
        // the tile's -lse (-inf past Lq, so P = 0 there) and -D rows, 4 per lane
        float4* rows = reinterpret_cast<float4*>(gbase + C::kOffRow + st * 1024);
        rows[lane] = load_row4_neg(lse_h, q0 + 4 * lane, p.Lq, -INFINITY);
        rows[32 + lane] = load_row4_neg(dsum_h, q0 + 4 * lane, p.Lq, 0.f);
        __syncwarp();  // the lanes' stores precede lane 0's arrive (a release)
        if (lane == 0) {
          mbar_expect_tx(bar(C::bFull(st)), 2 * C::kTileBytes);
          for (int kb = 0; kb < C::KB; ++kb) {
            tma_load_3d(base + C::kOffQ + st * C::kTileBytes + kb * kSub, &tmQ,
                        bar(C::bFull(st)), kb * 64, q0, bh);
            tma_load_3d(base + C::kOffDO + st * C::kTileBytes + kb * kSub, &tmDO,
                        bar(C::bFull(st)), kb * 64, q0, bh);
          }
        }
        issued = j + 1;
      }
      if (lane == 0) {
        wait_drain(bar(C::bKV), 0, p.limit_ns);
        for (int j = max(0, issued - C::NST); j < issued; ++j)
          wait_drain(bar(C::bFull(j % C::NST)), (j / C::NST) & 1, p.limit_ns);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && n_qt > 0) {
      constexpr uint32_t kIdT = idesc_bf16_f32(kTile, kTile, false, false);   // S^T, dP^T
      constexpr uint32_t kIdG = idesc_bf16_f32(kTile, D, false, true);       // dV, dK
      const uint64_t k_desc = sdesc_sw128(base + C::kOffK, 16, 1024);
      const uint64_t v_desc = sdesc_sw128(base + C::kOffV, 16, 1024);
      const uint64_t q_desc = sdesc_sw128(base + C::kOffQ, 16, 1024);
      const uint64_t q_mn = sdesc_sw128(base + C::kOffQ, kSub, 1024);
      const uint64_t do_desc = sdesc_sw128(base + C::kOffDO, 16, 1024);
      const uint64_t do_mn = sdesc_sw128(base + C::kOffDO, kSub, 1024);
      // d-step products of 128-row tiles: 16 elements = 32 bytes in a
      // 128-byte row, 64-column blocks kSub apart
      auto issue_t = [&](uint32_t d_tmem, uint64_t a, uint64_t bd) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t off = static_cast<uint64_t>(((ks >> 2) * kSub + (ks & 3) * 32) >> 4);
          umma_ss(d_tmem, a + off, bd + off, kIdT, ks > 0 ? 1u : 0u);
        }
      };
      // products over the 64 queries of half h: A = bf16 pairs in TMEM at
      // columns 64 h + 8 k (16 queries per step), B MN-major (16 rows of 128
      // bytes per step)
      auto issue_g = [&](uint32_t d_tmem, uint32_t a_tmem, uint64_t bd, int h, bool first) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ts(d_tmem, a_tmem + 64 * h + 8 * k,
                  bd + static_cast<uint64_t>(((64 * h + 16 * k) * 128) >> 4), kIdG,
                  (first && h == 0 && k == 0) ? 0u : 1u);
      };
      auto stage_off = [](int j) {
        return static_cast<uint64_t>(((j % C::NST) * C::kTileBytes) >> 4);
      };
      bool ok = mbar_wait_s(bar(C::bKV), 0, ctl) && mbar_wait_s(bar(C::bFull(0)), 0, ctl);
      if (ok) {
        tc_fence_after();
        issue_t(tmem + C::tS, k_desc, q_desc);
        umma_commit(bar(C::bS));
        issue_t(tmem + C::tDP, v_desc, do_desc);
        umma_commit(bar(C::bDP));
      }
      for (int j = 0; ok && j < n_qt; ++j) {
        const uint32_t par = j & 1;
        const uint64_t soff = stage_off(j);
        const bool more = j + 1 < n_qt;
        // dV += P^T dO, each half as soon as its warps stored it
        if (!(ok = mbar_wait_s(bar(C::bP0), par, ctl))) break;
        tc_fence_after();
        issue_g(tmem + C::tDV, tmem + C::tS, do_mn + soff, 0, j == 0);
        if (!(ok = mbar_wait_s(bar(C::bP1), par, ctl))) break;
        tc_fence_after();
        issue_g(tmem + C::tDV, tmem + C::tS, do_mn + soff, 1, j == 0);
        // S^T of the next tile over the S columns: P^T was read by the
        // products just issued (MMAs run in issue order)
        if (more) {
          const int j1 = j + 1;
          if (!(ok = mbar_wait_s(bar(C::bFull(j1 % C::NST)), (j1 / C::NST) & 1, ctl))) break;
          tc_fence_after();
          issue_t(tmem + C::tS, k_desc, q_desc + stage_off(j1));
          umma_commit(bar(C::bS));
        }
        if (!(ok = mbar_wait_s(bar(C::bDS), par, ctl))) break;
        tc_fence_after();
        issue_g(tmem + C::tDK, tmem + C::tDP, q_mn + soff, 0, j == 0);
        issue_g(tmem + C::tDK, tmem + C::tDP, q_mn + soff, 1, j == 0);
        umma_commit(bar(C::bEmpty(j % C::NST)));
        // dP^T of the next tile over dS^T, which dK just read
        if (more) {
          issue_t(tmem + C::tDP, v_desc, do_desc + stage_off(j + 1));
          umma_commit(bar(C::bDP));
        }
      }
      umma_commit(bar(C::bFinal));
      umma_commit(bar(C::bDrain));
      wait_drain(bar(C::bDrain), 0, p.limit_ns);
    }
  } else {
    // ------------------------- P and dS (lane = a key, half = 64 queries)
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int L = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int key = k0 + L;
    const bool key_live = key < len;
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    bool ok = true;
    for (int j = 0; j < n_qt; ++j) {
      const int st = j % C::NST;
      const uint32_t par = j & 1;
      const int qh = (qt_begin + j) * kTile + half * 64;   // first query of this half
      const float* nrow = reinterpret_cast<const float*>(gbase + C::kOffRow + st * 1024);
      if (!(ok = mbar_wait_s_warp(bar(C::bS), par, ctl))) break;
      if (!(ok = mbar_wait_s_warp(bar(C::bFull(st)), (j / C::NST) & 1, ctl))) break;
      tc_fence_after();
      // ---- P^T of this key over the half's 64 queries, kept as bf16 pairs;
      // query qh + c sees the key when key_live and (not causal or key <= qh + c)
      uint32_t pk[32];
      {
        uint32_t s[64];
        tmem_ld32(tl + C::tS + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld32(tl + C::tS + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_ld_wait(s);
        // visible columns are c >= first; expressed as a limit on 63 - c
        const int first = !key_live ? 64 : (causal ? max(0, key - qh) : 0);
        if (first == 0) {
          exp_tile64<true>(s, sl2, nrow + half * 64, 0.f, 64, pk);
        } else if (first >= 64) {
#pragma unroll
          for (int c = 0; c < 32; ++c) pk[c] = 0u;
        } else {
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const float2 nl = *reinterpret_cast<const float2*>(nrow + half * 64 + c);
            const float2 x =
                ffma2(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2, nl);
            pk[c / 2] = pack_bf16x2(c >= first ? ex2_approx(x.x) : 0.f,
                                    c + 1 >= first ? ex2_approx(x.y) : 0.f);
          }
        }
        // queries of half h -> bf16 pairs at columns 64 h .. 64 h + 31 (their
        // S^T values are in registers; the other half's warps read only
        // columns 64 (1 - h) ..).  Reconverge before the collective store.
        __syncwarp();
        tmem_st32(tl + C::tS + half * 64, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(half == 0 ? C::bP0 : C::bP1));
      }
      // ---- dS^T = P^T (dP^T - D) over the half, 32 queries at a time; bf16
      // pairs into TMEM at dP^T columns 64 h .. (already read)
      if (!(ok = mbar_wait_s_warp(bar(C::bDP), par, ctl))) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t dp[32];
        tmem_ld32(tl + C::tDP + half * 64 + cc * 32, dp);
        tmem_ld_wait(dp);
        uint32_t dsk[16];
        ds_tile32<true>(dp, pk, cc * 32, nrow + 128 + half * 64, 0.f, dsk);
        tmem_st16(tl + C::tDP + half * 64 + cc * 16, dsk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::bDS));
    }
    // ---- epilogue: half h writes columns [h d/2, (h + 1) d/2) of dV and dK
    bool have = ok && n_qt > 0;
    if (have) {
      have = mbar_wait_s_warp(bar(C::bFinal), 0, ctl);
      tc_fence_after();
    }
    const size_t row = (static_cast<size_t>(bh) * p.Lk + key) * D + half * (D / 2);
    store_row<D / 64>(tl + C::tDV + half * (D / 2), have, 1.f, p.dv, row, key < p.Lk,
                      p.out_f32 != 0);
    store_row<D / 64>(tl + C::tDK + half * (D / 2), have, p.scale, p.dk, row, key < p.Lk,
                      p.out_f32 != 0);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc<kTmemCols>(tmem);
}

// ================================================================ dQ kernel
template <int D>
__global__ void __maxnreg__(168)
    sdpa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmDO, const BwdParams p) {
  using C = CfgQ<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  if (base - raw + C::kUsed > static_cast<uint32_t>(C::kSmemBytes)) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemLayout);
    return;
  }
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffMisc + 4);
  auto bar = [base](int i) -> uint32_t { return base + C::kOffBar + 8u * i; };
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtl ctl{abort_flag, p.err, p.limit_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(C::bQ), 1);
    for (int s = 0; s < C::NK; ++s) {
      mbar_init(bar(C::bKFull(s)), 1);
      mbar_init(bar(C::bKEmpty(s)), 1);
    }
    for (int s = 0; s < C::NV; ++s) {
      mbar_init(bar(C::bVFull(s)), 1);
      mbar_init(bar(C::bVEmpty(s)), 1);
    }
    mbar_init(bar(C::bS0), 1);
    mbar_init(bar(C::bS0 + 1), 1);
    mbar_init(bar(C::bDP), 1);
    mbar_init(bar(C::bDPR), 32 * kCompWarps);
    mbar_init(bar(C::bDS0), 32 * kCompWarps);
    mbar_init(bar(C::bDS0 + 1), 32 * kCompWarps);
    mbar_init(bar(C::bFinal), 1);
    mbar_init(bar(C::bDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc<kTmemCols>(smem_u32(tmem_slot));
    tmem_relinquish();
  }
  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  // this CTA's (b, h) and query tile: head-major; causal query tiles go from
  // the last (which sees the most key tiles) to the first
  const bool causal = (p.mask_kind & MHA_MASK_CAUSAL) != 0;
  const bool padded = (p.mask_kind & MHA_MASK_KEY_PADDING) != 0;
  const int bh = static_cast<int>(blockIdx.x) / p.num_q_tiles;
  const int r = static_cast<int>(blockIdx.x) - bh * p.num_q_tiles;
  const int qt = causal ? p.num_q_tiles - 1 - r : r;
  const int b = bh / p.H;
  const int q0 = qt * kTile;
  int len = p.Lk;
  bool bad_len = false;
  if (padded) {
    len = __ldg(p.key_lengths + b);
    if (len < 1 || len > p.Lk) bad_len = true;
  }
  if (bad_len && r == 0 && threadIdx.x == 0) atomicOr(p.err, kErrKeyLength);
  const int n_len = (len + kTile - 1) / kTile;
  const int n_kt = bad_len ? 0 : (causal ? min(qt + 1, n_len) : n_len);

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_kt > 0) {
      mbar_expect_tx(bar(C::bQ), 2 * C::kTileBytes);
      for (int kb = 0; kb < C::KB; ++kb) {
        tma_load_3d(base + C::kOffQ + kb * kSub, &tmQ, bar(C::bQ), kb * 64, q0, bh);
        tma_load_3d(base + C::kOffDO + kb * kSub, &tmDO, bar(C::bQ), kb * 64, q0, bh);
      }
      // K runs up to NK tiles ahead, V up to NV: each stage frees as soon as
      // its last reader (dQ for K, dP for V) has completed
      int kissued = 0, vissued = 0;
      bool ok = true;
      for (int i = 0; ok && i < n_kt; ++i) {
        const int sk = i % C::NK;
        if (!(ok = mbar_wait_s(bar(C::bKEmpty(sk)), ((i / C::NK) & 1) ^ 1u, ctl))) break;
        mbar_expect_tx(bar(C::bKFull(sk)), C::kTileBytes);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(base + C::kOffK + sk * C::kTileBytes + kb * kSub, &tmK, bar(C::bKFull(sk)),
                      kb * 64, i * kTile, bh);
        kissued = i + 1;
        const int sv = i % C::NV;
        if (!(ok = mbar_wait_s(bar(C::bVEmpty(sv)), ((i / C::NV) & 1) ^ 1u, ctl))) break;
        mbar_expect_tx(bar(C::bVFull(sv)), C::kTileBytes);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(base + C::kOffV + sv * C::kTileBytes + kb * kSub, &tmV, bar(C::bVFull(sv)),
                      kb * 64, i * kTile, bh);
        vissued = i + 1;
      }
      wait_drain(bar(C::bQ), 0, p.limit_ns);
      for (int i = max(0, kissued - C::NK); i < kissued; ++i)
        wait_drain(bar(C::bKFull(i % C::NK)), (i / C::NK) & 1, p.limit_ns);
      for (int i = max(0, vissued - C::NV); i < vissued; ++i)
        wait_drain(bar(C::bVFull(i % C::NV)), (i / C::NV) & 1, p.limit_ns);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && n_kt > 0) {
      constexpr uint32_t kIdT = idesc_bf16_f32(kTile, kTile, false, false);   // S, dP
      constexpr uint32_t kIdG = idesc_bf16_f32(kTile, D, false, true);       // dQ
      const uint64_t q_desc = sdesc_sw128(base + C::kOffQ, 16, 1024);
      const uint64_t do_desc = sdesc_sw128(base + C::kOffDO, 16, 1024);
      const uint64_t k_desc = sdesc_sw128(base + C::kOffK, 16, 1024);
      const uint64_t k_mn = sdesc_sw128(base + C::kOffK, kSub, 1024);
      const uint64_t v_desc = sdesc_sw128(base + C::kOffV, 16, 1024);
      auto koff = [](int i) {
        return static_cast<uint64_t>(((i % C::NK) * C::kTileBytes) >> 4);
      };
      auto voff = [](int i) {
        return static_cast<uint64_t>(((i % C::NV) * C::kTileBytes) >> 4);
      };
      auto issue_t = [&](uint32_t d_tmem, uint64_t a, uint64_t bd) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t off = static_cast<uint64_t>(((ks >> 2) * kSub + (ks & 3) * 32) >> 4);
          umma_ss(d_tmem, a + off, bd + off, kIdT, ks > 0 ? 1u : 0u);
        }
      };
      auto issue_s = [&](int i) -> bool {
        if (!mbar_wait_s(bar(C::bKFull(i % C::NK)), (i / C::NK) & 1, ctl)) return false;
        tc_fence_after();
        issue_t(tmem + C::tS0 + (i & 1) * kTile, q_desc, k_desc + koff(i));
        umma_commit(bar(C::bS0 + (i & 1)));
        return true;
      };
      auto issue_dp = [&](int i) -> bool {
        if (!mbar_wait_s(bar(C::bVFull(i % C::NV)), (i / C::NV) & 1, ctl)) return false;
        tc_fence_after();
        issue_t(tmem + C::tDP, do_desc, v_desc + voff(i));
        umma_commit(bar(C::bDP));
        umma_commit(bar(C::bVEmpty(i % C::NV)));   // V(i) is read by dP(i) only
        return true;
      };
      bool ok = mbar_wait_s(bar(C::bQ), 0, ctl) && issue_s(0) && issue_dp(0) &&
                (n_kt < 2 || issue_s(1));
      for (int i = 0; ok && i < n_kt; ++i) {
        const int bsel = i & 1;
        // dP of the next tile as soon as this one has been read out of TMEM
        if (i + 1 < n_kt) {
          if (!(ok = mbar_wait_s(bar(C::bDPR), i & 1, ctl))) break;
          tc_fence_after();
          if (!(ok = issue_dp(i + 1))) break;
        }
        // dQ += dS K: A = dS pairs in the S buffer (16 keys = 8 columns per
        // step), B = K MN-major (16 rows of 128 bytes per step)
        if (!(ok = mbar_wait_s(bar(C::bDS0 + bsel), (i >> 1) & 1, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks) {
          const int h = ks >> 2, k = ks & 3;
          umma_ts(tmem + C::tDQ, tmem + C::tS0 + bsel * kTile + 64 * h + 8 * k,
                  k_mn + koff(i) + static_cast<uint64_t>(((64 * h + 16 * k) * 128) >> 4), kIdG,
                  (i == 0 && ks == 0) ? 0u : 1u);
        }
        umma_commit(bar(C::bKEmpty(i % C::NK)));
        // S of the tile after next into this buffer: dS was just read by the
        // dQ products (issue order)
        if (i + 2 < n_kt && !(ok = issue_s(i + 2))) break;
      }
      umma_commit(bar(C::bFinal));
      umma_commit(bar(C::bDrain));
      wait_drain(bar(C::bDrain), 0, p.limit_ns);
    }
  } else {
    // ---------------------- P and dS (lane = a query, half = 64 keys)
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int q = q0 + quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    // -lse (-inf past Lq: P = 0) and -D of this thread's query
    const size_t qrow = static_cast<size_t>(bh) * p.Lq + q;
    const float nl = q < p.Lq ? -__ldg(p.lse + qrow) : -INFINITY;
    const float nd = q < p.Lq ? -__ldg(p.dsum + qrow) : 0.f;
    bool ok = true;
    for (int i = 0; i < n_kt; ++i) {
      const int bsel = i & 1;
      const uint32_t tsb = C::tS0 + bsel * kTile + half * 64;
      const int kh = i * kTile + half * 64;   // first key of this half
      if (!(ok = mbar_wait_s_warp(bar(C::bS0 + bsel), (i >> 1) & 1, ctl))) break;
      tc_fence_after();
      // ---- P of this query over the half's 64 keys, kept as bf16 pairs:
      // key kh + c is visible when c < lim
      uint32_t pk[32];
      {
        uint32_t s[64];
        tmem_ld32(tl + tsb, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld32(tl + tsb + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_ld_wait(s);
        int lim = len - kh;
        if (causal) lim = min(lim, q - kh + 1);
        exp_tile64<false>(s, sl2, nullptr, nl, lim, pk);
      }
      // ---- dS = P (dP - D) over the half, into the S buffer as bf16 pairs
      // (columns 64 h .. 64 h + 31: read above, and only by this half)
      if (!(ok = mbar_wait_s_warp(bar(C::bDP), i & 1, ctl))) break;
      tc_fence_after();
      uint32_t dp[64];
      tmem_ld32(tl + C::tDP + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
      tmem_ld32(tl + C::tDP + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
      tmem_ld_wait(dp);
      tc_fence_before();
      mbar_arrive(bar(C::bDPR));
      __syncwarp();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t dsk[16];
        ds_tile32<false>(*reinterpret_cast<const uint32_t(*)[32]>(&dp[cc * 32]), pk, cc * 32,
                         nullptr, nd, dsk);
        tmem_st16(tl + tsb + cc * 16, dsk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::bDS0 + bsel));
    }
    // ---- epilogue: half h writes columns [h d/2, (h + 1) d/2) of scale dQ
    bool have = ok && n_kt > 0;
    if (have) {
      have = mbar_wait_s_warp(bar(C::bFinal), 0, ctl);
      tc_fence_after();
    }
    store_row<D / 64>(tl + C::tDQ + half * (D / 2), have, p.scale, p.dq,
                      qrow * D + half * (D / 2), q < p.Lq, true);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc<kTmemCols>(tmem);
}

// D_i = <dO_i, O_i> for every query row: one warp per row, fp32 sum.
template <int D>
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const __nv_bfloat16* __restrict__ dO,
                                                         const __nv_bfloat16* __restrict__ O,
                                                         float* __restrict__ dsum, long long rows) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (long long r = static_cast<long long>(blockIdx.x) * 8 + warp; r < rows;
       r += static_cast<long long>(gridDim.x) * 8) {
    const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(dO + r * D);
    const __nv_bfloat162* c = reinterpret_cast<const __nv_bfloat162*>(O + r * D);
    float acc = 0.f;
#pragma unroll
    for (int i = lane; i < D / 2; i += 32) {
      const float2 x = __bfloat1622float2(__ldg(a + i));
      const float2 y = __bfloat1622float2(__ldg(c + i));
      acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) dsum[r] = acc;
  }
}

template <int D>
cudaError_t launch_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                       const float* lse, float* dsum, float* dq, void* dk, void* dv, int B, int H,
                       int Lq, int Lk, float scale, int mask_kind, const int32_t* key_lengths,
                       bool out_f32, const DeviceCtl& ctl, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * H * Lq;
  int sms = 148, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long want = (rows + 7) / 8;
  const int blocks = static_cast<int>(want < 16LL * sms ? want : 16LL * sms);
  if (rows > 0) {
    bwd_rowdot_kernel<D><<<blocks, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(dO),
                                                      static_cast<const __nv_bfloat16*>(O), dsum,
                                                      rows);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  CUtensorMap maps[4];
  const void* ptrs[4] = {Q, K, V, dO};
  const int lens[4] = {Lq, Lk, Lk, Lq};
  for (int i = 0; i < 4; ++i) {
    const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(lens[i]),
                              static_cast<uint64_t>(B) * H};
    const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2,
                                 static_cast<uint64_t>(lens[i]) * D * 2};
    const uint32_t box[3] = {64, kTile, 1};
    if (!encode_tensor_map(&maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                           const_cast<void*>(ptrs[i]), dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  BwdParams p;
  p.lse = lse;
  p.dsum = dsum;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.B = B;
  p.H = H;
  p.Lq = Lq;
  p.Lk = Lk;
  p.num_k_tiles = (Lk + kTile - 1) / kTile;
  p.num_q_tiles = (Lq + kTile - 1) / kTile;
  p.mask_kind = mask_kind;
  p.key_lengths = key_lengths;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.out_f32 = out_f32 ? 1 : 0;
  p.err = ctl.err;
  p.limit_ns = ctl.limit_ns;
  const long long grid_kv = static_cast<long long>(p.num_k_tiles) * B * H;
  const long long grid_q = static_cast<long long>(p.num_q_tiles) * B * H;
  if (grid_kv > 0x7fffffffLL || grid_q > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (grid_kv > 0) {
    auto kern = sdpa_bwd_dkdv_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         CfgKV<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(grid_kv), kThreads, CfgKV<D>::kSmemBytes, stream>>>(
        maps[0], maps[1], maps[2], maps[3], p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (grid_q > 0) {
    auto kern = sdpa_bwd_dq_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         CfgQ<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(grid_q), kThreads, CfgQ<D>::kSmemBytes, stream>>>(
        maps[0], maps[1], maps[2], maps[3], p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace
}  // namespace mha

using namespace mha;

extern "C" {

mha_status sdpa_forward_lse(const void* Q, const void* K, const void* V, void* O, float* lse,
                            int B, int H, int Lq, int Lk, int d, float scale, int mask_kind,
                            const int32_t* key_lengths, mha_dtype out_dtype, mha_stream stream) {
  const mha_status st = validate_sdpa(Q, K, V, O, B, H, Lq, Lk, d, scale, mask_kind,
                                      key_lengths, MHA_BF16, out_dtype);
  if (st != MHA_OK) return st;
  if (static_cast<long long>(B) * H * Lq == 0) return MHA_OK;
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u)) return MHA_ERR_INVALID_ARG;
  DeviceCtl ctl;
  if (!device_ctl(&ctl)) return MHA_ERR_CUDA;
  SdpaArgs a{Q, K, V, O, B, H, Lq, Lk, d,
             scale == 0.f ? static_cast<float>(1.0 / sqrt(static_cast<double>(d))) : scale,
             mask_kind, key_lengths, MHA_BF16, out_dtype, false,
             reinterpret_cast<cudaStream_t>(stream), nullptr, 0, 0, lse};
  const cudaError_t e = launch_sdpa_bf16(a, ctl);
  return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

size_t sdpa_backward_workspace_bytes(int B, int H, int Lq) {
  if (B < 0 || H < 0 || Lq < 0) return 0;
  return static_cast<size_t>(B) * H * Lq * sizeof(float);
}

mha_status sdpa_backward(const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* lse, float* dQ, void* dK, void* dV, int B,
                         int H, int Lq, int Lk, int d, float scale, int mask_kind,
                         const int32_t* key_lengths, mha_dtype grad_dtype, void* workspace,
                         size_t workspace_bytes, mha_stream stream) {
  const mha_status st = validate_sdpa(Q, K, V, O, B, H, Lq, Lk, d, scale, mask_kind,
                                      key_lengths, MHA_BF16, MHA_BF16);
  if (st != MHA_OK) return st;
  if (grad_dtype != MHA_BF16 && grad_dtype != MHA_F32) return MHA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * (Lq + Lk) == 0) return MHA_OK;
  const void* ptrs[6] = {dO, dQ, dK, dV, lse, workspace};
  for (const void* ptr : ptrs)
    if (!ptr || (reinterpret_cast<uintptr_t>(ptr) & 15u)) return MHA_ERR_INVALID_ARG;
  if (workspace_bytes < sdpa_backward_workspace_bytes(B, H, Lq)) return MHA_ERR_INVALID_ARG;
  DeviceCtl ctl;
  if (!device_ctl(&ctl)) return MHA_ERR_CUDA;
  const float sc = scale == 0.f ? static_cast<float>(1.0 / sqrt(static_cast<double>(d))) : scale;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* dsum = static_cast<float*>(workspace);
  const cudaError_t e =
      d == 64 ? launch_bwd<64>(Q, K, V, O, dO, lse, dsum, dQ, dK, dV, B, H, Lq, Lk, sc, mask_kind,
                               key_lengths, grad_dtype == MHA_F32, ctl, s)
              : launch_bwd<128>(Q, K, V, O, dO, lse, dsum, dQ, dK, dV, B, H, Lq, Lk, sc,
                                mask_kind, key_lengths, grad_dtype == MHA_F32, ctl, s);
  return e == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // extern "C"
