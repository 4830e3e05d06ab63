// sdpa_backward.cu -- the backward pass of scaled dot-product attention
// (training), bf16 in, fp32 accumulate, on sm_103a tcgen05 tensor cores.
//
// Given dO = dL/dO for O = softmax(S) V, S = scale Q K^T + M, and the row
// log-sum-exp of the forward pass (lse, base 2):
//   P    = 2^(S log2(e) - lse)               recomputed per tile
//   dV  += P^T dO
//   dP   = dO V^T
//   dS   = P (dP - D),  D_i = <dO_i, O_i>    (= sum_j P_ij dP_ij)
//   dK  += scale dS^T Q
//   dQ  += scale dS K
// (the chain rule through the attention formula of "How Transformers Work"
// (worksonmygpu.com), "Scaled dot-product attention"; the softmax gradient
// "32 Transformer" (ml-canon-en), "Why we divide by sqrt(dk)", discusses).
//
// CTA = one tile of 128 keys of one (b, h); it walks the 128-query tiles
// that can see those keys and keeps dK and dV in tensor memory throughout.
// Keys sit on the MMA's M side (TMEM lanes):
//   S^T  = K Q^T        M 128 keys, N 128 queries, K = d      TMEM cols 0-127
//   dP^T = V dO^T       same shape                            TMEM cols 128-255
//   P^T  -> bf16 pairs: queries 0-63 in S^T cols 0-31, 64-127 in cols 64-95
//   dS^T -> bf16 pairs in the same places of dP^T, and into shared memory
//   dV  += P^T dO       A = P^T from TMEM, B = dO (MN-major)  TMEM dV
//   dK  += dS^T Q       A = dS^T from TMEM, B = Q (MN-major)  TMEM dK
//   dQ^T = K^T dS^T     A = K (MN-major), B = dS^T (MN-major, the shared
//                       copy): M = d on the TMEM lanes (d = 64 pads M to 128
//                       with rows that are never read), N 128 queries;
//                       d = 128 writes it over dP^T, d = 64 into cols 384-511
// and the dQ tile is added to an fp32 dQ accumulator in global memory: a
// warp's lanes hold 32 consecutive d of one query row, so each reduction
// instruction covers 128 contiguous bytes.
//
// Warps 0-7 compute P and dS: warp w takes the keys on TMEM lanes
// 32 (w % 4) .. +31 and the 64 queries of half w / 4, two such warps per
// SM sub-partition.  Each half writes P and dS only inside the columns it
// alone reads.  Warps 8-11 move the dQ tile out (one d per lane) and write
// dK at the end, warp 12 loads (TMA, and the tile's -lse and -D rows into
// shared memory), warp 13 issues the MMAs in the order dV(j), S^T(j+1),
// dK(j), dQ^T(j), dP^T(j+1), so the next tile's exponentials run under this
// tile's dK and dQ products.  Every wait is bounded; waiting threads sleep
// on the barrier instead of spinning.
#include <math.h>
#include <stdint.h>

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "ptx_cluster.cuh"

namespace mha {
namespace {

constexpr int kTile = 128;       // keys per CTA = queries per step
constexpr int kSub = 16384;      // one 128-row x 64-column bf16 box
constexpr int kPdsWarps = 8;     // warps 0-7; warps 8-11 move dQ out
constexpr int kLoadWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxSmem = 232448;  // per-CTA opt-in limit

template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int KB = D / 64;
  static constexpr int kTileBytes = KB * kSub;   // a 128-row tile of K, V, Q or dO
  static constexpr int NST = D == 128 ? 2 : 3;    // Q/dO stages
  // shared memory from a 1024-byte aligned base
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;                 // NST stages
  static constexpr int kOffDO = kOffQ + NST * kTileBytes;          // NST stages
  static constexpr int kOffDS = kOffDO + NST * kTileBytes;         // dS, 2 x 64 queries
  static constexpr int kOffRow = kOffDS + 2 * kSub;                // NST x {-lse[128], -D[128]}
  static constexpr int kOffBar = kOffRow + NST * 1024;
  // barriers
  static constexpr int bKV = 0;
  __host__ __device__ static constexpr int bFull(int s) { return 1 + s; }
  __host__ __device__ static constexpr int bEmpty(int s) { return 1 + NST + s; }
  static constexpr int bS = 1 + 2 * NST;   // S^T(j) complete
  static constexpr int bDP = bS + 1;       // dP^T(j) complete
  static constexpr int bP0 = bS + 2;       // P^T(j) queries 0-63 in TMEM
  static constexpr int bP1 = bS + 3;       // P^T(j) queries 64-127 in TMEM
  static constexpr int bDS = bS + 4;       // dS(j) in TMEM and shared memory
  static constexpr int bDQ = bS + 5;       // dQ^T(j) complete
  static constexpr int bDQF = bS + 6;      // dQ^T(j) read out of TMEM
  static constexpr int bFinal = bS + 7;
  static constexpr int bDrain = bS + 8;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kUsed = kOffMisc + 16;   // bytes from the aligned base
  static_assert(kUsed <= kMaxSmem, "shared memory");
  // the allocation leaves room to align the base; d = 128 has 896 bytes of
  // slack (the dynamic window starts 1024-byte aligned in practice, and the
  // kernel checks)
  static constexpr int kSmemBytes = kUsed + 1024 <= kMaxSmem ? kUsed + 1024 : kMaxSmem;
  // tensor memory
  static constexpr uint32_t tS = 0, tDP = 128, tDV = 256, tDK = 256 + D;
  static constexpr bool kDqOverDp = D == 128;
  static constexpr uint32_t tDQ = kDqOverDp ? tDP : 384;
};

struct BwdParams {
  const float* lse;     // [B, H, Lq], base 2
  const float* dsum;    // [B, H, Lq], D_i = <dO_i, O_i>
  float* dq;            // [B, H, Lq, d] fp32 accumulator (zeroed by the caller)
  void* dk;             // [B, H, Lk, d]
  void* dv;
  int B, H, Lq, Lk;
  int num_k_tiles;
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

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
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
  float4 v;
  if ((Lq & 3) == 0 && q + 3 < Lq) {
    v = __ldg(reinterpret_cast<const float4*>(row + q));
    return make_float4(-v.x, -v.y, -v.z, -v.w);
  }
  return make_float4(q < Lq ? -__ldg(row + q) : fill, q + 1 < Lq ? -__ldg(row + q + 1) : fill,
                     q + 2 < Lq ? -__ldg(row + q + 2) : fill,
                     q + 3 < Lq ? -__ldg(row + q + 3) : fill);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

// NCB x 32 columns of dK or dV of this thread's key from TMEM (whole warp;
// zeros when `have` is false), times `mul`, stored from column `c0` for a
// key below Lk.
template <int NCB>
__device__ __forceinline__ void store_key_grad(uint32_t taddr, bool have, float mul, void* out,
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

// 14 warps: two SM sub-partitions hold four of them, and a sub-partition has
// 16K registers, so 128 per thread at most
template <int D>
__global__ void __maxnreg__(128)
    sdpa_bwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmDO, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  if (base - raw + C::kUsed > static_cast<uint32_t>(C::kSmemBytes)) {
    // before any barrier or TMEM allocation: the whole CTA leaves
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
    mbar_init(bar(C::bDS), 32 * kPdsWarps);
    mbar_init(bar(C::bDQ), 1);
    mbar_init(bar(C::bDQF), 128);
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

  // ---- this CTA's (b, h) and key tile: head-major, so the CTAs resident at
  // once share a head's Q and dO in L2; causal key tiles go from the first
  // (which sees the most query tiles) to the last.
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
  const int n_qt_all = (p.Lq + kTile - 1) / kTile;
  const int qt_begin = causal ? k0 / kTile : 0;
  const int n_qt = (bad_len || k0 >= len) ? 0 : max(0, n_qt_all - qt_begin);

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
      constexpr uint32_t kIdQ = idesc_bf16_f32(kTile, kTile, true, true);    // dQ^T
      const uint64_t k_desc = sdesc_sw128(base + C::kOffK, 16, 1024);
      const uint64_t v_desc = sdesc_sw128(base + C::kOffV, 16, 1024);
      // K^T as the MN-major A of dQ^T: M = d in 64-element blocks kSub apart
      // (for d = 64 the second block is the V tile: rows never read)
      const uint64_t kt_mn = sdesc_sw128(base + C::kOffK, kSub, 1024);
      const uint64_t q_desc = sdesc_sw128(base + C::kOffQ, 16, 1024);
      const uint64_t q_mn = sdesc_sw128(base + C::kOffQ, kSub, 1024);
      const uint64_t do_desc = sdesc_sw128(base + C::kOffDO, 16, 1024);
      const uint64_t do_mn = sdesc_sw128(base + C::kOffDO, kSub, 1024);
      const uint64_t ds_mn = sdesc_sw128(base + C::kOffDS, kSub, 1024);
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
        // dV += P^T dO, each half as soon as its softmax warps stored it
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
        // dQ^T = K^T dS^T over the 128 keys, 16 per step
        if (!C::kDqOverDp && j > 0) {
          if (!(ok = mbar_wait_s(bar(C::bDQF), par ^ 1u, ctl))) break;
          tc_fence_after();
        }
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks) {
          const uint64_t off = static_cast<uint64_t>((ks * 16 * 128) >> 4);
          umma_ss(tmem + C::tDQ, kt_mn + off, ds_mn + off, kIdQ, ks > 0 ? 1u : 0u);
        }
        umma_commit(bar(C::bDQ));
        umma_commit(bar(C::bEmpty(j % C::NST)));
        if (more) {
          // d = 128: dQ^T sits over dP^T until it has been read out
          if (C::kDqOverDp) {
            if (!(ok = mbar_wait_s(bar(C::bDQF), par, ctl))) break;
            tc_fence_after();
          }
          issue_t(tmem + C::tDP, v_desc, do_desc + stage_off(j + 1));
          umma_commit(bar(C::bDP));
        }
      }
      umma_commit(bar(C::bFinal));
      umma_commit(bar(C::bDrain));
      wait_drain(bar(C::bDrain), 0, p.limit_ns);
    }
  } else if (warp < kPdsWarps) {
    // ------------------------- P and dS (lane = a key, half = 64 queries)
    const int quarter = warp & 3;
    const int half = warp >> 2;
    const int L = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int key = k0 + L;
    const bool key_live = key < len;
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    uint8_t* ds_row = gbase + C::kOffDS + half * kSub + (L >> 3) * 1024 + (L & 7) * 128;
    bool ok = true;
    for (int j = 0; j < n_qt; ++j) {
      const int st = j % C::NST;
      const uint32_t par = j & 1;
      const int qh = (qt_begin + j) * kTile + half * 64;   // first query of this half
      const float* nrow = reinterpret_cast<const float*>(gbase + C::kOffRow + st * 1024);
      const float* nlse = nrow + half * 64;
      const float* nd = nrow + 128 + half * 64;
      if (!(ok = mbar_wait_s_warp(bar(C::bS), par, ctl))) break;
      if (!(ok = mbar_wait_s_warp(bar(C::bFull(st)), (j / C::NST) & 1, ctl))) break;
      tc_fence_after();
      // ---- P^T of this key over the half's 64 queries, kept as bf16 pairs
      uint32_t pk[32];
      {
        uint32_t s[64];
        tmem_ld32(tl + C::tS + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld32(tl + C::tS + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_ld_wait(s);
        // every query of the half sees this key / none does / some do
        const bool all_vis = key_live && (!causal || key <= qh);
        const bool none_vis = !key_live || (causal && key > qh + 63);
        if (all_vis) {
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            const float4 nl = *reinterpret_cast<const float4*>(nlse + c);
            const float2 x01 = ffma2(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])),
                                     sl2, make_float2(nl.x, nl.y));
            const float2 x23 = ffma2(
                make_float2(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3])), sl2,
                make_float2(nl.z, nl.w));
            pk[c / 2] = pack_bf16x2(ex2_approx(x01.x), ex2_approx(x01.y));
            pk[c / 2 + 1] = pack_bf16x2(ex2_approx(x23.x), ex2_approx(x23.y));
          }
        } else if (none_vis) {
#pragma unroll
          for (int c = 0; c < 32; ++c) pk[c] = 0u;
        } else {
          // the diagonal tile: query q sees this key when key <= q
          const int first = key - qh;   // first visible column, in (0, 63]
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const float2 nl = *reinterpret_cast<const float2*>(nlse + c);
            const float2 x = ffma2(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])),
                                   sl2, nl);
            pk[c / 2] = pack_bf16x2(c >= first ? ex2_approx(x.x) : 0.f,
                                    c + 1 >= first ? ex2_approx(x.y) : 0.f);
          }
        }
        // queries of half h -> bf16 pairs at columns 64 h .. 64 h + 31 (their
        // S^T values are already in registers; the other half's warps read
        // only columns 64 (1 - h) ..).  The branches above may split the
        // warp on the diagonal tile: reconverge before the collective store.
        __syncwarp();
        tmem_st32(tl + C::tS + half * 64, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(half == 0 ? C::bP0 : C::bP1));
      }
      // ---- dS^T = P^T (dP^T - D) over the half, 32 queries at a time; bf16
      // pairs into TMEM at dP^T columns 64 h .. (already read) and into
      // shared memory as the MN-major B of the dQ product (row = key,
      // 64-query blocks).  The dQ product of the previous tile, the last
      // reader of that buffer, has completed: dP^T(j) was committed after it.
      if (!(ok = mbar_wait_s_warp(bar(C::bDP), par, ctl))) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t dp[32];
        tmem_ld32(tl + C::tDP + half * 64 + cc * 32, dp);
        tmem_ld_wait(dp);
        uint32_t dsk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 ndv = *reinterpret_cast<const float4*>(nd + cc * 32 + i);
          const float2 d01 = fadd2(make_float2(__uint_as_float(dp[i]), __uint_as_float(dp[i + 1])),
                                   make_float2(ndv.x, ndv.y));
          const float2 d23 = fadd2(
              make_float2(__uint_as_float(dp[i + 2]), __uint_as_float(dp[i + 3])),
              make_float2(ndv.z, ndv.w));
          const float2 s01 = fmul2(unpack_bf16x2(pk[cc * 16 + i / 2]), d01);
          const float2 s23 = fmul2(unpack_bf16x2(pk[cc * 16 + i / 2 + 1]), d23);
          dsk[i / 2] = pack_bf16x2(s01.x, s01.y);
          dsk[i / 2 + 1] = pack_bf16x2(s23.x, s23.y);
        }
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
            "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(
                tl + C::tDP + half * 64 + cc * 16),
            "r"(dsk[0]), "r"(dsk[1]), "r"(dsk[2]), "r"(dsk[3]), "r"(dsk[4]), "r"(dsk[5]),
            "r"(dsk[6]), "r"(dsk[7]), "r"(dsk[8]), "r"(dsk[9]), "r"(dsk[10]), "r"(dsk[11]),
            "r"(dsk[12]), "r"(dsk[13]), "r"(dsk[14]), "r"(dsk[15])
            : "memory");
        // shared memory: queries [32 cc, 32 cc + 32) of the half in row L,
        // 16-byte chunks (q % 64) / 8, swizzled by L % 8
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int chunk = cc * 4 + u;
          *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (L & 7)) << 4)) =
              make_uint4(dsk[4 * u], dsk[4 * u + 1], dsk[4 * u + 2], dsk[4 * u + 3]);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::bDS));
    }
    // ---- epilogue: half h writes dV columns [h d/2, (h + 1) d/2) of its key
    bool have = ok && n_qt > 0;
    if (have) {
      have = mbar_wait_s_warp(bar(C::bFinal), 0, ctl);
      tc_fence_after();
    }
    store_key_grad<D / 64>(tl + C::tDV + half * (D / 2), have, 1.f, p.dv,
                           (static_cast<size_t>(bh) * p.Lk + key) * D + half * (D / 2),
                           key < p.Lk, p.out_f32 != 0);
  } else {
    // ---------------------------------------- dQ tile out (lane = a d index)
    const int quarter = warp & 3;
    const int t = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float* dq_h = p.dq + static_cast<size_t>(bh) * p.Lq * D;
    bool ok = true;
    for (int j = 0; j < n_qt; ++j) {
      const int q0 = (qt_begin + j) * kTile;
      if (!(ok = mbar_wait_s_warp(bar(C::bDQ), j & 1, ctl))) break;
      tc_fence_after();
      uint32_t g[kTile];
#pragma unroll
      for (int cb = 0; cb < kTile / 32; ++cb)
        tmem_ld32(tl + C::tDQ + cb * 32, *reinterpret_cast<uint32_t(*)[32]>(&g[cb * 32]));
      tmem_ld_wait(g);
      tc_fence_before();
      mbar_arrive(bar(C::bDQF));
      if (t < D) {
        const int nq = min(kTile, p.Lq - q0);
        float* col = dq_h + static_cast<size_t>(q0) * D + t;
#pragma unroll
        for (int q = 0; q < kTile; ++q)
          if (q < nq) red_add_f32(col + q * D, __uint_as_float(g[q]) * p.scale);
      }
    }
    // ---- epilogue: scale dK of the key on this TMEM lane
    bool have = ok && n_qt > 0;
    if (have) {
      have = mbar_wait_s_warp(bar(C::bFinal), 0, ctl);
      tc_fence_after();
    }
    const int key = k0 + t;
    store_key_grad<D / 32>(tl + C::tDK, have, p.scale, p.dk,
                           (static_cast<size_t>(bh) * p.Lk + key) * D, key < p.Lk,
                           p.out_f32 != 0);
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
  using C = BwdCfg<D>;
  const long long rows = static_cast<long long>(B) * H * Lq;
  int sms = 148, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long want = (rows + 7) / 8;
  const int blocks = static_cast<int>(want < 16LL * sms ? want : 16LL * sms);
  bwd_rowdot_kernel<D><<<blocks, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(dO),
                                                    static_cast<const __nv_bfloat16*>(O), dsum,
                                                    rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(dq, 0, static_cast<size_t>(rows) * D * sizeof(float), stream);
  if (e != cudaSuccess) return e;
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
  p.mask_kind = mask_kind;
  p.key_lengths = key_lengths;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.out_f32 = out_f32 ? 1 : 0;
  p.err = ctl.err;
  p.limit_ns = ctl.limit_ns;
  const long long grid = static_cast<long long>(p.num_k_tiles) * B * H;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  auto kern = sdpa_bwd_bf16_kernel<D>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, stream>>>(maps[0], maps[1],
                                                                         maps[2], maps[3], p);
  return cudaGetLastError();
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
