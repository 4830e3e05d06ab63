// sdpa_decode.cu -- attention of a few new queries against a key/value cache
// (decoding): Lq <= 16 queries per (batch item, head), bottom-right causal
// alignment, the cached keys split across the CTAs of one thread-block
// cluster, and the partial softmaxes merged exactly through distributed
// shared memory.
//
// The decoder attends to earlier positions only while it generates left to
// right, and the keys and values of the tokens it has produced are kept and
// reused ("How Transformers Work" (worksonmygpu.com), "What changed since
// 2017"; "The Transformer" (hoshank.vercel.app), "The Breakthrough"; "The
// Transformer" (rayaq.ca), "The decoder stack").  The Lq new queries are the
// last Lq of the len_b cached positions, so query i sees keys
// j <= len_b - Lq + i.
//
// One CTA = one split of one (b, h): key tiles [t_begin, t_end) of 128 keys.
//   S^T = K_tile Q^T      tcgen05, M = 128 keys, N = 16 query slots, K = d
//   softmax over keys     warps 0-3, one key (TMEM lane) per thread; the
//                         per-query maximum of a tile is a warp redux plus
//                         an exchange of four warps through shared memory
//   O^T = V_tile^T P^T    tcgen05, M = d, N = 16, K = 128 keys; V is read
//                         MN-major exactly as TMA stored it.  For d = 64 the
//                         M = 128 operand's upper half is whatever 16 KB of
//                         shared memory follows the V tile (the next stage);
//                         the output rows it produces are never read.
//   merge (cluster)       o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s
//                         with M = max_s m_s: the same result as one softmax
//                         over all keys (exact up to rounding)
//
// The pass streams every visible cached key and value once from HBM; with
// 16 query slots the tensor work per byte is 16 flops, far below the
// machine's balance point, so the pipeline is sized to keep enough bytes in
// flight (2-3 stages of 48-64 KB per CTA) and the per-tile softmax short.
#include <math.h>
#include <stdint.h>

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx_cluster.cuh"

namespace mha {
namespace {

constexpr int kKeys = 128;      // keys per tile: MMA M of S^T, MMA K of O^T
constexpr int kSlots = 16;      // query slots: MMA N of both products
constexpr int kSub = 16384;     // one 128-row x 64-column bf16 box
constexpr int kQBox = 2048;     // one 16-row x 64-column bf16 box
constexpr int kPBuf = 4096;     // P^T of one tile: 16 rows x 128 keys bf16
constexpr int kThreads = 192;   // warps 0-3 softmax, 4 TMA, 5 MMA
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 64;  // S^T x 2 (cols 0-31), O^T x 2 (cols 32-63)
constexpr int kMaxSplits = 16;

template <int D>
struct DecCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int KB = D / 64;
  // d = 128: three 64 KB stages, one CTA per SM.  d = 64: three 32 KB stages
  // (~111 KB in all), so two CTAs share an SM and hide each other's setup
  // and softmax latency.
  static constexpr int NST = 3;
  static constexpr int kCtasPerSm = D == 128 ? 1 : 2;
  static constexpr int kKTile = KB * kSub;
  static constexpr int kVTile = KB * kSub;
  // shared memory from a 1024-byte aligned base.  V comes first, then K: the
  // 16 KB after any V tile is valid shared memory (the M = 128 operand of a
  // d = 64 product reads it as its unused upper half).
  static constexpr int kOffV = 0;
  static constexpr int kOffK = kOffV + NST * kVTile;
  static constexpr int kOffQ = kOffK + NST * kKTile;
  static constexpr int kOffP = kOffQ + KB * kQBox;
  static constexpr int kOffRed = kOffP + 2 * kPBuf;         // [3][4 warps][16] f32
  // m[16], l[16], o[16][D] f32 of the merge.  They are written once every
  // MMA has completed, so when they fit (d = 64) they share the P^T buffers;
  // that keeps a d = 64 CTA under half an SM's shared memory.
  static constexpr int kXBytes = (2 * kSlots + kSlots * D) * 4;
  static constexpr bool kXInP = kXBytes <= 2 * kPBuf;
  static constexpr int kOffX = kXInP ? kOffP : kOffRed + 3 * 4 * kSlots * 4;
  static constexpr int kOffBar = kXInP ? kOffRed + 3 * 4 * kSlots * 4 : kOffX + kXBytes;
  // barriers
  static constexpr int bQ = 0;
  __host__ __device__ static constexpr int bKF(int s) { return 1 + s; }
  __host__ __device__ static constexpr int bKE(int s) { return 1 + NST + s; }
  __host__ __device__ static constexpr int bVF(int s) { return 1 + 2 * NST + s; }
  __host__ __device__ static constexpr int bVE(int s) { return 1 + 3 * NST + s; }
  __host__ __device__ static constexpr int bS(int i) { return 1 + 4 * NST + i; }
  __host__ __device__ static constexpr int bP(int i) { return 3 + 4 * NST + i; }
  __host__ __device__ static constexpr int bO(int i) { return 5 + 4 * NST + i; }
  __host__ __device__ static constexpr int bRed(int i) { return 7 + 4 * NST + i; }
  static constexpr int bDrain = 9 + 4 * NST;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static_assert(kOffP % 1024 == 0, "P^T swizzle atoms must be 1024-byte aligned");
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(kCtasPerSm == 1 || kSmemBytes + 1024 <= 112 * 1024, "two CTAs per SM");
};

// Batch sizes up to this get their items ordered longest-first (below).
constexpr int kMaxSortedBatch = 256;

struct DecodeParams {
  int B, H, Lq, Lk;  // Lk: cache capacity (rows per (b, h))
  int splits;     // CTAs per (b, h) = cluster size
  int causal;     // bottom-right causal
  const int32_t* kv_len;  // [B] or nullptr (every item holds Lk tokens)
  float scale_log2;       // scale * log2(e)
  void* O;                // [B, H, Lq, D]
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

// Named barrier of the four softmax warps.
__device__ __forceinline__ void softmax_bar() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

template <int D>
__global__ void __launch_bounds__(kThreads, DecCfg<D>::kCtasPerSm)
    sdpa_decode_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  using C = DecCfg<D>;
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
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar(C::bKF(s)), 1);
      mbar_init(bar(C::bKE(s)), 1);
      mbar_init(bar(C::bVF(s)), 1);
      mbar_init(bar(C::bVE(s)), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::bS(i)), 1);
      mbar_init(bar(C::bP(i)), 128);
      mbar_init(bar(C::bO(i)), 1);
      mbar_init(bar(C::bRed(i)), 128);
    }
    mbar_init(bar(C::bDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc<kTmemCols>(smem_u32(tmem_slot));
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  float* red = reinterpret_cast<float*>(gbase + C::kOffRed);
  float* xm = reinterpret_cast<float*>(gbase + C::kOffX);
  float* xl = xm + kSlots;
  float* xo = xl + kSlots;

  // ---- this CTA's (b, h) and key tiles.  Cluster rank = split: the grid's
  // x dimension is (rank_b * H + h) * splits + split and the cluster spans
  // the splits.  CTAs start roughly in grid order, so batch items are taken
  // longest-first (rank_b = position of b when the lengths are sorted in
  // decreasing order, ties by index): the long items do not trail alone at
  // the end of the grid.  Every CTA ranks the (at most kMaxSortedBatch)
  // lengths itself from a copy in shared memory; larger batches keep
  // index order.
  const int split = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.splits));
  const int slot = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.splits));
  const int h = slot % p.H;
  int b = slot / p.H;
  if (p.kv_len && p.B > 1 && p.B <= kMaxSortedBatch) {
    int* lens_s = reinterpret_cast<int*>(xo);  // free until the merge
    int* pick = reinterpret_cast<int*>(xm);
    for (int i = threadIdx.x; i < p.B; i += kThreads) lens_s[i] = __ldg(p.kv_len + i);
    __syncthreads();
    const int want = b;
    for (int c = threadIdx.x; c < p.B; c += kThreads) {
      const int lc = lens_s[c];
      int rank = 0;
      for (int o = 0; o < p.B; ++o) {
        const int lo = lens_s[o];
        rank += (lo > lc || (lo == lc && o < c)) ? 1 : 0;
      }
      if (rank == want) *pick = c;
    }
    __syncthreads();
    b = *pick;
    __syncthreads();  // xm is written again only after the main loop
  }
  const int bh = b * p.H + h;
  int len = p.Lk;
  bool bad_len = false;
  if (p.kv_len) {
    len = __ldg(p.kv_len + b);
    if (len < 1 || len > p.Lk || (p.causal && len < p.Lq)) bad_len = true;
  }
  const int n_tiles = bad_len ? 0 : (len + kKeys - 1) / kKeys;
  const int t_begin = static_cast<int>(static_cast<long long>(n_tiles) * split / p.splits);
  const int t_end = static_cast<int>(static_cast<long long>(n_tiles) * (split + 1) / p.splits);
  const int T = t_end - t_begin;
  if (bad_len && split == 0 && threadIdx.x == 0) atomicOr(p.err, kErrKeyLength);

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && T > 0) {
      mbar_expect_tx(bar(C::bQ), C::KB * kQBox);
      for (int kb = 0; kb < C::KB; ++kb)
        tma_load_3d(base + C::kOffQ + kb * kQBox, &tmQ, bar(C::bQ), kb * 64, 0, bh);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < T; ++j) {
        const int st = j % C::NST;
        const uint32_t ph = (j / C::NST) & 1;
        const int row = (t_begin + j) * kKeys;
        if (!mbar_wait(bar(C::bKE(st)), ph ^ 1u, ctl)) break;
        mbar_expect_tx(bar(C::bKF(st)), C::kKTile);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(base + C::kOffK + st * C::kKTile + kb * kSub, &tmK, bar(C::bKF(st)),
                      kb * 64, row, bh);
        k_issued = j + 1;
        if (!mbar_wait(bar(C::bVE(st)), ph ^ 1u, ctl)) break;
        mbar_expect_tx(bar(C::bVF(st)), C::KB * kSub);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(base + C::kOffV + st * C::kVTile + kb * kSub, &tmV, bar(C::bVF(st)),
                      kb * 64, row, bh);
        v_issued = j + 1;
      }
      // let every issued copy land before the CTA can exit
      wait_drain(bar(C::bQ), 0, p.limit_ns);
      for (int j = max(0, k_issued - C::NST); j < k_issued; ++j)
        wait_drain(bar(C::bKF(j % C::NST)), (j / C::NST) & 1, p.limit_ns);
      for (int j = max(0, v_issued - C::NST); j < v_issued; ++j)
        wait_drain(bar(C::bVF(j % C::NST)), (j / C::NST) & 1, p.limit_ns);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // Order: S(0), S(1), then per tile j: O(j) once P(j) is published, and
    // S(j+2) into the S buffer that P(j)'s publication has just released.
    if (lane == 0 && T > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(kKeys, kSlots, false, false);
      constexpr uint32_t kIdO = idesc_bf16_f32(128, kSlots, true, false);
      const uint64_t q_desc = sdesc_sw128(base + C::kOffQ, 16, 1024);
      const uint64_t k_desc = sdesc_sw128(base + C::kOffK, 16, 1024);
      const uint64_t v_desc = sdesc_sw128(base + C::kOffV, kSub, 1024);
      const uint64_t p_desc = sdesc_sw128(base + C::kOffP, 16, 1024);
      auto issue_s = [&](int st, int buf) {
        const uint64_t kd = k_desc + static_cast<uint64_t>((st * C::kKTile) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          // 16 elements = 32 bytes inside a 128-byte row; 64-column blocks apart
          const uint64_t koff = static_cast<uint64_t>(((ks >> 2) * kSub + (ks & 3) * 32) >> 4);
          const uint64_t qoff = static_cast<uint64_t>(((ks >> 2) * kQBox + (ks & 3) * 32) >> 4);
          umma_ss(tmem + buf * kSlots, kd + koff, q_desc + qoff, kIdS, ks > 0 ? 1u : 0u);
        }
      };
      auto issue_o = [&](int st, int buf) {
        const uint64_t vd = v_desc + static_cast<uint64_t>((st * C::kVTile) >> 4);
        const uint64_t pd = p_desc + static_cast<uint64_t>((buf * kPBuf) >> 4);
#pragma unroll
        for (int ks = 0; ks < kKeys / 16; ++ks) {
          // V^T: 16 keys = 16 rows of 128 bytes; P^T: 64-key atoms 2048 bytes apart
          const uint64_t voff = static_cast<uint64_t>((ks * 16 * 128) >> 4);
          const uint64_t poff = static_cast<uint64_t>(((ks >> 2) * 2048 + (ks & 3) * 32) >> 4);
          umma_ss(tmem + 2 * kSlots + buf * kSlots, vd + voff, pd + poff, kIdO,
                  ks > 0 ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(bar(C::bQ), 0, ctl);
      for (int j = 0; ok && j < 2 && j < T; ++j) {
        const int st = j % C::NST;
        if (!(ok = mbar_wait(bar(C::bKF(st)), (j / C::NST) & 1, ctl))) break;
        tc_fence_after();
        issue_s(st, j);
        umma_commit(bar(C::bS(j)));
        umma_commit(bar(C::bKE(st)));
      }
      for (int j = 0; ok && j < T; ++j) {
        const int st = j % C::NST;
        const int buf = j & 1;
        if (!(ok = mbar_wait(bar(C::bP(buf)), (j >> 1) & 1, ctl))) break;
        if (!(ok = mbar_wait(bar(C::bVF(st)), (j / C::NST) & 1, ctl))) break;
        tc_fence_after();
        issue_o(st, buf);
        umma_commit(bar(C::bO(buf)));
        umma_commit(bar(C::bVE(st)));
        if (j + 2 < T) {
          const int st2 = (j + 2) % C::NST;
          if (!(ok = mbar_wait(bar(C::bKF(st2)), ((j + 2) / C::NST) & 1, ctl))) break;
          tc_fence_after();
          issue_s(st2, buf);
          umma_commit(bar(C::bS(buf)));
          umma_commit(bar(C::bKE(st2)));
        }
      }
      // every issued MMA completes before tensor memory is released
      umma_commit(bar(C::bDrain));
      wait_drain(bar(C::bDrain), 0, p.limit_ns);
    }
  } else {
    // ------------------------------------------------------------- softmax
    // Thread r (warp w may touch TMEM lanes [32w, 32w + 32)) owns key r of
    // every S^T tile and row r (= output column r) of every O^T tile.
    const int r = warp * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_bits;
    const uint32_t tO = tmem + lane_bits + 2 * kSlots;
    const bool o_rows = warp * 32 < D;  // warp-uniform
    const float sl2 = p.scale_log2;
    const int diag = len - p.Lq;  // query q sees keys <= diag + q
    // m: running maximum (log2 units) per query slot; l: this thread's share
    // of the running denominator; acc: this thread's output column, all
    // relative to m.  alpha_prev rescales acc when the previous tile's O^T
    // partial is added (one tile behind, so O(j) overlaps softmax(j + 1)).
    float m[kSlots], l[kSlots], acc[kSlots], alpha_prev[kSlots];
#pragma unroll
    for (int q = 0; q < kSlots; ++q) {
      m[q] = -INFINITY;
      l[q] = 0.f;
      acc[q] = 0.f;
      alpha_prev[q] = 1.f;
    }
    // P^T store address of key r: 64-key atom, 16-byte chunk, 2-byte slot
    const int kk = r & 63;
    uint8_t* p_key = gbase + C::kOffP + (r >> 6) * 2048 + (kk & 7) * 2;
    const int chunk = kk >> 3;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int buf = j & 1;
      const uint32_t par = (j >> 1) & 1;
      if (!(ok = mbar_wait_warp(bar(C::bS(buf)), par, ctl))) break;
      tc_fence_after();
      uint32_t sr[kSlots];
      tmem_ld16_sync(tS + buf * kSlots, sr);
      const int key = (t_begin + j) * kKeys + r;
      float s[kSlots];
#pragma unroll
      for (int q = 0; q < kSlots; ++q) {
        const bool vis = q < p.Lq && key < len && (!p.causal || key <= diag + q);
        s[q] = vis ? __uint_as_float(sr[q]) * sl2 : -INFINITY;
      }
      // per-query maximum of the tile: warp redux, then four warps via smem
      float* rb = red + buf * 4 * kSlots;
      {
        float wm[kSlots];
#pragma unroll
        for (int q = 0; q < kSlots; ++q) wm[q] = warp_max_f32(s[q]);
        if (lane == 0) {
          float4* dst = reinterpret_cast<float4*>(rb + warp * kSlots);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_float4(wm[4 * i], wm[4 * i + 1], wm[4 * i + 2], wm[4 * i + 3]);
        }
      }
      mbar_arrive(bar(C::bRed(buf)));
      if (!(ok = mbar_wait_warp(bar(C::bRed(buf)), par, ctl))) break;
      float alpha[kSlots];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 a0 = reinterpret_cast<const float4*>(rb)[i];
        const float4 a1 = reinterpret_cast<const float4*>(rb + kSlots)[i];
        const float4 a2 = reinterpret_cast<const float4*>(rb + 2 * kSlots)[i];
        const float4 a3 = reinterpret_cast<const float4*>(rb + 3 * kSlots)[i];
        const float t4[4] = {fmaxf(fmax3(a0.x, a1.x, a2.x), a3.x),
                             fmaxf(fmax3(a0.y, a1.y, a2.y), a3.y),
                             fmaxf(fmax3(a0.z, a1.z, a2.z), a3.z),
                             fmaxf(fmax3(a0.w, a1.w, a2.w), a3.w)};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int q = 4 * i + u;
          const float mn = fmaxf(m[q], t4[u]);
          const float ref = mn == -INFINITY ? 0.f : mn;  // a slot with no visible key yet
          alpha[q] = ex2_approx(m[q] - ref);
          const float pq = ex2_approx(s[q] - ref);
          l[q] = fmaf(l[q], alpha[q], pq);
          m[q] = mn;
          s[q] = pq;
        }
      }
      // P^T(j): row q, key r, 128-byte swizzle (16-byte chunk index ^ row % 8)
      uint8_t* pb = p_key + buf * kPBuf;
#pragma unroll
      for (int q = 0; q < kSlots; ++q)
        *reinterpret_cast<__nv_bfloat16*>(pb + (q >> 3) * 1024 + (q & 7) * 128 +
                                          ((chunk ^ (q & 7)) << 4)) = __float2bfloat16_rn(s[q]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::bP(buf)));
      if (j > 0) {
        const int pj = j - 1;
        if (!(ok = mbar_wait_warp(bar(C::bO(pj & 1)), (pj >> 1) & 1, ctl))) break;
        tc_fence_after();
        if (o_rows) {
          uint32_t orr[kSlots];
          tmem_ld16_sync(tO + (pj & 1) * kSlots, orr);
#pragma unroll
          for (int q = 0; q < kSlots; ++q)
            acc[q] = fmaf(acc[q], alpha_prev[q], __uint_as_float(orr[q]));
        }
      }
#pragma unroll
      for (int q = 0; q < kSlots; ++q) alpha_prev[q] = alpha[q];
    }
    if (ok && T > 0) {
      const int pj = T - 1;
      if ((ok = mbar_wait_warp(bar(C::bO(pj & 1)), (pj >> 1) & 1, ctl))) {
        tc_fence_after();
        if (o_rows) {
          uint32_t orr[kSlots];
          tmem_ld16_sync(tO + (pj & 1) * kSlots, orr);
#pragma unroll
          for (int q = 0; q < kSlots; ++q)
            acc[q] = fmaf(acc[q], alpha_prev[q], __uint_as_float(orr[q]));
        }
      }
    }
    tc_fence_before();
    // denominator: sum l over the 128 key lanes
#pragma unroll
    for (int q = 0; q < kSlots; ++q) {
#pragma unroll
      for (int sh = 16; sh > 0; sh >>= 1) l[q] += __shfl_xor_sync(0xffffffffu, l[q], sh);
    }
    float* lsum = red + 2 * 4 * kSlots;
    if (lane == 0) {
      float4* dst = reinterpret_cast<float4*>(lsum + warp * kSlots);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        dst[i] = make_float4(l[4 * i], l[4 * i + 1], l[4 * i + 2], l[4 * i + 3]);
    }
    softmax_bar();
    const bool failed = *abort_flag != 0;
    if (threadIdx.x < kSlots) {
      const int q = threadIdx.x;
      xm[q] = failed ? -INFINITY : m[q];
      xl[q] = failed ? 0.f
                     : lsum[q] + lsum[kSlots + q] + lsum[2 * kSlots + q] + lsum[3 * kSlots + q];
    }
    if (o_rows && r < D) {
#pragma unroll
      for (int q = 0; q < kSlots; ++q) xo[q * D + r] = acc[q];
    }
  }

  // ---- merge the splits of this (b, h) through distributed shared memory
  __syncwarp();
  cluster_sync();  // every split's m, l and O are in its shared memory
  if (warp < 4) {
    const int S = p.splits;
    const int total = p.Lq * D;
    const int per = (total + S - 1) / S;
    const int e0 = split * per;
    const int e1 = min(total, e0 + per);
    const uint32_t xm_s = smem_u32(xm), xl_s = smem_u32(xl), xo_s = smem_u32(xo);
    for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += 128) {
      const int q = e / D;
      const int c = e - q * D;
      float M = -INFINITY;
      for (int s = 0; s < S; ++s)
        M = fmaxf(M, ld_cluster_f32(cluster_map(xm_s + 4u * q, static_cast<uint32_t>(s))));
      float o = 0.f;
      if (M != -INFINITY) {
        float num = 0.f, den = 0.f;
        for (int s = 0; s < S; ++s) {
          const uint32_t rk = static_cast<uint32_t>(s);
          const float w = ex2_approx(ld_cluster_f32(cluster_map(xm_s + 4u * q, rk)) - M);
          num = fmaf(w, ld_cluster_f32(cluster_map(xo_s + 4u * (q * D + c), rk)), num);
          den = fmaf(w, ld_cluster_f32(cluster_map(xl_s + 4u * q, rk)), den);
        }
        o = num / den;
      }
      const size_t idx = (static_cast<size_t>(bh) * p.Lq + q) * D + c;
      if (p.out_f32)
        reinterpret_cast<float*>(p.O)[idx] = o;
      else
        reinterpret_cast<__nv_bfloat16*>(p.O)[idx] = __float2bfloat16_rn(o);
    }
  }
  __syncwarp();
  cluster_sync();  // no CTA leaves while another still reads its shared memory
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc<kTmemCols>(tmem);
  }
}

// Dynamic shared memory size, and the whole unified L1/shared array given to
// shared memory so that two d = 64 CTAs share an SM.
template <int D>
cudaError_t set_kernel_attributes() {
  auto kern = sdpa_decode_bf16_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       DecCfg<D>::kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

template <int D>
cudaError_t launch_impl(const DecodeArgs& a, const DeviceCtl& ctl) {
  using C = DecCfg<D>;
  CUtensorMap maps[3];
  const void* ptrs[3] = {a.Q, a.K, a.V};
  const int rows[3] = {a.Lq, a.Lk, a.Lk};
  const uint32_t box_rows[3] = {kSlots, kKeys, kKeys};
  for (int i = 0; i < 3; ++i) {
    const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(rows[i]),
                              static_cast<uint64_t>(a.B) * a.H};
    const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2,
                                 static_cast<uint64_t>(rows[i]) * D * 2};
    const uint32_t box[3] = {64, box_rows[i], 1};
    if (!encode_tensor_map(&maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                           const_cast<void*>(ptrs[i]), dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  DecodeParams p;
  p.B = a.B;
  p.H = a.H;
  p.Lq = a.Lq;
  p.Lk = a.Lk;
  p.splits = a.splits;
  p.causal = a.causal ? 1 : 0;
  p.kv_len = a.kv_len;
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.O = a.O;
  p.out_f32 = a.out_dtype == MHA_F32 ? 1 : 0;
  p.err = ctl.err;
  p.limit_ns = ctl.limit_ns;

  auto kern = sdpa_decode_bf16_kernel<D>;
  cudaError_t e = set_kernel_attributes<D>();
  if (e == cudaSuccess && a.splits > 8)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long long>(a.B) * a.H * a.splits));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(a.splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Stand-in for the decode kernel in occupancy queries: same block size and
// shared memory, no body.  The runtime occupancy calculator answers one CTA
// per SM for the decode kernel itself whatever its shared memory, while the
// hardware keeps two d = 64 CTAs resident (profiled warps-active average:
// 10.7 warps per SM, above the 6 of one CTA); the stand-in's answer matches
// what the hardware does.
__global__ void __launch_bounds__(kThreads) decode_occupancy_proxy_kernel() {}

// Clusters of `splits` CTAs of the d-kernel that the device holds at once
// (cached per device; 0 when the query fails).
template <int D>
int max_active_clusters(int splits) {
  constexpr int kDevs = 16;
  static int cache[kDevs][kMaxSplits + 1];
  static bool filled[kDevs][kMaxSplits + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  const bool cacheable = dev < kDevs;
  if (cacheable && filled[dev][splits]) return cache[dev][splits];
  auto kern = decode_occupancy_proxy_kernel;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           DecCfg<D>::kSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
      (splits > 8 &&
       cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
           cudaSuccess)) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(splits));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = DecCfg<D>::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  if (cacheable) {
    cache[dev][splits] = n;
    filled[dev][splits] = true;
  }
  return n;
}

}  // namespace

int decode_default_splits(int B, int H, int Lk, int d) {
  const long long bh = static_cast<long long>(B) * H;
  const int tiles = (Lk + kKeys - 1) / kKeys;
  // The largest split count whose B*H clusters are all resident at once
  // (one wave).  A second, partial wave costs more than the SMs a single
  // wave leaves idle, because each CTA keeps enough copies in flight to draw
  // more than its share of HBM bandwidth; and how many clusters fit depends
  // on their size (a cluster must sit inside one GPC), so the count is asked
  // of the device for every size.  Never more splits than key tiles.
  int best = 1;
  for (int s = 2; s <= kMaxSplits && s <= tiles; ++s) {
    const int n = d == 64 ? max_active_clusters<64>(s) : max_active_clusters<128>(s);
    if (n >= bh) best = s;
  }
  return best;
}

cudaError_t launch_sdpa_decode_bf16(const DecodeArgs& a, const DeviceCtl& ctl) {
  if (a.splits < 1 || a.splits > kMaxSplits || a.Lq < 1 || a.Lq > kSlots)
    return cudaErrorInvalidValue;
  if (a.d == 64) return launch_impl<64>(a, ctl);
  if (a.d == 128) return launch_impl<128>(a, ctl);
  return cudaErrorInvalidValue;
}

}  // namespace mha

using namespace mha;

extern "C" {

mha_status sdpa_decode(const void* Q, const void* K_cache, const void* V_cache, void* O, int B,
                       int H, int Lq, int Lk, int d, float scale, int mask_kind,
                       const int32_t* kv_lengths, mha_dtype out_dtype, int num_splits,
                       mha_stream stream) {
  if (B < 0 || H < 0 || Lq < 1 || Lq > MHA_DECODE_MAX_QUERIES || Lk < 1)
    return Lq > MHA_DECODE_MAX_QUERIES ? MHA_ERR_UNSUPPORTED : MHA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return MHA_ERR_UNSUPPORTED;
  if (out_dtype != MHA_BF16 && out_dtype != MHA_F32) return MHA_ERR_INVALID_ARG;
  if (!(scale >= 0.f) || isinf(scale)) return MHA_ERR_INVALID_ARG;
  if (mask_kind & ~(MHA_MASK_CAUSAL_BOTTOM_RIGHT | MHA_MASK_KEY_PADDING))
    return MHA_ERR_INVALID_ARG;
  const bool causal = (mask_kind & MHA_MASK_CAUSAL_BOTTOM_RIGHT) != 0;
  const bool padded = (mask_kind & MHA_MASK_KEY_PADDING) != 0;
  if (padded != (kv_lengths != nullptr)) return MHA_ERR_INVALID_ARG;
  if (kv_lengths && (reinterpret_cast<uintptr_t>(kv_lengths) & 3u)) return MHA_ERR_INVALID_ARG;
  if (causal && !padded && Lq > Lk) return MHA_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > kMaxSplits) return MHA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H == 0) return MHA_OK;
  const void* ptrs[4] = {Q, K_cache, V_cache, O};
  for (const void* ptr : ptrs)
    if (!ptr || (reinterpret_cast<uintptr_t>(ptr) & 15u)) return MHA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * kMaxSplits > 0x7fffffffLL) return MHA_ERR_UNSUPPORTED;
  DeviceCtl ctl;
  if (!device_ctl(&ctl)) return MHA_ERR_CUDA;
  DecodeArgs a;
  a.Q = Q;
  a.K = K_cache;
  a.V = V_cache;
  a.O = O;
  a.B = B;
  a.H = H;
  a.Lq = Lq;
  a.Lk = Lk;
  a.d = d;
  a.scale = scale == 0.f ? static_cast<float>(1.0 / sqrt(static_cast<double>(d))) : scale;
  a.causal = causal;
  a.kv_len = kv_lengths;
  a.out_dtype = out_dtype;
  a.splits = num_splits > 0 ? num_splits : decode_default_splits(B, H, Lk, d);
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = launch_sdpa_decode_bf16(a, ctl);
  if (e == cudaSuccess) return MHA_OK;
  return e == cudaErrorMemoryAllocation ? MHA_ERR_OOM : MHA_ERR_CUDA;
}

int sdpa_decode_splits(int B, int H, int Lk, int d) {
  if (B < 1 || H < 1 || Lk < 1 || (d != 64 && d != 128)) return 0;
  return decode_default_splits(B, H, Lk, d);
}

}  // extern "C"
