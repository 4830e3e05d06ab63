// gemm_ln_bf16.cu -- a projection whose epilogue is the post-norm sublayer
// wrapper: C = LayerNorm(R + A @ W + bias) * gamma + beta, bf16 operands,
// fp32 accumulation and statistics, on sm_103a tcgen05 tensor cores.
//
// In the post-norm encoder layer every sublayer's output is added to its
// input and the sum is normalised per position ("The Transformer"
// (hoshank.vercel.app), "The Mathematics": output = LayerNorm(x +
// Sublayer(x)); "The Transformer" (rayaq.ca), "Residuals and LayerNorm").
// The attention output projection (R = x) and the second FFN matrix
// (R = x1) are the last steps of their sublayers, so the residual add and
// the LayerNorm run in those GEMMs' epilogues: the sublayer output never
// goes to memory, and it is never rounded to bf16 before the sum.
//
// A CTA's output tile is 128 rows x N columns with N = d_model <= 512, i.e.
// whole rows: the fp32 accumulator holds N of the 512 tensor-memory columns
// and each epilogue thread owns one row, half of its columns.
//
// When N is an even number of 64-column blocks, two CTAs on two SMs (a
// cluster) share a tile of 256 rows: the even CTA issues M = 256 products
// (tcgen05 .cta_group::2) whose A rows and W columns are split between the
// two CTAs' shared memory, so each SM stages 128 rows of A and half of W per
// k-step (48 KB at N = 512 instead of 80 KB, three stages instead of two),
// and each CTA's tensor memory receives its own 128 rows.  Odd block counts
// run the same code as one CTA per tile.
//
// The epilogue makes two passes over the row in tensor memory, two warps per
// lane quarter, each taking half of the row's 64-column chunks:
//   1. v = acc + bias + R (R arrives by TMA, 32 rows x 64 columns per warp
//      and chunk, in a two-buffer ring whose first chunks load while the
//      MMAs run; bias, gamma and beta sit in shared memory); per
//      64-column chunk the mean and the centred sum of squares, merged
//      chunk by chunk with the pairwise update of Chan, Golub and LeVeque
//      ("Updating formulae and a pairwise algorithm for computing sample
//      variances", 1979): no E[v^2] - E[v]^2 cancellation; v goes back into
//      tensor memory.  The two warps of a quarter then swap their halves'
//      (mean, M2) through shared memory and merge them the same way, in the
//      same order, so both normalise with identical values;
//   2. y = (v - mean) / sqrt(var + eps) * gamma + beta, population variance
//      (divisor N), stored as bf16 or fp32 through a per-warp shared-memory
//      transpose, so that each store instruction writes four whole 128-byte
//      row pieces.
// Tile t walks its k-steps starting at t mod (K / 64): all CTAs share W, and
// staggering keeps them from asking the same L2 lines at once.
// Warp roles: warp 0 TMA producer, warp 1 MMA issuer and TMEM owner (the
// even CTA's issues for the pair), warps 2-9 epilogue.  One accumulator: the
// next tile's MMAs wait for the epilogue (of both CTAs), while the TMA ring
// keeps loading ahead.  Launched with programmatic dependent launch: the
// kernel sets itself up while the launch before it finishes, and waits for it
// before touching A, the residual or C.
#include "internal.h"
#include "ptx.cuh"
#include "ptx_cluster.cuh"
#include "ptx_pdl.cuh"
#include "ptx_pair.cuh"

namespace mha {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB: 128 rows x 64 k
constexpr int kWBox = 64 * 64 * 2;      // 8 KB: one 64(N) x 64(K) box of W
constexpr int kEpiWarps = 8;   // two per TMEM lane quarter, each half of the row's columns
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kStageWarpBytes = 32 * 128;  // one residual / staging buffer: 32 rows x 128 bytes

// N = 64 * NB output columns = whole rows.  kPair: the CTA pair form (a
// cluster of two; M = 256 products issued by the even CTA, each CTA staging
// its own 128 rows of A and half of every MMA's W columns), which needs every
// column chunk to split into whole 64-column blocks, i.e. NB even.
template <int NB, bool kPair>
struct LnCfg {
  static_assert(NB >= 1 && NB <= 8, "N = 64..512");
  static_assert(!kPair || NB % 2 == 0, "the pair form splits chunks into 64-column halves");
  static constexpr int N = 64 * NB;
  static constexpr int kTileM = kPair ? 2 * kBM : kBM;   // rows of one tile (both CTAs)
  static constexpr int kWBlocks = kPair ? NB / 2 : NB;   // 64-column W blocks this CTA stages
  // W blocks per copy in the pair form: a chunk's half is two blocks when
  // every chunk is 256 columns wide (NB a multiple of 4), else one per copy
  static constexpr int kPB = kPair ? (NB % 4 == 0 ? 2 : 1) : NB;
  static constexpr int kStageBytes = kABytes + kWBlocks * kWBox;
  // residual ring per epilogue warp: kRB buffers of 32 rows x 64 columns
  static constexpr int kRB = 2;
  // operand stages: as many as fit beside the residual rings (which also
  // stage the output), bias / gamma / beta, the statistics exchange and the
  // barriers (up to four)
  static constexpr int kStatBytes = 4 * 2 * 32 * 8 + 4 * 2 * 4;  // (mean, m2) per row, verdicts
  static constexpr int kStageBudget =
      232448 - 1024 - 512 - kEpiWarps * kRB * kStageWarpBytes - 3 * N * 2 - kStatBytes;
  static constexpr int kStages = kStageBudget / kStageBytes >= 4 ? 4 : kStageBudget / kStageBytes;
  static_assert(kStages >= 2, "operand stages");
  static constexpr uint32_t kTmemCols = N <= 64 ? 64u : N <= 128 ? 128u : N <= 256 ? 256u : 512u;
  // MMA column chunks of at most 256 (the largest N of one M = 128 MMA)
  static constexpr int kChunks = (N + 255) / 256;
  __host__ __device__ static constexpr int chunk_n(int c) { return N - 256 * c < 256 ? N - 256 * c : 256; }
  // barriers: full[S], empty[S], acc_full, acc_empty, drain, residual[kEpiWarps][kRB]
  __host__ __device__ static constexpr int bFull(int s) { return s; }
  __host__ __device__ static constexpr int bEmpty(int s) { return kStages + s; }
  static constexpr int bAccFull = 2 * kStages;
  static constexpr int bAccEmpty = 2 * kStages + 1;
  static constexpr int bDrain = 2 * kStages + 2;
  __host__ __device__ static constexpr int bRes(int w, int b) { return 2 * kStages + 3 + w * kRB + b; }
  static constexpr int kNumBars = 2 * kStages + 3 + kEpiWarps * kRB;
  // acc_empty arrivals: one per epilogue warp of each CTA of the tile
  static constexpr int kAccArrivals = kPair ? 2 * kEpiWarps : kEpiWarps;
  // the two epilogue warps of a lane quarter split the row's NB chunks
  __host__ __device__ static constexpr int cb_begin(int chalf) { return chalf ? (NB + 1) / 2 : 0; }
  __host__ __device__ static constexpr int cb_end(int chalf) { return chalf ? NB : (NB + 1) / 2; }
  // shared memory from a 1024-byte aligned base: stages, residual rings
  // (1024-byte aligned: the TMA's 128-byte swizzle), output staging,
  // bias / gamma / beta, barriers, misc
  static constexpr int kOffRes = kStages * kStageBytes;
  static constexpr int kOffStat = kOffRes + kEpiWarps * kRB * kStageWarpBytes;
  static constexpr int kOffVec = kOffStat + kStatBytes;
  static constexpr int kOffBar = kOffVec + 3 * N * 2;
  static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory");
};

struct GemmLnParams {
  void* C;                          // [M, N], bf16 or fp32
  const __nv_bfloat16* bias;        // [N]
  const __nv_bfloat16* resid;       // [M, N] (read through its tensor map)
  const __nv_bfloat16* gamma;       // [N]
  const __nv_bfloat16* beta;        // [N]
  float eps;
  int out_f32;
  int M, K;
  int mt;                           // row tiles
  unsigned* err;
  uint64_t limit_ns;
};

__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return;
  }
}

__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Barrier `id` (1..15) among `count` threads (whole warps).
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int NB, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_ln_bf16_kernel(const __grid_constant__ CUtensorMap tA,
                        const __grid_constant__ CUtensorMap tW,
                        const __grid_constant__ CUtensorMap tR, const GemmLnParams p) {
  using C = LnCfg<NB, kPair>;
  constexpr int N = C::N;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffMisc + 4);
  auto bar = [base](int i) -> uint32_t { return base + C::kOffBar + 8u * i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitCtl ctl{abort_flag, p.err, p.limit_ns};
  // tiles of kTileM rows: one per CTA, or in the pair form one per cluster
  // of two, whose rank-0 CTA issues the MMAs and owns the barriers that
  // gather both CTAs' stage bytes and both epilogues' releases
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const int tile0 = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tstride = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  auto row_base = [&](int t) { return t * C::kTileM + static_cast<int>(rank) * kBM; };
  auto lead_bar = [&](int i) -> uint32_t { return kPair ? cluster_map(bar(i), 0u) : bar(i); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::bFull(s)), 1);
      mbar_init(bar(C::bEmpty(s)), 1);
    }
    mbar_init(bar(C::bAccFull), 1);
    mbar_init(bar(C::bAccEmpty), C::kAccArrivals);
    mbar_init(bar(C::bDrain), 1);
    for (int w = 0; w < kEpiWarps; ++w)
      for (int b = 0; b < C::kRB; ++b) mbar_init(bar(C::bRes(w, b)), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair<C::kTmemCols>(smem_u32(tmem_slot));
      tmem_relinquish_pair();
    } else {
      tmem_alloc<C::kTmemCols>(smem_u32(tmem_slot));
      tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tA);
    tma_prefetch_desc(&tW);
    tma_prefetch_desc(&tR);
  }
  if (warp >= 2) {
    // bias, gamma and beta for every tile of this CTA, in shared memory
    uint4* vec = reinterpret_cast<uint4*>(gbase + C::kOffVec);
    for (int i = threadIdx.x - 64; i < 3 * N / 8; i += 32 * kEpiWarps) {
      const int which = i / (N / 8), piece = i - which * (N / 8);
      const __nv_bfloat16* src = which == 0 ? p.bias : which == 1 ? p.gamma : p.beta;
      vec[i] = __ldg(reinterpret_cast<const uint4*>(src) + piece);
    }
  }
  tc_fence_before();
  if constexpr (kPair) {
    // both CTAs' barriers and tensor memory exist before either touches the other's
    __syncthreads();
    cluster_sync();
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  // the launch that follows may set itself up from here on; every access to
  // data an earlier launch produced (A, the residual, C) comes after it ends
  pdl_launch_dependents();
  pdl_wait();
  const int num_k = (p.K + kBK - 1) / kBK;

  if (warp == 0) {
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int t = tile0; ok && t < p.mt; t += tstride) {
        const int m0 = row_base(t);
        for (int kt = 0; kt < num_k; ++kt, ++g) {
          const int st = g % C::kStages;
          const uint32_t ph = (g / C::kStages) & 1;
          // Row tile t starts its k walk at k-step t mod num_k: the CTAs
          // running at once then read different rows of W, instead of all of
          // them asking the same L2 lines for the same k-step at once.
          const int kk = (kt + t) % num_k;
          if (!(ok = mbar_wait(bar(C::bEmpty(st)), ph ^ 1u, ctl))) break;
          const uint32_t sa = base + st * C::kStageBytes;
          if constexpr (kPair) {
            // this CTA's rows of A and its half of each chunk's W columns
            // (chunk c covers blocks 4c.. of W; rank r takes the r-th half),
            // all reported to rank 0's full barrier
            if (rank == 0) mbar_expect_tx(bar(C::bFull(st)), 2 * C::kStageBytes);
            const uint32_t full = lead_bar(C::bFull(st));
            tma_load_2d_pair(sa, &tA, full, kk * kBK, m0);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
              const int half = C::chunk_n(c) / 128;  // blocks per CTA in chunk c
#pragma unroll
              for (int u = 0; u < half / C::kPB; ++u)
                tma_load_3d_pair(sa + kABytes + (2 * c + u * C::kPB) * kWBox, &tW, full, 0,
                                 kk * kBK, 4 * c + static_cast<int>(rank) * half + u * C::kPB);
            }
          } else {
            mbar_expect_tx(bar(C::bFull(st)), C::kStageBytes);
            tma_load_2d(sa, &tA, bar(C::bFull(st)), kk * kBK, m0);
            // all NB 64 x 64 blocks of W in one copy (W viewed as [NB][K][64])
            tma_load_3d(sa + kABytes, &tW, bar(C::bFull(st)), 0, kk * kBK, 0);
          }
        }
      }
      // Every copy lands before the CTA exits.  In the pair form all of
      // them (the other CTA's too) report to rank 0's full barriers, so rank
      // 0 waits on those; the other CTA leaves only after the final cluster
      // barrier, which rank 0 reaches after this wait.
      if (rank == 0)
        for (int q = max(0, g - C::kStages); q < g; ++q)
          wait_drain(bar(C::bFull(q % C::kStages)), (q / C::kStages) & 1, p.limit_ns);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      int g = 0, i = 0;
      bool ok = true;
      for (int t = tile0; ok && t < p.mt; t += tstride, ++i) {
        // the single accumulator, once the epilogue (both CTAs' in the pair
        // form) has drained the last tile
        if (!(ok = kPair ? mbar_wait_cluster(bar(C::bAccEmpty), (i & 1) ^ 1u, ctl)
                         : mbar_wait(bar(C::bAccEmpty), (i & 1) ^ 1u, ctl)))
          break;
        tc_fence_after();
        for (int kt = 0; kt < num_k; ++kt, ++g) {
          const int st = g % C::kStages;
          const uint32_t ph = (g / C::kStages) & 1;
          if (!(ok = mbar_wait(bar(C::bFull(st)), ph, ctl))) break;
          tc_fence_after();
          const uint32_t sa = base + st * C::kStageBytes;
          const uint32_t sw = sa + kABytes;
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks) {
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
              // A: K-major, +32 bytes per 16 k; W: MN-major, +16 rows of 128
              // bytes per 16 k, 64-column boxes kWBox apart (the pair form
              // stages half of each chunk: 2 blocks per chunk)
              const uint64_t da = sdesc_sw128(sa + ks * 32, 16, 1024);
              const uint32_t acc = tmem + static_cast<uint32_t>(256 * c);
              const uint32_t accum = (kt > 0 || ks > 0) ? 1u : 0u;
              if constexpr (kPair)
                umma_ss_pair(acc, da, sdesc_sw128(sw + c * 2 * kWBox + ks * 16 * 128, kWBox, 1024),
                             idesc_bf16_f32(C::kTileM, C::chunk_n(c), false, true), accum);
              else
                umma_ss(acc, da, sdesc_sw128(sw + c * 4 * kWBox + ks * 16 * 128, kWBox, 1024),
                        idesc_bf16_f32(kBM, C::chunk_n(c), false, true), accum);
            }
          }
          if constexpr (kPair)
            umma_commit_pair_mc(bar(C::bEmpty(st)), 0x3);  // the stage is free in both CTAs
          else
            umma_commit(bar(C::bEmpty(st)));
        }
        if (ok) {
          if constexpr (kPair)
            umma_commit_pair_mc(bar(C::bAccFull), 0x3);
          else
            umma_commit(bar(C::bAccFull));
        }
      }
      if constexpr (kPair)
        umma_commit_pair(bar(C::bDrain));
      else
        umma_commit(bar(C::bDrain));
      wait_drain(bar(C::bDrain), 0, p.limit_ns);
    }
  } else {
    // epilogue: warp w may touch TMEM lanes [32 (w % 4), 32 (w % 4) + 32); the
    // two warps of a quarter (chalf 0 and 1) take the row's 64-column chunks
    // [cb_begin, cb_end) each, and merge their row statistics through shared
    // memory before the second pass
    const int quarter = warp & 3;
    const int ew = warp - 2;          // epilogue warp 0..7: its residual ring
    const int chalf = ew >> 2;
    const int cb0 = C::cb_begin(chalf), cb1 = C::cb_end(chalf);
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint4* vec = reinterpret_cast<const uint4*>(gbase + C::kOffVec);
    const uint32_t res_base = base + C::kOffRes + ew * C::kRB * kStageWarpBytes;
    const uint4* res = reinterpret_cast<const uint4*>(gbase + C::kOffRes +
                                                      ew * C::kRB * kStageWarpBytes);
    // pass 2 stages its output in the warp's first residual buffer: every
    // residual chunk of the tile has been read by then
    uint4* stg = reinterpret_cast<uint4*>(gbase + C::kOffRes + ew * C::kRB * kStageWarpBytes);
    float2* stat = reinterpret_cast<float2*>(gbase + C::kOffStat);  // [quarter][chalf][lane]
    volatile int* verdict = reinterpret_cast<volatile int*>(gbase + C::kOffStat + 4 * 2 * 32 * 8);
    const int q = lane & 7;  // the 16-byte piece this lane moves in the store transpose
    // The warp's residual rows (32 rows x 64 columns per chunk) arrive by TMA
    // in a ring of kRB buffers, 128-byte swizzled: 16-byte piece qq of row r
    // at slot qq ^ (r & 7).  Chunk g of this warp (counted across tiles)
    // uses buffer g % kRB with phase (g / kRB) & 1.
    int g_issue = 0, g_use = 0;
    auto issue_res = [&](int t_next, int cb) {
      if (lane == 0) {
        const int b = g_issue % C::kRB;
        fence_proxy_async_shared();  // the warp's reads of this buffer came first
        mbar_expect_tx(bar(C::bRes(ew, b)), kStageWarpBytes);
        tma_load_2d(res_base + b * kStageWarpBytes, &tR, bar(C::bRes(ew, b)), cb * 64,
                    row_base(t_next) + quarter * 32);
      }
      ++g_issue;
    };
    const int first = tile0;
    if (first < p.mt)
      for (int cb = cb0; cb < cb0 + C::kRB && cb < cb1; ++cb) issue_res(first, cb);
    int i = 0;
    bool ok = true;
    // Both warps of a quarter take every tile, meet at every statistics
    // exchange (a warp whose wait failed brings its verdict there) and leave
    // the loop together, so neither can wait at the exchange for a partner
    // that has gone.
    for (int t = first; t < p.mt; t += tstride, ++i) {
      ok = num_k > 0 && mbar_wait_warp(bar(C::bAccFull), i & 1, ctl);
      tc_fence_after();
      const int row0 = row_base(t) + quarter * 32;  // this warp's first row
      // ---- pass 1: v = acc + bias + R, row statistics, v back to TMEM
      float mean = 0.f, m2 = 0.f;
#pragma unroll 1
      for (int cb = cb0; ok && cb < cb1; ++cb) {
        const int n = cb * 64;
        uint32_t v[64];
        tmem_ld32(lane_base + n, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(lane_base + n + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        const int b = g_use % C::kRB;
        ok = mbar_wait_warp(bar(C::bRes(ew, b)), (g_use / C::kRB) & 1, ctl);
        ++g_use;
        tmem_ld_wait(v);
        if (!ok) break;
        const uint4* rb = res + b * (kStageWarpBytes / 16);
        float s = 0.f;
#pragma unroll
        for (int qq = 0; qq < 8; ++qq) {
          const uint4 r = rb[lane * 8 + (qq ^ (lane & 7))];
          const uint4 bi = vec[n / 8 + qq];
          const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
          const uint32_t bw[4] = {bi.x, bi.y, bi.z, bi.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float lo = __uint_as_float(v[8 * qq + 2 * k]) + bf16_lo(bw[k]) + bf16_lo(rw[k]);
            const float hi =
                __uint_as_float(v[8 * qq + 2 * k + 1]) + bf16_hi(bw[k]) + bf16_hi(rw[k]);
            v[8 * qq + 2 * k] = __float_as_uint(lo);
            v[8 * qq + 2 * k + 1] = __float_as_uint(hi);
            s += lo + hi;
          }
        }
        __syncwarp();  // every lane has read the buffer before it is refilled
        if (cb + C::kRB < cb1) issue_res(t, cb + C::kRB);
        // this chunk's mean and centred sum of squares, then the pairwise merge
        const float mc = s * (1.f / 64.f);
        float qc = 0.f;
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          const float d = __uint_as_float(v[k]) - mc;
          qc = fmaf(d, d, qc);
        }
        if (cb == cb0) {
          mean = mc;
          m2 = qc;
        } else {
          const float na = 64.f * (cb - cb0), nt = na + 64.f;
          const float delta = mc - mean;
          mean = fmaf(delta, 64.f / nt, mean);
          m2 = m2 + qc + delta * delta * (na * 64.f / nt);
        }
        tmem_st32(lane_base + n, *reinterpret_cast<const uint32_t(*)[32]>(&v[0]));
        tmem_st32(lane_base + n + 32, *reinterpret_cast<const uint32_t(*)[32]>(&v[32]));
      }
      ok = __all_sync(0xffffffffu, ok);
      tmem_st_wait();
      // the two halves' statistics, merged in the same order by both warps
      // of the quarter (so that they normalise with identical values)
      stat[(quarter * 2 + chalf) * 32 + lane] = make_float2(mean, m2);
      if (lane == 0) verdict[quarter * 2 + chalf] = ok ? 1 : 0;
      named_barrier_sync(1 + quarter, 64);
      const float2 sa = stat[(quarter * 2 + 0) * 32 + lane];
      const float2 sb = stat[(quarter * 2 + 1) * 32 + lane];
      const bool both = verdict[quarter * 2] != 0 && verdict[quarter * 2 + 1] != 0;
      named_barrier_sync(1 + quarter, 64);  // both have read before the next tile writes
      if (!both) break;
      {
        const float na = 64.f * C::cb_end(0), nb = 64.f * (NB - C::cb_end(0));
        const float delta = sb.x - sa.x;
        mean = nb > 0.f ? fmaf(delta, nb / static_cast<float>(N), sa.x) : sa.x;
        m2 = nb > 0.f ? sa.y + sb.y + delta * delta * (na * nb / static_cast<float>(N)) : sa.y;
      }
      const float inv = 1.f / sqrtf(m2 * (1.f / static_cast<float>(N)) + p.eps);
      // ---- pass 2: y = (v - mean) * inv * gamma + beta, stored row-major
#pragma unroll 1
      for (int cb = cb0; cb < cb1; ++cb) {
        const int n = cb * 64;
        uint32_t v[64];
        tmem_ld32(lane_base + n, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(lane_base + n + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_ld_wait(v);
#pragma unroll
        for (int qq = 0; qq < 8; ++qq) {
          const uint4 gv = vec[N / 8 + n / 8 + qq];
          const uint4 bv = vec[2 * (N / 8) + n / 8 + qq];
          const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
          const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float lo = fmaf((__uint_as_float(v[8 * qq + 2 * k]) - mean) * inv, bf16_lo(gw[k]),
                                  bf16_lo(bw[k]));
            const float hi = fmaf((__uint_as_float(v[8 * qq + 2 * k + 1]) - mean) * inv,
                                  bf16_hi(gw[k]), bf16_hi(bw[k]));
            v[8 * qq + 2 * k] = __float_as_uint(lo);
            v[8 * qq + 2 * k + 1] = __float_as_uint(hi);
          }
        }
        if (!p.out_f32) {
#pragma unroll
          for (int qq = 0; qq < 8; ++qq) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[8 * qq + 0]), __uint_as_float(v[8 * qq + 1]));
            w.y = pack_bf16x2(__uint_as_float(v[8 * qq + 2]), __uint_as_float(v[8 * qq + 3]));
            w.z = pack_bf16x2(__uint_as_float(v[8 * qq + 4]), __uint_as_float(v[8 * qq + 5]));
            w.w = pack_bf16x2(__uint_as_float(v[8 * qq + 6]), __uint_as_float(v[8 * qq + 7]));
            stg[lane * 8 + (qq ^ (lane & 7))] = w;
          }
          __syncwarp();
          __nv_bfloat16* Cb = static_cast<__nv_bfloat16*>(p.C);
#pragma unroll
          for (int g4 = 0; g4 < 8; ++g4) {
            const int rr = 4 * g4 + (lane >> 3);
            const uint4 w = stg[rr * 8 + (q ^ (rr & 7))];
            if (row0 + rr < p.M)
              reinterpret_cast<uint4*>(Cb + static_cast<size_t>(row0 + rr) * N + n)[q] = w;
          }
          __syncwarp();
        } else {
          // fp32: 32 columns (128 bytes) of every row per round
          float* Cf = static_cast<float*>(p.C);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int qq = 0; qq < 8; ++qq)
              stg[lane * 8 + (qq ^ (lane & 7))] =
                  make_uint4(v[32 * h + 4 * qq], v[32 * h + 4 * qq + 1], v[32 * h + 4 * qq + 2],
                             v[32 * h + 4 * qq + 3]);
            __syncwarp();
#pragma unroll
            for (int g4 = 0; g4 < 8; ++g4) {
              const int rr = 4 * g4 + (lane >> 3);
              const uint4 w = stg[rr * 8 + (q ^ (rr & 7))];
              if (row0 + rr < p.M)
                reinterpret_cast<uint4*>(Cf + static_cast<size_t>(row0 + rr) * N + n + 32 * h)[q] = w;
            }
            __syncwarp();
          }
        }
      }
      // the accumulator may take the next tile once every epilogue warp (of
      // both CTAs in the pair form) has read it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kPair)
          mbar_arrive_cluster(lead_bar(C::bAccEmpty));
        else
          mbar_arrive(bar(C::bAccEmpty));
      }
      // the next tile's first residual chunks load while its MMAs run (the
      // staging buffer has been read: the __syncwarp above)
      if (t + tstride < p.mt)
        for (int cb = cb0; cb < cb0 + C::kRB && cb < cb1; ++cb) issue_res(t + tstride, cb);
    }
    // every residual copy this warp issued lands before the CTA exits
    for (int g = max(0, g_issue - C::kRB); g < g_issue; ++g)
      if (lane == 0) wait_drain(bar(C::bRes(ew, g % C::kRB)), (g / C::kRB) & 1, p.limit_ns);
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) {
    // no CTA of the pair leaves (or frees its tensor memory) while the
    // other's products, copies or barrier arrivals may still reach it
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair<C::kTmemCols>(tmem);
  } else {
    tc_fence_after();
    if (warp == 1) tmem_dealloc<C::kTmemCols>(tmem);
  }
}

int current_sm_count() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
    return v;
  return 1;
}

// Clusters of two of this kernel that can be resident at once on the current
// device (each CTA fills an SM, and a cluster sits inside one GPC), asked
// once per device; half the SM count if the query fails.
template <int NB>
int pair_slots() {
  constexpr int kDevs = 16;
  static int cache[kDevs];
  int dev = 0;
  const int fallback = current_sm_count() / 2 > 0 ? current_sm_count() / 2 : 1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return fallback;
  if (dev < kDevs && cache[dev] > 0) return cache[dev];
  using C = LnCfg<NB, true>;
  auto kern = gemm_ln_bf16_kernel<NB, true>;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  if (n <= 0) n = fallback;
  if (dev < kDevs) cache[dev] = n;
  return n;
}

template <int NB>
cudaError_t launch_nb(const GemmLnArgs& g, const DeviceCtl& ctl) {
  // the pair form wherever the column chunks split into whole blocks
  constexpr bool kPair = NB % 2 == 0;
  using C = LnCfg<NB, kPair>;
  CUtensorMap ta, tw, tr;
  const uint64_t adims[2] = {static_cast<uint64_t>(g.K), static_cast<uint64_t>(g.M)};
  const uint64_t astr[1] = {static_cast<uint64_t>(g.K) * 2};
  const uint32_t abox[2] = {64, 128};
  // W [K, N] as a 3-D tensor (64 columns, K rows, NB column blocks): one
  // copy brings kPB blocks (all NB of them in the single-CTA form)
  const uint64_t wdims[3] = {64, static_cast<uint64_t>(g.K), static_cast<uint64_t>(NB)};
  const uint64_t wstr[2] = {static_cast<uint64_t>(C::N) * 2, 128};
  const uint32_t wbox[3] = {64, 64, static_cast<uint32_t>(C::kPB)};
  if (!encode_tensor_map(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(g.A), adims,
                         astr, abox, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(g.W), wdims,
                         wstr, wbox, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // the residual [M, N]: 32-row x 64-column boxes (one epilogue warp's chunk)
  const uint64_t rdims[2] = {static_cast<uint64_t>(C::N), static_cast<uint64_t>(g.M)};
  const uint64_t rstr[1] = {static_cast<uint64_t>(C::N) * 2};
  const uint32_t rbox[2] = {64, 32};
  if (!encode_tensor_map(&tr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(g.resid),
                         rdims, rstr, rbox, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  GemmLnParams p{};
  p.C = g.C;
  p.bias = static_cast<const __nv_bfloat16*>(g.bias);
  p.resid = static_cast<const __nv_bfloat16*>(g.resid);
  p.gamma = static_cast<const __nv_bfloat16*>(g.gamma);
  p.beta = static_cast<const __nv_bfloat16*>(g.beta);
  p.eps = g.eps;
  p.out_f32 = g.out_dtype == MHA_F32 ? 1 : 0;
  p.M = g.M;
  p.K = g.K;
  p.mt = (g.M + C::kTileM - 1) / C::kTileM;
  p.err = ctl.err;
  p.limit_ns = ctl.limit_ns;
  auto kern = gemm_ln_bf16_kernel<NB, kPair>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  if constexpr (kPair) {
    // one cluster of two per tile, as many as can be resident at once
    const int slots = pair_slots<NB>();
    const int pairs = p.mt < slots ? p.mt : slots;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = g.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, ta, tw, tr, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  } else {
    // one CTA per SM at most (tensor memory and shared memory admit no second)
    const int sms = current_sm_count();
    const int grid = p.mt < sms ? p.mt : sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = g.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, ta, tw, tr, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
}

}  // namespace

bool gemm_ln_bf16_supported(int N) { return N >= 64 && N <= 512 && N % 64 == 0; }

cudaError_t launch_gemm_ln_bf16(const GemmLnArgs& g, const DeviceCtl& ctl) {
  if (g.M == 0) return cudaSuccess;
  if (!gemm_ln_bf16_supported(g.N) || g.K < 1) return cudaErrorInvalidValue;
  switch (g.N / 64) {
    case 1: return launch_nb<1>(g, ctl);
    case 2: return launch_nb<2>(g, ctl);
    case 3: return launch_nb<3>(g, ctl);
    case 4: return launch_nb<4>(g, ctl);
    case 5: return launch_nb<5>(g, ctl);
    case 6: return launch_nb<6>(g, ctl);
    case 7: return launch_nb<7>(g, ctl);
    default: return launch_nb<8>(g, ctl);
  }
}

}  // namespace mha
