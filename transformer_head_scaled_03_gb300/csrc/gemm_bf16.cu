// gemm_bf16.cu -- the Q/K/V/O projections, C = A @ W (bf16 in, fp32
// accumulate in tensor memory, bf16 out), on sm_103a tcgen05 tensor cores.
//
// y = x @ W with W stored [d_in, d_out] ("32 Transformer" (ml-canon-en),
// "PyTorch Implementation"; "The Transformer" (hoshank.vercel.app), the
// multi-head equation).  The head split is folded into the store: column n
// of the projection belongs to head n / d and lands in the [B, H, L, d]
// tensor the attention kernel reads.  The output projection reads the
// concatenated heads [B, Lq, H*d] that the attention kernel writes, so the
// concat is a store layout too, never a copy.
//
// CTA tile 128 x 256, k-step 64, a 4-stage TMA ring.  A (activations) is
// K-major; W is row-major [K, N], i.e. MN-major for the MMA's B operand, and
// is loaded as four 64 x 64 blocks (64 N-columns of 128 bytes, 64 K-rows)
// by one copy: the tensor map views W as [N/64][K][64], so the box lands as
// the four blocks in a row.  (Each copy instruction costs the producer
// thread about 100 cycles; five per stage would take as long as the stage's
// MMAs.)  Warp roles: warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2-9 epilogue, two per TMEM lane quarter, each half of the
// columns (TMEM -> registers, one row per thread; then a 32-row x 64-column
// piece through a 128-byte-swizzled shared-memory buffer, which one TMA store
// writes out, or, for head splits the store's box cannot express, the
// threads themselves with whole 128-byte row segments per instruction).  The
// stores travel by TMA rather than through L1, whose bandwidth the MMAs'
// operand reads share.
// Up to three problems of one shape share a launch, which is how the Q, K
// and V projections of self-attention run as one launch.
//
// The kernel is persistent: one CTA per SM walks the output tiles (problem,
// then row tile, then column tile, so the CTAs running at once share W and
// A tiles in L2).  Two 256-column
// accumulators in tensor memory alternate, so one tile's epilogue drains
// while the next tile's MMAs run, and the TMA ring runs on across tiles.
// Launched with programmatic dependent launch: the kernel sets itself up
// while the launch before it finishes, and waits for it before touching data.
#include "internal.h"
#include "ptx.cuh"
#include "ptx_cluster.cuh"
#include "ptx_pdl.cuh"
#include "ptx_store.cuh"

namespace mha {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;           // 16 KB
constexpr int kWBox = 64 * 64 * 2;               // 8 KB: one 64(N) x 64(K) box
constexpr int kWBytes = kBK * kBN * 2;           // 32 KB
constexpr int kStageBytes = kABytes + kWBytes;   // 48 KB
constexpr int kEpiWarps = 8;   // two per TMEM lane quarter, each half of the 256 columns
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr uint32_t kTmemCols = 512;   // two kBN-column accumulators
// barriers: full[kStages], empty[kStages], acc_full[2], acc_empty[2], drain
__host__ __device__ constexpr int bFull(int s) { return s; }
__host__ __device__ constexpr int bEmpty(int s) { return kStages + s; }
__host__ __device__ constexpr int bAccFull(int b) { return 2 * kStages + b; }
__host__ __device__ constexpr int bAccEmpty(int b) { return 2 * kStages + 2 + b; }
constexpr int bDrain = 2 * kStages + 4;
constexpr int kNumBars = 2 * kStages + 5;
constexpr int kOffBar = kStages * kStageBytes;
constexpr int kOffMisc = kOffBar + 8 * kNumBars;
// epilogue staging: per epilogue warp, 32 rows x 128 bytes (64 bf16 columns),
// 1024-byte aligned: the layout is the TMA's 128-byte swizzle
constexpr int kOffStage = (kOffMisc + 16 + 1023) & ~1023;
constexpr int kStageWarpBytes = 32 * 128;
constexpr int kSmemBytes = kOffStage + kEpiWarps * kStageWarpBytes + 1024;
static_assert(kSmemBytes <= 232448, "shared memory");

struct GemmParams {
  void* C[3];
  const __nv_bfloat16* bias[3];
  int relu[3];
  int store[3];
  int L[3];
  int dh[3];
  int tstore[3];      // 1: the output leaves by TMA stores through tC*
  int M, N, K;
  int count;          // problems in the launch (1..3)
  int mt, nt;         // row and column tiles per problem
  unsigned* err;
  uint64_t limit_ns;
};

__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tA0, const __grid_constant__ CUtensorMap tA1,
                     const __grid_constant__ CUtensorMap tA2, const __grid_constant__ CUtensorMap tW0,
                     const __grid_constant__ CUtensorMap tW1, const __grid_constant__ CUtensorMap tW2,
                     const __grid_constant__ CUtensorMap tC0, const __grid_constant__ CUtensorMap tC1,
                     const __grid_constant__ CUtensorMap tC2, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kOffMisc + 4);
  auto bar = [base](int i) -> uint32_t { return base + kOffBar + 8u * i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitCtl ctl{abort_flag, p.err, p.limit_ns};
  auto map_a = [&](int z) { return z == 0 ? &tA0 : (z == 1 ? &tA1 : &tA2); };
  auto map_w = [&](int z) { return z == 0 ? &tW0 : (z == 1 ? &tW1 : &tW2); };
  auto map_c = [&](int z) { return z == 0 ? &tC0 : (z == 1 ? &tC1 : &tC2); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(bFull(s)), 1);
      mbar_init(bar(bEmpty(s)), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(bAccFull(b)), 1);
      mbar_init(bar(bAccEmpty(b)), 32 * kEpiWarps);
    }
    mbar_init(bar(bDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<kTmemCols>(smem_u32(tmem_slot));
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    for (int z = 0; z < p.count; ++z) {
      tma_prefetch_desc(map_a(z));
      tma_prefetch_desc(map_w(z));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  // the launch that follows may set itself up from here on; every access to
  // data an earlier launch may touch (A, and C it may still read) comes after
  // it ends
  pdl_launch_dependents();
  pdl_wait();

  const int num_k = (p.K + kBK - 1) / kBK;
  const int num_tiles = p.mt * p.count * p.nt;
  // tile t: problem, then row tile, then column tile, so the CTAs running
  // at once share one problem's W (and a few rows of A) in L2
  auto decode = [&](int t, int& z, int& m0, int& n0) {
    const int per_z = p.mt * p.nt;
    z = t / per_z;
    const int r = t - z * per_z;
    const int mi = r / p.nt;
    n0 = (r - mi * p.nt) * kBN;
    m0 = mi * kBM;
  };

  if (warp == 0) {
    if (lane == 0) {
      // one ring of stages across all of this CTA's tiles
      int g = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        int z, m0, n0;
        decode(t, z, m0, n0);
        const CUtensorMap* tA = map_a(z);
        const CUtensorMap* tW = map_w(z);
        for (int kt = 0; kt < num_k; ++kt, ++g) {
          const int st = g % kStages;
          const uint32_t ph = (g / kStages) & 1;
          if (!(ok = mbar_wait(bar(bEmpty(st)), ph ^ 1u, ctl))) break;
          const uint32_t sa = base + st * kStageBytes;
          mbar_expect_tx(bar(bFull(st)), kStageBytes);
          tma_load_2d(sa, tA, bar(bFull(st)), kt * kBK, m0);
          // all four 64 x 64 boxes of W in one copy (W viewed as
          // [N/64][K][64], so the box lands as four consecutive 8 KB blocks)
          tma_load_3d(sa + kABytes, tW, bar(bFull(st)), 0, kt * kBK, n0 / 64);
        }
      }
      for (int q = max(0, g - kStages); q < g; ++q)
        wait_drain(bar(bFull(q % kStages)), (q / kStages) & 1, p.limit_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN, false, true);
      int g = 0, i = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x, ++i) {
        // accumulator i % 2, once the epilogue has drained its previous tile
        const int b = i & 1;
        const uint32_t acc = tmem + static_cast<uint32_t>(b * kBN);
        if (!(ok = mbar_wait(bar(bAccEmpty(b)), ((i >> 1) & 1) ^ 1u, ctl))) break;
        tc_fence_after();
        for (int kt = 0; kt < num_k; ++kt, ++g) {
          const int st = g % kStages;
          const uint32_t ph = (g / kStages) & 1;
          if (!(ok = mbar_wait(bar(bFull(st)), ph, ctl))) break;
          tc_fence_after();
          const uint32_t sa = base + st * kStageBytes;
          const uint32_t sw = sa + kABytes;
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks) {
            // A: K-major, +32 bytes per 16 k; W: MN-major, +16 rows of 128 bytes
            umma_ss(acc, sdesc_sw128(sa + ks * 32, 16, 1024),
                    sdesc_sw128(sw + ks * 16 * 128, kWBox, 1024), kIdesc,
                    (kt > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit(bar(bEmpty(st)));
        }
        if (ok) umma_commit(bar(bAccFull(b)));
      }
      umma_commit(bar(bDrain));
      wait_drain(bar(bDrain), 0, p.limit_ns);
    }
  } else {
    // epilogue: warp w may read TMEM lanes [32*(w%4), 32*(w%4)+32); the two
    // warps of a quarter take the tile's columns [0, 128) and [128, 256)
    const int quarter = warp & 3;
    const int chalf = (warp - 2) / 4;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    int i = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++i) {
      int z, m0, n0;
      decode(t, z, m0, n0);
      const int b = i & 1;
      const bool ok = num_k > 0 && mbar_wait_warp(bar(bAccFull(b)), (i >> 1) & 1, ctl);
      if (!ok) break;
      tc_fence_after();
      const int m = m0 + row;
      const int store = p.store[z];
      const int L = p.L[z], dh = p.dh[z];
      const __nv_bfloat16* bias = p.bias[z];
      const int relu = p.relu[z];
      __nv_bfloat16* C = static_cast<__nv_bfloat16*>(p.C[z]);
      const uint32_t tbase = lane_base + static_cast<uint32_t>(b * kBN);
      // An element's offset is a row part plus a column part: row-major
      // m * N + n, or for the head split ((bb * H + hh) * L + l) * dh + c
      // with m = bb * L + l and n = hh * dh + c.  Each lane computes the row
      // part of its own row (row `row` of the tile) once per tile.
      const bool split = store == static_cast<int>(GemmStore::kHeadSplit);
      const bool tstore = p.tstore[z] != 0;
      long long row_part;
      if (split) {
        const int bb = m / L, l = m - bb * L;
        row_part = (static_cast<long long>(bb) * (p.N / dh) * L + l) * dh;
      } else {
        row_part = static_cast<long long>(m) * p.N;
      }
      auto col_part = [&](int n) -> long long {
        if (!split) return n;
        const int hh = n / dh, c = n - hh * dh;
        return static_cast<long long>(hh) * L * dh + c;
      };
      // bias (bf16) added and ReLU applied to 8 accumulators
      auto finish8 = [&](uint32_t* v8, int n) -> uint4 {
        float f[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) f[k] = __uint_as_float(v8[k]);
        if (bias) {
          const uint4 bv = __ldg(reinterpret_cast<const uint4*>(bias + n));
          const __nv_bfloat16* b8 = reinterpret_cast<const __nv_bfloat16*>(&bv);
#pragma unroll
          for (int k = 0; k < 8; ++k) f[k] += __bfloat162float(b8[k]);
        }
        if (relu) {
#pragma unroll
          for (int k = 0; k < 8; ++k) f[k] = fmaxf(f[k], 0.f);
        }
        uint4 w;
        w.x = pack_bf16x2(f[0], f[1]);
        w.y = pack_bf16x2(f[2], f[3]);
        w.z = pack_bf16x2(f[4], f[5]);
        w.w = pack_bf16x2(f[6], f[7]);
        return w;
      };
      // this warp's staging rows: 32 x 128 bytes, 16-byte piece q of row r at
      // slot q ^ (r & 7), so that both the row-wise writes and the
      // piece-wise reads take the minimum four 128-byte wavefronts
      uint4* stg = reinterpret_cast<uint4*>(gbase + kOffStage + (warp - 2) * kStageWarpBytes);
      const int cb_end = (chalf + 1) * (kBN / 64);
      int cb = chalf * (kBN / 64);
      for (; cb + 2 <= cb_end && n0 + cb * 32 + 64 <= p.N; cb += 2) {
        const int n = n0 + cb * 32;
        uint32_t v[64];
        tmem_ld32(tbase + cb * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(tbase + cb * 32 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_ld_wait(v);
        if (tstore) {
          // the previous piece's TMA store has read the staging rows
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) stg[lane * 8 + (q ^ (lane & 7))] = finish8(&v[8 * q], n + 8 * q);
        if (tstore) {
          // the warp's 32 rows x 64 columns leave in one TMA store: 2-D
          // (n, m) row-major, or 4-D (c, l, head, batch) for the head split
          fence_proxy_async_smem();
          __syncwarp();
          const int mw = m0 + quarter * 32;
          if (lane == 0 && mw < p.M) {
            const uint32_t src = smem_u32(stg);
            if (split) {
              const int bb = mw / L, hh = n / dh;
              tma_store_4d(map_c(z), src, n - hh * dh, mw - bb * L, hh, bb);
            } else {
              tma_store_2d(map_c(z), src, n, mw);
            }
            bulk_commit();
          }
          continue;
        }
        __syncwarp();
        // four rows of 128 bytes per store instruction: lane l takes piece
        // l % 8 of row 4 g4 + l / 8
        const int q = lane & 7;
        const long long cp = col_part(n + 8 * q);
#pragma unroll
        for (int g4 = 0; g4 < 8; ++g4) {
          const int rr = 4 * g4 + (lane >> 3);
          const uint4 w = stg[rr * 8 + (q ^ (rr & 7))];
          const long long rp = __shfl_sync(0xffffffffu, row_part, rr);
          if (m0 + quarter * 32 + rr < p.M) *reinterpret_cast<uint4*>(C + rp + cp) = w;
        }
        __syncwarp();  // the staging rows are rewritten by the next pair
      }
      // a trailing 32-column block (N not a multiple of 64): row by row
      for (; cb < cb_end; ++cb) {
        const int n = n0 + cb * 32;
        if (n >= p.N) break;  // uniform across the warp
        uint32_t v[32];
        tmem_ld32(tbase + cb * 32, v);
        tmem_ld_wait(v);
        if (m < p.M) {
          uint4* dst = reinterpret_cast<uint4*>(C + row_part + col_part(n));
#pragma unroll
          for (int k = 0; k < 4; ++k) dst[k] = finish8(&v[8 * k], n + 8 * k);
        }
      }
      // this accumulator may take the tile after next
      tc_fence_before();
      mbar_arrive(bar(bAccEmpty(b)));
    }
    // every TMA store of this warp has written global memory before the CTA ends
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<kTmemCols>(tmem);
}

// SMs of the current device, asked at every launch (the runtime answers from
// its cached device properties), so that each device gets its own count; 1
// if the query fails, which only shrinks the grid.
int num_sms() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
    return v;
  return 1;
}

}  // namespace

cudaError_t launch_gemm_bf16(const GemmArgs& g, const DeviceCtl& ctl) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  if (g.N % 64 != 0) return cudaErrorInvalidValue;  // W is copied in 64-column blocks
  CUtensorMap ta[3], tw[3], tc[3];
  GemmParams p{};
  for (int i = 0; i < 3; ++i) {
    const GemmProblem& pr = g.prob[i < g.count ? i : 0];
    const uint64_t adims[2] = {static_cast<uint64_t>(g.K), static_cast<uint64_t>(g.M)};
    const uint64_t astr[1] = {static_cast<uint64_t>(g.K) * 2};
    const uint32_t abox[2] = {64, 128};
    // W [K, N] as a 3-D tensor (64 columns, K rows, N/64 column blocks)
    const uint64_t wdims[3] = {64, static_cast<uint64_t>(g.K), static_cast<uint64_t>(g.N) / 64};
    const uint64_t wstr[2] = {static_cast<uint64_t>(g.N) * 2, 128};
    const uint32_t wbox[3] = {64, 64, kBN / 64};
    if (!encode_tensor_map(&ta[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pr.A),
                           adims, astr, abox, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map(&tw[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pr.W),
                           wdims, wstr, wbox, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    // C by TMA stores of 32 rows x 64 columns: row-major [M, N], or the head
    // split [B, H, L, dh] as 4-D (dh, L, H, B) when a 64-column piece lies in
    // one head and a warp's 32 rows in one batch item; otherwise (or if the
    // map cannot be made, e.g. an unaligned C) by the threads' own stores
    p.tstore[i] = 0;
    if (pr.store == GemmStore::kRowMajor) {
      const uint64_t cdims[2] = {static_cast<uint64_t>(g.N), static_cast<uint64_t>(g.M)};
      const uint64_t cstr[1] = {static_cast<uint64_t>(g.N) * 2};
      const uint32_t cbox[2] = {64, 32};
      p.tstore[i] = encode_tensor_map(&tc[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pr.C, cdims,
                                      cstr, cbox, CU_TENSOR_MAP_SWIZZLE_128B) ? 1 : 0;
    } else if (pr.dh > 0 && pr.dh % 64 == 0 && pr.L > 0 && pr.L % 32 == 0 && g.M % pr.L == 0 &&
               g.N % pr.dh == 0) {
      const uint64_t H = static_cast<uint64_t>(g.N / pr.dh), L = static_cast<uint64_t>(pr.L);
      const uint64_t dh = static_cast<uint64_t>(pr.dh);
      const uint64_t cdims[4] = {dh, L, H, static_cast<uint64_t>(g.M / pr.L)};
      const uint64_t cstr[3] = {dh * 2, L * dh * 2, H * L * dh * 2};
      const uint32_t cbox[4] = {64, 32, 1, 1};
      p.tstore[i] = encode_tensor_map(&tc[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, pr.C, cdims,
                                      cstr, cbox, CU_TENSOR_MAP_SWIZZLE_128B) ? 1 : 0;
    }
    if (!p.tstore[i]) tc[i] = tw[i];  // unused; any valid map fills the slot
    p.C[i] = pr.C;
    p.bias[i] = static_cast<const __nv_bfloat16*>(pr.bias);
    p.relu[i] = pr.relu;
    p.store[i] = static_cast<int>(pr.store);
    p.L[i] = pr.L > 0 ? pr.L : 1;
    p.dh[i] = pr.dh > 0 ? pr.dh : 1;
  }
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.count = g.count;
  p.mt = (g.M + kBM - 1) / kBM;
  p.nt = (g.N + kBN - 1) / kBN;
  p.err = ctl.err;
  p.limit_ns = ctl.limit_ns;
  cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (shared memory admits no second), or fewer
  // when there are fewer tiles
  const long long tiles = static_cast<long long>(p.mt) * p.nt * g.count;
  const int grid = static_cast<int>(tiles < num_sms() ? tiles : num_sms());
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = g.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemm_bf16_kernel, ta[0], ta[1], ta[2], tw[0], tw[1], tw[2], tc[0],
                         tc[1], tc[2], p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mha
