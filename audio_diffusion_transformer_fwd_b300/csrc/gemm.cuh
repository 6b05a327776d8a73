// Persistent tcgen05 GEMMs for the block's four projections:
//   C[m][n] = epilogue( sum_k A[m][k] * B[n][k] )     A, B BF16, K-major
// A = activations [M tokens][K], B = a Linear weight [N out][K in].
// Two kernels compute the same sums in the same order: the CTA-pair kernel
// at the end of this file (the one the library launches) and the
// single-CTA kernel below (kept as its A/B reference and for the int8-code
// variant in gemm_i8.cuh).
//
// Single-CTA kernel: one CTA per SM walks output tiles of 128 x 256.  Warp 0 streams A/B
// k-blocks (64 wide) into a 4-deep shared-memory ring with TMA (128-byte
// swizzle); one thread of warp 1 issues tcgen05.mma (M=128, N=256, K=16)
// into one of two fp32 TMEM accumulators; warps 2-5 drain the other
// accumulator through the epilogue, so the epilogue of tile i overlaps the
// main loop of tile i+1.
//
// Epilogues:
//   kEpiStore  C = bf16(acc)                          (out-projection, FC2)
//   kEpiGelu   C = bf16(GELU_tanh(acc))               (FC1)
//   kEpiQKV    3D RoPE on the Q and K thirds, then Q/K stored head-major
//              [H][M][Dh] and V transposed [H][Dh][ld] for the attention
//              kernel's K-major operands ([linlog] "h3.c 的核心设计": Q/K/V
//              routed straight into head-major attention inputs).
#pragma once
#include "ptx.cuh"

namespace h3 {

enum { kEpiStore = 0, kEpiGelu = 1, kEpiQKV = 2 };

constexpr int kGemmBM = 128;
constexpr int kGemmBN = 256;
constexpr int kGemmBK = 64;
constexpr int kGemmStages = 4;
constexpr int kGemmThreads = 192;
constexpr int kGemmABytes = kGemmBM * kGemmBK * 2;   // 16 KB
constexpr int kGemmBBytes = kGemmBN * kGemmBK * 2;   // 32 KB
constexpr int kGemmStageBytes = kGemmABytes + kGemmBBytes;
constexpr int kGemmTmemCols = 2 * kGemmBN;           // two accumulators
constexpr int kGemmGroupN = 16;                      // default tile raster: bands of 16 N-tiles
constexpr size_t kGemmSmemBytes = 1024 /*align slack*/ + kGemmStages * kGemmStageBytes + 256;

struct GemmArgs {
  int M, N, K;
  int tiles_m, tiles_n, num_tiles;
  __nv_bfloat16* c;   // kEpiStore / kEpiGelu
  int ldc;
  // kEpiQKV
  __nv_bfloat16* q;
  __nv_bfloat16* k;
  __nv_bfloat16* vt;
  int vt_ld;
  int d;
  int head_dim;
  const float2* rope;  // [M][head_dim/2] (cos, sin)
  // Test hook, -1 in every normal launch: the producer of CTA 0 stops before
  // k-block `stall_kb` of its first tile and issues nothing more, so the MMA
  // thread's wait on that stage runs out (see h3dit_test_stall_next_gemm).
  int stall_kb;
  int band_n;   // tile raster: output tiles are walked in bands of band_n N-tiles, M fastest within a band
  // CTA-pair kernel: tiles full_tiles .. num_tiles-1 (a last wave that would
  // leave at least half of the pairs idle) are computed as two 256 x 128
  // halves each; num_units = full_tiles + 2 * (num_tiles - full_tiles).
  // Other kernels walk num_tiles whole tiles.
  int full_tiles, num_units;
};

// GELU, tanh form: 0.5 x (1 + tanh(u)) with u = sqrt(2/pi) (x + 0.044715 x^3),
// evaluated as x / (1 + exp(-2u)) (the same function: 1 + tanh(u) =
// 2 / (1 + exp(-2u))) with the fast exponential and division intrinsics;
// their relative error (~1e-6) is far below the BF16 rounding of the
// result.  Large |x|: exp(-2u) -> inf gives -0, exp(-2u) -> 0 gives x.
__device__ __forceinline__ float gelu_tanh_f(float x) {
  const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
  const float k1 = 0.044715f;
  const float u = k0 * fmaf(k1 * x, x * x, x);
  return __fdividef(x, 1.0f + __expf(-2.0f * u));
}

__device__ __forceinline__ void gemm_tile_coords(int t, const GemmArgs& a, int& mb, int& nb) {
  const int per_group = a.band_n * a.tiles_m;
  const int g = t / per_group;
  const int r = t - g * per_group;
  const int n_first = g * a.band_n;
  const int gn = min(a.band_n, a.tiles_n - n_first);
  mb = r / gn;
  nb = n_first + (r - mb * gn);
}

template <int EPI>
__device__ __forceinline__ void gemm_epilogue_chunk(const GemmArgs& a, float (&v)[32], int grow,
                                                    int gcol) {
  if (grow >= a.M) return;
  if (EPI == kEpiStore || EPI == kEpiGelu) {
    uint32_t p[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float x0 = v[2 * i], x1 = v[2 * i + 1];
      if (EPI == kEpiGelu) {
        x0 = gelu_tanh_f(x0);
        x1 = gelu_tanh_f(x1);
      }
      p[i] = pack_bf16x2(x0, x1);
    }
    uint4* dst = reinterpret_cast<uint4*>(a.c + static_cast<size_t>(grow) * a.ldc + gcol);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
  } else {
    const int region = gcol / a.d;          // 0 = Q, 1 = K, 2 = V
    const int cin = gcol - region * a.d;
    const int head = cin / a.head_dim;
    const int dh0 = cin - head * a.head_dim;
    if (region < 2) {
      const float4* cs = reinterpret_cast<const float4*>(
          a.rope + static_cast<size_t>(grow) * (a.head_dim / 2) + dh0 / 2);
      uint32_t p[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 t = __ldg(cs + i);   // (cos, sin) of two consecutive pairs
        const float a0 = v[4 * i], b0 = v[4 * i + 1], a1 = v[4 * i + 2], b1 = v[4 * i + 3];
        p[2 * i] = pack_bf16x2(a0 * t.x - b0 * t.y, a0 * t.y + b0 * t.x);
        p[2 * i + 1] = pack_bf16x2(a1 * t.z - b1 * t.w, a1 * t.w + b1 * t.z);
      }
      __nv_bfloat16* base = region == 0 ? a.q : a.k;
      uint4* dst = reinterpret_cast<uint4*>(
          base + (static_cast<size_t>(head) * a.M + grow) * a.head_dim + dh0);
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
    } else {
      __nv_bfloat16* dst = a.vt + (static_cast<size_t>(head) * a.head_dim + dh0) * a.vt_ld + grow;
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[static_cast<size_t>(i) * a.vt_ld] = __float2bfloat16_rn(v[i]);
    }
  }
}

template <int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const GemmArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kGemmStages * kGemmABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kGemmStages * kGemmStageBytes);
  // bars: full[S], empty[S], tfull[2], tempty[2], drain
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * kGemmStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + kGemmStages);
  const uint32_t tfull0 = smem_u32(bars + 2 * kGemmStages);
  const uint32_t tempty0 = smem_u32(bars + 2 * kGemmStages + 2);
  const uint32_t drain = smem_u32(bars + 2 * kGemmStages + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull0 + 8 * i, 1);
      mbar_init(tempty0 + 8 * i, 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), kGemmTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int kblocks = args.K / kGemmBK;
  grid_dep_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const int stall_kb = blockIdx.x == 0 ? args.stall_kb : -1;
      for (int t = blockIdx.x; t < args.num_tiles && ok; t += gridDim.x) {
        int mb, nb;
        gemm_tile_coords(t, args, mb, nb);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (t == blockIdx.x && kb == stall_kb) { ok = false; break; }
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag)) { ok = false; break; }
          const uint32_t fb = full0 + 8 * stage;
          mbar_arrive_expect_tx(fb, kGemmStageBytes);
          tma_load_2d(smem_u32(sA + stage * kGemmABytes), &tmA, fb, kb * kGemmBK, mb * kGemmBM);
          tma_load_2d(smem_u32(sB + stage * kGemmBBytes), &tmB, fb, kb * kGemmBK, nb * kGemmBN);
          if (++stage == kGemmStages) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        // let loads already in flight land before the CTA exits
        for (int s = 0; s < kGemmStages; ++s) mbar_wait_drain(full0 + 8 * s, phase);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(kGemmBM, kGemmBN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < args.num_tiles && ok; t += gridDim.x, ++it) {
        const int acc = it & 1;
        if (!mbar_wait(tempty0 + 8 * acc, ((it >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kGemmBN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * kGemmABytes);
          const uint32_t b0 = smem_u32(sB + stage * kGemmBBytes);
#pragma unroll
          for (int k = 0; k < kGemmBK / 16; ++k) {
            tc_mma_bf16(d_tmem, sdesc_k128(a0 + 32 * k), sdesc_k128(b0 + 32 * k), idesc,
                        (kb | k) != 0);
          }
          tc_commit(empty0 + 8 * stage);
          if (++stage == kGemmStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(tfull0 + 8 * acc);
      }
      // every MMA issued by this thread has completed once `drain` flips
      tc_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ---------------- epilogue warps 2..5: TMEM lane quarter = warp % 4
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    int it = 0;
    for (int t = blockIdx.x; t < args.num_tiles; t += gridDim.x, ++it) {
      int mb, nb;
      gemm_tile_coords(t, args, mb, nb);
      const int acc = it & 1;
      if (!mbar_wait(tfull0 + 8 * acc, (it >> 1) & 1, abort_flag)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kGemmBN;
      const int grow = mb * kGemmBM + row;
#pragma unroll 1
      for (int c = 0; c < kGemmBN / 32; ++c) {
        float v[32];
        tmem_ld32(tbase + c * 32, v);
        gemm_epilogue_chunk<EPI>(args, v, grow, nb * kGemmBN + c * 32);
      }
      tc_fence_before();
      mbar_arrive(tempty0 + 8 * acc);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kGemmTmemCols);
}

}  // namespace h3

namespace h3 {

// ---------------------------------------------------------------------------
// The same GEMM on CTA pairs (tcgen05 cta_group::2).  A cluster of two CTAs
// on two SMs computes 256 x 256 output tiles: each CTA streams its own 128 A
// rows and half (128 rows) of the 256 weight rows of a k-block, and rank 0
// issues one M = 256, N = 256 MMA per 16 channels that reads both CTAs'
// shared memory; each CTA's tensor memory receives its own 128 rows.  Per SM
// a k-block is 32 KB of operands instead of 48 KB, so the same shared memory
// holds a 6-deep ring (3072 cycles of MMA work in flight instead of 2048)
// and a third less data crosses L2.  Roles per CTA as in the single-CTA
// kernel: warp 0 TMA, warp 1 MMA (rank 0 only; both allocate), warps 2-5
// epilogue.  Stage completion: rank 0 expects both CTAs' bytes on its own
// full barrier, which both CTAs' copies complete; the MMA commit arrives on
// the empty (and accumulator-full) barriers of both CTAs; the epilogue
// threads of both CTAs arrive on rank 0's accumulator-empty barrier.
// Tail: when the last wave of whole tiles would occupy at most half of the
// pairs, those tiles are split into 256 x 128 halves (M256 N128 MMAs, each
// CTA loading 64 weight rows), so twice as many pairs share the last wave.
constexpr int kPairStages = 6;
constexpr int kPairRows = 128;                       // A rows and B rows per CTA per tile
constexpr int kPairABytes = kPairRows * kGemmBK * 2;  // 16 KB
constexpr int kPairBBytes = kPairRows * kGemmBK * 2;  // 16 KB
constexpr int kPairStageBytes = kPairABytes + kPairBBytes;
constexpr size_t kPairSmemBytes = 1024 + kPairStages * kPairStageBytes + 256;

// Work unit u of the CTA-pair kernel: a whole 256 x 256 tile (half = -1) or
// the left (0) / right (1) 128 columns of one.  Every output element is the
// same k-ordered sum either way.
__device__ __forceinline__ void pair_unit(int u, const GemmArgs& a, int& mb, int& nb, int& half) {
  if (u < a.full_tiles) {
    gemm_tile_coords(u, a, mb, nb);
    half = -1;
  } else {
    const int h = u - a.full_tiles;
    gemm_tile_coords(a.full_tiles + (h >> 1), a, mb, nb);
    half = h & 1;
  }
}

template <int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmBh, const GemmArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kPairStages * kPairABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPairStages * kPairStageBytes);
  // bars: full[S], empty[S], tfull[2], tempty[2], drain
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * kPairStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster = blockIdx.x >> 1;
  const int clusters = gridDim.x >> 1;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + kPairStages);
  const uint32_t tfull0 = smem_u32(bars + 2 * kPairStages);
  const uint32_t tempty0 = smem_u32(bars + 2 * kPairStages + 2);
  const uint32_t drain = smem_u32(bars + 2 * kPairStages + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull0 + 8 * i, 1);
      mbar_init(tempty0 + 8 * i, 2 * 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_holder), kGemmTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  // both CTAs' barriers are initialised before either CTA signals the other
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int kblocks = args.K / kGemmBK;
  grid_dep_wait();
  const uint32_t full0_lead = mapa_shared(full0, 0);
  const uint32_t tempty0_lead = mapa_shared(tempty0, 0);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const int stall_kb = blockIdx.x == 0 ? args.stall_kb : -1;
      for (int u = cluster; u < args.num_units && ok; u += clusters) {
        int mb, nb, half;
        pair_unit(u, args, mb, nb, half);
        // a half unit: 64 of its 128 weight rows per CTA
        const uint32_t bytes = half < 0 ? 2 * kPairStageBytes : 2 * (kPairABytes + kPairBBytes / 2);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (u == cluster && kb == stall_kb) { ok = false; break; }
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag)) { ok = false; break; }
          if (rank == 0) mbar_arrive_expect_tx(full0 + 8 * stage, bytes);
          const uint32_t fb = full0_lead + 8 * stage;
          tma_load_2d_pair(smem_u32(sA + stage * kPairABytes), &tmA, fb, kb * kGemmBK,
                           mb * (2 * kPairRows) + rank * kPairRows);
          if (half < 0)
            tma_load_2d_pair(smem_u32(sB + stage * kPairBBytes), &tmB, fb, kb * kGemmBK,
                             nb * kGemmBN + rank * kPairRows);
          else
            tma_load_2d_pair(smem_u32(sB + stage * kPairBBytes), &tmBh, fb, kb * kGemmBK,
                             nb * kGemmBN + half * (kGemmBN / 2) + rank * (kPairRows / 2));
          if (++stage == kPairStages) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok && rank == 0) {
        // let copies already in flight (this CTA's and the peer's, all
        // counted here) land before the CTA exits
        for (int s = 0; s < kPairStages; ++s) mbar_wait_drain(full0 + 8 * s, phase);
      }
    }
  } else if (warp == 1) {
    if (rank == 0) {
      // ---------------- MMA issuer (rank 0 of the pair): the whole warp runs
      // the loop converged, one elected lane issues the MMAs and commits
      auto wait_all = [&](uint32_t bar, uint32_t par) {
        return __all_sync(0xffffffffu, mbar_wait(bar, par, abort_flag));
      };
      constexpr uint32_t idesc_full = idesc_bf16_f32(2 * kPairRows, kGemmBN);
      constexpr uint32_t idesc_half = idesc_bf16_f32(2 * kPairRows, kGemmBN / 2);
      const uint32_t a_lo0 = sdesc_lo(smem_u32(sA));
      const uint32_t b_lo0 = sdesc_lo(smem_u32(sB));
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int u = cluster; u < args.num_units && ok; u += clusters, ++it) {
        const uint32_t idesc = u < args.full_tiles ? idesc_full : idesc_half;
        const int acc = it & 1;
        if (!wait_all(tempty0 + 8 * acc, ((it >> 1) & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kGemmBN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_all(full0 + 8 * stage, phase)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_lo = a_lo0 + stage * (kPairABytes >> 4);
          const uint32_t b_lo = b_lo0 + stage * (kPairBBytes >> 4);
          static_assert(kGemmBK == 64, "one four-MMA group per k-block");
          tc_mma_k64_elect<true>(d_tmem, a_lo, b_lo, idesc, kb != 0);
          tc_commit_pair_elect(empty0 + 8 * stage, 0x3);
          if (++stage == kPairStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit_pair_elect(tfull0 + 8 * acc, 0x3);
      }
      // every MMA issued by the elected lane has completed once `drain` flips
      tc_commit_pair_elect(drain, 0x1);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ---------------- epilogue warps 2..5 (both CTAs): TMEM lane quarter = warp % 4
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    int it = 0;
    for (int u = cluster; u < args.num_units; u += clusters, ++it) {
      int mb, nb, half;
      pair_unit(u, args, mb, nb, half);
      const int acc = it & 1;
      if (!mbar_wait(tfull0 + 8 * acc, (it >> 1) & 1, abort_flag)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kGemmBN;
      const int grow = mb * (2 * kPairRows) + static_cast<int>(rank) * kPairRows + row;
      const int col0 = nb * kGemmBN + (half < 0 ? 0 : half * (kGemmBN / 2));
      const int chunks = (half < 0 ? kGemmBN : kGemmBN / 2) / 32;
#pragma unroll 1
      for (int c = 0; c < chunks; ++c) {
        float v[32];
        tmem_ld32(tbase + c * 32, v);
        gemm_epilogue_chunk<EPI>(args, v, grow, col0 + c * 32);
      }
      tc_fence_before();
      mbar_arrive_cluster(tempty0_lead + 8 * acc);
    }
  }

  // neither CTA frees its tensor memory (or exits) while the pair's MMAs or
  // the other CTA's copies may still touch it
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kGemmTmemCols);
}

}  // namespace h3
