// Dynamic-int8 projections with exact integer accumulation on the BF16
// tensor cores ([linlog] "int8 量化：从 36 秒到 19 秒": per-token activation
// scales, per-output-channel weight scales, one activation scale per 1024
// FC2 input channels, scaled partial sums kept per group).
//
// sm_103a has no integer tcgen05.mma kind, so the int8 codes are fed to
// kind::f16 as BF16 values.  Every code is an integer in [-127, 127], exact
// in BF16, and every product is an integer of magnitude <= 16129.  A chunk
// of at most 1024 k-columns therefore has partial sums of magnitude
// <= 16129 * 1024 < 2^24: every partial sum is an integer that fp32 holds
// exactly, so the fp32 TMEM accumulator of one chunk is the exact integer
// sum whatever order the tensor core adds in.  Each chunk is drained from
// TMEM as soon as it is complete and combined in registers:
//   kI8Int:   acc = sum of the chunks in int32 (exact); the output is
//             acc * s_a[row] * s_b[col], or acc itself (kEpiAcc).
//   kI8Group: chunk g (one activation-scale group) adds s_a[row][g] * acc_g
//             to an fp32 sum in ascending g; the output is sum * s_b[col].
//
// Same pipeline as gemm_bf16_tc_kernel (128 x 256 tiles, 64-wide k-blocks in
// a 4-deep TMA ring, one thread issuing M128 N256 K16 MMAs), except that the
// two TMEM accumulators alternate per chunk rather than per tile, and eight
// epilogue warps hold the tile's running sums in registers: warp w reads
// TMEM lane quarter w % 4 and column half (w - 2) / 4, 128 columns each.
#pragma once
#include "gemm.cuh"

namespace h3 {

enum { kEpiAcc = 3 };            // raw int32 accumulator output (kI8Int only)
enum { kI8Int = 0, kI8Group = 1 };

constexpr int kI8Threads = 320;  // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue
constexpr int kI8MaxChunkKb = 16;  // 16 k-blocks of 64 = 1024 k-columns

struct I8Args {
  const float* sa;    // kI8Int: [M] per-row scales; kI8Group: [M][groups]
  int groups;         // kI8Group: scales per row (= K / (chunk_kb * 64))
  const float* sb;    // [N] per-output-channel scales
  int chunk_kb;       // k-blocks per chunk, 1..16
  int32_t* acc;       // kEpiAcc: [M][N] int32 output
};

// The epilogues of gemm_epilogue_chunk on 16 columns (a 16-column group
// never straddles a head: head_dim is 64 or 128).
// Where a thread's 128 output columns (col0, a multiple of 128) fall in the
// QKV projection: its region (Q, K or V) and the column within that region
// (head_dim is a power of two, so heads and head dims follow by shifts).
struct QkvPlace {
  int region, cin0, hd_shift;
};
__device__ __forceinline__ QkvPlace qkv_place(const GemmArgs& a, int col0) {
  QkvPlace p;
  p.region = col0 / a.d;   // d is a multiple of 256: 128 columns never straddle regions
  p.cin0 = col0 - p.region * a.d;
  p.hd_shift = a.head_dim == 128 ? 7 : 6;
  return p;
}

// The QKV epilogue on 16 columns cin .. cin+15 of a region (they never
// straddle a head): RoPE and head-major stores for Q and K (QK), V
// transposed otherwise.
template <bool QK>
__device__ __forceinline__ void i8_qkv16(const GemmArgs& a, const float (&v)[16], int grow, const QkvPlace& pl,
                                         int cin) {
  const int head = cin >> pl.hd_shift;
  const int dh0 = cin & (a.head_dim - 1);
  if constexpr (QK) {
    const float4* cs = reinterpret_cast<const float4*>(a.rope + static_cast<size_t>(grow) * (a.head_dim / 2) + dh0 / 2);
    uint32_t p[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 t = __ldg(cs + i);   // (cos, sin) of two consecutive pairs
      const float a0 = v[4 * i], b0 = v[4 * i + 1], a1 = v[4 * i + 2], b1 = v[4 * i + 3];
      p[2 * i] = pack_bf16x2(a0 * t.x - b0 * t.y, a0 * t.y + b0 * t.x);
      p[2 * i + 1] = pack_bf16x2(a1 * t.z - b1 * t.w, a1 * t.w + b1 * t.z);
    }
    __nv_bfloat16* base = pl.region == 0 ? a.q : a.k;
    uint4* dst = reinterpret_cast<uint4*>(base + (static_cast<size_t>(head) * a.M + grow) * a.head_dim + dh0);
    dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
    dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
  } else {
    __nv_bfloat16* dst = a.vt + (static_cast<size_t>(head) * a.head_dim + dh0) * a.vt_ld + grow;
#pragma unroll
    for (int i = 0; i < 16; ++i) dst[static_cast<size_t>(i) * a.vt_ld] = __float2bfloat16_rn(v[i]);
  }
}

template <int EPI>
__device__ __forceinline__ void i8_epilogue16(const GemmArgs& a, const float (&v)[16], int grow, int gcol) {
  if constexpr (EPI == kEpiStore || EPI == kEpiGelu) {
    uint32_t p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float x0 = v[2 * i], x1 = v[2 * i + 1];
      if constexpr (EPI == kEpiGelu) {
        x0 = gelu_tanh_f(x0);
        x1 = gelu_tanh_f(x1);
      }
      p[i] = pack_bf16x2(x0, x1);
    }
    uint4* dst = reinterpret_cast<uint4*>(a.c + static_cast<size_t>(grow) * a.ldc + gcol);
    dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
    dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
  } else {
    const int region = gcol / a.d;   // 0 = Q, 1 = K, 2 = V
    const int cin = gcol - region * a.d;
    const int head = cin / a.head_dim;
    const int dh0 = cin - head * a.head_dim;
    if (region < 2) {
      const float4* cs = reinterpret_cast<const float4*>(
          a.rope + static_cast<size_t>(grow) * (a.head_dim / 2) + dh0 / 2);
      uint32_t p[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 t = __ldg(cs + i);   // (cos, sin) of two consecutive pairs
        const float a0 = v[4 * i], b0 = v[4 * i + 1], a1 = v[4 * i + 2], b1 = v[4 * i + 3];
        p[2 * i] = pack_bf16x2(a0 * t.x - b0 * t.y, a0 * t.y + b0 * t.x);
        p[2 * i + 1] = pack_bf16x2(a1 * t.z - b1 * t.w, a1 * t.w + b1 * t.z);
      }
      __nv_bfloat16* base = region == 0 ? a.q : a.k;
      uint4* dst = reinterpret_cast<uint4*>(base + (static_cast<size_t>(head) * a.M + grow) * a.head_dim + dh0);
      dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
      dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
    } else {
      __nv_bfloat16* dst = a.vt + (static_cast<size_t>(head) * a.head_dim + dh0) * a.vt_ld + grow;
#pragma unroll
      for (int i = 0; i < 16; ++i) dst[static_cast<size_t>(i) * a.vt_ld] = __float2bfloat16_rn(v[i]);
    }
  }
}

// PAIR: the same kernel on CTA pairs (tcgen05 cta_group::2), as the BF16
// projections run (gemm.cuh): 256 x 256 tiles over two SMs, each CTA
// streaming its 128 A rows and 128 of the 256 weight rows per k-block into
// a 6-deep ring, rank 0 issuing M = 256 MMAs, each CTA's eight epilogue
// warps draining its own 128 rows of every chunk.  A short last wave runs
// as 256 x 128 half tiles (pair_unit), drained by the column-half-0 warps.
template <int EPI, int MODE, bool PAIR>
__global__ void __launch_bounds__(kI8Threads, 1)
    gemm_i8x_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmBh,
                       const GemmArgs args, const I8Args qa) {
  constexpr int kStages = PAIR ? kPairStages : kGemmStages;
  constexpr int kABytes = PAIR ? kPairABytes : kGemmABytes;
  constexpr int kBBytes = PAIR ? kPairBBytes : kGemmBBytes;
  constexpr int kTileM = PAIR ? 2 * kPairRows : kGemmBM;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * (kABytes + kBBytes));
  // bars: full[S], empty[S], tfull[2], tempty[2], drain
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int first = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + kStages);
  const uint32_t tfull0 = smem_u32(bars + 2 * kStages);
  const uint32_t tempty0 = smem_u32(bars + 2 * kStages + 2);
  const uint32_t drain = smem_u32(bars + 2 * kStages + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull0 + 8 * i, 1);
      mbar_init(tempty0 + 8 * i, PAIR ? 2 * 256 : 256);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_holder), kGemmTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_holder), kGemmTmemCols);
      tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync_all();
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int kblocks = args.K / kGemmBK;
  grid_dep_wait();
  const int nchunks = (kblocks + qa.chunk_kb - 1) / qa.chunk_kb;
  const uint32_t full0_lead = PAIR ? mapa_shared(full0, 0) : full0;
  // work units: whole tiles, and on CTA pairs the 256 x 128 halves of a
  // short last wave (pair_unit; the single-CTA launch has whole tiles only)
  const int units = PAIR ? args.num_units : args.num_tiles;
  const uint32_t tempty0_lead = PAIR ? mapa_shared(tempty0, 0) : tempty0;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs of a pair)
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = first; u < units && ok; u += step) {
        int mb, nb, half;
        pair_unit(u, args, mb, nb, half);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag)) { ok = false; break; }
          if constexpr (PAIR) {
            if (rank == 0)
              mbar_arrive_expect_tx(full0 + 8 * stage, half < 0 ? 2 * (kABytes + kBBytes) : 2 * (kABytes + kBBytes / 2));
            const uint32_t fb = full0_lead + 8 * stage;
            tma_load_2d_pair(smem_u32(sA + stage * kABytes), &tmA, fb, kb * kGemmBK,
                             mb * kTileM + static_cast<int>(rank) * kPairRows);
            if (half < 0)
              tma_load_2d_pair(smem_u32(sB + stage * kBBytes), &tmB, fb, kb * kGemmBK,
                               nb * kGemmBN + static_cast<int>(rank) * kPairRows);
            else
              tma_load_2d_pair(smem_u32(sB + stage * kBBytes), &tmBh, fb, kb * kGemmBK,
                               nb * kGemmBN + half * (kGemmBN / 2) + static_cast<int>(rank) * (kPairRows / 2));
          } else {
            const uint32_t fb = full0 + 8 * stage;
            mbar_arrive_expect_tx(fb, kABytes + kBBytes);
            tma_load_2d(smem_u32(sA + stage * kABytes), &tmA, fb, kb * kGemmBK, mb * kTileM);
            tma_load_2d(smem_u32(sB + stage * kBBytes), &tmB, fb, kb * kGemmBK, nb * kGemmBN);
          }
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok && rank == 0) {
        for (int s = 0; s < kStages; ++s) mbar_wait_drain(full0 + 8 * s, phase);
      }
    }
  } else if (warp == 1) {
    if (rank == 0) {
      // ---------------- MMA issuer: one accumulator per chunk, alternating;
      // the whole warp runs the loop converged, one elected lane issues
      auto wait_all = [&](uint32_t bar, uint32_t par) {
        return __all_sync(0xffffffffu, mbar_wait(bar, par, abort_flag));
      };
      constexpr uint32_t idesc_full = idesc_bf16_f32(kTileM, kGemmBN);
      constexpr uint32_t idesc_half = idesc_bf16_f32(kTileM, kGemmBN / 2);
      const uint32_t a_lo0 = sdesc_lo(smem_u32(sA));
      const uint32_t b_lo0 = sdesc_lo(smem_u32(sB));
      int stage = 0;
      uint32_t phase = 0;
      int cc = 0;   // chunks issued so far by this CTA
      bool ok = true;
      for (int u = first; u < units && ok; u += step) {
        const uint32_t idesc = u < args.full_tiles ? idesc_full : idesc_half;
        for (int ch = 0; ch < nchunks && ok; ++ch, ++cc) {
          const int acc = cc & 1;
          if (!wait_all(tempty0 + 8 * acc, ((cc >> 1) & 1) ^ 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * kGemmBN;
          const int kb0 = ch * qa.chunk_kb;
          const int kb1 = min(kblocks, kb0 + qa.chunk_kb);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!wait_all(full0 + 8 * stage, phase)) { ok = false; break; }
            tc_fence_after();
            const uint32_t a_lo = a_lo0 + stage * (kABytes >> 4);
            const uint32_t b_lo = b_lo0 + stage * (kBBytes >> 4);
            static_assert(kGemmBK == 64, "one four-MMA group per k-block");
            tc_mma_k64_elect<PAIR>(d_tmem, a_lo, b_lo, idesc, kb != kb0);
            if constexpr (PAIR) tc_commit_pair_elect(empty0 + 8 * stage, 0x3);
            else tc_commit_elect(empty0 + 8 * stage);
            if (++stage == kStages) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          if constexpr (PAIR) tc_commit_pair_elect(tfull0 + 8 * acc, 0x3);
          else tc_commit_elect(tfull0 + 8 * acc);
        }
      }
      if constexpr (PAIR) tc_commit_pair_elect(drain, 0x1);
      else tc_commit_elect(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ---------------- epilogue warps 2..9
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    int cc = 0;
    bool ok = true;
    for (int u = first; u < units && ok; u += step) {
      int mb, nb, unit_half;
      pair_unit(u, args, mb, nb, unit_half);
      const int grow = mb * kTileM + static_cast<int>(rank) * kPairRows * (PAIR ? 1 : 0) + row;
      // a half unit's 128 columns are column half 0 of the accumulator: the
      // other four warps only keep the barrier counts
      const bool cols = unit_half < 0 || half == 0;
      const bool live = cols && grow < args.M;
      const int col0 = nb * kGemmBN + (unit_half < 0 ? half : unit_half) * 128;
      int iacc[128];
      float facc[128];
      for (int ch = 0; ch < nchunks; ++ch, ++cc) {
        const int acc = cc & 1;
        __syncwarp();
        if (!mbar_wait(tfull0 + 8 * acc, (cc >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tbase =
            tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kGemmBN + half * 128;
        float sg = 0.f;
        if constexpr (MODE == kI8Group) {
          if (live) sg = __ldg(qa.sa + static_cast<size_t>(grow) * qa.groups + ch);
        }
        // 16 columns per TMEM load keeps the 128 running sums plus the
        // loaded values within the 168 registers a thread of this 10-warp
        // CTA can have (three warps share one SM sub-partition's registers)
        if (cols) {   // warp-uniform: the tensor-memory loads are warp-collective
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            float v[16];
            tmem_ld16(tbase + c8 * 16, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              if constexpr (MODE == kI8Int) {
                const int x = __float2int_rn(v[i]);   // an exact integer below 2^24
                iacc[c8 * 16 + i] = ch == 0 ? x : iacc[c8 * 16 + i] + x;
              } else {
                facc[c8 * 16 + i] = ch == 0 ? v[i] * sg : fmaf(v[i], sg, facc[c8 * 16 + i]);
              }
            }
          }
        }
        tc_fence_before();
        if constexpr (PAIR) mbar_arrive_cluster(tempty0_lead + 8 * acc);
        else mbar_arrive(tempty0 + 8 * acc);
      }
      if (!ok) break;
      if (!live) continue;
      if constexpr (EPI == kEpiAcc) {
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          int4* dst = reinterpret_cast<int4*>(qa.acc + static_cast<size_t>(grow) * args.N + col0 + c4 * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_int4(iacc[c4 * 32 + 4 * i], iacc[c4 * 32 + 4 * i + 1], iacc[c4 * 32 + 4 * i + 2],
                               iacc[c4 * 32 + 4 * i + 3]);
        }
      } else {
        float sa = 1.f;
        if constexpr (MODE == kI8Int) sa = __ldg(qa.sa + grow);
        // the 16 dequantised values of column group c8
        auto group16 = [&](int c8, float (&v)[16]) {
          const float4* sb4 = reinterpret_cast<const float4*>(qa.sb + col0 + c8 * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 s = __ldg(sb4 + i);
            const float sbv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = c8 * 16 + 4 * i + e;
              if constexpr (MODE == kI8Int) v[4 * i + e] = (static_cast<float>(iacc[j]) * sa) * sbv[e];
              else v[4 * i + e] = facc[j] * sbv[e];
            }
          }
        };
        if constexpr (EPI == kEpiQKV) {
          // the region is the same for all 128 columns: one loop per region
          // keeps the unrolled code (and its registers) to one epilogue form
          const QkvPlace pl = qkv_place(args, col0);
          if (pl.region < 2) {
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
              float v[16];
              group16(c8, v);
              i8_qkv16<true>(args, v, grow, pl, pl.cin0 + c8 * 16);
              // keep the next group's loads behind this group's stores:
              // hoisting them would need registers the running sums hold
              asm volatile("" ::: "memory");
            }
          } else {
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
              float v[16];
              group16(c8, v);
              i8_qkv16<false>(args, v, grow, pl, pl.cin0 + c8 * 16);
              asm volatile("" ::: "memory");
            }
          }
        } else {
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            float v[16];
            group16(c8, v);
            i8_epilogue16<EPI>(args, v, grow, col0 + c8 * 16);
          }
        }
      }
    }
  }

  tc_fence_before();
  if constexpr (PAIR) cluster_sync_all();
  else __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, kGemmTmemCols);
    else tmem_dealloc(tmem_base, kGemmTmemCols);
  }
}

}  // namespace h3
