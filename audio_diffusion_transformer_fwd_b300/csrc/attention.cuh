// Flash-style full attention on tcgen05 ([alphalab] model facts: the public
// H3-Base runs full, non-causal attention over the joint sequence).
//
// One CTA owns 128 query rows of one head and walks all keys in tiles of 128:
//   S_j   = Q K_j^T            tcgen05.mma into one of two TMEM S buffers
//   P_j   = exp2(S_j * c - m)  4 softmax warps, one query row per thread,
//                               written as BF16 into one of two shared P tiles
//   O    += P_j V_j            tcgen05.mma accumulating in TMEM
// with c = log2(e)/sqrt(Dh).  The running max m is only raised when a tile's
// max exceeds it by more than 8 (a factor 256): then the row's O in TMEM and
// its running sum are rescaled first.  Otherwise the stale max is kept; the
// result is the same softmax because O and the sum use the same m.
//
// Operands are K-major BF16 in the 128-byte swizzle: Q and K come from the
// head-major [H][N][Dh] tensors, V from its transpose [H][Dh][ld] written by
// the QKV epilogue, and P is written by the softmax warps in the same
// swizzled layout.  Keys past N read as zeros (TMA bounds) and are masked to
// -inf; query rows past N are computed and not stored.
#pragma once
#include "ptx.cuh"

namespace h3 {

constexpr int kAttnBQ = 128;
constexpr int kAttnBKV = 128;
constexpr int kAttnThreads = 192;   // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr float kAttnRescaleLog2 = 8.0f;

template <int DH>
struct AttnSmem {
  static constexpr int kQBytes = kAttnBQ * DH * 2;
  static constexpr int kKBytes = kAttnBKV * DH * 2;
  static constexpr int kVBytes = DH * kAttnBKV * 2;
  static constexpr int kPBytes = kAttnBQ * kAttnBKV * 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBytes;                 // 2 stages
  static constexpr int kVOff = kKOff + 2 * kKBytes;             // 2 stages
  static constexpr int kPOff = kVOff + 2 * kVBytes;             // 2 buffers
  static constexpr int kBarOff = kPOff + 2 * kPBytes;
  static constexpr size_t kTotal = 1024 + kBarOff + 256;
};

struct AttnArgs {
  int n;          // tokens
  int heads;
  __nv_bfloat16* o;   // [n][heads*DH]
  float scale_log2;
};

template <int DH>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const AttnArgs args) {
  using L = AttnSmem<DH>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  // bars: q_full, kv_full[2], kv_empty[2], s_full[2], s_empty[2], p_full[2], pv_done[2], drain
  const uint32_t b_qfull = smem_u32(bars + 0);
  const uint32_t b_kvfull = smem_u32(bars + 1);
  const uint32_t b_kvempty = smem_u32(bars + 3);
  const uint32_t b_sfull = smem_u32(bars + 5);
  const uint32_t b_sempty = smem_u32(bars + 7);
  const uint32_t b_pfull = smem_u32(bars + 9);
  const uint32_t b_pvdone = smem_u32(bars + 11);
  const uint32_t b_drain = smem_u32(bars + 13);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * kAttnBQ;
  const int head = blockIdx.y;
  const int nkv = (args.n + kAttnBKV - 1) / kAttnBKV;

  if (threadIdx.x == 0) {
    mbar_init(b_qfull, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_kvfull + 8 * i, 1);
      mbar_init(b_kvempty + 8 * i, 1);
      mbar_init(b_sfull + 8 * i, 1);
      mbar_init(b_sempty + 8 * i, 128);
      mbar_init(b_pfull + 8 * i, 128);
      mbar_init(b_pvdone + 8 * i, 1);
    }
    mbar_init(b_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // TMEM columns: S buffers at 0 and 128, O at 256
  const uint32_t t_s = tmem_base;
  const uint32_t t_o = tmem_base + 256;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(b_qfull, L::kQBytes);
#pragma unroll
      for (int a = 0; a < DH / 64; ++a)
        tma_load_3d(smem_u32(smem + L::kQOff + a * kAttnBQ * 128), &tmQ, b_qfull, a * 64, q0, head);
      for (int j = 0; j < nkv; ++j) {
        const int st = j & 1;
        if (!mbar_wait(b_kvempty + 8 * st, ((j >> 1) & 1) ^ 1, abort_flag)) break;
        const uint32_t fb = b_kvfull + 8 * st;
        mbar_arrive_expect_tx(fb, L::kKBytes + L::kVBytes);
        uint8_t* sk = smem + L::kKOff + st * L::kKBytes;
        uint8_t* sv = smem + L::kVOff + st * L::kVBytes;
#pragma unroll
        for (int a = 0; a < DH / 64; ++a)
          tma_load_3d(smem_u32(sk + a * kAttnBKV * 128), &tmK, fb, a * 64, j * kAttnBKV, head);
#pragma unroll
        for (int a = 0; a < 2; ++a)
          tma_load_3d(smem_u32(sv + a * DH * 128), &tmV, fb, j * kAttnBKV + a * 64, 0, head);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t id_s = idesc_bf16_f32(kAttnBQ, kAttnBKV);
      constexpr uint32_t id_o = idesc_bf16_f32(kAttnBQ, DH);
      const uint32_t sq = smem_u32(smem + L::kQOff);
      bool ok = mbar_wait(b_qfull, 0, abort_flag);
      for (int j = 0; j <= nkv && ok; ++j) {
        if (j < nkv) {
          // S_j = Q K_j^T
          const int st = j & 1;
          if (!mbar_wait(b_kvfull + 8 * st, (j >> 1) & 1, abort_flag)) { ok = false; break; }
          if (!mbar_wait(b_sempty + 8 * st, ((j >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sk = smem_u32(smem + L::kKOff + st * L::kKBytes);
#pragma unroll
          for (int kk = 0; kk < DH / 16; ++kk) {
            const uint32_t off = (kk >> 2) * (kAttnBQ * 128) + (kk & 3) * 32;
            const uint32_t offk = (kk >> 2) * (kAttnBKV * 128) + (kk & 3) * 32;
            tc_mma_bf16(t_s + st * kAttnBKV, sdesc_k128(sq + off), sdesc_k128(sk + offk), id_s, kk != 0);
          }
          tc_commit(b_sfull + 8 * st);
        }
        if (j >= 1) {
          // O += P_{j-1} V_{j-1}
          const int jp = j - 1;
          const int pb = jp & 1;
          if (!mbar_wait(b_pfull + 8 * pb, (jp >> 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sp = smem_u32(smem + L::kPOff + pb * L::kPBytes);
          const uint32_t sv = smem_u32(smem + L::kVOff + pb * L::kVBytes);
#pragma unroll
          for (int kk = 0; kk < kAttnBKV / 16; ++kk) {
            const uint32_t offp = (kk >> 2) * (kAttnBQ * 128) + (kk & 3) * 32;
            const uint32_t offv = (kk >> 2) * (DH * 128) + (kk & 3) * 32;
            tc_mma_bf16(t_o, sdesc_k128(sp + offp), sdesc_k128(sv + offv), id_o, (jp | kk) != 0);
          }
          tc_commit(b_kvempty + 8 * pb);
          tc_commit(b_pvdone + 8 * pb);
        }
      }
      tc_commit(b_drain);
      mbar_wait_drain(b_drain, 0);
    }
  } else {
    // ---------------- softmax / correction warps 2..5
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = args.scale_log2;
    float m_eff = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int st = j & 1;
      if (!mbar_wait(b_sfull + 8 * st, (j >> 1) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      float s[kAttnBKV];
#pragma unroll
      for (int cc = 0; cc < kAttnBKV / 32; ++cc) {
        float v[32];
        tmem_ld32(t_s + lane_off + st * kAttnBKV + cc * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[cc * 32 + i] = v[i];
      }
      tc_fence_before();
      mbar_arrive(b_sempty + 8 * st);
      const int valid = args.n - j * kAttnBKV;
      if (valid < kAttnBKV) {
#pragma unroll
        for (int i = 0; i < kAttnBKV; ++i)
          if (i >= valid) s[i] = -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < kAttnBKV; ++i) mx = fmaxf(mx, s[i]);
      mx *= c;
      float alpha = 1.f;
      bool rescale = false;
      if (j == 0) {
        m_eff = mx;
      } else if (mx > m_eff + kAttnRescaleLog2) {
        alpha = fast_exp2(m_eff - mx);
        m_eff = mx;
        rescale = true;
      }
      l *= alpha;
      // P_j -> shared buffer j&1 (its previous reader PV_{j-2} finished:
      // waited for below at iteration j-1)
      const int pb = j & 1;
      uint8_t* sp = smem + L::kPOff + pb * L::kPBytes;
      float sum = 0.f;
#pragma unroll
      for (int ch = 0; ch < kAttnBKV / 8; ++ch) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = fast_exp2(fmaf(s[ch * 8 + 2 * e], c, -m_eff));
          const float p1 = fast_exp2(fmaf(s[ch * 8 + 2 * e + 1], c, -m_eff));
          sum += p0 + p1;
          pk[e] = pack_bf16x2(p0, p1);
        }
        // 128-byte swizzle: 16-byte chunk (ch % 8) of row `row` in atom ch / 8
        const int atom = ch >> 3;
        const int chunk = (ch & 7) ^ (row & 7);
        *reinterpret_cast<uint4*>(sp + atom * (kAttnBQ * 128) + row * 128 + chunk * 16) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      l += sum;
      // PV_{j-1} must be complete before O is rescaled, and before P buffer
      // (j+1)&1 is overwritten at the next iteration.
      if (j >= 1) {
        const int jp = j - 1;
        if (!mbar_wait(b_pvdone + 8 * (jp & 1), (jp >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int cc = 0; cc < DH / 32; ++cc) {
            float v[32];
            tmem_ld32(t_o + lane_off + cc * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= alpha;
            tmem_st32(t_o + lane_off + cc * 32, v);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(b_pfull + 8 * pb);
    }
    if (ok) {
      const int jl = nkv - 1;
      if (mbar_wait(b_pvdone + 8 * (jl & 1), (jl >> 1) & 1, abort_flag)) {
        tc_fence_after();
        const int grow = q0 + row;
        const float inv = 1.f / l;
        const int d = args.heads * DH;
#pragma unroll 1
        for (int cc = 0; cc < DH / 32; ++cc) {
          float v[32];
          tmem_ld32(t_o + lane_off + cc * 32, v);
          if (grow < args.n) {
            uint32_t p[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) p[i] = pack_bf16x2(v[2 * i] * inv, v[2 * i + 1] * inv);
            uint4* dst = reinterpret_cast<uint4*>(args.o + static_cast<size_t>(grow) * d + head * DH + cc * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

}  // namespace h3
