// Flash-style full attention on tcgen05 ([alphalab] model facts: the public
// H3-Base runs full, non-causal attention over the joint sequence).
//
// One CTA owns 256 query rows of one head as two tiles of 128 (Q0, Q1) and
// walks all keys in tiles of 128; both query tiles share every K/V tile it
// loads.  Per key tile j and query tile i:
//   S_i   = Q_i K_j^T           tcgen05.mma (both operands in shared memory)
//                               into TMEM columns [128 i, 128 i + 128)
//   P_i   = exp2(S_i * c - m_i) softmax warpgroup i (one query row per
//                               thread), written back as BF16 into the first
//                               64 columns of S_i's own TMEM
//   O_i  += P_i V_j             tcgen05.mma with P_i read from TMEM
// with c = log2(e)/sqrt(Dh).  The MMA thread alternates the two tiles, so
// the tensor cores compute one tile's products while the other tile's
// softmax runs.  The running max m_i is raised only when a tile's max
// exceeds it by more than 8 (a factor 256): then the row's O in TMEM and its
// running sum are rescaled first; otherwise the stale max is kept, which
// gives the same softmax because O and the sum use the same m.
//
// Ordering through TMEM: S_i(j+1) overwrites the columns PV_i(j) reads P
// from; both are issued by the one MMA thread in that order and tcgen05.mma
// operations of a thread execute in issue order.  (The MMA warp runs
// converged and elect.sync over the full warp picks its issuing lane, the
// same lane every time, so every MMA and commit comes from one thread.)  The completion of S_i(j)
// (signalled by tcgen05.commit, which covers every earlier MMA of the
// thread) also implies PV_i(j-1) is complete, so the softmax warpgroup may
// rescale O_i as soon as S_i(j) has landed.
//
// The softmax of a row costs about 2 instructions per score: one 128-column
// TMEM load, 3-input max, packed (f32x2) scale-and-subtract and sums, MUFU
// exp2 (its rate on this part keeps it off the critical path), one BF16
// pack per pair and two TMEM stores.
//
// Operands are K-major BF16 in the 128-byte swizzle: Q and K come from the
// head-major [H][N][Dh] tensors, V from its transpose [H][Dh][ld] written by
// the QKV epilogue.  Keys past N read as zeros (TMA bounds) and are masked
// to probability 0; query rows past N are computed and not stored.  The
// MMA thread's operands are descriptor low words advanced by constant
// offsets (the high word is the same for all), and at Dh 128 each group of
// eight MMAs is one asm statement: that thread's instruction count shows in
// the kernel's speed.  Its whole warp runs the issue loop (waits, operand
// arithmetic, all warp-uniform) and one elected lane issues, rather than
// one lane in a divergent branch: 7 % faster.
//
// Work units are (head, 256 query rows).  A launch's CTAs are persistent:
// each walks units first, first + grid, ... with every barrier phase
// counting on, loading the next unit's query tiles (q_empty) while it
// finishes the current one, and starting the next unit's products on O
// once the epilogue has read it (o_free).  A launch with
// split = 1 runs each of its units on a cluster of two CTAs instead, key tiles
// [0, nkv/2) on rank 0 and the rest on rank 1, each with its own running
// max and sum; at the end each CTA hands its partner the partner's query
// tile (unnormalised O, max, sum) through distributed shared memory and
// finishes its own tile (rank r: tile r) by the usual two-part combine.
// The library uses it for the units of a short last wave.
#pragma once
#include <type_traits>

#include "ptx.cuh"

namespace h3 {

constexpr int kAttnBQ = 128;        // rows of one query tile
constexpr int kAttnTilesQ = 2;      // query tiles per CTA
constexpr int kAttnBKV = 128;       // keys per tile
constexpr int kAttnThreads = 384;   // warp 0 TMA, warp 1 MMA, warps 4-7 / 8-11 softmax
constexpr float kAttnRescaleLog2 = 8.0f;

template <int DH>
struct AttnSmem {
  static constexpr int kQBytes = kAttnBQ * DH * 2;
  static constexpr int kKBytes = kAttnBKV * DH * 2;
  static constexpr int kVBytes = DH * kAttnBKV * 2;
  static constexpr int kQOff = 0;                               // 2 query tiles
  static constexpr int kKOff = kQOff + kAttnTilesQ * kQBytes;   // 2 stages
  static constexpr int kVOff = kKOff + 2 * kKBytes;             // 2 stages
  static constexpr int kBarOff = kVOff + 2 * kVBytes;
  static constexpr size_t kTotal = 1024 + kBarOff + 256;
};

struct AttnArgs {
  int n;          // tokens
  int heads;
  __nv_bfloat16* o;   // [n][heads*DH]
  float scale_log2;
  int qpairs;     // 256-row query units per head
  int unit0;      // first unit (head * qpairs + query unit) of this launch
  int units;      // units of this launch; a CTA (or CTA pair) walks unit0 + first + k * stride
  int split;      // 1: CTA pairs share a unit, each taking half of the key tiles
};

template <int DH>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const AttnArgs args) {
  using L = AttnSmem<DH>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  // bars: q_full, q_empty, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2], pv_done[2],
  // o_free[2], drain
  const uint32_t b_qfull = smem_u32(bars + 0);
  const uint32_t b_qempty = smem_u32(bars + 1);
  const uint32_t b_kfull = smem_u32(bars + 2);
  const uint32_t b_kempty = smem_u32(bars + 4);
  const uint32_t b_vfull = smem_u32(bars + 6);
  const uint32_t b_vempty = smem_u32(bars + 8);
  const uint32_t b_sfull = smem_u32(bars + 10);
  const uint32_t b_pfull = smem_u32(bars + 12);
  const uint32_t b_pvdone = smem_u32(bars + 14);
  const uint32_t b_ofree = smem_u32(bars + 16);
  const uint32_t b_drain = smem_u32(bars + 18);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 19);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Units (head, 256 query rows): this CTA (pair) takes unit0 + first,
  // + stride, ...; every barrier phase below counts on across units.  With
  // split, the two CTAs of a cluster share one unit: key tiles [0, nkv/2)
  // on rank 0, the rest on rank 1.
  const uint32_t rank = args.split ? cluster_ctarank() : 0u;
  const int first = static_cast<int>(args.split ? (blockIdx.x >> 1) : blockIdx.x);
  const int stride = static_cast<int>(args.split ? (gridDim.x >> 1) : gridDim.x);
  const int my_units = first < args.units ? (args.units - first + stride - 1) / stride : 0;
  const int nkv_all = (args.n + kAttnBKV - 1) / kAttnBKV;
  const int jt0 = rank == 0 ? 0 : nkv_all / 2;                        // first key tile
  const int nkv = args.split ? (rank == 0 ? nkv_all / 2 : nkv_all - nkv_all / 2) : nkv_all;   // key tiles here

  if (threadIdx.x == 0) {
    mbar_init(b_qfull, 1);
    mbar_init(b_qempty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_kfull + 8 * i, 1);
      mbar_init(b_kempty + 8 * i, 1);
      mbar_init(b_vfull + 8 * i, 1);
      mbar_init(b_vempty + 8 * i, 1);
      mbar_init(b_sfull + 8 * i, 1);
      mbar_init(b_pfull + 8 * i, 128);
      mbar_init(b_pvdone + 8 * i, 1);
      mbar_init(b_ofree + 8 * i, 128);
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
  // TMEM columns: S_0 (and P_0) at 0, S_1 (and P_1) at 128, O_0 at 256, O_1 at 256 + DH
  grid_dep_wait();
  // a softmax thread's running max and sum at the end of its (one) unit,
  // for the split exchange; sm_ok: that unit's key tiles and products all
  // completed (warp-uniform)
  float sm_m = -INFINITY, sm_l = 0.f;
  bool sm_ok = false;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: per unit its two query tiles, then
      // its key and V^T tiles through the two-stage rings (global count g)
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int issued_k = 0, issued_v = 0, issued_q = 0;
      bool ok = true;
      for (int k = 0; k < my_units && ok; ++k) {
        const int unit = args.unit0 + first + k * stride;
        const int head = unit / args.qpairs;
        const int q0 = (unit - head * args.qpairs) * (kAttnTilesQ * kAttnBQ);
        // the previous unit's S products have all read its query tiles
        if (k > 0 && !mbar_wait(b_qempty, (k - 1) & 1, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(b_qfull, kAttnTilesQ * L::kQBytes);
#pragma unroll
        for (int i = 0; i < kAttnTilesQ; ++i)
#pragma unroll
          for (int a = 0; a < DH / 64; ++a)
            tma_load_3d(smem_u32(smem + L::kQOff + i * L::kQBytes + a * kAttnBQ * 128), &tmQ, b_qfull, a * 64,
                        q0 + i * kAttnBQ, head);
        ++issued_q;
        for (int j = 0; j < nkv; ++j) {
          const int g = k * nkv + j;
          const int st = g & 1;
          const uint32_t par = ((g >> 1) & 1) ^ 1;
          if (!mbar_wait(b_kempty + 8 * st, par, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(b_kfull + 8 * st, L::kKBytes);
          uint8_t* sk = smem + L::kKOff + st * L::kKBytes;
#pragma unroll
          for (int a = 0; a < DH / 64; ++a)
            tma_load_3d(smem_u32(sk + a * kAttnBKV * 128), &tmK, b_kfull + 8 * st, a * 64, (jt0 + j) * kAttnBKV,
                        head);
          ++issued_k;
          if (!mbar_wait(b_vempty + 8 * st, par, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(b_vfull + 8 * st, L::kVBytes);
          uint8_t* sv = smem + L::kVOff + st * L::kVBytes;
#pragma unroll
          for (int a = 0; a < 2; ++a)
            tma_load_3d(smem_u32(sv + a * DH * 128), &tmV, b_vfull + 8 * st, (jt0 + j) * kAttnBKV + a * 64, 0,
                        head);
          ++issued_v;
        }
      }
      if (!ok) {
        // let the loads still in flight land before the CTA exits
        for (int g = max(0, issued_k - 2); g < issued_k; ++g) mbar_wait_drain(b_kfull + 8 * (g & 1), (g >> 1) & 1);
        for (int g = max(0, issued_v - 2); g < issued_v; ++g) mbar_wait_drain(b_vfull + 8 * (g & 1), (g >> 1) & 1);
        if (issued_q > 0) mbar_wait_drain(b_qfull, (issued_q - 1) & 1);
      }
    }
  } else if (warp == 1) {
    {
      // ---------------- MMA issuer (whole warp converged; one elected lane issues)
      auto wait_all = [&](uint32_t bar, uint32_t par) {
        return __all_sync(0xffffffffu, mbar_wait(bar, par, abort_flag));
      };
      constexpr uint32_t id_s = idesc_bf16_f32(kAttnBQ, kAttnBKV);
      constexpr uint32_t id_o = idesc_bf16_f32(kAttnBQ, DH);
      // operand descriptors as their low words (start address >> 4 plus
      // offsets; the high word is the same for all of them)
      const uint32_t q_lo = sdesc_lo(smem_u32(smem + L::kQOff));
      const uint32_t k_lo = sdesc_lo(smem_u32(smem + L::kKOff));
      const uint32_t v_lo = sdesc_lo(smem_u32(smem + L::kVOff));
      auto issue_s = [&](int i, int g) {
        const uint32_t ka = k_lo + (g & 1) * (L::kKBytes >> 4);
        const uint32_t qa = q_lo + i * (L::kQBytes >> 4);
        if constexpr (DH == 128) {
          tc_mma_ss_k128(tmem_base + i * kAttnBKV, qa, ka, id_s, 0);
        } else {
#pragma unroll
          for (int kk = 0; kk < DH / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * (kAttnBQ * 128) + (kk & 3) * 32) >> 4;
            const uint32_t offk = ((kk >> 2) * (kAttnBKV * 128) + (kk & 3) * 32) >> 4;
            if (elect_one()) tc_mma_ss_lo(tmem_base + i * kAttnBKV, qa + off, ka + offk, id_s, kk != 0);
          }
        }
        tc_commit_elect(b_sfull + 8 * i);
      };
      auto issue_pv = [&](int i, int g, bool acc) {
        const uint32_t va = v_lo + (g & 1) * (L::kVBytes >> 4);
        if constexpr (DH == 128) {
          tc_mma_ts_k128(tmem_base + 256 + i * DH, tmem_base + i * kAttnBKV, va, id_o, acc);
        } else {
#pragma unroll
          for (int kk = 0; kk < kAttnBKV / 16; ++kk) {
            const uint32_t offv = ((kk >> 2) * (DH * 128) + (kk & 3) * 32) >> 4;
            if (elect_one())
              tc_mma_ts_lo(tmem_base + 256 + i * DH, tmem_base + i * kAttnBKV + kk * 8, va + offv, id_o,
                           acc || kk != 0);
          }
        }
      };
      bool ok = true;
      for (int k = 0; k < my_units && ok; ++k) {
        const int base = k * nkv;
        if (!wait_all(b_qfull, k & 1) || !wait_all(b_kfull + 8 * (base & 1), (base >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(0, base);
        issue_s(1, base);
        tc_commit_elect(b_kempty + 8 * (base & 1));
        // a unit's first products overwrite O_0 / O_1, which the previous
        // unit's epilogue must have read (waited for before the loop, so
        // that the per-tile loop stays as lean as in a single-unit CTA)
        if (k > 0 && (!wait_all(b_ofree, (k - 1) & 1) || !wait_all(b_ofree + 8, (k - 1) & 1))) {
          ok = false;
          break;
        }
        // one key tile: PV of both query tiles, and (MORE) the next tile's S
        auto step = [&](int j, auto more_tag) -> bool {
          constexpr bool kMore = decltype(more_tag)::value;
          const int g = base + j;
          const int st = g & 1;
          if (!wait_all(b_vfull + 8 * st, (g >> 1) & 1)) return false;
          // tile 0: O_0 += P_0 V_j, then S_0 of the next key tile
          if (!wait_all(b_pfull, g & 1)) return false;
          tc_fence_after();
          issue_pv(0, g, j != 0);
          if constexpr (kMore) {
            if (!wait_all(b_kfull + 8 * ((g + 1) & 1), ((g + 1) >> 1) & 1)) return false;
            tc_fence_after();
            issue_s(0, g + 1);
          }
          // tile 1
          if (!wait_all(b_pfull + 8, g & 1)) return false;
          tc_fence_after();
          issue_pv(1, g, j != 0);
          tc_commit_elect(b_vempty + 8 * st);
          if constexpr (kMore) {
            issue_s(1, g + 1);
            tc_commit_elect(b_kempty + 8 * ((g + 1) & 1));
          }
          return true;
        };
        for (int j = 0; j + 1 < nkv && ok; ++j) ok = step(j, std::true_type{});
        if (ok) ok = step(nkv - 1, std::false_type{});
        if (!ok) break;
        tc_commit_elect(b_qempty);   // every S product of the unit is complete with it
        tc_commit_elect(b_pvdone);
        tc_commit_elect(b_pvdone + 8);
      }
      tc_commit_elect(b_drain);
      mbar_wait_drain(b_drain, 0);
    }
  } else if (warp >= 4) {
    // ---------------- softmax warpgroups: warps 4-7 query tile 0, 8-11 tile 1
    const int ti = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem_base + lane_off + ti * kAttnBKV;
    const uint32_t t_o = tmem_base + lane_off + 256 + ti * DH;
    const uint32_t b_s = b_sfull + 8 * ti;
    const uint32_t b_p = b_pfull + 8 * ti;
    const float c = args.scale_log2;
    bool ok = true;
    for (int k = 0; k < my_units && ok; ++k) {
      const int unit = args.unit0 + first + k * stride;
      const int head = unit / args.qpairs;
      const int q0 = (unit - head * args.qpairs) * (kAttnTilesQ * kAttnBQ);
      float m_eff = -INFINITY;
      float l = 0.f;
      for (int j = 0; j < nkv; ++j) {
        const int g = k * nkv + j;
        if (!mbar_wait(b_s, g & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        float s[kAttnBKV];
        tmem_ld128(t_s, s);
        const int valid = args.n - (jt0 + j) * kAttnBKV;
        if (valid < kAttnBKV) {
#pragma unroll
          for (int i = 0; i < kAttnBKV; ++i)
            if (i >= valid) s[i] = -INFINITY;
        }
        float mx4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
        for (int i = 4; i < kAttnBKV - 4; i += 8) {
#pragma unroll
          for (int e = 0; e < 4; ++e) mx4[e] = fmax3(mx4[e], s[i + 2 * e], s[i + 2 * e + 1]);
        }
        const float mx = fmax3(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]),
                               fmax3(s[kAttnBKV - 4], s[kAttnBKV - 3], fmaxf(s[kAttnBKV - 2], s[kAttnBKV - 1]))) * c;
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          m_eff = mx;
        } else if (mx > m_eff + kAttnRescaleLog2) {
          alpha = fast_exp2(m_eff - mx);
          m_eff = mx;
          rescale = true;
        }
        const float neg_m = -m_eff;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // 4 packed partial sums
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int i = half * 64 + 2 * e;
            float x0, x1;
            ffma2(x0, x1, s[i], s[i + 1], c, c, neg_m, neg_m);
            const float p0 = fast_exp2(x0);
            const float p1 = fast_exp2(x1);
            const int a = 2 * (e & 3);
            fadd2(acc[a], acc[a + 1], acc[a], acc[a + 1], p0, p1);
            pk[e] = pack_bf16x2(p0, p1);
          }
          tmem_st32u(t_s + half * 32, pk);
        }
        l = l * alpha + (((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7])));
        // O_i holds the products up to key tile j-1 (complete: S_i(j) was
        // issued after them); rescale it to the new max before PV_i(j).
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int cc = 0; cc < DH / 32; ++cc) {
            float v[32];
            tmem_ld32(t_o + cc * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= alpha;
            tmem_st32(t_o + cc * 32, v);
          }
        }
        tc_fence_before();
        mbar_arrive(b_p);
      }
      sm_ok = __all_sync(0xffffffffu, ok) && __all_sync(0xffffffffu, mbar_wait(b_pvdone + 8 * ti, k & 1, abort_flag));
      ok = sm_ok;
      sm_m = m_eff;
      sm_l = l;
      if (sm_ok && !args.split) {
        tc_fence_after();
        const int grow = q0 + ti * kAttnBQ + row;
        const float inv = 1.f / l;
        const int d = args.heads * DH;
#pragma unroll 1
        for (int cc = 0; cc < DH / 32; ++cc) {
          float v[32];
          tmem_ld32(t_o + cc * 32, v);
          if (grow < args.n) {
            uint32_t p[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) p[i] = pack_bf16x2(v[2 * i] * inv, v[2 * i + 1] * inv);
            uint4* dst = reinterpret_cast<uint4*>(args.o + static_cast<size_t>(grow) * d + head * DH + cc * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
          }
        }
        // O_i has been read: the next unit's first PV_i may overwrite it
        tc_fence_before();
        mbar_arrive(b_ofree + 8 * ti);
      }
    }
  }

  if (args.split) {
    const int unit = args.unit0 + first;   // a split launch gives each pair one unit
    const int head = unit / args.qpairs;
    const int q0 = (unit - head * args.qpairs) * (kAttnTilesQ * kAttnBQ);
    // Combine the pair's halves of the keys: rank r finishes query tile r.
    // Its partner sends the other tile's unnormalised O rows, running max
    // and sum into r's shared memory (the K/V ring, idle now: both CTAs'
    // copies and products have completed before the first cluster barrier),
    // O as float4 [DH / 4][128 rows] so that a warp's stores are contiguous,
    // then m[128] and l[128].
    float* xo = reinterpret_cast<float*>(smem + L::kKOff);
    const int ti = (warp - 4) >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t t_o = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) + 256 + ti * DH;
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    if (warp >= 4 && ti != static_cast<int>(rank) && sm_ok) {
      const uint32_t dst = mapa_shared(smem_u32(xo), rank ^ 1u);
#pragma unroll 1
      for (int cc = 0; cc < DH / 32; ++cc) {
        float v[32];
        tmem_ld32(t_o + cc * 32, v);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          st_cluster_f4(dst + ((cc * 8 + q) * kAttnBQ + row) * 16, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
      st_cluster_f32(dst + (DH * kAttnBQ + row) * 4, sm_m);
      st_cluster_f32(dst + (DH * kAttnBQ + kAttnBQ + row) * 4, sm_l);
    }
    __syncwarp();
    cluster_sync_all();
    if (warp >= 4 && ti == static_cast<int>(rank) && sm_ok) {
      const float m1 = xo[DH * kAttnBQ + row];
      const float l1 = xo[DH * kAttnBQ + kAttnBQ + row];
      const float m = fmaxf(sm_m, m1);
      const float a0 = fast_exp2(sm_m - m), a1 = fast_exp2(m1 - m);
      const float inv = 1.f / (sm_l * a0 + l1 * a1);
      const float4* o1 = reinterpret_cast<const float4*>(xo);
      const int grow = q0 + ti * kAttnBQ + row;
      const int d = args.heads * DH;
#pragma unroll 1
      for (int cc = 0; cc < DH / 32; ++cc) {
        float v[32];
        tmem_ld32(t_o + cc * 32, v);
        if (grow < args.n) {
          uint32_t p[16];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 w = o1[(cc * 8 + q) * kAttnBQ + row];
            const float y0 = (v[4 * q] * a0 + w.x * a1) * inv, y1 = (v[4 * q + 1] * a0 + w.y * a1) * inv;
            const float y2 = (v[4 * q + 2] * a0 + w.z * a1) * inv, y3 = (v[4 * q + 3] * a0 + w.w * a1) * inv;
            p[2 * q] = pack_bf16x2(y0, y1);
            p[2 * q + 1] = pack_bf16x2(y2, y3);
          }
          uint4* dst = reinterpret_cast<uint4*>(args.o + static_cast<size_t>(grow) * d + head * DH + cc * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
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
