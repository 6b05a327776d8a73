// Final layer of the denoiser ([linlog] "DiT 融合内核"): each output head
// (video, audio) normalises its own rows of the residual stream in place --
// no slice copies -- with its own AdaLN vectors, and projects them with a
// BF16 weight [c_out][d], the AdaLN applied while the projection's operand
// tiles are loaded, so no normalised copy of the rows is ever stored:
//   out[r][c] = bf16( sum_k bf16(LN(x_r)_k (1 + scale_k) + shift_k) * w[c][k] )
//
// Two kernels, each one launch for all heads:
//  * head_stats_kernel: one warp per row, coalesced passes for the mean and
//    the centred variance; (mean, rstd) are parked in the first 8 bytes of
//    the row's own output, which the head kernel reads before it overwrites
//    the row -- the layer needs no workspace.
//  * final_head_kernel: 128 rows of a head per CTA (blockIdx.y = head), the
//    d columns split over a cluster of `ksplit` CTAs (one range of k-blocks
//    each) so that the launch fills the SMs.  320 threads: warp 8 streams
//    raw x tiles (128 rows x 64 columns, 128-byte swizzle), weight tiles
//    (c_out x 64) and the k-block's scale/shift slices with TMA through a
//    ring of up to 8 stages; warps 0-7 (two threads per row, 32 columns
//    each) normalise and modulate the tile in place, in the same swizzled
//    position, and hand the stage to warp 9, whose elected thread issues
//    tcgen05.mma M128 N c_out K16 into TMEM.  At the end each CTA but the
//    cluster's first parks its fp32 partial sums in its own shared memory;
//    the first CTA adds them (distributed shared memory), rounds to BF16 and
//    stores the rows.
#pragma once
#include "ptx.cuh"

namespace h3 {

constexpr int kHeadThreads = 320;           // warps 0-7 transform, 8 TMA, 9 MMA
constexpr int kHeadMaxSplit = 4;           // CTAs per cluster splitting d
constexpr int kHeadMaxStages = 8;
constexpr int kHeadBK = 64;
constexpr int kHeadXBytes = 128 * kHeadBK * 2;   // 16 KB raw x tile, transformed in place
constexpr int kHeadMaxN = 256;
constexpr size_t kHeadSmemLimit = 200u << 10;

// A stage: the raw x tile (transformed in place), the weight tile, and the
// k-block's 64 scale and 64 shift values, rounded up to 1 KB so every
// stage's tiles stay 1024-byte aligned for the 128-byte swizzle.
__host__ __device__ constexpr uint32_t head_stage_bytes(int c_out) {
  return static_cast<uint32_t>((kHeadXBytes + c_out * kHeadBK * 2 + 2 * kHeadBK * 4 + 1023) / 1024 * 1024);
}
__host__ __device__ constexpr uint32_t head_mod_offset(int c_out) {
  return static_cast<uint32_t>(kHeadXBytes + c_out * kHeadBK * 2);
}
// The epilogue parks a CTA's fp32 partial sums (128 rows of c_out + 4
// floats) over the stage buffers, so the ring is never smaller than that.
__host__ __device__ constexpr uint32_t head_part_bytes(int c_out) {
  return static_cast<uint32_t>(128 * (c_out + 4) * 4);
}
__host__ __device__ constexpr int head_stages(int c_out) {
  const int fit = static_cast<int>(kHeadSmemLimit / head_stage_bytes(c_out)) < kHeadMaxStages
                      ? static_cast<int>(kHeadSmemLimit / head_stage_bytes(c_out))
                      : kHeadMaxStages;
  const int need = static_cast<int>((head_part_bytes(c_out) + head_stage_bytes(c_out) - 1) / head_stage_bytes(c_out));
  return fit > need ? fit : need;
}
static_assert(head_stages(kHeadMaxN) <= kHeadMaxStages, "the widest head's partial sums fit the ring");
__host__ __device__ constexpr size_t head_smem_bytes(int c_out) {
  return 1024 + static_cast<size_t>(head_stages(c_out)) * head_stage_bytes(c_out) + 512;
}
// the most any supported width (16 .. kHeadMaxN, multiples of 16) asks for
constexpr size_t head_smem_max() {
  size_t m = 0;
  for (int c = 16; c <= kHeadMaxN; c += 16) m = head_smem_bytes(c) > m ? head_smem_bytes(c) : m;
  return m;
}

constexpr int kMaxHeads = 4;

struct HeadArgs {
  int row_start, rows, d;
  const float* shift;       // [d]
  const float* scale;       // [d]
  int c_out;
  __nv_bfloat16* out;       // [rows][c_out]; first 8 bytes of a row hold its (mean, rstd) on entry
  uint32_t tmem_cols;       // power of two >= max(32, c_out)
  int stages;
};

// All heads of one final layer, launched together (blockIdx.y = head).
struct HeadBatch {
  CUtensorMap tmX;                // the residual stream [n][d]
  CUtensorMap tmW[kMaxHeads];     // each head's weight [c_out][d]
  HeadArgs a[kMaxHeads];
  int ksplit;                     // cluster size along blockIdx.x (1..kHeadMaxSplit)
};

// The rows of every head for the statistics pass (one launch).
struct HeadRows {
  int n_heads;
  int first_warp[kMaxHeads + 1];  // prefix sums of the heads' row counts
  int row_start[kMaxHeads];
  int c_out[kMaxHeads];
  __nv_bfloat16* out[kMaxHeads];
};

// (mean, rstd) of every head row of x, one warp per row, stored as two
// floats at the start of the row's output.
__global__ void __launch_bounds__(256)
    head_stats_kernel(const __nv_bfloat16* __restrict__ x, const __grid_constant__ HeadRows hr, int d, float eps) {
  grid_dep_wait();
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= hr.first_warp[hr.n_heads]) return;
  int h = 0;
  while (gw >= hr.first_warp[h + 1]) ++h;
  const int warp = gw - hr.first_warp[h];
  const int row_start = hr.row_start[h];
  const int c_out = hr.c_out[h];
  __nv_bfloat16* out = hr.out[h];
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(row_start + warp) * d);
  const int nvec = d >> 3;
  float sum = 0.f;
  for (int v = lane; v < nvec; v += 32) {
    const uint4 u = src[v];
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 t = __bfloat1622float2(b[e]);
      sum += t.x;
      sum += t.y;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float mean = sum / static_cast<float>(d);
  float sq = 0.f;
  for (int v = lane; v < nvec; v += 32) {
    const uint4 u = src[v];
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 t = __bfloat1622float2(b[e]);
      const float d0 = t.x - mean, d1 = t.y - mean;
      sq = fmaf(d0, d0, sq);
      sq = fmaf(d1, d1, sq);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  if (lane == 0) {
    float2* st = reinterpret_cast<float2*>(out + static_cast<size_t>(warp) * c_out);
    *st = make_float2(mean, rsqrtf(sq / static_cast<float>(d) + eps));
  }
}

__global__ void __launch_bounds__(kHeadThreads, 1) final_head_kernel(const __grid_constant__ HeadBatch hb) {
  const HeadArgs& a = hb.a[blockIdx.y];
  const CUtensorMap* tmX = &hb.tmX;
  const CUtensorMap* tmW = &hb.tmW[blockIdx.y];
  const int ksplit = hb.ksplit;
  const int tile0 = (blockIdx.x / ksplit) * 128;
  // a head with fewer tiles: the whole cluster (same tile) leaves together
  if (tile0 >= a.rows) return;
  const int ks = static_cast<int>(blockIdx.x % ksplit);   // == rank in the cluster
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t stage_bytes = head_stage_bytes(a.c_out);
  const int S = a.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * stage_bytes);
  // bars: full[S], ready[S], empty[S], acc_full, drain
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3 * kHeadMaxStages + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t ready0 = smem_u32(bars + kHeadMaxStages);
  const uint32_t empty0 = smem_u32(bars + 2 * kHeadMaxStages);
  const uint32_t acc_full = smem_u32(bars + 3 * kHeadMaxStages);
  const uint32_t drain = smem_u32(bars + 3 * kHeadMaxStages + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kblocks = a.d / kHeadBK;
  const int kb0 = ks * kblocks / ksplit, kb1 = (ks + 1) * kblocks / ksplit;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(ready0 + 8 * s, 256);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_holder), a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  // transform warps: rows (warp & 3) * 32 + lane, column half warp >> 2
  const int r = (warp & 3) * 32 + lane;
  const int hh = (warp >> 2) & 1;
  const int grow = tile0 + r;
  const bool live = grow < a.rows;
  bool ok = true;

  if (warp < 8) {
    // ---------------- in-place AdaLN of the x tiles
    float mean = 0.f, rstd = 0.f;
    // the statistics launch writes (mean, rstd) into the output rows: wait
    // for it (launch overlap) before reading them; these warps also write
    // the outputs.  The other roles read only x, the weights and the
    // modulation vectors, which that launch does not write, so the x tiles
    // start streaming before it has finished.
    grid_dep_wait();
    if (live) {
      const float2 st = *reinterpret_cast<const float2*>(a.out + static_cast<size_t>(grow) * a.c_out);
      mean = st.x;
      rstd = st.y;
    }
    const uint32_t mod_off = head_mod_offset(a.c_out);
    int stage = 0;
    uint32_t phase = 0;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait(full0 + 8 * stage, phase, abort_flag)) { ok = false; break; }
      uint8_t* st_base = smem + stage * stage_bytes;
      uint8_t* row = st_base + r * 128;
      const float4* sc4 = reinterpret_cast<const float4*>(st_base + mod_off);            // 64 scales
      const float4* sh4 = reinterpret_cast<const float4*>(st_base + mod_off + kHeadBK * 4);   // 64 shifts
      // this thread's four 16-byte chunks of the row first, then the writes:
      // the loads are not ordered behind earlier stores to the same tile
      uint4 raw[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = hh * 4 + q;
        raw[q] = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) * 16));   // 128-byte swizzle
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c = hh * 4 + q;
        uint4 packed = make_uint4(0u, 0u, 0u, 0u);
        if (live) {
          const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw[q]);
          const float4 s0 = sc4[2 * c], s1 = sc4[2 * c + 1];
          const float4 h0 = sh4[2 * c], h1 = sh4[2 * c + 1];
          const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
          const float sh[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
          uint32_t p[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 t = __bfloat1622float2(b[e]);
            const float o0 = fmaf((t.x - mean) * rstd, 1.f + sc[2 * e], sh[2 * e]);
            const float o1 = fmaf((t.y - mean) * rstd, 1.f + sc[2 * e + 1], sh[2 * e + 1]);
            p[e] = pack_bf16x2(o0, o1);
          }
          packed = make_uint4(p[0], p[1], p[2], p[3]);
        }
        // rows past the head (other rows of x, or zero fill) become zeros
        *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) * 16)) = packed;
      }
      fence_proxy_async_smem();
      mbar_arrive(ready0 + 8 * stage);
      if (++stage == S) { stage = 0; phase ^= 1; }
    }
    ok = ok && mbar_wait(acc_full, 0, abort_flag);
    if (ok) tc_fence_after();
  } else if (warp == 8) {
    if (lane == 0) {
      // ---------------- raw x tiles and weight tiles by TMA
      tma_prefetch_desc(tmX);
      tma_prefetch_desc(tmW);
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag)) break;
        const uint32_t fb = full0 + 8 * stage;
        const uint32_t base = smem_u32(smem + stage * stage_bytes);
        const uint32_t mod_off = head_mod_offset(a.c_out);
        mbar_arrive_expect_tx(fb, mod_off + 2 * kHeadBK * 4);
        tma_load_2d(base, tmX, fb, kb * kHeadBK, a.row_start + tile0);
        tma_load_2d(base + kHeadXBytes, tmW, fb, kb * kHeadBK, 0);
        bulk_load(base + mod_off, a.scale + kb * kHeadBK, kHeadBK * 4, fb);
        bulk_load(base + mod_off + kHeadBK * 4, a.shift + kb * kHeadBK, kHeadBK * 4, fb);
        ++issued;
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
      if (issued < kb1 - kb0) {
        // after a timeout: let the loads in flight land before exiting
        for (int i = max(0, issued - S); i < issued; ++i) mbar_wait_drain(full0 + 8 * (i % S), (i / S) & 1);
      }
    }
  } else {
    if (lane == 0) {
      // ---------------- MMA issuer
      const uint32_t idesc = idesc_bf16_f32(128, a.c_out);
      int stage = 0;
      uint32_t phase = 0;
      bool mok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(ready0 + 8 * stage, phase, abort_flag)) { mok = false; break; }
        tc_fence_after();
        const uint32_t a0 = smem_u32(smem + stage * stage_bytes);
        const uint32_t b0 = a0 + kHeadXBytes;
#pragma unroll
        for (int k = 0; k < kHeadBK / 16; ++k)
          tc_mma_bf16(tmem_base, sdesc_k128(a0 + 32 * k), sdesc_k128(b0 + 32 * k), idesc, (kb != kb0 || k != 0));
        tc_commit(empty0 + 8 * stage);
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
      if (mok) tc_commit(acc_full);
      tc_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  }

  // ---------------- epilogue: warps w and w + 4 share TMEM lanes 32 (w & 3)
  // and take alternate halves of the 16-column groups.  All stage buffers
  // are consumed (acc_full), so the partial sums reuse shared memory from 0.
  const int groups = a.c_out / 16;
  const int gh = (groups + 1) / 2;
  const int g0 = hh * gh, g1 = min(groups, g0 + gh);
  const uint32_t tl = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const int pstride = a.c_out + 4;   // floats per partial row (16-byte shift per row)
  float* part = reinterpret_cast<float*>(smem);
  if (ksplit > 1) {
    if (warp < 8 && ok && ks != 0) {
#pragma unroll 1
      for (int cg = g0; cg < g1; ++cg) {
        float v[16];
        tmem_ld16(tl + cg * 16, v);
        float4* dst = reinterpret_cast<float4*>(part + r * pstride + cg * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
    }
    // every thread of every CTA of the cluster, whatever happened above
    cluster_sync_all();
  }
  if (warp < 8 && ok && ks == 0) {
#pragma unroll 1
    for (int cg = g0; cg < g1; ++cg) {
      float v[16];
      tmem_ld16(tl + cg * 16, v);
      for (int peer = 1; peer < ksplit; ++peer) {
        const uint32_t src = mapa_shared(smem_u32(part + r * pstride + cg * 16), static_cast<uint32_t>(peer));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 q = ld_cluster_f4(src + 16 * i);
          v[4 * i] += q.x;
          v[4 * i + 1] += q.y;
          v[4 * i + 2] += q.z;
          v[4 * i + 3] += q.w;
        }
      }
      if (live) {
        uint32_t p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) p[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
        uint4* o = reinterpret_cast<uint4*>(a.out + static_cast<size_t>(grow) * a.c_out + cg * 16);
        o[0] = make_uint4(p[0], p[1], p[2], p[3]);
        o[1] = make_uint4(p[4], p[5], p[6], p[7]);
      }
    }
  }
  // the peers' partial sums stay readable until the first CTA is done
  if (ksplit > 1) cluster_sync_all();

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem_base, a.tmem_cols);
}

}  // namespace h3
