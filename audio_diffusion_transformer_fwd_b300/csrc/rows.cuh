// HBM-bound row kernels: AdaLN, the gated residual fused with the next AdaLN,
// dynamic int8 quantisation, horizontal-pair token reduce/restore, and the
// RoPE cos/sin table.  One CTA of 128 threads per row, 16-byte loads and
// stores, warp-shuffle reductions; a row of up to 8192 BF16 stays in
// registers between the residual, the statistics and the normalisation.
#pragma once
#include "ptx.cuh"

namespace h3 {

constexpr int kRowThreads = 128;
constexpr int kRowMaxVec = 8;   // 8 x 128 threads x 8 values = 8192 columns

// Sum over the 128 threads of the CTA.  red[4] must be this reduction's
// own shared slots (not read by an earlier reduction of the same row), so a
// single barrier suffices.
__device__ __forceinline__ float block_sum_128(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  return red[0] + red[1] + red[2] + red[3];
}

__device__ __forceinline__ void unpack8(const uint4 u, float (&f)[8]) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(b[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// A group's quantisation scale s = absmax / 127 and its correctly rounded
// reciprocal r (0 when s is too small for a normal reciprocal).
struct QuantScale {
  float s, r;
};
__device__ __forceinline__ QuantScale quant_scale(float s) {
  QuantScale q;
  q.s = s;
  q.r = s >= 0x1p-100f ? __frcp_rn(s) : 0.f;
  return q;
}

// int8 code of x at scale s (s = absmax / 127 of x's group): x / s correctly
// rounded in fp32, rounded half to even, clamped to [-127, 127]; s = 0 gives 0.
// Returned as a float holding the integer.  The quotient is formed as
// t = x * r: |x / s| <= 127.x, so t lies within 128 * 2^-23 (two roundings)
// of x / s, and the correctly rounded quotient within 2^-24 * 128 of it; both
// round to the same integer unless t is within 2.3e-5 of a half-integer.
// Where t is within 1e-4 of one (|t - rint(t)| >= 0.4999, rare) the division
// itself decides.
__device__ __forceinline__ float quant_code(float x, const QuantScale& q) {
  if (q.s == 0.f) return 0.f;
  const float t = x * q.r;
  float c = rintf(t);
  if (q.r == 0.f || fabsf(t - c) >= 0.4999f) c = rintf(__fdiv_rn(x, q.s));
  return fminf(127.f, fmaxf(-127.f, c));
}

// max |v| over 8 BF16 values, exact (taken on the BF16 pairs).
__device__ __forceinline__ __nv_bfloat162 absmax8(const uint4 u, __nv_bfloat162 m) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) m = __hmax2(m, __habs2(b[i]));
  return m;
}
__device__ __forceinline__ float absmax_of(__nv_bfloat162 m) {
  return fmaxf(__bfloat162float(m.x), __bfloat162float(m.y));
}

// x_out = bf16(x + gate * branch) (if GATE) and h = bf16(LN(x_out)(1+scale)+shift)
// (if NORM).  LN statistics in fp32 over the rounded row: mean, then the
// biased variance of (x - mean) from the register copy.
// QUANT (dynamic-int8 path, [linlog] "int8 量化"): instead of h the row's
// int8 codes of bf16(h) at s = absmax(bf16(h)) / 127 are written into h as
// BF16 values, and s into hs[row] -- the same codes h3dit_quantize_act gives
// for the BF16 h.
// Token segments with their own modulation vectors ([linlog] "音频处理": the
// reference audio is conditioned at its own timestep): segment k covers rows
// start[k] .. start[k+1]-1, and its vectors sit `stride` floats after the
// previous segment's.
struct SegMap {
  int count;      // 1..4
  int start[4];   // start[0] = 0, increasing
  int stride;
};

__device__ __forceinline__ int seg_offset(const SegMap& m, int row) {
  int k = 0;
#pragma unroll
  for (int i = 1; i < 4; ++i) k += (i < m.count && row >= m.start[i]) ? 1 : 0;
  return k * m.stride;
}

// A thread's part of a row: NV vectors of 8 values, held either as fp32 or
// as packed BF16 pairs (exact when every value is a BF16 number; half the
// registers).
template <int NV, bool PACKED>
struct RowRegs;
template <int NV>
struct RowRegs<NV, true> {
  uint4 p[NV];
  __device__ __forceinline__ void get(int i, float (&v)[8]) const { unpack8(p[i], v); }
  __device__ __forceinline__ void set(int i, const float (&v)[8]) { p[i] = pack8(v); }
  __device__ __forceinline__ void set_packed(int i, uint4 u) { p[i] = u; }
};
template <int NV>
struct RowRegs<NV, false> {
  float f[NV][8];
  __device__ __forceinline__ void get(int i, float (&v)[8]) const {
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = f[i][e];
  }
  __device__ __forceinline__ void set(int i, const float (&v)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) f[i][e] = v[e];
  }
  __device__ __forceinline__ void set_packed(int i, uint4 u) { unpack8(u, f[i]); }
};

// NV = ceil(d / (8 * 128)) 16-byte vectors per thread: the row's register
// copy is sized to the actual width.  The kernel is latency-bound on its two
// block reductions, so resident rows per SM set its bandwidth: with the row
// held as packed BF16 pairs, up to NV = 5 (d <= 5120) the registers are
// capped for 10 CTAs per SM.  The gated residual + AdaLN (no quantisation)
// keeps its row in fp32 at 8 CTAs per SM: its gate and branch values need
// the registers and the unpacking costs it more than the residency gains
// (measured at d = 5120).
template <bool GATE, bool NORM, bool QUANT>
__host__ __device__ constexpr bool row_packed() { return !(GATE && NORM && !QUANT); }
template <bool GATE, bool NORM, bool QUANT, int NV>
constexpr int row_min_blocks() { return NV > 5 ? 8 : row_packed<GATE, NORM, QUANT>() ? 10 : 8; }

template <bool GATE, bool NORM, bool QUANT, int NV>
__global__ void __launch_bounds__(kRowThreads, row_min_blocks<GATE, NORM, QUANT, NV>())
    gate_adaln_kernel(__nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ branch,
                      const float* __restrict__ gate, const float* __restrict__ shift,
                      const float* __restrict__ scale, __nv_bfloat16* __restrict__ h,
                      float* __restrict__ hs, int d, float eps, SegMap sm) {
  grid_dep_wait();
  __shared__ float red[12];   // mean, variance and absmax: four slots each
  const size_t row = blockIdx.x;
  if (sm.count > 1) {
    const int so = seg_offset(sm, static_cast<int>(row));
    if (GATE) gate += so;
    if (NORM) {
      shift += so;
      scale += so;
    }
  }
  const int nvec = d >> 3;
  uint4* xr = reinterpret_cast<uint4*>(x + row * d);
  const uint4* br = reinterpret_cast<const uint4*>(branch + (GATE ? row * d : 0));
  // Every value of the row is exactly a BF16 number (the input, or the
  // residual after its BF16 rounding), so packing it loses nothing.
  RowRegs<NV, row_packed<GATE, NORM, QUANT>()> pv;
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int idx = i * kRowThreads + threadIdx.x;
    if (idx < nvec) {
      float v[8];
      pv.set_packed(i, xr[idx]);
      pv.get(i, v);
      if (GATE) {
        float b[8];
        unpack8(br[idx], b);
        const float4 g0 = __ldg(reinterpret_cast<const float4*>(gate) + 2 * idx);
        const float4 g1 = __ldg(reinterpret_cast<const float4*>(gate) + 2 * idx + 1);
        const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = fmaf(g[e], b[e], v[e]);
        const uint4 packed = pack8(v);
        xr[idx] = packed;
        pv.set_packed(i, packed);
        pv.get(i, v);   // continue with the rounded residual
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) sum += v[e];
    }
  }
  if (!NORM) return;
  const float mean = block_sum_128(sum, red) / static_cast<float>(d);
  float sq = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int idx = i * kRowThreads + threadIdx.x;
    if (idx < nvec) {
      float v[8];
      pv.get(i, v);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float t = v[e] - mean;
        sq = fmaf(t, t, sq);
      }
    }
  }
  const float var = block_sum_128(sq, red + 4) / static_cast<float>(d);
  const float rstd = rsqrtf(var + eps);
  uint4* hr = reinterpret_cast<uint4*>(h + row * d);
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int idx = i * kRowThreads + threadIdx.x;
    if (idx < nvec) {
      float v[8];
      pv.get(i, v);
      const float4 s0 = __ldg(reinterpret_cast<const float4*>(scale) + 2 * idx);
      const float4 s1 = __ldg(reinterpret_cast<const float4*>(scale) + 2 * idx + 1);
      const float4 b0 = __ldg(reinterpret_cast<const float4*>(shift) + 2 * idx);
      const float4 b1 = __ldg(reinterpret_cast<const float4*>(shift) + 2 * idx + 1);
      const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
      const float sh[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = fmaf((v[e] - mean) * rstd, 1.f + sc[e], sh[e]);
      if (QUANT) {
        pv.set_packed(i, pack8(o));   // keep bf16(h) for the codes below
      } else {
        hr[idx] = pack8(o);
      }
    }
  }
  if (!QUANT) return;
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int idx = i * kRowThreads + threadIdx.x;
    if (idx < nvec) {
      float v[8];
      pv.get(i, v);
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[8 + (threadIdx.x >> 5)] = amax;
  __syncthreads();
  amax = fmaxf(fmaxf(red[8], red[9]), fmaxf(red[10], red[11]));
  const QuantScale sq8 = quant_scale(__fdiv_rn(amax, 127.0f));
  if (threadIdx.x == 0) hs[row] = sq8.s;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int idx = i * kRowThreads + threadIdx.x;
    if (idx < nvec) {
      float v[8];
      pv.get(i, v);
      float c[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) c[e] = quant_code(v[e], sq8);
      hr[idx] = pack8(c);   // integers in [-127, 127]: exact in BF16
    }
  }
}

// The quantiser of quantize_kernel writing the codes as BF16 values (the
// operand form of the int8 projections).  q may be x itself: every thread
// reads each 16-byte chunk it overwrites, after the group's absmax is known.
__global__ void __launch_bounds__(kRowThreads)
    quantize_codes_kernel(const __nv_bfloat16* x, int cols, int group, __nv_bfloat16* q,
                          float* __restrict__ scales) {
  grid_dep_wait();
  __shared__ float red[4];
  const int groups = cols / group;
  const size_t row = blockIdx.x / groups;
  const int g = blockIdx.x - static_cast<int>(row) * groups;
  const size_t base = row * cols + static_cast<size_t>(g) * group;
  const uint4* src = reinterpret_cast<const uint4*>(x + base);
  uint4* dst = reinterpret_cast<uint4*>(q + base);
  const int nvec = group >> 3;
  __nv_bfloat162 m2 = __float2bfloat162_rn(0.f);
  for (int idx = threadIdx.x; idx < nvec; idx += kRowThreads) m2 = absmax8(src[idx], m2);
  float amax = absmax_of(m2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  const QuantScale s = quant_scale(__fdiv_rn(amax, 127.0f));
  if (threadIdx.x == 0) scales[row * groups + g] = s.s;
  for (int idx = threadIdx.x; idx < nvec; idx += kRowThreads) {
    float f[8];
    unpack8(src[idx], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = quant_code(f[e], s);
    dst[idx] = pack8(f);
  }
}

// Groups of up to 1024 columns (NV * 256): one warp per group, the group
// held in registers (NV 16-byte vectors per lane, all loaded before any
// store, so q may be x), the absmax by warp shuffles.  CODES: the codes as
// BF16 values into q16, else as int8 into q8.
template <int NV, bool CODES>
__global__ void __launch_bounds__(256)
    quantize_warp_kernel(const __nv_bfloat16* x, int cols, int group, long long n_groups, __nv_bfloat16* q16,
                         int8_t* q8, float* __restrict__ scales) {
  grid_dep_wait();
  const long long gw = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (gw >= n_groups) return;
  const int lane = threadIdx.x & 31;
  const int groups = cols / group;
  const long long row = gw / groups;
  const int g = static_cast<int>(gw - row * groups);
  const size_t base = static_cast<size_t>(row) * cols + static_cast<size_t>(g) * group;
  const uint4* src = reinterpret_cast<const uint4*>(x + base);
  uint4 u[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) u[i] = src[lane + 32 * i];
  __nv_bfloat162 m2 = __float2bfloat162_rn(0.f);
#pragma unroll
  for (int i = 0; i < NV; ++i) m2 = absmax8(u[i], m2);
  float amax = absmax_of(m2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const QuantScale s = quant_scale(__fdiv_rn(amax, 127.0f));
  if (lane == 0) scales[gw] = s.s;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    float f[8];
    unpack8(u[i], f);
    if (CODES) {
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = quant_code(f[e], s);
      reinterpret_cast<uint4*>(q16 + base)[lane + 32 * i] = pack8(f);
    } else {
      uint32_t w[2] = {0u, 0u};
#pragma unroll
      for (int e = 0; e < 8; ++e)
        w[e >> 2] |= (static_cast<uint32_t>(static_cast<int>(quant_code(f[e], s))) & 0xFFu) << (8 * (e & 3));
      reinterpret_cast<uint2*>(q8 + base)[lane + 32 * i] = make_uint2(w[0], w[1]);
    }
  }
}

// int8 codes -> the same integers as BF16 values (exact), 8 per thread.
__global__ void widen_codes_kernel(const int8_t* __restrict__ q, size_t n8,
                                   __nv_bfloat16* __restrict__ out) {
  grid_dep_wait();
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const uint2 w = reinterpret_cast<const uint2*>(q)[i];
  const uint32_t ww[2] = {w.x, w.y};
  float f[8];
#pragma unroll
  for (int e = 0; e < 8; ++e)
    f[e] = static_cast<float>(static_cast<int8_t>((ww[e >> 2] >> (8 * (e & 3))) & 0xFFu));
  reinterpret_cast<uint4*>(out)[i] = pack8(f);
}

// Symmetric absmax int8 quantisation of groups of `group` columns; one CTA
// per (row, group).  s = absmax / 127 and x / s both correctly rounded fp32
// divisions; round half to even; clamp to [-127, 127]; zero group -> 0.
__global__ void __launch_bounds__(kRowThreads)
    quantize_kernel(const __nv_bfloat16* __restrict__ x, int cols, int group, int8_t* __restrict__ q,
                    float* __restrict__ scales) {
  __shared__ float red[4];
  const int groups = cols / group;
  const size_t row = blockIdx.x / groups;
  const int g = blockIdx.x - static_cast<int>(row) * groups;
  const uint4* src = reinterpret_cast<const uint4*>(x + row * cols + static_cast<size_t>(g) * group);
  const int nvec = group >> 3;
  __nv_bfloat162 m2 = __float2bfloat162_rn(0.f);
  for (int idx = threadIdx.x; idx < nvec; idx += kRowThreads) m2 = absmax8(src[idx], m2);
  float amax = absmax_of(m2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  const QuantScale s = quant_scale(__fdiv_rn(amax, 127.0f));
  if (threadIdx.x == 0) scales[row * groups + g] = s.s;
  uint2* dst = reinterpret_cast<uint2*>(q + row * cols + static_cast<size_t>(g) * group);
  for (int idx = threadIdx.x; idx < nvec; idx += kRowThreads) {
    float f[8];
    unpack8(src[idx], f);
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int c = static_cast<int>(quant_code(f[e], s));
      w[e >> 2] |= (static_cast<uint32_t>(c) & 0xFFu) << (8 * (e & 3));
    }
    dst[idx] = make_uint2(w[0], w[1]);
  }
}

// Core residual reuse ([linlog] speed/quality presets, "--core-reuse"):
// delta = x_out - x_in in fp32 (exact for BF16 streams whose exponents are
// within 16 of each other), and a reuse step x = bf16(x + delta).  Eight
// elements per thread, 16-byte loads.
__global__ void core_residual_kernel(const __nv_bfloat16* __restrict__ x_in, const __nv_bfloat16* __restrict__ x_out,
                                     size_t n8, float* __restrict__ delta) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  float a[8], b[8];
  unpack8(reinterpret_cast<const uint4*>(x_in)[i], a);
  unpack8(reinterpret_cast<const uint4*>(x_out)[i], b);
  float4* o = reinterpret_cast<float4*>(delta) + 2 * i;
  o[0] = make_float4(b[0] - a[0], b[1] - a[1], b[2] - a[2], b[3] - a[3]);
  o[1] = make_float4(b[4] - a[4], b[5] - a[5], b[6] - a[6], b[7] - a[7]);
}

__global__ void core_reuse_kernel(__nv_bfloat16* __restrict__ x, const float* __restrict__ delta, size_t n8) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  float a[8];
  unpack8(reinterpret_cast<const uint4*>(x)[i], a);
  const float4 d0 = reinterpret_cast<const float4*>(delta)[2 * i];
  const float4 d1 = reinterpret_cast<const float4*>(delta)[2 * i + 1];
  const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
  for (int e = 0; e < 8; ++e) a[e] += dd[e];
  reinterpret_cast<uint4*>(x)[i] = pack8(a);
}

// Row maps of the horizontal-pair reduction.  Full row i -> reduced row.
struct PairGrid {
  int offset, T, Hh, W, Wr;   // Wr = ceil(W/2)
  int n_full, n_red;
};

// Reduced row r -> first full row and member count (1 or 2).
__device__ __forceinline__ void reduced_to_full(const PairGrid& g, int r, int& i0, int& cnt) {
  const int nv_red = g.T * g.Hh * g.Wr;
  if (r < g.offset) { i0 = r; cnt = 1; return; }
  if (r < g.offset + nv_red) {
    const int k = r - g.offset;
    const int rowi = k / g.Wr;
    const int j = k - rowi * g.Wr;
    i0 = g.offset + rowi * g.W + 2 * j;
    cnt = (2 * j + 1 < g.W) ? 2 : 1;
    return;
  }
  i0 = r + (g.T * g.Hh * g.W - nv_red);
  cnt = 1;
}

// One CTA per reduced row: mean of the pair (fp32, rounded to BF16), or a
// copy; optionally also copies the members into `side`.
__global__ void __launch_bounds__(kRowThreads)
    token_reduce_kernel(const __nv_bfloat16* __restrict__ xf, int d, PairGrid g,
                        __nv_bfloat16* __restrict__ xr, __nv_bfloat16* __restrict__ side) {
  const int r = blockIdx.x;
  int i0, cnt;
  reduced_to_full(g, r, i0, cnt);
  const uint4* a = reinterpret_cast<const uint4*>(xf + static_cast<size_t>(i0) * d);
  const uint4* b = reinterpret_cast<const uint4*>(xf + static_cast<size_t>(i0 + (cnt - 1)) * d);
  uint4* o = reinterpret_cast<uint4*>(xr + static_cast<size_t>(r) * d);
  const int nvec = d >> 3;
  for (int idx = threadIdx.x; idx < nvec; idx += kRowThreads) {
    const uint4 ua = a[idx];
    if (cnt == 2) {
      const uint4 ub = b[idx];
      float fa[8], fb[8], m[8];
      unpack8(ua, fa);
      unpack8(ub, fb);
#pragma unroll
      for (int e = 0; e < 8; ++e) m[e] = (fa[e] + fb[e]) * 0.5f;
      o[idx] = pack8(m);
      if (side) {
        reinterpret_cast<uint4*>(side + static_cast<size_t>(i0) * d)[idx] = ua;
        reinterpret_cast<uint4*>(side + static_cast<size_t>(i0 + 1) * d)[idx] = ub;
      }
    } else {
      o[idx] = ua;
      if (side) reinterpret_cast<uint4*>(side + static_cast<size_t>(i0) * d)[idx] = ua;
    }
  }
}

// One CTA per reduced row: writes its one or two full rows.  A paired member
// becomes side[i] + (x_red[p] - bf16(mean(side pair))) in fp32, rounded.
// x_full may be the same buffer as side (each CTA reads its pair before
// writing it).
__global__ void __launch_bounds__(kRowThreads)
    token_restore_kernel(const __nv_bfloat16* __restrict__ xr, const __nv_bfloat16* side, int d,
                         PairGrid g, __nv_bfloat16* xf) {
  const int r = blockIdx.x;
  int i0, cnt;
  reduced_to_full(g, r, i0, cnt);
  const uint4* red = reinterpret_cast<const uint4*>(xr + static_cast<size_t>(r) * d);
  const int nvec = d >> 3;
  for (int idx = threadIdx.x; idx < nvec; idx += kRowThreads) {
    const uint4 ur = red[idx];
    if (cnt == 2) {
      const uint4 ua = reinterpret_cast<const uint4*>(side + static_cast<size_t>(i0) * d)[idx];
      const uint4 ub = reinterpret_cast<const uint4*>(side + static_cast<size_t>(i0 + 1) * d)[idx];
      float fa[8], fb[8], fr[8], m[8], oa[8], ob[8];
      unpack8(ua, fa);
      unpack8(ub, fb);
      unpack8(ur, fr);
#pragma unroll
      for (int e = 0; e < 8; ++e) m[e] = (fa[e] + fb[e]) * 0.5f;
      const uint4 um = pack8(m);   // the value the pair held when reduced
      unpack8(um, m);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float upd = fr[e] - m[e];
        oa[e] = fa[e] + upd;
        ob[e] = fb[e] + upd;
      }
      reinterpret_cast<uint4*>(xf + static_cast<size_t>(i0) * d)[idx] = pack8(oa);
      reinterpret_cast<uint4*>(xf + static_cast<size_t>(i0 + 1) * d)[idx] = pack8(ob);
    } else {
      reinterpret_cast<uint4*>(xf + static_cast<size_t>(i0) * d)[idx] = ur;
    }
  }
}

__global__ void reduced_positions_kernel(const float* __restrict__ pos, PairGrid g,
                                         float* __restrict__ out) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= g.n_red) return;
  int i0, cnt;
  reduced_to_full(g, r, i0, cnt);
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    const float p0 = pos[static_cast<size_t>(i0) * 3 + a];
    const float p1 = pos[static_cast<size_t>(i0 + cnt - 1) * 3 + a];
    out[static_cast<size_t>(r) * 3 + a] = cnt == 2 ? (p0 + p1) * 0.5f : p0;
  }
}

// cos/sin of pos[axis] * theta^(-2i/sec) for every (token, pair); pairs are
// numbered across the head in section order (t, y, x).
struct RopeSpec {
  int head_dim;
  int sec[3];
  float theta;
};

__global__ void rope_table_kernel(const float* __restrict__ pos, int n, RopeSpec rs,
                                  float2* __restrict__ table) {
  grid_dep_wait();
  const int half = rs.head_dim / 2;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n * half) return;
  const int t = idx / half;
  const int p = idx - t * half;
  int axis = 0, start = 0;
  while (axis < 2 && 2 * p >= start + rs.sec[axis]) {
    start += rs.sec[axis];
    ++axis;
  }
  const float i = static_cast<float>(p - start / 2);
  const float omega = powf(rs.theta, -2.0f * i / static_cast<float>(rs.sec[axis]));
  const float ang = pos[static_cast<size_t>(t) * 3 + axis] * omega;
  float s, c;
  sincosf(ang, &s, &c);
  table[idx] = make_float2(c, s);
}

}  // namespace h3
