// Attention-input prologue fused with the tile quantiser: per row of Q or K,
// RMSNorm with per-channel gains, then the rotary embedding, then the per
// 128-row tile E4M3 quantisation of dm_quantize, in one pass over the
// pre-normalisation rows.  The pages' models normalise queries and keys with
// learned channel gains ("Delta-Matching for reliable FP8 attention
// training", section 02, where the gains are the tracked quantity) and use
// RoPE (section 05, "Attention variants change when failure appears").
// Readings (no epsilon, rotary layout or base on the pages): RMSNorm
// y_k = x_k / sqrt(mean x^2 + eps) * g_k; rotate-half rotary, channel i < d/2
// paired with i + d/2, angle n * base^(-2i/d) at sequence position n.
//
// HBM-bound: one CTA per 128-row x d tile, d/16 threads per row.  Thread p
// of a row holds channels [8p, 8p + 8) and the same range shifted by d/2, so
// each rotary pair sits in one thread and the row's sum of squares needs a
// few shuffles; every load (row and angles) is issued before any arithmetic.
// The rotary table ([N][d/2] cos and sin, FP32) is shared by every head and
// stays in L2.
#include <cuda_bf16.h>

#include "dm_device.cuh"
#include "dm_internal.h"

namespace dm {
namespace {

// One 128-row tile per CTA, D / 16 threads per row: every thread holds 8
// channels of each half of its row (16-byte loads of bf16 rows).
template <int D>
__host__ __device__ constexpr int row_threads() { return D / 16; }
template <int D>
__host__ __device__ constexpr int tile_threads() { return kTile * row_threads<D>(); }

template <typename T>
struct RowLoad;
template <>
struct RowLoad<float> {
  // n consecutive values (n a multiple of 4, 16-byte aligned)
  template <int n>
  __device__ static void load(const float* p, float* out) {
#pragma unroll
    for (int k = 0; k < n; k += 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(p + k));
      out[k] = v.x, out[k + 1] = v.y, out[k + 2] = v.z, out[k + 3] = v.w;
    }
  }
};
template <>
struct RowLoad<__nv_bfloat16> {
  template <int n>
  __device__ static void load(const __nv_bfloat16* p, float* out) {
#pragma unroll
    for (int k = 0; k < n; k += 8) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(p + k));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        out[k + 2 * e] = __uint_as_float(w[e] << 16);
        out[k + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
      }
    }
  }
};

template <typename T, int D>
__global__ void __launch_bounds__(tile_threads<D>(), 1) prologue_kernel(const PrologueBatch batch, float eps) {
  constexpr int kRowThreads = row_threads<D>(), kPThreads = tile_threads<D>();
  constexpr int Q = D / (2 * kRowThreads);  // channels per thread and half-row
  static_assert(Q == 8, "eight channels per thread and half-row");
  __shared__ float s_red[kPThreads / 32];

  int j = 0;
  while (j + 1 < batch.count && (int)blockIdx.x >= batch.first_tile[j + 1]) ++j;
  const PrologueJob& job = batch.job[j];
  const int N = job.N, T_tiles = job.T_tiles;
  const int tile = (int)blockIdx.x - batch.first_tile[j];
  const int bh = tile / T_tiles, t = tile % T_tiles;
  const int row = threadIdx.x / kRowThreads, part = threadIdx.x % kRowThreads;
  const int n = t * kTile + row;  // sequence position
  const bool valid = n < N;
  const int ca = part * Q, cb = D / 2 + part * Q;  // first channel of each half-row
  const size_t off = ((size_t)bh * N + n) * D;
  const bool rope = job.rope_cos != nullptr;

  // every load first: the row's channels and, with rope, its angles
  float a[Q], b[Q], c[Q], sn[Q];
  if (valid) {
    RowLoad<T>::template load<Q>(static_cast<const T*>(job.x) + off + ca, a);
    RowLoad<T>::template load<Q>(static_cast<const T*>(job.x) + off + cb, b);
    if (rope) {
      RowLoad<float>::template load<Q>(job.rope_cos + (size_t)n * (D / 2) + ca, c);
      RowLoad<float>::template load<Q>(job.rope_sin + (size_t)n * (D / 2) + ca, sn);
    }
  } else {
#pragma unroll
    for (int k = 0; k < Q; ++k) a[k] = b[k] = 0.0f;
  }
  // RMSNorm: the row's sum of squares over its kRowThreads threads
  float ss = 0.0f;
#pragma unroll
  for (int k = 0; k < Q; ++k) ss = fmaf(a[k], a[k], ss);
#pragma unroll
  for (int k = 0; k < Q; ++k) ss = fmaf(b[k], b[k], ss);
#pragma unroll
  for (int o = 1; o < kRowThreads; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  // eps > 0 (checked by the API), so an all-zero row normalises to zeros
  const float inv = valid ? __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ss * (1.0f / D), eps))) : 0.0f;
  if (job.gain) {
    float ga[Q], gb[Q];
    RowLoad<float>::template load<Q>(job.gain + ca, ga);
    RowLoad<float>::template load<Q>(job.gain + cb, gb);
#pragma unroll
    for (int k = 0; k < Q; ++k) {
      a[k] = __fmul_rn(a[k], inv) * ga[k];
      b[k] = __fmul_rn(b[k], inv) * gb[k];
    }
  } else {
#pragma unroll
    for (int k = 0; k < Q; ++k) a[k] = __fmul_rn(a[k], inv), b[k] = __fmul_rn(b[k], inv);
  }
  // rotary embedding: channel ca + k pairs with cb + k, angle index ca + k
  if (rope && valid) {
#pragma unroll
    for (int k = 0; k < Q; ++k) {
      const float x0 = a[k], x1 = b[k];
      a[k] = fmaf(x0, c[k], -__fmul_rn(x1, sn[k]));
      b[k] = fmaf(x1, c[k], __fmul_rn(x0, sn[k]));
    }
  }
  // tile amax, scale and E4M3 codes (the rule of dm_quantize)
  float amax = 0.0f;
#pragma unroll
  for (int k = 0; k < Q; ++k) amax = max3(amax, fabsf(a[k]), fabsf(b[k]));
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = s_red[0];
#pragma unroll
  for (int w = 1; w < kPThreads / 32; ++w) amax = fmaxf(amax, s_red[w]);
  float r;
  const float sc = tile_scale<0>(amax, r);
  if (threadIdx.x == 0) job.scales[tile] = sc;
  if (!valid) return;
  const bool flushed = sc == 0.0f;  // all codes +0
  uint32_t wa[Q / 4], wb[Q / 4];
#pragma unroll
  for (int k = 0; k < Q / 4; ++k) {
    wa[k] = flushed ? 0u
                    : pack4<0>(__fmul_rn(a[4 * k], r), __fmul_rn(a[4 * k + 1], r), __fmul_rn(a[4 * k + 2], r),
                               __fmul_rn(a[4 * k + 3], r));
    wb[k] = flushed ? 0u
                    : pack4<0>(__fmul_rn(b[4 * k], r), __fmul_rn(b[4 * k + 1], r), __fmul_rn(b[4 * k + 2], r),
                               __fmul_rn(b[4 * k + 3], r));
  }
  uint8_t* dst = job.codes + off;
  *reinterpret_cast<uint2*>(dst + ca) = make_uint2(wa[0], wa[1]);
  *reinterpret_cast<uint2*>(dst + cb) = make_uint2(wb[0], wb[1]);
}

// cos and sin of n * base^(-2i/d) in FP64, rounded to FP32; one thread per entry.
__global__ void rope_table_kernel(int N, int d, double base, float* __restrict__ cos_t, float* __restrict__ sin_t) {
  const int h = d / 2;
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)N * h) return;
  const int n = (int)(e / h), i = (int)(e % h);
  const double theta = (double)n * pow(base, -2.0 * i / d);
  double s, c;
  sincos(theta, &s, &c);
  cos_t[e] = (float)c;
  sin_t[e] = (float)s;
}

template <typename T>
cudaError_t prologue_t(const PrologueBatch& b, int d, float eps, cudaStream_t st) {
  const unsigned grid = (unsigned)b.first_tile[b.count];
  if (d == 128)
    prologue_kernel<T, 128><<<grid, tile_threads<128>(), 0, st>>>(b, eps);
  else
    prologue_kernel<T, 64><<<grid, tile_threads<64>(), 0, st>>>(b, eps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prologue(const PrologueBatch& b, dm_dtype xt, int d, float eps, cudaStream_t st) {
  if (b.first_tile[b.count] == 0) return cudaSuccess;
  return xt == DM_BF16 ? prologue_t<__nv_bfloat16>(b, d, eps, st) : prologue_t<float>(b, d, eps, st);
}

cudaError_t launch_rope_table(int N, int d, double base, float* cos_t, float* sin_t, cudaStream_t st) {
  const long long total = (long long)N * (d / 2);
  if (total == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((total + 255) / 256);
  rope_table_kernel<<<grid, 256, 0, st>>>(N, d, base, cos_t, sin_t);
  return cudaGetLastError();
}

}  // namespace dm
