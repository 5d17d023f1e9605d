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
// HBM-bound: one persistent CTA per SM streams 128-row x d tiles through a
// shared-memory ring filled by bulk copies; d/32 threads per row (at d = 256
// each thread takes two rows of a tile).  Thread p
// of a row holds channels [16p, 16p + 16) and the same range shifted by d/2,
// so each rotary pair sits in one thread and the row's sum of squares needs a
// shuffle or two.
// The rotary table ([N][d/2] cos and sin, FP32) is shared by every head and
// stays in L2.
#include <cuda_bf16.h>

#include "dm_device.cuh"
#include "dm_internal.h"

namespace dm {
namespace {

// D / 32 threads per row: every thread holds 16 channels of each half of its
// row, so that the per-tile fixed work (waits, cursor, scale) is shared by 32
// elements per thread.
template <int D>
__host__ __device__ constexpr int row_threads() { return D / 32; }

template <typename T>
struct RowLoad;
template <>
struct RowLoad<float> {
  // n consecutive values (n a multiple of 4, 16-byte aligned), from global
  // memory through the read-only path, or from shared memory
  template <int n>
  __device__ static void load(const float* p, float* out) {
#pragma unroll
    for (int k = 0; k < n; k += 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(p + k));
      out[k] = v.x, out[k + 1] = v.y, out[k + 2] = v.z, out[k + 3] = v.w;
    }
  }
  template <int n>
  __device__ static void load_shared(const float* p, float* out) {
#pragma unroll
    for (int k = 0; k < n; k += 4) {
      const float4 v = *reinterpret_cast<const float4*>(p + k);
      out[k] = v.x, out[k + 1] = v.y, out[k + 2] = v.z, out[k + 3] = v.w;
    }
  }
};
template <>
struct RowLoad<__nv_bfloat16> {
  template <int n>
  __device__ static void load_shared(const __nv_bfloat16* p, float* out) {
#pragma unroll
    for (int k = 0; k < n; k += 8) {
      const uint4 v = *reinterpret_cast<const uint4*>(p + k);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        out[k + 2 * e] = __uint_as_float(w[e] << 16);
        out[k + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
      }
    }
  }
};

// Where tile g (over all jobs) lives: job index j, tile index in the job,
// (b, h) and row tile t.  Fields are read from the kernel parameters by
// index, never through a pointer, which would copy the whole batch to local
// memory.  A CTA walks its tiles with a stride of gridDim.x, so the cursor is
// advanced by subtraction instead of a division per tile.
struct TileRef {
  int j, tile, bh, t, rows;
};
__device__ __forceinline__ void tile_set(const PrologueBatch& batch, int g, TileRef& r) {
  r.j = 0;
  while (r.j + 1 < batch.count && g >= batch.first_tile[r.j + 1]) ++r.j;
  r.tile = g - batch.first_tile[r.j];
  const int T_tiles = batch.job[r.j].T_tiles;
  r.bh = r.tile / T_tiles;
  r.t = r.tile - r.bh * T_tiles;
  r.rows = min(kTile, batch.job[r.j].N - r.t * kTile);
}
__device__ __forceinline__ void tile_advance(const PrologueBatch& batch, int g, int step, TileRef& r) {
  if (r.j + 1 < batch.count && g >= batch.first_tile[r.j + 1]) {  // crossed into a later job
    tile_set(batch, g, r);
    return;
  }
  r.tile += step;
  r.t += step;
  const int T_tiles = batch.job[r.j].T_tiles;
  while (r.t >= T_tiles) r.t -= T_tiles, ++r.bh;
  r.rows = min(kTile, batch.job[r.j].N - r.t * kTile);
}

template <typename T, int D>
struct PrologueCfg {
  static constexpr int kRowThreads = row_threads<D>();
  // d = 256: a 128-row tile is taken as two groups of 64 rows (each thread
  // one row of each), so that 512 threads hold the whole tile in registers
  // under the 128-register cap until its scale is known
  static constexpr int kRowGroups = D > 128 ? 2 : 1;
  static constexpr int kRowsPerGroup = kTile / kRowGroups;
  static constexpr int kThreads = kRowsPerGroup * kRowThreads;
  static constexpr int Q = D / (2 * kRowThreads);  // channels per thread and half-row
  // one row group: the gains stay in registers; two: read through L1 where used
  static constexpr bool kHoldGains = kRowGroups == 1;
  static constexpr int kTileBytes = kTile * D * (int)sizeof(T);
  static constexpr int kStages = 4 * kTileBytes <= 160 * 1024 ? 4 : (2 * kTileBytes <= 200 * 1024 ? 2 : 1);
  static constexpr int kSmem = kStages * kTileBytes;
};

// Persistent: CTA c takes tiles c, c + grid, ...; thread 0 keeps the next
// kStages tiles in flight as bulk copies into a shared-memory ring (each tile
// of one head is one contiguous block of rows), so the SM always has loads
// outstanding while it normalises, rotates and encodes the current tile.
template <typename T, int D>
__global__ void __launch_bounds__(PrologueCfg<T, D>::kThreads, 1)
    prologue_kernel(const PrologueBatch batch, float eps) {
  using C = PrologueCfg<T, D>;
  constexpr int Q = C::Q, kRowThreads = C::kRowThreads, G = C::kRowGroups;
  static_assert(Q == 16, "sixteen channels per thread and half-row");
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ float s_red[2][C::kThreads / 32];
  __shared__ uint64_t full[C::kStages];
  __shared__ int s_abort;

  const int total = batch.first_tile[batch.count];
  Watchdog wd{&s_abort, batch.status, batch.wait_limit_ns};
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < C::kStages; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](int g, int stage) {
    TileRef r;
    tile_set(batch, g, r);
    const uint32_t bytes = (uint32_t)(r.rows * D * (int)sizeof(T));
    const T* src = static_cast<const T*>(batch.job[r.j].x) + ((size_t)r.bh * batch.job[r.j].N + (size_t)r.t * kTile) * D;
    mbar_arrive_expect_tx(&full[stage], bytes);
    bulk_load(ring + stage * C::kTileBytes, src, bytes, &full[stage]);
  };
  if (threadIdx.x == 0)
    for (int k = 0; k < C::kStages; ++k)
      if ((int)blockIdx.x + k * (int)gridDim.x < total) issue((int)blockIdx.x + k * (int)gridDim.x, k);

  const int row = threadIdx.x / kRowThreads, part = threadIdx.x % kRowThreads;
  const int ca = part * Q, cb = D / 2 + part * Q;  // first channel of each half-row
  // this thread's channel gains (ones without gains), reloaded when the job changes
  float ga[C::kHoldGains ? Q : 1], gb[C::kHoldGains ? Q : 1];
  int gain_job = -1;
  int it = 0;
  TileRef r;
  tile_set(batch, blockIdx.x, r);
  for (int g = blockIdx.x; g < total; g += gridDim.x, ++it) {
    if (it > 0) tile_advance(batch, g, gridDim.x, r);
    const int stage = it % C::kStages;
    const float* gain = batch.job[r.j].gain;
    const float* rope_cos = batch.job[r.j].rope_cos;
    const float* rope_sin = batch.job[r.j].rope_sin;
    const int N = batch.job[r.j].N;
    if constexpr (C::kHoldGains) {
      if (r.j != gain_job) {
        gain_job = r.j;
        if (gain) {
          RowLoad<float>::template load<Q>(gain + ca, ga);
          RowLoad<float>::template load<Q>(gain + cb, gb);
        } else {
#pragma unroll
          for (int k = 0; k < Q; ++k) ga[k] = gb[k] = 1.0f;
        }
      }
    }
    const bool rope = rope_cos != nullptr;
    float a[G][Q], b[G][Q];  // this thread's channels of its row in each group
    float amax = 0.0f;
#pragma unroll
    for (int rg = 0; rg < G; ++rg) {
      const int rr = rg * C::kRowsPerGroup + row;  // row within the tile
      const int n = r.t * kTile + rr;              // sequence position
      const bool valid = rr < r.rows;
      // the row's angles (L2) while the rows arrive (two row groups: read
      // where used, which keeps the other group's row in registers)
      float c[C::kHoldGains ? Q : 1], sn[C::kHoldGains ? Q : 1];
      if (C::kHoldGains && rope && valid) {
        RowLoad<float>::template load<Q>(rope_cos + (size_t)n * (D / 2) + ca, c);
        RowLoad<float>::template load<Q>(rope_sin + (size_t)n * (D / 2) + ca, sn);
      }
      if (rg == 0) wait(&full[stage], (uint32_t)(it / C::kStages) & 1, wd, 401);
      float(&x)[Q] = a[rg];
      float(&y)[Q] = b[rg];
      if (valid) {
        const T* xr = reinterpret_cast<const T*>(ring + stage * C::kTileBytes) + rr * D;
        RowLoad<T>::template load_shared<Q>(xr + ca, x);
        RowLoad<T>::template load_shared<Q>(xr + cb, y);
      } else {
#pragma unroll
        for (int k = 0; k < Q; ++k) x[k] = y[k] = 0.0f;
      }
      // RMSNorm: the row's sum of squares over its kRowThreads threads (pairs of
      // adjacent channels in packed FP32x2 arithmetic throughout)
      float2 ss2 = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int k = 0; k < Q; k += 2) {
        ss2 = __ffma2_rn(make_float2(x[k], x[k + 1]), make_float2(x[k], x[k + 1]), ss2);
        ss2 = __ffma2_rn(make_float2(y[k], y[k + 1]), make_float2(y[k], y[k + 1]), ss2);
      }
      float ss = ss2.x + ss2.y;
#pragma unroll
      for (int o = 1; o < kRowThreads; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      // eps > 0 (checked by the API), so an all-zero row normalises to zeros
      const float inv = valid ? __frsqrt_rn(__fadd_rn(ss * (1.0f / D), eps)) : 0.0f;
      const float2 inv2 = make_float2(inv, inv);
#pragma unroll
      for (int k = 0; k < Q; k += 2) {
        float2 g0, g1;
        if constexpr (C::kHoldGains) {
          g0 = make_float2(ga[k], ga[k + 1]);
          g1 = make_float2(gb[k], gb[k + 1]);
        } else if (gain) {
          g0 = __ldg(reinterpret_cast<const float2*>(gain + ca + k));
          g1 = __ldg(reinterpret_cast<const float2*>(gain + cb + k));
        } else {
          g0 = g1 = make_float2(1.0f, 1.0f);
        }
        const float2 ya = __fmul2_rn(__fmul2_rn(make_float2(x[k], x[k + 1]), inv2), g0);
        const float2 yb = __fmul2_rn(__fmul2_rn(make_float2(y[k], y[k + 1]), inv2), g1);
        x[k] = ya.x, x[k + 1] = ya.y, y[k] = yb.x, y[k + 1] = yb.y;
      }
      // rotary embedding: channel ca + k pairs with cb + k, angle index ca + k
      if (rope && valid) {
#pragma unroll
        for (int k = 0; k < Q; k += 2) {
          const float2 x0 = make_float2(x[k], x[k + 1]), x1 = make_float2(y[k], y[k + 1]);
          float2 c2, s2;
          if constexpr (C::kHoldGains) {
            c2 = make_float2(c[k], c[k + 1]);
            s2 = make_float2(sn[k], sn[k + 1]);
          } else {
            c2 = __ldg(reinterpret_cast<const float2*>(rope_cos + (size_t)n * (D / 2) + ca + k));
            s2 = __ldg(reinterpret_cast<const float2*>(rope_sin + (size_t)n * (D / 2) + ca + k));
          }
          const float2 t1 = __fmul2_rn(x1, s2), t0 = __fmul2_rn(x0, s2);
          const float2 ra = __ffma2_rn(x0, c2, make_float2(-t1.x, -t1.y));
          const float2 rb = __ffma2_rn(x1, c2, t0);
          x[k] = ra.x, x[k + 1] = ra.y, y[k] = rb.x, y[k + 1] = rb.y;
        }
      }
#pragma unroll
      for (int k = 0; k < Q; ++k) amax = fmaxf(amax, fmaxf(fabsf(x[k]), fabsf(y[k])));  // |x| folds into the max
    }
    // tile amax, scale and E4M3 codes (the rule of dm_quantize)
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) s_red[it & 1][threadIdx.x >> 5] = amax;
    __syncthreads();
    // every thread has its rows in registers: the stage takes a later tile
    if (threadIdx.x == 0 && g + C::kStages * (int)gridDim.x < total) issue(g + C::kStages * (int)gridDim.x, stage);
    {  // every warp reduces the warp maxima itself (one per lane)
      const int lane = threadIdx.x & 31;
      amax = warp_max(lane < C::kThreads / 32 ? s_red[it & 1][lane] : 0.0f);
    }
    float rcp;
    const float sc = tile_scale<0>(amax, rcp);
    if (threadIdx.x == 0) batch.job[r.j].scales[r.tile] = sc;
    const bool flushed = sc == 0.0f;  // all codes +0
    const float2 r2 = make_float2(rcp, rcp);
#pragma unroll
    for (int rg = 0; rg < G; ++rg) {
      const int rr = rg * C::kRowsPerGroup + row;
      if (rr >= r.rows) continue;
      const int n = r.t * kTile + rr;
      uint32_t wa[Q / 4], wb[Q / 4];
#pragma unroll
      for (int k = 0; k < Q / 4; ++k) {
        const float2 a01 = __fmul2_rn(make_float2(a[rg][4 * k], a[rg][4 * k + 1]), r2);
        const float2 a23 = __fmul2_rn(make_float2(a[rg][4 * k + 2], a[rg][4 * k + 3]), r2);
        const float2 b01 = __fmul2_rn(make_float2(b[rg][4 * k], b[rg][4 * k + 1]), r2);
        const float2 b23 = __fmul2_rn(make_float2(b[rg][4 * k + 2], b[rg][4 * k + 3]), r2);
        wa[k] = flushed ? 0u : pack4<0>(a01.x, a01.y, a23.x, a23.y);
        wb[k] = flushed ? 0u : pack4<0>(b01.x, b01.y, b23.x, b23.y);
      }
      uint8_t* dst = batch.job[r.j].codes + ((size_t)r.bh * N + n) * D;
      *reinterpret_cast<uint4*>(dst + ca) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
      *reinterpret_cast<uint4*>(dst + cb) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
    }
  }
  // after a timeout the loop ran on without the data: wait (bounded by time
  // alone) for copies still landing in this CTA's shared memory
  if (threadIdx.x == 0 && s_abort) {
    const int issued = (total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    for (int k = max(0, issued - C::kStages); k < issued; ++k)
      wait_drain(&full[k % C::kStages], (uint32_t)(k / C::kStages) & 1, wd, 402);
  }
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

template <typename T, int D>
cudaError_t prologue_d(const PrologueBatch& b, float eps, cudaStream_t st) {
  using C = PrologueCfg<T, D>;
  auto k = prologue_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const unsigned grid = (unsigned)min(b.first_tile[b.count], sms);
  k<<<grid, C::kThreads, C::kSmem, st>>>(b, eps);
  return cudaGetLastError();
}

template <typename T>
cudaError_t prologue_t(const PrologueBatch& b, int d, float eps, cudaStream_t st) {
  if (d == 256) return prologue_d<T, 256>(b, eps, st);
  return d == 128 ? prologue_d<T, 128>(b, eps, st) : prologue_d<T, 64>(b, eps, st);
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
