// Bandwidth-bound kernels: the per-tile FP8 quantiser, the stale row
// corrections, and a zero fill.
//
// Quantiser: block scales of "Delta-Matching for reliable FP8 attention
// training", section 01 ("What changes in FP8?"), with the amax rule stated
// in dm.h; one CTA per 128-row x d tile, the tile held in registers between
// the amax reduction and the encode, 16-byte coalesced loads.
//
// Stale corrections: delta_i = <dO_i, O_i> (section 01, "Why can we reuse the
// forward output?") and delta_i = <dO^_i, O_i> (section 03), one warp per row.
//
// Key-block merges (context parallelism over the sequence; the project page's
// section 06 extends the context to 64K tokens): the attention of every query
// row over disjoint key blocks r merges as LSE = ln sum_r exp(LSE_r),
// O = sum_r exp(LSE_r - LSE) O_r, and the matched delta as
// sum_r (sum_j P dP^)_r / sum_r (sum_j P)_r.
#include <cuda_bf16.h>

#include "dm_device.cuh"
#include "dm_pdl.cuh"
#include "dm_internal.h"

namespace dm {
namespace {

// Threads per quantiser CTA: d = 256 tiles (64 KB of bf16) are spread over
// 1024 threads, so that each holds as many values as at d = 128 (the tile sits
// in registers between the amax reduction and the encode).
template <int D>
__host__ __device__ constexpr int quant_threads() { return D > 128 ? 1024 : 256; }

// 16-byte vectors of the input, held raw (bf16 words stay packed, so that a
// tile takes half the registers and more tiles are in flight per SM) and
// widened to FP32 where used.
template <typename T>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int kElems = 4;
  __device__ static uint4 load(const float* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
  __device__ static void widen(const uint4& r, float* out) {
    out[0] = __uint_as_float(r.x), out[1] = __uint_as_float(r.y);
    out[2] = __uint_as_float(r.z), out[3] = __uint_as_float(r.w);
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int kElems = 8;
  __device__ static uint4 load(const __nv_bfloat16* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
  __device__ static void widen(const uint4& r, float* out) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      out[2 * k] = __uint_as_float(w[k] << 16);
      out[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
};

// One CTA per 128-row x D tile of one of up to kMaxJobs tensors (one launch
// quantises Q, K, V and dO together); the CTA finds its tensor from the
// running tile counts.  fmt is per tensor (0 E4M3, 1 E5M2).
template <typename T, int D>
__global__ void __launch_bounds__(quant_threads<D>(), 1024 / quant_threads<D>()) quantize_kernel(const QuantBatch batch) {
  constexpr int kQThreads = quant_threads<D>();
  constexpr int V = Vec<T>::kElems;
  constexpr int kVecs = kTile * D / V;     // vectors in a full tile
  constexpr int kPer = kVecs / kQThreads;  // per thread
  __shared__ float s_red[kQThreads / 32];
  extern __shared__ __align__(16) uint8_t s_codes[];  // [kTile * D] when a transposed copy is wanted

  grid_dependency_sync();
  int j = 0;
  while (j + 1 < batch.count && (int)blockIdx.x >= batch.first_tile[j + 1]) ++j;
  const QuantJob& job = batch.job[j];
  const T* __restrict__ x = static_cast<const T*>(job.x);
  const int N = job.N, T_tiles = job.T_tiles;
  const int tile = (int)blockIdx.x - batch.first_tile[j];
  const int bh = tile / T_tiles, t = tile % T_tiles;
  const int rows = min(kTile, N - t * kTile);
  const size_t base = ((size_t)bh * N + (size_t)t * kTile) * D;
  const int nvec = rows * D / V;

  uint4 raw[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int idx = threadIdx.x + i * kQThreads;
    raw[i] = idx < nvec ? Vec<T>::load(x + base + (size_t)idx * V) : make_uint4(0u, 0u, 0u, 0u);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    float f[V];
    Vec<T>::widen(raw[i], f);
#pragma unroll
    for (int k = 0; k < V; ++k) amax = fmaxf(amax, fabsf(f[k]));
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = s_red[0];
#pragma unroll
  for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, s_red[w]);
  const bool e5m2 = job.fmt != 0;  // uniform over the CTA
  float r;
  const float s = e5m2 ? tile_scale<1>(amax, r) : tile_scale<0>(amax, r);
  if (threadIdx.x == 0) job.scales[tile] = s;
  const bool flushed = (s == 0.0f);  // flushed tile: all codes +0 (x * 0 would give -0 for x < 0)
  uint8_t* codes_t = job.codes_t;

#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int idx = threadIdx.x + i * kQThreads;
    if (idx >= nvec) continue;
    float f[V];
    Vec<T>::widen(raw[i], f);
    uint32_t w[V / 4];
#pragma unroll
    for (int k = 0; k < V / 4; ++k) {
      const float x0 = __fmul_rn(f[4 * k], r), x1 = __fmul_rn(f[4 * k + 1], r);
      const float x2 = __fmul_rn(f[4 * k + 2], r), x3 = __fmul_rn(f[4 * k + 3], r);
      w[k] = flushed ? 0u : (e5m2 ? pack4<1>(x0, x1, x2, x3) : pack4<0>(x0, x1, x2, x3));
    }
    uint8_t* dst = job.codes + base + (size_t)idx * V;
    if constexpr (V == 8) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
      if (codes_t) *reinterpret_cast<uint2*>(s_codes + idx * V) = make_uint2(w[0], w[1]);
    } else {
      *reinterpret_cast<uint32_t*>(dst) = w[0];
      if (codes_t) *reinterpret_cast<uint32_t*>(s_codes + idx * V) = w[0];
    }
  }
  if (codes_t) {
    // transposed copy [bh][d][N]
    __syncthreads();
    uint8_t* out = codes_t + (size_t)bh * D * N + (size_t)t * kTile;
    for (int e = threadIdx.x; e < D * kTile; e += kQThreads) {
      const int c = e / kTile, rr = e % kTile;
      if (rr < rows) out[(size_t)c * N + rr] = s_codes[rr * D + c];
    }
  }
}

template <typename T>
cudaError_t quantize_t(const QuantBatch& b, int d, cudaStream_t st) {
  bool any_t = false;
  for (int j = 0; j < b.count; ++j) any_t = any_t || b.job[j].codes_t;
  const int smem = any_t ? kTile * d : 0;
  const unsigned grid = (unsigned)b.first_tile[b.count];
  if (d == 256)
    quantize_kernel<T, 256><<<grid, quant_threads<256>(), smem, st>>>(b);
  else if (d == 192)
    quantize_kernel<T, 192><<<grid, quant_threads<192>(), smem, st>>>(b);
  else if (d == 128)
    quantize_kernel<T, 128><<<grid, quant_threads<128>(), smem, st>>>(b);
  else
    quantize_kernel<T, 64><<<grid, quant_threads<64>(), smem, st>>>(b);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- stale delta
__device__ __forceinline__ void load_row(const float* p, int k0, int n, float* out) {
  for (int k = 0; k < n; k += 2) {
    const float2 v = *reinterpret_cast<const float2*>(p + k0 + k);
    out[k] = v.x, out[k + 1] = v.y;
  }
}
__device__ __forceinline__ void load_row(const __nv_bfloat16* p, int k0, int n, float* out) {
  for (int k = 0; k < n; k += 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p + k0 + k);
    out[k] = __uint_as_float(w << 16), out[k + 1] = __uint_as_float(w & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void store_row(float* p, int k0, int n, const float* v) {
  for (int k = 0; k < n; k += 2) *reinterpret_cast<float2*>(p + k0 + k) = make_float2(v[k], v[k + 1]);
}
__device__ __forceinline__ void store_row(__nv_bfloat16* p, int k0, int n, const float* v) {
  for (int k = 0; k < n; k += 2)
    *reinterpret_cast<__nv_bfloat162*>(p + k0 + k) = __floats2bfloat162_rn(v[k], v[k + 1]);
}

// MODE 1: delta = <dO, O>; MODE 2: delta = s_dO * <codes(dO^), O>.  Each
// warp takes kStaleRows rows and issues all of their loads before the first
// reduction (each lane d/32 consecutive channels of a row, 16-byte loads of O
// where a lane's share allows), so that enough bytes are in flight per SM.
constexpr int kStaleRows = 4;

template <int PER>
__device__ __forceinline__ void load_vals(const float* p, float* out) {
  if constexpr (PER % 4 == 0) {
#pragma unroll
    for (int k = 0; k < PER; k += 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(p + k));
      out[k] = v.x, out[k + 1] = v.y, out[k + 2] = v.z, out[k + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < PER; k += 2) {
      const float2 v = __ldg(reinterpret_cast<const float2*>(p + k));
      out[k] = v.x, out[k + 1] = v.y;
    }
  }
}
template <int PER>
__device__ __forceinline__ void load_vals(const __nv_bfloat16* p, float* out) {
  if constexpr (PER % 4 == 0) {
#pragma unroll
    for (int k = 0; k < PER; k += 4) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(p + k));
      out[k] = __uint_as_float(w.x << 16), out[k + 1] = __uint_as_float(w.x & 0xFFFF0000u);
      out[k + 2] = __uint_as_float(w.y << 16), out[k + 3] = __uint_as_float(w.y & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int k = 0; k < PER; k += 2) {
      const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(p + k));
      out[k] = __uint_as_float(w << 16), out[k + 1] = __uint_as_float(w & 0xFFFF0000u);
    }
  }
}

template <int MODE, int D, typename TD, typename TO>
__global__ void __launch_bounds__(256) stale_delta_kernel(const TD* __restrict__ dO,
                                                          const uint8_t* __restrict__ do_codes,
                                                          const float* __restrict__ do_scales,
                                                          const TO* __restrict__ O, long long rows, int N,
                                                          int T_tiles, float* __restrict__ delta) {
  constexpr int PER = D / 32;
  const long long row0 = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * kStaleRows;
  const int lane = threadIdx.x & 31;
  if (row0 >= rows) return;
  float o[kStaleRows][PER], g[kStaleRows][PER];
#pragma unroll
  for (int rr = 0; rr < kStaleRows; ++rr) {
    const long long row = row0 + rr < rows ? row0 + rr : rows - 1;  // a ragged last warp rereads its last row
    const size_t off = (size_t)row * D + lane * PER;
    load_vals<PER>(O + off, o[rr]);
    if (MODE == 1) {
      load_vals<PER>(dO + off, g[rr]);
    } else {
#pragma unroll
      for (int k = 0; k < PER; k += 2) {
        const float2 f = unpack2<1>(__ldg(reinterpret_cast<const unsigned short*>(do_codes + off + k)));
        g[rr][k] = f.x, g[rr][k + 1] = f.y;
      }
    }
  }
#pragma unroll
  for (int rr = 0; rr < kStaleRows; ++rr) {
    const long long row = row0 + rr;
    float acc = 0.0f;
#pragma unroll
    for (int k = 0; k < PER; ++k) acc = fmaf(g[rr][k], o[rr][k], acc);
    acc = warp_sum(acc);
    if (lane == 0 && row < rows) {
      float sc = 1.0f;
      if (MODE == 2) sc = do_scales[(row / N) * T_tiles + (int)(row % N) / kTile];
      delta[row] = acc * sc;
    }
  }
}

template <int MODE, int D, typename TD>
cudaError_t stale_o(const TD* dO, const uint8_t* codes, const float* scales, const void* O, dm_dtype o_t,
                    long long rows, int N, int T, float* delta, cudaStream_t st) {
  const unsigned grid = (unsigned)((rows + 8 * kStaleRows - 1) / (8 * kStaleRows));
  if (o_t == DM_BF16)
    stale_delta_kernel<MODE, D, TD, __nv_bfloat16><<<grid, 256, 0, st>>>(
        dO, codes, scales, reinterpret_cast<const __nv_bfloat16*>(O), rows, N, T, delta);
  else
    stale_delta_kernel<MODE, D, TD, float><<<grid, 256, 0, st>>>(dO, codes, scales,
                                                                 reinterpret_cast<const float*>(O), rows, N, T,
                                                                 delta);
  return cudaGetLastError();
}

template <int D>
cudaError_t stale_d(const AttnArgs& a, dm_delta_mode mode, const void* dO, dm_dtype do_t, const uint8_t* codes,
                    const void* O, dm_dtype o_t, float* delta, cudaStream_t st) {
  const long long rows = (long long)a.B * a.Hq * a.N;
  if (mode == DM_DELTA_STALE_DOHAT)
    return stale_o<2, D, float>(nullptr, codes, a.do_scales, O, o_t, rows, a.N, a.T, delta, st);
  if (do_t == DM_BF16)
    return stale_o<1, D, __nv_bfloat16>(reinterpret_cast<const __nv_bfloat16*>(dO), nullptr, nullptr, O, o_t,
                                        rows, a.N, a.T, delta, st);
  return stale_o<1, D, float>(reinterpret_cast<const float*>(dO), nullptr, nullptr, O, o_t, rows, a.N, a.T,
                              delta, st);
}

// Merge of nparts stacked key-block results, one warp per row, each lane
// holding D/32 consecutive channels: O_parts [nparts][rows][D] fp32,
// lse_parts [nparts][rows].  Blocks that see none of a row's keys carry
// LSE = -inf and weigh zero; a row no block sees gets O = 0, LSE = -inf.
template <int D, typename TO>
__global__ void __launch_bounds__(256) merge_kernel(int nparts, const float* __restrict__ O_parts,
                                                    const float* __restrict__ lse_parts, long long rows,
                                                    TO* __restrict__ O, float* __restrict__ lse) {
  constexpr int PER = D / 32;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float m = -INFINITY;
  for (int r = 0; r < nparts; ++r) m = fmaxf(m, __ldg(lse_parts + r * rows + row));
  float o[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) o[k] = 0.0f;
  float lse_row = -INFINITY;
  if (m != -INFINITY) {
    float wsum = 0.0f;
    for (int r = 0; r < nparts; ++r) {
      const float w = expf(__ldg(lse_parts + r * rows + row) - m);
      wsum += w;
      if (w == 0.0f) continue;  // uniform over the warp (one row)
      float x[PER];
      load_row(O_parts + ((size_t)r * rows + row) * D, lane * PER, PER, x);
#pragma unroll
      for (int k = 0; k < PER; ++k) o[k] = fmaf(w, x[k], o[k]);
    }
    const float inv = 1.0f / wsum;
#pragma unroll
    for (int k = 0; k < PER; ++k) o[k] *= inv;
    lse_row = m + logf(wsum);
  }
  store_row(O + (size_t)row * D, lane * PER, PER, o);
  if (lane == 0) lse[row] = lse_row;
}

// delta = sum_r num_r / sum_r den_r per row (0 where no block sees the row).
__global__ void __launch_bounds__(256) delta_combine_kernel(int nparts, const float* __restrict__ num,
                                                            const float* __restrict__ den, long long rows,
                                                            float* __restrict__ delta) {
  for (long long row = (long long)blockIdx.x * blockDim.x + threadIdx.x; row < rows;
       row += (long long)gridDim.x * blockDim.x) {
    float a = 0.0f, b = 0.0f;
    for (int r = 0; r < nparts; ++r) {
      a += __ldg(num + r * rows + row);
      b += __ldg(den + r * rows + row);
    }
    delta[row] = b > 0.0f ? a / b : 0.0f;
  }
}

template <int D>
cudaError_t merge_d(int nparts, const float* O_parts, const float* lse_parts, long long rows, void* O, bool o_bf16,
                    float* lse, cudaStream_t st) {
  const unsigned grid = (unsigned)((rows + 7) / 8);
  if (o_bf16)
    merge_kernel<D, __nv_bfloat16><<<grid, 256, 0, st>>>(nparts, O_parts, lse_parts, rows,
                                                          reinterpret_cast<__nv_bfloat16*>(O), lse);
  else
    merge_kernel<D, float><<<grid, 256, 0, st>>>(nparts, O_parts, lse_parts, rows, reinterpret_cast<float*>(O), lse);
  return cudaGetLastError();
}

// Zero fill of several FP32 buffers in one launch.  Each buffer is written
// with 16-byte stores between its first and last 16-byte boundary and with
// scalar stores at its ragged ends, so any 4-byte aligned pointer works.
__global__ void zero_kernel(const ZeroList z) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int s = 0; s < z.count; ++s) {
    float* p = z.p[s];
    const size_t n = z.n[s];
    size_t head = ((16 - ((uintptr_t)p & 15)) & 15) / 4;
    if (head > n) head = n;
    const size_t n4 = (n - head) / 4;
    float4* p4 = reinterpret_cast<float4*>(p + head);
    for (size_t i = i0; i < n4; i += stride) p4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i0 < head) p[i0] = 0.0f;
    for (size_t i = head + 4 * n4 + i0; i < n; i += stride) p[i] = 0.0f;
  }
}

}  // namespace

cudaError_t launch_quantize(const QuantBatch& b, dm_dtype xt, int d, cudaStream_t st) {
  if (b.count == 0 || b.first_tile[b.count] == 0) return cudaSuccess;
  return xt == DM_BF16 ? quantize_t<__nv_bfloat16>(b, d, st) : quantize_t<float>(b, d, st);
}

cudaError_t launch_delta_stale(const AttnArgs& a, int d, dm_delta_mode mode, const void* dO, dm_dtype do_t,
                               const uint8_t* do_codes, const void* O, dm_dtype o_t, float* delta,
                               cudaStream_t st) {
  if (d == 256) return stale_d<256>(a, mode, dO, do_t, do_codes, O, o_t, delta, st);
  if (d == 192) return stale_d<192>(a, mode, dO, do_t, do_codes, O, o_t, delta, st);
  return d == 128 ? stale_d<128>(a, mode, dO, do_t, do_codes, O, o_t, delta, st)
                  : stale_d<64>(a, mode, dO, do_t, do_codes, O, o_t, delta, st);
}

cudaError_t launch_attn_merge(int nparts, const float* O_parts, const float* lse_parts, long long rows, int dv,
                              void* O, bool o_bf16, float* lse, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  if (dv == 256) return merge_d<256>(nparts, O_parts, lse_parts, rows, O, o_bf16, lse, st);
  if (dv == 192) return merge_d<192>(nparts, O_parts, lse_parts, rows, O, o_bf16, lse, st);
  return dv == 128 ? merge_d<128>(nparts, O_parts, lse_parts, rows, O, o_bf16, lse, st)
                   : merge_d<64>(nparts, O_parts, lse_parts, rows, O, o_bf16, lse, st);
}

cudaError_t launch_delta_combine(int nparts, const float* num_parts, const float* den_parts, long long rows,
                                 float* delta, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  long long blocks = (rows + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  delta_combine_kernel<<<(unsigned)blocks, 256, 0, st>>>(nparts, num_parts, den_parts, rows, delta);
  return cudaGetLastError();
}

cudaError_t launch_zero(const ZeroList& z, cudaStream_t st) {
  size_t total = 0;
  for (int s = 0; s < z.count; ++s) total += z.n[s];
  if (total == 0) return cudaSuccess;
  size_t blocks = (total / 4 + 255) / 256 + 1;
  if (blocks > 152 * 16) blocks = 152 * 16;
  zero_kernel<<<(unsigned)blocks, 256, 0, st>>>(z);
  return cudaGetLastError();
}

}  // namespace dm
