// Forward: O = P^ V^ and LSE, one CTA per (batch, query head, 128-row query
// tile), with both matmuls on tcgen05 FP8 MMAs ("Delta-Matching for reliable
// FP8 attention training", section 01: "What changes in FP8?").
//
// Warp roles (320 threads):
//   warp 0      TMA producer: Q tile once, K/V tiles double-buffered
//   warp 1      MMA issuer (+ TMEM owner): S(t) = Q K_t^T into TMEM S[t%2];
//               O_t = P^_t V_t into TMEM O[t%2]
//   warps 2-5   softmax: one thread per query row; online row max, P~ in FP32,
//               per-tile amax -> E4M3 codes written to shared memory
//   warps 6-9   correction: O accumulated in registers in true units,
//               acc = alpha * acc + (s_P * s_V) * O_t, then O / l
//
// Each key tile t brings its own FP32 scale product s_P,t * s_V,t, so the
// tiles' products are summed outside the tensor core; the S/O double buffers
// let S(t+1) run on the tensor core while the softmax works on S(t).
//
// TMEM columns (512 allocated): S[0] 0-127, S[1] 128-255, O[0] 256.., O[1] 384..
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "dm_device.cuh"
#include "dm_internal.h"

namespace dm {
namespace {

constexpr int kThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct FwdLayout {
  static constexpr int kTileBytes = kTile * D;  // one FP8 Q/K/V tile
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;           // 2 stages
  static constexpr int kV = kK + 2 * kTileBytes;       // 2 stages
  static constexpr int kP = kV + 2 * kTileBytes;       // 2 x (128 x 128) P^ codes
  static constexpr int kBytes = kP + 2 * kTile * kTile;
  static constexpr int kDynSmem = kBytes + 1024;       // + alignment slack
};

struct FwdBars {
  uint64_t q, kfull[2], kempty[2], vfull[2], vempty[2], sfull[2], sempty[2], pfull[2], ofull[2], oempty[2],
      fin, stall, mma_done;
};

template <int D, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnArgs a, void* __restrict__ O,
                    float* __restrict__ lse) {
  using L = FwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ FwdBars bars;
  __shared__ float s_alpha[2][kTile];
  __shared__ float s_cs[2];
  __shared__ float s_linv[kTile];
  __shared__ float s_red[2][4];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = a.B * a.Hq;
  const int qt = a.T - 1 - (int)(blockIdx.x / BH);  // longest causal rows first
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / a.Hq, h = bh % a.Hq;
  const int bg = b * a.Hkv + h / (a.Hq / a.Hkv);
  const int q0 = qt * kTile;
  const int nkv = a.causal ? qt + 1 : a.T;

  Watchdog wd{&s_abort, a.status, a.wait_limit_ns};
  if (tid == 0) {
    s_abort = 0;
    mbar_init(&bars.q, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.kfull[s], 1);
      mbar_init(&bars.kempty[s], 1);
      mbar_init(&bars.vfull[s], 1);
      mbar_init(&bars.vempty[s], 1);
      mbar_init(&bars.sfull[s], 1);
      mbar_init(&bars.sempty[s], 4);
      mbar_init(&bars.pfull[s], 4);
      mbar_init(&bars.ofull[s], 1);
      mbar_init(&bars.oempty[s], 4);
    }
    mbar_init(&bars.fin, 4);
    mbar_init(&bars.stall, 1);
    mbar_init(&bars.mma_done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(&bars.q, L::kTileBytes);
      tma_load_3d(sm + L::kQ, &tmQ, &bars.q, 0, q0, bh);
      int issued = 0;  // K/V tiles whose loads were issued (stops early on abort)
      for (int t = 0; t < nkv; ++t) {
        const int s = t & 1;
        const uint32_t ph = (t >> 1) & 1;
        if (!wait(&bars.kempty[s], ph ^ 1, wd, 101)) break;
        if (!wait(&bars.vempty[s], ph ^ 1, wd, 102)) break;
        mbar_arrive_expect_tx(&bars.kfull[s], L::kTileBytes);
        tma_load_3d(sm + L::kK + s * L::kTileBytes, &tmK, &bars.kfull[s], 0, t * kTile, bg);
        mbar_arrive_expect_tx(&bars.vfull[s], L::kTileBytes);
        tma_load_3d(sm + L::kV + s * L::kTileBytes, &tmV, &bars.vfull[s], 0, t * kTile, bg);
        issued = t + 1;
      }
      // every issued load has landed before the CTA may exit
      wait_drain(&bars.q, 0, wd, 116);
      for (int t = max(0, issued - 2); t < issued; ++t) {
        wait_drain(&bars.kfull[t & 1], (t >> 1) & 1, wd, 117);
        wait_drain(&bars.vfull[t & 1], (t >> 1) & 1, wd, 118);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f8(0, 0, 0, 0, kTile, kTile);  // Q K^T, both K-major
      constexpr uint32_t kIdO = idesc_f8(0, 0, 0, 1, kTile, D);      // P^ (K-major) V (MN-major)
      bool ok = true;
      if (a.stall_test) ok = wait(&bars.stall, 0, wd, 103);  // watchdog test: never signalled
      ok = ok && wait(&bars.q, 0, wd, 104);
      tc_fence_after();
      const uint32_t sQ = smem_u32(sm + L::kQ);
      for (int t = 0; t <= nkv && ok; ++t) {
        if (t < nkv) {
          const int s = t & 1;
          const uint32_t ph = (t >> 1) & 1;
          ok = wait(&bars.kfull[s], ph, wd, 105) && wait(&bars.sempty[s], ph ^ 1, wd, 106);
          if (!ok) break;
          tc_fence_after();
          const uint32_t sK = smem_u32(sm + L::kK + s * L::kTileBytes);
#pragma unroll
          for (int k = 0; k < D / 32; ++k)
            mma_f8(tmem + s * 128, SwTile<D>::kmajor(sQ, k), SwTile<D>::kmajor(sK, k), kIdS, k > 0);
          mma_commit(&bars.sfull[s]);
          mma_commit(&bars.kempty[s]);
        }
        if (t >= 1) {
          const int u = t - 1, s = u & 1;
          const uint32_t ph = (u >> 1) & 1;
          ok = wait(&bars.pfull[s], ph, wd, 107) && wait(&bars.vfull[s], ph, wd, 108) && wait(&bars.oempty[s], ph ^ 1, wd, 109);
          if (!ok) break;
          tc_fence_after();
          const uint32_t sP = smem_u32(sm + L::kP + s * kTile * kTile);
          const uint32_t sV = smem_u32(sm + L::kV + s * L::kTileBytes);
#pragma unroll
          for (int k = 0; k < kTile / 32; ++k)
            mma_f8(tmem + 256 + s * 128, SwTile<128>::kmajor(sP, k), SwTile<D>::mnmajor(sV, k), kIdO, k > 0);
          mma_commit(&bars.ofull[s]);
          mma_commit(&bars.vempty[s]);
        }
      }
      mma_commit(&bars.mma_done);
      wait_drain(&bars.mma_done, 0, wd, 119);
    }
  } else if (warp < 6) {
    // -------------------------------------------------------------- softmax
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int qi = q0 + row;
    const bool row_valid = qi < a.N;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sq = a.q_scales[bh * a.T + qt];
    const float* ksc = a.k_scales + (size_t)bg * a.T;
    const float* vsc = a.v_scales + (size_t)bg * a.T;
    float sk_next = ksc[0], sv_next = vsc[0];  // per-tile scales, loaded one tile ahead
    float m = -INFINITY, l = 0.0f;  // running max (log2 units) and row sum
    for (int t = 0; t < nkv; ++t) {
      const int s = t & 1;
      const uint32_t ph = (t >> 1) & 1;
      const float c1 = a.sigma * sq * sk_next * kLog2e;
      const float sv = sv_next;
      if (t + 1 < nkv) {
        sk_next = ksc[t + 1];
        sv_next = vsc[t + 1];
      }
      const int j0 = t * kTile;
      int jlim = min(kTile, a.N - j0);
      if (a.causal) jlim = min(jlim, qi - j0 + 1);

      wait(&bars.sfull[s], ph, wd, 110);
      tc_fence_after();
      float v[kTile];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tl + s * 128 + c * 32, *reinterpret_cast<float(*)[32]>(&v[c * 32]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.sempty[s]);

      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kTile; ++c)
        if (c < jlim) mx = fmaxf(mx, v[c]);
      const float tmax = mx * c1;
      const float m_new = fmaxf(m, tmax);
      // amax of this tile of P~ = max over its rows of exp2(tile row max - running max)
      float arow = row_valid ? ex2(tmax - m_new) : 0.0f;
      arow = warp_max(arow);
      if (lane == 0) s_red[s][quarter] = arow;
      named_bar_sync(1, 128);
      const float amax = fmaxf(fmaxf(s_red[s][0], s_red[s][1]), fmaxf(s_red[s][2], s_red[s][3]));
      float r;
      const float sp = tile_scale<0>(amax, r);

      const float alpha = ex2(m - m_new);
      float rowsum = 0.0f;
      uint32_t packed[kTile / 4];
#pragma unroll
      for (int c = 0; c < kTile; c += 4) {
        float p[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) p[k] = (c + k < jlim) ? ex2(fmaf(v[c + k], c1, -m_new)) : 0.0f;
        rowsum += (p[0] + p[1]) + (p[2] + p[3]);
        packed[c / 4] = pack4_e4m3(__fmul_rn(p[0], r), __fmul_rn(p[1], r), __fmul_rn(p[2], r), __fmul_rn(p[3], r));
      }
      l = alpha * l + rowsum;
      m = m_new;

      if (t >= 2) {
        wait(&bars.ofull[s], ph ^ 1, wd, 111);   // PV(t-2) has read P buffer s
        wait(&bars.oempty[s], ph ^ 1, wd, 112);  // correction has read alpha/cs of t-2
      }
      uint8_t* sP = sm + L::kP + s * kTile * kTile;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(sP + SwTile<128>::chunk_offset(row, c)) =
            make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
      s_alpha[s][row] = alpha;
      if (row == 0) s_cs[s] = sp * sv;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.pfull[s]);
    }
    if (row_valid) lse[(size_t)bh * a.N + qi] = m * kLn2 + logf(l);
    s_linv[row] = 1.0f / l;
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.fin);
  } else {
    // ----------------------------------------------------------- correction
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int qi = q0 + row;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    float acc[D];
#pragma unroll
    for (int k = 0; k < D; ++k) acc[k] = 0.0f;
    for (int t = 0; t < nkv; ++t) {
      const int s = t & 1;
      const uint32_t ph = (t >> 1) & 1;
      wait(&bars.pfull[s], ph, wd, 113);
      wait(&bars.ofull[s], ph, wd, 114);
      tc_fence_after();
      const float alpha = s_alpha[s][row];
      const float cs = s_cs[s];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float v[32];
        tmem_ld32(tl + 256 + s * 128 + c * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) acc[c * 32 + k] = fmaf(cs, v[k], alpha * acc[c * 32 + k]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.oempty[s]);
    }
    wait(&bars.fin, 0, wd, 115);
    const float linv = s_linv[row];
    if (qi < a.N) {
      if (OUT_BF16) {
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(O) + ((size_t)bh * a.N + qi) * D;
#pragma unroll
        for (int k = 0; k < D; k += 8) {
          uint4 w;
          uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[k + 2 * e] * linv, acc[k + 2 * e + 1] * linv);
            wp[e] = *reinterpret_cast<uint32_t*>(&h2);
          }
          *reinterpret_cast<uint4*>(o + k) = w;
        }
      } else {
        float* o = reinterpret_cast<float*>(O) + ((size_t)bh * a.N + qi) * D;
#pragma unroll
        for (int k = 0; k < D; k += 4)
          *reinterpret_cast<float4*>(o + k) =
              make_float4(acc[k] * linv, acc[k + 1] * linv, acc[k + 2] * linv, acc[k + 3] * linv);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BF16>
cudaError_t launch_fwd_t(const FwdLaunch& f, cudaStream_t st) {
  auto k = attn_fwd_kernel<D, BF16>;
  constexpr int smem = FwdLayout<D>::kDynSmem;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(f.args.B * f.args.Hq * f.args.T);
  k<<<grid, kThreads, smem, st>>>(f.tmQ, f.tmK, f.tmV, f.args, f.O, f.lse);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const FwdLaunch& f, int d, bool o_bf16, cudaStream_t st) {
  if (d == 128) return o_bf16 ? launch_fwd_t<128, true>(f, st) : launch_fwd_t<128, false>(f, st);
  return o_bf16 ? launch_fwd_t<64, true>(f, st) : launch_fwd_t<64, false>(f, st);
}

}  // namespace dm
