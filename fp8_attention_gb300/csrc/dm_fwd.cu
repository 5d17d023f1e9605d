// Forward: O = P^ V^ and LSE, one CTA per (batch, query head, 128-row query
// tile), with both matmuls on tcgen05 FP8 MMAs ("Delta-Matching for reliable
// FP8 attention training", section 01: "What changes in FP8?").
//
// Warp roles (384 threads):
//   warp 0      TMA producer: Q tile once, K/V tiles in kKV stages (K one
//               tile ahead of V)
//   warp 1      S issuer (+ TMEM owner): S(t) = Q K_t^T into TMEM S[t%2]
//   warp 3      O issuer: O_t = P^_t V_t into TMEM O[t%2]
//   warp 2      idle (each warpgroup starts at a multiple of four warps)
//   warps 4-11  two warpgroups; thread = query row (TMEM lane), warpgroup =
//               half of the key columns for the softmax and half of the d
//               columns for O.  Per key tile t: online row max (the halves
//               exchange partial maxima through shared memory), P~ in FP32,
//               the tile's amax -> E4M3 codes into shared memory; then, one
//               tile behind, O_acc = alpha * O_acc + (s_P * s_V) * O_{t-1} in
//               registers.
//
// Each key tile brings its own FP32 scale product s_P,t * s_V,t, so the
// tiles' products are summed outside the tensor core.  The O update lags one
// tile: it runs while the tensor core computes the next S and P V products.
//
// TMEM columns (512 allocated): S[0] 0-127, S[1] 128-255, O[0] 256.., O[1] 384..
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <type_traits>

#include "dm_device.cuh"
#include "dm_internal.h"

namespace dm {
namespace {

constexpr int kGroups = 2;                // compute warpgroups
constexpr int kWarps = 4 * kGroups;      // compute warps
constexpr int kThreads = 128 + 32 * kWarps;  // warps 0-3: TMA, MMA, two idle; then the compute warpgroups
constexpr int kCols = kTile / kGroups;    // key columns per thread
constexpr int kKV = 4;                    // K and V shared-memory stages (loads run ahead of the products)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct FwdBars {
  uint64_t q, kfull[kKV], kempty[kKV], vfull[kKV], vempty[kKV], sfull[2], sempty[2], pfull[2], ofull[2], oempty[2],
      stall, mma_done, mma_done2;
};

// Everything lives in dynamic shared memory (no static shared variables), so
// the 1024-byte aligned tile region starts at the window's base.
template <int D>
struct FwdLayout {
  static constexpr int kTileBytes = kTile * D;  // one FP8 Q/K/V tile
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;              // kKV stages
  static constexpr int kV = kK + kKV * kTileBytes;        // kKV stages
  static constexpr int kP = kV + kKV * kTileBytes;        // 2 x (128 x 128) P^ codes
  static constexpr int kRmax = kP + 2 * kTile * kTile;          // float [2][kGroups][128] partial row maxima
  static constexpr int kRed = kRmax + 2 * kGroups * kTile * 4;  // float [2][kWarps] tile amax partials
  static constexpr int kL = kRed + 2 * kWarps * 4;              // float [kGroups][128] row sums
  static constexpr int kBars = kL + kGroups * kTile * 4;
  static constexpr int kMisc = kBars + ((int)(sizeof(FwdBars) + 15) / 16) * 16;  // tmem address, abort flag
  static constexpr int kBytes = kMisc + 16;
};

template <int D, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnArgs a, void* __restrict__ O,
                    float* __restrict__ lse) {
  using L = FwdLayout<D>;
  constexpr int DH = D / kGroups;  // O columns per warpgroup
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  FwdBars& bars = *reinterpret_cast<FwdBars*>(sm + L::kBars);
  float(*s_rmax)[kGroups][kTile] = reinterpret_cast<float(*)[kGroups][kTile]>(sm + L::kRmax);
  float(*s_red)[kWarps] = reinterpret_cast<float(*)[kWarps]>(sm + L::kRed);
  float(*s_l)[kTile] = reinterpret_cast<float(*)[kTile]>(sm + L::kL);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  int* s_abort = reinterpret_cast<int*>(sm + L::kMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = a.B * a.Hq;
  const int qt = a.T - 1 - (int)(blockIdx.x / BH);  // longest causal rows first
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / a.Hq, h = bh % a.Hq;
  const int bg = b * a.Hkv + h / (a.Hq / a.Hkv);
  const int q0 = qt * kTile;
  const int nkv = a.causal ? qt + 1 : a.T;

  // the swizzled tiles need a 1024-byte aligned window (no static shared variables)
  if (smem_u32(smem_raw) & 1023u) {
    if (tid == 0) atomicCAS(a.status, 0u, (unsigned)DM_ERR_UNSUPPORTED);
    return;
  }
  Watchdog wd{s_abort, a.status, a.wait_limit_ns};
  if (tid == 0) {
    *s_abort = 0;
    mbar_init(&bars.q, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.sfull[s], 1);
      mbar_init(&bars.sempty[s], kWarps);
      mbar_init(&bars.pfull[s], kWarps);
      mbar_init(&bars.ofull[s], 1);
      mbar_init(&bars.oempty[s], kWarps);
    }
    for (int s = 0; s < kKV; ++s) {
      mbar_init(&bars.kfull[s], 1);
      mbar_init(&bars.kempty[s], 1);
      mbar_init(&bars.vfull[s], 1);
      mbar_init(&bars.vempty[s], 1);
    }
    mbar_init(&bars.stall, 1);
    mbar_init(&bars.mma_done, 1);
    mbar_init(&bars.mma_done2, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(&bars.q, L::kTileBytes);
      tma_load_3d(sm + L::kQ, &tmQ, &bars.q, 0, q0, bh);
      // K runs one tile ahead of V: K(t) needs only S(t-2) to have finished
      // with its stage, V(t) needs P V(t-2), which completes a tile later.
      int k_issued = 0, v_issued = 0;  // loads issued (both stop early on abort)
      for (int t = 0; t <= nkv; ++t) {
        if (t < nkv) {
          const int s = t % kKV;
          if (!wait(&bars.kempty[s], ((t / kKV) & 1) ^ 1, wd, 101)) break;
          mbar_arrive_expect_tx(&bars.kfull[s], L::kTileBytes);
          tma_load_3d(sm + L::kK + s * L::kTileBytes, &tmK, &bars.kfull[s], 0, t * kTile, bg);
          k_issued = t + 1;
        }
        if (t >= 1) {
          const int u = t - 1, s = u % kKV;
          if (!wait(&bars.vempty[s], ((u / kKV) & 1) ^ 1, wd, 102)) break;
          mbar_arrive_expect_tx(&bars.vfull[s], L::kTileBytes);
          tma_load_3d(sm + L::kV + s * L::kTileBytes, &tmV, &bars.vfull[s], 0, u * kTile, bg);
          v_issued = u + 1;
        }
      }
      // every issued load has landed before the CTA may exit
      wait_drain(&bars.q, 0, wd, 116);
      for (int t = max(0, k_issued - kKV); t < k_issued; ++t)
        wait_drain(&bars.kfull[t % kKV], (t / kKV) & 1, wd, 117);
      for (int t = max(0, v_issued - kKV); t < v_issued; ++t)
        wait_drain(&bars.vfull[t % kKV], (t / kKV) & 1, wd, 118);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- S = Q K^T issuer
    // (two issuing threads: one thread's barrier waits stall its own
    // tcgen05.mma stream, and the other keeps the tensor pipe fed meanwhile)
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f8(0, 0, 0, 0, kTile, kTile);  // Q K^T, both K-major
      bool ok = true;
      if (a.stall_test) {
        // watchdog test: a barrier nothing signals, with half the limit so
        // that it expires before the waits that depend on it
        const Watchdog wd_half{wd.abort_flag, wd.status, wd.limit_ns / 2};
        ok = wait(&bars.stall, 0, wd_half, 103);
      }
      ok = ok && wait(&bars.q, 0, wd, 104);
      tc_fence_after();
      const uint32_t sQ = smem_u32(sm + L::kQ);
      for (int t = 0; t < nkv && ok; ++t) {
        const int s = t & 1;
        const uint32_t ph = (t >> 1) & 1;
        const int ks = t % kKV;
        ok = wait(&bars.kfull[ks], (t / kKV) & 1, wd, 105) && wait(&bars.sempty[s], ph ^ 1, wd, 106);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sK = smem_u32(sm + L::kK + ks * L::kTileBytes);
#pragma unroll
        for (int k = 0; k < D / 32; ++k)
          mma_f8(tmem + s * 128, SwTile<D>::kmajor(sQ, k), SwTile<D>::kmajor(sK, k), kIdS, k > 0);
        mma_commit(&bars.sfull[s]);
        mma_commit(&bars.kempty[ks]);
      }
      mma_commit(&bars.mma_done);
      wait_drain(&bars.mma_done, 0, wd, 119);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------- O_u = P^ V issuer
    if (lane == 0) {
      constexpr uint32_t kIdO = idesc_f8(0, 0, 0, 1, kTile, D);  // P^ (K-major) V (MN-major)
      bool ok = true;
      for (int u = 0; u < nkv && ok; ++u) {
        const int s = u & 1;
        const uint32_t ph = (u >> 1) & 1;
        const int vs = u % kKV;
        ok = wait(&bars.pfull[s], ph, wd, 107) && wait(&bars.vfull[vs], (u / kKV) & 1, wd, 108) &&
             wait(&bars.oempty[s], ph ^ 1, wd, 109);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sP = smem_u32(sm + L::kP + s * kTile * kTile);
        const uint32_t sV = smem_u32(sm + L::kV + vs * L::kTileBytes);
#pragma unroll
        for (int k = 0; k < kTile / 32; ++k)
          mma_f8(tmem + 256 + s * 128, SwTile<128>::kmajor(sP, k), SwTile<D>::mnmajor(sV, k), kIdO, k > 0);
        mma_commit(&bars.ofull[s]);
        mma_commit(&bars.vempty[vs]);
      }
      mma_commit(&bars.mma_done2);
      wait_drain(&bars.mma_done2, 0, wd, 120);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ softmax and O update
    constexpr int kCT = 32 * kWarps;  // compute threads
    const int wg = (warp - 4) >> 2;   // key-column and O-column quarter
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int qi = q0 + row;
    const bool row_valid = qi < a.N;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sq = a.q_scales[bh * a.T + qt];
    const float* ksc = a.k_scales + (size_t)bg * a.T;
    const float* vsc = a.v_scales + (size_t)bg * a.T;
    float sk_next = ksc[0], sv_next = vsc[0];  // per-tile scales, loaded one tile ahead
    float m = -INFINITY, l = 0.0f;             // running max (log2 units), row sum of this quarter
    float2 acc[DH / 2];                        // O / unit, packed pairs of d columns
#pragma unroll
    for (int k = 0; k < DH / 2; ++k) acc[k] = make_float2(0.0f, 0.0f);
    float unit = 0.0f;                         // O in true units = unit * acc (0: nothing added yet)
    float alpha_prev = 0.0f, c_prev = 0.0f;    // the previous tile's rescale and scale product

    // O_true = alpha * O_true + c * O_u over this warpgroup's d columns, kept
    // in units of the latest scale product: acc = acc * (alpha * unit / c) + O_u
    // (one packed FMA per pair).  When c is zero (a flushed P or V tile) or
    // so small that the factor would exceed 2^64, the unit stays and the
    // general form acc = acc * alpha + O_u * (c / unit) is used.
    auto update_o = [&](int u, float alpha, float c) {
      const int su = u & 1;
      wait(&bars.ofull[su], (u >> 1) & 1, wd, 114);
      tc_fence_after();
      const float f_fast = __fdividef(alpha * unit, c);
      const bool fast = c != 0.0f && f_fast <= 0x1p64f;  // false for NaN
      const float f = fast ? f_fast : alpha;
      const float g = fast || c == 0.0f ? 0.0f : __fdividef(c, unit);
      if (fast) unit = c;
      const float2 f2 = make_float2(f, f), g2 = make_float2(g, g);
      float v[DH];  // warp-collective load: before any branch
      tmem_load_cols<DH>(tl + 256 + su * 128 + wg * DH, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.oempty[su]);
      if (fast) {
#pragma unroll
        for (int k = 0; k < DH; k += 2) acc[k / 2] = __ffma2_rn(acc[k / 2], f2, make_float2(v[k], v[k + 1]));
      } else {
#pragma unroll
        for (int k = 0; k < DH; k += 2)
          acc[k / 2] = __ffma2_rn(make_float2(v[k], v[k + 1]), g2, __fmul2_rn(acc[k / 2], f2));
      }
    };

    for (int t = 0; t < nkv; ++t) {
      const int s = t & 1;
      const uint32_t ph = (t >> 1) & 1;
      const float c1 = a.sigma * sq * sk_next * kLog2e;
      const float sv = sv_next;
      if (t + 1 < nkv) {
        sk_next = ksc[t + 1];
        sv_next = vsc[t + 1];
      }
      const int j0 = t * kTile + wg * kCols;
      int jlim = min(kCols, a.N - j0);
      if (a.causal) jlim = min(jlim, qi - j0 + 1);

      wait(&bars.sfull[s], ph, wd, 110);
      tc_fence_after();
      float v[kCols];
      tmem_load_cols<kCols>(tl + s * 128 + wg * kCols, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.sempty[s]);

      // row max over the four quarters (raw units; c1 > 0 preserves the order)
      const bool full = jlim >= kCols;  // no masked column here (all but the diagonal/ragged tile)
      float mx = -INFINITY;
      if (full) {
        float m4[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
        for (int c = 4; c < kCols; c += 8) {
          m4[0] = max3(m4[0], v[c], v[c + 1]);
          m4[1] = max3(m4[1], v[c + 2], v[c + 3]);
          m4[2] = max3(m4[2], v[c + 4], v[c + 5]);
          m4[3] = max3(m4[3], v[c + 6], v[c + 7]);
        }
        mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      } else {
#pragma unroll
        for (int c = 0; c < kCols; ++c)
          if (c < jlim) mx = fmaxf(mx, v[c]);
      }
      s_rmax[s][wg][row] = mx;
      named_bar_sync(1, kCT);
      float tmax = s_rmax[s][0][row];
#pragma unroll
      for (int g = 1; g < kGroups; ++g) tmax = fmaxf(tmax, s_rmax[s][g][row]);
      tmax *= c1;
      const float m_new = fmaxf(m, tmax);
      // amax of this tile of P~ = max over its rows of exp2(tile row max - running max)
      float arow = row_valid ? ex2(tmax - m_new) : 0.0f;
      arow = warp_max(arow);
      if (lane == 0) s_red[s][warp - 4] = arow;
      named_bar_sync(1, kCT);
      float amax = s_red[s][0];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) amax = fmaxf(amax, s_red[s][w]);
      float r;
      const float sp = tile_scale_fast<0>(amax, r);
      const float alpha = ex2(m - m_new);

      // P~ r = exp2(S c1 - m + log2 r) straight into E4M3 codes (P buffer s;
      // its last reader, the P V product of tile t-2, completed before this
      // thread's O update of tile t-2); the unquantised row sum of this
      // quarter is sum(P~ r) * s_P.  A flushed tile (r = 0) gives codes 0.
      const float bias = (r > 0.0f ? __log2f(r) : -INFINITY) - m_new;
      const float2 c1_2 = make_float2(c1, c1), b2 = make_float2(bias, bias);
      float2 rs2 = make_float2(0.0f, 0.0f);
      uint8_t* sP = sm + L::kP + s * kTile * kTile;
      // two instances: full tiles carry no masking selects
      auto p_codes = [&](auto full_tile) {
#pragma unroll
        for (int c = 0; c < kCols; c += 16) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int cc = c + 4 * e;
            const float2 x01 = __ffma2_rn(make_float2(v[cc], v[cc + 1]), c1_2, b2);
            const float2 x23 = __ffma2_rn(make_float2(v[cc + 2], v[cc + 3]), c1_2, b2);
            float2 q01 = make_float2(ex2(x01.x), ex2(x01.y)), q23 = make_float2(ex2(x23.x), ex2(x23.y));
            if (!decltype(full_tile)::value) {
              q01.x = cc < jlim ? q01.x : 0.0f;
              q01.y = cc + 1 < jlim ? q01.y : 0.0f;
              q23.x = cc + 2 < jlim ? q23.x : 0.0f;
              q23.y = cc + 3 < jlim ? q23.y : 0.0f;
            }
            rs2 = __fadd2_rn(rs2, __fadd2_rn(q01, q23));
            w4[e] = pack4_e4m3(q01.x, q01.y, q23.x, q23.y);
          }
          *reinterpret_cast<uint4*>(sP + SwTile<128>::chunk_offset(row, (wg * kCols + c) / 16)) =
              make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      };
      if (full)
        p_codes(std::true_type{});
      else
        p_codes(std::false_type{});
      l = alpha * l + (rs2.x + rs2.y) * sp;
      m = m_new;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.pfull[s]);

      // O update for the previous tile, while the tensor core works on this one
      if (t >= 1) update_o(t - 1, alpha_prev, c_prev);
      alpha_prev = alpha;
      c_prev = sp * sv;
    }
    update_o(nkv - 1, alpha_prev, c_prev);

    // row sum over the quarters, LSE, and O / l
    s_l[wg][row] = l;
    named_bar_sync(1, kCT);
    float lt = s_l[0][row];
#pragma unroll
    for (int g = 1; g < kGroups; ++g) lt += s_l[g][row];
    if (wg == 0 && row_valid) lse[(size_t)bh * a.N + qi] = m * kLn2 + logf(lt);
    const float linv = unit / lt;
    if (row_valid) {
      if (OUT_BF16) {
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(O) + ((size_t)bh * a.N + qi) * D + wg * DH;
#pragma unroll
        for (int k = 0; k < DH; k += 8) {
          uint4 w;
          uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 x = acc[k / 2 + e];
            __nv_bfloat162 h2 = __floats2bfloat162_rn(x.x * linv, x.y * linv);
            wp[e] = *reinterpret_cast<uint32_t*>(&h2);
          }
          *reinterpret_cast<uint4*>(o + k) = w;
        }
      } else {
        float* o = reinterpret_cast<float*>(O) + ((size_t)bh * a.N + qi) * D + wg * DH;
#pragma unroll
        for (int k = 0; k < DH; k += 4)
          *reinterpret_cast<float4*>(o + k) = make_float4(acc[k / 2].x * linv, acc[k / 2].y * linv,
                                                          acc[k / 2 + 1].x * linv, acc[k / 2 + 1].y * linv);
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
  constexpr int smem = FwdLayout<D>::kBytes;
  static_assert(smem <= 232448, "forward shared memory exceeds the per-block limit");
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
