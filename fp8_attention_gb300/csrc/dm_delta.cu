// Matched softmax row correction ("Delta-Matching for reliable FP8 attention
// training", section 03): delta_i = sum_j P_ij * dP^_ij / sum_j P_ij with
// P = exp(S - LSE) the FP32 softmax before quantisation and dP^ = dO^ V^T the
// FP32 result of the FP8 matmul.  Section 03 cancels the row sum of dS by
// using that each row of P sums to one; with P held in FP32 (and LSE stored
// in FP32) that sum is 1 + eta, and dividing by it makes the cancellation
// hold for the P the backward actually uses (identical to the undivided form
// when P sums to 1).  This is the separate correction pass: one CTA per
// (batch, query head, 128-row query tile), recomputing S = Q K^T and dP^ = dO^ V^T
// on tcgen05 tile by tile.
//
// Warp roles (640 threads):
//   warp 0      TMA: Q and dO tiles once, K/V tiles double-buffered
//   warps 1, 3  MMA issuers: S(t) into TMEM S[t%2] (warp 1), dP(t) into TMEM dP[t%2] (warp 3)
//   warp 2      idle (each warpgroup starts at a multiple of four warps)
//   warps 4-19  four warpgroups, one thread per (query row, quarter of the
//               key columns): P = exp2(S*c1 - LSE*log2e), sums of P*dP
//               (scaled by s_dO * s_V,t per key tile) and of P.  Sixteen
//               compute warps (four per SM sub-partition) hide the TMEM load
//               latency of each other.
// TMEM columns: S[0] 0, S[1] 128, dP[0] 256, dP[1] 384.
#include <cudaTypedefs.h>

#include <type_traits>

#include "dm_device.cuh"
#include "dm_internal.h"

namespace dm {
namespace {

constexpr int kGroups = 4;            // compute warpgroups
constexpr int kThreads = 128 + 128 * kGroups;  // warps 0-3: TMA, S issuer, idle, dP issuer; then compute
constexpr int kCols = kTile / kGroups;  // key columns per thread
constexpr float kLog2e = 1.4426950408889634f;
// K/V shared-memory stages: loads run up to kKV - 1 tiles ahead of the
// products, which covers the L2 latency of a tile load.
constexpr int kKV = 2;

template <int D>
struct DeltaLayout {
  static constexpr int kTileBytes = kTile * D;
  static constexpr int kQ = 0;
  static constexpr int kDO = kQ + kTileBytes;
  static constexpr int kK = kDO + kTileBytes;      // 2 stages
  static constexpr int kV = kK + kKV * kTileBytes;  // kKV stages
  static constexpr int kBytes = kV + kKV * kTileBytes;
  static constexpr int kDynSmem = kBytes + 1024;
};

struct DeltaBars {
  uint64_t q, kfull[kKV], kempty[kKV], vfull[kKV], vempty[kKV], sfull[2], dpfull[2], tempty[2], mma_done, mma_done2;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_delta_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                      const AttnArgs a, const float* __restrict__ lse, float* __restrict__ delta) {
  using L = DeltaLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ DeltaBars bars;
  __shared__ float s_part[kGroups][kTile], s_psum[kGroups][kTile];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = a.B * a.Hq;
  const int qt = a.T - 1 - (int)(blockIdx.x / BH);
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / a.Hq, h = bh % a.Hq;
  const int bg = b * a.Hkv + h / (a.Hq / a.Hkv);
  const int q0 = qt * kTile;
  const int nkv = a.causal ? qt + 1 : a.T;

  Watchdog wd{&s_abort, a.status, a.wait_limit_ns};
  if (tid == 0) {
    s_abort = 0;
    mbar_init(&bars.q, 1);
    for (int s = 0; s < kKV; ++s) {
      mbar_init(&bars.kfull[s], 1);
      mbar_init(&bars.kempty[s], 1);
      mbar_init(&bars.vfull[s], 1);
      mbar_init(&bars.vempty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.sfull[s], 1);
      mbar_init(&bars.dpfull[s], 1);
      mbar_init(&bars.tempty[s], 4 * kGroups);
    }
    mbar_init(&bars.mma_done, 1);
    mbar_init(&bars.mma_done2, 1);
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
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      mbar_arrive_expect_tx(&bars.q, 2 * L::kTileBytes);
      tma_load_3d(sm + L::kQ, &tmQ, &bars.q, 0, q0, bh);
      tma_load_3d(sm + L::kDO, &tmDO, &bars.q, 0, q0, bh);
      int issued = 0;
      for (int t = 0; t < nkv; ++t) {
        const int s = t % kKV;
        const uint32_t ph = (t / kKV) & 1;
        if (!wait(&bars.kempty[s], ph ^ 1, wd, 201)) break;
        if (!wait(&bars.vempty[s], ph ^ 1, wd, 202)) break;
        mbar_arrive_expect_tx(&bars.kfull[s], L::kTileBytes);
        tma_load_3d(sm + L::kK + s * L::kTileBytes, &tmK, &bars.kfull[s], 0, t * kTile, bg);
        mbar_arrive_expect_tx(&bars.vfull[s], L::kTileBytes);
        tma_load_3d(sm + L::kV + s * L::kTileBytes, &tmV, &bars.vfull[s], 0, t * kTile, bg);
        issued = t + 1;
      }
      wait_drain(&bars.q, 0, wd, 209);
      for (int t = max(0, issued - kKV); t < issued; ++t) {
        wait_drain(&bars.kfull[t % kKV], (t / kKV) & 1, wd, 210);
        wait_drain(&bars.vfull[t % kKV], (t / kKV) & 1, wd, 211);
      }
    }
  } else if (warp == 1 || warp == 3) {
    // Two MMA issuers: warp 1 issues S = Q K^T, warp 3 dP = dO^ V^T.  A
    // thread that issues tcgen05.mma stalls on its own mbarrier operations;
    // with two issuers one keeps the tensor pipe fed while the other waits.
    if (lane == 0) {
      const bool is_s = warp == 1;
      const uint32_t idesc = is_s ? idesc_f8(0, 0, 0, 0, kTile, kTile)   // Q K^T
                                  : idesc_f8(1, 0, 0, 0, kTile, kTile);  // dO^ (E5M2) V^T (E4M3)
      uint64_t* full = is_s ? bars.sfull : bars.dpfull;
      uint64_t* operand_full = is_s ? bars.kfull : bars.vfull;
      uint64_t* operand_empty = is_s ? bars.kempty : bars.vempty;
      const uint32_t dcol = is_s ? 0u : 256u;
      bool ok = wait(&bars.q, 0, wd, 203);
      tc_fence_after();
      const uint32_t sA = smem_u32(sm + (is_s ? L::kQ : L::kDO));
      const uint32_t sB0 = smem_u32(sm + (is_s ? L::kK : L::kV));
      for (int t = 0; t < nkv && ok; ++t) {
        const int s = t & 1;  // TMEM buffers
        const uint32_t ph = (t >> 1) & 1;
        const int ks = t % kKV;  // K/V stage
        const uint32_t kph = (t / kKV) & 1;
        ok = wait(&bars.tempty[s], ph ^ 1, wd, 204) && wait(&operand_full[ks], kph, wd, is_s ? 205 : 206);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sB = sB0 + ks * L::kTileBytes;
#pragma unroll
        for (int k = 0; k < D / 32; ++k)
          mma_f8(tmem + dcol + s * 128, SwTile<D>::kmajor(sA, k), SwTile<D>::kmajor(sB, k), idesc, k > 0);
        mma_commit(&full[s]);
        mma_commit(&operand_empty[ks]);
      }
      uint64_t* done = is_s ? &bars.mma_done : &bars.mma_done2;
      mma_commit(done);
      wait_drain(done, 0, wd, is_s ? 212 : 213);
    }
  } else if (warp >= 4) {
    const int wg = (warp - 4) >> 2;  // key-column quarter
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int qi = q0 + row;
    const bool row_valid = qi < a.N;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16) + wg * kCols;
    const float sq = a.q_scales[bh * a.T + qt];
    const float sdo = a.do_scales[bh * a.T + qt];
    const float lse2 = row_valid ? lse[(size_t)bh * a.N + qi] * kLog2e : 0.0f;
    const float* ksc = a.k_scales + (size_t)bg * a.T;
    const float* vsc = a.v_scales + (size_t)bg * a.T;
    float sk_next = ksc[0], sv_next = vsc[0];  // per-tile scales, loaded one tile ahead
    float dl = 0.0f, psum = 0.0f;
    for (int t = 0; t < nkv; ++t) {
      const int s = t & 1;
      const uint32_t ph = (t >> 1) & 1;
      const float c1 = a.sigma * sq * sk_next * kLog2e;
      const float c2 = sdo * sv_next;
      if (t + 1 < nkv) {
        sk_next = ksc[t + 1];
        sv_next = vsc[t + 1];
      }
      const int j0 = t * kTile + wg * kCols;
      int jlim = min(kCols, a.N - j0);
      if (a.causal) jlim = min(jlim, qi - j0 + 1);
      float x[2 * kCols];  // S then dP of this thread's columns
      const float* sv = x;
      const float* dp = x + kCols;
      wait(&bars.sfull[s], ph, wd, 207);
      wait(&bars.dpfull[s], ph, wd, 208);
      tc_fence_after();
      tmem_load64(tl + s * 128, tl + 256 + s * 128, x);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.tempty[s]);
      // P = exp2(S c1 - LSE log2e) on packed pairs; masks only on the
      // diagonal or ragged tile (a separate instance without selects)
      const float2 c1_2 = make_float2(c1, c1), nl2 = make_float2(-lse2, -lse2);
      float2 acc0 = make_float2(0.0f, 0.0f), acc1 = acc0, ps0 = acc0, ps1 = acc0;
      auto accumulate = [&](auto full_tile) {
#pragma unroll
        for (int c = 0; c < kCols; c += 4) {
          const float2 x0 = __ffma2_rn(make_float2(sv[c], sv[c + 1]), c1_2, nl2);
          const float2 x1 = __ffma2_rn(make_float2(sv[c + 2], sv[c + 3]), c1_2, nl2);
          float2 p0 = make_float2(ex2(x0.x), ex2(x0.y)), p1 = make_float2(ex2(x1.x), ex2(x1.y));
          if (!decltype(full_tile)::value) {
            p0.x = c < jlim ? p0.x : 0.0f;
            p0.y = c + 1 < jlim ? p0.y : 0.0f;
            p1.x = c + 2 < jlim ? p1.x : 0.0f;
            p1.y = c + 3 < jlim ? p1.y : 0.0f;
          }
          acc0 = __ffma2_rn(p0, make_float2(dp[c], dp[c + 1]), acc0);
          acc1 = __ffma2_rn(p1, make_float2(dp[c + 2], dp[c + 3]), acc1);
          ps0 = __fadd2_rn(ps0, p0);
          ps1 = __fadd2_rn(ps1, p1);
        }
      };
      if (jlim >= kCols)
        accumulate(std::true_type{});
      else
        accumulate(std::false_type{});
      dl = fmaf((acc0.x + acc0.y) + (acc1.x + acc1.y), c2, dl);
      psum += (ps0.x + ps0.y) + (ps1.x + ps1.y);
    }
    s_part[wg][row] = dl;
    s_psum[wg][row] = psum;
    named_bar_sync(1, 4 * kGroups * 32);
    if (wg == 0 && row_valid) {
      float num = 0.0f, den = 0.0f;
#pragma unroll
      for (int g = 0; g < kGroups; ++g) {
        num += s_part[g][row];
        den += s_psum[g][row];
      }
      delta[(size_t)bh * a.N + qi] = num / den;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_t(const DeltaLaunch& f, cudaStream_t st) {
  auto k = attn_delta_kernel<D>;
  constexpr int smem = DeltaLayout<D>::kDynSmem;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(f.args.B * f.args.Hq * f.args.T);
  k<<<grid, kThreads, smem, st>>>(f.tmQ, f.tmK, f.tmV, f.tmDO, f.args, f.lse, f.delta);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_delta_matched(const DeltaLaunch& f, int d, cudaStream_t st) {
  return d == 128 ? launch_t<128>(f, st) : launch_t<64>(f, st);
}

}  // namespace dm
