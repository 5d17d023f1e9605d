// Matched softmax row correction ("Delta-Matching for reliable FP8 attention
// training", section 03): delta_i = sum_j P_ij * dP^_ij / sum_j P_ij with
// P = exp(S - LSE) the FP32 softmax before quantisation and dP^ = dO^ V^T the
// FP32 result of the FP8 matmul.  Section 03 cancels the row sum of dS by
// using that each row of P sums to one; with P held in FP32 (and LSE stored
// in FP32) that sum is 1 + eta, and dividing by it makes the cancellation
// hold for the P the backward actually uses (identical to the undivided form
// when P sums to 1).  This is the separate correction pass: one CTA per
// (batch, query head, 128-row query tile), recomputing S = Q K^T and
// dP^ = dO^ V^T on tcgen05 tile by tile.  Over a key block (context
// parallelism) the two sums can be written apart (den != NULL), so that the
// blocks' sums add up before the one division.
//
// For d = 64 and 128 two CTAs share an SM (192 threads, 256 TMEM columns,
// ~97 KB of shared memory each): one CTA's reductions overlap the other's
// products, and each SM has two MMA issuers.  For d = 256 (192 KB of tiles)
// one CTA holds the SM and double-buffers S and dP in TMEM instead, so that
// the products of tile t+1 run while the warpgroup reduces tile t.
//
// Warp roles (192 threads):
//   warps 0-3   one warpgroup, thread = query row (TMEM lane), all key
//               columns in 32-column chunks: P = exp2(S*c1 - LSE*log2e),
//               sums of P*dP (scaled by s_dO * s_V,t per key tile) and of P
//   warp 4      TMA: Q and dO tiles once, K/V tiles double-buffered; when
//               the backward computes delta itself, the clearing of its
//               outputs (dQ, dK, dV, diagnostics) after the last loads
//   warp 5      MMA issuer (+ TMEM owner): S(t) and dP(t)
// TMEM columns: S 0-127, dP 128-255 (d = 256: a second pair at 256-511 for
// odd key tiles).
#include <cudaTypedefs.h>

#include <type_traits>

#include "dm_device.cuh"
#include "dm_pdl.cuh"
#include "dm_internal.h"

namespace dm {
namespace {

constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kKV = 2;  // K/V shared-memory stages
constexpr uint32_t kColS = 0, kColDP = 128;

template <int D>
struct DeltaCfg {
  static constexpr int kTBuf = D > 128 ? 2 : 1;  // (S, dP) buffer pairs in TMEM
  static constexpr uint32_t kTmemCols = 256u * kTBuf;
  static constexpr int kCTAsPerSM = D > 128 ? 1 : 2;
};

template <int D, int DV>
struct DeltaLayout {
  static constexpr int kTileBytes = kTile * D;   // Q, K (OpTile<D>)
  static constexpr int kVBytes = kTile * DV;     // dO, V (OpTile<DV>)
  static constexpr int kQ = 0;
  static constexpr int kDO = kQ + kTileBytes;
  static constexpr int kK = kDO + kVBytes;          // kKV stages
  static constexpr int kV = kK + kKV * kTileBytes;  // kKV stages
  static constexpr int kBars = kV + kKV * kVBytes;
  static constexpr int kMisc = kBars + 256;  // tmem address, abort flag
  static constexpr int kBytes = kMisc + 16;
};

struct DeltaBars {
  uint64_t q, kfull[kKV], kempty[kKV], vfull[kKV], vempty[kKV], tfull[2], tempty[2], mma_done;
};
static_assert(sizeof(DeltaBars) <= 256, "delta barriers");

// D: head dimension of Q and K; DV: of dO and V (DV <= D).
template <int D, int DV>
__global__ void __launch_bounds__(kThreads, DeltaCfg<D>::kCTAsPerSM)
    attn_delta_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                      const AttnArgs a, const float* __restrict__ lse, float* __restrict__ delta,
                      float* __restrict__ den, const DeltaClear clr) {
  using L = DeltaLayout<D, DV>;
  using C = DeltaCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  DeltaBars& bars = *reinterpret_cast<DeltaBars*>(sm + L::kBars);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  int* s_abort = reinterpret_cast<int*>(sm + L::kMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = a.B * a.Hq;
  const int qt = a.T - 1 - (int)(blockIdx.x / BH);
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / a.Hq, h = bh % a.Hq;
  const int bg = b * a.Hkv + h / (a.Hq / a.Hkv);
  const int q0 = qt * kTile;
  // key tiles of the block this query tile sees (0: none)
  const int nkv = a.causal ? max(0, min(qt + 1 - a.kt_off, a.Tk)) : a.Tk;

  // the swizzled tiles need a 1024-byte aligned window (no static shared
  // variables); the status word is written only after the wait for the
  // previous kernel, like every other global access of this kernel
  if (smem_u32(smem_raw) & 1023u) {
    grid_dependency_sync();
    if (tid == 0) atomicCAS(a.status, 0u, (unsigned)DM_ERR_UNSUPPORTED);
    return;
  }
  Watchdog wd{s_abort, a.status, a.wait_limit_ns};
  if (tid == 0) {
    *s_abort = 0;
    mbar_init(&bars.q, 1);
    for (int s = 0; s < kKV; ++s) {
      mbar_init(&bars.kfull[s], 1);
      mbar_init(&bars.kempty[s], 1);
      mbar_init(&bars.vfull[s], 1);
      mbar_init(&bars.vempty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.tfull[s], 1);
      mbar_init(&bars.tempty[s], 4);
    }
    mbar_init(&bars.mma_done, 1);
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(s_tmem, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dependency_sync();  // barriers and TMEM are set up; inputs of earlier kernels from here on
  const uint32_t tmem = *s_tmem;

  if (warp == 4) {
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      mbar_arrive_expect_tx(&bars.q, L::kTileBytes + L::kVBytes);
      tma_load_tile<D>(sm + L::kQ, &tmQ, &bars.q, q0, bh);
      tma_load_tile<DV>(sm + L::kDO, &tmDO, &bars.q, q0, bh);
      int issued = 0;
      for (int t = 0; t < nkv; ++t) {
        const int s = t % kKV;
        const uint32_t ph = (t / kKV) & 1;
        if (!wait(&bars.kempty[s], ph ^ 1, wd, 201)) break;
        if (!wait(&bars.vempty[s], ph ^ 1, wd, 202)) break;
        mbar_arrive_expect_tx(&bars.kfull[s], L::kTileBytes);
        tma_load_tile<D>(sm + L::kK + s * L::kTileBytes, &tmK, &bars.kfull[s], t * kTile, bg);
        mbar_arrive_expect_tx(&bars.vfull[s], L::kVBytes);
        tma_load_tile<DV>(sm + L::kV + s * L::kVBytes, &tmV, &bars.vfull[s], t * kTile, bg);
        issued = t + 1;
      }
      wait_drain(&bars.q, 0, wd, 209);
      for (int t = max(0, issued - kKV); t < issued; ++t) {
        wait_drain(&bars.kfull[t % kKV], (t / kKV) & 1, wd, 210);
        wait_drain(&bars.vfull[t % kKV], (t / kKV) & 1, wd, 211);
      }
    }
    __syncwarp();
    if (clr.dQ) {
      // the backward's outputs of this query tile (and, in a group's first
      // query head, of the key tile with its index) start at zero: 16-byte
      // stores of whole rows (d and d_v are multiples of 64), the
      // diagnostics rows one float at a time
      const int rows = min(kTile, a.N - q0);
      auto clear = [&](float* base, size_t first, size_t n) {
        float4* p4 = reinterpret_cast<float4*>(base + first);
        for (size_t i = lane; i < n / 4; i += 32) p4[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      };
      clear(clr.dQ, ((size_t)bh * a.N + q0) * a.dqk, (size_t)rows * a.dqk);
      if (h % (a.Hq / a.Hkv) == 0) {
        clear(clr.dK, ((size_t)bg * a.N + q0) * a.dqk, (size_t)rows * a.dqk);
        clear(clr.dV, ((size_t)bg * a.N + q0) * a.dv, (size_t)rows * a.dv);
      }
      for (int j = 0; j < 4; ++j)
        if (clr.rows[j])
          for (int i = lane; i < rows; i += 32) clr.rows[j][(size_t)bh * a.N + q0 + i] = 0.0f;
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f8(0, 0, 0, 0, kTile, kTile);   // Q K^T
      constexpr uint32_t kIdDP = idesc_f8(1, 0, 0, 0, kTile, kTile);  // dO^ (E5M2) V^T (E4M3)
      bool ok = wait(&bars.q, 0, wd, 203);
      tc_fence_after();
      const uint32_t sQ = smem_u32(sm + L::kQ), sDO = smem_u32(sm + L::kDO);
      for (int t = 0; t < nkv && ok; ++t) {
        const int ks = t % kKV, tb = t % C::kTBuf;
        const uint32_t kph = (t / kKV) & 1;
        // S(t) and dP(t) once K(t), V(t) have landed and the tile that last
        // used the TMEM pair, t - kTBuf, has been read
        ok = (t < C::kTBuf || wait(&bars.tempty[tb], ((t / C::kTBuf) & 1) ^ 1, wd, 204)) &&
             wait(&bars.kfull[ks], kph, wd, 205) && wait(&bars.vfull[ks], kph, wd, 206);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sK = smem_u32(sm + L::kK + ks * L::kTileBytes);
        const uint32_t sV = smem_u32(sm + L::kV + ks * L::kVBytes);
        const uint32_t tpair = tmem + 256u * tb;
#pragma unroll
        for (int k = 0; k < D / 32; ++k)
          mma_f8(tpair + kColS, OpTile<D>::kmajor(sQ, k), OpTile<D>::kmajor(sK, k), kIdS, k > 0);
#pragma unroll
        for (int k = 0; k < DV / 32; ++k)
          mma_f8(tpair + kColDP, OpTile<DV>::kmajor(sDO, k), OpTile<DV>::kmajor(sV, k), kIdDP, k > 0);
        mma_commit(&bars.tfull[tb]);
        mma_commit(&bars.kempty[ks]);
        mma_commit(&bars.vempty[ks]);
      }
      mma_commit(&bars.mma_done);
      wait_drain(&bars.mma_done, 0, wd, 212);
    }
  } else if (warp < 4) {
    const int row = warp * 32 + lane;
    const int qi = q0 + row;
    const bool row_valid = qi < a.N;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    const float sq = a.q_scales[bh * a.T + qt];
    const float sdo = a.do_scales[bh * a.T + qt];
    const float lse2 = row_valid ? lse[(size_t)bh * a.N + qi] * kLog2e : 0.0f;
    const float* ksc = a.k_scales + (size_t)bg * a.Tk;
    const float* vsc = a.v_scales + (size_t)bg * a.Tk;
    float sk_next = ksc[0], sv_next = vsc[0];  // per-tile scales, loaded one tile ahead
    float dl = 0.0f, psum = 0.0f;
    for (int t = 0; t < nkv; ++t) {
      const float c1 = a.sigma * sq * sk_next * kLog2e;
      const float c2 = sdo * sv_next;
      if (t + 1 < nkv) {
        sk_next = ksc[t + 1];
        sv_next = vsc[t + 1];
      }
      const int j0 = t * kTile;
      int jlim = min(kTile, a.Nk - j0);
      if (a.causal) jlim = min(jlim, qi - (j0 + a.kt_off * kTile) + 1);
      // warp-uniform: the TMEM loads below are warp-collective
      const bool full = __all_sync(0xffffffffu, jlim >= kTile);
      const int tb = t % C::kTBuf;
      const uint32_t tp = tl + 256u * tb;  // this tile's S, dP pair
      wait(&bars.tfull[tb], (t / C::kTBuf) & 1, wd, 207);
      tc_fence_after();
      // P = exp2(S c1 - LSE log2e) on packed pairs, 32 columns at a time;
      // masks only on the diagonal or ragged tile
      const float2 c1_2 = make_float2(c1, c1), nl2 = make_float2(-lse2, -lse2);
      float2 acc0 = make_float2(0.0f, 0.0f), acc1 = acc0, ps0 = acc0, ps1 = acc0;
      // two halves of 64 columns: S and dP of a half in registers at once;
      // TMEM is released as soon as the second half is loaded
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float x[128];  // S of 64 columns, then dP of the same columns
        tmem_load128(tp + kColS + 64 * hh, tp + kColS + 64 * hh + 32, tp + kColDP + 64 * hh,
                     tp + kColDP + 64 * hh + 32, x);
        if (hh == 1) {
          // S and dP of tile t have been read: the tensor core may write the pair again
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.tempty[tb]);
        }
        auto accumulate = [&](auto full_tile) {
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            const int col = 64 * hh + c;
            const float2 x0 = __ffma2_rn(make_float2(x[c], x[c + 1]), c1_2, nl2);
            const float2 x1 = __ffma2_rn(make_float2(x[c + 2], x[c + 3]), c1_2, nl2);
            float2 p0 = make_float2(ex2(x0.x), ex2(x0.y)), p1 = make_float2(ex2(x1.x), ex2(x1.y));
            if (!decltype(full_tile)::value) {
              p0.x = col < jlim ? p0.x : 0.0f;
              p0.y = col + 1 < jlim ? p0.y : 0.0f;
              p1.x = col + 2 < jlim ? p1.x : 0.0f;
              p1.y = col + 3 < jlim ? p1.y : 0.0f;
            }
            acc0 = __ffma2_rn(p0, make_float2(x[64 + c], x[64 + c + 1]), acc0);
            acc1 = __ffma2_rn(p1, make_float2(x[64 + c + 2], x[64 + c + 3]), acc1);
            ps0 = __fadd2_rn(ps0, p0);
            ps1 = __fadd2_rn(ps1, p1);
          }
        };
        if (full)
          accumulate(std::true_type{});
        else
          accumulate(std::false_type{});
      }
      dl = fmaf((acc0.x + acc0.y) + (acc1.x + acc1.y), c2, dl);
      psum += (ps0.x + ps0.y) + (ps1.x + ps1.y);
    }
    if (row_valid) {
      const size_t o = (size_t)bh * a.N + qi;
      if (den) {  // the block's two sums, apart
        delta[o] = dl;
        den[o] = psum;
      } else {
        delta[o] = psum > 0.0f ? dl / psum : 0.0f;  // 0 for a row that sees no key of the block
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int DV>
cudaError_t launch_t(const DeltaLaunch& f, cudaStream_t st) {
  auto k = attn_delta_kernel<D, DV>;
  constexpr int smem = DeltaLayout<D, DV>::kBytes;
  static_assert(DeltaCfg<D>::kCTAsPerSM * (smem + 1024) <= 233472, "the delta CTAs must fit in one SM's shared memory");
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(f.args.B * f.args.Hq * f.args.T);
  return launch_overlapped(k, grid, kThreads, smem, st, f.tmQ, f.tmK, f.tmV, f.tmDO, f.args, f.lse, f.delta,
                           f.den, f.clear);
}

}  // namespace

cudaError_t launch_delta_matched(const DeltaLaunch& f, int d, int dv, cudaStream_t st) {
  if (d == 256) return dv == 128 ? launch_t<256, 128>(f, st) : launch_t<256, 256>(f, st);
  return d == 128 ? launch_t<128, 128>(f, st) : launch_t<64, 64>(f, st);
}

}  // namespace dm
