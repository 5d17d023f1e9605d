// Backward: dQ, dK, dV with the five backward matmuls on tcgen05 FP8 MMAs
// ("Delta-Matching for reliable FP8 attention training", section 01, "Write
// down softmax backward", and section 03 for delta).  One CTA per (batch, kv
// head, 128-row key tile); it loops over the query heads of the kv head's
// group and over the query tiles that see the key tile, so dK and dV are
// summed over the group inside the CTA.  Computed transposed (key rows on
// TMEM lanes) so that dV and dK accumulate in TMEM:
//   S^T  = K Q^T           (MMA, TMEM cols 0..127)
//   dP^T = V dO^T          (MMA, TMEM cols 128..255)
//   P    = exp(S - LSE) in FP32, P^ = E4M3 per 128x128 tile
//   dS   = P (dP - delta) in FP32, dS^ = E5M2 per 128x128 tile
//   dV  += P^T dO          (MMA, TMEM cols 256..)
//   dK  += dS^T Q          (MMA, TMEM cols 384..)
//   dQ_i = dS^ K           (MMA into cols 128.., staged in shared memory and
//                           added into global dQ with a TMA bulk reduce-add)
// dV and dK accumulate in TMEM in units of the current iteration's scale
// product (s_P * s_dO, resp. sigma * s_dS * s_Q): before each accumulation the
// compute warps rescale the accumulator by old/new unit.  Iterations whose
// product is below 2^-100 (a flushed or negligible tile) add nothing.
//
// Warp roles (320 threads): warp 0 TMA, warp 1 MMA, warps 2-9 two compute
// warpgroups; thread = key row, warpgroup = half of the query columns (and
// half of the d columns for the dV/dK/dQ epilogues).
#include <cudaTypedefs.h>

#include "dm_device.cuh"
#include "dm_internal.h"

namespace dm {
namespace {

constexpr int kThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMinUnit = 0x1p-100f;

template <int D>
struct BwdLayout {
  static constexpr int kTileBytes = kTile * D;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;        // 2 stages
  static constexpr int kDO = kQ + 2 * kTileBytes;   // 2 stages
  static constexpr int kPt = kDO + 2 * kTileBytes;  // P^T codes, [key row][128 query bytes]
  static constexpr int kDSt = kPt + kTile * kTile;  // dS^T codes
  static constexpr int kDQ = kDSt + kTile * kTile;   // dQ tile staging: D/32 boxes of [128 rows][32 fp32]
  static constexpr int kBytes = kDQ + kTile * D * 4;
  static constexpr int kDynSmem = kBytes + 1024;
};

struct BwdBars {
  uint64_t kv, qfull[2], qempty[2], sfull, dpfull, pds, mma2, dqempty, mma_done;
};

// Column sums over the 32 lanes of a warp: on return lane l holds the sum over
// all lanes of their v[l] (recursive halving, 31 shuffles).
__device__ __forceinline__ float lane_column_sum(float (&v)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = upper ? v[i] : v[i + s];
      const float keep = upper ? v[i + s] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  return v[0];
}

// Rescale `ncols` (multiple of 32) TMEM columns of this warp's lanes by f.
__device__ __forceinline__ void tmem_scale(uint32_t taddr, int ncols, float f) {
  for (int c = 0; c < ncols; c += 32) {
    float v[32];
    tmem_ld32(taddr + c, v);
    tmem_wait_ld();
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] *= f;
    tmem_st32(taddr + c, v);
  }
  tmem_wait_st();
}

// Unit bookkeeping for one TMEM accumulator; every compute thread holds an
// identical copy.  Returns the MMA mode: 0 skip, 1 overwrite, 2 accumulate.
__device__ __forceinline__ int next_unit(float& unit, float c, uint32_t taddr, int ncols) {
  if (!(c >= kMinUnit)) return 0;
  if (unit == 0.0f) {
    unit = c;
    return 1;
  }
  if (unit != c) tmem_scale(taddr, ncols, unit / c);
  unit = c;
  return 2;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmDQ, const AttnArgs a, const float* __restrict__ lse,
                    const float* __restrict__ delta, float* __restrict__ dK, float* __restrict__ dV,
                    const dm_diag diag) {
  using L = BwdLayout<D>;
  constexpr int DH = D / 2;  // d columns per compute warpgroup
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ BwdBars bars;
  __shared__ float s_lse[2][kTile], s_dl[2][kTile];
  __shared__ float s_red[2][2][8];
  __shared__ int s_mode[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BG = a.B * a.Hkv;
  const int kt = (int)(blockIdx.x / BG);  // key tile 0 sees the most query tiles: first
  const int bg = (int)(blockIdx.x % BG);
  const int b = bg / a.Hkv, g = bg % a.Hkv;
  const int G = a.Hq / a.Hkv;
  const int qt0 = a.causal ? kt : 0;
  const int nq = a.T - qt0;
  const int n_iter = G * nq;
  const bool want_diag = diag.rowsum_pre || diag.abssum_pre || diag.rowsum_post || diag.abssum_post;

  Watchdog wd{&s_abort, a.status, a.wait_limit_ns};
  if (tid == 0) {
    s_abort = 0;
    mbar_init(&bars.kv, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.qfull[s], 1);
      mbar_init(&bars.qempty[s], 1);
    }
    mbar_init(&bars.sfull, 1);
    mbar_init(&bars.dpfull, 1);
    mbar_init(&bars.pds, 8);
    mbar_init(&bars.mma2, 1);
    mbar_init(&bars.dqempty, 8);
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
      tma_prefetch_desc(&tmDO);
      mbar_arrive_expect_tx(&bars.kv, 2 * L::kTileBytes);
      tma_load_3d(sm + L::kK, &tmK, &bars.kv, 0, kt * kTile, bg);
      tma_load_3d(sm + L::kV, &tmV, &bars.kv, 0, kt * kTile, bg);
      int issued = 0;
      for (int n = 0; n < n_iter; ++n) {
        const int s = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        const int bh = b * a.Hq + g * G + n / nq;
        const int qt = qt0 + n % nq;
        if (!wait(&bars.qempty[s], ph ^ 1, wd, 301)) break;
        mbar_arrive_expect_tx(&bars.qfull[s], 2 * L::kTileBytes);
        tma_load_3d(sm + L::kQ + s * L::kTileBytes, &tmQ, &bars.qfull[s], 0, qt * kTile, bh);
        tma_load_3d(sm + L::kDO + s * L::kTileBytes, &tmDO, &bars.qfull[s], 0, qt * kTile, bh);
        issued = n + 1;
      }
      wait_drain(&bars.kv, 0, wd, 309);
      for (int n = max(0, issued - 2); n < issued; ++n)
        wait_drain(&bars.qfull[n & 1], (n >> 1) & 1, wd, 310);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f8(0, 0, 0, 0, kTile, kTile);   // K Q^T
      constexpr uint32_t kIdDP = idesc_f8(0, 1, 0, 0, kTile, kTile);  // V (E4M3) dO^T (E5M2)
      constexpr uint32_t kIdDV = idesc_f8(0, 1, 0, 1, kTile, D);      // P^T (K-major) dO (MN-major)
      constexpr uint32_t kIdDK = idesc_f8(1, 0, 0, 1, kTile, D);      // dS^T (K-major) Q (MN-major)
      constexpr uint32_t kIdDQ = idesc_f8(1, 0, 1, 1, kTile, D);      // dS (MN-major) K (MN-major)
      const uint32_t sK = smem_u32(sm + L::kK), sV = smem_u32(sm + L::kV);
      const uint32_t sPt = smem_u32(sm + L::kPt), sDSt = smem_u32(sm + L::kDSt);
      bool ok = wait(&bars.kv, 0, wd, 302);
      for (int n = 0; n < n_iter && ok; ++n) {
        const int s = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        const uint32_t sQ = smem_u32(sm + L::kQ + s * L::kTileBytes);
        const uint32_t sDO = smem_u32(sm + L::kDO + s * L::kTileBytes);
        if (!(ok = wait(&bars.qfull[s], ph, wd, 303))) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 32; ++k)
          mma_f8(tmem + 0, SwTile<D>::kmajor(sK, k), SwTile<D>::kmajor(sQ, k), kIdS, k > 0);
        mma_commit(&bars.sfull);
        if (n >= 1 && !(ok = wait(&bars.dqempty, (n - 1) & 1, wd, 304))) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 32; ++k)
          mma_f8(tmem + 128, SwTile<D>::kmajor(sV, k), SwTile<D>::kmajor(sDO, k), kIdDP, k > 0);
        mma_commit(&bars.dpfull);
        if (!(ok = wait(&bars.pds, n & 1, wd, 305))) break;
        tc_fence_after();
        const int mode_dv = s_mode[0], mode_dk = s_mode[1];
        if (mode_dv) {
#pragma unroll
          for (int k = 0; k < kTile / 32; ++k)
            mma_f8(tmem + 256, SwTile<128>::kmajor(sPt, k), SwTile<D>::mnmajor(sDO, k), kIdDV,
                   (k > 0 || mode_dv == 2) ? 1u : 0u);
        }
        if (mode_dk) {
#pragma unroll
          for (int k = 0; k < kTile / 32; ++k)
            mma_f8(tmem + 384, SwTile<128>::kmajor(sDSt, k), SwTile<D>::mnmajor(sQ, k), kIdDK,
                   (k > 0 || mode_dk == 2) ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < kTile / 32; ++k)
          mma_f8(tmem + 128, SwTile<128>::mnmajor(sDSt, k), SwTile<D>::mnmajor(sK, k), kIdDQ, k > 0);
        mma_commit(&bars.mma2);
        mma_commit(&bars.qempty[s]);
      }
      mma_commit(&bars.mma_done);
      wait_drain(&bars.mma_done, 0, wd, 311);
    }
  } else {
    // -------------------------------------------------------------- compute
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // key row within the tile (TMEM lane)
    const int kj = kt * kTile + r;
    const bool kv_valid = kj < a.N;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const int ct = tid - 64;  // 0..255
    const float sk = a.k_scales[bg * a.T + kt];
    const float svv = a.v_scales[bg * a.T + kt];
    float unit_dv = 0.0f, unit_dk = 0.0f;
    // Per-iteration global values are loaded one iteration ahead: this
    // thread's element of the query tile's LSE (threads 0-127; +inf for absent
    // rows) or delta (threads 128-255; 0 for absent rows), and the tile's Q and
    // dO scales.
    auto row_value = [&](int n) -> float {
      const int bh_n = b * a.Hq + g * G + n / nq;
      const int qi = (qt0 + n % nq) * kTile + (ct & 127);
      if (ct < 128) return qi < a.N ? lse[(size_t)bh_n * a.N + qi] : INFINITY;
      return qi < a.N ? delta[(size_t)bh_n * a.N + qi] : 0.0f;
    };
    auto tile_index = [&](int n) { return (b * a.Hq + g * G + n / nq) * a.T + qt0 + n % nq; };
    float pre_row = row_value(0);
    float pre_sq = a.q_scales[tile_index(0)], pre_sdo = a.do_scales[tile_index(0)];

    for (int n = 0; n < n_iter; ++n) {
      const int hh = n / nq, qt = qt0 + n % nq;
      const int bh = b * a.Hq + g * G + hh;
      const int qi0 = qt * kTile;
      const int buf = n & 1;
      if (ct < 128)
        s_lse[buf][ct] = pre_row * kLog2e;
      else
        s_dl[buf][ct - 128] = pre_row;
      const float sq = pre_sq, sdo = pre_sdo;
      if (n + 1 < n_iter) {
        pre_row = row_value(n + 1);
        pre_sq = a.q_scales[tile_index(n + 1)];
        pre_sdo = a.do_scales[tile_index(n + 1)];
      }
      // the previous iteration's dQ reduce has finished reading the staging tile
      if (ct == 0) bulk_wait_read_all();
      named_bar_sync(1, 256);
      const float c1 = a.sigma * sq * sk * kLog2e;
      const float cdp = sdo * svv;
      const int cmin = !kv_valid ? (1 << 30) : (a.causal && qt == kt) ? r - wg * 64 : 0;

      // P = exp(S - LSE), its tile amax and E4M3 codes
      float p[64];
      wait(&bars.sfull, n & 1, wd, 306);
      tc_fence_after();
      tmem_ld32(tl + wg * 64, *reinterpret_cast<float(*)[32]>(&p[0]));
      tmem_ld32(tl + wg * 64 + 32, *reinterpret_cast<float(*)[32]>(&p[32]));
      tmem_wait_ld();
      float pmax = 0.0f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        p[c] = (c >= cmin) ? ex2(fmaf(p[c], c1, -s_lse[buf][wg * 64 + c])) : 0.0f;
        pmax = fmaxf(pmax, p[c]);
      }
      pmax = warp_max(pmax);
      if (lane == 0) s_red[buf][0][warp - 2] = pmax;
      named_bar_sync(1, 256);
      float amax = s_red[buf][0][0];
#pragma unroll
      for (int w = 1; w < 8; ++w) amax = fmaxf(amax, s_red[buf][0][w]);
      float rp;
      const float sp = tile_scale<0>(amax, rp);
      {
        uint8_t* dst = sm + L::kPt;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float* q4 = &p[16 * c + 4 * e];
            w4[e] = pack4_e4m3(__fmul_rn(q4[0], rp), __fmul_rn(q4[1], rp), __fmul_rn(q4[2], rp),
                               __fmul_rn(q4[3], rp));
          }
          *reinterpret_cast<uint4*>(dst + SwTile<128>::chunk_offset(r, wg * 4 + c)) =
              make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
      const int mode_dv = next_unit(unit_dv, sp * sdo, tl + 256 + wg * DH, DH);

      // dS = P (dP - delta), its tile amax and E5M2 codes
      float ds[64];
      wait(&bars.dpfull, n & 1, wd, 307);
      tc_fence_after();
      tmem_ld32(tl + 128 + wg * 64, *reinterpret_cast<float(*)[32]>(&ds[0]));
      tmem_ld32(tl + 128 + wg * 64 + 32, *reinterpret_cast<float(*)[32]>(&ds[32]));
      tmem_wait_ld();
      float dmax = 0.0f;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        ds[c] = p[c] * fmaf(ds[c], cdp, -s_dl[buf][wg * 64 + c]);
        dmax = fmaxf(dmax, fabsf(ds[c]));
      }
      dmax = warp_max(dmax);
      if (lane == 0) s_red[buf][1][warp - 2] = dmax;
      named_bar_sync(1, 256);
      amax = s_red[buf][1][0];
#pragma unroll
      for (int w = 1; w < 8; ++w) amax = fmaxf(amax, s_red[buf][1][w]);
      float rs;
      const float sds = tile_scale<1>(amax, rs);
      uint32_t dcode[16];
      {
        uint8_t* dst = sm + L::kDSt;
#pragma unroll
        for (int c = 0; c < 16; ++c)
          dcode[c] = pack4_e5m2(__fmul_rn(ds[4 * c], rs), __fmul_rn(ds[4 * c + 1], rs), __fmul_rn(ds[4 * c + 2], rs),
                                __fmul_rn(ds[4 * c + 3], rs));
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(dst + SwTile<128>::chunk_offset(r, wg * 4 + c)) =
              make_uint4(dcode[4 * c], dcode[4 * c + 1], dcode[4 * c + 2], dcode[4 * c + 3]);
      }
      const int mode_dk = next_unit(unit_dk, a.sigma * sds * sq, tl + 384 + wg * DH, DH);
      if (ct == 0) {
        s_mode[0] = mode_dv;
        s_mode[1] = mode_dk;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.pds);

      // per-query-row diagnostics (column sums over the key rows)
      if (want_diag) {
        const size_t rowbase = (size_t)bh * a.N + qi0 + wg * 64;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int col = half * 32 + lane;
          const bool col_ok = qi0 + wg * 64 + col < a.N;
          float v[32];
          if (diag.rowsum_pre) {
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = ds[half * 32 + k];
            const float sum = lane_column_sum(v, lane);
            if (col_ok) atomicAdd(diag.rowsum_pre + rowbase + col, sum);
          }
          if (diag.abssum_pre) {
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = fabsf(ds[half * 32 + k]);
            const float sum = lane_column_sum(v, lane);
            if (col_ok) atomicAdd(diag.abssum_pre + rowbase + col, sum);
          }
          if (diag.rowsum_post || diag.abssum_post) {
            float w2[32];
#pragma unroll
            for (int k = 0; k < 32; k += 4) {
              const uint32_t w = dcode[(half * 32 + k) / 4];
              const float2 lo = unpack2<1>((uint16_t)(w & 0xFFFF));
              const float2 hi = unpack2<1>((uint16_t)(w >> 16));
              v[k] = lo.x * sds, v[k + 1] = lo.y * sds, v[k + 2] = hi.x * sds, v[k + 3] = hi.y * sds;
            }
#pragma unroll
            for (int k = 0; k < 32; ++k) w2[k] = fabsf(v[k]);
            if (diag.rowsum_post) {
              const float sum = lane_column_sum(v, lane);
              if (col_ok) atomicAdd(diag.rowsum_post + rowbase + col, sum);
            }
            if (diag.abssum_post) {
              const float sum = lane_column_sum(w2, lane);
              if (col_ok) atomicAdd(diag.abssum_post + rowbase + col, sum);
            }
          }
        }
      }

      // dQ tile (query rows on TMEM lanes): scaled, staged in shared memory with
      // the 128-byte swizzle of the dQ tensor map, then added into global dQ
      // by one bulk reduce per 32-column box.  TMEM loads are warp-collective:
      // every lane loads; rows beyond N are clipped by the tensor map.
      wait(&bars.mma2, n & 1, wd, 312);
      tc_fence_after();
      {
        const float cdq = a.sigma * sds * sk;
        float v[DH];
#pragma unroll
        for (int c = 0; c < DH; c += 32) tmem_ld32(tl + 128 + wg * DH + c, *reinterpret_cast<float(*)[32]>(&v[c]));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.dqempty);
#pragma unroll
        for (int c = 0; c < DH; c += 32) {
          uint8_t* box = sm + L::kDQ + ((wg * DH + c) / 32) * (kTile * 128);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            *reinterpret_cast<float4*>(box + SwTile<128>::chunk_offset(r, e)) =
                make_float4(v[c + 4 * e] * cdq, v[c + 4 * e + 1] * cdq, v[c + 4 * e + 2] * cdq,
                            v[c + 4 * e + 3] * cdq);
        }
        fence_proxy_async_smem();
        named_bar_sync(2, 256);
        if (ct == 0 && cdq != 0.0f) {
#pragma unroll
          for (int bx = 0; bx < D / 32; ++bx)
            tma_reduce_add_3d(&tmDQ, sm + L::kDQ + bx * (kTile * 128), bx * 32, qi0, bh);
          bulk_commit();
        }
      }
    }

    if (ct == 0) bulk_wait_all();

    // epilogue: dV and dK rows of this key tile, in true units (an
    // accumulator that never received a contribution holds garbage: write 0).
    // All lanes load (warp-collective); only the stores are guarded.
#pragma unroll
    for (int c = 0; c < DH; c += 32) {
      float v[32], u[32];
      tmem_ld32(tl + 256 + wg * DH + c, v);
      tmem_ld32(tl + 384 + wg * DH + c, u);
      tmem_wait_ld();
      if (kv_valid) {
        float* dv = dV + ((size_t)bg * a.N + kj) * D + wg * DH + c;
        float* dk = dK + ((size_t)bg * a.N + kj) * D + wg * DH + c;
        const float fv = unit_dv, fk = unit_dk;
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
          *reinterpret_cast<float4*>(dv + k) =
              fv == 0.0f ? make_float4(0.f, 0.f, 0.f, 0.f)
                         : make_float4(v[k] * fv, v[k + 1] * fv, v[k + 2] * fv, v[k + 3] * fv);
          *reinterpret_cast<float4*>(dk + k) =
              fk == 0.0f ? make_float4(0.f, 0.f, 0.f, 0.f)
                         : make_float4(u[k] * fk, u[k + 1] * fk, u[k + 2] * fk, u[k + 3] * fk);
        }
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

template <int D>
cudaError_t launch_t(const BwdLaunch& f, cudaStream_t st) {
  auto k = attn_bwd_kernel<D>;
  constexpr int smem = BwdLayout<D>::kDynSmem;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(f.args.B * f.args.Hkv * f.args.T);
  k<<<grid, kThreads, smem, st>>>(f.tmQ, f.tmK, f.tmV, f.tmDO, f.tmDQ, f.args, f.lse, f.delta, f.dK, f.dV, f.diag);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd(const BwdLaunch& f, int d, cudaStream_t st) {
  return d == 128 ? launch_t<128>(f, st) : launch_t<64>(f, st);
}

}  // namespace dm
