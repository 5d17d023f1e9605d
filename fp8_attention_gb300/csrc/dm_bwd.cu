// Backward: dQ, dK, dV with the five backward matmuls on tcgen05 FP8 MMAs
// ("Delta-Matching for reliable FP8 attention training", section 01, "Write
// down softmax backward", and section 03 for delta).  One CTA per (batch,
// query head, 128-row key tile), launched longest first; it loops over the
// query tiles that see the key tile (iterations n).  The key tiles from
// a.bwd_pair_kt on (the short ones under a causal mask) are taken by CTAs
// that walk two query heads of a GQA group, head by head, so that each CTA's
// fill and drain serve twice the work and its dV and dK sum over both heads
// before one reduction; pairing the long ones as well would leave a longer
// tail of CTAs at the end of the launch.  A CTA's dK and dV tiles (its
// heads' share of the kv head's gradients) are added into global dK and dV
// with TMA bulk reduce-adds, like dQ.  Over a key block (context
// parallelism) the CTAs take the block's key tiles only (kt is the block's
// own tile index, kt + kt_off the global one), and dQ holds the block's
// partial sums.  Products are computed transposed (key
// rows on TMEM lanes) so that dV and dK accumulate in TMEM:
//   S^T  = K Q^T                 P  = exp(S - LSE) in FP32,   P^  = E4M3 per 128x128 tile
//   dP^T = V dO^T                dS = P (dP - delta) in FP32, dS^ = E5M2 per 128x128 tile
//   dV  += P^T dO     dK += dS^T Q     dQ_i = dS^ K (each staged, then bulk reduce-added)
//
// TMEM (512 columns): two 128-column work buffers and the two accumulators.
// Iteration n uses work buffer n%2 three times in a row: S(n), then dP(n) once
// S(n) has been read, then dQ(n) once dP(n) has been read.  The other buffer
// meanwhile carries iteration n-1's dQ and n+1's S, so the tensor core runs
// S(n+1), [dV dK dQ](n) and dP(n+1) while the compute warps work on n:
//   cols 0-127 work buffer 0, 128-255 work buffer 1, 256.. dV, 384.. dK.
// dV and dK accumulate in units of the current iteration's scale product
// (s_P * s_dO, resp. s_dS * sigma * s_Q): before each accumulation the compute
// warps rescale the accumulator by old/new unit.  Each unit is held as its two
// factors, so that neither a unit nor a ratio of two units leaves the FP32
// range for any tile scales the quantiser produces (down to its 2^-96 flush).
// An iteration adds nothing when one of its scales is zero (a flushed tile)
// or its product is below 2^-64 of the accumulator's unit.
//
// Warp roles (384 threads): warp 0 TMA, warp 1 MMA, warp 2 the dQ reducer,
// warp 3 idle (each warpgroup starts at a multiple of four warps), warps 4-11
// two compute warpgroups; thread = key row, warpgroup = half of the query
// columns (and half of the d columns for the dV/dK/dQ epilogues).
//
// d = 256 splits the head dimension over two CTAs per key tile ("halves"):
// dV, dK and dQ of 128 key/query rows x 256 columns, plus the work buffers,
// do not fit one SM's 512 TMEM columns.  Each half owns 128 of the d columns
// of dV, dK and dQ (its accumulators take the same TMEM columns as d = 128)
// and computes S and dP itself over the full d (four K steps on each
// 128-column sub-tile; the products dV, dK, dQ only over its columns).  Shared memory (227 KB) holds K
// and V whole, this half's columns of Q and dO in two stages, the other
// columns in one stage (needed only by S and dP, which finish early in an
// iteration), one P^ and one dS^ code tile, and a 64-column dQ staging tile
// drained in two passes.
#include <cudaTypedefs.h>

#include "dm_device.cuh"
#include "dm_internal.h"

namespace dm {
namespace {

constexpr int kThreads = 384;  // warps 0-3: TMA, MMA, dQ reducer, idle; warps 4-11: compute
constexpr float kLog2e = 1.4426950408889634f;

struct BwdBars {
  uint64_t kv, qfull[2], qempty[2], sfull[2], sread[2], dpfull[2], bfree[2], pds, mma2, mma_done, dq_staged,
      dq_free, ofull, oempty;
};

template <int D>
struct BwdCfg {
  static constexpr bool kSplit = D > 128;            // two CTAs per key tile, one per 128 d columns
  static constexpr int kDC = kSplit ? 128 : D;       // d columns of dV, dK, dQ this CTA accumulates
  static constexpr int kDH = kDC / 2;                // ... per compute warpgroup
  static constexpr int kCodeBufs = kSplit ? 1 : 2;   // P^T and dS^T code tiles
  static constexpr int kStageCols = kSplit ? 64 : kDC;  // fp32 columns per staged dQ/dK/dV pass
  static constexpr int kPasses = kDC / kStageCols;
};

// Everything lives in dynamic shared memory (no static shared variables), so
// the 1024-byte aligned tile region starts at the window's base.
template <int D>
struct BwdLayout {
  using C = BwdCfg<D>;
  static constexpr int kTileBytes = kTile * D;    // K, V (OpTile<D>)
  static constexpr int kOwnBytes = kTile * C::kDC;  // this CTA's columns of a Q or dO tile
  static constexpr int kOtherBytes = C::kSplit ? kTile * 128 : 0;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;             // 2 stages
  static constexpr int kDO = kQ + 2 * kOwnBytes;         // 2 stages
  static constexpr int kQo = kDO + 2 * kOwnBytes;        // split: the other half's Q columns, one stage
  static constexpr int kDOo = kQo + kOtherBytes;         // split: ... and dO columns
  static constexpr int kPt = kDOo + kOtherBytes;         // P^T codes, [key row][128 query bytes]
  static constexpr int kDSt = kPt + C::kCodeBufs * kTile * kTile;  // dS^T codes
  static constexpr int kDQ = kDSt + C::kCodeBufs * kTile * kTile;  // staging: boxes of [128 rows][32 fp32]
  static constexpr int kLse = kDQ + kTile * C::kStageCols * 4;      // float [2][128]
  static constexpr int kDl = kLse + 2 * kTile * 4;      // float [2][128]
  static constexpr int kRed = kDl + 2 * kTile * 4;      // float [2][2][8]
  static constexpr int kMode = kRed + 2 * 2 * 8 * 4;    // int [2][2]
  static constexpr int kBars = kMode + 16;              // BwdBars
  static constexpr int kMisc = kBars + ((int)(sizeof(BwdBars) + 15) / 16) * 16;  // tmem address, abort flag
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kDynSmem = kBytes;
  // the unsplit epilogue stages dK over the Q/dO stages and dV over the code tiles
  static_assert(C::kSplit || kPt - kQ >= kTile * C::kStageCols * 4, "Q/dO stages hold a staging tile");
  static_assert(C::kSplit || kDQ - kPt >= kTile * C::kStageCols * 4, "code tiles hold a staging tile");
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

// Largest of the eight warp maxima (16-byte aligned): two vector loads.
__device__ __forceinline__ float max8(const float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(v)[0], b = reinterpret_cast<const float4*>(v)[1];
  return fmaxf(max3(a.x, a.y, a.z), max3(a.w, b.x, max3(b.y, b.z, b.w)));
}

// Unit bookkeeping for one TMEM accumulator; every compute thread holds an
// identical copy.  The accumulator's true value is ua * ub * D_tmem; the
// iteration's product comes in units ca * cb (ra = 1 / ca, known from the
// tile's quantisation).  Sets f to the factor the accumulator must be
// multiplied by (1 when it stays) and returns the MMA mode: 0 skip,
// 1 overwrite, 2 accumulate.
__device__ __forceinline__ int unit_step(float& ua, float& ub, float ca, float ra, float cb, float& f) {
  f = 1.0f;
  if (ca == 0.0f || cb == 0.0f) return 0;  // a flushed tile adds exactly nothing
  if (ua == 0.0f) {
    ua = ca;
    ub = cb;
    return 1;
  }
  f = (ua * ra) * __fdividef(ub, cb);  // unit / c
  if (!(f >= 0x1p-100f && f <= 0x1p64f)) {
    // out of the common range (or a ratio of the factors out of FP32 range):
    // decide on the logarithm
    const float lg = (__log2f(ua) - __log2f(ca)) + (__log2f(ub) - __log2f(cb));
    if (lg > 64.0f) {  // below 2^-64 of the accumulator's unit
      f = 1.0f;
      return 0;
    }
    f = ex2(lg);  // a tiny factor only shrinks what the new product outweighs
  }
  ua = ca;
  ub = cb;
  return 2;
}

// dV *= fv and dK *= fk over this warp's lanes and this warpgroup's DH
// columns of each, with one TMEM load and one store of both.
template <int DH>
__device__ __forceinline__ void rescale_pair(uint32_t tdv, float fv, uint32_t tdk, float fk) {
  static_assert(DH == 32 || DH == 64, "unsupported column split");
  float v[2 * DH];
  if constexpr (DH == 64)
    tmem_load128(tdv, tdv + 32, tdk, tdk + 32, v);
  else
    tmem_load64(tdv, tdk, v);
#pragma unroll
  for (int k = 0; k < 2 * DH; k += 2) {
    const float f = k < DH ? fv : fk;
    const float2 x = __fmul2_rn(make_float2(v[k], v[k + 1]), make_float2(f, f));
    v[k] = x.x;
    v[k + 1] = x.y;
  }
  if constexpr (DH == 64) {
    tmem_store128(tdv, tdv + 32, tdk, tdk + 32, v);
  } else {
    tmem_store32(tdv, *reinterpret_cast<const float(*)[32]>(&v[0]));
    tmem_store32(tdk, *reinterpret_cast<const float(*)[32]>(&v[32]));
  }
}

// dK *= fk over this warp's lanes and this warpgroup's DH columns (a CTA
// that holds no dV columns).
template <int DH>
__device__ __forceinline__ void rescale_single(uint32_t tdk, float fk) {
  static_assert(DH == 32 || DH == 64, "unsupported column split");
  float v[64];
  if constexpr (DH == 64)
    tmem_load64(tdk, tdk + 32, v);
  else
    tmem_load32(tdk, *reinterpret_cast<float(*)[32]>(&v[0]));
#pragma unroll
  for (int k = 0; k < DH; k += 2) {
    const float2 x = __fmul2_rn(make_float2(v[k], v[k + 1]), make_float2(fk, fk));
    v[k] = x.x;
    v[k + 1] = x.y;
  }
  tmem_store32(tdk, *reinterpret_cast<const float(*)[32]>(&v[0]));
  if constexpr (DH == 64) tmem_store32(tdk + 32, *reinterpret_cast<const float(*)[32]>(&v[32]));
}

// PARTIAL (d = 256 kernels only): the value or query/key head dimension is
// narrower than D, so a half may own fewer dV, dK or dQ columns than its 128
// (checked at run time); without it every half owns all of its columns.
template <int D, bool PARTIAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmDK,
                    const __grid_constant__ CUtensorMap tmDV, const AttnArgs a, const float* __restrict__ lse,
                    const float* __restrict__ delta, const dm_diag diag) {
  using L = BwdLayout<D>;
  using C = BwdCfg<D>;
  constexpr int DH = C::kDH;  // d columns per compute warpgroup
  constexpr int SH = C::kStageCols / 2;  // ... per staging pass
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  BwdBars& bars = *reinterpret_cast<BwdBars*>(sm + L::kBars);
  float(*s_lse)[kTile] = reinterpret_cast<float(*)[kTile]>(sm + L::kLse);
  float(*s_dl)[kTile] = reinterpret_cast<float(*)[kTile]>(sm + L::kDl);
  float(*s_red)[2][8] = reinterpret_cast<float(*)[2][8]>(sm + L::kRed);
  int(*s_mode)[2] = reinterpret_cast<int(*)[2]>(sm + L::kMode);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  int* s_abort = reinterpret_cast<int*>(sm + L::kMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = a.B * a.Hq;
  // split: the two halves of a key tile are neighbouring CTAs
  const int hf = C::kSplit ? (int)(blockIdx.x & 1u) : 0;
  const int blk = (int)(C::kSplit ? blockIdx.x >> 1 : blockIdx.x);
  // key tile 0 sees the most query tiles: first.  Key tiles below
  // a.bwd_pair_kt have one CTA per query head, the rest one per head pair.
  const int n_single = a.bwd_pair_kt * BH;
  const int hpc = blk < n_single ? 1 : 2;  // query heads of this CTA
  const int kt = blk < n_single ? blk / BH : a.bwd_pair_kt + (blk - n_single) / (BH / 2);
  const int bh0 = blk < n_single ? blk % BH : ((blk - n_single) % (BH / 2)) * 2;  // first b * Hq + h
  const int col0 = hf * C::kDC;  // this CTA's first d column
  // dV columns exist only below the value head dimension (narrower than the
  // kernel's d for heads shaped like multi-head latent attention; the
  // unsplit kernels run only with the value dimension equal to d)
  constexpr bool kPart = C::kSplit && PARTIAL;
  const bool own_dv = !kPart || col0 < a.dv;
  // dQ/dK columns this CTA holds below the query/key head dimension (split:
  // 0, 64 or 128 of its 128; the rest hold zeros) and the dQ staging passes
  // they need
  const int own_qk = kPart ? max(0, min(C::kDC, a.dqk - col0)) : C::kDC;
  const int n_passes = kPart ? (own_qk + C::kStageCols - 1) / C::kStageCols : C::kPasses;
  const int bg = (bh0 / a.Hq) * a.Hkv + (bh0 % a.Hq) / (a.Hq / a.Hkv);
  const int ktg = kt + a.kt_off;  // the key tile's index in the whole sequence
  const int qt0 = a.causal ? ktg : 0;
  const int n_head = a.T - qt0;  // iterations per query head (>= 1)
  const int n_iter = hpc * n_head;
  // query head (b * Hq + h) and query tile of iteration n
  auto head_of = [&](int n) { return bh0 + (hpc == 2 && n >= n_head ? 1 : 0); };
  auto qtile_of = [&](int n) { return qt0 + (n >= n_head ? n - n_head : n); };
  // the halves of a split key tile compute the same dS: one adds the diagnostics
  const bool want_diag =
      hf == 0 && (diag.rowsum_pre || diag.abssum_pre || diag.rowsum_post || diag.abssum_post);

  // The swizzled tiles need a 1024-byte aligned base; the window is expected
  // to start aligned (no static shared variables).  Checked uniformly before
  // anything is initialised: a misaligned window reports an error instead.
  if (smem_u32(smem_raw) & 1023u) {
    if (tid == 0) atomicCAS(a.status, 0u, (unsigned)DM_ERR_UNSUPPORTED);
    return;
  }
  Watchdog wd{s_abort, a.status, a.wait_limit_ns};
  if (tid == 0) {
    *s_abort = 0;
    mbar_init(&bars.kv, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.qfull[s], 1);
      mbar_init(&bars.qempty[s], 1);
      mbar_init(&bars.sfull[s], 1);
      mbar_init(&bars.sread[s], 8);
      mbar_init(&bars.dpfull[s], 1);
      mbar_init(&bars.bfree[s], 8);
    }
    mbar_init(&bars.pds, 8);
    mbar_init(&bars.mma2, 1);
    mbar_init(&bars.mma_done, 1);
    mbar_init(&bars.dq_staged, 8);
    mbar_init(&bars.dq_free, 1);
    mbar_init(&bars.ofull, 1);
    mbar_init(&bars.oempty, 1);
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
      tma_prefetch_desc(&tmDO);
      tma_prefetch_desc(&tmDQ);
      tma_prefetch_desc(&tmDK);
      tma_prefetch_desc(&tmDV);
      mbar_arrive_expect_tx(&bars.kv, 2 * L::kTileBytes);
      tma_load_tile<D>(sm + L::kK, &tmK, &bars.kv, kt * kTile, bg);
      tma_load_tile<D>(sm + L::kV, &tmV, &bars.kv, kt * kTile, bg);
      int issued = 0, o_issued = 0;
      for (int n = 0; n < n_iter; ++n) {
        const int s = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        const int bh = head_of(n), qt = qtile_of(n);
        // this CTA's columns: stage s, free once dV/dK(n-2) have read it
        if (!wait(&bars.qempty[s], ph ^ 1, wd, 301)) break;
        mbar_arrive_expect_tx(&bars.qfull[s], 2 * L::kOwnBytes);
        if constexpr (C::kSplit) {
          tma_load_3d(sm + L::kQ + s * L::kOwnBytes, &tmQ, &bars.qfull[s], col0, qt * kTile, bh);
          tma_load_3d(sm + L::kDO + s * L::kOwnBytes, &tmDO, &bars.qfull[s], col0, qt * kTile, bh);
        } else {
          tma_load_tile<D>(sm + L::kQ + s * L::kOwnBytes, &tmQ, &bars.qfull[s], qt * kTile, bh);
          tma_load_tile<D>(sm + L::kDO + s * L::kOwnBytes, &tmDO, &bars.qfull[s], qt * kTile, bh);
        }
        issued = n + 1;
        if constexpr (C::kSplit) {
          // the other half's columns: one stage, free once S(n-1) and dP(n-1) are done
          if (n >= 1 && !wait(&bars.oempty, (n - 1) & 1, wd, 317)) break;
          mbar_arrive_expect_tx(&bars.ofull, 2 * L::kOtherBytes);
          tma_load_3d(sm + L::kQo, &tmQ, &bars.ofull, 128 - col0, qt * kTile, bh);
          tma_load_3d(sm + L::kDOo, &tmDO, &bars.ofull, 128 - col0, qt * kTile, bh);
          o_issued = n + 1;
        }
      }
      wait_drain(&bars.kv, 0, wd, 302);
      for (int n = max(0, issued - 2); n < issued; ++n) wait_drain(&bars.qfull[n & 1], (n >> 1) & 1, wd, 303);
      if (o_issued > 0) wait_drain(&bars.ofull, (o_issued - 1) & 1, wd, 318);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f8(0, 0, 0, 0, kTile, kTile);   // K Q^T
      constexpr uint32_t kIdDP = idesc_f8(0, 1, 0, 0, kTile, kTile);  // V (E4M3) dO^T (E5M2)
      constexpr int DC = C::kDC;
      constexpr uint32_t kIdDV = idesc_f8(0, 1, 0, 1, kTile, DC);     // P^T (K-major) dO (MN-major)
      constexpr uint32_t kIdDK = idesc_f8(1, 0, 0, 1, kTile, DC);     // dS^T (K-major) Q (MN-major)
      constexpr uint32_t kIdDQ = idesc_f8(1, 0, 1, 1, kTile, DC);     // dS (MN-major) K (MN-major)
      const uint32_t sK = smem_u32(sm + L::kK), sV = smem_u32(sm + L::kV);
      // this CTA's columns of K (split: its sub-tile) for dQ
      const uint32_t sKown = sK + (C::kSplit ? (uint32_t)hf * OpTile<D>::kSubBytes : 0u);
      // dV, dK and dQ of iteration m (its work buffer now takes dQ)
      auto tail = [&](int m) {
        const int bm = m & 1, cb = C::kCodeBufs == 2 ? bm : 0;
        const uint32_t sQ = smem_u32(sm + L::kQ + bm * L::kOwnBytes);
        const uint32_t sDO = smem_u32(sm + L::kDO + bm * L::kOwnBytes);
        const uint32_t sPt = smem_u32(sm + L::kPt + cb * kTile * kTile);
        const uint32_t sDSt = smem_u32(sm + L::kDSt + cb * kTile * kTile);
        const int mode_dv = s_mode[bm][0], mode_dk = s_mode[bm][1];
        if (mode_dv) {
#pragma unroll
          for (int k = 0; k < kTile / 32; ++k)
            mma_f8(tmem + 256, SwTile<128>::kmajor(sPt, k), SwTile<DC>::mnmajor(sDO, k), kIdDV,
                   (k > 0 || mode_dv == 2) ? 1u : 0u);
        }
        if (mode_dk) {
#pragma unroll
          for (int k = 0; k < kTile / 32; ++k)
            mma_f8(tmem + 384, SwTile<128>::kmajor(sDSt, k), SwTile<DC>::mnmajor(sQ, k), kIdDK,
                   (k > 0 || mode_dk == 2) ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < kTile / 32; ++k)
          mma_f8(tmem + bm * 128, SwTile<128>::mnmajor(sDSt, k), SwTile<DC>::mnmajor(sKown, k), kIdDQ, k > 0);
        mma_commit(&bars.mma2);
        mma_commit(&bars.qempty[bm]);
      };
      // A (key rows) x B (query rows) over the full d: split, this half's
      // sub-tile of A with its own columns of B, then the other sub-tile with
      // the other half's columns
      auto full_d = [&](uint32_t d_tmem, uint32_t sA, uint32_t sBown, uint32_t sBother, uint32_t idesc) {
        if constexpr (C::kSplit) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f8(d_tmem, SwTile<128>::kmajor(sA + (uint32_t)hf * OpTile<D>::kSubBytes, k),
                   SwTile<128>::kmajor(sBown, k), idesc, k > 0);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f8(d_tmem, SwTile<128>::kmajor(sA + (uint32_t)(1 - hf) * OpTile<D>::kSubBytes, k),
                   SwTile<128>::kmajor(sBother, k), idesc, 1u);
        } else {
#pragma unroll
          for (int k = 0; k < D / 32; ++k)
            mma_f8(d_tmem, SwTile<D>::kmajor(sA, k), SwTile<D>::kmajor(sBown, k), idesc, k > 0);
        }
      };
      const uint32_t sQo = smem_u32(sm + L::kQo), sDOo = smem_u32(sm + L::kDOo);
      bool ok = wait(&bars.kv, 0, wd, 304);
      for (int n = 0; n < n_iter && ok; ++n) {
        const int bn = n & 1;
        const uint32_t ph = (n >> 1) & 1;
        const uint32_t sQ = smem_u32(sm + L::kQ + bn * L::kOwnBytes);
        const uint32_t sDO = smem_u32(sm + L::kDO + bn * L::kOwnBytes);
        if (!(ok = wait(&bars.qfull[bn], ph, wd, 305))) break;
        if (C::kSplit && !(ok = wait(&bars.ofull, n & 1, wd, 319))) break;
        if (n >= 2 && !(ok = wait(&bars.bfree[bn], ph ^ 1, wd, 306))) break;  // dQ(n-2) drained
        tc_fence_after();
        full_d(tmem + bn * 128, sK, sQ, sQo, kIdS);
        mma_commit(&bars.sfull[bn]);
        if (n >= 1) {
          if (!(ok = wait(&bars.pds, (n - 1) & 1, wd, 307))) break;
          tc_fence_after();
          tail(n - 1);
        }
        if (!(ok = wait(&bars.sread[bn], ph, wd, 308))) break;  // S(n) read: the buffer takes dP(n)
        tc_fence_after();
        full_d(tmem + bn * 128, sV, sDO, sDOo, kIdDP);
        mma_commit(&bars.dpfull[bn]);
        if (C::kSplit) mma_commit(&bars.oempty);  // S(n) and dP(n) have read the other half's columns
      }
      if (ok && n_iter > 0 && wait(&bars.pds, (n_iter - 1) & 1, wd, 309)) {
        tc_fence_after();
        tail(n_iter - 1);
      }
      mma_commit(&bars.mma_done);
      wait_drain(&bars.mma_done, 0, wd, 310);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ dQ reducer
    // Adds each staged dQ pass into global dQ (one bulk reduce per 32-column
    // box) and frees the staging tile once the copies have read it, so that
    // no compute thread waits on the bulk copies.
    if (lane == 0) {
      for (int g = 0; g < n_iter * n_passes; ++g) {
        if (!wait(&bars.dq_staged, g & 1, wd, 314)) break;
        const int m = g / n_passes, ps = g % n_passes;
#pragma unroll
        for (int bx = 0; bx < C::kStageCols / 32; ++bx) {
          const int x = col0 + ps * C::kStageCols + bx * 32;
          if (!kPart || x < a.dqk)  // boxes beyond the head dimension hold zeros
            tma_reduce_add_3d(&tmDQ, sm + L::kDQ + bx * (kTile * 128), x, qtile_of(m) * kTile, head_of(m));
        }
        bulk_commit();
        bulk_wait_read_all();
        mbar_arrive(&bars.dq_free);
      }
      bulk_wait_all();
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- compute
    const int wg = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // key row within the tile (TMEM lane)
    // swizzled offsets of this thread's row in 128-byte row tiles: chunk c at
    // (tile + rsw) ^ 16 c; rsw_wg starts at this warpgroup's 64-byte half
    const uint32_t rsw = SwTile<128>::row_base(r);
    const uint32_t rsw_wg = rsw ^ (64u * wg);
    const bool kv_valid = kt * kTile + r < a.Nk;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const int ct = tid - 128;  // 0..255
    const float sk = a.k_scales[bg * a.Tk + kt];
    const float svv = a.v_scales[bg * a.Tk + kt];
    float udv_a = 0.0f, udv_b = 0.0f, udk_a = 0.0f, udk_b = 0.0f;  // accumulator units (two factors each)
    // Per-iteration global values are loaded one iteration ahead: this
    // thread's element of the query tile's LSE (threads 0-127; +inf for absent
    // rows) or delta (threads 128-255; 0 for absent rows), and the tile's Q and
    // dO scales.
    auto row_value = [&](int bh_n, int qt_n) -> float {
      const int qi = qt_n * kTile + (ct & 127);
      if (ct < 128) return qi < a.N ? lse[(size_t)bh_n * a.N + qi] : INFINITY;
      return qi < a.N ? delta[(size_t)bh_n * a.N + qi] : 0.0f;
    };
    // Stores this thread's element of iteration m's LSE (negated, log2
    // units) or delta (negated) into the double-buffered shared copy.  The
    // copy for m + 1 is written during m, before m's dS barrier, which orders
    // it before every read in m + 1 (and after every read of the same buffer
    // in m - 1).
    auto stage_row = [&](int m, float value) {
      if (ct < 128)
        s_lse[m & 1][ct] = -value * kLog2e;  // one packed FMA per pair below
      else
        s_dl[m & 1][ct - 128] = -value;
    };
    if (n_iter > 0) stage_row(0, row_value(head_of(0), qtile_of(0)));
    float row_next = n_iter > 1 ? row_value(head_of(1), qtile_of(1)) : 0.0f;  // staged during iteration 0
    float pre_sq = n_iter > 0 ? a.q_scales[head_of(0) * a.T + qtile_of(0)] : 0.0f;
    float pre_sdo = n_iter > 0 ? a.do_scales[head_of(0) * a.T + qtile_of(0)] : 0.0f;
    float prev_cdq = 0.0f;  // dQ scale of the previous iteration, drained one iteration late
    named_bar_sync(1, 256);

    // dQ(m) (query rows on TMEM lanes of buffer m%2): scaled, staged in shared
    // memory with the 128-byte swizzle of the dQ tensor map, then added into
    // global dQ by one bulk reduce per 32-column box.  TMEM loads are
    // warp-collective: every lane loads; rows beyond N are clipped by the map.
    // The reducer warp adds each staged pass into global dQ; a pass waits
    // until it has read the one before.  Pass ps stages columns
    // [ps * kStageCols, (ps + 1) * kStageCols) of this CTA's, each warpgroup
    // half of them.  Passes [p0, p1) of the n_passes run here; the TMEM
    // buffer is released after the last (at once when there is none).
    auto drain_dq = [&](int m, float cdq, int p0, int p1) {
      const int bm = m & 1;
      if (p0 == 0) wait(&bars.mma2, m & 1, wd, 311);
      if (p0 == 0 && n_passes == 0) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.bfree[bm]);
      }
#pragma unroll
      for (int ps = 0; ps < C::kPasses; ++ps) {
        if (ps < p0 || ps >= p1 || ps >= n_passes) continue;
        const int g = m * n_passes + ps;
        if (g >= 1) wait(&bars.dq_free, (g - 1) & 1, wd, 315);
        tc_fence_after();
        // 32 columns at a time (the P registers of the current iteration are live)
#pragma unroll
        for (int c = 0; c < SH; c += 32) {
          float v[32];
          tmem_load32(tl + bm * 128 + ps * C::kStageCols + wg * SH + c, v);
          const uint32_t box = L::kDQ + ((wg * SH + c) / 32) * (kTile * 128) + rsw;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 a01 = __fmul2_rn(make_float2(v[4 * e], v[4 * e + 1]), make_float2(cdq, cdq));
            const float2 a23 = __fmul2_rn(make_float2(v[4 * e + 2], v[4 * e + 3]), make_float2(cdq, cdq));
            *reinterpret_cast<float4*>(sm + (box ^ (16u * e))) = make_float4(a01.x, a01.y, a23.x, a23.y);
          }
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (ps == n_passes - 1) mbar_arrive(&bars.bfree[bm]);
          mbar_arrive(&bars.dq_staged);
        }
      }
    };

    for (int n = 0; n < n_iter; ++n) {
      const int bh = head_of(n), qt = qtile_of(n);  // this iteration's query head and tile
      const int qi0 = qt * kTile;
      const int bn = n & 1;
      const uint32_t ph = (n >> 1) & 1;
      const float sq = pre_sq, sdo = pre_sdo;
      if (n + 1 < n_iter) {
        pre_sq = a.q_scales[head_of(n + 1) * a.T + qtile_of(n + 1)];
        pre_sdo = a.do_scales[head_of(n + 1) * a.T + qtile_of(n + 1)];
      }
      const float c1 = a.sigma * sq * sk * kLog2e;
      const float cdp = sdo * svv;
      const int cmin = !kv_valid ? (1 << 30) : (a.causal && qt == ktg) ? r - wg * 64 : 0;

      // P = exp(S - LSE), its tile amax and E4M3 codes
      float p[64];
      wait(&bars.sfull[bn], ph, wd, 312);
      tc_fence_after();
      tmem_load64(tl + bn * 128 + wg * 64, tl + bn * 128 + wg * 64 + 32, p);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.sread[bn]);
      // The exponents x = S c1 - LSE log2e first, masked ones -inf; the tile
      // amax of P = exp2(x) is exp2 of the exponents' maximum (exp2 is
      // monotonic), so the maximum is reduced and exchanged while the
      // exponentials are still in flight.
      const float2 c1_2 = make_float2(c1, c1);
      const float4* nlse4 = reinterpret_cast<const float4*>(&s_lse[bn][wg * 64]);  // broadcast reads
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float4 l4 = nlse4[c / 4];
        const float2 x01 = __ffma2_rn(make_float2(p[c], p[c + 1]), c1_2, make_float2(l4.x, l4.y));
        const float2 x23 = __ffma2_rn(make_float2(p[c + 2], p[c + 3]), c1_2, make_float2(l4.z, l4.w));
        p[c] = x01.x;
        p[c + 1] = x01.y;
        p[c + 2] = x23.x;
        p[c + 3] = x23.y;
      }
      if (cmin > 0) {  // diagonal tile or absent key row: mask
#pragma unroll
        for (int c = 0; c < 64; ++c) p[c] = c >= cmin ? p[c] : -INFINITY;
      }
      float xm0 = -INFINITY, xm1 = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        xm0 = max3(xm0, p[c], p[c + 1]);
        xm1 = max3(xm1, p[c + 2], p[c + 3]);
      }
#pragma unroll
      for (int c = 0; c < 64; ++c) p[c] = ex2(p[c]);  // exp2(-inf) = +0 where masked
      const float xmax = warp_max_any(fmaxf(xm0, xm1));
      if (lane == 0) s_red[bn][0][warp - 4] = xmax;
      named_bar_sync(1, 256);
      float amax;
      {
        const float4 a4 = reinterpret_cast<const float4*>(s_red[bn][0])[0];
        const float4 b4 = reinterpret_cast<const float4*>(s_red[bn][0])[1];
        amax = ex2(fmaxf(max3(a4.x, a4.y, a4.z), max3(a4.w, b4.x, max3(b4.y, b4.z, b4.w))));
      }
      float rp;
      const float sp = tile_scale_fast<0>(amax, rp);
      // P^T codes and the next iteration's LSE / delta (read after this
      // iteration's dS barrier), and the previous iteration's dQ (its
      // completion also means dV/dK(n-1) are done).  The two warpgroups take
      // the two in opposite order, so that on every SM sub-partition one
      // warp's code conversion overlaps the other's TMEM loads and staging.
      const int cb = C::kCodeBufs == 2 ? bn : 0;  // code tiles of this iteration
      // one code tile of each kind: dV/dK/dQ(n-1) must have read it
      if (C::kCodeBufs == 1 && n >= 1) wait(&bars.mma2, (n - 1) & 1, wd, 320);
      auto write_p = [&]() {
        const uint32_t dst = L::kPt + cb * kTile * kTile + rsw_wg;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float* q4 = &p[16 * c + 4 * e];
            const float2 a01 = __fmul2_rn(make_float2(q4[0], q4[1]), make_float2(rp, rp));
            const float2 a23 = __fmul2_rn(make_float2(q4[2], q4[3]), make_float2(rp, rp));
            w4[e] = pack4_e4m3(a01.x, a01.y, a23.x, a23.y);
          }
          *reinterpret_cast<uint4*>(sm + (dst ^ (16u * c))) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        if (n + 1 < n_iter) {
          stage_row(n + 1, row_next);
          if (n + 2 < n_iter) row_next = row_value(head_of(n + 2), qtile_of(n + 2));
        }
      };
      // split: the first dQ pass here, the second after dS (the reducer
      // reads the first meanwhile)
      constexpr int kEarlyPasses = C::kSplit ? 1 : C::kPasses;
      if (wg == 0) {
        write_p();
        if (n >= 1) drain_dq(n - 1, prev_cdq, 0, kEarlyPasses);
      } else {
        if (n >= 1) drain_dq(n - 1, prev_cdq, 0, kEarlyPasses);
        write_p();
      }

      // dS = P (dP - delta), computed in place over p (P in FP32 is not needed
      // once its codes are written), its tile amax and E5M2 codes
      float* ds = p;
      wait(&bars.dpfull[bn], ph, wd, 313);
      tc_fence_after();
      const float2 cdp2 = make_float2(cdp, cdp);
      const float4* ndl4 = reinterpret_cast<const float4*>(&s_dl[bn][wg * 64]);  // broadcast reads
      float dm0 = 0.0f, dm1 = 0.0f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float dp[32];
        tmem_load32(tl + bn * 128 + wg * 64 + h * 32, dp);
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const int cc = h * 32 + c;
          const float4 l4 = ndl4[cc / 4];
          const float2 d01 = __fmul2_rn(make_float2(p[cc], p[cc + 1]),
                                        __ffma2_rn(make_float2(dp[c], dp[c + 1]), cdp2, make_float2(l4.x, l4.y)));
          const float2 d23 = __fmul2_rn(make_float2(p[cc + 2], p[cc + 3]),
                                        __ffma2_rn(make_float2(dp[c + 2], dp[c + 3]), cdp2, make_float2(l4.z, l4.w)));
          ds[cc] = d01.x;
          ds[cc + 1] = d01.y;
          ds[cc + 2] = d23.x;
          ds[cc + 3] = d23.y;
          // plain fmaxf: |x| folds into the max (the three-input asm max cannot take it)
          dm0 = fmaxf(dm0, fmaxf(fabsf(d01.x), fabsf(d01.y)));
          dm1 = fmaxf(dm1, fmaxf(fabsf(d23.x), fabsf(d23.y)));
        }
      }
      if (kEarlyPasses < C::kPasses && n >= 1) drain_dq(n - 1, prev_cdq, kEarlyPasses, C::kPasses);
      float dmax = fmaxf(dm0, dm1);
      dmax = warp_max_nonneg(dmax);  // |dS|
      if (lane == 0) s_red[bn][1][warp - 4] = dmax;
      named_bar_sync(1, 256);
      amax = max8(s_red[bn][1]);
      float rs;
      const float sds = tile_scale_fast<1>(amax, rs);
      // both accumulators into the units of this iteration's products (dV/dK
      // of n - 1 completed before the drain above), after the dS codes
      float fv = 1.0f, fk;
      const int mode_dv = own_dv ? unit_step(udv_a, udv_b, sp, rp, sdo, fv) : 0;
      // 1 / s = FMAX / amax = the tile's code reciprocal r
      const int mode_dk = own_qk > 0 ? unit_step(udk_a, udk_b, sds, rs, a.sigma * sq, fk) : (fk = 1.0f, 0);
      auto write_ds = [&]() {
        uint32_t dcode[16];
        {
          const uint32_t dst = L::kDSt + cb * kTile * kTile + rsw_wg;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float2 a01 = __fmul2_rn(make_float2(ds[4 * c], ds[4 * c + 1]), make_float2(rs, rs));
            const float2 a23 = __fmul2_rn(make_float2(ds[4 * c + 2], ds[4 * c + 3]), make_float2(rs, rs));
            dcode[c] = pack4_e5m2(a01.x, a01.y, a23.x, a23.y);
          }
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4*>(sm + (dst ^ (16u * c))) =
                make_uint4(dcode[4 * c], dcode[4 * c + 1], dcode[4 * c + 2], dcode[4 * c + 3]);
        }
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
      };
      write_ds();
      if (own_dv && own_qk == C::kDC) {
        if (fv != 1.0f || fk != 1.0f) rescale_pair<DH>(tl + 256 + wg * DH, fv, tl + 384 + wg * DH, fk);
      } else if constexpr (kPart) {
        // a split CTA with part of the accumulators: dV whole or absent, dK
        // whole, half (its first 64 columns, 32 per warpgroup) or absent
        if (own_dv && fv != 1.0f) rescale_single<DH>(tl + 256 + wg * DH, fv);
        if (fk != 1.0f) {
          if (own_qk == C::kDC)
            rescale_single<DH>(tl + 384 + wg * DH, fk);
          else if (own_qk == C::kDC / 2)
            rescale_single<DH / 2>(tl + 384 + wg * (DH / 2), fk);
        }
      }
      if (ct == 0) {
        s_mode[bn][0] = mode_dv;
        s_mode[bn][1] = mode_dk;
      }
      prev_cdq = a.sigma * sds * sk;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.pds);

    }
    if (n_iter > 0) {
      drain_dq(n_iter - 1, prev_cdq, 0, C::kPasses);
      // split: the epilogue stages over the dQ staging tile, which the
      // reducer must have read (unsplit: dV and dK go elsewhere; the reducer
      // waits for its own copies before the CTA exits)
      if (C::kSplit && n_passes > 0) wait(&bars.dq_free, (n_iter * n_passes - 1) & 1, wd, 316);
    }
    // epilogue: this head's dV and dK tiles in true units, staged like dQ
    // (after the last dQ reduce has read the staging tile) and added into
    // global dV and dK.  An accumulator that never received a contribution
    // holds garbage and is skipped.  TMEM loads are warp-collective.
    // base: the staging tile; reuse: it held an earlier reduction's source
    auto reduce_acc = [&](uint32_t col, float ua, float ub, const CUtensorMap* map, int width, uint32_t base,
                          bool reuse) {
#pragma unroll
      for (int ps = 0; ps < C::kPasses; ++ps) {
        if (ct == 0 && (reuse || ps > 0)) bulk_wait_read_all();
        named_bar_sync(1, 256);
        // uniform; passes past the width hold zeros (split kernels only)
        if (ua != 0.0f && (!kPart || (int)col0 + ps * C::kStageCols < width)) {
#pragma unroll
          for (int c = 0; c < SH; c += 32) {
            float v[32];
            tmem_load32(tl + col + ps * C::kStageCols + wg * SH + c, v);
            const uint32_t box = base + ((wg * SH + c) / 32) * (kTile * 128) + rsw;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              // two products, so that the unit's factors never underflow together
              const float2 a01 = __fmul2_rn(__fmul2_rn(make_float2(v[4 * e], v[4 * e + 1]), make_float2(ua, ua)),
                                            make_float2(ub, ub));
              const float2 a23 = __fmul2_rn(__fmul2_rn(make_float2(v[4 * e + 2], v[4 * e + 3]), make_float2(ua, ua)),
                                            make_float2(ub, ub));
              *reinterpret_cast<float4*>(sm + (box ^ (16u * e))) =
                  make_float4(a01.x, a01.y, a23.x, a23.y);
            }
          }
          fence_proxy_async_smem();
          named_bar_sync(2, 256);
          if (ct == 0) {
#pragma unroll
            for (int bx = 0; bx < C::kStageCols / 32; ++bx) {
              const int x = col0 + ps * C::kStageCols + bx * 32;
              if (!kPart || x < width) tma_reduce_add_3d(map, sm + base + bx * (kTile * 128), x, kt * kTile, bg);
            }
            bulk_commit();
          }
        }
      }
    };
    // unsplit: dV is staged over the P/dS code tiles and dK over the Q/dO
    // stages (both free once the last products have completed), so the two
    // reductions are in flight together and neither waits for the reducer
    // to have read the last dQ tile
    if constexpr (C::kSplit) {
      reduce_acc(256, udv_a, udv_b, &tmDV, a.dv, L::kDQ, true);
      reduce_acc(384, udk_a, udk_b, &tmDK, a.dqk, L::kDQ, true);
    } else {
      reduce_acc(256, udv_a, udv_b, &tmDV, a.dv, L::kPt, false);
      reduce_acc(384, udk_a, udk_b, &tmDK, a.dqk, L::kQ, false);
    }
    if (ct == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool PARTIAL>
cudaError_t launch_t(const BwdLaunch& f, cudaStream_t st) {
  auto k = attn_bwd_kernel<D, PARTIAL>;
  constexpr int smem = BwdLayout<D>::kDynSmem;
  static_assert(smem <= 232448, "backward shared memory exceeds the per-block limit");
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int BH = f.args.B * f.args.Hq, pk = f.args.bwd_pair_kt;
  const unsigned grid = (unsigned)((pk * BH + (f.args.Tk - pk) * (BH / 2)) * (BwdCfg<D>::kSplit ? 2 : 1));
  k<<<grid, kThreads, smem, st>>>(f.tmQ, f.tmK, f.tmV, f.tmDO, f.tmDQ, f.tmDK, f.tmDV, f.args, f.lse, f.delta,
                                  f.diag);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd(const BwdLaunch& f, int d, cudaStream_t st) {
  if (d == 256)
    return (f.args.dqk == 256 && f.args.dv == 256) ? launch_t<256, false>(f, st) : launch_t<256, true>(f, st);
  return d == 128 ? launch_t<128, false>(f, st) : launch_t<64, false>(f, st);
}

}  // namespace dm
