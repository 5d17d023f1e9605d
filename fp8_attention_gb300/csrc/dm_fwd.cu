// Forward: O = P^ V^ and LSE, one CTA per (batch, query head, 128-row query
// tile), with both matmuls on tcgen05 FP8 MMAs ("Delta-Matching for reliable
// FP8 attention training", section 01: "What changes in FP8?").
//
// For d = 64 and 128 two CTAs share an SM (192 threads, 256 TMEM columns and
// ~97 KB of shared memory each), so that one CTA's softmax overlaps the
// other's products and each SM has two independent MMA issuers.  For d = 256
// (160 KB of tiles) one CTA holds the SM, and S is double-buffered in TMEM
// instead: the tensor core computes S(t+1) while the warpgroup works on S(t).
//
// Warp roles (192 threads):
//   warps 0-3   one warpgroup; thread = query row (TMEM lane), all key
//               columns.  Per key tile t: row max, the tile amax of P~ (one
//               exchange through shared memory), P~ in FP32 straight into
//               E4M3 codes in shared memory, the row sum from the unquantised
//               P~, and the rescale of the O accumulator in TMEM to the units
//               of tile t's scale product before P^_t V_t is added; at the
//               end O / l, staged in shared memory for TMA tile stores
//   warp 4      TMA producer: Q tile once, K and V tiles in two stages each
//               (K one tile ahead of V)
//   warp 5      MMA issuer (+ TMEM owner): S(t) = Q K_t^T, O += P^_t V_t
//
// Each key tile brings its own FP32 scale product c_t = s_P,t * s_V,t.  O is
// kept in TMEM in units of the latest c: before tile t's product is added,
// every row is multiplied by alpha_t * c_{t-1} / c_t (alpha_t the online
// softmax rescale).  The unit is held as its two factors (s_P and s_V of the
// tile it came from), so that neither the unit nor a ratio of two units
// leaves the FP32 range for any pair of tile scales the quantiser produces.
// A tile adds nothing when its product is zero (a flushed P or V tile), or
// when alpha_t * c_{t-1} / c_t exceeds 2^64 in every row (its contribution is
// below 2^-64 of every row's accumulator unit); a row whose maximum jumped in
// tile t (alpha_t tiny) keeps the tile however small c_t is.
//
// TMEM columns: d <= 128: S 0-127, O 128..128+d-1 (256 allocated);
// d = 256: S(t even) 0-127, S(t odd) 128-255, O from 256 (512 allocated; O
// takes 128 columns when V is 128 wide).
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <type_traits>

#include "dm_device.cuh"
#include "dm_pdl.cuh"
#include "dm_internal.h"

namespace dm {
namespace {

constexpr int kThreads = 192;
constexpr int kKV = 2;  // K shared-memory stages (V has one: it is needed a whole tile later than K)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2FmaxE4M3 = 8.807354922057604f;  // log2 448

template <int D>
struct FwdCfg {
  static constexpr int kSBuf = D > 128 ? 2 : 1;  // S buffers in TMEM
  static constexpr uint32_t kColO = 128u * kSBuf;
  static constexpr uint32_t kTmemCols = D > 128 ? 512 : 256;
  static constexpr int kCTAsPerSM = D > 128 ? 1 : 2;
};

struct FwdBars {
  uint64_t q, kfull[kKV], kempty[kKV], vfull, vempty, sfull[2], sempty[2], pready, ofull, stall, mma_done;
};

// Everything lives in dynamic shared memory (no static shared variables), so
// the 1024-byte aligned tile region starts at the window's base.
template <int D, int DV>
struct FwdLayout {
  static constexpr int kTileBytes = kTile * D;   // one FP8 Q or K tile (OpTile<D>)
  static constexpr int kVBytes = kTile * DV;     // one FP8 V tile (OpTile<DV>)
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;          // kKV stages
  static constexpr int kV = kK + kKV * kTileBytes;    // one stage
  static constexpr int kP = kV + kVBytes;             // 2 x (128 x 128) P^ codes
  static constexpr int kRed = kP + 2 * kTile * kTile;  // float [2][4] per-warp amax exponents
  static constexpr int kMode = kRed + 2 * 4 * 4;      // int [2] per-tile P V mode
  static constexpr int kBars = kMode + 16;
  static constexpr int kMisc = kBars + ((int)(sizeof(FwdBars) + 15) / 16) * 16;  // tmem address, abort flag
  static constexpr int kBytes = kMisc + 16;
  // the epilogue stages O (up to 4 bytes x DV columns a row) over K, V and P
  static_assert(kRed - kK >= kTile * DV * 4, "K, V and P buffers hold an fp32 O tile");
  static_assert(kK % 1024 == 0, "staging boxes need 1024-byte alignment");
};

// O (this warp's lanes, D columns at taddr) *= f, 64 columns per TMEM round trip.
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t taddr, float f) {
  const float2 f2 = make_float2(f, f);
#pragma unroll
  for (int c = 0; c < D; c += 64) {
    float v[64];
    tmem_load64(taddr + c, taddr + c + 32, v);
#pragma unroll
    for (int k = 0; k < 64; k += 2) {
      const float2 x = __fmul2_rn(make_float2(v[k], v[k + 1]), f2);
      v[k] = x.x;
      v[k + 1] = x.y;
    }
    tmem_store32(taddr + c, *reinterpret_cast<const float(*)[32]>(&v[0]));
    tmem_store32(taddr + c + 32, *reinterpret_cast<const float(*)[32]>(&v[32]));
  }
}

// D: head dimension of Q and K; DV: of V and O (DV <= D).
template <int D, int DV, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, FwdCfg<D>::kCTAsPerSM)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const AttnArgs a, float* __restrict__ lse) {
  using L = FwdLayout<D, DV>;
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  FwdBars& bars = *reinterpret_cast<FwdBars*>(sm + L::kBars);
  float(*s_red)[4] = reinterpret_cast<float(*)[4]>(sm + L::kRed);
  int* s_mode = reinterpret_cast<int*>(sm + L::kMode);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + L::kMisc);
  int* s_abort = reinterpret_cast<int*>(sm + L::kMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = a.B * a.Hq;
  const int qt = a.T - 1 - (int)(blockIdx.x / BH);  // longest causal rows first
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / a.Hq, h = bh % a.Hq;
  const int bg = b * a.Hkv + h / (a.Hq / a.Hkv);
  const int q0 = qt * kTile;
  // key tiles of the block this query tile sees (0: none, for a causal query
  // tile before the block)
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
    }
    mbar_init(&bars.vfull, 1);
    mbar_init(&bars.vempty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.sfull[s], 1);
      mbar_init(&bars.sempty[s], 4);
    }
    mbar_init(&bars.pready, 4);
    mbar_init(&bars.ofull, 1);
    mbar_init(&bars.stall, 1);
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
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmO);
      mbar_arrive_expect_tx(&bars.q, L::kTileBytes);
      tma_load_tile<D>(sm + L::kQ, &tmQ, &bars.q, q0, bh);
      // K runs one tile ahead of V: K(t) needs only S(t-2) to have finished
      // with its stage, V(t) needs P V(t-1), which completes a tile later.
      int k_issued = 0, v_issued = 0;  // loads issued (both stop early on abort)
      for (int t = 0; t <= nkv; ++t) {
        if (t < nkv) {
          const int s = t % kKV;
          if (!wait(&bars.kempty[s], ((t / kKV) & 1) ^ 1, wd, 101)) break;
          mbar_arrive_expect_tx(&bars.kfull[s], L::kTileBytes);
          tma_load_tile<D>(sm + L::kK + s * L::kTileBytes, &tmK, &bars.kfull[s], t * kTile, bg);
          k_issued = t + 1;
        }
        if (t >= 1) {
          const int u = t - 1;
          if (!wait(&bars.vempty, (u & 1) ^ 1, wd, 102)) break;
          mbar_arrive_expect_tx(&bars.vfull, L::kVBytes);
          tma_load_tile<DV>(sm + L::kV, &tmV, &bars.vfull, u * kTile, bg);
          v_issued = u + 1;
        }
      }
      // every issued load has landed before the CTA may exit
      wait_drain(&bars.q, 0, wd, 116);
      for (int t = max(0, k_issued - kKV); t < k_issued; ++t)
        wait_drain(&bars.kfull[t % kKV], (t / kKV) & 1, wd, 117);
      if (v_issued > 0) wait_drain(&bars.vfull, (v_issued - 1) & 1, wd, 118);
    }
  } else if (warp == 5) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f8(0, 0, 0, 0, kTile, kTile);  // Q K^T, both K-major
      constexpr uint32_t kIdO = idesc_f8(0, 0, 0, 1, kTile, DV);     // P^ (K-major) V (MN-major)
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
      for (int t = 0; t <= nkv && ok; ++t) {
        if (t < nkv) {
          // S(t) once K(t) has landed and the warpgroup has read the S that
          // last used its buffer, S(t - kSBuf)
          const int ks = t % kKV, sb = t % C::kSBuf;
          ok = wait(&bars.kfull[ks], (t / kKV) & 1, wd, 105) &&
               (t < C::kSBuf || wait(&bars.sempty[sb], ((t / C::kSBuf) & 1) ^ 1, wd, 106));
          if (!ok) break;
          tc_fence_after();
          const uint32_t sK = smem_u32(sm + L::kK + ks * L::kTileBytes);
#pragma unroll
          for (int k = 0; k < D / 32; ++k)
            mma_f8(tmem + 128u * sb, OpTile<D>::kmajor(sQ, k), OpTile<D>::kmajor(sK, k), kIdS, k > 0);
          mma_commit(&bars.sfull[sb]);
          mma_commit(&bars.kempty[ks]);
        }
        if (t >= 1) {
          // O += P^(u) V(u) once the codes are written and O is rescaled
          const int u = t - 1;
          ok = wait(&bars.pready, u & 1, wd, 107) && wait(&bars.vfull, u & 1, wd, 108);
          if (!ok) break;
          tc_fence_after();
          const int mode = s_mode[u & 1];  // 0 skip, 1 overwrite, 2 accumulate
          if (mode) {
            const uint32_t sV = smem_u32(sm + L::kV);
            const uint32_t sP = smem_u32(sm + L::kP + (u & 1) * kTile * kTile);
#pragma unroll
            for (int k = 0; k < kTile / 32; ++k)
              mma_f8(tmem + C::kColO, SwTile<128>::kmajor(sP, k), OpTile<DV>::mnmajor(sV, k), kIdO,
                     (k > 0 || mode == 2) ? 1u : 0u);
          }
          mma_commit(&bars.ofull);
          mma_commit(&bars.vempty);
        }
      }
      mma_commit(&bars.mma_done);
      wait_drain(&bars.mma_done, 0, wd, 119);
    }
  } else if (warp < 4) {
    // ---------------------------------------- softmax, P codes and O rescale
    const int row = warp * 32 + lane;
    const int qi = q0 + row;
    const bool row_valid = qi < a.N;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    const float sq = a.q_scales[bh * a.T + qt];
    const float* ksc = a.k_scales + (size_t)bg * a.Tk;
    const float* vsc = a.v_scales + (size_t)bg * a.Tk;
    float sk_next = ksc[0], sv_next = vsc[0];  // per-tile scales, loaded one tile ahead
    float m = -INFINITY, l = 0.0f;             // running max (log2 units), row sum
    float u_p = 0.0f, u_v = 0.0f;              // O in true units = u_p * u_v * O_tmem

    for (int t = 0; t < nkv; ++t) {
      const float c1 = a.sigma * sq * sk_next * kLog2e;
      const float sv = sv_next;
      if (t + 1 < nkv) {
        sk_next = ksc[t + 1];
        sv_next = vsc[t + 1];
      }
      const int j0 = t * kTile;  // first key of the tile within the block
      int jlim = min(kTile, a.Nk - j0);
      if (a.causal) jlim = min(jlim, qi - (j0 + a.kt_off * kTile) + 1);
      // no masked column in this warp's rows (all but the diagonal/ragged
      // tile); warp-uniform, because the masked and unmasked paths both issue
      // warp-collective TMEM loads
      const bool full = __all_sync(0xffffffffu, jlim >= kTile);

      const int sb = t % C::kSBuf;
      const uint32_t tS = tl + 128u * sb;  // this tile's S
      wait(&bars.sfull[sb], (t / C::kSBuf) & 1, wd, 110);
      tc_fence_after();

      // row max (raw units; c1 > 0 preserves the order), S read in halves;
      // the second half stays in registers for its codes, the first is read
      // again (half a row of registers live at a time)
      float mx = -INFINITY;
      float v1[64];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float v0[64];
        float(&v)[64] = hh == 0 ? v0 : v1;
        tmem_load64(tS + 64 * hh, tS + 64 * hh + 32, v);
        if (full) {
          float m4[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
          for (int c = 4; c < 64; c += 8) {
            m4[0] = max3(m4[0], v[c], v[c + 1]);
            m4[1] = max3(m4[1], v[c + 2], v[c + 3]);
            m4[2] = max3(m4[2], v[c + 4], v[c + 5]);
            m4[3] = max3(m4[3], v[c + 6], v[c + 7]);
          }
          mx = max3(mx, fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (64 * hh + c < jlim) mx = fmaxf(mx, v[c]);
        }
      }
      // The tile amax of P~ = max over rows of exp2(tmax_i - m_new_i) =
      // exp2(min(0, max over rows of (tmax_i - m_i))): one exchange.
      const float tmax = mx * c1;
      float x = (row_valid && mx != -INFINITY) ? tmax - m : -INFINITY;
      x = warp_max_any(x);
      if (lane == 0) s_red[t & 1][warp] = x;
      named_bar_sync(1, 128);
      const float m_new = fmaxf(m, tmax);
      const float4 x4 = *reinterpret_cast<const float4*>(s_red[t & 1]);  // 16-byte aligned row
      const float xmax = fmaxf(max3(x4.x, x4.y, x4.z), x4.w);
      const float xm = fminf(xmax, 0.0f);  // log2 of the tile amax of P~
      const float amax = ex2(xm);
      float r;
      const float sp = tile_scale_fast<0>(amax, r);
      const float alpha = ex2(m - m_new);
      // How O enters the units of this tile's product (uniform over the CTA:
      // the scales are the same for every row, only alpha differs; the
      // largest rise of a row maximum in this tile is max(xmax, 0)), decided
      // here so that fewer values stay live across the code conversion.
      // mode 0: the tile adds nothing (O *= alpha); 1: O holds nothing yet
      // (or only zeros), overwrite; 2: O *= g, then accumulate.
      int mode;
      float g = alpha;
      if (u_p == 0.0f) {
        mode = 1;
      } else if (sp == 0.0f || sv == 0.0f) {
        mode = 0;  // a flushed P or V tile adds exactly nothing
      } else {
        // unit / c, with 1 / s_P = r (the tile's code reciprocal); up to 2^64
        // every row accumulates (its factor is at most unit / c)
        const float ratio = (u_p * r) * __fdividef(u_v, sv);  // s_V <= FLT_MAX / 448 < 2^126
        if (ratio <= 0x1p64f) {
          mode = 2;
          g = alpha * ratio;
        } else {
          // the smallest per-row factor is 2^(lg - max rise), lg = log2(unit / c)
          const float lg = (__log2f(u_p) - __log2f(sp)) + (__log2f(u_v) - __log2f(sv));
          if (lg - fmaxf(xmax, 0.0f) > 64.0f) {
            mode = 0;  // below 2^-64 of every row's accumulator unit
          } else {
            mode = 2;
            g = alpha * ratio;
            // a ratio of the factors out of range (inf, or 0 * inf): the same
            // factor from its logarithm, capped where FP32 ends
            if (!(g <= 0x1p100f)) g = ex2(fminf((m - m_new) + lg, 126.0f));
          }
        }
      }
      if (mode != 0) {
        u_p = sp;
        u_v = sv;
      }

      // P~ r = exp2(S c1 - m + log2 r) straight into E4M3 codes (P buffer
      // t%2, last read by P V(t-2), whose completion this thread saw before
      // its rescale of tile t-1); the
      // unquantised row sum is sum(P~ r) * s_P.  A flushed tile (r = 0)
      // gives codes 0.
      // log2 r = log2 FMAX - log2 amax, formed without a logarithm
      const float bias = (r > 0.0f ? kLog2FmaxE4M3 - xm : -INFINITY) - m_new;
      const float2 c1_2 = make_float2(c1, c1), b2 = make_float2(bias, bias);
      float2 rs2 = make_float2(0.0f, 0.0f);
      const uint32_t sP = L::kP + (t & 1) * kTile * kTile + SwTile<128>::row_base(row);  // chunk c at sP ^ 16 c
      auto p_codes = [&](auto full_tile) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int hh = 1 - i;  // the kept second half first
          float v0[64];
          float(&v)[64] = hh == 1 ? v1 : v0;
          if (hh == 0) {
            tmem_load64(tS, tS + 32, v);
            // S has been read: the tensor core may write the buffer again
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.sempty[sb]);
          }
#pragma unroll
          for (int c = 0; c < 64; c += 16) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int cc = c + 4 * e, col = 64 * hh + cc;
              const float2 x01 = __ffma2_rn(make_float2(v[cc], v[cc + 1]), c1_2, b2);
              const float2 x23 = __ffma2_rn(make_float2(v[cc + 2], v[cc + 3]), c1_2, b2);
              float2 q01 = make_float2(ex2(x01.x), ex2(x01.y)), q23 = make_float2(ex2(x23.x), ex2(x23.y));
              if (!decltype(full_tile)::value) {
                q01.x = col < jlim ? q01.x : 0.0f;
                q01.y = col + 1 < jlim ? q01.y : 0.0f;
                q23.x = col + 2 < jlim ? q23.x : 0.0f;
                q23.y = col + 3 < jlim ? q23.y : 0.0f;
              }
              rs2 = __fadd2_rn(rs2, __fadd2_rn(q01, q23));
              w4[e] = pack4_e4m3(q01.x, q01.y, q23.x, q23.y);
            }
            *reinterpret_cast<uint4*>(sm + (sP ^ (uint32_t)(4 * hh + c / 16) * 16u)) =
                make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      };
      if (full)
        p_codes(std::true_type{});
      else
        p_codes(std::false_type{});
      l = alpha * l + (rs2.x + rs2.y) * sp;
      m = m_new;

      // O into the units of this tile's product
      if (t >= 1) {
        wait(&bars.ofull, (t - 1) & 1, wd, 114);  // P V(t-1) has been added into O
        tc_fence_after();
      }
      if (mode != 1) rescale_o<DV>(tl + C::kColO, g);
      if (tid == 0) s_mode[t & 1] = mode;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.pready);
    }

    // LSE and O / l; O rows are a.dv wide (the kernel's d columns of O hold
    // zeros beyond the value head dimension).  A query tile that sees no key
    // of the block writes LSE = -inf and O = 0.
    if (row_valid) lse[(size_t)bh * a.N + qi] = nkv > 0 ? m * kLn2 + logf(l) : -INFINITY;
    if (nkv > 0) {
      wait(&bars.ofull, (nkv - 1) & 1, wd, 115);
      tc_fence_after();
    }
    const float linv = nkv > 0 ? u_p / l : 0.0f;  // O = O_tmem * (u_p / l) * u_v, two products so that no factor underflows
    // O / l staged over the K, V and P buffers (every product has completed)
    // in boxes of 128 rows x 128 bytes with the 128-byte swizzle, then
    // written by TMA tile stores (rows past N are not written); O rows are
    // a.dv wide (the kernel's columns past the value head dimension are
    // not stored)
    constexpr int kBoxCols = OUT_BF16 ? 64 : 32;  // O columns per 128-byte box row
    const uint32_t rsw = SwTile<128>::row_base(row);
    const int dv = a.dv;
#pragma unroll
    for (int c0 = 0; c0 < DV; c0 += 64) {
      if (c0 >= dv) break;  // uniform over the CTA
      float o[64];
      if (nkv > 0) {  // uniform: TMEM loads are warp-collective
        tmem_load64(tl + C::kColO + c0, tl + C::kColO + c0 + 32, o);
      } else {
#pragma unroll
        for (int k = 0; k < 64; ++k) o[k] = 0.0f;
      }
      if (OUT_BF16) {
        const uint32_t box = L::kK + (uint32_t)(c0 / kBoxCols) * (kTile * 128) + rsw;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn((o[8 * e + 2 * j] * linv) * u_v,
                                                      (o[8 * e + 2 * j + 1] * linv) * u_v);
            w[j] = *reinterpret_cast<uint32_t*>(&h2);
          }
          *reinterpret_cast<uint4*>(sm + (box ^ (16u * e))) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const uint32_t box = L::kK + (uint32_t)((c0 + 32 * b) / kBoxCols) * (kTile * 128) + rsw;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float* x = &o[32 * b + 4 * e];
            *reinterpret_cast<float4*>(sm + (box ^ (16u * e))) =
                make_float4((x[0] * linv) * u_v, (x[1] * linv) * u_v, (x[2] * linv) * u_v, (x[3] * linv) * u_v);
          }
        }
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1, 128);
    if (tid == 0) {
      for (int bx = 0; bx * kBoxCols < dv && bx * kBoxCols < DV; ++bx)
        tma_store_3d(&tmO, sm + L::kK + bx * (kTile * 128), bx * kBoxCols, q0, bh);
      bulk_commit();
      bulk_wait_all();  // the staging tile is read and O written before the CTA ends
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int DV, bool BF16>
cudaError_t launch_fwd_t(const FwdLaunch& f, cudaStream_t st) {
  auto k = attn_fwd_kernel<D, DV, BF16>;
  constexpr int smem = FwdLayout<D, DV>::kBytes;
  static_assert(FwdCfg<D>::kCTAsPerSM * (smem + 1024) <= 233472, "the forward CTAs must fit in one SM's shared memory");
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(f.args.B * f.args.Hq * f.args.T);
  return launch_overlapped(k, grid, kThreads, smem, st, f.tmQ, f.tmK, f.tmV, f.tmO, f.args, f.lse);
}

}  // namespace

cudaError_t launch_attn_fwd(const FwdLaunch& f, int d, int dv, bool o_bf16, cudaStream_t st) {
  if (d == 256 && dv == 128) return o_bf16 ? launch_fwd_t<256, 128, true>(f, st) : launch_fwd_t<256, 128, false>(f, st);
  if (d == 256) return o_bf16 ? launch_fwd_t<256, 256, true>(f, st) : launch_fwd_t<256, 256, false>(f, st);
  if (d == 128) return o_bf16 ? launch_fwd_t<128, 128, true>(f, st) : launch_fwd_t<128, 128, false>(f, st);
  return o_bf16 ? launch_fwd_t<64, 64, true>(f, st) : launch_fwd_t<64, 64, false>(f, st);
}

}  // namespace dm
