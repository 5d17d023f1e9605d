// Host-side launch interfaces between the API layer (dm_api.cu) and the
// kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <utility>

#include "dm_common.h"

namespace dm {

// Launches kernel `k` with programmatic stream serialisation: it may start
// while the kernel before it in the stream finishes, and waits for that
// kernel's completion in grid_dependency_sync() before touching global memory.
template <typename... P, typename... A>
inline cudaError_t launch_overlapped(void (*k)(P...), unsigned grid, unsigned threads, size_t smem,
                                     cudaStream_t st, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, std::forward<A>(args)...);
}

struct FwdLaunch {
  CUtensorMap tmQ, tmK, tmV;  // [B*H][N][d] FP8 codes, box 128 x d, hardware swizzle of width d
  CUtensorMap tmO;            // O [B*Hq][N][d_v] fp32 or bf16, box 128 rows x 128 bytes, 128-byte swizzle
  AttnArgs args;
  float* lse;
};

// The backward's outputs that the matched delta pass sets to zero on its way
// (the backward adds into them), when the backward computes delta itself:
// each CTA clears the dQ rows and diagnostics rows of its query tile, and
// the CTAs of a GQA group's first query head the dK and dV rows of the key
// tile with the same index.  All null: nothing is cleared.
struct DeltaClear {
  float* dQ;       // [B*Hq][N][d]
  float* dK;       // [B*Hkv][N][d]
  float* dV;       // [B*Hkv][N][d_v]
  float* rows[4];  // nullable [B*Hq][N] each
};

struct DeltaLaunch {
  CUtensorMap tmQ, tmK, tmV, tmDO;
  AttnArgs args;
  const float* lse;
  float* delta;  // delta, or (with den) sum_j P dP^ over the key block
  float* den;    // nullable: sum_j P over the key block
  DeltaClear clear;
};

struct BwdLaunch {
  CUtensorMap tmQ, tmK, tmV, tmDO;
  CUtensorMap tmDQ;       // fp32 [B*Hq][N][d], box 128 rows x 32 columns, 128-byte swizzle
  CUtensorMap tmDK, tmDV;  // fp32 [B*Hkv][N][d], same boxes
  AttnArgs args;
  const float* lse;
  const float* delta;
  float *dQ, *dK, *dV;
  dm_diag diag;
};

// Tensors one quantiser launch processes (same input dtype and d).
struct QuantJob {
  const void* x;
  int N, T_tiles, fmt;
  uint8_t* codes;
  float* scales;
  uint8_t* codes_t;
};
struct QuantBatch {
  static constexpr int kMaxJobs = 8;
  QuantJob job[kMaxJobs];
  int first_tile[kMaxJobs + 1];  // running tile counts; first_tile[count] = total
  int count;
};

cudaError_t launch_quantize(const QuantBatch& b, dm_dtype xt, int d, cudaStream_t st);

// Tensors one prologue launch processes (same input dtype, d and eps).
struct PrologueJob {
  const void* x;
  int N, T_tiles;
  const float* gain;      // nullable
  const float* rope_cos;  // nullable (no rotary embedding)
  const float* rope_sin;
  uint8_t* codes;
  float* scales;
};
struct PrologueBatch {
  static constexpr int kMaxJobs = 4;
  PrologueJob job[kMaxJobs];
  int first_tile[kMaxJobs + 1];
  int count;
  unsigned int* status;  // device status word (bounded waits)
  unsigned long long wait_limit_ns;
};
cudaError_t launch_prologue(const PrologueBatch& b, dm_dtype xt, int d, float eps, cudaStream_t st);
cudaError_t launch_rope_table(int N, int d, double base, float* cos_t, float* sin_t, cudaStream_t st);
// d: the kernel's Q/K head dimension; dv: its V/O head dimension (d, or 128
// with d = 256).
cudaError_t launch_attn_fwd(const FwdLaunch& f, int d, int dv, bool o_bf16, cudaStream_t st);
cudaError_t launch_delta_matched(const DeltaLaunch& f, int d, int dv, cudaStream_t st);
cudaError_t launch_delta_stale(const AttnArgs& a, int d, dm_delta_mode mode, const void* dO, dm_dtype do_t,
                               const uint8_t* do_codes, const void* O, dm_dtype o_t, float* delta,
                               cudaStream_t st);
// FP32 buffers (4-byte aligned) that one launch sets to zero.
struct ZeroList {
  static constexpr int kMax = 8;
  float* p[kMax];
  size_t n[kMax];
  int count;
  void add(float* ptr, size_t len) {
    if (ptr && len) {
      p[count] = ptr;
      n[count] = len;
      ++count;
    }
  }
};

cudaError_t launch_zero(const ZeroList& z, cudaStream_t st);
// Key-block merges (context parallelism), rows = B * Hq * N: O [rows][dv]
// (fp32 or bf16) and LSE from nparts stacked block results; delta from
// nparts stacked (sum P dP^, sum P) pairs.
cudaError_t launch_attn_merge(int nparts, const float* O_parts, const float* lse_parts, long long rows, int dv,
                              void* O, bool o_bf16, float* lse, cudaStream_t st);
cudaError_t launch_delta_combine(int nparts, const float* num_parts, const float* den_parts, long long rows,
                                 float* delta, cudaStream_t st);
cudaError_t launch_attn_bwd(const BwdLaunch& f, int d, cudaStream_t st);

// The checks dm_attn_bwd makes on its problem description and delta mode
// before anything else (DM_OK, DM_ERR_INVALID_ARG or DM_ERR_SHAPE), for entry
// points that wrap it.
dm_status check_attn_problem(const dm_attn_params* p, dm_delta_mode mode);
// Whether the call covers a key block rather than the whole sequence.
bool is_key_block(const dm_attn_params* p);

}  // namespace dm
