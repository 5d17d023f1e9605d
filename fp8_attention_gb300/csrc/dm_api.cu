// Host side of the C ABI declared in include/dm.h: argument validation, TMA
// descriptor encoding, the device status word, and dispatch to the kernels.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "dm_internal.h"

namespace {

using dm::kDefaultWaitLimitNs;

constexpr int kMaxDevices = 64;
constexpr int kTileRows = 128;

// [0]: DM_OK or the first error a kernel recorded; [1]: site of the first expired wait
__device__ unsigned int g_status_word[2];

std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
unsigned int* g_status_ptr[kMaxDevices] = {};
int g_dev_ok[kMaxDevices] = {};  // 0 unknown, 1 sm_103, -1 other
unsigned long long g_wait_limit_ns = 0;
unsigned int g_last_site = 0;
int g_stall_test = 0;

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks the current device once (sm_103), and looks up the status word's
// device address and the TMA descriptor encoder.
dm_status device_state(unsigned int** status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_dev_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return DM_ERR_CUDA;
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (g_dev_ok[dev] != 1) return DM_ERR_UNSUPPORTED;
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return DM_ERR_CUDA;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
  }
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return DM_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *status = g_status_ptr[dev];
  return DM_OK;
}

// FP8 codes viewed as [BH][N][d]; box = 128 rows x min(kw, 128) bytes with
// the hardware swizzle of that width, kw the kernel's head dimension (a
// kw = 256 row is loaded as two boxes; channels from d to kw lie outside the
// tensor and are read as zeros).
dm_status encode_codes_map(CUtensorMap* m, const uint8_t* codes, int BH, int N, int d, int kw) {
  const int box_x = kw < 128 ? kw : 128;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)d * (cuuint64_t)N};
  cuuint32_t box[3] = {(cuuint32_t)box_x, (cuuint32_t)kTileRows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(codes), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        box_x == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DM_OK : DM_ERR_CUDA;
}

// fp32 [BH][N][d] (dQ), box = 128 rows x 32 columns with the 128-byte swizzle.
dm_status encode_f32_rows_map(CUtensorMap* m, const float* x, int BH, int N, int d) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)d * 4 * (cuuint64_t)N};
  cuuint32_t box[3] = {32, (cuuint32_t)kTileRows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(x), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DM_OK : DM_ERR_CUDA;
}

// bf16 [BH][N][d] (O), box = 128 rows x 64 columns with the 128-byte swizzle.
dm_status encode_bf16_rows_map(CUtensorMap* m, void* x, int BH, int N, int d) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * (cuuint64_t)N};
  cuuint32_t box[3] = {64, (cuuint32_t)kTileRows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DM_OK : DM_ERR_CUDA;
}

// Head dimension of V, dO, O and dV (0 selects d).
inline int value_dim(const dm_attn_params* p) { return p->d_v ? p->d_v : p->d; }

// Rows of K, V, dK and dV: the key block's length (kv_len <= 0: every key
// from kv_offset on; the whole sequence by default).
inline int key_rows(const dm_attn_params* p) { return p->kv_len > 0 ? p->kv_len : p->N - p->kv_offset; }
inline bool key_block(const dm_attn_params* p) { return p->kv_offset != 0 || p->kv_len != 0; }

// The kernels' head dimension: d itself when Q/K and V share one of the
// widths the kernels are built for, else 256 (missing channels read as zeros).
inline int kernel_dim(const dm_attn_params* p) {
  const int dv = value_dim(p);
  return (p->d == dv && p->d != 192) ? p->d : 256;
}

// The forward's and delta pass's V/O head dimension: 128 for a 128-wide V
// beside wider Q/K, else the kernel's head dimension.
inline int kernel_value_dim(const dm_attn_params* p) {
  const int kw = kernel_dim(p);
  return (kw == 256 && value_dim(p) == 128) ? 128 : kw;
}

dm_status check_params(const dm_attn_params* p) {
  if (!p) return DM_ERR_INVALID_ARG;
  if (p->B < 0 || p->Hq <= 0 || p->Hkv <= 0 || p->N < 0) return DM_ERR_SHAPE;
  const int dv = value_dim(p);
  auto wide = [](int x) { return x == 128 || x == 192 || x == 256; };
  if (p->d == dv) {
    if (p->d != 64 && !wide(p->d)) return DM_ERR_SHAPE;
  } else if (!wide(p->d) || !wide(dv)) {
    return DM_ERR_SHAPE;
  }
  if (p->Hq % p->Hkv != 0) return DM_ERR_SHAPE;
  if ((long long)p->B * p->Hq * p->N * (p->d > dv ? p->d : dv) >= (1ll << 31)) return DM_ERR_SHAPE;
  if (!std::isfinite(p->softmax_scale)) return DM_ERR_INVALID_ARG;
  // key block: 128-aligned start inside the sequence, at least one key
  if (p->kv_offset < 0 || p->kv_offset % kTileRows != 0 || p->kv_len < 0) return DM_ERR_SHAPE;
  if (p->N > 0 && (p->kv_offset >= p->N || (long long)p->kv_offset + key_rows(p) > p->N)) return DM_ERR_SHAPE;
  return DM_OK;
}

bool is_empty(const dm_attn_params* p) { return p->B == 0 || p->N == 0; }

dm_status check_fp8(const dm_fp8_tensor& t) {
  if (!t.codes || !t.scales) return DM_ERR_INVALID_ARG;
  if (!aligned16(t.codes) || !aligned16(t.scales)) return DM_ERR_ALIGNMENT;
  return DM_OK;
}

dm_status check_ptr(const void* ptr) {
  if (!ptr) return DM_ERR_INVALID_ARG;
  return aligned16(ptr) ? DM_OK : DM_ERR_ALIGNMENT;
}

bool valid_dtype(dm_dtype t) { return t == DM_F32 || t == DM_BF16; }
bool valid_mode(dm_delta_mode m) {
  return m == DM_DELTA_MATCHED || m == DM_DELTA_STALE_DO || m == DM_DELTA_STALE_DOHAT;
}

// The backward's first key tile taken by CTAs that walk two query heads:
// with a causal mask and an even group size, the key tiles that see at most
// half of the query tiles (all of them up to 32 query tiles, where the
// per-CTA fill and drain weigh more); none otherwise (equal-length CTAs
// would only fill fewer, longer waves).
// The key tiles are counted in the sequence's numbering and the result is
// given in the key block's (Tk tiles from kt_off on).
int bwd_pair_kt(const dm_attn_params* p, int T, int Tk, int kt_off) {
  if (!p->causal || (p->Hq / p->Hkv) % 2 != 0) return Tk;
  const int global = T <= 32 ? 0 : T - T / 2;
  return std::min(Tk, std::max(0, global - kt_off));
}

dm::AttnArgs make_args(const dm_attn_params* p, unsigned int* status) {
  dm::AttnArgs a{};
  a.B = p->B, a.Hq = p->Hq, a.Hkv = p->Hkv, a.N = p->N;
  a.T = (p->N + kTileRows - 1) / kTileRows;
  a.Nk = key_rows(p);
  a.Tk = (a.Nk + kTileRows - 1) / kTileRows;
  a.kt_off = p->kv_offset / kTileRows;
  a.bwd_pair_kt = bwd_pair_kt(p, a.T, a.Tk, a.kt_off);
  a.causal = p->causal ? 1 : 0;
  a.dqk = p->d;
  a.dv = value_dim(p);
  a.sigma = p->softmax_scale > 0.f ? p->softmax_scale : (float)(1.0 / std::sqrt((double)p->d));
  a.status = status;
  std::lock_guard<std::mutex> lock(g_mu);
  a.wait_limit_ns = g_wait_limit_ns ? g_wait_limit_ns : kDefaultWaitLimitNs;
  return a;
}

#define DM_TRY(expr)            \
  do {                          \
    dm_status _s = (expr);      \
    if (_s != DM_OK) return _s; \
  } while (0)

inline dm_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DM_OK : DM_ERR_CUDA; }

dm_status check_delta_inputs(dm_delta_mode mode, dm_fp8_tensor q, dm_fp8_tensor k, dm_fp8_tensor v,
                             dm_fp8_tensor do_hat, const float* lse, const void* dO, dm_dtype do_dtype,
                             const void* O, dm_dtype o_dtype) {
  switch (mode) {
    case DM_DELTA_MATCHED:
      DM_TRY(check_fp8(q));
      DM_TRY(check_fp8(k));
      DM_TRY(check_fp8(v));
      DM_TRY(check_fp8(do_hat));
      DM_TRY(check_ptr(lse));
      return DM_OK;
    case DM_DELTA_STALE_DO:
      DM_TRY(check_ptr(dO));
      DM_TRY(check_ptr(O));
      if (!valid_dtype(do_dtype) || !valid_dtype(o_dtype)) return DM_ERR_DTYPE;
      return DM_OK;
    case DM_DELTA_STALE_DOHAT:
      DM_TRY(check_fp8(do_hat));
      DM_TRY(check_ptr(O));
      if (!valid_dtype(o_dtype)) return DM_ERR_DTYPE;
      return DM_OK;
  }
  return DM_ERR_INVALID_ARG;
}

dm_status delta_impl(const dm_attn_params* p, dm_delta_mode mode, dm_fp8_tensor q, dm_fp8_tensor k,
                     dm_fp8_tensor v, dm_fp8_tensor do_hat, const float* lse, const void* dO, dm_dtype do_dtype,
                     const void* O, dm_dtype o_dtype, float* delta, unsigned int* status, cudaStream_t st,
                     float* den = nullptr, const dm::DeltaClear* clear = nullptr) {
  dm::AttnArgs a = make_args(p, status);
  if (mode == DM_DELTA_MATCHED) {
    dm::DeltaLaunch f{};
    const int kw = kernel_dim(p), dv = value_dim(p);
    DM_TRY(encode_codes_map(&f.tmQ, q.codes, p->B * p->Hq, p->N, p->d, kw));
    DM_TRY(encode_codes_map(&f.tmK, k.codes, p->B * p->Hkv, key_rows(p), p->d, kw));
    DM_TRY(encode_codes_map(&f.tmV, v.codes, p->B * p->Hkv, key_rows(p), dv, kw));
    DM_TRY(encode_codes_map(&f.tmDO, do_hat.codes, p->B * p->Hq, p->N, dv, kw));
    a.q_scales = q.scales, a.k_scales = k.scales, a.v_scales = v.scales, a.do_scales = do_hat.scales;
    f.args = a;
    f.lse = lse;
    f.delta = delta;
    f.den = den;
    if (clear) f.clear = *clear;
    return cuda_status(dm::launch_delta_matched(f, kw, kernel_value_dim(p), st));
  }
  a.do_scales = do_hat.scales;
  return cuda_status(
      dm::launch_delta_stale(a, value_dim(p), mode, dO, do_dtype, do_hat.codes, O, o_dtype, delta, st));
}

}  // namespace

dm_status dm::check_attn_problem(const dm_attn_params* p, dm_delta_mode mode) {
  DM_TRY(check_params(p));
  return valid_mode(mode) ? DM_OK : DM_ERR_INVALID_ARG;
}

bool dm::is_key_block(const dm_attn_params* p) { return key_block(p); }

extern "C" {

int dm_version(void) { return 100; }

const char* dm_status_string(dm_status s) {
  switch (s) {
    case DM_OK: return "DM_OK";
    case DM_ERR_INVALID_ARG: return "DM_ERR_INVALID_ARG";
    case DM_ERR_SHAPE: return "DM_ERR_SHAPE";
    case DM_ERR_DTYPE: return "DM_ERR_DTYPE";
    case DM_ERR_ALIGNMENT: return "DM_ERR_ALIGNMENT";
    case DM_ERR_UNSUPPORTED: return "DM_ERR_UNSUPPORTED";
    case DM_ERR_CUDA: return "DM_ERR_CUDA";
    case DM_ERR_TIMEOUT: return "DM_ERR_TIMEOUT";
  }
  return "DM_ERR_UNKNOWN";
}

dm_status dm_set_knob(dm_knob knob, long long value) {
  if (value < 0) return DM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  switch (knob) {
    case DM_KNOB_WAIT_LIMIT_NS: g_wait_limit_ns = (unsigned long long)value; return DM_OK;
    case DM_KNOB_STALL_TEST: g_stall_test = value ? 1 : 0; return DM_OK;
  }
  return DM_ERR_INVALID_ARG;
}

dm_status dm_get_status(void* stream) {
  unsigned int* status = nullptr;
  DM_TRY(device_state(&status));
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return DM_ERR_CUDA;
  unsigned int v[2] = {0, 0};
  if (cudaMemcpyFromSymbol(v, g_status_word, sizeof(v)) != cudaSuccess) return DM_ERR_CUDA;
  if (v[0] != 0 || v[1] != 0) {
    const unsigned int zero[2] = {0, 0};
    if (cudaMemcpyToSymbol(g_status_word, zero, sizeof(zero)) != cudaSuccess) return DM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    g_last_site = v[1];
  }
  return v[0] == 0 ? DM_OK : (dm_status)v[0];
}

unsigned int dm_last_timeout_site(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  return g_last_site;
}

static_assert(DM_QUANTIZE_MAX_JOBS == dm::QuantBatch::kMaxJobs, "quantiser batch size");
static_assert(DM_PROLOGUE_MAX_JOBS == dm::PrologueBatch::kMaxJobs, "prologue batch size");

namespace {
dm_status check_quantize_job(const dm_quantize_job& j, int d) {
  if (j.fmt != DM_E4M3 && j.fmt != DM_E5M2) return DM_ERR_INVALID_ARG;
  if (j.B < 0 || j.H <= 0 || j.N < 0 || j.d != d) return DM_ERR_SHAPE;
  if ((long long)j.B * j.H * j.N * j.d >= (1ll << 31)) return DM_ERR_SHAPE;
  if (j.B == 0 || j.N == 0) return DM_OK;  // empty tensor: pointers may be NULL
  DM_TRY(check_ptr(j.x));
  DM_TRY(check_ptr(j.codes));
  DM_TRY(check_ptr(j.scales));
  if (j.codes_t && !aligned16(j.codes_t)) return DM_ERR_ALIGNMENT;
  return DM_OK;
}
}  // namespace

dm_status dm_quantize_batch(const dm_quantize_job* jobs, int njobs, dm_dtype x_dtype, void* stream) {
  if (!valid_dtype(x_dtype)) return DM_ERR_DTYPE;
  if (njobs < 0 || njobs > DM_QUANTIZE_MAX_JOBS) return DM_ERR_INVALID_ARG;
  if (njobs == 0) return DM_OK;
  if (!jobs) return DM_ERR_INVALID_ARG;
  const int d = jobs[0].d;
  if (d != 64 && d != 128 && d != 192 && d != 256) return DM_ERR_SHAPE;
  dm::QuantBatch b{};
  long long tiles = 0;
  for (int i = 0; i < njobs; ++i) {
    DM_TRY(check_quantize_job(jobs[i], d));
    if (jobs[i].B == 0 || jobs[i].N == 0) continue;
    dm::QuantJob& q = b.job[b.count];
    q.x = jobs[i].x;
    q.N = jobs[i].N;
    q.T_tiles = (jobs[i].N + 127) / 128;
    q.fmt = jobs[i].fmt == DM_E5M2 ? 1 : 0;
    q.codes = jobs[i].codes;
    q.scales = jobs[i].scales;
    q.codes_t = jobs[i].codes_t;
    b.first_tile[b.count] = (int)tiles;
    tiles += (long long)jobs[i].B * jobs[i].H * q.T_tiles;
    ++b.count;
  }
  if (b.count == 0) return DM_OK;  // every tensor empty
  if (tiles >= (1ll << 31)) return DM_ERR_SHAPE;
  b.first_tile[b.count] = (int)tiles;
  unsigned int* status = nullptr;
  DM_TRY(device_state(&status));
  return cuda_status(dm::launch_quantize(b, x_dtype, d, as_stream(stream)));
}

dm_status dm_quantize(const void* x, dm_dtype x_dtype, int B, int H, int N, int d, dm_fp8 fmt, uint8_t* codes,
                      float* scales, uint8_t* codes_t, void* stream) {
  const dm_quantize_job job{x, B, H, N, d, fmt, codes, scales, codes_t};
  if (d != 64 && d != 128 && d != 192 && d != 256) return valid_dtype(x_dtype) ? DM_ERR_SHAPE : DM_ERR_DTYPE;
  return dm_quantize_batch(&job, 1, x_dtype, stream);
}

namespace {
dm_status check_prologue_job(const dm_prologue_job& j, int d) {
  if (j.B < 0 || j.H <= 0 || j.N < 0 || j.d != d) return DM_ERR_SHAPE;
  if ((long long)j.B * j.H * j.N * j.d >= (1ll << 31)) return DM_ERR_SHAPE;
  if ((j.rope_cos == nullptr) != (j.rope_sin == nullptr)) return DM_ERR_INVALID_ARG;
  if (j.B == 0 || j.N == 0) return DM_OK;  // empty tensor: pointers may be NULL
  DM_TRY(check_ptr(j.x));
  DM_TRY(check_ptr(j.codes));
  DM_TRY(check_ptr(j.scales));
  if (j.gain && !aligned16(j.gain)) return DM_ERR_ALIGNMENT;
  if (j.rope_cos && (!aligned16(j.rope_cos) || !aligned16(j.rope_sin))) return DM_ERR_ALIGNMENT;
  return DM_OK;
}
}  // namespace

dm_status dm_qk_prologue_batch(const dm_prologue_job* jobs, int njobs, dm_dtype x_dtype, float eps, void* stream) {
  if (!valid_dtype(x_dtype)) return DM_ERR_DTYPE;
  if (njobs < 0 || njobs > DM_PROLOGUE_MAX_JOBS) return DM_ERR_INVALID_ARG;
  if (!(eps > 0.0f) || !(eps < INFINITY)) return DM_ERR_INVALID_ARG;
  if (njobs == 0) return DM_OK;
  if (!jobs) return DM_ERR_INVALID_ARG;
  const int d = jobs[0].d;
  if (d != 64 && d != 128 && d != 256) return DM_ERR_SHAPE;
  dm::PrologueBatch b{};
  long long tiles = 0;
  for (int i = 0; i < njobs; ++i) {
    DM_TRY(check_prologue_job(jobs[i], d));
    if (jobs[i].B == 0 || jobs[i].N == 0) continue;
    dm::PrologueJob& q = b.job[b.count];
    q.x = jobs[i].x;
    q.N = jobs[i].N;
    q.T_tiles = (jobs[i].N + 127) / 128;
    q.gain = jobs[i].gain;
    q.rope_cos = jobs[i].rope_cos;
    q.rope_sin = jobs[i].rope_sin;
    q.codes = jobs[i].codes;
    q.scales = jobs[i].scales;
    b.first_tile[b.count] = (int)tiles;
    tiles += (long long)jobs[i].B * jobs[i].H * q.T_tiles;
    ++b.count;
  }
  if (b.count == 0) return DM_OK;
  if (tiles >= (1ll << 31)) return DM_ERR_SHAPE;
  b.first_tile[b.count] = (int)tiles;
  unsigned int* status = nullptr;
  DM_TRY(device_state(&status));
  b.status = status;
  b.wait_limit_ns = g_wait_limit_ns ? g_wait_limit_ns : kDefaultWaitLimitNs;
  return cuda_status(dm::launch_prologue(b, x_dtype, d, eps, as_stream(stream)));
}

dm_status dm_rope_table(int N, int d, double base, float* cos_table, float* sin_table, void* stream) {
  if (N < 0 || d <= 0 || (d % 8)) return DM_ERR_SHAPE;
  if ((long long)N * (d / 2) >= (1ll << 31)) return DM_ERR_SHAPE;
  if (!(base > 1.0) || !(base < INFINITY)) return DM_ERR_INVALID_ARG;
  if (N == 0) return DM_OK;
  DM_TRY(check_ptr(cos_table));
  DM_TRY(check_ptr(sin_table));
  unsigned int* status = nullptr;
  DM_TRY(device_state(&status));
  return cuda_status(dm::launch_rope_table(N, d, base, cos_table, sin_table, as_stream(stream)));
}

dm_status dm_attn_fwd(const dm_attn_params* p, dm_fp8_tensor q, dm_fp8_tensor k, dm_fp8_tensor v, void* O,
                      dm_dtype o_dtype, float* lse, void* stream) {
  DM_TRY(check_params(p));
  if (!valid_dtype(o_dtype)) return DM_ERR_DTYPE;
  if (is_empty(p)) return DM_OK;  // empty input: nothing to do, pointers may be NULL
  DM_TRY(check_fp8(q));
  DM_TRY(check_fp8(k));
  DM_TRY(check_fp8(v));
  DM_TRY(check_ptr(O));
  DM_TRY(check_ptr(lse));
  unsigned int* status = nullptr;
  DM_TRY(device_state(&status));
  dm::FwdLaunch f{};
  const int kw = kernel_dim(p);
  DM_TRY(encode_codes_map(&f.tmQ, q.codes, p->B * p->Hq, p->N, p->d, kw));
  DM_TRY(encode_codes_map(&f.tmK, k.codes, p->B * p->Hkv, key_rows(p), p->d, kw));
  DM_TRY(encode_codes_map(&f.tmV, v.codes, p->B * p->Hkv, key_rows(p), value_dim(p), kw));
  f.args = make_args(p, status);
  f.args.q_scales = q.scales, f.args.k_scales = k.scales, f.args.v_scales = v.scales;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    f.args.stall_test = g_stall_test;
    g_stall_test = 0;
  }
  if (o_dtype == DM_BF16)
    DM_TRY(encode_bf16_rows_map(&f.tmO, O, p->B * p->Hq, p->N, value_dim(p)));
  else
    DM_TRY(encode_f32_rows_map(&f.tmO, static_cast<float*>(O), p->B * p->Hq, p->N, value_dim(p)));
  f.lse = lse;
  return cuda_status(dm::launch_attn_fwd(f, kw, kernel_value_dim(p), o_dtype == DM_BF16, as_stream(stream)));
}

dm_status dm_attn_delta(const dm_attn_params* p, dm_delta_mode mode, dm_fp8_tensor q, dm_fp8_tensor k,
                        dm_fp8_tensor v, dm_fp8_tensor do_hat, const float* lse, const void* dO, dm_dtype do_dtype,
                        const void* O, dm_dtype o_dtype, float* delta, void* stream) {
  DM_TRY(check_params(p));
  if (!valid_mode(mode)) return DM_ERR_INVALID_ARG;
  if (is_empty(p)) return DM_OK;
  DM_TRY(check_delta_inputs(mode, q, k, v, do_hat, lse, dO, do_dtype, O, o_dtype));
  DM_TRY(check_ptr(delta));
  unsigned int* status = nullptr;
  DM_TRY(device_state(&status));
  return delta_impl(p, mode, q, k, v, do_hat, lse, dO, do_dtype, O, o_dtype, delta, status, as_stream(stream));
}

size_t dm_attn_bwd_workspace_size(const dm_attn_params* p) {
  if (check_params(p) != DM_OK) return 0;
  const size_t bytes = (size_t)p->B * p->Hq * p->N * sizeof(float);
  return (bytes + 255) & ~(size_t)255;
}

dm_status dm_attn_bwd(const dm_attn_params* p, dm_delta_mode mode, dm_fp8_tensor q, dm_fp8_tensor k,
                      dm_fp8_tensor v, dm_fp8_tensor do_hat, const float* lse, const float* delta, const void* dO,
                      dm_dtype do_dtype, const void* O, dm_dtype o_dtype, float* dQ, float* dK, float* dV,
                      const dm_diag* diag, void* workspace, size_t workspace_bytes, void* stream) {
  DM_TRY(check_params(p));
  if (!valid_mode(mode)) return DM_ERR_INVALID_ARG;
  if (is_empty(p)) return DM_OK;
  DM_TRY(check_fp8(q));
  DM_TRY(check_fp8(k));
  DM_TRY(check_fp8(v));
  DM_TRY(check_fp8(do_hat));
  DM_TRY(check_ptr(lse));
  DM_TRY(check_ptr(dQ));
  DM_TRY(check_ptr(dK));
  DM_TRY(check_ptr(dV));
  dm_diag dg{};
  if (diag) {
    dg = *diag;
    for (float* ptr : {dg.rowsum_pre, dg.abssum_pre, dg.rowsum_post, dg.abssum_post})
      if (ptr && !aligned16(ptr)) return DM_ERR_ALIGNMENT;
  }
  const float* dl = delta;
  if (delta) {
    DM_TRY(check_ptr(delta));
  } else if (key_block(p)) {
    return DM_ERR_INVALID_ARG;  // a key block's backward needs the merged delta of the whole sequence
  } else {
    DM_TRY(check_delta_inputs(mode, q, k, v, do_hat, lse, dO, do_dtype, O, o_dtype));
    DM_TRY(check_ptr(workspace));
    if (workspace_bytes < dm_attn_bwd_workspace_size(p)) return DM_ERR_INVALID_ARG;
  }
  unsigned int* status = nullptr;
  DM_TRY(device_state(&status));
  cudaStream_t st = as_stream(stream);
  // the backward's tensor maps first: nothing is launched before every
  // argument has passed, these encodings included
  const int kw = kernel_dim(p), dv = value_dim(p);
  const int nk = key_rows(p);
  dm::BwdLaunch f{};
  DM_TRY(encode_codes_map(&f.tmQ, q.codes, p->B * p->Hq, p->N, p->d, kw));
  DM_TRY(encode_codes_map(&f.tmK, k.codes, p->B * p->Hkv, nk, p->d, kw));
  DM_TRY(encode_codes_map(&f.tmV, v.codes, p->B * p->Hkv, nk, dv, kw));
  DM_TRY(encode_codes_map(&f.tmDO, do_hat.codes, p->B * p->Hq, p->N, dv, kw));
  DM_TRY(encode_f32_rows_map(&f.tmDQ, dQ, p->B * p->Hq, p->N, p->d));
  DM_TRY(encode_f32_rows_map(&f.tmDK, dK, p->B * p->Hkv, nk, p->d));
  DM_TRY(encode_f32_rows_map(&f.tmDV, dV, p->B * p->Hkv, nk, dv));
  // dQ, dK and dV are sums of bulk reduce-adds, the diagnostics sums of
  // atomics: all start at zero.  When the matched delta is computed here, its
  // kernel clears them on the way (no key block here: dK and dV have N rows);
  // otherwise one fill launch does.
  const bool clear_in_delta = !delta && mode == DM_DELTA_MATCHED;
  if (!delta) {
    float* ws = static_cast<float*>(workspace);
    const dm::DeltaClear clr{dQ, dK, dV, {dg.rowsum_pre, dg.abssum_pre, dg.rowsum_post, dg.abssum_post}};
    DM_TRY(delta_impl(p, mode, q, k, v, do_hat, lse, dO, do_dtype, O, o_dtype, ws, status, st, nullptr,
                      clear_in_delta ? &clr : nullptr));
    dl = ws;
  }
  if (!clear_in_delta) {
    dm::ZeroList z{};
    z.add(dQ, (size_t)p->B * p->Hq * p->N * p->d);
    z.add(dK, (size_t)p->B * p->Hkv * nk * p->d);
    z.add(dV, (size_t)p->B * p->Hkv * nk * dv);
    const size_t nrow = (size_t)p->B * p->Hq * p->N;
    for (float* ptr : {dg.rowsum_pre, dg.abssum_pre, dg.rowsum_post, dg.abssum_post}) z.add(ptr, nrow);
    DM_TRY(cuda_status(dm::launch_zero(z, st)));
  }
  f.args = make_args(p, status);
  f.args.q_scales = q.scales, f.args.k_scales = k.scales, f.args.v_scales = v.scales;
  f.args.do_scales = do_hat.scales;
  f.lse = lse;
  f.delta = dl;
  f.dQ = dQ, f.dK = dK, f.dV = dV;
  f.diag = dg;
  return cuda_status(dm::launch_attn_bwd(f, kw, st));
}

dm_status dm_attn_delta_partial(const dm_attn_params* p, dm_fp8_tensor q, dm_fp8_tensor k, dm_fp8_tensor v,
                                dm_fp8_tensor do_hat, const float* lse, float* num, float* den, void* stream) {
  DM_TRY(check_params(p));
  if (is_empty(p)) return DM_OK;
  DM_TRY(check_delta_inputs(DM_DELTA_MATCHED, q, k, v, do_hat, lse, nullptr, DM_F32, nullptr, DM_F32));
  DM_TRY(check_ptr(num));
  DM_TRY(check_ptr(den));
  unsigned int* status = nullptr;
  DM_TRY(device_state(&status));
  return delta_impl(p, DM_DELTA_MATCHED, q, k, v, do_hat, lse, nullptr, DM_F32, nullptr, DM_F32, num, status,
                    as_stream(stream), den);
}

dm_status dm_attn_merge(const dm_attn_params* p, int nparts, const float* O_parts, const float* lse_parts, void* O,
                        dm_dtype o_dtype, float* lse, void* stream) {
  DM_TRY(check_params(p));
  if (nparts < 1) return DM_ERR_INVALID_ARG;
  if (!valid_dtype(o_dtype)) return DM_ERR_DTYPE;
  if (is_empty(p)) return DM_OK;
  DM_TRY(check_ptr(O_parts));
  DM_TRY(check_ptr(lse_parts));
  DM_TRY(check_ptr(O));
  DM_TRY(check_ptr(lse));
  const long long rows = (long long)p->B * p->Hq * p->N;
  if (rows * nparts * value_dim(p) >= (1ll << 40)) return DM_ERR_SHAPE;
  unsigned int* status = nullptr;
  DM_TRY(device_state(&status));
  return cuda_status(dm::launch_attn_merge(nparts, O_parts, lse_parts, rows, value_dim(p), O, o_dtype == DM_BF16,
                                           lse, as_stream(stream)));
}

dm_status dm_attn_delta_combine(const dm_attn_params* p, int nparts, const float* num_parts, const float* den_parts,
                                float* delta, void* stream) {
  DM_TRY(check_params(p));
  if (nparts < 1) return DM_ERR_INVALID_ARG;
  if (is_empty(p)) return DM_OK;
  DM_TRY(check_ptr(num_parts));
  DM_TRY(check_ptr(den_parts));
  DM_TRY(check_ptr(delta));
  unsigned int* status = nullptr;
  DM_TRY(device_state(&status));
  return cuda_status(dm::launch_delta_combine(nparts, num_parts, den_parts, (long long)p->B * p->Hq * p->N, delta,
                                              as_stream(stream)));
}

}  // extern "C"
