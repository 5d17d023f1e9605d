// dm_attn_bwd_noalloc: the backward with the softmax row correction computed
// on the fly, for callers that cannot allocate device memory.
//
// dm_attn_bwd needs a caller-provided workspace to hold delta when it computes
// delta itself.  Some callers have no way to provide one: a training runtime
// that plans every device byte ahead of the step and forbids allocations
// inside it, or a host program that reaches this library only through the C
// ABI and has no device allocator of its own.  This entry point keeps delta in
// a fixed, file-scope device array instead, so the caller passes only its
// inputs and outputs.
//
// The array holds DM_NOALLOC_MAX_DELTA_ROWS floats (8 MiB) on every GPU that
// loads the library, for the life of the process.  All calls share it; each
// call rewrites every delta row it reads before reading it, so nothing has to
// be cleared between calls, but two calls whose kernels overlap on the GPU
// race on it.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "dm_internal.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_delta[DM_NOALLOC_MAX_DELTA_ROWS];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the host-side symbol is only a stand-in for it).
dm_status scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_delta) != cudaSuccess || !ptr) return DM_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<float*>(ptr);
  }
  *out = g_noalloc_ptr[dev];
  return DM_OK;
}

bool aligned_nonnull(const void* ptr) { return ptr && (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// The backward's own pointer requirements, checked before the delta pass is
// launched so that a bad argument launches nothing.
dm_status precheck(const dm_fp8_tensor* t4, const float* lse, float* dQ, float* dK, float* dV, const dm_diag* diag) {
  for (int i = 0; i < 4; ++i) {
    if (!t4[i].codes || !t4[i].scales) return DM_ERR_INVALID_ARG;
    if (!aligned_nonnull(t4[i].codes) || !aligned_nonnull(t4[i].scales)) return DM_ERR_ALIGNMENT;
  }
  for (const void* ptr : {(const void*)lse, (const void*)dQ, (const void*)dK, (const void*)dV}) {
    if (!ptr) return DM_ERR_INVALID_ARG;
    if (!aligned_nonnull(ptr)) return DM_ERR_ALIGNMENT;
  }
  if (diag)
    for (const float* ptr : {diag->rowsum_pre, diag->abssum_pre, diag->rowsum_post, diag->abssum_post})
      if (ptr && !aligned_nonnull(ptr)) return DM_ERR_ALIGNMENT;
  return DM_OK;
}

}  // namespace

extern "C" dm_status dm_attn_bwd_noalloc(const dm_attn_params* p, dm_delta_mode mode, dm_fp8_tensor q,
                                         dm_fp8_tensor k, dm_fp8_tensor v, dm_fp8_tensor do_hat,
                                         const float* lse, const void* dO, dm_dtype do_dtype, const void* O,
                                         dm_dtype o_dtype, float* dQ, float* dK, float* dV, const dm_diag* diag,
                                         void* stream) {
  // the same problem checks as dm_attn_bwd first, so that a bad empty call
  // gets the same status from both entry points
  const dm_status pv = dm::check_attn_problem(p, mode);
  if (pv != DM_OK) return pv;
  if (dm::is_key_block(p)) return DM_ERR_INVALID_ARG;  // a key block needs the merged delta: dm_attn_bwd
  if ((long long)p->B * p->Hq * p->N > (long long)DM_NOALLOC_MAX_DELTA_ROWS) return DM_ERR_SHAPE;
  if (p->B == 0 || p->N == 0) return DM_OK;
  const dm_fp8_tensor t4[4] = {q, k, v, do_hat};
  const dm_status pc = precheck(t4, lse, dQ, dK, dV, diag);
  if (pc != DM_OK) return pc;
  float* delta = nullptr;
  const dm_status s = scratch_for_current_device(&delta);
  if (s != DM_OK) return s;
  const dm_status sd =
      dm_attn_delta(p, mode, q, k, v, do_hat, lse, dO, do_dtype, O, o_dtype, delta, stream);
  if (sd != DM_OK) return sd;
  return dm_attn_bwd(p, mode, q, k, v, do_hat, lse, delta, dO, do_dtype, O, o_dtype, dQ, dK, dV, diag, nullptr,
                     0, stream);
}
