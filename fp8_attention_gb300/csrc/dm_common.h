// Definitions shared by the host API and the kernels of libdm.
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/dm.h"

namespace dm {

constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;  // 2 s


// Arguments common to the attention kernels (all device pointers).
struct AttnArgs {
  int B, Hq, Hkv, N, T;      // T = ceil(N / 128)
  int dqk, dv;               // head dimensions of Q/K and of V/dO/O; the kernel's
                             // width may be larger (missing channels read as zeros)
  int causal;
  float sigma;               // softmax scale
  const float* q_scales;     // [B][Hq][T]
  const float* k_scales;     // [B][Hkv][T]
  const float* v_scales;     // [B][Hkv][T]
  const float* do_scales;    // [B][Hq][T]
  unsigned int* status;      // device status word
  unsigned long long wait_limit_ns;
  int stall_test;            // 1: the MMA warp waits on a barrier nothing signals
  int bwd_pair_kt;           // backward: key tiles from this one on are taken by CTAs
                             // that walk two query heads of a group (Tk: none)
  // Key block: K, V (and dK, dV) hold Nk rows, the keys at sequence positions
  // [128 * kt_off, 128 * kt_off + Nk); key tile t of the block is global key
  // tile t + kt_off.  The whole sequence: Nk = N, Tk = T, kt_off = 0.
  int Nk, Tk, kt_off;
};

}  // namespace dm
