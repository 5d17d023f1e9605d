// Device-side building blocks for the sm_103a kernels: mbarriers with bounded
// waits, TMA tile loads, tcgen05 (TMEM allocation, FP8 MMA, TMEM loads and
// stores), shared-memory matrix descriptors, and packed FP8 conversions.
// Everything is inline PTX written from the PTX ISA; no CUTLASS/CuTe.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "dm_common.h"

namespace dm {

constexpr int kTile = 128;  // rows of a query/key tile and of an MMA M dimension

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// A waiting thread is suspended in hardware until the phase completes or the
// hint (in ns) runs out, instead of spinning on the issue slots that the
// other warps of its SM sub-partition need.
constexpr uint32_t kSuspendHintNs = 1000000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "n"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Watchdog shared by all waits of one CTA.  Every wait is bounded: after
// `limit_ns` without progress the waiting thread records DM_ERR_TIMEOUT in the
// device status word and raises the CTA's abort flag; from then on every wait
// of the CTA returns immediately, so all roles run their (counted) loops to
// the end without blocking and the kernel exits normally.
// status[0] holds the status code, status[1] the site id (kernel * 100 + wait
// number) of the first wait that expired.
struct Watchdog {
  volatile int* abort_flag;  // shared memory
  unsigned int* status;      // global status words [2]
  unsigned long long limit_ns;
};

static __device__ __noinline__ void record_timeout(const Watchdog& wd, unsigned int site) {
  *wd.abort_flag = 1;
  atomicCAS(wd.status, 0u, (unsigned)DM_ERR_TIMEOUT);
  atomicCAS(wd.status + 1, 0u, site);
  __threadfence();
}

static __device__ __noinline__ bool wait_slow(uint64_t* bar, uint32_t parity, const Watchdog& wd,
                                              unsigned int site) {
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*wd.abort_flag) return false;
    if (globaltimer() - t0 > wd.limit_ns) {
      record_timeout(wd, site);
      return false;
    }
  }
}

// Returns true when the phase with `parity` completed, false on abort.
__device__ __forceinline__ bool wait(uint64_t* bar, uint32_t parity, const Watchdog& wd, unsigned int site) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, wd, site);
}

// Wait bounded only by time (not by the abort flag): used at teardown so that
// a CTA never exits while its own TMA copies or MMAs are still in flight.
static __device__ __noinline__ bool wait_drain(uint64_t* bar, uint32_t parity, const Watchdog& wd,
                                               unsigned int site) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > wd.limit_ns) {
      record_timeout(wd, site);
      return false;
    }
  return true;
}

// ----------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load: coordinates (c0 innermost, c1, c2) in elements.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Plain bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Bulk tensor reduce-add of a shared-memory tile into global memory (the
// element type and the add come from the tensor map); completion is tracked by
// the issuing thread's bulk async-groups.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Tile store of a shared-memory box into a 3-D tensor (rows past the
// tensor's extent are not written).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the source shared memory of every committed group has been read
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every committed group has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T with FP8 operands, FP32 accumulation.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier tracks completion of all prior tcgen05 async ops of this thread.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Instruction descriptor for kind::f8f6f4 with FP32 accumulator.
//   bits 4-5 D format (1 = F32), 7-9 A format, 10-12 B format (0 = E4M3,
//   1 = E5M2), 15 A major, 16 B major (0 = K-major, 1 = MN-major),
//   17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_f8(uint32_t a_fmt, uint32_t b_fmt, uint32_t a_mn, uint32_t b_mn,
                                                uint32_t M, uint32_t N) {
  return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}

// Shared-memory matrix descriptor (tcgen05 format): start address >> 4 in
// bits 0-13, leading-dimension byte offset >> 4 in 16-29, stride-dimension
// byte offset >> 4 in 32-45, fixed 0b001 in 46-48, swizzle mode in 61-63
// (2 = 128-byte, 4 = 64-byte).
enum : uint32_t { kSwizzle128 = 2, kSwizzle64 = 4 };
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | ((uint64_t)swz << 61);
}

// A [rows][row_bytes] FP8 tile in shared memory, rows contiguous, written by
// TMA (or by threads) with the hardware swizzle of width row_bytes (128 or
// 64).  Two views:
//  * K-major: MMA rows = tile rows, K = the row's bytes.  K step k (32 FP8
//    elements) starts 32*k bytes into the row.
//  * MN-major: MMA M/N = the row's bytes, K = tile rows.  K step k starts at
//    row 32*k.
// In both views 8 rows form one swizzle atom (SBO = 8 * row_bytes).
template <int ROW_BYTES>
struct SwTile {
  static_assert(ROW_BYTES == 128 || ROW_BYTES == 64, "row width");
  static constexpr uint32_t kSwz = ROW_BYTES == 128 ? kSwizzle128 : kSwizzle64;
  static constexpr uint32_t kSbo = 8 * ROW_BYTES;
  __device__ static uint64_t kmajor(uint32_t base, int kstep) {
    return smem_desc(base + 32u * kstep, 16u, kSbo, kSwz);
  }
  __device__ static uint64_t mnmajor(uint32_t base, int kstep) {
    return smem_desc(base + 32u * ROW_BYTES * kstep, 16u * 1024u, kSbo, kSwz);
  }
  // Byte offset of 16-byte chunk `c` of row `r` (for threads writing the
  // tile): the swizzle XORs address bits [4, 4+b) with bits [7, 7+b), b = 3
  // for 128-byte rows and 2 for 64-byte rows (tile base 1024-byte aligned).
  __device__ static uint32_t chunk_offset(int r, int c) {
    const uint32_t a = (uint32_t)(r * ROW_BYTES + c * 16);
    constexpr uint32_t kMask = ROW_BYTES == 128 ? 7u : 3u;
    return a ^ (((a >> 7) & kMask) << 4);
  }
  // The same with the row part hoisted: chunk c of row r sits at
  // row_base(r) ^ 16 c, also after adding a 1024-byte aligned tile offset to
  // row_base (which leaves bits [4, 7) alone), so a thread writing its row
  // pays one XOR per chunk.
  __device__ static uint32_t row_base(int r) {
    constexpr uint32_t kMask = ROW_BYTES == 128 ? 7u : 3u;
    return (uint32_t)r * ROW_BYTES | (((uint32_t)r & kMask) << 4);
  }
};

// An FP8 [128][D] operand tile for D = 64, 128 or 256.  The 128-byte swizzle
// spans at most 128 bytes of a row, so D = 256 is held as two [128][128]
// sub-tiles, d columns 0-127 then 128-255, kSubBytes apart (each loaded by its
// own TMA box).
//  * K-major (K = d): K step k lies in sub-tile k / 4.
//  * MN-major (N = d): the sub-tiles are the swizzle atoms along N, and the
//    descriptor's leading byte offset (16 KB in SwTile<128>) steps between
//    them.
template <int D>
struct OpTile {
  static_assert(D == 64 || D == 128 || D == 256, "head dimension");
  static constexpr int kRowBytes = D > 128 ? 128 : D;
  static constexpr int kSubTiles = D / kRowBytes;
  static constexpr uint32_t kSubBytes = (uint32_t)kTile * kRowBytes;
  static constexpr int kStepsPerSub = kRowBytes / 32;
  __device__ static uint64_t kmajor(uint32_t base, int kstep) {
    return SwTile<kRowBytes>::kmajor(base + (uint32_t)(kstep / kStepsPerSub) * kSubBytes, kstep % kStepsPerSub);
  }
  __device__ static uint64_t mnmajor(uint32_t base, int kstep) {
    static_assert(kSubTiles == 1 || kSubBytes == 16u * 1024u, "sub-tile stride = leading byte offset");
    return SwTile<kRowBytes>::mnmajor(base, kstep);
  }
};

// Loads rows [row, row + 128) of plane `plane` of a [planes][N][D] FP8 tensor
// (map box: 128 rows x min(D, 128) bytes) as OpTile<D>; completes on `bar`
// (kTile * D bytes in all).
template <int D>
__device__ __forceinline__ void tma_load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int row,
                                              int plane) {
#pragma unroll
  for (int s = 0; s < OpTile<D>::kSubTiles; ++s)
    tma_load_3d(dst + s * OpTile<D>::kSubBytes, map, bar, s * OpTile<D>::kRowBytes, row, plane);
}

// 32 lanes x 32 consecutive 32-bit columns.  Lane quarter of the warp is
// (warp_id % 4); taddr must carry that lane base in bits 16+.
// Each load below issues tcgen05.ld and tcgen05.wait::ld in one statement:
// the destination registers are written asynchronously, and a separate wait
// statement would leave the compiler free to read (or copy) them before the
// wait.  Stores likewise wait in the same statement.
__device__ __forceinline__ void tmem_load32(uint32_t taddr, float (&v)[32]) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// Two 32-column loads (v[0..31] from taddr0, v[32..63] from taddr1), one wait.
__device__ __forceinline__ void tmem_load64(uint32_t taddr0, uint32_t taddr1, float (&v)[64]) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr0), "r"(taddr1)
      : "memory");
}
// Four 32-column loads (v[32k..32k+31] from taddr_k), one wait.
__device__ __forceinline__ void tmem_load128(uint32_t t0, uint32_t t1, uint32_t t2, uint32_t t3, float (&v)[128]) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%129];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%130];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%131];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(t0), "r"(t1), "r"(t2), "r"(t3)
      : "memory");
}
// Four 32-column stores (the counterpart of tmem_load128), one wait.
__device__ __forceinline__ void tmem_store128(uint32_t t0, uint32_t t1, uint32_t t2, uint32_t t3,
                                              const float (&v)[128]) {
  const uint32_t* r = reinterpret_cast<const uint32_t*>(v);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35};\n\t"
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%1], {%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67};\n\t"
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%2], {%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99};\n\t"
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%3], {%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127,%128,%129,%130,%131};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(t0), "r"(t1), "r"(t2), "r"(t3),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63]), "r"(r[64]), "r"(r[65]), "r"(r[66]), "r"(r[67]), "r"(r[68]), "r"(r[69]), "r"(r[70]), "r"(r[71]), "r"(r[72]), "r"(r[73]), "r"(r[74]), "r"(r[75]), "r"(r[76]), "r"(r[77]), "r"(r[78]), "r"(r[79]), "r"(r[80]), "r"(r[81]), "r"(r[82]), "r"(r[83]), "r"(r[84]), "r"(r[85]), "r"(r[86]), "r"(r[87]), "r"(r[88]), "r"(r[89]), "r"(r[90]), "r"(r[91]), "r"(r[92]), "r"(r[93]), "r"(r[94]), "r"(r[95]), "r"(r[96]), "r"(r[97]), "r"(r[98]), "r"(r[99]), "r"(r[100]), "r"(r[101]), "r"(r[102]), "r"(r[103]), "r"(r[104]), "r"(r[105]), "r"(r[106]), "r"(r[107]), "r"(r[108]), "r"(r[109]), "r"(r[110]), "r"(r[111]), "r"(r[112]), "r"(r[113]), "r"(r[114]), "r"(r[115]), "r"(r[116]), "r"(r[117]), "r"(r[118]), "r"(r[119]), "r"(r[120]), "r"(r[121]), "r"(r[122]), "r"(r[123]), "r"(r[124]), "r"(r[125]), "r"(r[126]), "r"(r[127])
      : "memory");
}
__device__ __forceinline__ void tmem_store32(uint32_t taddr, const float (&v)[32]) {
  const uint32_t* r = reinterpret_cast<const uint32_t*>(v);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// ------------------------------------------------------------------ numerics
// Four FP32 values -> four FP8 codes (round to nearest even, saturating),
// byte k of the result holds value k.
__device__ __forceinline__ uint32_t pack4_e4m3(float x0, float x1, float x2, float x3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  return r;
}
__device__ __forceinline__ uint32_t pack4_e5m2(float x0, float x1, float x2, float x3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e5m2x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e5m2x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  return r;
}
template <int FMT>
__device__ __forceinline__ uint32_t pack4(float x0, float x1, float x2, float x3) {
  return FMT == 0 ? pack4_e4m3(x0, x1, x2, x3) : pack4_e5m2(x0, x1, x2, x3);
}

// Two FP8 codes (low byte first) -> two exact FP32 values, via f16x2.
template <int FMT>
__device__ __forceinline__ float2 unpack2(uint16_t codes) {
  uint32_t h2;
  if (FMT == 0)
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
  else
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(codes));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Tile quantiser scale rule (see dm.h): returns s and sets r; s = r = 0 when
// the tile is flushed.
template <int FMT>
__device__ __forceinline__ float tile_scale(float amax, float& r) {
  constexpr float kFmax = FMT == 0 ? 448.0f : 57344.0f;
  if (!(amax >= 0x1p-96f)) {
    r = 0.0f;
    return 0.0f;
  }
  r = __fdiv_rn(kFmax, amax);
  return __fdiv_rn(amax, kFmax);
}

// Scale rule for tiles that stay on chip (P^, dS^): the same rule with a
// hardware reciprocal instead of IEEE divisions.  The codes only feed the
// tensor core, so a last-place difference in r moves a code only when P r
// sits within one ulp of a rounding boundary.
template <int FMT>
__device__ __forceinline__ float tile_scale_fast(float amax, float& r) {
  constexpr float kFmax = FMT == 0 ? 448.0f : 57344.0f;
  if (!(amax >= 0x1p-96f)) {
    r = 0.0f;
    return 0.0f;
  }
  r = __fdividef(kFmax, amax);
  return amax * (1.0f / kFmax);
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// Largest of a non-negative, non-NaN value over the warp in one integer
// reduction: such floats (+0 included, -0 not) order like their bit patterns
// read as unsigned integers.
__device__ __forceinline__ float warp_max_nonneg(float v) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}
// Largest value over the warp, of any sign (-inf included, no NaN), in one
// integer reduction: the bit patterns are first mapped to unsigned integers
// in the same order (negative values complemented, the sign bit set on the
// others) and mapped back after.
__device__ __forceinline__ float warp_max_any(float v) {
  const uint32_t u = __float_as_uint(v);
  const uint32_t m = __reduce_max_sync(0xffffffffu, (u & 0x80000000u) ? ~u : (u | 0x80000000u));
  return __uint_as_float((m & 0x80000000u) ? (m & 0x7fffffffu) : ~m);
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace dm
