/*
 * dm.h -- C ABI of libdm: FP8 flash attention with the Delta-Matching
 * softmax correction, for one NVIDIA GB300 (sm_103a).
 *
 * Method: "Delta-Matching for reliable FP8 attention training" (project
 * page).  Section 01 ("Write down softmax backward") defines the attention
 * forward S = sigma*Q*K^T, P = softmax_row(S), O = P*V and its backward
 * dV = P^T dO, dP = dO V^T, dS = P o (dP - delta), dQ = sigma*dS*K,
 * dK = sigma*dS^T*Q with the row correction delta_i.  Section 01 ("What
 * changes in FP8?") puts every matmul on decoded block-scaled FP8 operands
 * with FP32 accumulation; section 03 defines the matched correction
 * delta_i = sum_j P_ij * dP^_ij, with P the FP32 softmax before it is
 * quantised and dP^ the FP32 result of the FP8 product dO^ V^T.  The two
 * stale corrections, <dO_i, O_i> (section 01) and <dO^_i, O_i> (section 03,
 * last paragraph), are kept as diagnostic modes.
 *
 * Conventions shared by every call
 *  - Tensors are contiguous row-major [B][H][N][d] (d fastest).  Query heads
 *    are Hq, key/value heads Hkv; query head h reads kv head h / (Hq/Hkv).
 *  - Every pointer is DEVICE memory owned by the caller, except `p`/`diag`
 *    struct pointers, which are host memory read during the call.  The library
 *    allocates no memory and keeps no state between calls other than the TMA
 *    entry point it looks up once, a device status word, and the fixed 8 MiB
 *    device array that dm_attn_bwd_noalloc keeps delta in (on every GPU that
 *    loads the library, until the process exits).
 *  - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and is asynchronous; the call returns after the launches.
 *    Stream order holds as usual.  The forward and delta kernels are launched
 *    with programmatic stream serialisation: their blocks may be scheduled
 *    while the previous kernel of the stream finishes, but they touch no
 *    memory until it has completed.  The quantiser, forward and delta kernels
 *    allow a following kernel that was itself launched that way to be
 *    scheduled early; such a kernel must wait (griddepcontrol.wait) before it
 *    reads their outputs.
 *  - Arguments are validated before any launch.  On an error nothing is
 *    launched and no output is touched.
 *  - FP8 tensors (dm_fp8_tensor) hold codes uint8 [B][H][N][d] and one FP32
 *    scale per 128-row x d tile, scales float [B][H][ceil(N/128)]; the decoded
 *    value of a code is scale * value(code).
 *  - Supported shapes: d = d_v in {64, 128, 192, 256}, or d != d_v with both in
 *    {128, 192, 256} (see dm_attn_params); any N >= 0 (ragged tails are masked);
 *    Hq % Hkv == 0; B*Hq*N*d < 2^31.  B == 0 or N == 0 is a valid no-op.
 *  - Device pointers must be 16-byte aligned.
 *  - The device must be compute capability 10.3 (sm_103a build).
 *
 * Precision contract (the pages leave these steps open; this is the reading
 * implemented and checked against the CPU oracle):
 *  - tile quantiser: amax = max|x| over the tile; if amax < 2^-96 the tile
 *    gets scale 0 and all-zero codes; else s = amax/FMAX, r = FMAX/amax (IEEE
 *    fp32 divisions), code = RNE_satfinite(fp32(x*r)); FMAX = 448 (E4M3) or
 *    57344 (E5M2);
 *  - forward P is quantised in one pass: key tiles in ascending order,
 *    P~ = exp(S - running row max) in FP32, one E4M3 scale per 128x128 tile
 *    of P~, the row sum l taken from the unquantised P~;
 *  - backward P = exp(S - LSE) in FP32, quantised E4M3 per 128x128 tile;
 *    dS = P*(dP^ - delta) in FP32, quantised E5M2 per 128x128 tile;
 *  - the P~, P and dS tiles never leave the chip, and their scales are formed
 *    with a hardware reciprocal (r = FMAX/amax to within 2 ulp, s = amax *
 *    (1/FMAX)) instead of IEEE divisions, and the forward forms P~ * r as one
 *    base-2 exponential exp2(S*c - m + log2 r): a code of these tiles can
 *    differ from the oracle's where P~ * r lies within FP32 rounding of a code
 *    boundary (the Q, K, V and dO codes of dm_quantize are bit-exact);
 *  - accumulator units: each key tile (forward) or query tile (backward)
 *    contributes in units of its own scale product; a tile adds nothing when
 *    one of its scales is zero (a flushed tile) or when its contribution is
 *    below 2^-64 of the accumulator's current unit in every row.  dQ is exact
 *    down to sigma * s_dS * s_K >= 2^-126 (the FP32 normal range of one
 *    iteration's dQ unit); the forward's O stays finite while the V tiles one
 *    query row sees have scales within about 2^90 of each other.
 */
#ifndef DM_H_
#define DM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DM_OK = 0,
  DM_ERR_INVALID_ARG = 1, /* null pointer, bad enum value, bad flag */
  DM_ERR_SHAPE = 2,       /* unsupported or inconsistent B/H/N/d */
  DM_ERR_DTYPE = 3,       /* dtype not accepted for that argument */
  DM_ERR_ALIGNMENT = 4,   /* a device pointer is not 16-byte aligned */
  DM_ERR_UNSUPPORTED = 5, /* device is not sm_103, or feature not built */
  DM_ERR_CUDA = 6,        /* a CUDA runtime/driver call or launch failed */
  DM_ERR_TIMEOUT = 7      /* a kernel's bounded wait expired (see dm_get_status) */
} dm_status;

typedef enum { DM_F32 = 0, DM_BF16 = 1 } dm_dtype;
typedef enum { DM_E4M3 = 0, DM_E5M2 = 1 } dm_fp8;
typedef enum {
  DM_DELTA_MATCHED = 0,    /* delta_i = sum_j P_ij dP^_ij (section 03)          */
  DM_DELTA_STALE_DO = 1,   /* delta_i = <dO_i, O_i>, dO before its FP8 cast      */
  DM_DELTA_STALE_DOHAT = 2 /* delta_i = <dO^_i, O_i>, "match dO only" (sec. 03)  */
} dm_delta_mode;

/* Problem description.  causal: key j visible to query i iff j <= i.
 * softmax_scale: sigma in S = sigma*Q*K^T; <= 0 selects 1/sqrt(d).
 * d is the head dimension of Q, K, dQ and dK; d_v that of V, dO, O and dV
 * (0 selects d).  They may differ (heads shaped like multi-head latent
 * attention, e.g. d = 192, d_v = 128) when both are 128, 192 or 256; such
 * heads run on the d = 256 kernels, which read the missing channels as
 * zeros and write only the real ones.
 *
 * Key block (context parallelism over the sequence; the project page's
 * section 06 extends the context from 8K to 64K tokens and does not say how
 * the sequence is split): with kv_offset or kv_len set, a call sees only the
 * keys at sequence positions [kv_offset, kv_offset + kv_len) (kv_len <= 0:
 * up to N), and K, V, dK, dV hold just those kv_len rows ([B][Hkv][kv_len][.],
 * scales [B][Hkv][ceil(kv_len/128)]); queries, dO, O, LSE, delta and dQ keep
 * all N rows.  kv_offset is a multiple of 128 (the key tiles then are the
 * sequence's own, so K and V quantised by block match the whole tensor's
 * codes and scales), 0 <= kv_offset < N and kv_offset + kv_len <= N.  Both 0
 * (a zero-initialised struct) is the whole sequence. */
typedef struct {
  int B, Hq, Hkv, N, d;
  int causal;
  float softmax_scale;
  int d_v;
  int kv_offset, kv_len;
} dm_attn_params;

/* A block-scaled FP8 tensor: codes [B][H][N][d], scales [B][H][ceil(N/128)]. */
typedef struct {
  const uint8_t* codes;
  const float* scales;
} dm_fp8_tensor;

/* Optional per-query-row dS diagnostics, each float [B][Hq][N] (any may be
 * NULL): sum_j dS_ij and sum_j |dS_ij| before the E5M2 cast, and the same two
 * sums of the decoded dS^ after it (project page section 03: the post-cast
 * row-sum residual). */
typedef struct {
  float* rowsum_pre;
  float* abssum_pre;
  float* rowsum_post;
  float* abssum_post;
} dm_diag;

/* dm_quantize -- per-tile FP8 quantisation (block scales of section 01,
 * "What changes in FP8?").  x: [B][H][N][d] of x_dtype (DM_F32 or DM_BF16).
 * fmt: DM_E4M3 (Q, K, V) or DM_E5M2 (dO).  Writes codes [B][H][N][d], scales
 * [B][H][ceil(N/128)], and, if codes_t != NULL, the codes transposed per
 * (b, h) as [B][H][d][N].  Bit-exact with the tile quantiser rule above. */
dm_status dm_quantize(const void* x, dm_dtype x_dtype, int B, int H, int N, int d, dm_fp8 fmt,
                      uint8_t* codes, float* scales, uint8_t* codes_t, void* stream);

/* dm_quantize_batch -- dm_quantize of up to DM_QUANTIZE_MAX_JOBS tensors in one
 * launch (the pages quantise Q, K, V and dO with the same rule; one launch
 * avoids a short kernel per tensor).  All jobs share x_dtype and d; fmt,
 * shapes and buffers are per job, with the meaning, layout and ownership of
 * dm_quantize.  Every job is validated before the launch (DM_ERR_SHAPE if the
 * jobs' d differ, DM_ERR_INVALID_ARG for njobs outside 0..MAX or jobs == NULL
 * with njobs > 0); empty tensors are skipped.  Results are bit-identical to
 * separate dm_quantize calls. */
#define DM_QUANTIZE_MAX_JOBS 8
typedef struct {
  const void* x;
  int B, H, N, d;
  dm_fp8 fmt;
  uint8_t* codes;
  float* scales;
  uint8_t* codes_t; /* nullable */
} dm_quantize_job;
dm_status dm_quantize_batch(const dm_quantize_job* jobs, int njobs, dm_dtype x_dtype, void* stream);

/* dm_rope_table -- cos and sin of the rotary angles theta(n, i) = n *
 * base^(-2i/d), n < N, i < d/2, written as float [N][d/2] each (row n = the
 * sequence position), computed in FP64 on the device and rounded to FP32.
 * The pages' models use RoPE (project page, section 05, "Attention variants
 * change when failure appears", where removing it is the NoPE variant) but
 * give no base; 10000 is the usual one.  d must be a multiple of 8 (so rows
 * stay 16-byte aligned), base > 1; the caller owns both tables (16-byte
 * aligned).  DM_ERR_SHAPE / DM_ERR_INVALID_ARG / DM_ERR_ALIGNMENT on bad
 * arguments, before any launch. */
dm_status dm_rope_table(int N, int d, double base, float* cos_table, float* sin_table, void* stream);

/* dm_qk_prologue_batch -- the attention-input prologue of a QK-normalised
 * rotary model fused with the tile quantiser, for up to
 * DM_PROLOGUE_MAX_JOBS tensors (typically Q and K) in one launch.  The pages'
 * models normalise queries and keys with RMSNorm and learned per-channel
 * gains (project page, section 02: the gains are the quantity that drifts
 * under stale delta) before attention.  Per row of x ([B][H][N][d] of x_dtype,
 * DM_F32 or DM_BF16, row n = sequence position n):
 *   y_k = x_k / sqrt(mean_k x_k^2 + eps) * gain_k     (gain [d] float shared by
 *                                                      the heads; NULL = ones)
 *   if rope_cos: channel i < d/2 and channel i + d/2 rotate by theta(n, i):
 *     (a, b) <- (a cos - b sin, b cos + a sin), cos/sin from rope_cos/rope_sin
 *     ([N][d/2] float, e.g. from dm_rope_table; both or neither)
 * then y is quantised to E4M3 with the rule of dm_quantize (one FP32 scale per
 * 128-row x d tile): codes [B][H][N][d], scales [B][H][ceil(N/128)], ready
 * for dm_attn_fwd.  All arithmetic is FP32 (correctly rounded 1/sqrt), so
 * codes can differ from an exact evaluation only where y * (448 / amax) lies
 * within FP32 rounding of a code boundary.  All jobs share x_dtype, d (64,
 * 128 or 256) and eps (finite, > 0); x, codes, scales, gain and the tables are
 * 16-byte aligned.  Every job is validated before the launch;
 * empty tensors are skipped.  Errors: DM_ERR_DTYPE, DM_ERR_SHAPE,
 * DM_ERR_INVALID_ARG (njobs out of range, bad eps, one table without the
 * other), DM_ERR_ALIGNMENT. */
#define DM_PROLOGUE_MAX_JOBS 4
typedef struct {
  const void* x;
  int B, H, N, d;
  const float* gain;     /* nullable */
  const float* rope_cos; /* nullable */
  const float* rope_sin; /* nullable */
  uint8_t* codes;
  float* scales;
} dm_prologue_job;
dm_status dm_qk_prologue_batch(const dm_prologue_job* jobs, int njobs, dm_dtype x_dtype, float eps, void* stream);

/* dm_attn_fwd -- O = P^ V^ and LSE (section 01).  q, k, v: E4M3 tensors of
 * shapes [B][Hq][N][d], [B][Hkv][N][d], [B][Hkv][N][d_v].  O: [B][Hq][N][d_v]
 * of o_dtype (DM_F32 or DM_BF16).  lse: float [B][Hq][N], natural log of the
 * softmax denominator including the scale sigma, i.e. LSE_i = ln sum_j
 * exp(S_ij).  O and LSE are the only saved forward outputs.  Over a key block
 * (see dm_attn_params) O and LSE are the block's own attention (its one-pass
 * quantisation starting at the block's first key tile); a row that sees no
 * key of the block gets O = 0 and LSE = -inf.  dm_attn_merge combines blocks. */
dm_status dm_attn_fwd(const dm_attn_params* p, dm_fp8_tensor q, dm_fp8_tensor k, dm_fp8_tensor v,
                      void* O, dm_dtype o_dtype, float* lse, void* stream);

/* dm_attn_delta -- the softmax row correction, float delta [B][Hq][N].
 * dO, do_hat and O are [B][Hq][N][d_v].
 *  DM_DELTA_MATCHED:     needs q, k, v, do_hat (E5M2), lse; recomputes S and
 *                        dP^ = dO^ V^T tile by tile in FP32 (the separate
 *                        correction pass).  dO and O may be NULL.  Over a key
 *                        block: the block's own correction (for the blocks of
 *                        one sequence use dm_attn_delta_partial).
 *  DM_DELTA_STALE_DO:    needs dO (do_dtype) and O (o_dtype).
 *  DM_DELTA_STALE_DOHAT: needs do_hat and O (o_dtype).  */
dm_status dm_attn_delta(const dm_attn_params* p, dm_delta_mode mode, dm_fp8_tensor q, dm_fp8_tensor k,
                        dm_fp8_tensor v, dm_fp8_tensor do_hat, const float* lse, const void* dO,
                        dm_dtype do_dtype, const void* O, dm_dtype o_dtype, float* delta,
                        void* stream);

/* dm_attn_bwd -- dQ, dK, dV (section 01) with the five backward matmuls in
 * FP8.  delta: float [B][Hq][N] from dm_attn_delta, or NULL, in which case it
 * is computed first for `mode` into `workspace` (which then needs
 * dm_attn_bwd_workspace_size(p) bytes, 16-byte aligned, and must not overlap
 * the outputs or the diagnostics buffers).  dQ float
 * [B][Hq][N][d] (overwritten, not accumulated), dK float [B][Hkv][N][d] and
 * dV float [B][Hkv][N][d_v] (summed over each kv head's query heads).  diag: optional
 * row-sum diagnostics (NULL = off).  dO/O are needed only when delta is NULL
 * and the mode is stale.  The outputs start at zero inside the call (with
 * delta NULL and the matched mode, the delta kernel clears them on its way;
 * otherwise one fill launch does).  Over a key block: lse and delta must be the whole
 * sequence's (merged; delta NULL gives DM_ERR_INVALID_ARG), dK and dV are the
 * block's rows ([B][Hkv][kv_len][.]) and dQ and diag hold the block's partial
 * sums (the blocks' dQ add up to the sequence's). */
dm_status dm_attn_bwd(const dm_attn_params* p, dm_delta_mode mode, dm_fp8_tensor q, dm_fp8_tensor k,
                      dm_fp8_tensor v, dm_fp8_tensor do_hat, const float* lse, const float* delta,
                      const void* dO, dm_dtype do_dtype, const void* O, dm_dtype o_dtype, float* dQ,
                      float* dK, float* dV, const dm_diag* diag, void* workspace,
                      size_t workspace_bytes, void* stream);

/* Bytes of workspace dm_attn_bwd needs when delta == NULL (0 on bad params). */
size_t dm_attn_bwd_workspace_size(const dm_attn_params* p);

/* dm_attn_bwd_noalloc -- dm_attn_bwd with delta computed for `mode`, for
 * callers that cannot allocate device memory and so cannot hand
 * dm_attn_bwd a workspace: a training runtime that plans every device byte
 * ahead of the step and forbids allocations inside it, or a host program that
 * reaches this library only through this C ABI with no device allocator of its
 * own.  The method's pages have no counterpart to this call; it exists only
 * for such callers.  A key block (dm_attn_params) is rejected with
 * DM_ERR_INVALID_ARG: its delta must be the merged one of the whole sequence.
 *
 * Arguments are those of dm_attn_bwd without delta and workspace.  delta is
 * kept in a fixed device array of DM_NOALLOC_MAX_DELTA_ROWS floats (8 MiB),
 * held on every GPU that loads the library until the process exits; problems
 * with B*Hq*N above that limit are rejected with DM_ERR_SHAPE before anything
 * is launched.  The call allocates nothing.  Its first call on a device looks
 * up that array's device address (once per device, with the device current);
 * make that first call before any stream capture.  All calls on a device
 * share that device's array, which keeps the last call's contents: each call
 * rewrites every delta row before reading it, so nothing needs clearing, but
 * calls whose kernels overlap on the same GPU (for example on two streams)
 * race on it and must be serialised by the caller. */
#define DM_NOALLOC_MAX_DELTA_ROWS (1u << 21)
dm_status dm_attn_bwd_noalloc(const dm_attn_params* p, dm_delta_mode mode, dm_fp8_tensor q, dm_fp8_tensor k,
                              dm_fp8_tensor v, dm_fp8_tensor do_hat, const float* lse, const void* dO,
                              dm_dtype do_dtype, const void* O, dm_dtype o_dtype, float* dQ, float* dK,
                              float* dV, const dm_diag* diag, void* stream);

/* dm_attn_delta_partial -- the two sums of the matched correction over a key
 * block (section 03's delta_i = sum_j P_ij dP^_ij / sum_j P_ij, split by key
 * blocks so that the blocks of one sequence add up before the division):
 * num_i = sum_{j in block} P_ij dP^_ij and den_i = sum_{j in block} P_ij, each
 * float [B][Hq][N] (0 for a row that sees no key of the block), with P =
 * exp(S - LSE) from the whole sequence's (merged) lse.  Arguments as
 * dm_attn_delta in DM_DELTA_MATCHED mode.  dm_attn_delta_combine divides. */
dm_status dm_attn_delta_partial(const dm_attn_params* p, dm_fp8_tensor q, dm_fp8_tensor k, dm_fp8_tensor v,
                                dm_fp8_tensor do_hat, const float* lse, float* num, float* den, void* stream);

/* dm_attn_merge -- the attention of every query row over the union of nparts
 * disjoint key blocks from the blocks' own results (dm_attn_fwd over each):
 * LSE_i = ln sum_r exp(LSE_r,i) and O_i = sum_r exp(LSE_r,i - LSE_i) O_r,i.
 * O_parts: float [nparts][B][Hq][N][d_v] (the blocks' fp32 O, stacked, e.g. by
 * an all-gather), lse_parts: float [nparts][B][Hq][N]; O: [B][Hq][N][d_v] of
 * o_dtype (DM_F32 or DM_BF16), lse: float [B][Hq][N].  Blocks with LSE = -inf
 * weigh zero; a row that no block sees gets O = 0 and LSE = -inf.  p gives B,
 * Hq, N and d_v (its key block is ignored).  Errors: DM_ERR_INVALID_ARG
 * (nparts < 1, NULL pointer), DM_ERR_DTYPE, DM_ERR_ALIGNMENT, DM_ERR_SHAPE. */
dm_status dm_attn_merge(const dm_attn_params* p, int nparts, const float* O_parts, const float* lse_parts, void* O,
                        dm_dtype o_dtype, float* lse, void* stream);

/* dm_attn_delta_combine -- delta_i = sum_r num_r,i / sum_r den_r,i from
 * nparts stacked dm_attn_delta_partial results (num_parts and den_parts each
 * float [nparts][B][Hq][N]; nparts = 1 after the sums were reduced across
 * devices), 0 where every den is 0.  delta: float [B][Hq][N].  p gives B, Hq
 * and N.  Errors as dm_attn_merge. */
dm_status dm_attn_delta_combine(const dm_attn_params* p, int nparts, const float* num_parts, const float* den_parts,
                                float* delta, void* stream);

/* Synchronises `stream`, then returns and clears the device status word of
 * the current device: DM_ERR_TIMEOUT if a kernel's bounded wait expired since
 * the last call (its outputs are then undefined), DM_ERR_CUDA if the stream
 * reports an error, else DM_OK. */
dm_status dm_get_status(void* stream);

/* Where the last DM_ERR_TIMEOUT reported by dm_get_status came from:
 * kernel * 100 + wait number (kernel 1 forward, 2 delta pass, 3 backward),
 * 0 if no wait has expired.  A diagnostic for bug reports. */
unsigned int dm_last_timeout_site(void);

/* Human-readable name of a status code (static string). */
const char* dm_status_string(dm_status s);

/* Library version, 100*major + minor. */
int dm_version(void);

/* Test and debug knobs (process-wide, default 0):
 *  DM_KNOB_WAIT_LIMIT_NS: limit of every bounded wait inside the kernels in
 *                         nanoseconds (0 = built-in default of 2 s);
 *  DM_KNOB_STALL_TEST:    1 makes the next dm_attn_fwd launch wait on a barrier
 *                         that nothing signals, so that its bounded wait
 *                         expires and the kernel returns DM_ERR_TIMEOUT
 *                         through dm_get_status (used to test the watchdog;
 *                         the knob resets itself after that launch). */
typedef enum { DM_KNOB_WAIT_LIMIT_NS = 0, DM_KNOB_STALL_TEST = 1 } dm_knob;
dm_status dm_set_knob(dm_knob knob, long long value);

#ifdef __cplusplus
}
#endif

#endif /* DM_H_ */
