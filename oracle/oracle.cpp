// CPU oracle for Delta-Matching FP8 attention.  TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, FP64 restatement of what the GPU path computes, written from
// the project page "Delta-Matching for reliable FP8 attention training"
// (sections 01-03) and from the quantisation contract stated below.  Only the
// test suite, the smoke check and the benchmark's CPU-baseline leg load this
// library; the product path never does.  It shares no code, header, table or
// constant with the CUDA sources.
//
// Conventions
//   * every tensor is contiguous [B][H][N][d] (d fastest); row i = query,
//     j = key, k = value channel; kv head of query head h is h / (Hq/Hkv);
//   * causal means key j is visible to query i iff j <= i;
//   * tiles are 128 rows (query or key), so tile t covers rows [128t, 128t+128)
//     clipped to N;
//   * the decoded FP8 operands (codes times their tile scale) are passed in as
//     FP64 arrays; quantising them is a separate call (or_quantize), exactly as
//     the GPU path quantises Q, K, V and dO before the attention calls.
//
// Parity pins (tests/test_oracle_*.py): the FP8 codec against torch's CPU
// float8 casts and exhaustive decode; exact-mode forward/backward against
// central finite differences and torch autograd in FP64; the identities of
// sections 01-03 (saved-output shortcut, zero row sum, shift invariance, the
// two-term split of the stale residual, dS_stale = dS_centered + eps*P); the
// backward's P^ / dS^ tile quantisation and the multi-tile one-pass forward
// against independent torch-cast emulations on exact grid inputs
// (tests/test_oracle_tile_pins.py); the attention-input prologue against textbook rotary values, the rotation as
// complex multiplication, the relative-position property and the RMSNorm
// invariants (tests/test_oracle_prologue.py).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <cstddef>
#include <vector>
#include <algorithm>
#include <limits>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

constexpr int kTile = 128;

// ---------------------------------------------------------------------------
// OFP8 formats (OCP 8-bit floating point specification v1.0).  The pages name
// E4M3 for the forward and E5M2 for the backward ("Delta-Matching Reports FP8
// LLM Training Parity...", section "The correction preserves FP8 through
// attention"); the bit layouts below are the OCP definitions.
//   E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa; no infinities;
//                S.1111.111 is NaN; largest finite 448; smallest subnormal 2^-9.
//   E5M2:        1 sign, 5 exponent (bias 15), 2 mantissa; IEEE-like inf/NaN;
//                largest finite 57344; smallest subnormal 2^-16.
struct Fp8Fmt {
  int ebits, mbits, bias;
  double fmax;
};
const Fp8Fmt kFmt[2] = {{4, 3, 7, 448.0}, {5, 2, 15, 57344.0}};

double fp8_decode(uint8_t c, int f) {
  const Fp8Fmt& F = kFmt[f];
  const int sign = c >> 7;
  const int e = (c >> F.mbits) & ((1 << F.ebits) - 1);
  const int m = c & ((1 << F.mbits) - 1);
  const int emax_field = (1 << F.ebits) - 1;
  double v;
  if (f == 0 && e == emax_field && m == (1 << F.mbits) - 1) {
    return std::numeric_limits<double>::quiet_NaN();
  } else if (f == 1 && e == emax_field) {
    v = m ? std::numeric_limits<double>::quiet_NaN()
          : std::numeric_limits<double>::infinity();
  } else if (e == 0) {
    v = std::ldexp((double)m, 1 - F.bias - F.mbits);  // subnormal
  } else {
    v = std::ldexp((double)((1 << F.mbits) + m), e - F.bias - F.mbits);
  }
  return sign ? -v : v;
}

// Round-to-nearest-even from the exact fp32 value onto the format's grid,
// saturating to the largest finite magnitude (satfinite); NaN stays NaN.
uint8_t fp8_encode(float x, int f) {
  const Fp8Fmt& F = kFmt[f];
  if (std::isnan(x)) return 0x7F;
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  double a = std::fabs((double)x);
  const int emin = 1 - F.bias;  // exponent of the smallest normal
  if (a >= F.fmax) {
    a = F.fmax;
  } else if (a > 0.0) {
    int e2;
    std::frexp(a, &e2);                       // a = f * 2^e2, f in [0.5, 1)
    const int E = std::max(e2 - 1, emin);     // binade of a (normal or subnormal)
    const double quantum = std::ldexp(1.0, E - F.mbits);
    a = std::nearbyint(a / quantum) * quantum;  // ties to even (default mode)
    if (a > F.fmax) a = F.fmax;
  }
  if (a == 0.0) return sign;
  int e2;
  std::frexp(a, &e2);
  const int E = e2 - 1;
  uint8_t code;
  if (E < emin) {
    code = (uint8_t)(a / std::ldexp(1.0, emin - F.mbits));  // subnormal field
  } else {
    const int mant = (int)(a / std::ldexp(1.0, E - F.mbits)) - (1 << F.mbits);
    code = (uint8_t)(((E + F.bias) << F.mbits) | mant);
  }
  return code | sign;
}

// Tile quantiser Qz: one FP32 scale per tile, derived from the tile's amax.
// The pages name per-block scales but give no rule (project page, section 01,
// "What changes in FP8?"); the rule used here is the plain amax rule:
//   amax = max |x| over the tile (exact),
//   if amax < 2^-96 (zero, subnormal or tiny tile): scale 0, all codes +0,
//   else s = fl32(amax / FMAX), r = fl32(FMAX / amax), code = enc(fl32(x * r)).
// The decoded value is s * dec(code).  `valid(i, j)` selects the tile entries
// that exist (ragged edges, causal mask); absent entries get code 0.
template <class Get, class Valid>
float qz_tile(int rows, int cols, int f, Get get, Valid valid, uint8_t* codes /*rows*cols*/) {
  float amax = 0.0f;
  for (int i = 0; i < rows; ++i)
    for (int j = 0; j < cols; ++j)
      if (valid(i, j)) {
        const float a = std::fabs(get(i, j));
        if (a > amax) amax = a;
      }
  if (!(amax >= 0x1p-96f)) {
    std::memset(codes, 0, (size_t)rows * cols);
    return 0.0f;
  }
  const float fmax = (float)kFmt[f].fmax;
  const float s = amax / fmax;
  const float r = fmax / amax;
  for (int i = 0; i < rows; ++i)
    for (int j = 0; j < cols; ++j) {
      const float xr = valid(i, j) ? get(i, j) * r : 0.0f;
      codes[(size_t)i * cols + j] = fp8_encode(xr, f);
    }
  return s;
}

inline float fl32(double x) { return (float)x; }

// d is the query/key head dimension, dv the value head dimension (V, dO, O
// and dV rows); they differ for heads shaped like multi-head latent attention.
struct Dims {
  int B, Hq, Hkv, N, d, dv, causal;
  double sigma;
  int kb = 0, ke = 0;  // key range [kb, ke): the keys this call sees (ke = N: all)
  int G() const { return Hq / Hkv; }
  int T() const { return (N + kTile - 1) / kTile; }
  size_t qoff(int b, int h) const { return ((size_t)b * Hq + h) * N * d; }
  size_t kvoff(int b, int g) const { return ((size_t)b * Hkv + g) * N * d; }
  size_t qvoff(int b, int h) const { return ((size_t)b * Hq + h) * N * dv; }
  size_t kvvoff(int b, int g) const { return ((size_t)b * Hkv + g) * N * dv; }
  size_t rowoff(int b, int h) const { return ((size_t)b * Hq + h) * N; }
};

bool visible(const Dims& D, int i, int j) { return j >= D.kb && j < D.ke && (!D.causal || j <= i); }

double dot(const double* a, const double* b, int n) {
  double s = 0.0;
  for (int k = 0; k < n; ++k) s += a[k] * b[k];
  return s;
}

// Selection helpers: a NULL list selects every tile.
std::vector<int> tiles_or_all(const int* sel, int n, int T) {
  std::vector<int> v;
  if (!sel) {
    for (int t = 0; t < T; ++t) v.push_back(t);
  } else {
    for (int k = 0; k < n; ++k)
      if (sel[k] >= 0 && sel[k] < T) v.push_back(sel[k]);
  }
  return v;
}

struct Group { int b, g; };
std::vector<Group> groups_or_all(const int* sel /*pairs b,g*/, int n, const Dims& D) {
  std::vector<Group> v;
  if (!sel) {
    for (int b = 0; b < D.B; ++b)
      for (int g = 0; g < D.Hkv; ++g) v.push_back({b, g});
  } else {
    for (int k = 0; k < n; ++k) v.push_back({sel[2 * k], sel[2 * k + 1]});
  }
  return v;
}

// Scores of one (query tile, key tile) pair: S_ij = sigma * <Q_i, K_j>.
void score_tile(const Dims& D, const double* Qh, const double* Kg, int qt, int kt,
                std::vector<double>& S, int& rows, int& cols) {
  const int i0 = qt * kTile, j0 = kt * kTile;
  rows = std::min(kTile, D.N - i0);
  cols = std::min(kTile, D.N - j0);
  S.assign((size_t)rows * cols, 0.0);
  for (int r = 0; r < rows; ++r)
    for (int c = 0; c < cols; ++c)
      if (visible(D, i0 + r, j0 + c))
        S[(size_t)r * cols + c] = D.sigma * dot(Qh + (size_t)(i0 + r) * D.d, Kg + (size_t)(j0 + c) * D.d, D.d);
}

// Key tiles a query tile sees: [first_key_tile, last_key_tile] (empty when
// first > last).
int first_key_tile(const Dims& D) { return D.kb / kTile; }
int last_key_tile(const Dims& D, int qt) {
  const int last = (D.ke - 1) / kTile;
  return D.causal ? std::min(qt, last) : last;
}

// Key range [kb, ke) of a call: kv_end <= 0 selects every key from kv_begin on.
bool set_key_range(Dims& D, int kv_begin, int kv_end) {
  D.kb = kv_begin;
  D.ke = kv_end > 0 ? kv_end : D.N;
  return kv_begin >= 0 && D.ke <= D.N && (D.N == 0 || kv_begin < D.ke);
}

}  // namespace

extern "C" {

enum {
  OR_QUANT_P_FWD = 1,   // quantise the forward probabilities P~ per 128x128 tile (E4M3)
  OR_QUANT_P_BWD = 2,   // quantise the backward probabilities P per 128x128 tile (E4M3)
  OR_QUANT_DS = 4,      // quantise dS per 128x128 tile (E5M2)
  OR_ROUND32 = 8,       // round P~, P and dS to FP32 where the GPU holds them in FP32
};
enum { OR_DELTA_MATCHED = 0, OR_DELTA_STALE_DO = 1, OR_DELTA_STALE_DOHAT = 2 };

double or_fp8_decode(uint8_t code, int fmt) { return fp8_decode(code, fmt); }
uint8_t or_fp8_encode(float x, int fmt) { return fp8_encode(x, fmt); }

// Elementwise encode of n fp32 values (used by the exhaustive codec test).
void or_fp8_encode_array(const float* x, int64_t n, int fmt, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < n; ++k) out[k] = fp8_encode(x[k], fmt);
}

// Quantise a [B][H][N][d] fp32 tensor with one scale per 128-row x d tile.
// codes: [B][H][N][d] uint8, scales: [B][H][ceil(N/128)] float.
int or_quantize(const float* x, int B, int H, int N, int d, int fmt, uint8_t* codes, float* scales) {
  if (fmt < 0 || fmt > 1 || B < 0 || H < 0 || N < 0 || d <= 0) return 1;
  const int T = (N + kTile - 1) / kTile;
  const int64_t units = (int64_t)B * H * T;
#pragma omp parallel for schedule(dynamic)
  for (int64_t u = 0; u < units; ++u) {
    const int64_t bh = u / T;
    const int t = (int)(u % T);
    const int rows = std::min(kTile, N - t * kTile);
    const float* xt = x + ((size_t)bh * N + (size_t)t * kTile) * d;
    uint8_t* ct = codes + ((size_t)bh * N + (size_t)t * kTile) * d;
    scales[bh * T + t] = qz_tile(
        rows, d, fmt, [&](int i, int j) { return xt[(size_t)i * d + j]; },
        [](int, int) { return true; }, ct);
  }
  return 0;
}

// Decoded value s * dec(code) of a quantised [B][H][N][d] tensor, in FP64.
void or_dequantize(const uint8_t* codes, const float* scales, int B, int H, int N, int d, int fmt, double* out) {
  const int T = (N + kTile - 1) / kTile;
  const int64_t rows = (int64_t)B * H * N;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const int64_t bh = r / N;
    const int n = (int)(r % N);
    const double s = scales[bh * T + n / kTile];
    for (int k = 0; k < d; ++k) out[r * d + k] = s * fp8_decode(codes[r * d + k], fmt);
  }
}

// ---------------------------------------------------------------------------
// Forward (project page, section 01, "Write down softmax backward" for the
// definition S = sigma Q K^T, P = softmax_row(S), O = P V; "What changes in
// FP8?" for O = P^ V^).  sigma <= 0 selects 1/sqrt(d) (the pages do not print
// the scale; the standard one is used).
//
// Without OR_QUANT_P_FWD this is the plain definition, row by row, in FP64.
// With it, the probabilities are quantised the only way a one-pass kernel can
// (the pages leave this step open; their analysis takes P as normalised so
// that only the rounding of the operands enters): key tiles t = 0, 1, ... in ascending order, running row max
// m^(t), P~_ij = exp(S_ij - m^(t)_i) (rounded to FP32 under OR_ROUND32),
// P~ quantised per 128x128 tile (E4M3), l_i accumulated from the unquantised
// P~, and earlier partial sums rescaled by exp(m^(t-1) - m^(t)).  Then
// O_i = acc_i / l_i and LSE_i = m_i + ln l_i.
//
// Pfwd (nullable, [B][Hq][N][N]) receives the effective forward
// probabilities, i.e. the matrix with O = Pfwd V exactly.
//
// Key range [kv_begin, kv_end) (kv_end <= 0: to N): the attention of every
// query row over those keys only, a key block of context-parallel attention
// (project page section 06 extends the context from 8K to 64K tokens; the
// pages do not say how the sequence is split).  A row that sees none of them
// gets O = 0 and LSE = -inf.  The one-pass quantised forward walks the range's
// key tiles only, so its running maximum starts at the block's first tile.
int or_attn_fwd(int B, int Hq, int Hkv, int N, int d, int dv, int causal, double sigma, int flags,
                const double* Q, const double* K, const double* V,
                const int* q_tiles, int n_q_tiles, const int* groups, int n_groups,
                double* O, double* LSE, double* Pfwd, int kv_begin, int kv_end) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || N < 0 || d <= 0 || dv <= 0) return 1;
  Dims D{B, Hq, Hkv, N, d, dv, causal, sigma > 0 ? sigma : 1.0 / std::sqrt((double)d)};
  if (!set_key_range(D, kv_begin, kv_end)) return 1;
  const int T = D.T();
  const std::vector<int> qts = tiles_or_all(q_tiles, n_q_tiles, T);
  const std::vector<Group> gs = groups_or_all(groups, n_groups, D);
  const int G = D.G();
  const int64_t units = (int64_t)gs.size() * G * qts.size();
#pragma omp parallel for schedule(dynamic)
  for (int64_t u = 0; u < units; ++u) {
    const Group gr = gs[u / ((int64_t)G * qts.size())];
    const int h = gr.g * G + (int)((u / qts.size()) % G);
    const int qt = qts[u % qts.size()];
    const double* Qh = Q + D.qoff(gr.b, h);
    const double* Kg = K + D.kvoff(gr.b, gr.g);
    const double* Vg = V + D.kvvoff(gr.b, gr.g);
    double* Oh = O + D.qvoff(gr.b, h);
    double* Lh = LSE + D.rowoff(gr.b, h);
    double* Ph = Pfwd ? Pfwd + ((size_t)gr.b * Hq + h) * N * N : nullptr;
    const int i0 = qt * kTile;
    const int rows = std::min(kTile, N - i0);
    const int ktmax = last_key_tile(D, qt);

    if (!(flags & OR_QUANT_P_FWD)) {
      std::vector<double> s(N);
      for (int r = 0; r < rows; ++r) {
        const int i = i0 + r;
        double m = -INFINITY;
        for (int j = 0; j < N; ++j)
          if (visible(D, i, j)) {
            s[j] = D.sigma * dot(Qh + (size_t)i * d, Kg + (size_t)j * d, d);
            m = std::max(m, s[j]);
          }
        double l = 0.0;
        for (int j = 0; j < N; ++j)
          if (visible(D, i, j)) l += std::exp(s[j] - m);
        for (int k = 0; k < dv; ++k) Oh[(size_t)i * dv + k] = 0.0;
        if (l == 0.0) {  // no visible key
          Lh[i] = -INFINITY;
          if (Ph)
            for (int j = 0; j < N; ++j) Ph[(size_t)i * N + j] = 0.0;
          continue;
        }
        for (int j = 0; j < N; ++j) {
          const double p = visible(D, i, j) ? std::exp(s[j] - m) / l : 0.0;
          if (Ph) Ph[(size_t)i * N + j] = p;
          if (p != 0.0)
            for (int k = 0; k < dv; ++k) Oh[(size_t)i * dv + k] += p * Vg[(size_t)j * dv + k];
        }
        Lh[i] = m + std::log(l);
      }
      continue;
    }

    // One-pass online forward with per-tile quantisation of P~.
    std::vector<double> m(rows, -INFINITY), l(rows, 0.0), acc((size_t)rows * dv, 0.0);
    const int ktmin = first_key_tile(D);
    std::vector<double> mt((size_t)std::max(ktmax + 1, 1) * rows);  // m^(t) per tile, for Pfwd
    std::vector<double> S;
    std::vector<float> pt;
    std::vector<uint8_t> codes;
    for (int kt = ktmin; kt <= ktmax; ++kt) {
      int rr, cols;
      score_tile(D, Qh, Kg, qt, kt, S, rr, cols);
      const int j0 = kt * kTile;
      std::vector<double> mnew(rows);
      for (int r = 0; r < rows; ++r) {
        double mx = m[r];
        for (int c = 0; c < cols; ++c)
          if (visible(D, i0 + r, j0 + c)) mx = std::max(mx, S[(size_t)r * cols + c]);
        mnew[r] = mx;
      }
      pt.assign((size_t)rows * cols, 0.0f);
      std::vector<double> pd((size_t)rows * cols, 0.0);
      for (int r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c)
          if (visible(D, i0 + r, j0 + c)) {
            const double p = std::exp(S[(size_t)r * cols + c] - mnew[r]);
            pd[(size_t)r * cols + c] = (flags & OR_ROUND32) ? (double)fl32(p) : p;
            pt[(size_t)r * cols + c] = fl32(p);
          }
      codes.resize((size_t)rows * cols);
      auto valid = [&](int r, int c) { return visible(D, i0 + r, j0 + c); };
      const float sP = qz_tile(rows, cols, 0, [&](int r, int c) { return (float)pd[(size_t)r * cols + c]; },
                               valid, codes.data());
      for (int r = 0; r < rows; ++r) {
        const double alpha = std::exp(m[r] - mnew[r]);  // exp(-inf) = 0 on the first tile
        double rowsum = 0.0;
        for (int c = 0; c < cols; ++c) rowsum += pd[(size_t)r * cols + c];
        l[r] = alpha * l[r] + rowsum;
        double* a = &acc[(size_t)r * dv];
        for (int k = 0; k < dv; ++k) a[k] *= alpha;
        for (int c = 0; c < cols; ++c) {
          const double ph = (double)sP * fp8_decode(codes[(size_t)r * cols + c], 0);
          if (Ph) Ph[(size_t)(i0 + r) * N + j0 + c] = ph;  // finalised below
          if (ph != 0.0)
            for (int k = 0; k < dv; ++k) a[k] += ph * Vg[(size_t)(j0 + c) * dv + k];
        }
        m[r] = mnew[r];
        mt[(size_t)kt * rows + r] = mnew[r];
      }
    }
    for (int r = 0; r < rows; ++r) {
      const int i = i0 + r;
      if (l[r] == 0.0) {  // no visible key
        for (int k = 0; k < dv; ++k) Oh[(size_t)i * dv + k] = 0.0;
        Lh[i] = -INFINITY;
        if (Ph)
          for (int j = 0; j < N; ++j) Ph[(size_t)i * N + j] = 0.0;
        continue;
      }
      for (int k = 0; k < dv; ++k) Oh[(size_t)i * dv + k] = acc[(size_t)r * dv + k] / l[r];
      Lh[i] = m[r] + std::log(l[r]);
      if (Ph) {
        for (int j = 0; j < std::min(N, ktmin * kTile); ++j) Ph[(size_t)i * N + j] = 0.0;
        for (int kt = ktmin; kt <= ktmax; ++kt) {
          const double w = std::exp(mt[(size_t)kt * rows + r] - m[r]) / l[r];
          for (int c = 0; c < std::min(kTile, N - kt * kTile); ++c)
            Ph[(size_t)i * N + kt * kTile + c] *= w;
        }
        for (int j = (ktmax + 1) * kTile; j < N; ++j) Ph[(size_t)i * N + j] = 0.0;
      }
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Softmax row correction delta (project page sections 01 and 03).
//   matched      (section 03): delta_i = sum_j P_ij dP^_ij / sum_j P_ij with
//                P the FP32 softmax before quantisation, P_ij = exp(S_ij -
//                LSE_i), and dP^ = dO^ V^T accumulated exactly over the decoded
//                operands.  Section 03 cancels the row sum of dS by using that
//                each row of P sums to one; P in FP32 with a stored FP32 LSE sums to
//                1 + eta, and the division makes the cancellation hold for the
//                P the backward uses (no change when P sums to 1 exactly);
//   stale_dO     (section 01, "Why can we reuse the forward output?" and
//                "What changes in FP8?"): delta_i = <dO_i, O_i>, dO before
//                its FP8 cast, O as stored by the forward;
//   stale_dOhat  (section 03, last paragraph): delta_i = <dO^_i, O_i>.
// LSE is the stored forward value (the caller rounds it to FP32).
//
// Key range [kv_begin, kv_end) (matched mode): the sums run over those keys
// only.  With den != NULL the two sums are returned apart, delta_i = sum_j
// P_ij dP^_ij and den_i = sum_j P_ij (0 for a row that sees none of the keys),
// so that the blocks of a split key range add up before the one division.
int or_attn_delta(int B, int Hq, int Hkv, int N, int d, int dv, int causal, double sigma, int flags, int mode,
                  const double* Q, const double* K, const double* V, const double* dOhat,
                  const double* dO, const double* O, const double* LSE,
                  const int* q_tiles, int n_q_tiles, const int* groups, int n_groups, double* delta,
                  int kv_begin, int kv_end, double* den) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || N < 0 || d <= 0 || dv <= 0 || mode < 0 || mode > 2) return 1;
  Dims D{B, Hq, Hkv, N, d, dv, causal, sigma > 0 ? sigma : 1.0 / std::sqrt((double)d)};
  if (!set_key_range(D, kv_begin, kv_end)) return 1;
  if (den && mode != OR_DELTA_MATCHED) return 1;
  const std::vector<int> qts = tiles_or_all(q_tiles, n_q_tiles, D.T());
  const std::vector<Group> gs = groups_or_all(groups, n_groups, D);
  const int G = D.G();
  const int64_t units = (int64_t)gs.size() * G * qts.size();
#pragma omp parallel for schedule(dynamic)
  for (int64_t u = 0; u < units; ++u) {
    const Group gr = gs[u / ((int64_t)G * qts.size())];
    const int h = gr.g * G + (int)((u / qts.size()) % G);
    const int qt = qts[u % qts.size()];
    const size_t qo = D.qoff(gr.b, h), ko = D.kvoff(gr.b, gr.g), ro = D.rowoff(gr.b, h);
    const size_t qvo = D.qvoff(gr.b, h), kvo = D.kvvoff(gr.b, gr.g);
    const int i0 = qt * kTile, rows = std::min(kTile, N - i0);
    for (int r = 0; r < rows; ++r) {
      const int i = i0 + r;
      double dl = 0.0;
      if (mode == OR_DELTA_STALE_DO) {
        dl = dot(dO + qvo + (size_t)i * dv, O + qvo + (size_t)i * dv, dv);
      } else if (mode == OR_DELTA_STALE_DOHAT) {
        dl = dot(dOhat + qvo + (size_t)i * dv, O + qvo + (size_t)i * dv, dv);
      } else {
        double psum = 0.0;
        for (int j = 0; j < N; ++j) {
          if (!visible(D, i, j)) continue;
          const double s = D.sigma * dot(Q + qo + (size_t)i * d, K + ko + (size_t)j * d, d);
          double p = std::exp(s - LSE[ro + i]);
          if (flags & OR_ROUND32) p = fl32(p);
          const double dp = dot(dOhat + qvo + (size_t)i * dv, V + kvo + (size_t)j * dv, dv);
          dl += p * dp;
          psum += p;
        }
        if (den)
          den[ro + i] = psum;
        else
          dl /= psum;
      }
      delta[ro + i] = dl;
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Backward (project page section 01, "Write down softmax backward", and
// section 03): per (query tile, key tile) pair
//   P_ij   = exp(S_ij - LSE_i)           (FP32 under OR_ROUND32)
//   P^     = Qz_E4M3(P) per 128x128 tile (OR_QUANT_P_BWD)
//   dP^_ij = <dO^_i, V^_j>
//   dS_ij  = P_ij (dP^_ij - delta_i)     (FP32 under OR_ROUND32)
//   dS^    = Qz_E5M2(dS) per 128x128 tile (OR_QUANT_DS)
//   dV_j  += sum_i P^_ij dO^_i ;  dQ_i += sigma sum_j dS^_ij K^_j ;
//   dK_j  += sigma sum_i dS^_ij Q^_i
// dK and dV of a kv head sum over the query heads of its group.
// dQ (and the row-sum diagnostics) are written for the selected query tiles,
// dK/dV for the selected key tiles, within the selected (b, kv head) groups.
// diag (nullable) is [4][B][Hq][N]: sum_j dS, sum_j |dS|, sum_j dS^, sum_j |dS^|.
// dS, dShat, Phat (nullable, [B][Hq][N][N]) receive the tiles computed for
// the selected query tiles (small test cases only).
//
// Key range [kv_begin, kv_end): only those keys take part; dQ (and the
// diagnostics) are then the block's partial sums, and dK, dV of keys outside
// the range are zero.
int or_attn_bwd(int B, int Hq, int Hkv, int N, int d, int dv, int causal, double sigma, int flags,
                const double* Q, const double* K, const double* V, const double* dOhat,
                const double* LSE, const double* delta,
                const int* q_tiles, int n_q_tiles, const int* kv_tiles, int n_kv_tiles,
                const int* groups, int n_groups,
                double* dQ, double* dK, double* dV, double* diag,
                double* dS_out, double* dShat_out, double* Phat_out, int kv_begin, int kv_end) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || N < 0 || d <= 0 || dv <= 0) return 1;
  Dims D{B, Hq, Hkv, N, d, dv, causal, sigma > 0 ? sigma : 1.0 / std::sqrt((double)d)};
  if (!set_key_range(D, kv_begin, kv_end)) return 1;
  const int T = D.T(), G = D.G();
  const std::vector<int> qts = tiles_or_all(q_tiles, n_q_tiles, T);
  const std::vector<int> kts = tiles_or_all(kv_tiles, n_kv_tiles, T);
  const std::vector<Group> gs = groups_or_all(groups, n_groups, D);

  // All tile-level quantities of one (b, h, qt, kt) pair.
  struct PairTile {
    int rows = 0, cols = 0;
    std::vector<double> P, Ph, dS, dSh;
  };
  auto compute_pair = [&](int b, int h, int qt, int kt, PairTile& pt) {
    const int g = h / G;
    const double* Qh = Q + D.qoff(b, h);
    const double* Kg = K + D.kvoff(b, g);
    const double* Vg = V + D.kvvoff(b, g);
    const double* dOh = dOhat + D.qvoff(b, h);
    const double* Lh = LSE + D.rowoff(b, h);
    const double* dl = delta + D.rowoff(b, h);
    std::vector<double> S;
    score_tile(D, Qh, Kg, qt, kt, S, pt.rows, pt.cols);
    const int rows = pt.rows, cols = pt.cols, i0 = qt * kTile, j0 = kt * kTile;
    auto valid = [&](int r, int c) { return visible(D, i0 + r, j0 + c); };
    pt.P.assign((size_t)rows * cols, 0.0);
    pt.dS.assign((size_t)rows * cols, 0.0);
    for (int r = 0; r < rows; ++r)
      for (int c = 0; c < cols; ++c) {
        if (!valid(r, c)) continue;
        double p = std::exp(S[(size_t)r * cols + c] - Lh[i0 + r]);
        if (flags & OR_ROUND32) p = fl32(p);
        const double dp = dot(dOh + (size_t)(i0 + r) * dv, Vg + (size_t)(j0 + c) * dv, dv);
        double ds = p * (dp - dl[i0 + r]);
        if (flags & OR_ROUND32) ds = fl32(ds);
        pt.P[(size_t)r * cols + c] = p;
        pt.dS[(size_t)r * cols + c] = ds;
      }
    std::vector<uint8_t> codes((size_t)rows * cols);
    pt.Ph = pt.P;
    if (flags & OR_QUANT_P_BWD) {
      const float s = qz_tile(rows, cols, 0, [&](int r, int c) { return (float)pt.P[(size_t)r * cols + c]; },
                              valid, codes.data());
      for (size_t k = 0; k < codes.size(); ++k) pt.Ph[k] = (double)s * fp8_decode(codes[k], 0);
    }
    pt.dSh = pt.dS;
    if (flags & OR_QUANT_DS) {
      const float s = qz_tile(rows, cols, 1, [&](int r, int c) { return (float)pt.dS[(size_t)r * cols + c]; },
                              valid, codes.data());
      for (size_t k = 0; k < codes.size(); ++k) pt.dSh[k] = (double)s * fp8_decode(codes[k], 1);
    }
  };

  // Pass A: dQ and diagnostics, one unit per (group, query head, query tile).
  {
    const int64_t units = (int64_t)gs.size() * G * qts.size();
#pragma omp parallel for schedule(dynamic)
    for (int64_t u = 0; u < units; ++u) {
      const Group gr = gs[u / ((int64_t)G * qts.size())];
      const int h = gr.g * G + (int)((u / qts.size()) % G);
      const int qt = qts[u % qts.size()];
      const int i0 = qt * kTile, rows = std::min(kTile, N - i0);
      const double* Kg = K + D.kvoff(gr.b, gr.g);
      double* dQh = dQ + D.qoff(gr.b, h);
      for (int r = 0; r < rows; ++r) {
        for (int k = 0; k < d; ++k) dQh[(size_t)(i0 + r) * d + k] = 0.0;
        if (diag)
          for (int q = 0; q < 4; ++q) diag[(size_t)q * B * Hq * N + D.rowoff(gr.b, h) + i0 + r] = 0.0;
      }
      PairTile pt;
      for (int kt = first_key_tile(D); kt <= last_key_tile(D, qt); ++kt) {
        compute_pair(gr.b, h, qt, kt, pt);
        const int j0 = kt * kTile;
        for (int r = 0; r < pt.rows; ++r) {
          const int i = i0 + r;
          double* dq = dQh + (size_t)i * d;
          for (int c = 0; c < pt.cols; ++c) {
            const double v = pt.dSh[(size_t)r * pt.cols + c];
            if (v != 0.0)
              for (int k = 0; k < d; ++k) dq[k] += D.sigma * v * Kg[(size_t)(j0 + c) * d + k];
            if (diag) {
              const size_t o = D.rowoff(gr.b, h) + i;
              const size_t st = (size_t)B * Hq * N;
              const double x = pt.dS[(size_t)r * pt.cols + c];
              diag[o] += x;
              diag[st + o] += std::fabs(x);
              diag[2 * st + o] += v;
              diag[3 * st + o] += std::fabs(v);
            }
          }
          if (dS_out || dShat_out || Phat_out) {
            const size_t base = ((size_t)gr.b * Hq + h) * N * N + (size_t)i * N + j0;
            for (int c = 0; c < pt.cols; ++c) {
              if (dS_out) dS_out[base + c] = pt.dS[(size_t)r * pt.cols + c];
              if (dShat_out) dShat_out[base + c] = pt.dSh[(size_t)r * pt.cols + c];
              if (Phat_out) Phat_out[base + c] = pt.Ph[(size_t)r * pt.cols + c];
            }
          }
        }
      }
    }
  }

  // Pass B: dK and dV, one unit per (group, key tile); sums over the group's heads.
  {
    const int64_t units = (int64_t)gs.size() * kts.size();
#pragma omp parallel for schedule(dynamic)
    for (int64_t u = 0; u < units; ++u) {
      const Group gr = gs[u / kts.size()];
      const int kt = kts[u % kts.size()];
      const int j0 = kt * kTile, cols = std::min(kTile, N - j0);
      double* dKg = dK + D.kvoff(gr.b, gr.g);
      double* dVg = dV + D.kvvoff(gr.b, gr.g);
      for (int c = 0; c < cols; ++c) {
        for (int k = 0; k < d; ++k) dKg[(size_t)(j0 + c) * d + k] = 0.0;
        for (int k = 0; k < dv; ++k) dVg[(size_t)(j0 + c) * dv + k] = 0.0;
      }
      PairTile pt;
      for (int hh = 0; hh < G; ++hh) {
        const int h = gr.g * G + hh;
        const double* Qh = Q + D.qoff(gr.b, h);
        const double* dOh = dOhat + D.qvoff(gr.b, h);
        for (int qt = D.causal ? kt : 0; qt < T; ++qt) {
          compute_pair(gr.b, h, qt, kt, pt);
          const int i0 = qt * kTile;
          for (int r = 0; r < pt.rows; ++r)
            for (int c = 0; c < pt.cols; ++c) {
              const double ph = pt.Ph[(size_t)r * pt.cols + c];
              const double ds = pt.dSh[(size_t)r * pt.cols + c];
              double* dvr = dVg + (size_t)(j0 + c) * dv;
              double* dk = dKg + (size_t)(j0 + c) * d;
              const double* dor = dOh + (size_t)(i0 + r) * dv;
              const double* qr = Qh + (size_t)(i0 + r) * d;
              if (ph != 0.0)
                for (int k = 0; k < dv; ++k) dvr[k] += ph * dor[k];
              if (ds != 0.0)
                for (int k = 0; k < d; ++k) dk[k] += D.sigma * ds * qr[k];
            }
        }
      }
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Merge of the attention of one query row over disjoint key blocks (context
// parallelism): with block r's LSE_r = ln sum_{j in r} exp(S_ij) and
// O_r = sum_{j in r} exp(S_ij - LSE_r) V_j, the whole row has
//   LSE = ln sum_r exp(LSE_r),   O = sum_r exp(LSE_r - LSE) O_r,
// which is the softmax over the union of the blocks written out.  Blocks with
// LSE_r = -inf (no visible key) weigh zero; a row with none at all gets O = 0
// and LSE = -inf.  O_parts [nparts][rows][dv], LSE_parts [nparts][rows].
int or_attn_merge(int nparts, int64_t rows, int dv, const double* O_parts, const double* LSE_parts, double* O,
                  double* LSE) {
  if (nparts <= 0 || rows < 0 || dv <= 0) return 1;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < rows; ++i) {
    double m = -INFINITY;
    for (int r = 0; r < nparts; ++r) m = std::max(m, LSE_parts[(size_t)r * rows + i]);
    double* o = O + (size_t)i * dv;
    for (int k = 0; k < dv; ++k) o[k] = 0.0;
    if (m == -INFINITY) {
      LSE[i] = -INFINITY;
      continue;
    }
    double wsum = 0.0;
    for (int r = 0; r < nparts; ++r) wsum += std::exp(LSE_parts[(size_t)r * rows + i] - m);
    LSE[i] = m + std::log(wsum);
    for (int r = 0; r < nparts; ++r) {
      const double w = std::exp(LSE_parts[(size_t)r * rows + i] - LSE[i]);
      const double* orow = O_parts + ((size_t)r * rows + i) * dv;
      for (int k = 0; k < dv; ++k) o[k] += w * orow[k];
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Attention-input prologue of a QK-normalised rotary model.  The models on the
// project page normalise queries and keys with RMSNorm and learned per-channel
// gains ("Delta-Matching for reliable FP8 attention training", section 02:
// the gains are the RMSNorm scales on query and key channels, and one of them
// grows to about 5.4 under stale delta) and use rotary position embedding
// (section 05, "Attention variants change when failure appears": QK
// normalisation can be removed, and removing RoPE gives the NoPE variant).
// The pages give no epsilon, rotary layout or base; readings:
//   RMSNorm  y_k = x_k / sqrt(mean_k x_k^2 + eps) * g_k   (g shared by heads)
//   rotary   channel i < d/2 pairs with channel i + d/2 ("rotate half"), at
//            the row's sequence position n, angle theta = n * base^(-2i/d):
//            (a, b) <- (a cos theta - b sin theta, b cos theta + a sin theta).
// Everything in FP64; the quantised result is or_quantize of fl32(y).

// cos and sin of the rotary angles, [N][d/2] each.
void or_rope_table(int N, int d, double base, double* cosv, double* sinv) {
  const int h = d / 2;
  for (int n = 0; n < N; ++n)
    for (int i = 0; i < h; ++i) {
      const double theta = (double)n * std::pow(base, -2.0 * i / d);
      cosv[(size_t)n * h + i] = std::cos(theta);
      sinv[(size_t)n * h + i] = std::sin(theta);
    }
}

// y = rotary(RMSNorm(x) * gain) for every row of a [B][H][N][d] tensor.
// gain: [d] or NULL (all ones); rope = 0 skips the rotation.
int or_qk_prologue(const float* x, int B, int H, int N, int d, const double* gain, double eps, int rope,
                   double base, double* y) {
  if (B < 0 || H < 0 || N < 0 || d <= 0 || (d % 2) || !(eps >= 0.0)) return 1;
  const int h = d / 2;
  std::vector<double> cosv, sinv;
  if (rope) {
    cosv.resize((size_t)N * h);
    sinv.resize((size_t)N * h);
    or_rope_table(N, d, base, cosv.data(), sinv.data());
  }
  const int64_t rows = (int64_t)B * H * N;
#pragma omp parallel for schedule(static)
  for (int64_t row = 0; row < rows; ++row) {
    const float* xr = x + (size_t)row * d;
    double* yr = y + (size_t)row * d;
    double ss = 0.0;
    for (int k = 0; k < d; ++k) ss += (double)xr[k] * (double)xr[k];
    const double inv = 1.0 / std::sqrt(ss / d + eps);
    for (int k = 0; k < d; ++k) yr[k] = (double)xr[k] * inv * (gain ? gain[k] : 1.0);
    if (rope) {
      const int n = (int)(row % N);
      for (int i = 0; i < h; ++i) {
        const double c = cosv[(size_t)n * h + i], sn = sinv[(size_t)n * h + i];
        const double a = yr[i], b = yr[i + h];
        yr[i] = a * c - b * sn;
        yr[i + h] = b * c + a * sn;
      }
    }
  }
  return 0;
}

int or_num_threads() {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

}  // extern "C"
