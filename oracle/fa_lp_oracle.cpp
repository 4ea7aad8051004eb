// fa_lp_oracle.cpp -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, obviously-correct CPU oracle for the low-precision packed-varlen attention
// forward. Only the test suite, the smoke check and the CPU-baseline leg of the benchmark load
// it; the CUDA library never does, and the two share no code, headers or tables.
//
// What it follows:
//  * SGLang PR #40175 "add fp8_fa_sm120 FP8 backend for SM120 GPUs", section Modifications
//    (kernel.py: E4M3 QK and PV with FP32 accumulation, online softmax, probabilities packed to
//    E4M3; fused_prep.py: per-head amax then pack of strided BF16 Q/K/V).
//  * SGLang PR #40116 "Add SM120 Sage compute for SubBlock sparse attention", Modifications
//    (Q64 x K64 blocks, partial blocks, variable per-row block counts, mixed sparse and dense
//    rows) and Accuracy Tests (ragged lengths, variable block counts, empty rows).
//  * FlashInfer docs, flashinfer.diffusion_ops.minimax_h3_sm120_varlen_attention_nvfp4, the
//    description paragraph (SageAttention3 FP4 recipe: K centred by the segment's per-channel
//    mean, Q by its 128-row block mean with qm K^T added back, E2M1 codes with one UE4M3 scale per
//    16 elements = block amax / 6, V transposed with per-16-key scales, two-level P with the row
//    maximum brought to 448*6) and its Parameters list (cu_seqlens contract, default scale).
//
// Readings taken where the pages are silent (each is stated again where it is used):
//  r1  FP8 amax is per (tensor, head) over all tokens of the packed input. Opt-in alternative
//      (the per-segment FP8 mode): one amax per (segment, tensor, head) over the segment's own
//      tokens, so that one long segment does not set a short segment's scale.
//  r2  inv = fl32(448/amax), code = E4M3(fl32(x*inv)), descale = fl32(amax/448); amax==0 -> 1.
//  r3  E4M3: round to nearest, ties to even, saturate to +-448, sign of zero kept, subnormals kept.
//  r4  FP8 P is the unscaled exp(S - m) in [0,1], rounded through fp32 then to E4M3 (shift p = 0;
//      p is a parameter so that a kernel using a power-of-two shift can be replayed).
//  r5  online softmax over key tiles of n_kv keys counted from the segment start. The reference
//      maximum m starts at the first tile's maximum and moves to a later tile's maximum only when
//      that exceeds m by more than tau (in log2 units, i.e. by a factor 2^tau in probability);
//      tau = 0 is the exact running maximum. Both are parameters so that the kernel's own rule
//      is replayed.
//  r6  the softmax denominator l sums the quantized probabilities.
//  r7  NVFP4 Q blocks and V key groups start at each segment's first token; partial last block's
//      mean is over present rows; padded V keys are zero.
//  r8  K / Q means: FP64 sums in canonical order (128-token chunks in order, then chunk sums in
//      order), mean = fl32(sum / n), centred value = fl32(x - mean).
//  r9  UE4M3 scale = E4M3(fl32(amax16/6)); code = E2M1(fl32(x / deq(scale))); scale 0 -> codes 0.
//  r10 E2M1: round to nearest even on {0,.5,1,1.5,2,3,4,6}, saturate to 6, sign of zero kept.
//  r11 NVFP4 P first level: P' = fl32(2688 * exp(S' - m_running)).
//  r12 the qm K^T term uses the dequantized centred K.
//  r15 LSE of a row = m + log(l) in the natural units of S = q.k scale: the log of the normalizer
//      of the (quantized) softmax the output divides by (exact attention: log sum exp(s)).
//  r16 block-sparse attention (SGLang PR #40116, Modifications and Accuracy Tests): a query row
//      in the g-th 64-row block of its segment attends to the keys of the 64-key blocks listed
//      for (head, g), blocks counted from the segment start, the last one partial; lists are
//      strictly ascending; a row with an empty list outputs 0 and has LSE -inf. The FP8 replay
//      takes the listed blocks, in list order, as the online softmax's key tiles.
//
// Build: g++ -std=c++17 -O2 -ffp-contract=off -fPIC -shared -pthread (no fast-math), so that fp32
// products and quotients are single IEEE round-to-nearest operations on any host.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <limits>
#include <thread>
#include <vector>

namespace {

constexpr int kD = 128;  // head dimension fixed by the pages' op (q/k/v are [tokens, heads, 128])

// ---------------------------------------------------------------------------------------------
// Number formats, from their definitions.
// E4M3 (OCP FP8, "fn" flavour): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinity,
// S.1111.111 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448.
// E2M1 (OCP FP4): 1 sign, 2 exponent bits (bias 1), 1 mantissa bit: 0, .5, 1, 1.5, 2, 3, 4, 6.
// ---------------------------------------------------------------------------------------------

double e4m3_magnitude(int code7) {  // code7 in [0, 126]
  const int e = (code7 >> 3) & 0xF;
  const int m = code7 & 7;
  if (e == 0) return std::ldexp(m / 8.0, -6);
  return std::ldexp(1.0 + m / 8.0, e - 7);
}

const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

// Nearest entry of an ascending magnitude table, ties to the even code (mantissa LSB 0).
int nearest_even(const double* table, int n, double a) {
  if (a >= table[n - 1]) return n - 1;  // saturate to the largest finite magnitude
  int lo = 0, hi = n - 1;               // invariant: table[lo] <= a < table[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) / 2;
    if (table[mid] <= a) lo = mid; else hi = mid;
  }
  const double dlo = a - table[lo];
  const double dhi = table[hi] - a;
  if (dlo < dhi) return lo;
  if (dhi < dlo) return hi;
  return (lo & 1) ? hi : lo;
}

struct E4M3Table {
  double mag[127];
  E4M3Table() { for (int c = 0; c < 127; ++c) mag[c] = e4m3_magnitude(c); }
};
const E4M3Table& e4m3_table() { static const E4M3Table t; return t; }

uint8_t e4m3_encode(float x) {
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  if (std::isnan(x)) return sign | 0x7F;  // out of contract (non-finite inputs)
  const double a = std::fabs(static_cast<double>(x));
  return sign | static_cast<uint8_t>(nearest_even(e4m3_table().mag, 127, a));
}

double e4m3_decode(uint8_t c) {
  const double s = (c & 0x80) ? -1.0 : 1.0;
  if ((c & 0x7F) == 0x7F) return std::numeric_limits<double>::quiet_NaN();
  return s * e4m3_magnitude(c & 0x7F);
}

uint8_t e2m1_encode(float x) {
  const uint8_t sign = std::signbit(x) ? 0x8 : 0x0;
  const double a = std::fabs(static_cast<double>(x));
  return sign | static_cast<uint8_t>(nearest_even(kE2M1, 8, a));
}

double e2m1_decode(uint8_t c) {
  const double s = (c & 0x8) ? -1.0 : 1.0;
  return s * kE2M1[c & 7];
}

float bf16_to_f32(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// Round a double to the nearest BF16 (8 significant bits, fp32 exponent range), ties to even.
uint16_t f64_to_bf16(double x) {
  if (std::isnan(x)) return 0x7FC0;
  const bool neg = std::signbit(x);
  const double a = std::fabs(x);
  uint16_t mag;
  if (a == 0.0) {
    mag = 0;
  } else {
    int e;
    std::frexp(a, &e);                         // a = f * 2^e, f in [0.5, 1)
    const int exp_unbiased = std::max(e - 1, -126);  // below 2^-126 the spacing stays 2^-133
    const double ulp = std::ldexp(1.0, exp_unbiased - 7);
    const double q = std::nearbyint(a / ulp) * ulp;  // default rounding mode: nearest-even
    float qf = static_cast<float>(q);                // exact: q has <= 8 significant bits
    if (q > 3.3895313892515355e38) qf = std::numeric_limits<float>::infinity();
    uint32_t u;
    std::memcpy(&u, &qf, 4);
    mag = static_cast<uint16_t>(u >> 16);
  }
  return static_cast<uint16_t>(mag | (neg ? 0x8000 : 0));
}

// ---------------------------------------------------------------------------------------------
// Small helpers: thread pool over an index range, segment lookup.
// ---------------------------------------------------------------------------------------------

void parallel_for(int64_t n, int nthreads, const std::function<void(int64_t)>& fn) {
  if (nthreads <= 0) nthreads = static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
  if (nthreads == 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  std::vector<std::thread> pool;
  const int64_t per = (n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    const int64_t b = t * per, e = std::min(n, b + per);
    if (b >= e) break;
    pool.emplace_back([b, e, &fn] { for (int64_t i = b; i < e; ++i) fn(i); });
  }
  for (auto& th : pool) th.join();
}

int segment_of(const int32_t* cu, int nseg, int64_t t) {  // s with cu[s] <= t < cu[s+1]
  int lo = 0, hi = nseg;  // cu[lo] <= t < cu[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) / 2;
    if (cu[mid] <= t) lo = mid; else hi = mid;
  }
  // skip empty segments that share the same start
  while (lo + 1 < nseg && cu[lo + 1] <= t) ++lo;
  return lo;
}

inline float load_bf16(const uint16_t* base, int64_t t, int h, int c, int64_t st, int64_t sh) {
  return bf16_to_f32(base[t * st + h * sh + c]);
}

// Sum a sequence of doubles in the canonical order of reading r8: consecutive chunks of 128
// values summed left to right, then the chunk sums left to right.
template <class Get>
double canonical_sum(int64_t n, Get get) {
  double total = 0.0;
  for (int64_t c0 = 0; c0 < n; c0 += 128) {
    double chunk = 0.0;
    const int64_t c1 = std::min(n, c0 + 128);
    for (int64_t i = c0; i < c1; ++i) chunk += get(i);
    total += chunk;
  }
  return total;
}

// One group of 16 values -> UE4M3 scale and 16 E2M1 codes (reading r9).
void nvfp4_group(const float* x, int n, uint8_t* codes, uint8_t* sf_out) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) amax = std::max(amax, std::fabs(x[i]));
  const float s = amax / 6.0f;  // IEEE single division
  const uint8_t sf = e4m3_encode(s);
  *sf_out = sf;
  const float ds = static_cast<float>(e4m3_decode(sf));  // exact in fp32
  for (int i = 0; i < n; ++i) {
    if (sf == 0) { codes[i] = 0; continue; }
    const float y = x[i] / ds;
    codes[i] = e2m1_encode(y);
  }
}

// Key ranges [j0, j1) of one query row, in the order the online softmax visits them.
using Ranges = std::vector<std::pair<int64_t, int64_t>>;

// Exact FP64 attention of query row (t, h) over the keys of `keys`; no key gives 0 and LSE -inf.
void exact_row(const uint16_t* q, int64_t qst, int64_t qsh, const uint16_t* k, int64_t kst,
               int64_t ksh, const uint16_t* v, int64_t vst, int64_t vsh, int64_t t, int h,
               const Ranges& keys, double scale, double* out, double* lse) {
  std::vector<double> qi(kD), sc;
  for (int c = 0; c < kD; ++c) qi[c] = load_bf16(q, t, h, c, qst, qsh);
  double m = -std::numeric_limits<double>::infinity();
  for (const auto& kr : keys)
    for (int64_t j = kr.first; j < kr.second; ++j) {
      double acc = 0.0;
      for (int c = 0; c < kD; ++c) acc += qi[c] * static_cast<double>(load_bf16(k, j, h, c, kst, ksh));
      sc.push_back(acc * scale);
      m = std::max(m, sc.back());
    }
  double l = 0.0;
  std::vector<double> o(kD, 0.0);
  size_t i = 0;
  for (const auto& kr : keys)
    for (int64_t j = kr.first; j < kr.second; ++j, ++i) {
      const double p = std::exp(sc[i] - m);
      l += p;
      for (int c = 0; c < kD; ++c) o[c] += p * load_bf16(v, j, h, c, vst, vsh);
    }
  for (int c = 0; c < kD; ++c) out[c] = l > 0.0 ? o[c] / l : 0.0;
  if (lse) lse[0] = l > 0.0 ? m + std::log(l) : -std::numeric_limits<double>::infinity();
}

// FP8-emulating attention of query row (t, h) (C2 below) over the key tiles `tiles`, in order.
void fp8_row(const uint8_t* cq, const uint8_t* ck, const uint8_t* cv, const float* dq,
             const float* dk, const float* dv, int H, int64_t t, int h, const Ranges& tiles,
             double scale, int p_shift, double tau, double* out64, uint16_t* out16, double* lse) {
  const double inf = std::numeric_limits<double>::infinity();
  const double pscale = std::ldexp(1.0, p_shift);
  const double tau_nat = tau * std::log(2.0);  // threshold in the natural-log units of S
  const double sfac = static_cast<double>(dq[h]) * static_cast<double>(dk[h]) * scale;
  double qi[kD];
  for (int c = 0; c < kD; ++c) qi[c] = e4m3_decode(cq[(t * H + h) * kD + c]);
  double m = -inf, l = 0.0;
  std::vector<double> o(kD, 0.0), sc;
  for (const auto& tile : tiles) {
    const int64_t j0 = tile.first, j1 = tile.second;
    sc.assign(j1 - j0, 0.0);
    double mt = -inf;
    for (int64_t j = j0; j < j1; ++j) {
      double acc = 0.0;  // exact: products are multiples of 2^-18, |sum| < 2^25
      for (int c = 0; c < kD; ++c) acc += qi[c] * e4m3_decode(ck[(j * H + h) * kD + c]);
      sc[j - j0] = acc * sfac;
      mt = std::max(mt, sc[j - j0]);
    }
    const double m_new = (m == -inf || mt > m + tau_nat) ? mt : m;
    const double alpha = (m == -inf) ? 0.0 : std::exp(m - m_new);
    l *= alpha;
    for (int c = 0; c < kD; ++c) o[c] *= alpha;
    for (int64_t j = j0; j < j1; ++j) {
      const float pt = static_cast<float>(std::exp(sc[j - j0] - m_new) * pscale);
      const double pq = e4m3_decode(e4m3_encode(pt)) / pscale;
      if (pq == 0.0) continue;
      l += pq;
      for (int c = 0; c < kD; ++c) o[c] += pq * e4m3_decode(cv[(j * H + h) * kD + c]);
    }
    m = m_new;
  }
  for (int c = 0; c < kD; ++c) {
    const double y = l > 0.0 ? o[c] * static_cast<double>(dv[h]) / l : 0.0;
    out64[c] = y;
    if (out16) out16[c] = f64_to_bf16(y);
  }
  // r15: the log of the quantized softmax normalizer, in the natural units of S
  if (lse) lse[0] = l > 0.0 ? m + std::log(l) : -inf;
}

// r16: 64-row query blocks and 64-key key blocks, counted from each segment's first token.
constexpr int kSparseBlock = 64;

// First query block of every segment (qb0[s]) and the total G over the packed batch.
int64_t sparse_qblock_offsets(const int32_t* cu, int nseg, std::vector<int64_t>& qb0) {
  qb0.assign(nseg + 1, 0);
  for (int s = 0; s < nseg; ++s)
    qb0[s + 1] = qb0[s] + (cu[s + 1] - cu[s] + kSparseBlock - 1) / kSparseBlock;
  return qb0[nseg];
}

// Key tiles of row (t, h) under the block lists; false if the list breaks the contract
// (an index outside the segment's key blocks, or not strictly ascending).
bool sparse_tiles(const int32_t* cu, int nseg, const std::vector<int64_t>& qb0, int64_t G,
                  const int32_t* blk_off, const int32_t* blk_idx, int64_t t, int h, Ranges& out) {
  const int s = segment_of(cu, nseg, t);
  const int64_t a = cu[s], b = cu[s + 1];
  const int64_t nkb = (b - a + kSparseBlock - 1) / kSparseBlock;
  const int64_t g = qb0[s] + (t - a) / kSparseBlock;
  out.clear();
  int64_t prev = -1;
  for (int64_t i = blk_off[h * G + g]; i < blk_off[h * G + g + 1]; ++i) {
    const int64_t kb = blk_idx[i];
    if (kb < 0 || kb >= nkb || kb <= prev) return false;
    prev = kb;
    out.push_back({a + kSparseBlock * kb, std::min(b, a + kSparseBlock * (kb + 1))});
  }
  return true;
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------------------------
// Converters (exported for the exhaustive table tests).
// ---------------------------------------------------------------------------------------------
uint8_t orc_e4m3_encode(float x) { return e4m3_encode(x); }
double orc_e4m3_decode(uint8_t c) { return e4m3_decode(c); }
uint8_t orc_e2m1_encode(float x) { return e2m1_encode(x); }
double orc_e2m1_decode(uint8_t c) { return e2m1_decode(c); }
uint16_t orc_f64_to_bf16(double x) { return f64_to_bf16(x); }

void orc_e4m3_encode_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode(x[i]);
}
void orc_e2m1_encode_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e2m1_encode(x[i]);
}

// ---------------------------------------------------------------------------------------------
// FP8 quantization of one tensor (SGLang #40175, Modifications, fused_prep.py: amax per head,
// then pack). x: BF16 [T, H, 128] with element strides (tok, head), channel stride 1.
// codes: [T, H, 128] E4M3 bytes (natural order); descale: [H] fp32 (readings r1, r2, r3).
// ---------------------------------------------------------------------------------------------
void orc_fp8_quantize(const uint16_t* x, int64_t T, int H, int64_t st, int64_t sh,
                      uint8_t* codes, float* descale, int nthreads) {
  parallel_for(H, nthreads, [&](int64_t h) {
    float amax = 0.0f;
    for (int64_t t = 0; t < T; ++t)
      for (int c = 0; c < kD; ++c) amax = std::max(amax, std::fabs(load_bf16(x, t, h, c, st, sh)));
    float inv = 1.0f, d = 1.0f;
    if (amax > 0.0f) {
      inv = 448.0f / amax;
      d = amax / 448.0f;
    }
    descale[h] = d;
    for (int64_t t = 0; t < T; ++t)
      for (int c = 0; c < kD; ++c) {
        const float y = load_bf16(x, t, h, c, st, sh) * inv;
        codes[(t * H + h) * kD + c] = e4m3_encode(y);
      }
  });
}

// The per-segment alternative of reading r1 (same arithmetic, r2 and r3, with the amax taken
// over the tokens of one segment): descale: [nseg][H]; an empty segment gets descale 1 and no
// codes.
void orc_fp8_quantize_seg(const uint16_t* x, int64_t T, int H, int64_t st, int64_t sh,
                          const int32_t* cu, int nseg, uint8_t* codes, float* descale,
                          int nthreads) {
  (void)T;
  parallel_for(static_cast<int64_t>(nseg) * H, nthreads, [&](int64_t sh_idx) {
    const int s = static_cast<int>(sh_idx / H), h = static_cast<int>(sh_idx % H);
    const int64_t a = cu[s], b = cu[s + 1];
    float amax = 0.0f;
    for (int64_t t = a; t < b; ++t)
      for (int c = 0; c < kD; ++c) amax = std::max(amax, std::fabs(load_bf16(x, t, h, c, st, sh)));
    float inv = 1.0f, d = 1.0f;
    if (amax > 0.0f) {
      inv = 448.0f / amax;
      d = amax / 448.0f;
    }
    descale[sh_idx] = d;
    for (int64_t t = a; t < b; ++t)
      for (int c = 0; c < kD; ++c) {
        const float y = load_bf16(x, t, h, c, st, sh) * inv;
        codes[(t * H + h) * kD + c] = e4m3_encode(y);
      }
  });
}

// ---------------------------------------------------------------------------------------------
// C1: exact attention in FP64 for a list of query rows (token, head). The plain definition from
// the FlashInfer docs' formula: out[i] = softmax(q_i k^T * scale) v over the keys of i's segment.
// rows: [nrows][2] = (token, head). out: [nrows][128] fp64.
// ---------------------------------------------------------------------------------------------
void orc_attn_exact(const uint16_t* q, int64_t qst, int64_t qsh,
                    const uint16_t* k, int64_t kst, int64_t ksh,
                    const uint16_t* v, int64_t vst, int64_t vsh,
                    int64_t T, int H, const int32_t* cu, int nseg, double scale,
                    const int64_t* rows, int64_t nrows, double* out, double* lse, int nthreads) {
  (void)T; (void)H;
  parallel_for(nrows, nthreads, [&](int64_t r) {
    const int64_t t = rows[2 * r];
    const int h = static_cast<int>(rows[2 * r + 1]);
    const int s = segment_of(cu, nseg, t);
    const Ranges keys{{cu[s], cu[s + 1]}};
    exact_row(q, qst, qsh, k, kst, ksh, v, vst, vsh, t, h, keys, scale, out + r * kD,
              lse ? lse + r : nullptr);
  });
}

// ---------------------------------------------------------------------------------------------
// C2: FP8 quantization-emulating attention for a list of query rows (SGLang #40175,
// Modifications, kernel.py): scores from E4M3 codes with exact accumulation, times
// dq*dk*scale; online softmax over key tiles of n_kv keys from the segment start with the exact
// running maximum (r5); P = exp(S - m) rounded through fp32 to E4M3 after a 2^p shift (r4);
// l sums the quantized P (r6); O accumulates quantized P times V codes; out = O * dv / l.
// codes_*: [T, H, 128] natural order. out64: [nrows][128] fp64; out16 (optional): BF16 bits.
// ---------------------------------------------------------------------------------------------
void orc_attn_fp8(const uint8_t* cq, const uint8_t* ck, const uint8_t* cv,
                  const float* dq, const float* dk, const float* dv,
                  int64_t T, int H, const int32_t* cu, int nseg, double scale, int n_kv,
                  int p_shift, double tau, const int64_t* rows, int64_t nrows, double* out64,
                  uint16_t* out16, double* lse, int nthreads, int seg_scales) {
  (void)T;
  parallel_for(nrows, nthreads, [&](int64_t r) {
    const int64_t t = rows[2 * r];
    const int h = static_cast<int>(rows[2 * r + 1]);
    const int s = segment_of(cu, nseg, t);
    Ranges tiles;
    for (int64_t j0 = cu[s]; j0 < cu[s + 1]; j0 += n_kv)
      tiles.push_back({j0, std::min<int64_t>(cu[s + 1], j0 + n_kv)});
    // per-segment scales: the descale rows of the query's segment ([nseg][H] arrays)
    const int64_t so = seg_scales ? static_cast<int64_t>(s) * H : 0;
    fp8_row(cq, ck, cv, dq + so, dk + so, dv + so, H, t, h, tiles, scale, p_shift, tau,
            out64 + r * kD, out16 ? out16 + r * kD : nullptr, lse ? lse + r : nullptr);
  });
}

// ---------------------------------------------------------------------------------------------
// C1 and C2 under block-sparse lists (r16). blk_off: int32 [H * G + 1], the list of (head h,
// query block g) is blk_idx[blk_off[h G + g], blk_off[h G + g + 1]); G = sum over segments of
// ceil(L_s / 64). Return 0, or -1 when a row's list breaks the contract (its output is then 0).
// ---------------------------------------------------------------------------------------------
int orc_attn_exact_sparse(const uint16_t* q, int64_t qst, int64_t qsh,
                          const uint16_t* k, int64_t kst, int64_t ksh,
                          const uint16_t* v, int64_t vst, int64_t vsh, int64_t T, int H,
                          const int32_t* cu, int nseg, double scale, const int32_t* blk_off,
                          const int32_t* blk_idx, const int64_t* rows, int64_t nrows,
                          double* out, double* lse, int nthreads) {
  (void)T; (void)H;
  std::vector<int64_t> qb0;
  const int64_t G = sparse_qblock_offsets(cu, nseg, qb0);
  std::vector<int> bad(nrows, 0);
  parallel_for(nrows, nthreads, [&](int64_t r) {
    const int64_t t = rows[2 * r];
    const int h = static_cast<int>(rows[2 * r + 1]);
    Ranges keys;
    if (!sparse_tiles(cu, nseg, qb0, G, blk_off, blk_idx, t, h, keys)) {
      bad[r] = 1;
      keys.clear();
    }
    exact_row(q, qst, qsh, k, kst, ksh, v, vst, vsh, t, h, keys, scale, out + r * kD,
              lse ? lse + r : nullptr);
  });
  return std::count(bad.begin(), bad.end(), 1) ? -1 : 0;
}

int orc_attn_fp8_sparse(const uint8_t* cq, const uint8_t* ck, const uint8_t* cv,
                        const float* dq, const float* dk, const float* dv, int64_t T, int H,
                        const int32_t* cu, int nseg, double scale, const int32_t* blk_off,
                        const int32_t* blk_idx, int p_shift, double tau, const int64_t* rows,
                        int64_t nrows, double* out64, uint16_t* out16, double* lse,
                        int nthreads, int seg_scales) {
  (void)T;
  std::vector<int64_t> qb0;
  const int64_t G = sparse_qblock_offsets(cu, nseg, qb0);
  std::vector<int> bad(nrows, 0);
  parallel_for(nrows, nthreads, [&](int64_t r) {
    const int64_t t = rows[2 * r];
    const int h = static_cast<int>(rows[2 * r + 1]);
    Ranges tiles;
    if (!sparse_tiles(cu, nseg, qb0, G, blk_off, blk_idx, t, h, tiles)) {
      bad[r] = 1;
      tiles.clear();
    }
    const int64_t so = seg_scales ? static_cast<int64_t>(segment_of(cu, nseg, t)) * H : 0;
    fp8_row(cq, ck, cv, dq + so, dk + so, dv + so, H, t, h, tiles, scale, p_shift, tau,
            out64 + r * kD, out16 ? out16 + r * kD : nullptr, lse ? lse + r : nullptr);
  });
  return std::count(bad.begin(), bad.end(), 1) ? -1 : 0;
}

// ---------------------------------------------------------------------------------------------
// NVFP4 quantization (FlashInfer docs, minimax_h3_sm120_varlen_attention_nvfp4, description).
// ---------------------------------------------------------------------------------------------

// a6: per (segment, head, channel) mean of K over the segment (r8). km: [nseg][H][128] fp32;
// empty segments get 0.
void orc_nvfp4_kmean(const uint16_t* k, int64_t kst, int64_t ksh, int64_t T, int H,
                     const int32_t* cu, int nseg, float* km, int nthreads) {
  (void)T;
  parallel_for(static_cast<int64_t>(nseg) * H, nthreads, [&](int64_t sh) {
    const int s = static_cast<int>(sh / H), h = static_cast<int>(sh % H);
    const int64_t a = cu[s], n = cu[s + 1] - cu[s];
    for (int c = 0; c < kD; ++c) {
      if (n == 0) { km[sh * kD + c] = 0.0f; continue; }
      const double sum = canonical_sum(n, [&](int64_t i) {
        return static_cast<double>(load_bf16(k, a + i, h, c, kst, ksh));
      });
      km[sh * kD + c] = static_cast<float>(sum / static_cast<double>(n));
    }
  });
}

// Number of 128-row Q blocks before segment s, and in total (r7).
int64_t orc_nvfp4_qblock_offsets(const int32_t* cu, int nseg, int64_t* offs) {
  int64_t acc = 0;
  for (int s = 0; s < nseg; ++s) {
    offs[s] = acc;
    acc += (static_cast<int64_t>(cu[s + 1]) - cu[s] + 127) / 128;
  }
  offs[nseg] = acc;
  return acc;
}

// Number of 16-key V groups before segment s, and in total (r7).
int64_t orc_nvfp4_vgroup_offsets(const int32_t* cu, int nseg, int64_t* offs) {
  int64_t acc = 0;
  for (int s = 0; s < nseg; ++s) {
    offs[s] = acc;
    acc += (static_cast<int64_t>(cu[s + 1]) - cu[s] + 15) / 16;
  }
  offs[nseg] = acc;
  return acc;
}

// a7 for Q: 128-row block means from each segment start (r7, r8), centring, then per 16
// channels UE4M3 scale + E2M1 codes (r9, r10).
// qm: [QB_total][H][128] fp32; codes: [T, H, 128] (one 4-bit code per byte); sf: [T, H, 8].
void orc_nvfp4_quantize_q(const uint16_t* q, int64_t qst, int64_t qsh, int64_t T, int H,
                          const int32_t* cu, int nseg, float* qm, uint8_t* codes, uint8_t* sf,
                          int nthreads) {
  (void)T;
  std::vector<int64_t> qoff(nseg + 1);
  const int64_t nqb = orc_nvfp4_qblock_offsets(cu, nseg, qoff.data());
  // block table: (segment, block-in-segment)
  std::vector<std::pair<int, int64_t>> blocks;
  blocks.reserve(nqb);
  for (int s = 0; s < nseg; ++s)
    for (int64_t b = 0; b < qoff[s + 1] - qoff[s]; ++b) blocks.emplace_back(s, b);
  parallel_for(nqb * H, nthreads, [&](int64_t idx) {
    const int64_t qb = idx / H;
    const int h = static_cast<int>(idx % H);
    const int s = blocks[qb].first;
    const int64_t r0 = cu[s] + blocks[qb].second * 128;
    const int64_t r1 = std::min<int64_t>(cu[s + 1], r0 + 128);
    float mean[kD];
    for (int c = 0; c < kD; ++c) {
      const double sum = canonical_sum(r1 - r0, [&](int64_t i) {
        return static_cast<double>(load_bf16(q, r0 + i, h, c, qst, qsh));
      });
      mean[c] = static_cast<float>(sum / static_cast<double>(r1 - r0));
      qm[(qb * H + h) * kD + c] = mean[c];
    }
    float xc[kD];
    for (int64_t t = r0; t < r1; ++t) {
      for (int c = 0; c < kD; ++c) xc[c] = load_bf16(q, t, h, c, qst, qsh) - mean[c];
      for (int g = 0; g < kD / 16; ++g)
        nvfp4_group(xc + 16 * g, 16, codes + (t * H + h) * kD + 16 * g, sf + (t * H + h) * 8 + g);
    }
  });
}

// r15 helper: q . km per (token, head), BF16 q and the fp32 segment mean, summed in FP64 over the
// channels in order. out: [T][H].
void orc_nvfp4_qkm(const uint16_t* q, int64_t qst, int64_t qsh, int64_t T, int H,
                   const int32_t* cu, int nseg, const float* km, double* out, int nthreads) {
  parallel_for(T * H, nthreads, [&](int64_t idx) {
    const int64_t t = idx / H;
    const int h = static_cast<int>(idx % H);
    const int s = segment_of(cu, nseg, t);
    double acc = 0.0;
    for (int c = 0; c < kD; ++c)
      acc += static_cast<double>(load_bf16(q, t, h, c, qst, qsh)) *
             static_cast<double>(km[(static_cast<int64_t>(s) * H + h) * kD + c]);
    out[t * H + h] = acc;
  });
}

// a7 for K: centring by the segment mean km (from orc_nvfp4_kmean), then per 16 channels.
void orc_nvfp4_quantize_k(const uint16_t* k, int64_t kst, int64_t ksh, int64_t T, int H,
                          const int32_t* cu, int nseg, const float* km, uint8_t* codes,
                          uint8_t* sf, int nthreads) {
  parallel_for(T * H, nthreads, [&](int64_t idx) {
    const int64_t t = idx / H;
    const int h = static_cast<int>(idx % H);
    const int s = segment_of(cu, nseg, t);
    float xc[kD];
    for (int c = 0; c < kD; ++c) xc[c] = load_bf16(k, t, h, c, kst, ksh) - km[(static_cast<int64_t>(s) * H + h) * kD + c];
    for (int g = 0; g < kD / 16; ++g)
      nvfp4_group(xc + 16 * g, 16, codes + (t * H + h) * kD + 16 * g, sf + (t * H + h) * 8 + g);
  });
}

// a7 for V (transposed operand): per channel, groups of 16 consecutive keys from each segment
// start, the last group zero-padded (r7). codes: [T, H, 128]; sf: [H][128][G_total].
void orc_nvfp4_quantize_v(const uint16_t* v, int64_t vst, int64_t vsh, int64_t T, int H,
                          const int32_t* cu, int nseg, uint8_t* codes, uint8_t* sf,
                          int nthreads) {
  (void)T;
  std::vector<int64_t> goff(nseg + 1);
  const int64_t G = orc_nvfp4_vgroup_offsets(cu, nseg, goff.data());
  parallel_for(static_cast<int64_t>(H) * kD, nthreads, [&](int64_t hc) {
    const int h = static_cast<int>(hc / kD), c = static_cast<int>(hc % kD);
    float x[16];
    uint8_t cd[16];
    for (int s = 0; s < nseg; ++s) {
      const int64_t a = cu[s], b = cu[s + 1];
      for (int64_t g = 0; g < goff[s + 1] - goff[s]; ++g) {
        const int64_t j0 = a + 16 * g;
        const int n = static_cast<int>(std::min<int64_t>(16, b - j0));
        for (int i = 0; i < 16; ++i) x[i] = (i < n) ? load_bf16(v, j0 + i, h, c, vst, vsh) : 0.0f;
        nvfp4_group(x, 16, cd, sf + (static_cast<int64_t>(h) * kD + c) * G + goff[s] + g);
        for (int i = 0; i < n; ++i) codes[((j0 + i) * H + h) * kD + c] = cd[i];
      }
    }
  });
}

// ---------------------------------------------------------------------------------------------
// C3: NVFP4 emulating attention for a list of query rows. Scores S' = scale * (deq(Qc) deq(Kc)^T
// + qm deq(Kc)^T) (r12); online softmax over tiles of n_kv keys (a multiple of 16) from the
// segment start with the exact running max (r5 with tau = 0); P' = fl32(2688 exp(S' - m)) (r11);
// per 16 keys of the tile a UE4M3 scale and E2M1 codes (r9); l sums deq(P'); O sums deq(P')
// deq(V); out = O / l.
// ---------------------------------------------------------------------------------------------
void orc_attn_nvfp4(const uint8_t* cq, const uint8_t* sfq, const float* qm, const double* qkm,
                    const uint8_t* ck, const uint8_t* sfk,
                    const uint8_t* cv, const uint8_t* sfv,
                    int64_t T, int H, const int32_t* cu, int nseg, double scale, int n_kv,
                    const int64_t* rows, int64_t nrows, double* out64, uint16_t* out16,
                    double* lse, int nthreads) {
  (void)T;
  const double inf = std::numeric_limits<double>::infinity();
  std::vector<int64_t> qoff(nseg + 1), goff(nseg + 1);
  orc_nvfp4_qblock_offsets(cu, nseg, qoff.data());
  const int64_t G = orc_nvfp4_vgroup_offsets(cu, nseg, goff.data());
  parallel_for(nrows, nthreads, [&](int64_t r) {
    const int64_t t = rows[2 * r];
    const int h = static_cast<int>(rows[2 * r + 1]);
    const int s = segment_of(cu, nseg, t);
    const int64_t a = cu[s], b = cu[s + 1];
    const int64_t qb = qoff[s] + (t - a) / 128;
    double qd[kD], qmean[kD];
    for (int c = 0; c < kD; ++c) {
      qd[c] = e2m1_decode(cq[(t * H + h) * kD + c]) * e4m3_decode(sfq[(t * H + h) * 8 + c / 16]);
      qmean[c] = qm[(qb * H + h) * kD + c];
    }
    double m = -inf, l = 0.0;
    std::vector<double> o(kD, 0.0), sc;
    for (int64_t j0 = a; j0 < b; j0 += n_kv) {
      const int64_t j1 = std::min(b, j0 + n_kv);
      sc.assign(j1 - j0, 0.0);
      double mt = -inf;
      for (int64_t j = j0; j < j1; ++j) {
        double acc = 0.0;
        for (int c = 0; c < kD; ++c) {
          const double kd = e2m1_decode(ck[(j * H + h) * kD + c]) * e4m3_decode(sfk[(j * H + h) * 8 + c / 16]);
          acc += (qd[c] + qmean[c]) * kd;
        }
        sc[j - j0] = acc * scale;
        mt = std::max(mt, sc[j - j0]);
      }
      const double m_new = std::max(m, mt);
      const double alpha = (m == -inf) ? 0.0 : std::exp(m - m_new);
      l *= alpha;
      for (int c = 0; c < kD; ++c) o[c] *= alpha;
      for (int64_t g0 = j0; g0 < j1; g0 += 16) {
        const int n = static_cast<int>(std::min<int64_t>(16, j1 - g0));
        float pp[16];
        uint8_t pc[16], psf;
        for (int i = 0; i < 16; ++i)
          pp[i] = (i < n) ? static_cast<float>(2688.0 * std::exp(sc[g0 + i - j0] - m_new)) : 0.0f;
        nvfp4_group(pp, 16, pc, &psf);
        const double ds = e4m3_decode(psf);
        const int64_t vg = goff[s] + (g0 - a) / 16;
        for (int i = 0; i < n; ++i) {
          const double pd = ds * e2m1_decode(pc[i]);
          if (pd == 0.0) continue;
          l += pd;
          const int64_t j = g0 + i;
          for (int c = 0; c < kD; ++c) {
            const double vd = e2m1_decode(cv[(j * H + h) * kD + c]) *
                              e4m3_decode(sfv[(static_cast<int64_t>(h) * kD + c) * G + vg]);
            o[c] += pd * vd;
          }
        }
      }
      m = m_new;
    }
    for (int c = 0; c < kD; ++c) {
      const double y = o[c] / l;
      out64[r * kD + c] = y;
      if (out16) out16[r * kD + c] = f64_to_bf16(y);
    }
    // r15: l sums deq(P') = 2688 exp(S' - m) quantized, so the normalizer is l / 2688; the scores
    // are those of the centred K, and q . km scale (BF16 q) restores the uncentred ones
    if (lse) lse[r] = m + std::log(l) - std::log(2688.0) + qkm[t * H + h] * scale;
  });
}

}  // extern "C"
