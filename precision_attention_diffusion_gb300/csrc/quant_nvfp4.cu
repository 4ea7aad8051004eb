// quant_nvfp4.cu -- NVFP4 (SageAttention3-style) quantization of BF16 Q/K/V into the workspace.
//
// Passage: FlashInfer docs, flashinfer.diffusion_ops.minimax_h3_sm120_varlen_attention_nvfp4,
// description: K rows centred by the segment's per-channel mean, Q rows by their 128-row block's
// mean; Q / K / V stored as E2M1 codes with one UE4M3 scale per 16 elements (block amax / 6); V
// transposed with per-16-key scales; segments of any length, including empty ones.
//
// Arithmetic (readings r7-r10): means are FP64 sums in canonical order -- 128-token chunks from
// the segment start summed left to right, then the chunk sums left to right -- and
// mean = fl32(sum / n); centred x = fl32(x - mean); per group of 16: s = E4M3_rn(fl32(amax / 6)),
// code = E2M1_rn_sat(fl32(x / deq(s))), codes 0 when s == 0. The scale's division by 6 is IEEE
// (__fdiv_rn); x / deq(s) is the correctly rounded quotient by Markstein's correction (see
// div_rn), the same value as IEEE division.
//
// Layouts written (padded token axis as for FP8: segment s on rows [row0_s, row0_s + L_s)):
//   Q, K codes : u8 [H][Tpad][64]    two E2M1 codes per byte, even channel in the low nibble
//   Q, K scales: u8 [H][Tpad][8]     UE4M3, one per 16 channels
//   V^T codes  : u8 [H][128][Tpad/2] two keys per byte, even key in the low nibble
//   V scales   : u8 [H][Tpad/128][128][8] one per 16 keys (groups start at the segment start);
//                each 128-key tile's scales are one contiguous 1 KB record
//   Q means    : f32 [H][Tpad/128][128]; K means: f32 [num_segments][H][128]
//   q . km     : f32 [H][Tpad], the BF16 query row times its segment's K mean (for the row LSE)
// Padding rows / keys hold code 0 and scale 0.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_lp_internal.h"
#include "sm103_ptx.cuh"

namespace falp {
namespace {

__device__ __forceinline__ float e4m3_value(uint8_t code) {
  const uint32_t h2 = cvt_e4m3x2_to_f16x2(uint16_t(code));
  return __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFF)));
}

// x / d rounded to nearest even, for a normal d and its correctly rounded reciprocal y = RN(1/d),
// by Markstein's correction (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): q = RN(x y) lies within an ulp of
// x / d, the residual r = x - q d is exact in one FMA, and RN(q + r y) = RN(x / d). A zero x keeps
// its sign (x / d would). Checked on GB300 against IEEE division for every E4M3 divisor and every
// dividend with a quotient in [2^-3, 16), both signs (1.5e10 cases), and 4.3e9 random ones.
__device__ __forceinline__ float div_rn(float x, float d, float y) {
  const float q = __fmul_rn(x, y);
  const float r = fmaf(-q, d, x);
  const float q1 = fmaf(r, y, q);
  return x == 0.f ? x : q1;
}

// One 16-element group held by one thread: UE4M3 scale and the 16 E2M1 codes, element 2i in the
// low nibble of byte i.
__device__ __forceinline__ uint2 group16(const float (&x)[16], uint8_t* sf_out) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(x[i]));
  const uint8_t sf = uint8_t(cvt_e4m3x2(__fdiv_rn(a, 6.f), 0.f) & 0xFF);
  *sf_out = sf;
  if (sf == 0) return make_uint2(0u, 0u);
  const float ds = e4m3_value(sf);
  const float y = __frcp_rn(ds);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i >> 2] |= cvt_e2m1x2(div_rn(x[2 * i], ds, y), div_rn(x[2 * i + 1], ds, y)) << (8 * (i & 3));
  return make_uint2(w[0], w[1]);
}

// Pass 1: per (128-row block, head) column sums, equal to the FP64 sums of the rows in order. For
// Q (z = 0) the block is one mean's whole extent: write the block mean. For K (z = 1) store the
// chunk sum. The block's rows are staged in shared memory with 16-byte loads; two threads share a
// column (rows 0-63 and 64-127).
//
// A nonzero BF16 value is +-s 2^k with an integer significand s < 256 and k = exponent - 134
// (subnormals: k = -133). If a column's k span at most 38, every partial sum of the column is a
// multiple of 2^kmin below 2^53 in magnitude, so each FP64 addition of the in-order sum is exact
// and that sum is the exact sum: computed here as an int64 fixed-point sum in any order, then
// converted exactly. Otherwise (rare: values 2^38 apart in one column) the column is summed in
// FP64, rows in order, as the definition reads.
__global__ void __launch_bounds__(256) nvfp4_block_sums_kernel(
    const uint16_t* __restrict__ q, int64_t qst, int64_t qsh, const uint16_t* __restrict__ k,
    int64_t kst, int64_t ksh, const BlockInfo* __restrict__ blocks, int H, int64_t nblk,
    float* __restrict__ qmean, double* __restrict__ kchunk) {
  __shared__ __align__(16) uint16_t tile[kTile][kD + 8];  // +8: rows start on distinct banks
  __shared__ int kmin_s[2][kD], kmax_s[2][kD];
  __shared__ long long part_s[kD];
  const int b = blockIdx.x, h = blockIdx.y, z = blockIdx.z;
  const BlockInfo bi = blocks[b];
  const uint16_t* x = z == 0 ? q : k;
  const int64_t st = z == 0 ? qst : kst, sh = z == 0 ? qsh : ksh;
  // 128 rows x 16 chunks of 8 BF16: all eight loads of a thread in flight, then the stores
  {
    uint4 w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = threadIdx.x + 256 * j, r = i >> 4, c8 = (i & 15) * 8;
      w[j] = make_uint4(0u, 0u, 0u, 0u);
      if (r < bi.nvalid)
        w[j] = __ldg(reinterpret_cast<const uint4*>(x + int64_t(bi.tok0 + r) * st +
                                                    int64_t(h) * sh + c8));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = threadIdx.x + 256 * j, r = i >> 4, c8 = (i & 15) * 8;
      *reinterpret_cast<uint4*>(&tile[r][c8]) = w[j];
    }
  }
  __syncthreads();
  const int c = threadIdx.x & (kD - 1), half = threadIdx.x >> 7;
  const int r0 = half * 64, r1 = min(r0 + 64, bi.nvalid);
  int kmn = 0x7fffffff, kmx = -0x7fffffff;
  for (int r = r0; r < r1; ++r) {
    const uint32_t v = tile[r][c];
    if ((v & 0x7FFFu) == 0) continue;
    const int e = int((v >> 7) & 0xFFu);
    const int kk = e ? e - 134 : -133;
    kmn = min(kmn, kk);
    kmx = max(kmx, kk);
  }
  kmin_s[half][c] = kmn;
  kmax_s[half][c] = kmx;
  __syncthreads();
  kmn = min(kmin_s[0][c], kmin_s[1][c]);
  kmx = max(kmax_s[0][c], kmax_s[1][c]);
  // all zero, or every partial sum exact in FP64 (the same decision for both threads of c)
  const bool exact = kmx < kmn || kmx - kmn <= 38;
  long long acc = 0;
  if (exact) {
    for (int r = r0; r < r1; ++r) {
      const uint32_t v = tile[r][c];
      if ((v & 0x7FFFu) == 0) continue;
      const int e = int((v >> 7) & 0xFFu);
      const long long sig = (e ? 128 : 0) + (v & 0x7Fu);
      const long long mag = sig << ((e ? e - 134 : -133) - kmn);
      acc += (v & 0x8000u) ? -mag : mag;
    }
  }
  if (half == 1) part_s[c] = acc;
  __syncthreads();
  if (half == 1) return;
  double sum = 0.0;
  if (exact) {
    if (kmx >= kmn) sum = ldexp(double(acc + part_s[c]), kmn);
  } else {
    for (int r = 0; r < bi.nvalid; ++r) sum += double(__uint_as_float(uint32_t(tile[r][c]) << 16));
  }
  if (z == 0)
    qmean[(int64_t(h) * nblk + b) * kD + c] = __double2float_rn(sum / double(bi.nvalid));
  else
    kchunk[(int64_t(b) * H + h) * kD + c] = sum;
}

// Pass 2: K segment means from the chunk sums, chunks in order.
__global__ void __launch_bounds__(128) nvfp4_kmean_kernel(const SegInfo* __restrict__ segs, int H,
                                                          const double* __restrict__ kchunk,
                                                          float* __restrict__ kmean) {
  const int s = blockIdx.x, h = blockIdx.y, c = threadIdx.x;
  const SegInfo sg = segs[s];
  float m = 0.f;
  if (sg.len > 0) {
    const int b0 = sg.row0 / kTile;
    double sum = 0.0;
    for (int i = 0; i < sg.nblk; ++i) sum += kchunk[(int64_t(b0 + i) * H + h) * kD + c];
    m = __double2float_rn(sum / double(sg.len));
  }
  kmean[(int64_t(s) * H + h) * kD + c] = m;
}

// Pass 3: Q and K codes and scales. One thread per (row, 16-channel group): 8 threads per row; a
// 256-thread CTA covers 32 rows per step and its 128-row block in 4 steps, every load of a thread
// issued before its arithmetic.
__global__ void __launch_bounds__(256) nvfp4_pack_qk_kernel(
    const uint16_t* __restrict__ q, int64_t qst, int64_t qsh, const uint16_t* __restrict__ k,
    int64_t kst, int64_t ksh, const BlockInfo* __restrict__ blocks, int H, int64_t Tp,
    int64_t nblk, const float* __restrict__ qmean, const float* __restrict__ kmean,
    uint8_t* __restrict__ qc, uint8_t* __restrict__ kc, uint8_t* __restrict__ qs,
    uint8_t* __restrict__ ks, float* __restrict__ qkm) {
  const int b = blockIdx.x, h = blockIdx.y, z = blockIdx.z;
  const int g = threadIdx.x & 7, rr = threadIdx.x >> 3, c0 = 16 * g;
  const BlockInfo bi = blocks[b];
  const uint16_t* x = z == 0 ? q : k;
  const int64_t st = z == 0 ? qst : kst, sh = z == 0 ? qsh : ksh;
  const float* mean = z == 0 ? qmean + (int64_t(h) * nblk + b) * kD
                             : kmean + (int64_t(bi.seg) * H + h) * kD;
  const float* kmu = kmean + (int64_t(bi.seg) * H + h) * kD;  // for q . km (Q only)
  uint8_t* codes = (z == 0 ? qc : kc) + (int64_t(h) * Tp + int64_t(b) * kTile) * 64;
  uint8_t* scales = (z == 0 ? qs : ks) + (int64_t(h) * Tp + int64_t(b) * kTile) * 8;
  uint4 w[4][2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 32 * i + rr;
    w[i][0] = w[i][1] = make_uint4(0u, 0u, 0u, 0u);
    if (r < bi.nvalid) {
      const uint4* src =
          reinterpret_cast<const uint4*>(x + int64_t(bi.tok0 + r) * st + int64_t(h) * sh + c0);
      w[i][0] = __ldg(src);
      w[i][1] = __ldg(src + 1);
    }
  }
  float mu[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) mu[e] = mean[c0 + e];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 32 * i + rr;
    const uint32_t u[8] = {w[i][0].x, w[i][0].y, w[i][0].z, w[i][0].w,
                           w[i][1].x, w[i][1].y, w[i][1].z, w[i][1].w};
    float v[16];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      v[2 * e] = __uint_as_float(u[e] << 16);
      v[2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
    }
    uint2 packed = make_uint2(0u, 0u);
    uint8_t sf = 0;
    if (r < bi.nvalid) {
      float xc[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) xc[e] = __fsub_rn(v[e], mu[e]);
      packed = group16(xc, &sf);
    }
    *reinterpret_cast<uint2*>(codes + int64_t(r) * 64 + 8 * g) = packed;
    scales[int64_t(r) * 8 + g] = sf;
    if (z == 0) {  // the BF16 query row times its segment's K mean (rows past the block: 0)
      float qk = 0.f;
      if (r < bi.nvalid) {
#pragma unroll
        for (int e = 0; e < 16; ++e) qk = fmaf(v[e], kmu[c0 + e], qk);
      }
      qk += __shfl_xor_sync(0xffffffffu, qk, 1);
      qk += __shfl_xor_sync(0xffffffffu, qk, 2);
      qk += __shfl_xor_sync(0xffffffffu, qk, 4);
      if (g == 0) qkm[int64_t(h) * Tp + int64_t(b) * kTile + r] = qk;
    }
  }
}

// Pass 4: V^T codes and scales. One CTA per (128-key block, head): the BF16 tile goes through
// shared memory with 16-byte loads; then one thread per (channel, 16-key group).
__global__ void __launch_bounds__(256) nvfp4_pack_vt_kernel(
    const uint16_t* __restrict__ v, int64_t vst, int64_t vsh, const BlockInfo* __restrict__ blocks,
    int H, int64_t Tp, uint8_t* __restrict__ vt, uint8_t* __restrict__ vs) {
  __shared__ __align__(16) uint16_t tile[kTile][kD + 8];  // +8: rows start on distinct banks
  const int b = blockIdx.x, h = blockIdx.y;
  const BlockInfo bi = blocks[b];
  {  // all eight 16-byte loads of a thread in flight, then the shared-memory stores
    uint4 w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = threadIdx.x + 256 * j, r = i >> 4, c8 = (i & 15) * 8;
      w[j] = make_uint4(0u, 0u, 0u, 0u);
      if (r < bi.nvalid)
        w[j] = __ldg(reinterpret_cast<const uint4*>(v + int64_t(bi.tok0 + r) * vst +
                                                    int64_t(h) * vsh + c8));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = threadIdx.x + 256 * j, r = i >> 4, c8 = (i & 15) * 8;
      *reinterpret_cast<uint4*>(&tile[r][c8]) = w[j];
    }
  }
  __syncthreads();
  // 128 channels x 8 groups; a warp takes 32 consecutive channels of one group
  for (int task = threadIdx.x; task < kD * 8; task += 256) {
    const int c = task & (kD - 1), g = task >> 7;
    float x[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) x[e] = __uint_as_float(uint32_t(tile[16 * g + e][c]) << 16);
    uint8_t sf;
    const uint2 packed = group16(x, &sf);
    *reinterpret_cast<uint2*>(vt + (int64_t(h) * kD + c) * (Tp / 2) + int64_t(b) * (kTile / 2) +
                              8 * g) = packed;
    vs[((int64_t(h) * (Tp / kTile) + b) * kD + c) * 8 + g] = sf;
  }
}

}  // namespace

int launch_nvfp4_quantize(const fa_lp_plan& p, uint8_t* ws, const void* q, int64_t qst,
                          int64_t qsh, const void* k, int64_t kst, int64_t ksh, const void* v,
                          int64_t vst, int64_t vsh, cudaStream_t stream) {
  const int H = p.heads;
  const int64_t nblk = int64_t(p.blocks.size());
  const auto* qb = static_cast<const uint16_t*>(q);
  const auto* kb = static_cast<const uint16_t*>(k);
  const auto* vb = static_cast<const uint16_t*>(v);
  float* qmean = reinterpret_cast<float*>(ws + p.ws.q_mean);
  float* kmean = reinterpret_cast<float*>(ws + p.ws.k_mean);
  double* kchunk = reinterpret_cast<double*>(ws + p.ws.k_chunk);
  nvfp4_block_sums_kernel<<<dim3(unsigned(nblk), unsigned(H), 2), 256, 0, stream>>>(
      qb, qst, qsh, kb, kst, ksh, p.d_blocks, H, nblk, qmean, kchunk);
  nvfp4_kmean_kernel<<<dim3(unsigned(p.nseg), unsigned(H)), 128, 0, stream>>>(p.d_segs, H,
                                                                             kchunk, kmean);
  nvfp4_pack_qk_kernel<<<dim3(unsigned(nblk), unsigned(H), 2), 256, 0, stream>>>(
      qb, qst, qsh, kb, kst, ksh, p.d_blocks, H, p.tpad, nblk, qmean, kmean, ws + p.ws.q_codes,
      ws + p.ws.k_codes, ws + p.ws.q_sf, ws + p.ws.k_sf, reinterpret_cast<float*>(ws + p.ws.q_km));
  nvfp4_pack_vt_kernel<<<dim3(unsigned(nblk), unsigned(H)), 256, 0, stream>>>(
      vb, vst, vsh, p.d_blocks, H, p.tpad, ws + p.ws.v_codes, ws + p.ws.v_sf);
  const int st = cuda_status(cudaGetLastError());
  if (st != FA_LP_OK) return st;
  // the qm K^T table from the means and K codes, when the plan holds all of it (a ring of
  // head-group slots is filled by the forward instead)
  return p.tbl_slots == 1 ? launch_nvfp4_qmk(p, ws, 0, stream) : FA_LP_OK;
}

}  // namespace falp
