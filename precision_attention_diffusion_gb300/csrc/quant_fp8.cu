// quant_fp8.cu -- FP8 E4M3 quantization of strided BF16 Q/K/V into the attention workspace.
//
// Passage: SGLang PR #40175 "add fp8_fa_sm120 FP8 backend for SM120 GPUs", Modifications
// (fused_prep.py: two passes that quantize strided BF16 Q/K/V views per head straight into the
// kernel buffers -- amax, then pack -- with no FP32 intermediates and no layout copy) and the
// review reply (the pack pass writes every padding position, so a 0xFF-filled workspace keeps no
// undefined byte).
//
// Arithmetic (readings r1-r3): amax over all tokens of a (tensor, head); inv = fl32(448/amax),
// descale = fl32(amax/448) (IEEE divisions, 1 when amax == 0); code = E4M3_rn_satfinite(
// fl32(x * inv)) by the hardware cvt.
//
// Layouts written (padded token axis: segment s occupies rows [row0_s, row0_s + L_s), every
// segment starts on a 128-row boundary, rows past L_s are zero):
//   Q, K codes : u8 [H][Tpad][128]  (K-major tiles for the QK^T tensor-core product)
//   V codes    : u8 [H][128][Tpad]  (V^T, K-major along keys for the PV product)
//   descale    : f32 [3][R][H], R = 1 (one scale per (tensor, head)) or the number of segments
//                (the per-segment mode: amax over the segment's own tokens)
// Both passes are HBM-bound streaming kernels: 16-byte vector loads and stores, grid sized to the
// data (many waves over the 152 SMs).
#include <cuda_bf16.h>

#include "fa_lp_internal.h"
#include "sm103_ptx.cuh"

namespace falp {
namespace {

constexpr int kAmaxTok = 256;  // tokens per amax block

// Pass 1: per (tensor, head) max |x| as the bit pattern of a non-negative float (integer order ==
// float order for non-negative values, so atomicMax is exact and order-independent).
__global__ void __launch_bounds__(256) fp8_amax_kernel(const uint16_t* __restrict__ q,
                                                       int64_t qst, int64_t qsh,
                                                       const uint16_t* __restrict__ k,
                                                       int64_t kst, int64_t ksh,
                                                       const uint16_t* __restrict__ v,
                                                       int64_t vst, int64_t vsh, int64_t T, int H,
                                                       uint32_t* __restrict__ amax) {
  const int z = blockIdx.z, h = blockIdx.y;
  const uint16_t* x = z == 0 ? q : (z == 1 ? k : v);
  const int64_t st = z == 0 ? qst : (z == 1 ? kst : vst);
  const int64_t sh = z == 0 ? qsh : (z == 1 ? ksh : vsh);
  const int64_t t0 = int64_t(blockIdx.x) * kAmaxTok;
  const int64_t t1 = min(T, t0 + kAmaxTok);
  const int tid = threadIdx.x;
  const int sub = tid & 15;  // 16 lanes x 16 bytes = one 256-byte row
  uint32_t m = 0;            // max of (bf16 bits & 0x7FFF) in both halves
  for (int64_t t = t0 + (tid >> 4); t < t1; t += 16) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(x + t * st + int64_t(h) * sh) + sub);
    m = __vmaxu2(m, w.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, w.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, w.z & 0x7FFF7FFFu);
    m = __vmaxu2(m, w.w & 0x7FFF7FFFu);
  }
  m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t red[8];
  if ((tid & 31) == 0) red[tid >> 5] = m;
  __syncthreads();
  if (tid == 0) {
    uint32_t r = red[0];
    for (int i = 1; i < 8; ++i) r = max(r, red[i]);
    atomicMax(amax + z * H + h, r << 16);  // BF16 magnitude -> fp32 bit pattern
  }
}

// Pass 1 of the per-segment mode: per (tensor, segment, head) max |x| over the 128-row blocks of
// the padded token axis (every block lies in one segment), one block of 256 threads per (block,
// head, tensor): 16 lanes x 16 bytes per row, eight rows per thread, loads issued together.
__global__ void __launch_bounds__(256) fp8_amax_seg_kernel(
    const uint16_t* __restrict__ q, int64_t qst, int64_t qsh, const uint16_t* __restrict__ k,
    int64_t kst, int64_t ksh, const uint16_t* __restrict__ v, int64_t vst, int64_t vsh,
    const BlockInfo* __restrict__ blocks, int H, int R, uint32_t* __restrict__ amax) {
  const int b = blockIdx.x, h = blockIdx.y, z = blockIdx.z;
  const BlockInfo bi = blocks[b];
  const uint16_t* x = z == 0 ? q : (z == 1 ? k : v);
  const int64_t st = z == 0 ? qst : (z == 1 ? kst : vst);
  const int64_t sh = z == 0 ? qsh : (z == 1 ? ksh : vsh);
  const int tid = threadIdx.x, sub = tid & 15;
  uint4 w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int r = (tid >> 4) + 16 * j;
    w[j] = make_uint4(0u, 0u, 0u, 0u);
    if (r < bi.nvalid)
      w[j] = __ldg(reinterpret_cast<const uint4*>(x + int64_t(bi.tok0 + r) * st + int64_t(h) * sh) +
                   sub);
  }
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    m = __vmaxu2(m, w[j].x & 0x7FFF7FFFu);
    m = __vmaxu2(m, w[j].y & 0x7FFF7FFFu);
    m = __vmaxu2(m, w[j].z & 0x7FFF7FFFu);
    m = __vmaxu2(m, w[j].w & 0x7FFF7FFFu);
  }
  m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t red[8];
  if ((tid & 31) == 0) red[tid >> 5] = m;
  __syncthreads();
  if (tid == 0) {
    uint32_t r = red[0];
    for (int i = 1; i < 8; ++i) r = max(r, red[i]);
    atomicMax(amax + (int64_t(z) * R + bi.seg) * H + h, r << 16);
  }
}

// Descales of the per-segment mode, one thread per (tensor, segment, head); a segment without
// tokens keeps amax 0 and gets descale 1.
__global__ void fp8_descale_kernel(const uint32_t* __restrict__ amax, int n,
                                   float* __restrict__ descale) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float a = __uint_as_float(amax[i]);
  descale[i] = a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
}

__device__ __forceinline__ float inv_of(uint32_t amax_bits) {
  const float a = __uint_as_float(amax_bits);
  return a > 0.f ? __fdiv_rn(448.f, a) : 1.f;
}

// 8 BF16 (one uint4) times inv -> 8 E4M3 codes (one uint2).
__device__ __forceinline__ uint2 pack8(const uint4 w, float inv) {
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  uint32_t out[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float a = __fmul_rn(__uint_as_float(in[2 * i] << 16), inv);
    const float b = __fmul_rn(__uint_as_float(in[2 * i] & 0xFFFF0000u), inv);
    const float c = __fmul_rn(__uint_as_float(in[2 * i + 1] << 16), inv);
    const float d = __fmul_rn(__uint_as_float(in[2 * i + 1] & 0xFFFF0000u), inv);
    out[i] = uint32_t(cvt_e4m3x2(a, b)) | (uint32_t(cvt_e4m3x2(c, d)) << 16);
  }
  return make_uint2(out[0], out[1]);
}

// Pass 2a: Q and K codes, one block per (128-row block, head, tensor).
__global__ void __launch_bounds__(256) fp8_pack_qk_kernel(
    const uint16_t* __restrict__ q, int64_t qst, int64_t qsh, const uint16_t* __restrict__ k,
    int64_t kst, int64_t ksh, const BlockInfo* __restrict__ blocks, int H, int64_t Tp,
    const uint32_t* __restrict__ amax, int R, uint8_t* __restrict__ qc, uint8_t* __restrict__ kc,
    float* __restrict__ descale) {
  const int b = blockIdx.x, h = blockIdx.y, z = blockIdx.z;
  const BlockInfo bi = blocks[b];
  const uint16_t* x = z == 0 ? q : k;
  const int64_t st = z == 0 ? qst : kst, sh = z == 0 ? qsh : ksh;
  uint8_t* dst = (z == 0 ? qc : kc) + (int64_t(h) * Tp + int64_t(b) * kTile) * kD;
  // R == 1: one scale per (tensor, head), descales written here; R == nseg: per segment, the
  // descales come from fp8_descale_kernel
  const uint32_t ab = amax[(int64_t(z) * R + (R > 1 ? bi.seg : 0)) * H + h];
  const float inv = inv_of(ab);
  if (R == 1 && b == 0 && threadIdx.x == 0) {
    const float a = __uint_as_float(ab);
    descale[z * H + h] = a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
  }
  const int sub = threadIdx.x & 15;
#pragma unroll 4
  for (int r = threadIdx.x >> 4; r < kTile; r += 16) {
    uint2 c = make_uint2(0u, 0u);
    if (r < bi.nvalid) {
      const uint4 w =
          __ldg(reinterpret_cast<const uint4*>(x + int64_t(bi.tok0 + r) * st + int64_t(h) * sh) + sub);
      c = pack8(w, inv);
    }
    reinterpret_cast<uint2*>(dst + int64_t(r) * kD)[sub] = c;
  }
}

// Pass 2b: V^T codes, one block per (128-row block, head): quantize a 128-token x 128-channel
// tile into shared memory, then write it transposed (128 channel rows x 128 key bytes).
__global__ void __launch_bounds__(256) fp8_pack_vt_kernel(const uint16_t* __restrict__ v,
                                                          int64_t vst, int64_t vsh,
                                                          const BlockInfo* __restrict__ blocks,
                                                          int H, int64_t Tp,
                                                          const uint32_t* __restrict__ amax,
                                                          int R, uint8_t* __restrict__ vt,
                                                          float* __restrict__ descale) {
  __shared__ __align__(16) uint8_t tile[kTile][kD + 4];
  const int b = blockIdx.x, h = blockIdx.y;
  const BlockInfo bi = blocks[b];
  const uint32_t ab = amax[(2 * int64_t(R) + (R > 1 ? bi.seg : 0)) * H + h];
  const float inv = inv_of(ab);
  if (R == 1 && b == 0 && threadIdx.x == 0) {
    const float a = __uint_as_float(ab);
    descale[2 * H + h] = a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
  }
  const int sub = threadIdx.x & 15;
  {
    // all eight 16-byte loads of a thread in flight before any is packed
    uint4 w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = (threadIdx.x >> 4) + 16 * j;
      w[j] = make_uint4(0u, 0u, 0u, 0u);
      if (r < bi.nvalid)
        w[j] = __ldg(reinterpret_cast<const uint4*>(v + int64_t(bi.tok0 + r) * vst +
                                                    int64_t(h) * vsh) + sub);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = (threadIdx.x >> 4) + 16 * j;
      const uint2 c = r < bi.nvalid ? pack8(w[j], inv) : make_uint2(0u, 0u);
      uint32_t* row = reinterpret_cast<uint32_t*>(&tile[r][sub * 8]);
      row[0] = c.x;
      row[1] = c.y;
    }
  }
  __syncthreads();
  uint8_t* dst = vt + int64_t(h) * kD * Tp + int64_t(b) * kTile;
  for (int i = threadIdx.x; i < kD * 8; i += 256) {
    const int chunk = i & 7, c = i >> 3;  // 8 threads write one channel row of 128 keys
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = chunk * 16 + 4 * j;
      w[j] = uint32_t(tile[r][c]) | (uint32_t(tile[r + 1][c]) << 8) |
             (uint32_t(tile[r + 2][c]) << 16) | (uint32_t(tile[r + 3][c]) << 24);
    }
    *reinterpret_cast<uint4*>(dst + int64_t(c) * Tp + chunk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__global__ void encode_kernel(int format, const float* __restrict__ x, int64_t n,
                              uint8_t* __restrict__ codes) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  if (format == 0) {
    codes[i] = static_cast<uint8_t>(cvt_e4m3x2(x[i], 0.f) & 0xFF);
  } else {
    codes[i] = cvt_e2m1x2(x[i], 0.f) & 0xF;
  }
}

}  // namespace

int launch_fp8_quantize(const fa_lp_plan& p, uint8_t* ws, const void* q, int64_t qst, int64_t qsh,
                        const void* k, int64_t kst, int64_t ksh, const void* v, int64_t vst,
                        int64_t vsh, cudaStream_t stream) {
  const int H = p.heads, R = fp8_scale_rows(p);
  uint32_t* amax = reinterpret_cast<uint32_t*>(ws + p.ws.amax);
  float* descale = reinterpret_cast<float*>(ws + p.ws.descale);
  if (cudaMemsetAsync(amax, 0, size_t(3) * R * H * sizeof(uint32_t), stream) != cudaSuccess)
    return FA_LP_ERR_CUDA;
  const auto* qb = static_cast<const uint16_t*>(q);
  const auto* kb = static_cast<const uint16_t*>(k);
  const auto* vb = static_cast<const uint16_t*>(v);
  const unsigned nblk = unsigned(p.blocks.size());
  if (R == 1) {
    dim3 g1(unsigned((p.tokens + kAmaxTok - 1) / kAmaxTok), unsigned(H), 3);
    fp8_amax_kernel<<<g1, 256, 0, stream>>>(qb, qst, qsh, kb, kst, ksh, vb, vst, vsh, p.tokens, H,
                                            amax);
  } else {
    dim3 g1(nblk, unsigned(H), 3);
    fp8_amax_seg_kernel<<<g1, 256, 0, stream>>>(qb, qst, qsh, kb, kst, ksh, vb, vst, vsh,
                                                p.d_blocks, H, R, amax);
    const int n = 3 * R * H;
    fp8_descale_kernel<<<(n + 255) / 256, 256, 0, stream>>>(amax, n, descale);
  }
  dim3 g2(nblk, unsigned(H), 2);
  fp8_pack_qk_kernel<<<g2, 256, 0, stream>>>(qb, qst, qsh, kb, kst, ksh, p.d_blocks, H, p.tpad,
                                             amax, R, ws + p.ws.q_codes, ws + p.ws.k_codes,
                                             descale);
  dim3 g3(nblk, unsigned(H));
  fp8_pack_vt_kernel<<<g3, 256, 0, stream>>>(vb, vst, vsh, p.d_blocks, H, p.tpad, amax, R,
                                             ws + p.ws.v_codes, descale);
  return cuda_status(cudaGetLastError());
}

int launch_encode(int format, const float* x, int64_t n, uint8_t* codes, cudaStream_t stream) {
  const int64_t blocks = (n + 255) / 256;
  encode_kernel<<<unsigned(blocks), 256, 0, stream>>>(format, x, n, codes);
  return cuda_status(cudaGetLastError());
}

}  // namespace falp
