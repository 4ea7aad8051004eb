// qmk_nvfp4.cu -- the qm K^T term of NVFP4 attention as a table, on the BF16 tensor cores.
//
// Passage: FlashInfer docs, flashinfer.diffusion_ops.minimax_h3_sm120_varlen_attention_nvfp4,
// description: Q is centred by its 128-row block mean qm and the qm K^T term is added back to the
// scores. The term does not depend on the query row inside a block, so for every segment s and
// head h it is the product of the block means and the dequantized centred keys (reading r12):
//
//     Tq[s][h][b][j] = qm_b . deq(Kc_j)                                  (raw units of S)
//
// for the segment's query blocks b and its padded keys j (zero codes past the segment). The
// attention kernel adds Tq to its scores. Layout: segment s at float offset c_off[s], then
// [H][nb_s][128 nb_s].
//
// One CTA = one (segment, 128-block M tile, head) and a run of up to kQmkTilesPer 256-key N tiles
// (A is built once per CTA; B, the MMAs and the stores repeat per N tile). qm is split into three BF16
// pieces (hi + mid + lo carries its 24 significant bits) and deq(Kc) = e2m1 x ue4m3 has at most 6
// significant bits, exact in BF16; one tcgen05.mma kind::f16 stream (M=128, N=256, K=16 steps over
// 3 x 128 channels) accumulates in FP32 in tensor memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_lp_internal.h"
#include "sm103_ptx.cuh"

namespace falp {
namespace {

constexpr int kQmkThreads = 128;
constexpr int kNKeys = 256;                         // keys per N tile
constexpr uint32_t kAChunk = 128 * 128;             // 128 rows x 64 BF16 (one 128-byte row)
constexpr uint32_t kBChunk = kNKeys * 128;          // 256 rows x 64 BF16
// kind::f16: D f32 (1 << 4), A and B BF16 (format 1), both K-major
constexpr uint32_t kIdescQmk = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t(kNKeys) >> 3) << 17) |
                               ((128u >> 4) << 24);
constexpr long long kQmkWaitProbes = 20000;         // ~2 s of parked probes


struct QmkSmem {
  uint8_t a[6][kAChunk];  // qm pieces: piece p, channels 64c..64c+63 -> chunk 2p + c
  uint8_t b[2][kBChunk];  // deq(Kc): channels 64c..64c+63 -> chunk c
  uint64_t bar;
  uint32_t tmem_base;
};
constexpr size_t kQmkSmemBytes = sizeof(QmkSmem) + 1024;

// byte offset of (row r, 16-byte unit u) in a K-major chunk with 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(int r, int u) {
  return uint32_t(r) * 128u + (uint32_t(u ^ (r & 7)) << 4);
}

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float e4m3f(uint32_t code) {
  const uint32_t h2 = cvt_e4m3x2_to_f16x2(uint16_t(code & 0xFF));
  return __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFF)));
}

__global__ void __launch_bounds__(kQmkThreads, 1) nvfp4_qmk_kernel(
    const QmkItem* __restrict__ items, const SegInfo* __restrict__ segs,
    const int64_t* __restrict__ c_off, const float* __restrict__ qmean,
    const uint8_t* __restrict__ kcodes, const uint8_t* __restrict__ ksf, int64_t Tp,
    int64_t nblk, int H, float* __restrict__ table, int* err) {
  extern __shared__ uint8_t smem_raw[];
  QmkSmem& S = *reinterpret_cast<QmkSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int i = threadIdx.x, warp = i >> 5, lane = i & 31;
  const QmkItem it = items[blockIdx.x];
  const int h = blockIdx.y;
  const SegInfo sg = segs[it.seg];
  const int nb = sg.nblk, lp = sg.nblk * kTile;
  if (i == 0) {
    mbar_init(smem_u32(&S.bar), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&S.tmem_base), 256);
    tmem_relinquish();
  }
  // A: row i = query block mt * 128 + i of the segment, three BF16 pieces of qm
  {
    const int bl = it.mt * 128 + i;
    const bool valid = bl < nb;
    const float4* qrow =
        reinterpret_cast<const float4*>(qmean + (int64_t(h) * nblk + sg.row0 / kTile + bl) * kD);
    for (int c8 = 0; c8 < kD; c8 += 8) {  // 8 channels = one 16-byte unit per piece
      uint32_t w[3][4];
      float xv[8];
      {
        const float4 f0 = valid ? qrow[c8 / 4] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 f1 = valid ? qrow[c8 / 4 + 1] : make_float4(0.f, 0.f, 0.f, 0.f);
        xv[0] = f0.x; xv[1] = f0.y; xv[2] = f0.z; xv[3] = f0.w;
        xv[4] = f1.x; xv[5] = f1.y; xv[6] = f1.z; xv[7] = f1.w;
      }
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        float x0 = xv[e], x1 = xv[e + 1];
#pragma unroll
        for (int p = 0; p < 3; ++p) {
          const uint32_t v = bf16x2(x0, x1);
          w[p][e >> 1] = v;
          // the remainder is exact in FP32 (x and its BF16 rounding share the leading bits)
          x0 = x0 - __uint_as_float(v << 16);
          x1 = x1 - __uint_as_float(v & 0xFFFF0000u);
        }
      }
      const int chunk = c8 >> 6, unit = (c8 & 63) >> 3;
#pragma unroll
      for (int p = 0; p < 3; ++p)
        *reinterpret_cast<uint4*>(S.a[2 * p + chunk] + sw128(i, unit)) =
            make_uint4(w[p][0], w[p][1], w[p][2], w[p][3]);
    }
  }
  // the barrier after the A build publishes the tensor-memory base
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  bool ok = true;
  for (int n = 0; n < it.ntiles && ok; ++n) {
    const int nt = it.nt + n;
    if (n > 0) {  // the previous tile's MMAs have finished (waited below); B may be rewritten
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
    // B: rows i and i + 128 = keys nt * 256 + row of the segment, dequantized to BF16 (exact)
    for (int kr = i; kr < kNKeys; kr += kQmkThreads) {
      const int key = nt * kNKeys + kr;
      const bool valid = key < lp;
      const int64_t row = int64_t(h) * Tp + sg.row0 + key;
      uint4 cw[4] = {};
      uint2 sw = make_uint2(0u, 0u);
      if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(kcodes + row * 64);
  #pragma unroll
        for (int x = 0; x < 4; ++x) cw[x] = src[x];
        sw = *reinterpret_cast<const uint2*>(ksf + row * 8);
      }
      const uint32_t words[16] = {cw[0].x, cw[0].y, cw[0].z, cw[0].w, cw[1].x, cw[1].y,
                                  cw[1].z, cw[1].w, cw[2].x, cw[2].y, cw[2].z, cw[2].w,
                                  cw[3].x, cw[3].y, cw[3].z, cw[3].w};
  #pragma unroll
      for (int g = 0; g < 8; ++g) {  // 16 channels: words 2g, 2g + 1; scale byte g
        const float ds = e4m3f((g < 4 ? sw.x : sw.y) >> (8 * (g & 3)));
        uint32_t o[8];
  #pragma unroll
        for (int bq = 0; bq < 8; ++bq) {
          const uint32_t byte = (words[2 * g + (bq >> 2)] >> (8 * (bq & 3))) & 0xFFu;
          const uint32_t h2 = cvt_e2m1x2_to_f16x2(byte);
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
          o[bq] = bf16x2(f.x * ds, f.y * ds);  // e2m1 x ue4m3: exact in FP32 and in BF16
        }
        const int c = 16 * g;  // first channel of the group
        const int chunk = c >> 6, unit = (c & 63) >> 3;
        *reinterpret_cast<uint4*>(S.b[chunk] + sw128(kr, unit)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(S.b[chunk] + sw128(kr, unit + 1)) =
            make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {
      // K step kk (16 channels = 32 bytes): chunk kk / 4, 32-byte offset (kk % 4) in the row
  #pragma unroll
      for (int p = 0; p < 3; ++p)
  #pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = sdesc_kmajor_sw128(smem_u32(S.a[2 * p + (kk >> 2)]) + 32u * (kk & 3));
          const uint64_t bd = sdesc_kmajor_sw128(smem_u32(S.b[kk >> 2]) + 32u * (kk & 3));
          mma_f16_ss_elect(tmem, ad, bd, kIdescQmk, (p > 0 || kk > 0) ? 1u : 0u);
        }
      mma_commit_elect(smem_u32(&S.bar));
    }
    bool done = false;
    for (long long pr = 0; pr < kQmkWaitProbes && !done; ++pr)
      done = mbar_try_wait_sleep(smem_u32(&S.bar), uint32_t(n) & 1, 100000);
    // one decision for the whole CTA, so that every thread leaves the loop together
    ok = __syncthreads_and(done) != 0;
    if (!ok) {
      if (i == 0) atomicCAS(err, 0, 0x100 | 6);
    } else {
      tc_fence_after();
      // D row = lane of this warp's quarter = query block; 256 key columns
      const int bl = it.mt * 128 + warp * 32 + lane;
      const bool valid = bl < nb;
      float* dst = table + c_off[it.seg] + (int64_t(h) * nb + bl) * lp + int64_t(nt) * kNKeys;
      const int ncol = min(kNKeys, lp - nt * kNKeys);
      const uint32_t taddr = tmem + (uint32_t(warp * 32) << 16);
  #pragma unroll
      for (int c32 = 0; c32 < kNKeys; c32 += 32) {
        uint32_t r[32];
        tmem_ld32(taddr + c32, r);
        tmem_wait_ld();
        if (valid && c32 < ncol) {
  #pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + c32 + e) =
                make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                            __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace

int launch_nvfp4_qmk(const fa_lp_plan& p, uint8_t* ws, cudaStream_t stream) {
  if (p.qmk_items.empty()) return FA_LP_OK;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(nvfp4_qmk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kQmkSmemBytes)) != cudaSuccess)
      return FA_LP_ERR_CUDA;
    attr_set = true;
  }
  nvfp4_qmk_kernel<<<dim3(unsigned(p.qmk_items.size()), unsigned(p.heads)), kQmkThreads,
                     kQmkSmemBytes, stream>>>(
      p.d_qmk, p.d_segs, p.d_coff, reinterpret_cast<const float*>(ws + p.ws.q_mean),
      ws + p.ws.k_codes, ws + p.ws.k_sf, p.tpad, int64_t(p.blocks.size()), p.heads,
      reinterpret_cast<float*>(ws + p.ws.qmk), p.d_err);
  return cuda_status(cudaGetLastError());
}

}  // namespace falp
