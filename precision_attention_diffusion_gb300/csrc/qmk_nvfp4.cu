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
// attention kernel adds Tq to its scores. One launch writes the tables of a group of heads
// [h0, h0 + gridDim.y) into one table slot: segment s at float offset c_off[s] of the slot, then
// [head - h0][nb_s][128 nb_s].
//
// One CTA = one (segment, 128-block M tile, head) and a run of up to 16 256-key N tiles (the plan
// picks the run per segment so that the CTAs fill whole waves; A is built once per CTA; B, the
// MMAs and the stores repeat per N tile). qm is split into three BF16
// pieces (hi + mid + lo carries its 24 significant bits) and deq(Kc) = e2m1 x ue4m3 has at most 6
// significant bits, exact in BF16; one tcgen05.mma kind::f16 stream (M=128, N=256, K=16 steps over
// 3 x 128 channels) accumulates in FP32 in tensor memory. B tiles and accumulators are double
// buffered: the MMAs of tile n run while the 256 threads store tile n - 1 (the table's HBM writes
// bound the kernel) and then build the B tile of n + 1.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_lp_internal.h"
#include "sm103_ptx.cuh"

namespace falp {
namespace {

constexpr int kQmkThreads = 256;
constexpr int kNKeys = 256;                         // keys per N tile
constexpr uint32_t kAChunk = 128 * 128;             // 128 rows x 64 BF16 (one 128-byte row)
constexpr uint32_t kBChunk = kNKeys * 128;          // 256 rows x 64 BF16
// kind::f16: D f32 (1 << 4), A and B BF16 (format 1), both K-major
constexpr uint32_t kIdescQmk = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t(kNKeys) >> 3) << 17) |
                               ((128u >> 4) << 24);
constexpr long long kQmkWaitProbes = 20000;         // ~2 s of parked probes


struct QmkSmem {
  uint8_t a[6][kAChunk];     // qm pieces: piece p, channels 64c..64c+63 -> chunk 2p + c
  uint8_t b[2][2][kBChunk];  // [buffer] deq(Kc): channels 64c..64c+63 -> chunk c
  uint64_t bar[2];           // [buffer]: the MMAs of the tile in that buffer have finished
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

// The codes and scale record of key nt * 256 + kr of the segment (one key per thread); zero past
// the segment. Loaded a tile ahead, so that their latency hides behind the current tile's store.
struct KeyRec {
  uint4 cw[4];
  uint2 sw;
};
__device__ __forceinline__ KeyRec load_key(int nt, int kr, int64_t row0, int lp,
                                           const uint8_t* __restrict__ kcodes,
                                           const uint8_t* __restrict__ ksf) {
  KeyRec r = {};
  const int key = nt * kNKeys + kr;
  if (key < lp) {
    const uint4* src = reinterpret_cast<const uint4*>(kcodes + (row0 + key) * 64);
#pragma unroll
    for (int x = 0; x < 4; ++x) r.cw[x] = src[x];
    r.sw = *reinterpret_cast<const uint2*>(ksf + (row0 + key) * 8);
  }
  return r;
}

// B tile row kr in buffer b from that key's record, dequantized to BF16 (exact).
__device__ __forceinline__ void build_b(QmkSmem& S, int b, int kr, const KeyRec& k) {
  const uint4 (&cw)[4] = k.cw;
  const uint2 sw = k.sw;
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
    *reinterpret_cast<uint4*>(S.b[b][chunk] + sw128(kr, unit)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(S.b[b][chunk] + sw128(kr, unit + 1)) =
        make_uint4(o[4], o[5], o[6], o[7]);
  }
}

__global__ void __launch_bounds__(kQmkThreads, 1) nvfp4_qmk_kernel(
    const QmkItem* __restrict__ items, const SegInfo* __restrict__ segs,
    const int64_t* __restrict__ c_off, const float* __restrict__ qmean,
    const uint8_t* __restrict__ kcodes, const uint8_t* __restrict__ ksf, int64_t Tp,
    int64_t nblk, int h0, float* __restrict__ table, int* err) {
  extern __shared__ uint8_t smem_raw[];
  QmkSmem& S = *reinterpret_cast<QmkSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int i = threadIdx.x, warp = i >> 5, lane = i & 31;
  const QmkItem it = items[blockIdx.x];
  const int hs = blockIdx.y, h = h0 + hs;  // head inside the slot, head
  const SegInfo sg = segs[it.seg];
  const int nb = sg.nblk, lp = sg.nblk * kTile;
  const int64_t krow0 = int64_t(h) * Tp + sg.row0;
  if (i == 0) {
    mbar_init(smem_u32(&S.bar[0]), 1);
    mbar_init(smem_u32(&S.bar[1]), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&S.tmem_base), 512);
    tmem_relinquish();
  }
  // A: row = query block mt * 128 + (i & 127) of the segment, three BF16 pieces of qm; threads
  // i and i + 128 take channels [0, 64) and [64, 128)
  {
    const int ar = i & 127, chalf = i >> 7;
    const int bl = it.mt * 128 + ar;
    const bool valid = bl < nb;
    const float4* qrow =
        reinterpret_cast<const float4*>(qmean + (int64_t(h) * nblk + sg.row0 / kTile + bl) * kD);
    for (int c8 = 64 * chalf; c8 < 64 * chalf + 64; c8 += 8) {  // one 16-byte unit per piece
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
        *reinterpret_cast<uint4*>(S.a[2 * p + chunk] + sw128(ar, unit)) =
            make_uint4(w[p][0], w[p][1], w[p][2], w[p][3]);
    }
  }
  if (it.ntiles > 0) build_b(S, 0, i, load_key(it.nt, i, krow0, lp, kcodes, ksf));
  fence_proxy_async_smem();
  // the barrier after the A / first B build publishes the tensor-memory base
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  // issue the 24 MMAs of the tile in buffer b into accumulator b (tensor-memory columns 256 b)
  auto issue = [&](int b) {
    if (warp == 0) {
      // K step kk (16 channels = 32 bytes): chunk kk / 4, 32-byte offset (kk % 4) in the row
#pragma unroll
      for (int p = 0; p < 3; ++p)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = sdesc_kmajor_sw128(smem_u32(S.a[2 * p + (kk >> 2)]) + 32u * (kk & 3));
          const uint64_t bd = sdesc_kmajor_sw128(smem_u32(S.b[b][kk >> 2]) + 32u * (kk & 3));
          mma_f16_ss_elect(tmem + 256u * uint32_t(b), ad, bd, kIdescQmk,
                           (p > 0 || kk > 0) ? 1u : 0u);
        }
      mma_commit_elect(smem_u32(&S.bar[b]));
    }
  };
  // wait (whole CTA, one decision) for the MMAs of the n-th tile, kept in buffer n & 1
  auto wait_tile = [&](int n) {
    bool done = false;
    for (long long pr = 0; pr < kQmkWaitProbes && !done; ++pr)
      done = mbar_try_wait_sleep(smem_u32(&S.bar[n & 1]), uint32_t(n >> 1) & 1, 100000);
    const bool all = __syncthreads_and(done) != 0;
    if (!all && i == 0) atomicCAS(err, 0, 0x100 | 6);
    return all;
  };
  // store the n-th tile: warp w reads lanes 32 (w & 3) + [0, 32) (query blocks) and columns
  // 128 (w >> 2) + [0, 128) (keys) of accumulator n & 1, and writes them through a 32 x 32
  // transpose in the tile's own B buffer (its MMAs have finished), so that a warp store covers 4
  // rows x 128 contiguous bytes of the table
  auto store = [&](int n) {
    const int nt = it.nt + n;
    const int k0 = 128 * (warp >> 2);
    const int ncol = min(kNKeys, lp - nt * kNKeys) - k0;
    const int row0 = it.mt * 128 + (warp & 3) * 32;
    float* stg = reinterpret_cast<float*>(&S.b[n & 1][0][0]) + warp * (32 * 33);
    const uint32_t taddr = tmem + 256u * uint32_t(n & 1) + uint32_t(k0) + (uint32_t((warp & 3) * 32) << 16);
    const float* base =
        table + c_off[it.seg] + (int64_t(hs) * nb + row0) * lp + int64_t(nt) * kNKeys + k0;
#pragma unroll 1
    for (int c32 = 0; c32 < 128; c32 += 32) {
      uint32_t r[32];
      tmem_ld32(taddr + c32, r);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) stg[lane * 33 + e] = __uint_as_float(r[e]);
      __syncwarp();
      const int cq = 4 * (lane & 7);  // this thread's 4 columns of the chunk
#pragma unroll
      for (int i4 = 0; i4 < 8; ++i4) {
        const int rr = 4 * i4 + (lane >> 3);
        if (row0 + rr < nb && c32 + cq < ncol)
          *reinterpret_cast<float4*>(const_cast<float*>(base) + int64_t(rr) * lp + c32 + cq) =
              make_float4(stg[rr * 33 + cq], stg[rr * 33 + cq + 1], stg[rr * 33 + cq + 2],
                          stg[rr * 33 + cq + 3]);
      }
      __syncwarp();
    }
  };
  bool ok = true;
  int issued = 0;  // tiles whose MMAs were issued (tile m commits to bar[m & 1], phase m >> 1)
  for (int n = 0; n < it.ntiles && ok; ++n) {
    issue(n & 1);  // B tile n is built and visible (barrier at the end of the previous step)
    issued = n + 1;
    // the next tile's key record, in flight during the wait and the store below
    const KeyRec next = n + 1 < it.ntiles ? load_key(it.nt + n + 1, i, krow0, lp, kcodes, ksf)
                                          : KeyRec{};
    if (n > 0) {
      if (!(ok = wait_tile(n - 1))) break;
      tc_fence_after();
      store(n - 1);
      __syncthreads();  // the staging area (B buffer (n + 1) & 1) is rebuilt next
    }
    if (n + 1 < it.ntiles) {
      // buffer (n + 1) & 1 was last read by the MMAs of tile n - 1, finished above
      build_b(S, (n + 1) & 1, i, next);
      fence_proxy_async_smem();
    }
    // B tile n + 1 visible to the MMA issuer; accumulator (n + 1) & 1 (tile n - 1) fully read
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (ok && it.ntiles > 0 && (ok = wait_tile(it.ntiles - 1))) {
    tc_fence_after();
    store(it.ntiles - 1);
  }
  if (!ok) {  // no MMA of this CTA may still be running when its tensor memory is released
    for (int m = max(0, issued - 2); m < issued; ++m)
      for (long long pr = 0; pr < kQmkWaitProbes; ++pr)
        if (mbar_try_wait_sleep(smem_u32(&S.bar[m & 1]), uint32_t(m >> 1) & 1, 100000)) break;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int launch_nvfp4_qmk(const fa_lp_plan& p, uint8_t* ws, int g, cudaStream_t stream) {
  const int h0 = g * p.tbl_hg, nh = std::min(p.tbl_hg, p.heads - h0);
  if (p.qmk_items.empty() || nh <= 0) return FA_LP_OK;
  static std::atomic<uint64_t> smem_set{0};
  if (set_smem_limit_once(reinterpret_cast<const void*>(nvfp4_qmk_kernel), int(kQmkSmemBytes), p.device,
                          smem_set) != FA_LP_OK)
    return FA_LP_ERR_CUDA;
  float* slot = reinterpret_cast<float*>(ws + p.ws.qmk) + size_t(g % p.tbl_slots) * p.tbl_slot_floats;
  nvfp4_qmk_kernel<<<dim3(unsigned(p.qmk_items.size()), unsigned(nh)), kQmkThreads, kQmkSmemBytes,
                     stream>>>(p.d_qmk, p.d_segs, p.d_coff,
                               reinterpret_cast<const float*>(ws + p.ws.q_mean), ws + p.ws.k_codes,
                               ws + p.ws.k_sf, p.tpad, int64_t(p.blocks.size()), h0, slot, p.d_err);
  return cuda_status(cudaGetLastError());
}

}  // namespace falp
