// attn_fp8.cu -- FP8 E4M3 packed-varlen attention forward on 5th-generation tensor cores.
//
// Passage: SGLang PR #40175 "add fp8_fa_sm120 FP8 backend for SM120 GPUs", Modifications
// (kernel.py: E4M3 QK and PV with FP32 accumulation, online softmax, K/V prefetch overlapping the
// math, probabilities packed to E4M3 without a shared-memory round trip); FlashInfer docs,
// minimax_h3_sm120_varlen_attention_nvfp4, description (non-causal packed varlen over cu_seqlens,
// empty segments and segments shorter than a tile, output rounded to BF16 once).
//
// GB300 design (the SM120 kernel's 128x32 mma.sync tile is prior art, not the blueprint):
//   * one CTA = one (segment, head) and two 128-row query tiles Q0, Q1 sharing every K/V tile;
//   * warp 8 issues TMA loads (Q once; K_j and V^T_j into a 3-stage ring, 128-byte swizzle);
//   * warp 9 allocates the 512 tensor-memory columns and issues tcgen05.mma kind::f8f6f4:
//       S_t = Q_t K_j^T   (A, B from shared memory, FP32 accumulator in TMEM columns [128t, +128))
//       O_t += P_t V_j    (A = P_t from TMEM, E4M3, 4 per column; O_t in columns [256+128t, +128))
//     in the order S0_0 S1_0 | PV0_j S0_{j+1} PV1_j S1_{j+1} ..., so that one tile's softmax
//     overlaps the other tile's tensor work;
//   * warps 0-3 / 4-7 run the online softmax of Q0 / Q1, one thread per query row (row == TMEM
//     lane). The reference maximum m is the first tile's maximum and moves to a later tile's
//     maximum M only when (M - m) c > 8 (reading r5 with tau = 8; the pages leave the rule open):
//       alpha = 2^((m - m') c);  P_j = E4M3(2^(S_j c - m' c)) <= 256
//       l = l alpha + sum_j P_j (the quantized P, reading r6);  O = O alpha before P V_j
//       accumulates (only when some row of the warp moved its reference; alpha == 1 otherwise),
//     where S is the raw E4M3 dot product and c = dq dk softmax_scale log2(e);
//   * epilogue: out = BF16_rn(O dv / l) for rows inside the segment only.
// Every barrier wait is bounded; on expiry the kernel records an error, drains its in-flight
// copies and MMAs, frees its tensor memory and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_lp_internal.h"
#include "sm103_ptx.cuh"

namespace falp {
namespace {

constexpr int kStages = 3;
constexpr int kThreads = 320;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTileBytes = 128 * 128;
constexpr uint32_t kIdesc = idesc_f8f6f4(128, 128, 0, 0);  // E4M3 x E4M3 -> F32, M=N=128
constexpr long long kDrainSpins = 1ll << 20;
// Threshold (log2 units) by which a key tile's maximum must exceed the reference maximum before
// the reference moves (and O, l are rescaled). P = 2^(S c - m c) <= 2^kTau stays inside E4M3.
constexpr float kTau = 8.0f;

struct Smem {
  uint8_t q[2][kTileBytes];
  uint8_t k[kStages][kTileBytes];
  uint8_t v[kStages][kTileBytes];
  uint64_t bar_q;
  uint64_t bar_k[kStages];
  uint64_t bar_v[kStages];
  uint64_t bar_free[kStages];
  uint64_t bar_s[2];
  uint64_t bar_p[2];
  uint64_t bar_o[2];
  uint64_t bar_drain;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

struct AttnArgs {
  const SegInfo* segs;
  const WorkItem* work;
  const float* descale;  // [3][H]
  __nv_bfloat16* out;
  int64_t ost, osh;
  float scale_log2;
  int H;
  int* err;          // sticky error word of the plan (read and cleared by the host)
  int* abort_word;   // launch generation that aborted, shared by every CTA of the launch
  int gen;           // this launch's generation
  long long spin_limit;
};

enum Role : int { kRoleProducer = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleEpilogue = 4 };

// Bounded wait on one mbarrier phase. Returns false when the CTA aborts (this wait expired, or
// another role's did).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, Smem& S,
                                           const AttnArgs& a, int role) {
  long long n = 0;
  while (!mbar_try_wait(bar, parity)) {
    if (*reinterpret_cast<volatile int*>(&S.abort_flag)) return false;
    ++n;
    // another CTA of this launch gave up: stop too (polled rarely, off the fast path)
    if ((n & 1023) == 0 && *reinterpret_cast<volatile int*>(a.abort_word) == a.gen) {
      *reinterpret_cast<volatile int*>(&S.abort_flag) = 1;
      return false;
    }
    if (n >= a.spin_limit) {
      *reinterpret_cast<volatile int*>(&S.abort_flag) = 1;
      atomicExch(a.abort_word, a.gen);
      atomicCAS(a.err, 0, 0x100 | role);
      return false;
    }
  }
  return true;
}

// Wait used while draining after an abort: ignores the abort flag, bounded separately.
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity) {
  for (long long n = 0; n < kDrainSpins; ++n)
    if (mbar_try_wait(bar, parity)) return;
}

__device__ __forceinline__ void producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                         const CUtensorMap* tm_v, Smem& S, const AttnArgs& a,
                                         const WorkItem& wi, const SegInfo& sg) {
  const int n_kv = sg.nblk;
  const int rq = sg.row0 + wi.qt0 * kTile;
  mbar_arrive_expect_tx(smem_u32(&S.bar_q), uint32_t(wi.nq) * kTileBytes);
  tma_load_3d(smem_u32(S.q[0]), tm_q, smem_u32(&S.bar_q), 0, rq, wi.head);
  if (wi.nq == 2) tma_load_3d(smem_u32(S.q[1]), tm_q, smem_u32(&S.bar_q), 0, rq + kTile, wi.head);
  int issued = 0;
  for (int j = 0; j < n_kv; ++j) {
    const int st = j % kStages;
    if (j >= kStages &&
        !wait_phase(smem_u32(&S.bar_free[st]), ((j / kStages) - 1) & 1, S, a, kRoleProducer))
      break;
    const int row = sg.row0 + j * kTile;
    mbar_arrive_expect_tx(smem_u32(&S.bar_k[st]), kTileBytes);
    tma_load_3d(smem_u32(S.k[st]), tm_k, smem_u32(&S.bar_k[st]), 0, row, wi.head);
    mbar_arrive_expect_tx(smem_u32(&S.bar_v[st]), kTileBytes);
    tma_load_3d(smem_u32(S.v[st]), tm_v, smem_u32(&S.bar_v[st]), row, 0, wi.head);
    issued = j + 1;
  }
  // No copy may still be landing in shared memory when the CTA exits.
  drain_phase(smem_u32(&S.bar_q), 0);
  for (int j = max(0, issued - kStages); j < issued; ++j) {
    const int st = j % kStages;
    drain_phase(smem_u32(&S.bar_k[st]), (j / kStages) & 1);
    drain_phase(smem_u32(&S.bar_v[st]), (j / kStages) & 1);
  }
}

__device__ __forceinline__ void mma_issuer(Smem& S, const AttnArgs& a, const WorkItem& wi,
                                           const SegInfo& sg, uint32_t tmem) {
  const int n_kv = sg.nblk;
  const int nq = wi.nq;
  const uint32_t s_t[2] = {tmem, tmem + 128};
  const uint32_t o_t[2] = {tmem + 256, tmem + 384};
  const uint32_t qa[2] = {smem_u32(S.q[0]), smem_u32(S.q[1])};
  auto issue_s = [&](int t, int st) {
    const uint32_t kb = smem_u32(S.k[st]);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_f8f6f4_ss(s_t[t], sdesc_kmajor_sw128(qa[t] + 32 * kk), sdesc_kmajor_sw128(kb + 32 * kk),
                    kIdesc, kk > 0);
    mma_commit(smem_u32(&S.bar_s[t]));
  };
  auto issue_pv = [&](int t, int st, bool acc) {
    const uint32_t vb = smem_u32(S.v[st]);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_f8f6f4_ts(o_t[t], s_t[t] + 8 * kk, sdesc_kmajor_sw128(vb + 32 * kk), kIdesc,
                    (acc || kk > 0) ? 1u : 0u);
    mma_commit(smem_u32(&S.bar_o[t]));
  };
  do {
    if (!wait_phase(smem_u32(&S.bar_q), 0, S, a, kRoleMma)) break;
    if (!wait_phase(smem_u32(&S.bar_k[0]), 0, S, a, kRoleMma)) break;
    tc_fence_after();
    issue_s(0, 0);
    if (nq == 2) issue_s(1, 0);
    for (int j = 0; j < n_kv; ++j) {
      const int st = j % kStages;
      const int j1 = j + 1, st1 = j1 % kStages;
      if (!wait_phase(smem_u32(&S.bar_v[st]), (j / kStages) & 1, S, a, kRoleMma)) break;
      if (!wait_phase(smem_u32(&S.bar_p[0]), j & 1, S, a, kRoleMma)) break;
      tc_fence_after();
      issue_pv(0, st, j > 0);
      if (j1 < n_kv) {
        if (!wait_phase(smem_u32(&S.bar_k[st1]), (j1 / kStages) & 1, S, a, kRoleMma)) break;
        tc_fence_after();
        issue_s(0, st1);
      }
      if (nq == 2) {
        if (!wait_phase(smem_u32(&S.bar_p[1]), j & 1, S, a, kRoleMma)) break;
        tc_fence_after();
        issue_pv(1, st, j > 0);
      }
      mma_commit(smem_u32(&S.bar_free[st]));
      if (nq == 2 && j1 < n_kv) issue_s(1, st1);
    }
  } while (false);
  // Every MMA issued so far must finish before the tensor memory is released.
  mma_commit(smem_u32(&S.bar_drain));
  drain_phase(smem_u32(&S.bar_drain), 0);
}

// Row maximum of 128 values: eight independent 3-input-max chains, then a 3-level combine
// (depth 10 instead of a 127-deep serial chain).
__device__ __forceinline__ float row_max128(const float (&s)[128]) {
  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    acc[k] = s[k];
#pragma unroll
    for (int i = 1; i < 16; i += 2)
      acc[k] = max3f(acc[k], s[k + 8 * i], s[k + 8 * (i + 1 < 16 ? i + 1 : i)]);
  }
  return max3f(max3f(acc[0], acc[1], acc[2]), max3f(acc[3], acc[4], acc[5]), fmaxf(acc[6], acc[7]));
}

__device__ __forceinline__ void softmax_and_epilogue(Smem& S, const AttnArgs& a,
                                                     const WorkItem& wi, const SegInfo& sg,
                                                     uint32_t tmem, int t, int wq, int lane) {
  const int n_kv = sg.nblk;
  const int h = wi.head;
  const float c = a.descale[h] * a.descale[a.H + h] * a.scale_log2;
  const float dv = a.descale[2 * a.H + h];
  const uint32_t lane_off = uint32_t(wq * 32) << 16;
  const uint32_t s_addr = tmem + uint32_t(128 * t) + lane_off;
  const uint32_t o_addr = tmem + 256u + uint32_t(128 * t) + lane_off;
  const int last_valid = sg.len - (n_kv - 1) * kTile;  // keys of the last tile, 1..128
  float m = -INFINITY, l = 0.f;                          // reference maximum (raw units), sum
  bool ok = true;
  for (int j = 0; j < n_kv; ++j) {
    ok = __all_sync(0xffffffffu, wait_phase(smem_u32(&S.bar_s[t]), j & 1, S, a, kRoleSoftmax));
    if (!ok) break;
    tc_fence_after();
    uint32_t r[4][32];
#pragma unroll
    for (int i = 0; i < 4; ++i) tmem_ld32(s_addr + 32 * i, r[i]);
    tmem_wait_ld();
    float s[128];
#pragma unroll
    for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(r[i >> 5][i & 31]);
    if (j == n_kv - 1 && last_valid < kTile) {
#pragma unroll
      for (int i = 0; i < 128; ++i)
        if (i >= last_valid) s[i] = -INFINITY;
    }
    // Reference maximum: moves only when the tile's maximum exceeds it by more than kTau (log2
    // units), so P stays below 2^kTau = 256 < 448 and O needs rescaling only on such moves.
    const float mx = row_max128(s);
    const bool move = (m == -INFINITY) || ((mx - m) * c > kTau);
    const float m_new = move ? mx : m;
    const float alpha = move ? ex2_approx((m - m_new) * c) : 1.f;  // m = -inf gives 0
    const float nmc = -m_new * c;
    uint32_t pk[32];
    float rs = 0.f;
#pragma unroll
    for (int g = 0; g < 4; ++g) {  // 32 keys per group
      uint32_t hs[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // 4 keys
        const int k0 = 32 * g + 4 * i;
        float x0, x1, x2, x3;
        fma2(x0, x1, s[k0], s[k0 + 1], c, nmc);
        fma2(x2, x3, s[k0 + 2], s[k0 + 3], c, nmc);
        const uint16_t c01 = cvt_e4m3x2(ex2_approx(x0), ex2_approx(x1));
        const uint16_t c23 = cvt_e4m3x2(ex2_approx(x2), ex2_approx(x3));
        pk[8 * g + i] = uint32_t(c01) | (uint32_t(c23) << 16);
        // the quantized values, back in f16 (exact), summed pairwise
        hs[i] = hadd2_u32(cvt_e4m3x2_to_f16x2(c01), cvt_e4m3x2_to_f16x2(c23));
      }
      const uint32_t h4 = hadd2_u32(hadd2_u32(hadd2_u32(hs[0], hs[1]), hadd2_u32(hs[2], hs[3])),
                                    hadd2_u32(hadd2_u32(hs[4], hs[5]), hadd2_u32(hs[6], hs[7])));
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h4));
      rs += f.x + f.y;
    }
    l = l * alpha + rs;
    tmem_st32(s_addr, pk);
    if (j > 0 && __any_sync(0xffffffffu, move)) {
      ok = __all_sync(0xffffffffu,
                      wait_phase(smem_u32(&S.bar_o[t]), (j - 1) & 1, S, a, kRoleSoftmax));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t o[32];
        tmem_ld32(o_addr + 32 * i, o);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st32(o_addr + 32 * i, o);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(smem_u32(&S.bar_p[t]));
    m = m_new;
  }
  if (!ok) return;
  ok = __all_sync(0xffffffffu,
                  wait_phase(smem_u32(&S.bar_o[t]), (n_kv - 1) & 1, S, a, kRoleEpilogue));
  if (!ok) return;
  tc_fence_after();
  const float f = dv / l;
  const int qrow = (wi.qt0 + t) * kTile + wq * 32 + lane;
  const bool valid = qrow < sg.len;
  __nv_bfloat16* dst = a.out + int64_t(sg.tok0 + qrow) * a.ost + int64_t(h) * a.osh;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t o[32];
    tmem_ld32(o_addr + 32 * i, o);
    tmem_wait_ld();
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(o[2 * e]) * f,
                                                     __uint_as_float(o[2 * e + 1]) * f);
      w[e] = *reinterpret_cast<const uint32_t*>(&b);
    }
    if (valid) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * i);
#pragma unroll
      for (int e = 0; e < 4; ++e) d4[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_fp8_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WorkItem wi = a.work[blockIdx.x];
  const SegInfo sg = a.segs[wi.seg];

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&S.bar_q), 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&S.bar_k[i]), 1);
      mbar_init(smem_u32(&S.bar_v[i]), 1);
      mbar_init(smem_u32(&S.bar_free[i]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&S.bar_s[t]), 1);
      mbar_init(smem_u32(&S.bar_p[t]), 128);
      mbar_init(smem_u32(&S.bar_o[t]), 1);
    }
    mbar_init(smem_u32(&S.bar_drain), 1);
    S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kTmaWarp && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&S.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == kTmaWarp) {
    if (lane == 0) producer(&tm_q, &tm_k, &tm_v, S, a, wi, sg);
  } else if (warp == kMmaWarp) {
    if (lane == 0) mma_issuer(S, a, wi, sg, tmem);
    __syncwarp();
  } else {
    const int t = warp >> 2;
    if (t < wi.nq) softmax_and_epilogue(S, a, wi, sg, tmem, t, warp & 3, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int launch_fp8_attention(const fa_lp_plan& p, uint8_t* ws, void* out, int64_t ost, int64_t osh,
                         cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attn_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSmemBytes)) != cudaSuccess)
      return FA_LP_ERR_CUDA;
    attr_set = true;
  }
  const uint64_t H = uint64_t(p.heads), Tp = uint64_t(p.tpad);
  CUtensorMap tq, tk, tv;
  int st = encode_tmap_3d_u8(&tq, ws + p.ws.q_codes, 128, Tp, H, 128, Tp * 128, 128, 128,
                             CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == FA_LP_OK)
    st = encode_tmap_3d_u8(&tk, ws + p.ws.k_codes, 128, Tp, H, 128, Tp * 128, 128, 128,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == FA_LP_OK)
    st = encode_tmap_3d_u8(&tv, ws + p.ws.v_codes, Tp, 128, H, Tp, Tp * 128, 128, 128,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != FA_LP_OK) return st;
  AttnArgs a;
  a.segs = p.d_segs;
  a.work = p.d_work;
  a.descale = reinterpret_cast<const float*>(ws + p.ws.descale);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ost = ost;
  a.osh = osh;
  a.scale_log2 = p.scale * 1.4426950408889634f;
  a.H = p.heads;
  a.err = p.d_err;
  a.abort_word = p.d_err + 1;
  a.gen = next_launch_generation();
  a.spin_limit = p.spin_limit;
  attn_fp8_kernel<<<unsigned(p.work.size()), kThreads, kSmemBytes, stream>>>(tq, tk, tv, a);
  return cuda_status(cudaGetLastError());
}

}  // namespace falp
