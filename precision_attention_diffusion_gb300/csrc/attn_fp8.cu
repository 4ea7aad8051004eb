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
//   * warp 16 issues TMA loads: Q once, then 128-key K and V^T tiles into a 4-stage ring with
//     128-byte swizzle;
//   * warp 17 allocates tensor memory; warps 17 and 18 issue the tcgen05.mma kind::f8f6f4 of query
//     tiles 0 and 1 (two independent in-order streams) on 64-key sub-tiles u, one elect.sync per
//     group of MMAs and its commit:
//       S_t(u) = Q_t K(u)^T   (M=128, N=64;  A, B from shared memory)
//       O_t += P_t(u) V(u)    (M=128, N=128; A = P_t from tensor memory)
//   * tensor memory (all 512 columns): per query tile two 64-column S buffers and a 128-column O;
//     P_t(u) (64 E4M3 per row = 16 columns) is written over the S buffer it was computed from, and
//     S_t(u+2) is issued into that buffer right after PV_t(u), so S is always one sub-tile ahead
//     of the softmax;
//   * warps 0-7 / 8-15 run the online softmax of Q0 / Q1, two threads per query row: with the
//     16x32bx2 tensor-memory shapes, warp w of a tile covers the 16 rows (lanes) 32 (w & 3) +
//     16 (w >> 2) + [0, 16), thread t and t ^ 16 of the warp holding keys [0, 32) and [32, 64)
//     of the row's sub-tile (and channels [0, 64) and [64, 128) of its O); the load returns each
//     half's maximum and one shuffle combines the halves. Four softmax warps per SM
//     sub-partition hide each other's MUFU and tensor-memory latencies. The reference maximum m
//     is the first sub-tile's maximum and moves to a later sub-tile's maximum M only when
//     (M - m) c > 8 (reading r5 with tau = 8; the pages leave the rule open): alpha =
//     2^((m - M) c), O *= alpha (only when a row of the warp moved), P = E4M3(2^(S c - m c)) <=
//     256, l = l alpha + sum of the quantized P (reading r6; each thread sums its half, the
//     halves are added at the end), where S is the raw E4M3 dot product and c = dq dk
//     softmax_scale log2(e);
//   * steady-state waits first park the warp in hardware (try_wait with a suspend-time hint) so
//     that waiting warps take no issue slots from the warps they share a scheduler with; warp 19
//     has no role (the 20-warp block keeps the register budget at 96 per thread);
//   * epilogue: out = BF16_rn(O dv / l) for rows inside the segment only.
// Every barrier wait is bounded; on expiry the kernel records an error, drains its in-flight
// copies and MMAs, frees its tensor memory and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_lp_internal.h"
#include "sm103_ptx.cuh"

namespace falp {
namespace {

constexpr int kStages = 4;
constexpr int kThreads = 640;   // 20 warps: 16 softmax, TMA, 2 MMA, one idle (see the header)
constexpr int kTmaWarp = 16;
constexpr int kMmaWarp = 17;    // warps 17 and 18 issue the MMAs of query tiles 0 and 1
constexpr int kSub = 64;                            // keys per sub-tile
constexpr uint32_t kTileBytes = 128 * 128;          // one 128x128 E4M3 tile
constexpr uint32_t kIdescS = idesc_f8f6f4(128, kSub, 0, 0);   // E4M3 x E4M3 -> F32, N=64
constexpr uint32_t kIdescPV = idesc_f8f6f4(128, 128, 0, 0);   // N = 128 channels
constexpr uint32_t kProbeNs = 100000;         // one parked probe: at most ~100 us
constexpr int kSpinProbes = 64;                 // plain probes before parking
constexpr long long kDrainProbes = 20000;      // drains give up after ~2 s
constexpr uint32_t kHintNs = 20000;           // first probe of a steady-state wait: park up to 20 us
// Threshold (log2 units) by which a sub-tile's maximum must exceed the reference maximum before
// the reference moves (and O, l are rescaled). P = 2^(S c - m c) <= 2^kTau stays inside E4M3.
constexpr float kTau = 8.0f;
// tensor-memory columns of query tile t: S buffer b at 128t + 64b (P of that sub-tile is written
// over its first 16 columns once S has been read), O at 256 + 128t
__device__ __forceinline__ uint32_t col_s(int t, int b) { return 128u * uint32_t(t) + 64u * uint32_t(b); }
__device__ __forceinline__ uint32_t col_o(int t) { return 256u + 128u * uint32_t(t); }

struct Smem {
  uint8_t q[2][kTileBytes];
  uint8_t k[kStages][kTileBytes];
  uint8_t v[kStages][kTileBytes];
  uint64_t bar_q;
  uint64_t bar_ld[kStages];  // K and V^T tiles of the stage landed
  uint64_t bar_free[kStages];
  uint64_t bar_s[2][2];  // [t][u & 1]: S_t(u) written (MMA commit)
  uint64_t bar_p[2][2];  // [t][u & 1]: P_t(u) written, O rescaled (128 arrivals)
  uint64_t bar_o[2][2];  // [t][u & 1]: PV_t(u) done (MMA commit)
  uint64_t bar_drain[2];
  uint32_t tmem_base;
  int abort_flag;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

struct AttnArgs {
  const SegInfo* segs;
  const WorkItem* work;
  const float* descale;  // [3][R][H]: R = 1, or one row per segment (per-segment scales)
  int scale_rows;        // R
  __nv_bfloat16* out;
  int64_t ost, osh;
  float* lse;        // optional: FP32 row log-sum-exp at lse[h * lse_sh + token]
  int64_t lse_sh;
  float scale_log2;
  int H;
  int* err;          // sticky error word of the plan (read and cleared by the host)
  int* abort_word;   // launch generation that aborted, shared by every CTA of the launch
  int gen;           // this launch's generation
  long long spin_limit;
};

enum Role : int { kRoleProducer = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleEpilogue = 4 };

// Bounded wait on one mbarrier phase. The first kSpinProbes probes are plain try_waits (the
// hardware holds the thread briefly and wakes it as the phase completes: the lowest latency for
// the short waits of the steady state); later probes park the thread for up to kProbeNs each.
// Every probe counts toward a.spin_limit; reaching it expires the wait. A limit shorter than the
// spin phase (a test configuration) makes every probe a non-blocking poll, so that the limit
// counts polls exactly. Returns false when the CTA aborts (this wait expired, or another wait of
// this launch did). The first probe is inlined; the rest lives out of line to keep code small.
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, Smem& S,
                                             const AttnArgs& a, int role) {
  const bool exact = a.spin_limit < kSpinProbes;
  long long n = exact ? 0 : 1;  // the inlined fast path made one probe already
  for (;;) {
    if (n >= a.spin_limit) {
      *reinterpret_cast<volatile int*>(&S.abort_flag) = 1;
      atomicExch(a.abort_word, a.gen);
      atomicCAS(a.err, 0, 0x100 | role);
      return false;
    }
    const bool parked = n >= kSpinProbes;
    bool done;
    if (exact) done = mbar_test_wait(bar, parity);
    else if (parked) done = mbar_try_wait_sleep(bar, parity, kProbeNs);
    else done = mbar_try_wait(bar, parity);
    if (done) return true;
    ++n;
    if (parked) {
      if (*reinterpret_cast<volatile int*>(&S.abort_flag)) return false;
      if (*reinterpret_cast<volatile int*>(a.abort_word) == a.gen) {  // another CTA gave up
        *reinterpret_cast<volatile int*>(&S.abort_flag) = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, Smem& S,
                                           const AttnArgs& a, int role) {
  if (a.spin_limit >= kSpinProbes && mbar_try_wait(bar, parity)) return true;
  return wait_phase_slow(bar, parity, S, a, role);
}

// Warp-uniform wait of the steady state: one probe that parks the warp in hardware until the phase
// completes (or kHintNs passes), so that a waiting warp takes no issue slots from the warps it
// shares a scheduler with; then the bounded wait.
__device__ __forceinline__ bool wait_hinted(uint32_t bar, uint32_t parity, Smem& S,
                                            const AttnArgs& a, int role) {
  if (__all_sync(0xffffffffu, mbar_try_wait_sleep(bar, parity, kHintNs))) return true;
  return __all_sync(0xffffffffu, wait_phase(bar, parity, S, a, role)) != 0;
}

// Wait used while draining after an abort: ignores the abort flag, bounded separately.
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity) {
  for (long long n = 0; n < kDrainProbes; ++n)
    if (mbar_try_wait_sleep(bar, parity, kProbeNs)) return;
}

// TMA role, on a whole warp, converged (a lone active lane beside 31 lanes parked at a CTA
// barrier is scheduled poorly); one elected lane issues the copies.
__device__ __forceinline__ void producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                         const CUtensorMap* tm_v, Smem& S, const AttnArgs& a,
                                         const WorkItem& wi, const SegInfo& sg) {
  const int n_kv = sg.nblk;
  const int rq = sg.row0 + wi.qt0 * kTile;
  mbar_arrive_expect_tx_elect(smem_u32(&S.bar_q), uint32_t(wi.nq) * kTileBytes);
  tma_load_3d_elect(smem_u32(S.q[0]), tm_q, smem_u32(&S.bar_q), 0, rq, wi.head);
  if (wi.nq == 2)
    tma_load_3d_elect(smem_u32(S.q[1]), tm_q, smem_u32(&S.bar_q), 0, rq + kTile, wi.head);
  int issued = 0;
  // two stages per iteration (see the sub-tile loops)
#pragma unroll 2
  for (int j = 0; j < n_kv; ++j) {
    const int st = j % kStages;
    if (j >= kStages &&
        !wait_hinted(smem_u32(&S.bar_free[st]), ((j / kStages) - 1) & 1, S, a, kRoleProducer))
      break;
    const int row = sg.row0 + j * kTile;
    mbar_arrive_expect_tx_elect(smem_u32(&S.bar_ld[st]), 2 * kTileBytes);
    tma_load_3d_elect(smem_u32(S.k[st]), tm_k, smem_u32(&S.bar_ld[st]), 0, row, wi.head);
    tma_load_3d_elect(smem_u32(S.v[st]), tm_v, smem_u32(&S.bar_ld[st]), row, 0, wi.head);
    issued = j + 1;
  }
  // No copy may still be landing in shared memory when the CTA exits.
  drain_phase(smem_u32(&S.bar_q), 0);
  for (int j = max(0, issued - kStages); j < issued; ++j) {
    const int st = j % kStages;
    drain_phase(smem_u32(&S.bar_ld[st]), (j / kStages) & 1);
  }
}

// MMA role of query tile t, on a whole warp, converged; only the MMA and commit instructions are
// issued, by one elected lane (lane 0 every time: tcgen05.commit tracks that lane's MMAs). The two
// query tiles have independent in-order MMA streams. S is computed two sub-tiles ahead: S_t(u+2)
// goes to the buffer of S_t(u) right after PV_t(u), which read P_t(u) from that buffer (the
// tensor pipe executes one thread's MMAs in issue order).
__device__ __forceinline__ void mma_issuer(Smem& S, const AttnArgs& a, const WorkItem& wi,
                                           const SegInfo& sg, uint32_t tmem, int t) {
  const int n_sub = (sg.len + kSub - 1) / kSub;
  // Descriptors are built once; the start-address field holds (address >> 4), so moving an
  // operand by `off` bytes (a K step, a sub-tile, a stage) adds off >> 4 to the descriptor.
  const uint64_t dq = sdesc_kmajor_sw128(smem_u32(S.q[0]) + uint32_t(t) * kTileBytes);
  const uint64_t dk = sdesc_kmajor_sw128(smem_u32(S.k[0]));
  const uint64_t dvv = sdesc_kmajor_sw128(smem_u32(S.v[0]));
  const uint32_t d_o = tmem + col_o(t);
  // S_t(u) = Q_t K(u)^T: K rows [64h, 64h + 64) of the stage holding key tile u / 2
  auto issue_s = [&](int u) {
    const uint32_t j = uint32_t(u) >> 1, h = uint32_t(u) & 1;
    const uint64_t kb = dk + (((j % kStages) * kTileBytes + h * (kSub * 128)) >> 4);
    const uint32_t d = tmem + col_s(t, h);
    mma_f8f6f4_ss_k128_commit_elect(d, dq, kb, kIdescS, smem_u32(&S.bar_s[t][h]));
  };
  // O_t += P_t(u) V(u): keys [64h, 64h + 64) are bytes [64h, 64h + 64) of each V^T row; P from
  // the first 16 columns of S buffer h
  // the group also releases the stage after the tile's last use of it (h = 1, or the segment's
  // last sub-tile)
  auto issue_pv = [&](int u) {
    const uint32_t j = uint32_t(u) >> 1, h = uint32_t(u) & 1;
    const uint64_t vb = dvv + (((j % kStages) * kTileBytes + h * kSub) >> 4);
    const uint32_t pa = tmem + col_s(t, h);
    const uint32_t release = (h == 1 || u + 1 == n_sub) ? 1u : 0u;
    mma_f8f6f4_ts_k64_commit2_elect(d_o, pa, vb, kIdescPV, u > 0 ? 1u : 0u,
                                    smem_u32(&S.bar_o[t][h]), release,
                                    smem_u32(&S.bar_free[j % kStages]));
  };
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return wait_hinted(smem_u32(bar), parity, S, a, kRoleMma);
  };
  do {
    if (!wait(&S.bar_q, 0)) break;
    if (!wait(&S.bar_ld[0], 0)) break;
    tc_fence_after();
    issue_s(0);
    if (n_sub > 1) issue_s(1);  // sub-tile 1 lies in key tile 0 as well
    bool ok = true;
    // two sub-tiles per iteration: the buffer and barrier parities become constants of each copy
#pragma unroll 2
    for (int u = 0; u < n_sub && ok; ++u) {
      const int h = u & 1;
      // the stage's V^T landed with its K, waited for before S of its first sub-tile
      ok = wait(&S.bar_p[t][h], (u >> 1) & 1);
      if (!ok) break;
      tc_fence_after();
      issue_pv(u);
      const int u2 = u + 2;
      if (u2 < n_sub) {
        if ((u2 & 1) == 0) {  // sub-tile u+2 opens key tile j+1
          const int j2 = u2 >> 1;
          ok = wait(&S.bar_ld[j2 % kStages], (j2 / kStages) & 1);
          if (!ok) break;
          tc_fence_after();
        }
        issue_s(u2);
      }
    }
  } while (false);
  // Every MMA issued so far must finish before the tensor memory is released.
  mma_commit_elect(smem_u32(&S.bar_drain[t]));
  drain_phase(smem_u32(&S.bar_drain[t]), 0);
}

__device__ __forceinline__ void softmax_and_epilogue(Smem& S, const AttnArgs& a,
                                                     const WorkItem& wi, const SegInfo& sg,
                                                     uint32_t tmem, int t, int wq, int lane) {
  const int n_sub = (sg.len + kSub - 1) / kSub;
  const int h = wi.head;
  const int64_t d0 = (a.scale_rows > 1 ? wi.seg : 0) * int64_t(a.H) + h;  // this tile's scales
  const int64_t dstride = int64_t(a.scale_rows) * a.H;
  const float c = a.descale[d0] * a.descale[dstride + d0] * a.scale_log2;
  const float dv = a.descale[2 * dstride + d0];
  // warp wq (0..7) of the tile: lane quarter wq & 3, half wq >> 2; the row is shared by threads
  // lane and lane ^ 16, which hold keys [0, 32) and [32, 64) of every sub-tile
  const int rbase = 32 * (wq & 3) + 16 * (wq >> 2);
  const int kh = lane >> 4;
  const uint32_t lane_off = uint32_t(rbase) << 16;
  const uint32_t o_addr = tmem + col_o(t) + lane_off;
  const int last_valid = sg.len - (n_sub - 1) * kSub;  // keys of the last sub-tile, 1..64
  float m = -INFINITY, l = 0.f;                         // reference maximum, this half's sum
  bool ok = true;
  // two sub-tiles per iteration: the buffer and barrier parities become constants of each copy
#pragma unroll 2
  for (int u = 0; u < n_sub; ++u) {
    const int b = u & 1;
    const uint32_t s_addr = tmem + col_s(t, b) + lane_off;
    ok = wait_hinted(smem_u32(&S.bar_s[t][b]), (u >> 1) & 1, S, a, kRoleSoftmax);
    if (!ok) break;
    tc_fence_after();
    uint32_t r[32];
    const float mxh = tmem_ld32x2_max<32>(s_addr, r);
    tmem_wait_ld();
    float s[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(r[i]);
    float mx = mxh;
    if (u == n_sub - 1 && last_valid < kSub) {  // keys past the segment: mask, then reduce
      mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (32 * kh + i >= last_valid) s[i] = -INFINITY;
        mx = fmaxf(mx, s[i]);
      }
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const bool move = (m == -INFINITY) || ((mx - m) * c > kTau);
    const float m_new = move ? mx : m;
    const float alpha = move ? ex2_approx((m - m_new) * c) : 1.f;  // m = -inf gives 0
    const float nmc = -m_new * c;
    uint32_t pk[8];
    uint32_t hs[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // 4 keys
      float x0, x1, x2, x3;
      fma2(x0, x1, s[4 * i], s[4 * i + 1], c, nmc);
      fma2(x2, x3, s[4 * i + 2], s[4 * i + 3], c, nmc);
      const uint16_t c01 = cvt_e4m3x2(ex2_approx(x0), ex2_approx(x1));
      const uint16_t c23 = cvt_e4m3x2(ex2_approx(x2), ex2_approx(x3));
      pk[i] = uint32_t(c01) | (uint32_t(c23) << 16);
      // the quantized values, back in f16 (exact), summed pairwise (reading r6)
      hs[i] = hadd2_u32(cvt_e4m3x2_to_f16x2(c01), cvt_e4m3x2_to_f16x2(c23));
    }
    const uint32_t h8 = hadd2_u32(hadd2_u32(hadd2_u32(hs[0], hs[1]), hadd2_u32(hs[2], hs[3])),
                                  hadd2_u32(hadd2_u32(hs[4], hs[5]), hadd2_u32(hs[6], hs[7])));
    const float2 fs = __half22float2(*reinterpret_cast<const __half2*>(&h8));
    l = l * alpha + (fs.x + fs.y);
    tmem_st8x2<8>(s_addr, pk);  // P over the first 16 columns of the S buffer just read
    if (u > 0 && __any_sync(0xffffffffu, move)) {
      // rescale O between PV_t(u-1) and PV_t(u): this thread's 64 channels
      ok = __all_sync(0xffffffffu, wait_phase(smem_u32(&S.bar_o[t][b ^ 1]), ((u - 1) >> 1) & 1,
                                              S, a, kRoleSoftmax));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        uint32_t o[32];
        tmem_ld32x2<64>(o_addr + 32 * i, o);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st32x2<64>(o_addr + 32 * i, o);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(smem_u32(&S.bar_p[t][b]));
    m = m_new;
  }
  if (!ok) {
    tmem_wait_st();  // a P store or O rescale may still be in flight
    return;
  }
  // PV_t(n_sub - 1) done implies every earlier PV of this in-order stream is done
  ok = __all_sync(0xffffffffu, wait_phase(smem_u32(&S.bar_o[t][(n_sub - 1) & 1]),
                                          ((n_sub - 1) >> 1) & 1, S, a, kRoleEpilogue));
  if (!ok) return;
  tc_fence_after();
  l += __shfl_xor_sync(0xffffffffu, l, 16);
  const float f = dv / l;
  const int qrow = (wi.qt0 + t) * kTile + rbase + (lane & 15);
  const bool valid = qrow < sg.len;
  // LSE in the units of S = q.k scale: m c (log2 units) + log2(l), times ln 2
  if (a.lse && valid && kh == 0)
    a.lse[int64_t(h) * a.lse_sh + sg.tok0 + qrow] = (m * c + log2f(l)) * 0.6931471805599453f;
  // this thread's channels: [0, 64) (kh = 0) or [64, 128) (kh = 1)
  __nv_bfloat16* dst = a.out + int64_t(sg.tok0 + qrow) * a.ost + int64_t(h) * a.osh + 64 * kh;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t o[32];
    tmem_ld32x2<64>(o_addr + 32 * i, o);
    tmem_wait_ld();
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const __nv_bfloat162 bb = __floats2bfloat162_rn(__uint_as_float(o[2 * e]) * f,
                                                      __uint_as_float(o[2 * e + 1]) * f);
      w[e] = *reinterpret_cast<const uint32_t*>(&bb);
    }
    if (valid) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * i);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        d4[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
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
      mbar_init(smem_u32(&S.bar_ld[i]), 1);
      mbar_init(smem_u32(&S.bar_free[i]), wi.nq);  // one commit per query tile
    }
    for (int t = 0; t < 2; ++t) {
      for (int x = 0; x < 2; ++x) {
        mbar_init(smem_u32(&S.bar_s[t][x]), 1);
        mbar_init(smem_u32(&S.bar_p[t][x]), 256);
        mbar_init(smem_u32(&S.bar_o[t][x]), 1);
      }
      mbar_init(smem_u32(&S.bar_drain[t]), 1);
    }
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
    producer(&tm_q, &tm_k, &tm_v, S, a, wi, sg);
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    const int t = warp - kMmaWarp;
    if (t < wi.nq) mma_issuer(S, a, wi, sg, tmem, t);
  } else if (warp < 16) {
    const int t = warp >> 3;
    if (t < wi.nq) softmax_and_epilogue(S, a, wi, sg, tmem, t, warp & 7, lane);
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
                         float* lse, int64_t lse_sh, cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};
  if (set_smem_limit_once(reinterpret_cast<const void*>(attn_fp8_kernel), int(kSmemBytes), p.device,
                          smem_set) != FA_LP_OK)
    return FA_LP_ERR_CUDA;
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
  a.scale_rows = fp8_scale_rows(p);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ost = ost;
  a.osh = osh;
  a.lse = lse;
  a.lse_sh = lse_sh;
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
