// attn_fp8_sparse.cu -- block-sparse FP8 E4M3 attention forward on 5th-generation tensor cores.
//
// Passage: SGLang PR #40116 "Add SM120 Sage compute for SubBlock sparse attention", Modifications
// (64-row query blocks x 64-key blocks, a key block being n_k = 4 pooling cells of 16 keys;
// partial blocks; variable per-row block counts, mixed sparse and dense query rows) and Accuracy
// Tests (ragged lengths, variable block counts, empty rows). The per-block arithmetic is the
// dense FP8 path's (SGLang PR #40175, Modifications, kernel.py): E4M3 QK and PV with FP32
// accumulation, online softmax, P packed to E4M3. The pages' SM120 mode computes QK in INT8;
// sm_103a has no INT8 tcgen05.mma (ptxas rejects kind::i8 for this target), so both products
// stay in E4M3 here.
//
// Semantics (reading r16): a query row in the g-th 64-row block of its segment attends to the
// keys of the 64-key blocks listed for (head, g) -- block kb covers keys [64 kb, 64 kb + 64) of
// the segment, the last one partial -- and a row whose list is empty is written as 0.
//
// GB300 design:
//   * the tensor cores take 128-row query tiles, i.e. two 64-row query blocks; a prologue kernel
//     merges the two ascending lists of every tile into one ascending list of key blocks, each
//     entry tagged with the halves (rows 0-63, 64-127) that listed it, and stores it in place of
//     the two lists (the merged list is never longer than the two together);
//   * a second prologue kernel orders the query tiles of every group (one segment, up to 8 heads,
//     the CTAs that run together and share K/V in L2) by merged-list length, longest first, and
//     the attention CTAs take them two at a time: the two tiles of a CTA have about the same
//     length (a CTA lasts as long as its longer tile) and long tiles start first;
//   * one CTA = two query tiles, each with its own pipeline over its own merged list: TMA warp
//     16 / 19 streams the tile's K blocks (64 keys x 128 channels, 128-byte
//     swizzle) and V^T blocks (128 channels x 64 keys, 64-byte swizzle) through a 5-stage ring;
//     MMA warp 17 / 18 issues S = Q K^T (N = 64) and O += P V (K = 64), S one block ahead in the
//     second tensor-memory buffer; softmax warps 0-7 / 8-15 as in the dense kernel (two threads
//     per row, lazy reference maximum with tau = 8, l from the quantized P);
//   * a softmax warp owns 16 rows of one half: on a block only the other half listed, it stores
//     P = 0 over its rows (the shared PV then adds exactly 0 to them) and leaves m and l alone;
//   * a row whose half listed nothing ends with l = 0 and is written as 0 (LSE -inf); a tile
//     whose merged list is empty issues no copy and no MMA.
// Every barrier wait is bounded; on expiry the kernel records an error, drains its in-flight
// copies and MMAs, frees its tensor memory and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_sync.cuh"
#include "fa_lp_internal.h"

namespace falp {
namespace {

constexpr int kSt = 5;                        // ring stages per query tile
constexpr int kThreads = 640;                 // 16 softmax warps, 2 TMA, 2 MMA
constexpr int kTmaWarp0 = 16, kTmaWarp1 = 19; // producers of query tiles 0 and 1
constexpr int kMmaWarp = 17;                  // warps 17 and 18 issue the MMAs of tiles 0 and 1
constexpr int kBlk = 64;                      // rows of a query block, keys of a key block
constexpr uint32_t kQBytes = 128 * 128;       // one 128-row query tile (E4M3)
constexpr uint32_t kKBytes = kBlk * 128;      // K block: 64 keys x 128 channels
constexpr uint32_t kVBytes = 128 * kBlk;      // V^T block: 128 channels x 64 keys
constexpr uint32_t kKbMask = 0x3FFFFFFFu;     // merged entry: key block | half 0 << 30 | half 1 << 31
constexpr uint32_t kIdescS = idesc_f8f6f4(128, kBlk, 0, 0);
constexpr uint32_t kIdescPV = idesc_f8f6f4(128, 128, 0, 0);
constexpr uint32_t kHintNs = 20000;
constexpr float kTau = 8.0f;                  // reference-maximum threshold, log2 units (r5)
constexpr int kErrBadList = 0x200;            // device status: a block list broke its contract

__device__ __forceinline__ uint32_t col_s(int t, int b) { return 128u * uint32_t(t) + 64u * uint32_t(b); }
__device__ __forceinline__ uint32_t col_o(int t) { return 256u + 128u * uint32_t(t); }

struct Smem {
  uint8_t q[2][kQBytes];
  uint8_t k[2][kSt][kKBytes];
  uint8_t v[2][kSt][kVBytes];
  uint64_t bar_q[2];
  uint64_t bar_ld[2][kSt];  // K block and V^T block of the stage landed
  uint64_t bar_free[2][kSt];
  uint64_t bar_s[2][2];  // [t][u & 1]: S_t(u) written
  uint64_t bar_p[2][2];  // [t][u & 1]: P_t(u) written, O rescaled (256 arrivals)
  uint64_t bar_o[2][2];  // [t][u & 1]: PV_t(u) done
  uint64_t bar_drain[2];
  uint32_t tmem_base;
  int abort_flag;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

struct SpArgs {
  const SegInfo* segs;
  const float* descale;    // [3][R][H]: R = 1, or one row per segment (per-segment scales)
  int scale_rows;          // R
  const uint32_t* uni;     // merged lists
  const int64_t* tbase;    // [H][nblocks] first entry of each tile's merged list
  const int32_t* tcnt;     // [H][nblocks] entries
  const int32_t* order;    // tile ids (h nblocks + block) by group, longest list first
  const SparseCta* ctas;   // slots of each CTA
  const BlockInfo* blocks;
  int nblocks;
  __nv_bfloat16* out;
  int64_t ost, osh;
  float* lse;
  int64_t lse_sh;
  float scale_log2;
  int H;
  WaitCtx w;
};

enum Role : int { kRoleProducer = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleEpilogue = 4 };

__device__ __forceinline__ bool wait_hinted(uint32_t bar, uint32_t parity, Smem& S,
                                            const SpArgs& a, int role) {
  if (__all_sync(0xffffffffu, mbar_try_wait_sleep(bar, parity, kHintNs))) return true;
  return __all_sync(0xffffffffu, wait_phase(bar, parity, &S.abort_flag, a.w, role)) != 0;
}

// ---------------------------------------------------------------------------------------------
// Prologue: merge the lists of the two 64-row query blocks of every 128-row tile.
// One CTA per (tile, head). Each list is checked (offsets inside [0, num_indices], indices inside
// the segment's key blocks and strictly ascending); an offending entry is dropped and the plan's
// device status records kErrBadList. Bitmaps of the two lists in shared memory, then one warp
// writes the set bits in ascending order.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(128) sparse_merge_kernel(
    const int32_t* __restrict__ off, const int32_t* __restrict__ idx, int64_t n_idx,
    const BlockInfo* __restrict__ blocks, const SegInfo* __restrict__ segs,
    const int32_t* __restrict__ qb0, int64_t G, int nblocks, uint32_t* __restrict__ uni,
    int64_t* __restrict__ tbase, int32_t* __restrict__ tcnt, int* __restrict__ err) {
  extern __shared__ uint32_t bm[];  // [2][nw]
  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const BlockInfo bi = blocks[b];
  const SegInfo sg = segs[bi.seg];
  const int nkb = (sg.len + kBlk - 1) / kBlk;
  const int nw = (nkb + 31) >> 5;
  const int64_t g0 = int64_t(qb0[bi.seg]) + 2 * int64_t(bi.blk);
  const int nlist = (int64_t(bi.blk) * 128 + kBlk < sg.len) ? 2 : 1;
  for (int i = tid; i < 2 * nw; i += 128) bm[i] = 0u;
  __syncthreads();
  const int64_t o0 = int64_t(h) * G + g0;
  bool bad = false;
  // list L of the tile: [lo_L, hi_L) of the indices (empty when its offsets are invalid)
  auto range = [&](int L, int64_t& lo, int64_t& hi) {
    lo = hi = 0;
    if (L >= nlist) return;
    const int64_t a0 = off[o0 + L], a1 = off[o0 + L + 1];
    if (a0 < 0 || a1 < a0 || a1 > n_idx) {
      bad = true;
      return;
    }
    lo = a0;
    hi = a1;
  };
  int64_t lo0, hi0, lo1, hi1;
  range(0, lo0, hi0);
  range(1, lo1, hi1);
  auto mark = [&](int L, int64_t lo, int64_t hi) {
    for (int64_t i = lo + tid; i < hi; i += 128) {
      const int kb = idx[i];
      const int prev = i > lo ? idx[i - 1] : -1;
      if (kb < 0 || kb >= nkb || kb <= prev) {
        bad = true;
        continue;
      }
      atomicOr(&bm[L * nw + (kb >> 5)], 1u << (kb & 31));
    }
  };
  mark(0, lo0, hi0);
  mark(1, lo1, hi1);
  if (bad) atomicCAS(err, 0, kErrBadList);
  __syncthreads();
  if (tid >= 32) return;
  // the merged list goes where the two lists were: [off[h G + g0], off[h G + g0 + nlist])
  const int64_t base = (hi0 > lo0 || nlist == 1) ? lo0 : lo1;
  const bool contiguous = nlist == 1 || hi0 == lo1 || hi0 == lo0 || hi1 == lo1;
  int64_t pos = 0;
  for (int w0 = 0; w0 < nw; w0 += 32) {
    const int w = w0 + tid;
    const uint32_t ma = w < nw ? bm[w] : 0u, mb = w < nw ? bm[nw + w] : 0u;
    uint32_t u = ma | mb;
    const int c = __popc(u);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (tid >= o) incl += y;
    }
    int64_t p = pos + incl - c;
    while (u) {
      const int bit = __ffs(u) - 1;
      u &= u - 1;
      const uint32_t kb = uint32_t(32 * w + bit);
      uni[base + p++] = kb | (((ma >> bit) & 1u) << 30) | (((mb >> bit) & 1u) << 31);
    }
    pos += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (tid == 0) {
    // a merged list may only use the room of the two lists it replaces
    const bool fits = contiguous && pos <= (hi0 - lo0) + (hi1 - lo1);
    tbase[int64_t(h) * nblocks + b] = base;
    tcnt[int64_t(h) * nblocks + b] = fits ? int32_t(pos) : 0;
    if (!fits) atomicCAS(err, 0, kErrBadList);
  }
}

// Prologue 2: within each group (one segment, heads [h0, h0 + nh)), the tile ids in descending
// order of merged-list length (a counting sort on min(length, 4095); ties in any order).
constexpr int kOrderBins = 4096;
__global__ void __launch_bounds__(256) sparse_order_kernel(const SparseGroup* __restrict__ groups,
                                                           const SegInfo* __restrict__ segs,
                                                           const int32_t* __restrict__ tcnt,
                                                           int nblocks, int32_t* __restrict__ order) {
  __shared__ int bins[kOrderBins];
  const SparseGroup gr = groups[blockIdx.x];
  const SegInfo sg = segs[gr.seg];
  const int nb = sg.nblk, nt = gr.nh * nb, b0 = sg.row0 / kTile;
  for (int i = threadIdx.x; i < kOrderBins; i += 256) bins[i] = 0;
  __syncthreads();
  auto tile = [&](int j) { return (gr.h0 + j / nb) * nblocks + b0 + j % nb; };
  auto key = [&](int id) { return kOrderBins - 1 - min(tcnt[id], kOrderBins - 1); };
  for (int j = threadIdx.x; j < nt; j += 256) atomicAdd(&bins[key(tile(j))], 1);
  __syncthreads();
  // exclusive scan of the bins: 256 threads x 16 consecutive bins
  constexpr int kPer = kOrderBins / 256;
  __shared__ int part[256];
  int loc[kPer], sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    loc[i] = sum;
    sum += bins[threadIdx.x * kPer + i];
  }
  part[threadIdx.x] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int i = 0; i < 256; ++i) {
      const int x = part[i];
      part[i] = acc;
      acc += x;
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kPer; ++i) bins[threadIdx.x * kPer + i] = part[threadIdx.x] + loc[i];
  __syncthreads();
  for (int j = threadIdx.x; j < nt; j += 256) {
    const int id = tile(j);
    order[gr.slot0 + atomicAdd(&bins[key(id)], 1)] = id;
  }
}

// ---------------------------------------------------------------------------------------------
// Attention roles. A query tile of a CTA: its segment, head and tile index in the segment.
struct TileRef {
  SegInfo sg;
  int seg, head, qt;
};

// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                         const CUtensorMap* tm_v, Smem& S, const SpArgs& a,
                                         const TileRef& tr, int t, const uint32_t* ent, int n) {
  if (n == 0) return;
  const SegInfo& sg = tr.sg;
  const int rq = sg.row0 + tr.qt * kTile;
  mbar_arrive_expect_tx_elect(smem_u32(&S.bar_q[t]), kQBytes);
  tma_load_3d_elect(smem_u32(S.q[t]), tm_q, smem_u32(&S.bar_q[t]), 0, rq, tr.head);
  int issued = 0;
  for (int j = 0; j < n; ++j) {
    const int st = j % kSt;
    if (j >= kSt &&
        !wait_hinted(smem_u32(&S.bar_free[t][st]), ((j / kSt) - 1) & 1, S, a, kRoleProducer))
      break;
    const int row = sg.row0 + kBlk * int(__ldg(ent + j) & kKbMask);
    mbar_arrive_expect_tx_elect(smem_u32(&S.bar_ld[t][st]), kKBytes + kVBytes);
    tma_load_3d_elect(smem_u32(S.k[t][st]), tm_k, smem_u32(&S.bar_ld[t][st]), 0, row, tr.head);
    tma_load_3d_elect(smem_u32(S.v[t][st]), tm_v, smem_u32(&S.bar_ld[t][st]), row, 0, tr.head);
    issued = j + 1;
  }
  drain_phase(smem_u32(&S.bar_q[t]), 0);
  for (int j = max(0, issued - kSt); j < issued; ++j) {
    const int st = j % kSt;
    drain_phase(smem_u32(&S.bar_ld[t][st]), (j / kSt) & 1);
  }
}

__device__ __forceinline__ void mma_issuer(Smem& S, const SpArgs& a, uint32_t tmem, int t, int n) {
  if (n == 0) return;
  const uint64_t dq = sdesc_kmajor_sw128(smem_u32(S.q[t]));
  const uint64_t dk = sdesc_kmajor_sw128(smem_u32(S.k[t][0]));
  const uint64_t dv = sdesc_kmajor_sw64(smem_u32(S.v[t][0]));
  const uint32_t d_o = tmem + col_o(t);
  auto issue_s = [&](int u) {
    const uint64_t kb = dk + ((uint32_t(u % kSt) * kKBytes) >> 4);
    mma_f8f6f4_ss_k128_commit_elect(tmem + col_s(t, u & 1), dq, kb, kIdescS,
                                    smem_u32(&S.bar_s[t][u & 1]));
  };
  // the group also releases the block's stage (its K was read by S(u), issued earlier)
  auto issue_pv = [&](int u) {
    const uint64_t vb = dv + ((uint32_t(u % kSt) * kVBytes) >> 4);
    mma_f8f6f4_ts_k64_commit2_elect(d_o, tmem + col_s(t, u & 1), vb, kIdescPV, u > 0 ? 1u : 0u,
                                    smem_u32(&S.bar_o[t][u & 1]), 1u,
                                    smem_u32(&S.bar_free[t][u % kSt]));
  };
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return wait_hinted(smem_u32(bar), parity, S, a, kRoleMma);
  };
  do {
    if (!wait(&S.bar_q[t], 0)) break;
    if (!wait(&S.bar_ld[t][0], 0)) break;
    tc_fence_after();
    issue_s(0);
    if (n > 1) {
      if (!wait(&S.bar_ld[t][1 % kSt], 0)) break;
      tc_fence_after();
      issue_s(1);
    }
    bool ok = true;
    // two sub-tiles per iteration: the buffer and barrier parities become constants of each copy
#pragma unroll 2
    for (int u = 0; u < n && ok; ++u) {
      // V(u) landed with K(u), waited for before S(u)
      ok = wait(&S.bar_p[t][u & 1], (u >> 1) & 1);
      if (!ok) break;
      tc_fence_after();
      issue_pv(u);
      const int u2 = u + 2;
      if (u2 < n) {
        ok = wait(&S.bar_ld[t][u2 % kSt], (u2 / kSt) & 1);
        if (!ok) break;
        tc_fence_after();
        issue_s(u2);
      }
    }
  } while (false);
  mma_commit_elect(smem_u32(&S.bar_drain[t]));
  drain_phase(smem_u32(&S.bar_drain[t]), 0);
}

__device__ __forceinline__ void softmax_and_epilogue(Smem& S, const SpArgs& a, const TileRef& tr,
                                                     uint32_t tmem, int t, int wq, int lane,
                                                     const uint32_t* ent, int n) {
  const SegInfo& sg = tr.sg;
  const int h = tr.head;
  const int64_t d0 = (a.scale_rows > 1 ? tr.seg : 0) * int64_t(a.H) + h;  // this tile's scales
  const int64_t dstride = int64_t(a.scale_rows) * a.H;
  const float c = a.descale[d0] * a.descale[dstride + d0] * a.scale_log2;
  const float dv = a.descale[2 * dstride + d0];
  const int rbase = 32 * (wq & 3) + 16 * (wq >> 2);  // rows of this warp: rbase + [0, 16)
  const int kh = lane >> 4;                           // keys [32 kh, 32 kh + 32) of a block
  const uint32_t half_bit = 1u << (30 + ((wq & 3) >> 1));
  const uint32_t lane_off = uint32_t(rbase) << 16;
  const uint32_t o_addr = tmem + col_o(t) + lane_off;
  const int kb_last = (sg.len + kBlk - 1) / kBlk - 1;
  const int last_valid = sg.len - kBlk * kb_last;  // keys of the segment's last block, 1..64
  float m = -INFINITY, l = 0.f;
  bool started = false, ok = true;
  uint32_t e_next = n > 0 ? __ldg(ent) : 0u;
  // two sub-tiles per iteration: the buffer and barrier parities become constants of each copy
#pragma unroll 2
  for (int u = 0; u < n; ++u) {
    const uint32_t e = e_next;
    if (u + 1 < n) e_next = __ldg(ent + u + 1);
    const int b = u & 1;
    const uint32_t s_addr = tmem + col_s(t, b) + lane_off;
    ok = wait_hinted(smem_u32(&S.bar_s[t][b]), (u >> 1) & 1, S, a, kRoleSoftmax);
    if (!ok) break;
    tc_fence_after();
    if (!(e & half_bit)) {  // the other half's block: P = 0 over these rows
      const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      tmem_st8x2<8>(s_addr, z);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&S.bar_p[t][b]));
      continue;
    }
    uint32_t r[32];
    const float mxh = tmem_ld32x2_max<32>(s_addr, r);
    tmem_wait_ld();
    float s[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(r[i]);
    float mx = mxh;
    if (int(e & kKbMask) == kb_last && last_valid < kBlk) {  // keys past the segment
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
    uint32_t pk[8], hs[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float x0, x1, x2, x3;
      fma2(x0, x1, s[4 * i], s[4 * i + 1], c, nmc);
      fma2(x2, x3, s[4 * i + 2], s[4 * i + 3], c, nmc);
      const uint16_t c01 = cvt_e4m3x2(ex2_approx(x0), ex2_approx(x1));
      const uint16_t c23 = cvt_e4m3x2(ex2_approx(x2), ex2_approx(x3));
      pk[i] = uint32_t(c01) | (uint32_t(c23) << 16);
      hs[i] = hadd2_u32(cvt_e4m3x2_to_f16x2(c01), cvt_e4m3x2_to_f16x2(c23));
    }
    const uint32_t h8 = hadd2_u32(hadd2_u32(hadd2_u32(hs[0], hs[1]), hadd2_u32(hs[2], hs[3])),
                                  hadd2_u32(hadd2_u32(hs[4], hs[5]), hadd2_u32(hs[6], hs[7])));
    const float2 fs = __half22float2(*reinterpret_cast<const __half2*>(&h8));
    l = l * alpha + (fs.x + fs.y);
    tmem_st8x2<8>(s_addr, pk);
    // Before this half's first block its O rows hold exactly 0 (every earlier P of theirs was
    // 0), so only a move after that needs the rescale.
    if (started && __any_sync(0xffffffffu, move)) {
      ok = __all_sync(0xffffffffu, wait_phase(smem_u32(&S.bar_o[t][b ^ 1]), ((u - 1) >> 1) & 1,
                                              &S.abort_flag, a.w, kRoleSoftmax));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        uint32_t o[32];
        tmem_ld32x2<64>(o_addr + 32 * i, o);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
        tmem_st32x2<64>(o_addr + 32 * i, o);
      }
    }
    started = true;
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(smem_u32(&S.bar_p[t][b]));
    m = m_new;
  }
  if (!ok) {
    tmem_wait_st();
    return;
  }
  if (n > 0) {
    ok = __all_sync(0xffffffffu, wait_phase(smem_u32(&S.bar_o[t][(n - 1) & 1]),
                                            ((n - 1) >> 1) & 1, &S.abort_flag, a.w,
                                            kRoleEpilogue));
    if (!ok) return;
    tc_fence_after();
  }
  l += __shfl_xor_sync(0xffffffffu, l, 16);
  const bool any = l > 0.f;  // false: this half listed no block
  const float f = any ? dv / l : 0.f;
  const int qrow = tr.qt * kTile + rbase + (lane & 15);
  const bool valid = qrow < sg.len;
  if (a.lse && valid && kh == 0)
    a.lse[int64_t(h) * a.lse_sh + sg.tok0 + qrow] =
        any ? (m * c + log2f(l)) * 0.6931471805599453f : -INFINITY;
  __nv_bfloat16* dst = a.out + int64_t(sg.tok0 + qrow) * a.ost + int64_t(h) * a.osh + 64 * kh;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t o[32];
    if (n > 0) {  // a warp-uniform condition: the load is collective
      tmem_ld32x2<64>(o_addr + 32 * i, o);
      tmem_wait_ld();
    }
    uint32_t w[16];
#pragma unroll
    for (int x = 0; x < 16; ++x) {
      if (any) {
        const __nv_bfloat162 bb = __floats2bfloat162_rn(__uint_as_float(o[2 * x]) * f,
                                                        __uint_as_float(o[2 * x + 1]) * f);
        w[x] = *reinterpret_cast<const uint32_t*>(&bb);
      } else {
        w[x] = 0u;
      }
    }
    if (valid) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * i);
#pragma unroll
      for (int x = 0; x < 4; ++x)
        d4[x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_fp8_sparse_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ SpArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const SparseCta cta = a.ctas[blockIdx.x];
  // the query tile this warp serves (TMA 16 / MMA 17 / softmax 0-7: tile 0; 19 / 18 / 8-15:
  // tile 1), its merged list and length (0 for a second tile the CTA does not hold); one tile
  // per warp, so nothing here is indexed by a runtime tile number (no local memory)
  const int t = warp < 16 ? (warp >> 3) : ((warp == kTmaWarp0 || warp == kMmaWarp) ? 0 : 1);
  const int id = t < cta.count ? a.order[cta.slot + t] : a.order[cta.slot];
  const int hh = id / a.nblocks;
  const BlockInfo bi = a.blocks[id - hh * a.nblocks];
  TileRef tr;
  tr.sg = a.segs[bi.seg];
  tr.seg = bi.seg;
  tr.head = hh;
  tr.qt = bi.blk;
  const uint32_t* ent = a.uni + a.tbase[id];
  const int n = t < cta.count ? a.tcnt[id] : 0;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&S.bar_q[t]), 1);
      for (int i = 0; i < kSt; ++i) {
        mbar_init(smem_u32(&S.bar_ld[t][i]), 1);
        mbar_init(smem_u32(&S.bar_free[t][i]), 1);
      }
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
  if (warp == kTmaWarp0 && lane == 0) {
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

  if (warp == kTmaWarp0 || warp == kTmaWarp1) {
    producer(&tm_q, &tm_k, &tm_v, S, a, tr, t, ent, n);
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    mma_issuer(S, a, tmem, t, n);
  } else if (warp < 16) {
    if (t < cta.count) softmax_and_epilogue(S, a, tr, tmem, t, warp & 7, lane, ent, n);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int launch_fp8_sparse(const fa_lp_plan& p, uint8_t* ws, const int32_t* off, const int32_t* idx,
                      int64_t n_idx, void* out, int64_t ost, int64_t osh, float* lse,
                      int64_t lse_sh, cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};
  if (set_smem_limit_once(reinterpret_cast<const void*>(attn_fp8_sparse_kernel), int(kSmemBytes), p.device,
                          smem_set) != FA_LP_OK)
    return FA_LP_ERR_CUDA;
  const int nblocks = int(p.blocks.size());
  uint32_t* uni = static_cast<uint32_t*>(p.sp_buf);
  int64_t* tbase = reinterpret_cast<int64_t*>(static_cast<uint8_t*>(p.sp_buf) + p.sp_tables);
  int32_t* tcnt = reinterpret_cast<int32_t*>(tbase + int64_t(p.heads) * nblocks);
  int32_t* order = tcnt + int64_t(p.heads) * nblocks;
  const size_t merge_smem = size_t(2) * p.sp_nw_max * sizeof(uint32_t);
  dim3 gm(unsigned(nblocks), unsigned(p.heads));
  sparse_merge_kernel<<<gm, 128, merge_smem, stream>>>(off, idx, n_idx, p.d_blocks, p.d_segs,
                                                       p.d_sp_qb0, p.sp_G, nblocks, uni, tbase,
                                                       tcnt, p.d_err);
  if (cudaGetLastError() != cudaSuccess) return FA_LP_ERR_CUDA;
  sparse_order_kernel<<<unsigned(p.sp_groups.size()), 256, 0, stream>>>(p.d_sp_groups, p.d_segs,
                                                                        tcnt, nblocks, order);
  if (cudaGetLastError() != cudaSuccess) return FA_LP_ERR_CUDA;

  const uint64_t H = uint64_t(p.heads), Tp = uint64_t(p.tpad);
  CUtensorMap tq, tk, tv;
  int st = encode_tmap_3d_u8(&tq, ws + p.ws.q_codes, 128, Tp, H, 128, Tp * 128, 128, 128,
                             CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == FA_LP_OK)
    st = encode_tmap_3d_u8(&tk, ws + p.ws.k_codes, 128, Tp, H, 128, Tp * 128, 128, kBlk,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == FA_LP_OK)
    st = encode_tmap_3d_u8(&tv, ws + p.ws.v_codes, Tp, 128, H, Tp, Tp * 128, kBlk, 128,
                           CU_TENSOR_MAP_SWIZZLE_64B);
  if (st != FA_LP_OK) return st;
  SpArgs a;
  a.segs = p.d_segs;
  a.order = order;
  a.ctas = p.d_sp_ctas;
  a.blocks = p.d_blocks;
  a.descale = reinterpret_cast<const float*>(ws + p.ws.descale);
  a.scale_rows = fp8_scale_rows(p);
  a.uni = uni;
  a.tbase = tbase;
  a.tcnt = tcnt;
  a.nblocks = nblocks;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ost = ost;
  a.osh = osh;
  a.lse = lse;
  a.lse_sh = lse_sh;
  a.scale_log2 = p.scale * 1.4426950408889634f;
  a.H = p.heads;
  a.w.err = p.d_err;
  a.w.abort_word = p.d_err + 1;
  a.w.gen = next_launch_generation();
  a.w.spin_limit = p.spin_limit;
  attn_fp8_sparse_kernel<<<unsigned(p.sp_ctas.size()), kThreads, kSmemBytes, stream>>>(tq, tk, tv,
                                                                                      a);
  return cuda_status(cudaGetLastError());
}

}  // namespace falp
