// attn_nvfp4.cu -- NVFP4 packed-varlen attention forward on 5th-generation tensor cores with
// block-scaled FP4 operands (tcgen05.mma kind::mxf4nvf4: E2M1 values, one UE4M3 scale per 16
// elements along the contraction).
//
// Passage: FlashInfer docs, flashinfer.diffusion_ops.minimax_h3_sm120_varlen_attention_nvfp4,
// description: SageAttention3-style FP4 attention -- K centred by its segment's per-channel mean
// (which leaves softmax unchanged), Q centred by its 128-row block mean with qm K^T added back,
// E2M1 codes with UE4M3 scales per 16 elements, V transposed with per-16-key scales, and a
// two-level P: the row maximum is brought to 448 * 6 = 2688 and every 16 keys get their own scale.
//
// What one CTA computes (readings r5 with tau = 0, r9, r11, r12): for the two 128-row query tiles
// Q0, Q1 of one (segment, head), over 64-key sub-tiles u from the segment start,
//   s''(i, j)  = (deq(Qc_i) . deq(Kc_j) + Tq_t(j)) c,  Tq_t(j) = qm_t . deq(Kc_j) (the table
//                qmk_nvfp4.cu writes, during quantization or right before the launch of a
//                group of heads, added to S by a TF32 MMA),
//                with c = softmax_scale log2(e)            (log2 units)
//   m_i        = running row maximum of s'' (exact: it moves whenever a sub-tile exceeds it)
//   P'(i, j)   = 2^(s'' - m_i + log2 2688)                  (= 2688 exp(S' - m) of the pages)
//   per 16 keys: sf = UE4M3(max P' / 6), code = E2M1(P' / deq(sf)), both evaluated in the
//                exponent: max P' / 6 = 2^(max s'' - m + log2 448), P' / deq(sf) =
//                2^(s'' - m + log2 2688 - log2 deq(sf)) (one exp2 per key, no division)
//   l_i        = l_i 2^(m_old - m_new) + sum deq(P),   O_i likewise with deq(P) deq(V); l is
//                accumulated by the PV MMA itself: every V^T stage carries 16 rows of E2M1 1.0
//                (scale 1.0) after its 128 channels, so O has 144 columns and column 128 is l
//   out        = BF16(O / l) for rows inside the segment.
//
// Roles (640 threads, 96 registers each):
//   warps 0-7 / 8-15  softmax of query tile 0 / 1, two threads per row through the 16x32bx2
//               tensor-memory shapes: warp w of a tile covers lanes 32 (w & 3) + 16 (w >> 2) +
//               [0, 16); threads t and t ^ 16 hold keys [0, 32) and [32, 64) of the row's
//               sub-tile (two 16-key scale groups each) and share the row maximum through one
//               shuffle; they also write the row's Q scale factors into tensor memory once;
//   warp 16     TMA: Q codes and (bulk copies) Q scale records once; per 128-key tile K codes, the
//               K scale record, the query tiles' 128-entry rows of the qm K^T table, V^T codes and
//               the V scale record, into a 4-stage ring;
//   warps 17/18 MMA issue for query tile 0/1 (two independent in-order streams; warp 17 allocates
//               tensor memory), each with the tcgen05.cp copies of the K and V scale factors its
//               MMAs read, from shared into its tile's tensor memory (ordered before its MMAs):
//                 S_t(u)  = deq(Qc_t) deq(Kc(u))^T   2 MMAs M=128 N=64  K=64, A, B in smem
//                 S_t(u) += 1 Tq_t(u)^T              1 kind::tf32 MMA M=128 N=64 K=8 (A =
//                                                    rows [1, 1, 1, 0...], B = the table
//                                                    entries as three TF32 pieces)
//                 O_t    += deq(P_t(u)) deq(V(u))    1 MMA  M=128 N=144 K=64, A = P in TMEM
//                                                    (N 128-143: the 1.0 rows, giving l)
//               S_t(u+1) is issued as soon as the softmax has read S_t(u), so the scores of the
//               next sub-tile are computed while the softmax works on the current ones;
//   warp 19     per sub-tile, from the stage's records: the K and V scale factors re-laid out as
//               32-row x 16-byte blocks for tcgen05.cp, and each query tile's fold tile (every
//               key's qm K^T table entry as three TF32 pieces, exact).
// Tensor memory (512 columns), per query tile t at 256 t: O [0, 144) (column 128: l), P codes
// [144, 152), P scales [152, 156) (A side: row r in lane r, column r / 32; [156, 160) takes the
// second thread's copy of the word), Q scales [160, 168), K scales [168, 184) (two buffers of two
// K steps), V scales [184, 189) (column 188: scale 1.0 of the 1.0 rows), S [192, 256).
// Every barrier wait is bounded; on expiry the kernel records an error, drains its in-flight
// copies and MMAs, frees its tensor memory and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_sync.cuh"
#include "fa_lp_internal.h"
#include "sm103_ptx.cuh"

namespace falp {
namespace {

constexpr int kStages = 4;
constexpr int kThreads = 640;
constexpr int kTmaWarp = 16;
constexpr int kMmaWarp = 17;     // warps 17 and 18 issue the MMAs of query tiles 0 and 1
constexpr int kAuxWarp = 19;
constexpr int kSub = 64;         // keys per sub-tile
constexpr int kAuxBufs = 4;      // re-laid-out scale blocks and fold tiles (two stages)
constexpr uint32_t kCodeTile = 128 * 64;  // 128 rows of 128 E2M1 codes
constexpr uint32_t kSfTile = 128 * 8;     // 128 rows of 8 UE4M3 scales
constexpr uint32_t kIdescS = idesc_mxf4nvf4(128, kSub);
constexpr uint32_t kVTile = 144 * 64;    // V^T stage: 128 channel rows + 16 rows of E2M1 1.0
constexpr uint32_t kIdescPV = idesc_mxf4nvf4(128, 144);  // channels + 16 row-sum columns
// kind::tf32: D f32, A and B TF32 (format 2), K-major, M=128, N=64
constexpr uint32_t kIdescFold = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t(kSub) >> 3) << 17) |
                                ((128u >> 4) << 24);
constexpr float kLog2_2688 = 11.392317422778761f;  // log2(448 * 6)
constexpr float kLog2_6 = 2.5849625007211562f;
constexpr uint32_t kHintNs = 20000;  // first probe of a steady-state wait: park up to 20 us

__device__ __forceinline__ uint32_t col_o(int t) { return 256u * uint32_t(t); }
__device__ __forceinline__ uint32_t col_p(int t) { return 256u * uint32_t(t) + 144u; }
__device__ __forceinline__ uint32_t col_psf(int t) { return 256u * uint32_t(t) + 152u; }
__device__ __forceinline__ uint32_t col_qsf(int t) { return 256u * uint32_t(t) + 160u; }
__device__ __forceinline__ uint32_t col_ksf(int t, int b) {
  return 256u * uint32_t(t) + 168u + 8u * uint32_t(b);
}
__device__ __forceinline__ uint32_t col_vsf(int t) { return 256u * uint32_t(t) + 184u; }
__device__ __forceinline__ uint32_t col_s(int t) { return 256u * uint32_t(t) + 192u; }

struct Smem {
  uint8_t q[2][kCodeTile];
  uint8_t k[kStages][kCodeTile];
  uint8_t v[kStages][kVTile];      // V^T: 128 channel rows of 128 keys, 16 rows of 1.0
  // qm K^T fold into S (one kind::tf32 MMA per sub-tile and query tile): A = 128 identical rows
  // [1, 1, 1, 0 | 0, 0, 0, 0] (one core matrix repeated, then a zero core matrix), B = per key the
  // table entry as three TF32 pieces (64 keys x 16 bytes, then 1 KB of zeros for K 4..7)
  uint8_t fb[kAuxBufs][2][2048];   // [u mod 4][t]
  uint8_t ksf_cp[kAuxBufs][2][512];  // [u mod 4][K step]: row i = scales of keys i, 32 + i, 0, 0
  uint8_t vsf_cp[kAuxBufs][512];     // [u mod 4]: row i = scales of channels i, 32+i, 64+i, 96+i
  uint8_t ones_cp[512];              // row i = scale 1.0 (x4) for i < 16, else 0
  uint8_t fa[256];
  uint8_t qsf[2][kSfTile];
  uint8_t ksf[kStages][kSfTile];   // [key][8]
  uint8_t vsf[kStages][kSfTile];   // [channel][8]
  float cq[kStages][2][kTile];     // [stage][t][key]: the qm K^T table row of query tile t
  uint64_t bar_q;
  uint64_t bar_qsf[2];             // [t]: Q scale factors in tensor memory (256 arrivals)
  uint64_t bar_ld[kStages];        // K, V codes, their scale records and the table rows landed
  uint64_t bar_free[kStages];      // MMA commits + the auxiliary warp
  uint64_t bar_aux[kAuxBufs];      // [u mod 4]: scale blocks and fold tiles of u written (32);
                                   // implies the stage of u has landed
  uint64_t bar_auxfree[kAuxBufs];  // [u mod 4]: the MMAs and copies of u that read them done
  uint64_t bar_s[2];               // [t]: S_t(u) written (MMA commit)
  uint64_t bar_sr[2];              // [t]: S_t(u) read by the softmax (256 arrivals)
  uint64_t bar_p[2][2];            // [t][u & 1]: P_t(u) written and O rescaled (256 arrivals)
  uint64_t bar_o[2][2];            // [t][u & 1]: PV_t(u) done (MMA commit)
  uint64_t bar_drain[2];
  uint32_t tmem_base;
  int abort_flag;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per block");

struct Nvfp4Args {
  const SegInfo* segs;
  const WorkItem* work;
  const uint8_t* q_sf;     // [H][Tp][8]
  const uint8_t* k_sf;     // [H][Tp][8]
  const uint8_t* v_sf;     // [H][Tp/128][128][8]
  const float* qmk;        // qm K^T table slot: segment s at c_off[s], [h - tbl_h0][nb_s][128 nb_s]
  const int64_t* c_off;
  int tbl_h0;              // first head of the slot
  const float* q_km;       // [H][Tp]: q . km per query row
  __nv_bfloat16* out;
  int64_t ost, osh;
  float* lse;              // optional: FP32 row log-sum-exp at lse[h * lse_sh + token]
  int64_t lse_sh;
  float scale;
  int64_t tpad;
  float scale_log2;
  WaitCtx w;
};

enum Role : int { kRoleProducer = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleEpilogue = 4,
                  kRoleScales = 5 };

// Warp-uniform bounded wait.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, Smem& S,
                                         const Nvfp4Args& a, int role) {
  return __all_sync(0xffffffffu, wait_phase(smem_u32(bar), parity, &S.abort_flag, a.w, role));
}

// Warp-uniform wait of the steady state: one probe that parks the warp in hardware until the phase
// completes (or kHintNs passes), so that a waiting warp takes no issue slots from the warps it
// shares a scheduler with; then the bounded wait.
__device__ __forceinline__ bool wait_hinted(uint64_t* bar, uint32_t parity, Smem& S,
                                            const Nvfp4Args& a, int role) {
  if (__all_sync(0xffffffffu, mbar_try_wait_sleep(smem_u32(bar), parity, kHintNs))) return true;
  return wait_all(bar, parity, S, a, role);
}

// One elect.sync for the whole S group of a query tile and sub-tile (a tcgen05 instruction group
// behind a single elect costs the issuing warp far less than one elect per instruction): the two K
// scale blocks into tensor memory, the two block-scaled K = 64 MMAs (the first overwriting S), the
// TF32 fold MMA adding the qm K^T term, and the commit of all of them to `bar`.
__device__ __forceinline__ void s_group_elect(uint32_t d, uint64_t qa, uint64_t kb, uint32_t sfa,
                                              uint32_t ks, uint64_t ksf0, uint64_t ksf1,
                                              uint64_t fa, uint64_t fb, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e, p0, p1;\n\t.reg .b64 qa1, kb1;\n\t.reg .b32 sfa1, ks1;\n\t"
      "setp.ne.b32 p0, 0, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
      "add.s64 qa1, %1, 2;\n\tadd.s64 kb1, %2, 2;\n\t"
      "add.s32 sfa1, %3, 4;\n\tadd.s32 ks1, %4, 4;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%4], %5;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [ks1], %6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %9, "
      "[%3], [%4], p0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], qa1, kb1, %9, "
      "[sfa1], [ks1], p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %7, %8, %10, p1;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%11];\n\t}"
      ::"r"(d), "l"(qa), "l"(kb), "r"(sfa), "r"(ks), "l"(ksf0), "l"(ksf1), "l"(fa), "l"(fb),
      "r"(kIdescS), "r"(kIdescFold), "r"(bar)
      : "memory");
}

// One elect.sync for the PV group: the V scale block into tensor memory, the block-scaled PV MMA
// (A = P from tensor memory; accumulating unless `first`), and the commits to the PV barrier and the
// auxiliary-buffer barrier, plus the stage barrier when `release`.
__device__ __forceinline__ void pv_group_elect(uint32_t d, uint32_t pa, uint64_t vb, uint32_t psf,
                                               uint32_t vs, uint64_t vsf, uint32_t accumulate,
                                               uint32_t bar_o, uint32_t bar_aux,
                                               uint32_t release, uint32_t bar_free) {
  asm volatile(
      "{\n\t.reg .pred e, p, r;\n\t"
      "setp.ne.b32 p, %6, 0;\n\tsetp.ne.b32 r, %9, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%4], %5;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], [%1], %2, %11, "
      "[%3], [%4], p;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%8];\n\t"
      "and.pred r, r, e;\n\t"
      "@r tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%10];\n\t}"
      ::"r"(d), "r"(pa), "l"(vb), "r"(psf), "r"(vs), "l"(vsf), "r"(accumulate), "r"(bar_o),
      "r"(bar_aux), "r"(release), "r"(bar_free), "r"(kIdescPV)
      : "memory");
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  const uint32_t h2 = cvt_e4m3x2_to_f16x2(uint16_t(code & 0xFF));
  return __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFF)));
}

// ---------------------------------------------------------------------------------------------
// TMA / bulk-copy producer (whole warp, converged; one elected lane issues).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                         const CUtensorMap* tm_v, Smem& S, const Nvfp4Args& a,
                                         const WorkItem& wi, const SegInfo& sg) {
  const int n_kv = sg.nblk;
  const int64_t Tp = a.tpad, h = wi.head;
  const int rq = sg.row0 + wi.qt0 * kTile;
  mbar_arrive_expect_tx_elect(smem_u32(&S.bar_q), uint32_t(wi.nq) * (kCodeTile + kSfTile));
  for (int t = 0; t < wi.nq; ++t) {
    const int row = rq + t * kTile;
    tma_load_3d_elect(smem_u32(S.q[t]), tm_q, smem_u32(&S.bar_q), 0, row, wi.head);
    bulk_load_elect(smem_u32(S.qsf[t]), a.q_sf + (h * Tp + row) * 8, kSfTile, smem_u32(&S.bar_q));
  }
  // rows of the qm K^T table of this (segment, head) for the CTA's query tiles
  const int64_t lp = int64_t(sg.nblk) * kTile;
  const float* tab = a.qmk + a.c_off[wi.seg] + ((h - a.tbl_h0) * sg.nblk + wi.qt0) * lp;
  int issued = 0;
  for (int j = 0; j < n_kv; ++j) {
    const int st = j % kStages;
    if (j >= kStages &&
        !wait_hinted(&S.bar_free[st], ((j / kStages) - 1) & 1, S, a, kRoleProducer))
      break;
    const int row = sg.row0 + j * kTile;
    const uint32_t bar = smem_u32(&S.bar_ld[st]);
    mbar_arrive_expect_tx_elect(bar, 2 * (kCodeTile + kSfTile) + uint32_t(wi.nq) * kTile * 4);
    tma_load_3d_elect(smem_u32(S.k[st]), tm_k, bar, 0, row, wi.head);
    bulk_load_elect(smem_u32(S.ksf[st]), a.k_sf + (h * Tp + row) * 8, kSfTile, bar);
    for (int t = 0; t < wi.nq; ++t)
      bulk_load_elect(smem_u32(S.cq[st][t]), tab + t * lp + int64_t(j) * kTile, kTile * 4, bar);
    tma_load_3d_elect(smem_u32(S.v[st]), tm_v, bar, row / 2, 0, wi.head);
    bulk_load_elect(smem_u32(S.vsf[st]), a.v_sf + (h * (Tp / kTile) + row / kTile) * kSfTile,
                    kSfTile, bar);
    issued = j + 1;
  }
  // No copy may still be landing in shared memory when the CTA exits.
  drain_phase(smem_u32(&S.bar_q), 0);
  for (int j = max(0, issued - kStages); j < issued; ++j)
    drain_phase(smem_u32(&S.bar_ld[j % kStages]), (j / kStages) & 1);
}

// ---------------------------------------------------------------------------------------------
// MMA issue for query tile t (whole warp, converged; one elected lane issues). Order per step u:
// S_t(u) as soon as the softmax has read S_t(u-1) (and the K tile and the auxiliary blocks of u are
// in shared memory), then PV_t(u-1) once P_t(u-1) is written: the tensor pipe computes the next
// scores while the softmax works on the current ones. The scale factors reach tensor memory by
// tcgen05.cp from this thread, ordered before its later MMAs.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void mma_issuer(Smem& S, const Nvfp4Args& a, const WorkItem& wi,
                                           const SegInfo& sg, uint32_t tmem, int t) {
  const int n_sub = (sg.len + kSub - 1) / kSub;
  // The start-address field holds (address >> 4): moving an operand by `off` bytes (a K step of
  // 64 E2M1 codes = 32 bytes, a sub-tile, a stage) adds off >> 4.
  const uint64_t dq = sdesc_kmajor_sw64(smem_u32(S.q[t]));
  const uint64_t dk = sdesc_kmajor_sw64(smem_u32(S.k[0]));
  const uint64_t dv = sdesc_kmajor_sw64(smem_u32(S.v[0]));
  const uint64_t dfa = sdesc_kmajor_noswz(smem_u32(S.fa), 128, 0);
  // 32 rows x 16 bytes, row i at byte 16 i (core matrices of 8 rows 128 bytes apart)
  const uint64_t dksf = sdesc_kmajor_noswz(smem_u32(S.ksf_cp[0][0]), 128, 128);
  const uint64_t dvsf = sdesc_kmajor_noswz(smem_u32(S.vsf_cp[0]), 128, 128);
  const uint64_t dones = sdesc_kmajor_noswz(smem_u32(S.ones_cp), 128, 128);
  const uint32_t d_s = tmem + col_s(t);
  auto issue_s = [&](int u) {
    const int x = u % kAuxBufs, h = u & 1, st = (u >> 1) % kStages;
    // K scales of u into buffer u & 1, last read by S_t(u-2): complete, since the softmax has
    // read S_t(u-1); S += 1 . (hi + mid + lo) of the table (TF32 pieces whose sum is the FP32
    // entry exactly): the qm K^T term, to FP32 accumulation
    const uint64_t kb = dk + (((st * kCodeTile) + h * (kSub * 64)) >> 4);
    s_group_elect(d_s, dq, kb, tmem + col_qsf(t), tmem + col_ksf(t, u & 1),
                  dksf + ((uint32_t(x) * 1024u) >> 4), dksf + ((uint32_t(x) * 1024u + 512u) >> 4),
                  dfa, sdesc_kmajor_noswz(smem_u32(S.fb[x][t]), 1024, 128),
                  smem_u32(&S.bar_s[t]));
  };
  // keys [64h, 64h + 64) of a 128-key tile are bytes [32h, 32h + 32) of each V^T row
  auto issue_pv = [&](int u) {
    const int x = u % kAuxBufs, h = u & 1, st = (u >> 1) % kStages;
    // V scales of u (the columns were last read by PV_t(u-1), complete before the softmax wrote
    // P_t(u)); the 1.0 rows' scale column was written once
    const uint64_t vb = dv + ((uint32_t(st) * kVTile) >> 4) + 2 * h;
    pv_group_elect(tmem + col_o(t), tmem + col_p(t), vb, tmem + col_psf(t), tmem + col_vsf(t),
                   dvsf + ((uint32_t(x) * 512u) >> 4), u > 0 ? 1u : 0u,
                   smem_u32(&S.bar_o[t][u & 1]), smem_u32(&S.bar_auxfree[x]),
                   (h == 1 || u + 1 == n_sub) ? 1u : 0u, smem_u32(&S.bar_free[st]));
  };
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return wait_hinted(bar, parity, S, a, kRoleMma);
  };
  // scale 1.0 of the 1.0 rows: columns [188, 192) of the tile are written by nothing else
  tmem_cp_32x128b_warpx4_elect(tmem + col_vsf(t) + 4, dones);
  do {
    if (!wait(&S.bar_q, 0)) break;
    if (!wait(&S.bar_qsf[t], 0)) break;
    bool ok = true;
    // four sub-tiles per iteration: the slot and barrier parities become constants of each copy
#pragma unroll 4
    for (int u = 0; u <= n_sub && ok; ++u) {
      if (u < n_sub) {
        // the auxiliary warp's blocks of u (written after the stage of u landed; the auxiliary
        // warp runs well ahead, so this wait is done before the one S_t(u) really waits for:
        // the softmax's read of S_t(u-1))
        if (!(ok = wait(&S.bar_aux[u % kAuxBufs], (u / kAuxBufs) & 1))) break;
        if (u > 0 && !(ok = wait(&S.bar_sr[t], (u - 1) & 1))) break;
        tc_fence_after();
        issue_s(u);
      }
      if (u > 0) {
        const int w = u - 1;
        if (!(ok = wait(&S.bar_p[t][w & 1], (w >> 1) & 1))) break;
        tc_fence_after();
        issue_pv(w);
      }
    }
  } while (false);
  // Every MMA and copy issued so far must finish before the tensor memory is released.
  mma_commit_elect(smem_u32(&S.bar_drain[t]));
  drain_phase(smem_u32(&S.bar_drain[t]), 0);
}

// ---------------------------------------------------------------------------------------------
// Auxiliary warp: once per 128-key stage, for both of its sub-tiles, the two K scale blocks and the
// V scale block in the row layout tcgen05.cp takes, and the fold tile of every query tile.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void aux_warp(Smem& S, const Nvfp4Args& a, const WorkItem& wi,
                                         const SegInfo& sg, int lane) {
  const int n_sub = (sg.len + kSub - 1) / kSub;
  const int n_kv = sg.nblk;
  const bool two = wi.nq == 2;
  for (int j = 0; j < n_kv; ++j) {
    const int st = j % kStages, u0 = 2 * j;
    if (!wait_hinted(&S.bar_ld[st], (j / kStages) & 1, S, a, kRoleScales)) break;
    // the blocks of u0 - 4 and u0 - 3 (same buffers) must have been consumed by every query
    // tile: the commit after PV(u0 - 3) covers every earlier MMA and copy of the issuing thread
    if (u0 >= kAuxBufs && !wait_hinted(&S.bar_auxfree[(u0 - 3) % kAuxBufs],
                                       ((u0 - 3) / kAuxBufs) & 1, S, a, kRoleScales))
      break;
    const int nh = min(2, n_sub - u0);  // sub-tiles of this stage inside the segment
    // K scale records of the stage's 128 keys, V scale words of its 128 channels, table entries
    uint2 kw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      kw[i] = *reinterpret_cast<const uint2*>(S.ksf[st] + (32 * i + lane) * 8);
    uint2 vw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      vw[i] = *reinterpret_cast<const uint2*>(S.vsf[st] + (32 * i + lane) * 8);
    float cv[2][4];
#pragma unroll
    for (int ft = 0; ft < 2; ++ft)
#pragma unroll
      for (int i = 0; i < 4; ++i) cv[ft][i] = (ft == 0 || two) ? S.cq[st][ft][32 * i + lane] : 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (h >= nh) break;
      const int x = (u0 + h) % kAuxBufs;
      // K scale blocks, one per K step kk: row i = (key i, key 32 + i) of the sub-tile, then two
      // zero words (an N = 64 MMA reads the first two columns)
      *reinterpret_cast<uint4*>(S.ksf_cp[x][0] + 16 * lane) =
          make_uint4(kw[2 * h].x, kw[2 * h + 1].x, 0u, 0u);
      *reinterpret_cast<uint4*>(S.ksf_cp[x][1] + 16 * lane) =
          make_uint4(kw[2 * h].y, kw[2 * h + 1].y, 0u, 0u);
      // V scale block: row i = channels i, 32 + i, 64 + i, 96 + i, the word of keys [64h, 64h+64)
      *reinterpret_cast<uint4*>(S.vsf_cp[x] + 16 * lane) =
          h ? make_uint4(vw[0].y, vw[1].y, vw[2].y, vw[3].y)
            : make_uint4(vw[0].x, vw[1].x, vw[2].x, vw[3].x);
      // fold B tiles: key row `key` = the table entry of query tile ft as three TF32 pieces:
      // hi = the entry's top 11 significant bits, mid = the next 11 of the exact remainder, lo =
      // the rest (at most 2 bits); each is exact in TF32 and hi + mid + lo is the entry
#pragma unroll
      for (int ft = 0; ft < 2; ++ft) {
        if (ft == 1 && !two) break;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int key = lane + 32 * r;
          const float v = cv[ft][2 * h + r];
          const uint32_t hi = __float_as_uint(v) & 0xFFFFE000u;
          const float rem = v - __uint_as_float(hi);
          const uint32_t mid = __float_as_uint(rem) & 0xFFFFE000u;
          const float lo = rem - __uint_as_float(mid);
          *reinterpret_cast<uint4*>(S.fb[x][ft] + (key >> 3) * 128 + (key & 7) * 16) =
              make_uint4(hi, mid, __float_as_uint(lo), 0u);
        }
      }
      fence_proxy_async_smem();  // the copies and the fold MMAs read these through the async proxy
      mbar_arrive(smem_u32(&S.bar_aux[x]));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&S.bar_free[st]));
  }
}

// ---------------------------------------------------------------------------------------------
// Softmax of query tile t (two threads per row) and the epilogue.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void softmax_and_epilogue(Smem& S, const Nvfp4Args& a,
                                                     const WorkItem& wi, const SegInfo& sg,
                                                     uint32_t tmem, int t, int wq, int lane) {
  const int n_sub = (sg.len + kSub - 1) / kSub;
  const float cs = a.scale_log2;
  const int q4 = wq & 3;
  const int rbase = 32 * q4 + 16 * (wq >> 2);  // rows of this warp: rbase + [0, 16)
  const int kh = lane >> 4;                    // keys [32 kh, 32 kh + 32) of every sub-tile
  const uint32_t lane_off = uint32_t(rbase) << 16;
  const uint32_t o_addr = tmem + col_o(t) + lane_off;
  const int last_valid = sg.len - (n_sub - 1) * kSub;  // keys of the last sub-tile, 1..64
  // Q scale factors, A side: row r reads lane r, column r / 32 of each K step's 4-column block;
  // thread kh writes K step kh's word (the 16x32bx2 store's second half lands 4 columns on)
  if (!wait_all(&S.bar_q, 0, S, a, kRoleSoftmax)) return;
  {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(S.qsf[t] + (rbase + (lane & 15)) * 8 +
                                                          4 * kh);
    tmem_st1x2<4>(tmem + col_qsf(t) + uint32_t(q4) + lane_off, w);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(smem_u32(&S.bar_qsf[t]));
  }
  const uint32_t s_addr = tmem + col_s(t) + lane_off;
  float m = -INFINITY;  // running maximum (log2 units)
  bool ok = true;
  // four sub-tiles per iteration: the slot and barrier parities become constants of each copy
#pragma unroll 4
  for (int u = 0; u < n_sub; ++u) {
    if (!(ok = wait_hinted(&S.bar_s[t], uint32_t(u) & 1, S, a, kRoleSoftmax))) break;
    tc_fence_after();
    // S already holds the qm K^T term (the fold MMA); the loads also return the maxima of this
    // thread's two 16-key scale groups
    uint32_t r[2][16];
    float gm[2];
    gm[0] = tmem_ld16x2_max<32>(s_addr, r[0]);
    gm[1] = tmem_ld16x2_max<32>(s_addr + 16, r[1]);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(smem_u32(&S.bar_sr[t]));  // S_t(u+1) may now overwrite S
    float s[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(r[i >> 4][i & 15]);
    if (u == n_sub - 1 && last_valid < kSub) {  // keys past the segment: mask, then reduce
      gm[0] = gm[1] = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (32 * kh + i >= last_valid) s[i] = -INFINITY;
        gm[i >> 4] = fmaxf(gm[i >> 4], s[i]);
      }
    }
    // raw S; s'' = S c enters only as the exp2 argument S c + gb (one FMA). c > 0, so the group
    // maxima of s'' are the raw maxima times c, exactly.
    gm[0] *= cs;
    gm[1] *= cs;
    float mx = fmaxf(gm[0], gm[1]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const bool move = mx > m;  // exact running maximum
    const float m_new = move ? mx : m;
    const float alpha = move ? ex2_approx(m - m_new) : 1.f;  // m = -inf gives 0
    const float bias = kLog2_2688 - m_new;                  // s'' + bias = log2 P'
    uint32_t pk[4];
    uint32_t sfw = 0u;
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {  // 16 keys per scale group
      // second level: UE4M3 scale of the group = E4M3(max P' / 6), max P' / 6 = 2^(gm + bias) / 6;
      // codes E2M1(P' / deq(scale)) = E2M1(2^(s'' + bias - log2 deq(scale))); scale 0 -> codes 0
      const uint32_t sf = cvt_e4m3x2(ex2_approx(gm[gi] + (bias - kLog2_6)), 0.f) & 0xFFu;
      const float ds = e4m3_to_f32(sf);
      const float gb = sf ? bias - lg2_approx(ds) : -INFINITY;
      uint32_t bt[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float x0, x1;
        fma2(x0, x1, s[16 * gi + 2 * i], s[16 * gi + 2 * i + 1], cs, gb);
        bt[i] = uint32_t(cvt_e2m1x2(ex2_approx(x0), ex2_approx(x1)));
      }
      pk[2 * gi] = __byte_perm(__byte_perm(bt[0], bt[1], 0x0040),
                               __byte_perm(bt[2], bt[3], 0x0040), 0x5410);
      pk[2 * gi + 1] = __byte_perm(__byte_perm(bt[4], bt[5], 0x0040),
                                   __byte_perm(bt[6], bt[7], 0x0040), 0x5410);
      sfw |= sf << (8 * gi);
    }
    // the row's four group scales: groups 0, 1 from thread kh = 0, groups 2, 3 from kh = 1
    const uint32_t other = __shfl_xor_sync(0xffffffffu, sfw, 16);
    const uint32_t sfrow = kh ? (other | (sfw << 16)) : (sfw | (other << 16));
    // the P slot was last read by PV_t(u-1)
    if (u >= 1) {
      if (!(ok = wait_hinted(&S.bar_o[t][(u - 1) & 1], ((u - 1) >> 1) & 1, S, a, kRoleSoftmax)))
        break;
      tc_fence_after();
    }
    // P codes (thread kh: keys 32 kh.., columns 4 kh..), the A-side P scales in column row / 32
    tmem_st4x2<4>(tmem + col_p(t) + lane_off, pk);
    tmem_st1x2<4>(tmem + col_psf(t) + uint32_t(q4) + lane_off, sfrow);
    if (u > 0 && __any_sync(0xffffffffu, move)) {
      // rescale O between PV_t(u-1) and PV_t(u): this thread's 72 of the 144 columns
#pragma unroll 1
      for (int i = 0; i < 2; ++i) {
        uint32_t o[32];
        tmem_ld32x2<72>(o_addr + 32 * i, o);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float a0, a1;
          fma2(a0, a1, __uint_as_float(o[e]), __uint_as_float(o[e + 1]), alpha, 0.f);
          o[e] = __float_as_uint(a0);
          o[e + 1] = __float_as_uint(a1);
        }
        tmem_st32x2<72>(o_addr + 32 * i, o);
      }
      uint32_t o3[8];  // the last 8 of this thread's columns (l among them for kh = 1)
      tmem_ld8x2<72>(o_addr + 64, o3);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 8; ++e) o3[e] = __float_as_uint(__uint_as_float(o3[e]) * alpha);
      tmem_st8x2<72>(o_addr + 64, o3);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(smem_u32(&S.bar_p[t][u & 1]));
    m = m_new;
  }
  if (!ok) {
    tmem_wait_st();
    return;
  }
  // PV_t(n_sub - 1) done implies every earlier PV of the in-order stream is done
  if (!wait_all(&S.bar_o[t][(n_sub - 1) & 1], ((n_sub - 1) >> 1) & 1, S, a, kRoleEpilogue))
    return;
  tc_fence_after();
  // sum of the dequantized P: columns 128 and 129 both hold it (the 16 row-sum columns agree)
  const float l = __uint_as_float(tmem_ld1x2<1>(o_addr + 128));
  tmem_wait_ld();
  const float f = __frcp_rn(l);
  const int qrow = (wi.qt0 + t) * kTile + rbase + (lane & 15);
  const bool valid = qrow < sg.len;
  // LSE of the uncentred scores: (m + log2(l) - log2 2688) ln 2 + (q . km) scale
  if (a.lse && valid && kh == 0)
    a.lse[int64_t(wi.head) * a.lse_sh + sg.tok0 + qrow] =
        (m + log2f(l) - kLog2_2688) * 0.6931471805599453f +
        a.q_km[int64_t(wi.head) * a.tpad + sg.row0 + qrow] * a.scale;
  // this thread's channels: [0, 64) (kh = 0) or [64, 128) (kh = 1)
  __nv_bfloat16* dst =
      a.out + int64_t(sg.tok0 + qrow) * a.ost + int64_t(wi.head) * a.osh + 64 * kh;
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
    attn_nvfp4_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ Nvfp4Args a) {
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
      mbar_init(smem_u32(&S.bar_free[i]), wi.nq + 1);  // MMA commits + the auxiliary warp
    }
    for (int x = 0; x < kAuxBufs; ++x) {
      mbar_init(smem_u32(&S.bar_aux[x]), 32);
      mbar_init(smem_u32(&S.bar_auxfree[x]), wi.nq);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&S.bar_qsf[t]), 256);
      mbar_init(smem_u32(&S.bar_s[t]), 1);
      mbar_init(smem_u32(&S.bar_sr[t]), 256);
      for (int x = 0; x < 2; ++x) {
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
  // fold operands: A rows [1, 1, 1, 0] (TF32 1.0 = 0x3F800000) then a zero core matrix; B zero
  // halves; the 1.0 rows' scale block; the 1.0 rows of every V^T stage
  if (threadIdx.x < 16) {
    const uint4 v1 = threadIdx.x < 8 ? make_uint4(0x3F800000u, 0x3F800000u, 0x3F800000u, 0u)
                                     : make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(S.fa)[threadIdx.x] = v1;
  }
  for (int i = threadIdx.x; i < kAuxBufs * 2 * 64; i += kThreads)
    reinterpret_cast<uint4*>(S.fb[i >> 7][(i >> 6) & 1] + 1024)[i & 63] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x < 32) {  // UE4M3 1.0 = 0x38 for the 16 rows of 1.0 (lanes 0-15)
    const uint32_t one = threadIdx.x < 16 ? 0x38383838u : 0u;
    reinterpret_cast<uint4*>(S.ones_cp)[threadIdx.x] = make_uint4(one, 0u, 0u, 0u);
  }
  for (int i = threadIdx.x; i < kStages * 64; i += kThreads)  // E2M1 1.0 = 0x2, two per byte
    reinterpret_cast<uint4*>(S.v[i >> 6] + kCodeTile)[i & 63] =
        make_uint4(0x22222222u, 0x22222222u, 0x22222222u, 0x22222222u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == kTmaWarp) {
    producer(&tm_q, &tm_k, &tm_v, S, a, wi, sg);
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    const int t = warp - kMmaWarp;
    if (t < wi.nq) mma_issuer(S, a, wi, sg, tmem, t);
  } else if (warp == kAuxWarp) {
    aux_warp(S, a, wi, sg, lane);
  } else {
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

int launch_nvfp4_attention(const fa_lp_plan& p, uint8_t* ws, int g, void* out, int64_t ost,
                           int64_t osh, float* lse, int64_t lse_sh, cudaStream_t stream) {
  const int w0 = p.tbl_work_off[g], nw = p.tbl_work_off[g + 1] - w0;
  if (nw <= 0) return FA_LP_OK;
  static std::atomic<uint64_t> smem_set{0};
  if (set_smem_limit_once(reinterpret_cast<const void*>(attn_nvfp4_kernel), int(kSmemBytes), p.device,
                          smem_set) != FA_LP_OK)
    return FA_LP_ERR_CUDA;
  const uint64_t H = uint64_t(p.heads), Tp = uint64_t(p.tpad);
  CUtensorMap tq, tk, tv;
  // Q, K codes: [H][Tp][64 bytes]; V^T codes: [H][128][Tp / 2 bytes]; boxes of 128 rows x 64 B
  int st = encode_tmap_3d_u8(&tq, ws + p.ws.q_codes, 64, Tp, H, 64, Tp * 64, 64, 128,
                             CU_TENSOR_MAP_SWIZZLE_64B);
  if (st == FA_LP_OK)
    st = encode_tmap_3d_u8(&tk, ws + p.ws.k_codes, 64, Tp, H, 64, Tp * 64, 64, 128,
                           CU_TENSOR_MAP_SWIZZLE_64B);
  if (st == FA_LP_OK)
    st = encode_tmap_3d_u8(&tv, ws + p.ws.v_codes, Tp / 2, 128, H, Tp / 2, 128 * (Tp / 2), 64,
                           128, CU_TENSOR_MAP_SWIZZLE_64B);
  if (st != FA_LP_OK) return st;
  Nvfp4Args a;
  a.segs = p.d_segs;
  a.work = p.d_work + w0;
  a.q_sf = ws + p.ws.q_sf;
  a.k_sf = ws + p.ws.k_sf;
  a.v_sf = ws + p.ws.v_sf;
  a.qmk = reinterpret_cast<const float*>(ws + p.ws.qmk) + size_t(g % p.tbl_slots) * p.tbl_slot_floats;
  a.c_off = p.d_coff;
  a.tbl_h0 = g * p.tbl_hg;
  a.q_km = reinterpret_cast<const float*>(ws + p.ws.q_km);
  a.lse = lse;
  a.lse_sh = lse_sh;
  a.scale = p.scale;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ost = ost;
  a.osh = osh;
  a.tpad = p.tpad;
  a.scale_log2 = p.scale * 1.4426950408889634f;
  a.w.err = p.d_err;
  a.w.abort_word = p.d_err + 1;
  a.w.gen = next_launch_generation();
  a.w.spin_limit = p.spin_limit;
  attn_nvfp4_kernel<<<unsigned(nw), kThreads, kSmemBytes, stream>>>(tq, tk, tv, a);
  return cuda_status(cudaGetLastError());
}

}  // namespace falp
