// fa_lp_api.cu -- the C ABI entry points of libfa_lp.so: plan building and caching, argument
// validation, the per-device grow-only workspace, and dispatch to the CUDA launchers.
//
// Passages: FlashInfer docs, flashinfer.diffusion_ops.minimax_h3_sm120_varlen_attention_nvfp4,
// Parameters (cu_seqlens contract, host copy, plan cache keyed by (cu_seqlens, heads, device),
// default softmax scale) and description (grow-only per-device workspace shared by the FP8 and
// NVFP4 ops); SGLang PR #40175, review replies (no input references retained, output owned by the
// caller, allocation stream-ordered on the calling stream).
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "fa_lp_internal.h"

using falp::BlockInfo;
using falp::SegInfo;
using falp::WorkItem;
using falp::QmkItem;

namespace {

std::mutex g_mu;

// ---- plan cache, keyed by (cu_seqlens, tokens, heads, scale bits, mode, device) ---------------
using PlanKey = std::tuple<std::vector<int32_t>, int64_t, int, uint32_t, int, int>;
std::map<PlanKey, fa_lp_plan*> g_plans;

PlanKey key_of(const fa_lp_plan& p) {
  uint32_t sb;
  std::memcpy(&sb, &p.scale, 4);
  return PlanKey(p.cu, p.tokens, p.heads, sb, p.mode, p.device);
}

bool log_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("FA_LP_LOG");
    return e && e[0] == '1';
  }();
  return on;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---- per-device workspace ----------------------------------------------------------------------
struct DevWs {
  void* ptr = nullptr;
  size_t bytes = 0;
  // the plan whose codes the workspace holds (the last quantize on this device) and that
  // quantize's generation: a forward of any other plan finds its codes overwritten
  const fa_lp_plan* owner = nullptr;
  uint64_t gen = 0;
};
std::map<int, DevWs> g_ws;
uint64_t g_quant_gen = 0;  // generations of fa_lp_quantize calls (under g_mu)

// Workspace base of plan p for a forward, or FA_LP_ERR_STATE when the workspace no longer holds
// p's codes (never quantized, released, grown, or another plan quantized since). Under g_mu.
int workspace_of_plan(const fa_lp_plan* p, void** base) {
  const DevWs& w = g_ws[p->device];
  if (!w.ptr || w.bytes < p->ws.total || w.owner != p || w.gen != p->quant_gen)
    return FA_LP_ERR_STATE;
  *base = w.ptr;
  return FA_LP_OK;
}

// ---- device capability check ---------------------------------------------------------------------
int check_device(int device) {
  static std::mutex mu;
  static std::map<int, int> cache;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(device);
  if (it != cache.end()) return it->second;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess) {
    cudaGetLastError();
    return FA_LP_ERR_CUDA;
  }
  const int st = (major == 10 && minor == 3) ? FA_LP_OK : FA_LP_ERR_UNSUPPORTED;
  cache[device] = st;
  return st;
}

int check_current_device(const fa_lp_plan* p) {
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return FA_LP_ERR_CUDA;
  if (cur != p->device) return FA_LP_ERR_INVALID_ARG;
  return check_device(p->device);
}

// Upload the plan's segment / block / work tables once (stream-ordered).
int ensure_device_meta(fa_lp_plan* p, cudaStream_t stream) {
  if (p->dmeta) return FA_LP_OK;
  const size_t n_seg = p->segs.size() * sizeof(SegInfo);
  const size_t n_blk = p->blocks.size() * sizeof(BlockInfo);
  const size_t n_wrk = p->work.size() * sizeof(WorkItem);
  const size_t n_qmk = p->qmk_items.size() * sizeof(QmkItem);
  const size_t n_cof = p->c_off.size() * sizeof(int64_t);
  const size_t n_qb0 = p->sp_qb0.size() * sizeof(int32_t);
  const size_t n_spg = p->sp_groups.size() * sizeof(falp::SparseGroup);
  const size_t n_spc = p->sp_ctas.size() * sizeof(falp::SparseCta);
  const size_t o_seg = 0;
  const size_t o_blk = align_up(o_seg + n_seg, 256);
  const size_t o_wrk = align_up(o_blk + n_blk, 256);
  const size_t o_qmk = align_up(o_wrk + n_wrk, 256);
  const size_t o_cof = align_up(o_qmk + n_qmk, 256);
  const size_t o_qb0 = align_up(o_cof + n_cof, 256);
  const size_t o_spg = align_up(o_qb0 + n_qb0, 256);
  const size_t o_spc = align_up(o_spg + n_spg, 256);
  const size_t o_err = align_up(o_spc + n_spc, 256);
  const size_t total = o_err + 256;
  void* d = nullptr;
  if (cudaMalloc(&d, total) != cudaSuccess) {
    cudaGetLastError();
    return FA_LP_ERR_OOM;
  }
  std::vector<uint8_t> host(total, 0);
  if (n_seg) std::memcpy(host.data() + o_seg, p->segs.data(), n_seg);
  if (n_blk) std::memcpy(host.data() + o_blk, p->blocks.data(), n_blk);
  if (n_wrk) std::memcpy(host.data() + o_wrk, p->work.data(), n_wrk);
  if (n_qmk) std::memcpy(host.data() + o_qmk, p->qmk_items.data(), n_qmk);
  if (n_cof) std::memcpy(host.data() + o_cof, p->c_off.data(), n_cof);
  if (n_qb0) std::memcpy(host.data() + o_qb0, p->sp_qb0.data(), n_qb0);
  if (n_spg) std::memcpy(host.data() + o_spg, p->sp_groups.data(), n_spg);
  if (n_spc) std::memcpy(host.data() + o_spc, p->sp_ctas.data(), n_spc);
  if (cudaMemcpyAsync(d, host.data(), total, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaFree(d);
    cudaGetLastError();
    return FA_LP_ERR_CUDA;
  }
  p->dmeta = d;
  uint8_t* b = static_cast<uint8_t*>(d);
  p->d_segs = reinterpret_cast<SegInfo*>(b + o_seg);
  p->d_blocks = reinterpret_cast<BlockInfo*>(b + o_blk);
  p->d_work = reinterpret_cast<WorkItem*>(b + o_wrk);
  p->d_qmk = reinterpret_cast<QmkItem*>(b + o_qmk);
  p->d_coff = reinterpret_cast<int64_t*>(b + o_cof);
  p->d_sp_qb0 = reinterpret_cast<int32_t*>(b + o_qb0);
  p->d_sp_groups = reinterpret_cast<falp::SparseGroup*>(b + o_spg);
  p->d_sp_ctas = reinterpret_cast<falp::SparseCta*>(b + o_spc);
  p->d_err = reinterpret_cast<int*>(b + o_err);
  if (log_enabled())
    std::fprintf(stderr, "[fa_lp] plan %p: device tables %zu bytes on device %d\n", (void*)p,
                 total, p->device);
  return FA_LP_OK;
}

bool bad_view(const void* ptr, int64_t st, int64_t sh) {
  if (!ptr) return true;
  if (st <= 0 || sh <= 0) return true;
  if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return true;
  if (st % 8 != 0 || sh % 8 != 0) return true;  // 16-byte aligned rows of 128 BF16
  return false;
}

// ---- host-buffer pipeline ------------------------------------------------------------------------
// Copy heads [h0, h0 + n) of a BF16 [T, H, 128] view (element strides st, sh) into or out of a
// dense [T, n, 128] device buffer: one 2D copy when the heads are adjacent, else one per head.
cudaError_t copy_heads(void* dst, int64_t dst_st, int64_t dst_sh, const void* src, int64_t src_st,
                       int64_t src_sh, int64_t T, int n, cudaMemcpyKind kind, cudaStream_t s) {
  const size_t row = size_t(FA_LP_HEAD_DIM) * 2;
  if (dst_sh == FA_LP_HEAD_DIM && src_sh == FA_LP_HEAD_DIM)
    return cudaMemcpy2DAsync(dst, size_t(dst_st) * 2, src, size_t(src_st) * 2, row * n, size_t(T),
                             kind, s);
  for (int h = 0; h < n; ++h) {
    const cudaError_t e = cudaMemcpy2DAsync(
        static_cast<uint8_t*>(dst) + size_t(h) * dst_sh * 2, size_t(dst_st) * 2,
        static_cast<const uint8_t*>(src) + size_t(h) * src_sh * 2, size_t(src_st) * 2, row,
        size_t(T), kind, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Device address of a page-locked host view the current device can read directly, or nullptr
// (pageable memory, device memory, or a view not 16-byte aligned in its base and strides).
const void* device_mapping(const void* host, int64_t st, int64_t sh) {
  if ((reinterpret_cast<uintptr_t>(host) & 15) != 0 || (st * 2) % 16 != 0 || (sh * 2) % 16 != 0)
    return nullptr;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// Copy-in of one tensor of a chunk: a 2D DMA copy, or, for the first chunk (whose copy-in no
// compute overlaps) from page-locked memory, the gather kernel, which is not slowed by the DMA
// engine's per-row cost.
cudaError_t copy_in(void* dst, const void* src, int64_t st, int64_t sh, int64_t T, int n,
                    bool gather, cudaStream_t s) {
  const void* d = gather ? device_mapping(src, st, sh) : nullptr;
  if (d) return falp::launch_gather_heads(dst, d, st, sh, T, n, s) == FA_LP_OK ? cudaSuccess
                                                                              : cudaErrorUnknown;
  return copy_heads(dst, int64_t(n) * FA_LP_HEAD_DIM, FA_LP_HEAD_DIM, src, st, sh, T, n,
                    cudaMemcpyHostToDevice, s);
}

// Chunks of heads for the host-buffer pipeline: equal chunks (the last may be shorter) of
// heads_per_chunk heads, or, when the caller leaves it open, of the size that gives 4 to 8 chunks
// whose CTAs fill the GPU's waves best (ties: more chunks, so that the first copy-in and the last
// copy-out, which nothing overlaps, are shorter).
std::vector<int> host_schedule(const fa_lp_plan& p, int heads_per_chunk, bool sparse) {
  const int H = p.heads;
  int nh = heads_per_chunk;
  if (nh <= 0) {
    nh = H < 4 ? 1 : (H + 3) / 4;
    if (H >= 4) {
      int sms = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p.device) != cudaSuccess ||
          sms <= 0) {
        cudaGetLastError();
        sms = 152;
      }
      const double cph = double(p.work.size()) / H;  // CTAs per head
      double best_eff = -1.0;
      for (int n = 1; n <= H; ++n) {
        const int nc = (H + n - 1) / n;
        if (nc < 4 || nc > 8) continue;
        double ctas = 0.0, slots = 0.0;
        for (int h0 = 0; h0 < H; h0 += n) {
          const double c = cph * std::min(n, H - h0);
          ctas += c;
          slots += std::ceil(c / sms) * sms;
        }
        const double eff = slots > 0 ? ctas / slots : 0.0;
        if (eff > best_eff + 1e-9 || (std::fabs(eff - best_eff) <= 1e-9 && n < nh)) {
          best_eff = eff;
          nh = n;
        }
      }
    }
  }
  std::vector<int> out;
  if (heads_per_chunk <= 0 && nh >= 2 && H >= 3 * nh) {
    // the library's choice: a short first chunk, whose copy-in nothing overlaps, then chunks of
    // nh, the last one the remainder (its copy-out overlaps nothing either). The first chunk
    // computes about as long as the next chunk's copy-in takes: half a chunk for NVFP4 and the
    // block-sparse forward; for the dense FP8 forward, which computes a head in ~0.22 ms while a
    // 14-head chunk's DMA copy-in moves one in ~0.15 ms, two thirds of a chunk (at S=30272,
    // H=56: [9, 14, 14, 14, 5], median host-entry step 14.00 ms against 14.25 ms for
    // [7, 14, 14, 14, 7])
    const int first = (falp::is_fp8(p) && !sparse) ? (2 * nh + 1) / 3 : (nh + 1) / 2;
    int rest = H - first;
    out.push_back(first);
    while (rest > nh) {
      out.push_back(nh);
      rest -= nh;
    }
    if (rest > 0) out.push_back(rest);
    return out;
  }
  for (int h0 = 0; h0 < H; h0 += nh) out.push_back(std::min(nh, H - h0));
  return out;
}

// Streams and events of the NVFP4 table ring (device already current).
int table_ring_release(fa_lp_plan* p) {
  int st = FA_LP_OK;
  for (int i = 0; i < 2; ++i) {
    if (p->tbl_stream[i]) {
      if (cudaStreamSynchronize(p->tbl_stream[i]) != cudaSuccess) st = FA_LP_ERR_CUDA;
      cudaStreamDestroy(p->tbl_stream[i]);
      p->tbl_stream[i] = nullptr;
    }
    if (p->tbl_join[i]) cudaEventDestroy(p->tbl_join[i]);
    p->tbl_join[i] = nullptr;
  }
  if (p->tbl_fork) cudaEventDestroy(p->tbl_fork);
  p->tbl_fork = nullptr;
  if (st != FA_LP_OK) cudaGetLastError();
  return st;
}

// NVFP4 forward with the qm K^T table held as a ring of two head-group slots. Group g's table
// build and attention launch go to internal stream g % 2: a slot is rewritten only after the
// attention launch that read it (stream order), and one stream's table build and attention run
// beside the other stream's attention. Both streams start after the work already queued on
// `stream`, and `stream` continues after both.
int nvfp4_ring_forward(fa_lp_plan* p, uint8_t* base, void* out, int64_t ost, int64_t osh,
                       float* lse, int64_t lse_sh, cudaStream_t stream) {
  if (!p->tbl_fork) {
    bool ok = cudaEventCreateWithFlags(&p->tbl_fork, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; i < 2 && ok; ++i)
      ok = cudaStreamCreateWithFlags(&p->tbl_stream[i], cudaStreamNonBlocking) == cudaSuccess &&
           cudaEventCreateWithFlags(&p->tbl_join[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      table_ring_release(p);
      return FA_LP_ERR_CUDA;
    }
  }
  if (cudaEventRecord(p->tbl_fork, stream) != cudaSuccess ||
      cudaStreamWaitEvent(p->tbl_stream[0], p->tbl_fork, 0) != cudaSuccess ||
      cudaStreamWaitEvent(p->tbl_stream[1], p->tbl_fork, 0) != cudaSuccess) {
    cudaGetLastError();
    return FA_LP_ERR_CUDA;
  }
  const int ng = int(p->tbl_work_off.size()) - 1;
  int st = FA_LP_OK;
  for (int g = 0; g < ng && st == FA_LP_OK; ++g) {
    cudaStream_t sg = p->tbl_stream[g & 1];
    st = falp::launch_nvfp4_qmk(*p, base, g, sg);
    if (st == FA_LP_OK)
      st = falp::launch_nvfp4_attention(*p, base, g, out, ost, osh, lse, lse_sh, sg);
  }
  // joined after a failed launch as well, so that `stream` never runs ahead of queued work
  for (int i = 0; i < 2; ++i)
    if (cudaEventRecord(p->tbl_join[i], p->tbl_stream[i]) != cudaSuccess ||
        cudaStreamWaitEvent(stream, p->tbl_join[i], 0) != cudaSuccess) {
      cudaGetLastError();
      st = FA_LP_ERR_CUDA;
    }
  return st;
}

// Free the pipeline's device buffer, streams and events (device already current); hands the
// sub-plans to the caller, which releases them outside the plan-cache lock.
int host_pipe_release(fa_lp_plan* p, fa_lp_plan* subs[4]) {
  falp::HostPipe& hp = p->host;
  int st = FA_LP_OK;
  if (hp.s_in && cudaStreamSynchronize(hp.s_in) != cudaSuccess) st = FA_LP_ERR_CUDA;
  if (hp.s_out && cudaStreamSynchronize(hp.s_out) != cudaSuccess) st = FA_LP_ERR_CUDA;
  if (hp.buf && cudaFree(hp.buf) != cudaSuccess) st = FA_LP_ERR_CUDA;
  if (hp.lists && cudaFree(hp.lists) != cudaSuccess) st = FA_LP_ERR_CUDA;
  for (cudaEvent_t* e : {&hp.start, &hp.end, &hp.in_done[0], &hp.in_done[1], &hp.in_free[0],
                         &hp.in_free[1], &hp.out_ready[0], &hp.out_ready[1], &hp.out_free[0],
                         &hp.out_free[1]})
    if (*e) cudaEventDestroy(*e);
  if (hp.s_in) cudaStreamDestroy(hp.s_in);
  if (hp.s_out) cudaStreamDestroy(hp.s_out);
  for (int i = 0; i < 4; ++i) subs[i] = hp.sub[i];
  hp = falp::HostPipe();
  if (st != FA_LP_OK) cudaGetLastError();
  return st;
}

// Heads per block of the work list (and per block-sparse tile group).
constexpr int kHeadGroup = 8;
// Largest NVFP4 qm K^T table a plan holds whole (bytes); a larger one is held as a ring of two
// head-group slots that the forward fills group by group. Holding the whole table keeps its build
// in the quantize, where it runs alone at full width (0.61 ms at S = 30272, H = 56, against
// 0.84 ms spread over the forward's head groups); above 4 GB (one segment of about 49.5k tokens at
// H = 56) the ring bounds it.
constexpr size_t kTableLimitDefault = size_t(4) << 30;

// Segments, longest first (ties in index order).
std::vector<int> lpt_order(const fa_lp_plan* p) {
  std::vector<int> order(p->nseg);
  for (int s = 0; s < p->nseg; ++s) order[s] = s;
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return p->segs[a].len > p->segs[b].len; });
  return order;
}

void layout_work_and_workspace(fa_lp_plan* p);

void build_plan(fa_lp_plan* p) {
  const int ns = p->nseg;
  p->row_off.assign(ns + 1, 0);
  p->segs.resize(ns);
  int64_t row = 0;
  for (int s = 0; s < ns; ++s) {
    const int64_t L = int64_t(p->cu[s + 1]) - p->cu[s];
    const int64_t nb = (L + falp::kTile - 1) / falp::kTile;
    p->row_off[s] = row;
    p->segs[s] = SegInfo{p->cu[s], int32_t(L), int32_t(row), int32_t(nb)};
    for (int64_t b = 0; b < nb; ++b) {
      const int64_t nv = std::min<int64_t>(falp::kTile, L - b * falp::kTile);
      p->blocks.push_back(BlockInfo{int32_t(p->cu[s] + b * falp::kTile), int32_t(nv), s, int32_t(b)});
    }
    row += nb * falp::kTile;
  }
  p->row_off[ns] = row;
  p->tpad = row;
  // block-sparse lists: 64-row query blocks and 64-key blocks per segment
  p->sp_qb0.assign(ns, 0);
  for (int s = 0; s < ns; ++s) {
    const int64_t nkb = (int64_t(p->cu[s + 1]) - p->cu[s] + 63) / 64;
    p->sp_qb0[s] = int32_t(p->sp_G);
    p->sp_G += nkb;
    p->sp_nw_max = std::max<int>(p->sp_nw_max, int((nkb + 31) / 32));
  }

  std::vector<int> order = lpt_order(p);
  // Block-sparse forward: the same segment / head-group order; a group's tiles are paired on the
  // device once their list lengths are known.
  int32_t slot = 0;
  for (int s : order) {
    const int nb = p->segs[s].nblk;
    if (nb == 0) continue;
    for (int h0 = 0; h0 < p->heads; h0 += kHeadGroup) {
      const int nh = std::min(kHeadGroup, p->heads - h0);
      const int nt = nh * nb;
      p->sp_groups.push_back(falp::SparseGroup{slot, h0, nh, s});
      for (int i = 0; i < nt; i += 2)
        p->sp_ctas.push_back(falp::SparseCta{slot + i, std::min(2, nt - i)});
      slot += nt;
    }
  }
  layout_work_and_workspace(p);
}

// Table groups of the NVFP4 qm K^T table (heads per group, slots), the work list ordered by
// group, and the workspace layout. Re-run when the plan's table limit changes.
void layout_work_and_workspace(fa_lp_plan* p) {
  const int ns = p->nseg;
  const std::vector<int> order = lpt_order(p);
  // one head's table, in floats, over all segments
  size_t head_floats = 0;
  for (int s = 0; s < ns; ++s)
    head_floats += size_t(p->segs[s].nblk) * size_t(p->segs[s].nblk) * 128;
  p->tbl_hg = p->heads;
  p->tbl_slots = 1;
  if (!falp::is_fp8(*p) && head_floats > 0) {
    const size_t limit = p->tbl_limit ? p->tbl_limit : kTableLimitDefault;
    if (size_t(p->heads) * head_floats * 4 > limit) {
      // a ring of two slots of at most limit / 2 bytes each (one head's table at the least);
      // groups of equal size
      const size_t fit = std::max<size_t>(1, (limit / 2) / (head_floats * 4));
      const int ng = int((size_t(p->heads) + fit - 1) / fit);
      p->tbl_hg = (p->heads + ng - 1) / ng;
      p->tbl_slots = 2;
    }
  }
  p->tbl_slot_floats = size_t(p->tbl_hg) * head_floats;

  // Work list, per table group (one group of all heads unless the table is held as a ring):
  // longest segment first (LPT); within a segment, blocks of kHeadGroup heads, and in a block
  // the query-tile pairs of its heads interleaved. The CTAs resident at one time then read the
  // K/V of a few heads (a working set that stays in L2) while no single K/V line is requested by
  // all of them at once.
  p->work.clear();
  p->tbl_work_off.clear();
  for (int g0 = 0; g0 < p->heads; g0 += p->tbl_hg) {
    const int g1 = std::min(p->heads, g0 + p->tbl_hg);
    p->tbl_work_off.push_back(int32_t(p->work.size()));
    for (int s : order) {
      const int nb = p->segs[s].nblk;
      if (nb == 0) continue;
      for (int h0 = g0; h0 < g1; h0 += kHeadGroup)
        for (int t = 0; t < nb; t += 2)
          for (int h = h0; h < std::min(g1, h0 + kHeadGroup); ++h)
            p->work.push_back(WorkItem{s, h, t, std::min(2, nb - t)});
    }
  }
  p->tbl_work_off.push_back(int32_t(p->work.size()));

  // Workspace layout.
  const size_t H = size_t(p->heads), Tp = size_t(p->tpad);
  p->ws = falp::WsLayout();
  falp::WsLayout& w = p->ws;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + std::max<size_t>(bytes, 1), 1024);
    return o;
  };
  if (falp::is_fp8(*p)) {
    const size_t R = size_t(falp::fp8_scale_rows(*p));
    w.q_codes = take(H * Tp * 128);
    w.k_codes = take(H * Tp * 128);
    w.v_codes = take(H * 128 * Tp);
    w.amax = take(3 * R * H * 4);
    w.descale = take(3 * R * H * 4);
  } else {
    w.q_codes = take(H * Tp * 64);
    w.k_codes = take(H * Tp * 64);
    w.v_codes = take(H * 128 * Tp / 2);
    w.q_sf = take(H * Tp * 8);
    w.k_sf = take(H * Tp * 8);
    w.v_sf = take(H * 128 * (Tp / 16));
    w.q_mean = take(H * (Tp / 128) * 128 * 4);
    w.k_mean = take(size_t(p->nseg) * H * 128 * 4);
    w.k_chunk = take(p->blocks.size() * H * 128 * 8);
    w.q_km = take(H * Tp * 4);
    // qm K^T table slot: segment s holds [tbl_hg][nb_s][128 nb_s] floats (quadratic in the
    // segment length: 1.6 GB for one 30272-token segment at H = 56 when one slot holds every
    // head)
    p->c_off.assign(ns, 0);
    p->qmk_items.clear();
    size_t floats = 0;
    // N tiles per table CTA: one run r for every segment, since the table kernel launches all
    // segments' tiles of a head group in one grid: the r whose CTAs (sum over segments of M tiles
    // x runs, times the group's heads) fill the GPU's waves best, i.e. the least
    // ceil(CTAs / SMs) * r (a CTA's time grows with its run); ties go to the longer run. r is at
    // least 4 when one launch covers every head (the per-CTA set-up then stays small against
    // its run), at least 1 for a head group
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess ||
        sms <= 0) {
      cudaGetLastError();
      sms = 152;
    }
    auto ntiles_of = [&](int s) { return (int64_t(p->segs[s].nblk) * 128 + 255) / 256; };
    auto nm_of = [&](int s) { return (int64_t(p->segs[s].nblk) + 127) / 128; };
    int run = falp::kQmkTilesPer;
    double best = 1e300;
    for (int r = p->tbl_slots == 1 ? 4 : 1; r <= 16; ++r) {
      double ctas = 0.0;
      for (int s = 0; s < ns; ++s)
        ctas += double(nm_of(s)) * double((ntiles_of(s) + r - 1) / r) * double(p->tbl_hg);
      const double cost = std::ceil(ctas / sms) * r;
      if (cost < best - 1e-9 || (std::fabs(cost - best) <= 1e-9 && r > run)) {
        best = cost;
        run = r;
      }
    }
    for (int s = 0; s < ns; ++s) {
      const int64_t nb = p->segs[s].nblk;
      p->c_off[s] = int64_t(floats);
      floats += size_t(p->tbl_hg) * size_t(nb) * size_t(nb) * 128;
      const int64_t ntiles = ntiles_of(s);
      for (int64_t mt = 0; mt * 128 < nb; ++mt)
        for (int64_t nt = 0; nt < ntiles; nt += run)
          p->qmk_items.push_back(falp::QmkItem{
              s, int32_t(mt), int32_t(nt), int32_t(std::min<int64_t>(run, ntiles - nt))});
    }
    w.qmk = take(floats * 4 * size_t(p->tbl_slots));
  }
  w.total = off;
}

}  // namespace

namespace falp {

int next_launch_generation() {
  static std::atomic<int> g{0};
  int v = g.fetch_add(1) + 1;
  if (v <= 0) {  // wrapped: restart at 1
    g.store(1);
    v = 1;
  }
  return v;
}

int workspace_acquire(int device, size_t bytes, cudaStream_t stream, void** base) {
  std::lock_guard<std::mutex> lk(g_mu);
  DevWs& w = g_ws[device];
  if (w.bytes < bytes) {
    if (w.ptr) {
      if (cudaFreeAsync(w.ptr, stream) != cudaSuccess) {
        cudaGetLastError();
        return FA_LP_ERR_CUDA;
      }
      w.ptr = nullptr;
      w.bytes = 0;
    }
    void* p = nullptr;
    if (cudaMallocAsync(&p, bytes, stream) != cudaSuccess) {
      cudaGetLastError();
      return FA_LP_ERR_OOM;
    }
    w.ptr = p;
    w.bytes = bytes;
    if (log_enabled())
      std::fprintf(stderr, "[fa_lp] workspace on device %d grown to %zu bytes\n", device, bytes);
  }
  *base = w.ptr;
  return FA_LP_OK;
}

int encode_tmap_3d_u8(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
                      uint32_t box1, CUtensorMapSwizzle swz) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    else
      cudaGetLastError();
  });
  if (!fn) return FA_LP_ERR_CUDA;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_LP_OK : FA_LP_ERR_CUDA;
}

}  // namespace falp

extern "C" {

const char* fa_lp_status_string(int status) {
  switch (status) {
    case FA_LP_OK: return "ok";
    case FA_LP_ERR_INVALID_ARG: return "invalid argument";
    case FA_LP_ERR_UNSUPPORTED: return "unsupported (this library serves sm_103 GPUs only)";
    case FA_LP_ERR_CUDA: return "CUDA error";
    case FA_LP_ERR_OOM: return "out of device memory";
    case FA_LP_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait expired";
    case FA_LP_ERR_STATE:
      return "call out of order (quantize this plan before its forward; another plan's quantize "
             "on the same device in between overwrites the shared workspace)";
    default: return "unknown status";
  }
}

int fa_lp_plan_create(int64_t tokens, int heads, const int32_t* cu, int num_segments,
                      float softmax_scale, int mode, int device, fa_lp_plan** out) {
  if (!out || !cu) return FA_LP_ERR_INVALID_ARG;
  *out = nullptr;
  if (tokens < 0 || tokens > (int64_t(1) << 30)) return FA_LP_ERR_INVALID_ARG;
  if (heads < 1 || heads > 1024 || num_segments < 1 || device < 0) return FA_LP_ERR_INVALID_ARG;
  if (mode != FA_LP_MODE_FP8 && mode != FA_LP_MODE_NVFP4 && mode != FA_LP_MODE_FP8_SEGMENT)
    return FA_LP_ERR_INVALID_ARG;
  if (cu[0] != 0 || int64_t(cu[num_segments]) != tokens) return FA_LP_ERR_INVALID_ARG;
  for (int s = 0; s < num_segments; ++s)
    if (cu[s + 1] < cu[s]) return FA_LP_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
    softmax_scale = 1.0f / std::sqrt(float(FA_LP_HEAD_DIM));

  auto* p = new fa_lp_plan();
  p->tokens = tokens;
  p->heads = heads;
  p->nseg = num_segments;
  p->scale = softmax_scale;
  p->mode = mode;
  p->device = device;
  p->cu.assign(cu, cu + num_segments + 1);

  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_plans.find(key_of(*p));
  if (it != g_plans.end()) {
    delete p;
    it->second->refcount++;
    *out = it->second;
    return FA_LP_OK;
  }
  build_plan(p);
  g_plans[key_of(*p)] = p;
  if (log_enabled())
    std::fprintf(stderr, "[fa_lp] plan %p: T=%lld H=%d segs=%d Tpad=%lld items=%zu ws=%zu\n",
                 (void*)p, (long long)tokens, heads, num_segments, (long long)p->tpad,
                 p->work.size(), p->ws.total);
  *out = p;
  return FA_LP_OK;
}

int fa_lp_plan_destroy(fa_lp_plan* p) {
  if (!p) return FA_LP_OK;
  fa_lp_plan* subs[4] = {nullptr, nullptr, nullptr, nullptr};
  int st = FA_LP_OK;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (--p->refcount > 0) return FA_LP_OK;
    g_plans.erase(key_of(*p));
    if (p->dmeta || p->host.buf || p->host.s_in || p->sp_buf || p->tbl_fork) {
      int cur = -1;
      cudaGetDevice(&cur);
      if (cur != p->device) cudaSetDevice(p->device);
      st = host_pipe_release(p, subs);
      if (table_ring_release(p) != FA_LP_OK) st = FA_LP_ERR_CUDA;
      if (p->sp_buf &&
          (cudaDeviceSynchronize() != cudaSuccess || cudaFree(p->sp_buf) != cudaSuccess)) {
        cudaGetLastError();
        st = FA_LP_ERR_CUDA;
      }
      if (p->dmeta &&
          (cudaDeviceSynchronize() != cudaSuccess || cudaFree(p->dmeta) != cudaSuccess)) {
        cudaGetLastError();
        st = FA_LP_ERR_CUDA;
      }
      if (cur >= 0 && cur != p->device) cudaSetDevice(cur);
    }
    delete p;
  }
  // the sub-plans of the host pipeline are plans of the cache like any other (never p itself)
  for (fa_lp_plan* sp : subs)
    if (sp && sp != p) fa_lp_plan_destroy(sp);
  return st;
}

int fa_lp_plan_info(const fa_lp_plan* p, int64_t* padded_tokens, int64_t* work_items,
                    size_t* workspace_bytes) {
  if (!p) return FA_LP_ERR_INVALID_ARG;
  if (padded_tokens) *padded_tokens = p->tpad;
  if (work_items) *work_items = int64_t(p->work.size());
  if (workspace_bytes) *workspace_bytes = p->ws.total;
  return FA_LP_OK;
}

int fa_lp_workspace_bytes(const fa_lp_plan* p, size_t* bytes) {
  if (!p || !bytes) return FA_LP_ERR_INVALID_ARG;
  *bytes = p->ws.total;
  return FA_LP_OK;
}

int fa_lp_plan_row_offsets(const fa_lp_plan* p, int64_t* row_offsets) {
  if (!p || !row_offsets) return FA_LP_ERR_INVALID_ARG;
  std::copy(p->row_off.begin(), p->row_off.end(), row_offsets);
  return FA_LP_OK;
}

int fa_lp_plan_set_wait_limit(fa_lp_plan* p, int64_t spins) {
  if (!p || spins < 1) return FA_LP_ERR_INVALID_ARG;
  p->spin_limit = spins;
  return FA_LP_OK;
}

int fa_lp_plan_set_table_limit(fa_lp_plan* p, size_t bytes) {
  if (!p) return FA_LP_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  if (falp::is_fp8(*p) || bytes == p->tbl_limit) return FA_LP_OK;
  if (p->dmeta) {  // the device copy of the work list is rebuilt on next use
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != p->device) cudaSetDevice(p->device);
    const bool ok = cudaDeviceSynchronize() == cudaSuccess && cudaFree(p->dmeta) == cudaSuccess;
    if (cur >= 0 && cur != p->device) cudaSetDevice(cur);
    p->dmeta = nullptr;
    if (!ok) {
      cudaGetLastError();
      return FA_LP_ERR_CUDA;
    }
  }
  p->tbl_limit = bytes;
  layout_work_and_workspace(p);
  p->quantized = false;
  return FA_LP_OK;
}

int fa_lp_plan_table_layout(const fa_lp_plan* p, int* heads_per_slot, int* slots,
                            size_t* slot_bytes) {
  if (!p) return FA_LP_ERR_INVALID_ARG;
  const bool fp8 = falp::is_fp8(*p);
  if (heads_per_slot) *heads_per_slot = fp8 ? 0 : p->tbl_hg;
  if (slots) *slots = fp8 ? 0 : p->tbl_slots;
  if (slot_bytes) *slot_bytes = fp8 ? 0 : p->tbl_slot_floats * 4;
  return FA_LP_OK;
}

int fa_lp_quantize(fa_lp_plan* p, const void* q, int64_t qst, int64_t qsh, const void* k,
                   int64_t kst, int64_t ksh, const void* v, int64_t vst, int64_t vsh,
                   void* stream_) {
  if (!p) return FA_LP_ERR_INVALID_ARG;
  if (p->tokens > 0 && (bad_view(q, qst, qsh) || bad_view(k, kst, ksh) || bad_view(v, vst, vsh)))
    return FA_LP_ERR_INVALID_ARG;
  int st = check_current_device(p);
  if (st != FA_LP_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if ((st = ensure_device_meta(p, stream)) != FA_LP_OK) return st;
  void* base = nullptr;
  if ((st = falp::workspace_acquire(p->device, p->ws.total, stream, &base)) != FA_LP_OK) return st;
  if (p->tokens > 0) {
    st = falp::is_fp8(*p)
             ? falp::launch_fp8_quantize(*p, static_cast<uint8_t*>(base), q, qst, qsh, k, kst, ksh,
                                         v, vst, vsh, stream)
             : falp::launch_nvfp4_quantize(*p, static_cast<uint8_t*>(base), q, qst, qsh, k, kst,
                                           ksh, v, vst, vsh, stream);
    if (st != FA_LP_OK) return st;
  }
  {
    std::lock_guard<std::mutex> lk(g_mu);
    DevWs& w = g_ws[p->device];
    w.owner = p;
    w.gen = ++g_quant_gen;
    p->quant_gen = w.gen;
  }
  p->quantized = true;
  return FA_LP_OK;
}

int fa_lp_forward_varlen_lse(fa_lp_plan* p, const int32_t* cu_seqlens_dev, void* out,
                             int64_t ost, int64_t osh, float* lse, int64_t lse_stride_head,
                             void* stream_) {
  (void)cu_seqlens_dev;
  if (!p) return FA_LP_ERR_INVALID_ARG;
  if (!p->quantized) return FA_LP_ERR_STATE;
  if (p->tokens > 0 && bad_view(out, ost, osh)) return FA_LP_ERR_INVALID_ARG;
  if (lse && p->tokens > 0 &&
      (lse_stride_head < p->tokens || reinterpret_cast<uintptr_t>(lse) % 4 != 0))
    return FA_LP_ERR_INVALID_ARG;
  int st = check_current_device(p);
  if (st != FA_LP_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = workspace_of_plan(p, &base)) != FA_LP_OK) return st;
  }
  if (p->work.empty()) return FA_LP_OK;
  uint8_t* ws = static_cast<uint8_t*>(base);
  if (falp::is_fp8(*p))
    return falp::launch_fp8_attention(*p, ws, out, ost, osh, lse, lse_stride_head, stream);
  if (p->tbl_slots == 2)
    return nvfp4_ring_forward(p, ws, out, ost, osh, lse, lse_stride_head, stream);
  return falp::launch_nvfp4_attention(*p, ws, 0, out, ost, osh, lse, lse_stride_head, stream);
}

int fa_lp_forward_varlen(fa_lp_plan* p, const int32_t* cu_seqlens_dev, void* out, int64_t ost,
                         int64_t osh, void* stream_) {
  return fa_lp_forward_varlen_lse(p, cu_seqlens_dev, out, ost, osh, nullptr, 0, stream_);
}

int fa_lp_sparse_query_blocks(const fa_lp_plan* p, int64_t* num_query_blocks) {
  if (!p || !num_query_blocks) return FA_LP_ERR_INVALID_ARG;
  *num_query_blocks = p->sp_G;
  return FA_LP_OK;
}

int fa_lp_forward_sparse(fa_lp_plan* p, const int32_t* cu_seqlens_dev,
                         const int32_t* block_offsets, const int32_t* block_indices,
                         int64_t num_indices, void* out, int64_t ost, int64_t osh, float* lse,
                         int64_t lse_stride_head, void* stream_) {
  (void)cu_seqlens_dev;
  if (!p) return FA_LP_ERR_INVALID_ARG;
  if (!falp::is_fp8(*p)) return FA_LP_ERR_UNSUPPORTED;
  if (!p->quantized) return FA_LP_ERR_STATE;
  if (p->tokens > 0 && bad_view(out, ost, osh)) return FA_LP_ERR_INVALID_ARG;
  if (num_indices < 0 || (p->tokens > 0 && !block_offsets) || (num_indices > 0 && !block_indices))
    return FA_LP_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(block_offsets) % 4 != 0 ||
      reinterpret_cast<uintptr_t>(block_indices) % 4 != 0)
    return FA_LP_ERR_INVALID_ARG;
  if (lse && p->tokens > 0 &&
      (lse_stride_head < p->tokens || reinterpret_cast<uintptr_t>(lse) % 4 != 0))
    return FA_LP_ERR_INVALID_ARG;
  // the list merge keeps two key-block bitmaps of the longest segment in 48 KB of shared memory
  if (size_t(p->sp_nw_max) * 8 > 48 * 1024) return FA_LP_ERR_UNSUPPORTED;
  int st = check_current_device(p);
  if (st != FA_LP_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = workspace_of_plan(p, &base)) != FA_LP_OK) return st;
    // per-plan scratch: merged lists (as many entries as the lists) + tile tables; grow-only,
    // stream-ordered
    const size_t nb = p->blocks.size(), H = size_t(p->heads);
    const size_t tables = align_up(size_t(std::max<int64_t>(num_indices, 1)) * 4, 256);
    const size_t need = tables + H * nb * (8 + 4 + 4);
    if (p->sp_bytes < need) {
      if (p->sp_buf && cudaFreeAsync(p->sp_buf, stream) != cudaSuccess) {
        cudaGetLastError();
        return FA_LP_ERR_CUDA;
      }
      p->sp_buf = nullptr;
      p->sp_bytes = 0;
      if (cudaMallocAsync(&p->sp_buf, need, stream) != cudaSuccess) {
        cudaGetLastError();
        p->sp_buf = nullptr;
        return FA_LP_ERR_OOM;
      }
      p->sp_bytes = need;
    }
    p->sp_tables = align_up(size_t(std::max<int64_t>(num_indices, 1)) * 4, 256);
  }
  if (p->sp_ctas.empty()) return FA_LP_OK;
  return falp::launch_fp8_sparse(*p, static_cast<uint8_t*>(base), block_offsets, block_indices,
                                 num_indices, out, ost, osh, lse, lse_stride_head, stream);
}

int fa_lp_attention(fa_lp_plan* p, const void* q, int64_t qst, int64_t qsh, const void* k,
                    int64_t kst, int64_t ksh, const void* v, int64_t vst, int64_t vsh,
                    const int32_t* cu_seqlens_dev, void* out, int64_t ost, int64_t osh,
                    void* stream) {
  const int st = fa_lp_quantize(p, q, qst, qsh, k, kst, ksh, v, vst, vsh, stream);
  if (st != FA_LP_OK) return st;
  return fa_lp_forward_varlen(p, cu_seqlens_dev, out, ost, osh, stream);
}

}  // extern "C"

namespace {

// Block lists of the block-sparse host entry (host arrays), or none for the dense forward.
struct HostLists {
  const int32_t* off;
  const int32_t* idx;
  int64_t n_idx;
};

int host_pipeline(fa_lp_plan* p, const void* q, int64_t qst, int64_t qsh, const void* k,
                  int64_t kst, int64_t ksh, const void* v, int64_t vst, int64_t vsh, void* out,
                  int64_t ost, int64_t osh, int heads_per_chunk, void* stream_,
                  const HostLists* lists) {
  if (!p) return FA_LP_ERR_INVALID_ARG;
  if (heads_per_chunk < 0 || heads_per_chunk > p->heads) return FA_LP_ERR_INVALID_ARG;
  if (p->tokens > 0 && (bad_view(q, qst, qsh) || bad_view(k, kst, ksh) || bad_view(v, vst, vsh) ||
                        bad_view(out, ost, osh)))
    return FA_LP_ERR_INVALID_ARG;
  int st = check_current_device(p);
  if (st != FA_LP_OK) return st;
  if (p->tokens == 0) return FA_LP_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const int H = p->heads;
  const int64_t T = p->tokens;
  falp::HostPipe& hp = p->host;
  const int key = 2 * heads_per_chunk + (lists ? 1 : 0);
  if (hp.key != key) {  // (re)build the pipeline for this chunking
    fa_lp_plan* old[4] = {nullptr, nullptr, nullptr, nullptr};
    st = host_pipe_release(p, old);
    for (fa_lp_plan* sp : old)
      if (sp) fa_lp_plan_destroy(sp);
    if (st != FA_LP_OK) return st;
    hp.sizes = host_schedule(*p, heads_per_chunk, lists != nullptr);
    hp.maxn = *std::max_element(hp.sizes.begin(), hp.sizes.end());
    const size_t bytes = size_t(8) * size_t(T) * size_t(hp.maxn) * FA_LP_HEAD_DIM * 2;
    if (cudaMalloc(&hp.buf, bytes) != cudaSuccess) {
      cudaGetLastError();
      hp.buf = nullptr;
      hp.sizes.clear();
      return FA_LP_ERR_OOM;
    }
    bool ok = cudaStreamCreateWithFlags(&hp.s_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.s_out, cudaStreamNonBlocking) == cudaSuccess;
    for (cudaEvent_t* e : {&hp.start, &hp.end, &hp.in_done[0], &hp.in_done[1], &hp.in_free[0],
                           &hp.in_free[1], &hp.out_ready[0], &hp.out_ready[1], &hp.out_free[0],
                           &hp.out_free[1]})
      ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    // chunks of fewer heads than the plan run on plans of their own (a chunk of all the heads
    // runs on this plan: a plan never holds itself)
    int nsub = 0;
    for (int n : hp.sizes) {
      if (!ok || n == H || std::find(hp.sub_n, hp.sub_n + nsub, n) != hp.sub_n + nsub) continue;
      if (nsub == 4) { ok = false; break; }
      ok = fa_lp_plan_create(T, n, p->cu.data(), p->nseg, p->scale, p->mode, p->device,
                             &hp.sub[nsub]) == FA_LP_OK;
      ok = ok && hp.sub[nsub] != p;
      hp.sub_n[nsub++] = n;
    }
    hp.key = key;
    if (!ok) {
      cudaGetLastError();
      host_pipe_release(p, old);
      for (fa_lp_plan* sp : old)
        if (sp) fa_lp_plan_destroy(sp);
      return FA_LP_ERR_CUDA;
    }
  }
  for (fa_lp_plan* sp : hp.sub) {
    if (!sp) continue;
    sp->spin_limit = p->spin_limit;
    // the chunk plans hold the NVFP4 table under the caller's limit (a no-op when unchanged)
    if ((st = fa_lp_plan_set_table_limit(sp, p->tbl_limit)) != FA_LP_OK) return st;
  }
  const size_t tb = size_t(T) * size_t(hp.maxn) * FA_LP_HEAD_DIM * 2;  // one tensor of one slot
  uint8_t* base = static_cast<uint8_t*>(hp.buf);
  auto dev = [&](int slot, int which) { return base + (size_t(slot) * 4 + which) * tb; };
  auto ok_ = [](cudaError_t e) { return e == cudaSuccess; };
  auto plan_of = [&](int n) -> fa_lp_plan* {
    if (n == H) return p;
    for (int i = 0; i < 4; ++i)
      if (hp.sub_n[i] == n) return hp.sub[i];
    return nullptr;
  };
  // the copies start after the work already on `stream` (which may still use the slots)
  if (!ok_(cudaEventRecord(hp.start, stream)) || !ok_(cudaStreamWaitEvent(hp.s_in, hp.start, 0)) ||
      !ok_(cudaStreamWaitEvent(hp.s_out, hp.start, 0))) {
    cudaGetLastError();
    return FA_LP_ERR_CUDA;
  }
  // block lists: one copy ahead of the first chunk's inputs on the copy-in stream (so every
  // chunk's in_done event covers it); chunk [h0, h0 + n) reads offsets from h0 G on
  const int32_t* d_off = nullptr;
  const int32_t* d_idx = nullptr;
  if (lists) {
    const size_t n_off = size_t(H) * size_t(p->sp_G) + 1;
    const size_t need = (n_off + size_t(std::max<int64_t>(lists->n_idx, 1))) * sizeof(int32_t);
    if (hp.lists_bytes < need) {
      if (hp.lists && cudaFree(hp.lists) != cudaSuccess) {
        cudaGetLastError();
        return FA_LP_ERR_CUDA;
      }
      hp.lists = nullptr;
      hp.lists_bytes = 0;
      if (cudaMalloc(&hp.lists, need) != cudaSuccess) {
        cudaGetLastError();
        hp.lists = nullptr;
        return FA_LP_ERR_OOM;
      }
      hp.lists_bytes = need;
    }
    int32_t* lo = static_cast<int32_t*>(hp.lists);
    if (!ok_(cudaMemcpyAsync(lo, lists->off, n_off * sizeof(int32_t), cudaMemcpyHostToDevice,
                             hp.s_in)) ||
        (lists->n_idx > 0 &&
         !ok_(cudaMemcpyAsync(lo + n_off, lists->idx, size_t(lists->n_idx) * sizeof(int32_t),
                              cudaMemcpyHostToDevice, hp.s_in)))) {
      cudaGetLastError();
      return FA_LP_ERR_CUDA;
    }
    d_off = lo;
    d_idx = lo + n_off;
  }
  const int nchunks = int(hp.sizes.size());
  for (int c = 0, h0 = 0; c < nchunks; h0 += hp.sizes[c], ++c) {
    const int n = hp.sizes[c], slot = c & 1;
    fa_lp_plan* sp = plan_of(n);
    if (!sp) return FA_LP_ERR_CUDA;
    const int64_t dst = int64_t(n) * FA_LP_HEAD_DIM, dsh = FA_LP_HEAD_DIM;  // dense [T, n, 128]
    const uint8_t* hq = static_cast<const uint8_t*>(q) + size_t(h0) * qsh * 2;
    const uint8_t* hk = static_cast<const uint8_t*>(k) + size_t(h0) * ksh * 2;
    const uint8_t* hv = static_cast<const uint8_t*>(v) + size_t(h0) * vsh * 2;
    uint8_t* ho = static_cast<uint8_t*>(out) + size_t(h0) * osh * 2;
    // copy-in of chunk c once the quantize of chunk c - 2 has consumed the slot
    const bool gather = c == 0;
    bool good = (c < 2 || ok_(cudaStreamWaitEvent(hp.s_in, hp.in_free[slot], 0))) &&
                ok_(copy_in(dev(slot, 0), hq, qst, qsh, T, n, gather, hp.s_in)) &&
                ok_(copy_in(dev(slot, 1), hk, kst, ksh, T, n, gather, hp.s_in)) &&
                ok_(copy_in(dev(slot, 2), hv, vst, vsh, T, n, gather, hp.s_in)) &&
                ok_(cudaEventRecord(hp.in_done[slot], hp.s_in)) &&
                ok_(cudaStreamWaitEvent(stream, hp.in_done[slot], 0));
    if (!good) {
      cudaGetLastError();
      return FA_LP_ERR_CUDA;
    }
    // quantize and attention of chunk c on the caller's stream
    st = fa_lp_quantize(sp, dev(slot, 0), dst, dsh, dev(slot, 1), dst, dsh, dev(slot, 2), dst, dsh,
                        stream);
    if (st != FA_LP_OK) return st;
    good = ok_(cudaEventRecord(hp.in_free[slot], stream)) &&
           (c < 2 || ok_(cudaStreamWaitEvent(stream, hp.out_free[slot], 0)));
    if (!good) {
      cudaGetLastError();
      return FA_LP_ERR_CUDA;
    }
    st = lists ? fa_lp_forward_sparse(sp, nullptr, d_off + int64_t(h0) * p->sp_G, d_idx,
                                      lists->n_idx, dev(slot, 3), dst, dsh, nullptr, 0, stream)
               : fa_lp_forward_varlen(sp, nullptr, dev(slot, 3), dst, dsh, stream);
    if (st != FA_LP_OK) return st;
    // copy-out of chunk c
    good = ok_(cudaEventRecord(hp.out_ready[slot], stream)) &&
           ok_(cudaStreamWaitEvent(hp.s_out, hp.out_ready[slot], 0)) &&
           ok_(copy_heads(ho, ost, osh, dev(slot, 3), dst, dsh, T, n, cudaMemcpyDeviceToHost,
                          hp.s_out)) &&
           ok_(cudaEventRecord(hp.out_free[slot], hp.s_out));
    if (!good) {
      cudaGetLastError();
      return FA_LP_ERR_CUDA;
    }
  }
  // `stream` completes only after the last copy-out
  if (!ok_(cudaEventRecord(hp.end, hp.s_out)) || !ok_(cudaStreamWaitEvent(stream, hp.end, 0))) {
    cudaGetLastError();
    return FA_LP_ERR_CUDA;
  }
  return FA_LP_OK;
}

}  // namespace

extern "C" {

int fa_lp_attention_host(fa_lp_plan* p, const void* q, int64_t qst, int64_t qsh, const void* k,
                         int64_t kst, int64_t ksh, const void* v, int64_t vst, int64_t vsh,
                         void* out, int64_t ost, int64_t osh, int heads_per_chunk,
                         void* stream) {
  return host_pipeline(p, q, qst, qsh, k, kst, ksh, v, vst, vsh, out, ost, osh, heads_per_chunk,
                       stream, nullptr);
}

int fa_lp_attention_sparse_host(fa_lp_plan* p, const void* q, int64_t qst, int64_t qsh,
                                const void* k, int64_t kst, int64_t ksh, const void* v,
                                int64_t vst, int64_t vsh, const int32_t* block_offsets,
                                const int32_t* block_indices, int64_t num_indices, void* out,
                                int64_t ost, int64_t osh, int heads_per_chunk, void* stream) {
  if (!p) return FA_LP_ERR_INVALID_ARG;
  if (!falp::is_fp8(*p)) return FA_LP_ERR_UNSUPPORTED;
  if (num_indices < 0 || (p->tokens > 0 && !block_offsets) || (num_indices > 0 && !block_indices))
    return FA_LP_ERR_INVALID_ARG;
  const HostLists lists{block_offsets, block_indices, num_indices};
  return host_pipeline(p, q, qst, qsh, k, kst, ksh, v, vst, vsh, out, ost, osh, heads_per_chunk,
                       stream, &lists);
}

int fa_lp_get_quantized(const fa_lp_plan* p, int which, fa_lp_array_desc* d) {
  if (!p || !d) return FA_LP_ERR_INVALID_ARG;
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_ws.find(p->device);
    if (it == g_ws.end() || !it->second.ptr || it->second.bytes < p->ws.total)
      return FA_LP_ERR_STATE;
    base = it->second.ptr;
  }
  const uint8_t* b = static_cast<const uint8_t*>(base);
  const int64_t H = p->heads, Tp = p->tpad;
  std::memset(d, 0, sizeof(*d));
  auto set = [&](size_t off, int64_t d0, int64_t d1, int64_t d2, int eb) {
    d->data = b + off;
    d->dims[0] = d0; d->dims[1] = d1; d->dims[2] = d2;
    d->strides[2] = eb;
    d->strides[1] = d2 * eb;
    d->strides[0] = d1 * d2 * eb;
    d->elem_bytes = eb;
    return FA_LP_OK;
  };
  if (falp::is_fp8(*p)) {
    switch (which) {
      case FA_LP_Q_CODES: return set(p->ws.q_codes, H, Tp, 128, 1);
      case FA_LP_K_CODES: return set(p->ws.k_codes, H, Tp, 128, 1);
      case FA_LP_V_CODES: return set(p->ws.v_codes, H, 128, Tp, 1);
      case FA_LP_DESCALE:
        return p->mode == FA_LP_MODE_FP8_SEGMENT ? set(p->ws.descale, 3, p->nseg, H, 4)
                                                 : set(p->ws.descale, 1, 3, H, 4);
      default: return FA_LP_ERR_INVALID_ARG;
    }
  }
  switch (which) {
    case FA_LP_Q_CODES: return set(p->ws.q_codes, H, Tp, 64, 1);
    case FA_LP_K_CODES: return set(p->ws.k_codes, H, Tp, 64, 1);
    case FA_LP_V_CODES: return set(p->ws.v_codes, H, 128, Tp / 2, 1);
    case FA_LP_Q_SCALES: return set(p->ws.q_sf, H, Tp, 8, 1);
    case FA_LP_K_SCALES: return set(p->ws.k_sf, H, Tp, 8, 1);
    case FA_LP_V_SCALES: return set(p->ws.v_sf, H, Tp / 128, 1024, 1);
    case FA_LP_Q_MEANS: return set(p->ws.q_mean, H, Tp / 128, 128, 4);
    case FA_LP_K_MEANS: return set(p->ws.k_mean, p->nseg, H, 128, 4);
    case FA_LP_Q_KM: return set(p->ws.q_km, 1, H, Tp, 4);
    case FA_LP_QMK_TABLE: {
      if (p->tbl_slots != 1) return FA_LP_ERR_UNSUPPORTED;  // built per head group in the forward
      int64_t n = 0;
      for (const auto& sg : p->segs) n += int64_t(H) * sg.nblk * sg.nblk * 128;
      return set(p->ws.qmk, 1, 1, n, 4);
    }
    default: return FA_LP_ERR_INVALID_ARG;
  }
}

int fa_lp_copy_quantized(const fa_lp_plan* p, int which, void* dst, size_t dst_bytes,
                         void* stream) {
  if (!p || !dst) return FA_LP_ERR_INVALID_ARG;
  fa_lp_array_desc d;
  const int st = fa_lp_get_quantized(p, which, &d);
  if (st != FA_LP_OK) return st;
  const size_t bytes = size_t(d.dims[0]) * size_t(d.dims[1]) * size_t(d.dims[2]) * d.elem_bytes;
  if (dst_bytes < bytes) return FA_LP_ERR_INVALID_ARG;
  return falp::cuda_status(cudaMemcpyAsync(dst, d.data, bytes, cudaMemcpyDeviceToDevice,
                                           static_cast<cudaStream_t>(stream)));
}

int fa_lp_get_last_error(fa_lp_plan* p, int* device_status) {
  if (!p || !device_status) return FA_LP_ERR_INVALID_ARG;
  *device_status = 0;
  int v = 0;
  if (p->dmeta) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != p->device) cudaSetDevice(p->device);
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&v, p->d_err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(p->d_err, 0, sizeof(int));
    if (cur >= 0 && cur != p->device) cudaSetDevice(cur);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return FA_LP_ERR_CUDA;
    }
  }
  // launches of the host-buffer entry point record their status in its sub-plans (plans of
  // fewer heads, so this recursion ends)
  for (fa_lp_plan* sp : p->host.sub) {
    if (!sp || sp == p) continue;
    int sv = 0;
    const int st = fa_lp_get_last_error(sp, &sv);
    if (st == FA_LP_ERR_CUDA) return st;
    if (v == 0) v = sv;
  }
  *device_status = v;
  if (v == 0) return FA_LP_OK;
  return (v & 0xF00) == 0x200 ? FA_LP_ERR_INVALID_ARG : FA_LP_ERR_DEVICE_TIMEOUT;
}

int fa_lp_release_workspace(int device, void* stream) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_ws.find(device);
  if (it == g_ws.end() || !it->second.ptr) return FA_LP_OK;
  const cudaError_t e = cudaFreeAsync(it->second.ptr, static_cast<cudaStream_t>(stream));
  it->second = DevWs{};
  for (auto& kv : g_plans)
    if (kv.second->device == device) kv.second->quantized = false;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FA_LP_ERR_CUDA;
  }
  return FA_LP_OK;
}

int fa_lp_encode(int format, const float* x, int64_t n, uint8_t* codes, void* stream) {
  if (n < 0 || (n > 0 && (!x || !codes)) || (format != 0 && format != 1))
    return FA_LP_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_LP_ERR_CUDA;
  const int st = check_device(dev);
  if (st != FA_LP_OK) return st;
  if (n == 0) return FA_LP_OK;
  return falp::launch_encode(format, x, n, codes, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
