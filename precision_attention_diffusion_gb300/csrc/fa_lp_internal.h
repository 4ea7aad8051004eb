// fa_lp_internal.h -- declarations shared by the translation units of libfa_lp.so (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <vector>

#include "fa_lp.h"  // include/ is on the include path

namespace falp {

constexpr int kD = FA_LP_HEAD_DIM;  // 128
constexpr int kTile = 128;          // rows of a query tile / keys of a key tile / padding quantum

// One segment of the packed batch, as the kernels see it.
struct SegInfo {
  int32_t tok0;     // first token of the segment in the packed input (cu_seqlens[s])
  int32_t len;      // L_s
  int32_t row0;     // first row of the segment on the padded token axis
  int32_t nblk;     // ceil(L_s / 128)
};

// 128-row block of the padded token axis (quantize passes).
struct BlockInfo {
  int32_t tok0;     // token of the block's first row, or -1 (never: every block has a segment)
  int32_t nvalid;   // rows of the block that hold tokens (the rest are zero padding)
  int32_t seg;      // segment index
  int32_t blk;      // block index inside its segment
};

// Attention work item: a pair of 128-row query tiles of one (segment, head).
struct WorkItem {
  int32_t seg;
  int32_t head;
  int32_t qt0;      // index of the first query tile inside the segment
  int32_t nq;       // 1 or 2 query tiles
};

// Block-sparse forward: a group of query tiles (one segment, up to 8 heads) whose CTAs run
// together; the tiles of a group are ordered by their merged-list length on the device and taken
// two per CTA.
struct SparseGroup {
  int32_t slot0;    // first slot of the group in the tile order
  int32_t h0, nh;   // heads [h0, h0 + nh)
  int32_t seg;
};
struct SparseCta {
  int32_t slot;     // first of this CTA's slots
  int32_t count;    // 1 or 2 tiles
};

// Tile of the NVFP4 qm K^T table: (segment, 128-block M tile, 256-key N tile).
struct QmkItem {
  int32_t seg;
  int32_t mt;       // 128-block M tile
  int32_t nt;       // first 256-key N tile
  int32_t ntiles;   // N tiles of this CTA
};
constexpr int kQmkTilesPer = 8;  // N tiles per table CTA (default; the plan picks per segment)

// Workspace layout of one plan (byte offsets from the workspace base, 1024-aligned).
struct WsLayout {
  size_t q_codes = 0, k_codes = 0, v_codes = 0;  // FP8: [H][Tp][128], [H][Tp][128], [H][128][Tp]
  size_t q_sf = 0, k_sf = 0, v_sf = 0;           // NVFP4 scale bytes
  size_t q_mean = 0, k_mean = 0;                 // NVFP4 means (f32)
  size_t k_chunk = 0;                            // NVFP4 scratch: f64 [nblk][H][128] chunk sums
  size_t q_km = 0;                               // NVFP4: f32 [H][Tp] q . km (row LSE term)
  size_t qmk = 0;                                // NVFP4: f32 qm K^T table (per segment)
  size_t amax = 0, descale = 0;                  // FP8: u32 / f32 [3][R][H], R = 1 or nseg
  size_t total = 0;
};

// State of the host-buffer entry point (fa_lp_attention_host): head-chunk pipeline.
struct HostPipe {
  int key = -1;                               // 2 heads_per_chunk + (block-sparse call) it was
                                              // built for
  std::vector<int> sizes;                     // heads of each chunk, in order
  int maxn = 0;                               // largest chunk
  fa_lp_plan* sub[4] = {nullptr, nullptr, nullptr, nullptr};  // plans of the chunk sizes
  int sub_n[4] = {0, 0, 0, 0};                // (fewer heads than the plan; a chunk of all
                                              // the heads runs on the plan itself)
  void* buf = nullptr;                        // 2 slots x {q, k, v, out} x tokens x maxn x 128 BF16
  void* lists = nullptr;                      // block-sparse entry: device copy of the lists
  size_t lists_bytes = 0;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t in_done[2] = {}, in_free[2] = {}, out_ready[2] = {}, out_free[2] = {};
};

}  // namespace falp

struct fa_lp_plan {
  // key
  int64_t tokens = 0;
  int heads = 0;
  int nseg = 0;
  float scale = 0.f;
  int mode = 0;
  int device = 0;
  std::vector<int32_t> cu;
  // derived
  int64_t tpad = 0;
  std::vector<int64_t> row_off;  // nseg + 1
  std::vector<falp::SegInfo> segs;
  std::vector<falp::BlockInfo> blocks;
  std::vector<falp::WorkItem> work;
  std::vector<falp::QmkItem> qmk_items;          // NVFP4 qm K^T table tiles
  std::vector<int64_t> c_off;                    // NVFP4: float offset of each segment's table
                                                 // inside a table slot
  // NVFP4 qm K^T table held per group of tbl_hg heads. tbl_slots == 1: one slot holds every
  // head's table (tbl_hg = heads), written by the quantize. tbl_slots == 2: a ring of two slots;
  // the forward builds group g's table into slot g % 2 right before group g's attention launch.
  // The work list is ordered by group; group g's items are [tbl_work_off[g], tbl_work_off[g+1]).
  int tbl_hg = 0;
  int tbl_slots = 1;
  size_t tbl_slot_floats = 0;
  size_t tbl_limit = 0;                          // bytes; 0 = the library default
  std::vector<int32_t> tbl_work_off;
  cudaStream_t tbl_stream[2] = {nullptr, nullptr};  // ring forward: one stream per slot
  cudaEvent_t tbl_fork = nullptr;
  cudaEvent_t tbl_join[2] = {nullptr, nullptr};
  falp::WsLayout ws;
  // block-sparse forward (FP8 plans): 64-row query blocks
  int64_t sp_G = 0;                   // query blocks over the packed batch
  std::vector<int32_t> sp_qb0;        // first query block of every segment
  int sp_nw_max = 0;                  // 32-bit words of the largest segment's key-block bitmap
  std::vector<falp::SparseGroup> sp_groups;
  std::vector<falp::SparseCta> sp_ctas;
  void* sp_buf = nullptr;             // merged lists (u32 [num_indices]) + tile tables
  size_t sp_bytes = 0, sp_tables = 0; // its size; byte offset of the tables (i64 base, i32 count,
                                      // i32 order, each [H][nb])
  int64_t spin_limit = 20000;  // parked probes of <= 100 us each: about 2 s per wait
  // device metadata (created on first use on the plan's device)
  void* dmeta = nullptr;
  falp::SegInfo* d_segs = nullptr;
  falp::BlockInfo* d_blocks = nullptr;
  falp::WorkItem* d_work = nullptr;
  falp::QmkItem* d_qmk = nullptr;
  int64_t* d_coff = nullptr;
  int32_t* d_sp_qb0 = nullptr;
  falp::SparseGroup* d_sp_groups = nullptr;
  falp::SparseCta* d_sp_ctas = nullptr;
  int* d_err = nullptr;  // [0]: sticky device status, [1]: abort word (launch generation)
  bool quantized = false;
  uint64_t quant_gen = 0;  // generation of this plan's last quantize (the workspace's owner tag)
  int refcount = 1;
  falp::HostPipe host;  // created by the first fa_lp_attention_host call
};

namespace falp {

// Per-device shared workspace (grow-only). Returns FA_LP_OK and the base pointer.
int workspace_acquire(int device, size_t bytes, cudaStream_t stream, void** base);

// Tensor-map encoder from the driver (resolved once through the runtime's entry-point query).
int encode_tmap_3d_u8(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
                      uint32_t box1, CUtensorMapSwizzle swz);

// Launchers (defined next to their kernels). All enqueue on `stream` and return a status.
int launch_fp8_quantize(const fa_lp_plan& p, uint8_t* ws, const void* q, int64_t qst,
                        int64_t qsh, const void* k, int64_t kst, int64_t ksh, const void* v,
                        int64_t vst, int64_t vsh, cudaStream_t stream);
int launch_fp8_attention(const fa_lp_plan& p, uint8_t* ws, void* out, int64_t ost, int64_t osh,
                         float* lse, int64_t lse_sh, cudaStream_t stream);
int launch_nvfp4_quantize(const fa_lp_plan& p, uint8_t* ws, const void* q, int64_t qst,
                          int64_t qsh, const void* k, int64_t kst, int64_t ksh, const void* v,
                          int64_t vst, int64_t vsh, cudaStream_t stream);
// NVFP4 attention over table group g's work items, reading the table from slot g % tbl_slots.
int launch_nvfp4_attention(const fa_lp_plan& p, uint8_t* ws, int g, void* out, int64_t ost,
                           int64_t osh, float* lse, int64_t lse_sh, cudaStream_t stream);
int launch_fp8_sparse(const fa_lp_plan& p, uint8_t* ws, const int32_t* block_offsets,
                      const int32_t* block_indices, int64_t num_indices, void* out, int64_t ost,
                      int64_t osh, float* lse, int64_t lse_sh, cudaStream_t stream);
// Dense [T][n][128] BF16 copy of n heads of a [T, H, 128] view (element strides st, sh) whose
// memory the device can read (`src_dev`: page-locked host memory through its device mapping).
int launch_gather_heads(void* dst, const void* src_dev, int64_t src_st, int64_t src_sh,
                        int64_t T, int n, cudaStream_t stream);
// The qm K^T table of table group g's heads into slot g % tbl_slots.
int launch_nvfp4_qmk(const fa_lp_plan& p, uint8_t* ws, int g, cudaStream_t stream);
int launch_encode(int format, const float* x, int64_t n, uint8_t* codes, cudaStream_t stream);

// Distinct positive id per kernel launch (device-side abort words compare against it).
int next_launch_generation();

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? FA_LP_OK : FA_LP_ERR_CUDA; }

// FP8 plans: one scale per (tensor, head), or per (segment, tensor, head).
inline bool is_fp8(const fa_lp_plan& p) {
  return p.mode == FA_LP_MODE_FP8 || p.mode == FA_LP_MODE_FP8_SEGMENT;
}
// Rows of the FP8 amax / descale arrays per tensor: 1, or the number of segments.
inline int fp8_scale_rows(const fa_lp_plan& p) {
  return p.mode == FA_LP_MODE_FP8_SEGMENT ? p.nseg : 1;
}

// Raise a kernel's dynamic shared-memory limit on `device` once (the attribute belongs to the
// device's context, so every device is set up on its own first launch). `done` holds one bit per
// device; safe to call from several host threads (a repeated set is harmless).
inline int set_smem_limit_once(const void* kernel, int bytes, int device,
                               std::atomic<uint64_t>& done) {
  const uint64_t bit = (device >= 0 && device < 64) ? (uint64_t(1) << device) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return FA_LP_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess) {
    cudaGetLastError();
    return FA_LP_ERR_CUDA;
  }
  done.fetch_or(bit, std::memory_order_acq_rel);
  return FA_LP_OK;
}

}  // namespace falp
