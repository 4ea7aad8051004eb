// noalloc.cu -- FP8 descales without any allocation by the library.
//
// Some callers cannot let a library call cudaMalloc: programs that hand all device memory to
// their own pool or allocator up front, deployments that fix their memory footprint at start-up
// and forbid later growth, and latency-critical loops where cudaMalloc's implicit device
// synchronization and unpredictable cost are not acceptable. fa_lp_fp8_descale_noalloc serves
// them: it runs the per-(tensor, head) amax pass of the FP8 quantizer with its scratch in a fixed
// file-scope device array instead of the plan workspace, and writes the descales (amax / 448, 1
// when amax is 0) to a buffer the caller owns.
//
// The scratch array holds 3 * kMaxHeadsNoAlloc words (12 KB). Every GPU that loads this library
// keeps it until the process exits. All calls on a device share it and each call clears it first:
// calls must be ordered on the GPU (one stream, or streams the caller synchronizes); calls that
// overlap on the GPU race on it. The first call on each device looks up the array's device
// address (cudaGetSymbolAddress, with that device current) and caches it for that device's CUDA
// context; make that first call before any stream capture begins (and, after cudaDeviceReset,
// the first call in the new context likewise).
#include "fa_lp_internal.h"

#include <mutex>

namespace falp {
namespace {

constexpr int kMaxHeadsNoAlloc = 1024;
constexpr int kNoAllocTok = 256;  // tokens per block of the amax pass

static __device__ __align__(256) uint32_t g_amax_scratch[3 * kMaxHeadsNoAlloc];

// Address of g_amax_scratch on each device, taken with that device current and kept together
// with the id of the CUDA context it belongs to: a context destroyed and re-created (after
// cudaDeviceReset) loads the module again, possibly at another address, so a new context id
// means a new lookup.
std::mutex g_sym_mu;
uint32_t* g_sym_addr[64] = {};
unsigned long long g_sym_ctx[64] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Id of the current context (0 when it cannot be read: the address is then looked up every call).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
    cudaGetLastError();
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

int scratch_address(int device, uint32_t** out) {
  if (device < 0 || device >= 64) return FA_LP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_sym_mu);
  const unsigned long long ctx = current_context_id();
  if (!g_sym_addr[device] || ctx == 0 || ctx != g_sym_ctx[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_amax_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      g_sym_addr[device] = nullptr;
      return FA_LP_ERR_CUDA;
    }
    g_sym_addr[device] = static_cast<uint32_t*>(p);
    g_sym_ctx[device] = ctx;
  }
  *out = g_sym_addr[device];
  return FA_LP_OK;
}

__global__ void noalloc_clear_kernel(uint32_t* scratch, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) scratch[i] = 0u;
}

// Per (tensor, head) max |x| as the bit pattern of a non-negative float (integer order equals
// float order there, so atomicMax is exact and independent of the order of blocks).
__global__ void __launch_bounds__(256) noalloc_amax_kernel(
    const uint16_t* __restrict__ q, int64_t qst, int64_t qsh, const uint16_t* __restrict__ k,
    int64_t kst, int64_t ksh, const uint16_t* __restrict__ v, int64_t vst, int64_t vsh,
    int64_t T, int H, uint32_t* __restrict__ scratch) {
  const int z = blockIdx.z, h = blockIdx.y;
  const uint16_t* x = z == 0 ? q : (z == 1 ? k : v);
  const int64_t st = z == 0 ? qst : (z == 1 ? kst : vst);
  const int64_t sh = z == 0 ? qsh : (z == 1 ? ksh : vsh);
  const int64_t t0 = int64_t(blockIdx.x) * kNoAllocTok;
  const int64_t t1 = min(T, t0 + kNoAllocTok);
  const int sub = threadIdx.x & 15;
  uint32_t m = 0;
  for (int64_t t = t0 + (threadIdx.x >> 4); t < t1; t += 16) {
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
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t r = red[0];
    for (int i = 1; i < 8; ++i) r = max(r, red[i]);
    atomicMax(scratch + z * H + h, r << 16);
  }
}

__global__ void noalloc_descale_kernel(const uint32_t* __restrict__ scratch, int n,
                                       float* __restrict__ descale) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float a = __uint_as_float(scratch[i]);
  descale[i] = a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
}

bool bad_view(const void* ptr, int64_t st, int64_t sh) {
  return !ptr || st <= 0 || sh <= 0 || reinterpret_cast<uintptr_t>(ptr) % 16 != 0 ||
         st % 8 != 0 || sh % 8 != 0;
}

}  // namespace
}  // namespace falp

extern "C" int fa_lp_fp8_descale_noalloc(const void* q, int64_t q_stride_tok,
                                         int64_t q_stride_head, const void* k,
                                         int64_t k_stride_tok, int64_t k_stride_head,
                                         const void* v, int64_t v_stride_tok,
                                         int64_t v_stride_head, int64_t tokens, int heads,
                                         float* descale, void* stream_) {
  using namespace falp;
  if (heads < 1 || heads > kMaxHeadsNoAlloc || tokens < 0 || !descale ||
      reinterpret_cast<uintptr_t>(descale) % 4 != 0)
    return FA_LP_ERR_INVALID_ARG;
  if (tokens > 0 && (bad_view(q, q_stride_tok, q_stride_head) ||
                     bad_view(k, k_stride_tok, k_stride_head) ||
                     bad_view(v, v_stride_tok, v_stride_head)))
    return FA_LP_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_LP_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return FA_LP_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return FA_LP_ERR_UNSUPPORTED;
  uint32_t* scratch = nullptr;
  int st = scratch_address(dev, &scratch);
  if (st != FA_LP_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const int n = 3 * heads;
  noalloc_clear_kernel<<<(n + 255) / 256, 256, 0, stream>>>(scratch, n);
  if (tokens > 0) {
    dim3 grid(unsigned((tokens + kNoAllocTok - 1) / kNoAllocTok), unsigned(heads), 3);
    noalloc_amax_kernel<<<grid, 256, 0, stream>>>(
        static_cast<const uint16_t*>(q), q_stride_tok, q_stride_head,
        static_cast<const uint16_t*>(k), k_stride_tok, k_stride_head,
        static_cast<const uint16_t*>(v), v_stride_tok, v_stride_head, tokens, heads, scratch);
  }
  noalloc_descale_kernel<<<(n + 255) / 256, 256, 0, stream>>>(scratch, n, descale);
  return cuda_status(cudaGetLastError());
}
