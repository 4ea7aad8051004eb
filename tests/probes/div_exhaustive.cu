// Exhaustive check of the NVFP4 quantizer's division (div_rn in quant_nvfp4.cu, included here so
// that the product's own function is tested) against IEEE division (__fdiv_rn): every positive
// E4M3 divisor d, every f32 dividend x whose quotient lies in [2^-3, 16) (both signs), plus
// 2^32 random dividends over [2^-40, 2^10) d. Compares the quotient bits and the E2M1 codes.
// Prints one line: "cases <n> quotient_mismatches <a> code_mismatches <b> zero_sign <ok>".
#include <cstdio>

#include "../../precision_attention_diffusion_gb300/csrc/quant_nvfp4.cu"

// the included file's quantize launcher refers to the table pass; this program never calls it
int falp::launch_nvfp4_qmk(const fa_lp_plan&, uint8_t*, int, cudaStream_t) { return FA_LP_OK; }

namespace falp {
namespace {
__device__ unsigned long long g_bad_q, g_bad_c, g_n;

__global__ void k_exhaustive(int exp_lo, int exp_hi) {
  const int code = blockIdx.y + 1;  // E4M3 codes 1..126: every positive finite value
  const float d = e4m3_value(uint8_t(code));
  const float y = __frcp_rn(d);
  unsigned long long bq = 0, bc = 0, n = 0;
  const uint32_t total = uint32_t(exp_hi - exp_lo) << 23;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int e = exp_lo + int(i >> 23);
    const uint32_t xb = (__float_as_uint(ldexpf(d, e)) & 0xFF800000u) + (i & 0x7FFFFFu);
    for (int sgn = 0; sgn < 2; ++sgn) {
      const float x = __uint_as_float(xb | (sgn ? 0x80000000u : 0u));
      const float a = __fdiv_rn(x, d), b = div_rn(x, d, y);
      ++n;
      bq += __float_as_uint(a) != __float_as_uint(b);
      bc += cvt_e2m1x2(a, a) != cvt_e2m1x2(b, b);
    }
  }
  atomicAdd(&g_bad_q, bq);
  atomicAdd(&g_bad_c, bc);
  atomicAdd(&g_n, n);
}

__global__ void k_random(unsigned seed, int iters) {
  unsigned s = seed ^ (blockIdx.x * 747796405u + threadIdx.x * 2891336453u);
  unsigned long long bq = 0, bc = 0, n = 0;
  for (int it = 0; it < iters; ++it) {
    s = s * 1664525u + 1013904223u;
    const int code = 1 + int((s >> 8) % 126);
    s = s * 1664525u + 1013904223u;
    const int e = -40 + int((s >> 8) % 50);
    s = s * 1664525u + 1013904223u;
    const float d = e4m3_value(uint8_t(code)), y = __frcp_rn(d);
    const float x = ldexpf(__uint_as_float(0x3F800000u | (s >> 9)), e) * ((s & 1) ? -1.f : 1.f) * d;
    const float a = __fdiv_rn(x, d), b = div_rn(x, d, y);
    ++n;
    bq += __float_as_uint(a) != __float_as_uint(b);
    bc += cvt_e2m1x2(a, a) != cvt_e2m1x2(b, b);
  }
  atomicAdd(&g_bad_q, bq);
  atomicAdd(&g_bad_c, bc);
  atomicAdd(&g_n, n);
}

__global__ void k_zero(unsigned* out) {
  const float d = 1.5f, y = __frcp_rn(d);
  out[0] = __float_as_uint(div_rn(-0.f, d, y)) == __float_as_uint(__fdiv_rn(-0.f, d)) &&
           __float_as_uint(div_rn(0.f, d, y)) == __float_as_uint(__fdiv_rn(0.f, d));
}
}  // namespace
}  // namespace falp

int main() {
  using namespace falp;
  falp::k_exhaustive<<<dim3(1024, 126), 256>>>(-3, 4);
  falp::k_random<<<4096, 256>>>(12345u, 4096);
  unsigned* z = nullptr;
  cudaMalloc(&z, 4);
  falp::k_zero<<<1, 1>>>(z);
  const cudaError_t e = cudaDeviceSynchronize();
  unsigned long long bq = 0, bc = 0, n = 0;
  unsigned zs = 0;
  cudaMemcpyFromSymbol(&bq, falp::g_bad_q, 8);
  cudaMemcpyFromSymbol(&bc, falp::g_bad_c, 8);
  cudaMemcpyFromSymbol(&n, falp::g_n, 8);
  cudaMemcpy(&zs, z, 4, cudaMemcpyDeviceToHost);
  std::printf("cases %llu quotient_mismatches %llu code_mismatches %llu zero_sign %u status %s\n",
              n, bq, bc, zs, cudaGetErrorString(e));
  return e == cudaSuccess ? 0 : 1;
}
