// FP8 (E4M3) rows for the low-precision indexer.  "DeepSeek V4 technical
// review", section 5: the indexer's QK product runs in low precision.  Each
// row (one compressed indexer key, or one indexer query head) is stored as
// E4M3 codes with one power-of-two scale 2^e, e the smallest integer with
// max|row| <= 448 * 2^e (clamped to [-126, 127]; an all-zero row gets e = 0):
// the division by the scale is exact and the rounding to the code (nearest,
// ties to even) is the only inexact step.
#include "common.cuh"
#include "kernels.h"

namespace csa {

namespace {

constexpr int kRowsPerBlock = 8;  // one warp per row

// Two fp32 values -> two E4M3 codes (round to nearest even, saturating):
// ``lo`` goes to the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// 2^e as fp32 bits, for a normal exponent e in [-126, 127]
__device__ __forceinline__ float pow2(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }

// The scale exponent of a row whose largest magnitude is amax (exact in fp32):
// e = lead - 8 where 2^lead is amax's leading bit, plus one when amax exceeds
// 448 * 2^(lead - 8) = 1.75 * 2^lead; at least -126 (then at most 120).
__device__ __forceinline__ int row_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  const uint32_t u = __float_as_uint(amax);
  const int field = static_cast<int>((u >> 23) & 0xFFu);
  // exponent of the leading bit (subnormal amax: from the highest mantissa bit)
  const int lead = field ? field - 127 : (31 - __clz(static_cast<int>(u & 0x7FFFFFu))) - 149;
  int e = lead - 8 < -126 ? -126 : lead - 8;
  const float limit = __uint_as_float((static_cast<uint32_t>(e + 8 + 127) << 23) | 0x600000u);  // 448 * 2^e
  if (amax > limit) ++e;
  return e;
}

// V values of a D = 32 V row per lane.
template <int V>
__global__ void __launch_bounds__(32 * kRowsPerBlock) quantize_kernel(const __nv_bfloat16* __restrict__ x,
                                                                     uint8_t* __restrict__ codes,
                                                                     float* __restrict__ scales, long long rows) {
  pdl_wait_then_release();
  constexpr int D = 32 * V;
  const int lane = threadIdx.x & 31;
  const long long r = static_cast<long long>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  if (r >= rows) return;
  // lane owns the V consecutive elements [lane * V, lane * V + V)
  float v[V];
  const uint16_t* src = reinterpret_cast<const uint16_t*>(x) + r * D + lane * V;
#pragma unroll
  for (int i = 0; i < V; ++i) v[i] = __uint_as_float(static_cast<uint32_t>(src[i]) << 16);
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e = row_exponent(amax);
  const float inv = pow2(-e);  // exact: -e in [-120, 126]
  uint8_t* dst = codes + r * D + lane * V;
  if constexpr (V == 1) {
    dst[0] = static_cast<uint8_t>(cvt_e4m3x2(v[0] * inv, 0.f) & 0xFFu);
  } else {
#pragma unroll
    for (int i = 0; i < V; i += 2) {
      const uint32_t c = cvt_e4m3x2(v[i] * inv, v[i + 1] * inv);
      *reinterpret_cast<uint16_t*>(dst + i) = static_cast<uint16_t>(c);
    }
  }
  if (lane == 0) scales[r] = pow2(e);
}

}  // namespace

cudaError_t launch_quantize_fp8(const void* x, long long rows, int D, void* codes, float* scales,
                                cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  if (blocks > 0x7fffffffLL) return cudaErrorNotSupported;
  const dim3 grid(static_cast<unsigned>(blocks)), block(32 * kRowsPerBlock);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  uint8_t* cb = static_cast<uint8_t*>(codes);
  switch (D) {
    case 32: return launch_k(quantize_kernel<1>, grid, block, 0, s, 1, xb, cb, scales, rows);
    case 64: return launch_k(quantize_kernel<2>, grid, block, 0, s, 1, xb, cb, scales, rows);
    case 128: return launch_k(quantize_kernel<4>, grid, block, 0, s, 1, xb, cb, scales, rows);
    case 256: return launch_k(quantize_kernel<8>, grid, block, 0, s, 1, xb, cb, scales, rows);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace csa
