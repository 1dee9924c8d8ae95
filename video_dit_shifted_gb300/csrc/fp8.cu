// wp_quantize_e4m3: bf16 rows -> e4m3 codes for wp_window_attn_fp8.
//
// code = e4m3(fp32(x) * inv_scale): the product is one fp32 multiply
// (round to nearest even), then rounded to the nearest e4m3 value (ties to
// even) and saturated to +-448 (the format's largest finite value).  The
// dequantised value is code * (1 / inv_scale).  HBM-bound: each thread moves
// 16 elements (32 bytes in, 16 bytes out) per chunk, six chunks at a time.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "wp_internal.h"

namespace wp {
namespace {

// Two fp32 values -> two e4m3 codes, lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  unsigned short d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// Thread t handles the 16-element chunks t, t + T, t + 2T, ... (T threads
// in the grid), kBatch of them at a time: every load of a batch is issued
// before the first chunk is converted, so a thread keeps kBatch * 32 bytes in
// flight.
constexpr int kBatch = 6;
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) quantize_e4m3_kernel(const uint8_t* __restrict__ src, int64_t src_stride,
                                                                 uint8_t* __restrict__ dst, int64_t dst_stride,
                                                                 int64_t rows, int chunks, float inv_scale) {
  const int64_t n = rows * chunks;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < n; i0 += step * kBatch) {
    uint4 a[kBatch], b[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t i = i0 + u * step;
      if (i < n) {
        const int64_t r = i / chunks;
        const int c = static_cast<int>(i - r * chunks);
        const uint4* s = reinterpret_cast<const uint4*>(src + r * src_stride + c * 32);
        a[u] = __ldcs(s);
        b[u] = __ldcs(s + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t i = i0 + u * step;
      if (i < n) {
        const int64_t r = i / chunks;
        const int c = static_cast<int>(i - r * chunks);
        const uint32_t w[8] = {a[u].x, a[u].y, a[u].z, a[u].w, b[u].x, b[u].y, b[u].z, b[u].w};
        uint32_t out[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t packed = 0;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t v = w[2 * q + h];  // two bf16: element 2k in the low half
            const float x0 = __uint_as_float(v << 16) * inv_scale;
            const float x1 = __uint_as_float(v & 0xffff0000u) * inv_scale;
            packed |= e4m3x2(x0, x1) << (16 * h);
          }
          out[q] = packed;
        }
        __stcs(reinterpret_cast<uint4*>(dst + r * dst_stride + c * 16), make_uint4(out[0], out[1], out[2], out[3]));
      }
    }
  }
}

}  // namespace
}  // namespace wp

using namespace wp;

extern "C" int wp_quantize_e4m3(const void* src, int64_t rows, int cols, int64_t src_row_stride_B, void* dst,
                                int64_t dst_row_stride_B, float inv_scale, void* stream) {
  if (!src || !dst) return fail(WP_EINVAL, "src or dst is NULL");
  if (rows < 0 || cols < 0) return fail(WP_EINVAL, "rows=%lld, cols=%d must be >= 0", (long long)rows, cols);
  if (!(inv_scale > 0.f) || !std::isfinite(inv_scale)) return fail(WP_EINVAL, "inv_scale must be finite and > 0");
  if (cols % 16 != 0) return fail(WP_EUNSUPPORTED, "cols=%d must be a multiple of 16", cols);
  if (!aligned16(src) || !aligned16(dst) || (src_row_stride_B & 15) || (dst_row_stride_B & 15) ||
      src_row_stride_B < 2LL * cols || dst_row_stride_B < cols)
    return fail(WP_EUNSUPPORTED, "pointers and row strides must be 16-byte aligned and hold a row");
  const int64_t n = rows * (cols / 16);
  if (n == 0) return ok();
  int dev = 0, sms = 0;
  if (int rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return rc;
  if (int rc = cuda_check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute"))
    return rc;
  // Two blocks per SM (80 registers a thread): fewer threads with more bytes
  // each measured faster than a full SM (6 chunks x 2 blocks: 97% of the copy
  // rate on 1.6 GB; 1 chunk x 8 blocks: 92%).
  const int64_t blocks = std::min<int64_t>((n + kThreads - 1) / kThreads, static_cast<int64_t>(sms) * 2);
  quantize_e4m3_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t*>(src), src_row_stride_B, static_cast<uint8_t*>(dst), dst_row_stride_B, rows,
      cols / 16, inv_scale);
  if (int rc = cuda_check(cudaGetLastError(), "quantize_e4m3_kernel launch")) return rc;
  return ok();
}
