// wp_permute: the regular <-> shifted (<-> canonical) re-layout of row data.
//
// "Window-Aligned Sequence Parallelism (SeedVR2)", §Motivation and §Plan A
// redistribution: when every row stays on one device, a layout boundary is a
// local permutation.  dst row q receives src row perm[q], where the plan's
// fused table perm[q] = pos_src[ids_dst[q]] was built on the host.
//
// The kernel is a pure HBM gather: every byte is read once and written once.
// One warp moves one row per iteration with 16-byte loads (read-only path)
// and stores, kChunks x 16 B per lane in flight before the stores: 12 for
// rows of up to 6 KB (a 5 KB hidden row in one batch), 8 for longer rows.
// The destination is walked in order, so writes stream; source rows arrive
// in runs of up to a window width of consecutive rows.  The grid is
// persistent with at most two 256-thread blocks per SM: measured on the
// sweep's rows, 16 warps per SM with 128-192 bytes in flight per lane beat
// 40 warps with 64 (5-7% more bandwidth, 96-100% of the measured copy
// rate on rows above 4x L2).
#include <cuda_runtime.h>

#include <algorithm>

#include "wp_internal.h"

namespace wp {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxBlocksPerSm = 2;

template <int kChunks>  // 16-byte chunks per lane per batch
__global__ void __launch_bounds__(kThreads)
permute_rows_kernel(const char* __restrict__ src, int64_t src_stride, char* __restrict__ dst,
                    int64_t dst_stride, int row_chunks, const int32_t* __restrict__ perm,
                    int64_t n_rows) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  for (int64_t q = warp0; q < n_rows; q += nwarps) {
    const int64_t p = perm ? static_cast<int64_t>(__ldg(perm + q)) : q;
    const int4* s = reinterpret_cast<const int4*>(src + p * src_stride);
    int4* d = reinterpret_cast<int4*>(dst + q * dst_stride);
    for (int c0 = 0; c0 < row_chunks; c0 += 32 * kChunks) {
      int4 r[kChunks];
#pragma unroll
      for (int u = 0; u < kChunks; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < row_chunks) r[u] = __ldg(s + c);
      }
#pragma unroll
      for (int u = 0; u < kChunks; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < row_chunks) d[c] = r[u];
      }
    }
  }
}

bool ranges_overlap(const void* a, int64_t a_len, const void* b, int64_t b_len) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(b_len) && b0 < a0 + static_cast<uintptr_t>(a_len);
}

}  // namespace
}  // namespace wp

using namespace wp;

extern "C" int wp_permute(const wp_plan* plan, int src_layout, int dst_layout, const void* src,
                          int64_t src_stride_B, void* dst, int64_t dst_stride_B, int64_t row_B,
                          void* stream) {
  if (!plan) return fail(WP_EINVAL, "plan is NULL");
  if (src_layout < 0 || src_layout >= kNumLayouts || dst_layout < 0 || dst_layout >= kNumLayouts)
    return fail(WP_EINVAL, "bad layout pair (%d -> %d)", src_layout, dst_layout);
  if (!src || !dst) return fail(WP_EINVAL, "src or dst is NULL");
  if (row_B <= 0 || (row_B & 15) != 0)
    return fail(WP_EUNSUPPORTED, "row_B=%lld must be a positive multiple of 16", (long long)row_B);
  if (row_B / 16 > (int64_t(1) << 30)) return fail(WP_EUNSUPPORTED, "row_B too large");
  if ((src_stride_B & 15) || (dst_stride_B & 15) || src_stride_B < row_B || dst_stride_B < row_B)
    return fail(WP_EUNSUPPORTED, "strides (%lld, %lld) must be multiples of 16 and >= row_B=%lld",
                (long long)src_stride_B, (long long)dst_stride_B, (long long)row_B);
  if (!aligned16(src) || !aligned16(dst))
    return fail(WP_EUNSUPPORTED, "src and dst must be 16-byte aligned");
  const int64_t N = plan->N;
  const int64_t src_len = (N - 1) * src_stride_B + row_B;
  const int64_t dst_len = (N - 1) * dst_stride_B + row_B;
  if (ranges_overlap(src, src_len, dst, dst_len))
    return fail(WP_EINVAL, "src and dst byte ranges overlap (in-place permutation is not supported)");
  if (int rc = require_uploaded(plan)) return rc;

  const int32_t* perm =
      (src_layout == dst_layout) ? nullptr : dev_ptr<int32_t>(plan, plan->perm_off[src_layout][dst_layout]);
  const int row_chunks = static_cast<int>(row_B / 16);
  auto kern = row_chunks <= 12 * 32 ? permute_rows_kernel<12> : permute_rows_kernel<8>;
  int sms = 0, per_sm = 0;
  if (int rc = cuda_check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, plan->device),
                          "cudaDeviceGetAttribute"))
    return rc;
  if (int rc = cuda_check(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0),
                          "cudaOccupancyMaxActiveBlocksPerMultiprocessor"))
    return rc;
  const int64_t warps_needed = N;
  int64_t blocks = static_cast<int64_t>(sms) * std::min(std::max(per_sm, 1), kMaxBlocksPerSm);
  blocks = std::min<int64_t>(blocks, (warps_needed * 32 + kThreads - 1) / kThreads);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  kern<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(static_cast<const char*>(src), src_stride_B,
                                                          static_cast<char*>(dst), dst_stride_B, row_chunks, perm, N);
  if (int rc = cuda_check(cudaGetLastError(), "permute_rows_kernel launch")) return rc;
  return ok();
}
