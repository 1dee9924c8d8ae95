// wp_rope: window-local 3D rotary position embedding of q and k, in place.
//
// "Window-Aligned Sequence Parallelism (SeedVR2)", §Reference quirks
// reproduced on purpose: a video token at window-local (dt, dh, dw) uses the
// axial indices (text_len + dt, dh, dw), every window restarting at 0; the
// rotary span is 3 * (head_dim / 3) channels, the rest pass through.
// Readings where the page is silent: axis blocks t, h, w of head_dim/3
// channels each; channels (2i, 2i+1) of a block rotate by pos * base^(-2i/d);
// a text token at position l uses (l, l, l).
//
// HBM-bound: every q and k element is read and written once.  One warp per
// row (video rows in layout order, then text rows): lane 0 finds the row's
// window (binary search of the window offsets) and its window-local
// position, the lanes fill a per-warp table of the 63 (cos, sin) pairs with
// sincosf, and then stream the row's q and k through 16-byte loads/stores
// (four chunks of each per lane in flight), the same angles serving every
// head.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "attn_internal.h"
#include "wp_internal.h"

namespace wp {
namespace {

constexpr int kHd = 128;
constexpr int kAxis = kHd / 3;         // 42 channels per axis
constexpr int kPairsPerAxis = kAxis / 2;  // 21
constexpr int kPairs = 3 * kPairsPerAxis;  // 63 rotated pairs; channels 126, 127 pass through
constexpr int kWarps = 8;

struct RopeParams {
  char *q, *k, *qt, *kt;
  int64_t stride, tstride;  // bytes
  char* kdst;               // rope_k_copy_kernel: destination rows (dstride bytes apart)
  int64_t dstride;
  char *qtdst, *ktdst;      // rope_text_copy_kernel: destination rows (tdstride bytes apart)
  int64_t tdstride;
  const int32_t *win_off, *ids, *boxes;
  int nwin, N, L, heads, H, W;
  float theta[kPairsPerAxis];  // base^(-2i/42)
};

// Rotates the pairs of one 16-byte chunk (chunk c of a row) in registers.
template <typename T>
__device__ __forceinline__ void rotate_chunk(int4& v, int c, const float2* cs) {
  constexpr int kPer = 16 / sizeof(T);  // elements per 16-byte chunk
  T* e = reinterpret_cast<T*>(&v);
  const int ch0 = (c * kPer) % kHd;  // first channel of the chunk within its head
#pragma unroll
  for (int u = 0; u < kPer; u += 2) {
    const int pair = (ch0 + u) >> 1;
    if (pair < kPairs) {
      const float2 t = cs[pair];
      float x0, x1;
      if constexpr (sizeof(T) == 2) {
        x0 = __bfloat162float(e[u]);
        x1 = __bfloat162float(e[u + 1]);
      } else {
        x0 = e[u];
        x1 = e[u + 1];
      }
      const float y0 = x0 * t.x - x1 * t.y, y1 = x0 * t.y + x1 * t.x;
      if constexpr (sizeof(T) == 2) {
        e[u] = __float2bfloat16_rn(y0);
        e[u + 1] = __float2bfloat16_rn(y1);
      } else {
        e[u] = y0;
        e[u + 1] = y1;
      }
    }
  }
}

// The q and k rows of one token, in batches of kBatch chunks per lane per
// row: all 2 * kBatch loads of a batch are issued before the first chunk is
// rotated and stored, so each lane keeps 2 * kBatch * 16 bytes in flight
// (one chunk at a time left the pass at 91% of the copy rate, four at 97%;
// more raise the register count past two blocks per SM and lose).
constexpr int kBatch = 4;

template <typename T>
__device__ __forceinline__ void rotate_rows(char* qrow, char* krow, int heads, const float2* cs, int lane) {
  constexpr int kPer = 16 / sizeof(T);
  const int chunks = heads * kHd / kPer;
  for (int c0 = 0; c0 < chunks; c0 += 32 * kBatch) {
    int4 a[kBatch], b[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int c = c0 + u * 32 + lane;
      if (c < chunks) {
        a[u] = *reinterpret_cast<const int4*>(qrow + static_cast<int64_t>(c) * 16);
        b[u] = *reinterpret_cast<const int4*>(krow + static_cast<int64_t>(c) * 16);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int c = c0 + u * 32 + lane;
      if (c < chunks) {
        rotate_chunk<T>(a[u], c, cs);
        rotate_chunk<T>(b[u], c, cs);
        *reinterpret_cast<int4*>(qrow + static_cast<int64_t>(c) * 16) = a[u];
        *reinterpret_cast<int4*>(krow + static_cast<int64_t>(c) * 16) = b[u];
      }
    }
  }
}

// The (cos, sin) table of row r (video rows in layout order, then text
// rows): one warp finds the row's window and window-local position and
// fills cs[0 .. 62].
__device__ __forceinline__ void row_table(const RopeParams& p, int64_t r, float2* cs, int lane) {
  int pos[3];
  if (r < p.N) {
    int lo = 0, hi = p.nwin - 1;  // window holding layout row r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.win_off + mid) <= r) lo = mid; else hi = mid - 1;
    }
    const int c = __ldg(p.ids + r);
    const int t = c / (p.H * p.W), h = (c / p.W) % p.H, w = c % p.W;
    const int32_t* box = p.boxes + lo * 6;  // t0,t1,h0,h1,w0,w1
    pos[0] = p.L + t - __ldg(box + 0);
    pos[1] = h - __ldg(box + 2);
    pos[2] = w - __ldg(box + 4);
  } else {
    pos[0] = pos[1] = pos[2] = static_cast<int>(r - p.N);
  }
  for (int q = lane; q < kPairs; q += 32) {
    float s, c;
    sincosf(static_cast<float>(pos[q / kPairsPerAxis]) * p.theta[q % kPairsPerAxis], &s, &c);
    cs[q] = make_float2(c, s);
  }
}

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) rope_kernel(const RopeParams p) {
  __shared__ float2 table[kWarps][kPairs + 1];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float2* cs = table[wib];
  const int64_t rows = static_cast<int64_t>(p.N) + p.L;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kWarps + wib; r < rows;
       r += static_cast<int64_t>(gridDim.x) * kWarps) {
    row_table(p, r, cs, lane);
    __syncwarp();
    if (r < p.N)
      rotate_rows<T>(p.q + r * p.stride, p.k + r * p.stride, p.heads, cs, lane);
    else
      rotate_rows<T>(p.qt + (r - p.N) * p.tstride, p.kt + (r - p.N) * p.tstride, p.heads, cs, lane);
    __syncwarp();
  }
}

// Video k only, rotated out of place (bf16): row r of p.k (stride p.stride)
// to row r of p.kdst (stride p.dstride), kCopyBatch chunks per lane in
// flight (a 24-head row is 32 lanes x 12 chunks; at two blocks per SM this
// runs at 97.5% of the copy rate, 8 chunks at eight blocks at 91%).
constexpr int kCopyBatch = 12;

__global__ void __launch_bounds__(kWarps * 32) rope_k_copy_kernel(const RopeParams p) {
  __shared__ float2 table[kWarps][kPairs + 1];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float2* cs = table[wib];
  constexpr int kPer = 8, kB = kCopyBatch;
  const int chunks = p.heads * kHd / kPer;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kWarps + wib; r < p.N;
       r += static_cast<int64_t>(gridDim.x) * kWarps) {
    row_table(p, r, cs, lane);
    __syncwarp();
    const char* src = p.k + r * p.stride;
    char* dst = p.kdst + r * p.dstride;
    for (int c0 = 0; c0 < chunks; c0 += 32 * kB) {
      int4 a[kB];
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < chunks) a[u] = __ldg(reinterpret_cast<const int4*>(src + static_cast<int64_t>(c) * 16));
      }
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < chunks) {
          rotate_chunk<__nv_bfloat16>(a[u], c, cs);
          *reinterpret_cast<int4*>(dst + static_cast<int64_t>(c) * 16) = a[u];
        }
      }
    }
    __syncwarp();
  }
}

// Text q and k rotated out of place (bf16): row l of p.qt / p.kt (stride
// p.tstride) to row l of p.qtdst / p.ktdst (stride p.tdstride), position
// (l, l, l); one warp per row as in rope_kernel (p.N = 0).
__global__ void __launch_bounds__(kWarps * 32) rope_text_copy_kernel(const RopeParams p) {
  __shared__ float2 table[kWarps][kPairs + 1];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float2* cs = table[wib];
  constexpr int kPer = 8;
  const int chunks = p.heads * kHd / kPer;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kWarps + wib; r < p.L;
       r += static_cast<int64_t>(gridDim.x) * kWarps) {
    row_table(p, r, cs, lane);
    __syncwarp();
    for (int tq = 0; tq < 2; ++tq) {
      const char* src = (tq ? p.kt : p.qt) + r * p.tstride;
      char* dst = (tq ? p.ktdst : p.qtdst) + r * p.tdstride;
      for (int c = lane; c < chunks; c += 32) {
        int4 a = __ldg(reinterpret_cast<const int4*>(src + static_cast<int64_t>(c) * 16));
        rotate_chunk<__nv_bfloat16>(a, c, cs);
        *reinterpret_cast<int4*>(dst + static_cast<int64_t>(c) * 16) = a;
      }
    }
    __syncwarp();
  }
}

}  // namespace

void rope_theta(float rope_base, float* theta21) {
  for (int i = 0; i < kPairsPerAxis; ++i)
    theta21[i] = static_cast<float>(std::pow(static_cast<double>(rope_base), -2.0 * i / kAxis));
}

int rope_text_copy(const void* qt, const void* kt, int64_t txt_stride_B, void* qt_out, void* kt_out, int L,
                   int heads, float rope_base, cudaStream_t stream) {
  if (L <= 0) return WP_OK;
  RopeParams p{};
  p.qt = static_cast<char*>(const_cast<void*>(qt));
  p.kt = static_cast<char*>(const_cast<void*>(kt));
  p.tstride = txt_stride_B;
  p.qtdst = static_cast<char*>(qt_out);
  p.ktdst = static_cast<char*>(kt_out);
  p.tdstride = static_cast<int64_t>(heads) * kHd * 2;
  p.N = 0;  // text rows only: positions (l, l, l)
  p.L = L;
  p.heads = heads;
  rope_theta(rope_base, p.theta);
  const unsigned blocks = static_cast<unsigned>((L + kWarps - 1) / kWarps);
  rope_text_copy_kernel<<<blocks, kWarps * 32, 0, stream>>>(p);
  return cuda_check(cudaGetLastError(), "rope_text_copy_kernel launch");
}

int rope_k_copy(const wp_plan* plan, int layout, const void* k, int64_t vid_stride_B, void* k_out, int heads, int L,
                float rope_base, cudaStream_t stream) {
  if (plan->N == 0) return WP_OK;
  RopeParams p{};
  p.k = static_cast<char*>(const_cast<void*>(k));
  p.stride = vid_stride_B;
  p.kdst = static_cast<char*>(k_out);
  p.dstride = static_cast<int64_t>(heads) * kHd * 2;
  p.win_off = dev_ptr<int32_t>(plan, plan->dlay[layout].win_off);
  p.ids = dev_ptr<int32_t>(plan, plan->dlay[layout].ids);
  p.boxes = dev_ptr<int32_t>(plan, plan->dlay[layout].boxes);
  p.nwin = plan->lay[layout].nwin;
  p.N = static_cast<int>(plan->N);
  p.L = L;  // positions only: video t offset by L
  p.heads = heads;
  p.H = plan->H;
  p.W = plan->W;
  rope_theta(rope_base, p.theta);
  int sms = 0;
  if (int rc = cuda_check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, plan->device),
                          "cudaDeviceGetAttribute"))
    return rc;
  const int64_t blocks = std::min<int64_t>((plan->N + kWarps - 1) / kWarps, static_cast<int64_t>(sms) * 2);
  rope_k_copy_kernel<<<static_cast<unsigned>(blocks), kWarps * 32, 0, stream>>>(p);
  return cuda_check(cudaGetLastError(), "rope_k_copy_kernel launch");
}

}  // namespace wp

using namespace wp;

extern "C" int wp_rope(const wp_plan* plan, int layout, int heads, int head_dim, int L, int dtype, void* q,
                       void* k, int64_t vid_row_stride_B, void* qt, void* kt, int64_t txt_row_stride_B,
                       float rope_base, void* stream) {
  if (!plan) return fail(WP_EINVAL, "plan is NULL");
  if (layout < 0 || layout >= kNumLayouts) return fail(WP_EINVAL, "bad layout %d", layout);
  if (heads < 1 || L < 0) return fail(WP_EINVAL, "heads=%d L=%d", heads, L);
  if (dtype != WP_BF16 && dtype != WP_FP32) return fail(WP_EINVAL, "bad dtype %d", dtype);
  if (head_dim != kHd) return fail(WP_EUNSUPPORTED, "wp_rope supports head_dim 128 (got %d)", head_dim);
  if (!(rope_base > 1.f)) return fail(WP_EINVAL, "rope_base must be > 1");
  if (!q || !k || (L > 0 && (!qt || !kt))) return fail(WP_EINVAL, "q/k (or text q/k with L > 0) is NULL");
  const int64_t row_B = static_cast<int64_t>(heads) * head_dim * (dtype == WP_BF16 ? 2 : 4);
  for (const void* ptr : {static_cast<const void*>(q), static_cast<const void*>(k)})
    if (!aligned16(ptr)) return fail(WP_EUNSUPPORTED, "q and k must be 16-byte aligned");
  if (L > 0)
    for (const void* ptr : {static_cast<const void*>(qt), static_cast<const void*>(kt)})
      if (!aligned16(ptr)) return fail(WP_EUNSUPPORTED, "text q and k must be 16-byte aligned");
  if (vid_row_stride_B < row_B || (vid_row_stride_B & 15) || (L > 0 && (txt_row_stride_B < row_B || (txt_row_stride_B & 15))))
    return fail(WP_EUNSUPPORTED, "row strides must be multiples of 16 and >= %lld", (long long)row_B);
  if (int rc = require_uploaded(plan)) return rc;
  RopeParams p;
  p.q = static_cast<char*>(q);
  p.k = static_cast<char*>(k);
  p.qt = static_cast<char*>(qt);
  p.kt = static_cast<char*>(kt);
  p.stride = vid_row_stride_B;
  p.tstride = txt_row_stride_B;
  p.win_off = dev_ptr<int32_t>(plan, plan->dlay[layout].win_off);
  p.ids = dev_ptr<int32_t>(plan, plan->dlay[layout].ids);
  p.boxes = dev_ptr<int32_t>(plan, plan->dlay[layout].boxes);
  p.nwin = plan->lay[layout].nwin;
  p.N = static_cast<int>(plan->N);
  p.L = L;
  p.heads = heads;
  p.H = plan->H;
  p.W = plan->W;
  rope_theta(rope_base, p.theta);
  int sms = 0;
  if (int rc = cuda_check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, plan->device),
                          "cudaDeviceGetAttribute"))
    return rc;
  const int64_t rows = plan->N + L;
  const int64_t blocks = std::min<int64_t>((rows + kWarps - 1) / kWarps, static_cast<int64_t>(sms) * 8);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == WP_BF16)
    rope_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(p);
  else
    rope_kernel<float><<<static_cast<unsigned>(blocks), kWarps * 32, 0, s>>>(p);
  if (int rc = cuda_check(cudaGetLastError(), "rope_kernel launch")) return rc;
  return ok();
}
