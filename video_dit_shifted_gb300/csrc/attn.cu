// wp_window_attn: argument checks, the fp32 parity kernel and the text mean.
//
// "Window-Aligned Sequence Parallelism (SeedVR2)":
//   §SeedVR2 integration -- one bidirectional attention per
//     [video window ; replicated text] segment, video rows back to canonical
//     order;
//   §Text stream -- text output = (sum over windows of T_w) / window count.
//
// The bf16 tensor-core kernel lives in attn_tc.cu.  This file holds
//   * attn_f32_kernel: fp32 SIMT attention (parity mode, head_dim 64/128),
//   * text_mean_kernel: o_txt = (sum_w T_w) / nwin, each output element
//     summed in window order by one thread (no atomics, so the result is
//     deterministic), and
//   * the C entry points wp_attn_workspace_bytes / wp_window_attn /
//     wp_read_status.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "attn_internal.h"

namespace wp {
namespace {

// ------------------------------------------------------------ fp32 path --
// One block = 32 query rows of one segment (window w, head h); 4 threads per
// row, each holding every 4th element of the row's head_dim.  Keys stream
// through shared memory 32 at a time; the softmax is the usual online
// (running max / running sum) form in fp32 with expf.
constexpr int kF32Rows = 32;
constexpr int kF32Keys = 32;
constexpr int kF32Tpr = 4;

struct F32Params {
  const float *q, *k, *v, *qt, *kt, *vt;
  int64_t vid_stride, txt_stride, o_stride;  // in floats
  float* o_vid;
  float* partial;
  const int32_t *win_off, *ids;
  int64_t n_rows;  // rows of o_vid (N)
  int* status;
  int heads, L, qblocks;
  float scale;
};

template <int HD>
__global__ void __launch_bounds__(kF32Rows * kF32Tpr) attn_f32_kernel(F32Params p) {
  constexpr int DPT = HD / kF32Tpr;
  __shared__ float Ks[kF32Keys][HD];
  __shared__ float Vs[kF32Keys][HD];
  const int w = blockIdx.x / p.qblocks;
  const int qb = blockIdx.x % p.qblocks;
  const int h = blockIdx.y;
  const int a = p.win_off[w];
  const int n_w = p.win_off[w + 1] - a;
  const int seg = n_w + p.L;
  if (qb * kF32Rows >= seg) return;  // uniform per block
  const int row = threadIdx.x / kF32Tpr, part = threadIdx.x % kF32Tpr;
  const int r = qb * kF32Rows + row;
  const bool live = r < seg;

  auto qrow = [&](int i) -> const float* {  // segment row i of q
    return i < n_w ? p.q + (a + i) * p.vid_stride + h * HD : p.qt + (i - n_w) * p.txt_stride + h * HD;
  };
  float qr[DPT], acc[DPT];
#pragma unroll
  for (int i = 0; i < DPT; ++i) {
    qr[i] = live ? qrow(r)[i * kF32Tpr + part] : 0.f;
    acc[i] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int k0 = 0; k0 < seg; k0 += kF32Keys) {
    __syncthreads();
    for (int e = threadIdx.x; e < kF32Keys * HD; e += blockDim.x) {
      const int j = e / HD, d = e % HD, kk = k0 + j;
      float kv = 0.f, vv = 0.f;
      if (kk < n_w) {
        kv = p.k[(a + kk) * p.vid_stride + h * HD + d];
        vv = p.v[(a + kk) * p.vid_stride + h * HD + d];
      } else if (kk < seg) {
        kv = p.kt[(kk - n_w) * p.txt_stride + h * HD + d];
        vv = p.vt[(kk - n_w) * p.txt_stride + h * HD + d];
      }
      Ks[j][d] = kv;
      Vs[j][d] = vv;
    }
    __syncthreads();
    const int nk = min(kF32Keys, seg - k0);
    float s[kF32Keys];
    float tmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < kF32Keys; ++j) {
      float dot = 0.f;
#pragma unroll
      for (int i = 0; i < DPT; ++i) dot = fmaf(qr[i], Ks[j][i * kF32Tpr + part], dot);
      dot += __shfl_xor_sync(0xffffffffu, dot, 1);
      dot += __shfl_xor_sync(0xffffffffu, dot, 2);
      s[j] = j < nk ? dot * p.scale : -INFINITY;
      tmax = fmaxf(tmax, s[j]);
    }
    const float m_new = fmaxf(m, tmax);
    const float alpha = expf(m - m_new);  // m = -inf on the first tile -> 0
    l *= alpha;
#pragma unroll
    for (int i = 0; i < DPT; ++i) acc[i] *= alpha;
#pragma unroll
    for (int j = 0; j < kF32Keys; ++j) {
      const float pj = j < nk ? expf(s[j] - m_new) : 0.f;
      l += pj;
#pragma unroll
      for (int i = 0; i < DPT; ++i) acc[i] = fmaf(pj, Vs[j][i * kF32Tpr + part], acc[i]);
    }
    m = m_new;
  }
  if (!live) return;
  const float inv = 1.f / l;
  const int64_t orow = r < n_w ? (p.ids ? static_cast<int64_t>(p.ids[a + r]) : static_cast<int64_t>(a + r)) : 0;
  if (r < n_w && static_cast<uint64_t>(orow) >= static_cast<uint64_t>(p.n_rows)) {
    atomicCAS(p.status, 0, WP_EDEVICE);  // table entry outside the output (plan buffer changed): not written
    return;
  }
  float* out = r < n_w ? p.o_vid + orow * p.o_stride + h * HD
                       : p.partial + ((static_cast<int64_t>(w) * p.L + (r - n_w)) * p.heads + h) * HD;
#pragma unroll
  for (int i = 0; i < DPT; ++i) out[i * kF32Tpr + part] = acc[i] * inv;
}

// ---------------------------------------------------------- text mean ----
// Thread i owns elements 4i .. 4i+3 (16-byte loads; n is a multiple of 4
// since head_dim is) and loads kAhead windows before adding them, in window
// order, so that each thread keeps 64 bytes in flight while the fp32 sum
// stays the ordered one (one thread per element at a time left the pass at
// 91% of the copy rate; this runs at 98%).
constexpr int kAhead = 4;

template <typename OutT>
__global__ void __launch_bounds__(256) text_mean_kernel(const float* __restrict__ part, int nwin, int64_t n,
                                                        OutT* __restrict__ out) {
  const int64_t n4 = n / 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const float count = static_cast<float>(nwin);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4* src = reinterpret_cast<const float4*>(part) + i;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int w = 0;
    for (; w + kAhead <= nwin; w += kAhead) {
      float4 v[kAhead];
#pragma unroll
      for (int u = 0; u < kAhead; ++u) v[u] = __ldcs(src + static_cast<int64_t>(w + u) * n4);
#pragma unroll
      for (int u = 0; u < kAhead; ++u) {
        acc.x += v[u].x;
        acc.y += v[u].y;
        acc.z += v[u].z;
        acc.w += v[u].w;
      }
    }
    for (; w < nwin; ++w) {
      const float4 v = __ldcs(src + static_cast<int64_t>(w) * n4);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const float m[4] = {acc.x / count, acc.y / count, acc.z / count, acc.w / count};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if constexpr (sizeof(OutT) == 2) {
        out[4 * i + c] = __float2bfloat16_rn(m[c]);
      } else {
        out[4 * i + c] = m[c];
      }
    }
  }
}

int launch_text_mean(const AttnCall& c) {
  const int64_t n = static_cast<int64_t>(c.L) * c.heads * c.hd;
  if (n == 0) return WP_OK;
  const int threads = 256;
  // One 16-byte group per thread up to 8 blocks per SM of a GB300 (152 SMs);
  // larger outputs loop.
  const int64_t blocks = std::min<int64_t>((n / 4 + threads - 1) / threads, 152 * 8);
  if (c.dtype == WP_BF16)
    text_mean_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), threads, 0, c.stream>>>(
        c.partial, c.nwin, n, static_cast<__nv_bfloat16*>(c.o_txt));
  else
    text_mean_kernel<float><<<static_cast<unsigned>(blocks), threads, 0, c.stream>>>(
        c.partial, c.nwin, n, static_cast<float*>(c.o_txt));
  return cuda_check(cudaGetLastError(), "text_mean_kernel launch");
}

}  // namespace

int launch_attn_f32(const AttnCall& c) {
  F32Params p;
  p.q = static_cast<const float*>(c.q);
  p.k = static_cast<const float*>(c.k);
  p.v = static_cast<const float*>(c.v);
  p.qt = static_cast<const float*>(c.qt);
  p.kt = static_cast<const float*>(c.kt);
  p.vt = static_cast<const float*>(c.vt);
  p.vid_stride = c.vid_stride_B / 4;
  p.txt_stride = c.txt_stride_B / 4;
  p.o_stride = c.o_stride_B / 4;
  p.o_vid = static_cast<float*>(c.o_vid);
  p.partial = c.partial;
  p.win_off = c.win_off;
  p.ids = c.ids;
  p.n_rows = c.N;
  p.status = c.status;
  p.heads = c.heads;
  p.L = c.L;
  p.qblocks = (c.max_tokens + c.L + kF32Rows - 1) / kF32Rows;
  p.scale = c.scale;
  const int64_t gx = static_cast<int64_t>(c.nwin) * p.qblocks;
  if (gx > 0x7fffffff) return fail(WP_EUNSUPPORTED, "fp32 grid too large");
  dim3 grid(static_cast<unsigned>(gx), c.heads);
  if (c.hd == 64)
    attn_f32_kernel<64><<<grid, kF32Rows * kF32Tpr, 0, c.stream>>>(p);
  else
    attn_f32_kernel<128><<<grid, kF32Rows * kF32Tpr, 0, c.stream>>>(p);
  return cuda_check(cudaGetLastError(), "attn_f32_kernel launch");
}

}  // namespace wp

using namespace wp;

namespace {

// Partial text outputs T_w start at kStatusBytes; with rope, the rotated
// text q and k (bf16, packed rows) follow them, then, 1024-byte aligned,
// the rotated video k (bf16, packed rows [N, heads * hd]).
int64_t partial_bytes(const wp_plan* plan, int layout, int heads, int hd, int L) {
  return static_cast<int64_t>(plan->lay[layout].nwin) * L * heads * hd * 4;
}

int64_t text_rot_offset(const wp_plan* plan, int layout, int heads, int hd, int L) {
  return static_cast<int64_t>(kStatusBytes) + partial_bytes(plan, layout, heads, hd, L);
}

int64_t krot_offset(const wp_plan* plan, int layout, int heads, int hd, int L) {
  const int64_t end = text_rot_offset(plan, layout, heads, hd, L) + 2 * static_cast<int64_t>(L) * heads * hd * 2;
  return (end + 1023) / 1024 * 1024;
}

int workspace_bytes(const wp_plan* plan, int layout, int heads, int hd, int L, size_t* bytes, bool rope = false) {
  *bytes = rope ? static_cast<size_t>(krot_offset(plan, layout, heads, hd, L) + plan->N * heads * hd * 2)
                : kStatusBytes + static_cast<size_t>(partial_bytes(plan, layout, heads, hd, L));
  return WP_OK;
}

int check_shape(const wp_plan* plan, int layout, int heads, int hd, int L, int dtype) {
  if (!plan) return fail(WP_EINVAL, "plan is NULL");
  if (layout != WP_REGULAR && layout != WP_SHIFTED)
    return fail(WP_EINVAL, "attention layout must be WP_REGULAR or WP_SHIFTED (got %d)", layout);
  if (heads < 1 || heads > 65535) return fail(WP_EINVAL, "heads=%d out of range [1, 65535]", heads);
  if (L < 0) return fail(WP_EINVAL, "L=%d < 0", L);
  if (dtype != WP_BF16 && dtype != WP_FP32) return fail(WP_EINVAL, "bad dtype %d", dtype);
  if (hd != 64 && hd != 128) return fail(WP_EUNSUPPORTED, "head_dim=%d (supported: 64, 128)", hd);
  return WP_OK;
}

}  // namespace

extern "C" int wp_attn_workspace_bytes(const wp_plan* plan, int layout, int heads, int head_dim,
                                       int L, int dtype, size_t* bytes) {
  if (int rc = check_shape(plan, layout, heads, head_dim, L, dtype)) return rc;
  if (!bytes) return fail(WP_EINVAL, "bytes is NULL");
  workspace_bytes(plan, layout, heads, head_dim, L, bytes);
  return ok();
}

extern "C" int wp_attn_rope_workspace_bytes(const wp_plan* plan, int layout, int heads, int head_dim, int L,
                                            int dtype, size_t* bytes) {
  if (int rc = check_shape(plan, layout, heads, head_dim, L, dtype)) return rc;
  if (!bytes) return fail(WP_EINVAL, "bytes is NULL");
  workspace_bytes(plan, layout, heads, head_dim, L, bytes, true);
  return ok();
}

namespace {

// The plan's tables for one call: windows of `layout`, and the output row
// of every input row for `out_layout`.
int set_tables(AttnCall& c, const wp_plan* plan, int layout, int out_layout, int L) {
  const LayoutTables& LT = plan->lay[layout];
  c.N = plan->N;
  c.nwin = LT.nwin;
  c.max_tokens = LT.max_tokens;
  c.win_off = dev_ptr<int32_t>(plan, plan->dlay[layout].win_off);
  // Row of the output layout for each row of the input layout:
  // canonical -> ids; the same layout -> identity (no table); another window
  // layout b -> pos_b[ids_layout[q]], which is the fused table perm[b -> layout].
  if (out_layout == WP_CANONICAL)
    c.ids = dev_ptr<int32_t>(plan, plan->dlay[layout].ids);
  else if (out_layout == layout)
    c.ids = nullptr;
  else
    c.ids = dev_ptr<int32_t>(plan, plan->perm_off[out_layout][layout]);
  c.pair_off[0] = dev_ptr<int32_t>(plan, plan->dlay[layout].pair_off[0]);
  c.pair_off[1] = dev_ptr<int32_t>(plan, plan->dlay[layout].pair_off[1]);
  c.text_tiles = (L + kTileM - 1) / kTileM;
  const int64_t pairs = static_cast<int64_t>(LT.pair_off[c.text_tiles & 1][LT.nwin]) +
                        static_cast<int64_t>(LT.nwin) * (c.text_tiles >> 1);
  if (pairs > 0x7fffffff) return fail(WP_EUNSUPPORTED, "too many query tiles");
  c.total_pairs = static_cast<int>(pairs);
  return WP_OK;
}

int window_attn_impl(const wp_plan* plan, int layout, int out_layout, int heads, int head_dim, int L,
                     int dtype, const void* q, const void* k, const void* v, int64_t vid_row_stride_B,
                     const void* qt, const void* kt, const void* vt, int64_t txt_row_stride_B,
                     void* o_vid, int64_t o_vid_row_stride_B, void* o_txt, void* workspace,
                     size_t ws_bytes, float softmax_scale, void* stream, float rope_base = 0.f) {
  const bool rope = rope_base != 0.f;
  if (int rc = check_shape(plan, layout, heads, head_dim, L, dtype)) return rc;
  if (rope) {
    if (!(rope_base > 1.f)) return fail(WP_EINVAL, "rope_base must be > 1");
    if (dtype != WP_BF16 || head_dim != 128)
      return fail(WP_EUNSUPPORTED, "RoPE attention supports bf16 with head_dim 128");
  }
  if (out_layout < 0 || out_layout >= kNumLayouts) return fail(WP_EINVAL, "bad output layout %d", out_layout);
  if (!q || !k || !v || !o_vid || !workspace) return fail(WP_EINVAL, "q, k, v, o_vid or workspace is NULL");
  if (L > 0 && (!qt || !kt || !vt || !o_txt)) return fail(WP_EINVAL, "text pointers are NULL with L=%d", L);
  const int64_t elem = dtype == WP_BF16 ? 2 : 4;
  const int64_t row_B = static_cast<int64_t>(heads) * head_dim * elem;
  for (const void* ptr : {q, k, v, static_cast<const void*>(o_vid), static_cast<const void*>(workspace)})
    if (!aligned16(ptr)) return fail(WP_EUNSUPPORTED, "q/k/v/o_vid/workspace must be 16-byte aligned");
  if (L > 0)
    for (const void* ptr : {qt, kt, vt, static_cast<const void*>(o_txt)})
      if (!aligned16(ptr)) return fail(WP_EUNSUPPORTED, "qt/kt/vt/o_txt must be 16-byte aligned");
  auto stride_ok = [&](int64_t s) { return s >= row_B && (s & 15) == 0; };
  if (!stride_ok(vid_row_stride_B) || !stride_ok(o_vid_row_stride_B) || (L > 0 && !stride_ok(txt_row_stride_B)))
    return fail(WP_EUNSUPPORTED,
                "row strides (video %lld, text %lld, out %lld) must be multiples of 16 and >= %lld",
                (long long)vid_row_stride_B, (long long)txt_row_stride_B, (long long)o_vid_row_stride_B,
                (long long)row_B);
  size_t need = 0;
  workspace_bytes(plan, layout, heads, head_dim, L, &need, rope);
  if (ws_bytes < need) return fail(WP_EINVAL, "workspace too small: %zu < %zu bytes", ws_bytes, need);
  if (int rc = require_uploaded(plan)) return rc;

  AttnCall c{};
  c.layout = layout; c.heads = heads; c.hd = head_dim; c.L = L; c.dtype = dtype;
  c.q = q; c.k = k; c.v = v; c.vid_stride_B = vid_row_stride_B; c.vid_v_stride_B = vid_row_stride_B;
  c.qt = qt; c.kt = kt; c.vt = vt; c.txt_stride_B = txt_row_stride_B; c.vt_stride_B = txt_row_stride_B;
  c.o_vid = o_vid; c.o_stride_B = o_vid_row_stride_B; c.o_txt = o_txt;
  c.status = static_cast<int*>(workspace);
  c.partial = reinterpret_cast<float*>(static_cast<char*>(workspace) + kStatusBytes);
  c.scale = softmax_scale > 0.f ? softmax_scale : 1.f / std::sqrt(static_cast<float>(head_dim));
  c.stream = static_cast<cudaStream_t>(stream);
  if (int rc = set_tables(c, plan, layout, out_layout, L)) return rc;
  if (rope) {
    c.rope = true;
    c.boxes = dev_ptr<int32_t>(plan, plan->dlay[layout].boxes);
    c.wt = plan->wt;
    c.wh = plan->wh;
    c.ww = plan->ww;
    rope_theta(rope_base, c.rope_theta);
  }

  if (int rc = cuda_check(cudaMemsetAsync(workspace, 0, kStatusBytes, c.stream), "cudaMemsetAsync(status)"))
    return rc;
  if (rope) {
    // Every video K tile is read by every work item of its (window, head):
    // rotate k once, into the workspace, and let the kernel read the copy
    // (the kernel rotates only the video Q tiles, each read by one item).
    char* krot = static_cast<char*>(workspace) + krot_offset(plan, layout, heads, head_dim, L);
    if (int rc = rope_k_copy(plan, layout, k, vid_row_stride_B, krot, heads, L, rope_base, c.stream)) return rc;
    c.k = krot;
    c.vid_k_stride_B = static_cast<int64_t>(heads) * head_dim * 2;
  }
  if (rope && L > 0) {
    // The text rows are shared by every window: rotate them once, into the
    // workspace, and let the kernel read the copies.
    char* rot = static_cast<char*>(workspace) + text_rot_offset(plan, layout, heads, head_dim, L);
    void* qt_rot = rot;
    void* kt_rot = rot + static_cast<int64_t>(L) * heads * head_dim * 2;
    if (int rc = rope_text_copy(qt, kt, txt_row_stride_B, qt_rot, kt_rot, L, heads, rope_base, c.stream)) return rc;
    c.qt = qt_rot;
    c.kt = kt_rot;
    c.txt_stride_B = static_cast<int64_t>(heads) * head_dim * 2;  // vt keeps vt_stride_B
  }
  int rc = dtype == WP_BF16 ? launch_attn_bf16_tc(c) : launch_attn_f32(c);
  if (rc) return rc;
  if (L > 0)
    if ((rc = launch_text_mean(c))) return rc;
  return ok();
}

}  // namespace

extern "C" int wp_window_attn(const wp_plan* plan, int layout, int heads, int head_dim, int L,
                              int dtype, const void* q, const void* k, const void* v,
                              int64_t vid_row_stride_B, const void* qt, const void* kt,
                              const void* vt, int64_t txt_row_stride_B, void* o_vid,
                              int64_t o_vid_row_stride_B, void* o_txt, void* workspace,
                              size_t ws_bytes, float softmax_scale, void* stream) {
  return window_attn_impl(plan, layout, WP_CANONICAL, heads, head_dim, L, dtype, q, k, v, vid_row_stride_B,
                          qt, kt, vt, txt_row_stride_B, o_vid, o_vid_row_stride_B, o_txt, workspace,
                          ws_bytes, softmax_scale, stream);
}

extern "C" int wp_window_attn_to(const wp_plan* plan, int layout, int out_layout, int heads, int head_dim,
                                 int L, int dtype, const void* q, const void* k, const void* v,
                                 int64_t vid_row_stride_B, const void* qt, const void* kt,
                                 const void* vt, int64_t txt_row_stride_B, void* o_vid,
                                 int64_t o_vid_row_stride_B, void* o_txt, void* workspace,
                                 size_t ws_bytes, float softmax_scale, void* stream) {
  return window_attn_impl(plan, layout, out_layout, heads, head_dim, L, dtype, q, k, v, vid_row_stride_B,
                          qt, kt, vt, txt_row_stride_B, o_vid, o_vid_row_stride_B, o_txt, workspace,
                          ws_bytes, softmax_scale, stream);
}

extern "C" int wp_window_attn_rope(const wp_plan* plan, int layout, int out_layout, int heads, int head_dim,
                                   int L, int dtype, const void* q, const void* k, const void* v,
                                   int64_t vid_row_stride_B, const void* qt, const void* kt,
                                   const void* vt, int64_t txt_row_stride_B, void* o_vid,
                                   int64_t o_vid_row_stride_B, void* o_txt, void* workspace,
                                   size_t ws_bytes, float softmax_scale, float rope_base, void* stream) {
  if (!(rope_base > 1.f)) return fail(WP_EINVAL, "rope_base must be > 1");
  return window_attn_impl(plan, layout, out_layout, heads, head_dim, L, dtype, q, k, v, vid_row_stride_B,
                          qt, kt, vt, txt_row_stride_B, o_vid, o_vid_row_stride_B, o_txt, workspace,
                          ws_bytes, softmax_scale, stream, rope_base);
}

extern "C" int wp_window_attn_fp8(const wp_plan* plan, int layout, int out_layout, int heads, int head_dim,
                                  int L, const void* q8, const void* k8, int64_t qk_row_stride_B, const void* v,
                                  int64_t v_row_stride_B, const void* qt8, const void* kt8,
                                  int64_t txt_qk_row_stride_B, const void* vt, int64_t txt_v_row_stride_B,
                                  float q_scale, float k_scale, void* o_vid, int64_t o_vid_row_stride_B,
                                  void* o_txt, void* workspace, size_t ws_bytes, float softmax_scale,
                                  void* stream) {
  if (int rc = check_shape(plan, layout, heads, head_dim, L, WP_BF16)) return rc;
  if (head_dim != 128) return fail(WP_EUNSUPPORTED, "e4m3 attention supports head_dim 128 (got %d)", head_dim);
  if (out_layout < 0 || out_layout >= kNumLayouts) return fail(WP_EINVAL, "bad output layout %d", out_layout);
  if (!(q_scale > 0.f) || !(k_scale > 0.f) || !std::isfinite(q_scale) || !std::isfinite(k_scale))
    return fail(WP_EINVAL, "q_scale and k_scale must be finite and > 0");
  if (!q8 || !k8 || !v || !o_vid || !workspace) return fail(WP_EINVAL, "q8, k8, v, o_vid or workspace is NULL");
  if (L > 0 && (!qt8 || !kt8 || !vt || !o_txt)) return fail(WP_EINVAL, "text pointers are NULL with L=%d", L);
  for (const void* ptr : {q8, k8, v, static_cast<const void*>(o_vid), static_cast<const void*>(workspace)})
    if (!aligned16(ptr)) return fail(WP_EUNSUPPORTED, "q8/k8/v/o_vid/workspace must be 16-byte aligned");
  if (L > 0)
    for (const void* ptr : {qt8, kt8, vt, static_cast<const void*>(o_txt)})
      if (!aligned16(ptr)) return fail(WP_EUNSUPPORTED, "qt8/kt8/vt/o_txt must be 16-byte aligned");
  const int64_t qk_B = static_cast<int64_t>(heads) * head_dim, bf_B = 2 * qk_B;
  auto ok_stride = [](int64_t s, int64_t min_B) { return s >= min_B && (s & 15) == 0; };
  if (!ok_stride(qk_row_stride_B, qk_B) || !ok_stride(v_row_stride_B, bf_B) || !ok_stride(o_vid_row_stride_B, bf_B) ||
      (L > 0 && (!ok_stride(txt_qk_row_stride_B, qk_B) || !ok_stride(txt_v_row_stride_B, bf_B))))
    return fail(WP_EUNSUPPORTED, "row strides must be multiples of 16 and hold a row (q/k %lld B, v/out %lld B)",
                (long long)qk_B, (long long)bf_B);
  size_t need = 0;
  workspace_bytes(plan, layout, heads, head_dim, L, &need);
  if (ws_bytes < need) return fail(WP_EINVAL, "workspace too small: %zu < %zu bytes", ws_bytes, need);
  if (int rc = require_uploaded(plan)) return rc;

  AttnCall c{};
  c.layout = layout; c.heads = heads; c.hd = head_dim; c.L = L; c.dtype = WP_BF16;
  c.fp8 = true;
  c.q = q8; c.k = k8; c.v = v; c.vid_stride_B = qk_row_stride_B; c.vid_v_stride_B = v_row_stride_B;
  c.qt = qt8; c.kt = kt8; c.vt = vt; c.txt_stride_B = txt_qk_row_stride_B; c.vt_stride_B = txt_v_row_stride_B;
  c.o_vid = o_vid; c.o_stride_B = o_vid_row_stride_B; c.o_txt = o_txt;
  c.status = static_cast<int*>(workspace);
  c.partial = reinterpret_cast<float*>(static_cast<char*>(workspace) + kStatusBytes);
  // scores = (q8 * q_scale) . (k8 * k_scale) * softmax_scale
  c.scale = (softmax_scale > 0.f ? softmax_scale : 1.f / std::sqrt(static_cast<float>(head_dim))) * q_scale * k_scale;
  c.stream = static_cast<cudaStream_t>(stream);
  if (int rc = set_tables(c, plan, layout, out_layout, L)) return rc;
  if (int rc = cuda_check(cudaMemsetAsync(workspace, 0, kStatusBytes, c.stream), "cudaMemsetAsync(status)"))
    return rc;
  if (int rc = launch_attn_bf16_tc(c)) return rc;
  if (L > 0)
    if (int rc = launch_text_mean(c)) return rc;
  return ok();
}

extern "C" int wp_debug_stall_next(int launches) {
  if (launches < 0) return fail(WP_EINVAL, "launches=%d < 0", launches);
  stall_next_launches(launches);
  return ok();
}

extern "C" int wp_read_status(const void* workspace, int* device_status, void* stream) {
  if (!device_status) return fail(WP_EINVAL, "device_status is NULL");
  if (!workspace) {
    // The fixed scratch of wp_window_attn_static on the current device.
    void* scratch = nullptr;
    if (int rc = static_scratch_address(&scratch)) return rc;
    workspace = scratch;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host = 0;
  if (int rc = cuda_check(cudaMemcpyAsync(&host, workspace, sizeof(int), cudaMemcpyDeviceToHost, s),
                          "cudaMemcpyAsync(status)"))
    return rc;
  if (int rc = cuda_check(cudaStreamSynchronize(s), "cudaStreamSynchronize(status)")) return rc;
  *device_status = host;
  return ok();
}
