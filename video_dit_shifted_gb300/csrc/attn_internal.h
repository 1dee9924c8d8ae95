// Shared between the attention translation units of libwp.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "wp_internal.h"

namespace wp {

// Workspace: a 256-byte status block, then the per-window text outputs
// T_w as fp32 [nwin, L, heads, head_dim].
constexpr size_t kStatusBytes = 256;

// Bound on every device-side wait (mbarrier or flag).  A wait that exceeds
// it records WP_ETIMEOUT in the status word and the kernel winds down.
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

struct AttnCall {
  int layout, heads, hd, L, dtype;
  const void *q, *k, *v;
  int64_t vid_stride_B;    // q and k
  int64_t vid_k_stride_B = 0;  // k, when it differs from q (0: vid_stride_B)
  int64_t vid_v_stride_B;  // v
  const void *qt, *kt, *vt;
  int64_t txt_stride_B;  // qt and kt
  int64_t vt_stride_B;
  void* o_vid;
  int64_t o_stride_B;
  void* o_txt;
  float* partial;  // [nwin, L, heads, hd] fp32
  int* status;     // device status word
  float scale;
  cudaStream_t stream;
  // from the plan
  int64_t N;
  int nwin, max_tokens;
  const int32_t* win_off;      // device
  const int32_t* ids;          // device: output row of each input row (NULL: same row)
  const int32_t* pair_off[2];  // device
  int total_pairs;             // query-tile pairs over all windows (tile kTileM)
  int text_tiles;              // ceil(L / kTileM)
  // q, k, qt, kt are e4m3 codes (wp_window_attn_fp8); their dequantisation
  // scales are folded into `scale`.
  bool fp8 = false;
  // Window-local RoPE of the video Q tiles applied inside the kernel
  // (wp_window_attn_rope): k and the text q/k passed in are already rotated.
  bool rope = false;
  const int32_t* boxes = nullptr;  // device: t0,t1,h0,h1,w0,w1 per window
  int wt = 0, wh = 0, ww = 0;      // window size
  float rope_theta[21] = {};       // base^(-2i/42)
};

// Tensor-core (tcgen05) bf16 path; head_dim 64 or 128.
int launch_attn_bf16_tc(const AttnCall& c);
// SIMT fp32 path (parity mode); head_dim 64 or 128.
int launch_attn_f32(const AttnCall& c);
// Test hook behind wp_debug_stall_next: the next n tensor-core launches
// stall on purpose (see attn_tc.cu).
void stall_next_launches(int n);

// Device address of the fixed scratch of wp_window_attn_static on the
// current device (looked up, and remembered, on the first call per device).
int static_scratch_address(void** out);

// RoPE angles base^(-2i/42), i < 21, as wp_rope uses them.
void rope_theta(float rope_base, float* theta21);
// Writes L rows of text q and k (bf16, heads x 128 per row, row stride
// txt_stride_B) to qt_out / kt_out (packed rows), rotated with the text
// positions (l, l, l) of wp_rope (the same values); qt and kt are not changed.
int rope_text_copy(const void* qt, const void* kt, int64_t txt_stride_B, void* qt_out, void* kt_out, int L,
                   int heads, float rope_base, cudaStream_t stream);
// Writes the N video rows of k (bf16, heads x 128 per row, layout order of
// `layout`, row stride vid_stride_B) rotated with wp_rope's window-local
// positions (text length L) to k_out (packed rows); k is not changed.
int rope_k_copy(const wp_plan* plan, int layout, const void* k, int64_t vid_stride_B, void* k_out, int heads, int L,
                float rope_base, cudaStream_t stream);

}  // namespace wp
