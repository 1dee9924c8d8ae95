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
  int64_t vid_stride_B;
  const void *qt, *kt, *vt;
  int64_t txt_stride_B;
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
};

// Tensor-core (tcgen05) bf16 path; head_dim 64 or 128.
int launch_attn_bf16_tc(const AttnCall& c);
// SIMT fp32 path (parity mode); head_dim 64 or 128.
int launch_attn_f32(const AttnCall& c);

}  // namespace wp
