// Internal declarations shared by the translation units of libwp.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "wp.h"

namespace wp {

// Record a one-line error message (printf-style) for wp_last_error() and
// return `code`.
int fail(int code, const char* fmt, ...);
// Clear the thread's error message and return WP_OK.
int ok();
// Check a cudaError_t (as int); on failure record it and return WP_ECUDA.
int cuda_check(int err, const char* what);

constexpr int kNumLayouts = 3;
// Query tile height of the tensor-core attention kernel; the plan's work-split
// prefix tables count query tiles of this many rows.
constexpr int kTileM = 128;

struct LayoutTables {
  int nwin = 0;
  int max_tokens = 0;
  std::vector<int32_t> win_off;   // nwin+1
  std::vector<int32_t> boxes;     // nwin*6: t0,t1,h0,h1,w0,w1
  std::vector<int32_t> ids;       // N: layout row -> canonical id
  std::vector<int32_t> pos;       // N: canonical id -> layout row
  // pair_off[b][w] = sum_{w' < w} (ceil(n_w'/kTileM) + b + 1) >> 1 for
  // b = 0, 1.  With tt text tiles, window w holds
  // (ceil(n_w/kTileM) + tt + 1) >> 1 pairs of query tiles, and their prefix
  // over windows is pair_off[tt & 1][w] + w * (tt >> 1).
  std::vector<int32_t> pair_off[2];
};

// Offsets (bytes) of each table inside the caller's device buffer.
struct DeviceLayout {
  size_t win_off = 0, ids = 0, pair_off[2] = {0, 0}, boxes = 0;
};

}  // namespace wp

struct wp_plan {
  int T = 0, H = 0, W = 0, nt = 0, nh = 0, nw = 0;
  int wt = 0, wh = 0, ww = 0;
  int64_t N = 0;
  unsigned flags = 0;  // WP_PLAN_HALF_CEIL
  wp::LayoutTables lay[wp::kNumLayouts];
  // device side (valid once uploaded)
  wp::DeviceLayout dlay[wp::kNumLayouts];
  size_t perm_off[wp::kNumLayouts][wp::kNumLayouts] = {};
  size_t dev_bytes = 0;
  char* dev = nullptr;
  int device = -1;
};

namespace wp {

// Validates that the plan was uploaded on the current device.
int require_uploaded(const wp_plan* plan);

template <typename T>
inline const T* dev_ptr(const wp_plan* p, size_t off) {
  return reinterpret_cast<const T*>(p->dev + off);
}

inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace wp
