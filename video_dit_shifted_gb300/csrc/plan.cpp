// Window planner and the host side of the C ABI (errors, plan, upload).
//
// Geometry follows "Window-Aligned Sequence Parallelism (SeedVR2)",
// §Window layouts.  The tables are produced arithmetically (interval
// formulas, then one pass over every window box), not by windowing an arange
// cube; the tests compare them bit for bit with an independent CPU
// implementation that does window an arange cube.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>

#include "wp_internal.h"

namespace wp {

namespace {
thread_local std::string g_err;

constexpr int kMaxTemporalWindow = 30;  // §Window layouts: min(T, 30)

struct Interval {
  int a, b;
};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// [i*w, min((i+1)*w, n)) for i = 0 .. ceil(n/w)-1.
std::vector<Interval> regular_axis(int n, int w) {
  std::vector<Interval> v;
  const int cnt = static_cast<int>(ceil_div(n, w));
  v.reserve(cnt);
  for (int i = 0; i < cnt; ++i) v.push_back({i * w, std::min((i + 1) * w, n)});
  return v;
}

// Interior cuts at floor((2k+1)*w/2) < n (ceil with half_ceil), i.e. every
// regular cut moved by half a window and the ends clipped to 0 and n.  An
// axis that one window covers keeps its single interval.
std::vector<Interval> shifted_axis(int n, int w, bool half_ceil) {
  if (w >= n) return {{0, n}};
  std::vector<Interval> v;
  int start = 0;
  for (int64_t k = 0;; ++k) {
    const int64_t cut = ((2 * k + 1) * static_cast<int64_t>(w) + (half_ceil ? 1 : 0)) / 2;
    if (cut >= n) break;
    if (cut > start) {
      v.push_back({start, static_cast<int>(cut)});
      start = static_cast<int>(cut);
    }
  }
  v.push_back({start, n});
  return v;
}

void build_layout(wp_plan* p, int layout) {
  LayoutTables& L = p->lay[layout];
  std::vector<Interval> ti, hi, wi;
  if (layout == WP_CANONICAL) {
    ti = {{0, p->T}};
    hi = {{0, p->H}};
    wi = {{0, p->W}};
  } else if (layout == WP_REGULAR) {
    ti = regular_axis(p->T, p->wt);
    hi = regular_axis(p->H, p->wh);
    wi = regular_axis(p->W, p->ww);
  } else {
    const bool up = (p->flags & WP_PLAN_HALF_CEIL) != 0;
    ti = shifted_axis(p->T, p->wt, up);
    hi = shifted_axis(p->H, p->wh, up);
    wi = shifted_axis(p->W, p->ww, up);
  }
  L.nwin = static_cast<int>(ti.size() * hi.size() * wi.size());
  L.win_off.assign(L.nwin + 1, 0);
  L.boxes.assign(static_cast<size_t>(L.nwin) * 6, 0);
  L.ids.assign(p->N, 0);
  L.pos.assign(p->N, 0);
  L.max_tokens = 0;
  int64_t r = 0;
  int win = 0;
  const int64_t HW = static_cast<int64_t>(p->H) * p->W;
  for (const Interval& iw : wi) {        // w outermost
    for (const Interval& ih : hi) {
      for (const Interval& it : ti) {    // t innermost
        int32_t* box = &L.boxes[static_cast<size_t>(win) * 6];
        box[0] = it.a; box[1] = it.b; box[2] = ih.a; box[3] = ih.b;
        box[4] = iw.a; box[5] = iw.b;
        L.win_off[win] = static_cast<int32_t>(r);
        for (int t = it.a; t < it.b; ++t)          // row-major (t, h, w)
          for (int h = ih.a; h < ih.b; ++h) {
            const int64_t base = t * HW + static_cast<int64_t>(h) * p->W;
            for (int w = iw.a; w < iw.b; ++w) L.ids[r++] = static_cast<int32_t>(base + w);
          }
        const int n_w = static_cast<int>(r - L.win_off[win]);
        L.max_tokens = std::max(L.max_tokens, n_w);
        ++win;
      }
    }
  }
  L.win_off[L.nwin] = static_cast<int32_t>(r);
  for (int64_t q = 0; q < p->N; ++q) L.pos[L.ids[q]] = static_cast<int32_t>(q);
  for (int b = 0; b < 2; ++b) {
    L.pair_off[b].assign(L.nwin + 1, 0);
    for (int w = 0; w < L.nwin; ++w) {
      const int n_w = L.win_off[w + 1] - L.win_off[w];
      const int vt = static_cast<int>(ceil_div(n_w, kTileM));
      L.pair_off[b][w + 1] = L.pair_off[b][w] + ((vt + b + 1) >> 1);
    }
  }
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Assigns every device-table offset and returns the total size.
size_t layout_device(wp_plan* p) {
  size_t off = 0;
  auto take = [&](size_t n_ints) {
    const size_t at = off;
    off = align256(off + n_ints * sizeof(int32_t));
    return at;
  };
  for (int l = 0; l < kNumLayouts; ++l) {
    const LayoutTables& L = p->lay[l];
    p->dlay[l].win_off = take(L.nwin + 1);
    p->dlay[l].ids = take(p->N);
    p->dlay[l].pair_off[0] = take(L.nwin + 1);
    p->dlay[l].pair_off[1] = take(L.nwin + 1);
    p->dlay[l].boxes = take(static_cast<size_t>(L.nwin) * 6);
  }
  for (int a = 0; a < kNumLayouts; ++a)
    for (int b = 0; b < kNumLayouts; ++b)
      p->perm_off[a][b] = (a == b) ? static_cast<size_t>(-1) : take(p->N);
  return off;
}

bool valid_layout(int layout) { return layout >= 0 && layout < kNumLayouts; }

}  // namespace

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int ok() {
  g_err.clear();
  return WP_OK;
}

int cuda_check(int err, const char* what) {
  if (err == cudaSuccess) return WP_OK;
  return fail(WP_ECUDA, "%s: %s", what, cudaGetErrorString(static_cast<cudaError_t>(err)));
}

int require_uploaded(const wp_plan* plan) {
  if (!plan) return fail(WP_EINVAL, "plan is NULL");
  if (!plan->dev) return fail(WP_ENOTREADY, "plan has not been uploaded (wp_plan_upload)");
  int dev = -1;
  if (int rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return rc;
  if (dev != plan->device)
    return fail(WP_ENOTREADY, "plan was uploaded on device %d, current device is %d",
                plan->device, dev);
  return WP_OK;
}

}  // namespace wp

using namespace wp;

extern "C" {

const char* wp_last_error(void) { return g_err.c_str(); }

int wp_abi_version(void) { return WP_ABI_VERSION; }

int wp_plan_create(int T, int H, int W, int nt, int nh, int nw, wp_plan** out) {
  return wp_plan_create_ex(T, H, W, nt, nh, nw, 0u, out);
}

int wp_plan_create_ex(int T, int H, int W, int nt, int nh, int nw, unsigned flags, wp_plan** out) {
  if (!out) return fail(WP_EINVAL, "out is NULL");
  if (flags & ~WP_PLAN_HALF_CEIL) return fail(WP_EINVAL, "unknown plan flags 0x%x", flags);
  if (T < 1 || H < 1 || W < 1 || nt < 1 || nh < 1 || nw < 1)
    return fail(WP_EINVAL, "grid and window counts must be >= 1 (T=%d H=%d W=%d nt=%d nh=%d nw=%d)",
                T, H, W, nt, nh, nw);
  const int64_t N = static_cast<int64_t>(T) * H * W;
  if (N >= (int64_t(1) << 31)) return fail(WP_EINVAL, "T*H*W = %lld does not fit int32", (long long)N);
  // §Window layouts: 720p-normalised window size.  round() ties to even:
  // nearbyint in the default rounding mode.
  const double scale = std::sqrt(45.0 * 80.0 / (static_cast<double>(H) * static_cast<double>(W)));
  const double rh = std::nearbyint(static_cast<double>(H) * scale);
  const double rw = std::nearbyint(static_cast<double>(W) * scale);
  if (!(rh >= 1.0) || !(rw >= 1.0) || rh > 2e9 || rw > 2e9)
    return fail(WP_EINVAL, "window size rounds to 0 (round(H*scale)=%g, round(W*scale)=%g)", rh, rw);
  wp_plan* p = new (std::nothrow) wp_plan();
  if (!p) return fail(WP_EINVAL, "out of host memory");
  p->T = T; p->H = H; p->W = W; p->nt = nt; p->nh = nh; p->nw = nw;
  p->N = N;
  p->flags = flags;
  p->wh = static_cast<int>(ceil_div(static_cast<int64_t>(rh), nh));
  p->ww = static_cast<int>(ceil_div(static_cast<int64_t>(rw), nw));
  p->wt = static_cast<int>(ceil_div(std::min(T, kMaxTemporalWindow), nt));
  try {
    for (int l = 0; l < kNumLayouts; ++l) build_layout(p, l);
  } catch (const std::bad_alloc&) {
    delete p;
    return fail(WP_EINVAL, "out of host memory building tables for N=%lld", (long long)N);
  }
  p->dev_bytes = layout_device(p);
  *out = p;
  return ok();
}

void wp_plan_destroy(wp_plan* plan) { delete plan; }

int wp_plan_info(const wp_plan* plan, int layout, int64_t* n_tokens, int* nwin, int* wt,
                 int* wh, int* ww, int* max_tokens) {
  if (!plan) return fail(WP_EINVAL, "plan is NULL");
  if (!valid_layout(layout)) return fail(WP_EINVAL, "bad layout %d", layout);
  const LayoutTables& L = plan->lay[layout];
  if (n_tokens) *n_tokens = plan->N;
  if (nwin) *nwin = L.nwin;
  if (wt) *wt = plan->wt;
  if (wh) *wh = plan->wh;
  if (ww) *ww = plan->ww;
  if (max_tokens) *max_tokens = L.max_tokens;
  return ok();
}

int wp_plan_host_tables(const wp_plan* plan, int layout, int32_t* win_off, int32_t* ids,
                        int32_t* boxes) {
  if (!plan) return fail(WP_EINVAL, "plan is NULL");
  if (!valid_layout(layout)) return fail(WP_EINVAL, "bad layout %d", layout);
  const LayoutTables& L = plan->lay[layout];
  if (win_off) std::memcpy(win_off, L.win_off.data(), L.win_off.size() * sizeof(int32_t));
  if (ids) std::memcpy(ids, L.ids.data(), L.ids.size() * sizeof(int32_t));
  if (boxes) std::memcpy(boxes, L.boxes.data(), L.boxes.size() * sizeof(int32_t));
  return ok();
}

int wp_plan_device_bytes(const wp_plan* plan, size_t* bytes) {
  if (!plan || !bytes) return fail(WP_EINVAL, "plan or bytes is NULL");
  *bytes = plan->dev_bytes;
  return ok();
}

int wp_plan_upload(wp_plan* plan, void* dev_buf, size_t bytes, void* stream) {
  if (!plan || !dev_buf) return fail(WP_EINVAL, "plan or dev_buf is NULL");
  if (bytes < plan->dev_bytes)
    return fail(WP_EINVAL, "device buffer too small: %zu < %zu bytes", bytes, plan->dev_bytes);
  if ((reinterpret_cast<uintptr_t>(dev_buf) & 255u) != 0)
    return fail(WP_EUNSUPPORTED, "device buffer must be 256-byte aligned");
  int dev = -1;
  if (int rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return rc;
  // One staging image of every table, then one copy.
  std::vector<char> img;
  try {
    img.assign(plan->dev_bytes, 0);
  } catch (const std::bad_alloc&) {
    return fail(WP_EINVAL, "out of host memory for the upload image");
  }
  auto put = [&](size_t off, const std::vector<int32_t>& v) {
    std::memcpy(img.data() + off, v.data(), v.size() * sizeof(int32_t));
  };
  for (int l = 0; l < kNumLayouts; ++l) {
    const LayoutTables& L = plan->lay[l];
    put(plan->dlay[l].win_off, L.win_off);
    put(plan->dlay[l].ids, L.ids);
    put(plan->dlay[l].pair_off[0], L.pair_off[0]);
    put(plan->dlay[l].pair_off[1], L.pair_off[1]);
    put(plan->dlay[l].boxes, L.boxes);
  }
  for (int a = 0; a < kNumLayouts; ++a)
    for (int b = 0; b < kNumLayouts; ++b) {
      if (a == b) continue;
      int32_t* perm = reinterpret_cast<int32_t*>(img.data() + plan->perm_off[a][b]);
      const std::vector<int32_t>& pos_a = plan->lay[a].pos;
      const std::vector<int32_t>& ids_b = plan->lay[b].ids;
      for (int64_t q = 0; q < plan->N; ++q) perm[q] = pos_a[ids_b[q]];
    }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (int rc = cuda_check(cudaMemcpyAsync(dev_buf, img.data(), img.size(), cudaMemcpyHostToDevice, s),
                          "cudaMemcpyAsync(plan upload)"))
    return rc;
  // The staging image is pageable and dies with this call: wait for the copy.
  if (int rc = cuda_check(cudaStreamSynchronize(s), "cudaStreamSynchronize(plan upload)")) return rc;
  plan->dev = static_cast<char*>(dev_buf);
  plan->device = dev;
  return ok();
}

}  // extern "C"

// ------------------------------------------------------------------------
// Window -> rank assignment and the Plan A exchange tables, for running the
// path on several devices ("Window-Aligned Sequence Parallelism (SeedVR2)",
// §Planner and §Plan A redistribution).  Host only.
namespace {

// LPT: windows by (-token count, window id); each goes to the rank with the
// smallest (assigned tokens, rank id).
void lpt_assign(const LayoutTables& L, int world, std::vector<int32_t>& win_rank,
                std::vector<int64_t>& load) {
  std::vector<int32_t> order(L.nwin);
  for (int w = 0; w < L.nwin; ++w) order[w] = w;
  auto size = [&](int w) { return L.win_off[w + 1] - L.win_off[w]; };
  std::sort(order.begin(), order.end(), [&](int a, int b) {
    return size(a) != size(b) ? size(a) > size(b) : a < b;
  });
  win_rank.assign(L.nwin, 0);
  load.assign(world, 0);
  for (int w : order) {
    int best = 0;
    for (int r = 1; r < world; ++r)
      if (load[r] < load[best]) best = r;  // ties keep the lower rank id
    win_rank[w] = best;
    load[best] += size(w);
  }
}

// Rank-local order: a rank lists its windows in ascending window id, tokens
// in layout order inside each.  For every layout row: owning rank and index
// in that rank's local order.
void local_rows(const LayoutTables& L, const std::vector<int32_t>& win_rank, int world,
                std::vector<int32_t>& rank_of_row, std::vector<int32_t>& local_of_row) {
  const int64_t N = L.win_off[L.nwin];
  rank_of_row.assign(N, 0);
  local_of_row.assign(N, 0);
  std::vector<int64_t> next(world, 0);
  for (int w = 0; w < L.nwin; ++w) {
    const int r = win_rank[w];
    for (int q = L.win_off[w]; q < L.win_off[w + 1]; ++q) {
      rank_of_row[q] = r;
      local_of_row[q] = static_cast<int32_t>(next[r]++);
    }
  }
}

}  // namespace

extern "C" int wp_plan_assign(const wp_plan* plan, int layout, int world, int32_t* win_rank,
                              int64_t* rank_tokens) {
  if (!plan) return fail(WP_EINVAL, "plan is NULL");
  if (!valid_layout(layout)) return fail(WP_EINVAL, "bad layout %d", layout);
  if (world < 1) return fail(WP_EINVAL, "world=%d < 1", world);
  std::vector<int32_t> wr;
  std::vector<int64_t> load;
  lpt_assign(plan->lay[layout], world, wr, load);
  if (win_rank) std::memcpy(win_rank, wr.data(), wr.size() * sizeof(int32_t));
  if (rank_tokens) std::memcpy(rank_tokens, load.data(), load.size() * sizeof(int64_t));
  return ok();
}

extern "C" int wp_plan_exchange(const wp_plan* plan, int src_layout, int dst_layout, int world, int rank,
                                int64_t* counts, int* exchange_required, int32_t* send_rows,
                                int32_t* recv_pos) {
  if (!plan) return fail(WP_EINVAL, "plan is NULL");
  if (!valid_layout(src_layout) || !valid_layout(dst_layout))
    return fail(WP_EINVAL, "bad layout pair (%d -> %d)", src_layout, dst_layout);
  if (world < 1 || rank < 0 || rank >= world) return fail(WP_EINVAL, "world=%d rank=%d", world, rank);
  const LayoutTables& S = plan->lay[src_layout];
  const LayoutTables& D = plan->lay[dst_layout];
  std::vector<int32_t> ws, wd, srank, slocal, drank, dlocal;
  std::vector<int64_t> ls, ld;
  lpt_assign(S, world, ws, ls);
  lpt_assign(D, world, wd, ld);
  local_rows(S, ws, world, srank, slocal);
  local_rows(D, wd, world, drank, dlocal);
  // C[r][d]: rows rank d needs from rank r (same canonical token).
  std::vector<int64_t> C(static_cast<size_t>(world) * world, 0);
  for (int64_t q = 0; q < plan->N; ++q) {
    const int32_t c = D.ids[q];
    const int32_t p = S.pos[c];
    C[static_cast<size_t>(srank[p]) * world + drank[q]]++;
  }
  if (counts) std::memcpy(counts, C.data(), C.size() * sizeof(int64_t));
  if (exchange_required) {
    int any = 0;
    for (int r = 0; r < world; ++r)
      for (int d = 0; d < world; ++d)
        if (r != d && C[static_cast<size_t>(r) * world + d]) any = 1;
    *exchange_required = any;
  }
  // Destination-local order of every rank's rows: walk the destination layout
  // window by window, which visits each destination rank's rows in its local
  // order.
  if (send_rows || recv_pos) {
    std::vector<std::vector<int32_t>> dst_rows(world);  // dst layout rows of each rank, local order
    for (int w = 0; w < D.nwin; ++w)
      for (int q = D.win_off[w]; q < D.win_off[w + 1]; ++q) dst_rows[wd[w]].push_back(q);
    if (send_rows) {
      // For each destination d in rank order: the rows this rank holds that d
      // needs, as this rank's local indices, in d's local order.
      int64_t k = 0;
      for (int d = 0; d < world; ++d)
        for (int32_t q : dst_rows[d]) {
          const int32_t p = S.pos[D.ids[q]];
          if (srank[p] == rank) send_rows[k++] = slocal[p];
        }
    }
    if (recv_pos) {
      // Received segments arrive in source-rank order; each segment is in
      // this rank's local order.  recv_pos[k] = local position of row k.
      int64_t k = 0;
      for (int r = 0; r < world; ++r)
        for (int32_t q : dst_rows[rank]) {
          const int32_t p = S.pos[D.ids[q]];
          if (srank[p] == r) recv_pos[k++] = dlocal[q];
        }
    }
  }
  return ok();
}
