// Window attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA), bf16
// in, fp32 accumulation.
//
// What it computes ("Window-Aligned Sequence Parallelism (SeedVR2)",
// §SeedVR2 integration and §Text stream): for every window w and head h, one
// full attention over the segment [video rows of w ; text rows]; video
// results are scattered to their canonical rows, text results T_w are written
// in fp32 for the ordered mean in attn.cu.
//
// Design.  Work items are pairs of 128-row query tiles of one (window, head);
// a persistent grid of one CTA per SM takes them from a global counter (the
// producer warp draws the next index and hands it to every role through a
// ring in shared memory), so the CTAs finish within a fraction of an item of
// each other; items of one (window, head) are handed out one after the other,
// so CTAs busy at the same time share K/V tiles through L2.  Roles inside a
// CTA (320 threads; 384 in the RoPE kernels):
//   warps 0-3   softmax + epilogue for query tile 0, warps 4-7 for tile 1:
//               one thread per query row (TMEM lane); one 128-column TMEM
//               load of S per tile, 2^x in the log2 domain against the
//               running max, P written back over S as packed bf16; O is
//               rescaled in TMEM only when a row max grows by more than
//               2^8 (the final O / l is exact either way), and the row max
//               is taken only when the row sum shows that some p may exceed
//               2^8 (a sum <= 2^8 proves every p <= 2^8); the epilogue
//               scatters video rows to their output rows and writes text
//               rows as fp32 T_w, with 32-byte stores when the output allows
//               it (a thread writes its own row, so each store instruction
//               touches 32 rows: 32-byte stores write whole sectors with
//               half the instructions, +5% end to end);
//   warp 8      TMA producer (whole warp, one elected lane issues): both Q
//               tiles of an item, then the item's K and V tiles (video
//               tiles of the window, then text tiles) in per-step payloads
//               [K_0], [V_0, K_1], [V_1, K_2], ... into two K and two V
//               slots, 128-byte swizzled, 64 columns per box; the next
//               item's loads start as soon as slots free up;
//   warp 9      TMEM allocator (512 columns: S0, S1, O0, O1) and MMA issuer:
//               S_i = Q_i K_j^T (both operands in shared memory) and
//               O_i += P_i V_j (P from TMEM, V MN-major);
//   warps 10-11 (RoPE kernels only) the window-local RoPE of the video Q
//               tiles in shared memory between the TMA and the MMA; the
//               RoPE kernels read K already rotated (a separate pass writes
//               every video K row once, rotated, to the workspace), so K/V
//               payloads go from the TMA to the MMA as in the plain kernels.
// The two query tiles share every K/V tile, and the issue order
// S0(j) S1(j) PV0(j) S0(j+1) PV1(j) S1(j+1) ... lets one tile's softmax run
// while the tensor core works on the other.  The issuer is the whole warp 9,
// converged, with tcgen05.mma and tcgen05.commit predicated on one elected
// lane: measured on this part, a barrier wait next to a commit costs ~27
// cycles of tensor-pipe time when one lane runs the loop inside a divergent
// branch and ~4 when the warp runs it converged (+9% end to end), while
// straight-line arithmetic between MMAs is free.  The loop is kept short all
// the same: the wait fast path is inlined, descriptors advance by constants,
// and the tile index is a compile-time constant.
//
// Masking: a segment is ragged, so the last video K/V tile of a window may
// run into the next window's rows (or past N, where TMA fills zeros).  Those
// key columns get probability exactly 0 and are left out of the max.  Query
// rows past the window are computed but never stored.
//
// Every mbarrier wait is bounded (kWaitTimeoutNs); on expiry the kernel sets
// WP_ETIMEOUT in the status word, raises a CTA-wide abort flag, drains its
// own TMA and MMA work and frees TMEM before returning.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <type_traits>

#include "attn_internal.h"
#include "tmem_io.cuh"

namespace wp {
namespace {

constexpr int kBM = 128;  // query rows per tile (TMEM lanes)
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kThreads = 320;       // warps 0-7 softmax, 8 TMA, 9 MMA
constexpr int kRopeThreads = 384;   // RoPE kernels: + warps 10-11 rotating Q tiles
constexpr int kRopeWarp0 = 10;
constexpr int kRopePairs = 21;      // rotated pairs per axis at head_dim 128 (42 channels)
constexpr int kRopeStride = 22;     // table entries per axis position (21 + 1 pad: 16-byte pairs)
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kTmemCols = 512;
static_assert(kBM == kTileM, "plan tables count tiles of kTileM rows");

// Shared-memory layout.  Q and K are bf16 or, in the e4m3 kernels, one byte
// per element; V is always bf16.  Every tile is stored as 128-row x 128-byte
// boxes (128-byte swizzle), one box per 128 bytes of a row.
template <int HD, bool kFp8 = false>
struct Cfg {
  static constexpr int kHalves = HD / 64;               // V: 64-column (128 B) boxes per row
  static constexpr int kQKElem = kFp8 ? 1 : 2;          // bytes per Q/K element
  static constexpr int kQKBoxes = HD * kQKElem / 128;   // Q/K: 128-byte boxes per row
  static constexpr int kQKBoxCols = 128 / kQKElem;      // Q/K: elements per box row
  static constexpr int kBoxBytes = 128 * 128;           // one 128-row x 128-byte box
  static constexpr int kQKTileBytes = kBM * HD * kQKElem;  // a Q or K tile
  static constexpr int kTileBytes = kBM * HD * 2;       // a V tile
  static constexpr int kQ = 0;                          // Q tile i at kQ + i*kQKTileBytes
  static constexpr int kK = 2 * kQKTileBytes;           // K stage s at kK + s*kQKTileBytes
  static constexpr int kV = 4 * kQKTileBytes;           // V stage s at kV + s*kTileBytes
  static constexpr int kBar = kV + 2 * kTileBytes;
  static constexpr int kTab = kBar + 256;          // RoPE kernels: cos/sin table
  static constexpr int kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + HD;
};
// Both head dims request the HD=128 footprint so that exactly one CTA (and
// one 512-column TMEM allocation) lives on an SM.
constexpr int kSmemBytes = Cfg<128>::kBar + 256 + 1024;
constexpr size_t kRopeMaxSmem = 227 * 1024;  // dynamic shared memory per CTA on sm_103a

struct Barriers {
  uint64_t q_full, q_empty;
  uint64_t pl_full[2], pl_empty[2];  // K/V payload slots (see the producer)
  uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
  uint64_t q_ready;                  // RoPE kernels: Q rotated
  uint64_t item_full[4], item_empty[4];  // ring of work-item indices (see the producer)
  uint64_t mma_done;
  uint64_t stall;                    // test hook: a barrier nothing arrives at
  uint32_t tmem_base;
  int abort_flag;
  int item_idx[4];
};
static_assert(sizeof(Barriers) <= 256, "barrier block");

struct TcParams {
  const int32_t* win_off;
  const int32_t* ids;       // output row of each input row (NULL: the same row)
  const int32_t* pair_off;  // pair_off[text_tiles & 1]
  int pair_add;             // text_tiles >> 1
  int nwin, L, heads, text_tiles, total_pairs;
  __nv_bfloat16* o_vid;
  int64_t o_stride;  // elements
  int64_t n_rows;    // rows of o_vid (N): every table entry must lie below it
  float* partial;
  int* status;
  int* counter;  // next work item (zero at launch)
  float scale_log2;
  int stall;   // test hook: CTA 0's MMA warp waits on `stall` (its bounded wait expires)
  int vid_v8;  // o_vid and o_stride are 32-byte aligned: 32-byte stores
  int txt_v8;  // partial is 32-byte aligned: 32-byte stores
  // RoPE kernels only: window boxes (t0,t1,h0,h1,w0,w1 per window), the
  // window size (rows of the cos/sin table per axis) and theta_i.
  const int32_t* boxes;
  int wt, wh, ww;
  float theta[kRopePairs];
};

// ------------------------------------------------------------ PTX helpers --
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Slow path of wait_phase: poll with a time limit.  Out of line, so that
// the hot path stays a single try_wait (a call costs ~200 cycles of
// register save/restore, which the MMA issue loop cannot afford).
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             int* status) {
  const uint64_t t0 = globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kWaitTimeoutNs) {
        *abort_flag = 1;
        atomicCAS(status, 0, WP_ETIMEOUT);
        return false;
      }
    }
  }
}

// Bounded wait for the phase with the given parity.  Returns false if the
// CTA is aborting (flag set by any thread) or this wait expired (then it
// sets the flag and the status word).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_phase_slow(bar, parity, abort_flag, status);
}

// Bounded wait that ignores the abort flag (used while draining).
__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > kWaitTimeoutNs) return;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x,
                                            int y) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (layout code 2 in bits
// 61-63), descriptor version 1 (bits 46-47), base offset 0 (every swizzle
// atom is 1024-byte aligned).  lbo/sbo in bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFF) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (uint64_t(1) << 46) |
         (uint64_t(2) << 61);
}

// Instruction descriptor for kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9, 10-12 = 1), B transposed (MN-major) via bit 16, N>>3 in bits
// 17-22, M>>4 in bits 24-28.
constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
// Instruction descriptor for kind::f8f6f4 with A and B both e4m3 (format
// code 0 in bits 7-9 and 10-12), both K-major, D fp32.
constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// MMA and commit wrappers: called by all 32 lanes of a converged warp; one
// elected lane issues the instruction.
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_ss_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void st_v8(void* dst, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  uint32_t u;
  memcpy(&u, &v, 4);
  return u;
}

// ------------------------------------------------------------------ kernel --
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Row max over the first `valid` of 128 scores (valid == 128: no masking).
template <bool kFull>
__device__ __forceinline__ float row_max(const uint32_t (&s)[128], int valid) {
  float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
  for (int e = 0; e < 128; e += 8) {
    float x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      x[u] = (kFull || e + u < valid) ? __uint_as_float(s[e + u]) : -INFINITY;
    m0 = fmax3(m0, x[0], x[1]);
    m1 = fmax3(m1, x[2], x[3]);
    m2 = fmax3(m2, x[4], x[5]);
    m3 = fmax3(m3, x[6], x[7]);
  }
  return fmaxf(fmax3(m0, m1, m2), m3);
}

// p = 2^(s*scale_log2 - m) for the valid columns (0 elsewhere), packed to
// bf16 pairs; returns the fp32 row sum of p.
template <bool kFull>
__device__ __forceinline__ float row_exp(const uint32_t (&s)[128], int valid, float scale_log2, float m,
                                         uint32_t (&pk)[64]) {
  const uint64_t sc = f2_pack(scale_log2, scale_log2);
  const uint64_t nm = f2_pack(-m, -m);
  uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
  for (int e = 0; e < 64; ++e) {
    float x0, x1;
    f2_unpack(ffma2(f2_pack(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])), sc, nm), x0, x1);
    float p0 = ex2(x0), p1 = ex2(x1);
    if (!kFull) {
      p0 = 2 * e < valid ? p0 : 0.f;
      p1 = 2 * e + 1 < valid ? p1 : 0.f;
    }
    acc[e & 3] = fadd2(acc[e & 3], f2_pack(p0, p1));
    pk[e] = pack_bf16(p0, p1);
  }
  float a0, a1, b0, b1;
  f2_unpack(fadd2(acc[0], acc[1]), a0, a1);
  f2_unpack(fadd2(acc[2], acc[3]), b0, b1);
  return (a0 + a1) + (b0 + b1);
}

// Rotate one bf16 pair (x0 low, x1 high) by the angle whose cosine and
// sine come as the bf16 pairs cc = (c, c) and ns = (-s, s):
// (x0 c - x1 s, x1 c + x0 s).
__device__ __forceinline__ uint32_t rot_bf16x2(uint32_t v, uint32_t cc, uint32_t ns) {
  uint32_t sw, t, r;
  asm("prmt.b32 %0, %1, %1, 0x1032;" : "=r"(sw) : "r"(v));
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(t) : "r"(sw), "r"(ns));
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(v), "r"(cc), "r"(t));
  return r;
}

// Window-local RoPE, in place, of the first `nrows` rows of a 128-row x 128
// column bf16 tile in shared memory, laid out as TMA wrote it (two 128-byte
// swizzled boxes of 64 columns: chunk c of row r at r*128 + (c ^ (r&7))*16).
// Row r is the window-local token tok0 + r, at (dt, dh, dw) in the window's
// (bh x bw) row-major order; channel pair i of axis block a (42 channels
// each: t, h, w) turns by pos_a * theta_i, pos = (L + dt, dh, dw); pair 63
// (channels 126, 127) is left alone.  tab (a shared-memory address) holds,
// per axis position and i, (c, c) and (-s, s) as bf16 pairs, kRopeStride
// entries of 8 bytes per position so that pairs i and i + 1 load as one
// 16-byte word: rows [0, wt) for t, then wh rows for h, then ww rows for w.
// inv_bhw = 1 / (bh bw) and inv_bw = 1 / bw turn the divisions into
// multiplies.  64 threads, rows rt and rt + 64.
__device__ __forceinline__ void rope_tile(uint32_t tile, int tok0, int nrows, int bh, int bw, int wt, int wh,
                                          uint32_t tab, float inv_bhw, float inv_bw, int rt) {
  const int bhw = bh * bw;
  for (int r = rt; r < nrows; r += 64) {
    const int tok = tok0 + r;
    // exact: (tok + 1/2) / bhw is at least 1/(2 bhw) away from an integer
    const int dt = __float2int_rz((static_cast<float>(tok) + 0.5f) * inv_bhw), rem = tok - dt * bhw;
    const int dh = __float2int_rz((static_cast<float>(rem) + 0.5f) * inv_bw), dw = rem - dh * bw;
    const uint32_t tr[3] = {tab + dt * (kRopeStride * 8), tab + (wt + dh) * (kRopeStride * 8),
                            tab + (wt + wh + dw) * (kRopeStride * 8)};
    const uint32_t row = tile + r * 128;
    // All 16 chunks of the row in flight at once, then rotate, then store.
    uint32_t v[16][4];
#pragma unroll
    for (int cc = 0; cc < 16; ++cc)
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(v[cc][0]), "=r"(v[cc][1]), "=r"(v[cc][2]), "=r"(v[cc][3])
                   : "r"(row + (cc >> 3) * (128 * 128) + (((cc & 7) ^ (r & 7)) << 4))
                   : "memory");
#pragma unroll
    for (int a = 0; a < 3; ++a)
#pragma unroll
      for (int i = 0; i < kRopePairs; i += 2) {  // pairs i and i + 1 of axis a: one 16-byte load
        uint32_t e0, e1, e2, e3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(e0), "=r"(e1), "=r"(e2), "=r"(e3)
                     : "r"(tr[a] + i * 8)
                     : "memory");
        const int w0 = a * kRopePairs + i;
        v[w0 >> 2][w0 & 3] = rot_bf16x2(v[w0 >> 2][w0 & 3], e0, e1);
        if (i + 1 < kRopePairs) {
          const int w1 = w0 + 1;
          v[w1 >> 2][w1 & 3] = rot_bf16x2(v[w1 >> 2][w1 & 3], e2, e3);
        }
      }
#pragma unroll
    for (int cc = 0; cc < 16; ++cc)
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (cc >> 3) * (128 * 128) +
                                                                    (((cc & 7) ^ (r & 7)) << 4)),
                   "r"(v[cc][0]), "r"(v[cc][1]), "r"(v[cc][2]), "r"(v[cc][3])
                   : "memory");
  }
}

// One work item: a pair of 128-row query tiles of one (window, head).
struct Item {
  int h, w, a, n_w, vt, nkv, t0, nq;
};

__device__ __forceinline__ Item decode_item(const TcParams& p, int it) {
  Item x;
  const int pidx = it % p.total_pairs;
  x.h = it / p.total_pairs;
  int lo = 0, hi = p.nwin - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.pair_off + mid) + mid * p.pair_add <= pidx) lo = mid; else hi = mid - 1;
  }
  x.w = lo;
  x.a = __ldg(p.win_off + lo);
  x.n_w = __ldg(p.win_off + lo + 1) - x.a;
  x.vt = (x.n_w + kBN - 1) / kBN;  // video tiles (queries and keys alike)
  x.nkv = x.vt + p.text_tiles;
  x.t0 = 2 * (pidx - (__ldg(p.pair_off + lo) + lo * p.pair_add));
  x.nq = min(2, x.nkv - x.t0);
  return x;
}

// Persistent: CTA b processes items b, b + gridDim.x, b + 2*gridDim.x, ...
// (items = query-tile pairs x heads, pairs of one (window, head) adjacent,
// so the CTAs working at the same time share K/V tiles through L2).  Every
// role walks the same item sequence; barrier phases follow running counters
// that all roles advance identically.
// 10 warps put 3 warps on one SM sub-partition (16K registers each), which
// caps a thread at 168 registers.
template <int HD, bool kRope, bool kFp8>
__global__ void __launch_bounds__(kRope ? kRopeThreads : kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_qt,
                   const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_vt,
                   const TcParams p) {
  static_assert(!(kRope && kFp8), "no RoPE on e4m3 tiles");
  using C = Cfg<HD, kFp8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 1024-aligned for 128 B swizzle
  uint8_t* smem = smem_raw + (base - raw);
  Barriers* bars = reinterpret_cast<Barriers*>(smem + C::kBar);
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.total_pairs * p.heads;

  const uint32_t bq_full = smem_addr(&bars->q_full), bq_empty = smem_addr(&bars->q_empty);
  auto bar = [](uint64_t& b) { return smem_addr(&b); };

  if (threadIdx.x == 0) {
    mbar_init(bq_full, 1);
    mbar_init(bq_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(bars->pl_full[s]), 1);
      mbar_init(bar(bars->pl_empty[s]), 1);
      mbar_init(bar(bars->s_full[s]), 1);
      mbar_init(bar(bars->p_full[s]), 128);
      mbar_init(bar(bars->o_full[s]), 1);
      mbar_init(bar(bars->o_empty[s]), 128);
    }
    mbar_init(bar(bars->mma_done), 1);
    mbar_init(bar(bars->stall), 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(bar(bars->item_full[s]), 1);
      // one arrival per consumer warp: MMA, 8 softmax (+ 2 RoPE)
      mbar_init(bar(bars->item_empty[s]), kRope ? 11 : 9);
    }
    if (kRope) {
      mbar_init(bar(bars->q_ready), 64);
    }
    // A CTA of this launch already failed: skip the work so that a broken
    // launch ends quickly instead of timing out CTA after CTA.
    bars->abort_flag = *reinterpret_cast<volatile int*>(p.status) != 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (bars->abort_flag) return;
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&bars->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  // Work items are handed out dynamically: the producer warp takes the next
  // item index from a global counter and publishes it in a ring of four
  // slots (item_full / item_empty); every role walks the same sequence, -1
  // ending it.  Items of one (window, head) are still taken one after the
  // other, so CTAs working at the same time share K/V tiles through L2.
  auto take_item = [&](int u, bool& good) -> int {
    const int slot = u & 3;
    good = __all_sync(0xffffffffu, wait_phase(bar(bars->item_full[slot]), (u >> 2) & 1, abort_flag, p.status));
    if (!good) return -1;
    const int it = *reinterpret_cast<volatile int*>(&bars->item_idx[slot]);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(bars->item_empty[slot]));
    return it;
  };

  if (warp == kProducerWarp) {
    // ======================= TMA producer ===============================
    {
      // K/V tiles travel in "payloads", one per MMA step, so that the MMA
      // thread waits once and releases once per step: an item starts with
      // [K_0]; step j of the item brings [V_j, K_{j+1}] (K only while the
      // item has a next tile).  Payload e fills K slot e&1 and V slot e&1 and
      // may load once payload e-2 is released, i.e. once the MMAs of the
      // step that consumed it have completed.
      int e = 0;  // payloads issued
      int k = 0;  // items whose Q load was issued
      bool good = true;
      for (int u = 0; good; ++u) {
        const int slot = u & 3;
        if (u >= 4 &&
            !(good = wait_phase(bar(bars->item_empty[slot]), ((u >> 2) - 1) & 1, abort_flag, p.status)))
          break;
        int it = 0;
        if (lane == 0) it = atomicAdd(p.counter, 1);
        it = __shfl_sync(0xffffffffu, it, 0);
        if (it >= n_items) it = -1;
        if (lane == 0) {
          bars->item_idx[slot] = it;
          mbar_arrive(bar(bars->item_full[slot]));
        }
        __syncwarp();
        if (it < 0) break;
        const Item x = decode_item(p, it);
        // Q smem is free once the previous item's last Q K^T has completed.
        if (k > 0 && !(good = wait_phase(bq_empty, (k - 1) & 1, abort_flag, p.status))) break;
        mbar_expect_tx(bq_full, x.nq * C::kQKTileBytes);
        for (int i = 0; i < x.nq; ++i) {
          const int t = x.t0 + i;
          const CUtensorMap* map = t < x.vt ? &tm_q : &tm_qt;
          const int row = t < x.vt ? x.a + t * kBM : (t - x.vt) * kBM;
          for (int hf = 0; hf < C::kQKBoxes; ++hf)
            tma_load_2d(base + C::kQ + i * C::kQKTileBytes + hf * C::kBoxBytes, map, bq_full,
                        x.h * HD + hf * C::kQKBoxCols, row);
        }
        ++k;
        auto tile_row = [&](int j) { return j < x.vt ? x.a + j * kBN : (j - x.vt) * kBN; };
        for (int pl = 0; pl <= x.nkv; ++pl, ++e) {
          const int slot = e & 1;
          if (e >= 2 && !(good = wait_phase(bar(bars->pl_empty[slot]), ((e >> 1) - 1) & 1, abort_flag, p.status)))
            break;
          const int kt = pl;      // K tile of this payload (none when pl == nkv)
          const int vt_ = pl - 1;  // V tile of this payload (none when pl == 0)
          const uint32_t fb = bar(bars->pl_full[slot]);
          mbar_expect_tx(fb, (kt < x.nkv ? C::kQKTileBytes : 0) + (vt_ >= 0 ? C::kTileBytes : 0));
          if (vt_ >= 0)
            for (int hf = 0; hf < C::kHalves; ++hf)
              tma_load_2d(base + C::kV + slot * C::kTileBytes + hf * C::kBoxBytes, vt_ < x.vt ? &tm_v : &tm_vt,
                          fb, x.h * HD + hf * 64, tile_row(vt_));
          if (kt < x.nkv)
            for (int hf = 0; hf < C::kQKBoxes; ++hf)
              tma_load_2d(base + C::kK + slot * C::kQKTileBytes + hf * C::kBoxBytes, kt < x.vt ? &tm_k : &tm_kt,
                          fb, x.h * HD + hf * C::kQKBoxCols, tile_row(kt));
        }
      }
      if (*abort_flag) {
        // Let every copy this thread started land before the CTA exits.
        if (k > 0) drain_wait(bq_full, (k - 1) & 1);
        for (int u = e - 2; u < e; ++u)
          if (u >= 0) drain_wait(bar(bars->pl_full[u & 1]), (u >> 1) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ======================= MMA issuer (whole warp, converged) ==========
    {
      constexpr uint32_t kIdescQK = kFp8 ? idesc_e4m3(kBM, kBN) : idesc_bf16(kBM, kBN, false);
      constexpr uint32_t kIdescPV = idesc_bf16(kBM, HD, true);
      // Descriptors are built once per tile and advanced by constant offsets
      // (the start-address field holds address >> 4 and never carries out of
      // its 14 bits for a shared-memory address), keeping the issue loop short.
      auto issue_qk = [&](int i, int s) {
        const uint32_t dS = tmem + (i ? C::kColS1 : C::kColS0);
        const uint64_t qd = sw128_desc(base + C::kQ + i * C::kQKTileBytes, 16, 1024);
        const uint64_t kd = sw128_desc(base + C::kK + s * C::kQKTileBytes, 16, 1024);
        // one MMA per 32 bytes of the head dimension (16 bf16 or 32 e4m3
        // elements): 4 per 128-byte box
#pragma unroll
        for (int kk = 0; kk < HD * C::kQKElem / 32; ++kk) {
          const uint32_t off16 = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          if constexpr (kFp8)
            mma_ss_f8(dS, qd + off16, kd + off16, kIdescQK, kk > 0);
          else
            mma_ss(dS, qd + off16, kd + off16, kIdescQK, kk > 0);
        }
      };
      auto issue_pv = [&](int i, int s, bool first) {
        const uint32_t dO = tmem + (i ? C::kColO1 : C::kColO0);
        const uint32_t aP = tmem + (i ? C::kColS1 : C::kColS0);
        const uint64_t vd = sw128_desc(base + C::kV + s * C::kTileBytes, C::kBoxBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(dO, aP + kk * 8, vd + ((kk * 2048) >> 4), kIdescPV, (!first || kk > 0) ? 1u : 0u);
      };
      int k = 0;                  // items
      int cs0 = 0, cs1 = 0;       // tiles per softmax warpgroup (s_full / p_full phases)
      int co0 = 0, co1 = 0;       // items per softmax warpgroup (o_full / o_empty phases)
      bool good = true;
      // One query tile's share of step j: O_i += P_i V_j, then S_i = Q_i K_{j+1}^T.
      // The tile index is a compile-time constant so that every phase counter
      // and TMEM address stays in registers.
      auto tile_step = [&](auto I, int j, int s, int sn, bool more, int cs, int co) -> bool {
        constexpr int i = decltype(I)::value;
        if (!wait_phase(bar(bars->p_full[i]), (cs + j) & 1, abort_flag, p.status)) return false;
        // O_i is overwritten by this item's first P V: the previous item's
        // epilogue must have read it out.
        if (j == 0 && co > 0 && !wait_phase(bar(bars->o_empty[i]), (co - 1) & 1, abort_flag, p.status))
          return false;
        tc_fence_after();
        issue_pv(i, s, j == 0);
        if (more) {
          issue_qk(i, sn);
          mma_commit(bar(bars->s_full[i]));
        } else {
          mma_commit(bar(bars->o_full[i]));
        }
        return true;
      };
      int e = 0;  // payloads consumed (see the producer)
      for (int u = 0; good; ++u, ++k) {
        const int it = take_item(u, good);
        if (it < 0) break;
        // Test hook (wp_debug_stall_next): wait for a phase that never
        // completes, so that the bounded wait expires and the CTA winds down.
        if (p.stall && blockIdx.x == 0 && k == 0 &&
            !(good = wait_phase(bar(bars->stall), 0, abort_flag, p.status)))
          break;
        const Item x = decode_item(p, it);
        // payload [K_0]
        // (RoPE kernels: Q once warps 10-11 have rotated it.)
        if (!(good = wait_phase(kRope ? bar(bars->q_ready) : bq_full, k & 1, abort_flag, p.status) &&
                     wait_phase(bar(bars->pl_full[e & 1]), (e >> 1) & 1, abort_flag, p.status)))
          break;
        tc_fence_after();
        issue_qk(0, e & 1);
        mma_commit(bar(bars->s_full[0]));
        if (x.nq > 1) {
          issue_qk(1, e & 1);
          mma_commit(bar(bars->s_full[1]));
        }
        if (x.nkv == 1) mma_commit(bq_empty);
        mma_commit(bar(bars->pl_empty[e & 1]));
        ++e;
        for (int j = 0; j < x.nkv; ++j, ++e) {
          const int s = e & 1;  // payload [V_j, K_{j+1}]
          const bool more = j + 1 < x.nkv;
          if (!(good = wait_phase(bar(bars->pl_full[s]), (e >> 1) & 1, abort_flag, p.status))) break;
          if (!(good = tile_step(std::integral_constant<int, 0>{}, j, s, s, more, cs0, co0))) break;
          if (x.nq > 1 && !(good = tile_step(std::integral_constant<int, 1>{}, j, s, s, more, cs1, co1)))
            break;
          mma_commit(bar(bars->pl_empty[s]));
          if (j + 2 == x.nkv) mma_commit(bq_empty);  // the Q K^T just issued was the item's last
        }
        cs0 += x.nkv;
        co0 += 1;
        if (x.nq > 1) {
          cs1 += x.nkv;
          co1 += 1;
        }
      }
      // All MMAs this warp issued must finish before TMEM is freed.
      mma_commit(bar(bars->mma_done));
      drain_wait(bar(bars->mma_done), 0);
    }
    __syncwarp();
  } else if (kRope && warp >= kRopeWarp0) {
    // ======================= RoPE (warps 10-11, RoPE kernels) ===========
    // The window-local RoPE of the item's video Q tiles, in shared memory
    // between the TMA landing (q_full) and the MMA (q_ready).  Text Q tiles
    // arrive already rotated.  The producer loads the next item's Q only
    // after the MMA's last Q K^T of this one, which follows q_ready, so these
    // waits are never more than one phase behind.
    const int rt = threadIdx.x - kRopeWarp0 * 32;  // 0..63
    uint2* tab = reinterpret_cast<uint2*>(smem + C::kTab);
    const uint32_t tab_s = base + C::kTab;
    const int ntab = p.wt + p.wh + p.ww;
    for (int e = rt; e < ntab * kRopePairs; e += 64) {
      const int row = e / kRopePairs, i = e - row * kRopePairs;
      const int pos = row < p.wt ? p.L + row : (row < p.wt + p.wh ? row - p.wt : row - p.wt - p.wh);
      float sn, cs;
      sincosf(static_cast<float>(pos) * p.theta[i], &sn, &cs);
      tab[row * kRopeStride + i] = make_uint2(pack_bf16(cs, cs), pack_bf16(-sn, sn));
    }
    asm volatile("bar.sync 1, 64;" ::: "memory");
    int k = 0;
    bool good = true;
    for (int u = 0; good; ++u, ++k) {
      const int it = take_item(u, good);
      if (it < 0) break;
      const Item x = decode_item(p, it);
      const int bh = __ldg(p.boxes + 6 * x.w + 3) - __ldg(p.boxes + 6 * x.w + 2);
      const int bw = __ldg(p.boxes + 6 * x.w + 5) - __ldg(p.boxes + 6 * x.w + 4);
      const float inv_bhw = 1.f / static_cast<float>(bh * bw), inv_bw = 1.f / static_cast<float>(bw);
      if (!(good = wait_phase(bq_full, k & 1, abort_flag, p.status))) break;
      for (int i = 0; i < x.nq; ++i) {
        const int t = x.t0 + i;
        if (t < x.vt)
          rope_tile(base + C::kQ + i * C::kQKTileBytes, t * kBM, min(kBM, x.n_w - t * kBM), bh, bw, p.wt, p.wh, tab_s,
                    inv_bhw, inv_bw, rt);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(bar(bars->q_ready));
    }
  } else {
    // ======================= softmax + epilogue (warps 0-7) =============
    const int i = warp >> 2;        // query tile of this warpgroup
    const int quarter = warp & 3;   // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + (i == 0 ? C::kColS0 : C::kColS1) + lane_off;
    const uint32_t tO = tmem + (i == 0 ? C::kColO0 : C::kColO1) + lane_off;
    const uint32_t bs = bar(bars->s_full[i]), bp = bar(bars->p_full[i]);
    int cs = 0, co = 0;
    bool good = true;
    for (int u = 0; good; ++u) {
      const int it = take_item(u, good);
      if (it < 0) break;
      const Item x = decode_item(p, it);
      if (i >= x.nq) continue;
      float m_run = 0.f, l_run = 0.f;
      for (int j = 0; j < x.nkv; ++j) {
        const int valid = j < x.vt ? min(kBN, x.n_w - j * kBN) : min(kBN, p.L - (j - x.vt) * kBN);
        good = __all_sync(0xffffffffu, wait_phase(bs, (cs + j) & 1, abort_flag, p.status));
        if (!good) break;
        tc_fence_after();
        uint32_t s[128];
        tmem_ld_x128(tS, s);
        const bool full = valid == kBN;
        // Lazy rescale: O and l move to a new max only when some row's max
        // grew by more than 2^8 over the running max m_run; otherwise every
        // p <= 2^8, which fp32 and bf16 hold exactly enough, and the final
        // O / l is unchanged.  The exponentials are taken against m_run
        // first (for an item's first tile, the max of its first 16 scores);
        // a row sum <= 2^8 proves every p <= 2^8, and only when some row's
        // sum is larger (or not finite) is S read again, the true max taken
        // and the pass redone.
        if (j == 0) {
          float m16 = __uint_as_float(s[0]);
#pragma unroll
          for (int c = 1; c < 16; ++c) m16 = fmaxf(m16, (full || c < valid) ? __uint_as_float(s[c]) : m16);
          m_run = m16 * p.scale_log2;
        }
        bool rescale = false;
        float alpha = 1.f;
        uint32_t pk[64];
        float l_tile = full ? row_exp<true>(s, valid, p.scale_log2, m_run, pk)
                            : row_exp<false>(s, valid, p.scale_log2, m_run, pk);
        if (__any_sync(0xffffffffu, !(l_tile <= 256.f))) {
          tmem_ld_x128(tS, s);
          const float mx = (full ? row_max<true>(s, valid) : row_max<false>(s, valid)) * p.scale_log2;
          if (__any_sync(0xffffffffu, mx > m_run + 8.f)) {
            const float m_new = fmaxf(m_run, mx);
            alpha = ex2(m_run - m_new);
            l_run *= alpha;
            m_run = m_new;
            rescale = j > 0;  // at j == 0 the first P V overwrites O
          }
          l_tile = full ? row_exp<true>(s, valid, p.scale_log2, m_run, pk)
                        : row_exp<false>(s, valid, p.scale_log2, m_run, pk);
        }
        l_run = j == 0 ? l_tile : l_run + l_tile;
        // P (bf16, 2 per column) overwrites S columns 0..63, already read.
        tmem_st_x64(tS, pk);
        if (rescale) {
          // O += P V of the previous tile has completed: this tile's S was
          // committed after it.
          uint32_t o[HD];
          tmem_ld_x128_or_64<HD>(tO, o);
          const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
          for (int e = 0; e < HD; e += 2) {
            float x0, x1;
            f2_unpack(fmul2(f2_pack(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2), x0, x1);
            o[e] = __float_as_uint(x0);
            o[e + 1] = __float_as_uint(x1);
          }
          tmem_st_x128_or_64<HD>(tO, o);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bp);
      }
      if (!good) break;
      cs += x.nkv;
      good = __all_sync(0xffffffffu, wait_phase(bar(bars->o_full[i]), co & 1, abort_flag, p.status));
      if (!good) break;
      tc_fence_after();
      uint32_t o[HD];
      tmem_ld_x128_or_64<HD>(tO, o);
      // O is in registers: the MMA may start the next item's P V.
      tc_fence_before();
      mbar_arrive(bar(bars->o_empty[i]));
      ++co;
      const int t = x.t0 + i;
      const float inv_l = 1.f / l_run;
      if (t < x.vt) {
        const int tok = t * kBM + r;
        const int64_t orow =
            tok < x.n_w ? (p.ids ? static_cast<int64_t>(__ldg(p.ids + x.a + tok)) : static_cast<int64_t>(x.a + tok)) : 0;
        // An output row outside [0, N) can only come from a plan buffer
        // changed after its upload: record it and write nothing there.
        if (tok < x.n_w && static_cast<uint64_t>(orow) >= static_cast<uint64_t>(p.n_rows))
          atomicCAS(p.status, 0, WP_EDEVICE);
        else if (tok < x.n_w) {
          __nv_bfloat16* dst = p.o_vid + orow * p.o_stride + x.h * HD;
          if (p.vid_v8) {
            // 32-byte stores: whole sectors, half the instructions.
#pragma unroll
            for (int q8 = 0; q8 < HD / 16; ++q8) {
              uint32_t pk8[8];
#pragma unroll
              for (int u = 0; u < 8; ++u)
                pk8[u] = pack_bf16(__uint_as_float(o[16 * q8 + 2 * u]) * inv_l,
                                   __uint_as_float(o[16 * q8 + 2 * u + 1]) * inv_l);
              st_v8(dst + 16 * q8, pk8);
            }
          } else {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int q4 = 0; q4 < HD / 8; ++q4) {
              uint32_t pk4[4];
#pragma unroll
              for (int u = 0; u < 4; ++u)
                pk4[u] = pack_bf16(__uint_as_float(o[8 * q4 + 2 * u]) * inv_l,
                                   __uint_as_float(o[8 * q4 + 2 * u + 1]) * inv_l);
              d4[q4] = make_uint4(pk4[0], pk4[1], pk4[2], pk4[3]);
            }
          }
        }
      } else {
        const int lt = (t - x.vt) * kBM + r;
        if (lt < p.L) {
          float* dp = p.partial + ((static_cast<int64_t>(x.w) * p.L + lt) * p.heads + x.h) * HD;
          if (p.txt_v8) {
#pragma unroll
            for (int q8 = 0; q8 < HD / 8; ++q8) {
              uint32_t v8[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) v8[u] = __float_as_uint(__uint_as_float(o[8 * q8 + u]) * inv_l);
              st_v8(dp + 8 * q8, v8);
            }
          } else {
            float4* d4 = reinterpret_cast<float4*>(dp);
#pragma unroll
            for (int q4 = 0; q4 < HD / 4; ++q4)
              d4[q4] = make_float4(__uint_as_float(o[4 * q4]) * inv_l, __uint_as_float(o[4 * q4 + 1]) * inv_l,
                                   __uint_as_float(o[4 * q4 + 2]) * inv_l, __uint_as_float(o[4 * q4 + 3]) * inv_l);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------------- host --
// Test hook: wp_debug_stall_next(n) makes the next n launches stall.
std::atomic<int> g_stall_launches{0};
bool take_stall() {
  int n = g_stall_launches.load();
  while (n > 0)
    if (g_stall_launches.compare_exchange_weak(n, n - 1)) return true;
  return false;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2D map over rows x (heads*hd) columns of bf16 (box 128 rows x 64 columns)
// or of one-byte e4m3 codes (box 128 rows x 128 columns): 128-byte rows of a
// box, 128-byte swizzle; reads past the last row return zeros.
int make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t stride_B, bool bytes = false) {
  auto fn = encode_fn();
  if (!fn) return fail(WP_ECUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride_B)};
  const cuuint32_t box[2] = {bytes ? 128u : 64u, 128};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(WP_ECUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
  return WP_OK;
}

template <int HD, bool kRope, bool kFp8>
int launch(const AttnCall& c) {
  static_assert(!kRope || HD == 128, "the RoPE kernels rotate 128-column heads");
  CUtensorMap mq, mk, mv, mqt, mkt, mvt;
  const int64_t cols = static_cast<int64_t>(c.heads) * HD;
  if (int rc = make_map(&mq, c.q, c.N, cols, c.vid_stride_B, kFp8)) return rc;
  if (int rc = make_map(&mk, c.k, c.N, cols, c.vid_k_stride_B ? c.vid_k_stride_B : c.vid_stride_B, kFp8)) return rc;
  if (int rc = make_map(&mv, c.v, c.N, cols, c.vid_v_stride_B)) return rc;
  if (c.L > 0) {
    if (int rc = make_map(&mqt, c.qt, c.L, cols, c.txt_stride_B, kFp8)) return rc;
    if (int rc = make_map(&mkt, c.kt, c.L, cols, c.txt_stride_B, kFp8)) return rc;
    if (int rc = make_map(&mvt, c.vt, c.L, cols, c.vt_stride_B)) return rc;
  } else {
    mqt = mq; mkt = mk; mvt = mv;  // never read: there are no text tiles
  }
  TcParams p;
  p.win_off = c.win_off;
  p.ids = c.ids;
  p.pair_off = c.pair_off[c.text_tiles & 1];
  p.pair_add = c.text_tiles >> 1;
  p.nwin = c.nwin;
  p.L = c.L;
  p.heads = c.heads;
  p.text_tiles = c.text_tiles;
  p.total_pairs = c.total_pairs;
  p.o_vid = static_cast<__nv_bfloat16*>(c.o_vid);
  p.o_stride = c.o_stride_B / 2;
  p.n_rows = c.N;
  p.partial = c.partial;
  p.status = c.status;
  p.counter = c.status + 16;  // inside the status block, cleared before every launch
  p.scale_log2 = c.scale * 1.4426950408889634f;  // e4m3: the dequantisation scales are folded into c.scale
  p.stall = take_stall() ? 1 : 0;
  p.vid_v8 = (reinterpret_cast<uintptr_t>(c.o_vid) % 32 == 0) && (c.o_stride_B % 32 == 0);
  p.txt_v8 = reinterpret_cast<uintptr_t>(c.partial) % 32 == 0;
  p.boxes = c.boxes;
  p.wt = c.wt;
  p.wh = c.wh;
  p.ww = c.ww;
  for (int i = 0; i < kRopePairs; ++i) p.theta[i] = c.rope_theta[i];
  size_t smem = kSmemBytes;
  if (kRope) {
    smem = static_cast<size_t>(Cfg<HD, kFp8>::kTab) + static_cast<size_t>(c.wt + c.wh + c.ww) * kRopeStride * 8 + 1024;
    if (smem > kRopeMaxSmem)
      return fail(WP_EUNSUPPORTED, "window %dx%dx%d too large for the RoPE table", c.wt, c.wh, c.ww);
  }
  // Every variant asks for at least the bf16 footprint (kSmemBytes, more than
  // half of an SM's shared memory) so that exactly one CTA, and one
  // 512-column TMEM allocation, lives on an SM.
  auto kern = attn_tc_kernel<HD, kRope, kFp8>;
  if (int rc = cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem)),
                          "cudaFuncSetAttribute(attn_tc_kernel)"))
    return rc;
  int dev = 0, sms = 0;
  if (int rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return rc;
  if (int rc = cuda_check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
                          "cudaDeviceGetAttribute"))
    return rc;
  // Persistent: one CTA per SM (shared memory and TMEM allow no second).
  const int64_t items = static_cast<int64_t>(c.total_pairs) * c.heads;
  if (items > 0x7fffffff) return fail(WP_EUNSUPPORTED, "too many work items");
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(items, sms));
  kern<<<grid, kRope ? kRopeThreads : kThreads, smem, c.stream>>>(mq, mk, mv, mqt, mkt, mvt, p);
  return cuda_check(cudaGetLastError(), "attn_tc_kernel launch");
}

}  // namespace

void stall_next_launches(int n) { g_stall_launches.store(n < 0 ? 0 : n); }

int launch_attn_bf16_tc(const AttnCall& c) {
  if (c.fp8) {
    if (c.hd != 128 || c.rope) return fail(WP_EUNSUPPORTED, "e4m3 attention needs head_dim 128 and no RoPE");
    return launch<128, false, true>(c);
  }
  if (c.rope) return c.hd == 128 ? launch<128, true, false>(c) : fail(WP_EUNSUPPORTED, "RoPE attention needs head_dim 128");
  return c.hd == 64 ? launch<64, false, false>(c) : launch<128, false, false>(c);
}

}  // namespace wp
