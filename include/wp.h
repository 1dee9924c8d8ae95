/*
 * wp.h -- C ABI of libwp: shifted-window video attention on GB300 (sm_103a).
 *
 * What it computes is defined on the page "Window-Aligned Sequence
 * Parallelism (SeedVR2)" (vLLM-Omni design docs):
 *
 *   §Window layouts      window size normalised to the 720p latent area,
 *                        regular and half-window-shifted (clipped) layouts,
 *                        window enumeration w -> h -> t, row-major (t,h,w)
 *                        token order inside a window, canonical id
 *                        (t*H + h)*W + w.
 *   §Motivation, §Plan A at SP=1 a layout boundary is a local permutation.
 *   §SeedVR2 integration one packed-varlen attention per
 *                        [video window ; replicated text] segment; video
 *                        results return to canonical token order.
 *   §Text stream         next text state = (sum over windows of the
 *                        window's text output) / (window count of the
 *                        current layout).
 *
 * Conventions shared by every entry point:
 *   - Every function validates its arguments on the host first and returns a
 *     wp_status; on any error nothing is launched and wp_last_error() holds a
 *     one-line message (thread-local, valid until the next call on the same
 *     thread).
 *   - Device pointers are plain CUDA device addresses; the caller owns all
 *     device memory (the library never allocates device memory; the one
 *     fixed array that wp_window_attn_static uses is part of the library's
 *     device image).  `stream`
 *     is a cudaStream_t passed as void* (NULL = legacy default stream).  All
 *     device work is asynchronous on that stream.
 *   - Faults detected on the device (a bounded wait that expired, a failed
 *     bounds check) are written to a status word in the attention workspace
 *     (or in wp_window_attn_static's fixed scratch) and read back with
 *     wp_read_status(); no kernel traps or spins forever.
 *   - Batch is 1: a batch of videos is more windows.
 *   - There is no CPU fallback: without a usable sm_103a device every
 *     launching call returns WP_ECUDA.
 */
#ifndef WP_H_
#define WP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define WP_ABI_VERSION 1

typedef struct wp_plan wp_plan; /* opaque, host-owned, immutable once uploaded */

enum wp_layout {
  WP_CANONICAL = 0, /* row-major (t,h,w): row i holds canonical token i      */
  WP_REGULAR = 1,   /* §Window layouts, regular windows                       */
  WP_SHIFTED = 2    /* §Window layouts, cuts moved by half a window, clipped  */
};

enum wp_dtype {
  WP_BF16 = 0, /* bf16 in/out, fp32 accumulation (tcgen05 tensor cores)       */
  WP_FP32 = 1  /* fp32 in/out, fp32 arithmetic throughout (parity mode)        */
};

enum wp_status {
  WP_OK = 0,
  WP_EINVAL = 1,       /* bad argument (null pointer, size, layout, range)    */
  WP_EUNSUPPORTED = 2, /* valid but not supported (head_dim, alignment, ...)  */
  WP_ECUDA = 3,        /* a CUDA runtime/driver call failed                   */
  WP_ETIMEOUT = 4,     /* device: a bounded wait expired (status word only)   */
  WP_EDEVICE = 5,      /* device: a bounds check failed (status word only)    */
  WP_ENOTREADY = 6     /* plan not uploaded, or uploaded on another device    */
};

/* ------------------------------------------------------------------ plan --
 * wp_plan_create -- window geometry for a post-patch token grid (T, H, W)
 * (§Window layouts):
 *   scale = sqrt(45*80 / (H*W)) (IEEE double),
 *   wh = ceil(round(H*scale)/nh), ww = ceil(round(W*scale)/nw) (round: ties
 *   to even), wt = ceil(min(T, 30)/nt).
 * Regular intervals per axis are [i*w, min((i+1)*w, n)).  Shifted intervals
 * cut at floor((2k+1)*w/2) (half window, floored -- a reading: the page does
 * not say how an odd half is rounded; wp_plan_create_ex takes the other)
 * clipped to [0, n]; an axis a single window already covers is not
 * shifted.  Windows are enumerated w outermost,
 * then h, then t.  All host work; no CUDA call.
 * Errors: WP_EINVAL if any argument < 1, T*H*W >= 2^31, or a window
 * dimension comes out as 0.  *out is set only on success; free it with
 * wp_plan_destroy. */
int wp_plan_create(int T, int H, int W, int nt, int nh, int nw, wp_plan** out);

/* wp_plan_create_ex -- wp_plan_create with options.  flags = 0 is
 * wp_plan_create; WP_PLAN_HALF_CEIL rounds an odd half window up instead:
 * shifted cuts at ceil((2k+1)*w/2) (w = 15: 8, 23, 38, ... instead of 7,
 * 22, 37, ...), the other reading of "moved by half a window" that the page
 * leaves open.  Regular layouts and even window sizes are the same either
 * way.  WP_EINVAL also for unknown flag bits. */
#define WP_PLAN_HALF_CEIL 1u
int wp_plan_create_ex(int T, int H, int W, int nt, int nh, int nw, unsigned flags, wp_plan** out);
void wp_plan_destroy(wp_plan* plan); /* NULL is a no-op */

/* Geometry of one layout.  n_tokens = T*H*W; nwin = window count (1 for
 * WP_CANONICAL); (wt, wh, ww) = window size; max_tokens = largest window.
 * Any output pointer may be NULL. */
int wp_plan_info(const wp_plan* plan, int layout, int64_t* n_tokens, int* nwin,
                 int* wt, int* wh, int* ww, int* max_tokens);

/* Host copies of a layout's tables (for tests and callers that index rows):
 *   win_off[nwin+1]  row offset of each window in layout order,
 *   ids[N]           canonical id of the token at each layout row,
 *   boxes[nwin*6]    (t0,t1,h0,h1,w0,w1) half-open box of each window.
 * Any output pointer may be NULL. */
int wp_plan_host_tables(const wp_plan* plan, int layout, int32_t* win_off,
                        int32_t* ids, int32_t* boxes);

/* Device tables: the caller provides a device buffer of at least
 * *bytes (wp_plan_device_bytes, 256-byte aligned) and wp_plan_upload copies
 * every table into it with cudaMemcpyAsync on `stream` from host memory the
 * plan owns (pageable: the copy is complete when the call returns).  The
 * plan then refers to that buffer, which must stay alive and unmodified
 * until the plan is destroyed or uploaded again; it is bound to the current
 * device.  Tables: per layout win_off, ids and two work-split prefix tables;
 * the six fused permutation tables perm[a->b][q] = pos_a[ids_b[q]]. */
int wp_plan_device_bytes(const wp_plan* plan, size_t* bytes);
int wp_plan_upload(wp_plan* plan, void* dev_buf, size_t bytes, void* stream);

/* Window -> rank assignment for running a layout on `world` devices
 * (§Planner): windows taken by (-token count, window id), each placed on the
 * rank with the smallest (assigned tokens, rank id); a rank lists its windows
 * in ascending window id.  win_rank[nwin] receives each window's rank and
 * rank_tokens[world] each rank's token count (either may be NULL).  Host
 * only; WP_EINVAL for world < 1 or a bad layout. */
int wp_plan_assign(const wp_plan* plan, int layout, int world, int32_t* win_rank,
                   int64_t* rank_tokens);

/* Plan A exchange between two layouts on `world` devices (§Plan A
 * redistribution), seen from rank `rank`; host only.  With both layouts
 * assigned as in wp_plan_assign and each rank's rows in its local order:
 *   counts[world*world]  C[r*world + d] = rows rank d needs from rank r
 *                        (row r = input split sizes of rank r, column d =
 *                        output split sizes of rank d);
 *   *exchange_required   1 if any row changes rank (then every rank must
 *                        join the all-to-all), 0 if the switch is a local
 *                        permutation (always the case for world == 1);
 *   send_rows[...]       the rows this rank sends, as indices in its source
 *                        local order, grouped by destination rank 0..world-1
 *                        and, inside a group, in the destination's local
 *                        order (sum over d of C[rank][d] entries);
 *   recv_pos[...]        for the rows this rank receives (segments from
 *                        ranks 0..world-1 concatenated), the position of
 *                        each in its destination local order (sum over r of
 *                        C[r][rank] entries); argsort of it, or a scatter by
 *                        it, gives the local order.
 * Any output pointer may be NULL. */
int wp_plan_exchange(const wp_plan* plan, int src_layout, int dst_layout, int world,
                     int rank, int64_t* counts, int* exchange_required,
                     int32_t* send_rows, int32_t* recv_pos);

/* --------------------------------------------------------------- permute --
 * wp_permute -- §Motivation/§Plan A at SP=1: the layout switch as a local row
 * permutation.  For every destination row q of dst_layout:
 *     dst[q*dst_stride_B .. +row_B) = src[p*src_stride_B .. +row_B),
 *     p = row of src_layout that holds canonical token ids_dst[q].
 * Rows are opaque bytes (any dtype); the copy is exact.  N = T*H*W rows.
 * src_layout == dst_layout is a strided copy.
 * Requirements (WP_EUNSUPPORTED otherwise): src, dst 16-byte aligned;
 * row_B > 0 and a multiple of 16; strides multiples of 16 and >= row_B.
 * WP_EINVAL: null pointer, bad layout, or the byte ranges of src and dst
 * overlap (in-place permutation is not supported).  WP_ENOTREADY: plan not
 * uploaded on the current device. */
int wp_permute(const wp_plan* plan, int src_layout, int dst_layout,
               const void* src, int64_t src_stride_B, void* dst,
               int64_t dst_stride_B, int64_t row_B, void* stream);

/* ------------------------------------------------------------------ rope --
 * wp_rope -- window-local 3D rotary position embedding of q and k, in place
 * (§Reference quirks reproduced on purpose): a video token at window-local
 * (dt, dh, dw) of `layout` uses the axial indices (L + dt, dh, dw), every
 * window restarting at 0; the rotary span is 3*(head_dim/3) = 126 channels,
 * the last two pass through.  Readings where the page is silent: axis
 * blocks t, h, w of 42 channels; channels (2i, 2i+1) of a block rotate by
 * pos * rope_base^(-2i/42) (rope_base 10000 is the usual value); a text
 * token at position l uses (l, l, l).
 * q, k: [N, heads, 128] rows in `layout` order (shared row stride); qt, kt:
 * [L, heads, 128] (shared stride; may be NULL iff L == 0).  dtype WP_BF16
 * (rotated in fp32, rounded to nearest even) or WP_FP32.
 * WP_EUNSUPPORTED: head_dim != 128, misaligned pointers or strides;
 * WP_EINVAL: bad layout/dtype, NULL pointers, rope_base <= 1. */
int wp_rope(const wp_plan* plan, int layout, int heads, int head_dim, int L,
            int dtype, void* q, void* k, int64_t vid_row_stride_B, void* qt,
            void* kt, int64_t txt_row_stride_B, float rope_base, void* stream);

/* ------------------------------------------------------------- attention --
 * wp_attn_workspace_bytes -- device workspace wp_window_attn needs: a
 * 256-byte status block plus the per-window text outputs
 * [nwin, L, heads, head_dim] in fp32. */
int wp_attn_workspace_bytes(const wp_plan* plan, int layout, int heads,
                            int head_dim, int L, int dtype, size_t* bytes);

/* wp_window_attn -- one layer of window attention (§SeedVR2 integration,
 * §Text stream) over layout `layout` (WP_REGULAR or WP_SHIFTED).
 * For every window w and head h, with segment X = [video rows of w ; text]:
 *     Y = softmax(Q_X K_X^T * s) V_X     (full, no mask; s = softmax_scale,
 *                                         or 1/sqrt(head_dim) if <= 0)
 * Video rows of Y are written to o_vid at their CANONICAL row ids; the text
 * rows of Y are T_w (fp32, written to the workspace), and
 * o_txt = (T_0 + ... + T_{nwin-1}) / nwin, summed in fp32 in window order by
 * a second kernel (deterministic, no atomics).
 * Layout (element type = dtype):
 *   q, k, v   [N, heads, head_dim] rows in `layout` order; row r of q starts
 *             at q + r*vid_row_stride_B (q, k, v share the stride, e.g. a
 *             packed [N, 3, heads, head_dim] buffer).  Inner dims contiguous.
 *   qt,kt,vt  [L, heads, head_dim] with row stride txt_row_stride_B.
 *   o_vid     [N, heads, head_dim], canonical order, row stride
 *             o_vid_row_stride_B.
 *   o_txt     [L, heads, head_dim], contiguous.  May be NULL iff L == 0.
 *   workspace at least wp_attn_workspace_bytes; its status word is cleared
 *             at the start of the call.
 * All rows of q/k/v (including rows of neighbouring windows) must be finite.
 * An output row the plan's device tables place outside [0, N) (possible only
 * if the plan's buffer changed after wp_plan_upload) is not written, and
 * WP_EDEVICE goes to the status word.
 * Supported (WP_EUNSUPPORTED otherwise): head_dim 64 or 128; pointers and
 * strides multiples of 16 bytes; heads*head_dim*elem <= stride.
 * WP_EINVAL: null pointer, heads < 1, L < 0, layout not REGULAR/SHIFTED,
 * workspace too small.  WP_ENOTREADY: plan not uploaded on this device. */
int wp_window_attn(const wp_plan* plan, int layout, int heads, int head_dim,
                   int L, int dtype, const void* q, const void* k,
                   const void* v, int64_t vid_row_stride_B, const void* qt,
                   const void* kt, const void* vt, int64_t txt_row_stride_B,
                   void* o_vid, int64_t o_vid_row_stride_B, void* o_txt,
                   void* workspace, size_t ws_bytes, float softmax_scale,
                   void* stream);

/* wp_window_attn_to -- wp_window_attn with the video output written in
 * layout `out_layout` instead of canonical order: video row r of the input
 * layout lands at the row of `out_layout` that holds the same canonical
 * token.  With out_layout = the next layer's layout this fuses the
 * re-layout of §Motivation/§Plan A into the attention epilogue; the result
 * is bit-identical to wp_window_attn followed by wp_permute(CANONICAL ->
 * out_layout).  out_layout == layout keeps the input order.  o_txt and all
 * other arguments as wp_window_attn; WP_EINVAL for a bad out_layout. */
int wp_window_attn_to(const wp_plan* plan, int layout, int out_layout, int heads,
                      int head_dim, int L, int dtype, const void* q,
                      const void* k, const void* v, int64_t vid_row_stride_B,
                      const void* qt, const void* kt, const void* vt,
                      int64_t txt_row_stride_B, void* o_vid,
                      int64_t o_vid_row_stride_B, void* o_txt, void* workspace,
                      size_t ws_bytes, float softmax_scale, void* stream);

/* wp_attn_rope_workspace_bytes -- device workspace wp_window_attn_rope
 * needs: wp_attn_workspace_bytes plus the rotated text q and k
 * (2 * L * heads * head_dim bf16 values), then, from the next multiple of
 * 1024 bytes, the rotated video k (N * heads * head_dim bf16 values). */
int wp_attn_rope_workspace_bytes(const wp_plan* plan, int layout, int heads,
                                 int head_dim, int L, int dtype, size_t* bytes);

/* wp_window_attn_rope -- wp_window_attn_to on UN-rotated q and k: applies
 * the window-local 3D RoPE of wp_rope ("Window-Aligned Sequence Parallelism
 * (SeedVR2)", §Reference quirks reproduced on purpose; same positions,
 * angles base^(-2i/42) and channel pairs) as part of the call, so that q
 * is never rotated in HBM.  q, k, qt, kt are the projections before RoPE
 * and are not modified; v, vt, the outputs, the scatter (`out_layout`) and
 * the text mean are as in wp_window_attn_to.  k and the text q/k, read by
 * many work items, are rotated once per call into the workspace (in fp32,
 * one rounding to bf16: the values wp_rope writes); each video Q tile,
 * read by one work item, is rotated in shared memory after it lands, in
 * bf16 arithmetic (cos, sin rounded to bf16; two roundings per value), so
 * results agree with wp_rope followed by wp_window_attn_to to within the
 * bf16 attention tolerance, not bit for bit.
 * Supported (WP_EUNSUPPORTED otherwise): dtype WP_BF16, head_dim 128, the
 * plan's window size (wt + wh + ww) <= 196 (the cos/sin table lives in
 * shared memory), the alignment rules of wp_window_attn.  WP_EINVAL:
 * rope_base <= 1, workspace smaller than wp_attn_rope_workspace_bytes, and
 * the wp_window_attn_to cases. */
int wp_window_attn_rope(const wp_plan* plan, int layout, int out_layout, int heads,
                        int head_dim, int L, int dtype, const void* q,
                        const void* k, const void* v, int64_t vid_row_stride_B,
                        const void* qt, const void* kt, const void* vt,
                        int64_t txt_row_stride_B, void* o_vid,
                        int64_t o_vid_row_stride_B, void* o_txt, void* workspace,
                        size_t ws_bytes, float softmax_scale, float rope_base,
                        void* stream);

/* wp_window_attn_fp8 -- wp_window_attn_to with Q K^T on e4m3 operands
 * (tcgen05 kind::f8f6f4, twice the bf16 rate per instruction); P V, the
 * softmax, the outputs and the text mean as in the bf16 call.  The pages
 * mention low-precision training only as context ("Scaling Video Training
 * with Parallelism", §Key claims: NVFP4 for LongLive-2.0) and define no such
 * path; this is an opt-in variant for callers whose q/k projection already
 * emits e4m3, with per-tensor scales:
 *     scores = (q8 * q_scale) . (k8 * k_scale) * softmax_scale
 * (softmax_scale <= 0: 1/sqrt(head_dim)).  Its error against exact attention
 * on the unquantised q/k is that of e4m3 rounding (3 mantissa bits) and is
 * larger than the bf16 call's.
 * Layout: q8, k8 [N, heads, 128] one byte per element (e4m3 codes, layout
 * `layout` order, shared row stride qk_row_stride_B); v [N, heads, 128] bf16
 * (row stride v_row_stride_B); qt8, kt8 [L, heads, 128] e4m3 (stride
 * txt_qk_row_stride_B); vt [L, heads, 128] bf16 (stride txt_v_row_stride_B);
 * o_vid, o_txt, workspace (wp_attn_workspace_bytes with WP_BF16) as in
 * wp_window_attn_to.
 * Supported (WP_EUNSUPPORTED otherwise): head_dim 128; pointers and strides
 * multiples of 16 bytes, each stride at least one row.  WP_EINVAL: scales
 * not finite and > 0, and the wp_window_attn_to cases. */
int wp_window_attn_fp8(const wp_plan* plan, int layout, int out_layout, int heads,
                       int head_dim, int L, const void* q8, const void* k8,
                       int64_t qk_row_stride_B, const void* v, int64_t v_row_stride_B,
                       const void* qt8, const void* kt8, int64_t txt_qk_row_stride_B,
                       const void* vt, int64_t txt_v_row_stride_B, float q_scale,
                       float k_scale, void* o_vid, int64_t o_vid_row_stride_B,
                       void* o_txt, void* workspace, size_t ws_bytes,
                       float softmax_scale, void* stream);

/* wp_quantize_e4m3 -- bf16 rows to e4m3 codes for wp_window_attn_fp8:
 *     code = e4m3(fp32(x) * inv_scale)
 * one fp32 multiply (round to nearest even), then the nearest e4m3 value
 * (ties to even), saturated to +-448; dequantised value = code / inv_scale
 * (pass q_scale = 1 / inv_scale to the attention call; a power of two keeps
 * that exact).  src [rows, cols] bf16 with row stride src_row_stride_B; dst
 * [rows, cols] bytes with row stride dst_row_stride_B.  WP_EUNSUPPORTED:
 * cols not a multiple of 16, pointers or strides not 16-byte aligned, or a
 * stride shorter than a row.  WP_EINVAL: NULL pointers, negative sizes,
 * inv_scale not finite and > 0.  Asynchronous on `stream`. */
int wp_quantize_e4m3(const void* src, int64_t rows, int cols, int64_t src_row_stride_B,
                     void* dst, int64_t dst_row_stride_B, float inv_scale, void* stream);

/* wp_window_attn_static -- wp_window_attn for callers that cannot allocate
 * device memory when they run attention (a runtime that owns a fixed memory
 * pool and forbids allocation from plugins, a latency-bound loop that cannot
 * afford the implicit device synchronisation of cudaMalloc, a caller with no
 * allocator at hand).  The pages define nothing like it: it is a convenience
 * of this library with no counterpart in the method.
 * Same arguments, layout and results as wp_window_attn, minus the workspace:
 * the scratch comes from one array of WP_STATIC_SCRATCH_BYTES bytes compiled
 * into the library's device image.  The call allocates nothing and calls no
 * allocating routine.
 *   - Size limit: the call needs 256 + nwin*L*heads*head_dim*4 bytes of
 *     scratch (wp_attn_workspace_bytes); larger requests return
 *     WP_EUNSUPPORTED with a message, and nothing is launched.
 *   - Set-up: the first call on each device looks up the array's device
 *     address (cudaGetSymbolAddress) with that device current and remembers
 *     it.  With CUDA's lazy module loading (the default) that lookup is also
 *     when the runtime loads the library's device code onto the device and
 *     reserves the array, so the first call may take device memory and can
 *     fail with WP_ECUDA if none is left: make it before a fixed pool claims
 *     the device, and before capturing any stream into a graph.  Later calls
 *     allocate nothing.  Only devices on which this set-up ran hold the
 *     array (until the process exits).  After cudaDeviceReset the remembered
 *     address is stale: do not call this entry point on that device again.
 *   - Sharing: every call on a device uses the same array, which keeps the
 *     last call's contents (the call clears what must start at zero).  Calls
 *     whose work overlaps on the GPU (e.g. on two streams at once) race on
 *     it: order them on one stream or synchronise between them.
 *   - Device faults: wp_read_status(NULL, ...) reads the array's status
 *     word (WP_ETIMEOUT after a bounded wait expired) like a workspace's. */
#define WP_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)
int wp_window_attn_static(const wp_plan* plan, int layout, int heads, int head_dim,
                          int L, int dtype, const void* q, const void* k,
                          const void* v, int64_t vid_row_stride_B,
                          const void* qt, const void* kt, const void* vt,
                          int64_t txt_row_stride_B, void* o_vid,
                          int64_t o_vid_row_stride_B, void* o_txt,
                          float softmax_scale, void* stream);

/* wp_read_status -- copies the device status word of `workspace` to
 * *device_status (a wp_status value: WP_OK, WP_ETIMEOUT or WP_EDEVICE),
 * synchronising `stream` first.  workspace == NULL reads the status word of
 * wp_window_attn_static's fixed scratch on the current device (the set-up
 * described there happens here if it has not yet).  No device memory is
 * allocated.  Returns WP_ECUDA if the copy fails. */
int wp_read_status(const void* workspace, int* device_status, void* stream);

/* wp_debug_stall_next -- test hook for the failure path: the next
 * `launches` bf16 attention launches (wp_window_attn*, any entry point) make
 * the MMA warp of CTA 0 wait for an mbarrier phase that nothing completes.
 * Its bounded wait (2 s) expires: the CTA records WP_ETIMEOUT in the status
 * word, winds down (its copies and MMAs drained, TMEM freed) and the launch
 * ends; the other CTAs finish their own items, and the context stays
 * usable.  The results of a stalled launch are undefined.  0 cancels.
 * Process-wide; WP_EINVAL for a negative count. */
int wp_debug_stall_next(int launches);

/* ---------------------------------------------------------------- misc --- */
const char* wp_last_error(void); /* never NULL; "" when there is no error */
int wp_abi_version(void);        /* WP_ABI_VERSION */

#ifdef __cplusplus
}
#endif
#endif /* WP_H_ */
