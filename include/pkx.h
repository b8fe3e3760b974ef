/*
 * pkx.h -- C ABI of libpkx: extend attention over a page-size-1 KV pool and
 * its companions (decode attention, unified KV-index build, merge_state, the
 * KV write into the pool and the KV-index gather from the request table),
 * as hand-written CUDA kernels for sm_103a (GB300).
 *
 * Conventions for every call below
 * --------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller.  Outputs
 *    are preallocated by the caller and written in place.  A call never
 *    allocates device memory and never synchronises the host with the
 *    device; everything is enqueued on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream).  Kernels run on the calling thread's
 *    current CUDA device: `stream` and every pointer must belong to it.
 *  - bf16 means IEEE bfloat16 (16 bits).  Shapes are written outermost
 *    first; the last dimension is always contiguous.  Strides are in
 *    ELEMENTS.
 *  - Alignment: every bf16 tensor base pointer must be 16-byte aligned, and
 *    every row stride must be a multiple of 8 elements (16 bytes); index and
 *    indptr arrays must be 4-byte (int32) / 8-byte (int64) aligned.
 *  - Return value: PKX_OK (0) or an error code.  Argument errors are found
 *    on the host before anything is enqueued (nothing is written then).
 *    pkx_last_error_string() gives a human-readable reason for the last
 *    failing call on the calling thread.  No call aborts or throws.
 *  - Index values that point outside the pool ([0, num_slots)) are not
 *    dereferenced: the kernel reads a zero row instead and records
 *    PKX_EDEVICE in the workspace's status word, which
 *    pkx_workspace_status() reads back.
 *  - Array extents are the caller's: an array described by an indptr (for
 *    example kv_indices[kv_indptr[b] .. kv_indptr[b+1])) must hold every
 *    entry the indptr names, as a C array argument must; its length is not
 *    checked.  Such an array may be NULL only when the indptr names no entry.
 *  - Every wait inside a kernel is bounded (about two seconds); a wait that
 *    runs out records PKX_ETIMEOUT in the same status word and the kernel
 *    returns instead of hanging.
 *
 * Notation (the pages' own): per sequence b, P_b prefix (cached) tokens and
 * E_b extend (new) tokens, T_b = P_b + E_b keys at positions 0..T_b-1; extend
 * query i sits at position P_b + i.  Hq query heads, Hkv KV heads, query head
 * h reads KV head h / (Hq / Hkv).  Lq = query/key head dim, Lv = value head
 * dim.
 */
#ifndef PKX_H
#define PKX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define PKX_OK 0
#define PKX_EINVAL 1        /* bad argument: null, misaligned, inconsistent */
#define PKX_EUNSUPPORTED 2  /* valid but not built: head dims, group size   */
#define PKX_ECUDA 3         /* a CUDA runtime call or a launch failed        */
#define PKX_ETIMEOUT 4      /* a bounded device wait ran out (status word)   */
#define PKX_EDEVICE 5       /* device-side index check failed (status word)  */
#define PKX_EWORKSPACE 6    /* workspace null or smaller than required       */

/*
 * Element format of the KV pool (kv_dtype arguments).
 * Source: sglang flashinfer_backend.py: the KV cache dtype may be bf16 or
 * float8_e4m3fn / float8_e5m2, and the attention call takes the layer's
 * k_scale and v_scale.  In an fp8 pool a key element reads code * k_scale
 * and a value element code * v_scale (k_scale, v_scale positive host
 * floats; ignored for bf16).  An fp8 pool's strides are in bytes (its
 * elements are one byte); the 16-byte alignment rule for rows still
 * applies.  Built for Lq = Lv = 64 or 128 and for the MLA head Lq / Lv =
 * 576 / 512 (v_buffer a view of k_buffer's codes), with or without a custom
 * mask, and for the split head dims 192 / 128 and 288 / 256 in the two
 * extend forms (no mask, no decode); other fp8 calls return
 * PKX_EUNSUPPORTED.  The extend rows of the two-stage form (k_extend /
 * v_extend) stay bf16.
 */
#define PKX_KV_BF16 0
#define PKX_KV_FP8_E4M3 1
#define PKX_KV_FP8_E5M2 2

/* Reason for the last failing call on this thread ("" if none). */
const char *pkx_last_error_string(void);

/* Library version string. */
const char *pkx_version(void);

/*
 * Workspace bytes the attention calls need for the given problem on the
 * CURRENT device (it depends on the device's SM count).  The workspace holds
 * the device-built work list and the split-KV partial results; it must be
 * 256-byte aligned.  Its content need not be initialised and may be reused
 * by later calls on the same stream.  Returns 0 on bad arguments.
 *   num_q_tokens: rows of q_extend (sum of E_b) for extend; batch for decode.
 */
size_t pkx_extend_workspace_size(int batch, int num_q_tokens, int hq, int hkv,
                                 int lq, int lv);
size_t pkx_decode_workspace_size(int batch, int hq, int hkv, int lq, int lv);
/*
 * The smallest workspace decode attention accepts.  With at least
 * pkx_decode_workspace_size bytes every decode unit runs two key streams (the
 * faster schedule); with less, but at least this many, one stream.
 */
size_t pkx_decode_workspace_min_size(int batch, int hq, int hkv, int lq, int lv);

/*
 * Device status word of the last attention call that used `workspace`:
 * copies it to the host (synchronising `stream`) and returns PKX_OK,
 * PKX_EDEVICE or PKX_ETIMEOUT.  Returns PKX_ECUDA if the copy fails.
 */
int pkx_workspace_status(const void *workspace, void *stream);

/*
 * Profiling hook: when `before` / `after` are non-null cudaEvent_t handles,
 * every later attention call made on this thread records `before` on its
 * stream immediately before the attention kernel launch and `after`
 * immediately after it (the scheduler and split-KV combine launches fall
 * outside the pair), so the caller can time the attention kernel alone with
 * cudaEventElapsedTime.  Pass NULL, NULL to stop.  Events are owned by the
 * caller.
 */
void pkx_set_attention_events(void *before, void *after);

/*
 * Time limit of every bounded wait inside the attention kernels launched
 * later on this thread, in nanoseconds (0 restores the default of two
 * seconds).  A wait that runs out records PKX_ETIMEOUT in the status word,
 * raises the CTA's abort flag, lets the tensor core and its own copies
 * finish, frees its tensor memory and returns; the call's outputs are then
 * undefined but the context stays usable.  This serves the library's own
 * failure handling (no device wait may hang); the pages have no
 * counterpart.
 */
void pkx_set_wait_limit_ns(uint64_t ns);

/*
 * Test hook for the timeout path above: when `on` is non-zero, the softmax
 * warps of every attention kernel launched later on this thread first wait
 * on a barrier no thread arrives at, so that their bounded wait runs out and
 * the call reports PKX_ETIMEOUT.  Pass 0 to stop.  Not for production use;
 * the pages have no counterpart.
 */
void pkx_set_stall_injection(int on);

/*
 * Extend attention, two-stage form.
 * Source: sglang extend_attention.py (diff 0.5.3rc2 -> 0.5.4.post1),
 * extend_attention_fwd and its _fwd_kernel (prefix K/V read from the pool
 * through kv_indptr/kv_indices, extend K/V read from k_extend/v_extend); the
 * masks, cap and online softmax follow _fwd_kernel_unified on the same page.
 *
 * For every sequence b, q head h and extend query i (position P_b + i):
 *   keys j <  P_b: k_buffer/v_buffer row (kv_indices[kv_indptr[b] + j], h_kv)
 *   keys j >= P_b: k_extend/v_extend row (qo_indptr[b] + j - P_b, h_kv)
 *   s_j = sm_scale * <q, k_j>;  s_j = logit_cap * tanh(s_j / logit_cap) if
 *   logit_cap > 0; key j is visible iff j <= P_b + i and, if
 *   sliding_window > 0, (P_b + i) - j <= sliding_window;
 *   o = softmax over visible keys of s, applied to v;  lse = log sum exp s.
 * With a custom mask (speculative tree verification, _fwd_kernel_unified
 * "Apply custom mask"), key j is visible iff
 * custom_mask[mask_indptr[b] + i * T_b + j] != 0 (T_b = P_b + E_b keys of
 * the sequence) and the window holds: the mask replaces the causal term.
 * With sinks (_fwd_kernel_unified "Handle sink tokens"), each row's softmax
 * denominator gains exp(sinks[h] - m): o is scaled down, lse includes it.
 *
 *   q_extend   bf16 [num_q_tokens, hq, lq] contiguous
 *   k_extend   bf16 row (t, h) at k_extend + t*ke_st + h*ke_sh, lq elements
 *   v_extend   bf16 row (t, h) at v_extend + t*ve_st + h*ve_sh, lv elements
 *   o_extend   bf16 [num_q_tokens, hq, lv] contiguous (written)
 *   k_buffer   bf16 row (slot, h) at k_buffer + slot*kb_ss + h*kb_sh (lq)
 *   v_buffer   bf16 row (slot, h) at v_buffer + slot*vb_ss + h*vb_sh (lv);
 *              may alias k_buffer (MLA: V is the first lv dims of K)
 *   qo_indptr  int32 [batch+1], qo_indptr[0] = 0, non-decreasing,
 *              qo_indptr[batch] = num_q_tokens
 *   kv_indptr  int32 [batch+1] over kv_indices: the PREFIX keys only
 *   kv_indices int32 [kv_indptr[batch]] pool slots
 *   sm_scale   <= 0 selects 1/sqrt(lq)
 *   logit_cap  <= 0: no cap
 *   sliding_window <= 0: no window
 *   custom_mask nullable uint8, one byte per (extend row, key) of every
 *              sequence, sequence b's rows at mask_indptr[b]
 *   mask_indptr int32 [batch+1] element offsets into custom_mask (needed
 *              with a mask; NULL otherwise)
 *   sinks      nullable fp32 [hq] sink logit per query head
 *   kv_dtype, k_scale, v_scale  the pool's format and scales (PKX_KV_*)
 *   lse_out    nullable fp32 [num_q_tokens, hq] (natural log)
 *   workspace  >= pkx_extend_workspace_size(...) bytes
 * Supported (lq, lv): (64, 64), (128, 128), (576, 512), and the split head
 * dims (192, 128) and (288, 256) (no custom mask for those; an fp8 pool in
 * the extend forms only);
 * hq % hkv == 0 and hq / hkv <= 128.
 */
int pkx_extend_attention_fwd(
    const void *q_extend, const void *k_extend, const void *v_extend,
    void *o_extend, const void *k_buffer, const void *v_buffer,
    const int32_t *qo_indptr, const int32_t *kv_indptr,
    const int32_t *kv_indices, int batch, int num_q_tokens, int hq, int hkv,
    int lq, int lv, int64_t ke_st, int64_t ke_sh, int64_t ve_st,
    int64_t ve_sh, int64_t kb_ss, int64_t kb_sh, int64_t vb_ss, int64_t vb_sh,
    int64_t num_slots, float sm_scale, float logit_cap, int sliding_window,
    const uint8_t *custom_mask, const int32_t *mask_indptr, const float *sinks,
    int kv_dtype, float k_scale, float v_scale, float *lse_out,
    void *workspace, size_t workspace_bytes, void *stream);

/*
 * Extend attention, two-stage form, with the KV write fused in.
 * Source: sglang flashinfer_backend.py, forward_extend: the new tokens' K
 * and V rows are saved into the pool (token_to_kv_pool.set_kv_buffer(layer,
 * cache_loc, k, v, ...)) before attention runs.  This call computes what
 * pkx_set_kv_buffer (or pkx_set_kv_buffer_fp8 for an fp8 pool) followed by
 * pkx_extend_attention_fwd computes:
 *   k_buffer[cache_loc[t], h, :] = k_extend[t, h, :]  and likewise for v
 * for every extend token t < num_q_tokens and KV head h, and the same o_extend
 * and lse.  Arguments as pkx_extend_attention_fwd, with the pools writable and
 *   cache_loc  int64 [num_q_tokens] pool slot of each extend token; the slots
 *              are the new tokens' own, so none of them appears among the
 *              prefix indices (kv_indices).  A slot outside the pool is
 *              skipped.
 * For a bf16 pool with Lq = Lv (64, 128) or the split head dims the attention
 * kernel does the write itself (idle warps copy each unit's own tokens'
 * rows, beside the attention); for the MLA pool (only K rows are written)
 * and fp8 pools the standalone write kernel runs first on the stream.
 */
int pkx_extend_attention_fwd_kv_write(
    const void *q_extend, const void *k_extend, const void *v_extend,
    void *o_extend, void *k_buffer, void *v_buffer,
    const int32_t *qo_indptr, const int32_t *kv_indptr,
    const int32_t *kv_indices, int batch, int num_q_tokens, int hq, int hkv,
    int lq, int lv, int64_t ke_st, int64_t ke_sh, int64_t ve_st,
    int64_t ve_sh, int64_t kb_ss, int64_t kb_sh, int64_t vb_ss, int64_t vb_sh,
    int64_t num_slots, float sm_scale, float logit_cap, int sliding_window,
    const uint8_t *custom_mask, const int32_t *mask_indptr, const float *sinks,
    int kv_dtype, float k_scale, float v_scale, float *lse_out,
    const int64_t *cache_loc, void *workspace, size_t workspace_bytes,
    void *stream);

/*
 * Extend attention, ragged + paged split.
 * Source: sglang flashinfer_backend.py, forward_extend with use_ragged (taken
 * there for 4096 or more extend tokens): a causal pass over the extend keys
 * alone (the ragged pass, k_extend / v_extend), a pass over the prefix keys
 * alone in which every prefix key is visible to every extend query (the
 * paged pass, the pool through kv_indptr / kv_indices), and merge_state of
 * the two (o, lse) pairs.  The result is the two-stage form's up to bf16
 * rounding of the two partial outputs (each pass writes bf16, as the pages'
 * wrappers do); a sequence without prefix takes the ragged result alone
 * (the paged pass gives it lse = -inf, weight 0).
 * Arguments as pkx_extend_attention_fwd, without custom_mask / mask_indptr /
 * sinks (the pages' ragged path has neither), and
 *   workspace  >= pkx_ragged_paged_workspace_size(...) bytes: the passes'
 *              scratch, the paged pass's output and both passes' lse.
 * Runs three kernels' worth of launches in order on `stream`; o_extend holds
 * the ragged pass's output in between.
 */
size_t pkx_ragged_paged_workspace_size(int batch, int num_q_tokens, int hq,
                                       int hkv, int lq, int lv);
int pkx_extend_attention_fwd_ragged_paged(
    const void *q_extend, const void *k_extend, const void *v_extend,
    void *o_extend, const void *k_buffer, const void *v_buffer,
    const int32_t *qo_indptr, const int32_t *kv_indptr,
    const int32_t *kv_indices, int batch, int num_q_tokens, int hq, int hkv,
    int lq, int lv, int64_t ke_st, int64_t ke_sh, int64_t ve_st,
    int64_t ve_sh, int64_t kb_ss, int64_t kb_sh, int64_t vb_ss, int64_t vb_sh,
    int64_t num_slots, float sm_scale, float logit_cap, int sliding_window,
    int kv_dtype, float k_scale, float v_scale, float *lse_out,
    void *workspace, size_t workspace_bytes, void *stream);

/*
 * Extend attention, unified form.
 * Source: sglang extend_attention.py, extend_attention_fwd_unified and
 * _fwd_kernel_unified: prefix and extend keys alike are pool slots
 * kv_indices[kv_indptr[b] + j], j < T_b = kv_indptr[b+1] - kv_indptr[b]; the
 * first prefix_lens[b] of them are the prefix, so extend query i sits at
 * position prefix_lens[b] + i.  The window start position is 0 for every
 * sequence (the launcher's default).  Same math and arguments as the
 * two-stage form, except:
 *   q, o       as q_extend / o_extend
 *   kv_indptr  int32 [batch+1] over ALL keys of each sequence
 *   kv_indices int64 [kv_indptr[batch]] (as build_unified_kv_indices makes)
 *   prefix_lens int32 [batch]
 */
int pkx_extend_attention_fwd_unified(
    const void *q, void *o, const void *k_buffer, const void *v_buffer,
    const int32_t *qo_indptr, const int32_t *kv_indptr,
    const int64_t *kv_indices, const int32_t *prefix_lens, int batch,
    int num_q_tokens, int hq, int hkv, int lq, int lv, int64_t kb_ss,
    int64_t kb_sh, int64_t vb_ss, int64_t vb_sh, int64_t num_slots,
    float sm_scale, float logit_cap, int sliding_window,
    const uint8_t *custom_mask, const int32_t *mask_indptr, const float *sinks,
    int kv_dtype, float k_scale, float v_scale, float *lse_out,
    void *workspace, size_t workspace_bytes, void *stream);

/*
 * Decode attention.
 * Source: sglang flashinfer_backend.py, forward_decode (the token's K/V are
 * saved into the pool first, then one query per sequence attends to all
 * T_b = kv_indptr[b+1] - kv_indptr[b] keys) and the sliding-window decode
 * index updater (the last min(T_b, W + 1) keys).  Same math as extend with
 * the query at position T_b - 1.  A sequence with T_b = 0 (padding) gets
 * o = 0 and lse = -inf.
 *   q  bf16 [batch, hq, lq] contiguous;  o  bf16 [batch, hq, lv] contiguous
 *   kv_indptr int32 [batch+1]; kv_indices int32 [kv_indptr[batch]]
 *   kv_dtype, k_scale, v_scale  the pool's format and scales (PKX_KV_*)
 *   workspace >= pkx_decode_workspace_size(...) bytes for the two-key-stream
 *             schedule; at least pkx_decode_workspace_min_size(...) bytes
 *             runs one stream per unit (same results)
 */
int pkx_decode_attention_fwd(
    const void *q, void *o, const void *k_buffer, const void *v_buffer,
    const int32_t *kv_indptr, const int32_t *kv_indices, int batch, int hq,
    int hkv, int lq, int lv, int64_t kb_ss, int64_t kb_sh, int64_t vb_ss,
    int64_t vb_sh, int64_t num_slots, float sm_scale, float logit_cap,
    int sliding_window, int kv_dtype, float k_scale, float v_scale,
    float *lse_out, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Decode attention without a workspace argument, for callers that cannot
 * allocate device memory: a plugin whose host framework owns every device
 * allocation and offers it no allocator, or a latency-critical decode loop
 * that must not call cudaMalloc (which synchronises the device).  The pages
 * have no counterpart to this call; it is this library's own addition.
 * Same arguments and results as pkx_decode_attention_fwd minus
 * workspace/workspace_bytes and the pool format (a bf16 pool).  Its scratch
 * is a fixed 96 MiB device array inside the library that every GPU loading
 * the library holds until exit.  The first call on each device looks up
 * that array's address (make it before any stream capture); the address
 * stays cached for the process, so after cudaDeviceReset this call must not
 * be used again.  Calls share the array: calls that overlap on the GPU race
 * and must be serialised.  A problem whose smallest decode scratch
 * (pkx_decode_workspace_min_size) exceeds 96 MiB returns PKX_EWORKSPACE
 * before anything is enqueued; when pkx_decode_workspace_size also fits,
 * the call runs the two-key-stream schedule, otherwise one stream per unit
 * (same results).  Nothing is allocated.  Device-side errors go to the
 * array's status word, read by pkx_decode_no_alloc_status.
 */
int pkx_decode_attention_fwd_no_alloc(
    const void *q, void *o, const void *k_buffer, const void *v_buffer,
    const int32_t *kv_indptr, const int32_t *kv_indices, int batch, int hq,
    int hkv, int lq, int lv, int64_t kb_ss, int64_t kb_sh, int64_t vb_ss,
    int64_t vb_sh, int64_t num_slots, float sm_scale, float logit_cap,
    int sliding_window, float *lse_out, void *stream);

/*
 * Device status word of the last pkx_decode_attention_fwd_no_alloc call on
 * the current device, as pkx_workspace_status reads a workspace's: copies it
 * to the host (synchronising `stream`) and returns PKX_OK, PKX_EDEVICE or
 * PKX_ETIMEOUT; PKX_ECUDA if the copy fails.  PKX_OK when no such call has
 * run on the device.  Like the entry point it serves, it has no counterpart
 * on the pages.
 */
int pkx_decode_no_alloc_status(void *stream);

/*
 * merge_state.
 * Source: sglang flashinfer_backend.py, forward_extend (the ragged causal
 * extend result and the non-causal paged prefix result, each with its
 * log-sum-exp, combined into one).  For every row r = (token, head):
 *   s = log(exp(s_a) + exp(s_b))
 *   v = exp(s_a - s) * v_a + exp(s_b - s) * v_b
 * A side with s = -inf has weight 0; both -inf gives v = 0, s = -inf.
 *   v_a, v_b, v_out  bf16 [n_tokens, h, dv] contiguous; dv % 8 == 0
 *   s_a, s_b         fp32 [n_tokens, h] (natural log)
 *   s_out            nullable fp32 [n_tokens, h]
 * v_out may alias v_a or v_b (and s_out s_a or s_b): each row is read
 * before it is written.
 */
int pkx_merge_state(const void *v_a, const float *s_a, const void *v_b,
                    const float *s_b, void *v_out, float *s_out,
                    int64_t n_tokens, int h, int dv, void *stream);

/*
 * Unified KV-index build.
 * Source: sglang extend_attention.py, build_unified_kv_indices and
 * _copy_unified_indices_kernel.  For b < batch:
 *   prefix_lens[b]           = prefix_kv_indptr[b+1] - prefix_kv_indptr[b]
 *   unified_kv_indptr[0]     = 0
 *   unified_kv_indptr[b+1]   = unified_kv_indptr[b] + prefix_lens[b]
 *                              + extend_seq_lens[b]
 *   unified_kv_indices[unified_kv_indptr[b] + j]
 *       = prefix_kv_indices[prefix_kv_indptr[b] + j]          (j < P_b)
 *       = extend_kv_indices[extend_start_loc[b] + j - P_b]    (P_b <= j < T_b)
 * Entries of unified_kv_indices past unified_kv_indptr[batch] are left as
 * they were.  Inputs int32; unified_kv_indptr and prefix_lens int32 (written);
 * unified_kv_indices int64 (written), sized >= len(prefix) + len(extend).
 * extend_start_loc[b] is any start offset (it need not be a running sum).
 */
int pkx_build_unified_kv_indices(
    const int32_t *prefix_kv_indptr, const int32_t *prefix_kv_indices,
    const int32_t *extend_start_loc, const int32_t *extend_seq_lens,
    const int32_t *extend_kv_indices, int batch, int32_t *unified_kv_indptr,
    int64_t *unified_kv_indices, int32_t *prefix_lens, void *stream);

/*
 * KV write into the pool.
 * Source: sglang flashinfer_backend.py, forward_extend and forward_decode:
 * before the paged pass, token_to_kv_pool.set_kv_buffer(layer, cache_loc, k,
 * v, ...) stores each new token's K and V rows at its pool slot.  For
 * t < n_tokens and every KV head h:
 *   k_buffer[cache_loc[t], h, :lk] = k[t, h, :lk]
 *   v_buffer[cache_loc[t], h, :lv] = v[t, h, :lv]
 *   k         bf16 [n_tokens, hkv, lk], strides (k_ts, k_hs)
 *   v         bf16 [n_tokens, hkv, lv], strides (v_ts, v_hs), or NULL for a
 *             K-only pool (the MLA pool, whose V is the first lv dims of K):
 *             then v_buffer and its strides are ignored
 *   cache_loc int64 [n_tokens] pool slots (the batch's out_cache_loc)
 *   k_buffer / v_buffer  bf16 pools [num_slots, hkv, lk] / [.., lv] (written)
 * The pool has the inputs' dtype, so the write is an exact copy (the fp8
 * scales of the pages' call do not apply to a bf16 pool).  lk and lv are any
 * positive multiples of 8.  Slots outside [0, num_slots) are skipped, so a
 * bad slot never writes out of the pool.  Two tokens with the same slot leave
 * either one's row there.  Slots not in cache_loc keep their contents.
 */
int pkx_set_kv_buffer(
    const void *k, int64_t k_ts, int64_t k_hs, const void *v, int64_t v_ts,
    int64_t v_hs, const int64_t *cache_loc, int64_t n_tokens, int hkv, int lk,
    int lv, void *k_buffer, int64_t kb_ss, int64_t kb_hs, void *v_buffer,
    int64_t vb_ss, int64_t vb_hs, int64_t num_slots, void *stream);

/*
 * KV write into an fp8 pool.
 * Source: sglang flashinfer_backend.py, set_kv_buffer(layer, cache_loc, k,
 * v, k_scale, v_scale) with an fp8 KV cache.  For t < n_tokens, every KV
 * head h and element d:
 *   k_buffer[cache_loc[t], h, d] = fp8(k[t, h, d] / k_scale)
 *   v_buffer[cache_loc[t], h, d] = fp8(v[t, h, d] / v_scale)
 * where the quotient is an IEEE fp32 division and fp8() rounds to the
 * nearest code, ties to even, and saturates at the largest finite code
 * (448 for e4m3, 57344 for e5m2).  kv_dtype PKX_KV_FP8_E4M3 or
 * PKX_KV_FP8_E5M2; pools of one-byte codes, strides in bytes (multiples of
 * 8); other arguments and rules as pkx_set_kv_buffer.
 */
int pkx_set_kv_buffer_fp8(
    const void *k, int64_t k_ts, int64_t k_hs, const void *v, int64_t v_ts,
    int64_t v_hs, const int64_t *cache_loc, int64_t n_tokens, int hkv, int lk,
    int lv, float k_scale, float v_scale, int kv_dtype, void *k_buffer,
    int64_t kb_ss, int64_t kb_hs, void *v_buffer, int64_t vb_ss,
    int64_t vb_hs, int64_t num_slots, void *stream);

/*
 * KV-index gather from the request-to-token table.
 * Source: sglang flashinfer_backend.py, create_flashinfer_kv_indices_triton
 * and the decode / prefill index updaters that build its kv_indptr.  For
 * b < batch, with kv_start[b] = kv_start_idx[b] (0 when kv_start_idx is
 * NULL):
 *   kv_indptr[0]   = 0
 *   kv_indptr[b+1] = kv_indptr[b] + paged_kernel_lens[b]
 *   kv_indices[kv_indptr[b] + j]
 *       = req_to_token[req_pool_indices[b] * req_to_token_stride
 *                      + kv_start[b] + j]             (j < paged_kernel_lens[b])
 *   req_to_token       int32 [req_to_token_rows, req_to_token_stride]
 *   req_pool_indices,
 *   paged_kernel_lens,
 *   kv_start_idx       int64 [batch] (kv_start_idx nullable); lengths and
 *                      starts are taken as 32-bit, as the pages' gather does
 *   kv_indptr          int32 [batch+1] (written: this call does the running
 *                      sum the pages' callers do before the gather)
 *   kv_indices         int32 [kv_indices_capacity] (written up to
 *                      min(kv_indptr[batch], capacity); the rest untouched)
 * The window updaters pass paged_kernel_lens = the kept tail and
 * kv_start_idx = seq_lens - paged_kernel_lens.  An entry whose source lies
 * outside the table is written as -1 instead of being read.  batch <= 12000
 * (PKX_EUNSUPPORTED above).
 */
int pkx_create_kv_indices(
    const int32_t *req_to_token, int64_t req_to_token_rows,
    int64_t req_to_token_stride, const int64_t *req_pool_indices,
    const int64_t *paged_kernel_lens, const int64_t *kv_start_idx, int batch,
    int32_t *kv_indptr, int32_t *kv_indices, int64_t kv_indices_capacity,
    void *stream);

/*
 * Paged KV indices (page size > 1) to per-token pool slots.
 * Source: sglang flashinfer_backend.py, the paged KV format the wrappers'
 * plan takes: indptr over pages, page indices, last_page_len (entries in
 * each sequence's last page) and page_size, the pool viewed as
 * [pages, page_size, heads, dim].  For b < batch:
 *   pages_b          = kv_indptr[b+1] - kv_indptr[b]
 *   T_b              = pages_b > 0 ? (pages_b - 1) * page_size
 *                                    + kv_last_page_len[b] : 0
 *   token_indptr     = [0, running sum of T_b]                   (written)
 *   token_indices[token_indptr[b] + j]
 *       = kv_indices[kv_indptr[b] + j / page_size] * page_size
 *         + j % page_size                                          (written)
 * The result is the page-size-1 index list every attention call above
 * takes (for the pool viewed as [pages * page_size, heads, dim]).  All
 * arrays int32; token_indices holds token_indices_capacity entries, and
 * none past it is written.  A key whose page would lie past its sequence's
 * pages (kv_last_page_len[b] > page_size) is written as -1, which the
 * attention calls report instead of reading.  batch <= 12000.
 */
int pkx_expand_paged_kv_indices(
    const int32_t *kv_indptr, const int32_t *kv_indices,
    const int32_t *kv_last_page_len, int page_size, int batch,
    int32_t *token_indptr, int32_t *token_indices,
    int64_t token_indices_capacity, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PKX_H */
