// api.cu -- the extern "C" entry points of libpkx (declared in include/pkx.h):
// host-side argument validation, then the launchers.  No entry point
// allocates device memory or synchronises the stream (except
// pkx_workspace_status, whose job is to read the device status word).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cuda_runtime.h>

#include "pkx_internal.h"

namespace pkx {

static thread_local char g_err[512] = "";
static thread_local cudaEvent_t g_ev_before = nullptr, g_ev_after = nullptr;
static thread_local uint64_t g_wait_ns = 0;
static thread_local int g_stall = 0;

void attention_events(cudaEvent_t *before, cudaEvent_t *after) {
  *before = g_ev_before;
  *after = g_ev_after;
}

void wait_settings(uint64_t *wait_ns, int *stall) {
  *wait_ns = g_wait_ns ? g_wait_ns : 2000000000ull;
  *stall = g_stall;
}

int set_error(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

static bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static int check_heads(int hq, int hkv, int lq, int lv) {
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0)
    return set_error(PKX_EINVAL, "hq=%d must be a positive multiple of hkv=%d", hq, hkv);
  if (hq / hkv > kBlockM)
    return set_error(PKX_EUNSUPPORTED, "group size hq/hkv=%d > %d not built", hq / hkv, kBlockM);
  const bool ok = (lq == 64 && lv == 64) || (lq == 128 && lv == 128) || (lq == 576 && lv == 512) ||
                  split_head_dims(lq, lv);
  if (!ok) return set_error(PKX_EUNSUPPORTED, "head dims (lq=%d, lv=%d) not built", lq, lv);
  return PKX_OK;
}

static int check_rows(const char *name, const void *p, int64_t s0, int64_t s1) {
  if (!p) return set_error(PKX_EINVAL, "%s is null", name);
  if (!aligned(p, 16)) return set_error(PKX_EINVAL, "%s must be 16-byte aligned", name);
  if (s0 < 0 || s1 < 0 || s0 % 8 || s1 % 8)
    return set_error(PKX_EINVAL, "%s strides (%lld, %lld) must be non-negative multiples of 8",
                     name, (long long)s0, (long long)s1);
  return PKX_OK;
}

// A custom mask needs its offsets.
static int check_mask_sinks(const uint8_t *custom_mask, const int32_t *mask_indptr,
                            const float *sinks) {
  if (custom_mask && (!mask_indptr || !aligned(mask_indptr, 4)))
    return set_error(PKX_EINVAL, "custom_mask needs an aligned int32 mask_indptr");
  if (sinks && !aligned(sinks, 4)) return set_error(PKX_EINVAL, "sinks misaligned");
  return PKX_OK;
}

// The pool's element format and its scales (an fp8 pool: Lq = Lv = 64 or
// 128, or the MLA head 576 / 512; with or without a custom mask).
static int check_kv_format(int kv_dtype, float k_scale, float v_scale, int lq, int lv,
                           bool decode) {
  if (kv_dtype == kKvBf16) return PKX_OK;
  if (kv_dtype != kKvFp8E4M3 && kv_dtype != kKvFp8E5M2)
    return set_error(PKX_EINVAL, "kv_dtype %d is not a PKX_KV_* value", kv_dtype);
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return set_error(PKX_EINVAL, "k_scale and v_scale must be positive and finite");
  if (!((lq == 64 && lv == 64) || (lq == 128 && lv == 128) || (lq == 576 && lv == 512) ||
        (split_head_dims(lq, lv) && !decode)))
    return set_error(PKX_EUNSUPPORTED,
                     "an fp8 pool is built for Lq = Lv = 64 or 128, for Lq / Lv = 576 / 512 and, "
                     "in extend, for the split head dims 192 / 128 and 288 / 256");
  return PKX_OK;
}

static int check_scalars(float sm_scale, float logit_cap) {
  if (!std::isfinite(sm_scale) || !std::isfinite(logit_cap))
    return set_error(PKX_EINVAL, "sm_scale and logit_cap must be finite");
  return PKX_OK;
}

}  // namespace pkx

using namespace pkx;

extern "C" {

const char *pkx_last_error_string(void) { return g_err; }

const char *pkx_version(void) { return "pkx 0.1 (sm_103a)"; }

void pkx_set_attention_events(void *before, void *after) {
  g_ev_before = static_cast<cudaEvent_t>(before);
  g_ev_after = static_cast<cudaEvent_t>(after);
}

void pkx_set_wait_limit_ns(uint64_t ns) { g_wait_ns = ns; }

void pkx_set_stall_injection(int on) { g_stall = on ? 1 : 0; }

size_t pkx_extend_workspace_size(int batch, int num_q_tokens, int hq, int hkv, int lq, int lv) {
  if (batch < 0 || num_q_tokens < 0 || hkv <= 0 || hq <= 0 || hq % hkv || hq / hkv > kBlockM ||
      lv <= 0)
    return 0;
  return ws_layout(batch, num_q_tokens, hkv, hq / hkv, lq, lv, num_sms_current_device(), false)
      .total;
}

size_t pkx_decode_workspace_min_size(int batch, int hq, int hkv, int lq, int lv) {
  if (batch < 0 || hkv <= 0 || hq <= 0 || hq % hkv || hq / hkv > kBlockM || lv <= 0) return 0;
  return ws_layout(batch, batch, hkv, hq / hkv, lq, lv, num_sms_current_device(), true, false)
      .total;
}

size_t pkx_decode_workspace_size(int batch, int hq, int hkv, int lq, int lv) {
  if (batch < 0 || hkv <= 0 || hq <= 0 || hq % hkv || hq / hkv > kBlockM || lv <= 0) return 0;
  return ws_layout(batch, batch, hkv, hq / hkv, lq, lv, num_sms_current_device(), true)
      .total;
}

int pkx_workspace_status(const void *workspace, void *stream) {
  if (!workspace) return set_error(PKX_EINVAL, "workspace is null");
  int32_t st = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&st, workspace, sizeof st, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_error(PKX_ECUDA, "status read: %s", cudaGetErrorString(e));
  if (st == PKX_EDEVICE) return set_error(PKX_EDEVICE, "device-side index or indptr check failed");
  if (st == PKX_ETIMEOUT) return set_error(PKX_ETIMEOUT, "a device wait ran out of time");
  if (st != 0) return set_error(st, "device status %d", st);
  return PKX_OK;
}

}  // extern "C"

// Validation and argument packing shared by the two-stage entry points.
static int two_stage_args(AttnArgs &a, const void *q_extend, const void *k_extend,
                          const void *v_extend, void *o_extend, const void *k_buffer,
                          const void *v_buffer, const int32_t *qo_indptr,
                          const int32_t *kv_indptr, const int32_t *kv_indices, int batch,
                          int num_q_tokens, int hq, int hkv, int lq, int lv, int64_t ke_st,
                          int64_t ke_sh, int64_t ve_st, int64_t ve_sh, int64_t kb_ss,
                          int64_t kb_sh, int64_t vb_ss, int64_t vb_sh, int64_t num_slots,
                          float sm_scale, float logit_cap, int sliding_window,
                          const uint8_t *custom_mask, const int32_t *mask_indptr,
                          const float *sinks, int kv_dtype, float k_scale, float v_scale,
                          float *lse_out, bool *nothing_to_do) {
  int rc;
  *nothing_to_do = false;
  if (batch < 0 || num_q_tokens < 0) return set_error(PKX_EINVAL, "negative batch or token count");
  if ((rc = check_heads(hq, hkv, lq, lv))) return rc;
  if ((rc = check_scalars(sm_scale, logit_cap))) return rc;
  if ((rc = check_mask_sinks(custom_mask, mask_indptr, sinks))) return rc;
  if ((rc = check_kv_format(kv_dtype, k_scale, v_scale, lq, lv, false))) return rc;
  if (batch == 0 || num_q_tokens == 0) {
    *nothing_to_do = true;
    return PKX_OK;
  }
  if ((rc = check_rows("q_extend", q_extend, 8, 8))) return rc;
  if ((rc = check_rows("o_extend", o_extend, 8, 8))) return rc;
  if ((rc = check_rows("k_extend", k_extend, ke_st, ke_sh))) return rc;
  if ((rc = check_rows("v_extend", v_extend, ve_st, ve_sh))) return rc;
  if ((rc = check_rows("k_buffer", k_buffer, kb_ss, kb_sh))) return rc;
  if ((rc = check_rows("v_buffer", v_buffer, vb_ss, vb_sh))) return rc;
  if (!qo_indptr || !kv_indptr || !aligned(qo_indptr, 4) || !aligned(kv_indptr, 4))
    return set_error(PKX_EINVAL, "qo_indptr / kv_indptr null or misaligned");
  if (kv_indices && !aligned(kv_indices, 4)) return set_error(PKX_EINVAL, "kv_indices misaligned");
  if (lse_out && !aligned(lse_out, 4)) return set_error(PKX_EINVAL, "lse_out misaligned");
  if (num_slots <= 0) return set_error(PKX_EINVAL, "num_slots must be positive");
  a.mode = kTwoStage;
  a.q = q_extend;
  a.o = o_extend;
  a.lse = lse_out;
  a.k_ext = k_extend;
  a.v_ext = v_extend;
  a.ke_st = ke_st; a.ke_sh = ke_sh; a.ve_st = ve_st; a.ve_sh = ve_sh;
  a.k_buf = k_buffer;
  a.v_buf = v_buffer;
  a.kb_ss = kb_ss; a.kb_sh = kb_sh; a.vb_ss = vb_ss; a.vb_sh = vb_sh;
  a.num_slots = num_slots;
  a.qo_indptr = qo_indptr;
  a.kv_indptr = kv_indptr;
  a.prefix_lens = nullptr;
  a.kv_indices = kv_indices;
  a.batch = batch; a.num_q_tokens = num_q_tokens; a.hq = hq; a.hkv = hkv; a.lq = lq; a.lv = lv;
  a.sm_scale = sm_scale; a.logit_cap = logit_cap; a.window = sliding_window;
  a.custom_mask = custom_mask; a.mask_indptr = mask_indptr; a.sinks = sinks;
  a.kv_fmt = kv_dtype; a.k_scale = k_scale; a.v_scale = v_scale;
  return PKX_OK;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace of the ragged + paged split: one attention pass's scratch (the
// passes run one after the other on the stream and share it), the paged
// pass's bf16 output and both passes' lse.
struct SplitLayout {
  size_t attn, o_paged, lse_paged, lse_ragged, total;
};

static SplitLayout split_layout(int batch, int num_q_tokens, int hq, int hkv, int lq, int lv) {
  SplitLayout L;
  L.attn = 0;
  const size_t attn = align256(ws_layout(batch, num_q_tokens, hkv, hq / hkv, lq, lv,
                                         num_sms_current_device(), false).total);
  const size_t rows = (size_t)num_q_tokens * hq;
  L.o_paged = attn;
  L.lse_paged = L.o_paged + align256(rows * lv * 2);
  L.lse_ragged = L.lse_paged + align256(rows * 4);
  L.total = L.lse_ragged + align256(rows * 4);
  return L;
}

extern "C" {

int pkx_extend_attention_fwd(const void *q_extend, const void *k_extend, const void *v_extend,
                             void *o_extend, const void *k_buffer, const void *v_buffer,
                             const int32_t *qo_indptr, const int32_t *kv_indptr,
                             const int32_t *kv_indices, int batch, int num_q_tokens, int hq,
                             int hkv, int lq, int lv, int64_t ke_st, int64_t ke_sh,
                             int64_t ve_st, int64_t ve_sh, int64_t kb_ss, int64_t kb_sh,
                             int64_t vb_ss, int64_t vb_sh, int64_t num_slots, float sm_scale,
                             float logit_cap, int sliding_window, const uint8_t *custom_mask,
                             const int32_t *mask_indptr, const float *sinks, int kv_dtype,
                             float k_scale, float v_scale, float *lse_out, void *workspace,
                             size_t workspace_bytes, void *stream) {
  AttnArgs a{};
  bool done;
  int rc = two_stage_args(a, q_extend, k_extend, v_extend, o_extend, k_buffer, v_buffer,
                          qo_indptr, kv_indptr, kv_indices, batch, num_q_tokens, hq, hkv, lq, lv,
                          ke_st, ke_sh, ve_st, ve_sh, kb_ss, kb_sh, vb_ss, vb_sh, num_slots,
                          sm_scale, logit_cap, sliding_window, custom_mask, mask_indptr, sinks,
                          kv_dtype, k_scale, v_scale, lse_out, &done);
  if (rc != PKX_OK || done) return rc;
  a.workspace = workspace; a.workspace_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  return launch_attention(a);
}

int pkx_extend_attention_fwd_kv_write(
    const void *q_extend, const void *k_extend, const void *v_extend, void *o_extend,
    void *k_buffer, void *v_buffer, const int32_t *qo_indptr, const int32_t *kv_indptr,
    const int32_t *kv_indices, int batch, int num_q_tokens, int hq, int hkv, int lq, int lv,
    int64_t ke_st, int64_t ke_sh, int64_t ve_st, int64_t ve_sh, int64_t kb_ss, int64_t kb_sh,
    int64_t vb_ss, int64_t vb_sh, int64_t num_slots, float sm_scale, float logit_cap,
    int sliding_window, const uint8_t *custom_mask, const int32_t *mask_indptr,
    const float *sinks, int kv_dtype, float k_scale, float v_scale, float *lse_out,
    const int64_t *cache_loc, void *workspace, size_t workspace_bytes, void *stream) {
  AttnArgs a{};
  bool done;
  int rc = two_stage_args(a, q_extend, k_extend, v_extend, o_extend, k_buffer, v_buffer,
                          qo_indptr, kv_indptr, kv_indices, batch, num_q_tokens, hq, hkv, lq, lv,
                          ke_st, ke_sh, ve_st, ve_sh, kb_ss, kb_sh, vb_ss, vb_sh, num_slots,
                          sm_scale, logit_cap, sliding_window, custom_mask, mask_indptr, sinks,
                          kv_dtype, k_scale, v_scale, lse_out, &done);
  if (rc != PKX_OK || done) return rc;
  if (!cache_loc || !aligned(cache_loc, 8))
    return set_error(PKX_EINVAL, "cache_loc null or misaligned");
  a.workspace = workspace; a.workspace_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  const bool mla = lq == 576 && lv == 512;
  if (mla || kv_dtype != kKvBf16) {
    // not fused for these pools: the standalone write first, as the pages
    // order it (the MLA pool stores only the K row; V is its first 512 dims)
    rc = kv_dtype != kKvBf16
             ? pkx_set_kv_buffer_fp8(k_extend, ke_st, ke_sh, mla ? nullptr : v_extend, ve_st,
                                     ve_sh, cache_loc, num_q_tokens, hkv, lq, lv, k_scale,
                                     v_scale, kv_dtype, k_buffer, kb_ss, kb_sh, v_buffer, vb_ss,
                                     vb_sh, num_slots, stream)
             : pkx_set_kv_buffer(k_extend, ke_st, ke_sh, nullptr, ve_st, ve_sh, cache_loc,
                                 num_q_tokens, hkv, lq, lv, k_buffer, kb_ss, kb_sh, v_buffer,
                                 vb_ss, vb_sh, num_slots, stream);
    if (rc != PKX_OK) return rc;
    return launch_attention(a);
  }
  a.cache_loc = cache_loc;
  return launch_attention(a);
}

size_t pkx_ragged_paged_workspace_size(int batch, int num_q_tokens, int hq, int hkv, int lq,
                                       int lv) {
  if (batch < 0 || num_q_tokens < 0 || hkv <= 0 || hq <= 0 || hq % hkv || hq / hkv > kBlockM ||
      lv <= 0)
    return 0;
  return split_layout(batch, num_q_tokens, hq, hkv, lq, lv).total;
}

int pkx_extend_attention_fwd_ragged_paged(
    const void *q_extend, const void *k_extend, const void *v_extend, void *o_extend,
    const void *k_buffer, const void *v_buffer, const int32_t *qo_indptr,
    const int32_t *kv_indptr, const int32_t *kv_indices, int batch, int num_q_tokens, int hq,
    int hkv, int lq, int lv, int64_t ke_st, int64_t ke_sh, int64_t ve_st, int64_t ve_sh,
    int64_t kb_ss, int64_t kb_sh, int64_t vb_ss, int64_t vb_sh, int64_t num_slots,
    float sm_scale, float logit_cap, int sliding_window, int kv_dtype, float k_scale,
    float v_scale, float *lse_out, void *workspace, size_t workspace_bytes, void *stream) {
  AttnArgs a{};
  bool done;
  int rc = two_stage_args(a, q_extend, k_extend, v_extend, o_extend, k_buffer, v_buffer,
                          qo_indptr, kv_indptr, kv_indices, batch, num_q_tokens, hq, hkv, lq, lv,
                          ke_st, ke_sh, ve_st, ve_sh, kb_ss, kb_sh, vb_ss, vb_sh, num_slots,
                          sm_scale, logit_cap, sliding_window, nullptr, nullptr, nullptr,
                          kv_dtype, k_scale, v_scale, lse_out, &done);
  if (rc != PKX_OK || done) return rc;
  const SplitLayout L = split_layout(batch, num_q_tokens, hq, hkv, lq, lv);
  if (!workspace || workspace_bytes < L.total)
    return set_error(PKX_EWORKSPACE, "workspace of %zu bytes given, %zu needed", workspace_bytes,
                     L.total);
  if (reinterpret_cast<uintptr_t>(workspace) & 255)
    return set_error(PKX_EINVAL, "workspace must be 256-byte aligned");
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  void *o_paged = ws + L.o_paged;
  float *lse_paged = reinterpret_cast<float *>(ws + L.lse_paged);
  float *lse_ragged = reinterpret_cast<float *>(ws + L.lse_ragged);
  a.workspace = ws + L.attn;
  a.workspace_bytes = L.o_paged - L.attn;
  a.stream = static_cast<cudaStream_t>(stream);
  // ragged pass: extend keys only, causal, straight into o_extend
  a.key_set = kExtendKeys;
  a.lse = lse_ragged;
  if ((rc = launch_attention(a)) != PKX_OK) return rc;
  // paged pass: prefix keys only, all visible, into the workspace
  a.key_set = kPrefixKeys;
  a.keep_status = 1;
  a.o = o_paged;
  a.lse = lse_paged;
  if ((rc = launch_attention(a)) != PKX_OK) return rc;
  // merge the two states in place
  return launch_merge_state(o_extend, lse_ragged, o_paged, lse_paged, o_extend, lse_out,
                            num_q_tokens, hq, lv, a.stream);
}

int pkx_extend_attention_fwd_unified(const void *q, void *o, const void *k_buffer,
                                     const void *v_buffer, const int32_t *qo_indptr,
                                     const int32_t *kv_indptr, const int64_t *kv_indices,
                                     const int32_t *prefix_lens, int batch, int num_q_tokens,
                                     int hq, int hkv, int lq, int lv, int64_t kb_ss,
                                     int64_t kb_sh, int64_t vb_ss, int64_t vb_sh,
                                     int64_t num_slots, float sm_scale, float logit_cap,
                                     int sliding_window, const uint8_t *custom_mask,
                                     const int32_t *mask_indptr, const float *sinks,
                                     int kv_dtype, float k_scale, float v_scale, float *lse_out,
                                     void *workspace, size_t workspace_bytes, void *stream) {
  int rc;
  if (batch < 0 || num_q_tokens < 0) return set_error(PKX_EINVAL, "negative batch or token count");
  if ((rc = check_heads(hq, hkv, lq, lv))) return rc;
  if ((rc = check_scalars(sm_scale, logit_cap))) return rc;
  if ((rc = check_mask_sinks(custom_mask, mask_indptr, sinks))) return rc;
  if ((rc = check_kv_format(kv_dtype, k_scale, v_scale, lq, lv, false))) return rc;
  if (batch == 0 || num_q_tokens == 0) return PKX_OK;
  if ((rc = check_rows("q", q, 8, 8))) return rc;
  if ((rc = check_rows("o", o, 8, 8))) return rc;
  if ((rc = check_rows("k_buffer", k_buffer, kb_ss, kb_sh))) return rc;
  if ((rc = check_rows("v_buffer", v_buffer, vb_ss, vb_sh))) return rc;
  if (!qo_indptr || !kv_indptr || !prefix_lens || !aligned(qo_indptr, 4) ||
      !aligned(kv_indptr, 4) || !aligned(prefix_lens, 4))
    return set_error(PKX_EINVAL, "qo_indptr / kv_indptr / prefix_lens null or misaligned");
  if (kv_indices && !aligned(kv_indices, 8)) return set_error(PKX_EINVAL, "kv_indices misaligned");
  if (lse_out && !aligned(lse_out, 4)) return set_error(PKX_EINVAL, "lse_out misaligned");
  if (num_slots <= 0) return set_error(PKX_EINVAL, "num_slots must be positive");
  AttnArgs a{};
  a.mode = kUnified;
  a.q = q;
  a.o = o;
  a.lse = lse_out;
  a.k_buf = k_buffer;
  a.v_buf = v_buffer;
  a.kb_ss = kb_ss; a.kb_sh = kb_sh; a.vb_ss = vb_ss; a.vb_sh = vb_sh;
  a.num_slots = num_slots;
  a.qo_indptr = qo_indptr;
  a.kv_indptr = kv_indptr;
  a.prefix_lens = prefix_lens;
  a.kv_indices = kv_indices;
  a.batch = batch; a.num_q_tokens = num_q_tokens; a.hq = hq; a.hkv = hkv; a.lq = lq; a.lv = lv;
  a.sm_scale = sm_scale; a.logit_cap = logit_cap; a.window = sliding_window;
  a.custom_mask = custom_mask; a.mask_indptr = mask_indptr; a.sinks = sinks;
  a.kv_fmt = kv_dtype; a.k_scale = k_scale; a.v_scale = v_scale;
  a.workspace = workspace; a.workspace_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  return launch_attention(a);
}

int pkx_decode_attention_fwd(const void *q, void *o, const void *k_buffer, const void *v_buffer,
                             const int32_t *kv_indptr, const int32_t *kv_indices, int batch,
                             int hq, int hkv, int lq, int lv, int64_t kb_ss, int64_t kb_sh,
                             int64_t vb_ss, int64_t vb_sh, int64_t num_slots, float sm_scale,
                             float logit_cap, int sliding_window, int kv_dtype, float k_scale,
                             float v_scale, float *lse_out, void *workspace,
                             size_t workspace_bytes, void *stream) {
  int rc;
  if (batch < 0) return set_error(PKX_EINVAL, "negative batch");
  if ((rc = check_heads(hq, hkv, lq, lv))) return rc;
  if ((rc = check_scalars(sm_scale, logit_cap))) return rc;
  if ((rc = check_kv_format(kv_dtype, k_scale, v_scale, lq, lv, true))) return rc;
  if (batch == 0) return PKX_OK;
  if ((rc = check_rows("q", q, 8, 8))) return rc;
  if ((rc = check_rows("o", o, 8, 8))) return rc;
  if ((rc = check_rows("k_buffer", k_buffer, kb_ss, kb_sh))) return rc;
  if ((rc = check_rows("v_buffer", v_buffer, vb_ss, vb_sh))) return rc;
  if (!kv_indptr || !aligned(kv_indptr, 4))
    return set_error(PKX_EINVAL, "kv_indptr null or misaligned");
  if (kv_indices && !aligned(kv_indices, 4)) return set_error(PKX_EINVAL, "kv_indices misaligned");
  if (lse_out && !aligned(lse_out, 4)) return set_error(PKX_EINVAL, "lse_out misaligned");
  if (num_slots <= 0) return set_error(PKX_EINVAL, "num_slots must be positive");
  AttnArgs a{};
  a.mode = kDecode;
  a.q = q;
  a.o = o;
  a.lse = lse_out;
  a.k_buf = k_buffer;
  a.v_buf = v_buffer;
  a.kb_ss = kb_ss; a.kb_sh = kb_sh; a.vb_ss = vb_ss; a.vb_sh = vb_sh;
  a.num_slots = num_slots;
  a.qo_indptr = nullptr;
  a.kv_indptr = kv_indptr;
  a.prefix_lens = nullptr;
  a.kv_indices = kv_indices;
  a.batch = batch; a.num_q_tokens = batch; a.hq = hq; a.hkv = hkv; a.lq = lq; a.lv = lv;
  a.sm_scale = sm_scale; a.logit_cap = logit_cap; a.window = sliding_window;
  a.kv_fmt = kv_dtype; a.k_scale = k_scale; a.v_scale = v_scale;
  a.workspace = workspace; a.workspace_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  return launch_attention(a);
}

int pkx_merge_state(const void *v_a, const float *s_a, const void *v_b, const float *s_b,
                    void *v_out, float *s_out, int64_t n_tokens, int h, int dv, void *stream) {
  if (n_tokens < 0 || h <= 0 || dv <= 0 || dv % 8)
    return set_error(PKX_EINVAL, "merge_state: n_tokens >= 0, h > 0, dv a positive multiple of 8");
  if (n_tokens == 0) return PKX_OK;
  if (!v_a || !v_b || !v_out || !s_a || !s_b)
    return set_error(PKX_EINVAL, "merge_state: null input or output");
  if (!aligned(v_a, 16) || !aligned(v_b, 16) || !aligned(v_out, 16) || !aligned(s_a, 4) ||
      !aligned(s_b, 4) || (s_out && !aligned(s_out, 4)))
    return set_error(PKX_EINVAL, "merge_state: misaligned pointer");
  return launch_merge_state(v_a, s_a, v_b, s_b, v_out, s_out, n_tokens, h, dv,
                            static_cast<cudaStream_t>(stream));
}

int pkx_build_unified_kv_indices(const int32_t *prefix_kv_indptr,
                                 const int32_t *prefix_kv_indices,
                                 const int32_t *extend_start_loc, const int32_t *extend_seq_lens,
                                 const int32_t *extend_kv_indices, int batch,
                                 int32_t *unified_kv_indptr, int64_t *unified_kv_indices,
                                 int32_t *prefix_lens, void *stream) {
  if (batch < 0) return set_error(PKX_EINVAL, "negative batch");
  if (!prefix_kv_indptr || !unified_kv_indptr)
    return set_error(PKX_EINVAL, "prefix_kv_indptr / unified_kv_indptr null");
  if (batch > 0 && (!extend_start_loc || !extend_seq_lens || !prefix_lens || !unified_kv_indices))
    return set_error(PKX_EINVAL, "null argument");
  if (!aligned(unified_kv_indices, 8)) return set_error(PKX_EINVAL, "unified_kv_indices misaligned");
  return launch_build_unified(prefix_kv_indptr, prefix_kv_indices, extend_start_loc,
                              extend_seq_lens, extend_kv_indices, batch, unified_kv_indptr,
                              unified_kv_indices, prefix_lens, static_cast<cudaStream_t>(stream));
}

int pkx_set_kv_buffer(const void *k, int64_t k_ts, int64_t k_hs, const void *v, int64_t v_ts,
                      int64_t v_hs, const int64_t *cache_loc, int64_t n_tokens, int hkv, int lk,
                      int lv, void *k_buffer, int64_t kb_ss, int64_t kb_hs, void *v_buffer,
                      int64_t vb_ss, int64_t vb_hs, int64_t num_slots, void *stream) {
  if (n_tokens < 0 || hkv <= 0 || lk <= 0 || lk % 8 || (v && (lv <= 0 || lv % 8)))
    return set_error(PKX_EINVAL,
                     "set_kv_buffer: n_tokens >= 0, hkv > 0, lk (and lv) positive multiples of 8");
  if (num_slots < 0) return set_error(PKX_EINVAL, "set_kv_buffer: negative num_slots");
  if (n_tokens == 0) return PKX_OK;
  if (!cache_loc || !aligned(cache_loc, 8))
    return set_error(PKX_EINVAL, "set_kv_buffer: cache_loc null or misaligned");
  int rc;
  if ((rc = check_rows("k", k, k_ts, k_hs)) != PKX_OK) return rc;
  if ((rc = check_rows("k_buffer", k_buffer, kb_ss, kb_hs)) != PKX_OK) return rc;
  if (v) {
    if ((rc = check_rows("v", v, v_ts, v_hs)) != PKX_OK) return rc;
    if ((rc = check_rows("v_buffer", v_buffer, vb_ss, vb_hs)) != PKX_OK) return rc;
  }
  return launch_set_kv_buffer(k, k_ts, k_hs, v, v_ts, v_hs, cache_loc, n_tokens, hkv, lk, lv,
                              k_buffer, kb_ss, kb_hs, v_buffer, vb_ss, vb_hs, num_slots,
                              static_cast<cudaStream_t>(stream));
}

int pkx_set_kv_buffer_fp8(const void *k, int64_t k_ts, int64_t k_hs, const void *v,
                          int64_t v_ts, int64_t v_hs, const int64_t *cache_loc, int64_t n_tokens,
                          int hkv, int lk, int lv, float k_scale, float v_scale, int kv_dtype,
                          void *k_buffer, int64_t kb_ss, int64_t kb_hs, void *v_buffer,
                          int64_t vb_ss, int64_t vb_hs, int64_t num_slots, void *stream) {
  if (kv_dtype != kKvFp8E4M3 && kv_dtype != kKvFp8E5M2)
    return set_error(PKX_EINVAL, "set_kv_buffer_fp8: kv_dtype must be an fp8 PKX_KV_* value");
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return set_error(PKX_EINVAL, "set_kv_buffer_fp8: scales must be positive and finite");
  if (n_tokens < 0 || hkv <= 0 || lk <= 0 || lk % 8 || (v && (lv <= 0 || lv % 8)))
    return set_error(PKX_EINVAL,
                     "set_kv_buffer_fp8: n_tokens >= 0, hkv > 0, lk (and lv) multiples of 8");
  if (num_slots < 0) return set_error(PKX_EINVAL, "set_kv_buffer_fp8: negative num_slots");
  if (n_tokens == 0) return PKX_OK;
  if (!cache_loc || !aligned(cache_loc, 8))
    return set_error(PKX_EINVAL, "set_kv_buffer_fp8: cache_loc null or misaligned");
  int rc;
  if ((rc = check_rows("k", k, k_ts, k_hs)) != PKX_OK) return rc;
  if ((rc = check_rows("k_buffer", k_buffer, kb_ss, kb_hs)) != PKX_OK) return rc;
  if (v) {
    if ((rc = check_rows("v", v, v_ts, v_hs)) != PKX_OK) return rc;
    if ((rc = check_rows("v_buffer", v_buffer, vb_ss, vb_hs)) != PKX_OK) return rc;
  }
  return launch_set_kv_buffer_fp8(k, k_ts, k_hs, v, v_ts, v_hs, cache_loc, n_tokens, hkv, lk, lv,
                                  k_scale, v_scale, kv_dtype, k_buffer, kb_ss, kb_hs, v_buffer,
                                  vb_ss, vb_hs, num_slots, static_cast<cudaStream_t>(stream));
}

int pkx_expand_paged_kv_indices(const int32_t *kv_indptr, const int32_t *kv_indices,
                                const int32_t *kv_last_page_len, int page_size, int batch,
                                int32_t *token_indptr, int32_t *token_indices,
                                int64_t token_indices_capacity, void *stream) {
  if (batch < 0 || batch > kGatherMaxBatch)
    return set_error(PKX_EUNSUPPORTED, "expand_paged_kv_indices: batch %d outside [0, %d]",
                     batch, kGatherMaxBatch);
  if (page_size <= 0) return set_error(PKX_EINVAL, "expand_paged_kv_indices: page_size <= 0");
  if (token_indices_capacity < 0)
    return set_error(PKX_EINVAL, "expand_paged_kv_indices: negative capacity");
  if (!token_indptr || !aligned(token_indptr, 4))
    return set_error(PKX_EINVAL, "expand_paged_kv_indices: token_indptr null or misaligned");
  if (batch > 0) {
    if (!kv_indptr || !kv_last_page_len || !aligned(kv_indptr, 4) ||
        !aligned(kv_last_page_len, 4) || (kv_indices && !aligned(kv_indices, 4)))
      return set_error(PKX_EINVAL, "expand_paged_kv_indices: null or misaligned input");
    if (token_indices_capacity > 0 && (!token_indices || !aligned(token_indices, 4)))
      return set_error(PKX_EINVAL, "expand_paged_kv_indices: token_indices null or misaligned");
  }
  return launch_expand_paged(kv_indptr, kv_indices, kv_last_page_len, page_size, batch,
                             token_indptr, token_indices, token_indices_capacity,
                             static_cast<cudaStream_t>(stream));
}

int pkx_create_kv_indices(const int32_t *req_to_token, int64_t req_to_token_rows,
                          int64_t req_to_token_stride, const int64_t *req_pool_indices,
                          const int64_t *paged_kernel_lens, const int64_t *kv_start_idx,
                          int batch, int32_t *kv_indptr, int32_t *kv_indices,
                          int64_t kv_indices_capacity, void *stream) {
  if (batch < 0 || batch > kGatherMaxBatch)
    return set_error(PKX_EUNSUPPORTED, "create_kv_indices: batch %d outside [0, %d]", batch,
                     kGatherMaxBatch);
  if (req_to_token_rows < 0 || req_to_token_stride < 0 || kv_indices_capacity < 0)
    return set_error(PKX_EINVAL, "create_kv_indices: negative table size or capacity");
  if (!kv_indptr || !aligned(kv_indptr, 4))
    return set_error(PKX_EINVAL, "create_kv_indices: kv_indptr null or misaligned");
  if (batch > 0) {
    if (!req_pool_indices || !paged_kernel_lens || !aligned(req_pool_indices, 8) ||
        !aligned(paged_kernel_lens, 8) || (kv_start_idx && !aligned(kv_start_idx, 8)))
      return set_error(PKX_EINVAL, "create_kv_indices: null or misaligned per-sequence array");
    if (kv_indices_capacity > 0 && (!kv_indices || !aligned(kv_indices, 4)))
      return set_error(PKX_EINVAL, "create_kv_indices: kv_indices null or misaligned");
    if (req_to_token_rows > 0 && req_to_token_stride > 0 &&
        (!req_to_token || !aligned(req_to_token, 4)))
      return set_error(PKX_EINVAL, "create_kv_indices: req_to_token null or misaligned");
  }
  return launch_create_kv_indices(req_to_token, req_to_token_rows, req_to_token_stride,
                                  req_pool_indices, paged_kernel_lens, kv_start_idx, batch,
                                  kv_indptr, kv_indices, kv_indices_capacity,
                                  static_cast<cudaStream_t>(stream));
}

}  // extern "C"
