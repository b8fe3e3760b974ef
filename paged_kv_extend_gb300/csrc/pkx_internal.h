// pkx_internal.h -- declarations shared by the translation units of libpkx
// (host side): error reporting, workspace layout and the kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <utility>

#include "../../include/pkx.h"

namespace pkx {

// Per-thread error message (pkx_last_error_string).
int set_error(int code, const char *fmt, ...);

// Which key source an attention launch reads.
enum KeyMode : int {
  kTwoStage = 0,  // prefix via int32 kv_indices, extend rows from k/v_extend
  kUnified = 1,   // every key via int64 kv_indices, prefix_lens given
  kDecode = 2,    // every key via int32 kv_indices, query at position T-1
};

// Element format of the KV pool (the values of include/pkx.h's PKX_KV_*).
enum KvFormat : int { kKvBf16 = 0, kKvFp8E4M3 = 1, kKvFp8E5M2 = 2 };

// Which keys a two-stage pass attends to (the ragged + paged split runs the
// extend keys and the prefix keys as two passes and merges them).
enum KeySet : int {
  kAllKeys = 0,
  kPrefixKeys = 1,  // prefix only: every prefix key visible to every extend query
  kExtendKeys = 2,  // extend only: causal over the extend keys
};

// Rows of one query tile (tcgen05 M) and keys of one KV tile.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
// Smallest number of KV tiles a split-KV chunk holds.
constexpr int kMinSplitTiles = 4;
// Upper bound on the shares of a stream partition (CTA pairs of one launch).
constexpr int kMaxStreamParts = 256;

// One unit of attention work: a block of query tokens of one sequence and one
// KV head (up to two Q tiles; in a tile, row = token * group + head-in-group),
// over the key range [k_begin, k_end).
struct __align__(16) WorkUnit {
  int32_t q_tok0;   // first query row in q/o (token index)
  int32_t n_tok;    // tokens in the block
  int32_t qpos0;    // position of the first query token in its sequence
  int32_t kvh;      // KV head
  int32_t k_begin;  // key positions [k_begin, k_end)
  int32_t k_end;
  int32_t k_split;  // keys >= k_split come from the extend rows (two-stage)
  int32_t n_tiles;  // K/V tiles (no tile straddles k_split)
  int32_t b;        // sequence
  int32_t slot;     // -1: write o/lse; else split-KV partial slot
  int32_t dq;       // value-dim slice (0: the kernels take all value dims)
  int32_t claim;    // claim key (cost bucket, largest cost first), for the scheduler
};

// A query block whose key range was split: its partials live in slots
// [slot0, slot0 + n_split).
struct __align__(16) CombineEntry {
  int32_t q_tok0;
  int32_t n_tok;
  int32_t kvh;
  int32_t slot0;
  int32_t n_split;
  int32_t pad[3];
};

// Header at the start of every attention workspace.
struct WsHeader {
  int32_t status;      // PKX_OK / PKX_EDEVICE / PKX_ETIMEOUT (first error wins)
  int32_t n_units;
  int32_t n_combine;
  int32_t split_tiles; // chunk size chosen by the scheduler (tiles)
  int32_t next_unit;   // position in the cost order of the next unclaimed unit
  int32_t pad[59];
};

// Byte offsets of the workspace regions for one problem.
struct WsLayout {
  size_t seq_off;      // int32 [8][batch + 1] per-sequence scratch (five used)
  size_t qb_off;       // int32 [6][qb_max] per-query-block scheduler arrays
  size_t part_off;     // int32 [kMaxStreamParts + 1] first claim position of each share
  size_t units_off;    // WorkUnit [unit_max]
  size_t uorder_off;   // int32 [unit_max] units by cost, largest first
  size_t comb_off;     // CombineEntry [comb_max]
  size_t plse_off;     // float [slot_max][rows_per_slot]
  size_t po_off;       // float [slot_max][rows_per_slot][lv]
  size_t total;
  int qb_max, unit_max, comb_max, slot_max, unit_target, rows_per_slot;
};

int num_sms_current_device();

// Launch `kernel` with programmatic stream serialization: it may start while
// the previous kernel on the stream runs, and waits for it in-kernel
// (grid_dep_wait) before reading its results.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
// Events set by pkx_set_attention_events for this thread (may be null).
void attention_events(cudaEvent_t *before, cudaEvent_t *after);
// Wait limit (ns) and stall hook set by pkx_set_wait_limit_ns /
// pkx_set_stall_injection for this thread.
void wait_settings(uint64_t *wait_ns, int *stall);
int tokens_per_block(int group);
// The split head dims Lq / Lv = 192 / 128 and 288 / 256.
bool split_head_dims(int lq, int lv);
// Q tiles (of 128 rows) per work unit: 2 for Lq = Lv <= 128, else 1.
int q_tiles_per_unit(int lq, int lv);
int rows_per_slot(bool decode, int group, int nqt);
// two_streams: the decode layout with two partial slots per unit (the GQA
// kernel's two key streams); without it decode units run one stream.
WsLayout ws_layout(int batch, int num_q_tokens, int hkv, int group, int lq, int lv, int num_sms,
                   bool decode, bool two_streams = true);

// Arguments of one attention launch (any key mode).
struct AttnArgs {
  int mode;
  const void *q;
  void *o;
  float *lse;
  const void *k_ext, *v_ext;
  int64_t ke_st, ke_sh, ve_st, ve_sh;
  const void *k_buf, *v_buf;
  int64_t kb_ss, kb_sh, vb_ss, vb_sh;
  int64_t num_slots;
  const int32_t *qo_indptr, *kv_indptr, *prefix_lens;
  const void *kv_indices;
  int batch, num_q_tokens, hq, hkv, lq, lv;
  float sm_scale, logit_cap;
  int window;
  const uint8_t *custom_mask;   // nullable: replaces the causal mask
  const int32_t *mask_indptr;   // [batch+1] offsets into custom_mask
  const float *sinks;           // nullable [hq] sink logits
  int kv_fmt = 0;               // pool format: kKvBf16, kKvFp8E4M3, kKvFp8E5M2
  float k_scale = 1.f, v_scale = 1.f;  // fp8 pool: key = code * k_scale, value = code * v_scale
  int key_set = kAllKeys;       // two-stage form: which keys this pass sees
  int keep_status = 0;          // a later pass of one call keeps the status word
  const int64_t *cache_loc = nullptr;  // two-stage: fused KV write of the extend rows
  void *workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
};

int launch_attention(const AttnArgs &a);
int launch_merge_state(const void *v_a, const float *s_a, const void *v_b, const float *s_b,
                       void *v_out, float *s_out, int64_t n, int h, int dv, cudaStream_t s);
int launch_build_unified(const int32_t *prefix_kv_indptr, const int32_t *prefix_kv_indices,
                         const int32_t *extend_start_loc, const int32_t *extend_seq_lens,
                         const int32_t *extend_kv_indices, int batch, int32_t *unified_kv_indptr,
                         int64_t *unified_kv_indices, int32_t *prefix_lens, cudaStream_t s);
int launch_set_kv_buffer(const void *k, int64_t k_ts, int64_t k_hs, const void *v, int64_t v_ts,
                         int64_t v_hs, const int64_t *cache_loc, int64_t n_tokens, int hkv, int lk,
                         int lv, void *k_buffer, int64_t kb_ss, int64_t kb_hs, void *v_buffer,
                         int64_t vb_ss, int64_t vb_hs, int64_t num_slots, cudaStream_t s);
int launch_set_kv_buffer_fp8(const void *k, int64_t k_ts, int64_t k_hs, const void *v,
                             int64_t v_ts, int64_t v_hs, const int64_t *cache_loc,
                             int64_t n_tokens, int hkv, int lk, int lv, float k_scale,
                             float v_scale, int fmt, void *k_buffer, int64_t kb_ss,
                             int64_t kb_hs, void *v_buffer, int64_t vb_ss, int64_t vb_hs,
                             int64_t num_slots, cudaStream_t s);
// Largest batch the index gather takes (its running sum lives in 48 KB of
// shared memory).
constexpr int kGatherMaxBatch = 12000;
int launch_expand_paged(const int32_t *kv_indptr, const int32_t *kv_indices,
                        const int32_t *last_page_len, int page_size, int batch,
                        int32_t *token_indptr, int32_t *token_indices, int64_t capacity,
                        cudaStream_t s);
int launch_create_kv_indices(const int32_t *req_to_token, int64_t rows, int64_t stride,
                             const int64_t *req_pool_indices, const int64_t *paged_kernel_lens,
                             const int64_t *kv_start_idx, int batch, int32_t *kv_indptr,
                             int32_t *kv_indices, int64_t capacity, cudaStream_t s);

}  // namespace pkx
