// kv_cache_ops.cu -- the two steps on either side of the attention call in
// sglang flashinfer_backend.py:
//
//  * set_kv_buffer (forward_extend / forward_decode): each new token's K and
//    V rows go into the page-size-1 pool at slot cache_loc[t], every KV head.
//  * create_flashinfer_kv_indices_triton (decode and prefill index updaters):
//    kv_indptr = [0, running sum of paged_kernel_lens], and sequence b's
//    kv_indices are the row slice req_to_token[req_pool_indices[b],
//    kv_start[b] .. kv_start[b] + paged_kernel_lens[b]).
//
// Both are pure data movement, bounded by HBM bandwidth.
//
// KV write: the work is a flat list of 16-byte chunks, (token, head, chunk of
// the K row then of the V row).  A (token, head) row is contiguous in the
// input and in the pool, so consecutive threads move consecutive 16-byte
// chunks of one row and each row's stores are whole 32-byte sectors.  Every
// thread keeps kUnroll chunks in flight (all loads, then all stores).  The
// grid is a multiple of the SM count with a grid-stride loop.
//
// Index gather: one launch does both the running sum and the copy.  Every CTA
// loads the lengths of the whole batch into shared memory and scans them
// (the batch is small next to the index count: a few KB of L2 reads per CTA),
// CTA 0 writes kv_indptr, and the index range [0, kv_indptr[batch]) is split
// evenly over the CTAs, so one long sequence does not serialise on one CTA as
// it would with a CTA per sequence.  A thread finds the sequence of its entry
// by binary search in the shared running sum.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "pkx_internal.h"

namespace pkx {

// ------------------------------------------------------------ KV write
constexpr int kKvThreads = 256;
constexpr int kUnroll = 4;

struct KvWriteArgs {
  const uint4 *k, *v;
  int64_t k_ts, k_hs, v_ts, v_hs;  // strides in 16-byte chunks
  const int64_t *cache_loc;
  uint4 *k_buf, *v_buf;
  int64_t kb_ss, kb_hs, vb_ss, vb_hs;
  int64_t num_slots;
  uint32_t hkv, ck, cv;            // heads, chunks per K row, per V row (0: K only)
  uint64_t total;                  // n_tokens * hkv * (ck + cv)
};

// Source chunk i and the token it belongs to.  The source address does not
// depend on the slot, so the data load and the slot load go out together.
__device__ __forceinline__ const uint4 *kv_chunk_src(const KvWriteArgs &a, uint32_t i,
                                                     uint32_t &t, uint32_t &h, uint32_t &c) {
  const uint32_t per_row = a.ck + a.cv;
  const uint32_t row = i / per_row;
  c = i - row * per_row;
  t = row / a.hkv;
  h = row - t * a.hkv;
  return c < a.ck ? a.k + (int64_t)t * a.k_ts + (int64_t)h * a.k_hs + c
                  : a.v + (int64_t)t * a.v_ts + (int64_t)h * a.v_hs + (c - a.ck);
}

__global__ void __launch_bounds__(kKvThreads) set_kv_buffer_kernel(const KvWriteArgs a) {
  // i < total < 2^31 (the launcher checks): 32-bit indices cannot overflow
  const uint32_t total = (uint32_t)a.total;
  const uint32_t stride = gridDim.x * kKvThreads;
  for (uint32_t base = blockIdx.x * kKvThreads + threadIdx.x; base < total;
       base += stride * kUnroll) {
    uint4 val[kUnroll];
    int64_t slot[kUnroll];
    uint32_t hh[kUnroll], cc[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t i = base + u * stride;
      slot[u] = -1;
      if (i < total) {
        uint32_t t;
        const uint4 *src = kv_chunk_src(a, i, t, hh[u], cc[u]);
        slot[u] = __ldg(a.cache_loc + t);
        val[u] = __ldg(src);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (slot[u] < 0 || slot[u] >= a.num_slots) continue;  // outside the pool: skipped
      uint4 *dst = cc[u] < a.ck
                       ? a.k_buf + slot[u] * a.kb_ss + (int64_t)hh[u] * a.kb_hs + cc[u]
                       : a.v_buf + slot[u] * a.vb_ss + (int64_t)hh[u] * a.vb_hs + (cc[u] - a.ck);
      *dst = val[u];
    }
  }
}

int launch_set_kv_buffer(const void *k, int64_t k_ts, int64_t k_hs, const void *v, int64_t v_ts,
                         int64_t v_hs, const int64_t *cache_loc, int64_t n_tokens, int hkv, int lk,
                         int lv, void *k_buffer, int64_t kb_ss, int64_t kb_hs, void *v_buffer,
                         int64_t vb_ss, int64_t vb_hs, int64_t num_slots, cudaStream_t st) {
  KvWriteArgs a;
  a.k = static_cast<const uint4 *>(k);
  a.v = static_cast<const uint4 *>(v);
  a.k_ts = k_ts / 8; a.k_hs = k_hs / 8; a.v_ts = v_ts / 8; a.v_hs = v_hs / 8;
  a.cache_loc = cache_loc;
  a.k_buf = static_cast<uint4 *>(k_buffer);
  a.v_buf = static_cast<uint4 *>(v_buffer);
  a.kb_ss = kb_ss / 8; a.kb_hs = kb_hs / 8; a.vb_ss = vb_ss / 8; a.vb_hs = vb_hs / 8;
  a.num_slots = num_slots;
  a.hkv = (uint32_t)hkv;
  a.ck = (uint32_t)(lk / 8);
  a.cv = v ? (uint32_t)(lv / 8) : 0u;
  a.total = (uint64_t)n_tokens * a.hkv * (a.ck + a.cv);
  if (a.total == 0) return PKX_OK;
  if (a.total >= (1ull << 31))
    return set_error(PKX_EUNSUPPORTED, "set_kv_buffer: 2^31 or more 16-byte chunks in one call");
  const int nsm = num_sms_current_device();
  const uint64_t need = (a.total + kKvThreads * kUnroll - 1) / (kKvThreads * kUnroll);
  static int resident = 0;  // CTAs per SM at this kernel's register count
  if (resident == 0) {
    int r = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, set_kv_buffer_kernel, kKvThreads, 0) !=
            cudaSuccess || r < 1)
      r = 4;
    resident = r;
  }
  const uint64_t cap = (uint64_t)nsm * resident;  // one resident wave
  const unsigned grid = (unsigned)(need < cap ? need : cap);
  set_kv_buffer_kernel<<<grid, kKvThreads, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_error(PKX_ECUDA, "set_kv_buffer launch: %s", cudaGetErrorString(e));
  return PKX_OK;
}

// ------------------------------------------------------------ KV write, fp8 pool
// The same flat list of 16-byte input chunks (8 bf16); each becomes 8 fp8
// codes (an 8-byte store): element / scale in IEEE fp32, then the nearest
// code, ties to even, saturating at the largest finite one.
struct KvWriteFp8Args {
  const uint4 *k, *v;
  int64_t k_ts, k_hs, v_ts, v_hs;  // input strides in 16-byte chunks
  const int64_t *cache_loc;
  uint2 *k_buf, *v_buf;
  int64_t kb_ss, kb_hs, vb_ss, vb_hs;  // pool strides in 8-byte chunks
  int64_t num_slots;
  uint32_t hkv, ck, cv;
  uint64_t total;
  float k_scale, v_scale;
};

template <int FMT>
__device__ __forceinline__ uint2 bf16x8_to_fp8x8(uint4 in, float scale) {
  constexpr __nv_fp8_interpretation_t kind = FMT == 1 ? __NV_E4M3 : __NV_E5M2;
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  uint32_t out[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
    const float2 f = __bfloat1622float2(b);
    const float2 q = make_float2(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale));
    const uint32_t two = __nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, kind);
    out[i >> 1] |= (two & 0xFFFFu) << (16 * (i & 1));
  }
  return make_uint2(out[0], out[1]);
}

template <int FMT>
__global__ void __launch_bounds__(kKvThreads) set_kv_buffer_fp8_kernel(const KvWriteFp8Args a) {
  const uint32_t total = (uint32_t)a.total;  // < 2^31 (the launcher checks)
  const uint32_t stride = gridDim.x * kKvThreads;
  const uint32_t per_row = a.ck + a.cv;
  for (uint32_t base = blockIdx.x * kKvThreads + threadIdx.x; base < total;
       base += stride * kUnroll) {
    uint4 val[kUnroll];
    int64_t slot[kUnroll];
    uint32_t hh[kUnroll], cc[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t i = base + u * stride;
      slot[u] = -1;
      if (i < total) {
        const uint32_t row = i / per_row;
        cc[u] = i - row * per_row;
        const uint32_t t = row / a.hkv;
        hh[u] = row - t * a.hkv;
        slot[u] = __ldg(a.cache_loc + t);
        val[u] = __ldg(cc[u] < a.ck
                           ? a.k + (int64_t)t * a.k_ts + (int64_t)hh[u] * a.k_hs + cc[u]
                           : a.v + (int64_t)t * a.v_ts + (int64_t)hh[u] * a.v_hs + (cc[u] - a.ck));
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (slot[u] < 0 || slot[u] >= a.num_slots) continue;  // outside the pool: skipped
      if (cc[u] < a.ck)
        a.k_buf[slot[u] * a.kb_ss + (int64_t)hh[u] * a.kb_hs + cc[u]] =
            bf16x8_to_fp8x8<FMT>(val[u], a.k_scale);
      else
        a.v_buf[slot[u] * a.vb_ss + (int64_t)hh[u] * a.vb_hs + (cc[u] - a.ck)] =
            bf16x8_to_fp8x8<FMT>(val[u], a.v_scale);
    }
  }
}

int launch_set_kv_buffer_fp8(const void *k, int64_t k_ts, int64_t k_hs, const void *v,
                             int64_t v_ts, int64_t v_hs, const int64_t *cache_loc,
                             int64_t n_tokens, int hkv, int lk, int lv, float k_scale,
                             float v_scale, int fmt, void *k_buffer, int64_t kb_ss,
                             int64_t kb_hs, void *v_buffer, int64_t vb_ss, int64_t vb_hs,
                             int64_t num_slots, cudaStream_t st) {
  KvWriteFp8Args a;
  a.k = static_cast<const uint4 *>(k);
  a.v = static_cast<const uint4 *>(v);
  a.k_ts = k_ts / 8; a.k_hs = k_hs / 8; a.v_ts = v_ts / 8; a.v_hs = v_hs / 8;
  a.cache_loc = cache_loc;
  a.k_buf = static_cast<uint2 *>(k_buffer);
  a.v_buf = static_cast<uint2 *>(v_buffer);
  a.kb_ss = kb_ss / 8; a.kb_hs = kb_hs / 8; a.vb_ss = vb_ss / 8; a.vb_hs = vb_hs / 8;
  a.num_slots = num_slots;
  a.hkv = (uint32_t)hkv;
  a.ck = (uint32_t)(lk / 8);
  a.cv = v ? (uint32_t)(lv / 8) : 0u;
  a.total = (uint64_t)n_tokens * a.hkv * (a.ck + a.cv);
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  if (a.total == 0) return PKX_OK;
  if (a.total >= (1ull << 31))
    return set_error(PKX_EUNSUPPORTED, "set_kv_buffer_fp8: 2^31 or more chunks in one call");
  const int nsm = num_sms_current_device();
  const uint64_t need = (a.total + kKvThreads * kUnroll - 1) / (kKvThreads * kUnroll);
  const uint64_t cap = (uint64_t)nsm * 4;
  const unsigned grid = (unsigned)(need < cap ? need : cap);
  if (fmt == kKvFp8E4M3) set_kv_buffer_fp8_kernel<1><<<grid, kKvThreads, 0, st>>>(a);
  else set_kv_buffer_fp8_kernel<2><<<grid, kKvThreads, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_error(PKX_ECUDA, "set_kv_buffer_fp8 launch: %s", cudaGetErrorString(e));
  return PKX_OK;
}

// ------------------------------------------------------------ index gather
constexpr int kGatherThreads = 512;
constexpr int kGatherPerThread = 8;  // entries a thread moves per CTA pass

__global__ void __launch_bounds__(kGatherThreads) create_kv_indices_kernel(
    const int32_t *__restrict__ req_to_token, int64_t rows, int64_t stride,
    const int64_t *__restrict__ req_pool_indices, const int64_t *__restrict__ paged_kernel_lens,
    const int64_t *__restrict__ kv_start_idx, int batch, int32_t *kv_indptr, int32_t *kv_indices,
    int64_t capacity) {
  extern __shared__ int32_t s_ptr[];  // [batch + 1] running sum
  __shared__ int32_t s_warp[kGatherThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Exclusive running sum of the 32-bit lengths, each thread over one
  // contiguous run of the batch.
  const int per = (batch + kGatherThreads - 1) / kGatherThreads;
  const int b0 = tid * per < batch ? tid * per : batch;
  const int b1 = b0 + per < batch ? b0 + per : batch;
  int32_t run = 0;
  for (int b = b0; b < b1; ++b) run += (int32_t)paged_kernel_lens[b];
  int32_t incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = lane < kGatherThreads / 32 ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kGatherThreads / 32) s_warp[lane] = w;
  }
  __syncthreads();
  int32_t acc = incl - run + (warp > 0 ? s_warp[warp - 1] : 0);
  for (int b = b0; b < b1; ++b) {
    s_ptr[b] = acc;
    acc += (int32_t)paged_kernel_lens[b];
  }
  if (tid == kGatherThreads - 1) s_ptr[batch] = s_warp[kGatherThreads / 32 - 1];
  __syncthreads();
  if (blockIdx.x == 0)
    for (int b = tid; b <= batch; b += kGatherThreads) kv_indptr[b] = s_ptr[b];

  // This CTA's share of the index range, never past the caller's buffer.
  int64_t total = s_ptr[batch];
  if (total > capacity) total = capacity;
  if (total < 0) total = 0;
  const int64_t share = (total + gridDim.x - 1) / gridDim.x;
  const int64_t f0 = (int64_t)blockIdx.x * share;
  const int64_t f1 = f0 + share < total ? f0 + share : total;
  for (int64_t base = f0 + tid; base < f1; base += (int64_t)kGatherThreads * kGatherPerThread) {
    int32_t val[kGatherPerThread];
#pragma unroll
    for (int u = 0; u < kGatherPerThread; ++u) {
      const int64_t f = base + (int64_t)u * kGatherThreads;
      val[u] = -1;
      if (f < f1) {
        int lo = 0, hi = batch - 1;  // last b with s_ptr[b] <= f
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (s_ptr[mid] <= f) lo = mid; else hi = mid - 1;
        }
        const int64_t r = req_pool_indices[lo];
        const int64_t col = (kv_start_idx ? (int64_t)(int32_t)kv_start_idx[lo] : 0) +
                            (f - s_ptr[lo]);
        if (r >= 0 && r < rows && col >= 0 && col < stride)
          val[u] = __ldg(req_to_token + r * stride + col);
      }
    }
#pragma unroll
    for (int u = 0; u < kGatherPerThread; ++u) {
      const int64_t f = base + (int64_t)u * kGatherThreads;
      if (f < f1) kv_indices[f] = val[u];
    }
  }
}

// ------------------------------------------------------------ page tables
// Paged KV indices (indptr over pages, page ids, entries in each sequence's
// last page, page size) to per-token pool slots, the layout every attention
// call here takes: key j of sequence b is slot
// kv_indices[kv_indptr[b] + j / page_size] * page_size + j % page_size.
// Same shape as the gather above: every CTA scans the key counts, CTA 0
// writes token_indptr, the token range is split evenly over the CTAs.
__global__ void __launch_bounds__(kGatherThreads) expand_paged_kernel(
    const int32_t *__restrict__ kv_indptr, const int32_t *__restrict__ kv_indices,
    const int32_t *__restrict__ last_page_len, int page_size, int batch, int32_t *token_indptr,
    int32_t *token_indices, int64_t capacity) {
  extern __shared__ int32_t s_ptr[];  // [batch + 1] running sum of key counts
  __shared__ int32_t s_warp[kGatherThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto keys_of = [&](int b) -> int32_t {
    const int32_t pages = kv_indptr[b + 1] - kv_indptr[b];
    return pages > 0 ? (pages - 1) * page_size + last_page_len[b] : 0;
  };
  const int per = (batch + kGatherThreads - 1) / kGatherThreads;
  const int b0 = tid * per < batch ? tid * per : batch;
  const int b1 = b0 + per < batch ? b0 + per : batch;
  int32_t run = 0;
  for (int b = b0; b < b1; ++b) run += keys_of(b);
  int32_t incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = lane < kGatherThreads / 32 ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kGatherThreads / 32) s_warp[lane] = w;
  }
  __syncthreads();
  int32_t acc = incl - run + (warp > 0 ? s_warp[warp - 1] : 0);
  for (int b = b0; b < b1; ++b) {
    s_ptr[b] = acc;
    acc += keys_of(b);
  }
  if (tid == kGatherThreads - 1) s_ptr[batch] = s_warp[kGatherThreads / 32 - 1];
  __syncthreads();
  if (blockIdx.x == 0)
    for (int b = tid; b <= batch; b += kGatherThreads) token_indptr[b] = s_ptr[b];

  int64_t total = s_ptr[batch];
  if (total > capacity) total = capacity;
  if (total < 0) total = 0;
  const int64_t share = (total + gridDim.x - 1) / gridDim.x;
  const int64_t f0 = (int64_t)blockIdx.x * share;
  const int64_t f1 = f0 + share < total ? f0 + share : total;
  for (int64_t base = f0 + tid; base < f1; base += (int64_t)kGatherThreads * kGatherPerThread) {
    int32_t val[kGatherPerThread];
#pragma unroll
    for (int u = 0; u < kGatherPerThread; ++u) {
      const int64_t f = base + (int64_t)u * kGatherThreads;
      val[u] = -1;
      if (f < f1) {
        int lo = 0, hi = batch - 1;  // last b with s_ptr[b] <= f
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (s_ptr[mid] <= f) lo = mid; else hi = mid - 1;
        }
        const int64_t j = f - s_ptr[lo];
        const int64_t pg = kv_indptr[lo] + j / page_size;
        if (pg >= kv_indptr[lo] && pg < kv_indptr[lo + 1])  // a page of this sequence
          val[u] = __ldg(kv_indices + pg) * page_size + (int32_t)(j % page_size);
      }
    }
#pragma unroll
    for (int u = 0; u < kGatherPerThread; ++u) {
      const int64_t f = base + (int64_t)u * kGatherThreads;
      if (f < f1) token_indices[f] = val[u];
    }
  }
}

int launch_expand_paged(const int32_t *kv_indptr, const int32_t *kv_indices,
                        const int32_t *last_page_len, int page_size, int batch,
                        int32_t *token_indptr, int32_t *token_indices, int64_t capacity,
                        cudaStream_t st) {
  if (batch == 0) {
    cudaError_t e = cudaMemsetAsync(token_indptr, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) return set_error(PKX_ECUDA, "memset: %s", cudaGetErrorString(e));
    return PKX_OK;
  }
  const int nsm = num_sms_current_device();
  const int64_t per_cta = batch * 2 > 1024 ? (int64_t)batch * 2 : 1024;
  int64_t grid = (capacity + per_cta - 1) / per_cta;
  if (grid < 1) grid = 1;
  if (grid > (int64_t)nsm * 4) grid = (int64_t)nsm * 4;
  const size_t smem = sizeof(int32_t) * (size_t)(batch + 1);
  expand_paged_kernel<<<(unsigned)grid, kGatherThreads, smem, st>>>(
      kv_indptr, kv_indices, last_page_len, page_size, batch, token_indptr, token_indices,
      capacity);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_error(PKX_ECUDA, "expand_paged_kv_indices launch: %s", cudaGetErrorString(e));
  return PKX_OK;
}

int launch_create_kv_indices(const int32_t *req_to_token, int64_t rows, int64_t stride,
                             const int64_t *req_pool_indices, const int64_t *paged_kernel_lens,
                             const int64_t *kv_start_idx, int batch, int32_t *kv_indptr,
                             int32_t *kv_indices, int64_t capacity, cudaStream_t st) {
  if (batch == 0) {
    cudaError_t e = cudaMemsetAsync(kv_indptr, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) return set_error(PKX_ECUDA, "memset: %s", cudaGetErrorString(e));
    return PKX_OK;
  }
  // Every CTA scans the whole batch, so a CTA takes at least twice the batch
  // in entries (and at least 1K); at most four CTAs per SM.
  const int nsm = num_sms_current_device();
  const int64_t per_cta = batch * 2 > 1024 ? (int64_t)batch * 2 : 1024;
  int64_t grid = (capacity + per_cta - 1) / per_cta;
  if (grid < 1) grid = 1;
  if (grid > (int64_t)nsm * 4) grid = (int64_t)nsm * 4;
  const size_t smem = sizeof(int32_t) * (size_t)(batch + 1);
  create_kv_indices_kernel<<<(unsigned)grid, kGatherThreads, smem, st>>>(
      req_to_token, rows, stride, req_pool_indices, paged_kernel_lens, kv_start_idx, batch,
      kv_indptr, kv_indices, capacity);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_error(PKX_ECUDA, "create_kv_indices launch: %s", cudaGetErrorString(e));
  return PKX_OK;
}

}  // namespace pkx
