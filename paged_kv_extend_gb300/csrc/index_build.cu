// index_build.cu -- unified KV-index construction (sglang extend_attention.py,
// build_unified_kv_indices and _copy_unified_indices_kernel):
//   prefix_lens[b] = prefix_kv_indptr[b+1] - prefix_kv_indptr[b]
//   unified_kv_indptr = [0, running sum of prefix_lens + extend_seq_lens]
//   unified row b = prefix slice of b, then extend slice of b (int32 -> int64)
//
// One kernel, one CTA per sequence: the CTA finds its output offset itself
// (the prefix part of the running sum is prefix_kv_indptr[b] -
// prefix_kv_indptr[0]; the extend part is a block reduction over
// extend_seq_lens[0..b)), writes its indptr entry and prefix length, then
// copies its two slices with coalesced 4-byte loads and 8-byte stores, eight
// loads in flight per thread.  No separate scan launch and no host sync.
#include <cuda_runtime.h>

#include "pkx_internal.h"
#include "ptx.cuh"

namespace pkx {

// dst[j] = src[j] for j < n by the block's 256 threads, eight independent
// loads in flight per thread before their stores (a long prefix is
// thousands of entries; one load-then-store per step would serialise on
// the memory latency).
__device__ __forceinline__ void copy_widen(const int32_t *__restrict__ src, int64_t *dst, int n,
                                           int tid) {
  constexpr int U = 8;
  for (int base = tid; base < n; base += 256 * U) {
    int32_t v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = base + u * 256;
      v[u] = j < n ? __ldg(src + j) : 0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = base + u * 256;
      if (j < n) dst[j] = v[u];
    }
  }
}

__global__ void __launch_bounds__(256) build_unified_kernel(
    const int32_t *__restrict__ prefix_kv_indptr, const int32_t *__restrict__ prefix_kv_indices,
    const int32_t *__restrict__ extend_start_loc, const int32_t *__restrict__ extend_seq_lens,
    const int32_t *__restrict__ extend_kv_indices, int batch, int32_t *unified_kv_indptr,
    int64_t *unified_kv_indices, int32_t *prefix_lens) {
  __shared__ long long red[256];
  grid_dep_launch();  // the scheduler may start (it waits for this grid's writes)
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  long long ext_before = 0;
  for (int c = tid; c < b; c += 256) ext_before += extend_seq_lens[c];
  red[tid] = ext_before;
  __syncthreads();
  for (int off = 128; off > 0; off >>= 1) {
    if (tid < off) red[tid] += red[tid + off];
    __syncthreads();
  }
  const int p0 = prefix_kv_indptr[b], p1 = prefix_kv_indptr[b + 1];
  const int plen = p1 - p0;
  const int elen = extend_seq_lens[b];
  const long long start = (long long)(p0 - prefix_kv_indptr[0]) + red[0];
  if (tid == 0) {
    prefix_lens[b] = plen;
    unified_kv_indptr[b + 1] = (int32_t)(start + plen + elen);
    if (b == 0) unified_kv_indptr[0] = 0;
  }
  int64_t *dst = unified_kv_indices + start;
  copy_widen(prefix_kv_indices + p0, dst, plen, tid);
  copy_widen(extend_kv_indices + extend_start_loc[b], dst + plen, elen, tid);
}

int launch_build_unified(const int32_t *prefix_kv_indptr, const int32_t *prefix_kv_indices,
                         const int32_t *extend_start_loc, const int32_t *extend_seq_lens,
                         const int32_t *extend_kv_indices, int batch, int32_t *unified_kv_indptr,
                         int64_t *unified_kv_indices, int32_t *prefix_lens, cudaStream_t st) {
  if (batch == 0) {
    // indptr[0] = 0 still has to be written
    cudaError_t e = cudaMemsetAsync(unified_kv_indptr, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) return set_error(PKX_ECUDA, "memset: %s", cudaGetErrorString(e));
    return PKX_OK;
  }
  build_unified_kernel<<<batch, 256, 0, st>>>(prefix_kv_indptr, prefix_kv_indices,
                                              extend_start_loc, extend_seq_lens,
                                              extend_kv_indices, batch, unified_kv_indptr,
                                              unified_kv_indices, prefix_lens);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_error(PKX_ECUDA, "build_unified_kv_indices launch: %s", cudaGetErrorString(e));
  return PKX_OK;
}

}  // namespace pkx
