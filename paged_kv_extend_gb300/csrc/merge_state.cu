// merge_state.cu -- merge two partial attention states by their log-sum-exp
// (sglang flashinfer_backend.py, forward_extend: the ragged causal extend
// result and the non-causal paged prefix result are combined with
// merge_state).  For each row: s = log(exp(s_a) + exp(s_b)),
// v = exp(s_a - s) v_a + exp(s_b - s) v_b; an s = -inf side has weight 0.
//
// HBM-bound elementwise work: one thread per 16-byte chunk (8 bf16) of a
// row, 16-byte loads and stores, the row's two lse values read once per
// chunk (they stay in L1).  Grid sized to a multiple of the SM count.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pkx_internal.h"
#include "ptx.cuh"

namespace pkx {

// PLAIN: v_out aliases v_a or v_b, so the inputs are not read-only for the
// kernel's lifetime and take ordinary loads (each chunk is still read before
// the same thread writes it).  WRITE_S: s_out is written here; when it
// aliases s_a or s_b it is written by merge_lse_kernel afterwards instead,
// since the threads of one row (several warps for a wide row) all read the
// row's s_a and s_b.
template <bool PLAIN, bool WRITE_S>
__global__ void __launch_bounds__(256) merge_state_kernel(
    const uint4 *v_a, const float *s_a, const uint4 *v_b, const float *s_b, uint4 *v_out,
    float *s_out, int64_t rows, int chunks_per_row) {
  const int64_t total = rows * chunks_per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / chunks_per_row;
    const int c = (int)(i - r * chunks_per_row);
    const float sa = __ldg(s_a + r), sb = __ldg(s_b + r);
    uint4 a, b;
    if constexpr (PLAIN) {
      a = v_a[i];
      b = v_b[i];
    } else {
      a = __ldg(v_a + i);
      b = __ldg(v_b + i);
    }
    float wa, wb, s;
    if (sa == -INFINITY && sb == -INFINITY) {
      wa = wb = 0.f;
      s = -INFINITY;
    } else {
      const float m = fmaxf(sa, sb);
      const float ea = __expf(sa - m), eb = __expf(sb - m);
      const float sum = ea + eb;
      wa = ea / sum;
      wb = eb / sum;
      s = m + __logf(sum);
    }
    const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&a);
    const __nv_bfloat162 *pb = reinterpret_cast<const __nv_bfloat162 *>(&b);
    uint4 out;
    uint32_t *po = reinterpret_cast<uint32_t *>(&out);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 fa = __bfloat1622float2(pa[k]);
      const float2 fb = __bfloat1622float2(pb[k]);
      po[k] = pack_bf16(wa * fa.x + wb * fb.x, wa * fa.y + wb * fb.y);
    }
    v_out[i] = out;
    if (WRITE_S && s_out && c == 0) s_out[r] = s;
  }
}

// The merged log-sum-exp, one thread per row (each row's inputs read and its
// output written by the same thread, so s_out may alias s_a or s_b).
__global__ void __launch_bounds__(256) merge_lse_kernel(const float *s_a, const float *s_b,
                                                         float *s_out, int64_t rows) {
  for (int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; r < rows;
       r += (int64_t)gridDim.x * blockDim.x) {
    const float sa = s_a[r], sb = s_b[r];
    float s = -INFINITY;
    if (!(sa == -INFINITY && sb == -INFINITY)) {
      const float m = fmaxf(sa, sb);
      s = m + __logf(__expf(sa - m) + __expf(sb - m));
    }
    s_out[r] = s;
  }
}

int launch_merge_state(const void *v_a, const float *s_a, const void *v_b, const float *s_b,
                       void *v_out, float *s_out, int64_t n, int h, int dv, cudaStream_t st) {
  const int64_t rows = n * h;
  if (rows == 0) return PKX_OK;
  const int cpr = dv / 8;
  const int nsm = num_sms_current_device();
  const int64_t need = (rows * cpr + 255) / 256;
  const unsigned grid = (unsigned)(need < (int64_t)nsm * 8 ? need : (int64_t)nsm * 8);
  const bool v_alias = v_out == v_a || v_out == v_b;
  const bool s_alias = s_out != nullptr && (s_out == s_a || s_out == s_b);
  auto *va = static_cast<const uint4 *>(v_a);
  auto *vb = static_cast<const uint4 *>(v_b);
  auto *vo = static_cast<uint4 *>(v_out);
  if (s_alias) {
    if (v_alias) merge_state_kernel<true, false><<<grid, 256, 0, st>>>(va, s_a, vb, s_b, vo, s_out, rows, cpr);
    else merge_state_kernel<false, false><<<grid, 256, 0, st>>>(va, s_a, vb, s_b, vo, s_out, rows, cpr);
    const int64_t need_s = (rows + 255) / 256;
    const unsigned grid_s = (unsigned)(need_s < (int64_t)nsm * 8 ? need_s : (int64_t)nsm * 8);
    merge_lse_kernel<<<grid_s, 256, 0, st>>>(s_a, s_b, s_out, rows);
  } else if (v_alias) {
    merge_state_kernel<true, true><<<grid, 256, 0, st>>>(va, s_a, vb, s_b, vo, s_out, rows, cpr);
  } else {
    merge_state_kernel<false, true><<<grid, 256, 0, st>>>(va, s_a, vb, s_b, vo, s_out, rows, cpr);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(PKX_ECUDA, "merge_state launch: %s", cudaGetErrorString(e));
  return PKX_OK;
}

}  // namespace pkx
