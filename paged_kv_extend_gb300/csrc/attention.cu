// attention.cu -- extend and decode attention over a page-size-1 KV pool for
// sm_103a: a device-side work scheduler, a warp-specialised tcgen05/TMEM
// attention kernel with a cp.async paged gather, and the split-KV combine.
//
// Method (sglang extend_attention.py, _fwd_kernel_unified and
// extend_attention_fwd; flashinfer_backend.py, forward_decode):
//   for each query row and each visible key j:  s_j = sm_scale * <q, k_j>,
//   optionally s_j = cap * tanh(s_j / cap); visible iff j <= qpos and, with a
//   window W > 0, qpos - j <= W; o = sum_j softmax(s)_j v_j; lse = log sum
//   exp s.  The online softmax keeps a running max and sum per row and
//   rescales the accumulator when the max moves.
//
// GB300 design (differs from the pages' Triton kernel, which launches one
// program per (sequence, q head, 128-row block) and re-reads K/V per q head):
//  * one tile = 128 rows = (tokens x the Hq/Hkv query heads of one KV head),
//    so K/V of a KV head are gathered once for all of its query heads;
//  * QK^T and PV are tcgen05.mma (M=128, bf16 in, fp32 accumulate in TMEM);
//    S is double-buffered in TMEM so the tensor core computes S_{j+1} while
//    the softmax warps work on S_j;
//  * the KV loop stops at the causal diagonal and starts at the window edge
//    (the Triton kernel walks every tile and masks);
//  * a device-built work list (no host sync, graph-safe) splits long key
//    ranges across CTAs (split-KV) and a combine kernel merges the partial
//    (o, lse) pairs with the merge_state formula;
//  * a persistent grid of one CTA per SM walks the work list.
#include <cstdio>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pkx_internal.h"
#include "ptx.cuh"

namespace pkx {

using bf16 = __nv_bfloat16;

// ============================================================ scheduler ====
struct SchedParams {
  int mode;
  const int32_t *qo_indptr, *kv_indptr, *prefix_lens;
  int batch, hkv, tok, window, num_q_tokens;
  int unit_target, qb_max, unit_max, comb_max, slot_max;
  int32_t *seq;  // 8 arrays of batch+1 ints
  int32_t *qbt;  // tiles per query block
  WorkUnit *units;
  CombineEntry *comb;
  WsHeader *hdr;
};

struct SeqDims {
  int P, E, T, qbase, nqb;
};

__device__ __forceinline__ void record_status(int32_t *status, int code) {
  atomicCAS(status, 0, code);
}

// Prefix length, extend length, key count and first query row of sequence b.
// Inconsistent values are recorded and the sequence is treated as empty.
__device__ SeqDims seq_dims(const SchedParams &p, int b) {
  SeqDims d;
  if (p.mode == kDecode) {
    d.T = p.kv_indptr[b + 1] - p.kv_indptr[b];
    d.E = 1;
    d.P = d.T - 1;
    d.qbase = b;
    if (d.T < 0 || p.kv_indptr[b] < 0) {
      record_status(&p.hdr->status, PKX_EDEVICE);
      d.T = 0;
      d.P = -1;
    }
    d.nqb = 1;
    return d;
  }
  d.qbase = p.qo_indptr[b];
  d.E = p.qo_indptr[b + 1] - d.qbase;
  if (p.mode == kTwoStage) {
    d.P = p.kv_indptr[b + 1] - p.kv_indptr[b];
    d.T = d.P + d.E;
  } else {
    d.T = p.kv_indptr[b + 1] - p.kv_indptr[b];
    d.P = p.prefix_lens[b];
    if (d.P + d.E != d.T) record_status(&p.hdr->status, PKX_EDEVICE);
  }
  bool bad = d.E < 0 || d.P < 0 || d.T < 0 || d.qbase < 0 || p.kv_indptr[b] < 0 ||
             (long long)d.qbase + d.E > p.num_q_tokens;
  if (bad) {
    record_status(&p.hdr->status, PKX_EDEVICE);
    d.E = 0;
  }
  d.nqb = d.E > 0 ? (d.E + p.tok - 1) / p.tok : 0;
  return d;
}

// Key range [lo, hi) of query block qb of a sequence.
__device__ __forceinline__ void qblock_range(const SchedParams &p, const SeqDims &d, int qb,
                                             int &lo, int &hi, int &i0, int &i1) {
  i0 = qb * p.tok;
  i1 = min(d.E, i0 + p.tok);
  const int qmin = d.P + i0, qmax = d.P + i1 - 1;
  hi = min(qmax + 1, d.T);
  lo = p.window > 0 ? max(0, qmin - p.window) : 0;
  if (hi < lo) hi = lo;
}

// Exclusive scan of in[0..n) into out[0..n) by the whole 1024-thread block;
// returns the total.  in and out may alias.
__device__ int block_exclusive_scan(const int32_t *in, int32_t *out, int n, int *sh) {
  const int tid = threadIdx.x;
  const int ch = (n + 1023) / 1024;
  const int beg = min(n, tid * ch), end = min(n, beg + ch);
  int local = 0;
  for (int i = beg; i < end; ++i) local += in[i];
  __syncthreads();
  sh[tid] = local;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    int v = tid >= off ? sh[tid - off] : 0;
    __syncthreads();
    sh[tid] += v;
    __syncthreads();
  }
  int run = sh[tid] - local;
  const int total = sh[1023];
  for (int i = beg; i < end; ++i) {
    int v = in[i];
    out[i] = run;
    run += v;
  }
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(1024, 1) sched_kernel(SchedParams p) {
  __shared__ int sh[1024];
  __shared__ int s_c;
  const int tid = threadIdx.x;
  const int B = p.batch;
  int32_t *nqb = p.seq;                 // [B]  query blocks per sequence
  int32_t *qboff = p.seq + 1 * (B + 1); // [B]  first query block of sequence
  int32_t *work = p.seq + 2 * (B + 1);  // [B]  KV tiles of the sequence
  int32_t *order = p.seq + 3 * (B + 1); // [B]  rank -> sequence
  int32_t *ucnt = p.seq + 4 * (B + 1);  // [B]  by rank: units, then offsets
  int32_t *scnt = p.seq + 5 * (B + 1);  // [B]  by rank: partial slots
  int32_t *ccnt = p.seq + 6 * (B + 1);  // [B]  by rank: combine entries

  if (tid == 0) p.hdr->status = 0;
  __syncthreads();

  // 1. query blocks per sequence and their offsets
  for (int b = tid; b < B; b += 1024) nqb[b] = seq_dims(p, b).nqb;
  __syncthreads();
  const int total_qb = block_exclusive_scan(nqb, qboff, B, sh);
  if (total_qb > p.qb_max) {  // cannot happen for consistent indptrs
    if (tid == 0) {
      record_status(&p.hdr->status, PKX_EDEVICE);
      p.hdr->n_units = 0;
      p.hdr->n_combine = 0;
    }
    return;
  }

  // 2. KV tiles per query block and per sequence; total tiles
  long long my_tiles = 0;
  for (int b = tid; b < B; b += 1024) {
    SeqDims d = seq_dims(p, b);
    int w = 0;
    for (int qb = 0; qb < d.nqb; ++qb) {
      int lo, hi, i0, i1;
      qblock_range(p, d, qb, lo, hi, i0, i1);
      int nt = (hi - lo + kBlockN - 1) / kBlockN;
      p.qbt[qboff[b] + qb] = nt;
      w += nt;
    }
    work[b] = w;
    my_tiles += w;
  }
  __syncthreads();
  // block reduce of the tile count (as 64-bit via two 32-bit halves is
  // unnecessary: tiles of any sane problem fit in 31 bits)
  sh[tid] = (int)min(my_tiles, (long long)0x3fffffff);
  __syncthreads();
  for (int off = 512; off > 0; off >>= 1) {
    if (tid < off) sh[tid] = min(sh[tid] + sh[tid + off], 0x3fffffff);
    __syncthreads();
  }
  const long long total_tiles = (long long)sh[0] * p.hkv;
  __syncthreads();
  if (tid == 0) {
    long long c = (total_tiles + p.unit_target - 1) / p.unit_target;
    s_c = (int)max((long long)kMinSplitTiles, c);
    p.hdr->split_tiles = s_c;
  }
  __syncthreads();
  const int C = s_c;

  // 3. order sequences by work, largest first (ties by index); identity for
  //    very large batches
  if (B <= 8192) {
    for (int b = tid; b < B; b += 1024) {
      const int wb = work[b];
      int rank = 0;
      for (int c = 0; c < B; ++c) {
        const int wc = work[c];
        rank += (wc > wb) || (wc == wb && c < b);
      }
      order[rank] = b;
    }
  } else {
    for (int b = tid; b < B; b += 1024) order[b] = b;
  }
  __syncthreads();

  // 4. units, partial slots and combine entries per sequence (by rank)
  for (int rk = tid; rk < B; rk += 1024) {
    const int b = order[rk];
    const int n = nqb[b];
    int u = 0, s = 0, c = 0;
    for (int qb = 0; qb < n; ++qb) {
      const int nt = p.qbt[qboff[b] + qb];
      const int S = nt > 0 ? (nt + C - 1) / C : 1;
      u += S;
      if (S > 1) {
        s += S;
        c += 1;
      }
    }
    ucnt[rk] = u * p.hkv;
    scnt[rk] = s * p.hkv;
    ccnt[rk] = c * p.hkv;
  }
  __syncthreads();
  const int n_units = block_exclusive_scan(ucnt, ucnt, B, sh);
  const int n_slots = block_exclusive_scan(scnt, scnt, B, sh);
  const int n_comb = block_exclusive_scan(ccnt, ccnt, B, sh);
  if (n_units > p.unit_max || n_slots > p.slot_max || n_comb > p.comb_max) {
    if (tid == 0) {
      record_status(&p.hdr->status, PKX_EDEVICE);
      p.hdr->n_units = 0;
      p.hdr->n_combine = 0;
    }
    return;
  }

  // 5. emit: for each sequence (largest first), each KV head, each query
  //    block from the last (longest key range) to the first, each split.
  for (int rk = tid; rk < B; rk += 1024) {
    const int b = order[rk];
    SeqDims d = seq_dims(p, b);
    int uo = ucnt[rk], so = scnt[rk], co = ccnt[rk];
    for (int kvh = 0; kvh < p.hkv; ++kvh) {
      for (int qb = d.nqb - 1; qb >= 0; --qb) {
        int lo, hi, i0, i1;
        qblock_range(p, d, qb, lo, hi, i0, i1);
        const int nt = p.qbt[qboff[b] + qb];
        const int S = nt > 0 ? (nt + C - 1) / C : 1;
        const int tps = nt > 0 ? (nt + S - 1) / S : 0;
        if (S > 1) {
          CombineEntry e;
          e.q_tok0 = d.qbase + i0;
          e.n_tok = i1 - i0;
          e.kvh = kvh;
          e.slot0 = so;
          e.n_split = S;
          e.pad[0] = e.pad[1] = e.pad[2] = 0;
          p.comb[co++] = e;
        }
        for (int s = 0; s < S; ++s) {
          WorkUnit w;
          w.q_tok0 = d.qbase + i0;
          w.n_tok = i1 - i0;
          w.qpos0 = d.P + i0;
          w.kvh = kvh;
          w.k_begin = min(hi, lo + s * tps * kBlockN);
          w.k_end = min(hi, lo + (s + 1) * tps * kBlockN);
          w.b = b;
          w.slot = S > 1 ? so + s : -1;
          p.units[uo++] = w;
        }
        if (S > 1) so += S;
      }
    }
  }
  if (tid == 0) {
    p.hdr->n_units = n_units;
    p.hdr->n_combine = n_comb;
  }
}

// ============================================================ attention ====
struct KParams {
  const bf16 *q;
  bf16 *o;
  float *lse;
  const bf16 *k_ext, *v_ext;
  int64_t ke_st, ke_sh, ve_st, ve_sh;
  const bf16 *k_buf, *v_buf;
  int64_t kb_ss, kb_sh, vb_ss, vb_sh;
  int64_t num_slots;
  const int32_t *qo_indptr, *kv_indptr;
  const void *kv_indices;
  int hq, group, window, use_cap;
  float scale_log2;  // sm_scale * log2(e)           (no cap)
  float cap_pre;     // sm_scale / cap                (cap)
  float cap_log2;    // cap * log2(e)                 (cap)
  const WorkUnit *units;
  const WsHeader *hdr;
  int32_t *status;
  float *plse, *po;
};

template <int HD>
struct Cfg {
  static constexpr int BM = kBlockM, BN = kBlockN, HDV = HD;
  static constexpr int NS = HD == 128 ? 2 : 4;  // K/V pipeline stages
  static constexpr int Q_BYTES = BM * HD * 2;
  static constexpr int K_BYTES = BN * HD * 2;
  static constexpr int V_BYTES = BN * HDV * 2;
  static constexpr int P_BYTES = BM * BN * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + NS * K_BYTES;
  static constexpr int OFF_P = OFF_V + NS * V_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int N_BARS = 8 + 2 * NS;
  static constexpr int SMEM = OFF_BAR + N_BARS * 8 + 1024;  // + alignment slack
  static constexpr int S_COL = 0;       // two S buffers: columns 0 and 128
  static constexpr int O_COL = 2 * BN;  // O accumulator
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, 0);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, HDV, 1);
  static constexpr int THREADS = 256;  // 4 softmax warps, 1 MMA warp, 3 load warps
  static constexpr int LOAD_THREADS = 96;
};

// barrier indices
enum {
  B_Q_FULL = 0,
  B_Q_EMPTY = 1,
  B_S_FULL0 = 2,
  B_S_FULL1 = 3,
  B_P_FULL = 4,
  B_O_DONE = 5,
  B_FINAL = 6,
  B_KV_FULL = 8,  // + stage
};

__device__ __forceinline__ int unit_tiles(const WorkUnit &w) {
  return w.k_end > w.k_begin ? (w.k_end - w.k_begin + kBlockN - 1) / kBlockN : 0;
}

__device__ __forceinline__ void abort_cta(volatile int *abort_flag, int32_t *status, int code) {
  *abort_flag = 1;
  record_status(status, code);
}

template <int HD, int MODE>
__global__ void __launch_bounds__(Cfg<HD>::THREADS, 1) attn_kernel(const KParams p) {
  using C = Cfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *bar_kv_full = bars + B_KV_FULL;
  uint64_t *bar_kv_empty = bars + B_KV_FULL + C::NS;
  volatile int *abort_flag = &s_abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(&bars[B_Q_FULL], C::LOAD_THREADS);
    mbar_init(&bars[B_Q_EMPTY], 1);
    mbar_init(&bars[B_S_FULL0], 1);
    mbar_init(&bars[B_S_FULL1], 1);
    mbar_init(&bars[B_P_FULL], 128);
    mbar_init(&bars[B_O_DONE], 1);
    mbar_init(&bars[B_FINAL], 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&bar_kv_full[s], C::LOAD_THREADS);
      mbar_init(&bar_kv_empty[s], 1);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 4) {
    tmem_alloc(&s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int n_units = p.hdr->n_units;

  if (warp < 4) {
    // ------------------------------------------------ softmax + epilogue
    const int r = tid;  // TMEM lane == tile row
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    uint32_t s_cnt = 0, o_cnt = 0;
    for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x) {
      const WorkUnit w = p.units[u];
      const int nt = unit_tiles(w);
      const int rows_valid = w.n_tok * p.group;
      const bool valid = r < rows_valid;
      const bool warp_active = warp * 32 < rows_valid;
      const int t = r / p.group, g = r - (r / p.group) * p.group;
      const int qpos = w.qpos0 + t;
      const int qpos_max = w.qpos0 + w.n_tok - 1;
      if (nt == 0) {
        if (valid) {
          if (w.slot < 0) {
            bf16 *orow = p.o + ((int64_t)(w.q_tok0 + t) * p.hq + w.kvh * p.group + g) * C::HDV;
            for (int c = 0; c < C::HDV; c += 8)
              *reinterpret_cast<uint4 *>(orow + c) = make_uint4(0, 0, 0, 0);
            if (p.lse) p.lse[(int64_t)(w.q_tok0 + t) * p.hq + w.kvh * p.group + g] = -INFINITY;
          } else {
            float *prow = p.po + ((int64_t)w.slot * C::BM + r) * C::HDV;
            for (int c = 0; c < C::HDV; c += 4)
              *reinterpret_cast<float4 *>(prow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            p.plse[(int64_t)w.slot * C::BM + r] = -INFINITY;
          }
        }
        continue;
      }
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j) {
        const int kb = w.k_begin + j * C::BN;
        const uint32_t sb = s_cnt & 1u;
        if (!mbar_wait(&bars[B_S_FULL0 + sb], (s_cnt >> 1) & 1u, abort_flag)) {
          abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
          break;
        }
        ++s_cnt;
        tc_fence_after();
        float x[C::BN];
        float mt = -INFINITY;
        if (warp_active) {
          uint32_t v[32];
#pragma unroll
          for (int c = 0; c < C::BN / 32; ++c) {
            tmem_ld32(lane_base + C::S_COL + sb * C::BN + c * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(v[i]);
          }
          if (p.use_cap) {
#pragma unroll
            for (int i = 0; i < C::BN; ++i) x[i] = p.cap_log2 * tanh_approx(x[i] * p.cap_pre);
          } else {
#pragma unroll
            for (int i = 0; i < C::BN; ++i) x[i] *= p.scale_log2;
          }
          const bool need_mask = (kb + C::BN - 1 > w.qpos0) || (kb + C::BN > w.k_end) ||
                                 (p.window > 0 && kb < qpos_max - p.window);
          if (need_mask) {
#pragma unroll
            for (int i = 0; i < C::BN; ++i) {
              const int kpos = kb + i;
              const bool vis = kpos < w.k_end && kpos <= qpos &&
                               (p.window <= 0 || qpos - kpos <= p.window);
              if (!vis) x[i] = -INFINITY;
            }
          }
#pragma unroll
          for (int i = 0; i < C::BN; ++i) mt = fmaxf(mt, x[i]);
        }
        if (j > 0) {
          if (!mbar_wait(&bars[B_O_DONE], o_cnt & 1u, abort_flag)) {
            abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
            break;
          }
          ++o_cnt;
          tc_fence_after();
        }
        if (warp_active) {
          const float m_new = fmaxf(m, mt);
          // Rescale only when the max grows by more than 2^8: exponents of
          // the stale max stay below 256, which fp32 sums and bf16 P hold.
          const bool grow = m_new > m + 8.0f;
          const float alpha = grow ? ex2_approx(m - m_new) : 1.0f;
          const bool o_needs = grow && j > 0 && l > 0.f;
          if (grow) {
            l *= alpha;
            m = m_new;
          }
          const float mref = m == -INFINITY ? 0.f : m;
          uint8_t *prow_base = smem + C::OFF_P;
#pragma unroll
          for (int c = 0; c < C::BN / 8; ++c) {
            float e[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              e[i] = ex2_approx(x[c * 8 + i] - mref);
              l += e[i];
            }
            uint4 pk;
            pk.x = pack_bf16(e[0], e[1]);
            pk.y = pack_bf16(e[2], e[3]);
            pk.z = pack_bf16(e[4], e[5]);
            pk.w = pack_bf16(e[6], e[7]);
            const uint32_t off = (c >> 3) * (C::BM * 128) + sw128_off(r, c & 7);
            *reinterpret_cast<uint4 *>(prow_base + off) = pk;
          }
          // O *= alpha once P is out of registers (PV_j is issued only after
          // this warp arrives on the P barrier below).
          if (__any_sync(0xffffffffu, o_needs)) {
            const float a = o_needs ? alpha : 1.0f;
            uint32_t v[32];
#pragma unroll
            for (int c = 0; c < C::HDV / 32; ++c) {
              const uint32_t ta = lane_base + C::O_COL + c * 32;
              tmem_ld32(ta, v);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * a);
              tmem_st32(ta, v);
            }
            tmem_wait_st();
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars[B_P_FULL]);
      }
      if (*abort_flag) break;
      // epilogue: wait for the last PV, normalise, store
      if (!mbar_wait(&bars[B_O_DONE], o_cnt & 1u, abort_flag)) {
        abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
        break;
      }
      ++o_cnt;
      tc_fence_after();
      if (warp_active) {
        const float inv = l > 0.f ? 1.0f / l : 0.f;
        const float lse_v = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        const int64_t orow_idx = (int64_t)(w.q_tok0 + t) * p.hq + w.kvh * p.group + g;
        uint32_t v[32];
#pragma unroll
        for (int c = 0; c < C::HDV / 32; ++c) {
          tmem_ld32(lane_base + C::O_COL + c * 32, v);
          tmem_wait_ld();
          if (valid) {
            if (w.slot < 0) {
              bf16 *orow = p.o + orow_idx * C::HDV + c * 32;
#pragma unroll
              for (int i = 0; i < 32; i += 8) {
                uint4 pk;
                pk.x = pack_bf16(__uint_as_float(v[i + 0]) * inv, __uint_as_float(v[i + 1]) * inv);
                pk.y = pack_bf16(__uint_as_float(v[i + 2]) * inv, __uint_as_float(v[i + 3]) * inv);
                pk.z = pack_bf16(__uint_as_float(v[i + 4]) * inv, __uint_as_float(v[i + 5]) * inv);
                pk.w = pack_bf16(__uint_as_float(v[i + 6]) * inv, __uint_as_float(v[i + 7]) * inv);
                *reinterpret_cast<uint4 *>(orow + i) = pk;
              }
            } else {
              float *prow = p.po + ((int64_t)w.slot * C::BM + r) * C::HDV + c * 32;
#pragma unroll
              for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4 *>(prow + i) =
                    make_float4(__uint_as_float(v[i]) * inv, __uint_as_float(v[i + 1]) * inv,
                                __uint_as_float(v[i + 2]) * inv, __uint_as_float(v[i + 3]) * inv);
            }
          }
        }
        if (valid) {
          if (w.slot < 0) {
            if (p.lse) p.lse[orow_idx] = lse_v;
          } else {
            p.plse[(int64_t)w.slot * C::BM + r] = lse_v;
          }
        }
      }
      tc_fence_before();
    }
  } else if (warp == 4) {
    // ------------------------------------------------ MMA issue (one thread)
    if (lane == 0) {
      uint32_t q_cnt = 0, kv_cnt = 0, s_cnt = 0, p_cnt = 0;
      const uint32_t sQ = sbase + C::OFF_Q, sP = sbase + C::OFF_P;
      bool ok = true;
      auto issue_pv = [&](int jj, int stage) -> bool {
        if (!mbar_wait(&bars[B_P_FULL], p_cnt & 1u, abort_flag)) return false;
        ++p_cnt;
        tc_fence_after();
        const uint32_t sV = sbase + C::OFF_V + stage * C::V_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          const uint64_t ad = sw128_desc(sP + (kk >> 2) * (C::BM * 128) + (kk & 3) * 32, 0, 1024);
          const uint64_t bd = sw128_desc(sV + kk * 2048, C::BN * 128, 1024);
          tc_mma_ss(tmem + C::O_COL, ad, bd, C::IDESC_PV, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&bars[B_O_DONE]);
        tc_commit(&bar_kv_empty[stage]);
        return true;
      };
      for (int u = blockIdx.x; u < n_units && ok && !*abort_flag; u += gridDim.x) {
        const WorkUnit w = p.units[u];
        const int nt = unit_tiles(w);
        if (nt == 0) continue;
        if (!mbar_wait(&bars[B_Q_FULL], q_cnt & 1u, abort_flag)) { ok = false; break; }
        ++q_cnt;
        tc_fence_after();
        int prev_stage = -1;
        for (int j = 0; j < nt; ++j) {
          const int stage = kv_cnt % C::NS;
          if (!mbar_wait(&bar_kv_full[stage], (kv_cnt / C::NS) & 1u, abort_flag)) { ok = false; break; }
          ++kv_cnt;
          tc_fence_after();
          const uint32_t sb = s_cnt & 1u;
          ++s_cnt;
          const uint32_t sK = sbase + C::OFF_K + stage * C::K_BYTES;
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint64_t ad = sw128_desc(sQ + (kk >> 2) * (C::BM * 128) + (kk & 3) * 32, 0, 1024);
            const uint64_t bd = sw128_desc(sK + (kk >> 2) * (C::BN * 128) + (kk & 3) * 32, 0, 1024);
            tc_mma_ss(tmem + C::S_COL + sb * C::BN, ad, bd, C::IDESC_QK, kk > 0 ? 1u : 0u);
          }
          tc_commit(&bars[B_S_FULL0 + sb]);
          if (j == nt - 1) tc_commit(&bars[B_Q_EMPTY]);
          if (j > 0 && !issue_pv(j - 1, prev_stage)) { ok = false; break; }
          prev_stage = stage;
        }
        if (!ok) break;
        if (!issue_pv(nt - 1, prev_stage)) { ok = false; break; }
      }
      if (!ok) abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
      // drain: every MMA issued above must finish before TMEM is freed
      tc_commit(&bars[B_FINAL]);
      if (!mbar_wait_drain(&bars[B_FINAL], 0)) record_status(p.status, PKX_ETIMEOUT);
    }
  } else {
    // ------------------------------------------------ paged K/V gather
    const int lt = tid - 160;
    uint32_t q_cnt = 0, kv_cnt = 0;
    constexpr int CPR = HD / 8;                  // 16-byte chunks per row
    constexpr int KPP = C::LOAD_THREADS / CPR;   // rows per pass of the load warps
    const int ch = lt % CPR;
    const int row0 = lt / CPR;
    for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x) {
      const WorkUnit w = p.units[u];
      const int nt = unit_tiles(w);
      if (nt == 0) continue;
      if (q_cnt > 0 && !mbar_wait(&bars[B_Q_EMPTY], (q_cnt - 1) & 1u, abort_flag)) {
        abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
        break;
      }
      // Q tile: row r = token * group + head-in-group; rows past the block
      // are zero-filled.
      {
        const uint32_t sQ = sbase + C::OFF_Q;
        const int rows_valid = w.n_tok * p.group;
#pragma unroll 4
        for (int rr = row0; rr < C::BM; rr += KPP) {
          const bool v = rr < rows_valid;
          const int t = rr / p.group, g = rr - t * p.group;
          const bf16 *src = v ? p.q + ((int64_t)(w.q_tok0 + t) * p.hq + w.kvh * p.group + g) * HD + ch * 8
                              : p.q;
          cp_async_16(sQ + (ch >> 3) * (C::BM * 128) + sw128_off(rr, ch & 7), src, v ? 16u : 0u);
        }
        cp_async_commit();
        cp_async_wait_group<0>();
        fence_proxy_async_smem();
        mbar_arrive(&bars[B_Q_FULL]);
        ++q_cnt;
      }
      // key sources of this sequence
      int64_t kv_base = p.kv_indptr[w.b];
      int P_pool;  // keys [0, P_pool) are pool slots, the rest extend rows
      int64_t ext_base = 0;
      if (MODE == kTwoStage) {
        P_pool = p.kv_indptr[w.b + 1] - (int)kv_base;
        ext_base = p.qo_indptr[w.b];
      } else {
        P_pool = 0x7fffffff;
      }
      int pending = -1;
      for (int j = 0; j < nt; ++j) {
        const int stage = kv_cnt % C::NS;
        if (kv_cnt >= (uint32_t)C::NS) {
          // Publish the tile still in flight before blocking on a free stage:
          // the MMA warp frees this stage only after it has consumed that tile.
          if (pending >= 0) {
            cp_async_wait_group<0>();
            fence_proxy_async_smem();
            mbar_arrive(&bar_kv_full[pending]);
            pending = -1;
          }
          if (!mbar_wait(&bar_kv_empty[stage], ((kv_cnt / C::NS) - 1) & 1u, abort_flag)) {
            abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
            break;
          }
        }
        const int kb = w.k_begin + j * C::BN;
        const uint32_t sK = sbase + C::OFF_K + stage * C::K_BYTES;
        const uint32_t sV = sbase + C::OFF_V + stage * C::V_BYTES;
        // All of this thread's slot indices first (independent loads in
        // flight together), then the row copies.
        constexpr int NK = (C::BN + KPP - 1) / KPP;
        int64_t slot[NK];
#pragma unroll
        for (int i = 0; i < NK; ++i) {
          const int key = row0 + i * KPP;
          const int jpos = kb + key;
          slot[i] = -1;
          if (key < C::BN && jpos < w.k_end && !(MODE == kTwoStage && jpos >= P_pool)) {
            if (MODE == kUnified)
              slot[i] = __ldg(static_cast<const int64_t *>(p.kv_indices) + kv_base + jpos);
            else
              slot[i] = __ldg(static_cast<const int32_t *>(p.kv_indices) + kv_base + jpos);
          }
        }
#pragma unroll
        for (int i = 0; i < NK; ++i) {
          const int key = row0 + i * KPP;
          if (key >= C::BN) break;
          const int jpos = kb + key;
          bool v = jpos < w.k_end;
          const bf16 *krow = p.k_buf, *vrow = p.v_buf;
          if (v) {
            if (MODE == kTwoStage && jpos >= P_pool) {
              const int64_t te = ext_base + (jpos - P_pool);
              krow = p.k_ext + te * p.ke_st + (int64_t)w.kvh * p.ke_sh;
              vrow = p.v_ext + te * p.ve_st + (int64_t)w.kvh * p.ve_sh;
            } else if (slot[i] < 0 || slot[i] >= p.num_slots) {
              record_status(p.status, PKX_EDEVICE);
              v = false;
            } else {
              krow = p.k_buf + slot[i] * p.kb_ss + (int64_t)w.kvh * p.kb_sh;
              vrow = p.v_buf + slot[i] * p.vb_ss + (int64_t)w.kvh * p.vb_sh;
            }
          }
          const uint32_t off = (ch >> 3) * (C::BN * 128) + sw128_off(key, ch & 7);
          cp_async_16(sK + off, v ? krow + ch * 8 : p.k_buf, v ? 16u : 0u);
          cp_async_16(sV + off, v ? vrow + ch * 8 : p.v_buf, v ? 16u : 0u);
        }
        cp_async_commit();
        if (pending >= 0) {
          cp_async_wait_group<1>();
          fence_proxy_async_smem();
          mbar_arrive(&bar_kv_full[pending]);
        }
        pending = stage;
        ++kv_cnt;
      }
      if (pending >= 0) {
        cp_async_wait_group<0>();
        fence_proxy_async_smem();
        mbar_arrive(&bar_kv_full[pending]);
      }
    }
    cp_async_wait_group<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ============================================================== combine ====
// Merge the split-KV partials of every split query block: with lse_i the
// partial log-sum-exps and o_i the partial (normalised) outputs,
//   lse = log sum_i exp(lse_i),  o = sum_i exp(lse_i - lse) o_i
// (the merge_state formula applied n ways).
__global__ void __launch_bounds__(256) combine_kernel(const WsHeader *hdr, const CombineEntry *ce,
                                                      const float *plse, const float *po,
                                                      bf16 *o, float *lse, int hq, int group,
                                                      int hdv) {
  const int n_comb = hdr->n_combine;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int64_t idx = gw; idx < (int64_t)n_comb * kBlockM; idx += nw) {
    const int e = (int)(idx / kBlockM), r = (int)(idx % kBlockM);
    const CombineEntry E = ce[e];
    if (r >= E.n_tok * group) continue;
    float mx = -INFINITY;
    for (int i = 0; i < E.n_split; ++i) mx = fmaxf(mx, plse[(int64_t)(E.slot0 + i) * kBlockM + r]);
    const int t = r / group, g = r - t * group;
    const int64_t orow = (int64_t)(E.q_tok0 + t) * hq + E.kvh * group + g;
    if (mx == -INFINITY) {
      for (int c = lane * 8; c < hdv; c += 256)
        *reinterpret_cast<uint4 *>(o + orow * hdv + c) = make_uint4(0, 0, 0, 0);
      if (lane == 0 && lse) lse[orow] = -INFINITY;
      continue;
    }
    float wsum = 0.f;
    for (int i = 0; i < E.n_split; ++i)
      wsum += exp2f((plse[(int64_t)(E.slot0 + i) * kBlockM + r] - mx) * 1.4426950408889634f);
    const float inv = 1.0f / wsum;
    for (int c = lane * 8; c < hdv; c += 256) {
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      for (int i = 0; i < E.n_split; ++i) {
        const float wi =
            exp2f((plse[(int64_t)(E.slot0 + i) * kBlockM + r] - mx) * 1.4426950408889634f) * inv;
        const float *src = po + ((int64_t)(E.slot0 + i) * kBlockM + r) * hdv + c;
        const float4 a = *reinterpret_cast<const float4 *>(src);
        const float4 b = *reinterpret_cast<const float4 *>(src + 4);
        acc[0] += wi * a.x; acc[1] += wi * a.y; acc[2] += wi * a.z; acc[3] += wi * a.w;
        acc[4] += wi * b.x; acc[5] += wi * b.y; acc[6] += wi * b.z; acc[7] += wi * b.w;
      }
      uint4 pk;
      pk.x = pack_bf16(acc[0], acc[1]);
      pk.y = pack_bf16(acc[2], acc[3]);
      pk.z = pack_bf16(acc[4], acc[5]);
      pk.w = pack_bf16(acc[6], acc[7]);
      *reinterpret_cast<uint4 *>(o + orow * hdv + c) = pk;
    }
    if (lane == 0 && lse) lse[orow] = mx + logf(wsum);
  }
}

// ================================================================= host ====
int num_sms_current_device() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

int tokens_per_block(int group) { return group >= 1 && group <= kBlockM ? kBlockM / group : 0; }

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

WsLayout ws_layout(int batch, int num_q_tokens, int hkv, int group, int lv, int num_sms) {
  WsLayout L{};
  const int tok = tokens_per_block(group);
  L.unit_target = 4 * (num_sms > 0 ? num_sms : 160);
  L.qb_max = (tok > 0 ? (num_q_tokens + tok - 1) / tok : 0) + batch + 1;
  L.unit_max = L.unit_target + hkv * L.qb_max;
  L.slot_max = 2 * L.unit_target;
  L.comb_max = L.unit_target;
  size_t off = align256(sizeof(WsHeader));
  L.seq_off = off;
  off = align256(off + sizeof(int32_t) * 8 * (size_t)(batch + 1));
  L.qb_off = off;
  off = align256(off + sizeof(int32_t) * (size_t)L.qb_max);
  L.units_off = off;
  off = align256(off + sizeof(WorkUnit) * (size_t)L.unit_max);
  L.comb_off = off;
  off = align256(off + sizeof(CombineEntry) * (size_t)L.comb_max);
  L.plse_off = off;
  off = align256(off + sizeof(float) * (size_t)L.slot_max * kBlockM);
  L.po_off = off;
  off = align256(off + sizeof(float) * (size_t)L.slot_max * kBlockM * lv);
  L.total = off;
  return L;
}

template <int HD, int MODE>
static int launch_attn_kernel(const KParams &kp, int grid, cudaStream_t s) {
  using C = Cfg<HD>;
  static bool configured = false;  // per instantiation; attribute is per device
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<HD, MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess)
      return set_error(PKX_ECUDA, "cudaFuncSetAttribute(attn_kernel): %s", cudaGetErrorString(e));
    configured = true;
  }
  attn_kernel<HD, MODE><<<grid, C::THREADS, C::SMEM, s>>>(kp);
  return PKX_OK;
}

int launch_attention(const AttnArgs &a) {
  const int group = a.hq / a.hkv;
  const int nsm = num_sms_current_device();
  if (nsm <= 0) return set_error(PKX_ECUDA, "cannot query the current device");
  const int nq = a.mode == kDecode ? a.batch : a.num_q_tokens;
  WsLayout L = ws_layout(a.batch, nq, a.hkv, group, a.lv, nsm);
  if (a.workspace == nullptr || a.workspace_bytes < L.total)
    return set_error(PKX_EWORKSPACE, "workspace of %zu bytes given, %zu needed",
                     a.workspace_bytes, L.total);
  if (reinterpret_cast<uintptr_t>(a.workspace) & 255)
    return set_error(PKX_EINVAL, "workspace must be 256-byte aligned");
  uint8_t *ws = static_cast<uint8_t *>(a.workspace);
  WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);

  SchedParams sp;
  sp.mode = a.mode;
  sp.qo_indptr = a.qo_indptr;
  sp.kv_indptr = a.kv_indptr;
  sp.prefix_lens = a.prefix_lens;
  sp.batch = a.batch;
  sp.hkv = a.hkv;
  sp.tok = tokens_per_block(group);
  sp.window = a.window;
  sp.num_q_tokens = nq;
  sp.unit_target = L.unit_target;
  sp.qb_max = L.qb_max;
  sp.unit_max = L.unit_max;
  sp.comb_max = L.comb_max;
  sp.slot_max = L.slot_max;
  sp.seq = reinterpret_cast<int32_t *>(ws + L.seq_off);
  sp.qbt = reinterpret_cast<int32_t *>(ws + L.qb_off);
  sp.units = reinterpret_cast<WorkUnit *>(ws + L.units_off);
  sp.comb = reinterpret_cast<CombineEntry *>(ws + L.comb_off);
  sp.hdr = hdr;
  sched_kernel<<<1, 1024, 0, a.stream>>>(sp);

  KParams kp;
  kp.q = static_cast<const bf16 *>(a.q);
  kp.o = static_cast<bf16 *>(a.o);
  kp.lse = a.lse;
  kp.k_ext = static_cast<const bf16 *>(a.k_ext);
  kp.v_ext = static_cast<const bf16 *>(a.v_ext);
  kp.ke_st = a.ke_st;
  kp.ke_sh = a.ke_sh;
  kp.ve_st = a.ve_st;
  kp.ve_sh = a.ve_sh;
  kp.k_buf = static_cast<const bf16 *>(a.k_buf);
  kp.v_buf = static_cast<const bf16 *>(a.v_buf);
  kp.kb_ss = a.kb_ss;
  kp.kb_sh = a.kb_sh;
  kp.vb_ss = a.vb_ss;
  kp.vb_sh = a.vb_sh;
  kp.num_slots = a.num_slots;
  kp.qo_indptr = a.qo_indptr;
  kp.kv_indptr = a.kv_indptr;
  kp.kv_indices = a.kv_indices;
  kp.hq = a.hq;
  kp.group = group;
  kp.window = a.window;
  const float log2e = 1.4426950408889634f;
  const float sm_scale = a.sm_scale > 0.f ? a.sm_scale : 1.0f / sqrtf((float)a.lq);
  kp.use_cap = a.logit_cap > 0.f;
  kp.scale_log2 = sm_scale * log2e;
  kp.cap_pre = kp.use_cap ? sm_scale / a.logit_cap : 0.f;
  kp.cap_log2 = kp.use_cap ? a.logit_cap * log2e : 0.f;
  kp.units = sp.units;
  kp.hdr = hdr;
  kp.status = &hdr->status;
  kp.plse = reinterpret_cast<float *>(ws + L.plse_off);
  kp.po = reinterpret_cast<float *>(ws + L.po_off);

  int rc;
  const int grid = nsm;
  cudaEvent_t ev_before = nullptr, ev_after = nullptr;
  attention_events(&ev_before, &ev_after);
  if (ev_before) cudaEventRecord(ev_before, a.stream);
  if (a.lq == 128 && a.lv == 128) {
    if (a.mode == kTwoStage) rc = launch_attn_kernel<128, kTwoStage>(kp, grid, a.stream);
    else if (a.mode == kUnified) rc = launch_attn_kernel<128, kUnified>(kp, grid, a.stream);
    else rc = launch_attn_kernel<128, kDecode>(kp, grid, a.stream);
  } else if (a.lq == 64 && a.lv == 64) {
    if (a.mode == kTwoStage) rc = launch_attn_kernel<64, kTwoStage>(kp, grid, a.stream);
    else if (a.mode == kUnified) rc = launch_attn_kernel<64, kUnified>(kp, grid, a.stream);
    else rc = launch_attn_kernel<64, kDecode>(kp, grid, a.stream);
  } else {
    return set_error(PKX_EUNSUPPORTED, "head dims (%d, %d) not built", a.lq, a.lv);
  }
  if (rc != PKX_OK) return rc;
  if (ev_after) cudaEventRecord(ev_after, a.stream);
  combine_kernel<<<nsm * 2, 256, 0, a.stream>>>(hdr, sp.comb, kp.plse, kp.po, kp.o, a.lse, a.hq,
                                               group, a.lv);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(PKX_ECUDA, "attention launch: %s", cudaGetErrorString(e));
  return PKX_OK;
}

}  // namespace pkx
