// attention.cu -- extend and decode attention over a page-size-1 KV pool for
// sm_103a: a device-side work scheduler, a warp-specialised tcgen05/TMEM
// attention kernel whose K/V rows are gathered by cp.async copy warps, and
// the split-KV combine.
//
// Method (sglang extend_attention.py, _fwd_kernel_unified and
// extend_attention_fwd; flashinfer_backend.py, forward_decode):
//   for each query row and each visible key j:  s_j = sm_scale * <q, k_j>,
//   optionally s_j = cap * tanh(s_j / cap); visible iff j <= qpos (or, with a
//   custom mask, iff its mask byte is set) and, with a window W > 0,
//   qpos - j <= W; o = sum_j softmax(s)_j v_j (a sink logit per head joins
//   the denominator); lse = log sum exp s.  The online softmax keeps a
//   running max and sum per row and rescales the accumulator when the max
//   moves.
//
// GB300 design (differs from the pages' Triton kernel, which launches one
// program per (sequence, q head, 128-row block) and re-reads K/V per q head):
//  * a Q tile = 128 rows = (tokens x the Hq/Hkv query heads of one KV head),
//    and a CTA runs two Q tiles of consecutive tokens against each K/V tile:
//    K/V of a KV head are gathered once for 2 x 128 query rows;
//  * K and V rows are gathered from the pool by four warps with 16-byte
//    cp.async copies placed straight into the 128-byte-swizzled layout the
//    MMA descriptors read (random 256-byte rows need many copying threads
//    to reach HBM bandwidth; a TMA gather4 moves only four 128-byte rows
//    per instruction and stalls on its issue rate); each copying thread
//    arrives on the stage barrier when its own copies land.  An index warp
//    claims work units, resolves every tile's slot indices into a small smem
//    ring ahead of the copy warps and loads the Q tiles (3-D TMA boxes).
//    setmaxnreg moves registers from these warps to the softmax warpgroups;
//  * QK^T and PV are tcgen05.mma (M=128, bf16 in, fp32 accumulate in TMEM).
//    TMEM holds S and O of both Q tiles (4 x 128 columns).  The softmax
//    warpgroup of a tile writes P (bf16) back over its S columns and PV
//    reads A = P straight from TMEM.  While one warpgroup runs its softmax,
//    the tensor core runs the other tile's PV and QK^T;
//  * a unit with one Q tile (every decode unit; split extend units of at
//    most 128/G tokens) runs two key streams instead: the two warpgroups
//    take alternate K/V tiles with their own S/P and O, and the combine
//    merges the two partials;
//  * an fp8 pool (e4m3 / e5m2 codes with k_scale, v_scale) is staged as
//    codes and converted in place to exact bf16 (f16 for decode) by the
//    copy warps; the scales go into the logit scale and P (or the output);
//  * the KV loop stops at the causal diagonal and starts at the window edge
//    (the Triton kernel walks every tile and masks);
//  * a device-built work list (no host sync, graph-safe) splits long key
//    ranges across CTAs (split-KV); a combine kernel merges the partial
//    (o, lse) pairs with the merge_state formula;
//  * a persistent grid of one CTA per SM claims the work units in cost
//    order.
#include <algorithm>
#include <climits>
#include <cstdio>
#include <cstring>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "pkx_internal.h"
#include "ptx.cuh"

namespace pkx {

using bf16 = __nv_bfloat16;

// ============================================================ scheduler ====
struct SchedParams {
  int mode;
  const int32_t *qo_indptr, *kv_indptr, *prefix_lens;
  int batch, hkv, tok, window, num_q_tokens;
  int bn;        // keys per K/V tile
  int q_tile_tok;  // query tokens of one Q tile
  int no_causal;   // a custom mask replaces the causal mask: blocks see every key
  int key_set;     // two-stage form only: kAllKeys, kPrefixKeys or kExtendKeys
  int keep_status; // leave the status word as an earlier pass left it
  int two_streams; // GQA kernel: decode units run two key streams, each with its own
                   // partial slot; split extend units of one query tile run two
                   // streams into the two halves of their slot
  int n_dsplit;  // units per (block, split): value-dim slices (1, or 4 for MLA)
  int unit_target, qb_max, unit_max, comb_max, slot_max;
  // Stream partition (parts > 0, a multiple of hkv): per KV head, the
  // blocks' key tiles laid end to end, each weighted by its block's Q tiles,
  // are cut into parts / hkv equal shares of that cost (the same cuts for
  // every head), a block is split at the first tile boundary of each share,
  // each piece is claimed by its share's CTA (or CTA pair), and
  // part_first[k] is the first claim position of share k (k <= parts).
  int parts;
  int32_t *part_first;
  int32_t *seq;  // 8 arrays of batch+1 ints
  int32_t *qbt;  // [6][qb_max]: tiles, sequence, unit / slot / combine offsets, tile offset per block
  int seq_in_smem, blk_in_smem;  // those arrays in dynamic shared memory instead
  WorkUnit *units;
  int32_t *uorder;  // units by cost, largest first
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
    // One half of the ragged + paged split: the prefix keys alone (every
    // one visible to every extend query), or the extend keys alone with
    // causal positions counted from the first extend token.
    if (p.key_set == kPrefixKeys) d.T = d.P;
    else if (p.key_set == kExtendKeys) { d.P = 0; d.T = d.E; }
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
  hi = p.no_causal ? d.T : min(qmax + 1, d.T);
  lo = p.window > 0 ? max(0, qmin - p.window) : 0;
  if (hi < lo) hi = lo;
}

// Number of K/V tiles of the key range [kb, ke) when tiles may not straddle
// `split` (the prefix / extend boundary of the two-stage form).
__device__ __forceinline__ int range_tiles(int kb, int ke, int split, int bn) {
  const int pe = min(ke, split), eb = max(kb, split);
  const int n_pre = pe > kb ? (pe - kb + bn - 1) / bn : 0;
  const int n_ext = ke > eb ? (ke - eb + bn - 1) / bn : 0;
  return n_pre + n_ext;
}

// Exclusive scan of one value per thread over the 1024-thread block (warp
// shuffles, then one warp over the 32 warp totals: three block barriers);
// the total goes to *total.  sh must hold 32 ints.
__device__ int block_scan_value(int v, int *sh, int &total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int t = sh[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    sh[lane] = t;
  }
  __syncthreads();
  const int excl = (wid ? sh[wid - 1] : 0) + x - v;
  total = sh[31];
  __syncthreads();  // sh may be reused by the caller
  return excl;
}

// Maximum of one value per thread over the 1024-thread block.
__device__ int block_max(int v, int *sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) sh[wid] = v;
  __syncthreads();
  int m = sh[lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __syncthreads();  // sh may be reused by the caller
  return m;
}

// Exclusive scan of in[0..n) into out[0..n) by the whole 1024-thread block
// (each thread a contiguous chunk); returns the total.  in and out may
// alias.
__device__ int block_exclusive_scan(const int32_t *in, int32_t *out, int n, int *sh) {
  const int tid = threadIdx.x;
  const int ch = (n + 1023) / 1024;
  const int beg = min(n, tid * ch), end = min(n, beg + ch);
  int local = 0;
  for (int i = beg; i < end; ++i) local += in[i];
  int total;
  int run = block_scan_value(local, sh, total);
  for (int i = beg; i < end; ++i) {
    int v = in[i];
    out[i] = run;
    run += v;
  }
  __syncthreads();
  return total;
}

// Buckets of the counting sorts (claim order, sequence ranks).
constexpr int kCostBuckets = 2048;
// Dynamic shared memory the scheduler may take: the histogram always, and
// the per-sequence and per-block arrays when they fit (else they live in
// the workspace, which is slower but has no size limit).
constexpr int kSchedSmemMax = 200 * 1024;
// Per-sequence and per-block arrays of the scheduler.
constexpr int kSchedSeqArrays = 5, kSchedBlockArrays = 6;

// Relative cost of a unit: its K/V tiles times its Q tiles, plus one for the
// per-unit prologue and epilogue (clamped to the sort's bucket range).
__device__ __forceinline__ int unit_cost(const WorkUnit &w, int q_tile_tok) {
  const int nq = (w.n_tok + q_tile_tok - 1) / q_tile_tok;
  return min(w.n_tiles * max(nq, 1) + 1, kCostBuckets - 1);
}

// Device-side work list.  Only the first phase reads global memory (the
// indptrs); the per-sequence and per-block values then live in shared memory
// (or, for very large batches, in the workspace), so the later phases are
// throughput-bound rather than chains of dependent global loads.
//   1. per sequence: P, E, T, first query row and query blocks; a scan gives
//      each sequence's first block;
//   2. per query block (of one KV head): its K/V tiles; their total sets the
//      split-KV chunk C;
//   3. per block: units (splits x value slices), partial slots and combine
//      entries, and their offsets (scans);
//   4-6. combine entries; every unit written and counted by its claim key
//      (its cost, largest first), then placed in the claim order.
// Largest first balances the CTAs, which claim units at run time.  (Orders
// that keep a sequence's units together cut DRAM re-reads of K/V but cost
// more in balance than they save: the kernel is not bound by DRAM.)
__global__ void __launch_bounds__(1024, 1) sched_kernel(SchedParams p) {
  extern __shared__ int sdyn[];
  __shared__ int sh[32];
  __shared__ int s_c, s_share;
  const int tid = threadIdx.x;
  const int B = p.batch;
  const int S1 = B + 1;
  int *hist = sdyn;
  int *seqa = p.seq_in_smem ? sdyn + kCostBuckets : p.seq;
  int *sP = seqa, *sE = seqa + S1, *sT = seqa + 2 * S1, *sQ0 = seqa + 3 * S1;
  int *sOff = seqa + 4 * S1;   // first query block of each sequence; [B] = total
  int *blk = p.blk_in_smem ? sdyn + kCostBuckets + (p.seq_in_smem ? kSchedSeqArrays * S1 : 0)
                           : p.qbt;
  int *bNt = blk, *bSeq = blk + p.qb_max, *bUo = blk + 2 * p.qb_max;
  int *bSo = blk + 3 * p.qb_max, *bCo = blk + 4 * p.qb_max;
  int *bTo = blk + 5 * p.qb_max;  // stream partition: first tile of the block in the stream

  grid_dep_wait();    // inputs written by the previous kernel on the stream
  grid_dep_launch();  // the attention grid may start its prologue now
  if (tid == 0) {
    if (!p.keep_status) p.hdr->status = 0;
    p.hdr->next_unit = 0;
  }

  // 1. per sequence
  for (int b = tid; b < B; b += 1024) {
    const SeqDims d = seq_dims(p, b);
    sP[b] = d.P;
    sE[b] = d.E;
    sT[b] = d.T;
    sQ0[b] = d.qbase;
    sOff[b] = d.nqb;
  }
  __syncthreads();
  const int total_qb = block_exclusive_scan(sOff, sOff, B, sh);
  if (tid == 0) sOff[B] = total_qb;
  if (total_qb >= p.qb_max) {  // cannot happen for consistent indptrs (one entry spare)
    if (tid == 0) {
      record_status(&p.hdr->status, PKX_EDEVICE);
      p.hdr->n_units = 0;
      p.hdr->n_combine = 0;
    }
    return;
  }
  __syncthreads();
  auto dims = [&](int b) {
    SeqDims d;
    d.P = sP[b];
    d.E = sE[b];
    d.T = sT[b];
    d.qbase = sQ0[b];
    d.nqb = sOff[b + 1] - sOff[b];
    return d;
  };
  // the sequence of query block qb: the last b with sOff[b] <= qb
  auto seq_of = [&](int qb) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sOff[mid] <= qb) lo = mid;
      else hi = mid - 1;
    }
    return lo;
  };

  // 2. K/V tiles per query block; total tiles -> chunk size C
  int my_tiles = 0;
  for (int qb = tid; qb < total_qb; qb += 1024) {
    const int b = seq_of(qb);
    const SeqDims d = dims(b);
    int lo, hi, i0, i1;
    qblock_range(p, d, qb - sOff[b], lo, hi, i0, i1);
    const int nt = (hi - lo + p.bn - 1) / p.bn;
    bNt[qb] = nt;
    bSeq[qb] = b;
    my_tiles = min(my_tiles + nt, 0x1fffff);
    // stream partition: the block's cost, its tiles times its Q tiles
    if (p.parts > 0) bTo[qb] = nt * max(1, (i1 - i0 + p.q_tile_tok - 1) / p.q_tile_tok);
  }
  int tiles_all;
  block_scan_value(my_tiles, sh, tiles_all);
  const bool stream = p.parts > 0;
  int cost_all = 0;
  if (stream) {
    __syncthreads();
    cost_all = block_exclusive_scan(bTo, bTo, total_qb, sh);  // first cost of each block
    if (tid == 0) bTo[total_qb] = cost_all;
  }
  if (tid == 0) {
    const long long total_tiles = (long long)tiles_all * p.hkv * p.n_dsplit;
    const long long c = (total_tiles + p.unit_target - 1) / p.unit_target;
    s_c = (int)max((long long)kMinSplitTiles, c);
    const int ppk = stream ? p.parts / p.hkv : 1;  // shares per KV head
    // at least two, the largest tile cost, so that every share holds a tile
    // boundary and no piece is empty
    s_share = stream ? max(2, (cost_all + ppk - 1) / ppk) : 0;
    p.hdr->split_tiles = stream ? s_share : s_c;
  }
  __syncthreads();
  const int C = s_c, share = s_share;

  // 3. per query block: units, slots, combine entries; their offsets
  const int nd = p.n_dsplit;
  // splits of block qb: chunks of C tiles, or (stream partition) one piece
  // per share its tiles touch
  auto splits = [&](int qb) {
    const int nt = bNt[qb];
    if (nt <= 0) return 1;
    if (!stream) return (nt + C - 1) / C;
    // a tile belongs to the share its first cost falls in
    const int g0 = bTo[qb], wq = (bTo[qb + 1] - g0) / nt;
    return (g0 + (nt - 1) * wq) / share - g0 / share + 1;
  };
  // two key streams: every decode unit has two partial slots and every
  // block a combine entry
  const bool dec2 = p.two_streams && p.mode == kDecode;
  const int spu = dec2 ? 2 : 1;
  auto combined = [&](int S) { return S > 1 || dec2; };
  const int chunk = (total_qb + 1023) / 1024;
  const int qb_beg = min(total_qb, tid * chunk), qb_end = min(total_qb, qb_beg + chunk);
  int lu = 0, ls = 0, lc = 0;
  for (int qb = qb_beg; qb < qb_end; ++qb) {
    const int S = splits(qb);
    lu += S * nd;
    if (combined(S)) {
      ls += S * spu;
      lc += 1;
    }
  }
  int tu, ts, tcm;
  int u0 = block_scan_value(lu, sh, tu);
  int s0 = block_scan_value(ls, sh, ts);
  int c0 = block_scan_value(lc, sh, tcm);
  for (int qb = qb_beg; qb < qb_end; ++qb) {
    bUo[qb] = u0;
    bSo[qb] = s0;
    bCo[qb] = c0;
    const int S = splits(qb);
    u0 += S * nd;
    if (combined(S)) {
      s0 += S * spu;
      c0 += 1;
    }
  }
  const long long n_units_l = (long long)tu * p.hkv, n_slots_l = (long long)ts * p.hkv,
                  n_comb_l = (long long)tcm * p.hkv;
  if (n_units_l > p.unit_max || n_slots_l > p.slot_max || n_comb_l > p.comb_max) {
    if (tid == 0) {
      record_status(&p.hdr->status, PKX_EDEVICE);
      p.hdr->n_units = 0;
      p.hdr->n_combine = 0;
    }
    return;
  }
  const int n_units = (int)n_units_l, n_comb = (int)n_comb_l;

  // 4. claim keys: the unit's cost, largest first
  for (int i = tid; i < kCostBuckets; i += 1024) hist[i] = 0;
  __syncthreads();
  auto claim_key = [&](const WorkUnit &w) { return kCostBuckets - 1 - unit_cost(w, p.q_tile_tok); };

  // 5. combine entries, one (KV head, query block) pair per thread
  const int n_pairs = p.hkv * total_qb;
  for (int idx = tid; idx < n_pairs; idx += 1024) {
    const int kvh = idx / total_qb, qb = idx - kvh * total_qb;
    const int S = splits(qb);
    if (!combined(S)) continue;
    const int b = bSeq[qb];
    const SeqDims d = dims(b);
    int lo, hi, i0, i1;
    qblock_range(p, d, qb - sOff[b], lo, hi, i0, i1);
    CombineEntry e;
    e.q_tok0 = d.qbase + i0;
    e.n_tok = i1 - i0;
    e.kvh = kvh;
    e.slot0 = kvh * ts + bSo[qb];
    e.n_split = S * spu;
    // a split extend block of one query tile: its units' second stream
    // fills the second half of each slot
    e.pad[0] = p.two_streams && p.mode != kDecode && S > 1 && i1 - i0 <= p.q_tile_tok ? 2 : 1;
    e.pad[1] = e.pad[2] = 0;
    p.comb[kvh * tcm + bCo[qb]] = e;
  }
  // Unit u: KV head u / tu; within the head, query block qb is the last
  // block with bUo[qb] <= rest, and the unit is its (split, value slice)
  // number rest - bUo[qb].
  auto unit_at = [&](int u) {
    const int kvh = u / tu, rest = u - kvh * tu;
    int lo_b = 0, hi_b = total_qb - 1;
    while (lo_b < hi_b) {
      const int mid = (lo_b + hi_b + 1) >> 1;
      if (bUo[mid] <= rest) lo_b = mid;
      else hi_b = mid - 1;
    }
    const int qb = lo_b, k = rest - bUo[qb];
    const int sp = k / nd, dq = k - sp * nd;
    const int b = bSeq[qb];
    const SeqDims d = dims(b);
    const int split_at = p.mode == kTwoStage ? d.P : INT_MAX;
    int lo, hi, i0, i1;
    qblock_range(p, d, qb - sOff[b], lo, hi, i0, i1);
    const int nt = bNt[qb], S = splits(qb);
    // split sp covers tiles [sp nt / S, (sp + 1) nt / S) (sizes differ by
    // one at most), or (stream partition) the block's tiles inside share
    // g0 / share + sp
    int t0 = (int)((long long)sp * nt / S), t1 = (int)((long long)(sp + 1) * nt / S);
    int part = 0;
    if (stream) {
      // share k of the head takes the block's tiles whose first cost lies
      // in [k share, (k + 1) share); a tile costs wq (the block's Q tiles),
      // at most share, so every share between the first and the last tile's
      // holds a tile
      const int g0 = bTo[qb], ppk = p.parts / p.hkv;
      const int wq = nt > 0 ? (bTo[qb + 1] - g0) / nt : 1;
      const int k = min(g0 / share + sp, ppk - 1);  // the share within the head
      t0 = sp == 0 ? 0 : min(nt, (k * share - g0 + wq - 1) / wq);
      t1 = sp == S - 1 ? nt : min(nt, ((k + 1) * share - g0 + wq - 1) / wq);
      part = kvh * ppk + k;
    }
    WorkUnit w;
    w.q_tok0 = d.qbase + i0;
    w.n_tok = i1 - i0;
    w.qpos0 = d.P + i0;
    w.kvh = kvh;
    w.k_begin = min(hi, lo + t0 * p.bn);
    w.k_end = min(hi, lo + t1 * p.bn);
    w.k_split = split_at;
    w.n_tiles = range_tiles(w.k_begin, w.k_end, split_at, p.bn);
    w.b = b;
    w.slot = combined(S) ? kvh * ts + bSo[qb] + sp * spu : -1;
    w.dq = dq;
    w.claim = stream ? part : 0;
    return w;
  };

  // 6. units, consecutive threads on consecutive units (their records go
  //    out as 16-byte stores); pass 0 builds and writes them with their
  //    claim keys and counts the keys, pass 1 reads the keys back and places
  //    the units in the claim order.  Lanes of a warp whose units share a
  //    key make one atomic for the group (units of one sequence and cost
  //    class share a key, so per-unit atomics serialise).
  const int lane = tid & 31;
  for (int pass = 0; pass < 2; ++pass) {
    for (int base = tid - lane; base < n_units; base += 1024) {
      const int u = base + lane;
      const bool act = u < n_units;
      WorkUnit w;
      int key = -1;
      if (act) {
        if (pass == 0) {
          w = unit_at(u);
          key = stream ? w.claim : claim_key(w);  // stream partition: the share, in order
          w.claim = key;
        } else {
          key = p.units[u].claim;  // written in pass 0 (the block barrier between passes orders it)
        }
      }
      const unsigned grp = __match_any_sync(0xffffffffu, key);
      const int leader = __ffs(grp) - 1;
      int first = 0;
      if (act && lane == leader) first = atomicAdd(&hist[key], __popc(grp));
      first = __shfl_sync(0xffffffffu, first, leader);
      if (act) {
        if (pass == 0) p.units[u] = w;
        else p.uorder[first + __popc(grp & ((1u << lane) - 1u))] = u;
      }
    }
    __syncthreads();
    if (pass == 0) {
      block_exclusive_scan(hist, hist, kCostBuckets, sh);
      // each share's first claim position (keys are shares, all below parts)
      if (stream)
        for (int k = tid; k <= p.parts; k += 1024) p.part_first[k] = hist[k];
    }
  }
  if (tid == 0) {
    p.hdr->n_units = n_units;
    p.hdr->n_combine = n_comb;
  }
}

// ============================================================ attention ====
struct KParams {
  const bf16 *q;  // read directly by the MLA kernel (the GQA kernel uses the TMA map)
  bf16 *o;
  float *lse;
  const bf16 *k_pool, *v_pool, *k_ext, *v_ext;
  int64_t kb_ss, vb_ss, ke_st, ve_st;  // row strides (elements): slot / token
  int64_t kb_sh, vb_sh, ke_sh, ve_sh;  // head strides (elements)
  int64_t num_slots;
  const int32_t *qo_indptr, *kv_indptr;
  const void *kv_indices;
  int hq, group, tok, q_box_tok, window, use_cap, rows_per_slot;
  float scale_log2;  // sm_scale * log2(e)           (no cap)
  float cap_pre;     // sm_scale / cap                (cap)
  float cap_log2;    // cap * log2(e)                 (cap)
  const uint8_t *custom_mask;   // nullable: byte per (extend row, key); replaces causal
  const int32_t *mask_indptr;   // [batch+1] offsets of each sequence's mask rows
  const float *sinks;           // nullable [hq] sink logits (natural log)
  // fp8 pool: a key reads code * k_scale, a value code * v_scale.  The codes
  // go to shared memory as exact bf16; k_scale is folded into the logit
  // scale of pool tiles, v_scale into their P through the exponent
  // (2^(s - m + log2 v_scale)), and the tile's row sum is divided back
  float scale_log2_k, cap_pre_k, log2_v_scale, inv_v_scale, v_scale;
  int dec_two;  // decode units run two key streams (else one)
  const int32_t *prefix_lens;   // unified form: prefix length per sequence
  const WorkUnit *units;
  const int32_t *uorder;  // units by cost, largest first
  const WsHeader *hdr;
  int32_t *next_unit;     // claim counter over uorder (zeroed by the scheduler)
  const int32_t *part_first;  // MLA pairs: each pair's claim positions (stream partition), or null
  int32_t *status;
  float *plse, *po;
  // two-stage form with the fused KV write: the pool slot of each extend
  // token (nullable), and the pools as writable pointers
  const int64_t *cache_loc;
  bf16 *k_pool_w, *v_pool_w;
  uint64_t wait_ns;       // time limit of every bounded wait
  int stall;              // test hook: the softmax warps first wait on a barrier
                          // no thread arrives at, so that the limit runs out
};

// TMA descriptor of q (3-D: dim, head, token).
struct TMaps {
  CUtensorMap q;
};

// Head configuration HD: 64 and 128 are Lq = Lv = HD (two Q tiles per unit);
// 192 and 288 are the split head dims Lq = 192 / Lv = 128 and Lq = 288 /
// Lv = 256 (sglang extend_attention.py, _get_block_sizes_for_extend_attention:
// 192 = 128 + 64 rope, 288 = 256 + 32 rope), run with one Q tile per unit and
// one key stream: S (128 columns) and O (Lv columns) of the one tile fit TMEM,
// and a K stage of 128 keys fits shared memory next to the larger Q tile.
template <int HD>
struct Cfg {
  static constexpr bool SPLIT = HD == 192 || HD == 288;
  static constexpr int BM = kBlockM, BN = kBlockN;
  static constexpr int LQ = HD;
  static constexpr int HDV = HD == 192 ? 128 : HD == 288 ? 256 : HD;
  static constexpr int QA = (LQ + 63) / 64;  // 64-dim swizzle atoms of a Q / K row
  static constexpr int VA = HDV / 64;        // ... of a V row
  static constexpr int NQT = SPLIT ? 1 : 2;  // Q tiles per unit
  static constexpr bool TWO_OK = !SPLIT;     // two key streams for one-tile units
  static constexpr int NK = HD == 128 ? 3 : HD == 64 ? 5 : HD == 192 ? 2 : 1;  // K ring stages
  static constexpr int NV = HD == 128 ? 2 : HD == 64 ? 5 : HD == 192 ? 2 : 1;  // V ring stages
  static constexpr int NI = HD == 64 ? 4 : 3;     // row-index ring stages
  static constexpr int Q_BYTES = BM * QA * 128;   // one Q tile (a 288-dim row fills 4.5 atoms)
  static constexpr int K_BYTES = BN * QA * 128;
  static constexpr int V_BYTES = BN * VA * 128;
  static constexpr int I_BYTES = BN * 4;        // int32 row of each key
  static constexpr int OFF_Q = 0;               // NQT Q tiles
  static constexpr int OFF_K = OFF_Q + NQT * Q_BYTES;
  static constexpr int OFF_V = OFF_K + NK * K_BYTES;
  static constexpr int OFF_I = OFF_V + NV * V_BYTES;
  static constexpr int OFF_BAR = OFF_I + NI * I_BYTES;
  // decode over an fp8 pool: the codes land in a ring of NRAW slots (the
  // unused second Q tile and K stage 0) and are converted from there
  static constexpr int NRAW = 4;
  static constexpr int RAW_BYTES = BN * LQ;  // the fp8 codes of one K or V tile
  static constexpr int OFF_RAW = OFF_Q + Q_BYTES;
  static constexpr int N_BARS = 17 + 2 * NK + 2 * NV + 2 * NI + 2 * NRAW;
  static constexpr int SMEM = OFF_BAR + N_BARS * 8 + 1024;  // + alignment slack
  // S0 | S1 | O0 | O1, 128 columns each (split dims: S0 | unused | O0 of Lv)
  static constexpr int TMEM_COLS = 512;
  static_assert(2 * BN + NQT * HDV <= TMEM_COLS, "TMEM budget");
  static constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, 0);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, HDV, 1);
  // warps 0-7: two softmax warpgroups; 8: MMA; 9: row indices + Q;
  // 10-13: copies; 14-15: idle
  static constexpr int THREADS = 512;
  static constexpr int COPY_WARP0 = 10;
  static constexpr int COPY_THREADS = 128;
  // keys per copy pass: whole rows per thread group for 64 / 128 dims; by
  // swizzle atom (chunk t % 8 of every atom, keys t / 8 + 16 i) for the
  // split dims, whose 24 or 36 chunks per row do not divide 128 threads
  static constexpr int KPP = SPLIT ? 16 : COPY_THREADS / (HD / 8);
  // Registers: the kernel launches with REGS_LAUNCH per thread (checked at
  // build time); the softmax warpgroups take REGS_SOFTMAX, the other two
  // give back down to REGS_OTHER.  The split must add up exactly.
  static constexpr int REGS_LAUNCH = 128, REGS_SOFTMAX = 168, REGS_OTHER = 88;
  static_assert(256 * REGS_SOFTMAX + 256 * REGS_OTHER == THREADS * REGS_LAUNCH,
                "register split must match the launch allocation");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(SPLIT || NRAW * RAW_BYTES == Q_BYTES + K_BYTES,
                "the raw ring fills the second Q tile and K stage 0");
};

// barrier indices
enum {
  B_Q_FULL = 0,
  B_Q_EMPTY = 1,
  B_S_FULL = 2,  // + Q tile
  B_P_FULL = 4,  // + Q tile
  B_O_DONE = 6,  // + Q tile
  B_FINAL = 8,
  B_U_FULL = 9,    // + unit ring slot (kUnitRing)
  B_U_EMPTY = 12,  // + unit ring slot
  B_Q_CONV = 15,   // decode over fp8: the query rows converted to f16
  B_NEVER = 16,    // no thread ever arrives (the stall hook waits on it)
  B_RING = 17,  // K full[NK], K empty[NK], V full[NV], V empty[NV],
                // I full[NI], I empty[NI], raw full[NRAW], raw empty[NRAW]
};

// Key range [kb, ke) of tile j of a unit (tiles never straddle k_split).
template <int BN = kBlockN>
__device__ __forceinline__ void tile_keys(const WorkUnit &w, int j, int &kb, int &ke) {
  const int pe = min(w.k_end, w.k_split);
  const int n_pre = pe > w.k_begin ? (pe - w.k_begin + BN - 1) / BN : 0;
  if (j < n_pre) {
    kb = w.k_begin + j * BN;
    ke = min(kb + BN, pe);
  } else {
    kb = max(w.k_begin, w.k_split) + (j - n_pre) * BN;
    ke = min(kb + BN, w.k_end);
  }
}

__device__ __forceinline__ void abort_cta(volatile int *abort_flag, int32_t *status, int code) {
  *abort_flag = 1;
  record_status(status, code);
}

// Units are claimed at run time: the index warp takes the next position of
// the cost order (largest first) from a global counter and passes the unit
// to the CTA's other warps through a small ring in shared memory (-1 ends
// the stream).  A CTA that finishes early simply claims more, so the work
// evens out without a cost model.
constexpr int kUnitRing = 3;
// Consumer side: the uc-th unit of this CTA, or -1 at the end or on a
// timeout (then *ok is cleared).  The slot is released as soon as it is
// read: by every lane of a warp (lane 0 arrives) or by a lone thread.
__device__ __forceinline__ int ring_unit(uint64_t *u_full, uint64_t *u_empty,
                                         const volatile int *ring, uint32_t uc,
                                         volatile int *abort_flag, bool whole_warp, bool &ok,
                                         uint64_t limit_ns) {
  const int slot = uc % kUnitRing;
  if (!mbar_wait(&u_full[slot], (uc / kUnitRing) & 1u, abort_flag, limit_ns)) {
    ok = false;
    return -1;
  }
  const int u = ring[slot];
  if (whole_warp) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&u_empty[slot]);
  } else {
    mbar_arrive(&u_empty[slot]);
  }
  return u;
}

// MASK: a custom mask replaces the causal mask (its own instantiation, so
// the unmasked kernel carries none of the mask code).
// Eight fp8 codes (e4m3 for FMT 1, e5m2 for FMT 2) as eight bf16 of the same
// values (exact: every code is a bf16 value), in element order (the code in
// the lowest byte first).
template <int FMT>
__device__ __forceinline__ uint4 fp8x8_to_bf16x8(uint2 raw) {
  constexpr __nv_fp8_interpretation_t kind = FMT == 1 ? __NV_E4M3 : __NV_E5M2;
  const uint32_t w[2] = {raw.x, raw.y};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h(__nv_cvt_fp8x2_to_halfraw2(
        static_cast<__nv_fp8x2_storage_t>(w[i >> 1] >> (16 * (i & 1))), kind));
    const float2 f = __half22float2(h);
    out[i] = pack_bf16(f.x, f.y);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Eight fp8 codes as eight f16 of the same values (exact), element order
// kept: an e5m2 code is the top byte of its f16; e4m3 goes through the
// converter.
template <int FMT>
__device__ __forceinline__ uint4 fp8x8_to_f16x8(uint2 raw) {
  uint32_t out[4];
  if constexpr (FMT == 2) {
    out[0] = __byte_perm(raw.x, 0u, 0x1404);
    out[1] = __byte_perm(raw.x, 0u, 0x3424);
    out[2] = __byte_perm(raw.y, 0u, 0x1404);
    out[3] = __byte_perm(raw.y, 0u, 0x3424);
  } else {
    const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
          static_cast<__nv_fp8x2_storage_t>(w[i >> 1] >> (16 * (i & 1))), __NV_E4M3);
      out[i] = (uint32_t)h.x | ((uint32_t)h.y << 16);
    }
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Eight bf16 times 2^-8 as eight f16 (round to nearest): the power of two
// keeps any bf16 of magnitude below 2^24 inside the f16 range; the logit
// scale takes the 2^8 back.
constexpr float kQF16Down = 0x1p-8f, kQF16Up = 256.0f;
__device__ __forceinline__ uint4 bf16x8_to_f16x8_scaled(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16) * kQF16Down;
    const float hi = __uint_as_float(w[i] & 0xFFFF0000u) * kQF16Down;
    const __half2 h = __floats2half2_rn(lo, hi);
    out[i] = *reinterpret_cast<const uint32_t *>(&h);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// FMT: the pool's element format (0 bf16; 1 fp8 e4m3, 2 fp8 e5m2 with
// k_scale / v_scale).  Extend rows of the two-stage form are always bf16.
template <int HD, int MODE, bool MASK, int FMT = 0>
__global__ void __launch_bounds__(Cfg<HD>::THREADS, 1)
    attn_kernel(const __grid_constant__ TMaps tm, const KParams p) {
  using C = Cfg<HD>;
  // Decode over an fp8 pool runs its products in f16: a code becomes f16 in
  // one step (exact), the unit's query rows are converted once (times 2^-8),
  // P is written as f16 and v_scale is applied to the output.
  constexpr bool F16 = FMT != 0 && MODE == kDecode;
  constexpr uint32_t IDQK = F16 ? idesc_f16_f32(C::BM, C::BN, 0) : C::IDESC_QK;
  constexpr uint32_t IDPV = F16 ? idesc_f16_f32(C::BM, C::HDV, 1) : C::IDESC_PV;
  // K ring: decode over fp8 gives stage 0 to the raw-code ring
  constexpr int NK_ = F16 ? C::NK - 1 : C::NK;
  constexpr uint32_t K0 = C::OFF_K + (F16 ? C::K_BYTES : 0);
  // decode over fp8: warps 10-11 copy the codes, warps 12-13 convert the K
  // tiles and 14-15 the V tiles
  constexpr int RAW_THREADS = 64, CONV_THREADS = 64;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_unit[kUnitRing];

  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *k_full = bars + B_RING;
  uint64_t *k_empty = k_full + C::NK;
  uint64_t *v_full = k_empty + C::NK;
  uint64_t *v_empty = v_full + C::NV;
  uint64_t *i_full = v_empty + C::NV;
  uint64_t *i_empty = i_full + C::NI;
  uint64_t *raw_full = i_empty + C::NI;
  uint64_t *raw_empty = raw_full + C::NRAW;
  volatile int *abort_flag = &s_abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const bool kv_write = MODE == kTwoStage && p.cache_loc != nullptr;

  if (tid == 0) {
    mbar_init(&bars[B_Q_FULL], 1);
    mbar_init(&bars[B_Q_CONV], C::COPY_THREADS);  // decode over fp8: warps 12-15
    mbar_init(&bars[B_Q_EMPTY], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_S_FULL + i], 1);
      mbar_init(&bars[B_P_FULL + i], 4);  // one arrival per softmax warp
      mbar_init(&bars[B_O_DONE + i], 1);
    }
    mbar_init(&bars[B_FINAL], 1);
    mbar_init(&bars[B_NEVER], 1);
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(&bars[B_U_FULL + i], 1);
      // softmax, MMA and copy warps (+ the two writer warps with the fused
      // KV write)
      mbar_init(&bars[B_U_EMPTY + i],
                8 + 1 + C::COPY_THREADS / 32 + (kv_write || F16 ? 2 : 0));
    }
    // stages are filled by the copy warps, or by the converting warps in
    // decode over fp8
    for (int s = 0; s < C::NK; ++s) {
      mbar_init(&k_full[s], F16 ? CONV_THREADS : C::COPY_THREADS);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::NV; ++s) {
      mbar_init(&v_full[s], F16 ? CONV_THREADS : C::COPY_THREADS);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < C::NRAW; ++s) {
      mbar_init(&raw_full[s], RAW_THREADS);
      mbar_init(&raw_empty[s], CONV_THREADS);
    }
    for (int s = 0; s < C::NI; ++s) {
      mbar_init(&i_full[s], 32);
      mbar_init(&i_empty[s], (F16 ? RAW_THREADS : C::COPY_THREADS) / 32);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(&s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the prologue above reads no global memory; the work list, indices and
  // Q come from the kernels before this one on the stream
  grid_dep_wait();
  grid_dep_launch();  // the combine may be scheduled (it waits for this grid)
  const uint32_t tmem = s_tmem;
  const int n_units = p.hdr->n_units;
  const int G = p.group, TOK = p.tok;

  if (warp < 8) {
    regs_increase<C::REGS_SOFTMAX>();
    // ------------------------------------------- softmax + epilogue (x2)
    const int wg = warp >> 2;  // Q tile of this warpgroup
    const int wq = warp & 3;   // TMEM lane quarter
    const int r = tid & 127;   // tile row == TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t s_col = wg * C::BN;
    const uint32_t o_col = 2 * C::BN + wg * C::HDV;
    uint32_t s_cnt = 0, o_cnt = 0;
    bool ring_ok = true;
    // test hook: a wait that cannot succeed, so that the time limit runs out
    // and the abort path (flag, drain, TMEM release, return) runs
    if (p.stall && !mbar_wait(&bars[B_NEVER], 0, abort_flag, p.wait_ns))
      abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
    for (uint32_t uc = 0; !*abort_flag; ++uc) {
      const int u = ring_unit(&bars[B_U_FULL], &bars[B_U_EMPTY], s_unit, uc, abort_flag, true, ring_ok, p.wait_ns);
      if (u < 0) {
        if (!ring_ok) abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
        break;
      }
      const WorkUnit w = p.units[p.uorder[u]];
      // decode: warpgroup wg takes the unit's tiles wg, wg + 2, ... of the
      // one query tile (two key streams, merged by the combine)
      // Two key streams (decode units; split units of one query tile):
      // warpgroup wg takes the unit's tiles wg, wg + 2, ... of the one query
      // tile and writes its own partial, which the combine merges.
      const bool two = C::TWO_OK && (MODE == kDecode ? p.dec_two != 0 : (w.slot >= 0 && w.n_tok <= TOK));
      // this warpgroup's tiles: j0, j0 + jstep, ... below the unit's n_tiles
      const int j0 = two ? wg : 0, jstep = two ? 2 : 1;
      const int nt = w.n_tiles - j0;  // > 0 when the warpgroup has a tile
      const int tok0 = two ? 0 : wg * TOK;  // first token of this warpgroup's Q rows
      if (!two && wg == 1 && w.n_tok <= TOK) continue;
      const int n_tok_i = min(TOK, w.n_tok - tok0);
      const int rows_valid = n_tok_i * G;
      const bool valid = r < rows_valid;
      const bool warp_active = wq * 32 < rows_valid;
      const int t = tok0 + r / G, g = r - (r / G) * G;
      const int qpos = w.qpos0 + t;
      const int qmin = w.qpos0 + tok0, qmax = w.qpos0 + tok0 + n_tok_i - 1;
      const int64_t orow_idx = (int64_t)(w.q_tok0 + t) * p.hq + w.kvh * G + g;
      const int64_t prow_idx =
          MODE == kDecode ? (int64_t)(w.slot + wg) * p.rows_per_slot + r
                          : (int64_t)w.slot * p.rows_per_slot + wg * TOK * G + r;
      // custom mask rows: a byte per key of the sequence for each extend
      // token; mbase is the row of this Q tile's first token
      const uint8_t *mbase = nullptr;
      int64_t mstride = 0;
      if (MASK) {
        const int qo0 = p.qo_indptr[w.b];
        mstride = MODE == kTwoStage ? (int64_t)(p.kv_indptr[w.b + 1] - p.kv_indptr[w.b]) +
                                          (p.qo_indptr[w.b + 1] - qo0)
                                    : (int64_t)(p.kv_indptr[w.b + 1] - p.kv_indptr[w.b]);
        mbase = p.custom_mask + p.mask_indptr[w.b] + (int64_t)(w.q_tok0 + tok0 - qo0) * mstride;
      }
      if (nt <= 0) {
        if (valid) {
          if (w.slot < 0) {
            bf16 *orow = p.o + orow_idx * C::HDV;
            for (int c = 0; c < C::HDV; c += 8)
              *reinterpret_cast<uint4 *>(orow + c) = make_uint4(0, 0, 0, 0);
            if (p.lse) p.lse[orow_idx] = -INFINITY;
          } else {
            float *prow = p.po + prow_idx * C::HDV;
            for (int c = 0; c < C::HDV; c += 4)
              *reinterpret_cast<float4 *>(prow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            p.plse[prow_idx] = -INFINITY;
          }
        }
        continue;
      }
      float m = -INFINITY, l = 0.f;
      for (int j = j0; j < w.n_tiles; j += jstep) {
        int kb, ke;
        tile_keys(w, j, kb, ke);
        // Mask bits of this thread's row for keys kb + 32 q + bit (q < 4).
        // The G heads of a token share its mask row, so the warp walks its
        // rows' tokens: all lanes read 32 consecutive bytes of the token's
        // row (one sector per load), a ballot turns them into a word, and
        // the lanes of that token keep it.  Issued before the S wait.
        uint32_t mb[4] = {0u, 0u, 0u, 0u};
        if constexpr (MASK) {
          if (warp_active) {
            const int t_lo = (wq * 32) / G, t_hi = min((wq * 32 + 31) / G, n_tok_i - 1);
            const int my_t = r / G;
            // eight tokens at a time: all loads first, so their latencies overlap
            for (int tc = t_lo; tc <= t_hi; tc += 8) {
              uint8_t by[8][4];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const uint8_t *rowp = mbase + (int64_t)(tc + u) * mstride;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                  const int kpos = kb + 32 * q4 + lane;
                  by[u][q4] = (tc + u <= t_hi && kpos < ke) ? __ldg(rowp + kpos) : (uint8_t)0;
                }
              }
#pragma unroll
              for (int u = 0; u < 8; ++u) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                  const uint32_t word = __ballot_sync(0xffffffffu, by[u][q4] != 0);
                  if (my_t == tc + u) mb[q4] = word;
                }
              }
            }
          }
        }
        if (!mbar_wait(&bars[B_S_FULL + wg], s_cnt & 1u, abort_flag, p.wait_ns)) {
          abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
          break;
        }
        ++s_cnt;
        tc_fence_after();
        if (warp_active) {
          float x[C::BN];
          {
            uint32_t v0[32], v1[32], v2[32], v3[32];
            tmem_ld32(lane_base + s_col + 0, v0);
            tmem_ld32(lane_base + s_col + 32, v1);
            tmem_ld32(lane_base + s_col + 64, v2);
            tmem_ld32(lane_base + s_col + 96, v3);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              x[i] = __uint_as_float(v0[i]);
              x[32 + i] = __uint_as_float(v1[i]);
              x[64 + i] = __uint_as_float(v2[i]);
              x[96 + i] = __uint_as_float(v3[i]);
            }
          }
          // Logits in the log2 domain are sc * x.  The plain path keeps the
          // raw dot products and folds sc into the exponent's FMA; a capped
          // or masked tile is first mapped into the log2 domain (sc = 1).
          // A tile of an fp8 pool holds the codes: its logits take k_scale
          // in the scale, its P takes v_scale.
          const bool pool8 = FMT != 0 && !(MODE == kTwoStage && kb >= w.k_split);
          float sc = pool8 ? p.scale_log2_k * (F16 ? kQF16Up : 1.0f) : p.scale_log2;
          if (p.use_cap) {
            const float pre = pool8 ? p.cap_pre_k * (F16 ? kQF16Up : 1.0f) : p.cap_pre;
#pragma unroll
            for (int i = 0; i < C::BN; ++i) x[i] = p.cap_log2 * tanh_approx(x[i] * pre);
            sc = 1.0f;
          }
          const bool need_mask = MASK || (ke - 1 > qmin) || (ke - kb < C::BN) ||
                                 (p.window > 0 && kb < qmax - p.window);
          if constexpr (MASK) {
            // the custom mask replaces the causal term; the window stays.
            // A row that sees every key of the tile (all bits set, the
            // window does not cut) keeps the plain path.
            const bool every = (mb[0] & mb[1] & mb[2] & mb[3]) == 0xffffffffu &&
                               (p.window <= 0 || qpos - kb <= p.window);
            if (!every) {
#pragma unroll
              for (int i = 0; i < C::BN; ++i) {
                const int kpos = kb + i;
                const bool vis = ((mb[i >> 5] >> (i & 31)) & 1u) &&
                                 (p.window <= 0 || qpos - kpos <= p.window);
                x[i] = vis ? x[i] * sc : -INFINITY;
              }
              sc = 1.0f;
            }
          } else if (need_mask) {
#pragma unroll
            for (int i = 0; i < C::BN; ++i) {
              const int kpos = kb + i;
              const bool vis =
                  kpos < ke && kpos <= qpos && (p.window <= 0 || qpos - kpos <= p.window);
              x[i] = vis ? x[i] * sc : -INFINITY;
            }
            sc = 1.0f;
          }
          // row max of sc * x: sc * max(x), or sc * min(x) for a negative sc
          float mt;
          if (sc >= 0.f) {
            float mt0 = x[0], mt1 = x[1], mt2 = x[2], mt3 = x[3];
#pragma unroll
            for (int i = 4; i < C::BN; i += 4) {
              mt0 = fmaxf(mt0, x[i]);
              mt1 = fmaxf(mt1, x[i + 1]);
              mt2 = fmaxf(mt2, x[i + 2]);
              mt3 = fmaxf(mt3, x[i + 3]);
            }
            mt = fmaxf(fmaxf(mt0, mt1), fmaxf(mt2, mt3)) * sc;
          } else {
            float mt0 = x[0], mt1 = x[1], mt2 = x[2], mt3 = x[3];
#pragma unroll
            for (int i = 4; i < C::BN; i += 4) {
              mt0 = fminf(mt0, x[i]);
              mt1 = fminf(mt1, x[i + 1]);
              mt2 = fminf(mt2, x[i + 2]);
              mt3 = fminf(mt3, x[i + 3]);
            }
            mt = fminf(fminf(mt0, mt1), fminf(mt2, mt3)) * sc;
          }
          const float m_new = fmaxf(m, mt);
          // Rescale only when the max grows by more than 2^8: exponents of
          // the stale max stay below 256, which fp32 sums and bf16 P hold.
          // (S_full of this tile completes after the previous PV, so O is
          // quiescent here.)
          const bool grow = m_new > m + 8.0f;
          const float alpha = grow ? ex2_approx(m - m_new) : 1.0f;
          const bool o_needs = grow && j > j0 && l > 0.f;
          if (grow) {
            l *= alpha;
            m = m_new;
          }
          const float mref = m == -INFINITY ? 0.f : m;
          // p = 2^(sc * x - m): one FMA into each exp2
          float nm = -mref;
          float lscale = 1.0f;
          if constexpr (FMT != 0 && !F16) {
            if (pool8) {
              nm += p.log2_v_scale;
              lscale = p.inv_v_scale;
            }
          }
          float l0 = 0.f, l1 = 0.f;
          uint32_t pk[C::BN / 2];
#pragma unroll
          for (int i = 0; i < C::BN; i += 2) {
            const float e0 = ex2_approx(fmaf(x[i], sc, nm));
            const float e1 = ex2_approx(fmaf(x[i + 1], sc, nm));
            l0 += e0;
            l1 += e1;
            if constexpr (F16) {
              const __half2 h = __floats2half2_rn(e0, e1);
              pk[i / 2] = *reinterpret_cast<const uint32_t *>(&h);
            } else {
              pk[i / 2] = pack_bf16(e0, e1);
            }
          }
          if constexpr (FMT != 0) l += (l0 + l1) * lscale;
          else l += l0 + l1;
          // P (bf16 pairs) over the first 64 columns of this tile's S.
          {
            uint32_t a[32], b[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              a[i] = pk[i];
              b[i] = pk[32 + i];
            }
            tmem_st32(lane_base + s_col + 0, a);
            tmem_st32(lane_base + s_col + 32, b);
          }
          if (__any_sync(0xffffffffu, o_needs)) {
            const float a = o_needs ? alpha : 1.0f;
            uint32_t v[32];
#pragma unroll
            for (int c = 0; c < C::HDV / 32; ++c) {
              const uint32_t ta = lane_base + o_col + c * 32;
              tmem_ld32(ta, v);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * a);
              tmem_st32(ta, v);
            }
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_P_FULL + wg]);
      }
      if (*abort_flag) break;
      // epilogue: wait for the last PV of this tile, normalise, store
      if (!mbar_wait(&bars[B_O_DONE + wg], o_cnt & 1u, abort_flag, p.wait_ns)) {
        abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
        break;
      }
      ++o_cnt;
      tc_fence_after();
      if (warp_active) {
        float inv = l > 0.f ? 1.0f / l : 0.f;
        float lse_v = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        if (p.sinks && w.slot < 0) {
          // the head's sink joins the denominator (a split row gets it in
          // the combine): with M = max(m, sink), l' = l 2^(m-M) + 2^(sink-M)
          const float s2 = __ldg(p.sinks + w.kvh * G + g) * 1.4426950408889634f;
          const float M = fmaxf(m, s2);
          const float a_m = m == -INFINITY ? 0.f : ex2_approx(m - M);
          const float lt = l * a_m + ex2_approx(s2 - M);
          inv = a_m / lt;
          lse_v = (M + __log2f(lt)) * 0.69314718055994531f;
        }
        if constexpr (F16) inv *= p.v_scale;  // V was read as its codes
        uint32_t v[32];
#pragma unroll
        for (int c = 0; c < C::HDV / 32; ++c) {
          tmem_ld32(lane_base + o_col + c * 32, v);
          tmem_wait_ld();
          if (valid) {
            if (w.slot < 0) {
              bf16 *orow = p.o + orow_idx * C::HDV + c * 32;
#pragma unroll
              for (int i = 0; i < 32; i += 8) {
                uint4 q4;
                q4.x = pack_bf16(__uint_as_float(v[i + 0]) * inv, __uint_as_float(v[i + 1]) * inv);
                q4.y = pack_bf16(__uint_as_float(v[i + 2]) * inv, __uint_as_float(v[i + 3]) * inv);
                q4.z = pack_bf16(__uint_as_float(v[i + 4]) * inv, __uint_as_float(v[i + 5]) * inv);
                q4.w = pack_bf16(__uint_as_float(v[i + 6]) * inv, __uint_as_float(v[i + 7]) * inv);
                *reinterpret_cast<uint4 *>(orow + i) = q4;
              }
            } else {
              float *prow = p.po + prow_idx * C::HDV + c * 32;
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
            p.plse[prow_idx] = lse_v;
          }
        }
      }
      tc_fence_before();
    }
  } else {
  regs_decrease<C::REGS_OTHER>();
  if (warp == 8) {
    // ------------------------------------------------ MMA issue (one warp)
    // All 32 lanes run the loop (and its waits), so the descriptors and
    // counters stay warp-uniform; one elected lane issues each tcgen05
    // operation.  The same loop run by lane 0 alone issued about 25 %
    // slower.
    {
      const bool leader = elect_one();
      uint32_t q_cnt = 0, kc = 0, vc = 0, p_cnt0 = 0, p_cnt1 = 0;
      const uint32_t sQ0 = sbase + C::OFF_Q, sQ1 = sQ0 + C::Q_BYTES;
      bool ok = true;
      // Descriptors are built once per tile and stepped by constants: the
      // issue path is a single thread, and a per-MMA dependent chain of
      // address arithmetic starves the tensor pipe.
      constexpr uint32_t K_LO = sw128_desc_lo(0), K_HI = sw128_desc_hi(1024);
      constexpr uint32_t V_LO = sw128_desc_lo(C::BN * 128), V_HI = sw128_desc_hi(1024);
      auto issue_s = [&](int qt, uint32_t sK) {
        const uint32_t a_lo = K_LO | desc_addr(qt ? sQ1 : sQ0), b_lo = K_LO | desc_addr(sK);
        const uint32_t d = tmem + qt * C::BN;
        static_for<0, C::LQ / 16>([&](auto kk_c) {
          constexpr int kk = decltype(kk_c)::value;
          constexpr uint32_t ao = ((kk / 4) * (C::BM * 128) + (kk % 4) * 32) / 16;
          constexpr uint32_t bo = ((kk / 4) * (C::BN * 128) + (kk % 4) * 32) / 16;
          if (leader) tc_mma_ss_step<ao, bo>(d, a_lo, b_lo, K_HI, IDQK, kk > 0 ? 1u : 0u);
        });
        if (leader) tc_commit(&bars[B_S_FULL + qt]);
      };
      // S of query tile 0 into S/P buffer `buf` (the decode streams)
      auto issue_s_q0 = [&](int buf, uint32_t sK) {
        const uint32_t a_lo = K_LO | desc_addr(sQ0), b_lo = K_LO | desc_addr(sK);
        const uint32_t d = tmem + buf * C::BN;
        static_for<0, C::LQ / 16>([&](auto kk_c) {
          constexpr int kk = decltype(kk_c)::value;
          constexpr uint32_t ao = ((kk / 4) * (C::BM * 128) + (kk % 4) * 32) / 16;
          constexpr uint32_t bo = ((kk / 4) * (C::BN * 128) + (kk % 4) * 32) / 16;
          if (leader) tc_mma_ss_step<ao, bo>(d, a_lo, b_lo, K_HI, IDQK, kk > 0 ? 1u : 0u);
        });
        if (leader) tc_commit(&bars[B_S_FULL + buf]);
      };
      auto issue_pv = [&](int qt, uint32_t sV, bool acc_first) {
        const uint32_t b_lo = V_LO | desc_addr(sV);
        const uint32_t d = tmem + 2 * C::BN + qt * C::HDV, a = tmem + qt * C::BN;
        const uint32_t acc0 = acc_first ? 1u : 0u;
        static_for<0, C::BN / 16>([&](auto kk_c) {
          constexpr int kk = decltype(kk_c)::value;
          if (leader) tc_mma_ts_step<kk * 8, kk * 128>(d, a, b_lo, V_HI, IDPV, kk > 0 ? 1u : acc0);
        });
      };
      for (uint32_t uc = 0; ok && !*abort_flag; ++uc) {
        const int u = ring_unit(&bars[B_U_FULL], &bars[B_U_EMPTY], s_unit, uc, abort_flag, true, ok, p.wait_ns);
        if (u < 0) break;
        const WorkUnit w = p.units[p.uorder[u]];
        const int nt = w.n_tiles;
        if (nt == 0) continue;
        const bool q1 = w.n_tok > TOK;
        if (!mbar_wait(&bars[F16 ? B_Q_CONV : B_Q_FULL], q_cnt & 1u, abort_flag, p.wait_ns)) {
          ok = false;
          break;
        }
        ++q_cnt;
        tc_fence_after();
        if (C::TWO_OK && (MODE == kDecode ? p.dec_two != 0 : (w.slot >= 0 && !q1))) {
          // Two key streams over the one query tile: even tiles into S/P
          // buffer 0 (softmax warpgroup 0, O 0), odd tiles into buffer 1
          // (warpgroup 1, O 1).  S(j) waits only for PV(j-2), which reads
          // the P it overwrites, so one stream's softmax runs while the
          // other's products do.
          for (int j = 0; j < nt && ok; ++j) {
            const int b = j & 1;
            if (j >= 2) {
              const int vs = vc % C::NV;
              uint32_t &pc = b ? p_cnt1 : p_cnt0;
              if (!mbar_wait(&v_full[vs], (vc / C::NV) & 1u, abort_flag, p.wait_ns) ||
                  !mbar_wait(&bars[B_P_FULL + b], pc & 1u, abort_flag, p.wait_ns)) {
                ok = false;
                break;
              }
              ++pc;
              fence_proxy_async_smem();
              tc_fence_after();
              issue_pv(b, sbase + C::OFF_V + vs * C::V_BYTES, j >= 4);
              if (leader) tc_commit(&v_empty[vs]);
              ++vc;
            }
            const int ks = kc % NK_;
            if (!mbar_wait(&k_full[ks], (kc / NK_) & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
            fence_proxy_async_smem();
            tc_fence_after();
            issue_s_q0(b, sbase + K0 + ks * C::K_BYTES);
            if (leader) tc_commit(&k_empty[ks]);
            ++kc;
            if (j == nt - 1 && leader) tc_commit(&bars[B_Q_EMPTY]);
          }
          // the last PV of each stream, in tile order
          for (int j = nt >= 2 ? nt - 2 : 0; j < nt && ok; ++j) {
            const int b = j & 1;
            const int vs = vc % C::NV;
            uint32_t &pc = b ? p_cnt1 : p_cnt0;
            if (!mbar_wait(&v_full[vs], (vc / C::NV) & 1u, abort_flag, p.wait_ns) ||
                !mbar_wait(&bars[B_P_FULL + b], pc & 1u, abort_flag, p.wait_ns)) {
              ok = false;
              break;
            }
            ++pc;
            fence_proxy_async_smem();
            tc_fence_after();
            issue_pv(b, sbase + C::OFF_V + vs * C::V_BYTES, j >= 2);
            if (leader) tc_commit(&bars[B_O_DONE + b]);
            if (leader) tc_commit(&v_empty[vs]);
            ++vc;
          }
          continue;
        }
        // tile 0: S of both Q tiles
        {
          const int ks = kc % NK_;
          if (!mbar_wait(&k_full[ks], (kc / NK_) & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
          fence_proxy_async_smem();  // cp.async (generic proxy) -> tcgen05.mma reads
          tc_fence_after();
          const uint32_t sK = sbase + K0 + ks * C::K_BYTES;
          issue_s(0, sK);
          if (q1) issue_s(1, sK);
          if (leader) tc_commit(&k_empty[ks]);
          ++kc;
          if (nt == 1 && leader) tc_commit(&bars[B_Q_EMPTY]);
        }
        for (int j = 1; j < nt && ok; ++j) {
          const int ks = kc % NK_, vs = vc % C::NV;
          if (!mbar_wait(&k_full[ks], (kc / NK_) & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
          if (!mbar_wait(&v_full[vs], (vc / C::NV) & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
          if (!mbar_wait(&bars[B_P_FULL + 0], p_cnt0 & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
          ++p_cnt0;
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t sK = sbase + K0 + ks * C::K_BYTES;
          const uint32_t sV = sbase + C::OFF_V + vs * C::V_BYTES;
          issue_pv(0, sV, j > 1);
          issue_s(0, sK);
          if (q1) {
            if (!mbar_wait(&bars[B_P_FULL + 1], p_cnt1 & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
            ++p_cnt1;
            tc_fence_after();
            issue_pv(1, sV, j > 1);
            issue_s(1, sK);
          }
          if (leader) tc_commit(&v_empty[vs]);
          ++vc;
          if (leader) tc_commit(&k_empty[ks]);
          ++kc;
          if (j == nt - 1 && leader) tc_commit(&bars[B_Q_EMPTY]);
        }
        if (!ok) break;
        // last PV of both Q tiles
        {
          const int vs = vc % C::NV;
          if (!mbar_wait(&v_full[vs], (vc / C::NV) & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
          if (!mbar_wait(&bars[B_P_FULL + 0], p_cnt0 & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
          ++p_cnt0;
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t sV = sbase + C::OFF_V + vs * C::V_BYTES;
          issue_pv(0, sV, nt > 1);
          if (leader) tc_commit(&bars[B_O_DONE + 0]);
          if (q1) {
            if (!mbar_wait(&bars[B_P_FULL + 1], p_cnt1 & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
            ++p_cnt1;
            tc_fence_after();
            issue_pv(1, sV, nt > 1);
            if (leader) tc_commit(&bars[B_O_DONE + 1]);
          }
          if (leader) tc_commit(&v_empty[vs]);
          ++vc;
        }
      }
      if (!ok) abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
      // drain: every MMA issued above must finish before TMEM is freed
      if (leader) tc_commit(&bars[B_FINAL]);
      if (!mbar_wait_drain(&bars[B_FINAL], 0)) record_status(p.status, PKX_ETIMEOUT);
    }
  } else if (warp == 9) {
    // --------------------------------------- Q tiles and row indices
    // Lane 0 loads each unit's Q tiles (3-D TMA box: 64 dims, G heads,
    // q_box_tok tokens; rows t * G + g).  Every lane resolves 4 keys of each
    // tile to a pool slot (or extend row) into the index ring, ahead of the
    // copy warps; -1 marks a key to zero-fill (past the tile's end, or an
    // out-of-range slot, which is also recorded).
    uint32_t q_cnt = 0, ic = 0;
    if (lane == 0) prefetch_tensormap(&tm.q);
    const uint32_t q_box_bytes = 64u * 2u * G * p.q_box_tok;
    bool ok = true;
    for (uint32_t uc = 0; ok && !*abort_flag; ++uc) {
      // claim the next unit and hand it to the other warps
      int u = -1;
      if (lane == 0) {
        if (p.part_first) {  // stream partition: this CTA's share, in order
          const int pos = p.part_first[blockIdx.x] + (int)uc;
          u = pos < p.part_first[blockIdx.x + 1] ? pos : -1;
        } else {
          const int pos = atomicAdd(p.next_unit, 1);
          u = pos < n_units ? pos : -1;
        }
      }
      u = __shfl_sync(0xffffffffu, u, 0);
      {
        const int slot = uc % kUnitRing;
        if (uc >= (uint32_t)kUnitRing &&
            !mbar_wait(&bars[B_U_EMPTY + slot], ((uc / kUnitRing) - 1) & 1u, abort_flag, p.wait_ns)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          s_unit[slot] = u;
          mbar_arrive(&bars[B_U_FULL + slot]);
        }
      }
      if (u < 0) break;
      const WorkUnit w = p.units[p.uorder[u]];
      const int nt = w.n_tiles;
      if (nt == 0) continue;
      const bool q1 = w.n_tok > TOK;
      if (lane == 0) {
        if (q_cnt > 0 && !mbar_wait(&bars[B_Q_EMPTY], (q_cnt - 1) & 1u, abort_flag, p.wait_ns)) ok = false;
        if (ok) {
          const int nq = q1 ? 2 : 1;
          mbar_arrive_expect_tx(&bars[B_Q_FULL], q_box_bytes * C::QA * nq);
          for (int qt = 0; qt < nq; ++qt)
            for (int h = 0; h < C::QA; ++h)
              tma_load_3d(sbase + C::OFF_Q + qt * C::Q_BYTES + h * (C::BM * 128), &tm.q, h * 64,
                          w.kvh * G, w.q_tok0 + qt * TOK, &bars[B_Q_FULL]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ++q_cnt;
      const int64_t kv_base = p.kv_indptr[w.b];
      const int64_t ext_base = MODE == kTwoStage ? p.qo_indptr[w.b] : 0;
      for (int j = 0; j < nt; ++j) {
        int kb, ke;
        tile_keys(w, j, kb, ke);
        const bool from_ext = MODE == kTwoStage && kb >= w.k_split;
        int rows[4];
        bool bad = false;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int jpos = kb + 4 * lane + i;
          int64_t row = -1;
          if (jpos < ke) {
            if (from_ext) {
              row = ext_base + (jpos - w.k_split);
            } else {
              row = MODE == kUnified
                        ? __ldg(static_cast<const int64_t *>(p.kv_indices) + kv_base + jpos)
                        : (int64_t)__ldg(static_cast<const int32_t *>(p.kv_indices) + kv_base + jpos);
              if (row < 0 || row >= p.num_slots) {
                bad = true;
                row = -1;
              }
            }
          }
          rows[i] = (int)row;
        }
        if (bad) record_status(p.status, PKX_EDEVICE);
        const int is = ic % C::NI;
        if (ic >= (uint32_t)C::NI &&
            !mbar_wait(&i_empty[is], ((ic / C::NI) - 1) & 1u, abort_flag, p.wait_ns)) {
          ok = false;
          break;
        }
        {
          // ring[key % KPP][key / KPP]: each copy thread's rows contiguous
          constexpr int KPP = C::KPP, NK_T = C::BN / KPP;
          int *ring = reinterpret_cast<int *>(smem + C::OFF_I + is * C::I_BYTES);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int key = 4 * lane + i;
            ring[(key % KPP) * NK_T + key / KPP] = rows[i];
          }
        }
        mbar_arrive(&i_full[is]);
        ++ic;
      }
    }
    if (!ok) abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
    // the last Q load this warp issued lands before the CTA may exit (after
    // an abort nobody else may have waited for it)
    if (lane == 0 && q_cnt > 0 && !mbar_wait_drain(&bars[B_Q_FULL], (q_cnt - 1) & 1u))
      record_status(p.status, PKX_ETIMEOUT);
    __syncwarp();
  } else if (F16 && warp >= 12) {
    // ------------------------------- fp8 codes -> f16 stages (warps 12-15)
    // Decode over an fp8 pool: each raw slot (K(j) and V(j) alternate, in
    // the order the copying warps issue them) is converted into the next
    // stage of its ring once its codes have landed and the stage is free;
    // warps 12-13 take the K slots and 14-15 the V slots, so that neither
    // ring waits behind the other.  Chunk c of a slot holds the eight codes
    // of key c / CPR, dims 8 (c % CPR) + [0, 8); thread cv of a group
    // converts chunks cv + 64 m, so a warp reads 256 contiguous bytes and
    // writes whole 128-byte rows of the swizzled stage.  Its chunk index
    // (c % CPR) and the key's swizzle phase are the same for every m, so
    // source and destination step by constants.  All four warps convert
    // each unit's query rows to f16 (Q_CONV).
    if constexpr (F16) {
    constexpr int CPR = HD / 8;
    constexpr int NCH = C::BN * CPR / CONV_THREADS;
    constexpr int KSTEP = CONV_THREADS / CPR;  // keys between a thread's chunks
    // swizzle phases (key % 8) a thread's keys cycle through
    constexpr int NPH = KSTEP % 8 == 0 ? 1 : 8 / KSTEP;
    static_assert(C::BN * CPR % CONV_THREADS == 0 && NCH % NPH == 0 &&
                      (KSTEP % 8 == 0 || 8 % KSTEP == 0),
                  "conversion geometry");
    const int grp = warp >= 14;                // 0: K slots, 1: V slots
    const int cq = tid - 12 * 32;              // 0 .. 127 for the query rows
    const int cv = cq - grp * CONV_THREADS;    // 0 .. 63 within the group
    const int ck = cv % CPR, key0 = cv / CPR;
    const uint32_t sthr = (uint32_t)cv * 8u;
    uint32_t dthr[NPH];  // chunk m = NPH mm + ph: key key0 + KSTEP m
#pragma unroll
    for (int ph = 0; ph < NPH; ++ph) {
      const int key = key0 + KSTEP * ph;
      dthr[ph] = (uint32_t)(ck >> 3) * (C::BN * 128) + (uint32_t)key * 128u +
                 ((uint32_t)((ck & 7) ^ (key & 7)) << 4);
    }
    uint32_t rc = grp, kc = 0, vc = 0, qc = 0;  // rc: slot use (K even, V odd)
    bool ok = true;
    // the group's next slot into `stage` once both are ready
    auto convert_slot = [&](uint64_t *st_empty, uint32_t n_used, int n_stages, uint32_t stage,
                            uint64_t *st_full) -> bool {
      const int s = rc % C::NRAW;
      if (!mbar_wait(&raw_full[s], (rc / C::NRAW) & 1u, abort_flag, p.wait_ns)) return false;
      if (n_used >= (uint32_t)n_stages &&
          !mbar_wait(st_empty, ((n_used / n_stages) - 1) & 1u, abort_flag, p.wait_ns))
        return false;
      const uint32_t src = sbase + C::OFF_RAW + s * C::RAW_BYTES + sthr;
#pragma unroll 2
      for (int mm = 0; mm < NCH / NPH; ++mm) {
#pragma unroll
        for (int ph = 0; ph < NPH; ++ph)
          st_shared_u4(stage + dthr[ph] + mm * (KSTEP * NPH * 128),
                       fp8x8_to_f16x8<FMT>(
                           ld_shared_u2(src + (mm * NPH + ph) * (CONV_THREADS * 8))));
      }
      fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
      mbar_arrive(st_full);
      mbar_arrive(&raw_empty[s]);
      rc += 2;
      return true;
    };
    for (uint32_t uc = 0; ok && !*abort_flag; ++uc) {
      const int u = ring_unit(&bars[B_U_FULL], &bars[B_U_EMPTY], s_unit, uc, abort_flag, true, ok, p.wait_ns);
      if (u < 0) break;
      const WorkUnit w = p.units[p.uorder[u]];
      const int nt = w.n_tiles;
      if (nt == 0) continue;
      // the unit's query rows (tokens x G heads of query tile 0) to f16 in
      // place once their load has landed, 16 bytes at a time (the swizzle
      // only permutes whole chunks within a row)
      if (!mbar_wait(&bars[B_Q_FULL], qc & 1u, abort_flag, p.wait_ns)) {
        ok = false;
        break;
      }
      ++qc;
      const int n_chunks = w.n_tok * G * (HD / 8);
      for (int c = cq; c < n_chunks; c += 2 * CONV_THREADS) {
        const int row = c / (HD / 8), k = c % (HD / 8);
        const uint32_t off = C::OFF_Q + (uint32_t)(k >> 3) * (C::BM * 128) + (uint32_t)row * 128u +
                             (uint32_t)(k & 7) * 16u;
        const uint4 v = *reinterpret_cast<const uint4 *>(smem + off);
        st_shared_u4(sbase + off, bf16x8_to_f16x8_scaled(v));
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[B_Q_CONV]);
      for (int j = 0; j < nt; ++j) {
        const int ks = kc % NK_, vs = vc % C::NV;
        if (grp == 0 ? !convert_slot(&k_empty[ks], kc, NK_, sbase + K0 + ks * C::K_BYTES, &k_full[ks])
                     : !convert_slot(&v_empty[vs], vc, C::NV, sbase + C::OFF_V + vs * C::V_BYTES,
                                     &v_full[vs])) {
          ok = false;
          break;
        }
        if (grp == 0) ++kc;
        else ++vc;
      }
    }
    if (!ok) abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
    }
  } else if (F16) {
    // ------------------------------------ fp8 codes into raw slots (warps 10-11)
    // Decode over an fp8 pool: the codes of each K and V tile go
    // fire-and-forget into the next slot of the raw ring (row-major, 8 bytes
    // per (key, chunk)) once the converting warps have read what it held;
    // each thread arrives (noinc) on the slot's barrier when its own copies
    // land.  Thread ct copies chunk ct % CPR of keys ct / CPR + KG i.
    if constexpr (F16) {
    constexpr int CPR = HD / 8, KG = RAW_THREADS / CPR, NKEYS = C::BN / KG;
    constexpr int KPP = C::KPP, NK_T = C::BN / KPP;  // the index ring's layout
    static_assert(KG * CPR == RAW_THREADS && C::BN % KG == 0, "copy geometry");
    const int ct = tid - C::COPY_WARP0 * 32;
    const int ch = ct % CPR, kg = ct / CPR;
    const uint32_t rthr = (uint32_t)(kg * CPR + ch) * 8u;
    uint32_t rc = 0, ic = 0;
    bool ok = true;
    for (uint32_t uc = 0; ok && !*abort_flag; ++uc) {
      const int u = ring_unit(&bars[B_U_FULL], &bars[B_U_EMPTY], s_unit, uc, abort_flag, true, ok, p.wait_ns);
      if (u < 0) break;
      const WorkUnit w = p.units[p.uorder[u]];
      const int nt = w.n_tiles;
      if (nt == 0) continue;
      const uint8_t *kp8 =
          reinterpret_cast<const uint8_t *>(p.k_pool) + (int64_t)w.kvh * p.kb_sh + ch * 8;
      const uint8_t *vp8 =
          reinterpret_cast<const uint8_t *>(p.v_pool) + (int64_t)w.kvh * p.vb_sh + ch * 8;
      for (int j = 0; j < nt && ok; ++j) {
        // this thread's rows (the index ring holds key's row at
        // [key % KPP][key / KPP])
        const int is = ic % C::NI;
        if (!mbar_wait(&i_full[is], (ic / C::NI) & 1u, abort_flag, p.wait_ns)) {
          ok = false;
          break;
        }
        int rows[NKEYS];
        {
          const int *ring = reinterpret_cast<const int *>(smem + C::OFF_I + is * C::I_BYTES);
#pragma unroll
          for (int i = 0; i < NKEYS; ++i) {
            const int key = kg + KG * i;
            rows[i] = ring[(key % KPP) * NK_T + key / KPP];
          }
        }
        __syncwarp();  // the warp is done with the ring slot
        if (lane == 0) mbar_arrive(&i_empty[is]);
        ++ic;
        for (int t = 0; t < 2; ++t) {  // K(j), then V(j)
          const int s = rc % C::NRAW;
          if (rc >= (uint32_t)C::NRAW &&
              !mbar_wait(&raw_empty[s], ((rc / C::NRAW) - 1) & 1u, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          const uint8_t *base = t == 0 ? kp8 : vp8;
          const int64_t stride = t == 0 ? p.kb_ss : p.vb_ss;
          const uint32_t slot = sbase + C::OFF_RAW + s * C::RAW_BYTES + rthr;
          static_for<0, NKEYS>([&](auto i_c) {
            constexpr int i = decltype(i_c)::value;
            const int r = rows[i];
            const uint8_t *src = base + (int64_t)max(r, 0) * stride;
            cp_async_8_at<i * KG * CPR * 8>(slot, src, r >= 0 ? 8u : 0u);
          });
          cp_async_arrive_noinc(&raw_full[s]);
          ++rc;
        }
      }
    }
    if (!ok) abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
    cp_async_wait_all();
    }
  } else if (warp < C::COPY_WARP0 + C::COPY_THREADS / 32) {
    // ------------------------------------------------ K/V copies (4 warps)
    // Thread ct copies 16-byte chunk ch = ct % CPR of keys key0 + KPP * i
    // (key0 = ct / CPR): every copy instruction of a warp reads whole rows.
    // KPP is a multiple of 8, so the swizzle term (ch ^ key % 8) is fixed
    // per thread and key i lands at a constant offset from the thread's
    // destination base.  The index warp stores each thread's rows
    // contiguously (ring[key0][i]).  A thread arrives (noinc) on the stage
    // barrier when its own copies have landed.
    // Split head dims: thread ct copies chunk ct % 8 of every 64-dim atom of
    // keys ct / 8 + 16 i (KPP = 16), so the swizzle term is again fixed per
    // thread; a warp instruction reads four rows' 128-byte segments.
    const int ct = tid - C::COPY_WARP0 * 32;
    constexpr int CPR = C::SPLIT ? 8 : C::LQ / 8;  // chunk lanes of a key
    constexpr int KPP = C::KPP;                    // keys per pass
    constexpr int NKEYS = C::BN / KPP;             // keys per thread
    static_assert(KPP * CPR == C::COPY_THREADS, "copy geometry");
    static_assert(KPP % 8 == 0 && C::BN % KPP == 0, "constant swizzle per thread");
    const int ch = ct % CPR, key0 = ct / CPR;
    const uint32_t dthr = (uint32_t)(ch >> 3) * (C::BN * 128) + (uint32_t)key0 * 128u +
                          ((uint32_t)((ch & 7) ^ (key0 & 7)) << 4);
    // the thread's chunks of its NKEYS rows (of L elements) into a stage
    auto copy_rows = [&](uint32_t stage, const bf16 *base, int64_t stride, const int *rows,
                         auto l_c) {
      constexpr int L = decltype(l_c)::value;
      static_for<0, NKEYS>([&](auto i_c) {
        constexpr int i = decltype(i_c)::value;
        const int r = rows[i];
        const uint32_t bytes = r >= 0 ? 16u : 0u;
        const bf16 *src = base + (int64_t)max(r, 0) * stride;
        if constexpr (!C::SPLIT) {
          static_assert(L == C::LQ || L == C::HDV, "row length");
          cp_async_16_at<i * KPP * 128, 0>(stage + dthr, src, bytes);
        } else {
          static_for<0, (L + 63) / 64>([&](auto a_c) {
            constexpr int a = decltype(a_c)::value;
            if (a * 8 + ch < L / 8)  // the last atom of a 288-dim row holds 4 chunks
              cp_async_16_at<a * C::BN * 128 + i * KPP * 128, a * 128>(stage + dthr, src, bytes);
          });
        }
      });
    };
    constexpr std::integral_constant<int, C::LQ> K_LEN{};
    constexpr std::integral_constant<int, C::HDV> V_LEN{};
    uint32_t kc = 0, vc = 0, ic = 0;
    [[maybe_unused]] uint32_t qc = 0;
    bool ok = true;
    if constexpr (FMT == 0) {
      for (uint32_t uc = 0; ok && !*abort_flag; ++uc) {
        const int u = ring_unit(&bars[B_U_FULL], &bars[B_U_EMPTY], s_unit, uc, abort_flag, true, ok, p.wait_ns);
        if (u < 0) break;
        const WorkUnit w = p.units[p.uorder[u]];
        const int nt = w.n_tiles;
        if (nt == 0) continue;
        const bf16 *kp = p.k_pool + (int64_t)w.kvh * p.kb_sh + ch * 8;
        const bf16 *vp = p.v_pool + (int64_t)w.kvh * p.vb_sh + ch * 8;
        const bf16 *kx = p.k_ext + (int64_t)w.kvh * p.ke_sh + ch * 8;
        const bf16 *vx = p.v_ext + (int64_t)w.kvh * p.ve_sh + ch * 8;
        for (int j = 0; j < nt; ++j) {
          int kb, ke;
          tile_keys(w, j, kb, ke);
          const bool from_ext = MODE == kTwoStage && kb >= w.k_split;
          // this thread's rows from the index ring
          const int is = ic % C::NI;
          if (!mbar_wait(&i_full[is], (ic / C::NI) & 1u, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          int rows[NKEYS];
          {
            const int4 *ring =
                reinterpret_cast<const int4 *>(smem + C::OFF_I + is * C::I_BYTES) + key0 * (NKEYS / 4);
  #pragma unroll
            for (int q = 0; q < NKEYS / 4; ++q) {
              const int4 v = ring[q];
              rows[4 * q] = v.x;
              rows[4 * q + 1] = v.y;
              rows[4 * q + 2] = v.z;
              rows[4 * q + 3] = v.w;
            }
          }
          __syncwarp();  // the warp is done with the ring slot
          if (lane == 0) mbar_arrive(&i_empty[is]);
          ++ic;
          // K tile
          const int ks = kc % NK_;
          if (kc >= (uint32_t)NK_ &&
              !mbar_wait(&k_empty[ks], ((kc / NK_) - 1) & 1u, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          copy_rows(sbase + K0 + ks * C::K_BYTES, from_ext ? kx : kp,
                    from_ext ? p.ke_st : p.kb_ss, rows, K_LEN);
          cp_async_arrive_noinc(&k_full[ks]);
          ++kc;
          // V tile
          const int vs = vc % C::NV;
          if (vc >= (uint32_t)C::NV &&
              !mbar_wait(&v_empty[vs], ((vc / C::NV) - 1) & 1u, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          copy_rows(sbase + C::OFF_V + vs * C::V_BYTES, from_ext ? vx : vp,
                    from_ext ? p.ve_st : p.vb_ss, rows, V_LEN);
          cp_async_arrive_noinc(&v_full[vs]);
          ++vc;
        }
      }
    } else {
    // extend over an fp8 pool.  A pool tile's codes are copied 8 bytes per (thread, key)
    // into the first half of the 16-byte chunk the same thread later
    // writes, and converted there in place to bf16 once they have landed, so no thread overwrites another's codes.  The copies
    // of tile j+1 go out before tile j is converted, in the order
    // K(j+1), convert K(j), V(j+1), convert V(j): V(j+1) reuses the stage of
    // V(j-1), which the tensor core frees only after K(j) is full.  Extend
    // tiles (bf16 rows of the two-stage form) take the plain copy.  One
    // cp.async group is committed per issued tile.
    // (split head dims: by 64-dim atom, as copy_rows does; a row of L codes)
    auto issue_raw = [&](uint32_t stage, const uint8_t *base, int64_t stride, const int *rows,
                         auto l_c) {
      constexpr int L = decltype(l_c)::value;
      static_for<0, NKEYS>([&](auto i_c) {
        constexpr int i = decltype(i_c)::value;
        const int r = rows[i];
        const uint8_t *src = base + (int64_t)max(r, 0) * stride;
        if constexpr (!C::SPLIT) {
          static_assert(L == C::LQ || L == C::HDV, "row length");
          cp_async_8_at<i * KPP * 128>(stage + dthr, src, r >= 0 ? 8u : 0u);
        } else {
          static_for<0, (L + 63) / 64>([&](auto a_c) {
            constexpr int a = decltype(a_c)::value;
            if (a * 8 + ch < L / 8)
              cp_async_8_at<a * C::BN * 128 + i * KPP * 128>(stage + dthr, src + a * 64,
                                                             r >= 0 ? 8u : 0u);
          });
        }
      });
    };
    auto convert = [&](uint32_t stage, auto l_c) {
      constexpr int L = decltype(l_c)::value;
      static_for<0, NKEYS>([&](auto i_c) {
        constexpr int i = decltype(i_c)::value;
        if constexpr (!C::SPLIT) {
          const uint32_t a = stage + dthr + i * KPP * 128;
          st_shared_u4(a, fp8x8_to_bf16x8<FMT>(ld_shared_u2(a)));
        } else {
          static_for<0, (L + 63) / 64>([&](auto a_c) {
            constexpr int a = decltype(a_c)::value;
            if (a * 8 + ch < L / 8) {
              const uint32_t at = stage + dthr + a * C::BN * 128 + i * KPP * 128;
              st_shared_u4(at, fp8x8_to_bf16x8<FMT>(ld_shared_u2(at)));
            }
          });
        }
      });
      fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
    };
    for (uint32_t uc = 0; ok && !*abort_flag; ++uc) {
      const int u = ring_unit(&bars[B_U_FULL], &bars[B_U_EMPTY], s_unit, uc, abort_flag, true, ok, p.wait_ns);
      if (u < 0) break;
      const WorkUnit w = p.units[p.uorder[u]];
      const int nt = w.n_tiles;
      if (nt == 0) continue;
      const uint8_t *kp8 =
          reinterpret_cast<const uint8_t *>(p.k_pool) + (int64_t)w.kvh * p.kb_sh + ch * 8;
      const uint8_t *vp8 =
          reinterpret_cast<const uint8_t *>(p.v_pool) + (int64_t)w.kvh * p.vb_sh + ch * 8;
      const bf16 *kx = p.k_ext + (int64_t)w.kvh * p.ke_sh + ch * 8;
      const bf16 *vx = p.v_ext + (int64_t)w.kvh * p.ve_sh + ch * 8;
      int rows[NKEYS];
      auto tile_from_ext = [&](int j) {
        int kb, ke;
        tile_keys(w, j, kb, ke);
        return MODE == kTwoStage && kb >= w.k_split;
      };
      auto fetch = [&]() -> bool {
        const int is = ic % C::NI;
        if (!mbar_wait(&i_full[is], (ic / C::NI) & 1u, abort_flag, p.wait_ns)) return false;
        const int4 *ring =
            reinterpret_cast<const int4 *>(smem + C::OFF_I + is * C::I_BYTES) + key0 * (NKEYS / 4);
#pragma unroll
        for (int q = 0; q < NKEYS / 4; ++q) {
          const int4 v = ring[q];
          rows[4 * q] = v.x;
          rows[4 * q + 1] = v.y;
          rows[4 * q + 2] = v.z;
          rows[4 * q + 3] = v.w;
        }
        __syncwarp();  // the warp is done with the ring slot
        if (lane == 0) mbar_arrive(&i_empty[is]);
        ++ic;
        return true;
      };
      auto issue_k = [&](bool from_ext) -> bool {
        const int ks = kc % NK_;
        if (kc >= (uint32_t)NK_ &&
            !mbar_wait(&k_empty[ks], ((kc / NK_) - 1) & 1u, abort_flag, p.wait_ns))
          return false;
        const uint32_t stage = sbase + K0 + ks * C::K_BYTES;
        if (from_ext) {
          copy_rows(stage, kx, p.ke_st, rows, K_LEN);
          cp_async_arrive_noinc(&k_full[ks]);
        } else {
          issue_raw(stage, kp8, p.kb_ss, rows, K_LEN);
        }
        cp_async_commit();
        ++kc;
        return true;
      };
      auto issue_v = [&](bool from_ext) -> bool {
        const int vs = vc % C::NV;
        if (vc >= (uint32_t)C::NV &&
            !mbar_wait(&v_empty[vs], ((vc / C::NV) - 1) & 1u, abort_flag, p.wait_ns))
          return false;
        const uint32_t stage = sbase + C::OFF_V + vs * C::V_BYTES;
        if (from_ext) {
          copy_rows(stage, vx, p.ve_st, rows, V_LEN);
          cp_async_arrive_noinc(&v_full[vs]);
        } else {
          issue_raw(stage, vp8, p.vb_ss, rows, V_LEN);
        }
        cp_async_commit();
        ++vc;
        return true;
      };
      if constexpr (NK_ < 2 || C::NV < 2) {
        // one K or one V stage (the 288 / 256 layout): the next tile's codes
        // could only go into the stage this tile holds, so each tile's codes
        // are converted as soon as they land
        for (int j = 0; j < nt; ++j) {
          const bool ext = tile_from_ext(j);
          if (!fetch() || !issue_k(ext)) {
            ok = false;
            break;
          }
          if (!ext) {
            cp_async_wait_group<0>();
            const int ks = (kc - 1) % NK_;
            convert(sbase + K0 + ks * C::K_BYTES, K_LEN);
            mbar_arrive(&k_full[ks]);
          }
          if (!issue_v(ext)) {
            ok = false;
            break;
          }
          if (!ext) {
            cp_async_wait_group<0>();
            const int vs = (vc - 1) % C::NV;
            convert(sbase + C::OFF_V + vs * C::V_BYTES, V_LEN);
            mbar_arrive(&v_full[vs]);
          }
        }
        continue;
      }
      bool ext_j = tile_from_ext(0);
      if (!fetch() || !issue_k(ext_j) || !issue_v(ext_j)) {
        ok = false;
        break;
      }
      for (int j = 0; j < nt; ++j) {
        const int ks_j = (kc - 1) % NK_, vs_j = (vc - 1) % C::NV;
        const bool more = j + 1 < nt;
        const bool ext_n = more && tile_from_ext(j + 1);
        if (more && (!fetch() || !issue_k(ext_n))) {
          ok = false;
          break;
        }
        if (!ext_j) {
          // groups issued after K(j): V(j), and K(j+1) if there is one
          if (more) cp_async_wait_group<2>();
          else cp_async_wait_group<1>();
          convert(sbase + K0 + ks_j * C::K_BYTES, K_LEN);
          mbar_arrive(&k_full[ks_j]);
        }
        if (more && !issue_v(ext_n)) {
          ok = false;
          break;
        }
        if (!ext_j) {
          // groups issued after V(j): K(j+1) and V(j+1) if there are
          if (more) cp_async_wait_group<2>();
          else cp_async_wait_group<0>();
          convert(sbase + C::OFF_V + vs_j * C::V_BYTES, V_LEN);
          mbar_arrive(&v_full[vs_j]);
        }
        ext_j = ext_n;
      }
    }
    }
    if (!ok) abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
    cp_async_wait_all();
  } else if (kv_write) {
    // ------------------------------------------ fused KV write (warps 14-15)
    // The pages store the new tokens' K/V rows in the pool before attending
    // (set_kv_buffer(layer, cache_loc, k, v)).  The two-stage form reads the
    // extend keys from k_extend / v_extend, so the store can run beside the
    // attention: each unit copies the rows of its own tokens whose key
    // positions lie in its key range (split-KV units of one block cover
    // disjoint ranges, so every (token, KV head) row is written once).  A
    // slot outside the pool is skipped.
    constexpr int CK = C::LQ / 8, CV = C::HDV / 8;  // 16-byte chunks of a K / V row
    const int wt = tid - 14 * 32;                    // 0 .. 63
    bool ok = true;
    for (uint32_t uc = 0; ok && !*abort_flag; ++uc) {
      const int u = ring_unit(&bars[B_U_FULL], &bars[B_U_EMPTY], s_unit, uc, abort_flag, true, ok, p.wait_ns);
      if (u < 0) break;
      const WorkUnit w = p.units[p.uorder[u]];
      const int t0 = max(w.k_begin, w.qpos0) - w.qpos0;
      const int t1 = min(w.k_end, w.qpos0 + w.n_tok) - w.qpos0;
      const int n = (t1 - t0) * (CK + CV);
      const bf16 *kx = p.k_ext + (int64_t)w.kvh * p.ke_sh;
      const bf16 *vx = p.v_ext + (int64_t)w.kvh * p.ve_sh;
      bf16 *kp = p.k_pool_w + (int64_t)w.kvh * p.kb_sh;
      bf16 *vp = p.v_pool_w + (int64_t)w.kvh * p.vb_sh;
      // four chunks in flight per thread: loads first, then the stores
      for (int c0 = wt; c0 < n; c0 += 4 * 64) {
        uint4 v[4];
        bf16 *dst[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = c0 + k * 64;
          dst[k] = nullptr;
          if (c < n) {
            const int t = t0 + c / (CK + CV), ch = c % (CK + CV);
            const int64_t row = w.q_tok0 + t;
            const int64_t slot = __ldg(p.cache_loc + row);
            if (slot >= 0 && slot < p.num_slots) {
              const bool is_k = ch < CK;
              const int e = (is_k ? ch : ch - CK) * 8;
              v[k] = __ldg(reinterpret_cast<const uint4 *>(
                  (is_k ? kx + row * p.ke_st : vx + row * p.ve_st) + e));
              dst[k] = (is_k ? kp + slot * p.kb_ss : vp + slot * p.vb_ss) + e;
            }
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (dst[k]) *reinterpret_cast<uint4 *>(dst[k]) = v[k];
      }
    }
    if (!ok) abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
  }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ================================================================== MLA ====
#include "mla_pair_kernel.cuh"

// ============================================================== combine ====
// Merge the split-KV partials of every split query block: with lse_i the
// partial log-sum-exps and o_i the partial (normalised) outputs,
//   lse = log sum_i exp(lse_i),  o = sum_i exp(lse_i - lse) o_i
// (the merge_state formula applied n ways).
__global__ void __launch_bounds__(256) combine_kernel(const WsHeader *hdr, const CombineEntry *ce,
                                                      const float *__restrict__ plse,
                                                      const float *__restrict__ po,
                                                      bf16 *__restrict__ o, float *__restrict__ lse,
                                                      const float *sinks, int hq, int group,
                                                      int hdv, int rows_per_slot) {
  grid_dep_wait();  // the attention kernel's partials
  const int n_comb = hdr->n_combine;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int64_t idx = gw; idx < (int64_t)n_comb * rows_per_slot; idx += nw) {
    const int e = (int)(idx / rows_per_slot), r = (int)(idx % rows_per_slot);
    const CombineEntry E = ce[e];
    if (r >= E.n_tok * group) continue;
    // partial i: slot slot0 + i / halves, half i % halves (halves = 2 when
    // the block's two key streams share each slot)
    const int halves = E.pad[0] == 2 ? 2 : 1, n_part = E.n_split * halves;
    auto prow = [&](int i) {
      return (int64_t)(E.slot0 + i / halves) * rows_per_slot + (i % halves) * (rows_per_slot / 2) +
             r;
    };
    float mx = -INFINITY;
    for (int i = 0; i < n_part; ++i) mx = fmaxf(mx, plse[prow(i)]);
    const int t = r / group, g = r - t * group;
    const int64_t orow = (int64_t)(E.q_tok0 + t) * hq + E.kvh * group + g;
    // a sink (natural-log logit of the head) joins the denominator once
    const float sink = sinks ? __ldg(sinks + E.kvh * group + g) : -INFINITY;
    const float mx_p = mx;
    mx = fmaxf(mx, sink);
    if (mx_p == -INFINITY) {
      for (int c = lane * 4; c < hdv; c += 128)
        *reinterpret_cast<uint2 *>(o + orow * hdv + c) = make_uint2(0, 0);
      if (lane == 0 && lse) lse[orow] = sink;  // -inf without a sink
      continue;
    }
    float wsum = sinks ? exp2f((sink - mx) * 1.4426950408889634f) : 0.f;
    for (int i = 0; i < n_part; ++i) wsum += exp2f((plse[prow(i)] - mx) * 1.4426950408889634f);
    const float inv = 1.0f / wsum;
    // every lane takes 4 consecutive value dims of each 128-dim pass (at
    // most four passes: Lv <= 512); a partial's loads for all passes go out
    // together, and the row is stored once every partial is added
    constexpr int kPasses = 4;
    float acc[kPasses][4] = {};
    for (int i = 0; i < n_part; ++i) {
      const int64_t sr = prow(i);
      const float wi = exp2f((plse[sr] - mx) * 1.4426950408889634f) * inv;
      const float *src = po + sr * hdv + lane * 4;
#pragma unroll
      for (int k = 0; k < kPasses; ++k) {
        if (k * 128 + lane * 4 < hdv) {
          const float4 a = *reinterpret_cast<const float4 *>(src + k * 128);
          acc[k][0] += wi * a.x; acc[k][1] += wi * a.y; acc[k][2] += wi * a.z; acc[k][3] += wi * a.w;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kPasses; ++k) {
      const int c = k * 128 + lane * 4;
      if (c < hdv)
        *reinterpret_cast<uint2 *>(o + orow * hdv + c) =
            make_uint2(pack_bf16(acc[k][0], acc[k][1]), pack_bf16(acc[k][2], acc[k][3]));
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

constexpr int kMaxDevicesCfg = 64;

// Rows of one split-KV partial slot: both Q tiles of an extend block, or the
// group's rows of a decode query.
bool split_head_dims(int lq, int lv) { return (lq == 192 && lv == 128) || (lq == 288 && lv == 256); }

int q_tiles_per_unit(int lq, int lv) {
  return (lq == 576 && lv == 512) || split_head_dims(lq, lv) ? 1 : 2;
}

int rows_per_slot(bool decode, int group, int nqt) {
  return decode ? group : nqt * tokens_per_block(group) * group;
}

WsLayout ws_layout(int batch, int num_q_tokens, int hkv, int group, int lq, int lv, int num_sms,
                   bool decode, bool two_streams) {
  WsLayout L{};
  const bool mla = lq == 576 && lv == 512;
  // tokens of a query block: two Q tiles (GQA kernel, Lq = Lv <= 128) or one
  // (MLA kernel, split head dims)
  const int nqt = q_tiles_per_unit(lq, lv);
  const int tok = nqt * tokens_per_block(group);
  L.unit_target = 4 * (num_sms > 0 ? num_sms : 160);
  L.qb_max = (tok > 0 ? (num_q_tokens + tok - 1) / tok : 0) + batch + 1;
  L.unit_max = (L.unit_target + hkv * L.qb_max) * (mla ? 4 : 1);
  L.slot_max = 2 * L.unit_target;
  L.comb_max = L.unit_target;
  if (decode && !mla && !split_head_dims(lq, lv) && two_streams) {
    // two key streams per unit: two partial slots per unit, a combine entry
    // per (query block, KV head)
    L.slot_max = 2 * L.unit_max;
    L.comb_max = L.unit_target + hkv * L.qb_max;
  }
  L.rows_per_slot = rows_per_slot(decode, group, nqt);
  size_t off = align256(sizeof(WsHeader));
  L.seq_off = off;
  off = align256(off + sizeof(int32_t) * 8 * (size_t)(batch + 1));
  L.qb_off = off;
  off = align256(off + sizeof(int32_t) * kSchedBlockArrays * (size_t)L.qb_max);
  L.part_off = off;
  off = align256(off + sizeof(int32_t) * (size_t)(kMaxStreamParts + 1));
  L.units_off = off;
  off = align256(off + sizeof(WorkUnit) * (size_t)L.unit_max);
  L.uorder_off = off;
  off = align256(off + sizeof(int32_t) * (size_t)L.unit_max);
  L.comb_off = off;
  off = align256(off + sizeof(CombineEntry) * (size_t)L.comb_max);
  L.plse_off = off;
  off = align256(off + sizeof(float) * (size_t)L.slot_max * L.rows_per_slot);
  L.po_off = off;
  off = align256(off + sizeof(float) * (size_t)L.slot_max * L.rows_per_slot * lv);
  L.total = off;
  return L;
}

// Whether a kernel's dynamic shared-memory limit has been raised on the
// current device (the attribute is per device; one flag array per kernel).
static bool needs_config(bool (&done)[kMaxDevicesCfg]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesCfg) return true;
  return !done[dev];
}
static void mark_configured(bool (&done)[kMaxDevicesCfg]) {
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevicesCfg) done[dev] = true;
}

// cuTensorMapEncodeTiled from the driver, looked up once.
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 3-D map over q [n, hq, lq]: box = 64 dims x G heads x tok tokens.
static int make_q_map(CUtensorMap *m, const void *q, int64_t n, int hq, int lq, int G, int tok) {
  auto fn = encode_fn();
  if (!fn) return set_error(PKX_ECUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[3] = {(cuuint64_t)lq, (cuuint64_t)hq, (cuuint64_t)n};
  cuuint64_t strides[2] = {(cuuint64_t)lq * 2, (cuuint64_t)hq * lq * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)tok};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(PKX_EINVAL, "q tensor map rejected: %d", (int)r);
  return PKX_OK;
}

template <int HD, int MODE, bool MASK = false, int FMT = 0>
static int launch_attn_kernel(const TMaps &tmaps, const KParams &kp, int grid, cudaStream_t s) {
  using C = Cfg<HD>;
  static bool configured[kMaxDevicesCfg] = {};  // per instantiation and device
  if (needs_config(configured)) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<HD, MODE, MASK, FMT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess)
      return set_error(PKX_ECUDA, "cudaFuncSetAttribute(attn_kernel): %s", cudaGetErrorString(e));
    mark_configured(configured);
  }
  cudaError_t e = launch_pdl(attn_kernel<HD, MODE, MASK, FMT>, dim3(grid), dim3(C::THREADS),
                             C::SMEM, s, tmaps, kp);
  if (e != cudaSuccess)
    return set_error(PKX_ECUDA, "attn_kernel launch: %s", cudaGetErrorString(e));
  return PKX_OK;
}

// The three key modes of one head size over an fp8 pool (the two extend
// forms with or without a custom mask).
template <int HD, int FMT>
static int launch_attn_fp8(int mode, bool masked, const TMaps &tmaps, const KParams &kp,
                           int grid, cudaStream_t s) {
  if (mode == kTwoStage)
    return masked ? launch_attn_kernel<HD, kTwoStage, true, FMT>(tmaps, kp, grid, s)
                  : launch_attn_kernel<HD, kTwoStage, false, FMT>(tmaps, kp, grid, s);
  if (mode == kUnified)
    return masked ? launch_attn_kernel<HD, kUnified, true, FMT>(tmaps, kp, grid, s)
                  : launch_attn_kernel<HD, kUnified, false, FMT>(tmaps, kp, grid, s);
  return launch_attn_kernel<HD, kDecode, false, FMT>(tmaps, kp, grid, s);
}

// Pair kernel launch: clusters of two CTAs, programmatic dependent launch.
template <int MODE, bool MASK, int FMT = 0, bool SG = false>
static cudaError_t launch_pair(int pairs, cudaStream_t s, const KParams &kp, bool query_only,
                               int *max_pairs) {
  using C = std::conditional_t<SG, std::conditional_t<FMT != 0, MlaPairDec8Cfg, MlaPairDecCfg>,
                               MlaPairCfg>;
  static bool configured[kMaxDevicesCfg] = {};
  if (needs_config(configured)) {
    cudaError_t e = cudaFuncSetAttribute(mla_pair_kernel<MODE, MASK, FMT, SG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    mark_configured(configured);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = query_only ? 1 : 2;
  if (query_only)
    return cudaOccupancyMaxActiveClusters(max_pairs, mla_pair_kernel<MODE, MASK, FMT, SG>, &cfg);
  return cudaLaunchKernelEx(&cfg, mla_pair_kernel<MODE, MASK, FMT, SG>, kp);
}

// CTA pairs of the MLA kernel that run at once on the current device (an SM
// group with an odd count of free SMs leaves one idle), queried once per
// device; 0 on error.
static int mla_pairs(int nsm) {
  static int cached[kMaxDevicesCfg] = {};
  int dev = 0;
  const bool cache = cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevicesCfg;
  if (cache && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (launch_pair<kUnified, false>(nsm / 2, nullptr, KParams{}, true, &n) != cudaSuccess) {
    set_error(PKX_ECUDA, "cudaOccupancyMaxActiveClusters(mla_pair_kernel) failed");
    return 0;
  }
  n = std::min(n, nsm / 2);
  if (cache && n > 0) cached[dev] = n;
  return n;
}

template <int MODE, bool MASK = false, int FMT = 0>
static int launch_mla_pair(const KParams &kp, int pairs, cudaStream_t s) {
  cudaError_t e;
  if constexpr (MODE == kDecode && !MASK) {
    // decode of at most 32 rows per unit: the five-stage layout
    e = kp.group <= MlaPairDecCfg::XR ? launch_pair<MODE, false, FMT, true>(pairs, s, kp, false, nullptr)
                                      : launch_pair<MODE, false, FMT>(pairs, s, kp, false, nullptr);
  } else {
    e = launch_pair<MODE, MASK, FMT>(pairs, s, kp, false, nullptr);
  }
  if (e != cudaSuccess)
    return set_error(PKX_ECUDA, "mla_pair_kernel launch: %s", cudaGetErrorString(e));
  return PKX_OK;
}

int launch_attention(const AttnArgs &a) {
  const int group = a.hq / a.hkv;
  const int nsm = num_sms_current_device();
  if (nsm <= 0) return set_error(PKX_ECUDA, "cannot query the current device");
  const bool decode = a.mode == kDecode;
  const bool mla = a.lq == 576 && a.lv == 512;
  const int nq = decode ? a.batch : a.num_q_tokens;
  const bool split = split_head_dims(a.lq, a.lv);
  WsLayout L = ws_layout(a.batch, nq, a.hkv, group, a.lq, a.lv, nsm, decode);
  // Decode runs two key streams when the workspace holds their partial
  // slots (pkx_decode_workspace_size asks for that), else one stream.  The
  // MLA kernel and the split head dims run one stream.
  bool dec_two = decode && !mla && !split;
  if (dec_two && a.workspace_bytes < L.total) {
    const WsLayout L1 = ws_layout(a.batch, nq, a.hkv, group, a.lq, a.lv, nsm, decode, false);
    if (a.workspace_bytes >= L1.total) {
      L = L1;
      dec_two = false;
    }
  }
  if (mla) {
    // V must be the first 512 dims of each K row (the MLA layout).
    const bool pool_alias = a.v_buf == a.k_buf && a.vb_ss == a.kb_ss && a.vb_sh == a.kb_sh;
    const bool ext_alias = a.mode != kTwoStage ||
                           (a.v_ext == a.k_ext && a.ve_st == a.ke_st && a.ve_sh == a.ke_sh);
    if (!pool_alias || !ext_alias)
      return set_error(PKX_EUNSUPPORTED,
                       "Lq=576/Lv=512 needs V to be the first 512 dims of each K row");
  }
  // the MLA kernel runs on CTA pairs: units for four rounds of the pairs
  int pairs = 0;
  if (mla) {
    pairs = mla_pairs(nsm);
    if (pairs <= 0) return set_error(PKX_ECUDA, "no CTA pair of the MLA kernel fits the device");
  }
  if (a.workspace == nullptr || a.workspace_bytes < L.total)
    return set_error(PKX_EWORKSPACE, "workspace of %zu bytes given, %zu needed",
                     a.workspace_bytes, L.total);
  if (reinterpret_cast<uintptr_t>(a.workspace) & 255)
    return set_error(PKX_EINVAL, "workspace must be 256-byte aligned");
  if (a.num_slots >= (int64_t)INT_MAX)
    return set_error(PKX_EUNSUPPORTED, "more than 2^31 pool slots");
  uint8_t *ws = static_cast<uint8_t *>(a.workspace);
  WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
  const int tok = tokens_per_block(group);

  // tensor maps
  TMaps tm;
  memset(&tm, 0, sizeof tm);
  int rc = PKX_OK;
  if (!mla && (rc = make_q_map(&tm.q, a.q, nq, a.hq, a.lq, group, decode ? 1 : tok)) != PKX_OK)
    return rc;

  SchedParams sp;
  sp.mode = a.mode;
  sp.qo_indptr = a.qo_indptr;
  sp.kv_indptr = a.kv_indptr;
  sp.prefix_lens = a.prefix_lens;
  sp.batch = a.batch;
  sp.hkv = a.hkv;
  sp.tok = q_tiles_per_unit(a.lq, a.lv) * tok;
  sp.bn = mla ? MlaPairCfg::BN : kBlockN;
  sp.q_tile_tok = tok > 0 ? tok : 1;
  sp.no_causal = a.custom_mask != nullptr;
  sp.key_set = a.mode == kTwoStage ? a.key_set : kAllKeys;
  sp.keep_status = a.keep_status;
  sp.two_streams = !mla && !split && (!decode || dec_two);
  sp.n_dsplit = 1;
  sp.window = a.window;
  sp.num_q_tokens = nq;
  sp.unit_target = mla ? 4 * pairs : L.unit_target;
  // MLA decode with one KV head: a stream partition, one share of the key
  // tiles per CTA pair (equal shares, where run-time claims of equal units
  // leave some pairs one unit more than others)
  // GQA decode over a bf16 pool: one share per CTA, nsm / hkv per KV head
  // (over an fp8 pool the conversion-bound pipeline does better with the
  // run-time claims of smaller units: 0.48 against 0.54 ms on decode_gqa)
  const bool stream =
      decode && (mla ? a.hkv == 1 && pairs <= kMaxStreamParts
                     : !split && a.kv_fmt == kKvBf16 && nsm <= kMaxStreamParts &&
                           nsm % a.hkv == 0);
  sp.parts = stream ? (mla ? pairs : nsm) : 0;
  sp.part_first = reinterpret_cast<int32_t *>(ws + L.part_off);
  sp.qb_max = L.qb_max;
  sp.unit_max = L.unit_max;
  sp.comb_max = L.comb_max;
  sp.slot_max = L.slot_max;
  sp.seq = reinterpret_cast<int32_t *>(ws + L.seq_off);
  sp.qbt = reinterpret_cast<int32_t *>(ws + L.qb_off);
  sp.units = reinterpret_cast<WorkUnit *>(ws + L.units_off);
  sp.uorder = reinterpret_cast<int32_t *>(ws + L.uorder_off);
  sp.comb = reinterpret_cast<CombineEntry *>(ws + L.comb_off);
  sp.hdr = hdr;
  size_t sched_smem = kCostBuckets * sizeof(int);
  {
    const size_t seq_b = (size_t)kSchedSeqArrays * (a.batch + 1) * sizeof(int);
    const size_t blk_b = (size_t)kSchedBlockArrays * L.qb_max * sizeof(int);
    sp.seq_in_smem = sched_smem + seq_b <= (size_t)kSchedSmemMax;
    if (sp.seq_in_smem) sched_smem += seq_b;
    sp.blk_in_smem = sched_smem + blk_b <= (size_t)kSchedSmemMax;
    if (sp.blk_in_smem) sched_smem += blk_b;
    static bool configured[kMaxDevicesCfg] = {};
    if (needs_config(configured)) {
      cudaError_t e = cudaFuncSetAttribute(sched_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kSchedSmemMax);
      if (e != cudaSuccess)
        return set_error(PKX_ECUDA, "cudaFuncSetAttribute(sched_kernel): %s", cudaGetErrorString(e));
      mark_configured(configured);
    }
  }
  {
    cudaError_t e = launch_pdl(sched_kernel, dim3(1), dim3(1024), sched_smem, a.stream, sp);
    if (e != cudaSuccess)
      return set_error(PKX_ECUDA, "sched_kernel launch: %s", cudaGetErrorString(e));
  }

  KParams kp;
  kp.q = static_cast<const bf16 *>(a.q);
  kp.o = static_cast<bf16 *>(a.o);
  kp.lse = a.lse;
  kp.k_pool = static_cast<const bf16 *>(a.k_buf);
  kp.v_pool = static_cast<const bf16 *>(a.v_buf);
  kp.k_ext = static_cast<const bf16 *>(a.mode == kTwoStage ? a.k_ext : a.k_buf);
  kp.v_ext = static_cast<const bf16 *>(a.mode == kTwoStage ? a.v_ext : a.v_buf);
  kp.kb_ss = a.kb_ss;
  kp.vb_ss = a.vb_ss;
  kp.ke_st = a.ke_st;
  kp.ve_st = a.ve_st;
  kp.kb_sh = a.kb_sh;
  kp.vb_sh = a.vb_sh;
  kp.ke_sh = a.ke_sh;
  kp.ve_sh = a.ve_sh;
  kp.num_slots = a.num_slots;
  kp.qo_indptr = a.qo_indptr;
  kp.kv_indptr = a.kv_indptr;
  kp.kv_indices = a.kv_indices;
  kp.hq = a.hq;
  kp.group = group;
  kp.tok = tok;
  kp.q_box_tok = decode ? 1 : tok;
  kp.window = a.window;
  kp.rows_per_slot = L.rows_per_slot;
  const float log2e = 1.4426950408889634f;
  const float sm_scale = a.sm_scale > 0.f ? a.sm_scale : 1.0f / sqrtf((float)a.lq);
  kp.use_cap = a.logit_cap > 0.f;
  kp.scale_log2 = sm_scale * log2e;
  kp.cap_pre = kp.use_cap ? sm_scale / a.logit_cap : 0.f;
  kp.cap_log2 = kp.use_cap ? a.logit_cap * log2e : 0.f;
  kp.scale_log2_k = kp.scale_log2 * a.k_scale;
  kp.cap_pre_k = kp.cap_pre * a.k_scale;
  kp.custom_mask = a.custom_mask;
  kp.mask_indptr = a.mask_indptr;
  kp.sinks = a.sinks;
  kp.dec_two = dec_two ? 1 : 0;
  kp.log2_v_scale = log2f(a.v_scale);
  kp.v_scale = a.v_scale;
  kp.inv_v_scale = 1.0f / a.v_scale;
  kp.prefix_lens = a.prefix_lens;
  kp.units = sp.units;
  kp.uorder = sp.uorder;
  kp.next_unit = &hdr->next_unit;
  kp.part_first = stream ? sp.part_first : nullptr;
  kp.hdr = hdr;
  kp.status = &hdr->status;
  kp.plse = reinterpret_cast<float *>(ws + L.plse_off);
  kp.po = reinterpret_cast<float *>(ws + L.po_off);
  wait_settings(&kp.wait_ns, &kp.stall);
  kp.cache_loc = a.cache_loc;
  kp.k_pool_w = static_cast<bf16 *>(const_cast<void *>(a.k_buf));
  kp.v_pool_w = static_cast<bf16 *>(const_cast<void *>(a.v_buf));

  const int grid = nsm;
  cudaEvent_t ev_before = nullptr, ev_after = nullptr;
  attention_events(&ev_before, &ev_after);
  if (ev_before) cudaEventRecord(ev_before, a.stream);
  const bool masked = a.custom_mask != nullptr;
  if (a.kv_fmt != kKvBf16 && mla) {
    // the MLA pair kernel over an fp8 pool
    const bool e4 = a.kv_fmt == kKvFp8E4M3;
    if (a.mode == kTwoStage)
      rc = masked ? (e4 ? launch_mla_pair<kTwoStage, true, 1>(kp, pairs, a.stream)
                        : launch_mla_pair<kTwoStage, true, 2>(kp, pairs, a.stream))
                  : (e4 ? launch_mla_pair<kTwoStage, false, 1>(kp, pairs, a.stream)
                        : launch_mla_pair<kTwoStage, false, 2>(kp, pairs, a.stream));
    else if (a.mode == kUnified)
      rc = masked ? (e4 ? launch_mla_pair<kUnified, true, 1>(kp, pairs, a.stream)
                        : launch_mla_pair<kUnified, true, 2>(kp, pairs, a.stream))
                  : (e4 ? launch_mla_pair<kUnified, false, 1>(kp, pairs, a.stream)
                        : launch_mla_pair<kUnified, false, 2>(kp, pairs, a.stream));
    else
      rc = e4 ? launch_mla_pair<kDecode, false, 1>(kp, pairs, a.stream)
              : launch_mla_pair<kDecode, false, 2>(kp, pairs, a.stream);
  } else if (a.kv_fmt != kKvBf16 && split) {
    // the split head dims over an fp8 pool: the two extend forms, no mask
    if (a.mode == kDecode || masked)
      return set_error(PKX_EUNSUPPORTED,
                       "an fp8 pool with split head dims is built for extend without a mask");
    const bool e4 = a.kv_fmt == kKvFp8E4M3, two = a.mode == kTwoStage;
    if (a.lq == 192)
      rc = two ? (e4 ? launch_attn_kernel<192, kTwoStage, false, 1>(tm, kp, grid, a.stream)
                     : launch_attn_kernel<192, kTwoStage, false, 2>(tm, kp, grid, a.stream))
               : (e4 ? launch_attn_kernel<192, kUnified, false, 1>(tm, kp, grid, a.stream)
                     : launch_attn_kernel<192, kUnified, false, 2>(tm, kp, grid, a.stream));
    else
      rc = two ? (e4 ? launch_attn_kernel<288, kTwoStage, false, 1>(tm, kp, grid, a.stream)
                     : launch_attn_kernel<288, kTwoStage, false, 2>(tm, kp, grid, a.stream))
               : (e4 ? launch_attn_kernel<288, kUnified, false, 1>(tm, kp, grid, a.stream)
                     : launch_attn_kernel<288, kUnified, false, 2>(tm, kp, grid, a.stream));
  } else if (a.kv_fmt != kKvBf16) {
    if (!((a.lq == 128 && a.lv == 128) || (a.lq == 64 && a.lv == 64)))
      return set_error(PKX_EUNSUPPORTED,
                       "an fp8 pool is built for Lq = Lv = 64 or 128, for Lq / Lv = 576 / 512 and "
                       "for the split head dims in extend");
    const bool e4 = a.kv_fmt == kKvFp8E4M3;
    if (a.lq == 128)
      rc = e4 ? launch_attn_fp8<128, 1>(a.mode, masked, tm, kp, grid, a.stream)
              : launch_attn_fp8<128, 2>(a.mode, masked, tm, kp, grid, a.stream);
    else
      rc = e4 ? launch_attn_fp8<64, 1>(a.mode, masked, tm, kp, grid, a.stream)
              : launch_attn_fp8<64, 2>(a.mode, masked, tm, kp, grid, a.stream);
  } else if (a.lq == 128 && a.lv == 128) {
    if (a.mode == kTwoStage)
      rc = masked ? launch_attn_kernel<128, kTwoStage, true>(tm, kp, grid, a.stream)
                  : launch_attn_kernel<128, kTwoStage>(tm, kp, grid, a.stream);
    else if (a.mode == kUnified)
      rc = masked ? launch_attn_kernel<128, kUnified, true>(tm, kp, grid, a.stream)
                  : launch_attn_kernel<128, kUnified>(tm, kp, grid, a.stream);
    else rc = launch_attn_kernel<128, kDecode>(tm, kp, grid, a.stream);
  } else if (a.lq == 64 && a.lv == 64) {
    if (a.mode == kTwoStage)
      rc = masked ? launch_attn_kernel<64, kTwoStage, true>(tm, kp, grid, a.stream)
                  : launch_attn_kernel<64, kTwoStage>(tm, kp, grid, a.stream);
    else if (a.mode == kUnified)
      rc = masked ? launch_attn_kernel<64, kUnified, true>(tm, kp, grid, a.stream)
                  : launch_attn_kernel<64, kUnified>(tm, kp, grid, a.stream);
    else rc = launch_attn_kernel<64, kDecode>(tm, kp, grid, a.stream);
  } else if (split) {
    if (masked)
      return set_error(PKX_EUNSUPPORTED, "a custom mask is not built for head dims (%d, %d)",
                       a.lq, a.lv);
    if (a.lq == 192) {
      if (a.mode == kTwoStage) rc = launch_attn_kernel<192, kTwoStage>(tm, kp, grid, a.stream);
      else if (a.mode == kUnified) rc = launch_attn_kernel<192, kUnified>(tm, kp, grid, a.stream);
      else rc = launch_attn_kernel<192, kDecode>(tm, kp, grid, a.stream);
    } else {
      if (a.mode == kTwoStage) rc = launch_attn_kernel<288, kTwoStage>(tm, kp, grid, a.stream);
      else if (a.mode == kUnified) rc = launch_attn_kernel<288, kUnified>(tm, kp, grid, a.stream);
      else rc = launch_attn_kernel<288, kDecode>(tm, kp, grid, a.stream);
    }
  } else if (mla) {
    if (a.mode == kTwoStage)
      rc = masked ? launch_mla_pair<kTwoStage, true>(kp, pairs, a.stream)
                  : launch_mla_pair<kTwoStage>(kp, pairs, a.stream);
    else if (a.mode == kUnified)
      rc = masked ? launch_mla_pair<kUnified, true>(kp, pairs, a.stream)
                  : launch_mla_pair<kUnified>(kp, pairs, a.stream);
    else rc = launch_mla_pair<kDecode>(kp, pairs, a.stream);
  } else {
    return set_error(PKX_EUNSUPPORTED, "head dims (%d, %d) not built", a.lq, a.lv);
  }
  if (rc != PKX_OK) return rc;
  if (ev_after) cudaEventRecord(ev_after, a.stream);
  // one warp per combined row: enough CTAs for a full wave of warps (the
  // rows' partial reads are latency-bound), eight per SM at most
  const size_t comb_rows = (size_t)L.comb_max * L.rows_per_slot;
  const int comb_grid = (int)std::min<size_t>((comb_rows + 7) / 8, (size_t)nsm * 8);
  cudaError_t e = launch_pdl(combine_kernel, dim3(comb_grid > 0 ? comb_grid : 1), dim3(256), 0,
                             a.stream,
                             (const WsHeader *)hdr, (const CombineEntry *)sp.comb,
                             (const float *)kp.plse, (const float *)kp.po, kp.o, a.lse, a.sinks,
                             a.hq, group, a.lv, L.rows_per_slot);
  if (e != cudaSuccess) return set_error(PKX_ECUDA, "attention launch: %s", cudaGetErrorString(e));
  return PKX_OK;
}

}  // namespace pkx
