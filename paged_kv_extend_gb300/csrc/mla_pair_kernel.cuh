// mla_pair_kernel.cuh -- extend / decode attention for the MLA head shape
// (Lq = 576 = 512 latent + 64 rope dims, Lv = 512, one KV head, V = the first
// 512 dims of each K row) on a pair of CTAs, included by attention.cu.
//
// The MLA layout (sglang cpu_graph_runner.py, qkv_proj_with_rope fake: V is a
// narrow view of K; extend_attention.py, _get_block_sizes_for_extend_attention:
// 576 = 512 + 64) makes the score one 576-dim dot product and lets the K tile
// double as V.  A 128-row tile's O over all 512 value dims (512 TMEM columns)
// does not fit one SM's TMEM next to Q and S, so the two CTAs of a cluster
// split the dims instead of recomputing S per value slice:
//   rank r holds value dims [256 r, 256 r + 256) and rope dims
//   [512 + 32 r, 512 + 32 r + 32) of Q and K (288 dims each);
//   each computes its partial S = Q_r K_r^T (64 keys per tile), sends it to
//   the other, and adds the other's: fp32 addition commutes, so both hold the
//   same S bit for bit, run the same softmax and get the same P;
//   each then computes O for its own value dims, the first 256 of its K dims.
// No product is recomputed: per (row, key) the pair does 2 x 576 + 2 x 512
// FLOP, the algorithmic count.
//
//   TMEM (per CTA)  [0, 144) Q_r as bf16 pairs
//                   [160, 192) P (bf16 pairs, 64 keys)
//                   [192, 256) S, the partial of this rank (fp32)
//                   [256, 512) O, 256 value dims (fp32)
//   SMEM  four stages of a 64-key K tile (four 64-dim swizzle atoms of value
//         dims and one atom whose first half holds the rope dims), two
//         receive buffers of the other rank's partial S (tile t in buffer
//         t & 1; 16-byte chunk c of row r at c * 128 * 16 + r * 16), a ring
//         of resolved row indices.
//
// The exchange runs one tile ahead of the softmax, so that its latency hides
// behind the softmax of the previous tile, and QK^T runs two tiles ahead of
// PV.  In the iteration of tile j each softmax thread
//   adds its own partial of tile j (kept in registers) to the other rank's
//   (received in shared memory; XFULL of the buffer);
//   reads S(j + 1) into registers and releases it (S_FREE; QK^T of tile
//   j + 2 follows) and writes its row of S(j + 1) into the other rank's
//   buffer (j + 1) & 1 with asynchronous remote stores whose bytes complete
//   that buffer's XFULL there;
//   runs the softmax of tile j and writes P(j).
// A buffer's XFULL is armed (one arrival that expects the tile's bytes) by
// thread 0 once the buffer's previous phase has completed; the bytes may
// land first.  No barrier frees a buffer: a thread sends tile t only after
// tile t - 1 of all exchanging threads of the other rank landed here, and
// each of them read its row of tile t - 2 from the buffer before it sent
// tile t - 1 (the complete-tx of its stores releases at cluster scope, the
// wait here acquires).  Extend exchanges all 128 rows; in decode, whose
// units all hold G rows, only the warps with real rows exchange.
// Both CTAs of a pair take the same units in the same order, so their tile
// counters stay in step: one thread of rank 0 claims them from the global
// cost order (largest first) and writes each into slot uc % 4 of both ranks'
// unit rings (a remote store, then a remote arrive that releases it on the
// slot's U_FULL there); every consuming warp releases the slot on its own
// CTA's U_EMPTY (a CTA-scope release, which does not wait for the warp's
// earlier global stores to reach the cluster), and one thread of rank 1
// forwards each completed phase of rank 1's U_EMPTY to rank 0's.  The
// claimer takes unit uc only once every warp of both ranks has taken unit
// uc - 2, so a pair holds at most three units and the rest stay free for
// whichever pair finishes first.  Under a stream partition (MLA decode with
// one KV head) the pair walks its own share of the claim order instead.
// The row-index warp, which runs tiles ahead, prefetches each unit's query
// rows into L2.
// Warps: 0-3 softmax (one row per thread; they also write Q into TMEM), 4 MMA
// issue, 5 row indices, 6-9 K-row copies (cp.async), 10 unit claims (one
// thread of rank 0) and slot releases forwarded (one thread of rank 1), 11
// idle.

// NK_: K stages; XR_: rows a receive buffer holds (the rows that exchange);
// NRAW_: raw fp8 code slots per copy thread's ring (0: codes converted in
// place in the stages).
template <int NK_, int XR_, int NRAW_ = 0>
struct MlaPairCfgT {
  static constexpr int BM = kBlockM, BN = 64;
  static constexpr int LQ = 576, LV = 512;
  static constexpr int DV = LV / 2;             // value dims per rank
  static constexpr int DR = (LQ - LV) / 2;      // rope dims per rank
  static constexpr int KSTEPS = (DV + DR) / 16;  // K-steps of QK^T: 18
  static constexpr int NK = NK_, NI = 4;
  static constexpr int XR = XR_;
  static constexpr int K_BYTES = BN * 5 * 128;  // four value atoms + the rope atom
  static constexpr int X_BYTES = XR * BN * 4;   // a partial S
  static constexpr int I_BYTES = BN * 4;
  static constexpr int NRAW = NRAW_;
  // a raw slot: the codes of a tile, four 64-byte value atoms per key
  // (atom-major, key rows of 64 bytes) and then the 32-byte rope rows
  static constexpr int RAW_BYTES = BN * (DV + DR);
  static constexpr int OFF_K = 0;
  static constexpr int OFF_RAW = NK * K_BYTES;
  static constexpr int OFF_X = OFF_RAW + NRAW * RAW_BYTES;  // received from the other rank
  static constexpr int OFF_I = OFF_X + 2 * X_BYTES;
  static constexpr int OFF_BAR = OFF_I + NI * I_BYTES;
  static constexpr int URING = 4;               // unit ring slots
  static constexpr int CLAIM_AHEAD = 2;         // units claimed past the slowest warp's
  static constexpr int UNIT_WARPS = 10;         // warps per CTA that take units
  static constexpr int N_BARS = 18 + 2 * NK + 2 * NI;
  static constexpr int SMEM = OFF_BAR + N_BARS * 8 + 1024;
  static constexpr int TMEM_COLS = 512;
  static constexpr int Q_COL = 0, P_COL = 160, S_COL = 192, O_COL = 256;
  static constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, 0);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, DV, 1);
  static constexpr int THREADS = 384;
  static constexpr int COPY_WARP0 = 6, COPY_THREADS = 128;
  // Registers: the kernel launches with REGS_LAUNCH per thread (checked at
  // build time); the softmax warpgroup takes REGS_SOFTMAX, the other two
  // give back down to REGS_OTHER.  The split must add up exactly.
  static constexpr int REGS_LAUNCH = 168, REGS_SOFTMAX = 232, REGS_OTHER = 136;
  static_assert(128 * REGS_SOFTMAX + 256 * REGS_OTHER == THREADS * REGS_LAUNCH,
                "register split");
  static_assert(SMEM + 256 <= 232448, "shared memory budget (dynamic + static, padded)");
  static_assert(DR == 32 && KSTEPS == 18, "the rope dims fill half an atom");
  static_assert(XR % 32 == 0 && XR <= BM, "whole warps exchange");
};
// Extend, and decode of more than 32 rows per unit: four K stages, every
// row exchanged.
using MlaPairCfg = MlaPairCfgT<4, kBlockM>;
// Decode of at most 32 rows per unit (G <= 32): only warp 0 exchanges, so
// the receive buffers shrink to 32 rows and a fifth K stage fits.  QK^T runs
// two tiles ahead of PV and holds three stages, so the fifth doubles the
// stages being copied.
using MlaPairDecCfg = MlaPairCfgT<5, 32>;
// The same over an fp8 pool: a copy thread stages its codes of a tile in
// one of four private raw slots and converts them into one of three stages
// three tiles later, so a stage is taken only from conversion to PV and the
// copies' latency is covered by the raw ring.
using MlaPairDec8Cfg = MlaPairCfgT<3, 32, 4>;

enum {
  X_Q_FULL = 0,
  X_S_FULL = 1,   // the partial S landed
  X_P_FULL = 2,   // P written
  X_O_DONE = 3,   // last PV of a unit landed
  X_FINAL = 4,
  X_S_FREE = 5,   // S read into registers: the next QK^T may overwrite it
  X_PV_DONE = 6,  // one phase per PV: P and O are free again
  X_NEVER = 7,    // no thread ever arrives (the stall hook waits on it)
  X_XFULL = 8,    // + buffer: the other rank's partial landed (one arrival + its bytes)
  X_U_FULL = 10,  // + slot: a unit written into the slot (the claimer's arrival)
  X_U_EMPTY = 14, // + slot: every consuming warp of the CTA read it (rank 0: and rank 1's, forwarded)
  X_RING = 18
};

// The record of unit uc of this pair from the claim ring (copied there by
// the claimer); n_tiles < 0 marks the end.  Every lane of the calling warp
// takes it; lane 0 then releases the slot on this CTA's U_EMPTY.  ok is
// cleared (and the end returned) if the wait gave up.
__device__ __forceinline__ WorkUnit pair_take(uint64_t *bars, const WorkUnit *recs, uint32_t uc,
                                              volatile int *abort_flag, uint64_t limit_ns,
                                              bool &ok) {
  const int slot = uc % MlaPairCfg::URING;
  WorkUnit w;
  if (!mbar_wait_cluster(&bars[X_U_FULL + slot], (uc / MlaPairCfg::URING) & 1u, abort_flag,
                         limit_ns)) {
    ok = false;
    w.n_tiles = -1;
    return w;
  }
  w = recs[slot];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&bars[X_U_EMPTY + slot]);
  return w;
}

// FMT: the pool's element format (0 bf16; 1 fp8 e4m3, 2 fp8 e5m2 with
// k_scale / v_scale: the copy warps stage a tile's codes and convert them in
// place to bf16, exact, one tile behind their copies; k_scale joins the
// logit scale of pool tiles and v_scale their P).  Extend rows of the
// two-stage form are always bf16.
// SG: decode with at most 32 rows per unit (the launcher checks G <= 32),
// laid out by MlaPairDecCfg.
template <int MODE, bool MASK, int FMT = 0, bool SG = false>
__global__ void __launch_bounds__(MlaPairCfg::THREADS, 1) mla_pair_kernel(const KParams p) {
  static_assert(!SG || (MODE == kDecode && !MASK), "the small-group layout is for decode");
  using C = std::conditional_t<SG, std::conditional_t<FMT != 0, MlaPairDec8Cfg, MlaPairDecCfg>,
                               MlaPairCfg>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ WorkUnit s_rec[MlaPairCfg::URING];  // the claimed units' records

  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *k_full = bars + X_RING;
  uint64_t *k_empty = k_full + C::NK;
  uint64_t *i_full = k_empty + C::NK;
  uint64_t *i_empty = i_full + C::NI;
  volatile int *abort_flag = &s_abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
  const int dv0 = (int)rank * C::DV;            // first value dim of this rank
  const int dr0 = C::LV + (int)rank * C::DR;    // first rope dim of this rank

  if (tid == 0) {
    mbar_init(&bars[X_Q_FULL], 128);
    mbar_init(&bars[X_S_FULL], 1);
    mbar_init(&bars[X_P_FULL], 4);  // one arrival per softmax warp
    mbar_init(&bars[X_O_DONE], 1);
    mbar_init(&bars[X_FINAL], 1);
    mbar_init(&bars[X_S_FREE], 4);
    mbar_init(&bars[X_PV_DONE], 1);
    mbar_init(&bars[X_NEVER], 1);
    for (int b = 0; b < 2; ++b) mbar_init(&bars[X_XFULL + b], 1);
    for (int s = 0; s < C::URING; ++s) {
      mbar_init(&bars[X_U_FULL + s], 1);
      mbar_init(&bars[X_U_EMPTY + s], rank == 0 ? C::UNIT_WARPS + 1 : C::UNIT_WARPS);
    }
    for (int s = 0; s < C::NK; ++s) {
      mbar_init(&k_full[s], C::COPY_THREADS);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::NI; ++s) {
      mbar_init(&i_full[s], 32);
      mbar_init(&i_empty[s], C::COPY_THREADS);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 4) {
    tmem_alloc(&s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  // both CTAs' barriers exist before either arrives on the other's
  cluster_sync();
  tc_fence_after();
  grid_dep_wait();
  grid_dep_launch();
  const uint32_t tmem = s_tmem;
  const int n_units = p.hdr->n_units;
  const int G = p.group;
  if (warp < 4) regs_increase<C::REGS_SOFTMAX>();
  else regs_decrease<C::REGS_OTHER>();

  if (warp < 4) {
    // ------------------------- Q -> TMEM, partial-S exchange, softmax, epilogue
    const int r = tid;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    uint32_t s_cnt = 0, o_cnt = 0;
    uint32_t n_sent = 0, n_recv = 0;  // tiles sent / combined so far
    uint32_t pv_base = 0;  // PVs of earlier units (X_PV_DONE phases)
    const uint32_t xfull_peer = cluster_addr(smem_u32(&bars[X_XFULL]), peer);
    // this thread's row of receive buffer 0 (chunk c at c * XR * 16), here
    // and in the other rank
    const uint8_t *recv_row = smem + C::OFF_X + r * 16;
    const uint32_t send_row = cluster_addr(sbase + C::OFF_X + r * 16, peer);
    uint32_t own[C::BN];  // this rank's partial S of the next tile
    // S of the next tile into registers, released for the next QK^T, and
    // sent to the other rank
    // Warps that exchange: every decode unit holds G rows (one token), so
    // only the warps with real rows send and receive, and a tile's phase
    // expects their bytes; extend units exchange all 128 rows.  (The
    // receive buffers hold C::XR rows: the decode layout takes G <= 32.)
    const int xw = MODE == kDecode ? min(C::XR / 32, (G + 31) / 32) : C::XR / 32;
    const bool xch = warp < xw;
    const uint32_t xbytes = (uint32_t)xw * 32u * (C::BN * 4u);
    auto send = [&]() -> bool {
      if (!mbar_wait(&bars[X_S_FULL], s_cnt & 1u, abort_flag, p.wait_ns)) return false;
      ++s_cnt;
      tc_fence_after();
      if (xch) {
        tmem_ld32(lane_base + C::S_COL, *reinterpret_cast<uint32_t (*)[32]>(own));
        tmem_ld32(lane_base + C::S_COL + 32, *reinterpret_cast<uint32_t (*)[32]>(own + 32));
        tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[X_S_FREE]);
      const uint32_t b = n_sent & 1u;
      if (xch) {
#pragma unroll
        for (int c = 0; c < 16; ++c)
          st_async_cluster_u4(send_row + b * C::X_BYTES + c * (C::XR * 16),
                              make_uint4(own[4 * c], own[4 * c + 1], own[4 * c + 2], own[4 * c + 3]),
                              xfull_peer + b * 8u);
      }
      ++n_sent;
      return true;
    };
    // both partials of the current tile added (own + other in both ranks:
    // the same sum bit for bit)
    auto combine = [&](float (&x)[C::BN]) -> bool {
      const uint32_t b = n_recv & 1u;
      if (xch &&
          !mbar_wait_cluster(&bars[X_XFULL + b], (n_recv >> 1) & 1u, abort_flag, p.wait_ns))
        return false;
      ++n_recv;
      // the buffer's phase for tile n_recv + 1 (its bytes cannot land before
      // every exchanging warp here has read this tile; warp 0 always exchanges)
      if (tid == 0) mbar_arrive_expect_tx(&bars[X_XFULL + b], xbytes);
      if (!xch) return true;  // no real rows: x is not used
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint4 o4 =
            *reinterpret_cast<const uint4 *>(recv_row + b * C::X_BYTES + c * (C::XR * 16));
        x[4 * c + 0] = __uint_as_float(own[4 * c + 0]) + __uint_as_float(o4.x);
        x[4 * c + 1] = __uint_as_float(own[4 * c + 1]) + __uint_as_float(o4.y);
        x[4 * c + 2] = __uint_as_float(own[4 * c + 2]) + __uint_as_float(o4.z);
        x[4 * c + 3] = __uint_as_float(own[4 * c + 3]) + __uint_as_float(o4.w);
      }
      return true;
    };
    if (tid == 0) {  // the first two tiles
      mbar_arrive_expect_tx(&bars[X_XFULL], xbytes);
      mbar_arrive_expect_tx(&bars[X_XFULL + 1], xbytes);
    }
    // this rank's Q dims of unit wq into TMEM as bf16 pairs: four value
    // atoms in columns [0, 128), the rope dims in [128, 144) (zeros up to
    // 160); rows past the block get zeros.  The previous unit's products
    // have all completed (its epilogue waited for them).
    auto write_q = [&](const WorkUnit &wq) {
      const bool vq = r < wq.n_tok * G;
      const int tq = r / G, gq = r - (r / G) * G;
      const int64_t oq = (int64_t)(wq.q_tok0 + tq) * p.hq + wq.kvh * G + gq;
      const uint4 *qrow = reinterpret_cast<const uint4 *>(p.q + oq * C::LQ);
#pragma unroll 1
      for (int c = 0; c < 5; ++c) {
        uint32_t v[32];
        const int q0 = c < 4 ? (dv0 + 64 * c) / 8 : dr0 / 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 x = vq && (c < 4 || i < C::DR / 8) ? __ldg(qrow + q0 + i)
                                                         : make_uint4(0, 0, 0, 0);
          v[4 * i + 0] = x.x;
          v[4 * i + 1] = x.y;
          v[4 * i + 2] = x.z;
          v[4 * i + 3] = x.w;
        }
        tmem_st32(lane_base + C::Q_COL + c * 32, v);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars[X_Q_FULL]);
    };
    if (p.stall && !mbar_wait(&bars[X_NEVER], 0, abort_flag, p.wait_ns))
      abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
    for (uint32_t uc = 0; !*abort_flag; ++uc) {
      bool took = true;
      const WorkUnit w = pair_take(bars, s_rec, uc, abort_flag, p.wait_ns, took);
      if (!took) abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
      if (w.n_tiles < 0) break;
      const int nt = w.n_tiles;
      const int rows_valid = w.n_tok * G;
      const bool valid = r < rows_valid;
      const bool warp_active = warp * 32 < rows_valid;
      const int t = r / G, g = r - (r / G) * G;
      const int qpos = w.qpos0 + t;
      const int qmax = w.qpos0 + w.n_tok - 1;
      const int64_t orow_idx = (int64_t)(w.q_tok0 + t) * p.hq + w.kvh * G + g;
      const int64_t prow_idx = (int64_t)w.slot * p.rows_per_slot + r;
      const uint8_t *mbase = nullptr;
      int64_t mstride = 0;
      if (MASK) {
        const int qo0 = p.qo_indptr[w.b];
        mstride = MODE == kTwoStage ? (int64_t)(p.kv_indptr[w.b + 1] - p.kv_indptr[w.b]) +
                                          (p.qo_indptr[w.b + 1] - qo0)
                                    : (int64_t)(p.kv_indptr[w.b + 1] - p.kv_indptr[w.b]);
        mbase = p.custom_mask + p.mask_indptr[w.b] + (int64_t)(w.q_tok0 - qo0) * mstride;
      }
      if (nt == 0) {
        if (valid) {
          if (w.slot < 0) {
            bf16 *orow = p.o + orow_idx * C::LV + dv0;
            for (int c = 0; c < C::DV; c += 8)
              *reinterpret_cast<uint4 *>(orow + c) = make_uint4(0, 0, 0, 0);
            if (p.lse && rank == 0) p.lse[orow_idx] = -INFINITY;
          } else {
            float *prow = p.po + prow_idx * C::LV + dv0;
            for (int c = 0; c < C::DV; c += 4)
              *reinterpret_cast<float4 *>(prow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            if (rank == 0) p.plse[prow_idx] = -INFINITY;
          }
        }
        continue;
      }
      if constexpr (!SG) write_q(w);  // (small-group decode: the MMA warp writes Q)
      if (!send()) {  // the unit's first tile
        abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
        break;
      }
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j) {
        int kb, ke;
        tile_keys<C::BN>(w, j, kb, ke);
        uint32_t mb[2] = {0u, 0u};
        if constexpr (MASK) {
          if (warp_active) {
            const int t_lo = (warp * 32) / G, t_hi = min((warp * 32 + 31) / G, w.n_tok - 1);
            for (int tc = t_lo; tc <= t_hi; tc += 4) {
              uint8_t by[4][2];
#pragma unroll
              for (int u2 = 0; u2 < 4; ++u2) {
                const uint8_t *rowp = mbase + (int64_t)(tc + u2) * mstride;
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                  const int kpos = kb + 32 * q2 + lane;
                  by[u2][q2] = (tc + u2 <= t_hi && kpos < ke) ? __ldg(rowp + kpos) : (uint8_t)0;
                }
              }
#pragma unroll
              for (int u2 = 0; u2 < 4; ++u2) {
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                  const uint32_t word = __ballot_sync(0xffffffffu, by[u2][q2] != 0);
                  if (t == tc + u2) mb[q2] = word;
                }
              }
            }
          }
        }
        float x[C::BN];
        if (!combine(x) || (j + 1 < nt && !send())) {
          abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
          break;
        }
        float alpha = 1.0f;
        bool o_needs = false;
        uint32_t pk[32];
        if (warp_active) {
          // a pool tile of an fp8 pool holds codes: k_scale joins the logit
          // scale, v_scale its P (through the exponent; the row sum divides
          // it back out)
          const bool pool8 = FMT != 0 && !(MODE == kTwoStage && kb >= w.k_split);
          float sc = pool8 ? p.scale_log2_k : p.scale_log2;
          if (p.use_cap) {
            const float pre = pool8 ? p.cap_pre_k : p.cap_pre;
#pragma unroll
            for (int i = 0; i < C::BN; ++i) x[i] = p.cap_log2 * tanh_approx(x[i] * pre);
            sc = 1.0f;
          }
          const bool need_mask = (ke - 1 > w.qpos0) || (ke - kb < C::BN) ||
                                 (p.window > 0 && kb < qmax - p.window);
          if constexpr (MASK) {
            const bool every = (mb[0] & mb[1]) == 0xffffffffu &&
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
          float mt;
          if (sc >= 0.f) {
            float mt0 = x[0], mt1 = x[1];
#pragma unroll
            for (int i = 2; i < C::BN; i += 2) {
              mt0 = fmaxf(mt0, x[i]);
              mt1 = fmaxf(mt1, x[i + 1]);
            }
            mt = fmaxf(mt0, mt1) * sc;
          } else {
            float mt0 = x[0], mt1 = x[1];
#pragma unroll
            for (int i = 2; i < C::BN; i += 2) {
              mt0 = fminf(mt0, x[i]);
              mt1 = fminf(mt1, x[i + 1]);
            }
            mt = fminf(mt0, mt1) * sc;
          }
          const float m_new = fmaxf(m, mt);
          const bool grow = m_new > m + 8.0f;
          alpha = grow ? ex2_approx(m - m_new) : 1.0f;
          o_needs = grow && j > 0 && l > 0.f;
          if (grow) {
            l *= alpha;
            m = m_new;
          }
          float nm = m == -INFINITY ? 0.f : -m;
          if (pool8) nm += p.log2_v_scale;
          float l0 = 0.f, l1 = 0.f;
#pragma unroll
          for (int i = 0; i < C::BN; i += 2) {
            const float e0 = ex2_approx(fmaf(x[i], sc, nm));
            const float e1 = ex2_approx(fmaf(x[i + 1], sc, nm));
            l0 += e0;
            l1 += e1;
            pk[i / 2] = pack_bf16(e0, e1);
          }
          l += pool8 ? (l0 + l1) * p.inv_v_scale : l0 + l1;
        }
        // P's columns and O are free once the previous tile's PV has landed.
        // Every warp waits, also one without rows, so that no warp arrives
        // on P_FULL twice in one phase.
        if (j > 0 && !mbar_wait(&bars[X_PV_DONE], (pv_base + j - 1) & 1u, abort_flag, p.wait_ns)) {
          abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
        }
        tc_fence_after();
        if (warp_active) {
          tmem_st32(lane_base + C::P_COL, pk);
          if (__any_sync(0xffffffffu, o_needs)) {
            const float a = o_needs ? alpha : 1.0f;
            uint32_t v[32];
#pragma unroll 1
            for (int c = 0; c < C::DV / 32; ++c) {
              const uint32_t ta = lane_base + C::O_COL + c * 32;
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
        if (lane == 0) mbar_arrive(&bars[X_P_FULL]);
      }
      if (*abort_flag) break;
      if (!mbar_wait(&bars[X_O_DONE], o_cnt & 1u, abort_flag, p.wait_ns)) {
        abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
        break;
      }
      ++o_cnt;
      pv_base += nt;
      tc_fence_after();
      if (warp_active) {
        float inv = l > 0.f ? 1.0f / l : 0.f;
        float lse_v = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        if (p.sinks && w.slot < 0) {
          const float s2 = __ldg(p.sinks + w.kvh * G + g) * 1.4426950408889634f;
          const float M = fmaxf(m, s2);
          const float a_m = m == -INFINITY ? 0.f : ex2_approx(m - M);
          const float lt = l * a_m + ex2_approx(s2 - M);
          inv = a_m / lt;
          lse_v = (M + __log2f(lt)) * 0.69314718055994531f;
        }
        uint32_t v[32];
#pragma unroll 1
        for (int c = 0; c < C::DV / 32; ++c) {
          tmem_ld32(lane_base + C::O_COL + c * 32, v);
          tmem_wait_ld();
          if (valid) {
            if (w.slot < 0) {
              bf16 *orow = p.o + orow_idx * C::LV + dv0 + c * 32;
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
              float *prow = p.po + prow_idx * C::LV + dv0 + c * 32;
#pragma unroll
              for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4 *>(prow + i) =
                    make_float4(__uint_as_float(v[i]) * inv, __uint_as_float(v[i + 1]) * inv,
                                __uint_as_float(v[i + 2]) * inv, __uint_as_float(v[i + 3]) * inv);
            }
          }
        }
        if (valid && rank == 0) {
          if (w.slot < 0) {
            if (p.lse) p.lse[orow_idx] = lse_v;
          } else {
            p.plse[prow_idx] = lse_v;
          }
        }
      }
      tc_fence_before();
    }
  } else if (warp == 4) {
    // ------------------------------------------------ MMA issue (one warp)
    // QK^T runs two tiles ahead of PV: S(j + 2) = Q_r K_r(j + 2)^T as soon
    // as the softmax has read S(j + 1) (it does so before it writes P(j)),
    // then O += P(j) V_r(j) once P(j) is written.  The whole warp runs the
    // loop; one elected lane issues.
    const bool leader = elect_one();
    uint32_t q_cnt = 0, kc = 0, p_cnt = 0, f_cnt = 0;
    bool ok = true;
    constexpr uint32_t K_LO = sw128_desc_lo(0), K_HI = sw128_desc_hi(1024);
    constexpr uint32_t V_LO = sw128_desc_lo(C::BN * 128), V_HI = sw128_desc_hi(1024);
    auto issue_s = [&](uint32_t sK) {
      const uint32_t b_lo = K_LO | desc_addr(sK);
      static_for<0, C::KSTEPS>([&](auto kk_c) {
        constexpr int kk = decltype(kk_c)::value;
        constexpr uint32_t bo = ((kk / 4) * (C::BN * 128) + (kk % 4) * 32) / 16;
        if (leader)
          tc_mma_ts_step<kk * 8, bo>(tmem + C::S_COL, tmem + C::Q_COL, b_lo, K_HI, C::IDESC_QK,
                                     kk > 0 ? 1u : 0u);
      });
      if (leader) tc_commit(&bars[X_S_FULL]);
    };
    auto issue_pv = [&](uint32_t sV, bool acc_first) {
      const uint32_t b_lo = V_LO | desc_addr(sV);
      const uint32_t acc0 = acc_first ? 1u : 0u;
      static_for<0, C::BN / 16>([&](auto kk_c) {
        constexpr int kk = decltype(kk_c)::value;
        if (leader)
          tc_mma_ts_step<kk * 8, kk * 128>(tmem + C::O_COL, tmem + C::P_COL, b_lo, V_HI,
                                           C::IDESC_PV, kk > 0 ? 1u : acc0);
      });
      if (leader) tc_commit(&bars[X_PV_DONE]);
    };
    auto k_tile = [&](uint32_t kpos) { return sbase + C::OFF_K + (kpos % C::NK) * C::K_BYTES; };
    // QK^T of the tile at ring position kpos, once its K rows have landed
    auto qk = [&](uint32_t kpos) -> bool {
      if (!mbar_wait(&k_full[kpos % C::NK], (kpos / C::NK) & 1u, abort_flag, p.wait_ns))
        return false;
      fence_proxy_async_smem();  // cp.async (generic proxy) -> tcgen05.mma reads
      tc_fence_after();
      issue_s(k_tile(kpos));
      return true;
    };
    auto s_free = [&]() -> bool {
      if (!mbar_wait(&bars[X_S_FREE], f_cnt & 1u, abort_flag, p.wait_ns)) return false;
      ++f_cnt;
      tc_fence_after();
      return true;
    };
    for (uint32_t uc = 0; ok && !*abort_flag; ++uc) {
      const WorkUnit w = pair_take(bars, s_rec, uc, abort_flag, p.wait_ns, ok);
      if (w.n_tiles < 0) break;
      const int nt = w.n_tiles;
      if (nt == 0) continue;
      if constexpr (SG) {
        // Decode of at most 32 rows: only TMEM lanes 0-31 matter, and this
        // warp (lanes 0-31) writes the unit's Q itself.  Every QK^T of the
        // previous unit has landed: this warp waited for its last P, which
        // the softmax wrote after it saw the last S.  Lanes 32-127 keep
        // whatever they hold; their rows are never read.
        const bool vq = lane < w.n_tok * G;
        const int64_t oq = (int64_t)(w.q_tok0 + lane / G) * p.hq + w.kvh * G + lane % G;
        const uint4 *qrow = reinterpret_cast<const uint4 *>(p.q + oq * C::LQ);
        static_for<0, 3>([&](auto h_c) {  // loads of 16, 16 and 4 chunks
          constexpr int h = decltype(h_c)::value;
          constexpr int c0 = 2 * h, nc = h < 2 ? 2 : 1;  // 32-column groups
          uint32_t v[nc][32];
#pragma unroll
          for (int c = 0; c < nc; ++c) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int k = 8 * (c0 + c) + i;  // 16-byte chunk: 32 value, then 4 rope
              const int q0 = k < C::DV / 8 ? dv0 / 8 + k : dr0 / 8 + (k - C::DV / 8);
              const uint4 x = vq && k < (C::DV + C::DR) / 8 ? __ldg(qrow + q0)
                                                            : make_uint4(0, 0, 0, 0);
              v[c][4 * i + 0] = x.x;
              v[c][4 * i + 1] = x.y;
              v[c][4 * i + 2] = x.z;
              v[c][4 * i + 3] = x.w;
            }
          }
#pragma unroll
          for (int c = 0; c < nc; ++c) tmem_st32(tmem + C::Q_COL + (c0 + c) * 32, v[c]);
        });
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        tc_fence_after();
      } else {
        if (!mbar_wait(&bars[X_Q_FULL], q_cnt & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
        ++q_cnt;
        tc_fence_after();
      }
      const uint32_t k0 = kc;
      // S(0); S(1) once S(0) is read
      if (!qk(k0) || !s_free() || (nt > 1 && !qk(k0 + 1))) { ok = false; break; }
      for (int j = 0; j < nt; ++j) {
        // S(j + 1) read: S(j + 2) may overwrite it
        if (j + 1 < nt && (!s_free() || (j + 2 < nt && !qk(k0 + j + 2)))) { ok = false; break; }
        if (!mbar_wait(&bars[X_P_FULL], p_cnt & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
        ++p_cnt;
        tc_fence_after();
        issue_pv(k_tile(k0 + j), j > 0);
        if (leader) tc_commit(&k_empty[(k0 + j) % C::NK]);
      }
      if (!ok) break;
      kc = k0 + nt;
      if (leader) tc_commit(&bars[X_O_DONE]);
    }
    if (!ok) abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
    if (leader) tc_commit(&bars[X_FINAL]);
    if (!mbar_wait_drain(&bars[X_FINAL], 0)) record_status(p.status, PKX_ETIMEOUT);
  } else if (warp == 5) {
    // ------------------------------------------------ row indices (one warp)
    uint32_t ic = 0;
    bool ok = true;
    for (uint32_t uc = 0; ok && !*abort_flag; ++uc) {
      const WorkUnit w = pair_take(bars, s_rec, uc, abort_flag, p.wait_ns, ok);
      if (w.n_tiles < 0) break;
      const int nt = w.n_tiles;
      if (nt == 0) continue;
      const int64_t kv_base = p.kv_indptr[w.b];
      const int64_t ext_base = MODE == kTwoStage ? p.qo_indptr[w.b] : 0;
      // the unit's query rows (G consecutive rows per token) into L2: this
      // warp runs tiles ahead of the softmax, which loads them into TMEM
      for (int t = lane; t < w.n_tok; t += 32)
        prefetch_l2_bulk(p.q + ((int64_t)(w.q_tok0 + t) * p.hq + w.kvh * G) * C::LQ,
                         (uint32_t)(G * C::LQ * 2));
      for (int j = 0; j < nt; ++j) {
        int kb, ke;
        tile_keys<C::BN>(w, j, kb, ke);
        const bool from_ext = MODE == kTwoStage && kb >= w.k_split;
        int rows[2];
        bool bad = false;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int jpos = kb + 2 * lane + i;
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
        *reinterpret_cast<int2 *>(smem + C::OFF_I + is * C::I_BYTES + lane * 8) =
            make_int2(rows[0], rows[1]);
        mbar_arrive(&i_full[is]);
        ++ic;
      }
    }
    if (!ok) abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
  } else if (warp < C::COPY_WARP0 + C::COPY_THREADS / 32) {
    // ------------------------------------------------ K-row copies (4 warps)
    // Thread ct copies chunk ct % 8 of each of this rank's four value atoms,
    // and of its rope dims if ct % 8 < 4, for keys ct / 8 + 16 i (i < 4): the
    // swizzle term (chunk ^ key % 8) is fixed per thread, and a warp
    // instruction reads four rows' 128-byte segments.
    const int ct = tid - C::COPY_WARP0 * 32;
    const int ch = ct & 7, key0 = ct >> 3;
    const uint32_t dthr = (uint32_t)key0 * 128u + ((uint32_t)(ch ^ (key0 & 7)) << 4);
    uint32_t kc = 0, ic = 0;
    bool ok = true;
    if constexpr (FMT == 0) {
      for (uint32_t uc = 0; ok && !*abort_flag; ++uc) {
        const WorkUnit w = pair_take(bars, s_rec, uc, abort_flag, p.wait_ns, ok);
        if (w.n_tiles < 0) break;
        const int nt = w.n_tiles;
        if (nt == 0) continue;
        const bf16 *kp = p.k_pool + (int64_t)w.kvh * p.kb_sh + dv0 + ch * 8;
        const bf16 *kx = p.k_ext + (int64_t)w.kvh * p.ke_sh + dv0 + ch * 8;
        for (int j = 0; j < nt; ++j) {
          int kb, ke;
          tile_keys<C::BN>(w, j, kb, ke);
          const bool from_ext = MODE == kTwoStage && kb >= w.k_split;
          const int is = ic % C::NI;
          if (!mbar_wait(&i_full[is], (ic / C::NI) & 1u, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          const int *ring = reinterpret_cast<const int *>(smem + C::OFF_I + is * C::I_BYTES);
          int rows[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) rows[i] = ring[key0 + 16 * i];
          mbar_arrive(&i_empty[is]);
          ++ic;
          const int ks = kc % C::NK;
          if (kc >= (uint32_t)C::NK &&
              !mbar_wait(&k_empty[ks], ((kc / C::NK) - 1) & 1u, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          const bf16 *base = from_ext ? kx : kp;
          const int64_t st = from_ext ? p.ke_st : p.kb_ss;
          const uint32_t sK = sbase + C::OFF_K + ks * C::K_BYTES + dthr;
          static_for<0, 4>([&](auto i_c) {
            constexpr int i = decltype(i_c)::value;
            const int row = rows[i];
            const bf16 *src = base + (int64_t)max(row, 0) * st;
            const uint32_t bytes = row >= 0 ? 16u : 0u;
            static_for<0, 4>([&](auto a_c) {
              constexpr int a = decltype(a_c)::value;
              cp_async_16_at<a * C::BN * 128 + i * 16 * 128, a * 128>(sK, src, bytes);
            });
            // the rope dims dr0 + 8 ch (value dims start at dv0 + 8 ch)
            if (ch < C::DR / 8)
              cp_async_16_at<4 * C::BN * 128 + i * 16 * 128, 0>(sK, src + (dr0 - dv0), bytes);
          });
          cp_async_arrive_noinc(&k_full[ks]);
          ++kc;
        }
      }
    } else if constexpr (C::NRAW > 0) {
      // fp8 pool, decode of at most 32 rows: tile t's codes go to this
      // thread's raw slot t % NRAW (8 bytes per key, atom and chunk, at
      // offsets fixed per thread), and tile t is converted into its stage
      // once tile t + NRAW - 1 is issued: the stage is taken (k_empty) only
      // then.  A unit's last tiles are converted before the next unit is
      // taken: its claim may wait for this unit's products, which wait for
      // these tiles.  One cp.async group per issued tile.
      static_assert(MODE == kDecode, "the raw ring serves decode (no extend rows)");
      const uint32_t rthr = (uint32_t)key0 * 64u + (uint32_t)ch * 8u;        // value atoms
      const uint32_t rthr_r = (uint32_t)key0 * 32u + (uint32_t)ch * 8u;      // rope rows
      constexpr uint32_t RAW_ROPE = 4u * C::BN * 64u;
      uint32_t issued = 0, conv = 0;
      int rows[4];
      auto convert = [&](bool drain) -> bool {
        const int ks = conv % C::NK;
        if (conv >= (uint32_t)C::NK &&
            !mbar_wait(&k_empty[ks], ((conv / C::NK) - 1) & 1u, abort_flag, p.wait_ns))
          return false;
        // tile conv's group: NRAW - 1 groups were issued after it, or fewer
        // while draining
        if (drain) cp_async_wait_group<0>();
        else cp_async_wait_group<C::NRAW - 1>();
        const uint32_t sR = sbase + C::OFF_RAW + (conv % C::NRAW) * C::RAW_BYTES;
        const uint32_t sK = sbase + C::OFF_K + ks * C::K_BYTES + dthr;
        static_for<0, 4>([&](auto i_c) {
          constexpr int i = decltype(i_c)::value;
          static_for<0, 4>([&](auto a_c) {
            constexpr int a = decltype(a_c)::value;
            st_shared_u4(sK + a * C::BN * 128 + i * 16 * 128,
                         fp8x8_to_bf16x8<FMT>(ld_shared_u2(sR + rthr + a * (C::BN * 64) + i * (16 * 64))));
          });
          if (ch < C::DR / 8)
            st_shared_u4(sK + 4 * C::BN * 128 + i * 16 * 128,
                         fp8x8_to_bf16x8<FMT>(ld_shared_u2(sR + RAW_ROPE + rthr_r + i * (16 * 32))));
        });
        fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
        mbar_arrive(&k_full[ks]);
        ++conv;
        return true;
      };
      for (uint32_t uc = 0; ok && !*abort_flag; ++uc) {
        const WorkUnit w = pair_take(bars, s_rec, uc, abort_flag, p.wait_ns, ok);
        if (w.n_tiles < 0) break;
        const int nt = w.n_tiles;
        if (nt == 0) continue;
        const uint8_t *kp8 =
            reinterpret_cast<const uint8_t *>(p.k_pool) + (int64_t)w.kvh * p.kb_sh + dv0 + ch * 8;
        for (int j = 0; j < nt && ok; ++j) {
          const int is = ic % C::NI;
          if (!mbar_wait(&i_full[is], (ic / C::NI) & 1u, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          const int *ring = reinterpret_cast<const int *>(smem + C::OFF_I + is * C::I_BYTES);
#pragma unroll
          for (int i = 0; i < 4; ++i) rows[i] = ring[key0 + 16 * i];
          mbar_arrive(&i_empty[is]);
          ++ic;
          // this thread converted tile issued - NRAW (the slot's last tile)
          // before it got here, in program order
          const uint32_t sR = sbase + C::OFF_RAW + (issued % C::NRAW) * C::RAW_BYTES;
          static_for<0, 4>([&](auto i_c) {
            constexpr int i = decltype(i_c)::value;
            const int row = rows[i];
            const uint8_t *src = kp8 + (int64_t)max(row, 0) * p.kb_ss;
            const uint32_t bytes = row >= 0 ? 8u : 0u;
            static_for<0, 4>([&](auto a_c) {
              constexpr int a = decltype(a_c)::value;
              cp_async_8_at<a * C::BN * 64 + i * 16 * 64>(sR + rthr, src + a * 64, bytes);
            });
            if (ch < C::DR / 8)
              cp_async_8_at<RAW_ROPE + i * 16 * 32>(sR + rthr_r, src + (dr0 - dv0), bytes);
          });
          cp_async_commit();
          ++issued;
          if (issued - conv > (uint32_t)(C::NRAW - 1) && !convert(false)) ok = false;
        }
        while (ok && conv < issued)
          if (!convert(true)) ok = false;
      }
    } else {
      // fp8 pool.  A pool tile's codes are copied 8 bytes per (thread, key,
      // chunk) into the first half of the 16-byte chunk the same thread
      // later writes, and converted there in place to bf16 once they have
      // landed, so no thread overwrites another's codes.  Tile j is
      // converted (and its stage marked full) after tile j + 1's copies are
      // issued; extend tiles of the two-stage form are bf16 rows and take
      // the plain copy.  One cp.async group per issued tile.
      int rows[4];
      auto fetch = [&]() -> bool {
        const int is = ic % C::NI;
        if (!mbar_wait(&i_full[is], (ic / C::NI) & 1u, abort_flag, p.wait_ns)) return false;
        const int *ring = reinterpret_cast<const int *>(smem + C::OFF_I + is * C::I_BYTES);
#pragma unroll
        for (int i = 0; i < 4; ++i) rows[i] = ring[key0 + 16 * i];
        mbar_arrive(&i_empty[is]);
        ++ic;
        return true;
      };
      for (uint32_t uc = 0; ok && !*abort_flag; ++uc) {
        const WorkUnit w = pair_take(bars, s_rec, uc, abort_flag, p.wait_ns, ok);
        if (w.n_tiles < 0) break;
        const int nt = w.n_tiles;
        if (nt == 0) continue;
        const uint8_t *kp8 =
            reinterpret_cast<const uint8_t *>(p.k_pool) + (int64_t)w.kvh * p.kb_sh + dv0 + ch * 8;
        const bf16 *kx = p.k_ext + (int64_t)w.kvh * p.ke_sh + dv0 + ch * 8;
        auto tile_ext = [&](int j) {
          int kb, ke;
          tile_keys<C::BN>(w, j, kb, ke);
          return MODE == kTwoStage && kb >= w.k_split;
        };
        // tile j's rows into the next stage; returns the stage, or -1
        auto issue = [&](bool from_ext) -> int {
          const int ks = kc % C::NK;
          if (kc >= (uint32_t)C::NK &&
              !mbar_wait(&k_empty[ks], ((kc / C::NK) - 1) & 1u, abort_flag, p.wait_ns))
            return -1;
          const uint32_t sK = sbase + C::OFF_K + ks * C::K_BYTES + dthr;
          if (from_ext) {
            static_for<0, 4>([&](auto i_c) {
              constexpr int i = decltype(i_c)::value;
              const int row = rows[i];
              const bf16 *src = kx + (int64_t)max(row, 0) * p.ke_st;
              const uint32_t bytes = row >= 0 ? 16u : 0u;
              static_for<0, 4>([&](auto a_c) {
                constexpr int a = decltype(a_c)::value;
                cp_async_16_at<a * C::BN * 128 + i * 16 * 128, a * 128>(sK, src, bytes);
              });
              if (ch < C::DR / 8)
                cp_async_16_at<4 * C::BN * 128 + i * 16 * 128, 0>(sK, src + (dr0 - dv0), bytes);
            });
            cp_async_arrive_noinc(&k_full[ks]);
          } else {
            static_for<0, 4>([&](auto i_c) {
              constexpr int i = decltype(i_c)::value;
              const int row = rows[i];
              const uint8_t *src = kp8 + (int64_t)max(row, 0) * p.kb_ss;
              const uint32_t bytes = row >= 0 ? 8u : 0u;
              static_for<0, 4>([&](auto a_c) {
                constexpr int a = decltype(a_c)::value;
                cp_async_8_at<a * C::BN * 128 + i * 16 * 128>(sK, src + a * 64, bytes);
              });
              if (ch < C::DR / 8)
                cp_async_8_at<4 * C::BN * 128 + i * 16 * 128>(sK, src + (dr0 - dv0), bytes);
            });
          }
          cp_async_commit();
          ++kc;
          return ks;
        };
        // the thread's codes of a stage to bf16, in place
        auto convert = [&](int ks) {
          const uint32_t sK = sbase + C::OFF_K + ks * C::K_BYTES + dthr;
          static_for<0, 4>([&](auto i_c) {
            constexpr int i = decltype(i_c)::value;
            static_for<0, 4>([&](auto a_c) {
              constexpr int a = decltype(a_c)::value;
              const uint32_t at = sK + a * C::BN * 128 + i * 16 * 128;
              st_shared_u4(at, fp8x8_to_bf16x8<FMT>(ld_shared_u2(at)));
            });
            if (ch < C::DR / 8) {
              const uint32_t at = sK + 4 * C::BN * 128 + i * 16 * 128;
              st_shared_u4(at, fp8x8_to_bf16x8<FMT>(ld_shared_u2(at)));
            }
          });
          fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
        };
        bool ext_j = tile_ext(0);
        int st_j = fetch() ? issue(ext_j) : -1;
        if (st_j < 0) {
          ok = false;
          break;
        }
        for (int j = 0; j < nt; ++j) {
          const bool more = j + 1 < nt;
          bool ext_n = false;
          int st_n = 0;
          if (more) {
            ext_n = tile_ext(j + 1);
            st_n = fetch() ? issue(ext_n) : -1;
            if (st_n < 0) {
              ok = false;
              break;
            }
          }
          if (!ext_j) {
            // groups issued after tile j's: tile j + 1's, if there is one
            if (more) cp_async_wait_group<1>();
            else cp_async_wait_group<0>();
            convert(st_j);
            mbar_arrive(&k_full[st_j]);
          }
          ext_j = ext_n;
          st_j = st_n;
        }
      }
    }
    if (!ok) abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
    cp_async_wait_all();
  } else if (warp == 10) {
    // ------------------------------------- unit claims (one thread of rank 0)
    // Claims the next unit of the cost order and writes it into the next
    // slot of both ranks' rings once all consuming warps of both ranks have
    // released the slot's previous unit; -1 (after the last unit, or after
    // an abort) ends every consumer.
    if (rank == 0 && lane == 0) {
      const uint32_t rec_peer = cluster_addr(smem_u32(&s_rec[0]), 1);
      static_assert(sizeof(WorkUnit) % 16 == 0, "records move as 16-byte chunks");
      constexpr int RCH = (int)(sizeof(WorkUnit) / 16);
      const uint32_t full_peer = cluster_addr(smem_u32(&bars[X_U_FULL]), 1);
      static_assert(C::CLAIM_AHEAD >= 1 && C::CLAIM_AHEAD <= C::URING, "claim lag");
      for (uint32_t uc = 0;; ++uc) {
        const int slot = uc % C::URING;
        // every warp of both ranks took unit uc - CLAIM_AHEAD, and so the
        // slot's previous unit uc - URING
        if (uc >= (uint32_t)C::CLAIM_AHEAD) {
          const uint32_t e = uc - C::CLAIM_AHEAD;
          if (!mbar_wait_cluster(&bars[X_U_EMPTY + e % C::URING], (e / C::URING) & 1u, abort_flag,
                                 p.wait_ns)) {
            abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
            break;
          }
        }
        int u = -1;
        if (!*abort_flag) {
          if (p.part_first) {  // stream partition: this pair's share, in order
            const int pair = (int)(blockIdx.x >> 1);
            const int pos = p.part_first[pair] + (int)uc;
            if (pos < p.part_first[pair + 1]) u = p.uorder[pos];
          } else {
            const int pos = atomicAdd(p.next_unit, 1);
            if (pos < n_units) u = p.uorder[pos];
          }
        }
        // the record (or the end marker), here and in rank 1
        WorkUnit rec;
        if (u >= 0) {
          rec = p.units[u];
        } else {
          rec = WorkUnit{};
          rec.n_tiles = -1;
        }
        const uint4 *src = reinterpret_cast<const uint4 *>(&rec);
        uint4 *dst = reinterpret_cast<uint4 *>(&s_rec[slot]);
#pragma unroll
        for (int i = 0; i < RCH; ++i) {
          dst[i] = src[i];
          st_cluster_u4(rec_peer + (uint32_t)(slot * (int)sizeof(WorkUnit) + 16 * i), src[i]);
        }
        mbar_arrive(&bars[X_U_FULL + slot]);
        mbar_arrive_cluster(full_peer + (uint32_t)slot * 8u);
        if (u < 0) break;
      }
    } else if (rank == 1 && lane == 0) {
      // Each completed phase of this CTA's U_EMPTY (every consuming warp
      // read the slot) becomes one arrival on rank 0's, up to the end
      // marker.  The record is intact until this arrival lets the claimer
      // reuse the slot.
      const uint32_t empty_peer = cluster_addr(smem_u32(&bars[X_U_EMPTY]), 0);
      for (uint32_t uc = 0;; ++uc) {
        const int slot = uc % C::URING;
        if (!mbar_wait(&bars[X_U_EMPTY + slot], (uc / C::URING) & 1u, abort_flag, p.wait_ns)) {
          abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
          break;
        }
        const bool end = s_rec[slot].n_tiles < 0;
        mbar_arrive_cluster(empty_peer + (uint32_t)slot * 8u);
        if (end) break;
      }
    }
  }

  tc_fence_before();
  // neither CTA leaves while the other may still store into its receive
  // buffer or arrive on its barriers
  cluster_sync();
  if (warp == 4) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}
