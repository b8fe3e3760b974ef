// mla_kernel.cuh -- extend / decode attention for the MLA head shape
// (Lq = 576 = 512 latent + 64 rope dims, Lv = 512, one KV head, V = the first
// 512 dims of each K row), included by attention.cu.
//
// The MLA layout (sglang cpu_graph_runner.py, qkv_proj_with_rope fake: V is a
// narrow view of K; extend_attention.py, _get_block_sizes_for_extend_attention:
// 576 = 512 + 64) makes the score a single 576-dim dot product, and V need not
// be loaded separately: the K tile in shared memory is also the V operand.
//
// TMEM holds 512 columns of 32 bits.  A 128-row tile of O over all 512 value
// dims would fill it, leaving no room for S, so each work unit produces one
// 128-dim slice of the value dims (w.dq) and recomputes S for it:
//   TMEM  [0, 288)   Q tile, bf16 pairs (A operand of QK^T, TMEM form)
//         [288, 320) P (bf16 pairs, 64 keys)
//         [320, 384) S (fp32)
//         [384, 512) O slice (fp32)
// The softmax releases S as soon as it holds the tile in registers, so QK^T
// of the next K tile runs while it computes P and while PV runs.
//   SMEM  three stages of a 64-key K tile (64 x 576 bf16, 128-byte swizzle,
//         nine 64-dim blocks) + a ring of resolved row indices.
// QK^T reads A = Q from TMEM and B = K from SMEM; PV reads A = P from TMEM and
// B = columns [128 dq, 128 dq + 128) of the same K tile, as an MN-major
// operand.  Warps: 0-3 softmax (one row per thread; they also write Q into
// TMEM), 4 MMA issue, 5 row indices, 6-11 K-row copies (cp.async).

template <int MODE>
struct MlaCfg {
  static constexpr int BM = kBlockM, BN = 64;
  static constexpr int LQ = 576, LV = 512, DVS = 128;  // value dims per unit
  static constexpr int NK = 3, NI = 4;
  static constexpr int K_BYTES = BN * LQ * 2;  // 73728
  static constexpr int I_BYTES = BN * 4;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_I = NK * K_BYTES;
  static constexpr int OFF_BAR = OFF_I + NI * I_BYTES;
  static constexpr int N_BARS = 16 + 2 * NK + 2 * NI;
  static constexpr int SMEM = OFF_BAR + N_BARS * 8 + 1024;
  static constexpr int TMEM_COLS = 512;
  static constexpr int Q_COL = 0, P_COL = 288, S_COL = 320, O_COL = 384;
  static constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, 0);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, DVS, 1);
  static constexpr int THREADS = 384;
  static constexpr int COPY_THREADS = 192;
  static_assert(SMEM <= 232448, "shared memory budget");
};

enum {
  M_Q_FULL = 0,
  M_S_FULL = 1,   // S landed
  M_P_FULL = 2,   // P written
  M_O_DONE = 3,   // last PV of a unit landed
  M_FINAL = 4,
  M_S_FREE = 5,   // S read into registers: the next QK^T may overwrite it
  M_PV_DONE = 6,  // one phase per PV: P and O are free again
  M_NEVER = 7,    // no thread ever arrives (the stall hook waits on it)
  M_U_FULL = 8,   // + unit ring slot
  M_U_EMPTY = 11, // + unit ring slot
  M_RING = 16
};

// MASK: a custom mask replaces the causal mask (own instantiation).
template <int MODE, bool MASK>
__global__ void __launch_bounds__(MlaCfg<MODE>::THREADS, 1) mla_kernel(const KParams p) {
  using C = MlaCfg<MODE>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_unit[kUnitRing];

  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *k_full = bars + M_RING;
  uint64_t *k_empty = k_full + C::NK;
  uint64_t *i_full = k_empty + C::NK;
  uint64_t *i_empty = i_full + C::NI;
  volatile int *abort_flag = &s_abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(&bars[M_Q_FULL], 128);
    mbar_init(&bars[M_S_FULL], 1);
    mbar_init(&bars[M_P_FULL], 4);  // one arrival per softmax warp
    mbar_init(&bars[M_O_DONE], 1);
    mbar_init(&bars[M_FINAL], 1);
    mbar_init(&bars[M_S_FREE], 4);  // one arrival per softmax warp
    mbar_init(&bars[M_PV_DONE], 1);
    mbar_init(&bars[M_NEVER], 1);
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(&bars[M_U_FULL + i], 1);
      mbar_init(&bars[M_U_EMPTY + i], 4 + 1 + C::COPY_THREADS / 32);
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
  __syncthreads();
  tc_fence_after();
  // the prologue above reads no global memory; the work list, indices and
  // Q come from the kernels before this one on the stream
  grid_dep_wait();
  grid_dep_launch();
  const uint32_t tmem = s_tmem;
  const int n_units = p.hdr->n_units;
  const int G = p.group;

  if (warp < 4) {
    // ------------------------------------------- Q -> TMEM, softmax, epilogue
    const int r = tid;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    uint32_t s_cnt = 0, o_cnt = 0;
    uint32_t pv_base = 0;  // PVs of earlier units (M_PV_DONE phases)
    bool ring_ok = true;
    // test hook: a wait that cannot succeed (see attn_kernel)
    if (p.stall && !mbar_wait(&bars[M_NEVER], 0, abort_flag, p.wait_ns))
      abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
    for (uint32_t uc = 0; !*abort_flag; ++uc) {
      const int u = ring_unit(&bars[M_U_FULL], &bars[M_U_EMPTY], s_unit, uc, abort_flag, true,
                              ring_ok, p.wait_ns);
      if (u < 0) {
        if (!ring_ok) abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
        break;
      }
      const WorkUnit w = p.units[p.uorder[u]];
      const int nt = w.n_tiles;
      const int rows_valid = w.n_tok * G;
      const bool valid = r < rows_valid;
      const bool warp_active = warp * 32 < rows_valid;
      const int t = r / G, g = r - (r / G) * G;
      const int qpos = w.qpos0 + t;
      const int qmax = w.qpos0 + w.n_tok - 1;
      const int64_t orow_idx = (int64_t)(w.q_tok0 + t) * p.hq + w.kvh * G + g;
      const int64_t prow_idx = (int64_t)w.slot * p.rows_per_slot + r;
      const int dv0 = w.dq * C::DVS;
      // custom mask rows: a byte per key of the sequence for each extend
      // token; mbase is the row of the unit's first token
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
            for (int c = 0; c < C::DVS; c += 8)
              *reinterpret_cast<uint4 *>(orow + c) = make_uint4(0, 0, 0, 0);
            if (p.lse && w.dq == 0) p.lse[orow_idx] = -INFINITY;
          } else {
            float *prow = p.po + prow_idx * C::LV + dv0;
            for (int c = 0; c < C::DVS; c += 4)
              *reinterpret_cast<float4 *>(prow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            if (w.dq == 0) p.plse[prow_idx] = -INFINITY;
          }
        }
        continue;
      }
      // Q row (576 bf16) into TMEM columns [0, 288) as bf16 pairs; rows past
      // the block get zeros.  The previous unit's MMAs have all completed
      // (its epilogue waited for them), so Q's columns are free.
      {
        const uint4 *qrow = reinterpret_cast<const uint4 *>(p.q + orow_idx * C::LQ);
#pragma unroll 1
        for (int c = 0; c < C::LQ / 64; ++c) {
          uint32_t v[32];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 x = valid ? __ldg(qrow + c * 8 + i) : make_uint4(0, 0, 0, 0);
            v[4 * i + 0] = x.x;
            v[4 * i + 1] = x.y;
            v[4 * i + 2] = x.z;
            v[4 * i + 3] = x.w;
          }
          tmem_st32(lane_base + C::Q_COL + c * 32, v);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars[M_Q_FULL]);
      }
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nt; ++j) {
        int kb, ke;
        tile_keys<C::BN>(w, j, kb, ke);
        // mask bits of this thread's row for keys kb + 32 q + bit (q < 2):
        // the warp's rows cover 32 / G tokens; all lanes read 32 consecutive
        // bytes of a token's row per load, a ballot packs them
        uint32_t mb[2] = {0u, 0u};
        if constexpr (MASK) {
          if (warp_active) {
            const int t_lo = (warp * 32) / G, t_hi = min((warp * 32 + 31) / G, w.n_tok - 1);
            for (int tc = t_lo; tc <= t_hi; tc += 4) {
              uint8_t by[4][2];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint8_t *rowp = mbase + (int64_t)(tc + u) * mstride;
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                  const int kpos = kb + 32 * q2 + lane;
                  by[u][q2] = (tc + u <= t_hi && kpos < ke) ? __ldg(rowp + kpos) : (uint8_t)0;
                }
              }
#pragma unroll
              for (int u = 0; u < 4; ++u) {
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                  const uint32_t word = __ballot_sync(0xffffffffu, by[u][q2] != 0);
                  if (t == tc + u) mb[q2] = word;
                }
              }
            }
          }
        }
        if (!mbar_wait(&bars[M_S_FULL], s_cnt & 1u, abort_flag, p.wait_ns)) {
          abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
          break;
        }
        ++s_cnt;
        tc_fence_after();
        float x[C::BN];
        if (warp_active) {
          uint32_t v0[32], v1[32];
          tmem_ld32(lane_base + C::S_COL + 0, v0);
          tmem_ld32(lane_base + C::S_COL + 32, v1);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            x[i] = __uint_as_float(v0[i]);
            x[32 + i] = __uint_as_float(v1[i]);
          }
        }
        // S is in registers: the next QK^T may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[M_S_FREE]);
        float alpha = 1.0f;
        bool o_needs = false;
        uint32_t pk[32];
        if (warp_active) {
          // Logits in the log2 domain are sc * x; a capped or masked tile
          // is first mapped into the log2 domain (sc = 1).
          float sc = p.scale_log2;
          if (p.use_cap) {
#pragma unroll
            for (int i = 0; i < C::BN; ++i) x[i] = p.cap_log2 * tanh_approx(x[i] * p.cap_pre);
            sc = 1.0f;
          }
          const bool need_mask = (ke - 1 > w.qpos0) || (ke - kb < C::BN) ||
                                 (p.window > 0 && kb < qmax - p.window);
          if constexpr (MASK) {
            // the custom mask replaces the causal term; the window stays; a
            // row that sees every key of the tile keeps the plain path
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
          // row max of sc * x: sc * max(x), or sc * min(x) for a negative sc
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
          const float nm = m == -INFINITY ? 0.f : -m;
          float l0 = 0.f, l1 = 0.f;
#pragma unroll
          for (int i = 0; i < C::BN; i += 2) {
            const float e0 = ex2_approx(fmaf(x[i], sc, nm));
            const float e1 = ex2_approx(fmaf(x[i + 1], sc, nm));
            l0 += e0;
            l1 += e1;
            pk[i / 2] = pack_bf16(e0, e1);
          }
          l += l0 + l1;
        }
        // P's columns and O are free once the previous tile's PV has landed.
        // Every warp waits, also one without rows: S of the next tile can
        // land before this tile's P, and a warp that ran ahead would arrive
        // on P_FULL twice in one phase.
        if (j > 0 && !mbar_wait(&bars[M_PV_DONE], (pv_base + j - 1) & 1u, abort_flag, p.wait_ns)) {
          abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
        }
        tc_fence_after();
        if (warp_active) {
          tmem_st32(lane_base + C::P_COL, pk);
          if (__any_sync(0xffffffffu, o_needs)) {
            const float a = o_needs ? alpha : 1.0f;
            uint32_t v[32];
#pragma unroll 1
            for (int c = 0; c < C::DVS / 32; ++c) {
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
        if (lane == 0) mbar_arrive(&bars[M_P_FULL]);
      }
      if (*abort_flag) break;
      if (!mbar_wait(&bars[M_O_DONE], o_cnt & 1u, abort_flag, p.wait_ns)) {
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
          // the head's sink joins the denominator (split rows: in the combine)
          const float s2 = __ldg(p.sinks + w.kvh * G + g) * 1.4426950408889634f;
          const float M = fmaxf(m, s2);
          const float a_m = m == -INFINITY ? 0.f : ex2_approx(m - M);
          const float lt = l * a_m + ex2_approx(s2 - M);
          inv = a_m / lt;
          lse_v = (M + __log2f(lt)) * 0.69314718055994531f;
        }
        uint32_t v[32];
#pragma unroll
        for (int c = 0; c < C::DVS / 32; ++c) {
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
        if (valid && w.dq == 0) {
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
    // ------------------------------------------------ MMA issue (one thread)
    // Per K tile j: S(j+1) = Q K(j+1)^T as soon as the softmax has read S(j),
    // then O += P(j) V(j) once P(j) is written.  Descriptors are formed once
    // per tile and stepped by constants.  The whole warp runs the loop (the
    // values stay warp-uniform); one elected lane issues.
    {
      const bool leader = elect_one();
      uint32_t q_cnt = 0, kc = 0, p_cnt = 0, f_cnt = 0;
      bool ok = true;
      constexpr uint32_t K_LO = sw128_desc_lo(0), K_HI = sw128_desc_hi(1024);
      constexpr uint32_t V_LO = sw128_desc_lo(C::BN * 128), V_HI = sw128_desc_hi(1024);
      auto issue_s = [&](uint32_t sK) {
        const uint32_t b_lo = K_LO | (sK >> 4);
        static_for<0, C::LQ / 16>([&](auto kk_c) {
          constexpr int kk = decltype(kk_c)::value;
          constexpr uint32_t bo = ((kk / 4) * (C::BN * 128) + (kk % 4) * 32) / 16;
          if (leader) tc_mma_ts_step<kk * 8, bo>(tmem + C::S_COL, tmem + C::Q_COL, b_lo, K_HI, C::IDESC_QK,
                                     kk > 0 ? 1u : 0u);
        });
        if (leader) tc_commit(&bars[M_S_FULL]);
      };
      auto issue_pv = [&](uint32_t sV, bool acc_first) {
        const uint32_t b_lo = V_LO | (sV >> 4);
        const uint32_t acc0 = acc_first ? 1u : 0u;
        static_for<0, C::BN / 16>([&](auto kk_c) {
          constexpr int kk = decltype(kk_c)::value;
          if (leader) tc_mma_ts_step<kk * 8, kk * 128>(tmem + C::O_COL, tmem + C::P_COL, b_lo, V_HI,
                                           C::IDESC_PV, kk > 0 ? 1u : acc0);
        });
        if (leader) tc_commit(&bars[M_PV_DONE]);
      };
      auto k_tile = [&](uint32_t kpos) { return sbase + C::OFF_K + (kpos % C::NK) * C::K_BYTES; };
      for (uint32_t uc = 0; ok && !*abort_flag; ++uc) {
        const int u = ring_unit(&bars[M_U_FULL], &bars[M_U_EMPTY], s_unit, uc, abort_flag, true,
                                ok, p.wait_ns);
        if (u < 0) break;
        const WorkUnit w = p.units[p.uorder[u]];
        const int nt = w.n_tiles;
        if (nt == 0) continue;
        if (!mbar_wait(&bars[M_Q_FULL], q_cnt & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
        ++q_cnt;
        tc_fence_after();
        const uint32_t k0 = kc;  // ring position of this unit's first K tile
        if (!mbar_wait(&k_full[k0 % C::NK], (k0 / C::NK) & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
        fence_proxy_async_smem();  // cp.async (generic proxy) -> tcgen05.mma reads
        tc_fence_after();
        issue_s(k_tile(k0));
        const uint32_t dv_off = (w.dq * (C::DVS / 64)) * (C::BN * 128);
        for (int j = 0; j < nt; ++j) {
          if (!mbar_wait(&bars[M_S_FREE], f_cnt & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
          ++f_cnt;
          tc_fence_after();
          if (j + 1 < nt) {
            const uint32_t kn = k0 + j + 1;
            if (!mbar_wait(&k_full[kn % C::NK], (kn / C::NK) & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
            fence_proxy_async_smem();
            tc_fence_after();
            issue_s(k_tile(kn));
          }
          if (!mbar_wait(&bars[M_P_FULL], p_cnt & 1u, abort_flag, p.wait_ns)) { ok = false; break; }
          ++p_cnt;
          tc_fence_after();
          issue_pv(k_tile(k0 + j) + dv_off, j > 0);
          if (leader) tc_commit(&k_empty[(k0 + j) % C::NK]);
        }
        if (!ok) break;
        kc = k0 + nt;
        if (leader) tc_commit(&bars[M_O_DONE]);
      }
      if (!ok) abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
      if (leader) tc_commit(&bars[M_FINAL]);
      if (!mbar_wait_drain(&bars[M_FINAL], 0)) record_status(p.status, PKX_ETIMEOUT);
    }
  } else if (warp == 5) {
    // ------------------------------------------------ row indices (one warp)
    uint32_t ic = 0;
    bool ok = true;
    for (uint32_t uc = 0; ok && !*abort_flag; ++uc) {
      // claim the next unit and hand it to the other warps
      int u = -1;
      if (lane == 0) {
        const int pos = atomicAdd(p.next_unit, 1);
        u = pos < n_units ? pos : -1;
      }
      u = __shfl_sync(0xffffffffu, u, 0);
      {
        const int slot = uc % kUnitRing;
        if (uc >= (uint32_t)kUnitRing &&
            !mbar_wait(&bars[M_U_EMPTY + slot], ((uc / kUnitRing) - 1) & 1u, abort_flag, p.wait_ns)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          s_unit[slot] = u;
          mbar_arrive(&bars[M_U_FULL + slot]);
        }
      }
      if (u < 0) break;
      const WorkUnit w = p.units[p.uorder[u]];
      const int nt = w.n_tiles;
      if (nt == 0) continue;
      const int64_t kv_base = p.kv_indptr[w.b];
      const int64_t ext_base = MODE == kTwoStage ? p.qo_indptr[w.b] : 0;
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
  } else {
    // ------------------------------------------------ K-row copies (6 warps)
    // Thread ct copies flat chunks c = ct + 192 i (key c / 72, 16-byte chunk
    // c % 72), so consecutive lanes read consecutive bytes of a row.  Since
    // 3 x 192 = 8 rows, steps i and i + 3 share the chunk and the key mod 8:
    // three destination bases cover all steps, the rest is a constant
    // offset of 1024 bytes per 3 steps.
    const int ct = tid - 6 * 32;
    constexpr int CPR = C::LQ / 8;  // 72 chunks of 16 bytes per row
    constexpr int NCH = C::BN * CPR / C::COPY_THREADS;  // 24 chunks per thread
    static_assert(C::BN * CPR % C::COPY_THREADS == 0 && 3 * C::COPY_THREADS == 8 * CPR &&
                      NCH % 3 == 0,
                  "copy steps repeat every 8 rows");
    int kq[3], cq[3];
    uint32_t dq[3];
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int c = ct + q * C::COPY_THREADS;
      kq[q] = c / CPR;
      cq[q] = c - kq[q] * CPR;
      dq[q] = (uint32_t)(cq[q] >> 3) * (C::BN * 128) + sw128_off(kq[q], cq[q] & 7);
    }
    uint32_t kc = 0, ic = 0;
    bool ok = true;
    for (uint32_t uc = 0; ok && !*abort_flag; ++uc) {
      const int u = ring_unit(&bars[M_U_FULL], &bars[M_U_EMPTY], s_unit, uc, abort_flag, true, ok, p.wait_ns);
      if (u < 0) break;
      const WorkUnit w = p.units[p.uorder[u]];
      const int nt = w.n_tiles;
      if (nt == 0) continue;
      const bf16 *kp = p.k_pool + (int64_t)w.kvh * p.kb_sh;
      const bf16 *kx = p.k_ext + (int64_t)w.kvh * p.ke_sh;
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
        ++ic;
        const int ks = kc % C::NK;
        if (kc >= (uint32_t)C::NK &&
            !mbar_wait(&k_empty[ks], ((kc / C::NK) - 1) & 1u, abort_flag, p.wait_ns)) {
          ok = false;
          break;
        }
        const bf16 *base = from_ext ? kx : kp;
        const int64_t st = from_ext ? p.ke_st : p.kb_ss;
        const uint32_t sK = sbase + C::OFF_K + ks * C::K_BYTES;
        static_for<0, NCH>([&](auto i_c) {
          constexpr int i = decltype(i_c)::value, q = i % 3, step = i / 3;
          const int row = ring[kq[q] + 8 * step];
          const bool v = row >= 0;
          cp_async_16_at<step * 1024, 0>(sK + dq[q], (v ? base + (int64_t)row * st : base) + cq[q] * 8,
                                         v ? 16u : 0u);
        });
        cp_async_arrive_noinc(&k_full[ks]);
        mbar_arrive(&i_empty[is]);
        ++kc;
      }
    }
    if (!ok) abort_cta(abort_flag, p.status, PKX_ETIMEOUT);
    cp_async_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}
