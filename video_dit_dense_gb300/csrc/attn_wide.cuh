// Attention kernel for head dim 256 with double-buffered scores (included by
// attn_fwd.cu inside its anonymous namespace; uses its helpers).
//
// One 128-row query tile per CTA.  At head dim 256 a 128-key tile costs 2048
// tensor cycles (S = Q K^T and O += P V, 1024 each) against about 1500 SM
// cycles of softmax, so the kernel is tensor-bound if the softmax of tile j
// overlaps the products of its neighbours.  Tensor memory (512 columns):
//   S_0, S_1   [0, 128), [128, 256)   scores of even / odd key tiles (fp32);
//                                     P of a tile (bf16 pairs) is written over
//                                     the first 64 columns of its score buffer
//   O          [256, 512)             output accumulator (fp32, 256 channels)
// Q (128 rows x 256 channels, 64 KiB) sits in shared memory; K and V stream
// through a ring of NSTAGE half-tile stages (128 keys x 128 channels, 32 KiB:
// two 64-channel swizzle columns), consumed by 8 MMAs each.
//
// MMA thread (warp 5):
//   prologue: S_0 = Q K_0^T; S_1 = Q K_1^T
//   for j = 0, 1, ...: wait P_j; O[:, 0:128] += P_j V_j[:, 0:128];
//     O[:, 128:256] += P_j V_j[:, 128:256]; commit; then, once that product
//     has completed (P_j sits in S_{j mod 2}, and the tensor pipe orders only
//     MMAs that share an accumulator), S_{j mod 2} = Q K_{j+2}^T; commit.
// The softmax of tile j + 1 runs on the other buffer meanwhile.  s_full and
// p_ready are barriers per buffer, so a waiter can never be passed by a
// completion two phases ahead; the epilogue waits on the MMA thread's
// one-shot drain barrier, not on a parity of pv_done (with two buffers the
// product of tile n - 2 can still run when P_{n-1} is stored).
//
//   warps 0-3  softmax (thread t = query row t = TMEM lane t)
//   warp 4     TMA producer: Q, then K_0, K_1, then V_j, K_{j+2} (half tiles)
//   warp 5     MMA thread (allocates TMEM)
//   warp 6     zeroes the V rows past kv_len in the tile that straddles kv_len
//   warp 7     idle
template <int NSTAGE>
struct WideCfg {
  static constexpr int D = 256;
  static constexpr int kHalfBytes = kBlockN * 128 * 2;  // 32 KiB: 128 keys x 128 channels
  static constexpr int kChunk = kBlockN * 128;          // 16 KiB: one 64-channel swizzle column
  static constexpr int kQBytes = kBlockM * D * 2;       // 64 KiB
  static constexpr int kSmemKV = NSTAGE * kHalfBytes;
  // q_full, kv_full[NSTAGE], kv_empty[NSTAGE], s_full[2], p_ready[2], pv_done, drain, v_clean, o_staged
  static constexpr int kNumBars = 1 + 2 * NSTAGE + 2 + 2 + 4;
  static constexpr int kSmemBytes = 1024 + kQBytes + kSmemKV + kNumBars * 8 + 16;
  static constexpr int kThreads = 256;
  static constexpr int kProducerWarp = 4;
  static constexpr int kMmaWarp = 5;
  static constexpr int kPadWarp = 6;
  static constexpr int kColO = 256;
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kBlockN, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, false, true);  // one 128-channel half of O
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(NSTAGE >= 4, "K_0 and K_1 (two halves each) resident before the first P V");
};

template <int NSTAGE>
__global__ void __launch_bounds__(256, 1) attn_wide_kernel(const __grid_constant__ AttnArgs a) {
  using C = WideCfg<NSTAGE>;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sKV = base + C::kQBytes;
  const uint32_t bars = sKV + C::kSmemKV;
  const uint32_t bar_q_full = bars;
  auto bar_kv_full = [&](int s) { return bars + 8u * (1 + s); };
  auto bar_kv_empty = [&](int s) { return bars + 8u * (1 + NSTAGE + s); };
  auto bar_s_full = [&](int bf) { return bars + 8u * (1 + 2 * NSTAGE + bf); };
  auto bar_p_ready = [&](int bf) { return bars + 8u * (3 + 2 * NSTAGE + bf); };
  const uint32_t bar_pv_done = bars + 8u * (5 + 2 * NSTAGE);
  const uint32_t bar_drain = bars + 8u * (6 + 2 * NSTAGE);
  const uint32_t bar_v_clean = bars + 8u * (7 + 2 * NSTAGE);
  const uint32_t bar_o_staged = bars + 8u * (8 + 2 * NSTAGE);  // o rows staged for the TMA store (128 softmax)
  uint8_t* gmisc = gbase + C::kQBytes + C::kSmemKV + C::kNumBars * 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gmisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gmisc + 4);
  const uint32_t pad_issued = smem_u32(gmisc + 8);  // 1 once V of the tile straddling kv_len is requested

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work unit: (b, h, 128-row query tile), longest (causal) first --------
  const int b = blockIdx.z;
  const int h = blockIdx.y;
  const int kvh = h / (a.Hq / a.Hkv);
  const int qb = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);
  const int q0 = qb * kBlockM;
  int kv_lim = a.Sk;
  if (a.kv_len) kv_lim = min(kv_lim, max(a.kv_len[b], 0));
  const bool causal = a.causal || (a.causal_b && a.causal_b[b]);
  int q_lim = a.Sq;
  if (a.q_len) q_lim = min(q_lim, max(a.q_len[b], 0));
  int kv_end = kv_lim;
  if (causal) kv_end = min(kv_end, q0 + kBlockM);
  const int n_tiles = (q0 < q_lim && kv_end > 0) ? (kv_end + kBlockN - 1) / kBlockN : 0;
  // Iteration j visits key tile (j + rot) mod n_tiles (spreads the CTAs that
  // run at the same time over different K/V lines).
  const int rot = n_tiles > 0 ? static_cast<int>(blockIdx.x) % n_tiles : 0;
  auto tile_of = [rot, n_tiles](int j) { return j + rot < n_tiles ? j + rot : j + rot - n_tiles; };
  // Half-tile load order: K_0, K_1 (two halves each), then V_j, K_{j+2}.  A
  // tile's two halves are consecutive loads; these give the first one's index.
  const int n_lead = min(n_tiles, 2);
  auto ld_v = [n_tiles, n_lead](int j) { return 2 * n_lead + 2 * j + 2 * max(0, min(j, n_tiles - 2)); };
  auto ld_k = [&](int j) { return j < 2 ? 2 * j : ld_v(j - 2) + 2; };
  auto stage_of = [](int pos) { return pos % NSTAGE; };
  auto phase_of = [](int pos) { return static_cast<uint32_t>((pos / NSTAGE) & 1); };
  auto bpar = [](int j) { return static_cast<uint32_t>((j >> 1) & 1); };  // j-th use of buffer j mod 2
  int j_pad = -1;  // iteration of the key tile that straddles kv_len, or -1
  if (n_tiles > 0 && kv_lim < a.Sk && (kv_lim % kBlockN) != 0) {
    const int tb = kv_lim / kBlockN;
    if (tb < n_tiles) j_pad = tb >= rot ? tb - rot : tb - rot + n_tiles;
  }

  WaitCtl ctl{abort_flag, &g_status_word, a.wait_limit_ns, static_cast<int>(H3ATTN_ERR_TIMEOUT)};

  if (warp == C::kProducerWarp && lane == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    mbar_init(bar_q_full, 1);
    for (int bf = 0; bf < 2; ++bf) {
      mbar_init(bar_s_full(bf), 1);
      mbar_init(bar_p_ready(bf), 128);
    }
    mbar_init(bar_pv_done, 1);
    mbar_init(bar_drain, 1);
    mbar_init(bar_v_clean, 1);
    mbar_init(bar_o_staged, 128);
    *abort_flag = 0u;
    *reinterpret_cast<volatile uint32_t*>(gmisc + 8) = 0u;  // pad_issued
    fence_barrier_init();
    if (n_tiles > 0 && !a.debug_skip_producer) {
      // Q and the halves of K_0, K_1 (ring positions 0 .. 2 n_lead - 1, first
      // use of their stages) go out before the block-wide set-up completes
      mbar_arrive_expect_tx(bar_q_full, C::kQBytes);
      for (int c = 0; c < D / 64; ++c) tma_load_4d(sQ + c * C::kChunk, &a.tm_q, bar_q_full, c * 64, h, q0, b);
      for (int p = 0; p < 2 * n_lead; ++p) {
        mbar_arrive_expect_tx(bar_kv_full(p), C::kHalfBytes);
        for (int c = 0; c < 2; ++c)
          tma_load_4d(sKV + p * C::kHalfBytes + c * C::kChunk, &a.tm_k, bar_kv_full(p), (2 * (p & 1) + c) * 64, kvh,
                      tile_of(p >> 1) * kBlockN, b);
      }
    }
    prefetch_tmap(&a.tm_v);
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::kProducerWarp) {
    // ======================= TMA producer ==================================
    if (lane == 0 && n_tiles > 0 && !a.debug_skip_producer) {
      int pos = 2 * n_lead;  // Q, K_0 and K_1 went out during the set-up
      bool ok = true;
      auto load = [&](int kind, int j) {  // both halves of K_j (kind 0) or V_j (kind 1)
        for (int half = 0; ok && half < 2; ++half) {
          const int s = stage_of(pos);
          if (!(ok = mbar_wait<kWaitParked>(bar_kv_empty(s), phase_of(pos) ^ 1u, ctl))) return;
          mbar_arrive_expect_tx(bar_kv_full(s), C::kHalfBytes);
          const CUtensorMap* m = kind == 0 ? &a.tm_k : &a.tm_v;
          for (int c = 0; c < 2; ++c)
            tma_load_4d(sKV + s * C::kHalfBytes + c * C::kChunk, m, bar_kv_full(s), (2 * half + c) * 64, kvh,
                        tile_of(j) * kBlockN, b);
          ++pos;
        }
        if (ok && kind == 1 && j == j_pad) st_release_cta(pad_issued, 1u);
      };
      for (int j = 0; ok && j < n_tiles; ++j) {
        load(1, j);
        if (ok && j + 2 < n_tiles) load(0, j + 2);
      }
      // Drain: every issued copy has landed before the CTA can retire.
      mbar_wait_drain(bar_q_full, 0, a.wait_limit_ns);
      for (int i = pos > NSTAGE ? pos - NSTAGE : 0; i < pos; ++i)
        mbar_wait_drain(bar_kv_full(stage_of(i)), phase_of(i), a.wait_limit_ns);
    }
  } else if (warp == C::kMmaWarp) {
    // ======================= MMA thread ====================================
    if (lane == 0 && n_tiles > 0) {
      bool ok = mbar_wait<kWaitParked>(bar_q_full, 0, ctl);
      tc_fence_after();
      // S_{j mod 2} = Q K_j^T: 16 MMAs of 16 channels, 8 on each half of K_j
      auto issue_qk = [&](int j) -> bool {
        const uint32_t tS = tmem + (j & 1) * 128;
        for (int half = 0; half < 2; ++half) {
          const int pos = ld_k(j) + half, s = stage_of(pos);
          if (!mbar_wait<kWaitParked>(bar_kv_full(s), phase_of(pos), ctl)) return false;
          tc_fence_after();
          const uint32_t kb = sKV + s * C::kHalfBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ko = (kk >> 2) * C::kChunk + (kk & 3) * 32;
            const uint32_t qo = (2 * half + (kk >> 2)) * C::kChunk + (kk & 3) * 32;
            mma_ss(tS, sdesc_sw128(sQ + qo, 16, 1024), sdesc_sw128(kb + ko, 16, 1024), C::kIdescQK,
                   (half > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bar_kv_empty(s));
        }
        tc_commit(bar_s_full(j & 1));
        return true;
      };
      if (ok) ok = issue_qk(0);
      if (ok && n_tiles > 1) ok = issue_qk(1);
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (!(ok = mbar_wait<kWaitParked>(bar_p_ready(j & 1), bpar(j), ctl))) break;
        if (j == j_pad && !(ok = mbar_wait<kWaitParked>(bar_v_clean, 0, ctl))) break;  // padding rows zeroed
        // O[:, 128 half ...] += P_j V_j[:, 128 half ...]: A = P over S_{j mod 2}
        const uint32_t tP = tmem + (j & 1) * 128;
        for (int half = 0; half < 2; ++half) {
          const int pos = ld_v(j) + half, s = stage_of(pos);
          if (!(ok = mbar_wait<kWaitParked>(bar_kv_full(s), phase_of(pos), ctl))) break;
          tc_fence_after();
          const uint32_t vb = sKV + s * C::kHalfBytes;
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk)
            mma_ts(tmem + C::kColO + half * 128, tP + kk * 8, sdesc_sw128(vb + kk * 2048, C::kChunk, 1024),
                   C::kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
          tc_commit(bar_kv_empty(s));
        }
        if (!ok) break;
        tc_commit(bar_pv_done);
        if (j + 2 < n_tiles) {
          // the next scores of this buffer overwrite P_j: once O += P V has read it
          if (!(ok = mbar_wait<kWaitParked>(bar_pv_done, j & 1, ctl))) break;
          tc_fence_after();
          ok = issue_qk(j + 2);
        }
      }
      // Drain every MMA issued by this thread before tensor memory is freed;
      // the softmax's epilogue waits on the same one-shot barrier.
      tc_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0, a.wait_limit_ns);
    }
  } else if (warp == C::kPadWarp) {
    // ======================= padding rows of the tile straddling kv_len ====
    if (j_pad >= 0) {
      const int pos = ld_v(j_pad);
      const bool ok = __all_sync(0xFFFFFFFFu, count_wait_sleep(pad_issued, 1u, ctl) &&
                                                  mbar_wait<kWaitParked>(bar_kv_full(stage_of(pos)), phase_of(pos), ctl) &&
                                                  mbar_wait<kWaitParked>(bar_kv_full(stage_of(pos + 1)), phase_of(pos + 1), ctl));
      if (ok) {  // both halves of V landed; their stages are refilled only after O += P V of them
        zero_padding_rows<128>(sKV + stage_of(pos) * C::kHalfBytes, kv_lim % kBlockN, lane, 32);
        zero_padding_rows<128>(sKV + stage_of(pos + 1) * C::kHalfBytes, kv_lim % kBlockN, lane, 32);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_v_clean);
      }
    }
  } else if (warp < 4) {
    // ======================= softmax / correction / epilogue ===============
    const int wq = warp & 3;
    const int t = wq * 32 + lane;
    const int row = q0 + t;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tO = tmem + lane_off + C::kColO;
    const float sl = a.scale_log2;
    const int64_t bit_words = (a.Sk + 31) / 32;
    float m_ref = -INFINITY;  // running max in scaled (log2) units
    float l = 0.0f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      ok = mbar_wait<kWaitParked>(bar_s_full(j & 1), bpar(j), ctl);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + (j & 1) * 128;
      const int kbase = tile_of(j) * kBlockN;
      const bool need_mask = (kbase + kBlockN > kv_lim) || (causal && kbase + kBlockN - 1 > q0) || a.bits;
      // First pass against the running max as it stands; a tile row sum
      // <= 2^kRescaleThreshold proves no score exceeded it by more than the
      // rescale threshold.  Otherwise (and on a row's first tile) a second
      // pass takes the row max, rescales O and l if it grew past the
      // threshold, and recomputes.
      bool with_max = __any_sync(0xFFFFFFFFu, m_ref == -INFINITY);
      float tile_sum = 0.0f;
      uint32_t pr[2][32];
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
        float s[kBlockN];
#pragma unroll
        for (int c = 0; c < kBlockN; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
        if (need_mask) {
          int lim = kv_lim - kbase;
          if (causal) lim = min(lim, row + 1 - kbase);
          uint32_t wbits[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
          if (a.bits && row < a.Sq) {
            const uint32_t* br = a.bits + (static_cast<int64_t>(b) * a.Sq + row) * bit_words;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const int64_t wi = kbase / 32 + w;
              wbits[w] = wi < bit_words ? br[wi] : 0u;
            }
          }
#pragma unroll
          for (int c = 0; c < kBlockN; ++c)
            s[c] = ((c < lim) && ((wbits[c >> 5] >> (c & 31)) & 1u)) ? s[c] : -INFINITY;
        }
        if (with_max) {
          float mx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
          for (int c = 16; c < kBlockN; c += 16) {
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[c + 2 * i], s[c + 2 * i + 1]);
          }
          const float mt = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7]));
          const float mt_s = mt * sl;
          const bool grow = mt_s > m_ref + kRescaleThreshold;
          float alpha = 1.0f;
          if (grow) {
            alpha = ex2(m_ref - mt_s);  // m_ref = -inf gives 0
            l *= alpha;
            m_ref = mt_s;
          }
          if (j > 0 && __any_sync(0xFFFFFFFFu, grow)) {
            // O must hold every product of tiles < j before it is rescaled;
            // they are sequential, so the last one completing is enough.  The
            // parity wait is unambiguous: S_j exists, so the MMA thread has
            // seen tile j - 2's product complete, and tile j's waits for P_j.
            ok = mbar_wait<kWaitParked>(bar_pv_done, (j - 1) & 1, ctl);
            if (!__all_sync(0xFFFFFFFFu, ok)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
              tmem_ld_wait(o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st32(tO + c * 32, o);
            }
            tmem_st_wait();
          }
        }
        const float mu = (m_ref == -INFINITY) ? 0.0f : m_ref;
        float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < kBlockN; c += 2) {
          float t0, t1;
          ffma2(t0, t1, s[c], s[c + 1], sl, sl, -mu, -mu);
          const float p0 = ex2(t0);
          const float p1 = ex2(t1);
          const int a2 = ((c >> 1) & 3) * 2;
          fadd2(ls[a2], ls[a2 + 1], ls[a2], ls[a2 + 1], p0, p1);
          pr[c >> 6][(c >> 1) & 31] = pack_bf16x2(p0, p1);
        }
        tile_sum = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        if (with_max) break;
        with_max = __any_sync(0xFFFFFFFFu, !(tile_sum <= kFastPassSumLimit));
        if (!with_max) break;
      }
      if (!ok) break;
      l += tile_sum;
      // P over the first 64 columns of this tile's score buffer (read above)
      tmem_st32(tS, pr[0]);
      tmem_st32(tS + 32, pr[1]);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p_ready(j & 1));
    }
    // ---- epilogue: O / l -> bf16, once every product has completed ---------
    if (ok && n_tiles > 0) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait<kWaitParked>(bar_drain, 0, ctl));
      tc_fence_after();
    }
    if (ok) {
      // o = O / l as bf16, staged over Q in shared memory (every product has
      // completed) in the 128-byte swizzled layout of the o map's box, then
      // one TMA store of the tile; rows past Sq are not written.
      const bool zero_row = row >= q_lim || n_tiles == 0 || !(l > 0.0f);
      const float inv = zero_row ? 0.0f : 1.0f / l;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (n_tiles > 0) {
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait(o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        // channels [32c, 32c + 32): 16-byte units 4(c mod 2) .. +3 of row t in swizzle column c / 2
        const uint32_t rowp = sQ + (c >> 1) * C::kChunk + t * 128;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = zero_row ? 0u
                            : pack_bf16x2(__uint_as_float(o[v * 8 + 2 * e]) * inv,
                                          __uint_as_float(o[v * 8 + 2 * e + 1]) * inv);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                           rowp + ((((c & 1) * 4 + v) ^ (t & 7)) << 4)),
                       "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                       : "memory");
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar_o_staged);
      if (t == 0 && mbar_wait<kWaitParked>(bar_o_staged, 0, ctl)) {
        for (int c = 0; c < D / 64; ++c) tma_store_4d(&a.tm_o, sQ + c * C::kChunk, c * 64, h, q0, b);
        bulk_commit_group();
        bulk_wait_group_read0();  // the shared-memory source is read before the CTA retires
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int NSTAGE>
cudaError_t launch_wide(const AttnArgs& a, cudaStream_t stream) {
  using C = WideCfg<NSTAGE>;
  auto kern = attn_wide_kernel<NSTAGE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Sq + kBlockM - 1) / kBlockM, a.Hq, a.B);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}
