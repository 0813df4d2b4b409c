// Attention kernel with one 128-row query tile per CTA, two MMA-issuing
// threads and a separate P buffer (included by attn_fwd.cu inside its
// anonymous namespace; uses its helpers).
//
// Tensor memory (512 columns x 128 lanes):
//   S_0, S_1  [0,128), [128,256)     scores of even / odd key tiles (fp32)
//   P         [256, 320)             probabilities of the current tile (bf16 pairs)
//   O         [320, 320+D)           output accumulator (fp32)
//   Q         [320+D, 320+D+D/2)     this CTA's query rows (bf16 pairs), the A
//                                    operand of S = Q K^T
//
// Score tile S_j lives in buffer S_{j mod 2}.  Once P_j is ready, MMA thread
// p = j mod 2 issues the burst
//     O += P_j V_j;   S_{j+3} = Q K_{j+3}^T  into S_{(j+1) mod 2}
// (the second half waits until softmax j+1 has read S_{j+1} out of that
// buffer, which it does at the start of its turn).  The tensor pipe thus runs
// the product that frees P right away and computes scores three tiles ahead,
// so the softmax warpgroup, which handles the tiles in order, finds S_{j+1}
// ready when it finishes tile j and finds the P buffer free when it wants to
// write P_{j+1}.  Prologue: S_0 (thread 0), S_1 and S_2 (thread 1).
// Two issuing threads on two SM sub-partitions alternate these bursts: while
// one does its commits and barrier polls (slow when it shares a sub-partition
// with a busy softmax warp) the other keeps the tensor pipe fed.
//
// P has a single buffer, so softmax j writes P_j only after O += P_{j-1} V_{j-1}
// has completed; this also makes the O += P V products strictly sequential.
//
//   warps 0-3  softmax warpgroup, thread t = query row t = TMEM lane t
//   warp 4     TMA producer: K_0, K_1, K_2, then K_{j+3}, V_j for j = 0, 1, ...
//   warps 5-6  MMA issuers for even / odd key tiles (warp 5 allocates TMEM)
//   warp 7     padding: in the key tile that straddles kv_len, zeroes the V
//              rows past kv_len (they may hold anything; 0 * NaN in O += P V
//              would leak) before that tile's O += P V (barrier v_clean)
template <int D, int NSTAGE>
struct PipeCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kBlockM * D * 2;
  static constexpr int kChunkBytes = kBlockM * 128;
  static constexpr int kSmemKV = NSTAGE * kTileBytes;
  // q_full, kv_full[NSTAGE], kv_empty[NSTAGE], s_full[2], s_read[2], p_ready[2], pv_done[2], drain[2],
  // v_clean, o_staged
  static constexpr int kNumBars = 1 + 2 * NSTAGE + 12;
  static constexpr int kSmemBytes = 1024 + kSmemKV + kNumBars * 8 + 16;
  static constexpr int kThreads = 256;
  static constexpr int kProducerWarp = 4;
  static constexpr int kMmaWarp = 5;  // and kMmaWarp + 1
  static constexpr int kColP = 256;
  static constexpr int kColO = 320;
  static constexpr int kColQ = kColO + D;
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kBlockN, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
  static_assert(kColQ + D / 2 <= static_cast<int>(kTmemCols), "tensor memory budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(NSTAGE >= 4, "K_{j+3}, V_j and the other thread's pair resident together");
};

// WIN: chunked-window tile lists and masking (a.win_ct > 0); the dense
// instantiation carries none of that code.
// SPLIT: the split-key tail (dense only; 1-D grid).  CTAs [0, split_full)
// are whole units, taken in the order of the 3-D grid (query block fastest,
// then head, then batch item); CTA split_full + i computes key-range piece
// i % split_pieces of unit split_full + i / split_pieces and writes its
// partial (unnormalised O, running max, row sum) to slot i of split_ws.
template <int D, int NSTAGE, bool WIN, bool SPLIT = false>
__global__ void __launch_bounds__(256, 1) attn_pipe_kernel(const __grid_constant__ AttnArgs a) {
  using C = PipeCfg<D, NSTAGE>;
  static_assert(!(WIN && SPLIT), "the split tail is for dense attention");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sKV = base;
  const uint32_t bars = sKV + C::kSmemKV;
  const uint32_t bar_q_full = bars;
  auto bar_kv_full = [&](int s) { return bars + 8u * (1 + s); };
  auto bar_kv_empty = [&](int s) { return bars + 8u * (1 + NSTAGE + s); };
  // Per parity p = j mod 2 of key tile j: s_full (S_j computed into S_p),
  // s_read (softmax has read S_j out of S_p), p_ready (P_j written), pv_done
  // (O += P_j V_j complete); drain: end of MMA thread p.
  auto bar_s_full = [&](int p) { return bars + 8u * (1 + 2 * NSTAGE + p); };
  auto bar_s_read = [&](int p) { return bars + 8u * (3 + 2 * NSTAGE + p); };
  auto bar_p_ready = [&](int p) { return bars + 8u * (5 + 2 * NSTAGE + p); };
  auto bar_pv_done = [&](int p) { return bars + 8u * (7 + 2 * NSTAGE + p); };
  auto bar_drain = [&](int p) { return bars + 8u * (9 + 2 * NSTAGE + p); };
  const uint32_t bar_v_clean = bars + 8u * (11 + 2 * NSTAGE);
  const uint32_t bar_o_staged = bars + 8u * (12 + 2 * NSTAGE);  // o rows staged for the TMA store (128 softmax)
  uint8_t* gmisc = gbase + C::kSmemKV + C::kNumBars * 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gmisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gmisc + 4);
  const uint32_t pad_issued = smem_u32(gmisc + 8);  // 1 once V of the tile straddling kv_len is requested

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) H3_TRACE(kEvCtaStart, 0);
  // Split launch: the combine kernel, launched after this grid with
  // programmatic stream serialization, may be scheduled as soon as every CTA
  // of this grid has started; it waits for this grid's completion itself.
  if constexpr (SPLIT) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- work unit: (b, h, 128-row query tile) -------------------------------
  int ux = static_cast<int>(blockIdx.x), uy = static_cast<int>(blockIdx.y), uz = static_cast<int>(blockIdx.z);
  int piece = -1;  // split tail: this CTA's key-range piece of its unit
  const int nqb = SPLIT ? (a.Sq + kBlockM - 1) / kBlockM : static_cast<int>(gridDim.x);
  if constexpr (SPLIT) {
    int unit = static_cast<int>(blockIdx.x);
    if (unit >= a.split_full) {
      const int i = unit - a.split_full;
      unit = a.split_full + i / a.split_pieces;
      piece = i % a.split_pieces;
    }
    ux = unit % nqb;
    uy = (unit / nqb) % a.Hq;
    uz = unit / (nqb * a.Hq);
  }
  const int b = uz;
  const int h = uy;
  const int kvh = h / (a.Hq / a.Hkv);
  // Longest units first: with a causal mask the last query blocks; under the
  // chunked window the first ones (blocks holding anchor rows see every key,
  // and the last chunk's window is cut at the sequence end).
  const int qb = WIN ? ux : nqb - 1 - ux;
  const int q0 = qb * kBlockM;
  int kv_lim = a.Sk;
  if (a.kv_len) kv_lim = min(kv_lim, max(a.kv_len[b], 0));
  const bool causal = a.causal || (a.causal_b && a.causal_b[b]);
  int q_lim = a.Sq;
  if (a.q_len) q_lim = min(q_lim, max(a.q_len[b], 0));
  int kv_end = kv_lim;
  if (causal) kv_end = min(kv_end, q0 + kBlockM);
  // Key tiles of this CTA: [0, n_lead) and [mid0, mid0 + n_tiles - n_lead).
  // Dense: one range [0, ceil(kv_end / 128)).  Chunked window (self-attention,
  // win_ct > 0): blocks holding an anchor row see every key; any other block
  // sees the anchor keys [0, win_af) and the keys of the chunks within
  // win_r of its rows' chunks.
  int n_lead = 0, mid0 = 0, n_tiles = 0;
  // keys every row of the block may attend: [0, full_a) and [full_lo, full_hi)
  int full_a = kv_end, full_lo = 0, full_hi = 0;
  if (q0 < q_lim && kv_end > 0) {
    const int n_all = (kv_end + kBlockN - 1) / kBlockN;
    n_tiles = n_all;
    if constexpr (WIN) {
      const int q_last = min(q0 + kBlockM, a.Sq) - 1;
      if (q0 >= a.win_af) {
        const int64_t af = a.win_af, ct = a.win_ct, r = a.win_r;
        const int64_t c_lo = (q0 - af) / ct, c_hi = (q_last - af) / ct;
        const int lo = static_cast<int>(af + max(c_lo - r, int64_t{0}) * ct);
        const int hi = static_cast<int>(min(af + (c_hi + r + 1) * ct, static_cast<int64_t>(kv_end)));
        n_lead = (min(a.win_af, kv_end) + kBlockN - 1) / kBlockN;
        mid0 = max(lo / kBlockN, n_lead);
        const int mid1 = hi > lo ? (hi + kBlockN - 1) / kBlockN : 0;
        n_tiles = n_lead + max(mid1 - mid0, 0);
        full_a = min(a.win_af, kv_end);
        full_lo = static_cast<int>(min(af + max(c_hi - r, int64_t{0}) * ct, static_cast<int64_t>(INT_MAX)));
        full_hi = static_cast<int>(min(af + (c_lo + r + 1) * ct, static_cast<int64_t>(kv_end)));
      } else if (q_last >= a.win_af) {
        full_a = 0;  // anchor rows and windowed rows share the block: mask every tile
      }
    }
  }
  int tile_lo = 0;  // first key tile of the CTA's range (a split piece's share of its unit)
  if constexpr (SPLIT) {
    if (piece >= 0) {
      const int lo = piece * n_tiles / a.split_pieces, hi = (piece + 1) * n_tiles / a.split_pieces;
      tile_lo = lo;
      n_tiles = hi - lo;
    }
  }
  // Load order = consumption order: K_0, K_1, K_2, then K_{j+3} (if any) and
  // V_j for j = 0, 1, ...  Load index of V_j: the K loads up to
  // K_{min(j+3, n-1)} and the V loads before it; K_j (j >= 3) sits right
  // before V_{j-3}.
  auto ld_v = [n_tiles](int j) { return min(j + 4, n_tiles) + j; };
  auto ld_k = [](int j) { return j < 3 ? j : 2 * j - 3; };
  auto stage_of = [](int load) { return load % NSTAGE; };
  auto phase_of = [](int load) { return static_cast<uint32_t>((load / NSTAGE) & 1); };
  // Iteration j visits entry (j + rot) mod n_tiles of the CTA's tile list.
  // The online softmax
  // does not depend on the order of the key tiles; rotating the start by the
  // query block spreads the CTAs that run at the same time (neighbouring
  // query blocks of one head) over different K/V tiles instead of having all
  // of them read the same tile's lines at once.
  const int rot = n_tiles > 0 ? ux % n_tiles : 0;
  auto tile_of = [rot, n_lead, mid0, n_tiles, tile_lo](int j) {
    const int m = j + rot < n_tiles ? j + rot : j + rot - n_tiles;  // position in the CTA's tile list
    if constexpr (WIN) {
      return m < n_lead ? m : mid0 + (m - n_lead);
    } else {
      return tile_lo + m;
    }
  };
  // Tile j's barriers of parity j % 2 complete for the (j / 2)-th time.
  auto bpar = [](int j) { return static_cast<uint32_t>((j >> 1) & 1); };
  // Iteration of the key tile that straddles kv_len (keys from kv_len on are
  // padding, read into the tile but never attended), or -1: none is loaded,
  // or kv_len is Sk or a tile edge.
  int j_pad = -1;
  if (n_tiles > 0 && kv_lim < a.Sk && (kv_lim % kBlockN) != 0) {
    const int tb = kv_lim / kBlockN;
    int m = -1;  // position of tile tb in the CTA's tile list
    if constexpr (WIN) {
      if (tb < n_lead) m = tb;
      else if (tb >= mid0 && tb < mid0 + n_tiles - n_lead) m = n_lead + (tb - mid0);
    } else {
      if (tb >= tile_lo && tb < tile_lo + n_tiles) m = tb - tile_lo;
    }
    if (m >= 0) j_pad = m >= rot ? m - rot : m - rot + n_tiles;
  }

  WaitCtl ctl{abort_flag, &g_status_word, a.wait_limit_ns, static_cast<int>(H3ATTN_ERR_TIMEOUT)};

  if (warp == C::kProducerWarp && lane == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    mbar_init(bar_q_full, 128);  // the 128 query rows stored to tensor memory
    for (int p = 0; p < 2; ++p) {
      mbar_init(bar_s_full(p), 1);
      mbar_init(bar_s_read(p), 128);
      mbar_init(bar_p_ready(p), 128);
      mbar_init(bar_pv_done(p), 1);
      mbar_init(bar_drain(p), 1);
    }
    mbar_init(bar_v_clean, 1);
    mbar_init(bar_o_staged, 128);
    *abort_flag = 0u;
    *reinterpret_cast<volatile uint32_t*>(gmisc + 8) = 0u;  // pad_issued
    fence_barrier_init();
    prefetch_tmap(&a.tm_k);
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
      int ld = 0;
      bool ok = true;
      auto load = [&](int kind, int j) {
        const int s = stage_of(ld);
        if (!(ok = mbar_wait(bar_kv_empty(s), phase_of(ld) ^ 1u, ctl))) return;
        H3_TRACE(kind == 0 ? kEvProdK : kEvProdV, j);
        mbar_arrive_expect_tx(bar_kv_full(s), C::kTileBytes);
        const CUtensorMap* m = kind == 0 ? &a.tm_k : &a.tm_v;
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(sKV + s * C::kTileBytes + c * C::kChunkBytes, m, bar_kv_full(s), c * 64, kvh,
                      tile_of(j) * kBlockN, b);
        if (kind == 1 && j == j_pad) st_release_cta(pad_issued, 1u);
        ++ld;
      };
      for (int j = 0; ok && j < 3 && j < n_tiles; ++j) load(0, j);
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 3 < n_tiles) load(0, j + 3);
        if (ok) load(1, j);
      }
      // Drain: every issued copy has landed before the CTA can retire.
      for (int i = ld > NSTAGE ? ld - NSTAGE : 0; i < ld; ++i)
        mbar_wait_drain(bar_kv_full(stage_of(i)), phase_of(i), a.wait_limit_ns);
    }
  } else if (warp == C::kMmaWarp || warp == C::kMmaWarp + 1) {
    // ======================= MMA issuers, one per tile parity ==============
    const int p = warp - C::kMmaWarp;
    if (lane == 0 && n_tiles > p) {
      bool ok = mbar_wait(bar_q_full, 0, ctl);
      tc_fence_after();
      // S_{i mod 2} = Q K_i^T (A = Q from tensor memory: channels
      // [16kk, 16kk+16) are columns [8kk, 8kk+8) of the Q region).
      auto issue_qk = [&](int i) -> bool {
        const int ld = ld_k(i), s = stage_of(ld);
        if (!mbar_wait(bar_kv_full(s), phase_of(ld), ctl)) return false;
        // S_{i-2} has been read out of the buffer
        if (i >= 2 && !mbar_wait(bar_s_read(i & 1), bpar(i - 2), ctl)) return false;
        tc_fence_after();
        H3_TRACE(kEvMmaQK0, i);
        const uint32_t kb = sKV + s * C::kTileBytes;
        const uint32_t tS = tmem + (i & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ts(tS, tmem + C::kColQ + kk * 8, sdesc_sw128(kb + off, 16, 1024), C::kIdescQK, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar_s_full(i & 1));
        tc_commit(bar_kv_empty(s));
        return true;
      };
      // prologue: S_0 on thread 0; S_1 and S_2 on thread 1
      if (ok) ok = issue_qk(p);
      if (ok && p == 1 && n_tiles > 2) ok = issue_qk(2);
      for (int j = p; ok && j < n_tiles; j += 2) {
        const int ldv = ld_v(j), sv = stage_of(ldv);
        if (!(ok = mbar_wait(bar_kv_full(sv), phase_of(ldv), ctl))) break;
        H3_TRACE(kEvMmaV, j);
        if (!(ok = mbar_wait(bar_p_ready(p), bpar(j), ctl))) break;
        // V_j's padding rows are zeroed (warp 7)
        if (j == j_pad && !(ok = mbar_wait(bar_v_clean, 0, ctl))) break;
        H3_TRACE(kEvMmaPV0, j);
        tc_fence_after();
        const uint32_t vb = sKV + sv * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
          mma_ts(tmem + C::kColO, tmem + C::kColP + kk * 8, sdesc_sw128(vb + kk * 2048, C::kChunkBytes, 1024),
                 C::kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar_pv_done(p));
        tc_commit(bar_kv_empty(sv));
        H3_TRACE(kEvMmaPV1, j);
        if (j + 3 < n_tiles) ok = issue_qk(j + 3);
      }
      // Drain every MMA issued by this thread before tensor memory is freed.
      tc_commit(bar_drain(p));
      mbar_wait_drain(bar_drain(p), 0, a.wait_limit_ns);
    }
  } else if (warp == 7) {
    // ======================= padding rows of the tile straddling kv_len ====
    if (j_pad >= 0) {
      const int ldv = ld_v(j_pad), sv = stage_of(ldv);
      const bool ok = __all_sync(0xFFFFFFFFu, count_wait_sleep(pad_issued, 1u, ctl) &&
                                                  mbar_wait(bar_kv_full(sv), phase_of(ldv), ctl));
      if (ok) {  // V tile landed; its stage is refilled only after O += P V of it
        zero_padding_rows<D>(sKV + sv * C::kTileBytes, kv_lim % kBlockN, lane, 32);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_v_clean);
      }
    }
  } else if (warp < 4) {
    // ======================= softmax / correction / epilogue ===============
    const int wq = warp & 3;         // lane quarter of tensor memory
    const int t = wq * 32 + lane;    // row within the tile
    const int row = q0 + t;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tO = tmem + lane_off + C::kColO;
    const uint32_t tP = tmem + lane_off + C::kColP;
    const float sl = a.scale_log2;
    const int64_t bit_words = (a.Sk + 31) / 32;
    // this row's window: anchor keys [0, win_a) and chunk keys [win_lo, win_hi)
    int win_a = INT_MAX, win_lo = 0, win_hi = 0;
    if (WIN && row >= a.win_af) {
      const int64_t af = a.win_af, ct = a.win_ct, r = a.win_r;
      const int64_t ci = (row - af) / ct;
      win_a = a.win_af;
      win_lo = static_cast<int>(min(af + max(ci - r, int64_t{0}) * ct, static_cast<int64_t>(INT_MAX)));
      win_hi = static_cast<int>(min(af + (ci + r + 1) * ct, static_cast<int64_t>(INT_MAX)));
    }
    float m_ref = -INFINITY;  // running max in scaled (log2) units
    float l = 0.0f;
    bool ok = true;
    // O += P V of tile i has completed
    auto wait_pv = [&](int i) { return mbar_wait(bar_pv_done(i & 1), bpar(i), ctl); };
    // This thread's query row (D bf16) into tensor-memory lane t as bf16
    // pairs, the A-operand layout of S = Q K^T; rows past Sq are zeros.
    if (n_tiles > 0) {
      const uint4* src = reinterpret_cast<const uint4*>(a.q_ptr + ((static_cast<int64_t>(b) * a.Sq + row) * a.Hq + h) * D);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = row < a.Sq ? __ldg(src + c * 8 + v) : make_uint4(0u, 0u, 0u, 0u);
          w[4 * v] = x.x;
          w[4 * v + 1] = x.y;
          w[4 * v + 2] = x.z;
          w[4 * v + 3] = x.w;
        }
        tmem_st32(tmem + lane_off + C::kColQ + c * 32, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_q_full);
    }
    for (int j = 0; j < n_tiles; ++j) {
      ok = mbar_wait(bar_s_full(j & 1), bpar(j), ctl);
      if (t == 0) H3_TRACE(kEvSmS0, j);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + (j & 1) * 128;
      const int kbase = tile_of(j) * kBlockN;
      bool need_mask = (kbase + kBlockN > kv_lim) || (causal && kbase + kBlockN - 1 > q0) || a.bits;
      if constexpr (WIN) need_mask = need_mask || (kbase + kBlockN > full_a && (kbase < full_lo || kbase + kBlockN > full_hi));
      // First pass: exponentials against the running max as it stands.  That
      // is exactly the result of the rescale rule below whenever no score of
      // the tile exceeds the running max by more than kRescaleThreshold, and
      // a tile row sum <= 2^kRescaleThreshold proves that.  Otherwise (and on
      // a row's first tile) a second pass reloads the scores, takes the row
      // max, rescales if it grew past the threshold and recomputes.  The pass
      // decision is per warp: tensor-memory loads are warp-collective.
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
        if (t == 0) H3_TRACE(kEvSmLd0, j);
        float s[kBlockN];
#pragma unroll
        for (int c = 0; c < kBlockN; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
        if (need_mask) {
          int lim = kv_lim - kbase;
          if (causal) lim = min(lim, row + 1 - kbase);
          // window: keys [0, w_a) and [w_lo, w_hi) relative to the tile
          int w_a = INT_MAX, w_lo = 0, w_hi = 0;
          if constexpr (WIN) {
            w_a = win_a - kbase;
            w_lo = win_lo - kbase;
            w_hi = win_hi - kbase;
          }
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
          for (int c = 0; c < kBlockN; ++c) {
            bool allowed = (c < lim) && ((wbits[c >> 5] >> (c & 31)) & 1u);
            if constexpr (WIN) allowed = allowed && (c < w_a || (c >= w_lo && c < w_hi));
            s[c] = allowed ? s[c] : -INFINITY;
          }
        }
        if (with_max) {
          // row max: 3-input max in 8 independent chains
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
            // O must hold every P V product of tiles < j before it is
            // rescaled; the products are sequential, so the last one
            // completing is enough.
            ok = wait_pv(j - 1);
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
        // p = exp2(s * scale*log2e - m): packed FMA, ex2, packed row-sum
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
      if (t == 0) H3_TRACE(kEvSmExp0, j);
      tc_fence_before();
      mbar_arrive(bar_s_read(j & 1));  // S_{j mod 2} may be overwritten by S_{j+2}
      // The single P buffer is free once O += P_{j-1} V_{j-1} has completed.
      if (j > 0) {
        ok = wait_pv(j - 1);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      tmem_st32(tP, pr[0]);
      tmem_st32(tP + 32, pr[1]);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p_ready(j & 1));
      if (t == 0) H3_TRACE(kEvSmArr0, j);
    }
    // ---- epilogue: O / l -> bf16 ------------------------------------------
    if (ok && n_tiles > 0) {
      ok = __all_sync(0xFFFFFFFFu, wait_pv(n_tiles - 1));
      tc_fence_after();
    }
    if (SPLIT && ok && piece >= 0) {
      // Partial of this key range: unnormalised O, the running max in scaled
      // log2 units (-inf when no key of the range was allowed) and the row
      // sum; the combine kernel weighs the pieces by 2^(m - max m).
      float* part = a.split_ws + static_cast<size_t>(static_cast<int>(blockIdx.x) - a.split_full) * (kBlockM * (D + 2));
      float4* prow = reinterpret_cast<float4*>(part + t * D);
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
#pragma unroll
        for (int v = 0; v < 8; ++v)
          prow[c * 8 + v] = make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]),
                                        __uint_as_float(o[4 * v + 2]), __uint_as_float(o[4 * v + 3]));
      }
      part[kBlockM * D + t] = m_ref;
      part[kBlockM * D + kBlockM + t] = l;
    } else if (ok) {
      // o = O / l as bf16, staged in the K/V ring (idle now: every load has
      // landed and been consumed once the last P V is complete) in the
      // 128-byte swizzled layout of the o map's box, then one TMA store of
      // the tile; rows past Sq lie outside the tensor and are not written.
      // (One row per thread straight to global memory writes 32 rows apart
      // per warp instruction; the CTA's end took ~4.8 k cycles that way.)
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
        const uint32_t rowp = sKV + (c >> 1) * C::kChunkBytes + t * 128;
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
      if (t == 0 && mbar_wait(bar_o_staged, 0, ctl)) {
        for (int c = 0; c < C::kChunks; ++c) tma_store_4d(&a.tm_o, sKV + c * C::kChunkBytes, c * 64, h, q0, b);
        bulk_commit_group();
        bulk_wait_group_read0();  // the shared-memory source is read before the CTA retires
      }
    }
  }

  if (threadIdx.x == 0) H3_TRACE(kEvCtaEnd, 0);
  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Output rows of the split tail's units from their pieces' partials:
// M = max_p m_p, o = (sum_p 2^(m_p - M) O_p) / (sum_p 2^(m_p - M) l_p),
// rounded once to bf16; rows past q_len and rows with no allowed key are
// zeros.  One warp per output row: lanes read the pieces' (m, l) side by side
// (lane i takes pieces i, i + 32, ...; max and sum by a fixed butterfly), then
// every lane accumulates its D/32 channels over the pieces in order, with the
// loads of several pieces in flight.  Deterministic: a fixed order throughout.
template <int D>
__global__ void __launch_bounds__(256) split_combine_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int V = D / 32;
  // Launched as a programmatic dependent of the split kernel: wait until that
  // grid has completed and its partials are visible (a no-op when launched
  // without the dependency).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int gw = static_cast<int>((blockIdx.x * 256u + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= a.split_tail * kBlockM) return;  // warp-uniform
  const int tu = gw / kBlockM, t = gw % kBlockM;
  const int nqb = (a.Sq + kBlockM - 1) / kBlockM;
  const int unit = a.split_full + tu;
  const int ux = unit % nqb, h = (unit / nqb) % a.Hq, b = unit / (nqb * a.Hq);
  const int row = (nqb - 1 - ux) * kBlockM + t;
  if (row >= a.Sq) return;  // warp-uniform
  int q_lim = a.Sq;
  if (a.q_len) q_lim = min(q_lim, max(a.q_len[b], 0));
  const int P = a.split_pieces;
  const size_t stride = static_cast<size_t>(kBlockM) * (D + 2);
  const float* part0 = a.split_ws + static_cast<size_t>(tu) * P * stride;
  float M = -INFINITY;
  for (int p = lane; p < P; p += 32) M = fmaxf(M, part0[p * stride + kBlockM * D + t]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
  float L = 0.0f, acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.0f;
  if (M != -INFINITY) {
    for (int p0 = 0; p0 < P; p0 += 32) {
      const int p = p0 + lane;
      float w = 0.0f, lw = 0.0f;
      if (p < P) {
        w = exp2f(part0[p * stride + kBlockM * D + t] - M);  // a piece with m = -inf weighs 0
        lw = w * part0[p * stride + kBlockM * D + kBlockM + t];
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) lw += __shfl_xor_sync(0xFFFFFFFFu, lw, off);
      L += lw;
      const int n = min(32, P - p0);
      const float* orow = part0 + static_cast<size_t>(p0) * stride + t * D + lane * V;
#pragma unroll 8
      for (int i = 0; i < n; ++i) {
        const float wi = __shfl_sync(0xFFFFFFFFu, w, i);
        float x[V];
        if constexpr (V == 4) {
          const float4 f = __ldg(reinterpret_cast<const float4*>(orow + i * stride));
          x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
        } else {
          const float2 f = __ldg(reinterpret_cast<const float2*>(orow + i * stride));
          x[0] = f.x; x[1] = f.y;
        }
#pragma unroll
        for (int c = 0; c < V; ++c) acc[c] = fmaf(wi, x[c], acc[c]);
      }
    }
  }
  const bool zero = row >= q_lim || !(L > 0.0f);
  const float inv = zero ? 0.0f : 1.0f / L;
  uint16_t* dst = a.o + ((static_cast<int64_t>(b) * a.Sq + row) * a.Hq + h) * D + lane * V;
  if constexpr (V == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
}

template <int D, int NSTAGE>
cudaError_t launch_pipe(const AttnArgs& a, cudaStream_t stream) {
  using C = PipeCfg<D, NSTAGE>;
  if (a.split_pieces > 0) {
    auto kern = attn_pipe_kernel<D, NSTAGE, false, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int ctas = a.split_full + a.split_tail * a.split_pieces;
    kern<<<ctas, C::kThreads, C::kSmemBytes, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // The combine as a programmatic dependent launch: its CTAs are placed
    // while the split kernel's last pieces run and start the moment it ends.
    const int warps = a.split_tail * kBlockM;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((warps + 7) / 8);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_combine_kernel<D>, a);
  }
  auto kern = a.win_ct > 0 ? attn_pipe_kernel<D, NSTAGE, true> : attn_pipe_kernel<D, NSTAGE, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Sq + kBlockM - 1) / kBlockM, a.Hq, a.B);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}
