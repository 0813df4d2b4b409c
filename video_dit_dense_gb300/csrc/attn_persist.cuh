// Persistent attention kernel (dense prefill, head_dim 64/128, every mask
// but the chunked window): one CTA per SM walks a static list of work units
// (batch, head, 128-row query block) with two MMA-issuing threads and a
// separate P buffer.  Included by attn_fwd.cu inside its anonymous namespace
// (uses its helpers); chosen with kernel = 3.  The default one-query-tile
// kernel (one CTA per unit, scheduled by the hardware onto the SMs in the
// same order) runs the same per-tile pipeline and measures faster in steady
// state, so this one is opt-in.
//
// Scheduling (per-batch and per-head work over a persistent grid, FastVideo
// PR #1799 "Implementation" and TeleFuser PR #37 section 2.3): unit u
// enumerates (b, h, query block) with the query block fastest and the longest
// (causal) block of each head first; CTA c of G takes units c, c + G, c + 2G,
// ...  Units of one head run side by side, so their K/V tiles are shared in
// L2.  A unit's key range stops at kv_len[b] and the causal limit; units past
// q_len[b] or with no key only write their zero rows.
//
// Within a CTA the key tiles of all its units form one stream, numbered
// J = 0, 1, ... across unit boundaries; the pipeline below runs on that
// stream, so loads and score products of the next unit start while the
// current one finishes.
//
// Tensor memory (512 columns x 128 lanes):
//   S_0, S_1  [0,128), [128,256)     scores of even / odd key tiles (fp32)
//   P         [256, 320)             probabilities of the current tile (bf16 pairs)
//   O         [320, 320+D)           output accumulator (fp32)
//   Q         [320+D, 320+D+D/2)     the current unit's query rows (bf16 pairs),
//                                    the A operand of S = Q K^T
//
// Score tile S_J lives in buffer S_{J mod 2}.  Once P_J is ready, MMA thread
// p = J mod 2 issues the burst
//     O += P_J V_J;   S_{J+3} = Q K_{J+3}^T  into S_{(J+1) mod 2}
// (the second half waits until softmax has read S_{J+1} out of that buffer,
// which it does at the start of its turn).  The tensor pipe thus runs the
// product that frees P right away and computes scores three tiles ahead.
// Prologue: S_0 (thread 0), S_1 and S_2 (thread 1).  Two issuing threads on
// two SM sub-partitions alternate these bursts: while one does its commits and
// barrier polls (slow when it shares a sub-partition with a busy softmax warp)
// the other keeps the tensor pipe fed.
//
// P has a single buffer, so softmax J writes P_J only after O += P_{J-1}
// V_{J-1} has completed; this also makes the O += P V products strictly
// sequential.  The first O += P V of a unit overwrites O (no accumulate); it
// is issued only after softmax has read the previous unit's O out, because
// softmax writes that P after its epilogue.
//
// Q has a single buffer.  Softmax writes the next unit's Q when it has seen
// the current unit's last score tile complete (every Q K^T of the unit is
// then done); each softmax thread then adds 1 to q_ready, a count in shared
// memory (128 per unit whose Q has been written), and an MMA thread waits for
// that count before its first Q K^T of each unit.  (A phase bit cannot stand
// in for the count: an MMA thread may skip a unit whose only tile the other
// thread issued, and then one parity no longer tells unit k's Q from unit
// k-2's.)
//
//   warps 0-3  softmax warpgroup, thread t = query row t = TMEM lane t
//   warp 4     TMA producer: K_0, K_1, K_2, then K_{J+3}, V_J for J = 0, 1, ...
//   warps 5-6  MMA issuers for even / odd key tiles (warp 5 allocates TMEM)
//   warp 7     idle
template <int D, int NSTAGE>
struct PersistCfg {
  static_assert(NSTAGE == 7 || NSTAGE == 12, "padding-row phase wait reasoned for these ring depths");
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = kBlockM * D * 2;
  static constexpr int kChunkBytes = kBlockM * 128;
  static constexpr int kSmemKV = NSTAGE * kTileBytes;
  // kv_full[NSTAGE], kv_empty[NSTAGE], s_full[2], s_read[2], p_ready[2], pv_done[2], drain[2]
  static constexpr int kNumBars = 2 * NSTAGE + 10;
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
  static_assert(NSTAGE >= 4, "K_{J+3}, V_J and the other thread's pair resident together");
};

// One work unit: a 128-row query block of one (batch, head) and its key
// tiles [0, n_tiles) in 128-key tile units, n_tiles = ceil(kv_end / 128).
struct PipeUnit {
  int b, h, kvh, q0;
  int kv_lim, q_lim;
  int causal;
  int n_tiles, rot;
};

// Out of line: every role decodes units, and one copy keeps the hot loops
// compact in the instruction cache.
__device__ __noinline__ PipeUnit pipe_unit(const AttnArgs& a, int u, int n_qb) {
  PipeUnit w;
  const int qbr = u % n_qb;  // blocks of a head from the last (longest when causal) down
  const int bh = u / n_qb;
  w.h = bh % a.Hq;
  w.b = bh / a.Hq;
  w.kvh = w.h / (a.Hq / a.Hkv);
  w.q0 = (n_qb - 1 - qbr) * kBlockM;
  w.kv_lim = a.Sk;
  if (a.kv_len) w.kv_lim = min(w.kv_lim, max(a.kv_len[w.b], 0));
  w.causal = a.causal || (a.causal_b && a.causal_b[w.b]);
  w.q_lim = a.Sq;
  if (a.q_len) w.q_lim = min(w.q_lim, max(a.q_len[w.b], 0));
  int kv_end = w.kv_lim;
  if (w.causal) kv_end = min(kv_end, w.q0 + kBlockM);
  w.n_tiles = 0;
  if (w.q0 < w.q_lim && kv_end > 0) {
    w.n_tiles = (kv_end + kBlockN - 1) / kBlockN;
  }
  // Iteration j visits entry (j + rot) mod n_tiles of the unit's tile list.
  // The online softmax does not depend on the order of the key tiles;
  // rotating the start by the query block spreads the CTAs that run at the
  // same time (neighbouring query blocks of one head) over different K/V
  // tiles instead of having all of them read the same tile's lines at once.
  w.rot = w.n_tiles > 0 ? qbr % w.n_tiles : 0;
  return w;
}

// Key tile (in 128-key units) of iteration j of unit w.
__device__ __forceinline__ int pipe_tile(const PipeUnit& w, int j) {
  return j + w.rot < w.n_tiles ? j + w.rot : j + w.rot - w.n_tiles;
}

// Walks the key-tile stream of this CTA: the tiles of its units with at
// least one tile, in order.  seq counts those units (unit seq's Q is in
// tensor memory once q_ready >= 128 (seq + 1)).
struct PipeCursor {
  const AttnArgs* a;
  int n_qb, n_units;
  int i;    // position in this CTA's unit list
  int j;    // tile within the unit
  int seq;  // units with tiles before this one
  bool valid;
  PipeUnit w;

  __device__ __forceinline__ void start(const AttnArgs* args, int nqb, int nunits) {
    a = args;
    n_qb = nqb;
    n_units = nunits;
    i = -1;
    seq = -1;
    next_unit();
  }
  __device__ __forceinline__ void next_unit() {
    valid = false;
    while (++i < n_units) {
      w = pipe_unit(*a, static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x), n_qb);
      if (w.n_tiles > 0) {
        valid = true;
        ++seq;
        j = 0;
        return;
      }
    }
  }
  __device__ __forceinline__ void advance() {
    if (++j >= w.n_tiles) next_unit();
  }
};


template <int D, int NSTAGE>
__global__ void __launch_bounds__(256, 1) attn_persist_kernel(const __grid_constant__ AttnArgs a) {
  using C = PersistCfg<D, NSTAGE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sKV = base;
  const uint32_t bars = sKV + C::kSmemKV;
  auto bar_kv_full = [&](int s) { return bars + 8u * s; };
  auto bar_kv_empty = [&](int s) { return bars + 8u * (NSTAGE + s); };
  // Per parity p = J mod 2 of key tile J: s_full (S_J computed into S_p),
  // s_read (softmax has read S_J out of S_p), p_ready (P_J written), pv_done
  // (O += P_J V_J complete); drain: end of MMA thread p.
  auto bar_s_full = [&](int p) { return bars + 8u * (2 * NSTAGE + p); };
  auto bar_s_read = [&](int p) { return bars + 8u * (2 + 2 * NSTAGE + p); };
  auto bar_p_ready = [&](int p) { return bars + 8u * (4 + 2 * NSTAGE + p); };
  auto bar_pv_done = [&](int p) { return bars + 8u * (6 + 2 * NSTAGE + p); };
  auto bar_drain = [&](int p) { return bars + 8u * (8 + 2 * NSTAGE + p); };
  uint8_t* gmisc = gbase + C::kSmemKV + C::kNumBars * 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gmisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gmisc + 4);
  const uint32_t q_ready = smem_u32(gmisc + 8);  // 128 x units whose Q is in tensor memory

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- this CTA's units: c, c + G, c + 2G, ... ------------------------------
  const int n_qb = (a.Sq + kBlockM - 1) / kBlockM;
  const int n_all = n_qb * a.Hq * a.B;
  const int G = static_cast<int>(gridDim.x);
  const int c = static_cast<int>(blockIdx.x);
  const int n_units = c < n_all ? (n_all - c + G - 1) / G : 0;
  auto unit_at = [&](int i) { return pipe_unit(a, c + i * G, n_qb); };

  // Load order = consumption order over the CTA's key-tile stream: K_0, K_1,
  // K_2, then K_{J+3} (if any) and V_J for J = 0, 1, ...  With N tiles in the
  // stream, V_J comes after the K loads up to K_{min(J+3, N-1)} and the V
  // loads before it; K_J (J >= 3) sits right before V_{J-3}.
  auto stage_of = [](int load) { return load % NSTAGE; };
  auto phase_of = [](int load) { return static_cast<uint32_t>((load / NSTAGE) & 1); };
  // Tile J's barriers of parity J % 2 complete for the (J / 2)-th time.
  auto bpar = [](int J) { return static_cast<uint32_t>((J >> 1) & 1); };

  WaitCtl ctl{abort_flag, &g_status_word, a.wait_limit_ns, static_cast<int>(H3ATTN_ERR_TIMEOUT)};
  int N = 0;  // key tiles in this CTA's stream
  if (warp != C::kProducerWarp)
    for (int i = 0; i < n_units; ++i) N += unit_at(i).n_tiles;
  auto ld_v = [N](int J) { return min(J + 4, N) + J; };

  if (warp == C::kProducerWarp && lane == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(bar_s_full(p), 1);
      mbar_init(bar_s_read(p), 128);
      mbar_init(bar_p_ready(p), 128);
      mbar_init(bar_pv_done(p), 1);
      mbar_init(bar_drain(p), 1);
    }
    *abort_flag = 0u;
    *reinterpret_cast<volatile uint32_t*>(gmisc + 8) = 0u;  // q_ready
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
    if (lane == 0 && n_units > 0 && !a.debug_skip_producer) {
      int ld = 0, jk = 0, jv = 0;
      bool ok = true;
      PipeCursor ck, cv;  // next K and next V tile of the stream
      ck.start(&a, n_qb, n_units);
      cv = ck;
      auto load = [&](int kind, const PipeCursor& cur, int J) {
        const int s = stage_of(ld);
        if (!(ok = mbar_wait(bar_kv_empty(s), phase_of(ld) ^ 1u, ctl))) return;
        H3_TRACE(kind == 0 ? kEvProdK : kEvProdV, J);
        mbar_arrive_expect_tx(bar_kv_full(s), C::kTileBytes);
        const CUtensorMap* m = kind == 0 ? &a.tm_k : &a.tm_v;
        const int key0 = pipe_tile(cur.w, cur.j) * kBlockN;
        for (int ch = 0; ch < C::kChunks; ++ch)
          tma_load_4d(sKV + s * C::kTileBytes + ch * C::kChunkBytes, m, bar_kv_full(s), ch * 64, cur.w.kvh, key0,
                      cur.w.b);
        ++ld;
      };
      for (int n = 0; ok && n < 3 && ck.valid; ++n) {
        load(0, ck, jk++);
        ck.advance();
      }
      while (ok && cv.valid) {
        if (ck.valid) {
          load(0, ck, jk++);
          ck.advance();
        }
        if (ok) {
          load(1, cv, jv++);
          cv.advance();
        }
      }
      // Drain: every issued copy has landed before the CTA can retire.
      for (int i = ld > NSTAGE ? ld - NSTAGE : 0; i < ld; ++i)
        mbar_wait_drain(bar_kv_full(stage_of(i)), phase_of(i), a.wait_limit_ns);
    }
  } else if (warp == C::kMmaWarp || warp == C::kMmaWarp + 1) {
    // ======================= MMA issuers, one per tile parity ==============
    const int p = warp - C::kMmaWarp;
    if (lane == 0 && N > p) {
      auto ld_k = [](int J) { return J < 3 ? J : 2 * J - 3; };
      PipeCursor cq, cv;  // this thread's next Q K^T tile and next P V tile
      cq.start(&a, n_qb, n_units);
      cv = cq;
      int jq = 0, jv = 0;  // their positions in the stream
      int q_seq = -1;      // the unit whose Q this thread has seen written
      bool ok = true;
      // S_{J mod 2} = Q K_J^T (A = Q from tensor memory: channels
      // [16kk, 16kk+16) are columns [8kk, 8kk+8) of the Q region).
      auto issue_qk = [&](int J) -> bool {
        while (jq < J) {
          cq.advance();
          ++jq;
        }
        if (cq.seq != q_seq) {
          if (!count_wait(q_ready, 128u * static_cast<uint32_t>(cq.seq + 1), ctl)) return false;
          q_seq = cq.seq;
        }
        const int ld = ld_k(J), s = stage_of(ld);
        if (!mbar_wait(bar_kv_full(s), phase_of(ld), ctl)) return false;
        // S_{J-2} has been read out of the buffer
        if (J >= 2 && !mbar_wait(bar_s_read(J & 1), bpar(J - 2), ctl)) return false;
        tc_fence_after();
        H3_TRACE(kEvMmaQK0, J);
        const uint32_t kb = sKV + s * C::kTileBytes;
        const uint32_t tS = tmem + (J & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_ts(tS, tmem + C::kColQ + kk * 8, sdesc_sw128(kb + off, 16, 1024), C::kIdescQK, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar_s_full(J & 1));
        tc_commit(bar_kv_empty(s));
        return true;
      };
      // prologue: S_0 on thread 0; S_1 and S_2 on thread 1
      ok = issue_qk(p);
      if (ok && p == 1 && N > 2) ok = issue_qk(2);
      for (int J = p; ok && J < N; J += 2) {
        while (jv < J) {
          cv.advance();
          ++jv;
        }
        const int ldv = ld_v(J), sv = stage_of(ldv);
        if (!(ok = mbar_wait(bar_kv_full(sv), phase_of(ldv), ctl))) break;
        H3_TRACE(kEvMmaV, J);
        if (!(ok = mbar_wait(bar_p_ready(p), bpar(J), ctl))) break;
        H3_TRACE(kEvMmaPV0, J);
        tc_fence_after();
        const uint32_t vb = sKV + sv * C::kTileBytes;
        // the first tile of a unit starts O afresh
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
          mma_ts(tmem + C::kColO, tmem + C::kColP + kk * 8, sdesc_sw128(vb + kk * 2048, C::kChunkBytes, 1024),
                 C::kIdescPV, (cv.j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar_pv_done(p));
        tc_commit(bar_kv_empty(sv));
        H3_TRACE(kEvMmaPV1, J);
        if (J + 3 < N) ok = issue_qk(J + 3);
      }
      // Drain every MMA issued by this thread before tensor memory is freed.
      tc_commit(bar_drain(p));
      mbar_wait_drain(bar_drain(p), 0, a.wait_limit_ns);
    }
  } else if (warp < 4) {
    // ======================= softmax / correction / epilogue ===============
    const int wq = warp & 3;         // lane quarter of tensor memory
    const int t = wq * 32 + lane;    // row within the query block
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tO = tmem + lane_off + C::kColO;
    const uint32_t tP = tmem + lane_off + C::kColP;
    const float sl = a.scale_log2;
    const int64_t bit_words = (a.Sk + 31) / 32;
    bool ok = true;
    int J = 0;  // position in the CTA's key-tile stream
    // O += P V of tile I has completed
    auto wait_pv = [&](int I) { return mbar_wait(bar_pv_done(I & 1), bpar(I), ctl); };
    auto q_row = [&](const PipeUnit& w) {
      return a.q_ptr + ((static_cast<int64_t>(w.b) * a.Sq + (w.q0 + t)) * a.Hq + w.h) * D;
    };
    // This thread's query row of unit w (D bf16) into tensor-memory lane t as
    // bf16 pairs, the A-operand layout of S = Q K^T; rows past Sq are zeros.
    // q_ready counts the row once it is stored.
    auto write_q = [&](const PipeUnit& w) {
      const bool live = w.q0 + t < a.Sq;
      const uint4* src = reinterpret_cast<const uint4*>(q_row(w));
#pragma unroll
      for (int ch = 0; ch < D / 64; ++ch) {
        uint32_t r[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = live ? __ldg(src + ch * 8 + v) : make_uint4(0u, 0u, 0u, 0u);
          r[4 * v] = x.x;
          r[4 * v + 1] = x.y;
          r[4 * v + 2] = x.z;
          r[4 * v + 3] = x.w;
        }
        tmem_st32(tmem + lane_off + C::kColQ + ch * 32, r);
      }
      tmem_st_wait();
      tc_fence_before();
      add_release_cta(q_ready, 1u);
    };
    // first unit at or after position i with a key tile (n_units if none)
    auto next_tiled = [&](int i, PipeUnit& w) {
      for (; i < n_units; ++i) {
        w = unit_at(i);
        if (w.n_tiles > 0) break;
      }
      return i;
    };
    {
      PipeUnit w0;
      if (next_tiled(0, w0) < n_units) write_q(w0);
    }
#pragma unroll 1
    for (int i = 0; ok && i < n_units; ++i) {
      const PipeUnit w = unit_at(i);
      const int row = w.q0 + t;
      const bool live_row = row < a.Sq;
      if (w.n_tiles == 0) {
        // no key for this block (past q_len, or kv_len 0): zero rows
        if (live_row) {
          uint4* dst = reinterpret_cast<uint4*>(a.o + ((static_cast<int64_t>(w.b) * a.Sq + row) * a.Hq + w.h) * D);
#pragma unroll
          for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      // The next unit with key tiles: its query rows go into tensor memory
      // once this unit's last score tile is complete; pull them into L2 now.
      {
        PipeUnit wn;
        if (next_tiled(i + 1, wn) < n_units && wn.q0 + t < a.Sq) {
          const char* pf = reinterpret_cast<const char*>(q_row(wn));
#pragma unroll
          for (int off = 0; off < D * 2; off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(pf + off));
        }
      }
      float m_ref = -INFINITY;  // running max in scaled (log2) units
      float l = 0.0f;
#pragma unroll 1
      for (int j = 0; j < w.n_tiles; ++j, ++J) {
        ok = mbar_wait(bar_s_full(J & 1), bpar(J), ctl);
        if (t == 0) H3_TRACE(kEvSmS0, J);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tS = tmem + lane_off + (J & 1) * 128;
        const int kbase = pipe_tile(w, j) * kBlockN;
        bool need_mask = (kbase + kBlockN > w.kv_lim) || (w.causal && kbase + kBlockN - 1 > w.q0) || a.bits;
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
          for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, sr[q]);
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_ld_wait(sr[q]);
          if (t == 0) H3_TRACE(kEvSmLd0, J);
          float s[kBlockN];
#pragma unroll
          for (int q = 0; q < kBlockN; ++q) s[q] = __uint_as_float(sr[q >> 5][q & 31]);
          if (need_mask) {
            int lim = w.kv_lim - kbase;
            if (w.causal) lim = min(lim, row + 1 - kbase);
            uint32_t wbits[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
            if (a.bits && live_row) {
              const uint32_t* br = a.bits + (static_cast<int64_t>(w.b) * a.Sq + row) * bit_words;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int64_t wi = kbase / 32 + q;
                wbits[q] = wi < bit_words ? br[wi] : 0u;
              }
            }
#pragma unroll
            for (int q = 0; q < kBlockN; ++q) {
              bool allowed = (q < lim) && ((wbits[q >> 5] >> (q & 31)) & 1u);
              s[q] = allowed ? s[q] : -INFINITY;
            }
          }
          if (with_max) {
            // row max: 3-input max in 8 independent chains
            float mx[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) mx[q] = fmaxf(s[2 * q], s[2 * q + 1]);
#pragma unroll
            for (int q = 16; q < kBlockN; q += 16) {
#pragma unroll
              for (int e = 0; e < 8; ++e) mx[e] = fmax3(mx[e], s[q + 2 * e], s[q + 2 * e + 1]);
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
              // O must hold every P V product of this unit's tiles before it
              // is rescaled; the products are sequential, so the last one
              // completing is enough.
              ok = wait_pv(J - 1);
              if (!__all_sync(0xFFFFFFFFu, ok)) {
                ok = false;
                break;
              }
              tc_fence_after();
#pragma unroll 1
              for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                tmem_ld32(tO + q * 32, o);
                tmem_ld_wait(o);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                tmem_st32(tO + q * 32, o);
              }
              tmem_st_wait();
            }
          }
          const float mu = (m_ref == -INFINITY) ? 0.0f : m_ref;
          // p = exp2(s * scale*log2e - m): packed FMA, ex2, packed row-sum
          float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int q = 0; q < kBlockN; q += 2) {
            float t0, t1;
            ffma2(t0, t1, s[q], s[q + 1], sl, sl, -mu, -mu);
            const float p0 = ex2(t0);
            const float p1 = ex2(t1);
            const int a2 = ((q >> 1) & 3) * 2;
            fadd2(ls[a2], ls[a2 + 1], ls[a2], ls[a2 + 1], p0, p1);
            pr[q >> 6][(q >> 1) & 31] = pack_bf16x2(p0, p1);
          }
          tile_sum = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
          if (with_max) break;
          with_max = __any_sync(0xFFFFFFFFu, !(tile_sum <= kFastPassSumLimit));
          if (!with_max) break;
        }
        if (!ok) break;
        l += tile_sum;
        if (t == 0) H3_TRACE(kEvSmExp0, J);
        tc_fence_before();
        mbar_arrive(bar_s_read(J & 1));  // S_{J mod 2} may be overwritten by S_{J+2}
        // The single P buffer is free once O += P_{J-1} V_{J-1} has completed.
        if (J > 0) {
          ok = wait_pv(J - 1);
          if (!__all_sync(0xFFFFFFFFu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (w.kv_lim < a.Sk && kbase + kBlockN > w.kv_lim) {
          // the tile straddles kv_len: zero V_J's padding rows once V_J has
          // landed.  The stage's previous fill (K_J with 7 stages, V_{J-6}
          // with 12) has landed by now, so this phase wait is exact.
          const int ldv = ld_v(J);
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_kv_full(stage_of(ldv)), phase_of(ldv), ctl));
          if (!ok) break;
          zero_padding_rows<D>(sKV + stage_of(ldv) * C::kTileBytes, w.kv_lim - kbase, t, kBlockM);
        }
        tmem_st32(tP, pr[0]);
        tmem_st32(tP + 32, pr[1]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_p_ready(J & 1));
        if (t == 0) H3_TRACE(kEvSmArr0, J);
      }
      // ---- epilogue: O / l -> bf16 ----------------------------------------
      if (ok) {
        PipeUnit wn;
        if (next_tiled(i + 1, wn) < n_units) write_q(wn);
      }
      if (ok) {
        ok = __all_sync(0xFFFFFFFFu, wait_pv(J - 1));
        tc_fence_after();
      }
      if (!ok) break;
      uint16_t* orow = a.o + ((static_cast<int64_t>(w.b) * a.Sq + row) * a.Hq + w.h) * D;
      const bool zero_row = row >= w.q_lim || !(l > 0.0f);
      const float inv = zero_row ? 0.0f : 1.0f / l;
#pragma unroll 1
      for (int q = 0; q < D / 32; ++q) {
        uint32_t o[32];
        tmem_ld32(tO + q * 32, o);
        tmem_ld_wait(o);
        if (live_row) {
          uint4* dst = reinterpret_cast<uint4*>(orow + q * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = zero_row ? 0.0f : __uint_as_float(o[v * 8 + e]) * inv;
            dst[v] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                                pack_bf16x2(f[6], f[7]));
          }
        }
      }
      // the next unit's first P (and so its O-overwriting product) follows
      // these loads in program order
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int NSTAGE>
cudaError_t launch_persist(const AttnArgs& a, cudaStream_t stream) {
  using C = PersistCfg<D, NSTAGE>;
  auto kern = attn_persist_kernel<D, NSTAGE>;
  if (a.win_ct > 0) return cudaErrorInvalidValue;  // the chunked window runs on the default kernel
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  // one CTA per SM (the kernel holds all of tensor memory), never more CTAs than units
  const int64_t units = static_cast<int64_t>((a.Sq + kBlockM - 1) / kBlockM) * a.Hq * a.B;
  const int grid = static_cast<int>(units < sms ? units : sms);
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}
