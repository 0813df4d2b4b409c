// Attention kernel that chains work units per CTA (included by attn_fwd.cu
// inside its anonymous namespace; uses its helpers).  Head dim 128.
//
// One CTA per SM walks the work units c, c + G, c + 2G, ... (G = grid size;
// a unit is 128 query rows of one batch item and head, in the order of the
// 3-D grid of the other kernels).  A CTA of the one-tile kernel pays its start
// (tensor-memory allocation, barrier set-up, Q load, first K tiles, first
// scores) and its end (last P V, epilogue) once per unit; here they are paid
// once per CTA, and a unit's Q hand-off and epilogue run on warps of their own
// beside the next unit's tiles.  This is what short units need
// (cross-attention against a few hundred text keys, short sequences).
//
// The key tiles of all the CTA's units form one stream J = 0, 1, ...; the
// per-tile protocol on that stream is the one-tile kernel's: scores three
// tiles ahead in S_{J mod 2}, a single P buffer written once the previous
// P V has completed, two MMA-issuing threads alternating bursts
//     O += P_J V_J;   S_{J+3} = Q K_{J+3}^T.
//
// Tensor memory (512 columns x 128 lanes):
//   S_0, S_1  [0,128), [128,256)   scores of even / odd stream tiles (fp32)
//   P         [256, 320)           probabilities of the current tile (bf16 pairs)
//   O         [320, 448)           output accumulator of the current unit (fp32)
//   Q         [448, 512)           query rows of the current unit (bf16 pairs),
//                                  the A operand of S = Q K^T
// Shared memory: one 32 KiB buffer through which Q tiles come in and o tiles
// go out (TMA, 128-byte swizzle), a ring of NSTAGE K/V tiles (32 KiB each),
// barriers, the row sums handed from the softmax to the epilogue (two slots).
//
// Unit changes (kappa = rank of a unit among the CTA's units with key tiles;
// units without any, rows past q_len or kv_len 0, only get zero rows):
//   Q: the unit warps copy Q_kappa from the buffer into tensor memory once
//      the softmax has seen the last score tile of unit kappa - 1 (every
//      Q K^T of that unit has then completed), count the copy into q_ready,
//      and load Q_{kappa+1} into the buffer themselves once o of unit
//      kappa - 1 has gone out through it.  An MMA thread
//      waits for q_ready >= 128 (kappa + 1) before its first Q K^T of unit
//      kappa: a count, because a thread may issue no score product of a
//      one-tile unit, after which a phase bit no longer tells unit kappa's Q
//      from unit kappa - 2's.  (Were the producer to load Q, it would wait for
//      the copy before its next K load while running three tiles ahead, over
//      several short units: the copy waits for the epilogue of an earlier
//      unit, whose P V needs a V load queued behind that K.)
//   O: the MMA thread of a unit's last tile commits o_full after its P V; the
//      unit warps read O and the row sums and free O (the next unit's first
//      P V, no accumulate, waits for that), stage o = O / l as bf16 in the
//      buffer and write it with one TMA store.
// Every hand-off is a barrier that completes once per use (or a count), and
// each waiter can show that at most the awaited phase is pending; the CPU
// model of this protocol in the tests runs random interleavings of it.
//
//   warps 0-3   softmax warpgroup, thread t = query row t = TMEM lane t
//   warps 4-7   unit warps: Q staging -> tensor memory, epilogue
//   warp 8      TMA producer: K_0, K_1, K_2, then K_{J+3}, V_J for J = 0, 1, ...
//   warps 9-10  MMA issuers (warp 9 allocates tensor memory)
//   warp 11     padding: in each unit's key tile that straddles kv_len, zeroes
//               the V rows past kv_len before that tile's P V
template <int NSTAGE>
struct ChainCfg {
  static constexpr int D = 128;
  static constexpr int kTileBytes = kBlockN * D * 2;  // one K or V tile
  static constexpr int kChunk = kBlockN * 128;        // one 64-channel swizzle column of a tile
  static constexpr int kQBytes = kBlockM * D * 2;
  static constexpr int kSmemKV = NSTAGE * kTileBytes;
  // kv_full[NSTAGE], kv_empty[NSTAGE], s_full[2], s_read[2], p_ready[2], pv_done[2], drain[2],
  // q_sfull, buf_free, q_free, o_full, o_free, l_full[2], l_free[2]
  static constexpr int kNumBars = 2 * NSTAGE + 10 + 5 + 4;
  static constexpr int kMiscBytes = 32 + 2 * kBlockM * 4;  // slot, abort, counts; row sums [2][128]
  static constexpr int kSmemBytes = 1024 + kQBytes + kSmemKV + kNumBars * 8 + kMiscBytes;
  static constexpr int kThreads = 384;
  static constexpr int kUnitWarp = 4;  // warps 4-7
  static constexpr int kProducerWarp = 8;
  static constexpr int kMmaWarp = 9;   // and 10
  static constexpr int kPadWarp = 11;
  static constexpr int kColP = 256;
  static constexpr int kColO = 320;
  static constexpr int kColQ = 448;
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kBlockN, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
  // Register split: 12 warps launch with 168 registers a thread (three warps
  // per SM sub-partition); the control and unit warpgroups drop to 96 and the
  // softmax warpgroup rises to 232.
  static constexpr int kLaunchRegs = 168;
  static constexpr int kCtlRegs = 96;
  static constexpr int kUnitRegs = 96;
  static constexpr int kSoftRegs = 232;
  static_assert(128 * (kSoftRegs + kCtlRegs + kUnitRegs) <= kThreads * kLaunchRegs, "register split");
  static_assert(kColQ + D / 2 <= static_cast<int>(kTmemCols), "tensor memory budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(NSTAGE >= 4, "K_{J+3}, V_J and the other thread's pair resident together");
};

// The rows, key range and key-tile count of work unit u.
struct ChainUnit {
  int b, h, q0, x;    // batch item, query head, first query row, index in the grid's x order
  int rot;            // first iteration's key tile (x mod n)
  int kv_lim, q_lim;  // keys [0, kv_lim) may be attended; rows from q_lim on are zeros
  bool causal;
  int n;              // key tiles
};

__device__ __forceinline__ ChainUnit chain_unit(const AttnArgs& a, int u, int nqb) {
  ChainUnit c;
  c.x = u % nqb;
  c.h = (u / nqb) % a.Hq;
  c.b = u / (nqb * a.Hq);
  c.q0 = (nqb - 1 - c.x) * kBlockM;  // longest (causal) first within each (b, h)
  c.kv_lim = a.Sk;
  if (a.kv_len) c.kv_lim = min(c.kv_lim, max(a.kv_len[c.b], 0));
  c.causal = a.causal || (a.causal_b && a.causal_b[c.b]);
  c.q_lim = a.Sq;
  if (a.q_len) c.q_lim = min(c.q_lim, max(a.q_len[c.b], 0));
  int kv_end = c.kv_lim;
  if (c.causal) kv_end = min(kv_end, c.q0 + kBlockM);
  c.n = (c.q0 < c.q_lim && kv_end > 0) ? (kv_end + kBlockN - 1) / kBlockN : 0;
  c.rot = c.n > 0 ? c.x % c.n : 0;
  return c;
}

// Key tile of iteration j of a unit: the start is rotated by the unit's x
// index so that the CTAs running at the same time read different K/V lines.
__device__ __forceinline__ int chain_tile(const ChainUnit& c, int j) {
  return j + c.rot < c.n ? j + c.rot : j + c.rot - c.n;
}

// Iteration of a unit's key tile that straddles kv_len (loaded with padding
// rows), or -1.
__device__ __forceinline__ int chain_pad_iter(const AttnArgs& a, const ChainUnit& c) {
  if (c.n == 0 || c.kv_lim >= a.Sk || (c.kv_lim % kBlockN) == 0) return -1;
  const int tb = c.kv_lim / kBlockN;
  if (tb >= c.n) return -1;
  return tb >= c.rot ? tb - c.rot : tb - c.rot + c.n;
}

// Position in the stream of a CTA's key tiles: unit u (rank kap among the
// units with key tiles), its iteration j, and the count of earlier units with
// a padded tile.
struct ChainIt {
  int u, kap, j, pads, j_pad;
  ChainUnit c;
};

__device__ __forceinline__ void chain_skip_empty(ChainIt& it, const AttnArgs& a, int nqb, int n_units, int G) {
  while (it.u < n_units) {
    it.c = chain_unit(a, it.u, nqb);
    if (it.c.n > 0) break;
    it.u += G;
  }
  it.j_pad = it.u < n_units ? chain_pad_iter(a, it.c) : -1;
}

__device__ __forceinline__ void chain_begin(ChainIt& it, const AttnArgs& a, int nqb, int n_units, int G) {
  it.u = static_cast<int>(blockIdx.x);
  it.kap = 0;
  it.j = 0;
  it.pads = 0;
  chain_skip_empty(it, a, nqb, n_units, G);
}

__device__ __forceinline__ void chain_next(ChainIt& it, const AttnArgs& a, int nqb, int n_units, int G) {
  if (++it.j < it.c.n) return;
  if (it.j_pad >= 0) ++it.pads;
  ++it.kap;
  it.j = 0;
  it.u += G;
  chain_skip_empty(it, a, nqb, n_units, G);
}

template <int NSTAGE>
__global__ void __launch_bounds__(384, 1) attn_chain_kernel(const __grid_constant__ AttnArgs a) {
  using C = ChainCfg<NSTAGE>;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sKV = base + C::kQBytes;
  const uint32_t bars = sKV + C::kSmemKV;
  auto bar_kv_full = [&](int s) { return bars + 8u * s; };
  auto bar_kv_empty = [&](int s) { return bars + 8u * (NSTAGE + s); };
  // per parity p = J mod 2 of stream tile J (as in the one-tile kernel)
  auto bar_s_full = [&](int p) { return bars + 8u * (2 * NSTAGE + p); };
  auto bar_s_read = [&](int p) { return bars + 8u * (2 * NSTAGE + 2 + p); };
  auto bar_p_ready = [&](int p) { return bars + 8u * (2 * NSTAGE + 4 + p); };
  auto bar_pv_done = [&](int p) { return bars + 8u * (2 * NSTAGE + 6 + p); };
  auto bar_drain = [&](int p) { return bars + 8u * (2 * NSTAGE + 8 + p); };
  // once per unit with key tiles
  const uint32_t bar_q_sfull = bars + 8u * (2 * NSTAGE + 10);  // Q_kappa in the staging buffer
  const uint32_t bar_buf_free = bars + 8u * (2 * NSTAGE + 11);  // the unit threads are done with the buffer
  const uint32_t bar_q_free = bars + 8u * (2 * NSTAGE + 12);   // every Q K^T of the unit done (128 softmax)
  const uint32_t bar_o_full = bars + 8u * (2 * NSTAGE + 13);   // the unit's last P V done
  const uint32_t bar_o_free = bars + 8u * (2 * NSTAGE + 14);   // O read out (128 unit threads)
  // per row-sum slot kappa mod 2
  auto bar_l_full = [&](int s) { return bars + 8u * (2 * NSTAGE + 15 + s); };
  auto bar_l_free = [&](int s) { return bars + 8u * (2 * NSTAGE + 17 + s); };
  uint8_t* gmisc = gbase + C::kQBytes + C::kSmemKV + C::kNumBars * 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gmisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gmisc + 4);
  const uint32_t q_ready = smem_u32(gmisc + 8);   // 128 x units whose Q is in tensor memory
  const uint32_t v_issued = smem_u32(gmisc + 12); // V tiles the producer has issued
  const uint32_t cleaned = smem_u32(gmisc + 16);  // padded tiles the padding warp has zeroed
  float* lbuf = reinterpret_cast<float*>(gmisc + 32);  // [2][128] row sums

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nqb = (a.Sq + kBlockM - 1) / kBlockM;
  const int n_units = nqb * a.Hq * a.B;
  const int G = static_cast<int>(gridDim.x);
  // stream length, and the units with key tiles
  int N = 0, n_kap = 0;
  for (int u = blockIdx.x; u < n_units; u += G) {
    const int n = chain_unit(a, u, nqb).n;
    N += n;
    n_kap += n > 0;
  }
  // ring positions: K_0, K_1, K_2, then K_{J+3} (if any) and V_J
  auto ld_v = [N](int J) { return min(J + 4, N) + J; };
  auto ld_k = [](int J) { return J < 3 ? J : 2 * J - 3; };
  auto stage_of = [](int pos) { return pos % NSTAGE; };
  auto phase_of = [](int pos) { return static_cast<uint32_t>((pos / NSTAGE) & 1); };
  auto bpar = [](int J) { return static_cast<uint32_t>((J >> 1) & 1); };

  WaitCtl ctl{abort_flag, &g_status_word, a.wait_limit_ns, static_cast<int>(H3ATTN_ERR_TIMEOUT)};

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
      mbar_init(bar_l_full(p), 128);
      mbar_init(bar_l_free(p), 128);
    }
    mbar_init(bar_q_sfull, 1);
    mbar_init(bar_buf_free, 128);
    mbar_init(bar_q_free, 128);
    mbar_init(bar_o_full, 1);
    mbar_init(bar_o_free, 128);
    *abort_flag = 0u;
    for (int i = 8; i < 32; i += 4) *reinterpret_cast<volatile uint32_t*>(gmisc + i) = 0u;
    fence_barrier_init();
    prefetch_tmap(&a.tm_q);
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

  if (warp >= C::kProducerWarp) {
   regs_dec<C::kCtlRegs>();
   if (warp == C::kProducerWarp) {
    // ======================= TMA producer ==================================
    if (lane == 0 && N > 0 && !a.debug_skip_producer) {
      int pos = 0;
      bool ok = true;
      ChainIt kit, vit;  // next K and next V tile of the stream
      chain_begin(kit, a, nqb, n_units, G);
      chain_begin(vit, a, nqb, n_units, G);
      auto load = [&](int kind, ChainIt& it, int J) {
        const int s = stage_of(pos);
        if (!(ok = mbar_wait(bar_kv_empty(s), phase_of(pos) ^ 1u, ctl))) return;
        H3_TRACE(kind == 0 ? kEvProdK : kEvProdV, J);
        mbar_arrive_expect_tx(bar_kv_full(s), C::kTileBytes);
        const CUtensorMap* m = kind == 0 ? &a.tm_k : &a.tm_v;
        const int kvh = it.c.h / (a.Hq / a.Hkv);
        const int row = chain_tile(it.c, it.j) * kBlockN;
        for (int ch = 0; ch < 2; ++ch)
          tma_load_4d(sKV + s * C::kTileBytes + ch * C::kChunk, m, bar_kv_full(s), ch * 64, kvh, row, it.c.b);
        if (kind == 1) st_release_cta(v_issued, static_cast<uint32_t>(J + 1));
        ++pos;
        chain_next(it, a, nqb, n_units, G);
      };
      for (int J = 0; ok && J < 3 && J < N; ++J) load(0, kit, J);
      for (int J = 0; ok && J < N; ++J) {
        if (J + 3 < N) load(0, kit, J + 3);
        if (ok) load(1, vit, J);
      }
      // Drain: every issued copy has landed before the CTA can retire.
      for (int i = pos > NSTAGE ? pos - NSTAGE : 0; i < pos; ++i)
        mbar_wait_drain(bar_kv_full(stage_of(i)), phase_of(i), a.wait_limit_ns);
    }
   } else if (warp == C::kMmaWarp || warp == C::kMmaWarp + 1) {
    // ======================= MMA issuers ===================================
    // Thread p issues P V of the stream tiles J = p mod 2 and, after each,
    // S_{J+3}; prologue S_0 (thread 0), S_1 and S_2 (thread 1).
    const int p = warp - C::kMmaWarp;
    if (lane == 0 && N > p) {
      bool ok = true;
      int q_seen = -1;  // last unit whose Q this thread has waited for
      ChainIt qi, vi;   // next score tile and next P V tile of this thread
      chain_begin(qi, a, nqb, n_units, G);
      chain_begin(vi, a, nqb, n_units, G);
      int qJ = 0;
      auto seek = [&](ChainIt& it, int& at, int J) {
        for (; at < J; ++at) chain_next(it, a, nqb, n_units, G);
      };
      // S_{J mod 2} = Q K_J^T (A = Q from tensor memory: channels [16kk, 16kk+16)
      // are columns [8kk, 8kk+8) of the Q region)
      auto issue_qk = [&](int J) -> bool {
        seek(qi, qJ, J);
        if (qi.kap != q_seen) {
          if (!count_wait(q_ready, 128u * static_cast<uint32_t>(qi.kap + 1), ctl)) return false;
          q_seen = qi.kap;
        }
        const int pk = ld_k(J), sk = stage_of(pk);
        if (!mbar_wait(bar_kv_full(sk), phase_of(pk), ctl)) return false;
        // S_{J-2} has been read out of the buffer
        if (J >= 2 && !mbar_wait(bar_s_read(J & 1), bpar(J - 2), ctl)) return false;
        tc_fence_after();
        H3_TRACE(kEvMmaQK0, J);
        const uint32_t kb = sKV + sk * C::kTileBytes;
        const uint32_t tS = tmem + (J & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kChunk + (kk & 3) * 32;
          mma_ts(tS, tmem + C::kColQ + kk * 8, sdesc_sw128(kb + off, 16, 1024), C::kIdescQK, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar_s_full(J & 1));
        tc_commit(bar_kv_empty(sk));
        return true;
      };
      ok = issue_qk(p);
      if (ok && p == 1 && N > 2) ok = issue_qk(2);
      int vJ = 0;
      for (int J = p; ok && J < N; J += 2) {
        seek(vi, vJ, J);
        const int pv = ld_v(J), sv = stage_of(pv);
        if (!(ok = mbar_wait(bar_kv_full(sv), phase_of(pv), ctl))) break;
        H3_TRACE(kEvMmaV, J);
        if (!(ok = mbar_wait(bar_p_ready(J & 1), bpar(J), ctl))) break;
        // a unit's first product overwrites O: the unit warps have read the previous unit's
        if (vi.j == 0 && vi.kap >= 1 && !(ok = mbar_wait(bar_o_free, (vi.kap - 1) & 1, ctl))) break;
        // V_J's padding rows are zeroed (warp 11)
        if (vi.j == vi.j_pad && !(ok = count_wait(cleaned, static_cast<uint32_t>(vi.pads + 1), ctl))) break;
        tc_fence_after();
        H3_TRACE(kEvMmaPV0, J);
        const uint32_t vb = sKV + sv * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          mma_ts(tmem + C::kColO, tmem + C::kColP + kk * 8, sdesc_sw128(vb + kk * 2048, C::kChunk, 1024),
                 C::kIdescPV, (vi.j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(bar_pv_done(p));
        tc_commit(bar_kv_empty(sv));
        if (vi.j == vi.c.n - 1) tc_commit(bar_o_full);
        H3_TRACE(kEvMmaPV1, J);
        if (J + 3 < N) ok = issue_qk(J + 3);
      }
      // Drain every MMA issued by this thread before tensor memory is freed.
      tc_commit(bar_drain(p));
      mbar_wait_drain(bar_drain(p), 0, a.wait_limit_ns);
    }
   } else {
    // ======================= padding rows of each unit's straddling tile ===
    int J = 0, pads = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < n_units; u += G) {
      const ChainUnit c = chain_unit(a, u, nqb);
      const int j_pad = chain_pad_iter(a, c);
      if (j_pad >= 0) {
        const int Jp = J + j_pad, pos = ld_v(Jp), s = stage_of(pos);
        ok = __all_sync(0xFFFFFFFFu, count_wait_sleep(v_issued, static_cast<uint32_t>(Jp + 1), ctl) &&
                                         mbar_wait(bar_kv_full(s), phase_of(pos), ctl));
        if (!ok) break;
        // V_Jp landed; its stage is refilled only after O += P V of it
        zero_padding_rows<D>(sKV + s * C::kTileBytes, c.kv_lim % kBlockN, lane, 32);
        __syncwarp();
        ++pads;
        if (lane == 0) st_release_cta(cleaned, static_cast<uint32_t>(pads));
      }
      J += c.n;
    }
   }
  } else if (warp < 4) {
    regs_inc<C::kSoftRegs>();
    // ======================= softmax =======================================
    const int wq = warp & 3;
    const int t = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tO = tmem + lane_off + C::kColO;
    const uint32_t tP = tmem + lane_off + C::kColP;
    const float sl = a.scale_log2;
    const int64_t bit_words = (a.Sk + 31) / 32;
    bool ok = true;
    int J = 0, kap = -1;
    // O += P V of stream tile i has completed
    auto wait_pv = [&](int i) { return mbar_wait(bar_pv_done(i & 1), bpar(i), ctl); };
    for (int u = blockIdx.x; ok && u < n_units; u += G) {
      const ChainUnit c = chain_unit(a, u, nqb);
      if (c.n == 0) continue;
      ++kap;
      const int row = c.q0 + t;
      float m_ref = -INFINITY;  // running max in scaled (log2) units
      float l = 0.0f;
      for (int j = 0; j < c.n; ++j, ++J) {
        ok = mbar_wait(bar_s_full(J & 1), bpar(J), ctl);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (t == 0) H3_TRACE(kEvSmS0, J);
        // every Q K^T of the unit has completed: the unit warps may replace Q
        if (j == c.n - 1) mbar_arrive(bar_q_free);
        const uint32_t tS = tmem + lane_off + (J & 1) * 128;
        const int kbase = chain_tile(c, j) * kBlockN;
        const bool need_mask = (kbase + kBlockN > c.kv_lim) || (c.causal && kbase + kBlockN - 1 > c.q0) || a.bits;
        // First pass against the running max as it stands, a second one with
        // the tile's max when a row's sum says it may have grown by more than
        // the rescale threshold (the one-tile kernel's rule).
        bool with_max = __any_sync(0xFFFFFFFFu, m_ref == -INFINITY);
        float tile_sum = 0.0f;
        uint32_t pr[2][32];
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
          uint32_t sr[4][32];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, sr[cc]);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) tmem_ld_wait(sr[cc]);
          if (t == 0) H3_TRACE(kEvSmLd0, J);
          float s[kBlockN];
#pragma unroll
          for (int cc = 0; cc < kBlockN; ++cc) s[cc] = __uint_as_float(sr[cc >> 5][cc & 31]);
          if (need_mask) {
            int lim = c.kv_lim - kbase;
            if (c.causal) lim = min(lim, row + 1 - kbase);
            uint32_t wbits[4] = {0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu};
            if (a.bits && row < a.Sq) {
              const uint32_t* br = a.bits + (static_cast<int64_t>(c.b) * a.Sq + row) * bit_words;
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                const int64_t wi = kbase / 32 + w;
                wbits[w] = wi < bit_words ? br[wi] : 0u;
              }
            }
#pragma unroll
            for (int cc = 0; cc < kBlockN; ++cc)
              s[cc] = ((cc < lim) && ((wbits[cc >> 5] >> (cc & 31)) & 1u)) ? s[cc] : -INFINITY;
          }
          if (with_max) {
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
            for (int cc = 16; cc < kBlockN; cc += 16) {
#pragma unroll
              for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[cc + 2 * i], s[cc + 2 * i + 1]);
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
              // O holds every product of the unit's earlier tiles once the
              // last one has completed (the products are sequential)
              ok = wait_pv(J - 1);
              if (!__all_sync(0xFFFFFFFFu, ok)) {
                ok = false;
                break;
              }
              tc_fence_after();
#pragma unroll 1
              for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                tmem_ld32(tO + cc * 32, o);
                tmem_ld_wait(o);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                tmem_st32(tO + cc * 32, o);
              }
              tmem_st_wait();
            }
          }
          const float mu = (m_ref == -INFINITY) ? 0.0f : m_ref;
          float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int cc = 0; cc < kBlockN; cc += 2) {
            float t0, t1;
            ffma2(t0, t1, s[cc], s[cc + 1], sl, sl, -mu, -mu);
            const float p0 = ex2(t0);
            const float p1 = ex2(t1);
            const int a2 = ((cc >> 1) & 3) * 2;
            fadd2(ls[a2], ls[a2 + 1], ls[a2], ls[a2 + 1], p0, p1);
            pr[cc >> 6][(cc >> 1) & 31] = pack_bf16x2(p0, p1);
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
        // The single P buffer is free once O += P V of the previous stream tile has completed.
        if (J > 0) {
          ok = wait_pv(J - 1);
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
        mbar_arrive(bar_p_ready(J & 1));
        if (t == 0) H3_TRACE(kEvSmArr0, J);
      }
      if (!ok) break;
      // row sums to the epilogue: slot kap mod 2, once its previous unit's were read
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_l_free(kap & 1), bpar(kap) ^ 1u, ctl));
      if (!ok) break;
      lbuf[(kap & 1) * kBlockM + t] = l;
      mbar_arrive(bar_l_full(kap & 1));
    }
  } else {
    regs_dec<C::kUnitRegs>();
    // ======================= unit warps: Q hand-off, epilogue ==============
    // One shared-memory buffer serves both hand-offs.  Per unit with key
    // tiles: Q_kap is copied out of it into tensor memory; o of the previous
    // unit is staged into it (128-byte swizzled rows, the o map's box) once
    // that unit's O and row sums are complete; then, once every unit thread is
    // done with the buffer, one thread writes that o with one TMA store and,
    // when the store has read the buffer, loads Q_{kap+1} into it.  (One row
    // per thread stored straight to global memory took 3.5-4.2 k cycles per
    // unit and held back the next unit's first P V.)  The waits park the
    // warps in the barrier wait: they share SM sub-partitions with the
    // softmax warps, whose issue slots set the pace.
    const int wq = warp & 3;
    const int t = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tO = tmem + lane_off + C::kColO;
    bool ok = true;
    // thread 0: phases of buf_free waited, units whose Q was loaded / copied out
    int kap = -1, uses = 0, q_loaded = -1, q_taken = -1;
    auto load_q = [&](int u) {  // Q of unit u (with key tiles) into the buffer
      const ChainUnit c = chain_unit(a, u, nqb);
      mbar_arrive_expect_tx(bar_q_sfull, C::kQBytes);
      for (int ch = 0; ch < 2; ++ch)
        tma_load_4d(sQ + ch * C::kChunk, &a.tm_q, bar_q_sfull, ch * 64, c.h, c.q0, c.b);
      ++q_loaded;
    };
    auto next_with_tiles = [&](int u) {
      for (u += G; u < n_units; u += G)
        if (chain_unit(a, u, nqb).n > 0) return u;
      return n_units;
    };
    // o = O / l as bf16 rows of the unit of rank pk (row-sum slot pk mod 2) into the buffer
    auto stage_o = [&](const ChainUnit& c, int pk) -> bool {
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_parked(bar_o_full, pk & 1, ctl) &&
                                       mbar_wait_parked(bar_l_full(pk & 1), bpar(pk), ctl)))
        return false;
      if (t == 0) H3_TRACE(kEvSmLd1, pk);
      tc_fence_after();
      const float l = lbuf[(pk & 1) * kBlockM + t];
      mbar_arrive(bar_l_free(pk & 1));
      const bool zero_row = c.q0 + t >= c.q_lim || !(l > 0.0f);
      const float inv = zero_row ? 0.0f : 1.0f / l;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + cc * 32, o);
        tmem_ld_wait(o);
        if (cc == D / 32 - 1) {
          tc_fence_before();
          mbar_arrive(bar_o_free);  // O read out: the next unit's first P V may overwrite it
          if (t == 0) H3_TRACE(kEvCtaEnd, pk);
        }
        // channels [32cc, 32cc + 32): 16-byte units 4(cc mod 2) .. +3 of row t in swizzle column cc / 2
        const uint32_t rowp = sQ + (cc >> 1) * C::kChunk + t * 128;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = zero_row ? 0u
                            : pack_bf16x2(__uint_as_float(o[v * 8 + 2 * e]) * inv,
                                          __uint_as_float(o[v * 8 + 2 * e + 1]) * inv);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                           rowp + ((((cc & 1) * 4 + v) ^ (t & 7)) << 4)),
                       "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                       : "memory");
        }
      }
      fence_proxy_async_smem();
      return true;
    };
    // Every unit thread is done with the buffer: thread 0 stores the staged o
    // of unit pc (if has_o), then loads the Q of the next unit with key tiles
    // after unit u (if any).
    auto flush = [&](bool has_o, const ChainUnit& pc, int u) -> bool {
      mbar_arrive(bar_buf_free);
      bool r = true;
      if (t == 0) {
        r = mbar_wait_parked(bar_buf_free, uses & 1, ctl);
        ++uses;
        if (r && has_o) {
          for (int ch = 0; ch < 2; ++ch) tma_store_4d(&a.tm_o, sQ + ch * C::kChunk, ch * 64, pc.h, pc.q0, pc.b);
          bulk_commit_group();
          bulk_wait_group_read0();  // the buffer is read out before the next Q lands in it
        }
        if (r && u < n_units) {
          const int nu = next_with_tiles(u);
          if (nu < n_units) load_q(nu);
        }
      }
      return __all_sync(0xFFFFFFFFu, r);
    };
    if (t == 0 && n_kap > 0) load_q(next_with_tiles(static_cast<int>(blockIdx.x) - G));
    ChainUnit prev{};
    for (int u = blockIdx.x; ok && u < n_units; u += G) {
      const ChainUnit c = chain_unit(a, u, nqb);
      if (c.n == 0) {  // nothing to attend: zero rows
        const int row = c.q0 + t;
        if (row < a.Sq) {
          uint4* dst = reinterpret_cast<uint4*>(a.o + ((static_cast<int64_t>(c.b) * a.Sq + row) * a.Hq + c.h) * D);
#pragma unroll
          for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      ++kap;
      // Q_kap into tensor memory once every Q K^T of the previous unit is done
      ok = __all_sync(0xFFFFFFFFu, (kap == 0 || mbar_wait_parked(bar_q_free, (kap - 1) & 1, ctl)) &&
                                       mbar_wait_parked(bar_q_sfull, kap & 1, ctl));
      if (!ok) break;
      if (t == 0) q_taken = kap;
      if (t == 0) H3_TRACE(kEvSmS1, kap);
      tc_fence_after();
      {
        // row t of the buffer: 16-byte unit i of a 128-byte row sits at i ^ (t mod 8)
        const uint32_t src = sQ + t * 128;
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t w[32];
#pragma unroll
          for (int v = 0; v < 8; ++v)
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[4 * v]), "=r"(w[4 * v + 1]), "=r"(w[4 * v + 2]), "=r"(w[4 * v + 3])
                         : "r"(src + ch * C::kChunk + ((v ^ (t & 7)) << 4))
                         : "memory");
          tmem_st32(tmem + lane_off + C::kColQ + ch * 32, w);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      add_release_cta(q_ready, 1u);
      if (t == 0) H3_TRACE(kEvCtaStart, kap);
      // o of the previous unit through the buffer (this thread's rows only: it
      // read its own Q row above), then the next Q into it
      if (kap >= 1 && !(ok = stage_o(prev, kap - 1))) break;
      if (!(ok = flush(kap >= 1, prev, u))) break;
      prev = c;
    }
    if (ok && kap >= 0) ok = stage_o(prev, kap) && flush(true, prev, n_units);
    // Drain: a Q load issued but never waited for (the CTA aborted) lands before the CTA retires.
    if (t == 0 && q_loaded > q_taken) mbar_wait_drain(bar_q_sfull, q_loaded & 1, a.wait_limit_ns);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int NSTAGE>
cudaError_t launch_chain(const AttnArgs& a, cudaStream_t stream) {
  using C = ChainCfg<NSTAGE>;
  auto kern = attn_chain_kernel<NSTAGE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // The softmax warpgroup's register increase waits until the other
  // warpgroups' decreases leave enough of the block's launch registers: a
  // build that launched with fewer than the split assumes is refused here.
  static const int launch_regs = [kern] {
    cudaFuncAttributes fa{};
    return cudaFuncGetAttributes(&fa, kern) == cudaSuccess ? fa.numRegs : 0;
  }();
  if (launch_regs * C::kThreads < 128 * (C::kSoftRegs + C::kCtlRegs + C::kUnitRegs)) return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int64_t units = static_cast<int64_t>((a.Sq + kBlockM - 1) / kBlockM) * a.Hq * a.B;
  const int grid = static_cast<int>(min(static_cast<int64_t>(sms), units));
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}
