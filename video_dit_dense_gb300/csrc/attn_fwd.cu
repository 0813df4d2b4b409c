// Dense prefill attention o = softmax(q k^T * scale) v on BSHD bf16 tensors
// for sm_103a (FastVideo PR #1832 "Add FlashInfer attention backend support
// for MiniMax H3", section "Summary": dense non-causal self-attention on
// [batch, sequence, heads, head_dim] with head_dim 128; FastVideo PR #1799
// "Add opt-in FlashInfer attention backend for Wan", section
// "Implementation": cross-attention, GQA, causal and boolean [Q, K] masks).
//
// One CTA owns NQ query tiles of 128 rows of one (batch, head) and streams
// that head's K/V through shared memory in 128-key tiles:
//
//   warp 4*NQ      TMA producer: Q tiles once, then K_j, V_j into a ring of
//                  NSTAGE shared-memory stages (mbarrier full/empty pairs).
//   warp 4*NQ+1    MMA issuer (one thread): S_q = Q_q K_j^T with
//                  tcgen05.mma (both operands in shared memory, fp32
//                  accumulator in tensor memory), then O_q += P_q V_j with
//                  P_q read from tensor memory.  Also allocates tensor memory.
//   warp 4*NQ+2    zeroes the V rows past kv_len of the key tile that
//                  straddles kv_len, before that tile's O += P V.
//   warps 4q..4q+3 softmax warpgroup of tile q: thread t owns query row t
//                  (tensor-memory lane t).  It reads its 128 scores, applies
//                  the mask, keeps a running max and sum, writes
//                  P = exp2(s*scale*log2e - m) as bf16 back into tensor
//                  memory over the scores, rescales its O row when the max
//                  grows by more than 2^8, and finally writes O / l.
//
// Tensor memory (128 lanes; all 512 columns, or 256 when two CTAs share an
// SM): S_q at columns [128q, 128q+128), P_q over the first 64 columns of S_q
// (bf16 pairs), O_q at [128*NQ + D*q, 128*NQ + D*(q+1)).
//
// The next S_q = Q_q K^T overwrites P_q, and tcgen05 only orders MMAs that
// share an accumulator, so the issuer waits for O_q += P_q V to complete
// before it issues the next S_q; the other tile's MMA is queued meanwhile,
// which keeps the tensor pipe busy across that wait.
//
// Masking: tiles entirely inside the allowed region run unmasked; the
// kv_len boundary tile, causal diagonal tiles and every tile of a packed-bit
// mask set disallowed scores to -inf before the max.  Key tiles past the
// last allowed key of the CTA are never loaded.
#include <cuda_bf16.h>

#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace h3 {
namespace {

constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8
// A tile row sum at most 2^kRescaleThreshold bounds every probability of the
// tile by 2^kRescaleThreshold: no score exceeds the running max by more.
constexpr float kFastPassSumLimit = 256.0f;

// CTAS: resident CTAs per SM the configuration is built for (1, or 2 for one
// query tile with a short ring: one CTA's prologue and epilogue then overlap
// the other's products).
template <int D, int NQ, int NSTAGE, int CTAS = 1>
struct Cfg {
  static constexpr int kChunks = D / 64;                  // 128-byte swizzle columns per row
  static constexpr int kTileBytes = kBlockM * D * 2;      // one 128-row tile of Q, K or V
  static constexpr int kChunkBytes = kBlockM * 128;       // 16 KiB: one swizzle column of a tile
  static constexpr int kSmemQ = NQ * kTileBytes;
  static constexpr int kSmemKV = NSTAGE * kTileBytes;
  static constexpr int kNumBars = 1 + 2 * NSTAGE + 4 * NQ + 3;
  static constexpr int kSmemBytes = 1024 /*alignment slack*/ + kSmemQ + kSmemKV + kNumBars * 8 + 16;
  // NQ softmax warpgroups + one control warpgroup (producer, MMA issuer, the warp that zeroes V
  // padding rows, one idle warp)
  static constexpr int kThreads = NQ * 128 + 128;
  static constexpr int kProducerWarp = NQ * 4;
  static constexpr int kMmaWarp = NQ * 4 + 1;
  // Register split: launch budget kThreads * floor(65536 / (kThreads * CTAS)) (rounded to 8);
  // the control warpgroup drops to kCtlRegs, softmax warpgroups rise to kSoftRegs.
  static constexpr int kLaunchRegs = (65536 / (kThreads * CTAS)) / 8 * 8;
  static constexpr int kCtlRegs = CTAS == 1 ? 96 : 56;
  static constexpr int kSoftRegs =
      ((kThreads * kLaunchRegs - 128 * kCtlRegs) / (NQ * 128)) / 8 * 8 > 232
          ? 232
          : ((kThreads * kLaunchRegs - 128 * kCtlRegs) / (NQ * 128)) / 8 * 8;
  static_assert(NQ * 128 * kSoftRegs + 128 * kCtlRegs <= kThreads * kLaunchRegs, "register split");
  // Only needed when the launch budget per thread is below what softmax wants.
  static constexpr bool kRebalance = kLaunchRegs < 200;
  static constexpr int kColO = NQ * 128;
  // Head dim 64 with one query tile: P gets tensor-memory columns of its own
  // after O (S 128 + O 64 + P 64 = the CTA's 256), so the next tile's scores
  // may overwrite S as soon as the softmax has read it, instead of after the
  // P V that reads P over S.
  static constexpr bool kSepP = D == 64 && NQ == 1;
  static constexpr int kColP = kColO + NQ * D;
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kBlockN, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
  // tensor memory per CTA: all of it, or an equal share (a power of two >= 32 columns)
  static constexpr uint32_t kTmemAlloc = CTAS == 1 ? kTmemCols : kTmemCols / CTAS;
  static_assert((kSepP ? kColP + 64 : kColO + NQ * D) <= static_cast<int>(kTmemAlloc), "tensor memory budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(CTAS * (kSmemBytes + 1024) <= 233472, "shared memory of CTAS resident CTAs");
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Wait that ignores the abort flag: used to drain copies/MMAs already in flight.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

__device__ int g_status_word = 0;

// Shared-memory count: each producer thread adds with release, the waiter
// reads with acquire (CTA scope).
__device__ __forceinline__ void add_release_cta(uint32_t addr, uint32_t v) {
  asm volatile("red.release.cta.shared::cta.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_cta(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
// Wait until the count at addr reaches target; bounded like mbar_wait.
__device__ __forceinline__ bool count_wait(uint32_t addr, uint32_t target, const WaitCtl& ctl) {
  if (ld_acquire_cta(addr) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (ld_acquire_cta(addr) >= target) return true;
    if (*ctl.abort_flag) return false;
    if (globaltimer_ns() - t0 > ctl.limit_ns) {
      *ctl.abort_flag = 1u;
      atomicExch(ctl.status, ctl.timeout_code);
      return false;
    }
  }
}
__device__ __forceinline__ void st_release_cta(uint32_t addr, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// count_wait for a warp with nothing else to do: sleeps between polls so that
// it takes no issue slots from the warps that share its SM sub-partition.
__device__ __forceinline__ bool count_wait_sleep(uint32_t addr, uint32_t target, const WaitCtl& ctl) {
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_cta(addr) < target) {
    if (*ctl.abort_flag) return false;
    if (globaltimer_ns() - t0 > ctl.limit_ns) {
      *ctl.abort_flag = 1u;
      atomicExch(ctl.status, ctl.timeout_code);
      return false;
    }
    __nanosleep(256);
  }
  return true;
}
// mbar_wait for the same kind of warp: each poll parks the thread in the
// barrier wait (woken when the phase completes, or after the hint) instead of
// spinning.
__device__ __forceinline__ bool mbar_wait_parked(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_hint(bar, parity, 1000000u)) {
    if (*ctl.abort_flag) return false;
    if (globaltimer_ns() - t0 > ctl.limit_ns) {
      *ctl.abort_flag = 1u;
      atomicExch(ctl.status, ctl.timeout_code);
      return false;
    }
  }
  return true;
}

// Keys past kv_len may hold anything (uninitialised padding, NaN, Inf).  Their
// scores are masked by selection, but in O += P V a zero probability times a
// NaN or Inf value is still NaN, so in the key tile that straddles kv_len the
// V rows r0 = kv_len mod 128 .. 127 are zeroed in shared memory before that
// tile's O += P V is issued.  128-byte swizzle: row r of 64-channel chunk c is
// the 128 bytes at c * 16 KiB + r * 128, its 16-byte units permuted among
// themselves, so whole rows are contiguous: the calling thread `lane` of
// `stride` writes 16-byte units lane, lane + stride, ... of that range
// (neighbouring lanes on neighbouring units, no bank conflicts).  The proxy fence orders these generic writes before the
// tensor core's reads, which follow a barrier the caller arrives on.
// The zeroing warp learns that the V tile has landed in two steps: the
// producer raises a flag in shared memory when it issues that load (the
// stage's previous fill has then landed and been consumed), and only then
// does the warp wait for the stage's phase, which from there on is
// unambiguous; waiting on the phase alone from the kernel's start could pass
// on a fill two rounds older (same parity).
template <int D>
__device__ __forceinline__ void zero_padding_rows(uint32_t tile, int r0, int lane, int stride) {
  const int units = (kBlockN - r0) * 8;  // 16-byte units of rows r0 .. 127 in one chunk
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    const uint32_t first = tile + c * 16384 + r0 * 128;
    for (int k = lane; k < units; k += stride)
      asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(first + k * 16), "r"(0u) : "memory");
  }
  fence_proxy_async_smem();
}

#ifdef H3ATTN_TRACE
// Optional pipeline trace (compile with -DH3ATTN_TRACE): clock64 stamps of
// the first CTA's producer, MMA issuer and softmax threads, per key tile.
constexpr int kTraceTiles = 512;
enum TraceEv {
  kEvProdK, kEvProdV, kEvMmaK, kEvMmaQK0, kEvMmaQK1, kEvMmaV, kEvMmaPV0, kEvMmaPV1,
  kEvSmS0, kEvSmLd0, kEvSmExp0, kEvSmArr0, kEvSmS1, kEvSmLd1, kEvSmExp1, kEvSmArr1, kEvCtaStart, kEvCtaEnd, kNumEv
};
__device__ unsigned long long g_trace[kNumEv][kTraceTiles];
#define H3_TRACE(ev, j)                                                                     \
  do {                                                                                      \
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (j) < kTraceTiles)         \
      g_trace[(ev)][(j)] = clock64();                                                       \
  } while (0)
#else
#define H3_TRACE(ev, j) \
  do {                  \
  } while (0)
#endif

template <int D, int NQ, int NSTAGE, int CTAS>
__global__ void __launch_bounds__(Cfg<D, NQ, NSTAGE, CTAS>::kThreads, CTAS)
    attn_fwd_kernel(const __grid_constant__ AttnArgs a) {
  using C = Cfg<D, NQ, NSTAGE, CTAS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t sQ = base;
  const uint32_t sKV = base + C::kSmemQ;
  const uint32_t bars = sKV + C::kSmemKV;
  const uint32_t bar_q_full = bars;
  auto bar_kv_full = [&](int s) { return bars + 8u * (1 + s); };
  auto bar_kv_empty = [&](int s) { return bars + 8u * (1 + NSTAGE + s); };
  auto bar_s_full = [&](int q) { return bars + 8u * (1 + 2 * NSTAGE + q); };
  auto bar_p_ready = [&](int q) { return bars + 8u * (1 + 2 * NSTAGE + NQ + q); };
  auto bar_pv_done = [&](int q) { return bars + 8u * (1 + 2 * NSTAGE + 2 * NQ + q); };
  const uint32_t bar_drain = bars + 8u * (1 + 2 * NSTAGE + 3 * NQ);
  const uint32_t bar_v_clean = bars + 8u * (2 + 2 * NSTAGE + 3 * NQ);  // padding rows of V zeroed
  // o rows of query tile q staged for the TMA store (its 128 softmax threads)
  auto bar_o_staged = [&](int q) { return bars + 8u * (3 + 2 * NSTAGE + 3 * NQ + q); };
  // separate-P form: the softmax has read the scores out of S (128 softmax threads)
  const uint32_t bar_s_read = bars + 8u * (3 + 2 * NSTAGE + 4 * NQ);
  uint8_t* gmisc = gbase + C::kSmemQ + C::kSmemKV + C::kNumBars * 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gmisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gmisc + 4);
  const uint32_t pad_issued = smem_u32(gmisc + 8);  // 1 once V of the tile straddling kv_len is requested

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work unit of this CTA -------------------------------------------
  const int b = blockIdx.z;
  const int h = blockIdx.y;
  const int kvh = h / (a.Hq / a.Hkv);
  const int n_qblocks = gridDim.x;
  const int qb = n_qblocks - 1 - static_cast<int>(blockIdx.x);  // longest (causal) units first
  const int q0 = qb * (NQ * kBlockM);
  int kv_lim = a.Sk;
  if (a.kv_len) kv_lim = min(kv_lim, max(a.kv_len[b], 0));
  const bool causal = a.causal || (a.causal_b && a.causal_b[b]);
  int q_lim = a.Sq;
  if (a.q_len) q_lim = min(q_lim, max(a.q_len[b], 0));
  int kv_end = kv_lim;
  if (causal) kv_end = min(kv_end, q0 + NQ * kBlockM);
  int n_tiles = (q0 >= q_lim || kv_end <= 0) ? 0 : (kv_end + kBlockN - 1) / kBlockN;
  // The key tile that straddles kv_len (keys from kv_len on are padding, read
  // into the tile but never attended), or -1: none is loaded, or kv_len is Sk
  // or a tile edge.  Its V rows past kv_len are zeroed before O += P V.
  const int j_pad =
      (kv_lim < a.Sk && (kv_lim % kBlockN) != 0 && kv_lim / kBlockN < n_tiles) ? kv_lim / kBlockN : -1;

  WaitCtl ctl{abort_flag, &g_status_word, a.wait_limit_ns, static_cast<int>(H3ATTN_ERR_TIMEOUT)};

  // ---- setup ---------------------------------------------------------------
  if (warp == C::kProducerWarp && lane == 0) {
    mbar_init(bar_q_full, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    for (int q = 0; q < NQ; ++q) {
      mbar_init(bar_s_full(q), 1);
      mbar_init(bar_p_ready(q), 128);
      mbar_init(bar_pv_done(q), 1);
      mbar_init(bar_o_staged(q), 128);
    }
    mbar_init(bar_s_read, 128);
    mbar_init(bar_drain, 1);
    mbar_init(bar_v_clean, 1);
    *abort_flag = 0u;
    *reinterpret_cast<volatile uint32_t*>(gmisc + 8) = 0u;  // pad_issued
    fence_barrier_init();
    if (n_tiles > 0 && !a.debug_skip_producer) {
      // Q and the first key tile's K and V (ring positions 0 and 1, first use
      // of their stages) go out before the block-wide set-up completes
      mbar_arrive_expect_tx(bar_q_full, C::kSmemQ);
      for (int q = 0; q < NQ; ++q)
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(sQ + q * C::kTileBytes + c * C::kChunkBytes, &a.tm_q, bar_q_full, c * 64, h,
                      q0 + q * kBlockM, b);
      for (int kind = 0; kind < 2; ++kind) {
        mbar_arrive_expect_tx(bar_kv_full(kind), C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(sKV + kind * C::kTileBytes + c * C::kChunkBytes, kind == 0 ? &a.tm_k : &a.tm_v,
                      bar_kv_full(kind), c * 64, kvh, 0, b);
      }
      if (j_pad == 0) st_release_cta(pad_issued, 1u);
    }
    prefetch_tmap(&a.tm_q);
    prefetch_tmap(&a.tm_k);
    prefetch_tmap(&a.tm_v);
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemAlloc);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= NQ * 4) {
   if constexpr (C::kRebalance) regs_dec<C::kCtlRegs>();
   if (warp == C::kProducerWarp) {
    // ======================= TMA producer ==================================
    if (lane == 0 && n_tiles > 0 && !a.debug_skip_producer) {
      int it = 2;  // Q, K_0 and V_0 went out during the set-up
      for (int j = 1; j < n_tiles; ++j) {
        bool ok = true;
        for (int kind = 0; kind < 2; ++kind, ++it) {
          const int s = it % NSTAGE;
          const uint32_t ph = (it / NSTAGE) & 1;
          if (!mbar_wait<kWaitParked>(bar_kv_empty(s), ph ^ 1u, ctl)) {
            ok = false;
            break;
          }
          H3_TRACE(kind == 0 ? kEvProdK : kEvProdV, j);
          mbar_arrive_expect_tx(bar_kv_full(s), C::kTileBytes);
          const CUtensorMap* m = kind == 0 ? &a.tm_k : &a.tm_v;
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d(sKV + s * C::kTileBytes + c * C::kChunkBytes, m, bar_kv_full(s), c * 64,
                        kvh, j * kBlockN, b);
          if (kind == 1 && j == j_pad) st_release_cta(pad_issued, 1u);
        }
        if (!ok) break;
      }
      // Drain: every issued copy has landed before the CTA can retire.
      mbar_wait_drain(bar_q_full, 0, a.wait_limit_ns);
      const int first = it > NSTAGE ? it - NSTAGE : 0;
      for (int i = first; i < it; ++i)
        mbar_wait_drain(bar_kv_full(i % NSTAGE), (i / NSTAGE) & 1, a.wait_limit_ns);
    }
  } else if (warp == C::kMmaWarp + 1) {
    // ======================= padding rows of the tile straddling kv_len ====
    if (j_pad >= 0) {
      const int it_v = 2 * j_pad + 1;  // load index of V_{j_pad}
      const bool ok = __all_sync(0xFFFFFFFFu, count_wait_sleep(pad_issued, 1u, ctl) &&
                                                  mbar_wait<kWaitParked>(bar_kv_full(it_v % NSTAGE), (it_v / NSTAGE) & 1, ctl));
      if (ok) {  // V tile landed; its stage is refilled only after O += P V of it
        zero_padding_rows<D>(sKV + (it_v % NSTAGE) * C::kTileBytes, kv_lim % kBlockN, lane, 32);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_v_clean);
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ======================= MMA issuer ====================================
    if (lane == 0 && n_tiles > 0) {
      bool ok = mbar_wait<kWaitParked>(bar_q_full, 0, ctl);
      tc_fence_after();
      if constexpr (C::kSepP) {
        // S = Q K_0^T; then per key tile j: S = Q K_{j+1}^T once the softmax
        // has read S_j out, and O += P_j V_j (A = P in its own columns).
        // Ring positions: K_j at 2j, V_j at 2j + 1.
        auto issue_qk = [&](int j) -> bool {
          const int s = (2 * j) % NSTAGE;
          if (!mbar_wait<kWaitParked>(bar_kv_full(s), ((2 * j) / NSTAGE) & 1, ctl)) return false;
          if (j > 0 && !mbar_wait<kWaitParked>(bar_s_read, (j - 1) & 1, ctl)) return false;
          tc_fence_after();
          H3_TRACE(kEvMmaQK0, j);
          const uint32_t kb = sKV + s * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
            mma_ss(tmem, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024), C::kIdescQK,
                   kk > 0 ? 1u : 0u);
          }
          tc_commit(bar_s_full(0));
          tc_commit(bar_kv_empty(s));
          return true;
        };
        ok = ok && issue_qk(0);
        for (int j = 0; ok && j < n_tiles; ++j) {
          if (j + 1 < n_tiles && !(ok = issue_qk(j + 1))) break;
          const int s = (2 * j + 1) % NSTAGE;
          if (!(ok = mbar_wait<kWaitParked>(bar_kv_full(s), ((2 * j + 1) / NSTAGE) & 1, ctl))) break;
          if (j == j_pad && !(ok = mbar_wait<kWaitParked>(bar_v_clean, 0, ctl))) break;  // padding rows zeroed
          if (!(ok = mbar_wait<kWaitParked>(bar_p_ready(0), j & 1, ctl))) break;
          H3_TRACE(kEvMmaPV0, j);
          tc_fence_after();
          const uint32_t vb = sKV + s * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk)
            mma_ts(tmem + C::kColO, tmem + C::kColP + kk * 8, sdesc_sw128(vb + kk * 2048, C::kChunkBytes, 1024),
                   C::kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
          tc_commit(bar_pv_done(0));
          tc_commit(bar_kv_empty(s));
        }
      } else {
      int it = 0;
      for (int j = 0; ok && j < n_tiles; ++j) {
        // S_q = Q_q K_j^T
        {
          const int s = it % NSTAGE;
          const uint32_t ph = (it / NSTAGE) & 1;
          ++it;
          if (!(ok = mbar_wait<kWaitParked>(bar_kv_full(s), ph, ctl))) break;
          H3_TRACE(kEvMmaK, j);
          tc_fence_after();
          for (int q = 0; q < NQ; ++q) {
            if (j > 0) {
              if (!(ok = mbar_wait<kWaitParked>(bar_pv_done(q), (j - 1) & 1, ctl))) break;
              tc_fence_after();
            }
            H3_TRACE(kEvMmaQK0 + q, j);
            const uint32_t qa = sQ + q * C::kTileBytes;
            const uint32_t kb = sKV + s * C::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
              mma_ss(tmem + q * 128, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                     C::kIdescQK, kk > 0 ? 1u : 0u);
            }
            tc_commit(bar_s_full(q));
          }
          if (!ok) break;
          tc_commit(bar_kv_empty(s));
        }
        // O_q += P_q V_j
        {
          const int s = it % NSTAGE;
          const uint32_t ph = (it / NSTAGE) & 1;
          ++it;
          if (!(ok = mbar_wait<kWaitParked>(bar_kv_full(s), ph, ctl))) break;
          if (j == j_pad && !(ok = mbar_wait<kWaitParked>(bar_v_clean, 0, ctl))) break;  // padding rows zeroed
          H3_TRACE(kEvMmaV, j);
          tc_fence_after();
          const uint32_t vb = sKV + s * C::kTileBytes;
          for (int q = 0; q < NQ; ++q) {
            if (!(ok = mbar_wait<kWaitParked>(bar_p_ready(q), j & 1, ctl))) break;
            H3_TRACE(kEvMmaPV0 + q, j);
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kBlockN / 16; ++kk) {
              mma_ts(tmem + C::kColO + q * D, tmem + q * 128 + kk * 8,
                     sdesc_sw128(vb + kk * 2048, C::kChunkBytes, 1024), C::kIdescPV,
                     (j > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(bar_pv_done(q));
          }
          if (!ok) break;
          tc_commit(bar_kv_empty(s));
        }
      }
      }
      // Drain every MMA issued by this thread before tensor memory is freed.
      tc_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0, a.wait_limit_ns);
    }
   }
  } else {
    if constexpr (C::kRebalance) regs_inc<C::kSoftRegs>();
    // ======================= softmax / correction / epilogue ===============
    const int q = warp >> 2;         // query tile of this warpgroup
    const int wq = warp & 3;         // lane quarter of tensor memory
    const int t = wq * 32 + lane;    // row within the tile
    const int row = q0 + q * kBlockM + t;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + q * 128;
    const uint32_t tO = tmem + lane_off + C::kColO + q * D;
    const float sl = a.scale_log2;
    const int64_t bit_words = (a.Sk + 31) / 32;
    float m_ref = -INFINITY;  // running max in scaled (log2) units
    float l = 0.0f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      ok = mbar_wait<kWaitParked>(bar_s_full(q), j & 1, ctl);
      if (t == 0) H3_TRACE(kEvSmS0 + 4 * q, j);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
      if (t == 0) H3_TRACE(kEvSmLd0 + 4 * q, j);
      float s[kBlockN];
#pragma unroll
      for (int c = 0; c < kBlockN; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);

      const int kbase = j * kBlockN;
      const bool need_mask = (kbase + kBlockN > kv_lim) ||
                             (causal && kbase + kBlockN - 1 > q0 + q * kBlockM) || a.bits;
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
        for (int c = 0; c < kBlockN; ++c) {
          const bool allowed = (c < lim) && ((wbits[c >> 5] >> (c & 31)) & 1u);
          s[c] = allowed ? s[c] : -INFINITY;
        }
      }
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
        // O_q holds every earlier product once O_q += P V of the previous
        // tile has completed (P over S: before this tile's S_q was issued, so
        // the wait returns at once; separate P: it may still be running).
        ok = mbar_wait<kWaitParked>(bar_pv_done(q), (j - 1) & 1, ctl);
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
      const float mu = (m_ref == -INFINITY) ? 0.0f : m_ref;
      // p = exp2(s * scale*log2e - m): packed FMA, ex2, packed row-sum
      float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t p[2][32];
#pragma unroll
      for (int c = 0; c < kBlockN; c += 2) {
        float t0, t1;
        ffma2(t0, t1, s[c], s[c + 1], sl, sl, -mu, -mu);
        const float p0 = ex2(t0);
        const float p1 = ex2(t1);
        const int a2 = ((c >> 1) & 3) * 2;
        fadd2(ls[a2], ls[a2 + 1], ls[a2], ls[a2 + 1], p0, p1);
        p[c >> 6][(c >> 1) & 31] = pack_bf16x2(p0, p1);
      }
      l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      if (t == 0) H3_TRACE(kEvSmExp0 + 4 * q, j);
      if constexpr (C::kSepP) {
        // S is read out: the next tile's scores may overwrite it.  P's own
        // buffer is free once O += P V of the previous tile has completed.
        tc_fence_before();
        mbar_arrive(bar_s_read);
        if (j > 0) {
          ok = mbar_wait<kWaitParked>(bar_pv_done(q), (j - 1) & 1, ctl);
          if (!__all_sync(0xFFFFFFFFu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        tmem_st32(tmem + lane_off + C::kColP, p[0]);
        tmem_st32(tmem + lane_off + C::kColP + 32, p[1]);
      } else {
        tmem_st32(tS, p[0]);
        tmem_st32(tS + 32, p[1]);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p_ready(q));
      if (t == 0) H3_TRACE(kEvSmArr0 + 4 * q, j);
    }
    // ---- epilogue: O / l -> bf16 ------------------------------------------
    if (ok && n_tiles > 0) {
      ok = mbar_wait<kWaitParked>(bar_pv_done(q), (n_tiles - 1) & 1, ctl);
      ok = __all_sync(0xFFFFFFFFu, ok);
      tc_fence_after();
    }
    if (ok) {
      // o = O / l as bf16, staged over this query tile's Q in shared memory
      // (every Q K^T has completed once the last P V has) in the 128-byte
      // swizzled layout of the o map's box, then one TMA store of the tile;
      // rows past Sq lie outside the tensor and are not written.  One row
      // per thread straight to global memory writes 32 rows apart per warp
      // instruction: cross-attention against 512 keys ran 815 vs 952 TFLOP/s.
      const bool zero_row = row >= q_lim || n_tiles == 0 || !(l > 0.0f);
      const float inv = zero_row ? 0.0f : 1.0f / l;
      const uint32_t sO = sQ + q * C::kTileBytes;
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
        const uint32_t rowp = sO + (c >> 1) * C::kChunkBytes + t * 128;
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
      mbar_arrive(bar_o_staged(q));
      if (t == 0 && mbar_wait<kWaitParked>(bar_o_staged(q), 0, ctl)) {
        for (int c = 0; c < C::kChunks; ++c)
          tma_store_4d(&a.tm_o, sO + c * C::kChunkBytes, c * 64, h, q0 + q * kBlockM, b);
        bulk_commit_group();
        bulk_wait_group_read0();  // the shared-memory source is read before the CTA retires
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemAlloc);
  }
}

#include "attn_pipe.cuh"
#include "attn_persist.cuh"
#include "attn_wide.cuh"
#include "attn_chain.cuh"

template <int D, int NQ, int NSTAGE, int CTAS = 1>
cudaError_t launch_cfg(const AttnArgs& a, cudaStream_t stream) {
  using C = Cfg<D, NQ, NSTAGE, CTAS>;
  auto kern = attn_fwd_kernel<D, NQ, NSTAGE, CTAS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int rows_per_cta = NQ * kBlockM;
  dim3 grid((a.Sq + rows_per_cta - 1) / rows_per_cta, a.Hq, a.B);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

#ifdef H3ATTN_TRACE
extern "C" int h3attn_trace_read(unsigned long long* dst, int n) {
  const int total = kNumEv * kTraceTiles;
  if (n < total) return -1;
  return cudaMemcpyFromSymbol(dst, g_trace, sizeof(unsigned long long) * total) == cudaSuccess ? total : -2;
}
#endif

int* status_word_ptr() {
  static int* cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cache[dev]) {
    int* p = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_status_word) != cudaSuccess) return nullptr;
    cache[dev] = p;
  }
  return cache[dev];
}

namespace {
// Clears the status word if it still holds `seen`: a report that another
// stream's kernel wrote after the read is kept for the next check.
__global__ void clear_status_if_kernel(int seen) { atomicCAS(&g_status_word, seen, 0); }
}  // namespace

// The read and the conditional clear both run in the order of `stream`.
int read_and_clear_status(cudaStream_t stream, int* value) {
  int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_status_word, sizeof(int), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return 1;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return 1;
  if (v != 0) {
    clear_status_if_kernel<<<1, 1, 0, stream>>>(v);
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(stream) != cudaSuccess) return 1;
  }
  *value = v;
  return 0;
}

// Split-key tail.  With units of equal length and one resident CTA per SM,
// the last U mod #SMs units run as a wave of their own while the other SMs
// idle.  The plan keeps the first U - r units whole and cuts each of the last
// r units into P = min(#SMs / r, key tiles / 2) key ranges, so that the tail
// runs on r * P SMs at once.  Only for the one-query-tile kernel's dense
// path without causal masks (under a causal mask the last units launched are
// already the shortest ones, and per-sample causal flags are device data).
SplitPlan plan_split(const AttnArgs& a) {
  SplitPlan p{0, 0, 0, 0};
  const bool pipe = (a.D == 64 || a.D == 128) &&
                    (a.kernel == 1 || (a.kernel == 0 && a.D == 128 && a.Sk >= kOneTileMinKeys));
  if (!pipe || a.win_ct > 0 || a.causal || a.causal_b) return p;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return p;
  const int64_t units = static_cast<int64_t>((a.Sq + kBlockM - 1) / kBlockM) * a.Hq * a.B;
  const int64_t r = units % sms;
  if (r == 0) return p;
  const int64_t n_max = (a.Sk + kBlockN - 1) / kBlockN;
  const int64_t pieces = min(static_cast<int64_t>(sms) / r, max(int64_t{1}, n_max / 2));
  if (pieces < 2) return p;
  p.full = static_cast<int>(units - r);
  p.tail = static_cast<int>(r);
  p.pieces = static_cast<int>(pieces);
  p.bytes = static_cast<size_t>(r) * pieces * kBlockM * (a.D + 2) * sizeof(float);
  return p;
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream) {
  // Kernels (measured on GB300 with the workloads' shapes):
  //   1  one 128-row query tile per CTA, Q in tensor memory, two MMA-issuing
  //      threads, 7-stage ring (12 for head_dim 64): head_dim 128 from 1024
  //      keys on, and the chunked window;
  //   4  the two-tile kernel's code with one query tile per CTA, a short ring
  //      and two CTAs per SM (one CTA's prologue and epilogue overlap the
  //      other's products; at head_dim 64 P has tensor-memory columns of its
  //      own): head_dim 128 below 1024 keys, head_dim 64;
  //   5  head_dim 256: one query tile per CTA with double-buffered scores
  //      (P over its score buffer, Q and half-tiles of K/V in shared memory);
  //   2  two query tiles per CTA sharing each K/V tile (head_dim 256: one
  //      tile with a single score buffer), only on request;
  //   3  the persistent kernel (one CTA per SM over all units), on request;
  //   6  head_dim 128: one CTA per SM chaining its work units (a unit's Q
  //      hand-off and epilogue run on warps of their own beside the next
  //      unit's tiles), on request.
  // a.kernel: 0 = by shape, else the kernel above (head dims it lacks fall
  // back to the shape rule's next choice).
  if (a.split_pieces > 0) {  // planned by plan_split: the one-query-tile kernel
    if (a.D == 64) return launch_pipe<64, 12>(a, stream);
    if (a.D == 128) return launch_pipe<128, 7>(a, stream);
    return cudaErrorInvalidValue;
  }
  if (a.kernel == 6 && a.D == 128 && a.win_ct == 0) return launch_chain<6>(a, stream);
  if ((a.kernel == 5 && a.D != 256) || a.kernel == 6) {  // head dims without that kernel: the shape rule below
    AttnArgs b = a;
    b.kernel = 0;
    return launch_attention(b, stream);
  }
  if (a.kernel == 3 && a.win_ct == 0) {
    if (a.D == 64) return launch_persist<64, 12>(a, stream);
    if (a.D == 128) return launch_persist<128, 7>(a, stream);
  }
  const bool one_tile = a.kernel == 1 || (a.kernel == 0 && a.D == 128 && a.Sk >= kOneTileMinKeys);
  const bool two_ctas = !one_tile && a.win_ct == 0 && (a.kernel == 4 || a.kernel == 0);
  switch (a.D) {
    case 64:
      return one_tile ? launch_pipe<64, 12>(a, stream)
                      : (two_ctas ? launch_cfg<64, 1, 4, 2>(a, stream) : launch_cfg<64, 2, 8>(a, stream));
    case 128:
      return one_tile ? launch_pipe<128, 7>(a, stream)
                      : (two_ctas ? launch_cfg<128, 1, 2, 2>(a, stream) : launch_cfg<128, 2, 4>(a, stream));
    case 256:  // double-buffered scores; the two-tile kernel's code on request ("2", and "3"/"4" fall back to it)
      return (a.kernel == 0 || a.kernel == 1 || a.kernel == 5) ? launch_wide<5>(a, stream)
                                                               : launch_cfg<256, 1, 2>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace h3
