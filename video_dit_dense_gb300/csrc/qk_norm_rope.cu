// Fused Q/K RMSNorm -> bf16 boundary -> partial rotate-half RoPE, in place or
// into separate output tensors.
//
// The step MiniMax-H3 runs on Q and K before attention (FastVideo PR #1832
// "Add FlashInfer attention backend support for MiniMax H3", section
// "Preserve H3-specific attention behavior": Q/K RMSNorm then RoPE on 96 of
// the 128 head channels; TeleFuser PR #37 "perf(minimax-h3): optimize Ulysses
// attention and DiT kernels", section 2.2: norm, BF16-compatible rounding and
// RoPE fused in one kernel).  Memory-bound: every row is read once and
// written once.
//
// Layout of the work: a row is one (token, head) vector of D bf16 channels.
// q rows ([B*S*Hq, D]) and k rows ([B*S*Hkv, D]) are contiguous, so the work
// is a list of 16 KiB chunks of whole rows.  A persistent grid walks the
// chunk list; in each CTA one producer warp streams chunks into a ring of
// shared-memory stages with 1-D bulk copies (completion on an mbarrier),
// together with the RoPE table rows of the chunk's tokens, and eight compute
// warps read rows from shared memory, compute, and store the results
// straight to global memory.  D/16 lanes own a row, each holding two groups
// of 8 channels (two 16-byte accesses): lane l < rotary_dim/16 holds a whole
// rotation pair (channels 8l.. and 8l + rotary_dim/2..), so the rotation
// needs no data from other lanes.
//
// Arithmetic (float32, fixed order -- reproducible bit for bit):
//   lane partial: acc = fma(x, x, acc) over its first group's 8 channels in
//   order, then its second group's, from 0 (first group l or D/16 + l,
//   second l + rotary_dim/16);
//   butterfly over the row's lanes (xor offsets D/32 .. 1): acc = acc + partner;
//   ms = acc * (1/D); r = 1 / sqrt(ms + eps), correctly rounded;
//   n = bf16((x * r) * w); rotation with y_i = fma(a, c, -(b*s)),
//   y_{i+h} = fma(b, c, a*s); store bf16(y) (round to nearest even).
// Explicit round-to-nearest intrinsics and packed f32x2 instructions (each
// lane rounded once) keep the compiler from contracting or reassociating.
//
// rotary_dim need only be even.  When it is not a multiple of 16 (h8 =
// floor(rotary_dim/16) in the partition above), a rotation pair can straddle
// two lanes' groups, so that instantiation (GEN) writes each row's boundary
// values n^ to a per-warp shared-memory row, then every lane rotates its 16
// channels one at a time with the partner read from that row and the
// coefficients read from global memory (same formulas, same rounding).  The
// GEN instantiation never stages table rows; its row buffers use the space
// of the table slots.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace h3 {
namespace {

constexpr int kComputeWarps = 8;
constexpr int kStages = 3;     // row stages
constexpr int kTabSlots = 6;   // RoPE table slots, released later than the rows
constexpr int kNormThreads = (kComputeWarps + 1) * 32;  // + one producer warp
constexpr int kChunkBytes = 16384;
constexpr int kUnroll = 2;  // rows per lane slot per chunk; also rows sharing one sqrt/div pass

template <int D>
struct NormCfg {
  static constexpr int LPR = D / 16;                        // lanes per row (16 channels each)
  static constexpr int RPW = 32 / LPR;                      // rows per warp per access
  static constexpr int kRows = kChunkBytes / (D * 2);       // rows per chunk
  static_assert(kRows == kComputeWarps * RPW * kUnroll, "chunk = compute warps x rows per warp");
  // Tokens whose RoPE table rows a slot holds: a chunk of kRows rows spans at
  // most 8 tokens once a token has kRows / 7 heads or more.
  static constexpr int kTabTokens = D == 256 ? 4 : 8;
  static constexpr int kTabBytes = kTabTokens * (D / 2) * 4;  // one table, rows of at most D/2 floats
  static constexpr int kSlotBytes = 2 * kTabBytes;            // cos rows, then sin rows
  static constexpr int kTabBase = kStages * kChunkBytes;
  static constexpr int kBarBase = kTabBase + kTabSlots * kSlotBytes;
  // full[kStages], empty[kStages], tab_empty[kTabSlots]
  static constexpr int kSmem = kBarBase + (2 * kStages + kTabSlots) * 8 + 16;
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// Two floats -> one bf16x2 word (round to nearest even), low half = lo.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  return f.one ? n : static_cast<uint32_t>(__umul64hi(f.M, static_cast<uint64_t>(n)));
}

__device__ __forceinline__ void chunk_of(const NormRopeArgs& a, uint32_t c, uint32_t rows_per_chunk,
                                         uint32_t n_q_chunks, bool& is_q, uint32_t& row0, uint32_t& nrows) {
  is_q = c < n_q_chunks;
  const uint32_t cc = is_q ? c : c - n_q_chunks;
  const uint32_t limit = is_q ? a.rows_q : a.rows_k;
  row0 = cc * rows_per_chunk;
  nrows = min(rows_per_chunk, limit - row0);
}

template <int D, bool GEN>
__global__ void __launch_bounds__(kNormThreads, 3) qk_norm_rope_kernel(const __grid_constant__ NormRopeArgs a) {
  using C = NormCfg<D>;
  // GEN: a warp's row buffer (RPW rows of D bf16) fits in its share of the table slots
  static_assert(kComputeWarps * (32 / (D / 16)) * D * 2 <= kTabSlots * C::kSlotBytes, "GEN row buffers");
  constexpr int LPR = C::LPR, RPW = C::RPW, U = kUnroll;
  constexpr float kInvD = 1.0f / static_cast<float>(D);
  static_assert(LPR >= U, "each row needs a lane per unrolled row for the shared sqrt/div pass");
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + C::kBarBase;
  auto bar_full = [&](int st) { return bars + 8u * st; };
  auto bar_empty = [&](int st) { return bars + 8u * (kStages + st); };
  auto bar_tab_empty = [&](int ts) { return bars + 8u * (2 * kStages + ts); };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kBarBase + (2 * kStages + kTabSlots) * 8);
  WaitCtl ctl{abort_flag, a.status, a.wait_limit_ns, static_cast<int>(H3ATTN_ERR_TIMEOUT)};

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(bar_full(st), 1);
      mbar_init(bar_empty(st), kComputeWarps);
    }
    for (int ts = 0; ts < kTabSlots; ++ts) mbar_init(bar_tab_empty(ts), kComputeWarps);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  __syncthreads();

  const uint32_t n_q_chunks = (a.rows_q + C::kRows - 1) / C::kRows;
  const uint32_t n_chunks = n_q_chunks + (a.rows_k + C::kRows - 1) / C::kRows;
  const int half = a.rotary_dim >> 1;
  // Tokens [tok0, tok0 + ntok) of a chunk; their table rows are staged with
  // the chunk when they fit and ntok <= S, so that their positions form at
  // most two runs (tok0 and ntok are recomputed by both sides).
  auto chunk_tokens = [&](bool is_q, uint32_t row0, uint32_t nrows, uint32_t& tok0, uint32_t& ntok) {
    const FastDiv& dh = is_q ? a.div_hq : a.div_hkv;
    tok0 = fdiv(row0, dh);
    ntok = fdiv(row0 + nrows - 1, dh) - tok0 + 1;
  };

  if (warp == kComputeWarps) {
    // ---------------- producer: chunk -> shared-memory stage ----------------
    if (lane == 0) {
      uint32_t it = 0;
      for (uint32_t c = blockIdx.x; c < n_chunks; c += gridDim.x, ++it) {
        const int st = it % kStages;
        const int ts = it % kTabSlots;
        if (!mbar_wait(bar_empty(st), ((it / kStages) & 1) ^ 1u, ctl)) break;
        if (!mbar_wait(bar_tab_empty(ts), ((it / kTabSlots) & 1) ^ 1u, ctl)) break;
        bool is_q;
        uint32_t row0, nrows;
        chunk_of(a, c, C::kRows, n_q_chunks, is_q, row0, nrows);
        const uint16_t* src = (is_q ? a.q_in : a.k_in) + static_cast<size_t>(row0) * D;
        uint32_t tok0, ntok;
        chunk_tokens(is_q, row0, nrows, tok0, ntok);
        const bool staged = !GEN && half > 0 && ntok <= static_cast<uint32_t>(C::kTabTokens) && ntok <= a.div_s.d;
        const uint32_t tab_bytes = staged ? ntok * half * 4 : 0u;
        const uint32_t stage = sbase + st * kChunkBytes;
        const uint32_t slot_c = sbase + C::kTabBase + ts * C::kSlotBytes;  // cos rows; sin rows follow
        mbar_arrive_expect_tx(bar_full(st), nrows * D * 2 + 2 * tab_bytes);
        bulk_load(stage, src, nrows * D * 2, bar_full(st));
        if (staged) {
          // positions tok % S: one run, or two when the chunk crosses a sample boundary
          const uint32_t pos0 = tok0 - fdiv(tok0, a.div_s) * a.div_s.d;
          const uint32_t n1 = min(ntok, a.div_s.d - pos0);
          const uint32_t b1 = n1 * half * 4;
          bulk_load(slot_c, a.cos + static_cast<size_t>(pos0) * half, b1, bar_full(st));
          bulk_load(slot_c + C::kTabBytes, a.sin + static_cast<size_t>(pos0) * half, b1, bar_full(st));
          if (n1 < ntok) {
            bulk_load(slot_c + b1, a.cos, tab_bytes - b1, bar_full(st));
            bulk_load(slot_c + C::kTabBytes + b1, a.sin, tab_bytes - b1, bar_full(st));
          }
        }
      }
      // every issued copy has landed before the CTA retires
      const uint32_t first = it > kStages ? it - kStages : 0;
      for (uint32_t i = first; i < it; ++i) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar_full(i % kStages), (i / kStages) & 1))
          if (globaltimer_ns() - t0 > a.wait_limit_ns) break;
      }
    }
    return;
  }

  // ---------------- compute warps ----------------
  // A row's LPR = D/16 lanes each hold two 8-channel groups: first g0 = lr
  // (lr < h8) or LPR + lr, second g1 = lr + h8, h8 = rotary_dim/16.  Lane
  // lr < h8 thus holds a whole rotation pair (channel i and i + half); the
  // others hold pass-through channels.  (Reading g0 then g1 is also free of
  // shared-memory bank conflicts for D = 128.)
  const uint32_t lr = lane % LPR;  // lane within its row
  const uint32_t slot = lane / LPR;
  const uint32_t row_lane0 = lane - lr;
  const uint32_t h8 = static_cast<uint32_t>(half >> 3);
  const bool rotating = lr < h8;
  const uint32_t g0 = rotating ? lr : LPR + lr, g1 = lr + h8;
  const uint32_t ti = lr * 8;  // table column of a rotating lane's channel 0

  uint32_t it = 0;
  for (uint32_t c = blockIdx.x; c < n_chunks; c += gridDim.x, ++it) {
    const int st = it % kStages;
    const bool ok = mbar_wait(bar_full(st), (it / kStages) & 1, ctl);
    if (!__all_sync(0xFFFFFFFFu, ok)) break;
    bool is_q;
    uint32_t row0, nrows;
    chunk_of(a, c, C::kRows, n_q_chunks, is_q, row0, nrows);
    const uint8_t* stage = smem + st * kChunkBytes;
    const int ts = it % kTabSlots;
    const float* tab_c = reinterpret_cast<const float*>(smem + C::kTabBase + ts * C::kSlotBytes);
    const float* tab_s = tab_c + C::kTabBytes / 4;
    uint32_t tok0, ntok;
    chunk_tokens(is_q, row0, nrows, tok0, ntok);
    const bool staged = !GEN && half > 0 && ntok <= static_cast<uint32_t>(C::kTabTokens) && ntok <= a.div_s.d;

    uint4 xa[U], xb[U];
    uint32_t lrow[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      lrow[u] = (warp * U + u) * RPW + slot;
      const uint8_t* rp = stage + lrow[u] * (D * 2);
      const bool live = lrow[u] < nrows;
      xa[u] = live ? *reinterpret_cast<const uint4*>(rp + g0 * 16) : make_uint4(0u, 0u, 0u, 0u);
      xb[u] = live ? *reinterpret_cast<const uint4*>(rp + g1 * 16) : make_uint4(0u, 0u, 0u, 0u);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty(st));  // the stage may be refilled

    // Sum of squares: g0's channels then g1's in order, then the butterfly.
    float acc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t w[8] = {xa[u].x, xa[u].y, xa[u].z, xa[u].w, xb[u].x, xb[u].y, xb[u].z, xb[u].w};
      float t = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float x0 = bf16lo(w[e]), x1 = bf16hi(w[e]);
        t = __fmaf_rn(x0, x0, t);
        t = __fmaf_rn(x1, x1, t);
      }
      acc[u] = t;
    }
#pragma unroll
    for (int off = LPR / 2; off >= 1; off >>= 1) {
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = __fadd_rn(acc[u], __shfl_xor_sync(0xFFFFFFFFu, acc[u], off));
    }
    // r = 1/sqrt(ms + eps): lane lr of a row evaluates it for unrolled row
    // lr % U (one IEEE sqrt and divide per lane instead of U), then every
    // lane fetches the value of each of its rows.  Same operations per row.
    float mine = acc[0];
#pragma unroll
    for (int u = 1; u < U; ++u) mine = (lr % U) == static_cast<uint32_t>(u) ? acc[u] : mine;
    const float r_mine = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(mine, kInvD), a.eps)));
    float rinv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) rinv[u] = __shfl_sync(0xFFFFFFFFu, r_mine, row_lane0 + u);

    const float* wp = is_q ? a.wq : a.wk;
    const float4 wa0 = __ldg(reinterpret_cast<const float4*>(wp + g0 * 8));
    const float4 wa1 = __ldg(reinterpret_cast<const float4*>(wp + g0 * 8 + 4));
    const float4 wb0 = __ldg(reinterpret_cast<const float4*>(wp + g1 * 8));
    const float4 wb1 = __ldg(reinterpret_cast<const float4*>(wp + g1 * 8 + 4));
    const float wv[16] = {wa0.x, wa0.y, wa0.z, wa0.w, wa1.x, wa1.y, wa1.z, wa1.w,
                          wb0.x, wb0.y, wb0.z, wb0.w, wb1.x, wb1.y, wb1.z, wb1.w};
    const FastDiv& dh = is_q ? a.div_hq : a.div_hkv;
    uint16_t* gbase = is_q ? a.q_out : a.k_out;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool live = lrow[u] < nrows;
      if (!GEN && !live) continue;  // GEN: every lane takes part in the row buffer's warp syncs
      const uint32_t xw[8] = {xa[u].x, xa[u].y, xa[u].z, xa[u].w, xb[u].x, xb[u].y, xb[u].z, xb[u].w};
      // boundary values n^ = bf16((x * r) * w), kept as bf16 pairs
      uint32_t nb[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float t0, t1, n0, n1;
        fmul2(t0, t1, bf16lo(xw[e]), bf16hi(xw[e]), rinv[u], rinv[u]);
        fmul2(n0, n1, t0, t1, wv[2 * e], wv[2 * e + 1]);
        nb[e] = pack_bf16(n0, n1);
      }
      const uint32_t r = row0 + lrow[u];
      uint32_t ob[8] = {nb[0], nb[1], nb[2], nb[3], nb[4], nb[5], nb[6], nb[7]};
      if constexpr (GEN) {
        // Row buffer of this warp's row slot: the whole row of n^ values.
        uint16_t* wrow = reinterpret_cast<uint16_t*>(smem + C::kTabBase) + (warp * RPW + slot) * D;
        *reinterpret_cast<uint4*>(wrow + g0 * 8) = make_uint4(nb[0], nb[1], nb[2], nb[3]);
        *reinterpret_cast<uint4*>(wrow + g1 * 8) = make_uint4(nb[4], nb[5], nb[6], nb[7]);
        __syncwarp();
        const uint32_t tok = fdiv(r, dh);
        const size_t pos = tok - fdiv(tok, a.div_s) * a.div_s.d;
        const int rot = 2 * half;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int d = static_cast<int>((e < 8 ? g0 : g1) * 8) + (e & 7);
          if (!live || d >= rot) continue;
          const int i = d < half ? d : d - half;  // pair (n_i, n_{i+half})
          const float av = __uint_as_float(static_cast<uint32_t>(wrow[i]) << 16);
          const float bv = __uint_as_float(static_cast<uint32_t>(wrow[i + half]) << 16);
          const float cs = __ldg(a.cos + pos * half + i), sn = __ldg(a.sin + pos * half + i);
          const float y = d < half ? __fmaf_rn(av, cs, -__fmul_rn(bv, sn)) : __fmaf_rn(bv, cs, __fmul_rn(av, sn));
          const uint32_t yb = pack_bf16(y, 0.0f) & 0xFFFFu;
          uint32_t& word = ob[(e >> 1)];
          word = (e & 1) ? ((word & 0xFFFFu) | (yb << 16)) : ((word & 0xFFFF0000u) | yb);
        }
        __syncwarp();  // the row buffer is rewritten by the next unrolled row
      } else if (rotating) {
        const uint32_t tok = fdiv(r, dh);
        float4 c0, c1, s0, s1;
        if (staged) {
          const float* ct = tab_c + (tok - tok0) * half + ti;
          const float* stb = tab_s + (tok - tok0) * half + ti;
          c0 = *reinterpret_cast<const float4*>(ct);
          c1 = *reinterpret_cast<const float4*>(ct + 4);
          s0 = *reinterpret_cast<const float4*>(stb);
          s1 = *reinterpret_cast<const float4*>(stb + 4);
        } else {
          const uint32_t pos = tok - fdiv(tok, a.div_s) * a.div_s.d;
          const float* ct = a.cos + static_cast<size_t>(pos) * half + ti;
          const float* stb = a.sin + static_cast<size_t>(pos) * half + ti;
          c0 = __ldg(reinterpret_cast<const float4*>(ct));
          c1 = __ldg(reinterpret_cast<const float4*>(ct + 4));
          s0 = __ldg(reinterpret_cast<const float4*>(stb));
          s1 = __ldg(reinterpret_cast<const float4*>(stb + 4));
        }
        const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
        // pair (a, b) = (n_i, n_{i+half}):  y_i = fma(a, c, -(b*s)) with
        // -(b*s) = b*(-s) exactly;  y_{i+half} = fma(b, c, a*s)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a0 = bf16lo(nb[e]), a1 = bf16hi(nb[e]);
          const float b0 = bf16lo(nb[4 + e]), b1 = bf16hi(nb[4 + e]);
          float t0, t1, u0, u1, y0, y1, z0, z1;
          fmul2(t0, t1, b0, b1, -sv[2 * e], -sv[2 * e + 1]);
          ffma2(y0, y1, a0, a1, cv[2 * e], cv[2 * e + 1], t0, t1);
          fmul2(u0, u1, a0, a1, sv[2 * e], sv[2 * e + 1]);
          ffma2(z0, z1, b0, b1, cv[2 * e], cv[2 * e + 1], u0, u1);
          ob[e] = pack_bf16(y0, y1);
          ob[4 + e] = pack_bf16(z0, z1);
        }
      }
      if (!live) continue;
      uint16_t* orow = gbase + static_cast<size_t>(r) * D;
      *reinterpret_cast<uint4*>(orow + g0 * 8) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
      *reinterpret_cast<uint4*>(orow + g1 * 8) = make_uint4(ob[4], ob[5], ob[6], ob[7]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_tab_empty(ts));  // this warp is done with the table slot
  }
}

template <int D, bool GEN>
cudaError_t launch_d(const NormRopeArgs& a, cudaStream_t stream) {
  using C = NormCfg<D>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(qk_norm_rope_kernel<D, GEN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t chunks = (static_cast<int64_t>(a.rows_q) + C::kRows - 1) / C::kRows +
                         (static_cast<int64_t>(a.rows_k) + C::kRows - 1) / C::kRows;
  int64_t blocks = static_cast<int64_t>(sms) * 3;  // three resident CTAs per SM
  if (blocks > chunks) blocks = chunks;
  if (blocks == 0) return cudaSuccess;
  qk_norm_rope_kernel<D, GEN><<<static_cast<unsigned>(blocks), kNormThreads, C::kSmem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qk_norm_rope(const NormRopeArgs& a, cudaStream_t stream) {
  const bool gen = (a.rotary_dim % 16) != 0;  // rotation pairs may straddle two lanes
  switch (a.D) {
    case 64: return gen ? launch_d<64, true>(a, stream) : launch_d<64, false>(a, stream);
    case 128: return gen ? launch_d<128, true>(a, stream) : launch_d<128, false>(a, stream);
    case 256: return gen ? launch_d<256, true>(a, stream) : launch_d<256, false>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace h3
