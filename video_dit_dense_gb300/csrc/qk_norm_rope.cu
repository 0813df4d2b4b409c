// Fused Q/K RMSNorm -> bf16 boundary -> partial rotate-half RoPE, in place.
//
// The step MiniMax-H3 runs on Q and K before attention (FastVideo PR #1832
// "Add FlashInfer attention backend support for MiniMax H3", section
// "Preserve H3-specific attention behavior": Q/K RMSNorm then RoPE on 96 of
// the 128 head channels; TeleFuser PR #37 "perf(minimax-h3): optimize Ulysses
// attention and DiT kernels", section 2.2: norm, BF16-compatible rounding and
// RoPE fused in one kernel).  Memory-bound: every row is read once and
// written once.
//
// Layout of the work: a row is one (token, head) vector of D bf16 channels
// (D*2 bytes).  D/8 consecutive lanes own a row, each holding 8 channels in
// one 16-byte load, so a warp covers 32*8/D rows per instruction and every
// load/store instruction of a warp touches 512 contiguous bytes.  Each warp
// keeps UNROLL such loads in flight before it computes.
//
// Arithmetic (float32, fixed order -- reproducible bit for bit):
//   lane partial: acc = fma(x, x, acc) over its 8 channels in order, from 0;
//   butterfly over the row's lanes (xor offsets D/16 .. 1): acc = acc + partner;
//   ms = acc * (1/D); r = 1 / sqrt(ms + eps), correctly rounded;
//   n = bf16((x * r) * w); rotation with y_i = fma(a, c, -(b*s)),
//   y_{i+h} = fma(b, c, a*s); store bf16(y) (round to nearest even).
// Explicit __f*_rn intrinsics keep the compiler from contracting or
// reassociating any of it.
#include <cuda_bf16.h>

#include "internal.h"

namespace h3 {
namespace {

constexpr int kNormThreads = 256;
constexpr int kNormUnroll = 4;  // rows per lane slot in flight; also the rows sharing one sqrt/div pass

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

template <int D>
__global__ void __launch_bounds__(kNormThreads) qk_norm_rope_kernel(const __grid_constant__ NormRopeArgs a) {
  constexpr int LPR = D / 8;     // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp per load instruction
  constexpr int U = kNormUnroll;
  constexpr float kInvD = 1.0f / static_cast<float>(D);
  static_assert(LPR >= U, "each row needs a lane per unrolled row for the shared sqrt/div pass");
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t lr = lane % LPR;  // lane within its row
  const uint32_t slot = lane / LPR;
  const uint32_t row_lane0 = lane - lr;
  const int half = a.rotary_dim >> 1;
  const uint32_t hl = static_cast<uint32_t>(half >> 3);  // lanes per rotated half
  const bool rotating = lr < 2 * hl;
  // Rotation partner: lanes [0, hl) pair with [hl, 2hl) of the same row.
  const uint32_t partner = lr < hl ? lane + hl : (rotating ? lane - hl : lane);
  const uint32_t ti = rotating ? (lr < hl ? lr : lr - hl) * 8 : 0;  // table column of channel 0 of this lane
  const uint32_t neg = lr < hl ? 0x80000000u : 0u;                 // y_i takes -(b*s), y_{i+h} takes +(a*s)
  const uint32_t total = a.rows_q + a.rows_k;
  const uint32_t warp = (blockIdx.x * kNormThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kNormThreads) >> 5;

  for (uint32_t base = warp * (RPW * U); base < total; base += nwarps * (RPW * U)) {
    uint4 xv[U];
    uint32_t row[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      row[u] = base + u * RPW + slot;
      xv[u] = make_uint4(0u, 0u, 0u, 0u);
      if (row[u] < total) {
        const uint16_t* p = row[u] < a.rows_q ? a.q + static_cast<size_t>(row[u]) * D
                                              : a.k + static_cast<size_t>(row[u] - a.rows_q) * D;
        xv[u] = *reinterpret_cast<const uint4*>(p + lr * 8);
      }
    }
    // Sum of squares: lane partial in channel order, then the butterfly.
    float acc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t w[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
      float t = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
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

#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool is_q = row[u] < a.rows_q;
      const uint32_t r = is_q ? row[u] : row[u] - a.rows_q;
      const float* wp = (is_q ? a.wq : a.wk) + lr * 8;
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(wp));
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(wp + 4));
      const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      const uint32_t xw[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
      // boundary values n^ = bf16((x * r) * w), kept as bf16 pairs
      uint32_t nb[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float n0 = __fmul_rn(__fmul_rn(bf16lo(xw[e]), rinv[u]), wv[2 * e]);
        const float n1 = __fmul_rn(__fmul_rn(bf16hi(xw[e]), rinv[u]), wv[2 * e + 1]);
        nb[e] = pack_bf16(n0, n1);
      }
      uint32_t pb[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) pb[e] = __shfl_sync(0xFFFFFFFFu, nb[e], partner);
      if (row[u] >= total) continue;
      uint32_t ob[4] = {nb[0], nb[1], nb[2], nb[3]};
      if (rotating) {
        const uint32_t tok = fdiv(r, is_q ? a.div_hq : a.div_hkv);
        const uint32_t pos = tok - fdiv(tok, a.div_s) * a.div_s.d;
        const float* ct = a.cos + static_cast<size_t>(pos) * half + ti;
        const float* st = a.sin + static_cast<size_t>(pos) * half + ti;
        const float4 c0 = __ldg(reinterpret_cast<const float4*>(ct));
        const float4 c1 = __ldg(reinterpret_cast<const float4*>(ct + 4));
        const float4 s0 = __ldg(reinterpret_cast<const float4*>(st));
        const float4 s1 = __ldg(reinterpret_cast<const float4*>(st + 4));
        const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float own0 = bf16lo(nb[e]), own1 = bf16hi(nb[e]);
          const float oth0 = bf16lo(pb[e]), oth1 = bf16hi(pb[e]);
          const float t0 = __uint_as_float(__float_as_uint(__fmul_rn(oth0, sv[2 * e])) ^ neg);
          const float t1 = __uint_as_float(__float_as_uint(__fmul_rn(oth1, sv[2 * e + 1])) ^ neg);
          ob[e] = pack_bf16(__fmaf_rn(own0, cv[2 * e], t0), __fmaf_rn(own1, cv[2 * e + 1], t1));
        }
      }
      uint16_t* p = is_q ? a.q + static_cast<size_t>(r) * D : a.k + static_cast<size_t>(r) * D;
      *reinterpret_cast<uint4*>(p + lr * 8) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
    }
  }
}

template <int D>
cudaError_t launch_d(const NormRopeArgs& a, cudaStream_t stream) {
  constexpr int RPW = 32 / (D / 8);
  const int64_t total = static_cast<int64_t>(a.rows_q) + a.rows_k;
  const int64_t rows_per_block = static_cast<int64_t>(kNormThreads / 32) * RPW * kNormUnroll;
  int64_t blocks = (total + rows_per_block - 1) / rows_per_block;
  if (blocks > 65536) blocks = 65536;  // the kernel's grid-stride loop covers the rest
  if (blocks == 0) return cudaSuccess;
  qk_norm_rope_kernel<D><<<static_cast<unsigned>(blocks), kNormThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qk_norm_rope(const NormRopeArgs& a, cudaStream_t stream) {
  switch (a.D) {
    case 64: return launch_d<64>(a, stream);
    case 128: return launch_d<128>(a, stream);
    case 256: return launch_d<256>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace h3
