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
constexpr int kNormUnroll = 4;

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float round_bf16(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

template <int D>
__global__ void __launch_bounds__(kNormThreads) qk_norm_rope_kernel(NormRopeArgs a) {
  constexpr int LPR = D / 8;     // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp per load instruction
  constexpr float kInvD = 1.0f / static_cast<float>(D);
  const int lane = threadIdx.x & 31;
  const int lr = lane % LPR;  // lane within its row
  const int slot = lane / LPR;
  const int half = a.rotary_dim >> 1;
  const int hl = half >> 3;  // lanes holding one half of the rotated channels
  const int64_t total = a.rows_q + a.rows_k;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kNormThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kNormThreads) >> 5;

  // Rotation partner: lanes [0, hl) pair with [hl, 2hl) of the same row.
  const int partner = (lr < hl) ? lane + hl : (lr < 2 * hl ? lane - hl : lane);
  const int ti = (lr < hl ? lr : lr - hl) * 8;  // table column of this lane's first channel

  for (int64_t base = warp * (RPW * kNormUnroll); base < total;
       base += nwarps * (RPW * kNormUnroll)) {
    uint4 xv[kNormUnroll];
    int64_t row[kNormUnroll];
#pragma unroll
    for (int u = 0; u < kNormUnroll; ++u) {
      row[u] = base + u * RPW + slot;
      xv[u] = make_uint4(0u, 0u, 0u, 0u);
      if (row[u] < total) {
        const uint16_t* p = row[u] < a.rows_q ? a.q + row[u] * D
                                              : a.k + (row[u] - a.rows_q) * D;
        xv[u] = *reinterpret_cast<const uint4*>(p + lr * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < kNormUnroll; ++u) {
      const bool is_q = row[u] < a.rows_q;
      const int64_t r = is_q ? row[u] : row[u] - a.rows_q;
      const int heads = is_q ? a.Hq : a.Hkv;
      const float* w = is_q ? a.wq : a.wk;
      float x[8] = {bf16lo(xv[u].x), bf16hi(xv[u].x), bf16lo(xv[u].y), bf16hi(xv[u].y),
                    bf16lo(xv[u].z), bf16hi(xv[u].z), bf16lo(xv[u].w), bf16hi(xv[u].w)};
      float acc = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc = __fmaf_rn(x[e], x[e], acc);
#pragma unroll
      for (int off = LPR / 2; off >= 1; off >>= 1)
        acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, off));
      const float ms = __fmul_rn(acc, kInvD);
      const float rinv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));

      float n[8];
      if (row[u] < total) {
        const float4 w0 = *reinterpret_cast<const float4*>(w + lr * 8);
        const float4 w1 = *reinterpret_cast<const float4*>(w + lr * 8 + 4);
        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) n[e] = round_bf16(__fmul_rn(__fmul_rn(x[e], rinv), wv[e]));
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) n[e] = 0.0f;
      }
      // Exchange the boundary values with the rotation partner (exact: bf16 pairs).
      uint32_t mine[4] = {pack_bf16(n[0], n[1]), pack_bf16(n[2], n[3]), pack_bf16(n[4], n[5]),
                          pack_bf16(n[6], n[7])};
      uint32_t other[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) other[e] = __shfl_sync(0xFFFFFFFFu, mine[e], partner);
      if (row[u] >= total) continue;
      const float pn[8] = {bf16lo(other[0]), bf16hi(other[0]), bf16lo(other[1]),
                           bf16hi(other[1]), bf16lo(other[2]), bf16hi(other[2]),
                           bf16lo(other[3]), bf16hi(other[3])};
      float y[8];
      if (lr < 2 * hl) {
        const int64_t pos = (r / heads) % a.S;
        const float* ct = a.cos + pos * half + ti;
        const float* st = a.sin + pos * half + ti;
        const float4 c0 = *reinterpret_cast<const float4*>(ct);
        const float4 c1 = *reinterpret_cast<const float4*>(ct + 4);
        const float4 s0 = *reinterpret_cast<const float4*>(st);
        const float4 s1 = *reinterpret_cast<const float4*>(st + 4);
        const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
        if (lr < hl) {  // own = n_i (a), partner = n_{i+h} (b): y_i = a c - b s
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = __fmaf_rn(n[e], cv[e], -__fmul_rn(pn[e], sv[e]));
        } else {  // own = n_{i+h} (b), partner = n_i (a): y_{i+h} = b c + a s
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = __fmaf_rn(n[e], cv[e], __fmul_rn(pn[e], sv[e]));
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = n[e];
      }
      uint16_t* p = is_q ? a.q + r * D : a.k + r * D;
      *reinterpret_cast<uint4*>(p + lr * 8) =
          make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                     pack_bf16(y[6], y[7]));
    }
  }
}

template <int D>
cudaError_t launch_d(const NormRopeArgs& a, cudaStream_t stream) {
  constexpr int RPW = 32 / (D / 8);
  const int64_t total = a.rows_q + a.rows_k;
  const int64_t rows_per_block = static_cast<int64_t>(kNormThreads / 32) * RPW * kNormUnroll;
  int64_t blocks = (total + rows_per_block - 1) / rows_per_block;
  if (blocks > (1LL << 30)) blocks = 1LL << 30;  // the kernel's loop covers the rest
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
