// Fused RMSNorm -> indexed AdaLN scale/shift modulation of DiT hidden rows
// (TeleFuser PR #37 "perf(minimax-h3): optimize Ulysses attention and DiT
// kernels", section 2.5: one kernel for "RMSNorm -> indexed scale/shift
// modulation" that keeps the bf16 store/load rounding boundaries of the
// unfused norm-then-modulate path, element-wise bit-exact with it).
// Memory-bound: every row of x is read once and y written once (one warp per
// row, the row held in registers between the two passes); the scale / shift
// tables and the norm weight are small and stay in L1/L2.
//
// For a row t of C channels, with s = scale[idx[t]], h = shift[idx[t]]:
//   r = 1 / sqrt(mean_c(x_c^2) + eps)
//   n = bf16((x * r) * w)     (n = bf16(x * r) without a weight)
//   a = bf16(1 + s);  m = bf16(n * a);  y = bf16(m + h)
// Float32 operation order (reproducible bit for bit): 8-channel groups
// g = 0 .. C/8-1, group g on lane g mod 32 of the row's warp; per lane
// acc = fma(x, x, acc) over its groups in increasing g, channels in order;
// butterfly over the 32 lanes (xor 16 .. 1): acc = acc + partner;
// ms = acc / C; r = 1 / sqrt(ms + eps), each correctly rounded; every
// bf16 store rounds to nearest even.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace h3 {
namespace {

constexpr int kModWarps = 8;  // rows per CTA, one warp per row

__device__ __forceinline__ float lo16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// bf16x2 add / multiply, each result rounded once to nearest even.  For bf16
// operands this equals rounding the float32 result to bf16: a product of
// two 8-bit significands is exact in float32, and a float32 sum of two bf16
// values is exact unless their exponents differ by more than 16, where both
// roundings return the larger operand.
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// K = groups of 8 channels per lane (upper bound; groups past C/8 are skipped).
template <int K>
__global__ void __launch_bounds__(kModWarps * 32) rmsnorm_modulate_kernel(const __grid_constant__ ModArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kModWarps + (threadIdx.x >> 5);
  if (t >= a.T) return;
  const int G = a.C >> 3;
  const uint4* xr = reinterpret_cast<const uint4*>(a.x + t * a.C);
  uint4* yr = reinterpret_cast<uint4*>(a.y + t * a.C);
  const int32_t ix = a.idx ? a.idx[t] : 0;
  if (ix < 0 || ix >= a.N) {
    // no table row for this index: zeros, and the call reports an invalid argument
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int g = lane + 32 * k;
      if (g < G) yr[g] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (lane == 0) atomicExch(a.status, static_cast<int>(H3ATTN_ERR_INVALID_ARG));
    return;
  }
  uint4 xv[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int g = lane + 32 * k;
    xv[k] = g < G ? xr[g] : make_uint4(0u, 0u, 0u, 0u);
  }
  // sum of squares: this lane's groups in increasing g, channels in order
  float acc = 0.0f;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    if (lane + 32 * k < G) {
      const uint32_t w4[4] = {xv[k].x, xv[k].y, xv[k].z, xv[k].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = __fmaf_rn(lo16(w4[e]), lo16(w4[e]), acc);
        acc = __fmaf_rn(hi16(w4[e]), hi16(w4[e]), acc);
      }
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, off));
  const float ms = __fdiv_rn(acc, static_cast<float>(a.C));
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));

  const uint4* sr = reinterpret_cast<const uint4*>(a.scale + static_cast<int64_t>(ix) * a.C);
  const uint4* hr = reinterpret_cast<const uint4*>(a.shift + static_cast<int64_t>(ix) * a.C);
  const uint32_t one2 = 0x3F803F80u;  // bf16x2 (1, 1)
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int g = lane + 32 * k;
    if (g >= G) continue;
    const uint4 sv = __ldg(sr + g), hv = __ldg(hr + g);
    const uint32_t x4[4] = {xv[k].x, xv[k].y, xv[k].z, xv[k].w};
    const uint32_t s4[4] = {sv.x, sv.y, sv.z, sv.w};
    const uint32_t h4[4] = {hv.x, hv.y, hv.z, hv.w};
    float wv[8];
    if (a.w) {
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(a.w + 8 * g));
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(a.w + 8 * g + 4));
      wv[0] = w0.x; wv[1] = w0.y; wv[2] = w0.z; wv[3] = w0.w;
      wv[4] = w1.x; wv[5] = w1.y; wv[6] = w1.z; wv[7] = w1.w;
    }
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float n0, n1;
      fmul2(n0, n1, lo16(x4[e]), hi16(x4[e]), r, r);
      if (a.w) fmul2(n0, n1, n0, n1, wv[2 * e], wv[2 * e + 1]);
      const uint32_t nb = pack2(n0, n1);           // n = bf16(...)
      const uint32_t ab = add_bf16x2(one2, s4[e]);  // a = bf16(1 + s)
      const uint32_t mb = mul_bf16x2(nb, ab);       // m = bf16(n * a)
      out[e] = add_bf16x2(mb, h4[e]);               // y = bf16(m + h)
    }
    yr[g] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

template <int K>
cudaError_t launch_k(const ModArgs& a, cudaStream_t stream) {
  const int64_t blocks = (a.T + kModWarps - 1) / kModWarps;
  rmsnorm_modulate_kernel<K><<<static_cast<unsigned>(blocks), kModWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rmsnorm_modulate(const ModArgs& a, cudaStream_t stream) {
  const int per_lane = (a.C / 8 + 31) / 32;  // groups of 8 channels per lane
  if (per_lane <= 1) return launch_k<1>(a, stream);
  if (per_lane <= 2) return launch_k<2>(a, stream);
  if (per_lane <= 4) return launch_k<4>(a, stream);
  if (per_lane <= 8) return launch_k<8>(a, stream);
  if (per_lane <= 12) return launch_k<12>(a, stream);
  if (per_lane <= 16) return launch_k<16>(a, stream);
  if (per_lane <= 24) return launch_k<24>(a, stream);
  if (per_lane <= 32) return launch_k<32>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace h3
