// Fused RMSNorm -> indexed AdaLN scale/shift modulation of DiT hidden rows
// (TeleFuser PR #37 "perf(minimax-h3): optimize Ulysses attention and DiT
// kernels", section 2.5: one kernel for "RMSNorm -> indexed scale/shift
// modulation" that keeps the bf16 store/load rounding boundaries of the
// unfused norm-then-modulate path, element-wise bit-exact with it).
// Memory-bound: every row of x is read once (bulk-copied into a shared-memory
// ring by a producer warp) and y written once; the scale / shift tables and
// the norm weight are small and stay in L1/L2.
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

// Count of rows the producer has issued, published with release semantics
// (shared memory, CTA scope), and the bounded wait on it.
__device__ __forceinline__ void st_release_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ bool issued_wait(uint32_t addr, uint32_t need, const WaitCtl& ctl) {
  if (ld_acquire_u32(addr) >= need) return true;
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_u32(addr) < need) {
    if (*ctl.abort_flag) return false;
    if (globaltimer_ns() - t0 > ctl.limit_ns) {
      *ctl.abort_flag = 1u;
      atomicExch(ctl.status, ctl.timeout_code);
      return false;
    }
  }
  return true;
}

// A persistent CTA streams a contiguous range of rows through a ring of NS
// one-row shared-memory stages: one producer warp bulk-copies rows ahead as
// stages free up, and compute warp w takes rows w, w + W, ... of the CTA's
// range.  The ring keeps up to NS - W rows of HBM reads in flight per CTA
// beyond the rows the compute warps hold.  With stage_w the float32 norm
// weight is copied once into shared memory after the ring, so the per-row
// loads through L1 are only the scale / shift rows.
//
// Phase aliasing.  Warp w waits for row i as fill f = i / NS of stage
// i % NS.  A parity wait passes when fill f has landed, but also when only
// fills up to f - 2 have (fill f - 1, row i - NS, still in flight): row
// i - NS belongs to another warp unless NS == W, and bulk copies complete in
// any order, so a warp could take the stale row i - 2 NS.  The producer
// therefore publishes how many rows it has issued, and warp w first waits
// for row i to be issued: that happens only after row i - NS was consumed,
// hence landed, so the parity then names fill f alone.  This holds for any
// NS; the launcher's NS >= W + 2 is for read-ahead.
template <int W>
__global__ void __launch_bounds__((W + 1) * 32, W == 8 ? 4 : 2)
    rmsnorm_modulate_kernel(const __grid_constant__ ModArgs a, int NS, int stage_w) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int C = a.C, G = C >> 3;
  const uint32_t row_bytes = static_cast<uint32_t>(C) * 2;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + NS * row_bytes;
  auto bar_full = [&](int st) { return bars + 8u * st; };
  auto bar_empty = [&](int st) { return bars + 8u * (NS + st); };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + NS * row_bytes + 16 * NS);
  const uint32_t issued = smem_u32(smem + NS * row_bytes + 16 * NS + 4);  // rows issued by the producer
  // staged norm weight: after the barriers and the abort word (16-byte aligned: row_bytes and 16 NS are)
  float* wsm = reinterpret_cast<float*>(smem + NS * row_bytes + 16 * NS + 16);
  WaitCtl ctl{abort_flag, a.status, a.wait_limit_ns, static_cast<int>(H3ATTN_ERR_TIMEOUT)};
  // Launched with programmatic stream serialization: the next kernel of the
  // stream may be scheduled as soon as every CTA of this grid has started
  // (its CTAs take an SM once one of these exits), and this grid touches
  // global memory only after the previous kernel of the stream has completed
  // (griddepcontrol.wait below; a no-op without the dependency).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int st = 0; st < NS; ++st) {
      mbar_init(bar_full(st), 1);
      mbar_init(bar_empty(st), 1);
    }
    *abort_flag = 0u;
    *reinterpret_cast<volatile uint32_t*>(smem + NS * row_bytes + 16 * NS + 4) = 0u;
    fence_barrier_init();
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (stage_w) {
    for (int i = threadIdx.x; i < (C >> 2); i += blockDim.x)
      reinterpret_cast<float4*>(wsm)[i] = __ldg(reinterpret_cast<const float4*>(a.w) + i);
  }
  __syncthreads();
  // rows of this CTA: a contiguous range t_i = r0 + i, i < n (neighbouring
  // rows share their table row, which then stays in L1)
  const int64_t per = (a.T + gridDim.x - 1) / gridDim.x;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * per;
  const int64_t n = a.T > r0 ? min(per, a.T - r0) : 0;

  if (warp == W) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int64_t i = 0;
      for (; i < n; ++i) {
        const int st = static_cast<int>(i % NS);
        if (!mbar_wait(bar_empty(st), static_cast<uint32_t>((i / NS) & 1) ^ 1u, ctl)) break;
        mbar_arrive_expect_tx(bar_full(st), row_bytes);
        bulk_load(sbase + st * row_bytes, a.x + (r0 + i) * C, row_bytes, bar_full(st));
        st_release_u32(issued, static_cast<uint32_t>(i + 1));
      }
      // every issued copy has landed before the CTA retires
      for (int64_t k = i > NS ? i - NS : 0; k < i; ++k) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar_full(static_cast<int>(k % NS)), static_cast<uint32_t>((k / NS) & 1)))
          if (globaltimer_ns() - t0 > a.wait_limit_ns) break;
      }
    }
    return;
  }

  // ---------------- compute warps ----------------
  const uint32_t one2 = 0x3F803F80u;  // bf16x2 (1, 1)
  for (int64_t i = warp; i < n; i += W) {
    const int st = static_cast<int>(i % NS);
    const bool ok = issued_wait(issued, static_cast<uint32_t>(i + 1), ctl) &&
                    mbar_wait(bar_full(st), static_cast<uint32_t>((i / NS) & 1), ctl);
    if (!__all_sync(0xFFFFFFFFu, ok)) break;
    const int64_t t = r0 + i;
    const uint4* xs = reinterpret_cast<const uint4*>(smem + st * row_bytes);
    uint4* yr = reinterpret_cast<uint4*>(a.y + t * C);
    const int32_t ix = a.idx ? a.idx[t] : 0;
    if (ix < 0 || ix >= a.N) {
      // no table row for this index: zeros, and the call reports an invalid argument
      for (int g = lane; g < G; g += 32) yr[g] = make_uint4(0u, 0u, 0u, 0u);
      if (lane == 0) atomicExch(a.status, static_cast<int>(H3ATTN_ERR_INVALID_ARG));
    } else {
      // sum of squares: this lane's groups in increasing g, channels in order
      float acc = 0.0f;
      for (int g = lane; g < G; g += 32) {
        const uint4 v = xs[g];
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc = __fmaf_rn(lo16(w4[e]), lo16(w4[e]), acc);
          acc = __fmaf_rn(hi16(w4[e]), hi16(w4[e]), acc);
        }
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, off));
      const float ms = __fdiv_rn(acc, static_cast<float>(C));
      const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));
      const uint4* sr = reinterpret_cast<const uint4*>(a.scale + static_cast<int64_t>(ix) * C);
      const uint4* hr = reinterpret_cast<const uint4*>(a.shift + static_cast<int64_t>(ix) * C);
#pragma unroll 2
      for (int g = lane; g < G; g += 32) {
        const uint4 xv = xs[g], sv = __ldg(sr + g), hv = __ldg(hr + g);
        const uint32_t x4[4] = {xv.x, xv.y, xv.z, xv.w};
        const uint32_t s4[4] = {sv.x, sv.y, sv.z, sv.w};
        const uint32_t h4[4] = {hv.x, hv.y, hv.z, hv.w};
        float wv[8];
        if (a.w) {
          float4 w0, w1;
          if (stage_w) {
            w0 = reinterpret_cast<const float4*>(wsm)[2 * g];
            w1 = reinterpret_cast<const float4*>(wsm)[2 * g + 1];
          } else {
            w0 = __ldg(reinterpret_cast<const float4*>(a.w + 8 * g));
            w1 = __ldg(reinterpret_cast<const float4*>(a.w + 8 * g + 4));
          }
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
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty(st));  // the stage may be refilled
  }
}

template <int W>
cudaError_t launch_with(const ModArgs& a, int ctas_per_sm, int NS, int stage_w, size_t smem, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(rmsnorm_modulate_kernel<W>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  int64_t blocks = static_cast<int64_t>(sms) * ctas_per_sm;
  if (blocks > a.T) blocks = a.T;
  // A programmatic dependent launch: back to back, the next launch's CTAs are
  // placed while this one's last rows drain (+3 % at T 32760 x C 3072).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3((W + 1) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, rmsnorm_modulate_kernel<W>, a, NS, stage_w);
}

}  // namespace

// Shape: as many compute warps per SM as the rings allow (the kernel is
// latency-bound per warp: 16 compute warps per SM reached 4.44 TB/s, 32
// reached 5.3 TB/s on T 32760 x C 3072), each ring holding at least W + 2
// rows (one per compute warp plus two of read-ahead), then the deepest ring
// that fits beside the other CTAs of the SM.  The weight is staged in
// shared memory when the shape that leaves room for it keeps at least 3/4 of
// the compute warps of the shape without it (C 3072: 28 warps with the staged
// weight measured 2.2 % faster than 32 loading it through L1).
cudaError_t launch_rmsnorm_modulate(const ModArgs& a, cudaStream_t stream) {
  constexpr int64_t kSmemPerSm = 233472;  // 228 KiB, of which 1 KiB per CTA is reserved
  constexpr int64_t kMaxNS = 48;
  const int64_t stage = static_cast<int64_t>(a.C) * 2 + 16;  // one row + its two barriers
  struct Shape {
    int W, ctas;
    int64_t NS;
  };
  const Shape shapes[] = {{16, 2, 0}, {14, 2, 0}, {8, 4, 0}, {8, 3, 0}, {16, 1, 0}, {8, 2, 0}, {8, 1, 0}};
  // first shape of the table whose ring fits beside `extra` bytes per CTA
  auto pick = [&](int64_t extra, Shape* out) {
    for (const Shape& sh : shapes) {
      const int64_t per_cta = kSmemPerSm / sh.ctas - 1024 - 16 - extra;  // ring (+ abort word and issued count, extra)
      int64_t NS = per_cta / stage;
      if (NS < sh.W + 2) continue;
      *out = {sh.W, sh.ctas, NS > kMaxNS ? kMaxNS : NS};
      return true;
    }
    return false;
  };
  const int64_t wbytes = static_cast<int64_t>(a.C) * 4;
  Shape plain{}, staged{};
  const bool has_plain = pick(0, &plain);
  const bool has_staged = a.w != nullptr && pick(wbytes, &staged);
  const bool use_staged =
      has_staged && (!has_plain || 4 * staged.W * staged.ctas >= 3 * plain.W * plain.ctas);
  if (!use_staged && !has_plain) return cudaErrorInvalidValue;  // a row larger than an SM's shared memory
  const Shape sh = use_staged ? staged : plain;
  const size_t smem = static_cast<size_t>(sh.NS * stage + 16 + (use_staged ? wbytes : 0));
  const int NS = static_cast<int>(sh.NS), sw = use_staged ? 1 : 0;
  if (sh.W == 16) return launch_with<16>(a, sh.ctas, NS, sw, smem, stream);
  if (sh.W == 14) return launch_with<14>(a, sh.ctas, NS, sw, smem, stream);
  return launch_with<8>(a, sh.ctas, NS, sw, smem, stream);
}

}  // namespace h3
