// Internal launcher interface between the C-ABI layer (api.cu) and the
// kernels.  Arguments arriving here are already validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/h3attn.h"

namespace h3 {

// Reads and clears the current device's status word (see h3attn_check_device_status).
int read_and_clear_status(int* value);

// ---- fused Q/K RMSNorm + bf16 boundary + partial RoPE (in place) ----
struct NormRopeArgs {
  uint16_t* q;
  uint16_t* k;
  const float* wq;
  const float* wk;
  const float* cos;
  const float* sin;
  int64_t rows_q;  // B * S * Hq
  int64_t rows_k;  // B * S * Hkv
  int S, Hq, Hkv, D, rotary_dim;
  float eps;
};
cudaError_t launch_qk_norm_rope(const NormRopeArgs& a, cudaStream_t stream);

// ---- dense prefill attention ----
struct AttnArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // 4-D (D, H, S, B) bf16 maps, 64-element inner box, 128B swizzle
  uint16_t* o;
  const int32_t* kv_len;
  const int32_t* q_len;
  const uint8_t* causal_b;
  const uint32_t* bits;
  int B, Sq, Sk, Hq, Hkv, D;
  int causal;
  float scale_log2;  // scale * log2(e)
  uint64_t wait_limit_ns;
  int debug_skip_producer;  // fault injection for the bounded-wait test: 1 = never load K/V
};
// Box rows of the Q/K/V maps built by the launcher.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream);

}  // namespace h3
