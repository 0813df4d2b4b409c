// Internal launcher interface between the C-ABI layer (api.cu) and the
// kernels.  Arguments arriving here are already validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/h3attn.h"

namespace h3 {

// Reads the current device's status word in the order of `stream`, then
// clears it only if it still holds the value read (see
// h3attn_check_device_status).  Returns nonzero on a CUDA error.
int read_and_clear_status(cudaStream_t stream, int* value);
// Device address of the current device's status word (nullptr on failure).
int* status_word_ptr();

// ---- fused Q/K RMSNorm + bf16 boundary + partial RoPE (in place or out of place) ----
// Division of 32-bit unsigned integers by a runtime constant d with one
// 64x64 multiply-high: q = floor(M * n / 2^64), M = floor((2^64 - 1) / d) + 1,
// exact for every 32-bit n (Lemire, Kaser and Kurz, "Faster remainder by
// direct computation", Software: Practice and Experience 49(6), 2019).
// d == 1 is handled by the caller-visible flag `one`.
struct FastDiv {
  uint64_t M;
  uint32_t d;
  uint32_t one;
};
inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d;
  f.one = d == 1 ? 1u : 0u;
  f.M = d == 1 ? 0ull : (~0ull) / d + 1ull;
  return f;
}

struct NormRopeArgs {
  const uint16_t* q_in;   // rows read (== q_out / k_out for the in-place call)
  const uint16_t* k_in;
  uint16_t* q_out;        // rows written
  uint16_t* k_out;
  const float* wq;
  const float* wk;
  const float* cos;
  const float* sin;
  uint32_t rows_q;  // B * S * Hq   (host guarantees rows_q + rows_k < 2^31)
  uint32_t rows_k;  // B * S * Hkv
  FastDiv div_hq, div_hkv, div_s;  // row -> token = row / H, position = token % S
  int D, rotary_dim;
  float eps;
  int* status;             // device status word (bounded-wait timeouts)
  uint64_t wait_limit_ns;  // per-wait limit
};
cudaError_t launch_qk_norm_rope(const NormRopeArgs& a, cudaStream_t stream);

// ---- RMSNorm -> indexed AdaLN scale/shift modulation ----
struct ModArgs {
  const uint16_t* x;      // [T, C] bf16
  uint16_t* y;            // [T, C] bf16 (may be x)
  const float* w;         // [C] or nullptr
  const uint16_t* scale;  // [N, C] bf16
  const uint16_t* shift;  // [N, C] bf16
  const int32_t* idx;     // [T] or nullptr (row 0 for every token)
  int64_t T;
  int C, N;
  float eps;
  int* status;            // device status word (out-of-range index, timeout)
  uint64_t wait_limit_ns; // per-wait limit
};
// Largest C: a 16 KiB row per shared-memory stage, at least two stages per CTA.
constexpr int kModMaxChannels = 8192;
cudaError_t launch_rmsnorm_modulate(const ModArgs& a, cudaStream_t stream);

// ---- dense prefill attention ----
struct AttnArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // 4-D (D, H, S, B) bf16 maps, 64-element inner box, 128B swizzle
  CUtensorMap tm_o;              // the same over o (epilogues that store a staged tile with TMA)
  const uint16_t* q_ptr;         // q itself (kernels that stage Q through registers)
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
  // 0 = choose by head dim and key length; 1 = one query tile per CTA (Q in tensor memory),
  // 2 = two query tiles per CTA, 3 = persistent (one CTA per SM), 4 = one query tile, two CTAs per SM,
  // 5 = head dim 256 with double-buffered scores, 6 = head dim 128, one CTA per SM chaining its units
  int kernel;
  // chunked window (self-attention, one-query-tile kernel only): tokens per
  // chunk (0 = dense), anchor tokens, radius in chunks
  int win_ct, win_af, win_r;
  // Split-key tail (one-query-tile kernel, dense): the first split_full work
  // units run whole; each of the remaining split_tail units is cut into
  // split_pieces key ranges whose partial (O, m, l) go to split_ws, and a
  // combine kernel writes their output rows.  split_pieces == 0: no split.
  int split_full, split_tail, split_pieces;
  float* split_ws;
};
// Plan of the split-key tail for a prefill call on the current device (all
// zero when the call runs without it) and the workspace bytes it needs.
struct SplitPlan {
  int full, tail, pieces;
  size_t bytes;
};
SplitPlan plan_split(const AttnArgs& a);
// Key length from which the one-query-tile kernel is chosen (head_dim 64/128).
constexpr int kOneTileMinKeys = 1024;
// Box rows of the Q/K/V maps built by the launcher.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream);

}  // namespace h3
