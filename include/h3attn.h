/*
 * libh3attn -- the MiniMax-H3 / Wan video-DiT attention step on one GB300
 * (sm_103a): fused Q/K RMSNorm + bf16 boundary + partial RoPE, then dense
 * prefill attention.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensors are bf16, contiguous, in BSHD layout [batch, sequence, heads,
 *   head_dim] (FastVideo PR #1832 "Add FlashInfer attention backend support
 *   for MiniMax H3", section "Summary": query/key/value are
 *   [batch, sequence, heads, head_dim]).  bf16 is passed as raw 16-bit words.
 * - Pointers are DEVICE pointers unless stated otherwise.  The caller owns
 *   every buffer; the library allocates no per-call memory.  It keeps one
 *   4-byte device status word per device, created on the first call on that
 *   device.
 * - Every call is asynchronous on `stream` (0 = the legacy default stream).
 *   Argument errors are detected on the host and returned before anything is
 *   launched; nothing is written in that case.
 * - Device-side bounded waits: the attention kernel never spins forever.  If
 *   a pipeline wait exceeds its limit the kernel records H3ATTN_ERR_TIMEOUT
 *   in the status word and returns; h3attn_check_device_status() reports it.
 * - Inference only: there is no backward pass (FastVideo PR #1799 "Add
 *   opt-in FlashInfer attention backend for Wan", section "Implementation":
 *   grad-enabled inputs are rejected; the Python binding enforces that).
 */
#ifndef H3ATTN_H_
#define H3ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque stream handle; pass a cudaStream_t. */
typedef void* h3attn_stream_t;

typedef enum {
  H3ATTN_OK = 0,
  H3ATTN_ERR_INVALID_ARG = 1,          /* null pointer, bad size, aliasing, causal with Sq != Sk, ... */
  H3ATTN_ERR_MISALIGNED = 2,           /* a tensor pointer is not 16-byte aligned */
  H3ATTN_ERR_UNSUPPORTED_HEAD_DIM = 3, /* head_dim not in {64, 128, 256} */
  H3ATTN_ERR_UNSUPPORTED_DEVICE = 4,   /* current device is not compute capability 10.3 */
  H3ATTN_ERR_UNSUPPORTED_MASK = 5,     /* mask form that has no representation here */
  H3ATTN_ERR_LAUNCH = 6,               /* a CUDA runtime/driver call failed */
  H3ATTN_ERR_TIMEOUT = 7               /* a device-side wait hit its limit (see check_device_status) */
} h3attn_status_t;

/*
 * Attention mask descriptor.  Every field is an optional DEVICE pointer
 * (NULL = absent), indexed per batch item and never per head: the pages'
 * boolean [Q, K] custom mask is per batch item, and per-head [B, H, Q, K]
 * masks are rejected (FastVideo PR #1799, sections "Implementation" and
 * "Limitations").  The fields combine by logical AND of "may attend":
 *
 *   allowed(b, i, j) = j < Sk
 *                    and (kv_len == NULL or j < kv_len[b])          key padding
 *                    and (not causal_eff(b) or j <= i)               causal, top-left aligned
 *                    and (bits == NULL or bit (j & 31) of bits[b, i, j >> 5])
 *   causal_eff(b)    = causal argument != 0 or (causal_b != NULL and causal_b[b] != 0)
 *
 * kv_len[b] may be any int32: values <= 0 mask every key, values >= Sk mask
 * none.  K and V rows j >= kv_len[b] are padding and may hold anything
 * (NaN, Inf): they never reach the output.  Keys masked only by causal or
 * bits must hold finite K and V (their probability is zero, and 0 * NaN is
 * NaN).  A query row with no allowed key produces an all-zero output row.
 * q_len[b]: rows i >= q_len[b] of sample b are written as zeros (the
 * fixed-valid zero-tail mode of TeleFuser PR #37 "perf(minimax-h3): optimize
 * Ulysses attention and DiT kernels", sections 2.3 and 2.4).
 * bits: uint32 words, shape [B, Sq, ceil(Sk / 32)], row-major, 4-byte
 * aligned; bit value 1 = attend, and bits for j >= Sk are ignored.
 */
typedef struct {
  const int32_t* kv_len;   /* [B] valid keys per sample, or NULL */
  const int32_t* q_len;    /* [B] valid query rows per sample, or NULL */
  const uint8_t* causal_b; /* [B] per-sample causal flag, or NULL */
  const uint32_t* bits;    /* [B, Sq, ceil(Sk/32)] packed boolean mask, or NULL */
} h3attn_mask_t;

/*
 * Fused Q/K RMSNorm -> bf16 rounding boundary -> partial rotate-half RoPE,
 * IN PLACE on q and k.
 *
 * The step H3 runs on Q and K before attention: per-(token, head) RMSNorm,
 * a BF16-compatible rounding, then RoPE on the first rotary_dim channels
 * (FastVideo PR #1832, section "Preserve H3-specific attention behavior":
 * H3 rotates 96 of its 128 head channels after Q/K RMSNorm; TeleFuser PR #37
 * section 2.2, steps 1-3 of the fused kernel).  For every row x of D
 * channels at sequence position s:
 *   r      = 1 / sqrt(mean_d(x_d^2) + eps)
 *   n_d    = bf16((x_d * r) * w_d)
 *   for i < rotary_dim/2, with c = cos[s, i], t = sin[s, i], h = rotary_dim/2:
 *     y_i     = n_i * c - n_{i+h} * t
 *     y_{i+h} = n_{i+h} * c + n_i * t
 *   y_d = n_d for d >= rotary_dim;  x <- bf16(y)
 * The float32 operation order is fixed (lane partial sums of 8 channels,
 * butterfly across lanes, correctly rounded sqrt and divide, separate
 * multiplies, fused multiply-adds in the rotation, round-to-nearest-even
 * stores), so results are reproducible bit for bit.  Any even rotary_dim is
 * accepted; multiples of 16 (96 of 128 in H3) take the fast path in which a
 * lane holds whole rotation pairs, other values a slower path that rotates
 * channel by channel through shared memory (same results bit for bit as the
 * fixed order above).
 *
 * q: [B, S, Hq, D] bf16, k: [B, S, Hkv, D] bf16 (device, in place, must not
 *    overlap each other).  Either may be NULL with its head count 0 to
 *    process only the other.
 * wq, wk: [D] float32 RMSNorm weights (device), shared by all heads.
 * cos, sin: [S, rotary_dim/2] float32 (device); row = sequence position.
 *    May be NULL when rotary_dim == 0.
 * D in {64, 128, 256}; rotary_dim even with 0 <= rotary_dim <= D;
 * eps >= 0 and finite.  Every pointer 16-byte aligned (rows, weights and
 * tables alike).
 * Errors: INVALID_ARG, MISALIGNED, UNSUPPORTED_HEAD_DIM, UNSUPPORTED_DEVICE,
 * LAUNCH.
 */
h3attn_status_t h3attn_qk_norm_rope(void* q, void* k, const float* wq, const float* wk,
                                    const float* cos, const float* sin, int B, int S, int Hq,
                                    int Hkv, int D, int rotary_dim, float eps,
                                    h3attn_stream_t stream);

/*
 * The same fused Q/K RMSNorm -> bf16 boundary -> partial RoPE, written to
 * separate output tensors so that the raw q and k stay available (SGLang PR
 * #37903 "[diffusion] model: support VDN-H3 ...", section "Modifications",
 * hybrid attention module: an out-of-place fused QK-norm + RoPE, bit-equal to
 * the in-place one, lets the linear branch keep the raw q/k).  Every output
 * element is bit-identical to what h3attn_qk_norm_rope() writes in place.
 *
 * q, k: inputs as above (device, read only); q_out: [B, S, Hq, D] and
 *    k_out: [B, S, Hkv, D] bf16 outputs (device), present exactly when the
 *    matching input is.  An output may be its own input (then the call is the
 *    in-place one); any other overlap among q, k, q_out, k_out is rejected.
 * Other arguments, alignment and errors as for h3attn_qk_norm_rope().
 */
h3attn_status_t h3attn_qk_norm_rope_out(const void* q, const void* k, void* q_out, void* k_out,
                                        const float* wq, const float* wk, const float* cos,
                                        const float* sin, int B, int S, int Hq, int Hkv, int D,
                                        int rotary_dim, float eps, h3attn_stream_t stream);

/*
 * Dense prefill attention  o = softmax(q k^T * scale) v  per (batch, query
 * head), on BSHD bf16 tensors (FastVideo PR #1832, section "Summary": dense
 * non-causal self-attention with head_dim 128; FastVideo PR #1799, section
 * "Implementation": self- and cross-attention, MHA and GQA, causal,
 * padding masks as a boolean [Q, K] mask, combined with causal when both are
 * present; head dims 64, 128, 256).
 *
 * q: [B, Sq, Hq, D] bf16; k, v: [B, Sk, Hkv, D] bf16; o: [B, Sq, Hq, D] bf16
 *    (all device; o must not overlap q, k or v).  Query head h reads key/value
 *    head h / (Hq / Hkv) (GQA, contiguous groups).
 * scale: finite and > 0 (typically 1/sqrt(D)); 0, negative or non-finite
 *    values are rejected (INVALID_ARG).
 * mask: NULL (dense) or a descriptor as above.  causal: nonzero applies the
 *    causal mask to every sample; causal masking requires Sq == Sk.
 * D in {64, 128, 256}; Hq % Hkv == 0; B, Sq, Sk, Hq, Hkv >= 1 (B*Sq == 0 is
 * a no-op); B, Hq <= 65535 and ceil(Sq/128)*Hq*B < 2^31 (work units).
 * Scheduling: a work unit is 128 query rows of one batch item and head; the
 * units are launched longest (causal) first and the hardware places them on
 * the SMs as they free up (one resident CTA per SM for head dim 128 from 1024
 * keys on and for head dim 256, two for head dim 64 and for head dim 128
 * below 1024 keys).
 * Accumulation is float32 on the tensor cores; softmax in float32
 * with exp2; the output is rounded once to bf16.
 * Errors: INVALID_ARG, MISALIGNED, UNSUPPORTED_HEAD_DIM, UNSUPPORTED_DEVICE,
 * UNSUPPORTED_MASK, LAUNCH.  A device-side pipeline timeout is reported by
 * h3attn_check_device_status().
 */
h3attn_status_t h3attn_prefill(const void* q, const void* k, const void* v, void* o, int B, int Sq,
                               int Sk, int Hq, int Hkv, int D, float scale,
                               const h3attn_mask_t* mask, int causal, h3attn_stream_t stream);

/*
 * Dense prefill attention as h3attn_prefill(), with a caller-owned workspace
 * for the split-key tail.  The work units (128 query rows of one batch item
 * and head) of a long-sequence call are equal in length, and the last
 * (units mod number-of-SMs) of them would run as a partial wave of their own
 * while the other SMs idle.  With a workspace those last units are cut into
 * key ranges that run side by side on the idle SMs; each range writes its
 * unnormalised output, running max and row sum to the workspace, and a
 * combine kernel merges the ranges of a unit in a fixed order
 * (o = sum 2^(m_i - M) O_i / sum 2^(m_i - M) l_i, M = max m_i), so results
 * are deterministic.  This is the split-key (O, m, l) combination of the
 * online softmax over key blocks; the pages' own kernels run one launch per
 * batch item (FastVideo PR #1799 "Add opt-in FlashInfer attention backend for
 * Wan", section "Implementation": single prefill per item) and pack batch-1
 * long sequences (FastVideo PR #1832, section "Performance considerations").
 *
 * workspace: device memory of at least h3attn_prefill_workspace_size() bytes
 *    for the same arguments, 16-byte aligned, not overlapping q, k, v or o;
 *    its contents on entry do not matter and are overwritten.  NULL (or a
 *    size of 0 from the query) runs the call exactly as h3attn_prefill().
 *    Calls that share a workspace must be ordered (one stream, or events):
 *    the tail of one call and the combine of another would race on it.
 * The split applies to the head-dim-128 kernel from 1024 keys (and to head
 * dim 64 when that kernel is forced), without causal masks.  Other arguments
 * and errors as for h3attn_prefill(); a workspace smaller than required is
 * INVALID_ARG.
 */
h3attn_status_t h3attn_prefill_ws(const void* q, const void* k, const void* v, void* o, int B, int Sq,
                                  int Sk, int Hq, int Hkv, int D, float scale,
                                  const h3attn_mask_t* mask, int causal, void* workspace,
                                  size_t workspace_bytes, h3attn_stream_t stream);

/*
 * Workspace bytes h3attn_prefill_ws() needs for these arguments on the
 * current device (0 when the call would not split), written to *bytes.  The
 * size depends on the device's SM count; it is at most
 * SMs * 128 * (D + 2) * 4 bytes (10.1 MB for head dim 128 on 152 SMs).
 * Errors: INVALID_ARG, UNSUPPORTED_HEAD_DIM, UNSUPPORTED_DEVICE, LAUNCH.
 */
h3attn_status_t h3attn_prefill_workspace_size(int B, int Sq, int Sk, int Hq, int Hkv, int D,
                                              const h3attn_mask_t* mask, int causal, size_t* bytes);

/*
 * Dense prefill attention that allocates nothing, for callers that cannot
 * allocate device memory.  The pages have no counterpart to this call; it
 * exists for hosts that must not call cudaMalloc (or let a library do so):
 * runtimes and plugin interfaces that own every device allocation and plan
 * memory ahead of time, inference servers that keep allocation (which can
 * synchronise the device) off the serving path, and code running while a
 * stream is being captured, where an allocation would fail.  It computes
 * what h3attn_prefill_ws() computes with a workspace, but the split-key
 * tail's scratch is a fixed 12 MiB array inside the library's device code
 * instead of caller memory.  Every device that loads the library holds that
 * array until the process exits, whether or not this call is used.
 *
 * The caller still passes q, k, v and o; arguments, layout and errors as for
 * h3attn_prefill().  A call whose tail would need more than 12 MiB of scratch
 * (h3attn_prefill_workspace_size() above 12582912 bytes; at most 10.1 MB at
 * head dim 128 on 152 SMs) is rejected with H3ATTN_ERR_INVALID_ARG before
 * anything is launched.  Calls that need no scratch run exactly as
 * h3attn_prefill().
 * The first call on each device looks up the array's device address (and may
 * load the library's device code on that device); make that first call
 * before any stream capture.
 * All calls on a device share the one array, and it keeps the last call's
 * partial results: each call overwrites every slot it reads, so nothing needs
 * clearing, but calls whose kernels can overlap on the GPU (different streams,
 * or host threads racing on one stream) race on the array and must be
 * ordered by the caller.
 */
h3attn_status_t h3attn_prefill_noalloc(const void* q, const void* k, const void* v, void* o, int B, int Sq,
                                       int Sk, int Hq, int Hkv, int D, float scale,
                                       const h3attn_mask_t* mask, int causal, h3attn_stream_t stream);

/*
 * Fused RMSNorm -> indexed AdaLN scale/shift modulation of DiT hidden rows
 * (TeleFuser PR #37 "perf(minimax-h3): optimize Ulysses attention and DiT
 * kernels", section 2.5: "RMSNorm -> indexed scale/shift modulation" in one
 * kernel, keeping the bf16 store/load rounding boundaries of the unfused
 * path).  For every row t of C channels, with s = scale[idx[t]] and
 * h = shift[idx[t]]:
 *   r = 1 / sqrt(mean_c(x_c^2) + eps)
 *   n = bf16((x * r) * w)       (bf16(x * r) when w is NULL)
 *   y = bf16(bf16(n * bf16(1 + s)) + h)
 * The float32 operation order is fixed (8-channel groups dealt round-robin to
 * 32 lanes, per-lane fused multiply-adds in channel order, a 32-lane
 * butterfly, correctly rounded divide and square root, round-to-nearest-even
 * stores), so results are reproducible bit for bit.
 *
 * x: [T, C] bf16 (device); y: [T, C] bf16 output (device), may be x itself.
 * w: [C] float32 RMSNorm weight (device) or NULL.
 * scale, shift: [N, C] bf16 modulation tables (device), row = index value.
 * idx: [T] int32 (device): the table row of each token, or NULL for row 0.
 *    A row whose index is outside [0, N) is written as zeros and
 *    h3attn_check_device_status() then reports H3ATTN_ERR_INVALID_ARG.
 * C a multiple of 8, 8 <= C <= 8192; N >= 1; eps >= 0 and finite; T == 0 is a
 * no-op.  x, y, scale, shift, w 16-byte aligned, idx 4-byte aligned; y must not
 * overlap scale, shift, w, idx or (unless equal) x.
 * Stream order as for any kernel.  The kernel is launched as a programmatic
 * dependent of the kernel before it in the stream: it reads and writes memory
 * only after that kernel has completed, while its CTAs may be placed as that
 * kernel's last CTAs finish; a later launch that is itself a programmatic
 * dependent may likewise start its set-up before this kernel ends.
 * Errors: INVALID_ARG, MISALIGNED, UNSUPPORTED_DEVICE, LAUNCH.
 */
h3attn_status_t h3attn_rmsnorm_modulate(const void* x, void* y, const float* w, const void* scale,
                                        const void* shift, const int32_t* idx, int T, int C, int N,
                                        float eps, h3attn_stream_t stream);

/*
 * Chunked window of video self-attention with anchor frames (SGLang PR
 * #37903 "[diffusion] model: support VDN-H3 ...", section "Modifications",
 * hybrid_window_attn_h3: a chunk-5 / radius-1 window with anchor frames,
 * dense-query rows against all keys; section "Accuracy Tests": the anchor
 * frames shift the chunk grid).  Rows are frame-major video tokens; token t
 * is in frame t / frame_tokens.  With af = anchor_frames * frame_tokens and
 * ct = chunk_frames * frame_tokens:
 *   allowed(i, j) = i < af  or  j < af  or  |(i - af) / ct - (j - af) / ct| <= radius
 * (integer division), AND-ed with the key padding / zero tail of the mask.
 */
typedef struct {
  int frame_tokens;   /* tokens per frame, >= 1 */
  int anchor_frames;  /* leading frames whose queries and keys are dense, >= 0 */
  int chunk_frames;   /* frames per chunk of the window grid, >= 1 */
  int radius;         /* a query in chunk c attends chunks c - radius .. c + radius, >= 0 */
} h3attn_window_t;

/*
 * Prefill self-attention (Sq = Sk = S) under the chunked window above; key
 * tiles outside a query block's window are never loaded or computed.
 * q, k, v, o, B, Hq, Hkv, scale as for h3attn_prefill(); D in {64, 128}.
 * win: required.  mask: NULL or a descriptor whose kv_len / q_len apply as in
 *    h3attn_prefill(); causal_b and bits are rejected (UNSUPPORTED_MASK).
 * Errors: INVALID_ARG, MISALIGNED, UNSUPPORTED_HEAD_DIM (D = 256),
 * UNSUPPORTED_DEVICE, UNSUPPORTED_MASK, LAUNCH.
 */
h3attn_status_t h3attn_prefill_window(const void* q, const void* k, const void* v, void* o, int B, int S,
                                      int Hq, int Hkv, int D, float scale, const h3attn_window_t* win,
                                      const h3attn_mask_t* mask, h3attn_stream_t stream);

/* Static English description of a status code (never NULL). */
const char* h3attn_status_string(h3attn_status_t status);

/*
 * Synchronises `stream`, then reads the current device's status word and
 * clears it.  Returns H3ATTN_ERR_TIMEOUT if a kernel gave up on a bounded wait
 * (H3ATTN_ERR_INVALID_ARG for an out-of-range modulation index) since the
 * last check, H3ATTN_ERR_LAUNCH if the stream reports a CUDA error, else
 * H3ATTN_OK.
 * The status word is one per device, shared by every stream and host thread
 * on it: a kernel on any stream can set it, and a check on any stream reports
 * it.  The read and the clear are issued on `stream` (after its work), and the
 * word is cleared only if it still holds the value read, so a report that
 * another stream's kernel writes in between is kept for the next check rather
 * than lost.  The word holds one code; several reports before a check merge.
 */
h3attn_status_t h3attn_check_device_status(h3attn_stream_t stream);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int h3attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* H3ATTN_H_ */
