// C-ABI entry points of libh3attn: argument validation, device gate, TMA
// descriptor construction and error mapping.  No entry point allocates
// device memory; all work is enqueued on the caller's stream.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include <atomic>

#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;

// Per device: 0 = not yet known, 1 = supported, 2 = not supported.  Stored
// only after both attribute queries succeeded, so a failed query is retried
// on the next call instead of marking the device unsupported for good.
std::atomic<int> g_dev_state[kMaxDevices];

// Gate on compute capability 10.3 (the only target the kernels are built for).
h3attn_status_t check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return H3ATTN_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return H3ATTN_ERR_UNSUPPORTED_DEVICE;
  int state = g_dev_state[dev].load(std::memory_order_acquire);
  if (state == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return H3ATTN_ERR_LAUNCH;
    state = (major == 10 && minor == 3) ? 1 : 2;
    g_dev_state[dev].store(state, std::memory_order_release);  // racing callers store the same value
  }
  return state == 1 ? H3ATTN_OK : H3ATTN_ERR_UNSUPPORTED_DEVICE;
}

// The driver's tensor-map encoder, looked up until a lookup succeeds.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
  if (f) return f;
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  fn.store(f, std::memory_order_release);
  return f;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, int64_t na, const void* b, int64_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(nb) && b0 < a0 + static_cast<uintptr_t>(na);
}

// 4-D map over a BSHD bf16 tensor: dims (D, H, S, B), box (64, 1, 128, 1),
// 128-byte swizzle, zero fill outside the tensor.
bool make_bshd_map(CUtensorMap* m, const void* ptr, int B, int S, int H, int D) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                                 static_cast<cuuint64_t>(S) * H * D * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(h3::kBlockM), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

uint64_t wait_limit_ns() {
  const char* s = getenv("H3ATTN_WAIT_LIMIT_MS");
  long ms = s ? strtol(s, nullptr, 10) : 0;
  if (ms <= 0) ms = 2000;
  return static_cast<uint64_t>(ms) * 1000000ull;
}

bool head_dim_ok(int D) { return D == 64 || D == 128 || D == 256; }

}  // namespace

extern "C" {

int h3attn_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char* h3attn_status_string(h3attn_status_t s) {
  switch (s) {
    case H3ATTN_OK: return "ok";
    case H3ATTN_ERR_INVALID_ARG: return "invalid argument";
    case H3ATTN_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
    case H3ATTN_ERR_UNSUPPORTED_HEAD_DIM: return "unsupported head dimension (64, 128 or 256)";
    case H3ATTN_ERR_UNSUPPORTED_DEVICE: return "unsupported device (compute capability 10.3 required)";
    case H3ATTN_ERR_UNSUPPORTED_MASK: return "unsupported mask form";
    case H3ATTN_ERR_LAUNCH: return "CUDA launch or runtime error";
    case H3ATTN_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

}  // extern "C"

namespace {

// Shared body of the in-place and out-of-place norm/RoPE entry points.  An
// output may be its own input (in place); any other overlap between the four
// row tensors is rejected.
h3attn_status_t norm_rope(const void* q, const void* k, void* q_out, void* k_out, const float* wq,
                          const float* wk, const float* cos, const float* sin, int B, int S, int Hq, int Hkv,
                          int D, int rotary_dim, float eps, h3attn_stream_t stream) {
  if (B < 0 || S < 0 || Hq < 0 || Hkv < 0) return H3ATTN_ERR_INVALID_ARG;
  if (!head_dim_ok(D)) return H3ATTN_ERR_UNSUPPORTED_HEAD_DIM;
  if (rotary_dim < 0 || rotary_dim > D || rotary_dim % 2 != 0) return H3ATTN_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || !isfinite(eps)) return H3ATTN_ERR_INVALID_ARG;
  if ((q == nullptr) != (Hq == 0) || (k == nullptr) != (Hkv == 0)) return H3ATTN_ERR_INVALID_ARG;
  if ((q_out == nullptr) != (q == nullptr) || (k_out == nullptr) != (k == nullptr)) return H3ATTN_ERR_INVALID_ARG;
  if (q && !wq) return H3ATTN_ERR_INVALID_ARG;
  if (k && !wk) return H3ATTN_ERR_INVALID_ARG;
  if (rotary_dim > 0 && (!cos || !sin)) return H3ATTN_ERR_INVALID_ARG;
  const int64_t rows_q = static_cast<int64_t>(B) * S * Hq;
  const int64_t rows_k = static_cast<int64_t>(B) * S * Hkv;
  if (rows_q + rows_k == 0) return H3ATTN_OK;
  if (rows_q + rows_k >= (1LL << 31)) return H3ATTN_ERR_INVALID_ARG;
  if ((q && !aligned16(q)) || (k && !aligned16(k)) || (q_out && !aligned16(q_out)) || (k_out && !aligned16(k_out)) ||
      (wq && !aligned16(wq)) || (wk && !aligned16(wk)) || (cos && !aligned16(cos)) || (sin && !aligned16(sin)))
    return H3ATTN_ERR_MISALIGNED;
  const int64_t nq = rows_q * D * 2, nk = rows_k * D * 2;
  if (q && k && overlap(q, nq, k, nk)) return H3ATTN_ERR_INVALID_ARG;
  if (q && k && (overlap(q_out, nq, k, nk) || overlap(q_out, nq, k_out, nk) || overlap(k_out, nk, q, nq)))
    return H3ATTN_ERR_INVALID_ARG;
  if (q && q_out != q && overlap(q_out, nq, q, nq)) return H3ATTN_ERR_INVALID_ARG;
  if (k && k_out != k && overlap(k_out, nk, k, nk)) return H3ATTN_ERR_INVALID_ARG;
  h3attn_status_t st = check_device();
  if (st != H3ATTN_OK) return st;
  h3::NormRopeArgs a;
  a.q_in = static_cast<const uint16_t*>(q);
  a.k_in = static_cast<const uint16_t*>(k);
  a.q_out = static_cast<uint16_t*>(q_out);
  a.k_out = static_cast<uint16_t*>(k_out);
  a.wq = wq;
  a.wk = wk;
  a.cos = cos;
  a.sin = sin;
  a.rows_q = static_cast<uint32_t>(rows_q);
  a.rows_k = static_cast<uint32_t>(rows_k);
  a.div_hq = h3::make_fastdiv(static_cast<uint32_t>(Hq > 0 ? Hq : 1));
  a.div_hkv = h3::make_fastdiv(static_cast<uint32_t>(Hkv > 0 ? Hkv : 1));
  a.div_s = h3::make_fastdiv(static_cast<uint32_t>(S > 0 ? S : 1));
  a.D = D;
  a.rotary_dim = rotary_dim;
  a.eps = eps;
  a.status = h3::status_word_ptr();
  if (!a.status) return H3ATTN_ERR_LAUNCH;
  a.wait_limit_ns = wait_limit_ns();
  cudaError_t e = h3::launch_qk_norm_rope(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? H3ATTN_OK : H3ATTN_ERR_LAUNCH;
}

}  // namespace

extern "C" {

h3attn_status_t h3attn_qk_norm_rope(void* q, void* k, const float* wq, const float* wk,
                                    const float* cos, const float* sin, int B, int S, int Hq,
                                    int Hkv, int D, int rotary_dim, float eps,
                                    h3attn_stream_t stream) {
  return norm_rope(q, k, q, k, wq, wk, cos, sin, B, S, Hq, Hkv, D, rotary_dim, eps, stream);
}

h3attn_status_t h3attn_qk_norm_rope_out(const void* q, const void* k, void* q_out, void* k_out,
                                        const float* wq, const float* wk, const float* cos,
                                        const float* sin, int B, int S, int Hq, int Hkv, int D,
                                        int rotary_dim, float eps, h3attn_stream_t stream) {
  return norm_rope(q, k, q_out, k_out, wq, wk, cos, sin, B, S, Hq, Hkv, D, rotary_dim, eps, stream);
}

}  // extern "C"

namespace {

// Kernel choice override (tests run every case on every kernel): "1" .. "5".
int kernel_override() {
  const char* kern = getenv("H3ATTN_ATTN_KERNEL");
  return (kern && kern[0] >= '1' && kern[0] <= '6') ? kern[0] - '0' : 0;
}

// The fields of AttnArgs that decide the kernel and the split-key plan.
void plan_fields(h3::AttnArgs* a, int B, int Sq, int Sk, int Hq, int Hkv, int D, const h3attn_mask_t* mask,
                 int causal, const h3attn_window_t* win) {
  a->B = B;
  a->Sq = Sq;
  a->Sk = Sk;
  a->Hq = Hq;
  a->Hkv = Hkv;
  a->D = D;
  a->causal = causal ? 1 : 0;
  a->kv_len = mask ? mask->kv_len : nullptr;
  a->q_len = mask ? mask->q_len : nullptr;
  a->causal_b = mask ? mask->causal_b : nullptr;
  a->bits = mask ? mask->bits : nullptr;
  a->kernel = win ? 1 : kernel_override();  // the window's tile ranges live in the one-query-tile kernel
  a->win_ct = win ? win->frame_tokens * win->chunk_frames : 0;
  a->split_full = a->split_tail = a->split_pieces = 0;
  a->split_ws = nullptr;
}

// Shared body of the dense and windowed prefill entry points (win == nullptr:
// dense).  ws: the split-key tail's workspace (nullptr: no split).
h3attn_status_t prefill(const void* q, const void* k, const void* v, void* o, int B, int Sq, int Sk, int Hq,
                        int Hkv, int D, float scale, const h3attn_mask_t* mask, int causal,
                        const h3attn_window_t* win, void* ws, size_t ws_bytes, h3attn_stream_t stream) {
  if (B < 0 || Sq < 0 || Sk < 1 || Hq < 1 || Hkv < 1) return H3ATTN_ERR_INVALID_ARG;
  if (!head_dim_ok(D)) return H3ATTN_ERR_UNSUPPORTED_HEAD_DIM;
  if (Hq % Hkv != 0) return H3ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.0f) || !isfinite(scale)) return H3ATTN_ERR_INVALID_ARG;
  if (B > 65535 || Hq > 65535) return H3ATTN_ERR_INVALID_ARG;
  // work units (128-row query blocks x heads x batch items) are counted in 32 bits
  if ((static_cast<int64_t>(Sq) + 127) / 128 * Hq * B > INT32_MAX) return H3ATTN_ERR_INVALID_ARG;
  if (win) {
    if (Sq != Sk || win->frame_tokens < 1 || win->chunk_frames < 1 || win->anchor_frames < 0 || win->radius < 0)
      return H3ATTN_ERR_INVALID_ARG;
    // token counts of the window grid must fit 32 bits
    if (static_cast<int64_t>(win->frame_tokens) * win->chunk_frames > INT32_MAX ||
        static_cast<int64_t>(win->frame_tokens) * win->anchor_frames > INT32_MAX)
      return H3ATTN_ERR_INVALID_ARG;
    if (D == 256) return H3ATTN_ERR_UNSUPPORTED_HEAD_DIM;
    if (causal || (mask && (mask->causal_b || mask->bits))) return H3ATTN_ERR_UNSUPPORTED_MASK;
  }
  if (B == 0 || Sq == 0) return H3ATTN_OK;
  if (!q || !k || !v || !o) return H3ATTN_ERR_INVALID_ARG;
  const bool any_causal = causal || (mask && mask->causal_b);
  if (any_causal && Sq != Sk) return H3ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return H3ATTN_ERR_MISALIGNED;
  if (mask && mask->bits && (reinterpret_cast<uintptr_t>(mask->bits) & 3u))
    return H3ATTN_ERR_MISALIGNED;
  if (mask && ((mask->kv_len && (reinterpret_cast<uintptr_t>(mask->kv_len) & 3u)) ||
               (mask->q_len && (reinterpret_cast<uintptr_t>(mask->q_len) & 3u))))
    return H3ATTN_ERR_MISALIGNED;
  const int64_t nq = static_cast<int64_t>(B) * Sq * Hq * D * 2;
  const int64_t nk = static_cast<int64_t>(B) * Sk * Hkv * D * 2;
  if (overlap(o, nq, q, nq) || overlap(o, nq, k, nk) || overlap(o, nq, v, nk))
    return H3ATTN_ERR_INVALID_ARG;
  if (ws && !aligned16(ws)) return H3ATTN_ERR_MISALIGNED;
  h3attn_status_t st = check_device();
  if (st != H3ATTN_OK) return st;

  h3::AttnArgs a;
  plan_fields(&a, B, Sq, Sk, Hq, Hkv, D, mask, causal, win);
  if (ws) {
    const h3::SplitPlan sp = h3::plan_split(a);
    if (sp.pieces > 0) {
      const int64_t nb = static_cast<int64_t>(sp.bytes);
      if (ws_bytes < sp.bytes) return H3ATTN_ERR_INVALID_ARG;
      if (overlap(ws, nb, q, nq) || overlap(ws, nb, k, nk) || overlap(ws, nb, v, nk) || overlap(ws, nb, o, nq))
        return H3ATTN_ERR_INVALID_ARG;
      a.split_full = sp.full;
      a.split_tail = sp.tail;
      a.split_pieces = sp.pieces;
      a.split_ws = static_cast<float*>(ws);
    }
  }
  if (!make_bshd_map(&a.tm_q, q, B, Sq, Hq, D) || !make_bshd_map(&a.tm_k, k, B, Sk, Hkv, D) ||
      !make_bshd_map(&a.tm_v, v, B, Sk, Hkv, D) || !make_bshd_map(&a.tm_o, o, B, Sq, Hq, D))
    return H3ATTN_ERR_LAUNCH;
  a.q_ptr = static_cast<const uint16_t*>(q);
  a.o = static_cast<uint16_t*>(o);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit_ns = wait_limit_ns();
  const char* inj = getenv("H3ATTN_FAULT_INJECT_STALL_PRODUCER");
  a.debug_skip_producer = (inj && inj[0] == '1') ? 1 : 0;
  a.win_af = a.win_r = 0;
  if (win) {
    a.win_af = static_cast<int>(min(static_cast<int64_t>(win->frame_tokens) * win->anchor_frames,
                                    static_cast<int64_t>(Sk)));
    a.win_r = static_cast<int>(min(static_cast<int64_t>(win->radius), static_cast<int64_t>(Sk)));
  }
  cudaError_t e = h3::launch_attention(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? H3ATTN_OK : H3ATTN_ERR_LAUNCH;
}

}  // namespace

extern "C" {

h3attn_status_t h3attn_prefill(const void* q, const void* k, const void* v, void* o, int B, int Sq,
                               int Sk, int Hq, int Hkv, int D, float scale,
                               const h3attn_mask_t* mask, int causal, h3attn_stream_t stream) {
  return prefill(q, k, v, o, B, Sq, Sk, Hq, Hkv, D, scale, mask, causal, nullptr, nullptr, 0, stream);
}

h3attn_status_t h3attn_prefill_workspace_size(int B, int Sq, int Sk, int Hq, int Hkv, int D,
                                              const h3attn_mask_t* mask, int causal, size_t* bytes) {
  if (!bytes) return H3ATTN_ERR_INVALID_ARG;
  *bytes = 0;
  if (B < 0 || Sq < 0 || Sk < 1 || Hq < 1 || Hkv < 1) return H3ATTN_ERR_INVALID_ARG;
  if (!head_dim_ok(D)) return H3ATTN_ERR_UNSUPPORTED_HEAD_DIM;
  if (Hq % Hkv != 0 || B > 65535 || Hq > 65535) return H3ATTN_ERR_INVALID_ARG;
  if ((static_cast<int64_t>(Sq) + 127) / 128 * Hq * B > INT32_MAX) return H3ATTN_ERR_INVALID_ARG;
  if (B == 0 || Sq == 0) return H3ATTN_OK;
  h3attn_status_t st = check_device();
  if (st != H3ATTN_OK) return st;
  h3::AttnArgs a;
  plan_fields(&a, B, Sq, Sk, Hq, Hkv, D, mask, causal, nullptr);
  *bytes = h3::plan_split(a).bytes;
  return H3ATTN_OK;
}

h3attn_status_t h3attn_prefill_ws(const void* q, const void* k, const void* v, void* o, int B, int Sq, int Sk,
                                  int Hq, int Hkv, int D, float scale, const h3attn_mask_t* mask, int causal,
                                  void* workspace, size_t workspace_bytes, h3attn_stream_t stream) {
  return prefill(q, k, v, o, B, Sq, Sk, Hq, Hkv, D, scale, mask, causal, nullptr, workspace, workspace_bytes,
                 stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Prefill for callers that cannot allocate device memory (h3attn_prefill_noalloc).
// The split-key tail's partials go to one fixed array that the library's
// device code owns; it exists on every device that loads the library, from
// the moment the device code is loaded until the process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t{12} << 20;  // 12 MiB: 152 SMs x 128 rows x 130 floats fit
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

// Device address of the array on each device.  In host code the array's name
// is only a stand-in that the runtime maps to the device copy, so a kernel
// must be given the address cudaGetSymbolAddress returns for the current
// device, never the name itself.  Looked up on the first call on a device.
std::atomic<void*> g_noalloc_addr[kMaxDevices];

h3attn_status_t noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return H3ATTN_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return H3ATTN_ERR_UNSUPPORTED_DEVICE;
  void* p = g_noalloc_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return H3ATTN_ERR_LAUNCH;
    g_noalloc_addr[dev].store(p, std::memory_order_release);  // racing first calls store the same address
  }
  *out = p;
  return H3ATTN_OK;
}

}  // namespace

extern "C" {

h3attn_status_t h3attn_prefill_noalloc(const void* q, const void* k, const void* v, void* o, int B, int Sq,
                                       int Sk, int Hq, int Hkv, int D, float scale, const h3attn_mask_t* mask,
                                       int causal, h3attn_stream_t stream) {
  size_t need = 0;
  h3attn_status_t st = h3attn_prefill_workspace_size(B, Sq, Sk, Hq, Hkv, D, mask, causal, &need);
  if (st != H3ATTN_OK) return st;
  if (need > kNoAllocScratchBytes) return H3ATTN_ERR_INVALID_ARG;  // more scratch than the fixed array holds
  void* scratch = nullptr;
  if (need > 0) {
    st = noalloc_scratch(&scratch);
    if (st != H3ATTN_OK) return st;
  }
  // Every slot the combine reads is written by this call's pieces in full, so
  // nothing left in the array by an earlier call needs clearing.
  return prefill(q, k, v, o, B, Sq, Sk, Hq, Hkv, D, scale, mask, causal, nullptr, scratch, kNoAllocScratchBytes,
                 stream);
}

h3attn_status_t h3attn_prefill_window(const void* q, const void* k, const void* v, void* o, int B, int S,
                                      int Hq, int Hkv, int D, float scale, const h3attn_window_t* win,
                                      const h3attn_mask_t* mask, h3attn_stream_t stream) {
  if (!win) return H3ATTN_ERR_INVALID_ARG;
  if (S == 0) {  // no tokens: nothing to do once the window itself is well formed
    const bool ok = win->frame_tokens >= 1 && win->chunk_frames >= 1 && win->anchor_frames >= 0 && win->radius >= 0;
    return ok ? H3ATTN_OK : H3ATTN_ERR_INVALID_ARG;
  }
  return prefill(q, k, v, o, B, S, S, Hq, Hkv, D, scale, mask, 0, win, nullptr, 0, stream);
}

h3attn_status_t h3attn_rmsnorm_modulate(const void* x, void* y, const float* w, const void* scale,
                                        const void* shift, const int32_t* idx, int T, int C, int N,
                                        float eps, h3attn_stream_t stream) {
  if (T < 0 || C <= 0 || C % 8 != 0 || C > h3::kModMaxChannels || N < 1) return H3ATTN_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || !isfinite(eps)) return H3ATTN_ERR_INVALID_ARG;
  if (T == 0) return H3ATTN_OK;
  if (!x || !y || !scale || !shift) return H3ATTN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(scale) || !aligned16(shift) || (w && !aligned16(w)) ||
      (idx && (reinterpret_cast<uintptr_t>(idx) & 3u)))
    return H3ATTN_ERR_MISALIGNED;
  const int64_t ny = static_cast<int64_t>(T) * C * 2, nt = static_cast<int64_t>(N) * C * 2;
  if (y != x && overlap(y, ny, x, ny)) return H3ATTN_ERR_INVALID_ARG;
  if (overlap(y, ny, scale, nt) || overlap(y, ny, shift, nt) || (w && overlap(y, ny, w, static_cast<int64_t>(C) * 4)) ||
      (idx && overlap(y, ny, idx, static_cast<int64_t>(T) * 4)))
    return H3ATTN_ERR_INVALID_ARG;
  h3attn_status_t st = check_device();
  if (st != H3ATTN_OK) return st;
  h3::ModArgs a;
  a.x = static_cast<const uint16_t*>(x);
  a.y = static_cast<uint16_t*>(y);
  a.w = w;
  a.scale = static_cast<const uint16_t*>(scale);
  a.shift = static_cast<const uint16_t*>(shift);
  a.idx = idx;
  a.T = T;
  a.C = C;
  a.N = N;
  a.eps = eps;
  a.status = h3::status_word_ptr();
  if (!a.status) return H3ATTN_ERR_LAUNCH;
  a.wait_limit_ns = wait_limit_ns();
  cudaError_t e = h3::launch_rmsnorm_modulate(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? H3ATTN_OK : H3ATTN_ERR_LAUNCH;
}

h3attn_status_t h3attn_check_device_status(h3attn_stream_t stream) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return H3ATTN_ERR_LAUNCH;
  int v = 0;
  if (h3::read_and_clear_status(s, &v) != 0) return H3ATTN_ERR_LAUNCH;
  return v == 0 ? H3ATTN_OK : static_cast<h3attn_status_t>(v);
}

}  // extern "C"
