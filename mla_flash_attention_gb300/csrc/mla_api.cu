// Host side of the C ABI declared in include/mla.h: argument validation, the
// device error word, decode workspace sizing and kernel dispatch.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "../../include/mla.h"
#include "../../include/mla_testing.h"
#include "common.cuh"

namespace mla {
cudaError_t launch_prefill_sm103_bf16(const void* q_nope, const void* q_rope, const void* k_nope,
                                      const void* k_rope, const void* v, void* out, float* lse,
                                      int B, int H, int S, float softmax_scale, int causal,
                                      bool out_f32, unsigned int* err, cudaStream_t stream);
cudaError_t launch_prefill_sm103_fp8(const void* q_nope, const void* q_rope, const void* k_nope,
                                     const void* k_rope, const void* v, const float* q_scale,
                                     const float* k_scale, void* out, float* lse, int B, int H,
                                     int S, float softmax_scale, int causal, bool out_f32,
                                     unsigned int* err, cudaStream_t stream);
cudaError_t launch_decode_sm103(const void* q_latent, const void* q_rope, const void* kv_cache,
                                const float* kv_scale, const int* page_table,
                                const int* cache_lens, int B, int H, int T, int max_pages,
                                int num_pages, float softmax_scale, int causal, bool fp8,
                                float* part_o, float* part_lse, int* counters, void* out,
                                float* lse, int G, unsigned int* err, cudaStream_t stream);
cudaError_t launch_decode_t_sm103(const void* q_latent, const void* q_rope, const void* kv_cache,
                                  const float* kv_scale, const int* page_table,
                                  const int* cache_lens, int B, int H, int T, int max_pages,
                                  int num_pages, float softmax_scale, int causal, float* part_o,
                                  float* part_lse, int* counters, void* out, float* lse, int G,
                                  unsigned int* err, long long wait_limit, int skip_unit,
                                  cudaStream_t stream);
cudaError_t launch_absorb_sm103(const void* x, const void* w, void* y, int R, int H, int K, int N,
                                unsigned int* err, cudaStream_t stream);
size_t prefill_bwd_workspace_bytes(int B, int H, int S);
cudaError_t launch_prefill_bwd_sm103(const void* q_nope, const void* q_rope, const void* k_nope,
                                     const void* k_rope, const void* v, const void* out,
                                     const float* lse, const void* d_out, void* dq_nope,
                                     void* dq_rope, void* dk_nope, float* dk_rope, void* dv,
                                     int B, int H, int S, float softmax_scale, int causal,
                                     void* workspace, unsigned int* err, cudaStream_t stream);
cudaError_t launch_cache_append(const void* c_new, void* cache, float* kv_scale,
                                const int* page_table, const int* cache_lens, int B, int T,
                                int max_pages, int num_pages, bool fp8, unsigned int* err,
                                cudaStream_t stream);
}  // namespace mla

namespace {

thread_local std::string g_last_error;

__device__ unsigned int g_device_error = 0;

mla_status fail(mla_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

mla_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MLA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Address of the device error word on the current device (looked up once per device).  The
// cache entries are atomics: host threads may make their first calls concurrently, and two
// threads that both look the address up store the same value.
unsigned int* device_error_word() {
  static std::atomic<unsigned int*> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  unsigned int* w = cache[dev].load(std::memory_order_acquire);
  if (!w) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    w = static_cast<unsigned int*>(p);
    cache[dev].store(w, std::memory_order_release);
  }
  return w;
}

int num_sms_current() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Decode work units of the split kernel: each unit is served by a pair of CTAs (one per half
// of the latent output columns), one CTA per SM.
int decode_units() { return num_sms_current() / 2; }

// The transposed decode kernel (one CTA per SM and work unit) serves an fp8 cache when a
// sequence has at most 32 query rows (q_len * H).
constexpr int kTransposedMaxRows = 32;
bool decode_transposed(bool fp8, int TH) { return fp8 && TH <= kTransposedMaxRows; }

// Test hooks (mla_testing.h): a decode launch of the transposed kernel leaves raw unit
// `g_skip_unit` unloaded and gives each pipeline wait `g_wait_limit` SM clocks.
std::atomic<int> g_skip_unit{-1};
std::atomic<long long> g_wait_limit{1000000000LL};
// ... and launches report the output buffer `g_out_shrink` bytes smaller to the store checks
// of the bounds-checked build
std::atomic<size_t> g_out_shrink{0};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct DecodeWorkspace {
  float* part_o;
  float* part_lse;
  int* counters;
  size_t bytes;
};

// The q_len*H query rows of a sequence are processed in tiles of (up to) 128 rows; each
// (sequence, tile) is planned as its own work item, so there are G + B * NQT partial slots of
// TQ = min(q_len*H, 128) rows each: O partials (fp32, 512 columns), LSE partials (one copy per
// column half), and two split counters per work item for the merge.
DecodeWorkspace decode_workspace_layout(void* base, int B, int TH, int d_latent, int G) {
  DecodeWorkspace w;
  const size_t nqt = (size_t)(TH + 127) / 128, tq = TH < 128 ? TH : 128;
  const size_t slots = (size_t)G + (size_t)B * nqt;
  const size_t o_bytes = align_up(slots * tq * d_latent * sizeof(float), 256);
  const size_t l_bytes = align_up(2 * slots * tq * sizeof(float), 256);
  const size_t c_bytes = align_up(2 * (size_t)B * nqt * sizeof(int), 256);
  w.part_o = static_cast<float*>(base);
  w.part_lse = reinterpret_cast<float*>(static_cast<char*>(base) + o_bytes);
  w.counters = reinterpret_cast<int*>(static_cast<char*>(base) + o_bytes + l_bytes);
  w.bytes = o_bytes + l_bytes + c_bytes;
  return w;
}

// Workspace of the transposed kernel: G = SMs units, S = G + B slots of TQ = q_len*H rows:
// O partials [S][TQ][d_latent] fp32, LSE partials [S][TQ] fp32, one split counter per sequence.
DecodeWorkspace decode_workspace_layout_t(void* base, int B, int TH, int d_latent, int G) {
  DecodeWorkspace w;
  const size_t slots = (size_t)G + (size_t)B;
  const size_t o_bytes = align_up(slots * TH * d_latent * sizeof(float), 256);
  const size_t l_bytes = align_up(slots * TH * sizeof(float), 256);
  const size_t c_bytes = align_up((size_t)B * sizeof(int), 256);
  w.part_o = static_cast<float*>(base);
  w.part_lse = reinterpret_cast<float*>(static_cast<char*>(base) + o_bytes);
  w.counters = reinterpret_cast<int*>(static_cast<char*>(base) + o_bytes + l_bytes);
  w.bytes = o_bytes + l_bytes + c_bytes;
  return w;
}

}  // namespace

namespace mla {
size_t testing_out_shrink() { return g_out_shrink.load(); }

// The device error word's address on the current device (for entry points in other files).
unsigned int* error_word_address() { return device_error_word(); }

// Records `fmt` as this thread's last-error message (for entry points in other files).
mla_status set_last_error(mla_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}
}  // namespace mla

extern "C" {

const char* mla_last_error(void) { return g_last_error.c_str(); }

void mla_testing_decode_stall(int skip_unit, long long wait_limit_cycles) {
  g_skip_unit.store(skip_unit < 0 ? -1 : skip_unit);
  g_wait_limit.store(wait_limit_cycles > 0 ? wait_limit_cycles : 1000000000LL);
}

void mla_testing_bounds_shrink(long long bytes) { g_out_shrink.store(bytes > 0 ? (size_t)bytes : 0); }

int mla_testing_bounds_checked(void) {
#ifdef MLA_DEBUG
  return 1;
#else
  return 0;
#endif
}

int mla_version(void) { return 100; }

mla_status mla_check_device_error(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int* w = device_error_word();
  if (!w) return fail(MLA_ERR_CUDA, "device error word not reachable");
  unsigned int v = 0;
  e = cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  const unsigned int zero = 0;
  e = cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
  if (v & mla::kErrTimeout) return fail(MLA_ERR_TIMEOUT, "a device-side pipeline wait timed out (word 0x%x)", v);
  if (v & mla::kErrBadPage)
    return fail(MLA_ERR_DEVICE_CHECK, "a page-table entry or cache length was out of range (word 0x%x)", v);
  if (v & mla::kErrBounds)
    return fail(MLA_ERR_DEVICE_CHECK, "a store fell outside its buffer and was skipped (word 0x%x)", v);
  return MLA_OK;
}

mla_status mla_prefill(const void* q_nope, const void* q_rope, const void* k_nope,
                       const void* k_rope, const void* v, const float* q_scale,
                       const float* k_scale, void* out, float* lse, int B, int H, int S,
                       int d_nope, int d_rope, int d_v, float softmax_scale, int causal,
                       mla_dtype qkv_dtype, mla_dtype out_dtype, void* stream) {
  if (!q_nope || !q_rope || !k_nope || !k_rope || !v || !out || !lse)
    return fail(MLA_ERR_INVALID_ARG, "mla_prefill: null tensor pointer");
  if (B <= 0 || H <= 0 || S <= 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_prefill: B, H, S must be positive (got %d, %d, %d)", B, H, S);
  if (B > 65535 || H > 65535)
    return fail(MLA_ERR_UNSUPPORTED, "mla_prefill: B and H must be at most 65535");
  if (d_nope != 128 || d_rope != 64 || d_v != 128)
    return fail(MLA_ERR_UNSUPPORTED, "mla_prefill: only d_nope=128, d_rope=64, d_v=128 are built (got %d, %d, %d)",
                d_nope, d_rope, d_v);
  if (!std::isfinite(softmax_scale) || softmax_scale <= 0.f)
    return fail(MLA_ERR_INVALID_ARG, "mla_prefill: softmax_scale must be finite and positive");
  const bool fp8 = qkv_dtype == MLA_FP8_E4M3;
  if (qkv_dtype != MLA_BF16 && !fp8)
    return fail(MLA_ERR_UNSUPPORTED, "mla_prefill: qkv_dtype must be MLA_BF16 or MLA_FP8_E4M3");
  if (out_dtype != MLA_BF16 && out_dtype != MLA_FP32)
    return fail(MLA_ERR_UNSUPPORTED, "mla_prefill: out_dtype must be MLA_BF16 or MLA_FP32");
  if (fp8 && (!q_scale || !k_scale))
    return fail(MLA_ERR_INVALID_ARG, "mla_prefill: fp8 inputs need q_scale and k_scale");
  if (!fp8 && (q_scale || k_scale))
    return fail(MLA_ERR_INVALID_ARG, "mla_prefill: q_scale/k_scale must be NULL for bf16 inputs");
  const void* ptrs[] = {q_nope, q_rope, k_nope, k_rope, v, out, lse};
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(MLA_ERR_INVALID_ARG, "mla_prefill: tensors must be 16-byte aligned");
  if ((double)B * S * H * 128 >= 9.0e18)
    return fail(MLA_ERR_UNSUPPORTED, "mla_prefill: problem too large");
  unsigned int* err = device_error_word();
  if (!err) return fail(MLA_ERR_CUDA, "mla_prefill: device error word not reachable");
  cudaError_t e;
  if (!fp8)
    e = mla::launch_prefill_sm103_bf16(q_nope, q_rope, k_nope, k_rope, v, out, lse, B, H, S,
                                       softmax_scale, causal != 0, out_dtype == MLA_FP32, err,
                                       static_cast<cudaStream_t>(stream));
  else
    e = mla::launch_prefill_sm103_fp8(q_nope, q_rope, k_nope, k_rope, v, q_scale, k_scale, out,
                                      lse, B, H, S, softmax_scale, causal != 0,
                                      out_dtype == MLA_FP32, err,
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_prefill launch");
  return MLA_OK;
}

size_t mla_prefill_backward_workspace_size(int B, int H, int S) {
  if (B <= 0 || H <= 0 || S <= 0) return 0;
  return mla::prefill_bwd_workspace_bytes(B, H, S);
}

mla_status mla_prefill_backward(const void* q_nope, const void* q_rope, const void* k_nope,
                                const void* k_rope, const void* v, const void* out,
                                const float* lse, const void* d_out, void* dq_nope,
                                void* dq_rope, void* dk_nope, float* dk_rope, void* dv, int B,
                                int H, int S, int d_nope, int d_rope, int d_v,
                                float softmax_scale, int causal, void* workspace,
                                size_t workspace_bytes, void* stream) {
  if (!q_nope || !q_rope || !k_nope || !k_rope || !v || !out || !lse || !d_out || !dq_nope ||
      !dq_rope || !dk_nope || !dk_rope || !dv)
    return fail(MLA_ERR_INVALID_ARG, "mla_prefill_backward: null tensor pointer");
  if (B <= 0 || H <= 0 || S <= 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_prefill_backward: B, H, S must be positive (got %d, %d, %d)", B, H, S);
  if (B > 65535 || H > 65535)
    return fail(MLA_ERR_UNSUPPORTED, "mla_prefill_backward: B and H must be at most 65535");
  if (d_nope != 128 || d_rope != 64 || d_v != 128)
    return fail(MLA_ERR_UNSUPPORTED, "mla_prefill_backward: only d_nope=128, d_rope=64, d_v=128 are built (got %d, %d, %d)",
                d_nope, d_rope, d_v);
  if (!std::isfinite(softmax_scale) || softmax_scale <= 0.f)
    return fail(MLA_ERR_INVALID_ARG, "mla_prefill_backward: softmax_scale must be finite and positive");
  const void* ptrs[] = {q_nope, q_rope, k_nope, k_rope, v, out, lse, d_out, dq_nope, dq_rope,
                        dk_nope, dk_rope, dv, workspace};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return fail(MLA_ERR_INVALID_ARG, "mla_prefill_backward: tensors must be 16-byte aligned");
  if ((double)B * S * H * 128 >= 9.0e18 || 2.0 * B * H * ((S + 127) / 128) > 2147483647.0)
    return fail(MLA_ERR_UNSUPPORTED, "mla_prefill_backward: problem too large");
  const size_t need = mla::prefill_bwd_workspace_bytes(B, H, S);
  if (!workspace || workspace_bytes < need)
    return fail(MLA_ERR_WORKSPACE, "mla_prefill_backward: workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, need);
  unsigned int* err = device_error_word();
  if (!err) return fail(MLA_ERR_CUDA, "mla_prefill_backward: device error word not reachable");
  cudaError_t e = mla::launch_prefill_bwd_sm103(q_nope, q_rope, k_nope, k_rope, v, out, lse, d_out,
                                                dq_nope, dq_rope, dk_nope, dk_rope, dv, B, H, S,
                                                softmax_scale, causal != 0, workspace, err,
                                                static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_prefill_backward launch");
  return MLA_OK;
}

size_t mla_decode_workspace_size(int B, int H, int q_len, int d_latent) {
  if (B <= 0 || H <= 0 || q_len <= 0 || d_latent <= 0) return 0;
  const int G = decode_units();
  if (G <= 0) return 0;
  size_t bytes = decode_workspace_layout(nullptr, B, H * q_len, d_latent, G).bytes;
  if (decode_transposed(true, H * q_len))  // the size cannot depend on the cache type
    bytes = std::max(bytes, decode_workspace_layout_t(nullptr, B, H * q_len, d_latent, 2 * G).bytes);
  return bytes;
}

mla_status mla_decode(const void* q_latent, const void* q_rope, const void* kv_cache,
                      const float* kv_scale, const int* page_table, const int* cache_lens,
                      void* out, float* lse, int B, int H, int q_len, int d_latent,
                      int d_rope, int page_size, int max_pages_per_seq, int num_pages,
                      float softmax_scale, int causal, mla_dtype kv_dtype, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!q_latent || !q_rope || !kv_cache || !page_table || !cache_lens || !out || !lse)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: null tensor pointer");
  if (B <= 0 || H <= 0 || q_len <= 0 || max_pages_per_seq <= 0 || num_pages <= 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: B, H, q_len, max_pages_per_seq, num_pages must be positive");
  if (d_latent != 512 || d_rope != 64)
    return fail(MLA_ERR_UNSUPPORTED, "mla_decode: only d_latent=512, d_rope=64 are built (got %d, %d)", d_latent, d_rope);
  if (page_size != 64)
    return fail(MLA_ERR_UNSUPPORTED, "mla_decode: only page_size=64 is built (got %d)", page_size);
  if ((long long)H * q_len > 65536)
    return fail(MLA_ERR_UNSUPPORTED, "mla_decode: q_len*H must be at most 65536 (got %lld)", (long long)H * q_len);
  if ((long long)B * ((H * q_len + 127) / 128) > (1LL << 24))
    return fail(MLA_ERR_UNSUPPORTED, "mla_decode: B * ceil(q_len*H / 128) must be at most 2^24");
  if (B > 65535) return fail(MLA_ERR_UNSUPPORTED, "mla_decode: B must be at most 65535");
  if ((long long)max_pages_per_seq * page_size > 0x7fffffffLL)
    return fail(MLA_ERR_UNSUPPORTED, "mla_decode: max_pages_per_seq*page_size overflows int32");
  if (!std::isfinite(softmax_scale) || softmax_scale <= 0.f)
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: softmax_scale must be finite and positive");
  const bool fp8 = kv_dtype == MLA_FP8_E4M3;
  if (kv_dtype != MLA_BF16 && !fp8)
    return fail(MLA_ERR_UNSUPPORTED, "mla_decode: kv_dtype must be MLA_BF16 or MLA_FP8_E4M3");
  if (fp8 != (kv_scale != nullptr))
    return fail(MLA_ERR_INVALID_ARG, "mla_decode: kv_scale is required for fp8 and must be NULL for bf16");
  const void* ptrs[] = {q_latent, q_rope, kv_cache, kv_scale, out, lse, workspace};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return fail(MLA_ERR_INVALID_ARG, "mla_decode: tensors must be 16-byte aligned");
  const int G = decode_units();
  if (G <= 0) return fail(MLA_ERR_CUDA, "mla_decode: cannot query the SM count");
  const bool tr = decode_transposed(fp8, H * q_len);
  DecodeWorkspace ws = tr ? decode_workspace_layout_t(workspace, B, H * q_len, d_latent, 2 * G)
                          : decode_workspace_layout(workspace, B, H * q_len, d_latent, G);
  if (!workspace || workspace_bytes < ws.bytes)
    return fail(MLA_ERR_WORKSPACE, "mla_decode: workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, ws.bytes);
  unsigned int* err = device_error_word();
  if (!err) return fail(MLA_ERR_CUDA, "mla_decode: device error word not reachable");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e =
      tr ? mla::launch_decode_t_sm103(q_latent, q_rope, kv_cache, kv_scale, page_table, cache_lens, B, H,
                                      q_len, max_pages_per_seq, num_pages, softmax_scale, causal != 0,
                                      ws.part_o, ws.part_lse, ws.counters, out, lse, 2 * G, err,
                                      g_wait_limit.load(), g_skip_unit.load(), st)
         : mla::launch_decode_sm103(q_latent, q_rope, kv_cache, kv_scale, page_table, cache_lens, B, H,
                                    q_len, max_pages_per_seq, num_pages, softmax_scale, causal != 0, fp8,
                                    ws.part_o, ws.part_lse, ws.counters, out, lse, G, err, st);
  if (e != cudaSuccess) return cuda_fail(e, "mla_decode launch");
  return MLA_OK;
}

mla_status mla_absorb(const void* x, const void* w, void* y, int R, int H, int K, int N,
                      void* stream) {
  if (!x || !w || !y) return fail(MLA_ERR_INVALID_ARG, "mla_absorb: null tensor pointer");
  if (R <= 0 || H <= 0 || K <= 0 || N <= 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_absorb: R, H, K, N must be positive");
  if (K % 64 != 0 || N % 128 != 0)
    return fail(MLA_ERR_UNSUPPORTED, "mla_absorb: K must be a multiple of 64 and N of 128 (got %d, %d)", K, N);
  if (H > 65535 || (long long)R * H * (K > N ? K : N) > 0x7fffffffffLL)
    return fail(MLA_ERR_UNSUPPORTED, "mla_absorb: tensor too large");
  const void* ptrs[] = {x, w, y};
  for (const void* q : ptrs)
    if (!aligned16(q)) return fail(MLA_ERR_INVALID_ARG, "mla_absorb: tensors must be 16-byte aligned");
  unsigned int* err = device_error_word();
  if (!err) return fail(MLA_ERR_CUDA, "mla_absorb: device error word not reachable");
  cudaError_t e = mla::launch_absorb_sm103(x, w, y, R, H, K, N, err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_absorb launch");
  return MLA_OK;
}

mla_status mla_cache_append(const void* c_new, void* kv_cache, float* kv_scale,
                            const int* page_table, const int* cache_lens, int B, int q_len,
                            int d_latent, int d_rope, int page_size, int max_pages_per_seq,
                            int num_pages, mla_dtype kv_dtype, void* stream) {
  if (!c_new || !kv_cache || !page_table || !cache_lens)
    return fail(MLA_ERR_INVALID_ARG, "mla_cache_append: null tensor pointer");
  if (B <= 0 || q_len <= 0 || max_pages_per_seq <= 0 || num_pages <= 0)
    return fail(MLA_ERR_INVALID_ARG, "mla_cache_append: B, q_len, max_pages_per_seq, num_pages must be positive");
  if (d_latent != 512 || d_rope != 64)
    return fail(MLA_ERR_UNSUPPORTED, "mla_cache_append: only d_latent=512, d_rope=64 are built (got %d, %d)", d_latent, d_rope);
  if (page_size != 64)
    return fail(MLA_ERR_UNSUPPORTED, "mla_cache_append: only page_size=64 is built (got %d)", page_size);
  if ((long long)B * q_len > 0x7fffffffLL / 4)
    return fail(MLA_ERR_UNSUPPORTED, "mla_cache_append: B*q_len too large");
  if ((long long)max_pages_per_seq * page_size > 0x7fffffffLL)
    return fail(MLA_ERR_UNSUPPORTED, "mla_cache_append: max_pages_per_seq*page_size overflows int32");
  const bool fp8 = kv_dtype == MLA_FP8_E4M3;
  if (kv_dtype != MLA_BF16 && !fp8)
    return fail(MLA_ERR_UNSUPPORTED, "mla_cache_append: kv_dtype must be MLA_BF16 or MLA_FP8_E4M3");
  if (fp8 != (kv_scale != nullptr))
    return fail(MLA_ERR_INVALID_ARG, "mla_cache_append: kv_scale is required for fp8 and must be NULL for bf16");
  const void* ptrs[] = {c_new, kv_cache};
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(MLA_ERR_INVALID_ARG, "mla_cache_append: tensors must be 16-byte aligned");
  if (kv_scale && (reinterpret_cast<uintptr_t>(kv_scale) & 3))
    return fail(MLA_ERR_INVALID_ARG, "mla_cache_append: kv_scale must be 4-byte aligned");
  unsigned int* err = device_error_word();
  if (!err) return fail(MLA_ERR_CUDA, "mla_cache_append: device error word not reachable");
  cudaError_t e = mla::launch_cache_append(c_new, kv_cache, kv_scale, page_table, cache_lens, B,
                                           q_len, max_pages_per_seq, num_pages, fp8, err,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_cache_append launch");
  return MLA_OK;
}

}  // extern "C"
