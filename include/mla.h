/*
 * mla.h -- C ABI of the GB300 (sm_103a) fused multi-head latent attention library.
 *
 * Two operations, both exact attention in flash form (scores S = Q K', online
 * softmax, O += P V -- Modular API docs, "KVPipelineGeneric" (nn/attention/gpu/
 * nvidia/sm100/mla_decode_utils), struct description and Parameters):
 *
 *   mla_prefill  causal (or full) self-attention over split nope+rope head depths,
 *                optionally with fp8 e4m3 Q_nope/K_nope/V and one fp32 scale per
 *                query and per key token ("MLASmemStorage" of nn/attention/gpu/
 *                nvidia/sm100/mla_prefill_per_token_scale: Fields q_smem, kv_smem,
 *                q_scale_smem, k_scale_smem).
 *   mla_decode   absorbed decode: T new query tokens per sequence attend to one
 *                shared latent head (d_latent + d_rope columns per token) kept in a
 *                paged cache; V is the first d_latent columns of the same rows.
 *                Split over the key axis across CTAs, then merged by log-sum-exp.
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers, contiguous, innermost dimension
 *     last, 16-byte aligned.  The caller owns every buffer (including the decode
 *     workspace); the library allocates no device memory and keeps no pointer
 *     after a call returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Inputs are only read; `out` and `lse` are written in full.
 *   - Argument errors are detected on the host before any launch and return a
 *     non-zero mla_status with nothing launched; mla_last_error() then returns a
 *     message (thread-local, valid until the next call on the same thread).
 *   - A launch failure returns MLA_ERR_CUDA.  Errors found by the device itself
 *     (a bounded pipeline wait that ran out) are latched in a device word and
 *     reported by mla_check_device_error().
 *   - No C++ exception crosses this boundary.
 *
 * Softmax scale and LSE: the score of query row i and key j is
 *   s_ij = softmax_scale * (q_nope_i . k_nope_j + q_rope_i . k_rope_j)
 * (fp8: q_nope_i scaled by q_scale_i, k_nope_j by k_scale_j); LSE_i is the natural
 * log of sum_j exp(s_ij) over the keys row i may see, stored as fp32.  A row that
 * sees no key gets O = 0 and LSE = -inf.
 */
#ifndef MLA_GB300_H_
#define MLA_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,  /* null pointer, negative/zero size, misalignment */
  MLA_ERR_UNSUPPORTED = 2,  /* valid but not built: head depths, dtypes, page size */
  MLA_ERR_WORKSPACE = 3,    /* decode workspace missing or too small */
  MLA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
  MLA_ERR_TIMEOUT = 5,      /* a device-side bounded wait ran out (device word) */
  MLA_ERR_DEVICE_CHECK = 6  /* a device-side bounds check failed (device word) */
} mla_status;

typedef enum {
  MLA_BF16 = 0,
  MLA_FP8_E4M3 = 1,
  MLA_FP32 = 2
} mla_dtype;

/*
 * mla_prefill -- O = softmax(S) V per (batch, head), S as above.
 *
 * Layouts (element type in brackets):
 *   q_nope  [B, S, H, d_nope]  (qkv_dtype)      q_rope [B, S, H, d_rope] (bf16)
 *   k_nope  [B, S, H, d_nope]  (qkv_dtype)      k_rope [B, S, d_rope]    (bf16)
 *           one rope key per token, shared by all H heads
 *   v       [B, S, H, d_v]     (qkv_dtype)
 *   q_scale [B, S] fp32, k_scale [B, S] fp32 -- required iff qkv_dtype is
 *           MLA_FP8_E4M3 (then k_scale also dequantises V), must be NULL for bf16
 *   out     [B, S, H, d_v]     (out_dtype: MLA_BF16, or MLA_FP32)
 *   lse     [B, H, S] fp32
 * causal != 0: query i sees keys 0..i (square problem).  causal == 0: all keys.
 * Supported: d_nope = 128, d_rope = 64, d_v = 128; qkv_dtype MLA_BF16 or
 * MLA_FP8_E4M3; S >= 1; B, H <= 65535 (offsets are 64-bit; B*S*H*128 must stay below
 * 9e18).  Larger sizes return MLA_ERR_UNSUPPORTED.
 */
mla_status mla_prefill(const void* q_nope, const void* q_rope, const void* k_nope,
                       const void* k_rope, const void* v, const float* q_scale,
                       const float* k_scale, void* out, float* lse, int B, int H, int S,
                       int d_nope, int d_rope, int d_v, float softmax_scale, int causal,
                       mla_dtype qkv_dtype, mla_dtype out_dtype, void* stream);

/*
 * mla_decode_workspace_size -- bytes of device workspace mla_decode needs for a
 * batch of B sequences with H heads and q_len new tokens each.  Independent of
 * the cache lengths (the split plan is sized for its worst case).
 */
size_t mla_decode_workspace_size(int B, int H, int q_len, int d_latent);

/*
 * mla_decode -- absorbed MLA decode over a paged latent cache.
 *
 *   q_latent   [B, q_len, H, d_latent] bf16     q_rope [B, q_len, H, d_rope] bf16
 *   kv_cache   [num_pages, page_size, d_latent + d_rope]  (kv_dtype: bf16 or e4m3)
 *   kv_scale   [num_pages, page_size] fp32 -- one scale per cache row; required iff
 *              kv_dtype is MLA_FP8_E4M3, must be NULL for bf16
 *   page_table [B, max_pages_per_seq] int32 -- token j of sequence b is row
 *              j % page_size of page page_table[b][j / page_size]; entries past
 *              the sequence's last page are never read
 *   cache_lens [B] int32 -- L_b, counting the q_len new tokens, which occupy
 *              positions L_b - q_len .. L_b - 1 (0 <= L_b <= max_pages*page_size)
 *   out        [B, q_len, H, d_latent] bf16
 *   lse        [B, H, q_len] fp32
 *   workspace  device buffer of at least mla_decode_workspace_size() bytes
 * causal != 0: new token t sees keys 0 .. L_b - q_len + t; causal == 0: keys
 * 0 .. L_b - 1.  Cache rows past L_b may hold anything (even NaN): they are
 * never mixed into a result.  Page indices must lie in [0, num_pages): entries
 * outside are reported through MLA_ERR_DEVICE_CHECK (that page is skipped).
 * Supported: d_latent = 512, d_rope = 64, page_size = 64, q_len * H <= 65536 (rows beyond
 * 128 are processed in tiles of 128 rows: q_len > 1 new tokens over a cached prefix is
 * chunked prefill in absorbed form, after mla_cache_append has written the chunk's rows),
 * B <= 65535, B * ceil(q_len * H / 128) <= 2^24, max_pages_per_seq * page_size < 2^31.
 * Larger sizes return MLA_ERR_UNSUPPORTED.
 */
mla_status mla_decode(const void* q_latent, const void* q_rope, const void* kv_cache,
                      const float* kv_scale, const int* page_table, const int* cache_lens,
                      void* out, float* lse, int B, int H, int q_len, int d_latent,
                      int d_rope, int page_size, int max_pages_per_seq, int num_pages,
                      float softmax_scale, int causal, mla_dtype kv_dtype, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * mla_decode_noalloc -- mla_decode for callers that cannot allocate device memory.
 * (This entry point has no counterpart in the source pages: it exists for callers that run
 * where cudaMalloc and other allocating calls are not allowed -- e.g. an inference engine
 * that owns all device memory from start-up, or a plugin hook that may not allocate -- and
 * therefore cannot supply mla_decode's workspace.)
 *
 * Arguments, layouts and results are those of mla_decode without the workspace: the split
 * partials and merge counters go to a scratch array compiled into the library, of
 * mla_decode_noalloc_max_workspace() bytes (48 MiB).  No call allocates or frees device memory
 * through this library or the CUDA runtime's allocator.
 *   - Set-up: the array lives in its own module.  Under CUDA's lazy module loading (the
 *     default) the driver loads that module, and reserves the 48 MiB on the device, the first
 *     time the array's address is looked up on that device; it is then held until the
 *     process exits.  A call with B = 0 does only that set-up on the current device (looks up
 *     the array's address with cudaGetSymbolAddress, loads the decode kernels and the device
 *     error word), ignores every other argument and launches nothing.  A caller that reserves
 *     device memory at start-up makes this call first, before its reservation and before any
 *     stream capture; without it, the first ordinary call on the device does the set-up.
 *   - A batch whose mla_decode_workspace_size() exceeds that size is rejected with
 *     MLA_ERR_WORKSPACE before anything is launched.
 *   - All calls on a device share the array, which keeps the last call's contents.  Every
 *     call writes its partials before reading them and zeroes the merge counters (with a
 *     kernel queued ahead of the decode kernel) before counting, so nothing has to be cleared
 *     by the caller.  Calls that overlap on the GPU race on the array; the caller must
 *     serialise them (one stream, or ordered streams).
 */
mla_status mla_decode_noalloc(const void* q_latent, const void* q_rope, const void* kv_cache,
                              const float* kv_scale, const int* page_table, const int* cache_lens,
                              void* out, float* lse, int B, int H, int q_len, int d_latent,
                              int d_rope, int page_size, int max_pages_per_seq, int num_pages,
                              float softmax_scale, int causal, mla_dtype kv_dtype, void* stream);

/* Bytes of the built-in scratch array used by mla_decode_noalloc. */
size_t mla_decode_noalloc_max_workspace(void);

/*
 * mla_cache_append -- write the q_len new tokens of every sequence into the paged latent
 * cache, where mla_decode reads them (the step before decode).  The pages say nothing about
 * how the cache is filled; this follows mla_decode's cache layout and cache_lens reading.
 *
 *   c_new      [B, q_len, d_latent + d_rope] bf16 -- the new tokens' latent then rope row
 *   kv_cache   [num_pages, page_size, d_latent + d_rope]  (kv_dtype: bf16 or e4m3), written
 *   kv_scale   [num_pages, page_size] fp32, written -- required iff kv_dtype is
 *              MLA_FP8_E4M3, must be NULL for bf16
 *   page_table [B, max_pages_per_seq] int32, cache_lens [B] int32 -- as for mla_decode:
 *              L_b counts the new tokens, token t goes to position L_b - q_len + t
 * bf16 cache: the row is copied.  e4m3 cache: per token, scale = max|x| / 448 (1 when the row
 * is all zero) in fp32, codes = e4m3(clamp(x / scale, -448, 448)) rounded to nearest even;
 * the scale is stored next to the row.  Positions below 0 (L_b < q_len) are not written;
 * a page index outside [0, num_pages) (or a position past max_pages_per_seq pages) skips the
 * row and is reported through MLA_ERR_DEVICE_CHECK.  Only the target rows are touched.
 * Supported: d_latent = 512, d_rope = 64, page_size = 64.
 */
mla_status mla_cache_append(const void* c_new, void* kv_cache, float* kv_scale,
                            const int* page_table, const int* cache_lens, int B, int q_len,
                            int d_latent, int d_rope, int page_size, int max_pages_per_seq,
                            int num_pages, mla_dtype kv_dtype, void* stream);

/*
 * mla_absorb -- the per-head absorption product either side of absorbed decode:
 *     y[r, h, :] = x[r, h, :] @ w[h]      (fp32 accumulation, bf16 round-to-nearest-even out)
 *   x [R, H, K] bf16, w [H, K, N] bf16, y [R, H, N] bf16 (all contiguous, 16-byte aligned).
 * Before decode: x = q_nope [B*q_len, H, d_nope], w = W_UK [H, d_nope, d_latent] gives
 * q_latent; after it: x = O_latent [B*q_len, H, d_latent], w = W_UV [H, d_latent, d_v] gives
 * the output.  The pages only name the absorbed (latent) form of decode; this entry point is
 * the plain product that feeds and follows it.
 * Supported: K a multiple of 64, N a multiple of 128, R >= 1, H <= 65535.
 */
mla_status mla_absorb(const void* x, const void* w, void* y, int R, int H, int K, int N,
                      void* stream);

/*
 * mla_prefill_backward_workspace_size -- bytes of device workspace mla_prefill_backward
 * needs (two fp32 vectors of B * H * ceil(S / 128) * 128 entries).
 */
size_t mla_prefill_backward_workspace_size(int B, int H, int S);

/*
 * mla_prefill_backward -- gradients of bf16 MLA prefill with respect to its operands.
 * The pages define the forward step only (S = Q K', O += P V); this is its exact derivative
 * for an upstream gradient d_out, reusing the forward's O and LSE:
 *   P = exp(s - LSE),  dV = P' dO,  dP = dO V',  D_i = sum_d dO_id O_id,  dS = P * (dP - D),
 *   dQ = softmax_scale dS [Kn|Kr],  dK = softmax_scale dS' [Qn|Qr]
 * per (batch, head); the rope key is shared by the heads, so dk_rope is the sum over heads.
 *
 *   q_nope, q_rope, k_nope, k_rope, v   the forward's bf16 inputs (layouts of mla_prefill)
 *   out     [B, S, H, d_v] bf16 -- the forward's output;  lse [B, H, S] fp32 -- its LSE
 *   d_out   [B, S, H, d_v] bf16 -- upstream gradient
 *   dq_nope [B, S, H, d_nope] bf16, dq_rope [B, S, H, d_rope] bf16,
 *   dk_nope [B, S, H, d_nope] bf16, dv [B, S, H, d_v] bf16   -- written in full
 *   dk_rope [B, S, d_rope] fp32 -- written in full (zeroed, then accumulated over heads)
 *   workspace  device buffer of at least mla_prefill_backward_workspace_size() bytes
 * causal as for mla_prefill.  All gradients are accumulated in fp32; P and dS enter the
 * products as bf16.  Supported: d_nope = 128, d_rope = 64, d_v = 128, bf16 only,
 * B, H <= 65535 (larger: MLA_ERR_UNSUPPORTED).
 */
mla_status mla_prefill_backward(const void* q_nope, const void* q_rope, const void* k_nope,
                                const void* k_rope, const void* v, const void* out,
                                const float* lse, const void* d_out, void* dq_nope,
                                void* dq_rope, void* dk_nope, float* dk_rope, void* dv, int B,
                                int H, int S, int d_nope, int d_rope, int d_v,
                                float softmax_scale, int causal, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * mla_check_device_error -- synchronise `stream`, then read and clear the device
 * error word latched by earlier kernels of this library on the current device.
 * Returns MLA_OK, MLA_ERR_TIMEOUT or MLA_ERR_DEVICE_CHECK (or MLA_ERR_CUDA if the
 * synchronisation itself failed).
 */
mla_status mla_check_device_error(void* stream);

/* Message describing the last non-OK status returned on this thread. */
const char* mla_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_H_ */
