/*
 * lat_attn.h — fused grouped-query attention for one NVIDIA GB300 GPU (sm_103a).
 *
 * The operation is scaled-dot-product softmax attention with grouped-query heads:
 *
 *   for query row i of sequence b and query head h (G = n_heads / n_kv_heads,
 *   KV head hk = h / G, query position p = i + (kv_len - seq_len)):
 *     s_j   = scale * sum_d q[b,i,h,d] * k[b,j,hk,d]       over visible keys j
 *     out   = sum_j exp(s_j - m) * v[b,j,hk,:] / Z,   m = max_j s_j,  Z = sum_j exp(s_j - m)
 *     lse   = m + ln Z                                  (natural log)
 *
 * This is the row-wise attention of the larql "Inference Engine" page (section
 * "BLAS-Fused Attention": scores from K times Q, head scale, softmax, V^T times the
 * weights, GQA with any Q/KV ratio, causal masking built in), computed the way the
 * lattice-inference DESIGN page's fused Metal kernel does it ("Current Design":
 * fused attention with online softmax in registers, head_dim a compile-time
 * specialisation).  Visibility of key j from position p:
 *   causal != 0  ->  j <= p
 *   window  > 0  ->  p - j < window        (window keys including the query's own;
 *                                          Gemma 4 sliding layers use 1024, hf2q
 *                                          "Current Inference Path" page, section 2)
 * A row with no visible key gets out = 0 and lse = -inf.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers are caller-owned DEVICE memory unless stated otherwise.  The library
 *   allocates nothing; scratch space is passed in by the caller.
 * - Strides and row strides are in ELEMENTS of the call's dtype.  Within a row the
 *   heads of a tensor sit side by side with stride head_dim, so Q, K and V can be
 *   column slices of one packed QKV buffer read with the parent's row stride (the
 *   rlx-metal DESIGN page, "Cross-crate contract": per-tensor q/k/v row strides let
 *   attention read straight from the fused QKV output).
 * - head_dim is one of 64, 80, 128, 256, 512 (the Qwen3 and Gemma 4 head sizes named
 *   by the lattice-inference DESIGN page's compatibility matrix and the hf2q page);
 *   anything else returns LAT_ERR_UNSUPPORTED.
 * - n_heads % n_kv_heads != 0 returns LAT_ERR_INVALID_ARG (the same rule as
 *   INV-3 on the lattice-inference DESIGN page, without its CPU fallback: there is
 *   no fallback here, ever).
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *   stream).  Errors found on the host return at once and launch nothing.  Errors
 *   found on the device are written to `*status` (a device int32, nullable; it is
 *   set from 0 to the first error code seen and never cleared by the library);
 *   read it after synchronising.
 * - No global mutable state; calls on different streams are independent as long as
 *   their output and scratch buffers do not overlap.
 */
#ifndef LAT_ATTN_H
#define LAT_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { LAT_F32 = 0, LAT_BF16 = 1 } lat_dtype;

typedef enum {
    LAT_OK = 0,
    LAT_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad stride, bad ratio   */
    LAT_ERR_UNSUPPORTED = 2, /* head_dim or dtype not built, or a size past a limit  */
    LAT_ERR_WORKSPACE = 3,   /* decode workspace missing or too small                */
    LAT_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (launch, attribute) */
    LAT_ERR_BOUNDS = 5,      /* device: a cache position or kv_len out of range       */
    LAT_ERR_TIMEOUT = 6      /* device: a bounded pipeline wait ran out; kernel quit   */
} lat_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *lat_status_string(lat_status s);

/*
 * lat_attn_prefill — attention for seq_len query rows per sequence over kv_len keys.
 *
 * Layout (r = row index):
 *   q   element (b,i,h,d) at q[(b*seq_len + i)*q_rs + h*head_dim + d]
 *   k   element (b,j,hk,d) at k[(b*kv_len + j)*k_rs + hk*head_dim + d]; v likewise with v_rs
 *   out element (b,i,h,d) at out[(b*seq_len + i)*out_rs + h*head_dim + d], dtype dt
 *   lse (nullable) fp32 at lse[(b*seq_len + i)*n_heads + h]
 * kv_len >= seq_len >= 0 (kv_len > seq_len is a chunk of new queries appended after
 * kv_len - seq_len earlier keys).  dt = LAT_BF16 runs on the tensor cores
 * (bf16 operands, fp32 accumulation, one bf16 rounding of the output); dt = LAT_F32
 * runs exact fp32 arithmetic on the CUDA cores.
 * For LAT_BF16, q, k, v and out must be 16-byte aligned and q_rs, k_rs, v_rs, out_rs
 * multiples of 8 (the tensor-memory-access unit reads 16-byte aligned rows and the
 * epilogue writes 16-byte vectors), else LAT_ERR_INVALID_ARG.
 * Size limits (LAT_ERR_UNSUPPORTED): batch <= 65535, ceil(seq_len / 128) <= 65535, and
 * for LAT_BF16 at most 2^30 work items, an item being one 128-row query tile of one
 * query head (two items per tile and head at head_dim 512).
 * `out` must not overlap q, k or v.
 */
lat_status lat_attn_prefill(lat_dtype dt, const void *q, int64_t q_rs, const void *k,
                            int64_t k_rs, const void *v, int64_t v_rs, void *out,
                            int64_t out_rs, float *lse, int batch, int seq_len, int kv_len,
                            int n_heads, int n_kv_heads, int head_dim, int causal,
                            int window, float scale, int32_t *status, void *stream);

/*
 * lat_attn_prefill_softcap — lat_attn_prefill with the Gemma 2 score cap: each scaled
 * score s is replaced by softcap * tanh(s / softcap) before the softmax (the larql
 * "Inference Engine" page, section "BLAS-Fused Attention", step 2, "Scale + softcap",
 * listed there as a supported Gemma 2 feature).  softcap must be finite and >= 0; 0 means
 * no cap (the result of lat_attn_prefill); otherwise LAT_ERR_INVALID_ARG.  The lse is
 * taken over the capped scores.  All other arguments and rules are lat_attn_prefill's.
 */
lat_status lat_attn_prefill_softcap(lat_dtype dt, const void *q, int64_t q_rs, const void *k,
                                    int64_t k_rs, const void *v, int64_t v_rs, void *out,
                                    int64_t out_rs, float *lse, int batch, int seq_len,
                                    int kv_len, int n_heads, int n_kv_heads, int head_dim,
                                    int causal, int window, float scale, float softcap,
                                    int32_t *status, void *stream);

/*
 * lat_attn_prefill_cached — lat_attn_prefill reading K and V from an in-place KV cache:
 * a chunk of seq_len new query rows per sequence at positions kv_len - seq_len ..
 * kv_len - 1, attending to cache rows 0 .. kv_len - 1 (the chunk's own keys appended
 * first, e.g. by lat_kv_append).  This is the "full" (seq_len > 1) SDPA over a cache
 * that the hf2q target page leaves open for chunked prefill (open question Q2), in the
 * cache layout of its section 3.3.
 *
 * Layout: q, out and lse as in lat_attn_prefill; caches as in lat_attn_decode
 *   (element (b,j,hk,d) at cache[b*cache_seq_stride + j*cache_rs + hk*cache_head_stride + d],
 *   token-major or head-major).  Every sequence uses the same seq_len and kv_len
 *   (kv_len >= seq_len) and its cache must hold at least kv_len rows; slots at or past
 *   kv_len never reach the result (they may hold anything, NaN included).
 * For LAT_BF16, q, out and the cache bases must be 16-byte aligned and q_rs, out_rs and
 * the three cache strides multiples of 8, else LAT_ERR_INVALID_ARG.  Other rules and
 * errors are those of lat_attn_prefill.
 */
lat_status lat_attn_prefill_cached(lat_dtype dt, const void *q, int64_t q_rs,
                                   const void *k_cache, const void *v_cache, int64_t cache_rs,
                                   int64_t cache_head_stride, int64_t cache_seq_stride,
                                   void *out, int64_t out_rs, float *lse, int batch,
                                   int seq_len, int kv_len, int n_heads, int n_kv_heads,
                                   int head_dim, int causal, int window, float scale,
                                   int32_t *status, void *stream);

/*
 * lat_attn_decode_workspace_size — bytes of scratch lat_attn_decode needs for these
 * sizes (its split-KV partial results and merge counters).  Returns 0 for sizes the
 * library rejects.
 */
size_t lat_attn_decode_workspace_size(lat_dtype dt, int batch, int n_heads, int n_kv_heads,
                                      int head_dim, int max_kv_len);

/*
 * lat_attn_decode — one query token per sequence against an in-place KV cache.
 *
 * The decode step of the hf2q "Current Inference Path" page (section 3: attention at
 * seq_len 1 over the KV cache, right after the cache append).  The query of
 * sequence b sits at position kv_lens[b] - 1 and reads cached keys
 * max(0, kv_lens[b] - window) .. kv_lens[b] - 1 (all of 0 .. kv_lens[b]-1 when
 * window <= 0), so it equals the last row of a causal prefill over those keys.
 *
 * Layout:
 *   q      element (b,h,d) at q[b*q_rs + h*head_dim + d]
 *   caches element (b,j,hk,d) at cache[b*cache_seq_stride + j*cache_rs +
 *                                      hk*cache_head_stride + d]   (k_cache and v_cache)
 *          token-major [B, cap, Hkv*D]: cache_rs = Hkv*D, cache_head_stride = D;
 *          head-major  [B, Hkv, cap, D]: cache_rs = D, cache_head_stride = cap*D
 *          (the hf2q target page's per-layer cache [1, kv_heads, max_cache, head_dim]).
 *   kv_lens device int32 [batch], each in [0, max_kv_len]; a value outside that
 *          range sets *status = LAT_ERR_BOUNDS and that row's output is left unwritten.
 *   out    element (b,h,d) at out[b*out_rs + h*head_dim + d], dtype dt
 *   lse    nullable fp32 [batch, n_heads]
 * max_kv_len is a host-side upper bound used to size the launch; every sequence's
 * cache must hold at least max_kv_len rows (the kernel may load any row below
 * max_kv_len in whole tiles).  Cache slots at or past kv_lens[b] never reach the result
 * (they may hold anything, NaN included).
 * workspace: device scratch of at least lat_attn_decode_workspace_size(...) bytes,
 * 256-byte aligned; it must be zero-filled before its first use with a given layout
 * (the kernel returns its merge counters to zero, so later calls need no reset, except
 * after a call that reported LAT_ERR_TIMEOUT: zero it again), and calls sharing one
 * workspace must not overlap on the GPU.  Too small ->
 * LAT_ERR_WORKSPACE.  The size depends on the current device's SM count: size the
 * workspace with the device current that will run the call.  LAT_F32 needs no
 * workspace (its size is 0 and the pointer may be NULL).
 * For LAT_BF16, q, out and the cache base pointers must be 16-byte aligned and q_rs,
 * out_rs, cache_rs, cache_head_stride, cache_seq_stride multiples of 8 (tiles arrive
 * through the tensor-memory-access unit and results leave in 16-byte vectors), else
 * LAT_ERR_INVALID_ARG.
 * Size limits (LAT_ERR_UNSUPPORTED): batch <= 65535 and, for LAT_BF16, fewer than 2^23
 * work units, a unit being one sequence, one KV head and a block of up to 8 of its
 * query heads (batch * n_kv_heads * ceil(n_heads / n_kv_heads / 8)).
 */
lat_status lat_attn_decode(lat_dtype dt, const void *q, int64_t q_rs, const void *k_cache,
                           const void *v_cache, int64_t cache_rs, int64_t cache_head_stride,
                           int64_t cache_seq_stride, const int32_t *kv_lens, int max_kv_len,
                           void *out, int64_t out_rs, float *lse, int batch, int n_heads,
                           int n_kv_heads, int head_dim, int window, float scale,
                           void *workspace, size_t workspace_bytes, int32_t *status,
                           void *stream);

/*
 * lat_attn_decode_softcap — lat_attn_decode with the score cap of lat_attn_prefill_softcap
 * (softcap finite and >= 0, 0 = none).  Same arguments, workspace and rules otherwise.
 */
lat_status lat_attn_decode_softcap(lat_dtype dt, const void *q, int64_t q_rs,
                                   const void *k_cache, const void *v_cache, int64_t cache_rs,
                                   int64_t cache_head_stride, int64_t cache_seq_stride,
                                   const int32_t *kv_lens, int max_kv_len, void *out,
                                   int64_t out_rs, float *lse, int batch, int n_heads,
                                   int n_kv_heads, int head_dim, int window, float scale,
                                   float softcap, void *workspace, size_t workspace_bytes,
                                   int32_t *status, void *stream);

/*
 * lat_attn_decode_ring — lat_attn_decode over a ring cache for sliding-window layers: each
 * sequence's cache holds ring_capacity rows and the key at absolute position j sits in
 * row j % ring_capacity (the cache keeps the last ring_capacity positions).  kv_lens are
 * absolute lengths (they may exceed ring_capacity) and the visible keys are the last
 * `window` positions, which may wrap past the end of the ring: the cache-offset case
 * the hf2q pages flag for sliding layers (Current Inference Path, section 2 step 1:
 * sliding window 1024; Target Architecture, section 3.3 per-layer caches).
 * Requires 0 < window <= ring_capacity, else LAT_ERR_INVALID_ARG; size the workspace with
 * lat_attn_decode_workspace_size(..., max_kv_len = ring_capacity).  Rows of the ring
 * outside the window never reach the result.  All other rules are lat_attn_decode's.
 */
lat_status lat_attn_decode_ring(lat_dtype dt, const void *q, int64_t q_rs, const void *k_cache,
                                const void *v_cache, int64_t cache_rs, int64_t cache_head_stride,
                                int64_t cache_seq_stride, int ring_capacity,
                                const int32_t *kv_lens, int max_kv_len, void *out,
                                int64_t out_rs, float *lse, int batch, int n_heads,
                                int n_kv_heads, int head_dim, int window, float scale,
                                void *workspace, size_t workspace_bytes, int32_t *status,
                                void *stream);

/*
 * lat_attn_decode_static — lat_attn_decode without a caller workspace.  The pages have
 * no counterpart to this call; it exists for callers that cannot allocate device
 * memory: code running inside a host framework that owns all device memory, plugins
 * whose host forbids allocation after start-up, and latency-critical paths that cannot
 * afford an allocation's implicit synchronisation.
 *
 * Same arguments, layout and results as lat_attn_decode, minus workspace and
 * workspace_bytes.  The split-KV scratch is one fixed 16 MiB array in device global
 * memory that belongs to the library (every GPU the library is used on holds it until
 * the process exits).  The call allocates nothing and calls no allocating routine.
 * - Shapes whose scratch need (lat_attn_decode_workspace_size) exceeds 16 MiB return
 *   LAT_ERR_WORKSPACE and launch nothing.
 * - The first call on a device looks up the array's device address with that device
 *   current and caches it; make that first call before any stream capture.
 * - Every call on a device shares the array and it keeps the last call's contents: the
 *   call clears the part that must start at zero (an asynchronous memset on `stream`
 *   before the kernel), but calls that overlap on the GPU race on it, so serialise
 *   them (one stream, or explicit events).
 * - LAT_F32 needs no scratch and behaves exactly like lat_attn_decode.
 */
lat_status lat_attn_decode_static(lat_dtype dt, const void *q, int64_t q_rs,
                                  const void *k_cache, const void *v_cache, int64_t cache_rs,
                                  int64_t cache_head_stride, int64_t cache_seq_stride,
                                  const int32_t *kv_lens, int max_kv_len, void *out,
                                  int64_t out_rs, float *lse, int batch, int n_heads,
                                  int n_kv_heads, int head_dim, int window, float scale,
                                  int32_t *status, void *stream);

/*
 * lat_kv_append — in-place KV-cache append: row pos[b] + t of sequence b's cache
 * takes new row t, for t < n_new (the in-place "slice_set" append of the hf2q
 * "Current Inference Path" page, sections 1 and 3, and the kv_cache_write step of
 * the hf2q target page, section 6.1 step 6: "stride arithmetic must match exactly").
 *
 * Layout: caches as in lat_attn_decode; new element (b,t,hk,d) at
 *   k_new[(b*n_new + t)*new_rs + hk*head_dim + d] (v_new likewise), so the new rows can
 *   be column slices of a packed QKV buffer.  pos: device int32 [batch].
 * A sequence whose rows would fall outside [0, capacity) is skipped whole and sets
 * *status = LAT_ERR_BOUNDS.  New rows must not overlap the cache.
 */
lat_status lat_kv_append(lat_dtype dt, void *k_cache, void *v_cache, int64_t cache_rs,
                         int64_t cache_head_stride, int64_t cache_seq_stride, int capacity,
                         const void *k_new, const void *v_new, int64_t new_rs,
                         const int32_t *pos, int n_new, int batch, int n_kv_heads,
                         int head_dim, int32_t *status, void *stream);

/*
 * lat_kv_append_ring — lat_kv_append into a ring cache: new row t of sequence b goes to
 * row (pos[b] + t) % ring_capacity (positions are absolute and never out of range).
 * n_new must not exceed ring_capacity (rows would overwrite each other), else
 * LAT_ERR_INVALID_ARG; pos[b] < 0 sets *status = LAT_ERR_BOUNDS and skips the sequence.
 */
lat_status lat_kv_append_ring(lat_dtype dt, void *k_cache, void *v_cache, int64_t cache_rs,
                              int64_t cache_head_stride, int64_t cache_seq_stride,
                              int ring_capacity, const void *k_new, const void *v_new,
                              int64_t new_rs, const int32_t *pos, int n_new, int batch,
                              int n_kv_heads, int head_dim, int32_t *status, void *stream);

/*
 * lat_qkv_norm_rope_append — the steps right before attention, fused for the new token
 * rows of a fused QKV projection: Q norm and K norm (RMS norm over head_dim with a
 * head_dim weight), rotary position embedding, V unit norm or copy, then the KV-cache
 * append (the hf2q "Current Inference Path" page, section 3: Q norm, K norm, V unit norm,
 * RoPE apply, KV cache append; the lattice-inference DESIGN page's fused_qk_norm_rope).
 *
 * For new row t of sequence b at position p = pos[b] + t, with x one head of that row:
 *   Q, K heads:  y = x / sqrt(mean(x^2) + eps) * w   (w = q_norm_w or k_norm_w; NULL = 1)
 *                then element i < D/2 and element i + D/2 rotate by theta_i = p *
 *                rope_base^(-2i/D):  (a, b) -> (a cos - b sin, a sin + b cos)
 *   V heads:     x, or x / sqrt(mean(x^2) + eps) when v_unit_norm != 0
 * Layout: qkv row (b,t) at qkv[(b*n_new + t)*qkv_rs]: n_heads Q heads, then n_kv_heads K
 *   heads, then n_kv_heads V heads, each head_dim wide (the packed layout of
 *   lat_attn_prefill); q_out row (b,t) at q_out[(b*n_new + t)*q_out_rs] (n_heads heads);
 *   caches, capacity and pos as in lat_kv_append (rows p of sequence b).  Norm weights are
 *   head_dim elements of dtype dt.  fp32 arithmetic, one rounding to dt.
 * eps must be finite and >= 0 and rope_base finite and > 1, else LAT_ERR_INVALID_ARG.  A
 * sequence whose rows would fall outside [0, capacity) is skipped whole (nothing of it is
 * written, Q included) and sets *status = LAT_ERR_BOUNDS.
 */
lat_status lat_qkv_norm_rope_append(lat_dtype dt, const void *qkv, int64_t qkv_rs,
                                    const void *q_norm_w, const void *k_norm_w, float eps,
                                    double rope_base, int v_unit_norm, void *q_out,
                                    int64_t q_out_rs, void *k_cache, void *v_cache,
                                    int64_t cache_rs, int64_t cache_head_stride,
                                    int64_t cache_seq_stride, int capacity, const int32_t *pos,
                                    int n_new, int batch, int n_heads, int n_kv_heads,
                                    int head_dim, int32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LAT_ATTN_H */
