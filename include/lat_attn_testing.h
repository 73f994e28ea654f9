/*
 * lat_attn_testing.h — test hooks of the lat_attn library.  Not part of the compute API.
 *
 * lat_test_prefill_timeout runs the bf16 prefill kernel (causal, kv_len = seq_len,
 * scale 1/8, no lse) with its first K tile never loaded, so the tensor-core pipeline's
 * bounded wait for that tile must run out after `timeout_ns` nanoseconds.  Each CTA then
 * records LAT_ERR_TIMEOUT in *status (device int32, must be non-NULL and start at 0),
 * drains its in-flight copies and MMAs, frees its tensor memory and exits, leaving the
 * CUDA context usable.  Arguments and layout are those of lat_attn_prefill; the return
 * value reports host-side validation and launch errors only.  The output is unspecified.
 *
 * lat_test_decode_timeout runs the bf16 decode (window 0, scale 1/8, no lse) with the
 * first K/V stage of every CTA never filled, so the compute warps' bounded wait for it
 * (and the producer's wait for that stage to be released) must run out after
 * `timeout_ns` nanoseconds.  Each CTA then records LAT_ERR_TIMEOUT in *status (device
 * int32, non-NULL, starting at 0), drains its issued copies and exits; a deferred merge
 * kernel, if the shape uses one, still runs and finishes.  Arguments, layout and
 * workspace rules are those of lat_attn_decode; the output is unspecified, and the
 * workspace must be zero-filled again before its next use.
 *
 * lat_test_capped_scores evaluates the score cap of the bf16 kernels (the Gemma 2 softcap
 * of the larql "BLAS-Fused Attention" step 2, folded into the log2 domain) on n raw dot
 * products: out[i] = softcap * log2(e) * tanh(raw[i] * scale / softcap), formed exactly as
 * lat_attn_prefill_softcap and lat_attn_decode_softcap form it.  raw and out are device
 * arrays of n floats (n >= 0) that do not overlap; softcap > 0 and scale finite, else
 * LAT_ERR_INVALID_ARG.  Asynchronous on `stream`.
 */
#ifndef LAT_ATTN_TESTING_H
#define LAT_ATTN_TESTING_H

#include "lat_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

lat_status lat_test_prefill_timeout(const void *q, int64_t q_rs, const void *k, int64_t k_rs,
                                    const void *v, int64_t v_rs, void *out, int64_t out_rs,
                                    int batch, int seq_len, int n_heads, int n_kv_heads,
                                    int head_dim, uint64_t timeout_ns, int32_t *status,
                                    void *stream);
lat_status lat_test_decode_timeout(const void *q, int64_t q_rs, const void *k_cache,
                                   const void *v_cache, int64_t cache_rs,
                                   int64_t cache_head_stride, int64_t cache_seq_stride,
                                   const int32_t *kv_lens, int max_kv_len, void *out,
                                   int64_t out_rs, int batch, int n_heads, int n_kv_heads,
                                   int head_dim, void *workspace, size_t workspace_bytes,
                                   uint64_t timeout_ns, int32_t *status, void *stream);
lat_status lat_test_capped_scores(const float *raw, int64_t n, float scale, float softcap,
                                  float *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LAT_ATTN_TESTING_H */
