// api.cu — the C ABI declared in include/lat_attn.h: argument validation, launch planning,
// tensor-map encoding and dispatch to the kernels.  No allocation, no global mutable state
// (the driver entry point for tensor-map encoding is resolved once and then read-only).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "kernels.h"
#include "lat_attn.h"
#include "lat_attn_testing.h"

namespace {

bool supported_head_dim(int d) { return d == 64 || d == 80 || d == 128 || d == 256 || d == 512; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 4-D bf16 map over (head-dim d, head, row, batch) with a [64, 1, box_rows, 1] box and
// 128-byte swizzle.  Columns past head_dim and rows past `rows` read as zero.
bool make_head_map(CUtensorMap *m, const void *base, int head_dim, int heads, int rows,
                   int batch, int64_t row_stride, int box_rows) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)heads, (cuuint64_t)rows,
                                (cuuint64_t)batch};
    const cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2, (cuuint64_t)row_stride * 2,
                                   (cuuint64_t)row_stride * 2 * (cuuint64_t)rows};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D bf16 map over a KV cache: (head-dim d, KV head, row < rows, sequence) with the
// cache's own element strides, a [64, 1, box_rows, 1] box and 128-byte swizzle.
bool make_cache_map(CUtensorMap *m, const void *base, int head_dim, int heads, int rows,
                    int batch, int64_t row_stride, int64_t head_stride, int64_t seq_stride,
                    int box_rows,
                    CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)heads, (cuuint64_t)rows,
                                (cuuint64_t)batch};
    const cuuint64_t strides[3] = {(cuuint64_t)head_stride * 2, (cuuint64_t)row_stride * 2,
                                   (cuuint64_t)seq_stride * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 5-D bf16 map over the same tensor as make_cache_map, with the head dimension split into
// 64-column chunks: (d in chunk, row < rows, chunk, head, batch), 128-byte swizzle, box
// [64, box_rows, box_chunks, 1, 1].  One box lands as box_chunks consecutive
// [box_rows x 128 B] chunks: a whole multi-chunk tile in one copy.
bool make_chunked_map(CUtensorMap *m, const void *base, int head_dim, int heads, int rows,
                      int batch, int64_t row_stride, int64_t head_stride, int64_t seq_stride,
                      int box_rows, int box_chunks,
                      CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_128B) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr || head_dim % 64 != 0) return false;
    const cuuint64_t dims[5] = {64, (cuuint64_t)rows, (cuuint64_t)(head_dim / 64),
                                (cuuint64_t)heads, (cuuint64_t)batch};
    const cuuint64_t strides[4] = {(cuuint64_t)row_stride * 2, 128, (cuuint64_t)head_stride * 2,
                                   (cuuint64_t)seq_stride * 2};
    const cuuint32_t box[5] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_chunks, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map over decode queries: (head-dim d, query head, sequence), 8-head boxes
bool make_query_map(CUtensorMap *m, const void *base, int head_dim, int heads, int batch,
                    int64_t row_stride) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)heads, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)row_stride * 2};
    const cuuint32_t box[3] = {64, 8, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map over a prefill output: (column < heads * head_dim, row < rows, batch) with
// 32-row boxes of box_cols columns, swizzled to the box's row width (128 or 64 bytes).
// Stores clip at the row extent, so rows past a sequence's end are never written.
bool make_out_map(CUtensorMap *m, void *base, int head_dim, int heads, int rows, int batch,
                  int64_t row_stride, int box_cols) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (fn == nullptr || (box_cols != 64 && box_cols != 32)) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)heads * (cuuint64_t)head_dim, (cuuint64_t)rows,
                                (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)row_stride * 2,
                                   (cuuint64_t)row_stride * 2 * (cuuint64_t)rows};
    const cuuint32_t box[3] = {(cuuint32_t)box_cols, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE,
              box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int current_sm_count(int *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    return cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;  // 4 s per CTA

// Where K and V element (b, j, hk, d) live: base + b*seq + j*row + hk*head + d (elements).
struct KvStrides {
    int64_t k_row, k_head, k_seq, v_row, v_head, v_seq;
};

lat_status prefill_impl(lat_dtype dt, const void *q, int64_t q_rs, const void *k, const void *v,
                        const KvStrides &kv, void *out, int64_t out_rs, float *lse, int batch,
                        int seq_len, int kv_len, int n_heads, int n_kv_heads, int head_dim,
                        int causal, int window, float scale, float softcap, int32_t *status,
                        void *stream, uint64_t timeout_ns, int skip_kv_load) {
    if (dt != LAT_F32 && dt != LAT_BF16) return LAT_ERR_INVALID_ARG;
    if (!(softcap >= 0.f) || !isfinite(softcap)) return LAT_ERR_INVALID_ARG;
    if (batch < 0 || seq_len < 0 || kv_len < seq_len || n_heads <= 0 || n_kv_heads <= 0 ||
        n_heads % n_kv_heads != 0)
        return LAT_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim)) return LAT_ERR_UNSUPPORTED;
    if (!isfinite(scale)) return LAT_ERR_INVALID_ARG;
    if (batch == 0 || seq_len == 0) return LAT_OK;
    if (!q || !k || !v || !out) return LAT_ERR_INVALID_ARG;
    if (q_rs < (int64_t)n_heads * head_dim || out_rs < (int64_t)n_heads * head_dim ||
        kv.k_row <= 0 || kv.k_head <= 0 || kv.k_seq <= 0 || kv.v_row <= 0 || kv.v_head <= 0 ||
        kv.v_seq <= 0)
        return LAT_ERR_INVALID_ARG;
    if (batch > 65535 || (seq_len + 127) / 128 > 65535) return LAT_ERR_UNSUPPORTED;
    if (window < 0) window = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    if (dt == LAT_F32) {
        lat::RowAttnArgs a{};
        a.q = static_cast<const float *>(q);
        a.q_rs = q_rs;
        a.k = static_cast<const float *>(k);
        a.v = static_cast<const float *>(v);
        a.k_seq = kv.k_seq;
        a.k_row = kv.k_row;
        a.k_head = kv.k_head;
        a.v_seq = kv.v_seq;
        a.v_row = kv.v_row;
        a.v_head = kv.v_head;
        a.out = static_cast<float *>(out);
        a.out_rs = out_rs;
        a.lse = lse;
        a.batch = batch;
        a.seq_len = seq_len;
        a.kv_len = kv_len;
        a.n_heads = n_heads;
        a.n_kv_heads = n_kv_heads;
        a.head_dim = head_dim;
        a.causal = causal != 0;
        a.window = window;
        a.scale = scale;
        a.softcap = softcap;
        a.kv_lens = nullptr;
        a.max_kv_len = kv_len;
        a.status = status;
        return lat::launch_row_attention_f32(a, s) == cudaSuccess ? LAT_OK : LAT_ERR_CUDA;
    }

    // bf16: tensor-memory-access reads need 16-byte aligned bases and row strides
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || q_rs % 8 ||
        out_rs % 8 || kv.k_row % 8 || kv.k_head % 8 || kv.k_seq % 8 || kv.v_row % 8 ||
        kv.v_head % 8 || kv.v_seq % 8)
        return LAT_ERR_INVALID_ARG;
    if (lat::prefill_tc_items(batch, n_heads, head_dim, seq_len) > lat::kPrefillMaxItems)
        return LAT_ERR_UNSUPPORTED;
    lat::PrefillTcArgs a{};
    a.wide = lat::prefill_tc_wide(head_dim, seq_len, kv_len, causal, window) ? 1 : 0;
    a.pair = lat::prefill_tc_pair(head_dim, n_heads, n_kv_heads) ? 1 : 0;
    const int k_box = lat::prefill_tc_box_rows(head_dim, a.wide != 0, a.pair != 0, false);
    const int v_box = lat::prefill_tc_box_rows(head_dim, a.wide != 0, a.pair != 0, true);
    // K/V maps span exactly kv_len rows per sequence: rows past it read as zeros, so cache
    // slots beyond the visible keys (which may hold anything) never reach the MMA.  Head
    // dims that are whole 64-column chunks move each tile in one copy (chunked maps: Q all
    // chunks of 128 rows, K all chunks of its rows, V the chunks of this CTA's columns).
    a.chunked = lat::prefill_tc_chunked(head_dim, a.pair != 0) ? 1 : 0;
    if (a.chunked) {
        const int v_chunks = lat::prefill_tc_v_chunks(head_dim, a.pair != 0);
        if (!make_chunked_map(&a.tm_q, q, head_dim, n_heads, seq_len, batch, q_rs, head_dim,
                              (int64_t)seq_len * q_rs, 128, head_dim / 64) ||
            !make_chunked_map(&a.tm_k, k, head_dim, n_kv_heads, kv_len, batch, kv.k_row,
                              kv.k_head, kv.k_seq, k_box, head_dim / 64) ||
            !make_chunked_map(&a.tm_v, v, head_dim, n_kv_heads, kv_len, batch, kv.v_row,
                              kv.v_head, kv.v_seq, v_box, v_chunks))
            return LAT_ERR_CUDA;
    } else if (!make_head_map(&a.tm_q, q, head_dim, n_heads, seq_len, batch, q_rs, 128) ||
        !make_cache_map(&a.tm_k, k, head_dim, n_kv_heads, kv_len, batch, kv.k_row, kv.k_head,
                        kv.k_seq, k_box, CU_TENSOR_MAP_L2_PROMOTION_L2_128B) ||
        !make_cache_map(&a.tm_v, v, head_dim, n_kv_heads, kv_len, batch, kv.v_row, kv.v_head,
                        kv.v_seq, v_box, CU_TENSOR_MAP_L2_PROMOTION_L2_128B))
        return LAT_ERR_CUDA;
    const int out_box = lat::prefill_tc_out_box_cols(head_dim, a.pair != 0);
    if (out_box > 0 &&
        !make_out_map(&a.tm_out, out, head_dim, n_heads, seq_len, batch, out_rs, out_box))
        return LAT_ERR_CUDA;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.out_rs = out_rs;
    a.out_v8 = reinterpret_cast<uintptr_t>(out) % 32 == 0 && out_rs % 16 == 0;
    a.lse = lse;
    a.batch = batch;
    a.seq_len = seq_len;
    a.kv_len = kv_len;
    a.n_heads = n_heads;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.causal = causal != 0;
    a.window = window;
    a.scale_log2 = scale * kLog2e;
    a.cap_log2 = softcap > 0.f ? softcap * kLog2e : 0.f;
    a.raw_over_cap = softcap > 0.f ? scale / softcap : 0.f;
    a.status = status;
    a.timeout_ns = timeout_ns;
    a.test_skip_kv_load = skip_kv_load;
    int sms = 0;
    if (!current_sm_count(&sms)) return LAT_ERR_CUDA;
    return lat::launch_prefill_tc(a, sms, s) == cudaSuccess ? LAT_OK : LAT_ERR_CUDA;
}

}  // namespace

extern "C" {

const char *lat_status_string(lat_status st) {
    switch (st) {
        case LAT_OK: return "LAT_OK";
        case LAT_ERR_INVALID_ARG: return "LAT_ERR_INVALID_ARG";
        case LAT_ERR_UNSUPPORTED: return "LAT_ERR_UNSUPPORTED";
        case LAT_ERR_WORKSPACE: return "LAT_ERR_WORKSPACE";
        case LAT_ERR_CUDA: return "LAT_ERR_CUDA";
        case LAT_ERR_BOUNDS: return "LAT_ERR_BOUNDS";
        case LAT_ERR_TIMEOUT: return "LAT_ERR_TIMEOUT";
    }
    return "LAT_ERR_UNKNOWN";
}

lat_status lat_attn_prefill(lat_dtype dt, const void *q, int64_t q_rs, const void *k,
                            int64_t k_rs, const void *v, int64_t v_rs, void *out,
                            int64_t out_rs, float *lse, int batch, int seq_len, int kv_len,
                            int n_heads, int n_kv_heads, int head_dim, int causal, int window,
                            float scale, int32_t *status, void *stream) {
    if (k_rs < (int64_t)n_kv_heads * head_dim || v_rs < (int64_t)n_kv_heads * head_dim)
        return LAT_ERR_INVALID_ARG;
    const KvStrides kv{k_rs, head_dim, (int64_t)kv_len * k_rs, v_rs, head_dim, (int64_t)kv_len * v_rs};
    return prefill_impl(dt, q, q_rs, k, v, kv, out, out_rs, lse, batch, seq_len, kv_len, n_heads,
                        n_kv_heads, head_dim, causal, window, scale, 0.f, status, stream,
                        kDefaultTimeoutNs, 0);
}

lat_status lat_attn_prefill_softcap(lat_dtype dt, const void *q, int64_t q_rs, const void *k,
                                    int64_t k_rs, const void *v, int64_t v_rs, void *out,
                                    int64_t out_rs, float *lse, int batch, int seq_len,
                                    int kv_len, int n_heads, int n_kv_heads, int head_dim,
                                    int causal, int window, float scale, float softcap,
                                    int32_t *status, void *stream) {
    if (k_rs < (int64_t)n_kv_heads * head_dim || v_rs < (int64_t)n_kv_heads * head_dim)
        return LAT_ERR_INVALID_ARG;
    const KvStrides kv{k_rs, head_dim, (int64_t)kv_len * k_rs, v_rs, head_dim, (int64_t)kv_len * v_rs};
    return prefill_impl(dt, q, q_rs, k, v, kv, out, out_rs, lse, batch, seq_len, kv_len, n_heads,
                        n_kv_heads, head_dim, causal, window, scale, softcap, status, stream,
                        kDefaultTimeoutNs, 0);
}

lat_status lat_attn_prefill_cached(lat_dtype dt, const void *q, int64_t q_rs,
                                   const void *k_cache, const void *v_cache, int64_t cache_rs,
                                   int64_t cache_head_stride, int64_t cache_seq_stride,
                                   void *out, int64_t out_rs, float *lse, int batch,
                                   int seq_len, int kv_len, int n_heads, int n_kv_heads,
                                   int head_dim, int causal, int window, float scale,
                                   int32_t *status, void *stream) {
    const KvStrides kv{cache_rs, cache_head_stride, cache_seq_stride,
                       cache_rs, cache_head_stride, cache_seq_stride};
    return prefill_impl(dt, q, q_rs, k_cache, v_cache, kv, out, out_rs, lse, batch, seq_len,
                        kv_len, n_heads, n_kv_heads, head_dim, causal, window, scale, 0.f, status,
                        stream, kDefaultTimeoutNs, 0);
}

lat_status lat_test_prefill_timeout(const void *q, int64_t q_rs, const void *k, int64_t k_rs,
                                    const void *v, int64_t v_rs, void *out, int64_t out_rs,
                                    int batch, int seq_len, int n_heads, int n_kv_heads,
                                    int head_dim, uint64_t timeout_ns, int32_t *status,
                                    void *stream) {
    const KvStrides kv{k_rs, head_dim, (int64_t)seq_len * k_rs, v_rs, head_dim,
                       (int64_t)seq_len * v_rs};
    return prefill_impl(LAT_BF16, q, q_rs, k, v, kv, out, out_rs, nullptr, batch, seq_len,
                        seq_len, n_heads, n_kv_heads, head_dim, 1, 0, 0.125f, 0.f, status, stream,
                        timeout_ns, 1);
}

size_t lat_attn_decode_workspace_size(lat_dtype dt, int batch, int n_heads, int n_kv_heads,
                                      int head_dim, int max_kv_len) {
    if (dt == LAT_F32) return 0;
    if (dt != LAT_BF16 || batch < 0 || n_heads <= 0 || n_kv_heads <= 0 ||
        n_heads % n_kv_heads != 0 || !supported_head_dim(head_dim) || max_kv_len < 0)
        return 0;
    int sms = 0;
    if (!current_sm_count(&sms)) return 0;
    lat::DecodePlan plan;
    if (!lat::plan_decode_bf16(batch, n_heads, n_kv_heads, head_dim, max_kv_len, 0, sms, &plan))
        return 0;
    return plan.total_bytes;
}

}  // extern "C"

namespace {

lat_status decode_impl(lat_dtype dt, const void *q, int64_t q_rs, const void *k_cache,
                       const void *v_cache, int64_t cache_rs, int64_t cache_head_stride,
                       int64_t cache_seq_stride, const int32_t *kv_lens, int max_kv_len,
                       void *out, int64_t out_rs, float *lse, int batch, int n_heads,
                       int n_kv_heads, int head_dim, int window, float scale, float softcap,
                       int ring, void *workspace, size_t workspace_bytes, int32_t *status,
                       void *stream, uint64_t timeout_ns, int skip_load) {
    if (dt != LAT_F32 && dt != LAT_BF16) return LAT_ERR_INVALID_ARG;
    if (!(softcap >= 0.f) || !isfinite(softcap)) return LAT_ERR_INVALID_ARG;
    // a ring cache keeps only the last `ring` positions: the window must fit in it
    if (ring < 0 || (ring > 0 && (window <= 0 || window > ring))) return LAT_ERR_INVALID_ARG;
    if (batch < 0 || max_kv_len < 0 || n_heads <= 0 || n_kv_heads <= 0 ||
        n_heads % n_kv_heads != 0)
        return LAT_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim)) return LAT_ERR_UNSUPPORTED;
    if (!isfinite(scale)) return LAT_ERR_INVALID_ARG;
    if (batch == 0) return LAT_OK;
    if (!q || !k_cache || !v_cache || !kv_lens || !out) return LAT_ERR_INVALID_ARG;
    if (q_rs < (int64_t)n_heads * head_dim || out_rs < (int64_t)n_heads * head_dim ||
        cache_rs <= 0 || cache_head_stride <= 0 || cache_seq_stride <= 0)
        return LAT_ERR_INVALID_ARG;
    if (batch > 65535) return LAT_ERR_UNSUPPORTED;
    if (window < 0) window = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    if (dt == LAT_F32) {
        lat::RowAttnArgs a{};
        a.q = static_cast<const float *>(q);
        a.q_rs = q_rs;
        a.k = static_cast<const float *>(k_cache);
        a.v = static_cast<const float *>(v_cache);
        a.k_seq = a.v_seq = cache_seq_stride;
        a.k_row = a.v_row = cache_rs;
        a.k_head = a.v_head = cache_head_stride;
        a.out = static_cast<float *>(out);
        a.out_rs = out_rs;
        a.lse = lse;
        a.batch = batch;
        a.seq_len = 1;
        a.kv_len = 0;
        a.n_heads = n_heads;
        a.n_kv_heads = n_kv_heads;
        a.head_dim = head_dim;
        a.causal = 1;
        a.window = window;
        a.scale = scale;
        a.softcap = softcap;
        a.kv_lens = kv_lens;
        a.max_kv_len = max_kv_len;
        a.ring = ring;
        a.status = status;
        return lat::launch_row_attention_f32(a, s) == cudaSuccess ? LAT_OK : LAT_ERR_CUDA;
    }

    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        q_rs % 8 || cache_rs % 8 || cache_head_stride % 8 || cache_seq_stride % 8 || out_rs % 8)
        return LAT_ERR_INVALID_ARG;
    if (lat::decode_bf16_units(batch, n_heads, n_kv_heads) >= lat::kDecodeMaxUnits)
        return LAT_ERR_UNSUPPORTED;
    int sms = 0;
    if (!current_sm_count(&sms)) return LAT_ERR_CUDA;
    // rows per sequence: the ring, or every position up to max_kv_len; the scratch layout
    // is sized by the same count (a ring's visible keys never exceed it)
    const int rows = ring > 0 ? ring : max_kv_len;
    lat::DecodePlan plan;
    if (!lat::plan_decode_bf16(batch, n_heads, n_kv_heads, head_dim, rows, window, sms, &plan))
        return LAT_ERR_UNSUPPORTED;
    if (workspace == nullptr || workspace_bytes < plan.total_bytes ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return LAT_ERR_WORKSPACE;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    lat::DecodeArgs a{};
    if (max_kv_len > 0) {
        const int box = lat::decode_bf16_tile_keys(head_dim);
        // head dims of up to four whole 64-column chunks take each K (or V) tile in one
        // copy (at head_dim 512, eight 32-row chunks per copy measured 2.4 % slower than
        // eight copies)
        a.chunked = head_dim % 64 == 0 && head_dim <= 256 ? 1 : 0;
        const bool maps_ok =
            a.chunked
                ? make_chunked_map(&a.tm_k, k_cache, head_dim, n_kv_heads, rows, batch, cache_rs,
                                   cache_head_stride, cache_seq_stride, box, head_dim / 64,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B) &&
                      make_chunked_map(&a.tm_v, v_cache, head_dim, n_kv_heads, rows, batch,
                                       cache_rs, cache_head_stride, cache_seq_stride, box,
                                       head_dim / 64, CU_TENSOR_MAP_L2_PROMOTION_L2_256B)
                : make_cache_map(&a.tm_k, k_cache, head_dim, n_kv_heads, rows, batch, cache_rs,
                                 cache_head_stride, cache_seq_stride, box) &&
                      make_cache_map(&a.tm_v, v_cache, head_dim, n_kv_heads, rows, batch,
                                     cache_rs, cache_head_stride, cache_seq_stride, box);
        const bool partial_ok =
            make_cache_map(&a.tm_k16, k_cache, head_dim, n_kv_heads, rows, batch, cache_rs,
                           cache_head_stride, cache_seq_stride, 16) &&
            make_cache_map(&a.tm_v16, v_cache, head_dim, n_kv_heads, rows, batch, cache_rs,
                           cache_head_stride, cache_seq_stride, 16);
        if (!maps_ok || !partial_ok ||
            !make_query_map(&a.tm_q, q, head_dim, n_heads, batch, q_rs))
            return LAT_ERR_CUDA;
    }
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.q_rs = q_rs;
    a.k_cache = static_cast<const __nv_bfloat16 *>(k_cache);
    a.v_cache = static_cast<const __nv_bfloat16 *>(v_cache);
    a.cache_rs = cache_rs;
    a.cache_head = cache_head_stride;
    a.cache_seq = cache_seq_stride;
    a.kv_lens = kv_lens;
    a.max_kv_len = max_kv_len;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.out_rs = out_rs;
    a.lse = lse;
    a.batch = batch;
    a.n_heads = n_heads;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.window = window;
    a.ring = ring;
    a.scale_log2 = scale * kLog2e;
    a.cap_log2 = softcap > 0.f ? softcap * kLog2e : 0.f;
    a.raw_over_cap = softcap > 0.f ? scale / softcap : 0.f;
    a.part_o = reinterpret_cast<float *>(ws);
    a.part_lse = reinterpret_cast<float *>(ws + plan.part_o_bytes);
    a.counters = reinterpret_cast<int32_t *>(ws + plan.part_o_bytes + plan.part_lse_bytes);
    a.max_splits = plan.max_splits;
    a.min_seg = plan.min_seg;
    a.defer_merge = plan.defer_merge;
    a.piece_count = a.counters;  // the same scratch region, used one way or the other
    a.timeout_ns = timeout_ns;
    a.test_skip_load = skip_load;
    a.status = status;
    return lat::launch_decode_bf16(a, plan.grid, s) == cudaSuccess ? LAT_OK : LAT_ERR_CUDA;
}

}  // namespace

extern "C" {

lat_status lat_attn_decode(lat_dtype dt, const void *q, int64_t q_rs, const void *k_cache,
                           const void *v_cache, int64_t cache_rs, int64_t cache_head_stride,
                           int64_t cache_seq_stride, const int32_t *kv_lens, int max_kv_len,
                           void *out, int64_t out_rs, float *lse, int batch, int n_heads,
                           int n_kv_heads, int head_dim, int window, float scale,
                           void *workspace, size_t workspace_bytes, int32_t *status,
                           void *stream) {
    return decode_impl(dt, q, q_rs, k_cache, v_cache, cache_rs, cache_head_stride,
                       cache_seq_stride, kv_lens, max_kv_len, out, out_rs, lse, batch, n_heads,
                       n_kv_heads, head_dim, window, scale, 0.f, 0, workspace,
                       workspace_bytes, status, stream,
                       kDefaultTimeoutNs, 0);
}

lat_status lat_attn_decode_ring(lat_dtype dt, const void *q, int64_t q_rs, const void *k_cache,
                                const void *v_cache, int64_t cache_rs, int64_t cache_head_stride,
                                int64_t cache_seq_stride, int ring_capacity,
                                const int32_t *kv_lens, int max_kv_len, void *out,
                                int64_t out_rs, float *lse, int batch, int n_heads,
                                int n_kv_heads, int head_dim, int window, float scale,
                                void *workspace, size_t workspace_bytes, int32_t *status,
                                void *stream) {
    if (ring_capacity <= 0) return LAT_ERR_INVALID_ARG;
    return decode_impl(dt, q, q_rs, k_cache, v_cache, cache_rs, cache_head_stride,
                       cache_seq_stride, kv_lens, max_kv_len, out, out_rs, lse, batch, n_heads,
                       n_kv_heads, head_dim, window, scale, 0.f, ring_capacity, workspace,
                       workspace_bytes, status, stream,
                       kDefaultTimeoutNs, 0);
}

lat_status lat_attn_decode_softcap(lat_dtype dt, const void *q, int64_t q_rs,
                                   const void *k_cache, const void *v_cache, int64_t cache_rs,
                                   int64_t cache_head_stride, int64_t cache_seq_stride,
                                   const int32_t *kv_lens, int max_kv_len, void *out,
                                   int64_t out_rs, float *lse, int batch, int n_heads,
                                   int n_kv_heads, int head_dim, int window, float scale,
                                   float softcap, void *workspace, size_t workspace_bytes,
                                   int32_t *status, void *stream) {
    return decode_impl(dt, q, q_rs, k_cache, v_cache, cache_rs, cache_head_stride,
                       cache_seq_stride, kv_lens, max_kv_len, out, out_rs, lse, batch, n_heads,
                       n_kv_heads, head_dim, window, scale, softcap, 0, workspace,
                       workspace_bytes, status, stream,
                       kDefaultTimeoutNs, 0);
}

lat_status lat_test_decode_timeout(const void *q, int64_t q_rs, const void *k_cache,
                                   const void *v_cache, int64_t cache_rs,
                                   int64_t cache_head_stride, int64_t cache_seq_stride,
                                   const int32_t *kv_lens, int max_kv_len, void *out,
                                   int64_t out_rs, int batch, int n_heads, int n_kv_heads,
                                   int head_dim, void *workspace, size_t workspace_bytes,
                                   uint64_t timeout_ns, int32_t *status, void *stream) {
    return decode_impl(LAT_BF16, q, q_rs, k_cache, v_cache, cache_rs, cache_head_stride,
                       cache_seq_stride, kv_lens, max_kv_len, out, out_rs, nullptr, batch,
                       n_heads, n_kv_heads, head_dim, 0, 0.125f, 0.f, 0, workspace,
                       workspace_bytes, status, stream, timeout_ns, 1);
}

lat_status lat_test_capped_scores(const float *raw, int64_t n, float scale, float softcap,
                                  float *out, void *stream) {
    if (n < 0 || !(softcap > 0.f) || !isfinite(scale)) return LAT_ERR_INVALID_ARG;
    if (n == 0) return LAT_OK;
    if (raw == nullptr || out == nullptr) return LAT_ERR_INVALID_ARG;
    // the same two factors the attention entry points hand their kernels
    return lat::launch_capped_scores(raw, n, scale / softcap, softcap * kLog2e, out,
                                     static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? LAT_OK
               : LAT_ERR_CUDA;
}

}  // extern "C"

namespace {

lat_status append_impl(lat_dtype dt, void *k_cache, void *v_cache, int64_t cache_rs,
                       int64_t cache_head_stride, int64_t cache_seq_stride, int capacity,
                       const void *k_new, const void *v_new, int64_t new_rs, const int32_t *pos,
                       int n_new, int batch, int n_kv_heads, int head_dim, int ring,
                       int32_t *status, void *stream) {
    if (dt != LAT_F32 && dt != LAT_BF16) return LAT_ERR_INVALID_ARG;
    if (batch < 0 || n_new < 0 || capacity < 0 || n_kv_heads <= 0) return LAT_ERR_INVALID_ARG;
    if (ring > 0 && n_new > ring) return LAT_ERR_INVALID_ARG;  // rows would overwrite each other
    if (!supported_head_dim(head_dim)) return LAT_ERR_UNSUPPORTED;
    if (batch == 0 || n_new == 0) return LAT_OK;
    if (!k_cache || !v_cache || !k_new || !v_new || !pos) return LAT_ERR_INVALID_ARG;
    if (cache_rs <= 0 || cache_head_stride <= 0 || cache_seq_stride <= 0 ||
        new_rs < (int64_t)n_kv_heads * head_dim)
        return LAT_ERR_INVALID_ARG;
    lat::AppendArgs a{};
    a.k_cache = static_cast<char *>(k_cache);
    a.v_cache = static_cast<char *>(v_cache);
    a.k_new = static_cast<const char *>(k_new);
    a.v_new = static_cast<const char *>(v_new);
    a.cache_rs = cache_rs;
    a.cache_head = cache_head_stride;
    a.cache_seq = cache_seq_stride;
    a.new_rs = new_rs;
    a.pos = pos;
    a.capacity = capacity;
    a.n_new = n_new;
    a.batch = batch;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.elem_bytes = dt == LAT_F32 ? 4 : 2;
    a.ring = ring;
    a.status = status;
    return lat::launch_kv_append(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? LAT_OK
               : LAT_ERR_CUDA;
}

}  // namespace

extern "C" {

lat_status lat_kv_append(lat_dtype dt, void *k_cache, void *v_cache, int64_t cache_rs,
                         int64_t cache_head_stride, int64_t cache_seq_stride, int capacity,
                         const void *k_new, const void *v_new, int64_t new_rs,
                         const int32_t *pos, int n_new, int batch, int n_kv_heads,
                         int head_dim, int32_t *status, void *stream) {
    return append_impl(dt, k_cache, v_cache, cache_rs, cache_head_stride, cache_seq_stride,
                       capacity, k_new, v_new, new_rs, pos, n_new, batch, n_kv_heads, head_dim,
                       0, status, stream);
}

lat_status lat_qkv_norm_rope_append(lat_dtype dt, const void *qkv, int64_t qkv_rs,
                                    const void *q_norm_w, const void *k_norm_w, float eps,
                                    double rope_base, int v_unit_norm, void *q_out,
                                    int64_t q_out_rs, void *k_cache, void *v_cache,
                                    int64_t cache_rs, int64_t cache_head_stride,
                                    int64_t cache_seq_stride, int capacity, const int32_t *pos,
                                    int n_new, int batch, int n_heads, int n_kv_heads,
                                    int head_dim, int32_t *status, void *stream) {
    if (dt != LAT_F32 && dt != LAT_BF16) return LAT_ERR_INVALID_ARG;
    if (batch < 0 || n_new < 0 || capacity < 0 || n_heads <= 0 || n_kv_heads <= 0 ||
        n_heads % n_kv_heads != 0)
        return LAT_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim)) return LAT_ERR_UNSUPPORTED;
    if (!(eps >= 0.f) || !isfinite(eps) || !(rope_base > 1.0) || !isfinite(rope_base))
        return LAT_ERR_INVALID_ARG;
    if (batch == 0 || n_new == 0) return LAT_OK;
    if (!qkv || !q_out || !k_cache || !v_cache || !pos) return LAT_ERR_INVALID_ARG;
    if (qkv_rs < (int64_t)(n_heads + 2 * n_kv_heads) * head_dim ||
        q_out_rs < (int64_t)n_heads * head_dim || cache_rs <= 0 || cache_head_stride <= 0 ||
        cache_seq_stride <= 0)
        return LAT_ERR_INVALID_ARG;
    lat::ProducerArgs a{};
    a.qkv = qkv;
    a.qkv_rs = qkv_rs;
    a.q_w = q_norm_w;
    a.k_w = k_norm_w;
    a.eps = eps;
    a.v_unit_norm = v_unit_norm != 0;
    a.q_out = q_out;
    a.q_out_rs = q_out_rs;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.cache_rs = cache_rs;
    a.cache_head = cache_head_stride;
    a.cache_seq = cache_seq_stride;
    a.capacity = capacity;
    a.pos = pos;
    a.n_new = n_new;
    a.batch = batch;
    a.n_heads = n_heads;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.status = status;
    for (int i = 0; i < head_dim / 2; ++i)  // the rotation frequencies, in double
        a.inv_freq[i] = pow(rope_base, -2.0 * i / head_dim);
    return lat::launch_qkv_producer(a, dt == LAT_BF16, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? LAT_OK
               : LAT_ERR_CUDA;
}

lat_status lat_kv_append_ring(lat_dtype dt, void *k_cache, void *v_cache, int64_t cache_rs,
                              int64_t cache_head_stride, int64_t cache_seq_stride,
                              int ring_capacity, const void *k_new, const void *v_new,
                              int64_t new_rs, const int32_t *pos, int n_new, int batch,
                              int n_kv_heads, int head_dim, int32_t *status, void *stream) {
    if (ring_capacity <= 0) return LAT_ERR_INVALID_ARG;
    return append_impl(dt, k_cache, v_cache, cache_rs, cache_head_stride, cache_seq_stride,
                       ring_capacity, k_new, v_new, new_rs, pos, n_new, batch, n_kv_heads,
                       head_dim, ring_capacity, status, stream);
}

}  // extern "C"
