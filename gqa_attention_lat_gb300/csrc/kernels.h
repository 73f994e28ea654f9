// kernels.h — internal launch interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Host-only declarations; every argument has been validated by the
// caller before a launcher runs.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lat {

// ---------------------------------------------------------------- KV-cache append
struct AppendArgs {
    char *k_cache, *v_cache;          // byte pointers
    const char *k_new, *v_new;
    int64_t cache_rs, cache_head, cache_seq, new_rs;  // element strides
    const int32_t *pos;
    int capacity, n_new, batch, n_kv_heads, head_dim, elem_bytes;
    int ring;                         // > 0: position p lives in slot p % ring (no bounds)
    int32_t *status;
};
cudaError_t launch_kv_append(const AppendArgs &a, cudaStream_t s);

// ---------------------------------------------------------------- attention-input producer
// Q/K RMS norm + neox RoPE + V (copy or unit norm) + cache append, one CTA per new row.
struct ProducerArgs {
    const void *qkv;                 // [batch * n_new rows, qkv_rs]: Q heads, K heads, V heads
    int64_t qkv_rs;
    const void *q_w, *k_w;           // [head_dim] norm weights (nullable: weight 1)
    float eps;
    int v_unit_norm;
    void *q_out;                     // [batch * n_new rows, q_out_rs]
    int64_t q_out_rs;
    void *k_cache, *v_cache;
    int64_t cache_rs, cache_head, cache_seq;
    int capacity;
    const int32_t *pos;
    int n_new, batch, n_heads, n_kv_heads, head_dim;
    int32_t *status;
    double inv_freq[256];            // base^(-2i/D), i < head_dim/2, from the host in double
};
cudaError_t launch_qkv_producer(const ProducerArgs &a, bool bf16, cudaStream_t s);

// ---------------------------------------------------------------- fp32 row kernel
// One warp per (query row, query head); used for every fp32 prefill and decode.
// Element (b, j, hk, d) of K is k[b*k_seq + j*k_row + hk*k_head + d] (V alike);
// in decode mode (kv_lens != nullptr) seq_len is 1 and sequence b has kv_lens[b] keys.
struct RowAttnArgs {
    const float *q;
    int64_t q_rs;
    const float *k, *v;
    int64_t k_seq, k_row, k_head, v_seq, v_row, v_head;
    float *out;
    int64_t out_rs;
    float *lse;
    int batch, seq_len, kv_len, n_heads, n_kv_heads, head_dim, causal, window;
    float scale;
    float softcap;                 // > 0: score s becomes softcap * tanh(s / softcap)
    const int32_t *kv_lens;
    int max_kv_len;
    int ring;                      // > 0: key j sits in row j % ring of its sequence
    int32_t *status;
};
cudaError_t launch_row_attention_f32(const RowAttnArgs &a, cudaStream_t s);

// ---------------------------------------------------------------- bf16 split-KV decode
struct DecodeArgs {
    CUtensorMap tm_k, tm_v;  // 4-D maps (d, head, row < max_kv_len, sequence), 128-byte swizzle
    CUtensorMap tm_k16, tm_v16;  // the same with 16-row boxes: a sequence's partial last tile
    CUtensorMap tm_q;        // 3-D map (d, query head, sequence), 8-head boxes, 128-byte swizzle
    const __nv_bfloat16 *q;
    int64_t q_rs;
    const __nv_bfloat16 *k_cache, *v_cache;
    int64_t cache_rs, cache_head, cache_seq;
    const int32_t *kv_lens;
    int max_kv_len;
    __nv_bfloat16 *out;
    int64_t out_rs;
    float *lse;
    int batch, n_heads, n_kv_heads, head_dim, window;
    int ring;           // > 0: ring cache of `ring` rows, key j in row j % ring (window <= ring)
    float scale_log2;   // scale * log2(e): scores are exponentiated with exp2
    float cap_log2, raw_over_cap;  // score cap, as in PrefillTcArgs (cap_log2 0: none)
    // split-KV scratch: partial outputs, partial lse and arrival counters
    float *part_o;      // [batch, n_heads, max_splits, head_dim]
    float *part_lse;    // [batch, n_heads, max_splits]
    int32_t *counters;  // [batch, n_kv_heads, head_blocks]
    int max_splits;  // partial slots per (sequence, KV head, head block)
    int min_seg;     // shortest stretch of one unit's keys a CTA takes (multiple of the tile)
    // few long units: the key stream is cut across every CTA and the pieces are merged by
    // a second kernel; piece_count[b, h] (in the counters' place) tells it how many
    int defer_merge;
    int32_t *piece_count;  // [batch, n_heads] when defer_merge
    int chunked;           // tm_k/tm_v are chunked 5-D maps: one copy per K or V tile
    uint64_t timeout_ns;   // budget of every bounded wait, per CTA
    int test_skip_load;    // test hook: never load a CTA's first K/V stage (forces a timeout)
    int32_t *status;
};
struct DecodePlan {
    int head_blocks, max_splits, min_seg, grid, defer_merge;
    size_t part_o_bytes, part_lse_bytes, counter_bytes, total_bytes;
};
// Chooses the split size and the scratch layout; false when the shape is not built.
bool plan_decode_bf16(int batch, int n_heads, int n_kv_heads, int head_dim, int max_kv_len,
                      int window, int num_sms, DecodePlan *plan);
// work units of one decode launch (sequence x KV head x block of <= 8 query heads); the
// split-KV merge tickets carry a unit index in 23 bits, so plans stop below kDecodeMaxUnits
int64_t decode_bf16_units(int batch, int n_heads, int n_kv_heads);
constexpr int64_t kDecodeMaxUnits = int64_t(1) << 23;
int decode_bf16_tile_keys(int head_dim);     // cache rows per TMA box for this head_dim
cudaError_t launch_decode_bf16(const DecodeArgs &a, int grid, cudaStream_t s);

// ---------------------------------------------------------------- bf16 tensor-core prefill
struct PrefillTcArgs {
    CUtensorMap tm_q, tm_k, tm_v;  // 4-D maps (d, head, row, batch), 128-byte swizzle
    // 3-D map over the output (column, row < seq_len, batch), 32-row boxes of
    // prefill_tc_out_box_cols columns; used where that is nonzero
    CUtensorMap tm_out;
    __nv_bfloat16 *out;
    int64_t out_rs;
    int out_v8;                    // out and out_rs allow 32-byte row stores
    float *lse;
    int batch, seq_len, kv_len, n_heads, n_kv_heads, head_dim, causal, window;
    float scale_log2;              // scale * log2(e)
    // score cap: when cap_log2 > 0 a raw dot product x scores cap_log2 * tanh(x * raw_over_cap)
    // in the log2 domain (softcap * log2(e) and scale / softcap), replacing x * scale_log2
    float cap_log2, raw_over_cap;
    int32_t *status;
    uint64_t timeout_ns;
    int test_skip_kv_load;         // test hook: never load KV tile 0 (forces a timeout)
    int wide;                      // head_dim 64: the 96-key-tile form (prefill_tc_wide)
    int pair;                      // head_dim 512, even GQA group: the CTA-pair form
    int chunked;                   // tm_q/k/v are chunked 5-D maps: one copy per tile
};
// the 96-key-tile form of head_dim 64 for long key ranges (a query tile visiting ~1K keys)
bool prefill_tc_wide(int head_dim, int seq_len, int kv_len, int causal, int window);
int prefill_tc_block_n(int head_dim, bool wide);  // keys per KV tile
// head_dim 512 with an even number of query heads per KV head runs on CTA pairs
bool prefill_tc_pair(int head_dim, int n_heads, int n_kv_heads);
// rows of the K (v = false) or V (v = true) tensor-map box of the chosen form
int prefill_tc_box_rows(int head_dim, bool wide, bool pair, bool v);
// forms that move each tile in one copy through chunked 5-D maps, and the 64-column
// chunks of one V copy
bool prefill_tc_chunked(int head_dim, bool pair);
// columns of one output box where the epilogue stores through tm_out, else 0
int prefill_tc_out_box_cols(int head_dim, bool pair);
int prefill_tc_v_chunks(int head_dim, bool pair);
// work items of one prefill launch (query tile x head x output-column part); the kernel
// numbers them in int32, so the host refuses shapes above kPrefillMaxItems
int64_t prefill_tc_items(int batch, int n_heads, int head_dim, int seq_len);
constexpr int64_t kPrefillMaxItems = int64_t(1) << 30;
cudaError_t launch_prefill_tc(const PrefillTcArgs &a, int num_sms, cudaStream_t s);
// out[i] = the capped score (log2 domain) of raw[i], as the bf16 kernels form it
cudaError_t launch_capped_scores(const float *raw, int64_t n, float raw_over_cap,
                                 float cap_log2, float *out, cudaStream_t s);

}  // namespace lat
