// decode_bf16.cu — bandwidth-bound split-KV decode over an in-place bf16 KV cache.
//
// What it computes: for each sequence b and query head h, attention of the single query
// row (at position kv_len-1) over the visible cached keys — the decode ("vector") SDPA
// step of the hf2q "Current Inference Path" page (section 3: attention at seq_len 1 over
// the KV cache right after the append) and of the hf2q target page (section 3.2,
// sdpa_vector).  The online-softmax recurrence is the one the lattice-inference DESIGN
// page's fused kernel keeps in registers ("Current Design").
//
// How (GB300 design, not the pages'):
//  * grid = (KV split, KV head x head block, sequence).  One CTA streams one contiguous
//    chunk of one sequence's keys for one KV head, and serves ALL query heads of that
//    GQA group from the same K/V bytes (up to 8 heads per head block), so each cached
//    element is read from HBM once per decode step.
//  * One producer thread streams K and V tiles with TMA (a 4-D tensor map over the
//    cache's (head-dim, head, row, sequence) strides, 128-byte swizzled 64-column
//    chunks) into a ring of stages guarded by mbarriers; the compute warps only run
//    ldmatrix + mma.  Rows past the visible range are masked in S and, on the ragged
//    last tile, zeroed in V by the warp that owns them (cache slots there may hold NaN).
//  * The contraction runs on the tensor cores with keys in the M dimension:
//      S^T[16 keys x 8 heads]   = K[16 x D] . Q^T[D x 8]        (mma m16n8k16)
//      O^T[D x 8 heads]        += V^T[D x 16 keys] . P^T[16 x 8]
//    so a GQA group of 8 heads fills the N=8 operand exactly.  P^T's fragment comes from
//    S^T's accumulator by an in-register 8x8 transpose (movmatrix).
//  * Each warp owns 16 keys of every tile and keeps its own running max/sum, refreshed
//    only when the max grows by more than 2^8 (so the O rescale is rare); the CTA's
//    warps are merged through shared memory, and the splits of one (sequence, KV head)
//    are merged by log-sum-exp by whichever CTA arrives last (an atomic ticket), so a
//    decode step is one launch.
//  * Every mbarrier wait is bounded; on expiry the CTA records LAT_ERR_TIMEOUT, drains
//    its in-flight copies and skips its output.
#include <math.h>

#include <algorithm>

#include "device_common.cuh"
#include "kernels.h"

namespace lat {

namespace {

constexpr int kHeadsPerBlock = 8;  // N of the mma: query heads served per CTA
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint64_t kTimeoutNs = 4000000000ull;

template <int D>
struct DecodeCfg {
    static constexpr int kWarps = D >= 256 ? 2 : 4;           // compute warps
    static constexpr int kThreads = 32 * (kWarps + 1);        // + one producer warp
    static constexpr int kTile = 16 * kWarps;                 // keys per pipeline stage
    static constexpr int kStages = D == 64 ? 4 : 3;
    static constexpr int kChunks = D / 8;                     // 16-byte chunks per row
    static constexpr int kCols64 = (D + 63) / 64;             // 64-column TMA chunks per row
    static constexpr int kTileBytes = kCols64 * kTile * 128;  // one K (or V) tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kQRowChunks = (kChunks + 7) / 8 * 8; // Q rows padded for the swizzle
    static constexpr int kQRowBytes = kQRowChunks * 16;
    static constexpr int kQBytes = kHeadsPerBlock * kQRowBytes;
    static constexpr int kBarBytes = 128;
    static constexpr int kSmem = 1024 /*align slack*/ + kStages * kStageBytes + kQBytes + kBarBytes;
    // merge scratch (aliases the stage ring after the main loop)
    static constexpr int kMergeBytes = kWarps * (kHeadsPerBlock * D + 2 * kHeadsPerBlock) * 4;
    static_assert(kMergeBytes <= kStages * kStageBytes, "merge scratch must fit the ring");
    static_assert(kSmem <= 232448, "shared memory budget");
};

// byte offset of 16-byte chunk c of row r in a tile stored as 64-column, 128-byte
// swizzled regions of `rows` rows each (the TMA SWIZZLE_128B layout)
__device__ __forceinline__ uint32_t tile_off(int r, int c, int rows) {
    return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}
// byte offset of 16-byte chunk c of Q row r (rows padded to a multiple of 8 chunks)
__device__ __forceinline__ uint32_t q_off(int r, int c, int row_bytes) {
    return (uint32_t)(r * row_bytes + ((c ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(DecodeCfg<D>::kThreads)
decode_bf16_kernel(const __grid_constant__ DecodeArgs a) {
    using C = DecodeCfg<D>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *sRing = smem;                                   // [stage][K tile | V tile]
    unsigned char *sQ = smem + C::kStages * C::kStageBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(sQ + C::kQBytes);  // [kStages]
    uint64_t *empty = full + C::kStages;                           // [kStages]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + C::kStages);
    int *s_last = const_cast<int *>(abort_flag + 1);

    const int split = blockIdx.x;
    const int HB = (a.n_heads / a.n_kv_heads + kHeadsPerBlock - 1) / kHeadsPerBlock;
    const int hk = blockIdx.y / HB, hb = blockIdx.y % HB;
    const int b = blockIdx.z;
    const int G = a.n_heads / a.n_kv_heads;
    const int g_base = hb * kHeadsPerBlock;
    const int g_cnt = min(kHeadsPerBlock, G - g_base);
    const int h0 = hk * G + g_base;  // first query head of this block
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const int kv_len = a.kv_lens[b];
    if (kv_len < 0 || kv_len > a.max_kv_len) {
        if (split == 0 && hk == 0 && hb == 0 && tid == 0) report_status(a.status, kErrBounds);
        return;
    }
    const int lo = a.window > 0 ? max(0, kv_len - a.window) : 0;  // keys lo .. kv_len-1
    const int n_keys = kv_len - lo;
    const int n_splits = (n_keys + a.chunk - 1) / a.chunk;
    if (n_keys == 0) {  // nothing visible: out = 0, lse = -inf
        if (split == 0) {
            for (int i = tid; i < g_cnt * D; i += blockDim.x)
                a.out[(int64_t)b * a.out_rs + (int64_t)(h0 + i / D) * D + i % D] =
                    __float2bfloat16_rn(0.f);
            if (a.lse != nullptr && tid < g_cnt) a.lse[(int64_t)b * a.n_heads + h0 + tid] = -INFINITY;
        }
        return;
    }
    if (split >= n_splits) return;
    const int kb = lo + split * a.chunk;
    const int ke = min(kv_len, kb + a.chunk);
    const int n_tiles = (ke - kb + C::kTile - 1) / C::kTile;
    const uint64_t deadline = globaltimer_ns() + kTimeoutNs;

    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::kWarps);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    // Q rows of this head block (rows >= g_cnt are zero); the producer warp helps
    for (int i = tid; i < kHeadsPerBlock * C::kQRowChunks; i += C::kThreads) {
        const int g = i / C::kQRowChunks, c = i % C::kQRowChunks;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (g < g_cnt && c < C::kChunks)
            v = *reinterpret_cast<const uint4 *>(a.q + (int64_t)b * a.q_rs + (int64_t)(h0 + g) * D + c * 8);
        *reinterpret_cast<uint4 *>(sQ + q_off(g, c, C::kQRowBytes)) = v;
    }
    __syncthreads();

    // per-thread state: this thread's two head columns g0 = 2*(lane%4), g0+1
    float m_ref[2] = {-INFINITY, -INFINITY};  // reference maxima (log2 domain, scaled)
    float l_run[2] = {0.f, 0.f};
    float acc[D / 16][4];
#pragma unroll
    for (int i = 0; i < D / 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

    if (warp == C::kWarps) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&a.tm_k);
            tma_prefetch_desc(&a.tm_v);
            int last_issued[C::kStages];
            for (int s = 0; s < C::kStages; ++s) last_issued[s] = -1;
            for (int t = 0; t < n_tiles; ++t) {
                const int s = t % C::kStages;
                if (!mbar_wait_bounded(&empty[s], ((t / C::kStages) & 1) ^ 1, abort_flag, deadline))
                    break;
                mbar_arrive_expect_tx(&full[s], C::kStageBytes);
                unsigned char *dk = sRing + s * C::kStageBytes;
                unsigned char *dv = dk + C::kTileBytes;
                const int key0 = kb + t * C::kTile;
#pragma unroll
                for (int c = 0; c < C::kCols64; ++c) {
                    tma_load_4d(dk + c * C::kTile * 128, &a.tm_k, &full[s], c * 64, hk, key0, b);
                    tma_load_4d(dv + c * C::kTile * 128, &a.tm_v, &full[s], c * 64, hk, key0, b);
                }
                last_issued[s] = t;
            }
            // drain: every issued copy must land before the ring is reused or the CTA exits
            const uint64_t drain_deadline = globaltimer_ns() + 100000000ull;
            volatile int no_abort = 0;
            for (int s = 0; s < C::kStages; ++s)
                if (last_issued[s] >= 0)
                    mbar_wait_bounded(&full[s], (last_issued[s] / C::kStages) & 1, &no_abort,
                                      drain_deadline);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ compute warps
        const int row0 = warp * 16;
        for (int t = 0; t < n_tiles; ++t) {
            const int s = t % C::kStages;
            const bool got = mbar_wait_bounded(&full[s], (t / C::kStages) & 1, abort_flag, deadline);
            if (!__all_sync(0xffffffffu, got)) break;
            unsigned char *tk = sRing + s * C::kStageBytes;
            unsigned char *tv = tk + C::kTileBytes;
            const int key0 = kb + t * C::kTile;
            // this warp's rows past the chunk end: zero their V (their K is masked below)
            const int valid_rows = ke - (key0 + row0);
            if (valid_rows < 16) {
                for (int i = lane; i < 16 * C::kChunks; i += 32) {
                    const int r = i / C::kChunks, c = i % C::kChunks;
                    if (r >= valid_rows)
                        *reinterpret_cast<uint4 *>(tv + tile_off(row0 + r, c, C::kTile)) =
                            make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }

            // S^T = K . Q^T for this warp's 16 keys
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < D / 16; ks += 2) {
                uint32_t qf[4];  // b0,b1 for k-step ks and ks+1
                {
                    const int r = lane & 7, c = 2 * ks + (lane >> 3);
                    ldmatrix_x4(qf, sQ + q_off(r, c < C::kChunks ? c : 0, C::kQRowBytes));
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (ks + u < D / 16) {
                        uint32_t af[4];
                        const int r = row0 + (lane & 7) + 8 * ((lane >> 3) & 1);
                        const int c = 2 * (ks + u) + (lane >> 4);
                        ldmatrix_x4(af, tk + tile_off(r, c, C::kTile));
                        mma_bf16_16816(sc, af, qf[2 * u], qf[2 * u + 1]);
                    }
                }
            }
            // scale into the log2 domain and mask keys past the chunk
            const int key_a = key0 + row0 + (lane >> 2);
            const bool va = key_a < ke, vb = key_a + 8 < ke;
            sc[0] = va ? sc[0] * a.scale_log2 : -INFINITY;
            sc[1] = va ? sc[1] * a.scale_log2 : -INFINITY;
            sc[2] = vb ? sc[2] * a.scale_log2 : -INFINITY;
            sc[3] = vb ? sc[3] * a.scale_log2 : -INFINITY;

            float p[4];
            bool refresh_any = false;
            float corr[2];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float tmax = fmaxf(sc[c], sc[c + 2]);
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
                // refresh the reference only when the max grew by more than the threshold
                const bool refresh = tmax > m_ref[c] + kRescaleThreshold;
                const float m_new = refresh ? tmax : m_ref[c];
                const float m_use = m_new == -INFINITY ? 0.f : m_new;  // no key seen yet
                corr[c] = refresh ? fast_exp2(m_ref[c] - m_use) : 1.f;
                p[c] = fast_exp2(sc[c] - m_use);
                p[c + 2] = fast_exp2(sc[c + 2] - m_use);
                l_run[c] = l_run[c] * corr[c] + p[c] + p[c + 2];
                m_ref[c] = m_new;
                refresh_any |= refresh;
            }
            if (__any_sync(0xffffffffu, refresh_any)) {
#pragma unroll
                for (int i = 0; i < D / 16; ++i) {
                    acc[i][0] *= corr[0];
                    acc[i][1] *= corr[1];
                    acc[i][2] *= corr[0];
                    acc[i][3] *= corr[1];
                }
            }
            // P^T fragments: transpose the two 8x8 (key x head) quadrants
            const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p[0], p[1]));
            const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p[2], p[3]));
            // O^T += V^T . P^T
#pragma unroll
            for (int i = 0; i < D / 16; ++i) {
                uint32_t vf[4];
                const int r = row0 + (lane & 7) + 8 * (lane >> 4);
                const int c = 2 * i + ((lane >> 3) & 1);
                ldmatrix_x4_trans(vf, tv + tile_off(r, c, C::kTile));
                mma_bf16_16816(acc[i], vf, pb0, pb1);
            }
            // release the stage; zeroed rows (generic writes) must precede the next TMA
            if (valid_rows < 16) fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }
    __syncthreads();  // the ring is free from here on: reuse it as merge scratch
    if (*abort_flag) {
        if (tid == 0) report_status(a.status, kErrTimeout);
        return;
    }

    // ---- merge the warps of this CTA ---------------------------------------------
    float *w_o = reinterpret_cast<float *>(sRing);                // [warp][g][D]
    float *w_m = w_o + C::kWarps * kHeadsPerBlock * D;            // [warp][g]
    float *w_l = w_m + C::kWarps * kHeadsPerBlock;                // [warp][g]
    if (warp < C::kWarps) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            l_run[c] += __shfl_xor_sync(0xffffffffu, l_run[c], 4);
            l_run[c] += __shfl_xor_sync(0xffffffffu, l_run[c], 8);
            l_run[c] += __shfl_xor_sync(0xffffffffu, l_run[c], 16);
        }
        const int g0 = 2 * (lane & 3);
        float *wo = w_o + warp * kHeadsPerBlock * D;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
            const int d = 16 * i + (lane >> 2);
            wo[g0 * D + d] = acc[i][0];
            wo[(g0 + 1) * D + d] = acc[i][1];
            wo[g0 * D + d + 8] = acc[i][2];
            wo[(g0 + 1) * D + d + 8] = acc[i][3];
        }
        if (lane < 4) {
            w_m[warp * kHeadsPerBlock + g0] = m_ref[0];
            w_m[warp * kHeadsPerBlock + g0 + 1] = m_ref[1];
            w_l[warp * kHeadsPerBlock + g0] = l_run[0];
            w_l[warp * kHeadsPerBlock + g0 + 1] = l_run[1];
        }
    }
    __syncthreads();

    const bool single = n_splits == 1;
    for (int i = tid; i < g_cnt * D; i += C::kThreads) {
        const int g = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::kWarps; ++w) M = fmaxf(M, w_m[w * kHeadsPerBlock + g]);
        const float Mu = M == -INFINITY ? 0.f : M;
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < C::kWarps; ++w) {
            const float f = fast_exp2(w_m[w * kHeadsPerBlock + g] - Mu);
            L += w_l[w * kHeadsPerBlock + g] * f;
            O += w_o[(w * kHeadsPerBlock + g) * D + d] * f;
        }
        const int h = h0 + g;
        const float o = O / L;
        const float lse2 = Mu + log2f(L);  // log2-domain log-sum-exp of this chunk
        if (single) {
            a.out[(int64_t)b * a.out_rs + (int64_t)h * D + d] = __float2bfloat16_rn(o);
            if (d == 0 && a.lse != nullptr) a.lse[(int64_t)b * a.n_heads + h] = lse2 * 0.69314718055994531f;
        } else {
            const int64_t row = ((int64_t)b * a.n_heads + h) * a.max_splits + split;
            a.part_o[row * D + d] = o;
            if (d == 0) a.part_lse[row] = lse2;
        }
    }
    if (single) return;

    // ---- the last CTA of this (sequence, KV head, head block) merges the splits ------
    __threadfence();
    __syncthreads();
    int32_t *counter = a.counters + ((int64_t)b * a.n_kv_heads + hk) * HB + hb;
    if (tid == 0) *s_last = (atomicAdd(counter, 1) == n_splits - 1);
    __syncthreads();
    if (!*s_last) return;
    __threadfence();

    float *wt = reinterpret_cast<float *>(sRing);         // [g][n_splits] weights
    float *tot = wt + kHeadsPerBlock * n_splits;          // [g] merged log2-lse
    for (int g = warp; g < g_cnt; g += C::kWarps + 1) {
        const int64_t rb = ((int64_t)b * a.n_heads + h0 + g) * a.max_splits;
        float M = -INFINITY;
        for (int sp = lane; sp < n_splits; sp += 32) M = fmaxf(M, __ldcg(a.part_lse + rb + sp));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float Z = 0.f;
        for (int sp = lane; sp < n_splits; sp += 32) {
            const float e = fast_exp2(__ldcg(a.part_lse + rb + sp) - M);
            wt[g * n_splits + sp] = e;
            Z += e;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, off);
        const float inv = 1.f / Z;
        for (int sp = lane; sp < n_splits; sp += 32) wt[g * n_splits + sp] *= inv;
        if (lane == 0) tot[g] = M + log2f(Z);
    }
    __syncthreads();
    for (int i = tid; i < g_cnt * D; i += C::kThreads) {
        const int g = i / D, d = i % D;
        const int64_t rb = ((int64_t)b * a.n_heads + h0 + g) * a.max_splits;
        float o = 0.f;
        for (int sp = 0; sp < n_splits; ++sp)
            o += wt[g * n_splits + sp] * __ldcg(a.part_o + (rb + sp) * D + d);
        a.out[(int64_t)b * a.out_rs + (int64_t)(h0 + g) * D + d] = __float2bfloat16_rn(o);
        if (d == 0 && a.lse != nullptr)
            a.lse[(int64_t)b * a.n_heads + h0 + g] = tot[g] * 0.69314718055994531f;
    }
    if (tid == 0) *counter = 0;  // ready for the next call
}

template <int D>
cudaError_t launch_decode_d(const DecodeArgs &a, cudaStream_t s) {
    using C = DecodeCfg<D>;
    cudaError_t e = cudaFuncSetAttribute(decode_bf16_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    const int HB = (a.n_heads / a.n_kv_heads + kHeadsPerBlock - 1) / kHeadsPerBlock;
    const int range = a.window > 0 ? min(a.max_kv_len, a.window) : a.max_kv_len;
    const int grid_splits = max(1, (range + a.chunk - 1) / a.chunk);
    dim3 grid(grid_splits, a.n_kv_heads * HB, a.batch);
    decode_bf16_kernel<D><<<grid, C::kThreads, C::kSmem, s>>>(a);
    return cudaGetLastError();
}

template <int D>
int tile_keys() { return DecodeCfg<D>::kTile; }
template <int D>
int ctas_per_sm() { return (228 * 1024) / (DecodeCfg<D>::kSmem + 1024); }

}  // namespace

int decode_bf16_tile_keys(int head_dim) {
    switch (head_dim) {
        case 64: return tile_keys<64>();
        case 80: return tile_keys<80>();
        case 128: return tile_keys<128>();
        case 256: return tile_keys<256>();
        case 512: return tile_keys<512>();
        default: return 0;
    }
}

bool plan_decode_bf16(int batch, int n_heads, int n_kv_heads, int head_dim, int max_kv_len,
                      int window, int num_sms, DecodePlan *p) {
    int T, occ;
    switch (head_dim) {
        case 64: T = tile_keys<64>(); occ = ctas_per_sm<64>(); break;
        case 80: T = tile_keys<80>(); occ = ctas_per_sm<80>(); break;
        case 128: T = tile_keys<128>(); occ = ctas_per_sm<128>(); break;
        case 256: T = tile_keys<256>(); occ = ctas_per_sm<256>(); break;
        case 512: T = tile_keys<512>(); occ = ctas_per_sm<512>(); break;
        default: return false;
    }
    if (occ < 1) occ = 1;
    const int G = n_heads / n_kv_heads;
    const int HB = (G + kHeadsPerBlock - 1) / kHeadsPerBlock;
    const int64_t units = (int64_t)batch * n_kv_heads * HB;
    const int range = window > 0 ? std::min(max_kv_len, window) : max_kv_len;
    // The scratch layout depends on the window-free plan only, so a workspace sized by
    // lat_attn_decode_workspace_size fits every window.
    auto splits_for = [&](int rng) {
        const int64_t target = (int64_t)num_sms * occ * 2;  // ~2 CTA waves for balance
        int64_t sp = (target + units - 1) / std::max<int64_t>(units, 1);
        sp = std::min<int64_t>(sp, (rng + T - 1) / T);
        sp = std::min<int64_t>(sp, 512);
        return (int)std::max<int64_t>(sp, 1);
    };
    const int layout_splits = splits_for(std::max(max_kv_len, 1));
    const int sp = splits_for(std::max(range, 1));
    int chunk = (std::max(range, 1) + sp - 1) / sp;
    chunk = (chunk + T - 1) / T * T;
    p->head_blocks = HB;
    p->chunk = chunk;
    p->max_splits = layout_splits;
    auto round256 = [](size_t x) { return (x + 255) / 256 * 256; };
    p->part_o_bytes = round256((size_t)batch * n_heads * layout_splits * head_dim * 4);
    p->part_lse_bytes = round256((size_t)batch * n_heads * layout_splits * 4);
    p->counter_bytes = round256((size_t)units * 4);
    p->total_bytes = p->part_o_bytes + p->part_lse_bytes + p->counter_bytes;
    return true;
}

cudaError_t launch_decode_bf16(const DecodeArgs &a, cudaStream_t s) {
    switch (a.head_dim) {
        case 64: return launch_decode_d<64>(a, s);
        case 80: return launch_decode_d<80>(a, s);
        case 128: return launch_decode_d<128>(a, s);
        case 256: return launch_decode_d<256>(a, s);
        case 512: return launch_decode_d<512>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lat
