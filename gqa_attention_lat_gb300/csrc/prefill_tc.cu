// prefill_tc.cu — bf16 grouped-query attention prefill on the 5th-generation tensor cores.
//
// What it computes: for every query row and query head, softmax(scale * q K^T) V over the
// keys the causal / sliding-window mask leaves visible, plus the row's log-sum-exp — the
// fused attention of the lattice-inference DESIGN page ("Current Design": fused attention
// with online softmax in registers; head_dim and the GQA mapping fixed per compiled
// variant) and the prefill ("full", seq_len > 1) SDPA of the hf2q pages (Current
// Inference Path, section 7; target architecture, open question Q2).
//
// How (GB300 design; the pages' Metal kernels are prior art only):
//  * One CTA owns a 128-row query tile of one head (one TMEM lane per query row).
//  * Warp roles: warps 0-3 run the softmax (thread t <-> query row t), warp 4 issues TMA
//    loads, warp 5 issues tcgen05.mma.  Synchronisation is by mbarriers only.
//  * S = Q K^T is accumulated in tensor memory (fp32, double-buffered so the MMA of tile
//    j+1 overlaps the softmax of tile j); P = exp2(S*scale*log2e - m) is written as bf16
//    to shared memory and O += P V accumulates in tensor memory.
//  * K and V reach shared memory as [BN keys x 64 head-dims] chunks with 128-byte
//    swizzle, through one ring of chunk slots that the MMA warp consumes in issue order.
//    Q and K enter the MMA K-major; V enters MN-major, one 64-column chunk per MMA.
//  * Tiles wholly outside the causal / window band are never loaded or computed; tiles
//    wholly inside it skip the per-element mask.
//  * The running maximum is refreshed only when it grows by more than 2^8 (the stale
//    maximum keeps every weight <= 256, well inside fp32/bf16 range), so the O rescale
//    in tensor memory is rare; the result is exact up to rounding because O and l always
//    share the same reference maximum.
//  * head_dim 80 runs as two chunks (64 + 16 live columns; the tensor map zero-fills
//    columns past 80).  head_dim 512 splits O across two CTAs of 256 columns each (a
//    128 x 512 fp32 accumulator alone would fill tensor memory); each recomputes S.
//  * Every mbarrier wait is bounded by a wall-clock budget; on expiry the CTA records
//    LAT_ERR_TIMEOUT, drains its in-flight copies and MMAs, frees tensor memory and exits.
#include <math.h>

#include "device_common.cuh"
#include "kernels.h"

namespace lat {

namespace {

constexpr int kBM = 128;             // query rows per CTA (= TMEM lanes)
constexpr int kThreads = 192;        // 4 softmax warps + producer warp + MMA warp
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kChunkCols = 64;       // head-dim columns per swizzled chunk (128 bytes)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;       // O accumulator columns [0, 256)
constexpr uint32_t kTmemS = 256;     // S buffers at 256 and 256 + BN
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct TcCfg {
    static constexpr int kQkChunks = (D + kChunkCols - 1) / kChunkCols;   // Q/K chunks
    static constexpr int kKSteps = (D + 15) / 16;                          // S MMA k-steps
    static constexpr int kBN = D <= 128 ? 128 : 64;                        // keys per tile
    static constexpr int kSplitO = D == 512 ? 2 : 1;                       // CTAs per O row
    static constexpr int kOCols = D / kSplitO;                             // O cols per CTA
    static constexpr int kVChunks = (kOCols + kChunkCols - 1) / kChunkCols;
    static constexpr int kSlotBytes = kBN * 128;
    static constexpr int kQBytes = kQkChunks * kBM * 128;
    static constexpr int kPChunks = kBN / 64;
    static constexpr int kPBytes = kPChunks * kBM * 128;
    static constexpr int kSlots = D == 512 ? 10 : (D == 256 ? 16 : 8);
    static constexpr int kBarBytes = 1024;
    static constexpr int kSmem = 1024 /*align slack*/ + kQBytes + kPBytes +
                                 kSlots * kSlotBytes + kBarBytes;
    static_assert(kSmem <= 232448, "shared memory budget");
    static_assert(kOCols <= 256 && kTmemS + 2 * kBN <= kTmemCols, "tensor memory budget");
};

// ---- tcgen05 descriptors ----------------------------------------------------------

// Shared-memory matrix descriptor, 128-byte swizzle.  Bits: [0,14) start address >> 4,
// [16,30) leading byte offset >> 4, [32,46) stride byte offset >> 4, [46,49) = 0b001,
// [49,52) base offset, bit 52 LBO mode, [61,64) swizzle mode (2 = 128-byte).
// Every operand tile here is one swizzle atom wide in its contiguous dimension, so the
// only stride that matters is the 1024 bytes between 8-row groups; both offset fields
// carry it.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)(1024 >> 4) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A and B
// (bits 7-9, 10-12 = 1), A K-major (bit 15 = 0), B K-major or MN-major (bit 16),
// N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct Band {  // the KV tiles one query tile must visit
    int t_begin, t_end;
};

__device__ __forceinline__ Band kv_band(int m0, int rows, int S, int L, int causal, int window,
                                        int BN) {
    const int p_min = m0 + (L - S);
    const int p_max = m0 + rows - 1 + (L - S);
    const int j_lo = window > 0 ? max(0, p_min - window + 1) : 0;
    const int j_hi = causal ? min(L, p_max + 1) : L;
    Band b;
    b.t_begin = j_lo / BN;
    b.t_end = j_hi > j_lo ? (j_hi + BN - 1) / BN : b.t_begin;
    return b;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ PrefillTcArgs a) {
    using C = TcCfg<D>;
    constexpr int BN = C::kBN;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *sQ = smem;
    unsigned char *sP = sQ + C::kQBytes;
    unsigned char *sSlots = sP + C::kPBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sSlots + C::kSlots * C::kSlotBytes);
    uint64_t *bar_q = bars + 0;
    uint64_t *bar_s = bars + 1;        // [2]
    uint64_t *bar_p = bars + 3;
    uint64_t *bar_o = bars + 4;
    uint64_t *bar_done = bars + 5;     // final MMA drain
    uint64_t *bar_full = bars + 6;     // [kSlots]
    uint64_t *bar_empty = bar_full + C::kSlots;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_empty + C::kSlots);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int head_sel = blockIdx.x;               // h * kSplitO + half
    const int h = head_sel / C::kSplitO;
    const int half = head_sel % C::kSplitO;
    const int b = blockIdx.y;
    const int n_mtiles = (a.seq_len + kBM - 1) / kBM;
    const int mt = n_mtiles - 1 - (int)blockIdx.z;  // heaviest (latest) query tiles first
    const int m0 = mt * kBM;
    const int rows = min(kBM, a.seq_len - m0);
    const int hk = h / (a.n_heads / a.n_kv_heads);
    const int v_col0 = half * C::kOCols;
    const Band band = kv_band(m0, rows, a.seq_len, a.kv_len, a.causal, a.window, BN);
    const int n_tiles = band.t_end - band.t_begin;
    const uint64_t deadline = globaltimer_ns() + a.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        mbar_init(&bar_s[0], 1);
        mbar_init(&bar_s[1], 1);
        mbar_init(bar_p, 128);
        mbar_init(bar_o, 1);
        mbar_init(bar_done, 1);
        for (int s = 0; s < C::kSlots; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], 1);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == kMmaWarp) {  // whole warp: allocate tensor memory
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&a.tm_q);
            tma_prefetch_desc(&a.tm_k);
            tma_prefetch_desc(&a.tm_v);
            mbar_arrive_expect_tx(bar_q, C::kQBytes);
            for (int c = 0; c < C::kQkChunks; ++c)
                tma_load_4d(sQ + c * kBM * 128, &a.tm_q, bar_q, c * kChunkCols, h, m0, b);
            int issued[C::kSlots];
            for (int s = 0; s < C::kSlots; ++s) issued[s] = 0;
            int r = 0;
            bool ok = true;
            auto push = [&](const CUtensorMap *tm, int col, int key0) {
                const int s = r % C::kSlots;
                if (!mbar_wait_bounded(&bar_empty[s], ((r / C::kSlots) & 1) ^ 1, abort_flag,
                                       deadline)) {
                    ok = false;
                    return;
                }
                mbar_arrive_expect_tx(&bar_full[s], C::kSlotBytes);
                tma_load_4d(sSlots + s * C::kSlotBytes, tm, &bar_full[s], col, hk, key0, b);
                ++issued[s];
                ++r;
            };
            for (int t = 0; t <= n_tiles && ok; ++t) {
                if (t < n_tiles) {
                    const int key0 = (band.t_begin + t) * BN;
                    for (int c = 0; c < C::kQkChunks && ok; ++c) {
                        if (a.test_skip_kv_load && t == 0 && c == 0) {  // test hook
                            ++r;
                            continue;
                        }
                        push(&a.tm_k, c * kChunkCols, key0);
                    }
                }
                if (t > 0) {
                    const int key0 = (band.t_begin + t - 1) * BN;
                    for (int c = 0; c < C::kVChunks && ok; ++c)
                        push(&a.tm_v, v_col0 + c * kChunkCols, key0);
                }
            }
            // drain: every issued copy must land before the CTA may exit
            const uint64_t drain_deadline = globaltimer_ns() + 100000000ull;
            volatile int no_abort = 0;
            mbar_wait_bounded(bar_q, 0, &no_abort, drain_deadline);
            for (int s = 0; s < C::kSlots; ++s)
                if (issued[s] > 0)
                    mbar_wait_bounded(&bar_full[s], (issued[s] - 1) & 1, &no_abort,
                                      drain_deadline);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = instr_desc(kBM, BN, false);
            const uint32_t q_base = smem_u32(sQ);
            const uint32_t p_base = smem_u32(sP);
            const uint32_t slot_base = smem_u32(sSlots);
            bool ok = mbar_wait_bounded(bar_q, 0, abort_flag, deadline);
            int r = 0;
            tc_fence_after();
            auto take = [&](int &s) {
                s = r % C::kSlots;
                if (!mbar_wait_bounded(&bar_full[s], (r / C::kSlots) & 1, abort_flag, deadline))
                    return false;
                tc_fence_after();
                return true;
            };
            for (int t = 0; t <= n_tiles && ok; ++t) {
                if (t < n_tiles) {
                    // S(t) = Q K(t)^T into S buffer t % 2
                    const uint32_t d_s = tmem + kTmemS + (uint32_t)((t & 1) * BN);
                    for (int c = 0; c < C::kQkChunks && ok; ++c) {
                        int s;
                        if (!take(s)) { ok = false; break; }
                        const uint32_t k_addr = slot_base + s * C::kSlotBytes;
                        const uint32_t q_addr = q_base + c * kBM * 128;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            if (c * 4 + kk < C::kKSteps)
                                tc_mma_ss(d_s, sw128_desc(q_addr + kk * 32),
                                          sw128_desc(k_addr + kk * 32), idesc_s,
                                          (c > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc_commit(&bar_empty[s]);
                        ++r;
                    }
                    if (!ok) break;
                    tc_commit(&bar_s[t & 1]);
                }
                if (t > 0) {
                    // O += P(t-1) V(t-1), one 64-column chunk of V at a time
                    const int tp = t - 1;
                    if (!mbar_wait_bounded(bar_p, tp & 1, abort_flag, deadline)) { ok = false; break; }
                    tc_fence_after();
                    for (int c = 0; c < C::kVChunks && ok; ++c) {
                        int s;
                        if (!take(s)) { ok = false; break; }
                        const uint32_t v_addr = slot_base + s * C::kSlotBytes;
                        const int ncols = min(kChunkCols, C::kOCols - c * kChunkCols);
                        const uint32_t idesc_pv = instr_desc(kBM, ncols, true);
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk) {
                            // A = P, K-major: keys 16kk..16kk+15 live in chunk kk/4 at +32B*(kk%4)
                            const uint32_t a_addr = p_base + (kk >> 2) * kBM * 128 + (kk & 3) * 32;
                            // B = V, MN-major: 16 keys = two 8-row groups = 2048 bytes
                            const uint32_t b_addr = v_addr + kk * 2048;
                            tc_mma_ss(tmem + kTmemO + c * kChunkCols, sw128_desc(a_addr),
                                      sw128_desc(b_addr), idesc_pv, (tp > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc_commit(&bar_empty[s]);
                        ++r;
                    }
                    if (!ok) break;
                    tc_commit(bar_o);
                }
            }
            // drain: all issued MMAs must finish before tensor memory is freed
            tc_commit(bar_done);
            volatile int no_abort = 0;
            mbar_wait_bounded(bar_done, 0, &no_abort, globaltimer_ns() + 100000000ull);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax warps
        const int row = threadIdx.x;                  // 0..127, TMEM lane
        const int i = m0 + row;                       // query row within the sequence
        const int p = i + (a.kv_len - a.seq_len);     // its absolute position
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        float m_ref = -INFINITY;  // reference maximum (log2 domain, scaled)
        float l_sum = 0.f;
        bool ok = true;
        // tcgen05.ld/st are warp-collective, so a wait's outcome is made warp-uniform
        auto wait_warp = [&](uint64_t *bar, uint32_t parity) {
            const bool r = mbar_wait_bounded(bar, parity, abort_flag, deadline);
            return __all_sync(0xffffffffu, r) != 0;
        };
        for (int t = 0; t < n_tiles; ++t) {
            if (!wait_warp(&bar_s[t & 1], (t >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            float sv[BN];
#pragma unroll
            for (int c = 0; c < BN; c += 16)
                tmem_ld16(lane_base + kTmemS + (t & 1) * BN + c, reinterpret_cast<uint32_t *>(sv + c));
            tc_wait_ld();

            const int key0 = (band.t_begin + t) * BN;
            const bool need_mask = (key0 + BN > a.kv_len) ||
                                   (a.causal && key0 + BN - 1 > m0 + (a.kv_len - a.seq_len)) ||
                                   (a.window > 0 && key0 < m0 + rows - 1 + (a.kv_len - a.seq_len) - a.window + 1);
            float mx = -INFINITY;
            if (need_mask) {
#pragma unroll
                for (int c = 0; c < BN; ++c) {
                    const int j = key0 + c;
                    const bool vis = j < a.kv_len && (!a.causal || j <= p) &&
                                     (a.window <= 0 || p - j < a.window);
                    sv[c] = vis ? sv[c] * a.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, sv[c]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < BN; ++c) {
                    sv[c] *= a.scale_log2;
                    mx = fmaxf(mx, sv[c]);
                }
            }
            // refresh the reference maximum only when it grew by more than the threshold
            const bool refresh = mx > m_ref + kRescaleThreshold;
            const float m_new = refresh ? mx : m_ref;
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            float rowsum = 0.f;
#pragma unroll
            for (int c = 0; c < BN; ++c) {
                sv[c] = fast_exp2(sv[c] - m_use);
                rowsum += sv[c];
            }
            const float corr = refresh ? fast_exp2(m_ref - m_use) : 1.f;  // 0 when m_ref = -inf

            // P and O are free once P(t-1) V(t-1) has completed
            if (t > 0) {
                if (!wait_warp(bar_o, (t - 1) & 1)) { ok = false; break; }
                tc_fence_after();
            }
            // P (bf16) into shared memory, K-major with 128-byte swizzle: row `row`,
            // keys 8u..8u+7 of chunk c at 16-byte unit u ^ (row & 7)
#pragma unroll
            for (int c = 0; c < C::kPChunks; ++c) {
                unsigned char *prow = sP + c * kBM * 128 + row * 128;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float *x = sv + c * 64 + u * 8;
                    uint4 pk;
                    pk.x = pack_bf16x2(x[0], x[1]);
                    pk.y = pack_bf16x2(x[2], x[3]);
                    pk.z = pack_bf16x2(x[4], x[5]);
                    pk.w = pack_bf16x2(x[6], x[7]);
                    *reinterpret_cast<uint4 *>(prow + ((u ^ (row & 7)) << 4)) = pk;
                }
            }
            // rescale O in tensor memory when any row of this warp refreshed its maximum
            if (t > 0 && __any_sync(0xffffffffu, refresh)) {
#pragma unroll 1
                for (int c = 0; c < C::kOCols; c += 16) {
                    uint32_t ov[16];
                    tmem_ld16(lane_base + kTmemO + c, ov);
                    tc_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        ov[e] = __float_as_uint(__uint_as_float(ov[e]) * corr);
                    tmem_st16(lane_base + kTmemO + c, ov);
                }
                tc_wait_st();
            }
            l_sum = l_sum * corr + rowsum;
            m_ref = m_new;
            fence_proxy_async_smem();  // P writes -> visible to the tensor core
            tc_fence_before();
            mbar_arrive(bar_p);
        }
        // ---- epilogue: O / l -> bf16 rows, lse -----------------------------------
        if (ok && n_tiles > 0) {
            ok = wait_warp(bar_o, (n_tiles - 1) & 1);
            tc_fence_after();
        }
        if (ok) {
            const bool live = row < rows;  // rows past the sequence end are not stored
            const int64_t qrow = (int64_t)b * a.seq_len + i;
            __nv_bfloat16 *orow = a.out + qrow * a.out_rs + (int64_t)h * D + v_col0;
            const bool empty = !(l_sum > 0.f);
            const float inv_l = empty ? 0.f : 1.f / l_sum;
            if (n_tiles > 0) {
#pragma unroll 1
                for (int c = 0; c < C::kOCols; c += 16) {
                    uint32_t ov[16];
                    tmem_ld16(lane_base + kTmemO + c, ov);  // warp-wide: every lane takes part
                    tc_wait_ld();
                    uint32_t pk[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv_l,
                                            __uint_as_float(ov[2 * e + 1]) * inv_l);
                    if (live) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + c);
                        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                }
            } else if (live) {
                for (int c = 0; c < C::kOCols; ++c) orow[c] = __float2bfloat16_rn(0.f);
            }
            if (live && a.lse != nullptr && half == 0)
                a.lse[qrow * a.n_heads + h] =
                    empty ? -INFINITY : (m_ref + log2f(l_sum)) * 0.69314718055994531f;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) report_status(a.status, kErrTimeout);
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D>
cudaError_t launch_d(const PrefillTcArgs &a, cudaStream_t s) {
    using C = TcCfg<D>;
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    const int n_mtiles = (a.seq_len + kBM - 1) / kBM;
    dim3 grid(a.n_heads * C::kSplitO, a.batch, n_mtiles);
    prefill_tc_kernel<D><<<grid, kThreads, C::kSmem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

int prefill_tc_block_n(int head_dim) {
    switch (head_dim) {
        case 64: return TcCfg<64>::kBN;
        case 80: return TcCfg<80>::kBN;
        case 128: return TcCfg<128>::kBN;
        case 256: return TcCfg<256>::kBN;
        case 512: return TcCfg<512>::kBN;
        default: return 0;
    }
}

cudaError_t launch_prefill_tc(const PrefillTcArgs &a, cudaStream_t s) {
    if (a.seq_len == 0 || a.batch == 0) return cudaSuccess;
    switch (a.head_dim) {
        case 64: return launch_d<64>(a, s);
        case 80: return launch_d<80>(a, s);
        case 128: return launch_d<128>(a, s);
        case 256: return launch_d<256>(a, s);
        case 512: return launch_d<512>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lat
