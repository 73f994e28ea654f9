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
//  * Work unit = one (sequence, KV head, head block of <= 8 query heads): all query
//    heads of a GQA group are served from the same K/V bytes, so each cached element is
//    read from HBM once per decode step.
//  * Persistent, statically balanced ("stream-K") schedule: the visible keys of all
//    units, laid end to end, form one key stream; CTA c takes the c-th equal share of it
//    (never less than a minimum stretch), which may cut units at both ends.  A CTA
//    streams its share without draining its pipeline between units; a unit cut across
//    CTAs leaves one partial (normalised output and log-sum-exp) per piece, merged by
//    the CTA that finishes the unit's last piece (an atomic ticket), after its stream.
//    With few units (one long sequence, say) the stream is cut across every CTA and a
//    second kernel, launched as a programmatic dependent, merges the pieces instead.
//  * One producer thread streams K and V tiles with TMA (tensor maps over the cache's
//    (head-dim, head, row, sequence) strides, 128-byte swizzled 64-column chunks: one
//    copy per K or V tile where head_dim is 64-256, a copy per chunk at 512, and a part's
//    partial last tile in 16-row boxes) into a ring of stages, each tagged with a record
//    of what it holds; each unit's query rows arrive by TMA into a double buffer.  Rows
//    past a piece's end are masked in S and zeroed in V by the warp that owns them
//    (cache slots there may hold NaN).
//  * The contraction runs on the tensor cores with keys in the M dimension:
//      S^T[16 keys x 8 heads]   = K[16 x D] . Q^T[D x 8]        (mma m16n8k16)
//      O^T[D x 8 heads]        += V^T[D x 16 keys] . P^T[16 x 8]
//    so a GQA group of 8 heads fills the N=8 operand exactly; P^T's fragment comes from
//    S^T's accumulator by an in-register 8x8 transpose (movmatrix).
//  * Each warp owns 16 keys of every tile and keeps its own running max/sum, refreshed
//    only when the max grows by more than 2^8 (so the O rescale is rare); at the end of
//    a piece the warps park their states in shared memory and each combines a share of
//    the heads from all of them and writes it out.
//  * Every wait is bounded (the budget comes with the launch); on expiry the CTA records
//    LAT_ERR_TIMEOUT, drains its copies and quits.
#include <math.h>

#include <algorithm>

#include "device_common.cuh"
#include "kernels.h"

namespace lat {

namespace {

constexpr int kHeadsPerBlock = 8;          // N of the mma: query heads served per unit
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kMaxMerges = 2;              // multi-piece units a CTA can finish last
constexpr float kLn2 = 0.69314718055994531f;

template <int D>
struct DecodeCfg {
    static constexpr int kWarps = D >= 256 ? 2 : 4;           // compute warps
    static constexpr int kThreads = 32 * (kWarps + 1);        // + one producer warp
    static constexpr int kTile = 16 * kWarps;                 // keys per pipeline stage
    // Two stages up to head_dim 256: as fast as three on the ragged 32-sequence decode at
    // head_dim 128 and on the ring decode at 256, and faster where every CTA's first stages
    // dominate (one long sequence at 128: 4 %; B32 H16/8 up to 4096 keys: 4.5 % at head_dim
    // 64 against four stages, 2.7 % at 256): requested all at once, fewer land sooner.
    // head_dim 512 (one CTA per SM) needs its three 64 KB stages (two: 3 % slower).
    static constexpr int kStages = D == 512 ? 3 : 2;
    static constexpr int kMinBlocks = D == 512 ? 1 : (D == 64 ? 3 : 2);  // CTAs per SM
    static constexpr int kChunks = D / 8;                     // 16-byte chunks per row
    static constexpr int kCols64 = (D + 63) / 64;             // 64-column TMA chunks per row
    static constexpr int kTileBytes = kCols64 * kTile * 128;  // one K (or V) tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kQBytes = kCols64 * kHeadsPerBlock * 128;   // 8 query rows
    static constexpr int kMiscBytes = 640;                           // records, barriers, flags
    static constexpr int kSmem = 1024 /*align slack*/ + kStages * kStageBytes + 2 * kQBytes +
                                 kMiscBytes;
    static_assert(kSmem <= 232448, "shared memory budget");
    static_assert(kHeadsPerBlock * 66 * 4 + 64 <= kStages * kStageBytes, "merge weights");
    static_assert(256 + (2 * kStages + 6) * 8 + 24 + 8 + 8 * 4 + kWarps * 2 * 16 <= kMiscBytes,
                  "misc area");
    // a warp's parked piece state fits in its own 16 rows of a stage's K and V tiles
    static constexpr int kParkML = kHeadsPerBlock * D;        // accumulators, then m[8], l[8]
    static constexpr int kHpw = kHeadsPerBlock / kWarps;      // heads each warp merges
    static_assert(kParkML + 2 * kHeadsPerBlock <= 2 * kCols64 * 512, "parked state");
    static_assert(kHeadsPerBlock % kWarps == 0, "merge split");
};

struct StageRec {
    int b, hk, hb;      // unit
    int key0;           // cache row of the tile's first key
    int ke;             // end (exclusive) of the cache rows of the tile's part of the unit
    int first, last;    // first / last tile of the piece
    int kq;             // piece number within this CTA (selects the query buffer)
    int slot, nseg;     // partial slot of the piece, pieces of the unit
    int end;            // no more tiles
    int pad;
};

// byte offset of 16-byte chunk c of row r in a tile stored as 64-column, 128-byte
// swizzled regions of `rows` rows each (the TMA SWIZZLE_128B layout)
__device__ __forceinline__ uint32_t tile_off(int r, int c, int rows) {
    return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Visible keys of one sequence as cache rows: n1 rows from row s1, then (a ring cache
// that wrapped) n2 rows from row 0.  Each part is tiled separately, so no tile crosses
// the end of the ring.
struct SeqKeys {
    int s1, n1, n2, n;
};
__device__ __forceinline__ SeqKeys seq_keys_of(const DecodeArgs &a, int kv_len) {
    SeqKeys s;
    if (kv_len < 0 || kv_len > a.max_kv_len) {  // reported once, by CTA 0
        s.s1 = s.n1 = s.n2 = s.n = 0;
        return s;
    }
    const int lo = a.window > 0 ? max(0, kv_len - a.window) : 0;
    s.n = kv_len - lo;
    if (a.ring > 0) {
        s.s1 = lo % a.ring;
        s.n1 = min(s.n, a.ring - s.s1);
    } else {
        s.s1 = lo;
        s.n1 = s.n;
    }
    s.n2 = s.n - s.n1;
    return s;
}
template <int T>
__device__ __forceinline__ int seq_tiles(const SeqKeys &s) {  // tiles of one unit
    return (s.n1 + T - 1) / T + (s.n2 + T - 1) / T;
}
__device__ __forceinline__ SeqKeys seq_keys(const DecodeArgs &a, int b) {
    return seq_keys_of(a, a.kv_lens[b]);
}

template <int D>
__global__ void __launch_bounds__(DecodeCfg<D>::kThreads, DecodeCfg<D>::kMinBlocks)
decode_bf16_kernel(const __grid_constant__ DecodeArgs a) {
    using C = DecodeCfg<D>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *sRing = smem;                                          // [stage][K | V]
    unsigned char *sQ = sRing + C::kStages * C::kStageBytes;              // [2] query blocks
    unsigned char *misc = sQ + 2 * C::kQBytes;
    StageRec *rec = reinterpret_cast<StageRec *>(misc);                   // [kStages]
    uint64_t *full = reinterpret_cast<uint64_t *>(misc + 256);            // [kStages]
    uint64_t *empty = full + C::kStages;                                  // [kStages]
    uint64_t *q_full = empty + C::kStages;                                // [2]
    uint64_t *q_empty = q_full + 2;                                       // [2]
    uint64_t *parked = q_empty + 2;                                       // piece states parked
    uint64_t *merge_bar = parked + 1;                                     // partials staged
    long long *total_p = reinterpret_cast<long long *>(parked + 2);       // key-stream length
    long long *start_p = total_p + 1;                                     // first sequence's offset
    int *start_b = reinterpret_cast<int *>(start_p + 1);                  // CTA's first sequence
    volatile int *abort_flag = start_b + 1;
    int *n_merge = const_cast<int *>(abort_flag + 1);
    int *merge_unit = n_merge + 1;                                        // [kMaxMerges][4]
    int *tickets = merge_unit + 4 * kMaxMerges;                           // [kWarps][2][4]
    // per-thread key counts; the ring is free until the first copy is issued
    long long *scan = reinterpret_cast<long long *>(sRing);               // [warps] totals

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.n_heads / a.n_kv_heads;
    const int HB = (G + kHeadsPerBlock - 1) / kHeadsPerBlock;
    const int HU = a.n_kv_heads * HB;  // units per sequence

    // ---- the tile stream: unit u of a sequence with n visible keys contributes
    // ceil(n / kTile) tiles, units laid end to end; per-thread sums over a slice of the
    // sequences, then a block-wide exclusive scan --------------------------------------
    constexpr int T = C::kTile;
    const int per_thread = (a.batch + C::kThreads - 1) / C::kThreads;
    const int b_lo = min(a.batch, tid * per_thread), b_hi = min(a.batch, b_lo + per_thread);
    if (tid == 0) {
        *start_b = -1;
        *start_p = 0;
    }
    long long my_sum = 0;
    for (int b = b_lo; b < b_hi; ++b) {
        const int kv_len = a.kv_lens[b];
        const SeqKeys sk = seq_keys_of(a, kv_len);
        my_sum += (long long)seq_tiles<T>(sk) * HU;
        if (blockIdx.x == 0) {  // CTA 0 handles sequences with nothing to stream
            if (a.defer_merge && (kv_len < 0 || kv_len > a.max_kv_len || sk.n == 0))
                for (int h = 0; h < a.n_heads; ++h)  // the merge kernel leaves them alone
                    a.piece_count[(int64_t)b * a.n_heads + h] = 0;
            if (kv_len < 0 || kv_len > a.max_kv_len) {
                report_status(a.status, kErrBounds);
            } else if (sk.n == 0) {
                for (int i = 0; i < a.n_heads * D; ++i)
                    a.out[(int64_t)b * a.out_rs + i] = __float2bfloat16_rn(0.f);
                if (a.lse != nullptr)
                    for (int h = 0; h < a.n_heads; ++h) a.lse[(int64_t)b * a.n_heads + h] = -INFINITY;
            }
        }
    }
    long long incl = my_sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) scan[warp] = incl;
    __syncthreads();
    long long total = 0, my_start = incl - my_sum;
#pragma unroll
    for (int w = 0; w < C::kWarps + 1; ++w) {
        const long long v = scan[w];
        if (w < warp) my_start += v;
        total += v;
    }
    const long long per_cta = max((total + gridDim.x - 1) / gridDim.x, (long long)(a.min_seg / T));
    const long long r0 = (long long)blockIdx.x * per_cta;
    const long long r1 = min(total, r0 + per_cta);
    const bool has_work = r0 < total;
    if (has_work && r0 >= my_start && r0 < my_start + my_sum) {  // r0 is in this slice
        long long p = my_start;
        for (int b = b_lo; b < b_hi; ++b) {
            const SeqKeys sk = seq_keys(a, b);
            const long long w = (long long)seq_tiles<T>(sk) * HU;
            if (r0 >= p && r0 < p + w) {
                *start_b = b;
                *start_p = p;
            }
            p += w;
        }
    }
    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::kWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], C::kWarps);
        }
        mbar_init(parked, C::kWarps);
        mbar_init(merge_bar, 1);
        *abort_flag = 0;
        *n_merge = 0;
        fence_mbarrier_init();
    }
    fence_proxy_async_smem();  // the scan's generic writes precede the ring's first copies
    __syncthreads();
    const uint64_t deadline = globaltimer_ns() + a.timeout_ns;
    // a deferred merge kernel may be set up now; it waits for this grid before reading
    if (a.defer_merge) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == C::kWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&a.tm_k);
            tma_prefetch_desc(&a.tm_v);
            tma_prefetch_desc(&a.tm_k16);
            tma_prefetch_desc(&a.tm_v16);
            tma_prefetch_desc(&a.tm_q);
            int tg = 0, kq = 0;  // stage fills issued, query blocks issued
            bool ok = true;
            if (has_work && *start_b >= 0) {
                int b = *start_b;
                long long pb = *start_p;  // stream offset of sequence b's first unit
                long long pos = r0;
                SeqKeys sk = seq_keys(a, b);
                int next_len = b + 1 < a.batch ? a.kv_lens[b + 1] : 0;  // fetched ahead
                while (pos < r1 && ok) {
                    const int nt = seq_tiles<T>(sk);
                    const long long w = (long long)nt * HU;
                    if (pos >= pb + w) {  // nothing (left) of this sequence in our share
                        pb += w;
                        if (++b >= a.batch) break;
                        sk = seq_keys_of(a, next_len);
                        next_len = b + 1 < a.batch ? a.kv_lens[b + 1] : 0;
                        continue;
                    }
                    const int idx = (int)((pos - pb) / nt);  // unit within the sequence
                    const int hk = idx / HB, hb = idx % HB;
                    const long long ustart = pb + (long long)idx * nt;
                    const int t0 = (int)(pos - ustart);
                    const int t1 = (int)min((long long)nt, r1 - ustart);
                    const long long first_cta = ustart / per_cta;
                    const long long last_cta = (ustart + nt - 1) / per_cta;
                    const int nseg = (int)(last_cta - first_cta + 1);
                    const int slot = (int)(blockIdx.x - first_cta);
                    // query rows of the unit's heads
                    const int qs = kq & 1;
                    if (!mbar_wait_bounded(&q_empty[qs], ((kq >> 1) & 1) ^ 1, abort_flag, deadline)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&q_full[qs], C::kQBytes);
                    const int h0 = hk * G + hb * kHeadsPerBlock;
                    for (int c = 0; c < C::kCols64; ++c)
                        tma_load_3d(sQ + qs * C::kQBytes + c * kHeadsPerBlock * 128, &a.tm_q,
                                    &q_full[qs], c * 64, h0, b);
                    const int nt1 = (sk.n1 + T - 1) / T;  // tiles of the first part
                    for (int t = t0; t < t1; ++t) {
                        // cache row of the tile's first key and the end of its part
                        const int key0 = t < nt1 ? sk.s1 + t * T : (t - nt1) * T;
                        const int kend = t < nt1 ? sk.s1 + sk.n1 : sk.n2;
                        const int s = tg % C::kStages;
                        if (!mbar_wait_bounded(&empty[s], ((tg / C::kStages) & 1) ^ 1, abort_flag,
                                               deadline)) {
                            ok = false;
                            break;
                        }
                        StageRec r;
                        r.b = b; r.hk = hk; r.hb = hb; r.key0 = key0; r.ke = kend;
                        r.first = t == t0; r.last = t == t1 - 1;
                        r.kq = kq; r.slot = slot; r.nseg = nseg; r.end = 0; r.pad = 0;
                        rec[s] = r;
                        if (a.test_skip_load && tg == 0) {  // test hook: never filled
                            ++tg;
                            continue;
                        }
                        unsigned char *dk = sRing + s * C::kStageBytes;
                        unsigned char *dv = dk + C::kTileBytes;
                        const int rows_valid = kend - key0;  // > 0: the part's rows in the tile
                        if (rows_valid < T) {
                            // a part's partial last tile: only its 16-row groups that hold
                            // keys, each landing where the whole tile would put those rows
                            // (rows past them are masked in S and zeroed in V as before)
                            const int nb = (rows_valid + 15) / 16;
                            mbar_arrive_expect_tx(&full[s], 2 * C::kCols64 * nb * 16 * 128);
                            for (int c = 0; c < C::kCols64; ++c)
                                for (int i = 0; i < nb; ++i) {
                                    const uint32_t off = c * C::kTile * 128 + i * 16 * 128;
                                    tma_load_4d(dk + off, &a.tm_k16, &full[s], c * 64, hk,
                                                key0 + 16 * i, b);
                                    tma_load_4d(dv + off, &a.tm_v16, &full[s], c * 64, hk,
                                                key0 + 16 * i, b);
                                }
                            ++tg;
                            continue;
                        }
                        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
                        if (a.chunked) {  // each tile's 64-column chunks in one copy
                            tma_load_5d(dk, &a.tm_k, &full[s], 0, key0, 0, hk, b);
                            tma_load_5d(dv, &a.tm_v, &full[s], 0, key0, 0, hk, b);
                        } else {
                            for (int c = 0; c < C::kCols64; ++c) {
                                tma_load_4d(dk + c * C::kTile * 128, &a.tm_k, &full[s], c * 64,
                                            hk, key0, b);
                                tma_load_4d(dv + c * C::kTile * 128, &a.tm_v, &full[s], c * 64,
                                            hk, key0, b);
                            }
                        }
                        ++tg;
                    }
                    ++kq;
                    pos = ustart + t1;
                }
            }
            if (ok) {  // end-of-stream record
                const int s = tg % C::kStages;
                if (mbar_wait_bounded(&empty[s], ((tg / C::kStages) & 1) ^ 1, abort_flag, deadline)) {
                    rec[s].end = 1;
                    mbar_arrive(&full[s]);
                    ++tg;  // the drain must wait on this phase, not an older one
                }
            }
            // drain: every issued copy must land before the CTA may exit.  Fills go round
            // the ring in order, so stage s last held fill s + k*kStages, the largest below tg.
            const uint64_t drain_deadline = globaltimer_ns() + 100000000ull;
            volatile int no_abort = 0;
#pragma unroll
            for (int s = 0; s < C::kStages; ++s)
                if (s < tg) {
                    const int last = s + (tg - 1 - s) / C::kStages * C::kStages;
                    if (!(a.test_skip_load && last == 0))  // the hook's fill was never issued
                        mbar_wait_bounded(&full[s], (last / C::kStages) & 1, &no_abort, drain_deadline);
                }
#pragma unroll
            for (int i = 0; i < 2; ++i)
                if (i < kq) {
                    const int last = i + (kq - 1 - i) / 2 * 2;
                    mbar_wait_bounded(&q_full[i], (last >> 1) & 1, &no_abort, drain_deadline);
                }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ compute warps
        const int row0 = warp * 16;
        float m_ref[2] = {-INFINITY, -INFINITY};  // reference maxima (log2 domain, scaled)
        float l_run[2] = {0.f, 0.f};
        float acc[D / 16][4];
#pragma unroll
        for (int i = 0; i < D / 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
        int mk = 0;  // pieces finished
        constexpr int kParkML = C::kParkML, kHpw = C::kHpw;
        // float f of warp w's parked state: 512 floats per 64-column chunk of its 16 rows,
        // K tile chunks first, then V tile chunks
        auto park_at = [](unsigned char *tk_, unsigned char *tv_, int w, int f) -> float * {
            const int p = f >> 9;
            unsigned char *base = p < C::kCols64 ? tk_ + p * C::kTile * 128
                                                 : tv_ + (p - C::kCols64) * C::kTile * 128;
            return reinterpret_cast<float *>(base + w * 16 * 128) + (f & 511);
        };
        // split pieces' merge tickets (at most two per CTA: its first and last piece), kept
        // as {ticket, nseg | unit << 8, b, h_base | g_cnt << 24}
        int n_tickets = 0;
        int *my_tickets = tickets + warp * 8;
        for (int tg = 0;; ++tg) {
            const int s = tg % C::kStages;
            const bool got = mbar_wait_bounded(&full[s], (tg / C::kStages) & 1, abort_flag, deadline);
            if (!__all_sync(0xffffffffu, got)) break;
            const StageRec r = rec[s];
            if (r.end) break;
            const int qs = r.kq & 1;
            if (r.first) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    m_ref[c] = -INFINITY;
                    l_run[c] = 0.f;
                }
#pragma unroll
                for (int i = 0; i < D / 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
                const bool qgot = mbar_wait_bounded(&q_full[qs], (r.kq >> 1) & 1, abort_flag, deadline);
                if (!__all_sync(0xffffffffu, qgot)) break;
            }
            unsigned char *tk = sRing + s * C::kStageBytes;
            unsigned char *tv = tk + C::kTileBytes;
            const unsigned char *tq = sQ + qs * C::kQBytes;
            // this warp's rows past the piece's end: zero their V (their K is masked below)
            const int valid_rows = r.ke - (r.key0 + row0);
            if (valid_rows < 16) {
                for (int i = lane; i < 16 * C::kChunks; i += 32) {
                    const int rr = i / C::kChunks, c = i % C::kChunks;
                    if (rr >= valid_rows)
                        *reinterpret_cast<uint4 *>(tv + tile_off(row0 + rr, c, C::kTile)) =
                            make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }

            // S^T = K . Q^T for this warp's 16 keys
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < D / 16; ks += 2) {
                uint32_t qf[4];  // b0,b1 for k-steps ks and ks+1
                {
                    const int c = 2 * ks + (lane >> 3);
                    ldmatrix_x4(qf, tq + tile_off(lane & 7, c < C::kChunks ? c : 0, kHeadsPerBlock));
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (ks + u < D / 16) {
                        uint32_t af[4];
                        const int rr = row0 + (lane & 7) + 8 * ((lane >> 3) & 1);
                        const int c = 2 * (ks + u) + (lane >> 4);
                        ldmatrix_x4(af, tk + tile_off(rr, c, C::kTile));
                        mma_bf16_16816(sc, af, qf[2 * u], qf[2 * u + 1]);
                    }
                }
            }
            // scale (and cap) into the log2 domain and mask keys past the piece
            if (a.cap_log2 > 0.f) {
                const float k2 = a.raw_over_cap * kTwoLog2e;
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[e] = capped_score_log2(sc[e], k2, a.cap_log2);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[e] *= a.scale_log2;
            }
            const int key_a = r.key0 + row0 + (lane >> 2);
            const bool va = key_a < r.ke, vb = key_a + 8 < r.ke;
            sc[0] = va ? sc[0] : -INFINITY;
            sc[1] = va ? sc[1] : -INFINITY;
            sc[2] = vb ? sc[2] : -INFINITY;
            sc[3] = vb ? sc[3] : -INFINITY;

            float p[4], corr[2];
            bool refresh_any = false;
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
                const int rr = row0 + (lane & 7) + 8 * (lane >> 4);
                const int c = 2 * i + ((lane >> 3) & 1);
                ldmatrix_x4_trans(vf, tv + tile_off(rr, c, C::kTile));
                mma_bf16_16816(acc[i], vf, pb0, pb1);
            }
            // zeroed rows (generic writes) must precede the stage's next copy
            if (valid_rows < 16) fence_proxy_async_smem();
            __syncwarp();
            if (!r.last) {  // release the stage
                if (lane == 0) mbar_arrive(&empty[s]);
                continue;
            }

            // ---- end of a piece: release the query block, merge the warps ----------
            // Every warp parks its state in its own rows of this stage, which no other warp
            // reads while computing: accumulator register j = 4i+e of lane l at float
            // 32j + (l ^ (j & 31)) (the XOR spreads the merge's reads over the banks), then
            // m[8] and l[8].  Once all warps have parked, warp w combines heads
            // [w*kHpw, (w+1)*kHpw) of every state, writes them out and releases the stage.
            if (lane == 0) mbar_arrive(&q_empty[qs]);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                l_run[c] += __shfl_xor_sync(0xffffffffu, l_run[c], 4);
                l_run[c] += __shfl_xor_sync(0xffffffffu, l_run[c], 8);
                l_run[c] += __shfl_xor_sync(0xffffffffu, l_run[c], 16);
            }
            {
                const int g0 = 2 * (lane & 3);
#pragma unroll
                for (int i = 0; i < D / 16; ++i)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = 4 * i + e;
                        *park_at(tk, tv, warp, 32 * j + (lane ^ (j & 31))) = acc[i][e];
                    }
                if (lane < 4) {
                    float *ml = park_at(tk, tv, warp, kParkML);
                    ml[g0] = m_ref[0];
                    ml[g0 + 1] = m_ref[1];
                    ml[kHeadsPerBlock + g0] = l_run[0];
                    ml[kHeadsPerBlock + g0 + 1] = l_run[1];
                }
            }
            fence_proxy_async_smem();  // the parked writes precede the stage's next copy
            __syncwarp();
            if (lane == 0) mbar_arrive(parked);
            const bool pk = mbar_wait_bounded(parked, mk & 1, abort_flag, deadline);
            if (!__all_sync(0xffffffffu, pk)) break;

            const int h_base = r.hk * G + r.hb * kHeadsPerBlock;
            const int g_cnt = min(kHeadsPerBlock, G - r.hb * kHeadsPerBlock);
            const bool single = r.nseg == 1;
            const int64_t prow = ((int64_t)r.b * a.n_heads + h_base) * a.max_splits + r.slot;
            constexpr int kV8 = D / 8;  // 8-element vectors per head row
            for (int v = lane; v < kHpw * kV8; v += 32) {
                const int g = warp * kHpw + v / kV8, x = 8 * (v % kV8);
                if (g >= g_cnt) continue;
                float mx = -INFINITY;
#pragma unroll
                for (int w = 0; w < C::kWarps; ++w) mx = fmaxf(mx, park_at(tk, tv, w, kParkML)[g]);
                const float mu = mx == -INFINITY ? 0.f : mx;
                float f[C::kWarps], l = 0.f;
#pragma unroll
                for (int w = 0; w < C::kWarps; ++w) {
                    const float *ml = park_at(tk, tv, w, kParkML);
                    f[w] = fast_exp2(ml[g] - mu);
                    l += ml[kHeadsPerBlock + g] * f[w];
                }
                const float rl = 1.f / l;
                // element (g, x+k) sits in register j = 4*(x/16) + (g&1) + 2*((x/8)&1) of
                // lane 4k + g/2 (the m16n8 accumulator layout with keys' D in M)
                const int j = 4 * (x >> 4) + (g & 1) + 2 * ((x >> 3) & 1);
                float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int w = 0; w < C::kWarps; ++w) {
                    const float *row = park_at(tk, tv, w, 32 * j);
#pragma unroll
                    for (int k = 0; k < 8; ++k) o[k] += f[w] * row[(4 * k + (g >> 1)) ^ (j & 31)];
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] *= rl;
                const float lse2 = mu + log2f(l);  // log2 domain
                if (a.defer_merge && x == 0 && r.slot == 0)
                    a.piece_count[(int64_t)r.b * a.n_heads + h_base + g] = r.nseg;
                if (single) {
                    *reinterpret_cast<uint4 *>(a.out + (int64_t)r.b * a.out_rs +
                                               (int64_t)(h_base + g) * D + x) =
                        make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                                   pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7]));
                    if (x == 0 && a.lse != nullptr) a.lse[(int64_t)r.b * a.n_heads + h_base + g] = lse2 * kLn2;
                } else {
                    float *dst = a.part_o + (prow + (int64_t)g * a.max_splits) * D + x;
                    *reinterpret_cast<float4 *>(dst) = make_float4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<float4 *>(dst + 4) = make_float4(o[4], o[5], o[6], o[7]);
                    if (x == 0) a.part_lse[prow + (int64_t)g * a.max_splits] = lse2;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage
            if (!single && !a.defer_merge) {
                // Ticket: the warp that brings the unit's count to nseg * kWarps is the last
                // writer of its partials and queues the unit for merging after the stream.
                // The result is only examined after the stream, so the round trip overlaps it.
                __threadfence();
                __syncwarp();
                if (lane == 0) {
                    const int unit = (r.b * a.n_kv_heads + r.hk) * HB + r.hb;
                    const int t = atomicAdd(a.counters + unit, 1);
                    if (n_tickets < 2) {
                        int *tk4 = my_tickets + 4 * n_tickets;
                        tk4[0] = t;
                        tk4[1] = r.nseg | (unit << 8);
                        tk4[2] = r.b;
                        tk4[3] = h_base | (g_cnt << 24);
                    }
                    ++n_tickets;
                }
            }
            ++mk;
        }
        if (lane == 0) {  // queue the units whose last partial this warp wrote
            if (n_tickets > 2) report_status(a.status, kErrCuda);  // cannot happen by construction
            for (int k = 0; k < min(n_tickets, 2); ++k) {
                const int *tk4 = my_tickets + 4 * k;
                if (tk4[0] != (tk4[1] & 0xff) * C::kWarps - 1) continue;
                const int n = atomicAdd(n_merge, 1);
                if (n < kMaxMerges) {
                    merge_unit[4 * n + 0] = tk4[2];
                    merge_unit[4 * n + 1] = tk4[3] & 0xffffff;
                    merge_unit[4 * n + 2] = tk4[3] >> 24;
                    merge_unit[4 * n + 3] = tk4[1];
                } else {
                    report_status(a.status, kErrCuda);  // cannot happen by construction
                }
            }
        }
    }
    __syncthreads();
    if (*abort_flag) {
        if (tid == 0) report_status(a.status, kErrTimeout);
        return;
    }

    // ---- merge the units this CTA finished last: lse-weighted sum of their pieces ----
    // The partial rows of a head sit side by side in the scratch, so one bulk copy per
    // head stages all of them in the (now idle) ring: one round trip to L2 per unit.
    // Meanwhile each warp turns its heads' partial lse values into weights.
    __threadfence();
    const int n_merges = min(*n_merge, kMaxMerges);
    float *wts = reinterpret_cast<float *>(sQ);  // [g][nseg] weights, then [g] lse
    int n_staged = 0;  // completed phases of merge_bar: only staged merges use it
    for (int mi = 0; mi < n_merges; ++mi) {
        const int b = merge_unit[4 * mi + 0], h_base = merge_unit[4 * mi + 1];
        const int g_cnt = merge_unit[4 * mi + 2];
        const int nseg = merge_unit[4 * mi + 3] & 0xff, unit = merge_unit[4 * mi + 3] >> 8;
        const uint32_t row_bytes = (uint32_t)nseg * D * 4;
        const bool staged = nseg <= 96 &&
                            (size_t)g_cnt * row_bytes <= (size_t)C::kStages * C::kStageBytes &&
                            kHeadsPerBlock * (nseg + 1) * 4 <= 2 * C::kQBytes;
        if (staged && tid == 0) {
            fence_proxy_async_global();
            mbar_arrive_expect_tx(merge_bar, (uint32_t)g_cnt * row_bytes);
            for (int g = 0; g < g_cnt; ++g)
                bulk_load(sRing + g * row_bytes,
                          a.part_o + ((int64_t)b * a.n_heads + h_base + g) * a.max_splits * D,
                          row_bytes, merge_bar);
        }
        if (staged) {
            for (int g = warp; g < g_cnt; g += C::kWarps + 1) {
                const int64_t rb = ((int64_t)b * a.n_heads + h_base + g) * a.max_splits;
                float lv[3];  // nseg <= 96 (the scratch layout keeps it near 66)
#pragma unroll
                for (int k = 0; k < 3; ++k)
                    lv[k] = lane + 32 * k < nseg ? __ldcg(a.part_lse + rb + lane + 32 * k) : -INFINITY;
                float M = fmaxf(fmaxf(lv[0], lv[1]), lv[2]);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
                float e[3], Z = 0.f;
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    e[k] = lv[k] == -INFINITY ? 0.f : fast_exp2(lv[k] - M);
                    Z += e[k];
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, off);
                const float rz = 1.f / Z;
#pragma unroll
                for (int k = 0; k < 3; ++k)
                    if (lane + 32 * k < nseg) wts[g * nseg + lane + 32 * k] = e[k] * rz;
                if (lane == 0) wts[kHeadsPerBlock * nseg + g] = M + log2f(Z);
            }
            __syncthreads();
            const bool got = mbar_wait_bounded(merge_bar, n_staged & 1, abort_flag, deadline);
            if (!__syncthreads_and(got)) {  // the copies must land before the CTA may go
                volatile int no_abort = 0;
                mbar_wait_bounded(merge_bar, n_staged & 1, &no_abort, globaltimer_ns() + 100000000ull);
                if (tid == 0) report_status(a.status, kErrTimeout);
                return;
            }
            constexpr int kV4 = D / 4;
            for (int i = tid; i < g_cnt * kV4; i += C::kThreads) {
                const int g = i / kV4, x = 4 * (i % kV4);
                const float *src = reinterpret_cast<const float *>(sRing + g * row_bytes) + x;
                float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int sp = 0; sp < nseg; ++sp) {
                    const float w = wts[g * nseg + sp];
                    const float4 v = *reinterpret_cast<const float4 *>(src + sp * D);
                    o.x += w * v.x; o.y += w * v.y; o.z += w * v.z; o.w += w * v.w;
                }
                *reinterpret_cast<uint2 *>(a.out + (int64_t)b * a.out_rs + (int64_t)(h_base + g) * D + x) =
                    make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
                if (x == 0 && a.lse != nullptr)
                    a.lse[(int64_t)b * a.n_heads + h_base + g] = wts[kHeadsPerBlock * nseg + g] * kLn2;
            }
            ++n_staged;
            __syncthreads();  // the ring and weights are reused by the next unit
        } else {
            // too many pieces to stage: one thread per 4 outputs, partials straight from L2
            constexpr int kV4 = D / 4;
            for (int i = tid; i < g_cnt * kV4; i += C::kThreads) {
                const int g = i / kV4, x = 4 * (i % kV4);
                const int64_t rb = ((int64_t)b * a.n_heads + h_base + g) * a.max_splits;
                float M = -INFINITY, Z = 0.f;
                float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int sp = 0; sp < nseg; ++sp) {
                    const float l = __ldcg(a.part_lse + rb + sp);
                    const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.part_o + (rb + sp) * D + x));
                    const float mn = fmaxf(M, l);
                    const float c = M == -INFINITY ? 0.f : fast_exp2(M - mn);
                    const float e = fast_exp2(l - mn);
                    Z = Z * c + e;
                    o.x = o.x * c + e * v.x; o.y = o.y * c + e * v.y;
                    o.z = o.z * c + e * v.z; o.w = o.w * c + e * v.w;
                    M = mn;
                }
                const float rz = 1.f / Z;
                *reinterpret_cast<uint2 *>(a.out + (int64_t)b * a.out_rs + (int64_t)(h_base + g) * D + x) =
                    make_uint2(pack_bf16x2(o.x * rz, o.y * rz), pack_bf16x2(o.z * rz, o.w * rz));
                if (x == 0 && a.lse != nullptr)
                    a.lse[(int64_t)b * a.n_heads + h_base + g] = (M + log2f(Z)) * kLn2;
            }
        }
        if (tid == 0) a.counters[unit] = 0;  // ready for the next call
    }
}

// The deferred split-KV merge for few long units: the pieces of one (sequence, query
// head), lse_c and normalised o_c, combine as
//   lse = log2 sum_c 2^{lse_c} (log2 domain),  out = sum_c 2^{lse_c - lse} o_c.
// Each head's columns are split over kMergeSplit<D> CTAs of kMergeV4<D> 16-byte vectors;
// within a CTA thread t takes column vector t % w4 of pieces t / w4, t / w4 + groups, ...
// It issues the loads of its first kMergeBatch pieces (lse and partial) at once, so the
// whole merge costs about one round trip to L2; the maximum lse is a block reduction.
constexpr int kMergeThreads = 256;
constexpr int kMergeBatch = 8;  // pieces per thread held in registers
template <int D>
constexpr int kMergeV4 = D >= 256 ? 32 : 8;
template <int D>
constexpr int kMergeSplit = (D / 4 + kMergeV4<D> - 1) / kMergeV4<D>;

template <int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const DecodeArgs a) {
    constexpr int kV4 = D / 4;
    __shared__ float4 red[kMergeThreads];
    __shared__ float red_m[kMergeThreads / 32], red_z[kMergeThreads];
    // launched as a programmatic dependent of the stream: wait until that grid has
    // finished and its partial results are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int bh = blockIdx.x / kMergeSplit<D>, cb = blockIdx.x % kMergeSplit<D>;
    // (clamped: a stream that gave up early may leave counts of an earlier call)
    const int nseg = min(a.piece_count[bh], a.max_splits);
    if (nseg <= 1) return;  // written whole by its only piece (or nothing to write)
    const int v0 = cb * kMergeV4<D>, w4 = min(kMergeV4<D>, kV4 - v0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int groups = kMergeThreads / w4;  // w4 divides the block (a power of two or 4)
    const int g = tid / w4, col = v0 + tid % w4;
    const bool active = g < groups;
    const float *pl = a.part_lse + (int64_t)bh * a.max_splits;
    const float4 *po = reinterpret_cast<const float4 *>(a.part_o + (int64_t)bh * a.max_splits * D) + col;
    float lv[kMergeBatch];
    float4 ov[kMergeBatch];
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
        const int sp = g + k * groups;
        const bool ok = active && sp < nseg;
        lv[k] = ok ? __ldcg(pl + sp) : -INFINITY;
        ov[k] = ok ? __ldcg(po + (int64_t)sp * kV4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) m = fmaxf(m, lv[k]);
    for (int sp = g + kMergeBatch * groups; active && sp < nseg; sp += groups) m = fmaxf(m, __ldcg(pl + sp));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) red_m[warp] = m;
    __syncthreads();
    float M = red_m[0];
#pragma unroll
    for (int w = 1; w < kMergeThreads / 32; ++w) M = fmaxf(M, red_m[w]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float z = 0.f;
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
        const float wt = lv[k] == -INFINITY ? 0.f : fast_exp2(lv[k] - M);
        z += wt;
        acc.x += wt * ov[k].x; acc.y += wt * ov[k].y; acc.z += wt * ov[k].z; acc.w += wt * ov[k].w;
    }
    for (int sp = g + kMergeBatch * groups; active && sp < nseg; sp += groups) {
        const float l = __ldcg(pl + sp);
        const float wt = l == -INFINITY ? 0.f : fast_exp2(l - M);
        const float4 v = __ldcg(po + (int64_t)sp * kV4);
        z += wt;
        acc.x += wt * v.x; acc.y += wt * v.y; acc.z += wt * v.z; acc.w += wt * v.w;
    }
    red[tid] = acc;
    red_z[tid] = z;
    __syncthreads();
    if (tid < w4) {  // column vector v0 + tid: sum over the piece groups
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        float zt = 0.f;
        for (int gg = 0; gg < groups; ++gg) {
            const float4 v = red[gg * w4 + tid];
            o.x += v.x; o.y += v.y; o.z += v.z; o.w += v.w;
            zt += red_z[gg * w4];  // every column's threads saw the same weights
        }
        const float rz = 1.f / zt;
        const int b = bh / a.n_heads, h = bh % a.n_heads;
        *reinterpret_cast<uint2 *>(a.out + (int64_t)b * a.out_rs + (int64_t)h * D + 4 * (v0 + tid)) =
            make_uint2(pack_bf16x2(o.x * rz, o.y * rz), pack_bf16x2(o.z * rz, o.w * rz));
        if (cb == 0 && tid == 0 && a.lse != nullptr) a.lse[bh] = (M + log2f(zt)) * kLn2;
    }
}

template <int D>
cudaError_t launch_decode_d(const DecodeArgs &a, int grid, cudaStream_t s) {
    using C = DecodeCfg<D>;
    cudaError_t e = cudaFuncSetAttribute(decode_bf16_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    decode_bf16_kernel<D><<<grid, C::kThreads, C::kSmem, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess || !a.defer_merge) return e;
    // programmatic dependent launch: the merge grid is set up while the stream runs
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(a.batch * a.n_heads * kMergeSplit<D>);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, a)) != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int D>
int tile_keys() { return DecodeCfg<D>::kTile; }
template <int D>
int ctas_per_sm() {  // resident CTAs per SM as the runtime sees them (smem and registers)
    using C = DecodeCfg<D>;
    int n = 0;
    if (cudaFuncSetAttribute(decode_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_bf16_kernel<D>, C::kThreads,
                                                      C::kSmem) != cudaSuccess)
        return 1;
    return std::max(1, n);
}

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

// Pieces are at least min_seg keys long, so a unit of at most `range` keys falls into at
// most range / min_seg + 2 pieces; min_seg grows with the range so that the count stays
// near 64 (the scratch layout is sized for it).  Shapes with few units, where that would
// leave CTAs idle, take the deferred-merge plan below instead.
constexpr int64_t kDeferPieces = 8;
static int min_seg_for(int range, int T) {
    const int m = std::max(4 * T, (range + 63) / 64);
    return (m + T - 1) / T * T;
}

int64_t decode_bf16_units(int batch, int n_heads, int n_kv_heads) {
    const int G = n_heads / n_kv_heads;
    return (int64_t)batch * n_kv_heads * ((G + kHeadsPerBlock - 1) / kHeadsPerBlock);
}

bool plan_decode_bf16(int batch, int n_heads, int n_kv_heads, int head_dim, int max_kv_len,
                      int window, int num_sms, DecodePlan *p) {
    if (decode_bf16_units(batch, n_heads, n_kv_heads) >= kDecodeMaxUnits) return false;
    int T, occ;
    switch (head_dim) {
        case 64: T = tile_keys<64>(); occ = ctas_per_sm<64>(); break;
        case 80: T = tile_keys<80>(); occ = ctas_per_sm<80>(); break;
        case 128: T = tile_keys<128>(); occ = ctas_per_sm<128>(); break;
        case 256: T = tile_keys<256>(); occ = ctas_per_sm<256>(); break;
        case 512: T = tile_keys<512>(); occ = ctas_per_sm<512>(); break;
        default: return false;
    }
    const int G = n_heads / n_kv_heads;
    const int HB = (G + kHeadsPerBlock - 1) / kHeadsPerBlock;
    const int64_t units = (int64_t)batch * n_kv_heads * HB;
    const int grid = num_sms * occ;
    // the scratch layout uses the window-free bound, so one workspace fits every window
    const int layout_range = std::max(max_kv_len, 1);
    // pieces per unit that would keep every CTA streaming; beyond a few, the last CTA of a
    // unit would merge many pieces after its stream (about 8 us at head_dim 512, measured),
    // so cut the stream that finely and merge in a second kernel
    const int64_t target = (grid + units - 1) / units;
    const bool defer = target > kDeferPieces;
    int min_seg = min_seg_for(layout_range, T);
    if (defer) {
        const int64_t m = std::max<int64_t>(4 * T, (layout_range + target - 1) / target);
        min_seg = (int)((m + T - 1) / T * T);
    }
    const int layout_splits = (layout_range + min_seg - 1) / min_seg + 2;
    p->head_blocks = HB;
    p->min_seg = min_seg;
    p->max_splits = layout_splits;
    p->grid = grid;
    p->defer_merge = defer ? 1 : 0;
    auto round256 = [](size_t x) { return (x + 255) / 256 * 256; };
    p->part_o_bytes = round256((size_t)batch * n_heads * layout_splits * head_dim * 4);
    p->part_lse_bytes = round256((size_t)batch * n_heads * layout_splits * 4);
    // merge counters per unit, or (deferred merge) piece counts per (sequence, head)
    p->counter_bytes = round256((size_t)(defer ? (int64_t)batch * n_heads : units) * 4);
    p->total_bytes = p->part_o_bytes + p->part_lse_bytes + p->counter_bytes;
    (void)window;
    return true;
}

cudaError_t launch_decode_bf16(const DecodeArgs &a, int grid, cudaStream_t s) {
    switch (a.head_dim) {
        case 64: return launch_decode_d<64>(a, grid, s);
        case 80: return launch_decode_d<80>(a, grid, s);
        case 128: return launch_decode_d<128>(a, grid, s);
        case 256: return launch_decode_d<256>(a, grid, s);
        case 512: return launch_decode_d<512>(a, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lat
