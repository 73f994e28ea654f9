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
//  * A unit of work ("item") is a 128-row query tile of one head (one TMEM lane per query
//    row).  The grid is persistent, one CTA per SM (two for head_dim 64), and CTA c walks
//    the items heaviest first, dealt forwards and backwards in turn; its K/V rings, S
//    buffers and barrier phases run on across items.  head_dim 64 uses 64-key tiles, or
//    96-key tiles where a query tile visits about 1K keys or more (prefill_tc_wide).
//  * Warp roles: warps 0-7 run the softmax as two warpgroups that split each S tile's
//    columns (thread t of a warpgroup <-> query row t; the two halves meet through a
//    small shared-memory exchange for the row max and sum), warp 8 loads Q and K tiles
//    with TMA, warp 9 loads V tiles, warp 10 issues tcgen05.mma.  Synchronisation is by
//    mbarriers only.
//  * S = Q K^T is accumulated in tensor memory (fp32, double-buffered so the MMA of tile
//    j+1 overlaps the softmax of tile j); P = exp2(S*scale*log2e - m) is written as bf16
//    back into the S buffer it came from, and O += P V reads it straight from tensor
//    memory (one MMA per 16 keys covering all of this CTA's O columns).
//  * K and V tiles reach shared memory through two rings (one for K tiles, one for V
//    tiles), each tile a set of [BN keys x 64 head-dims] chunks with 128-byte swizzle
//    filled by its own producer warp under ONE mbarrier per tile: a TMA producer that
//    arms a barrier per small chunk spends most of its time on the barrier round trip,
//    and the consumer would wait once per chunk.  Q and K enter the MMA K-major; V
//    enters MN-major, one 64-column chunk per MMA.
//  * Tiles wholly outside the causal / window band are never loaded or computed; tiles
//    wholly inside it skip the per-element mask.
//  * The running maximum is refreshed only when it grows by more than 2^8 (the stale
//    maximum keeps every weight <= 256, well inside fp32/bf16 range), so the O rescale
//    in tensor memory is rare; the result is exact up to rounding because O and l always
//    share the same reference maximum.
//  * head_dim 80 runs as two chunks (64 + 16 live columns; the tensor map zero-fills
//    columns past 80).  head_dim 512 splits O into two 256-column halves (a 128 x 512 fp32
//    accumulator alone would fill tensor memory), each half an item of its own.
//  * head_dim 512 with an even GQA group runs on CTA pairs (a 2-CTA cluster on the two SMs
//    of a TPC, tcgen05 .cta_group::2): the pair takes one query tile of two query heads
//    that share a KV head, CTA r holding head 2j+r's 128 query rows.  Each pair MMA is
//    M = 256 (both heads' rows) x N = 128 keys, with every CTA holding only its 64 keys of
//    the K tile and its 128 columns of the V tile, so a 128-key tile fits next to a
//    128 x 512 query tile in shared memory and the S MMA runs at N = 128 (a single CTA
//    could only afford N = 64, which the tensor pipe runs at about half rate).  The even
//    CTA issues the MMAs; both CTAs' copies count on its barriers, and its commits arrive
//    on the barriers of both.
//  * Every mbarrier wait is bounded by a wall-clock budget; on expiry the CTA records
//    LAT_ERR_TIMEOUT, drains its in-flight copies and MMAs, frees tensor memory and exits.
#include <math.h>

#include <algorithm>

#include "device_common.cuh"
#include "kernels.h"

namespace lat {

namespace {

constexpr int kBM = 128;             // query rows per CTA (= TMEM lanes)
constexpr int kThreads = 352;        // 8 softmax warps + K and V producer warps + MMA warp
constexpr int kSoftmaxThreads = 256;
constexpr int kKProducerWarp = 8;
constexpr int kVProducerWarp = 9;
constexpr int kMmaWarp = 10;
constexpr int kChunkCols = 64;       // head-dim columns per swizzled chunk (128 bytes)
constexpr uint32_t kTmemO = 0;       // O accumulator columns [0, kOCols)
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D, bool W = false, bool P = false>
struct TcCfg {
    static_assert(!P || D == 512, "the CTA-pair form exists for head_dim 512");
    static constexpr int kQkChunks = (D + kChunkCols - 1) / kChunkCols;   // Q/K chunks
    static constexpr int kKSteps = (D + 15) / 16;                          // S MMA k-steps
    // keys per tile; head_dim 64 takes 64-key tiles so that two CTAs fit one SM (256 tensor
    // memory columns and under 113 KB of shared memory each): at that size a CTA's serial
    // chain of S MMA, softmax and P.V leaves the SM idle, and a second CTA fills the gaps
    // W (head_dim 64 with long key ranges): 96-key tiles, which halve the per-tile fixed
    // costs where a query tile visits a thousand keys or more, still two CTAs per SM
    // P (head_dim 512 on a CTA pair): 128-key tiles, 64 keys of K in each CTA
    static constexpr int kBN = P ? 128 : (D == 64 ? (W ? 96 : 64) : (D <= 256 ? 128 : 64));
    static constexpr int kKRows = P ? kBN / 2 : kBN;                       // K rows per CTA
    static constexpr int kCtasPerSm = D == 64 ? 2 : 1;
    static constexpr uint32_t kTmemS = D == 64 ? 64 : 256;     // S buffers at kTmemS (+ BN)
    static constexpr uint32_t kTmemCols = D == 64 ? 256 : 512;
    static constexpr int kSplitO = D == 512 ? 2 : 1;                       // O column halves
    static constexpr int kOCols = D / kSplitO;                             // O cols per CTA
    static constexpr int kVCols = P ? kOCols / 2 : kOCols;                 // V cols per CTA
    static constexpr int kVChunks = (kVCols + kChunkCols - 1) / kChunkCols;
    static constexpr int kKChunkBytes = kKRows * 128;                      // [rows x 64] chunk
    static constexpr int kVChunkBytes = kBN * 128;
    static constexpr int kKTileBytes = kQkChunks * kKChunkBytes;
    static constexpr int kVTileBytes = kVChunks * kVChunkBytes;
    // Few tiles in flight: with deeper rings (and the next item's query tile loaded ahead)
    // every CTA's requests queue behind one another and each load lands later, while the
    // per-tile chain is set by the MMAs and the softmax.  Measured: head_dim 64, 2 + 2
    // slots and one query tile 25.7 vs 26.5 us (4 + 4 and two) on the Qwen3 shape, 1 + 1
    // for the 96-key tiles 70.1 vs 75.2 us (3 + 3) on the chunked prefill; head_dim 128,
    // 1 + 1 and one query tile 555.8 vs 574.0 us (3 + 2 and two) on B1 S8192 H32/8 and
    // 49.5 vs 51.4 us on B8 S512.
    static constexpr int kKStages = D == 64 && !W ? 2 : 1;
    static constexpr int kVStages = D == 64 && !W ? 2 : 1;
    static constexpr int kQBytes = kQkChunks * kBM * 128;
    static constexpr int kQStages = 1;
    // Output staging: each softmax warp writes its 32 rows x kEpiCols output columns per
    // pass into one of its kEpiBufs swizzled boxes and hands the box to one TMA store.
    // Row-per-thread global stores touch 32 rows per instruction, and at head_dim 256 they
    // held the softmax warps for most of a 3 us item boundary.  Single-CTA head_dim 128/256
    // stage in boxes of their own; the CTA pair (no shared memory left) stages in its V
    // slot, which is free from the item's last P.V until the next item's first V copy, and
    // that copy waits until the boxes have been read.  Head_dim 64 (two stores per thread),
    // 80 (no whole boxes) and single-CTA 512 (no room) store rows directly.
    static constexpr bool kEpiOwn = !P && (D == 128 || D == 256);
    static constexpr bool kEpiInV = P;
    static constexpr bool kEpiTma = kEpiOwn || kEpiInV;
    static constexpr int kEpiCols = 64;                                   // box columns
    static constexpr int kEpiBufs = 1;                                    // boxes per warp
    static constexpr int kEpiPasses = kEpiTma ? kOCols / 2 / kEpiCols : 0;  // boxes per item
    static constexpr int kEpiBoxBytes = 32 * kEpiCols * 2;
    static constexpr int kEpiStageBytes = kSoftmaxThreads / 32 * kEpiBufs * kEpiBoxBytes;
    static constexpr int kEpiBytes = kEpiOwn ? kEpiStageBytes : 0;
    static_assert(!kEpiTma || 2 * kEpiPasses * kEpiCols == kOCols, "boxes cover the columns");
    static_assert(!kEpiInV || (kVStages == 1 && kEpiStageBytes <= kVTileBytes),
                  "the boxes fit the V slot");
    static constexpr int kBarBytes = 256 + 4 * kBM * 4;  // barriers + row exchange
    static constexpr int kPayload = kQStages * kQBytes + kKStages * kKTileBytes +
                                    kVStages * kVTileBytes + kEpiBytes + kBarBytes;
    // 1 KB of slack lets the 1024-byte aligned carve-up start anywhere; a shape that
    // cannot afford it relies on the dynamic shared memory base being 1024-byte aligned
    // (checked at run time)
    static constexpr int kSlack = kPayload + 1024 <= 232448 ? 1024 : 0;
    static constexpr int kSmem = kSlack + kPayload;
    static_assert(kSmem <= 232448, "shared memory budget");
    static_assert(kOCols <= kTmemS && kTmemS + 2 * kBN <= kTmemCols, "tensor memory budget");
    static_assert(kBN % 32 == 0, "P columns per warpgroup must fill whole TMEM stores");
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

// The same for an MN-major operand whose 64-column atoms sit `atom_stride` bytes apart:
// the leading byte offset is the stride between atoms along N, the stride byte offset
// the 1024 bytes between 8-row groups along K.
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t saddr, uint32_t atom_stride) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)(atom_stride >> 4) << 16;
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

// One unit of work: a 128-row query tile of one query head (and one O half for D = 512).
// On a CTA pair the unit is the same tile of two query heads of one GQA group, CTA r
// taking head 2j + r.
struct Item {
    int b, h, half, m0, rows, hk;
    Band band;
};

// Items are numbered heaviest first (latest query tiles, which see the most keys under a
// causal mask), then by sequence and head.
template <int D, bool W, bool P>
__device__ __forceinline__ Item item_at(const PrefillTcArgs &a, int idx, int rank) {
    using C = TcCfg<D, W, P>;
    const int head_slots = P ? a.n_heads / 2 : a.n_heads;  // heads, or head pairs
    const int per_tile = a.batch * head_slots * C::kSplitO;
    const int n_mtiles = (a.seq_len + kBM - 1) / kBM;
    const int z = idx / per_tile, rem = idx % per_tile;
    const int mt = n_mtiles - 1 - z;
    Item it;
    it.b = rem / (head_slots * C::kSplitO);
    const int head_sel = rem % (head_slots * C::kSplitO);
    const int hs = head_sel / C::kSplitO;
    it.h = P ? 2 * hs + rank : hs;
    it.half = head_sel % C::kSplitO;
    it.m0 = mt * kBM;
    it.rows = min(kBM, a.seq_len - it.m0);
    it.hk = it.h / (a.n_heads / a.n_kv_heads);
    it.band = kv_band(it.m0, it.rows, a.seq_len, a.kv_len, a.causal, a.window, C::kBN);
    return it;
}

// The k-th item of CTA c in a grid of G: rounds of G items in heaviest-first order, dealt
// forwards and backwards in turn (a "snake"), so that the CTA with the heaviest item of
// one round gets the lightest of the next.  -1 past the end.
__device__ __forceinline__ int item_index(int k, int c, int G, int n_items) {
    const int idx = k * G + ((k & 1) ? G - 1 - c : c);
    return idx < n_items ? idx : -1;
}

template <int D, bool W, bool P>
__global__ void __launch_bounds__(kThreads, TcCfg<D, W, P>::kCtasPerSm)
prefill_tc_kernel(const __grid_constant__ PrefillTcArgs a) {
    using C = TcCfg<D, W, P>;
    constexpr int BN = C::kBN;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if (C::kSlack == 0 && smem != smem_raw) {  // no room to realign: refuse to run (both
        if (threadIdx.x == 0) report_status(a.status, kErrCuda);  // CTAs of a pair alike)
        return;
    }
    unsigned char *sQ = smem;                                 // [kQStages] Q tiles
    unsigned char *sK = sQ + C::kQStages * C::kQBytes;        // [kKStages] K tiles
    unsigned char *sV = sK + C::kKStages * C::kKTileBytes;    // [kVStages] V tiles
    unsigned char *sEpi = sV + C::kVStages * C::kVTileBytes;  // output boxes, one per warp
    uint64_t *bars = reinterpret_cast<uint64_t *>(sEpi + C::kEpiBytes);
    unsigned char *sStage = C::kEpiInV ? sV : sEpi;            // where the boxes are staged
    uint64_t *q_full = bars + 0;       // [2]
    uint64_t *q_empty = bars + 2;      // [2]
    uint64_t *bar_s = bars + 4;        // [2] S(g) ready, by global tile parity
    uint64_t *bar_p = bars + 6;        // [2] P(g) ready
    uint64_t *bar_o = bars + 8;        // one phase per P.V MMA group (global tile order)
    uint64_t *o_full = bars + 9;       // one phase per item: its O is complete
    uint64_t *bar_done = bars + 10;    // every MMA complete (drain)
    uint64_t *bar_x = bars + 11;       // [4] softmax row exchange, one per TMEM lane quarter
    uint64_t *k_full = bars + 15;      // [kKStages]
    uint64_t *k_empty = k_full + C::kKStages;
    uint64_t *v_full = k_empty + C::kKStages;   // [kVStages]
    uint64_t *v_empty = v_full + C::kVStages;
    uint64_t *epi_done = v_empty + C::kVStages;  // one phase per item: its boxes are read
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(epi_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *xchg = reinterpret_cast<float *>(bars + 32);   // [2 parities][2 warpgroups][kBM]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int head_slots = P ? a.n_heads / 2 : a.n_heads;
    const int n_items = a.batch * head_slots * C::kSplitO * ((a.seq_len + kBM - 1) / kBM);
    // a pair walks its items together: the cluster is the unit of the schedule
    const uint32_t rank = P ? cluster_ctarank() : 0;
    const bool leader = rank == 0;
    const int cta = P ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int G = P ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    const uint64_t deadline = globaltimer_ns() + a.timeout_ns;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
            mbar_init(&bar_s[i], 1);
            // one arrival per softmax warp (of both CTAs on a pair, at the even CTA)
            mbar_init(&bar_p[i], (P ? 2 : 1) * kSoftmaxThreads / 32);
        }
        for (int q = 0; q < 4; ++q) mbar_init(&bar_x[q], 2);  // one arrival per warp
        mbar_init(bar_o, 1);
        mbar_init(o_full, 1);
        mbar_init(bar_done, 1);
        mbar_init(epi_done, kSoftmaxThreads / 32);  // one arrival per softmax warp
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == kMmaWarp) {  // whole warp: allocate tensor memory (both CTAs of a pair)
        if constexpr (P) {
            tmem_alloc_pair(tmem_slot, C::kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, C::kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    if constexpr (P)
        cluster_sync_all();  // the peer's barriers are initialised before any remote signal
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // waits on barriers the peer CTA (or the pair's MMAs) also signals
    auto wait_bar = [&](uint64_t *bar, uint32_t parity) {
        if constexpr (P)
            return mbar_wait_bounded_cluster(bar, parity, abort_flag, deadline);
        else
            return mbar_wait_bounded(bar, parity, abort_flag, deadline);
    };

    if (warp == kKProducerWarp || warp == kVProducerWarp) {
        // ------------------------------------------------------------ TMA producers
        // warp 8 loads each item's Q, then its K tiles; warp 9 loads its V tiles (this
        // item's O columns).  The rings run on across items.  One mbarrier per tile
        // carries all of the tile's chunk copies.  On a pair, both CTAs' copies of a tile
        // count on the even CTA's barrier, which that CTA arms for both.
        if (lane == 0) {
            const bool is_k = warp == kKProducerWarp;
            const int stages = is_k ? C::kKStages : C::kVStages;
            const int tile_bytes = is_k ? C::kKTileBytes : C::kVTileBytes;
            const int chunk_bytes = is_k ? C::kKChunkBytes : C::kVChunkBytes;
            const int chunks = is_k ? C::kQkChunks : C::kVChunks;
            const int arm = P ? 2 : 1;  // CTAs whose copies a barrier counts
            unsigned char *ring = is_k ? sK : sV;
            uint64_t *full = is_k ? k_full : v_full;
            uint64_t *empty = is_k ? k_empty : v_empty;
            const CUtensorMap *tm = is_k ? &a.tm_k : &a.tm_v;
            tma_prefetch_desc(tm);
            if (is_k) tma_prefetch_desc(&a.tm_q);
            int g = 0, qi = 0;  // tiles and query tiles issued
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int idx = item_index(k, cta, G, n_items);
                if (idx < 0) break;
                const Item it = item_at<D, W, P>(a, idx, rank);
                // the V slot held the previous item's output boxes until their stores read them
                if (C::kEpiInV && !is_k && k > 0 &&
                    !mbar_wait_bounded(epi_done, (k - 1) & 1, abort_flag, deadline)) {
                    ok = false;
                    break;
                }
                if (is_k) {
                    const int qs = qi % C::kQStages;
                    if (!wait_bar(&q_empty[qs], ((qi / C::kQStages) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(&q_full[qs], arm * C::kQBytes);
                    if constexpr (P) {  // the whole query tile in one copy
                        tma_load_5d_pair(sQ + qs * C::kQBytes, &a.tm_q,
                                         cluster_addr(&q_full[qs], 0), 0, it.m0, 0, it.h, it.b);
                    } else if (a.chunked) {
                        tma_load_5d(sQ + qs * C::kQBytes, &a.tm_q, &q_full[qs], 0, it.m0, 0,
                                    it.h, it.b);
                    } else {
                        for (int c = 0; c < C::kQkChunks; ++c)
                            tma_load_4d(sQ + qs * C::kQBytes + c * kBM * 128, &a.tm_q,
                                        &q_full[qs], c * kChunkCols, it.h, it.m0, it.b);
                    }
                    ++qi;
                }
                // K: this CTA's rows of the tile (all of them, or its half on a pair); V: its
                // columns of the item's O columns
                const int col0 = is_k ? 0 : it.half * C::kOCols + (int)rank * C::kVCols;
                const int row_off = is_k ? (int)rank * C::kKRows : 0;
                for (int t = it.band.t_begin; t < it.band.t_end; ++t, ++g) {
                    const int s = g % stages;
                    if (!wait_bar(&empty[s], ((g / stages) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    if (is_k && a.test_skip_kv_load && g == 0) continue;  // test hook: never load
                    if (leader) mbar_arrive_expect_tx(&full[s], arm * tile_bytes);
                    if constexpr (P) {  // this CTA's part of the tile in one copy
                        tma_load_5d_pair(ring + s * tile_bytes, tm, cluster_addr(&full[s], 0), 0,
                                         t * BN + row_off, col0 / kChunkCols, it.hk, it.b);
                    } else if (a.chunked) {
                        tma_load_5d(ring + s * tile_bytes, tm, &full[s], 0, t * BN + row_off,
                                    col0 / kChunkCols, it.hk, it.b);
                    } else {
                        for (int c = 0; c < chunks; ++c)
                            tma_load_4d(ring + s * tile_bytes + c * chunk_bytes, tm, &full[s],
                                        col0 + c * kChunkCols, it.hk, t * BN + row_off, it.b);
                    }
                }
            }
            // drain: every issued copy must land before the CTA may exit.  Fills go round
            // each ring in order, so slot s last held fill s + j*stages, the largest below
            // the count issued.  On a pair the even CTA's barriers count both CTAs' copies,
            // and the odd CTA stays at the closing cluster barrier until the even one
            // has drained.
            const uint64_t drain_deadline = globaltimer_ns() + 100000000ull;
            volatile int no_abort = 0;
            if (leader) {
                for (int s = 0; s < stages; ++s)
                    if (s < g) {
                        const int last = s + (g - 1 - s) / stages * stages;
                        if (!(is_k && a.test_skip_kv_load && last == 0))
                            mbar_wait_bounded(&full[s], (last / stages) & 1, &no_abort,
                                              drain_deadline);
                    }
                if (is_k)
                    for (int s = 0; s < C::kQStages; ++s)
                        if (s < qi) {
                            const int last = s + (qi - 1 - s) / C::kQStages * C::kQStages;
                            mbar_wait_bounded(&q_full[s], (last / C::kQStages) & 1, &no_abort,
                                              drain_deadline);
                        }
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // (on a pair, the even CTA's warp issues for both; the odd CTA's warp only waits
        // for the last MMA before the tensor memory is freed)
        if (lane == 0 && leader) {
            constexpr int kM = P ? 2 * kBM : kBM;
            constexpr uint32_t idesc_s = instr_desc(kM, BN, false);
            constexpr uint32_t idesc_pv = instr_desc(kM, P ? 2 * C::kVCols : C::kOCols, true);
            auto mma_ss = [&](uint32_t d, uint64_t ad, uint64_t bd, uint32_t id, uint32_t acc) {
                if constexpr (P) tc_mma_ss_pair(d, ad, bd, id, acc);
                else tc_mma_ss(d, ad, bd, id, acc);
            };
            auto mma_ts = [&](uint32_t d, uint32_t at, uint64_t bd, uint32_t id, uint32_t acc) {
                if constexpr (P) tc_mma_ts_pair(d, at, bd, id, acc);
                else tc_mma_ts(d, at, bd, id, acc);
            };
            auto commit = [&](uint64_t *bar) {
                if constexpr (P) tc_commit_pair(bar);
                else tc_commit(bar);
            };
            // Descriptors are built once; advancing an operand by B bytes adds B >> 4 to
            // the start-address field (all smem addresses here are below 256 KB, so the
            // 14-bit field never carries), which keeps the issue loop to a few
            // instructions per MMA.
            const uint64_t dq0 = sw128_desc(smem_u32(sQ));
            const uint64_t dk0 = sw128_desc(smem_u32(sK));
            bool ok = true;
            int g = 0;  // global tile index: S buffer g % 2, ring slots, barrier phases
            for (int k = 0, qi = 0; ok; ++k, ++qi) {
                const int idx = item_index(k, cta, G, n_items);
                if (idx < 0) break;
                const Item it = item_at<D, W, P>(a, idx, rank);
                const int n_tiles = it.band.t_end - it.band.t_begin;
                const int qs = qi % C::kQStages;
                if (!wait_bar(&q_full[qs], (qi / C::kQStages) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t dq = dq0 + (uint64_t)((qs * C::kQBytes) >> 4);
                for (int t = 0; t <= n_tiles && ok; ++t) {
                    if (t < n_tiles) {
                        // S(g+t) = Q K^T into S buffer (g+t) % 2
                        const int gt = g + t;
                        const int s = gt % C::kKStages;
                        if (!wait_bar(&k_full[s], (gt / C::kKStages) & 1)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d_s = tmem + C::kTmemS + (uint32_t)((gt & 1) * BN);
                        const uint64_t dk = dk0 + (uint64_t)((s * C::kKTileBytes) >> 4);
#pragma unroll
                        for (int c = 0; c < C::kQkChunks; ++c) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                if (c * 4 + kk < C::kKSteps)
                                    mma_ss(d_s, dq + (uint64_t)((c * kBM * 128 + kk * 32) >> 4),
                                           dk + (uint64_t)((c * C::kKChunkBytes + kk * 32) >> 4),
                                           idesc_s, (c > 0 || kk > 0) ? 1u : 0u);
                            }
                        }
                        commit(&k_empty[s]);
                        commit(&bar_s[gt & 1]);
                        if (t == n_tiles - 1) commit(&q_empty[qs]);  // Q read for the last time
                    }
                    if (t > 0) {
                        // O += P V for tile g+t-1: A = P from tensor memory (the S buffer it
                        // was computed from, 8 columns per 16 keys), B = V MN-major with its
                        // 64-column atoms kVChunkBytes apart, N = every O column of the item.
                        // The first group overwrites O: the previous item's epilogue read it
                        // before its softmax published this item's first P.
                        const int gp = g + t - 1;
                        const int s = gp % C::kVStages;
                        if (!wait_bar(&bar_p[gp & 1], (gp >> 1) & 1) ||
                            !wait_bar(&v_full[s], (gp / C::kVStages) & 1)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t dv = sw128_desc_mn(smem_u32(sV) + s * C::kVTileBytes,
                                                          C::kVChunkBytes);
                        const uint32_t p_tmem = tmem + C::kTmemS + (uint32_t)((gp & 1) * BN);
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk)
                            mma_ts(tmem + kTmemO, p_tmem + kk * 8, dv + (uint64_t)((kk * 2048) >> 4),
                                   idesc_pv, (t > 1 || kk > 0) ? 1u : 0u);
                        commit(&v_empty[s]);
                        commit(bar_o);
                    }
                }
                if (!ok) break;
                if (n_tiles == 0) commit(&q_empty[qs]);  // nothing read this Q
                commit(o_full);  // the item's O is complete once every MMA above is
                g += n_tiles;
            }
            // drain: all issued MMAs must finish before tensor memory is freed
            commit(bar_done);
            volatile int no_abort = 0;
            mbar_wait_bounded(bar_done, 0, &no_abort, globaltimer_ns() + 100000000ull);
        } else if (P && lane == 0) {
            // the odd CTA of a pair: its tensor memory is written by the pair's MMAs
            volatile int no_abort = 0;
            mbar_wait_bounded_cluster(bar_done, 0, &no_abort, deadline + 100000000ull);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax warps
        // Two warpgroups share every row: warp w and warp w+4 read the same TMEM lane
        // quarter; warpgroup g owns S columns [g*BN/2, (g+1)*BN/2) of each tile and O
        // column chunks k (16 wide) with k % 2 == g.  Their partial row maxima meet in
        // shared memory once per tile (an mbarrier per lane quarter, double-buffered).
        constexpr int HC = BN / 2;                    // S columns per thread
        const int wg = warp >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;          // query row in the tile = TMEM lane
        const int col0 = wg * HC;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        const bool capped = a.cap_log2 > 0.f;
        const float sl2 = capped ? 1.f : a.scale_log2;  // capped scores arrive pre-scaled
        const bool max_mode = sl2 >= 0.f;             // a negative scale flips max and min
        const float hide = max_mode ? -INFINITY : INFINITY;  // raw value that never wins
        // P(g) ready: this CTA's barrier, or on a pair the even CTA's (which issues P.V)
        const uint32_t bar_p_pair[2] = {P ? cluster_addr(&bar_p[0], 0) : 0u,
                                        P ? cluster_addr(&bar_p[1], 0) : 0u};
        bool ok = true;
        int xn = 0;  // exchanges done (selects the exchange buffer and barrier phase)
        // tcgen05.ld/st are warp-collective, so a wait's outcome is made warp-uniform
        auto wait_warp = [&](uint64_t *bar, uint32_t parity) {
            const bool r = wait_bar(bar, parity);
            return __all_sync(0xffffffffu, r) != 0;
        };
        // publish v for the partner warp and read the partner's value (the warp barrier
        // orders every lane's store before lane 0's arrival, whose release makes them
        // visible to the partner warp's acquire)
        auto exchange = [&](float v, float &other) {
            const int n = xn++;
            xchg[((n & 1) * 2 + wg) * kBM + row] = v;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_x[quarter]);
            if (!wait_warp(&bar_x[quarter], n & 1)) return false;
            other = xchg[((n & 1) * 2 + (wg ^ 1)) * kBM + row];
            return true;
        };
        int g = 0;  // global tile index
        for (int k = 0; ok; ++k) {
            const int idx = item_index(k, cta, G, n_items);
            if (idx < 0) break;
            const Item it = item_at<D, W, P>(a, idx, rank);
            const int n_tiles = it.band.t_end - it.band.t_begin;
            const int i = it.m0 + row;                       // query row within the sequence
            const int p = i + (a.kv_len - a.seq_len);        // its absolute position
            const int p_min = it.m0 + (a.kv_len - a.seq_len);
            float m_ref = -INFINITY;  // reference maximum (log2 domain, scaled)
            float l_part = 0.f;       // this warpgroup's share of the row sum
            for (int t = 0; t < n_tiles; ++t) {
                const int gt = g + t;
                if (!wait_warp(&bar_s[gt & 1], (gt >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                float sv[HC];
#pragma unroll
                for (int c = 0; c < HC; c += 16)
                    tmem_ld16(lane_base + C::kTmemS + (gt & 1) * BN + col0 + c,
                              reinterpret_cast<uint32_t *>(sv + c));
                tc_wait_ld();
                if (capped) {  // Gemma 2 score cap, in the log2 domain
                    const float k2 = a.raw_over_cap * kTwoLog2e;
#pragma unroll
                    for (int c = 0; c < HC; ++c) sv[c] = capped_score_log2(sv[c], k2, a.cap_log2);
                }

                const int key0 = (it.band.t_begin + t) * BN;
                const bool need_mask = (key0 + BN > a.kv_len) || (a.causal && key0 + BN - 1 > p_min) ||
                                       (a.window > 0 && key0 < p_min + it.rows - 1 - a.window + 1);
                // visible columns of this thread's half: [vlo, vhi)
                int vlo = 0, vhi = HC;
                if (need_mask) {
                    const int kc0 = key0 + col0;
                    int jhi = a.kv_len;
                    if (a.causal) jhi = min(jhi, p + 1);
                    vhi = max(0, min(HC, jhi - kc0));
                    if (a.window > 0) vlo = min(HC, max(0, p - a.window + 1 - kc0));
#pragma unroll
                    for (int c = 0; c < HC; ++c)
                        if (c < vlo || c >= vhi) sv[c] = hide;
                }
                float e[4] = {hide, hide, hide, hide};
                if (max_mode) {
#pragma unroll
                    for (int c = 0; c < HC; ++c) e[c & 3] = fmaxf(e[c & 3], sv[c]);
                } else {
#pragma unroll
                    for (int c = 0; c < HC; ++c) e[c & 3] = fminf(e[c & 3], sv[c]);
                }
                const float ext = max_mode ? fmaxf(fmaxf(e[0], e[1]), fmaxf(e[2], e[3]))
                                           : fminf(fminf(e[0], e[1]), fminf(e[2], e[3]));
                const float mx_part = vhi > vlo ? ext * sl2 : -INFINITY;
                float mx_other;
                if (!exchange(mx_part, mx_other)) { ok = false; break; }
                const float mx = fmaxf(mx_part, mx_other);

                // refresh the reference maximum only when it grew by more than the threshold
                const bool refresh = mx > m_ref + kRescaleThreshold;
                const float m_new = refresh ? mx : m_ref;
                const float m_use = m_new == -INFINITY ? 0.f : m_new;  // no key seen yet
                float rs[4] = {0.f, 0.f, 0.f, 0.f};
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < HC; ++c) {
                        const float w = fast_exp2(fmaf(sv[c], sl2, -m_use));
                        sv[c] = (c >= vlo && c < vhi) ? w : 0.f;
                        rs[c & 3] += sv[c];
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < HC; ++c) {
                        sv[c] = fast_exp2(fmaf(sv[c], sl2, -m_use));
                        rs[c & 3] += sv[c];
                    }
                }
                const float corr = refresh ? fast_exp2(m_ref - m_use) : 1.f;  // 0 when m_ref = -inf

                // this half of P (bf16 pairs) into the S buffer it came from: both
                // warpgroups have read their S columns (the exchange above orders that),
                // and P sits where its P.V MMA will read it
                {
                    const uint32_t pcol = lane_base + C::kTmemS + (gt & 1) * BN + col0 / 2;
#pragma unroll
                    for (int c = 0; c < HC / 2; c += 8) {
                        uint32_t pk[8];
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            pk[kk] = pack_bf16x2(sv[2 * (c + kk)], sv[2 * (c + kk) + 1]);
                        tmem_st8(pcol + c, pk);
                    }
                }
                // rescale this warpgroup's O chunks when any row of the warp refreshed; O
                // is stable once the previous tile's P.V completes (the S commit of this
                // tile already covered the one before, so that is the next phase of bar_o)
                if (t > 0 && __any_sync(0xffffffffu, refresh)) {
                    if (!wait_warp(bar_o, (gt - 1) & 1)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 16 * wg; c < C::kOCols; c += 32) {
                        uint32_t ov[16];
                        tmem_ld16(lane_base + kTmemO + c, ov);
                        tc_wait_ld();
#pragma unroll
                        for (int kk = 0; kk < 16; ++kk)
                            ov[kk] = __float_as_uint(__uint_as_float(ov[kk]) * corr);
                        tmem_st16(lane_base + kTmemO + c, ov);
                    }
                }
                tc_wait_st();
                l_part = l_part * corr + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
                m_ref = m_new;
                // P(g) is published once per warp: every lane's tensor-memory stores are
                // complete (wait::st) and fenced before the warp barrier, then lane 0 arrives
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (P)
                        mbar_arrive_cluster(bar_p_pair[gt & 1]);
                    else
                        mbar_arrive(&bar_p[gt & 1]);
                }
            }
            if (!ok) break;
            g += n_tiles;
            // ---- epilogue of the item: O / l -> bf16 rows, lse ---------------------------
            if (!wait_warp(o_full, k & 1)) { ok = false; break; }
            tc_fence_after();
            float l_other = 0.f;
            if (!exchange(l_part, l_other)) { ok = false; break; }
            const float l_sum = l_part + l_other;
            const bool live = row < it.rows;  // rows past the sequence end are not stored
            const int64_t qrow = (int64_t)it.b * a.seq_len + i;
            __nv_bfloat16 *orow = a.out + qrow * a.out_rs + (int64_t)it.h * D + it.half * C::kOCols;
            const bool empty = !(l_sum > 0.f);
            const float inv_l = empty ? 0.f : 1.f / l_sum;
            if constexpr (C::kEpiTma) {
                // warpgroup wg takes O columns [wg, wg + 1) * kOCols / 2, one box of
                // kEpiCols per pass: lane r writes row r of the box (16-byte pieces placed
                // by the swizzle the map expects), then lane 0 stores the box.  Rows past
                // the sequence end fall outside the map and are not written.
                constexpr uint32_t kRowBytes = C::kEpiCols * 2;   // bytes per box row
                constexpr uint32_t kSwMask = kRowBytes / 16 - 1;  // the swizzle of that width
                unsigned char *boxes = sStage + warp * C::kEpiBufs * C::kEpiBoxBytes;
                const uint32_t row_off = (uint32_t)lane * kRowBytes;
                const uint32_t sw = (row_off >> 7) & kSwMask;
#pragma unroll 1
                for (int ps = 0; ps < C::kEpiPasses; ++ps) {
                    unsigned char *box = boxes + (ps % C::kEpiBufs) * C::kEpiBoxBytes;
                    const uint32_t my_row = smem_u32(box) + row_off;
                    const int c0 = wg * (C::kOCols / 2) + ps * C::kEpiCols;  // O column
                    uint32_t pk[C::kEpiCols / 2];
                    if (n_tiles > 0) {
                        uint32_t ov[C::kEpiCols];
#pragma unroll
                        for (int c = 0; c < C::kEpiCols; c += 16)
                            tmem_ld16(lane_base + kTmemO + c0 + c, ov + c);  // warp-wide
                        tc_wait_ld();
#pragma unroll
                        for (int kk = 0; kk < C::kEpiCols / 2; ++kk)
                            pk[kk] = pack_bf16x2(__uint_as_float(ov[2 * kk]) * inv_l,
                                                 __uint_as_float(ov[2 * kk + 1]) * inv_l);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < C::kEpiCols / 2; ++kk) pk[kk] = 0u;
                    }
                    if (lane == 0) bulk_wait_read<C::kEpiBufs - 1>();  // the box is free again
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < (int)(kRowBytes / 16); ++j)
                        st_shared_v4(my_row + (((uint32_t)j ^ sw) << 4), pk[4 * j],
                                     pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    fence_proxy_async_smem();  // the generic writes before the async read
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&a.tm_out, box, it.h * D + it.half * C::kOCols + c0,
                                     it.m0 + quarter * 32, it.b);
                        bulk_commit_group();
                    }
                }
                // hand the V slot back once the boxes are read.  Every item visits at least
                // one key tile (kv_len >= seq_len), so the V producer, which waits for each
                // item's boxes before the next item's first V copy, never falls two phases
                // behind this barrier.
                if constexpr (C::kEpiInV) {
                    if (lane == 0) {
                        bulk_wait_read<0>();
                        mbar_arrive(epi_done);
                    }
                }
            } else if (n_tiles > 0) {
#pragma unroll 1
                for (int c = 16 * wg; c < C::kOCols; c += 32) {
                    uint32_t ov[16];
                    tmem_ld16(lane_base + kTmemO + c, ov);  // warp-wide: every lane takes part
                    tc_wait_ld();
                    uint32_t pk[8];
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        pk[kk] = pack_bf16x2(__uint_as_float(ov[2 * kk]) * inv_l,
                                             __uint_as_float(ov[2 * kk + 1]) * inv_l);
                    if (live) {
                        if (a.out_v8) {
                            st_global_v8(orow + c, pk);
                        } else {
                            uint4 *dst = reinterpret_cast<uint4 *>(orow + c);
                            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                        }
                    }
                }
            } else if (live) {
                for (int c = 16 * wg; c < C::kOCols; c += 32)
                    for (int kk = 0; kk < 16; ++kk) orow[c + kk] = __float2bfloat16_rn(0.f);
            }
            if (live && wg == 0 && a.lse != nullptr && it.half == 0)
                a.lse[qrow * a.n_heads + it.h] =
                    empty ? -INFINITY : (m_ref + log2f(l_sum)) * 0.69314718055994531f;
            // the O reads above complete before this thread's next P is published, and the
            // next item's first P.V (which overwrites O) waits for that P
        }
        if constexpr (C::kEpiTma) {
            if (lane == 0) bulk_wait_all();  // output stores done before shared memory goes
        }
    }

    tc_fence_before();
    if constexpr (P)
        cluster_sync_all();  // neither CTA leaves while the pair's MMAs or copies may touch it
    else
        __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) report_status(a.status, kErrTimeout);
    if (warp == kMmaWarp) {
        tc_fence_after();
        if constexpr (P)
            tmem_dealloc_pair(tmem, C::kTmemCols);
        else
            tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool W = false>
cudaError_t launch_d(const PrefillTcArgs &a, int num_sms, cudaStream_t s) {
    using C = TcCfg<D, W>;
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D, W, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    const int64_t n_items = (int64_t)a.batch * a.n_heads * C::kSplitO * ((a.seq_len + kBM - 1) / kBM);
    const int grid = (int)std::min<int64_t>(n_items, std::max(1, num_sms) * C::kCtasPerSm);
    prefill_tc_kernel<D, W, false><<<grid, kThreads, C::kSmem, s>>>(a);
    return cudaGetLastError();
}

// The CTA-pair form: a persistent grid of as many 2-CTA clusters as fit the GPU at once
// (one per TPC whose two SMs are both available), capped by the number of items.
cudaError_t launch_pair_512(const PrefillTcArgs &a, cudaStream_t s) {
    using C = TcCfg<512, false, true>;
    auto kern = prefill_tc_kernel<512, false, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    static int clusters_per_dev[64] = {};  // co-resident clusters, asked once per device
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (clusters_per_dev[dev] == 0) {
        int sms = 0, n = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        cfg.gridDim = dim3(2 * (sms / 2));
        if ((e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg)) != cudaSuccess) return e;
        clusters_per_dev[dev] = std::max(1, n);
    }
    const int64_t n_items = (int64_t)a.batch * (a.n_heads / 2) * C::kSplitO *
                            ((a.seq_len + kBM - 1) / kBM);
    const int clusters = (int)std::min<int64_t>(n_items, clusters_per_dev[dev]);
    cfg.gridDim = dim3(2 * clusters);
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool prefill_tc_wide(int head_dim, int seq_len, int kv_len, int causal, int window) {
    if (head_dim != 64) return false;
    // mean keys a query tile visits (bottom-right causal alignment, window cap)
    double keys = causal ? (kv_len - seq_len) + seq_len / 2.0 + kBM / 2.0 : (double)kv_len;
    if (window > 0) keys = std::min(keys, (double)window + kBM);
    return keys >= 1024.0;
}

bool prefill_tc_pair(int head_dim, int n_heads, int n_kv_heads) {
    return head_dim == 512 && (n_heads / n_kv_heads) % 2 == 0;
}

int prefill_tc_block_n(int head_dim, bool wide) {
    switch (head_dim) {
        case 64: return wide ? TcCfg<64, true>::kBN : TcCfg<64>::kBN;
        case 80: return TcCfg<80>::kBN;
        case 128: return TcCfg<128>::kBN;
        case 256: return TcCfg<256>::kBN;
        case 512: return TcCfg<512>::kBN;
        default: return 0;
    }
}

int prefill_tc_box_rows(int head_dim, bool wide, bool pair, bool v) {
    if (pair) return v ? TcCfg<512, false, true>::kBN : TcCfg<512, false, true>::kKRows;
    return prefill_tc_block_n(head_dim, wide);
}

int prefill_tc_out_box_cols(int head_dim, bool pair) {
    if (pair) return TcCfg<512, false, true>::kEpiCols;
    switch (head_dim) {
        case 128: return TcCfg<128>::kEpiCols;
        case 256: return TcCfg<256>::kEpiCols;
        default: return 0;
    }
}

bool prefill_tc_chunked(int head_dim, bool pair) {
    return pair || head_dim == 128 || head_dim == 256 || head_dim == 512;
}

int prefill_tc_v_chunks(int head_dim, bool pair) {
    if (pair) return TcCfg<512, false, true>::kVChunks;
    switch (head_dim) {
        case 128: return TcCfg<128>::kVChunks;
        case 256: return TcCfg<256>::kVChunks;
        case 512: return TcCfg<512>::kVChunks;
        default: return 0;
    }
}

int64_t prefill_tc_items(int batch, int n_heads, int head_dim, int seq_len) {
    const int split = head_dim == 512 ? TcCfg<512>::kSplitO : 1;
    return (int64_t)batch * n_heads * split * ((seq_len + kBM - 1) / kBM);
}

cudaError_t launch_prefill_tc(const PrefillTcArgs &a, int num_sms, cudaStream_t s) {
    if (a.seq_len == 0 || a.batch == 0) return cudaSuccess;
    if (prefill_tc_items(a.batch, a.n_heads, a.head_dim, a.seq_len) > kPrefillMaxItems)
        return cudaErrorInvalidValue;
    if (a.pair) {
        if (!prefill_tc_pair(a.head_dim, a.n_heads, a.n_kv_heads)) return cudaErrorInvalidValue;
        return launch_pair_512(a, s);
    }
    switch (a.head_dim) {
        case 64: return a.wide ? launch_d<64, true>(a, num_sms, s) : launch_d<64>(a, num_sms, s);
        case 80: return launch_d<80>(a, num_sms, s);
        case 128: return launch_d<128>(a, num_sms, s);
        case 256: return launch_d<256>(a, num_sms, s);
        case 512: return launch_d<512>(a, num_sms, s);
        default: return cudaErrorInvalidValue;
    }
}

// the score cap alone, for testing it against tanh (grid-stride over n values)
__global__ void capped_scores_kernel(const float *raw, int64_t n, float raw_over_cap,
                                     float cap_log2, float *out) {
    const float k2 = raw_over_cap * kTwoLog2e;  // formed as the attention kernels form it
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = capped_score_log2(raw[i], k2, cap_log2);
}

cudaError_t launch_capped_scores(const float *raw, int64_t n, float raw_over_cap,
                                 float cap_log2, float *out, cudaStream_t s) {
    const int64_t blocks = (n + 255) / 256;
    capped_scores_kernel<<<(int)(blocks < 1184 ? blocks : 1184), 256, 0, s>>>(
        raw, n, raw_over_cap, cap_log2, out);
    return cudaGetLastError();
}

}  // namespace lat
