// row_attention_f32.cu — exact-fp32 attention on the CUDA cores, one CTA of four warps
// per (query row, query head).  Serves every LAT_F32 call (prefill and decode).
//
// The arithmetic is the row-wise online softmax of the lattice-inference DESIGN page
// ("Current Design": fused attention, online softmax in registers): keys are visited in
// order, a few at a time; each score s = scale * q.k is reduced across the warp (then
// capped as softcap * tanh(s / softcap) when a cap is set: the larql page, "BLAS-Fused
// Attention", step 2), and for a block of scores s_u the running maximum m, normaliser l
// and output accumulator o are updated as
//   m' = max(m, max_u s_u),  l' = l*e^(m-m') + sum_u e^(s_u-m'),
//   o' = o*e^(m-m') + sum_u e^(s_u-m')*v_u.
// The four warps take interleaved blocks of the row's keys, each keeping its own (m, l, o),
// and meet in shared memory at the end, where the states combine as
//   M = max_w m_w,  l = sum_w l_w e^(m_w - M),  out = sum_w o_w e^(m_w - M) / l,
// so a row waits for a quarter of the memory round trips one warp would.
// fp32 inputs keep fp32 products (no tf32), so the result stays within ~1e-6 of fp64.
// Lane `lane` owns head dimensions d = lane + 32*t, t < NT.
#include <math.h>

#include "device_common.cuh"
#include "kernels.h"

namespace lat {

constexpr int kRowWarps = 4;

template <int NT>
__global__ void __launch_bounds__(32 * kRowWarps) row_attention_f32_kernel(RowAttnArgs a) {
    __shared__ float part_m[kRowWarps], part_l[kRowWarps];
    __shared__ float part_o[kRowWarps][32 * NT];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t unit = blockIdx.x;
    const int h = (int)(unit % a.n_heads);
    const int64_t r = unit / a.n_heads;  // flattened query row b*seq_len + i
    const int b = (int)(r / a.seq_len), i = (int)(r % a.seq_len);
    const int D = a.head_dim;

    int L = a.kv_len;
    if (a.kv_lens != nullptr) {
        L = a.kv_lens[b];
        if (L < 0 || L > a.max_kv_len) {  // the whole CTA leaves
            if (threadIdx.x == 0 && h == 0) report_status(a.status, kErrBounds);
            return;
        }
    }
    const int p = i + (L - a.seq_len);                 // absolute query position
    const int hi = a.causal ? min(L, p + 1) : L;       // causal: keys j <= p
    const int lo = a.window > 0 ? max(0, p - a.window + 1) : 0;  // window: p - j < W
    const int hk = h / (a.n_heads / a.n_kv_heads);

    const float *qrow = a.q + r * a.q_rs + (int64_t)h * D;
    float qv[NT], o[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int d = lane + 32 * t;
        qv[t] = d < D ? qrow[d] : 0.f;
        o[t] = 0.f;
    }
    const float *kb = a.k + (int64_t)b * a.k_seq + (int64_t)hk * a.k_head;
    const float *vb = a.v + (int64_t)b * a.v_seq + (int64_t)hk * a.v_head;
    // Keys are taken KB at a time: the block's K and V rows are loaded together, so the
    // warp waits for one memory round trip per block instead of one per key; the scores
    // of the block then enter the running maximum and sums together.
    constexpr int KB = NT <= 2 ? 8 : (NT <= 4 ? 4 : (NT <= 8 ? 2 : 1));
    float m = -INFINITY, l = 0.f;
    for (int j0 = lo + warp * KB; j0 < hi; j0 += kRowWarps * KB) {
        float kx[KB][NT], vx[KB][NT];
#pragma unroll
        for (int u = 0; u < KB; ++u) {
            const int j = j0 + u;
            const bool live = j < hi;
            const int64_t jr = a.ring > 0 ? j % a.ring : j;  // ring cache slot
            const float *kr = kb + jr * a.k_row;
            const float *vr = vb + jr * a.v_row;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const int d = lane + 32 * t;
                kx[u][t] = (live && d < D) ? kr[d] : 0.f;
                vx[u][t] = (live && d < D) ? vr[d] : 0.f;
            }
        }
        float sc[KB];
#pragma unroll
        for (int u = 0; u < KB; ++u) {
            float part = 0.f;
#pragma unroll
            for (int t = 0; t < NT; ++t) part = fmaf(qv[t], kx[u][t], part);
            sc[u] = part;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int u = 0; u < KB; ++u) sc[u] += __shfl_xor_sync(0xffffffffu, sc[u], off);
        float mb = -INFINITY;
#pragma unroll
        for (int u = 0; u < KB; ++u) {
            float x = sc[u] * a.scale;
            if (a.softcap > 0.f) x = a.softcap * tanhf(x / a.softcap);  // Gemma 2 score cap
            sc[u] = j0 + u < hi ? x : -INFINITY;
            mb = fmaxf(mb, sc[u]);
        }
        const float m_new = fmaxf(m, mb);  // finite: key j0 is visible
        const float corr = expf(m - m_new);
        l *= corr;
#pragma unroll
        for (int t = 0; t < NT; ++t) o[t] *= corr;
#pragma unroll
        for (int u = 0; u < KB; ++u) {
            const float w = expf(sc[u] - m_new);  // 0 for keys past the end
            l += w;
#pragma unroll
            for (int t = 0; t < NT; ++t) o[t] = fmaf(w, vx[u][t], o[t]);
        }
        m = m_new;
    }
    // the four warps' states meet in shared memory; warp 0 combines and writes the row
#pragma unroll
    for (int t = 0; t < NT; ++t) part_o[warp][lane + 32 * t] = o[t];
    if (lane == 0) {
        part_m[warp] = m;
        part_l[warp] = l;
    }
    __syncthreads();
    if (warp != 0) return;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kRowWarps; ++w) M = fmaxf(M, part_m[w]);
    const bool empty = !(M > -INFINITY);  // no visible key
    float f[kRowWarps], lt = 0.f;
#pragma unroll
    for (int w = 0; w < kRowWarps; ++w) {
        f[w] = empty ? 0.f : expf(part_m[w] - M);  // 0 for a warp that saw no key
        lt += part_l[w] * f[w];
    }
    const float inv_l = empty ? 0.f : 1.f / lt;
    float *orow = a.out + r * a.out_rs + (int64_t)h * D;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int d = lane + 32 * t;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kRowWarps; ++w) acc = fmaf(part_o[w][d], f[w], acc);
        if (d < D) orow[d] = acc * inv_l;
    }
    if (a.lse != nullptr && lane == 0)
        a.lse[r * a.n_heads + h] = empty ? -INFINITY : M + logf(lt);
}

cudaError_t launch_row_attention_f32(const RowAttnArgs &a, cudaStream_t s) {
    const int64_t n_units = (int64_t)a.batch * a.seq_len * a.n_heads;
    if (n_units == 0) return cudaSuccess;
    const int64_t blocks = n_units;  // one CTA per (row, head)
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    constexpr int kT = 32 * kRowWarps;
    switch (a.head_dim) {
        case 64: row_attention_f32_kernel<2><<<(unsigned)blocks, kT, 0, s>>>(a); break;
        case 80: row_attention_f32_kernel<3><<<(unsigned)blocks, kT, 0, s>>>(a); break;
        case 128: row_attention_f32_kernel<4><<<(unsigned)blocks, kT, 0, s>>>(a); break;
        case 256: row_attention_f32_kernel<8><<<(unsigned)blocks, kT, 0, s>>>(a); break;
        case 512: row_attention_f32_kernel<16><<<(unsigned)blocks, kT, 0, s>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace lat
