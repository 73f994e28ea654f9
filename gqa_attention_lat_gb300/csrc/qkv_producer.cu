// qkv_producer.cu — the steps right before attention, fused: Q/K RMS norm, rotary position
// embedding, V (unit norm or copy), and the KV-cache append.
//
// What it computes, for new row t of sequence b at absolute position p = pos[b] + t
// (the hf2q "Current Inference Path" page, section 3: Q norm and K norm (RmsNorm), V unit
// norm, RoPE apply, KV cache append; the lattice-inference DESIGN page's
// fused_qk_norm_rope: one RMS norm over head_dim, then head_dim/2 rotation pairs):
//   Q and K heads:  y = x / sqrt(mean(x^2) + eps) * w        (w the head-dim norm weight)
//                   element i < D/2 pairs with i + D/2 and both rotate by
//                   theta_i = p * base^(-2i/D)  (the neox pairing the hf2q page names)
//   V heads:        copied, or x / sqrt(mean(x^2) + eps) when unit-normed (Gemma 4)
// Q goes to q_out (the attention input); K and V go to cache row p.
//
// How: one CTA per new row, in two forms (a vectorised one for head_dim 64/128/256 with
// 16-byte aligned rows and strides, and a general one).  The row's threads turn its
// position into cos/sin of every rotation angle, in shared memory: p * base^(-2i/D) is
// formed in double precision (the host passes the inverse frequencies in double) and
// reduced by 2*pi there, so the fp32 sine and cosine see an argument below pi even at
// positions in the hundreds of thousands.  The general form then takes one head per warp
// at a time (a warp-shuffle sum of squares, the scaled head staged in shared memory, each
// lane writing the rotated elements it owns); the vectorised form is described at its
// kernel.  fp32 arithmetic throughout, one rounding to the output type.
#include <math.h>

#include <algorithm>

#include "device_common.cuh"
#include "kernels.h"

namespace lat {

namespace {

constexpr int kWarps = 4;
constexpr double kTwoPi = 6.283185307179586;

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) qkv_producer_kernel(const __grid_constant__ ProducerArgs a) {
    extern __shared__ float smem[];
    const int D = a.head_dim, half = D / 2;
    float *cs = smem;                 // [half] cos
    float *sn = smem + half;          // [half] sin
    float *stage = smem + 2 * half;   // [kWarps][D] normed rows
    const int row = blockIdx.x;
    const int b = row / a.n_new, t = row % a.n_new;
    const int p0 = a.pos[b];
    // a sequence whose rows fall outside the cache is skipped whole (every CTA of the
    // sequence sees the same pos[b]), like the plain append
    if (p0 < 0 || (int64_t)p0 + a.n_new > (int64_t)a.capacity) {
        if (t == 0 && threadIdx.x == 0) report_status(a.status, kErrBounds);
        return;
    }
    const int p = p0 + t;
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        double th = (double)p * a.inv_freq[i];
        th -= rint(th * (1.0 / kTwoPi)) * kTwoPi;
        float s, c;
        sincosf((float)th, &s, &c);
        cs[i] = c;
        sn[i] = s;
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *st = stage + warp * D;
    const T *src_row = static_cast<const T *>(a.qkv) + ((int64_t)b * a.n_new + t) * a.qkv_rs;
    const int n_q = a.n_heads, n_k = a.n_kv_heads;
    const int total = n_q + 2 * n_k;
    for (int hh = warp; hh < total; hh += kWarps) {
        const T *x = src_row + (int64_t)hh * D;
        const bool is_q = hh < n_q, is_k = !is_q && hh < n_q + n_k, is_v = hh >= n_q + n_k;
        float ss = 0.f;
        for (int e = lane; e < D; e += 32) {
            const float v = to_f<T>(x[e]);
            st[e] = v;
            ss = fmaf(v, v, ss);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const bool normed = !is_v || a.v_unit_norm;
        const float r = normed ? 1.f / sqrtf(ss / (float)D + a.eps) : 1.f;
        const T *w = is_q ? static_cast<const T *>(a.q_w) : (is_k ? static_cast<const T *>(a.k_w) : nullptr);
        __syncwarp();
        for (int e = lane; e < D; e += 32) st[e] = st[e] * r * (w != nullptr ? to_f<T>(w[e]) : 1.f);
        __syncwarp();
        T *dst;
        if (is_q) {
            dst = static_cast<T *>(a.q_out) + ((int64_t)b * a.n_new + t) * a.q_out_rs + (int64_t)hh * D;
        } else {
            const int hk = is_k ? hh - n_q : hh - n_q - n_k;
            T *cache = static_cast<T *>(is_k ? a.k_cache : a.v_cache);
            dst = cache + (int64_t)b * a.cache_seq + (int64_t)p * a.cache_rs + (int64_t)hk * a.cache_head;
        }
        if (is_v) {
            for (int e = lane; e < D; e += 32) dst[e] = from_f<T>(st[e]);
        } else {  // rotation pair (i, i + D/2)
            for (int i = lane; i < half; i += 32) {
                const float x0 = st[i], x1 = st[i + half], c = cs[i], sv = sn[i];
                dst[i] = from_f<T>(x0 * c - x1 * sv);
                dst[i + half] = from_f<T>(x0 * sv + x1 * c);
            }
        }
        __syncwarp();  // the stage is rewritten by the next head
    }
}

// 8 consecutive elements from registers, as 16-byte stores
template <typename T>
__device__ __forceinline__ void store8(T *p, const float v[8]);
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16 *p, const float v[8]) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                               pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}
template <>
__device__ __forceinline__ void store8<float>(float *p, const float v[8]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// Vectorised form for head_dim 64/128/256 and 16-byte aligned rows.  A head is D/16
// lanes; lane j holds elements [8j, 8j+8) and their rotation partners [D/2 + 8j,
// D/2 + 8j + 8) as two 16-byte vectors, so the rotation needs no data from other lanes
// and the sum of squares is a shuffle reduction over the head's D/16 lanes.  A warp holds
// 512/D heads; the CTA has just enough warps (up to 8) for one row's heads per pass.
//
// Only the rotation needs the position: the first pass's head rows, norm weights and the
// position are all loaded up front, the norm of the first pass is done before the one
// barrier that publishes the cos/sin table, and the rotation and the stores follow it.
constexpr int kFastMaxWarps = 8;

// 8 elements held as raw 16-byte words until they are needed as floats (fewer registers)
template <typename T>
struct Raw8 {
    static constexpr int kWords = (int)sizeof(T) / 2;  // uint4 words: 1 for bf16, 2 for fp32
    uint4 u[kWords];
    __device__ __forceinline__ void load(const T *p) {
#pragma unroll
        for (int i = 0; i < kWords; ++i) u[i] = reinterpret_cast<const uint4 *>(p)[i];
    }
    __device__ __forceinline__ void fill(uint32_t bits) {
#pragma unroll
        for (int i = 0; i < kWords; ++i) u[i] = make_uint4(bits, bits, bits, bits);
    }
    __device__ __forceinline__ float get(int k) const;
};
template <>
__device__ __forceinline__ float Raw8<__nv_bfloat16>::get(int k) const {
    const uint32_t w = k < 2 ? u[0].x : k < 4 ? u[0].y : k < 6 ? u[0].z : u[0].w;
    return __uint_as_float((k & 1) ? (w & 0xffff0000u) : (w << 16));
}
template <>
__device__ __forceinline__ float Raw8<float>::get(int k) const {
    const uint4 &q = u[k >> 2];
    const int m = k & 3;
    return __uint_as_float(m == 0 ? q.x : m == 1 ? q.y : m == 2 ? q.z : q.w);
}

template <typename T, int D>
struct FastHead {  // one lane's 2 x 8 elements of one head, through norm and rotation
    static constexpr int LPH = D / 16;
    Raw8<T> xlo, xhi, wlo, whi;
    float lo[8], hi[8];

    __device__ __forceinline__ void load(const T *row, const ProducerArgs &a, int hh, int j, bool live,
                                         bool is_q, bool is_k) {
        const T *wp = is_q ? static_cast<const T *>(a.q_w) : (is_k ? static_cast<const T *>(a.k_w) : nullptr);
        const uint32_t one = sizeof(T) == 2 ? 0x3f803f80u : 0x3f800000u;  // 1.0
        xlo.fill(0u), xhi.fill(0u), wlo.fill(one), whi.fill(one);
        if (live) {
            const T *h = row + (int64_t)hh * D + 8 * j;
            xlo.load(h);
            xhi.load(h + D / 2);
        }
        if (live && wp != nullptr) {
            wlo.load(wp + 8 * j);
            whi.load(wp + D / 2 + 8 * j);
        }
    }
    // x <- x / sqrt(mean(x^2) + eps) * w (or x for a V head that is not normed)
    __device__ __forceinline__ void norm(const ProducerArgs &a, bool normed) {
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            lo[k] = xlo.get(k);
            hi[k] = xhi.get(k);
            ss = fmaf(lo[k], lo[k], ss);
            ss = fmaf(hi[k], hi[k], ss);
        }
#pragma unroll
        for (int off = LPH / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float r = normed ? rsqrtf(fmaf(ss, 1.f / (float)D, a.eps)) : 1.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            lo[k] *= r * wlo.get(k);
            hi[k] *= r * whi.get(k);
        }
    }
    // (a, b) -> (a cos - b sin, a sin + b cos) for pair index i0 + k
    __device__ __forceinline__ void rotate(const float *cs, const float *sn, int i0) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float c = cs[i0 + k], s = sn[i0 + k];
            const float a0 = lo[k], b0 = hi[k];
            lo[k] = fmaf(a0, c, -b0 * s);
            hi[k] = fmaf(a0, s, b0 * c);
        }
    }
};

template <typename T, int D>
__global__ void __launch_bounds__(kFastMaxWarps * 32) qkv_producer_fast(const __grid_constant__ ProducerArgs a) {
    constexpr int LPH = D / 16, HPW = 32 / LPH, HALF = D / 2;
    __shared__ float cs[HALF], sn[HALF];
    const int row = blockIdx.x;
    const int b = row / a.n_new, t = row - b * a.n_new;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int sub = lane / LPH, j = lane % LPH;
    const T *src_row = static_cast<const T *>(a.qkv) + (int64_t)row * a.qkv_rs;
    const int n_q = a.n_heads, n_k = a.n_kv_heads, total = n_q + 2 * n_k;
    const int i0 = 8 * j;  // pair index of the lane's first element

    FastHead<T, D> h;
    int hh = warp * HPW + sub;
    bool live = hh < total, is_q = hh < n_q, is_k = !is_q && hh < n_q + n_k;
    h.load(src_row, a, hh, j, live, is_q, is_k);
    const int p0 = a.pos[b];
    h.norm(a, is_q || is_k || a.v_unit_norm);
    const bool skip = p0 < 0 || (int64_t)p0 + a.n_new > (int64_t)a.capacity;  // CTA-uniform
    if (skip) {  // the sequence is skipped whole
        if (t == 0 && threadIdx.x == 0) report_status(a.status, kErrBounds);
        return;
    }
    const int p = p0 + t;
    for (int i = threadIdx.x; i < HALF; i += blockDim.x) {
        double th = (double)p * a.inv_freq[i];
        th -= rint(th * (1.0 / kTwoPi)) * kTwoPi;
        float sv, cv;
        __sincosf((float)th, &sv, &cv);  // |th| <= pi: the hardware form is accurate to ~2^-21
        cs[i] = cv;
        sn[i] = sv;
    }
    __syncthreads();
    for (;;) {  // warp-uniform passes over the row's heads
        if (live) {
            if (is_q || is_k) h.rotate(cs, sn, i0);
            T *dst;
            if (is_q) {
                dst = static_cast<T *>(a.q_out) + (int64_t)row * a.q_out_rs + (int64_t)hh * D;
            } else {
                const int hk = is_k ? hh - n_q : hh - n_q - n_k;
                T *cache = static_cast<T *>(is_k ? a.k_cache : a.v_cache);
                dst = cache + (int64_t)b * a.cache_seq + (int64_t)p * a.cache_rs + (int64_t)hk * a.cache_head;
            }
            store8<T>(dst + 8 * j, h.lo);
            store8<T>(dst + D / 2 + 8 * j, h.hi);
        }
        hh += nwarps * HPW;
        if (hh - sub >= total) break;
        live = hh < total, is_q = hh < n_q, is_k = !is_q && hh < n_q + n_k;
        h.load(src_row, a, hh, j, live, is_q, is_k);
        h.norm(a, is_q || is_k || a.v_unit_norm);
    }
}

template <typename T>
cudaError_t launch_t(const ProducerArgs &a, unsigned blocks, bool vec, cudaStream_t s) {
    if (vec) {
        // warps for one pass over the row's heads (512 / D heads per warp), at most 8
        const int heads = a.n_heads + 2 * a.n_kv_heads, hpw = 512 / a.head_dim;
        const int threads = 32 * std::min(kFastMaxWarps, (heads + hpw - 1) / hpw);
        switch (a.head_dim) {
            case 64: qkv_producer_fast<T, 64><<<blocks, threads, 0, s>>>(a); return cudaGetLastError();
            case 128: qkv_producer_fast<T, 128><<<blocks, threads, 0, s>>>(a); return cudaGetLastError();
            case 256: qkv_producer_fast<T, 256><<<blocks, threads, 0, s>>>(a); return cudaGetLastError();
            default: break;
        }
    }
    const size_t smem = (size_t)(a.head_dim + kWarps * a.head_dim) * sizeof(float);
    qkv_producer_kernel<T><<<blocks, kWarps * 32, smem, s>>>(a);
    return cudaGetLastError();
}

bool aligned16_all(const ProducerArgs &a, int64_t es) {
    auto ok = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    return ok(a.qkv) && ok(a.q_out) && ok(a.k_cache) && ok(a.v_cache) &&
           (a.q_w == nullptr || ok(a.q_w)) && (a.k_w == nullptr || ok(a.k_w)) &&
           (a.qkv_rs * es) % 16 == 0 && (a.q_out_rs * es) % 16 == 0 && (a.cache_rs * es) % 16 == 0 &&
           (a.cache_head * es) % 16 == 0 && (a.cache_seq * es) % 16 == 0;
}

}  // namespace

cudaError_t launch_qkv_producer(const ProducerArgs &a, bool bf16, cudaStream_t s) {
    const int64_t blocks = (int64_t)a.batch * a.n_new;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // the vectorised form needs 16-byte aligned rows; anything else takes the general one
    const bool vec = aligned16_all(a, bf16 ? 2 : 4);
    return bf16 ? launch_t<__nv_bfloat16>(a, (unsigned)blocks, vec, s)
                : launch_t<float>(a, (unsigned)blocks, vec, s);
}

}  // namespace lat
