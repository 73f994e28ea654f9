// kv_append.cu — in-place KV-cache append.
//
// Row pos[b] + t of sequence b's K and V caches takes new row t (t < n_new): the in-place
// "slice_set" cache append of the hf2q "Current Inference Path" page (sections 1 and 3)
// and the kv_cache_write step of the hf2q target page (section 6.1, step 6, whose note
// is that the stride arithmetic must match exactly).  Pure copy, one CTA per new row.
// A ring cache (sliding-window layers) stores position p in slot p % ring instead.
#include "device_common.cuh"
#include "kernels.h"

namespace lat {

template <typename U>  // copy unit: uint4 (16 B) when everything is 16-byte aligned
__global__ void __launch_bounds__(128) kv_append_kernel(AppendArgs a) {
    const int b = blockIdx.x / a.n_new;
    const int t = blockIdx.x % a.n_new;
    const int p = a.pos[b];
    // A sequence whose rows fall outside the cache is skipped whole (every CTA of the
    // sequence sees the same pos[b], so none of its rows is written).
    if (p < 0 || (a.ring == 0 && (int64_t)p + a.n_new > (int64_t)a.capacity)) {
        if (t == 0 && threadIdx.x == 0) report_status(a.status, kErrBounds);
        return;
    }
    const int64_t eb = a.elem_bytes;
    const int units_per_head = (int)((int64_t)a.head_dim * eb / (int64_t)sizeof(U));
    const int total = units_per_head * a.n_kv_heads;
    const int64_t src_row = ((int64_t)b * a.n_new + t) * a.new_rs;
    const int64_t slot = a.ring > 0 ? ((int64_t)p + t) % a.ring : (int64_t)p + t;
    const int64_t dst_row = (int64_t)b * a.cache_seq + slot * a.cache_rs;
    for (int u = threadIdx.x; u < total; u += blockDim.x) {
        const int hk = u / units_per_head, w = u % units_per_head;
        const int64_t src = (src_row + (int64_t)hk * a.head_dim) * eb;
        const int64_t dst = (dst_row + (int64_t)hk * a.cache_head) * eb;
        reinterpret_cast<U *>(a.k_cache + dst)[w] = reinterpret_cast<const U *>(a.k_new + src)[w];
        reinterpret_cast<U *>(a.v_cache + dst)[w] = reinterpret_cast<const U *>(a.v_new + src)[w];
    }
}

static bool aligned_to(const AppendArgs &a, int64_t unit) {
    auto ok_ptr = [&](const void *p) { return (reinterpret_cast<uintptr_t>(p) % unit) == 0; };
    const int64_t eb = a.elem_bytes;
    return ok_ptr(a.k_cache) && ok_ptr(a.v_cache) && ok_ptr(a.k_new) && ok_ptr(a.v_new) &&
           (a.cache_rs * eb) % unit == 0 && (a.cache_head * eb) % unit == 0 &&
           (a.cache_seq * eb) % unit == 0 && (a.new_rs * eb) % unit == 0 &&
           ((int64_t)a.head_dim * eb) % unit == 0;
}

cudaError_t launch_kv_append(const AppendArgs &a, cudaStream_t s) {
    const int64_t blocks = (int64_t)a.batch * a.n_new;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (aligned_to(a, 16))
        kv_append_kernel<uint4><<<(unsigned)blocks, 128, 0, s>>>(a);
    else if (aligned_to(a, 4))
        kv_append_kernel<uint32_t><<<(unsigned)blocks, 128, 0, s>>>(a);
    else
        kv_append_kernel<uint16_t><<<(unsigned)blocks, 128, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace lat
