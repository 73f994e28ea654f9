// decode_static.cu — lat_attn_decode_static: the bf16/fp32 decode step for callers that
// cannot allocate device memory.
//
// Some callers have no allocator to hand: code that runs inside a framework that owns
// all device memory and exposes none of it, plugins loaded into a host process that
// forbids cudaMalloc after start-up (the allocation could fail or fragment a pool the
// host sized), and real-time paths where a device allocation's implicit
// synchronisation and unbounded latency are not acceptable.  lat_attn_decode needs a
// caller-provided workspace for its split-KV partial results; this entry point instead
// takes its scratch from one fixed-size array in device global memory that is part of
// the library's device image, so the caller passes only inputs and outputs.
//
// The array lives as long as the library is loaded, on every GPU the library is used
// on.  All calls on a device share it, so calls that can overlap on the GPU (different
// streams, or graphs replayed concurrently) race on it and must be serialised by the
// caller.  The merge counters inside it are cleared on the call's stream before every
// launch, because the previous call may have left other data at those offsets.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kernels.h"
#include "lat_attn.h"

namespace {

// The stated maximum: enough for the decode shapes of this library's workloads (for
// example batch 8, 16 query heads, head_dim 512 at 32768 cached tokens needs ~10 MB).
constexpr size_t kStaticScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of g_decode_scratch for `dev`, resolved once per device with that
// device current (in host code the symbol itself is only a host-side stand-in).
unsigned char *scratch_on_device(int dev) {
    static std::mutex mu;
    static unsigned char *addr[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
            return nullptr;
        addr[dev] = static_cast<unsigned char *>(p);
    }
    return addr[dev];
}

}  // namespace

extern "C" lat_status lat_attn_decode_static(
    lat_dtype dt, const void *q, int64_t q_rs, const void *k_cache, const void *v_cache,
    int64_t cache_rs, int64_t cache_head_stride, int64_t cache_seq_stride,
    const int32_t *kv_lens, int max_kv_len, void *out, int64_t out_rs, float *lse, int batch,
    int n_heads, int n_kv_heads, int head_dim, int window, float scale, int32_t *status,
    void *stream) {
    if (dt == LAT_F32)  // the fp32 decode path uses no scratch
        return lat_attn_decode(dt, q, q_rs, k_cache, v_cache, cache_rs, cache_head_stride,
                               cache_seq_stride, kv_lens, max_kv_len, out, out_rs, lse, batch,
                               n_heads, n_kv_heads, head_dim, window, scale, nullptr, 0, status,
                               stream);
    if (dt != LAT_BF16 || batch < 0 || max_kv_len < 0 || n_heads <= 0 || n_kv_heads <= 0 ||
        n_heads % n_kv_heads != 0)
        return LAT_ERR_INVALID_ARG;
    if (batch == 0) return LAT_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return LAT_ERR_CUDA;
    lat::DecodePlan plan;
    if (!lat::plan_decode_bf16(batch, n_heads, n_kv_heads, head_dim, max_kv_len,
                               window < 0 ? 0 : window, sms, &plan))
        return LAT_ERR_UNSUPPORTED;
    if (plan.total_bytes > kStaticScratchBytes) return LAT_ERR_WORKSPACE;  // beyond the maximum
    unsigned char *scratch = scratch_on_device(dev);
    if (scratch == nullptr) return LAT_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the merge counters must start at zero; the last call may have left partial
    // results of another shape at these offsets
    if (cudaMemsetAsync(scratch + plan.part_o_bytes + plan.part_lse_bytes, 0,
                        plan.counter_bytes, s) != cudaSuccess)
        return LAT_ERR_CUDA;
    return lat_attn_decode(dt, q, q_rs, k_cache, v_cache, cache_rs, cache_head_stride,
                           cache_seq_stride, kv_lens, max_kv_len, out, out_rs, lse, batch,
                           n_heads, n_kv_heads, head_dim, window, scale, scratch,
                           kStaticScratchBytes, status, stream);
}
