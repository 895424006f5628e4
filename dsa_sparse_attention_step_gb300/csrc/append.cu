// append.cu -- write new tokens' index keys and latents into the paged caches.
//
// "vLLM's Kimi K3.1 Pro day-0 support", section "Fused low-latency decode for
// DSA layers": the indexer front produces the new token's index key and the MLA
// query path writes the new token's latent into the KV cache.  Key: per-token
// scale amax/448 (fp32), codes E4M3 round-to-nearest-even saturating of
// x/scale; latent: E4M3 of x/kv_scale.
#include "common.cuh"

namespace dsa {

namespace {

constexpr int kWarpsPerCta = 4;

__device__ __forceinline__ uint8_t to_e4m3(float v) {
    return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

__global__ void __launch_bounds__(kWarpsPerCta * 32)
append_cache_kernel(BatchArgs bt, const float* __restrict__ keys, const float* __restrict__ lat,
                    float kv_scale, uint8_t* __restrict__ index_pages,
                    uint8_t* __restrict__ latent_pages, int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    if (t >= bt.total_q) return;
    const int b = request_of(bt, t);
    if (!token_ok(bt, b, t, status)) return;
    const int pos = visible_of(bt, b, t) - 1;
    const int page = page_lookup(bt, b, pos / kPage, status);
    if (page < 0) return;
    const int slot = pos % kPage;

    if (keys != nullptr && index_pages != nullptr) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(keys + (int64_t)t * kIdxDim) + lane);
        float amax = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
        amax = warp_max(amax);
        const float scale = (amax > 0.f) ? __fdiv_rn(amax, 448.0f) : 1.0f;
        uint32_t packed = (uint32_t)to_e4m3(__fdiv_rn(x.x, scale)) |
                          ((uint32_t)to_e4m3(__fdiv_rn(x.y, scale)) << 8) |
                          ((uint32_t)to_e4m3(__fdiv_rn(x.z, scale)) << 16) |
                          ((uint32_t)to_e4m3(__fdiv_rn(x.w, scale)) << 24);
        uint8_t* base = index_pages + (int64_t)page * kFp8PageBytes;
        reinterpret_cast<uint32_t*>(base + slot * kIdxDim)[lane] = packed;
        if (lane == 0) reinterpret_cast<float*>(base + kPage * kIdxDim)[slot] = scale;
    }
    if (lat != nullptr && latent_pages != nullptr) {
        const float* src = lat + (int64_t)t * kLatDim;
        uint8_t* dst = latent_pages + (int64_t)page * kLatPageBytes + (int64_t)slot * kLatDim;
        // 576 = 144 groups of 4 -> 4.5 groups per lane
        for (int g = lane; g < kLatDim / 4; g += 32) {
            const float4 x = __ldg(reinterpret_cast<const float4*>(src) + g);
            uint32_t packed = (uint32_t)to_e4m3(__fdiv_rn(x.x, kv_scale)) |
                              ((uint32_t)to_e4m3(__fdiv_rn(x.y, kv_scale)) << 8) |
                              ((uint32_t)to_e4m3(__fdiv_rn(x.z, kv_scale)) << 16) |
                              ((uint32_t)to_e4m3(__fdiv_rn(x.w, kv_scale)) << 24);
            reinterpret_cast<uint32_t*>(dst)[g] = packed;
        }
    }
}

}  // namespace

cudaError_t launch_append_cache(const BatchArgs& bt, const float* keys, const float* lat,
                                float kv_scale, void* index_pages, void* latent_pages,
                                int32_t* status, cudaStream_t stream) {
    if (bt.total_q == 0) return cudaSuccess;
    const int grid = (bt.total_q + kWarpsPerCta - 1) / kWarpsPerCta;
    append_cache_kernel<<<grid, kWarpsPerCta * 32, 0, stream>>>(
        bt, keys, lat, kv_scale, static_cast<uint8_t*>(index_pages),
        static_cast<uint8_t*>(latent_pages), status);
    return cudaGetLastError();
}

}  // namespace dsa
