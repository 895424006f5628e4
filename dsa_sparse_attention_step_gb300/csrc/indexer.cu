// indexer.cu -- DSA indexer scores.
//
// score[t,s] = sum_h w[t,h]*q_scale[t,h] * ReLU(q8[t,h,:] . k8[s,:]) * kscale[s]
// (FP8 keys; the positive per-token key scale and per-head query scale are
// pulled through the ReLU) or, for MXFP4 keys, the same sum with the key
// dequantised per 32-element block before the dot product.
//
// "vLLM's Kimi K3.1 Pro day-0 support", section "What changed": 32 indexer
// heads x 128 dims, one FP8 key (132 B with scale) per token, every earlier
// token scored; section "Native MXFP4 indexer": 68-B MXFP4 keys, fp32
// accumulation, weighted reduction across heads.
#include "common.cuh"

namespace dsa {

namespace {

constexpr int kTileKeys = 128;   // keys per CTA (one thread per key)
constexpr int kTokChunk = 8;     // query tokens per CTA (grid z covers the rest)

// Decode 16 consecutive key elements (FP8 bytes in `raw`) into floats.
__device__ __forceinline__ void decode16_fp8(const uint4& raw, float* k) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 a = e4m3x2_to_float2((uint16_t)(w[i] & 0xFFFF));
        float2 b = e4m3x2_to_float2((uint16_t)(w[i] >> 16));
        k[4 * i + 0] = a.x;
        k[4 * i + 1] = a.y;
        k[4 * i + 2] = b.x;
        k[4 * i + 3] = b.y;
    }
}

// E2M1 magnitudes in code order.
__device__ __forceinline__ float e2m1_value(uint32_t nib) {
    const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
    float v = mag[nib & 7];
    return (nib & 8) ? -v : v;
}

// Decode 16 consecutive MXFP4 elements (8 packed bytes, element 2i in the low
// nibble) and multiply by the block scale 2^(e-127).
__device__ __forceinline__ void decode16_mx(uint2 raw, float scale, float* k) {
    const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) k[8 * i + j] = e2m1_value((w[i] >> (4 * j)) & 0xF) * scale;
}

template <int kFormat>
__global__ void __launch_bounds__(kTileKeys)
indexer_scores_kernel(BatchArgs bt, const uint8_t* __restrict__ q8,
                      const float* __restrict__ qscale, const float* __restrict__ w,
                      const uint8_t* __restrict__ pages, float* __restrict__ scores,
                      int64_t ld, int32_t* status) {
    __shared__ float q_s[kIdxHeads * kIdxDim];
    __shared__ float wq_s[kIdxHeads];

    const int b = blockIdx.y;
    if (!request_ok(bt, b, blockIdx.x == 0 && blockIdx.z == 0 ? status : nullptr)) return;
    const int seq = __ldg(bt.seq_lens + b);
    const int q0 = __ldg(bt.q_offsets + b);
    const int nb = __ldg(bt.q_offsets + b + 1) - q0;
    const int tile0 = blockIdx.x * kTileKeys;
    const int j0 = blockIdx.z * kTokChunk;
    if (tile0 >= seq || j0 >= nb) return;
    const int j1 = min(nb, j0 + kTokChunk);

    const int s = tile0 + threadIdx.x;
    const bool in_seq = s < seq;
    int page = -1;
    if (in_seq) page = page_lookup(bt, b, s / kPage, status);
    const int slot = s % kPage;

    // the key of this thread, kept raw in registers
    uint4 kraw[8];
    uint2 mraw[8];
    float kscale = 0.f;
    float bscale[4] = {0.f, 0.f, 0.f, 0.f};
    if (page >= 0) {
        if (kFormat == DSA_KEYS_FP8_E4M3) {
            const uint8_t* base = pages + (int64_t)page * kFp8PageBytes;
            const uint4* src = reinterpret_cast<const uint4*>(base + slot * kIdxDim);
#pragma unroll
            for (int c = 0; c < 8; ++c) kraw[c] = __ldg(src + c);
            kscale = __ldg(reinterpret_cast<const float*>(base + kPage * kIdxDim) + slot);
        } else {
            const uint8_t* base = pages + (int64_t)page * kMxPageBytes;
            const uint2* src = reinterpret_cast<const uint2*>(base + slot * (kIdxDim / 2));
#pragma unroll
            for (int c = 0; c < 8; ++c) mraw[c] = __ldg(src + c);
            const uint8_t* sc = base + kPage * (kIdxDim / 2) + slot * 4;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t e = sc[i];
                bscale[i] = (e == 0xFF) ? __int_as_float(0x7fffffff)
                                        : ldexpf(1.0f, (int)e - 127);
            }
        }
    }

    for (int j = j0; j < j1; ++j) {
        const int t = q0 + j;
        __syncthreads();
        for (int i = threadIdx.x; i < kIdxHeads * kIdxDim / 2; i += kTileKeys) {
            float2 v = e4m3x2_to_float2(
                reinterpret_cast<const uint16_t*>(q8 + (int64_t)t * kIdxHeads * kIdxDim)[i]);
            q_s[2 * i] = v.x;
            q_s[2 * i + 1] = v.y;
        }
        if (threadIdx.x < kIdxHeads)
            wq_s[threadIdx.x] = __ldg(w + (int64_t)t * kIdxHeads + threadIdx.x) *
                                __ldg(qscale + (int64_t)t * kIdxHeads + threadIdx.x);
        __syncthreads();
        if (!in_seq) continue;

        float acc[kIdxHeads];
#pragma unroll
        for (int h = 0; h < kIdxHeads; ++h) acc[h] = 0.f;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
            float k[16];
            if (kFormat == DSA_KEYS_FP8_E4M3) decode16_fp8(kraw[c], k);
            else decode16_mx(mraw[c], bscale[c / 2], k);
#pragma unroll
            for (int h = 0; h < kIdxHeads; ++h) {
                const float4* qh = reinterpret_cast<const float4*>(q_s + h * kIdxDim + c * 16);
#pragma unroll
                for (int d4 = 0; d4 < 4; ++d4) {
                    float4 qv = qh[d4];
                    acc[h] = fmaf(qv.x, k[4 * d4 + 0], acc[h]);
                    acc[h] = fmaf(qv.y, k[4 * d4 + 1], acc[h]);
                    acc[h] = fmaf(qv.z, k[4 * d4 + 2], acc[h]);
                    acc[h] = fmaf(qv.w, k[4 * d4 + 3], acc[h]);
                }
            }
        }
        float score = 0.f;
#pragma unroll
        for (int h = 0; h < kIdxHeads; ++h) score = fmaf(wq_s[h], fmaxf(acc[h], 0.f), score);
        if (kFormat == DSA_KEYS_FP8_E4M3) score *= kscale;
        const int vis = seq - nb + j + 1;
        // positions past the causal limit, or whose page failed the range check
        scores[(int64_t)t * ld + s] = (s < vis && page >= 0) ? score : -INFINITY;
    }
}

}  // namespace

bool indexer_tc_supported(const BatchArgs& bt);
cudaError_t launch_index_scores_fp8_tc(const BatchArgs& bt, const uint8_t* q8, const float* qscale,
                                       const float* w, const void* pages, float* scores,
                                       int64_t ld, int32_t* status, cudaStream_t stream);

cudaError_t launch_index_scores(const BatchArgs& bt, const uint8_t* q8, const float* qscale,
                                const float* w, const void* pages, int key_format,
                                float* scores, int64_t ld, int32_t* status,
                                cudaStream_t stream) {
    if (key_format == DSA_KEYS_FP8_E4M3 && indexer_tc_supported(bt))
        return launch_index_scores_fp8_tc(bt, q8, qscale, w, pages, scores, ld, status, stream);
    dim3 grid((bt.max_seq + kTileKeys - 1) / kTileKeys, bt.num_requests,
              (bt.max_q + kTokChunk - 1) / kTokChunk);
    if (key_format == DSA_KEYS_FP8_E4M3)
        indexer_scores_kernel<DSA_KEYS_FP8_E4M3><<<grid, kTileKeys, 0, stream>>>(
            bt, q8, qscale, w, static_cast<const uint8_t*>(pages), scores, ld, status);
    else
        indexer_scores_kernel<DSA_KEYS_MXFP4><<<grid, kTileKeys, 0, stream>>>(
            bt, q8, qscale, w, static_cast<const uint8_t*>(pages), scores, ld, status);
    return cudaGetLastError();
}

}  // namespace dsa
