// sparse_mla.cu -- absorbed-form MLA over the selected tokens.
//
// For query token t and head h over the selected positions I:
//   z[h,s] = sm_scale * kv_scale * (q_lat[t,h,:] . E4M3(latent[s,:]))   (576 dims)
//   out[t,h,:] = kv_scale * sum_s softmax_s(z)[s] * E4M3(latent[s,0:512])
// "vLLM's Kimi K3.1 Pro day-0 support", section "What changed" (MLA run
// exactly on the 2048 selected tokens) and section "Sparse attention cuts
// long-context decode bandwidth" (576-byte FP8 latents read for the selected
// tokens only).  Online softmax over chunks of 32 selected tokens.
#include "common.cuh"

namespace dsa {

namespace {

constexpr int kHeadsPerCta = 8;          // one warp per head
constexpr int kThreads = kHeadsPerCta * 32;
constexpr int kChunk = 32;               // selected tokens per step
constexpr int kLatStride = kLatDim + 1;  // padded smem row (bank-conflict free)

__global__ void __launch_bounds__(kThreads)
sparse_mla_kernel(BatchArgs bt, const __nv_bfloat16* __restrict__ q_lat,
                  const uint8_t* __restrict__ latent_pages, float kv_scale, float sm_scale,
                  const int32_t* __restrict__ indices, int K, __nv_bfloat16* __restrict__ out,
                  float* __restrict__ lse, int32_t* status) {
    extern __shared__ float smem[];
    float* lat_s = smem;                                  // [kChunk][kLatStride]
    float* q_s = lat_s + kChunk * kLatStride;             // [kHeadsPerCta][576]
    __shared__ int64_t src_off[kChunk];

    const int t = blockIdx.x;
    const int h0 = blockIdx.y * kHeadsPerCta;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = h0 + warp;
    const int b = request_of(bt, t);
    if (!token_ok(bt, b, t, status)) return;
    const int seq = __ldg(bt.seq_lens + b);

    for (int i = threadIdx.x; i < kHeadsPerCta * kLatDim; i += kThreads)
        q_s[i] = __bfloat162float(q_lat[((int64_t)t * kMlaHeads + h0) * kLatDim + i]);

    const float zscale = sm_scale * kv_scale;
    float m = -INFINITY, l = 0.f;
    float o[kVDim / 32];
#pragma unroll
    for (int i = 0; i < kVDim / 32; ++i) o[i] = 0.f;

    for (int c0 = 0; c0 < K; c0 += kChunk) {
        __syncthreads();
        if (threadIdx.x < kChunk) {
            int s = __ldg(indices + (int64_t)t * K + c0 + threadIdx.x);
            int64_t off = -1;
            if (s >= seq) {
                record_error(status, DSA_ERR_DEVICE_CHECK);
            } else if (s >= 0) {
                int p = page_lookup(bt, b, s / kPage, status);
                if (p >= 0) off = (int64_t)p * kLatPageBytes + (int64_t)(s % kPage) * kLatDim;
            }
            src_off[threadIdx.x] = off;
        }
        __syncthreads();
        // gather + dequantise: 32 rows x 36 16-byte vectors
        for (int v = threadIdx.x; v < kChunk * (kLatDim / 16); v += kThreads) {
            int r = v / (kLatDim / 16), c = v % (kLatDim / 16);
            int64_t off = src_off[r];
            float* dst = lat_s + r * kLatStride + c * 16;
            if (off >= 0) {
                uint4 raw = __ldg(reinterpret_cast<const uint4*>(latent_pages + off) + c);
                const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float2 a = e4m3x2_to_float2((uint16_t)(wv[i] & 0xFFFF));
                    float2 bb = e4m3x2_to_float2((uint16_t)(wv[i] >> 16));
                    dst[4 * i + 0] = a.x;
                    dst[4 * i + 1] = a.y;
                    dst[4 * i + 2] = bb.x;
                    dst[4 * i + 3] = bb.y;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) dst[i] = 0.f;
            }
        }
        __syncthreads();
        // scores: lane = selected token of the chunk
        const bool valid = src_off[lane] >= 0;
        float z = 0.f;
        const float* qh = q_s + warp * kLatDim;
        const float* lr = lat_s + lane * kLatStride;
#pragma unroll 8
        for (int d = 0; d < kLatDim; ++d) z = fmaf(qh[d], lr[d], z);
        z = valid ? z * zscale : -INFINITY;
        const float m_new = fmaxf(m, warp_max(z));
        const float corr = (m == -INFINITY) ? 0.f : expf(m - m_new);
        const float p = valid ? expf(z - m_new) : 0.f;
        l = l * corr + warp_sum(p);
#pragma unroll
        for (int i = 0; i < kVDim / 32; ++i) o[i] *= corr;
#pragma unroll 4
        for (int j = 0; j < kChunk; ++j) {
            const float pj = __shfl_sync(0xffffffffu, p, j);
            const float* lj = lat_s + j * kLatStride + lane;
#pragma unroll
            for (int i = 0; i < kVDim / 32; ++i) o[i] = fmaf(pj, lj[32 * i], o[i]);
        }
        m = m_new;
    }
    const float inv = (l > 0.f) ? kv_scale / l : 0.f;
    __nv_bfloat16* dst = out + ((int64_t)t * kMlaHeads + h) * kVDim;
#pragma unroll
    for (int i = 0; i < kVDim / 32; ++i) dst[lane + 32 * i] = __float2bfloat16_rn(o[i] * inv);
    if (lse && lane == 0) lse[(int64_t)t * kMlaHeads + h] = (l > 0.f) ? m + logf(l) : -INFINITY;
}

}  // namespace

size_t sparse_mla_smem_bytes() {
    return sizeof(float) * (kChunk * kLatStride + kHeadsPerCta * kLatDim);
}

cudaError_t launch_sparse_mla(const BatchArgs& bt, const uint16_t* q_lat, const void* latent_pages,
                              float kv_scale, float sm_scale, const int32_t* indices, int K,
                              uint16_t* out, float* lse, int32_t* status, cudaStream_t stream) {
    if (bt.total_q == 0) return cudaSuccess;
    const size_t smem = sparse_mla_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(sparse_mla_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(bt.total_q, kMlaHeads / kHeadsPerCta);
    sparse_mla_kernel<<<grid, kThreads, smem, stream>>>(
        bt, reinterpret_cast<const __nv_bfloat16*>(q_lat),
        static_cast<const uint8_t*>(latent_pages), kv_scale, sm_scale, indices, K,
        reinterpret_cast<__nv_bfloat16*>(out), lse, status);
    return cudaGetLastError();
}

}  // namespace dsa
