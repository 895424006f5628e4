// common.cuh -- shared device helpers of the DSA step library (sm_103a).
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "../../include/dsa.h"

namespace dsa {

constexpr int kPage = 64;
constexpr int kIdxHeads = 32;
constexpr int kIdxDim = 128;
constexpr int kMlaHeads = 96;
constexpr int kLatDim = 576;
constexpr int kVDim = 512;
constexpr int kTopK = 2048;
constexpr int kFp8PageBytes = kPage * kIdxDim + kPage * 4;           // 8448
constexpr int kMxPageBytes = kPage * kIdxDim / 2 + kPage * 4;        // 4352
constexpr int kLatPageBytes = kPage * kLatDim;                       // 36864

// Request metadata passed by value to every kernel.
struct BatchArgs {
    int32_t num_requests;
    int32_t total_q;
    int32_t max_q;
    int32_t max_seq;
    int32_t num_pages;
    int32_t max_pages;
    const int32_t* q_offsets;
    const int32_t* seq_lens;
    const int32_t* block_table;
};

// Request of query token t: the b with q_offsets[b] <= t < q_offsets[b+1]
// (binary search over the non-decreasing prefix array).
__device__ __forceinline__ int request_of(const BatchArgs& bt, int t) {
    int lo = 0, hi = bt.num_requests - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(bt.q_offsets + mid) <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Device-side consistency of request b's metadata with the host-side sizes
// that bound every index (q_offsets within [0, total_q], n_b <= max_q,
// n_b <= seq_len <= max_seq).  A failing request is skipped by the caller and
// DSA_ERR_DEVICE_CHECK is recorded.
__device__ __forceinline__ bool request_ok(const BatchArgs& bt, int b, int32_t* status) {
    const int q0 = __ldg(bt.q_offsets + b);
    const int q1 = __ldg(bt.q_offsets + b + 1);
    const int seq = __ldg(bt.seq_lens + b);
    const bool ok = q0 >= 0 && q1 >= q0 && q1 <= bt.total_q && (q1 - q0) <= bt.max_q &&
                    seq >= (q1 - q0) && seq <= bt.max_seq;
    if (!ok && status) atomicCAS(status, 0, (int32_t)DSA_ERR_DEVICE_CHECK);
    return ok;
}

// Same check for the request that owns query token t (t must lie in it).
__device__ __forceinline__ bool token_ok(const BatchArgs& bt, int b, int t, int32_t* status) {
    if (!request_ok(bt, b, status)) return false;
    const bool ok = t >= __ldg(bt.q_offsets + b) && t < __ldg(bt.q_offsets + b + 1);
    if (!ok && status) atomicCAS(status, 0, (int32_t)DSA_ERR_DEVICE_CHECK);
    return ok;
}

// Number of positions query token t (of request b) may see.
__device__ __forceinline__ int visible_of(const BatchArgs& bt, int b, int t) {
    int q0 = __ldg(bt.q_offsets + b);
    int nb = __ldg(bt.q_offsets + b + 1) - q0;
    return __ldg(bt.seq_lens + b) - nb + (t - q0) + 1;
}

// Physical page of logical page lp of request b, or -1 after recording a
// device-check failure when the table entry is outside the pool.
__device__ __forceinline__ int page_lookup(const BatchArgs& bt, int b, int lp, int32_t* status) {
    int p = __ldg(bt.block_table + (int64_t)b * bt.max_pages + lp);
    if (p < 0 || p >= bt.num_pages) {
        if (status) atomicCAS(status, 0, (int32_t)DSA_ERR_DEVICE_CHECK);
        return -1;
    }
    return p;
}

__device__ __forceinline__ void record_error(int32_t* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Two E4M3 bytes (low byte first) -> two floats, exact.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
    return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// Order-preserving map of a float to uint32 (larger float -> larger key),
// with -0.0 mapped onto +0.0 so the two signed zeros tie.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}


// ---- programmatic dependent launch ------------------------------------------
// A kernel launched with `pdl` may start while the previous kernel of the
// stream is still running; it must call grid_dependency_wait() before it reads
// anything that kernel writes (the wait returns once that grid has completed
// and its writes are visible; without the launch attribute it returns at
// once).  grid_dependents_launch() lets the next kernel start launching.
__device__ __forceinline__ void grid_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// cudaLaunchKernelEx with optional programmatic serialisation and cluster size.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, bool pdl, int cluster, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace dsa
