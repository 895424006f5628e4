// topk.cu -- exact top-k over the indexer scores.
//
// "vLLM's Kimi K3.1 Pro day-0 support", section "What changed": the indexer
// keeps the top 2048 tokens; section "Fused low-latency decode for DSA
// layers": an exact top-k selection follows the scorer.
//
// Per query token: a most-significant-digit radix select over order-preserving
// uint32 keys (digits of 11, 11 and 10 bits) finds the k-th largest key tau
// and how many keys equal to tau are still needed; a final pass in position
// order emits every position with key > tau plus the lowest positions with
// key == tau, which gives ascending output and the lower-position tie-break.
#include "common.cuh"

namespace dsa {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;

// Block-wide exclusive prefix count of `flag`; returns the prefix of this
// thread and writes the block total to *total.  Uses `warp_tot` (kWarps ints).
__device__ __forceinline__ int block_excl_count(bool flag, int* warp_tot, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned m = __ballot_sync(0xffffffffu, flag);
    int pre = __popc(m & ((1u << lane) - 1u));
    if (lane == 0) warp_tot[warp] = __popc(m);
    __syncthreads();
    if (warp == 0) {
        int v = warp_tot[lane];
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int u = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += u;
        }
        warp_tot[lane] = inc - v;  // exclusive
        if (lane == 31) warp_tot[kWarps] = inc;
    }
    __syncthreads();
    int r = pre + warp_tot[warp];
    *total = warp_tot[kWarps];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kThreads)
topk_radix_kernel(BatchArgs bt, const float* __restrict__ scores, int64_t ld, int K,
                  int32_t* __restrict__ out) {
    __shared__ uint32_t hist[kBins];
    __shared__ int warp_tot[kWarps + 1];
    __shared__ uint32_t s_digit, s_remaining;

    const int t = blockIdx.x;
    const int b = request_of(bt, t);
    int32_t* o = out + (int64_t)t * K;
    if (!token_ok(bt, b, t, nullptr)) {  // inconsistent metadata: select nothing
        for (int i = threadIdx.x; i < K; i += kThreads) o[i] = -1;
        return;
    }
    const int vis = visible_of(bt, b, t);
    const float* row = scores + (int64_t)t * ld;

    if (vis <= K) {
        for (int i = threadIdx.x; i < K; i += kThreads) o[i] = (i < vis) ? i : -1;
        return;
    }

    uint32_t prefix = 0, pmask = 0, remaining = (uint32_t)K;
    const int shifts[3] = {21, 10, 0};
    const uint32_t masks[3] = {0x7FFu, 0x7FFu, 0x3FFu};
    for (int d = 0; d < 3; ++d) {
        const int sh = shifts[d];
        const uint32_t mk = masks[d];
        for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
        __syncthreads();
        for (int s = threadIdx.x; s < vis; s += kThreads) {
            uint32_t key = order_key(__ldg(row + s));
            if ((key & pmask) == prefix) atomicAdd(&hist[(key >> sh) & mk], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            // lane owns bins [64*lane, 64*lane + 64); higher lanes hold larger keys
            uint32_t c = 0;
            for (int i = 0; i < 64; ++i) c += hist[64 * lane + i];
            // count in lanes above this one (suffix sum, exclusive)
            uint32_t incl = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                uint32_t u = __shfl_down_sync(0xffffffffu, incl, off);
                if (lane + off < 32) incl += u;
            }
            uint32_t above = incl - c;
            if (above < remaining && remaining <= above + c) {
                uint32_t run = above;
                for (int i = 63; i >= 0; --i) {
                    uint32_t h = hist[64 * lane + i];
                    if (run + h >= remaining) {
                        s_digit = (uint32_t)(64 * lane + i);
                        s_remaining = remaining - run;
                        break;
                    }
                    run += h;
                }
            }
        }
        __syncthreads();
        prefix |= s_digit << sh;
        pmask |= mk << sh;
        remaining = s_remaining;
        __syncthreads();
    }
    // prefix is now the k-th largest key tau; `remaining` keys equal to tau are
    // taken, lowest positions first.
    const uint32_t tau = prefix;
    const int need_eq = (int)remaining;
    int base = 0, eq_seen = 0;
    for (int c = 0; c < vis; c += kThreads) {
        const int s = c + threadIdx.x;
        uint32_t key = (s < vis) ? order_key(__ldg(row + s)) : 0u;
        bool is_eq = (s < vis) && key == tau;
        bool is_gt = (s < vis) && key > tau;
        int eq_tot;
        int eq_rank = eq_seen + block_excl_count(is_eq, warp_tot, &eq_tot);
        bool sel = is_gt || (is_eq && eq_rank < need_eq);
        int sel_tot;
        int pos = base + block_excl_count(sel, warp_tot, &sel_tot);
        if (sel) o[pos] = s;
        base += sel_tot;
        eq_seen += eq_tot;
    }
}

}  // namespace

cudaError_t launch_topk(const BatchArgs& bt, const float* scores, int64_t ld, int K,
                        int32_t* out, cudaStream_t stream) {
    if (bt.total_q == 0) return cudaSuccess;
    topk_radix_kernel<<<bt.total_q, kThreads, 0, stream>>>(bt, scores, ld, K, out);
    return cudaGetLastError();
}

}  // namespace dsa
