// topk.cu -- exact top-k over the indexer scores.
//
// "vLLM's Kimi K3.1 Pro day-0 support", section "What changed": the indexer
// keeps the top 2048 tokens; section "Fused low-latency decode for DSA
// layers": an exact top-k selection follows the scorer.
//
// For query token t with `vis` visible positions (vis > k): the k positions
// with the largest scores, ties to the lower position, in ascending order.
// Scores are mapped to order-preserving uint32 keys (-0 folded onto +0) and the
// k-th largest key tau is found by a most-significant-digit radix select with
// digits of 12, 10 and 10 bits.
//
// One thread-block cluster of `cs` CTAs per query token; CTA r owns a
// contiguous, 32-aligned slice of the positions and keeps its slice's results
// in shared memory.  Per digit the CTAs build histograms of their slice
// (streaming the scores from global memory), the cluster sums them through
// distributed shared memory, and every CTA derives the same digit.  As soon as
// the keys sharing the threshold prefix fit the candidate buffers, one more
// streaming pass marks the positions above the prefix in a bitmap and copies
// the candidates (key, position) into shared memory; the remaining digits are
// resolved on the candidates only.  Keys equal to tau are taken lowest
// position first across the cluster (prefix of per-CTA counts), and each CTA
// writes its selected positions in order at its offset in the output row.
// Inputs whose threshold bin keeps more keys than the buffers hold (e.g. huge
// runs of equal scores) resolve all digits by streaming and select in a final
// ordered streaming pass.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace dsa {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
constexpr int kBins = 4096;                  // first digit: 12 bits
constexpr int kCandCap = 8192;               // candidates per CTA
constexpr int kSliceMax = 1 << 18;           // positions per CTA (bitmap capacity)
constexpr int kWords = kSliceMax / 32;       // 8192 bitmap words

struct TopkShared {
    uint32_t hist[kBins];       // this CTA's histogram (read remotely by the cluster)
    uint32_t tot[kBins];        // cluster-wide histogram
    uint32_t bits[kWords];      // selected positions of the slice
    uint32_t cand_key[kCandCap];
    int32_t cand_pos[kCandCap];
    int32_t warp_tot[kWarps + 1];
    uint32_t xchg[4];           // per-CTA values read by the cluster
    uint32_t s_digit, s_rem, s_count;
};

// Radix digits: bits 31..20, 19..10, 9..0 of the order key.
__device__ __forceinline__ int dig_shift(int level) { return level == 0 ? 20 : (level == 1 ? 10 : 0); }
__device__ __forceinline__ uint32_t dig_mask(int level) { return level == 0 ? 0xFFFu : 0x3FFu; }

// Block-wide exclusive prefix sum of v (1024 threads); returns the prefix and
// the total through *total.
__device__ __forceinline__ int block_excl_sum(int v, int* warp_tot, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = warp_tot[lane];
        int inc = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += u;
        }
        warp_tot[lane] = inc - w;
        if (lane == 31) warp_tot[kWarps] = inc;
    }
    __syncthreads();
    const int r = incl - v + warp_tot[warp];
    *total = warp_tot[kWarps];
    __syncthreads();
    return r;
}

// Warp-aggregated shared-memory histogram increment.
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool active) {
    const unsigned act = __ballot_sync(0xffffffffu, active);
    if (!active) return;
    const unsigned peers = __match_any_sync(act, bin);
    if ((__ffs(peers) - 1) == (int)(threadIdx.x & 31)) atomicAdd(&hist[bin], __popc(peers));
}

// Sum the cluster's histograms (nb bins) into tot, then find the digit d such
// that count(digits > d) < rem <= count(digits >= d); stores the digit, the
// remaining count within it and the count of the digit's bin.
__device__ void cluster_digit(TopkShared& S, cg::cluster_group& cluster, int nb, uint32_t rem) {
    const int cs = (int)cluster.num_blocks();
    cluster.sync();  // every histogram of the cluster is complete
    for (int i = threadIdx.x; i < nb; i += kThreads) {
        uint32_t v = 0;
        for (int r = 0; r < cs; ++r) v += cluster.map_shared_rank(S.hist, r)[i];
        S.tot[i] = v;
    }
    cluster.sync();  // remote reads done before any histogram is reset
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int per = nb / 32;
        uint32_t c = 0;
        for (int i = 0; i < per; ++i) c += S.tot[per * lane + i];
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_down_sync(0xffffffffu, incl, o);
            if (lane + o < 32) incl += u;
        }
        const uint32_t above = incl - c;
        if (above < rem && rem <= above + c) {
            uint32_t run = above;
            for (int i = per - 1; i >= 0; --i) {
                const uint32_t h = S.tot[per * lane + i];
                if (run + h >= rem) {
                    S.s_digit = (uint32_t)(per * lane + i);
                    S.s_rem = rem - run;
                    S.s_count = h;
                    break;
                }
                run += h;
            }
        }
    }
    __syncthreads();
}

// Exclusive prefix over the cluster ranks of the per-CTA value in xchg[slot];
// also returns the cluster total.
__device__ uint32_t cluster_prefix(TopkShared& S, cg::cluster_group& cluster, int slot,
                                   uint32_t* total) {
    cluster.sync();
    const int cs = (int)cluster.num_blocks(), me = (int)cluster.block_rank();
    uint32_t before = 0, tot = 0;
    for (int r = 0; r < cs; ++r) {
        const uint32_t v = cluster.map_shared_rank(S.xchg, r)[slot];
        if (r < me) before += v;
        tot += v;
    }
    *total = tot;
    return before;
}

__global__ void __launch_bounds__(kThreads, 1)
topk_cluster_kernel(BatchArgs bt, const float* __restrict__ scores, int64_t ld, int K,
                    int32_t* __restrict__ out) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    TopkShared& S = *reinterpret_cast<TopkShared*>(smem_raw);
    cg::cluster_group cluster = cg::this_cluster();
    const int cs = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int t = blockIdx.x / cs;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = request_of(bt, t);
    int32_t* o = out + (int64_t)t * K;
    // uniform over the cluster: every CTA of token t takes the same branch
    const bool ok = token_ok(bt, b, t, nullptr);
    const int vis = ok ? visible_of(bt, b, t) : 0;
    if (vis <= K) {
        if (rank == 0)
            for (int i = tid; i < K; i += kThreads) o[i] = (i < vis) ? i : -1;
        return;
    }
    const float* row = scores + (int64_t)t * ld;
    // 32-aligned slice [lo, hi) of the visible positions
    const int per = ((vis + cs - 1) / cs + 31) & ~31;
    const int lo = min(vis, rank * per);
    const int hi = min(vis, lo + per);
    const int nwords = (hi - lo + 31) / 32;

    uint32_t prefix = 0, pmask = 0, rem = (uint32_t)K;
    int level = 0;
    bool collected = false;
    int ncand = 0;
    // ---- streaming digits until the threshold prefix is small enough ----
    while (level < 3) {
        const int nb = (level == 0) ? kBins : 1024;
        for (int i = tid; i < nb; i += kThreads) S.hist[i] = 0;
        __syncthreads();
        for (int s0 = lo + warp * 32; s0 < hi; s0 += kThreads) {
            const int s = s0 + lane;
            const bool in = s < hi;
            const uint32_t key = in ? order_key(__ldg(row + s)) : 0u;
            const bool match = in && (key & pmask) == prefix;
            hist_add(S.hist, (key >> dig_shift(level)) & dig_mask(level), match);
        }
        cluster_digit(S, cluster, nb, rem);
        const uint32_t d = S.s_digit;
        // the local count of the threshold digit decides whether candidates fit
        S.xchg[0] = S.hist[d];
        prefix |= d << dig_shift(level);
        pmask |= dig_mask(level) << dig_shift(level);
        rem = S.s_rem;
        ++level;
        // largest local count over the cluster (all CTAs agree on the branch)
        cluster.sync();
        uint32_t mx = 0;
        for (int r = 0; r < cs; ++r) mx = max(mx, cluster.map_shared_rank(S.xchg, r)[0]);
        cluster.sync();
        if (level < 3 && mx <= (uint32_t)kCandCap) break;
    }

    if (level < 3) {
        // ---- collection pass: bitmap of positions above the prefix, candidates ----
        if (tid == 0) S.s_count = 0;
        __syncthreads();
        for (int s0 = lo + warp * 32; s0 < hi; s0 += kThreads) {
            const int s = s0 + lane;
            const bool in = s < hi;
            const uint32_t key = in ? order_key(__ldg(row + s)) : 0u;
            const uint32_t top = key & pmask;
            const unsigned above = __ballot_sync(0xffffffffu, in && top > prefix);
            const bool cand = in && top == prefix;
            const unsigned cm = __ballot_sync(0xffffffffu, cand);
            if (lane == 0) S.bits[(s0 - lo) >> 5] = above;
            int base = 0;
            if (lane == 0 && cm) base = atomicAdd(&S.s_count, __popc(cm));
            base = __shfl_sync(0xffffffffu, base, 0);
            if (cand) {
                const int c = base + __popc(cm & ((1u << lane) - 1u));
                S.cand_key[c] = key;
                S.cand_pos[c] = s;
            }
        }
        __syncthreads();
        ncand = (int)S.s_count;
        collected = true;
        // ---- remaining digits on the candidates ----
        while (level < 3) {
            for (int i = tid; i < 1024; i += kThreads) S.hist[i] = 0;
            __syncthreads();
            for (int c0 = 0; c0 < ncand; c0 += kThreads) {
                const int c = c0 + tid;
                const bool in = c < ncand;
                const uint32_t key = in ? S.cand_key[c] : 0u;
                const bool match = in && (key & pmask) == prefix;
                hist_add(S.hist, (key >> dig_shift(level)) & dig_mask(level), match);
            }
            cluster_digit(S, cluster, 1024, rem);
            prefix |= S.s_digit << dig_shift(level);
            pmask |= dig_mask(level) << dig_shift(level);
            rem = S.s_rem;
            ++level;
        }
    }
    // prefix is now the k-th largest key tau; `rem` keys equal to tau are taken,
    // lowest positions first across the cluster
    const uint32_t tau = prefix;
    const uint32_t need_eq = rem;

    if (collected) {
        // count this CTA's keys equal to tau, exchange, take the lowest ones
        int eq_local = 0;
        for (int c = tid; c < ncand; c += kThreads) eq_local += (S.cand_key[c] == tau) ? 1 : 0;
        int eq_tot;
        (void)block_excl_sum(eq_local, S.warp_tot, &eq_tot);
        S.xchg[1] = (uint32_t)eq_tot;
        uint32_t eq_all;
        const uint32_t eq_before = cluster_prefix(S, cluster, 1, &eq_all);
        const int take = (int)min((uint32_t)eq_tot, need_eq > eq_before ? need_eq - eq_before : 0u);
        // candidates above tau are selected; equal ones by position rank
        for (int c0 = 0; c0 < ncand; c0 += kThreads) {
            const int c = c0 + tid;
            if (c < ncand) {
                const uint32_t key = S.cand_key[c];
                const int pos = S.cand_pos[c];
                bool sel = key > tau;
                if (key == tau && take > 0) {
                    // rank among this CTA's tau-equal candidates by position
                    int rank_eq = 0;
                    for (int j = 0; j < ncand; ++j)
                        rank_eq += (S.cand_key[j] == tau && S.cand_pos[j] < pos) ? 1 : 0;
                    sel = rank_eq < take;
                }
                if (sel) atomicOr(&S.bits[(pos - lo) >> 5], 1u << ((pos - lo) & 31));
            }
        }
        __syncthreads();
    } else {
        // ---- fallback: selection by streaming with the full key known ----
        // keys above tau: one bitmap word per warp iteration
        int eq = 0;
        for (int s0 = lo + warp * 32; s0 < hi; s0 += kThreads) {
            const int s = s0 + lane;
            const bool in = s < hi;
            const uint32_t key = in ? order_key(__ldg(row + s)) : 0u;
            const unsigned gtm = __ballot_sync(0xffffffffu, in && key > tau);
            eq += (in && key == tau) ? 1 : 0;
            if (lane == 0) S.bits[(s0 - lo) >> 5] = gtm;
        }
        int eq_tot;
        (void)block_excl_sum(eq, S.warp_tot, &eq_tot);
        S.xchg[1] = (uint32_t)eq_tot;
        uint32_t eq_all;
        const uint32_t eq_before = cluster_prefix(S, cluster, 1, &eq_all);
        const int take =
            (int)min((uint32_t)eq_tot, need_eq > eq_before ? need_eq - eq_before : 0u);
        // keys equal to tau, lowest positions first: a block-ordered pass over words
        int eq_seen = 0;
        for (int w0 = 0; w0 < nwords; w0 += kThreads) {
            const int w = w0 + tid;
            uint32_t eqm = 0;
            if (w < nwords) {
                const int s0 = lo + 32 * w;
                for (int j = 0; j < 32 && s0 + j < hi; ++j)
                    eqm |= (order_key(__ldg(row + s0 + j)) == tau ? 1u : 0u) << j;
            }
            int cnt;
            const int before = eq_seen + block_excl_sum(__popc(eqm), S.warp_tot, &cnt);
            if (eqm) {
                int r = before;
                uint32_t m = eqm, keep = 0;
                while (m) {
                    const int j = __ffs(m) - 1;
                    if (r < take) keep |= 1u << j;
                    ++r;
                    m &= m - 1;
                }
                S.bits[w] |= keep;
            }
            eq_seen += cnt;
        }
        __syncthreads();
    }

    // ---- ordered output: this CTA's selected positions at its cluster offset ----
    int sel_local = 0;
    for (int w = tid; w < nwords; w += kThreads) sel_local += __popc(S.bits[w]);
    int sel_tot;
    (void)block_excl_sum(sel_local, S.warp_tot, &sel_tot);
    S.xchg[2] = (uint32_t)sel_tot;
    uint32_t all;
    const uint32_t off = cluster_prefix(S, cluster, 2, &all);
    // words are assigned to threads in contiguous runs so the order is kept
    const int wpt = (nwords + kThreads - 1) / kThreads;
    const int w_begin = min(nwords, tid * wpt), w_end = min(nwords, w_begin + wpt);
    int mine = 0;
    for (int w = w_begin; w < w_end; ++w) mine += __popc(S.bits[w]);
    int tot2;
    int pos = (int)off + block_excl_sum(mine, S.warp_tot, &tot2);
    for (int w = w_begin; w < w_end; ++w) {
        uint32_t m = S.bits[w];
        while (m) {
            const int j = __ffs(m) - 1;
            if (pos < K) o[pos] = lo + 32 * w + j;
            ++pos;
            m &= m - 1;
        }
    }
    cluster.sync();  // no CTA leaves while others may still read its shared memory
}

}  // namespace

// CTAs per query token: spread few tokens over more SMs, and keep every
// slice within the per-CTA bitmap.
int topk_cluster_size(int total_q, int max_seq) {
    int cs = 1;
    while (cs < kMaxCluster && total_q * cs * 2 <= 152) cs <<= 1;
    while (cs < kMaxCluster && (max_seq + cs - 1) / cs > kSliceMax) cs <<= 1;
    return cs;
}

bool topk_supported(int max_seq) { return max_seq <= kSliceMax * kMaxCluster; }

cudaError_t launch_topk(const BatchArgs& bt, const float* scores, int64_t ld, int K,
                        int32_t* out, cudaStream_t stream) {
    if (bt.total_q == 0) return cudaSuccess;
    const int cs = topk_cluster_size(bt.total_q, bt.max_seq);
    const size_t smem = sizeof(TopkShared);
    cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(bt.total_q * cs, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, topk_cluster_kernel, bt, scores, ld, K, out);
}

}  // namespace dsa
