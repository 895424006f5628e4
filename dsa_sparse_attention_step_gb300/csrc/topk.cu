// topk.cu -- exact top-k over the indexer scores.
//
// "vLLM's Kimi K3.1 Pro day-0 support", section "What changed": the indexer
// keeps the top 2048 tokens; section "Fused low-latency decode for DSA
// layers": an exact top-k selection follows the scorer.
//
// For query token t with `vis` visible positions (vis > k): the k positions
// with the largest scores, ties to the lower position, written in ascending
// position order.  Scores are mapped to order-preserving uint32 keys (-0
// folded onto +0); tau denotes the k-th largest key.
//
// Four paths, by batch shape:
//   - rows of at most 32,768 positions: one CTA per query token with the row
//     resident in shared memory (topk_resident_kernel, below);
//   - at most 8 query tokens over longer rows: every row split over the whole
//     GPU by radix levels (topk_split_*, below);
//   - more query tokens over rows of at most 2^18 positions: a sampled
//     threshold, one candidate pass over all rows at once and a per-row exact
//     select (topk_rows.cu);
//   - otherwise one thread-block cluster of `cs` CTAs per query token, as
//     follows.  CTA r owns a contiguous, 32-aligned slice of the positions.
//   1. Threshold estimate.  A histogram over the top 12 key bits of a sample
//      (every 16th 32-position chunk of the slice; every position when the row
//      is resident) is summed over the cluster through distributed shared
//      memory, and the bin b_lo holding the sample's ~1.25k-th largest key
//      (exactly the k-th when every position is sampled) is chosen.
//   2. One pass over the slice copies every key in a bin >= b_lo, with its
//      position, into shared memory (warp-aggregated appends).
//   3. If the cluster holds at least k candidates (so every key >= tau is
//      among them) and nothing overflowed, CTA 0 gathers the candidates,
//      resolves tau exactly by radix select (digits of 12, 10, 10 bits) and
//      tells every CTA how many of its keys equal to tau it takes (lowest
//      positions first).  Otherwise an exact fallback resolves the digits by
//      passes over the whole slice.
//   4. Each CTA marks its selected positions in a bitmap and writes them in
//      order at its offset in the output row (block-wide scan).
// Global reads are 16-byte vectors, four in flight per thread.
#include <cstddef>

#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace dsa {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
constexpr int kBins = 4096;                   // first digit: 12 bits
constexpr int kSampleStride = 16;             // sample one 32-position chunk in 16
constexpr int kResidentMax = 32768;           // rows kept in shared memory
constexpr int kSliceMax = 1 << 18;            // streaming positions per CTA

template <bool kRes>
struct Cfg {
    static constexpr int kWords = kRes ? kResidentMax / 32 : kSliceMax / 32;
    static constexpr int kCand = kRes ? 4096 : 8192;
    static constexpr int kKeys = kRes ? kResidentMax : 4;
};

template <bool kRes>
struct TopkSmem {
    uint32_t hist[kBins];                      // this CTA's histogram (cluster-visible)
    uint32_t tot[kBins];                       // cluster-wide histogram
    uint32_t bits[Cfg<kRes>::kWords];          // selected positions of the slice
    uint32_t eqbits[Cfg<kRes>::kWords];        // positions whose key equals tau
    uint32_t cand_key[Cfg<kRes>::kCand];
    int32_t cand_pos[Cfg<kRes>::kCand];
    int32_t warp_tot[kWarps + 1];
    uint32_t xchg[16];                         // per-CTA values read or written by the cluster
    uint32_t s_digit, s_rem, s_count, s_flag;
    alignas(16) uint32_t keys[Cfg<kRes>::kKeys];  // resident rows: the order keys (16-B loads)
};
static_assert(offsetof(TopkSmem<true>, keys) % 16 == 0, "vector loads of the resident keys");

// Radix digits: bits 31..20, 19..10, 9..0 of the order key.
__device__ __forceinline__ int dig_shift(int level) { return level == 0 ? 20 : (level == 1 ? 10 : 0); }
__device__ __forceinline__ uint32_t dig_mask(int level) { return level == 0 ? 0xFFFu : 0x3FFu; }

// Block-wide exclusive prefix sum (1024 threads); *total gets the block sum.
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

// Shared-memory histogram increment (the atomic unit serialises only lanes
// of a warp that hit the same bin).
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool active) {
    if (active) atomicAdd(&hist[bin], 1u);
}

// Find digit d over nb bins of h with count(> d) < rem <= count(>= d): sets
// s_digit and s_rem (= rem minus the count above d).  All threads call it.
template <bool kRes>
__device__ void find_digit(TopkSmem<kRes>& S, const uint32_t* h, int nb, uint32_t rem) {
    const int per = nb / kThreads;  // 4 or 1
    const int tid = threadIdx.x;
    // thread tid owns the bins of descending rank [per*tid, per*tid + per)
    uint32_t part = 0;
    for (int i = 0; i < per; ++i) part += h[nb - 1 - (per * tid + i)];
    int tot;
    const uint32_t above = (uint32_t)block_excl_sum((int)part, S.warp_tot, &tot);
    if (above < rem && rem <= above + part) {
        uint32_t run = above;
        for (int i = 0; i < per; ++i) {
            const int bin = nb - 1 - (per * tid + i);
            if (run + h[bin] >= rem) {
                S.s_digit = (uint32_t)bin;
                S.s_rem = rem - run;
                break;
            }
            run += h[bin];
        }
    }
    __syncthreads();
}

// Sum the cluster's histograms into tot (cs > 1) or use the local one.
template <bool kRes>
__device__ const uint32_t* cluster_hist(TopkSmem<kRes>& S, cg::cluster_group& cluster, int cs,
                                        int nb) {
    if (cs == 1) {
        __syncthreads();
        return S.hist;
    }
    cluster.sync();
    for (int i = threadIdx.x; i < nb; i += kThreads) {
        uint32_t v[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
            v[r] = (r < cs) ? cluster.map_shared_rank(S.hist, r)[i] : 0u;
        uint32_t s = 0;
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) s += v[r];
        S.tot[i] = s;
    }
    cluster.sync();
    return S.tot;
}

// Visit the slice [lo, hi) in steps of 32 positions per thread: f(i, kv)
// gets, for u = 0..7, the keys of positions i[u] .. i[u]+3 (kv[u]); positions
// >= hi carry key 0 and must be masked by the caller.  Eight 16-byte loads per
// thread are in flight per step.  Called by every thread (warp-uniform).
constexpr int kVec = 8;
template <bool kRes, typename F>
__device__ __forceinline__ void sweep(const float* row, const uint32_t* keys, int lo, int hi,
                                      F&& f) {
    const int tid = threadIdx.x;
    for (int base = lo; base < hi; base += 4 * kVec * kThreads) {
        uint4 kv[kVec];
        int i[kVec];
#pragma unroll
        for (int u = 0; u < kVec; ++u) {
            i[u] = base + u * 4 * kThreads + 4 * tid;
            if (kRes) {
                kv[u] = (i[u] < hi) ? *reinterpret_cast<const uint4*>(keys + (i[u] - lo))
                                    : make_uint4(0u, 0u, 0u, 0u);
            } else {
                const float4 x = (i[u] < hi) ? __ldg(reinterpret_cast<const float4*>(row + i[u]))
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                kv[u] = make_uint4(order_key(x.x), order_key(x.y), order_key(x.z), order_key(x.w));
            }
        }
        f(i, kv);
    }
}

// Per-position form of sweep: g(pos, key, valid) for every position.
template <bool kRes, typename G>
__device__ __forceinline__ void sweep_each(const float* row, const uint32_t* keys, int lo, int hi,
                                           G&& g) {
    sweep<kRes>(row, keys, lo, hi, [&](const int (&i)[kVec], const uint4 (&kv)[kVec]) {
#pragma unroll
        for (int u = 0; u < kVec; ++u) {
            g(i[u] + 0, kv[u].x, i[u] + 0 < hi);
            g(i[u] + 1, kv[u].y, i[u] + 1 < hi);
            g(i[u] + 2, kv[u].z, i[u] + 2 < hi);
            g(i[u] + 3, kv[u].w, i[u] + 3 < hi);
        }
    });
}

// Block-ordered pass over the eq bitmap: keep the first `take` set bits (in
// position order) and add them to the selection bitmap.
template <bool kRes>
__device__ void take_lowest_eq(TopkSmem<kRes>& S, int nwords, int take) {
    int seen = 0;
    for (int w0 = 0; w0 < nwords; w0 += kThreads) {
        const int w = w0 + threadIdx.x;
        const uint32_t m0 = (w < nwords) ? S.eqbits[w] : 0u;
        int cnt;
        int r = seen + block_excl_sum(__popc(m0), S.warp_tot, &cnt);
        if (m0 && r < take) {
            uint32_t m = m0, keep = 0;
            while (m && r < take) {
                keep |= m & (~m + 1u);  // lowest set bit
                m &= m - 1;
                ++r;
            }
            S.bits[w] |= keep;
        }
        seen += cnt;
    }
    __syncthreads();
}

template <bool kRes>
__global__ void __launch_bounds__(kThreads, 1)
topk_kernel(BatchArgs bt, const float* __restrict__ scores, int64_t ld, int K,
            int32_t* __restrict__ out) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    TopkSmem<kRes>& S = *reinterpret_cast<TopkSmem<kRes>*>(smem_raw);
    cg::cluster_group cluster = cg::this_cluster();
    const int cs = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int t = blockIdx.x / cs;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    grid_dependents_launch();
    const int b = request_of(bt, t);
    int32_t* o = out + (int64_t)t * K;
    // uniform over the cluster: every CTA of token t takes the same branches
    const bool ok = token_ok(bt, b, t, nullptr);
    const int vis = ok ? visible_of(bt, b, t) : 0;
    grid_dependency_wait();  // the scores come from the previous kernel
    if (vis <= K) {
        if (rank == 0)
            for (int i = tid; i < K; i += kThreads) o[i] = (i < vis) ? i : -1;
        return;
    }
    const float* row = scores + (int64_t)t * ld;
    const int per = ((vis + cs - 1) / cs + 31) & ~31;  // 32-aligned slices
    const int lo = min(vis, rank * per);
    const int hi = min(vis, lo + per);
    const int nwords = (hi - lo + 31) / 32;
    constexpr int kCand = Cfg<kRes>::kCand;

    if (kRes) {
        sweep_each<false>(row, nullptr, lo, hi, [&](int pos, uint32_t key, bool valid) {
            if (valid) S.keys[pos - lo] = key;
        });
    }
    for (int i = tid; i < kBins; i += kThreads) S.hist[i] = 0;
    if (tid == 0) S.s_count = 0;
    __syncthreads();

    // ---- 1. threshold estimate from a sample -------------------------------
    int sampled = 0;
    if (kRes) {
        sweep_each<true>(row, S.keys, lo, hi, [&](int, uint32_t key, bool valid) {
            hist_add(S.hist, key >> 20, valid);
        });
        sampled = hi - lo;
    } else {
        // chunks 16*w + 512*u + 4096*j: every 16th chunk exactly once
        for (int c0 = warp * kSampleStride; c0 < nwords; c0 += kWarps * kSampleStride * 8) {
            float x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int pos = lo + 32 * (c0 + u * kWarps * kSampleStride) + lane;
                x[u] = (pos < hi) ? __ldg(row + pos) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int pos = lo + 32 * (c0 + u * kWarps * kSampleStride) + lane;
                hist_add(S.hist, order_key(x[u]) >> 20, pos < hi);
            }
        }
        for (int c = 0; c < nwords; c += kSampleStride) sampled += min(32, hi - (lo + 32 * c));
    }
    S.xchg[4] = (uint32_t)sampled;
    const uint32_t* th = cluster_hist(S, cluster, cs, kBins);
    uint32_t sampled_all = (uint32_t)sampled;
    if (cs > 1) {
        sampled_all = 0;
        for (int r = 0; r < cs; ++r) sampled_all += cluster.map_shared_rank(S.xchg, r)[4];
    }
    uint32_t need_s;
    if (sampled_all >= (uint32_t)vis) {
        need_s = (uint32_t)K;  // every position sampled: the exact threshold bin
    } else {
        // ceil(1.25 K sampled / vis) + 16 in exact integer arithmetic (the
        // FP64 units of this GPU are far too slow for per-thread use)
        const uint64_t num = 5ull * (uint64_t)K * sampled_all;
        const uint64_t den = 4ull * (uint64_t)vis;
        const uint64_t want = (num + den - 1) / den + 16ull;
        need_s = (want < (uint64_t)sampled_all) ? (uint32_t)want : sampled_all;
    }
    find_digit(S, th, kBins, need_s);
    const uint32_t key_lo = S.s_digit << 20;

    // ---- 2. candidates: every key in a bin >= b_lo -------------------------
    // A float compare against the smallest float of bin b_lo (order keys are
    // monotone in the float value); order keys are formed for the candidates
    // only, and a thread's write loop visits only its vectors that hold one.
    {
        const float thr = (key_lo == 0u) ? -INFINITY
                        : __uint_as_float((key_lo & 0x80000000u) ? (key_lo & 0x7FFFFFFFu) : ~key_lo);
        for (int base0 = lo; base0 < hi; base0 += 4 * kVec * kThreads) {
            float4 x[kVec];
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const int i0 = base0 + u * 4 * kThreads + 4 * tid;
                x[u] = (i0 < hi) ? __ldg(reinterpret_cast<const float4*>(row + i0))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            uint32_t mask = 0;  // bit 4u+e: element e of vector u is a candidate
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const int i0 = base0 + u * 4 * kThreads + 4 * tid;
                const float xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    mask |= (i0 + e < hi && xv[e] >= thr) ? (1u << (4 * u + e)) : 0u;
            }
            const int n = __popc(mask);
            int incl = n;
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o2);
                if (lane >= o2) incl += v;
            }
            const int wsum = __shfl_sync(0xffffffffu, incl, 31);
            if (wsum == 0) continue;
            int base = 0;
            if (lane == 31) base = (int)atomicAdd(&S.s_count, (uint32_t)wsum);
            base = __shfl_sync(0xffffffffu, base, 31) + incl - n;
            if (mask == 0u) continue;
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const uint32_t mu = (mask >> (4 * u)) & 0xFu;
                if (mu == 0u) continue;
                const int i0 = base0 + u * 4 * kThreads + 4 * tid;
                const float xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (mu & (1u << e)) {
                        if (base < kCand) {
                            S.cand_key[base] = order_key(xv[e]);
                            S.cand_pos[base] = i0 + e;
                        }
                        ++base;
                    }
                }
            }
        }
    }
    __syncthreads();
    const uint32_t ncand_raw = S.s_count;
    S.xchg[0] = ncand_raw;
    uint32_t total = ncand_raw, maxc = ncand_raw;
    if (cs > 1) {
        cluster.sync();
        total = 0;
        maxc = 0;
        for (int r = 0; r < cs; ++r) {
            const uint32_t v = cluster.map_shared_rank(S.xchg, r)[0];
            total += v;
            maxc = max(maxc, v);
        }
    }
    const bool fast = total >= (uint32_t)K && maxc <= (uint32_t)kCand && total <= (uint32_t)kCand;
    const int ncand = (int)min(ncand_raw, (uint32_t)kCand);

    int take = 0;
    if (fast) {
        // ---- 3. exact tau on the candidates (gathered in CTA 0) -------------
        if (cs > 1) {
            cluster.sync();  // every candidate list is complete
            if (rank == 0) {
                uint32_t off = (uint32_t)ncand;
                for (int r = 1; r < cs; ++r) {
                    const uint32_t n = cluster.map_shared_rank(S.xchg, r)[0];
                    const uint32_t* rk = cluster.map_shared_rank(S.cand_key, r);
                    const int32_t* rp = cluster.map_shared_rank(S.cand_pos, r);
                    for (uint32_t i = tid; i < n; i += kThreads) {
                        S.cand_key[off + i] = rk[i];
                        S.cand_pos[off + i] = rp[i];
                    }
                    off += n;
                }
            }
        }
        if (rank == 0) {
            __syncthreads();
            const int n_all = (int)total;
            uint32_t prefix = 0, pmask = 0, rem = (uint32_t)K;
            for (int level = 0; level < 3; ++level) {
                const int nb = (level == 0) ? kBins : 1024;
                for (int i = tid; i < nb; i += kThreads) S.hist[i] = 0;
                __syncthreads();
                for (int c0 = 0; c0 < n_all; c0 += kThreads) {
                    const int c = c0 + tid;
                    const uint32_t key = (c < n_all) ? S.cand_key[c] : 0u;
                    hist_add(S.hist, (key >> dig_shift(level)) & dig_mask(level),
                             c < n_all && (key & pmask) == prefix);
                }
                __syncthreads();
                find_digit(S, S.hist, nb, rem);
                prefix |= S.s_digit << dig_shift(level);
                pmask |= dig_mask(level) << dig_shift(level);
                rem = S.s_rem;
            }
            // keys equal to tau per source CTA (candidates are in rank order);
            // tot is free at this point: [0,8) counts, [8,16) first candidate
            if (tid < kMaxCluster) {
                S.tot[tid] = 0u;
                uint32_t first = 0;
                for (int r = 0; r < tid && r < cs; ++r)
                    first += (cs > 1) ? cluster.map_shared_rank(S.xchg, r)[0] : (uint32_t)ncand;
                S.tot[8 + tid] = (tid < cs) ? first : 0xFFFFFFFFu;
            }
            __syncthreads();
            for (int c = tid; c < n_all; c += kThreads) {
                if (S.cand_key[c] == prefix) {
                    int r = 0;
                    while (r + 1 < cs && (uint32_t)c >= S.tot[8 + r + 1]) ++r;
                    atomicAdd(&S.tot[r], 1u);
                }
            }
            __syncthreads();
            if (tid == 0) {
                uint32_t before = 0;
                for (int r = 0; r < cs; ++r) {
                    const uint32_t e = S.tot[r];
                    const uint32_t tk = rem > before ? min(e, rem - before) : 0u;
                    before += e;
                    uint32_t* x = (cs > 1) ? cluster.map_shared_rank(S.xchg, r) : S.xchg;
                    x[1] = prefix;
                    x[2] = tk;
                }
            }
        }
        if (cs > 1) cluster.sync();
        else __syncthreads();
        const uint32_t tau = S.xchg[1];
        take = (int)S.xchg[2];
        // ---- 4a. bitmap from this CTA's own candidates -----------------------
        for (int w = tid; w < nwords; w += kThreads) {
            S.bits[w] = 0u;
            S.eqbits[w] = 0u;
        }
        __syncthreads();
        for (int c = tid; c < ncand; c += kThreads) {
            const uint32_t key = S.cand_key[c];
            const int p = S.cand_pos[c] - lo;
            if (key > tau) atomicOr(&S.bits[p >> 5], 1u << (p & 31));
            else if (key == tau) atomicOr(&S.eqbits[p >> 5], 1u << (p & 31));
        }
        __syncthreads();
        take_lowest_eq(S, nwords, take);
    } else {
        // ---- 3'. exact fallback: digits by passes over the slice -------------
        uint32_t prefix = 0, pmask = 0, rem = (uint32_t)K;
        for (int level = 0; level < 3; ++level) {
            const int nb = (level == 0) ? kBins : 1024;
            if (cs > 1) cluster.sync();  // remote readers of the last histogram are done
            for (int i = tid; i < nb; i += kThreads) S.hist[i] = 0;
            __syncthreads();
            sweep_each<kRes>(row, kRes ? S.keys : nullptr, lo, hi,
                             [&](int, uint32_t key, bool valid) {
                hist_add(S.hist, (key >> dig_shift(level)) & dig_mask(level),
                         valid && (key & pmask) == prefix);
            });
            const uint32_t* h = cluster_hist(S, cluster, cs, nb);
            find_digit(S, h, nb, rem);
            prefix |= S.s_digit << dig_shift(level);
            pmask |= dig_mask(level) << dig_shift(level);
            rem = S.s_rem;
        }
        const uint32_t tau = prefix;
        // bitmaps of the keys above / equal to tau: a 32-position word spans 8
        // lanes of 4 positions; their nibbles are OR-combined by shuffles
        int eq_local = 0;
        sweep_each<kRes>(row, kRes ? S.keys : nullptr, lo, hi,
                         [&](int pos, uint32_t key, bool valid) {
            const int e = pos & 3;
            const int sh = 4 * (lane & 7) + e;
            unsigned gw = (valid && key > tau) ? (1u << sh) : 0u;
            unsigned ew = (valid && key == tau) ? (1u << sh) : 0u;
            eq_local += ew ? 1 : 0;
#pragma unroll
            for (int o2 = 1; o2 < 8; o2 <<= 1) {
                gw |= __shfl_xor_sync(0xffffffffu, gw, o2);
                ew |= __shfl_xor_sync(0xffffffffu, ew, o2);
            }
            const int word_pos = (pos & ~3) - 4 * (lane & 7);  // first position of the word
            if ((lane & 7) == 0 && word_pos < hi) {
                const int w = (word_pos - lo) >> 5;
                if (e == 0) {
                    S.bits[w] = gw;
                    S.eqbits[w] = ew;
                } else {
                    S.bits[w] |= gw;
                    S.eqbits[w] |= ew;
                }
            }
        });
        __syncthreads();
        int eq_tot;
        (void)block_excl_sum(eq_local, S.warp_tot, &eq_tot);
        S.xchg[3] = (uint32_t)eq_tot;
        uint32_t eq_before = 0;
        if (cs > 1) {
            cluster.sync();
            for (int r = 0; r < rank; ++r) eq_before += cluster.map_shared_rank(S.xchg, r)[3];
        }
        take = (int)(rem > eq_before ? min((uint32_t)eq_tot, rem - eq_before) : 0u);
        take_lowest_eq(S, nwords, take);
    }

    // ---- 4b. ordered output: this CTA's positions at its cluster offset ------
    int sel_local = 0;
    for (int w = tid; w < nwords; w += kThreads) sel_local += __popc(S.bits[w]);
    int sel_tot;
    (void)block_excl_sum(sel_local, S.warp_tot, &sel_tot);
    S.xchg[5] = (uint32_t)sel_tot;
    uint32_t off = 0;
    if (cs > 1) {
        cluster.sync();
        for (int r = 0; r < rank; ++r) off += cluster.map_shared_rank(S.xchg, r)[5];
    }
    const int wpt = (nwords + kThreads - 1) / kThreads;  // contiguous runs keep the order
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
    if (cs > 1) cluster.sync();  // no CTA leaves while others may read its shared memory
}

// ---------------------------------------------------------------------------
// Rows of at most 32768 visible positions: one CTA per query token, the whole
// row resident in shared memory.
//   A. Load the row once (every load in flight at the same time), store its
//      order keys, and build a 12-bit histogram over the row's key range
//      [kmin, kmax] (digit (key - kmin) >> sh, sh = bit length of kmax - kmin
//      minus 12): bins spread over the values actually present, so that few
//      lanes of a warp add to the same bin.
//   B. Bin b holding the k-th largest key, and rem = how many keys bin b must
//      still give.
//   C. Radix levels of up to 10 bits over the resident keys of bin b (the sh
//      bits below it) give tau, the k-th largest key, and eq_take, how many
//      keys equal to tau are selected.
//   D. Thread i owns positions [32i, 32i + 32): it selects the keys above tau
//      and, among those equal to tau, the lowest positions still needed (one
//      block-wide scan of packed counts), and writes them in order.
// Every pass stops at the row's visible length.  Keys are stored in 16-byte
// chunks permuted within groups of eight (chunk c at c ^ ((c >> 3) & 7)), so
// the strided passes of A/C and the contiguous per-thread reads of D are free
// of bank conflicts.
struct ResSmem {
    alignas(16) uint32_t keys[kResidentMax];
    uint32_t hist[kBins];
    uint32_t warp_tot[kWarps + 1];
    uint32_t wmin[kWarps], wmax[kWarps];
    uint32_t s_digit, s_rem, pad0, pad1;
};

__device__ __forceinline__ int swz_chunk(int c) { return c ^ ((c >> 3) & 7); }

// Block-wide exclusive prefix sum of unsigned values (1024 threads).
__device__ __forceinline__ uint32_t block_excl_sum_u(uint32_t v, uint32_t* warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t w = warp_tot[lane];
        uint32_t inc = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += u;
        }
        warp_tot[lane] = inc - w;
    }
    __syncthreads();
    return incl - v + warp_tot[warp];
}

// Digit d over nb bins of h with count(> d) < rem <= count(>= d): sets
// s_digit and s_rem (= rem minus the count above d).  All threads call it.
__device__ void res_find_digit(ResSmem& S, const uint32_t* h, int nb, uint32_t rem) {
    const int per = nb / kThreads;  // 4 or 1
    const int tid = threadIdx.x;
    uint32_t part = 0;
    for (int i = 0; i < per; ++i) part += h[nb - 1 - (per * tid + i)];
    const uint32_t above = block_excl_sum_u(part, S.warp_tot);
    if (above < rem && rem <= above + part) {
        uint32_t run = above;
        for (int i = 0; i < per; ++i) {
            const int bin = nb - 1 - (per * tid + i);
            if (run + h[bin] >= rem) {
                S.s_digit = (uint32_t)bin;
                S.s_rem = rem - run;
                break;
            }
            run += h[bin];
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1)
topk_resident_kernel(BatchArgs bt, const float* __restrict__ scores, int64_t ld, int K,
                     int32_t* __restrict__ out) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    ResSmem& S = *reinterpret_cast<ResSmem*>(smem_raw);
    const int t = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5;
    grid_dependents_launch();
    const int b = request_of(bt, t);
    int32_t* o = out + (int64_t)t * K;
    const bool ok = token_ok(bt, b, t, nullptr);
    const int vis = ok ? visible_of(bt, b, t) : 0;
    for (int i = tid; i < kBins; i += kThreads) S.hist[i] = 0;
    grid_dependency_wait();  // the scores come from the previous kernel
    if (vis <= K) {
        for (int i = tid; i < K; i += kThreads) o[i] = (i < vis) ? i : -1;
        return;
    }
    __syncthreads();
    const float* row = scores + (int64_t)t * ld;
    constexpr int kChunksPerThread = kResidentMax / 4 / kThreads;  // 8
    // strided passes: chunk c = tid + 1024u holds positions 4c..4c+3; a warp
    // stops once its first chunk lies past the row
    const int nchunk = (vis + 3) / 4;
    auto warp_live = [&](int u) { return 32 * warp + kThreads * u < nchunk; };

    // ---- A. load, order keys, key range, 12-bit histogram over the range ----
    {
        uint32_t k[kChunksPerThread][4];
        uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
        for (int u = 0; u < kChunksPerThread; ++u) {
            const int c = tid + kThreads * u;
            // positions 4c..4c+3 lie below round_up(vis, 4) <= ld
            const float4 x = (c < nchunk) ? __ldg(reinterpret_cast<const float4*>(row) + c)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
            const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) k[u][e] = order_key(xv[e]);
        }
#pragma unroll
        for (int u = 0; u < kChunksPerThread; ++u) {
            const int c = tid + kThreads * u;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (4 * c + e < vis) {
                    kmin = min(kmin, k[u][e]);
                    kmax = max(kmax, k[u][e]);
                }
            }
            if (warp_live(u))
                *reinterpret_cast<uint4*>(&S.keys[4 * swz_chunk(c)]) =
                    make_uint4(k[u][0], k[u][1], k[u][2], k[u][3]);
        }
        kmin = __reduce_min_sync(0xffffffffu, kmin);
        kmax = __reduce_max_sync(0xffffffffu, kmax);
        if ((tid & 31) == 0) {
            S.wmin[warp] = kmin;
            S.wmax[warp] = kmax;
        }
        __syncthreads();
        kmin = 0xFFFFFFFFu;
        kmax = 0u;
#pragma unroll 8
        for (int w = 0; w < kWarps; ++w) {
            kmin = min(kmin, S.wmin[w]);
            kmax = max(kmax, S.wmax[w]);
        }
        S.pad0 = kmin;  // every thread writes the same value
        const int bits = 32 - __clz((int)(kmax - kmin));
        const int sh = bits > 12 ? bits - 12 : 0;
        S.pad1 = (uint32_t)sh;
#pragma unroll
        for (int u = 0; u < kChunksPerThread; ++u) {
            if (!warp_live(u)) break;
            const int c = tid + kThreads * u;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (4 * c + e < vis) atomicAdd(&S.hist[(k[u][e] - kmin) >> sh], 1u);
        }
    }
    __syncthreads();

    // ---- B. the bin of the k-th largest key --------------------------------
    const uint32_t kbase = S.pad0;
    int low = (int)S.pad1;  // bits of the key range below the bin
    res_find_digit(S, S.hist, kBins, (uint32_t)K);
    uint32_t vpre = S.s_digit << low;  // key - kbase of the bin's lower edge
    uint32_t rem = S.s_rem;

    // ---- C. radix levels of up to 10 bits below the bin --------------------
    while (low > 0) {
        const int shift = low > 10 ? low - 10 : 0;
        const int w = low - shift;
        for (int i = tid; i < 1024; i += kThreads) S.hist[i] = 0;
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kChunksPerThread; ++u) {
            if (!warp_live(u)) break;
            const int c = tid + kThreads * u;
            const uint4 kv = *reinterpret_cast<const uint4*>(&S.keys[4 * swz_chunk(c)]);
            const uint32_t k4[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t v = k4[e] - kbase;
                if (4 * c + e < vis && k4[e] >= kbase && (v >> low) == (vpre >> low))
                    atomicAdd(&S.hist[(v >> shift) & ((1u << w) - 1u)], 1u);
            }
        }
        __syncthreads();
        res_find_digit(S, S.hist, 1024, rem);
        vpre |= S.s_digit << shift;
        rem = S.s_rem;
        low = shift;
    }
    const uint32_t tau = kbase + vpre;
    const uint32_t eq_take = rem;  // keys equal to tau that are selected (lowest positions)

    // ---- D. ordered output --------------------------------------------------
    uint32_t mgt = 0, meq = 0;
    if (32 * 32 * warp < vis) {  // the warp's 1024 positions start inside the row
#pragma unroll
        for (int j = 0; j < kChunksPerThread; ++j) {
            const int c = kChunksPerThread * tid + j;
            const uint4 kv = *reinterpret_cast<const uint4*>(&S.keys[4 * swz_chunk(c)]);
            const uint32_t k4[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool valid = 4 * c + e < vis;
                mgt |= (valid && k4[e] > tau) ? (1u << (4 * j + e)) : 0u;
                meq |= (valid && k4[e] == tau) ? (1u << (4 * j + e)) : 0u;
            }
        }
    }
    // counts packed as (eq << 16) | gt: per-row totals stay below 2^16 each
    const uint32_t before = block_excl_sum_u((uint32_t)__popc(mgt) | ((uint32_t)__popc(meq) << 16),
                                             S.warp_tot);
    const uint32_t gt_before = before & 0xFFFFu, eq_before = before >> 16;
    uint32_t take = eq_take > eq_before ? min(eq_take - eq_before, (uint32_t)__popc(meq)) : 0u;
    uint32_t sel = mgt;
    for (uint32_t m = meq; take > 0; --take) {
        sel |= m & (~m + 1u);  // lowest remaining equal position
        m &= m - 1;
    }
    int pos = (int)(gt_before + min(eq_before, eq_take));
    const int p0 = 32 * tid;
    while (sel) {
        const int j = __ffs(sel) - 1;
        o[pos++] = p0 + j;
        sel &= sel - 1;
    }
}

// ---------------------------------------------------------------------------
// Split-row top-k, for a few query tokens over long rows: P CTAs per row, each
// owning a contiguous slice (a multiple of 4 positions), so that every SM
// works on the few rows.  Four kernels, each one pass over its slice (the rows
// stay in L2 between them):
//   L1   histogram of key bits 31..20 -> the bin d1 holding the k-th largest
//   L2   keys above d1 counted; histogram of bits 19..8 of the keys in d1 -> d2;
//        the keys in d1 are also appended to a list of up to 4096 (low 20 key
//        bits, slice).  When the list holds all of them, the last CTA resolves
//        tau and the per-slice counts from it in shared memory, and the L3
//        kernel writes the output instead (OUT then returns at once).
//   L3   keys of d1 above d2 counted; histogram of bits 7..0 of the keys whose
//        top 24 bits are (d1, d2) -> tau, and how many keys equal to tau are
//        taken (the lowest positions); every CTA stores the suffix sums of its
//        own level-3 histogram
//   OUT  every CTA adds up the counts of the CTAs before it (keys above tau,
//        keys equal to tau: two suffix-sum entries and two counts each) and
//        writes its selected positions in order at its offset
// Each level's row histogram is accumulated in the workspace with atomics (the
// accumulators are cleared by a memset before L1), and the last CTA of the row
// to finish its atomics (counter incremented after a memory fence) resolves the
// digit; no CTA ever waits for another.
constexpr int kSplitThreads = 512;
constexpr int kSplitWarps = kSplitThreads / 32;
constexpr int kSplitVec = 4;                    // float4 loads in flight per thread
constexpr int kSplitMinSlice = 2048;            // positions per CTA, at least
constexpr int kSplitMaxRows = 8;
constexpr int kSplitMinSeq = kResidentMax + 1;  // shorter rows: resident kernel
// accumulators per row (cleared): h1[4096], h2[4096], h3[256], done[3], list length
constexpr int kAccH1 = 0, kAccH2 = 4096, kAccH3 = 8192, kAccDone = 8448, kAccCand = 8451,
              kAccWords = 8456;
constexpr int kSplitCand = 4096;  // candidate list of the threshold bin
// per-row words after all rows' accumulators: state[8], cnt[P][2], suf[P][257],
// cand[kSplitCand]
__host__ __device__ constexpr size_t split_row_words(int P) {
    return 8 + (size_t)P * 259 + kSplitCand;
}

struct SplitArgs {
    BatchArgs bt;
    const float* scores;
    int64_t ld;
    int K;
    int32_t* out;
    uint32_t* ws;
    int P;  // CTAs per row
};

struct SplitRow {
    int vis, lo, hi;
    uint32_t* acc;   // cleared accumulators of the row
    uint32_t* st;    // state[8]: d1, rem1, d2, rem2, tau, rem3
    uint32_t* cnt;   // [P][2]: keys above d1; keys of d1 above (d1, d2)
    uint32_t* suf;   // [P][257]: suffix sums of each CTA's level-3 histogram
    uint32_t* cand;  // [kSplitCand]: (key bits 19..0) << 12 | slice, keys in d1
    int per;         // positions per slice
};

__device__ __forceinline__ SplitRow split_row(const SplitArgs& a, int t, int c) {
    SplitRow g;
    const int b = request_of(a.bt, t);
    g.vis = token_ok(a.bt, b, t, nullptr) ? visible_of(a.bt, b, t) : 0;
    const int per = ((g.vis + a.P - 1) / a.P + 3) & ~3;
    g.lo = min(g.vis, c * per);
    g.hi = min(g.vis, g.lo + per);
    g.acc = a.ws + (size_t)t * kAccWords;
    uint32_t* rest = a.ws + (size_t)a.bt.total_q * kAccWords + (size_t)t * split_row_words(a.P);
    g.st = rest;
    g.cnt = rest + 8;
    g.suf = g.cnt + 2 * a.P;
    g.cand = g.suf + 257 * a.P;
    g.per = per;
    return g;
}

// f(pos, key, valid) over the slice, kSplitVec 16-byte loads in flight per
// thread (positions past hi are read inside the row's padding and masked).
template <typename F>
__device__ __forceinline__ void split_pass(const float* row, int lo, int hi, F&& f) {
    for (int base = lo; base < hi; base += 4 * kSplitVec * kSplitThreads) {
        float4 x[kSplitVec];
#pragma unroll
        for (int u = 0; u < kSplitVec; ++u) {
            const int i0 = base + 4 * (u * kSplitThreads + (int)threadIdx.x);
            x[u] = (i0 < hi) ? __ldg(reinterpret_cast<const float4*>(row + i0))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kSplitVec; ++u) {
            const int i0 = base + 4 * (u * kSplitThreads + (int)threadIdx.x);
            f(i0 + 0, order_key(x[u].x), i0 + 0 < hi);
            f(i0 + 1, order_key(x[u].y), i0 + 1 < hi);
            f(i0 + 2, order_key(x[u].z), i0 + 2 < hi);
            f(i0 + 3, order_key(x[u].w), i0 + 3 < hi);
        }
    }
}

// Block-wide exclusive sum over kSplitThreads threads; *total gets the sum.
__device__ __forceinline__ uint32_t split_excl_sum(uint32_t v, uint32_t* warp_tot, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t w = (lane < kSplitWarps) ? warp_tot[lane] : 0u;
        uint32_t inc = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += u;
        }
        if (lane < kSplitWarps) warp_tot[lane] = inc - w;
        if (lane == 31) warp_tot[kSplitWarps] = inc;
    }
    __syncthreads();
    const uint32_t r = incl - v + warp_tot[warp];
    *total = warp_tot[kSplitWarps];
    __syncthreads();
    return r;
}

// Flush this CTA's histogram into the row's accumulator, then report whether
// this CTA is the row's last to do so (its atomics, and every other CTA's, are
// then visible to it).
__device__ __forceinline__ bool split_flush_last(const uint32_t* hist, int nb, uint32_t* acc_h,
                                                 uint32_t* done, int P, int* s_last) {
    for (int i = threadIdx.x; i < nb; i += kSplitThreads)
        if (hist[i]) atomicAdd(&acc_h[i], hist[i]);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *s_last = (atomicAdd(done, 1u) == (uint32_t)(P - 1)) ? 1 : 0;
    __syncthreads();
    if (*s_last) __threadfence();
    return *s_last != 0;
}

// Digit d over the nb = kPer * kSplitThreads (or fewer) bins of the row
// histogram h (read once from L2) with count(> d) < rem <= count(>= d); writes
// d and rem - count(> d) to s_out.
template <int kPer, bool kGlobal = true>
__device__ __forceinline__ void split_find(const uint32_t* h, int nb, uint32_t rem,
                                           uint32_t* warp_tot, uint32_t* s_out) {
    const int tid = threadIdx.x;
    uint32_t v[kPer], part = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int r = kPer * tid + i;  // descending rank of the bin
        v[i] = (r < nb) ? (kGlobal ? __ldcg(h + nb - 1 - r) : h[nb - 1 - r]) : 0u;
        part += v[i];
    }
    uint32_t tot;
    const uint32_t above = split_excl_sum(part, warp_tot, &tot);
    if (above < rem && rem <= above + part) {
        uint32_t run = above;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            if (run < rem && run + v[i] >= rem) {
                s_out[0] = (uint32_t)(nb - 1 - (kPer * tid + i));
                s_out[1] = rem - run;
            }
            run += v[i];
        }
    }
    __syncthreads();
}

__device__ __forceinline__ uint32_t split_block_sum(uint32_t v, uint32_t* warp_tot) {
    uint32_t tot;
    split_excl_sum(v, warp_tot, &tot);
    return tot;
}

// The ordered output of slice c of row t: every CTA adds up the counts of the
// CTAs before it (keys above tau and keys equal to tau) and writes its
// selected positions in ascending order at its offset.
__device__ __forceinline__ void split_output(const SplitArgs& a, const SplitRow& g, int t, int c,
                                             uint32_t* warp_tot) {
    int32_t* o = a.out + (int64_t)t * a.K;
    // thread i owns 16 consecutive positions of each 8192-position chunk; the
    // first chunk's loads are issued before the counts are read
    const float* row = a.scores + (size_t)t * a.ld;
    float4 x[4];
    auto load = [&](int base) {
        const int p0 = base + 16 * (int)threadIdx.x;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            x[u] = (p0 + 4 * u < g.hi) ? __ldg(reinterpret_cast<const float4*>(row + p0 + 4 * u))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    load(g.lo);
    const uint32_t tau = __ldcg(g.st + 4), rem3 = __ldcg(g.st + 5);
    const uint32_t d3 = tau & 0xFFu;
    // keys above tau and keys equal to tau of slice cc
    auto counts = [&](int cc, uint32_t* gt, uint32_t* eq) {
        const uint32_t s0 = __ldcg(g.suf + 257 * cc + d3), s1 = __ldcg(g.suf + 257 * cc + d3 + 1);
        *gt = __ldcg(g.cnt + 2 * cc) + __ldcg(g.cnt + 2 * cc + 1) + s1;
        *eq = s0 - s1;
    };
    uint32_t gb = 0, eb = 0;
    for (int cc = threadIdx.x; cc < c; cc += kSplitThreads) {
        uint32_t gv, ev;
        counts(cc, &gv, &ev);
        gb += gv;
        eb += ev;
    }
    const uint32_t gt_before = split_block_sum(gb, warp_tot);
    const uint32_t eq_before = split_block_sum(eb, warp_tot);
    uint32_t my_gt, my_eq;
    counts(c, &my_gt, &my_eq);
    const uint32_t my_take = rem3 > eq_before ? min(my_eq, rem3 - eq_before) : 0u;
    const uint32_t base_out = gt_before + min(eq_before, rem3);
    uint32_t gt_run = 0, eq_run = 0;
    for (int base = g.lo; base < g.hi; base += 16 * kSplitThreads) {
        const int p0 = base + 16 * (int)threadIdx.x;
        if (base != g.lo) load(base);
        uint32_t gm = 0, em = 0;  // bit j: position p0 + j is above / equal to tau
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = 4 * u + e;
                if (p0 + j < g.hi) {
                    const uint32_t key = order_key(xv[e]);
                    gm |= (key > tau) ? (1u << j) : 0u;
                    em |= (key == tau) ? (1u << j) : 0u;
                }
            }
        }
        uint32_t tot;
        const uint32_t pre = split_excl_sum(((uint32_t)__popc(em) << 16) | (uint32_t)__popc(gm),
                                            warp_tot, &tot);
        uint32_t eq_seen = eq_run + (pre >> 16);
        uint32_t pos = base_out + gt_run + (pre & 0xFFFFu) + min(eq_seen, my_take);
        for (uint32_t m = gm | em; m; m &= m - 1) {
            const int j = __ffs(m) - 1;
            // (pos < K always holds: the per-CTA counts add up to K exactly)
            if (gm & (1u << j)) {
                if (pos < (uint32_t)a.K) o[pos] = p0 + j;
                ++pos;
            } else {
                if (eq_seen < my_take) {
                    if (pos < (uint32_t)a.K) o[pos] = p0 + j;
                    ++pos;
                }
                ++eq_seen;
            }
        }
        gt_run += tot & 0xFFFFu;
        eq_run += tot >> 16;
    }
}

__global__ void __launch_bounds__(kSplitThreads) topk_split_l1(SplitArgs a) {
    __shared__ uint32_t hist[4096];
    __shared__ uint32_t warp_tot[kSplitWarps + 1];
    __shared__ uint32_t s_out[2];
    __shared__ int s_last;
    grid_dependents_launch();
    const int t = blockIdx.x / a.P, c = blockIdx.x % a.P;
    grid_dependency_wait();  // the scores come from the previous kernel
    const SplitRow g = split_row(a, t, c);
    if (g.vis <= a.K) return;  // the same for every CTA of the row
    for (int i = threadIdx.x; i < 4096; i += kSplitThreads) hist[i] = 0;
    __syncthreads();
    split_pass(a.scores + (size_t)t * a.ld, g.lo, g.hi, [&](int, uint32_t key, bool v) {
        if (v) atomicAdd(&hist[key >> 20], 1u);
    });
    __syncthreads();
    if (!split_flush_last(hist, 4096, g.acc + kAccH1, g.acc + kAccDone + 0, a.P, &s_last)) return;
    split_find<4096 / kSplitThreads>(g.acc + kAccH1, 4096, (uint32_t)a.K, warp_tot, s_out);
    if (threadIdx.x == 0) {
        g.st[0] = s_out[0];
        g.st[1] = s_out[1];
    }
}

__global__ void __launch_bounds__(kSplitThreads) topk_split_l2(SplitArgs a) {
    __shared__ uint32_t hist[4096];
    __shared__ uint32_t hsm[1024];
    __shared__ uint32_t warp_tot[kSplitWarps + 1];
    __shared__ uint32_t s_out[2];
    __shared__ int s_last;
    __shared__ volatile int s_full;
    grid_dependents_launch();
    const int t = blockIdx.x / a.P, c = blockIdx.x % a.P;
    grid_dependency_wait();
    const SplitRow g = split_row(a, t, c);
    if (g.vis <= a.K) return;
    const uint32_t d1 = __ldcg(g.st + 0), rem1 = __ldcg(g.st + 1);
    for (int i = threadIdx.x; i < 4096; i += kSplitThreads) hist[i] = 0;
    if (threadIdx.x == 0) s_full = 0;
    __syncthreads();
    uint32_t gt = 0;
    split_pass(a.scores + (size_t)t * a.ld, g.lo, g.hi, [&](int pos, uint32_t key, bool v) {
        const uint32_t b1 = key >> 20;
        gt += (v && b1 > d1) ? 1u : 0u;
        if (v && b1 == d1) {  // rare: the keys of the threshold bin
            atomicAdd(&hist[(key >> 8) & 0xFFFu], 1u);
            // append to the list; once a CTA sees it full it stops appending
            if (!s_full) {
                const uint32_t slot = atomicAdd(g.acc + kAccCand, 1u);
                if (slot < (uint32_t)kSplitCand) g.cand[slot] = ((key & 0xFFFFFu) << 12) | (uint32_t)c;
                else s_full = 1;
            }
        }
    });
    gt = split_block_sum(gt, warp_tot);
    if (threadIdx.x == 0) g.cnt[2 * c + 0] = gt;
    __syncthreads();
    if (!split_flush_last(hist, 4096, g.acc + kAccH2, g.acc + kAccDone + 1, a.P, &s_last)) return;
    const uint32_t ncand = __ldcg(g.acc + kAccCand);
    if (ncand > (uint32_t)kSplitCand) {  // the list overflowed: level 3 resolves tau
        split_find<4096 / kSplitThreads>(g.acc + kAccH2, 4096, rem1, warp_tot, s_out);
        if (threadIdx.x == 0) {
            g.st[2] = s_out[0];
            g.st[3] = s_out[1];
            g.st[6] = 0u;
        }
        return;
    }
    // tau from the list: bits 19..10, then 9..0 of the keys in d1
    uint32_t* cl = hist;  // the list (this CTA's histogram is flushed)
    for (int i = threadIdx.x; i < (int)ncand; i += kSplitThreads) cl[i] = __ldcg(g.cand + i);
    for (int i = threadIdx.x; i < 1024; i += kSplitThreads) hsm[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < (int)ncand; i += kSplitThreads) atomicAdd(&hsm[cl[i] >> 22], 1u);
    __syncthreads();
    split_find<1024 / kSplitThreads, false>(hsm, 1024, rem1, warp_tot, s_out);
    const uint32_t da = s_out[0], rema = s_out[1];
    for (int i = threadIdx.x; i < 1024; i += kSplitThreads) hsm[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < (int)ncand; i += kSplitThreads)
        if ((cl[i] >> 22) == da) atomicAdd(&hsm[(cl[i] >> 12) & 0x3FFu], 1u);
    __syncthreads();
    split_find<1024 / kSplitThreads, false>(hsm, 1024, rema, warp_tot, s_out);
    const uint32_t tau20 = (da << 10) | s_out[0], rem3 = s_out[1];
    const uint32_t tau = (d1 << 20) | tau20;
    // per slice: keys of d1 above tau (hsm[0, P)) and keys equal to tau
    // (hsm[512, 512 + P)), written where the output kernel reads them
    for (int i = threadIdx.x; i < 1024; i += kSplitThreads) hsm[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < (int)ncand; i += kSplitThreads) {
        const uint32_t k20 = cl[i] >> 12, sl = cl[i] & 0xFFFu;
        if (k20 > tau20) atomicAdd(&hsm[sl], 1u);
        else if (k20 == tau20) atomicAdd(&hsm[512 + sl], 1u);
    }
    __syncthreads();
    const uint32_t d3 = tau & 0xFFu;
    for (int cc = threadIdx.x; cc < a.P; cc += kSplitThreads) {
        g.cnt[2 * cc + 1] = hsm[cc];
        g.suf[257 * cc + d3] = hsm[512 + cc];
        g.suf[257 * cc + d3 + 1] = 0u;
    }
    if (threadIdx.x == 0) {
        g.st[4] = tau;
        g.st[5] = rem3;
        g.st[6] = 1u;
    }
}

__global__ void __launch_bounds__(kSplitThreads) topk_split_l3(SplitArgs a) {
    __shared__ uint32_t hist[256];
    __shared__ uint32_t warp_tot[kSplitWarps + 1];
    __shared__ uint32_t s_out[2];
    __shared__ int s_last;
    grid_dependents_launch();
    const int t = blockIdx.x / a.P, c = blockIdx.x % a.P;
    grid_dependency_wait();
    const SplitRow g = split_row(a, t, c);
    if (g.vis <= a.K) return;
    if (__ldcg(g.st + 6)) {  // tau resolved from the list: write the output
        split_output(a, g, t, c, warp_tot);
        return;
    }
    const uint32_t d1 = __ldcg(g.st + 0), d2 = __ldcg(g.st + 2), rem2 = __ldcg(g.st + 3);
    const uint32_t p24 = (d1 << 12) | d2;
    for (int i = threadIdx.x; i < 256; i += kSplitThreads) hist[i] = 0;
    __syncthreads();
    uint32_t gt = 0;
    split_pass(a.scores + (size_t)t * a.ld, g.lo, g.hi, [&](int, uint32_t key, bool v) {
        const uint32_t k24 = key >> 8;
        gt += (v && (key >> 20) == d1 && k24 > p24) ? 1u : 0u;
        if (v && k24 == p24) atomicAdd(&hist[key & 0xFFu], 1u);
    });
    gt = split_block_sum(gt, warp_tot);
    if (threadIdx.x == 0) g.cnt[2 * c + 1] = gt;
    {   // suf[b] = keys of this slice in level-3 bins >= b (suf[256] = 0):
        // thread i < 256 takes bin 255 - i of a scan in descending bin order
        const int i = threadIdx.x;
        const uint32_t hv = (i < 256) ? hist[255 - i] : 0u;
        uint32_t tot;
        const uint32_t ex = split_excl_sum(hv, warp_tot, &tot);
        if (i < 256) g.suf[257 * c + 255 - i] = ex + hv;
        if (i == 0) g.suf[257 * c + 256] = 0u;
    }
    if (!split_flush_last(hist, 256, g.acc + kAccH3, g.acc + kAccDone + 2, a.P, &s_last)) return;
    split_find<1>(g.acc + kAccH3, 256, rem2, warp_tot, s_out);
    if (threadIdx.x == 0) {
        g.st[4] = (p24 << 8) | s_out[0];
        g.st[5] = s_out[1];
    }
}

__global__ void __launch_bounds__(kSplitThreads) topk_split_out(SplitArgs a) {
    __shared__ uint32_t warp_tot[kSplitWarps + 1];
    grid_dependents_launch();
    const int t = blockIdx.x / a.P, c = blockIdx.x % a.P;
    int32_t* o = a.out + (int64_t)t * a.K;
    grid_dependency_wait();
    const SplitRow g = split_row(a, t, c);
    if (g.vis <= a.K) {  // every visible position, then -1
        const int chunk = (a.K + a.P - 1) / a.P;
        for (int i = c * chunk + (int)threadIdx.x; i < min(a.K, (c + 1) * chunk); i += kSplitThreads)
            o[i] = (i < g.vis) ? i : -1;
        return;
    }
    if (__ldcg(g.st + 6)) return;  // written by the level-3 kernel
    split_output(a, g, t, c, warp_tot);
}

// CTAs per row of the split path.
int split_ctas(int total_q, int max_seq) {
    const int by_sm = 152 / (total_q > 0 ? total_q : 1);
    const int by_len = (max_seq + kSplitMinSlice - 1) / kSplitMinSlice;
    const int p = by_sm < by_len ? by_sm : by_len;
    return p > 0 ? p : 1;
}

bool use_split(int total_q, int max_seq) {
    return total_q <= kSplitMaxRows && max_seq >= kSplitMinSeq;
}

cudaError_t launch_split(const BatchArgs& bt, const float* scores, int64_t ld, int K,
                         int32_t* out, void* ws, bool pdl, cudaStream_t stream) {
    SplitArgs a;
    a.bt = bt;
    a.scores = scores;
    a.ld = ld;
    a.K = K;
    a.out = out;
    a.ws = static_cast<uint32_t*>(ws);
    a.P = split_ctas(bt.total_q, bt.max_seq);
    const dim3 grid((unsigned)(bt.total_q * a.P));
    cudaError_t e = cudaMemsetAsync(ws, 0, (size_t)bt.total_q * kAccWords * sizeof(uint32_t), stream);
    (void)pdl;  // the first kernel follows the memset
    if (e == cudaSuccess) e = launch_kernel(topk_split_l1, grid, dim3(kSplitThreads), 0, stream, false, 1, a);
    if (e == cudaSuccess) e = launch_kernel(topk_split_l2, grid, dim3(kSplitThreads), 0, stream, true, 1, a);
    if (e == cudaSuccess) e = launch_kernel(topk_split_l3, grid, dim3(kSplitThreads), 0, stream, true, 1, a);
    if (e == cudaSuccess) e = launch_kernel(topk_split_out, grid, dim3(kSplitThreads), 0, stream, true, 1, a);
    return e;
}

cudaError_t launch_streaming(const BatchArgs& bt, const float* scores, int64_t ld, int K,
                             int32_t* out, int cs, bool pdl, cudaStream_t stream) {
    const size_t smem = sizeof(TopkSmem<false>);
    cudaError_t e = cudaFuncSetAttribute(topk_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(topk_kernel<false>, dim3(bt.total_q * cs), dim3(kThreads), smem, stream,
                         pdl, cs, bt, scores, ld, K, out);
}

cudaError_t launch_resident(const BatchArgs& bt, const float* scores, int64_t ld, int K,
                            int32_t* out, bool pdl, cudaStream_t stream) {
    const size_t smem = sizeof(ResSmem);
    cudaError_t e = cudaFuncSetAttribute(topk_resident_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(topk_resident_kernel, dim3(bt.total_q), dim3(kThreads), smem, stream, pdl,
                         1, bt, scores, ld, K, out);
}

}  // namespace

bool topk_rows_eligible(int total_q, int max_seq, bool split);
size_t topk_rows_workspace_bytes(int total_q);
cudaError_t launch_topk_rows(const BatchArgs& bt, const float* scores, int64_t ld, int K,
                             int32_t* out, void* ws, bool pdl, cudaStream_t stream);

// CTAs per query token for rows that stream from global memory: spread few
// tokens over more SMs, and keep every slice within the per-CTA bitmap.
int topk_cluster_size(int total_q, int max_seq) {
    int cs = 1;
    while (cs < kMaxCluster && total_q * cs * 2 <= 152) cs <<= 1;
    while (cs < kMaxCluster && (max_seq + cs - 1) / cs > kSliceMax) cs <<= 1;
    return cs;
}

bool topk_supported(int max_seq) { return max_seq <= kSliceMax * kMaxCluster; }

// Device scratch of the top-k: the split path's histograms and counts, or the
// many-rows path's thresholds and candidate lists.
size_t topk_workspace_bytes(int total_q, int max_seq) {
    if (topk_rows_eligible(total_q, max_seq, use_split(total_q, max_seq)))
        return topk_rows_workspace_bytes(total_q);
    if (!use_split(total_q, max_seq)) return 0;
    return ((size_t)total_q * kAccWords +
            (size_t)total_q * split_row_words(split_ctas(total_q, max_seq))) * sizeof(uint32_t);
}

int topk_launches(int total_q, int max_seq) {
    if (use_split(total_q, max_seq)) return 4;
    return topk_rows_eligible(total_q, max_seq, false) ? 3 : 1;
}

cudaError_t launch_topk(const BatchArgs& bt, const float* scores, int64_t ld, int K,
                        int32_t* out, void* ws, bool pdl, cudaStream_t stream) {
    if (bt.total_q == 0) return cudaSuccess;
    if (use_split(bt.total_q, bt.max_seq)) return launch_split(bt, scores, ld, K, out, ws, pdl, stream);
    if (topk_rows_eligible(bt.total_q, bt.max_seq, false))
        return launch_topk_rows(bt, scores, ld, K, out, ws, pdl, stream);
    if (bt.max_seq <= kResidentMax) return launch_resident(bt, scores, ld, K, out, pdl, stream);
    return launch_streaming(bt, scores, ld, K, out, topk_cluster_size(bt.total_q, bt.max_seq), pdl,
                            stream);
}

}  // namespace dsa
