// dcp.cu -- decode context parallelism (DCP) for the sparse indexer, emulated
// on one GPU: the exact one-round top-k merge and the log-sum-exp combine.
//
// "vLLM's Kimi K3.1 Pro day-0 support", section "Decode context parallelism
// with the sparse indexer": with DCP over W ranks, rank r stores every W-th
// token (positions s = r mod W) and ranks only its own tokens, so the global
// top-2048 must be merged across ranks before attention, and the partial
// attention outputs are combined by log-sum-exp.  Section "Exact top-k merge
// with about 10x less traffic": each rank selects its best ceil(1.5 * 2048 /
// W) candidates directly from BF16 scores and packs each with its score into
// 32 bits; every rank radix-selects the same global top-2048 from the gathered
// candidates; a rank holding more of the top-2048 than it sent is detected by
// that selection and resends its full local top-k for the row.
//
// Here the W ranks' shards are the interleaved positions of one score row on
// one GPU, and an exchange buffer in device memory stands for what the ranks
// put on the wire.  A candidate word is (k << 16) | i: k = the order-preserving
// 16-bit key of the BF16-rounded score, i = the position within the rank's
// shard (s = i * W + r).  The merged order is BF16 score descending, position
// ascending.
//
// Kernels (launched in this order, each one CTA per query row):
//   dcp_candidates_kernel<false>  every rank's top `cand`: a list of the
//                                 rank's tokens at or above a sampled key
//                                 threshold (or all of them), then a radix
//                                 select on (k << 16) | (0xFFFF - i), four
//                                 8-bit levels, over the list (over the whole
//                                 row when the list missed)
//   dcp_merge_kernel<false>       the top-k of the gathered candidates (radix
//                                 select on 48-bit (k, ~s) keys in shared
//                                 memory); a rank all of whose candidates are
//                                 selected while it holds more tokens is
//                                 flagged; a row without flags is final
//   dcp_candidates_kernel<true>   flagged ranks only: their local top-k
//   dcp_merge_kernel<true>        flagged rows only: the top-k of the flagged
//                                 ranks' full lists and the others' candidates
// A rank that is not flagged has its lowest candidate outside the top-k of a
// subset of all tokens, hence outside the global top-k, and so are its unsent
// tokens (they rank below that candidate); so the second selection is exact.
#include <climits>

#include "common.cuh"
#include "sm100.cuh"

namespace dsa {

using namespace sm100;

namespace {

constexpr int kDcpThreads = 1024;
constexpr int kDcpMaxWorld = 8;
constexpr int kDcpPool = 24576;   // first round: candidate words of all ranks of a row (96 KB)
constexpr int kDcpSamples = 4;    // first round: sampled positions per thread, at most
constexpr int kStageRounds = 3;   // row passes: rounds of vectors in flight per thread
// dynamic shared memory of the candidate kernel: the first round's list pool,
// then the row passes' staging ring (two 16-byte vectors per thread and round)
constexpr size_t kCandSmem = (size_t)kDcpPool * 4 + (size_t)kStageRounds * 2 * 16 * kDcpThreads;

// Wait until at most n of this thread's cp.async groups are pending.
template <int n>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(n) : "memory");
}

// Order-preserving 16-bit key of a score rounded to BF16 (round to nearest
// even), -0 folded onto +0.
__device__ __forceinline__ uint32_t bf16_key(float f) {
    uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(f));
    if (b == 0x8000u) b = 0u;
    return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}

struct DcpArgs {
    BatchArgs bt;
    const float* scores;
    int64_t ld;
    int world;
    int cand;               // candidates per rank
    int K;                  // selected per row
    uint32_t* sent;         // [T][W][cand]
    int32_t* sent_n;        // [T][W]
    uint32_t* full;         // [T][W][K]  flagged ranks' local top-k
    int32_t* full_n;        // [T][W]
    int32_t* flags;         // [T][W]
    int32_t* indices;       // [T][K]
    int32_t* rank_indices;  // [W][T][K] or null
    int32_t* resent;        // [T][W] or null
};

// Warp-wide, over hist[0..256): the digit d with count(> d) < need <=
// count(>= d), and count(> d); returned to every lane.  Lane l sums bins
// 255-8l .. 248-8l (descending digits), then a warp scan locates the lane.
__device__ __forceinline__ void find_digit(const uint32_t* hist, uint32_t need, int lane,
                                           uint32_t& digit, uint32_t& above) {
    uint32_t v[8], sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        v[j] = hist[255 - 8 * lane - j];
        sum += v[j];
    }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const uint32_t excl = incl - sum;
    const uint32_t ballot = __ballot_sync(0xffffffffu, excl < need && need <= incl);
    const int src = ballot ? __ffs(ballot) - 1 : 0;
    uint32_t d = 0, c = excl;
    if (lane == src) {
        int j = 0;
        while (j < 7 && c + v[j] < need) c += v[j++];
        d = 255u - 8u * (uint32_t)lane - (uint32_t)j;
    }
    digit = __shfl_sync(0xffffffffu, d, src);
    above = __shfl_sync(0xffffffffu, c, src);
}

// Shared-memory histogram increment aggregated over the warp: lanes with the
// same bin are counted by one atomic (the top digits of BF16 keys take few
// distinct values, so unaggregated atomics would serialise on a few bins).
// Called by every lane of the warp; `active` lanes contribute.
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool active, int lane) {
    const unsigned am = __ballot_sync(0xffffffffu, active);
    if (active) {
        const unsigned peers = __match_any_sync(am, bin);
        if ((int)(__ffs(peers) - 1) == lane) atomicAdd(hist + bin, (uint32_t)__popc(peers));
    }
}

// Append `val` to rank r's list (pool + r * cap, count in lcnt[r]); words
// past the list's capacity are counted but not stored.  (Few lanes append
// at a time, so plain shared atomics do.)
__device__ __forceinline__ void list_append(uint32_t* pool, int cap, int* lcnt, int r, uint32_t val) {
    const int slot = atomicAdd(lcnt + r, 1);
    if (slot < cap) pool[r * cap + slot] = val;
}

// Radix select by one warp of the c largest (unique) words of list[0, n),
// four 8-bit levels with a histogram of the warp's own (hist, 256 bins);
// returns the c-th largest word, tau, to every lane.
__device__ __forceinline__ uint32_t warp_list_select(const uint32_t* list, int n, uint32_t c,
                                                     uint32_t* hist, int lane) {
    uint32_t prefix = 0u, need = c;
    for (int level = 0; level < 4; ++level) {
        const int shift = 24 - 8 * level;
        const uint32_t hi_mask = level == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
        for (int i = lane; i < 256; i += 32) hist[i] = 0u;
        __syncwarp();
        for (int j = lane; j < n; j += 32) {
            const uint32_t wv = list[j];
            if ((wv & hi_mask) == (prefix & hi_mask)) atomicAdd(hist + ((wv >> shift) & 255u), 1u);
        }
        __syncwarp();
        uint32_t d, above;
        find_digit(hist, need, lane, d, above);
        prefix |= d << shift;
        need -= above;
        __syncwarp();
    }
    return prefix;
}

// Rank and rank-local index of position s (shifts when W is a power of two).
__device__ __forceinline__ void rank_of(int s, int W, int lw, int& r, uint32_t& i) {
    if (lw >= 0) {
        r = s & (W - 1);
        i = (uint32_t)(s >> lw);
    } else {
        r = s % W;
        i = (uint32_t)(s / W);
    }
}

// Local top-C of every rank of row t (kResend: only flagged ranks, C = K).
//
// First round: a rank with at most `cap` tokens lists them all; for a larger
// rank, a sample of the row (every stride-th 32-position chunk) gives a BF16
// key threshold at about the 2 C-th largest of its tokens, and one pass over
// the row lists the rank's tokens at or above it.  The C best of a list are
// found by a radix select over the list in shared memory.  A list that holds
// fewer than C tokens or overflows falls back to the radix select over the
// whole row, which the resend round (flagged ranks, C = K) always uses.  The
// threshold only decides which path a rank takes: the result is exact either
// way.
template <bool kResend>
__global__ void __launch_bounds__(kDcpThreads) dcp_candidates_kernel(const DcpArgs a) {
    extern __shared__ uint4 s_dyn[];      // kCandSmem bytes
    uint32_t* s_pool = reinterpret_cast<uint32_t*>(s_dyn);  // first round: the ranks' candidate lists
    __shared__ uint32_t s_hist[kDcpMaxWorld][256];
    __shared__ uint32_t s_prefix[kDcpMaxWorld];
    __shared__ uint32_t s_need[kDcpMaxWorld];
    __shared__ int s_cnt[kDcpMaxWorld];
    __shared__ int s_lcnt[kDcpMaxWorld];          // tokens listed
    __shared__ uint32_t s_keylo[kDcpMaxWorld];    // list threshold (16-bit key)
    __shared__ uint32_t s_d1[kDcpMaxWorld], s_need2[kDcpMaxWorld];
    // 0: idle, 1: select (first round: over its list; resend: over the row),
    // 2: take all, 3: first round, select over the row
    __shared__ int s_mode[kDcpMaxWorld];
    __shared__ int s_samp[kDcpMaxWorld];          // threshold from the sample
    const int t = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int W = a.world;
    const int C = kResend ? a.K : a.cand;
    const int b = request_of(a.bt, t);
    if (!token_ok(a.bt, b, t, nullptr)) return;
    const int vis = visible_of(a.bt, b, t);
    const float* row = a.scores + (int64_t)t * a.ld;
    const int lw = (W & (W - 1)) == 0 ? __ffs(W) - 1 : -1;
    const int cap = min(8 * C, kDcpPool / W);  // first round: list capacity per rank
    if (tid < W) {
        const int r = tid;
        const int n_r = vis > r ? (vis - 1 - r) / W + 1 : 0;
        const int c = min(C, n_r);
        const bool on = !kResend || a.flags[(int64_t)t * W + r] != 0;
        s_mode[r] = !on ? 0 : (c == n_r ? 2 : 1);
        s_samp[r] = (!kResend && s_mode[r] == 1 && n_r > cap) ? 1 : 0;
        s_prefix[r] = 0u;
        s_need[r] = (uint32_t)c;
        s_cnt[r] = 0;
        s_lcnt[r] = 0;
        s_keylo[r] = 0u;
        if (on) (kResend ? a.full_n : a.sent_n)[(int64_t)t * W + r] = c;
    }
    __syncthreads();
    bool any = false, radix = false, samp = false;
    for (int r = 0; r < W; ++r) {
        any |= s_mode[r] != 0;
        radix |= s_mode[r] == 1;
        samp |= s_samp[r] != 0;
    }
    if (!any) return;
    uint32_t* out = kResend ? a.full : a.sent;
    const int stride = kResend ? a.K : a.cand;
    // One pass over the row's visible positions: every thread loads two
    // 16-byte vectors per round (rows are 16-byte aligned and score_ld is a
    // multiple of 4, so a vector starting below vis stays in the row; values
    // at or past vis are never used), then every lane calls body(s, f, valid,
    // e) for each of its eight positions (e = s % 4), in step with the warp.
    // The vectors go through a ring of kStageRounds rounds in shared memory
    // (cp.async, each thread into slots of its own, so only its own waits
    // order them): a round is consumed while the next two are in flight.
    float4* stg = reinterpret_cast<float4*>(s_pool + kDcpPool);  // [round % 3][2][threads]
    auto row_pass = [&](auto&& body) {
        constexpr int kRound = 8 * kDcpThreads;
        const int nround = (vis + kRound - 1) / kRound;
        auto issue = [&](int rd) {  // every thread commits one group per round, maybe empty
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int s0 = rd * kRound + 4 * (tid + q * kDcpThreads);
                if (rd < nround && s0 < vis)
                    cp_async16(stg + ((rd % kStageRounds) * 2 + q) * kDcpThreads + tid, row + s0);
            }
            cp_async_commit();
        };
        for (int rd = 0; rd < kStageRounds - 1; ++rd) issue(rd);
        for (int rd = 0; rd < nround; ++rd) {  // warp-uniform trip count
            cp_async_wait_group<kStageRounds - 2>();  // round rd has landed
            float4 v[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) v[q] = stg[((rd % kStageRounds) * 2 + q) * kDcpThreads + tid];
            issue(rd + kStageRounds - 1);  // into the slots of round rd - 1, already read
            const int base = rd * kRound;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int s0 = base + 4 * (tid + q * kDcpThreads);
                body(s0 + 0, v[q].x, s0 + 0 < vis, 0);
                body(s0 + 1, v[q].y, s0 + 1 < vis, 1);
                body(s0 + 2, v[q].z, s0 + 2 < vis, 2);
                body(s0 + 3, v[q].w, s0 + 3 < vis, 3);
            }
        }
        cp_async_wait_group<0>();  // no copy lands after the pass
    };
    if (!kResend) {
        if (samp) {
            // ---- thresholds: the n_s-th largest sampled key of each sampling
            // rank, n_s = ceil(3 c samples / n_r), found in two 8-bit levels
            const int nch = (vis + 31) / 32;
            const int cstride = max(8, (nch + 32 * kDcpSamples - 1) / (32 * kDcpSamples));
            uint32_t key[kDcpSamples];
            int rk[kDcpSamples];
#pragma unroll
            for (int u = 0; u < kDcpSamples; ++u) {
                const int ch = (warp + 32 * u) * cstride;
                const int sp = 32 * ch + lane;
                rk[u] = -1;
                key[u] = 0u;
                if (ch < nch && sp < vis) {
                    int r;
                    uint32_t i;
                    rank_of(sp, W, lw, r, i);
                    if (s_samp[r]) {
                        rk[u] = r;
                        key[u] = bf16_key(__ldcg(row + sp));
                    }
                }
            }
            for (int i = tid; i < W * 256; i += kDcpThreads) (&s_hist[0][0])[i] = 0u;
            __syncthreads();
#pragma unroll
            for (int u = 0; u < kDcpSamples; ++u)
                hist_add(&s_hist[0][0], (uint32_t)max(rk[u], 0) * 256u + (key[u] >> 8), rk[u] >= 0, lane);
            __syncthreads();
            if (warp < W && s_samp[warp]) {
                uint32_t tot = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) tot += s_hist[warp][8 * lane + j];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
                const int n_r = (vis - 1 - warp) / W + 1;
                const uint32_t c = s_need[warp];
                uint32_t ns = (uint32_t)((3ull * c * tot + (uint64_t)n_r - 1) / (uint64_t)n_r);
                ns = max(1u, min(ns, tot));
                uint32_t d = 0, above = 0;
                if (tot > 0) find_digit(s_hist[warp], ns, lane, d, above);
                if (lane == 0) {
                    s_d1[warp] = d;
                    s_need2[warp] = ns - above;
                    if (tot == 0) s_samp[warp] = 0;  // no sample: list from key 0 (may overflow)
                }
            }
            __syncthreads();
            for (int i = tid; i < W * 256; i += kDcpThreads) (&s_hist[0][0])[i] = 0u;
            __syncthreads();
#pragma unroll
            for (int u = 0; u < kDcpSamples; ++u) {
                const bool in = rk[u] >= 0 && s_samp[max(rk[u], 0)] && (key[u] >> 8) == s_d1[max(rk[u], 0)];
                hist_add(&s_hist[0][0], (uint32_t)max(rk[u], 0) * 256u + (key[u] & 255u), in, lane);
            }
            __syncthreads();
            if (warp < W && s_samp[warp]) {
                uint32_t d, above;
                find_digit(s_hist[warp], s_need2[warp], lane, d, above);
                if (lane == 0) s_keylo[warp] = (s_d1[warp] << 8) | d;
            }
            __syncthreads();
        }
        // ---- one pass over the row: the lists, and every token of the
        // take-all ranks written out.  With W a power of two a thread's four
        // consecutive positions always fall on the same four ranks (vectors
        // start at multiples of 4, rounds at multiples of 8192), whose mode
        // and threshold it keeps in registers (threshold 0x10000: no list).
        uint32_t klo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = lw >= 0 ? ((4 * tid + e) & (W - 1)) : 0;
            klo[e] = s_mode[r] == 1 ? s_keylo[r] : (s_mode[r] == 2 ? 0u : 0x10000u);
        }
        row_pass([&](int s, float f, bool valid, int e) {
            if (!valid) return;
            int r;
            uint32_t i;
            rank_of(s, W, lw, r, i);
            const uint32_t k = bf16_key(f);
            const uint32_t lo = lw >= 0 ? klo[e]
                                        : (s_mode[r] == 1 ? s_keylo[r] : (s_mode[r] == 2 ? 0u : 0x10000u));
            if (k < lo) return;
            if (s_mode[r] == 2) {
                const int slot = atomicAdd(&s_cnt[r], 1);
                if (slot < stride) out[((int64_t)t * W + r) * stride + slot] = (k << 16) | i;
            } else {
                list_append(s_pool, cap, s_lcnt, r, (k << 16) | (0xFFFFu - i));
            }
        });
        __syncthreads();
        // a list that missed: the rank selects over the whole row instead
        if (tid < W && s_mode[tid] == 1 && (s_lcnt[tid] < (int)s_need[tid] || s_lcnt[tid] > cap))
            s_mode[tid] = 3;
        __syncthreads();
        // ---- the c largest words of each list: warp r selects on list r
        // (histogram in its row of s_hist), then the CTA writes them out
        if (warp < W && s_mode[warp] == 1) {
            const uint32_t tau =
                warp_list_select(s_pool + warp * cap, s_lcnt[warp], s_need[warp], s_hist[warp], lane);
            if (lane == 0) s_prefix[warp] = tau;
        }
        __syncthreads();
        for (int r = 0; r < W; ++r) {
            if (s_mode[r] != 1) continue;
            const int n = s_lcnt[r];
            const uint32_t tau = s_prefix[r];
            for (int j = tid; j < n; j += kDcpThreads) {
                const uint32_t wv = s_pool[r * cap + j];
                if (wv >= tau) {
                    const int slot = atomicAdd(&s_cnt[r], 1);
                    if (slot < stride)
                        out[((int64_t)t * W + r) * stride + slot] = (wv & 0xFFFF0000u) | (0xFFFFu - (wv & 0xFFFFu));
                }
            }
        }
        radix = false;
        for (int r = 0; r < W; ++r) radix |= s_mode[r] == 3;
    }
    // ---- radix select over the whole row (resend round; first-round ranks
    // whose list missed), on comp = (k << 16) | (0xFFFF - i): the C largest
    // are the best C of the rank (larger score, then lower position); the
    // composite is unique per token, so the C-th largest, tau, selects
    // exactly C
    const int kRow = kResend ? 1 : 3;
    for (int level = 0; radix && level < 4; ++level) {
        const int shift = 24 - 8 * level;
        const uint32_t hi_mask = level == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
        for (int i = tid; i < W * 256; i += kDcpThreads) (&s_hist[0][0])[i] = 0u;
        __syncthreads();
        row_pass([&](int s, float f, bool valid, int) {
            bool act = false;
            uint32_t bin = 0;
            if (valid) {
                int r;
                uint32_t i;
                rank_of(s, W, lw, r, i);
                if (s_mode[r] == kRow) {
                    const uint32_t comp = (bf16_key(f) << 16) | (0xFFFFu - i);
                    act = (comp & hi_mask) == (s_prefix[r] & hi_mask);
                    bin = (uint32_t)r * 256u + ((comp >> shift) & 255u);
                }
            }
            hist_add(&s_hist[0][0], bin, act, lane);
        });
        __syncthreads();
        if (warp < W && s_mode[warp] == kRow) {
            uint32_t d, above;
            find_digit(s_hist[warp], s_need[warp], lane, d, above);
            if (lane == 0) {
                s_prefix[warp] |= d << shift;
                s_need[warp] -= above;
            }
        }
        __syncthreads();
    }
    // output: every token of a row-select rank with comp >= tau, and (resend
    // round) every token of a take-all rank
    if (!radix && !kResend) return;
    row_pass([&](int s, float f, bool valid, int) {
        if (!valid) return;
        int r;
        uint32_t i;
        rank_of(s, W, lw, r, i);
        const int mode = s_mode[r];
        if (mode == 0 || (!kResend && mode != 3)) return;
        const uint32_t k = bf16_key(f);
        const uint32_t comp = (k << 16) | (0xFFFFu - i);
        const uint32_t tau = mode == 2 ? 0u : s_prefix[r];
        if (comp >= tau) {
            const int slot = atomicAdd(&s_cnt[r], 1);
            if (slot < stride) out[((int64_t)t * W + r) * stride + slot] = (k << 16) | i;
        }
    });
}

// Block-wide exclusive scan of one int per thread (1024 threads); returns the
// exclusive prefix and sets *total.
__device__ __forceinline__ int block_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int x = s_warp[lane];
        int wi = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        s_warp[lane] = wi - x;
        if (lane == 31) s_warp[32] = wi;
    }
    __syncthreads();
    const int r = s_warp[warp] + incl - v;
    *total = s_warp[32];
    __syncthreads();
    return r;
}

// Shared memory of the merge: this struct, then the candidate area -- the
// gathered keys (k << 32) | (0xFFFFFFFF - s), later the row's position bitmap
// -- sized per round by merge_cand_bytes.
struct MergeSmem {
    int pos[kTopK];                        // selected positions, sorted
    uint32_t hist[256];
    int warp_tot[33];
    int off[kDcpMaxWorld + 1];
    int taken[kDcpMaxWorld];
    int flag[kDcpMaxWorld];
    unsigned long long prefix;
    uint32_t need;
    int count;
    int any_flag;
};
constexpr size_t kMergeFixed = (sizeof(MergeSmem) + 15) / 16 * 16;

// Candidate-area bytes of a merge round: its gathered words (round 1: at most
// `cand` per rank; round 2: a flagged rank's full top-K) or the bitmap of the
// longest row, whichever is larger.
size_t merge_cand_bytes(bool second, int world, int cand, int K, int max_seq) {
    const size_t words = (size_t)world * (second ? K : cand) * sizeof(unsigned long long);
    const size_t bitmap = (size_t)(max_seq + 31) / 32 * sizeof(uint32_t);
    return ((words > bitmap ? words : bitmap) + 15) / 16 * 16;
}

// Top-K of the gathered candidates of row t.  Round 1 (kSecond = false): all
// ranks' candidates; ranks whose candidates were all selected while they hold
// more tokens are flagged, and a row without flags writes its outputs.
// Round 2: rows with flags, flagged ranks contributing their local top-K.
template <bool kSecond>
__global__ void __launch_bounds__(kDcpThreads) dcp_merge_kernel(const DcpArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    MergeSmem& sm = *reinterpret_cast<MergeSmem*>(smem_raw);
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(smem_raw + kMergeFixed);
    const int t = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int W = a.world;
    const int b = request_of(a.bt, t);
    if (!token_ok(a.bt, b, t, nullptr)) return;
    const int vis = visible_of(a.bt, b, t);
    if (tid == 0) {
        int any = 0, o = 0;
        for (int r = 0; r < W; ++r) {
            const int f = kSecond ? a.flags[(int64_t)t * W + r] : 0;
            sm.flag[r] = f;
            any |= f;
            sm.off[r] = o;
            o += f ? a.full_n[(int64_t)t * W + r] : a.sent_n[(int64_t)t * W + r];
            sm.taken[r] = 0;
        }
        sm.off[W] = o;
        sm.any_flag = any;
        sm.prefix = 0ull;
        sm.count = 0;
    }
    __syncthreads();
    if (kSecond && !sm.any_flag) return;  // final after round 1
    const int N = sm.off[W];
    // gather the candidate words into (k << 32) | ~s keys
    for (int r = 0; r < W; ++r) {
        const int n = sm.off[r + 1] - sm.off[r];
        const uint32_t* src = sm.flag[r] ? a.full + ((int64_t)t * W + r) * a.K
                                         : a.sent + ((int64_t)t * W + r) * a.cand;
        for (int j = tid; j < n; j += kDcpThreads) {
            const uint32_t w = __ldcg(src + j);
            const uint32_t s = (w & 0xFFFFu) * (uint32_t)W + (uint32_t)r;
            cand[sm.off[r] + j] = ((unsigned long long)(w >> 16) << 32) | (0xFFFFFFFFu - s);
        }
    }
    const int K = min(a.K, N);
    if (tid == 0) sm.need = (uint32_t)K;
    __syncthreads();
    // radix select of the K-th largest over 48 bits (six 8-bit levels);
    // keys are unique, so exactly K keys are >= it
    if (K < N) {
        for (int level = 0; level < 6; ++level) {
            const int shift = 40 - 8 * level;
            const unsigned long long hi_mask = level == 0 ? 0ull : (~0ull << (shift + 8));
            if (tid < 256) sm.hist[tid] = 0u;
            __syncthreads();
            for (int base = 0; base < N; base += kDcpThreads) {  // warp-uniform trip count
                const int j = base + tid;
                const unsigned long long c = j < N ? cand[j] : 0ull;
                const bool act = j < N && (c & hi_mask) == (sm.prefix & hi_mask);
                hist_add(sm.hist, (uint32_t)((c >> shift) & 255u), act, lane);
            }
            __syncthreads();
            if (warp == 0) {
                uint32_t d, above;
                find_digit(sm.hist, sm.need, lane, d, above);
                if (lane == 0) {
                    sm.prefix |= (unsigned long long)d << shift;
                    sm.need -= above;
                }
            }
            __syncthreads();
        }
    }
    const unsigned long long tau = K < N ? sm.prefix : 0ull;
    for (int j = tid; j < N; j += kDcpThreads) {
        const unsigned long long c = cand[j];
        if (c >= tau) {
            const int s = (int)(0xFFFFFFFFu - (uint32_t)(c & 0xFFFFFFFFull));
            const int slot = atomicAdd(&sm.count, 1);
            if (slot < kTopK) sm.pos[slot] = s;
            if (!kSecond) atomicAdd(&sm.taken[s % W], 1);
        }
    }
    __syncthreads();
    if (!kSecond) {
        if (tid == 0) {
            int any = 0;
            for (int r = 0; r < W; ++r) {
                const int n_r = vis > r ? (vis - 1 - r) / W + 1 : 0;
                const int sr = sm.off[r + 1] - sm.off[r];
                const int f = (sr > 0 && sm.taken[r] == sr && n_r > sr) ? 1 : 0;
                a.flags[(int64_t)t * W + r] = f;
                if (a.resent) a.resent[(int64_t)t * W + r] = f;
                any |= f;
            }
            sm.any_flag = any;
        }
        __syncthreads();
        if (sm.any_flag) return;  // round 2 finishes this row
    }
    // the K positions in ascending order: marked in a bitmap of the row's
    // positions (in the candidate area, no longer read), then every thread
    // ranks the set bits of its run of words by one block-wide scan
    {
        uint32_t* bm = reinterpret_cast<uint32_t*>(cand);
        const int nwords = (vis + 31) >> 5;  // the area holds the longest row's bitmap
        for (int j = tid; j < nwords; j += kDcpThreads) bm[j] = 0u;
        __syncthreads();
        for (int j = tid; j < K; j += kDcpThreads) {
            const int s = sm.pos[j];
            atomicOr(bm + (s >> 5), 1u << (s & 31));
        }
        __syncthreads();
        const int per = (nwords + kDcpThreads - 1) / kDcpThreads;
        const int w0 = min(tid * per, nwords), w1 = min(w0 + per, nwords);
        int mine = 0;
        for (int j = w0; j < w1; ++j) mine += __popc(bm[j]);
        int total;
        int o = block_scan(mine, sm.warp_tot, &total);
        for (int j = w0; j < w1; ++j)
            for (uint32_t m = bm[j]; m != 0u; m &= m - 1u) sm.pos[o++] = 32 * j + __ffs(m) - 1;
        __syncthreads();
    }
    for (int j = tid; j < a.K; j += kDcpThreads)
        a.indices[(int64_t)t * a.K + j] = j < K ? sm.pos[j] : -1;
    if (a.rank_indices) {
        // each rank's share of the selection, ascending, -1 padded
        constexpr int kPer = kTopK / kDcpThreads;  // 2 positions per thread
        for (int r = 0; r < W; ++r) {
            int mine = 0;
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int j = kPer * tid + u;
                mine += (j < K && sm.pos[j] % W == r);
            }
            int total;
            int o = block_scan(mine, sm.warp_tot, &total);
            int32_t* dst = a.rank_indices + ((int64_t)r * a.bt.total_q + t) * a.K;
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int j = kPer * tid + u;
                if (j < K && sm.pos[j] % W == r) dst[o++] = sm.pos[j];
            }
            for (int j = total + tid; j < a.K; j += kDcpThreads) dst[j] = -1;
        }
    }
}

// out[t,h,:] = sum_r exp(lse_r - L) part_r[t,h,:], L = log sum_r exp(lse_r);
// thread = (row (t, h), 8 dims): one 16-byte load per rank, all in flight.
constexpr int kCombThreads = 128;  // two (t, h) rows per block
__global__ void __launch_bounds__(kCombThreads)
dcp_lse_combine_kernel(int total_q, int world, const __nv_bfloat16* __restrict__ part,
                       const float* __restrict__ part_lse, __nv_bfloat16* __restrict__ out,
                       float* __restrict__ lse) {
    const int64_t rows = (int64_t)total_q * kMlaHeads;
    const int64_t row = (int64_t)blockIdx.x * 2 + (threadIdx.x >> 6);
    if (row >= rows) return;
    const int d0 = 8 * (threadIdx.x & 63);
    float l[kDcpMaxWorld];
    uint4 v[kDcpMaxWorld];
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < kDcpMaxWorld; ++r) {
        l[r] = r < world ? __ldg(part_lse + (int64_t)r * rows + row) : -INFINITY;
        v[r] = r < world ? __ldg(reinterpret_cast<const uint4*>(part + ((int64_t)r * rows + row) * kVDim + d0))
                         : make_uint4(0u, 0u, 0u, 0u);
        M = fmaxf(M, l[r]);
    }
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float tot = 0.f;
    if (M > -INFINITY) {
#pragma unroll
        for (int r = 0; r < kDcpMaxWorld; ++r) {
            const float wgt = __expf(l[r] - M);  // 0 for an absent or empty rank
            tot += wgt;
            const uint32_t wv[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                acc[2 * k] = fmaf(wgt, __uint_as_float(wv[k] << 16), acc[2 * k]);
                acc[2 * k + 1] = fmaf(wgt, __uint_as_float(wv[k] & 0xFFFF0000u), acc[2 * k + 1]);
            }
        }
    }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 p2 = __floats2bfloat162_rn(acc[2 * k] * inv, acc[2 * k + 1] * inv);
        o[k] = *reinterpret_cast<const uint32_t*>(&p2);
    }
    *reinterpret_cast<uint4*>(out + row * kVDim + d0) = make_uint4(o[0], o[1], o[2], o[3]);
    if (lse && d0 == 0) lse[row] = tot > 0.f ? M + __logf(tot) : -INFINITY;
}

}  // namespace

// ceil(1.5 K / W), capped at K (a rank never needs to send more than K)
int dcp_default_cand(int world, int K) {
    const int c = (3 * K + 2 * world - 1) / (2 * world);
    return c < K ? c : K;
}

struct DcpWs {
    size_t sent, sent_n, full, full_n, flags, total;
};

DcpWs dcp_ws_layout(int total_q, int world, int cand, int K) {
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    const size_t tw = (size_t)total_q * world;
    DcpWs w;
    w.sent = 0;
    w.sent_n = up(tw * cand * 4);
    w.full = w.sent_n + up(tw * 4);
    w.full_n = w.full + up(tw * (size_t)K * 4);
    w.flags = w.full_n + up(tw * 4);
    w.total = w.flags + up(tw * 4);
    return w;
}

bool dcp_supported(int world, int max_seq) {
    return world >= 1 && world <= kDcpMaxWorld && (int64_t)max_seq <= (int64_t)65536 * world;
}

cudaError_t launch_dcp_topk(const BatchArgs& bt, const float* scores, int64_t ld, int world,
                            int cand, int K, int32_t* indices, int32_t* rank_indices,
                            int32_t* resent, void* ws, cudaStream_t stream) {
    if (bt.total_q == 0) return cudaSuccess;
    const DcpWs w = dcp_ws_layout(bt.total_q, world, cand, K);
    uint8_t* base = static_cast<uint8_t*>(ws);
    DcpArgs a;
    a.bt = bt;
    a.scores = scores;
    a.ld = ld;
    a.world = world;
    a.cand = cand;
    a.K = K;
    a.sent = reinterpret_cast<uint32_t*>(base + w.sent);
    a.sent_n = reinterpret_cast<int32_t*>(base + w.sent_n);
    a.full = reinterpret_cast<uint32_t*>(base + w.full);
    a.full_n = reinterpret_cast<int32_t*>(base + w.full_n);
    a.flags = reinterpret_cast<int32_t*>(base + w.flags);
    a.indices = indices;
    a.rank_indices = rank_indices;
    a.resent = resent;
    const size_t msmem1 = kMergeFixed + merge_cand_bytes(false, world, cand, K, bt.max_seq);
    const size_t msmem2 = kMergeFixed + merge_cand_bytes(true, world, cand, K, bt.max_seq);
    cudaError_t e = cudaFuncSetAttribute(dcp_merge_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)msmem1);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(dcp_merge_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)msmem2);
    const dim3 grid((unsigned)bt.total_q);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(dcp_candidates_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kCandSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(dcp_candidates_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kCandSmem);
    if (e == cudaSuccess)
        e = launch_kernel(dcp_candidates_kernel<false>, grid, dim3(kDcpThreads), kCandSmem, stream, false,
                          1, a);
    if (e == cudaSuccess)
        e = launch_kernel(dcp_merge_kernel<false>, grid, dim3(kDcpThreads), msmem1, stream, false, 1, a);
    if (e == cudaSuccess)
        e = launch_kernel(dcp_candidates_kernel<true>, grid, dim3(kDcpThreads), kCandSmem, stream, false, 1,
                          a);
    if (e == cudaSuccess)
        e = launch_kernel(dcp_merge_kernel<true>, grid, dim3(kDcpThreads), msmem2, stream, false, 1, a);
    return e;
}

cudaError_t launch_lse_combine(int total_q, int world, const uint16_t* part, const float* part_lse,
                               uint16_t* out, float* lse, cudaStream_t stream) {
    const int64_t rows = (int64_t)total_q * kMlaHeads;
    if (rows == 0) return cudaSuccess;
    return launch_kernel(dcp_lse_combine_kernel, dim3((unsigned)((rows + 1) / 2)),
                         dim3(kCombThreads), 0, stream, false, 1, total_q, world,
                         reinterpret_cast<const __nv_bfloat16*>(part), part_lse,
                         reinterpret_cast<__nv_bfloat16*>(out), lse);
}

}  // namespace dsa
