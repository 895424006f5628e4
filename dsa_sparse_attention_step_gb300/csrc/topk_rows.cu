// topk_rows.cu -- exact top-k for batches of many long rows: every row is
// spread over the whole GPU by three short kernels.
//
// "vLLM's Kimi K3.1 Pro day-0 support", section "What changed" (the indexer
// keeps the top 2048 tokens) and section "Fused low-latency decode for DSA
// layers" (an exact top-k follows the scorer).  The result is the one every
// top-k path of this library gives: the k positions with the largest scores,
// ties to the lower position, in ascending position order; scores are
// compared through order-preserving uint32 keys (-0 folded onto +0).
//
// One CTA per row reads its row at a fraction of what an SM can draw while
// it also runs the row's sequential phases, and a batch of a few hundred rows
// leaves the last wave of such CTAs almost empty.  Here the row is cut into
// units of 8192 positions:
//   1. rows_threshold_kernel, one CTA per row: draws every S-th 32-position
//      chunk of the row (S >= 16, at most 128 chunks) and finds the bin of
//      the n_s-th largest sampled key, n_s = ceil(1.5 k sampled / vis) + 16,
//      among 4096 bins over the sampled key range (a second digit of 12 bits
//      splits that bin when it holds more than 8 samples); key_lo is the
//      bin's lower edge.  Rows with vis <= k are written out at once.
//   2. rows_candidates_kernel, two persistent CTAs per SM over the units of
//      all rows: appends each key >= key_lo and its position to the row's
//      candidate list (one global atomic per warp and unit reserves slots).
//   3. rows_select_kernel, one CTA per row: when the row holds n candidates
//      with k <= n <= kRowsCandMax, every key >= tau (the k-th largest key of
//      the row) is among them, and the candidates (held in registers) are
//      digited, 8 bits at a time over [key_lo, max key], until the bin of
//      tau holds at most 128 of them; those are ranked pairwise (key, then
//      position), which gives tau and, among keys equal to it, the last
//      position taken.  Otherwise the same select runs over the whole row
//      (exact fallback; a bin of many equal keys is settled by a radix
//      select over positions).  The selection is marked in a bitmap and each
//      selected position is written at its rank (per-word prefix counts).
// The sample only steers how many candidates there are: the result is exact
// whatever it draws.
#include <climits>
#include <cstddef>

#include "common.cuh"
#include "sm100.cuh"

namespace dsa {

using namespace sm100;

namespace {

constexpr int kRowsMaxSeq = 1 << 18;      // positions per row (the bitmap: 32 KB)
constexpr int kRowsMinSeq = 32769;        // shorter rows stay in one CTA's shared memory
constexpr int kRowsCandMax = 6144;        // candidates kept per row
constexpr int kBins0 = 4096;              // first digit: 12 bits
constexpr int kThrThreads = 256;
constexpr int kSampleChunks = 128;        // sampled 32-position chunks per row, at most
constexpr int kSampleStride = 16;         // sample at most one chunk in 16
constexpr int kUnit = 8192;               // positions per unit of the candidate pass (32 KB)
constexpr int kStages = 3;                // shared-memory ring of the candidate pass
constexpr int kConsWarps = 8;             // each takes 1024 positions of a unit
constexpr int kLaneVec = kUnit / kConsWarps / 128;  // 16-byte vectors per lane and unit
constexpr int kStreamThreads = 32 * (kConsWarps + 1);  // + one producer warp
constexpr uint32_t kCountPoison = 1u << 30;  // a count above any row's length
constexpr int kSelThreads = 256;
constexpr int kSelPer = kRowsCandMax / kSelThreads;   // candidates per select thread
constexpr int kRowVec = 8;                // 16-byte loads in flight per thread, whole-row select

static_assert(kRowsCandMax % kSelThreads == 0, "candidates split evenly over the select threads");
static_assert(kUnit == 128 * kLaneVec * kConsWarps, "units split evenly over the consumer lanes");
static_assert(4 * kLaneVec <= 32, "a lane's candidates fit one 32-bit mask");
static_assert((kUnit * 4) % 16 == 0, "bulk copies of whole 16-byte vectors");

struct RowInfo {
    int32_t vis;      // positions the row selects from; 0 once the row is written
    uint32_t key_lo;  // candidates are the keys >= key_lo
    uint32_t count;   // candidates appended (may exceed kRowsCandMax)
    uint32_t pad;
};

struct RowsArgs {
    BatchArgs bt;
    const float* scores;
    int64_t ld;
    int K;
    int32_t* out;
    RowInfo* info;         // [total_q]
    uint32_t* cand_key;    // [total_q][kRowsCandMax]
    int32_t* cand_pos;     // [total_q][kRowsCandMax]
    int units_per_row;
};

// Block-wide exclusive prefix sum over NT threads; *total gets the block sum.
// wsum holds NT/32 + 1 ints.  Every thread calls it.
template <int NT>
__device__ __forceinline__ int block_scan_excl(int v, int* wsum, int* total) {
    constexpr int kW = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = (lane < kW) ? wsum[lane] : 0;
        int inc = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += u;
        }
        if (lane < kW) wsum[lane] = inc - w;
        if (lane == kW - 1) wsum[kW] = inc;
    }
    __syncthreads();
    const int r = incl - v + wsum[warp];
    *total = wsum[kW];
    __syncthreads();
    return r;
}

// Histogram increment with the lanes of a warp that hit the same bin merged
// into one atomic (rows of equal keys would otherwise serialise 32-fold).
// Called by all 32 lanes of the warp.
__device__ __forceinline__ void hist_add_merged(uint32_t* hist, uint32_t bin, bool active) {
    const unsigned act = __ballot_sync(0xffffffffu, active);
    if (!active) return;
    const unsigned peers = __match_any_sync(act, bin);
    if ((threadIdx.x & 31) == (unsigned)(__ffs(peers) - 1)) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
}

// The digit d of nb bins (bin i counts the keys whose digit is i) with
// count(> d) < rem <= count(>= d): res[0] = d, res[1] = rem - count(> d),
// res[2] = count(d).  nb and NT are powers of two, NT <= nb <= 32 NT.
// Every thread calls it.
template <int NT>
__device__ void find_digit_desc(const uint32_t* h, int nb, uint32_t rem, int* wsum,
                                uint32_t* res) {
    const int per = nb / NT;  // 1..32 bins per thread, in descending order
    const int tid = threadIdx.x;
    if (tid == 0) {  // a defined result should the counts not reach rem
        res[0] = 0u;
        res[1] = 1u;
        res[2] = 0u;
    }
    // the per bins of a thread are summed starting at a rotated offset, so
    // that the 32 lanes of a warp read 32 different banks at each step
    const int rot = tid / (32 / per);
    uint32_t part = 0;
    for (int i = 0; i < per; ++i) part += h[nb - 1 - (per * tid + ((i + rot) & (per - 1)))];
    int tot;
    const uint32_t above = (uint32_t)block_scan_excl<NT>((int)part, wsum, &tot);
    if (above < rem && rem <= above + part) {
        uint32_t run = above;
        for (int i = 0; i < per; ++i) {
            const int bin = nb - 1 - (per * tid + i);
            if (run + h[bin] >= rem) {
                res[0] = (uint32_t)bin;
                res[1] = rem - run;
                res[2] = h[bin];
                break;
            }
            run += h[bin];
        }
    }
    __syncthreads();
}

// Radix select, most significant digit first, over the values v = key - base
// of the items src.each() reports valid whose key lies in [base, base + 2^L)
// (the others take no part): digits of up to kDigit bits, at most max_levels.  Finds the
// digit prefix of the rem-th largest value.  On return, value = that prefix
// and low = the number of bits below it (0 once every digit is resolved: then
// value is the rem-th largest value itself); rem = how many of the items with
// that prefix the rem largest take; eq = how many items have it.  With kMerge
// the lanes of a warp that add to the same bin are merged into one atomic
// (for sources where one bin may take nearly everything).
struct RadixResult {
    uint32_t value, rem, eq;
    int low;
};

template <int NT, int kDigit, bool kMerge, typename Src>
__device__ __forceinline__ RadixResult radix_select_desc(uint32_t* hist, int* wsum, uint32_t* res, const Src& src,
                                         uint32_t base, int L, uint32_t rem, int max_levels) {
    const int tid = threadIdx.x;
    uint32_t hi = 0u, eq = 0u;
    int top = L;  // an item is active while (v >> top) == hi
    for (int level = 0; level < max_levels; ++level) {
        const int sh = max(0, top - kDigit);
        const int w = top - sh;  // digit: bits [sh, top)
        const uint32_t dmask = (1u << w) - 1u;
        const int nb = max(1 << w, NT);
        for (int i = tid; i < nb; i += NT) hist[i] = 0u;
        __syncthreads();
        src.each([&](uint32_t key, int, bool valid) {
            const uint32_t v = key - base;
            const bool act = valid && ((uint64_t)v >> top) == (uint64_t)hi;
            const uint32_t d = (v >> sh) & dmask;
            if (kMerge) hist_add_merged(hist, d, act);
            else if (act) atomicAdd(&hist[d], 1u);
        });
        __syncthreads();
        find_digit_desc<NT>(hist, nb, rem, wsum, res);
        hi = (w == 0) ? hi : ((hi << w) | res[0]);
        rem = res[1];
        eq = res[2];
        top = sh;
        if (sh == 0) break;
    }
    return RadixResult{hi, rem, eq, top};
}

// Bit length of x (0 for x = 0).
__device__ __forceinline__ int bit_length(uint32_t x) { return 32 - __clz((int)x); }

// ---- 1. threshold ----------------------------------------------------------
constexpr int kPerWarp = kSampleChunks / (kThrThreads / 32);  // sampled chunks per warp

struct ThrSmem {
    uint32_t hist[kBins0];
    int wsum[kThrThreads / 32 + 1];
    uint32_t res[4];
    uint32_t wmin[kThrThreads / 32], wmax[kThrThreads / 32];
};

// The sampled keys, held in registers: lane l of warp w has position l of
// the sampled chunks w + 8 i.
struct SampleSource {
    uint32_t key[kPerWarp];
    int nsc, stride, vis;
    template <typename F>
    __device__ __forceinline__ void each(F&& f) const {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
        for (int i = 0; i < kPerWarp; ++i) {
            const int j = warp + (kThrThreads / 32) * i;
            f(key[i], 0, j < nsc && 32 * j * stride + lane < vis);
        }
    }
};

__global__ void __launch_bounds__(kThrThreads, 4)
rows_threshold_kernel(RowsArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    ThrSmem& S = *reinterpret_cast<ThrSmem*>(smem_raw);
    const int t = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = request_of(a.bt, t);
    const bool ok = token_ok(a.bt, b, t, nullptr);
    const int vis = ok ? visible_of(a.bt, b, t) : 0;
    grid_dependents_launch();
    grid_dependency_wait();  // the scores come from the previous kernel
    RowInfo* info = a.info + t;
    if (vis <= a.K) {
        int32_t* o = a.out + (int64_t)t * a.K;
        for (int i = tid; i < a.K; i += kThrThreads) o[i] = (i < vis) ? i : -1;
        if (tid == 0) {
            info->vis = 0;
            info->key_lo = 0u;
            info->count = 0u;
        }
        return;
    }
    const float* row = a.scores + (int64_t)t * a.ld;
    const int nch = (vis + 31) / 32;
    const int stride = max(kSampleStride, (nch + kSampleChunks - 1) / kSampleChunks);
    const int nsc = (nch + stride - 1) / stride;  // sampled chunks, <= kSampleChunks
    float x[kPerWarp];
#pragma unroll
    for (int i = 0; i < kPerWarp; ++i) {
        const int j = warp + (kThrThreads / 32) * i;
        const int p = 32 * j * stride + lane;
        x[i] = (j < nsc && p < vis) ? __ldg(row + p) : 0.f;
    }
    SampleSource src;
    src.nsc = nsc;
    src.stride = stride;
    src.vis = vis;
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
    for (int i = 0; i < kPerWarp; ++i) {
        const int j = warp + (kThrThreads / 32) * i;
        src.key[i] = order_key(x[i]);
        if (j < nsc && 32 * j * stride + lane < vis) {
            kmin = min(kmin, src.key[i]);
            kmax = max(kmax, src.key[i]);
        }
    }
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    if (lane == 0) {
        S.wmin[warp] = kmin;
        S.wmax[warp] = kmax;
    }
    const int last = 32 * (nsc - 1) * stride;
    const int ns = 32 * (nsc - 1) + min(32, vis - last);
    // n_s = ceil(1.5 k ns / vis) + 16, at most ns (exact integer arithmetic)
    const uint64_t num = 3ull * (uint64_t)a.K * (uint64_t)ns;
    const uint64_t den = 2ull * (uint64_t)vis;
    const uint64_t want = (num + den - 1) / den + 16ull;
    const uint32_t need = (want < (uint64_t)ns) ? (uint32_t)want : (uint32_t)ns;
    __syncthreads();
    kmin = 0xFFFFFFFFu;
    kmax = 0u;
#pragma unroll
    for (int w = 0; w < kThrThreads / 32; ++w) {
        kmin = min(kmin, S.wmin[w]);
        kmax = max(kmax, S.wmax[w]);
    }
    // one 12-bit digit over the sampled range [kmin, kmax]; a second one when
    // the chosen bin is crowded (the candidates beyond the k-th come from it)
    // (values outside [base, base + 2^L) take no part in a select)
    const RadixResult r = radix_select_desc<kThrThreads, 12, false>(
        S.hist, S.wsum, S.res, src, kmin, bit_length(kmax - kmin), need, 1);
    uint32_t key_lo = kmin + (r.value << r.low);  // the lower edge of the chosen bin
    if (r.low > 0 && r.eq > 8u) {
        const RadixResult r2 = radix_select_desc<kThrThreads, 12, false>(S.hist, S.wsum, S.res, src,
                                                                     key_lo, r.low, r.rem, 1);
        key_lo += r2.value << r2.low;
    }
    if (tid == 0) {
        info->vis = vis;
        info->key_lo = key_lo;
        info->count = 0u;
    }
}

// ---- 2. candidates ---------------------------------------------------------
// A persistent grid: CTA c walks the units [c U / G, (c+1) U / G) of the
// row-major unit space (U = rows x units per row).  One producer thread
// streams each unit (32 KB) into a ring of shared-memory stages with bulk
// copies; eight consumer warps take 1024 positions of each unit apiece and
// reserve slots in the row's candidate list with one atomic per warp.
struct StreamSmem {
    float buf[kStages][kUnit];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int abort_flag;
};

__global__ void __launch_bounds__(kStreamThreads, 2)
rows_candidates_kernel(RowsArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    StreamSmem& S = *reinterpret_cast<StreamSmem*>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &S.abort_flag;
    if (threadIdx.x == 0) {
        for (int st = 0; st < kStages; ++st) {
            mbar_init(&S.full[st], 1);
            mbar_init(&S.empty[st], kConsWarps);
        }
        S.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_dependents_launch();
    grid_dependency_wait();  // the thresholds come from the previous kernel
    const int upr = a.units_per_row;
    const int64_t total = (int64_t)a.bt.total_q * upr;
    const int64_t u_begin = total * blockIdx.x / gridDim.x;
    const int64_t u_end = total * (blockIdx.x + 1) / gridDim.x;
    const int t_begin = (int)(u_begin / upr), ui_begin = (int)(u_begin % upr);
    if (warp == kConsWarps) {
        // ---- producer: one thread ----
        if (lane == 0) {
            int t = t_begin, ui = ui_begin, t_cur = -1, vis = 0, k = 0;
            int st = 0;           // stage of copy k
            uint32_t phase = 0u;  // parity of copy k's use of that stage
            for (int64_t i = u_begin; i < u_end; ++i, ++ui) {
                if (ui == upr) {
                    ui = 0;
                    ++t;
                }
                const int base = ui * kUnit;
                if (t != t_cur) {
                    t_cur = t;
                    vis = __ldcg(&a.info[t].vis);
                }
                if (base >= vis) continue;  // past the row, or the row is written
                if (k >= kStages && !mbar_wait(&S.empty[st], phase ^ 1u, abort_flag)) break;
                // whole 16-byte vectors: the row is padded to a multiple of 4
                const uint32_t bytes = (uint32_t)(((min(kUnit, vis - base) + 3) & ~3) * 4);
                mbar_arrive_expect_tx(&S.full[st], bytes);
                bulk_copy_g2s(S.buf[st], a.scores + (int64_t)t * a.ld + base, bytes, &S.full[st]);
                ++k;
                if (++st == kStages) {
                    st = 0;
                    phase ^= 1u;
                }
            }
            // copies in flight land before the CTA may exit (also after an abort)
            for (int j = max(0, k - kStages); j < k; ++j)
                (void)mbar_drain(&S.full[j % kStages], (j / kStages) & 1);
        }
    } else {
        // ---- consumers: positions base + 512 warp + 128 u + 4 lane + e ----
        // A unit's slot reservation (a global atomic) is used one unit later,
        // so its latency overlaps the next unit's test; its stage is handed
        // back once its candidates are written.
        int t = t_begin, ui = ui_begin, t_cur = -1, vis = 0;
        int st = 0;
        uint32_t phase = 0u, key_lo = 0u, thr = 0u;
        bool nonneg = true;
        uint32_t* ck = nullptr;
        int32_t* cp = nullptr;
        // the previous unit
        bool have_prev = false, prev_cands = false;
        int prev_st = 0, prev_excl = 0, prev_p0 = 0;
        uint32_t prev_mask = 0u, prev_slot = 0u;
        uint32_t* prev_ck = nullptr;
        int32_t* prev_cp = nullptr;
        auto finish_prev = [&]() {
            if (prev_cands) {
                uint32_t slot = __shfl_sync(0xffffffffu, prev_slot, 31) + (uint32_t)prev_excl;
                const float* xs = &S.buf[prev_st][128 * kLaneVec * warp + 4 * lane];
                uint32_t m = prev_mask;
                while (m) {  // candidates are rare
                    const int j = __ffs(m) - 1;
                    m &= m - 1;
                    const int off = 128 * (j >> 2) + (j & 3);
                    if (slot < (uint32_t)kRowsCandMax) {
                        prev_ck[slot] = order_key(xs[off]);
                        prev_cp[slot] = prev_p0 + off;
                    }
                    ++slot;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[prev_st]);
        };
        bool ok = true;
        for (int64_t i = u_begin; i < u_end; ++i, ++ui) {
            if (ui == upr) {
                ui = 0;
                ++t;
            }
            const int base = ui * kUnit;
            if (t != t_cur) {
                t_cur = t;
                vis = __ldcg(&a.info[t].vis);
                key_lo = __ldcg(&a.info[t].key_lo);
                ck = a.cand_key + (int64_t)t * kRowsCandMax;
                cp = a.cand_pos + (int64_t)t * kRowsCandMax;
                // key >= key_lo, tested on the raw bits.  Above +0's key: as
                // signed integers (every negative float, -0 included, is a
                // negative integer and below the bound).  Otherwise on the
                // sign-flipped bits, where -0 sits one under +0: the bound
                // +0's key drops by one to take -0 in as well.
                nonneg = key_lo > 0x80000000u;
                thr = nonneg ? (key_lo & 0x7FFFFFFFu)
                             : ((key_lo == 0x80000000u) ? 0x7FFFFFFFu : key_lo);
            }
            if (base >= vis) continue;
            if (!mbar_wait(&S.full[st], phase, abort_flag)) {
                ok = false;
                break;
            }
            const float* xs = &S.buf[st][128 * kLaneVec * warp + 4 * lane];  // + 128 u + e
            const int p0 = base + 128 * kLaneVec * warp + 4 * lane;
            uint32_t mask = 0u;  // bit 4u+e: position p0 + 128u + e is a candidate
            if (nonneg) {
#pragma unroll
                for (int u = 0; u < kLaneVec; ++u) {
                    const int4 x = *reinterpret_cast<const int4*>(xs + 128 * u);
                    mask |= (x.x >= (int32_t)thr ? 1u : 0u) << (4 * u + 0);
                    mask |= (x.y >= (int32_t)thr ? 1u : 0u) << (4 * u + 1);
                    mask |= (x.z >= (int32_t)thr ? 1u : 0u) << (4 * u + 2);
                    mask |= (x.w >= (int32_t)thr ? 1u : 0u) << (4 * u + 3);
                }
            } else {
#pragma unroll
                for (int u = 0; u < kLaneVec; ++u) {
                    const uint4 x = *reinterpret_cast<const uint4*>(xs + 128 * u);
                    const uint32_t xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t raw = xv[e] ^ ((uint32_t)((int32_t)xv[e] >> 31) | 0x80000000u);
                        mask |= (raw >= thr ? 1u : 0u) << (4 * u + e);
                    }
                }
            }
            if (base + kUnit > vis) {  // the row's last unit: drop positions >= vis
#pragma unroll
                for (int j = 0; j < 4 * kLaneVec; ++j)
                    if (p0 + 128 * (j >> 2) + (j & 3) >= vis) mask &= ~(1u << j);
            }
            const int n = __popc(mask);
            int incl = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            const int wsum = __shfl_sync(0xffffffffu, incl, 31);
            uint32_t slot_raw = 0u;
            if (wsum != 0 && lane == 31) slot_raw = atomicAdd(&a.info[t].count, (uint32_t)wsum);
            if (have_prev) finish_prev();
            have_prev = true;
            prev_cands = wsum != 0;
            prev_st = st;
            prev_mask = mask;
            prev_slot = slot_raw;
            prev_excl = incl - n;
            prev_p0 = p0;
            prev_ck = ck;
            prev_cp = cp;
            if (++st == kStages) {
                st = 0;
                phase ^= 1u;
            }
        }
        if (ok && have_prev) finish_prev();
    }
    __syncthreads();
    if (*abort_flag) {
        // a wait ran out: the rows this CTA touched get an impossible count,
        // so the select reads them whole (the result stays exact)
        const int t0 = t_begin;
        const int t1 = (int)((u_end - 1) / upr);
        for (int t = t0 + (int)threadIdx.x; t <= t1; t += kStreamThreads)
            atomicOr(&a.info[t].count, kCountPoison);
    }
}

// ---- 3. exact select -------------------------------------------------------
// Words of the selection bitmap a select thread owns: an odd number, so that
// the threads of a warp, reading word i of their runs, hit 32 different banks.
constexpr int kSelWordsMax = (kRowsMaxSeq / 32 / kSelThreads) | 1;

constexpr int kSmallBin = 128;  // a bin this small is finished by pairwise ranks

struct SelSmem {
    union {
        uint32_t hist[kBins0];
        struct {
            uint32_t key[kSmallBin];
            int32_t pos[kSmallBin];
        } list;  // the items of the threshold bin
        struct {
            uint32_t bits[kSelWordsMax * kSelThreads];  // the selection
            uint32_t pre[kSelWordsMax * kSelThreads];   // selected positions before word w
        } b;
    } u;
    int wsum[kSelThreads / 32 + 1];
    uint32_t res[4];
    uint32_t n_list;
};

// The candidates, held in registers: thread i has candidates i + 256 j.
// each(f) calls f(key, position, valid) for all of them (every thread the
// same number of times).
struct CandSource {
    uint32_t key[kSelPer];
    int32_t pos[kSelPer];
    int n;
    template <typename F>
    __device__ __forceinline__ void each(F&& f) const {
#pragma unroll
        for (int j = 0; j < kSelPer; ++j) f(key[j], pos[j], j * kSelThreads + (int)threadIdx.x < n);
    }
};

// The whole row, read from global memory (rows of <= 2^18 positions; the row
// is padded to a multiple of 4 floats, so each 16-byte vector is in bounds).
// Same each(f) contract.
struct RowSource {
    const float* row;
    int vis;
    template <typename F>
    __device__ __forceinline__ void each(F&& f) const {
        const int nvec = (vis + 3) / 4;
        for (int v0 = 0; v0 < nvec; v0 += kRowVec * kSelThreads) {
            float4 x[kRowVec];
#pragma unroll
            for (int u = 0; u < kRowVec; ++u) {
                const int v = v0 + u * kSelThreads + threadIdx.x;
                x[u] = (v < nvec) ? __ldg(reinterpret_cast<const float4*>(row) + v)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kRowVec; ++u) {
                const int p = 4 * (v0 + u * kSelThreads + threadIdx.x);
                f(order_key(x[u].x), p + 0, p + 0 < vis);
                f(order_key(x[u].y), p + 1, p + 1 < vis);
                f(order_key(x[u].z), p + 2, p + 2 < vis);
                f(order_key(x[u].w), p + 3, p + 3 < vis);
            }
        }
    }
};

// Positions of the keys equal to tau, mirrored so that the lowest position
// is the largest value (positions < 2^18).
template <typename Src>
struct EqPosSource {
    const Src& src;
    uint32_t tau;
    template <typename F>
    __device__ __forceinline__ void each(F&& f) const {
        src.each([&](uint32_t key, int pos, bool valid) {
            f((uint32_t)(kRowsMaxSeq - 1 - pos), pos, valid && key == tau);
        });
    }
};

// Select over a source whose valid keys are all >= base and < base + 2^L, and
// write the row's ascending top-K positions.
template <bool kMerge, typename Src>
__device__ __forceinline__ void select_and_write(SelSmem& S, const Src& src, uint32_t base, int L,
                                                 int vis, int K, int32_t* o) {
    const int tid = threadIdx.x, lane = tid & 31;
    // The selection is every key above tau (the K-th largest key) and, of
    // the keys equal to tau, those at positions <= pthr.  Radix digits narrow
    // tau down to a bin [bin_lo, bin_lo + 2^low) holding eq items, of which
    // the rem largest (by key, then lower position) are taken.
    uint32_t bin_lo = base, rem = (uint32_t)K, eq = 0u;
    int low = L;
    do {
        const RadixResult r = radix_select_desc<kSelThreads, 8, kMerge>(S.u.hist, S.wsum, S.res,
                                                                        src, bin_lo, low, rem, 1);
        bin_lo += r.value << r.low;
        rem = r.rem;
        eq = r.eq;
        low = r.low;
    } while (low > 0 && eq > (uint32_t)kSmallBin);
    uint32_t tau;
    int pthr = INT_MAX;
    if (eq <= (uint32_t)kSmallBin) {
        // gather the bin's items; the one ranked rem-th (key descending, then
        // position ascending) gives tau and pthr
        if (tid == 0) S.n_list = 0u;
        __syncthreads();
        const uint32_t span = (low >= 32) ? 0xFFFFFFFFu : ((1u << low) - 1u);
        src.each([&](uint32_t key, int p, bool valid) {
            const bool in = valid && key - bin_lo <= span;
            const unsigned m = __ballot_sync(0xffffffffu, in);
            if (m == 0u) return;
            uint32_t b0 = 0u;
            if (lane == __ffs(m) - 1) b0 = atomicAdd(&S.n_list, (uint32_t)__popc(m));
            b0 = __shfl_sync(0xffffffffu, b0, __ffs(m) - 1);
            if (in) {
                const uint32_t slot = b0 + (uint32_t)__popc(m & ((1u << lane) - 1u));
                if (slot < (uint32_t)kSmallBin) {
                    S.u.list.key[slot] = key;
                    S.u.list.pos[slot] = p;
                }
            }
        });
        __syncthreads();
        const int m = (int)min(S.n_list, (uint32_t)kSmallBin);
        for (int i = tid; i < m; i += kSelThreads) {
            const uint32_t ki = S.u.list.key[i];
            const int pi = S.u.list.pos[i];
            uint32_t before = 0u;
#pragma unroll 8
            for (int j = 0; j < m; ++j) {
                const uint32_t kj = S.u.list.key[j];
                const int pj = S.u.list.pos[j];
                before += (kj > ki) | ((kj == ki) & (pj < pi));
            }
            if (before == rem - 1u) {
                S.res[0] = ki;
                S.res[1] = (uint32_t)pi;
            }
        }
        __syncthreads();
        tau = S.res[0];
        pthr = (int)S.res[1];
        __syncthreads();  // the list is overwritten by the bitmap below
    } else {
        // every item of the bin carries the key bin_lo: the rem lowest
        // positions among them
        tau = bin_lo;
        const EqPosSource<Src> eqs{src, tau};
        const RadixResult pr = radix_select_desc<kSelThreads, 8, kMerge>(
            S.u.hist, S.wsum, S.res, eqs, 0u, 18, rem, 3);
        pthr = kRowsMaxSeq - 1 - (int)pr.value;
    }
    // bitmap of the selection; thread i owns words [wpt i, wpt i + wpt)
    const int nwords = (vis + 31) / 32;
    const int wpt = ((nwords + kSelThreads - 1) / kSelThreads) | 1;
    for (int w = tid; w < wpt * kSelThreads; w += kSelThreads) S.u.b.bits[w] = 0u;
    __syncthreads();
    auto selected = [&](uint32_t key, int p, bool valid) {
        return valid && key >= tau && (key > tau || p <= pthr);
    };
    src.each([&](uint32_t key, int p, bool valid) {
        if (selected(key, p, valid)) atomicOr(&S.u.b.bits[p >> 5], 1u << (p & 31));
    });
    __syncthreads();
    // the output index of a selected position is the number selected before
    // it: per-word prefix counts, then each selected item writes itself
    int mine = 0;
    for (int i = 0; i < wpt; ++i) {
        S.u.b.pre[wpt * tid + i] = (uint32_t)mine;
        mine += __popc(S.u.b.bits[wpt * tid + i]);
    }
    int tot;
    const uint32_t off = (uint32_t)block_scan_excl<kSelThreads>(mine, S.wsum, &tot);
    for (int i = 0; i < wpt; ++i) S.u.b.pre[wpt * tid + i] += off;
    __syncthreads();
    src.each([&](uint32_t key, int p, bool valid) {
        if (selected(key, p, valid)) {
            const uint32_t below = S.u.b.bits[p >> 5] & ((1u << (p & 31)) - 1u);
            const uint32_t q = S.u.b.pre[p >> 5] + (uint32_t)__popc(below);
            if (q < (uint32_t)K) o[q] = p;
        }
    });
}

__global__ void __launch_bounds__(kSelThreads, 3)
rows_select_kernel(RowsArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SelSmem& S = *reinterpret_cast<SelSmem*>(smem_raw);
    const int t = blockIdx.x;
    grid_dependents_launch();
    grid_dependency_wait();  // the candidates come from the previous kernel
    const int vis = __ldcg(&a.info[t].vis);
    if (vis == 0) return;
    const uint32_t n = __ldcg(&a.info[t].count);
    int32_t* o = a.out + (int64_t)t * a.K;
    if (n >= (uint32_t)a.K && n <= (uint32_t)kRowsCandMax) {
        const uint32_t* ck = a.cand_key + (int64_t)t * kRowsCandMax;
        const int32_t* cp = a.cand_pos + (int64_t)t * kRowsCandMax;
        const uint32_t key_lo = __ldcg(&a.info[t].key_lo);
        CandSource src;
        src.n = (int)n;
        uint32_t kmax = key_lo;
#pragma unroll
        for (int j = 0; j < kSelPer; ++j) {
            const int c = j * kSelThreads + (int)threadIdx.x;
            src.key[j] = (c < (int)n) ? __ldcg(ck + c) : key_lo;
            src.pos[j] = (c < (int)n) ? __ldcg(cp + c) : 0;
            kmax = max(kmax, src.key[j]);
        }
        // digits over [key_lo, max key]: every candidate is >= key_lo
        kmax = __reduce_max_sync(0xffffffffu, kmax);
        if ((threadIdx.x & 31) == 0) S.wsum[threadIdx.x >> 5] = (int)kmax;
        __syncthreads();
        kmax = key_lo;
        for (int w = 0; w < kSelThreads / 32; ++w) kmax = max(kmax, (uint32_t)S.wsum[w]);
        __syncthreads();
        select_and_write<false>(S, src, key_lo, bit_length(kmax - key_lo), vis, a.K, o);
    } else {
        const RowSource src{a.scores + (int64_t)t * a.ld, vis};
        select_and_write<true>(S, src, 0u, 32, vis, a.K, o);
    }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

// This path takes batches whose rows are too long for one CTA's shared memory
// but short enough for the selection bitmap, unless the rows are so few that
// the split path (rows over the whole GPU by radix levels) serves them.
bool topk_rows_eligible(int total_q, int max_seq, bool split) {
    return !split && total_q > 0 && max_seq >= kRowsMinSeq && max_seq <= kRowsMaxSeq;
}

size_t topk_rows_workspace_bytes(int total_q) {
    const size_t q = (size_t)total_q;
    return align256(q * sizeof(RowInfo)) + 2 * align256(q * kRowsCandMax * sizeof(uint32_t));
}

cudaError_t launch_topk_rows(const BatchArgs& bt, const float* scores, int64_t ld, int K,
                             int32_t* out, void* ws, bool pdl, cudaStream_t stream) {
    RowsArgs a;
    a.bt = bt;
    a.scores = scores;
    a.ld = ld;
    a.K = K;
    a.out = out;
    uint8_t* p = static_cast<uint8_t*>(ws);
    const size_t q = (size_t)bt.total_q;
    a.info = reinterpret_cast<RowInfo*>(p);
    p += align256(q * sizeof(RowInfo));
    a.cand_key = reinterpret_cast<uint32_t*>(p);
    p += align256(q * kRowsCandMax * sizeof(uint32_t));
    a.cand_pos = reinterpret_cast<int32_t*>(p);
    a.units_per_row = (bt.max_seq + kUnit - 1) / kUnit;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)bt.total_q * a.units_per_row;
    const int grid2 = (int)(units < 2 * (int64_t)sms ? units : 2 * (int64_t)sms);
    e = cudaFuncSetAttribute(rows_threshold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(ThrSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rows_candidates_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(StreamSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rows_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(SelSmem));
    if (e == cudaSuccess)
        e = launch_kernel(rows_threshold_kernel, dim3(bt.total_q), dim3(kThrThreads),
                          sizeof(ThrSmem), stream, pdl, 1, a);
    if (e == cudaSuccess)
        e = launch_kernel(rows_candidates_kernel, dim3((unsigned)grid2), dim3(kStreamThreads),
                          sizeof(StreamSmem), stream, true, 1, a);
    if (e == cudaSuccess)
        e = launch_kernel(rows_select_kernel, dim3(bt.total_q), dim3(kSelThreads),
                          sizeof(SelSmem), stream, true, 1, a);
    return e;
}

}  // namespace dsa
