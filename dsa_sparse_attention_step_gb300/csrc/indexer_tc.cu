// indexer_tc.cu -- DSA indexer scores for FP8 keys on tcgen05 tensor cores.
//
//   score[t,s] = kscale[s] * sum_h (w[t,h] * q_scale[t,h]) * ReLU(q8[t,h,:] . k8[s,:])
// i.e. sum_h w[t,h] ReLU(qhat[t,h,:] . khat[s,:]) with the positive key and
// query scales pulled through the ReLU.
// "vLLM's Kimi K3.1 Pro day-0 support", section "What changed": 32 indexer
// heads x 128 dims, one FP8 key of 132 bytes with its scale per token, every
// earlier token scored; section "Fused low-latency decode for DSA layers": a
// key-balanced scorer.
//
// The work is a list of units (request b, query group g of up to G tokens,
// tile of 128 keys = two 64-token pages); every group of a request covers all
// of the request's tiles (positions past a token's causal limit get -inf).
// A persistent grid splits the unit list into equal contiguous ranges, so the
// keys, not the queries, are balanced across SMs.  Per unit:
//   D[128 keys x N] = K8[128 x 128] . Q8[N x 128]^T,  N = 32 heads x G tokens,
// tcgen05.mma kind::f8f6f4 (E4M3 x E4M3, fp32 accumulator in TMEM).  Key pages
// arrive by TMA (128-byte swizzle) into a ring of six stages (eight for query
// groups of one or two tokens), their 64 scale words by bulk copy beside them,
// and the query group by TMA into a double buffer.  The epilogue warps read the
// accumulator (thread = key), apply ReLU, the weighted head sum, the key scale
// and the causal mask, and store fp32 scores.
//
// Roles: producer warps (each looks up pages and one lane issues the copies),
// then MMA warps (the first allocates TMEM; lane 0 issues MMAs), then for
// MXFP4 keys four converter warps, then epilogue warps in sets of four (one
// warp per TMEM lane quarter).  With FP8 keys two producer and two MMA warps
// take alternate units (one thread spends about a thousand cycles of
// instruction latency on a unit's copies, or on its waits, MMAs and commits,
// more than the unit's share of the memory bandwidth allows), and the
// accumulators depend on the query-group size (IdxCfg below): six for groups
// of one or two tokens, a ring of three for groups of 3-5, two accumulators of
// two token halves for groups of 6-8.  With MXFP4 keys one MMA thread feeds
// four accumulators per token and two epilogue sets each take every second
// token.  A key of an absent page carries all-ones scale bits (copied in place
// of the page's scales), so the epilogue needs no block-table read.  Every
// wait is bounded.
#include <climits>
#include <cstring>
#include <mutex>
#include <type_traits>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm100.cuh"

namespace dsa {

using namespace sm100;

namespace {

constexpr int kTile = 128;                     // keys per unit
constexpr int kMaxStages = 8;                  // key-tile ring: at most 8 stages
constexpr int kStageBytes = kTile * kIdxDim;   // 16384: E4M3 A operand of one unit
constexpr int kQBufBytes = 8 * kIdxHeads * kIdxDim;  // 32768: up to 8 tokens x 32 heads
constexpr int kMaxReq = 4096;
constexpr int kStgSlots = 4;                   // MXFP4: packed-key staging ring
constexpr int kStgBytes = 2 * kPage * kIdxDim / 2;   // 8192: two pages of packed E2M1
constexpr int kMetaBytes = 2 * kPage * 4;        // 512: the 64 scale words of two pages

// Per-format layout of the kernel.  FP8 keys go straight from TMA to the MMA;
// MXFP4 keys are staged packed and expanded to E4M3 by four converter warps,
// and each 32-element block gets its own accumulator (its E8M0 scale is
// applied in the epilogue), which limits a query group to 2 tokens.
// FP8 keys: two MMA warps take alternate units (one thread's waits, MMAs and
// commits of a unit take longer than the tensor pipe needs for them).  kDual
// (query groups of one or two tokens, where the epilogue has time to spare):
// six accumulators, three per MMA warp, and two epilogue sets.  Groups of 3-5
// tokens: a ring of three accumulators shared by the two MMA warps.  kWide
// (FP8 keys, query groups of 6-8 tokens): two accumulators of two token halves
// each, MMA warp m filling accumulator m (the units of parity m), and four
// epilogue sets, set s draining half s % 2 of accumulator s / 2.
template <int kFmt, bool kDual, bool kWide = false>
struct IdxCfg {
    static constexpr bool kMx = (kFmt == DSA_KEYS_MXFP4);
    static_assert(!(kMx && kDual), "MXFP4 keys use one producer and one MMA warp");
    static_assert(!(kWide && (kMx || kDual)), "four epilogue sets only for FP8 groups of 6-8 tokens");
    // FP8 keys: two producer warps taking alternate units (one thread's copy
    // issue for a unit takes longer than the unit's keys take to arrive);
    // MXFP4 keys: one (the converters pace the stream)
    static constexpr int kProdWarps = kMx ? 1 : 2;
    static constexpr int kMmaWarp = kProdWarps;    // allocates TMEM
    static constexpr int kMmaWarps = kMx ? 1 : 2;  // MMA-issuing threads (alternate units)
    static constexpr int kConvWarp0 = kMmaWarp + kMmaWarps;
    static constexpr int kConvWarps = kMx ? 4 : 0;
    static constexpr int kEpiWarp0 = kConvWarp0 + kConvWarps;
    // epilogue warps in sets of four (one warp per TMEM lane quarter).  FP8:
    // a set takes whole units, round robin (two sets with two MMA threads,
    // else one set per TMEM accumulator, so every accumulator is drained while
    // the MMA fills another), or token halves of units; MXFP4: two sets, each
    // every second token
    static constexpr int kEpiSets = (kMx || kDual) ? 2 : (kWide ? 4 : 3);
    static constexpr int kEpiWarps = 4 * kEpiSets;
    static constexpr int kEpiThreads = kEpiWarps * 32;
    static constexpr int kTokSplit = 2;                        // MXFP4 token stride
    static constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;  // 384 (kDual), 512, 640 (kWide) or 448
    static constexpr int kMaxG = kMx ? 2 : 8;                  // tokens per group
    // enough key bytes in flight per SM to cover the memory latency at full
    // load: six stages (96 KB) on the paths of groups of 3-8 tokens (six ran
    // 1-2 % faster than eight there, four slower), eight for groups of 1-2
    static constexpr int kStages = (kMx || !kDual) ? 6 : 8;
    // scale words of a unit: a slot is free again S + 3 units later with one
    // MMA thread (MXFP4); S + 6 with kDual, whose accumulators repeat every
    // sixth unit; S + 4 with kWide (the MMA of unit i - S waited for the
    // epilogue of unit i - S - 2 of the same parity, and each set drains its
    // half's units in order, so an even distance of at least S + 2 is
    // needed); S + 7 with the ring of three (the argument is at the MMA loop)
    static constexpr int kMetaSlots = kStages + (kMx ? 3 : (kDual ? 6 : (kWide ? 4 : 7)));
    static constexpr int kOffStage = 0;
    static constexpr int kOffQ = kOffStage + kStages * kStageBytes;
    static constexpr int kOffW = kOffQ + 2 * kQBufBytes;
    static constexpr int kOffReq = kOffW + kEpiSets * 8 * kIdxHeads * 4;  // w x q_scale: [sets][8][32]
    static constexpr int kOffStg = (kOffReq + (kMaxReq + 1) * 4 + 1023) / 1024 * 1024;
    static constexpr int kOffMeta = kOffStg + (kMx ? kStgSlots * kStgBytes : 0);
    static constexpr int kOffBar = kOffMeta + kMetaSlots * kMetaBytes;
    static constexpr int kSmemAlloc = kOffBar + 512 + 1024;
    static_assert(kSmemAlloc <= 227 * 1024, "shared memory budget");
    static_assert(kStages <= kMaxStages, "the barrier arrays cover every key stage");
};

// Scale words of a page that is absent (past the sequence) or out of range:
// all bits set, which is NaN as an fp32 key scale and NaN in every E8M0 byte.
// The producers copy them into the unit's scale slot in place of the page's
// own, through the same barrier as the keys, and the epilogue masks every key
// whose scale word reads so (valid key scales are positive).
__device__ __align__(16) uint32_t g_absent_scales[kPage] = {
    0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu,
    0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu,
    0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu,
    0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu,
    0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu,
    0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu,
    0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu,
    0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu,
    0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu,
    0xFFFFFFFFu};

struct Bars {
    uint64_t full[kMaxStages];   // TMA / converters -> MMA: key tile ready
    uint64_t empty[kMaxStages];  // MMA -> TMA / converters: stage free (commit)
    uint64_t tfull[6];        // MMA -> epilogue: accumulator ready (commit)
    uint64_t tempty[6];       // epilogue -> MMA: accumulator drained (epilogue arrivals)
    uint64_t qfull[2];        // TMA -> MMA: query group landed
    uint64_t qempty[2];       // MMA -> TMA: query buffer free (commit)
    uint64_t sfull[kStgSlots];   // MXFP4: packed keys landed (bulk copy)
    uint64_t sempty[kStgSlots];  // MXFP4: staging slot converted (128 arrivals)
    uint64_t done;            // MMA issuer: all its MMAs have completed
    uint32_t tmem_base;
    int abort_flag;
    int total_units;
};

static_assert(sizeof(Bars) <= 512, "barrier block of the shared-memory layout");

struct IdxParams {
    BatchArgs bt;
    const float* qscale;
    const float* w;
    const uint8_t* pages;
    float* scores;
    int64_t ld;
    int G;                    // tokens per group (1..8)
    int N;                    // 32 * G
    int32_t* status;
};

// Per-request unit count: groups x tiles.
__device__ __forceinline__ int request_units(const BatchArgs& bt, int b, int G) {
    if (!request_ok(bt, b, nullptr)) return 0;
    const int nb = __ldg(bt.q_offsets + b + 1) - __ldg(bt.q_offsets + b);
    const int seq = __ldg(bt.seq_lens + b);
    return ((nb + G - 1) / G) * ((seq + kTile - 1) / kTile);
}

// Cursor over the unit list of this CTA.
struct Cursor {
    int b, g, tile;     // current unit
    int ntile;          // tiles of request b
    int ngroup;         // groups of request b
    int q0, nb, seq;    // request metadata
};

__device__ __forceinline__ void cursor_load_request(Cursor& c, const BatchArgs& bt, int G) {
    c.q0 = __ldg(bt.q_offsets + c.b);
    c.nb = __ldg(bt.q_offsets + c.b + 1) - c.q0;
    c.seq = __ldg(bt.seq_lens + c.b);
    const bool ok = request_ok(bt, c.b, nullptr);
    c.ngroup = ok ? (c.nb + G - 1) / G : 0;
    c.ntile = ok ? (c.seq + kTile - 1) / kTile : 0;
}

// Position the cursor on global unit u (req_units = exclusive prefix, B+1).
__device__ __forceinline__ void cursor_seek(Cursor& c, const BatchArgs& bt, const int* req_units,
                                            int G, int u) {
    int lo = 0, hi = bt.num_requests - 1;
    while (lo < hi) {  // last b with req_units[b] <= u
        const int mid = (lo + hi + 1) >> 1;
        if (req_units[mid] <= u) lo = mid;
        else hi = mid - 1;
    }
    c.b = lo;
    cursor_load_request(c, bt, G);
    const int r = u - req_units[lo];
    c.g = (c.ntile > 0) ? r / c.ntile : 0;
    c.tile = (c.ntile > 0) ? r % c.ntile : 0;
}

__device__ __forceinline__ void cursor_next(Cursor& c, const BatchArgs& bt, int G) {
    if (++c.tile < c.ntile) return;
    c.tile = 0;
    if (++c.g < c.ngroup) return;
    c.g = 0;
    do {
        ++c.b;
        if (c.b >= bt.num_requests) return;
        cursor_load_request(c, bt, G);
    } while (c.ngroup == 0 || c.ntile == 0);
}

// Packed pairs of fp32 (low word = first element) and their fused multiply-add
// (one instruction for two lanes of the FMA pipe on this GPU).
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
// Four consecutive fp32 of shared memory in one 128-bit load (plain float4
// reads here executed twice as many shared-load instructions).
__device__ __forceinline__ float4 lds_f32x4(const float* p) {
    float4 r;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "r"(smem_u32(p)));
    return r;
}
// (max(a, 0), max(b, 0)) as a pair, formed in the pair's own registers
__device__ __forceinline__ uint64_t relu_pair(uint32_t a, uint32_t b) {
    uint64_t d;
    asm("{\n\t.reg .f32 x, y;\n\tmax.f32 x, %1, 0f00000000;\n\tmax.f32 y, %2, 0f00000000;\n\t"
        "mov.b64 %0, {x, y};\n\t}"
        : "=l"(d)
        : "f"(__uint_as_float(a)), "f"(__uint_as_float(b)));
    return d;
}
__device__ __forceinline__ uint64_t pair_f32(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ float lo_f32x2(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_f32x2(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// E2M1 magnitude code -> E4M3 code of the same value (0, 0.5, 1, 1.5, 2, 3,
// 4, 6), as byte lanes of two words for PRMT lookups.
constexpr uint32_t kE2m1ToE4m3Lo = 0x3C383000u;  // codes 0..3
constexpr uint32_t kE2m1ToE4m3Hi = 0x4C484440u;  // codes 4..7

// Eight packed E2M1 elements (element 2i in the low nibble of byte i) -> eight
// E4M3 bytes (exact: every E2M1 value is an E4M3 value).
__device__ __forceinline__ uint2 e2m1x8_to_e4m3x8(uint32_t w) {
    uint2 r;
    const uint32_t mag = w & 0x77777777u;      // 3-bit magnitude codes
    const uint32_t sgn = w & 0x88888888u;      // sign bits (bit 3 of each nibble)
    // PRMT selector nibbles pick a byte among the 8 table bytes
    const uint32_t sel_lo = (mag & 0x7u) | ((mag >> 4) & 0x7u) << 4 | ((mag >> 8) & 0x7u) << 8 |
                            ((mag >> 12) & 0x7u) << 12;
    const uint32_t sel_hi = ((mag >> 16) & 0x7u) | ((mag >> 20) & 0x7u) << 4 |
                            ((mag >> 24) & 0x7u) << 8 | ((mag >> 28) & 0x7u) << 12;
    r.x = __byte_perm(kE2m1ToE4m3Lo, kE2m1ToE4m3Hi, sel_lo);
    r.y = __byte_perm(kE2m1ToE4m3Lo, kE2m1ToE4m3Hi, sel_hi);
    // sign of nibble k -> bit 7 of output byte k
    const uint32_t s_lo = sgn & 0xFFFFu, s_hi = sgn >> 16;
    r.x |= ((s_lo >> 3) & 1u) << 7 | ((s_lo >> 7) & 1u) << 15 | ((s_lo >> 11) & 1u) << 23 |
           ((s_lo >> 15) & 1u) << 31;
    r.y |= ((s_hi >> 3) & 1u) << 7 | ((s_hi >> 7) & 1u) << 15 | ((s_hi >> 11) & 1u) << 23 |
           ((s_hi >> 15) & 1u) << 31;
    return r;
}

template <int kFmt, bool kDual, bool kWide>
__global__ void __launch_bounds__(IdxCfg<kFmt, kDual, kWide>::kThreads, 1)
indexer_tc_kernel(const __grid_constant__ CUtensorMap tm_keys,
                  const __grid_constant__ CUtensorMap tm_q, const IdxParams p) {
    using C = IdxCfg<kFmt, kDual, kWide>;
    constexpr bool kMx = C::kMx;
    constexpr int kThreads = C::kThreads;
    grid_dependents_launch();  // the top-k may start its preamble
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    uint8_t* sStage = sm + C::kOffStage;
    uint8_t* sQ = sm + C::kOffQ;
    float* sW = reinterpret_cast<float*>(sm + C::kOffW);     // [sets][8][32]
    int* sReq = reinterpret_cast<int*>(sm + C::kOffReq);      // [B+1]
    uint8_t* sStg = sm + C::kOffStg;                          // MXFP4 staging ring
    uint8_t* sMeta = sm + C::kOffMeta;                        // scale words per unit
    Bars* bars = reinterpret_cast<Bars*>(sm + C::kOffBar);
    __shared__ int s_warp_sum[kThreads / 32];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const BatchArgs& bt = p.bt;
    const int G = p.G, N = p.N;
    // TMEM accumulators: columns per unit, and three buffers when they fit in
    // the 512 columns (the MMA then runs two units ahead of the epilogue).
    // kDual (N <= 64): each MMA thread owns three of six buffers and cycles
    // through them in its own unit order: unit i uses buffer
    // 3 (i % 2) + (i / 2) % 3 for the (i / 6)-th time.  Were a buffer shared
    // by the two threads with one drain barrier, the thread at unit i could
    // reach its wait for the epilogue of unit i - 3 while that of unit i - 6
    // (issued by the same thread, same buffer) is still running, and the
    // parity wait would take the older, unfinished phase for the awaited
    // one; the ring of three below shares its buffers and therefore splits
    // the drain barrier by unit parity.
    const int acc_cols = kMx ? 4 * N : N;
    const int nacc = kDual ? 6 : ((3 * acc_cols <= 512) ? 3 : 2);
    // FP8 groups of 6-8 tokens (kWide; the host routes them here, and only
    // two accumulators fit): each token half is an MMA of its own on its own
    // barrier pair, drained by its own epilogue set, so that an accumulator
    // half waits only for its own drain (with three accumulators the extra
    // MMAs and waits cost the MMA threads more than they save)
    const bool tsplit = kWide;
    // FP8 groups of 3-5 tokens (the host routes 6-8 to kWide): the two MMA
    // threads share a ring of three accumulators, unit i on accumulator i % 3
    const bool ring3 = !kMx && !kDual && !kWide && nacc == 3;
    // with token halves, tokens [0, H) and [H, G) of a group are two MMAs on
    // their own column ranges of the accumulator, with their own barriers
    const int H = (G + 1) >> 1;
    volatile int* abort_flag = &bars->abort_flag;

    if (tid == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&bars->full[i], kMx ? 128 : 1);
            mbar_init(&bars->empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->qfull[i], 1);
            mbar_init(&bars->qempty[i], C::kMmaWarps);  // one commit per MMA thread
        }
        for (int i = 0; i < 6; ++i) {
            mbar_init(&bars->tfull[i], 1);
            // FP8: the set of four warps that takes the unit arrives (the two
            // sets of its token halves when they are split)
            mbar_init(&bars->tempty[i], kMx ? C::kEpiThreads : 128);
        }
        for (int i = 0; i < kStgSlots; ++i) {
            mbar_init(&bars->sfull[i], 1);
            mbar_init(&bars->sempty[i], 128);
        }
        mbar_init(&bars->done, C::kMmaWarps);
        bars->abort_flag = 0;
        fence_mbar_init();
        if (!kMx) tma_prefetch_desc(&tm_keys);
        tma_prefetch_desc(&tm_q);
    }
    if (warp == C::kMmaWarp) {
        tmem_alloc(&bars->tmem_base, 512);
        tmem_relinquish();
    }
    // Everything below reads the caller's inputs: wait for the previous grid
    // of the stream (the launch may overlap its tail; the setup above does
    // not touch global memory).
    grid_dependency_wait();
    // ---- unit table: exclusive prefix of per-request unit counts ----
    int carry = 0;
    for (int b0 = 0; b0 < bt.num_requests; b0 += kThreads) {
        const int b = b0 + tid;
        const int u = (b < bt.num_requests) ? request_units(bt, b, G) : 0;
        int incl = u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) s_warp_sum[warp] = incl;
        __syncthreads();
        int before = 0, chunk = 0;
        for (int w2 = 0; w2 < kThreads / 32; ++w2) {
            const int s2 = s_warp_sum[w2];
            if (w2 < warp) before += s2;
            chunk += s2;
        }
        if (b < bt.num_requests) sReq[b] = carry + before + incl - u;
        carry += chunk;
        __syncthreads();
    }
    if (tid == 0) {
        sReq[bt.num_requests] = carry;
        bars->total_units = carry;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int total = bars->total_units;
    const uint32_t tmem = bars->tmem_base;
    const int u_begin = (int)(((int64_t)total * blockIdx.x) / gridDim.x);
    const int u_end = (int)(((int64_t)total * (blockIdx.x + 1)) / gridDim.x);
    const int n_units = u_end - u_begin;

    if (warp < C::kProdWarps) {
        // ---------------- producers: query groups and key pages ----------------
        // Every producer warp follows the unit cursor; warp pw issues the keys
        // of units i = pw (mod kProdWarps) and warp 0 also the query groups.
        // Page ids come from two windows of 32 consecutive table entries (lane
        // l holds one), each loaded with one coalesced read one window ahead
        // of its use and range-checked only when it becomes current, so that
        // the read's latency never stalls the copies; lane 0 issues the copies.
        // Stage and meta-slot reuse: unit i waits for the MMA of unit i - S
        // (S = key stages, a multiple of 2, so the same producer and MMA
        // thread), which itself waited for unit i - S's keys and for earlier
        // epilogues; the meta ring (kMetaSlots, set per variant with its
        // argument) is long enough that the slot of unit i is then free.
        const int pw = warp;
        bool ok = true;
        int gcount = 0, pb = -1, pg = -1;
        int q_issued = 0;      // query groups whose copy was issued (lane 0)
        int last_issued = -1;  // last unit whose key copies were issued (lane 0)
        Cursor c;
        if (n_units > 0) cursor_seek(c, bt, sReq, G, u_begin);
        int wb = -1, wlp0 = 0, wcur = -1, wnext = -1;
        auto fetch = [&](int lp) {  // raw table entry, -1 past the sequence
            return (lp * kPage < c.seq) ? __ldg(bt.block_table + (int64_t)c.b * bt.max_pages + lp) : -1;
        };
        auto check = [&](int raw, int lp) {  // -1 (and the status set) for a bad page id
            if (lp * kPage < c.seq && (raw < 0 || raw >= bt.num_pages)) {
                record_error(p.status, DSA_ERR_DEVICE_CHECK);
                return -1;
            }
            return raw;
        };
        for (int i = 0; i < n_units && ok; ++i) {
            const int cb = c.b, cg = c.g, cq0 = c.q0;
            const bool mine = C::kProdWarps == 1 || i % C::kProdWarps == pw;
            const bool qnew = pw == 0 && (cb != pb || cg != pg);  // warp-uniform
            int go = 1;
            if (qnew) {
                if (lane == 0) {
                    const int x = gcount & 1;
                    if (gcount >= 2 &&
                        !mbar_wait(&bars->qempty[x], ((gcount >> 1) - 1) & 1, abort_flag))
                        go = 0;
                    if (go) {
                        mbar_arrive_expect_tx(&bars->qfull[x], (uint32_t)N * kIdxDim);
                        tma_load_2d(sQ + x * kQBufBytes, &tm_q, 0, (cq0 + cg * G) * kIdxHeads,
                                    &bars->qfull[x]);
                        ++q_issued;
                    }
                }
                ++gcount;
                pb = cb;
                pg = cg;
            }
            if (mine) {
                const int lp = c.tile * 2;
                if (c.b != wb || lp < wlp0 || lp >= wlp0 + 64) {
                    wb = c.b;
                    wlp0 = lp;
                    wnext = fetch(lp + 32 + lane);
                    wcur = check(fetch(lp + lane), lp + lane);
                } else if (lp >= wlp0 + 32) {
                    wlp0 += 32;
                    wcur = check(wnext, wlp0 + lane);
                    wnext = fetch(wlp0 + 32 + lane);
                }
                const int pages[2] = {__shfl_sync(0xffffffffu, wcur, lp - wlp0),
                                      __shfl_sync(0xffffffffu, wcur, lp - wlp0 + 1)};
                if (lane == 0 && go) {
                    uint32_t bytes = 0;
                    for (int h = 0; h < 2; ++h)
                        bytes += (pages[h] >= 0 ? (kMx ? kPage * kIdxDim / 2 : kPage * kIdxDim) : 0) +
                                 kPage * 4;
                    // the 64 scale words of each page land in meta slot
                    // i % (S + 3), completing on the same barrier as the keys
                    uint8_t* meta = sMeta + (i % C::kMetaSlots) * kMetaBytes;
                    if (!kMx) {
                        const int st = i % C::kStages, kq = i / C::kStages;
                        if (kq >= 1 && !mbar_wait(&bars->empty[st], (kq - 1) & 1, abort_flag)) go = 0;
                        if (go) {
                            last_issued = i;
                            mbar_arrive_expect_tx(&bars->full[st], bytes);
                            for (int h = 0; h < 2; ++h) {
                                if (pages[h] >= 0)
                                    tma_load_2d(sStage + st * kStageBytes + h * (kPage * kIdxDim),
                                                &tm_keys, 0, pages[h] * (kFp8PageBytes / kIdxDim),
                                                &bars->full[st]);
                                bulk_copy_g2s(meta + h * kPage * 4,
                                              pages[h] >= 0 ? (const void*)(p.pages + (int64_t)pages[h] * kFp8PageBytes +
                                                                            kPage * kIdxDim)
                                                            : (const void*)g_absent_scales,
                                              (uint32_t)(kPage * 4), &bars->full[st]);
                            }
                        }
                    } else {
                        // packed E2M1 bytes of the two pages into a staging
                        // slot; the wait for the MMA of unit i - S frees meta
                        // slot i % (S + 3) (as for FP8 keys)
                        const int ss = i % kStgSlots, kq = i / kStgSlots;
                        if (kq >= 1 && !mbar_wait(&bars->sempty[ss], (kq - 1) & 1, abort_flag)) go = 0;
                        if (go && i >= C::kStages &&
                            !mbar_wait(&bars->empty[i % C::kStages], ((i / C::kStages) - 1) & 1, abort_flag))
                            go = 0;
                        if (go) {
                            last_issued = i;
                            mbar_arrive_expect_tx(&bars->sfull[ss], bytes);
                            for (int h = 0; h < 2; ++h) {
                                if (pages[h] >= 0)
                                    bulk_copy_g2s(sStg + ss * kStgBytes + h * (kPage * kIdxDim / 2),
                                                  p.pages + (int64_t)pages[h] * kMxPageBytes,
                                                  (uint32_t)(kPage * kIdxDim / 2), &bars->sfull[ss]);
                                bulk_copy_g2s(meta + h * kPage * 4,
                                              pages[h] >= 0 ? (const void*)(p.pages + (int64_t)pages[h] * kMxPageBytes +
                                                                            kPage * kIdxDim / 2)
                                                            : (const void*)g_absent_scales,
                                              (uint32_t)(kPage * 4), &bars->sfull[ss]);
                            }
                        }
                    }
                }
            }
            if (mine || qnew) {
                if (!__shfl_sync(0xffffffffu, go, 0)) {
                    ok = false;
                    break;
                }
            }
            cursor_next(c, bt, G);
        }
        // The copies this warp issued must have landed before the CTA exits,
        // also after an abort (their destination is this CTA's shared
        // memory).  Units are issued in order, so the pending ones are among
        // the last ring's worth; in a normal run these phases have completed.
        if (lane == 0) {
            constexpr int kRing = kMx ? kStgSlots : C::kStages;
            for (int j = 0; j < kRing; ++j) {
                const int u = last_issued - j;
                if (u < 0) break;
                if (C::kProdWarps > 1 && u % C::kProdWarps != pw) continue;
                if (kMx) mbar_drain(&bars->sfull[u % kStgSlots], (u / kStgSlots) & 1);
                else mbar_drain(&bars->full[u % C::kStages], (u / C::kStages) & 1);
            }
            for (int gq = q_issued - 1; gq >= 0 && gq >= q_issued - 2; --gq)
                mbar_drain(&bars->qfull[gq & 1], (gq >> 1) & 1);
        }
        __syncwarp();
    } else if (warp < C::kMmaWarp + C::kMmaWarps) {
        // ---------------- MMA issue ----------------
        // FP8 keys: two issuing threads (lane 0 of two warps) take alternate
        // units, since one thread's waits, MMAs and commits of a unit take
        // longer than the unit's keys take to arrive or the tensor pipe needs
        // for the unit's MMAs.  Both follow every
        // query-group change: each releases the old query buffer with its own
        // commit (the buffer's barrier counts both) and waits for the new one.
        // Each unit's stage, accumulator and scale slot belong to that unit
        // alone, so the two threads' MMAs never share an operand they write.
        const int mw = warp - C::kMmaWarp;
        if (lane == 0 && n_units > 0) {
            Cursor c;
            cursor_seek(c, bt, sReq, G, u_begin);
            const uint32_t idesc = make_idesc(kFmtE4M3, kFmtE4M3, 128, N, false, false);
            const uint32_t idesc_h0 = make_idesc(kFmtE4M3, kFmtE4M3, 128, kIdxHeads * H, false, false);
            const uint32_t idesc_h1 = make_idesc(kFmtE4M3, kFmtE4M3, 128, kIdxHeads * (G - H), false, false);
            // descriptors of stage 0 and query buffer 0; a byte offset o moves
            // the start-address field (16-byte units, 14 bits) by o >> 4
            const uint64_t a0 = smem_desc(smem_u32(sStage), 16, 1024, kSwizzle128B);
            const uint64_t b0 = smem_desc(smem_u32(sQ), 16, 1024, kSwizzle128B);
            int gcount = 0, pb = -1, pg = -1;
            // accumulator and its use count of this thread's next unit, kept
            // as counters (the unit index divided by a run-time count costs
            // tens of instructions): one thread cycles through nacc
            // accumulators; kDual: thread mw through its own three; kWide:
            // thread mw always fills accumulator mw; ring of three: unit i
            // uses accumulator i % 3, so a thread's accumulator steps by 2.
            //
            // Ring of three, barrier pairing: tfull[a] completes once per unit
            // on a, in unit order (the MMA of unit i waits for the epilogue of
            // unit i - 3, which waited for tfull of i - 3), and set a, the only
            // one draining a, waits for its units in that order.  The epilogue
            // of unit j arrives on tempty[2 (j % 3) + (j & 1)], whose phase n is
            // the unit j = 6 n + const; the thread of parity p waits at unit i
            // for unit j = i - 3 there, and that barrier's previous phase (unit
            // i - 9) has completed, since the same thread's unit i - 6 waited
            // for it: the parity wait cannot alias.  Meta slots: the producer
            // of unit i reuses the slot of unit i - S - 7 once the MMA of unit
            // i - S has completed; that thread's units i - S, i - S - 2 and
            // i - S - 4 waited for the epilogues of units i - S - 3, - 5 and
            // - 7, one per accumulator, and each set drains its accumulator's
            // units in order.
            const int a_period = kDual ? 3 : (kWide ? 1 : nacc);
            const int a_base = kDual ? 3 * mw : (kWide ? mw : 0);
            int a_next = 0, u_next = 0;
            int r3 = mw;  // ring of three: this thread's next accumulator
            bool ok = true;
            for (int i = 0; i < n_units && ok; ++i) {
                if (c.b != pb || c.g != pg) {
                    if (gcount >= 1) mma_commit(&bars->qempty[(gcount - 1) & 1]);
                    ok = mbar_wait(&bars->qfull[gcount & 1], (gcount >> 1) & 1, abort_flag);
                    ++gcount;
                    pb = c.b;
                    pg = c.g;
                }
                if (ok && (C::kMmaWarps == 1 || i % C::kMmaWarps == mw)) {
                    const int st = i % C::kStages;
                    const int acc = ring3 ? r3 : a_base + a_next, use = u_next;
                    if (ring3) {
                        r3 = (r3 == 0) ? 2 : r3 - 1;
                    } else if (++a_next == a_period) {
                        a_next = 0;
                        ++u_next;
                    }
                    ok = mbar_wait(&bars->full[st], (i / C::kStages) & 1, abort_flag);
                    if (!ok) break;
                    const uint64_t ad = a0 + (uint64_t)((st * kStageBytes) >> 4);
                    const uint64_t bd = b0 + (uint64_t)((((gcount - 1) & 1) * kQBufBytes) >> 4);
                    if (tsplit) {
                        // each token half waits only for the set that drained
                        // the same half of this accumulator one use earlier;
                        // its query rows start 32 H rows (of 128 B) further on
                        for (int hh = 0; hh < 2; ++hh) {
                            const int bi = 2 * acc + hh;
                            if (use >= 1 && !mbar_wait(&bars->tempty[bi], (use - 1) & 1, abort_flag)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint64_t bh = bd + (uint64_t)((hh * H * kIdxHeads * kIdxDim) >> 4);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_f8f6f4(tmem + acc * acc_cols + hh * kIdxHeads * H, ad + 2 * kk, bh + 2 * kk,
                                           hh ? idesc_h1 : idesc_h0, kk > 0 ? 1u : 0u);
                            mma_commit(&bars->tfull[bi]);
                        }
                        if (!ok) break;
                    } else {
                        if (ring3) {
                            if (i >= 3 && !mbar_wait(&bars->tempty[2 * acc + ((i - 3) & 1)], ((i - 3) / 6) & 1,
                                                     abort_flag))
                                break;
                        } else if (use >= 1 && !mbar_wait(&bars->tempty[acc], (use - 1) & 1, abort_flag)) {
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            if (kMx)  // one accumulator per 32-element block
                                mma_f8f6f4(tmem + acc * acc_cols + kk * N, ad + 2 * kk, bd + 2 * kk, idesc, 0u);
                            else
                                mma_f8f6f4(tmem + acc * acc_cols, ad + 2 * kk, bd + 2 * kk, idesc,
                                           kk > 0 ? 1u : 0u);
                        }
                        mma_commit(&bars->tfull[acc]);
                    }
                    mma_commit(&bars->empty[st]);
                }
                cursor_next(c, bt, G);
            }
        }
        if (lane == 0) {
            // nothing may still write TMEM when it is released, also after an
            // abort
            mma_commit(&bars->done);
            mbar_drain(&bars->done, 0);
        }
        __syncwarp();
    } else if (warp < C::kEpiWarp0) {
        // ---------------- MXFP4 converters: E2M1 -> E4M3 A-operand tiles ----------
        const int ctid = tid - 32 * C::kConvWarp0;  // 0..127
        for (int i = 0; i < n_units; ++i) {
            const int ss = i % kStgSlots, st = i % C::kStages;
            if (!mbar_wait(&bars->sfull[ss], (i / kStgSlots) & 1, abort_flag)) break;
            if (i >= C::kStages && !mbar_wait(&bars->empty[st], ((i / C::kStages) - 1) & 1, abort_flag))
                break;
            const uint8_t* src = sStg + ss * kStgBytes;
            uint8_t* dst = sStage + st * kStageBytes;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                // 1024 chunks of 16 elements: key r, elements 16c .. 16c+15
                const int q = ctid + 128 * k;
                const int r = q >> 3, cidx = q & 7;
                const uint2 packed = *reinterpret_cast<const uint2*>(src + r * 64 + cidx * 8);
                const uint2 a = e2m1x8_to_e4m3x8(packed.x);
                const uint2 b2 = e2m1x8_to_e4m3x8(packed.y);
                *reinterpret_cast<uint4*>(dst + sw128(r, cidx * 16)) = make_uint4(a.x, a.y, b2.x, b2.y);
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars->full[st]);
            mbar_arrive(&bars->sempty[ss]);
        }
    } else {
        // ---------------- epilogue (thread = key) ----------------
        const int etid = tid - 32 * C::kEpiWarp0;
        const int quarter = warp & 3;                 // TMEM lanes 32*quarter..+31
        const int half = (warp - C::kEpiWarp0) >> 2;  // warp set (FP8: unit parity, MXFP4: token parity)
        constexpr int kTS = C::kTokSplit;
        // the unit loop, specialised on token halves (kSplit) at compile time
        auto drain = [&](auto split_tag) {
            constexpr bool kSplit = decltype(split_tag)::value;
            Cursor c;
            cursor_seek(c, bt, sReq, G, u_begin);
            int gcount = 0, pb = -1, pg = -1;
            // FP8: the warp sets take whole units round robin (the per-unit
            // bookkeeping runs on four warps, and the sets drain different
            // accumulators at once): with the ring of three, set `half` takes
            // the units i = half (mod 3), all on accumulator `half`; kDual: the
            // units of parity `half`, on MMA thread half's accumulators in
            // turn.  MXFP4: every set takes every unit.  With token halves
            // (kSplit, kWide) the work items are (unit, half) and set s takes
            // every half s % 2 of the units of parity s / 2 (accumulator
            // s / 2, filled by MMA thread s / 2 for the (i / 2)-th time at
            // unit i), so each barrier pair has one producer thread and one
            // consuming set, and a set's previous item was the previous phase
            // of the barrier it waits on.
            const int step = kMx ? 1 : (kDual ? 2 : nacc);
            const int first = kMx ? 0 : ((kDual || half < nacc) ? half : n_units);
            const int a_period = kMx ? nacc : (kDual ? 3 : 1);
            const int a_base = kMx ? 0 : (kDual ? 3 * half : half);
            int a_next = 0, u_next = 0;
            const int n_items = kSplit ? 2 * n_units : n_units;
            const int item0 = kSplit ? half : first;
            const int istep = kSplit ? C::kEpiSets : step;
            int cur = 0;  // the unit the cursor is on
            for (int it = item0; it < n_items; it += istep) {
                const int i = kSplit ? (it >> 1) : it;
                for (; cur < i; ++cur) cursor_next(c, bt, G);
                const int gtok0 = c.g * G;                    // first token of the group
                const int gr = min(G, c.nb - gtok0);          // real tokens in the group
                // this item's tokens [jlo, jhi) of the group
                const int jlo = kSplit ? (it & 1) * H : 0;
                const int jhi = kSplit ? min(gr, jlo + H) : gr;
                if (c.b != pb || c.g != pg) {
                    if (kMx) {
                        float* wdst = sW + (gcount & 1) * (8 * kIdxHeads);
                        for (int e = etid; e < gr * kIdxHeads; e += C::kEpiThreads) {
                            const int64_t t = c.q0 + gtok0 + e / kIdxHeads;
                            const int h = e % kIdxHeads;
                            wdst[e] = __ldg(p.w + t * kIdxHeads + h) * __ldg(p.qscale + t * kIdxHeads + h);
                        }
                        asm volatile("bar.sync 2, %0;" ::"n"(C::kEpiThreads) : "memory");
                    } else {
                        // each warp set keeps its own copy (barrier 3 + set over
                        // its 128 threads, which follow the same units)
                        float* wdst = sW + half * (8 * kIdxHeads);
                        asm volatile("bar.sync %0, 128;" ::"r"(3 + half) : "memory");
                        for (int e = etid - 128 * half; e < gr * kIdxHeads; e += 128) {
                            const int64_t t = c.q0 + gtok0 + e / kIdxHeads;
                            const int h = e % kIdxHeads;
                            wdst[e] = __ldg(p.w + t * kIdxHeads + h) * __ldg(p.qscale + t * kIdxHeads + h);
                        }
                        asm volatile("bar.sync %0, 128;" ::"r"(3 + half) : "memory");
                    }
                    ++gcount;
                    pb = c.b;
                    pg = c.g;
                }
                const float* wq = kMx ? sW + ((gcount - 1) & 1) * (8 * kIdxHeads)
                                      : sW + half * (8 * kIdxHeads);
                const int s = c.tile * kTile + quarter * 32 + lane;
                const bool in_seq = s < c.seq;
                int acc, use;
                if (kSplit) {
                    acc = i & 1;
                    use = i >> 1;
                } else {
                    acc = a_base + a_next;
                    use = u_next;
                    if (++a_next == a_period) {
                        a_next = 0;
                        ++u_next;
                    }
                }
                // the barriers of the accumulator (of its token half); with the
                // ring of three, the drain barrier also by the unit's parity
                const int bi = kSplit ? 2 * acc + (it & 1) : acc;
                const int be = (!kSplit && ring3) ? 2 * acc + (i & 1) : bi;
                if (!mbar_wait(&bars->tfull[bi], use & 1, abort_flag)) break;
                tc_fence_after();
                // the unit's scale words arrived with its keys (before tfull)
                const uint32_t sw = reinterpret_cast<const uint32_t*>(
                    sMeta + (i % C::kMetaSlots) * kMetaBytes)[quarter * 32 + lane];
                // a key of an absent or out-of-range page has all scale bits set
                const bool page_ok = sw != 0xFFFFFFFFu;
                float kscale = 0.f;                   // FP8: per-key scale
                float bsc[4] = {0.f, 0.f, 0.f, 0.f};  // MXFP4: block scales 2^(e-127)
                if (!kMx) {
                    kscale = __uint_as_float(sw);
                } else {
#pragma unroll
                    for (int bb = 0; bb < 4; ++bb) {
                        const int ev = (sw >> (8 * bb)) & 0xFF;
                        bsc[bb] = (ev == 0xFF) ? __int_as_float(0x7fffffff) : ldexpf(1.0f, ev - 127);
                    }
                }
                if (!kMx) {
                    // the key's score cell of the group's first token, and the
                    // number of visible positions the key needs (one more per
                    // later token): a page-absent or out-of-range key is masked
                    // as if no token saw it
                    float* cell = p.scores + (int64_t)(c.q0 + gtok0 + jlo) * p.ld + s;
                    const int need = (in_seq && page_ok) ? s - (c.seq - c.nb + gtok0) : INT_MAX;
                    // one token's 32 head logits -> its weighted ReLU sum, stored
                    auto score = [&](const uint32_t(&v)[32], int jt) {
                        const float* wt = wq + jt * kIdxHeads;
                        // two independent packed (f32x2) partial sums, heads
                        // (4i, 4i+1) and (4i+2, 4i+3)
                        uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
                        for (int h4 = 0; h4 < 8; ++h4) {
                            const float4 ww = lds_f32x4(wt + 4 * h4);
                            if constexpr (kWide) {
                                acc2[0] = fma_f32x2(pair_f32(ww.x, ww.y),
                                                    relu_pair(v[4 * h4 + 0], v[4 * h4 + 1]), acc2[0]);
                                acc2[1] = fma_f32x2(pair_f32(ww.z, ww.w),
                                                    relu_pair(v[4 * h4 + 2], v[4 * h4 + 3]), acc2[1]);
                            } else {
                                acc2[0] = fma_f32x2(
                                    pack_f32x2(ww.x, ww.y),
                                    pack_f32x2(fmaxf(__uint_as_float(v[4 * h4 + 0]), 0.f),
                                               fmaxf(__uint_as_float(v[4 * h4 + 1]), 0.f)),
                                    acc2[0]);
                                acc2[1] = fma_f32x2(
                                    pack_f32x2(ww.z, ww.w),
                                    pack_f32x2(fmaxf(__uint_as_float(v[4 * h4 + 2]), 0.f),
                                               fmaxf(__uint_as_float(v[4 * h4 + 3]), 0.f)),
                                    acc2[1]);
                            }
                        }
                        const float sc = ((lo_f32x2(acc2[0]) + hi_f32x2(acc2[0])) +
                                          (lo_f32x2(acc2[1]) + hi_f32x2(acc2[1]))) * kscale;
                        // token jt sees s when s < seq - nb + gtok0 + jt + 1
                        if (in_seq) *cell = (need <= jt) ? sc : -INFINITY;
                        cell += p.ld;
                    };
                    const uint32_t tcol = tmem_addr(tmem, 32 * quarter, acc * acc_cols);
                    if (kWide) {
                        // one token per TMEM load (the register budget of 19
                        // warps; four sets hide the load latency)
                        for (int j = jlo; j < jhi; ++j) {
                            uint32_t v[32];
                            tmem_ld32(tcol + 32 * j, v);
                            tmem_wait_ld();
                            score(v, j);
                        }
                    } else {
                        // tokens two at a time: both TMEM loads, then one wait
                        for (int j = jlo; j < jhi; j += 2) {
                            uint32_t v[2][32];
                            tmem_ld32(tcol + 32 * j, v[0]);
                            if (j + 1 < jhi) tmem_ld32(tcol + 32 * (j + 1), v[1]);
                            tmem_wait_ld();
                            score(v[0], j);
                            if (j + 1 < jhi) score(v[1], j + 1);
                        }
                    }
                } else {
                    for (int j = half; j < gr; j += kTS) {
                        float x[32];
#pragma unroll
                        for (int h = 0; h < 32; ++h) x[h] = 0.f;
#pragma unroll
                        for (int bb = 0; bb < 4; ++bb) {
                            uint32_t v[32];
                            tmem_ld32(tmem_addr(tmem, 32 * quarter, acc * acc_cols + bb * N + 32 * j), v);
                            tmem_wait_ld();
#pragma unroll
                            for (int h = 0; h < 32; ++h) x[h] = fmaf(bsc[bb], __uint_as_float(v[h]), x[h]);
                        }
                        const float4* w4 = reinterpret_cast<const float4*>(wq + j * kIdxHeads);
                        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                        for (int h4 = 0; h4 < 8; ++h4) {
                            const float4 ww = w4[h4];
                            s0 = fmaf(ww.x, fmaxf(x[4 * h4 + 0], 0.f), s0);
                            s1 = fmaf(ww.y, fmaxf(x[4 * h4 + 1], 0.f), s1);
                            s2 = fmaf(ww.z, fmaxf(x[4 * h4 + 2], 0.f), s2);
                            s3 = fmaf(ww.w, fmaxf(x[4 * h4 + 3], 0.f), s3);
                        }
                        const float sc = (s0 + s1) + (s2 + s3);
                        if (in_seq) {
                            const int vis = c.seq - c.nb + gtok0 + j + 1;
                            p.scores[(int64_t)(c.q0 + gtok0 + j) * p.ld + s] =
                                (s < vis && page_ok) ? sc : -INFINITY;
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars->tempty[be]);
            }
        };
        if (n_units > 0) {
            if (tsplit) drain(std::integral_constant<bool, true>{});
            else drain(std::integral_constant<bool, false>{});
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && tid == 0) record_error(p.status, DSA_ERR_TIMEOUT);
    if (warp == C::kMmaWarp) tmem_dealloc(tmem, 512);
}

}  // namespace

// The driver's tensor-map encoder, looked up once (shared with front.cu).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

namespace {

// 2-D byte tensor [rows, 128] with 128-byte rows, box [box_rows, 128], 128-B swizzle.
bool encode_rows128(CUtensorMap* tm, const void* base, uint64_t rows, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {128, rows};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}


template <int kFmt, bool kDual, bool kWide = false>
cudaError_t launch_tc(const BatchArgs& bt, const uint8_t* q8, const float* qscale, const float* w,
                      const void* pages, float* scores, int64_t ld, int32_t* status,
                      cudaStream_t stream) {
    using C = IdxCfg<kFmt, kDual, kWide>;
    IdxParams p;
    p.bt = bt;
    p.qscale = qscale;
    p.w = w;
    p.pages = static_cast<const uint8_t*>(pages);
    p.scores = scores;
    p.ld = ld;
    p.G = bt.max_q < C::kMaxG ? (bt.max_q > 0 ? bt.max_q : 1) : C::kMaxG;
    p.N = kIdxHeads * p.G;
    p.status = status;
    CUtensorMap tm_keys, tm_q;
    memset(&tm_keys, 0, sizeof(tm_keys));
    // FP8 index pool as rows of 128 bytes: page p = rows [66p, 66p + 64) + 2 scale rows
    if (!C::kMx && !encode_rows128(&tm_keys, pages,
                                   (uint64_t)bt.num_pages * (kFp8PageBytes / kIdxDim), kPage))
        return cudaErrorInvalidValue;
    if (!encode_rows128(&tm_q, q8, (uint64_t)bt.total_q * kIdxHeads, (uint32_t)p.N))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(indexer_tc_kernel<kFmt, kDual, kWide>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    // programmatic dependent launch is safe after any predecessor: the kernel
    // reads no global memory before its grid-dependency wait
    return launch_kernel(indexer_tc_kernel<kFmt, kDual, kWide>, dim3(sms), dim3(C::kThreads),
                         (size_t)C::kSmemAlloc, stream, true, 1, tm_keys, tm_q, p);
}

}  // namespace

bool indexer_supported(const BatchArgs& bt) { return bt.num_requests <= kMaxReq; }

cudaError_t launch_index_scores(const BatchArgs& bt, const uint8_t* q8, const float* qscale,
                                const float* w, const void* pages, int key_format,
                                float* scores, int64_t ld, int32_t* status,
                                cudaStream_t stream) {
    if (key_format == DSA_KEYS_MXFP4)
        return launch_tc<DSA_KEYS_MXFP4, false>(bt, q8, qscale, w, pages, scores, ld, status, stream);
    // groups of one or two tokens: the copies and MMAs of a unit, not its
    // epilogue, bound the rate, so two threads issue each
    if (bt.max_q <= 2)
        return launch_tc<DSA_KEYS_FP8_E4M3, true>(bt, q8, qscale, w, pages, scores, ld, status, stream);
    // groups of 6-8 tokens (two accumulators): one MMA thread per accumulator
    // and four epilogue sets, one per accumulator half; groups of 3-5: three
    // accumulators shared by two MMA threads, one epilogue set each
    if (bt.max_q >= 6)
        return launch_tc<DSA_KEYS_FP8_E4M3, false, true>(bt, q8, qscale, w, pages, scores, ld, status,
                                                          stream);
    return launch_tc<DSA_KEYS_FP8_E4M3, false>(bt, q8, qscale, w, pages, scores, ld, status, stream);
}

}  // namespace dsa
