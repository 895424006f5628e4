// sparse_mla.cu -- absorbed-form MLA over the selected tokens, on tcgen05.
//
// For query token t and head h over the selected positions I:
//   z[h,s]     = sm_scale * kv_scale * (q_lat[t,h,:] . E4M3(latent[s,:]))   (576 dims)
//   out[t,h,:] = kv_scale * sum_s softmax_s(z)[s] * E4M3(latent[s,0:512])
// "vLLM's Kimi K3.1 Pro day-0 support", section "What changed" (MLA run
// exactly on the 2048 selected tokens) and section "Sparse attention cuts
// long-context decode bandwidth" (the 576-byte FP8 latents are read for the
// selected tokens only).
//
// One CTA = one query token x one contiguous split of its index slots, taken
// in tiles of 64 selected tokens.  The batch runs as whole waves of one CTA
// per token, and the tokens left for a last, partial wave are split into as
// many pieces as keep that wave full (powers of two, up to 16); the pieces'
// partial results are merged by a second kernel.
//   S   = Q . L^T    tcgen05 kind::f16, M = 128 (96 heads + 32 unused rows),
//                    N = 64 selected tokens, K = 576; accumulator in TMEM
//   O^T = V^T . P^T  M = 128 latent dims (4 tiles cover 512), N = 96 heads,
//                    K = 64 tokens; accumulator in TMEM (4 x 96 columns)
// An MMA with N <= 64 costs about as much as one with N = 128, so the tile is
// as wide as shared memory allows: the query (110.6 KB of f16) and one latent
// tile (73.7 KB of f16) leave no room for a second latent stage.  Instead the
// tile is refilled in five slab groups (latent dims 0-127, 128-255, 256-383,
// 384-511 and 512-575): a group is overwritten with the next tile's latents as
// soon as the MMAs reading it have completed, so the next S = Q . L^T starts
// while the current O^T update is still running.
//
// Latents are gathered with 16-byte loads from the paged cache (each group one
// tile ahead, in registers) and lifted E4M3 -> f16 exactly into a
// 128-byte-swizzled tile that serves both as the K-major B operand of S and as
// the MN-major A operand of O^T.  The bf16 query is converted in the kernel to
// f16 after a per-token power-of-two scale (exact for every element within
// 2^-14 of the largest).  Softmax runs online in the log2 domain with
// conditional rescaling: a head's reference maximum only moves when a new
// maximum exceeds it by more than 2^8, and the O^T columns are then rescaled
// in TMEM.
//
// Warp roles (256 threads, so a thread may hold up to 255 registers): warps
// 0-3 softmax (thread = head), warps 4-6 gather/convert producers, warp 7 TMEM
// allocation and the single MMA-issuing thread; all eight warps share the
// epilogue (thread = latent dim), which stages the result in shared memory and
// writes it with one bulk copy.  Every wait is bounded.
#include <cuda_fp4.h>

#include "common.cuh"
#include "sm100.cuh"

namespace dsa {

using namespace sm100;

namespace {

constexpr int kTileKeys = 64;
constexpr int kThreads = 256;
constexpr int kProducers = 96;                                // warps 4-6
constexpr int kMmaWarp = 7;
constexpr int kQRows = 96;
constexpr int kSlabs = kLatDim / 64;                          // 9 K-slabs of 64 dims
constexpr int kGroups = 5;                                    // slab groups of a latent tile
constexpr int kQSlabBytes = kQRows * 128;                     // 12288
constexpr int kQBytes = kSlabs * kQSlabBytes;                 // 110592
constexpr int kPBytes = kQRows * 128;                         // 12288: 96 heads x 64 keys f16
constexpr int kLSlabBytes = kTileKeys * 128;                  // 8192
constexpr int kLBytes = kSlabs * kLSlabBytes;                 // 73728
constexpr int kOutBytes = kMlaHeads * kVDim * 2;              // 98304 (bf16 or f16)
constexpr int kMaxSplitKeys = kTopK;                          // index slots per CTA, max
constexpr int kOffQ = 0;
// The M = 128 reads of a 96-row Q slab run 4 KB past it; for the last slab
// that lands in the P buffer (valid shared memory, unused accumulator rows).
constexpr int kOffP = kOffQ + kQBytes;
constexpr int kOffL = kOffP + kPBytes;
constexpr int kOffRow = kOffL + kLBytes;                      // int32 row ids
constexpr int kOffMask = kOffRow + kMaxSplitKeys * 4;         // valid-slot mask per tile
constexpr int kOffF = kOffMask + (kMaxSplitKeys / kTileKeys) * 8;  // per-head floats
constexpr int kOffBar = kOffF + 512 * 4;
constexpr int kSmemBytes = kOffBar + 256;
constexpr int kSmemAlloc = kSmemBytes + 1024;                 // slack for 1024-B alignment
static_assert(kSmemAlloc <= 227 * 1024, "shared memory budget");
static_assert(kOffP % 1024 == 0 && kOffL % 1024 == 0, "swizzled tiles are 1024-B aligned");
static_assert(kOutBytes <= kQBytes, "the epilogue stages the output in the query buffer");

// TMEM columns
constexpr uint32_t kColS = 0;     // one 64-column S buffer
constexpr uint32_t kColO = 64;    // four 96-column O^T tiles
constexpr uint32_t kTmemCols = 512;

constexpr float kRescaleLog2 = 8.0f;  // move the reference max when exceeded by > 2^8

constexpr uint32_t kIdescQK = make_idesc(kFmtF16, kFmtF16, 128, kTileKeys, false, false);
constexpr uint32_t kIdescPV = make_idesc(kFmtF16, kFmtF16, 128, kQRows, true, false);

struct Bars {
    uint64_t lfull[kGroups];   // producers -> MMA: slab group of the latent tile written
    uint64_t lempty[kGroups];  // MMA -> producers: slab group free (commit)
    uint64_t sfull;            // MMA -> softmax: S ready, every earlier O^T update done
    uint64_t pfull;            // softmax -> MMA: P written, S read (128 arrivals)
    uint64_t done;             // MMA -> epilogue: everything finished
    uint32_t tmem_base;
    int abort_flag;
};

// 2^x by the special-function unit (flushes results below 2^-126 to zero;
// 2^-inf = +0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Pairs of fp32 in one 64-bit register (low word = first element) and their
// packed arithmetic; f16 pairs in one 32-bit register.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float lo_f32(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_f32(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// (lo, hi) fp32 -> f16 pair, round to nearest even
__device__ __forceinline__ uint32_t f32x2_to_f16x2(uint64_t v) {
    __half2 h = __floats2half2_rn(lo_f32(v), hi_f32(v));
    return *reinterpret_cast<uint32_t*>(&h);
}
// max(a, b, c) in one instruction
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// s_lo += lo(e), s_hi += hi(e) for an f16 pair e, each f16 value converted
// exactly and added in fp32 with one rounding
__device__ __forceinline__ void add_f16x2_to_f32(uint32_t e, float& s_lo, float& s_hi) {
    asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.f16 %0, l, %0;\n\tadd.rn.f32.f16 %1, h, %1;\n\t}"
        : "+f"(s_lo), "+f"(s_hi)
        : "r"(e));
}
// 2^x of an f16 pair by the special-function unit (2^-inf = +0)
__device__ __forceinline__ uint32_t ex2_f16x2(uint32_t x) {
    uint32_t y;
    asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Barrier over the 128 softmax threads (warps 0-3), returning whether any of the 128 threads passed `pred`.
__device__ __forceinline__ bool softmax_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred q, o;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred o, 1, 128, q;\n\tselp.u32 %0, 1, 0, o;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u)
        : "memory");
    return r != 0;
}

// Shared -> global bulk copy of `bytes` (16-byte aligned, multiple of 16),
// waited for until the source has been read.
__device__ __forceinline__ void bulk_store_s2g(void* gdst, const void* ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Four f16 pairs from eight E4M3 bytes (exact).
__device__ __forceinline__ void e4m3x8_to_f16x8(uint32_t w0, uint32_t w1, uint32_t (&h)[4]) {
    const uint32_t wv[2] = {w0, w1};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(wv[k] & 0xFFFF), __NV_E4M3);
        __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(wv[k] >> 16), __NV_E4M3);
        h[2 * k] = *reinterpret_cast<uint32_t*>(&lo);
        h[2 * k + 1] = *reinterpret_cast<uint32_t*>(&hi);
    }
}

// Eight packed E2M1 elements (element 2i in the low nibble of byte i) -> eight
// f16 values, exact (every E2M1 value is an f16 value): one hardware
// conversion per byte.
__device__ __forceinline__ uint4 e2m1x8_to_f16x8(uint32_t w) {
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __half2_raw h = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((w >> (8 * j)) & 0xFFu),
                                                         __NV_E2M1);
        o[j] = (uint32_t)h.x | ((uint32_t)h.y << 16);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// NVFP4 latent row (352 B): packed E2M1 of dims 0..511, 32 E4M3 block scales
// (one per 16 elements), E4M3 of dims 512..575.
constexpr int kNvRowBytes = kVDim / 2 + kVDim / 16 + (kLatDim - kVDim);  // 352
constexpr int kNvScaleOff = kVDim / 2;                                   // 256
constexpr int kNvTailOff = kNvScaleOff + kVDim / 16;                     // 288

struct MlaParams {
    BatchArgs bt;
    const __nv_bfloat16* q_lat;  // [T][96][576]
    const uint8_t* latent_pages;
    const int32_t* indices;
    int K;                 // index slots per token
    int full_tokens;       // tokens [0, full_tokens) run as one CTA each
    int tail_splits;       // the other tokens as tail_splits CTAs each
    float kv_scale;
    float sm_scale;
    __nv_bfloat16* out;    // final outputs (tokens run whole)
    float* lse;            // final lse, nullable
    __half* part_o;        // [T - full_tokens, tail_splits, 512, 96] normalised partial outputs
    float* part_lse;       // [T - full_tokens, tail_splits, 96] partial lse, log2 domain
    int32_t* status;
};

// kWaitTest: the variant of the test-only export -- the producers withhold one
// arrival (the latent slab group 512-575 of the first tile) and every wait has
// a budget of 2^20 cycles, so the MMA thread's wait runs out and the kernel
// takes its abort path.  kLat: latent pages as FP8 (0, 576 B per token) or
// NVFP4 (1, 352 B per token); both are lifted exactly to f16 by the producers.
template <bool kWaitTest, int kLat>
__global__ void __launch_bounds__(kThreads, 1) sparse_mla_tc_kernel(const MlaParams p) {
    constexpr long long kBudget = kWaitTest ? (1ll << 20) : kWaitCycles;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = sm + kOffQ;
    uint8_t* sP = sm + kOffP;
    uint8_t* sL = sm + kOffL;
    int32_t* sRow = reinterpret_cast<int32_t*>(sm + kOffRow);
    uint64_t* sMask = reinterpret_cast<uint64_t*>(sm + kOffMask);
    // [0,128): rescale factors, [256,384): output scale per head, [384,400): reductions
    float* sF = reinterpret_cast<float*>(sm + kOffF);
    Bars* bars = reinterpret_cast<Bars*>(sm + kOffBar);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    grid_dependents_launch();
    const bool whole = (int)blockIdx.x < p.full_tokens;
    const int tail_cta = (int)blockIdx.x - p.full_tokens;  // >= 0 for a split token
    const int t = whole ? (int)blockIdx.x : p.full_tokens + tail_cta / p.tail_splits;
    const int split = whole ? 0 : tail_cta % p.tail_splits;
    const int split_keys = whole ? p.K : p.K / p.tail_splits;
    const int64_t piece = whole ? -1 : (int64_t)tail_cta;  // partial slot of a split token
    const int b = request_of(p.bt, t);
    const bool ok_tok = token_ok(p.bt, b, t, split == 0 ? p.status : nullptr);
    const int seq = __ldg(p.bt.seq_lens + b);
    const int n_tiles = split_keys / kTileKeys;
    const int slot0 = split * split_keys;
    volatile int* abort_flag = &bars->abort_flag;

    if (tid == 0) {
        for (int g = 0; g < kGroups; ++g) {
            mbar_init(&bars->lfull[g], kProducers);
            mbar_init(&bars->lempty[g], 1);
        }
        mbar_init(&bars->sfull, 1);
        mbar_init(&bars->pfull, 128);
        mbar_init(&bars->done, 1);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }

    // ---- preamble 1: the query, bf16 -> f16 after a power-of-two scale 2^-e --
    // (e = 0 unless max|q| >= 2^15 or < 2^-8; then max|q| * 2^-e lies in
    // [2^14, 2^15)), written in the 128-byte-swizzled slabs the MMA reads.
    // One pass converts with e = 0 while finding max|q|; a token that needs
    // e != 0 is converted again.
    constexpr int kQVec = kMlaHeads * kLatDim / 8 / kThreads;  // 27 vectors of 8 per thread
    static_assert(kQVec * kThreads * 8 == kMlaHeads * kLatDim, "query split");
    const uint4* qsrc = reinterpret_cast<const uint4*>(p.q_lat + (int64_t)t * kMlaHeads * kLatDim);
    auto convert_q = [&](float qmul) {
        float amax = 0.f;
#pragma unroll 9
        for (int u = 0; u < kQVec; ++u) {
            const int v = tid + kThreads * u;
            const uint4 r = ok_tok ? __ldg(qsrc + v) : make_uint4(0u, 0u, 0u, 0u);
            const int h = v / (kLatDim / 8), c = v % (kLatDim / 8);
            const uint32_t wv[4] = {r.x, r.y, r.z, r.w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float lo = __uint_as_float(wv[i] << 16), hi = __uint_as_float(wv[i] & 0xFFFF0000u);
                amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
                o[i] = pack_half2(lo * qmul, hi * qmul);
            }
            *reinterpret_cast<uint4*>(sQ + (c / 8) * kQSlabBytes + sw128(h, (c % 8) * 16)) =
                make_uint4(o[0], o[1], o[2], o[3]);
        }
        return amax;
    };
    int e = 0;
    {
        const float amax = warp_max(convert_q(1.0f));
        if (lane == 0) sF[384 + warp] = amax;
        __syncthreads();
        float qmax = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) qmax = fmaxf(qmax, sF[384 + w]);
        if (qmax > 0.f && (qmax >= 32768.f || qmax < 0.00390625f)) {
            int ex;
            frexpf(qmax, &ex);  // qmax = f * 2^ex, f in [0.5, 1)
            e = ex - 15;
            (void)convert_q(ldexpf(1.0f, -e));  // uniform over the CTA
        }
    }

    grid_dependency_wait();  // the indices come from the previous kernel
    // ---- preamble 2: row ids (page * 64 + slot) of this CTA's index slots ----
    // every index load of a thread, then every table load (unconditional, at
    // a clamped page), so the dependent global reads overlap
    {
        constexpr int kPer = (kMaxSplitKeys + kThreads - 1) / kThreads;  // 8
        int s[kPer], pg[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int k = tid + kThreads * u;
            s[u] = (ok_tok && k < split_keys) ? __ldg(p.indices + (int64_t)t * p.K + slot0 + k) : -1;
        }
        const int32_t* table = p.bt.block_table + (int64_t)b * p.bt.max_pages;
#pragma unroll
        for (int u = 0; u < kPer; ++u)
            pg[u] = __ldg(table + ((s[u] >= 0 && s[u] < seq) ? s[u] / kPage : 0));
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int k = tid + kThreads * u;
            if (k < split_keys) {
                int row = -1;
                if (s[u] >= seq) {
                    record_error(p.status, DSA_ERR_DEVICE_CHECK);
                } else if (s[u] >= 0) {
                    if (pg[u] < 0 || pg[u] >= p.bt.num_pages) record_error(p.status, DSA_ERR_DEVICE_CHECK);
                    else row = pg[u] * kPage + (s[u] % kPage);
                }
                sRow[k] = row;
            }
        }
    }
    __syncthreads();
    // valid-slot mask per tile (one ballot per 32 slots)
    for (int i = warp; i < n_tiles; i += kThreads / 32) {
        const uint32_t lo = __ballot_sync(0xffffffffu, sRow[i * kTileKeys + lane] >= 0);
        const uint32_t hi = __ballot_sync(0xffffffffu, sRow[i * kTileKeys + 32 + lane] >= 0);
        if (lane == 0) sMask[i] = ((uint64_t)hi << 32) | lo;
    }
    if (tid < 128) sF[tid] = 1.f;
    fence_proxy_async_smem();  // the query slabs are read by the tensor cores
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem = bars->tmem_base;
    // z in log2 units per unit of the f16 accumulator
    const float zscale = p.sm_scale * p.kv_scale * ldexpf(1.0f, e) * 1.4426950408889634f;
    // tiles after the last one holding a selected position have only empty
    // slots (p = 0, zero latents): every role stops before them, which leaves
    // the result bit-for-bit unchanged
    int n_used = n_tiles;
    while (n_used > 0 && sMask[n_used - 1] == 0ull) --n_used;

    if (warp >= 4 && warp < kMmaWarp) {
        // ---------------- producers: gather + E4M3 -> f16 ----------------
        // a tile is 64 rows x 36 chunks of 16 bytes; slab group g < 4 holds
        // chunks 8g..8g+7 of every row (512 chunks: 6 per thread of warp 4,
        // 5 per thread of warps 5-6), group 4 chunks 32..35 (256 chunks: 3 per
        // thread of warps 4-5, 2 per thread of warp 6).  A group is refilled
        // as soon as it is free, and its next tile is then loaded into the
        // same registers.
        const int pt = tid - 128;
        // NVFP4 (kLat == 1): group g < 4 is 64 rows x 4 items of 32 elements
        // (16 packed bytes + their two block scales), group 4 is 64 rows x 4
        // chunks of 16 E4M3 bytes (dims 512-575): 256 items per group, three
        // per thread of warps 4-5, two per thread of warp 6
        uint4 raw[kGroups][kLat == 0 ? 6 : 3];
        uint32_t rsc[4][kLat == 0 ? 1 : 3];
        (void)rsc;
#define DSA_MLA_CHUNK(g_, u_, r_, c_)                                          \
    const int r_ = ((g_) < 4) ? ((ptv >> 3) + 12 * (u_)) : ((ptv >> 2) + 24 * (u_)); \
    const int c_ = ((g_) < 4) ? (8 * (g_) + (ptv & 7)) : (32 + (ptv & 3));
#define DSA_MLA_NCHUNK(g_) ((g_) < 4 ? 6 : 3)
#define DSA_MLA_HAS(g_, u_) (pt + kProducers * (u_) < ((g_) < 4 ? 512 : 256))
#define DSA_MLA_LOAD(i_, g_)                                                   \
    _Pragma("unroll") for (int u = 0; u < DSA_MLA_NCHUNK(g_); ++u) {            \
        if (!DSA_MLA_HAS(g_, u)) continue;                                      \
        DSA_MLA_CHUNK(g_, u, r, c)                                              \
        const int row = sRow[(i_) * kTileKeys + r];                             \
        raw[g_][u] = (row >= 0) ? __ldg(reinterpret_cast<const uint4*>(          \
                                            p.latent_pages + (int64_t)row * kLatDim) + c) \
                                : make_uint4(0u, 0u, 0u, 0u);                   \
    }
#define DSA_NV_HAS(u_) (pt + kProducers * (u_) < 256)
#define DSA_NV_LOAD(i_, g_)                                                    \
    _Pragma("unroll") for (int u = 0; u < 3; ++u) {                             \
        if (!DSA_NV_HAS(u)) continue;                                           \
        const int q = ptv + kProducers * u, r = q >> 2, h = q & 3;              \
        const int row = sRow[(i_) * kTileKeys + r];                             \
        const uint8_t* src = p.latent_pages + (int64_t)(row >= 0 ? row : 0) * kNvRowBytes; \
        if ((g_) < 4) {                                                         \
            raw[g_][u] = (row >= 0) ? __ldg(reinterpret_cast<const uint4*>(src + 64 * (g_) + 16 * h)) \
                                    : make_uint4(0u, 0u, 0u, 0u);               \
            rsc[(g_) & 3][u] = (row >= 0) ? (uint32_t)__ldg(reinterpret_cast<const unsigned short*>( \
                                                src + kNvScaleOff + 8 * (g_) + 2 * h)) : 0u; \
        } else {                                                                \
            raw[g_][u] = (row >= 0) ? __ldg(reinterpret_cast<const uint4*>(src + kNvTailOff + 16 * h)) \
                                    : make_uint4(0u, 0u, 0u, 0u);               \
        }                                                                       \
    }
#define DSA_NV_STORE(g_)                                                       \
    _Pragma("unroll") for (int u = 0; u < 3; ++u) {                             \
        if (!DSA_NV_HAS(u)) continue;                                           \
        const int q = ptv + kProducers * u, r = q >> 2, h = q & 3;              \
        if ((g_) < 4) {                                                         \
            const __half2_raw sc = __nv_cvt_fp8x2_to_halfraw2(                  \
                (__nv_fp8x2_storage_t)(rsc[(g_) & 3][u] & 0xFFFFu), __NV_E4M3);   \
            const uint32_t s_lo = (uint32_t)sc.x | ((uint32_t)sc.x << 16);      \
            const uint32_t s_hi = (uint32_t)sc.y | ((uint32_t)sc.y << 16);      \
            uint8_t* base = sL + (2 * (g_) + (h >> 1)) * kLSlabBytes;           \
            const uint32_t wv[4] = {raw[g_][u].x, raw[g_][u].y, raw[g_][u].z, raw[g_][u].w}; \
            _Pragma("unroll") for (int j = 0; j < 4; ++j) {                     \
                const uint4 f = e2m1x8_to_f16x8(wv[j]);                         \
                const uint32_t sj = (j < 2) ? s_lo : s_hi;                       \
                *reinterpret_cast<uint4*>(base + sw128(r, (h & 1) * 64 + 16 * j)) = \
                    make_uint4(hmul2_u32(f.x, sj), hmul2_u32(f.y, sj), hmul2_u32(f.z, sj), \
                               hmul2_u32(f.w, sj));                              \
            }                                                                   \
        } else {                                                                \
            uint32_t h0[4], h1[4];                                              \
            e4m3x8_to_f16x8(raw[g_][u].x, raw[g_][u].y, h0);                    \
            e4m3x8_to_f16x8(raw[g_][u].z, raw[g_][u].w, h1);                    \
            uint8_t* base = sL + 8 * kLSlabBytes;                               \
            *reinterpret_cast<uint4*>(base + sw128(r, h * 32)) =                \
                make_uint4(h0[0], h0[1], h0[2], h0[3]);                         \
            *reinterpret_cast<uint4*>(base + sw128(r, h * 32 + 16)) =           \
                make_uint4(h1[0], h1[1], h1[2], h1[3]);                         \
        }                                                                       \
    }
#define DSA_MLA_STORE(g_)                                                      \
    _Pragma("unroll") for (int u = 0; u < DSA_MLA_NCHUNK(g_); ++u) {            \
        if (!DSA_MLA_HAS(g_, u)) continue;                                      \
        DSA_MLA_CHUNK(g_, u, r, c)                                              \
        uint32_t h0[4], h1[4];                                                  \
        e4m3x8_to_f16x8(raw[g_][u].x, raw[g_][u].y, h0);                        \
        e4m3x8_to_f16x8(raw[g_][u].z, raw[g_][u].w, h1);                        \
        uint8_t* base = sL + (c >> 2) * kLSlabBytes;                            \
        *reinterpret_cast<uint4*>(base + sw128(r, (c & 3) * 32)) =              \
            make_uint4(h0[0], h0[1], h0[2], h0[3]);                             \
        *reinterpret_cast<uint4*>(base + sw128(r, (c & 3) * 32 + 16)) =         \
            make_uint4(h1[0], h1[1], h1[2], h1[3]);                             \
    }
        if (n_used > 0) {
            const int ptv = pt;
#pragma unroll
            for (int g = 0; g < kGroups; ++g) {
                if constexpr (kLat == 0) { DSA_MLA_LOAD(0, g) }
                else { DSA_NV_LOAD(0, g) }
            }
        }
        bool ok = true;
        for (int i = 0; i < n_used && ok; ++i) {
            // index arithmetic is redone every tile rather than kept live
            int ptv = pt;
            asm volatile("" : "+r"(ptv));
            // group 4 (latent dims 512-575) is freed first: S alone reads it
#pragma unroll
            for (int gi = 0; gi < kGroups; ++gi) {
                const int g = (gi == 0) ? 4 : gi - 1;
                if (i > 0 && !mbar_wait<kBudget>(&bars->lempty[g], (i - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                if constexpr (kLat == 0) { DSA_MLA_STORE(g) }
                else { DSA_NV_STORE(g) }
                fence_proxy_async_smem();
                if (!(kWaitTest && i == 0 && g == 4)) mbar_arrive(&bars->lfull[g]);
                if (i + 1 < n_used) {
                    if constexpr (kLat == 0) { DSA_MLA_LOAD(i + 1, g) }
                    else { DSA_NV_LOAD(i + 1, g) }
                }
            }
        }
#undef DSA_MLA_CHUNK
#undef DSA_MLA_NCHUNK
#undef DSA_MLA_HAS
#undef DSA_MLA_LOAD
#undef DSA_MLA_STORE
#undef DSA_NV_HAS
#undef DSA_NV_LOAD
#undef DSA_NV_STORE
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issue (one thread) ----------------
        // descriptors are built once; operand offsets are added in 16-byte
        // units (the start-address field cannot carry: shared addresses are
        // below 256 KB)
        if (lane == 0) {
            const uint64_t qd = smem_desc(smem_u32(sQ), 16, 1024, kSwizzle128B);
            const uint64_t ld = smem_desc(smem_u32(sL), 16, 1024, kSwizzle128B);
            const uint64_t vd = smem_desc(smem_u32(sL), kLSlabBytes, 1024, kSwizzle128B);
            const uint64_t pd = smem_desc(smem_u32(sP), 16, 1024, kSwizzle128B);
            bool ok = true;
            for (int i = 0; i < n_used && ok; ++i) {
                // S = Q . L^T, slab group by slab group in the order the
                // producers refill them: group 4 (dims 512-575, free once the
                // previous S completed) first, then groups 0-3 as the previous
                // O^T update releases them
#pragma unroll
                for (int gi = 0; gi < kGroups; ++gi) {
                    const int g = (gi == 0) ? 4 : gi - 1;
                    if (!mbar_wait<kBudget>(&bars->lfull[g], i & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int s = 2 * g; s < 2 * g + (g < 4 ? 2 : 1); ++s)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_f16(tmem + kColS,
                                    qd + (uint64_t)((s * kQSlabBytes + kk * 32) >> 4),
                                    ld + (uint64_t)((s * kLSlabBytes + kk * 32) >> 4), kIdescQK,
                                    (gi > 0 || kk > 0) ? 1u : 0u);
                }
                if (!ok) break;
                mma_commit(&bars->lempty[4]);
                mma_commit(&bars->sfull);
                // O^T += V^T . P^T once the softmax has written P
                if (!mbar_wait<kBudget>(&bars->pfull, i & 1, abort_flag)) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16(tmem + kColO + 96 * c,
                                vd + (uint64_t)((2 * c * kLSlabBytes + ks * 2048) >> 4),
                                pd + (uint64_t)((ks * 32) >> 4), kIdescPV,
                                (i > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(&bars->lempty[c]);
                }
            }
            // TMEM is released only after every MMA issued here has completed,
            // also after an abort
            mma_commit(&bars->done);
            mbar_drain<kBudget>(&bars->done, 0);
        }
        __syncwarp();
    } else {
        // ---------------- softmax (thread = head) ----------------
        const int h = tid;  // 0..127; rows 96..127 (warp 3) are padding
        float m_ref = -INFINITY, l = 0.f;
        for (int i = 0; i < n_used; ++i) {
            if (!mbar_wait<kBudget>(&bars->sfull, i & 1, abort_flag)) break;
            tc_fence_after();
            // S(i) is complete and so is every earlier O^T update; nothing
            // touches O^T again before this thread arrives on pfull
            float factor = 1.f;
            bool resc = false;
            if (warp < 3) {
                uint32_t r[64];
                tmem_ld32(tmem_addr(tmem, 32 * warp, kColS), *reinterpret_cast<uint32_t(*)[32]>(r));
                tmem_ld32(tmem_addr(tmem, 32 * warp, kColS + 32),
                          *reinterpret_cast<uint32_t(*)[32]>(r + 32));
                tmem_wait_ld();
                const uint64_t mask = sMask[i];
                if (mask != ~0ull) {
                    // empty slots score -inf
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        if (!((mask >> j) & 1u)) r[j] = __float_as_uint(-INFINITY);
                }
                // the maximum of the raw accumulators (zscale > 0 keeps the order)
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int j = 0; j < 64; j += 2)
                    mx[(j >> 1) & 3] = max3f(mx[(j >> 1) & 3], __uint_as_float(r[j]), __uint_as_float(r[j + 1]));
                const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * zscale;
                if (mt > -INFINITY && (m_ref == -INFINITY || mt > m_ref + kRescaleLog2)) {
                    factor = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - mt);
                    m_ref = mt;
                    resc = (i > 0);
                }
                // P(i) -> its shared-memory row (the buffer's last reader, the
                // previous O^T update, has completed).  p = 2^(z - m_ref) with
                // z = s * zscale; an empty slot gives 2^-inf = 0, and while
                // m_ref is -inf every slot so far was empty.
                const float nm = (m_ref == -INFINITY) ? 0.f : -m_ref;
                const bool none = (m_ref == -INFINITY);
                // two scores at a time: the exponent z - m_ref in fp32, rounded
                // to an f16 pair, raised by one f16x2 2^x (P is stored in f16
                // either way); the row sum adds the same f16 values in fp32,
                // in four chains
                const uint64_t zs2 = pack_f32x2(zscale, zscale), nm2 = pack_f32x2(nm, nm);
                float ps[4] = {0.f, 0.f, 0.f, 0.f};
                if (none) {
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(sP + sw128(h, 16 * c)) = make_uint4(0u, 0u, 0u, 0u);
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint32_t ph[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int j = 8 * c + 2 * k;
                            const uint64_t a2 = fma_f32x2(
                                pack_f32x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), zs2, nm2);
                            const uint32_t e2 = ex2_f16x2(f32x2_to_f16x2(a2));
                            ph[k] = e2;
                            add_f16x2_to_f32(e2, ps[2 * (k & 1)], ps[2 * (k & 1) + 1]);
                        }
                        *reinterpret_cast<uint4*>(sP + sw128(h, 16 * c)) =
                            make_uint4(ph[0], ph[1], ph[2], ph[3]);
                    }
                }
                l = l * factor + ((ps[0] + ps[2]) + (ps[1] + ps[3]));
            }
            sF[h] = resc ? factor : 1.f;
            if (softmax_any(resc)) {
                // every warp rescales the O^T lanes (latent dims) it may access
                for (int hg = 0; hg < 3; ++hg) {
                    float fac[32];
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float4 v4 = *reinterpret_cast<const float4*>(sF + 32 * hg + j);
                        fac[j] = v4.x; fac[j + 1] = v4.y; fac[j + 2] = v4.z; fac[j + 3] = v4.w;
                    }
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t a = tmem_addr(tmem, 32 * warp, kColO + 96 * c + 32 * hg);
                        uint32_t o[32];
                        tmem_ld32(a, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            o[j] = __float_as_uint(__uint_as_float(o[j]) * fac[j]);
                        tmem_st32(a, o);
                    }
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars->pfull);
        }
        // ---------------- end of softmax: per-head normaliser ----------------
        const bool ok = mbar_wait<kBudget>(&bars->done, 0, abort_flag);
        tc_fence_after();
        const float scale_out = whole ? p.kv_scale : 1.f;
        sF[256 + h] = (l > 0.f) ? scale_out / l : 0.f;
        if (ok && ok_tok && h < kQRows) {
            const float lse2 = (l > 0.f) ? m_ref + log2f(l) : -INFINITY;
            if (whole) {
                if (p.lse) p.lse[(int64_t)t * kMlaHeads + h] = lse2 * 0.6931471805599453f;
            } else {
                p.part_lse[piece * kMlaHeads + h] = lse2;
            }
        }
    }

    // ---------------- epilogue: O^T / l -> bf16 output or f16 partial ----------
    // warps 0-3 take latent-dim tiles 0-1, warps 4-7 tiles 2-3 (a warp reads
    // TMEM lanes 32*(warp%4)..+31); thread = one latent dim, 96 heads.  The
    // result is staged in the (now unused) query buffer and leaves with one
    // bulk copy: a final result as [96][512] bf16, a split partial dim-major
    // as [512][96] f16, row d's twelve 16-byte chunks (heads 8q..8q+7) stored
    // at chunk (q + d) mod 12 so that a warp's stores of 32 rows spread over
    // the banks; the combine reads them there.  (Stored from registers, the
    // 192-byte-strided pieces cost a transaction each: about 3 us per CTA.)
    {
        __syncthreads();  // the softmax warps have seen `done` and written 1/l
        tc_fence_after();
        const bool write = !*abort_flag && ok_tok;
        const int lq = warp & 3;
        const int mt0 = (warp < 4) ? 0 : 2;
        if (write) {
            for (int mt = mt0; mt < mt0 + 2; ++mt) {
                const int d = 128 * mt + 32 * lq + lane;
                uint32_t o[96];
#pragma unroll
                for (int hg = 0; hg < 3; ++hg)
                    tmem_ld32(tmem_addr(tmem, 32 * lq, kColO + 96 * mt + 32 * hg),
                              *reinterpret_cast<uint32_t(*)[32]>(o + 32 * hg));
                tmem_wait_ld();
                // the per-head scales go to registers first: a shared load
                // between the (possibly aliasing) stores would serialise them
                if (whole) {
                    __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(sQ) + d;
#pragma unroll
                    for (int hg = 0; hg < 3; ++hg) {
                        float inv[32];
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            const float4 v4 = *reinterpret_cast<const float4*>(sF + 256 + 32 * hg + j);
                            inv[j] = v4.x; inv[j + 1] = v4.y; inv[j + 2] = v4.z; inv[j + 3] = v4.w;
                        }
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            st[(32 * hg + j) * kVDim] =
                                __float2bfloat16_rn(__uint_as_float(o[32 * hg + j]) * inv[j]);
                    }
                } else {
                    uint4* srow = reinterpret_cast<uint4*>(sQ) + 12 * d;
                    const int rot = d % 12;
                    float inv[96];  // the per-head scales, loaded before the stores
#pragma unroll
                    for (int j = 0; j < 96; j += 4) {
                        const float4 v4 = *reinterpret_cast<const float4*>(sF + 256 + j);
                        inv[j] = v4.x; inv[j + 1] = v4.y; inv[j + 2] = v4.z; inv[j + 3] = v4.w;
                    }
#pragma unroll
                    for (int q = 0; q < 12; ++q) {  // heads 8q .. 8q+7
                        const float* ov = reinterpret_cast<const float*>(o + 8 * q);
                        const float* iv = inv + 8 * q;
                        const int c = (q + rot >= 12) ? q + rot - 12 : q + rot;
                        srow[c] = make_uint4(pack_half2(ov[0] * iv[0], ov[1] * iv[1]),
                                             pack_half2(ov[2] * iv[2], ov[3] * iv[3]),
                                             pack_half2(ov[4] * iv[4], ov[5] * iv[5]),
                                             pack_half2(ov[6] * iv[6], ov[7] * iv[7]));
                    }
                }
            }
            fence_proxy_async_smem();  // the bulk copy reads the staged result
        }
        __syncthreads();
        if (write && tid == 0) {
            if (whole)
                bulk_store_s2g(p.out + (int64_t)t * kMlaHeads * kVDim, sQ, (uint32_t)kOutBytes);
            else
                bulk_store_s2g(p.part_o + piece * kVDim * kMlaHeads, sQ, (uint32_t)kOutBytes);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && tid == 0) record_error(p.status, DSA_ERR_TIMEOUT);
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// Merge the split partials of one token over 32 latent dims: out = kv_scale *
// sum_s 2^(lse_s - L) o_s with L = log2 sum_s 2^lse_s per head, in a fixed
// order over the splits.  The partials are dim-major ([512][96] f16 per
// split); thread = (latent dim, 8 heads): one 16-byte vector per split, all
// of them in flight at once.
constexpr int kCombineDims = 32;
constexpr int kMaxSplits = 16;
constexpr int kCombineThreads = kCombineDims * (kMlaHeads / 8);  // 384
__global__ void __launch_bounds__(kCombineThreads)
sparse_mla_combine_kernel(const __half* __restrict__ part_o, const float* __restrict__ part_lse,
                          int first_token, int splits, float kv_scale,
                          __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
    constexpr int kBlocksPerToken = kVDim / kCombineDims;  // 16
    __shared__ float s_w[kMaxSplits][kMlaHeads];
    __shared__ float s_inv[kMlaHeads];
    grid_dependents_launch();  // the next step's first kernel may start its setup
    grid_dependency_wait();  // the partials come from the previous kernel
    const int u = blockIdx.x / kBlocksPerToken;  // the u-th split token
    const int t = first_token + u;
    const int dblk = blockIdx.x % kBlocksPerToken;
    const int tid = threadIdx.x;
    const int d = dblk * kCombineDims + (tid & (kCombineDims - 1));
    const int h0 = 8 * (tid / kCombineDims);  // 0, 8, ..., 88
    const int chunk = (h0 / 8 + d) % 12;      // where the partial's row d keeps heads h0..h0+7
    uint4 v[kMaxSplits];
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s)
        v[s] = (s < splits) ? __ldg(reinterpret_cast<const uint4*>(
                                  part_o + (((int64_t)u * splits + s) * kVDim + d) * kMlaHeads + 8 * chunk))
                            : make_uint4(0u, 0u, 0u, 0u);
    if (tid < kMlaHeads) {
        const int h = tid;
        float ls[kMaxSplits];
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s)
            ls[s] = (s < splits) ? part_lse[((int64_t)u * splits + s) * kMlaHeads + h] : -INFINITY;
        float M = -INFINITY;
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s) M = fmaxf(M, ls[s]);
        float tot = 0.f;
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s) {
            if (s >= splits) break;
            const float wgt = (M == -INFINITY) ? 0.f : exp2f(ls[s] - M);
            s_w[s][h] = wgt;
            tot += wgt;
        }
        s_inv[h] = (tot > 0.f) ? kv_scale / tot : 0.f;
        if (dblk == 0 && lse)
            lse[(int64_t)t * kMlaHeads + h] =
                (tot > 0.f) ? (M + log2f(tot)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) {
        if (s >= splits) break;
        const uint32_t wv[4] = {v[s].x, v[s].y, v[s].z, v[s].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv[k]));
            acc[2 * k] = fmaf(s_w[s][h0 + 2 * k], f.x, acc[2 * k]);
            acc[2 * k + 1] = fmaf(s_w[s][h0 + 2 * k + 1], f.y, acc[2 * k + 1]);
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
        out[((int64_t)t * kMlaHeads + h0 + j) * kVDim + d] = __float2bfloat16_rn(acc[j] * s_inv[h0 + j]);
}

}  // namespace

// The wave of CTAs the plan fills: one CTA per SM (the kernel's shared memory
// admits one).  A fixed count, not the device's, so that the plan -- and with
// it every token's result -- depends on the batch alone.
constexpr int kWaveCtas = 152;

// How a batch of T tokens runs: whole waves of one CTA per token, then the
// remaining r tokens split into P pieces each, P the largest power of two
// with r P <= kWaveCtas (at most 16, and dividing the slots into whole tiles).
// For T < kWaveCtas this gives 16 splits up to 9 tokens, then 8, 4, 2, 1.
// The batch-invariant plan (whole_only) runs every token as one CTA.
struct MlaPlan {
    int full_tokens, tail_splits;
};

MlaPlan mla_plan(int total_q, int K, bool whole_only = false) {
    MlaPlan pl;
    const int r = total_q % kWaveCtas;
    int P = 1;
    while (!whole_only && r > 0 && 2 * P <= kMaxSplits && r * 2 * P <= kWaveCtas &&
           (K % (2 * P * kTileKeys)) == 0)
        P *= 2;
    pl.tail_splits = P;
    pl.full_tokens = (P > 1) ? total_q - r : total_q;
    return pl;
}

// Workspace: the f16 partial outputs [split tokens, P, 512, 96] and their lse
// [split tokens, P, 96], sized for the default plan (the batch-invariant plan
// needs none).
struct MlaWs {
    size_t part_o, part_lse, total;
};

MlaWs mla_ws_layout(int total_q, int K) {
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    const MlaPlan pl = mla_plan(total_q, K);
    const size_t pieces = (size_t)(total_q - pl.full_tokens) * pl.tail_splits;
    MlaWs w;
    w.part_o = 0;
    w.part_lse = up(pieces * kMlaHeads * kVDim * sizeof(__half));
    w.total = w.part_lse + up(pieces * kMlaHeads * sizeof(float));
    return w;
}

size_t sparse_mla_workspace_bytes(int total_q, int K) { return mla_ws_layout(total_q, K).total; }

// Kernels one sparse-MLA call launches: the MMA kernel and, when some tokens
// are split, the combine.
int sparse_mla_launches(int total_q, int K, bool whole_only) {
    const MlaPlan pl = mla_plan(total_q, K, whole_only);
    return pl.full_tokens < total_q ? 2 : 1;
}

cudaError_t launch_sparse_mla(const BatchArgs& bt, const uint16_t* q_lat, const void* latent_pages,
                              float kv_scale, float sm_scale, const int32_t* indices, int K,
                              uint16_t* out, float* lse, void* ws, int32_t* status, bool pdl,
                              cudaStream_t stream, bool wait_test, int latent_format,
                              bool whole_only) {
    if (bt.total_q == 0) return cudaSuccess;
    MlaParams p;
    p.bt = bt;
    const MlaWs w = mla_ws_layout(bt.total_q, K);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    p.q_lat = reinterpret_cast<const __nv_bfloat16*>(q_lat);
    p.latent_pages = static_cast<const uint8_t*>(latent_pages);
    p.indices = indices;
    p.K = K;
    const MlaPlan pl = mla_plan(bt.total_q, K, whole_only);
    p.full_tokens = pl.full_tokens;
    p.tail_splits = pl.tail_splits;
    const int split_tokens = bt.total_q - pl.full_tokens;
    p.kv_scale = kv_scale;
    p.sm_scale = sm_scale;
    p.out = reinterpret_cast<__nv_bfloat16*>(out);
    p.lse = lse;
    p.status = status;
    p.part_o = split_tokens > 0 ? reinterpret_cast<__half*>(wsb + w.part_o) : nullptr;
    p.part_lse = split_tokens > 0 ? reinterpret_cast<float*>(wsb + w.part_lse) : nullptr;
    auto kernel = latent_format == DSA_LATENT_NVFP4
                      ? sparse_mla_tc_kernel<false, DSA_LATENT_NVFP4>
                      : (wait_test ? sparse_mla_tc_kernel<true, DSA_LATENT_FP8_E4M3>
                                   : sparse_mla_tc_kernel<false, DSA_LATENT_FP8_E4M3>);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemAlloc);
    if (e != cudaSuccess) return e;
    e = launch_kernel(kernel, dim3(pl.full_tokens + split_tokens * pl.tail_splits), dim3(kThreads),
                      (size_t)kSmemAlloc, stream, pdl, 1, p);
    if (e != cudaSuccess || split_tokens == 0) return e;
    return launch_kernel(sparse_mla_combine_kernel, dim3(split_tokens * (kVDim / kCombineDims)),
                         dim3(kCombineThreads), 0, stream, true, 1, (const __half*)p.part_o,
                         (const float*)p.part_lse, pl.full_tokens, pl.tail_splits, kv_scale, p.out,
                         lse);
}

}  // namespace dsa
