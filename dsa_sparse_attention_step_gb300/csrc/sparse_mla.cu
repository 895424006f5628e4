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
// One CTA = one query token x one contiguous split of its index slots.
//   S   = Q . L^T    tcgen05 kind::f16, M = 128 (96 heads + 32 unused rows),
//                    N = 32 selected tokens, K = 576; accumulator in TMEM
//                    (double buffered, 2 x 32 columns)
//   O^T = V^T . P^T  M = 128 latent dims (4 tiles cover 512), N = 96 heads,
//                    K = 32 tokens; accumulator in TMEM (4 x 96 columns)
// Latents are gathered row by row with 16-byte loads from the paged cache and
// lifted E4M3 -> f16 exactly into a 128-byte-swizzled tile that serves both as
// the K-major B operand of S and as the MN-major A operand of O^T.  The bf16
// query is converted to f16 after a per-token power-of-two scale (exact for
// every element within 2^-14 of the largest).  Softmax runs online in the
// log2 domain with conditional rescaling: a head's reference maximum only
// moves when a new maximum exceeds it by more than 2^8, and the O^T columns
// are then rescaled in TMEM.
//
// Warp roles (256 threads, so a thread may hold up to 255 registers): warps
// 0-3 softmax (thread = head), warps 4-6 gather/convert producers, warp 7 TMEM
// allocation and the single MMA-issuing thread; all eight warps share the
// epilogue (thread = latent dim).  Every wait is bounded.
#include "common.cuh"
#include "sm100.cuh"

namespace dsa {

using namespace sm100;

namespace {

constexpr int kTileKeys = 32;
constexpr int kThreads = 256;
constexpr int kProducers = 96;                                // warps 4-6
constexpr int kVecPerProducer = kTileKeys * (kLatDim / 16) / kProducers;  // 12
constexpr int kQRows = 96;
constexpr int kSlabs = kLatDim / 64;                          // 9 K-slabs of 64 dims
constexpr int kQSlabBytes = kQRows * 128;                     // 12288
constexpr int kQBytes = kSlabs * kQSlabBytes;                 // 110592
constexpr int kPBytes = kQRows * 128;                         // 12288 per buffer
constexpr int kLSlabBytes = kTileKeys * 128;                  // 4096
constexpr int kLBytes = kSlabs * kLSlabBytes;                 // 36864 per stage
constexpr int kMaxSplitKeys = kTopK;                          // index slots per CTA, max
constexpr int kOffQ = 0;
// The M = 128 reads of a 96-row Q slab run 4 KB past it; for the last slab
// that lands in the P buffers (valid shared memory, unused accumulator rows).
constexpr int kOffP = kOffQ + kQBytes;
constexpr int kOffL = kOffP + 2 * kPBytes;
constexpr int kOffRow = kOffL + 2 * kLBytes;                  // int32 row ids
constexpr int kOffMask = kOffRow + kMaxSplitKeys * 4;         // valid-slot mask per tile
constexpr int kOffF = kOffMask + (kMaxSplitKeys / kTileKeys) * 4;  // per-head floats
constexpr int kOffBar = kOffF + 512 * 4;
constexpr int kSmemBytes = kOffBar + 256;
constexpr int kSmemAlloc = kSmemBytes + 1024;                 // slack for 1024-B alignment
static_assert(kSmemAlloc <= 227 * 1024, "shared memory budget");

// TMEM columns
constexpr uint32_t kColS = 0;     // two 32-column S buffers
constexpr uint32_t kColO = 64;    // four 96-column O^T tiles
constexpr uint32_t kTmemCols = 512;

constexpr float kRescaleLog2 = 8.0f;  // move the reference max when exceeded by > 2^8

constexpr uint32_t kIdescQK = make_idesc(kFmtF16, kFmtF16, 128, kTileKeys, false, false);
constexpr uint32_t kIdescPV = make_idesc(kFmtF16, kFmtF16, 128, kQRows, true, false);

struct Bars {
    uint64_t full[2];    // producer -> MMA: latent stage filled (96 arrivals)
    uint64_t empty[2];   // MMA -> producer: stage free (commit after PV)
    uint64_t sfull[2];   // MMA -> softmax: S buffer ready (commit after QK)
    uint64_t pfull[2];   // softmax -> MMA: P buffer written, S buffer read (128 arrivals)
    uint64_t pempty[2];  // MMA -> softmax: PV done with P buffer (commit)
    uint64_t done;       // MMA -> epilogue: everything finished
    uint64_t qbar;       // bulk copy of the prepared query landed
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Named barrier over the 128 softmax threads (warps 0-3).
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Same barrier, returning whether any of the 128 threads passed `pred`.
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

struct MlaParams {
    BatchArgs bt;
    const uint8_t* qf16;   // [T][110592] prepared query (f16, swizzled slabs)
    const int* qexp;       // [T] power-of-two exponent e of the query scale 2^-e
    const uint8_t* latent_pages;
    const int32_t* indices;
    int K;                 // index slots per token
    int splits;            // CTAs per token
    int split_keys;        // index slots per CTA (multiple of 32)
    float kv_scale;
    float sm_scale;
    __nv_bfloat16* out;    // final output (splits == 1)
    float* lse;            // final lse (splits == 1), nullable
    __half* part_o;        // [T, splits, 96, 512] normalised partial outputs (splits > 1)
    float* part_lse;       // [T, splits, 96] partial lse, log2 domain (splits > 1)
    int32_t* status;
};

__global__ void __launch_bounds__(kThreads, 1) sparse_mla_tc_kernel(const MlaParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = sm + kOffQ;
    uint8_t* sP = sm + kOffP;
    uint8_t* sL = sm + kOffL;
    int32_t* sRow = reinterpret_cast<int32_t*>(sm + kOffRow);
    uint32_t* sMask = reinterpret_cast<uint32_t*>(sm + kOffMask);
    // [0,256): rescale factors (two buffers of 128), [256,384): m, [384,512): l
    float* sF = reinterpret_cast<float*>(sm + kOffF);
    Bars* bars = reinterpret_cast<Bars*>(sm + kOffBar);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t = blockIdx.x / p.splits;
    const int split = blockIdx.x % p.splits;
    const int b = request_of(p.bt, t);
    const bool ok_tok = token_ok(p.bt, b, t, split == 0 ? p.status : nullptr);
    const int seq = __ldg(p.bt.seq_lens + b);
    const int n_tiles = p.split_keys / kTileKeys;
    const int slot0 = split * p.split_keys;
    volatile int* abort_flag = &bars->abort_flag;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->full[i], kProducers);
            mbar_init(&bars->empty[i], 1);
            mbar_init(&bars->sfull[i], 1);
            mbar_init(&bars->pfull[i], 128);
            mbar_init(&bars->pempty[i], 1);
        }
        mbar_init(&bars->done, 1);
        mbar_init(&bars->qbar, 1);
        bars->abort_flag = 0;
        fence_mbar_init();
        // the prepared query: one bulk copy into its shared-memory slabs
        if (ok_tok) {
            mbar_arrive_expect_tx(&bars->qbar, (uint32_t)kQBytes);
            bulk_copy_g2s(sQ, p.qf16 + (int64_t)t * kQBytes, (uint32_t)kQBytes, &bars->qbar);
        } else {
            mbar_arrive(&bars->qbar);
        }
    }
    if (warp == 7) {
        tmem_alloc(&bars->tmem_base, kTmemCols);
        tmem_relinquish();
    }

    // ---- preamble: row ids (page * 64 + slot) of this CTA's index slots -------
    for (int k = tid; k < p.split_keys; k += kThreads) {
        int row = -1;
        if (ok_tok) {
            const int s = __ldg(p.indices + (int64_t)t * p.K + slot0 + k);
            if (s >= seq) {
                record_error(p.status, DSA_ERR_DEVICE_CHECK);
            } else if (s >= 0) {
                const int pg = page_lookup(p.bt, b, s / kPage, p.status);
                if (pg >= 0) row = pg * kPage + (s % kPage);
            }
        }
        sRow[k] = row;
    }
    if (tid < 2 * 128) sF[tid] = 1.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const bool producer = (warp >= 4 && warp < 7);
    const int e = ok_tok ? __ldg(p.qexp + t) : 0;
    if (!producer) {
        // warps 0-3 and 7: valid-slot masks while the producers start gathering
        const int ctid = (warp == 7) ? 128 + lane : tid;  // 0..159
        for (int i = ctid; i < n_tiles; i += 160) {
            uint32_t m = 0;
            for (int j = 0; j < kTileKeys; ++j) m |= (sRow[i * kTileKeys + j] >= 0 ? 1u : 0u) << j;
            sMask[i] = m;
        }
        asm volatile("bar.sync 2, 160;" ::: "memory");
    }
    const uint32_t tmem = bars->tmem_base;
    // z in log2 units per unit of the f16 accumulator
    const float zscale = p.sm_scale * p.kv_scale * ldexpf(1.0f, e) * 1.4426950408889634f;

    if (producer) {
        // ---------------- producers: gather + E4M3 -> f16 ----------------
        // 32 rows x 36 vectors of 16 bytes = 1152 vectors -> 12 per thread per
        // tile; two tiles of loads are kept in flight (registers A and B)
        const int ptid = tid - 128;
        uint4 rawA[kVecPerProducer], rawB[kVecPerProducer];
#define DSA_MLA_LOAD(raw_, i_)                                                           \
    _Pragma("unroll") for (int u = 0; u < kVecPerProducer; ++u) {                        \
        const int v = ptid + kProducers * u;                                              \
        const int r = v / 36, c = v % 36;                                                 \
        const int row = sRow[(i_) * kTileKeys + r];                                       \
        raw_[u] = (row >= 0) ? __ldg(reinterpret_cast<const uint4*>(                      \
                                         p.latent_pages + (int64_t)row * kLatDim) + c)    \
                             : make_uint4(0, 0, 0, 0);                                    \
    }
#define DSA_MLA_STORE(raw_, st_)                                                         \
    _Pragma("unroll") for (int u = 0; u < kVecPerProducer; ++u) {                        \
        const int v = ptid + kProducers * u;                                              \
        const int r = v / 36, c = v % 36;                                                 \
        const uint32_t wv[4] = {raw_[u].x, raw_[u].y, raw_[u].z, raw_[u].w};              \
        uint32_t hv[8];                                                                   \
        _Pragma("unroll") for (int k = 0; k < 4; ++k) {                                   \
            __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(                                  \
                (__nv_fp8x2_storage_t)(wv[k] & 0xFFFF), __NV_E4M3);                       \
            __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(                                  \
                (__nv_fp8x2_storage_t)(wv[k] >> 16), __NV_E4M3);                          \
            hv[2 * k] = *reinterpret_cast<uint32_t*>(&lo);                                \
            hv[2 * k + 1] = *reinterpret_cast<uint32_t*>(&hi);                            \
        }                                                                                 \
        uint8_t* base = sL + (st_) * kLBytes + (c / 4) * kLSlabBytes;                     \
        *reinterpret_cast<uint4*>(base + sw128(r, (c % 4) * 32)) =                        \
            make_uint4(hv[0], hv[1], hv[2], hv[3]);                                       \
        *reinterpret_cast<uint4*>(base + sw128(r, (c % 4) * 32 + 16)) =                   \
            make_uint4(hv[4], hv[5], hv[6], hv[7]);                                       \
    }
        if (n_tiles > 0) { DSA_MLA_LOAD(rawA, 0) }
        if (n_tiles > 1) { DSA_MLA_LOAD(rawB, 1) }
        for (int i = 0; i < n_tiles; i += 2) {
            if (i >= 2 && !mbar_wait(&bars->empty[0], ((i - 2) >> 1) & 1, abort_flag)) break;
            DSA_MLA_STORE(rawA, 0)
            fence_proxy_async_smem();
            mbar_arrive(&bars->full[0]);
            if (i + 2 < n_tiles) { DSA_MLA_LOAD(rawA, i + 2) }
            if (i + 1 >= n_tiles) break;
            if (i + 1 >= 2 && !mbar_wait(&bars->empty[1], ((i - 1) >> 1) & 1, abort_flag)) break;
            DSA_MLA_STORE(rawB, 1)
            fence_proxy_async_smem();
            mbar_arrive(&bars->full[1]);
            if (i + 3 < n_tiles) { DSA_MLA_LOAD(rawB, i + 3) }
        }
#undef DSA_MLA_LOAD
#undef DSA_MLA_STORE
    } else if (warp == 7) {
        // ---------------- MMA issue (one thread) ----------------
        if (lane == 0) {
            const uint32_t qa = smem_u32(sQ), pa = smem_u32(sP), la = smem_u32(sL);
            auto issue_pv = [&](int i) -> bool {
                const int st = i & 1;
                if (!mbar_wait(&bars->pfull[st], (i >> 1) & 1, abort_flag)) return false;
                tc_fence_after();
#pragma unroll
                for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        const uint64_t ad = smem_desc(
                            la + st * kLBytes + (2 * mt) * kLSlabBytes + ks * 2048, kLSlabBytes,
                            1024, kSwizzle128B);
                        const uint64_t bd =
                            smem_desc(pa + st * kPBytes + ks * 32, 16, 1024, kSwizzle128B);
                        mma_f16(tmem + kColO + 96 * mt, ad, bd, kIdescPV,
                                (i > 0 || ks > 0) ? 1u : 0u);
                    }
                mma_commit(&bars->empty[st]);
                mma_commit(&bars->pempty[st]);
                return true;
            };
            bool ok = mbar_wait(&bars->qbar, 0, abort_flag);
            for (int i = 0; i < n_tiles && ok; ++i) {
                const int st = i & 1;
                ok = mbar_wait(&bars->full[st], (i >> 1) & 1, abort_flag);
                if (ok && i >= 2)
                    ok = mbar_wait(&bars->pfull[st], ((i - 2) >> 1) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                for (int j = 0; j < kSlabs; ++j)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad =
                            smem_desc(qa + j * kQSlabBytes + kk * 32, 16, 1024, kSwizzle128B);
                        const uint64_t bd = smem_desc(la + st * kLBytes + j * kLSlabBytes + kk * 32,
                                                      16, 1024, kSwizzle128B);
                        mma_f16(tmem + kColS + 32 * st, ad, bd, kIdescQK, (j | kk) ? 1u : 0u);
                    }
                mma_commit(&bars->sfull[st]);
                if (i >= 1) ok = issue_pv(i - 1);
            }
            if (ok && n_tiles > 0) issue_pv(n_tiles - 1);
            mma_commit(&bars->done);  // also drains whatever is in flight after an abort
        }
        __syncwarp();
    } else {
        // ---------------- softmax (thread = head) ----------------
        const int h = tid;  // 0..127; rows 96..127 are padding
        const bool real = h < kQRows;
        float m_ref = -INFINITY, l = 0.f;
        for (int i = 0; i < n_tiles; ++i) {
            const int st = i & 1;
            if (!mbar_wait(&bars->sfull[st], (i >> 1) & 1, abort_flag)) break;
            tc_fence_after();
            uint32_t r[32];
            tmem_ld32(tmem_addr(tmem, 32 * warp, kColS + 32 * st), r);
            tmem_wait_ld();
            const uint32_t mask = sMask[i];
            float z[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
                z[j] = ((mask >> j) & 1u) ? __uint_as_float(r[j]) * zscale : -INFINITY;
            // pairwise trees keep the dependency chains short
            float mx[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) mx[j] = fmaxf(z[2 * j], z[2 * j + 1]);
#pragma unroll
            for (int w2 = 8; w2 >= 1; w2 >>= 1)
#pragma unroll
                for (int j = 0; j < w2; ++j) mx[j] = fmaxf(mx[j], mx[j + w2]);
            const float mt = mx[0];
            float factor = 1.f;
            bool resc = false;
            if (real && mt > -INFINITY && (m_ref == -INFINITY || mt > m_ref + kRescaleLog2)) {
                factor = (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - mt);
                m_ref = mt;
                resc = (i > 0);
            }
            uint32_t ph[16];
            float ps[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float p0 = ((mask >> (2 * j)) & 1u) ? exp2f(z[2 * j] - m_ref) : 0.f;
                const float p1 = ((mask >> (2 * j + 1)) & 1u) ? exp2f(z[2 * j + 1] - m_ref) : 0.f;
                ps[j] = p0 + p1;
                ph[j] = pack_half2(p0, p1);
            }
#pragma unroll
            for (int w2 = 8; w2 >= 1; w2 >>= 1)
#pragma unroll
                for (int j = 0; j < w2; ++j) ps[j] += ps[j + w2];
            const float psum = ps[0];
            l = l * factor + psum;
            float* fac = sF + 128 * (i & 1);
            fac[h] = resc ? factor : 1.f;
            const bool any = softmax_any(resc);
            // P buffer st was last read by PV(i-2); O^T is complete up to PV(i-1)
            if (i >= 2 && !mbar_wait(&bars->pempty[st], ((i - 2) >> 1) & 1, abort_flag)) break;
            if (any) {
                if (!mbar_wait(&bars->pempty[(i - 1) & 1], ((i - 1) >> 1) & 1, abort_flag)) break;
                tc_fence_after();
                for (int mtile = 0; mtile < 4; ++mtile)
                    for (int c = 0; c < 3; ++c) {
                        const uint32_t a = tmem_addr(tmem, 32 * warp, kColO + 96 * mtile + 32 * c);
                        uint32_t o[32];
                        tmem_ld32(a, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            o[j] = __float_as_uint(__uint_as_float(o[j]) * fac[32 * c + j]);
                        tmem_st32(a, o);
                    }
                tmem_wait_st();
            }
            if (real) {
                uint8_t* row = sP + st * kPBytes;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4*>(row + sw128(h, 16 * c)) =
                        make_uint4(ph[4 * c], ph[4 * c + 1], ph[4 * c + 2], ph[4 * c + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars->pfull[st]);
        }
        // ---------------- end of softmax: per-head normaliser ----------------
        const bool ok = mbar_wait(&bars->done, 0, abort_flag);
        tc_fence_after();
        const float scale_out = (p.splits == 1) ? p.kv_scale : 1.f;
        sF[256 + h] = (l > 0.f) ? scale_out / l : 0.f;
        if (ok && ok_tok && real) {
            const float lse2 = (l > 0.f) ? m_ref + log2f(l) : -INFINITY;
            if (p.splits == 1) {
                if (p.lse) p.lse[(int64_t)t * kMlaHeads + h] = lse2 * 0.6931471805599453f;
            } else {
                p.part_lse[((int64_t)t * p.splits + split) * kMlaHeads + h] = lse2;
            }
        }
        tc_fence_before();
    }

    // ---------------- epilogue: O^T / l -> bf16 output or f16 partial ----------
    // warps 0-3 take latent-dim tiles 0-1, warps 4-7 tiles 2-3 (a warp reads
    // TMEM lanes 32*(warp%4)..+31); thread = one latent dim, 96 heads
    if (warp < 8) {
        asm volatile("bar.sync 3, 256;" ::: "memory");
        tc_fence_after();
        if (!*abort_flag && ok_tok) {
            const int lq = warp & 3;
            const int mt0 = (warp < 4) ? 0 : 2;
            for (int c = 0; c < 3; ++c) {
                float inv[32];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 v4 = *reinterpret_cast<const float4*>(sF + 256 + 32 * c + j);
                    inv[j] = v4.x; inv[j + 1] = v4.y; inv[j + 2] = v4.z; inv[j + 3] = v4.w;
                }
                for (int mt = mt0; mt < mt0 + 2; ++mt) {
                    const int d = 128 * mt + 32 * lq + lane;
                    uint32_t o[32];
                    tmem_ld32(tmem_addr(tmem, 32 * lq, kColO + 96 * mt + 32 * c), o);
                    tmem_wait_ld();
                    if (p.splits == 1) {
                        __nv_bfloat16* dst = p.out + ((int64_t)t * kMlaHeads + 32 * c) * kVDim + d;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            dst[(int64_t)j * kVDim] = __float2bfloat16_rn(__uint_as_float(o[j]) * inv[j]);
                    } else {
                        __half* dst = p.part_o +
                                      (((int64_t)t * p.splits + split) * kMlaHeads + 32 * c) * kVDim + d;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            dst[(int64_t)j * kVDim] = __float2half_rn(__uint_as_float(o[j]) * inv[j]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && tid == 0) record_error(p.status, DSA_ERR_TIMEOUT);
    if (warp == 7) tmem_dealloc(tmem, kTmemCols);
}

// Prepare each token's query once: bf16 -> f16 with a power-of-two scale 2^-e
// (e = 0 unless max|q| >= 2^15 or < 2^-8; then max|q| * 2^-e lies in
// [2^14, 2^15)), written in the 128-byte-swizzled slab layout the MMA reads,
// so every CTA of the token loads it with one bulk copy.
__global__ void __launch_bounds__(256)
sparse_mla_prep_q_kernel(const __nv_bfloat16* __restrict__ q_lat, uint8_t* __restrict__ qf16,
                         int* __restrict__ qexp) {
    constexpr int kVec = kMlaHeads * kLatDim / 8 / 256;  // 27 vectors of 8 per thread
    __shared__ float s_max[8];
    const int t = blockIdx.x, tid = threadIdx.x;
    const uint4* src = reinterpret_cast<const uint4*>(q_lat + (int64_t)t * kMlaHeads * kLatDim);
    uint4 raw[kVec];
    float amax = 0.f;
#pragma unroll
    for (int u = 0; u < kVec; ++u) {
        raw[u] = __ldg(src + tid + 256 * u);
        const uint32_t wv[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(wv[i] << 16)),
                                     fabsf(__uint_as_float(wv[i] & 0xFFFF0000u))));
    }
    amax = warp_max(amax);
    if ((tid & 31) == 0) s_max[tid >> 5] = amax;
    __syncthreads();
    float qmax = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) qmax = fmaxf(qmax, s_max[w]);
    int e = 0;
    if (qmax > 0.f && (qmax >= 32768.f || qmax < 0.00390625f)) {
        int ex;
        frexpf(qmax, &ex);  // qmax = f * 2^ex, f in [0.5, 1)
        e = ex - 15;
    }
    const float qmul = ldexpf(1.0f, -e);
    uint8_t* dst = qf16 + (int64_t)t * kQBytes;
#pragma unroll
    for (int u = 0; u < kVec; ++u) {
        const int v = tid + 256 * u;
        const int h = v / (kLatDim / 8), c = v % (kLatDim / 8);
        const uint32_t wv[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = pack_half2(__uint_as_float(wv[i] << 16) * qmul,
                              __uint_as_float(wv[i] & 0xFFFF0000u) * qmul);
        *reinterpret_cast<uint4*>(dst + (c / 8) * kQSlabBytes + sw128(h, (c % 8) * 16)) =
            make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (tid == 0) qexp[t] = e;
}

// Merge the split partials: out = sum_s 2^(lse_s - L) o_s with
// L = log2 sum_s 2^lse_s, in a fixed order over the splits.
__global__ void __launch_bounds__(128)
sparse_mla_combine_kernel(const __half* __restrict__ part_o, const float* __restrict__ part_lse,
                          int splits, float kv_scale, __nv_bfloat16* __restrict__ out,
                          float* __restrict__ lse) {
    const int t = blockIdx.x / kMlaHeads, h = blockIdx.x % kMlaHeads;
    __shared__ float w_s[64];
    __shared__ float s_total;
    if (threadIdx.x == 0) {
        float M = -INFINITY;
        for (int s = 0; s < splits; ++s)
            M = fmaxf(M, part_lse[((int64_t)t * splits + s) * kMlaHeads + h]);
        float tot = 0.f;
        for (int s = 0; s < splits; ++s) {
            const float ls = part_lse[((int64_t)t * splits + s) * kMlaHeads + h];
            const float wgt = (M == -INFINITY) ? 0.f : exp2f(ls - M);
            w_s[s] = wgt;
            tot += wgt;
        }
        s_total = tot;
        if (lse)
            lse[(int64_t)t * kMlaHeads + h] =
                (tot > 0.f) ? (M + log2f(tot)) * 0.6931471805599453f : -INFINITY;
    }
    __syncthreads();
    const float inv = (s_total > 0.f) ? kv_scale / s_total : 0.f;
    for (int d = threadIdx.x; d < kVDim; d += 128) {
        float acc = 0.f;
        for (int s = 0; s < splits; ++s)
            acc += w_s[s] *
                   __half2float(part_o[(((int64_t)t * splits + s) * kMlaHeads + h) * kVDim + d]);
        out[((int64_t)t * kMlaHeads + h) * kVDim + d] = __float2bfloat16_rn(acc * inv);
    }
}

}  // namespace

// Index-slot splits per token: more CTAs per token when there are few tokens.
// The count depends only on the number of query tokens, in steps, so a
// request's result is bit-identical across batches within one step.
int sparse_mla_splits(int total_q, int K) {
    int splits;
    if (total_q <= 9) splits = 16;
    else if (total_q <= 19) splits = 8;
    else if (total_q <= 38) splits = 4;
    else if (total_q <= 76) splits = 2;
    else splits = 1;
    while (splits > 1 && (K % (splits * kTileKeys)) != 0) splits >>= 1;
    return splits;
}

// Workspace: prepared queries [T][110592], exponents [T], then for split
// batches the f16 partial outputs [T, splits, 96, 512] and lse [T, splits, 96].
struct MlaWs {
    size_t q, qexp, part_o, part_lse, total;
};

MlaWs mla_ws_layout(int total_q, int K) {
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    const int splits = sparse_mla_splits(total_q, K);
    MlaWs w;
    w.q = 0;
    w.qexp = up((size_t)total_q * kQBytes);
    w.part_o = w.qexp + up((size_t)total_q * sizeof(int));
    const size_t po = splits > 1 ? (size_t)total_q * splits * kMlaHeads * kVDim * sizeof(__half) : 0;
    w.part_lse = w.part_o + up(po);
    const size_t pl = splits > 1 ? (size_t)total_q * splits * kMlaHeads * sizeof(float) : 0;
    w.total = w.part_lse + up(pl);
    return w;
}

size_t sparse_mla_workspace_bytes(int total_q, int K) { return mla_ws_layout(total_q, K).total; }

// Kernels one sparse-MLA call launches: query preparation, the MMA kernel and,
// for split batches, the combine.
int sparse_mla_launches(int total_q, int K) { return sparse_mla_splits(total_q, K) > 1 ? 3 : 2; }

cudaError_t launch_sparse_mla(const BatchArgs& bt, const uint16_t* q_lat, const void* latent_pages,
                              float kv_scale, float sm_scale, const int32_t* indices, int K,
                              uint16_t* out, float* lse, void* ws, int32_t* status,
                              cudaStream_t stream) {
    if (bt.total_q == 0) return cudaSuccess;
    MlaParams p;
    p.bt = bt;
    const MlaWs w = mla_ws_layout(bt.total_q, K);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    p.qf16 = wsb + w.q;
    p.qexp = reinterpret_cast<const int*>(wsb + w.qexp);
    p.latent_pages = static_cast<const uint8_t*>(latent_pages);
    p.indices = indices;
    p.K = K;
    p.splits = sparse_mla_splits(bt.total_q, K);
    p.split_keys = K / p.splits;
    p.kv_scale = kv_scale;
    p.sm_scale = sm_scale;
    p.out = reinterpret_cast<__nv_bfloat16*>(out);
    p.lse = lse;
    p.status = status;
    p.part_o = reinterpret_cast<__half*>(wsb + w.part_o);
    p.part_lse = reinterpret_cast<float*>(wsb + w.part_lse);
    sparse_mla_prep_q_kernel<<<bt.total_q, 256, 0, stream>>>(
        reinterpret_cast<const __nv_bfloat16*>(q_lat), wsb + w.q, reinterpret_cast<int*>(wsb + w.qexp));
    cudaError_t e = cudaFuncSetAttribute(sparse_mla_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    sparse_mla_tc_kernel<<<bt.total_q * p.splits, kThreads, kSmemAlloc, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess || p.splits == 1) return e;
    sparse_mla_combine_kernel<<<bt.total_q * kMlaHeads, 128, 0, stream>>>(
        p.part_o, p.part_lse, p.splits, kv_scale, p.out, lse);
    return cudaGetLastError();
}

}  // namespace dsa
