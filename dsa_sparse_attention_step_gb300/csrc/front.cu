// front.cu -- the fused indexer front on tcgen05 tensor cores.
//
// "vLLM's Kimi K3.1 Pro day-0 support", section "Fused low-latency decode for
// DSA layers", second step: one kernel does the query norm, the indexer query
// projection, FP8 quantisation with the head weights folded in, and the new
// token's index key.  For token t (query latent q_c [1536], hidden state
// x [7168], all bf16; synthetic projections W_q [4096, 1536] with the norm
// gain folded in, W_k [128, 7168], W_w [32, 7168]):
//   inv_rms = 1 / sqrt(mean(q_c^2) + 1e-6)
//   q[h, :] = inv_rms * (W_q q_c)[128 h .. 128 h + 127]  -> E4M3 with scale
//             amax/448 per (token, head): q_fp8, q_scale
//   w[h]    = (W_w x)[h]                                 head weights, fp32
//   key     = W_k x  -> E4M3 with scale amax/448, written into the token's
//             slot of the FP8 index cache
// (the indexer applies w * q_scale per head: the fold of the head weights into
// the quantised query).
//
// One CTA = one output tile x 128 tokens: D[128 features x 128 tokens] =
// W_tile[128 x K] . X[128 x K]^T with tcgen05.mma kind::f16 (bf16 x bf16, fp32
// accumulator in TMEM), operands by TMA (128-byte swizzle) into a 6-stage ring.
// The grid is launched as clusters of 8 CTAs: 4 clusters of query heads (8
// heads each, K = 1536), then the key and the head weights (K = 7168), each
// split over the 8 CTAs of its cluster by K (896 each); after its K range a
// split CTA leaves its fp32 partial in shared memory and rank 0 of the cluster
// adds the 8 partials in rank order through distributed shared memory (a fixed
// order: the result does not depend on timing) before the epilogue.
// Warp 0 issues the copies, warp 1 the MMAs, warp 2 (query tiles) sums the
// squares of the query latents from the same shared-memory tiles, warps 4-7
// run the epilogue (thread = feature, one TMEM lane each) in two halves of 64
// tokens: per-token amax over the tile's 128 features by warp max-reductions,
// the scale, the E4M3 codes (fp32 division, round to nearest even, saturating)
// and the stores.  Every wait is bounded.
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cooperative_groups.h>

#include "common.cuh"
#include "sm100.cuh"

namespace cg = cooperative_groups;

namespace dsa {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

namespace {

using namespace sm100;

constexpr int kDq = 1536;              // query latent
constexpr int kDh = 7168;              // hidden state
constexpr int kFTok = 128;             // tokens per CTA (MMA N)
constexpr int kFHalf = 64;             // epilogue columns per pass
constexpr int kFStages = 6;
constexpr int kFAStage = 128 * 128;    // 128 rows x 64 bf16
constexpr int kFBStage = kFTok * 128;  // 128 tokens x 64 bf16
constexpr int kFThreads = 256;
constexpr int kFCluster = 8;           // CTAs per cluster; K splits of the x tiles
constexpr int kTilesQ = kIdxHeads;     // 32 query tiles (one head each)
constexpr int kTileKey = kTilesQ;      // 32: key, split 8 ways (CTAs 32..39)
constexpr int kTileW = kTilesQ + 1;    // 33: head weights (CTAs 40..47)
constexpr int kFGridX = kTilesQ + 2 * kFCluster;  // 48
constexpr int kFOffA = 0;
constexpr int kFOffB = kFOffA + kFStages * kFAStage;
constexpr int kFOffF = kFOffB + kFStages * kFBStage;   // floats: inv_rms[128], amax[4][64]
constexpr int kFOffSlot = kFOffF + (kFTok + 4 * kFHalf) * 4;  // int64 key slot per token
constexpr int kFOffBar = kFOffSlot + kFTok * 8;
constexpr int kFSmemAlloc = kFOffBar + 256 + 1024;
static_assert(kFSmemAlloc <= 227 * 1024, "shared memory budget");
constexpr uint32_t kFIdesc = make_idesc(kFmtBF16, kFmtBF16, 128, kFTok, false, false);

struct FrontBars {
    uint64_t full[kFStages];
    uint64_t empty[kFStages];
    uint64_t done;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(FrontBars) <= 256, "barrier block");

struct FrontParams {
    BatchArgs bt;
    int T;
    uint8_t* q8;           // [T, 32, 128]
    float* qscale;         // [T, 32]
    float* w;              // [T, 32]
    uint8_t* index_pages;  // FP8 index pool or null
    float* q_f32;          // [T, 4096] or null
    float* k_f32;          // [T, 128] or null
    int32_t* status;
};

__global__ void __launch_bounds__(kFThreads, 1)
indexer_front_kernel(const __grid_constant__ CUtensorMap tm_wq,
                     const __grid_constant__ CUtensorMap tm_wk,
                     const __grid_constant__ CUtensorMap tm_ww,
                     const __grid_constant__ CUtensorMap tm_qc,
                     const __grid_constant__ CUtensorMap tm_x, const FrontParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    uint8_t* sA = sm + kFOffA;
    uint8_t* sB = sm + kFOffB;
    float* sInv = reinterpret_cast<float*>(sm + kFOffF);
    float* sAmax = sInv + kFTok;  // [4][64]
    int64_t* sSlot = reinterpret_cast<int64_t*>(sm + kFOffSlot);
    FrontBars* bars = reinterpret_cast<FrontBars*>(sm + kFOffBar);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool is_q = (int)blockIdx.x < kTilesQ;
    const int tile = is_q ? (int)blockIdx.x : kTilesQ + ((int)blockIdx.x - kTilesQ) / kFCluster;
    const int split = is_q ? 0 : ((int)blockIdx.x - kTilesQ) % kFCluster;  // = cluster rank
    const int t0 = blockIdx.y * kFTok;
    const int nk = is_q ? kDq / 64 : kDh / 64 / kFCluster;   // 24 or 14 chunks
    const int kc0 = split * nk;
    const CUtensorMap* tmA = is_q ? &tm_wq : (tile == kTileKey ? &tm_wk : &tm_ww);
    const CUtensorMap* tmB = is_q ? &tm_qc : &tm_x;
    const uint32_t a_bytes = (tile == kTileW) ? (uint32_t)(kIdxHeads * 128) : (uint32_t)kFAStage;
    // activation box: 64 tokens, or all of them when there are fewer
    const uint32_t b_bytes = (uint32_t)(min(p.T, kFTok) * 128);
    volatile int* abort_flag = &bars->abort_flag;

    if (tid == 0) {
        for (int s = 0; s < kFStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], is_q ? 2 : 1);  // the MMA commit (+ the norm warp)
        }
        mbar_init(&bars->done, 1);
        bars->abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(tmA);
        tma_prefetch_desc(tmB);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, kFTok);
        tmem_relinquish();
    }
    // key slots of this CTA's tokens (byte offset of the token's key in the
    // index pool, -1 when absent or out of range)
    if (tile == kTileKey && split == 0 && tid < kFTok) {
        int64_t off = -1;
        const int t = t0 + tid;
        if (t < p.T && p.index_pages) {
            const int b = request_of(p.bt, t);
            if (token_ok(p.bt, b, t, p.status)) {
                const int pos = visible_of(p.bt, b, t) - 1;  // the token's own position
                const int pg = page_lookup(p.bt, b, pos / kPage, p.status);
                if (pg >= 0) off = (int64_t)pg * kFp8PageBytes + (int64_t)(pos % kPage) * kIdxDim;
            }
        }
        sSlot[tid] = off;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int last = -1;
            for (int kc = 0; kc < nk; ++kc) {
                const int st = kc % kFStages;
                if (kc >= kFStages &&
                    !mbar_wait(&bars->empty[st], ((kc / kFStages) - 1) & 1, abort_flag))
                    break;
                mbar_arrive_expect_tx(&bars->full[st], a_bytes + b_bytes);
                tma_load_2d(sA + st * kFAStage, tmA, (kc0 + kc) * 64, is_q ? tile * 128 : 0, &bars->full[st]);
                tma_load_2d(sB + st * kFBStage, tmB, (kc0 + kc) * 64, t0, &bars->full[st]);
                last = kc;
            }
            // the copies must have landed before the CTA exits
            for (int j = 0; j < kFStages; ++j) {
                const int kc = last - j;
                if (kc < 0) break;
                mbar_drain(&bars->full[kc % kFStages], (kc / kFStages) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issue ----------------
        if (lane == 0) {
            const uint64_t ad = smem_desc(smem_u32(sA), 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(smem_u32(sB), 16, 1024, kSwizzle128B);
            for (int kc = 0; kc < nk; ++kc) {
                const int st = kc % kFStages;
                if (!mbar_wait(&bars->full[st], (kc / kFStages) & 1, abort_flag)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16(tmem, ad + (uint64_t)((st * kFAStage + 32 * kk) >> 4),
                            bd + (uint64_t)((st * kFBStage + 32 * kk) >> 4), kFIdesc,
                            (kc | kk) ? 1u : 0u);
                mma_commit(&bars->empty[st]);
            }
            mma_commit(&bars->done);
            mbar_drain(&bars->done, 0);
        }
        __syncwarp();
    } else if (warp == 2 && is_q) {
        // ---------------- query norm: sum of squares per token ----------------
        // lane l takes tokens l, l + 32, l + 64, l + 96 of each 64-element chunk
        float ss[4] = {0.f, 0.f, 0.f, 0.f};
        for (int kc = 0; kc < nk; ++kc) {
            const int st = kc % kFStages;
            if (!mbar_wait(&bars->full[st], (kc / kFStages) & 1, abort_flag)) break;
            const uint8_t* tileB = sB + st * kFBStage;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int r = lane + 32 * h;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = *reinterpret_cast<const uint4*>(tileB + sw128(r, 16 * c));
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float a = __uint_as_float(wv[k] << 16), b = __uint_as_float(wv[k] & 0xFFFF0000u);
                        ss[h] = fmaf(a, a, fmaf(b, b, ss[h]));
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->empty[st]);
        }
#pragma unroll
        for (int h = 0; h < 4; ++h) sInv[lane + 32 * h] = 1.0f / sqrtf(ss[h] / (float)kDq + 1e-6f);
    }

    // ---------------- epilogue (warps 4-7: thread = feature row) ----------------
    __syncthreads();  // the norm warp's 1/rms are in shared memory
    const int q4 = warp & 3;
    const int d = 32 * q4 + lane;  // feature row of the tile
    bool ok = true;
    if (warp >= 4) {
        ok = mbar_wait(&bars->done, 0, abort_flag);
        tc_fence_after();
    }
    // split tiles: each CTA's fp32 partial [128 rows][128 tokens] goes to its
    // own shared memory (the operand ring is idle now), rank 0 adds them
    float* sPart = reinterpret_cast<float*>(sA);
    if (!is_q) {
        if (warp >= 4 && ok) {
            for (int c = 0; c < kFTok; c += 32) {
                uint32_t v[32];
                tmem_ld32(tmem_addr(tmem, 32 * q4, c), v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4*>(sPart + d * kFTok + c + j) =
                        make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                    __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
            }
        }
        cg::this_cluster().sync();  // every partial is written
    }
    if (warp >= 4 && ok && (is_q || split == 0)) {
        for (int half = 0; half < kFTok / kFHalf; ++half) {
            const int c0 = half * kFHalf;
            float v[kFHalf];
            if (is_q) {
                uint32_t u[kFHalf];
                tmem_ld32(tmem_addr(tmem, 32 * q4, c0), *reinterpret_cast<uint32_t(*)[32]>(u));
                tmem_ld32(tmem_addr(tmem, 32 * q4, c0 + 32), *reinterpret_cast<uint32_t(*)[32]>(u + 32));
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < kFHalf; ++j) v[j] = __uint_as_float(u[j]) * sInv[c0 + j];
            } else {
                // the 8 partials of this row, added in rank order
#pragma unroll
                for (int j = 0; j < kFHalf; ++j) v[j] = 0.f;
                cg::cluster_group cl = cg::this_cluster();
                for (int r = 0; r < kFCluster; ++r) {
                    const float* src = cl.map_shared_rank(sPart, r) + d * kFTok + c0;
#pragma unroll
                    for (int j = 0; j < kFHalf; j += 4) {
                        const float4 x4 = *reinterpret_cast<const float4*>(src + j);
                        v[j] += x4.x; v[j + 1] += x4.y; v[j + 2] += x4.z; v[j + 3] += x4.w;
                    }
                }
            }
            if (tile == kTileW) {
                if (q4 == 0 && p.w) {
#pragma unroll
                    for (int j = 0; j < kFHalf; ++j)
                        if (t0 + c0 + j < p.T) p.w[(int64_t)(t0 + c0 + j) * kIdxHeads + d] = v[j];
                }
                continue;
            }
            // per-token amax over the 128 features: |x| compares as unsigned
#pragma unroll
            for (int j = 0; j < kFHalf; ++j) {
                const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(v[j]) & 0x7FFFFFFFu);
                if (lane == 0) sAmax[q4 * kFHalf + j] = __uint_as_float(m);
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
#pragma unroll
            for (int j = 0; j < kFHalf; ++j) {
                const int t = t0 + c0 + j;
                if (t >= p.T) continue;
                const float amax = fmaxf(fmaxf(sAmax[j], sAmax[kFHalf + j]),
                                         fmaxf(sAmax[2 * kFHalf + j], sAmax[3 * kFHalf + j]));
                const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
                const float x = v[j];
                const uint8_t code = (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(x, scale), __NV_SATFINITE, __NV_E4M3);
                if (is_q) {
                    p.q8[(int64_t)t * (kIdxHeads * kIdxDim) + tile * kIdxDim + d] = code;
                    if (p.q_f32) p.q_f32[(int64_t)t * (kIdxHeads * kIdxDim) + tile * kIdxDim + d] = x;
                    if (d == 0) p.qscale[(int64_t)t * kIdxHeads + tile] = scale;
                } else {
                    const int64_t off = sSlot[c0 + j];
                    if (off >= 0) {
                        p.index_pages[off + d] = code;
                        if (d == 0) {
                            const int64_t page0 = off - off % kFp8PageBytes;
                            const int slot = (int)((off % kFp8PageBytes) / kIdxDim);
                            *reinterpret_cast<float*>(p.index_pages + page0 + kPage * kIdxDim + 4 * slot) = scale;
                        }
                    }
                    if (p.k_f32) p.k_f32[(int64_t)t * kIdxDim + d] = x;
                }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");  // sAmax is reused by the next half
        }
    }
    if (!is_q) cg::this_cluster().sync();  // rank 0 has read every partial

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && tid == 0) record_error(p.status, DSA_ERR_TIMEOUT);
    if (warp == 1) tmem_dealloc(tmem, kFTok);
}

// bf16 matrix [rows, cols] row-major, box [box_rows, 64 columns], 128-B swizzle
bool encode_bf16(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_indexer_front(const BatchArgs& bt, const uint16_t* q_c, const uint16_t* x,
                                 const uint16_t* w_q, const uint16_t* w_k, const uint16_t* w_w,
                                 uint8_t* q8, float* qscale, float* w, void* index_pages,
                                 float* q_f32, float* k_f32, int32_t* status, cudaStream_t stream) {
    const int T = bt.total_q;
    if (T == 0) return cudaSuccess;
    CUtensorMap tm_wq, tm_wk, tm_ww, tm_qc, tm_x;
    memset(&tm_wq, 0, sizeof(tm_wq));
    memset(&tm_wk, 0, sizeof(tm_wk));
    memset(&tm_ww, 0, sizeof(tm_ww));
    memset(&tm_qc, 0, sizeof(tm_qc));
    memset(&tm_x, 0, sizeof(tm_x));
    if (!encode_bf16(&tm_wq, w_q, kIdxHeads * kIdxDim, kDq, 128) ||
        !encode_bf16(&tm_wk, w_k, kIdxDim, kDh, 128) ||
        !encode_bf16(&tm_ww, w_w, kIdxHeads, kDh, kIdxHeads) ||
        !encode_bf16(&tm_qc, q_c, (uint64_t)T, kDq, (uint32_t)(T < kFTok ? T : kFTok)) ||
        !encode_bf16(&tm_x, x, (uint64_t)T, kDh, (uint32_t)(T < kFTok ? T : kFTok)))
        return cudaErrorInvalidValue;
    FrontParams p;
    p.bt = bt;
    p.T = T;
    p.q8 = q8;
    p.qscale = qscale;
    p.w = w;
    p.index_pages = static_cast<uint8_t*>(index_pages);
    p.q_f32 = q_f32;
    p.k_f32 = k_f32;
    p.status = status;
    cudaError_t e = cudaFuncSetAttribute(indexer_front_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kFSmemAlloc);
    if (e != cudaSuccess) return e;
    const dim3 grid(kFGridX, (unsigned)((T + kFTok - 1) / kFTok));
    return launch_kernel(indexer_front_kernel, grid, dim3(kFThreads), (size_t)kFSmemAlloc, stream,
                         false, kFCluster, tm_wq, tm_wk, tm_ww, tm_qc, tm_x, p);
}

}  // namespace dsa
