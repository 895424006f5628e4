/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DSA sparse-attention step library
 * (libdsa.so).
 *
 * One layer of DeepSeek-style sparse attention as the web page "vLLM's Kimi
 * K3.1 Pro day-0 support: sparse attention, DCP, zero-mismatch RL"
 * (agentlenshq.com/ja/blogs/5e91cd0c...) describes it:
 *   - section "What changed" (table and text): a light indexer with 32 heads
 *     of 128 dims scores every earlier token of a query against one FP8 key per
 *     token (132 bytes with its scale); the top 2048 tokens are kept and MLA
 *     attention runs exactly on those tokens only;
 *   - section "Sparse attention cuts long-context decode bandwidth": the full
 *     576-byte FP8 latent is read only for the 2048 selected tokens;
 *   - section "Packed KV cache": index keys are 132 B (FP8) or 68 B (MXFP4) per
 *     token; kernels see small fixed-size pages through a block table that is
 *     translated to page addresses before each step;
 *   - section "Fused low-latency decode for DSA layers": a key-balanced scorer
 *     and an exact top-k selection feed sparse attention; the new tokens' key
 *     and latent are written into the caches.
 * The pages do not state the indexer formula.  This library computes
 *     score[t,s] = sum_h w[t,h] * ReLU( qhat[t,h,:] . khat[s,:] )
 * with qhat = E4M3(q) * q_scale[t,h] and khat the dequantised key, and selects
 * the top-k positions with ties broken toward the lower position.
 *
 * Conventions shared by every entry point
 *   - All pointers except the dsa_batch struct itself are DEVICE pointers owned
 *     by the caller.  The library allocates nothing, keeps no state between
 *     calls (apart from a launch counter, the batch-invariant switch and the
 *     fixed scratch array of dsa_decode_noalloc) and is safe to call from
 *     several host threads on different streams, except dsa_decode_noalloc
 *     calls whose executions overlap on the GPU (they share that array; see
 *     below).
 *   - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t;
 *     NULL = legacy default stream).  Argument errors the host can see are
 *     returned before anything is launched; nothing is written then.
 *   - Device-side checks (a block-table entry outside [0, num_pages), a selected
 *     position outside [0, seq_len)) skip the offending access and store the
 *     first error code (DSA_ERR_DEVICE_CHECK) into *dev_status when dev_status
 *     is not NULL.  The caller clears *dev_status to 0 and reads it after
 *     synchronising.
 *   - Query token t belongs to request b with q_offsets[b] <= t < q_offsets[b+1]
 *     (n_b = q_offsets[b+1]-q_offsets[b] tokens).  Token j of request b sits at
 *     position seq_lens[b] - n_b + j and sees positions
 *     0 .. seq_lens[b] - n_b + j (causal multi-token rule; n_b = 1 is plain
 *     decode, n_b new tokens is prefill-append).
 *   - Position s of request b lives in physical page block_table[b*max_pages +
 *     s/64], slot s%64.  page_size must be 64.
 *   - Cache page layouts (one layer; a page id indexes both pools):
 *       FP8 index page   (8448 B): 64 x 128 E4M3 key bytes, then 64 fp32 scales
 *       MXFP4 index page (4352 B): 64 x 64 bytes of packed E2M1 (element 2i in
 *                                  the low nibble), then 64 x 4 E8M0 scales,
 *                                  one per block of 32 elements
 *       latent page     (36864 B): 64 x 576 E4M3 bytes; one fp32 scale per layer
 *     Pool bases must be 16-byte aligned.
 *   - Only the shapes of the pages are supported: 32 indexer heads x 128 dims,
 *     96 MLA heads x 576 latent dims with values = dims 0..511, top-k = 2048.
 *     Other values return DSA_ERR_UNSUPPORTED.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dsa_stream_t; /* same type as cudaStream_t */

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1,  /* NULL/misaligned pointer, inconsistent sizes */
    DSA_ERR_UNSUPPORTED = 2,  /* a shape or format outside the supported set */
    DSA_ERR_WORKSPACE = 3,    /* workspace too small */
    DSA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    DSA_ERR_DEVICE_CHECK = 5, /* (device status word) page id or position out of range */
    DSA_ERR_TIMEOUT = 6       /* (device status word) a bounded device wait expired */
} dsa_status;

typedef enum { DSA_KEYS_FP8_E4M3 = 0, DSA_KEYS_MXFP4 = 1 } dsa_key_format;

/* Latent page format (section "Packed KV cache": 576 B FP8 or 352 B NVFP4 per
 * token).  The pages print only the NVFP4 width; the byte split used is the
 * one described at dsa_sparse_mla_ex. */
typedef enum { DSA_LATENT_FP8_E4M3 = 0, DSA_LATENT_NVFP4 = 1 } dsa_latent_format;

enum {
    DSA_PAGE_SIZE = 64,
    DSA_INDEX_HEADS = 32,
    DSA_INDEX_DIM = 128,
    DSA_MLA_HEADS = 96,
    DSA_LATENT_DIM = 576,
    DSA_VALUE_DIM = 512,
    DSA_TOPK = 2048,
    DSA_FP8_INDEX_PAGE_BYTES = 8448,
    DSA_MXFP4_INDEX_PAGE_BYTES = 4352,
    DSA_LATENT_PAGE_BYTES = 36864,
    DSA_NVFP4_LATENT_PAGE_BYTES = 22528
};

/* Request metadata of one step.  The struct lives in host memory; the three
 * arrays are device pointers.  The host copies (total_q, max_q_per_request,
 * max_seq_len) must agree with the device arrays; they size the grids. */
typedef struct {
    int32_t num_requests;       /* B >= 1 */
    int32_t total_q;            /* T = q_offsets[B] */
    int32_t max_q_per_request;  /* max_b n_b */
    int32_t max_seq_len;        /* max_b seq_lens[b] */
    int32_t num_pages;          /* pages in each cache pool */
    int32_t max_pages;          /* row stride of block_table, >= ceil(max_seq_len/64) */
    int32_t page_size;          /* must be 64 */
    const int32_t* q_offsets;   /* device [B+1], q_offsets[0] = 0, non-decreasing */
    const int32_t* seq_lens;    /* device [B], seq_lens[b] >= n_b */
    const int32_t* block_table; /* device [B * max_pages] physical page ids */
} dsa_batch;

/* Human-readable name of a status code (static string). */
const char* dsa_status_string(dsa_status s);

/* Number of kernels this library has launched in this process (monotonic). */
uint64_t dsa_launch_count(void);

/* ---- batch-invariant plan ----------------------------------------------------
 * Section "Zero-mismatch RL" (a switch under which a token's result does not
 * depend on the batch it runs in; the page's top-k is batch-invariant by
 * design).  The indexer and the exact top-k of this library always are.  The
 * sparse MLA by default runs whole waves of one CTA per token and splits each
 * token of a last, partial wave into pieces merged by log-sum-exp, the piece
 * count set by the batch size, so a token's out and lse can differ in rounding
 * between batches.  With enabled != 0 every token runs whole: out and lse of a
 * token depend on its own inputs alone, and equal the default plan's wherever
 * that plan runs the token whole.  Small batches then use fewer SMs.
 * Process-wide; read once by each later call of dsa_sparse_mla(_ex),
 * dsa_decode(_ex) and dsa_decode_noalloc.  Workspace sizes do not change.
 * Returns the previous setting (0 or 1); the default is 0. */
int32_t dsa_set_batch_invariant(int32_t enabled);

/* ---- indexer -------------------------------------------------------------
 * Section "What changed" (32 heads x 128 dims, FP8 key with its scale, every
 * earlier token scored) and, for MXFP4 keys, section "Native MXFP4 indexer"
 * (fp32 accumulation, weighted reduction across heads).
 *   q_fp8    [T,32,128] E4M3 bytes           (16-byte aligned)
 *   q_scale  [T,32] fp32, > 0                (dequantisation of q per head)
 *   w        [T,32] fp32                     (head weights)
 *   index_pages: the FP8 or MXFP4 index pool
 *   scores   [T, score_ld] fp32 output, score_ld >= max_seq_len and a multiple
 *            of 4.  For token t of request b: scores[t,s] for s < visible(t);
 *            -inf for visible(t) <= s < seq_lens[b]; entries s >= seq_lens[b]
 *            are not written.
 * The key scale (FP8) must be positive: the kernel applies it after the ReLU.
 * Batches of more than 4096 requests return DSA_ERR_UNSUPPORTED. */
dsa_status dsa_index_scores(const dsa_batch* batch, const uint8_t* q_fp8,
                            const float* q_scale, const float* w, const void* index_pages,
                            dsa_key_format key_format, float* scores, int64_t score_ld,
                            int32_t* dev_status, dsa_stream_t stream);

/* ---- exact top-k -----------------------------------------------------------
 * Section "What changed" (the top 2048 tokens are kept) and section "Fused
 * low-latency decode" (exact top-k after the scorer).  For each query token t:
 * the topk positions s < visible(t) with the largest scores[t,s], ties going to
 * the lower position, written to indices[t, 0..topk) in ascending position
 * order; when visible(t) <= topk all visible positions are written and the rest
 * is -1.  Scores must not be NaN.  -0.0 and +0.0 are equal.
 *   indices  [T, topk] int32 output (logical positions)
 *   ws       device scratch of at least dsa_topk_workspace_size() bytes,
 *            16-byte aligned (may be NULL when that size is 0).  The size is
 *            nonzero for batches of at most 8 query tokens with max_seq_len
 *            above 32768: their rows are split over the whole GPU and the
 *            scratch holds the row histograms and per-slice counts (it is
 *            cleared by the call; its contents need not be kept between
 *            calls).  Returns DSA_ERR_WORKSPACE when it is missing or short. */
size_t dsa_topk_workspace_size(const dsa_batch* batch, int32_t topk);
dsa_status dsa_topk(const dsa_batch* batch, const float* scores, int64_t score_ld,
                    int32_t topk, int32_t* indices, void* ws, size_t ws_bytes,
                    dsa_stream_t stream);

/* ---- sparse MLA (absorbed form) --------------------------------------------
 * Section "What changed" (MLA run exactly on the selected tokens) and section
 * "Sparse attention cuts long-context decode bandwidth" (576-byte FP8 latents
 * read for the selected tokens only).  For token t, head h (96 heads) over the
 * selected positions I = {indices[t,i] >= 0}:
 *   z[h,s] = sm_scale * kv_scale * (q_lat[t,h,:] . E4M3(latent[s,:]))  (576 dims)
 *   out[t,h,:] = kv_scale * sum_s softmax_s(z[h,s]) * E4M3(latent[s,0:512])
 *   lse[t,h]   = log sum_s exp(z[h,s])      (natural log; -inf if I is empty)
 *   q_lat    [T,96,576] bf16 bits            (16-byte aligned)
 *   indices  [T, topk] int32, entries -1 (skipped) or in [0, seq_lens[b])
 *   out      [T,96,512] bf16 output (round to nearest even; 0 if I is empty)
 *   lse      [T,96] fp32 output, may be NULL
 *   ws       device scratch of at least dsa_sparse_mla_workspace_size() bytes */
size_t dsa_sparse_mla_workspace_size(const dsa_batch* batch, int32_t topk);
dsa_status dsa_sparse_mla(const dsa_batch* batch, const uint16_t* q_lat,
                          const void* latent_pages, float kv_scale, float sm_scale,
                          const int32_t* indices, int32_t topk, uint16_t* out, float* lse,
                          void* ws, size_t ws_bytes, int32_t* dev_status,
                          dsa_stream_t stream);

/* dsa_sparse_mla with the latent format as an argument.  DSA_LATENT_FP8_E4M3 is
 * dsa_sparse_mla.  DSA_LATENT_NVFP4: section "Packed KV cache" (NVFP4
 * latents, 352 bytes per token); each token's 352 bytes, 64 tokens per page
 * (22528 B), are
 *   bytes   0..255  dims 0..511 as E2M1 (element 2i in the low nibble of byte i)
 *   bytes 256..287  one E4M3 scale per block of 16 of those elements
 *   bytes 288..351  dims 512..575 as E4M3
 * and the latent is lhat[d] = E2M1 * E4M3(block scale) * kv_scale for d < 512,
 * E4M3 * kv_scale for d >= 512.  Every such value is exact in f16, and the
 * kernel lifts it exactly, so the arithmetic after the lift is that of FP8
 * latents. */
dsa_status dsa_sparse_mla_ex(const dsa_batch* batch, const uint16_t* q_lat,
                             const void* latent_pages, dsa_latent_format latent_format,
                             float kv_scale, float sm_scale, const int32_t* indices, int32_t topk,
                             uint16_t* out, float* lse, void* ws, size_t ws_bytes,
                             int32_t* dev_status, dsa_stream_t stream);

/* ---- the fused step ---------------------------------------------------------
 * dsa_index_scores -> dsa_topk -> dsa_sparse_mla on one stream, the scores
 * kept in the workspace (section "Fused low-latency decode for DSA layers").
 * Arguments as above; indices [T, topk] is an output. */
size_t dsa_decode_workspace_size(const dsa_batch* batch, int32_t topk);
dsa_status dsa_decode(const dsa_batch* batch, const uint8_t* q_fp8, const float* q_scale,
                      const float* w, const void* index_pages, dsa_key_format key_format,
                      const uint16_t* q_lat, const void* latent_pages, float kv_scale,
                      float sm_scale, int32_t topk, uint16_t* out, float* lse,
                      int32_t* indices, void* ws, size_t ws_bytes, int32_t* dev_status,
                      dsa_stream_t stream);

/* dsa_decode with the latent format as an argument (see dsa_sparse_mla_ex);
 * DSA_LATENT_FP8_E4M3 is dsa_decode.  Same workspace size. */
dsa_status dsa_decode_ex(const dsa_batch* batch, const uint8_t* q_fp8, const float* q_scale,
                         const float* w, const void* index_pages, dsa_key_format key_format,
                         const uint16_t* q_lat, const void* latent_pages,
                         dsa_latent_format latent_format, float kv_scale, float sm_scale,
                         int32_t topk, uint16_t* out, float* lse, int32_t* indices, void* ws,
                         size_t ws_bytes, int32_t* dev_status, dsa_stream_t stream);

/* ---- the fused step without caller scratch ------------------------------------
 * No counterpart on the pages: an addition of this library.  Same arguments,
 * outputs and results as dsa_decode, minus the workspace: its scratch (the
 * score rows) lives in one file-scope device array of DSA_NOALLOC_SCRATCH_BYTES
 * bytes inside the library, so the call itself allocates nothing.  It is meant
 * for callers that cannot obtain device memory on the call path, such as an
 * engine whose device memory is entirely pre-reserved by its own pool (the KV
 * cache), or code running where the device-synchronising cudaMalloc/cudaFree
 * may not be called.
 *   - A batch whose dsa_decode_workspace_size() exceeds
 *     DSA_NOALLOC_SCRATCH_BYTES is rejected with DSA_ERR_WORKSPACE before
 *     anything is launched.
 *   - Each call outside stream capture looks up the device address of the
 *     current device's copy of the array (with that device current); a call
 *     made while `stream` is capturing uses the address found by the last
 *     call outside capture.  Make the first call on each device before any
 *     stream capture on it, and after a cudaDeviceReset make one call outside
 *     capture before capturing again (the reset may move the array).
 *   - Every GPU that loads the library holds the array until the process exits.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents; nothing in it needs to start at zero.  Calls whose executions
 *     overlap on the GPU (different streams, no ordering between them) race on
 *     it and give undefined results: order them on one stream or with events. */
enum { DSA_NOALLOC_SCRATCH_BYTES = 16 << 20 };
dsa_status dsa_decode_noalloc(const dsa_batch* batch, const uint8_t* q_fp8,
                              const float* q_scale, const float* w, const void* index_pages,
                              dsa_key_format key_format, const uint16_t* q_lat,
                              const void* latent_pages, float kv_scale, float sm_scale,
                              int32_t topk, uint16_t* out, float* lse, int32_t* indices,
                              int32_t* dev_status, dsa_stream_t stream);

/* ---- cache append -------------------------------------------------------------
 * Section "Fused low-latency decode for DSA layers" (the new token's index key
 * and latent are written into the caches).  The T = q_offsets[B] new tokens
 * are the query tokens of the batch; token j of request b goes to position
 * seq_lens[b] - n_b + j.
 *   new_keys   [T,128] fp32 (may be NULL: index pool untouched). FP8 pool only:
 *              scale = amax/448 (1 if amax == 0), code = E4M3 round-to-nearest-
 *              even saturating of (x / scale), both fp32 divisions.
 *   new_latent [T,576] fp32 (may be NULL): code = E4M3 RNE satfinite (x / kv_scale).
 * Only the new tokens' slots are written. */
dsa_status dsa_append_cache(const dsa_batch* batch, const float* new_keys,
                            const float* new_latent, float kv_scale, void* index_pages,
                            void* latent_pages, dsa_key_format key_format,
                            int32_t* dev_status, dsa_stream_t stream);

/* ---- fused indexer front --------------------------------------------------------
 * Section "Fused low-latency decode for DSA layers", second step: one kernel
 * does the query norm, the indexer query projection, FP8 quantisation with the
 * head weights folded in, and the new token's index key.  The pages give no
 * dimensions or formulas; this library reads them as follows, for each of the
 * batch's T query tokens (all matrices bf16, row-major):
 *   q_c  [T, 1536]   the token's query latent
 *   x    [T, 7168]   the token's hidden state
 *   w_q  [4096, 1536] indexer query projection (the query norm's gain folded in)
 *   w_k  [128, 7168]  index-key projection
 *   w_w  [32, 7168]   head-weight projection
 *   inv_rms = 1 / sqrt(mean(q_c^2) + 1e-6)
 *   q[t, h, :] = inv_rms * (w_q q_c)[128 h .. 128 h + 127]
 *   q_fp8[t, h, :] = E4M3(q / q_scale[t, h]),  q_scale[t, h] = amax(|q[t, h, :]|) / 448
 *   w[t, h] = (w_w x)[h]            (the indexer applies w * q_scale per head)
 *   key = w_k x -> 128 E4M3 codes with scale amax / 448, written into the token's
 *                  slot of the FP8 index cache (position seq_lens[b] - n_b + j,
 *                  as dsa_append_cache places it); index_pages may be NULL
 * Quantisation: the scale is 1 when amax is 0; codes are round-to-nearest-even
 * saturating of x / scale (fp32 division), as in dsa_append_cache.
 *   q_fp8 [T, 32, 128], q_scale [T, 32], w [T, 32]: outputs (16-byte aligned)
 *   q_f32 [T, 4096], k_f32 [T, 128]: optional fp32 outputs of the projections
 *          before quantisation (NULL to skip), for checking the codes
 * The outputs q_fp8, q_scale and w are the indexer's inputs (dsa_index_scores).
 * An MXFP4 index pool returns DSA_ERR_UNSUPPORTED for the key write. */
dsa_status dsa_indexer_front(const dsa_batch* batch, const uint16_t* q_c, const uint16_t* x,
                             const uint16_t* w_q, const uint16_t* w_k, const uint16_t* w_w,
                             uint8_t* q_fp8, float* q_scale, float* w, void* index_pages,
                             dsa_key_format key_format, float* q_f32, float* k_f32,
                             int32_t* dev_status, dsa_stream_t stream);

/* ---- decode context parallelism: exact top-k merge and LSE combine ---------------
 * Section "Decode context parallelism with the sparse indexer": with DCP over
 * W ranks, rank r holds every W-th token (positions s = r mod W) and ranks only
 * its own tokens, so the global top-2048 is merged across ranks before
 * attention, and the ranks' partial attention outputs are combined by
 * log-sum-exp.  Section "Exact top-k merge with about 10x less traffic": each
 * rank sends its best ceil(1.5 * 2048 / W) candidates, chosen from BF16
 * scores and packed with the score into 32 bits; every rank radix-selects the
 * same global top-2048 from the gathered candidates; a rank holding more of
 * it than it sent is detected and resends its full local top-k for that row.
 *
 * dsa_dcp_topk runs that protocol for all W ranks of each query row on one
 * GPU, the ranks' shards being the interleaved positions of the row in
 * `scores` (as dsa_index_scores writes them) and the exchange going through
 * the workspace.  Result: for each query token t, the topk visible positions
 * with the largest BF16-rounded scores (round to nearest even), ties to the
 * lower position, in ascending order, -1 padded -- exactly, whatever the
 * distribution of winners over ranks.
 *   world         W, 1..8
 *   cand          candidates per rank, 1..topk; 0 = min(ceil(1.5 * topk / W), topk)
 *   indices       [T, topk] int32 output
 *   rank_indices  [W, T, topk] int32 output (may be NULL): rank r's share of
 *                 the selection (the positions with s mod W == r), ascending,
 *                 -1 padded -- the index list rank r attends over
 *   resent        [T, W] int32 output (may be NULL): 1 where rank r had to
 *                 resend its local top-k for the row, else 0
 *   ws            device scratch of dsa_dcp_topk_workspace_size() bytes (the
 *                 exchanged candidate words and resend lists), 16-byte aligned
 * The packed word keeps a rank-local position in 16 bits, so max_seq_len must
 * be at most 65536 * W (DSA_ERR_UNSUPPORTED otherwise).  topk must be 2048.
 * Scores must not be NaN.  Four kernel launches. */
size_t dsa_dcp_topk_workspace_size(const dsa_batch* batch, int32_t world, int32_t cand,
                                   int32_t topk);
dsa_status dsa_dcp_topk(const dsa_batch* batch, const float* scores, int64_t score_ld,
                        int32_t world, int32_t cand, int32_t topk, int32_t* indices,
                        int32_t* rank_indices, int32_t* resent, void* ws, size_t ws_bytes,
                        dsa_stream_t stream);

/* The log-sum-exp combine of W partial attention results over disjoint token
 * sets (for instance the outputs of dsa_sparse_mla over each rank's
 * rank_indices):
 *   L = log sum_r exp(part_lse[r,t,h]),
 *   out[t,h,:] = sum_r exp(part_lse[r,t,h] - L) * part_out[r,t,h,:]
 *   part_out  [W, T, 96, 512] bf16 (16-byte aligned)
 *   part_lse  [W, T, 96] fp32, natural log; -inf for a rank with no tokens
 *   out       [T, 96, 512] bf16 output; lse [T, 96] fp32 output (may be NULL)
 * A (t, h) with no tokens on any rank gives out = 0 and lse = -inf.
 * world must be 1..8. */
dsa_status dsa_lse_combine(int32_t total_q, int32_t world, const uint16_t* part_out,
                           const float* part_lse, uint16_t* out, float* lse,
                           dsa_stream_t stream);

/* ---- token-sharded prefill planner (host only) ----------------------------------
 * Section "Token-sharded prefill improves time to first token": for a large
 * prefill step each rank of W runs the indexer and sparse MLA for a share of
 * the query tokens (all 96 heads) instead of a share of the heads; to balance
 * causal work every request is cut into 2W parts (16 for W = 8) and rank r
 * takes parts r and 2W - 1 - r.  Part i of a request with n new tokens is its
 * tokens [floor(i n / 2W), floor((i + 1) n / 2W)).
 * Each part is returned as a sub-request for a dsa_batch of the rank: its
 * tokens are the batch's query tokens token_begin .. token_begin + num_tokens
 * - 1 (indices into the original batch, whose request b holds q_counts[b]
 * tokens in order), its context ends at its last token (seq_len), and its
 * block-table row is that of `request`.  With that context the step's causal
 * rule gives every token exactly the positions it sees in the whole request,
 * so the rank's results for its tokens equal the unsharded step's.
 *   seq_lens, q_counts  host [num_requests]: context (incl. new tokens), new tokens
 *   parts               host output, up to max_parts entries (2 per request at
 *                       most; empty parts are skipped)
 * Returns the number of parts written, or a negated dsa_status:
 * -DSA_ERR_INVALID_ARG for bad sizes, -DSA_ERR_WORKSPACE when max_parts is
 * too small.  Pure host code: no device, stream or allocation. */
typedef struct {
    int32_t request;      /* index of the original request */
    int32_t token_begin;  /* first query token of the part, in the original batch */
    int32_t num_tokens;   /* query tokens in the part (> 0) */
    int32_t seq_len;      /* the part's context: position of its last token + 1 */
} dsa_shard_part;
int32_t dsa_plan_token_shards(const int32_t* seq_lens, const int32_t* q_counts,
                              int32_t num_requests, int32_t world, int32_t rank,
                              dsa_shard_part* parts, int32_t max_parts);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
