// api.cu -- the extern "C" boundary of libdsa.so: argument validation,
// workspace arithmetic and kernel launches.  See include/dsa.h.
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "../../include/dsa_testing.h"

namespace dsa {
cudaError_t launch_index_scores(const BatchArgs& bt, const uint8_t* q8, const float* qscale,
                                const float* w, const void* pages, int key_format,
                                float* scores, int64_t ld, int32_t* status, cudaStream_t stream);
bool indexer_supported(const BatchArgs& bt);
cudaError_t launch_topk(const BatchArgs& bt, const float* scores, int64_t ld, int K,
                        int32_t* out, void* ws, bool pdl, cudaStream_t stream);
size_t topk_workspace_bytes(int total_q, int max_seq);
int topk_launches(int total_q, int max_seq);
bool topk_supported(int max_seq);
cudaError_t launch_sparse_mla(const BatchArgs& bt, const uint16_t* q_lat, const void* latent_pages,
                              float kv_scale, float sm_scale, const int32_t* indices, int K,
                              uint16_t* out, float* lse, void* ws, int32_t* status, bool pdl,
                              cudaStream_t stream, bool wait_test, int latent_format,
                              bool whole_only);
size_t sparse_mla_workspace_bytes(int total_q, int K);
int sparse_mla_launches(int total_q, int K, bool whole_only);
cudaError_t launch_append_cache(const BatchArgs& bt, const float* keys, const float* lat,
                                float kv_scale, void* index_pages, void* latent_pages,
                                int32_t* status, cudaStream_t stream);

int dcp_default_cand(int world, int K);
struct DcpWs {
    size_t sent, sent_n, full, full_n, flags, total;
};
DcpWs dcp_ws_layout(int total_q, int world, int cand, int K);
bool dcp_supported(int world, int max_seq);
cudaError_t launch_dcp_topk(const BatchArgs& bt, const float* scores, int64_t ld, int world,
                            int cand, int K, int32_t* indices, int32_t* rank_indices,
                            int32_t* resent, void* ws, cudaStream_t stream);
cudaError_t launch_lse_combine(int total_q, int world, const uint16_t* part, const float* part_lse,
                               uint16_t* out, float* lse, cudaStream_t stream);

cudaError_t launch_indexer_front(const BatchArgs& bt, const uint16_t* q_c, const uint16_t* x,
                                 const uint16_t* w_q, const uint16_t* w_k, const uint16_t* w_w,
                                 uint8_t* q8, float* qscale, float* w, void* index_pages,
                                 float* q_f32, float* k_f32, int32_t* status, cudaStream_t stream);

std::atomic<uint64_t> g_launches{0};
std::atomic<int32_t> g_batch_invariant{0};  // dsa_set_batch_invariant
}  // namespace dsa

using namespace dsa;

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dsa_status check_batch(const dsa_batch* bt) {
    if (bt == nullptr) return DSA_ERR_INVALID_ARG;
    if (bt->page_size != kPage) return DSA_ERR_UNSUPPORTED;
    if (bt->num_requests < 1 || bt->total_q < 0 || bt->max_q_per_request < 0 ||
        bt->max_seq_len < 1 || bt->num_pages < 1 || bt->max_pages < 1)
        return DSA_ERR_INVALID_ARG;
    if ((int64_t)bt->max_pages * kPage < bt->max_seq_len) return DSA_ERR_INVALID_ARG;
    if (bt->max_q_per_request > bt->max_seq_len) return DSA_ERR_INVALID_ARG;
    if ((int64_t)bt->total_q > (int64_t)bt->num_requests * bt->max_q_per_request)
        return DSA_ERR_INVALID_ARG;
    if (!bt->q_offsets || !bt->seq_lens || !bt->block_table) return DSA_ERR_INVALID_ARG;
    return DSA_OK;
}

BatchArgs to_args(const dsa_batch* bt) {
    BatchArgs a;
    a.num_requests = bt->num_requests;
    a.total_q = bt->total_q;
    a.max_q = bt->max_q_per_request;
    a.max_seq = bt->max_seq_len;
    a.num_pages = bt->num_pages;
    a.max_pages = bt->max_pages;
    a.q_offsets = bt->q_offsets;
    a.seq_lens = bt->seq_lens;
    a.block_table = bt->block_table;
    return a;
}

inline dsa_status cuda_status(cudaError_t e) {
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline int64_t score_ld_for(const dsa_batch* bt) {
    return (int64_t)align_up((size_t)bt->max_seq_len, 128);
}

dsa_status check_index_args(const dsa_batch* bt, const uint8_t* q8, const float* qscale,
                            const float* w, const void* pages, dsa_key_format fmt,
                            const float* scores, int64_t ld) {
    if (fmt != DSA_KEYS_FP8_E4M3 && fmt != DSA_KEYS_MXFP4) return DSA_ERR_UNSUPPORTED;
    if (!indexer_supported(to_args(bt))) return DSA_ERR_UNSUPPORTED;
    if (!q8 || !qscale || !w || !pages || !scores) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q8) || !aligned16(pages) || !aligned16(scores) || !aligned16(qscale) ||
        !aligned16(w))
        return DSA_ERR_INVALID_ARG;
    if (ld < bt->max_seq_len || (ld % 4) != 0) return DSA_ERR_INVALID_ARG;
    return DSA_OK;
}

dsa_status check_mla_args(const dsa_batch* bt, const uint16_t* q_lat, const void* lat,
                          const int32_t* indices, int32_t topk, const uint16_t* out,
                          float kv_scale, float sm_scale) {
    (void)bt;
    if (topk != kTopK) return DSA_ERR_UNSUPPORTED;
    if (!q_lat || !lat || !indices || !out) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_lat) || !aligned16(lat) || !aligned16(indices) || !aligned16(out))
        return DSA_ERR_INVALID_ARG;
    if (!(kv_scale > 0.f) || !(sm_scale > 0.f)) return DSA_ERR_INVALID_ARG;
    return DSA_OK;
}

}  // namespace

extern "C" {

const char* dsa_status_string(dsa_status s) {
    switch (s) {
        case DSA_OK: return "ok";
        case DSA_ERR_INVALID_ARG: return "invalid argument";
        case DSA_ERR_UNSUPPORTED: return "unsupported shape or format";
        case DSA_ERR_WORKSPACE: return "workspace too small";
        case DSA_ERR_CUDA: return "CUDA error";
        case DSA_ERR_DEVICE_CHECK: return "device check failed (page id or position out of range)";
        case DSA_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

int32_t dsa_set_batch_invariant(int32_t enabled) {
    return g_batch_invariant.exchange(enabled != 0 ? 1 : 0);
}

uint64_t dsa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

dsa_status dsa_index_scores(const dsa_batch* batch, const uint8_t* q_fp8, const float* q_scale,
                            const float* w, const void* index_pages, dsa_key_format key_format,
                            float* scores, int64_t score_ld, int32_t* dev_status,
                            dsa_stream_t stream) {
    dsa_status st = check_batch(batch);
    if (st != DSA_OK) return st;
    st = check_index_args(batch, q_fp8, q_scale, w, index_pages, key_format, scores, score_ld);
    if (st != DSA_OK) return st;
    if (batch->total_q == 0) return DSA_OK;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(launch_index_scores(to_args(batch), q_fp8, q_scale, w, index_pages,
                                           (int)key_format, scores, score_ld, dev_status,
                                           (cudaStream_t)stream));
}

size_t dsa_topk_workspace_size(const dsa_batch* batch, int32_t topk) {
    if (check_batch(batch) != DSA_OK || topk != kTopK) return 0;
    return topk_workspace_bytes(batch->total_q, batch->max_seq_len);
}

dsa_status dsa_topk(const dsa_batch* batch, const float* scores, int64_t score_ld, int32_t topk,
                    int32_t* indices, void* ws, size_t ws_bytes, dsa_stream_t stream) {
    dsa_status st = check_batch(batch);
    if (st != DSA_OK) return st;
    if (topk != kTopK || !topk_supported(batch->max_seq_len)) return DSA_ERR_UNSUPPORTED;
    if (!scores || !indices) return DSA_ERR_INVALID_ARG;
    if (!aligned16(scores) || !aligned16(indices) || score_ld < batch->max_seq_len ||
        (score_ld % 4) != 0)
        return DSA_ERR_INVALID_ARG;
    const size_t need = dsa_topk_workspace_size(batch, topk);
    if (ws_bytes < need || (need > 0 && (!ws || !aligned16(ws)))) return DSA_ERR_WORKSPACE;
    if (batch->total_q == 0) return DSA_OK;
    g_launches.fetch_add((uint64_t)topk_launches(batch->total_q, batch->max_seq_len),
                         std::memory_order_relaxed);
    return cuda_status(launch_topk(to_args(batch), scores, score_ld, topk, indices, ws, false,
                                   (cudaStream_t)stream));
}

size_t dsa_sparse_mla_workspace_size(const dsa_batch* batch, int32_t topk) {
    if (check_batch(batch) != DSA_OK || topk != kTopK) return 0;
    return sparse_mla_workspace_bytes(batch->total_q, topk);
}

dsa_status dsa_sparse_mla(const dsa_batch* batch, const uint16_t* q_lat, const void* latent_pages,
                          float kv_scale, float sm_scale, const int32_t* indices, int32_t topk,
                          uint16_t* out, float* lse, void* ws, size_t ws_bytes,
                          int32_t* dev_status, dsa_stream_t stream) {
    return dsa_sparse_mla_ex(batch, q_lat, latent_pages, DSA_LATENT_FP8_E4M3, kv_scale, sm_scale,
                             indices, topk, out, lse, ws, ws_bytes, dev_status, stream);
}

dsa_status dsa_sparse_mla_ex(const dsa_batch* batch, const uint16_t* q_lat,
                             const void* latent_pages, dsa_latent_format latent_format,
                             float kv_scale, float sm_scale, const int32_t* indices, int32_t topk,
                             uint16_t* out, float* lse, void* ws, size_t ws_bytes,
                             int32_t* dev_status, dsa_stream_t stream) {
    if (latent_format != DSA_LATENT_FP8_E4M3 && latent_format != DSA_LATENT_NVFP4)
        return DSA_ERR_UNSUPPORTED;
    dsa_status st = check_batch(batch);
    if (st != DSA_OK) return st;
    st = check_mla_args(batch, q_lat, latent_pages, indices, topk, out, kv_scale, sm_scale);
    if (st != DSA_OK) return st;
    const size_t need = dsa_sparse_mla_workspace_size(batch, topk);
    if (ws_bytes < need || (need > 0 && (!ws || !aligned16(ws)))) return DSA_ERR_WORKSPACE;
    if (batch->total_q == 0) return DSA_OK;
    const bool whole_only = g_batch_invariant.load(std::memory_order_relaxed) != 0;
    g_launches.fetch_add((uint64_t)sparse_mla_launches(batch->total_q, topk, whole_only),
                         std::memory_order_relaxed);
    return cuda_status(launch_sparse_mla(to_args(batch), q_lat, latent_pages, kv_scale, sm_scale,
                                         indices, topk, out, lse, ws, dev_status, false,
                                         (cudaStream_t)stream, false, (int)latent_format,
                                         whole_only));
}

size_t dsa_decode_workspace_size(const dsa_batch* batch, int32_t topk) {
    if (check_batch(batch) != DSA_OK) return 0;
    size_t scores = align_up((size_t)batch->total_q * score_ld_for(batch) * sizeof(float), 256);
    return scores + align_up(dsa_topk_workspace_size(batch, topk), 256) +
           align_up(dsa_sparse_mla_workspace_size(batch, topk), 256);
}

dsa_status dsa_decode(const dsa_batch* batch, const uint8_t* q_fp8, const float* q_scale,
                      const float* w, const void* index_pages, dsa_key_format key_format,
                      const uint16_t* q_lat, const void* latent_pages, float kv_scale,
                      float sm_scale, int32_t topk, uint16_t* out, float* lse, int32_t* indices,
                      void* ws, size_t ws_bytes, int32_t* dev_status, dsa_stream_t stream) {
    return dsa_decode_ex(batch, q_fp8, q_scale, w, index_pages, key_format, q_lat, latent_pages,
                         DSA_LATENT_FP8_E4M3, kv_scale, sm_scale, topk, out, lse, indices, ws,
                         ws_bytes, dev_status, stream);
}

dsa_status dsa_decode_ex(const dsa_batch* batch, const uint8_t* q_fp8, const float* q_scale,
                         const float* w, const void* index_pages, dsa_key_format key_format,
                         const uint16_t* q_lat, const void* latent_pages,
                         dsa_latent_format latent_format, float kv_scale, float sm_scale,
                         int32_t topk, uint16_t* out, float* lse, int32_t* indices, void* ws,
                         size_t ws_bytes, int32_t* dev_status, dsa_stream_t stream) {
    if (latent_format != DSA_LATENT_FP8_E4M3 && latent_format != DSA_LATENT_NVFP4)
        return DSA_ERR_UNSUPPORTED;
    dsa_status st = check_batch(batch);
    if (st != DSA_OK) return st;
    const int64_t ld = score_ld_for(batch);
    float* scores = static_cast<float*>(ws);
    st = check_index_args(batch, q_fp8, q_scale, w, index_pages, key_format,
                          scores ? scores : reinterpret_cast<float*>(16), ld);
    if (st != DSA_OK) return st;
    st = check_mla_args(batch, q_lat, latent_pages, indices, topk, out, kv_scale, sm_scale);
    if (st != DSA_OK) return st;
    if (!topk_supported(batch->max_seq_len)) return DSA_ERR_UNSUPPORTED;
    if (!ws || !aligned16(ws) || ws_bytes < dsa_decode_workspace_size(batch, topk))
        return DSA_ERR_WORKSPACE;
    if (batch->total_q == 0) return DSA_OK;
    const BatchArgs a = to_args(batch);
    cudaStream_t s = (cudaStream_t)stream;
    uint8_t* base = static_cast<uint8_t*>(ws);
    const size_t off_topk = align_up((size_t)batch->total_q * ld * sizeof(float), 256);
    const size_t off_mla = off_topk + align_up(dsa_topk_workspace_size(batch, topk), 256);
    const bool whole_only = g_batch_invariant.load(std::memory_order_relaxed) != 0;
    g_launches.fetch_add(1 + (uint64_t)topk_launches(batch->total_q, batch->max_seq_len) +
                             (uint64_t)sparse_mla_launches(batch->total_q, topk, whole_only),
                         std::memory_order_relaxed);
    cudaError_t e = launch_index_scores(a, q_fp8, q_scale, w, index_pages, (int)key_format,
                                        scores, ld, dev_status, s);
    // the later kernels only read what the kernel before them writes after
    // their grid-dependency wait, so each may start while its predecessor runs
    if (e == cudaSuccess) e = launch_topk(a, scores, ld, topk, indices, base + off_topk, true, s);
    if (e == cudaSuccess)
        e = launch_sparse_mla(a, q_lat, latent_pages, kv_scale, sm_scale, indices, topk, out, lse,
                              base + off_mla, dev_status, true, s, false, (int)latent_format,
                              whole_only);
    return cuda_status(e);
}

size_t dsa_dcp_topk_workspace_size(const dsa_batch* batch, int32_t world, int32_t cand,
                                   int32_t topk) {
    if (check_batch(batch) != DSA_OK || topk != kTopK || world < 1 || world > 8) return 0;
    if (cand == 0) cand = dcp_default_cand(world, topk);
    if (cand < 1 || cand > topk) return 0;
    return dcp_ws_layout(batch->total_q, world, cand, topk).total;
}

dsa_status dsa_dcp_topk(const dsa_batch* batch, const float* scores, int64_t score_ld,
                        int32_t world, int32_t cand, int32_t topk, int32_t* indices,
                        int32_t* rank_indices, int32_t* resent, void* ws, size_t ws_bytes,
                        dsa_stream_t stream) {
    dsa_status st = check_batch(batch);
    if (st != DSA_OK) return st;
    if (topk != kTopK) return DSA_ERR_UNSUPPORTED;
    if (world < 1 || world > 8) return DSA_ERR_UNSUPPORTED;
    if (cand == 0) cand = dcp_default_cand(world, topk);
    if (cand < 1 || cand > topk) return DSA_ERR_INVALID_ARG;
    if (!dcp_supported(world, batch->max_seq_len)) return DSA_ERR_UNSUPPORTED;
    if (!scores || !indices || !aligned16(scores) || !aligned16(indices)) return DSA_ERR_INVALID_ARG;
    if ((rank_indices && !aligned16(rank_indices)) || (resent && !aligned16(resent)))
        return DSA_ERR_INVALID_ARG;
    if (score_ld < batch->max_seq_len || (score_ld % 4) != 0) return DSA_ERR_INVALID_ARG;
    const size_t need = dsa_dcp_topk_workspace_size(batch, world, cand, topk);
    if (!ws || !aligned16(ws) || ws_bytes < need) return DSA_ERR_WORKSPACE;
    if (batch->total_q == 0) return DSA_OK;
    g_launches.fetch_add(4, std::memory_order_relaxed);
    return cuda_status(launch_dcp_topk(to_args(batch), scores, score_ld, world, cand, topk,
                                       indices, rank_indices, resent, ws, (cudaStream_t)stream));
}

dsa_status dsa_lse_combine(int32_t total_q, int32_t world, const uint16_t* part_out,
                           const float* part_lse, uint16_t* out, float* lse,
                           dsa_stream_t stream) {
    if (total_q < 0) return DSA_ERR_INVALID_ARG;
    if (world < 1 || world > 8) return DSA_ERR_UNSUPPORTED;
    if (!part_out || !part_lse || !out || !aligned16(part_out) || !aligned16(out))
        return DSA_ERR_INVALID_ARG;
    if (total_q == 0) return DSA_OK;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(launch_lse_combine(total_q, world, part_out, part_lse, out, lse,
                                          (cudaStream_t)stream));
}

dsa_status dsa_indexer_front(const dsa_batch* batch, const uint16_t* q_c, const uint16_t* x,
                             const uint16_t* w_q, const uint16_t* w_k, const uint16_t* w_w,
                             uint8_t* q_fp8, float* q_scale, float* w, void* index_pages,
                             dsa_key_format key_format, float* q_f32, float* k_f32,
                             int32_t* dev_status, dsa_stream_t stream) {
    dsa_status st = check_batch(batch);
    if (st != DSA_OK) return st;
    if (index_pages && key_format != DSA_KEYS_FP8_E4M3) return DSA_ERR_UNSUPPORTED;
    if (!q_c || !x || !w_q || !w_k || !w_w || !q_fp8 || !q_scale || !w) return DSA_ERR_INVALID_ARG;
    const void* ptrs[] = {q_c, x, w_q, w_k, w_w, q_fp8, q_scale, w};
    for (const void* q : ptrs)
        if (!aligned16(q)) return DSA_ERR_INVALID_ARG;
    if ((index_pages && !aligned16(index_pages)) || (q_f32 && !aligned16(q_f32)) ||
        (k_f32 && !aligned16(k_f32)))
        return DSA_ERR_INVALID_ARG;
    if (batch->total_q == 0) return DSA_OK;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(launch_indexer_front(to_args(batch), q_c, x, w_q, w_k, w_w, q_fp8, q_scale,
                                            w, index_pages, q_f32, k_f32, dev_status,
                                            (cudaStream_t)stream));
}

dsa_status dsa_test_sparse_mla_wait_timeout(const dsa_batch* batch, const uint16_t* q_lat,
                                           const void* latent_pages, float kv_scale,
                                           float sm_scale, const int32_t* indices, int32_t topk,
                                           uint16_t* out, float* lse, void* ws, size_t ws_bytes,
                                           int32_t* dev_status, dsa_stream_t stream) {
    dsa_status st = check_batch(batch);
    if (st != DSA_OK) return st;
    st = check_mla_args(batch, q_lat, latent_pages, indices, topk, out, kv_scale, sm_scale);
    if (st != DSA_OK) return st;
    const size_t need = dsa_sparse_mla_workspace_size(batch, topk);
    if (ws_bytes < need || (need > 0 && (!ws || !aligned16(ws)))) return DSA_ERR_WORKSPACE;
    if (batch->total_q == 0) return DSA_OK;
    g_launches.fetch_add((uint64_t)sparse_mla_launches(batch->total_q, topk, false),
                         std::memory_order_relaxed);
    return cuda_status(launch_sparse_mla(to_args(batch), q_lat, latent_pages, kv_scale, sm_scale,
                                         indices, topk, out, lse, ws, dev_status, false,
                                         (cudaStream_t)stream, true, DSA_LATENT_FP8_E4M3, false));
}

dsa_status dsa_append_cache(const dsa_batch* batch, const float* new_keys,
                            const float* new_latent, float kv_scale, void* index_pages,
                            void* latent_pages, dsa_key_format key_format, int32_t* dev_status,
                            dsa_stream_t stream) {
    dsa_status st = check_batch(batch);
    if (st != DSA_OK) return st;
    if (new_keys && key_format != DSA_KEYS_FP8_E4M3) return DSA_ERR_UNSUPPORTED;
    if ((new_keys && !index_pages) || (new_latent && !latent_pages)) return DSA_ERR_INVALID_ARG;
    if ((new_keys && (!aligned16(new_keys) || !aligned16(index_pages))) ||
        (new_latent && (!aligned16(new_latent) || !aligned16(latent_pages))))
        return DSA_ERR_INVALID_ARG;
    if (new_latent && !(kv_scale > 0.f)) return DSA_ERR_INVALID_ARG;
    if (batch->total_q == 0 || (!new_keys && !new_latent)) return DSA_OK;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(launch_append_cache(to_args(batch), new_keys, new_latent, kv_scale,
                                           index_pages, latent_pages, dev_status,
                                           (cudaStream_t)stream));
}

}  // extern "C"
