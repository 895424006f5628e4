// shard_plan.cu -- host-side planner of token-sharded prefill.
//
// "vLLM's Kimi K3.1 Pro day-0 support", section "Token-sharded prefill
// improves time to first token": for a large prefill step the attention is
// sharded by query token instead of by head; to balance causal attention each
// request is cut into 16 parts and GPU r of 8 takes parts r and 15 - r (the
// split prefill context parallelism uses).  Generalised here to W ranks and
// 2W parts: rank r takes parts r and 2W - 1 - r.
//
// A part is a contiguous run of a request's new tokens.  It is emitted as a
// sub-request of its own whose context ends at its last token, so the causal
// rule of the step (token j of a request with n tokens and context s sees
// positions 0 .. s - n + j) gives each of its tokens exactly the positions it
// sees in the whole request.  Runs only on the host; launches nothing.
#include <cstdint>

#include "../../include/dsa.h"

extern "C" int32_t dsa_plan_token_shards(const int32_t* seq_lens, const int32_t* q_counts,
                                         int32_t num_requests, int32_t world, int32_t rank,
                                         dsa_shard_part* parts, int32_t max_parts) {
    if (!seq_lens || !q_counts || num_requests < 1 || world < 1 || rank < 0 || rank >= world ||
        max_parts < 0 || (max_parts > 0 && !parts))
        return -(int32_t)DSA_ERR_INVALID_ARG;
    const int64_t nparts = 2 * (int64_t)world;
    int64_t token0 = 0;  // first token of request b in the batch
    int32_t out = 0;
    for (int32_t b = 0; b < num_requests; ++b) {
        const int64_t n = q_counts[b], s = seq_lens[b];
        if (n < 0 || s < n || token0 + n > INT32_MAX) return -(int32_t)DSA_ERR_INVALID_ARG;
        const int64_t mine[2] = {rank, nparts - 1 - rank};
        for (int k = 0; k < 2; ++k) {
            // part i = tokens [floor(i n / P), floor((i + 1) n / P)) of the request
            const int64_t lo = mine[k] * n / nparts, hi = (mine[k] + 1) * n / nparts;
            if (hi <= lo) continue;
            if (out >= max_parts) return -(int32_t)DSA_ERR_WORKSPACE;
            dsa_shard_part& p = parts[out++];
            p.request = b;
            p.token_begin = (int32_t)(token0 + lo);
            p.num_tokens = (int32_t)(hi - lo);
            p.seq_len = (int32_t)(s - n + hi);  // position of the part's last token + 1
        }
        token0 += n;
    }
    return out;
}
