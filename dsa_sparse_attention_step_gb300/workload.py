"""Algorithmic byte and flop counts of the DSA step (host-side arithmetic for
roofline reporting; no device work).

Per request per layer the step reads the index keys of every context token
(132 B FP8 or 68 B MXFP4) and the 576-byte latents of the 2048 selected tokens
("vLLM's Kimi K3.1 Pro day-0 support", section "Sparse attention cuts
long-context decode bandwidth"), plus the query tensors of its tokens.
Outputs and the score scratch are not counted.
"""
KEY_BYTES = {0: 132, 1: 68}          # per token: FP8 (128 E4M3 + fp32), MXFP4 (64 + 4)
LATENT_BYTES = 576                   # per token, FP8
TOPK = 2048
# per query token: q8 [32x128] + q_scale [32] fp32 + w [32] fp32 + q_lat [96x576] bf16
QUERY_BYTES_INDEXER = 32 * 128 + 32 * 4 + 32 * 4
QUERY_BYTES_MLA = 96 * 576 * 2
OUT_BYTES = 96 * 512 * 2 + TOPK * 4  # bf16 output + int32 indices per query token


def step_bytes(seq_lens, q_counts, key_format=0, latent_per_token=False):
    """Bytes of one layer step: sum_b (key_bytes * ctx_b + 2048 * 576) + query
    bytes.  With latent_per_token, the latent term is counted once per query
    token (each token gathers its own selection) instead of once per request."""
    kb = KEY_BYTES[key_format]
    total = 0
    for s, n in zip(seq_lens, q_counts):
        sel = min(TOPK, s)
        lat = sel * LATENT_BYTES * (n if latent_per_token else 1)
        total += kb * s + lat + n * (QUERY_BYTES_INDEXER + QUERY_BYTES_MLA)
    return total


def indexer_bytes(seq_lens, q_counts, key_format=0):
    """Bytes the indexer kernel must read: every key once, plus its queries."""
    kb = KEY_BYTES[key_format]
    return sum(kb * s + n * QUERY_BYTES_INDEXER for s, n in zip(seq_lens, q_counts))


def topk_bytes(seq_lens, q_counts):
    """Scores read by the selection (fp32 per visible position)."""
    tot = 0
    for s, n in zip(seq_lens, q_counts):
        for j in range(n):
            tot += 4 * (s - n + j + 1)
    return tot


def mla_bytes(seq_lens, q_counts, latent_bytes=LATENT_BYTES):
    """Latents of each query token's selection plus its MLA query (latent_bytes
    per key: 576 FP8, 352 NVFP4)."""
    tot = 0
    for s, n in zip(seq_lens, q_counts):
        for j in range(n):
            vis = s - n + j + 1
            tot += min(TOPK, vis) * latent_bytes + QUERY_BYTES_MLA
    return tot


NVFP4_LATENT_BYTES = 352
FRONT_QLAT, FRONT_HIDDEN = 1536, 7168


def front_bytes(T):
    """Fused indexer front: the projections (bf16) once, each token's query
    latent and hidden state (bf16), and its outputs (q8, q_scale, w, key)."""
    weights = 2 * (4096 * FRONT_QLAT + (128 + 32) * FRONT_HIDDEN)
    return weights + T * (2 * (FRONT_QLAT + FRONT_HIDDEN) + 4096 + 4 * 32 + 4 * 32 + 132)


def front_flops(T):
    return 2 * T * (4096 * FRONT_QLAT + (128 + 32) * FRONT_HIDDEN)


def dcp_exchange_bytes(world, cand, k=TOPK):
    """Bytes one row puts on the wire in the candidate exchange (32-bit words
    from every rank) and in a merge of every rank's full top-k as fp32 score +
    int32 id pairs."""
    return world * cand * 4, world * k * 8


def indexer_flops(seq_lens, q_counts):
    """2 * 32 heads * 128 dims per visible (query, key) pair."""
    tot = 0
    for s, n in zip(seq_lens, q_counts):
        for j in range(n):
            tot += 2 * 32 * 128 * (s - n + j + 1)
    return tot


def mla_flops(seq_lens, q_counts):
    """2 * 96 heads * (576 + 512) per selected (query, key) pair."""
    tot = 0
    for s, n in zip(seq_lens, q_counts):
        for j in range(n):
            tot += 2 * 96 * (576 + 512) * min(TOPK, s - n + j + 1)
    return tot


def dense_mla_bytes(ctx):
    """What dense MLA reads per request per layer: every latent."""
    return LATENT_BYTES * ctx
