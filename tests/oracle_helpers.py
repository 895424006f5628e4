"""Test-side helpers that read the synthetic caches back with PyTorch's own
float8 / bfloat16 conversions (independent of the oracle's decoders), so that
library routines can serve as pins."""
import numpy as np
import torch

import dsa_inputs as di
import oracle


def batch_of(layer):
    return oracle.Batch(layer.q_offsets, layer.seq_lens, layer.block_table, layer.num_pages)


def fp8(t):
    return t.view(torch.float8_e4m3fn).to(torch.float64)


def dense_keys(layer, b):
    """Dequantised FP8 index keys of request b, [seq_len, 128] float64."""
    assert layer.key_format == di.KEYS_FP8
    n = layer.seq_lens_host[b]
    pages = layer.block_table[b, :(n + 63) // 64].long()
    raw = layer.index_pages[pages]                       # [p, 8448]
    vals = fp8(raw[:, :64 * 128].contiguous()).view(-1, 128)
    scales = raw[:, 64 * 128:].contiguous().view(torch.float32).to(torch.float64).view(-1, 1)
    return (vals * scales)[:n]


def dense_latents(layer, b):
    """Dequantised latents of request b, [seq_len, 576] float64."""
    n = layer.seq_lens_host[b]
    pages = layer.block_table[b, :(n + 63) // 64].long()
    raw = layer.latent_pages[pages].contiguous().view(-1, 576)
    return (fp8(raw) * float(layer.kv_scale))[:n]


def dense_q(layer, t):
    """Dequantised indexer query of token t, [32, 128] float64."""
    return fp8(layer.q8[t].contiguous()) * layer.qscale[t].to(torch.float64).view(32, 1)


def request_of(layer, t):
    off = layer.q_offsets.tolist()
    for b in range(layer.num_requests):
        if off[b] <= t < off[b + 1]:
            return b, t - off[b]
    raise IndexError(t)


def visible(layer, t):
    b, j = request_of(layer, t)
    return layer.seq_lens_host[b] - layer.q_counts_host[b] + j + 1


def oracle_scores(layer, rows=None, ld=None):
    return oracle.index_scores(batch_of(layer), layer.q8, layer.qscale, layer.w,
                               layer.index_pages, layer.key_format, rows=rows, ld=ld)


def remap_pages(layer, seed):
    """The same logical caches on a different physical page placement."""
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(layer.num_pages, generator=g)        # old -> new
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(layer.num_pages)
    bt = layer.block_table.clone()
    m = bt >= 0
    bt[m] = perm[bt[m].long()].to(torch.int32)
    d = dict(layer.__dict__)
    d["block_table"] = bt
    d["index_pages"] = layer.index_pages[inv]
    d["latent_pages"] = layer.latent_pages[inv]
    return di.Layer(**d)


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))
