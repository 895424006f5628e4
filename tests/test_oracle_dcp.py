"""Pins of the oracle's decode-context-parallelism functions ("vLLM's Kimi
K3.1 Pro day-0 support", sections "Decode context parallelism with the sparse
indexer" and "Exact top-k merge with about 10x less traffic").

- bf16_encode against PyTorch's own float -> bfloat16 rounding;
- the merged selection against a brute-force sort of PyTorch-rounded scores;
- the resend decision against an independent simulation of the protocol
  written here (candidates, gathered top-k, detection), and the exactness claim
  itself: after the detected ranks resend, the top-k of what was gathered is
  the global top-k, on random and on skewed inputs;
- the LSE combine against the oracle's own sparse MLA: attention over a union
  of disjoint token sets equals the combine of the attention over each set."""
import numpy as np
import pytest
import torch

import dsa_inputs as di
import oracle
from oracle_helpers import batch_of


def _bf16_values(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def test_bf16_encode_matches_pytorch():
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 10 ** rng.uniform(-30, 30, 20000).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.3895e38, -3.3895e38, 1e-40, -1e-40,
                  1.00390625, 1.01171875, 1.0078125, 65504.0], np.float32)])
    # ties to even: 1 + 2^-8 is halfway between 1 and 1 + 2^-7
    x = np.concatenate([x, np.float32(1.0) + np.float32(2.0 ** -8) * np.arange(1, 9, dtype=np.float32)])
    got = oracle.bf16_encode(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def _global_topk(scores, n, k):
    v = _bf16_values(scores[:n])
    order = sorted(range(n), key=lambda s: (-v[s], s))
    sel = sorted(order[:k])
    return np.array(sel + [-1] * (k - len(sel)), np.int32), order


def _simulate(scores, n, world, cand, k):
    """The protocol, step by step (independent of the oracle's code)."""
    v = _bf16_values(scores[:n])
    key = lambda s: (-v[s], s)
    local = {r: sorted(range(r, n, world), key=key) for r in range(world)}
    sent = {r: local[r][:cand] for r in range(world)}
    gathered = sorted([s for r in range(world) for s in sent[r]], key=key)
    top = set(gathered[:k])
    resend = [int(len(sent[r]) > 0 and all(s in top for s in sent[r]) and len(local[r]) > len(sent[r]))
              for r in range(world)]
    # second round: flagged ranks send their full local top-k
    pool = [s for r in range(world) for s in (local[r][:k] if resend[r] else sent[r])]
    merged = sorted(sorted(pool, key=key)[:k])
    return np.array(merged + [-1] * (k - len(merged)), np.int32), np.array(resend, np.int32)


@pytest.mark.parametrize("world,k,cand,n", [(8, 64, 12, 900), (4, 64, 24, 300), (8, 64, 12, 50),
                                            (3, 32, 16, 5000), (1, 64, 96, 400), (8, 64, 12, 64)])
def test_merge_and_resend_against_simulation(world, k, cand, n):
    rng = np.random.default_rng(world * 1000 + n)
    for trial in range(4):
        if trial == 0:      # random
            s = rng.standard_normal(n).astype(np.float32)
        elif trial == 1:    # heavy BF16 ties
            s = np.round(rng.standard_normal(n) * 4).astype(np.float32) / 4
        elif trial == 2:    # skew: rank 1's tokens score high
            s = rng.standard_normal(n).astype(np.float32)
            s[1 % world::world] += 8.0
        else:               # values that round together in BF16 only
            s = (1.0 + rng.integers(0, 64, n) * 2.0 ** -10).astype(np.float32)
        got, resend = oracle.dcp_topk(s, n, world, cand, k)
        want, want_resend = _simulate(s, n, world, cand, k)
        glob, _ = _global_topk(s, n, k)
        assert np.array_equal(got[0], glob)          # the oracle's definition
        assert np.array_equal(want, glob)            # the protocol reaches it
        assert np.array_equal(resend[0], want_resend)


def test_skewed_rank_is_detected():
    world, k, cand = 8, 2048, oracle.dcp_cand(8)
    assert cand == 384
    n = 40000
    s = np.random.default_rng(1).standard_normal(n).astype(np.float32)
    s[3::world] += 20.0   # rank 3 holds every one of the top 2048
    _, resend = oracle.dcp_topk(s, n, world, None, k)
    assert resend[0].tolist() == [0, 0, 0, 1, 0, 0, 0, 0]
    # spread evenly: nobody has more winners than it sent
    s = np.random.default_rng(2).standard_normal(n).astype(np.float32)
    _, resend = oracle.dcp_topk(s, n, world, None, k)
    assert resend[0].sum() == 0
    # every visible token fits in the candidates: nothing to resend
    _, resend = oracle.dcp_topk(s, 1000, world, None, k)
    assert resend[0].sum() == 0


def test_all_equal_scores_pick_the_lowest_positions():
    n, k = 5000, 2048
    got, resend = oracle.dcp_topk(np.full(n, 0.5, np.float32), n, 8, None, k)
    assert got[0].tolist() == list(range(k))
    assert resend[0].sum() == 0   # each rank holds 256 winners, below its 384


def test_lse_combine_equals_attention_over_the_union():
    layer = di.make_layer([3000], [1], seed=9)
    b = batch_of(layer)
    rng = np.random.default_rng(3)
    sel = np.sort(rng.choice(3000, 700, replace=False)).astype(np.int32)
    full = np.full((1, 2048), -1, np.int32)
    full[0, :sel.size] = sel
    ref_out, ref_lse = oracle.sparse_mla(b, layer.q_lat, layer.latent_pages, layer.kv_scale,
                                         layer.sm_scale, full)
    world = 8
    parts, lses = [], []
    for r in range(world + 1):   # one extra rank with no tokens at all
        mine = sel[sel % world == r] if r < world else sel[:0]
        idx = np.full((1, 2048), -1, np.int32)
        idx[0, :mine.size] = mine
        o, l = oracle.sparse_mla(b, layer.q_lat, layer.latent_pages, layer.kv_scale,
                                 layer.sm_scale, idx)
        parts.append(o)
        lses.append(l)
    out, lse = oracle.lse_combine(np.stack(parts), np.stack(lses))
    assert np.abs(out - ref_out).max() <= 1e-12 * max(1.0, np.abs(ref_out).max())
    assert np.abs(lse - ref_lse).max() <= 1e-12
    # nothing anywhere: zero output, -inf lse
    o, l = oracle.lse_combine(np.zeros((2, 3, 4)), np.full((2, 3), -np.inf))
    assert (o == 0).all() and np.isneginf(l).all()
