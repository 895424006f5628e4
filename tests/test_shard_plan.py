"""Token-sharded prefill planner ("Token-sharded prefill improves time to
first token": each request cut into 16 parts, GPU r of 8 takes parts r and
15 - r).  Host-only checks: every new token is planned exactly once, each
part's context makes the step's causal rule give its tokens the positions
they see in the whole request, and the causal work of the ranks balances."""
import pytest

import dsa_sparse_attention_step_gb300 as dsa


@pytest.fixture(scope="module", autouse=True)
def lib():
    from dsa_sparse_attention_step_gb300 import _build
    _build.build()
    dsa.load()


def _positions(part, q_counts, seq_lens):
    """Positions of the part's tokens, through the sub-request's causal rule."""
    return [part.seq_len - part.num_tokens + j for j in range(part.num_tokens)]


def _plan(seq_lens, q_counts, world):
    return [dsa.dsa_plan_token_shards(seq_lens, q_counts, world, r) for r in range(world)]


def test_eight_ranks_take_parts_r_and_15_minus_r():
    # one request of 2048 new tokens after a 153,600-token prefix: 16 parts of 128
    plans = _plan([153600 + 2048], [2048], 8)
    for r, parts in enumerate(plans):
        assert [p.token_begin for p in parts] == [128 * r, 128 * (15 - r)]
        assert all(p.num_tokens == 128 for p in parts)
        assert [p.seq_len for p in parts] == [153600 + 128 * (r + 1), 153600 + 128 * (16 - r)]


@pytest.mark.parametrize("seq_lens,q_counts,world", [
    ([153600 + 2048], [2048], 8),
    ([5000, 777, 300, 40], [1000, 777, 17, 3], 8),
    ([100, 9000], [100, 4001], 3),
    ([64] * 5, [1, 2, 3, 4, 5], 2),
])
def test_every_token_once_with_its_own_causal_positions(seq_lens, q_counts, world):
    starts = [sum(q_counts[:b]) for b in range(len(q_counts))]
    seen = {}
    for r, parts in enumerate(_plan(seq_lens, q_counts, world)):
        assert len(parts) <= 2 * len(seq_lens)
        for p in parts:
            b = p.request
            assert p.num_tokens > 0
            for j, pos in enumerate(_positions(p, q_counts, seq_lens)):
                t = p.token_begin + j
                assert starts[b] <= t < starts[b] + q_counts[b]
                # position of token t in the unsharded request
                assert pos == seq_lens[b] - q_counts[b] + (t - starts[b])
                assert t not in seen
                seen[t] = r
    assert sorted(seen) == list(range(sum(q_counts)))


def _indexer_work(parts):
    """Keys scored: token at position p sees p + 1 keys."""
    w = 0
    for p in parts:
        first = p.seq_len - p.num_tokens
        w += sum(first + j + 1 for j in range(p.num_tokens))
    return w


def _mla_work(parts):
    """Latents attended: min(2048, visible) per token."""
    return sum(min(2048, p.seq_len - p.num_tokens + j + 1)
               for p in parts for j in range(p.num_tokens))


def test_causal_work_is_balanced():
    # divisible: every rank does exactly the same indexer work
    plans = _plan([153600 + 2048], [2048], 8)
    work = [_indexer_work(p) for p in plans]
    assert len(set(work)) == 1
    # a plain prefill from position 0 (the most skewed causal triangle):
    # pairing part r with 15 - r balances it, contiguous eighths do not
    n = 16384
    plans = _plan([n], [n], 8)
    work = [_indexer_work(p) for p in plans]
    assert len(set(work)) == 1
    naive = [sum(range(r * n // 8 + 1, (r + 1) * n // 8 + 1)) for r in range(8)]
    assert max(naive) / min(naive) > 10
    # ragged: parts differ by at most one token
    plans = _plan([10007], [10007], 8)
    work = [_indexer_work(p) for p in plans]
    assert (max(work) - min(work)) / max(work) < 2e-3
    # sparse MLA attends min(2048, visible) latents per token: once the prefix
    # holds 2048 tokens that is constant, and equal part sizes balance it
    plans = _plan([153600 + 2048], [2048], 8)
    assert len({_mla_work(p) for p in plans}) == 1


def test_bad_arguments():
    with pytest.raises(dsa.DsaError):
        dsa.dsa_plan_token_shards([10], [11], 8, 0)  # more new tokens than context
    with pytest.raises(dsa.DsaError):
        dsa.dsa_plan_token_shards([10], [5], 8, 8)   # rank out of range


def _rank_plan(rank, world, port, out):
    import os
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dsa.load()
        parts = dsa.dsa_plan_token_shards([153600 + 2048, 4000], [2048, 100], world, rank)
        mine = torch.tensor([t for p in parts
                             for t in range(p.token_begin, p.token_begin + p.num_tokens)])
        n = torch.tensor([mine.numel()])
        sizes = [torch.zeros(1, dtype=torch.long) for _ in range(world)]
        dist.all_gather(sizes, n)
        buf = [torch.zeros(int(s.item()), dtype=torch.long) for s in sizes]
        dist.all_gather(buf, mine.long())
        out[rank] = sorted(torch.cat(buf).tolist())
    finally:
        dist.destroy_process_group()


def test_two_ranks_cover_the_batch_once():
    """Each of two gloo ranks plans its own share; gathered, the shares are
    the batch's tokens exactly once."""
    import socket
    import torch.multiprocessing as mp
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank_plan, args=(2, port, out), nprocs=2, start_method="spawn",
                       join=True)
    assert out[0] == out[1] == list(range(2148))
