"""dsa_topk on crafted score matrices (independent of the indexer), bit-exact
against the oracle's selection on the same fp32 scores: heavy ties, signed
zeros, negative scores, rows of every length class, and batches that take
each path: rows kept in shared memory (up to 32768 positions), rows split over
the whole GPU (at most 8 query tokens), many rows of up to 2^18 positions
(sampled threshold, candidate pass, per-row select) and one cluster per row
(more tokens over longer rows), including inputs that force the exact
fallbacks."""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_step_gb300 as dsa
import oracle

pytestmark = pytest.mark.gpu


def _batch(seq_lens, q_counts):
    dev = "cuda:0"
    off = [0]
    for n in q_counts:
        off.append(off[-1] + n)
    max_pages = (max(seq_lens) + 63) // 64
    return dsa.Batch(torch.tensor(off, dtype=torch.int32, device=dev),
                     torch.tensor(seq_lens, dtype=torch.int32, device=dev),
                     torch.zeros(len(seq_lens), max_pages, dtype=torch.int32, device=dev), 1,
                     seq_lens, q_counts)


def _visible(seq_lens, q_counts):
    vis = []
    for s, n in zip(seq_lens, q_counts):
        vis += [s - n + j + 1 for j in range(n)]
    return np.array(vis, np.int64)


def _run(seq_lens, q_counts, scores):
    b = _batch(seq_lens, q_counts)
    ld = scores.shape[1]
    S = torch.from_numpy(scores.astype(np.float32)).cuda()
    idx = torch.full((b.total_q, dsa.TOPK), -7, dtype=torch.int32, device="cuda:0")
    nws = dsa.dsa_topk_workspace_size(b)
    ws = torch.full((max(nws, 16),), 0xA5, dtype=torch.uint8, device="cuda:0")  # not zero
    dsa.dsa_topk(b, S, ld, dsa.TOPK, idx, ws if nws else None)
    torch.cuda.synchronize()
    want = oracle.topk(scores.astype(np.float32).astype(np.float64),
                       _visible(seq_lens, q_counts), dsa.TOPK)
    got = idx.cpu().numpy()
    for r in range(got.shape[0]):
        assert np.array_equal(got[r], want[r]), "row %d" % r


def _scores(rng, T, ld, kind):
    if kind == "normal":
        return rng.standard_normal((T, ld))
    if kind == "few_levels":          # heavy ties everywhere
        return rng.integers(-3, 4, size=(T, ld)).astype(np.float64) * 0.5
    if kind == "signed_zero":         # +0 / -0 and a few positives
        s = np.where(rng.random((T, ld)) < 0.5, 0.0, -0.0)
        s[rng.random((T, ld)) < 0.01] = 1.0
        return s
    if kind == "offset":              # narrow band far from zero (one first-digit bin)
        return 1000.0 + rng.random((T, ld)) * 1e-3
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["normal", "few_levels", "signed_zero", "offset"])
@pytest.mark.parametrize("shape", [([30000, 2049, 4096], [1, 1, 2]),     # resident rows
                                   ([131072], [1]),                      # one long row: split
                                   ([40000] * 5, [2] * 5),               # 10 tokens: many rows
                                   ([300000, 40000], [6, 4]),            # 10 tokens: clusters
                                   ([9000] * 40, [2] * 40),              # 80 short rows: one CTA each
                                   ([32768, 17000] * 9, [1] * 18)])      # 18 short rows: one CTA each
def test_topk_crafted(kind, shape):
    lens, counts = shape
    rng = np.random.default_rng(len(lens) * 7 + sum(counts))
    T = sum(counts)
    ld = ((max(lens) + 127) // 128) * 128
    _run(lens, counts, _scores(rng, T, ld, kind))


@pytest.mark.parametrize("lens,counts", [([70000, 300000], [1, 1]),   # split rows
                                         ([70000, 262144], [5, 5]),   # many rows
                                         ([70000, 300000], [5, 5])])  # clusters
def test_topk_all_equal_long_rows(lens, counts):
    # every key equals tau: split rows take the lowest positions across their
    # slices; on the other paths the threshold holds far more keys than the
    # candidate buffers, and the exact fallback selects by position
    ld = ((max(lens) + 127) // 128) * 128
    _run(lens, counts, np.full((sum(counts), ld), 2.5))


@pytest.mark.parametrize("lens", [[131072, 200000],    # 10 tokens: many rows
                                  [131072, 300000]])   # 10 tokens: one cluster per row
def test_topk_sample_misses_the_top(lens):
    """The large scores sit exactly in the sampled chunks (every 16th run of 32
    positions), so the sampled threshold is far too high: the candidate pass
    finds fewer than k keys and the exact fallback must take over."""
    counts = [5, 5]
    ld = ((max(lens) + 127) // 128) * 128
    rng = np.random.default_rng(5)
    s = rng.standard_normal((10, ld))
    pos = np.arange(ld)
    s[:, (pos // 32) % 16 == 0] += 100.0
    _run(lens, counts, s)


@pytest.mark.parametrize("kind", ["normal", "few_levels", "signed_zero", "offset"])
def test_topk_many_rows_ragged(kind):
    """Many-rows path: rows at and below k (all visible positions, then -1),
    a row of exactly 2^18 positions, ragged unit ends, causal multi-token
    requests; the workspace starts filled with garbage."""
    lens, counts = [40000, 1000, 2049, 262144, 33001], [3, 1, 1, 3, 2]
    rng = np.random.default_rng(31)
    ld = ((max(lens) + 127) // 128) * 128
    _run(lens, counts, _scores(rng, sum(counts), ld, kind))


def test_topk_many_rows_ties_within_the_candidates():
    """3,000 copies of one value near the 2048th largest score of each row:
    tau is that value, the candidates hold every copy, and the lowest
    positions among them are found by the select over positions."""
    lens, counts = [131072] * 4, [3] * 4
    rng = np.random.default_rng(17)
    T = sum(counts)
    s = rng.standard_normal((T, lens[0]))
    for r in range(T):
        s[r, rng.choice(lens[0], 3000, replace=False)] = 2.3
    _run(lens, counts, s)


def test_topk_many_rows_overflow():
    """A sample that draws low: the large scores sit outside the sampled
    chunks, so every row holds more candidates than its list keeps and the
    exact fallback over the row takes over."""
    lens, counts = [100000] * 5, [2] * 5
    rng = np.random.default_rng(19)
    s = rng.standard_normal((10, lens[0]))
    pos = np.arange(lens[0])
    s[:, (pos // 32) % 16 != 0] += 100.0
    _run(lens, counts, s)


def test_topk_one_million_positions():
    rng = np.random.default_rng(11)
    lens = [1 << 20]
    _run(lens, [1], rng.standard_normal((1, 1 << 20)))


@pytest.mark.parametrize("kind", ["equal", "normal", "few_levels"])
def test_topk_resident_row_limits(kind):
    """Rows at the resident-path size limit (32768 positions, where the packed
    counts of equal keys reach 2^15) next to rows at and just above k."""
    lens, counts = [32768, 2049, 2048, 1], [1, 1, 1, 1]
    ld = 32768
    rng = np.random.default_rng(3)
    if kind == "equal":
        s = np.full((4, ld), -1.25)
    else:
        s = _scores(rng, 4, ld, kind)
    _run(lens, counts, s)


@pytest.mark.parametrize("kind", ["normal", "few_levels", "signed_zero", "offset"])
def test_topk_split_rows(kind):
    """At most 8 query tokens with a row above 32768 positions: every row is
    split over the GPU.  Rows at and below k (all visible positions, then -1),
    ragged slice ends, and multi-token requests (causal visibility) in one
    batch; the workspace starts filled with garbage."""
    lens, counts = [33000, 1000, 70001, 2049, 500000], [1, 1, 3, 1, 2]
    rng = np.random.default_rng(21)
    ld = ((max(lens) + 127) // 128) * 128
    _run(lens, counts, _scores(rng, sum(counts), ld, kind))


def test_topk_split_ties_at_the_threshold():
    """Many keys equal to tau spread over every slice: the lowest positions are
    taken across slice boundaries."""
    lens, counts = [262144], [1]
    rng = np.random.default_rng(8)
    s = rng.standard_normal((1, lens[0]))
    s[0, rng.random(lens[0]) < 0.05] = 1.5  # ~13,000 copies of one value
    s[0, :100] = 9.0
    _run(lens, counts, s)


def test_topk_split_ties_within_the_list():
    """3,000 copies of 2.5 spread over the slices of a 262,144-position row:
    the threshold bin (about 3,800 keys) fits the candidate list, so tau and
    the lowest 428-or-so equal positions come from the list itself."""
    lens, counts = [262144], [1]
    rng = np.random.default_rng(13)
    s = rng.standard_normal((1, lens[0]))
    s[0, rng.choice(lens[0], 3000, replace=False)] = 2.5
    _run(lens, counts, s)
