"""GPU parity of every C-ABI entry point against the CPU oracle, on seeded
inputs that span several tiles and ragged tails, plus the edge cases: a
single token, page and tile boundaries, contexts at and around 2048,
multi-token causal rows, query groups of up to 9 tokens, MXFP4 keys, page
placement, batch invariance, determinism and device-side range checks."""
import zlib

import numpy as np
import pytest
import torch

import dsa_inputs as di
import dsa_sparse_attention_step_gb300 as dsa
import oracle
from gpu_helpers import (GpuLayer, check_out, check_scores, check_topk_against_oracle,
                         check_topk_against_scores)
from oracle_helpers import batch_of, remap_pages

pytestmark = pytest.mark.gpu

CASES = {
    "ctx1": ([1], 1, di.KEYS_FP8),
    "page_edges": ([63, 64, 65, 127, 128, 129], 1, di.KEYS_FP8),
    "around_topk": ([2047, 2048, 2049, 4096], 1, di.KEYS_FP8),
    "multi_token": ([5000, 2300, 40], [5, 3, 2], di.KEYS_FP8),
    "ragged_batch": ([9000, 3001, 130, 7777], [1, 2, 1, 4], di.KEYS_FP8),
    "mxfp4": ([2047, 6000, 300], [1, 3, 1], di.KEYS_MXFP4),
    # query groups of 6, 7 and 8 tokens (two TMEM accumulators, N >= 192) and
    # a request split into a group of 8 and a group of 1
    "wide_groups": ([3000, 2600, 1200, 5000], [6, 7, 8, 9], di.KEYS_FP8),
    # groups of 6 (token halves of 3 + 3) and of 7 (4 + 3), with short groups
    "groups_of_6": ([2500, 1400], [6, 5], di.KEYS_FP8),
    "groups_of_7": ([2200, 3100, 900], [7, 3, 1], di.KEYS_FP8),
    # groups of at most two tokens: two producer and two MMA threads taking
    # alternate units (odd unit counts per CTA, a request boundary mid-range)
    "two_token": ([5000, 2049, 700, 9001], [2, 1, 2, 2], di.KEYS_FP8),
}


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    lens, nq, fmt = CASES[request.param]
    layer = di.make_layer(lens, nq, fmt, seed=zlib.crc32(request.param.encode()) % 10000, extra_pages=3)
    return layer, GpuLayer(layer)


def test_index_scores(case):
    layer, gl = case
    st = gl.status()
    S = gl.scores(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    check_scores(layer, S)


def test_topk_exact(case):
    layer, gl = case
    S_gpu = gl.scores()
    idx = gl.topk(S_gpu)
    rows = list(range(layer.total_q))
    vis = batch_of(layer).visible(rows)
    check_topk_against_scores(idx, S_gpu, vis, rows)
    S, A, _ = check_scores(layer, S_gpu)
    check_topk_against_oracle(idx, S, A, vis, rows)


def test_sparse_mla(case):
    layer, gl = case
    S_gpu = gl.scores()
    idx = gl.topk(S_gpu)
    st = gl.status()
    out, lse = gl.mla(idx, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_out, ref_lse = oracle.sparse_mla(batch_of(layer), layer.q_lat, layer.latent_pages,
                                         layer.kv_scale, layer.sm_scale, idx.cpu().numpy())
    check_out(out, lse, ref_out, ref_lse, list(range(layer.total_q)))


def test_decode_fused(case):
    layer, gl = case
    st = gl.status()
    out, lse, idx = gl.decode(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_idx, ref_out, ref_lse = oracle.decode(
        batch_of(layer), layer.q8, layer.qscale, layer.w, layer.index_pages, layer.key_format,
        layer.q_lat, layer.latent_pages, layer.kv_scale, layer.sm_scale)
    rows = list(range(layer.total_q))
    vis = batch_of(layer).visible(rows)
    got = idx.cpu().numpy()
    # the selections are identical unless a threshold near-tie fell the other
    # way; in that case compare attention on the GPU's own selection
    if not np.array_equal(got, ref_idx):
        S, A, _ = check_scores(layer, gl.scores())
        check_topk_against_oracle(idx, S, A, vis, rows)
        ref_out, ref_lse = oracle.sparse_mla(batch_of(layer), layer.q_lat, layer.latent_pages,
                                             layer.kv_scale, layer.sm_scale, got)
    check_out(out, lse, ref_out, ref_lse, rows)


def test_small_context_selects_everything():
    layer = di.make_layer([1, 700, 2048], 1, seed=3)
    gl = GpuLayer(layer)
    _, _, idx = gl.decode()
    got = idx.cpu().numpy()
    for t, n in enumerate([1, 700, 2048]):
        assert np.array_equal(got[t, :n], np.arange(n)) and (got[t, n:] == -1).all()


def test_all_equal_scores_pick_lowest_positions():
    """Adversarial ties: w = 0 makes every score 0; the lowest 2048 positions win."""
    layer = di.make_layer([9000, 3000], [2, 1], seed=4)
    layer.w.zero_()
    gl = GpuLayer(layer)
    S = gl.scores()
    idx = gl.topk(S).cpu().numpy()
    assert (idx == np.arange(2048)[None, :]).all()


def test_page_placement_is_bit_identical():
    layer = di.make_layer([6000, 2500], [2, 1], seed=8, extra_pages=5)
    a = GpuLayer(layer).decode()
    b = GpuLayer(remap_pages(layer, 77)).decode()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_deterministic_repeat():
    layer = di.make_layer([20000, 17000], 1, seed=9)
    gl = GpuLayer(layer)
    a = gl.decode()
    b = gl.decode()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_batch_invariance():
    """A request's result does not depend on the other requests of the batch."""
    lens = [18000, 25000, 31000]
    layer = di.make_layer(lens, 1, seed=12)
    full = GpuLayer(layer).decode()
    for b in range(len(lens)):
        d = dict(layer.__dict__)
        d.update(q_offsets=torch.tensor([0, 1], dtype=torch.int32),
                 seq_lens=layer.seq_lens[b:b + 1].clone(),
                 block_table=layer.block_table[b:b + 1].clone(), q8=layer.q8[b:b + 1],
                 qscale=layer.qscale[b:b + 1], w=layer.w[b:b + 1], q_lat=layer.q_lat[b:b + 1],
                 seq_lens_host=[lens[b]], q_counts_host=[1])
        one = GpuLayer(di.Layer(**d)).decode()
        for x, y in zip(full, one):
            assert torch.equal(x[b:b + 1], y)


def test_batch_invariant_plan():
    """Under the batch-invariant plan a token's attention is bit-identical in a
    batch whose last, partial wave the default plan splits (200 tokens: the
    last 48 in two pieces) and alone (where the default plan takes 16 pieces);
    the tokens the default plan runs whole are unchanged by the switch, and the
    result matches the oracle."""
    n, nq = 40, 5
    lens = [2600 + 37 * b for b in range(n)]
    layer = di.make_layer(lens, nq, seed=21)
    gl = GpuLayer(layer)
    _, _, idx = gl.decode()
    out_d, lse_d = gl.mla(idx)
    b = n - 1
    d = dict(layer.__dict__)
    lo = nq * b
    d.update(q_offsets=torch.tensor([0, nq], dtype=torch.int32),
             seq_lens=layer.seq_lens[b:b + 1].clone(), block_table=layer.block_table[b:b + 1].clone(),
             q8=layer.q8[lo:lo + nq], qscale=layer.qscale[lo:lo + nq], w=layer.w[lo:lo + nq],
             q_lat=layer.q_lat[lo:lo + nq], seq_lens_host=[lens[b]], q_counts_host=[nq])
    one = GpuLayer(di.Layer(**d))
    prev = dsa.dsa_set_batch_invariant(True)
    try:
        out_i, lse_i = gl.mla(idx)
        out_1, lse_1 = one.mla(idx[lo:lo + nq].contiguous())
        dec_out, dec_lse, dec_idx = one.decode()
        assert dsa.dsa_set_batch_invariant(True)
    finally:
        dsa.dsa_set_batch_invariant(prev)
    torch.cuda.synchronize()
    assert torch.equal(out_i[lo:lo + nq], out_1) and torch.equal(lse_i[lo:lo + nq], lse_1)
    assert torch.equal(dec_idx, idx[lo:lo + nq])
    assert torch.equal(dec_out, out_1) and torch.equal(dec_lse, lse_1)
    assert torch.equal(out_i[:152], out_d[:152]) and torch.equal(lse_i[:152], lse_d[:152])
    rows = [0, 151, 152, 170, lo, lo + nq - 1]
    ref_out, ref_lse = oracle.sparse_mla(batch_of(layer), layer.q_lat, layer.latent_pages,
                                         layer.kv_scale, layer.sm_scale,
                                         idx[rows].cpu().numpy(), rows=rows)
    check_out(out_i, lse_i, ref_out, ref_lse, rows)


def test_prepared_decode_matches_the_direct_call():
    """A PreparedCall of dsa_decode issues the same call: identical results,
    and an error status raised the same way."""
    layer = di.make_layer([5000, 2600], [3, 2], seed=23)
    gl = GpuLayer(layer)
    out, lse, idx = gl.decode()
    g = gl.g
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    idx2 = torch.empty_like(idx)
    ws = torch.empty(dsa.dsa_decode_workspace_size(gl.batch), dtype=torch.uint8, device="cuda:0")
    st = gl.status()
    call = dsa.prepare_decode(gl.batch, g.q8, g.qscale, g.w, g.index_pages, layer.key_format,
                              g.q_lat, g.latent_pages, layer.kv_scale, layer.sm_scale, dsa.TOPK,
                              out2, lse2, idx2, ws, st)
    call()
    call()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out, out2) and torch.equal(lse, lse2) and torch.equal(idx, idx2)
    bad = dsa.prepare_decode(gl.batch, g.q8, g.qscale, g.w, g.index_pages, layer.key_format,
                             g.q_lat, g.latent_pages, layer.kv_scale, layer.sm_scale, dsa.TOPK,
                             out2, lse2, idx2, ws[:16], st)
    with pytest.raises(dsa.DsaError) as e:
        bad()
    assert e.value.status == 3  # DSA_ERR_WORKSPACE


def test_prepared_append_matches_the_direct_call():
    """A PreparedCall of dsa_append_cache writes the same cache bytes."""
    layer = di.make_layer([130, 3000], [5, 2], seed=43, extra_pages=1)
    keys, lat = di.append_payload(layer, seed=4)
    a, b = GpuLayer(layer), GpuLayer(layer)
    k_dev, l_dev = keys.cuda(), lat.cuda()
    dsa.dsa_append_cache(a.batch, k_dev, l_dev, layer.kv_scale, a.g.index_pages,
                         a.g.latent_pages, di.KEYS_FP8, a.status())
    call = dsa.prepare_append_cache(b.batch, k_dev, l_dev, layer.kv_scale, b.g.index_pages,
                                    b.g.latent_pages, di.KEYS_FP8, b.status())
    call()
    torch.cuda.synchronize()
    assert torch.equal(a.g.index_pages, b.g.index_pages)
    assert torch.equal(a.g.latent_pages, b.g.latent_pages)


def test_bad_page_id_sets_device_status():
    layer = di.make_layer([3000], 1, seed=13)
    layer.block_table[0, 5] = layer.num_pages + 10
    gl = GpuLayer(layer)
    st = gl.status()
    gl.decode(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 5  # DSA_ERR_DEVICE_CHECK


def test_bad_index_sets_device_status():
    layer = di.make_layer([3000], 1, seed=14)
    gl = GpuLayer(layer)
    idx = torch.full((1, 2048), -1, dtype=torch.int32, device="cuda:0")
    idx[0, 0] = 3000  # == seq_len: out of range
    idx[0, 1] = 17
    st = gl.status()
    out, lse = gl.mla(idx, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 5
    ref_out, _ = oracle.sparse_mla(batch_of(layer), layer.q_lat, layer.latent_pages,
                                   layer.kv_scale, layer.sm_scale,
                                   np.array([[17] + [-1] * 2047], np.int32))
    check_out(out, None, ref_out, None, [0])


def test_append_cache_bit_exact():
    layer = di.make_layer([130, 70, 64, 3000], [5, 1, 2, 7], seed=41, extra_pages=1)
    keys, lat = di.append_payload(layer, seed=3)
    keys[1] *= 1e-3
    keys[2] = 0.0
    gl = GpuLayer(layer)
    st = gl.status()
    dsa.dsa_append_cache(gl.batch, keys.cuda(), lat.cuda(), layer.kv_scale, gl.g.index_pages,
                         gl.g.latent_pages, di.KEYS_FP8, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ip, lp = oracle.append_cache(batch_of(layer), keys, lat, layer.kv_scale, layer.index_pages,
                                 layer.latent_pages)
    assert np.array_equal(gl.g.index_pages.cpu().numpy(), ip)
    assert np.array_equal(gl.g.latent_pages.cpu().numpy(), lp)


def test_host_validation_errors():
    layer = di.make_layer([100], 1, seed=1)
    gl = GpuLayer(layer)
    S = torch.empty(1, 128, dtype=torch.float32, device="cuda:0")
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_index_scores(gl.batch, gl.g.q8, gl.g.qscale, gl.g.w, gl.g.index_pages, 7, S, 128)
    assert e.value.status == 2
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_index_scores(gl.batch, gl.g.q8, gl.g.qscale, gl.g.w, gl.g.index_pages, 0, S, 50)
    assert e.value.status == 1
    idx = torch.empty(1, 1024, dtype=torch.int32, device="cuda:0")
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_topk(gl.batch, S, 128, 1024, idx)
    assert e.value.status == 2


@pytest.mark.parametrize("log2_scale", [16, -12])
def test_query_exponent_paths(log2_scale):
    """A query whose largest magnitude is >= 2^15 or < 2^-8 is rescaled by a
    power of two before it is lifted to f16.  Scaling q_lat by 2^s and the
    softmax scale by 2^-s leaves the exact result unchanged, so the oracle's
    output for the scaled inputs must be matched on that path too."""
    layer = di.make_layer([3000, 700, 2049], [2, 1, 1], di.KEYS_FP8, seed=77)
    gl = GpuLayer(layer)
    S_gpu = gl.scores()
    idx = gl.topk(S_gpu)
    q_scaled = (layer.q_lat.float() * 2.0 ** log2_scale).to(torch.bfloat16)
    sm_scale = layer.sm_scale * 2.0 ** -log2_scale
    out = torch.empty(gl.T, 96, 512, dtype=torch.bfloat16, device="cuda:0")
    lse = torch.empty(gl.T, 96, dtype=torch.float32, device="cuda:0")
    nws = dsa.dsa_sparse_mla_workspace_size(gl.batch)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda:0")
    st = gl.status()
    dsa.dsa_sparse_mla(gl.batch, q_scaled.to("cuda:0"), gl.g.latent_pages, layer.kv_scale,
                       sm_scale, idx, dsa.TOPK, out, lse, ws if nws else None, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_out, ref_lse = oracle.sparse_mla(batch_of(layer), q_scaled, layer.latent_pages,
                                         layer.kv_scale, sm_scale, idx.cpu().numpy())
    check_out(out, lse, ref_out, ref_lse, list(range(layer.total_q)))


def test_mla_whole_waves_and_split_tail():
    """160 query tokens: one wave of 152 tokens runs one CTA each, and the 8
    tokens left over are split into 16 pieces each (a full second wave) whose
    partials are merged; rows of both kinds, short rows with empty slots
    among them, against the oracle."""
    lens = [2100 + 613 * i for i in range(39)] + [1500]
    counts = [4] * 40
    layer = di.make_layer(lens, counts, seed=160, extra_pages=2)
    gl = GpuLayer(layer)
    st = gl.status()
    out, lse, idx = gl.decode(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = [0, 77, 151, 152, 153, 157, 158, 159]
    ref_out, ref_lse = oracle.sparse_mla(batch_of(layer), layer.q_lat, layer.latent_pages,
                                         layer.kv_scale, layer.sm_scale,
                                         idx[rows].cpu().numpy(), rows=rows)
    check_out(out, lse, ref_out, ref_lse, rows)
    # the last rows see fewer than 2048 positions: their trailing slots are empty
    assert (idx[159] < 0).any()
