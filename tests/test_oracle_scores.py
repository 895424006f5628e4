"""Pins of the oracle's indexer scores.

S[t,s] = sum_h w[t,h] ReLU(qhat[t,h].khat[s]) is pinned by
  * the one-hot case w = e_h, which reduces to ReLU of a plain GEMM (checked
    against torch.matmul in float64 on keys decoded by PyTorch), together with
  * linearity and positive homogeneity in w, which extend the one-hot case to
    any w;
and by the causal rule, scale folding, page-placement invariance and the
MXFP4/FP8 equivalence of equal dequantised keys.
"""
import numpy as np
import pytest
import torch

import dsa_inputs as di
import oracle
from oracle_helpers import (batch_of, dense_keys, dense_q, oracle_scores, remap_pages,
                            request_of, visible)


@pytest.fixture(scope="module")
def layer():
    # two requests, ragged lengths (partial last pages), multi-token causal rows
    return di.make_layer([200, 131], n_q=[3, 1], seed=11, extra_pages=3)


def _with_w(layer, w):
    d = dict(layer.__dict__)
    d["w"] = w
    return di.Layer(**d)


def test_one_hot_weights_reduce_to_relu_gemm(layer):
    T = layer.total_q
    for h in [0, 5, 17, 31]:
        w = torch.zeros(T, 32)
        w[:, h] = 1.0
        S, _ = oracle_scores(_with_w(layer, w))
        for t in range(T):
            b, _ = request_of(layer, t)
            K = dense_keys(layer, b)
            ref = torch.relu(dense_q(layer, t)[h] @ K.T).numpy()
            n = visible(layer, t)
            np.testing.assert_allclose(S[t, :n], ref[:n], rtol=1e-12, atol=1e-12)


def test_linear_and_positively_homogeneous_in_w(layer):
    g = torch.Generator().manual_seed(3)
    # multiples of 2^-10 of modest size, so that w1 + w2 is exact in fp32
    w1 = torch.round(torch.randn(layer.total_q, 32, generator=g) * 1024) / 1024
    w2 = torch.round(torch.randn(layer.total_q, 32, generator=g) * 1024) / 1024
    S1, _ = oracle_scores(_with_w(layer, w1))
    S2, _ = oracle_scores(_with_w(layer, w2))
    S12, _ = oracle_scores(_with_w(layer, w1 + w2))
    Sc, _ = oracle_scores(_with_w(layer, w1 * 0.5))
    fin = np.isfinite(S1)
    np.testing.assert_allclose(S12[fin], S1[fin] + S2[fin], rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(Sc[fin], 0.5 * S1[fin], rtol=1e-12, atol=0)


def test_weighted_sum_of_one_hot_rows(layer):
    """S(w) = sum_h w_h S(e_h): the one-hot pins extended to the drawn w."""
    T = layer.total_q
    S, _ = oracle_scores(layer)
    acc = np.zeros_like(S)
    for h in range(32):
        e = torch.zeros(T, 32)
        e[:, h] = 1.0
        Sh, _ = oracle_scores(_with_w(layer, e))
        acc += layer.w[:, h].double().numpy()[:, None] * np.where(np.isfinite(Sh), Sh, 0)
    fin = np.isfinite(S)
    np.testing.assert_allclose(S[fin], acc[fin], rtol=1e-9, atol=1e-9)


def test_causal_rule_and_padding(layer):
    ld = 256
    S, A = oracle_scores(layer, ld=ld)
    for t in range(layer.total_q):
        n = visible(layer, t)
        assert np.isfinite(S[t, :n]).all()
        assert np.isneginf(S[t, n:]).all() and (A[t, n:] == 0).all()
    # request 0 has 3 query tokens at positions 197, 198, 199
    assert [visible(layer, t) for t in range(4)] == [198, 199, 200, 131]


def test_abs_magnitude_bounds_scores(layer):
    S, A = oracle_scores(layer)
    fin = np.isfinite(S)
    assert (np.abs(S[fin]) <= A[fin] * (1 + 1e-12)).all()


def test_query_scale_folds_out(layer):
    d = dict(layer.__dict__)
    d["qscale"] = layer.qscale * 4.0
    S4, _ = oracle_scores(di.Layer(**d))
    S1, _ = oracle_scores(layer)
    fin = np.isfinite(S1)
    np.testing.assert_allclose(S4[fin], 4.0 * S1[fin], rtol=1e-12)


def test_page_placement_does_not_matter(layer):
    S1, _ = oracle_scores(layer)
    S2, _ = oracle_scores(remap_pages(layer, 5))
    assert np.array_equal(S1, S2)


def test_bad_page_id_is_reported(layer):
    d = dict(layer.__dict__)
    bt = layer.block_table.clone()
    bt[1, 0] = layer.num_pages  # out of range
    d["block_table"] = bt
    with pytest.raises(RuntimeError, match="page id"):
        oracle_scores(di.Layer(**d))


def test_mxfp4_keys_equal_fp8_keys_with_the_same_values():
    """Keys whose E2M1 x E8M0 values are exactly E4M3 values (scale 1) give the
    same scores in both formats."""
    lay = di.make_layer([150], n_q=2, seed=21)
    g = torch.Generator().manual_seed(9)
    ntok = lay.num_pages * 64
    codes = torch.randint(0, 16, (ntok, 128), generator=g, dtype=torch.uint8)
    exps = torch.randint(126, 130, (ntok, 4), generator=g, dtype=torch.uint8)  # 2^-1 .. 2^2
    mag = torch.tensor([0, .5, 1, 1.5, 2, 3, 4, 6], dtype=torch.float64)
    vals = mag[(codes & 7).long()] * torch.where(codes >= 8, -1.0, 1.0).double()
    vals = vals * torch.exp2(exps.double() - 127).repeat_interleave(32, dim=1)
    mx = torch.empty(lay.num_pages, di.MXFP4_PAGE_BYTES, dtype=torch.uint8)
    mx[:, :4096] = (codes[:, 0::2] | (codes[:, 1::2] << 4)).reshape(lay.num_pages, 4096)
    mx[:, 4096:] = exps.reshape(lay.num_pages, 256)
    f8 = torch.empty(lay.num_pages, di.FP8_PAGE_BYTES, dtype=torch.uint8)
    e4 = vals.to(torch.float32).to(torch.float8_e4m3fn)
    assert torch.equal(e4.to(torch.float64), vals)  # exact in E4M3
    f8[:, :8192] = e4.view(torch.uint8).reshape(lay.num_pages, 8192)
    f8[:, 8192:] = torch.ones(lay.num_pages, 64).view(torch.uint8).reshape(lay.num_pages, 256)
    b = batch_of(lay)
    S_mx, _ = oracle.index_scores(b, lay.q8, lay.qscale, lay.w, mx, di.KEYS_MXFP4)
    S_f8, _ = oracle.index_scores(b, lay.q8, lay.qscale, lay.w, f8, di.KEYS_FP8)
    assert np.array_equal(S_mx, S_f8)
