"""Pins of the oracle's sparse MLA: dense attention from PyTorch's
scaled_dot_product_attention (float64, different value width) over the
selected latents, logsumexp from torch.logsumexp, and the closed-form special
cases (identical latents, zero query, one selected token)."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import dsa_inputs as di
import oracle
from oracle_helpers import batch_of, dense_latents, fp8, request_of


@pytest.fixture(scope="module")
def layer():
    return di.make_layer([300, 77], n_q=[2, 1], seed=31, extra_pages=2)


def _sdpa(layer, t, sel):
    b, _ = request_of(layer, t)
    L = dense_latents(layer, b)[torch.as_tensor(sel, dtype=torch.long)]
    q = layer.q_lat[t].to(torch.float64)                       # [96, 576]
    o = F.scaled_dot_product_attention(q[None], L[None], L[None, :, :512],
                                       scale=layer.sm_scale)[0]
    lse = torch.logsumexp(layer.sm_scale * (q @ L.T), dim=-1)
    return o.numpy(), lse.numpy()


def _mla(layer, idx, rows):
    return oracle.sparse_mla(batch_of(layer), layer.q_lat, layer.latent_pages, layer.kv_scale,
                             layer.sm_scale, idx, rows=rows)


def test_all_tokens_selected_equals_dense_attention(layer):
    rows = [0, 1, 2]
    idx = np.full((3, 2048), -1, np.int32)
    idx[0, :300] = np.arange(300)
    idx[1, :300] = np.arange(300)
    idx[2, :77] = np.arange(77)
    out, lse = _mla(layer, idx, rows)
    for r, t in enumerate(rows):
        n = 300 if t < 2 else 77
        o_ref, l_ref = _sdpa(layer, t, np.arange(n))
        np.testing.assert_allclose(out[r], o_ref, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[r], l_ref, rtol=1e-12, atol=1e-12)


def test_scattered_subset_with_holes(layer):
    rng = np.random.default_rng(2)
    sel = np.sort(rng.choice(300, size=120, replace=False)).astype(np.int32)
    idx = np.full((1, 2048), -1, np.int32)
    pos = np.sort(rng.choice(2048, size=120, replace=False))
    idx[0, pos] = rng.permutation(sel)  # any order, -1 holes anywhere
    out, lse = _mla(layer, idx, [1])
    o_ref, l_ref = _sdpa(layer, 1, sel)
    np.testing.assert_allclose(out[0], o_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse[0], l_ref, rtol=1e-12)


def test_identical_latents_return_that_latent(layer):
    d = dict(layer.__dict__)
    lat = layer.latent_pages.clone()
    row = lat[0, :576].clone()
    lat.view(-1, 576)[:] = row
    d["latent_pages"] = lat
    lay = di.Layer(**d)
    idx = np.full((1, 2048), -1, np.int32)
    idx[0, :50] = np.arange(0, 250, 5)
    out, _ = _mla(lay, idx, [0])
    v = (fp8(row) * lay.kv_scale)[:512].numpy()
    np.testing.assert_allclose(out[0], np.broadcast_to(v, (96, 512)), rtol=1e-13, atol=1e-15)


def test_zero_query_gives_mean_of_selected_values(layer):
    d = dict(layer.__dict__)
    d["q_lat"] = torch.zeros_like(layer.q_lat)
    lay = di.Layer(**d)
    sel = np.array([3, 9, 64, 65, 199], np.int32)
    idx = np.full((1, 2048), -1, np.int32)
    idx[0, :5] = sel
    out, lse = _mla(lay, idx, [0])
    L = dense_latents(lay, 0)[torch.as_tensor(sel, dtype=torch.long)]
    np.testing.assert_allclose(out[0], np.broadcast_to(L[:, :512].mean(0).numpy(), (96, 512)),
                               rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse[0], math.log(5.0), rtol=1e-14)


def test_single_selected_token(layer):
    idx = np.full((1, 2048), -1, np.int32)
    idx[0, 700] = 42
    out, _ = _mla(layer, idx, [2])  # row 2 = request 1
    v = dense_latents(layer, 1)[42, :512].numpy()
    np.testing.assert_allclose(out[0], np.broadcast_to(v, (96, 512)), rtol=1e-13, atol=1e-15)


def test_empty_selection(layer):
    idx = np.full((1, 2048), -1, np.int32)
    out, lse = _mla(layer, idx, [0])
    assert (out == 0).all() and np.isneginf(lse).all()


def test_index_beyond_sequence_is_rejected(layer):
    idx = np.full((1, 2048), -1, np.int32)
    idx[0, 0] = 77  # request 1 has 77 tokens: 0..76
    with pytest.raises(RuntimeError, match="index"):
        _mla(layer, idx, [2])
