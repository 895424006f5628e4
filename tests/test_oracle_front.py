"""Pins of the oracle's fused indexer front ("vLLM's Kimi K3.1 Pro day-0
support", section "Fused low-latency decode for DSA layers": query norm,
indexer query projection, FP8 quantisation with the head weights folded in,
the new token's index key).

- the projections against torch.matmul in float64 on the same bf16 inputs
  (the definition is a matrix product after the norm);
- the query norm: invariance to scaling the query latent by 4 (exact in bf16
  and fp64), and the closed form for an all-ones latent;
- the per-row quantiser against PyTorch's float8 rounding of x / (amax/448)."""
import numpy as np
import torch

import oracle

DQ, DH = 1536, 7168


def _inputs(T, seed):
    g = torch.Generator().manual_seed(seed)
    q_c = torch.randn(T, DQ, generator=g).to(torch.bfloat16)
    x = torch.randn(T, DH, generator=g).to(torch.bfloat16)
    w_q = (torch.randn(4096, DQ, generator=g) / DQ ** 0.5).to(torch.bfloat16)
    w_k = (torch.randn(128, DH, generator=g) / DH ** 0.5).to(torch.bfloat16)
    w_w = (torch.randn(32, DH, generator=g) / DH ** 0.5).to(torch.bfloat16)
    return q_c, x, w_q, w_k, w_w


def test_projections_match_torch_matmul():
    q_c, x, w_q, w_k, w_w = _inputs(3, 1)
    q, w, key, inv = oracle.indexer_front(q_c, x, w_q, w_k, w_w)
    qc = q_c.double()
    r = 1.0 / torch.sqrt((qc * qc).mean(dim=1) + 1e-6)
    assert np.allclose(inv, r.numpy(), rtol=1e-14, atol=0)
    assert np.allclose(q, (r[:, None] * (qc @ w_q.double().T)).numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(w, (x.double() @ w_w.double().T).numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(key, (x.double() @ w_k.double().T).numpy(), rtol=1e-12, atol=1e-12)


def test_query_norm_scale_invariance_and_closed_form():
    q_c, x, w_q, w_k, w_w = _inputs(2, 2)
    q1, _, _, _ = oracle.indexer_front(q_c, x, w_q, w_k, w_w)
    q4, _, _, _ = oracle.indexer_front((q_c.float() * 4).to(torch.bfloat16), x, w_q, w_k, w_w)
    assert np.allclose(q1, q4, rtol=1e-6, atol=0)   # only the 1e-6 epsilon differs
    ones = torch.ones(1, DQ, dtype=torch.bfloat16)
    q, _, _, inv = oracle.indexer_front(ones, x[:1], w_q, w_k, w_w)
    assert inv[0] == 1.0 / np.sqrt(1.0 + 1e-6)
    rows = w_q.double().sum(dim=1).numpy()
    assert np.allclose(q[0], rows * inv[0], rtol=1e-12, atol=1e-12)


def test_quantize_rows_matches_pytorch():
    g = torch.Generator().manual_seed(3)
    v = torch.randn(50, 128, generator=g) * torch.logspace(-6, 6, 50).view(50, 1)
    v[7] = 0.0
    codes, scales = oracle.quantize_rows(v.numpy(), 128)
    amax = v.abs().amax(dim=1)
    sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    want = (v / sc[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(scales, sc.numpy())
    assert np.array_equal(codes, want)
