"""The fused indexer front through the C ABI ("vLLM's Kimi K3.1 Pro day-0
support", section "Fused low-latency decode for DSA layers": query norm,
indexer query projection, FP8 quantisation with the head weights folded in,
the new token's index key, in one kernel).

- the fp32 projections against the fp64 oracle within 1e-4 of sum |terms|;
- the query codes and scales bit-exact against the oracle's quantiser run on
  the kernel's own fp32 values (the same decision in the same precision);
- the index cache bit-exact against the oracle's cache writer given the
  kernel's fp32 keys (and every other byte untouched);
- the front's outputs drive the indexer to oracle-matching scores."""
import numpy as np
import pytest
import torch

import dsa_inputs as di
import dsa_sparse_attention_step_gb300 as dsa
import oracle
from gpu_helpers import GpuLayer, check_scores
from oracle_helpers import batch_of

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DQ, DH = dsa.FRONT_QLAT_DIM, dsa.FRONT_HIDDEN_DIM


def _weights(seed):
    g = torch.Generator().manual_seed(seed)
    w_q = (torch.randn(4096, DQ, generator=g) / DQ ** 0.5).to(torch.bfloat16)
    w_k = (torch.randn(128, DH, generator=g) / DH ** 0.5).to(torch.bfloat16)
    w_w = (torch.randn(32, DH, generator=g) / DH ** 0.5).to(torch.bfloat16)
    return w_q, w_k, w_w


@pytest.mark.parametrize("lens,nq", [([3000], [1]), ([5000, 700, 64], [3, 1, 1]),
                                     ([9000, 4000], [40, 30])])
def test_indexer_front_matches_oracle(lens, nq):
    layer = di.make_layer(lens, nq, seed=sum(lens) % 1000, extra_pages=2)
    gl = GpuLayer(layer)
    T = gl.T
    g = torch.Generator().manual_seed(T)
    q_c = torch.randn(T, DQ, generator=g).to(torch.bfloat16)
    x = torch.randn(T, DH, generator=g).to(torch.bfloat16)
    w_q, w_k, w_w = _weights(7)
    d = {k: v.to(DEV) for k, v in dict(q_c=q_c, x=x, w_q=w_q, w_k=w_k, w_w=w_w).items()}
    q8 = torch.empty(T, 32, 128, dtype=torch.uint8, device=DEV)
    qs = torch.empty(T, 32, dtype=torch.float32, device=DEV)
    w = torch.empty(T, 32, dtype=torch.float32, device=DEV)
    qf = torch.empty(T, 4096, dtype=torch.float32, device=DEV)
    kf = torch.empty(T, 128, dtype=torch.float32, device=DEV)
    pages = gl.g.index_pages.clone()
    st = gl.status()
    dsa.dsa_indexer_front(gl.batch, d["q_c"], d["x"], d["w_q"], d["w_k"], d["w_w"], q8, qs, w,
                          pages, dsa.KEYS_FP8, qf, kf, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    q_ref, w_ref, k_ref, inv = oracle.indexer_front(q_c, x, w_q, w_k, w_w)
    qcd, xd = q_c.double(), x.double()
    A_q = inv[:, None] * (qcd.abs() @ w_q.double().abs().T).numpy()
    A_x = xd.abs()
    assert (np.abs(qf.double().cpu().numpy() - q_ref) <= 1e-4 * A_q).all()
    assert (np.abs(w.double().cpu().numpy() - w_ref) <= 1e-4 * (A_x @ w_w.double().abs().T).numpy()).all()
    assert (np.abs(kf.double().cpu().numpy() - k_ref) <= 1e-4 * (A_x @ w_k.double().abs().T).numpy()).all()

    codes, scales = oracle.quantize_rows(qf.cpu().numpy(), 128)
    assert np.array_equal(q8.cpu().numpy().reshape(-1, 128), codes)
    assert np.array_equal(qs.cpu().numpy().reshape(-1), scales)

    ip, _ = oracle.append_cache(batch_of(layer), kf.cpu(), None, layer.kv_scale,
                                layer.index_pages, None)
    assert np.array_equal(pages.cpu().numpy(), ip)

    # the front's outputs are the indexer's inputs
    d2 = dict(layer.__dict__)
    d2.update(q8=q8.cpu(), qscale=qs.cpu(), w=w.cpu(), index_pages=pages.cpu())
    l2 = di.Layer(**d2)
    g2 = GpuLayer(l2)
    check_scores(l2, g2.scores(), rows=list(range(min(T, 6))))


def test_mxfp4_pool_is_rejected_for_the_key_write():
    layer = di.make_layer([300], [1], di.KEYS_MXFP4, seed=2)
    gl = GpuLayer(layer)
    z = lambda *s, dt=torch.bfloat16: torch.zeros(*s, dtype=dt, device=DEV)
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_indexer_front(gl.batch, z(1, DQ), z(1, DH), z(4096, DQ), z(128, DH), z(32, DH),
                              z(1, 32, 128, dt=torch.uint8), z(1, 32, dt=torch.float32),
                              z(1, 32, dt=torch.float32), gl.g.index_pages, dsa.KEYS_MXFP4)
    assert e.value.status == 2
