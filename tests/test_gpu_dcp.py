"""Decode context parallelism on one GPU ("vLLM's Kimi K3.1 Pro day-0
support", sections "Decode context parallelism with the sparse indexer" and
"Exact top-k merge with about 10x less traffic"): W ranks hold the
interleaved positions of each row; dsa_dcp_topk runs the one-round candidate
exchange with detection and resend, dsa_lse_combine merges the ranks' partial
attention.  Checked through the C ABI against the oracle: the merged indices
and the resend decisions bit-exact (both sides take them on the same fp32
scores, rounded to BF16), every rank's share, and the combined attention
output at the parity tolerances."""
import numpy as np
import pytest
import torch

import dsa_inputs as di
import dsa_sparse_attention_step_gb300 as dsa
import oracle
from gpu_helpers import GpuLayer, check_out
from oracle_helpers import batch_of

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _dcp(gl, S, world, cand=0):
    T = gl.T
    idx = torch.full((T, dsa.TOPK), -7, dtype=torch.int32, device=DEV)
    ridx = torch.full((world, T, dsa.TOPK), -7, dtype=torch.int32, device=DEV)
    resent = torch.full((T, world), -7, dtype=torch.int32, device=DEV)
    ws = torch.empty(dsa.dsa_dcp_topk_workspace_size(gl.batch, world, cand), dtype=torch.uint8,
                     device=DEV)
    dsa.dsa_dcp_topk(gl.batch, S, gl.ld, world, cand, dsa.TOPK, idx, ridx, resent, ws)
    torch.cuda.synchronize()
    return idx, ridx, resent


def _check_against_oracle(gl, S, idx, ridx, resent, world, cand, rows=None):
    layer = gl.host
    rows = list(range(gl.T)) if rows is None else rows
    vis = batch_of(layer).visible(rows)
    want, want_resend = oracle.dcp_topk(S[rows].cpu().numpy(), vis, world,
                                        cand if cand else None, dsa.TOPK)
    got = idx[rows].cpu().numpy()
    assert np.array_equal(got, want)
    assert np.array_equal(resent[rows].cpu().numpy(), want_resend)
    r_all = ridx.cpu().numpy()
    for i, t in enumerate(rows):
        sel = got[i][got[i] >= 0]
        for r in range(world):
            mine = sel[sel % world == r]
            exp = np.full(dsa.TOPK, -1, np.int32)
            exp[:mine.size] = mine
            assert np.array_equal(r_all[r, t], exp), (t, r)
    return want_resend


@pytest.mark.parametrize("world", [8, 6, 4, 3, 2, 1])
def test_dcp_topk_on_indexer_scores(world):
    layer = di.make_layer([40000, 23000, 2500, 9000], [2, 1, 3, 1], seed=500 + world, extra_pages=2)
    gl = GpuLayer(layer)
    S = gl.scores()
    idx, ridx, resent = _dcp(gl, S, world)
    _check_against_oracle(gl, S, idx, ridx, resent, world, 0)


@pytest.mark.parametrize("cand", [16, 200, 0])
def test_dcp_resend_path_on_skewed_scores(cand):
    """Rows where one or several ranks hold most winners: they are detected
    and resend; the merge stays exact."""
    world = 8
    layer = di.make_layer([30000, 30000, 30000, 700, 5], [1, 1, 1, 1, 1], seed=77, extra_pages=1)
    gl = GpuLayer(layer)
    g = torch.Generator().manual_seed(3)
    S = torch.randn(gl.T, gl.ld, generator=g)
    S[0, 3::world] += 20.0                    # rank 3 holds every winner
    S[1, 0::world] += 2.0                     # ranks 0 and 5 hold many
    S[1, 5::world] += 2.0
    S[2] = torch.round(S[2] * 2) / 2          # heavy BF16 ties
    S[3, :] = 1.0                             # 700 visible, all equal
    S = S.to(DEV)
    idx, ridx, resent = _dcp(gl, S, world, cand)
    want_resend = _check_against_oracle(gl, S, idx, ridx, resent, world, cand)
    assert want_resend[0, 3] == 1
    if cand == 16:
        assert want_resend.sum() >= 3


def test_dcp_attention_equals_merged_attention():
    """Each rank attends over its share of the merged selection (dsa_sparse_mla
    on rank_indices[r]); dsa_lse_combine of the ranks' outputs matches the
    oracle's attention over the whole merged selection."""
    world = 8
    layer = di.make_layer([131072, 20000, 3000], [5, 2, 1], seed=42, extra_pages=2)
    gl = GpuLayer(layer)
    S = gl.scores()
    idx, ridx, resent = _dcp(gl, S, world)
    rows = [0, 4, 5, 7]
    _check_against_oracle(gl, S, idx, ridx, resent, world, 0, rows)
    parts = torch.empty(world, gl.T, 96, 512, dtype=torch.bfloat16, device=DEV)
    lses = torch.empty(world, gl.T, 96, dtype=torch.float32, device=DEV)
    for r in range(world):
        o, l = gl.mla(ridx[r].contiguous())
        parts[r].copy_(o)
        lses[r].copy_(l)
    out = torch.empty(gl.T, 96, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(gl.T, 96, dtype=torch.float32, device=DEV)
    dsa.dsa_lse_combine(gl.T, world, parts, lses, out, lse)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.sparse_mla(batch_of(layer), layer.q_lat, layer.latent_pages,
                                         layer.kv_scale, layer.sm_scale,
                                         idx[rows].cpu().numpy(), rows=rows)
    check_out(out, lse, ref_out, ref_lse, rows)


def test_lse_combine_matches_oracle_combine():
    T, world = 3, 5
    g = torch.Generator().manual_seed(8)
    parts = torch.randn(world, T, 96, 512, generator=g).to(torch.bfloat16)
    lses = torch.randn(world, T, 96, generator=g) * 3
    lses[1, 0, :] = float("-inf")            # a rank with no tokens
    lses[:, 2, 7] = float("-inf")            # nothing anywhere for (2, 7)
    out = torch.empty(T, 96, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(T, 96, dtype=torch.float32, device=DEV)
    dsa.dsa_lse_combine(T, world, parts.to(DEV), lses.to(DEV), out, lse)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.lse_combine(parts.double().numpy(), lses.double().numpy())
    o = out.double().cpu().numpy()
    assert np.abs(o - ref).max() <= 1e-2 * max(1.0, np.abs(ref).max())
    fin = np.isfinite(ref_lse)
    l = lse.double().cpu().numpy()
    assert np.array_equal(np.isfinite(l), fin)
    assert np.abs(l[fin] - ref_lse[fin]).max() <= 1e-4
    assert (o[2, 7] == 0).all()


def test_dcp_limits_are_host_errors():
    layer = di.make_layer([70000], [1], seed=3)
    gl = GpuLayer(layer)
    S = torch.zeros(1, gl.ld, dtype=torch.float32, device=DEV)
    idx = torch.empty(1, dsa.TOPK, dtype=torch.int32, device=DEV)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    with pytest.raises(dsa.DsaError) as e:   # 70,000 positions do not fit 16 bits on one rank
        dsa.dsa_dcp_topk(gl.batch, S, gl.ld, 1, 0, dsa.TOPK, idx, None, None, ws)
    assert e.value.status == 2
    with pytest.raises(dsa.DsaError) as e:   # at most 8 ranks
        dsa.dsa_dcp_topk(gl.batch, S, gl.ld, 9, 0, dsa.TOPK, idx, None, None, ws)
    assert e.value.status == 2
