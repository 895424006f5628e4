"""NVFP4 latents (352 B per token; section "Packed KV cache") through the C
ABI: dsa_sparse_mla_ex and dsa_decode_ex with DSA_LATENT_NVFP4 against the
oracle, and bit-identity with the FP8 path on caches whose values are exact in
both formats (the kernel lifts both to the same f16 operands)."""
import numpy as np
import pytest
import torch

import dsa_inputs as di
import dsa_sparse_attention_step_gb300 as dsa
import oracle
from gpu_helpers import GpuLayer, check_out, check_topk_against_scores
from oracle_helpers import batch_of
from test_oracle_nvfp4 import _twin_layers

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _mla(gl, idx, latent_format):
    g = gl.g
    out = torch.full((gl.T, 96, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(gl.T, 96, dtype=torch.float32, device=DEV)
    nws = dsa.dsa_sparse_mla_workspace_size(gl.batch)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=DEV)
    st = gl.status()
    dsa.dsa_sparse_mla_ex(gl.batch, g.q_lat, g.latent_pages, latent_format, gl.host.kv_scale,
                          gl.host.sm_scale, idx, dsa.TOPK, out, lse, ws if nws else None, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out, lse


@pytest.mark.parametrize("lens,nq", [([3000, 700, 2049, 65], [2, 1, 1, 1]),
                                     ([20000, 9000], [5, 3]),
                                     ([1, 64, 129], [1, 1, 1])])
def test_sparse_mla_nvfp4_matches_oracle(lens, nq):
    layer = di.make_layer(lens, nq, seed=sum(lens) % 997, extra_pages=2,
                          latent_format=di.LATENT_NVFP4)
    gl = GpuLayer(layer)
    idx = gl.topk(gl.scores())
    out, lse = _mla(gl, idx, dsa.LATENT_NVFP4)
    rows = list(range(gl.T))
    ref_out, ref_lse = oracle.sparse_mla(batch_of(layer), layer.q_lat, layer.latent_pages,
                                         layer.kv_scale, layer.sm_scale, idx.cpu().numpy(),
                                         latent_format=1)
    check_out(out, lse, ref_out, ref_lse, rows)


def test_nvfp4_and_fp8_paths_agree_bitwise_on_shared_values():
    l8, l4 = _twin_layers(33)
    g8, g4 = GpuLayer(l8), GpuLayer(l4)
    idx = g8.topk(g8.scores())
    o8, s8 = _mla(g8, idx, dsa.LATENT_FP8)
    o4, s4 = _mla(g4, idx, dsa.LATENT_NVFP4)
    assert torch.equal(o8.view(torch.int16), o4.view(torch.int16))
    assert torch.equal(s8, s4)


def test_decode_nvfp4_full_step():
    layer = di.make_layer([131072, 40000, 3000], [5, 1, 2], seed=404, extra_pages=1,
                          latent_format=di.LATENT_NVFP4)
    gl = GpuLayer(layer)
    g = gl.g
    out = torch.empty(gl.T, 96, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(gl.T, 96, dtype=torch.float32, device=DEV)
    idx = torch.empty(gl.T, dsa.TOPK, dtype=torch.int32, device=DEV)
    ws = torch.empty(dsa.dsa_decode_workspace_size(gl.batch), dtype=torch.uint8, device=DEV)
    st = gl.status()
    dsa.dsa_decode_ex(gl.batch, g.q8, g.qscale, g.w, g.index_pages, layer.key_format, g.q_lat,
                      g.latent_pages, dsa.LATENT_NVFP4, layer.kv_scale, layer.sm_scale, dsa.TOPK,
                      out, lse, idx, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = [0, 4, 5, 7]
    S = gl.scores()
    check_topk_against_scores(idx, S, batch_of(layer).visible(rows), rows)
    ref_out, ref_lse = oracle.sparse_mla(batch_of(layer), layer.q_lat, layer.latent_pages,
                                         layer.kv_scale, layer.sm_scale, idx[rows].cpu().numpy(),
                                         rows=rows, latent_format=1)
    check_out(out, lse, ref_out, ref_lse, rows)


def test_unknown_latent_format_is_a_host_error():
    layer = di.make_layer([300], [1], seed=5)
    gl = GpuLayer(layer)
    idx = gl.topk(gl.scores())
    with pytest.raises(dsa.DsaError) as e:
        _mla(gl, idx, 7)
    assert e.value.status == 2
