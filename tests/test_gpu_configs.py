"""GPU parity at the five workloads' full sizes, in the launch configuration
the benchmark times (the fused dsa_decode over the whole batch; the append
before it for the prefill-append workload), checked on sampled query rows that
the oracle computes one by one (always the first and the last row)."""
import numpy as np
import pytest
import torch

import dsa_inputs as di
import dsa_sparse_attention_step_gb300 as dsa
import oracle
from gpu_helpers import (GpuLayer, check_out, check_scores, check_topk_against_oracle,
                         check_topk_against_scores)
from oracle_helpers import batch_of

pytestmark = pytest.mark.gpu

SAMPLES = {
    "c0_tiny": [0],
    "c1_batched": list(range(8)),
    "c2_agentic": [0, 4, 157, 319],
    "c3a_long_fp8": [0],
    "c3b_long_mxfp4": [0],
    "c4_prefill_append": [0, 1, 1024, 2047],
}


def _run(name):
    layer_dev = di.make_config(name, device="cuda")
    layer = layer_dev.to("cpu")
    gl = GpuLayer(layer)
    gl.g = layer_dev  # same bytes, already resident
    rows = SAMPLES[name]
    if name == "c4_prefill_append":
        keys, lat = di.append_payload(layer_dev, seed=4004)
        st = gl.status()
        dsa.dsa_append_cache(gl.batch, keys, lat, layer.kv_scale, layer_dev.index_pages,
                             layer_dev.latent_pages, di.KEYS_FP8, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ip, lp = oracle.append_cache(batch_of(layer), keys.cpu(), lat.cpu(), layer.kv_scale,
                                     layer.index_pages, layer.latent_pages)
        assert np.array_equal(layer_dev.index_pages.cpu().numpy(), ip)
        assert np.array_equal(layer_dev.latent_pages.cpu().numpy(), lp)
        layer.index_pages = torch.from_numpy(ip)
        layer.latent_pages = torch.from_numpy(lp)
    st = gl.status()
    out, lse, idx = gl.decode(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # scores of the same launch configuration, for the sampled rows
    S_gpu = gl.scores()
    vis = batch_of(layer).visible(rows)
    S, A, worst = check_scores(layer, S_gpu, rows)
    check_topk_against_scores(idx, S_gpu, vis, rows)
    check_topk_against_oracle(idx, S, A, vis, rows)
    ref_out, ref_lse = oracle.sparse_mla(batch_of(layer), layer.q_lat, layer.latent_pages,
                                         layer.kv_scale, layer.sm_scale,
                                         idx[rows].cpu().numpy(), rows=rows)
    rel, mx = check_out(out, lse, ref_out, ref_lse, rows)
    return worst, rel, mx


@pytest.mark.parametrize("name", ["c0_tiny", "c1_batched"])
def test_small_configs(name):
    _run(name)


@pytest.mark.parametrize("name", ["c2_agentic", "c3a_long_fp8", "c3b_long_mxfp4",
                                  "c4_prefill_append"])
def test_large_configs(name):
    _run(name)
