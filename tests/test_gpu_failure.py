"""Failure detection on the GPU without a fault: every wait in the library's
kernels is bounded, and a wait that runs out sets DSA_ERR_TIMEOUT in the
caller's status word and lets the kernel return.  A test-only export withholds
one barrier arrival inside the sparse-MLA kernel with a short wait budget; the
status must read DSA_ERR_TIMEOUT, the call must return, and the next normal
step on the same stream must still match the oracle."""
import numpy as np
import pytest
import torch

import dsa_inputs as di
import dsa_sparse_attention_step_gb300 as dsa
import oracle
from gpu_helpers import GpuLayer, check_out
from oracle_helpers import batch_of

pytestmark = pytest.mark.gpu

DSA_ERR_TIMEOUT = 6


@pytest.mark.parametrize("lens,nq", [([3000], [1]), ([5000, 2600] * 40, [1] * 80)])
def test_sparse_mla_wait_timeout_reports_and_the_stream_recovers(lens, nq):
    layer = di.make_layer(lens, nq, seed=91, extra_pages=1)
    gl = GpuLayer(layer)
    g = gl.g
    idx = gl.topk(gl.scores())
    out = torch.empty(gl.T, 96, 512, dtype=torch.bfloat16, device="cuda:0")
    lse = torch.empty(gl.T, 96, dtype=torch.float32, device="cuda:0")
    nws = dsa.dsa_sparse_mla_workspace_size(gl.batch)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda:0")
    st = gl.status()
    dsa.dsa_test_sparse_mla_wait_timeout(gl.batch, g.q_lat, g.latent_pages, layer.kv_scale,
                                         layer.sm_scale, idx, dsa.TOPK, out, lse,
                                         ws if nws else None, st)
    torch.cuda.synchronize()
    assert int(st.item()) == DSA_ERR_TIMEOUT

    # the context is usable: a normal fused step on the same stream passes
    st2 = gl.status()
    out2, lse2, idx2 = gl.decode(st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    rows = [0, gl.T - 1]
    r_idx, r_out, r_lse = oracle.decode(batch_of(layer), layer.q8, layer.qscale, layer.w,
                                        layer.index_pages, layer.key_format, layer.q_lat,
                                        layer.latent_pages, layer.kv_scale, layer.sm_scale,
                                        rows=rows)
    check_out(out2, lse2, r_out, r_lse, rows)
