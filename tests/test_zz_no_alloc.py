"""dsa_decode_noalloc: the fused step for callers that cannot allocate device
memory on the call path (for example an engine whose device memory is all
pre-reserved by its own pool, or code that must not run the device-synchronising
cudaMalloc/cudaFree).  Its scratch is a fixed array inside the library instead
of a caller workspace.

Checked through the C ABI against dsa_decode on the same inputs, at the
tolerances of the other parity tests, on calls in a row (each later call
reuses the array with the earlier calls' contents still in it).  The last
batch (one query token over a 40,000-position context) takes the split-row
top-k, whose histograms and counters live in the shared array and must be
cleared by every call.  The file name
puts it last in collection order; it also passes on its own in a fresh
process."""
import numpy as np
import pytest
import torch

import dsa_inputs as di
import dsa_sparse_attention_step_gb300 as dsa
from gpu_helpers import GpuLayer, check_out

pytestmark = pytest.mark.gpu


def _noalloc(gl, status):
    g = gl.g
    out = torch.full((gl.T, 96, 512), float("nan"), dtype=torch.bfloat16, device="cuda:0")
    lse = torch.full((gl.T, 96), float("nan"), dtype=torch.float32, device="cuda:0")
    idx = torch.full((gl.T, dsa.TOPK), -7, dtype=torch.int32, device="cuda:0")
    dsa.dsa_decode_noalloc(gl.batch, g.q8, g.qscale, g.w, g.index_pages, gl.host.key_format,
                           g.q_lat, g.latent_pages, gl.host.kv_scale, gl.host.sm_scale, dsa.TOPK,
                           out, lse, idx, status)
    return out, lse, idx


def test_noalloc_matches_decode_on_calls_in_a_row():
    layers = [di.make_layer([20000, 9000, 31000], [1, 3, 1], seed=71, extra_pages=2),
              di.make_layer([4096, 2500, 17000], [2, 1, 1], seed=72, extra_pages=1),
              di.make_layer([40000], [1], seed=73, extra_pages=3)]
    assert all(dsa.dsa_decode_workspace_size(GpuLayer(l).batch) <= dsa.NOALLOC_SCRATCH_BYTES
               for l in layers)
    for layer in layers:  # different batches, back to back on one stream
        gl = GpuLayer(layer)
        ref_out, ref_lse, ref_idx = gl.decode()
        st = gl.status()
        out, lse, idx = _noalloc(gl, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(idx, ref_idx)
        rows = list(range(gl.T))
        check_out(out, lse, ref_out.double().cpu().numpy(), ref_lse.double().cpu().numpy(),
                  rows)


def test_noalloc_rejects_batches_beyond_its_scratch():
    """8 query tokens over a 1M-position context need 32 MiB of fp32 scores,
    more than the fixed 16 MiB: rejected on the host, nothing launched (the
    data tensors are never touched, so tiny stand-ins suffice)."""
    dev = "cuda:0"
    lens = [1 << 20] + [64] * 7
    batch = dsa.Batch(torch.arange(9, dtype=torch.int32, device=dev),
                      torch.tensor(lens, dtype=torch.int32, device=dev),
                      torch.zeros(8, (1 << 20) // 64, dtype=torch.int32, device=dev), 1,
                      lens, [1] * 8)
    assert dsa.dsa_decode_workspace_size(batch) > dsa.NOALLOC_SCRATCH_BYTES
    u8 = torch.zeros(64, dtype=torch.uint8, device=dev)
    f32 = torch.zeros(16, dtype=torch.float32, device=dev)
    bf = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    i32 = torch.zeros(16, dtype=torch.int32, device=dev)
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_decode_noalloc(batch, u8, f32, f32, u8, 0, bf, u8, 1.0, 0.07, dsa.TOPK, bf, f32,
                               i32, i32)
    assert e.value.status == 3  # DSA_ERR_WORKSPACE
