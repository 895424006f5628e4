"""Token-sharded prefill on one GPU: each rank's parts, run as a batch of
their own through dsa_decode, give bit-for-bit the unsharded step's indices
and output for their tokens (the ranks are run one after another; nothing
waits on another rank)."""
import pytest
import torch

import dsa_inputs as di
import dsa_sparse_attention_step_gb300 as dsa
from gpu_helpers import GpuLayer

pytestmark = pytest.mark.gpu


def _rank_batch(layer, g, parts):
    dev = "cuda:0"
    toks = torch.cat([torch.arange(p.token_begin, p.token_begin + p.num_tokens) for p in parts])
    counts = [p.num_tokens for p in parts]
    lens = [p.seq_len for p in parts]
    q_off = torch.tensor([0] + list(torch.tensor(counts).cumsum(0).tolist()), dtype=torch.int32)
    bt = layer.block_table[[p.request for p in parts]].contiguous()
    batch = dsa.Batch(q_off.to(dev), torch.tensor(lens, dtype=torch.int32, device=dev),
                      bt.to(dev), layer.num_pages, lens, counts)
    td = toks.to(dev)
    q = (g.q8[td].contiguous(), g.qscale[td].contiguous(), g.w[td].contiguous(),
         g.q_lat[td].contiguous())
    return batch, toks, q


@pytest.mark.parametrize("world", [2, 4])
def test_sharded_prefill_equals_unsharded(world):
    # two requests appending 512 and 96 tokens to cached prefixes
    layer = di.make_layer([20000 + 512, 3000 + 96], [512, 96], seed=123, extra_pages=2)
    gl = GpuLayer(layer)
    st = gl.status()
    out_f, lse_f, idx_f = gl.decode(st)
    g = gl.g
    covered = 0
    for r in range(world):
        parts = dsa.dsa_plan_token_shards(layer.seq_lens_host, layer.q_counts_host, world, r)
        batch, toks, (q8, qs, w, ql) = _rank_batch(layer, g, parts)
        T = len(toks)
        out = torch.empty(T, 96, 512, dtype=torch.bfloat16, device="cuda:0")
        lse = torch.empty(T, 96, dtype=torch.float32, device="cuda:0")
        idx = torch.empty(T, dsa.TOPK, dtype=torch.int32, device="cuda:0")
        ws = torch.empty(dsa.dsa_decode_workspace_size(batch), dtype=torch.uint8, device="cuda:0")
        dsa.dsa_decode(batch, q8, qs, w, g.index_pages, layer.key_format, ql, g.latent_pages,
                       layer.kv_scale, layer.sm_scale, dsa.TOPK, out, lse, idx, ws, st)
        torch.cuda.synchronize()
        td = toks.to("cuda:0")
        assert torch.equal(idx, idx_f[td])
        assert torch.equal(out.view(torch.int16), out_f[td].view(torch.int16))
        assert torch.equal(lse, lse_f[td])
        covered += T
    assert int(st.item()) == 0
    assert covered == gl.T
