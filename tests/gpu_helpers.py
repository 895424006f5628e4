"""Helpers of the GPU parity tests: run the C-ABI entry points on a layer and
compare with the CPU oracle at the stated tolerances."""
import numpy as np
import torch

import dsa_inputs as di
import dsa_sparse_attention_step_gb300 as dsa
import oracle
from oracle_helpers import batch_of

# Tolerances of the parity contract
SCORE_REL_TO_ABS = 1e-4   # |S_gpu - S| <= 1e-4 * sum |terms|
OUT_REL_L2 = 1e-2         # attention output, relative L2 vs fp64
OUT_MAX_ABS = 3e-2        # attention output, max abs vs fp64
LSE_ABS = 1e-3            # log-sum-exp (natural log), absolute


class GpuLayer:
    """A layer's tensors on cuda:0 plus the library's Batch."""

    def __init__(self, layer):
        dev = torch.device("cuda:0")
        self.host = layer
        self.g = layer.to(dev)
        self.batch = dsa.Batch(self.g.q_offsets, self.g.seq_lens, self.g.block_table,
                               layer.num_pages, layer.seq_lens_host, layer.q_counts_host)
        self.T = layer.total_q
        self.ld = ((layer.max_seq_len + 127) // 128) * 128

    def status(self):
        return torch.zeros(1, dtype=torch.int32, device="cuda:0")

    def scores(self, status=None):
        S = torch.full((self.T, self.ld), float("nan"), dtype=torch.float32, device="cuda:0")
        g = self.g
        dsa.dsa_index_scores(self.batch, g.q8, g.qscale, g.w, g.index_pages, self.host.key_format,
                             S, self.ld, status)
        return S

    def topk(self, S):
        idx = torch.full((self.T, dsa.TOPK), -7, dtype=torch.int32, device="cuda:0")
        nws = dsa.dsa_topk_workspace_size(self.batch)
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda:0")
        dsa.dsa_topk(self.batch, S, self.ld, dsa.TOPK, idx, ws if nws else None)
        return idx

    def mla(self, idx, status=None):
        g = self.g
        out = torch.empty(self.T, 96, 512, dtype=torch.bfloat16, device="cuda:0")
        lse = torch.empty(self.T, 96, dtype=torch.float32, device="cuda:0")
        nws = dsa.dsa_sparse_mla_workspace_size(self.batch)
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda:0")
        dsa.dsa_sparse_mla(self.batch, g.q_lat, g.latent_pages, self.host.kv_scale,
                           self.host.sm_scale, idx, dsa.TOPK, out, lse, ws if nws else None,
                           status)
        return out, lse

    def decode(self, status=None):
        g = self.g
        out = torch.empty(self.T, 96, 512, dtype=torch.bfloat16, device="cuda:0")
        lse = torch.empty(self.T, 96, dtype=torch.float32, device="cuda:0")
        idx = torch.empty(self.T, dsa.TOPK, dtype=torch.int32, device="cuda:0")
        ws = torch.empty(dsa.dsa_decode_workspace_size(self.batch), dtype=torch.uint8,
                         device="cuda:0")
        dsa.dsa_decode(self.batch, g.q8, g.qscale, g.w, g.index_pages, self.host.key_format,
                       g.q_lat, g.latent_pages, self.host.kv_scale, self.host.sm_scale, dsa.TOPK,
                       out, lse, idx, ws, status)
        return out, lse, idx


def check_scores(layer, S_gpu, rows=None):
    """GPU scores vs fp64 oracle: |diff| <= 1e-4 * A on visible positions,
    -inf on the causally masked positions of the request."""
    rows = list(range(layer.total_q)) if rows is None else list(rows)
    ld = S_gpu.shape[1]
    S, A = oracle.index_scores(batch_of(layer), layer.q8, layer.qscale, layer.w,
                               layer.index_pages, layer.key_format, rows=rows, ld=ld)
    G = S_gpu[rows].double().cpu().numpy()
    vis = batch_of(layer).visible(rows)
    worst = 0.0
    for r, t in enumerate(rows):
        n = int(vis[r])
        b = int(np.searchsorted(layer.q_offsets.numpy(), t, side="right") - 1)
        seq = layer.seq_lens_host[b]
        err = np.abs(G[r, :n] - S[r, :n])
        bound = SCORE_REL_TO_ABS * A[r, :n]
        assert (err <= bound).all(), "row %d: worst err/bound %.3g" % (
            t, float((err / np.maximum(bound, 1e-300)).max()))
        assert np.isneginf(G[r, n:seq]).all(), "row %d: masked positions not -inf" % t
        worst = max(worst, float((err / np.maximum(bound, 1e-300)).max(initial=0.0)))
    return S, A, worst


def check_topk_against_scores(idx_gpu, S_gpu, vis, rows):
    """Bit-exact: the oracle's selection run on the GPU's own scores."""
    G = S_gpu[rows].double().cpu().numpy()
    want = oracle.topk(G, vis, dsa.TOPK)
    got = idx_gpu[rows].cpu().numpy()
    for r in range(len(rows)):
        assert np.array_equal(got[r], want[r]), "row %d differs" % rows[r]


def check_topk_against_oracle(idx_gpu, S, A, vis, rows):
    """Sets may differ from the oracle's only at near-ties of the threshold."""
    got = idx_gpu[rows].cpu().numpy()
    for r in range(len(rows)):
        n = int(vis[r])
        want = oracle.topk_row(S[r], n, dsa.TOPK)
        if n <= dsa.TOPK:
            assert np.array_equal(got[r], want)
            continue
        order = sorted(range(n), key=lambda s: (-S[r, s], s))
        tau_i = order[dsa.TOPK - 1]
        tau = S[r, tau_i]
        a, b = set(got[r].tolist()), set(want.tolist())
        for s in a ^ b:
            assert abs(S[r, s] - tau) <= SCORE_REL_TO_ABS * (A[r, s] + A[r, tau_i]), (
                "row %d: position %d is not a near-tie" % (rows[r], s))


def check_out(out_gpu, lse_gpu, ref_out, ref_lse, rows):
    o = out_gpu[rows].float().cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(o - ref_out) / max(np.linalg.norm(ref_out), 1e-300)
    mx = float(np.abs(o - ref_out).max(initial=0.0))
    assert rel <= OUT_REL_L2 and mx <= OUT_MAX_ABS, (rel, mx)
    if lse_gpu is not None:
        l = lse_gpu[rows].double().cpu().numpy()
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(l), fin)
        assert np.abs(l[fin] - ref_lse[fin]).max(initial=0.0) <= LSE_ABS
    return rel, mx
