"""Pins of the oracle's NVFP4 latent path ("vLLM's Kimi K3.1 Pro day-0
support", section "Packed KV cache": 352-byte NVFP4 latents; the byte split is
not printed and is read as 256 B of E2M1 for dims 0..511, one E4M3 scale per
16 of them, and 64 E4M3 bytes for dims 512..575, times one per-layer scale).

- the row decoder against a decode built from the OCP E2M1 golden table and
  PyTorch's float8_e4m3fn;
- NVFP4 pages whose values are also exactly E4M3 give bit-for-bit the result
  of the (already pinned) FP8 pages in sparse MLA and in the whole step;
- the 352-byte width against the pages' per-token totals."""
import numpy as np
import torch

import dsa_inputs as di
import oracle
from conftest import read_golden
from oracle_helpers import batch_of


def _e2m1_table():
    return {int(c, 16): float(v) for k, c, v in read_golden("mx_e2m1_e8m0.txt") if k == "e2m1"}


def _e4m3(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def test_latent_row_decoder_against_tables():
    rng = np.random.default_rng(4)
    tab = _e2m1_table()
    for _ in range(50):
        row = rng.integers(0, 256, 352, dtype=np.uint8)
        row[256:] &= 0x7E   # E4M3 scales / tail: finite, non-negative codes
        ks = float(rng.uniform(0.001, 0.1))
        want = np.empty(576)
        for d in range(512):
            nib = (row[d // 2] >> (4 * (d & 1))) & 15
            want[d] = tab[int(nib)] * _e4m3([row[256 + d // 16]])[0] * ks
        want[512:] = _e4m3(row[288:]) * ks
        assert np.array_equal(oracle.latent_row(row, ks, 1), want)
        # FP8 rows: E4M3 times the layer scale
        row8 = rng.integers(0, 256, 576, dtype=np.uint8) & 0x7E
        assert np.array_equal(oracle.latent_row(row8, ks, 0), _e4m3(row8) * ks)


def _twin_layers(seed):
    """An FP8 layer and an NVFP4 layer holding identical latent values:
    NVFP4 blocks with power-of-two E4M3 scales 2^k (k in -2..4) and E2M1
    elements, whose products are E4M3 values too."""
    layer = di.make_layer([2600, 900], [2, 1], seed=seed, extra_pages=1)
    n = layer.num_pages * di.PAGE
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, (n, 512)).astype(np.uint8)
    k = rng.integers(-2, 5, (n, 32))
    scale_codes = ((k + 7) << 3).astype(np.uint8)          # E4M3 2^k, mantissa 0
    tail = (rng.integers(0, 256, (n, 64)) & 0x7E).astype(np.uint8)
    tail[:, ::2] |= 0x80
    nv = np.concatenate([codes[:, 0::2] | (codes[:, 1::2] << 4), scale_codes, tail], axis=1)
    tab = _e2m1_table()
    vals = np.vectorize(tab.get)(codes) * (2.0 ** np.repeat(k, 16, axis=1))
    fp8 = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn)
    assert np.array_equal(fp8.to(torch.float64).numpy(), vals)   # exact in E4M3
    lat8 = np.concatenate([fp8.view(torch.uint8).numpy(), tail], axis=1)
    d8 = dict(layer.__dict__)
    d8["latent_pages"] = torch.from_numpy(lat8.reshape(layer.num_pages, -1).copy())
    dn = dict(layer.__dict__)
    dn["latent_pages"] = torch.from_numpy(nv.reshape(layer.num_pages, -1).copy())
    dn["latent_format"] = di.LATENT_NVFP4
    return di.Layer(**d8), di.Layer(**dn)


def test_nvfp4_pages_equal_fp8_pages_with_the_same_values():
    l8, l4 = _twin_layers(21)
    b = batch_of(l8)
    idx = np.full((3, 2048), -1, np.int32)
    rng = np.random.default_rng(0)
    for r, vis in enumerate(b.visible(range(3))):
        sel = np.sort(rng.choice(int(vis), min(int(vis), 1500), replace=False))
        idx[r, :sel.size] = sel
    o8, s8 = oracle.sparse_mla(b, l8.q_lat, l8.latent_pages, l8.kv_scale, l8.sm_scale, idx)
    o4, s4 = oracle.sparse_mla(b, l4.q_lat, l4.latent_pages, l4.kv_scale, l4.sm_scale, idx,
                               latent_format=1)
    assert np.array_equal(o8, o4) and np.array_equal(s8, s4)
    i8, d8, e8 = oracle.decode(b, l8.q8, l8.qscale, l8.w, l8.index_pages, l8.key_format,
                               l8.q_lat, l8.latent_pages, l8.kv_scale, l8.sm_scale)
    i4, d4, e4 = oracle.decode(b, l4.q8, l4.qscale, l4.w, l4.index_pages, l4.key_format,
                               l4.q_lat, l4.latent_pages, l4.kv_scale, l4.sm_scale,
                               latent_format=1)
    assert np.array_equal(i8, i4) and np.array_equal(d8, d4) and np.array_equal(e8, e4)


def test_nvfp4_width():
    assert di.NVFP4_LAT_BYTES == 352
    # the pages' per-token totals over 24 layers: NVFP4 latent + MXFP4 key = 10,080 B
    assert 24 * (di.NVFP4_LAT_BYTES + 68) == 10080
    layer = di.make_layer([200], [1], seed=1, latent_format=di.LATENT_NVFP4)
    assert layer.latent_pages.shape[1] == 64 * 352


def test_generator_quantisation_is_close():
    """The synthetic NVFP4 recipe (block scale E4M3(amax/6/kv_scale), nearest
    E2M1 element) reproduces N(0,1) latents within FP4's resolution."""
    layer = di.make_layer([128], [1], seed=2, latent_format=di.LATENT_NVFP4)
    ref = di.make_layer([128], [1], seed=2)
    a = np.stack([oracle.latent_row(r, layer.kv_scale, 1)
                  for r in layer.latent_pages.view(-1, 352)[:128].numpy()])
    b8 = np.stack([oracle.latent_row(r, ref.kv_scale, 0)
                   for r in ref.latent_pages.view(-1, 576)[:128].numpy()])
    rel = np.linalg.norm(a - b8) / np.linalg.norm(b8)
    assert rel < 0.12
