"""Pins of the oracle's cache writer against PyTorch's float8_e4m3fn rounding
(a library conversion independent of the oracle's encoder)."""
import numpy as np
import torch

import dsa_inputs as di
import oracle
from oracle_helpers import batch_of


def _layer():
    return di.make_layer([130, 70, 64], n_q=[5, 1, 2], seed=41, extra_pages=1)


def _slots(layer):
    """(page, slot) of each new token, in q_offsets order."""
    out = []
    for b in range(layer.num_requests):
        n, s = layer.q_counts_host[b], layer.seq_lens_host[b]
        for j in range(n):
            pos = s - n + j
            out.append((int(layer.block_table[b, pos // 64]), pos % 64))
    return out


def test_append_matches_library_rounding_and_touches_only_new_slots():
    lay = _layer()
    keys, lat = di.append_payload(lay, seed=3)
    keys[1] *= 1e-3           # a small-magnitude key: subnormal codes appear
    keys[2] = 0.0             # amax == 0: scale 1, all-zero codes
    ip, lp = oracle.append_cache(batch_of(lay), keys, lat, lay.kv_scale, lay.index_pages,
                                 lay.latent_pages)
    ip = torch.from_numpy(ip)
    lp = torch.from_numpy(lp)
    touched_i = torch.zeros_like(ip, dtype=torch.bool)
    touched_l = torch.zeros_like(lp, dtype=torch.bool)
    for t, (page, slot) in enumerate(_slots(lay)):
        x = keys[t]
        amax = x.abs().max()
        scale = amax / 448.0 if amax > 0 else torch.tensor(1.0)
        want = (x / scale).to(torch.float8_e4m3fn).view(torch.uint8)
        assert torch.equal(ip[page, slot * 128:(slot + 1) * 128], want)
        got_scale = ip[page, 8192 + 4 * slot: 8192 + 4 * slot + 4].view(torch.float32)[0]
        assert got_scale.item() == scale.to(torch.float32).item()
        touched_i[page, slot * 128:(slot + 1) * 128] = True
        touched_i[page, 8192 + 4 * slot: 8192 + 4 * slot + 4] = True
        y = lat[t] / torch.tensor(lay.kv_scale, dtype=torch.float32)
        y = y.clamp(-448, 448)  # satfinite (the library conversion does not saturate)
        assert torch.equal(lp[page, slot * 576:(slot + 1) * 576],
                           y.to(torch.float8_e4m3fn).view(torch.uint8))
        touched_l[page, slot * 576:(slot + 1) * 576] = True
    assert torch.equal(ip[~touched_i], lay.index_pages[~touched_i])
    assert torch.equal(lp[~touched_l], lay.latent_pages[~touched_l])
    assert (ip[_slots(lay)[2][0], _slots(lay)[2][1] * 128:][:128] == 0).all()


def test_append_then_scores_see_the_new_keys():
    """Written keys decode back to within E4M3 rounding of the fp32 input."""
    lay = _layer()
    keys, lat = di.append_payload(lay, seed=4)
    ip, _ = oracle.append_cache(batch_of(lay), keys, None, lay.kv_scale, lay.index_pages, None)
    for t, (page, slot) in enumerate(_slots(lay)):
        codes = ip[page, slot * 128:(slot + 1) * 128]
        scale = np.frombuffer(ip[page, 8192 + 4 * slot: 8192 + 4 * slot + 4].tobytes(),
                              np.float32)[0]
        back = oracle.e4m3_decode(codes) * scale
        x = keys[t].double().numpy()
        # E4M3 relative step is 2^-3 (half-step 2^-4) for normals; subnormals
        # are absolute steps of 2^-9 * scale
        assert np.all(np.abs(back - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * scale)
                      * (1 + 1e-6))
