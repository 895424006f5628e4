"""The oracle's cache formats against the byte figures the pages print."""
import pytest

import oracle
from conftest import read_golden


def _golden():
    g = {}
    for row in read_golden("kv_footprint.txt"):
        g[(row[0], row[1] if len(row) > 2 else None)] = float(row[-1])
    return g


def test_widths_and_page_sizes():
    c = oracle.constants()
    g = _golden()
    assert c["fp8_key_bytes_per_token"] == g[("width", "index_fp8")] == 132
    assert c["mxfp4_key_bytes_per_token"] == g[("width", "index_mxfp4")] == 68
    assert c["lat_bytes_per_token"] == g[("width", "latent_fp8")] == 576
    assert c["fp8_page_bytes"] == 64 * 132
    assert c["mxfp4_page_bytes"] == 64 * 68
    assert c["lat_page_bytes"] == 64 * 576
    assert c["idx_heads"] == 32 and c["idx_dim"] == 128
    assert c["mla_heads"] == 96 and c["lat_dim"] == 576 and c["v_dim"] == 512


def test_24_layer_footprints():
    c = oracle.constants()
    g = _golden()
    lat, key8, key4 = c["lat_bytes_per_token"], c["fp8_key_bytes_per_token"], \
        c["mxfp4_key_bytes_per_token"]
    nvfp4 = g[("width", "latent_nvfp4")]
    assert 24 * lat == g[("footprint24", "k3_fp8_latent")]
    assert 24 * (lat + key8) == g[("footprint24", "k31_fp8_latent_fp8_index")]
    assert 24 * (nvfp4 + key4) == g[("footprint24", "k31_nvfp4_latent_mxfp4_index")]


def test_mxfp4_saving_and_long_context_share():
    c = oracle.constants()
    g = _golden()
    key8, key4, lat = (c["fp8_key_bytes_per_token"], c["mxfp4_key_bytes_per_token"],
                       c["lat_bytes_per_token"])
    assert 1 - key4 / key8 == pytest.approx(g[("saving", "mxfp4_vs_fp8_index")], abs=5e-4)
    k = int(g[("topk", None)])
    share = lambda ctx: (key8 * ctx + k * lat) / (lat * ctx)
    # "about 23%" at long context; the limit is 132/576
    assert share(1 << 20) == pytest.approx(g[("dsa_share_long_context", None)], abs=0.005)
    assert share(1 << 30) == pytest.approx(key8 / lat, rel=1e-3)
    assert share(128 * 1024) > share(1 << 20)
