"""The byte/flop model used for roofline reporting, against the pages'
figures and closed forms."""
import pytest

from conftest import read_golden
from dsa_sparse_attention_step_gb300 import workload as wl


def test_dsa_reads_about_a_quarter_of_dense_at_long_context():
    g = {r[0]: float(r[-1]) for r in read_golden("kv_footprint.txt")}
    ctx = 1 << 20
    share = (wl.step_bytes([ctx], [1]) - wl.QUERY_BYTES_INDEXER - wl.QUERY_BYTES_MLA) \
        / wl.dense_mla_bytes(ctx)
    assert share == pytest.approx(g["dsa_share_long_context"], abs=0.005)
    assert share == pytest.approx((132 * ctx + 2048 * 576) / (576 * ctx))


def test_config_bytes():
    # 1M-token request: 132 B keys + 2048 latents + one query token
    b = wl.step_bytes([1 << 20], [1])
    assert b == 132 * (1 << 20) + 2048 * 576 + 4096 + 256 + 110592
    assert wl.step_bytes([1 << 20], [1], key_format=1) == b - 64 * (1 << 20)
    # short contexts gather only what exists
    assert wl.mla_bytes([100], [1]) == 100 * 576 + 110592


def test_prefill_append_flops():
    # 2048 queries appended to a 153600-token prefix: causal visible counts
    f = wl.indexer_flops([153600 + 2048], [2048])
    assert f == 2 * 32 * 128 * sum(153600 + i + 1 for i in range(2048))
    assert f / 1e12 == pytest.approx(2.594, abs=0.001)
    assert wl.mla_flops([153600 + 2048], [2048]) / 1e12 == pytest.approx(0.876, abs=0.001)
