"""The C-ABI library (CPU-only checks): it loads, exports every entry point
that include/dsa.h declares, and rejects invalid host arguments before any
CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for h in sorted(os.listdir(inc)):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(inc, h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from dsa_sparse_attention_step_gb300 import _build
    _build.build()
    import dsa_sparse_attention_step_gb300 as dsa
    return dsa.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"dsa_index_scores", "dsa_topk", "dsa_sparse_mla", "dsa_decode",
            "dsa_append_cache"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_batch_invariant_switch_returns_the_previous_setting(lib):
    import dsa_sparse_attention_step_gb300 as dsa
    prev = dsa.dsa_set_batch_invariant(True)
    try:
        assert dsa.dsa_set_batch_invariant(True) is True
        assert dsa.dsa_set_batch_invariant(False) is True
        assert dsa.dsa_set_batch_invariant(False) is False
    finally:
        dsa.dsa_set_batch_invariant(prev)


def test_status_strings(lib):
    import dsa_sparse_attention_step_gb300 as dsa
    assert dsa.dsa_status_string(0) == "ok"
    assert "workspace" in dsa.dsa_status_string(3)


def _cbatch(**kw):
    import dsa_sparse_attention_step_gb300 as dsa
    b = dsa._CBatch(1, 1, 1, 4096, 64, 64, 64, 16, 32, 48)
    for k, v in kw.items():
        setattr(b, k, v)
    return b


def test_invalid_host_arguments_return_before_launch(lib):
    fake = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    b = _cbatch()
    # unsupported key format
    assert lib.dsa_index_scores(ctypes.byref(b), fake, fake, fake, fake, 9, fake, 4096, None,
                                None) == 2
    # score row stride shorter than the longest sequence
    assert lib.dsa_index_scores(ctypes.byref(b), fake, fake, fake, fake, 0, fake, 100, None,
                                None) == 1
    # misaligned query pointer
    assert lib.dsa_index_scores(ctypes.byref(b), ctypes.c_void_p(4097), fake, fake, fake, 0,
                                fake, 4096, None, None) == 1
    # page size other than 64
    b2 = _cbatch(page_size=32)
    assert lib.dsa_topk(ctypes.byref(b2), fake, 4096, 2048, fake, None, 0, None) == 2
    # top-k other than 2048
    assert lib.dsa_topk(ctypes.byref(b), fake, 4096, 1000, fake, None, 0, None) == 2
    # block table too short for the longest sequence
    b3 = _cbatch(max_pages=10)
    assert lib.dsa_topk(ctypes.byref(b3), fake, 4096, 2048, fake, None, 0, None) == 1
    # NULL batch
    assert lib.dsa_sparse_mla(None, fake, fake, 1.0, 1.0, fake, 2048, fake, None, None, 0,
                              None, None) == 1
    # non-positive latent scale
    assert lib.dsa_sparse_mla(ctypes.byref(b), fake, fake, 0.0, 1.0, fake, 2048, fake, None,
                              None, 0, None, None) == 1
    # workspace too small for the fused step
    need = lib.dsa_decode_workspace_size(ctypes.byref(b), 2048)
    assert need >= 4096 * 4
    assert lib.dsa_decode(ctypes.byref(b), fake, fake, fake, fake, 0, fake, fake, 1.0, 0.07,
                          2048, fake, None, fake, fake, need - 1, None, None) == 3
    # MXFP4 append is not provided
    assert lib.dsa_append_cache(ctypes.byref(b), fake, None, 1.0, fake, None, 1, None,
                                None) == 2


def test_topk_workspace_follows_the_split_path(lib):
    """Only batches of at most 8 query tokens over rows longer than 32,768
    positions split their rows over the GPU and need top-k scratch; the fused
    step's workspace includes it, and a missing one is refused before launch."""
    fake = ctypes.c_void_p(4096)
    pages = (1 << 20) // 64

    def size(total_q, max_seq):
        b = _cbatch(total_q=total_q, num_requests=1, max_q_per_request=total_q,
                    max_seq_len=max_seq, num_pages=pages, max_pages=pages)
        return b, lib.dsa_topk_workspace_size(ctypes.byref(b), 2048)

    b1, one = size(1, 1 << 20)
    _, two = size(2, 1 << 20)
    _, eight = size(8, 1 << 20)
    assert one > 0 and two > one and eight > 0
    assert size(9, 1 << 20)[1] == 0       # one cluster per row
    assert size(8, 32768)[1] == 0         # rows kept in shared memory
    assert size(1, 32769)[1] > 0
    scores = (1 << 20) * 4
    assert lib.dsa_decode_workspace_size(ctypes.byref(b1), 2048) >= scores + one
    assert lib.dsa_topk(ctypes.byref(b1), fake, 1 << 20, 2048, fake, None, 0, None) == 3
    assert lib.dsa_topk(ctypes.byref(b1), fake, 1 << 20, 2048, fake, fake, one - 1, None) == 3
