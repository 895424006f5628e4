"""GB300-native DSA sparse-attention step.

Python binding of ``libdsa.so`` (the C ABI declared in ``include/dsa.h``):
argument marshalling only.  Every step of the path runs in the library's CUDA
kernels; PyTorch supplies device memory and streams.  There is no CPU
fallback: importing works without a GPU, but every call needs the built
library and a CUDA device, and raises otherwise.
"""
import ctypes
import os

import torch

__all__ = ["DsaError", "Batch", "KEYS_FP8", "KEYS_MXFP4", "TOPK", "library_path", "load",
           "dsa_status_string", "dsa_launch_count", "dsa_set_batch_invariant",
           "dsa_index_scores", "dsa_topk",
           "dsa_topk_workspace_size", "dsa_sparse_mla", "dsa_sparse_mla_workspace_size",
           "dsa_decode", "dsa_decode_workspace_size", "dsa_decode_noalloc",
           "NOALLOC_SCRATCH_BYTES", "dsa_append_cache", "ShardPart", "dsa_plan_token_shards",
           "dsa_dcp_topk_workspace_size", "dsa_dcp_topk", "dsa_lse_combine",
           "LATENT_FP8", "LATENT_NVFP4", "dsa_sparse_mla_ex", "dsa_decode_ex",
           "dsa_indexer_front", "FRONT_QLAT_DIM", "FRONT_HIDDEN_DIM", "PreparedCall",
           "prepare_decode", "prepare_append_cache"]

KEYS_FP8 = 0
KEYS_MXFP4 = 1
LATENT_FP8 = 0
LATENT_NVFP4 = 1
FRONT_QLAT_DIM = 1536    # query latent of dsa_indexer_front
FRONT_HIDDEN_DIM = 7168  # hidden state of dsa_indexer_front
TOPK = 2048
PAGE = 64
NOALLOC_SCRATCH_BYTES = 16 << 20  # DSA_NOALLOC_SCRATCH_BYTES of include/dsa.h

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB = None


def library_path():
    return os.path.join(_PKG, "libdsa.so")


class DsaError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, _status_str(status), status))


class _CBatch(ctypes.Structure):
    _fields_ = [("num_requests", ctypes.c_int32), ("total_q", ctypes.c_int32),
                ("max_q_per_request", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("q_offsets", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p)]


class ShardPart(ctypes.Structure):
    """One part of a request assigned to a rank (dsa_shard_part)."""
    _fields_ = [("request", ctypes.c_int32), ("token_begin", ctypes.c_int32),
                ("num_tokens", ctypes.c_int32), ("seq_len", ctypes.c_int32)]

    def __repr__(self):
        return "ShardPart(request=%d, token_begin=%d, num_tokens=%d, seq_len=%d)" % (
            self.request, self.token_begin, self.num_tokens, self.seq_len)


_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_sz = ctypes.c_size_t
_bp = ctypes.POINTER(_CBatch)

_SIGS = {
    "dsa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "dsa_launch_count": (ctypes.c_uint64, []),
    "dsa_set_batch_invariant": (ctypes.c_int32, [ctypes.c_int32]),
    "dsa_index_scores": (ctypes.c_int, [_bp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _i64, _vp, _vp]),
    "dsa_topk_workspace_size": (_sz, [_bp, _i32]),
    "dsa_topk": (ctypes.c_int, [_bp, _vp, _i64, _i32, _vp, _vp, _sz, _vp]),
    "dsa_sparse_mla_workspace_size": (_sz, [_bp, _i32]),
    "dsa_sparse_mla": (ctypes.c_int, [_bp, _vp, _vp, _f32, _f32, _vp, _i32, _vp, _vp, _vp, _sz,
                                      _vp, _vp]),
    "dsa_decode_workspace_size": (_sz, [_bp, _i32]),
    "dsa_sparse_mla_ex": (ctypes.c_int, [_bp, _vp, _vp, ctypes.c_int, _f32, _f32, _vp, _i32, _vp,
                                         _vp, _vp, _sz, _vp, _vp]),
    "dsa_decode_ex": (ctypes.c_int, [_bp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _vp, ctypes.c_int,
                                     _f32, _f32, _i32, _vp, _vp, _vp, _vp, _sz, _vp, _vp]),
    "dsa_decode": (ctypes.c_int, [_bp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _vp, _f32, _f32,
                                  _i32, _vp, _vp, _vp, _vp, _sz, _vp, _vp]),
    "dsa_decode_noalloc": (ctypes.c_int, [_bp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _vp, _f32,
                                          _f32, _i32, _vp, _vp, _vp, _vp, _vp]),
    "dsa_append_cache": (ctypes.c_int, [_bp, _vp, _vp, _f32, _vp, _vp, ctypes.c_int, _vp, _vp]),
    "dsa_dcp_topk_workspace_size": (_sz, [_bp, _i32, _i32, _i32]),
    "dsa_dcp_topk": (ctypes.c_int, [_bp, _vp, _i64, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _sz,
                                    _vp]),
    "dsa_lse_combine": (ctypes.c_int, [_i32, _i32, _vp, _vp, _vp, _vp, _vp]),
    "dsa_indexer_front": (ctypes.c_int, [_bp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                         ctypes.c_int, _vp, _vp, _vp, _vp]),
    "dsa_plan_token_shards": (ctypes.c_int32, [ctypes.POINTER(ctypes.c_int32),
                                               ctypes.POINTER(ctypes.c_int32), _i32, _i32, _i32,
                                               ctypes.POINTER(ShardPart), _i32]),
    "dsa_test_sparse_mla_wait_timeout": (ctypes.c_int, [_bp, _vp, _vp, _f32, _f32, _vp, _i32, _vp,
                                                        _vp, _vp, _sz, _vp, _vp]),
}


def load():
    """Load libdsa.so (built in-tree by ``__graft_entry__.build()``)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError("libdsa.so is not built (%s); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`" % path)
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _status_str(s):
    try:
        return load().dsa_status_string(int(s)).decode()
    except Exception:  # library missing while formatting an error
        return "status"


def dsa_status_string(s):
    return load().dsa_status_string(int(s)).decode()


def dsa_launch_count():
    return int(load().dsa_launch_count())


def dsa_set_batch_invariant(enabled):
    """Process-wide batch-invariant attention plan on (True) or off; returns
    the previous setting."""
    return bool(load().dsa_set_batch_invariant(1 if enabled else 0))


def _check(rc, what):
    if rc != 0:
        raise DsaError(rc, what)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError("%s has dtype %s" % (name, t.dtype))
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Batch:
    """Request metadata of one step: device int32 arrays plus the host copies
    the library uses to size its grids."""

    def __init__(self, q_offsets, seq_lens, block_table, num_pages, seq_lens_host=None,
                 q_counts_host=None):
        self.q_offsets = q_offsets.to(torch.int32).contiguous()
        self.seq_lens = seq_lens.to(torch.int32).contiguous()
        self.block_table = block_table.to(torch.int32).contiguous()
        if seq_lens_host is None:
            seq_lens_host = self.seq_lens.cpu().tolist()
        if q_counts_host is None:
            off = self.q_offsets.cpu().tolist()
            q_counts_host = [off[i + 1] - off[i] for i in range(len(off) - 1)]
        self.seq_lens_host = [int(v) for v in seq_lens_host]
        self.q_counts_host = [int(v) for v in q_counts_host]
        self.num_pages = int(num_pages)
        self._c = _CBatch(len(self.seq_lens_host), sum(self.q_counts_host),
                          max(self.q_counts_host), max(self.seq_lens_host), self.num_pages,
                          int(self.block_table.shape[-1]), PAGE,
                          self.q_offsets.data_ptr(), self.seq_lens.data_ptr(),
                          self.block_table.data_ptr())

    @property
    def total_q(self):
        return self._c.total_q

    @property
    def max_seq_len(self):
        return self._c.max_seq_len

    def ref(self):
        return ctypes.byref(self._c)


def dsa_index_scores(batch, q_fp8, q_scale, w, index_pages, key_format, scores, score_ld=None,
                     dev_status=None, stream=None):
    if score_ld is None:
        score_ld = scores.shape[-1]
    rc = load().dsa_index_scores(batch.ref(), _ptr(q_fp8, torch.uint8, "q_fp8"),
                                 _ptr(q_scale, torch.float32, "q_scale"),
                                 _ptr(w, torch.float32, "w"),
                                 _ptr(index_pages, torch.uint8, "index_pages"), int(key_format),
                                 _ptr(scores, torch.float32, "scores"), int(score_ld),
                                 _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(rc, "dsa_index_scores")


def dsa_topk_workspace_size(batch, topk=TOPK):
    return int(load().dsa_topk_workspace_size(batch.ref(), int(topk)))


def dsa_topk(batch, scores, score_ld, topk, indices, ws=None, stream=None):
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    rc = load().dsa_topk(batch.ref(), _ptr(scores, torch.float32, "scores"), int(score_ld),
                         int(topk), _ptr(indices, torch.int32, "indices"), _ptr(ws), nbytes,
                         _stream(stream))
    _check(rc, "dsa_topk")


def dsa_sparse_mla_workspace_size(batch, topk=TOPK):
    return int(load().dsa_sparse_mla_workspace_size(batch.ref(), int(topk)))


def dsa_sparse_mla(batch, q_lat, latent_pages, kv_scale, sm_scale, indices, topk, out, lse=None,
                   ws=None, dev_status=None, stream=None):
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    rc = load().dsa_sparse_mla(batch.ref(), _ptr(q_lat, (torch.bfloat16, torch.int16), "q_lat"),
                               _ptr(latent_pages, torch.uint8, "latent_pages"), float(kv_scale),
                               float(sm_scale), _ptr(indices, torch.int32, "indices"), int(topk),
                               _ptr(out, (torch.bfloat16, torch.int16), "out"),
                               _ptr(lse, torch.float32, "lse"), _ptr(ws), nbytes,
                               _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(rc, "dsa_sparse_mla")


def dsa_test_sparse_mla_wait_timeout(batch, q_lat, latent_pages, kv_scale, sm_scale, indices,
                                     topk, out, lse=None, ws=None, dev_status=None, stream=None):
    """Test-only (include/dsa_testing.h): dsa_sparse_mla with the kernel's
    bounded-wait failure path forced; the device status becomes 6."""
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    rc = load().dsa_test_sparse_mla_wait_timeout(
        batch.ref(), _ptr(q_lat, (torch.bfloat16, torch.int16), "q_lat"),
        _ptr(latent_pages, torch.uint8, "latent_pages"), float(kv_scale), float(sm_scale),
        _ptr(indices, torch.int32, "indices"), int(topk),
        _ptr(out, (torch.bfloat16, torch.int16), "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(ws), nbytes, _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(rc, "dsa_test_sparse_mla_wait_timeout")


def dsa_sparse_mla_ex(batch, q_lat, latent_pages, latent_format, kv_scale, sm_scale, indices,
                      topk, out, lse=None, ws=None, dev_status=None, stream=None):
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    rc = load().dsa_sparse_mla_ex(batch.ref(), _ptr(q_lat, (torch.bfloat16, torch.int16), "q_lat"),
                                  _ptr(latent_pages, torch.uint8, "latent_pages"),
                                  int(latent_format), float(kv_scale), float(sm_scale),
                                  _ptr(indices, torch.int32, "indices"), int(topk),
                                  _ptr(out, (torch.bfloat16, torch.int16), "out"),
                                  _ptr(lse, torch.float32, "lse"), _ptr(ws), nbytes,
                                  _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(rc, "dsa_sparse_mla_ex")


def dsa_decode_ex(batch, q_fp8, q_scale, w, index_pages, key_format, q_lat, latent_pages,
                  latent_format, kv_scale, sm_scale, topk, out, lse, indices, ws,
                  dev_status=None, stream=None):
    nbytes = ws.numel() * ws.element_size()
    rc = load().dsa_decode_ex(batch.ref(), _ptr(q_fp8, torch.uint8, "q_fp8"),
                              _ptr(q_scale, torch.float32, "q_scale"), _ptr(w, torch.float32, "w"),
                              _ptr(index_pages, torch.uint8, "index_pages"), int(key_format),
                              _ptr(q_lat, (torch.bfloat16, torch.int16), "q_lat"),
                              _ptr(latent_pages, torch.uint8, "latent_pages"),
                              int(latent_format), float(kv_scale), float(sm_scale), int(topk),
                              _ptr(out, (torch.bfloat16, torch.int16), "out"),
                              _ptr(lse, torch.float32, "lse"),
                              _ptr(indices, torch.int32, "indices"), _ptr(ws), nbytes,
                              _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(rc, "dsa_decode_ex")


def dsa_decode_workspace_size(batch, topk=TOPK):
    return int(load().dsa_decode_workspace_size(batch.ref(), int(topk)))


def dsa_decode(batch, q_fp8, q_scale, w, index_pages, key_format, q_lat, latent_pages, kv_scale,
               sm_scale, topk, out, lse, indices, ws, dev_status=None, stream=None):
    nbytes = ws.numel() * ws.element_size()
    rc = load().dsa_decode(batch.ref(), _ptr(q_fp8, torch.uint8, "q_fp8"),
                           _ptr(q_scale, torch.float32, "q_scale"), _ptr(w, torch.float32, "w"),
                           _ptr(index_pages, torch.uint8, "index_pages"), int(key_format),
                           _ptr(q_lat, (torch.bfloat16, torch.int16), "q_lat"),
                           _ptr(latent_pages, torch.uint8, "latent_pages"), float(kv_scale),
                           float(sm_scale), int(topk),
                           _ptr(out, (torch.bfloat16, torch.int16), "out"),
                           _ptr(lse, torch.float32, "lse"), _ptr(indices, torch.int32, "indices"),
                           _ptr(ws), nbytes, _ptr(dev_status, torch.int32, "dev_status"),
                           _stream(stream))
    _check(rc, "dsa_decode")


class PreparedCall:
    """One entry point with its arguments checked and converted once, for a
    step repeated on the same buffers (a serving loop): each call issues the
    same C-ABI call as the function it was prepared from, without the
    per-call argument handling in Python.  It keeps the tensors it was given
    alive; their storage must not move."""

    def __init__(self, name, fn, args, keep):
        self._name, self._fn, self._args, self._keep = name, fn, args, keep

    def __call__(self):
        rc = self._fn(*self._args)
        if rc != 0:
            raise DsaError(rc, self._name)


def prepare_decode(batch, q_fp8, q_scale, w, index_pages, key_format, q_lat, latent_pages,
                   kv_scale, sm_scale, topk, out, lse, indices, ws, dev_status=None, stream=None):
    """dsa_decode as a PreparedCall (same arguments)."""
    if stream is None:
        stream = torch.cuda.current_stream()
    args = (batch.ref(), _ptr(q_fp8, torch.uint8, "q_fp8"), _ptr(q_scale, torch.float32, "q_scale"),
            _ptr(w, torch.float32, "w"), _ptr(index_pages, torch.uint8, "index_pages"),
            int(key_format), _ptr(q_lat, (torch.bfloat16, torch.int16), "q_lat"),
            _ptr(latent_pages, torch.uint8, "latent_pages"), float(kv_scale), float(sm_scale),
            int(topk), _ptr(out, (torch.bfloat16, torch.int16), "out"),
            _ptr(lse, torch.float32, "lse"), _ptr(indices, torch.int32, "indices"), _ptr(ws),
            ws.numel() * ws.element_size(), _ptr(dev_status, torch.int32, "dev_status"),
            _stream(stream))
    keep = (batch, q_fp8, q_scale, w, index_pages, q_lat, latent_pages, out, lse, indices, ws,
            dev_status, stream)
    return PreparedCall("dsa_decode", load().dsa_decode, args, keep)


def prepare_append_cache(batch, new_keys, new_latent, kv_scale, index_pages, latent_pages,
                         key_format, dev_status=None, stream=None):
    """dsa_append_cache as a PreparedCall (same arguments)."""
    if stream is None:
        stream = torch.cuda.current_stream()
    args = (batch.ref(), _ptr(new_keys, torch.float32, "new_keys"),
            _ptr(new_latent, torch.float32, "new_latent"), float(kv_scale),
            _ptr(index_pages, torch.uint8, "index_pages"),
            _ptr(latent_pages, torch.uint8, "latent_pages"), int(key_format),
            _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    keep = (batch, new_keys, new_latent, index_pages, latent_pages, dev_status, stream)
    return PreparedCall("dsa_append_cache", load().dsa_append_cache, args, keep)


def dsa_decode_noalloc(batch, q_fp8, q_scale, w, index_pages, key_format, q_lat, latent_pages,
                       kv_scale, sm_scale, topk, out, lse, indices, dev_status=None, stream=None):
    """dsa_decode with no workspace argument, for callers that cannot allocate
    device memory on the call path: the scratch is a fixed array of
    NOALLOC_SCRATCH_BYTES inside the library, shared by all calls on a device
    (calls that overlap on the GPU race on it).  Batches that need more scratch
    raise DsaError with status 3."""
    rc = load().dsa_decode_noalloc(batch.ref(), _ptr(q_fp8, torch.uint8, "q_fp8"),
                                   _ptr(q_scale, torch.float32, "q_scale"),
                                   _ptr(w, torch.float32, "w"),
                                   _ptr(index_pages, torch.uint8, "index_pages"), int(key_format),
                                   _ptr(q_lat, (torch.bfloat16, torch.int16), "q_lat"),
                                   _ptr(latent_pages, torch.uint8, "latent_pages"),
                                   float(kv_scale), float(sm_scale), int(topk),
                                   _ptr(out, (torch.bfloat16, torch.int16), "out"),
                                   _ptr(lse, torch.float32, "lse"),
                                   _ptr(indices, torch.int32, "indices"),
                                   _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(rc, "dsa_decode_noalloc")


def dsa_dcp_topk_workspace_size(batch, world, cand=0, topk=TOPK):
    return int(load().dsa_dcp_topk_workspace_size(batch.ref(), int(world), int(cand), int(topk)))


def dsa_dcp_topk(batch, scores, score_ld, world, cand, topk, indices, rank_indices=None,
                 resent=None, ws=None, stream=None):
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    rc = load().dsa_dcp_topk(batch.ref(), _ptr(scores, torch.float32, "scores"), int(score_ld),
                             int(world), int(cand), int(topk),
                             _ptr(indices, torch.int32, "indices"),
                             _ptr(rank_indices, torch.int32, "rank_indices"),
                             _ptr(resent, torch.int32, "resent"), _ptr(ws), nbytes,
                             _stream(stream))
    _check(rc, "dsa_dcp_topk")


def dsa_lse_combine(total_q, world, part_out, part_lse, out, lse=None, stream=None):
    rc = load().dsa_lse_combine(int(total_q), int(world),
                                _ptr(part_out, (torch.bfloat16, torch.int16), "part_out"),
                                _ptr(part_lse, torch.float32, "part_lse"),
                                _ptr(out, (torch.bfloat16, torch.int16), "out"),
                                _ptr(lse, torch.float32, "lse"), _stream(stream))
    _check(rc, "dsa_lse_combine")


def dsa_indexer_front(batch, q_c, x, w_q, w_k, w_w, q_fp8, q_scale, w, index_pages=None,
                      key_format=KEYS_FP8, q_f32=None, k_f32=None, dev_status=None, stream=None):
    bf = (torch.bfloat16, torch.int16)
    rc = load().dsa_indexer_front(batch.ref(), _ptr(q_c, bf, "q_c"), _ptr(x, bf, "x"),
                                  _ptr(w_q, bf, "w_q"), _ptr(w_k, bf, "w_k"), _ptr(w_w, bf, "w_w"),
                                  _ptr(q_fp8, torch.uint8, "q_fp8"),
                                  _ptr(q_scale, torch.float32, "q_scale"),
                                  _ptr(w, torch.float32, "w"),
                                  _ptr(index_pages, torch.uint8, "index_pages"), int(key_format),
                                  _ptr(q_f32, torch.float32, "q_f32"),
                                  _ptr(k_f32, torch.float32, "k_f32"),
                                  _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check(rc, "dsa_indexer_front")


def dsa_plan_token_shards(seq_lens, q_counts, world, rank):
    """Parts of the batch's requests that rank `rank` of `world` runs in a
    token-sharded prefill (host only; see include/dsa.h)."""
    n = len(seq_lens)
    sl = (ctypes.c_int32 * n)(*[int(v) for v in seq_lens])
    qc = (ctypes.c_int32 * n)(*[int(v) for v in q_counts])
    cap = 2 * n
    parts = (ShardPart * max(cap, 1))()
    rc = load().dsa_plan_token_shards(sl, qc, n, int(world), int(rank), parts, cap)
    if rc < 0:
        raise DsaError(-rc, "dsa_plan_token_shards")
    return [ShardPart(p.request, p.token_begin, p.num_tokens, p.seq_len) for p in parts[:rc]]


def dsa_append_cache(batch, new_keys, new_latent, kv_scale, index_pages, latent_pages, key_format,
                     dev_status=None, stream=None):
    rc = load().dsa_append_cache(batch.ref(), _ptr(new_keys, torch.float32, "new_keys"),
                                 _ptr(new_latent, torch.float32, "new_latent"), float(kv_scale),
                                 _ptr(index_pages, torch.uint8, "index_pages"),
                                 _ptr(latent_pages, torch.uint8, "latent_pages"),
                                 int(key_format), _ptr(dev_status, torch.int32, "dev_status"),
                                 _stream(stream))
    _check(rc, "dsa_append_cache")
