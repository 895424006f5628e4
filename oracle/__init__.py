"""CPU oracle for the DSA sparse-attention step -- TEST INFRASTRUCTURE.

A plain, slow, fp64 C implementation (``dsa_oracle.c``) of what one DSA layer
step computes, behind ctypes.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg use it.  It shares no code with the CUDA library
and never calls it.

Every function takes plain numpy arrays (or anything ``np.asarray`` accepts)
in the layouts of the paged caches:

* FP8 index page: 64 x 128 E4M3 bytes then 64 fp32 scales (8448 B).
* MXFP4 index page: 64 x 64 packed E2M1 bytes (element 2i in the low nibble)
  then 64 x 4 E8M0 scales (4352 B).
* Latent page: 64 x 576 E4M3 bytes (36864 B), one scale per layer.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

ORC_ERRORS = {-1: "bad argument", -2: "page id out of range", -3: "index out of range",
              -4: "NaN score", -5: "out of memory"}

_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_e4m3_decode.restype = ctypes.c_double
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e2m1_decode.restype = ctypes.c_double
        L.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e8m0_decode.restype = ctypes.c_double
        L.oracle_e8m0_decode.argtypes = [ctypes.c_uint8]
        L.oracle_bf16_decode.restype = ctypes.c_double
        L.oracle_bf16_decode.argtypes = [ctypes.c_uint16]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_e4m3_decode_array.argtypes = [_u8p, _f64p, ctypes.c_int64]
        L.oracle_e4m3_encode_array.argtypes = [_f32p, _u8p, ctypes.c_int64]
        L.oracle_constants.argtypes = [_i32p, ctypes.c_int32]
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_index_scores.argtypes = [
            ctypes.c_int32, _i32p, _i32p, _i32p, ctypes.c_int32, ctypes.c_int32,
            _u8p, _f32p, _f32p, _u8p, ctypes.c_int32, _i32p, ctypes.c_int32,
            ctypes.c_int64, _f64p, _f64p]
        L.oracle_topk_row.argtypes = [_f64p, ctypes.c_int64, ctypes.c_int32, _i32p]
        L.oracle_topk.argtypes = [_f64p, ctypes.c_int64, _i64p, ctypes.c_int32,
                                  ctypes.c_int32, _i32p]
        L.oracle_visible.argtypes = [ctypes.c_int32, _i32p, _i32p, _i32p, ctypes.c_int32,
                                     _i64p]
        L.oracle_sparse_mla.argtypes = [
            ctypes.c_int32, _i32p, _i32p, _i32p, ctypes.c_int32, ctypes.c_int32,
            _u16p, _u8p, ctypes.c_double, ctypes.c_double, _i32p, ctypes.c_int32,
            _i32p, ctypes.c_int32, _f64p, _f64p]
        L.oracle_decode.argtypes = [
            ctypes.c_int32, _i32p, _i32p, _i32p, ctypes.c_int32, ctypes.c_int32,
            _u8p, _f32p, _f32p, _u8p, ctypes.c_int32, _u16p, _u8p, ctypes.c_double,
            ctypes.c_double, ctypes.c_int32, _i32p, ctypes.c_int32, _i32p, _f64p, _f64p]
        L.oracle_append_cache.argtypes = [
            ctypes.c_int32, _i32p, _i32p, _i32p, ctypes.c_int32, ctypes.c_int32,
            _f32p, _f32p, ctypes.c_float, _u8p, _u8p, ctypes.c_int32]
        L.oracle_latent_row.argtypes = [ctypes.c_int32, _u8p, ctypes.c_double, _f64p]
        L.oracle_sparse_mla_fmt.argtypes = [
            ctypes.c_int32, _i32p, _i32p, _i32p, ctypes.c_int32, ctypes.c_int32,
            _u16p, _u8p, ctypes.c_int32, ctypes.c_double, ctypes.c_double, _i32p, ctypes.c_int32,
            _i32p, ctypes.c_int32, _f64p, _f64p]
        L.oracle_decode_fmt.argtypes = [
            ctypes.c_int32, _i32p, _i32p, _i32p, ctypes.c_int32, ctypes.c_int32,
            _u8p, _f32p, _f32p, _u8p, ctypes.c_int32, _u16p, _u8p, ctypes.c_int32,
            ctypes.c_double, ctypes.c_double, ctypes.c_int32, _i32p, ctypes.c_int32, _i32p, _f64p,
            _f64p]
        for name in ("oracle_latent_row", "oracle_sparse_mla_fmt", "oracle_decode_fmt"):
            getattr(L, name).restype = ctypes.c_int
        L.oracle_indexer_front.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _u16p,
                                           _u16p, _u16p, _u16p, _u16p, _f64p, _f64p, _f64p, _f64p]
        L.oracle_quantize_rows.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int32, _u8p, _f32p]
        for name in ("oracle_indexer_front", "oracle_quantize_rows"):
            getattr(L, name).restype = ctypes.c_int
        L.oracle_bf16_encode.restype = ctypes.c_uint16
        L.oracle_bf16_encode.argtypes = [ctypes.c_float]
        L.oracle_bf16_encode_array.argtypes = [_f32p, _u16p, ctypes.c_int64]
        L.oracle_dcp_topk_row.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_int32, _i32p, _i32p]
        L.oracle_dcp_topk.argtypes = [_f32p, ctypes.c_int64, _i64p, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _i32p,
                                      _i32p]
        L.oracle_lse_combine.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, _f64p,
                                         _f64p, _f64p, _f64p]
        for name in ("oracle_index_scores", "oracle_topk_row", "oracle_topk", "oracle_visible",
                     "oracle_sparse_mla", "oracle_decode", "oracle_append_cache",
                     "oracle_constants", "oracle_dcp_topk_row", "oracle_dcp_topk",
                     "oracle_lse_combine"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _arr(x, dtype):
    """Contiguous numpy view/copy of x with the given dtype.  Same-width
    integer types and torch bf16 / fp8 tensors are reinterpreted bit-wise."""
    dtype = np.dtype(dtype)
    if hasattr(x, "detach"):  # torch tensor
        import torch
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            x = x.view(torch.int16)
        elif x.dtype == torch.float8_e4m3fn:
            x = x.view(torch.uint8)
        x = x.numpy()
    a = np.asarray(x)
    if a.dtype != dtype:
        if a.dtype.itemsize == dtype.itemsize and a.dtype.kind in "iu" and dtype.kind in "iu":
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return np.ascontiguousarray(a)


def _p(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _check(rc, what):
    if rc != 0:
        raise RuntimeError("oracle %s failed: %s" % (what, ORC_ERRORS.get(rc, rc)))


def constants():
    out = np.zeros(16, np.int32)
    n = lib().oracle_constants(_p(out, ctypes.c_int32), 16)
    names = ["page_tokens", "idx_heads", "idx_dim", "lat_dim", "v_dim", "mla_heads",
             "fp8_key_bytes_per_token", "fp8_page_bytes", "mxfp4_key_bytes_per_token",
             "mxfp4_page_bytes", "lat_bytes_per_token", "lat_page_bytes"]
    return dict(zip(names, out[:n].tolist()))


def num_threads():
    return lib().oracle_num_threads()


def e4m3_decode(codes):
    c = _arr(codes, np.uint8).ravel()
    out = np.empty(c.size, np.float64)
    lib().oracle_e4m3_decode_array(_p(c, ctypes.c_uint8), _p(out, ctypes.c_double), c.size)
    return out.reshape(np.shape(codes))


def e4m3_encode(values):
    v = _arr(values, np.float32).ravel()
    out = np.empty(v.size, np.uint8)
    lib().oracle_e4m3_encode_array(_p(v, ctypes.c_float), _p(out, ctypes.c_uint8), v.size)
    return out.reshape(np.shape(values))


def e2m1_decode(nibble):
    return lib().oracle_e2m1_decode(int(nibble))


def e8m0_decode(code):
    return lib().oracle_e8m0_decode(int(code))


def bf16_decode(bits):
    return lib().oracle_bf16_decode(int(bits))


class Batch:
    """Request metadata as the oracle reads it (host arrays)."""

    def __init__(self, q_offsets, seq_lens, block_table, num_pages):
        self.q_offsets = _arr(q_offsets, np.int32)
        self.seq_lens = _arr(seq_lens, np.int32)
        bt = _arr(block_table, np.int32)
        self.block_table = bt.reshape(len(self.seq_lens), -1)
        self.max_pages = self.block_table.shape[1]
        self.num_pages = int(num_pages)
        self.num_requests = len(self.seq_lens)
        self.total_q = int(self.q_offsets[-1])

    def args(self):
        return (self.num_requests, _p(self.q_offsets, ctypes.c_int32),
                _p(self.seq_lens, ctypes.c_int32), _p(self.block_table, ctypes.c_int32),
                self.max_pages, self.num_pages)

    def visible(self, rows):
        rows = _arr(rows, np.int32)
        vis = np.zeros(rows.size, np.int64)
        _check(lib().oracle_visible(self.num_requests, _p(self.q_offsets, ctypes.c_int32),
                                    _p(self.seq_lens, ctypes.c_int32),
                                    _p(rows, ctypes.c_int32), rows.size,
                                    _p(vis, ctypes.c_int64)), "visible")
        return vis


def _rows(batch, rows):
    if rows is None:
        rows = np.arange(batch.total_q, dtype=np.int32)
    return _arr(rows, np.int32)


def index_scores(batch, q8, qscale, w, index_pages, key_format=0, rows=None, ld=None,
                 with_abs=True):
    """fp64 indexer scores S [nrows, ld] (-inf past the causal limit) and the
    magnitude A = sum_h |w| sum_d |qhat khat| used for the tolerance."""
    rows = _rows(batch, rows)
    if ld is None:
        ld = int(batch.seq_lens.max())
    q8 = _arr(q8, np.uint8)
    qscale = _arr(qscale, np.float32)
    w = _arr(w, np.float32)
    pages = _arr(index_pages, np.uint8)
    S = np.empty((rows.size, ld), np.float64)
    A = np.empty((rows.size, ld), np.float64) if with_abs else None
    _check(lib().oracle_index_scores(*batch.args(), _p(q8, ctypes.c_uint8),
                                     _p(qscale, ctypes.c_float), _p(w, ctypes.c_float),
                                     _p(pages, ctypes.c_uint8), int(key_format),
                                     _p(rows, ctypes.c_int32), rows.size, ld,
                                     _p(S, ctypes.c_double),
                                     _p(A, ctypes.c_double) if with_abs else None),
           "index_scores")
    return S, A


def topk_row(scores, n_visible, k=2048):
    s = _arr(scores, np.float64)
    out = np.empty(k, np.int32)
    _check(lib().oracle_topk_row(_p(s, ctypes.c_double), int(n_visible), k,
                                 _p(out, ctypes.c_int32)), "topk_row")
    return out


def topk(scores, n_visible, k=2048):
    """Row-wise exact top-k of a [nrows, ld] score matrix; row r uses its first
    n_visible[r] entries.  Ascending positions, -1 padded."""
    s = _arr(scores, np.float64)
    nv = _arr(n_visible, np.int64)
    out = np.empty((s.shape[0], k), np.int32)
    _check(lib().oracle_topk(_p(s, ctypes.c_double), s.shape[1], _p(nv, ctypes.c_int64),
                             s.shape[0], k, _p(out, ctypes.c_int32)), "topk")
    return out


def latent_row(row_bytes, kv_scale, latent_format=0):
    """Dequantised latent [576] of one token from its stored bytes (576 B FP8
    or 352 B NVFP4)."""
    r = _arr(row_bytes, np.uint8)
    out = np.empty(576, np.float64)
    _check(lib().oracle_latent_row(int(latent_format), _p(r, ctypes.c_uint8), float(kv_scale),
                                   _p(out, ctypes.c_double)), "latent_row")
    return out


def sparse_mla(batch, q_lat_bf16, latent_pages, kv_scale, sm_scale, indices, rows=None,
               latent_format=0):
    """fp64 absorbed sparse MLA over the selected positions of each row.
    q_lat_bf16: bf16 bit patterns [T, 96, 576] (uint16 or torch.bfloat16).
    indices: [nrows, k] logical positions (-1 = unused).
    latent_format: 0 = FP8 pages (576 B per token), 1 = NVFP4 pages (352 B)."""
    rows = _rows(batch, rows)
    q = _arr(q_lat_bf16, np.uint16)
    lat = _arr(latent_pages, np.uint8)
    idx = _arr(indices, np.int32)
    k = idx.shape[1]
    out = np.empty((rows.size, 96, 512), np.float64)
    lse = np.empty((rows.size, 96), np.float64)
    _check(lib().oracle_sparse_mla_fmt(*batch.args(), _p(q, ctypes.c_uint16),
                                       _p(lat, ctypes.c_uint8), int(latent_format),
                                       float(kv_scale), float(sm_scale),
                                       _p(idx, ctypes.c_int32), k, _p(rows, ctypes.c_int32),
                                       rows.size, _p(out, ctypes.c_double),
                                       _p(lse, ctypes.c_double)), "sparse_mla")
    return out, lse


def decode(batch, q8, qscale, w, index_pages, key_format, q_lat_bf16, latent_pages, kv_scale,
           sm_scale, k=2048, rows=None, latent_format=0):
    """The whole step (scores -> top-k -> sparse MLA) for the listed rows."""
    rows = _rows(batch, rows)
    q8 = _arr(q8, np.uint8)
    qscale = _arr(qscale, np.float32)
    w = _arr(w, np.float32)
    pages = _arr(index_pages, np.uint8)
    q = _arr(q_lat_bf16, np.uint16)
    lat = _arr(latent_pages, np.uint8)
    idx = np.empty((rows.size, k), np.int32)
    out = np.empty((rows.size, 96, 512), np.float64)
    lse = np.empty((rows.size, 96), np.float64)
    _check(lib().oracle_decode_fmt(*batch.args(), _p(q8, ctypes.c_uint8),
                                   _p(qscale, ctypes.c_float), _p(w, ctypes.c_float),
                                   _p(pages, ctypes.c_uint8), int(key_format),
                                   _p(q, ctypes.c_uint16), _p(lat, ctypes.c_uint8),
                                   int(latent_format), float(kv_scale),
                                   float(sm_scale), k, _p(rows, ctypes.c_int32), rows.size,
                               _p(idx, ctypes.c_int32), _p(out, ctypes.c_double),
                               _p(lse, ctypes.c_double)), "decode")
    return idx, out, lse


def append_cache(batch, new_keys, new_latent, kv_scale, index_pages, latent_pages, key_format=0):
    """Returns updated copies of (index_pages, latent_pages)."""
    ip = None if index_pages is None else np.array(_arr(index_pages, np.uint8), copy=True)
    lp = None if latent_pages is None else np.array(_arr(latent_pages, np.uint8), copy=True)
    nk = None if new_keys is None else _arr(new_keys, np.float32)
    nl = None if new_latent is None else _arr(new_latent, np.float32)
    _check(lib().oracle_append_cache(*batch.args(),
                                     None if nk is None else _p(nk, ctypes.c_float),
                                     None if nl is None else _p(nl, ctypes.c_float),
                                     float(kv_scale),
                                     None if ip is None else _p(ip, ctypes.c_uint8),
                                     None if lp is None else _p(lp, ctypes.c_uint8),
                                     int(key_format)), "append_cache")
    return ip, lp


# ---- decode context parallelism ------------------------------------------------

def bf16_encode(values):
    """bfloat16 codes (round to nearest even) of binary32 values."""
    a = _arr(values, np.float32).reshape(-1)
    out = np.empty(a.size, np.uint16)
    lib().oracle_bf16_encode_array(_p(a, ctypes.c_float), _p(out, ctypes.c_uint16), a.size)
    return out.reshape(np.shape(values))


def dcp_cand(world, k=2048):
    """Candidates each rank sends: ceil(1.5 k / world), at most k (no rank
    needs to send more than the k it could contribute)."""
    return min(-(-3 * k // (2 * world)), k)


def dcp_topk(scores, n_visible, world, cand=None, k=2048):
    """Row-wise merged selection of decode context parallelism over `world`
    ranks (rank r holds positions s = r mod world): the k visible positions
    with the largest BF16-rounded scores, ties to the lower position, in
    ascending order, -1 padded; and per row which ranks resend their full local
    top-k.  scores: [rows, ld] binary32 (the scores as computed)."""
    s = _arr(scores, np.float32)
    if s.ndim == 1:
        s = s.reshape(1, -1)
    nv = _arr(np.atleast_1d(n_visible), np.int64)
    cand = dcp_cand(world, k) if cand is None else int(cand)
    out = np.empty((s.shape[0], k), np.int32)
    resend = np.empty((s.shape[0], world), np.int32)
    _check(lib().oracle_dcp_topk(_p(s, ctypes.c_float), s.shape[1], _p(nv, ctypes.c_int64),
                                 s.shape[0], int(world), cand, int(k), _p(out, ctypes.c_int32),
                                 _p(resend, ctypes.c_int32)), "dcp_topk")
    return out, resend


def lse_combine(parts, lses):
    """Log-sum-exp combine of partial attention results over disjoint token
    sets: parts [world, ..., dim], lses [world, ...] (natural log)."""
    p = _arr(parts, np.float64)
    l = _arr(lses, np.float64)
    world = p.shape[0]
    dim = p.shape[-1]
    rows = int(np.prod(p.shape[1:-1])) if p.ndim > 2 else 1
    out = np.empty((rows, dim), np.float64)
    lse = np.empty(rows, np.float64)
    _check(lib().oracle_lse_combine(world, rows, dim, _p(p, ctypes.c_double),
                                    _p(l, ctypes.c_double), _p(out, ctypes.c_double),
                                    _p(lse, ctypes.c_double)), "lse_combine")
    return out.reshape(p.shape[1:]), lse.reshape(l.shape[1:])


# ---- fused indexer front ------------------------------------------------------

def indexer_front(q_c, x, w_q, w_k, w_w):
    """fp64 indexer front for T tokens: q [T, 4096] (normed query projection),
    w [T, 32] head weights, key [T, 128] new index keys, inv_rms [T].
    Inputs are bf16 bit patterns (uint16 / int16 / torch.bfloat16):
    q_c [T, dq], x [T, dh], w_q [4096, dq], w_k [128, dh], w_w [32, dh]."""
    qc = _arr(q_c, np.uint16)
    xx = _arr(x, np.uint16)
    T, dq = qc.shape
    dh = xx.shape[1]
    wq = _arr(w_q, np.uint16)
    wk = _arr(w_k, np.uint16)
    ww = _arr(w_w, np.uint16)
    assert wq.shape == (4096, dq) and wk.shape == (128, dh) and ww.shape == (32, dh)
    q = np.empty((T, 4096), np.float64)
    w = np.empty((T, 32), np.float64)
    key = np.empty((T, 128), np.float64)
    inv = np.empty(T, np.float64)
    _check(lib().oracle_indexer_front(T, dq, dh, _p(qc, ctypes.c_uint16), _p(xx, ctypes.c_uint16),
                                      _p(wq, ctypes.c_uint16), _p(ww, ctypes.c_uint16),
                                      _p(wk, ctypes.c_uint16), _p(q, ctypes.c_double),
                                      _p(w, ctypes.c_double), _p(key, ctypes.c_double),
                                      _p(inv, ctypes.c_double)), "indexer_front")
    return q, w, key, inv


def quantize_rows(x, dim):
    """The cache writer's per-row FP8 rule on binary32 values: codes [n, dim]
    (uint8) and scales [n] (float32)."""
    v = _arr(x, np.float32).reshape(-1, dim)
    codes = np.empty(v.shape, np.uint8)
    scales = np.empty(v.shape[0], np.float32)
    _check(lib().oracle_quantize_rows(_p(v, ctypes.c_float), v.shape[0], dim,
                                      _p(codes, ctypes.c_uint8), _p(scales, ctypes.c_float)),
           "quantize_rows")
    return codes, scales
