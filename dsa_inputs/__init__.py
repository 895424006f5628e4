"""Seeded synthetic inputs for the DSA sparse-attention step.

This module only draws random numbers and lays bytes out in the cache page
formats; it holds none of the step's arithmetic.  Both the CPU oracle (in the
tests) and the CUDA library consume what it produces.  Quantisation of the
drawn values to FP8 uses PyTorch's own float8_e4m3fn conversion (a library
primitive); MXFP4 keys use a nearest-value table lookup written here.

Value recipe (one layer):
  index keys k ~ N(0,1) per token, FP8 E4M3 with fp32 scale amax/448 per token
             (or MXFP4: E2M1 elements with one E8M0 power-of-two scale per
             32-element block, shared exponent floor(log2(amax)) - 2)
  indexer query q ~ N(0,1) [T,32,128], FP8 with one scale amax/448 per token,
             stored per (token, head) in qscale [T,32]
  head weights w ~ N(0,1)/sqrt(32) [T,32] fp32
  MLA query q_lat ~ N(0,1) [T,96,576] bf16
  latents ~ N(0,1) [pool tokens, 576] FP8 E4M3 with one scale per layer
             kv_scale = amax(pool)/448; or NVFP4 (352 B per token): dims
             0..511 as E2M1 elements with one E4M3 scale per block of 16
             (block scale = E4M3(amax_block / 6 / kv_scale), element = nearest
             E2M1 value of x / (block scale * kv_scale)), dims 512..575 as
             E4M3(x / kv_scale)
  pages: each request's logical pages are placed on a seeded random
         permutation of one shared physical pool; unused block-table entries
         are -1.
"""
import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

PAGE = 64
IDX_HEADS = 32
IDX_DIM = 128
LAT_DIM = 576
V_DIM = 512
MLA_HEADS = 96
TOPK = 2048
FP8_PAGE_BYTES = PAGE * IDX_DIM + PAGE * 4        # 8448
MXFP4_PAGE_BYTES = PAGE * IDX_DIM // 2 + PAGE * 4  # 4352
LAT_PAGE_BYTES = PAGE * LAT_DIM                    # 36864
NVFP4_LAT_BYTES = V_DIM // 2 + V_DIM // 16 + (LAT_DIM - V_DIM)   # 256 + 32 + 64 = 352
NVFP4_LAT_PAGE_BYTES = PAGE * NVFP4_LAT_BYTES      # 22528
LATENT_FP8 = 0
LATENT_NVFP4 = 1
SM_SCALE = 1.0 / math.sqrt(192.0)
KEYS_FP8 = 0
KEYS_MXFP4 = 1

# E2M1 magnitudes in code order 0..7 (OCP MX element format).
_E2M1_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


@dataclass
class Layer:
    """One layer's paged caches plus one batch of queries for it."""
    q_offsets: torch.Tensor      # int32 [B+1]
    seq_lens: torch.Tensor       # int32 [B]
    block_table: torch.Tensor    # int32 [B, max_pages], -1 where unused
    num_pages: int
    key_format: int
    q8: torch.Tensor             # uint8 [T,32,128]
    qscale: torch.Tensor         # float32 [T,32]
    w: torch.Tensor              # float32 [T,32]
    index_pages: torch.Tensor    # uint8 [num_pages, page_bytes]
    q_lat: torch.Tensor          # bfloat16 [T,96,576]
    latent_pages: torch.Tensor   # uint8 [num_pages, 36864] (or [num_pages, 22528] NVFP4)
    kv_scale: float
    sm_scale: float = SM_SCALE
    seq_lens_host: List[int] = field(default_factory=list)
    q_counts_host: List[int] = field(default_factory=list)
    latent_format: int = LATENT_FP8

    @property
    def num_requests(self):
        return len(self.seq_lens_host)

    @property
    def total_q(self):
        return int(sum(self.q_counts_host))

    @property
    def max_pages(self):
        return int(self.block_table.shape[1])

    @property
    def max_seq_len(self):
        return int(max(self.seq_lens_host))

    def to(self, device):
        d = dict(self.__dict__)
        for k, v in d.items():
            if isinstance(v, torch.Tensor):
                d[k] = v.to(device)
        return Layer(**d)


def _fp8_per_row(x: torch.Tensor):
    """x [..., n] fp32 -> (E4M3 bytes, fp32 scale per row = amax/448)."""
    amax = x.abs().amax(dim=-1, keepdim=True)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (x / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale.squeeze(-1)


def _mxfp4_rows(x: torch.Tensor):
    """x [n, 128] fp32 -> (packed E2M1 bytes [n, 64], E8M0 bytes [n, 4])."""
    n = x.shape[0]
    blk = x.view(n, 4, 32)
    amax = blk.abs().amax(dim=-1)
    safe = torch.where(amax > 0, amax, torch.ones_like(amax))
    e = torch.floor(torch.log2(safe)) - 2.0
    e = torch.where(amax > 0, e, torch.full_like(e, -127.0)).clamp(-127.0, 127.0)
    scale_byte = (e + 127.0).to(torch.uint8)
    y = (blk / torch.exp2(e).unsqueeze(-1)).view(n, 128)
    mag = torch.tensor(_E2M1_MAG, device=x.device)
    bounds = (mag[1:] + mag[:-1]) / 2
    code = torch.bucketize(y.abs().clamp(max=6.0), bounds).to(torch.uint8)
    code = code | ((y < 0).to(torch.uint8) << 3)
    packed = code[:, 0::2] | (code[:, 1::2] << 4)
    return packed.contiguous(), scale_byte.contiguous()


def _e2m1_codes(y):
    """Nearest E2M1 code (sign in bit 3) of y, magnitudes clamped to 6."""
    mag = torch.tensor(_E2M1_MAG, device=y.device)
    bounds = (mag[1:] + mag[:-1]) / 2
    code = torch.bucketize(y.abs().clamp(max=6.0), bounds).to(torch.uint8)
    return code | ((y < 0).to(torch.uint8) << 3)


def _nvfp4_latent_rows(x, kv_scale):
    """x [n, 576] fp32 -> NVFP4 latent rows [n, 352]: packed E2M1 of dims
    0..511 (element 2i in the low nibble), 32 E4M3 block scales, E4M3 of
    dims 512..575."""
    n = x.shape[0]
    ks = torch.tensor(kv_scale, dtype=torch.float32, device=x.device)
    v = x[:, :V_DIM].reshape(n, V_DIM // 16, 16)
    sc = (v.abs().amax(dim=-1) / 6.0 / ks).to(torch.float8_e4m3fn)
    step = sc.to(torch.float32) * ks
    y = torch.where(step.unsqueeze(-1) > 0, v / step.unsqueeze(-1), torch.zeros_like(v))
    code = _e2m1_codes(y.reshape(n, V_DIM))
    packed = code[:, 0::2] | (code[:, 1::2] << 4)
    tail = (x[:, V_DIM:] / ks).to(torch.float8_e4m3fn).view(torch.uint8)
    return torch.cat([packed, sc.view(torch.uint8), tail], dim=1).contiguous()


def _randn(g, shape, device):
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)


def make_layer(seq_lens, n_q=1, key_format=KEYS_FP8, seed=0, device="cpu",
               extra_pages=0, chunk_tokens=1 << 18, latent_format=LATENT_FP8) -> Layer:
    """Build one layer for requests with the given context lengths (counted
    including the request's own query tokens) and n_q query tokens each."""
    seq_lens = [int(s) for s in seq_lens]
    B = len(seq_lens)
    q_counts = [int(n_q)] * B if isinstance(n_q, int) else [int(v) for v in n_q]
    assert len(q_counts) == B and all(1 <= q <= s for q, s in zip(q_counts, seq_lens))
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    pages_per_req = [(s + PAGE - 1) // PAGE for s in seq_lens]
    num_pages = sum(pages_per_req) + int(extra_pages)
    max_pages = max(pages_per_req)
    perm = torch.randperm(num_pages, generator=g, device=device).to(torch.int32)
    block_table = torch.full((B, max_pages), -1, dtype=torch.int32, device=device)
    o = 0
    for b, p in enumerate(pages_per_req):
        block_table[b, :p] = perm[o:o + p]
        o += p
    T = sum(q_counts)
    q_offsets = torch.tensor([0] + list(_cumsum(q_counts)), dtype=torch.int32, device=device)

    # indexer query: FP8 with one scale per token, broadcast over the 32 heads
    q = _randn(g, (T, IDX_HEADS * IDX_DIM), device)
    q8, qs = _fp8_per_row(q)
    q8 = q8.view(T, IDX_HEADS, IDX_DIM)
    qscale = qs.view(T, 1).expand(T, IDX_HEADS).contiguous()
    w = _randn(g, (T, IDX_HEADS), device) / math.sqrt(IDX_HEADS)
    q_lat = _randn(g, (T, MLA_HEADS, LAT_DIM), device).to(torch.bfloat16)

    # index key pool
    ntok = num_pages * PAGE
    if key_format == KEYS_FP8:
        pages = torch.empty((num_pages, FP8_PAGE_BYTES), dtype=torch.uint8, device=device)
        for t0 in range(0, ntok, chunk_tokens):
            t1 = min(ntok, t0 + chunk_tokens)
            p0, p1 = t0 // PAGE, t1 // PAGE
            k = _randn(g, (t1 - t0, IDX_DIM), device)
            codes, scale = _fp8_per_row(k)
            pages[p0:p1, :PAGE * IDX_DIM] = codes.view(p1 - p0, PAGE * IDX_DIM)
            pages[p0:p1, PAGE * IDX_DIM:] = scale.view(p1 - p0, PAGE).contiguous().view(
                torch.uint8).view(p1 - p0, PAGE * 4)
    elif key_format == KEYS_MXFP4:
        pages = torch.empty((num_pages, MXFP4_PAGE_BYTES), dtype=torch.uint8, device=device)
        for t0 in range(0, ntok, chunk_tokens):
            t1 = min(ntok, t0 + chunk_tokens)
            p0, p1 = t0 // PAGE, t1 // PAGE
            k = _randn(g, (t1 - t0, IDX_DIM), device)
            packed, sb = _mxfp4_rows(k)
            pages[p0:p1, :PAGE * IDX_DIM // 2] = packed.view(p1 - p0, PAGE * IDX_DIM // 2)
            pages[p0:p1, PAGE * IDX_DIM // 2:] = sb.view(p1 - p0, PAGE * 4)
    else:
        raise ValueError("key_format")

    # latent pool: one scale for the whole layer -> two passes over the same
    # seeded chunks (first for amax, then to quantise)
    lat_bytes = LAT_PAGE_BYTES if latent_format == LATENT_FP8 else NVFP4_LAT_PAGE_BYTES
    lat = torch.empty((num_pages, lat_bytes), dtype=torch.uint8, device=device)
    state = g.get_state()
    amax = torch.zeros((), device=device)
    for t0 in range(0, ntok, chunk_tokens):
        t1 = min(ntok, t0 + chunk_tokens)
        amax = torch.maximum(amax, _randn(g, (t1 - t0, LAT_DIM), device).abs().amax())
    kv_scale = float((amax / 448.0).to(torch.float32).item())  # an fp32 value
    g.set_state(state)
    for t0 in range(0, ntok, chunk_tokens):
        t1 = min(ntok, t0 + chunk_tokens)
        p0, p1 = t0 // PAGE, t1 // PAGE
        x = _randn(g, (t1 - t0, LAT_DIM), device)
        if latent_format == LATENT_FP8:
            codes = (x / torch.tensor(kv_scale, dtype=torch.float32, device=device)).to(
                torch.float8_e4m3fn).view(torch.uint8)
            lat[p0:p1] = codes.view(p1 - p0, LAT_PAGE_BYTES)
        else:
            lat[p0:p1] = _nvfp4_latent_rows(x, kv_scale).view(p1 - p0, NVFP4_LAT_PAGE_BYTES)

    return Layer(q_offsets=q_offsets, seq_lens=torch.tensor(seq_lens, dtype=torch.int32,
                                                            device=device),
                 block_table=block_table, num_pages=num_pages, key_format=key_format,
                 q8=q8, qscale=qscale, w=w, index_pages=pages, q_lat=q_lat,
                 latent_pages=lat, kv_scale=kv_scale, seq_lens_host=seq_lens,
                 q_counts_host=q_counts, latent_format=latent_format)


def _cumsum(v):
    s = 0
    for x in v:
        s += x
        yield s


# ---- the five workloads ------------------------------------------------------

CONFIGS = {
    "c0_tiny": "1 request, ctx 4096, 1 query token, 64 pages",
    "c1_batched": "8 requests, ctx ~ U[16384, 32768], 1 query token each",
    "c2_agentic": "64 requests, ctx 131072, 5 causal query tokens each",
    "c3a_long_fp8": "1 request, ctx 1048576, 1 query token, FP8 index keys",
    "c3b_long_mxfp4": "1 request, ctx 1048576, 1 query token, MXFP4 index keys",
    "c4_prefill_append": "1 request, 2048 new tokens appended to a 153600-token prefix",
}


def config_shape(name: str, seed: Optional[int] = None):
    """(seq_lens, n_q, key_format, seed) of a named workload.  'K' = 1024."""
    cid = {"c0_tiny": 0, "c1_batched": 1, "c2_agentic": 2, "c3a_long_fp8": 3,
           "c3b_long_mxfp4": 3, "c4_prefill_append": 4}[name]
    seed = 1000 + cid if seed is None else seed
    if name == "c0_tiny":
        return [4096], 1, KEYS_FP8, seed
    if name == "c1_batched":
        g = torch.Generator().manual_seed(seed)
        lens = torch.randint(16384, 32768 + 1, (8,), generator=g).tolist()
        return lens, 1, KEYS_FP8, seed
    if name == "c2_agentic":
        return [131072] * 64, 5, KEYS_FP8, seed
    if name == "c3a_long_fp8":
        return [1048576], 1, KEYS_FP8, seed
    if name == "c3b_long_mxfp4":
        return [1048576], 1, KEYS_MXFP4, seed
    if name == "c4_prefill_append":
        return [153600 + 2048], 2048, KEYS_FP8, seed
    raise KeyError(name)


def make_config(name: str, device="cpu", seed: Optional[int] = None) -> Layer:
    lens, nq, fmt, sd = config_shape(name, seed)
    return make_layer(lens, nq, fmt, sd, device)


def append_payload(layer: Layer, seed: int):
    """fp32 new-token keys [T,128] and latents [T,576] for a cache append (the
    new tokens are the query tokens of the batch), drawn N(0,1)."""
    g = torch.Generator(device=layer.q8.device)
    g.manual_seed(int(seed))
    T = layer.total_q
    keys = _randn(g, (T, IDX_DIM), layer.q8.device)
    lat = _randn(g, (T, LAT_DIM), layer.q8.device)
    return keys, lat
