"""Seeded synthetic inputs for MLA paged-KV decode.

This module only draws inputs.  It holds none of the decode arithmetic, and
both the CUDA path and the CPU oracle consume what it produces.  Everything
is drawn on the CPU from ``torch.Generator().manual_seed(seed)``.

Dense recipe (FlashMLA PR #183 layout: 64-token pages of 576 bf16 latent
entries, a block table per request):
  * cache_seqlens[b] ~ uniform integers in [lo, hi], i.i.d. per request;
  * pages per request = ceil(L_b / 64); the pool holds ceil(1.2 * total)
    pages and every request draws its pages without replacement from one
    random permutation of the pool, so logical order != physical order;
  * Q and KV ~ N(0, 1), rounded to bf16; ``q_scale`` multiplies Q before
    rounding (8 gives "peaky" softmax rows);
  * every slot no request uses (tail slots of a last page, unused pages) is
    filled with finite poison (+-1e3) so a masking error cannot hide;
  * block-table entries past ceil(L_b / 64) are -1.

Sparse FP8 recipe (FlashMLA PR #200: 656-byte records of 512 E4M3 codes,
four fp32 scales, 64 bf16 RoPE values; physical slot indices; topk_length):
  * each request owns ``pages_per_req`` pages of the pool, the page sets are
    disjoint and randomly placed (a random request-disjoint block table);
  * each query token selects ``topk`` distinct logical positions of its
    request, mapped to physical slots page*64 + position % 64;
  * topk_length[b, i] ~ uniform integers in [lo, hi]; entries at or past it
    are -1;
  * NoPE values x ~ N(0, 1) in fp32, quantised per 128-element group with
    scale = max|x| / 448 and codes = E4M3(x / scale) (round to nearest even,
    clamped to +-448); RoPE ~ N(0, 1) rounded to bf16.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

PAGE = 64
D_QK = 576
D_V = 512
RECORD = 656
POISON = 1.0e3


@dataclass
class DenseCase:
    q: torch.Tensor              # bf16 [B, s_q, h_q, 576]
    kv: torch.Tensor             # bf16 [num_pages, 64, 576]
    block_table: torch.Tensor    # int32 [B, max_pages], -1 past the used pages
    cache_seqlens: torch.Tensor  # int32 [B]
    causal: bool
    scale: float
    out_fp32: bool
    name: str = ""

    @property
    def batch(self):
        return self.q.shape[0]

    @property
    def s_q(self):
        return self.q.shape[1]

    @property
    def h_q(self):
        return self.q.shape[2]

    @property
    def h_kv(self):
        return 1 if self.kv.dim() == 3 else self.kv.shape[2]

    def kv_bytes(self) -> int:
        """Unique KV bytes read: every valid token's 576 16-bit entries once per KV head."""
        return int(self.cache_seqlens.to(torch.int64).sum().item()) * D_QK * 2 * self.h_kv


@dataclass
class SparseCase:
    q: torch.Tensor              # bf16 [B, s_q, h_q, 576]
    kv8: torch.Tensor            # uint8 [num_pages, 64, 656]
    indices: torch.Tensor        # int32 [B, s_q, topk]
    topk_length: torch.Tensor    # int32 [B, s_q]
    scale: float
    name: str = ""

    @property
    def batch(self):
        return self.q.shape[0]

    @property
    def s_q(self):
        return self.q.shape[1]

    @property
    def h_q(self):
        return self.q.shape[2]

    def kv_bytes(self) -> int:
        """Record bytes read: 656 per valid selected slot."""
        topk = self.indices.shape[2]
        t = torch.arange(topk)[None, None, :]
        valid = (t < self.topk_length[:, :, None]) & (self.indices != -1)
        return int(valid.sum().item()) * RECORD


def _gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed))


def dense_case(batch, s_q, h_q, seqlen_lo, seqlen_hi=None, *, causal=False, seed=0,
               pool_factor=1.2, q_scale=1.0, out_fp32=False, seqlens=None,
               scale=None, poison=True, name="", h_kv=1, dtype=torch.bfloat16) -> DenseCase:
    """Seeded dense case: N(0,1) latent rows in a shuffled 64-token page pool
    (1.2x the pages in use; unused slots hold +-1e3 poison), the block table,
    and q.  h_kv > 1 gives a [pages, 64, h_kv, 576] cache; dtype is that of q
    and the cache (bf16 or fp16)."""
    g = _gen(seed)
    if seqlens is None:
        hi = seqlen_lo if seqlen_hi is None else seqlen_hi
        seqlens = torch.randint(seqlen_lo, hi + 1, (batch,), generator=g, dtype=torch.int64)
    seqlens = torch.as_tensor(seqlens, dtype=torch.int64).reshape(batch)
    npg = [(int(L) + PAGE - 1) // PAGE for L in seqlens.tolist()]
    total = sum(npg)
    pool = max(int(math.ceil(pool_factor * total)), total, 1)
    perm = torch.randperm(pool, generator=g)
    max_pages = max(max(npg), 1)
    bt = torch.full((batch, max_pages), -1, dtype=torch.int32)
    pos = 0
    for b in range(batch):
        bt[b, :npg[b]] = perm[pos:pos + npg[b]].to(torch.int32)
        pos += npg[b]
    kv = torch.randn(pool, PAGE, D_QK, generator=g) if h_kv == 1 else torch.randn(pool, PAGE, h_kv, D_QK,
                                                                                      generator=g)
    if poison:
        used = torch.zeros(pool, PAGE, dtype=torch.bool)
        for b in range(batch):
            L = int(seqlens[b])
            for lp in range(npg[b]):
                n = min(PAGE, L - lp * PAGE)
                used[int(bt[b, lp]), :n] = True
        sign = torch.where(torch.rand(pool, PAGE, 1, generator=g) < 0.5, -1.0, 1.0)
        if h_kv > 1:
            used, sign = used[:, :, None], sign[:, :, None]
        kv = torch.where(used[..., None], kv, sign * POISON)
    kv = kv.to(dtype)
    q = (torch.randn(batch, s_q, h_q, D_QK, generator=g) * q_scale).to(dtype)
    return DenseCase(q=q, kv=kv, block_table=bt, cache_seqlens=seqlens.to(torch.int32),
                     causal=bool(causal), scale=(1.0 / math.sqrt(D_QK)) if scale is None else scale,
                     out_fp32=bool(out_fp32), name=name)


def _quantise_records(x: torch.Tensor, rope: torch.Tensor) -> torch.Tensor:
    """x: fp32 [n, 512], rope: bf16 [n, 64] -> uint8 [n, 656] records."""
    n = x.shape[0]
    groups = x.reshape(n, 4, 128)
    amax = groups.abs().amax(dim=2)
    sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).to(torch.float32)
    y = (groups / sc[:, :, None]).clamp(-448.0, 448.0)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(n, 512)
    rec = torch.empty(n, RECORD, dtype=torch.uint8)
    rec[:, :512] = codes
    rec[:, 512:528] = sc.contiguous().view(torch.uint8).reshape(n, 16)
    rec[:, 528:656] = rope.contiguous().view(torch.uint8).reshape(n, 128)
    return rec


@dataclass
class DenseFp8Case:
    q: torch.Tensor              # bf16 [B, s_q, h_q, 576]
    kv8: torch.Tensor            # uint8 [num_pages, 64, 656]
    block_table: torch.Tensor    # int32 [B, max_pages]
    cache_seqlens: torch.Tensor  # int32 [B]
    causal: bool
    scale: float
    name: str = ""

    @property
    def batch(self):
        return self.q.shape[0]

    @property
    def s_q(self):
        return self.q.shape[1]

    @property
    def h_q(self):
        return self.q.shape[2]

    def kv_bytes(self) -> int:
        """Record bytes read: every valid token's 656-byte record once."""
        return int(self.cache_seqlens.to(torch.int64).sum().item()) * RECORD


def dense_fp8_case(batch, s_q, h_q, seqlen_lo, seqlen_hi=None, *, causal=False, seed=0, pool_factor=1.2,
                   q_scale=1.0, seqlens=None, scale=None, poison=True, name="") -> DenseFp8Case:
    """Seeded paged cache of FP8 records (N(0,1) rows quantised as for the sparse cases, bf16
    RoPE), shuffled pages (1.2x the pages in use) and the block table; unused slots carry
    1e3x scales as poison."""
    g = _gen(seed)
    if seqlens is None:
        hi = seqlen_lo if seqlen_hi is None else seqlen_hi
        seqlens = torch.randint(seqlen_lo, hi + 1, (batch,), generator=g, dtype=torch.int64)
    seqlens = torch.as_tensor(seqlens, dtype=torch.int64).reshape(batch)
    npg = [(int(L) + PAGE - 1) // PAGE for L in seqlens.tolist()]
    total = sum(npg)
    pool = max(int(math.ceil(pool_factor * total)), total, 1)
    perm = torch.randperm(pool, generator=g)
    max_pages = max(max(npg), 1)
    bt = torch.full((batch, max_pages), -1, dtype=torch.int32)
    pos = 0
    for b in range(batch):
        bt[b, :npg[b]] = perm[pos:pos + npg[b]].to(torch.int32)
        pos += npg[b]
    x = torch.randn(pool * PAGE, 512, generator=g)
    rope = torch.randn(pool * PAGE, 64, generator=g).to(torch.bfloat16)
    kv8 = _quantise_records(x, rope).reshape(pool, PAGE, RECORD)
    if poison:
        used = torch.zeros(pool, PAGE, dtype=torch.bool)
        for b in range(batch):
            L = int(seqlens[b])
            for lp in range(npg[b]):
                used[int(bt[b, lp]), :min(PAGE, L - lp * PAGE)] = True
        flat = kv8.view(pool * PAGE, RECORD)
        scales = flat[:, 512:528].contiguous().view(torch.float32).reshape(-1, 4)
        scales[~used.reshape(-1)] *= POISON
        flat[:, 512:528] = scales.contiguous().view(torch.uint8).reshape(-1, 16)
    q = (torch.randn(batch, s_q, h_q, D_QK, generator=g) * q_scale).to(torch.bfloat16)
    return DenseFp8Case(q=q, kv8=kv8, block_table=bt, cache_seqlens=seqlens.to(torch.int32), causal=bool(causal),
                        scale=(1.0 / math.sqrt(D_QK)) if scale is None else scale, name=name)


def sparse_case(batch, s_q, h_q, *, topk=2048, pages_per_req=512, topk_lo=1024,
                topk_hi=2048, seed=0, q_scale=1.0, poison=True, topk_lengths=None,
                scale=None, name="") -> SparseCase:
    g = _gen(seed)
    num_pages = batch * pages_per_req
    perm = torch.randperm(num_pages, generator=g)
    bt = perm.reshape(batch, pages_per_req)
    n_log = pages_per_req * PAGE
    assert topk <= n_log
    indices = torch.empty(batch, s_q, topk, dtype=torch.int32)
    if topk_lengths is None:
        topk_lengths = torch.randint(topk_lo, topk_hi + 1, (batch, s_q), generator=g)
    topk_lengths = torch.as_tensor(topk_lengths, dtype=torch.int64).reshape(batch, s_q)
    for b in range(batch):
        for i in range(s_q):
            lpos = torch.randperm(n_log, generator=g)[:topk]
            phys = bt[b][lpos // PAGE] * PAGE + (lpos % PAGE)
            tl = int(topk_lengths[b, i])
            phys = phys.to(torch.int32)
            phys[tl:] = -1
            indices[b, i] = phys
    kv8 = torch.empty(num_pages, PAGE, RECORD, dtype=torch.uint8)
    chunk = 256
    for p0 in range(0, num_pages, chunk):
        p1 = min(num_pages, p0 + chunk)
        n = (p1 - p0) * PAGE
        x = torch.randn(n, 512, generator=g)
        rope = torch.randn(n, 64, generator=g).to(torch.bfloat16)
        kv8[p0:p1] = _quantise_records(x, rope).reshape(p1 - p0, PAGE, RECORD)
    if poison:
        sel = torch.zeros(num_pages * PAGE, dtype=torch.bool)
        valid = indices[indices >= 0].to(torch.int64)
        sel[valid] = True
        flat = kv8.view(num_pages * PAGE, RECORD)
        scales = flat[:, 512:528].contiguous().view(torch.float32).reshape(-1, 4)
        scales[~sel] = scales[~sel] * POISON
        flat[:, 512:528] = scales.contiguous().view(torch.uint8).reshape(-1, 16)
    q = (torch.randn(batch, s_q, h_q, D_QK, generator=g) * q_scale).to(torch.bfloat16)
    return SparseCase(q=q, kv8=kv8, indices=indices, topk_length=topk_lengths.to(torch.int32),
                      scale=(1.0 / math.sqrt(D_QK)) if scale is None else scale, name=name)


# The workloads the benchmark and the parity tests use, named by shape.
WORKLOADS = {
    "dense_b1_hq16_sk256_fp32out": dict(kind="dense", batch=1, s_q=1, h_q=16, seqlen_lo=256,
                                        seqlen_hi=256, out_fp32=True, seed=1001),
    "dense_b64_hq128_sk2048to4096": dict(kind="dense", batch=64, s_q=1, h_q=128, seqlen_lo=2048,
                                         seqlen_hi=4096, seed=1002),
    "dense_b1_hq64_sk65536": dict(kind="dense", batch=1, s_q=1, h_q=64, seqlen_lo=65536,
                                  seqlen_hi=65536, seed=1003),
    "dense_b16_sq2causal_hq128_sk4096to8192": dict(kind="dense", batch=16, s_q=2, h_q=128,
                                                   seqlen_lo=4096, seqlen_hi=8192, causal=True,
                                                   seed=1004),
    "sparse_fp8_b16_hq128_topk2048": dict(kind="sparse", batch=16, s_q=1, h_q=128, topk=2048,
                                          pages_per_req=512, topk_lo=1024, topk_hi=2048,
                                          seed=1005),
    # the dense page's fp16 instantiation and several latent KV heads
    "dense_b64_hq128_sk2048to4096_fp16": dict(kind="dense", batch=64, s_q=1, h_q=128, seqlen_lo=2048,
                                              seqlen_hi=4096, dtype=torch.float16, seed=1008),
    "dense_b32_hkv2_hq128_sk2048to4096": dict(kind="dense", batch=32, s_q=1, h_q=128, seqlen_lo=2048,
                                              seqlen_hi=4096, h_kv=2, seed=1009),
    # the dense decode over a paged cache of FP8 records
    "dense_fp8_b64_hq128_sk2048to4096": dict(kind="dense_fp8", batch=64, s_q=1, h_q=128, seqlen_lo=2048,
                                             seqlen_hi=4096, seed=1010),
    # the H=64 and S_q>1 query shapes of the packed-path page's grid, full top-k prefix
    "sparse_fp8_b4_sq4_hq64_topk2048": dict(kind="sparse", batch=4, s_q=4, h_q=64, topk=2048,
                                            pages_per_req=512, topk_lo=2048, topk_hi=2048,
                                            seed=1006),
    "sparse_fp8_b2_sq8_hq128_topk2048": dict(kind="sparse", batch=2, s_q=8, h_q=128, topk=2048,
                                             pages_per_req=512, topk_lo=2048, topk_hi=2048,
                                             seed=1007),
}


def make(name: str):
    spec = dict(WORKLOADS[name])
    kind = spec.pop("kind")
    if kind == "dense":
        return dense_case(name=name, **spec)
    if kind == "dense_fp8":
        return dense_fp8_case(name=name, **spec)
    return sparse_case(name=name, **spec)
