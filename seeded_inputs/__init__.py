"""Seeded synthetic inputs for the attention kernels and for the oracle.

This module is shared by the CUDA path's tests/benchmark and by the oracle's
tests.  It holds no attention arithmetic: it only draws random numbers, encodes
K/V into the int8 storage format the library consumes, and lays tensors out in
the contiguous or paged cache layouts.

Value recipe (the same for every workload):

* Q, K, V elements are N(0, 1) draws rounded to float16 (round-to-nearest-even),
  drawn from a ``torch.Generator`` seeded with the workload's seed.  Small cases
  are drawn on the CPU; full-size workloads may be drawn on the GPU (the oracle
  then reads the same bytes back, so both sides always see identical inputs).
* int8 K/V: each (token, kv-head) row of D f16 values x is encoded as
  ``s = f16(max|x| / 127)``, ``q = clamp(rint(x / float(s)), -127, 127)``
  (rint = round-half-even, division in fp32), ``q = 0`` where ``s == 0``.
  The attention inputs are then the dequantised values ``q * float(s)``; both
  the oracle and the kernels dequantise from (q, s) themselves.
* Paged caches: page ids come from a seeded random permutation of the page pool;
  sequence b takes the next ``ceil(L_b / P)`` ids in order; unused page-table
  slots hold -1.
* Variable lengths: ``kv_len[b]`` uniform on the integers of [lo, hi].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

__all__ = [
    "f16_normal",
    "quantize_int8_rows",
    "DecodeCase",
    "PrefillCase",
    "make_decode_case",
    "make_prefill_case",
    "paged_from_contiguous",
    "ring_from_contiguous",
    "TieredCase",
    "make_tiered_case",
    "ChunkCase",
    "make_chunked_case",
    "WORKLOADS",
]


def _gen(seed: int, device: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def f16_normal(shape, seed: int, device: str = "cpu", chunk: int = 1 << 26) -> torch.Tensor:
    """N(0,1) float16 tensor drawn from a seeded generator.

    Drawn in float32 and rounded to float16 (RNE); large tensors are drawn in
    chunks to bound the float32 temporary.
    """
    g = _gen(seed, device)
    out = torch.empty(shape, dtype=torch.float16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        flat[s:e] = torch.randn(e - s, generator=g, device=device, dtype=torch.float32).to(torch.float16)
    return out


def f32_normal(shape, seed: int, device: str = "cpu") -> torch.Tensor:
    """N(0,1) float32 tensor drawn from a seeded generator (queries of the f32-Q variant)."""
    return torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)


def quantize_int8_rows(x: torch.Tensor, chunk_rows: int = 1 << 20):
    """Encode f16 rows (last dim) as symmetric int8 with one f16 scale per row.

    Returns (codes int8 same shape, scales f16 shape[:-1]).  See the module
    docstring for the exact rule.
    """
    assert x.dtype == torch.float16
    D = x.shape[-1]
    rows = x.reshape(-1, D)
    codes = torch.empty(rows.shape, dtype=torch.int8, device=x.device)
    scales = torch.empty(rows.shape[0], dtype=torch.float16, device=x.device)
    for s in range(0, rows.shape[0], chunk_rows):
        e = min(rows.shape[0], s + chunk_rows)
        xf = rows[s:e].float()
        amax = xf.abs().amax(dim=1)
        sc = (amax / 127.0).to(torch.float16)
        scf = sc.float()
        safe = torch.where(scf > 0, scf, torch.ones_like(scf))
        qv = torch.round(xf / safe[:, None]).clamp_(-127, 127)
        qv = torch.where(scf[:, None] > 0, qv, torch.zeros_like(qv))
        codes[s:e] = qv.to(torch.int8)
        scales[s:e] = sc
    return codes.view(x.shape), scales.view(x.shape[:-1])


@dataclass
class DecodeCase:
    """Inputs of one decode call (all tensors on one device).

    Layouts (row-major):
      q            f16 [B, Hq, D]
      k, v         contiguous: [B, cap, Hkv, D]; paged: [n_pages, P, Hkv, D]
                   (f16, or int8 codes when ``int8``)
      k_scales/v_scales  f16; contiguous [B, Hkv, cap]; paged [n_pages, Hkv, P]
      kv_len       int32 [B]
      page_table   int32 [B, max_pages] or None
    """
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    kv_len: torch.Tensor
    batch: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    cap: int
    int8: bool = False
    k_scales: Optional[torch.Tensor] = None
    v_scales: Optional[torch.Tensor] = None
    page_table: Optional[torch.Tensor] = None
    page_size: int = 0
    max_pages: int = 0
    window: int = 0
    softcap: float = 0.0
    scale: float = 0.0
    lens: list = field(default_factory=list)
    ring: int = 0          # > 0: k/v [B, ring, Hkv, D] hold logical token t in slot t % ring

    @property
    def paged(self) -> bool:
        return self.page_table is not None

    @property
    def n_pages(self) -> int:
        return int(self.k.shape[0]) if self.paged else 0

    def to(self, device: str) -> "DecodeCase":
        kw = dict(self.__dict__)
        for name in ("q", "k", "v", "kv_len", "k_scales", "v_scales", "page_table"):
            t = kw[name]
            if t is not None:
                kw[name] = t.to(device)
        return DecodeCase(**kw)


@dataclass
class TieredCase(DecodeCase):
    """Inputs of one tiered decode call: the cold tier is the DecodeCase part
    (``kv_len`` = cold lengths, contiguous or paged, f16 or int8) and the hot
    tier an f16 ring:

      hot_k, hot_v   f16 [B, hot_ring, Hkv, D]; hot token i of sequence b in slot
                     (hot_start[b] + i) mod hot_ring
      hot_len        int32 [B]: hot tokens seen (the ring keeps the newest hot_ring)
      hot_start      int32 [B]: slot of hot token 0
    """
    hot_k: Optional[torch.Tensor] = None
    hot_v: Optional[torch.Tensor] = None
    hot_len: Optional[torch.Tensor] = None
    hot_start: Optional[torch.Tensor] = None
    hot_ring: int = 0
    hot_lens: list = field(default_factory=list)

    def to(self, device: str) -> "TieredCase":
        kw = dict(self.__dict__)
        for name in ("q", "k", "v", "kv_len", "k_scales", "v_scales", "page_table", "hot_k", "hot_v",
                     "hot_len", "hot_start"):
            t = kw[name]
            if t is not None:
                kw[name] = t.to(device)
        return TieredCase(**kw)


@dataclass
class PrefillCase:
    """Inputs of one prefill / vision call: q f16 [S, Hq, D]; k, v f16 [S, Hkv, D]."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    seq_len: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    causal: bool
    window: int = 0
    softcap: float = 0.0
    scale: float = 0.0

    def to(self, device: str) -> "PrefillCase":
        kw = dict(self.__dict__)
        for name in ("q", "k", "v"):
            kw[name] = kw[name].to(device)
        return PrefillCase(**kw)


@dataclass
class ChunkCase:
    """Inputs of one chunked-prefill / multi-token decode call over a paged cache.

    Layouts (row-major):
      q            f16 [total_q, Hq, D]: sequence b's new tokens are rows
                   q_start[b] .. q_start[b+1]-1
      k, v         f16 pool [n_pages, P, Hkv, D]; the new tokens' K/V are already
                   the last q_len[b] of sequence b's kv_len[b] cache tokens
      q_start      int32 [B+1]; kv_len int32 [B]; page_table int32 [B, max_pages]
    """
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    q_start: torch.Tensor
    kv_len: torch.Tensor
    page_table: torch.Tensor
    batch: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    max_pages: int
    max_q: int
    window: int = 0
    softcap: float = 0.0
    scale: float = 0.0
    q_lens: list = field(default_factory=list)
    kv_lens: list = field(default_factory=list)

    @property
    def total_q(self) -> int:
        return int(sum(self.q_lens))

    def to(self, device: str) -> "ChunkCase":
        kw = dict(self.__dict__)
        for name in ("q", "k", "v", "q_start", "kv_len", "page_table"):
            kw[name] = kw[name].to(device)
        return ChunkCase(**kw)


def _lengths(batch: int, lo: int, hi: int, seed: int) -> list:
    g = _gen(seed * 7919 + 17, "cpu")
    return torch.randint(lo, hi + 1, (batch,), generator=g).tolist()


def make_decode_case(batch: int, n_heads: int, n_kv_heads: int, head_dim: int,
                     lens, seed: int, *, cap: Optional[int] = None, int8: bool = False,
                     page_size: int = 0, n_pages: Optional[int] = None,
                     window: int = 0, softcap: float = 0.0, scale: Optional[float] = None,
                     ring: int = 0, q_f32: bool = False, device: str = "cpu") -> DecodeCase:
    """Build a decode case.

    ``lens`` is a list of per-sequence KV lengths, or a (lo, hi) tuple for
    seeded uniform lengths.  With ``page_size > 0`` the cache is paged: a pool of
    ``n_pages`` pages (default: just enough) filled with N(0,1) values, and a
    seeded permutation assigning pages to sequences.  With ``ring > 0`` the cache
    is a ring of ``ring`` slots per sequence, drawn directly (every slot holds
    N(0,1) values, as a ring does once its sequence has passed ``ring`` tokens);
    ``lens`` are then logical lengths and may exceed ``ring``.  ``q_f32`` draws the
    queries in float32 (not rounded to f16).
    """
    if isinstance(lens, tuple):
        lens = _lengths(batch, lens[0], lens[1], seed)
    lens = [int(x) for x in lens]
    assert len(lens) == batch
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    q = (f32_normal if q_f32 else f16_normal)((batch, n_heads, head_dim), seed * 1000 + 1, device)
    kv_len = torch.tensor(lens, dtype=torch.int32, device=device)
    if ring > 0:
        assert page_size <= 0
        cap = ring
    if page_size <= 0:
        if cap is None:
            cap = max(max(lens), 1)
            cap = (cap + 7) // 8 * 8
        k = f16_normal((batch, cap, n_kv_heads, head_dim), seed * 1000 + 2, device)
        v = f16_normal((batch, cap, n_kv_heads, head_dim), seed * 1000 + 3, device)
        ks = vs = None
        if int8:
            k, ks = quantize_int8_rows(k)
            v, vs = quantize_int8_rows(v)
            ks = ks.permute(0, 2, 1).contiguous()   # [B, Hkv, cap]
            vs = vs.permute(0, 2, 1).contiguous()
        return DecodeCase(q=q, k=k, v=v, kv_len=kv_len, batch=batch, n_heads=n_heads,
                          n_kv_heads=n_kv_heads, head_dim=head_dim, cap=cap, int8=int8,
                          k_scales=ks, v_scales=vs, window=window, softcap=softcap,
                          scale=float(scale), lens=lens, ring=ring)
    P = page_size
    need = [(L + P - 1) // P for L in lens]
    max_pages = max(max(need), 1)
    if n_pages is None:
        n_pages = max(sum(need), 1)
    assert sum(need) <= n_pages
    perm = torch.randperm(n_pages, generator=_gen(seed * 1000 + 4, "cpu"))
    pt = torch.full((batch, max_pages), -1, dtype=torch.int32)
    pos = 0
    for b in range(batch):
        pt[b, :need[b]] = perm[pos:pos + need[b]].to(torch.int32)
        pos += need[b]
    k = f16_normal((n_pages, P, n_kv_heads, head_dim), seed * 1000 + 2, device)
    v = f16_normal((n_pages, P, n_kv_heads, head_dim), seed * 1000 + 3, device)
    ks = vs = None
    if int8:
        k, ks = quantize_int8_rows(k)
        v, vs = quantize_int8_rows(v)
        ks = ks.permute(0, 2, 1).contiguous()        # [n_pages, Hkv, P]
        vs = vs.permute(0, 2, 1).contiguous()
    return DecodeCase(q=q, k=k, v=v, kv_len=kv_len, batch=batch, n_heads=n_heads,
                      n_kv_heads=n_kv_heads, head_dim=head_dim, cap=max_pages * P, int8=int8,
                      k_scales=ks, v_scales=vs, page_table=pt.to(device), page_size=P,
                      max_pages=max_pages, window=window, softcap=softcap,
                      scale=float(scale), lens=lens)


def ring_from_contiguous(case: DecodeCase, ring: int) -> DecodeCase:
    """The same logical tokens in a ring cache of ``ring`` slots per sequence:
    slot t % ring holds the newest token t that maps to it (older ones are
    overwritten, as a sliding-window cache does).  Slots no token has reached
    yet hold seeded filler values (finite, larger than the real ones), which no
    result may depend on.  The contiguous case must hold every logical token
    (cap >= max kv_len)."""
    assert not case.paged and not case.ring
    B = case.batch
    dev = case.k.device
    shape = (B, ring) + tuple(case.k.shape[2:])
    filler = f16_normal(shape, 7919 + ring, dev) * 4
    if case.int8:
        kr = filler.clamp(-127, 127).to(torch.int8)
        vr = kr.flip(-1).contiguous()
        ksr = (f16_normal((B, case.n_kv_heads, ring), 7927 + ring, dev).abs() + 0.5).to(torch.float16)
        vsr = ksr.flip(-1).contiguous()
    else:
        kr = filler.to(case.k.dtype)
        vr = kr.flip(-1).contiguous()
        ksr = vsr = None
    for b in range(B):
        L = int(case.lens[b])
        for t in range(max(0, L - ring), L):
            kr[b, t % ring] = case.k[b, t]
            vr[b, t % ring] = case.v[b, t]
            if case.int8:
                ksr[b, :, t % ring] = case.k_scales[b, :, t]
                vsr[b, :, t % ring] = case.v_scales[b, :, t]
    kw = dict(case.__dict__)
    kw.update(k=kr, v=vr, k_scales=ksr, v_scales=vsr, cap=ring, ring=ring)
    return DecodeCase(**kw)


def make_tiered_case(batch: int, n_heads: int, n_kv_heads: int, head_dim: int, cold_lens, hot_lens,
                     hot_ring: int, seed: int, *, hot_starts=None, int8: bool = False, page_size: int = 0,
                     n_pages: Optional[int] = None, cap: Optional[int] = None, window: int = 0,
                     softcap: float = 0.0, scale: Optional[float] = None, q_f32: bool = False,
                     device: str = "cpu") -> TieredCase:
    """Build a tiered decode case: the cold tier as make_decode_case builds a
    cache (``cold_lens`` tokens, contiguous or paged, f16 or int8) and an f16 hot
    ring of ``hot_ring`` slots holding N(0,1) values in every slot.  ``hot_lens``
    and ``cold_lens`` are lists or (lo, hi) tuples; ``hot_starts`` defaults to
    seeded slots in [0, hot_ring)."""
    cold = make_decode_case(batch, n_heads, n_kv_heads, head_dim, cold_lens, seed, cap=cap, int8=int8,
                            page_size=page_size, n_pages=n_pages, window=window, softcap=softcap,
                            scale=scale, q_f32=q_f32, device=device)
    if isinstance(hot_lens, tuple):
        hot_lens = _lengths(batch, hot_lens[0], hot_lens[1], seed * 7 + 3)
    hot_lens = [int(x) for x in hot_lens]
    assert len(hot_lens) == batch
    if hot_starts is None:
        g = _gen(seed * 7 + 4, "cpu")
        hot_starts = torch.randint(0, hot_ring, (batch,), generator=g).tolist()
    shape = (batch, hot_ring, n_kv_heads, head_dim)
    kw = dict(cold.__dict__)
    kw.update(hot_k=f16_normal(shape, seed * 1000 + 7, device), hot_v=f16_normal(shape, seed * 1000 + 8, device),
              hot_len=torch.tensor(hot_lens, dtype=torch.int32, device=device),
              hot_start=torch.tensor([int(x) for x in hot_starts], dtype=torch.int32, device=device),
              hot_ring=hot_ring, hot_lens=hot_lens)
    return TieredCase(**kw)


def paged_from_contiguous(case: DecodeCase, page_size: int, seed: int,
                          extra_pages: int = 3) -> DecodeCase:
    """Scatter a contiguous case into a paged pool holding the same values.

    Every logical token keeps its K/V (and scale) values, so attention over the
    paged case must equal attention over the contiguous one exactly.
    """
    assert not case.paged
    P = page_size
    B, Hkv, D = case.batch, case.n_kv_heads, case.head_dim
    max_pages = (case.cap + P - 1) // P
    n_pages = B * max_pages + extra_pages
    perm = torch.randperm(n_pages, generator=_gen(seed * 1000 + 5, "cpu"))
    pt = perm[:B * max_pages].view(B, max_pages).to(torch.int32)
    dev = case.k.device
    pool_shape = (n_pages, P, Hkv, D)
    kp = torch.zeros(pool_shape, dtype=case.k.dtype, device=dev)
    vp = torch.zeros(pool_shape, dtype=case.v.dtype, device=dev)
    ksp = vsp = None
    if case.int8:
        ksp = torch.zeros((n_pages, Hkv, P), dtype=torch.float16, device=dev)
        vsp = torch.zeros((n_pages, Hkv, P), dtype=torch.float16, device=dev)
    for b in range(B):
        for i in range(max_pages):
            t0, t1 = i * P, min((i + 1) * P, case.cap)
            pg = int(pt[b, i])
            kp[pg, :t1 - t0] = case.k[b, t0:t1]
            vp[pg, :t1 - t0] = case.v[b, t0:t1]
            if case.int8:
                ksp[pg, :, :t1 - t0] = case.k_scales[b, :, t0:t1]
                vsp[pg, :, :t1 - t0] = case.v_scales[b, :, t0:t1]
    kw = dict(case.__dict__)
    kw.update(k=kp, v=vp, k_scales=ksp, v_scales=vsp, page_table=pt.to(dev),
              page_size=P, max_pages=max_pages, cap=max_pages * P)
    return DecodeCase(**kw)


def make_chunked_case(batch: int, n_heads: int, n_kv_heads: int, head_dim: int, q_lens, ctx_lens,
                      seed: int, *, page_size: int, n_pages: Optional[int] = None, window: int = 0,
                      softcap: float = 0.0, scale: Optional[float] = None,
                      device: str = "cpu") -> ChunkCase:
    """Build a chunked-prefill case: sequence b has ctx_lens[b] cached tokens
    before a chunk of q_lens[b] new ones (kv_len = ctx + q_len).  Either list may
    be a (lo, hi) tuple for seeded uniform lengths.  Pages as in make_decode_case.
    """
    if isinstance(q_lens, tuple):
        q_lens = _lengths(batch, q_lens[0], q_lens[1], seed * 3 + 1)
    if isinstance(ctx_lens, tuple):
        ctx_lens = _lengths(batch, ctx_lens[0], ctx_lens[1], seed * 3 + 2)
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(c) + int(n) for c, n in zip(ctx_lens, q_lens)]
    assert len(q_lens) == batch and len(kv_lens) == batch
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    total_q = sum(q_lens)
    q = f16_normal((max(total_q, 1), n_heads, head_dim), seed * 1000 + 21, device)
    q_start = torch.tensor([0] + list(torch.tensor(q_lens).cumsum(0).tolist()), dtype=torch.int32,
                           device=device)
    P = page_size
    need = [(L + P - 1) // P for L in kv_lens]
    max_pages = max(max(need), 1)
    if n_pages is None:
        n_pages = max(sum(need), 1)
    assert sum(need) <= n_pages
    perm = torch.randperm(n_pages, generator=_gen(seed * 1000 + 24, "cpu"))
    pt = torch.full((batch, max_pages), -1, dtype=torch.int32)
    pos = 0
    for b in range(batch):
        pt[b, :need[b]] = perm[pos:pos + need[b]].to(torch.int32)
        pos += need[b]
    k = f16_normal((n_pages, P, n_kv_heads, head_dim), seed * 1000 + 22, device)
    v = f16_normal((n_pages, P, n_kv_heads, head_dim), seed * 1000 + 23, device)
    return ChunkCase(q=q, k=k, v=v, q_start=q_start,
                     kv_len=torch.tensor(kv_lens, dtype=torch.int32, device=device),
                     page_table=pt.to(device), batch=batch, n_heads=n_heads, n_kv_heads=n_kv_heads,
                     head_dim=head_dim, page_size=P, max_pages=max_pages, max_q=max(max(q_lens), 1),
                     window=window, softcap=softcap, scale=float(scale), q_lens=q_lens,
                     kv_lens=kv_lens)


def make_prefill_case(seq_len: int, n_heads: int, n_kv_heads: int, head_dim: int, seed: int, *,
                      causal: bool, window: int = 0, softcap: float = 0.0,
                      scale: Optional[float] = None, device: str = "cpu") -> PrefillCase:
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    q = f16_normal((seq_len, n_heads, head_dim), seed * 1000 + 11, device)
    k = f16_normal((seq_len, n_kv_heads, head_dim), seed * 1000 + 12, device)
    v = f16_normal((seq_len, n_kv_heads, head_dim), seed * 1000 + 13, device)
    return PrefillCase(q=q, k=k, v=v, seq_len=seq_len, n_heads=n_heads, n_kv_heads=n_kv_heads,
                       head_dim=head_dim, causal=causal, window=window, softcap=softcap,
                       scale=float(scale))


# The five seeded workloads, named by what they are.  Seeds are the workload
# numbers 1..5.
WORKLOADS = {
    "tiny_decode": dict(kind="decode", seed=1, batch=1, n_heads=4, n_kv_heads=2, head_dim=64,
                        lens=[128], int8=False, page_size=0, window=0, softcap=0.0,
                        scale=1.0 / 8.0),
    "vision_2304": dict(kind="prefill", seed=2, seq_len=2304, n_heads=16, n_kv_heads=16,
                        head_dim=64, causal=False, window=0, softcap=0.0, scale=1.0 / 8.0),
    "paged_gqa_decode": dict(kind="decode", seed=3, batch=32, n_heads=32, n_kv_heads=8,
                             head_dim=128, lens=(512, 8192), int8=False, page_size=16,
                             n_pages=32768, window=0, softcap=0.0,
                             scale=1.0 / math.sqrt(128.0)),
    "swa_softcap_prefill": dict(kind="prefill", seed=4, seq_len=4096, n_heads=8, n_kv_heads=4,
                                head_dim=256, causal=True, window=1024, softcap=50.0,
                                scale=1.0 / 16.0),
    "int8_long_decode": dict(kind="decode", seed=5, batch=16, n_heads=32, n_kv_heads=8,
                             head_dim=128, lens=[32768] * 16, int8=True, page_size=0,
                             window=0, softcap=0.0, scale=1.0 / math.sqrt(128.0)),
    # chunked prefill over a paged cache: 8 sequences append 512-token chunks to
    # 512..7680 cached tokens (16-token pages), the GQA shape of the paged decode
    # sliding-window decode over a 4096-slot ring cache: 32 sequences at logical
    # lengths 4K..64K (each keeps its newest 4096 tokens), the paged decode's GQA shape
    "ring_window_decode": dict(kind="decode", seed=7, batch=32, n_heads=32, n_kv_heads=8, head_dim=128,
                               lens=(4096, 65536), int8=False, page_size=0, ring=4096, window=0,
                               softcap=0.0, scale=1.0 / math.sqrt(128.0)),
    # tiered decode, the int8 tier of the pages: 32 sequences, an int8 cold tier of
    # 2K..16K tokens on 16-token pages plus an f16 hot ring of 1024 slots holding
    # the newest 256..1024 tokens
    # (f32 queries, as the pages' int8 tier requires)
    "tiered_int8_decode": dict(kind="tiered", seed=8, batch=32, n_heads=32, n_kv_heads=8, head_dim=128,
                               cold_lens=(2048, 16384), hot_lens=(256, 1024), hot_ring=1024, int8=True,
                               page_size=16, window=0, softcap=0.0, scale=1.0 / math.sqrt(128.0), q_f32=True),
    # the paged GQA decode with f32 queries and f32 outputs
    "paged_decode_f32io": dict(kind="decode", seed=9, batch=32, n_heads=32, n_kv_heads=8, head_dim=128,
                               lens=(512, 8192), int8=False, page_size=16, n_pages=None, window=0, softcap=0.0,
                               scale=1.0 / math.sqrt(128.0), q_f32=True, out_f32=True),
    "chunked_prefill_paged": dict(kind="chunked", seed=6, batch=8, n_heads=32, n_kv_heads=8,
                                  head_dim=128, q_lens=[512] * 8, ctx_lens=(512, 7680), page_size=16,
                                  window=0, softcap=0.0, scale=1.0 / math.sqrt(128.0)),
}

# Reduced cases of the same kernels for ncu captures (inputs still larger than
# the 129 MB L2, a few hundred MB on the device).
PROFILE_WORKLOADS = {
    "int8_decode_profile": dict(kind="decode", seed=5, batch=16, n_heads=32, n_kv_heads=8, head_dim=128,
                                lens=[4096] * 16, int8=True, page_size=0, window=0, softcap=0.0,
                                scale=1.0 / math.sqrt(128.0)),
    "paged_decode_profile": dict(kind="decode", seed=3, batch=32, n_heads=32, n_kv_heads=8,
                                 head_dim=128, lens=(512, 8192), int8=False, page_size=16,
                                 n_pages=None, window=0, softcap=0.0, scale=1.0 / math.sqrt(128.0)),
}
WORKLOADS.update(PROFILE_WORKLOADS)


def make_workload(name: str, device: str = "cpu"):
    w = dict(WORKLOADS[name])
    kind = w.pop("kind")
    seed = w.pop("seed")
    w.pop("out_f32", None)   # an output type: the caller allocates out
    if kind == "decode":
        b, hq, hkv, d, lens = (w.pop("batch"), w.pop("n_heads"), w.pop("n_kv_heads"),
                               w.pop("head_dim"), w.pop("lens"))
        return make_decode_case(b, hq, hkv, d, lens, seed, device=device, **w)
    if kind == "tiered":
        b, hq, hkv, d = w.pop("batch"), w.pop("n_heads"), w.pop("n_kv_heads"), w.pop("head_dim")
        return make_tiered_case(b, hq, hkv, d, w.pop("cold_lens"), w.pop("hot_lens"), w.pop("hot_ring"), seed,
                                device=device, **w)
    if kind == "chunked":
        b, hq, hkv, d = w.pop("batch"), w.pop("n_heads"), w.pop("n_kv_heads"), w.pop("head_dim")
        return make_chunked_case(b, hq, hkv, d, w.pop("q_lens"), w.pop("ctx_lens"), seed, device=device, **w)
    s, hq, hkv, d = w.pop("seq_len"), w.pop("n_heads"), w.pop("n_kv_heads"), w.pop("head_dim")
    return make_prefill_case(s, hq, hkv, d, seed, device=device, **w)
