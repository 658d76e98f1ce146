"""Seeded synthetic decode-step workloads.

This module only draws inputs: request lengths, the pages each request owns, the
request-to-token slot table, the query and the paged K/V cache (bf16, or int8 codes
with fp32 per-token-per-head scales), and an optional full-to-sliding-window slot
mapping.  It holds none of the path's arithmetic (no metadata formula, no attention),
so the CUDA path and the CPU oracle can both be fed from it.

All draws use a CPU ``torch.Generator`` seeded per workload, so the same seed gives
the same tensors on every host.

Cache layout (the layout the CUDA path reads): K and V are separate pools of shape
``[num_pages, num_kv_heads, page_size, head_dim]``; the int8 scales are
``[num_pages, num_kv_heads, page_size]`` float32.  Token slot ``page * page_size + off``
of the request-to-token table addresses row ``off`` of page ``page``.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import torch


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


@dataclasses.dataclass(frozen=True)
class Spec:
    """A decode-step workload shape.

    ``ctx`` is the number of cached tokens each request attends to (the value the
    metadata stage produces as ``cache_seqlens``); ``seq_lens = ctx - seqlen_offset``.
    ``ragged=(lo, hi)`` draws each request's ``ctx`` uniformly from ``lo..hi``.
    """

    name: str
    bs: int
    num_q_heads: int
    num_kv_heads: int
    num_pages: int
    ctx: int = 0
    ragged: Optional[tuple] = None
    head_dim: int = 128
    page_size: int = 64
    kv_dtype: str = "bf16"
    num_splits: int = 0            # 0: the library's split heuristic decides
    seqlen_offset: int = 0
    swa_window: Optional[int] = None
    seed: int = 0


# The five decode-step workloads the path is measured on.  Shapes and value
# distributions follow the workload list of the path's statement: Hq 32/Hkv 8
# (Hq 64 for the int8 case), head_dim 128, page_size 64, N(0,1) bf16 Q/K/V,
# int8 K/V with fp32 scales U[0.005, 0.05], shuffled page pools.
WORKLOADS = {
    "bs1_ctx1k": Spec("bs1_ctx1k", bs=1, num_q_heads=32, num_kv_heads=8, num_pages=64,
                      ctx=1024, num_splits=4, seqlen_offset=0, seed=1000),
    "bs8_ctx1k": Spec("bs8_ctx1k", bs=8, num_q_heads=32, num_kv_heads=8, num_pages=512,
                      ctx=1024, num_splits=4, seqlen_offset=1, seed=1001),
    "bs1_ctx8k": Spec("bs1_ctx8k", bs=1, num_q_heads=32, num_kv_heads=8, num_pages=256,
                      ctx=8192, num_splits=32, seqlen_offset=0, seed=1002),
    "bs32_ctx8k": Spec("bs32_ctx8k", bs=32, num_q_heads=32, num_kv_heads=8, num_pages=4096,
                       ctx=8192, num_splits=0, seqlen_offset=0, seed=1003),
    "bs64_ragged16k_int8_swa": Spec("bs64_ragged16k_int8_swa", bs=64, num_q_heads=64,
                                    num_kv_heads=8, num_pages=20000, ragged=(1, 16384),
                                    kv_dtype="int8", num_splits=0, seqlen_offset=0,
                                    swa_window=4096, seed=1004),
}
WORKLOAD_ORDER = list(WORKLOADS)


@dataclasses.dataclass
class Workload:
    spec: Spec
    ctx: list                      # attended tokens per request (python ints)
    pages: list                    # pages owned by each request, in token order
    req_pool_indices: torch.Tensor  # [bs] int64
    seq_lens: torch.Tensor         # [bs] int64
    req_to_token: torch.Tensor     # [bs, stride] int32
    max_seq_pages: int             # page-table width the caller asks for
    q: torch.Tensor                # [bs, Hq, d] bf16
    k_cache: torch.Tensor          # [num_pages, Hkv, page_size, d] bf16 or int8
    v_cache: torch.Tensor
    k_scale: Optional[torch.Tensor]  # [num_pages, Hkv, page_size] fp32 (int8 only)
    v_scale: Optional[torch.Tensor]
    full_to_swa_mapping: Optional[torch.Tensor]  # [num_pages*page_size + page_size + 1] int64
    swa_pages: Optional[list]      # per request: {page index in request: swa page}
    swa_window_start: Optional[list]  # per request: first in-window token position
    swa_num_pages: int = 0         # pages of the sliding-window pool
    # sliding-window pool (make(..., with_swa_cache=True)): same layouts as the full pool
    k_swa: Optional[torch.Tensor] = None
    v_swa: Optional[torch.Tensor] = None
    k_swa_scale: Optional[torch.Tensor] = None
    v_swa_scale: Optional[torch.Tensor] = None

    @property
    def sm_scale(self) -> float:
        """1/sqrt(head_dim) rounded to float32 (the value both sides are given)."""
        return float(torch.tensor(self.spec.head_dim ** -0.5, dtype=torch.float32))


def _draw_cache(spec: Spec, num_pages: int, g: torch.Generator):
    shape = (num_pages, spec.num_kv_heads, spec.page_size, spec.head_dim)
    if spec.kv_dtype == "bf16":
        k = torch.randn(shape, generator=g).to(torch.bfloat16)
        v = torch.randn(shape, generator=g).to(torch.bfloat16)
        return k, v, None, None
    if spec.kv_dtype == "int8":
        k = torch.randint(-127, 128, shape, generator=g, dtype=torch.int8)
        v = torch.randint(-127, 128, shape, generator=g, dtype=torch.int8)
        sshape = (num_pages, spec.num_kv_heads, spec.page_size)
        ks = torch.rand(sshape, generator=g) * 0.045 + 0.005
        vs = torch.rand(sshape, generator=g) * 0.045 + 0.005
        return k, v, ks, vs
    raise ValueError(spec.kv_dtype)


def make(spec: Spec, seed: Optional[int] = None, with_cache: bool = True,
         with_swa_cache: bool = False) -> Workload:
    """Draw one workload.  ``with_cache=False`` skips the (large) K/V pools;
    ``with_swa_cache`` also draws the sliding-window pool, from a generator of its own
    (seed + 0x5A5A), so neither it nor the other tensors depend on which pools are
    drawn."""
    g = torch.Generator().manual_seed(spec.seed if seed is None else seed)
    bs, P = spec.bs, spec.page_size
    if spec.ragged is not None:
        lo, hi = spec.ragged
        ctx = [int(x) for x in torch.randint(lo, hi + 1, (bs,), generator=g)]
        stride_tokens = _cdiv(hi, P) * P
    else:
        ctx = [spec.ctx] * bs
        stride_tokens = _cdiv(max(spec.ctx, 1), P) * P
    npages = [_cdiv(n, P) for n in ctx]
    if sum(npages) > spec.num_pages:
        raise ValueError(f"{spec.name}: {sum(npages)} pages needed, pool has {spec.num_pages}")
    perm = torch.randperm(spec.num_pages, generator=g).tolist()
    pages, cursor = [], 0
    for n_p in npages:
        pages.append(perm[cursor:cursor + n_p])
        cursor += n_p
    rpi = torch.randperm(bs, generator=g).to(torch.int64)
    seq_lens = torch.tensor([n - spec.seqlen_offset for n in ctx], dtype=torch.int64)

    req_to_token = torch.zeros((bs, stride_tokens), dtype=torch.int32)
    for i in range(bs):
        n = ctx[i]
        if n == 0:
            continue
        pg = torch.tensor(pages[i], dtype=torch.int32)
        t = torch.arange(n, dtype=torch.int32)
        req_to_token[int(rpi[i]), :n] = pg[t // P] * P + t % P
    max_seq_pages = max(max(npages), 1)

    q = torch.randn((bs, spec.num_q_heads, spec.head_dim), generator=g).to(torch.bfloat16)
    k_cache = v_cache = k_scale = v_scale = None
    if with_cache:
        k_cache, v_cache, k_scale, v_scale = _draw_cache(spec, spec.num_pages, g)

    mapping = swa_pages = window_start = None
    swa_num_pages = 0
    if spec.swa_window is not None:
        mapping, swa_pages, window_start, swa_num_pages = _swa_mapping(spec, ctx, pages, g)

    wl = Workload(spec, ctx, pages, rpi, seq_lens, req_to_token, max_seq_pages, q,
                  k_cache, v_cache, k_scale, v_scale, mapping, swa_pages, window_start,
                  swa_num_pages)
    if with_swa_cache:
        if spec.swa_window is None:
            raise ValueError(f"{spec.name}: no sliding window")
        g_swa = torch.Generator().manual_seed((spec.seed if seed is None else seed) + 0x5A5A)
        wl.k_swa, wl.v_swa, wl.k_swa_scale, wl.v_swa_scale = _draw_cache(spec, swa_num_pages,
                                                                         g_swa)
    return wl


def _swa_mapping(spec: Spec, ctx, pages, g):
    """Full-pool slot -> sliding-window-pool slot map, -1 where unmapped.

    For a request of length n, the window is token positions j >= n - window.  Every
    full-pool page that holds a window token gets its own page of a shuffled
    sliding-window pool, page for page: each slot of that page maps to the same offset
    in its sliding-window page (the pool allocates whole pages, so the first slot of a
    page the window starts inside is mapped too).  Every other entry, and the extra
    page_size + 1 tail, is -1.  Returns (mapping, per-request {page: swa page},
    per-request window start, sliding-window pool pages).
    """
    P, W = spec.page_size, spec.swa_window
    full_size = spec.num_pages * P
    mapping = torch.full((full_size + P + 1,), -1, dtype=torch.int64)
    swa_pool = sum(_cdiv(W, P) + 1 for _ in ctx)
    swa_perm = torch.randperm(swa_pool, generator=g).tolist()
    swa_pages, window_start, cursor = [], [], 0
    for n, pg in zip(ctx, pages):
        w0 = max(0, n - W)
        assigned = {}
        for p in range(w0 // P, _cdiv(n, P)):
            assigned[p] = swa_perm[cursor]
            cursor += 1
        offs = torch.arange(P, dtype=torch.int64)
        for p, sp in assigned.items():
            mapping[pg[p] * P + offs] = sp * P + offs
        swa_pages.append(assigned)
        window_start.append(w0)
    return mapping, swa_pages, window_start, swa_pool


def draw_query_lengths(bs: int, max_q_len: int, seed: int) -> torch.Tensor:
    """Query tokens per request for multi-token (speculative verify / extend) steps:
    uniform in 1..max_q_len, int64 [bs]."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(1, max_q_len + 1, (bs,), generator=g, dtype=torch.int64)


def draw_queries(total_q: int, num_q_heads: int, head_dim: int, seed: int) -> torch.Tensor:
    """Query rows ~ N(0, 1) in bf16, [total_q, num_q_heads, head_dim]."""
    g = torch.Generator().manual_seed(seed)
    return torch.randn((total_q, num_q_heads, head_dim), generator=g).to(torch.bfloat16)


def small_spec(seed: int, kv_dtype: str = "bf16", bs_max: int = 5, ctx_max: int = 300,
               group: Optional[int] = None, num_splits: Optional[int] = None,
               page_size: int = 64) -> Spec:
    """A small random shape: lengths that are not page multiples, empty splits."""
    g = torch.Generator().manual_seed(seed)
    bs = int(torch.randint(1, bs_max + 1, (1,), generator=g))
    hkv = int(torch.randint(1, 3, (1,), generator=g))
    grp = group if group is not None else [1, 2, 4, 8][int(torch.randint(0, 4, (1,), generator=g))]
    splits = num_splits if num_splits is not None else int(torch.randint(1, 8, (1,), generator=g))
    need = bs * _cdiv(ctx_max, page_size)
    return Spec(f"small{seed}", bs=bs, num_q_heads=hkv * grp, num_kv_heads=hkv,
                num_pages=need + 3, ragged=(1, ctx_max), page_size=page_size,
                kv_dtype=kv_dtype, num_splits=splits,
                seqlen_offset=int(torch.randint(0, 2, (1,), generator=g)), seed=seed)
