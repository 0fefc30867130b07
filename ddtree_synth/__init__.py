"""Seeded synthetic inputs for the DDTree tree-verify step.

This module only draws random numbers and lays them out in the shapes the
verify step consumes. It holds none of the method's arithmetic: no top-k, no
tree building, no attention, no accept rule. Both the fp64 oracle (``oracle/``)
and the CUDA path read their inputs from here, and nothing here imports either.

Workload shapes follow the five configurations the verify step is measured on
(a tiny parity case, a single-request latency case, a batched serving case, a
deep tree at high batch and a temperature case); the pages that describe the
method never name a public dataset, so every value is drawn from
``numpy.random.default_rng`` with a per-stream seed:

* stream 0: draft logits ``[B, D, V]`` (plus planted tokens) and root tokens
* stream 1: target logits ``[B, N, V]``, one fresh noise row per tree node
* stream 2: Q, tree K and tree V
* stream 3: the paged K/V cache and the page shuffle
* stream 4: context lengths

Separate streams keep every array independent of the order in which a caller
asks for them.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

__all__ = [
    "Workload", "CONFIGS", "config", "draft_inputs", "context_lengths",
    "paged_layout", "qkv_tree", "kv_cache", "target_logits",
    "f32_to_bf16_bits", "bf16_bits_to_f32", "sampling_params",
]


@dataclass(frozen=True)
class Workload:
    """Sizes and value distributions of one synthetic verify-step workload."""
    name: str
    B: int                 # requests
    D: int                 # draft depths
    V: int                 # vocabulary
    K: int                 # top-k cap (children per node)
    budget: int            # tree nodes excluding the root; N = budget + 1
    Hq: int
    Hkv: int
    Dh: int
    ctx_lo: int            # context length range [ctx_lo, ctx_hi] (equal -> fixed)
    ctx_hi: int
    page_size: int = 64
    paged_shuffle: bool = True     # False -> identity page table (contiguous context)
    draft_scale: float = 3.0       # draft logits = N(0,1) * draft_scale
    planted_boost: float = 0.0     # one planted token per depth gets +boost (0 -> none)
    target_sigma: float = 1.5      # target logits = draft row + N(0,1) * target_sigma
    temperature: float = 0.0       # 0 -> greedy accept
    seed: int = 0
    qkv_fp32_source: bool = False  # Q/K/V drawn as fp32 then rounded to bf16

    @property
    def N(self) -> int:
        return self.budget + 1

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def max_pages(self) -> int:
        return -(-self.ctx_hi // self.page_size)


CONFIGS = {
    "tiny": Workload(
        name="tiny", B=1, D=8, V=64, K=4, budget=16, Hq=4, Hkv=2, Dh=64,
        ctx_lo=256, ctx_hi=256, paged_shuffle=False, draft_scale=3.0,
        target_sigma=1.5, seed=0, qkv_fp32_source=True),
    "latency": Workload(
        name="latency", B=1, D=8, V=32000, K=8, budget=32, Hq=64, Hkv=8, Dh=128,
        ctx_lo=4096, ctx_hi=4096, paged_shuffle=False, draft_scale=4.0,
        planted_boost=6.0, target_sigma=2.0, seed=1000),
    "batched": Workload(
        name="batched", B=16, D=8, V=32000, K=8, budget=32, Hq=64, Hkv=8, Dh=128,
        ctx_lo=1024, ctx_hi=16384, paged_shuffle=True, draft_scale=3.0,
        target_sigma=1.5, seed=2000),
    "deep": Workload(
        name="deep", B=64, D=16, V=32000, K=8, budget=64, Hq=32, Hkv=8, Dh=128,
        ctx_lo=32768, ctx_hi=32768, paged_shuffle=True, draft_scale=4.0,
        planted_boost=5.0, target_sigma=2.5, seed=3000),
    "temperature": Workload(
        name="temperature", B=32, D=8, V=131072, K=8, budget=32, Hq=64, Hkv=8,
        Dh=128, ctx_lo=2048, ctx_hi=8192, paged_shuffle=True, draft_scale=3.0,
        target_sigma=1.5, temperature=0.7, seed=4000),
}


def config(name: str, **overrides) -> Workload:
    """Return a named workload, optionally with some fields replaced."""
    w = CONFIGS[name]
    return replace(w, **overrides) if overrides else w


def _rng(w: Workload, stream: int) -> np.random.Generator:
    return np.random.default_rng([w.seed, stream])


# ----------------------------------------------------------------------------
# bf16 storage format (round to nearest even); a data-format helper only
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return the raw uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------
# streams
# ----------------------------------------------------------------------------

def draft_inputs(w: Workload):
    """Draft logits fp32 ``[B, D, V]`` and root (anchor) tokens int32 ``[B]``.

    Logits are ``N(0,1) * draft_scale``; when ``planted_boost`` is set, one
    uniformly chosen token per (request, depth) gets ``+planted_boost``.
    Returns ``(draft_logits, root_tok, planted)`` where ``planted`` is
    ``[B, D]`` int32 (or None).
    """
    rng = _rng(w, 0)
    logits = rng.standard_normal((w.B, w.D, w.V), dtype=np.float32)
    logits *= np.float32(w.draft_scale)
    planted = None
    if w.planted_boost:
        planted = rng.integers(0, w.V, size=(w.B, w.D), dtype=np.int64).astype(np.int32)
        bi, di = np.meshgrid(np.arange(w.B), np.arange(w.D), indexing="ij")
        logits[bi, di, planted] += np.float32(w.planted_boost)
    root_tok = rng.integers(0, w.V, size=w.B, dtype=np.int64).astype(np.int32)
    return logits, root_tok, planted


def context_lengths(w: Workload) -> np.ndarray:
    """Per-request context length int32 ``[B]``: fixed or uniform in [lo, hi]."""
    if w.ctx_lo == w.ctx_hi:
        return np.full(w.B, w.ctx_lo, dtype=np.int32)
    rng = _rng(w, 4)
    return rng.integers(w.ctx_lo, w.ctx_hi + 1, size=w.B, dtype=np.int64).astype(np.int32)


def paged_layout(w: Workload, ctx_len: np.ndarray, spare_pages: int = 0, room: int = 0):
    """Page table int32 ``[B, max_pages]`` and the pool size.

    Request b owns ``ceil((ctx_len[b] + room) / page_size)`` pages (``room``
    token positions past the context, for a commit to write into). With
    ``paged_shuffle`` the pool's pages are handed out in a random order,
    otherwise in order (an identity layout for one contiguous context).
    Unused table entries hold -1. ``spare_pages`` extra pool pages are never
    referenced.
    """
    ps = w.page_size
    need = [-(-(int(L) + room) // ps) for L in ctx_len]
    total = sum(need) + spare_pages
    order = np.arange(total, dtype=np.int64)
    if w.paged_shuffle:
        order = _rng(w, 3).permutation(total)
    max_pages = max(w.max_pages(), max(need) if need else 0, 1)
    table = np.full((w.B, max_pages), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = order[k:k + n]
        k += n
    return table, total


def qkv_tree(w: Workload):
    """Tree-row Q ``[B,N,Hq,Dh]`` and tree K/V ``[B,N,Hkv,Dh]`` as bf16 bits.

    Values are N(0,1). When ``qkv_fp32_source`` is set the fp32 draws are also
    returned (the bf16 arrays are their rounding).
    """
    rng = _rng(w, 2)
    q = rng.standard_normal((w.B, w.N, w.Hq, w.Dh), dtype=np.float32)
    k = rng.standard_normal((w.B, w.N, w.Hkv, w.Dh), dtype=np.float32)
    v = rng.standard_normal((w.B, w.N, w.Hkv, w.Dh), dtype=np.float32)
    out = dict(q=f32_to_bf16_bits(q), k_tree=f32_to_bf16_bits(k), v_tree=f32_to_bf16_bits(v))
    if w.qkv_fp32_source:
        out.update(q_f32=q, k_tree_f32=k, v_tree_f32=v)
    return out


def kv_cache(w: Workload, num_pages: int):
    """Paged context K and V ``[num_pages, page_size, Hkv, Dh]`` as bf16 bits, N(0,1)."""
    rng = _rng(w, 3)
    rng.permutation(1)  # keep the stream distinct from the page shuffle's draw
    shape = (num_pages, w.page_size, w.Hkv, w.Dh)
    out = {}
    block = max(1, (1 << 24) // (w.page_size * w.Hkv * w.Dh))   # ~16M values per draw
    for name in ("k_cache", "v_cache"):
        bits = np.empty(shape, dtype=np.uint16)
        f32 = np.empty(shape, dtype=np.float32) if w.qkv_fp32_source else None
        for p0 in range(0, num_pages, block):
            p1 = min(num_pages, p0 + block)
            x = rng.standard_normal((p1 - p0,) + shape[1:], dtype=np.float32)
            bits[p0:p1] = f32_to_bf16_bits(x)
            if f32 is not None:
                f32[p0:p1] = x
        out[name] = bits
        if f32 is not None:
            out[name + "_f32"] = f32
    return out


def target_logits(w: Workload, draft_logits: np.ndarray, depth: np.ndarray,
                  n_nodes: np.ndarray) -> np.ndarray:
    """Target logits fp32 ``[B, N, V]`` for the nodes of a built tree.

    Row u is the target's prediction for the token that follows node u. For a
    node at depth d < D it is the draft row of depth d+1 plus
    ``N(0,1) * target_sigma`` noise drawn fresh for that node, so that siblings
    disagree; a node at depth D gets a fresh draft-like row plus noise. Rows of
    pad nodes (u >= n_nodes) are plain draft-like noise. ``depth`` is the tree's
    node depth array ``[B, N]`` and only selects rows; it is structure, not
    arithmetic of the method.
    """
    rng = _rng(w, 1)
    out = np.empty((w.B, w.N, w.V), dtype=np.float32)
    sig = np.float32(w.target_sigma)
    for b in range(w.B):
        for u in range(w.N):
            noise = rng.standard_normal(w.V, dtype=np.float32) * sig
            d = int(depth[b, u]) if u < int(n_nodes[b]) else -1
            if 0 <= d < w.D:
                out[b, u] = draft_logits[b, d] + noise
            else:
                fresh = rng.standard_normal(w.V, dtype=np.float32) * np.float32(w.draft_scale)
                out[b, u] = fresh + noise
    return out


def sampling_params(w: Workload):
    """Per-request temperature fp32 ``[B]`` and Philox seed uint64 ``[B]`` (seed = base + b)."""
    temp = np.full(w.B, w.temperature, dtype=np.float32)
    seed = (np.uint64(w.seed) * np.uint64(1000003) + np.arange(w.B, dtype=np.uint64)).astype(np.uint64)
    return temp, seed
