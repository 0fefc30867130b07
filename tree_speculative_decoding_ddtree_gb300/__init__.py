"""DDTree tree-verify step on one GB300: thin Python binding of ``libddtree.so``.

The calls of the C ABI (``include/ddtree.h``) are exposed under the same
names. This module only marshals arguments: it checks that tensors are CUDA,
contiguous and of the right dtype and shape, passes their device pointers and
the current stream, and raises :class:`DDTreeError` on a non-zero status. All
computation runs in the library's CUDA kernels; there is no fallback. PyTorch
serves for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

__all__ = [
    "DDTreeError", "load_library", "library_path", "ddtree_draft_topk", "ddtree_build", "tree_verify_attn",
    "tree_verify_attn_workspace_size", "ddtree_accept_greedy", "ddtree_accept_sample",
    "ddtree_accept_greedy_sample",
    "TreeBuffers", "alloc_tree", "DEV_ERRORS", "tree_verify_attn_noalloc", "ddtree_commit_kv",
    "StepArgs", "VerifyStep", "ddtree_accept_sample_ratio",
]

DEV_ERRORS = {
    1: "DDT_DEV_BAD_PAGE", 2: "DDT_DEV_BAD_CTX", 4: "DDT_DEV_BAD_TREE",
    8: "DDT_DEV_BAD_TEMPERATURE", 16: "DDT_DEV_BAD_TOKEN",
}

_lib = None


class DDTreeError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: status {status} ({detail})")


def library_path() -> str:
    return _build.LIB_PATH


def load_library(path: Optional[str] = None):
    """Load ``libddtree.so`` (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"DDTree CUDA library not found at {p}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (no CPU fallback exists)")
    lib = ctypes.CDLL(p)
    P, I, F, Z, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint64
    lib.ddtree_status_string.restype = ctypes.c_char_p
    lib.ddtree_status_string.argtypes = [I]
    lib.ddtree_last_error.restype = ctypes.c_char_p
    lib.ddtree_last_error.argtypes = []
    lib.ddtree_draft_topk.restype = I
    lib.ddtree_draft_topk.argtypes = [P, I, I, I, I, P, P, P]
    lib.ddtree_commit_kv.restype = I
    lib.ddtree_commit_kv.argtypes = [P, P, P, P, I, I, I, I, I, P, P, I, I, P, I, P, P, P, P]
    lib.ddtree_step_args_size.restype = Z
    lib.ddtree_step_args_size.argtypes = []
    lib.ddtree_step_create.restype = I
    lib.ddtree_step_create.argtypes = [ctypes.POINTER(StepArgs), ctypes.POINTER(P)]
    lib.ddtree_step_launch.restype = I
    lib.ddtree_step_launch.argtypes = [P, P]
    lib.ddtree_step_destroy.restype = None
    lib.ddtree_step_destroy.argtypes = [P]
    lib.ddtree_accept_sample_ratio.restype = I
    lib.ddtree_accept_sample_ratio.argtypes = [P, P, I, P, P, P, P, I, I, I, P, P, U64, P, P, P, P, P, P, P, P]
    lib.ddtree_build.restype = I
    lib.ddtree_build.argtypes = [P] * 4 + [I] * 4 + [P] * 10 + [P, P]
    lib.tree_verify_attn.restype = I
    lib.tree_verify_attn.argtypes = [P, P, P, P, P, I, I, P, I, P, P, P, I, I, I, I, I, F,
                                     P, P, P, Z, P, P]
    lib.tree_verify_attn_workspace_size.restype = Z
    lib.tree_verify_attn_workspace_size.argtypes = [I, I, I, I, I, I]
    lib.ddtree_accept_greedy.restype = I
    lib.ddtree_accept_greedy.argtypes = [P, I, P, P, P, P, I, I, I, P, P, P, P, P, P, P]
    lib.ddtree_accept_sample.restype = I
    lib.ddtree_accept_sample.argtypes = [P, I, P, P, P, P, I, I, I, P, P, U64, P, P, P, P, P, P, P, P]
    lib.ddtree_accept_greedy_sample.argtypes = [P, I, P, P, P, P, I, I, I, P, P, U64, P, P, P, P, P,
                                                P, P, P, P, P, P, P, P]
    if path is None:
        _lib = lib
    return lib


class StepArgs(ctypes.Structure):
    """Mirror of ``ddtree_step_args`` (include/ddtree.h), field for field."""
    _fields_ = (
        [(n, ctypes.c_int) for n in ("B", "D", "K", "budget", "V", "Hq", "Hkv", "Dh", "num_pages",
                                     "page_size", "max_pages")]
        + [("scale", ctypes.c_float), ("walk", ctypes.c_int), ("philox_offset", ctypes.c_uint64)]
        + [(n, ctypes.c_void_p) for n in ("topk_logp", "topk_tok", "root_tok", "ctx_len", "q", "k_tree",
                                          "v_tree", "k_cache", "v_cache", "page_table", "logits",
                                          "temperature", "seed", "draft_logits", "parent", "depth", "token", "rank",
                                          "pos", "score", "first_child", "next_sibling", "vis",
                                          "n_nodes", "attn_out", "lse", "workspace")]
        + [("workspace_bytes", ctypes.c_size_t)]
        + [(n, ctypes.c_void_p) for n in ("accept_len", "out_tokens", "out_nodes", "bonus",
                                          "new_ctx_len", "dev_status")])


def _check(status: int, where: str):
    if status != 0:
        lib = load_library()
        detail = lib.ddtree_status_string(status).decode()
        if status == -3:
            detail += ": " + lib.ddtree_last_error().decode()
        raise DDTreeError(status, where, detail)


def _ptr(t: Optional[torch.Tensor], dtype, name: str, shape=None) -> int:
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def ddtree_draft_topk(draft_logits: torch.Tensor, K: int, topk_logp: Optional[torch.Tensor] = None,
                      topk_tok: Optional[torch.Tensor] = None, stream=None):
    """Per-depth top-K tokens and log-probs of fp32 draft logits ``[B, D, V]``
    (see ``ddtree_draft_topk`` in include/ddtree.h). Returns ``(topk_logp, topk_tok)``."""
    lib = load_library()
    B, D, V = draft_logits.shape
    dev = draft_logits.device
    if topk_logp is None:
        topk_logp = torch.empty((B, D, K), dtype=torch.float32, device=dev)
    if topk_tok is None:
        topk_tok = torch.empty((B, D, K), dtype=torch.int32, device=dev)
    st = lib.ddtree_draft_topk(
        _ptr(draft_logits, torch.float32, "draft_logits", (B, D, V)), B, D, V, K,
        _ptr(topk_logp, torch.float32, "topk_logp", (B, D, K)),
        _ptr(topk_tok, torch.int32, "topk_tok", (B, D, K)), _stream(stream))
    _check(st, "ddtree_draft_topk")
    return topk_logp, topk_tok


class TreeBuffers:
    """Device outputs of ``ddtree_build`` for B requests and N = budget + 1 rows."""

    def __init__(self, B: int, N: int, device):
        W = (N + 31) // 32
        i32 = dict(dtype=torch.int32, device=device)
        self.B, self.N, self.W = B, N, W
        self.parent = torch.empty((B, N), **i32)
        self.depth = torch.empty((B, N), **i32)
        self.token = torch.empty((B, N), **i32)
        self.rank = torch.empty((B, N), **i32)
        self.pos = torch.empty((B, N), **i32)
        self.score = torch.empty((B, N), dtype=torch.float64, device=device)
        self.first_child = torch.empty((B, N), **i32)
        self.next_sibling = torch.empty((B, N), **i32)
        self.vis = torch.empty((B, N, W), dtype=torch.int32, device=device)  # uint32 bits
        self.n_nodes = torch.empty((B,), **i32)


def alloc_tree(B: int, N: int, device="cuda") -> TreeBuffers:
    return TreeBuffers(B, N, device)


def ddtree_build(topk_logp: torch.Tensor, topk_tok: torch.Tensor, root_tok: torch.Tensor,
                 ctx_len: torch.Tensor, budget: int, out: Optional[TreeBuffers] = None,
                 dev_status: Optional[torch.Tensor] = None, stream=None) -> TreeBuffers:
    """Best-first tree from per-depth top-k (see ``ddtree_build`` in include/ddtree.h)."""
    lib = load_library()
    B, D, K = topk_logp.shape
    N = budget + 1
    if out is None:
        out = TreeBuffers(B, N, topk_logp.device)
    st = lib.ddtree_build(
        _ptr(topk_logp, torch.float32, "topk_logp", (B, D, K)),
        _ptr(topk_tok, torch.int32, "topk_tok", (B, D, K)),
        _ptr(root_tok, torch.int32, "root_tok", (B,)),
        _ptr(ctx_len, torch.int32, "ctx_len", (B,)),
        B, D, K, budget,
        _ptr(out.parent, torch.int32, "parent", (B, N)), _ptr(out.depth, torch.int32, "depth", (B, N)),
        _ptr(out.token, torch.int32, "token", (B, N)), _ptr(out.rank, torch.int32, "rank", (B, N)),
        _ptr(out.pos, torch.int32, "pos", (B, N)), _ptr(out.score, torch.float64, "score", (B, N)),
        _ptr(out.first_child, torch.int32, "first_child", (B, N)),
        _ptr(out.next_sibling, torch.int32, "next_sibling", (B, N)),
        _ptr(out.vis, torch.int32, "vis", (B, N, (N + 31) // 32)),
        _ptr(out.n_nodes, torch.int32, "n_nodes", (B,)),
        _ptr(dev_status, torch.int32, "dev_status", (1,)), _stream(stream))
    _check(st, "ddtree_build")
    return out


def tree_verify_attn_workspace_size(B: int, N: int, Hq: int, Hkv: int, Dh: int, max_ctx: int) -> int:
    return int(load_library().tree_verify_attn_workspace_size(B, N, Hq, Hkv, Dh, max_ctx))


def tree_verify_attn(q: torch.Tensor, k_tree: torch.Tensor, v_tree: torch.Tensor,
                     k_cache: torch.Tensor, v_cache: torch.Tensor, page_table: torch.Tensor,
                     ctx_len: torch.Tensor, vis: torch.Tensor, n_nodes: torch.Tensor,
                     scale: float, out: Optional[torch.Tensor] = None,
                     lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                     dev_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Tree-verify attention (see ``tree_verify_attn`` in include/ddtree.h).

    ``q`` is bf16 ``[B, N, Hq, Dh]``; ``k_cache``/``v_cache`` are bf16
    ``[num_pages, page_size, Hkv, Dh]``. A workspace of the required size is
    allocated here when none is given.
    """
    lib = load_library()
    B, N, Hq, Dh = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    max_pages = page_table.shape[1]
    W = (N + 31) // 32
    if out is None:
        out = torch.empty_like(q)
    need = tree_verify_attn_workspace_size(B, N, Hq, Hkv, Dh, max_pages * page_size)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = lib.tree_verify_attn(
        _ptr(q, torch.bfloat16, "q", (B, N, Hq, Dh)),
        _ptr(k_tree, torch.bfloat16, "k_tree", (B, N, Hkv, Dh)),
        _ptr(v_tree, torch.bfloat16, "v_tree", (B, N, Hkv, Dh)),
        _ptr(k_cache, torch.bfloat16, "k_cache", (num_pages, page_size, Hkv, Dh)),
        _ptr(v_cache, torch.bfloat16, "v_cache", (num_pages, page_size, Hkv, Dh)),
        num_pages, page_size,
        _ptr(page_table, torch.int32, "page_table", (B, max_pages)), max_pages,
        _ptr(ctx_len, torch.int32, "ctx_len", (B,)),
        _ptr(vis, torch.int32, "vis", (B, N, W)),
        _ptr(n_nodes, torch.int32, "n_nodes", (B,)),
        B, N, Hq, Hkv, Dh, float(scale),
        _ptr(out, torch.bfloat16, "out", (B, N, Hq, Dh)),
        _ptr(lse, torch.float32, "lse", (B, N, Hq)),
        _ptr(workspace, torch.uint8, "workspace") if workspace is not None else 0,
        workspace.numel() if workspace is not None else 0,
        _ptr(dev_status, torch.int32, "dev_status", (1,)), _stream(stream))
    _check(st, "tree_verify_attn")
    return out


def _walk_outputs(B, D, device, out):
    if out is not None:
        return out
    i32 = dict(dtype=torch.int32, device=device)
    return dict(accept_len=torch.empty(B, **i32), out_tokens=torch.empty((B, D + 1), **i32),
                out_nodes=torch.empty((B, D + 1), **i32), bonus=torch.empty(B, **i32))


def ddtree_accept_greedy(logits: torch.Tensor, tree: TreeBuffers, D: int, out=None,
                         dev_status: Optional[torch.Tensor] = None, stream=None,
                         walk_stats: Optional[torch.Tensor] = None):
    """Greedy verify walk (see ``ddtree_accept_greedy`` in include/ddtree.h).

    ``walk_stats`` (optional int32 ``[B, 4]``) receives accepted depth, nodes
    built, tokens emitted and children compared without a match."""
    lib = load_library()
    B, N, V = logits.shape
    o = _walk_outputs(B, D, logits.device, out)
    st = lib.ddtree_accept_greedy(
        _ptr(logits, torch.float32, "logits", (B, N, V)), V,
        _ptr(tree.token, torch.int32, "token", (B, N)),
        _ptr(tree.first_child, torch.int32, "first_child", (B, N)),
        _ptr(tree.next_sibling, torch.int32, "next_sibling", (B, N)),
        _ptr(tree.n_nodes, torch.int32, "n_nodes", (B,)), B, N, D,
        _ptr(o["accept_len"], torch.int32, "accept_len", (B,)),
        _ptr(o["out_tokens"], torch.int32, "out_tokens", (B, D + 1)),
        _ptr(o["out_nodes"], torch.int32, "out_nodes", (B, D + 1)),
        _ptr(o["bonus"], torch.int32, "bonus", (B,)),
        _ptr(walk_stats, torch.int32, "walk_stats", (B, 4)),
        _ptr(dev_status, torch.int32, "dev_status", (1,)), _stream(stream))
    _check(st, "ddtree_accept_greedy")
    return o


def ddtree_accept_sample_ratio(logits: torch.Tensor, draft_logits: torch.Tensor, tree: TreeBuffers,
                               D: int, temperature: torch.Tensor, seed: torch.Tensor, philox_offset: int,
                               out=None, dev_status: Optional[torch.Tensor] = None, stream=None,
                               margin_stats: Optional[torch.Tensor] = None,
                               walk_stats: Optional[torch.Tensor] = None):
    """Temperature walk with the draft-ratio rule (see ``ddtree_accept_sample_ratio`` in
    include/ddtree.h). ``draft_logits`` fp32 ``[B, D, V]``; ``seed`` int64 ``[B]``
    holding the uint64 seeds; optional ``margin_stats`` fp32 ``[B]`` and
    ``walk_stats`` int32 ``[B, 4]``."""
    lib = load_library()
    B, N, V = logits.shape
    o = _walk_outputs(B, D, logits.device, out)
    st = lib.ddtree_accept_sample_ratio(
        _ptr(logits, torch.float32, "logits", (B, N, V)),
        _ptr(draft_logits, torch.float32, "draft_logits", (B, D, V)), V,
        _ptr(tree.token, torch.int32, "token", (B, N)),
        _ptr(tree.first_child, torch.int32, "first_child", (B, N)),
        _ptr(tree.next_sibling, torch.int32, "next_sibling", (B, N)),
        _ptr(tree.n_nodes, torch.int32, "n_nodes", (B,)), B, N, D,
        _ptr(temperature, torch.float32, "temperature", (B,)),
        _ptr(seed, torch.int64, "seed", (B,)), philox_offset,
        _ptr(o["accept_len"], torch.int32, "accept_len", (B,)),
        _ptr(o["out_tokens"], torch.int32, "out_tokens", (B, D + 1)),
        _ptr(o["out_nodes"], torch.int32, "out_nodes", (B, D + 1)),
        _ptr(o["bonus"], torch.int32, "bonus", (B,)),
        _ptr(margin_stats, torch.float32, "margin_stats", (B,)),
        _ptr(walk_stats, torch.int32, "walk_stats", (B, 4)),
        _ptr(dev_status, torch.int32, "dev_status", (1,)), _stream(stream))
    _check(st, "ddtree_accept_sample_ratio")
    return o


def ddtree_commit_kv(k_tree: torch.Tensor, v_tree: torch.Tensor, accept: dict,
                     ctx_len: torch.Tensor, page_table: torch.Tensor, k_cache: torch.Tensor,
                     v_cache: torch.Tensor, new_ctx_len: Optional[torch.Tensor] = None,
                     dev_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Append the committed path's K/V to the paged cache (see ``ddtree_commit_kv`` in
    include/ddtree.h). ``accept`` is a walk's output dict; ``new_ctx_len`` may be
    ``ctx_len`` itself (in-place advance). Returns ``new_ctx_len``."""
    lib = load_library()
    B, N, Hkv, Dh = k_tree.shape
    D = accept["out_nodes"].shape[1] - 1
    num_pages, page_size = k_cache.shape[0], k_cache.shape[1]
    max_pages = page_table.shape[1]
    if new_ctx_len is None:
        new_ctx_len = torch.empty_like(ctx_len)
    st = lib.ddtree_commit_kv(
        _ptr(k_tree, torch.bfloat16, "k_tree", (B, N, Hkv, Dh)),
        _ptr(v_tree, torch.bfloat16, "v_tree", (B, N, Hkv, Dh)),
        _ptr(accept["out_nodes"], torch.int32, "out_nodes", (B, D + 1)),
        _ptr(accept["accept_len"], torch.int32, "accept_len", (B,)), B, N, D, Hkv, Dh,
        _ptr(k_cache, torch.bfloat16, "k_cache", (num_pages, page_size, Hkv, Dh)),
        _ptr(v_cache, torch.bfloat16, "v_cache", (num_pages, page_size, Hkv, Dh)),
        num_pages, page_size, _ptr(page_table, torch.int32, "page_table", (B, max_pages)), max_pages,
        _ptr(ctx_len, torch.int32, "ctx_len", (B,)), _ptr(new_ctx_len, torch.int32, "new_ctx_len", (B,)),
        _ptr(dev_status, torch.int32, "dev_status", (1,)), _stream(stream))
    _check(st, "ddtree_commit_kv")
    return new_ctx_len


def ddtree_accept_sample(logits: torch.Tensor, tree: TreeBuffers, D: int,
                         temperature: torch.Tensor, seed: torch.Tensor, philox_offset: int,
                         out=None, dev_status: Optional[torch.Tensor] = None, stream=None,
                         margin_stats: Optional[torch.Tensor] = None,
                         walk_stats: Optional[torch.Tensor] = None):
    """Temperature verify walk (see ``ddtree_accept_sample`` in include/ddtree.h).

    ``seed`` is int64 on the device, read as uint64 bits. Optional
    ``margin_stats`` fp32 ``[B]`` receives each request's smallest decision
    margin and ``walk_stats`` int32 ``[B, 4]`` its walk statistics.
    """
    lib = load_library()
    B, N, V = logits.shape
    o = _walk_outputs(B, D, logits.device, out)
    st = lib.ddtree_accept_sample(
        _ptr(logits, torch.float32, "logits", (B, N, V)), V,
        _ptr(tree.token, torch.int32, "token", (B, N)),
        _ptr(tree.first_child, torch.int32, "first_child", (B, N)),
        _ptr(tree.next_sibling, torch.int32, "next_sibling", (B, N)),
        _ptr(tree.n_nodes, torch.int32, "n_nodes", (B,)), B, N, D,
        _ptr(temperature, torch.float32, "temperature", (B,)),
        _ptr(seed, torch.int64, "seed", (B,)), int(philox_offset),
        _ptr(o["accept_len"], torch.int32, "accept_len", (B,)),
        _ptr(o["out_tokens"], torch.int32, "out_tokens", (B, D + 1)),
        _ptr(o["out_nodes"], torch.int32, "out_nodes", (B, D + 1)),
        _ptr(o["bonus"], torch.int32, "bonus", (B,)),
        _ptr(margin_stats, torch.float32, "margin_stats", (B,)),
        _ptr(walk_stats, torch.int32, "walk_stats", (B, 4)),
        _ptr(dev_status, torch.int32, "dev_status", (1,)), _stream(stream))
    _check(st, "ddtree_accept_sample")
    return o


def ddtree_accept_greedy_sample(logits: torch.Tensor, tree: TreeBuffers, D: int,
                                temperature: torch.Tensor, seed: torch.Tensor, philox_offset: int,
                                out_greedy=None, out_sample=None,
                                dev_status: Optional[torch.Tensor] = None, stream=None,
                                greedy_walk_stats: Optional[torch.Tensor] = None,
                                sample_margin_stats: Optional[torch.Tensor] = None,
                                sample_walk_stats: Optional[torch.Tensor] = None):
    """The greedy and the temperature walk in one launch (see
    ``ddtree_accept_greedy_sample`` in include/ddtree.h); returns the two output
    dicts, each identical to what the separate call writes."""
    lib = load_library()
    B, N, V = logits.shape
    og = _walk_outputs(B, D, logits.device, out_greedy)
    os_ = _walk_outputs(B, D, logits.device, out_sample)
    st = lib.ddtree_accept_greedy_sample(
        _ptr(logits, torch.float32, "logits", (B, N, V)), V,
        _ptr(tree.token, torch.int32, "token", (B, N)),
        _ptr(tree.first_child, torch.int32, "first_child", (B, N)),
        _ptr(tree.next_sibling, torch.int32, "next_sibling", (B, N)),
        _ptr(tree.n_nodes, torch.int32, "n_nodes", (B,)), B, N, D,
        _ptr(temperature, torch.float32, "temperature", (B,)),
        _ptr(seed, torch.int64, "seed", (B,)), int(philox_offset),
        _ptr(og["accept_len"], torch.int32, "greedy accept_len", (B,)),
        _ptr(og["out_tokens"], torch.int32, "greedy out_tokens", (B, D + 1)),
        _ptr(og["out_nodes"], torch.int32, "greedy out_nodes", (B, D + 1)),
        _ptr(og["bonus"], torch.int32, "greedy bonus", (B,)),
        _ptr(greedy_walk_stats, torch.int32, "greedy_walk_stats", (B, 4)),
        _ptr(os_["accept_len"], torch.int32, "sample accept_len", (B,)),
        _ptr(os_["out_tokens"], torch.int32, "sample out_tokens", (B, D + 1)),
        _ptr(os_["out_nodes"], torch.int32, "sample out_nodes", (B, D + 1)),
        _ptr(os_["bonus"], torch.int32, "sample bonus", (B,)),
        _ptr(sample_margin_stats, torch.float32, "sample_margin_stats", (B,)),
        _ptr(sample_walk_stats, torch.int32, "sample_walk_stats", (B, 4)),
        _ptr(dev_status, torch.int32, "dev_status", (1,)), _stream(stream))
    _check(st, "ddtree_accept_greedy_sample")
    return og, os_


def tree_verify_attn_noalloc(q: torch.Tensor, k_tree: torch.Tensor, v_tree: torch.Tensor,
                             k_cache: torch.Tensor, v_cache: torch.Tensor,
                             page_table: torch.Tensor, ctx_len: torch.Tensor, vis: torch.Tensor,
                             n_nodes: torch.Tensor, scale: float, out: torch.Tensor,
                             lse: Optional[torch.Tensor] = None,
                             dev_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Tree-verify attention through ``tree_verify_attn_noalloc``: for callers that
    cannot allocate device memory at run time. The split-KV scratch is the library's
    own fixed 64 MiB device array (shared by all calls; calls that overlap on the GPU
    race on it), and ``out`` must be given, so this call allocates nothing."""
    lib = load_library()
    fn = lib.tree_verify_attn_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.restype = I
    fn.argtypes = [P, P, P, P, P, I, I, P, I, P, P, P, I, I, I, I, I, F, P, P, P, P]
    B, N, Hq, Dh = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    max_pages = page_table.shape[1]
    W = (N + 31) // 32
    st = fn(_ptr(q, torch.bfloat16, "q", (B, N, Hq, Dh)),
            _ptr(k_tree, torch.bfloat16, "k_tree", (B, N, Hkv, Dh)),
            _ptr(v_tree, torch.bfloat16, "v_tree", (B, N, Hkv, Dh)),
            _ptr(k_cache, torch.bfloat16, "k_cache", (num_pages, page_size, Hkv, Dh)),
            _ptr(v_cache, torch.bfloat16, "v_cache", (num_pages, page_size, Hkv, Dh)),
            num_pages, page_size,
            _ptr(page_table, torch.int32, "page_table", (B, max_pages)), max_pages,
            _ptr(ctx_len, torch.int32, "ctx_len", (B,)),
            _ptr(vis, torch.int32, "vis", (B, N, W)),
            _ptr(n_nodes, torch.int32, "n_nodes", (B,)),
            B, N, Hq, Hkv, Dh, float(scale),
            _ptr(out, torch.bfloat16, "out", (B, N, Hq, Dh)),
            _ptr(lse, torch.float32, "lse", (B, N, Hq)),
            _ptr(dev_status, torch.int32, "dev_status", (1,)), _stream(stream))
    _check(st, "tree_verify_attn_noalloc")
    return out


class VerifyStep:
    """The verify step (build -> attention -> walk -> commit) recorded by the
    library as one CUDA graph (``ddtree_step_*`` in include/ddtree.h).

    Every array is fixed at construction; ``launch()`` replays the graph on a
    stream and reads the arrays' current contents. Outputs not given are
    allocated here: ``tree`` (TreeBuffers), ``attn_out``, ``accept`` (walk
    dict). With ``new_ctx_len=None`` each launch advances ``ctx_len`` in place.
    The object keeps references to all tensors for the graph's lifetime.
    """

    def __init__(self, *, topk_logp, topk_tok, root_tok, ctx_len, q, k_tree, v_tree, k_cache, v_cache,
                 page_table, logits, budget: int, scale: float, walk: str = "greedy",
                 temperature=None, seed=None, philox_offset: int = 0, new_ctx_len=None,
                 dev_status=None, lse=None, draft_logits=None):
        lib = load_library()
        B, D, K = topk_logp.shape
        N = budget + 1
        _, _, Hq, Dh = q.shape
        num_pages, page_size, Hkv, _ = k_cache.shape
        max_pages = page_table.shape[1]
        V = logits.shape[2]
        dev = q.device
        walks = {"greedy": 0, "sampled": 1, "ratio": 2}
        if walk not in walks:
            raise ValueError("walk must be 'greedy', 'sampled' or 'ratio'")
        self.tree = TreeBuffers(B, N, dev)
        self.attn_out = torch.empty((B, N, Hq, Dh), dtype=torch.bfloat16, device=dev)
        self.accept = _walk_outputs(B, D, dev, None)
        need = tree_verify_attn_workspace_size(B, N, Hq, Hkv, Dh, max_pages * page_size)
        self.workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        self._keep = [topk_logp, topk_tok, root_tok, ctx_len, q, k_tree, v_tree, k_cache, v_cache,
                      page_table, logits, temperature, seed, new_ctx_len, dev_status, lse,
                      draft_logits]
        a = StepArgs()
        a.B, a.D, a.K, a.budget, a.V, a.Hq, a.Hkv, a.Dh = B, D, K, budget, V, Hq, Hkv, Dh
        a.num_pages, a.page_size, a.max_pages = num_pages, page_size, max_pages
        a.scale, a.walk, a.philox_offset = scale, walks[walk], philox_offset
        a.topk_logp = _ptr(topk_logp, torch.float32, "topk_logp", (B, D, K))
        a.topk_tok = _ptr(topk_tok, torch.int32, "topk_tok", (B, D, K))
        a.root_tok = _ptr(root_tok, torch.int32, "root_tok", (B,))
        a.ctx_len = _ptr(ctx_len, torch.int32, "ctx_len", (B,))
        a.q = _ptr(q, torch.bfloat16, "q", (B, N, Hq, Dh))
        a.k_tree = _ptr(k_tree, torch.bfloat16, "k_tree", (B, N, Hkv, Dh))
        a.v_tree = _ptr(v_tree, torch.bfloat16, "v_tree", (B, N, Hkv, Dh))
        a.k_cache = _ptr(k_cache, torch.bfloat16, "k_cache", (num_pages, page_size, Hkv, Dh))
        a.v_cache = _ptr(v_cache, torch.bfloat16, "v_cache", (num_pages, page_size, Hkv, Dh))
        a.page_table = _ptr(page_table, torch.int32, "page_table", (B, max_pages))
        a.logits = _ptr(logits, torch.float32, "logits", (B, N, V))
        a.temperature = _ptr(temperature, torch.float32, "temperature", (B,))
        a.seed = _ptr(seed, torch.int64, "seed", (B,))
        a.draft_logits = _ptr(draft_logits, torch.float32, "draft_logits", (B, D, V))
        t = self.tree
        a.parent, a.depth, a.token, a.rank, a.pos = (x.data_ptr() for x in (t.parent, t.depth, t.token,
                                                                             t.rank, t.pos))
        a.score, a.first_child, a.next_sibling = t.score.data_ptr(), t.first_child.data_ptr(), \
            t.next_sibling.data_ptr()
        a.vis, a.n_nodes = t.vis.data_ptr(), t.n_nodes.data_ptr()
        a.attn_out = self.attn_out.data_ptr()
        a.lse = _ptr(lse, torch.float32, "lse", (B, N, Hq))
        a.workspace, a.workspace_bytes = self.workspace.data_ptr(), self.workspace.numel()
        o = self.accept
        a.accept_len, a.out_tokens = o["accept_len"].data_ptr(), o["out_tokens"].data_ptr()
        a.out_nodes, a.bonus = o["out_nodes"].data_ptr(), o["bonus"].data_ptr()
        a.new_ctx_len = _ptr(new_ctx_len, torch.int32, "new_ctx_len", (B,))
        a.dev_status = _ptr(dev_status, torch.int32, "dev_status", (1,))
        self._args = a
        handle = ctypes.c_void_p()
        _check(lib.ddtree_step_create(ctypes.byref(a), ctypes.byref(handle)), "ddtree_step_create")
        self._handle = handle

    def launch(self, stream=None):
        _check(load_library().ddtree_step_launch(self._handle, _stream(stream)), "ddtree_step_launch")

    def close(self):
        if getattr(self, "_handle", None):
            load_library().ddtree_step_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
