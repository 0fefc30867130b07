"""Test helpers: seeded workloads (ddtree_synth) staged for the oracle and the GPU."""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

import ddtree_synth as S
import oracle as O


@dataclass
class Staged:
    w: S.Workload
    draft_logits: np.ndarray
    root: np.ndarray
    ctx: np.ndarray
    topk_logp: np.ndarray
    topk_tok: np.ndarray
    tree: O.Tree
    table: np.ndarray = None
    num_pages: int = 0
    qkv: dict = None
    kv: dict = None
    logits: np.ndarray = None


def stage(w: S.Workload, attention=True, logits=True, ctx=None) -> Staged:
    dl, root, _ = S.draft_inputs(w)
    ctx = S.context_lengths(w) if ctx is None else np.asarray(ctx, np.int32)
    lp, tok = O.draft_topk(dl, w.K)
    tree = O.build_tree(lp, tok, root, ctx, w.budget)
    st = Staged(w, dl, root, ctx, lp, tok, tree)
    if attention:
        st.table, st.num_pages = S.paged_layout(w, ctx)
        st.qkv = S.qkv_tree(w)
        st.kv = S.kv_cache(w, max(st.num_pages, 1))
    if logits:
        st.logits = S.target_logits(w, dl, tree.depth, tree.n_nodes)
    return st


def scale(w):
    return 1.0 / math.sqrt(w.Dh)


# ---------------------------------------------------------------------------
# GPU side (torch only for memory)
# ---------------------------------------------------------------------------

def dev(a, device="cuda"):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).to(device)
    if a.dtype == np.uint64:
        return torch.from_numpy(a.view(np.int64)).to(device)
    return torch.from_numpy(a).to(device)


def host_u32(t):
    return t.cpu().numpy().view(np.uint32)


def bf16_to_f64_t(t):
    return t.float().cpu().numpy().astype(np.float64)


def attn_tolerance(got, ref, atol=2e-2, rel_l2=1e-2):
    """Max abs and relative L2 error bars of the benchmark spec's tolerance."""
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)) if got.size else 0.0
    return err, rel, (err <= atol and rel <= rel_l2)
