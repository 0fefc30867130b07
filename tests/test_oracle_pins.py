"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each test ties one oracle function to a fact the pages or the mathematics fix:
a hand-worked example, a brute-force enumeration, a reduction to a textbook or
library routine, a closed form or a distributional law. A plausible mistake in
the oracle (a dropped term, a wrong index, a swapped operand, a wrong push
order) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
import ddtree_synth as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_topk(rng, B, D, K, V=1000):
    """Random per-depth top-k: sorted descending log-probs (all < 0), distinct tokens."""
    lp = -np.sort(rng.exponential(1.0, size=(B, D, K)), axis=-1).astype(np.float32)
    lp = np.minimum(lp, np.float32(-1e-3))
    tok = np.stack([np.stack([rng.choice(V, size=K, replace=False) for _ in range(D)])
                    for _ in range(B)]).astype(np.int32)
    return lp, tok


# ----------------------------------------------------------------------------
# a0: draft top-k
# ----------------------------------------------------------------------------

def test_draft_topk_matches_torch_logsoftmax_topk():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((3, 4, 500)) * 3).astype(np.float32)
    lp, tok = O.draft_topk(x, 8)
    ref = torch.log_softmax(torch.from_numpy(x).double(), dim=-1)
    v, i = torch.topk(ref, 8, dim=-1)
    assert np.array_equal(tok, i.numpy().astype(np.int32))
    assert np.array_equal(lp, v.numpy().astype(np.float32))


def test_draft_topk_ranks_by_logit_where_fp64_logprobs_merge():
    # 1e-10 and the next fp32 value above it differ by ~6e-18, far below the
    # fp64 spacing near the row's log-sum-exp (~30): their fp64 log-probs are
    # equal, but the larger logit still ranks first
    a = np.float32(1e-10)
    b = np.nextafter(a, np.float32(1))
    x = np.array([[[30.0, a, b, -5.0]]], dtype=np.float32)
    lse = 30.0 + math.log(sum(math.exp(float(v) - 30.0) for v in x[0, 0]))
    assert float(a) - lse == float(b) - lse
    lp, tok = O.draft_topk(x, 3)
    assert tok[0, 0].tolist() == [0, 2, 1]
    assert lp[0, 0, 1] == lp[0, 0, 2] == np.float32(float(b) - lse)


def test_draft_topk_tie_goes_to_lower_token():
    x = np.zeros((1, 1, 6), np.float32)
    x[0, 0, [4, 1, 3]] = 2.0
    lp, tok = O.draft_topk(x, 4)
    assert tok[0, 0].tolist() == [1, 3, 4, 0]
    # three equal maxima and three zeros: p = e^2 / (3 e^2 + 3)
    assert lp[0, 0, 0] == np.float32(math.log(math.exp(2) / (3 * math.exp(2) + 3)))


# ----------------------------------------------------------------------------
# a1: build
# ----------------------------------------------------------------------------

def test_build_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "hand_tree.json")))
    lp = np.array([g["topk_logp"]], np.float32)
    tok = np.array([g["topk_tok"]], np.int32)
    t = O.build_tree(lp, tok, np.array([g["root_tok"]]), np.array([g["ctx_len"]]), g["budget"])
    e = g["expect"]
    assert t.n_nodes[0] == e["n_nodes"]
    for key in ("parent", "depth", "token", "rank", "pos", "first_child", "next_sibling"):
        assert getattr(t, key)[0].tolist() == e[key], key
    np.testing.assert_allclose(t.score[0], e["score"], atol=1e-6)
    assert t.vis[0, :, 0].tolist() == e["vis"]


def _enumerate_candidates(lp_b, D, K):
    """Every node the tree could hold: rank tuples of length 1..D with fp64 path scores."""
    out = []
    for d in range(1, D + 1):
        for ranks in itertools.product(range(K), repeat=d):
            s = np.cumsum([0.0] + [float(lp_b[k, r]) for k, r in enumerate(ranks)])[-1]
            out.append((s, ranks))
    return out


def _tree_paths(t, b):
    paths = {}
    for i in range(int(t.n_nodes[b])):
        ranks = []
        j = i
        while t.parent[b, j] != -1:
            ranks.append(int(t.rank[b, j]))
            j = int(t.parent[b, j])
        paths[i] = tuple(reversed(ranks))
    return paths


@pytest.mark.parametrize("D,K,budget,seed", [(4, 3, 10, 0), (5, 4, 30, 1), (8, 4, 16, 2), (3, 5, 40, 3)])
def test_build_equals_top_budget_by_brute_force(D, K, budget, seed):
    """Scores fall along child and sibling edges, so best-first = the best `budget` candidates."""
    rng = np.random.default_rng(seed)
    lp, tok = _rand_topk(rng, 2, D, K)
    t = O.build_tree(lp, tok, np.array([7, 9]), np.array([0, 5]), budget)
    for b in range(2):
        cands = sorted(_enumerate_candidates(lp[b], D, K), key=lambda c: -c[0])
        want = {r for _, r in cands[:budget]}
        got = _tree_paths(t, b)
        assert t.n_nodes[b] == min(budget, len(cands)) + 1
        assert {p for i, p in got.items() if i > 0} == want
        for i, p in got.items():
            if i == 0:
                continue
            assert t.token[b, i] == tok[b, len(p) - 1, p[-1]]
            exact = np.cumsum([0.0] + [float(lp[b, k, r]) for k, r in enumerate(p)])[-1]
            assert t.score[b, i] == exact
        # pop order is descending score
        assert np.all(np.diff(t.score[b, 1:t.n_nodes[b]]) <= 0)


def test_build_topk1_is_linear_chain():
    """'The Tree That Couldn't Branch', experiment budget=7 topk_cap=1: a single chain."""
    rng = np.random.default_rng(5)
    lp, tok = _rand_topk(rng, 3, 8, 1)
    for budget in (7, 8, 20, 3):
        t = O.build_tree(lp, tok, np.array([1, 2, 3]), np.array([10, 0, 4]), budget)
        n = min(budget, 8) + 1
        for b in range(3):
            assert t.n_nodes[b] == n
            assert t.parent[b, :n].tolist() == [-1] + list(range(n - 1))
            assert t.token[b, 1:n].tolist() == tok[b, :n - 1, 0].tolist()
            assert t.depth[b, :n].tolist() == list(range(n))
            assert np.all(t.parent[b, n:] == -1) and np.all(t.token[b, n:] == -1)
            # a chain's mask is lower-triangular
            vb = O.unpack_vis(t.vis[b:b + 1], budget + 1)[0]
            assert np.array_equal(vb[:n, :n], np.tril(np.ones((n, n), bool)))


@pytest.mark.parametrize("seed", range(6))
def test_build_contains_greedy_chain_prefix(seed):
    """If any depth-d node is present, the all-rank-0 node of depth d is present."""
    rng = np.random.default_rng(100 + seed)
    D, K = 8, 8
    lp, tok = _rand_topk(rng, 4, D, K)
    t = O.build_tree(lp, tok, np.zeros(4, np.int32), np.zeros(4, np.int32), 32)
    for b in range(4):
        paths = _tree_paths(t, b)
        maxd = max(len(p) for p in paths.values())
        for d in range(1, maxd + 1):
            assert (0,) * d in paths.values()


@pytest.mark.parametrize("seed", range(4))
def test_build_structure(seed):
    rng = np.random.default_rng(200 + seed)
    D, K, budget = 6, 5, 40
    lp, tok = _rand_topk(rng, 3, D, K)
    ctx = np.array([0, 17, 4096])
    t = O.build_tree(lp, tok, np.array([3, 4, 5]), ctx, budget)
    N = budget + 1
    # ancestor-or-self via boolean transitive closure of the parent relation
    for b in range(3):
        n = int(t.n_nodes[b])
        A = np.zeros((N, N), bool)
        for i in range(1, n):
            assert 0 <= t.parent[b, i] < i
            A[i, t.parent[b, i]] = True
        reach = np.eye(N, dtype=bool)
        reach[n:, n:] = False
        step = reach.copy()
        for _ in range(N):
            step = (step.astype(np.int64) @ A.astype(np.int64)) > 0
            reach |= step
        assert np.array_equal(O.unpack_vis(t.vis[b:b + 1], N)[0], reach)
        kids = {}
        for i in range(1, n):
            kids.setdefault(int(t.parent[b, i]), []).append(i)
            assert t.depth[b, i] == t.depth[b, t.parent[b, i]] + 1 <= D
            assert t.pos[b, i] == ctx[b] + t.depth[b, i]
        for p, cs in kids.items():
            assert len(cs) <= K
            assert len({int(t.token[b, c]) for c in cs}) == len(cs)
            assert [int(t.rank[b, c]) for c in cs] == list(range(len(cs)))
            chain, c = [], int(t.first_child[b, p])
            while c != -1:
                chain.append(c)
                c = int(t.next_sibling[b, c])
            assert chain == cs
        pc = [bin(int(w)).count("1") for w in t.vis[b, :n, 0]] if N <= 32 else None
        if pc is not None:
            assert pc == [int(d) + 1 for d in t.depth[b, :n]]


def test_build_budget_exhaustion_pads():
    rng = np.random.default_rng(9)
    lp, tok = _rand_topk(rng, 1, 2, 2)       # only 2 + 4 = 6 candidates
    t = O.build_tree(lp, tok, np.array([1]), np.array([3]), 10)
    assert t.n_nodes[0] == 7
    assert np.all(t.parent[0, 7:] == -1) and np.all(t.depth[0, 7:] == -1)
    assert np.all(t.vis[0, 7:] == 0) and np.all(np.isneginf(t.score[0, 7:]))


# ----------------------------------------------------------------------------
# a2: attention
# ----------------------------------------------------------------------------

def _sdpa(q, k, v, mask=None, causal=False):
    """torch SDPA in fp64 on the CPU: q [H,n,Dh], k/v [H,m,Dh]."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        attn_mask=None if mask is None else torch.from_numpy(mask)[None, None],
        is_causal=causal)[0].numpy()


def test_attention_chain_no_context_is_causal_sdpa():
    rng = np.random.default_rng(11)
    N, Hq, Hkv, Dh = 9, 4, 2, 16
    parent = np.array([[-1] + list(range(N - 1))], np.int32)
    n_nodes = np.array([N], np.int32)
    vis = O.visibility_matrix(parent, n_nodes, N)
    q = rng.standard_normal((1, N, Hq, Dh))
    kt = rng.standard_normal((1, N, Hkv, Dh))
    vt = rng.standard_normal((1, N, Hkv, Dh))
    kc = np.zeros((1, 64, Hkv, Dh))
    out = O.tree_verify_attention(q, kt, vt, kc, kc, np.zeros((1, 1), np.int32),
                                  np.array([0]), vis, n_nodes, 1 / math.sqrt(Dh), 64)
    G = Hq // Hkv
    ref = _sdpa(q[0].transpose(1, 0, 2), np.repeat(kt[0].transpose(1, 0, 2), G, 0),
                np.repeat(vt[0].transpose(1, 0, 2), G, 0), causal=True)
    np.testing.assert_allclose(out[0], ref.transpose(1, 0, 2), rtol=1e-12, atol=1e-12)


def test_attention_paged_context_and_tree_mask_vs_sdpa():
    """Paged context plus a general tree mask equals SDPA over the contiguous keys."""
    rng = np.random.default_rng(12)
    B, N, Hq, Hkv, Dh, ps = 2, 11, 6, 2, 32, 16
    ctx = np.array([37, 0])
    lp, tok = _rand_topk(rng, B, 4, 3)
    t = O.build_tree(lp, tok, np.array([1, 2]), ctx, N - 1)
    vis = O.unpack_vis(t.vis, N)
    q = rng.standard_normal((B, N, Hq, Dh))
    kt = rng.standard_normal((B, N, Hkv, Dh))
    vt = rng.standard_normal((B, N, Hkv, Dh))
    # logical contiguous contexts, then scattered into a shuffled page pool
    kctx = [rng.standard_normal((L, Hkv, Dh)) for L in ctx]
    vctx = [rng.standard_normal((L, Hkv, Dh)) for L in ctx]
    npages = [-(-int(L) // ps) for L in ctx]
    perm = rng.permutation(sum(npages) + 3)
    kc = rng.standard_normal((len(perm), ps, Hkv, Dh)) * 100   # junk in unused slots
    vc = rng.standard_normal((len(perm), ps, Hkv, Dh)) * 100
    table = np.full((B, 4), -1, np.int32)
    k = 0
    for b in range(B):
        for p in range(npages[b]):
            page = perm[k]; k += 1
            table[b, p] = page
            lo, hi = p * ps, min((p + 1) * ps, ctx[b])
            kc[page, :hi - lo] = kctx[b][lo:hi]
            vc[page, :hi - lo] = vctx[b][lo:hi]
    out, lse = O.tree_verify_attention(q, kt, vt, kc, vc, table, ctx, vis, t.n_nodes,
                                       0.3, ps, want_lse=True)
    G = Hq // Hkv
    for b in range(B):
        L, n = int(ctx[b]), int(t.n_nodes[b])
        keys = np.concatenate([kctx[b], kt[b]], 0).transpose(1, 0, 2)   # [Hkv, L+N, Dh]
        vals = np.concatenate([vctx[b], vt[b]], 0).transpose(1, 0, 2)
        mask = np.concatenate([np.ones((N, L), bool), vis[b]], 1)
        mask[n:] = True      # pad rows: compared as zeros below
        ref = _sdpa(q[b].transpose(1, 0, 2) * (0.3 * math.sqrt(Dh)), np.repeat(keys, G, 0),
                    np.repeat(vals, G, 0), mask=mask)
        np.testing.assert_allclose(out[b, :n], ref.transpose(1, 0, 2)[:n], rtol=1e-10, atol=1e-10)
        assert np.all(out[b, n:] == 0)
        # lse closed form for one row
        s = 0.3 * (keys[0][mask[0]] @ q[b, 0, 0])
        assert abs(lse[b, 0, 0] - math.log(np.exp(s).sum())) < 1e-10


def test_attention_single_key_returns_value():
    rng = np.random.default_rng(13)
    q = rng.standard_normal((1, 1, 2, 8))
    kt = rng.standard_normal((1, 1, 1, 8))
    vt = rng.standard_normal((1, 1, 1, 8))
    out = O.tree_verify_attention(q, kt, vt, np.zeros((1, 4, 1, 8)), np.zeros((1, 4, 1, 8)),
                                  np.zeros((1, 1), np.int32), np.array([0]),
                                  np.ones((1, 1, 1), bool), np.array([1]), 0.5, 4)
    np.testing.assert_array_equal(out[0, 0, 0], vt[0, 0, 0])
    np.testing.assert_array_equal(out[0, 0, 1], vt[0, 0, 0])


def test_attention_row_matches_full():
    w = S.config("tiny")
    dl, root, _ = S.draft_inputs(w)
    lp, tok = O.draft_topk(dl, w.K)
    ctx = S.context_lengths(w)
    t = O.build_tree(lp, tok, root, ctx, w.budget)
    table, npg = S.paged_layout(w, ctx)
    qkv = S.qkv_tree(w)
    kv = S.kv_cache(w, npg)
    vis = O.unpack_vis(t.vis, w.N)
    f = O.bf16_to_f64
    full = O.tree_verify_attention(f(qkv["q"]), f(qkv["k_tree"]), f(qkv["v_tree"]),
                                   f(kv["k_cache"]), f(kv["v_cache"]), table, ctx, vis,
                                   t.n_nodes, 1 / math.sqrt(w.Dh), w.page_size)
    for (b, i, h) in [(0, 0, 0), (0, 5, 3), (0, 16, 1)]:
        row, _ = O.attention_row(qkv["q"], qkv["k_tree"], qkv["v_tree"], kv["k_cache"],
                                 kv["v_cache"], table, ctx, vis, t.n_nodes,
                                 1 / math.sqrt(w.Dh), w.page_size, b, i, h)
        np.testing.assert_allclose(row, full[b, i, h], rtol=1e-11, atol=1e-12)


# ----------------------------------------------------------------------------
# a3: greedy accept
# ----------------------------------------------------------------------------

def test_argmax_rule():
    assert O.argmax_lowest(np.array([1.0, 3.0, 3.0, 2.0])) == 1
    assert O.argmax_lowest(np.array([np.nan, 1.0, np.nan, 1.0])) == 1
    assert O.argmax_lowest(np.array([np.nan, -np.inf, np.nan])) == 1
    assert O.argmax_lowest(np.array([np.nan, np.nan])) == 0
    assert O.argmax_lowest(np.array([-np.inf, -np.inf])) == 0


def test_greedy_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "hand_tree.json")))
    lp = np.array([g["topk_logp"]], np.float32)
    tok = np.array([g["topk_tok"]], np.int32)
    t = O.build_tree(lp, tok, np.array([g["root_tok"]]), np.array([g["ctx_len"]]), g["budget"])
    gr = g["greedy"]
    logits = np.zeros((1, 4, gr["V"]), np.float32)
    for u, a in enumerate(gr["argmax_per_node"]):
        logits[0, u, a] = 1.0
    r = O.accept_greedy(logits, t, g["D"])
    assert r.accept_len[0] == gr["accept_len"]
    assert r.bonus[0] == gr["bonus"]
    n = gr["accept_len"] + 1
    assert r.out_tokens[0, :n].tolist() == gr["out_tokens"]
    assert r.out_nodes[0, :n].tolist() == gr["out_nodes"]
    assert np.all(r.out_tokens[0, n:] == -1)


def _brute_force_greedy(logits, t, b):
    """Enumerate every root path; keep those whose edges match the parent's argmax."""
    n = int(t.n_nodes[b])
    am = [int(np.argmax(logits[b, u])) for u in range(n)]
    best = [0]
    for leaf in range(n):
        path = []
        j = leaf
        while j != -1:
            path.append(j)
            j = int(t.parent[b, j])
        path = path[::-1]
        if all(t.token[b, path[k + 1]] == am[path[k]] for k in range(len(path) - 1)):
            if len(path) > len(best):
                best = path
    return best, am[best[-1]]


@pytest.mark.parametrize("seed", range(8))
def test_greedy_brute_force_paths(seed):
    rng = np.random.default_rng(300 + seed)
    B, D, K, V = 4, 5, 3, 12
    lp = -np.sort(rng.exponential(1.0, (B, D, K)), -1).astype(np.float32) - 1e-3
    tok = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(D)])
                    for _ in range(B)]).astype(np.int32)
    t = O.build_tree(lp, tok, np.zeros(B, np.int32), np.zeros(B, np.int32), 20)
    # bias logits toward tree tokens so that long paths occur
    logits = rng.standard_normal((B, 21, V)).astype(np.float32)
    for b in range(B):
        for u in range(int(t.n_nodes[b])):
            c = int(t.first_child[b, u])
            if c != -1 and rng.random() < 0.7:
                logits[b, u, t.token[b, c]] += 5.0
    r = O.accept_greedy(logits, t, D)
    for b in range(B):
        path, bonus = _brute_force_greedy(logits, t, b)
        assert r.accept_len[b] == len(path) - 1
        assert r.out_nodes[b, :len(path)].tolist() == path
        assert r.bonus[b] == bonus
        assert r.out_tokens[b, :len(path) - 1].tolist() == [int(t.token[b, c]) for c in path[1:]]


def test_greedy_chain_equals_sequential_argmax_matching():
    """Linear DFlash rule: accept draft i while the argmax at position i-1 equals it."""
    rng = np.random.default_rng(17)
    B, D, V = 6, 7, 10
    lp = -np.sort(rng.exponential(1.0, (B, D, 1)), -1).astype(np.float32) - 1e-3
    tok = rng.integers(0, V, (B, D, 1)).astype(np.int32)
    t = O.build_tree(lp, tok, np.zeros(B, np.int32), np.zeros(B, np.int32), 7)
    logits = rng.standard_normal((B, 8, V)).astype(np.float32)
    for b in range(B):
        stop = rng.integers(0, D + 1)
        for i in range(stop):
            logits[b, i, tok[b, i, 0]] += 10.0
    r = O.accept_greedy(logits, t, D)
    for b in range(B):
        draft = tok[b, :, 0]
        preds = logits[b].argmax(-1)
        k = 0
        while k < D and preds[k] == draft[k]:
            k += 1
        assert r.accept_len[b] == k
        assert r.bonus[b] == preds[k]


def test_greedy_planted_full_depth():
    w = S.config("latency")
    D, K = w.D, w.K
    rng = np.random.default_rng(19)
    lp, tok = _rand_topk(rng, 1, D, K, V=500)
    lp[..., 0] = -1e-3          # a confident drafter: the rank-0 chain is built to full depth
    lp[..., 1:] -= 3.0
    t = O.build_tree(lp, tok, np.array([0]), np.array([0]), 32)
    assert t.depth[0].max() == D
    logits = rng.standard_normal((1, 33, 500)).astype(np.float32)
    u = 0
    for d in range(D):                     # plant the rank-0 chain token at every chain node
        logits[0, u, tok[0, d, 0]] += 50.0
        u = int(t.first_child[0, u])
    logits[0, u, 123] += 50.0
    r = O.accept_greedy(logits, t, D)
    assert r.accept_len[0] == D
    assert r.out_tokens[0].tolist() == list(tok[0, :, 0]) + [123]


# ----------------------------------------------------------------------------
# a4: temperature accept
# ----------------------------------------------------------------------------

def test_philox_matches_triton_interpreter():
    """Philox4x32-10 against triton's own implementation, run by its CPU interpreter."""
    os.environ["TRITON_INTERPRET"] = "1"
    triton = pytest.importorskip("triton")
    import triton.language as tl

    @triton.jit
    def kern(out_ptr, seed, c0_ptr, c1_ptr, c2_ptr, c3_ptr, NUM: tl.constexpr):
        i = tl.arange(0, NUM)
        a, b, c, d = tl.philox(seed, tl.load(c0_ptr + i), tl.load(c1_ptr + i),
                               tl.load(c2_ptr + i), tl.load(c3_ptr + i))
        tl.store(out_ptr + 4 * i + 0, a)
        tl.store(out_ptr + 4 * i + 1, b)
        tl.store(out_ptr + 4 * i + 2, c)
        tl.store(out_ptr + 4 * i + 3, d)

    rng = np.random.default_rng(23)
    for seed in (0, 12345, 0xDEADBEEFCAFEF00D & 0x7FFFFFFFFFFFFFFF):
        ctr = rng.integers(0, 2 ** 32, size=(4, 16), dtype=np.uint64)
        ctr[:, 0] = 0
        ctr[:, 1] = 0xFFFFFFFF
        cols = [torch.from_numpy(ctr[k].astype(np.uint32)) for k in range(4)]
        out = torch.zeros(64, dtype=torch.uint32)
        kern[(1,)](out, seed, *cols, NUM=16)
        got = out.numpy().reshape(16, 4)
        for n in range(16):
            mine = O.philox4x32_10(ctr[:, n], (seed & 0xFFFFFFFF, seed >> 32))
            assert tuple(int(x) for x in got[n]) == mine
        vec = O.philox4x32_10_np(*ctr, seed & 0xFFFFFFFF, seed >> 32)
        assert np.array_equal(np.stack(vec, 1).astype(np.uint32), got)


def test_uniform_map_open_interval():
    u = O.to_uniform(np.array([0, 0xFF, 0xFFFFFFFF], dtype=np.uint64))
    assert u[0] == 0.5 * 2 ** -24 and u[1] == u[0] and u[2] == 1 - 0.5 * 2 ** -24


def _tiny_sampling_tree(rng, V=8, K=4, D=3, budget=12):
    lp = -np.sort(rng.exponential(1.0, (1, D, K)), -1).astype(np.float32) - 1e-3
    tok = np.stack([rng.choice(V, K, replace=False) for _ in range(D)])[None].astype(np.int32)
    return O.build_tree(lp, tok, np.array([0]), np.array([0]), budget)


def test_sampling_first_token_follows_target_softmax():
    """Chi-square: emitted tokens are distributed as softmax(logits / T) at the root,
    and the second token, given an accepted first child c, as softmax(logits_c / T)."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(29)
    V = 8
    t = _tiny_sampling_tree(rng, V=V)
    logits = (rng.standard_normal((1, 13, V)) * 1.5).astype(np.float32)
    c0 = int(t.first_child[0, 0])
    logits[0, 0, t.token[0, c0]] += 2.0      # make the first child likely, to condition on it
    T = 0.8
    n = 20000
    first = np.zeros(V, np.int64)
    second = np.zeros(V, np.int64)
    for s in range(n):
        r = O.accept_sample(logits, t, 3, np.array([T], np.float32),
                            np.array([1_000_000 + s], np.uint64), 7)
        first[r.out_tokens[0, 0]] += 1
        if r.accept_len[0] >= 1 and r.out_nodes[0, 1] == c0:
            second[r.out_tokens[0, 1]] += 1
    p = np.exp(logits[0, 0].astype(np.float64) / T)
    p /= p.sum()
    assert chisquare(first, p * n).pvalue > 0.001 / 2
    p2 = np.exp(logits[0, c0].astype(np.float64) / T)
    p2 /= p2.sum()
    m = second.sum()
    assert m > 500
    assert chisquare(second, p2 * m).pvalue > 0.001 / 2


def test_sampling_low_temperature_equals_greedy():
    rng = np.random.default_rng(31)
    B, D, K, V = 5, 4, 3, 40
    lp = -np.sort(rng.exponential(1.0, (B, D, K)), -1).astype(np.float32) - 1e-3
    tok = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(D)])
                    for _ in range(B)]).astype(np.int32)
    t = O.build_tree(lp, tok, np.zeros(B, np.int32), np.zeros(B, np.int32), 15)
    logits = (rng.standard_normal((B, 16, V)) * 5).astype(np.float32)
    for b in range(B):
        for u in range(16):
            c = int(t.first_child[b, u])
            if c != -1 and rng.random() < 0.6:
                logits[b, u, t.token[b, c]] += 30.0
    g = O.accept_greedy(logits, t, D)
    s = O.accept_sample(logits, t, D, np.full(B, 1e-3, np.float32),
                        np.arange(B, dtype=np.uint64) + 77, 0)
    assert np.array_equal(g.accept_len, s.accept_len)
    assert np.array_equal(g.out_tokens, s.out_tokens)
    assert np.array_equal(g.bonus, s.bonus)


def test_sampling_leaf_root_bonus_is_gumbel_max_sample():
    """A root with no children: the bonus is a plain sample of softmax(l/T)."""
    from scipy.stats import chisquare
    V = 6
    t = O.build_tree(np.zeros((1, 1, 1), np.float32) - 1, np.zeros((1, 1, 1), np.int32),
                     np.array([0]), np.array([0]), 0)
    assert t.n_nodes[0] == 1
    logits = np.array([[[0.0, 1.0, -1.0, 2.0, 0.5, -0.5]]], np.float32)
    cnt = np.zeros(V, np.int64)
    for s in range(12000):
        r = O.accept_sample(logits, t, 1, np.array([1.3], np.float32), np.array([s], np.uint64), 3)
        assert r.accept_len[0] == 0
        cnt[r.bonus[0]] += 1
    p = np.exp(logits[0, 0].astype(np.float64) / 1.3)
    p /= p.sum()
    assert chisquare(cnt, p * cnt.sum()).pvalue > 0.001


def test_sampling_rejects_nonpositive_temperature():
    t = O.build_tree(np.zeros((1, 1, 1), np.float32) - 1, np.zeros((1, 1, 1), np.int32),
                     np.array([0]), np.array([0]), 1)
    with pytest.raises(ValueError):
        O.accept_sample(np.zeros((1, 2, 4), np.float32), t, 1, np.array([0.0], np.float32),
                        np.array([1], np.uint64), 0)


def test_build_equal_scores_follow_push_order():
    """Reading for ties: the earlier push wins, and a popped node pushes its child first.

    Worked by hand: depth-1 log-probs (-0.5, -1.0), depth-2 (-0.5, -2.0). Pop node 1
    (score -0.5); its child (-0.5-0.5 = -1.0) is pushed before its sibling (0-1.0 = -1.0),
    so with budget 2 the second node is the depth-2 child.
    """
    lp = np.array([[[-0.5, -1.0], [-0.5, -2.0]]], np.float32)
    tok = np.array([[[1, 2], [3, 4]]], np.int32)
    t = O.build_tree(lp, tok, np.array([0]), np.array([0]), 2)
    assert t.token[0].tolist() == [0, 1, 3]
    assert t.parent[0].tolist() == [-1, 0, 1]
    t3 = O.build_tree(lp, tok, np.array([0]), np.array([0]), 3)
    assert t3.token[0].tolist() == [0, 1, 3, 2]


# ---------------------------------------------------------------------------
# commit of the verified path's K/V
# ---------------------------------------------------------------------------

def test_commit_hand_worked_example():
    # page_size 4, request 0 owns pages [2, 0, 1] (tokens 0-3 on page 2, 4-7 on
    # page 0, 8-11 on page 1) and holds 3 tokens; the path is rows 0, 2, 5
    # (accept_len 2). Worked by hand: token 3 -> page 2 slot 3, token 4 ->
    # page 0 slot 0, token 5 -> page 0 slot 1; the new length is 6.
    N, Hkv, Dh = 6, 1, 2
    k_tree = np.arange(1, N + 1, dtype=np.float64)[None, :, None, None] * np.ones((1, N, Hkv, Dh))
    v_tree = -k_tree
    k_cache = np.zeros((3, 4, Hkv, Dh))
    v_cache = np.zeros((3, 4, Hkv, Dh))
    kc, vc, new_ctx = O.commit_kv(k_tree, v_tree, np.array([[0, 2, 5, -1]]), np.array([2]),
                                  np.array([3]), np.array([[2, 0, 1]]), k_cache, v_cache, 4)
    assert new_ctx.tolist() == [6]
    expect = np.zeros((3, 4))
    expect[2, 3], expect[0, 0], expect[0, 1] = 1.0, 3.0, 6.0   # rows 0, 2, 5 hold 1, 3, 6
    assert np.array_equal(kc[:, :, 0, 0], expect) and np.array_equal(kc[:, :, 0, 1], expect)
    assert np.array_equal(vc[:, :, 0, 0], -expect)


@pytest.mark.parametrize("seed", range(4))
def test_commit_appends_the_path_to_the_token_sequence(seed):
    # the cache read as a token sequence after the commit is the old sequence
    # followed by the path rows in path order; no other slot changes
    rng = np.random.default_rng(seed)
    B, N, Hkv, Dh, page, D = 3, 9, 2, 4, 4, 4
    ctx = rng.integers(0, 12, B).astype(np.int32)
    max_pages = 5
    table = rng.permutation(B * max_pages).reshape(B, max_pages).astype(np.int32)
    k_cache = rng.standard_normal((B * max_pages, page, Hkv, Dh))
    v_cache = rng.standard_normal((B * max_pages, page, Hkv, Dh))
    k_tree = rng.standard_normal((B, N, Hkv, Dh))
    v_tree = rng.standard_normal((B, N, Hkv, Dh))
    acc = rng.integers(0, D + 1, B).astype(np.int32)
    nodes = np.full((B, D + 1), -1, np.int32)
    for b in range(B):
        nodes[b, 0] = 0
        nodes[b, 1:acc[b] + 1] = np.sort(rng.choice(np.arange(1, N), acc[b], replace=False))
    kc, vc, new_ctx = O.commit_kv(k_tree, v_tree, nodes, acc, ctx, table, k_cache, v_cache, page)
    assert np.array_equal(new_ctx, ctx + acc + 1)
    for b in range(B):
        path = nodes[b, :acc[b] + 1]
        for old, new, tree in ((k_cache, kc, k_tree), (v_cache, vc, v_tree)):
            seq_old = O.gather_context(old, table, b, int(ctx[b]), page)
            seq_new = O.gather_context(new, table, b, int(new_ctx[b]), page)
            assert np.array_equal(seq_new, np.concatenate([seq_old, tree[b, path]], axis=0))
    touched = np.zeros(k_cache.shape[:2], bool)
    for b in range(B):
        for t in range(int(ctx[b]), int(new_ctx[b])):
            touched[table[b, t // page], t % page] = True
    assert np.array_equal(kc[~touched], k_cache[~touched])
    assert np.array_equal(vc[~touched], v_cache[~touched])


def test_commit_of_a_chain_is_the_linear_dflash_commit():
    # top-k 1: the tree is the D-node chain (node index = depth), the greedy
    # walk accepts a prefix, and the commit appends verify rows 0..a in order
    w = S.config("tiny")
    dl, root, _ = S.draft_inputs(w)
    lp, tok = O.draft_topk(dl, 1)
    ctx = np.array([5], np.int32)
    tree = O.build_tree(lp, tok, root, ctx, w.D)
    assert tree.parent[0, 1:].tolist() == list(range(w.D))
    logits = np.zeros((1, w.D + 1, w.V))
    for d in range(w.D):   # the target agrees with the first three draft tokens
        logits[0, d, tree.token[0, d + 1] if d < 3 else (tree.token[0, d + 1] + 1) % w.V] = 1.0
    acc = O.accept_greedy(logits, tree, w.D)
    assert int(acc.accept_len[0]) == 3
    rng = np.random.default_rng(0)
    k_tree = rng.standard_normal((1, w.D + 1, 1, 4))
    v_tree = rng.standard_normal((1, w.D + 1, 1, 4))
    k_cache = rng.standard_normal((4, 4, 1, 4))
    v_cache = rng.standard_normal((4, 4, 1, 4))
    table = np.array([[3, 1, 0, 2]], np.int32)
    kc, _, new_ctx = O.commit_kv(k_tree, v_tree, acc.out_nodes, acc.accept_len, ctx, table,
                                 k_cache, v_cache, 4)
    assert new_ctx.tolist() == [9]
    seq = O.gather_context(kc, table, 0, 9, 4)
    assert np.array_equal(seq[5:9], k_tree[0, 0:4])


# ---------------------------------------------------------------------------
# draft-ratio temperature walk
# ---------------------------------------------------------------------------

def _star_tree(child_tokens):
    """Root 0 with children 1..k (depth 1, leaves) carrying the given tokens in rank order."""
    k = len(child_tokens)
    lp = -np.arange(1, k + 1, dtype=np.float32)[None, None, :] * 0.1
    tok = np.asarray(child_tokens, np.int32)[None, None, :]
    return O.build_tree(lp, tok, np.array([0]), np.array([0]), k)


def _softmax64(x, T):
    z = np.asarray(x, np.float64) / T
    e = np.exp(z - z.max())
    return e / e.sum()


@pytest.mark.parametrize("k", [1, 3])
def test_ratio_iid_candidates_emit_the_target_distribution(k):
    """Chi-square: with the k candidates drawn independently from the draft
    distribution p, the first emitted token follows q = softmax(target / T)
    (k = 1: the speculative-sampling theorem of the linear chain; k > 1: the
    multi-candidate residual update)."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(40 + k)
    V, T, n = 6, 0.9, 6000
    logits = (rng.standard_normal((1, k + 1, V)) * 1.2).astype(np.float32)
    draft = (rng.standard_normal((1, 1, V)) * 1.2).astype(np.float32)
    p = _softmax64(draft[0, 0], T)
    q = _softmax64(logits[0, 0], T)
    counts = np.zeros(V, np.int64)
    draws = rng.choice(V, size=(n, k), p=p)
    for s in range(n):
        t = _star_tree(draws[s])
        r = O.accept_sample_ratio(logits, draft, t, 1, np.array([T], np.float32),
                                  np.array([5_000_000 + s], np.uint64), 3)
        counts[r.out_tokens[0, 0]] += 1
    assert chisquare(counts, q * n).pvalue > 0.001 / 2


def test_ratio_single_child_is_accepted_with_min_one_q_over_p():
    """One fixed child x: accepted with probability min(1, q(x)/p(x)) (binomial, 4 sigma)."""
    rng = np.random.default_rng(7)
    V, T, n = 8, 0.7, 4000
    logits = (rng.standard_normal((1, 2, V)) * 1.5).astype(np.float32)
    draft = (rng.standard_normal((1, 1, V)) * 1.5).astype(np.float32)
    p = _softmax64(draft[0, 0], T)
    q = _softmax64(logits[0, 0], T)
    for x in (int(np.argmax(p)), int(np.argmax(q))):
        t = _star_tree([x])
        hits = sum(int(O.accept_sample_ratio(logits, draft, t, 1, np.array([T], np.float32),
                                             np.array([s], np.uint64), 11).accept_len[0])
                   for s in range(n))
        a = min(1.0, q[x] / p[x])
        assert abs(hits / n - a) <= 4 * math.sqrt(a * (1 - a) / n) + 1e-9


def test_ratio_equal_draft_and_target_accept_every_level():
    # p == q at every node: r(x)/p(x) = 1 > U, so the walk takes the top child
    # at each level and reaches depth D
    rng = np.random.default_rng(3)
    B, D, V = 3, 5, 20
    draft = (rng.standard_normal((B, D, V)) * 2).astype(np.float32)
    lp, tok = O.draft_topk(draft, 2)
    tree = O.build_tree(lp, tok, np.zeros(B, np.int32), np.zeros(B, np.int32), 12)
    logits = np.zeros((B, 13, V), np.float32)
    for b in range(B):
        for u in range(int(tree.n_nodes[b])):
            d = int(tree.depth[b, u])
            logits[b, u] = draft[b, d] if d < D else rng.standard_normal(V)
    for s in range(20):
        r = O.accept_sample_ratio(logits, draft, tree, D, np.full(B, 0.8, np.float32),
                                  np.arange(B, dtype=np.uint64) + 100 * s, 0)
        for b in range(B):
            path = r.out_nodes[b, 1:r.accept_len[b] + 1]
            assert all(int(tree.rank[b, c]) == 0 for c in path)   # always the first child
            last = int(r.out_nodes[b, r.accept_len[b]])
            assert int(tree.first_child[b, last]) == -1           # stopped at a leaf


def test_ratio_leaf_bonus_equals_the_renormalising_walk():
    # a node without children draws its bonus from q in both walks, from the
    # same Gumbel noise: the two oracles agree exactly (accept_sample is pinned
    # by its own chi-square tests)
    rng = np.random.default_rng(12)
    B, V = 4, 50
    lp = np.zeros((B, 1, 1), np.float32)
    tok = np.zeros((B, 1, 1), np.int32)
    tree = O.build_tree(lp, tok, np.zeros(B, np.int32), np.zeros(B, np.int32), 0)   # root only
    logits = (rng.standard_normal((B, 1, V)) * 2).astype(np.float32)
    draft = (rng.standard_normal((B, 1, V)) * 2).astype(np.float32)
    for s in range(10):
        T = np.full(B, 0.6 + 0.1 * s, np.float32)
        seed = np.arange(B, dtype=np.uint64) + 1000 * s
        a = O.accept_sample(logits, tree, 1, T, seed, 5)
        r = O.accept_sample_ratio(logits, draft, tree, 1, T, seed, 5)
        assert np.array_equal(a.bonus, r.bonus) and (r.accept_len == 0).all()
