"""GPU parity: every C-ABI call against the fp64 oracle on the same seeded inputs.

Bars: tree structure, masks, positions, fp64 scores, accept lengths and tokens
bit-exact; attention within max abs 2e-2 and relative L2 1e-2 of the oracle;
sampled accepts identical given the same Philox counters on every request
whose scaled decision margin exceeds 1e-4, with at most two requests per test
below it.

The sampled walk's bar, derived: the kernel's q(x) = expf((l - M) / T) / Z in
fp32 carries a relative error of at most about 3 * 2^-24 |l - M| / T (the
exponent's rounding, |l - M| / T <= 40 here) + 2 ulp (expf) + the fp32 sum Z
over V (at most about 2e-6), i.e. below 1e-5. A child test compares u with
q(x_j) / R, R = 1 - sum_{i<j} q(x_i) formed in fp64 from the fp32 q values, so
the threshold moves by at most about 1e-5 / R; the bonus compares perturbed
scores logits * (1/T) + g whose error is below 1e-5 as well. The oracle's
``margin_scaled`` divides each child test's margin by its conditioning 1/R,
so a scaled margin above 1e-4 is ten times the worst error of that decision.
"""
import math

import numpy as np
import pytest

import ddtree_synth as S
import oracle as O
from _stage import stage, scale, dev, host_u32, attn_tolerance

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import tree_speculative_decoding_ddtree_gb300 as dd  # noqa: E402

MARGIN = 1e-4
TREE_FIELDS = ("parent", "depth", "token", "rank", "pos", "first_child", "next_sibling", "n_nodes")


def status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def gpu_tree(st, stat=None):
    return dd.ddtree_build(dev(st.topk_logp), dev(st.topk_tok), dev(st.root), dev(st.ctx),
                           st.w.budget, dev_status=stat)


def assert_tree_equal(tree, ref):
    torch.cuda.synchronize()
    for name in TREE_FIELDS:
        got = getattr(tree, name).cpu().numpy()
        assert np.array_equal(got, getattr(ref, name)), name
    assert np.array_equal(tree.score.cpu().numpy(), ref.score)   # fp64 bit-exact
    assert np.array_equal(host_u32(tree.vis), ref.vis)


# ---------------------------------------------------------------------------
# ddtree_build
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "latency", "batched", "deep", "temperature"])
def test_build_matches_oracle(name):
    st = stage(S.config(name), attention=False, logits=False)
    s = status()
    assert_tree_equal(gpu_tree(st, s), st.tree)
    assert int(s.item()) == 0


def _random_topk(seed, B, D, K, V=5000, ties=False):
    rng = np.random.default_rng(seed)
    if ties:   # coarse log-probs: many exactly equal path scores
        lp = -np.sort(rng.integers(1, 4, size=(B, D, K)), axis=-1).astype(np.float32) * 0.5
    else:
        lp = -np.sort(rng.exponential(1.0, size=(B, D, K)), axis=-1).astype(np.float32) - 1e-3
    tok = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(D)])
                    for _ in range(B)]).astype(np.int32)
    return lp, tok


@pytest.mark.parametrize("B,D,K,budget,ties", [
    (3, 8, 1, 20, False),      # chain that runs out of candidates (n_nodes < N)
    (2, 8, 1, 7, False),       # budget 7, top-k cap 1: the linear chain
    (5, 4, 3, 0, False),       # budget 0: root only
    (4, 64, 32, 127, False),   # largest tree, widest cap, deepest draft
    (6, 6, 4, 50, True),       # many equal scores: push order decides
    (3, 5, 3, 20, True),       # equal scores, one-slot heap
    (4, 16, 8, 100, True),     # equal scores, four-slot heap
    (33, 5, 5, 31, True),      # more requests than one block holds
    (1, 2, 2, 10, False),      # every candidate fits
])
def test_build_edge_cases(B, D, K, budget, ties):
    lp, tok = _random_topk(1000 + B * 7 + K, B, D, K, ties=ties)
    root = np.arange(B, dtype=np.int32) + 3
    ctx = (np.arange(B, dtype=np.int32) * 97) % 5000
    ref = O.build_tree(lp, tok, root, ctx, budget)
    tree = dd.ddtree_build(dev(lp), dev(tok), dev(root), dev(ctx), budget)
    assert_tree_equal(tree, ref)


def test_build_nan_logprob_ranks_last():
    lp, tok = _random_topk(7, 2, 4, 3)
    lp[0, 1, 0] = np.nan
    lp[1, 0, 2] = np.nan
    root = np.zeros(2, np.int32)
    ctx = np.zeros(2, np.int32)
    ref = O.build_tree(lp, tok, root, ctx, 12)
    assert_tree_equal(dd.ddtree_build(dev(lp), dev(tok), dev(root), dev(ctx), 12), ref)


# ---------------------------------------------------------------------------
# tree_verify_attn
# ---------------------------------------------------------------------------

def run_attn(st, lse=False, stat=None):
    w = st.w
    tree = gpu_tree(st)
    out_lse = torch.empty((w.B, w.N, w.Hq), dtype=torch.float32, device="cuda") if lse else None
    out = dd.tree_verify_attn(dev(st.qkv["q"]), dev(st.qkv["k_tree"]), dev(st.qkv["v_tree"]),
                              dev(st.kv["k_cache"]), dev(st.kv["v_cache"]), dev(st.table),
                              dev(st.ctx), tree.vis, tree.n_nodes, scale(w), lse=out_lse,
                              dev_status=stat)
    torch.cuda.synchronize()
    return out, out_lse


def oracle_full(st, want_lse=False):
    f = O.bf16_to_f64
    w = st.w
    return O.tree_verify_attention(f(st.qkv["q"]), f(st.qkv["k_tree"]), f(st.qkv["v_tree"]),
                                   f(st.kv["k_cache"]), f(st.kv["v_cache"]), st.table, st.ctx,
                                   O.unpack_vis(st.tree.vis, w.N), st.tree.n_nodes, scale(w),
                                   w.page_size, want_lse=want_lse)


def oracle_slice(st, b, kvh):
    """Oracle output rows of one (request, KV head): ``[N, G, Dh]``, on that slice only."""
    w = st.w
    f = O.bf16_to_f64
    G = w.G
    L = int(st.ctx[b])
    npg = -(-L // w.page_size)
    pages = st.table[b, :npg]
    kc = f(st.kv["k_cache"][pages][:, :, kvh:kvh + 1, :])
    vc = f(st.kv["v_cache"][pages][:, :, kvh:kvh + 1, :])
    table = np.arange(max(npg, 1), dtype=np.int32)[None, :]
    if npg == 0:
        kc = np.zeros((1, w.page_size, 1, w.Dh))
        vc = kc
    q = f(st.qkv["q"][b:b + 1, :, kvh * G:(kvh + 1) * G, :])
    kt = f(st.qkv["k_tree"][b:b + 1, :, kvh:kvh + 1, :])
    vt = f(st.qkv["v_tree"][b:b + 1, :, kvh:kvh + 1, :])
    vis = O.unpack_vis(st.tree.vis[b:b + 1], w.N)
    out = O.tree_verify_attention(q, kt, vt, kc, vc, table, st.ctx[b:b + 1], vis,
                                  st.tree.n_nodes[b:b + 1], scale(w), w.page_size)
    return out[0]


def check_attn(got, ref, what):
    err, rel, ok = attn_tolerance(got, ref)
    assert ok, f"{what}: max abs {err:.3e}, rel L2 {rel:.3e}"
    assert np.isfinite(got).all()


def test_attn_tiny_full():
    st = stage(S.config("tiny"))
    out, lse = run_attn(st, lse=True)
    ref, ref_lse = oracle_full(st, want_lse=True)
    check_attn(out.float().cpu().numpy().astype(np.float64), ref, "tiny")
    got_lse = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(got_lse))
    assert np.abs(got_lse[fin] - ref_lse[fin]).max() < 2e-3
    # the tiny case also runs the oracle on the fp32 draws: bf16 rounding stays small
    w = st.w
    ref32 = O.tree_verify_attention(st.qkv["q_f32"].astype(np.float64),
                                    st.qkv["k_tree_f32"].astype(np.float64),
                                    st.qkv["v_tree_f32"].astype(np.float64),
                                    st.kv["k_cache_f32"].astype(np.float64),
                                    st.kv["v_cache_f32"].astype(np.float64), st.table, st.ctx,
                                    O.unpack_vis(st.tree.vis, w.N), st.tree.n_nodes, scale(w),
                                    w.page_size)
    assert np.abs(ref32 - ref).max() < 5e-2


@pytest.mark.parametrize("ctx,page_size,Hq,Hkv,Dh,budget,K,D", [
    ([0, 1, 100, 777], 16, 8, 2, 128, 19, 3, 5),    # empty / one-token / ragged contexts, many chunks
    ([64, 4095], 64, 16, 4, 64, 40, 4, 6),          # page-aligned and ragged tail, Dh 64
    ([300], 32, 6, 6, 128, 9, 2, 4),                # MHA (G = 1)
    ([5000, 20], 64, 32, 2, 128, 8, 8, 2),          # G = 16: 144 rows
    ([1500], 16, 48, 2, 128, 23, 5, 6),             # G = 24: 576 rows, several row groups
    ([0, 70, 1000, 3], 64, 64, 8, 128, 32, 8, 8),   # 264 rows: two tensor-core tiles + 8 leftover rows
    ([129, 4000], 128, 32, 8, 128, 64, 8, 16),      # 260 rows (4 leftover), page 128, two tree tiles
    ([2000], 32, 16, 2, 128, 32, 4, 6),             # 264 rows, page 32 (two page boxes per key tile)
    ([6000, 1], 16, 8, 8, 128, 127, 4, 9),          # MHA, N = 128: 128 rows, one tile, page 16
    # tensor-core row groups of 256 rows per (request, KV head)
    ([3000, 70], 64, 64, 8, 128, 64, 8, 9),         # 520 rows: 256 + (256 + 8 leftover)
    ([2500, 5], 16, 64, 4, 128, 32, 8, 8),          # G = 16, 528 rows: 256 + 256 + 16
    ([1200], 64, 32, 4, 128, 127, 4, 10),           # 1024 rows: four groups
    ([900, 4000], 32, 16, 4, 128, 99, 6, 9),        # 400 rows: 256 + 144 (a partial second tile)
    # GQA groups that do not divide 128: tiles of whole nodes (126, 125, 120 rows)
    ([2000, 300], 64, 28, 4, 128, 32, 8, 8),        # G = 7, 231 rows: 126 + 105
    ([1500], 64, 28, 4, 128, 36, 6, 7),             # G = 7, 259 rows: 126 + 126 + 7 leftover
    ([700], 32, 24, 8, 128, 64, 8, 9),              # G = 3, 195 rows
    ([5000], 64, 96, 8, 128, 32, 8, 8),             # G = 12, 396 rows: 240 + 156
    ([1100, 10], 64, 40, 8, 128, 52, 6, 7),         # G = 5, 265 rows: 250 + 15
])
def test_attn_ragged_shapes(ctx, page_size, Hq, Hkv, Dh, budget, K, D):
    w = S.Workload(name="ragged", B=len(ctx), D=D, V=300, K=K, budget=budget, Hq=Hq, Hkv=Hkv,
                   Dh=Dh, ctx_lo=0, ctx_hi=max(ctx), page_size=page_size, paged_shuffle=True,
                   seed=77 + budget)
    st = stage(w, logits=False, ctx=ctx)
    out, lse = run_attn(st, lse=True)
    ref, ref_lse = oracle_full(st, want_lse=True)
    check_attn(out.float().cpu().numpy().astype(np.float64), ref, "ragged")
    got_lse = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(got_lse))
    assert np.abs(got_lse[fin] - ref_lse[fin]).max() < 2e-3
    pad = np.arange(w.N)[None, :] >= st.tree.n_nodes[:, None]
    assert np.all(out.float().cpu().numpy()[pad] == 0)


def test_attn_latency_full():
    st = stage(S.config("latency"), logits=False)
    out, _ = run_attn(st)
    check_attn(out.float().cpu().numpy().astype(np.float64), oracle_full(st), "latency")


@pytest.mark.parametrize("name,picks", [
    ("batched", [(0, 0), (3, 7), (7, 2), (11, 5), (15, 1)]),
    ("temperature", [(0, 3), (17, 0), (31, 7)]),
])
def test_attn_full_size_sampled(name, picks):
    """Full-size workload in the bench's launch configuration; sampled (request, KV head) slices."""
    st = stage(S.config(name), logits=False)
    s = status()
    out, _ = run_attn(st, stat=s)
    assert int(s.item()) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    G = st.w.G
    for b, kvh in picks:
        check_attn(got[b, :, kvh * G:(kvh + 1) * G, :], oracle_slice(st, b, kvh), f"{name} b={b} kv={kvh}")


def test_attn_rescale_for_some_rows_of_a_warp():
    """A context key equal to 1.5 x one row's query lifts that row's running max
    by far more than 2^8 in the middle of a chunk, while the other rows of its
    warp keep theirs: the online softmax rescales O for some rows of a warp only."""
    st = stage(S.config("batched"), logits=False)
    w = st.w
    G, ps = w.G, w.page_size
    b, kvh = 3, 2
    L = int(st.ctx[b])
    kc, vc = st.kv["k_cache"], st.kv["v_cache"]
    targets = [(2, 1), (9, 6), (20, 0), (30, 5), (32, 2)]   # (node, head in group): both tiles + leftover
    v_mark = S.f32_to_bf16_bits(np.full(w.Dh, 3.0, np.float32))
    for k, (u, g) in enumerate(targets):
        i = L * (k + 1) // 6 + 11
        page, slot = int(st.table[b, i // ps]), i % ps
        kc[page, slot, kvh, :] = S.f32_to_bf16_bits(1.5 * S.bf16_bits_to_f32(st.qkv["q"][b, u, kvh * G + g, :]))
        vc[page, slot, kvh, :] = v_mark
    s = status()
    out, _ = run_attn(st, stat=s)
    assert int(s.item()) == 0
    got = out.float().cpu().numpy().astype(np.float64)[b, :, kvh * G:(kvh + 1) * G, :]
    ref = oracle_slice(st, b, kvh)
    for u, g in targets:
        if u < int(st.tree.n_nodes[b]):
            assert ref[u, g].mean() > 2.0          # the planted key dominates that row
    check_attn(got, ref, "planted keys")


@pytest.mark.slow
def test_attn_deep_sampled():
    st = stage(S.config("deep"), logits=False)
    out, _ = run_attn(st)
    got = out.float().cpu().numpy().astype(np.float64)
    G = st.w.G
    for b, kvh in [(0, 0), (40, 5), (63, 7)]:
        check_attn(got[b, :, kvh * G:(kvh + 1) * G, :], oracle_slice(st, b, kvh), f"deep b={b}")


def test_attn_bad_page_and_ctx_flagged():
    w = S.Workload(name="bad", B=3, D=3, V=50, K=2, budget=5, Hq=4, Hkv=2, Dh=64, ctx_lo=0,
                   ctx_hi=200, page_size=16, seed=5)
    st = stage(w, logits=False, ctx=[100, 150, 60])
    st.table = st.table.copy()
    st.table[1, 2] = st.num_pages + 5            # page outside the pool
    ctx_bad = st.ctx.copy()
    ctx_bad[2] = 10 ** 6                          # beyond the page table
    tree = gpu_tree(st)
    s = status()
    out = dd.tree_verify_attn(dev(st.qkv["q"]), dev(st.qkv["k_tree"]), dev(st.qkv["v_tree"]),
                              dev(st.kv["k_cache"]), dev(st.kv["v_cache"]), dev(st.table),
                              dev(ctx_bad), tree.vis, tree.n_nodes, scale(w), dev_status=s)
    torch.cuda.synchronize()
    bits = int(s.item())
    assert bits & 1 and bits & 2
    o = out.float().cpu().numpy()
    assert np.all(o[2] == 0)
    assert np.isfinite(o).all()
    ref = oracle_slice(st, 0, 1)                  # request 0 is untouched
    check_attn(o[0, :, 2:4, :].astype(np.float64), ref, "bad-case request 0")


def test_attn_tc_bad_requests_between_good_ones():
    """Tensor-core path: requests with an invalid length or node count get zero
    rows, lse -inf and the BAD_CTX bit; the requests around them are unaffected."""
    w = S.Workload(name="badtc", B=5, D=4, V=50, K=4, budget=20, Hq=16, Hkv=2, Dh=128, ctx_lo=0,
                   ctx_hi=3000, page_size=64, paged_shuffle=True, seed=9)
    st = stage(w, logits=False, ctx=[300, 700, 0, 2999, 65])
    ctx_bad = st.ctx.copy()
    ctx_bad[1] = 10 ** 6                          # beyond the page table
    tree = gpu_tree(st)
    nn = tree.n_nodes.clone()
    nn[3] = -1                                    # invalid node count
    s = status()
    lse = torch.empty((w.B, w.N, w.Hq), dtype=torch.float32, device="cuda")
    out = dd.tree_verify_attn(dev(st.qkv["q"]), dev(st.qkv["k_tree"]), dev(st.qkv["v_tree"]),
                              dev(st.kv["k_cache"]), dev(st.kv["v_cache"]), dev(st.table),
                              dev(ctx_bad), tree.vis, nn, scale(w), lse=lse, dev_status=s)
    torch.cuda.synchronize()
    assert int(s.item()) == 2
    o = out.float().cpu().numpy()
    assert np.all(o[1] == 0) and np.all(o[3] == 0)
    assert np.all(np.isneginf(lse.cpu().numpy()[[1, 3]]))
    G = w.G
    for b in (0, 2, 4):
        for kvh in range(w.Hkv):
            check_attn(o[b, :, kvh * G:(kvh + 1) * G, :].astype(np.float64), oracle_slice(st, b, kvh),
                       f"request {b} kv {kvh}")


def test_attn_tc_many_short_requests():
    """Tensor-core path with 40 short requests (0..699 cached tokens, 264 rows:
    two tensor-core tiles and 8 leftover rows), full oracle comparison."""
    rng = np.random.default_rng(31)
    ctx = rng.integers(0, 700, size=40).tolist()
    w = S.Workload(name="short", B=40, D=6, V=300, K=6, budget=32, Hq=64, Hkv=8, Dh=128, ctx_lo=0,
                   ctx_hi=max(ctx), page_size=64, paged_shuffle=True, seed=123)
    st = stage(w, logits=False, ctx=ctx)
    out, lse = run_attn(st, lse=True)
    ref, ref_lse = oracle_full(st, want_lse=True)
    check_attn(out.float().cpu().numpy().astype(np.float64), ref, "many short")
    got_lse = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(got_lse))
    assert np.abs(got_lse[fin] - ref_lse[fin]).max() < 2e-3


@pytest.mark.parametrize("name", ["tiny", "batched"])
def test_attn_repeatable(name):
    # every sum runs in a fixed order (the leftover rows' four-warp merge and
    # the split-KV merge included), so two calls agree bit for bit
    st = stage(S.config(name), logits=False)
    a, la = run_attn(st, lse=True)
    b, lb = run_attn(st, lse=True)
    assert torch.equal(a, b)
    assert torch.equal(la, lb)


# ---------------------------------------------------------------------------
# ddtree_accept_greedy
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "latency", "batched", "deep"])
def test_accept_greedy_matches_oracle(name):
    st = stage(S.config(name), attention=False)
    tree = gpu_tree(st)
    s = status()
    g = dd.ddtree_accept_greedy(dev(st.logits), tree, st.w.D, dev_status=s)
    r = O.accept_greedy(st.logits, st.tree, st.w.D)
    torch.cuda.synchronize()
    assert int(s.item()) == 0
    assert np.array_equal(g["accept_len"].cpu().numpy(), r.accept_len)
    assert np.array_equal(g["out_tokens"].cpu().numpy(), r.out_tokens)
    assert np.array_equal(g["out_nodes"].cpu().numpy(), r.out_nodes)
    assert np.array_equal(g["bonus"].cpu().numpy(), r.bonus)


def test_accept_greedy_walk_stats():
    # accepted depth, nodes built, tokens emitted (accepted + bonus) and the
    # children compared without a match, per request
    st = stage(S.config("batched"), attention=False)
    tree = gpu_tree(st)
    ws = torch.full((st.w.B, 4), -7, dtype=torch.int32, device="cuda")
    dd.ddtree_accept_greedy(dev(st.logits), tree, st.w.D, walk_stats=ws)
    r = O.accept_greedy(st.logits, st.tree, st.w.D)
    want = np.stack([r.accept_len, st.tree.n_nodes, r.accept_len + 1, r.rejected], axis=1)
    assert np.array_equal(ws.cpu().numpy(), want)


def test_accept_greedy_planted_deep_accepts():
    """Planted logits that agree with the rank-0 chain: the walk reaches full depth."""
    lp, tok = _random_topk(3, 2, 8, 4, V=100)
    lp[..., 0] = -1e-3
    lp[..., 1:] -= 3.0
    root = np.zeros(2, np.int32)
    ref = O.build_tree(lp, tok, root, np.zeros(2, np.int32), 32)
    logits = np.random.default_rng(4).standard_normal((2, 33, 100)).astype(np.float32)
    for b in range(2):
        u = 0
        for d in range(8):
            logits[b, u, tok[b, d, 0]] += 40.0
            u = int(ref.first_child[b, u])
    tree = dd.ddtree_build(dev(lp), dev(tok), dev(root), dev(np.zeros(2, np.int32)), 32)
    g = dd.ddtree_accept_greedy(dev(logits), tree, 8)
    r = O.accept_greedy(logits, ref, 8)
    assert np.array_equal(g["out_tokens"].cpu().numpy(), r.out_tokens)
    assert np.all(r.accept_len == 8)


def test_accept_greedy_ties_nan_inf_and_odd_vocab():
    lp, tok = _random_topk(11, 4, 3, 3, V=37)
    root = np.zeros(4, np.int32)
    ref = O.build_tree(lp, tok, root, np.zeros(4, np.int32), 9)
    rng = np.random.default_rng(12)
    logits = rng.integers(-2, 3, size=(4, 10, 37)).astype(np.float32)   # many ties
    logits[1, 0, :] = np.nan
    logits[2, 0, 5:] = np.nan
    logits[2, 0, :5] = -np.inf
    logits[3, 0, 7] = np.inf
    logits[3, 0, 9] = np.inf
    logits[0, 0, 3] = -0.0
    tree = dd.ddtree_build(dev(lp), dev(tok), dev(root), dev(np.zeros(4, np.int32)), 9)
    g = dd.ddtree_accept_greedy(dev(logits), tree, 3)
    r = O.accept_greedy(logits, ref, 3)
    assert np.array_equal(g["out_tokens"].cpu().numpy(), r.out_tokens)
    assert np.array_equal(g["bonus"].cpu().numpy(), r.bonus)


# ---------------------------------------------------------------------------
# ddtree_accept_sample
# ---------------------------------------------------------------------------

def compare_sampled(g, r, margin=None, stats=None, n_nodes=None):
    """Outputs identical on every request whose scaled margin clears the bar;
    the optional margin and stats outputs checked on the same requests (the
    margin within 1e-5 times the path's largest conditioning, the fp32 bound
    of any one decision). Returns the number of requests below the bar."""
    ok = r.margin_scaled > MARGIN
    for key, ref in (("accept_len", r.accept_len), ("out_tokens", r.out_tokens),
                     ("out_nodes", r.out_nodes), ("bonus", r.bonus)):
        got = g[key].cpu().numpy()
        assert np.array_equal(got[ok], ref[ok]), key
    if margin is not None:
        m = margin.cpu().numpy().astype(np.float64)
        fin = ok & np.isfinite(r.margin)
        assert np.all(np.abs(m[fin] - r.margin[fin]) <= 1e-5 * r.cond[fin] + 1e-6), \
            np.max(np.abs(m[fin] - r.margin[fin]))
        assert np.all(np.isinf(m[ok & np.isinf(r.margin)]))
    if stats is not None:
        emitted = r.accept_len + (r.bonus >= 0)
        want = np.stack([r.accept_len, n_nodes, emitted, r.rejected], axis=1)
        assert np.array_equal(stats.cpu().numpy()[ok], want[ok])
    return int((~ok).sum())


def walk_extras(B):
    return (torch.full((B,), -1.0, dtype=torch.float32, device="cuda"),
            torch.full((B, 4), -7, dtype=torch.int32, device="cuda"))


def test_accept_sample_temperature_config():
    st = stage(S.config("temperature"), attention=False)
    temp, seed = S.sampling_params(st.w)
    tree = gpu_tree(st)
    s = status()
    m, ws = walk_extras(st.w.B)
    g = dd.ddtree_accept_sample(dev(st.logits), tree, st.w.D, dev(temp), dev(seed), 1234,
                                dev_status=s, margin_stats=m, walk_stats=ws)
    r = O.accept_sample(st.logits, st.tree, st.w.D, temp, seed, 1234)
    torch.cuda.synchronize()
    assert int(s.item()) == 0
    assert compare_sampled(g, r, m, ws, st.tree.n_nodes) <= 2


@pytest.mark.parametrize("T,offset", [(0.3, 0), (1.0, 5), (2.5, (7 << 32) + 3)])
def test_accept_sample_many_seeds(T, offset):
    B = 64
    w = S.Workload(name="s", B=B, D=5, V=257, K=4, budget=24, Hq=1, Hkv=1, Dh=64, ctx_lo=10,
                   ctx_hi=10, draft_scale=2.0, target_sigma=1.0, seed=9)
    st = stage(w, attention=False)
    temp = np.full(B, T, np.float32)
    seed = np.arange(B, dtype=np.uint64) * np.uint64(2654435761) + np.uint64(1)
    tree = gpu_tree(st)
    m, ws = walk_extras(B)
    g = dd.ddtree_accept_sample(dev(st.logits), tree, w.D, dev(temp), dev(seed), offset,
                                margin_stats=m, walk_stats=ws)
    r = O.accept_sample(st.logits, st.tree, w.D, temp, seed, offset)
    assert compare_sampled(g, r, m, ws, st.tree.n_nodes) <= 2


def test_accept_sample_low_temperature_equals_greedy():
    st = stage(S.config("latency"), attention=False)
    tree = gpu_tree(st)
    g = dd.ddtree_accept_greedy(dev(st.logits), tree, st.w.D)
    s = dd.ddtree_accept_sample(dev(st.logits), tree, st.w.D, dev(np.full(1, 1e-4, np.float32)),
                                dev(np.array([5], np.uint64)), 0)
    for key in ("accept_len", "out_tokens", "bonus"):
        assert torch.equal(g[key], s[key]), key


def test_accept_sample_bad_temperature_flagged():
    st = stage(S.config("tiny"), attention=False)
    tree = gpu_tree(st)
    s = status()
    m, ws = walk_extras(1)
    g = dd.ddtree_accept_sample(dev(st.logits), tree, st.w.D, dev(np.zeros(1, np.float32)),
                                dev(np.array([1], np.uint64)), 0, dev_status=s, margin_stats=m, walk_stats=ws)
    torch.cuda.synchronize()
    assert int(s.item()) & 8
    assert int(g["accept_len"][0]) == 0 and int(g["bonus"][0]) == -1
    assert math.isnan(float(m[0])) and ws[0].tolist() == [0, int(st.tree.n_nodes[0]), 0, 0]
