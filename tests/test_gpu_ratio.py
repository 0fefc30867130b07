"""GPU parity of ddtree_accept_sample_ratio (the draft-ratio temperature walk).

The kernel keeps q and p in fp32 (softmax sums over V), c and R in fp64, and
forms each residual max(q - c p, 0) with one fused multiply-add; the oracle
works in fp64. After rejections a child's threshold r(x)/p(x) =
(q(x)/p(x) - c)/R inherits the fp32 error of q and p amplified by the
decision's conditioning (1 + c)/R (the bonus's log-scores by
(q + c p)/(q - c p)); the fp32 emulation of these formulas measured at most
6e-6 per unit of conditioning. The oracle's ``margin_scaled`` divides each
margin by its conditioning, and outputs are compared on every request whose
scaled margin exceeds 1e-4 (more than ten times the error), with at most two
requests per test below it, as for the renormalising walk. The margin and
stats outputs are checked on the same requests. Structural properties
(p == q accepts every level; bad inputs) are checked on every request.
"""
import numpy as np
import pytest

import ddtree_synth as S
import oracle as O
from _stage import dev, scale

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import tree_speculative_decoding_ddtree_gb300 as dd  # noqa: E402

MARGIN = 1e-4
WALK_FIELDS = ("accept_len", "out_tokens", "out_nodes", "bonus")


def status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def staged(w, T=0.7, seed0=17):
    dl, root, _ = S.draft_inputs(w)
    ctx = S.context_lengths(w)
    lp, tok = O.draft_topk(dl, w.K)
    tree = O.build_tree(lp, tok, root, ctx, w.budget)
    logits = S.target_logits(w, dl, tree.depth, tree.n_nodes)
    temp = np.full(w.B, T, np.float32)
    seed = np.arange(w.B, dtype=np.uint64) * 1009 + seed0
    return dl, lp, tok, root, ctx, tree, logits, temp, seed


def gpu_tree(lp, tok, root, ctx, budget):
    return dd.ddtree_build(dev(lp), dev(tok), dev(root), dev(ctx), budget)


def compare(got, ref, margin=None, stats=None, n_nodes=None):
    sure = ref.margin_scaled > MARGIN
    assert int((~sure).sum()) <= 2, f"{int((~sure).sum())} of {sure.size} requests below the margin"
    for k in WALK_FIELDS:
        g = got[k].cpu().numpy()
        assert np.array_equal(g[sure], getattr(ref, k)[sure]), k
    if margin is not None:
        m = margin.cpu().numpy().astype(np.float64)
        fin = sure & np.isfinite(ref.margin)
        assert np.all(np.abs(m[fin] - ref.margin[fin]) <= 1e-5 * ref.cond[fin] + 1e-6), \
            np.max(np.abs(m[fin] - ref.margin[fin]))
    if stats is not None:
        emitted = ref.accept_len + (ref.bonus >= 0)
        want = np.stack([ref.accept_len, n_nodes, emitted, ref.rejected], axis=1)
        assert np.array_equal(stats.cpu().numpy()[sure], want[sure])
    return int(sure.sum())


def extras(B):
    return (torch.full((B,), -1.0, dtype=torch.float32, device="cuda"),
            torch.full((B, 4), -7, dtype=torch.int32, device="cuda"))


@pytest.mark.parametrize("name,over", [("tiny", {}), ("latency", {}), ("batched", {}),
                                       ("temperature", {}), ("deep", dict(B=16))])
def test_ratio_walk_matches_oracle(name, over):
    w = S.config(name, **over)
    dl, lp, tok, root, ctx, tree, logits, temp, seed = staged(w)
    t = gpu_tree(lp, tok, root, ctx, w.budget)
    s = status()
    m, ws = extras(w.B)
    got = dd.ddtree_accept_sample_ratio(dev(logits), dev(dl), t, w.D, dev(temp), dev(seed.view(np.int64)),
                                        21, dev_status=s, margin_stats=m, walk_stats=ws)
    torch.cuda.synchronize()
    assert int(s.item()) == 0
    ref = O.accept_sample_ratio(logits, dl, tree, w.D, temp, seed, 21)
    compare(got, ref, m, ws, tree.n_nodes)


@pytest.mark.parametrize("T", [0.3, 1.0, 2.5])
def test_ratio_walk_temperatures_and_rejections(T):
    # the target far from the draft: many rejections per node, several
    # residual passes; high T flattens both
    w = S.config("batched", B=24, target_sigma=4.0, K=12, budget=40)
    dl, lp, tok, root, ctx, tree, logits, temp, seed = staged(w, T=T, seed0=3)
    t = gpu_tree(lp, tok, root, ctx, w.budget)
    m, ws = extras(w.B)
    got = dd.ddtree_accept_sample_ratio(dev(logits), dev(dl), t, w.D, dev(temp), dev(seed.view(np.int64)), 0,
                                        margin_stats=m, walk_stats=ws)
    torch.cuda.synchronize()
    ref = O.accept_sample_ratio(logits, dl, tree, w.D, temp, seed, 0)
    assert ref.rejected.sum() > w.B   # many rejections per request on average
    compare(got, ref, m, ws, tree.n_nodes)


def test_ratio_walk_scalar_path():
    w = S.config("batched", B=8, V=1001)
    dl, lp, tok, root, ctx, tree, logits, temp, seed = staged(w)
    t = gpu_tree(lp, tok, root, ctx, w.budget)
    got = dd.ddtree_accept_sample_ratio(dev(logits), dev(dl), t, w.D, dev(temp), dev(seed.view(np.int64)), 5)
    torch.cuda.synchronize()
    ref = O.accept_sample_ratio(logits, dl, tree, w.D, temp, seed, 5)
    compare(got, ref)


def test_ratio_walk_chain_is_linear_speculative_sampling():
    w = S.config("batched", B=16, K=1, budget=8)
    dl, lp, tok, root, ctx, tree, logits, temp, seed = staged(w)
    assert (tree.parent[:, 1:] == np.arange(w.D)).all()
    t = gpu_tree(lp, tok, root, ctx, w.budget)
    got = dd.ddtree_accept_sample_ratio(dev(logits), dev(dl), t, w.D, dev(temp), dev(seed.view(np.int64)), 2)
    torch.cuda.synchronize()
    ref = O.accept_sample_ratio(logits, dl, tree, w.D, temp, seed, 2)
    compare(got, ref)


def test_ratio_walk_equal_distributions_accept_every_level():
    # target row of a depth-d node = draft row d: r(x)/p(x) = 1 > U at every
    # test, so the walk takes the first child at every level down to a leaf
    w = S.config("batched", B=12)
    dl, lp, tok, root, ctx, tree, _, temp, seed = staged(w)
    logits = np.zeros((w.B, w.N, w.V), np.float32)
    rng = np.random.default_rng(1)
    for b in range(w.B):
        for u in range(int(tree.n_nodes[b])):
            d = int(tree.depth[b, u])
            logits[b, u] = dl[b, d] if d < w.D else rng.standard_normal(w.V)
    t = gpu_tree(lp, tok, root, ctx, w.budget)
    got = dd.ddtree_accept_sample_ratio(dev(logits), dev(dl), t, w.D, dev(temp), dev(seed.view(np.int64)), 0)
    torch.cuda.synchronize()
    acc = got["accept_len"].cpu().numpy()
    nodes = got["out_nodes"].cpu().numpy()
    for b in range(w.B):
        path = nodes[b, 1:acc[b] + 1]
        assert all(int(tree.rank[b, c]) == 0 for c in path)
        assert int(tree.first_child[b, nodes[b, acc[b]]]) == -1


def test_ratio_walk_bad_inputs():
    w = S.config("tiny", B=3)
    dl, lp, tok, root, ctx, tree, logits, temp, seed = staged(w)
    temp[1] = 0.0                               # bad temperature: nothing emitted
    t = gpu_tree(lp, tok, root, ctx, w.budget)
    bad_tok = t.token.clone()
    c0 = int(tree.first_child[2, 0])
    bad_tok[2, c0] = w.V + 5                    # a child token outside the vocabulary: skipped
    t.token.copy_(bad_tok)
    s = status()
    got = dd.ddtree_accept_sample_ratio(dev(logits), dev(dl), t, w.D, dev(temp), dev(seed.view(np.int64)),
                                        0, dev_status=s)
    torch.cuda.synchronize()
    assert int(s.item()) & 8 and int(s.item()) & 16
    assert int(got["accept_len"][1]) == 0 and int(got["bonus"][1]) == -1
    assert int(got["out_nodes"][2, 1]) != c0


def test_step_graph_ratio_walk_equals_the_call_alone():
    w = S.config("batched", ctx_lo=64, ctx_hi=900)
    dl, lp, tok, root, ctx, tree, logits, temp, seed = staged(w)
    table, npg = S.paged_layout(w, ctx, room=w.D + 1)
    qkv = S.qkv_tree(w)
    kv = S.kv_cache(w, npg)
    s = status()
    step_ctx = torch.empty(w.B, dtype=torch.int32, device="cuda")
    tens = dict(topk_logp=dev(lp), topk_tok=dev(tok), root_tok=dev(root), ctx_len=dev(ctx), q=dev(qkv["q"]),
                k_tree=dev(qkv["k_tree"]), v_tree=dev(qkv["v_tree"]), k_cache=dev(kv["k_cache"]),
                v_cache=dev(kv["v_cache"]), page_table=dev(table), logits=dev(logits))
    step = dd.VerifyStep(budget=w.budget, scale=scale(w), walk="ratio", temperature=dev(temp),
                         seed=dev(seed.view(np.int64)), philox_offset=4, draft_logits=dev(dl),
                         new_ctx_len=step_ctx, dev_status=s, **tens)
    step.launch()
    t = gpu_tree(lp, tok, root, ctx, w.budget)
    alone = dd.ddtree_accept_sample_ratio(dev(logits), dev(dl), t, w.D, dev(temp), dev(seed.view(np.int64)), 4)
    torch.cuda.synchronize()
    assert int(s.item()) == 0
    for k in WALK_FIELDS:
        assert torch.equal(step.accept[k], alone[k]), k
    assert torch.equal(step_ctx.cpu(), torch.from_numpy(ctx + alone["accept_len"].cpu().numpy() + 1))
    step.close()
