"""GPU parity of ddtree_commit_kv and of the graph-captured step (ddtree_step_*).

Bars: the cache after a commit, the new lengths, trees and walks bit-exact to
the oracle; attention within max abs 2e-2 and relative L2 1e-2; the sampled
walk inside the graph identical to the same call made alone.
"""
from dataclasses import dataclass

import numpy as np
import pytest

import ddtree_synth as S
import oracle as O
from _stage import attn_tolerance, dev, host_u32, scale

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import tree_speculative_decoding_ddtree_gb300 as dd  # noqa: E402

TREE_FIELDS = ("parent", "depth", "token", "rank", "pos", "first_child", "next_sibling", "n_nodes")
WALK_FIELDS = ("accept_len", "out_tokens", "out_nodes", "bonus")


@dataclass
class Setup:
    w: S.Workload
    lp: np.ndarray
    tok: np.ndarray
    root: np.ndarray
    ctx: np.ndarray
    tree: O.Tree
    table: np.ndarray
    qkv: dict
    kv: dict
    logits: np.ndarray
    acc: O.Accept


def setup(w):
    dl, root, _ = S.draft_inputs(w)
    ctx = S.context_lengths(w)
    lp, tok = O.draft_topk(dl, w.K)
    tree = O.build_tree(lp, tok, root, ctx, w.budget)
    table, npg = S.paged_layout(w, ctx, room=2 * (w.D + 1))   # room for two commits
    qkv = S.qkv_tree(w)
    kv = S.kv_cache(w, npg)
    logits = S.target_logits(w, dl, tree.depth, tree.n_nodes)
    return Setup(w, lp, tok, root, ctx, tree, table, qkv, kv, logits, O.accept_greedy(logits, tree, w.D))


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def walk_dev(acc):
    return {k: dev(getattr(acc, k)) for k in WALK_FIELDS}


def status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


CASES = [("tiny", {}), ("latency", {}), ("batched", dict(ctx_lo=64, ctx_hi=900)),
         ("deep", dict(B=6, ctx_lo=100, ctx_hi=3000))]


# ---------------------------------------------------------------------------
# ddtree_commit_kv
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name,over", CASES)
def test_commit_matches_oracle(name, over):
    st = setup(S.config(name, **over))
    w = st.w
    kc, vc = dev(st.kv["k_cache"]), dev(st.kv["v_cache"])
    s = status()
    new_ctx = dd.ddtree_commit_kv(dev(st.qkv["k_tree"]), dev(st.qkv["v_tree"]), walk_dev(st.acc),
                                  dev(st.ctx), dev(st.table), kc, vc, dev_status=s)
    ref_k, ref_v, ref_ctx = O.commit_kv(st.qkv["k_tree"], st.qkv["v_tree"], st.acc.out_nodes,
                                        st.acc.accept_len, st.ctx, st.table, st.kv["k_cache"],
                                        st.kv["v_cache"], w.page_size)
    torch.cuda.synchronize()
    assert int(s.item()) == 0
    assert np.array_equal(new_ctx.cpu().numpy(), ref_ctx)
    assert np.array_equal(bits(kc), ref_k)
    assert np.array_equal(bits(vc), ref_v)


def test_commit_in_place_advances_ctx_len():
    st = setup(S.config("latency"))
    ctx = dev(st.ctx)
    kc, vc = dev(st.kv["k_cache"]), dev(st.kv["v_cache"])
    out = dd.ddtree_commit_kv(dev(st.qkv["k_tree"]), dev(st.qkv["v_tree"]), walk_dev(st.acc), ctx,
                              dev(st.table), kc, vc, new_ctx_len=ctx)
    torch.cuda.synchronize()
    assert out is ctx
    assert ctx.cpu().tolist() == (st.ctx + st.acc.accept_len + 1).tolist()


def test_commit_bad_requests_write_nothing():
    w = S.config("batched", B=5, ctx_lo=64, ctx_hi=900)
    st = setup(w)
    acc = {k: getattr(st.acc, k).copy() for k in WALK_FIELDS}
    ctx = st.ctx.copy()
    table = st.table.copy()
    num_pages = st.kv["k_cache"].shape[0]
    for b in range(1, 5):   # give every bad request a path of at least two rows
        acc["accept_len"][b] = max(int(acc["accept_len"][b]), 1)
        acc["out_nodes"][b, :2] = [0, 1]
    acc["accept_len"][1] = w.D + 1                                      # walk longer than D
    acc["out_nodes"][2, 1] = w.N                                        # row outside the tree
    t = int(ctx[3])
    table[3, t // w.page_size] = num_pages                              # page outside the pool
    ctx[4] = table.shape[1] * w.page_size - 1                           # no room left
    kc, vc = dev(st.kv["k_cache"]), dev(st.kv["v_cache"])
    s = status()
    new_ctx = dd.ddtree_commit_kv(dev(st.qkv["k_tree"]), dev(st.qkv["v_tree"]),
                                  {k: dev(v) for k, v in acc.items()}, dev(ctx), dev(table), kc, vc,
                                  dev_status=s)
    torch.cuda.synchronize()
    assert int(s.item()) == 4 | 1 | 2
    # the oracle commits request 0 alone
    ref_k, ref_v, _ = O.commit_kv(st.qkv["k_tree"][:1], st.qkv["v_tree"][:1], acc["out_nodes"][:1],
                                  acc["accept_len"][:1], ctx[:1], table[:1], st.kv["k_cache"],
                                  st.kv["v_cache"], w.page_size)
    assert np.array_equal(bits(kc), ref_k) and np.array_equal(bits(vc), ref_v)
    got = new_ctx.cpu().numpy()
    assert got[0] == ctx[0] + acc["accept_len"][0] + 1
    assert got[1:].tolist() == ctx[1:].tolist()


# ---------------------------------------------------------------------------
# the graph-captured step
# ---------------------------------------------------------------------------

def make_step(st, walk="greedy", **kw):
    t = dict(topk_logp=dev(st.lp), topk_tok=dev(st.tok), root_tok=dev(st.root),
             ctx_len=dev(st.ctx), q=dev(st.qkv["q"]),
             k_tree=dev(st.qkv["k_tree"]), v_tree=dev(st.qkv["v_tree"]),
             k_cache=dev(st.kv["k_cache"]), v_cache=dev(st.kv["v_cache"]), page_table=dev(st.table),
             logits=dev(st.logits))
    step = dd.VerifyStep(budget=st.w.budget, scale=scale(st.w), walk=walk, **t, **kw)
    return step, t


def oracle_attention(st, ctx, k_cache, v_cache, tree):
    f = O.bf16_to_f64
    return O.tree_verify_attention(f(st.qkv["q"]), f(st.qkv["k_tree"]), f(st.qkv["v_tree"]),
                                   f(k_cache), f(v_cache), st.table, ctx,
                                   O.unpack_vis(tree.vis, st.w.N), tree.n_nodes, scale(st.w),
                                   st.w.page_size)


def assert_step_matches(step, t, st, tree, acc, ctx_before, k_before, v_before, s):
    torch.cuda.synchronize()
    assert int(s.item()) == 0
    for name in TREE_FIELDS:
        assert np.array_equal(getattr(step.tree, name).cpu().numpy(), getattr(tree, name)), name
    assert np.array_equal(host_u32(step.tree.vis), tree.vis)
    ref = oracle_attention(st, ctx_before, k_before, v_before, tree)
    err, rel, ok = attn_tolerance(step.attn_out.float().cpu().numpy().astype(np.float64), ref)
    assert ok, (err, rel)
    for k in WALK_FIELDS:
        assert np.array_equal(step.accept[k].cpu().numpy(), getattr(acc, k)), k
    ref_k, ref_v, ref_ctx = O.commit_kv(st.qkv["k_tree"], st.qkv["v_tree"], acc.out_nodes,
                                        acc.accept_len, ctx_before, st.table, k_before, v_before,
                                        st.w.page_size)
    assert np.array_equal(t["ctx_len"].cpu().numpy(), ref_ctx)
    assert np.array_equal(bits(t["k_cache"]), ref_k) and np.array_equal(bits(t["v_cache"]), ref_v)
    return ref_k, ref_v, ref_ctx


@pytest.mark.parametrize("name,over", CASES[:3])
def test_step_graph_matches_oracle_over_two_steps(name, over):
    st = setup(S.config(name, **over))
    s = status()
    step, t = make_step(st, dev_status=s)
    step.launch()
    k1, v1, ctx1 = assert_step_matches(step, t, st, st.tree, st.acc, st.ctx, st.kv["k_cache"],
                                       st.kv["v_cache"], s)
    # the second launch decodes over the committed context (same tree inputs)
    step.launch()
    tree2 = O.build_tree(st.lp, st.tok, st.root, ctx1, st.w.budget)
    acc2 = O.accept_greedy(st.logits, tree2, st.w.D)
    assert_step_matches(step, t, st, tree2, acc2, ctx1, k1, v1, s)
    step.close()


def test_step_graph_chain_is_the_linear_commit():
    # top-k 1: the tree is the D-node chain, the walk accepts a prefix of it,
    # and the commit appends verify rows 0..a in order
    w = S.config("batched", B=4, K=1, budget=8, ctx_lo=64, ctx_hi=700)
    st = setup(w)
    assert (st.tree.parent[:, 1:] == np.arange(w.D)).all()
    s = status()
    step, t = make_step(st, dev_status=s)
    step.launch()
    assert_step_matches(step, t, st, st.tree, st.acc, st.ctx, st.kv["k_cache"], st.kv["v_cache"], s)
    acc = step.accept["accept_len"].cpu().numpy()
    nodes = step.accept["out_nodes"].cpu().numpy()
    for b in range(w.B):
        assert nodes[b, :acc[b] + 1].tolist() == list(range(acc[b] + 1))
    step.close()


def test_step_graph_sampled_walk_equals_the_calls_alone():
    w = S.config("batched", ctx_lo=64, ctx_hi=900)
    st = setup(w)
    temp = dev(np.full(w.B, 0.7, np.float32))
    seed = dev((np.arange(w.B, dtype=np.uint64) * 7 + 3).view(np.int64))
    s = status()
    step_ctx = torch.empty(w.B, dtype=torch.int32, device="cuda")
    step, t = make_step(st, walk="sampled", temperature=temp, seed=seed, philox_offset=9,
                        new_ctx_len=step_ctx, dev_status=s)
    step.launch()
    torch.cuda.synchronize()
    # the same calls, one by one, on fresh copies of the inputs
    kc, vc = dev(st.kv["k_cache"]), dev(st.kv["v_cache"])
    tree = dd.ddtree_build(dev(st.lp), dev(st.tok), dev(st.root), dev(st.ctx), w.budget)
    dd.tree_verify_attn(dev(st.qkv["q"]), dev(st.qkv["k_tree"]), dev(st.qkv["v_tree"]), kc, vc,
                        dev(st.table), dev(st.ctx), tree.vis, tree.n_nodes, scale(w))
    walk = dd.ddtree_accept_sample(dev(st.logits), tree, w.D, temp, seed, 9)
    new_ctx = dd.ddtree_commit_kv(dev(st.qkv["k_tree"]), dev(st.qkv["v_tree"]), walk, dev(st.ctx),
                                  dev(st.table), kc, vc)
    torch.cuda.synchronize()
    assert int(s.item()) == 0
    for k in WALK_FIELDS:
        assert torch.equal(step.accept[k], walk[k]), k
    assert torch.equal(step_ctx, new_ctx)

    assert torch.equal(t["ctx_len"], dev(st.ctx))  # not advanced in place
    assert torch.equal(t["k_cache"], kc) and torch.equal(t["v_cache"], vc)
    ref = O.accept_sample(st.logits, st.tree, w.D, np.full(w.B, 0.7, np.float32),
                          np.arange(w.B, dtype=np.uint64) * 7 + 3, 9)
    sure = ref.margin > 1e-4
    assert np.array_equal(walk["accept_len"].cpu().numpy()[sure], ref.accept_len[sure])
    step.close()
