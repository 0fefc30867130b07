"""GPU tests of ddtree_accept_greedy_sample (the greedy and the temperature
walk of one tree in one launch).

Its outputs must be bit-identical to the separate ddtree_accept_greedy and
ddtree_accept_sample calls on the same inputs (those two are checked against
the fp64 oracle in test_gpu_parity.py); one case is also checked against the
oracle directly. Cases: every workload shape, several temperatures and Philox
offsets (walks that part at the root, later, or never), the margin and
statistics outputs, a bad temperature (the temperature walk stops at once
while the greedy one runs), a child token outside the vocabulary, and a
vocabulary that is not a multiple of four (element slices).
"""
import numpy as np
import pytest

import ddtree_synth as S
import oracle as O
from _stage import stage, dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import tree_speculative_decoding_ddtree_gb300 as dd  # noqa: E402

KEYS = ("accept_len", "out_tokens", "out_nodes", "bonus")


def status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def extras(B):
    return (torch.full((B, 4), -7, dtype=torch.int32, device="cuda"),
            torch.full((B,), -1.0, dtype=torch.float32, device="cuda"),
            torch.full((B, 4), -7, dtype=torch.int32, device="cuda"))


def run_both(st, temp, seed, offset, tree=None):
    """The fused call and the two separate calls; returns both sets and the statuses."""
    w = st.w
    tree = tree if tree is not None else dd.ddtree_build(dev(st.topk_logp), dev(st.topk_tok), dev(st.root),
                                                         dev(st.ctx), w.budget)
    logits = dev(st.logits)
    t, sd = dev(temp), dev(seed)
    s_f, s_g, s_s = status(), status(), status()
    gws, sm, sws = extras(w.B)
    fg, fs = dd.ddtree_accept_greedy_sample(logits, tree, w.D, t, sd, offset, dev_status=s_f,
                                            greedy_walk_stats=gws, sample_margin_stats=sm,
                                            sample_walk_stats=sws)
    gws2, sm2, sws2 = extras(w.B)
    g = dd.ddtree_accept_greedy(logits, tree, w.D, dev_status=s_g, walk_stats=gws2)
    s = dd.ddtree_accept_sample(logits, tree, w.D, t, sd, offset, dev_status=s_s, margin_stats=sm2,
                                walk_stats=sws2)
    torch.cuda.synchronize()
    return (fg, fs, gws, sm, sws, int(s_f.item())), (g, s, gws2, sm2, sws2, int(s_g.item()) | int(s_s.item()))


def assert_identical(fused, sep):
    fg, fs, gws, sm, sws, sf = fused
    g, s, gws2, sm2, sws2, ss = sep
    for k in KEYS:
        assert torch.equal(fg[k], g[k]), "greedy " + k
        assert torch.equal(fs[k], s[k]), "sample " + k
    assert torch.equal(gws, gws2)
    assert torch.equal(sws, sws2)
    # NaN (bad temperature) compares equal to NaN here
    assert torch.equal(torch.nan_to_num(sm, nan=-99.0), torch.nan_to_num(sm2, nan=-99.0))
    assert sf == ss


@pytest.mark.parametrize("name,over", [("tiny", {}), ("latency", {}), ("batched", {}),
                                       ("temperature", {}), ("deep", dict(B=16))])
def test_fused_walks_equal_the_separate_calls(name, over):
    st = stage(S.config(name, **over), attention=False)
    temp, seed = S.sampling_params(st.w)
    if not (temp > 0).all():
        temp = np.full(st.w.B, 0.8, np.float32)
    fused, sep = run_both(st, temp, seed, 77)
    assert fused[-1] == 0
    assert_identical(fused, sep)


@pytest.mark.parametrize("T,offset", [(0.05, 0), (0.3, 3), (1.0, 5), (2.5, (7 << 32) + 3)])
def test_fused_walks_many_seeds(T, offset):
    # low T: both walks mostly take the same children; high T: they part early
    B = 64
    w = S.Workload(name="s", B=B, D=5, V=257, K=4, budget=24, Hq=1, Hkv=1, Dh=64, ctx_lo=10,
                   ctx_hi=10, draft_scale=2.0, target_sigma=1.0, seed=9)
    st = stage(w, attention=False)
    temp = np.full(B, T, np.float32)
    seed = np.arange(B, dtype=np.uint64) * np.uint64(2654435761) + np.uint64(1)
    fused, sep = run_both(st, temp, seed, offset)
    assert_identical(fused, sep)
    # the walks do part on some requests and agree on others at these settings
    fg, fs = fused[0], fused[1]
    same = (fg["out_nodes"] == fs["out_nodes"]).all(dim=1)
    if T >= 1.0:
        assert not bool(same.all())


def test_fused_walks_match_the_oracle():
    st = stage(S.config("batched"), attention=False)
    w = st.w
    temp = np.full(w.B, 0.7, np.float32)
    seed = np.arange(w.B, dtype=np.uint64) * 1009 + 17
    fused, _ = run_both(st, temp, seed, 21)
    fg, fs = fused[0], fused[1]
    rg = O.accept_greedy(st.logits, st.tree, w.D)
    for k in KEYS:
        assert np.array_equal(fg[k].cpu().numpy(), getattr(rg, k)), k
    rs = O.accept_sample(st.logits, st.tree, w.D, temp, seed, 21)
    sure = rs.margin_scaled > 1e-4
    assert int((~sure).sum()) <= 2
    for k in KEYS:
        assert np.array_equal(fs[k].cpu().numpy()[sure], getattr(rs, k)[sure]), k


def test_fused_walks_bad_temperature_and_token():
    w = S.config("tiny", B=3)
    st = stage(w, attention=False)
    temp = np.full(w.B, 0.9, np.float32)
    temp[1] = 0.0                              # the temperature walk of request 1 stops at once
    seed = np.arange(w.B, dtype=np.uint64) + 3
    tree = dd.ddtree_build(dev(st.topk_logp), dev(st.topk_tok), dev(st.root), dev(st.ctx), w.budget)
    c0 = int(st.tree.first_child[2, 0])
    tree.token[2, c0] = w.V + 5                # a child token outside the vocabulary
    fused, sep = run_both(st, temp, seed, 0, tree=tree)
    assert_identical(fused, sep)
    assert fused[-1] & 8 and fused[-1] & 16
    fg, fs = fused[0], fused[1]
    assert int(fs["accept_len"][1]) == 0 and int(fs["bonus"][1]) == -1
    assert int(fg["bonus"][1]) >= 0            # the greedy walk of that request still ran


def test_fused_walks_odd_vocabulary():
    w = S.config("batched", B=8, V=1001)
    st = stage(w, attention=False)
    temp = np.full(w.B, 1.3, np.float32)
    seed = np.arange(w.B, dtype=np.uint64) * 7 + 1
    fused, sep = run_both(st, temp, seed, 9)
    assert_identical(fused, sep)
