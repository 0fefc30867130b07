"""GPU parity of ddtree_draft_topk against the oracle's draft top-k.

Tokens are compared bit-exactly (the ranking is decided on the fp32 logits on
both sides, ties to the lower id, NaN last). Log-probs: the oracle forms the
row's log-sum-exp in fp64. The kernel sums exp(x - max) in fp32 with the
__expf intrinsic (documented error: 2 ulp plus about 1.2 |x| ulp), at most
V / 512 + 16 terms per running sum, then combines 16 warp partials and takes
logf. Relative to the exp-sum S >= 1, the per-term errors weigh at most
(2 + 1.6 (ln V + 1)) ulp (terms with |x| > ln V + 1 are below 1/(eV) each),
the running sums and the combine (V / 512 + 37) ulp, and logf one ulp of
log S <= 16 ulp; rounding the fp64 log-prob to fp32 adds half an ulp of it.
The bar below, |got - ref| <= (V / 512 + 64) * 2^-22 + 2^-23 |ref|, is that
bound with a factor of 3 or more to spare.
"""
import numpy as np
import pytest

import ddtree_synth as S
import oracle as O
from _stage import dev, stage

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import tree_speculative_decoding_ddtree_gb300 as dd  # noqa: E402

TREE_FIELDS = ("parent", "depth", "token", "rank", "pos", "first_child", "next_sibling", "n_nodes")


def lp_bar(V, ref):
    return (V / 512 + 64) * 2.0 ** -22 + 2.0 ** -23 * np.abs(ref)


def check(x, K, x_dev=None):
    """Run the kernel on fp32 logits ``x`` [B, D, V] and compare with the oracle."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    B, D, V = x.shape
    lp, tok = dd.ddtree_draft_topk(dev(x) if x_dev is None else x_dev, K)
    torch.cuda.synchronize()
    lp, tok = lp.cpu().numpy(), tok.cpu().numpy()
    ref_lp, ref_tok = O.draft_topk(x, K)
    assert np.array_equal(tok, ref_tok)
    nan = np.isnan(ref_lp)
    assert np.array_equal(np.isnan(lp), nan)
    inf = np.isinf(ref_lp)
    assert np.array_equal(lp[inf], ref_lp[inf])
    fin = ~nan & ~inf
    err = np.abs(lp[fin].astype(np.float64) - ref_lp[fin])
    assert np.all(err <= lp_bar(V, ref_lp[fin].astype(np.float64))), float(err.max())
    return lp, tok


@pytest.mark.parametrize("name", ["tiny", "latency", "batched", "deep", "temperature"])
def test_draft_topk_matches_oracle(name):
    w = S.config(name)
    dl, _, _ = S.draft_inputs(w)
    check(dl, w.K)


@pytest.mark.parametrize("K", [1, 2, 7, 32])
@pytest.mark.parametrize("V", [32, 33, 1001, 4096, 50257])
def test_draft_topk_sizes(K, V):
    rng = np.random.default_rng(V * 100 + K)
    x = (rng.standard_normal((3, 5, V)) * 4).astype(np.float32)
    check(x, min(K, V))


@pytest.mark.parametrize("V", [1, 4, 5, 8, 31])
def test_draft_topk_vocab_below_a_warp(V):
    rng = np.random.default_rng(V)
    x = rng.standard_normal((2, 3, V)).astype(np.float32)
    check(x, V)
    check(x, 1)


def test_draft_topk_ties_go_to_the_lower_id():
    rng = np.random.default_rng(11)
    # few distinct values over a large vocabulary: every rank is decided by a tie
    x = rng.integers(-3, 4, size=(4, 6, 20000)).astype(np.float32)
    x[0, 0] = 1.0   # a whole row of one value: tokens 0..K-1
    x[0, 1, ::2] = -0.0
    x[0, 1, 1::2] = 0.0   # -0 equals +0
    _, tok = check(x, 32)
    assert tok[0, 0].tolist() == list(range(32))
    assert tok[0, 1].tolist() == list(range(32))


def test_draft_topk_ascending_and_descending_rows():
    # ascending: every element displaces the K-th best (the insert path each time)
    V = 40000
    up = np.linspace(-10, 10, V, dtype=np.float32)
    x = np.stack([up, up[::-1].copy(), np.roll(up, 12345)])[None]
    check(x, 32)
    check(x, 8)


def test_draft_topk_nan_inf_rows():
    rng = np.random.default_rng(5)
    V = 3000
    x = rng.standard_normal((1, 8, V)).astype(np.float32)
    x[0, 0, [7, 100, 2999]] = np.nan              # NaN ranks last, log-probs NaN
    x[0, 1, [3, 9]] = np.inf                       # +inf first, log-probs NaN
    x[0, 2, :] = -np.inf                           # all -inf: ranks by id, NaN log-probs
    x[0, 3, rng.choice(V, V - 5, replace=False)] = -np.inf   # five finite values
    x[0, 4, :] = np.nan                            # all NaN
    x[0, 5, ::3] = -np.inf                         # some -inf among finite
    x[0, 6, :] = np.float32(3.0e38)                # large but finite
    x[0, 7, :V // 2] = np.float32(-3.0e38)
    lp, tok = check(x, 10)
    assert tok[0, 1, :2].tolist() == [3, 9]
    assert tok[0, 2].tolist() == list(range(10))
    assert tok[0, 4].tolist() == list(range(10))
    assert np.isneginf(lp[0, 3, 5:]).all() and np.isfinite(lp[0, 3, :5]).all()


def test_draft_topk_unaligned_rows_take_the_scalar_path():
    rng = np.random.default_rng(9)
    B, D, V = 2, 4, 2048
    x = (rng.standard_normal((B, D, V)) * 3).astype(np.float32)
    buf = torch.empty(B * D * V + 1, dtype=torch.float32, device="cuda")
    buf[1:].copy_(torch.from_numpy(x.reshape(-1)))
    view = buf[1:].view(B, D, V)   # 4-byte aligned, not 16-byte aligned
    assert view.data_ptr() % 16 != 0
    check(x, 8, x_dev=view)


# Share layout of the kernel (512 threads, 4 units of 16 bytes, or of one
# float when V % 4 != 0, in flight per thread): thread (warp w, lane l) reads
# units w * 128 + l + it * 2048 + j * 32 (j < 4). The test below fills whole
# shares of six threads with large values, so that more than 1024 elements
# pass the threshold and the kernel takes its exact many-candidates path.
def _share(w, l, n_units, per_unit):
    units = [w * 128 + l + it * 2048 + j * 32 for it in range(n_units // 2048 + 1) for j in range(4)]
    units = [u for u in units if u < n_units]
    return np.array([u * per_unit + e for u in units for e in range(per_unit)])


@pytest.mark.parametrize("V", [131072, 131071])
def test_draft_topk_many_candidates_path(V):
    rng = np.random.default_rng(V)
    per_unit = 4 if V % 4 == 0 else 1
    n_units = V // per_unit
    x = rng.standard_normal((1, 2, V)).astype(np.float32)
    for d in range(2):
        for t in range(6):   # six whole shares above the threshold
            idx = _share(0, t, n_units, per_unit)
            assert len(idx) >= 200
            x[0, d, idx] = rng.uniform(600, 1000, len(idx)).astype(np.float32)
        for t in range(2):   # two more best elements set the threshold near 500
            idx = _share(1, t, n_units, per_unit)
            x[0, d, idx[5]] = np.float32(500 + t)
    x[0, 1, _share(0, 3, n_units, per_unit)] = np.float32(700.0)   # ties inside a share
    check(x, 8)
    check(x, 32)


def test_draft_topk_feeds_the_build():
    # the device top-k drives ddtree_build; the tree equals the oracle's on the
    # seeded batched workload (structure bit-exact, scores within the bar)
    w = S.config("batched")
    st = stage(w, attention=False, logits=False)
    lp, tok = dd.ddtree_draft_topk(dev(st.draft_logits), w.K)
    tree = dd.ddtree_build(lp, tok, dev(st.root), dev(st.ctx), w.budget)
    torch.cuda.synchronize()
    for name in TREE_FIELDS:
        assert np.array_equal(getattr(tree, name).cpu().numpy(), getattr(st.tree, name)), name
    sc = tree.score.cpu().numpy()
    ref = st.tree.score
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(sc), fin)
    assert np.all(np.abs(sc[fin] - ref[fin]) <= w.D * lp_bar(w.V, np.abs(ref[fin])))


def test_draft_topk_is_graph_capturable_and_deterministic():
    rng = np.random.default_rng(21)
    x = dev((rng.standard_normal((8, 8, 32000)) * 4).astype(np.float32))
    lp = torch.empty((8, 8, 8), dtype=torch.float32, device="cuda")
    tok = torch.empty((8, 8, 8), dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dd.ddtree_draft_topk(x, 8, lp, tok)
    torch.cuda.synchronize()
    first = (lp.clone(), tok.clone())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            dd.ddtree_draft_topk(x, 8, lp, tok)
    lp.zero_()
    tok.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(lp, first[0]) and torch.equal(tok, first[1])
