"""The C-ABI library without a GPU: it loads, exports every declared symbol, and
rejects bad arguments on the host before launching anything."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))

from tree_speculative_decoding_ddtree_gb300 import _build  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    path = _build.build()
    import tree_speculative_decoding_ddtree_gb300 as dd
    return dd.load_library(path)


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("ddtree_draft_topk", "ddtree_commit_kv", "ddtree_accept_sample_ratio", "ddtree_build", "tree_verify_attn",
              "ddtree_accept_greedy", "ddtree_accept_sample", "ddtree_accept_greedy_sample"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -6):
        assert lib.ddtree_status_string(code)
    assert lib.ddtree_last_error() == b""


FAKE = 4096   # an aligned non-null address; host checks fail before any launch


def build_args(B=2, D=3, K=4, budget=5, null=None):
    ptrs = [FAKE] * 4 + [FAKE] * 10
    if null is not None:
        ptrs[null] = 0
    return ptrs[:4] + [B, D, K, budget] + ptrs[4:] + [0, 0]


@pytest.mark.parametrize("D,K,budget,code", [(3, 0, 5, -2), (3, 33, 5, -2), (0, 4, 5, -2),
                                             (65, 4, 5, -2), (3, 4, 128, -2), (3, 4, -1, -2)])
def test_build_rejects_shapes(lib, D, K, budget, code):
    assert lib.ddtree_build(*build_args(D=D, K=K, budget=budget)) == code


@pytest.mark.parametrize("null", range(14))
def test_build_rejects_null_pointers(lib, null):
    assert lib.ddtree_build(*build_args(null=null)) == -1


def test_build_empty_batch_is_a_noop(lib):
    assert lib.ddtree_build(*build_args(B=0, null=3)) == 0


def topk_args(B=2, D=3, V=100, K=4, null=None):
    ptrs = [FAKE] * 3
    if null is not None:
        ptrs[null] = 0
    return [ptrs[0], B, D, V, K, ptrs[1], ptrs[2], 0]


@pytest.mark.parametrize("kw,code", [
    (dict(K=0), -2), (dict(K=33), -2), (dict(V=3, K=4), -2), (dict(D=0), -2), (dict(D=65), -2),
    (dict(B=1 << 30, D=4), -2), (dict(B=-1), -1), (dict(V=0), -1),
    (dict(null=0), -1), (dict(null=1), -1), (dict(null=2), -1)])
def test_draft_topk_rejects_bad_arguments(lib, kw, code):
    assert lib.ddtree_draft_topk(*topk_args(**kw)) == code


def test_draft_topk_empty_batch_is_a_noop(lib):
    assert lib.ddtree_draft_topk(*topk_args(B=0, null=0)) == 0


def commit_args(B=2, N=9, D=8, Hkv=8, Dh=128, num_pages=10, page=64, max_pages=4, null=None,
                unaligned=None):
    ptrs = [FAKE] * 9
    if null is not None:
        ptrs[null] = 0
    if unaligned is not None:
        ptrs[unaligned] = FAKE + 4
    k_tree, v_tree, nodes, acc, kc, vc, table, ctx, new_ctx = ptrs
    return [k_tree, v_tree, nodes, acc, B, N, D, Hkv, Dh, kc, vc, num_pages, page, table, max_pages,
            ctx, new_ctx, 0, 0]


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), -1), (dict(Hkv=0), -1), (dict(Dh=0), -1), (dict(page=0), -1), (dict(max_pages=0), -1),
    (dict(num_pages=0), -1), (dict(N=0), -2), (dict(N=129), -2), (dict(D=0), -2), (dict(D=65), -2),
    (dict(Hkv=1, Dh=4), -2)] + [(dict(null=i), -1) for i in range(9)]
    + [(dict(unaligned=i), -1) for i in (0, 1, 4, 5)])
def test_commit_rejects_bad_arguments(lib, kw, code):
    assert lib.ddtree_commit_kv(*commit_args(**kw)) == code


def test_commit_empty_batch_is_a_noop(lib):
    assert lib.ddtree_commit_kv(*commit_args(B=0, null=0)) == 0


def attn_args(**kw):
    a = dict(q=FAKE, kt=FAKE, vt=FAKE, kc=FAKE, vc=FAKE, num_pages=10, page_size=64, table=FAKE,
             max_pages=256, ctx=FAKE, vis=FAKE, nn=FAKE, B=2, N=33, Hq=64, Hkv=8, Dh=128, scale=0.1,
             out=FAKE, lse=0, ws=FAKE, ws_bytes=1 << 40, status=0, stream=0)
    a.update(kw)
    return [a[k] for k in ("q", "kt", "vt", "kc", "vc", "num_pages", "page_size", "table",
                           "max_pages", "ctx", "vis", "nn", "B", "N", "Hq", "Hkv", "Dh", "scale",
                           "out", "lse", "ws", "ws_bytes", "status", "stream")]


@pytest.mark.parametrize("kw,code", [
    (dict(Dh=96), -2), (dict(Hq=60), -2), (dict(N=129), -2), (dict(N=0), -2),
    (dict(page_size=8), -2), (dict(page_size=100), -2), (dict(num_pages=0), -2),
    (dict(scale=float("nan")), -1), (dict(q=0), -1), (dict(out=0), -1), (dict(vis=0), -1),
    (dict(q=FAKE + 8), -1), (dict(ws=0), -6), (dict(ws_bytes=16), -6), (dict(ws=FAKE + 16), -6),
    (dict(B=-1), -1), (dict(B=0, q=0), 0),
])
def test_attn_rejects_bad_arguments(lib, kw, code):
    if code == -6:
        # the workspace cases rely on these sizes needing one: make sure, so that
        # a call that is not refused can never launch on the placeholder pointers
        assert lib.tree_verify_attn_workspace_size(2, 33, 64, 8, 128, 64 * 256) > 16
    assert lib.tree_verify_attn(*attn_args(**kw)) == code


def test_workspace_size(lib):
    assert lib.tree_verify_attn_workspace_size(16, 33, 64, 8, 128, 16384) > 0
    assert lib.tree_verify_attn_workspace_size(16, 33, 64, 8, 96, 16384) == 0
    # a short context needs no split and no workspace
    assert lib.tree_verify_attn_workspace_size(1, 33, 64, 8, 128, 64) == 0
    small = lib.tree_verify_attn_workspace_size(1, 33, 64, 8, 128, 4096)
    big = lib.tree_verify_attn_workspace_size(1, 33, 64, 8, 128, 32768)
    assert 0 < small <= big


def _planned_workspace(B, N, Hq, Hkv, Dh, max_ctx, sms=152):
    """The split-KV planner's workspace, restated: a three-wave target gives the
    fewest chunks per full-length context; from there up to four times as many,
    the count whose equal work items (tiles + 11 tiles of fixed cost, in whole
    waves of the SMs) plus the merge's partial traffic (written and read, in
    32 KB per SM per tile time, + 5 tiles) finish first; then the shortest
    chunk length for that count."""
    R = N * (Hq // Hkv)
    groups = -(-R // 288)
    tiles = -(-max_ctx // 64)
    units = B * Hkv * groups
    tpc = max(4, -(-units * max(tiles, 1) // (sms * 3)))
    if tiles > 0:
        nch0 = -(-tiles // tpc)
        hi = max(nch0, min(4 * nch0, tiles // 4))
        best = None
        for n in range(nch0, hi + 1):
            t = -(-tiles // n)
            if -(-tiles // t) != n:
                continue
            cost = -(-units * n // sms) * (11 + t)
            if n > 1:
                cost += -(-(2 * units * n * (R // groups) * Dh * 4) // (sms * 32768)) + 5
            if best is None or cost < best[0]:
                best = (cost, n)
        tpc = max(4, -(-tiles // best[1]))
    chunks = -(-tiles // tpc) if tiles > 0 else 1
    if chunks <= 1:
        return 0
    rows = B * Hkv * chunks * R
    return -(-(rows * Dh * 4) // 256) * 256 + -(-(rows * 8) // 256) * 256


@pytest.mark.parametrize("B,N,Hq,Hkv,Dh,max_ctx", [
    (16, 33, 64, 8, 128, 16384),   # the bench batch: four chunks of 64 tiles
    (64, 65, 32, 8, 128, 32768),   # the deep batch: two chunks of 256 tiles
    (32, 33, 64, 8, 128, 8192),
    (1, 33, 64, 8, 128, 4096),     # one request: the 4-tile floor
    (3, 17, 16, 2, 64, 100000),
    (8, 128, 48, 8, 128, 65536),   # several row groups
    (40, 9, 8, 8, 128, 2048),
])
def test_workspace_size_follows_the_chunk_model(lib, B, N, Hq, Hkv, Dh, max_ctx):
    # on a host without a usable device the planner sizes for 152 SMs, as here
    assert lib.tree_verify_attn_workspace_size(B, N, Hq, Hkv, Dh, max_ctx) == \
        _planned_workspace(B, N, Hq, Hkv, Dh, max_ctx)


def walk_args(sample=False, **kw):
    a = dict(logits=FAKE, V=100, token=FAKE, fc=FAKE, ns=FAKE, nn=FAKE, B=2, N=33, D=8,
             acc=FAKE, toks=FAKE, nodes=FAKE, bonus=FAKE, margin=0, stats=0, status=0, stream=0,
             temp=FAKE, seed=FAKE, offset=0)
    a.update(kw)
    head = [a[k] for k in ("logits", "V", "token", "fc", "ns", "nn", "B", "N", "D")]
    outs = [a[k] for k in ("acc", "toks", "nodes", "bonus")]
    tail = [a[k] for k in ("status", "stream")]
    if sample:   # the sampled walks also take the (nullable) margin output
        return head + [a["temp"], a["seed"], a["offset"]] + outs + [a["margin"], a["stats"]] + tail
    return head + outs + [a["stats"]] + tail


@pytest.mark.parametrize("kw,code", [(dict(V=0), -1), (dict(N=200), -2), (dict(D=0), -2),
                                     (dict(logits=0), -1), (dict(bonus=0), -1), (dict(B=0, logits=0), 0)])
def test_walks_reject_bad_arguments(lib, kw, code):
    assert lib.ddtree_accept_greedy(*walk_args(**kw)) == code
    assert lib.ddtree_accept_sample(*walk_args(sample=True, **kw)) == code


def ratio_args(draft=FAKE, **kw):
    a = walk_args(sample=True, **kw)
    return a[:1] + [draft] + a[1:]


@pytest.mark.parametrize("kw,code", [(dict(V=0), -1), (dict(N=200), -2), (dict(D=0), -2),
                                     (dict(D=65), -2), (dict(B=-1), -1), (dict(logits=0), -1),
                                     (dict(token=0), -1), (dict(bonus=0), -1), (dict(draft=0), -1),
                                     (dict(temp=0), -1), (dict(seed=0), -1), (dict(offset=1 << 56), -1)])
def test_ratio_walk_rejects_bad_arguments(lib, kw, code):
    assert lib.ddtree_accept_sample_ratio(*ratio_args(**kw)) == code


def test_ratio_walk_empty_batch_is_a_noop(lib):
    assert lib.ddtree_accept_sample_ratio(*ratio_args(B=0, logits=0, draft=0)) == 0


def both_args(**kw):
    a = dict(logits=FAKE, V=100, token=FAKE, fc=FAKE, ns=FAKE, nn=FAKE, B=2, N=33, D=8, temp=FAKE,
             seed=FAKE, offset=0, g_acc=FAKE, g_toks=FAKE, g_nodes=FAKE, g_bonus=FAKE, g_stats=0,
             s_acc=FAKE, s_toks=FAKE, s_nodes=FAKE, s_bonus=FAKE, s_margin=0, s_stats=0, status=0, stream=0)
    a.update(kw)
    return [a[k] for k in ("logits", "V", "token", "fc", "ns", "nn", "B", "N", "D", "temp", "seed", "offset",
                           "g_acc", "g_toks", "g_nodes", "g_bonus", "g_stats", "s_acc", "s_toks", "s_nodes",
                           "s_bonus", "s_margin", "s_stats", "status", "stream")]


@pytest.mark.parametrize("kw,code", [(dict(V=0), -1), (dict(N=200), -2), (dict(D=0), -2), (dict(D=65), -2),
                                     (dict(logits=0), -1), (dict(token=0), -1), (dict(g_bonus=0), -1),
                                     (dict(s_bonus=0), -1), (dict(g_nodes=0), -1), (dict(s_acc=0), -1),
                                     (dict(temp=0), -1), (dict(seed=0), -1), (dict(offset=1 << 56), -1),
                                     (dict(B=0, logits=0), 0)])
def test_fused_walks_reject_bad_arguments(lib, kw, code):
    # the checks of the two separate calls, on both output sets; nothing launches
    assert lib.ddtree_accept_greedy_sample(*both_args(**kw)) == code


def test_sample_rejects_missing_rng_inputs_and_large_offset(lib):
    assert lib.ddtree_accept_sample(*walk_args(sample=True, temp=0)) == -1
    assert lib.ddtree_accept_sample(*walk_args(sample=True, seed=0)) == -1
    assert lib.ddtree_accept_sample(*walk_args(sample=True, offset=1 << 56)) == -1


def test_gumbel_probe_rejects_null_before_any_cuda_call(lib):
    fn = lib.ddtree_testing_gumbel
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    assert fn(None, None, 0, None) == 0    # nothing to do
    assert fn(None, None, 4, None) == -1   # DDT_EINVAL


def test_step_args_mirror_matches_the_c_struct(lib):
    import tree_speculative_decoding_ddtree_gb300 as dd
    assert lib.ddtree_step_args_size() == ctypes.sizeof(dd.StepArgs)


def test_step_create_rejects_before_any_cuda_call(lib):
    import tree_speculative_decoding_ddtree_gb300 as dd
    a = dd.StepArgs()
    a.B, a.walk = 2, 3
    h = ctypes.c_void_p()
    assert lib.ddtree_step_create(ctypes.byref(a), ctypes.byref(h)) == -1   # walk not 0, 1, 2
    a.walk, a.B = 0, 0
    assert lib.ddtree_step_create(ctypes.byref(a), ctypes.byref(h)) == -2   # empty batch
    assert lib.ddtree_step_create(None, ctypes.byref(h)) == -1
    assert lib.ddtree_step_create(ctypes.byref(a), None) == -1
    assert h.value is None
    lib.ddtree_step_destroy(None)
    assert lib.ddtree_step_launch(None, None) == -1


def test_testing_stall_entry_checks_its_limit_on_the_host(lib):
    # NULL pointers throughout: every outcome is a host-side refusal, so no
    # kernel can be launched whatever the order of the checks
    fn = lib.ddtree_testing_attn_stall
    P, I, F, Z, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint64
    fn.restype = I
    fn.argtypes = [P, P, P, P, P, I, I, P, I, P, P, P, I, I, I, I, I, F, P, P, P, Z, P, P, U64]
    args = [None] * 5 + [16, 64, None, 4, None, None, None, 2, 33, 64, 8, 128, 0.08, None, None, None, 0,
                         None, None]
    assert "ddtree_testing_attn_stall" in declared_functions()
    assert fn(*args, 0) == -1                 # no stall asked for
    assert fn(*args, 2_000_000_000) == -1     # above one second
    assert fn(*args, 100_000) == -1           # a valid limit, but NULL pointers
