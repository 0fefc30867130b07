"""Failure detection in the tensor-core attention kernel, without a GPU fault.

Every wait inside attn_tc_kernel is bounded: a wait that runs out sets the
CTA's abort flag and DDT_DEV_TIMEOUT in the caller's status word; the CTA then
stops its other waits, drains the copies and MMAs it already issued (under
their normal limits), frees TMEM and returns. The test-only entry point
ddtree_testing_attn_stall (include/ddtree_testing.h) makes one such wait run
out: in every CTA, row tile 0's MMA-issuing warp first waits on an mbarrier
that nothing completes, with a limit of a few hundred microseconds. Nothing
faults and nothing waits without a limit; the checks are that the call
returns, the status bit is set, the outputs are defined (row tile 0's rows are
zeros, nothing is NaN), and a normal call on the same stream afterwards gives
the same result as before the stall and matches the oracle.
"""
import ctypes
import time

import numpy as np
import pytest

import ddtree_synth as S
from _stage import stage, scale, dev, attn_tolerance
import oracle as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import tree_speculative_decoding_ddtree_gb300 as dd  # noqa: E402

DDT_DEV_TIMEOUT = 32


def stall_fn():
    lib = dd.load_library()
    fn = lib.ddtree_testing_attn_stall
    P, I, F, Z, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint64
    fn.restype = I
    fn.argtypes = [P, P, P, P, P, I, I, P, I, P, P, P, I, I, I, I, I, F, P, P, P, Z, P, P, U64]
    return fn


def test_attention_wait_timeout_is_reported_and_the_next_call_is_normal():
    w = S.config("batched", B=4)
    st = stage(w, logits=False)
    q, kt, vt = dev(st.qkv["q"]), dev(st.qkv["k_tree"]), dev(st.qkv["v_tree"])
    kc, vc, table, ctx = dev(st.kv["k_cache"]), dev(st.kv["v_cache"]), dev(st.table), dev(st.ctx)
    tree = dd.ddtree_build(dev(st.topk_logp), dev(st.topk_tok), dev(st.root), ctx, w.budget)
    num_pages, page, max_pages = kc.shape[0], kc.shape[1], table.shape[1]
    need = dd.tree_verify_attn_workspace_size(w.B, w.N, w.Hq, w.Hkv, w.Dh, max_pages * page)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")

    before = dd.tree_verify_attn(q, kt, vt, kc, vc, table, ctx, tree.vis, tree.n_nodes, scale(w),
                                 workspace=ws)
    torch.cuda.synchronize()

    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.N, w.Hq), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    rc = stall_fn()(q.data_ptr(), kt.data_ptr(), vt.data_ptr(), kc.data_ptr(), vc.data_ptr(), num_pages,
                    page, table.data_ptr(), max_pages, ctx.data_ptr(), tree.vis.data_ptr(),
                    tree.n_nodes.data_ptr(), w.B, w.N, w.Hq, w.Hkv, w.Dh, scale(w), out.data_ptr(),
                    lse.data_ptr(), ws.data_ptr(), ws.numel(), status.data_ptr(), stream, 300_000)
    assert rc == 0
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) & DDT_DEV_TIMEOUT
    assert elapsed < 30.0                           # bounded: the limits are milliseconds to seconds
    o = out.float()
    assert not torch.isnan(o).any() and not torch.isnan(lse).any()
    # row tile 0 holds rows r = node * G + head < 128, i.e. nodes 0..127/G: its
    # issuing warp never ran, so those rows are zeros with lse -inf
    nodes0 = 128 // w.G
    assert torch.count_nonzero(o[:, :nodes0]) == 0
    assert bool(torch.all(torch.isneginf(lse[:, :nodes0])))

    # the context is fine: the same call again gives what it gave before, bit
    # for bit (every sum in the call, the leftover rows' four-warp merge and
    # the split-KV merge included, runs in a fixed order)
    status.zero_()
    after = dd.tree_verify_attn(q, kt, vt, kc, vc, table, ctx, tree.vis, tree.n_nodes, scale(w),
                                workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(after, before)
    # and one (request, KV head) slice still matches the oracle
    b, kvh = 1, 3
    G = w.G
    L = int(st.ctx[b])
    npg = -(-L // w.page_size)
    f = O.bf16_to_f64
    pages = st.table[b, :npg]
    ref = O.tree_verify_attention(
        f(st.qkv["q"][b:b + 1, :, kvh * G:(kvh + 1) * G]), f(st.qkv["k_tree"][b:b + 1, :, kvh:kvh + 1]),
        f(st.qkv["v_tree"][b:b + 1, :, kvh:kvh + 1]), f(st.kv["k_cache"][pages][:, :, kvh:kvh + 1]),
        f(st.kv["v_cache"][pages][:, :, kvh:kvh + 1]), np.arange(npg, dtype=np.int32)[None], st.ctx[b:b + 1],
        O.unpack_vis(st.tree.vis[b:b + 1], w.N), st.tree.n_nodes[b:b + 1], scale(w), w.page_size)[0]
    got = after[b, :, kvh * G:(kvh + 1) * G].float().cpu().numpy().astype(np.float64)
    err, rel, ok = attn_tolerance(got, ref)
    assert ok, (err, rel)


def test_stall_entry_refuses_shapes_without_bounded_waits():
    # Dh 64 runs on the warp-MMA kernel, which has no mbarrier waits to stall
    w = S.config("tiny")
    st = stage(w, logits=False)
    q, kt, vt = dev(st.qkv["q"]), dev(st.qkv["k_tree"]), dev(st.qkv["v_tree"])
    kc, vc, table, ctx = dev(st.kv["k_cache"]), dev(st.kv["v_cache"]), dev(st.table), dev(st.ctx)
    tree = dd.ddtree_build(dev(st.topk_logp), dev(st.topk_tok), dev(st.root), ctx, w.budget)
    out = torch.empty_like(q)
    rc = stall_fn()(q.data_ptr(), kt.data_ptr(), vt.data_ptr(), kc.data_ptr(), vc.data_ptr(), kc.shape[0],
                    kc.shape[1], table.data_ptr(), table.shape[1], ctx.data_ptr(), tree.vis.data_ptr(),
                    tree.n_nodes.data_ptr(), w.B, w.N, w.Hq, w.Hkv, w.Dh, scale(w), out.data_ptr(), None,
                    None, 0, None, torch.cuda.current_stream().cuda_stream, 300_000)
    assert rc == -2
