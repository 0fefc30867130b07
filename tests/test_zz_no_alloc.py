"""The allocation-free attention entry point, for callers that cannot allocate.

Some callers (a serving engine that keeps nearly all of HBM in its own KV pool
and gives plugins no allocator; a hot loop that must not stall the device on a
cudaMalloc) cannot hand tree_verify_attn a workspace. tree_verify_attn_noalloc
takes its split-KV scratch from a fixed 64 MiB array inside the library. These
checks call it through the C ABI and compare it with tree_verify_attn, within
the attention tolerance the parity tests use, on two calls in a row; the
second call runs on different inputs so that stale scratch from the first
cannot pass unnoticed. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import ddtree_synth as S
from _stage import stage, scale, dev, attn_tolerance

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import tree_speculative_decoding_ddtree_gb300 as dd  # noqa: E402


def _inputs(st):
    return [dev(st.qkv["q"]), dev(st.qkv["k_tree"]), dev(st.qkv["v_tree"]), dev(st.kv["k_cache"]),
            dev(st.kv["v_cache"]), dev(st.table), dev(st.ctx)]


def test_noalloc_matches_tree_verify_attn_twice():
    lib = dd.load_library()
    cap = lib.tree_verify_attn_noalloc_max_scratch
    cap.restype = ctypes.c_size_t
    runs = []
    for seed in (1000, 1001):                       # latency workload: 16 KV chunks -> scratch used
        w = S.config("latency", seed=seed)
        st = stage(w, logits=False)
        need = dd.tree_verify_attn_workspace_size(w.B, w.N, w.Hq, w.Hkv, w.Dh,
                                                  st.table.shape[1] * w.page_size)
        assert 0 < need <= cap()
        q, kt, vt, kc, vc, table, ctx = _inputs(st)
        tree = dd.ddtree_build(dev(st.topk_logp), dev(st.topk_tok), dev(st.root), ctx, w.budget)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = dd.tree_verify_attn(q, kt, vt, kc, vc, table, ctx, tree.vis, tree.n_nodes, scale(w))
        lse_ref = torch.empty((w.B, w.N, w.Hq), dtype=torch.float32, device="cuda")
        dd.tree_verify_attn(q, kt, vt, kc, vc, table, ctx, tree.vis, tree.n_nodes, scale(w),
                            lse=lse_ref)
        out = torch.empty_like(q)
        lse = torch.empty_like(lse_ref)
        dd.tree_verify_attn_noalloc(q, kt, vt, kc, vc, table, ctx, tree.vis, tree.n_nodes,
                                    scale(w), out, lse=lse, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = out.float().cpu().numpy().astype(np.float64)
        want = ref.float().cpu().numpy().astype(np.float64)
        err, rel, ok = attn_tolerance(got, want)
        assert ok, f"max abs {err}, rel L2 {rel}"
        assert torch.allclose(lse, lse_ref, atol=2e-3, rtol=0)
        runs.append(got)
    assert not np.array_equal(runs[0], runs[1])


def test_noalloc_rejects_sizes_beyond_its_array():
    # Hq/Hkv = 6 does not divide 128, so the warp-MMA kernel takes the call:
    # 96 nodes x 6 heads = 576 rows (two row groups of 288) over up to 256k
    # tokens of context need more split-KV scratch than the array holds. The
    # need is checked with the library's own workspace_size first. Every
    # pointer is NULL: the entry point must return DDT_ESCRATCH on the host
    # before anything is launched, and if that check were ever lost the
    # attention call behind it would refuse the NULL pointers with DDT_EINVAL,
    # again on the host, so no kernel can be handed a bad address.
    lib = dd.load_library()
    B, N, Hq, Hkv, Dh, page, max_pages = 2, 96, 48, 8, 128, 64, 4096
    cap = lib.tree_verify_attn_noalloc_max_scratch
    cap.restype = ctypes.c_size_t
    need = lib.tree_verify_attn_workspace_size(B, N, Hq, Hkv, Dh, page * max_pages)
    assert need > cap(), "these sizes no longer exceed the scratch array; pick larger ones"
    fn = lib.tree_verify_attn_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.restype = I
    fn.argtypes = [P, P, P, P, P, I, I, P, I, P, P, P, I, I, I, I, I, F, P, P, P, P]
    null = None
    st = fn(null, null, null, null, null, 16 * max_pages, page, null, max_pages, null, null, null,
            B, N, Hq, Hkv, Dh, 0.1, null, null, null, null)
    assert st == -7
    assert b"scratch" in lib.ddtree_status_string(-7)
