"""GPU parity of the tensor-parallel split of one request (by KV head).

Attention: each rank's tree_verify_attn on its own KV heads (and their query
heads) gives that rank's columns of the unsplit result; checked by running
the slices one after another on this GPU against the oracle.

Walks: the ddtree_shard_walk_* kernels with the vocabulary cut into W slices.
One GPU stands in for the W ranks: each level runs the partial kernel on
every slice and stacks the records, which is exactly what the all-gather of
a W-rank process group returns; then the merge-and-step kernels. The greedy
walk must equal ddtree_accept_greedy (and the oracle) bit for bit; the
sampled walk the oracle on every request whose scaled decision margin clears
1e-4, with at most two below it.
"""
import numpy as np
import pytest

import ddtree_synth as S
import oracle as O
from _stage import stage, scale, dev, attn_tolerance

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import tree_speculative_decoding_ddtree_gb300 as dd  # noqa: E402
from tree_speculative_decoding_ddtree_gb300 import sharded  # noqa: E402


def emulated_walk(logits, tree, D, world, temperature=None, seed=None, offset=0, status=None):
    """shard_walk's level loop with the all-gather replaced by stacking the W slices' records."""
    B, N, V = logits.shape
    ops = sharded.CudaShardOps()
    slices = [sharded.vocab_slice(V, world, r) for r in range(world)]
    shards = [logits[:, :, v0:v0 + vs].contiguous() for v0, vs in slices]
    i32 = dict(dtype=torch.int32, device="cuda")
    out = dict(accept_len=torch.empty(B, **i32), out_tokens=torch.empty((B, D + 1), **i32),
               out_nodes=torch.empty((B, D + 1), **i32), bonus=torch.empty(B, **i32))
    state = torch.empty((B, 4), **i32)
    ops.begin(state, out, D)
    for _ in range(D + 1):
        recs = torch.stack([ops.partial(sh, v0, V, tree, temperature, state) for sh, (v0, _) in zip(shards, slices)])
        ops.advance(recs, V, tree, D, temperature, seed, offset, state, out, status)
        if temperature is not None:
            keys = torch.stack([ops.bonus(sh, v0, V, tree, temperature, seed, offset, state)
                                for sh, (v0, _) in zip(shards, slices)])
            ops.finish(keys, D, state, out)
    torch.cuda.synchronize()
    out["state"] = state
    return out


@pytest.mark.parametrize("name,world", [("batched", 2), ("batched", 8), ("latency", 4), ("tiny", 3)])
def test_greedy_walk_over_vocab_slices_equals_the_unsplit_walk(name, world):
    st = stage(S.config(name), attention=False)
    w = st.w
    tree = dd.ddtree_build(dev(st.topk_logp), dev(st.topk_tok), dev(st.root), dev(st.ctx), w.budget)
    logits = dev(st.logits)
    s = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = emulated_walk(logits, tree, w.D, world, status=s)
    full = dd.ddtree_accept_greedy(logits, tree, w.D)
    ref = O.accept_greedy(st.logits, st.tree, w.D)
    assert int(s.item()) == 0
    for k in ("accept_len", "out_tokens", "out_nodes", "bonus"):
        assert torch.equal(got[k], full[k]), k
        assert np.array_equal(got[k].cpu().numpy(), getattr(ref, k)), k
    assert np.array_equal(got["state"][:, 3].cpu().numpy(), ref.rejected)


@pytest.mark.parametrize("name,world,T", [("temperature", 4, 0.7), ("batched", 2, 1.0), ("batched", 8, 0.4)])
def test_sampled_walk_over_vocab_slices_matches_the_oracle(name, world, T):
    st = stage(S.config(name), attention=False)
    w = st.w
    temp = np.full(w.B, T, np.float32)
    seed = np.arange(w.B, dtype=np.uint64) * 104729 + 3
    tree = dd.ddtree_build(dev(st.topk_logp), dev(st.topk_tok), dev(st.root), dev(st.ctx), w.budget)
    got = emulated_walk(dev(st.logits), tree, w.D, world, dev(temp), dev(seed), 77)
    ref = O.accept_sample(st.logits, st.tree, w.D, temp, seed, 77)
    sure = ref.margin_scaled > 1e-4
    assert int((~sure).sum()) <= 2
    for k in ("accept_len", "out_tokens", "out_nodes", "bonus"):
        assert np.array_equal(got[k].cpu().numpy()[sure], getattr(ref, k)[sure]), k
    assert np.array_equal(got["state"][:, 3].cpu().numpy()[sure], ref.rejected[sure])


def test_one_rank_host_loop_equals_the_unsplit_walks():
    # shard_walk itself, world 1 (LocalComm): one slice holding the whole vocabulary
    st = stage(S.config("batched"), attention=False)
    w = st.w
    tree = dd.ddtree_build(dev(st.topk_logp), dev(st.topk_tok), dev(st.root), dev(st.ctx), w.budget)
    logits = dev(st.logits)
    got = sharded.shard_walk(logits, 0, w.V, tree, w.D)
    full = dd.ddtree_accept_greedy(logits, tree, w.D)
    for k in ("accept_len", "out_tokens", "out_nodes", "bonus"):
        assert torch.equal(got[k], full[k]), k
    temp = np.full(w.B, 0.7, np.float32)
    seed = np.arange(w.B, dtype=np.uint64) + 9
    got = sharded.shard_walk(logits, 0, w.V, tree, w.D, temperature=dev(temp), seed=dev(seed), philox_offset=5)
    ref = O.accept_sample(st.logits, st.tree, w.D, temp, seed, 5)
    sure = ref.margin_scaled > 1e-4
    for k in ("accept_len", "out_tokens", "bonus"):
        assert np.array_equal(got[k].cpu().numpy()[sure], getattr(ref, k)[sure]), k


@pytest.mark.parametrize("world", [2, 4])
def test_attention_split_by_kv_head(world):
    st = stage(S.config("batched", B=4))
    w = st.w
    tree = dd.ddtree_build(dev(st.topk_logp), dev(st.topk_tok), dev(st.root), dev(st.ctx), w.budget)
    q, kt, vt = dev(st.qkv["q"]), dev(st.qkv["k_tree"]), dev(st.qkv["v_tree"])
    kc, vc = dev(st.kv["k_cache"]), dev(st.kv["v_cache"])
    table, ctx = dev(st.table), dev(st.ctx)
    full = dd.tree_verify_attn(q, kt, vt, kc, vc, table, ctx, tree.vis, tree.n_nodes, scale(w))
    parts = []
    for r in range(world):
        q0, nq, k0, nk = sharded.kv_head_slice(w.Hq, w.Hkv, world, r)
        parts.append(dd.tree_verify_attn(q[:, :, q0:q0 + nq].contiguous(), kt[:, :, k0:k0 + nk].contiguous(),
                                         vt[:, :, k0:k0 + nk].contiguous(), kc[:, :, k0:k0 + nk].contiguous(),
                                         vc[:, :, k0:k0 + nk].contiguous(), table, ctx, tree.vis, tree.n_nodes,
                                         scale(w)))
    split = torch.cat(parts, dim=2).float().cpu().numpy().astype(np.float64)
    err, rel, ok = attn_tolerance(split, full.float().cpu().numpy().astype(np.float64))
    assert ok, (err, rel)
    # one (request, KV head) slice against the oracle
    b, kvh = 2, w.Hkv - 1
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
    err, rel, ok = attn_tolerance(split[b, :, kvh * G:(kvh + 1) * G], ref)
    assert ok, (err, rel)
