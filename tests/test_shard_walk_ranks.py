"""The vocabulary-parallel verify walks on two CPU ranks over gloo.

A request split over GPUs by KV head has each logits row split over the
ranks by vocabulary. ``sharded.shard_walk`` runs the walk one level at a
time: per-rank records, an all-gather over the process group, the same merge
and step on every rank. Here two gloo ranks each hold half of the vocabulary
and run the host loop with a CPU stand-in of the per-level kernels
(tests/_shard_cpu.py); both ranks must end with the unsplit oracle's
decisions: bit for bit for the greedy walk, and for the sampled walk on every
request whose scaled decision margin clears 1e-4.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

pytest.importorskip("torch")

import ddtree_synth as S
import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, os.path.join({root!r}, "tests"))
import numpy as np, torch, torch.distributed as dist
import ddtree_synth as S, oracle as O
from tree_speculative_decoding_ddtree_gb300 import sharded
from _shard_cpu import CpuShardOps
rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
dist.init_process_group("gloo", rank=rank, world_size=world)
w = S.config("tiny", B=6, V=997, K=4, budget=20, D=5, seed=31)
dl, root, _ = S.draft_inputs(w)
ctx = S.context_lengths(w)
lp, tok = O.draft_topk(dl, w.K)
tr = O.build_tree(lp, tok, root, ctx, w.budget)
logits = S.target_logits(w, dl, tr.depth, tr.n_nodes)
v0, vs = sharded.vocab_slice(w.V, world, rank)
class T: pass
tree = T()
for k in ("token", "first_child", "next_sibling", "n_nodes"):
    setattr(tree, k, torch.from_numpy(np.ascontiguousarray(getattr(tr, k))))
shard = torch.from_numpy(np.ascontiguousarray(logits[:, :, v0:v0 + vs]))
comm = sharded.TorchComm()
g = sharded.shard_walk(shard, v0, w.V, tree, w.D, comm=comm, ops=CpuShardOps())
temp = torch.full((w.B,), {T}, dtype=torch.float32)
seed = torch.from_numpy((np.arange(w.B, dtype=np.uint64) * 7919 + 5).view(np.int64))
s = sharded.shard_walk(shard, v0, w.V, tree, w.D, comm=comm, ops=CpuShardOps(), temperature=temp, seed=seed,
                       philox_offset={off})
res = dict(rank=rank, v0=v0, vs=vs, greedy={{k: v.tolist() for k, v in g.items()}},
           sample={{k: v.tolist() for k, v in s.items()}})
print(json.dumps(res))
dist.destroy_process_group()
"""


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def run_ranks(world, T=0.7, off=3):
    port = free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER.format(root=ROOT, T=T, off=off)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=300)
        assert p.returncode == 0, err[-3000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    return outs


@pytest.mark.parametrize("world,T,off", [(2, 0.7, 3), (3, 1.3, (5 << 32) + 1)])
def test_vocab_parallel_walks_equal_the_unsplit_oracle(world, T, off):
    outs = run_ranks(world, T, off)
    w = S.config("tiny", B=6, V=997, K=4, budget=20, D=5, seed=31)
    dl, root, _ = S.draft_inputs(w)
    ctx = S.context_lengths(w)
    lp, tok = O.draft_topk(dl, w.K)
    tr = O.build_tree(lp, tok, root, ctx, w.budget)
    logits = S.target_logits(w, dl, tr.depth, tr.n_nodes)
    rg = O.accept_greedy(logits, tr, w.D)
    temp = np.full(w.B, T, np.float32)
    seed = np.arange(w.B, dtype=np.uint64) * 7919 + 5
    rs = O.accept_sample(logits, tr, w.D, temp, seed, off)
    sure = rs.margin_scaled > 1e-4
    assert sure.sum() >= w.B - 1
    # the slices tile the vocabulary
    assert sorted((o["v0"], o["vs"]) for o in outs)[0][0] == 0
    assert sum(o["vs"] for o in outs) == w.V
    for o in outs:
        g, s = o["greedy"], o["sample"]
        assert g["accept_len"] == rg.accept_len.tolist()
        assert g["out_tokens"] == rg.out_tokens.tolist()
        assert g["out_nodes"] == rg.out_nodes.tolist()
        assert g["bonus"] == rg.bonus.tolist()
        assert [st[3] for st in g["state"]] == rg.rejected.tolist()
        for k, ref in (("accept_len", rs.accept_len), ("out_tokens", rs.out_tokens),
                       ("out_nodes", rs.out_nodes), ("bonus", rs.bonus)):
            got = np.array(s[k])
            assert np.array_equal(got[sure], ref[sure]), k
        assert np.array_equal(np.array([st[3] for st in s["state"]])[sure], rs.rejected[sure])
    # every rank holds the same outputs
    assert all(o["greedy"] == outs[0]["greedy"] and o["sample"] == outs[0]["sample"] for o in outs)


def test_slices():
    from tree_speculative_decoding_ddtree_gb300 import sharded
    for V, W in ((32000, 8), (997, 3), (5, 5)):
        sl = [sharded.vocab_slice(V, W, r) for r in range(W)]
        assert sl[0][0] == 0 and all(sl[i][0] + sl[i][1] == sl[i + 1][0] for i in range(W - 1))
        assert sl[-1][0] + sl[-1][1] == V and max(s for _, s in sl) - min(s for _, s in sl) <= 1
    assert sharded.kv_head_slice(64, 8, 4, 3) == (48, 16, 6, 2)
    with pytest.raises(ValueError):
        sharded.kv_head_slice(64, 8, 3, 0)
