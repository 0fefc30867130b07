"""Benchmark of the DDTree tree-verify step on GB300.

One step = the whole hot path over one batch: ddtree_build -> tree_verify_attn
-> the greedy and the temperature walk (the sampled walk runs on the same tree
at T = 0.7, as a server would for the temperature requests of a batch; both
walks run in one launch, ddtree_accept_greedy_sample, whose outputs equal the
separate ddtree_accept_greedy and ddtree_accept_sample calls; those two are
timed on their own as well).
The step's input, the per-depth top-k, is made once by ddtree_draft_topk
from the draft logits; that call, the draft-ratio walk
(ddtree_accept_sample_ratio), ddtree_commit_kv and the library's own step
graph (build, attention, greedy walk, commit: ddtree_step_*) are timed on
their own (`per_call_us`).

The default workload is the batched serving case: 16 requests with contexts
uniform in [1024, 16384] tokens (paged, page 64, shuffled pages), 64 query /
8 KV heads, head dim 128, budget 32 (33 verify rows), top-k cap 8, depth 8,
vocab 32000. Inputs are seeded synthetic data (ddtree_synth).

Prints one JSON line. `value` is tree-verify steps/s with inputs resident in
HBM; `e2e` is the same through the public API with host (pinned) buffers and
the copies inside the timed region, pipelined as a serving loop would (each
step's inputs copied in while the previous step computes, results read back
on a third stream); `roofline` reports tree_verify_attn's
achieved algorithmic HBM bandwidth against the measured copy peak.

`--impl reference` times the fp64 CPU oracle on a bounded sample instead.
Under torchrun each rank runs its own batch (replicas; weak scaling).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree-verify steps/s & attn HBM GB/s (% roofline), batch16 ctx8k budget32"
# DRAM traffic of one attn_tc_kernel launch on the batched workload:
# dram__bytes_read.sum + dram__bytes_write.sum from an ncu capture (a metric
# list, one launch) of `bench.py --steps 5 --warmup 3 --no-cpu-baseline
# --e2e-steps 3`, on the current kernel (profiles/attn_tc_batched16_ctx8k.md).
ATTN_TC_TRAFFIC_BYTES = 533692672 + 25800448
L2_FLUSH_BELOW = 256e6   # a paged KV cache smaller than this is timed with L2 flushed
WORKLOAD_DESC = ("batched serving: 16 requests, ctx ~U[1024,16384] paged (page 64, shuffled), "
                 "Hq 64 / Hkv 8 / Dh 128 bf16, budget 32 (N=33), top-k 8, depth 8, vocab 32000")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="batched")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-slices", type=int, default=4)
    ap.add_argument("--clocks-dir", default="",
                    help="folder for the raw nvidia-smi clock samples (default: the system temp folder)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ---------------------------------------------------------------------------
# workload (host side, numpy)
# ---------------------------------------------------------------------------

def make_host_inputs(w):
    import numpy as np
    import ddtree_synth as S
    dl, root, _ = S.draft_inputs(w)
    ctx = S.context_lengths(w)
    table, npg = S.paged_layout(w, ctx, room=w.D + 1)   # pages for the commit to write into
    qkv = S.qkv_tree(w)
    kv = S.kv_cache(w, npg)
    import dataclasses
    temp, seed = S.sampling_params(dataclasses.replace(w, temperature=0.7) if w.temperature == 0 else w)
    return dict(draft_logits=dl, root=root, ctx=ctx, table=table, num_pages=npg, qkv=qkv, kv=kv,
                temperature=temp, seed=seed)


def algorithmic_attn_bytes(w, ctx):
    """Bytes an ideal tree_verify_attn moves: context K+V read once, Q, O, tree K/V,
    page-table entries, masks and per-request scalars."""
    ctx_kv = sum(int(L) for L in ctx) * w.Hkv * w.Dh * 2 * 2
    q_o = 2 * w.B * w.N * w.Hq * w.Dh * 2
    tree_kv = 2 * w.B * w.N * w.Hkv * w.Dh * 2
    pages = sum(-(-int(L) // w.page_size) for L in ctx) * 4
    masks = w.B * w.N * ((w.N + 31) // 32) * 4 + 2 * w.B * 4
    return ctx_kv + q_o + tree_kv + pages + masks


def algorithmic_attn_flops(w, ctx, depth_sum):
    """4*N*Hq*Dh per context key (QK^T and PV), plus the visible tree pairs."""
    ctx_f = sum(4 * w.N * w.Hq * w.Dh * int(L) for L in ctx)
    tree_f = 4 * w.Hq * w.Dh * depth_sum
    return ctx_f + tree_f


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, out_dir: str = ""):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(out_dir or tempfile.gettempdir(), f"clocks_rank{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm.sort()
        loaded = [x for x in sm if x >= 0.5 * sm[-1]] or sm
        return {"sm_mhz": loaded[len(loaded) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU baseline and reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------

# One full oracle step over the whole batch: the tree build of every request,
# the attention of every (request, KV head) slice (all its query heads, over
# its whole context plus its tree rows) and both walks of every request. The
# slices and the requests are spread over a pool of worker processes (one per
# host core; each worker single-threaded), forked after the inputs are made:
# this process never touches a GPU. `reps` steps are timed one by one.
ORACLE_POOL_SNIPPET = r"""
import dataclasses, json, math, multiprocessing as mp, os, platform, sys, time
sys.path.insert(0, {root!r})
import numpy as np
import ddtree_synth as S
import oracle as O
w = S.config({name!r})
dl, root, _ = S.draft_inputs(w)
ctx = S.context_lengths(w)
table, npg = S.paged_layout(w, ctx)
qkv = S.qkv_tree(w)
kv = S.kv_cache(w, npg)
lp, tok = O.draft_topk(dl, w.K)
tree0 = O.build_tree(lp, tok, root, ctx, w.budget)
logits = S.target_logits(w, dl, tree0.depth, tree0.n_nodes)
temp, seed = S.sampling_params(dataclasses.replace(w, temperature=0.7))
vis0 = O.unpack_vis(tree0.vis, w.N)
f = O.bf16_to_f64
G = w.G

def attn_slice(bk):
    b, kvh = bk
    L = int(ctx[b])
    npb = -(-L // w.page_size)
    pages = table[b, :max(npb, 1)]
    O.tree_verify_attention(f(qkv["q"][b:b+1, :, kvh*G:(kvh+1)*G]), f(qkv["k_tree"][b:b+1, :, kvh:kvh+1]),
                            f(qkv["v_tree"][b:b+1, :, kvh:kvh+1]), f(kv["k_cache"][pages][:, :, kvh:kvh+1, :]),
                            f(kv["v_cache"][pages][:, :, kvh:kvh+1, :]), np.arange(max(npb, 1), dtype=np.int32)[None],
                            ctx[b:b+1], vis0[b:b+1], tree0.n_nodes[b:b+1], 1 / math.sqrt(w.Dh), w.page_size)
    return 0

def walks(b):
    tr = O.build_tree(lp[b:b+1], tok[b:b+1], root[b:b+1], ctx[b:b+1], w.budget)
    O.accept_greedy(logits[b:b+1], tr, w.D)
    O.accept_sample(logits[b:b+1], tr, w.D, temp[b:b+1], seed[b:b+1], 0)
    return 0

def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
        out = os.popen("lscpu 2>/dev/null").read()
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()

if __name__ == "__main__":
    cores = {cores} or (os.cpu_count() or 1)
    tasks = [(b, k) for b in range(w.B) for k in range(w.Hkv)]
    tasks.sort(key=lambda t: -int(ctx[t[0]]))          # longest slices first
    steps = []
    with mp.get_context("fork").Pool(cores) as pool:
        pool.map(walks, range(min(cores, w.B)))        # workers started and warmed, untimed
        for rep in range({reps}):
            t0 = time.perf_counter()
            r1 = pool.map_async(attn_slice, tasks, chunksize=1)
            r2 = pool.map_async(walks, range(w.B), chunksize=1)
            r1.get(); r2.get()
            steps.append(time.perf_counter() - t0)
    print(json.dumps(dict(steps=steps, cores=cores, cpu_model=cpu_model(), nproc=os.cpu_count(),
                          slices=len(tasks))))
"""


def run_oracle_pool(name: str, reps: int, cores: int = 0, timeout: float = 1800):
    """Full oracle steps on a pool of host cores, in a fresh process with no GPU."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"                                    # one thread per worker process
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = ORACLE_POOL_SNIPPET.format(root=ROOT, name=name, reps=reps, cores=cores)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=timeout)
    if r.returncode != 0:
        raise RuntimeError("oracle pool failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


CPU_SNIPPET = r"""
import dataclasses, json, math, os, sys, time
sys.path.insert(0, {root!r})
import numpy as np
import ddtree_synth as S
import oracle as O
w = S.config({name!r})
n_slices, reps = {n_slices}, {reps}
dl, root, _ = S.draft_inputs(w)
ctx = S.context_lengths(w)
table, npg = S.paged_layout(w, ctx)
qkv = S.qkv_tree(w)
kv = S.kv_cache(w, npg)
lp, tok = O.draft_topk(dl, w.K)
tree0 = O.build_tree(lp, tok, root, ctx, w.budget)
logits = S.target_logits(w, dl, tree0.depth, tree0.n_nodes)
temp, seed = S.sampling_params(dataclasses.replace(w, temperature=0.7))
f = O.bf16_to_f64
G = w.G
rng = np.random.default_rng(0)
total_keys = int(ctx.sum()) * w.Hkv
out = []
for rep in range(reps):
    t0 = time.perf_counter()
    tree = O.build_tree(lp, tok, root, ctx, w.budget)
    t_build = time.perf_counter() - t0
    vis = O.unpack_vis(tree.vis, w.N)
    t_attn, keys_done = 0.0, 0
    for _ in range(n_slices):
        b, kvh = int(rng.integers(w.B)), int(rng.integers(w.Hkv))
        L = int(ctx[b]); npb = -(-L // w.page_size); pages = table[b, :npb]
        t0 = time.perf_counter()
        kc = f(kv["k_cache"][pages][:, :, kvh:kvh + 1, :]); vc = f(kv["v_cache"][pages][:, :, kvh:kvh + 1, :])
        O.tree_verify_attention(f(qkv["q"][b:b+1, :, kvh*G:(kvh+1)*G]), f(qkv["k_tree"][b:b+1, :, kvh:kvh+1]),
                                f(qkv["v_tree"][b:b+1, :, kvh:kvh+1]), kc, vc,
                                np.arange(max(npb, 1), dtype=np.int32)[None], ctx[b:b+1], vis[b:b+1],
                                tree.n_nodes[b:b+1], 1 / math.sqrt(w.Dh), w.page_size)
        t_attn += time.perf_counter() - t0
        keys_done += L
    t0 = time.perf_counter()
    O.accept_greedy(logits, tree, w.D)
    t_greedy = time.perf_counter() - t0
    t0 = time.perf_counter()
    O.accept_sample(logits, tree, w.D, temp, seed, 0)
    t_sample = time.perf_counter() - t0
    t_attn_full = t_attn * total_keys / max(keys_done, 1)
    out.append(dict(step_s=t_build + t_attn_full + t_greedy + t_sample, t_build=t_build,
                    t_attn_sample=t_attn, t_attn_full=t_attn_full, t_greedy=t_greedy,
                    t_sample=t_sample, keys_done=keys_done, total_keys=total_keys))
print(json.dumps(out))
"""


def run_cpu_oracle(name: str, n_slices: int, reps: int = 1):
    """One thread: the oracle's build and walks for the whole batch and its
    attention on a few sampled slices, scaled to the whole step by key count."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = CPU_SNIPPET.format(root=ROOT, name=name, n_slices=n_slices, reps=reps)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=3600)
    if r.returncode != 0:
        raise RuntimeError("oracle baseline failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline_obj(pool, single, n_slices):
    steps = pool["steps"]
    step_s = sum(steps) / len(steps)
    return {"value": 1.0 / step_s, "unit": "steps/s", "cores": pool["cores"], "kind": "oracle",
            "cpu_model": pool["cpu_model"], "nproc": pool["nproc"],
            "sample": (f"fp64 numpy oracle, {pool['cores']} worker processes (one per host core, one "
                       f"thread each): {len(steps)} full steps of the whole batch (build, attention of "
                       f"all {pool['slices']} (request, KV head) slices over their whole contexts, "
                       f"greedy and sampled walks), each timed"),
            "single_thread": {
                "value": 1.0 / single["step_s"], "unit": "steps/s", "cores": 1,
                "sample": (f"1 thread: full build + greedy and sampled accept for all requests, attention "
                           f"on {n_slices} sampled (request, KV head) slices ({single['keys_done']} of "
                           f"{single['total_keys']} context key-heads), scaled to the whole step by key "
                           f"count")}}


def mean_context(w):
    """The workload's mean context length in tokens (its seeded lengths), the
    `seq_len` both arms report."""
    import ddtree_synth as S
    return int(S.context_lengths(w).sum()) // w.B


def rank_workload(name, rank, world):
    """The batch rank `rank` runs: the named workload, its seed offset by the
    rank when several ranks run (replicas: each GPU its own batch, no exchange)."""
    import ddtree_synth as S
    base = S.config(name)
    return S.config(name, seed=base.seed + 7919 * rank) if world > 1 else base


def max_over_ranks(x, world, device=None):
    """The largest of the ranks' values of x (an elapsed time): all-reduce MAX
    over the process group; x itself on one rank."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, units_per_rank, seconds):
    """Units per second of the whole job: every rank's units over the slowest rank's time."""
    return world * units_per_rank / seconds


def run_reference(args):
    rank, _, _ = dist_env()
    if rank != 0:
        return
    import ddtree_synth as S
    w = S.config(args.config)
    n_reps = max(args.warmup, 0) + args.steps
    t0 = time.perf_counter()
    res = run_oracle_pool(args.config, n_reps)
    elapsed = time.perf_counter() - t0
    per = res["steps"][max(args.warmup, 0):]
    step_s = sum(per) / len(per)
    value = 1.0 / step_s
    line = {"metric": METRIC, "value": value, "unit": "steps/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, ddtree_synth)",
            "config": {"workload": WORKLOAD_DESC if args.config == "batched" else args.config,
                       "global_batch": w.B, "seq_len": mean_context(w),
                       "parallelism": f"{res['cores']} host processes"},
            "cpu_baseline": {"value": value, "unit": "steps/s", "cores": res["cores"], "kind": "oracle",
                             "cpu_model": res["cpu_model"], "nproc": res["nproc"],
                             "sample": (f"every step is one full oracle step of the whole batch (no sample, "
                                        f"no extrapolation): build, attention of all {res['slices']} (request, "
                                        f"KV head) slices, greedy and sampled walks, over {res['cores']} worker "
                                        "processes, one thread each")},
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": elapsed}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------

def run_native(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    import ddtree_synth as S
    import tree_speculative_decoding_ddtree_gb300 as dd

    w = rank_workload(args.config, rank, world)

    # CPU baseline first, in fresh processes (rank 0, N = 1 only): two full
    # steps on all host cores, and one thread on a sample
    cpu_pool = cpu_single = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_pool = run_oracle_pool(w.name, 2)
        cpu_single = run_cpu_oracle(w.name, args.cpu_sample_slices)[0]

    h = make_host_inputs(w)
    stream = torch.cuda.current_stream(device)

    def to_dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
        if a.dtype == np.uint64:
            return torch.from_numpy(a.view(np.int64)).to(device)
        return torch.from_numpy(a).to(device)

    # per-depth top-k of the draft: the step's input, made by the library's own
    # kernel (timed per call below, outside the step)
    dl_d = to_dev(h["draft_logits"])
    topk_logp = torch.empty((w.B, w.D, w.K), dtype=torch.float32, device=device)
    topk_tok = torch.empty((w.B, w.D, w.K), dtype=torch.int32, device=device)
    dd.ddtree_draft_topk(dl_d, w.K, topk_logp, topk_tok)
    root = to_dev(h["root"])
    ctx = to_dev(h["ctx"])
    table = to_dev(h["table"])
    q = to_dev(h["qkv"]["q"])
    k_tree = to_dev(h["qkv"]["k_tree"])
    v_tree = to_dev(h["qkv"]["v_tree"])
    k_cache = to_dev(h["kv"]["k_cache"])
    v_cache = to_dev(h["kv"]["v_cache"])
    temp = to_dev(h["temperature"])
    seed = to_dev(h["seed"])
    status = torch.zeros(1, dtype=torch.int32, device=device)
    tree = dd.alloc_tree(w.B, w.N, device)
    dd.ddtree_build(topk_logp, topk_tok, root, ctx, w.budget, out=tree, dev_status=status)
    torch.cuda.synchronize()
    depth_h = tree.depth.cpu().numpy()
    nn_h = tree.n_nodes.cpu().numpy()
    logits = to_dev(S.target_logits(w, h["draft_logits"], depth_h, nn_h))
    depth_sum = int(sum(int(d) + 1 for b in range(w.B) for d in depth_h[b, :nn_h[b]]) * 1)

    out = torch.empty_like(q)
    ws_bytes = dd.tree_verify_attn_workspace_size(w.B, w.N, w.Hq, w.Hkv, w.Dh,
                                                  h["table"].shape[1] * w.page_size)
    workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device)
    go = dict(accept_len=torch.empty(w.B, dtype=torch.int32, device=device),
              out_tokens=torch.empty((w.B, w.D + 1), dtype=torch.int32, device=device),
              out_nodes=torch.empty((w.B, w.D + 1), dtype=torch.int32, device=device),
              bonus=torch.empty(w.B, dtype=torch.int32, device=device))
    so = {k: torch.empty_like(t) for k, t in go.items()}
    ro = {k: torch.empty_like(t) for k, t in go.items()}
    scale = 1.0 / math.sqrt(w.Dh)

    def step():
        dd.ddtree_build(topk_logp, topk_tok, root, ctx, w.budget, out=tree, dev_status=status)
        dd.tree_verify_attn(q, k_tree, v_tree, k_cache, v_cache, table, ctx, tree.vis, tree.n_nodes,
                            scale, out=out, workspace=workspace, dev_status=status)
        # the greedy and the temperature walk of the tree, in one launch (outputs
        # identical to the two separate calls, which the GPU does not overlap)
        dd.ddtree_accept_greedy_sample(logits, tree, w.D, temp, seed, 0, out_greedy=go, out_sample=so,
                                       dev_status=status)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    # The step is replayed as one CUDA graph (the four calls allocate nothing and
    # never synchronise, so they capture as they are); this removes the host's
    # per-call launch overhead from the device timeline.
    cap_stream = torch.cuda.Stream(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap_stream):
        with torch.cuda.graph(graph, stream=cap_stream):
            step()
    torch.cuda.synchronize()

    def graph_of(fn, reps):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap_stream):
            with torch.cuda.graph(gr, stream=cap_stream):
                for _ in range(reps):
                    fn()
        return gr

    # the commit and the whole step as the library's own graph: the new lengths
    # go to a scratch array, so every launch commits the same rows
    commit_ctx = torch.empty_like(ctx)
    native_step = dd.VerifyStep(topk_logp=topk_logp, topk_tok=topk_tok, root_tok=root, ctx_len=ctx, q=q,
                                k_tree=k_tree, v_tree=v_tree, k_cache=k_cache, v_cache=v_cache,
                                page_table=table, logits=logits, budget=w.budget, scale=scale,
                                new_ctx_len=commit_ctx, dev_status=status)
    calls = {
        "ddtree_draft_topk": lambda: dd.ddtree_draft_topk(dl_d, w.K, topk_logp, topk_tok),
        "ddtree_commit_kv": lambda: dd.ddtree_commit_kv(k_tree, v_tree, go, ctx, table, k_cache, v_cache,
                                                        new_ctx_len=commit_ctx, dev_status=status),
        "ddtree_build": lambda: dd.ddtree_build(topk_logp, topk_tok, root, ctx, w.budget, out=tree,
                                                dev_status=status),
        "tree_verify_attn": lambda: dd.tree_verify_attn(q, k_tree, v_tree, k_cache, v_cache, table, ctx,
                                                        tree.vis, tree.n_nodes, scale, out=out,
                                                        workspace=workspace, dev_status=status),
        "ddtree_accept_greedy": lambda: dd.ddtree_accept_greedy(logits, tree, w.D, out=go, dev_status=status),
        "ddtree_accept_sample": lambda: dd.ddtree_accept_sample(logits, tree, w.D, temp, seed, 0, out=so,
                                                                dev_status=status),
        "ddtree_accept_greedy_sample": lambda: dd.ddtree_accept_greedy_sample(logits, tree, w.D, temp, seed, 0,
                                                                              out_greedy=go, out_sample=so,
                                                                              dev_status=status),
        "ddtree_accept_sample_ratio": lambda: dd.ddtree_accept_sample_ratio(logits, dl_d, tree, w.D, temp, seed,
                                                                            0, out=ro, dev_status=status),
    }
    # A workload whose paged KV cache fits in L2 is timed one step at a time with
    # L2 flushed (a 256 MB write, outside the timed events) before every step;
    # larger ones run back to back (their inputs exceed L2).
    kv_bytes = h["kv"]["k_cache"].nbytes * 2
    flush_l2 = kv_bytes < L2_FLUSH_BELOW
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=device) if flush_l2 else None
    reps = 1 if flush_l2 else 10
    call_graphs = {n: graph_of(f, reps) for n, f in calls.items()}
    torch.cuda.synchronize()

    def time_replays(gr, n):
        """Milliseconds of n replays of gr on `stream`: one event pair around all of
        them, or, with L2 flushed, one pair per replay (the flush outside)."""
        if not flush_l2:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                gr.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for k, (e0, e1) in enumerate(evs):
            flush_buf.fill_(k & 255)
            e0.record(stream)
            gr.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return sum(e0.elapsed_time(e1) for e0, e1 in evs)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        graph.replay()
    torch.cuda.synchronize()
    barrier()
    launches_per_step = 3 + (1 if ws_bytes > 0 else 0)   # build, attention (+ merge), walks
    with ClockSampler(local, args.clocks_dir) as clk:
        torch.cuda.synchronize()
        barrier()
        elapsed_ms = time_replays(graph, args.steps)
        barrier()
        # tree_verify_attn alone on the same stream (roofline timing)
        attn_calls = max(20, args.steps // 10) // 10 * 10
        attn_avg_ms = time_replays(call_graphs["tree_verify_attn"], attn_calls // reps) / attn_calls
    per_call_us = {}
    for n, gr in call_graphs.items():
        gr.replay()
        torch.cuda.synchronize()
        per_call_us[n] = time_replays(gr, 50 // reps) * 1e3 / 50
    # the library's step graph, launched directly (a graph launch per step)
    for _ in range(3):
        native_step.launch()
    torch.cuda.synchronize()
    if flush_l2:
        step_ms = 0.0
        for k in range(50):
            flush_buf.fill_(k & 255)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            native_step.launch()
            e1.record(stream)
            torch.cuda.synchronize()
            step_ms += e0.elapsed_time(e1)
    else:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(50):
            native_step.launch()
        e1.record(stream)
        torch.cuda.synchronize()
        step_ms = e0.elapsed_time(e1)
    per_call_us["ddtree_step_graph"] = step_ms * 1e3 / 50
    elapsed_ms = max_over_ranks(elapsed_ms, world, device)
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    # end to end through the public API: host (pinned) inputs, copies in the timed
    # region. Like a serving loop, the steps are pipelined: two device sets of
    # inputs and outputs; step k's inputs are copied on a copy stream while step
    # k-1 computes, and its results are read back on a third stream, ordered by
    # events. Every step copies all of its inputs in and its results out.
    pin = lambda t: t.cpu().pin_memory()
    in_names = ("topk_logp", "topk_tok", "root", "ctx", "table", "q", "k_tree", "v_tree", "logits", "temp",
                "seed")
    d_in0 = dict(topk_logp=topk_logp, topk_tok=topk_tok, root=root, ctx=ctx, table=table, q=q,
                 k_tree=k_tree, v_tree=v_tree, logits=logits, temp=temp, seed=seed)
    h_in = {k: pin(d_in0[k]) for k in in_names}
    out0 = dict(out=out, **{f"g_{k}": t for k, t in go.items()}, **{f"s_{k}": t for k, t in so.items()})
    sets = [(d_in0, out0), ({k: torch.empty_like(t) for k, t in d_in0.items()},
                            {k: torch.empty_like(t) for k, t in out0.items()})]
    h_outs = [{k: torch.empty(t.shape, dtype=t.dtype).pin_memory() for k, t in out0.items()} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in out0.values())

    def step_on(di, do):
        dd.ddtree_build(di["topk_logp"], di["topk_tok"], di["root"], di["ctx"], w.budget, out=tree,
                        dev_status=status)
        dd.tree_verify_attn(di["q"], di["k_tree"], di["v_tree"], k_cache, v_cache, di["table"], di["ctx"],
                            tree.vis, tree.n_nodes, scale, out=do["out"], workspace=workspace, dev_status=status)
        dd.ddtree_accept_greedy_sample(di["logits"], tree, w.D, di["temp"], di["seed"], 0,
                                       out_greedy={k: do[f"g_{k}"] for k in go},
                                       out_sample={k: do[f"s_{k}"] for k in so}, dev_status=status)

    set_graphs = []
    for di, do in sets:
        for k in in_names:   # both sets hold valid inputs before capture
            di[k].copy_(h_in[k])
        torch.cuda.synchronize()
        set_graphs.append(graph_of(lambda di=di, do=do: step_on(di, do), 1))
    torch.cuda.synchronize()
    comp = torch.cuda.Stream(device)
    s_in = torch.cuda.Stream(device)      # one copy stream: more did not raise the host-link rate
    s_out = torch.cuda.Stream(device)
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_comp + ev_out:
        e.record(comp)

    def e2e_run(n):
        for k in range(n):
            sidx = k & 1
            di, do = sets[sidx]
            s_in.wait_event(ev_comp[sidx])        # step k-2 is done with this set's inputs
            with torch.cuda.stream(s_in):
                for name in in_names:
                    di[name].copy_(h_in[name], non_blocking=True)
            ev_in[sidx].record(s_in)
            comp.wait_event(ev_in[sidx])
            comp.wait_event(ev_out[sidx])         # step k-2's results are read out
            with torch.cuda.stream(comp):
                set_graphs[sidx].replay()
            ev_comp[sidx].record(comp)
            s_out.wait_event(ev_comp[sidx])
            with torch.cuda.stream(s_out):
                for name, t in do.items():
                    h_outs[sidx][name].copy_(t, non_blocking=True)
            ev_out[sidx].record(s_out)
        torch.cuda.synchronize()

    e2e_run(4)
    barrier()
    t0 = time.perf_counter()
    e2e_run(args.e2e_steps)
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, world, device)

    if rank == 0:
        peaks = {}
        try:
            peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        except Exception:
            pass
        hbm_peak = peaks.get("hbm_gbs", 6800.0)
        bf16_peak = peaks.get("bf16_tflops", 1900.0)
        peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
        ms_per_step = elapsed_ms / args.steps
        value = whole_job_rate(world, args.steps, elapsed_ms / 1e3)
        abytes = algorithmic_attn_bytes(w, h["ctx"])
        aflops = algorithmic_attn_flops(w, h["ctx"], depth_sum)
        achieved = abytes / (attn_avg_ms * 1e-3) / 1e9
        clocks = clk.summary()
        line = {
            "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded, ddtree_synth)",
            "config": {"workload": WORKLOAD_DESC if w.name == "batched" else w.name,
                       "global_batch": w.B * world, "seq_len": mean_context(w),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": (("L2 flushed before every timed step (256 MB write outside the events; "
                               "paged KV cache %.0f MB < 129 MB L2; the e2e leg is not flushed)" % (kv_bytes / 1e6))
                              if flush_l2 else
                              "inputs larger than L2 (paged KV cache %.0f MB > 129 MB L2)" % (kv_bytes / 1e6))},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak,
                         "traffic": ATTN_TC_TRAFFIC_BYTES if w.name == "batched" else None,
                         "traffic_source": "ncu dram read+write of one attn_tc_kernel launch, batched workload",
                         "kernel": "tree_verify_attn (split-KV main + combine launches)",
                         "peak_source": f"{peak_src} hbm_gbs",
                         "algorithmic_bytes": abytes, "attn_us": attn_avg_ms * 1e3,
                         "tensor_tflops": aflops / (attn_avg_ms * 1e-3) / 1e12,
                         "tensor_frac_of_measured_bf16": aflops / (attn_avg_ms * 1e-3) / 1e12 / bf16_peak},
            "e2e": {"value": whole_job_rate(world, args.e2e_steps, e2e_s), "unit": "steps/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "note": ("KV cache stays resident (it is the cache); every step copies all of its inputs "
                             "in from pinned host memory and its results out; steps pipelined on two "
                             "device buffer sets (inputs of step k copied while step k-1 computes, results "
                             "read back on a third stream)")},
            "per_call_us": per_call_us,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }
        if cpu_pool is not None:
            line["cpu_baseline"] = cpu_baseline_obj(cpu_pool, cpu_single, args.cpu_sample_slices)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
