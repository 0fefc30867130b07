"""One request split over GPUs by KV head: attention slices and the
vocabulary-parallel verify walks.

"The Pivot Point: Strategic Decision-Making in Speculative Decoding
Optimization", The Strategic Decision (TP8: each request spread over the
GPUs of a node); "The Architecture of Speculative Decoding: Dissecting
DDTree's Tree-Parallel Evaluation Strategy", Section 1 step 1 (the
vocabulary-parallel head: each rank holds a slice of every logits row).

* Attention needs no exchange: rank r takes KV heads
  [r * Hkv / W, (r + 1) * Hkv / W) and their query heads (contiguous GQA
  groups) and calls ``tree_verify_attn`` on its own slices.
* The walks need the whole vocabulary at every visited node. ``shard_walk``
  runs one level at a time: this rank's partial records (C ABI
  ``ddtree_shard_walk_partial``), an all-gather of the records over the
  ranks, the identical merge and step on every rank
  (``ddtree_shard_walk_advance``), and for the sampled walk the Gumbel-max
  bonus the same way (``ddtree_shard_walk_bonus`` / ``_finish``). Every rank
  ends with the same accept outputs.

This module is host orchestration only: every reduction and decision runs in
the library's kernels (``CudaShardOps``); the collective is the caller's
process group (``TorchComm``: NCCL on GPUs, gloo on CPU) or nothing for a
single rank (``LocalComm``).
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

RECORD_WORDS = 36   # key lo, key hi, max, sum, 32 child logits (int32 bit patterns)


def vocab_slice(V: int, world: int, rank: int):
    """This rank's vocabulary slice ``(v0, Vs)``: contiguous, sizes differing by at most one."""
    if not 0 <= rank < world or V < world:
        raise ValueError("need 0 <= rank < world <= V")
    base, extra = divmod(V, world)
    v0 = rank * base + min(rank, extra)
    return v0, base + (1 if rank < extra else 0)


def kv_head_slice(Hq: int, Hkv: int, world: int, rank: int):
    """This rank's heads: ``(q0, nq, kv0, nkv)`` for KV heads split evenly (GQA groups stay whole)."""
    if Hkv % world or Hq % Hkv:
        raise ValueError("KV heads must split evenly over the ranks")
    nkv = Hkv // world
    G = Hq // Hkv
    return rank * nkv * G, nkv * G, rank * nkv, nkv


class LocalComm:
    """One rank: the all-gather of a tensor is the tensor itself, with a leading axis of 1."""
    world = 1

    def all_gather(self, t: torch.Tensor) -> torch.Tensor:
        return t.unsqueeze(0)


class TorchComm:
    """All-gather over a ``torch.distributed`` process group (NCCL for GPU
    tensors, gloo for CPU tensors), on the current stream."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)

    def all_gather(self, t: torch.Tensor) -> torch.Tensor:
        t = t.contiguous()
        out = torch.empty((self.world * t.shape[0],) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
        self.dist.all_gather_into_tensor(out, t, group=self.group)   # rank blocks, concatenated
        return out.view((self.world,) + tuple(t.shape))


class CudaShardOps:
    """The per-level kernels of the vocabulary-parallel walks (C ABI ``ddtree_shard_walk_*``)."""

    def __init__(self):
        from . import _check, _ptr, _stream, load_library
        self._check, self._ptr, self._stream = _check, _ptr, _stream
        lib = load_library()
        P, I, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
        lib.ddtree_shard_walk_begin.restype = I
        lib.ddtree_shard_walk_begin.argtypes = [I, I, P, P, P, P, P, P]
        lib.ddtree_shard_walk_partial.restype = I
        lib.ddtree_shard_walk_partial.argtypes = [P, I, I, I, P, P, P, P, I, I, P, P, P, P]
        lib.ddtree_shard_walk_advance.restype = I
        lib.ddtree_shard_walk_advance.argtypes = [P, I, I, P, P, P, P, I, I, I, P, P, U64, P, P, P, P, P, P, P]
        lib.ddtree_shard_walk_bonus.restype = I
        lib.ddtree_shard_walk_bonus.argtypes = [P, I, I, I, P, P, P, P, I, I, P, P, U64, P, P, P]
        lib.ddtree_shard_walk_finish.restype = I
        lib.ddtree_shard_walk_finish.argtypes = [P, I, I, I, P, P, P, P, P]
        self.lib = lib

    def begin(self, state, out, D, stream=None):
        B = state.shape[0]
        p = self._ptr
        self._check(self.lib.ddtree_shard_walk_begin(
            B, D, p(state, torch.int32, "state", (B, 4)), p(out["accept_len"], torch.int32, "accept_len", (B,)),
            p(out["out_tokens"], torch.int32, "out_tokens", (B, D + 1)),
            p(out["out_nodes"], torch.int32, "out_nodes", (B, D + 1)), p(out["bonus"], torch.int32, "bonus", (B,)),
            self._stream(stream)), "ddtree_shard_walk_begin")

    def _tree(self, tree, B, N):
        p = self._ptr
        return (p(tree.token, torch.int32, "token", (B, N)), p(tree.first_child, torch.int32, "first_child", (B, N)),
                p(tree.next_sibling, torch.int32, "next_sibling", (B, N)), p(tree.n_nodes, torch.int32, "n_nodes", (B,)))

    def partial(self, logits_shard, v0, V, tree, temperature, state, stream=None):
        B, N, Vs = logits_shard.shape
        rec = torch.empty((B, RECORD_WORDS), dtype=torch.int32, device=logits_shard.device)
        p = self._ptr
        self._check(self.lib.ddtree_shard_walk_partial(
            p(logits_shard, torch.float32, "logits_shard", (B, N, Vs)), Vs, v0, V, *self._tree(tree, B, N), B, N,
            p(temperature, torch.float32, "temperature", (B,)), p(state, torch.int32, "state", (B, 4)),
            p(rec, torch.int32, "record", (B, RECORD_WORDS)), self._stream(stream)), "ddtree_shard_walk_partial")
        return rec

    def advance(self, records, V, tree, D, temperature, seed, offset, state, out, dev_status=None, stream=None):
        W, B, _ = records.shape
        N = tree.token.shape[1]
        p = self._ptr
        self._check(self.lib.ddtree_shard_walk_advance(
            p(records, torch.int32, "records", (W, B, RECORD_WORDS)), W, V, *self._tree(tree, B, N), B, N, D,
            p(temperature, torch.float32, "temperature", (B,)), p(seed, torch.int64, "seed", (B,)), int(offset),
            p(state, torch.int32, "state", (B, 4)), p(out["accept_len"], torch.int32, "accept_len", (B,)),
            p(out["out_tokens"], torch.int32, "out_tokens", (B, D + 1)),
            p(out["out_nodes"], torch.int32, "out_nodes", (B, D + 1)), p(out["bonus"], torch.int32, "bonus", (B,)),
            p(dev_status, torch.int32, "dev_status", (1,)), self._stream(stream)), "ddtree_shard_walk_advance")

    def bonus(self, logits_shard, v0, V, tree, temperature, seed, offset, state, stream=None):
        B, N, Vs = logits_shard.shape
        key = torch.empty(B, dtype=torch.int64, device=logits_shard.device)
        p = self._ptr
        self._check(self.lib.ddtree_shard_walk_bonus(
            p(logits_shard, torch.float32, "logits_shard", (B, N, Vs)), Vs, v0, V, *self._tree(tree, B, N), B, N,
            p(temperature, torch.float32, "temperature", (B,)), p(seed, torch.int64, "seed", (B,)), int(offset),
            p(state, torch.int32, "state", (B, 4)), p(key, torch.int64, "key", (B,)), self._stream(stream)),
            "ddtree_shard_walk_bonus")
        return key

    def finish(self, keys, D, state, out, stream=None):
        W, B = keys.shape
        p = self._ptr
        self._check(self.lib.ddtree_shard_walk_finish(
            p(keys, torch.int64, "keys", (W, B)), W, B, D, p(state, torch.int32, "state", (B, 4)),
            p(out["accept_len"], torch.int32, "accept_len", (B,)),
            p(out["out_tokens"], torch.int32, "out_tokens", (B, D + 1)), p(out["bonus"], torch.int32, "bonus", (B,)),
            self._stream(stream)), "ddtree_shard_walk_finish")


def shard_walk(logits_shard: torch.Tensor, v0: int, V: int, tree, D: int, comm=None, ops=None,
               temperature: Optional[torch.Tensor] = None, seed: Optional[torch.Tensor] = None,
               philox_offset: int = 0, out: Optional[dict] = None, dev_status: Optional[torch.Tensor] = None):
    """The greedy (``temperature=None``) or sampled verify walk of a request
    batch whose logits rows are split over the ranks of ``comm`` by
    vocabulary: this rank holds ``logits_shard[b, u, :] = logits[b, u, v0:v0+Vs]``.
    Returns the accept outputs (identical on every rank) as a dict like
    ``ddtree_accept_greedy``'s; ``state`` (``[B, 4]``) is added to it."""
    comm = comm if comm is not None else LocalComm()
    ops = ops if ops is not None else CudaShardOps()
    B, N, Vs = logits_shard.shape
    dev = logits_shard.device
    if out is None:
        i32 = dict(dtype=torch.int32, device=dev)
        out = dict(accept_len=torch.empty(B, **i32), out_tokens=torch.empty((B, D + 1), **i32),
                   out_nodes=torch.empty((B, D + 1), **i32), bonus=torch.empty(B, **i32))
    state = torch.empty((B, 4), dtype=torch.int32, device=dev)
    ops.begin(state, out, D)
    for _ in range(D + 1):   # a walk accepts at most D nodes, one level each, then stops
        rec = ops.partial(logits_shard, v0, V, tree, temperature, state)
        ops.advance(comm.all_gather(rec), V, tree, D, temperature, seed, philox_offset, state, out, dev_status)
        if temperature is not None:
            key = ops.bonus(logits_shard, v0, V, tree, temperature, seed, philox_offset, state)
            ops.finish(comm.all_gather(key), D, state, out)
    out["state"] = state
    return out
