"""CPU stand-in for the kernels of the vocabulary-parallel walks.

The product's ``ddtree_shard_walk_*`` kernels run on the GPU only. To test the
host orchestration (``sharded.shard_walk``) and the split of each reduction
into per-rank records and a rank-order merge on CPU ranks over gloo, this
module restates those kernels' record layout and merge rules with numpy on
CPU tensors: the packed argmax key (order key of the value, then the lowest
global index), the (max, sum of exp((x - max)/T)) pair merged in rank order,
the children's logits (-inf outside the slice), the child tests of the
renormalising walk and the Gumbel-max bonus with the oracle's Philox words.
Test infrastructure only.
"""
import numpy as np
import torch

import oracle as O

REC = 36


def order_key(x: np.float32) -> int:
    if np.isnan(x):
        return 0
    if x == 0:
        x = np.float32(0.0)
    u = int(np.array([x], np.float32).view(np.uint32)[0])
    return (~u & 0xFFFFFFFF) if (u & 0x80000000) else (u | 0x80000000)


def pack(key: int, idx: int) -> int:
    return (key << 32) | (0xFFFFFFFF - idx)


def unpack_idx(p: int) -> int:
    return 0xFFFFFFFF - (p & 0xFFFFFFFF)


def f32_bits(x) -> int:
    return int(np.array([x], np.float32).view(np.int32)[0])


def bits_f32(w) -> np.float32:
    return np.array([int(w) & 0xFFFFFFFF], np.uint32).view(np.float32)[0]


def kids_of(tree, b, u):
    fc, ns = tree.first_child.numpy(), tree.next_sibling.numpy()
    out, c = [], int(fc[b, u])
    while c != -1:
        out.append(c)
        c = int(ns[b, c])
    return out


class CpuShardOps:
    def begin(self, state, out, D):
        state.zero_()
        out["out_tokens"].fill_(-1)
        out["out_nodes"].fill_(-1)
        out["out_nodes"][:, 0] = 0
        out["accept_len"].zero_()
        out["bonus"].fill_(-1)

    def partial(self, logits_shard, v0, V, tree, temperature, state):
        B, N, Vs = logits_shard.shape
        rec = np.zeros((B, REC), np.int64)
        lg = logits_shard.numpy()
        tok = tree.token.numpy()
        for b in range(B):
            u, phase = int(state[b, 0]), int(state[b, 2])
            rec[b, 2] = f32_bits(-np.inf)
            rec[b, 3] = f32_bits(0.0)
            rec[b, 4:] = f32_bits(-np.inf)
            if phase != 0:
                continue
            row = lg[b, u]
            if temperature is None:
                best = max(pack(order_key(row[i]), v0 + i) for i in range(Vs))
                rec[b, 0], rec[b, 1] = best & 0xFFFFFFFF, best >> 32
            else:
                T = float(temperature[b])
                m = float(row.max())
                z = float(np.exp((row.astype(np.float64) - m) / T).sum())
                rec[b, 2], rec[b, 3] = f32_bits(m), f32_bits(z)
            for j, c in enumerate(kids_of(tree, b, u)):
                x = int(tok[b, c])
                if v0 <= x < v0 + Vs:
                    rec[b, 4 + j] = f32_bits(row[x - v0])
        rec = np.where(rec >= 2 ** 31, rec - 2 ** 32, rec)
        return torch.from_numpy(rec.astype(np.int32))

    def advance(self, records, V, tree, D, temperature, seed, offset, state, out, dev_status=None):
        W, B, _ = records.shape
        r = records.numpy().astype(np.int64) & 0xFFFFFFFF
        tok = tree.token.numpy()
        for b in range(B):
            if int(state[b, 2]) != 0:
                continue
            u, ln = int(state[b, 0]), int(state[b, 1])
            kids = kids_of(tree, b, u)
            match = -1
            if temperature is None:
                best = max(int(r[w, b, 0]) | (int(r[w, b, 1]) << 32) for w in range(W))
                a = unpack_idx(best)
                for c in kids:
                    if int(tok[b, c]) == a:
                        match = c
                        break
                    state[b, 3] += 1
            else:
                T = float(temperature[b])
                ms = [(float(bits_f32(r[w, b, 2])), float(bits_f32(r[w, b, 3]))) for w in range(W)]
                M = max(m for m, _ in ms)
                Z = sum(z * np.exp((m - M) / T) for m, z in ms if z > 0)
                R = 1.0
                for j, c in enumerate(kids):
                    lj = max(float(bits_f32(r[w, b, 4 + j])) for w in range(W))
                    q = np.exp((lj - M) / T) / Z
                    uj = float(O.to_uniform(O.draw_words(int(seed[b]), offset, O.PURPOSE_ACCEPT, u, j)[0]))
                    if uj * R < q:
                        match = c
                        break
                    R -= q
                    state[b, 3] += 1
            if match != -1:
                out["out_tokens"][b, ln] = int(tok[b, match])
                out["out_nodes"][b, ln + 1] = match
                state[b, 0], state[b, 1] = match, ln + 1
            elif temperature is None:
                out["out_tokens"][b, ln] = a
                out["bonus"][b] = a
                out["accept_len"][b] = ln
                state[b, 2] = 2
            else:
                state[b, 2] = 1

    def bonus(self, logits_shard, v0, V, tree, temperature, seed, offset, state):
        B, N, Vs = logits_shard.shape
        keys = np.zeros(B, np.uint64)
        lg = logits_shard.numpy()
        tok = tree.token.numpy()
        for b in range(B):
            if int(state[b, 2]) != 1:
                continue
            u = int(state[b, 0])
            kid_tok = {int(tok[b, c]) for c in kids_of(tree, b, u)}
            T = np.float32(1.0) / np.float32(temperature[b])
            vidx = np.arange(v0, v0 + Vs, dtype=np.uint64)
            words = np.stack(O.draw_words(int(seed[b]), offset, O.PURPOSE_GUMBEL, u, vidx >> np.uint64(2)))
            w = words[(vidx & np.uint64(3)).astype(np.int64), np.arange(Vs)]
            g = -np.log(-np.log(O.to_uniform(w)))
            best = 0
            for i in range(Vs):
                if v0 + i in kid_tok:
                    continue
                best = max(best, pack(order_key(np.float32(lg[b, u, i] * T + g[i])), v0 + i))
            keys[b] = best
        return torch.from_numpy(keys.view(np.int64))

    def finish(self, keys, D, state, out):
        W, B = keys.shape
        k = keys.numpy().view(np.uint64)
        for b in range(B):
            if int(state[b, 2]) != 1:
                continue
            best = int(k[:, b].max())
            ln = int(state[b, 1])
            a = unpack_idx(best) if best else -1
            out["out_tokens"][b, ln] = a
            out["bonus"][b] = a
            out["accept_len"][b] = ln
            state[b, 2] = 2
