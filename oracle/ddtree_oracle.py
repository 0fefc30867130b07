"""Plain fp64 CPU oracle for the DDTree tree-verify step.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or run
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it. It shares
no code with the CUDA path; both sides read their inputs from ``ddtree_synth``.

Every function follows the method as the pages state it, in their order, with
plain loops and fp64 arithmetic; numpy primitives (a matmul, an exp, an
argmax, a sort) serve as single steps, with no blocking, fusion or reordering
beyond what the definition states. Sources, cited by page title and section:

* [Arch]   "The Architecture of Speculative Decoding: Dissecting DDTree's
           Tree-Parallel Evaluation Strategy"
* [Verify] "The Architecture of Speculative Verification: Implementing
           Temperature-Aware Tree Sampling for DDTree"
* [Pivot]  "The Pivot Point: Strategic Decision-Making in Speculative Decoding
           Optimization"
* [Branch] "The Tree That Couldn't Branch: Diagnosing a 2x Acceptance
           Regression in DDTree Speculative Decoding"

Where the pages are silent the plainest reading is taken and named at the
function. Pins (checks against things other than this code) live in
``tests/test_oracle_pins.py``; every function here has at least one.
"""
from __future__ import annotations

import heapq
import math
from dataclasses import dataclass

import numpy as np

U32 = 0xFFFFFFFF


# ----------------------------------------------------------------------------
# bf16 -> fp64 widening (exact)
# ----------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bits (uint16) to fp64 exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# a0 (input preparation): per-depth top-k log-probs of the draft
# ----------------------------------------------------------------------------

def draft_topk(draft_logits: np.ndarray, K: int):
    """Per-depth top-K token ids and log-probs of the draft.

    [Arch] §"Section 1: The Five-Step Flow of DDTree", step 1: from each depth
    position of the single draft forward, the top-k candidate tokens are taken
    with their log-probs. [Branch] §"Hypothesis 4": each depth's distribution
    is conditioned on the anchor only, so one row per depth serves every node.

    Reading (pages silent): top-K tokens by the value of the draft logit
    (log-softmax subtracts one constant per row, so this is the log-prob
    order; ranking on the logit itself keeps distinct logits distinct where
    the fp64 subtraction would round them to one value), ties going to the
    lower token id; their log-probs are computed in fp64 over the row, then
    rounded to fp32. These fp32 arrays are what both the oracle and the CUDA
    path consume.

    Returns ``(topk_logp fp32 [B,D,K], topk_tok int32 [B,D,K])``.
    """
    x = np.asarray(draft_logits, dtype=np.float64)
    B, D, V = x.shape
    logp = np.empty_like(x)
    for b in range(B):
        for d in range(D):
            row = x[b, d]
            m = row.max()
            lse = m + math.log(np.exp(row - m).sum())
            logp[b, d] = row - lse
    tok = np.empty((B, D, K), dtype=np.int32)
    val = np.empty((B, D, K), dtype=np.float32)
    ids = np.arange(V)
    for b in range(B):
        for d in range(D):
            order = np.lexsort((ids, -x[b, d]))[:K]
            tok[b, d] = order
            val[b, d] = logp[b, d, order].astype(np.float32)
    return val, tok


# ----------------------------------------------------------------------------
# a1: best-first tree build, visibility and positions
# ----------------------------------------------------------------------------

def _nan_low(s: float) -> float:
    return -math.inf if s != s else s


@dataclass
class Tree:
    """Tree arrays for a batch; N = budget + 1 rows per request."""
    parent: np.ndarray        # int32 [B,N]; -1 for the root and for pad rows
    depth: np.ndarray         # int32 [B,N]; 0 for the root, -1 for pad rows
    token: np.ndarray         # int32 [B,N]; root_tok for the root, -1 for pad rows
    rank: np.ndarray          # int32 [B,N]; rank among the depth's top-k, 0 root, -1 pad
    pos: np.ndarray           # int32 [B,N]; ctx_len + depth, -1 pad
    score: np.ndarray         # fp64  [B,N]; cumulative log-prob, 0 root, -inf pad
    first_child: np.ndarray   # int32 [B,N]; -1 if none
    next_sibling: np.ndarray  # int32 [B,N]; -1 if none
    vis: np.ndarray           # uint32 [B,N,W]; bit j of row i: j is ancestor-or-self of i
    n_nodes: np.ndarray       # int32 [B]


def build_tree(topk_logp: np.ndarray, topk_tok: np.ndarray, root_tok: np.ndarray,
               ctx_len: np.ndarray, budget: int) -> Tree:
    """Best-first tree under a node budget and a per-node top-k cap.

    [Arch] §"Section 1", step 2: a heap keyed by cumulative log-prob; pop the
    best node and add it; push its best child and its next sibling; repeat
    until ``budget`` nodes are chosen, giving budget+1 nodes with the root.
    [Branch] §"Context: The Road to DDTree": the cap K bounds the children
    per node. [Branch] §"Hypothesis 4": every node at depth d draws its
    children from the same depth-(d+1) top-k.

    Readings (pages silent):
    * the root is node 0 (depth 0, token ``root_tok``, score 0); nodes are
      numbered in pop order, so a parent always precedes its children;
    * a node's score is its parent's score plus its own fp32 log-prob, added in
      fp64 along the path;
    * heap order: larger score first, then the earlier push; the child is
      pushed before the sibling;
    * the depth never exceeds D; if the heap empties first, n_nodes < N and the
      remaining rows are pads;
    * a NaN score (from a NaN log-prob) ranks as -inf.
    """
    lp = np.asarray(topk_logp, dtype=np.float32)
    tk = np.asarray(topk_tok, dtype=np.int32)
    B, D, K = lp.shape
    N = budget + 1
    parent = np.full((B, N), -1, np.int32)
    depth = np.full((B, N), -1, np.int32)
    token = np.full((B, N), -1, np.int32)
    rank = np.full((B, N), -1, np.int32)
    pos = np.full((B, N), -1, np.int32)
    score = np.full((B, N), -np.inf, np.float64)
    n_nodes = np.zeros(B, np.int32)
    for b in range(B):
        depth[b, 0] = 0
        token[b, 0] = int(root_tok[b])
        rank[b, 0] = 0
        score[b, 0] = 0.0
        heap = []
        seq = 0
        if D >= 1 and K >= 1 and budget >= 1:
            heapq.heappush(heap, (-_nan_low(0.0 + float(lp[b, 0, 0])), seq, 1, 0, 0))
            seq += 1
        count = 0
        while count < budget and heap:
            neg, _, d, r, p = heapq.heappop(heap)
            count += 1
            i = count
            parent[b, i] = p
            depth[b, i] = d
            rank[b, i] = r
            token[b, i] = int(tk[b, d - 1, r])
            score[b, i] = -neg
            if d < D:   # best child: rank 0 at depth d+1
                heapq.heappush(heap, (-_nan_low(score[b, i] + float(lp[b, d, 0])), seq, d + 1, 0, i))
                seq += 1
            if r + 1 < K:   # next sibling: same parent, rank r+1
                heapq.heappush(heap, (-_nan_low(score[b, p] + float(lp[b, d - 1, r + 1])), seq, d, r + 1, p))
                seq += 1
        n_nodes[b] = count + 1
        for i in range(count + 1):
            pos[b, i] = int(ctx_len[b]) + depth[b, i]
    first_child, next_sibling = child_lists(parent, n_nodes)
    vis = visibility_words(parent, n_nodes, N)
    return Tree(parent, depth, token, rank, pos, score, first_child, next_sibling, vis, n_nodes)


def child_lists(parent: np.ndarray, n_nodes: np.ndarray):
    """Children of each node as first-child / next-sibling links, in index order.

    [Arch] §"Section 3" (the stored child maps walked by the accept step).
    Index order equals rank order because siblings are popped in rank order.
    """
    B, N = parent.shape
    first = np.full((B, N), -1, np.int32)
    nxt = np.full((B, N), -1, np.int32)
    for b in range(B):
        last = {}
        for i in range(1, int(n_nodes[b])):
            p = int(parent[b, i])
            if p in last:
                nxt[b, last[p]] = i
            else:
                first[b, p] = i
            last[p] = i
    return first, nxt


def visibility_matrix(parent: np.ndarray, n_nodes: np.ndarray, N: int) -> np.ndarray:
    """Tree part of the verify mask: ``vis[b, i, j]`` iff node j is i or an ancestor of i.

    [Arch] §"Section 1", step 3: each node attends only to its ancestors plus
    the shared prefix (the prefix part is implicit: every valid row sees the
    whole context, [Arch] §"Section 2"). Reading: a node sees itself. Pad
    rows see nothing.
    """
    B = parent.shape[0]
    m = np.zeros((B, N, N), dtype=bool)
    for b in range(B):
        for i in range(int(n_nodes[b])):
            j = i
            while j != -1:
                m[b, i, j] = True
                j = int(parent[b, j])
    return m


def visibility_words(parent: np.ndarray, n_nodes: np.ndarray, N: int) -> np.ndarray:
    """``visibility_matrix`` packed as uint32 words: bit (j % 32) of word j // 32."""
    m = visibility_matrix(parent, n_nodes, N)
    B = m.shape[0]
    W = (N + 31) // 32
    out = np.zeros((B, N, W), dtype=np.uint32)
    for b in range(B):
        for i in range(N):
            for j in range(N):
                if m[b, i, j]:
                    out[b, i, j // 32] |= np.uint32(1 << (j % 32))
    return out


def unpack_vis(vis: np.ndarray, N: int) -> np.ndarray:
    """Inverse of ``visibility_words``: uint32 [B,N,W] -> bool [B,N,N]."""
    B = vis.shape[0]
    m = np.zeros((B, N, N), dtype=bool)
    for j in range(N):
        m[:, :, j] = (vis[:, :, j // 32] >> np.uint32(j % 32)) & np.uint32(1)
    return m


# ----------------------------------------------------------------------------
# a2: tree-verify attention over the paged context plus the tree rows
# ----------------------------------------------------------------------------

def gather_context(cache: np.ndarray, page_table: np.ndarray, b: int, L: int,
                   page_size: int) -> np.ndarray:
    """Context K (or V) of request b in token order: ``[L, Hkv, Dh]``."""
    n_pages = -(-L // page_size)
    pages = [int(p) for p in page_table[b, :n_pages]]
    if not pages:
        return cache[:0].reshape((0,) + cache.shape[2:])
    rows = np.concatenate([cache[p] for p in pages], axis=0)
    return rows[:L]


def tree_verify_attention(q, k_tree, v_tree, k_cache, v_cache, page_table, ctx_len,
                          vis_bool, n_nodes, scale, page_size, want_lse=False):
    """Attention of every tree row over its context plus its visible tree rows.

    [Arch] §"Section 1", step 4: all budget+1 nodes go through the target in
    one pass with the tree mask. [Arch] §"Section 2": every node sees the
    whole prefix ``[0, ctx_len)``, read from the cache once and shared.
    [Pivot] §"The Design Constraint: Load Contexts Once".

    For request b, row i and query head h (kv head ``h // (Hq/Hkv)``):
    ``o = softmax(scale * q k^T + mask) v`` over the context keys followed by
    the tree keys j with ``vis_bool[b, i, j]``. Inputs are fp64 arrays (bf16
    values widened exactly); the result is fp64 ``[B,N,Hq,Dh]``, with zeros for
    pad rows (i >= n_nodes). ``lse`` (natural log of the softmax denominator,
    fp64 ``[B,N,Hq]``, -inf for pad rows) is returned when asked.

    Readings (pages silent): GQA groups are contiguous (h // G); no soft-cap,
    window or bias; the root's own K/V is tree row 0, not part of the cache.
    """
    B, N, Hq, Dh = q.shape
    Hkv = k_tree.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, N, Hq, Dh), dtype=np.float64)
    lse = np.full((B, N, Hq), -np.inf, dtype=np.float64)
    for b in range(B):
        L = int(ctx_len[b])
        n = int(n_nodes[b])
        kc = gather_context(k_cache, page_table, b, L, page_size)
        vc = gather_context(v_cache, page_table, b, L, page_size)
        for h in range(Hq):
            kv = h // G
            keys = np.concatenate([kc[:, kv, :], k_tree[b, :, kv, :]], axis=0)
            vals = np.concatenate([vc[:, kv, :], v_tree[b, :, kv, :]], axis=0)
            s = scale * (q[b, :n, h, :] @ keys.T)              # [n, L+N]
            allow = np.concatenate([np.ones((n, L), bool), vis_bool[b, :n, :]], axis=1)
            s = np.where(allow, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            den = p.sum(axis=1, keepdims=True)
            out[b, :n, h, :] = (p @ vals) / den
            lse[b, :n, h] = (m + np.log(den))[:, 0]
    return (out, lse) if want_lse else out


def attention_row(q, k_tree, v_tree, k_cache, v_cache, page_table, ctx_len, vis_bool,
                  n_nodes, scale, page_size, b, i, h):
    """One output row ``o[b, i, h, :]`` (fp64) of ``tree_verify_attention``.

    Same definition, evaluated for a single (request, row, head) so that very
    large workloads can be checked on sampled rows.
    """
    Hq = q.shape[2]
    Hkv = k_tree.shape[2]
    kv = h // (Hq // Hkv)
    Dh = q.shape[3]
    if i >= int(n_nodes[b]):
        return np.zeros(Dh), -np.inf
    L = int(ctx_len[b])
    n_pages = -(-L // page_size)
    pages = [int(p) for p in page_table[b, :n_pages]]
    kc = (np.concatenate([bf16_to_f64(k_cache[p, :, kv, :]) for p in pages], axis=0)[:L]
          if pages else np.zeros((0, Dh)))
    vc = (np.concatenate([bf16_to_f64(v_cache[p, :, kv, :]) for p in pages], axis=0)[:L]
          if pages else np.zeros((0, Dh)))
    sel = np.nonzero(vis_bool[b, i])[0]
    keys = np.concatenate([kc, bf16_to_f64(k_tree[b, sel, kv, :])], axis=0)
    vals = np.concatenate([vc, bf16_to_f64(v_tree[b, sel, kv, :])], axis=0)
    s = scale * (keys @ bf16_to_f64(q[b, i, h, :]))
    m = s.max()
    p = np.exp(s - m)
    den = p.sum()
    return (p @ vals) / den, m + math.log(den)


# ----------------------------------------------------------------------------
# a3: greedy accept walk
# ----------------------------------------------------------------------------

def argmax_lowest(row: np.ndarray) -> int:
    """Index of the largest value, ties to the lowest index; NaN ranks below every number.

    Reading (pages silent on ties and NaN): the lowest index wins a tie; a NaN
    is never chosen unless the whole row is NaN, in which case index 0.
    """
    r = np.asarray(row, dtype=np.float64)
    nan = np.isnan(r)
    if nan.all():
        return 0
    r = np.where(nan, -np.inf, r)
    best = r.max()
    cand = np.nonzero(r == best)[0]
    if best == -np.inf:
        cand = np.nonzero((r == -np.inf) & ~nan)[0]
    return int(cand[0])


def children(tree: Tree, b: int, u: int):
    c = int(tree.first_child[b, u])
    out = []
    while c != -1:
        out.append(c)
        c = int(tree.next_sibling[b, c])
    return out


@dataclass
class Accept:
    accept_len: np.ndarray   # int32 [B]: accepted draft tokens (bonus excluded)
    out_tokens: np.ndarray   # int32 [B, D+1]: accepted tokens then the bonus, -1 after
    out_nodes: np.ndarray    # int32 [B, D+1]: root then accepted nodes, -1 after
    bonus: np.ndarray        # int32 [B]
    margin: np.ndarray = None  # fp64 [B]: smallest decision margin (sampling only)
    rejected: np.ndarray = None  # int32 [B]: child tests that rejected (sampling) or
    #                              children compared without a match (greedy)
    margin_scaled: np.ndarray = None  # fp64 [B]: smallest margin / conditioning (sampling only)
    cond: np.ndarray = None    # fp64 [B]: largest conditioning factor on the path (sampling only)


def accept_greedy(logits: np.ndarray, tree: Tree, D: int) -> Accept:
    """Longest root path whose tokens match the target argmax, plus one bonus token.

    [Arch] §"Section 1", step 5: walk from the root, follow the target's
    argmax at the current node into the child carrying that token, stop when
    no child matches; return the accepted chain and one bonus token (the
    argmax at the last node). [Verify] §"The Context": the same rule as the
    linear chain, where draft i is accepted if the argmax at position i-1
    equals it. ``logits[b, u]`` is the target's prediction for the token that
    follows node u.

    Reading: ``accept_len`` counts accepted draft tokens, the bonus excluded;
    the commit length is ``accept_len + 1``. ``out_nodes`` lists the root and
    then the accepted nodes (the rows whose K/V a server would keep).
    """
    B = logits.shape[0]
    acc = np.zeros(B, np.int32)
    toks = np.full((B, D + 1), -1, np.int32)
    nodes = np.full((B, D + 1), -1, np.int32)
    bonus = np.zeros(B, np.int32)
    rejected = np.zeros(B, np.int32)
    for b in range(B):
        u = 0
        path = []
        while True:
            a = argmax_lowest(logits[b, u])
            match = -1
            for c in children(tree, b, u):
                if int(tree.token[b, c]) == a:
                    match = c
                    break
                rejected[b] += 1
            if match == -1:
                bonus[b] = a
                break
            path.append(match)
            u = match
        acc[b] = len(path)
        nodes[b, 0] = 0
        for k, c in enumerate(path):
            toks[b, k] = tree.token[b, c]
            nodes[b, k + 1] = c
        toks[b, len(path)] = bonus[b]
    return Accept(acc, toks, nodes, bonus, rejected=rejected)


# ----------------------------------------------------------------------------
# Philox4x32-10 (Salmon, Moraes, Dror, Shaw: "Parallel random numbers: as easy
# as 1, 2, 3", SC'11), written from the paper's definition
# ----------------------------------------------------------------------------

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9   # golden ratio
PHILOX_W1 = 0xBB67AE85   # sqrt(3) - 1


def philox4x32_10(ctr, key):
    """Philox4x32 with 10 rounds on one 128-bit counter and 64-bit key.

    Each round multiplies counter words 0 and 2 by the two round constants,
    swaps the word pairs and xors the high halves with the other counter
    words and the round key; the key is bumped by the two Weyl constants
    between rounds. ``ctr``: 4 ints, ``key``: 2 ints (all < 2**32).
    """
    c0, c1, c2, c3 = (int(x) & U32 for x in ctr)
    k0, k1 = (int(x) & U32 for x in key)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + PHILOX_W0) & U32
            k1 = (k1 + PHILOX_W1) & U32
        p0 = PHILOX_M0 * c0
        p1 = PHILOX_M1 * c2
        hi0, lo0 = p0 >> 32, p0 & U32
        hi1, lo1 = p1 >> 32, p1 & U32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def philox4x32_10_np(c0, c1, c2, c3, k0, k1):
    """Elementwise ``philox4x32_10`` over numpy arrays (uint64 holding 32-bit words)."""
    m = np.uint64(U32)
    c0, c1, c2, c3 = (np.asarray(x, dtype=np.uint64) & m for x in (c0, c1, c2, c3))
    k0 = np.asarray(k0, dtype=np.uint64) & m
    k1 = np.asarray(k1, dtype=np.uint64) & m
    for rnd in range(10):
        if rnd:
            k0 = (k0 + np.uint64(PHILOX_W0)) & m
            k1 = (k1 + np.uint64(PHILOX_W1)) & m
        p0 = np.uint64(PHILOX_M0) * c0
        p1 = np.uint64(PHILOX_M1) * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & m
        hi1, lo1 = p1 >> np.uint64(32), p1 & m
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


PURPOSE_ACCEPT = 0
PURPOSE_GUMBEL = 1


def draw_words(seed: int, offset: int, purpose: int, node: int, index):
    """Philox words for one (request seed, step offset, purpose, node, index).

    Reading (the pages give no RNG): key = (seed low 32 bits, seed high 32
    bits); counter = (purpose | (offset >> 32) << 8, node, index, offset low
    32 bits). ``index`` may be an array.
    """
    idx = np.asarray(index, dtype=np.uint64)
    c0 = np.full(idx.shape, (purpose | ((int(offset) >> 32) << 8)) & U32, dtype=np.uint64)
    c1 = np.full(idx.shape, node, dtype=np.uint64)
    c3 = np.full(idx.shape, int(offset) & U32, dtype=np.uint64)
    return philox4x32_10_np(c0, c1, idx, c3, int(seed) & U32, (int(seed) >> 32) & U32)


def to_uniform(word) -> np.ndarray:
    """Map a 32-bit word to (0, 1): the top 24 bits plus one half, times 2**-24."""
    w = np.asarray(word, dtype=np.uint64)
    return ((w >> np.uint64(8)).astype(np.float64) + 0.5) * (2.0 ** -24)


# ----------------------------------------------------------------------------
# a4: temperature accept walk (recursive rejection sampling over siblings)
# ----------------------------------------------------------------------------

def accept_sample(logits: np.ndarray, tree: Tree, D: int, temperature: np.ndarray,
                  seed: np.ndarray, offset: int) -> Accept:
    """Tree verification at temperature T by recursive rejection over siblings.

    [Arch] §"Section 3: Temperature Support", tree case: at each node,
    reject-sample the children in turn; on an acceptance descend; once every
    child is rejected, draw the bonus from the residual and stop.
    [Verify] §"Path B: CPU-Side Tree Rejection Sampling" and §"The Knowledge
    Required …" item 3: the target distribution q = softmax(logits / T);
    accept with min(1, q/p), else renormalise q over what remains.

    Reading: a DDTree child is the deterministic top-k token of its depth, so
    the distribution it was proposed from is a point mass at that token. With
    p = a point mass, min(1, q(x)/p(x)) = q(x) and the residual max(q - p, 0)
    renormalised is q with x removed; applied to siblings in rank order this
    gives: child j (token x_j) is accepted with probability
    q(x_j) / (1 - sum_{i<j} q(x_i)). The bonus is drawn from q restricted to
    tokens that are not children of the final node (all of q at a leaf), by
    Gumbel-max. Emitted tokens are then distributed exactly as the target.

    Randomness: uniform ``U(node u, slot j)`` from ``draw_words`` with the
    accept purpose, word 0; Gumbel noise for vocab entry v from the Gumbel
    purpose at index v >> 2, word v & 3: g = -log(-log U).

    ``margin[b]`` is the smallest decision margin on the path:
    |u_j - q(x_j)/R| for each child test and the gap between the two best
    perturbed scores for the bonus. ``margin_scaled[b]`` divides each child
    test's margin by its conditioning 1/R (a relative error e in the q values
    moves the threshold q(x_j)/R by up to about e/R) before taking the
    minimum; the bonus gap is taken as it is. ``rejected[b]`` counts the
    child tests that rejected.
    """
    B, N, V = logits.shape
    acc = np.zeros(B, np.int32)
    toks = np.full((B, D + 1), -1, np.int32)
    nodes = np.full((B, D + 1), -1, np.int32)
    bonus = np.zeros(B, np.int32)
    margin = np.full(B, np.inf)
    margin_scaled = np.full(B, np.inf)
    rejected = np.zeros(B, np.int32)
    cond_max = np.ones(B)
    vidx = np.arange(V, dtype=np.uint64)
    for b in range(B):
        T = float(temperature[b])
        if not T > 0.0:
            raise ValueError("temperature must be > 0")
        sd = int(seed[b])
        u = 0
        path = []
        while True:
            row = np.asarray(logits[b, u], dtype=np.float64) / T
            m = row.max()
            e = np.exp(row - m)
            q = e / e.sum()
            R = 1.0
            kids = children(tree, b, u)
            chosen = -1
            for j, c in enumerate(kids):
                x = int(tree.token[b, c])
                uj = float(to_uniform(draw_words(sd, offset, PURPOSE_ACCEPT, u, j)[0]))
                if R > 0.0:
                    thr = q[x] / R
                    margin[b] = min(margin[b], abs(uj - thr))
                    margin_scaled[b] = min(margin_scaled[b], abs(uj - thr) * R)
                    cond_max[b] = max(cond_max[b], 1.0 / R)
                if uj * R < q[x]:
                    chosen = c
                    break
                R -= q[x]
                rejected[b] += 1
            if chosen != -1:
                path.append(chosen)
                u = chosen
                continue
            words = draw_words(sd, offset, PURPOSE_GUMBEL, u, vidx >> np.uint64(2))
            stacked = np.stack(words, axis=0)                   # [4, V]
            w = stacked[(vidx & np.uint64(3)).astype(np.int64), np.arange(V)]
            g = -np.log(-np.log(to_uniform(w)))
            pert = row + g
            allowed = np.ones(V, bool)
            for c in kids:
                allowed[int(tree.token[b, c])] = False
            cand = np.nonzero(allowed)[0]
            if cand.size == 0:      # every token is a child: nothing left to draw
                bonus[b] = -1
            else:
                best = int(cand[np.argmax(pert[cand])])
                if cand.size >= 2:
                    top2 = np.partition(pert[cand], -2)[-2:]
                    margin[b] = min(margin[b], float(top2[1] - top2[0]))
                    margin_scaled[b] = min(margin_scaled[b], float(top2[1] - top2[0]))
                bonus[b] = best
            break
        acc[b] = len(path)
        nodes[b, 0] = 0
        for k, c in enumerate(path):
            toks[b, k] = tree.token[b, c]
            nodes[b, k + 1] = c
        toks[b, len(path)] = bonus[b]
    return Accept(acc, toks, nodes, bonus, margin, rejected, margin_scaled, cond_max)


# ----------------------------------------------------------------------------
# commit: the verified path's K/V appended to the paged cache
# ----------------------------------------------------------------------------

def commit_kv(k_tree, v_tree, out_nodes, accept_len, ctx_len, page_table, k_cache, v_cache,
              page_size):
    """Append each request's committed path K/V to its paged cache.

    [Arch] §"Section 1", step 5: only the single longest verified path is
    committed; the other tree nodes are dropped. [Branch] §"Hypothesis 3": a
    node of depth d was verified at position ``ctx_len + d``.

    Reading (pages silent on the cache write): the committed rows are the
    root (tree row 0, whose K/V the verify pass computed at position
    ``ctx_len``) followed by the accepted nodes in path order, i.e.
    ``out_nodes[b, 0..accept_len[b]]``; path row i is written to token
    position ``ctx_len[b] + i`` (slot ``t % page_size`` of page
    ``page_table[b, t // page_size]``), which is its depth, so the position it
    was verified at. The bonus token is not written: it is the next step's
    root and its K/V comes from that pass. ``new_ctx_len = ctx_len +
    accept_len + 1``.

    Works on any element type (the bf16 bit patterns are copied as they are).
    Returns ``(k_cache', v_cache', new_ctx_len)`` as new arrays.
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    B = k_tree.shape[0]
    new_ctx = np.array(ctx_len, dtype=np.int32, copy=True)
    for b in range(B):
        a = int(accept_len[b])
        for i in range(a + 1):
            node = int(out_nodes[b, i])
            t = int(ctx_len[b]) + i
            page = int(page_table[b, t // page_size])
            slot = t % page_size
            kc[page, slot] = k_tree[b, node]
            vc[page, slot] = v_tree[b, node]
        new_ctx[b] = int(ctx_len[b]) + a + 1
    return kc, vc, new_ctx


# ----------------------------------------------------------------------------
# draft-ratio temperature walk (the min(1, q/p) rule with the draft softmax)
# ----------------------------------------------------------------------------

def accept_sample_ratio(logits: np.ndarray, draft_logits: np.ndarray, tree: Tree, D: int,
                        temperature: np.ndarray, seed: np.ndarray, offset: int) -> Accept:
    """Tree verification at temperature T with the draft-ratio rule.

    [Arch] §"Section 3: Temperature Support": linear case, accept draft token
    t with probability min(1, p_target(t) / p_draft(t)), else resample from
    the residual; tree case, reject-sample each node's children against their
    draft probabilities and, once they are all rejected, draw the bonus from
    the residual and stop. [Verify] §"The Knowledge Required …" item 3
    (accept with min(1, q/p); after a rejection the target distribution is
    renormalised over what remains) and §"Path B" (softmax only at the nodes
    visited). [Arch] §"Mistakes and Incorrect Assumptions" (the rule needs
    the draft's full distribution, not only its top-k): this walk takes the
    draft logits.

    Readings (pages silent):
    * p = softmax(draft_logits[b, d] / T) is the draft distribution the
      children of a depth-d node were taken from (the row whose top-k they
      are); q = softmax(logits[b, u] / T) at node u; one T for both.
    * Children are tested in rank order against a residual r that starts at
      q: child j (token x_j) is accepted when U_j * p(x_j) < r(x_j), i.e.
      with probability min(1, r(x_j) / p(x_j)); after a rejection
      r <- max(r - p, 0) / sum(max(r - p, 0)) (the SpecInfer-style update, so
      that candidates drawn independently from p emit tokens distributed as
      q). If a rejection leaves r without mass, no further child is tested
      and the bonus is drawn from q.
    * The bonus is drawn from the final r (r = q at a node without children,
      including every depth-D node) by Gumbel-max over the tokens with
      r > 0; the linear chain is the top-k-1 tree.

    Randomness as ``accept_sample``: U(node u, slot j) from the accept purpose,
    word 0; Gumbel noise of vocab entry v from the Gumbel purpose at index
    v >> 2, word v & 3. ``margin[b]`` is the smallest decision margin on the
    path: |U_j - r(x_j)/p(x_j)| for each child test and the gap between the
    two best perturbed scores for the bonus. ``rejected[b]`` counts the child
    tests that rejected.

    ``margin_scaled[b]`` divides each margin by its conditioning before the
    minimum. Written out, the residual after k rejections is
    r = max(q - C p, 0) / P with C = 0, P = 1 at first and C <- C + P,
    P <- P * mass at each rejection (tracked here beside the vector r, not
    used for the decisions). A relative error e in the q and p values moves a
    child's threshold r(x)/p(x) by up to about e (1 + C) / P, and the
    perturbed log-score log r(v) of a bonus candidate by about
    e (q(v) + C p(v)) / (q(v) - C p(v)); the conditioning of a child test is
    (1 + C) / P, that of the bonus gap the larger of that factor over the two
    best candidates.
    """
    B, N, V = logits.shape
    acc = np.zeros(B, np.int32)
    toks = np.full((B, D + 1), -1, np.int32)
    nodes = np.full((B, D + 1), -1, np.int32)
    bonus = np.zeros(B, np.int32)
    margin = np.full(B, np.inf)
    margin_scaled = np.full(B, np.inf)
    rejected = np.zeros(B, np.int32)
    cond_max = np.ones(B)
    vidx = np.arange(V, dtype=np.uint64)

    def softmax_t(row, T):
        z = np.asarray(row, dtype=np.float64) / T
        e = np.exp(z - z.max())
        return e / e.sum()

    for b in range(B):
        T = float(temperature[b])
        if not T > 0.0:
            raise ValueError("temperature must be > 0")
        sd = int(seed[b])
        u = 0
        path = []
        while True:
            q = softmax_t(logits[b, u], T)
            r = q
            C, P = 0.0, 1.0          # r = max(q - C p, 0) / P (bookkeeping for the conditioning)
            kids = children(tree, b, u) if len(path) < D else []
            chosen = -1
            if kids:
                p = softmax_t(draft_logits[b, len(path)], T)
                for j, c in enumerate(kids):
                    x = int(tree.token[b, c])
                    uj = float(to_uniform(draw_words(sd, offset, PURPOSE_ACCEPT, u, j)[0]))
                    if p[x] > 0.0:
                        margin[b] = min(margin[b], abs(uj - r[x] / p[x]))
                        margin_scaled[b] = min(margin_scaled[b], abs(uj - r[x] / p[x]) * P / (1.0 + C))
                        cond_max[b] = max(cond_max[b], (1.0 + C) / P)
                    if uj * p[x] < r[x]:
                        chosen = c
                        break
                    rejected[b] += 1
                    res = np.maximum(r - p, 0.0)
                    mass = res.sum()
                    if not mass > 0.0:   # nothing left to renormalise: the bonus comes from q
                        r = q
                        C, P = 0.0, 1.0
                        break
                    r = res / mass
                    C, P = C + P, P * mass
            if chosen != -1:
                path.append(chosen)
                u = chosen
                continue
            words = draw_words(sd, offset, PURPOSE_GUMBEL, u, vidx >> np.uint64(2))
            stacked = np.stack(words, axis=0)                   # [4, V]
            w = stacked[(vidx & np.uint64(3)).astype(np.int64), np.arange(V)]
            g = -np.log(-np.log(to_uniform(w)))
            cand = np.nonzero(r > 0.0)[0]
            if cand.size == 0:
                bonus[b] = -1
            else:
                pert = np.log(r[cand]) + g[cand]
                bonus[b] = int(cand[np.argmax(pert)])
                if cand.size >= 2:
                    order = np.argsort(pert)[-2:]
                    gap = float(pert[order[1]] - pert[order[0]])
                    margin[b] = min(margin[b], gap)
                    if C > 0.0:
                        pc = softmax_t(draft_logits[b, len(path)], T)
                        v2 = cand[order]
                        cond = float(np.max((q[v2] + C * pc[v2]) / (P * r[v2])))   # P r = q - C p
                    else:
                        cond = 1.0
                    margin_scaled[b] = min(margin_scaled[b], gap / cond)
                    cond_max[b] = max(cond_max[b], cond)
            break
        acc[b] = len(path)
        nodes[b, 0] = 0
        for k, c in enumerate(path):
            toks[b, k] = tree.token[b, c]
            nodes[b, k + 1] = c
        toks[b, len(path)] = bonus[b]
    return Accept(acc, toks, nodes, bonus, margin, rejected, margin_scaled, cond_max)
