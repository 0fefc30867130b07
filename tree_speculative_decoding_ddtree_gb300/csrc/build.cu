// ddtree_build: best-first DDTree construction, one warp per request.
//
// Method: "The Architecture of Speculative Decoding: Dissecting DDTree's
// Tree-Parallel Evaluation Strategy", Section 1 (The Five-Step Flow of
// DDTree), steps 2-3: pop the best node by cumulative log-prob, add it, push
// its best child and its next sibling, until `budget` nodes are chosen; the
// mask lets a node see its ancestors. "The Tree That Couldn't Branch",
// Context section (top-k cap per node) and Hypothesis 3 (position =
// ctx_len + depth).
//
// GPU design: one warp (one CTA) per request, with the request's top-k staged
// in shared memory. The heap is a warp-wide sorted list held in registers
// (entry p in slot p / 32 of lane p % 32), ordered by a 64-bit integer key
// that preserves the order of the fp64 score, newest last among equal keys.
// That is the heap's total order (score descending, earlier push first), so a
// pop takes entry 0 and an insert lands after every entry with a key >= its
// own: one ballot and one shift. Only lane 0 touches fp64 (two adds per pop,
// in path order, as in the definition); it also records each node's first
// child and next sibling as nodes are added. Masks and positions are then
// computed with every lane working on its own nodes.
#include "common.cuh"

namespace ddt {

constexpr int kMaxN = DDT_MAX_NODES;          // 128
constexpr int kMaxW = (kMaxN + 31) / 32;      // 4

struct BuildSmem {
    double n_score[kMaxN];
    int n_parent[kMaxN];
    int n_depth[kMaxN];
    int n_rank[kMaxN];
    int root_token;
    int n_first_child[kMaxN];
    int n_next_sibling[kMaxN];
};

// order-preserving key of a double (NaN ranks as -inf); 0 is below every key.
// Integer operations only: fp64 compares are slow on this GPU.
DDT_DEVINL unsigned long long score_key(double s) {
    unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(s));
    if ((b & 0x7FFFFFFFFFFFFFFFull) > 0x7FF0000000000000ull) b = 0xFFF0000000000000ull;   // NaN -> -inf
    return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}
DDT_DEVINL double key_score(unsigned long long k) {
    const unsigned long long b = (k >> 63) ? (k & 0x7FFFFFFFFFFFFFFFull) : ~k;
    return __longlong_as_double(static_cast<long long>(b));
}

// entry code: depth << 24 | previous sibling << 16 | rank << 8 | parent
// (depth <= 64, node indices <= 127, rank <= 31: each fits its byte)
DDT_DEVINL uint32_t entry_code(int d, int prev, int r, int p) {
    return (static_cast<uint32_t>(d) << 24) | (static_cast<uint32_t>(prev) << 16) |
           (static_cast<uint32_t>(r) << 8) | static_cast<uint32_t>(p);
}

template <int SLOTS>
struct WarpHeap {
    unsigned long long key[SLOTS];
    uint32_t code[SLOTS];   // entry_code()

    DDT_DEVINL void clear() {
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) { key[s] = 0ull; code[s] = 0u; }
    }
    // remove entry 0 (every other entry moves one place forward)
    DDT_DEVINL void pop_front(int lane) {
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            unsigned long long k = __shfl_down_sync(0xffffffffu, key[s], 1);
            uint32_t c = __shfl_down_sync(0xffffffffu, code[s], 1);
            const unsigned long long kn = s + 1 < SLOTS ? __shfl_sync(0xffffffffu, key[(s + 1) % SLOTS], 0) : 0ull;
            const uint32_t cn = s + 1 < SLOTS ? __shfl_sync(0xffffffffu, code[(s + 1) % SLOTS], 0) : 0u;
            if (lane == 31) { k = kn; c = cn; }
            key[s] = k;
            code[s] = c;
        }
    }
    // insert after every entry whose key is >= k (stable: later pushes go last)
    DDT_DEVINL void insert(unsigned long long k, uint32_t c, int lane) {
        int pos = 0;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) pos += __popc(__ballot_sync(0xffffffffu, key[s] >= k));
        unsigned long long carry_k = 0ull;
        uint32_t carry_c = 0u;
#pragma unroll
        for (int s = 0; s < SLOTS; ++s) {
            const unsigned long long up_k = __shfl_up_sync(0xffffffffu, key[s], 1);
            const uint32_t up_c = __shfl_up_sync(0xffffffffu, code[s], 1);
            const unsigned long long last_k = __shfl_sync(0xffffffffu, key[s], 31);
            const uint32_t last_c = __shfl_sync(0xffffffffu, code[s], 31);
            const int p = s * 32 + lane;
            const unsigned long long prev_k = lane == 0 ? carry_k : up_k;
            const uint32_t prev_c = lane == 0 ? carry_c : up_c;
            if (p == pos) { key[s] = k; code[s] = c; }
            else if (p > pos) { key[s] = prev_k; code[s] = prev_c; }
            carry_k = last_k;
            carry_c = last_c;
        }
    }
};

// lp: the request's top-k log-probs, already widened to fp64 (exactly), so
// the loop's only fp64 instructions are the two independent score adds per pop.
// Every lane computes both new scores from the same shared-memory values (no
// broadcast on the critical path); lane 0 alone records the node. The list
// keeps only entries that can still be popped: an entry at place p needs p + 1
// more pops to reach the front (inserts only move entries back), so with
// budget - count pops left anything past that place never matters, and
// SLOTS * 32 >= budget places suffice. An insert into a full list drops its
// last entry.
// A node's first child is its rank-0 child and the next sibling of a rank-r
// node the rank-(r+1) node it pushed (a sibling is pushed only when the one
// before it is added), so both links are known when a node is added.
template <int SLOTS>
DDT_DEVINL int build_pops(BuildSmem& s, const double* lp, const int32_t* tk, int D, int K, int budget,
                          int lane) {
    WarpHeap<SLOTS> h;
    h.clear();
    int count = 0, live = 0;
    if (budget >= 1) {
        h.insert(score_key(0.0 + lp[0]), entry_code(1, 0, 0, 0), lane);
        live = 1;
    }
    while (count < budget && live > 0) {
        const unsigned long long bk = __shfl_sync(0xffffffffu, h.key[0], 0);
        const uint32_t code = __shfl_sync(0xffffffffu, h.code[0], 0);
        h.pop_front(lane);
        --live;
        const int d = static_cast<int>(code >> 24), q = static_cast<int>((code >> 16) & 0xffu),
                  r = static_cast<int>((code >> 8) & 0xffu), p = static_cast<int>(code & 0xffu);
        ++count;
        const int i = count;
        const double sc = key_score(bk);
        const double cs = d < D ? sc + lp[d * K] : 0.0;                                // best child
        const double ss = r + 1 < K ? s.n_score[p] + lp[(d - 1) * K + r + 1] : 0.0;    // next sibling
        // the node's record (its token is looked up from depth and rank afterwards)
        if (lane == 0) {
            s.n_score[i] = sc;
            s.n_parent[i] = p;
            s.n_depth[i] = d;
            s.n_rank[i] = r;
            if (r == 0) s.n_first_child[p] = i;
            else s.n_next_sibling[q] = i;
        }
        const unsigned long long ck = score_key(cs);
        const unsigned long long sk = score_key(ss);
        if (d < D) {   // the child is pushed before the sibling
            h.insert(ck, entry_code(d + 1, 0, 0, i), lane);
            ++live;
        }
        if (r + 1 < K) {
            h.insert(sk, entry_code(d, i, r + 1, p), lane);
            ++live;
        }
        __syncwarp();
    }
    return count;
}

__global__ void __launch_bounds__(32)
ddtree_build_kernel(const float* __restrict__ topk_logp, const int32_t* __restrict__ topk_tok,
                    const int32_t* __restrict__ root_tok, const int32_t* __restrict__ ctx_len,
                    int B, int D, int K, int budget,
                    int32_t* __restrict__ parent, int32_t* __restrict__ depth,
                    int32_t* __restrict__ token, int32_t* __restrict__ rank,
                    int32_t* __restrict__ pos, double* __restrict__ score,
                    int32_t* __restrict__ first_child, int32_t* __restrict__ next_sibling,
                    uint32_t* __restrict__ vis, int32_t* __restrict__ n_nodes_out,
                    int32_t* dev_status) {
    __shared__ BuildSmem s;
    extern __shared__ __align__(16) unsigned char dyn[];   // staged top-k: D*K doubles then D*K ints
    // a programmatic dependent (the attention) may start now: it reads this
    // kernel's outputs only after waiting for the whole grid
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x;
    double* lp = reinterpret_cast<double*>(dyn);
    int32_t* tk = reinterpret_cast<int32_t*>(dyn + sizeof(double) * D * K);
    {
        const float* glp = topk_logp + static_cast<size_t>(b) * D * K;
        const int32_t* gtk = topk_tok + static_cast<size_t>(b) * D * K;
        for (int x = lane; x < D * K; x += 32) { lp[x] = static_cast<double>(glp[x]); tk[x] = gtk[x]; }
    }
    const int N = budget + 1;
    const int W = (N + 31) >> 5;
    const int L = ctx_len[b];
    if (lane == 0) {
        s.n_score[0] = 0.0;
        s.n_parent[0] = -1;
        s.n_depth[0] = 0;
        s.n_rank[0] = 0;
        s.root_token = root_tok[b];
    }
    for (int i = lane; i < N; i += 32) { s.n_first_child[i] = -1; s.n_next_sibling[i] = -1; }
    __syncwarp();

    int count;   // the list needs budget places (see build_pops)
    if (budget <= 32) count = build_pops<1>(s, lp, tk, D, K, budget, lane);
    else if (budget <= 64) count = build_pops<2>(s, lp, tk, D, K, budget, lane);
    else count = build_pops<4>(s, lp, tk, D, K, budget, lane);
    const int n = count + 1;
    __syncwarp();

    if (L < 0 && lane == 0) report(dev_status, DDT_DEV_BAD_CTX);
    const size_t base = static_cast<size_t>(b) * N;
    for (int i = lane; i < N; i += 32) {
        const bool real = i < n;
        uint32_t vw[kMaxW] = {0u, 0u, 0u, 0u};
        if (real)   // ancestor-or-self bits
            for (int a = i; a >= 0; a = s.n_parent[a]) vw[a >> 5] |= 1u << (a & 31);
        parent[base + i] = real ? s.n_parent[i] : -1;
        depth[base + i] = real ? s.n_depth[i] : -1;
        token[base + i] = !real ? -1 : (i == 0 ? s.root_token : tk[(s.n_depth[i] - 1) * K + s.n_rank[i]]);
        rank[base + i] = real ? s.n_rank[i] : -1;
        pos[base + i] = real ? L + s.n_depth[i] : -1;
        score[base + i] = real ? s.n_score[i] : -INFINITY;
        first_child[base + i] = real ? s.n_first_child[i] : -1;
        next_sibling[base + i] = real ? s.n_next_sibling[i] : -1;
        for (int w = 0; w < W; ++w) vis[(base + i) * W + w] = vw[w];
    }
    if (lane == 0) n_nodes_out[b] = n;
}

cudaError_t launch_build(const float* topk_logp, const int32_t* topk_tok, const int32_t* root_tok,
                         const int32_t* ctx_len, int B, int D, int K, int budget,
                         int32_t* parent, int32_t* depth, int32_t* token, int32_t* rank,
                         int32_t* pos, double* score, int32_t* first_child,
                         int32_t* next_sibling, uint32_t* vis, int32_t* n_nodes,
                         int32_t* dev_status, cudaStream_t stream) {
    const size_t dyn = static_cast<size_t>(D) * K * 12;
    ddtree_build_kernel<<<B, 32, dyn, stream>>>(
        topk_logp, topk_tok, root_tok, ctx_len, B, D, K, budget, parent, depth, token, rank,
        pos, score, first_child, next_sibling, vis, n_nodes, dev_status);
    return cudaGetLastError();
}

}  // namespace ddt
