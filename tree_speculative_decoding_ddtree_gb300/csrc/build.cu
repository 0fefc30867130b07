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
// GPU design: one warp (one CTA) per request. The request's per-depth top-k is
// staged in shared memory first, so the serial pop loop never waits on global
// memory. The frontier (the heap's contents) lives in shared memory as a flat
// array of at most budget+1 live entries; each pop is a warp-wide argmax over
// (score desc, push sequence asc), which is the heap's total order, so the pop
// sequence is the heap's exactly. Removal moves the last entry into the hole.
// Scores are fp64 sums in path order, as in the definition.
#include "common.cuh"

namespace ddt {

constexpr int kMaxN = DDT_MAX_NODES;          // 128
constexpr int kMaxW = (kMaxN + 31) / 32;      // 4
constexpr int kMaxFrontier = kMaxN;           // live entries <= 1 + budget <= 128

struct BuildSmem {
    double f_score[kMaxFrontier];
    int f_seq[kMaxFrontier];
    int f_code[kMaxFrontier];   // depth << 16 | rank << 8 | parent
    double n_score[kMaxN];
    int n_parent[kMaxN];
    int n_depth[kMaxN];
    int n_rank[kMaxN];
    int n_token[kMaxN];
    int n_first[kMaxN];
    int n_next[kMaxN];
    int n_last[kMaxN];
    uint32_t n_vis[kMaxN][kMaxW];
};

DDT_DEVINL double canon_score(double s) { return s != s ? -INFINITY : s; }

// true if entry (s, q) comes before (bs, bq) in pop order
DDT_DEVINL bool pops_before(double s, int q, double bs, int bq) {
    return s > bs || (s == bs && q < bq);
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
    extern __shared__ unsigned char dyn[];     // staged top-k: D*K floats then D*K ints
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x;
    float* lp = reinterpret_cast<float*>(dyn);
    int32_t* tk = reinterpret_cast<int32_t*>(dyn + sizeof(float) * D * K);
    {
        const float* glp = topk_logp + static_cast<size_t>(b) * D * K;
        const int32_t* gtk = topk_tok + static_cast<size_t>(b) * D * K;
        for (int x = lane; x < D * K; x += 32) { lp[x] = glp[x]; tk[x] = gtk[x]; }
        __syncwarp();
    }
    const int N = budget + 1;
    const int W = (N + 31) >> 5;

    if (lane == 0) {
        s.n_score[0] = 0.0;
        s.n_parent[0] = -1;
        s.n_depth[0] = 0;
        s.n_rank[0] = 0;
        s.n_token[0] = root_tok[b];
    }
    // warp-uniform bookkeeping (every lane keeps the same copy)
    int fsize = 0, seqc = 0, count = 0;
    if (budget >= 1) {
        if (lane == 0) {
            s.f_score[0] = canon_score(0.0 + static_cast<double>(lp[0]));
            s.f_seq[0] = 0;
            s.f_code[0] = (1 << 16) | (0 << 8) | 0;
        }
        fsize = 1;
        seqc = 1;
    }
    __syncwarp();

    while (count < budget && fsize > 0) {
        double bs = -INFINITY;
        int bq = 0x7fffffff, bi = -1;
        for (int e = lane; e < fsize; e += 32) {
            const double sc = s.f_score[e];
            const int q = s.f_seq[e];
            if (bi < 0 || pops_before(sc, q, bs, bq)) { bs = sc; bq = q; bi = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const double os = __shfl_xor_sync(0xffffffffu, bs, o);
            const int oq = __shfl_xor_sync(0xffffffffu, bq, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oi >= 0 && (bi < 0 || pops_before(os, oq, bs, bq))) { bs = os; bq = oq; bi = oi; }
        }
        const int code = s.f_code[bi];
        const int d = code >> 16, r = (code >> 8) & 0xff, p = code & 0xff;
        ++count;
        const int i = count;
        const bool push_child = d < D;
        const bool push_sib = r + 1 < K;
        __syncwarp();
        if (lane == 0) {
            --fsize;
            s.f_score[bi] = s.f_score[fsize];
            s.f_seq[bi] = s.f_seq[fsize];
            s.f_code[bi] = s.f_code[fsize];
            s.n_score[i] = bs;
            s.n_parent[i] = p;
            s.n_depth[i] = d;
            s.n_rank[i] = r;
            s.n_token[i] = tk[(d - 1) * K + r];
            int e = fsize, q = seqc;
            if (push_child) {   // best child: rank 0 of depth d+1
                s.f_score[e] = canon_score(bs + static_cast<double>(lp[d * K]));
                s.f_seq[e] = q++;
                s.f_code[e] = ((d + 1) << 16) | (0 << 8) | i;
                ++e;
            }
            if (push_sib) {     // next sibling: rank r+1 under the same parent
                s.f_score[e] = canon_score(s.n_score[p] + static_cast<double>(lp[(d - 1) * K + r + 1]));
                s.f_seq[e] = q++;
                s.f_code[e] = (d << 16) | ((r + 1) << 8) | p;
            }
        } else {
            --fsize;
        }
        fsize += static_cast<int>(push_child) + static_cast<int>(push_sib);
        seqc += static_cast<int>(push_child) + static_cast<int>(push_sib);
        __syncwarp();
    }
    const int n = count + 1;

    // children as first-child / next-sibling links (index order = rank order)
    for (int i = lane; i < n; i += 32) { s.n_first[i] = -1; s.n_next[i] = -1; s.n_last[i] = -1; }
    __syncwarp();
    if (lane == 0) {
        for (int i = 1; i < n; ++i) {
            const int p = s.n_parent[i];
            if (s.n_last[p] < 0) s.n_first[p] = i; else s.n_next[s.n_last[p]] = i;
            s.n_last[p] = i;
        }
    }
    // ancestor-or-self bitmask: vis[i] = vis[parent[i]] | bit(i), parents first
    for (int i = 0; i < n; ++i) {
        if (lane < W) {
            uint32_t v = (i == 0) ? 0u : s.n_vis[s.n_parent[i]][lane];
            if (lane == (i >> 5)) v |= 1u << (i & 31);
            s.n_vis[i][lane] = v;
        }
        __syncwarp();
    }

    const int L = ctx_len[b];
    if (L < 0 && lane == 0) report(dev_status, DDT_DEV_BAD_CTX);
    const size_t base = static_cast<size_t>(b) * N;
    for (int i = lane; i < N; i += 32) {
        const bool real = i < n;
        parent[base + i] = real ? s.n_parent[i] : -1;
        depth[base + i] = real ? s.n_depth[i] : -1;
        token[base + i] = real ? s.n_token[i] : -1;
        rank[base + i] = real ? s.n_rank[i] : -1;
        pos[base + i] = real ? L + s.n_depth[i] : -1;
        score[base + i] = real ? s.n_score[i] : -INFINITY;
        first_child[base + i] = real ? s.n_first[i] : -1;
        next_sibling[base + i] = real ? s.n_next[i] : -1;
    }
    for (int x = lane; x < N * W; x += 32) {
        const int i = x / W, w = x % W;
        vis[base * W + x] = i < n ? s.n_vis[i][w] : 0u;
    }
    if (lane == 0) n_nodes_out[b] = n;
}

cudaError_t launch_build(const float* topk_logp, const int32_t* topk_tok, const int32_t* root_tok,
                         const int32_t* ctx_len, int B, int D, int K, int budget,
                         int32_t* parent, int32_t* depth, int32_t* token, int32_t* rank,
                         int32_t* pos, double* score, int32_t* first_child,
                         int32_t* next_sibling, uint32_t* vis, int32_t* n_nodes,
                         int32_t* dev_status, cudaStream_t stream) {
    const size_t dyn = static_cast<size_t>(D) * K * 8;
    ddtree_build_kernel<<<B, 32, dyn, stream>>>(
        topk_logp, topk_tok, root_tok, ctx_len, B, D, K, budget, parent, depth, token, rank,
        pos, score, first_child, next_sibling, vis, n_nodes, dev_status);
    return cudaGetLastError();
}

}  // namespace ddt
