// ddtree_accept_greedy / ddtree_accept_sample: the verify walks.
//
// Greedy: "The Architecture of Speculative Decoding: Dissecting DDTree's
// Tree-Parallel Evaluation Strategy", Section 1, step 5 (follow the target
// argmax into the matching child; the argmax at the last node is the bonus).
// Temperature: the same page, Section 3 (tree case: reject-sample the children
// in turn, descend on acceptance, bonus from the residual), and "The
// Architecture of Speculative Verification: Implementing Temperature-Aware
// Tree Sampling for DDTree", Path B (lazy softmax of the visited nodes only).
//
// One cluster of kCluster CTAs per request walks the tree. Only the logits
// rows of visited nodes are read. Every pass over a row (argmax; running max
// and softmax denominator; the Gumbel-max bonus) is split over the cluster:
// CTA r streams slice r of the vocabulary with 16-byte loads, reduces it in
// the block, and publishes one partial in its shared memory; after a cluster
// barrier every CTA reads the kCluster partials through distributed shared
// memory and combines them in rank order, so all CTAs hold the same result
// and take the same step. The walk itself (child match, rejection tests) is
// done by every CTA on identical values; CTA 0 writes the outputs. Per level
// this costs one row slice (a memory round trip) and one cluster barrier,
// instead of streaming the whole row through one SM.
#include "walk.cuh"

namespace ddt {

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kWalkThreads)
accept_greedy_kernel(const float* __restrict__ logits, int V, bool vec4,
                     const int32_t* __restrict__ token, const int32_t* __restrict__ first_child,
                     const int32_t* __restrict__ next_sibling, const int32_t* __restrict__ n_nodes,
                     int N, int D, WalkOut o, int32_t* dev_status) {
    __shared__ unsigned long long scratch[32];
    __shared__ unsigned long long part[2];      // this CTA's partial argmax, by level parity
    __shared__ TreeRows tr;
    __shared__ int s_next;
    __shared__ int s_len;
    __shared__ int s_rej;
    const uint32_t rank = cluster_rank();
    const bool writer = rank == 0;
    const int b = static_cast<int>(blockIdx.x) / kCluster;
    const size_t tb = static_cast<size_t>(b) * N;
    const Slice sl = row_slice(V, vec4, rank);
    int32_t* toks = o.out_tokens + static_cast<size_t>(b) * (D + 1);
    int32_t* nodes = o.out_nodes + static_cast<size_t>(b) * (D + 1);
    if (writer)
        for (int k = threadIdx.x; k <= D; k += kWalkThreads) { toks[k] = -1; nodes[k] = -1; }
    if (threadIdx.x == 0) prefetch_slice_l2(logits + tb * static_cast<size_t>(V), vec4, sl);
    stage_tree(tr, token, first_child, next_sibling, tb, N);
    const int nn_read = n_nodes[b];
    int nn = nn_read;
    if (nn < 1 || nn > N) {
        if (threadIdx.x == 0 && writer) report(dev_status, DDT_DEV_BAD_TREE);
        nn = nn < 1 ? 1 : N;
    }
    if (threadIdx.x == 0) { s_len = 0; s_rej = 0; }
    __syncthreads();
    if (threadIdx.x == 0 && writer) nodes[0] = 0;
    int u = 0;
    for (int level = 0;; ++level) {
        const unsigned long long mine = slice_argmax(logits + (tb + u) * static_cast<size_t>(V), vec4, sl, scratch);
        if (threadIdx.x == 0) part[level & 1] = mine;
        cluster_barrier();
        if (threadIdx.x == 0) {
            // the same partials in the same order in every CTA: the same argmax
            const uint32_t a = argmax_unpack_idx(cluster_max_u64(&part[level & 1]));
            int match = -1, c = tr.fc[u], guard = 0;
            while (c != -1) {
                if (c < 1 || c >= nn || ++guard > kMaxKids) {
                    if (writer) report(dev_status, DDT_DEV_BAD_TREE);
                    break;
                }
                if (tr.tok[c] == static_cast<int32_t>(a)) { match = c; break; }
                ++s_rej;
                c = tr.ns[c];
            }
            const int len = s_len;
            if (match != -1 && len >= D) {
                if (writer) report(dev_status, DDT_DEV_BAD_TREE);
                match = -1;
            }
            if (match != -1) {
                if (writer) {
                    toks[len] = tr.tok[match];
                    nodes[len + 1] = match;
                }
                s_len = len + 1;
            } else if (writer) {
                toks[len] = static_cast<int32_t>(a);
                o.bonus[b] = static_cast<int32_t>(a);
                o.accept_len[b] = len;
                write_stats(o, b, len, nn_read, len + 1, s_rej);
            }
            s_next = match;
        }
        __syncthreads();
        u = s_next;
        if (u == -1) break;
    }
    cluster_barrier();   // peers may still be reading this CTA's partials
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kWalkThreads)
accept_sample_kernel(const float* __restrict__ logits, int V, bool vec4,
                     const int32_t* __restrict__ token, const int32_t* __restrict__ first_child,
                     const int32_t* __restrict__ next_sibling, const int32_t* __restrict__ n_nodes,
                     int N, int D, const float* __restrict__ temperature,
                     const uint64_t* __restrict__ seed, uint64_t offset, WalkOut o,
                     int32_t* dev_status) {
    __shared__ unsigned long long scratch_u[32];
    __shared__ float scratch_m[32];
    __shared__ float scratch_z[32];
    __shared__ float2 scratch_g[32];
    __shared__ float2 part_ms[2];               // this CTA's partial (max, sum), by level parity
    __shared__ unsigned long long part_g;       // this CTA's partial Gumbel-max (bonus)
    __shared__ float2 part_gap;                 // its two best perturbed scores (margin output only)
    __shared__ TreeRows tr;
    __shared__ int s_kid_tok[kMaxKids];
    __shared__ int s_kid_node[kMaxKids];
    __shared__ float s_kid_logit[kMaxKids];
    __shared__ float s_q[kMaxKids];
    __shared__ double s_u[kMaxKids];
    __shared__ int s_nkids;
    __shared__ int s_next;
    __shared__ int s_len;
    __shared__ int s_rej;
    __shared__ float s_margin;
    const uint32_t rank = cluster_rank();
    const bool writer = rank == 0;
    const int b = static_cast<int>(blockIdx.x) / kCluster;
    const size_t tb = static_cast<size_t>(b) * N;
    const Slice sl = row_slice(V, vec4, rank);
    int32_t* toks = o.out_tokens + static_cast<size_t>(b) * (D + 1);
    int32_t* nodes = o.out_nodes + static_cast<size_t>(b) * (D + 1);
    if (writer)
        for (int k = threadIdx.x; k <= D; k += kWalkThreads) { toks[k] = -1; nodes[k] = -1; }
    if (threadIdx.x == 0) prefetch_slice_l2(logits + tb * static_cast<size_t>(V), vec4, sl);
    stage_tree(tr, token, first_child, next_sibling, tb, N);
    const int nn_read = n_nodes[b];
    int nn = nn_read;
    if (nn < 1 || nn > N) {
        if (threadIdx.x == 0 && writer) report(dev_status, DDT_DEV_BAD_TREE);
        nn = nn < 1 ? 1 : N;
    }
    const float T = temperature[b];
    __syncthreads();
    if (!(T > 0.0f) || !isfinite(T)) {   // the same decision in every CTA of the cluster
        if (threadIdx.x == 0 && writer) {
            report(dev_status, DDT_DEV_BAD_TEMPERATURE);
            o.accept_len[b] = 0;
            o.bonus[b] = -1;
            if (o.margin) o.margin[b] = NAN;
            write_stats(o, b, 0, nn_read, 0, 0);
        }
        return;
    }
    const float inv_t = 1.0f / T;
    const float s2 = inv_t * 1.4426950408889634f;   // log2(e) / T
    const uint64_t sd = seed[b];
    const uint32_t k0 = static_cast<uint32_t>(sd), k1 = static_cast<uint32_t>(sd >> 32);
    const uint32_t off_lo = static_cast<uint32_t>(offset);
    const uint32_t off_hi8 = static_cast<uint32_t>(offset >> 32) << 8;
    if (threadIdx.x == 0) {
        s_len = 0;
        s_rej = 0;
        s_margin = INFINITY;
        if (writer) nodes[0] = 0;
    }
    int u = 0;
    for (int level = 0;; ++level) {
        const float* row = logits + (tb + u) * static_cast<size_t>(V);
        // the node's children, in rank order (thread 0, from shared memory)
        if (threadIdx.x == 0) {
            int c = tr.fc[u], j = 0;
            while (c != -1) {
                if (c < 1 || c >= nn || j >= kMaxKids) {
                    if (writer) report(dev_status, DDT_DEV_BAD_TREE);
                    break;
                }
                s_kid_node[j] = c;
                s_kid_tok[j] = tr.tok[c];
                ++j;
                c = tr.ns[c];
            }
            s_nkids = j;
        }
        __syncthreads();
        const int nk = s_nkids;
        // the children's logits are fetched while the slice streams, and their
        // uniforms drawn (they need no statistics of the row)
        if (threadIdx.x < nk) {
            const int j = threadIdx.x;
            const int x = s_kid_tok[j];
            s_kid_logit[j] = (x >= 0 && x < V) ? __ldg(row + x) : 0.0f;
            const uint4 w = philox4x32_10(make_uint4(0u | off_hi8, static_cast<uint32_t>(u),
                                                     static_cast<uint32_t>(j), off_lo), k0, k1);
            s_u[j] = uniform_exact(w.x);
        }
        // this CTA's slice: softmax statistics of logits / T in the exp2 domain
        SMaxSum ms{-INFINITY, 0.0f};
        if (vec4) {
            const float4* r4 = reinterpret_cast<const float4*>(row);
#pragma unroll 4
            for (int x = sl.g0 + static_cast<int>(threadIdx.x); x < sl.g1; x += kWalkThreads)
                sms_add4(ms, __ldg(r4 + x), s2);
        } else {
            for (int v = sl.g0 + static_cast<int>(threadIdx.x); v < sl.g1; v += kWalkThreads)
                sms_add1(ms, __ldg(row + v), s2);
        }
        ms = sms_block(ms, scratch_m, scratch_z);
        if (threadIdx.x == 0) part_ms[level & 1] = make_float2(ms.m, ms.z);
        cluster_barrier();
        if (threadIdx.x < 32) {
            // warp 0 alone: the same partials merged by the same shuffle tree in
            // every CTA, lane 0's result on every lane, q(x_j) of child j on lane j
            // (at most 32 children), then the decision on lane 0
            SMaxSum acc = sms_cluster(&part_ms[level & 1]);
            acc.m = __shfl_sync(0xffffffffu, acc.m, 0);
            acc.z = __shfl_sync(0xffffffffu, acc.z, 0);
            if (threadIdx.x < nk) {
                const int j = threadIdx.x;
                const int x = s_kid_tok[j];
                float q = 0.0f;
                if (x >= 0 && x < V) q = ex2_approx(fmaf(s_kid_logit[j], s2, -acc.m)) / acc.z;
                else if (writer) report(dev_status, DDT_DEV_BAD_TOKEN);
                s_q[j] = q;
            }
            __syncwarp();
        }
        // children in rank order: accept child j when u_j * R < q(x_j)
        if (threadIdx.x == 0) {
            int match = -1;
            double R = 1.0;
            for (int j = 0; j < nk; ++j) {
                if (o.margin && R > 0.0)   // fp32 is enough for the report; no fp64 divide on the walk's path
                    s_margin = fminf(s_margin, fabsf(static_cast<float>(s_u[j]) - s_q[j] / static_cast<float>(R)));
                if (s_u[j] * R < static_cast<double>(s_q[j])) { match = s_kid_node[j]; break; }
                R -= static_cast<double>(s_q[j]);
                ++s_rej;
            }
            const int len = s_len;
            if (match != -1 && len >= D) {
                if (writer) report(dev_status, DDT_DEV_BAD_TREE);
                match = -1;
            }
            if (match != -1) {
                if (writer) {
                    toks[len] = tr.tok[match];
                    nodes[len + 1] = match;
                }
                s_len = len + 1;
            }
            s_next = match;
        }
        __syncthreads();
        const int nxt = s_next;
        if (nxt != -1) { u = nxt; continue; }
        // bonus: Gumbel-max over this CTA's slice, tokens that are not children of u
        // (with a margin output, the two best scores too: their gap is the draw's margin)
        const bool want_gap = o.margin != nullptr;
        unsigned long long best = 0ull;
        Gap2 gap{-INFINITY, -INFINITY};
        const int g0 = vec4 ? sl.g0 : (sl.g0 >> 2), g1 = vec4 ? sl.g1 : ((sl.g1 + 3) >> 2);
        // does any child's token fall in this thread's groups of four (x = g0 + tid + 512 i)?
        bool kid_here = false;
        for (int k = 0; k < nk; ++k) {
            const int xk = s_kid_tok[k] >> 2;
            kid_here |= xk >= g0 && xk < g1 && (xk - g0 - static_cast<int>(threadIdx.x)) % kWalkThreads == 0;
        }
#pragma unroll 2
        for (int x = g0 + static_cast<int>(threadIdx.x); x < g1; x += kWalkThreads) {
            const uint4 w = philox4x32_10(make_uint4(1u | off_hi8, static_cast<uint32_t>(u),
                                                     static_cast<uint32_t>(x), off_lo), k0, k1);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
            float f[4];
            if (vec4) {
                const float4 t4 = __ldg(reinterpret_cast<const float4*>(row) + x);
                f[0] = t4.x; f[1] = t4.y; f[2] = t4.z; f[3] = t4.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) f[e] = (4 * x + e < V) ? __ldg(row + 4 * x + e) : 0.0f;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int v = 4 * x + e;
                // element slices: this CTA owns [g0, g1) of the elements only
                if (v >= V || (!vec4 && (v < sl.g0 || v >= sl.g1))) continue;
                if (kid_here) {   // only threads holding a child's token look for it
                    bool kid = false;
                    for (int k = 0; k < nk; ++k) kid |= (s_kid_tok[k] == v);
                    if (kid) continue;
                }
                const float g = gumbel_noise(ws[e]);
                const float sc = f[e] * inv_t + g;
                const unsigned long long pk = argmax_pack(float_order_key(sc), static_cast<uint32_t>(v));
                best = best > pk ? best : pk;
                if (want_gap) gap2_add(gap, sc);
            }
        }
        best = block_reduce(best, scratch_u, MaxU64(), 0ull);
        if (want_gap) gap = block_gap2(gap, scratch_g);
        if (threadIdx.x == 0) {
            part_g = best;
            part_gap = make_float2(gap.top, gap.sec);
        }
        cluster_barrier();
        if (threadIdx.x == 0 && writer) {
            const unsigned long long all = cluster_max_u64(&part_g);
            const int len = s_len;
            const int32_t a = all ? static_cast<int32_t>(argmax_unpack_idx(all)) : -1;
            toks[len] = a;
            o.bonus[b] = a;
            o.accept_len[b] = len;
            if (want_gap) o.margin[b] = fminf(s_margin, cluster_gap(&part_gap));
            write_stats(o, b, len, nn_read, len + (a >= 0 ? 1 : 0), s_rej);
        }
        break;
    }
    cluster_barrier();   // peers may still be reading this CTA's partials
}

cudaError_t launch_accept_greedy(const float* logits, int V, const int32_t* token,
                                 const int32_t* first_child, const int32_t* next_sibling,
                                 const int32_t* n_nodes, int B, int N, int D,
                                 int32_t* accept_len, int32_t* out_tokens, int32_t* out_nodes,
                                 int32_t* bonus, int32_t* walk_stats, int32_t* dev_status,
                                 cudaStream_t stream) {
    const bool vec4 = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
    WalkOut o{accept_len, out_tokens, out_nodes, bonus, nullptr, walk_stats};
    accept_greedy_kernel<<<B * kCluster, kWalkThreads, 0, stream>>>(logits, V, vec4, token, first_child,
                                                                    next_sibling, n_nodes, N, D, o, dev_status);
    return cudaGetLastError();
}

cudaError_t launch_accept_sample(const float* logits, int V, const int32_t* token,
                                 const int32_t* first_child, const int32_t* next_sibling,
                                 const int32_t* n_nodes, int B, int N, int D,
                                 const float* temperature, const uint64_t* seed, uint64_t offset,
                                 int32_t* accept_len, int32_t* out_tokens, int32_t* out_nodes,
                                 int32_t* bonus, float* margin_stats, int32_t* walk_stats,
                                 int32_t* dev_status, cudaStream_t stream) {
    const bool vec4 = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
    WalkOut o{accept_len, out_tokens, out_nodes, bonus, margin_stats, walk_stats};
    accept_sample_kernel<<<B * kCluster, kWalkThreads, 0, stream>>>(logits, V, vec4, token, first_child,
                                                                    next_sibling, n_nodes, N, D, temperature,
                                                                    seed, offset, o, dev_status);
    return cudaGetLastError();
}

// gumbel_noise of every word (the testing entry point's exhaustive check)
__global__ void gumbel_probe_kernel(const uint32_t* __restrict__ words, float* __restrict__ out, size_t n) {
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        out[i] = gumbel_noise(words[i]);
}

cudaError_t launch_gumbel_probe(const uint32_t* words, float* out, size_t n, cudaStream_t stream) {
    const size_t blocks = (n + 255) / 256;
    gumbel_probe_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(words, out, n);
    return cudaGetLastError();
}

}  // namespace ddt
