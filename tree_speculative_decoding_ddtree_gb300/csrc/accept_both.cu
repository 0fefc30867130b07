// ddtree_accept_greedy_sample: the greedy walk and the temperature walk of the
// same tree in one launch.
//
// Greedy: "The Architecture of Speculative Decoding: Dissecting DDTree's
// Tree-Parallel Evaluation Strategy", Section 1, step 5. Temperature: the same
// page, Section 3 (reject-sample the children in turn, descend on acceptance,
// bonus from the residual), and "The Architecture of Speculative
// Verification: Implementing Temperature-Aware Tree Sampling for DDTree",
// Path B (lazy softmax of the visited nodes only).
//
// Each walk alone is latency-bound: per level one row slice per CTA of an
// 8-CTA cluster and one cluster barrier. Here one cluster per request runs
// both walks level by level: in every round each walk still walking does its
// row pass (the greedy walk the argmax of its node's row; the temperature walk
// the softmax statistics of its node's row, or its bonus draw), and the two
// share the round's cluster barrier. When both walks stand on the same node
// the second pass over the row is served from the caches. Every pass, every
// reduction and every decision is the one ddtree_accept_greedy and
// ddtree_accept_sample make, in the same order, so the outputs are
// bit-identical to those two calls. The launch is a programmatic dependent of
// the work before it (the split-KV merge signals early); the kernel reads
// nothing before griddepcontrol.wait.
#include "walk.cuh"

namespace ddt {

// Two CTAs per SM (at most 64 registers per thread): with one, only 15 of the
// 16 eight-CTA clusters of a 16-request batch fit on the GPU at once.
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kWalkThreads, 2)
accept_both_kernel(const float* __restrict__ logits, int V, bool vec4,
                   const int32_t* __restrict__ token, const int32_t* __restrict__ first_child,
                   const int32_t* __restrict__ next_sibling, const int32_t* __restrict__ n_nodes,
                   int N, int D, const float* __restrict__ temperature, const uint64_t* __restrict__ seed,
                   uint64_t offset, WalkOut og, WalkOut os, int32_t* dev_status) {
    // a programmatic dependent of the work before it: nothing is read before
    // that work's grid has completed
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    __shared__ unsigned long long scratch_a[32];   // greedy argmax reduction
    __shared__ unsigned long long scratch_u[32];   // bonus reduction
    __shared__ float scratch_m[32];
    __shared__ float scratch_z[32];
    __shared__ float2 scratch_g[32];
    __shared__ unsigned long long part_a[2];       // this CTA's partial argmax, by round parity
    __shared__ float2 part_ms[2];                  // its partial (max, sum), by round parity
    __shared__ unsigned long long part_b;          // its partial Gumbel-max (bonus)
    __shared__ float2 part_gap;                    // its two best perturbed scores (margin output only)
    __shared__ TreeRows tr;
    __shared__ int s_kid_tok[kMaxKids];
    __shared__ int s_kid_node[kMaxKids];
    __shared__ float s_kid_logit[kMaxKids];
    __shared__ float s_q[kMaxKids];
    __shared__ double s_u[kMaxKids];
    __shared__ int s_nkids;
    __shared__ int s_gnext, s_snext;
    __shared__ int s_glen, s_grej, s_slen, s_srej;
    __shared__ float s_margin;
    const uint32_t rank = cluster_rank();
    const bool writer = rank == 0;
    const int b = static_cast<int>(blockIdx.x) / kCluster;
    const size_t tb = static_cast<size_t>(b) * N;
    const Slice sl = row_slice(V, vec4, rank);
    int32_t* gtoks = og.out_tokens + static_cast<size_t>(b) * (D + 1);
    int32_t* gnodes = og.out_nodes + static_cast<size_t>(b) * (D + 1);
    int32_t* stoks = os.out_tokens + static_cast<size_t>(b) * (D + 1);
    int32_t* snodes = os.out_nodes + static_cast<size_t>(b) * (D + 1);
    if (writer)
        for (int k = threadIdx.x; k <= D; k += kWalkThreads) {
            gtoks[k] = -1; gnodes[k] = -1; stoks[k] = -1; snodes[k] = -1;
        }
    if (threadIdx.x == 0) prefetch_slice_l2(logits + tb * static_cast<size_t>(V), vec4, sl);
    stage_tree(tr, token, first_child, next_sibling, tb, N);
    const int nn_read = n_nodes[b];
    int nn = nn_read;
    if (nn < 1 || nn > N) {
        if (threadIdx.x == 0 && writer) report(dev_status, DDT_DEV_BAD_TREE);
        nn = nn < 1 ? 1 : N;
    }
    const float T = temperature[b];
    const bool t_ok = (T > 0.0f) && isfinite(T);   // the same decision in every CTA of the cluster
    const float inv_t = t_ok ? 1.0f / T : 1.0f;
    const float s2 = inv_t * 1.4426950408889634f;   // log2(e) / T
    const uint64_t sd = seed[b];
    const uint32_t k0 = static_cast<uint32_t>(sd), k1 = static_cast<uint32_t>(sd >> 32);
    const uint32_t off_lo = static_cast<uint32_t>(offset);
    const uint32_t off_hi8 = static_cast<uint32_t>(offset >> 32) << 8;
    __syncthreads();
    if (threadIdx.x == 0) {
        s_glen = 0; s_grej = 0; s_slen = 0; s_srej = 0;
        s_margin = INFINITY;
        s_nkids = 0;
        if (writer) {
            gnodes[0] = 0;
            if (t_ok) {
                snodes[0] = 0;
            } else {
                report(dev_status, DDT_DEV_BAD_TEMPERATURE);
                os.accept_len[b] = 0;
                os.bonus[b] = -1;
                if (os.margin) os.margin[b] = NAN;
                write_stats(os, b, 0, nn_read, 0, 0);
            }
        }
    }
    int ug = 0, us = 0;
    bool g_on = true, s_on = t_ok, s_bonus = false;
    for (int round = 0;; ++round) {
        const int par = round & 1;
        const bool s_walk = s_on && !s_bonus;
        const float* grow = logits + (tb + ug) * static_cast<size_t>(V);
        const float* srow = logits + (tb + us) * static_cast<size_t>(V);
        // the temperature walk's node: its children, in rank order (thread 0, from shared memory)
        if (s_walk && threadIdx.x == 0) {
            int c = tr.fc[us], j = 0;
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
        if (s_walk && threadIdx.x < nk) {
            // child j's logit and its uniform (the uniform needs no statistics of
            // the row, so it is drawn before the round's cluster barrier)
            const int j = threadIdx.x;
            const int x = s_kid_tok[j];
            s_kid_logit[j] = (x >= 0 && x < V) ? __ldg(srow + x) : 0.0f;
            const uint4 w = philox4x32_10(make_uint4(0u | off_hi8, static_cast<uint32_t>(us),
                                                     static_cast<uint32_t>(j), off_lo), k0, k1);
            s_u[j] = uniform_exact(w.x);
        }
        // This round's row passes, in one loop so that both rows' loads are in
        // flight together (one load when both walks stand on the same node): the
        // greedy walk's argmax of its row, the temperature walk's running max and
        // softmax denominator of its row. Per thread, the same elements in the
        // same order as ddtree_accept_greedy's and ddtree_accept_sample's passes,
        // and the same reductions.
        if (g_on || s_walk) {
            const bool same = g_on && s_walk && ug == us;
            unsigned long long best = 0ull;
            SMaxSum ms{-INFINITY, 0.0f};
            auto arg = [&](float f, uint32_t v) {
                const unsigned long long pk = argmax_pack(float_order_key(f), v);
                return pk;
            };
            if (vec4) {
                const float4* g4 = reinterpret_cast<const float4*>(grow);
                const float4* s4 = reinterpret_cast<const float4*>(srow);
#pragma unroll 4
                for (int x = sl.g0 + static_cast<int>(threadIdx.x); x < sl.g1; x += kWalkThreads) {
                    float4 fg = make_float4(0.0f, 0.0f, 0.0f, 0.0f), fs = fg;
                    if (g_on) fg = __ldg(g4 + x);
                    if (s_walk) fs = same ? fg : __ldg(s4 + x);
                    if (g_on) {
                        const uint32_t v = static_cast<uint32_t>(x) << 2;
                        unsigned long long p0 = arg(fg.x, v), p1 = arg(fg.y, v + 1);
                        unsigned long long p2 = arg(fg.z, v + 2), p3 = arg(fg.w, v + 3);
                        p0 = p0 > p1 ? p0 : p1;
                        p2 = p2 > p3 ? p2 : p3;
                        p0 = p0 > p2 ? p0 : p2;
                        best = best > p0 ? best : p0;
                    }
                    if (s_walk) sms_add4(ms, fs, s2);
                }
            } else {
                for (int v = sl.g0 + static_cast<int>(threadIdx.x); v < sl.g1; v += kWalkThreads) {
                    float fg = 0.0f, fs = 0.0f;
                    if (g_on) fg = __ldg(grow + v);
                    if (s_walk) fs = same ? fg : __ldg(srow + v);
                    if (g_on) {
                        const unsigned long long p = arg(fg, static_cast<uint32_t>(v));
                        best = best > p ? best : p;
                    }
                    if (s_walk) sms_add1(ms, fs, s2);
                }
            }
            // both block reductions under one pair of barriers
            const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const unsigned long long ob = __shfl_xor_sync(0xffffffffu, best, off);
                best = best > ob ? best : ob;
                ms = sms_merge(ms, SMaxSum{__shfl_xor_sync(0xffffffffu, ms.m, off),
                                           __shfl_xor_sync(0xffffffffu, ms.z, off)});
            }
            __syncthreads();
            if (lane == 0) { scratch_a[warp] = best; scratch_m[warp] = ms.m; scratch_z[warp] = ms.z; }
            __syncthreads();
            if (warp == 0) {
                best = lane < kWalkThreads / 32 ? scratch_a[lane] : 0ull;
                ms.m = lane < kWalkThreads / 32 ? scratch_m[lane] : -INFINITY;
                ms.z = lane < kWalkThreads / 32 ? scratch_z[lane] : 0.0f;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const unsigned long long ob = __shfl_xor_sync(0xffffffffu, best, off);
                    best = best > ob ? best : ob;
                    ms = sms_merge(ms, SMaxSum{__shfl_xor_sync(0xffffffffu, ms.m, off),
                                               __shfl_xor_sync(0xffffffffu, ms.z, off)});
                }
                if (lane == 0) {
                    if (g_on) part_a[par] = best;
                    if (s_walk) part_ms[par] = make_float2(ms.m, ms.z);
                }
            }
        }
        const bool want_gap = os.margin != nullptr;
        if (s_bonus) {
            // Gumbel-max over this CTA's slice, tokens that are not children of us
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
                const uint4 w = philox4x32_10(make_uint4(1u | off_hi8, static_cast<uint32_t>(us),
                                                         static_cast<uint32_t>(x), off_lo), k0, k1);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                float f[4];
                if (vec4) {
                    const float4 t4 = __ldg(reinterpret_cast<const float4*>(srow) + x);
                    f[0] = t4.x; f[1] = t4.y; f[2] = t4.z; f[3] = t4.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) f[e] = (4 * x + e < V) ? __ldg(srow + 4 * x + e) : 0.0f;
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
                part_b = best;
                part_gap = make_float2(gap.top, gap.sec);
            }
        }
        cluster_barrier();
        // greedy: the child whose token is the target argmax at ug (one thread of
        // warp 1 in every CTA, beside the temperature walk's merge on thread 0)
        if (g_on && threadIdx.x == 32) {
            const uint32_t a = argmax_unpack_idx(cluster_max_u64(&part_a[par]));
            int match = -1, c = tr.fc[ug], guard = 0;
            while (c != -1) {
                if (c < 1 || c >= nn || ++guard > kMaxKids) {
                    if (writer) report(dev_status, DDT_DEV_BAD_TREE);
                    break;
                }
                if (tr.tok[c] == static_cast<int32_t>(a)) { match = c; break; }
                ++s_grej;
                c = tr.ns[c];
            }
            const int len = s_glen;
            if (match != -1 && len >= D) {
                if (writer) report(dev_status, DDT_DEV_BAD_TREE);
                match = -1;
            }
            if (match != -1) {
                if (writer) {
                    gtoks[len] = tr.tok[match];
                    gnodes[len + 1] = match;
                }
                s_glen = len + 1;
            } else if (writer) {
                gtoks[len] = static_cast<int32_t>(a);
                og.bonus[b] = static_cast<int32_t>(a);
                og.accept_len[b] = len;
                write_stats(og, b, len, nn_read, len + 1, s_grej);
            }
            s_gnext = match;
        }
        if (s_walk && threadIdx.x < 32) {
            // warp 0 alone: the same partials merged by the same shuffle tree in
            // every CTA, lane 0's result on every lane, q(x_j) of child j on lane j
            // (at most 32 children), then the decision on lane 0
            SMaxSum acc = sms_cluster(&part_ms[par]);
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
            // children in rank order: accept child j when u_j * R < q(x_j)
            if (threadIdx.x == 0) {
                int match = -1;
                double R = 1.0;
                for (int j = 0; j < nk; ++j) {
                    if (os.margin && R > 0.0)
                        s_margin = fminf(s_margin, fabsf(static_cast<float>(s_u[j]) - s_q[j] / static_cast<float>(R)));
                    if (s_u[j] * R < static_cast<double>(s_q[j])) { match = s_kid_node[j]; break; }
                    R -= static_cast<double>(s_q[j]);
                    ++s_srej;
                }
                const int len = s_slen;
                if (match != -1 && len >= D) {
                    if (writer) report(dev_status, DDT_DEV_BAD_TREE);
                    match = -1;
                }
                if (match != -1) {
                    if (writer) {
                        stoks[len] = tr.tok[match];
                        snodes[len + 1] = match;
                    }
                    s_slen = len + 1;
                }
                s_snext = match;
            }
        }
        if (s_bonus && threadIdx.x == 0 && writer) {
            const unsigned long long all = cluster_max_u64(&part_b);
            const int len = s_slen;
            const int32_t a = all ? static_cast<int32_t>(argmax_unpack_idx(all)) : -1;
            stoks[len] = a;
            os.bonus[b] = a;
            os.accept_len[b] = len;
            if (want_gap) os.margin[b] = fminf(s_margin, cluster_gap(&part_gap));
            write_stats(os, b, len, nn_read, len + (a >= 0 ? 1 : 0), s_srej);
        }
        __syncthreads();
        if (g_on) {
            ug = s_gnext;
            if (ug == -1) g_on = false;
        }
        if (s_walk) {
            if (s_snext != -1) us = s_snext;
            else s_bonus = true;
        } else if (s_bonus) {
            s_on = false;
            s_bonus = false;
        }
        if (!g_on && !s_on) break;
    }
    cluster_barrier();   // peers may still be reading this CTA's partials
}

cudaError_t launch_accept_both(const float* logits, int V, const int32_t* token, const int32_t* first_child,
                               const int32_t* next_sibling, const int32_t* n_nodes, int B, int N, int D,
                               const float* temperature, const uint64_t* seed, uint64_t offset,
                               const WalkOut& og, const WalkOut& os, int32_t* dev_status, cudaStream_t stream) {
    const bool vec4 = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B) * kCluster);
    cfg.blockDim = dim3(kWalkThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, accept_both_kernel, logits, V, vec4, token, first_child, next_sibling,
                              n_nodes, N, D, temperature, seed, offset, og, os, dev_status);
}

}  // namespace ddt
