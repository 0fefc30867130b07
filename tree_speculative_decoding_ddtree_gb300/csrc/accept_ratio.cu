// ddtree_accept_sample_ratio: the temperature walk with the draft-ratio rule.
//
// Method: "The Architecture of Speculative Decoding: Dissecting DDTree's
// Tree-Parallel Evaluation Strategy", Section 3 (linear case: accept draft
// token t with probability min(1, p_target(t) / p_draft(t)), else resample
// from the residual; tree case: reject-sample the children, bonus from the
// residual) and "The Architecture of Speculative Verification: Implementing
// Temperature-Aware Tree Sampling for DDTree", The Knowledge Required, item 3.
// p = softmax(draft row d / T) for the children of a depth-d node and
// q = softmax(target row / T). Children are tested in rank order against a
// residual r that starts at q; after a rejection r <- normalise(max(r - p, 0)).
// Written out, r = max(q - c p, 0) / R with c = 0, R = 1 at first and, after
// each rejection, c <- c + R and R <- sum_v max(q(v) - c p(v), 0): a rejection
// costs one pass over both rows. Child j (token x) is accepted when
// U_j * p(x) < r(x). The bonus is the Gumbel-max of log max(q - c p, 0); if
// the residual has no mass left the bonus is drawn from q.
//
// Precision: q and p are fp32 (softmax statistics in the exp2 domain, each
// power one ex2.approx of a fused multiply-add, fp32 sums); c and R are
// fp64 scalars (R summed in fp64 across the threads' fp32 partials), and
// every residual q - c p is formed with one fused multiply-add on the high
// part of c (the low part's product subtracted after), so the subtraction
// adds no rounding beyond that of its result. What remains is the fp32 error
// of q and p themselves, which a rejection chain amplifies by (1 + c) / R:
// that conditioning is the problem's, not the formula's.
//
// Same layout as the other walks: one 8-CTA cluster per request; every pass
// over a row is split into the CTAs' slices and combined through distributed
// shared memory in rank order, so every CTA holds identical values and takes
// identical decisions; CTA 0 writes the outputs.
#include "walk.cuh"

namespace ddt {

namespace {

enum ChildState { kAccept = 1, kReject = 2, kSkip = 3 };

// block-wide sum of one float per thread (every thread gets the result)
DDT_DEVINL float block_sum_f(float v, float* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum_f(v);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float x = lane < kWalkThreads / 32 ? scratch[lane] : 0.0f;
        x = warp_sum_f(x);
        if (lane == 0) scratch[0] = x;
    }
    __syncthreads();
    return scratch[0];
}

}  // namespace

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kWalkThreads)
accept_ratio_kernel(const float* __restrict__ logits, const float* __restrict__ draft, int V, bool vec4,
                    const int32_t* __restrict__ token, const int32_t* __restrict__ first_child,
                    const int32_t* __restrict__ next_sibling, const int32_t* __restrict__ n_nodes,
                    int N, int D, const float* __restrict__ temperature,
                    const uint64_t* __restrict__ seed, uint64_t offset, WalkOut o, int32_t* dev_status) {
    __shared__ unsigned long long scratch_u[32];
    __shared__ float scratch_a[32], scratch_b[32];
    __shared__ float2 scratch_g[32];
    __shared__ float4 part_s[2];                // (max, sum) of the target and the draft row, by round
    __shared__ double part_r[2];                // residual mass, by round (the cluster sums it in fp64)
    __shared__ unsigned long long part_g[2];    // Gumbel-max, by round
    __shared__ float2 part_gap[2];              // two best perturbed scores, by round (margin output only)
    __shared__ TreeRows tr;
    __shared__ int s_kid_tok[kMaxKids];
    __shared__ int s_kid_node[kMaxKids];
    __shared__ float s_kid_l[kMaxKids];         // target logit of the child's token
    __shared__ float s_kid_d[kMaxKids];         // draft logit of the child's token
    __shared__ double s_u[kMaxKids];
    __shared__ float s_mq, s_zq, s_mp, s_zp;
    __shared__ double s_R, s_c;                 // thread 0's fp64 residual mass and offset
    __shared__ float s_chi, s_clo;              // c = s_chi + s_clo for every thread
    __shared__ int s_rpos;                      // the residual still has mass
    __shared__ float s_margin;
    __shared__ unsigned long long s_best;
    __shared__ float s_gap;
    __shared__ int s_nkids, s_state, s_next, s_len, s_rej;
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
    const float s2 = inv_t * 1.4426950408889634f;   // log2(e) / T: the statistics' exp2 units
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
    int round = 0;   // cluster reductions so far: partial slots alternate by its parity
    int u = 0;
    for (;;) {
        const float* row = logits + (tb + u) * static_cast<size_t>(V);
        if (threadIdx.x == 0) {   // the node's children, in rank order
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
            if (j > 0 && s_len >= D) {   // a depth-D node has no children
                if (writer) report(dev_status, DDT_DEV_BAD_TREE);
                j = 0;
            }
            s_nkids = j;
        }
        __syncthreads();
        const int nk = s_nkids;
        const int len = s_len;
        const float* drow = draft + (static_cast<size_t>(b) * D + (nk > 0 ? len : 0)) * static_cast<size_t>(V);
        if (threadIdx.x < nk) {   // the children's logits and uniforms, one thread each
            const int j = threadIdx.x;
            const int x = s_kid_tok[j];
            const bool ok = x >= 0 && x < V;
            s_kid_l[j] = ok ? __ldg(row + x) : 0.0f;
            s_kid_d[j] = ok ? __ldg(drow + x) : 0.0f;
            const uint4 w = philox4x32_10(make_uint4(0u | off_hi8, static_cast<uint32_t>(u),
                                                     static_cast<uint32_t>(j), off_lo), k0, k1);
            s_u[j] = uniform_exact(w.x);
        }
        // pass 1: softmax statistics (exp2 domain) of the target row and, with
        // children, of the draft row
        SMaxSum mq{-INFINITY, 0.0f}, mp{-INFINITY, 0.0f};
        if (vec4) {
            const float4* r4 = reinterpret_cast<const float4*>(row);
            const float4* d4 = reinterpret_cast<const float4*>(drow);
#pragma unroll 2
            for (int x = sl.g0 + static_cast<int>(threadIdx.x); x < sl.g1; x += kWalkThreads) {
                sms_add4(mq, __ldg(r4 + x), s2);
                if (nk > 0) sms_add4(mp, __ldg(d4 + x), s2);
            }
        } else {
            for (int v = sl.g0 + static_cast<int>(threadIdx.x); v < sl.g1; v += kWalkThreads) {
                sms_add1(mq, __ldg(row + v), s2);
                if (nk > 0) sms_add1(mp, __ldg(drow + v), s2);
            }
        }
        mq = sms_block(mq, scratch_a, scratch_b);
        mp = sms_block(mp, scratch_a, scratch_b);
        if (threadIdx.x == 0) part_s[round & 1] = make_float4(mq.m, mq.z, mp.m, mp.z);
        cluster_barrier();
        if (threadIdx.x == 0) {   // the same partials merged in the same order in every CTA
            SMaxSum aq{-INFINITY, 0.0f}, ap{-INFINITY, 0.0f};
#pragma unroll
            for (int r = 0; r < kCluster; ++r) {
                const uint32_t a = cluster_addr(&part_s[round & 1], r);
                const float2 q2 = ld_cluster_f32x2(a);
                const float2 p2 = ld_cluster_f32x2(a + 8);
                aq = sms_merge(aq, SMaxSum{q2.x, q2.y});
                ap = sms_merge(ap, SMaxSum{p2.x, p2.y});
            }
            s_mq = aq.m; s_zq = aq.z; s_mp = ap.m; s_zp = ap.z;
            s_c = 0.0;
            s_R = 1.0;
        }
        ++round;
        __syncthreads();
        const float Mq = s_mq, rZq = 1.0f / s_zq, Mp = s_mp, rZp = nk > 0 ? 1.0f / s_zp : 0.0f;
        // children in rank order against the residual max(q - c p, 0) / R; thread 0
        // keeps c and R in fp64 and hands every thread c = c_hi + c_lo, the
        // residuals take fmaf on c_hi
        float c_hi = 0.0f, c_lo = 0.0f;
        auto resid = [&](float qv, float pv) { return fmaxf(fmaf(-c_hi, pv, qv) - c_lo * pv, 0.0f); };
        // the residual of vocabulary entry v from its target and draft logits
        auto qp = [&](float l, float d) {
            return resid(ex2_approx(fmaf(l, s2, -Mq)) * rZq, ex2_approx(fmaf(d, s2, -Mp)) * rZp);
        };
        int match = -1;
        for (int j = 0; j < nk; ++j) {
            if (threadIdx.x == 0) {
                int st;
                const int x = s_kid_tok[j];
                if (x < 0 || x >= V) {
                    if (writer) report(dev_status, DDT_DEV_BAD_TOKEN);
                    st = kSkip;
                } else {
                    const float qx = ex2_approx(fmaf(s_kid_l[j], s2, -Mq)) * rZq;
                    const float px = ex2_approx(fmaf(s_kid_d[j], s2, -Mp)) * rZp;
                    const double R = s_R;
                    const float ru = resid(qx, px);   // R r(x): the test U p(x) < r(x) without a divide
                    if (o.margin && px > 0.0f)        // fp32 is enough for the report
                        s_margin = fminf(s_margin, fabsf(static_cast<float>(s_u[j]) - ru / (px * static_cast<float>(R))));
                    st = s_u[j] * static_cast<double>(px) * R < static_cast<double>(ru) ? kAccept : kReject;
                    if (st == kReject) {
                        s_c += R;
                        s_chi = static_cast<float>(s_c);
                        s_clo = static_cast<float>(s_c - static_cast<double>(s_chi));
                    }
                    if (st == kReject) ++s_rej;
                }
                s_state = st;
            }
            __syncthreads();
            const int st = s_state;
            __syncthreads();   // every thread has read s_state before thread 0 writes it again
            if (st == kAccept) { match = s_kid_node[j]; break; }
            if (st == kSkip) continue;
            c_hi = s_chi;
            c_lo = s_clo;
            // the residual's mass for the next test, or to confirm the bonus has one
            float part = 0.0f;
            if (vec4) {
                const float4* r4 = reinterpret_cast<const float4*>(row);
                const float4* d4 = reinterpret_cast<const float4*>(drow);
#pragma unroll 1   // each thread takes about two groups per pass; unrolling only adds registers
                for (int x = sl.g0 + static_cast<int>(threadIdx.x); x < sl.g1; x += kWalkThreads) {
                    const float4 f = __ldg(r4 + x), g = __ldg(d4 + x);
                    part += qp(f.x, g.x) + qp(f.y, g.y) + qp(f.z, g.z) + qp(f.w, g.w);
                }
            } else {
                for (int v = sl.g0 + static_cast<int>(threadIdx.x); v < sl.g1; v += kWalkThreads)
                    part += qp(__ldg(row + v), __ldg(drow + v));
            }
            part = block_sum_f(part, scratch_a);
            if (threadIdx.x == 0) part_r[round & 1] = static_cast<double>(part);
            cluster_barrier();
            if (threadIdx.x == 0) {   // in rank order: the same sum in every CTA
                double all = 0.0;
#pragma unroll
                for (int r = 0; r < kCluster; ++r) all += ld_cluster_f64(cluster_addr(&part_r[round & 1], r));
                s_R = all;
                s_rpos = all > 0.0;
            }
            ++round;
            __syncthreads();
            if (!s_rpos) {   // no residual mass left: the bonus comes from q
                c_hi = c_lo = 0.0f;
                break;
            }
        }
        if (threadIdx.x == 0) {
            const int l0 = s_len;
            if (match != -1) {
                if (writer) {
                    toks[l0] = tr.tok[match];
                    nodes[l0 + 1] = match;
                }
                s_len = l0 + 1;
            }
            s_next = match;
        }
        __syncthreads();
        if (s_next != -1) { u = s_next; continue; }
        // bonus: Gumbel-max of log max(q - c p, 0) over this CTA's slice; if no
        // token keeps residual mass, once more with c = 0 (from q)
        const bool want_gap = o.margin != nullptr;
        for (;;) {
        const bool from_resid = c_hi > 0.0f;   // else from q
        unsigned long long best = 0ull;
        Gap2 gap{-INFINITY, -INFINITY};
        const int g0 = vec4 ? sl.g0 : (sl.g0 >> 2), g1 = vec4 ? sl.g1 : ((sl.g1 + 3) >> 2);
#pragma unroll 2
        for (int x = g0 + static_cast<int>(threadIdx.x); x < g1; x += kWalkThreads) {
            const uint4 w = philox4x32_10(make_uint4(1u | off_hi8, static_cast<uint32_t>(u),
                                                     static_cast<uint32_t>(x), off_lo), k0, k1);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
            float f[4], d[4];
            if (vec4) {
                const float4 t4 = __ldg(reinterpret_cast<const float4*>(row) + x);
                f[0] = t4.x; f[1] = t4.y; f[2] = t4.z; f[3] = t4.w;
                if (from_resid) {
                    const float4 d4 = __ldg(reinterpret_cast<const float4*>(drow) + x);
                    d[0] = d4.x; d[1] = d4.y; d[2] = d4.z; d[3] = d4.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int v = 4 * x + e;
                    f[e] = v < V ? __ldg(row + v) : 0.0f;
                    d[e] = (v < V && from_resid) ? __ldg(drow + v) : 0.0f;
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int v = 4 * x + e;
                if (v >= V || (!vec4 && (v < sl.g0 || v >= sl.g1))) continue;
                float sc;
                if (from_resid) {
                    const float r = qp(f[e], d[e]);
                    if (!(r > 0.0f)) continue;
                    sc = logf(r);
                } else {
                    sc = f[e] * inv_t;   // log q up to a constant (as the renormalising walk's bonus)
                }
                sc += gumbel_noise(ws[e]);
                const unsigned long long pk = argmax_pack(float_order_key(sc), static_cast<uint32_t>(v));
                best = best > pk ? best : pk;
                if (want_gap) gap2_add(gap, sc);
            }
        }
        best = block_reduce(best, scratch_u, MaxU64(), 0ull);
        if (want_gap) gap = block_gap2(gap, scratch_g);
        if (threadIdx.x == 0) {
            part_g[round & 1] = best;
            part_gap[round & 1] = make_float2(gap.top, gap.sec);
        }
        cluster_barrier();
        if (threadIdx.x == 0) {
            s_best = cluster_max_u64(&part_g[round & 1]);
            if (want_gap) s_gap = cluster_gap(&part_gap[round & 1]);
        }
        ++round;
        __syncthreads();
        if (s_best == 0ull && from_resid) {
            c_hi = c_lo = 0.0f;
            continue;
        }
        break;
        }
        if (threadIdx.x == 0 && writer) {
            const unsigned long long all = s_best;
            const int l0 = s_len;
            const int32_t a = all ? static_cast<int32_t>(argmax_unpack_idx(all)) : -1;
            toks[l0] = a;
            o.bonus[b] = a;
            o.accept_len[b] = l0;
            if (want_gap) o.margin[b] = fminf(s_margin, s_gap);
            write_stats(o, b, l0, nn_read, l0 + (a >= 0 ? 1 : 0), s_rej);
        }
        break;
    }
    cluster_barrier();   // peers may still be reading this CTA's partials
}

cudaError_t launch_accept_ratio(const float* logits, const float* draft_logits, int V, const int32_t* token,
                                const int32_t* first_child, const int32_t* next_sibling,
                                const int32_t* n_nodes, int B, int N, int D, const float* temperature,
                                const uint64_t* seed, uint64_t offset, int32_t* accept_len,
                                int32_t* out_tokens, int32_t* out_nodes, int32_t* bonus,
                                float* margin_stats, int32_t* walk_stats, int32_t* dev_status,
                                cudaStream_t stream) {
    const bool vec4 = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0) &&
                      (reinterpret_cast<uintptr_t>(draft_logits) % 16 == 0);
    WalkOut o{accept_len, out_tokens, out_nodes, bonus, margin_stats, walk_stats};
    accept_ratio_kernel<<<B * kCluster, kWalkThreads, 0, stream>>>(
        logits, draft_logits, V, vec4, token, first_child, next_sibling, n_nodes, N, D, temperature, seed,
        offset, o, dev_status);
    return cudaGetLastError();
}

}  // namespace ddt
