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
// One CTA per request walks the tree; only the logits rows of visited nodes
// are read, each streamed once per pass with 16-byte loads, eight in flight
// per thread so a row costs about one memory round trip.
#include "common.cuh"

namespace ddt {

constexpr int kAcceptThreads = 1024;
constexpr int kMaxKids = DDT_MAX_TOPK;

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., SC'11): two multiply-xor lanes per round,
// key bumped by the Weyl constants between rounds.
// ---------------------------------------------------------------------------
DDT_DEVINL uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
    constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) { k0 += W0; k1 += W1; }
        const uint32_t hi0 = __umulhi(M0, c.x), lo0 = M0 * c.x;
        const uint32_t hi1 = __umulhi(M1, c.z), lo1 = M1 * c.z;
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}

// -log(U) for U = ((w >> 8) + 0.5) * 2^-24, accurate in fp32 on both halves of
// (0, 1): log of U below one half, log1p of -(1 - U) above it.
DDT_DEVINL float neg_log_uniform(uint32_t w) {
    const uint32_t k = w >> 8;
    if (k < (1u << 23)) return -logf((static_cast<float>(k) + 0.5f) * 0x1p-24f);
    const float one_minus_u = (static_cast<float>((1u << 24) - 1u - k) + 0.5f) * 0x1p-24f;
    return -log1pf(-one_minus_u);
}

DDT_DEVINL double uniform_exact(uint32_t w) {
    return (static_cast<double>(w >> 8) + 0.5) * 0x1p-24;
}

// block-wide reductions over kAcceptThreads threads; every thread gets the result
template <typename T, typename Op>
DDT_DEVINL T block_reduce(T v, T* scratch, Op op, T identity) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    if (warp == 0) {
        T x = lane < kAcceptThreads / 32 ? scratch[lane] : identity;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x = op(x, __shfl_xor_sync(0xffffffffu, x, o));
        if (lane == 0) scratch[0] = x;
    }
    __syncthreads();
    return scratch[0];
}

struct MaxU64 { DDT_DEVINL unsigned long long operator()(unsigned long long a, unsigned long long b) const { return a > b ? a : b; } };
struct MaxF { DDT_DEVINL float operator()(float a, float b) const { return fmaxf(a, b); } };
struct SumF { DDT_DEVINL float operator()(float a, float b) const { return a + b; } };

// argmax of one row (largest value, lowest index, NaN lowest)
DDT_DEVINL uint32_t row_argmax(const float* __restrict__ row, int V, bool vec4,
                               unsigned long long* scratch) {
    unsigned long long best = 0ull;
    if (vec4) {
        const float4* r4 = reinterpret_cast<const float4*>(row);
#pragma unroll 8
        for (int x = threadIdx.x; x < (V >> 2); x += kAcceptThreads) {
            const float4 f = __ldg(r4 + x);
            const uint32_t v = static_cast<uint32_t>(x) << 2;
            unsigned long long p0 = argmax_pack(float_order_key(f.x), v);
            unsigned long long p1 = argmax_pack(float_order_key(f.y), v + 1);
            unsigned long long p2 = argmax_pack(float_order_key(f.z), v + 2);
            unsigned long long p3 = argmax_pack(float_order_key(f.w), v + 3);
            p0 = p0 > p1 ? p0 : p1;
            p2 = p2 > p3 ? p2 : p3;
            p0 = p0 > p2 ? p0 : p2;
            best = best > p0 ? best : p0;
        }
    } else {
        for (int v = threadIdx.x; v < V; v += kAcceptThreads) {
            const unsigned long long p = argmax_pack(float_order_key(__ldg(row + v)), v);
            best = best > p ? best : p;
        }
    }
    best = block_reduce(best, scratch, MaxU64(), 0ull);
    return argmax_unpack_idx(best);
}

struct WalkOut {
    int32_t* accept_len;
    int32_t* out_tokens;
    int32_t* out_nodes;
    int32_t* bonus;
};

// The request's token / first-child / next-sibling rows, staged in shared
// memory so the serial child scans never wait on global memory.
struct TreeRows {
    int tok[DDT_MAX_NODES];
    int fc[DDT_MAX_NODES];
    int ns[DDT_MAX_NODES];
};

DDT_DEVINL void stage_tree(TreeRows& t, const int32_t* token, const int32_t* first_child,
                           const int32_t* next_sibling, size_t tb, int N) {
    for (int i = threadIdx.x; i < N; i += kAcceptThreads) {
        t.tok[i] = token[tb + i];
        t.fc[i] = first_child[tb + i];
        t.ns[i] = next_sibling[tb + i];
    }
}

__global__ void __launch_bounds__(kAcceptThreads)
accept_greedy_kernel(const float* __restrict__ logits, int V, bool vec4,
                     const int32_t* __restrict__ token, const int32_t* __restrict__ first_child,
                     const int32_t* __restrict__ next_sibling, const int32_t* __restrict__ n_nodes,
                     int N, int D, WalkOut o, int32_t* dev_status) {
    __shared__ unsigned long long scratch[32];
    __shared__ TreeRows tr;
    __shared__ int s_next;
    __shared__ int s_len;
    const int b = blockIdx.x;
    const size_t tb = static_cast<size_t>(b) * N;
    int32_t* toks = o.out_tokens + static_cast<size_t>(b) * (D + 1);
    int32_t* nodes = o.out_nodes + static_cast<size_t>(b) * (D + 1);
    for (int k = threadIdx.x; k <= D; k += kAcceptThreads) { toks[k] = -1; nodes[k] = -1; }
    stage_tree(tr, token, first_child, next_sibling, tb, N);
    int nn = n_nodes[b];
    if (nn < 1 || nn > N) {
        if (threadIdx.x == 0) report(dev_status, DDT_DEV_BAD_TREE);
        nn = nn < 1 ? 1 : N;
    }
    if (threadIdx.x == 0) s_len = 0;
    __syncthreads();
    if (threadIdx.x == 0) nodes[0] = 0;
    int u = 0;
    while (true) {
        const uint32_t a = row_argmax(logits + (tb + u) * static_cast<size_t>(V), V, vec4, scratch);
        if (threadIdx.x == 0) {
            int match = -1, c = tr.fc[u], guard = 0;
            while (c != -1) {
                if (c < 1 || c >= nn || ++guard > kMaxKids) { report(dev_status, DDT_DEV_BAD_TREE); break; }
                if (tr.tok[c] == static_cast<int32_t>(a)) { match = c; break; }
                c = tr.ns[c];
            }
            const int len = s_len;
            if (match != -1 && len >= D) { report(dev_status, DDT_DEV_BAD_TREE); match = -1; }
            if (match != -1) {
                toks[len] = tr.tok[match];
                nodes[len + 1] = match;
                s_len = len + 1;
            } else {
                toks[len] = static_cast<int32_t>(a);
                o.bonus[b] = static_cast<int32_t>(a);
                o.accept_len[b] = len;
            }
            s_next = match;
        }
        __syncthreads();
        u = s_next;
        if (u == -1) break;
    }
}

// online (max, sum of exp((x - max) / T)) pair, merged in a block reduction
struct MaxSum {
    float m, z;
};

__global__ void __launch_bounds__(kAcceptThreads)
accept_sample_kernel(const float* __restrict__ logits, int V, bool vec4,
                     const int32_t* __restrict__ token, const int32_t* __restrict__ first_child,
                     const int32_t* __restrict__ next_sibling, const int32_t* __restrict__ n_nodes,
                     int N, int D, const float* __restrict__ temperature,
                     const uint64_t* __restrict__ seed, uint64_t offset, WalkOut o,
                     int32_t* dev_status) {
    __shared__ unsigned long long scratch_u[32];
    __shared__ float scratch_m[32];
    __shared__ float scratch_z[32];
    __shared__ TreeRows tr;
    __shared__ int s_kid_tok[kMaxKids];
    __shared__ int s_kid_node[kMaxKids];
    __shared__ float s_q[kMaxKids];
    __shared__ double s_u[kMaxKids];
    __shared__ int s_nkids;
    __shared__ int s_next;
    __shared__ int s_len;
    const int b = blockIdx.x;
    const size_t tb = static_cast<size_t>(b) * N;
    int32_t* toks = o.out_tokens + static_cast<size_t>(b) * (D + 1);
    int32_t* nodes = o.out_nodes + static_cast<size_t>(b) * (D + 1);
    for (int k = threadIdx.x; k <= D; k += kAcceptThreads) { toks[k] = -1; nodes[k] = -1; }
    stage_tree(tr, token, first_child, next_sibling, tb, N);
    int nn = n_nodes[b];
    if (nn < 1 || nn > N) {
        if (threadIdx.x == 0) report(dev_status, DDT_DEV_BAD_TREE);
        nn = nn < 1 ? 1 : N;
    }
    const float T = temperature[b];
    __syncthreads();
    if (!(T > 0.0f) || !isfinite(T)) {
        if (threadIdx.x == 0) {
            report(dev_status, DDT_DEV_BAD_TEMPERATURE);
            o.accept_len[b] = 0;
            o.bonus[b] = -1;
        }
        return;
    }
    const float inv_t = 1.0f / T;
    const uint64_t sd = seed[b];
    const uint32_t k0 = static_cast<uint32_t>(sd), k1 = static_cast<uint32_t>(sd >> 32);
    const uint32_t off_lo = static_cast<uint32_t>(offset);
    const uint32_t off_hi8 = static_cast<uint32_t>(offset >> 32) << 8;
    if (threadIdx.x == 0) { s_len = 0; nodes[0] = 0; }
    int u = 0;
    while (true) {
        const float* row = logits + (tb + u) * static_cast<size_t>(V);
        // the node's children, in rank order (thread 0, from shared memory)
        if (threadIdx.x == 0) {
            int c = tr.fc[u], j = 0;
            while (c != -1) {
                if (c < 1 || c >= nn || j >= kMaxKids) { report(dev_status, DDT_DEV_BAD_TREE); break; }
                s_kid_node[j] = c;
                s_kid_tok[j] = tr.tok[c];
                ++j;
                c = tr.ns[c];
            }
            s_nkids = j;
        }
        // one pass: running max and softmax denominator of logits / T
        float m = -INFINITY, z = 0.0f;
        auto add = [&](float x) {
            if (x > m) {
                z = z * expf((m - x) * inv_t) + 1.0f;
                m = x;
            } else {
                z += expf((x - m) * inv_t);
            }
        };
        if (vec4) {
            const float4* r4 = reinterpret_cast<const float4*>(row);
#pragma unroll 8
            for (int x = threadIdx.x; x < (V >> 2); x += kAcceptThreads) {
                const float4 f = __ldg(r4 + x);
                add(f.x); add(f.y); add(f.z); add(f.w);
            }
        } else {
            for (int v = threadIdx.x; v < V; v += kAcceptThreads) add(__ldg(row + v));
        }
        {
            const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
                const float z2 = __shfl_xor_sync(0xffffffffu, z, off);
                const float M = fmaxf(m, m2);
                z = (M == -INFINITY) ? 0.0f : z * expf((m - M) * inv_t) + z2 * expf((m2 - M) * inv_t);
                m = M;
            }
            __syncthreads();
            if (lane == 0) { scratch_m[warp] = m; scratch_z[warp] = z; }
            __syncthreads();
            if (warp == 0) {
                m = lane < kAcceptThreads / 32 ? scratch_m[lane] : -INFINITY;
                z = lane < kAcceptThreads / 32 ? scratch_z[lane] : 0.0f;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
                    const float z2 = __shfl_xor_sync(0xffffffffu, z, off);
                    const float M = fmaxf(m, m2);
                    z = (M == -INFINITY) ? 0.0f : z * expf((m - M) * inv_t) + z2 * expf((m2 - M) * inv_t);
                    m = M;
                }
                if (lane == 0) { scratch_m[0] = m; scratch_z[0] = z; }
            }
            __syncthreads();
            m = scratch_m[0];
            z = scratch_z[0];
        }
        // child j: q(x_j) and its uniform, one thread each
        const int nk = s_nkids;
        if (threadIdx.x < nk) {
            const int j = threadIdx.x;
            const int x = s_kid_tok[j];
            float q = 0.0f;
            if (x >= 0 && x < V) q = expf((row[x] - m) * inv_t) / z;
            else report(dev_status, DDT_DEV_BAD_TOKEN);
            const uint4 w = philox4x32_10(make_uint4(0u | off_hi8, static_cast<uint32_t>(u),
                                                     static_cast<uint32_t>(j), off_lo), k0, k1);
            s_q[j] = q;
            s_u[j] = uniform_exact(w.x);
        }
        __syncthreads();
        // children in rank order: accept child j when u_j * R < q(x_j)
        if (threadIdx.x == 0) {
            int match = -1;
            double R = 1.0;
            for (int j = 0; j < nk; ++j) {
                if (s_u[j] * R < static_cast<double>(s_q[j])) { match = s_kid_node[j]; break; }
                R -= static_cast<double>(s_q[j]);
            }
            const int len = s_len;
            if (match != -1 && len >= D) { report(dev_status, DDT_DEV_BAD_TREE); match = -1; }
            if (match != -1) {
                toks[len] = tr.tok[match];
                nodes[len + 1] = match;
                s_len = len + 1;
            }
            s_next = match;
        }
        __syncthreads();
        const int nxt = s_next;
        if (nxt != -1) { u = nxt; continue; }
        // bonus: Gumbel-max over tokens that are not children of u
        unsigned long long best = 0ull;
        const int groups = (V + 3) >> 2;
#pragma unroll 4
        for (int x = threadIdx.x; x < groups; x += kAcceptThreads) {
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
                if (v >= V) break;
                bool kid = false;
                for (int k = 0; k < nk; ++k) kid |= (s_kid_tok[k] == v);
                if (kid) continue;
                const float g = -logf(neg_log_uniform(ws[e]));
                const float sc = f[e] * inv_t + g;
                const unsigned long long p = argmax_pack(float_order_key(sc), static_cast<uint32_t>(v));
                best = best > p ? best : p;
            }
        }
        best = block_reduce(best, scratch_u, MaxU64(), 0ull);
        if (threadIdx.x == 0) {
            const int len = s_len;
            const int32_t a = best ? static_cast<int32_t>(argmax_unpack_idx(best)) : -1;
            toks[len] = a;
            o.bonus[b] = a;
            o.accept_len[b] = len;
        }
        break;
    }
}

cudaError_t launch_accept_greedy(const float* logits, int V, const int32_t* token,
                                 const int32_t* first_child, const int32_t* next_sibling,
                                 const int32_t* n_nodes, int B, int N, int D,
                                 int32_t* accept_len, int32_t* out_tokens, int32_t* out_nodes,
                                 int32_t* bonus, int32_t* dev_status, cudaStream_t stream) {
    const bool vec4 = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
    WalkOut o{accept_len, out_tokens, out_nodes, bonus};
    accept_greedy_kernel<<<B, kAcceptThreads, 0, stream>>>(logits, V, vec4, token, first_child,
                                                           next_sibling, n_nodes, N, D, o, dev_status);
    return cudaGetLastError();
}

cudaError_t launch_accept_sample(const float* logits, int V, const int32_t* token,
                                 const int32_t* first_child, const int32_t* next_sibling,
                                 const int32_t* n_nodes, int B, int N, int D,
                                 const float* temperature, const uint64_t* seed, uint64_t offset,
                                 int32_t* accept_len, int32_t* out_tokens, int32_t* out_nodes,
                                 int32_t* bonus, int32_t* dev_status, cudaStream_t stream) {
    const bool vec4 = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
    WalkOut o{accept_len, out_tokens, out_nodes, bonus};
    accept_sample_kernel<<<B, kAcceptThreads, 0, stream>>>(logits, V, vec4, token, first_child,
                                                           next_sibling, n_nodes, N, D, temperature,
                                                           seed, offset, o, dev_status);
    return cudaGetLastError();
}

}  // namespace ddt
