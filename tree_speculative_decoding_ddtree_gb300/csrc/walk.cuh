// Device helpers shared by the verify walks (greedy, sampled, draft-ratio):
// thread-block cluster primitives, Philox4x32-10, block reductions, the
// per-CTA vocabulary slices and the staged tree rows.
#pragma once

#include "common.cuh"

namespace ddt {

constexpr int kCluster = 8;               // CTAs per request (portable cluster size)
constexpr int kWalkThreads = 512;
constexpr int kMaxKids = DDT_MAX_TOPK;

// ---------------------------------------------------------------------------
// cluster helpers
// ---------------------------------------------------------------------------
DDT_DEVINL uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
// every thread of every CTA of the cluster; orders shared-memory writes before
// the barrier with reads after it, cluster-wide
DDT_DEVINL void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// shared::cluster address of the same variable in CTA `rank`
DDT_DEVINL uint32_t cluster_addr(const void* p, uint32_t rank) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
DDT_DEVINL unsigned long long ld_cluster_u64(uint32_t addr) {
    unsigned long long v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];\n" : "=l"(v) : "r"(addr) : "memory");
    return v;
}
DDT_DEVINL double ld_cluster_f64(uint32_t addr) {
    double v;
    asm volatile("ld.shared::cluster.f64 %0, [%1];\n" : "=d"(v) : "r"(addr) : "memory");
    return v;
}
DDT_DEVINL float2 ld_cluster_f32x2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];\n" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}

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

// Gumbel noise g = -log(-log U) for the Philox word w, U = ((w >> 8) + 0.5) 2^-24.
// E = -log U comes from the hardware base-2 logarithm (absolute error about
// 2^-22.6), at most about 2^-20 relative wherever 1 - U > 1/8 (|log2 U| >=
// 0.19 there; U itself is rounded to fp32, a further 2^-22 relative); for
// 1 - U = x <= 1/8, where those errors would grow, from the series
// x + x^2/2 + ... + x^8/8 of -log(1 - x), x exact in fp32 (truncation below
// 2^-26 relative). Then g = -log E from the base-2 logarithm again. Both forms
// of E are computed and one selected, so no warp diverges. Worst case over all
// 2^24 values of U: |g - exact| below 2e-6 (checked exhaustively against fp64
// in the tests).
DDT_DEVINL float gumbel_noise(uint32_t w) {
    constexpr float kLn2 = 0.69314718055994531f;
    const uint32_t k = w >> 8;
    const float u = (static_cast<float>(k) + 0.5f) * 0x1p-24f;
    // 1 - U: exact when U >= 1/2 (k >= 2^23), the only case it is used in
    const float x = (static_cast<float>((1u << 24) - 1u - k) + 0.5f) * 0x1p-24f;
    float t = fmaf(x, 0.125f, 1.0f / 7.0f);
    t = fmaf(x, t, 1.0f / 6.0f);
    t = fmaf(x, t, 0.2f);
    t = fmaf(x, t, 0.25f);
    t = fmaf(x, t, 1.0f / 3.0f);
    t = fmaf(x, t, 0.5f);
    t = fmaf(x, t, 1.0f);
    const float e_series = x * t;
    const float e_log = -__log2f(u) * kLn2;
    const float e = (k >= (1u << 23) && x <= 0.125f) ? e_series : e_log;
    return -__log2f(e) * kLn2;
}

DDT_DEVINL double uniform_exact(uint32_t w) {
    return (static_cast<double>(w >> 8) + 0.5) * 0x1p-24;
}

// block-wide reductions over kWalkThreads threads; every thread gets the result
template <typename T, typename Op>
DDT_DEVINL T block_reduce(T v, T* scratch, Op op, T identity) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    if (warp == 0) {
        T x = lane < kWalkThreads / 32 ? scratch[lane] : identity;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x = op(x, __shfl_xor_sync(0xffffffffu, x, o));
        if (lane == 0) scratch[0] = x;
    }
    __syncthreads();
    return scratch[0];
}

struct MaxU64 { DDT_DEVINL unsigned long long operator()(unsigned long long a, unsigned long long b) const { return a > b ? a : b; } };

// This CTA's slice of a row: float4 groups [g0, g1) when the row is read as
// float4, else elements [g0, g1).
struct Slice {
    int g0, g1;
};
DDT_DEVINL Slice row_slice(int V, bool vec4, uint32_t rank) {
    const int n = vec4 ? (V >> 2) : V;
    Slice s;
    s.g0 = static_cast<int>((static_cast<long long>(n) * rank) / kCluster);
    s.g1 = static_cast<int>((static_cast<long long>(n) * (rank + 1)) / kCluster);
    return s;
}

// Ask L2 for this CTA's slice of the root's logits row, which every walk reads
// first, while the tree is staged (a hint: nothing waits for it). The range is
// trimmed to 16-byte boundaries inside the slice, as the bulk prefetch needs.
DDT_DEVINL void prefetch_slice_l2(const float* row, bool vec4, Slice sl) {
    const uintptr_t unit = vec4 ? 16 : 4;
    const uintptr_t lo = (reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(sl.g0) * unit + 15) &
                         ~static_cast<uintptr_t>(15);
    const uintptr_t hi = (reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(sl.g1) * unit) &
                         ~static_cast<uintptr_t>(15);
    if (hi > lo)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n"
                     :: "l"(lo), "r"(static_cast<uint32_t>(hi - lo)) : "memory");
}

// argmax of this CTA's slice (largest value, lowest index, NaN lowest), packed
DDT_DEVINL unsigned long long slice_argmax(const float* __restrict__ row, bool vec4, Slice sl,
                                           unsigned long long* scratch) {
    unsigned long long best = 0ull;
    if (vec4) {
        const float4* r4 = reinterpret_cast<const float4*>(row);
#pragma unroll 4
        for (int x = sl.g0 + static_cast<int>(threadIdx.x); x < sl.g1; x += kWalkThreads) {
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
        for (int v = sl.g0 + static_cast<int>(threadIdx.x); v < sl.g1; v += kWalkThreads) {
            const unsigned long long p = argmax_pack(float_order_key(__ldg(row + v)), v);
            best = best > p ? best : p;
        }
    }
    return block_reduce(best, scratch, MaxU64(), 0ull);
}

// max over the cluster's partials (slot `part` in every CTA)
DDT_DEVINL unsigned long long cluster_max_u64(const unsigned long long* part) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int r = 0; r < kCluster; ++r) {
        const unsigned long long v = ld_cluster_u64(cluster_addr(part, r));
        best = best > v ? best : v;
    }
    return best;
}

struct WalkOut {
    int32_t* accept_len;
    int32_t* out_tokens;
    int32_t* out_nodes;
    int32_t* bonus;
    float* margin;        // nullable [B]: smallest decision margin on the path
    int32_t* stats;       // nullable [B, 4]: accepted depth, nodes built, tokens emitted,
                          //                  child tests that rejected (or did not match)
};

// Write one request's walk statistics (writer CTA, one thread).
DDT_DEVINL void write_stats(const WalkOut& o, int b, int len, int n_nodes, int emitted, int rejected) {
    if (!o.stats) return;
    int32_t* st = o.stats + static_cast<size_t>(b) * 4;
    st[0] = len;
    st[1] = n_nodes;
    st[2] = emitted;
    st[3] = rejected;
}

// ---------------------------------------------------------------------------
// The bonus draw's decision margin: the gap between the best and the
// runner-up perturbed score. Each thread keeps the two largest scores it saw
// (only when a caller asked for margins); pairs merge by (max of the tops,
// max of the smaller top and the runner-ups).
// ---------------------------------------------------------------------------
struct Gap2 {
    float top, sec;
};
DDT_DEVINL void gap2_add(Gap2& g, float sc) {
    g.sec = fmaxf(g.sec, fminf(g.top, sc));
    g.top = fmaxf(g.top, sc);
}
DDT_DEVINL Gap2 gap2_merge(Gap2 x, Gap2 y) {
    return Gap2{fmaxf(x.top, y.top), fmaxf(fminf(x.top, y.top), fmaxf(x.sec, y.sec))};
}
// block-wide merge over kWalkThreads threads; thread 0 gets the result
DDT_DEVINL Gap2 block_gap2(Gap2 g, float2* scratch /* [32] */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        g = gap2_merge(g, Gap2{__shfl_xor_sync(0xffffffffu, g.top, o), __shfl_xor_sync(0xffffffffu, g.sec, o)});
    __syncthreads();
    if (lane == 0) scratch[warp] = make_float2(g.top, g.sec);
    __syncthreads();
    if (warp == 0) {
        const float2 v = lane < kWalkThreads / 32 ? scratch[lane] : make_float2(-INFINITY, -INFINITY);
        g = Gap2{v.x, v.y};
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            g = gap2_merge(g, Gap2{__shfl_xor_sync(0xffffffffu, g.top, o), __shfl_xor_sync(0xffffffffu, g.sec, o)});
    }
    return g;
}
// merge of the cluster's partials (float2 `part` in every CTA, rank order): the gap
DDT_DEVINL float cluster_gap(const float2* part) {
    Gap2 g{-INFINITY, -INFINITY};
#pragma unroll
    for (int r = 0; r < kCluster; ++r) {
        const float2 v = ld_cluster_f32x2(cluster_addr(part, r));
        g = gap2_merge(g, Gap2{v.x, v.y});
    }
    return g.sec == -INFINITY ? INFINITY : g.top - g.sec;
}

// The request's token / first-child / next-sibling rows, staged in shared
// memory so the serial child scans never wait on global memory.
struct TreeRows {
    int tok[DDT_MAX_NODES];
    int fc[DDT_MAX_NODES];
    int ns[DDT_MAX_NODES];
};

DDT_DEVINL void stage_tree(TreeRows& t, const int32_t* token, const int32_t* first_child,
                           const int32_t* next_sibling, size_t tb, int N) {
    for (int i = threadIdx.x; i < N; i += kWalkThreads) {
        t.tok[i] = token[tb + i];
        t.fc[i] = first_child[tb + i];
        t.ns[i] = next_sibling[tb + i];
    }
}

// online (max, sum of exp((x - max) / T)) pair
struct MaxSum {
    float m, z;
};

DDT_DEVINL MaxSum merge_ms(MaxSum a, MaxSum b, float inv_t) {
    const float M = fmaxf(a.m, b.m);
    MaxSum r;
    r.m = M;
    r.z = (M == -INFINITY) ? 0.0f : a.z * expf((a.m - M) * inv_t) + b.z * expf((b.m - M) * inv_t);
    return r;
}

// ---------------------------------------------------------------------------
// The temperature walk's softmax statistics of a row in the exp2 domain:
// m = the largest x * s (s = log2(e) / T > 0, the rounded product), z = the
// sum over the row of 2^(x * s - m), each exponent one fused multiply-add
// (so its error is relative to the difference, as for exp((x - max) / T))
// and each power one ex2.approx. Merges and the children's probabilities use
// the same units: q(x) = 2^(x * s - m) / z.
// ---------------------------------------------------------------------------
DDT_DEVINL float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
struct SMaxSum {
    float m, z;
};
DDT_DEVINL SMaxSum sms_merge(SMaxSum a, SMaxSum b) {
    const float M = fmaxf(a.m, b.m);
    if (M == -INFINITY) return SMaxSum{-INFINITY, 0.0f};
    return SMaxSum{M, a.z * ex2_approx(a.m - M) + b.z * ex2_approx(b.m - M)};
}
// four elements at a time: one rescale at most, four fused exponents
DDT_DEVINL void sms_add4(SMaxSum& a, float4 f, float s) {
    const float mx = fmaxf(fmaxf(f.x, f.y), fmaxf(f.z, f.w)) * s;
    if (mx > a.m) {
        a.z = a.z * ex2_approx(a.m - mx);
        a.m = mx;
    }
    if (a.m == -INFINITY) return;
    a.z += (ex2_approx(fmaf(f.x, s, -a.m)) + ex2_approx(fmaf(f.y, s, -a.m))) +
           (ex2_approx(fmaf(f.z, s, -a.m)) + ex2_approx(fmaf(f.w, s, -a.m)));
}
DDT_DEVINL void sms_add1(SMaxSum& a, float f, float s) {
    const float mx = f * s;
    if (mx > a.m) {
        a.z = a.z * ex2_approx(a.m - mx);
        a.m = mx;
    }
    if (a.m == -INFINITY) return;
    a.z += ex2_approx(fmaf(f, s, -a.m));
}
// block-wide merge over kWalkThreads threads (fixed shuffle tree); warp 0 holds the result
DDT_DEVINL SMaxSum sms_block(SMaxSum ms, float* scratch_m, float* scratch_z) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        ms = sms_merge(ms, SMaxSum{__shfl_xor_sync(0xffffffffu, ms.m, off), __shfl_xor_sync(0xffffffffu, ms.z, off)});
    __syncthreads();
    if (lane == 0) { scratch_m[warp] = ms.m; scratch_z[warp] = ms.z; }
    __syncthreads();
    if (warp == 0) {
        ms.m = lane < kWalkThreads / 32 ? scratch_m[lane] : -INFINITY;
        ms.z = lane < kWalkThreads / 32 ? scratch_z[lane] : 0.0f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            ms = sms_merge(ms, SMaxSum{__shfl_xor_sync(0xffffffffu, ms.m, off), __shfl_xor_sync(0xffffffffu, ms.z, off)});
    }
    return ms;
}
// the cluster's partials (float2 `part` in every CTA), merged by a fixed
// shuffle tree over lanes 0..kCluster-1 of warp 0 (call from all of warp 0);
// every CTA gets the same result
DDT_DEVINL SMaxSum sms_cluster(const float2* part) {
    const int lane = threadIdx.x & 31;
    SMaxSum ms{-INFINITY, 0.0f};
    if (lane < kCluster) {
        const float2 v = ld_cluster_f32x2(cluster_addr(part, static_cast<uint32_t>(lane)));
        ms = SMaxSum{v.x, v.y};
    }
#pragma unroll
    for (int off = kCluster / 2; off > 0; off >>= 1)
        ms = sms_merge(ms, SMaxSum{__shfl_xor_sync(0xffffffffu, ms.m, off), __shfl_xor_sync(0xffffffffu, ms.z, off)});
    return ms;
}

}  // namespace ddt
