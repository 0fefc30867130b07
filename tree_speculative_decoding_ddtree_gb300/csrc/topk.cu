// ddtree_draft_topk: per-depth top-K tokens of the draft and their log-probs.
//
// Method: "The Architecture of Speculative Decoding: Dissecting DDTree's
// Tree-Parallel Evaluation Strategy", Section 1 (The Five-Step Flow of
// DDTree), step 1: from each depth position of the single draft forward, the
// top-k candidate tokens are taken with their log-probs; "The Tree That
// Couldn't Branch", Hypothesis 4 (one row per depth serves every node).
// Ranking is by the logit (the log-prob order), ties to the lower token id;
// log-prob = logit - log(sum exp(logits)) of the row.
//
// One CTA per (request, depth) row; the row is read once from HBM.
//  Pass A: every thread streams its share of the row (16-byte loads, several
//    in flight) keeping an online (max, sum of exp(x - max)) pair for the
//    log-sum-exp; the max with its lowest id is the thread's best element. A key packs the logit's
//    order key above the inverted token id, so a larger key is a larger logit
//    or, on a tie, a lower id; NaN ranks below every number.
//  Threshold: T = the K-th largest of the threads' best keys (a bitonic sort
//    per warp, then ranks across warps). At least K elements have a key >= T,
//    so every element of the top K has a key >= T and sits in a thread whose
//    best key is >= T: exactly K threads, keys being distinct.
//  Pass B: the warps re-read those threads' shares (from L2, one unit per
//    lane) and stage the elements with key >= T in shared memory; the K largest staged keys, ranked by
//    counting, are the answer. Rows with more candidates than the staging
//    array holds (many equal logits) take a slower exact path instead: a
//    sorted top-K list per warp, updated by ballot and shift, then merged.
// The exp-sum is accumulated and combined in fp32; the log-probs are formed
// as logit - (max + log(sum)) in fp64, then rounded to fp32.
#include "common.cuh"

namespace ddt {

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkCap = 1024;   // staged candidate keys
constexpr int kTopkUnroll = 4;   // loads in flight per thread (4 measured best of 4, 8, 16)

// descending bitonic sort of one key per lane across the warp
DDT_DEVINL unsigned long long warp_sort_desc(unsigned long long v, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, j);
            const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
            v = keep_max ? (o > v ? o : v) : (o < v ? o : v);
        }
    return v;
}

// insert key k into the warp's sorted list (lanes 0..K-1, descending); k is
// larger than the K-th key and differs from every key in the list
DDT_DEVINL void list_insert(unsigned long long& list, unsigned long long k, int K, int lane) {
    const int pos = __popc(__ballot_sync(0xffffffffu, lane < K && list > k));
    const unsigned long long up = __shfl_up_sync(0xffffffffu, list, 1);
    if (lane < K) list = lane < pos ? list : (lane == pos ? k : up);
}

// offer one key per lane to the warp's list; thr tracks the K-th key
DDT_DEVINL void list_offer(unsigned long long& list, unsigned long long& thr, unsigned long long key,
                           int K, int lane) {
    unsigned int m = __ballot_sync(0xffffffffu, key > thr);
    while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        const unsigned long long k = __shfl_sync(0xffffffffu, key, src);
        if (k > thr) {   // warp-uniform
            list_insert(list, k, K, lane);
            thr = __shfl_sync(0xffffffffu, list, K - 1);
        }
    }
}

// The calling thread's share of the row: units (one float4, or one float)
// first + it * kTopkThreads * kU + j * 32 for j < kU. fn(f, g) sees each group
// of kU loaded units, g[j] the unit index (>= n_units: absent, f = -inf).
template <int kL, int kU, class Fn>
DDT_DEVINL void scan_share(const float* __restrict__ x, int n_units, int first, Fn&& fn) {
    for (int base = first; base < n_units; base += kTopkThreads * kU) {
        float f[kU][kL];
        int g[kU];
#pragma unroll
        for (int j = 0; j < kU; ++j) {
            g[j] = base + j * 32;
            if (g[j] < n_units) {
                if constexpr (kL == 4) {
                    const float4 t = __ldg(reinterpret_cast<const float4*>(x) + g[j]);
                    f[j][0] = t.x; f[j][1] = t.y; f[j][2] = t.z; f[j][3] = t.w;
                } else {
                    f[j][0] = __ldg(x + g[j]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < kL; ++e) f[j][e] = -INFINITY;   // adds nothing to the sum
            }
        }
        fn(f, g);
    }
}

// ranks of the first K entries of each warp's descending list among all lists
// (an entry's own list counts its p predecessors): one binary search per list,
// all lists stepped together; calls out(rank, key) for every non-zero entry
template <class Out>
DDT_DEVINL void rank_lists(const unsigned long long (*keys)[32], int K, Out&& out) {
    if (threadIdx.x < kTopkWarps * K) {
        const int w = threadIdx.x / K, p = threadIdx.x - w * K;
        const unsigned long long c = keys[w][p];
        int pos[kTopkWarps];
#pragma unroll
        for (int w2 = 0; w2 < kTopkWarps; ++w2) pos[w2] = 0;
#pragma unroll
        for (int step = 16; step > 0; step >>= 1)
#pragma unroll
            for (int w2 = 0; w2 < kTopkWarps; ++w2)
                pos[w2] += keys[w2][pos[w2] + step - 1] > c ? step : 0;
        // the steps reach 0..31; a list with all 32 keys above c counts 32
        int rank = 0;
#pragma unroll
        for (int w2 = 0; w2 < kTopkWarps; ++w2) rank += pos[w2] + (keys[w2][pos[w2]] > c ? 1 : 0);
        if (c != 0ull) out(rank, c);
    }
}

template <int kL>
__global__ void __launch_bounds__(kTopkThreads)
draft_topk_kernel(const float* __restrict__ logits, int V, int K, float* __restrict__ out_lp,
                  int32_t* __restrict__ out_tok) {
    constexpr int kU = kTopkUnroll;
    __shared__ unsigned long long s_keys[kTopkWarps][32];
    __shared__ unsigned long long s_cand[kTopkCap];
    __shared__ float s_m[kTopkWarps], s_s[kTopkWarps];
    __shared__ int s_nan[kTopkWarps];
    __shared__ uint32_t s_win[32];
    __shared__ int s_sel[32];
    __shared__ unsigned long long s_T;
    __shared__ int s_count;
    __shared__ double s_lse;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t row = blockIdx.x;
    const float* x = logits + row * static_cast<size_t>(V);
    const int n_units = V / kL;
    const int first = warp * 32 * kU + lane;

    // pass A: exp-sum, and the thread's best element (the exp-sum's running
    // max; its lowest id is searched for only when a group raises the max)
    float m = -INFINITY, s = 0.0f;
    bool nan = false;
    uint32_t best_i = 0u;
    scan_share<kL, kU>(x, n_units, first, [&](const float (&f)[kU][kL], const int (&g)[kU]) {
        float mj[kL];   // kL independent chains; fmaxf skips NaN
#pragma unroll
        for (int e = 0; e < kL; ++e) mj[e] = f[0][e];
#pragma unroll
        for (int j = 1; j < kU; ++j)
#pragma unroll
            for (int e = 0; e < kL; ++e) mj[e] = fmaxf(mj[e], f[j][e]);
        float mloc = mj[0];
#pragma unroll
        for (int e = 1; e < kL; ++e) mloc = fmaxf(mloc, mj[e]);
        if (mloc > m) {
            bool found = false;   // the first (lowest id) element equal to the new max
#pragma unroll
            for (int j = 0; j < kU; ++j)
#pragma unroll
                for (int e = 0; e < kL; ++e)
                    if (!found && f[j][e] == mloc) {
                        found = true;
                        best_i = static_cast<uint32_t>(g[j] * kL + e);
                    }
            s = s != 0.0f ? s * __expf(m - mloc) : 0.0f;
            m = mloc;
        }
        if (m != -INFINITY) {
            float t[kL];   // kL independent chains; a NaN makes the sum NaN
#pragma unroll
            for (int e = 0; e < kL; ++e) t[e] = __expf(f[0][e] - m);
#pragma unroll
            for (int j = 1; j < kU; ++j)
#pragma unroll
                for (int e = 0; e < kL; ++e) t[e] += __expf(f[j][e] - m);
#pragma unroll
            for (int e = 1; e < kL; ++e) t[0] += t[e];
            s += t[0];
        } else {
#pragma unroll
            for (int j = 0; j < kU; ++j)
#pragma unroll
                for (int e = 0; e < kL; ++e) nan |= f[j][e] != f[j][e];
        }
    });
    unsigned long long my_key = 0ull;
    if (m != -INFINITY) {
        my_key = argmax_pack(float_order_key(m), best_i);
    } else if (first < n_units) {
        // every element of the share is -inf or NaN: the best is the first -inf,
        // else the first NaN (NaN ranks lowest)
        uint32_t first_ninf = 0xFFFFFFFFu;
        scan_share<kL, kU>(x, n_units, first, [&](const float (&f)[kU][kL], const int (&g)[kU]) {
#pragma unroll
            for (int j = 0; j < kU; ++j)
#pragma unroll
                for (int e = 0; e < kL; ++e)
                    if (g[j] < n_units && f[j][e] == -INFINITY && first_ninf == 0xFFFFFFFFu)
                        first_ninf = static_cast<uint32_t>(g[j] * kL + e);
        });
        my_key = first_ninf != 0xFFFFFFFFu ? argmax_pack(float_order_key(-INFINITY), first_ninf)
                                           : argmax_pack(0u, static_cast<uint32_t>(first * kL));
    }

    // warp partial of the exp-sum
    {
        const float mw = warp_max_f(m);
        float t = 0.0f;
        if (mw != -INFINITY && mw != INFINITY && m != -INFINITY) t = s * __expf(m - mw);   // NaN s propagates
        t = warp_sum_f(t);
        nan = __any_sync(0xffffffffu, nan);
        if (lane == 0) { s_m[warp] = mw; s_s[warp] = t; s_nan[warp] = nan; }
    }
    s_keys[warp][lane] = warp_sort_desc(my_key, lane);
    if (threadIdx.x < 32) { s_win[threadIdx.x] = 0u; s_sel[threadIdx.x] = -1; }
    if (threadIdx.x == 0) { s_T = 0ull; s_count = 0; }
    __syncthreads();

    if (warp == kTopkWarps - 1) {   // the row's log-sum-exp (beside the ranks below)
        const float mw = lane < kTopkWarps ? s_m[lane] : -INFINITY;
        const float sw = lane < kTopkWarps ? s_s[lane] : 0.0f;
        const bool any_nan = __any_sync(0xffffffffu, lane < kTopkWarps && s_nan[lane] != 0);
        const float M = warp_max_f(mw);
        float term = 0.0f;
        if (M != -INFINITY && M != INFINITY && sw != 0.0f) term = sw * expf(mw - M);
        term = warp_sum_f(term);
        if (lane == 0)
            s_lse = (any_nan || M == -INFINITY || M == INFINITY)
                        ? __longlong_as_double(0x7FF8000000000000ll)   // NaN, as the exp-sum is
                        : static_cast<double>(M) + static_cast<double>(logf(term));
    }
    // T = the K-th largest best key (stays 0 if fewer than K threads hold
    // elements); the threads holding the K largest best keys are selected. A
    // key's unit g = id / kL belongs to thread (warp, lane) with lane = g % 32
    // and warp = (g % (kTopkThreads * kU)) / (32 * kU).
    rank_lists(s_keys, K, [&](int rank, unsigned long long c) {
        if (rank < K) {
            const uint32_t g = argmax_unpack_idx(c) / kL;
            s_sel[rank] = static_cast<int>((g % (kTopkThreads * kU)) / (32 * kU) * 32 + g % 32);
        }
        if (rank == K - 1) s_T = c;
    });
    __syncthreads();
    const unsigned long long T = s_T;

    // pass B: each warp re-reads selected shares, one unit per lane, and
    // stages the keys >= T
    for (int q = warp; q < K; q += kTopkWarps) {
        const int tid = s_sel[q];
        if (tid < 0) continue;
        const int t_first = (tid >> 5) * 32 * kU + (tid & 31);
        for (int i0 = 0;; i0 += 32) {
            const int i = i0 + lane;
            // unit i of the share: group i / kU, slot i % kU
            if (static_cast<long long>(t_first) + static_cast<long long>(i0 / kU) * kTopkThreads * kU >= n_units)
                break;   // warp-uniform: no unit of this or a later batch exists
            const long long g = static_cast<long long>(t_first) +
                                static_cast<long long>(i / kU) * kTopkThreads * kU + (i % kU) * 32;
            if (g < n_units) {
                float f[kL];
                if constexpr (kL == 4) {
                    const float4 t = __ldg(reinterpret_cast<const float4*>(x) + g);
                    f[0] = t.x; f[1] = t.y; f[2] = t.z; f[3] = t.w;
                } else {
                    f[0] = __ldg(x + g);
                }
#pragma unroll
                for (int e = 0; e < kL; ++e) {
                    const unsigned long long k =
                        argmax_pack(float_order_key(f[e]), static_cast<uint32_t>(g * kL + e));
                    if (k >= T) {
                        const int slot = atomicAdd(&s_count, 1);
                        if (slot < kTopkCap) s_cand[slot] = k;
                    }
                }
            }
        }
    }
    __syncthreads();
    const int n = s_count;
    if (n <= kTopkCap) {
        // exact ranks among the staged keys (distinct; at least K of them)
        for (int c = threadIdx.x; c < n; c += kTopkThreads) {
            const unsigned long long key = s_cand[c];
            int rank = 0;
            for (int i = 0; i < n; ++i) rank += s_cand[i] > key;
            if (rank < K) s_win[rank] = argmax_unpack_idx(key);
        }
    } else {
        // many candidates: a sorted list per warp over the whole row (keys < T
        // dropped), then the lists' ranks
        unsigned long long list = 0ull, thr = 0ull;   // every element's key is > 0
        for (int base = warp * 32 * kU; base < n_units; base += kTopkThreads * kU) {
#pragma unroll
            for (int j = 0; j < kU; ++j) {
                const int g = base + j * 32 + lane;
                float f[kL];
                if (g < n_units) {
                    if constexpr (kL == 4) {
                        const float4 t = __ldg(reinterpret_cast<const float4*>(x) + g);
                        f[0] = t.x; f[1] = t.y; f[2] = t.z; f[3] = t.w;
                    } else {
                        f[0] = __ldg(x + g);
                    }
                }
#pragma unroll
                for (int e = 0; e < kL; ++e) {
                    unsigned long long key = 0ull;
                    if (g < n_units) {
                        key = argmax_pack(float_order_key(f[e]), static_cast<uint32_t>(g * kL + e));
                        if (key < T) key = 0ull;
                    }
                    list_offer(list, thr, key, K, lane);
                }
            }
        }
        s_keys[warp][lane] = lane < K ? list : 0ull;   // the earlier readers are past a barrier
        __syncthreads();
        rank_lists(s_keys, K, [&](int rank, unsigned long long c) {
            if (rank < K) s_win[rank] = argmax_unpack_idx(c);
        });
    }
    __syncthreads();
    if (threadIdx.x < K) {
        const uint32_t idx = s_win[threadIdx.x];
        out_tok[row * K + threadIdx.x] = static_cast<int32_t>(idx);
        out_lp[row * K + threadIdx.x] = static_cast<float>(static_cast<double>(__ldg(x + idx)) - s_lse);
    }
}

cudaError_t launch_draft_topk(const float* logits, int V, int B, int D, int K, float* topk_logp,
                              int32_t* topk_tok, cudaStream_t stream) {
    const unsigned rows = static_cast<unsigned>(B) * static_cast<unsigned>(D);
    if (V % 4 == 0 && reinterpret_cast<uintptr_t>(logits) % 16 == 0)
        draft_topk_kernel<4><<<rows, kTopkThreads, 0, stream>>>(logits, V, K, topk_logp, topk_tok);
    else
        draft_topk_kernel<1><<<rows, kTopkThreads, 0, stream>>>(logits, V, K, topk_logp, topk_tok);
    return cudaGetLastError();
}

}  // namespace ddt
