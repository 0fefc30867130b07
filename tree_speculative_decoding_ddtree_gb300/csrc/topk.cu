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
// One CTA per (request, depth) row. Each thread streams its share of the row
// (16-byte loads) keeping an online (max, sum of exp(x - max)) pair for the
// log-sum-exp, and each warp keeps the row's K best keys seen so far spread
// over its lanes (lane k holds the k-th best): a value above the K-th best is
// inserted with one ballot and one shift. Keys pack the logit's order key
// above the inverted token id, so a larger key is a larger logit or, on a
// tie, a lower id; NaN ranks below every number. Warp 0 merges the warps'
// lists. The log-sum-exp is combined in fp64 and the log-probs are formed in
// fp64, then rounded to fp32.
#include "common.cuh"

namespace ddt {

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;

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

// online (max, sum of exp(x - max)) of a row share; NaN only sets the flag
// (the row's log-sum-exp is then NaN, as is the case for a +inf or all -inf row)
struct Lse {
    float m, s;
    bool nan;
};

DDT_DEVINL Lse lse_merge(Lse a, Lse b) {
    Lse r;
    r.nan = a.nan || b.nan;
    r.m = fmaxf(a.m, b.m);
    if (r.m == -INFINITY || r.m == INFINITY) {
        r.s = 0.0f;   // only the flagged cases reach here with a non-empty share
    } else {
        r.s = (a.s > 0.0f ? a.s * expf(a.m - r.m) : 0.0f) + (b.s > 0.0f ? b.s * expf(b.m - r.m) : 0.0f);
    }
    return r;
}

// kL floats per load (4: 16-byte loads, needs V % 4 == 0 and an aligned row),
// kU loads in flight per lane
template <int kL>
__global__ void __launch_bounds__(kTopkThreads)
draft_topk_kernel(const float* __restrict__ logits, int V, int K,
                  float* __restrict__ out_lp, int32_t* __restrict__ out_tok) {
    constexpr int kU = 4;
    __shared__ unsigned long long s_keys[kTopkWarps][DDT_MAX_TOPK];
    __shared__ float s_m[kTopkWarps], s_s[kTopkWarps];
    __shared__ int s_nan[kTopkWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t row = blockIdx.x;
    const float* x = logits + row * static_cast<size_t>(V);
    const int n_units = V / kL;
    unsigned long long list = 0ull, thr = 0ull;   // every element's key is > 0
    Lse acc{-INFINITY, 0.0f, false};
    // warp-uniform trip count: the list operations always see all 32 lanes
    for (int base = warp * 32 * kU; base < n_units; base += kTopkThreads * kU) {
        float f[kU][kL];
#pragma unroll
        for (int j = 0; j < kU; ++j) {
            const int g = base + j * 32 + lane;
            if (g < n_units) {
                if constexpr (kL == 4) {
                    const float4 t = __ldg(reinterpret_cast<const float4*>(x) + g);
                    f[j][0] = t.x; f[j][1] = t.y; f[j][2] = t.z; f[j][3] = t.w;
                } else {
                    f[j][0] = __ldg(x + g);
                }
            } else {
#pragma unroll
                for (int e = 0; e < kL; ++e) f[j][e] = -INFINITY;   // adds nothing to the sum
            }
        }
        float mloc = -INFINITY;
        bool nanloc = false;
#pragma unroll
        for (int j = 0; j < kU; ++j)
#pragma unroll
            for (int e = 0; e < kL; ++e) {
                nanloc |= f[j][e] != f[j][e];
                mloc = fmaxf(mloc, f[j][e]);   // fmaxf skips NaN
            }
        const float m_new = fmaxf(acc.m, mloc);
        if (m_new != -INFINITY) {
            float s = acc.s > 0.0f ? acc.s * expf(acc.m - m_new) : 0.0f;
#pragma unroll
            for (int j = 0; j < kU; ++j)
#pragma unroll
                for (int e = 0; e < kL; ++e) s += expf(f[j][e] - m_new);
            acc.s = s;
            acc.m = m_new;
        }
        acc.nan |= nanloc;
#pragma unroll
        for (int j = 0; j < kU; ++j) {
            const int g = base + j * 32 + lane;
#pragma unroll
            for (int e = 0; e < kL; ++e) {
                const unsigned long long key =
                    g < n_units ? argmax_pack(float_order_key(f[j][e]), static_cast<uint32_t>(g * kL + e)) : 0ull;
                list_offer(list, thr, key, K, lane);
            }
        }
    }
    // warp partials of the log-sum-exp
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Lse other;
        other.m = __shfl_xor_sync(0xffffffffu, acc.m, o);
        other.s = __shfl_xor_sync(0xffffffffu, acc.s, o);
        other.nan = __shfl_xor_sync(0xffffffffu, static_cast<int>(acc.nan), o) != 0;
        acc = lse_merge(acc, other);
    }
    if (lane < K) s_keys[warp][lane] = list;
    if (lane == 0) { s_m[warp] = acc.m; s_s[warp] = acc.s; s_nan[warp] = acc.nan; }
    __syncthreads();
    if (warp != 0) return;
    // warp 0: merge the other warps' lists into its own (warp 0 has seen at
    // least min(V, 32) >= K elements, so its list is full and thr > 0: the
    // empty slots of shorter lists, key 0, never enter)
    for (int w = 1; w < kTopkWarps; ++w) {
        const unsigned long long cand = lane < K ? s_keys[w][lane] : 0ull;
        list_offer(list, thr, cand, K, lane);
    }
    bool nan = false;
    float M = -INFINITY;
    for (int w = 0; w < kTopkWarps; ++w) { M = fmaxf(M, s_m[w]); nan |= s_nan[w] != 0; }
    double lse;
    if (nan || M == -INFINITY || M == INFINITY) {
        lse = __longlong_as_double(0x7FF8000000000000ll);   // NaN, as the row's exp-sum is
    } else {
        double s = 0.0;
        for (int w = 0; w < kTopkWarps; ++w)
            if (s_s[w] > 0.0f)
                s += static_cast<double>(s_s[w]) * exp(static_cast<double>(s_m[w]) - static_cast<double>(M));
        lse = static_cast<double>(M) + log(s);
    }
    if (lane < K) {
        const uint32_t idx = argmax_unpack_idx(list);
        const float v = __ldg(x + idx);
        out_tok[row * K + lane] = static_cast<int32_t>(idx);
        out_lp[row * K + lane] = static_cast<float>(static_cast<double>(v) - lse);
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
