// The verify walks over a vocabulary-parallel logits shard, for a request
// split over GPUs by KV head ("The Pivot Point: Strategic Decision-Making in
// Speculative Decoding Optimization", The Strategic Decision: TP8). With
// tensor parallelism each rank holds the logits of its vocabulary slice
// [v0, v0 + Vs) only ("The Architecture of Speculative Decoding: Dissecting
// DDTree's Tree-Parallel Evaluation Strategy", Section 1 step 1, the
// vocab-parallel head). The walk itself is the same as ddtree_accept_greedy /
// ddtree_accept_sample; only the reductions over the vocabulary are split:
//
//   partial   each rank reduces its slice for the current node of every
//             request: the packed (value, global index) argmax, the online
//             (max, sum of exp) of logits/T, and the logits of the node's
//             children that fall in the slice (-inf for the others); one
//             36-word record per request
//   (the caller all-gathers the records: [world, B, 36])
//   advance   every rank merges the world's records in rank order (so all
//             ranks hold identical values) and takes the same step: greedy
//             match or bonus; sampled child tests, or marks the bonus due
//   bonus     (sampled) each rank's Gumbel-max over its slice for requests
//             whose bonus is due, all-gathered, then merged by `finish`
//
// One CTA (or one thread) per request; the state [B, 4] (current node,
// accepted length, phase, rejected tests) lives on the device between calls.
#include "walk.cuh"

namespace ddt {

namespace {

constexpr int kShardThreads = 256;
constexpr int kRec = 36;   // record words: key lo, key hi, max, sum, 32 child logits
enum Phase { kWalking = 0, kBonusDue = 1, kDone = 2 };

DDT_DEVINL unsigned long long block_max_u64_256(unsigned long long v, unsigned long long* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_max_u64(v);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    unsigned long long x = lane < kShardThreads / 32 ? scratch[lane] : 0ull;
    if (warp == 0) x = warp_max_u64(x);
    return x;   // valid in thread 0
}

DDT_DEVINL MaxSum block_ms_256(MaxSum ms, float inv_t, float2* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        ms = merge_ms(ms, MaxSum{__shfl_xor_sync(0xffffffffu, ms.m, o), __shfl_xor_sync(0xffffffffu, ms.z, o)}, inv_t);
    __syncthreads();
    if (lane == 0) scratch[warp] = make_float2(ms.m, ms.z);
    __syncthreads();
    if (warp == 0) {
        const float2 v = lane < kShardThreads / 32 ? scratch[lane] : make_float2(-INFINITY, 0.0f);
        ms = MaxSum{v.x, v.y};
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            ms = merge_ms(ms, MaxSum{__shfl_xor_sync(0xffffffffu, ms.m, o), __shfl_xor_sync(0xffffffffu, ms.z, o)}, inv_t);
    }
    return ms;   // valid in thread 0
}

// children of node u in rank order (at most kMaxKids); returns the count
DDT_DEVINL int node_children(const int32_t* fc, const int32_t* ns, size_t tb, int u, int nn, int* kids,
                             bool* bad) {
    int c = fc[tb + u], j = 0;
    while (c != -1) {
        if (c < 1 || c >= nn || j >= kMaxKids) { *bad = true; break; }
        kids[j++] = c;
        c = ns[tb + c];
    }
    return j;
}

__global__ void __launch_bounds__(kShardThreads)
shard_partial_kernel(const float* __restrict__ logits, int Vs, int v0, const int32_t* __restrict__ token,
                     const int32_t* __restrict__ first_child, const int32_t* __restrict__ next_sibling,
                     const int32_t* __restrict__ n_nodes, int N, const float* __restrict__ temperature,
                     const int32_t* __restrict__ state, int32_t* __restrict__ rec) {
    __shared__ unsigned long long scratch_u[32];
    __shared__ float2 scratch_ms[32];
    __shared__ int kids[kMaxKids];
    __shared__ int nk;
    const int b = blockIdx.x;
    int32_t* out = rec + static_cast<size_t>(b) * kRec;
    const int u = state[b * 4 + 0], phase = state[b * 4 + 2];
    if (phase != kWalking) {   // a neutral record: nothing to contribute
        for (int k = threadIdx.x; k < kRec; k += kShardThreads)
            out[k] = k < 2 ? 0 : (k == 3 ? __float_as_int(0.0f) : __float_as_int(-INFINITY));
        return;
    }
    const size_t tb = static_cast<size_t>(b) * N;
    int nn = n_nodes[b];
    nn = nn < 1 ? 1 : (nn > N ? N : nn);
    if (threadIdx.x == 0) {
        bool bad = false;
        nk = node_children(first_child, next_sibling, tb, u, nn, kids, &bad);
    }
    __syncthreads();
    const float* row = logits + (tb + u) * static_cast<size_t>(Vs);
    const bool sampled = temperature != nullptr;
    const float inv_t = sampled ? 1.0f / temperature[b] : 1.0f;
    unsigned long long best = 0ull;
    MaxSum ms{-INFINITY, 0.0f};
    for (int v = threadIdx.x; v < Vs; v += kShardThreads) {
        const float x = __ldg(row + v);
        if (sampled) {
            if (x > ms.m) { ms.z = ms.z * expf((ms.m - x) * inv_t) + 1.0f; ms.m = x; }
            else ms.z += expf((x - ms.m) * inv_t);
        } else {
            const unsigned long long p = argmax_pack(float_order_key(x), static_cast<uint32_t>(v0 + v));
            best = best > p ? best : p;
        }
    }
    if (sampled) ms = block_ms_256(ms, inv_t, scratch_ms);
    else best = block_max_u64_256(best, scratch_u);
    if (threadIdx.x == 0) {
        out[0] = static_cast<int32_t>(static_cast<uint32_t>(best));
        out[1] = static_cast<int32_t>(static_cast<uint32_t>(best >> 32));
        out[2] = __float_as_int(sampled ? ms.m : -INFINITY);
        out[3] = __float_as_int(sampled ? ms.z : 0.0f);
    }
    if (threadIdx.x < kMaxKids) {
        float l = -INFINITY;
        if (static_cast<int>(threadIdx.x) < nk) {
            const int x = token[tb + kids[threadIdx.x]];
            if (x >= v0 && x < v0 + Vs) l = __ldg(row + (x - v0));
        }
        out[4 + threadIdx.x] = __float_as_int(l);
    }
}

// one thread per request: merge the world's records in rank order, then step
__global__ void shard_advance_kernel(const int32_t* __restrict__ recs, int world, int B, int V,
                                     const int32_t* __restrict__ token,
                                     const int32_t* __restrict__ first_child,
                                     const int32_t* __restrict__ next_sibling,
                                     const int32_t* __restrict__ n_nodes, int N, int D,
                                     const float* __restrict__ temperature,
                                     const uint64_t* __restrict__ seed, uint64_t offset,
                                     int32_t* state, WalkOut o, int32_t* dev_status) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int32_t* st = state + b * 4;
    if (st[2] != kWalking) return;
    const int u = st[0], len = st[1];
    const size_t tb = static_cast<size_t>(b) * N;
    int nn = n_nodes[b];
    nn = nn < 1 ? 1 : (nn > N ? N : nn);
    int kids[kMaxKids];
    bool bad = false;
    int nk = node_children(first_child, next_sibling, tb, u, nn, kids, &bad);
    if (bad) report(dev_status, DDT_DEV_BAD_TREE);
    int32_t* toks = o.out_tokens + static_cast<size_t>(b) * (D + 1);
    int32_t* nodes = o.out_nodes + static_cast<size_t>(b) * (D + 1);
    const bool sampled = temperature != nullptr;
    int match = -1;
    uint32_t a = 0;
    if (!sampled) {
        unsigned long long best = 0ull;
        for (int w = 0; w < world; ++w) {
            const int32_t* r = recs + (static_cast<size_t>(w) * B + b) * kRec;
            const unsigned long long k = static_cast<uint32_t>(r[0]) | (static_cast<unsigned long long>(static_cast<uint32_t>(r[1])) << 32);
            best = best > k ? best : k;
        }
        a = argmax_unpack_idx(best);
        for (int j = 0; j < nk; ++j) {
            if (token[tb + kids[j]] == static_cast<int32_t>(a)) { match = kids[j]; break; }
            ++st[3];
        }
    } else {
        const float T = temperature[b];
        if (!(T > 0.0f) || !isfinite(T)) {
            report(dev_status, DDT_DEV_BAD_TEMPERATURE);
            o.accept_len[b] = 0;
            o.bonus[b] = -1;
            st[2] = kDone;
            return;
        }
        const float inv_t = 1.0f / T;
        MaxSum acc{-INFINITY, 0.0f};
        for (int w = 0; w < world; ++w) {
            const int32_t* r = recs + (static_cast<size_t>(w) * B + b) * kRec;
            acc = merge_ms(acc, MaxSum{__int_as_float(r[2]), __int_as_float(r[3])}, inv_t);
        }
        const uint64_t sd = seed[b];
        const uint32_t k0 = static_cast<uint32_t>(sd), k1 = static_cast<uint32_t>(sd >> 32);
        double R = 1.0;
        for (int j = 0; j < nk; ++j) {
            const int x = token[tb + kids[j]];
            float l = -INFINITY;
            for (int w = 0; w < world; ++w) l = fmaxf(l, __int_as_float(recs[(static_cast<size_t>(w) * B + b) * kRec + 4 + j]));
            float q = 0.0f;
            if (x >= 0 && x < V) q = expf((l - acc.m) * inv_t) / acc.z;
            else report(dev_status, DDT_DEV_BAD_TOKEN);
            const uint4 wd = philox4x32_10(make_uint4(0u | (static_cast<uint32_t>(offset >> 32) << 8), static_cast<uint32_t>(u),
                                                      static_cast<uint32_t>(j), static_cast<uint32_t>(offset)), k0, k1);
            if (uniform_exact(wd.x) * R < static_cast<double>(q)) { match = kids[j]; break; }
            R -= static_cast<double>(q);
            ++st[3];
        }
    }
    if (match != -1 && len >= D) {   // a walk longer than the draft depth: malformed tree
        report(dev_status, DDT_DEV_BAD_TREE);
        match = -1;
    }
    if (match != -1) {
        toks[len] = token[tb + match];
        nodes[len + 1] = match;
        st[0] = match;
        st[1] = len + 1;
    } else if (!sampled) {
        toks[len] = static_cast<int32_t>(a);
        o.bonus[b] = static_cast<int32_t>(a);
        o.accept_len[b] = len;
        st[2] = kDone;
    } else {
        st[2] = kBonusDue;
    }
}

__global__ void __launch_bounds__(kShardThreads)
shard_bonus_kernel(const float* __restrict__ logits, int Vs, int v0, const int32_t* __restrict__ token,
                   const int32_t* __restrict__ first_child, const int32_t* __restrict__ next_sibling,
                   const int32_t* __restrict__ n_nodes, int N, const float* __restrict__ temperature,
                   const uint64_t* __restrict__ seed, uint64_t offset, const int32_t* __restrict__ state,
                   unsigned long long* __restrict__ key) {
    __shared__ unsigned long long scratch_u[32];
    __shared__ int kid_tok[kMaxKids];
    __shared__ int nk;
    const int b = blockIdx.x;
    if (state[b * 4 + 2] != kBonusDue) {
        if (threadIdx.x == 0) key[b] = 0ull;
        return;
    }
    const int u = state[b * 4 + 0];
    const size_t tb = static_cast<size_t>(b) * N;
    int nn = n_nodes[b];
    nn = nn < 1 ? 1 : (nn > N ? N : nn);
    if (threadIdx.x == 0) {
        int kids[kMaxKids];
        bool bad = false;
        nk = node_children(first_child, next_sibling, tb, u, nn, kids, &bad);
        for (int j = 0; j < nk; ++j) kid_tok[j] = token[tb + kids[j]];
    }
    __syncthreads();
    const float* row = logits + (tb + u) * static_cast<size_t>(Vs);
    const float inv_t = 1.0f / temperature[b];
    const uint64_t sd = seed[b];
    const uint32_t k0 = static_cast<uint32_t>(sd), k1 = static_cast<uint32_t>(sd >> 32);
    const uint32_t off_lo = static_cast<uint32_t>(offset), off_hi8 = static_cast<uint32_t>(offset >> 32) << 8;
    unsigned long long best = 0ull;
    for (int i = threadIdx.x; i < Vs; i += kShardThreads) {
        const int v = v0 + i;   // the global vocabulary entry: its Gumbel noise is the unsplit walk's
        bool kid = false;
        for (int k = 0; k < nk; ++k) kid |= (kid_tok[k] == v);
        if (kid) continue;
        const uint4 w = philox4x32_10(make_uint4(1u | off_hi8, static_cast<uint32_t>(u), static_cast<uint32_t>(v >> 2),
                                                 off_lo), k0, k1);
        const uint32_t word = (v & 3) == 0 ? w.x : (v & 3) == 1 ? w.y : (v & 3) == 2 ? w.z : w.w;
        const float sc = __ldg(row + i) * inv_t + gumbel_noise(word);
        const unsigned long long p = argmax_pack(float_order_key(sc), static_cast<uint32_t>(v));
        best = best > p ? best : p;
    }
    best = block_max_u64_256(best, scratch_u);
    if (threadIdx.x == 0) key[b] = best;
}

__global__ void shard_finish_kernel(const unsigned long long* __restrict__ keys, int world, int B, int D,
                                    int32_t* state, WalkOut o) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int32_t* st = state + b * 4;
    if (st[2] != kBonusDue) return;
    unsigned long long best = 0ull;
    for (int w = 0; w < world; ++w) {
        const unsigned long long k = keys[static_cast<size_t>(w) * B + b];
        best = best > k ? best : k;
    }
    const int len = st[1];
    const int32_t a = best ? static_cast<int32_t>(argmax_unpack_idx(best)) : -1;
    o.out_tokens[static_cast<size_t>(b) * (D + 1) + len] = a;
    o.bonus[b] = a;
    o.accept_len[b] = len;
    st[2] = kDone;
}

__global__ void shard_begin_kernel(int B, int D, int32_t* state, WalkOut o) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    state[b * 4 + 0] = 0;
    state[b * 4 + 1] = 0;
    state[b * 4 + 2] = kWalking;
    state[b * 4 + 3] = 0;
    for (int k = 0; k <= D; ++k) {
        o.out_tokens[static_cast<size_t>(b) * (D + 1) + k] = -1;
        o.out_nodes[static_cast<size_t>(b) * (D + 1) + k] = k == 0 ? 0 : -1;
    }
    o.accept_len[b] = 0;
    o.bonus[b] = -1;
}

}  // namespace

cudaError_t launch_shard_begin(int B, int D, int32_t* state, int32_t* accept_len, int32_t* out_tokens,
                               int32_t* out_nodes, int32_t* bonus, cudaStream_t s) {
    WalkOut o{accept_len, out_tokens, out_nodes, bonus, nullptr, nullptr};
    shard_begin_kernel<<<(B + 127) / 128, 128, 0, s>>>(B, D, state, o);
    return cudaGetLastError();
}

cudaError_t launch_shard_partial(const float* logits, int Vs, int v0, const int32_t* token,
                                 const int32_t* first_child, const int32_t* next_sibling,
                                 const int32_t* n_nodes, int B, int N, const float* temperature,
                                 const int32_t* state, int32_t* rec, cudaStream_t s) {
    shard_partial_kernel<<<B, kShardThreads, 0, s>>>(logits, Vs, v0, token, first_child, next_sibling, n_nodes, N,
                                                     temperature, state, rec);
    return cudaGetLastError();
}

cudaError_t launch_shard_advance(const int32_t* recs, int world, int B, int V, const int32_t* token,
                                 const int32_t* first_child, const int32_t* next_sibling,
                                 const int32_t* n_nodes, int N, int D, const float* temperature,
                                 const uint64_t* seed, uint64_t offset, int32_t* state, int32_t* accept_len,
                                 int32_t* out_tokens, int32_t* out_nodes, int32_t* bonus, int32_t* dev_status,
                                 cudaStream_t s) {
    WalkOut o{accept_len, out_tokens, out_nodes, bonus, nullptr, nullptr};
    shard_advance_kernel<<<(B + 63) / 64, 64, 0, s>>>(recs, world, B, V, token, first_child, next_sibling, n_nodes,
                                                      N, D, temperature, seed, offset, state, o, dev_status);
    return cudaGetLastError();
}

cudaError_t launch_shard_bonus(const float* logits, int Vs, int v0, const int32_t* token,
                               const int32_t* first_child, const int32_t* next_sibling,
                               const int32_t* n_nodes, int B, int N, const float* temperature,
                               const uint64_t* seed, uint64_t offset, const int32_t* state,
                               unsigned long long* key, cudaStream_t s) {
    shard_bonus_kernel<<<B, kShardThreads, 0, s>>>(logits, Vs, v0, token, first_child, next_sibling, n_nodes, N,
                                                   temperature, seed, offset, state, key);
    return cudaGetLastError();
}

cudaError_t launch_shard_finish(const unsigned long long* keys, int world, int B, int D, int32_t* state,
                                int32_t* accept_len, int32_t* out_tokens, int32_t* bonus, cudaStream_t s) {
    WalkOut o{accept_len, out_tokens, nullptr, bonus, nullptr, nullptr};
    shard_finish_kernel<<<(B + 127) / 128, 128, 0, s>>>(keys, world, B, D, state, o);
    return cudaGetLastError();
}

}  // namespace ddt
