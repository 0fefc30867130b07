// ddtree_commit_kv: the committed path's K/V appended to the paged cache.
//
// Method: "The Architecture of Speculative Decoding: Dissecting DDTree's
// Tree-Parallel Evaluation Strategy", Section 1 step 5 (only the longest
// verified path is committed); "The Tree That Couldn't Branch", Hypothesis 3
// (a node of depth d is verified at position ctx_len + d). Path row i (the
// root, then the accepted nodes) goes to token position ctx_len + i.
//
// One CTA per request: its threads first check the path rows and their pages
// (any bad entry: nothing is written and the length is kept), then copy the
// rows with 16-byte loads and stores, K and V together. The new length is
// written last, after a barrier that every read of ctx_len precedes, so the
// output may alias ctx_len (an in-place advance).
#include "common.cuh"

namespace ddt {

constexpr int kCommitThreads = 256;

__global__ void __launch_bounds__(kCommitThreads)
commit_kv_kernel(const uint4* __restrict__ k_tree, const uint4* __restrict__ v_tree, int row_vec,
                 const int32_t* __restrict__ out_nodes, const int32_t* __restrict__ accept_len, int N,
                 int D, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int num_pages,
                 int page_size, const int32_t* __restrict__ page_table, int max_pages,
                 const int32_t* ctx_len, int32_t* new_ctx_len, int32_t* dev_status) {
    __shared__ long long s_src[DDT_MAX_DEPTH + 1];   // tree row (b * N + node)
    __shared__ long long s_dst[DDT_MAX_DEPTH + 1];   // cache row (page * page_size + slot)
    __shared__ int s_bad;
    const int b = blockIdx.x;
    const int ctx = ctx_len[b];
    const int acc = accept_len[b];
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    int len_bad = 0;
    if (acc < 0 || acc > D) len_bad = DDT_DEV_BAD_TREE;
    else if (ctx < 0 || static_cast<long long>(ctx) + acc + 1 > static_cast<long long>(max_pages) * page_size)
        len_bad = DDT_DEV_BAD_CTX;
    if (!len_bad) {
        for (int i = threadIdx.x; i <= acc; i += blockDim.x) {
            const int node = out_nodes[static_cast<size_t>(b) * (D + 1) + i];
            const long long t = static_cast<long long>(ctx) + i;
            const int page = page_table[static_cast<size_t>(b) * max_pages + t / page_size];
            int bits = 0;
            if (node < 0 || node >= N) bits |= DDT_DEV_BAD_TREE;
            if (page < 0 || page >= num_pages) bits |= DDT_DEV_BAD_PAGE;
            if (bits) atomicOr(&s_bad, bits);
            s_src[i] = static_cast<long long>(b) * N + node;
            s_dst[i] = static_cast<long long>(page) * page_size + t % page_size;
        }
    }
    __syncthreads();
    const int bad = len_bad | s_bad;
    if (!bad) {
        const long long total = static_cast<long long>(acc + 1) * row_vec;
        for (long long e = threadIdx.x; e < total; e += kCommitThreads) {
            const int i = static_cast<int>(e / row_vec);
            const long long v = e - static_cast<long long>(i) * row_vec;
            const uint4 kx = __ldg(k_tree + s_src[i] * row_vec + v);
            const uint4 vx = __ldg(v_tree + s_src[i] * row_vec + v);
            k_cache[s_dst[i] * row_vec + v] = kx;
            v_cache[s_dst[i] * row_vec + v] = vx;
        }
    }
    __syncthreads();   // every thread has read ctx_len[b]
    if (threadIdx.x == 0) {
        if (bad) report(dev_status, bad);
        new_ctx_len[b] = bad ? ctx : ctx + acc + 1;
    }
}

cudaError_t launch_commit_kv(const ddtree_bf16* k_tree, const ddtree_bf16* v_tree,
                             const int32_t* out_nodes, const int32_t* accept_len, int B, int N, int D,
                             int Hkv, int Dh, ddtree_bf16* k_cache, ddtree_bf16* v_cache, int num_pages,
                             int page_size, const int32_t* page_table, int max_pages,
                             const int32_t* ctx_len, int32_t* new_ctx_len, int32_t* dev_status,
                             cudaStream_t stream) {
    const int row_vec = Hkv * Dh / 8;   // 16-byte units per row
    commit_kv_kernel<<<B, kCommitThreads, 0, stream>>>(
        reinterpret_cast<const uint4*>(k_tree), reinterpret_cast<const uint4*>(v_tree), row_vec,
        out_nodes, accept_len, N, D, reinterpret_cast<uint4*>(k_cache), reinterpret_cast<uint4*>(v_cache),
        num_pages, page_size, page_table, max_pages, ctx_len, new_ctx_len, dev_status);
    return cudaGetLastError();
}

}  // namespace ddt
