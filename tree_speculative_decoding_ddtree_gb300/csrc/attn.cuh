// Parameters shared by the tree_verify_attn kernels.
#pragma once

#include "common.cuh"

namespace ddt {

typedef uint16_t bf16_t;

constexpr int kMaxRowsPerCta = 288;    // query rows one CTA carries (18 warps of 16)

struct AttnParams {
    const bf16_t* q;
    const bf16_t* k_tree;
    const bf16_t* v_tree;
    const bf16_t* k_cache;
    const bf16_t* v_cache;
    const int32_t* page_table;
    const int32_t* ctx_len;
    const uint32_t* vis;
    const int32_t* n_nodes;
    bf16_t* out;
    float* lse;
    float* ws_o;        // [B, Hkv, max_chunks, R, Dh] unnormalised partial outputs
    float2* ws_ml;      // [B, Hkv, max_chunks, R] (running max in log2 units, sum)
    int32_t* dev_status;
    int num_pages, page_size, max_pages;
    int B, N, Hq, Hkv, Dh, G, W, R;
    int rows_per_group, n_groups;
    int tiles_per_chunk, max_chunks;
    int merge_wide;      // split-KV merge with several chunk loads in flight per warp (few rows per SM)
    int tc_groups;       // tensor-core path: row groups of 256 rows per (request, KV head); the last
                         // group takes the rest (256 + up to 8 leftover rows, or fewer than 256)
    float scale_log2;
    uint64_t stall_ns;   // 0; else (testing entry point only) a wait that nothing completes, bounded by this limit
};

// warp-MMA path: any supported shape (split-KV main launch + combine)
cudaError_t launch_attn_mma(const AttnParams& p, cudaStream_t stream);
// tensor-core path (tcgen05 + TMA): Dh 128, G dividing 128, R <= 264, one row group
bool attn_tc_supported(const AttnParams& p);
cudaError_t launch_attn_tc(const AttnParams& p, cudaStream_t stream);
// merge split-KV partials (no-op launch when every request fits one chunk)
cudaError_t launch_attn_combine(const AttnParams& p, cudaStream_t stream);

}  // namespace ddt
