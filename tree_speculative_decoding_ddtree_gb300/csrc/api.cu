// C ABI of the DDTree verify step: host-side argument checks, then launches.
// Nothing here allocates or synchronises; every call is stream-ordered.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>

#include "attn.cuh"
#include "common.cuh"
#include "ddtree_testing.h"
#include "trace.h"
#include "walk.cuh"

namespace ddt {
cudaError_t launch_build(const float*, const int32_t*, const int32_t*, const int32_t*, int, int,
                         int, int, int32_t*, int32_t*, int32_t*, int32_t*, int32_t*, double*,
                         int32_t*, int32_t*, uint32_t*, int32_t*, int32_t*, cudaStream_t);
cudaError_t launch_accept_greedy(const float*, int, const int32_t*, const int32_t*,
                                 const int32_t*, const int32_t*, int, int, int, int32_t*,
                                 int32_t*, int32_t*, int32_t*, int32_t*, int32_t*, cudaStream_t);
cudaError_t launch_accept_sample(const float*, int, const int32_t*, const int32_t*,
                                 const int32_t*, const int32_t*, int, int, int, const float*,
                                 const uint64_t*, uint64_t, int32_t*, int32_t*, int32_t*,
                                 int32_t*, float*, int32_t*, int32_t*, cudaStream_t);
cudaError_t launch_accept_both(const float*, int, const int32_t*, const int32_t*, const int32_t*,
                               const int32_t*, int, int, int, const float*, const uint64_t*, uint64_t,
                               const WalkOut&, const WalkOut&, int32_t*, cudaStream_t);
cudaError_t launch_draft_topk(const float*, int, int, int, int, float*, int32_t*, cudaStream_t);
cudaError_t launch_gumbel_probe(const uint32_t*, float*, size_t, cudaStream_t);
cudaError_t launch_accept_ratio(const float*, const float*, int, const int32_t*, const int32_t*,
                                const int32_t*, const int32_t*, int, int, int, const float*,
                                const uint64_t*, uint64_t, int32_t*, int32_t*, int32_t*, int32_t*,
                                float*, int32_t*, int32_t*, cudaStream_t);
cudaError_t launch_commit_kv(const ddtree_bf16*, const ddtree_bf16*, const int32_t*, const int32_t*, int,
                             int, int, int, int, ddtree_bf16*, ddtree_bf16*, int, int, const int32_t*,
                             int, const int32_t*, int32_t*, int32_t*, cudaStream_t);

cudaError_t launch_shard_begin(int, int, int32_t*, int32_t*, int32_t*, int32_t*, int32_t*, cudaStream_t);
cudaError_t launch_shard_partial(const float*, int, int, const int32_t*, const int32_t*, const int32_t*,
                                 const int32_t*, int, int, const float*, const int32_t*, int32_t*, cudaStream_t);
cudaError_t launch_shard_advance(const int32_t*, int, int, int, const int32_t*, const int32_t*, const int32_t*,
                                 const int32_t*, int, int, const float*, const uint64_t*, uint64_t, int32_t*,
                                 int32_t*, int32_t*, int32_t*, int32_t*, int32_t*, cudaStream_t);
cudaError_t launch_shard_bonus(const float*, int, int, const int32_t*, const int32_t*, const int32_t*,
                               const int32_t*, int, int, const float*, const uint64_t*, uint64_t, const int32_t*,
                               unsigned long long*, cudaStream_t);
cudaError_t launch_shard_finish(const unsigned long long*, int, int, int, int32_t*, int32_t*, int32_t*, int32_t*,
                                cudaStream_t);

thread_local char g_last_error[256] = "";

// records the error text for ddtree_last_error(); shared with the step graph
int cuda_fail(cudaError_t e) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e),
                  cudaGetErrorString(e));
    return DDT_ECUDA;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kPlanWaves = 3;        // target CTAs per SM over a full-length batch (3 measured best of 2..8)
constexpr int kMaxPlanDevices = 64;
constexpr int kHostOnlySMs = 152;    // sizing on a host without a usable device (nothing launches there)

// SM count of the current device, queried once per device: the split-KV grid
// is sized in waves of it.
int plan_sms() {
    static std::atomic<int> cache[kMaxPlanDevices];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxPlanDevices) {
        cudaGetLastError();
        return kHostOnlySMs;
    }
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
            cudaGetLastError();
            return kHostOnlySMs;
        }
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}
constexpr int kKeyTile = 64;
// chunk-count model, in key-tile times of one SM (about 0.87 us for 264 rows of
// Dh 128 on the tensor-core path): a work item's fixed cost (start, Q, first
// tiles in flight, epilogue: about 9.6 us), the merge launch's fixed cost, and
// the bytes all SMs move in one key-tile time (one 32 KB K/V tile each)
constexpr long long kItemFixedTiles = 11;
constexpr long long kMergeFixedTiles = 5;
constexpr long long kTileBytesPerSm = 32768;

struct AttnPlan {
    int R, rows_per_group, n_groups, tiles_per_chunk, max_chunks;
    size_t ws_o_bytes, ws_ml_bytes;
};

bool plan_attn(int B, int N, int Hq, int Hkv, int Dh, long long max_ctx, AttnPlan* pl) {
    if (B < 1 || N < 1 || N > DDT_MAX_NODES || Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 ||
        (Dh != 64 && Dh != 128) || max_ctx < 0 || max_ctx > (1ll << 30))
        return false;
    const long long R = static_cast<long long>(N) * (Hq / Hkv);
    if (R > (1 << 20)) return false;
    pl->R = static_cast<int>(R);
    pl->n_groups = static_cast<int>((R + kMaxRowsPerCta - 1) / kMaxRowsPerCta);
    // spread rows evenly over the groups, in whole 16-row blocks
    const long long per = (R + pl->n_groups - 1) / pl->n_groups;
    pl->rows_per_group = static_cast<int>((per + 15) / 16 * 16);
    if (pl->rows_per_group > kMaxRowsPerCta) pl->rows_per_group = kMaxRowsPerCta;
    const long long tiles = (max_ctx + kKeyTile - 1) / kKeyTile;
    const long long units = static_cast<long long>(B) * Hkv * pl->n_groups;
    const long long total = units * (tiles > 0 ? tiles : 1);
    const int sms = plan_sms();
    const long long slots = static_cast<long long>(sms) * kPlanWaves;
    long long tpc = (total + slots - 1) / slots;
    if (tpc < 4) tpc = 4;
    if (tiles > 0) {
        // The wave target gives the fewest chunks per full-length context; from
        // there up to four times as many, take the count whose work items of a
        // batch of full-length contexts finish first: whole waves of equal items
        // (each its tiles plus a fixed cost) plus the merge's partial traffic,
        // all in key-tile times of one SM. Chunks are then as long as that count
        // needs and no longer.
        const long long nch0 = (tiles + tpc - 1) / tpc;
        long long nch_hi = 4 * nch0;
        if (nch_hi > tiles / 4) nch_hi = tiles / 4;
        if (nch_hi < nch0) nch_hi = nch0;
        long long best_n = nch0, best_cost = -1;
        for (long long n = nch0; n <= nch_hi; ++n) {
            const long long t = (tiles + n - 1) / n;
            if ((tiles + t - 1) / t != n) continue;   // no chunk length gives exactly n chunks
            const long long waves = (units * n + sms - 1) / sms;
            long long cost = waves * (kItemFixedTiles + t);
            if (n > 1) {
                const long long part = 2 * units * n * (R / pl->n_groups) * Dh * 4;   // written, then read
                cost += (part + static_cast<long long>(sms) * kTileBytesPerSm - 1) /
                            (static_cast<long long>(sms) * kTileBytesPerSm) + kMergeFixedTiles;
            }
            if (best_cost < 0 || cost < best_cost) { best_cost = cost; best_n = n; }
        }
        tpc = (tiles + best_n - 1) / best_n;
        if (tpc < 4) tpc = 4;
    }
    pl->tiles_per_chunk = static_cast<int>(tpc);
    pl->max_chunks = tiles > 0 ? static_cast<int>((tiles + tpc - 1) / tpc) : 1;
    const size_t rows = static_cast<size_t>(B) * Hkv * pl->max_chunks * R;
    pl->ws_o_bytes = pl->max_chunks > 1 ? (rows * Dh * sizeof(float) + 255) / 256 * 256 : 0;
    pl->ws_ml_bytes = pl->max_chunks > 1 ? (rows * sizeof(float2) + 255) / 256 * 256 : 0;
    return true;
}

}  // namespace

// Record a CUDA failure for ddtree_last_error() (used by entry points in other files).
void set_last_error(const char* what, cudaError_t e) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s: %s", what, cudaGetErrorName(e),
                  cudaGetErrorString(e));
}

}  // namespace ddt

using namespace ddt;

extern "C" {

const char* ddtree_status_string(int status) {
    switch (status) {
        case DDT_OK: return "DDT_OK";
        case DDT_EINVAL: return "DDT_EINVAL: null pointer or bad scalar argument";
        case DDT_ESHAPE: return "DDT_ESHAPE: sizes outside the supported range";
        case DDT_ECUDA: return "DDT_ECUDA: a CUDA call or launch failed";
        case DDT_ETIMEOUT: return "DDT_ETIMEOUT: a bounded device wait gave up";
        case DDT_EWORKSPACE: return "DDT_EWORKSPACE: workspace missing or too small";
        case DDT_ESCRATCH: return "DDT_ESCRATCH: sizes need more scratch than tree_verify_attn_noalloc's fixed array";
        default: return "unknown ddtree status";
    }
}

const char* ddtree_last_error(void) { return g_last_error; }

int ddtree_draft_topk(const float* draft_logits, int B, int D, int V, int K, float* topk_logp,
                      int32_t* topk_tok, void* stream) {
    TraceRange trace("ddtree_draft_topk");
    if (B < 0 || V < 1) return DDT_EINVAL;
    if (K < 1 || K > DDT_MAX_TOPK || K > V || D < 1 || D > DDT_MAX_DEPTH ||
        static_cast<long long>(B) * D > 0x7FFFFFFFll)
        return DDT_ESHAPE;
    if (B == 0) return DDT_OK;
    if (!draft_logits || !topk_logp || !topk_tok) return DDT_EINVAL;
    cudaError_t e = launch_draft_topk(draft_logits, V, B, D, K, topk_logp, topk_tok,
                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DDT_OK : cuda_fail(e);
}

int ddtree_build(const float* topk_logp, const int32_t* topk_tok, const int32_t* root_tok,
                 const int32_t* ctx_len, int B, int D, int K, int budget, int32_t* parent,
                 int32_t* depth, int32_t* token, int32_t* rank, int32_t* pos, double* score,
                 int32_t* first_child, int32_t* next_sibling, uint32_t* vis, int32_t* n_nodes,
                 int32_t* dev_status, void* stream) {
    TraceRange trace("ddtree_build");
    if (B < 0) return DDT_EINVAL;
    if (K < 1 || K > DDT_MAX_TOPK || D < 1 || D > DDT_MAX_DEPTH || budget < 0 ||
        budget + 1 > DDT_MAX_NODES)
        return DDT_ESHAPE;
    if (B == 0) return DDT_OK;
    if (!topk_logp || !topk_tok || !root_tok || !ctx_len || !parent || !depth || !token ||
        !rank || !pos || !score || !first_child || !next_sibling || !vis || !n_nodes)
        return DDT_EINVAL;
    cudaError_t e = launch_build(topk_logp, topk_tok, root_tok, ctx_len, B, D, K, budget, parent,
                                 depth, token, rank, pos, score, first_child, next_sibling, vis,
                                 n_nodes, dev_status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DDT_OK : cuda_fail(e);
}

size_t tree_verify_attn_workspace_size(int B, int N, int Hq, int Hkv, int Dh, int max_ctx) {
    AttnPlan pl;
    if (!plan_attn(B, N, Hq, Hkv, Dh, max_ctx, &pl)) return 0;
    return pl.ws_o_bytes + pl.ws_ml_bytes;
}

namespace {

// tree_verify_attn's checks and launches; stall_ns != 0 (the testing entry
// point only) makes the tensor-core kernel's bounded waits run out.
int attn_call(const ddtree_bf16* q, const ddtree_bf16* k_tree, const ddtree_bf16* v_tree,
              const ddtree_bf16* k_cache, const ddtree_bf16* v_cache, int num_pages, int page_size,
              const int32_t* page_table, int max_pages, const int32_t* ctx_len, const uint32_t* vis,
              const int32_t* n_nodes, int B, int N, int Hq, int Hkv, int Dh, float scale,
              ddtree_bf16* out, float* lse, void* workspace, size_t workspace_bytes,
              int32_t* dev_status, void* stream, uint64_t stall_ns) {
    if (B < 0 || !std::isfinite(scale)) return DDT_EINVAL;
    if (page_size < 16 || page_size > 1024 || page_size % 16 != 0 || num_pages < 1 ||
        max_pages < 1)
        return DDT_ESHAPE;
    const long long max_ctx = static_cast<long long>(max_pages) * page_size;
    AttnPlan pl;
    if (!plan_attn(B > 0 ? B : 1, N, Hq, Hkv, Dh, max_ctx, &pl)) return DDT_ESHAPE;
    if (B == 0) return DDT_OK;
    if (!q || !k_tree || !v_tree || !k_cache || !v_cache || !page_table || !ctx_len || !vis ||
        !n_nodes || !out)
        return DDT_EINVAL;
    if (!aligned16(q) || !aligned16(k_tree) || !aligned16(v_tree) || !aligned16(k_cache) ||
        !aligned16(v_cache) || !aligned16(out))
        return DDT_EINVAL;
    const size_t need = pl.ws_o_bytes + pl.ws_ml_bytes;
    if (need > 0 && (!workspace || workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return DDT_EWORKSPACE;
    AttnParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = q; p.k_tree = k_tree; p.v_tree = v_tree; p.k_cache = k_cache; p.v_cache = v_cache;
    p.page_table = page_table; p.ctx_len = ctx_len; p.vis = vis; p.n_nodes = n_nodes;
    p.out = out; p.lse = lse; p.dev_status = dev_status;
    p.ws_o = need ? static_cast<float*>(workspace) : nullptr;
    p.ws_ml = need ? reinterpret_cast<float2*>(static_cast<char*>(workspace) + pl.ws_o_bytes) : nullptr;
    p.num_pages = num_pages; p.page_size = page_size; p.max_pages = max_pages;
    p.B = B; p.N = N; p.Hq = Hq; p.Hkv = Hkv; p.Dh = Dh; p.G = Hq / Hkv; p.W = (N + 31) / 32;
    p.R = pl.R; p.rows_per_group = pl.rows_per_group; p.n_groups = pl.n_groups;
    p.tiles_per_chunk = pl.tiles_per_chunk; p.max_chunks = pl.max_chunks;
    // fewer merge rows than 32 warps per SM: occupancy cannot hide the loads
    p.merge_wide = static_cast<long long>(pl.R) * Hkv * B <= 32ll * plan_sms() ? 1 : 0;
    // tensor-core path: groups of two tiles of rpt rows (the whole nodes that fit in
    // 128 rows); up to 8 more rows ride in the last full group as leftover rows, a
    // longer rest takes a group of its own
    {
        const int G = Hq / Hkv;
        const int rpt = G <= 128 ? (128 / G) * G : 0;
        p.tc_groups = rpt == 0 ? 0 : pl.R <= 2 * rpt + 8 ? 1 : pl.R / (2 * rpt) + (pl.R % (2 * rpt) > 8 ? 1 : 0);
    }
    p.scale_log2 = scale * 1.4426950408889634f;
    p.stall_ns = stall_ns;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (attn_tc_supported(p)) {
        e = launch_attn_tc(p, st);
        if (e == cudaSuccess) e = launch_attn_combine(p, st);
    } else {
        if (stall_ns) return DDT_ESHAPE;   // only the tensor-core kernel has bounded waits
        e = launch_attn_mma(p, st);
    }
    return e == cudaSuccess ? DDT_OK : cuda_fail(e);
}

}  // namespace

int tree_verify_attn(const ddtree_bf16* q, const ddtree_bf16* k_tree, const ddtree_bf16* v_tree,
                     const ddtree_bf16* k_cache, const ddtree_bf16* v_cache, int num_pages,
                     int page_size, const int32_t* page_table, int max_pages,
                     const int32_t* ctx_len, const uint32_t* vis, const int32_t* n_nodes,
                     int B, int N, int Hq, int Hkv, int Dh, float scale, ddtree_bf16* out,
                     float* lse, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                     void* stream) {
    TraceRange trace("tree_verify_attn");
    return attn_call(q, k_tree, v_tree, k_cache, v_cache, num_pages, page_size, page_table, max_pages,
                     ctx_len, vis, n_nodes, B, N, Hq, Hkv, Dh, scale, out, lse, workspace,
                     workspace_bytes, dev_status, stream, 0);
}

int ddtree_testing_attn_stall(const ddtree_bf16* q, const ddtree_bf16* k_tree,
                              const ddtree_bf16* v_tree, const ddtree_bf16* k_cache,
                              const ddtree_bf16* v_cache, int num_pages, int page_size,
                              const int32_t* page_table, int max_pages, const int32_t* ctx_len,
                              const uint32_t* vis, const int32_t* n_nodes, int B, int N, int Hq,
                              int Hkv, int Dh, float scale, ddtree_bf16* out, float* lse,
                              void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              void* stream, uint64_t stall_ns) {
    TraceRange trace("ddtree_testing_attn_stall");
    if (stall_ns == 0 || stall_ns > 1000000000ull) return DDT_EINVAL;
    return attn_call(q, k_tree, v_tree, k_cache, v_cache, num_pages, page_size, page_table, max_pages,
                     ctx_len, vis, n_nodes, B, N, Hq, Hkv, Dh, scale, out, lse, workspace,
                     workspace_bytes, dev_status, stream, stall_ns);
}

int ddtree_testing_gumbel(const uint32_t* words, float* out, size_t n, void* stream) {
    TraceRange trace("ddtree_testing_gumbel");
    if (n == 0) return DDT_OK;
    if (!words || !out) return DDT_EINVAL;
    const cudaError_t e = launch_gumbel_probe(words, out, n, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DDT_OK : cuda_fail(e);
}

static int check_walk_args(const float* logits, int V, const int32_t* token,
                           const int32_t* first_child, const int32_t* next_sibling,
                           const int32_t* n_nodes, int B, int N, int D, int32_t* accept_len,
                           int32_t* out_tokens, int32_t* out_nodes, int32_t* bonus) {
    if (B < 0 || V < 1) return DDT_EINVAL;
    if (N < 1 || N > DDT_MAX_NODES || D < 1 || D > DDT_MAX_DEPTH) return DDT_ESHAPE;
    if (B == 0) return DDT_OK;
    if (!logits || !token || !first_child || !next_sibling || !n_nodes || !accept_len ||
        !out_tokens || !out_nodes || !bonus)
        return DDT_EINVAL;
    return DDT_OK;
}

int ddtree_accept_greedy(const float* logits, int V, const int32_t* token,
                         const int32_t* first_child, const int32_t* next_sibling,
                         const int32_t* n_nodes, int B, int N, int D, int32_t* accept_len,
                         int32_t* out_tokens, int32_t* out_nodes, int32_t* bonus,
                         int32_t* walk_stats, int32_t* dev_status, void* stream) {
    TraceRange trace("ddtree_accept_greedy");
    int st = check_walk_args(logits, V, token, first_child, next_sibling, n_nodes, B, N, D,
                             accept_len, out_tokens, out_nodes, bonus);
    if (st != DDT_OK || B == 0) return st;
    cudaError_t e = launch_accept_greedy(logits, V, token, first_child, next_sibling, n_nodes, B,
                                         N, D, accept_len, out_tokens, out_nodes, bonus, walk_stats,
                                         dev_status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DDT_OK : cuda_fail(e);
}

int ddtree_accept_sample(const float* logits, int V, const int32_t* token,
                         const int32_t* first_child, const int32_t* next_sibling,
                         const int32_t* n_nodes, int B, int N, int D, const float* temperature,
                         const uint64_t* seed, uint64_t philox_offset, int32_t* accept_len,
                         int32_t* out_tokens, int32_t* out_nodes, int32_t* bonus,
                         float* margin_stats, int32_t* walk_stats, int32_t* dev_status,
                         void* stream) {
    TraceRange trace("ddtree_accept_sample");
    int st = check_walk_args(logits, V, token, first_child, next_sibling, n_nodes, B, N, D,
                             accept_len, out_tokens, out_nodes, bonus);
    if (st != DDT_OK || B == 0) return st;
    if (!temperature || !seed) return DDT_EINVAL;
    if (philox_offset >> 56) return DDT_EINVAL;
    cudaError_t e = launch_accept_sample(logits, V, token, first_child, next_sibling, n_nodes, B,
                                         N, D, temperature, seed, philox_offset, accept_len,
                                         out_tokens, out_nodes, bonus, margin_stats, walk_stats,
                                         dev_status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DDT_OK : cuda_fail(e);
}

int ddtree_accept_greedy_sample(const float* logits, int V, const int32_t* token,
                                const int32_t* first_child, const int32_t* next_sibling,
                                const int32_t* n_nodes, int B, int N, int D, const float* temperature,
                                const uint64_t* seed, uint64_t philox_offset,
                                int32_t* greedy_accept_len, int32_t* greedy_out_tokens,
                                int32_t* greedy_out_nodes, int32_t* greedy_bonus, int32_t* greedy_walk_stats,
                                int32_t* sample_accept_len, int32_t* sample_out_tokens,
                                int32_t* sample_out_nodes, int32_t* sample_bonus, float* sample_margin_stats,
                                int32_t* sample_walk_stats, int32_t* dev_status, void* stream) {
    TraceRange trace("ddtree_accept_greedy_sample");
    int st = check_walk_args(logits, V, token, first_child, next_sibling, n_nodes, B, N, D,
                             greedy_accept_len, greedy_out_tokens, greedy_out_nodes, greedy_bonus);
    if (st != DDT_OK) return st;
    st = check_walk_args(logits, V, token, first_child, next_sibling, n_nodes, B, N, D,
                         sample_accept_len, sample_out_tokens, sample_out_nodes, sample_bonus);
    if (st != DDT_OK || B == 0) return st;
    if (!temperature || !seed) return DDT_EINVAL;
    if (philox_offset >> 56) return DDT_EINVAL;
    const WalkOut og{greedy_accept_len, greedy_out_tokens, greedy_out_nodes, greedy_bonus, nullptr,
                     greedy_walk_stats};
    const WalkOut os{sample_accept_len, sample_out_tokens, sample_out_nodes, sample_bonus, sample_margin_stats,
                     sample_walk_stats};
    cudaError_t e = launch_accept_both(logits, V, token, first_child, next_sibling, n_nodes, B, N, D,
                                       temperature, seed, philox_offset, og, os, dev_status,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DDT_OK : cuda_fail(e);
}

int ddtree_accept_sample_ratio(const float* logits, const float* draft_logits, int V,
                               const int32_t* token, const int32_t* first_child,
                               const int32_t* next_sibling, const int32_t* n_nodes, int B, int N,
                               int D, const float* temperature, const uint64_t* seed,
                               uint64_t philox_offset, int32_t* accept_len, int32_t* out_tokens,
                               int32_t* out_nodes, int32_t* bonus, float* margin_stats,
                               int32_t* walk_stats, int32_t* dev_status, void* stream) {
    TraceRange trace("ddtree_accept_sample_ratio");
    int st = check_walk_args(logits, V, token, first_child, next_sibling, n_nodes, B, N, D,
                             accept_len, out_tokens, out_nodes, bonus);
    if (st != DDT_OK || B == 0) return st;
    if (!draft_logits || !temperature || !seed) return DDT_EINVAL;
    if (philox_offset >> 56) return DDT_EINVAL;
    cudaError_t e = launch_accept_ratio(logits, draft_logits, V, token, first_child, next_sibling,
                                        n_nodes, B, N, D, temperature, seed, philox_offset,
                                        accept_len, out_tokens, out_nodes, bonus, margin_stats,
                                        walk_stats, dev_status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DDT_OK : cuda_fail(e);
}

int ddtree_commit_kv(const ddtree_bf16* k_tree, const ddtree_bf16* v_tree, const int32_t* out_nodes,
                     const int32_t* accept_len, int B, int N, int D, int Hkv, int Dh,
                     ddtree_bf16* k_cache, ddtree_bf16* v_cache, int num_pages, int page_size,
                     const int32_t* page_table, int max_pages, const int32_t* ctx_len,
                     int32_t* new_ctx_len, int32_t* dev_status, void* stream) {
    TraceRange trace("ddtree_commit_kv");
    if (B < 0 || Hkv < 1 || Dh < 1 || page_size < 1 || max_pages < 1 || num_pages < 1)
        return DDT_EINVAL;
    if (N < 1 || N > DDT_MAX_NODES || D < 1 || D > DDT_MAX_DEPTH ||
        (static_cast<long long>(Hkv) * Dh) % 8 != 0 || static_cast<long long>(Hkv) * Dh > (1 << 20))
        return DDT_ESHAPE;
    if (B == 0) return DDT_OK;
    if (!k_tree || !v_tree || !out_nodes || !accept_len || !k_cache || !v_cache || !page_table ||
        !ctx_len || !new_ctx_len)
        return DDT_EINVAL;
    if (!aligned16(k_tree) || !aligned16(v_tree) || !aligned16(k_cache) || !aligned16(v_cache))
        return DDT_EINVAL;
    cudaError_t e = launch_commit_kv(k_tree, v_tree, out_nodes, accept_len, B, N, D, Hkv, Dh, k_cache,
                                     v_cache, num_pages, page_size, page_table, max_pages, ctx_len,
                                     new_ctx_len, dev_status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DDT_OK : cuda_fail(e);
}

// ---------------------------------------------------------------------------
// the walks over a vocabulary-parallel logits shard (requests split over GPUs by KV head)
// ---------------------------------------------------------------------------

static int check_shard_tree(const int32_t* token, const int32_t* first_child, const int32_t* next_sibling,
                            const int32_t* n_nodes, int B, int N) {
    if (B < 0) return DDT_EINVAL;
    if (N < 1 || N > DDT_MAX_NODES) return DDT_ESHAPE;
    if (B > 0 && (!token || !first_child || !next_sibling || !n_nodes)) return DDT_EINVAL;
    return DDT_OK;
}

int ddtree_shard_walk_begin(int B, int D, int32_t* state, int32_t* accept_len, int32_t* out_tokens,
                            int32_t* out_nodes, int32_t* bonus, void* stream) {
    TraceRange trace("ddtree_shard_walk_begin");
    if (B < 0) return DDT_EINVAL;
    if (D < 1 || D > DDT_MAX_DEPTH) return DDT_ESHAPE;
    if (B == 0) return DDT_OK;
    if (!state || !accept_len || !out_tokens || !out_nodes || !bonus) return DDT_EINVAL;
    cudaError_t e = launch_shard_begin(B, D, state, accept_len, out_tokens, out_nodes, bonus,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DDT_OK : cuda_fail(e);
}

int ddtree_shard_walk_partial(const float* logits_shard, int Vs, int v0, int V, const int32_t* token,
                              const int32_t* first_child, const int32_t* next_sibling,
                              const int32_t* n_nodes, int B, int N, const float* temperature,
                              const int32_t* state, int32_t* record, void* stream) {
    TraceRange trace("ddtree_shard_walk_partial");
    int st = check_shard_tree(token, first_child, next_sibling, n_nodes, B, N);
    if (st != DDT_OK) return st;
    if (Vs < 1 || v0 < 0 || V < 1 || static_cast<long long>(v0) + Vs > V) return DDT_EINVAL;
    if (B == 0) return DDT_OK;
    if (!logits_shard || !state || !record) return DDT_EINVAL;
    cudaError_t e = launch_shard_partial(logits_shard, Vs, v0, token, first_child, next_sibling, n_nodes, B, N,
                                         temperature, state, record, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DDT_OK : cuda_fail(e);
}

int ddtree_shard_walk_advance(const int32_t* records, int world, int V, const int32_t* token,
                              const int32_t* first_child, const int32_t* next_sibling,
                              const int32_t* n_nodes, int B, int N, int D, const float* temperature,
                              const uint64_t* seed, uint64_t philox_offset, int32_t* state,
                              int32_t* accept_len, int32_t* out_tokens, int32_t* out_nodes, int32_t* bonus,
                              int32_t* dev_status, void* stream) {
    TraceRange trace("ddtree_shard_walk_advance");
    int st = check_shard_tree(token, first_child, next_sibling, n_nodes, B, N);
    if (st != DDT_OK) return st;
    if (world < 1 || world > 1024 || V < 1) return DDT_EINVAL;
    if (D < 1 || D > DDT_MAX_DEPTH) return DDT_ESHAPE;
    if (B == 0) return DDT_OK;
    if (!records || !state || !accept_len || !out_tokens || !out_nodes || !bonus) return DDT_EINVAL;
    if (temperature && (!seed || (philox_offset >> 56))) return DDT_EINVAL;
    cudaError_t e = launch_shard_advance(records, world, B, V, token, first_child, next_sibling, n_nodes, N, D,
                                         temperature, seed, philox_offset, state, accept_len, out_tokens,
                                         out_nodes, bonus, dev_status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DDT_OK : cuda_fail(e);
}

int ddtree_shard_walk_bonus(const float* logits_shard, int Vs, int v0, int V, const int32_t* token,
                            const int32_t* first_child, const int32_t* next_sibling, const int32_t* n_nodes,
                            int B, int N, const float* temperature, const uint64_t* seed,
                            uint64_t philox_offset, const int32_t* state, int64_t* key, void* stream) {
    TraceRange trace("ddtree_shard_walk_bonus");
    int st = check_shard_tree(token, first_child, next_sibling, n_nodes, B, N);
    if (st != DDT_OK) return st;
    if (Vs < 1 || v0 < 0 || V < 1 || static_cast<long long>(v0) + Vs > V) return DDT_EINVAL;
    if (B == 0) return DDT_OK;
    if (!logits_shard || !temperature || !seed || !state || !key || (philox_offset >> 56)) return DDT_EINVAL;
    cudaError_t e = launch_shard_bonus(logits_shard, Vs, v0, token, first_child, next_sibling, n_nodes, B, N,
                                       temperature, seed, philox_offset, state,
                                       reinterpret_cast<unsigned long long*>(key),
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DDT_OK : cuda_fail(e);
}

int ddtree_shard_walk_finish(const int64_t* keys, int world, int B, int D, int32_t* state,
                             int32_t* accept_len, int32_t* out_tokens, int32_t* bonus, void* stream) {
    TraceRange trace("ddtree_shard_walk_finish");
    if (B < 0 || world < 1 || world > 1024) return DDT_EINVAL;
    if (D < 1 || D > DDT_MAX_DEPTH) return DDT_ESHAPE;
    if (B == 0) return DDT_OK;
    if (!keys || !state || !accept_len || !out_tokens || !bonus) return DDT_EINVAL;
    cudaError_t e = launch_shard_finish(reinterpret_cast<const unsigned long long*>(keys), world, B, D, state,
                                        accept_len, out_tokens, bonus, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DDT_OK : cuda_fail(e);
}

}  // extern "C"
