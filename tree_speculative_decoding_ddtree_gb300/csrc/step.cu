// ddtree_step_*: the verify step (build -> attention -> walk -> commit)
// recorded once into a CUDA graph by stream capture and replayed per step.
//
// Method: "The Architecture of Speculative Decoding: Dissecting DDTree's
// Tree-Parallel Evaluation Strategy", Section 1 steps 2-5; "The Pivot Point",
// The Strategic Decision (the verify path runs under CUDA graphs). The calls
// are the public ones, so each checks its arguments as it does alone.
#include <new>

#include "common.cuh"
#include "trace.h"

namespace ddt {
int cuda_fail(cudaError_t e);
}

struct ddtree_step {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};

namespace {

int record_step(const ddtree_step_args& a, cudaStream_t s) {
    const int N = a.budget + 1;
    int st = ddtree_build(a.topk_logp, a.topk_tok, a.root_tok, a.ctx_len, a.B, a.D, a.K, a.budget,
                          a.parent, a.depth, a.token, a.rank, a.pos, a.score, a.first_child,
                          a.next_sibling, a.vis, a.n_nodes, a.dev_status, s);
    if (st != DDT_OK) return st;
    st = tree_verify_attn(a.q, a.k_tree, a.v_tree, a.k_cache, a.v_cache, a.num_pages, a.page_size,
                          a.page_table, a.max_pages, a.ctx_len, a.vis, a.n_nodes, a.B, N, a.Hq, a.Hkv,
                          a.Dh, a.scale, a.attn_out, a.lse, a.workspace, a.workspace_bytes,
                          a.dev_status, s);
    if (st != DDT_OK) return st;
    if (a.walk == 0)
        st = ddtree_accept_greedy(a.logits, a.V, a.token, a.first_child, a.next_sibling, a.n_nodes,
                                  a.B, N, a.D, a.accept_len, a.out_tokens, a.out_nodes, a.bonus,
                                  nullptr, a.dev_status, s);
    else if (a.walk == 1)
        st = ddtree_accept_sample(a.logits, a.V, a.token, a.first_child, a.next_sibling, a.n_nodes,
                                  a.B, N, a.D, a.temperature, a.seed, a.philox_offset, a.accept_len,
                                  a.out_tokens, a.out_nodes, a.bonus, nullptr, nullptr, a.dev_status, s);
    else
        st = ddtree_accept_sample_ratio(a.logits, a.draft_logits, a.V, a.token, a.first_child,
                                        a.next_sibling, a.n_nodes, a.B, N, a.D, a.temperature, a.seed,
                                        a.philox_offset, a.accept_len, a.out_tokens, a.out_nodes,
                                        a.bonus, nullptr, nullptr, a.dev_status, s);
    if (st != DDT_OK) return st;
    return ddtree_commit_kv(a.k_tree, a.v_tree, a.out_nodes, a.accept_len, a.B, N, a.D, a.Hkv, a.Dh,
                            a.k_cache, a.v_cache, a.num_pages, a.page_size, a.page_table,
                            a.max_pages, a.ctx_len, a.new_ctx_len ? a.new_ctx_len : a.ctx_len,
                            a.dev_status, s);
}

}  // namespace

extern "C" {

size_t ddtree_step_args_size(void) { return sizeof(ddtree_step_args); }

int ddtree_step_create(const ddtree_step_args* args, ddtree_step** out) {
    ddt::TraceRange trace("ddtree_step_create");
    if (!out) return DDT_EINVAL;
    *out = nullptr;
    if (!args || args->walk < 0 || args->walk > 2) return DDT_EINVAL;
    if (args->B < 1) return DDT_ESHAPE;   // an empty step has nothing to record
    cudaStream_t s = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e != cudaSuccess) return ddt::cuda_fail(e);
    e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
        cudaStreamDestroy(s);
        return ddt::cuda_fail(e);
    }
    const int st = record_step(*args, s);
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(s, &graph);
    cudaStreamDestroy(s);
    if (st != DDT_OK || e != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        return st != DDT_OK ? st : ddt::cuda_fail(e);
    }
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    if (e != cudaSuccess) {
        cudaGraphDestroy(graph);
        return ddt::cuda_fail(e);
    }
    ddtree_step* step = new (std::nothrow) ddtree_step;
    if (!step) {
        cudaGraphExecDestroy(exec);
        cudaGraphDestroy(graph);
        return DDT_EINVAL;
    }
    step->graph = graph;
    step->exec = exec;
    *out = step;
    return DDT_OK;
}

int ddtree_step_launch(ddtree_step* step, void* stream) {
    ddt::TraceRange trace("ddtree_step_launch");
    if (!step || !step->exec) return DDT_EINVAL;
    cudaError_t e = cudaGraphLaunch(step->exec, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DDT_OK : ddt::cuda_fail(e);
}

void ddtree_step_destroy(ddtree_step* step) {
    if (!step) return;
    if (step->exec) cudaGraphExecDestroy(step->exec);
    if (step->graph) cudaGraphDestroy(step->graph);
    delete step;
}

}  // extern "C"
