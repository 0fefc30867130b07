// tree_verify_attn_noalloc: tree attention for callers that cannot allocate.
//
// Some callers have no way to get device memory at run time: a serving engine
// that reserves nearly all of HBM for its own KV pool at start-up and gives
// its plugins no allocator, or a hot loop where a cudaMalloc would block the
// device and stall every stream. tree_verify_attn needs a scratch workspace
// for its split-KV partial results; this entry point takes that scratch from
// a fixed array compiled into the library instead of from the caller.
//
// The array is a file-scope __device__ object of kNoAllocScratchBytes. Every
// GPU on which the library's module is loaded holds it until the process
// exits. Its device address is looked up with cudaGetSymbolAddress by the
// first call on each device (with that device current) and cached together
// with the id of the CUDA context it belongs to; a later call under another
// context (after cudaDeviceReset, or under a context the caller made current
// through the driver API) looks it up again, so a stale address is never
// used. Make the first call on a device, and the first after a reset, before
// any stream capture. All calls share the one array and its contents persist
// between calls: the attention kernels write every scratch word they read
// within a call, so nothing needs clearing, but two calls that overlap on the
// GPU (different streams, no ordering between them) race on the array.
#include <climits>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "trace.h"

namespace ddt {
void set_last_error(const char* what, cudaError_t e);
}

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;   // 64 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
struct ScratchEntry {
    unsigned long long ctx_id;   // 0: not looked up yet
    void* ptr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

// Id of the CUDA context current on this thread (0 if none or unavailable).
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_attn_scratch in the current device's current context.
int scratch_on_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        ddt::set_last_error("cudaGetDevice", e);
        return DDT_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return DDT_EINVAL;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchEntry& ent = g_scratch[dev];
    const unsigned long long id = current_context_id();
    if (ent.ctx_id == 0 || id == 0 || id != ent.ctx_id) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_scratch);   // also makes the primary context current
        if (e != cudaSuccess || p == nullptr) {
            ddt::set_last_error("cudaGetSymbolAddress(g_attn_scratch)", e);
            return DDT_ECUDA;
        }
        ent.ptr = p;
        ent.ctx_id = current_context_id();   // 0 keeps the next call looking it up again
    }
    *out = ent.ptr;
    return DDT_OK;
}

}  // namespace

extern "C" {

size_t tree_verify_attn_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

int tree_verify_attn_noalloc(const ddtree_bf16* q, const ddtree_bf16* k_tree,
                             const ddtree_bf16* v_tree, const ddtree_bf16* k_cache,
                             const ddtree_bf16* v_cache, int num_pages, int page_size,
                             const int32_t* page_table, int max_pages, const int32_t* ctx_len,
                             const uint32_t* vis, const int32_t* n_nodes, int B, int N, int Hq,
                             int Hkv, int Dh, float scale, ddtree_bf16* out, float* lse,
                             int32_t* dev_status, void* stream) {
    ddt::TraceRange trace("tree_verify_attn_noalloc");
    const long long max_ctx = static_cast<long long>(max_pages) * page_size;
    if (max_pages > 0 && page_size > 0 && max_ctx <= INT_MAX && B > 0) {
        const size_t need = tree_verify_attn_workspace_size(B, N, Hq, Hkv, Dh,
                                                            static_cast<int>(max_ctx));
        if (need > kNoAllocScratchBytes) return DDT_ESCRATCH;
    }
    void* scratch = nullptr;
    const int st = scratch_on_current_device(&scratch);
    if (st != DDT_OK) return st;
    return tree_verify_attn(q, k_tree, v_tree, k_cache, v_cache, num_pages, page_size,
                            page_table, max_pages, ctx_len, vis, n_nodes, B, N, Hq, Hkv, Dh,
                            scale, out, lse, scratch, kNoAllocScratchBytes, dev_status, stream);
}

}  // extern "C"
