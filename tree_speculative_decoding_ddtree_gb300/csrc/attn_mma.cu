// tree_verify_attn, warp-MMA path: split-KV flash attention of all tree rows
// of one (request, KV head) over the paged context plus the tree rows.
//
// Method: "The Architecture of Speculative Decoding: Dissecting DDTree's
// Tree-Parallel Evaluation Strategy", Section 1 step 4 (all budget+1 nodes in
// one pass under the tree mask) and Section 2 (the context KV is read once
// and shared by every node); "The Pivot Point", The Design Constraint (load
// contexts once).
//
// Layout of the work: one CTA owns all R = N * (Hq/Hkv) query rows of one
// (request, KV head) (up to kMaxRowsPerCta; more rows go to further row
// groups) and one chunk of the context, so each K/V tile is fetched from HBM
// once and used by every tree row and every head of the GQA group. Row r of a
// CTA is (node r / G, head r % G). Keys stream through shared memory in tiles
// of 64 with cp.async double buffering; QK^T and PV run on mma.sync m16n8k16
// (bf16 in, fp32 accumulate) with an online softmax in the exp2 domain. The
// last chunk of a request also takes the tree keys, masked per row by the
// ancestor bitmask. Chunks of a multi-chunk request write unnormalised fp32
// partials that a second launch merges.
#include "common.cuh"
#include <type_traits>

#include "attn.cuh"

namespace ddt {

constexpr int kKeyTile = 64;
constexpr int kMaxWarps = kMaxRowsPerCta / 16;     // 18

DDT_DEVINL uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

DDT_DEVINL void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n"
                 :: "r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
DDT_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
DDT_DEVINL void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" :: "n"(N) : "memory"); }

DDT_DEVINL void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
DDT_DEVINL void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

DDT_DEVINL void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

DDT_DEVINL uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <int DH>
struct MmaTile {
    static constexpr int kRowBytes = DH * 2 + 16;             // +16 B: conflict-free ldmatrix
    static constexpr int kTileBytes = kKeyTile * kRowBytes;
    static constexpr int kChunks = DH / 8;                     // 16-byte chunks per row
};

template <int DH>
__global__ void __launch_bounds__(32 * kMaxWarps, 1)
attn_mma_kernel(AttnParams p) {
    using T = MmaTile<DH>;
    extern __shared__ __align__(128) unsigned char smem[];
    const int b = blockIdx.z;
    const int kvh = blockIdx.y / p.n_groups;
    const int grp = blockIdx.y % p.n_groups;
    const int chunk = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x;

    int L = p.ctx_len[b];
    bool bad = false;
    if (L < 0 || L > p.max_pages * p.page_size) { bad = true; L = 0; }
    const int nt_ctx = (L + kKeyTile - 1) / kKeyTile;
    const int nchunks = nt_ctx > 0 ? (nt_ctx + p.tiles_per_chunk - 1) / p.tiles_per_chunk : 1;
    if (chunk >= nchunks) return;
    int nn = p.n_nodes[b];
    if (nn < 0 || nn > p.N) { bad = true; nn = 0; }
    const int t_begin = chunk * p.tiles_per_chunk;
    const int n_ctx_tiles = max(0, min(nt_ctx, t_begin + p.tiles_per_chunk) - t_begin);
    const int n_tree_tiles = (chunk == nchunks - 1 && !bad) ? (p.N + kKeyTile - 1) / kKeyTile : 0;
    const int n_tiles = bad ? 0 : n_ctx_tiles + n_tree_tiles;
    if (bad && chunk == 0 && tid == 0) report(p.dev_status, DDT_DEV_BAD_CTX);

    const int row0 = grp * p.rows_per_group;
    const int rows = min(p.R - row0, p.rows_per_group);
    const int G = p.G;

    unsigned char* q_s = smem;
    unsigned char* k_s = q_s + kMaxRowsPerCta * T::kRowBytes;
    unsigned char* v_s = k_s + 2 * T::kTileBytes;

    // ---- Q rows of this (request, KV head, row group) -> shared memory
    for (int x = tid; x < nthreads / 2 * T::kChunks; x += nthreads) {
        const int lr = x / T::kChunks, ch = x % T::kChunks;
        if (lr >= ((rows + 15) & ~15)) continue;
        const int r = row0 + lr;
        const bool ok = lr < rows;
        const int i = ok ? r / G : 0, h = kvh * G + (ok ? r % G : 0);
        const bf16_t* src = p.q + ((static_cast<size_t>(b) * p.N + i) * p.Hq + h) * DH + ch * 8;
        cp_async16(smem_addr(q_s + lr * T::kRowBytes + ch * 16), src, ok);
    }

    auto load_tile = [&](int t, int stage) {
        unsigned char* ks = k_s + stage * T::kTileBytes;
        unsigned char* vs = v_s + stage * T::kTileBytes;
        if (t < n_ctx_tiles) {
            const int kt0 = (t_begin + t) * kKeyTile;
            for (int x = tid; x < kKeyTile * T::kChunks; x += nthreads) {
                const int key = x / T::kChunks, ch = x % T::kChunks;
                const int kk = kt0 + key;
                bool ok = kk < L;
                size_t off = 0;
                if (ok) {
                    const int page = p.page_table[static_cast<size_t>(b) * p.max_pages + kk / p.page_size];
                    if (page < 0 || page >= p.num_pages) {
                        ok = false;
                        if (ch == 0) report(p.dev_status, DDT_DEV_BAD_PAGE);
                    } else {
                        off = ((static_cast<size_t>(page) * p.page_size + kk % p.page_size) * p.Hkv + kvh) * DH + ch * 8;
                    }
                }
                cp_async16(smem_addr(ks + key * T::kRowBytes + ch * 16), p.k_cache + off, ok);
                cp_async16(smem_addr(vs + key * T::kRowBytes + ch * 16), p.v_cache + off, ok);
            }
        } else {
            const int j0 = (t - n_ctx_tiles) * kKeyTile;
            for (int x = tid; x < kKeyTile * T::kChunks; x += nthreads) {
                const int key = x / T::kChunks, ch = x % T::kChunks;
                const int j = j0 + key;
                const bool ok = j < nn;
                const size_t off = ok ? ((static_cast<size_t>(b) * p.N + j) * p.Hkv + kvh) * DH + ch * 8 : 0;
                cp_async16(smem_addr(ks + key * T::kRowBytes + ch * 16), p.k_tree + off, ok);
                cp_async16(smem_addr(vs + key * T::kRowBytes + ch * 16), p.v_tree + off, ok);
            }
        }
    };

    // per-thread rows: lane/4 and lane/4 + 8 of this warp's 16-row block
    const int lr_base = warp * 16 + (lane >> 2);
    uint32_t visw[2][4];
    int node_of[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int lr = lr_base + rr * 8;
        const int r = row0 + lr;
        const int i = (lr < rows) ? r / G : -1;
        node_of[rr] = i;
#pragma unroll
        for (int w = 0; w < 4; ++w)
            visw[rr][w] = (i >= 0 && i < nn && w < p.W) ? p.vis[(static_cast<size_t>(b) * p.N + i) * p.W + w] : 0u;
    }
    const bool warp_active = warp * 16 < rows;

    float o_acc[DH / 8][4];
#pragma unroll
    for (int d = 0; d < DH / 8; ++d) o_acc[d][0] = o_acc[d][1] = o_acc[d][2] = o_acc[d][3] = 0.0f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.0f, 0.0f};

    if (n_tiles > 0) load_tile(0, 0);
    cp_async_commit();

    for (int t = 0; t < n_tiles; ++t) {
        if (t + 1 < n_tiles) load_tile(t + 1, (t + 1) & 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (warp_active) {
            const unsigned char* ks = k_s + (t & 1) * T::kTileBytes;
            const unsigned char* vs = v_s + (t & 1) * T::kTileBytes;
            float s[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.0f;
#pragma unroll
            for (int kstep = 0; kstep < DH / 16; ++kstep) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(smem_addr(q_s + (warp * 16 + (lane & 15)) * T::kRowBytes + (kstep * 16 + (lane >> 4) * 8) * 2),
                        a0, a1, a2, a3);
#pragma unroll
                for (int nb2 = 0; nb2 < 4; ++nb2) {
                    uint32_t b0, b1, b2, b3;
                    const int key = nb2 * 16 + (lane >> 4) * 8 + (lane & 7);
                    ldsm_x4(smem_addr(ks + key * T::kRowBytes + (kstep * 16 + ((lane >> 3) & 1) * 8) * 2),
                            b0, b1, b2, b3);
                    mma_bf16(s[2 * nb2], a0, a1, a2, a3, b0, b1);
                    mma_bf16(s[2 * nb2 + 1], a0, a1, a2, a3, b2, b3);
                }
            }
            // scale into the log2 domain and mask
            const bool is_ctx = t < n_ctx_tiles;
            const int key0 = is_ctx ? (t_begin + t) * kKeyTile : (t - n_ctx_tiles) * kKeyTile;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int rr = e >> 1;
                    const int key = key0 + n * 8 + 2 * (lane & 3) + (e & 1);
                    bool ok;
                    if (is_ctx) ok = key < L;
                    else ok = key < nn && ((pick4(visw[rr], key >> 5) >> (key & 31)) & 1u);
                    s[n][e] = ok ? s[n][e] * p.scale_log2 : -INFINITY;
                }
            }
            // online softmax per row
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                float mx = -INFINITY;
#pragma unroll
                for (int n = 0; n < 8; ++n) mx = fmaxf(mx, fmaxf(s[n][2 * rr], s[n][2 * rr + 1]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_run[rr], mx);
                const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
                const float alpha = exp2f(m_run[rr] - m_use);
                float ls = 0.0f;
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    s[n][2 * rr] = exp2f(s[n][2 * rr] - m_use);
                    s[n][2 * rr + 1] = exp2f(s[n][2 * rr + 1] - m_use);
                    ls += s[n][2 * rr] + s[n][2 * rr + 1];
                }
                l_run[rr] = l_run[rr] * alpha + ls;
                m_run[rr] = m_new;
#pragma unroll
                for (int d = 0; d < DH / 8; ++d) { o_acc[d][2 * rr] *= alpha; o_acc[d][2 * rr + 1] *= alpha; }
            }
            // O += P V
#pragma unroll
            for (int kk = 0; kk < kKeyTile / 16; ++kk) {
                const uint32_t a0 = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
                const uint32_t a1 = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
                const uint32_t a2 = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
                const uint32_t a3 = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
                for (int dn2 = 0; dn2 < DH / 16; ++dn2) {
                    uint32_t b0, b1, b2, b3;
                    const int key = kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
                    ldsm_x4_t(smem_addr(vs + key * T::kRowBytes + (dn2 * 16 + (lane >> 4) * 8) * 2),
                              b0, b1, b2, b3);
                    mma_bf16(o_acc[2 * dn2], a0, a1, a2, a3, b0, b1);
                    mma_bf16(o_acc[2 * dn2 + 1], a0, a1, a2, a3, b2, b3);
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // ---- epilogue
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        float l = l_run[rr];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        l_run[rr] = l;
    }
    if (!warp_active) return;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int lr = lr_base + rr * 8;
        if (lr >= rows) continue;
        const int r = row0 + lr;
        const int i = r / G, h = kvh * G + r % G;
        const bool real = node_of[rr] >= 0 && i < nn && !bad;
        if (nchunks == 1) {
            const float l = l_run[rr];
            const float inv = (real && l > 0.0f) ? 1.0f / l : 0.0f;
            bf16_t* dst = p.out + ((static_cast<size_t>(b) * p.N + i) * p.Hq + h) * DH + 2 * (lane & 3);
#pragma unroll
            for (int d = 0; d < DH / 8; ++d) {
                const uint32_t v = pack_bf16(o_acc[d][2 * rr] * inv, o_acc[d][2 * rr + 1] * inv);
                *reinterpret_cast<uint32_t*>(dst + d * 8) = v;
            }
            if (p.lse && (lane & 3) == 0)
                p.lse[(static_cast<size_t>(b) * p.N + i) * p.Hq + h] =
                    (real && l > 0.0f) ? (m_run[rr] + log2f(l)) * 0.69314718055994531f : -INFINITY;
        } else {
            const size_t slot = (static_cast<size_t>(b) * p.Hkv + kvh) * p.max_chunks + chunk;
            float* dst = p.ws_o + (slot * p.R + r) * DH + 2 * (lane & 3);
#pragma unroll
            for (int d = 0; d < DH / 8; ++d)
                *reinterpret_cast<float2*>(dst + d * 8) = make_float2(o_acc[d][2 * rr], o_acc[d][2 * rr + 1]);
            if ((lane & 3) == 0) p.ws_ml[slot * p.R + r] = make_float2(m_run[rr], l_run[rr]);
        }
    }
}

// Merge the chunk partials of every multi-chunk (request, KV head): one warp
// per query row. The lanes read the chunks' (max, sum) pairs in parallel for
// the common max and the total; then each lane owns DH/32 contiguous features
// and adds the chunks' vectors, weighted by the chunk's exp2(max - M), with
// the weights handed round by shuffles so several chunk loads are in flight.
template <int DH>
__global__ void __launch_bounds__(256)
attn_combine_kernel(AttnParams p) {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");   // the walk may start; it waits for this grid
    const int b = blockIdx.z, kvh = blockIdx.y;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= p.R) return;
    int L = p.ctx_len[b];
    if (L < 0 || L > p.max_pages * p.page_size) return;
    const int nt_ctx = (L + kKeyTile - 1) / kKeyTile;
    const int nchunks = nt_ctx > 0 ? (nt_ctx + p.tiles_per_chunk - 1) / p.tiles_per_chunk : 1;
    if (nchunks == 1) return;
    int nn = p.n_nodes[b];
    const bool nn_ok = nn >= 0 && nn <= p.N;
    const int G = p.G;
    const int i = r / G, h = kvh * G + r % G;
    constexpr int PER = DH / 32;
    bf16_t* dst = p.out + ((static_cast<size_t>(b) * p.N + i) * p.Hq + h) * DH + lane * PER;
    if (!nn_ok) {
        // A malformed tree: the main kernel flagged it and may have left this
        // request's partials unwritten, so they are not read. Zeros, lse -inf.
#pragma unroll
        for (int e = 0; e < PER; e += 2) *reinterpret_cast<uint32_t*>(dst + e) = 0u;
        if (p.lse && lane == 0) p.lse[(static_cast<size_t>(b) * p.N + i) * p.Hq + h] = -INFINITY;
        return;
    }
    const size_t slot0 = (static_cast<size_t>(b) * p.Hkv + kvh) * p.max_chunks;
    const float2* ml = p.ws_ml + slot0 * p.R + r;            // chunk c at ml[c * R]
    float M = -INFINITY;
    for (int c = lane; c < nchunks; c += 32) M = fmaxf(M, ml[static_cast<size_t>(c) * p.R].x);
    M = warp_max_f(M);
    const float m_use = (M == -INFINITY) ? 0.0f : M;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.0f;
    float lpart = 0.0f;
    const float* o_row = p.ws_o + (slot0 * p.R + r) * DH + lane * PER;
    const size_t o_stride = static_cast<size_t>(p.R) * DH;   // one chunk
    for (int c0 = 0; c0 < nchunks; c0 += 32) {
        float wl = 0.0f;
        if (c0 + lane < nchunks) {
            const float2 v = ml[static_cast<size_t>(c0 + lane) * p.R];
            wl = exp2f(v.x - m_use);
            lpart += v.y * wl;
        }
        const int cn = min(32, nchunks - c0);
#pragma unroll 4
        for (int k = 0; k < cn; ++k) {
            const float w = __shfl_sync(0xffffffffu, wl, k);
            const float* src = o_row + static_cast<size_t>(c0 + k) * o_stride;
            if constexpr (PER == 4) {
                const float4 v = *reinterpret_cast<const float4*>(src);
                acc[0] += v.x * w; acc[1] += v.y * w; acc[2] += v.z * w; acc[3] += v.w * w;
            } else {
                const float2 v = *reinterpret_cast<const float2*>(src);
                acc[0] += v.x * w; acc[1] += v.y * w;
            }
        }
    }
    const float lsum = warp_sum_f(lpart);
    const bool real = i < nn;
    const float inv = (real && lsum > 0.0f) ? 1.0f / lsum : 0.0f;
#pragma unroll
    for (int e = 0; e < PER; e += 2)
        *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16(acc[e] * inv, acc[e + 1] * inv);
    if (p.lse && lane == 0)
        p.lse[(static_cast<size_t>(b) * p.N + i) * p.Hq + h] =
            (real && lsum > 0.0f) ? (M + log2f(lsum)) * 0.69314718055994531f : -INFINITY;
}

// The same merge for launches with few rows per SM (a small batch split into
// many chunks), where occupancy cannot hide the load latency: the chunks'
// vectors are loaded kMergeBatch at a time, all issued before any of them is
// used and before the common max is known (they do not depend on it); the
// lanes read the chunks' (max, sum) pairs in parallel for the common max and
// the total, and the weights exp2(max_c - M) reach every lane by shuffles.
// Same arithmetic in the same order as attn_combine_kernel.
constexpr int kMergeBatch = 8;
static_assert(32 % kMergeBatch == 0, "a batch of chunks stays within one lane word of weights");
template <int DH>
__global__ void __launch_bounds__(256)
attn_combine_wide_kernel(AttnParams p) {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");   // the walk may start; it waits for this grid
    const int b = blockIdx.z, kvh = blockIdx.y;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= p.R) return;
    int L = p.ctx_len[b];
    if (L < 0 || L > p.max_pages * p.page_size) return;
    const int nt_ctx = (L + kKeyTile - 1) / kKeyTile;
    const int nchunks = nt_ctx > 0 ? (nt_ctx + p.tiles_per_chunk - 1) / p.tiles_per_chunk : 1;
    if (nchunks == 1) return;
    int nn = p.n_nodes[b];
    const bool nn_ok = nn >= 0 && nn <= p.N;
    const int G = p.G;
    const int i = r / G, h = kvh * G + r % G;
    constexpr int PER = DH / 32;
    using VecT = typename std::conditional<PER == 4, float4, float2>::type;
    bf16_t* dst = p.out + ((static_cast<size_t>(b) * p.N + i) * p.Hq + h) * DH + lane * PER;
    if (!nn_ok) {
        // A malformed tree: the main kernel flagged it and may have left this
        // request's partials unwritten, so they are not read. Zeros, lse -inf.
#pragma unroll
        for (int e = 0; e < PER; e += 2) *reinterpret_cast<uint32_t*>(dst + e) = 0u;
        if (p.lse && lane == 0) p.lse[(static_cast<size_t>(b) * p.N + i) * p.Hq + h] = -INFINITY;
        return;
    }
    const size_t slot0 = (static_cast<size_t>(b) * p.Hkv + kvh) * p.max_chunks;
    const float2* ml = p.ws_ml + slot0 * p.R + r;            // chunk c at ml[c * R]
    const float* o_row = p.ws_o + (slot0 * p.R + r) * DH + lane * PER;
    const size_t o_stride = static_cast<size_t>(p.R) * DH;   // one chunk
    // the first batch of vectors and every chunk's (max, sum), all in flight together
    VecT v[kMergeBatch];
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k)
        if (k < nchunks) v[k] = *reinterpret_cast<const VecT*>(o_row + static_cast<size_t>(k) * o_stride);
    float2 mlv[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int c = lane + 32 * q;
        mlv[q] = c < nchunks ? ml[static_cast<size_t>(c) * p.R] : make_float2(-INFINITY, 0.0f);
    }
    float M = fmaxf(mlv[0].x, mlv[1].x);
    for (int c = lane + 64; c < nchunks; c += 32) M = fmaxf(M, ml[static_cast<size_t>(c) * p.R].x);
    M = warp_max_f(M);
    const float m_use = (M == -INFINITY) ? 0.0f : M;
    // lane l holds the weights of chunks l and l + 32
    const float w0 = exp2f(mlv[0].x - m_use), w1 = exp2f(mlv[1].x - m_use);
    float lpart = mlv[0].y * w0 + mlv[1].y * w1;
    for (int c = lane + 64; c < nchunks; c += 32) {
        const float2 mv = ml[static_cast<size_t>(c) * p.R];
        lpart += mv.y * exp2f(mv.x - m_use);
    }
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.0f;
    for (int c0 = 0; c0 < nchunks; c0 += kMergeBatch) {
        if (c0 > 0) {
#pragma unroll
            for (int k = 0; k < kMergeBatch; ++k)
                if (c0 + k < nchunks) v[k] = *reinterpret_cast<const VecT*>(o_row + static_cast<size_t>(c0 + k) * o_stride);
        }
        // a batch lies within chunks [0, 32) or [32, 64) (kMergeBatch divides 32)
        const float wsel = c0 < 32 ? w0 : w1;
#pragma unroll
        for (int k = 0; k < kMergeBatch; ++k) {
            const int c = c0 + k;
            float w;
            if (c0 < 64) w = __shfl_sync(0xffffffffu, wsel, c & 31);
            else w = c < nchunks ? exp2f(ml[static_cast<size_t>(c) * p.R].x - m_use) : 0.0f;
            if (c < nchunks) {
                if constexpr (PER == 4) {
                    acc[0] += v[k].x * w; acc[1] += v[k].y * w; acc[2] += v[k].z * w; acc[3] += v[k].w * w;
                } else {
                    acc[0] += v[k].x * w; acc[1] += v[k].y * w;
                }
            }
        }
    }
    const float lsum = warp_sum_f(lpart);
    const bool real = i < nn;
    const float inv = (real && lsum > 0.0f) ? 1.0f / lsum : 0.0f;
#pragma unroll
    for (int e = 0; e < PER; e += 2)
        *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16(acc[e] * inv, acc[e + 1] * inv);
    if (p.lse && lane == 0)
        p.lse[(static_cast<size_t>(b) * p.N + i) * p.Hq + h] =
            (real && lsum > 0.0f) ? (M + log2f(lsum)) * 0.69314718055994531f : -INFINITY;
}

template <int DH>
static cudaError_t launch_dh(const AttnParams& p, cudaStream_t stream) {
    using T = MmaTile<DH>;
    const size_t smem = kMaxRowsPerCta * T::kRowBytes + 4 * T::kTileBytes;
    cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int warps = (p.rows_per_group + 15) / 16;
    const dim3 grid(p.max_chunks, p.Hkv * p.n_groups, p.B);
    attn_mma_kernel<DH><<<grid, 32 * warps, smem, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_attn_combine(p, stream);
}

cudaError_t launch_attn_mma(const AttnParams& p, cudaStream_t stream) {
    return p.Dh == 128 ? launch_dh<128>(p, stream) : launch_dh<64>(p, stream);
}

cudaError_t launch_attn_combine(const AttnParams& p, cudaStream_t stream) {
    if (p.max_chunks <= 1) return cudaSuccess;
    const dim3 g2((p.R + 7) / 8, p.Hkv, p.B);
    if (p.merge_wide) {
        if (p.Dh == 128) attn_combine_wide_kernel<128><<<g2, 256, 0, stream>>>(p);
        else attn_combine_wide_kernel<64><<<g2, 256, 0, stream>>>(p);
    } else {
        if (p.Dh == 128) attn_combine_kernel<128><<<g2, 256, 0, stream>>>(p);
        else attn_combine_kernel<64><<<g2, 256, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace ddt
