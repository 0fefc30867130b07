// tree_verify_attn, tensor-core path for sm_103a (tcgen05 + TMA + TMEM).
//
// Method: "The Architecture of Speculative Decoding: Dissecting DDTree's
// Tree-Parallel Evaluation Strategy", Section 1 step 4 (all budget+1 tree
// rows in one pass under the tree mask) and Section 2 (the context KV is
// loaded once and shared by all rows); "The Pivot Point", The Design
// Constraint (load contexts once).
//
// One CTA owns one row group of one (request, KV head) and one chunk of its
// context (a request's context is cut into chunks of equal length; with a
// split context, warp 0 of each CTA first maps the block index to a work
// item so that the longest chunks are dispatched first). The R = N * G rows
// (node-major: row r = node r / G, head r % G) fall in row groups of two
// tensor-core tiles; a tile holds the whole nodes that fit in 128 rows (128
// rows when G divides 128, else 128 - 128 % G), and the last group takes the
// rest: two tiles plus up to 8 leftover rows, or fewer rows. A group's rows:
//
//   warp 0       TMA producer: Q once, then paged K/V tiles of 64 keys (one
//                page box per half of the head dim, 128-byte swizzle) into a
//                4-stage ring; zeroes V rows past the valid keys of a ragged
//                tile so masked keys contribute exact zeros.
//   warp 1       allocates TMEM; one lane issues tcgen05.mma:
//                S_t = Q_t K^T (Q from TMEM, K K-major in shared memory) and
//                O_t += P_t V (P from TMEM, V MN-major in shared memory),
//                ping-ponging the two tiles so the tensor core works on one
//                tile while the other tile's softmax runs.
//   warps 4-7,   one thread per row of tile 0 / tile 1 (its TMEM lane): load
//   warps 8-11   S, mask (context tail, ancestor bitmask on the tree tile),
//                online softmax in the exp2 domain with a lazy rescale of O
//                (only when the running max grows by more than 2^8), write P
//                as bf16 over S in TMEM; final normalisation and store, staged
//                per warp through the (then idle) Q region of shared memory
//                so that every store instruction writes whole rows.
//   warps 12-15  the leftover rows on mma.sync (keys on M, rows on N), reading
//                the same K/V stages through ldmatrix.
//
// TMEM columns: S/P of tile t at [64t, +64); Q of tile t at [128+64t, +64) (the A
// operand of QK^T, so Q is not re-read from shared memory for every key tile);
// O of tile t at [256+128t, +128). The tensor core works on one tile while the
// other tile's softmax runs.
// Every wait is bounded; a timeout sets DDT_DEV_TIMEOUT, drains the copies
// and MMAs already issued, frees TMEM and returns.
//
// The kernel is a programmatic dependent of the build (which signals its
// dependents as it starts): the work-item lookup reads only ctx_len, the
// producer streams Q and the context at once, and the tree (n_nodes, the
// masks) is read after griddepcontrol.wait, by the softmax warps once their Q
// is in TMEM, by the leftover-row warps, and by the producer before its first
// tree tile.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn.cuh"
#include "tc_ptx.cuh"

namespace ddt {

namespace {

using namespace tc;

constexpr int kKeys = 64;                 // keys per pipeline tile
constexpr int kStages = 4;
constexpr int kThreads = 512;
constexpr int kD = 128;                   // head dim of this path
constexpr int kMaxSide = 8;               // leftover rows handled on mma.sync
constexpr int kLptMaxB = 64;              // batches up to this size run their longest chunks first

constexpr uint32_t kQTileBytes = 128 * kD * 2;          // 32 KB (two 16 KB halves)
constexpr uint32_t kHalfBytes = kKeys * 128;            // 8 KB: 64 rows x 128 B
constexpr uint32_t kStageBytes = 4 * kHalfBytes;        // K0 K1 V0 V1
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffStages = 2 * kQTileBytes;                       // 64 KB
constexpr uint32_t kOffSideO = kOffStages + kStages * kStageBytes;     // 192 KB
constexpr uint32_t kSideOBytes = 4 * kMaxSide * kD * 4;                // 16 KB: one block per leftover-row warp
constexpr uint32_t kSmemBytes = kOffSideO + kSideOBytes + 1024;        // + alignment slack

constexpr uint32_t kColS = 0;     // + 64 * t: S of tile t, P written over its first 32 columns
constexpr uint32_t kColQ = 128;   // + 64 * t: Q of tile t (bf16 pairs), the A operand of QK^T
constexpr uint32_t kColO = 256;   // + 128 * t

struct TcMaps {
    CUtensorMap q;    // {Dh, G, Hkv, B*N}
    CUtensorMap kc;   // {Dh, Hkv, page_size, num_pages}
    CUtensorMap vc;
    CUtensorMap kt;   // {Dh, Hkv, B*N}
    CUtensorMap vt;
};

struct TcShared {
    uint64_t q_full;
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t q_tmem;          // Q rows copied from shared memory into TMEM
    uint64_t s_full[2];       // [tile]: S of the current key tile is in TMEM
    uint64_t p_full[2];       // [tile]: P written over it
    uint64_t o_final[2];      // row tile t's last PV done: its epilogue may read O
    uint64_t vfix[3];
    uint64_t never;           // completed by nothing: the testing entry point's stalled wait
    uint32_t tmem_base;
    int abort;
    float side_max[2][4][kMaxSide];
    float side_l[4][kMaxSide];
    float side_m[kMaxSide];
    int map_cnt[kLptMaxB];    // work-item counts in rank order (the CTA's item lookup)
    int map_off[kLptMaxB];    // their exclusive prefix sums
    int item[7];              // this CTA's (request, KV head, chunk, found, ctx_len, unused, row group)
};

struct Geometry {
    int b, kvh, chunk, L, nn, nchunks, t_begin, n_ctx, n_tree, n_tiles;
    int R, G, n_main, n_side;
    int grp, r0;              // row group and its first row (rows r0 .. r0 + R - 1 of the request's G * N)
    int rpt;                  // rows of a tile: the whole nodes that fit in 128 lanes
    bool bad;
};

// key range of pipeline tile j: first key, number of valid keys, and the
// index of its V fix-up barrier (-1: none)
struct TileInfo {
    bool ctx;
    int key0, valid, fix;
};

DDT_DEVINL TileInfo tile_info(const Geometry& g, int j) {
    TileInfo ti;
    if (j < g.n_ctx) {
        ti.ctx = true;
        ti.key0 = (g.t_begin + j) * kKeys;
        ti.valid = min(kKeys, g.L - ti.key0);
        ti.fix = ti.valid < kKeys ? 0 : -1;
    } else {
        const int tt = j - g.n_ctx;
        ti.ctx = false;
        ti.key0 = tt * kKeys;
        ti.valid = max(0, min(kKeys, g.nn - ti.key0));
        ti.fix = 1 + tt;
    }
    return ti;
}

DDT_DEVINL uint32_t bar_addr(const uint64_t& b) { return smem_u32(&b); }

// Work item of CTA i when the batch runs longest chunks first (warp 0, all
// lanes). Requests are ranked by their chunk length (tiles, descending; ties
// by index); each contributes Hkv * nch items (head-major, then chunk), in
// rank order. Writes (b, kvh, chunk, found) to `item`: found = 0 past the last
// item. The CTAs are dispatched in index order, so the longest chunks start
// first and the short ones fill the tail (longest processing time first).
DDT_DEVINL void lpt_item(const AttnParams& p, int i, int* cnt, int* off, int* item) {
    const int lane = threadIdx.x & 31;
    int key[2], nch[2], rnk[2], Lq[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int b = lane + 32 * q;
        Lq[q] = b < p.B ? p.ctx_len[b] : 0;
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int b = lane + 32 * q;
        key[q] = -1;
        nch[q] = 1;
        if (b < p.B) {
            const int L = Lq[q];
            const int nt = (L < 0 || L > p.max_pages * p.page_size) ? 0 : (L + kKeys - 1) / kKeys;
            nch[q] = nt > 0 ? (nt + p.tiles_per_chunk - 1) / p.tiles_per_chunk : 1;
            key[q] = nt > 0 ? (nt + nch[q] - 1) / nch[q] : 0;
        }
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int b = lane + 32 * q;
        int r = 0;
        for (int s2 = 0; s2 < p.B; ++s2) {
            const int ks = __shfl_sync(0xffffffffu, s2 < 32 ? key[0] : key[1], s2 & 31);
            r += (ks > key[q]) || (ks == key[q] && s2 < b);
        }
        rnk[q] = r;
        if (b < p.B) cnt[r] = nch[q] * p.Hkv * p.tc_groups;
    }
    __syncwarp();
    // exclusive prefix over the ranked counts (two entries per lane)
    const int c0 = 2 * lane < p.B ? cnt[2 * lane] : 0;
    const int c1 = 2 * lane + 1 < p.B ? cnt[2 * lane + 1] : 0;
    int incl = c0 + c1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const int excl = incl - c0 - c1;
    off[2 * lane] = excl;
    off[2 * lane + 1] = excl + c0;
    __syncwarp();
    int hit = -1, local = 0;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int b = lane + 32 * q;
        if (b < p.B) {
            const int o = off[rnk[q]];
            if (i >= o && i < o + nch[q] * p.Hkv * p.tc_groups) { hit = q; local = i - o; }
        }
    }
    const unsigned m = __ballot_sync(0xffffffffu, hit >= 0);
    if (m) {
        const int src = __ffs(m) - 1;
        if (lane == src) {
            const int b = lane + 32 * hit;
            item[0] = b;
            item[1] = local / (nch[hit] * p.tc_groups);
            item[2] = local % nch[hit];
            item[3] = 1;
            item[4] = Lq[hit];
            item[6] = (local / nch[hit]) % p.tc_groups;
        }
    } else if (lane == 0) {
        item[3] = 0;
    }
}

// kWholeTile: G divides 128, so a tile's rows are all 128 lanes (a compile-time
// constant in the row arithmetic); otherwise the whole nodes that fit.
template <bool kWholeTile>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const AttnParams p, const __grid_constant__ TcMaps maps) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ TcShared sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---------------- set-up: barriers, descriptors, TMEM ----------------
    // None of it depends on the work item (every CTA has the same rows), so it
    // runs beside the item lookup, under one barrier.
    // Barrier counts are the same in every CTA: the Q copy is acknowledged by the
    // softmax warps of n_main_all tiles (those of a tile a short row group does
    // not use arrive without work), and when the last row group has leftover
    // rows the leftover-row warps of every CTA take part in the K/V ring.
    const int n_main_all = p.R > (kWholeTile ? 128 : (128 / p.G) * p.G) ? 2 : 1;
    // rows of a 128-lane tile: whole nodes only (a tile's Q box holds 128 / G nodes)
    const int rpt = kWholeTile ? 128 : (128 / p.G) * p.G;
    const bool side_all = p.R - 2 * rpt * (p.tc_groups - 1) > 2 * rpt;
    {
        const int n_main = n_main_all;
        const bool side = side_all;
        if (tid == 64) {   // warp 2: idle during the lookup
            mbar_init(bar_addr(sh.q_full), 1);
            for (int s = 0; s < kStages; ++s) {
                mbar_init(bar_addr(sh.kv_full[s]), 1);
                mbar_init(bar_addr(sh.kv_empty[s]), side ? 5 : 1);   // MMA commit + 4 side warps
            }
            mbar_init(bar_addr(sh.q_tmem), 4 * n_main);   // one arrival per softmax warp
            for (int t = 0; t < 2; ++t) {
                mbar_init(bar_addr(sh.s_full[t]), 1);
                mbar_init(bar_addr(sh.p_full[t]), 4);
            }
            mbar_init(bar_addr(sh.o_final[0]), 1);
            mbar_init(bar_addr(sh.o_final[1]), 1);
            for (int k = 0; k < 3; ++k) mbar_init(bar_addr(sh.vfix[k]), 1);
            mbar_init(bar_addr(sh.never), 1);
            sh.abort = 0;
            fence_mbar_init();
            prefetch_tmap(&maps.q);
            prefetch_tmap(&maps.kc);
            prefetch_tmap(&maps.vc);
            prefetch_tmap(&maps.kt);
            prefetch_tmap(&maps.vt);
        }
        if (warp == 1) tmem_alloc(smem_u32(&sh.tmem_base), 512);
    }
    const bool lpt = p.B <= kLptMaxB && p.max_chunks > 1;
    if (lpt && warp == 0) lpt_item(p, static_cast<int>(blockIdx.x), sh.map_cnt, sh.map_off, sh.item);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sh.tmem_base;
    // a CTA without work frees its TMEM and leaves (nothing is in flight yet)
    auto leave = [&]() {
        if (warp == 1) tmem_dealloc(tbase, 512);
    };

    Geometry g;
    if (lpt) {   // one-dimensional grid, longest chunks first
        if (!sh.item[3]) { leave(); return; }
        g.b = sh.item[0];
        g.kvh = sh.item[1];
        g.chunk = sh.item[2];
        g.L = sh.item[4];
        g.grp = sh.item[6];
    } else {   // one-dimensional grid in (request, head, row group, chunk) order
        const int i = static_cast<int>(blockIdx.x);
        g.chunk = i % p.max_chunks;
        g.grp = (i / p.max_chunks) % p.tc_groups;
        g.kvh = (i / (p.max_chunks * p.tc_groups)) % p.Hkv;
        g.b = i / (p.max_chunks * p.tc_groups * p.Hkv);
        g.L = p.ctx_len[g.b];
    }
    g.G = p.G;
    g.rpt = rpt;
    g.r0 = 2 * rpt * g.grp;
    g.R = g.grp + 1 < p.tc_groups ? 2 * rpt : p.R - g.r0;
    g.bad = false;
    if (g.L < 0 || g.L > p.max_pages * p.page_size) { g.bad = true; g.L = 0; }
    const int nt_ctx = (g.L + kKeys - 1) / kKeys;
    g.nchunks = nt_ctx > 0 ? (nt_ctx + p.tiles_per_chunk - 1) / p.tiles_per_chunk : 1;
    if (g.chunk >= g.nchunks) { leave(); return; }
    // The tree (n_nodes, the masks) comes from the build, which may still be
    // running (this kernel is its programmatic dependent): the roles that need
    // it wait for the build's grid first (see read_tree). Everything before
    // uses only the call's inputs.
    g.nn = 0;
    auto read_tree = [&]() {
        asm volatile("griddepcontrol.wait;\n" ::: "memory");
        const int nn = p.n_nodes[g.b];
        if (nn < 0 || nn > p.N) {   // a malformed tree: no real rows (outputs zero, lse -inf)
            if (lane == 0) report(p.dev_status, DDT_DEV_BAD_CTX);
            g.nn = 0;
        } else {
            g.nn = nn;
        }
    };
    // the request's tiles in nchunks chunks of equal length (within one tile)
    g.t_begin = static_cast<int>(static_cast<long long>(nt_ctx) * g.chunk / g.nchunks);
    g.n_ctx = static_cast<int>(static_cast<long long>(nt_ctx) * (g.chunk + 1) / g.nchunks) - g.t_begin;
    g.n_tree = (g.chunk == g.nchunks - 1) ? (p.N + kKeys - 1) / kKeys : 0;
    g.n_tiles = g.n_ctx + g.n_tree;
    g.n_main = g.R > rpt ? 2 : 1;
    g.n_side = max(0, g.R - 2 * rpt);

    if (g.bad) {   // the request's rows are zeros
        if (g.chunk == 0) {
            if (tid == 0) report(p.dev_status, DDT_DEV_BAD_CTX);
            for (int x = tid; x < g.R * (kD / 8); x += kThreads) {
                const int r = g.r0 + x / (kD / 8), c = x % (kD / 8);
                const int i = r / g.G, h = g.kvh * g.G + r % g.G;
                *reinterpret_cast<uint4*>(p.out + ((static_cast<size_t>(g.b) * p.N + i) * p.Hq + h) * kD + c * 8) =
                    make_uint4(0, 0, 0, 0);
                if (p.lse && c == 0) p.lse[(static_cast<size_t>(g.b) * p.N + i) * p.Hq + h] = -INFINITY;
            }
        }
        leave();
        return;
    }

    const size_t slot = (static_cast<size_t>(g.b) * p.Hkv + g.kvh) * p.max_chunks + g.chunk;
    const bool split = g.nchunks > 1;

    volatile int* abort = &sh.abort;

    const uint32_t sQ = smem_u32(smem + kOffQ);
    const uint32_t sStage = smem_u32(smem + kOffStages);

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        const int box_keys = p.page_size < kKeys ? p.page_size : kKeys;
        int last_issued[kStages];
#pragma unroll
        for (int s = 0; s < kStages; ++s) last_issued[s] = -1;
        int pf_base = -1, pf_page = 0;
        if (lane == 0) {
            mbar_arrive_expect_tx(bar_addr(sh.q_full), g.n_main * (kQTileBytes / 128) * g.rpt);
            const int nodes_per_tile = 128 / g.G;
            for (int t = 0; t < g.n_main; ++t)
                for (int h = 0; h < 2; ++h)
                    tma_load_4d(sQ + t * kQTileBytes + h * (kQTileBytes / 2), &maps.q,
                                bar_addr(sh.q_full), 64 * h, 0, g.kvh,
                                g.b * p.N + g.r0 / g.G + t * nodes_per_tile);
        }
        for (int j = 0; j < g.n_tiles; ++j) {
            const int s = j % kStages;
            if (j >= kStages &&
                !__all_sync(0xffffffffu, mbar_wait_bounded(bar_addr(sh.kv_empty[s]), ((j / kStages) - 1) & 1, abort)))
                break;
            if (j == g.n_ctx) read_tree();   // the tree tiles' valid rows need n_nodes
            const TileInfo ti = tile_info(g, j);
            const uint32_t kdst = sStage + s * kStageBytes;
            const uint32_t vdst = kdst + 2 * kHalfBytes;
            const uint32_t full = bar_addr(sh.kv_full[s]);
            // page ids of the next 32 tiles are fetched by the 32 lanes at once
            // (one page per tile when pages hold at least 64 keys)
            int tile_page = p.num_pages;
            if (ti.ctx && box_keys == kKeys) {
                if (pf_base < 0 || j >= pf_base + 32) {
                    pf_base = j;
                    const int jj = j + lane;
                    const int kk = (g.t_begin + jj) * kKeys;
                    pf_page = p.num_pages;
                    if (jj < g.n_ctx && kk < g.L)
                        pf_page = p.page_table[static_cast<size_t>(g.b) * p.max_pages + kk / p.page_size];
                }
                tile_page = __shfl_sync(0xffffffffu, pf_page, j - pf_base);
            }
            mbar_arrive_expect_tx_elect(full, kStageBytes);
            if (ti.ctx) {
                for (int sub = 0; sub < kKeys / box_keys; ++sub) {
                    const int kk = ti.key0 + sub * box_keys;
                    int page = p.num_pages;   // past the pool: the box reads zeros
                    if (kk < g.L) {
                        page = box_keys == kKeys
                                   ? tile_page
                                   : p.page_table[static_cast<size_t>(g.b) * p.max_pages + kk / p.page_size];
                        if (page < 0 || page >= p.num_pages) {
                            if (lane == 0) report(p.dev_status, DDT_DEV_BAD_PAGE);
                            page = p.num_pages;
                        }
                    }
                    const int slot_in_page = kk % p.page_size;
                    for (int h = 0; h < 2; ++h) {
                        tma_load_4d_elect(kdst + h * kHalfBytes + sub * box_keys * 128, &maps.kc, full,
                                          64 * h, g.kvh, slot_in_page, page);
                        tma_load_4d_elect(vdst + h * kHalfBytes + sub * box_keys * 128, &maps.vc, full,
                                          64 * h, g.kvh, slot_in_page, page);
                    }
                }
            } else {
                for (int h = 0; h < 2; ++h) {
                    tma_load_3d_elect(kdst + h * kHalfBytes, &maps.kt, full, 64 * h, g.kvh,
                                      g.b * p.N + ti.key0);
                    tma_load_3d_elect(vdst + h * kHalfBytes, &maps.vt, full, 64 * h, g.kvh,
                                      g.b * p.N + ti.key0);
                }
            }
            last_issued[s] = j;
            __syncwarp();
            if (ti.fix >= 0) {
                // zero V rows [valid, 64) once the tile has landed
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(full, (j / kStages) & 1, abort))) break;
                const int rows = kKeys - ti.valid;
                for (int x = lane; x < rows * 16; x += 32) {
                    const int row = ti.valid + x / 16, part = x % 16;   // 16 x 16 B per row (two halves)
                    const int h = part / 8, c = part % 8;
                    unsigned char* dst = smem + kOffStages + s * kStageBytes + 2 * kHalfBytes +
                                         h * kHalfBytes + row * 128 + c * 16;
                    *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_addr(sh.vfix[ti.fix]));
            }
        }
        // drain: every copy issued must land before the CTA can exit
        if (lane == 0) {
            for (int s = 0; s < kStages; ++s)
                if (last_issued[s] >= 0) mbar_drain(bar_addr(sh.kv_full[s]), (last_issued[s] / kStages) & 1);
            mbar_drain(bar_addr(sh.q_full), 0);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        // The whole warp runs this loop so every operand is warp-uniform; one
        // elected lane issues each tcgen05 instruction.
        {
            const uint32_t id_s = idesc_bf16_f32(128, kKeys, 0, 0);
            const uint32_t id_o = idesc_bf16_f32(128, kD, 0, 1);
            // Descriptors: one base per operand; an MMA only adds its byte offset >> 4
            // to the start-address field (addresses stay below 256 KB, so no carry).
            const uint64_t dq = smem_desc(sQ, 16, 1024);
            const uint64_t dk = smem_desc(sStage, 16, 1024);
            const uint64_t dv = smem_desc(sStage + 2 * kHalfBytes, kHalfBytes, 1024);
            // S_t = Q_t K_j^T (Q from TMEM)
            auto qk = [&](int t, int j) {
                const uint32_t koff = ((j % kStages) * kStageBytes) >> 4;
                const uint32_t d = tbase + kColS + 64 * t;
                const uint32_t qa = tbase + kColQ + 64 * t;
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks) {
                    const uint32_t ko = koff + (((ks / 4) * kHalfBytes + (ks % 4) * 32) >> 4);
                    mma_ts_elect(d, qa + 8 * ks, dk + ko, id_s, ks > 0);
                }
                mma_commit_elect(bar_addr(sh.s_full[t]));
            };
            // O_t (+)= P_t V_j
            auto pv = [&](int t, int j) {
                const uint32_t voff = ((j % kStages) * kStageBytes) >> 4;
                const uint32_t a = tbase + kColS + 64 * t;
                const uint32_t o = tbase + kColO + 128 * t;
#pragma unroll
                for (int ks = 0; ks < kKeys / 16; ++ks)
                    mma_ts_elect(o, a + 8 * ks, dv + voff + ((ks * 2048) >> 4), id_o, (j > 0) || ks > 0);
            };
            auto wait_all = [&](uint32_t bar, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort));
            };
            // testing entry point only: a wait that nothing completes runs out after
            // stall_ns and aborts the CTA through the normal path
            const bool stalled = p.stall_ns != 0 &&
                                 !__all_sync(0xffffffffu, mbar_wait_bounded(bar_addr(sh.never), 0, abort, p.stall_ns));
            bool fin[2] = {false, false};   // o_final[t] committed
            bool ok = !stalled && wait_all(bar_addr(sh.q_tmem), 0) &&
                      (g.n_tiles == 0 || wait_all(bar_addr(sh.kv_full[0]), 0));
            if (ok && g.n_tiles > 0) {
                tc_fence_after();
                qk(0, 0);
                if (g.n_main == 2) qk(1, 0);
            }
            for (int j = 0; ok && j < g.n_tiles; ++j) {
                const TileInfo ti = tile_info(g, j);
                const bool more = j + 1 < g.n_tiles;
                if (ti.fix >= 0 && !wait_all(bar_addr(sh.vfix[ti.fix]), 0)) break;
                if (!wait_all(bar_addr(sh.p_full[0]), j & 1)) break;
                tc_fence_after();
                pv(0, j);
                if (!more) { mma_commit_elect(bar_addr(sh.o_final[0])); fin[0] = true; }
                if (more) {
                    if (!wait_all(bar_addr(sh.kv_full[(j + 1) % kStages]), ((j + 1) / kStages) & 1)) break;
                    tc_fence_after();
                    qk(0, j + 1);   // after PV_0(j) in issue order, so P_0 is consumed first
                }
                if (g.n_main == 2) {
                    if (!wait_all(bar_addr(sh.p_full[1]), j & 1)) break;
                    tc_fence_after();
                    pv(1, j);
                    if (!more) { mma_commit_elect(bar_addr(sh.o_final[1])); fin[1] = true; }
                }
                mma_commit_elect(bar_addr(sh.kv_empty[j % kStages]));   // K_j and V_j consumed
                if (g.n_main == 2 && more) qk(1, j + 1);
            }
            // a tile whose last PV was not reached (abort, or no tiles) is released here
            for (int t = 0; t < g.n_main; ++t)
                if (!fin[t]) mma_commit_elect(bar_addr(sh.o_final[t]));
            for (int t = 0; t < g.n_main; ++t)
                mbar_drain(bar_addr(sh.o_final[t]), 0);   // every MMA done before TMEM is freed
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 12) {
        // ---------------- softmax: one thread per row of tile t ----------------
        const int t = (warp - 4) / 4;
        const int qw = warp & 3;
        const int row_local = 32 * qw + lane;
        const int r = g.rpt * t + row_local;
        const bool active = t < g.n_main;
        const bool valid_row = active && row_local < g.rpt && r < g.R;
        const int node = valid_row ? (g.r0 + r) / g.G : 0;
        const uint32_t lane_off = static_cast<uint32_t>(32 * qw) << 16;
        const uint32_t tS = tbase + lane_off + kColS + 64 * t;
        const uint32_t tO = tbase + lane_off + kColO + 128 * t;
        // copy this thread's Q row (TMA-written, 128-byte swizzled) into TMEM
        if (active) {
            const bool q_ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar_addr(sh.q_full), 0, abort));
            const unsigned char* qrow = smem + kOffQ + t * kQTileBytes;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    // rows past the tile's whole nodes hold no Q: zeros
                    const uint4 v = (q_ok && row_local < g.rpt) ? *reinterpret_cast<const uint4*>(
                                               qrow + hh * (kQTileBytes / 2) + sw128_offset(row_local, c))
                                         : make_uint4(0, 0, 0, 0);
                    w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
                }
                tmem_st32(tbase + lane_off + kColQ + 64 * t + 32 * hh, w);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_addr(sh.q_tmem));   // one arrival per warp
        } else if (t < n_main_all && lane == 0) {
            mbar_arrive(bar_addr(sh.q_tmem));   // a tile this row group does not use
        }
        read_tree();   // after the Q copy: the tree is first needed by the masks
        const bool real = valid_row && node < g.nn;
        uint32_t visw[4] = {0u, 0u, 0u, 0u};
        if (real)
            for (int w = 0; w < p.W; ++w) visw[w] = p.vis[(static_cast<size_t>(g.b) * p.N + node) * p.W + w];
        const float sc = p.scale_log2;            // > 0 on this path
        float m_ref = -INFINITY;                  // reference max, scaled log2 units
        float l_sum = 0.0f;
        bool ok = active;
        for (int j = 0; ok && j < g.n_tiles; ++j) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar_addr(sh.s_full[t]), j & 1, abort))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t raw[2][32];
            tmem_ld32(tS, raw[0]);
            tmem_ld32(tS + 32, raw[1]);
            tmem_wait_ld();
            const TileInfo ti = tile_info(g, j);
            if (!(ti.ctx && ti.valid == kKeys)) {
                // ragged context tail or tree tile: masked scores become -inf
                uint32_t vlo = 0xFFFFFFFFu, vhi = 0xFFFFFFFFu;
                if (!ti.ctx) {
                    vlo = pick4(visw, ti.key0 >> 5);
                    vhi = pick4(visw, (ti.key0 >> 5) + 1);
                }
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const uint32_t bit = c < 32 ? (vlo >> c) & 1u : (vhi >> (c - 32)) & 1u;
                    if (!(c < ti.valid && bit)) raw[c >> 5][c & 31] = 0xFF800000u;   // -inf
                }
            }
            // row max of the raw scores (scale > 0 keeps the order): four chains of
            // three-input maxima over 16 columns each, then their maximum
            float mx;
            {
                float mc[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c0 = 16 * q;
                    float a = fmaxf(__uint_as_float(raw[c0 >> 5][c0 & 31]), __uint_as_float(raw[(c0 + 1) >> 5][(c0 + 1) & 31]));
#pragma unroll
                    for (int k = 2; k < 16; k += 2)
                        a = fmax3(a, __uint_as_float(raw[(c0 + k) >> 5][(c0 + k) & 31]),
                                  __uint_as_float(raw[(c0 + k + 1) >> 5][(c0 + k + 1) & 31]));
                    mc[q] = a;
                }
                mx = fmaxf(fmax3(mc[0], mc[1], mc[2]), mc[3]);
            }
            const float mxs = mx * sc;
            // Raise the reference max of a row when it grows by more than 2^8, and
            // rescale O and l. The decision is taken for the whole warp (the
            // TMEM loads and stores are warp-collective): rows that need no
            // rescale keep their reference and scale by exactly 1.
            const bool raise = mxs > m_ref + 8.0f;
            if (__any_sync(0xffffffffu, raise)) {
                const float m_new = raise ? mxs : m_ref;
                if (j > 0) {
                    // QK_t(j) was issued after PV_t(j-1), so S ready means O is complete
                    const float alpha = (raise && m_ref != -INFINITY) ? fast_exp2(m_ref - m_new) : 1.0f;
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + 32 * c, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tO + 32 * c, o);
                    }
                    l_sum *= alpha;
                }
                m_ref = m_new;
            }
            const float neg_m = (m_ref == -INFINITY) ? 0.0f : -m_ref;
            // P = 2^(s*scale - m) as bf16 pairs over the first 32 columns of this S buffer;
            // the scaling and the running sums take paired fp32 instructions
            const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(neg_m, neg_m);
            float2 ls[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float2 x = ffma2(make_float2(__uint_as_float(raw[(2 * c) >> 5][(2 * c) & 31]),
                                                   __uint_as_float(raw[(2 * c + 1) >> 5][(2 * c + 1) & 31])),
                                       sc2, nm2);
                const float2 pe = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                ls[c & 1] = fadd2(ls[c & 1], pe);
                __nv_bfloat162 v = __floats2bfloat162_rn(pe.x, pe.y);
                raw[0][c] = *reinterpret_cast<uint32_t*>(&v);
            }
            l_sum += (ls[0].x + ls[0].y) + (ls[1].x + ls[1].y);
            tmem_st32(tS, raw[0]);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_addr(sh.p_full[t]));   // one arrival per warp
        }
        if (active) {
            const bool done = __all_sync(0xffffffffu, mbar_wait_bounded(bar_addr(sh.o_final[t]), 0, abort));
            tc_fence_after();
            const int i = node, h = g.kvh * g.G + (valid_row ? (g.r0 + r) % g.G : 0);
            const bool good = done && ok;
            // Rows leave through a per-warp staging block in the (now idle) Q region of
            // shared memory, so that each store instruction writes whole rows.
            uint32_t* stage = reinterpret_cast<uint32_t*>(smem + kOffQ) + (warp - 4) * (32 * 36);
            if (!split) {
                const float inv = (real && good && l_sum > 0.0f) ? 1.0f / l_sum : 0.0f;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * c, o);
                    tmem_wait_ld();
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        __nv_bfloat162 v = __floats2bfloat162_rn(inv != 0.0f ? __uint_as_float(o[2 * e]) * inv : 0.0f,
                                                                 inv != 0.0f ? __uint_as_float(o[2 * e + 1]) * inv : 0.0f);
                        w[e] = *reinterpret_cast<uint32_t*>(&v);
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e)   // row stride 20 words: conflict-free 16-byte stores
                        *reinterpret_cast<uint4*>(stage + lane * 20 + 4 * e) =
                            make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 4; ++k) {   // 8 rows x 64 bytes per instruction
                        const int rr = 8 * k + (lane >> 2), q4 = lane & 3;
                        const int rg = g.rpt * t + 32 * qw + rr;
                        if (32 * qw + rr < g.rpt && rg < g.R) {
                            const int ir = (g.r0 + rg) / g.G, hr = g.kvh * g.G + (g.r0 + rg) % g.G;
                            *reinterpret_cast<uint4*>(p.out + ((static_cast<size_t>(g.b) * p.N + ir) * p.Hq + hr) * kD +
                                                      32 * c + 8 * q4) =
                                *reinterpret_cast<const uint4*>(stage + rr * 20 + 4 * q4);
                        }
                    }
                    __syncwarp();
                }
                if (p.lse && valid_row)
                    p.lse[(static_cast<size_t>(g.b) * p.N + i) * p.Hq + h] =
                        (real && good && l_sum > 0.0f) ? (m_ref + log2f(l_sum)) * 0.69314718055994531f
                                                       : -INFINITY;
            } else {
                float* fst = reinterpret_cast<float*>(stage);
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; ++e)   // row stride 36 words: conflict-free 16-byte stores
                        *reinterpret_cast<float4*>(fst + lane * 36 + 4 * e) =
                            good ? make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                               __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]))
                                 : make_float4(0.0f, 0.0f, 0.0f, 0.0f);   // aborted: defined zeros
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 8; ++k) {   // 4 rows x 128 bytes per instruction
                        const int rr = 4 * k + (lane >> 3), q4 = lane & 7;
                        const int rg = g.rpt * t + 32 * qw + rr;
                        if (32 * qw + rr < g.rpt && rg < g.R)
                            *reinterpret_cast<float4*>(p.ws_o + (slot * p.R + g.r0 + rg) * kD + 32 * c + 4 * q4) =
                                *reinterpret_cast<const float4*>(fst + rr * 36 + 4 * q4);
                    }
                    __syncwarp();
                }
                if (valid_row)
                    p.ws_ml[slot * p.R + g.r0 + r] = good ? make_float2(m_ref, l_sum) : make_float2(-INFINITY, 0.0f);
            }
        }
    } else if (warp >= 12 && side_all && g.n_side == 0) {
        // a row group without leftover rows in a launch whose last group has
        // them: these warps still release every K/V stage the ring counts on
        read_tree();   // tile_info below uses n_nodes
        bool ok = true;
        for (int j = 0; ok && j < g.n_tiles; ++j) {
            const int s = j % kStages;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar_addr(sh.kv_full[s]), (j / kStages) & 1, abort));
            if (ok && lane == 0) mbar_arrive(bar_addr(sh.kv_empty[s]));
        }
    } else if (warp >= 12 && g.n_side > 0) {
        // ---------------- leftover rows on mma.sync ----------------
        read_tree();
        const int sw = warp - 12;                      // keys 16*sw .. 16*sw+15 of each tile
        const int nrow = lane >> 2;                    // B-fragment row (n index)
        const int crow0 = 2 * (lane & 3);              // C-fragment rows crow0, crow0+1
        // Q rows as B fragments (k = dh, n = row)
        uint32_t qb[kD / 16][2];
        {
            const int sr = nrow;
            const bool ok = sr < g.n_side;
            const int r = g.r0 + 2 * g.rpt + (ok ? sr : 0);
            const int i = r / g.G, h = g.kvh * g.G + r % g.G;
            const bf16_t* qrow = p.q + ((static_cast<size_t>(g.b) * p.N + i) * p.Hq + h) * kD;
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
                const int k0 = ks * 16 + 2 * (lane & 3);
                qb[ks][0] = ok ? *reinterpret_cast<const uint32_t*>(qrow + k0) : 0u;
                qb[ks][1] = ok ? *reinterpret_cast<const uint32_t*>(qrow + k0 + 8) : 0u;
            }
        }
        int node_r[2];
        uint32_t visr[2][4];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int sr = crow0 + q;
            node_r[q] = sr < g.n_side ? (g.r0 + 2 * g.rpt + sr) / g.G : -1;
#pragma unroll
            for (int w = 0; w < 4; ++w)
                visr[q][w] = (node_r[q] >= 0 && node_r[q] < g.nn && w < p.W)
                                 ? p.vis[(static_cast<size_t>(g.b) * p.N + node_r[q]) * p.W + w] : 0u;
        }
        float m_run[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.0f, 0.0f};
        float oacc[kD / 16][4];
#pragma unroll
        for (int mb = 0; mb < kD / 16; ++mb) oacc[mb][0] = oacc[mb][1] = oacc[mb][2] = oacc[mb][3] = 0.0f;
        bool ok = true;
        // Each of the four warps runs its own online softmax over its 16 keys of
        // every tile; the four partial results are merged once at the end.
        for (int j = 0; j < g.n_tiles; ++j) {
            const int s = j % kStages;
            const TileInfo ti = tile_info(g, j);
            bool got = ok && mbar_wait_bounded(bar_addr(sh.kv_full[s]), (j / kStages) & 1, abort);
            if (got && ti.fix >= 0) got = mbar_wait_bounded(bar_addr(sh.vfix[ti.fix]), 0, abort);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            const unsigned char* kst = smem + kOffStages + s * kStageBytes;
            const unsigned char* vst = kst + 2 * kHalfBytes;
            // S^T (16 keys x 8 rows) = K Q^T, two accumulators to halve the dependency chain
            float c[4] = {0.0f, 0.0f, 0.0f, 0.0f}, c2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
                const int key = 16 * sw + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int chunk = ks * 2 + (lane >> 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(smem_u32(kst + (chunk >> 3) * kHalfBytes + sw128_offset(key, chunk & 7)), a0, a1, a2, a3);
                if (ks & 1) mma16816(c2, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
                else mma16816(c, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
            }
            // scale, mask; c0/c1: key kA rows crow0/crow0+1; c2/c3: key kA+8
            const int kA = 16 * sw + nrow;
            if (ti.ctx && ti.valid == kKeys) {   // a full context tile: only rows past R are masked
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    c[e] += c2[e];
                    c[e] = node_r[e & 1] >= 0 ? c[e] * p.scale_log2 : -INFINITY;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    c[e] += c2[e];
                    const int kl = kA + ((e >> 1) << 3);
                    const int q = e & 1;
                    bool vis_ok = node_r[q] >= 0 && kl < ti.valid;
                    if (!ti.ctx && vis_ok) {
                        const int key = ti.key0 + kl;
                        vis_ok = (pick4(visr[q], key >> 5) >> (key & 31)) & 1u;
                    }
                    c[e] = vis_ok ? c[e] * p.scale_log2 : -INFINITY;
                }
            }
            // Lazy rescale, as for the main rows: the reference max of a row moves
            // only when a score exceeds it by more than 2^8; most tiles then need
            // neither the row max nor a rescale of the accumulators.
            const bool up = fmaxf(c[0], c[2]) > m_run[0] + 8.0f || fmaxf(c[1], c[3]) > m_run[1] + 8.0f;
            float alpha[2] = {1.0f, 1.0f};
            if (__any_sync(0xffffffffu, up)) {
                float mx[2] = {fmaxf(c[0], c[2]), fmaxf(c[1], c[3])};
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    mx[q] = fmaxf(mx[q], __shfl_xor_sync(0xffffffffu, mx[q], 4));
                    mx[q] = fmaxf(mx[q], __shfl_xor_sync(0xffffffffu, mx[q], 8));
                    mx[q] = fmaxf(mx[q], __shfl_xor_sync(0xffffffffu, mx[q], 16));
                    if (mx[q] > m_run[q] + 8.0f) {
                        alpha[q] = m_run[q] == -INFINITY ? 1.0f : fast_exp2(m_run[q] - mx[q]);
                        m_run[q] = mx[q];
                    }
                }
#pragma unroll
                for (int mb = 0; mb < kD / 16; ++mb) {
                    oacc[mb][0] *= alpha[0]; oacc[mb][2] *= alpha[0];
                    oacc[mb][1] *= alpha[1]; oacc[mb][3] *= alpha[1];
                }
            }
            const float m_use[2] = {m_run[0] == -INFINITY ? 0.0f : m_run[0], m_run[1] == -INFINITY ? 0.0f : m_run[1]};
            float pe[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) pe[e] = fast_exp2(c[e] - m_use[e & 1]);
            l_part[0] = l_part[0] * alpha[0] + pe[0] + pe[2];
            l_part[1] = l_part[1] * alpha[1] + pe[1] + pe[3];
            __nv_bfloat162 p01 = __floats2bfloat162_rn(pe[0], pe[1]);
            __nv_bfloat162 p23 = __floats2bfloat162_rn(pe[2], pe[3]);
            const uint32_t b0 = movmatrix_t(*reinterpret_cast<uint32_t*>(&p01));
            const uint32_t b1 = movmatrix_t(*reinterpret_cast<uint32_t*>(&p23));
#pragma unroll
            for (int mb = 0; mb < kD / 16; ++mb) {
                const int key = 16 * sw + (lane & 7) + (lane >> 4) * 8;
                const int chunk = mb * 2 + ((lane >> 3) & 1);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(smem_u32(vst + (chunk >> 3) * kHalfBytes + sw128_offset(key, chunk & 7)), a0, a1, a2, a3);
                mma16816(oacc[mb], a0, a1, a2, a3, b0, b1);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_addr(sh.kv_empty[s]));   // this warp is done with the stage
        }
        // merge the four warps: common max per row, then rescaled sums
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            l_part[q] += __shfl_xor_sync(0xffffffffu, l_part[q], 4);
            l_part[q] += __shfl_xor_sync(0xffffffffu, l_part[q], 8);
            l_part[q] += __shfl_xor_sync(0xffffffffu, l_part[q], 16);
        }
        // [4 warps][kMaxSide rows][kD]: each warp writes every entry of its own block
        float* side_o = reinterpret_cast<float*>(smem + kOffSideO);
        if (lane < 4) {
            sh.side_max[0][sw][crow0] = m_run[0];
            sh.side_max[0][sw][crow0 + 1] = m_run[1];
        }
        named_bar_sync(1, 128);
        float wscale[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float M = sh.side_max[0][0][crow0 + q];
#pragma unroll
            for (int w2 = 1; w2 < 4; ++w2) M = fmaxf(M, sh.side_max[0][w2][crow0 + q]);
            wscale[q] = (M == -INFINITY) ? 0.0f : fast_exp2(m_run[q] - M);
            if (sw == 0 && lane < 4) sh.side_m[crow0 + q] = M;
        }
        if (lane < 4) {
            sh.side_l[sw][crow0] = l_part[0] * wscale[0];
            sh.side_l[sw][crow0 + 1] = l_part[1] * wscale[1];
        }
        {
            float* mine = side_o + sw * (kMaxSide * kD);
#pragma unroll
            for (int mb = 0; mb < kD / 16; ++mb) {
                const int d0 = 16 * mb + nrow;
                mine[crow0 * kD + d0] = oacc[mb][0] * wscale[0];
                mine[(crow0 + 1) * kD + d0] = oacc[mb][1] * wscale[1];
                mine[crow0 * kD + d0 + 8] = oacc[mb][2] * wscale[0];
                mine[(crow0 + 1) * kD + d0 + 8] = oacc[mb][3] * wscale[1];
            }
        }
        named_bar_sync(1, 128);
        // write: thread -> (row tid/16, 8 features), the four warps' blocks summed in
        // a fixed order
        const int st = tid - 384;
        const int sr = st >> 4, d0 = (st & 15) * 8;
        float o8[8];
        {
            const float* src = side_o + sr * kD + d0;
            const float4 a0 = *reinterpret_cast<const float4*>(src);
            const float4 a1 = *reinterpret_cast<const float4*>(src + 4);
            o8[0] = a0.x; o8[1] = a0.y; o8[2] = a0.z; o8[3] = a0.w;
            o8[4] = a1.x; o8[5] = a1.y; o8[6] = a1.z; o8[7] = a1.w;
#pragma unroll
            for (int w2 = 1; w2 < 4; ++w2) {
                const float4 b0 = *reinterpret_cast<const float4*>(src + w2 * (kMaxSide * kD));
                const float4 b1 = *reinterpret_cast<const float4*>(src + w2 * (kMaxSide * kD) + 4);
                o8[0] += b0.x; o8[1] += b0.y; o8[2] += b0.z; o8[3] += b0.w;
                o8[4] += b1.x; o8[5] += b1.y; o8[6] += b1.z; o8[7] += b1.w;
            }
        }
        if (sr < g.n_side) {
            const int r = g.r0 + 2 * g.rpt + sr;   // the request's row
            const int i = r / g.G, h = g.kvh * g.G + r % g.G;
            const float lt = sh.side_l[0][sr] + sh.side_l[1][sr] + sh.side_l[2][sr] + sh.side_l[3][sr];
            const float mrun = sh.side_m[sr];
            const bool real = i < g.nn && ok;
            if (!split) {
                const float inv = (real && lt > 0.0f) ? 1.0f / lt : 0.0f;
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    __nv_bfloat162 v = __floats2bfloat162_rn(inv != 0.0f ? o8[2 * e] * inv : 0.0f,
                                                             inv != 0.0f ? o8[2 * e + 1] * inv : 0.0f);
                    w[e] = *reinterpret_cast<uint32_t*>(&v);
                }
                *reinterpret_cast<uint4*>(p.out + ((static_cast<size_t>(g.b) * p.N + i) * p.Hq + h) * kD + d0) =
                    make_uint4(w[0], w[1], w[2], w[3]);
                if (p.lse && d0 == 0)
                    p.lse[(static_cast<size_t>(g.b) * p.N + i) * p.Hq + h] =
                        (real && lt > 0.0f) ? (mrun + log2f(lt)) * 0.69314718055994531f : -INFINITY;
            } else {
                float* dst = p.ws_o + (slot * p.R + r) * kD + d0;
                *reinterpret_cast<float4*>(dst) = ok ? make_float4(o8[0], o8[1], o8[2], o8[3]) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                *reinterpret_cast<float4*>(dst + 4) = ok ? make_float4(o8[4], o8[5], o8[6], o8[7]) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (d0 == 0) p.ws_ml[slot * p.R + r] = ok ? make_float2(mrun, lt) : make_float2(-INFINITY, 0.0f);
            }
        }
    }

    // ---------------- teardown ----------------
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, 512);
    if (tid == 0 && sh.abort) report(p.dev_status, DDT_DEV_TIMEOUT);
}

// ---------------------------------------------------------------------------
// host: tensor maps and launch
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

bool encode(PFN_cuTensorMapEncodeTiled_v12000 fn, CUtensorMap* m, const void* base, int rank,
            const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box) {
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                    strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

// True when tree_verify_attn's sizes fit the tensor-core kernel.
bool attn_tc_supported(const AttnParams& p) {
    if (p.Dh != kD || p.G > 128 || !(p.scale_log2 > 0.0f)) return false;
    const int rpt = (128 / p.G) * p.G;
    if (p.tc_groups < 1 || p.R > 2 * rpt * p.tc_groups + kMaxSide) return false;
    if (p.page_size < kKeys ? (kKeys % p.page_size) != 0 : (p.page_size % kKeys) != 0) return false;
    return true;
}

cudaError_t launch_attn_tc(const AttnParams& p, cudaStream_t stream) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = get_encode();
    if (!fn) return cudaErrorNotSupported;
    TcMaps maps;
    const cuuint64_t es = 2;
    {
        const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(p.G),
                                    static_cast<cuuint64_t>(p.Hkv), static_cast<cuuint64_t>(p.B) * p.N};
        const cuuint64_t str[3] = {kD * es, static_cast<cuuint64_t>(p.G) * kD * es,
                                   static_cast<cuuint64_t>(p.Hq) * kD * es};
        const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(p.G), 1, static_cast<cuuint32_t>(128 / p.G)};
        if (!encode(fn, &maps.q, p.q, 4, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(p.Hkv),
                                    static_cast<cuuint64_t>(p.page_size), static_cast<cuuint64_t>(p.num_pages)};
        const cuuint64_t str[3] = {kD * es, static_cast<cuuint64_t>(p.Hkv) * kD * es,
                                   static_cast<cuuint64_t>(p.page_size) * p.Hkv * kD * es};
        const cuuint32_t bk = static_cast<cuuint32_t>(p.page_size < kKeys ? p.page_size : kKeys);
        const cuuint32_t box[4] = {64, 1, bk, 1};
        if (!encode(fn, &maps.kc, p.k_cache, 4, dims, str, box)) return cudaErrorInvalidValue;
        if (!encode(fn, &maps.vc, p.v_cache, 4, dims, str, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(p.Hkv),
                                    static_cast<cuuint64_t>(p.B) * p.N};
        const cuuint64_t str[2] = {kD * es, static_cast<cuuint64_t>(p.Hkv) * kD * es};
        const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kKeys)};
        if (!encode(fn, &maps.kt, p.k_tree, 3, dims, str, box)) return cudaErrorInvalidValue;
        if (!encode(fn, &maps.vt, p.v_tree, 3, dims, str, box)) return cudaErrorInvalidValue;
    }
    const bool whole = 128 % p.G == 0;
    cudaError_t e = cudaFuncSetAttribute(whole ? attn_tc_kernel<true> : attn_tc_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    const long long ctas = static_cast<long long>(p.max_chunks) * p.Hkv * p.tc_groups * p.B;
    if (ctas > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    // a programmatic dependent of the build: the context streams while the
    // build finishes; the tree is read after griddepcontrol.wait
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return whole ? cudaLaunchKernelEx(&cfg, attn_tc_kernel<true>, p, maps)
                 : cudaLaunchKernelEx(&cfg, attn_tc_kernel<false>, p, maps);
}

}  // namespace ddt
