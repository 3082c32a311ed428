// Persistent tcgen05 / TMEM BF16 GEMM for the active-shape AG-GEMM and GEMM-RS.
//
// One kernel, two modes:
//  * MODE_AG -- the column-parallel linear after the all-gather (QKV / fc1 diagrams of
//    "Do tp overlap support thd..."): Y[chunk r rows] = UB[chunk r rows] * Wt^T. Tiles
//    are walked chunk by chunk in ring order from the self rank ("ring_exchange" of
//    "How to setup TP Overlap configs", with the chunk loop on the device as in its
//    "atomic_gemm"); the producer waits for a chunk's readiness flag, written by the
//    copy's stream after it lands the chunk, before loading any of its rows.
//  * MODE_RS -- the row-parallel linear followed by the reduce-scatter (MLP diagram):
//    the K loop runs over (shard j, k-block), so sum_j A_j * Bt_j^T accumulates in
//    TMEM, and the epilogue writes the rows of block r straight into Y_shards[r].
//
// M tiles never straddle a chunk: tile rows are counted inside chunk r, and every
// tensor map of an output block (and, for AG, of an input chunk) has exactly c = T/tp
// rows, so the tensor memory accelerator zero-fills loads and drops stores past the
// chunk end. No byte past the active prefix is read or written ("Support dynamic
// token counts in TP communication/GEMM overlap", "Implementation approach").
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: flag waits, A/B tiles into a 4-stage smem ring
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma 128x256x16, fp32 in TMEM
//   warps 2..5  epilogue: tcgen05.ld -> bf16 -> swizzled smem -> TMA store
// The accumulator is double-buffered (2 x 256 TMEM columns), so the epilogue of one
// tile overlaps the main loop of the next.
//
// Every wait is bounded (%globaltimer): when one runs out the CTA records
// UB_ERR_TIMEOUT in the status word, publishes the call's epoch in the abort word so
// the other CTAs stop too, drains its own outstanding copies and MMAs, frees its TMEM
// and returns. Nothing traps.
#include <cuda_bf16.h>

#include <mutex>
#include <utility>
#include <vector>

#include "ub_device.cuh"
#include "ub_internal.h"

namespace ubk {
namespace {

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both K-major,
// N = BN, M = BM.
constexpr uint32_t kIdesc = (1u << 4)                           // D format: f32
                            | (1u << 7)                         // A format: bf16
                            | (1u << 10)                        // B format: bf16
                            | (static_cast<uint32_t>(BN >> 3) << 17)  // N / 8
                            | (static_cast<uint32_t>(BM >> 4) << 24); // M / 16

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

// ---- CTA-pair (cta_group::2) helpers

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank)
{
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
    return d;
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// TMA load into this CTA's shared memory that completes bytes on an mbarrier which may
// live in either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar_cluster, int x,
                                                 int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Instruction descriptor for the pair MMA: M = 256 (128 rows in each CTA), N = 256.
constexpr uint32_t kIdescPair = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                                (static_cast<uint32_t>(PAIR_BM >> 4) << 24);

// idesc: kIdescPair, plus bit 15 (A MN-major) / bit 16 (B MN-major) when set.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the mbarrier at `bar` in both CTAs of the pair once the MMAs issued so far
// have completed.
__device__ __forceinline__ void umma_commit_pair_both(uint32_t bar)
{
    const uint16_t mask = 0x3;
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::
                     "r"(bar),
                 "h"(mask)
                 : "memory");
}

__device__ __forceinline__ void umma_commit_pair_local(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// ------------------------------------------------------------------ tile walk

struct Tile {
    int r;  // chunk (AG) / output row block (RS)
    int m;  // M tile inside the chunk
    int n;  // N tile
};

template <int MODE>
__device__ __forceinline__ Tile tile_at(int t, const GemmParams &p)
{
    const int per_chunk = p.m_tiles * p.n_tiles;
    const int q = t / per_chunk;  // position in the ring
    const int rem = t - q * per_chunk;
    Tile x;
    if (MODE != MODE_RS) {
        int r = p.self_rank + q;
        x.r = r >= p.tp ? r - p.tp : r;
    } else {
        x.r = q;
    }
    x.m = rem / p.n_tiles;
    x.n = rem - x.m * p.n_tiles;
    return x;
}

// ------------------------------------------------------------------ the kernel

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1) ub_gemm_kernel(const __grid_constant__ GemmParams p)
{
    constexpr bool IS_AG = MODE != MODE_RS;
    // SwiGLU: the 256-row B tile is 128 gate rows and the matching 128 up rows (F further
    // down), so accumulator columns 0..127 hold the gate and 128..255 the up projections
    // of the same 128 outputs.
    constexpr bool GLU = MODE == MODE_AG_GLU;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *smA = base;
    uint8_t *smB = smA + STAGES * A_STAGE_BYTES;
    uint8_t *smE = smB + STAGES * B_STAGE_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smE + EPI_WARPS * 2 * EPI_BUF_BYTES);
    // barrier slots: full[STAGES], empty[STAGES], tmem_full[2], tmem_empty[2], drain
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const WaitCtx w{p.abort_word, p.status, p.timeout_ns, p.epoch};

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (!p.after_gather) pdl_wait();
    pdl_trigger();

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------------- producer
        const int nmaps = IS_AG ? 1 : p.tp;
        for (int i = 0; i < nmaps; ++i) prefetch_tmap(&p.tmB[i]);
        uint32_t stage = 0, phase = 0, ready = 0;
        int issued = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
            const Tile x = tile_at<MODE>(t, p);
            if (IS_AG && x.r != p.self_rank && !((ready >> x.r) & 1u)) {
                if (!wait_flag(p.flags + x.r, w)) {
                    ok = false;
                    break;
                }
                ready |= 1u << x.r;
            }
            const int arow = IS_AG ? x.m * BM : x.r * p.c + x.m * BM;
            const int brow = GLU ? x.n * 128 : x.n * BN;
            for (int kb = 0; kb < p.k_blocks; ++kb) {
                if (!mbar_wait(empty_bar(stage), phase ^ 1u, w)) {
                    ok = false;
                    break;
                }
                const CUtensorMap *ma;
                const CUtensorMap *mb;
                int kx;
                if (IS_AG) {
                    ma = &p.tmA[x.r];
                    mb = &p.tmB[0];
                    kx = kb * BK;
                } else {
                    const int j = kb / p.k_blocks_per_shard;
                    kx = (kb - j * p.k_blocks_per_shard) * BK;
                    ma = &p.tmA[j];
                    mb = &p.tmB[j];
                }
                mbar_arrive_expect_tx(full_bar(stage), A_STAGE_BYTES + B_STAGE_BYTES);
                tma_load_2d(smem_u32(smA + stage * A_STAGE_BYTES), ma, full_bar(stage), kx, arow);
                tma_load_2d(smem_u32(smB + stage * B_STAGE_BYTES), mb, full_bar(stage), kx, brow);
                if (GLU)  // B map boxes are 128 rows: the up rows go to the second half
                    tma_load_2d(smem_u32(smB + stage * B_STAGE_BYTES) + B_STAGE_BYTES / 2, mb, full_bar(stage), kx,
                                brow + p.glu_f);
                ++issued;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // Drain: the last STAGES loads must have landed before the CTA may exit.
        for (int i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
            mbar_wait_drain(full_bar(i % STAGES), static_cast<uint32_t>(i / STAGES) & 1u, p.timeout_ns);
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------------- MMA issuer
        uint32_t stage = 0, phase = 0;
        int local = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x, ++local) {
            const uint32_t acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, w)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int kb = 0; kb < p.k_blocks; ++kb) {
                if (!mbar_wait(full_bar(stage), phase, w)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_u32(smA + stage * A_STAGE_BYTES);
                const uint32_t b0 = smem_u32(smB + stage * B_STAGE_BYTES);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma_bf16(d_tmem, smem_desc_sw128(a0 + 32u * k), smem_desc_sw128(b0 + 32u * k),
                              (kb | k) != 0 ? 1u : 0u);
                umma_commit(empty_bar(stage));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit(tfull_bar(acc));
        }
        // Drain: every MMA issued must be complete before TMEM is released.
        umma_commit(drain_bar);
        mbar_wait_drain(drain_bar, 0, p.timeout_ns);
    } else if (warp >= 2) {
        // ---------------------------------------------------------- epilogue
        if (IS_AG && p.fused_gather) fused_gather(p, static_cast<int>(threadIdx.x) - 64);
        const int quarter = warp & 3;  // TMEM lanes this warp may read: 32*quarter ...
        uint8_t *ebuf = smE + (warp - 2) * 2 * EPI_BUF_BYTES;
        const uint32_t ebuf0 = smem_u32(ebuf);
        int local = 0, nstore = 0;
        for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++local) {
            const Tile x = tile_at<MODE>(t, p);
            const uint32_t acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            // One lane waits and the warp follows its verdict, so the warp never splits
            // around the warp-wide tcgen05.ld below.
            int live = 0;
            if (lane == 0) live = mbar_wait(tfull_bar(acc), acc_phase, w) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, live, 0)) break;
            tc_fence_after();
            const int row0 = x.m * BM + quarter * 32;  // first row of this warp's slab, inside block r
            const bool rows_live = row0 < p.c;
            const uint32_t trow = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
            if constexpr (GLU) {
                // Two output groups of 64 features: Z[:, 128n + 64h + j] = silu(gate) * up
                // from gate column 64h + j and up column 128 + 64h + j, in fp32 (silu with
                // the fast division, as in the pair kernel).
#pragma unroll 1
                for (int hs = 0; hs < 2; ++hs) {
                    uint32_t pk[STORE_COLS / 2];
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int c0 = hs * STORE_COLS + hf * 32;
                        uint32_t g[32], u[32];
                        tmem_ld32(trow + c0, g);
                        tmem_ld32(trow + 128 + c0, u);
                        tmem_wait_ld();
                        if (hs == 1 && hf == 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(tempty_bar(acc));
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float g0 = __uint_as_float(g[2 * j]), g1 = __uint_as_float(g[2 * j + 1]);
                            const float z0 = __fdividef(g0, 1.0f + __expf(-g0)) * __uint_as_float(u[2 * j]);
                            const float z1 = __fdividef(g1, 1.0f + __expf(-g1)) * __uint_as_float(u[2 * j + 1]);
                            pk[hf * 16 + j] = pack_bf16x2(__float_as_uint(z0), __float_as_uint(z1));
                        }
                    }
                    const int col = x.n * 128 + hs * STORE_COLS;
                    if (!rows_live || col >= p.n_out) continue;
                    const uint32_t buf = ebuf0 + (nstore & 1) * EPI_BUF_BYTES;
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                    const uint32_t rowaddr = buf + lane * 128u;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(rowaddr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4), pk[4 * j],
                                     pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&p.tmY[x.r], buf, col, row0);
                        bulk_commit();
                    }
                    ++nstore;
                }
            } else {
#pragma unroll 1
                for (int sub = 0; sub < BN / STORE_COLS; ++sub) {
                    uint32_t v[STORE_COLS];
                    tmem_ld32(trow + sub * STORE_COLS, v);
                    tmem_ld32(trow + sub * STORE_COLS + 32, v + 32);
                    tmem_wait_ld();
                    if (sub == BN / STORE_COLS - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(tempty_bar(acc));
                    }
                    const int col = x.n * BN + sub * STORE_COLS;
                    if (!rows_live || col >= p.n_out) continue;
                    const uint32_t buf = ebuf0 + (nstore & 1) * EPI_BUF_BYTES;
                    if (lane == 0) bulk_wait_read<1>();  // the store that last used `buf` has read it
                    __syncwarp();
                    const uint32_t rowaddr = buf + lane * 128u;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        st_shared_v4(rowaddr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4),
                                     pack_bf16x2(v[8 * j + 0], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                                     pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
                    }
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&p.tmY[x.r], buf, col, row0);
                        bulk_commit();
                    }
                    ++nstore;
                }
            }
        }
        if (lane == 0) bulk_wait_all();
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if (p.after_gather && threadIdx.x == 0) pdl_wait();  // complete only after the gather
}


// ------------------------------------------------------------------ the CTA-pair kernel

// Work split of the pair kernel. Tiles [0, dp_tiles) go whole to the pairs in strided
// order (pair p: p, p + P, p + 2P, ...), so the tiles in flight across all pairs stay
// close together and share L2. The remaining R tiles (fewer than P) form the last wave;
// with tail_split = s > 1 each of them is cut into s equal k-ranges ("pieces") held by
// s consecutive pairs, so that up to R * s pairs work on the last wave instead of R.
// All pieces start together and have the same length, so pairs that share a weight
// panel stay in step. The pair holding piece 0 finishes the tile: it adds the other
// pieces' fp32 partials, which their pairs publish in the workspace with the call's
// epoch, in piece order — a deterministic result for a given launch shape.
struct SegIter {
    int pair, num_pairs, kb, dp_tiles, tiles, split, i;
    bool tail_done;
    __device__ __forceinline__ SegIter(const GemmParams &p, int pr)
        : pair(pr), num_pairs(p.num_pairs), kb(p.k_blocks), dp_tiles(p.dp_tiles),
          tiles(p.region_tile0[p.n_regions]), split(p.tail_split), i(0), tail_done(false)
    {
    }
    // Next segment: tile t, k-blocks [k0, k1). False when the pair is done.
    __device__ __forceinline__ bool next(int &t, int &k0, int &k1)
    {
        const int tdp = pair + i * num_pairs;
        if (tdp < dp_tiles) {
            ++i;
            t = tdp;
            k0 = 0;
            k1 = kb;
            return true;
        }
        if (tail_done) return false;
        tail_done = true;
        if (pair >= (tiles - dp_tiles) * split) return false;
        t = dp_tiles + pair / split;
        const int q = pair - (pair / split) * split;
        k0 = q * kb / split;
        k1 = (q + 1) * kb / split;
        return true;
    }
};

struct PTile {
    int q;  // region
    int m;  // 256-row pair tile inside the region
    int n;  // 256-column tile
};

__device__ __forceinline__ PTile pair_tile_at(int t, const GemmParams &p)
{
    int q = 0;
    while (q + 1 < p.n_regions && t >= p.region_tile0[q + 1]) ++q;
    const int rem = t - p.region_tile0[q];
    PTile x;
    x.q = q;
    if (p.group_m > 1) {
        // groups of group_m tile rows (the last group may be shorter), rows fastest: a
        // wave of P tiles spans group_m activation panels and about P / group_m weight
        // panels instead of every weight panel
        const int mt = (p.region_tile0[q + 1] - p.region_tile0[q]) / p.n_tiles;
        const int per_group = p.group_m * p.n_tiles;
        const int g = rem / per_group;
        const int m0 = g * p.group_m;
        const int gm = mt - m0 < p.group_m ? mt - m0 : p.group_m;
        const int r = rem - g * per_group;
        x.n = r / gm;
        x.m = m0 + (r - x.n * gm);
        return x;
    }
    x.m = rem / p.n_tiles;
    x.n = rem - x.m * p.n_tiles;
    return x;
}


// Same roles as ub_gemm_kernel, on a cluster of two CTAs that share 256 x 256 tiles.
// Both CTAs run a producer (own A rows, own half of B) whose loads complete on the even
// CTA's `full` barrier; the even CTA's MMA thread issues the cta_group::2 MMAs and
// multicasts stage releases and accumulator-ready signals to both CTAs; each CTA's
// epilogue drains its own 128 TMEM lanes and reports back to the even CTA. Work is
// split across pairs by stream-K (above); rows are tiled by region (see GemmParams).
// MN: the instantiation that also reads MN-major operands (p.a_mn / p.b_mn); the forward
// instantiations leave those branches out of the load and MMA loops.
template <int MODE, bool MN>
// The register cap leaves room on every SM for another kernel's CTA next to this one:
// same-device cudaMemcpyAsync (the all-gather's chunk copies) runs as a kernel on SMs on
// this platform, and the GEMM waits for those copies, so they must be able to start.
__global__ void __maxnreg__(PAIR_MAX_REGS) ub_gemm_pair_kernel(const __grid_constant__ GemmParams p)
{
    constexpr bool IS_AG = MODE != MODE_RS;     // A rows come from regions of the gathered input
    constexpr bool GLU = MODE == MODE_AG_GLU;   // B tile = 128 gate rows (even CTA) + 128 up rows (odd CTA)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *smA = base;
    uint8_t *smB = smA + PAIR_STAGES * PAIR_A_BYTES;
    uint8_t *smE = smB + PAIR_STAGES * PAIR_B_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smE + EPI_WARPS * 2 * EPI_BUF_BYTES);
    // barrier slots: full[S], empty[S], tmem_full[2], tmem_empty[2], drain
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * PAIR_STAGES + 5);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (PAIR_STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * PAIR_STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * PAIR_STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * PAIR_STAGES + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();  // 0 = even CTA (issues the MMAs), 1 = its peer
    const int pair = blockIdx.x >> 1;
    const WaitCtx w{p.abort_word, p.status, p.timeout_ns, p.epoch};
    const int KB = p.k_blocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < PAIR_STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 2 * EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    cluster_sync_all();  // barriers of both CTAs initialised before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (!p.after_gather) pdl_wait();
    pdl_trigger();

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------------- producer (both CTAs)
        const int nmaps = IS_AG ? 1 : p.tp;
        for (int i = 0; i < nmaps; ++i) prefetch_tmap(&p.tmB[i]);
        uint32_t stage = 0, phase = 0, ready = 0;
        int issued = 0;
        bool ok = true;
        const int half = static_cast<int>(rank) * 128;
        SegIter it(p, pair);
        int t, k0, k1;
        while (ok && it.next(t, k0, k1)) {
            const PTile x = pair_tile_at(t, p);
            const int lrow = x.m * PAIR_BM + half;  // row of this CTA's half inside the region
            if (IS_AG && p.region_ub[x.q]) {
                const int g0 = p.region_row0[x.q] + lrow;
                const int g1 = min(g0 + 128, p.region_row0[x.q] + p.region_rows[x.q]) - 1;
                for (int ch = g0 / p.c; ok && g0 <= g1 && ch <= g1 / p.c; ++ch) {
                    if ((ready >> ch) & 1u) continue;
                    if (!wait_flag(p.flags + ch, w)) ok = false;
                    ready |= 1u << ch;
                }
                if (!ok) break;
            }
            // GLU: the even CTA loads gate rows [128n, 128n + 128) and the odd CTA the
            // matching up rows, F further down, so TMEM columns 0..127 hold the gate and
            // 128..255 the up projections of the same 128 outputs.
            const int brow = GLU ? x.n * 128 + (rank ? p.glu_f : 0) : x.n * BN + half;
            for (int kb = k0; kb < k1; ++kb) {
                if (!mbar_wait(empty_bar(stage), phase ^ 1u, w)) {
                    ok = false;
                    break;
                }
                const CUtensorMap *ma;
                const CUtensorMap *mb;
                int kx;
                if (IS_AG) {
                    ma = &p.tmA[x.q];
                    mb = &p.tmB[0];
                    kx = kb * BK;
                } else {
                    const int j = kb / p.k_blocks_per_shard;
                    kx = (kb - j * p.k_blocks_per_shard) * BK;
                    ma = &p.tmA[j];
                    mb = &p.tmB[j];
                }
                const uint32_t fb = map_to_rank(full_bar(stage), 0);
                if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * (PAIR_A_BYTES + PAIR_B_BYTES));
                const uint32_t sa = smem_u32(smA + stage * PAIR_A_BYTES);
                const uint32_t sb = smem_u32(smB + stage * PAIR_B_BYTES);
                // K-major operands: one 128-row x 64-K box. MN-major operands: two boxes of
                // 64 MN x 64 K rows (the tensor map's inner dimension is MN).
                if (MN && p.a_mn) {
                    tma_load_2d_pair(sa, ma, fb, lrow, kx);
                    tma_load_2d_pair(sa + MN_BOX_BYTES, ma, fb, lrow + 64, kx);
                } else {
                    tma_load_2d_pair(sa, ma, fb, kx, lrow);
                }
                if (MN && p.b_mn) {
                    tma_load_2d_pair(sb, mb, fb, brow, kx);
                    tma_load_2d_pair(sb + MN_BOX_BYTES, mb, fb, brow + 64, kx);
                } else {
                    tma_load_2d_pair(sb, mb, fb, kx, brow);
                }
                ++issued;
                if (++stage == PAIR_STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (rank == 0) {
            // The even CTA's full barriers also count the peer's bytes: once its last
            // stages have completed, every load of both CTAs for them has landed.
            for (int i = issued > PAIR_STAGES ? issued - PAIR_STAGES : 0; i < issued; ++i)
                mbar_wait_drain(full_bar(i % PAIR_STAGES), static_cast<uint32_t>(i / PAIR_STAGES) & 1u, p.timeout_ns);
        }
        if (!ok) settle(100000);  // abort path: let copies already issued land
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ---------------------------------------------------------- MMA issuer (even CTA)
        const uint32_t idesc = kIdescPair | (MN && p.a_mn ? (1u << 15) : 0u) | (MN && p.b_mn ? (1u << 16) : 0u);
        uint32_t stage = 0, phase = 0;
        int local = 0;
        bool ok = true;
        SegIter it(p, pair);
        int t, k0, k1;
        for (; ok && it.next(t, k0, k1); ++local) {
            const uint32_t acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, w)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int kb = k0; kb < k1; ++kb) {
                if (!mbar_wait(full_bar(stage), phase, w)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_u32(smA + stage * PAIR_A_BYTES);
                const uint32_t b0 = smem_u32(smB + stage * PAIR_B_BYTES);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma_bf16_pair(d_tmem,
                                   MN && p.a_mn ? smem_desc_mn_sw128(a0 + 2048u * k) : smem_desc_sw128(a0 + 32u * k),
                                   MN && p.b_mn ? smem_desc_mn_sw128(b0 + 2048u * k) : smem_desc_sw128(b0 + 32u * k),
                                   idesc,
                                   (kb != k0 || k != 0) ? 1u : 0u);
                umma_commit_pair_both(empty_bar(stage));
                if (++stage == PAIR_STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit_pair_both(tfull_bar(acc));
        }
        umma_commit_pair_local(drain_bar);
        mbar_wait_drain(drain_bar, 0, p.timeout_ns);
    } else if (warp >= 2) {
        // ---------------------------------------------------------- epilogue (both CTAs)
        if (IS_AG && p.fused_gather) fused_gather(p, static_cast<int>(threadIdx.x) - 64);
        const int quarter = warp & 3;
        uint8_t *ebuf = smE + (warp - 2) * 2 * EPI_BUF_BYTES;
        const uint32_t ebuf0 = smem_u32(ebuf);
        const int my_slot = (pair * 2 + static_cast<int>(rank)) * EPI_WARPS + quarter;
        int local = 0, nstore = 0;
        SegIter it(p, pair);
        int t, k0, k1;
        for (; it.next(t, k0, k1); ++local) {
            const PTile x = pair_tile_at(t, p);
            const uint32_t acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            int live = 0;
            if (lane == 0) live = mbar_wait(tfull_bar(acc), acc_phase, w) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, live, 0)) break;
            tc_fence_after();
            const uint32_t trow = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
            const int lrow0 = x.m * PAIR_BM + static_cast<int>(rank) * 128 + quarter * 32;  // inside the region
            const int prow = quarter * 32 + lane;  // this thread's row inside the CTA's 128

            // A tile of the split last wave: its k-pieces are held by pairs p0 .. p0 + sp - 1
            // (piece q here), and each piece owns an equal share of the tile's output
            // units (64-column groups; with SwiGLU, 64-feature groups of gate and up
            // columns). A piece publishes its fp32 partial of the units it does not own,
            // then adds the other pieces' partials of its own units (own accumulator
            // first, then the pieces in order: deterministic for a given launch shape) and
            // stores them, so the fix-up of a tile is shared by its pairs. Whole tiles own
            // every unit and publish nothing.
            constexpr int UNITS = GLU ? 2 : BN / STORE_COLS;
            const bool split_seg = k1 - k0 < KB;
            const int sp = split_seg ? p.tail_split : 1;
            const int q = split_seg ? pair % sp : 0;
            const int p0 = pair - q;
            const int u_lo = q * UNITS / sp, u_hi = (q + 1) * UNITS / sp;
            auto owned = [&](int sub) {  // 64-column group `sub` of the accumulator (0..3)
                const int u = GLU ? (sub & 1) : sub;
                return u >= u_lo && u < u_hi;
            };
            if (split_seg) {
                float4 *dst = reinterpret_cast<float4 *>(p.ws + static_cast<size_t>(pair * 2 + rank) * PARTIAL_FLOATS);
#pragma unroll 1
                for (int sub = 0; sub < BN / STORE_COLS; ++sub) {
                    if (owned(sub)) continue;
                    uint32_t v[STORE_COLS];
                    tmem_ld32(trow + sub * STORE_COLS, v);
                    tmem_ld32(trow + sub * STORE_COLS + 32, v + 32);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < STORE_COLS / 4; ++i)
                        __stcg(dst + (sub * (STORE_COLS / 4) + i) * 128 + prow,
                               make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                           __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])));
                }
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    st_release_u32(p.ws_flags + my_slot, p.epoch);
                }
                if (u_lo == u_hi) {
                    // Nothing to store here: release the accumulator.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));
                    continue;
                }
                bool okw = true;
                for (int k = 0; okw && k < sp; ++k) {
                    if (k == q || p0 + k >= p.num_pairs) continue;
                    int got = 1;
                    if (lane == 0) {
                        const uint32_t *f = p.ws_flags + ((p0 + k) * 2 + static_cast<int>(rank)) * EPI_WARPS + quarter;
                        got = wait_partial(f, w) ? 1 : 0;
                    }
                    okw = __shfl_sync(0xffffffffu, got, 0) != 0;
                }
                if (!okw) {
                    // Abort: release the accumulator so the MMA side is not left waiting.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));
                    break;
                }
            }
            // The partials added into an owned unit: the other pieces' slots, in piece order.
            auto contrib = [&](int k) -> const float4 * {
                return reinterpret_cast<const float4 *>(p.ws + static_cast<size_t>((p0 + k) * 2 + rank) * PARTIAL_FLOATS);
            };

            if constexpr (GLU) {
                // Two output groups of 64 columns: gate columns [64h, 64h + 64) and up
                // columns 128 + [64h, 64h + 64) of the accumulator give
                // Z[:, 128n + 64h + j] = silu(gate) * up, computed in fp32. silu(g) =
                // g / (1 + e^-g) takes the fast division (__fdividef, within 2 ulp): with
                // the IEEE division the epilogue slowed the whole call by 3-9 % on GB300
                // (T = 2048: 80.9 against 74.2 us).
#pragma unroll 1
                for (int hs = u_lo; hs < u_hi; ++hs) {
                    // 32 columns at a time keeps the live registers low enough for the
                    // kernel's register cap.
                    uint32_t pk[STORE_COLS / 2];
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int c0 = hs * STORE_COLS + hf * 32;  // gate column; up is c0 + 128
                        uint32_t g[32], u[32];
                        tmem_ld32(trow + c0, g);
                        tmem_ld32(trow + 128 + c0, u);
                        tmem_wait_ld();
                        if (hs == u_hi - 1 && hf == 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));
                        }
                        for (int k = 0; k < sp; ++k) {
                            if (k == q) continue;
                            const float4 *src = contrib(k);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float4 a = __ldcg(src + (c0 / 4 + i) * 128 + prow);
                                const float4 b = __ldcg(src + ((128 + c0) / 4 + i) * 128 + prow);
                                g[4 * i + 0] = __float_as_uint(__uint_as_float(g[4 * i + 0]) + a.x);
                                g[4 * i + 1] = __float_as_uint(__uint_as_float(g[4 * i + 1]) + a.y);
                                g[4 * i + 2] = __float_as_uint(__uint_as_float(g[4 * i + 2]) + a.z);
                                g[4 * i + 3] = __float_as_uint(__uint_as_float(g[4 * i + 3]) + a.w);
                                u[4 * i + 0] = __float_as_uint(__uint_as_float(u[4 * i + 0]) + b.x);
                                u[4 * i + 1] = __float_as_uint(__uint_as_float(u[4 * i + 1]) + b.y);
                                u[4 * i + 2] = __float_as_uint(__uint_as_float(u[4 * i + 2]) + b.z);
                                u[4 * i + 3] = __float_as_uint(__uint_as_float(u[4 * i + 3]) + b.w);
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float g0 = __uint_as_float(g[2 * j]), g1 = __uint_as_float(g[2 * j + 1]);
                            const float z0 = __fdividef(g0, 1.0f + __expf(-g0)) * __uint_as_float(u[2 * j]);
                            const float z1 = __fdividef(g1, 1.0f + __expf(-g1)) * __uint_as_float(u[2 * j + 1]);
                            pk[hf * 16 + j] = pack_bf16x2(__float_as_uint(z0), __float_as_uint(z1));
                        }
                    }
                    const int col = x.n * 128 + hs * STORE_COLS;
                    if (col >= p.n_out || lrow0 >= p.region_rows[x.q]) continue;
                    const uint32_t buf = ebuf0 + (nstore & 1) * EPI_BUF_BYTES;
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                    const uint32_t rowaddr = buf + lane * 128u;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(rowaddr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4), pk[4 * j],
                                     pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&p.tmY[x.q], buf, col, lrow0);
                        bulk_commit();
                    }
                    ++nstore;
                }
            } else {
#pragma unroll 1
                for (int sub = u_lo; sub < u_hi; ++sub) {
                    uint32_t v[STORE_COLS];
                    tmem_ld32(trow + sub * STORE_COLS, v);
                    tmem_ld32(trow + sub * STORE_COLS + 32, v + 32);
                    tmem_wait_ld();
                    if (sub == u_hi - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));
                    }
                    for (int k = 0; k < sp; ++k) {
                        if (k == q) continue;
                        const float4 *src = contrib(k);
#pragma unroll
                        for (int i = 0; i < STORE_COLS / 4; ++i) {
                            const float4 q = __ldcg(src + (sub * (STORE_COLS / 4) + i) * 128 + prow);
                            v[4 * i + 0] = __float_as_uint(__uint_as_float(v[4 * i + 0]) + q.x);
                            v[4 * i + 1] = __float_as_uint(__uint_as_float(v[4 * i + 1]) + q.y);
                            v[4 * i + 2] = __float_as_uint(__uint_as_float(v[4 * i + 2]) + q.z);
                            v[4 * i + 3] = __float_as_uint(__uint_as_float(v[4 * i + 3]) + q.w);
                        }
                    }
                    const int col = x.n * BN + sub * STORE_COLS;
                    if (col >= p.n_out || lrow0 >= p.region_rows[x.q]) continue;
                    // Pack to bf16 (row-major, 8 x 16 bytes per thread).
                    uint32_t pk[STORE_COLS / 2];
#pragma unroll
                    for (int j = 0; j < STORE_COLS / 2; ++j) pk[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);

                    int chunk = 0;  // output block of a TMA store (RS), or -1 = direct stores
                    int brow = lrow0;
                    if (MODE == MODE_RS) {
                        const int last = min(lrow0 + 31, p.region_rows[0] - 1);
                        chunk = lrow0 / p.c;
                        if (last / p.c != chunk) {
                            chunk = -1;
                        } else {
                            brow = lrow0 - chunk * p.c;
                        }
                    } else {
                        chunk = x.q;
                    }
                    if (chunk < 0) {
                        // The 32 rows cross a chunk end: each thread writes its own row to the
                        // output block that owns it.
                        const int row = lrow0 + lane;
                        if (row < p.region_rows[0]) {
                            const int r = row / p.c;
                            const int i = row - r * p.c;
                            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.y_ptr[r]) +
                                                                   static_cast<size_t>(i) * p.ldy + col);
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                if (col + 8 * j < p.n_out) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                        }
                        continue;
                    }
                    const uint32_t buf = ebuf0 + (nstore & 1) * EPI_BUF_BYTES;
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                    const uint32_t rowaddr = buf + lane * 128u;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(rowaddr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4), pk[4 * j],
                                     pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&p.tmY[chunk], buf, col, brow);
                        bulk_commit();
                    }
                    ++nstore;
                }
            }
        }
        if (lane == 0) bulk_wait_all();
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync_all();  // neither CTA leaves while the pair's MMAs may touch its memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
    if (p.after_gather && threadIdx.x == 0) pdl_wait();  // complete only after the gather
}

}  // namespace

cudaError_t raise_smem_limit(const void *kernel, int bytes)
{
    static std::mutex mu;
    static std::vector<std::pair<const void *, int>> done;  // (kernel, device)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (const auto &d : done)
        if (d.first == kernel && d.second == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.emplace_back(kernel, dev);
    return e;
}

int max_pair_clusters(int mode)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = PAIR_SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e;
    if (mode == MODE_AG) {
        e = raise_smem_limit(reinterpret_cast<const void *>(ub_gemm_pair_kernel<MODE_AG, false>), PAIR_SMEM_BYTES);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, ub_gemm_pair_kernel<MODE_AG, false>, &cfg);
    } else if (mode == MODE_AG_GLU) {
        e = raise_smem_limit(reinterpret_cast<const void *>(ub_gemm_pair_kernel<MODE_AG_GLU, false>), PAIR_SMEM_BYTES);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, ub_gemm_pair_kernel<MODE_AG_GLU, false>, &cfg);
    } else {
        e = raise_smem_limit(reinterpret_cast<const void *>(ub_gemm_pair_kernel<MODE_RS, false>), PAIR_SMEM_BYTES);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, ub_gemm_pair_kernel<MODE_RS, false>, &cfg);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_gemm_pair(const GemmParams &p, int mode, int clusters, cudaStream_t stream)
{
    // MN-major operands only in the backward GEMMs' instantiations (never with SwiGLU)
    const bool mn = p.a_mn || p.b_mn;
    auto go = [&](void (*kernel)(GemmParams)) {
        cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(kernel), PAIR_SMEM_BYTES);
        return e == cudaSuccess ? launch_ex(kernel, p, 2 * clusters, THREADS, PAIR_SMEM_BYTES, 2, p.pdl != 0, stream) : e;
    };
    cudaError_t e;
    if (mode == MODE_AG)
        e = mn ? go(ub_gemm_pair_kernel<MODE_AG, true>) : go(ub_gemm_pair_kernel<MODE_AG, false>);
    else if (mode == MODE_AG_GLU)
        e = mn ? cudaErrorInvalidValue : go(ub_gemm_pair_kernel<MODE_AG_GLU, false>);
    else
        e = mn ? go(ub_gemm_pair_kernel<MODE_RS, true>) : go(ub_gemm_pair_kernel<MODE_RS, false>);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_gemm(const GemmParams &p, int mode, int grid, cudaStream_t stream)
{
    cudaError_t e;
    if (mode == MODE_AG_GLU) {
        e = raise_smem_limit(reinterpret_cast<const void *>(ub_gemm_kernel<MODE_AG_GLU>), SMEM_BYTES);
        if (e != cudaSuccess) return e;
        e = launch_ex(ub_gemm_kernel<MODE_AG_GLU>, p, grid, THREADS, SMEM_BYTES, 0, p.pdl != 0, stream);
        if (e != cudaSuccess) return e;
    } else if (mode == MODE_AG) {
        e = raise_smem_limit(reinterpret_cast<const void *>(ub_gemm_kernel<MODE_AG>), SMEM_BYTES);
        if (e != cudaSuccess) return e;
        e = launch_ex(ub_gemm_kernel<MODE_AG>, p, grid, THREADS, SMEM_BYTES, 0, p.pdl != 0, stream);
        if (e != cudaSuccess) return e;
    } else {
        e = raise_smem_limit(reinterpret_cast<const void *>(ub_gemm_kernel<MODE_RS>), SMEM_BYTES);
        if (e != cudaSuccess) return e;
        e = launch_ex(ub_gemm_kernel<MODE_RS>, p, grid, THREADS, SMEM_BYTES, 0, p.pdl != 0, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace ubk
