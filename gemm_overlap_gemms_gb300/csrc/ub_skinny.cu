// Skinny-token GEMM: the AG-GEMM, AG-GEMM + SwiGLU and GEMM-RS when the active token
// count is small (decode-like microbatches of "Support dynamic token counts in TP
// communication/GEMM overlap", TransformerEngine issue #3564, where T may be as low as tp).
//
// With few tokens the work is the weight read: every weight byte is used T times. A
// tile of 128 or 256 token rows on the tensor core's M dimension then computes mostly
// padding, and with one such tile per weight panel only a few dozen SMs pull weights.
// This kernel swaps the operand roles. The tensor core's M dimension runs over 128
// weight rows (output features) and its N dimension over the tokens, so one MMA computes
//
//   D[n, t] = sum_k W[n, k] * X[t, k]        (128 lanes x T columns of fp32 in TMEM)
//
// with N = the tokens rounded up to 16: the MMA work follows T, and the weight is read
// from HBM exactly once per call. The K range of each weight panel is cut into pieces
// so that about one work unit (panel, piece) runs per SM. Each piece owns an equal
// share of the token columns: it publishes its fp32 partial of the other columns in the
// workspace (with the call's epoch), adds the other pieces' partials of its own columns
// in a fixed order (deterministic for a given launch shape) and writes their outputs,
// so the pieces of a panel share its fix-up.
//
//  * AG (column-parallel, QKV / fc1): the tokens are the gathered chunks. Sub-tile r of
//    the token tile holds chunk r's c rows (the self chunk read in place from its shard,
//    the others from the user buffer once their readiness flags are set), so chunks of
//    any size stay apart and the rows past each chunk are zero-filled by the copy.
//  * AG + SwiGLU: each tile loads 128 gate rows and the 128 matching up rows of W; two
//    MMAs per k-step fill two accumulators, and every thread holds gate and up for its
//    own feature: Z[t, f] = silu(gate) * up needs no exchange.
//  * RS (row-parallel, attention out / fc2): the K loop runs over (shard j, k-block), so
//    the cross-shard sum accumulates in TMEM; token t of the result goes to row t - r*c
//    of Y_shards[r], r = t / c.
//
// Warp roles as in the other kernels: warp 0 loads (TMA), warp 1 owns TMEM and issues
// the MMAs, warps 2..5 drain TMEM. The weight load of a stage is issued before the
// chunk flags are checked, so the weight stream starts while the gather is in flight.
#include <cuda_bf16.h>

#include "ub_device.cuh"
#include "ub_internal.h"

namespace ubk {
namespace {

// kind::f16 instruction descriptor for M = 128 and N = n: fp32 accumulator, bf16 A and
// B, A (the weight) MN-major when `a_mn`.
__host__ __device__ constexpr uint32_t skinny_idesc(int n, bool a_mn)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn ? (1u << 15) : 0u) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(SK_BM >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16_id(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

struct Unit {
    int tile, piece, k0, k1;
};

// Partial tiles in the workspace are laid out per epilogue warp (quarter of the 128
// rows), so that one warp's share of a column range is contiguous:
//   float4 index = (quarter * cols4 + column / 4) * 32 + lane,   cols4 = slot columns / 4
// Fix-up chunks: columns per bulk-copied chunk, two chunks in flight per warp, each
// holding every other piece's partial of the chunk (SwiGLU: gate and up).
constexpr int FIX_CHUNK_COLS = 32;
constexpr int FIX_BUF_BYTES = (SK_MAX_SPLIT - 1) * FIX_CHUNK_COLS * 128;  // per warp per buffer
// The fix-up buffers (two per epilogue warp) reuse the stage buffers, which always hold
// at least SK_SMEM_LIMIT - 1536 - 64 KiB bytes (the pipeline is as deep as fits, a stage
// is at most 64 KiB).
static_assert(2 * EPI_WARPS * FIX_BUF_BYTES <= SK_SMEM_LIMIT - 1536 - 65536, "fix-up buffers exceed the stages");

__device__ __forceinline__ Unit unit_at(int u, const GemmParams &p)
{
    Unit x;
    x.piece = u / p.n_tiles;
    x.tile = u - x.piece * p.n_tiles;
    x.k0 = x.piece * p.k_blocks / p.sk_split;
    x.k1 = (x.piece + 1) * p.k_blocks / p.sk_split;
    return x;
}

// Workspace slot of a unit's published partial (SwiGLU units take two slots' room).
__device__ __forceinline__ int partial_slot(const Unit &x, const GemmParams &p) { return x.piece * p.n_tiles + x.tile; }

// The gather inside this kernel (UB_OPT_GATHER_KERNEL = 2; p.fused_gather == 3): the
// CTAs form groups of g_group; group k alone copies parts k, k + groups, ... (gather_part),
// each member a share, and CTAs past the last whole group copy nothing. A few-token
// call's chunks are small (T = 4, tp = 4: 8 KB), so a chunk is one CTA's or a few CTAs'
// work and its flag waits for no count across the grid (the tile kernels' part-by-part
// order, every CTA a share of every part, took 2-4 us longer here). The one-launch
// gather kernel on the side stream is still faster, by 2-5 us a call at T = 4-128 on
// GB300, and stays the default.
__device__ void fused_gather_grouped(const GemmParams &p, int et)
{
    const int gs = p.g_group;                           // 1 <= gs <= gridDim.x
    const int ng = static_cast<int>(gridDim.x) / gs;    // groups; group k copies parts k, k + ng, ...
    const int grp = static_cast<int>(blockIdx.x) / gs;
    if (grp >= ng) return;
    const int m = static_cast<int>(blockIdx.x) - grp * gs;
    const int np = gather_n_parts(p);
    for (int i = grp; i < np; i += ng) {
        const GatherPart g = gather_part(p, i);
        const int64_t per = (g.hi - g.lo + gs - 1) / gs;
        const int64_t v0 = g.lo + m * per;
        const int64_t v1 = v0 + per < g.hi ? v0 + per : g.hi;
        if (v1 > v0)
            copy_vecs(static_cast<const uint4 *>(p.g_src[g.r]) + v0,
                      static_cast<uint4 *>(p.g_ub) + static_cast<int64_t>(g.r) * p.g_chunk_vecs + v0, v1 - v0, et);
        if (!g.flag) continue;
        asm volatile("bar.sync 1, 128;" ::: "memory");  // this CTA's share is written
        if (et != 0) continue;
        __threadfence();
        if (gs > 1) {
            const uint32_t done = atomicAdd(p.g_counters + g.r, 1u) + 1u;
            if (done != static_cast<uint32_t>(gs)) continue;
            p.g_counters[g.r] = 0u;  // zero again for the next call
            __threadfence();
        }
        if (g.r != p.g_drop) st_release_u32(const_cast<uint32_t *>(p.flags) + g.r, p.epoch);
    }
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1) ub_gemm_skinny_kernel(const __grid_constant__ GemmParams p)
{
    constexpr bool IS_AG = MODE != MODE_RS;
    constexpr bool GLU = MODE == MODE_AG_GLU;
    constexpr int W_BYTES = GLU ? 2 * SK_W_BYTES : SK_W_BYTES;  // SwiGLU: gate rows, then up rows
    constexpr int SLOT_FLOATS = GLU ? 2 * PARTIAL_FLOATS : PARTIAL_FLOATS;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.sk_stages;
    const int sub_n = p.sk_sub_n;
    const int n_sub = p.sk_n_sub;
    const int acc_cols = n_sub * sub_n;
    const uint32_t x_bytes = static_cast<uint32_t>(acc_cols) * 128u;
    uint8_t *smW = base;
    uint8_t *smX = smW + S * W_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smX + S * x_bytes);
    // barrier slots: full[SK_MAX_STAGES], empty[SK_MAX_STAGES], tmem_full[2], tmem_empty[2],
    // drain, fix-up chunk[EPI_WARPS][2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * SK_MAX_STAGES + 5 + 2 * EPI_WARPS);
    volatile uint32_t *stop_flag = tmem_slot + 1;  // set by the producer when it gives up
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (SK_MAX_STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * SK_MAX_STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * SK_MAX_STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * SK_MAX_STAGES + 4);
    auto fix_bar = [&](int q, int b) { return bar0 + 8u * (2 * SK_MAX_STAGES + 5 + 2 * q + b); };
    // SwiGLU: one accumulator pair per unit (gate at column 0, up at sk_stride).
    // Otherwise two accumulators, at columns 0 and sk_stride, used alternately.
    const uint32_t tmem_cols = 2u * static_cast<uint32_t>(p.sk_stride) < 32u ? 32u : 2u * p.sk_stride;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const WaitCtx w{p.abort_word, p.status, p.timeout_ns, p.epoch};

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 2);  // one arrival with the weight bytes, one with the token bytes
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        for (int q = 0; q < EPI_WARPS; ++q) {
            mbar_init(fix_bar(q, 0), 1);
            mbar_init(fix_bar(q, 1), 1);
        }
        *stop_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (!p.after_gather) pdl_wait();
    pdl_trigger();

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------------- producer
        // With few tokens this thread issues a stage every few hundred ns, so the loop
        // keeps its per-stage work to a few instructions: shard and K offset advance
        // incrementally, no division or modulo.
        const int nw = IS_AG ? (GLU ? 2 : 1) : p.tp;
        for (int i = 0; i < nw; ++i) prefetch_tmap(&p.tmB[i]);
        for (int i = 0; i < p.tp; ++i) prefetch_tmap(&p.tmA[i]);
        const bool w_mn = p.b_mn != 0;
        const int kx_end = p.k_blocks_per_shard * BK;
        const uint32_t smW0 = smem_u32(smW), smX0 = smem_u32(smX);
        uint32_t stage = 0, phase = 0;
        int issued = 0;
        bool ok = true;
        bool ready = !IS_AG;  // AG: every chunk's flag seen
        for (int u = blockIdx.x; ok && u < p.sk_units; u += gridDim.x) {
            const Unit x = unit_at(u, p);
            const int n0 = x.tile * SK_BM;
            int j = IS_AG ? 0 : x.k0 / p.k_blocks_per_shard;  // shard of the current k-block (RS)
            int kx = (x.k0 - j * p.k_blocks_per_shard) * BK;   // its K offset inside the shard
            const CUtensorMap *mw = &p.tmB[j];
            const CUtensorMap *mx = &p.tmA[j];
            const int pend_kb = x.k0;     // AG before the flags: first k-block without token loads
            const int pend_issue = issued;
            for (int kb = x.k0; kb < x.k1; ++kb) {
                if (!mbar_wait(empty_bar(stage), phase ^ 1u, w)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = full_bar(stage);
                const uint32_t sw = smW0 + stage * W_BYTES;
                mbar_arrive_expect_tx(fb, W_BYTES);
                if (w_mn) {
                    // weight stored K x N: two boxes of 64 features x 64 K rows
                    tma_load_2d(sw, mw, fb, n0, kx);
                    tma_load_2d(sw + MN_BOX_BYTES, mw, fb, n0 + 64, kx);
                } else {
                    tma_load_2d(sw, mw, fb, kx, n0);
                    if (GLU) tma_load_2d(sw + SK_W_BYTES, &p.tmB[1], fb, kx, n0);
                }
                if (ready) {
                    const uint32_t sx = smX0 + stage * x_bytes;
                    mbar_arrive_expect_tx(fb, x_bytes);
                    if (IS_AG) {
                        for (int r = 0; r < p.tp; ++r)
                            tma_load_2d(sx + static_cast<uint32_t>(r * sub_n) * 128u, &p.tmA[r], fb, kx, 0);
                    } else {
                        tma_load_2d(sx, mx, fb, kx, 0);
                    }
                }
                ++issued;
                if (++stage == static_cast<uint32_t>(S)) {
                    stage = 0;
                    phase ^= 1u;
                }
                kx += BK;
                if (!IS_AG && kx == kx_end && kb + 1 < x.k1) {
                    kx = 0;
                    ++j;
                    mw = &p.tmB[j];
                    mx = &p.tmA[j];
                }
                if (!ready) {
                    // After each weight stage one look at the chunk flags, without waiting:
                    // where the gather has already landed them (it runs just ahead of this
                    // kernel), the token loads start with the first stages and the MMA with
                    // them. Only once the weight has run ahead as far as the stages allow
                    // (or the piece ended) does the producer wait for the flags. Then the
                    // token loads of the stages issued so far (k-blocks pend_kb .. kb).
                    // Measured on GB300 (one call after an L2 flush, AG + SwiGLU at T = 4):
                    // checking only once the stages were full saw the flags ~5 us into the
                    // kernel although the gather had set them as it started, the weight
                    // stream stalled meanwhile on stages the MMA could not use.
                    const uint32_t others = ((1u << p.tp) - 1u) & ~(1u << p.self_rank);
                    const bool full = issued - pend_issue == S || kb + 1 == x.k1;
                    if (!try_flags(p.flags, others, p.epoch)) {
                        if (!full) continue;
                        if (!wait_flags(p.flags, others, w)) ok = false;
                    }
                    if (!ok) break;
                    ready = true;
                    for (int q = pend_kb; q <= kb; ++q) {
                        const int slot = (pend_issue + (q - pend_kb)) % S;
                        const uint32_t sx = smX0 + static_cast<uint32_t>(slot) * x_bytes;
                        mbar_arrive_expect_tx(full_bar(slot), x_bytes);
                        for (int r = 0; r < p.tp; ++r)
                            tma_load_2d(sx + static_cast<uint32_t>(r * sub_n) * 128u, &p.tmA[r], full_bar(slot), q * BK,
                                        0);
                    }
                }
            }
            if (!ok) {
                // Stages whose weight is in flight but whose tokens were never requested:
                // make their second arrival, so that they complete once the weight lands
                // (the drain below waits for that); the MMA thread sees the stop flag.
                *stop_flag = 1u;
                if (!ready)
                    for (int i = pend_issue; i < issued; ++i) mbar_arrive(full_bar(i % S));
            }
        }
        // Drain: the last S loads must have landed before the CTA may exit.
        for (int i = issued > S ? issued - S : 0; i < issued; ++i)
            mbar_wait_drain(full_bar(i % S), static_cast<uint32_t>(i / S) & 1u, p.timeout_ns);
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------------- MMA issuer
        // One MMA per K=16 step covers every token sub-tile: they follow each other in
        // shared memory in the same 8-row swizzle atoms, so N = all token columns.
        // Descriptors advance by adding byte offsets / 16 to their start-address field.
        const uint32_t idesc = skinny_idesc(acc_cols, p.b_mn != 0);
        const uint64_t a_stage = W_BYTES >> 4, b_stage = x_bytes >> 4;
        const uint64_t a_k = p.b_mn ? (2048u >> 4) : (32u >> 4), b_k = 32u >> 4;
        const uint64_t a_base = p.b_mn ? smem_desc_mn_sw128(smem_u32(smW)) : smem_desc_sw128(smem_u32(smW));
        const uint64_t b_base = smem_desc_sw128(smem_u32(smX));
        constexpr uint64_t UP = SK_W_BYTES >> 4;  // SwiGLU: the up rows follow the gate rows
        uint32_t stage = 0, phase = 0;
        uint64_t ad = a_base, bd = b_base;
        int local = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < p.sk_units; u += gridDim.x, ++local) {
            const Unit x = unit_at(u, p);
            const uint32_t acc = GLU ? 0u : static_cast<uint32_t>(local & 1);
            const uint32_t acc_phase = GLU ? static_cast<uint32_t>(local & 1) : static_cast<uint32_t>((local >> 1) & 1);
            if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, w)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d0 = tmem_base + acc * static_cast<uint32_t>(p.sk_stride);
            const uint32_t d_up = d0 + static_cast<uint32_t>(p.sk_stride);
            for (int kb = x.k0; kb < x.k1; ++kb) {
                if (!mbar_wait(full_bar(stage), phase, w) || *stop_flag) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    const uint32_t accum = (kb != x.k0 || k != 0) ? 1u : 0u;
                    umma_bf16_id(d0, ad + k * a_k, bd + k * b_k, idesc, accum);
                    if (GLU) umma_bf16_id(d_up, ad + UP + k * a_k, bd + k * b_k, idesc, accum);
                }
                umma_commit(empty_bar(stage));
                ad += a_stage;
                bd += b_stage;
                if (++stage == static_cast<uint32_t>(S)) {
                    stage = 0;
                    phase ^= 1u;
                    ad = a_base;
                    bd = b_base;
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
        if (IS_AG && p.fused_gather) fused_gather_grouped(p, static_cast<int>(threadIdx.x) - 64);
        const int quarter = warp & 3;         // TMEM lanes this warp may read: 32*quarter ...
        const int row = quarter * 32 + lane;  // this thread's lane = weight row inside the tile
        const int T = p.tp * p.c;
        int local = 0;
        for (int u = blockIdx.x; u < p.sk_units; u += gridDim.x, ++local) {
            const Unit x = unit_at(u, p);
            const uint32_t acc = GLU ? 0u : static_cast<uint32_t>(local & 1);
            const uint32_t acc_phase = GLU ? static_cast<uint32_t>(local & 1) : static_cast<uint32_t>((local >> 1) & 1);
            int live = 0;
            if (lane == 0) live = mbar_wait(tfull_bar(acc), acc_phase, w) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, live, 0)) break;
            tc_fence_after();
            const uint32_t trow =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * static_cast<uint32_t>(p.sk_stride);

            constexpr int HALVES = GLU ? 2 : 1;
            constexpr int COLS4 = (GLU ? 2 * SK_MAX_COLS : SK_MAX_COLS) / 4;  // float4 columns of a slot
            // With the tile's K range cut into s pieces, piece q owns the token columns of
            // the 16-column groups [q * g16 / s, (q + 1) * g16 / s): it publishes its fp32
            // partial of every other column for the pieces that own them, then adds the
            // other pieces' partials of its own columns and writes their outputs, so the
            // fix-up of a tile is shared by its s CTAs (all resident: one unit per CTA).
            const int nsplit = p.sk_split;
            const int q = x.piece;
            const int g16 = acc_cols / 16;
            const int c_lo = q * g16 / nsplit * 16, c_hi = (q + 1) * g16 / nsplit * 16;
            const int np = nsplit - 1;  // partials added into the own columns
            if (np > 0) {
                float4 *dst = reinterpret_cast<float4 *>(p.ws + static_cast<size_t>(partial_slot(x, p)) * SLOT_FLOATS) +
                              quarter * COLS4 * 32 + lane;
#pragma unroll 1
                for (int c0 = 0; c0 < acc_cols; c0 += 16) {
                    if (c0 >= c_lo && c0 < c_hi) continue;
#pragma unroll
                    for (int h = 0; h < HALVES; ++h) {
                        const int tc = h * p.sk_stride + c0;
                        uint32_t v[16];
                        tmem_ld16(trow + tc, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            __stcg(dst + (tc / 4 + i) * 32,
                                   make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                               __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])));
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    st_release_u32(p.ws_flags + partial_slot(x, p) * EPI_WARPS + quarter, p.epoch);
                }
            }

            // The other pieces' partials of the own columns are streamed into this warp's
            // part of the (now idle) stage buffers by bulk copies, a chunk of columns at a
            // time, two chunks in flight; the sums run in a fixed order (own accumulator,
            // then the other pieces in piece order).
            int okw = 1;
            if (np > 0 && c_hi > c_lo && lane == 0) {
                for (int pc = 0; okw && pc < nsplit; ++pc)
                    if (pc != q) okw = wait_partial(p.ws_flags + (pc * p.n_tiles + x.tile) * EPI_WARPS + quarter, w) ? 1 : 0;
                asm volatile("fence.proxy.async.global;" ::: "memory");  // bulk copies read what was acquired
            }
            if (!__shfl_sync(0xffffffffu, okw, 0)) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(acc));
                break;
            }
            constexpr int CH = FIX_CHUNK_COLS / HALVES;  // columns per chunk
            const uint32_t fbuf = smem_u32(base) + static_cast<uint32_t>((warp - 2) * 2 * FIX_BUF_BYTES);
            const int n_chunks = (c_hi - c_lo + CH - 1) / CH;
            auto issue_chunk = [&](int ci) {
                const int ca = c_lo + ci * CH;
                const int cols = c_hi - ca < CH ? c_hi - ca : CH;
                const uint32_t bytes = static_cast<uint32_t>(cols) * 128u;
                const uint32_t bar = fix_bar(warp - 2, ci & 1);
                const uint32_t dst0 = fbuf + static_cast<uint32_t>((ci & 1) * FIX_BUF_BYTES);
                mbar_arrive_expect_tx(bar, bytes * static_cast<uint32_t>(np * HALVES));
                for (int k = 0; k < np; ++k) {
                    const int pc = k < q ? k : k + 1;
                    const float4 *src = reinterpret_cast<const float4 *>(
                                            p.ws + static_cast<size_t>(pc * p.n_tiles + x.tile) * SLOT_FLOATS) +
                                        quarter * COLS4 * 32;
                    for (int h = 0; h < HALVES; ++h)
                        bulk_load(dst0 + static_cast<uint32_t>((k * HALVES + h) * CH * 128),
                                  src + ((h * p.sk_stride + ca) / 4) * 32, bytes, bar);
                }
            };
            if (np > 0 && lane == 0) {
                if (n_chunks > 0) issue_chunk(0);
                if (n_chunks > 1) issue_chunk(1);
            }
            const int n = x.tile * SK_BM + row;  // output column (feature) of this thread
            const bool n_ok = n < p.n_out;
            int failed_chunk = -1;
#pragma unroll 1
            for (int ci = 0; ci < n_chunks; ++ci) {
                if (np > 0) {
                    int got = 1;
                    if (lane == 0) got = mbar_wait(fix_bar(warp - 2, ci & 1), static_cast<uint32_t>(ci >> 1) & 1u, w) ? 1 : 0;
                    if (!__shfl_sync(0xffffffffu, got, 0)) {
                        failed_chunk = ci;
                        break;
                    }
                }
                const uint32_t buf = fbuf + static_cast<uint32_t>((ci & 1) * FIX_BUF_BYTES);
                const int ca = c_lo + ci * CH;
                const int cb = ca + CH < c_hi ? ca + CH : c_hi;
#pragma unroll 1
                for (int c0 = ca; c0 < cb; c0 += 16) {
                    float a[16], b[16];
                    {
                        uint32_t v[16];
                        tmem_ld16(trow + c0, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) a[i] = __uint_as_float(v[i]);
                        if (GLU) {
                            tmem_ld16(trow + p.sk_stride + c0, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i) b[i] = __uint_as_float(v[i]);
                        }
                    }
                    for (int k = 0; k < np; ++k) {
#pragma unroll
                        for (int h = 0; h < HALVES; ++h) {
                            float *acc_h = h == 0 ? a : b;
                            const uint32_t src =
                                buf + static_cast<uint32_t>((k * HALVES + h) * CH * 128 + (c0 - ca) * 128) + lane * 16u;
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                float4 f;
                                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                             : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w)
                                             : "r"(src + i * 512u));
                                acc_h[4 * i] += f.x;
                                acc_h[4 * i + 1] += f.y;
                                acc_h[4 * i + 2] += f.z;
                                acc_h[4 * i + 3] += f.w;
                            }
                        }
                    }
                    if (!n_ok) continue;
                    // Output rows of tokens c0 .. c0+15, walked without division per token.
                    if (IS_AG) {
                        const int sb = c0 / sub_n;  // sub-tile (chunk) of these 16 columns
                        const int i0 = c0 - sb * sub_n;
                        __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(p.y_ptr[0]) +
                                           static_cast<int64_t>(sb * p.c + i0) * p.ldy + n;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float z = GLU ? __fdividef(a[i], 1.0f + __expf(-a[i])) * b[i] : a[i];
                            if (i0 + i < p.c) y[static_cast<int64_t>(i) * p.ldy] = __float2bfloat16_rn(z);
                        }
                    } else {
                        int r = c0 / p.c;
                        int ii = c0 - r * p.c;
                        __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(p.y_ptr[r]) + static_cast<int64_t>(ii) * p.ldy + n;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if (c0 + i >= T) break;
                            *y = __float2bfloat16_rn(a[i]);
                            y += p.ldy;
                            if (++ii == p.c && c0 + i + 1 < T) {
                                ii = 0;
                                ++r;
                                y = static_cast<__nv_bfloat16 *>(p.y_ptr[r]) + n;
                            }
                        }
                    }
                }
                if (np > 0 && ci + 2 < n_chunks) {
                    // every lane is done reading this buffer before the copy refills it
                    __syncwarp();
                    if (lane == 0) {
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        issue_chunk(ci + 2);
                    }
                }
            }
            if (failed_chunk >= 0 && lane == 0) {
                // Gave up waiting for chunk k = failed_chunk: chunks k and k + 1 may still be
                // in flight; let them land before the CTA exits.
                for (int k = failed_chunk; k < failed_chunk + 2 && k < n_chunks; ++k)
                    mbar_wait_drain(fix_bar(warp - 2, k & 1), static_cast<uint32_t>(k >> 1) & 1u, p.timeout_ns);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            if (failed_chunk >= 0) break;
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, tmem_cols);
    }
    if (p.after_gather && threadIdx.x == 0) pdl_wait();  // complete only after the gather
}

// Calibration read: each CTA streams one contiguous share of the bytes through a ring of
// SR_STAGES shared-memory buffers with 32 KB bulk copies (thread 0 issues, thread 32
// frees), the pipeline a few-token weight stream would use with nothing else to do.
constexpr int SR_STAGES = 6;
constexpr uint32_t SR_CHUNK = 32768;
constexpr int SR_SMEM = 128 + SR_STAGES * static_cast<int>(SR_CHUNK) + 2 * SR_STAGES * 8;

__global__ void __launch_bounds__(64, 1) stream_read_kernel(const __grid_constant__ StreamReadParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const uint32_t buf0 = smem_u32(base);
    const uint32_t bar0 = buf0 + SR_STAGES * SR_CHUNK;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (SR_STAGES + s); };
    if (threadIdx.x == 0) {
        for (int s = 0; s < SR_STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    const WaitCtx w{p.abort_word, p.status, p.timeout_ns, p.epoch};
    const int64_t vecs = p.bytes / 16;
    const int64_t per = (vecs + gridDim.x - 1) / gridDim.x * 16;
    const int64_t lo = static_cast<int64_t>(blockIdx.x) * per;
    const int64_t hi = lo + per < p.bytes ? lo + per : p.bytes;
    const int n = hi > lo ? static_cast<int>((hi - lo + SR_CHUNK - 1) / SR_CHUNK) : 0;
    if (threadIdx.x == 0) {
        int issued = 0;
        for (int i = 0; i < n; ++i) {
            const int s = i % SR_STAGES;
            if (!mbar_wait(empty_bar(s), ((i / SR_STAGES) & 1u) ^ 1u, w)) break;
            const int64_t o = lo + static_cast<int64_t>(i) * SR_CHUNK;
            const uint32_t bytes = static_cast<uint32_t>(hi - o < SR_CHUNK ? hi - o : SR_CHUNK);
            mbar_arrive_expect_tx(full_bar(s), bytes);
            bulk_load(buf0 + s * SR_CHUNK, p.src + o, bytes, full_bar(s));
            ++issued;
        }
        // the copies in flight must land before the CTA may exit
        for (int i = issued > SR_STAGES ? issued - SR_STAGES : 0; i < issued; ++i)
            mbar_wait_drain(full_bar(i % SR_STAGES), static_cast<uint32_t>(i / SR_STAGES) & 1u, p.timeout_ns);
    } else if (threadIdx.x == 32) {
        for (int i = 0; i < n; ++i) {
            const int s = i % SR_STAGES;
            if (!mbar_wait(full_bar(s), static_cast<uint32_t>(i / SR_STAGES) & 1u, w)) break;
            mbar_arrive(empty_bar(s));
        }
    }
}

}  // namespace

cudaError_t launch_stream_read(const StreamReadParams &p, int grid, cudaStream_t stream)
{
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(stream_read_kernel), SR_SMEM);
    if (e != cudaSuccess) return e;
    e = launch_ex(stream_read_kernel, p, grid, 64, SR_SMEM, 0, p.pdl != 0, stream);
    return e != cudaSuccess ? e : cudaGetLastError();
}

int skinny_smem_bytes(int stages, int w_bytes, int x_bytes)
{
    return 1024 /* alignment slack */ + stages * (w_bytes + x_bytes) + 512 /* barriers, TMEM slot, stop flag */;
}

cudaError_t launch_gemm_skinny(const GemmParams &p, int mode, int grid, cudaStream_t stream)
{
    const int wb = mode == MODE_AG_GLU ? 2 * SK_W_BYTES : SK_W_BYTES;
    const int smem = skinny_smem_bytes(p.sk_stages, wb, p.sk_n_sub * p.sk_sub_n * 128);
    if (smem > SK_SMEM_LIMIT || p.sk_stages < 1 || p.sk_stages > SK_MAX_STAGES) return cudaErrorInvalidValue;
    cudaError_t e;
    if (mode == MODE_AG) {
        e = raise_smem_limit(reinterpret_cast<const void *>(ub_gemm_skinny_kernel<MODE_AG>), SK_SMEM_LIMIT);
        if (e != cudaSuccess) return e;
        e = launch_ex(ub_gemm_skinny_kernel<MODE_AG>, p, grid, THREADS, smem, 0, p.pdl != 0, stream);
        if (e != cudaSuccess) return e;
    } else if (mode == MODE_AG_GLU) {
        e = raise_smem_limit(reinterpret_cast<const void *>(ub_gemm_skinny_kernel<MODE_AG_GLU>), SK_SMEM_LIMIT);
        if (e != cudaSuccess) return e;
        e = launch_ex(ub_gemm_skinny_kernel<MODE_AG_GLU>, p, grid, THREADS, smem, 0, p.pdl != 0, stream);
        if (e != cudaSuccess) return e;
    } else {
        e = raise_smem_limit(reinterpret_cast<const void *>(ub_gemm_skinny_kernel<MODE_RS>), SK_SMEM_LIMIT);
        if (e != cudaSuccess) return e;
        e = launch_ex(ub_gemm_skinny_kernel<MODE_RS>, p, grid, THREADS, smem, 0, p.pdl != 0, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace ubk
