// Internal interface between the host runtime (ub_api.cu) and the GEMM kernel
// (ub_gemm.cu). Not installed; the public ABI is include/ub.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ub.h"

namespace ubk {

// Tile shape of the persistent kernel: one CTA owns a 128 x 256 output tile at a
// time, accumulating in TMEM (128 lanes x 256 fp32 columns, double-buffered), with a
// 4-stage shared-memory ring of 128x64 (A) and 256x64 (B) BF16 tiles in the 128-byte
// swizzled layout the tensor memory accelerator writes.
constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;          // 64 bf16 = 128 bytes = one swizzle row
constexpr int STAGES = 4;
constexpr int EPI_WARPS = 4;
constexpr int THREADS = 64 + 32 * EPI_WARPS;  // producer warp, MMA warp, epilogue warps
constexpr int STORE_COLS = 64;  // epilogue store box: 64 columns x 32 rows
constexpr int A_STAGE_BYTES = BM * BK * 2;
constexpr int B_STAGE_BYTES = BN * BK * 2;
constexpr int EPI_BUF_BYTES = 32 * STORE_COLS * 2;  // 4 KiB per warp per buffer
constexpr int SMEM_BYTES = 1024 /* alignment slack */ + STAGES * (A_STAGE_BYTES + B_STAGE_BYTES) +
                           EPI_WARPS * 2 * EPI_BUF_BYTES + 256 /* barriers */;
constexpr int TMEM_COLS = 2 * BN;  // two accumulators

// CTA-pair variant (tcgen05 cta_group::2): a cluster of two CTAs on neighbouring SMs
// owns a 256 x 256 output tile. Each CTA loads its own 128 rows of A and its own
// 128-row half of B per k-block (32 KiB instead of 48 KiB), the even CTA issues one
// 256x256x16 MMA that reads both CTAs' shared memory, and each CTA's TMEM receives its
// 128 rows. Less shared memory per stage leaves room for 6 stages.
constexpr int PAIR_BM = 256;             // rows of a pair tile (128 per CTA)
constexpr int PAIR_MAX_REGS = 168;       // per thread: 192 x 168 leaves half of an SM's registers free
constexpr int PAIR_STAGES = 6;
constexpr int PAIR_A_BYTES = 128 * BK * 2;
constexpr int PAIR_B_BYTES = 128 * BK * 2;  // this CTA's half of the 256-row B tile
constexpr int PAIR_SMEM_BYTES = 1024 + PAIR_STAGES * (PAIR_A_BYTES + PAIR_B_BYTES) +
                                EPI_WARPS * 2 * EPI_BUF_BYTES + 256;
// One CTA's share of a partial pair tile: 128 rows x 256 fp32 columns.
constexpr int PARTIAL_FLOATS = 128 * BN;
// A split tail tile is never cut into pieces of fewer than this many k-blocks.
constexpr int MIN_KBLOCKS_PER_PIECE = 16;
// Nor into more than this many pieces.
constexpr int MAX_TAIL_SPLIT = 8;

// Skinny kernel (few active tokens): 128 weight rows per tile, pipeline depth chosen per
// call from the token tile's size, partial tiles of split pieces in the workspace.
constexpr int SK_BM = 128;
constexpr int SK_MAX_COLS = 256;         // token columns of one accumulator
constexpr int SK_AUTO_MAX_COLS = 128;    // chosen by default up to here (beyond, the tile kernels win)
constexpr int SK_MAX_STAGES = 12;
constexpr int SK_MIN_KBLOCKS = 8;        // a k-piece is never shorter than this
constexpr int SK_MAX_SPLIT = 6;          // nor is a tile cut into more pieces
constexpr int SK_SMEM_LIMIT = 232448;    // dynamic shared memory a CTA may opt into
constexpr int SK_W_BYTES = SK_BM * BK * 2;

enum Mode : int { MODE_AG = 0, MODE_RS = 1, MODE_AG_GLU = 2 /* AG-GEMM + SwiGLU epilogue */ };

// Kernel parameters, passed by value as a __grid_constant__ (tensor maps must live
// in parameter, constant or global memory).
struct GemmParams {
    CUtensorMap tmA[UB_MAX_TP];  // AG: chunk r ([c, hidden] view); RS: A_j ([T, K])
    CUtensorMap tmB[UB_MAX_TP];  // AG: [0] = Wt ([N, hidden]); RS: Bt_j ([hidden, K])
    CUtensorMap tmY[UB_MAX_TP];  // output block r: AG [c, N] of Y; RS Y_shards[r] [c, hidden]
    const uint32_t *flags;       // AG readiness flag per chunk (device)
    uint32_t *abort_word;        // epoch of an aborted call (device)
    int32_t *status;             // sticky UB_ERR_* (device)
    uint64_t timeout_ns;
    uint32_t epoch;
    int tp;
    int c;                       // rows per chunk = T / tp
    int n_out;                   // N (AG) or hidden (RS)
    int k_blocks;                // BK-blocks per tile (RS: over all tp shards)
    int k_blocks_per_shard;      // RS: BK-blocks of one shard's K
    int m_tiles;                 // per chunk: ceil(c / BM)
    int n_tiles;                 // ceil(n_out / BN)
    int num_tiles;               // tp * m_tiles * n_tiles
    int self_rank;               // AG: chunk read in place, no flag wait
    int self_head;               // AG: rows of the self chunk read in place (the CTA-pair
                                 // kernel reads the rest from the buffer); c elsewhere

    // ---- CTA-pair kernel only: row regions and the split last wave.
    // The pair kernel tiles rows by region instead of by chunk. RS has one region,
    // [0, T): its tiles may span chunks, and the epilogue splits stores at chunk ends.
    // AG has one region per source of A rows, in ring order: the self chunk (read in
    // place from its shard), then the chunks after it, then the chunks before it (both
    // read from the user buffer, each row only once its chunk's flag is set). Region q
    // uses tmA[q] and tmY[q], whose row extents end exactly at the region's end.
    int n_regions;
    int region_row0[3];          // first row of region q (global row of the active prefix)
    int region_rows[3];
    int region_ub[3];            // 1: rows come from the user buffer (flag waits)
    int region_tile0[4];         // first pair tile of region q; [n_regions] = total
    int num_pairs;               // clusters launched
    int dp_tiles;                // tiles [0, dp_tiles) go whole to pairs in strided order
                                 // (pair p: p, p + num_pairs, ...)
    int tail_split;              // the remaining tiles are cut into this many k-pieces
    int group_m;                 // > 1: tiles walked in groups of this many 256-row tile rows,
                                 // rows fastest inside a group (RS whose weight panels
                                 // together exceed L2; AG with chunks of >= 2 tile rows);
                                 // else N fastest
    int ldy;                     // RS: leading dimension of Y_shards (= hidden)
    void *y_ptr[UB_MAX_TP];      // RS: Y_shards[r], for stores that cross a chunk end
    int glu_f;                   // MODE_AG_GLU: F, the width of each half (gate, up) of Wt
    int a_mn;                    // 1: A is MN-major (stored K x M; tensor map inner dim = M)
    int b_mn;                    // 1: B is MN-major (stored K x N; tensor map inner dim = N)
    float *ws;                   // partial tiles of split tail tiles: [num_pairs][2][256/4][128][4] fp32
    uint32_t *ws_flags;          // [num_pairs][2][EPI_WARPS]: epoch of the partial written

    // ---- fused gather (tile kernels, AG modes): the epilogue warps copy the chunks into
    // the user buffer before their first tile and publish each chunk's readiness flag
    int fused_gather;            // 1: chunk by chunk; 2: the chunks end to end, one range per
                                 // CTA (one wave of tiles); 3: each chunk by its own group of
                                 // g_group CTAs (few tokens); the host then issues no copies
    int g_group;                 // fused_gather 3: CTAs per chunk
    int g_drop;                  // chunk whose flag is not published (-1: none)
    const void *g_src[UB_MAX_TP];  // shard r ([c, hidden])
    void *g_ub;                  // user buffer base
    uint32_t *g_counters;        // CTAs done per chunk (zero between calls)
    int64_t g_chunk_vecs;        // 16-byte vectors per chunk = c * hidden / 8
    int64_t g_self_head_vecs;    // vectors of the self chunk's first self_head rows

    // ---- skinny kernel only (few tokens): weight rows on the MMA's M dimension, tokens
    // on its N dimension. Tiles are SK_BM weight rows (SwiGLU: SK_BM gate + SK_BM up rows)
    // by all T tokens; work units are (tile, k-piece), unit u = piece * n_tiles + tile.
    int sk_sub_n;                // token columns per sub-tile (multiple of 16, <= 256)
    int sk_n_sub;                // sub-tiles: AG one per chunk (rows of chunk r), RS one
    int sk_stride;               // TMEM columns between the two accumulators (power of two)
    int sk_split;                // k-pieces per tile; the last piece finishes the tile
    int sk_stages;               // shared-memory pipeline depth (<= SK_MAX_STAGES)
    int sk_units;                // n_tiles * sk_split
    int pdl;                     // host: launch with programmatic stream serialization
    int after_gather;            // AG launched as the programmatic dependent of its gather kernel:
                                 // no wait at entry (the chunk flags order the buffer reads), one
                                 // thread waits for the gather at exit
};

// Launch the persistent GEMM (mode MODE_AG, MODE_AG_GLU or MODE_RS) with `grid` CTAs on
// `stream`. SwiGLU: the tensor map of Wt has 128-row boxes (gate at row 128n, up at
// glu_f + 128n) and n_tiles counts 128-feature tiles.
cudaError_t launch_gemm(const GemmParams &p, int mode, int grid, cudaStream_t stream);

// Launch the CTA-pair variant with `clusters` clusters of two CTAs. The tensor maps of
// B must have 128-row boxes and m_tiles must count 256-row pair tiles.
cudaError_t launch_gemm_pair(const GemmParams &p, int mode, int clusters, cudaStream_t stream);

// Clusters of two CTAs of the pair kernel that can be resident at once (0 on error).
int max_pair_clusters(int mode);

// Launch the skinny kernel (ub_skinny.cu) with `grid` CTAs; the tensor maps of the weight
// have 128-row boxes (K-major) or 64 x 64 boxes (MN-major), those of the tokens
// sk_sub_n-row boxes.
cudaError_t launch_gemm_skinny(const GemmParams &p, int mode, int grid, cudaStream_t stream);

// Dynamic shared memory of the skinny kernel for a pipeline of `stages`.
int skinny_smem_bytes(int stages, int w_bytes, int x_bytes);

// Calibration read (ub_skinny.cu): `bytes` of `src` streamed into shared memory by bulk
// copies, one contiguous share per CTA, and discarded: the cost of reading those bytes
// once in one kernel, which a few-token call (whose work is its weight read) cannot beat.
struct StreamReadParams {
    const char *src;
    int64_t bytes;               // multiple of 16
    uint32_t *abort_word;
    int32_t *status;
    uint64_t timeout_ns;
    uint32_t epoch;
    int pdl;                     // host: launch with programmatic stream serialization
};
cudaError_t launch_stream_read(const StreamReadParams &p, int grid, cudaStream_t stream);

// Standalone reduce-scatter (ub_bulk.cu): Y[r][i][:] = sum_j P[j][r*c + i][:].
struct BulkRsParams {
    const void *P[UB_MAX_TP];  // tp partials [T, H] bf16
    void *Y[UB_MAX_TP];        // tp row blocks [c, H] bf16
    int tp;
    int64_t T;
    int64_t H;                 // multiple of 8
    int64_t c;
    int pdl;                   // host: launch with programmatic stream serialization
    int beside;                // launched beside the GEMM before it: no entry wait, wait at exit
};
cudaError_t launch_bulk_rs(const BulkRsParams &p, int grid, cudaStream_t stream);

// One-launch gather (ub_bulk.cu): chunk r of the active shape into the user buffer, in
// ring order after the self rank, each chunk's readiness flag published (release) by
// the CTA that finishes it. Counters are reset by that CTA for the next call.
struct GatherParams {
    const void *src[UB_MAX_TP];  // shards [c, H]
    void *ub;                    // user buffer [T, H]
    uint32_t *flags;             // readiness flag per chunk
    uint32_t *counters;          // CTAs done per chunk (zero between calls)
    uint32_t epoch;
    int tp;
    int self_rank;
    int drop;                    // chunk whose flag is not published (-1: none)
    int ctas_per_chunk;
    int64_t chunk_vecs;          // 16-byte vectors per chunk = c * H / 8
    int pdl;                     // host: launch with programmatic stream serialization
    int beside;                  // launched beside the GEMM before it: no entry wait, wait at exit
};
cudaError_t launch_gather(const GatherParams &p, cudaStream_t stream);

// Record the message ub_last_error() returns on this host thread.
void set_last_error(const char *msg);

// Launch `kernel(params)` with `grid` x `threads`, `smem` dynamic shared memory, an
// optional cluster of `cluster_x` CTAs, and programmatic stream serialization if `pdl`.
template <typename P>
inline cudaError_t launch_ex(void (*kernel)(P), const P &params, int grid, int threads, int smem, int cluster_x,
                             bool pdl, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, params);
}

// Raise a kernel's dynamic shared memory limit to `bytes`, once per kernel and device
// (the runtime call costs microseconds of host time, paid once instead of per launch).
cudaError_t raise_smem_limit(const void *kernel, int bytes);

}  // namespace ubk
