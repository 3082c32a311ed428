// Host runtime of libubgemm: the C ABI declared in include/ub.h.
//
// A handle is the registered user buffer of "Support dynamic token counts in TP
// communication/GEMM overlap" (TransformerEngine issue #3564): one allocation at
// capacity [max_tokens, hidden], an active shape that is only a logical view (nothing
// allocated, freed or re-registered per microbatch), and chunk offsets computed from
// the active first dimension. The all-gather stands in for the "ring_exchange" method
// with copy-engine send/recv ("use_ce") of "How to setup TP Overlap configs"
// (TransformerEngine issue #1344), collapsed onto one GPU: each virtual rank's chunk is
// a device-to-device cudaMemcpyAsync on a side stream, followed by a stream memory
// write of the call's epoch into the chunk's readiness flag, which the persistent GEMM
// polls. On GB300 the driver runs such a same-device copy as a kernel on SMs, not on a
// copy engine; the GEMM kernels therefore leave each SM room for a copy CTA (see the
// register cap of the pair kernel), and every flag wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <new>
#include <vector>

#include "ub_internal.h"

using ubk::GemmParams;

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(UB_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define UB_CUDA(call)                                   \
    do {                                                \
        cudaError_t e_ = (call);                        \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
    } while (0)

// ---------------------------------------------------------------- driver entry points

typedef CUresult (*PFN_encodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                    const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*PFN_writeValue32)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

struct DriverFns {
    PFN_encodeTiled encode = nullptr;
    PFN_writeValue32 write_value32 = nullptr;
    int status = -1;  // -1 unresolved, 0 ok, else error
};

DriverFns &driver()
{
    static DriverFns fns;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q1, q2;
        void *f1 = nullptr, *f2 = nullptr;
        cudaError_t e1 = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f1, 12000, cudaEnableDefault, &q1);
        cudaError_t e2 = cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &f2, 12000, cudaEnableDefault, &q2);
        if (e1 == cudaSuccess && e2 == cudaSuccess && q1 == cudaDriverEntryPointSuccess &&
            q2 == cudaDriverEntryPointSuccess && f1 && f2) {
            fns.encode = reinterpret_cast<PFN_encodeTiled>(f1);
            fns.write_value32 = reinterpret_cast<PFN_writeValue32>(f2);
            fns.status = 0;
        } else {
            fns.status = 1;
        }
    });
    return fns;
}

// ---------------------------------------------------------------- tensor maps

// 2-D row-major bf16 tensor [outer, inner] with row pitch `pitch_bytes`, moved in boxes
// of [box_outer, box_inner] with the 128-byte swizzle (box_inner * 2 == 128).
int encode_2d(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t outer, uint64_t pitch_bytes,
              uint32_t box_inner, uint32_t box_outer)
{
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = driver().encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides,
                                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(UB_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%llu x %llu], pitch %llu", (int)r,
                    (unsigned long long)outer, (unsigned long long)inner, (unsigned long long)pitch_bytes);
    return UB_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Kernel parameters are cached by everything that determines them (mode, shape,
// pointers, ring start), so a repeated call encodes no tensor map.
struct CacheEntry {
    std::vector<const void *> key;
    GemmParams params;
    uint64_t last_use;
};

constexpr int kCacheEntries = 64;
constexpr int kMaxProfiled = 4096;

struct ProfileRing {
    std::vector<cudaEvent_t> start, stop;
    int count = 0;
};

}  // namespace

struct ub_handle {
    int device = 0;
    int sm_count = 0;
    int64_t max_tokens = 0, hidden = 0;
    int tp = 1;
    int64_t T = 0;  // active tokens
    void *ub = nullptr;      // [max_tokens, hidden] bf16
    uint32_t *ctrl = nullptr;  // flags[UB_MAX_TP] | abort | status | ... | partial-tile flags (from word 64)
    size_t ctrl_bytes = 0;
    float *ws = nullptr;       // partial tiles of split work: ws_slots x PARTIAL_FLOATS fp32
    int ws_slots = 0;          // 2 per SM: pair kernel (pair, rank) slots, skinny-kernel pieces
    int max_pairs = 0;         // pairs the workspace has room for
    cudaStream_t side = nullptr;                  // copy stream 0; also status reads
    cudaStream_t extra_side[UB_MAX_TP] = {};      // copy streams 1.. (created on demand)
    cudaEvent_t ev_join_extra[UB_MAX_TP] = {};
    int64_t copy_streams = 1;  // raised to min(tp, 4) at creation
    int64_t gather_kernel = -1; // 0: driver copies; 1: one kernel launch; 2: inside the GEMM; -1: by T
    bool gather_by_kernel = false;  // what the last issue_gather chose (join_gather follows it)
    bool gather_chained = false;    // ... and whether its kernel went on the call's own stream
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    uint32_t epoch = 0;
    // options
    int64_t sm_margin = 0;
    int64_t timeout_ns = 1000000000;
    int64_t self_rank = 0;
    int64_t drop_flag = -1;
    int64_t profile = 0;
    int64_t cta_pair = -1;  // -1 = chosen per call
    int64_t streamk = -1;   // -1 = chosen per call
    int64_t skinny = -1;    // -1 = whenever the few-token kernel is usable
    int64_t pdl = 1;        // programmatic dependent launch of every kernel
    int64_t bulk_beside = 0; // 1: ub_allgather / ub_reduce_scatter beside the kernel before them
    int64_t gather_chain = 1; // 1: the gather kernel on the call's stream, the GEMM its dependent
    int pair_clusters[3] = {-1, -1, -1};  // resident clusters of the pair kernel, per mode
    ub_counters_t counters{};
    std::vector<CacheEntry> cache;
    uint64_t use_clock = 0;
    ProfileRing prof[UB_NUM_OPS];
};

namespace {

// Control block, in 32-bit words: the readiness flags [0, UB_MAX_TP), the partial-tile
// flags [UB_MAX_TP, UB_MAX_TP + W) with W = ws_slots * EPI_WARPS, then the abort word, the
// status word and the gather's per-chunk counters (zero between calls). The words a
// captured call clears (flags and partial-tile flags) are one contiguous run.
size_t ws_flag_words(const ub_handle *h) { return static_cast<size_t>(h->ws_slots) * ubk::EPI_WARPS; }
uint32_t *flags_of(ub_handle *h) { return h->ctrl; }
uint32_t *ws_flags_of(ub_handle *h) { return h->ctrl + UB_MAX_TP; }
uint32_t *abort_of(ub_handle *h) { return h->ctrl + UB_MAX_TP + ws_flag_words(h); }
int32_t *status_of(ub_handle *h) { return reinterpret_cast<int32_t *>(abort_of(h) + 1); }
uint32_t *gather_counters_of(ub_handle *h) { return abort_of(h) + 8; }  // UB_MAX_TP words

// Makes the handle's device current for the duration of a call.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            return;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard()
    {
        if (ok && prev >= 0) cudaSetDevice(prev);
    }
};

int grid_for(ub_handle *h, int num_tiles)
{
    int g = h->sm_count - static_cast<int>(h->sm_margin);
    if (g < 1) g = 1;
    return g < num_tiles ? g : num_tiles;
}

// Clusters of the pair kernel to launch: as many as fit (resident at once, within the
// SM margin), but no more than there are pair tiles.
int clusters_for(ub_handle *h, int mode, int num_tiles)
{
    if (h->pair_clusters[mode] < 0) h->pair_clusters[mode] = ubk::max_pair_clusters(mode);
    int g = (h->sm_count - static_cast<int>(h->sm_margin)) / 2;
    if (h->pair_clusters[mode] > 0 && g > h->pair_clusters[mode]) g = h->pair_clusters[mode];
    if (g > h->max_pairs) g = h->max_pairs;
    if (g < 1) g = 1;
    return g < num_tiles ? g : num_tiles;
}

GemmParams *cache_lookup(ub_handle *h, const std::vector<const void *> &key)
{
    for (auto &e : h->cache)
        if (e.key == key) {
            e.last_use = ++h->use_clock;
            return &e.params;
        }
    return nullptr;
}

GemmParams *cache_insert(ub_handle *h, std::vector<const void *> key, const GemmParams &p)
{
    if (static_cast<int>(h->cache.size()) < kCacheEntries) {
        h->cache.push_back(CacheEntry{std::move(key), p, ++h->use_clock});
        return &h->cache.back().params;
    }
    size_t victim = 0;
    for (size_t i = 1; i < h->cache.size(); ++i)
        if (h->cache[i].last_use < h->cache[victim].last_use) victim = i;
    h->cache[victim] = CacheEntry{std::move(key), p, ++h->use_clock};
    return &h->cache[victim].params;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Row regions of the CTA-pair AG tiling, in ring order: the self chunk's first `head`
// rows, read in place from its shard; the user-buffer rows from there to T (the rest of
// the self chunk first, behind its readiness flag like the other chunks' rows); the
// user-buffer rows before the self chunk. With head = c the self chunk is read wholly
// in place; with head = its whole 256-row tiles only the second region ends in a partial
// tile (self rank 0: ceil(T / 256) row tiles, one fewer whenever 256 does not divide c).
struct AgRegion {
    int64_t row0, rows;
    const void *src;
    int ub_backed;
};
int ag_pair_regions(int64_t T, int64_t c, int64_t H, int self, int64_t head, const void *self_shard, char *ub,
                    AgRegion out[3])
{
    const int64_t row1 = self * c + head;
    const AgRegion all[3] = {{self * c, head, self_shard, 0},
                             {row1, T - row1, ub + row1 * H * 2, 1},
                             {0, self * c, ub, 1}};
    int n = 0;
    for (const AgRegion &r : all)
        if (r.rows > 0) out[n++] = r;
    return n;
}

int64_t ag_pair_row_tiles(int64_t T, int64_t c, int self, int64_t head)
{
    AgRegion reg[3];
    const int n = ag_pair_regions(T, c, 0, self, head, nullptr, nullptr, reg);
    int64_t tiles = 0;
    for (int i = 0; i < n; ++i) tiles += ceil_div(reg[i].rows, ubk::PAIR_BM);
    return tiles;
}

// How many of the self chunk's rows the CTA-pair AG kernel reads in place: all of them,
// unless reading only its whole 256-row tiles in place saves a wave of pairs. The rest
// then waits for the gather, which copies those rows first (measured on GB300: AG +
// SwiGLU at T = 1140 in two waves instead of three, 59 against 83 us; QKV at T = 1140,
// one wave either way, 39.4 against 36.0 us had it always been done).
int64_t self_head_for(int64_t T, int64_t c, int self, int64_t n_tiles, int64_t np)
{
    const int64_t split = c / ubk::PAIR_BM * ubk::PAIR_BM;
    if (split == c) return c;
    const int64_t waves_split = ceil_div(ag_pair_row_tiles(T, c, self, split) * n_tiles, np);
    const int64_t waves_whole = ceil_div(ag_pair_row_tiles(T, c, self, c) * n_tiles, np);
    return waves_split < waves_whole ? split : c;
}

int64_t ag_self_head(ub_handle *h, int mode, int64_t T, int64_t c, int self, int64_t n_tiles)
{
    return self_head_for(T, c, self, n_tiles, clusters_for(h, mode, 1 << 30));
}

// GEMM-RS on CTA pairs: tile rows walked in groups of kGroupM (rows fastest inside a
// group) when the weights exceed this many bytes, else N fastest.
constexpr int64_t kGroupedOrderBytes = int64_t(256) << 20;
constexpr int kGroupM = 8;

// AG-GEMM on CTA pairs: tile rows walked in groups of kGroupM (rows fastest inside a
// group), so that a wave reads each weight panel about once per group instead of once
// per wave (walked N fastest, fc1 at T = 8192 streams all 58.7 MB of W1 in every wave).
// That holds when the first wave reads only the self chunk's in-place rows
// (`head_tiles` >= the pairs): later waves start after the gather has moved on. Else
// the first wave reaches gathered rows, and a group of more tile rows than a chunk holds
// would start tiles of chunks late in the ring: there the group is one chunk's tile rows
// (none below two). Measured on GB300: fc1 AG + SwiGLU at T = 8192 269.4 against 275.6
// us, the benchmark step 1.1 % faster; groups of 8 at T = 2048 (first wave 56 self-chunk
// tiles and 20 gathered), which start tiles of all four chunks at once, 97.4 against
// 91.2 us.
int ag_group_m(int64_t c, int64_t head_tiles, int64_t pairs)
{
    if (head_tiles >= pairs) return kGroupM;
    const int64_t g = c / ubk::PAIR_BM;
    return g >= 2 ? static_cast<int>(g < kGroupM ? g : kGroupM) : 0;
}

constexpr int64_t kGatherKernelMaxT = 512;  // UB_OPT_GATHER_KERNEL = -1: kernel up to this T
// ... and inside the GEMM above it when the call has more than one wave of tiles: on
// GB300 (tp 4, hidden 4096) the whole AG call is 2-8 % faster than with the driver copies
// at T = 1024-8192 (the chunks land sooner: no copy launches, every SM copying; AG
// T = 2048: 73.2 vs 78.6 us). A call whose tiles fit one wave leaves SMs without a tile,
// and there the gather kernel, whose CTAs run on them, lands the chunks sooner than the
// GEMM's own epilogue warps: QKV (N = 3072) at T = 576-1536 37.0-41.5 against 39.4-45.6 us,
// tp 8 / hidden 8192 at T = 576-1024 55.8-61.9 against 60.2-64.5; with more than one wave
// the GEMM's warps win (QKV T = 2048: 51.7 against 61.6 us).
constexpr bool kFusedGatherAuto = true;
// Not for the few-token kernel: there the chunks are tiny, the weight stream hides the
// one-launch gather, and the gather inside the kernel (each chunk by its own few CTAs)
// measured 2-5 us slower per call (AG, AG + SwiGLU and QKV at T = 4-128, GB300).
constexpr bool kFusedGatherSkinnyAuto = false;

// Cost of the last, partial wave's tiles when each is cut into s k-pieces, in units of
// one whole tile on one pair: the longest piece, 1/s, plus the fix-up (each piece
// publishes its fp32 partial of the columns it does not own and adds the others' partials
// of its own). The fix-up is a fixed time rather than a share of the tile, fitted on
// GB300 in k-blocks of a 256 x 256 pair tile (0.34 us each) by running the same shapes
// whole and split in 2..8 pieces (bench.py --case ... --streamk 0 | n):
//  - GEMM-RS: kFixupKb0 + kFixupKb1 * (s - 1), about 10 us + 4.6 us per added piece; a
//    split pays off for its long K (tp shards of K = 1024 .. 3584: 2-27 % faster).
//  - AG-GEMM behind the gather (`gathered`): kFixupAgKb0 + kFixupAgKb1 * (s - 1), about
//    3.4 us + 2.6 us per added piece (K = 4096: QKV at T = 5120 90.5 us in 4 pieces against
//    96.1 whole, AG + SwiGLU at T = 3072 119.3 in 2 against 124.0). Its tail tiles are the
//    last rows of the gather, so with one whole wave before them they wait for the
//    gather whatever their length, and a split only adds its fix-up (QKV at T = 2048, one
//    whole wave: 55.8 us in 2 pieces, 62.0 in 3, against 53.8 whole). With no whole wave
//    (fewer tiles than pairs) every tile is in the split and spreads over idle pairs: QKV
//    at T = 256 31.7 us in 3 pieces against 34.5 whole, at T = 512 33.3 in 2 against 35.0.
constexpr double kFixupKb0 = 30.0;
constexpr double kFixupKb1 = 13.5;
constexpr double kFixupAgKb0 = 10.0;
constexpr double kFixupAgKb1 = 7.5;
constexpr int64_t kMinWavesAg = 2;
double split_tail_cost(int64_t s, int64_t kb, bool gathered)
{
    if (s <= 1) return 1.0;
    const double f = gathered ? kFixupAgKb0 + kFixupAgKb1 * static_cast<double>(s - 1)
                              : kFixupKb0 + kFixupKb1 * static_cast<double>(s - 1);
    return 1.0 / static_cast<double>(s) + f / static_cast<double>(kb);
}

// How many k-pieces the last wave's tiles are cut into. At most one piece per idle pair,
// MAX_TAIL_SPLIT pieces and MIN_KBLOCKS_PER_PIECE k-blocks per piece; within that the
// cheapest cut by split_tail_cost (1 when no cut beats whole tiles, or for a gathered
// AG-GEMM with at least one but fewer than kMinWavesAg whole waves), or with `force` = 1
// the most pieces
// allowed (the split forced on), with `force` = n >= 2 at most n pieces.
int64_t tail_split_for(int64_t tiles, int64_t np, int64_t kb, int64_t force, bool gathered)
{
    const int64_t rem = tiles % np;
    if (rem == 0) return 1;
    int64_t smax = np / rem;
    if (smax > ubk::MAX_TAIL_SPLIT) smax = ubk::MAX_TAIL_SPLIT;
    if (smax > kb / ubk::MIN_KBLOCKS_PER_PIECE) smax = kb / ubk::MIN_KBLOCKS_PER_PIECE;
    if (smax < 1) return 1;
    if (force == 1) return smax;
    if (force >= 2) return force < smax ? force : smax;
    if (gathered && tiles >= np && tiles / np < kMinWavesAg) return 1;
    int64_t best = 1;
    for (int64_t s = 2; s <= smax; ++s)
        if (split_tail_cost(s, kb, gathered) < split_tail_cost(best, kb, gathered)) best = s;
    return best;
}

// Launch shape of a pair-kernel call: whole tiles in strided waves, and (with the
// split on) the last, partial wave's tiles cut into k-pieces over the idle pairs. With
// `every_pair` (the gather runs inside the GEMM) every pair is launched even when there
// are fewer tiles, so that every SM copies its share of the gather.
void set_pairs(ub_handle *h, GemmParams &p, int mode, bool split, bool every_pair = false, bool gathered = false)
{
    const int64_t tiles = p.region_tile0[p.n_regions];
    int64_t np = clusters_for(h, mode, 1 << 30);
    int64_t sp = split ? tail_split_for(tiles, np, p.k_blocks, h->streamk > 0 ? h->streamk : 0, gathered) : 1;
    if (sp == 1 && np > tiles && !every_pair) np = tiles;
    if (np < 1) np = 1;
    p.num_pairs = static_cast<int>(np);
    p.dp_tiles = static_cast<int>((tiles / np) * np);
    p.tail_split = static_cast<int>(sp);
    if (p.dp_tiles == tiles) p.tail_split = 1;
    p.ws = h->ws;
    p.ws_flags = ws_flags_of(h);
}

// The few-token kernel runs a call when its token tile (`cols` TMEM columns) fits one
// accumulator and neither it nor the CTA-pair choice is forced the other way. Chosen
// automatically up to SK_AUTO_MAX_COLS columns: measured on GB300 (fc1 / fc2 of the
// SwiGLU MLP, hidden 4096, tp 4) it beats the tile kernels up to T = 128 and loses at
// T = 256, where the work is no longer bound by the weight read.
bool use_skinny(ub_handle *h, int64_t cols)
{
    if (cols > ubk::SK_MAX_COLS || h->skinny == 0) return false;
    if (h->skinny == 1) return true;
    return h->cta_pair < 0 && cols <= ubk::SK_AUTO_MAX_COLS;
}

// Launch shape of a skinny-kernel call: k-pieces per weight tile so that about one unit
// runs per SM (each piece at least SK_MIN_KBLOCKS long, the partials within the
// workspace), and the deepest pipeline that fits in shared memory.
void set_skinny(ub_handle *h, GemmParams &p, int slot_mult, int w_bytes)
{
    const int64_t slots = h->sm_count - h->sm_margin > 0 ? h->sm_count - h->sm_margin : 1;
    int64_t s = slots / p.n_tiles;
    if (s > ubk::SK_MAX_SPLIT) s = ubk::SK_MAX_SPLIT;
    if (s > p.k_blocks / ubk::SK_MIN_KBLOCKS) s = p.k_blocks / ubk::SK_MIN_KBLOCKS;
    const int64_t ws_cap = h->ws_slots / (static_cast<int64_t>(p.n_tiles) * slot_mult);  // every piece publishes
    if (s > ws_cap) s = ws_cap;
    if (s < 1) s = 1;
    p.sk_split = static_cast<int>(s);
    p.sk_units = p.n_tiles * p.sk_split;
    // split pieces run one unit per CTA (the finisher reuses its stage buffers): all
    // units fit in one wave of the grid the launch uses (grid_for: slots CTAs at most)
    const int x_bytes = p.sk_n_sub * p.sk_sub_n * 128;
    int st = (ubk::SK_SMEM_LIMIT - ubk::skinny_smem_bytes(0, w_bytes, x_bytes)) / (w_bytes + x_bytes);
    if (st > ubk::SK_MAX_STAGES) st = ubk::SK_MAX_STAGES;
    p.sk_stages = st < 1 ? 1 : st;
    int stride = 16;
    while (stride < p.sk_n_sub * p.sk_sub_n) stride *= 2;
    p.sk_stride = stride;
    p.ws = h->ws;
    p.ws_flags = ws_flags_of(h);
}

// Which kernel runs a call, from a wave-count cost model measured on GB300 (one unit =
// the time of one 128x256 tile on one SM, the same as one 256x256 tile on a pair):
//   single CTAs, chunk-aligned 128-row tiles:    waves
//   CTA pairs, whole tiles:                      0.91 * waves (a third less L2 traffic)
//   CTA pairs, last wave split into s k-pieces:  0.91 * (full waves + split_tail_cost(s))
// UB_OPT_CTA_PAIR / UB_OPT_STREAMK >= 0 force a choice. The choice depends only on the
// shapes and the SM count, so results stay bitwise reproducible.
void plan_path(int64_t slots, int64_t np, int cta_pair, int streamk, int64_t single_tiles, int64_t pair_tiles,
               int64_t kb, bool gathered, bool &pair, bool &split)
{
    const double c_single = static_cast<double>(ceil_div(single_tiles, slots));
    const double c_dp = 0.91 * static_cast<double>(ceil_div(pair_tiles, np));
    const int64_t s = tail_split_for(pair_tiles, np, kb, streamk > 0 ? streamk : 0, gathered);
    const double c_split =
        s > 1 ? 0.91 * (static_cast<double>(pair_tiles / np) + split_tail_cost(s, kb, gathered)) : c_dp;
    if (cta_pair == 0) {
        pair = false;
    } else if (cta_pair == 1) {
        pair = true;
    } else {
        pair = (c_dp < c_single) || (c_split < c_single);
    }
    if (!pair) {
        split = false;
    } else if (streamk >= 0) {
        split = streamk != 0;
    } else {
        split = c_split < c_dp;
    }
}

void choose_path(ub_handle *h, int mode, int64_t single_tiles, int64_t pair_tiles, int64_t kb, bool gathered,
                 bool &pair, bool &split)
{
    const int64_t slots = h->sm_count - h->sm_margin > 0 ? h->sm_count - h->sm_margin : 1;
    plan_path(slots, clusters_for(h, mode, 1 << 30), static_cast<int>(h->cta_pair), static_cast<int>(h->streamk),
              single_tiles, pair_tiles, kb, gathered, pair, split);
}

enum Path : int { PATH_SINGLE = 0, PATH_PAIR = 1, PATH_SKINNY = 2 };

int launch(ub_handle *h, GemmParams &p, int mode, int path, cudaStream_t s, int prof_op)
{
    p.pdl = static_cast<int>(h->pdl);
    // single CTAs: one per tile, or one per SM when the gather runs inside the GEMM
    const int grid = path == PATH_PAIR ? p.num_pairs
                                       : grid_for(h, path == PATH_SKINNY ? p.sk_units
                                                                         : (p.fused_gather ? 1 << 30 : p.num_tiles));
    if (path == PATH_SKINNY && p.sk_split > 1 && grid < p.sk_units)
        return fail(UB_ERR_ARG, "skinny launch: %d split units on %d CTAs", p.sk_units, grid);
    ProfileRing &ring = h->prof[prof_op];
    const bool timed = h->profile != 0 && ring.count < kMaxProfiled;
    if (timed) {
        if (static_cast<int>(ring.start.size()) <= ring.count) {
            cudaEvent_t a, b;
            UB_CUDA(cudaEventCreate(&a));
            UB_CUDA(cudaEventCreate(&b));
            ring.start.push_back(a);
            ring.stop.push_back(b);
        }
        UB_CUDA(cudaEventRecord(ring.start[ring.count], s));
    }
    cudaError_t e = path == PATH_PAIR     ? ubk::launch_gemm_pair(p, mode, grid, s)
                    : path == PATH_SKINNY ? ubk::launch_gemm_skinny(p, mode, grid, s)
                                          : ubk::launch_gemm(p, mode, grid, s);
    if (e != cudaSuccess) return cuda_fail(e, "GEMM kernel launch");
    h->counters.last_kernel = path == PATH_PAIR ? UB_KERNEL_PAIR : path == PATH_SKINNY ? UB_KERNEL_FEW_TOKEN : UB_KERNEL_SINGLE;
    h->counters.last_pieces = path == PATH_PAIR ? p.tail_split : path == PATH_SKINNY ? p.sk_split : 1;
    h->counters.last_gather = -1;  // an AG call sets it after the launch
    if (timed) {
        UB_CUDA(cudaEventRecord(ring.stop[ring.count], s));
        ++ring.count;
    }
    return UB_OK;
}


// The all-gather of the chunks into the user buffer: device-to-device copies dealt over
// the copy streams in ring order after the self rank (the self chunk last), each
// followed by a stream memory write of `epoch` into the chunk's readiness flag (skipped
// for chunk `drop`, a host-side fault injection). The copy streams first wait for the
// work already queued on `s`.
// Whether this AG call's gather runs inside the GEMM kernel (its epilogue warps copy the
// chunks before their first tile): UB_OPT_GATHER_KERNEL = 2, or the automatic choice.
bool gather_in_gemm(ub_handle *h, bool skinny, bool one_wave)
{
    if (h->gather_kernel == 2) return true;
    if (h->gather_kernel >= 0) return false;
    return skinny ? kFusedGatherSkinnyAuto : (kFusedGatherAuto && h->T > kGatherKernelMaxT && !one_wave);
}

// The copies of the all-gather in issue order: the self chunk's rows from `head` on (the
// rows the GEMM reads from the buffer; flag after them), the other chunks in ring order
// (flag after each), then the self chunk's first `head` rows (read in place by the GEMM;
// flagged only when they are the whole chunk).
struct GatherPart {
    int r;
    int64_t row_lo, row_hi;
    bool flag;
};
int gather_parts(int tp, int self, int64_t c, int64_t head, GatherPart out[UB_MAX_TP + 1])
{
    int n = 0;
    if (head < c) out[n++] = GatherPart{self, head, c, true};
    for (int q = 1; q < tp; ++q) out[n++] = GatherPart{(self + q) % tp, 0, c, true};
    if (head > 0) out[n++] = GatherPart{self, 0, head, head == c};
    return n;
}

// The gather kernel's launch parameters for the handle's active shape: about one CTA
// per SM in all (ceil(SMs / tp) per chunk, fewer for small chunks), ring order from the
// self rank, each chunk's flag published at `epoch` unless it is `drop`.
ubk::GatherParams gather_kernel_params(ub_handle *h, const void *const *shards, uint32_t epoch, int64_t drop)
{
    const int tp = h->tp;
    ubk::GatherParams g;
    memset(&g, 0, sizeof g);
    for (int r = 0; r < tp; ++r) g.src[r] = shards[r];
    g.ub = h->ub;
    g.flags = flags_of(h);
    g.counters = gather_counters_of(h);
    g.epoch = epoch;
    g.tp = tp;
    g.self_rank = static_cast<int>(h->self_rank);
    g.drop = static_cast<int>(drop);
    g.chunk_vecs = (h->T / tp) * h->hidden / 8;
    int64_t per = (h->sm_count + tp - 1) / tp;
    const int64_t need = (g.chunk_vecs + 511) / 512;  // at least two vectors per thread
    if (per > need) per = need;
    g.ctas_per_chunk = static_cast<int>(per < 1 ? 1 : per);
    g.pdl = static_cast<int>(h->pdl);
    return g;
}

int issue_gather(ub_handle *h, const void *const *shards, cudaStream_t s, uint32_t epoch, int64_t drop,
                 int64_t self_head, bool one_wave = false)
{
    const int tp = h->tp;
    const int64_t T = h->T, H = h->hidden, c = T / tp;
    const int self = static_cast<int>(h->self_rank);
    char *ub = static_cast<char *>(h->ub);
    // The one-launch gather kernel replaces tp copies and tp flag writes, each a driver
    // operation with its own host cost and launch latency; for few tokens those dominate
    // the call (GB300, tp 4: AG at T <= 512 takes 26-33 us with the kernel, 39-44 us with
    // the copies), while for many tokens the copies are as fast or faster.
    h->gather_by_kernel = h->gather_kernel == 1 || h->gather_kernel == 2 ||
                          (h->gather_kernel < 0 && (T <= kGatherKernelMaxT || one_wave));
    if (h->copy_streams == 0 && !h->gather_by_kernel) {
        // In-stream: the copies and flag writes go on `s` itself, ahead of the GEMM,
        // which then finds every flag set (no overlap, no cross-stream hops).
        GatherPart parts[UB_MAX_TP + 1];
        const int np = gather_parts(tp, self, c, self_head, parts);
        for (int i = 0; i < np; ++i) {
            const GatherPart &pt = parts[i];
            const int r = pt.r;
            UB_CUDA(cudaMemcpyAsync(ub + (r * c + pt.row_lo) * H * 2,
                                    static_cast<const char *>(shards[r]) + pt.row_lo * H * 2,
                                    static_cast<size_t>((pt.row_hi - pt.row_lo) * H * 2), cudaMemcpyDeviceToDevice, s));
            if (pt.flag && r != drop) {
                CUresult cr = driver().write_value32(reinterpret_cast<CUstream>(s),
                                                     reinterpret_cast<CUdeviceptr>(flags_of(h) + r), epoch,
                                                     CU_STREAM_WRITE_VALUE_DEFAULT);
                if (cr != CUDA_SUCCESS) return fail(UB_ERR_CUDA, "cuStreamWriteValue32 failed (%d)", (int)cr);
            }
        }
        return UB_OK;
    }
    h->gather_chained = false;
    if (h->gather_by_kernel) {
        // One launch: small CTAs (they fit beside the GEMM's), about one per SM per chunk,
        // each chunk's flag published by its last CTA.
        ubk::GatherParams g = gather_kernel_params(h, shards, epoch, drop);
        if (h->gather_chain && h->pdl) {
            // On the call's own stream: the kernel waits for the work before it, then lets
            // the next launch, so a GEMM launched next as its programmatic dependent starts
            // once every gather CTA holds its SM (the flags it waits on are then certain to
            // come) and finds every grid before the gather complete.
            cudaError_t e = ubk::launch_gather(g, s);
            if (e != cudaSuccess) return cuda_fail(e, "gather kernel launch");
            h->gather_chained = true;
            return UB_OK;
        }
        // On the side stream, forked from and joined back into the call's stream.
        UB_CUDA(cudaEventRecord(h->ev_fork, s));
        UB_CUDA(cudaStreamWaitEvent(h->side, h->ev_fork, 0));
        cudaError_t e = ubk::launch_gather(g, h->side);
        if (e != cudaSuccess) return cuda_fail(e, "gather kernel launch");
        return UB_OK;
    }
    const int ncs = static_cast<int>(h->copy_streams < tp ? h->copy_streams : tp);
    auto copy_stream = [&](int i) { return i == 0 ? h->side : h->extra_side[i]; };
    UB_CUDA(cudaEventRecord(h->ev_fork, s));
    for (int i = 0; i < ncs; ++i) UB_CUDA(cudaStreamWaitEvent(copy_stream(i), h->ev_fork, 0));
    GatherPart parts[UB_MAX_TP + 1];
    const int np = gather_parts(tp, self, c, self_head, parts);
    for (int i = 0; i < np; ++i) {
        const GatherPart &pt = parts[i];
        const int r = pt.r;
        cudaStream_t cs = copy_stream(i % ncs);
        UB_CUDA(cudaMemcpyAsync(ub + (r * c + pt.row_lo) * H * 2,
                                static_cast<const char *>(shards[r]) + pt.row_lo * H * 2,
                                static_cast<size_t>((pt.row_hi - pt.row_lo) * H * 2), cudaMemcpyDeviceToDevice, cs));
        if (pt.flag && r != drop) {
            CUresult cr = driver().write_value32(reinterpret_cast<CUstream>(cs),
                                                 reinterpret_cast<CUdeviceptr>(flags_of(h) + r), epoch,
                                                 CU_STREAM_WRITE_VALUE_DEFAULT);
            if (cr != CUDA_SUCCESS) return fail(UB_ERR_CUDA, "cuStreamWriteValue32 failed (%d)", (int)cr);
        }
    }
    return UB_OK;
}

// Make `s` wait for every copy stream the last gather used.
int join_gather(ub_handle *h, cudaStream_t s)
{
    if (h->copy_streams == 0 && !h->gather_by_kernel) return UB_OK;  // in-stream: nothing to join
    if (h->gather_chained) return UB_OK;  // the gather kernel ran on the call's stream
    const int ncs = h->gather_by_kernel ? 1 : static_cast<int>(h->copy_streams < h->tp ? h->copy_streams : h->tp);
    UB_CUDA(cudaEventRecord(h->ev_join, h->side));
    UB_CUDA(cudaStreamWaitEvent(s, h->ev_join, 0));
    for (int i = 1; i < ncs; ++i) {
        UB_CUDA(cudaEventRecord(h->ev_join_extra[i], h->extra_side[i]));
        UB_CUDA(cudaStreamWaitEvent(s, h->ev_join_extra[i], 0));
    }
    return UB_OK;
}

// A new call's epoch, unique per handle: every wait compares a flag for equality with
// it, so words left by other calls never match. When `s` is being captured into a CUDA
// graph the epoch becomes a constant of the graph, so every replay would find the words
// it waits on still holding it from the replay before. The captured call therefore
// starts, in stream order, by clearing the ones it uses -- the readiness flags (`gathered`:
// the call waits for chunk flags) and the partial-tile flags (`split`: tiles cut into
// k-pieces) -- in one memset of the contiguous run that covers them; a call that uses
// neither clears nothing. The abort word, which a timeout sets to the call's epoch, is
// cleared by ub_clear_status. An uncaptured call pays nothing.
int begin_call(ub_handle *h, cudaStream_t s, uint32_t &epoch, bool gathered, bool split)
{
    epoch = ++h->epoch;
    if (epoch == 0) epoch = ++h->epoch;  // 0 is what a cleared word holds
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    UB_CUDA(cudaStreamIsCapturing(s, &cs));
    if (cs == cudaStreamCaptureStatusActive && (gathered || split)) {
        const size_t lo = gathered ? 0 : UB_MAX_TP;
        const size_t hi = split ? UB_MAX_TP + ws_flag_words(h) : static_cast<size_t>(h->tp);
        UB_CUDA(cudaMemsetAsync(h->ctrl + lo, 0, (hi - lo) * sizeof(uint32_t), s));
    }
    return UB_OK;
}

// An NVTX range around one ABI call, named with the call and its active T, so that a
// timeline shows which GPU work each call issued and what of it stays exposed. Without
// an attached tool the push and pop cost a few nanoseconds.
struct NvtxRange {
    NvtxRange(const char *name, int64_t T)
    {
        char msg[64];
        snprintf(msg, sizeof msg, "%s T=%lld", name, static_cast<long long>(T));
        nvtxRangePushA(msg);
    }
    ~NvtxRange() { nvtxRangePop(); }
};

int check_handle(ub_handle *h)
{
    if (!h) return fail(UB_ERR_ARG, "null handle");
    return UB_OK;
}

}  // namespace

void ubk::set_last_error(const char *msg) { snprintf(g_err, sizeof g_err, "%s", msg); }

extern "C" {

const char *ub_last_error(void) { return g_err; }

int ub_validate_active_shape(int ndim, const int64_t *dims, int64_t max_tokens, int64_t hidden, int tp)
{
    if (ndim != 2) return fail(UB_ERR_RANK, "active shape must be two-dimensional, got %d dims", ndim);
    if (!dims) return fail(UB_ERR_ARG, "null shape");
    if (dims[0] <= 0 || dims[1] <= 0)
        return fail(UB_ERR_ZERO, "active shape [%lld, %lld] has a zero extent", (long long)dims[0],
                    (long long)dims[1]);
    if (dims[0] > max_tokens)
        return fail(UB_ERR_CAPACITY, "active tokens %lld exceed the registered capacity %lld", (long long)dims[0],
                    (long long)max_tokens);
    if (dims[1] != hidden)
        return fail(UB_ERR_HIDDEN, "hidden %lld differs from the registered hidden %lld", (long long)dims[1],
                    (long long)hidden);
    if (tp < 1 || dims[0] % tp != 0)
        return fail(UB_ERR_DIVISIBLE, "active tokens %lld not divisible by tp %d", (long long)dims[0], tp);
    return UB_OK;
}

int ub_create(int64_t max_tokens, int64_t hidden, int tp, ub_dtype_t dtype, ub_handle_t *out)
{
    if (!out) return fail(UB_ERR_ARG, "null output handle pointer");
    *out = nullptr;
    if (tp < 1 || tp > UB_MAX_TP) return fail(UB_ERR_ARG, "tp %d outside [1, %d]", tp, UB_MAX_TP);
    if (max_tokens <= 0 || hidden <= 0)
        return fail(UB_ERR_ZERO, "capacity [%lld, %lld] has a zero extent", (long long)max_tokens, (long long)hidden);
    if (dtype != UB_BF16) return fail(UB_ERR_DTYPE, "only UB_BF16 user buffers are supported");
    if (hidden % 8 != 0) return fail(UB_ERR_ALIGN, "hidden %lld is not a multiple of 8", (long long)hidden);
    if (max_tokens % tp != 0)
        return fail(UB_ERR_DIVISIBLE, "max_tokens %lld not divisible by tp %d", (long long)max_tokens, tp);
    if (max_tokens > (int64_t(1) << 31) - 1 || hidden > (int64_t(1) << 24))
        return fail(UB_ERR_ARG, "capacity [%lld, %lld] too large", (long long)max_tokens, (long long)hidden);

    int dev = 0;
    UB_CUDA(cudaGetDevice(&dev));
    if (driver().status != 0)
        return fail(UB_ERR_CUDA, "driver entry points cuTensorMapEncodeTiled / cuStreamWriteValue32 unavailable");
    ub_handle *h = new (std::nothrow) ub_handle();
    if (!h) return fail(UB_ERR_ARG, "out of host memory");
    h->device = dev;
    h->max_tokens = max_tokens;
    h->hidden = hidden;
    h->tp = tp;
    h->T = max_tokens;
    auto cleanup = [&](int code) {
        ub_destroy(h);
        return code;
    };
    cudaError_t e = cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cleanup(cuda_fail(e, "cudaDeviceGetAttribute"));
    e = cudaMalloc(&h->ub, static_cast<size_t>(max_tokens) * hidden * 2);
    if (e != cudaSuccess) return cleanup(cuda_fail(e, "cudaMalloc(user buffer)"));
    ++h->counters.device_allocations;
    h->max_pairs = h->sm_count / 2 > 0 ? h->sm_count / 2 : 1;
    h->ws_slots = 2 * (h->sm_count > 0 ? h->sm_count : 1);
    h->ctrl_bytes = (UB_MAX_TP + ws_flag_words(h) + 8 + UB_MAX_TP) * sizeof(uint32_t);
    e = cudaMalloc(reinterpret_cast<void **>(&h->ctrl), h->ctrl_bytes);
    if (e != cudaSuccess) return cleanup(cuda_fail(e, "cudaMalloc(control block)"));
    ++h->counters.device_allocations;
    e = cudaMalloc(reinterpret_cast<void **>(&h->ws),
                   static_cast<size_t>(h->ws_slots) * ubk::PARTIAL_FLOATS * sizeof(float));
    if (e != cudaSuccess) return cleanup(cuda_fail(e, "cudaMalloc(split workspace)"));
    ++h->counters.device_allocations;
    e = cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cleanup(cuda_fail(e, "cudaStreamCreateWithFlags"));
    if (int rc = ub_set_option(h, UB_OPT_COPY_STREAMS, tp < 4 ? tp : 4)) return cleanup(rc);
    e = cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming);
    if (e != cudaSuccess) return cleanup(cuda_fail(e, "cudaEventCreateWithFlags"));
    e = cudaMemsetAsync(h->ctrl, 0, h->ctrl_bytes, h->side);
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->side);
    if (e != cudaSuccess) return cleanup(cuda_fail(e, "clearing the control block"));
    *out = h;
    return UB_OK;
}

int ub_destroy(ub_handle_t h)
{
    if (!h) return fail(UB_ERR_ARG, "null handle");
    DeviceGuard g(h->device);
    if (h->side) cudaStreamSynchronize(h->side);
    for (auto &ring : h->prof) {
        for (auto ev : ring.start) cudaEventDestroy(ev);
        for (auto ev : ring.stop) cudaEventDestroy(ev);
    }
    if (h->ev_fork) cudaEventDestroy(h->ev_fork);
    if (h->ev_join) cudaEventDestroy(h->ev_join);
    if (h->side) cudaStreamDestroy(h->side);
    for (int i = 0; i < UB_MAX_TP; ++i) {
        if (h->extra_side[i]) {
            cudaStreamSynchronize(h->extra_side[i]);
            cudaStreamDestroy(h->extra_side[i]);
        }
        if (h->ev_join_extra[i]) cudaEventDestroy(h->ev_join_extra[i]);
    }
    if (h->ctrl) cudaFree(h->ctrl);
    if (h->ws) cudaFree(h->ws);
    if (h->ub) cudaFree(h->ub);
    delete h;
    return UB_OK;
}

int ub_set_active_shape_nd(ub_handle_t h, int ndim, const int64_t *dims)
{
    if (int rc = check_handle(h)) return rc;
    int rc = ub_validate_active_shape(ndim, dims, h->max_tokens, h->hidden, h->tp);
    if (rc != UB_OK) return rc;
    h->T = dims[0];
    return UB_OK;
}

int ub_set_active_shape(ub_handle_t h, int64_t T, int64_t hidden)
{
    const int64_t dims[2] = {T, hidden};
    return ub_set_active_shape_nd(h, 2, dims);
}

int ub_get_active_shape(ub_handle_t h, int64_t *T, int64_t *hidden)
{
    if (int rc = check_handle(h)) return rc;
    if (T) *T = h->T;
    if (hidden) *hidden = h->hidden;
    return UB_OK;
}

int ub_get_capacity(ub_handle_t h, int64_t *max_tokens, int64_t *hidden)
{
    if (int rc = check_handle(h)) return rc;
    if (max_tokens) *max_tokens = h->max_tokens;
    if (hidden) *hidden = h->hidden;
    return UB_OK;
}

int ub_get_tp(ub_handle_t h, int *tp)
{
    if (int rc = check_handle(h)) return rc;
    if (tp) *tp = h->tp;
    return UB_OK;
}

int ub_buffer(ub_handle_t h, void **dev_ptr, size_t *bytes)
{
    if (int rc = check_handle(h)) return rc;
    if (dev_ptr) *dev_ptr = h->ub;
    if (bytes) *bytes = static_cast<size_t>(h->max_tokens) * h->hidden * 2;
    return UB_OK;
}

int ub_grid_ctas(ub_handle_t h, int *ctas)
{
    if (int rc = check_handle(h)) return rc;
    DeviceGuard g(h->device);
    if (ctas) *ctas = h->cta_pair != 0 ? 2 * clusters_for(h, ubk::MODE_RS, 1 << 30) : grid_for(h, 1 << 30);
    return UB_OK;
}

int64_t ub_plan_tail_split(int64_t tiles, int64_t pairs, int64_t k_blocks, int widest, int gathered)
{
    if (tiles < 1 || pairs < 1 || k_blocks < 1) return fail(UB_ERR_ARG, "ub_plan_tail_split: sizes must be >= 1");
    return tail_split_for(tiles, pairs, k_blocks, widest != 0 ? 1 : 0, gathered != 0);
}

int ub_plan_path(int64_t single_tiles, int64_t pair_tiles, int64_t k_blocks, int64_t slots, int64_t pairs,
                 int cta_pair, int streamk, int gathered, int *pair, int *split)
{
    if (single_tiles < 1 || pair_tiles < 1 || k_blocks < 1 || slots < 1 || pairs < 1 || !pair || !split)
        return fail(UB_ERR_ARG, "ub_plan_path: sizes must be >= 1 and outputs non-null");
    bool pr = false, sp = false;
    plan_path(slots, pairs, cta_pair, streamk, single_tiles, pair_tiles, k_blocks, gathered != 0, pr, sp);
    *pair = pr ? 1 : 0;
    *split = sp ? 1 : 0;
    return UB_OK;
}

int ub_plan_gather_parts(int tp, int self, int64_t c, int64_t head, int *chunk, int64_t *row_lo,
                         int64_t *row_hi, int *flag)
{
    if (tp < 1 || tp > UB_MAX_TP || self < 0 || self >= tp || c < 1 || head < 0 || head > c || !chunk ||
        !row_lo || !row_hi || !flag)
        return fail(UB_ERR_ARG, "ub_plan_gather_parts: invalid arguments");
    GatherPart parts[UB_MAX_TP + 1];
    const int n = gather_parts(tp, self, c, head, parts);
    for (int i = 0; i < n; ++i) {
        chunk[i] = parts[i].r;
        row_lo[i] = parts[i].row_lo;
        row_hi[i] = parts[i].row_hi;
        flag[i] = parts[i].flag ? 1 : 0;
    }
    return n;
}

int64_t ub_plan_ag_self_head(int64_t T, int tp, int self, int64_t n_tiles, int64_t pairs)
{
    if (tp < 1 || tp > UB_MAX_TP || T < tp || T % tp != 0 || self < 0 || self >= tp || n_tiles < 1 || pairs < 1)
        return fail(UB_ERR_ARG, "ub_plan_ag_self_head: invalid shape");
    return self_head_for(T, T / tp, self, n_tiles, pairs);
}

int ub_plan_ag_group_m(int64_t T, int tp, int self, int64_t n_tiles, int64_t pairs)
{
    if (tp < 1 || tp > UB_MAX_TP || T < tp || T % tp != 0 || self < 0 || self >= tp || n_tiles < 1 || pairs < 1)
        return fail(UB_ERR_ARG, "ub_plan_ag_group_m: invalid shape");
    const int64_t c = T / tp;
    return ag_group_m(c, ceil_div(self_head_for(T, c, self, n_tiles, pairs), ubk::PAIR_BM) * n_tiles, pairs);
}

// AG-GEMM, optionally with the SwiGLU epilogue (glu_f > 0: Wt is [2 * glu_f, hidden],
// gate rows first, and Y receives [T, glu_f]), or with the weight stored hidden x N
// (b_kn: the tensor core reads it MN-major).
static int ag_gemm_impl(ub_handle_t h, const void *const *shards, const void *Wt, int64_t N, void *Y, void *stream,
                        int64_t glu_f, bool b_kn)
{
    if (int rc = check_handle(h)) return rc;
    if (!shards || !Wt || !Y) return fail(UB_ERR_ARG, "ag_gemm: null pointer argument");
    if (N <= 0) return fail(UB_ERR_ZERO, "ag_gemm: N = %lld", (long long)N);
    if (N % 8 != 0) return fail(UB_ERR_ALIGN, "ag_gemm: N = %lld is not a multiple of 8", (long long)N);
    if (N > (int64_t(1) << 24)) return fail(UB_ERR_ARG, "ag_gemm: N = %lld too large", (long long)N);
    if (!aligned16(Wt) || !aligned16(Y)) return fail(UB_ERR_ALIGN, "ag_gemm: Wt / Y not 16-byte aligned");
    const int tp = h->tp;
    for (int r = 0; r < tp; ++r) {
        if (!shards[r]) return fail(UB_ERR_ARG, "ag_gemm: shard %d is null", r);
        if (!aligned16(shards[r])) return fail(UB_ERR_ALIGN, "ag_gemm: shard %d not 16-byte aligned", r);
    }
    DeviceGuard g(h->device);
    if (!g.ok) return fail(UB_ERR_CUDA, "ag_gemm: cannot select the handle's device");
    NvtxRange range(glu_f > 0 ? "ag_gemm_swiglu" : b_kn ? "ag_gemm_kn" : "ag_gemm", h->T);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t T = h->T, H = h->hidden, c = T / tp;
    const int self = static_cast<int>(h->self_rank);
    char *ub = static_cast<char *>(h->ub);

    const bool glu = glu_f > 0;
    const int mode = glu ? ubk::MODE_AG_GLU : ubk::MODE_AG;
    const int prof_op = glu ? UB_OP_AG_SWIGLU : (b_kn ? UB_OP_AG_KN : UB_OP_AG);
    const int64_t n_out = glu ? glu_f : N;                    // columns of Y
    const int64_t n_tiles = glu ? (glu_f + 127) / 128 : (N + ubk::BN - 1) / ubk::BN;
    const int64_t self_head = ag_self_head(h, mode, T, c, self, n_tiles);
    AgRegion regions[3];
    const int n_regions = ag_pair_regions(T, c, H, self, self_head, shards[self], ub, regions);
    int64_t pair_rows_tiles = 0;
    for (int i = 0; i < n_regions; ++i) pair_rows_tiles += ceil_div(regions[i].rows, ubk::PAIR_BM);
    bool pair = false, streamk = false;
    choose_path(h, mode, tp * ceil_div(c, ubk::BM) * n_tiles, pair_rows_tiles * n_tiles,
                (H + ubk::BK - 1) / ubk::BK, true, pair, streamk);
    const int64_t c16 = ceil_div(c, 16) * 16;  // token columns of one chunk in the skinny kernel
    const bool skinny = use_skinny(h, tp * c16);
    if (skinny) pair = false;
    else if (b_kn) pair = true;  // otherwise MN-major operands need CTA pairs
    const int bm = pair ? ubk::PAIR_BM : ubk::BM;      // rows of a tile
    // rows of a B box: one CTA's half in a pair; SwiGLU: the gate or the up half of a tile
    const int bbox = pair || glu ? ubk::BN / 2 : ubk::BN;
    std::vector<const void *> key;
    key.reserve(tp + 7);
    key.push_back(reinterpret_cast<const void *>(uintptr_t(mode)));
    key.push_back(reinterpret_cast<const void *>(uintptr_t(pair + 2 * b_kn + 4 * skinny)));
    key.push_back(reinterpret_cast<const void *>(uintptr_t(T)));
    key.push_back(reinterpret_cast<const void *>(uintptr_t(N)));
    key.push_back(reinterpret_cast<const void *>(uintptr_t(self)));
    key.push_back(Wt);
    key.push_back(Y);
    for (int r = 0; r < tp; ++r) key.push_back(shards[r]);
    GemmParams *pp = cache_lookup(h, key);
    if (!pp) {
        GemmParams p;
        memset(&p, 0, sizeof p);
        p.tp = tp;
        p.c = static_cast<int>(c);
        p.n_out = static_cast<int>(n_out);
        p.glu_f = static_cast<int>(glu_f);
        p.k_blocks = static_cast<int>((H + ubk::BK - 1) / ubk::BK);
        p.k_blocks_per_shard = p.k_blocks;
        p.m_tiles = static_cast<int>((c + bm - 1) / bm);
        p.n_tiles = static_cast<int>(n_tiles);
        p.num_tiles = tp * p.m_tiles * p.n_tiles;
        p.self_rank = self;
        p.self_head = static_cast<int>(pair ? self_head : c);
        if (skinny) {
            // Token sub-tile r = chunk r (c rows, zero-filled to c16), the self chunk in place.
            for (int r = 0; r < tp; ++r) {
                const void *src = r == self ? shards[r] : static_cast<const void *>(ub + r * c * H * 2);
                if (int rc = encode_2d(&p.tmA[r], src, H, c, H * 2, ubk::BK, static_cast<uint32_t>(c16))) return rc;
            }
            if (b_kn) {
                if (int rc = encode_2d(&p.tmB[0], Wt, N, H, N * 2, 64, ubk::BK)) return rc;
                p.b_mn = 1;
            } else if (glu) {
                // gate rows [0, F) and up rows [F, 2F) of Wt as two maps of F rows each
                if (int rc = encode_2d(&p.tmB[0], Wt, H, glu_f, H * 2, ubk::BK, ubk::SK_BM)) return rc;
                if (int rc = encode_2d(&p.tmB[1], static_cast<const char *>(Wt) + glu_f * H * 2, H, glu_f, H * 2,
                                       ubk::BK, ubk::SK_BM))
                    return rc;
            } else if (int rc = encode_2d(&p.tmB[0], Wt, H, N, H * 2, ubk::BK, ubk::SK_BM)) {
                return rc;
            }
            h->counters.tensor_map_encodes += tp + (glu ? 2 : 1);
            p.y_ptr[0] = Y;
            p.ldy = static_cast<int>(n_out);
            p.n_tiles = static_cast<int>((n_out + ubk::SK_BM - 1) / ubk::SK_BM);
            p.sk_sub_n = static_cast<int>(c16);
            p.sk_n_sub = tp;
            pp = cache_insert(h, std::move(key), p);
        } else if (!pair) {
            for (int r = 0; r < tp; ++r) {
                // Chunk r is read from the user buffer, except the self chunk, which the
                // kernel reads in place from its shard while its copy stages it.
                const void *src = r == self ? shards[r] : static_cast<const void *>(ub + r * c * H * 2);
                if (int rc = encode_2d(&p.tmA[r], src, H, c, H * 2, ubk::BK, ubk::BM)) return rc;
                if (int rc = encode_2d(&p.tmY[r], static_cast<char *>(Y) + r * c * n_out * 2, n_out, c, n_out * 2,
                                       ubk::STORE_COLS, 32))
                    return rc;
            }
            h->counters.tensor_map_encodes += 2 * tp;
        } else {
            int nreg = 0;
            for (int i = 0; i < n_regions; ++i) {
                const AgRegion &rgn = regions[i];
                if (int rc = encode_2d(&p.tmA[nreg], rgn.src, H, rgn.rows, H * 2, ubk::BK, 128)) return rc;
                if (int rc = encode_2d(&p.tmY[nreg], static_cast<char *>(Y) + rgn.row0 * n_out * 2, n_out,
                                       rgn.rows, n_out * 2, ubk::STORE_COLS, 32))
                    return rc;
                p.region_row0[nreg] = static_cast<int>(rgn.row0);
                p.region_rows[nreg] = static_cast<int>(rgn.rows);
                p.region_ub[nreg] = rgn.ub_backed;
                p.region_tile0[nreg + 1] =
                    p.region_tile0[nreg] + static_cast<int>((rgn.rows + ubk::PAIR_BM - 1) / ubk::PAIR_BM) * p.n_tiles;
                ++nreg;
            }
            p.n_regions = nreg;
            h->counters.tensor_map_encodes += 2 * nreg;
        }
        if (!skinny) {
            if (b_kn) {
                // W is [hidden, N]: inner dimension N, boxes of 64 N x 64 K rows
                if (int rc = encode_2d(&p.tmB[0], Wt, N, H, N * 2, 64, ubk::BK)) return rc;
                p.b_mn = 1;
            } else if (int rc = encode_2d(&p.tmB[0], Wt, H, N, H * 2, ubk::BK, bbox)) {
                return rc;
            }
            h->counters.tensor_map_encodes += 1;
            pp = cache_insert(h, std::move(key), p);
        }
    }
    GemmParams &p = *pp;
    p.flags = flags_of(h);
    p.abort_word = abort_of(h);
    p.status = status_of(h);
    p.timeout_ns = static_cast<uint64_t>(h->timeout_ns);
    const bool fits_one_wave = pair ? pair_rows_tiles * n_tiles <= clusters_for(h, mode, 1 << 30)
                                    : tp * ceil_div(c, ubk::BM) * n_tiles <= grid_for(h, 1 << 30);
    const bool in_gemm = gather_in_gemm(h, skinny, fits_one_wave);
    if (skinny) set_skinny(h, p, glu ? 2 : 1, glu ? 2 * ubk::SK_W_BYTES : ubk::SK_W_BYTES);
    else if (pair) set_pairs(h, p, mode, streamk, in_gemm, true);
    p.group_m = pair ? ag_group_m(c, ceil_div(self_head, ubk::PAIR_BM) * n_tiles, p.num_pairs) : 0;
    uint32_t epoch = 0;
    if (int rc = begin_call(h, s, epoch, true, pair ? p.tail_split > 1 : skinny && p.sk_split > 1)) return rc;
    p.epoch = epoch;
    const int64_t drop = h->drop_flag;
    h->drop_flag = -1;

    // one wave of tiles: the gather end to end (every chunk needed at once), else part by
    // part (the chunks land in ring order, the first wave's soonest)
    const bool one_wave = pair ? p.region_tile0[p.n_regions] <= p.num_pairs : p.num_tiles <= grid_for(h, 1 << 30);
    p.fused_gather = in_gemm ? (one_wave ? 2 : 1) : 0;
    if (in_gemm && skinny) {
        // few tokens: each chunk copied by its own group of CTAs, at most 32 KB per CTA
        // (the self chunk is a part too); with fewer CTAs than chunks, one CTA per group
        // and some groups copy several chunks
        const int64_t grid = grid_for(h, p.sk_units), parts = tp;
        int64_t gs = (c * H / 8 + 2047) / 2048;
        if (gs > grid / parts) gs = grid / parts;
        p.fused_gather = 3;
        p.g_group = static_cast<int>(gs < 1 ? 1 : gs);
    }
    if (in_gemm) {
        for (int r = 0; r < tp; ++r) p.g_src[r] = shards[r];
        p.g_ub = h->ub;
        p.g_counters = gather_counters_of(h);
        p.g_chunk_vecs = c * H / 8;
        p.g_self_head_vecs = p.self_head * H / 8;
        p.g_drop = static_cast<int>(drop);
        p.after_gather = 0;
        int rc = launch(h, p, mode, skinny ? PATH_SKINNY : pair ? PATH_PAIR : PATH_SINGLE, s, prof_op);
        if (rc != UB_OK) return rc;
    } else {
        if (int rc = issue_gather(h, shards, s, epoch, drop, p.self_head, fits_one_wave)) return rc;
        // chained: the GEMM is the gather kernel's programmatic dependent (no wait at entry:
        // the chunk flags order its reads of the buffer; one thread waits for the gather at
        // exit, so that the call completes only after both)
        p.after_gather = h->gather_chained ? 1 : 0;
        int rc = launch(h, p, mode, skinny ? PATH_SKINNY : pair ? PATH_PAIR : PATH_SINGLE, s, prof_op);
        // Join the copy streams back into `s` even if the launch failed.
        if (int jrc = join_gather(h, s)) return jrc;
        if (rc != UB_OK) return rc;
    }
    h->counters.last_gather = in_gemm ? 2 : h->gather_by_kernel ? 1 : 0;
    ++h->counters.ag_calls;
    h->counters.last_T = T;
    return UB_OK;
}

int ag_gemm(ub_handle_t h, const void *const *shards, const void *Wt, int64_t N, void *Y, void *stream)
{
    return ag_gemm_impl(h, shards, Wt, N, Y, stream, 0, false);
}

int ag_gemm_kn(ub_handle_t h, const void *const *shards, const void *W, int64_t N, void *Y, void *stream)
{
    return ag_gemm_impl(h, shards, W, N, Y, stream, 0, true);
}

int ag_gemm_swiglu(ub_handle_t h, const void *const *shards, const void *Wt, int64_t F, void *Z, void *stream)
{
    if (F <= 0) return fail(UB_ERR_ZERO, "ag_gemm_swiglu: F = %lld", (long long)F);
    if (F % 8 != 0) return fail(UB_ERR_ALIGN, "ag_gemm_swiglu: F = %lld is not a multiple of 8", (long long)F);
    return ag_gemm_impl(h, shards, Wt, 2 * F, Z, stream, F, false);
}

// GEMM-RS; with b_kn the shard weights are stored K x hidden (read MN-major).
static int gemm_rs_impl(ub_handle_t h, const void *const *A, const void *const *Bt, int64_t K, void *const *Y_shards,
                        void *stream, bool b_kn)
{
    if (int rc = check_handle(h)) return rc;
    if (!A || !Bt || !Y_shards) return fail(UB_ERR_ARG, "gemm_rs: null pointer argument");
    if (K <= 0) return fail(UB_ERR_ZERO, "gemm_rs: K = %lld", (long long)K);
    if (K % 8 != 0) return fail(UB_ERR_ALIGN, "gemm_rs: K = %lld is not a multiple of 8", (long long)K);
    if (K > (int64_t(1) << 24)) return fail(UB_ERR_ARG, "gemm_rs: K = %lld too large", (long long)K);
    const int tp = h->tp;
    for (int j = 0; j < tp; ++j) {
        if (!A[j] || !Bt[j] || !Y_shards[j]) return fail(UB_ERR_ARG, "gemm_rs: pointer %d is null", j);
        if (!aligned16(A[j]) || !aligned16(Bt[j]) || !aligned16(Y_shards[j]))
            return fail(UB_ERR_ALIGN, "gemm_rs: pointer %d not 16-byte aligned", j);
    }
    DeviceGuard g(h->device);
    if (!g.ok) return fail(UB_ERR_CUDA, "gemm_rs: cannot select the handle's device");
    NvtxRange range(b_kn ? "gemm_rs_kn" : "gemm_rs", h->T);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t T = h->T, H = h->hidden, c = T / tp;

    const int64_t n_tiles = (H + ubk::BN - 1) / ubk::BN;
    bool pair = false, streamk = false;
    choose_path(h, ubk::MODE_RS, tp * ceil_div(c, ubk::BM) * n_tiles, ceil_div(T, ubk::PAIR_BM) * n_tiles,
                tp * ((K + ubk::BK - 1) / ubk::BK), false, pair, streamk);
    const int64_t T16 = ceil_div(T, 16) * 16;  // token columns in the skinny kernel
    const bool skinny = use_skinny(h, T16);
    if (skinny) pair = false;
    else if (b_kn) pair = true;  // otherwise MN-major operands need CTA pairs
    const int bm = pair ? ubk::PAIR_BM : ubk::BM;
    const int bbox = pair ? ubk::BN / 2 : ubk::BN;
    std::vector<const void *> key;
    key.reserve(3 * tp + 4);
    key.push_back(reinterpret_cast<const void *>(uintptr_t(ubk::MODE_RS)));
    key.push_back(reinterpret_cast<const void *>(uintptr_t(pair + 2 * b_kn + 4 * skinny)));
    key.push_back(reinterpret_cast<const void *>(uintptr_t(T)));
    key.push_back(reinterpret_cast<const void *>(uintptr_t(K)));
    for (int j = 0; j < tp; ++j) {
        key.push_back(A[j]);
        key.push_back(Bt[j]);
        key.push_back(Y_shards[j]);
    }
    GemmParams *pp = cache_lookup(h, key);
    if (!pp && skinny) {
        GemmParams p;
        memset(&p, 0, sizeof p);
        for (int j = 0; j < tp; ++j) {
            // all T tokens of A_j in one box (zero-filled to T16 rows)
            if (int rc = encode_2d(&p.tmA[j], A[j], K, T, K * 2, ubk::BK, static_cast<uint32_t>(T16))) return rc;
            if (b_kn) {
                if (int rc = encode_2d(&p.tmB[j], Bt[j], H, K, H * 2, 64, ubk::BK)) return rc;
            } else if (int rc = encode_2d(&p.tmB[j], Bt[j], K, H, K * 2, ubk::BK, ubk::SK_BM)) {
                return rc;
            }
            p.y_ptr[j] = Y_shards[j];
        }
        h->counters.tensor_map_encodes += 2 * tp;
        p.b_mn = b_kn ? 1 : 0;
        p.tp = tp;
        p.c = static_cast<int>(c);
        p.n_out = static_cast<int>(H);
        p.ldy = static_cast<int>(H);
        p.k_blocks_per_shard = static_cast<int>((K + ubk::BK - 1) / ubk::BK);
        p.k_blocks = tp * p.k_blocks_per_shard;
        p.n_tiles = static_cast<int>((H + ubk::SK_BM - 1) / ubk::SK_BM);
        p.sk_sub_n = static_cast<int>(T16);
        p.sk_n_sub = 1;
        pp = cache_insert(h, std::move(key), p);
    }
    if (!pp) {
        GemmParams p;
        memset(&p, 0, sizeof p);
        for (int j = 0; j < tp; ++j) {
            if (int rc = encode_2d(&p.tmA[j], A[j], K, T, K * 2, ubk::BK, ubk::BM)) return rc;
            if (b_kn) {
                // B_j is [K, hidden]: inner dimension hidden, boxes of 64 x 64 K rows
                if (int rc = encode_2d(&p.tmB[j], Bt[j], H, K, H * 2, 64, ubk::BK)) return rc;
            } else if (int rc = encode_2d(&p.tmB[j], Bt[j], K, H, K * 2, ubk::BK, bbox)) {
                return rc;
            }
            if (int rc = encode_2d(&p.tmY[j], Y_shards[j], H, c, H * 2, ubk::STORE_COLS, 32)) return rc;
            p.y_ptr[j] = Y_shards[j];
        }
        h->counters.tensor_map_encodes += 3 * tp;
        // The pair kernel tiles all T rows as one region; stores split at chunk ends.
        p.n_regions = 1;
        p.region_row0[0] = 0;
        p.region_rows[0] = static_cast<int>(T);
        p.region_ub[0] = 0;
        p.region_tile0[1] = static_cast<int>((T + ubk::PAIR_BM - 1) / ubk::PAIR_BM) *
                            static_cast<int>((H + ubk::BN - 1) / ubk::BN);
        p.ldy = static_cast<int>(H);
        p.b_mn = b_kn ? 1 : 0;
        p.tp = tp;
        p.c = static_cast<int>(c);
        p.n_out = static_cast<int>(H);
        p.k_blocks_per_shard = static_cast<int>((K + ubk::BK - 1) / ubk::BK);
        p.k_blocks = tp * p.k_blocks_per_shard;
        p.m_tiles = static_cast<int>((c + bm - 1) / bm);
        p.n_tiles = static_cast<int>((H + ubk::BN - 1) / ubk::BN);
        p.num_tiles = tp * p.m_tiles * p.n_tiles;
        p.self_rank = 0;
        pp = cache_insert(h, std::move(key), p);
    }
    GemmParams &p = *pp;
    p.flags = flags_of(h);
    p.abort_word = abort_of(h);
    p.status = status_of(h);
    p.timeout_ns = static_cast<uint64_t>(h->timeout_ns);
    if (skinny) set_skinny(h, p, 1, ubk::SK_W_BYTES);
    else if (pair) set_pairs(h, p, ubk::MODE_RS, streamk);
    // weight panels that together exceed L2 several times over (the large RS at K = 3584:
    // 470 MB) would be re-read from HBM by every wave walked N fastest
    p.group_m = pair && static_cast<int64_t>(tp) * K * H * 2 > kGroupedOrderBytes ? kGroupM : 0;
    uint32_t epoch = 0;
    if (int rc = begin_call(h, s, epoch, false, pair ? p.tail_split > 1 : skinny && p.sk_split > 1)) return rc;
    p.epoch = epoch;
    if (int rc = launch(h, p, ubk::MODE_RS, skinny ? PATH_SKINNY : pair ? PATH_PAIR : PATH_SINGLE, s,
                        b_kn ? UB_OP_RS_KN : UB_OP_RS))
        return rc;
    ++h->counters.rs_calls;
    h->counters.last_T = T;
    return UB_OK;
}

int gemm_rs(ub_handle_t h, const void *const *A, const void *const *Bt, int64_t K, void *const *Y_shards,
            void *stream)
{
    return gemm_rs_impl(h, A, Bt, K, Y_shards, stream, false);
}

int gemm_rs_kn(ub_handle_t h, const void *const *A, const void *const *B, int64_t K, void *const *Y_shards,
               void *stream)
{
    return gemm_rs_impl(h, A, B, K, Y_shards, stream, true);
}

int ub_allgather(ub_handle_t h, const void *const *shards, void *stream)
{
    if (int rc = check_handle(h)) return rc;
    if (!shards) return fail(UB_ERR_ARG, "ub_allgather: null pointer argument");
    for (int r = 0; r < h->tp; ++r) {
        if (!shards[r]) return fail(UB_ERR_ARG, "ub_allgather: shard %d is null", r);
        if (!aligned16(shards[r])) return fail(UB_ERR_ALIGN, "ub_allgather: shard %d not 16-byte aligned", r);
    }
    DeviceGuard g(h->device);
    if (!g.ok) return fail(UB_ERR_CUDA, "ub_allgather: cannot select the handle's device");
    NvtxRange range("ub_allgather", h->T);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t epoch = 0;
    if (int rc = begin_call(h, s, epoch, false, false)) return rc;
    if (h->bulk_beside) {
        // the gather kernel on `stream` itself, a programmatic dependent of the kernel
        // before it: about one CTA per SM, in the room that kernel's CTAs leave
        ubk::GatherParams g = gather_kernel_params(h, shards, epoch, -1);
        g.pdl = 1;
        g.beside = 1;
        cudaError_t e = ubk::launch_gather(g, s);
        if (e != cudaSuccess) return cuda_fail(e, "gather kernel launch");
        h->counters.last_T = h->T;
        return UB_OK;
    }
    if (int rc = issue_gather(h, shards, s, epoch, -1, h->T / h->tp)) return rc;
    if (int rc = join_gather(h, s)) return rc;
    h->counters.last_T = h->T;
    return UB_OK;
}

int ub_stream_read(ub_handle_t h, const void *src, int64_t bytes, void *stream)
{
    if (int rc = check_handle(h)) return rc;
    if (!src || bytes < 0) return fail(UB_ERR_ARG, "ub_stream_read: null source or negative size");
    if (!aligned16(src) || bytes % 16 != 0)
        return fail(UB_ERR_ALIGN, "ub_stream_read: source or size not a multiple of 16 bytes");
    if (bytes == 0) return UB_OK;
    DeviceGuard g(h->device);
    if (!g.ok) return fail(UB_ERR_CUDA, "ub_stream_read: cannot select the handle's device");
    NvtxRange range("ub_stream_read", bytes);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t epoch = 0;
    if (int rc = begin_call(h, s, epoch, false, false)) return rc;
    ubk::StreamReadParams p;
    memset(&p, 0, sizeof p);
    p.src = static_cast<const char *>(src);
    p.bytes = bytes;
    p.abort_word = abort_of(h);
    p.status = status_of(h);
    p.timeout_ns = static_cast<uint64_t>(h->timeout_ns);
    p.epoch = epoch;
    p.pdl = static_cast<int>(h->pdl);
    cudaError_t e = ubk::launch_stream_read(p, h->sm_count, s);
    if (e != cudaSuccess) return cuda_fail(e, "stream-read kernel launch");
    return UB_OK;
}

int ub_reduce_scatter(ub_handle_t h, const void *const *P, void *const *Y_shards, void *stream)
{
    if (int rc = check_handle(h)) return rc;
    if (!P || !Y_shards) return fail(UB_ERR_ARG, "ub_reduce_scatter: null pointer argument");
    const int tp = h->tp;
    ubk::BulkRsParams p;
    memset(&p, 0, sizeof p);
    for (int j = 0; j < tp; ++j) {
        if (!P[j] || !Y_shards[j]) return fail(UB_ERR_ARG, "ub_reduce_scatter: pointer %d is null", j);
        if (!aligned16(P[j]) || !aligned16(Y_shards[j]))
            return fail(UB_ERR_ALIGN, "ub_reduce_scatter: pointer %d not 16-byte aligned", j);
        p.P[j] = P[j];
        p.Y[j] = Y_shards[j];
    }
    DeviceGuard g(h->device);
    if (!g.ok) return fail(UB_ERR_CUDA, "ub_reduce_scatter: cannot select the handle's device");
    NvtxRange range("ub_reduce_scatter", h->T);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    p.tp = tp;
    p.T = h->T;
    p.H = h->hidden;
    p.c = h->T / tp;
    p.pdl = static_cast<int>(h->pdl);
    // Small CTAs, four per SM: alone, they keep enough loads in flight to stream HBM; beside
    // a persistent GEMM CTA one of them fits on each SM (the rest start as GEMM CTAs leave).
    // Beside mode: one per SM, all of them running beside the kernel before it on `s`
    // (a CTA that waits for that kernel at its exit would hold back any CTA queued behind).
    p.beside = h->bulk_beside ? 1 : 0;
    if (p.beside) p.pdl = 1;
    const int64_t vecs = p.T * (p.H / 8);
    int64_t grid = (p.beside ? 1 : 4) * static_cast<int64_t>(h->sm_count);
    if (grid > (vecs + 255) / 256) grid = (vecs + 255) / 256;
    ProfileRing &ring = h->prof[UB_OP_REDUCE_SCATTER];
    const bool timed = h->profile != 0 && ring.count < kMaxProfiled;
    if (timed) {
        if (static_cast<int>(ring.start.size()) <= ring.count) {
            cudaEvent_t e0, e1;
            UB_CUDA(cudaEventCreate(&e0));
            UB_CUDA(cudaEventCreate(&e1));
            ring.start.push_back(e0);
            ring.stop.push_back(e1);
        }
        UB_CUDA(cudaEventRecord(ring.start[ring.count], s));
    }
    cudaError_t e = ubk::launch_bulk_rs(p, static_cast<int>(grid), s);
    if (e != cudaSuccess) return cuda_fail(e, "reduce-scatter kernel launch");
    if (timed) {
        UB_CUDA(cudaEventRecord(ring.stop[ring.count], s));
        ++ring.count;
    }
    h->counters.last_T = h->T;
    return UB_OK;
}

int ub_wgrad(ub_handle_t h, const void *D, int64_t M, int ub_is_a, void *out, void *stream)
{
    if (int rc = check_handle(h)) return rc;
    if (!D || !out) return fail(UB_ERR_ARG, "ub_wgrad: null pointer argument");
    if (M <= 0) return fail(UB_ERR_ZERO, "ub_wgrad: M = %lld", (long long)M);
    if (M % 8 != 0) return fail(UB_ERR_ALIGN, "ub_wgrad: M = %lld is not a multiple of 8", (long long)M);
    if (M > (int64_t(1) << 24)) return fail(UB_ERR_ARG, "ub_wgrad: M = %lld too large", (long long)M);
    if (!aligned16(D) || !aligned16(out)) return fail(UB_ERR_ALIGN, "ub_wgrad: D / out not 16-byte aligned");
    if (ub_is_a != 0 && ub_is_a != 1) return fail(UB_ERR_ARG, "ub_wgrad: ub_is_a must be 0 or 1");
    DeviceGuard g(h->device);
    if (!g.ok) return fail(UB_ERR_CUDA, "ub_wgrad: cannot select the handle's device");
    NvtxRange range("ub_wgrad", h->T);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t T = h->T, H = h->hidden;
    // out = A^T B over the T active rows; A and B are [T, .] row-major (MN-major operands)
    const void *Aop = ub_is_a ? h->ub : D;
    const void *Bop = ub_is_a ? D : h->ub;
    const int64_t rows = ub_is_a ? H : M, cols = ub_is_a ? M : H;

    std::vector<const void *> key = {reinterpret_cast<const void *>(uintptr_t(100 + ub_is_a)),
                                     reinterpret_cast<const void *>(uintptr_t(T)),
                                     reinterpret_cast<const void *>(uintptr_t(M)), D, out};
    GemmParams *pp = cache_lookup(h, key);
    if (!pp) {
        GemmParams p;
        memset(&p, 0, sizeof p);
        if (int rc = encode_2d(&p.tmA[0], Aop, rows, T, rows * 2, 64, ubk::BK)) return rc;
        if (int rc = encode_2d(&p.tmB[0], Bop, cols, T, cols * 2, 64, ubk::BK)) return rc;
        if (int rc = encode_2d(&p.tmY[0], out, cols, rows, cols * 2, ubk::STORE_COLS, 32)) return rc;
        h->counters.tensor_map_encodes += 3;
        p.tp = h->tp;
        p.c = static_cast<int>(T / h->tp);
        p.n_out = static_cast<int>(cols);
        p.k_blocks = static_cast<int>((T + ubk::BK - 1) / ubk::BK);
        p.k_blocks_per_shard = p.k_blocks;
        p.n_tiles = static_cast<int>((cols + ubk::BN - 1) / ubk::BN);
        p.n_regions = 1;
        p.region_row0[0] = 0;
        p.region_rows[0] = static_cast<int>(rows);
        p.region_ub[0] = 0;  // the buffer already holds the gathered rows: no flags to wait for
        p.region_tile0[1] = static_cast<int>((rows + ubk::PAIR_BM - 1) / ubk::PAIR_BM) * p.n_tiles;
        p.a_mn = 1;
        p.b_mn = 1;
        pp = cache_insert(h, std::move(key), p);
    }
    GemmParams &p = *pp;
    p.flags = flags_of(h);
    p.abort_word = abort_of(h);
    p.status = status_of(h);
    p.timeout_ns = static_cast<uint64_t>(h->timeout_ns);
    bool pair = true, split = false;
    choose_path(h, ubk::MODE_AG, 1 << 30, p.region_tile0[1], p.k_blocks, false, pair, split);
    set_pairs(h, p, ubk::MODE_AG, split);
    uint32_t epoch = 0;
    if (int rc = begin_call(h, s, epoch, false, p.tail_split > 1)) return rc;
    p.epoch = epoch;
    if (int rc = launch(h, p, ubk::MODE_AG, PATH_PAIR, s, UB_OP_WGRAD)) return rc;
    h->counters.last_T = T;
    return UB_OK;
}

int ag_gemm_from_buffer(ub_handle_t h, const void *Wt, int64_t N, int64_t glu_f, void *Y, void *stream)
{
    if (int rc = check_handle(h)) return rc;
    if (!Wt || !Y) return fail(UB_ERR_ARG, "ag_gemm_from_buffer: null pointer argument");
    if (N <= 0) return fail(UB_ERR_ZERO, "ag_gemm_from_buffer: N = %lld", (long long)N);
    if (N % 8 != 0) return fail(UB_ERR_ALIGN, "ag_gemm_from_buffer: N = %lld is not a multiple of 8", (long long)N);
    if (glu_f < 0 || (glu_f > 0 && (N != 2 * glu_f || glu_f % 8 != 0)))
        return fail(UB_ERR_ARG, "ag_gemm_from_buffer: SwiGLU needs N = 2 * F with F a multiple of 8");
    if (N > (int64_t(1) << 24)) return fail(UB_ERR_ARG, "ag_gemm_from_buffer: N = %lld too large", (long long)N);
    if (!aligned16(Wt) || !aligned16(Y)) return fail(UB_ERR_ALIGN, "ag_gemm_from_buffer: Wt / Y not 16-byte aligned");
    DeviceGuard g(h->device);
    if (!g.ok) return fail(UB_ERR_CUDA, "ag_gemm_from_buffer: cannot select the handle's device");
    NvtxRange range("ag_gemm_from_buffer", h->T);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t T = h->T, H = h->hidden;
    const bool glu = glu_f > 0;
    const int mode = glu ? ubk::MODE_AG_GLU : ubk::MODE_AG;
    const int64_t n_out = glu ? glu_f : N;
    std::vector<const void *> key = {reinterpret_cast<const void *>(uintptr_t(200 + (glu ? 1 : 0))),
                                     reinterpret_cast<const void *>(uintptr_t(T)),
                                     reinterpret_cast<const void *>(uintptr_t(N)), Wt, Y};
    GemmParams *pp = cache_lookup(h, key);
    if (!pp) {
        GemmParams p;
        memset(&p, 0, sizeof p);
        // One region: all T rows of the buffer, no readiness flags (already gathered).
        if (int rc = encode_2d(&p.tmA[0], h->ub, H, T, H * 2, ubk::BK, 128)) return rc;
        if (int rc = encode_2d(&p.tmB[0], Wt, H, N, H * 2, ubk::BK, ubk::BN / 2)) return rc;
        if (int rc = encode_2d(&p.tmY[0], Y, n_out, T, n_out * 2, ubk::STORE_COLS, 32)) return rc;
        h->counters.tensor_map_encodes += 3;
        p.tp = h->tp;
        p.c = static_cast<int>(T / h->tp);
        p.n_out = static_cast<int>(n_out);
        p.glu_f = static_cast<int>(glu_f);
        p.k_blocks = static_cast<int>((H + ubk::BK - 1) / ubk::BK);
        p.k_blocks_per_shard = p.k_blocks;
        p.n_tiles = static_cast<int>(glu ? (glu_f + 127) / 128 : (N + ubk::BN - 1) / ubk::BN);
        p.self_head = static_cast<int>(T / h->tp);
        p.n_regions = 1;
        p.region_row0[0] = 0;
        p.region_rows[0] = static_cast<int>(T);
        p.region_ub[0] = 0;
        p.region_tile0[1] = static_cast<int>((T + ubk::PAIR_BM - 1) / ubk::PAIR_BM) * p.n_tiles;
        pp = cache_insert(h, std::move(key), p);
    }
    GemmParams &p = *pp;
    p.flags = flags_of(h);
    p.abort_word = abort_of(h);
    p.status = status_of(h);
    p.timeout_ns = static_cast<uint64_t>(h->timeout_ns);
    bool pair = true, split = false;
    choose_path(h, mode, 1 << 30, p.region_tile0[1], p.k_blocks, false, pair, split);
    set_pairs(h, p, mode, split);
    p.group_m = kGroupM;  // every row is in the buffer already: no chunk to wait for
    uint32_t epoch = 0;
    if (int rc = begin_call(h, s, epoch, false, p.tail_split > 1)) return rc;
    p.epoch = epoch;
    p.fused_gather = 0;
    if (int rc = launch(h, p, mode, PATH_PAIR, s, glu ? UB_OP_AG_SWIGLU : UB_OP_AG)) return rc;
    ++h->counters.ag_calls;
    h->counters.last_T = T;
    return UB_OK;
}

int ub_set_option(ub_handle_t h, int key, int64_t val)
{
    if (int rc = check_handle(h)) return rc;
    switch (key) {
    case UB_OPT_SM_MARGIN:
        if (val < 0 || val >= h->sm_count) return fail(UB_ERR_ARG, "sm_margin %lld outside [0, %d)", (long long)val, h->sm_count);
        h->sm_margin = val;
        return UB_OK;
    case UB_OPT_TIMEOUT_NS:
        if (val < 1000) return fail(UB_ERR_ARG, "timeout %lld ns below 1 us", (long long)val);
        h->timeout_ns = val;
        return UB_OK;
    case UB_OPT_SELF_RANK:
        if (val < 0 || val >= h->tp) return fail(UB_ERR_ARG, "self rank %lld outside [0, %d)", (long long)val, h->tp);
        h->self_rank = val;
        return UB_OK;
    case UB_OPT_DROP_FLAG:
        if (val < -1 || val >= h->tp) return fail(UB_ERR_ARG, "drop_flag %lld outside [-1, %d)", (long long)val, h->tp);
        h->drop_flag = val;
        return UB_OK;
    case UB_OPT_PROFILE:
        if (val != 0 && val != 1) return fail(UB_ERR_ARG, "profile must be 0 or 1");
        h->profile = val;
        return UB_OK;
    case UB_OPT_CTA_PAIR:
        if (val < -1 || val > 1) return fail(UB_ERR_ARG, "cta_pair must be -1, 0 or 1");
        h->cta_pair = val;
        return UB_OK;
    case UB_OPT_STREAMK:
        if (val < -1 || val > ubk::MAX_TAIL_SPLIT)
            return fail(UB_ERR_ARG, "streamk must be -1, 0, 1 or a piece count 2..%d", ubk::MAX_TAIL_SPLIT);
        h->streamk = val;
        return UB_OK;
    case UB_OPT_SKINNY:
        if (val < -1 || val > 1) return fail(UB_ERR_ARG, "UB_OPT_SKINNY must be -1, 0 or 1");
        h->skinny = val;
        return UB_OK;
    case UB_OPT_PDL:
        if (val != 0 && val != 1) return fail(UB_ERR_ARG, "UB_OPT_PDL must be 0 or 1");
        h->pdl = val;
        return UB_OK;
    case UB_OPT_BULK_BESIDE:
        if (val != 0 && val != 1) return fail(UB_ERR_ARG, "UB_OPT_BULK_BESIDE must be 0 or 1");
        h->bulk_beside = val;
        return UB_OK;
    case UB_OPT_GATHER_CHAIN:
        if (val != 0 && val != 1) return fail(UB_ERR_ARG, "UB_OPT_GATHER_CHAIN must be 0 or 1");
        h->gather_chain = val;
        return UB_OK;
    case UB_OPT_GATHER_KERNEL:
        if (val < -1 || val > 2) return fail(UB_ERR_ARG, "gather_kernel must be -1, 0, 1 or 2");
        h->gather_kernel = val;
        return UB_OK;
    case UB_OPT_COPY_STREAMS: {
        if (val < 0 || val > UB_MAX_TP) return fail(UB_ERR_ARG, "copy_streams must be in [0, %d]", UB_MAX_TP);
        DeviceGuard g(h->device);
        for (int i = 1; i < val; ++i) {
            if (!h->extra_side[i]) UB_CUDA(cudaStreamCreateWithFlags(&h->extra_side[i], cudaStreamNonBlocking));
            if (!h->ev_join_extra[i]) UB_CUDA(cudaEventCreateWithFlags(&h->ev_join_extra[i], cudaEventDisableTiming));
        }
        h->copy_streams = val;
        return UB_OK;
    }
    default:
        return fail(UB_ERR_ARG, "unknown option %d", key);
    }
}

int ub_get_option(ub_handle_t h, int key, int64_t *val)
{
    if (int rc = check_handle(h)) return rc;
    if (!val) return fail(UB_ERR_ARG, "null output");
    switch (key) {
    case UB_OPT_SM_MARGIN: *val = h->sm_margin; return UB_OK;
    case UB_OPT_TIMEOUT_NS: *val = h->timeout_ns; return UB_OK;
    case UB_OPT_SELF_RANK: *val = h->self_rank; return UB_OK;
    case UB_OPT_DROP_FLAG: *val = h->drop_flag; return UB_OK;
    case UB_OPT_PROFILE: *val = h->profile; return UB_OK;
    case UB_OPT_CTA_PAIR: *val = h->cta_pair; return UB_OK;
    case UB_OPT_STREAMK: *val = h->streamk; return UB_OK;
    case UB_OPT_COPY_STREAMS: *val = h->copy_streams; return UB_OK;
    case UB_OPT_GATHER_KERNEL: *val = h->gather_kernel; return UB_OK;
    case UB_OPT_SKINNY: *val = h->skinny; return UB_OK;
    case UB_OPT_PDL: *val = h->pdl; return UB_OK;
    case UB_OPT_BULK_BESIDE: *val = h->bulk_beside; return UB_OK;
    case UB_OPT_GATHER_CHAIN: *val = h->gather_chain; return UB_OK;
    default: return fail(UB_ERR_ARG, "unknown option %d", key);
    }
}

int ub_query_status(ub_handle_t h)
{
    if (int rc = check_handle(h)) return rc;
    DeviceGuard g(h->device);
    int32_t st = 0;
    UB_CUDA(cudaMemcpyAsync(&st, status_of(h), sizeof st, cudaMemcpyDeviceToHost, h->side));
    UB_CUDA(cudaStreamSynchronize(h->side));
    return st;
}

int ub_clear_status(ub_handle_t h)
{
    if (int rc = check_handle(h)) return rc;
    DeviceGuard g(h->device);
    UB_CUDA(cudaMemsetAsync(abort_of(h), 0, 2 * sizeof(uint32_t), h->side));  // abort and status words
    UB_CUDA(cudaStreamSynchronize(h->side));
    return UB_OK;
}

int ub_get_counters(ub_handle_t h, ub_counters_t *out)
{
    if (int rc = check_handle(h)) return rc;
    if (!out) return fail(UB_ERR_ARG, "null output");
    *out = h->counters;
    return UB_OK;
}

int ub_kernel_time(ub_handle_t h, int op, double *total_ms, int64_t *launches)
{
    if (int rc = check_handle(h)) return rc;
    if (op < 0 || op >= UB_NUM_OPS) return fail(UB_ERR_ARG, "unknown op %d", op);
    DeviceGuard g(h->device);
    ProfileRing &ring = h->prof[op];
    double sum = 0.0;
    if (ring.count > 0) UB_CUDA(cudaEventSynchronize(ring.stop[ring.count - 1]));
    for (int i = 0; i < ring.count; ++i) {
        float ms = 0.f;
        UB_CUDA(cudaEventElapsedTime(&ms, ring.start[i], ring.stop[i]));
        sum += ms;
    }
    if (total_ms) *total_ms = sum;
    if (launches) *launches = ring.count;
    ring.count = 0;
    return UB_OK;
}

}  // extern "C"
