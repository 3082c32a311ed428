/*
 * ub.h -- C ABI of libubgemm: active-shape tensor-parallel AG-GEMM and GEMM-RS on one
 * GB300 (sm_103a), with the tp "ranks" as virtual shards resident in the same HBM.
 *
 * The operations follow three public pages on tensor-parallel communication/GEMM
 * overlap:
 *  [P1] "Do tp overlap support thd, whose sequence length is flexible?"
 *       (Megatron-LM discussion #1240), answer: QKV and MLP diagrams
 *       (ColumnParallelLinear after the all-gather of [S, H]; RowParallelLinear
 *       whose [S, H] output is summed over ranks and split by rows); the user buffer
 *       is sized by the communicated tensor [S, hidden], not the GEMM output.
 *  [P2] "Support dynamic token counts in TP communication/GEMM overlap"
 *       (TransformerEngine issue #3564): "Proposed API" (initialize at
 *       [max_tokens, hidden], set an active shape per microbatch), "Implementation
 *       approach in the prototype" (capacity and active shape kept apart; nothing
 *       allocated, freed or re-registered; active data is a contiguous prefix; chunk
 *       offsets and counts use the active first dimension) and "Constrain the initial
 *       behavior" (2-D, nonzero, within capacity, hidden unchanged, T divisible by
 *       tp; unquantized 2-byte BF16 only).
 *  [P3] "How to setup TP Overlap configs" (TransformerEngine issue #1344): the
 *       "ring_exchange" method with copy-engine send/recv ("use_ce"), "num_splits"
 *       forced to the TP size, the on-device chunk loop of "atomic_gemm", and the
 *       "num_sm" / "set_sm_margin" SM reservation.
 *
 * Conventions for every call:
 *  - All matrices are row-major BF16. Linear weights are stored out x in, the layout
 *    of a PyTorch nn.Linear weight: the column-parallel weight is Wt[N][hidden]
 *    (Y = X * Wt^T), each row-parallel shard weight is Bt_j[hidden][K]
 *    (S = sum_j A_j * Bt_j^T). Accumulation is fp32; outputs are rounded to BF16
 *    (round to nearest even).
 *  - Device pointers must be 16-byte aligned and N, K, hidden multiples of 8
 *    (UB_ERR_ALIGN otherwise): rows are moved by the tensor memory accelerator.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are
 *    asynchronous on it; the caller keeps every buffer alive until the stream has
 *    passed the call. Results are deterministic run to run for a given launch shape:
 *    where a tile's K range is split over several CTAs (the last wave of the CTA-pair
 *    kernel, the few-token kernel) the fp32 partials are added in a fixed piece order,
 *    and atomics only count finished gather copies and record the status word; no
 *    result is accumulated atomically. The split depends only on the shapes and the
 *    SM count.
 *  - Every function returns UB_OK (0) or a negative UB_ERR_* code; on error the
 *    state of the handle is unchanged and ub_last_error() describes the failure.
 *  - A handle is used from one host thread at a time.
 */
#ifndef UB_H
#define UB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define UB_MAX_TP 8 /* virtual ranks per handle */

typedef struct ub_handle *ub_handle_t; /* opaque; owned by the library */

typedef enum { UB_BF16 = 0 } ub_dtype_t; /* [P2] "Constrain...": 2-byte BF16 only */

enum {
    UB_OK = 0,
    UB_ERR_ARG = -1,       /* null pointer, tp out of [1, UB_MAX_TP], bad option */
    UB_ERR_DTYPE = -2,     /* dtype other than UB_BF16 */
    UB_ERR_RANK = -3,      /* active shape not two-dimensional */
    UB_ERR_ZERO = -4,      /* a zero (or negative) extent */
    UB_ERR_CAPACITY = -5,  /* T larger than the registered max_tokens */
    UB_ERR_HIDDEN = -6,    /* hidden differs from the registered hidden */
    UB_ERR_DIVISIBLE = -7, /* T (or max_tokens) not divisible by tp */
    UB_ERR_ALIGN = -8,     /* pointer not 16-byte aligned, or N / K / hidden % 8 != 0 */
    UB_ERR_CUDA = -9,      /* a CUDA runtime or driver call failed */
    UB_ERR_TIMEOUT = -10   /* a bounded device-side wait expired (see ub_query_status) */
};

/* Options for ub_set_option / ub_get_option. */
enum {
    UB_OPT_SM_MARGIN = 1,  /* SMs left out of the GEMM grid ([P3] "num_sm"); default 0 */
    UB_OPT_TIMEOUT_NS = 2, /* bound of every device-side wait, ns; default 1e9 */
    UB_OPT_SELF_RANK = 3,  /* ring start of ag_gemm: the chunk read in place; default 0 */
    UB_OPT_DROP_FLAG = 4,  /* fault injection on the host: the next ag_gemm skips the
                              readiness-flag write of this chunk (-1 = off, one-shot) */
    UB_OPT_PROFILE = 5,    /* 1 = time every GEMM kernel launch with CUDA events */
    UB_OPT_CTA_PAIR = 6,   /* -1 (default) = chosen per call from the tile counts; 1 = 256x256
                              tiles on CTA pairs (tcgen05 cta_group::2); 0 = chunk-aligned
                              128x256 tiles on single CTAs */
    UB_OPT_STREAMK = 7,    /* pair tiles only. -1 (default) = chosen per call; 1 = the last,
                              partial wave's tiles are cut into equal k-pieces spread over the
                              idle pairs, as many as allowed (fixed-order fp32 fix-up:
                              deterministic); 2..8 = the same with at most that many pieces;
                              0 = whole tiles only */
    UB_OPT_COPY_STREAMS = 8, /* side streams the ag_gemm chunk copies are dealt over
                              (round-robin in ring order), 1..UB_MAX_TP; default min(tp, 4).
                              0 = no overlap: the copies and flag writes go on the call's own
                              stream ahead of the GEMM (a comparator; slower on GB300) */
    UB_OPT_GATHER_KERNEL = 9, /* 0: the gather is one cudaMemcpyAsync plus one stream flag write
                              per chunk; 1: one kernel launch on the side stream lands every
                              chunk in ring order and publishes each chunk's flag as its last
                              CTA finishes (fewer driver operations per call); 2: the GEMM's
                              own epilogue warps copy the chunks before their first tile and
                              publish the flags (the few-token kernel: each chunk by its own
                              few CTAs); -1 (default): the tile kernels 2 when T > 512 and
                              the call has more than one wave of tiles, else 1; the
                              few-token kernel 1 (ub_allgather uses 1 or 0 instead of 2) */
    UB_OPT_SKINNY = 10,    /* few-token kernel: weight rows on the MMA's M, tokens on its N, so
                              the work follows T and the weight is read once. Usable while the
                              token columns (ag_gemm*: tp * roundup(T/tp, 16); gemm_rs*:
                              roundup(T, 16)) are <= 256. -1 (default) = used up to 128 columns
                              unless UB_OPT_CTA_PAIR forces a tile kernel; 0 = never; 1 =
                              whenever usable */
    UB_OPT_PDL = 11,       /* 1 (default): kernels are launched with programmatic stream
                              serialization, so a kernel's launch and prologue overlap the end
                              of the kernel before it on the stream; 0: plain launches. Every
                              kernel lets the next one launch only after its own wait for the
                              grid before it, so a grid launched early finds every earlier
                              grid on the stream complete */
    UB_OPT_BULK_BESIDE = 12, /* 1: ub_allgather and ub_reduce_scatter run beside the kernel
                              issued just before them on their stream (see ub_allgather);
                              0 (default): they wait for the work before them, as any call */
    UB_OPT_GATHER_CHAIN = 13 /* when an AG call's gather is the one-launch gather kernel:
                              1 (default, with UB_OPT_PDL = 1): the kernel runs on the call's
                              stream and the GEMM is launched as its programmatic dependent,
                              starting once every gather CTA holds its SM (the chunk flags the
                              GEMM waits on are then certain to come) and completing only
                              after the gather; 0: the kernel runs on the handle's side
                              stream, forked from and joined back into the call's stream */
};

/* Operation ids for ub_kernel_time. */
enum {
    UB_OP_AG = 0,
    UB_OP_RS = 1,
    UB_OP_AG_SWIGLU = 2,
    UB_OP_AG_KN = 3,
    UB_OP_RS_KN = 4,
    UB_OP_WGRAD = 5,
    UB_OP_REDUCE_SCATTER = 6,
    UB_NUM_OPS = 7
};

/*
 * Register a user buffer at capacity [max_tokens, hidden] for tp virtual ranks
 * ([P2] "Proposed API", initialize_ub). Allocates, once, the buffer
 * (max_tokens * hidden * 2 bytes) and a small control block (tp readiness flags, an
 * abort word, a status word) on the current CUDA device, plus one side stream and two
 * events. The active shape starts at capacity. Requires max_tokens % tp == 0 so that
 * the initial active shape is itself valid. *out receives the handle.
 * Errors: UB_ERR_ARG, UB_ERR_ZERO, UB_ERR_DTYPE, UB_ERR_ALIGN, UB_ERR_DIVISIBLE,
 * UB_ERR_CUDA (no device, allocation failure).
 */
int ub_create(int64_t max_tokens, int64_t hidden, int tp, ub_dtype_t dtype, ub_handle_t *out);

/* Release everything the handle owns. Synchronises the handle's side stream. An
 * addition of this library: [P2] registers a buffer once and never releases it within
 * the run, so it names no release call. */
int ub_destroy(ub_handle_t h);

/*
 * Set the active shape [T, hidden] for the next calls ([P2] set_ub_active_shape,
 * "Implementation approach": a logical shape only -- nothing is allocated, freed or
 * re-registered, and no GPU work is issued). Constraints, checked in this order
 * ([P2] "Constrain the initial behavior"): two-dimensional (UB_ERR_RANK), nonzero
 * (UB_ERR_ZERO), T <= max_tokens (UB_ERR_CAPACITY), hidden unchanged
 * (UB_ERR_HIDDEN), T % tp == 0 (UB_ERR_DIVISIBLE). A rejected shape leaves the
 * previous active shape in place.
 */
int ub_set_active_shape(ub_handle_t h, int64_t T, int64_t hidden);
/* The same with the shape given as ndim extents (the rank is checked too). */
int ub_set_active_shape_nd(ub_handle_t h, int ndim, const int64_t *dims);

/* The same five checks without a handle: 0 or the UB_ERR_* of the first violation. */
int ub_validate_active_shape(int ndim, const int64_t *dims, int64_t max_tokens,
                             int64_t hidden, int tp);

/* Active and capacity shapes ([P2] "Proposed API": active/capacity shape getters). */
int ub_get_active_shape(ub_handle_t h, int64_t *T, int64_t *hidden);
int ub_get_capacity(ub_handle_t h, int64_t *max_tokens, int64_t *hidden);
int ub_get_tp(ub_handle_t h, int *tp);

/* Device address and byte size of the registered buffer. After ag_gemm its first T
 * rows hold the gathered input concat_r X_r (rows >= T are never touched): [P1]'s point
 * that the buffer stages the communicated activation [S, hidden]. The accessor itself is
 * an addition of this library (the pages expose the buffer only through the overlap
 * calls). */
int ub_buffer(ub_handle_t h, void **dev_ptr, size_t *bytes);

/*
 * All-gather + GEMM for the column-parallel linear ([P1] QKV / fc1 diagrams; [P3]
 * "ring_exchange" with "use_ce"): with T the active token count and c = T / tp,
 *     UB[r*c + i][:] = shards[r][i][:]            for r < tp, i < c
 *     Y[t][n]       = sum_h UB[t][h] * Wt[n][h]   for t < T, n < N.
 * shards: host array of tp device pointers, each [c, hidden]. Wt: device [N, hidden].
 * Y: device [T, N] (leading dimension N). The chunks are landed in the buffer by one of
 * three gathers (UB_OPT_GATHER_KERNEL): cudaMemcpyAsync calls on the handle's side
 * streams (the stand-in for copy-engine send/recv; on GB300 the driver runs a
 * same-device copy as a kernel on SMs, next to the GEMM, whose CTAs leave room for it),
 * each followed by a readiness-flag write; one gather kernel (default for the few-token
 * kernel, and for the tile kernels at T <= 512 or when the tiles fit one wave, so that
 * the gather's CTAs run on the SMs no tile holds), on `stream` with the GEMM launched as
 * its programmatic dependent (UB_OPT_GATHER_CHAIN) or on the side stream; or the
 * GEMM kernel's own epilogue warps before their first tile (default for tile-kernel
 * calls of more than one wave). One persistent GEMM kernel on `stream` walks the chunks in
 * ring order starting at UB_OPT_SELF_RANK (whose chunk it reads in place, without
 * waiting -- on CTA pairs, where that saves a wave, only the chunk's whole 256-row
 * tiles, its last rows from the buffer behind its flag, see ub_plan_ag_self_head),
 * waits for each other chunk's flag, and never reads or writes rows >= T.
 * Side streams are joined back into `stream` before return. A device wait that expires
 * is reported by ub_query_status (UB_ERR_TIMEOUT), never by a trap.
 * Concurrency: the GEMM kernels size their grids to be resident at once (at most one
 * CTA or CTA pair per SM) and some of their CTAs wait for others (the gather inside
 * the GEMM, split k-ranges). Calls of one handle are stream-ordered by the caller;
 * calls of this library that run at the same time on other streams must leave every
 * SM the room of one such CTA, or a wait may run out (UB_ERR_TIMEOUT, never a hang).
 * Errors: UB_ERR_ARG, UB_ERR_ZERO (N <= 0), UB_ERR_ALIGN, UB_ERR_CUDA.
 */
int ag_gemm(ub_handle_t h, const void *const *shards, const void *Wt, int64_t N, void *Y,
            void *stream);

/*
 * AG-GEMM with the SwiGLU activation fused into the epilogue: the column-parallel fc1
 * followed by the GELU/SwiGLU box of [P1]'s MLP diagram, whose output feeds fc2.
 * Wt is [2F, hidden] with the gate rows first and the up rows second (fc1's output row
 * is [gate | up]); the all-gather is the one of ag_gemm, and
 *     Z[t][f] = silu(g) * u,  g = sum_h UB[t][h] * Wt[f][h],  u = sum_h UB[t][h] * Wt[F + f][h],
 * with silu(x) = x / (1 + e^-x), evaluated in fp32 on the fp32 accumulators and rounded
 * once to BF16. Z: device [T, F]. Always runs on CTA pairs (the even CTA of a pair
 * loads 128 gate rows and the odd CTA the matching up rows of each 256-row B tile).
 * Errors: as ag_gemm; UB_ERR_ZERO (F <= 0), UB_ERR_ALIGN (F % 8 != 0).
 */
int ag_gemm_swiglu(ub_handle_t h, const void *const *shards, const void *Wt, int64_t F, void *Z,
                   void *stream);

/*
 * The same all-gather + GEMM with the weight stored in its mathematical layout,
 * W[hidden][N] row-major (the tensor core reads it MN-major):
 *     Y[t][n] = sum_h UB[t][h] * W[h][n].
 * This is also the input gradient of the row-parallel layer ([P1] MLP diagram, fc2, in
 * the backward pass): the shards are the output-gradient chunks dY_r [c, hidden] and W
 * is that layer's shard weight Bt_j [hidden, K] (N = K), giving dA_j = dS * Bt_j with dS
 * the gathered dY (left in the buffer for ub_wgrad). Always on CTA pairs.
 * Errors: as ag_gemm.
 */
int ag_gemm_kn(ub_handle_t h, const void *const *shards, const void *W, int64_t N, void *Y,
               void *stream);

/*
 * GEMM + reduce-scatter for the row-parallel linear ([P1] MLP diagram, fc2; [P2]
 * "Implementation approach": row blocks from the active first dimension):
 *     S[t][n]        = sum_{j<tp} sum_{k<K} A_j[t][k] * Bt_j[n][k]   (fp32, in TMEM)
 *     Y_shards[r][i] = bf16(S[r*c + i])                            for i < c = T / tp
 * A: host array of tp device pointers, each [T, K]. Bt: tp device pointers, each
 * [hidden, K]. Y_shards: tp device pointers, each [c, hidden]. The cross-shard sum
 * never leaves the accumulator; each rank's block is written directly, and no byte of
 * A_j beyond row T nor of Y_shards[r] beyond row c is touched.
 * Errors: UB_ERR_ARG, UB_ERR_ZERO (K <= 0), UB_ERR_ALIGN, UB_ERR_CUDA.
 */
int gemm_rs(ub_handle_t h, const void *const *A, const void *const *Bt, int64_t K,
            void *const *Y_shards, void *stream);

/*
 * The same GEMM + reduce-scatter with the shard weights stored K x hidden row-major
 * (B_j[k][n], read MN-major):  Y_shards[r][i][n] = sum_j sum_k A_j[r*c + i][k] * B_j[k][n].
 * This is also the input gradient of the column-parallel layer ([P1] QKV / fc1, in the
 * backward pass): A_j = dY_j [T, N_j] and B_j = that layer's weight shard Wt_j [N_j,
 * hidden] (K = N_j), so dX_r = rows_r of sum_j dY_j * Wt_j. Always on CTA pairs.
 * Errors: as gemm_rs.
 */
int gemm_rs_kn(ub_handle_t h, const void *const *A, const void *const *B, int64_t K,
               void *const *Y_shards, void *stream);

/*
 * An addition of this library, for the backward pass of [P1]'s two layers (the pages
 * show only the forward diagrams): the buffer still holds the communicated activation
 * after the all-gather, so the weight gradient reads it instead of gathering again.
 * Weight gradient over the active tokens, reading the gathered rows G = UB[0:T] that
 * the last ag_gemm / ag_gemm_kn / ag_gemm_swiglu of this handle left in the buffer:
 *   ub_is_a = 0:  out[m][h] = sum_{t<T} D[t][m] * G[t][h]   (out [M, hidden]: dWt of the
 *                 column-parallel layer, D = dY [T, M])
 *   ub_is_a = 1:  out[h][m] = sum_{t<T} G[t][h] * D[t][m]   (out [hidden, M]: dBt_j of
 *                 the row-parallel layer, G = the gathered dS, D = A_j [T, M])
 * fp32 accumulation over t, one BF16 rounding. Both operands are read MN-major; CTA
 * pairs. Call it on the stream of that gather (it reads the buffer without waiting).
 * Errors: UB_ERR_ARG, UB_ERR_ZERO (M <= 0), UB_ERR_ALIGN (M % 8, pointers), UB_ERR_CUDA.
 */
int ub_wgrad(ub_handle_t h, const void *D, int64_t M, int ub_is_a, void *out, void *stream);

/*
 * The "bulk" method of [P3] ("Overlap GEMM with an independent bulk all-gather or
 * reduce-scatter"): the collective alone, to run beside an unrelated GEMM (for example,
 * gather a layer's input for its weight gradient while its input-gradient GEMM runs, or
 * reduce the input-gradient partials while the weight-gradient GEMM runs).
 *
 * Two ways to run it beside the GEMM:
 *  - on a second stream (UB_OPT_BULK_BESIDE = 0). The GPU then decides which grid it
 *    places first: the GEMM first, the collective's CTAs fill the room beside the GEMM's;
 *    the collective first, its CTAs take the SMs and the two run one after the other.
 *  - beside mode (UB_OPT_BULK_BESIDE = 1): call it on the GEMM's own stream directly
 *    after the GEMM call. Its kernel is launched as a programmatic dependent of the GEMM:
 *    it starts once every GEMM CTA holds its SM, runs one CTA per SM in the room they
 *    leave, and completes only after the GEMM (it waits for it at exit), so work behind
 *    it on the stream sees both results. It does not wait for the GEMM at entry: what it
 *    reads must be complete before the GEMM starts, which holds for anything written
 *    before the GEMM on the stream when that GEMM is a call of this library (its kernels
 *    let the next grid launch only after their own wait). After a kernel of another
 *    library, which may let the next grid launch before its own predecessors finish,
 *    leave the option at 0. After a non-kernel operation (a copy, an event wait) the
 *    collective simply runs after it. The collective must not write what the GEMM reads
 *    (ub_allgather writes the user buffer: not beside an AG-GEMM of the same handle).
 *
 * ub_allgather: the all-gather of ag_gemm without the GEMM -- UB[r*c + i] = shards[r][i]
 * for the active shape, copies and readiness flags on the handle's side streams, joined
 * back into `stream` (beside mode: the gather kernel on `stream` itself). A following
 * ub_wgrad on `stream` reads the gathered rows.
 *
 * ub_reduce_scatter: Y_shards[r][i][n] = bf16(sum_{j<tp} P[j][r*c + i][n]) for the
 * active shape (P: tp device pointers [T, hidden]; Y_shards: tp pointers [c, hidden]);
 * fp32 sum in j order, one small HBM-bound kernel on `stream` whose CTAs fit beside a
 * persistent GEMM CTA (four per SM; beside mode one). Rows >= T of P and rows >= c of
 * each Y_shards[r] are untouched.
 * Errors: UB_ERR_ARG, UB_ERR_ALIGN (pointers not 16-byte aligned), UB_ERR_CUDA.
 */
int ub_allgather(ub_handle_t h, const void *const *shards, void *stream);
int ub_reduce_scatter(ub_handle_t h, const void *const *P, void *const *Y_shards, void *stream);

/*
 * An addition of this library, the column-parallel half of [P3]'s "bulk" method: the
 * all-gather is done ahead by ub_allgather, beside other work, and this call computes
 * from its result.
 * AG-GEMM over the user buffer as it stands: Y[t, :] = UB[t, :] . Wt^T for t < T (the
 * active shape), with no gather and no readiness-flag wait -- for a caller that landed
 * the chunks ahead of time with ub_allgather on this handle, for the same active shape
 * and shards, and ordered that call before this one (same stream, or an event), e.g.
 * the next microbatch's all-gather run beside the current GEMM-RS (the pages' "bulk"
 * overlap feeding the column-parallel GEMM). Nothing checks that the buffer holds the
 * chunks: an unordered or missing gather gives undefined results.
 *  - Wt: device [N, hidden] (out x in); Y: device [T, N] (rows >= T untouched).
 *  - glu_f > 0: the SwiGLU epilogue of ag_gemm_swiglu: N = 2 * glu_f (gate rows first),
 *    Y is [T, glu_f]; 0: plain.
 *  - Runs on CTA pairs, all T rows as one region (ceil(T / 256) row tiles).
 *  - Errors: UB_ERR_ARG (null pointers, bad glu_f), UB_ERR_ZERO, UB_ERR_ALIGN (N or glu_f
 *    not a multiple of 8, pointers not 16-byte aligned), UB_ERR_CUDA.
 */
int ag_gemm_from_buffer(ub_handle_t h, const void *Wt, int64_t N, int64_t glu_f, void *Y, void *stream);

/*
 * An addition of this library for measurement (the pages define no such call): read
 * `bytes` of device memory at `src` once and discard them -- one kernel on `stream`, one
 * CTA per SM, each streaming a contiguous share into shared memory with bulk copies. Its
 * time is what reading those bytes costs in one isolated kernel on this GPU (launch, ramp
 * and drain included): the floor of a few-token call, whose work is its weight read.
 *  - src: device pointer, 16-byte aligned; bytes: a multiple of 16 (0: nothing launched).
 *  - Errors: UB_ERR_ARG (null src, negative bytes), UB_ERR_ALIGN, UB_ERR_CUDA; a bounded
 *    wait that runs out is reported by ub_query_status (UB_ERR_TIMEOUT).
 */
int ub_stream_read(ub_handle_t h, const void *src, int64_t bytes, void *stream);

/* Options (UB_OPT_*). UB_ERR_ARG for an unknown key or an out-of-range value. */
int ub_set_option(ub_handle_t h, int key, int64_t val);
int ub_get_option(ub_handle_t h, int key, int64_t *val);

/*
 * Additions of this library (failure reporting of the bounded device waits; the pages
 * define none).
 * Sticky device status: UB_OK, or the first UB_ERR_* a kernel of this handle raised
 * (UB_ERR_TIMEOUT when a readiness flag or pipeline barrier wait ran out). Reads the
 * device word through the handle's side stream; call it after the stream of the
 * calls of interest has been synchronised. Returns UB_ERR_CUDA if the read fails.
 */
int ub_query_status(ub_handle_t h);
/* Reset the sticky device status to UB_OK, and the word through which a call whose wait
 * ran out stops the rest of its CTAs (stream-ordered on the side stream). A call replayed
 * from a CUDA graph keeps the epoch it was captured with, so after one replay has timed
 * out the later replays of that graph give up at once until this is called. */
int ub_clear_status(ub_handle_t h);

/* Counters of the handle: calls made, device allocations made (constant after
 * ub_create), last active T used by a GEMM call, and how the last GEMM call ran:
 * which kernel (UB_KERNEL_*), into how many k-pieces it cut a tile (the CTA-pair
 * kernel: the tiles of its last, partial wave; the few-token kernel: every weight tile;
 * 1 = whole tiles) and which all-gather fed it (a UB_OPT_GATHER_KERNEL value: 0 driver
 * copies, 1 one gather kernel, 2 inside the GEMM; -1 none, e.g. GEMM-RS). An addition
 * of this library; the pages define no counters. */
enum { UB_KERNEL_SINGLE = 0, UB_KERNEL_PAIR = 1, UB_KERNEL_FEW_TOKEN = 2 };
typedef struct {
    int64_t ag_calls;
    int64_t rs_calls;
    int64_t device_allocations;
    int64_t last_T;
    int64_t tensor_map_encodes;
    int64_t last_kernel;
    int64_t last_pieces;
    int64_t last_gather;
} ub_counters_t;
int ub_get_counters(ub_handle_t h, ub_counters_t *out);

/*
 * An addition of this library (kernel timing for the benchmark; the pages define none).
 * With UB_OPT_PROFILE = 1, every GEMM kernel launch of operation `op` (a UB_OP_* id) is
 * bracketed by CUDA events on its launch stream (up to 4096 launches are kept). This
 * call waits for the last recorded launch, returns the summed kernel time in
 * milliseconds and the launch count, and clears the record.
 */
int ub_kernel_time(ub_handle_t h, int op, double *total_ms, int64_t *launches);

/* Grid size a GEMM call of this handle launches (SM count minus the margin of [P3]'s
 * "num_sm" / "set_sm_margin"). The query is an addition of this library. */
int ub_grid_ctas(ub_handle_t h, int *ctas);

/*
 * AG-GEMM without any device allocation, for callers that cannot call cudaMalloc (code
 * running inside another framework's memory pool or a custom allocator that owns the
 * device, plugins whose allocations are audited, processes that must not grow their
 * device footprint after start-up). The paper has no counterpart to this entry point.
 *
 * Computes what ag_gemm computes for an active shape [T, hidden] split over tp
 * virtual ranks (shards: host array of tp device pointers, each [T/tp, hidden];
 * Wt: device [N, hidden]; Y: device [T, N]), with the ring starting at rank 0, using
 * the same kernel. Instead of a handle's user buffer and control block it uses one
 * file-scope device array of UB_NOALLOC_MAX_ELEMS bf16 elements (32 MiB) plus 256
 * bytes, which every GPU that loads the library holds until the process exits. It
 * calls no cudaMalloc or cudaFree and creates no stream or event: the copies of chunks
 * 1 .. tp-1 and their readiness flags are issued on `stream` itself, ahead of the kernel
 * (chunk 0 is read in place from its shard and not copied).
 *  - Every pointer and `stream` must belong to the current device: the scratch used is
 *    that device's copy of the array, and the kernel is launched there. The function
 *    cannot see the sizes behind the pointers: Y must hold T x N elements and Wt
 *    N x hidden, or the kernel reads or writes past them.
 *  - T * hidden must not exceed UB_NOALLOC_MAX_ELEMS (UB_ERR_CAPACITY otherwise);
 *    T % tp == 0 (UB_ERR_DIVISIBLE); hidden, N multiples of 8 and pointers 16-byte
 *    aligned (UB_ERR_ALIGN); 1 <= tp <= UB_MAX_TP (UB_ERR_ARG).
 *  - The first call on a device looks up the array's device address there
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - Every call on a device shares the one array, which keeps the last call's
 *    contents (the status word is cleared by each call; flags use growing epochs).
 *    Calls that overlap on the GPU -- on different streams, or from several host
 *    threads without ordering -- race on it and give undefined results.
 *  - Device-side wait timeouts are not reported by this entry point.
 */
#define UB_NOALLOC_MAX_ELEMS (16ll * 1024 * 1024)
int ag_gemm_noalloc(const void *const *shards, int tp, int64_t T, int64_t hidden, const void *Wt,
                    int64_t N, void *Y, void *stream);

/*
 * Planning queries, additions of this library (the pages define no launch planning):
 * the launch choices the library makes for a call, as pure functions of the shapes and
 * the GPU's unit counts -- no handle, no device, no CUDA call. Tools use them to predict
 * a call's launch; they are the same code the calls run.
 *
 * ub_plan_tail_split: into how many k-pieces the CTA-pair kernel cuts each tile of the
 * last, partial wave. `tiles` 256 x 256 output tiles over `pairs` CTA pairs, `k_blocks`
 * 64-wide k-blocks per tile (GEMM-RS: over all tp shards); `gathered` != 0 for an
 * AG-GEMM whose rows come through the all-gather. At most one piece per idle pair, 8
 * pieces and 16 k-blocks per piece; within that, widest != 0 (the split forced on,
 * UB_OPT_STREAMK = 1) gives the most pieces, else the cheapest cut by the fix-up cost
 * model (the longest piece plus a fixed fix-up time per added piece, fitted on GB300
 * separately for GEMM-RS and for a gathered AG-GEMM, which also needs two whole waves
 * before its last). Returns the piece count (1 = whole tiles), or UB_ERR_ARG for sizes
 * < 1.
 *
 * ub_plan_path: whether a tile-kernel call runs on CTA pairs (*pair = 1) or single CTAs
 * (*pair = 0), and whether the pairs split the last wave (*split). `single_tiles`
 * 128 x 256 tiles over `slots` SMs against `pair_tiles` 256 x 256 tiles over `pairs`
 * pairs; `cta_pair` and `streamk` as UB_OPT_CTA_PAIR and UB_OPT_STREAMK (-1: chosen by
 * the wave-count cost model; 0 / 1: forced); `gathered` as for ub_plan_tail_split.
 * Returns UB_OK, or UB_ERR_ARG for sizes < 1 or null outputs.
 *
 * ub_plan_ag_self_head: how many rows of the self chunk the CTA-pair AG kernel reads in
 * place from its shard (the rest from the user buffer, behind the chunk's readiness
 * flag): all c = T / tp rows, or only its whole 256-row tiles where that saves a wave of
 * `pairs` pairs over `n_tiles` N tiles (self: the ring's start rank). Returns the row
 * count, or UB_ERR_ARG for an invalid shape.
 *
 * ub_plan_ag_group_m: the tile order of a CTA-pair AG call: tile rows walked in groups of
 * the returned count, rows fastest inside a group (0: N fastest). Groups of 8 when the
 * first wave of `pairs` pairs reads only the self chunk's in-place rows (n_tiles N tiles
 * per tile row); else groups of one chunk's tile rows, 0 below two. Returns the count,
 * or UB_ERR_ARG for an invalid shape.
 */
int64_t ub_plan_tail_split(int64_t tiles, int64_t pairs, int64_t k_blocks, int widest, int gathered);
int ub_plan_path(int64_t single_tiles, int64_t pair_tiles, int64_t k_blocks, int64_t slots, int64_t pairs,
                 int cta_pair, int streamk, int gathered, int *pair, int *split);
int64_t ub_plan_ag_self_head(int64_t T, int tp, int self, int64_t n_tiles, int64_t pairs);
int ub_plan_ag_group_m(int64_t T, int tp, int self, int64_t n_tiles, int64_t pairs);

/*
 * ub_plan_gather_parts: the copies of an ag_gemm gather by driver copies, in issue
 * order, for tp chunks of c rows, ring start `self`, of which the CTA-pair kernel reads
 * the self chunk's first `head` rows in place (ub_plan_ag_self_head; c elsewhere).
 * Part i copies rows [row_lo[i], row_hi[i]) of chunk chunk[i] into the buffer and, when
 * flag[i] is 1, then publishes that chunk's readiness flag: the self chunk's rows from
 * `head` on (if any) first, the other chunks in ring order, then the self chunk's first
 * `head` rows (flagged only when they are the whole chunk). The gather inside the GEMM
 * copies in the same order. Outputs hold UB_MAX_TP + 1 entries. Returns the part count,
 * or UB_ERR_ARG.
 */
int ub_plan_gather_parts(int tp, int self, int64_t c, int64_t head, int *chunk, int64_t *row_lo,
                         int64_t *row_hi, int *flag);

/* Message of the last failed call on this host thread ("" if none). */
const char *ub_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* UB_H */
