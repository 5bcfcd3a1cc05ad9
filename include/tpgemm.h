/*
 * tpgemm.h - C ABI of the tile-partitioned dense GEMM library for GB300 (sm_103a)
 *
 *     D = alpha * A * B + beta * C
 *
 * A is bf16 [M, K], B is bf16 [K, N], C and D are [M, N] of the output dtype
 * (bf16 or fp32); all row-major with explicit row strides. Products are
 * accumulated in fp32 on the tensor cores; the epilogue applies alpha and beta
 * in fp32 and rounds once (round-to-nearest-even) to the output dtype.
 *
 * Sources for the operation and its conventions:
 *  - "TorchInductor ganha suporte a GEMMs de alta performance com CuteDSL":
 *    GEMMs in attention projections and fully-connected layers dominate a
 *    transformer forward pass (the paragraph on where GPU cycles go); tile
 *    sizes matched to the tensor-core pipeline, explicit shared-memory stages,
 *    warp specialisation and TMA are the design levers (same paragraph and the
 *    one on GEMM design decisions); the epilogue may load an auxiliary tensor
 *    and add it element-wise (the roadmap paragraph on epilogue fusion), which
 *    is beta * C here.
 *  - "cuTile Rust explained", "Ownership crosses the launch boundary" and "The
 *    useful boundary": the mutable output is split into disjoint tiles, each
 *    owned by exactly one tile program; inputs are shared and read-only. Here
 *    every D tile is written by exactly one CTA (or CTA pair), with no
 *    atomics. Partial sums reach global memory only in the opt-in K split of
 *    the last partial round (gemm_set_workspace); each element there is
 *    still stored once, by its owner. The small-M variant may split a
 *    panel's K range over the 2 to 4 CTAs of one cluster;
 *    the partial sums meet in distributed shared memory and the panel's owner
 *    adds them in a fixed order. So may the tiled kernel when an output has
 *    few 128 x 256 tiles: the 2 or 4 CTAs of a cluster share a tile's K range,
 *    each owns a quarter (or half) of the tile's columns, and each adds the
 *    others' partial sums of its columns in rank order before its epilogue.
 *  - Same page, "Why scoped graph capture helps borrowing": only operations
 *    that allocate nothing are safe to capture and replay. gemm_run allocates
 *    nothing and never synchronises.
 *  - "Implementing Tensor Parallelism Communication Overlays ...", "Preventing
 *    Rust Lifetime Pitfalls in Async GPU Operations": work is asynchronous on
 *    the caller's stream, so the caller keeps every buffer alive until the
 *    stream has passed the call.
 *  - Goldy "Rust Compute Kernels", "Shape contracts" and "Fusing invocations":
 *    shapes are checked before anything runs and failures are named; a written
 *    argument that overlaps another argument is rejected.
 *
 * Ownership: the caller owns A, B, C and D (device memory of the handle's
 * device). The library reads A, B, C and writes exactly the M x N elements of
 * D; bytes in the row-stride padding of D are never touched.
 *
 * Errors: every function returns a tpgemm_status. Argument errors are detected
 * on the host before anything is enqueued. A device-side timeout (a pipeline
 * wait that exceeded its limit) is recorded in the handle's status word and
 * reported by gemm_sync_status. No function aborts, exits or traps.
 *
 * Threads: gemm_run, gemm_run_epilogue, gemm_run_batched, gemm_run_grouped,
 * gemm_run_chunked and gemm_query_plan may be called on one handle from
 * several host threads at once. gemm_force_variant, gemm_set_workspace and
 * gemm_destroy must not overlap any other call on the handle.
 */
#ifndef TPGEMM_H
#define TPGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tpgemm_handle tpgemm_handle; /* opaque */

/* Output (and C) element type. */
enum tpgemm_out_dtype { TPGEMM_OUT_BF16 = 0, TPGEMM_OUT_F32 = 1 };

enum tpgemm_status {
    TPGEMM_OK = 0,
    TPGEMM_ERR_INVALID_ARG = -1,        /* null pointer, negative size, ld < extent, bad dtype */
    TPGEMM_ERR_ALIGNMENT = -2,          /* pointer or row stride in bytes not a multiple of 16 */
    TPGEMM_ERR_OVERLAP = -3,            /* D overlaps A or B, or partially overlaps C */
    TPGEMM_ERR_UNSUPPORTED_DEVICE = -4, /* device is not compute capability 10.3 */
    TPGEMM_ERR_CUDA = -5,               /* a CUDA runtime/driver call failed */
    TPGEMM_ERR_TIMEOUT = -6,            /* a device-side pipeline wait ran out (see gemm_sync_status) */
    TPGEMM_ERR_TOO_LARGE = -7           /* a dimension exceeds 2^31 - 1 */
};

/* Kernel variants, for gemm_force_variant and gemm_query_plan. */
enum tpgemm_variant {
    TPGEMM_VARIANT_AUTO = 0,   /* M <= 64: streaming; M <= 128: tiled; otherwise tiled pair */
    TPGEMM_VARIANT_TILED = 1,  /* persistent warp-specialised tcgen05 kernel, 128x256 tiles per CTA */
    TPGEMM_VARIANT_STREAM = 2, /* small-M weight-streaming kernel (swapped operands) */
    TPGEMM_VARIANT_EPILOGUE_ONLY = 3, /* K == 0: D = beta * C */
    TPGEMM_VARIANT_TILED_PAIR = 4 /* the tiled kernel on CTA pairs: 256x256 tiles, cta_group::2 MMA */
};

/* Activation of the fused epilogue. */
enum tpgemm_activation {
    TPGEMM_ACT_NONE = 0,
    TPGEMM_ACT_RELU = 1,    /* max(v, 0) */
    TPGEMM_ACT_SIGMOID = 2, /* 1 / (1 + exp(-v)) */
    TPGEMM_ACT_TANH = 3     /* tanh(v) */
};

/*
 * Fused epilogue: the element-wise work that follows a GEMM in a transformer
 * layer, done on the accumulator before the single rounding to the output
 * type, instead of in separate kernels that re-read D ("TorchInductor ganha
 * suporte a GEMMs de alta performance com CuteDSL", epilogue-fusion roadmap
 * paragraph: auxiliary tensor loads, element-wise add and mul, ReLU,
 * sigmoid, tanh). Per element, in fp32:
 *     v = alpha * acc + beta * C[m,n]
 *     v = v + bias[n]              (if bias != NULL)
 *     v = activation(v)
 *     v = v * aux[m,n]             (if aux != NULL)
 *     D[m,n] = round(v)
 * bias: N values of bias_dtype (TPGEMM_OUT_BF16 or TPGEMM_OUT_F32), 16-byte
 * aligned. aux: [M, N] of the output dtype, row stride ldaux >= N, 16-byte
 * aligned with ldaux * element size a multiple of 16; it may be D itself
 * (same stride) but may not otherwise overlap D. Both are read-only.
 */
typedef struct tpgemm_epilogue {
    const void *bias;
    int bias_dtype;
    int activation;
    const void *aux;
    int64_t ldaux;
} tpgemm_epilogue;

/*
 * Creates a handle for CUDA device `device`. Checks that the device is
 * compute capability 10.3, reads its SM count, resolves the driver's
 * tensor-map encoder, sets the kernels' shared-memory limits and allocates
 * the 8-byte device status word (the only allocation the library makes).
 * *out is set to NULL on failure. Not called on a hot path.
 * Everything that allocates or queries the device happens here, once, so
 * that the calls made per GEMM allocate nothing and can be captured into a
 * graph and replayed ("cuTile Rust explained", "Why scoped graph capture
 * helps borrowing": only operations that allocate nothing are safe to
 * capture). The handle owns its status word; the caller owns the handle.
 */
int gemm_create(tpgemm_handle **out, int device);

/*
 * Enqueues D = alpha*A*B + beta*C on `stream` (a cudaStream_t; NULL is the
 * legacy default stream) and returns without synchronising.
 *   M, N, K     >= 0, each <= 2^31 - 1.
 *   A, lda      bf16, row-major [M, K], lda >= K (elements).
 *   B, ldb      bf16, row-major [K, N], ldb >= N.
 *   C, ldc      out_dtype, row-major [M, N], ldc >= N. Not read when beta == 0,
 *               and may then be NULL.
 *   D, ldd      out_dtype, row-major [M, N], ldd >= N.
 *   out_dtype   TPGEMM_OUT_BF16 or TPGEMM_OUT_F32.
 * All non-NULL pointers must be 16-byte aligned and every row stride times
 * the element size a multiple of 16 bytes (TMA requirements); a stride of a
 * matrix with one row is not checked. M == 0 or N == 0 enqueues nothing;
 * K == 0 gives D = beta*C (zeros when beta == 0).
 * D == C with ldd == ldc (in place) is allowed; any other overlap of D with
 * A, B or C is TPGEMM_ERR_OVERLAP. Argument errors enqueue nothing. Launch
 * failures return TPGEMM_ERR_CUDA. Allocates nothing, so it may be captured
 * into a CUDA graph. Calls on different streams may run concurrently, unless
 * the handle has a workspace (gemm_set_workspace).
 */
int gemm_run(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
             const void *B, int64_t ldb, const void *C, int64_t ldc, void *D, int64_t ldd,
             float alpha, float beta, int out_dtype, void *stream);

/*
 * gemm_run with a fused epilogue (see tpgemm_epilogue). epi == NULL is exactly
 * gemm_run. Extra argument errors: TPGEMM_ERR_INVALID_ARG for a bad
 * activation or bias dtype or ldaux < N, TPGEMM_ERR_ALIGNMENT for a misaligned
 * bias, aux or ldaux, TPGEMM_ERR_OVERLAP when bias overlaps D or aux partially
 * overlaps D. Like gemm_run it allocates nothing and never synchronises.
 */
int gemm_run_epilogue(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, const void *A,
                      int64_t lda, const void *B, int64_t ldb, const void *C, int64_t ldc,
                      void *D, int64_t ldd, float alpha, float beta, int out_dtype,
                      const tpgemm_epilogue *epi, void *stream);

/*
 * Batched GEMM ("TorchInductor ganha suporte a GEMMs de alta performance com
 * CuteDSL", the enablement paragraph: NVGEMM covers mm, bmm, scaled_mm and
 * grouped_mm). For b in [0, batch):
 *     D_b = alpha * A_b * B_b + beta * C_b,   X_b = X + b * strideX (elements)
 * with every slice laid out as in gemm_run. A stride of 0 shares one slice of
 * A, B or C between all batches (e.g. one weight for every batch); D's slices
 * must not overlap (strideD >= (M-1)*ldd + N when batch > 1). Strides times
 * the element size must be multiples of 16 bytes. Runs the tiled kernel over
 * all batches' tiles in one launch. batch == 0 enqueues nothing.
 * Errors as gemm_run; overlap is checked over all slices.
 */
int gemm_run_batched(tpgemm_handle *h, int64_t batch, int64_t M, int64_t N, int64_t K,
                     const void *A, int64_t lda, int64_t strideA, const void *B, int64_t ldb,
                     int64_t strideB, const void *C, int64_t ldc, int64_t strideC, void *D,
                     int64_t ldd, int64_t strideD, float alpha, float beta, int out_dtype,
                     void *stream);

/* Most groups gemm_run_grouped takes. */
#define TPGEMM_MAX_GROUPS 256

/*
 * Grouped GEMM (grouped_mm of the same paragraph), as in a mixture-of-experts
 * layer: group g owns rows [r_g, r_g + group_rows[g]) of A [R, K], C and D
 * [R, N], stacked in group order (r_0 = 0, r_{g+1} = r_g + group_rows[g],
 * R = sum of group_rows), and its own weight B_g = B + g * strideB, a [K, N]
 * matrix with row stride ldb:
 *     D[r_g + i, :] = alpha * A[r_g + i, :] * B_g + beta * C[r_g + i, :]
 * group_rows is a host array of `groups` non-negative counts (empty groups are
 * allowed); groups <= TPGEMM_MAX_GROUPS. Every output row belongs to exactly
 * one group and is written by exactly one CTA. Layout, alignment and error
 * rules as gemm_run (strideB * 2 a multiple of 16 bytes when groups > 1).
 */
int gemm_run_grouped(tpgemm_handle *h, int64_t groups, const int64_t *group_rows, int64_t N,
                     int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
                     int64_t strideB, const void *C, int64_t ldc, void *D, int64_t ldd, float alpha,
                     float beta, int out_dtype, void *stream);

/*
 * M-chunked GEMM for overlapping a GEMM with the collective that consumes it
 * ("Implementing Tensor Parallelism Communication Overlays ...", "Pipelining
 * GEMM and Collectives: The Core Overlay Loop"): the rows of D are cut into
 * `chunks` consecutive chunks; for each chunk i the chunk's GEMM (the same
 * D = alpha*A*B + beta*C on its rows) is enqueued on `stream` and then
 * events[i] is recorded on `stream`. A communication stream can wait on
 * events[i] and start the collective on chunk i's rows of D while chunk i+1
 * is computed ("Performance Tradeoffs": more chunks expose more overlap but
 * make each GEMM smaller).
 *   chunks    1 .. 64.
 *   events    `chunks` cudaEvent_t handles created by the caller (with or
 *             without timing), all non-NULL; the library only records them.
 * Chunk boundaries are multiples of 128 rows: chunk i covers rows
 * [b_i, b_{i+1}) with b_i = floor(i*M/chunks / 128) * 128 (b_chunks = M); a
 * chunk may be empty, and its event is still recorded. Other arguments, rules
 * and errors as gemm_run. Allocates nothing and never synchronises.
 */
int gemm_run_chunked(tpgemm_handle *h, int chunks, int64_t M, int64_t N, int64_t K,
                     const void *A, int64_t lda, const void *B, int64_t ldb, const void *C,
                     int64_t ldc, void *D, int64_t ldd, float alpha, float beta, int out_dtype,
                     void *const *events, void *stream);

/*
 * Synchronises `stream`, then reads and clears the handle's device status
 * word. Returns TPGEMM_OK, TPGEMM_ERR_TIMEOUT if any kernel since the last
 * call gave up on a pipeline wait (its output is then incomplete), or
 * TPGEMM_ERR_CUDA if the synchronisation failed. A wait that cannot finish
 * must end in a reported error rather than a hang, and the error must reach
 * the host so that the caller can recover ("Implementing Tensor Parallelism
 * Communication Overlays ...", "Real-world Failure Modes: Deadlocks,
 * Timeouts, and Error Recovery"): every pipeline wait in the kernels has a
 * time limit, and this call is where its expiry is read.
 */
int gemm_sync_status(tpgemm_handle *h, void *stream);

/*
 * The argument checks of gemm_run on their own: returns the status gemm_run
 * would return for these arguments before launching anything (TPGEMM_OK when
 * they are acceptable). Needs no handle, no GPU and no valid memory: the
 * pointers are only compared and tested for alignment, never dereferenced.
 */
int gemm_check_args(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                    int64_t ldb, const void *C, int64_t ldc, const void *D, int64_t ldd, float beta,
                    int out_dtype);

/*
 * Frees the handle and its status word. NULL is accepted. Work is
 * asynchronous, so the handle (like every buffer a call reads or writes)
 * must outlive the calls enqueued with it: destroy it only after the streams
 * of those calls have passed them ("Implementing Tensor Parallelism
 * Communication Overlays ...", "Preventing Rust Lifetime Pitfalls in Async
 * GPU Operations").
 */
int gemm_destroy(tpgemm_handle *h);

/* Static, human-readable name of a tpgemm_status value. */
const char *gemm_status_string(int status);

/*
 * Forces a kernel variant for later gemm_run calls on this handle
 * (TPGEMM_VARIANT_AUTO restores the default choice). TILED, TILED_PAIR and
 * STREAM are accepted for any K >= 1; STREAM is used only when M <= 64 (larger
 * M falls back to TILED). Not thread-safe with concurrent gemm_run calls on
 * the same handle.
 */
int gemm_force_variant(tpgemm_handle *h, int variant);

/*
 * Reports what gemm_run would launch for this problem, without launching:
 * the variant, the output tile (rows x cols of D), the number of tiles, the
 * grid size in CTAs, the cluster size (2 for CTA pairs; for the streaming
 * variant the number of CTAs that share a panel's K range, 1 to 4; for 1-CTA
 * tiles the number that share a tile's K range, 1, 2 or 4), the
 * dynamic shared memory per CTA and the number of kernel launches. Any output
 * pointer may be NULL.
 */
int gemm_query_plan(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, int out_dtype,
                    int *variant, int *tile_m, int *tile_n, int64_t *num_tiles, int *grid,
                    int *cluster, int *smem_bytes, int *launches);

/*
 * Host copy of the persistent tile scheduler. For an mt x nt grid of output
 * tiles (256 columns wide; 128 rows, or 256 rows when pair != 0) and at most
 * `cap` persistent workers (CTAs, or CTA pairs), gemm_schedule_workers returns
 * how many workers the tiled kernels launch, and gemm_schedule_tiles writes
 * the work items of worker `worker`, in order, as triples out[3*i .. 3*i+2] =
 * (tile row, first column, width in columns) for i < cap_items, with the
 * grouped raster's band height set to group_m; it returns how many items that
 * worker owns (0 for a worker past the last; TPGEMM_ERR_INVALID_ARG on bad
 * arguments). With allow_split, the tiles of a nearly empty last round (or all
 * tiles, when there are fewer than workers) are cut into 2 or 4 column pieces
 * (2 at most for pairs) when that shortens the estimated time. The kernels run
 * the same functions, so this is what the partition tests check. No GPU is
 * needed.
 */
int gemm_schedule_workers(int64_t mt, int64_t nt, int cap, int pair, int allow_split);

/*
 * Host copy of the streaming variant's K-split choice. For nt panels of 128
 * columns, kb K blocks of 64 and mt_pad token rows (16, 32, 48 or 64),
 * returns the number s of CTAs (1..4) of a cluster that share each panel's K
 * range: the s with the least rounds(s) / s * (1 + 0.02 (s - 1)), rounds(s)
 * being the panels over the clusters of s CTAs that fit at once. s = 1 runs on
 * num_sms CTAs; clusters[s - 2] (three entries, s = 2..4) gives the clusters of
 * s CTAs the occupancy API reports (0: not possible). s is also limited to kb
 * and to splits whose reduction slots leave a ring of at least 4 stages.
 * gemm_run computes the cluster counts on the device and calls the same
 * function. Returns TPGEMM_ERR_INVALID_ARG on bad arguments. No GPU is needed.
 */
int gemm_stream_split(int64_t nt, int64_t kb, int mt_pad, int num_sms, const int *clusters);

/*
 * Host copy of the tiled kernel's K-split choice, made before the choice
 * between 1-CTA tiles and CTA pairs. For `tiles` 128 x 256 output tiles of kb
 * K blocks of 64, returns 4 when kb >= 4 and every tile gets a cluster of four
 * CTAs at once (tiles <= cap4, the clusters of four the occupancy API
 * reports), else 2 when kb >= 2 and tiles <= cap2, else 1: no split, the
 * persistent schedule of gemm_schedule_tiles. gemm_run and gemm_run_noalloc
 * call the same function (gemm_run only when no variant is forced). Returns
 * TPGEMM_ERR_INVALID_ARG on bad arguments. No GPU is needed.
 */
int gemm_tiled_ksplit(int64_t tiles, int64_t kb, int cap2, int cap4);
int64_t gemm_schedule_tiles(int64_t mt, int64_t nt, int group_m, int cap, int pair, int allow_split, int worker,
                            int32_t *out, int64_t cap_items);

/*
 * Watchdog self-test: launches one CTA that waits on a barrier no thread will
 * ever arrive at, with a limit of `timeout_ns` nanoseconds (1 us .. 1 s), then
 * synchronises `stream`. Returns TPGEMM_ERR_TIMEOUT when the wait ran out as
 * designed and the context is still usable, TPGEMM_OK if it (wrongly) did not
 * run out, or TPGEMM_ERR_CUDA. Leaves the handle's status word clear.
 */
int gemm_watchdog_selftest(tpgemm_handle *h, uint64_t timeout_ns, void *stream);

/* Number of SMs the handle schedules over, or a negative status. */
int gemm_num_sms(tpgemm_handle *h);

/*
 * Optional workspace for the K split of the last partial round of the CTA-pair
 * kernel. The persistent schedule gives every pair the same number of whole
 * 256 x 256 tiles; the tiles left over for a last, partial round are cut in
 * two pieces so that more pairs share them ("cuTile Rust explained",
 * "Ownership crosses the launch boundary": each piece keeps an exclusive
 * column half of its tile). Without a workspace a piece is a column half that
 * runs over all of K, and it costs about as long as a whole tile. With one,
 * and K of at least 2048, a piece runs over half of K and the full tile
 * width; the two pairs of a tile trade their fp32 partial sums of each
 * other's column half through the workspace and each adds the other's part
 * before its epilogue, so a piece takes about half as long. Each output element is still stored by one CTA,
 * with no atomics, and the sum of two fp32 parts does not depend on their
 * order, so results are the same on every run.
 *   ws, bytes   device memory of the handle's device, 256-byte aligned;
 *               bytes >= gemm_workspace_size(h) covers every shape (a smaller
 *               workspace covers the shapes whose tail fits, others run
 *               without the split). ws == NULL detaches the workspace (bytes
 *               is then ignored) and restores the behaviour without one.
 *   stream      the workspace's flags are cleared on this stream; enqueue the
 *               calls that use it after that point.
 * Co-residency: the two pairs that share a tail tile wait for each other's
 * partial sums, so the split assumes every CTA pair of the launch is resident
 * at once. The grid is sized to the number of CTA pairs the occupancy API
 * reports for the whole device, so that holds when the GPU runs this launch
 * alone or beside kernels that leave it room. Where fewer SMs are available
 * than the device reports (an MPS client limited to part of the GPU, a green
 * context, kernels on other streams holding SMs for a long time), a pair may
 * wait for a partner that cannot start until it exits: the wait then runs out
 * after the handle's time limit and gemm_sync_status reports
 * TPGEMM_ERR_TIMEOUT with the output incomplete. Such callers detach the
 * workspace (ws == NULL), which restores the plan without waits between
 * pairs.
 * Ownership stays with the caller: keep the memory allocated, and do not
 * touch it, until it is detached and every call that used it has finished.
 * Each call uses the whole workspace, so while one is attached, calls on the
 * handle must not overlap on the GPU: issue them on one stream, or order
 * them with events; two replays of a captured graph that contains such calls
 * must not overlap either. A call whose workspace wait ran out
 * (TPGEMM_ERR_TIMEOUT in gemm_sync_status) may leave stale flags: call
 * gemm_set_workspace again before the next call. Only gemm_run,
 * gemm_run_epilogue and gemm_run_chunked use it. TPGEMM_ERR_INVALID_ARG for a
 * null handle or bytes below one tail tile's need, TPGEMM_ERR_ALIGNMENT for a
 * misaligned ws, TPGEMM_ERR_CUDA if the clearing memset fails to enqueue; a
 * call whose operands overlap the part of the workspace it would use returns
 * TPGEMM_ERR_OVERLAP.
 */
int gemm_set_workspace(tpgemm_handle *h, void *ws, int64_t bytes, void *stream);

/* Workspace bytes that cover every shape on the handle's device, or a negative status. */
int64_t gemm_workspace_size(tpgemm_handle *h);

/*
 * 1 if gemm_run would split the last partial round over K for this problem
 * (CTA-pair plan, a tail of column halves, K >= 2048 and a large enough
 * workspace attached), 0 if not, or a negative status.
 */
int gemm_plan_tail_ksplit(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, int out_dtype);

/*
 * Host copies of the K split tail's rules (no GPU needed). gemm_tail_ksplit
 * returns 1 when a CTA-pair schedule whose left-over tiles are cut into
 * `split` column pieces (the split only applies to halves, split == 2), with
 * kb K blocks of 64 and `tail_tiles` left-over tiles, is split over K with a
 * workspace of ws_bytes bytes: kb >= 32 and ws_bytes >=
 * gemm_tail_workspace_bytes(tail_tiles); else 0. gemm_tail_workspace_bytes
 * is 4096 bytes of flags plus four 64 KB slots per left-over tile. gemm_run
 * calls the same rule. TPGEMM_ERR_INVALID_ARG on bad arguments.
 */
int gemm_tail_ksplit(int split, int64_t kb, int64_t tail_tiles, int64_t ws_bytes);
int64_t gemm_tail_workspace_bytes(int64_t tail_tiles);

/* FP8 element formats of the block-scaled GEMM (OCP Microscaling v1.0). */
enum tpgemm_fp8_format {
    TPGEMM_FP8_E4M3 = 0, /* bias 7, no infinities, largest finite 448 */
    TPGEMM_FP8_E5M2 = 1  /* bias 15, IEEE-style infinities and NaNs, largest finite 57344 */
};

/*
 * Block-scaled GEMM, MXFP8 (scaled_mm): "TorchInductor ganha suporte a GEMMs de
 * alta performance com CuteDSL" lists scaled_mm among the GEMMs its backend
 * covers (the enablement paragraph) and reports MXFP8 results (the results
 * paragraph). The page defines no format; the formats are those of the OCP
 * Microscaling (MX) v1.0 specification: every 32 consecutive elements along K
 * share one E8M0 scale (2^(e - 127), e = 255 is NaN), per row of A and per
 * column of B. With A_b, B_b the b-th 32-wide K block:
 *     D = alpha * sum_b (SA[:, b] SB[:, b]^T) .* (A_b * B_b) + beta * C
 * accumulated in fp32 on the tensor cores (tcgen05.mma kind::mxf8f6f4 applies
 * the scales), then alpha, beta*C and one rounding as in gemm_run.
 *   M, N, K     >= 0, each <= 2^31 - 1; K a multiple of 32.
 *   A, lda      FP8 codes (a_format), row-major [M, K], lda >= K bytes, a
 *               multiple of 16 (not checked for M == 1).
 *   B, ldb      FP8 codes (b_format) of B TRANSPOSED: row-major [N, K] (B in
 *               column-major order, as fp8 scaled_mm takes it), ldb >= K
 *               bytes, a multiple of 16 (not checked for N == 1).
 *   SA, SB      E8M0 scale codes of A's M rows and B's N columns, each in the
 *               blocked layout: 512-byte chunks of 128 rows x 4 scale columns,
 *               chunk (row block rb, column block cb) at byte
 *               (rb * ceil(K/128) + cb) * 512, and inside it the scale of row
 *               r, scale column c at byte (r % 32) * 16 + (r / 32) * 4 + c;
 *               gemm_mx_scale_bytes(M, K) and (N, K) bytes, 16-byte aligned.
 *               This is the layout NVIDIA's libraries take for MX scales, so
 *               scales prepared for them can be passed as they are. Bytes of
 *               rows past M (N) or scale columns past K/32 are read and must
 *               hold finite scales (any code but 255; zero is fine).
 *   C, ldc, D, ldd, alpha, beta, out_dtype   as gemm_run.
 * K == 0 gives D = beta*C. D may equal C (same stride); any other overlap of
 * D with A, B, SA, SB or C is TPGEMM_ERR_OVERLAP. Errors as gemm_run, plus
 * TPGEMM_ERR_INVALID_ARG for a bad format or K not a multiple of 32.
 * Allocates nothing and never synchronises. Runs a persistent kernel of
 * 256 x 256 tiles on CTA pairs when M and N are both above 128, else of
 * 128 x 192 tiles on single CTAs (128 x 128 when N <= 128).
 */
int gemm_run_mx(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, int a_format,
                const void *SA, const void *B, int64_t ldb, int b_format, const void *SB, const void *C,
                int64_t ldc, void *D, int64_t ldd, float alpha, float beta, int out_dtype, void *stream);

/* Bytes of one operand's scales in gemm_run_mx's blocked layout:
 * ceil(rows / 128) * ceil(K / 128) * 512; TPGEMM_ERR_INVALID_ARG for negative sizes. */
int64_t gemm_mx_scale_bytes(int64_t rows, int64_t K);

/* The argument checks of gemm_run_mx alone (no handle, no GPU; pointers are
 * only compared and tested for alignment). */
int gemm_mx_check_args(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, int a_format, const void *SA,
                       const void *B, int64_t ldb, int b_format, const void *SB, const void *C, int64_t ldc,
                       const void *D, int64_t ldd, float beta, int out_dtype);

/* What gemm_run_mx launches for this shape: tile rows and columns, tiles, grid
 * (CTAs, one per SM at most), cluster size (2 for CTA pairs) and dynamic
 * shared memory per CTA. Any output pointer may be NULL. */
int gemm_mx_query_plan(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, int out_dtype, int *tile_m, int *tile_n,
                       int64_t *num_tiles, int *grid, int *cluster, int *smem_bytes);

/* FP4 formats of the block-scaled GEMM (gemm_run_fp4). */
enum tpgemm_fp4_format {
    TPGEMM_NVFP4 = 0, /* E2M1 elements, one E4M3 scale per 16 elements along K */
    TPGEMM_MXFP4 = 1  /* E2M1 elements, one E8M0 scale per 32 elements along K (OCP MX) */
};

/*
 * Block-scaled GEMM, FP4 (scaled_mm): "TorchInductor ganha suporte a GEMMs de
 * alta performance com CuteDSL" names NVFP4 and MXF4 GEMMs among those its
 * backend covers (the enablement paragraph) and reports NVFP4 results on
 * decode shapes (the results paragraph). The page defines no format; read as:
 * an element is E2M1 (OCP MX v1.0: sign, two exponent bits with bias 1, one
 * mantissa bit; the values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives),
 * two to a byte with the even-numbered element (along K) in the low four
 * bits. NVFP4 gives every 16 consecutive elements along K one E4M3 scale
 * (unsigned: the sign bit must be clear); its per-tensor fp32 scale is the
 * caller's alpha. MXFP4 gives every 32 one E8M0 scale (2^(e - 127)). With
 * A_b, B_b the b-th block of K:
 *     D = alpha * sum_b (SA[:, b] SB[:, b]^T) .* (A_b * B_b) + beta * C
 * accumulated in fp32 on the tensor cores (tcgen05.mma kind::mxf4nvf4 applies
 * the scales), then alpha, beta*C and one rounding as in gemm_run.
 *   M, N, K     >= 0, each <= 2^31 - 1; K a multiple of 16 (NVFP4) or 32
 *               (MXFP4).
 *   format      TPGEMM_NVFP4 or TPGEMM_MXFP4.
 *   A, lda      packed E2M1 codes, row-major [M, K/2] bytes; lda is the row
 *               stride in BYTES, >= K/2, a multiple of 16 (not checked for
 *               M == 1).
 *   B, ldb      packed E2M1 codes of B TRANSPOSED: row-major [N, K/2] bytes,
 *               ldb >= K/2 bytes, a multiple of 16 (not checked for N == 1).
 *   SA, SB      scale codes of A's M rows and B's N columns (E4M3 for NVFP4,
 *               E8M0 for MXFP4) in the blocked layout of gemm_run_mx: 512-byte
 *               chunks of 128 rows x 4 scale columns, chunk (row block rb,
 *               column block cb) at byte (rb * ceil(K/(4*block)) + cb) * 512
 *               (block = 16 or 32), inside it the scale of row r, scale column
 *               c at byte (r % 32) * 16 + (r / 32) * 4 + c;
 *               gemm_fp4_scale_bytes(format, M, K) and (format, N, K) bytes,
 *               16-byte aligned. Bytes of rows past M (N) or of scale columns
 *               past K/block are read and must hold finite scales (not 0x7F
 *               or 0xFF for E4M3, not 255 for E8M0; zero is fine).
 *   C, ldc, D, ldd, alpha, beta, out_dtype   as gemm_run.
 * K == 0 gives D = beta*C. D may equal C (same stride); any other overlap of
 * D with A, B, SA, SB or C is TPGEMM_ERR_OVERLAP. Errors as gemm_run, plus
 * TPGEMM_ERR_INVALID_ARG for a bad format or K not a multiple of the block.
 * Allocates nothing and never synchronises. Runs a persistent kernel of
 * 256 x 256 tiles on CTA pairs when M and N are both above 128, else of
 * 128 x 128 tiles on single CTAs.
 */
int gemm_run_fp4(tpgemm_handle *h, int64_t M, int64_t N, int64_t K, int format, const void *A, int64_t lda,
                 const void *SA, const void *B, int64_t ldb, const void *SB, const void *C, int64_t ldc, void *D,
                 int64_t ldd, float alpha, float beta, int out_dtype, void *stream);

/* Bytes of one operand's scales in gemm_run_fp4's blocked layout:
 * ceil(rows / 128) * ceil(K / (4 * block)) * 512, block = 16 (NVFP4) or 32
 * (MXFP4); TPGEMM_ERR_INVALID_ARG for a bad format or negative sizes. */
int64_t gemm_fp4_scale_bytes(int format, int64_t rows, int64_t K);

/* The argument checks of gemm_run_fp4 alone (no handle, no GPU; pointers are
 * only compared and tested for alignment). */
int gemm_fp4_check_args(int64_t M, int64_t N, int64_t K, int format, const void *A, int64_t lda, const void *SA,
                        const void *B, int64_t ldb, const void *SB, const void *C, int64_t ldc, const void *D,
                        int64_t ldd, float beta, int out_dtype);

/* What gemm_run_fp4 launches for this shape, as gemm_mx_query_plan. */
int gemm_fp4_query_plan(tpgemm_handle *h, int format, int64_t M, int64_t N, int64_t K, int out_dtype, int *tile_m,
                        int *tile_n, int64_t *num_tiles, int *grid, int *cluster, int *smem_bytes);

/*
 * Allocation-free GEMM (no counterpart in the paper; it serves callers that
 * cannot allocate device memory). Some callers cannot call cudaMalloc: code
 * whose device memory must all come from a pool or arena owned by an outer
 * framework, and serving loops that forbid allocation after warm-up, where an
 * allocation can stall on the driver, fragment the pool or break a stream
 * capture in progress. gemm_create allocates (the handle's status word), so
 * such callers use this entry point instead. It needs no handle and runs on the
 * current device.
 *
 * Computes the same D = alpha*A*B + beta*C as gemm_run, with the same
 * arguments, layouts, alignment, aliasing and error rules, always with the
 * tiled kernel (K == 0 runs the D = beta*C kernel). The kernel's scratch, its
 * 4-byte status word, lives in a file-scope device array of 16 bytes (the
 * stated maximum) that every GPU that loads this library holds until the
 * process exits; the scratch needed does not grow with M, N or K, and sizes
 * beyond the library's limit (any dimension above 2^31 - 1) are rejected with
 * TPGEMM_ERR_TOO_LARGE. The caller still passes and owns A, B, C and D.
 * Nothing here calls cudaMalloc, cudaFree or any allocating library routine.
 *
 * The first call on a device does that device's one-time set-up (it looks up
 * the array's device address, resolves the tensor-map encoder, sets the
 * kernel's shared-memory limit and clears the array, synchronously); make
 * that first call before any stream capture. Every call shares the array and
 * it keeps the last call's contents: each call clears the status word on
 * `stream` before its launch, so calls that overlap on the GPU (on different
 * streams) race on it.
 *
 * check_status == 0: enqueue and return (launch errors only).
 * check_status != 0: also synchronise `stream`, read and clear the status
 * word, and return TPGEMM_ERR_TIMEOUT if a pipeline wait ran out.
 */
int gemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                     const void *B, int64_t ldb, const void *C, int64_t ldc, void *D,
                     int64_t ldd, float alpha, float beta, int out_dtype, void *stream,
                     int check_status);

#ifdef __cplusplus
}
#endif

#endif /* TPGEMM_H */
