/*
 * gemm_tcgen05.h -- C ABI of a dense GEMM library for NVIDIA GB300 (sm_103a).
 *
 *     C <- alpha * A * B + beta * C
 *
 * A is M x K, B is K x N, C is M x N; inputs fp16 or bf16, products accumulated
 * in fp32 by the fifth-generation tensor core (tcgen05, accumulator in Tensor
 * Memory), output fp32, bf16 or fp16.  The operation is the GEMM of "GEMM From
 * Naive CUDA to Tensor Cores" (leetllm.com/learn/gemm-naive-cuda-tensor-cores),
 * opening section: shapes [M,K] x [K,N] = [M,N], C <- alpha*AB + beta*C, and
 * with beta = 0 the old output is not read.  FLOPs are counted as 2*M*N*K
 * (same page, "Compute one output before launching a warp").
 *
 * Conventions for every entry point:
 *  - Pointers named A, B, C are DEVICE pointers of the current CUDA device,
 *    owned by the caller; the library never frees or retains them.  A and B are
 *    only read.  C is read (only when beta != 0) and written in place.
 *  - All work is enqueued on `stream` (a cudaStream_t passed as void*, NULL =
 *    legacy default stream) and the call returns without synchronising.  A fault
 *    inside the kernel surfaces at the caller's next synchronisation, and a
 *    timed-out internal wait through gemm_sync_status().
 *  - Sizes and leading dimensions are in ELEMENTS; leading dimensions are the
 *    distance between consecutive rows of the stored (row-major) array.
 *  - Thread safety: calls from several host threads are safe; the debug knobs
 *    (gemm_debug_set) are process-wide.
 *  - Status codes are returned; nothing is printed and nothing aborts.
 */
#ifndef GEMM_TCGEN05_H
#define GEMM_TCGEN05_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element formats. */
typedef enum {
  GEMM_F16 = 0,  /* IEEE binary16 */
  GEMM_BF16 = 1, /* bfloat16 (8-bit exponent, 7-bit mantissa) */
  GEMM_F32 = 2,  /* IEEE binary32 (output only) */
  GEMM_E4M3 = 3, /* OCP FP8 E4M3 (4-bit exponent, bias 7, 3-bit mantissa, no
                    infinities, max 448; input only) */
  GEMM_E5M2 = 4  /* OCP FP8 E5M2 (5-bit exponent, bias 15, 2-bit mantissa; input
                    only).  FP8 is the variant "A dense FP16 matrix-multiply kernel
                    for NVIDIA Ada" lists as written but untested; here the tensor
                    core multiplies it with tcgen05.mma kind::f8f6f4, fp32
                    accumulation.  FP8 operands must be K-major: layout
                    GEMM_A_ROW | GEMM_B_COL (other layouts: GEMM_ERR_UNSUPPORTED),
                    and lda, ldb multiples of 16 elements. */
} gemm_dtype_t;

/* Storage order of A and B (bit mask, OR one A flag with one B flag).  C is
 * always row-major [M, N] with ldc >= N.  "Layout is part of the type" (leetllm
 * page, section of that name): the flags say how memory is read; they never
 * transpose data.
 *   GEMM_A_ROW  A stored [M, K] row-major, lda >= K   (K-major)
 *   GEMM_A_COL  A stored [K, M] row-major (A column-major), lda >= M (M-major)
 *   GEMM_B_ROW  B stored [K, N] row-major, ldb >= N   (N-major)
 *   GEMM_B_COL  B stored [N, K] row-major (B column-major), ldb >= K (K-major;
 *               the A-row/B-col pairing is the "TN" layout of the Ada GEMM page,
 *               kd.iw.mk, that makes both operand copies identical) */
enum { GEMM_A_ROW = 0, GEMM_A_COL = 1, GEMM_B_ROW = 0, GEMM_B_COL = 2 };

typedef enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_ARG = 1, /* negative size, ld below its minimum, NULL operand
                               that would be read or written, size overflow */
  GEMM_ERR_UNSUPPORTED = 2, /* dtype not supported, pointer not 16-byte aligned,
                               ld * element size not a multiple of 16 bytes
                               (the tensor-copy engine's stride rule), a
                               dimension >= 2^31 */
  GEMM_ERR_ARCH = 3,        /* current device is not compute capability 10.3 */
  GEMM_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (no device,
                               launch failure, tensor-map encoding failure) */
  GEMM_ERR_TIMEOUT = 5,     /* a kernel wait gave up (see gemm_sync_status) */
  GEMM_ERR_SCRATCH = 6      /* gemm_ex_noalloc only: the launch needs more scratch
                               than its fixed buffer holds */
} gemm_status_t;

/*
 * gemm -- C <- alpha * A * B + beta * C on the current device.
 *
 * in_dtype  : GEMM_F16, GEMM_BF16, GEMM_E4M3 or GEMM_E5M2 (A and B share it).
 * out_dtype : GEMM_F32, GEMM_BF16 or GEMM_F16 (C in and C out share it).
 * layout    : GEMM_A_ROW|GEMM_A_COL combined with GEMM_B_ROW|GEMM_B_COL.
 * Requirements: A, B, C 16-byte aligned; lda*sizeof(in), ldb*sizeof(in) and
 * ldc*sizeof(out) multiples of 16 bytes.  Any M, N, K >= 0 (ragged edges are handled by the
 * copy engine's zero fill on loads and clipping on stores).
 * Quick returns: M == 0 or N == 0 -> GEMM_OK, nothing touched.  K == 0 ->
 * C <- beta * C (C is not read when beta == 0), A and B not read.
 * beta == 0: C is never read, so NaN/Inf already in C do not propagate.
 * Deterministic: the same call on the same device gives bitwise-identical C.
 * Accuracy: products are exact, sums are fp32 (order differs from a serial loop);
 * the result is alpha*acc + beta*C evaluated in fp32, then rounded to nearest even.
 */
gemm_status_t gemm(int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
                   const void* B, int64_t ldb, float beta, void* C, int64_t ldc, int in_dtype,
                   int out_dtype, int layout, void* stream);

/* Tile-configuration override for sweeps.  Zero fields mean "choose
 * automatically".
 *   bn        output columns per tile: 64, 128 or 256 for single-CTA tiles
 *             (128 rows); 128 or 256 for CTA-pair tiles (256 rows).
 *   group_m   tile-rows per group of the grouped tile order (>= 1).
 *   grid      number of persistent CTAs (clamped to the work available; even in
 *             pair mode).
 *   cta_group 1: one CTA per tile (tcgen05 cta_group::1); 2: a cluster of two
 *             CTAs per 256-row tile, one MMA spanning both SMs (cta_group::2),
 *             each SM loading its own half of A and of B.
 *   split_k   1: no split; 2 or 4: a cluster of that many CTAs shares each
 *             128-row tile, each accumulating 1/split_k of K, the partial sums
 *             reduced in distributed shared memory in a fixed order (needs
 *             cta_group 1; supported for bn 256 with split_k 2 or 4 and bn 128
 *             with split_k 2; one tile per cluster, so grid is ignored).
 *   stream_k  1: off; 2: on.  Stream-K runs all but the last whole wave of
 *             tiles data-parallel and splits the remaining tiles' k-groups evenly
 *             over all CTAs (or CTA pairs), each doing its stream-K share (from
 *             its last tile down) before its data-parallel tiles; a tile's
 *             partial sums are added by the CTA holding its last k-groups, in a
 *             fixed order, through a scratch buffer the library keeps per device
 *             and stream.  Ignored with split_k > 1.
 *             3: split-tile.  Every tile's k-groups are split over split_k CTAs
 *             (2 to 16; 0 means 2) of one-CTA tiles (bn 64, 128 or 256; 0 means
 *             128) without a cluster: the first CTA takes the first and larger
 *             share and finishes the tile, adding the other CTAs' partial sums
 *             (in CTA order) from the same scratch buffer; each of the others
 *             takes an even share of the rest.  Needs tiles x split_k <= the SM
 *             count (GEMM_ERR_UNSUPPORTED otherwise), a k-group (two 64-element
 *             k-blocks of 16-bit operands) per part, and cta_group 0 or 1.
 *   order     tile order of the persistent scheduler: 1 grouped (group_m
 *             tile-rows at a time, column-major inside the group; the default),
 *             2 Hilbert curve (the order the lecture "The Asynchronous Kernel:
 *             Tensor Cores & TMA", section "Scheduling is geometry", compares
 *             with the grouped one: every prefix of the walk stays compact).
 *             The Hilbert order walks the curve over the smallest power-of-two
 *             square holding the tile grid and keeps the cells inside the grid;
 *             when that square is more than 16 times the grid (a very elongated
 *             grid) or the grid has more than 2^22 tiles the grouped order is
 *             used.  Its table (8 bytes per tile) is built on the host and kept
 *             on the device per grid shape by the library (gemm_ex_noalloc
 *             always uses the grouped order).
 *   general   1: always launch the general kernel.  0 (the default): a call on
 *             the plain path -- the grouped tile order -- runs a kernel instance
 *             specialised for its layout when the plan's configuration has
 *             one.  With N times the output element size a multiple of 16
 *             bytes: the 256-wide CTA pair (beta == 0 with or without stream-K
 *             work, with or without a bias or activation; beta != 0 with or
 *             without stream-K work, without a bias or activation); with beta == 0 and no
 *             stream-K work, the single CTA of width 64 or 128 and the split-K
 *             clusters of 2 CTAs (width 64, 128 or 256), of 4 CTAs (width 64 or
 *             128) and of 8 CTAs (width 128) without a bias or activation, and
 *             the single CTA and the 2-CTA cluster of width 64 or 128 with one.
 *             With any N, beta == 0, no bias or activation and no stream-K
 *             work: the single CTA of width 64 or 128.  Both kernels compute
 *             the same result bit for bit.  Other values: GEMM_ERR_INVALID_ARG. */
enum { GEMM_ORDER_AUTO = 0, GEMM_ORDER_GROUPED = 1, GEMM_ORDER_HILBERT = 2 };

typedef struct {
  int32_t bn;
  int32_t group_m;
  int32_t grid;
  int32_t cta_group;
  int32_t split_k;
  int32_t stream_k;
  int32_t order;
  int32_t general;
} gemm_config_t;

/* gemm with an explicit configuration (cfg may be NULL = gemm()).  Same
 * contract and errors as gemm(); an invalid cfg field gives
 * GEMM_ERR_INVALID_ARG. */
gemm_status_t gemm_ex(int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
                      const void* B, int64_t ldb, float beta, void* C, int64_t ldc, int in_dtype,
                      int out_dtype, int layout, void* stream, const gemm_config_t* cfg);

/*
 * gemm_bias_act -- the GEMM with a fused epilogue:
 *
 *     C <- act(alpha * A * B + beta * C + bias)
 *
 * The bias + ReLU epilogue that "A dense FP16 matrix-multiply kernel for NVIDIA
 * Ada" (kd.iw.mk) folds into the GEMM (its paragraph on bias + ReLU after the
 * L2-rasterization table): the sum stays in an fp32 register through the bias
 * and the activation and is rounded to the output format once, with no extra
 * pass over C.  The per-row form is the per-row bias the "mma.sync and ldmatrix"
 * page (gpu-preview.ayushworks.com, day 73) names as coordinate-dependent
 * epilogue work.
 *
 * bias      : fp32, DEVICE pointer owned by the caller, only read, 16-byte
 *             aligned; N values (GEMM_BIAS_COL: bias[j] added to every row's
 *             column j) or M values (GEMM_BIAS_ROW: bias[i] added to row i).
 *             Unused (may be NULL) with GEMM_BIAS_NONE.
 * bias_kind : GEMM_BIAS_NONE, GEMM_BIAS_COL or GEMM_BIAS_ROW.
 * act       : GEMM_ACT_NONE or GEMM_ACT_RELU (negative results become +0; NaN
 *             stays NaN), applied after the bias.
 * The fp32 order is alpha*acc, then fmaf(beta, c, .), then + bias, then act,
 * then one round to nearest even.  Everything else (arguments, layouts, K == 0
 * -> C <- act(beta*C + bias), quick returns, determinism) is as for gemm_ex.
 * Errors: as gemm_ex, plus GEMM_ERR_INVALID_ARG for an unknown bias_kind or act
 * or a NULL bias that would be read, GEMM_ERR_UNSUPPORTED for a bias pointer
 * that is not 16-byte aligned.
 */
enum { GEMM_BIAS_NONE = 0, GEMM_BIAS_COL = 1, GEMM_BIAS_ROW = 2 };
enum { GEMM_ACT_NONE = 0, GEMM_ACT_RELU = 1 };

gemm_status_t gemm_bias_act(int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                            int64_t lda, const void* B, int64_t ldb, float beta, void* C,
                            int64_t ldc, int in_dtype, int out_dtype, int layout, const float* bias,
                            int bias_kind, int act, void* stream, const gemm_config_t* cfg);

/*
 * gemm_ex_noalloc -- gemm_ex that never allocates device memory.
 *
 * The pages have no counterpart: this entry point exists for callers that must
 * not allocate on the call path.  gemm_ex obtains a stream-K launch's scratch
 * (ready flags and fp32 partial tiles) from cudaMalloc the first time a stream
 * needs it (and again, after a cudaFree that synchronises the stream, when it
 * needs more).  A caller whose device memory is fully held by another
 * allocator, or whose steady-state loop must not synchronise or fail on
 * allocation, cannot accept that.  Here the scratch is a fixed device array of
 * GEMM_NOALLOC_SCRATCH_BYTES per device, built into the library.
 *
 * Same arguments, planning, kernels, results and errors as gemm_ex, plus:
 *  - GEMM_ERR_SCRATCH when the plan's scratch (gemm_plan_t.scratch_bytes)
 *    exceeds GEMM_NOALLOC_SCRATCH_BYTES (nothing is enqueued).  Plans without
 *    stream-K use no scratch and are never rejected.  A stream-K plan needs
 *    4 KB + (CTAs) * 128 * bn * 4 bytes with at most one CTA per SM, so on a
 *    152-SM GB300 the largest is 19.0 MiB and every plan fits.
 *  - Set-up: the first call on a device (that device current) looks up the
 *    array's device address and enqueues, on that call's stream, a clear of its
 *    4 KB of ready flags; make that first call before any stream capture.
 *  - The one array is shared by every call on the device: calls that may
 *    overlap on the device (different streams with no ordering between them,
 *    or several host threads) race on it and must be serialised by the caller.
 *    gemm_ex keeps its own per-stream scratch and does not touch this array.
 */
enum { GEMM_NOALLOC_SCRATCH_BYTES = 24 * 1024 * 1024 };

gemm_status_t gemm_ex_noalloc(int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                              int64_t lda, const void* B, int64_t ldb, float beta, void* C,
                              int64_t ldc, int in_dtype, int out_dtype, int layout, void* stream,
                              const gemm_config_t* cfg);

/*
 * gemm_host -- the same GEMM on HOST operands (end-to-end path).
 *
 * hA, hB, hC are host pointers (pinned memory gives asynchronous copies);
 * dA, dB, dC are caller-owned device buffers of at least the same extents
 * (rows * ld elements of each stored array), used as staging.  The call
 * enqueues copy hA -> dA and hB -> dB, copy hC -> dC when beta != 0, the GEMM
 * on the device buffers, and copy dC -> hC, all ordered after the work already
 * queued on `stream`.  It returns without synchronising; hC holds the result
 * after the caller synchronises `stream`.
 *   A problem that moves at least 64 MiB over the host link and has M >= 2048
 * is pipelined by row panels of C (about 8, each a multiple of 256 rows): B is
 * copied whole, then each panel's rows of A (and C) on an internal copy-in
 * stream, each panel's GEMM runs on `stream` once its rows are in, and its
 * rows of C return on an internal copy-out stream, so that copies in both
 * directions overlap the GEMMs; `stream` finally waits for both internal
 * streams.  Smaller problems run the four steps in order on `stream`.  Each
 * panel is a GEMM of its own (its plan may differ from the whole problem's).
 * Same argument rules and errors as gemm() (pointer checks apply to both sets);
 * GEMM_ERR_CUDA if a copy, stream or event call fails.
 */
gemm_status_t gemm_host(int64_t M, int64_t N, int64_t K, float alpha, const void* hA, int64_t lda,
                        const void* hB, int64_t ldb, float beta, void* hC, int64_t ldc,
                        int in_dtype, int out_dtype, int layout, void* dA, void* dB, void* dC,
                        void* stream);

/* Human-readable text for a status code (static storage, never NULL). */
const char* gemm_status_string(gemm_status_t status);

/*
 * gemm_sync_status -- synchronise `stream`, then report whether any GEMM kernel
 * on the current device gave up a wait since the last call.  Returns GEMM_OK,
 * GEMM_ERR_TIMEOUT (and stores the internal wait-site code, 1..8, in *site when
 * site != NULL; the word is then cleared), or GEMM_ERR_CUDA if the
 * synchronisation itself failed.  Meant for tests and benchmarks.
 */
gemm_status_t gemm_sync_status(void* stream, int* site);

/*
 * gemm_debug_set -- process-wide debug knobs, for tests only.
 * wait_timeout_ns: limit of every kernel wait (0 restores the default, 2 s).
 * inject_skip: when > 0, the copy producer of every CTA leaves its ring
 * iteration number (inject_skip - 1) unarmed, so the consumer's wait must run
 * out and the kernel must report GEMM_ERR_TIMEOUT and exit cleanly; 0 = off.
 */
void gemm_debug_set(uint64_t wait_timeout_ns, int32_t inject_skip);

/* The launch plan gemm() would use, computed on the host only (no CUDA call):
 * num_sms is the SM count to plan for.  Returns the same argument errors as
 * gemm() for the size/dtype/layout arguments. */
typedef struct {
  int32_t bm, bn, bk, stages;             /* bm: rows per tile (128, or 256 for a pair);
                                              bk: K per ring stage */
  int32_t m_tiles, n_tiles, k_blocks, num_tiles;
  int32_t grid, group_m, threads, smem_bytes;
  int32_t tmem_cols, a_mn, b_mn, epi_chunk_cols;
  int32_t cta_group, split_k;
  int32_t groups;      /* k-groups (ring stages) per tile */
  int32_t dp_tiles;    /* tiles of the data-parallel phase */
  int32_t order;       /* GEMM_ORDER_GROUPED or GEMM_ORDER_HILBERT */
  int32_t specialised; /* 1: a call under this plan with beta == 0 and no bias or
                          activation runs a specialised instance (see
                          gemm_config_t.general) */
  int64_t sk_iters;    /* stream-K iterations (tile k-groups) after it; 0 = none */
  int64_t scratch_bytes; /* stream-K / split-tile scratch the launch uses (0 = none) */
  int32_t tile_split;  /* split-tile parts per tile (gemm_config_t.stream_k 3); 0 = none */
  int32_t owner_groups; /* k-groups of the part that finishes a split tile */
} gemm_plan_t;

gemm_status_t gemm_plan(int64_t M, int64_t N, int64_t K, int in_dtype, int out_dtype, int layout,
                        int32_t num_sms, const gemm_config_t* cfg, gemm_plan_t* plan);

/* The grouped tile order (host copy of the device scheduler): tile index t ->
 * (m_blk, n_blk).  Covers every tile of an m_tiles x n_tiles grid exactly once
 * for t in [0, m_tiles * n_tiles). */
void gemm_tile_coord(int32_t t, int32_t m_tiles, int32_t n_tiles, int32_t group_m,
                     int32_t* m_blk, int32_t* n_blk);

/* A whole tile order on the host: order GEMM_ORDER_GROUPED (with group_m) or
 * GEMM_ORDER_HILBERT; writes the (m_blk, n_blk) of tiles 0 .. m_tiles*n_tiles-1
 * (at most max_tiles of them) and returns the tile count, or -1 when the order
 * is unknown or (Hilbert) not used for this grid shape.  The grouped order is
 * computed the kernel's way (gemm_fastdiv divisions); gemm_tile_coord computes
 * it with plain division, so the two agree tile for tile. */
int32_t gemm_tile_order(int order, int32_t m_tiles, int32_t n_tiles, int32_t group_m,
                        int32_t* m_blk, int32_t* n_blk, int32_t max_tiles);

/* The work split of one unit (a CTA, or a CTA pair) for a plan, computed on the
 * host exactly as the kernel walks it: the unit's even share of the sk_iters
 * stream-K iterations (sk_iters < 2^31), tile by tile from the share's last
 * tile down, then the whole tiles unit, unit + units, ... below dp_tiles.  Writes up to max_items (tile, first
 * k-group, end k-group) triples to items[3*i .. 3*i+2] and returns the number of
 * items the unit has (0 for invalid arguments). */
int32_t gemm_work_items(int32_t unit, int32_t units, int32_t dp_tiles, int64_t sk_iters,
                        int32_t groups, int32_t* items, int32_t max_items);

/* The one work item of unit `unit` under a split-tile plan (gemm_plan_t
 * tile_split and owner_groups, with the plan's groups), computed on the host
 * exactly as the kernel walks it: tile unit / tile_split, k-groups [0,
 * owner_groups) for the first part, an even share of the rest for the others.
 * Writes (tile, first k-group, end k-group) to item[0..2] and returns the number
 * of items the unit has (1), or 0 for invalid arguments. */
int32_t gemm_split_tile_item(int32_t unit, int32_t tile_split, int32_t owner_groups,
                             int32_t groups, int32_t* item);

/* n / d as the kernel divides by a run-time constant (a multiply and a shift
 * with host-computed constants), for host checks: 1 <= d < 2^31 and n < 2^31;
 * returns 0xFFFFFFFF for arguments outside that range. */
uint32_t gemm_fastdiv(uint32_t n, uint32_t d);

/* The tcgen05 descriptor encoders, exposed for host checks.  idesc: kind::f16
 * instruction descriptor; sdesc: 128B-swizzled shared-memory descriptor. */
uint32_t gemm_encode_idesc(int in_dtype, int a_mn, int b_mn, int m, int n);
uint64_t gemm_encode_sdesc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes);

/* Library version (major*10000 + minor*100 + patch). */
int32_t gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_TCGEN05_H */
