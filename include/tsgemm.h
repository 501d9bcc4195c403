/*
 * tsgemm.h -- C ABI of the GB300 (sm_103a) tile-level GEMM library.
 *
 * Operation.  C = A * B with A (M x K) and B (K x N) in row-major order and
 * C (M x N) row-major, accumulated in fp32.  This is the tile-level GEMM of
 * the TileLang single-device skeleton ("TileScale 与 TileLang比较",
 * yaopepe.com, section 核心抽象与编程模型对比): the accumulator tile is
 * cleared, every BK-slice product of an A tile and a B tile is added into it,
 * and the tile is copied to C.  C is overwritten; there is no alpha or beta.
 * The cluster form (two SMs computing one tile as a pair, which the TileScale
 * README, section on T.Scale, calls a distributed GEMM on two SMs sharing
 * operands over distributed shared memory) and the K split with a reduction
 * (TileScale README, "Example of GEMM": warpgroups split along K and reduce)
 * are implementation choices of the plan; they do not change the result
 * beyond the fp32 summation order.
 *
 * Supported (dtype_in, dtype_out): (F16, F32), (F16, F16), (BF16, BF16),
 * (BF16, F32), and the 8-bit float inputs (E4M3 or E5M2, both operands the
 * same format) with an F16, BF16 or F32 output: a low-precision GEMM on the
 * same skeleton, of the Dequant-GEMM family TileLang targets ("TileScale 与
 * TileLang比较", sections 设计目标、定位与适用场景 and 生态互操作、性能、
 * 局限与路线图).  8-bit inputs take the RCR layout only (A stored M x K, B stored N x K, the
 * K-major form both tensor-core operands are read in).  Everything else
 * returns TSGEMM_ERR_UNSUPPORTED.
 *
 * Numerics.  Products of the 16-bit or 8-bit inputs are exact; sums are fp32 in an
 * order fixed by the plan (tensor-core order inside a K-slice, K-slices in
 * increasing k, split-K partials added in split order 0..S-1), so results
 * are reproducible run to run.  fp32 -> bf16/fp16 output conversion rounds
 * to nearest, ties to even.
 *
 * Memory.  A, B and C are device pointers owned by the caller, on the device
 * that was current when the plan was made, 16-byte aligned, with C not
 * overlapping A or B.  Stored row strides must be multiples of 16 bytes: A's
 * (K * e, or M * e when A is stored K x M), B's (N * e, or K * e when B is
 * stored N x K), e the input element size (2, or 1 for 8-bit inputs), and
 * C's (N * sizeof(out)); otherwise TSGEMM_ERR_ALIGNMENT.
 *
 * Errors.  Every call returns a tsgemm_status_t.  Argument, alignment and
 * device errors are detected on the host before anything is launched.  A
 * kernel never waits without bound: each wait on the device gives up after
 * a time limit (default 1 s), records TSGEMM_ERR_TIMEOUT in the plan's
 * device status word and returns; tsgemm_status() reads that word after the
 * caller has synchronised the stream.
 */
#ifndef TSGEMM_H
#define TSGEMM_H

#include <stdint.h>

#if defined(__GNUC__)
#define TSGEMM_API __attribute__((visibility("default")))
#else
#define TSGEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tsgemm_plan_s* tsgemm_plan_t;

typedef enum {
    TSGEMM_F16 = 0,  /* IEEE binary16 */
    TSGEMM_BF16 = 1, /* bfloat16 */
    TSGEMM_F32 = 2,  /* IEEE binary32 (outputs only) */
    TSGEMM_E4M3 = 3, /* OCP 8-bit float E4M3 (bias 7, no infinities, max 448); inputs only */
    TSGEMM_E5M2 = 4  /* OCP 8-bit float E5M2 (bias 15, IEEE-style inf/NaN, max 57344); inputs only */
} tsgemm_dtype_t;

/* Operand storage.  C is always M x N row-major.  The transposed-B forms are
 * the T.gemm(..., transpose_B=True) of the TileScale examples (SUMMA and
 * Cannon local GEMMs in the project_analysis.md notes). */
typedef enum {
    TSGEMM_LAYOUT_RRR = 0, /* A M x K row-major, B K x N row-major */
    TSGEMM_LAYOUT_RCR = 1, /* A M x K row-major, B stored N x K row-major (B column-major) */
    TSGEMM_LAYOUT_CRR = 2, /* A stored K x M row-major (A column-major), B K x N row-major */
    TSGEMM_LAYOUT_CCR = 3  /* A stored K x M, B stored N x K */
} tsgemm_layout_t;

typedef enum {
    TSGEMM_OK = 0,
    TSGEMM_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, bad enum */
    TSGEMM_ERR_UNSUPPORTED = 2, /* dtype pair, layout, or device not CC 10.3 */
    TSGEMM_ERR_ALIGNMENT = 3,   /* pointer or row stride not 16-byte aligned */
    TSGEMM_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
    TSGEMM_ERR_TIMEOUT = 5,     /* a bounded device wait expired */
    TSGEMM_ERR_OOM = 6,         /* plan could not allocate its buffers */
    TSGEMM_ERR_SCRATCH_LIMIT = 7 /* problem needs more than the fixed scratch of
                                    tsgemm_run_splitk_noalloc */
} tsgemm_status_t;

/* Execution configuration of a plan.  In tsgemm_plan_ex every field left at
 * 0 is chosen by the planner; a non-zero field forces that value. */
typedef struct {
    int32_t block_m;      /* rows of C per MMA tile: 128 (one SM) or 256 (SM pair) */
    int32_t block_n;      /* columns of C per tile: 64, 128, 192 or 256; 512
                             for a CTA pair (block_m 256) whose tile's two
                             256-column halves fill tensor memory: each K
                             slice's A feeds two N = 256 MMAs.  The planner
                             takes 512 for whole-tile schedules of at least
                             four rounds (RRR, RCR); forced, it runs whole
                             tiles or stream-K, never a split. */
    int32_t splits;       /* K split factor S of the split tiles (1 = no split) */
    int32_t stages;       /* depth of the shared-memory operand ring */
    int32_t group_m;      /* tile rows per raster group (L2 reuse) */
    int32_t grid;         /* CTAs launched (persistent) */
    int64_t units;        /* work units = whole tiles + split_tiles * splits */
    int64_t workspace_bytes; /* split-K (stream-K) partials owned by the plan:
                                split_tiles * splits * block_m * block_n * 4
                                bytes (see stream_k_tiles) */
    int32_t timeout_ms;   /* limit of every device-side wait */
    int32_t debug_flags;  /* tests only: TSGEMM_DEBUG_* */
    int64_t split_tiles;  /* work units split into `splits` K parts: the last
                             ones of the schedule (all, or the last partial
                             wave). Forced with splits > 1; 0 then means all. */
    int64_t stream_k_tiles; /* stream-K: the last stream_k_tiles tiles (units)
                               of the schedule have their K slices spread
                               evenly over all CTAs (CTA pairs), after rounds
                               of whole tiles; a tile cut between CTAs is
                               finished by the CTA holding its first K slices.
                               Excludes splits > 1. Forced: > 0 a count, -1
                               none, 0 the planner's choice. The workspace is
                               then one block_m x block_n fp32 partial per
                               slot. */
    int32_t cluster_split;  /* 2, 4 or 8: the DSMEM split of K (block_m 128,
                               RRR layout, 16-bit inputs, at least that many
                               K slices): the cs CTAs of a cs x 1 cluster
                               compute cs consecutive parts of every tile's
                               K range; CTA r receives the fp32 sum of parts
                               0..r-1 from CTA r - 1 through distributed
                               shared memory, chunk by chunk, adds its own
                               and passes it on, and the last CTA stores C
                               (parts summed in K order); no workspace.
                               Forced only; the planner reports 1
                               otherwise. */
} tsgemm_config_t;

/* Tests only: the first CTA (or CTA pair) skips the first operand load of
 * its first work unit, so the MMA issuer's bounded wait runs out; the launch
 * ends with TSGEMM_ERR_TIMEOUT in the status word instead of hanging. */
#define TSGEMM_DEBUG_SKIP_FIRST_LOAD 1

/* Validate the problem, check that the current device is CC 10.3, choose the
 * tile shape, split factor and grid, and allocate the plan's device buffers
 * (status word; split-K workspace and tile counters when S > 1).  The plan
 * owns those buffers.  On success *out holds the plan; on failure *out is
 * NULL. */
TSGEMM_API tsgemm_status_t tsgemm_plan(tsgemm_plan_t* out, int64_t M, int64_t N, int64_t K,
                            tsgemm_dtype_t dtype_in, tsgemm_dtype_t dtype_out,
                            tsgemm_layout_t layout);

/* tsgemm_plan with some configuration fields forced (see tsgemm_config_t).
 * `force` may be NULL.  A forced value the kernel cannot run returns
 * TSGEMM_ERR_UNSUPPORTED.  The parts of a split (or stream-K) tile never
 * wait for one another: whichever part completes a chunk's set of partials
 * adds them, so any split factor runs on any grid, and a run stays correct
 * when some of its CTAs must wait for SMs held by other work. */
TSGEMM_API tsgemm_status_t tsgemm_plan_ex(tsgemm_plan_t* out, int64_t M, int64_t N, int64_t K,
                               tsgemm_dtype_t dtype_in, tsgemm_dtype_t dtype_out,
                               tsgemm_layout_t layout, const tsgemm_config_t* force);

/* Enqueue C = A * B on `stream` (a cudaStream_t; NULL is the legacy default
 * stream).  Asynchronous: returns after the launch.  Checks pointer
 * alignment and that A, B, C are device memory on the plan's device.  The
 * operand descriptors are re-encoded only when a pointer changed since the
 * previous call.  A plan may be in flight on one stream at a time (its
 * split-K workspace is not re-entrant). */
TSGEMM_API tsgemm_status_t tsgemm_run(tsgemm_plan_t plan, const void* A, const void* B, void* C,
                           void* stream);

/* Free the plan and its device buffers.  The caller must make sure no run of
 * the plan is still executing.  NULL is accepted. */
TSGEMM_API tsgemm_status_t tsgemm_destroy(tsgemm_plan_t plan);

/* The device status word of the plan: TSGEMM_OK, or TSGEMM_ERR_TIMEOUT when a
 * bounded wait of an earlier run expired.  Call after synchronising the
 * stream of the runs.  Reading a timeout clears the word and resets the
 * split-K tile counters so the plan can run again. */
TSGEMM_API tsgemm_status_t tsgemm_status(tsgemm_plan_t plan);

/* The configuration the plan runs with. */
TSGEMM_API tsgemm_status_t tsgemm_get_config(tsgemm_plan_t plan, tsgemm_config_t* out);

/* The planner alone, host only (no GPU needed): the configuration
 * tsgemm_plan_ex would choose for this problem on a device with `num_sms`
 * SMs.  Same validation and return codes as tsgemm_plan_ex, except that the
 * device is not queried. */
TSGEMM_API tsgemm_status_t tsgemm_choose_config(int64_t M, int64_t N, int64_t K,
                                     tsgemm_dtype_t dtype_in, tsgemm_dtype_t dtype_out,
                                     tsgemm_layout_t layout, int32_t num_sms,
                                     const tsgemm_config_t* force, tsgemm_config_t* out);

/* A static English description of a status code. */
TSGEMM_API const char* tsgemm_status_string(tsgemm_status_t s);

/* ---- Split-K GEMM without any allocation -------------------------------
 *
 * The pages this library follows have no counterpart of this entry point;
 * it exists for callers that cannot allocate device memory.  tsgemm_plan
 * allocates its split-K workspace, tile counters and status word with
 * cudaMalloc.  Some callers cannot do that: code that runs inside another
 * framework's allocator or memory hooks (where allocating would re-enter
 * it), plug-ins that are handed their buffers and own no allocator, and
 * real-time loops that forbid cudaMalloc/cudaFree after start-up because
 * those calls can synchronise the whole device.  This entry point needs no
 * plan: the split-K scratch lives in one fixed device array inside the
 * library (TSGEMM_NOALLOC_SCRATCH_BYTES, about 34 MiB), which every GPU that
 * loads the library holds until the process exits.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 * Computes C = A * B exactly like tsgemm_run with the K dimension split in
 * `splits` parts (0 lets the planner choose; 1 means no split).  A, B, C as
 * for tsgemm_run: device memory of the current device, 16-byte aligned, C
 * overlapping neither A nor B.  `status` may be NULL; otherwise it is a
 * device int (or mapped pinned host int) the kernel sets to
 * TSGEMM_ERR_TIMEOUT if a bounded device wait expires (it is cleared to 0
 * on `stream` before the launch).
 *
 * Limits: at most TSGEMM_NOALLOC_MAX_TILES output tiles and at most
 * TSGEMM_NOALLOC_WS_BYTES of fp32 partials (split tiles * S * 128 * block_n *
 * 4 bytes); larger problems return TSGEMM_ERR_SCRATCH_LIMIT before anything
 * is enqueued.
 *
 * Every call uses the same scratch array, which keeps the previous call's
 * contents; each call clears the tile counters it needs on `stream` before
 * its launch.  Calls whose kernels overlap on the GPU (on different streams,
 * or from different host threads without ordering) race on that array and
 * give wrong results: order them on one stream.
 *
 * The first call on each device does a one-time set-up with that device
 * current (it looks up the device address of the scratch array and sets the
 * kernels' shared-memory limit); make that first call before any stream
 * capture.  Asynchronous otherwise: returns after the launch. */
#define TSGEMM_NOALLOC_MAX_TILES 16384
#define TSGEMM_NOALLOC_WS_BYTES (32u << 20)
/* status word, 32 counters per tile at most, the fp32 partials */
#define TSGEMM_NOALLOC_SCRATCH_BYTES (256u + TSGEMM_NOALLOC_MAX_TILES * 128u + TSGEMM_NOALLOC_WS_BYTES)

TSGEMM_API tsgemm_status_t tsgemm_run_splitk_noalloc(int64_t M, int64_t N, int64_t K,
                                                     tsgemm_dtype_t dtype_in,
                                                     tsgemm_dtype_t dtype_out, int32_t splits,
                                                     const void* A, const void* B, void* C,
                                                     int* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TSGEMM_H */
