/*
 * gf -- fused GEMM + epilogue on GB300 (sm_103a): the C ABI.
 *
 * One dense half-precision matrix multiply per call, with the epilogue run
 * inside the same kernel while the fp32 accumulator is still on chip:
 *
 *   out[M,N] = epilog( A[M,K] . B[K,N] )      fp16/bf16 in, fp32 accumulate
 *
 * The operations follow these web pages on fused matmul epilogs:
 *  - "Fusing Matmul Epilogs with nvmath-python": "The problem addressed by
 *    fused epilogs" (product + bias per output column + ReLU in one call),
 *    "Forward-pass capabilities in the source" (RELU_BIAS, RELU_AUX_BIAS and
 *    its bit-encoded relu_aux mask; the stateful plan / execute split),
 *    "Backward-pass path shown in the example" (DRELU_BGRAD: the product with
 *    the transposed weight, masked by relu_aux, plus the column-wise sum that
 *    is the bias gradient).
 *  - "nvmath-python 封装 cuBLASLt ..." (nvmath-python over cuBLASLt): step 1
 *    (fp16 operands, bias of shape (m,1)), step 2 (plan with
 *    COMPUTE_32F_FAST_16F: fp32 accumulation; epilog and epilog inputs fixed
 *    at plan time), step 3 (execute is asynchronous on a stream; free
 *    releases the plan), "plan reuse" (planning is the expensive step,
 *    execute is light and reused for equal shape, dtype and epilog), "other
 *    epilogs" (BIAS, GELU_BIAS).
 *
 * Conventions for every call:
 *  - Matrices are dense and row-major. A is [m, k]. B is [k, n]
 *    (GF_B_KN, the default) or given as an [n, k] matrix W with B = W^T
 *    (GF_B_NK: an nn.Linear weight, or the transposed weight of a backward
 *    pass). out is [m, n].
 *  - Device pointers are caller-owned device memory (for example torch
 *    tensors), 16-byte aligned. The library never frees them.
 *  - relu_aux words: uint32 [ceil(m/32), n] row-major. Bit (i % 32) of word
 *    [i/32][j] is 1 when the fp32 pre-activation z[i][j] = acc + bias is
 *    strictly greater than 0. Bits of rows >= m are 0.
 *  - Errors: a call that fails returns a gf_status (or NULL for the plan
 *    constructors) and records it for gf_last_error() on the calling thread.
 *    Invalid arguments are rejected before anything is enqueued.
 *  - The stream argument is a cudaStream_t (NULL: the legacy default stream),
 *    declared through its underlying struct so this header needs no CUDA
 *    header.
 */
#ifndef GF_H
#define GF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GF_API __attribute__((visibility("default")))
#else
#define GF_API
#endif

struct CUstream_st; /* cudaStream_t == struct CUstream_st* */

typedef enum gf_status {
  GF_OK = 0,
  GF_ERR_INVALID_VALUE = 1,   /* bad argument: NULL, size, alignment, enum  */
  GF_ERR_UNSUPPORTED = 2,     /* valid but not handled (shape rule, device) */
  GF_ERR_NO_DEVICE = 3,       /* no CUDA device could be queried            */
  GF_ERR_CUDA = 4,            /* a CUDA runtime or driver call failed       */
  GF_ERR_OUT_OF_MEMORY = 5,   /* plan workspace could not be allocated      */
  GF_ERR_DEVICE_TIMEOUT = 6   /* a bounded wait inside a kernel gave up     */
} gf_status;

typedef enum gf_dtype {
  GF_F16 = 0, /* IEEE binary16 in and out */
  GF_BF16 = 1 /* bfloat16 in and out      */
} gf_dtype;

typedef enum gf_epilog {
  GF_EPILOG_NONE = 0,          /* out = acc                                      */
  GF_EPILOG_RELU_BIAS = 1,     /* out = max(acc + bias, 0)                       */
  GF_EPILOG_RELU_AUX_BIAS = 2, /* RELU_BIAS, and aux_out = relu_aux words        */
  GF_EPILOG_DRELU_BGRAD = 3,   /* out = acc masked by aux_in; bgrad = colsum(out) */
  GF_EPILOG_BIAS = 4,          /* out = acc + bias                               */
  GF_EPILOG_GELU_BIAS = 5,     /* out = gelu(acc + bias), tanh form              */
  GF_EPILOG_GELU_AUX_BIAS = 6, /* GELU_BIAS, and aux_out = acc + bias (dtype)    */
  GF_EPILOG_DGELU_BGRAD = 7    /* out = acc * gelu'(aux_in); bgrad = colsum(out) */
} gf_epilog;
/* GELU is the tanh form 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))
 * (Hendrycks & Gimpel 2016), named as GELU_BIAS on the nvmath-python /
 * cuBLASLt page ("other epilogs"). Its aux is the pre-activation z = acc +
 * bias rounded to dtype, [m, n] row-major: what DGELU_BGRAD reads back. */

typedef enum gf_bias_axis {
  GF_BIAS_COL = 0, /* bias[n]: one value per output column, broadcast down rows */
  GF_BIAS_ROW = 1  /* bias[m]: one value per output row (a (m,1) bias)          */
} gf_bias_axis;

typedef enum gf_b_layout {
  GF_B_KN = 0, /* B stored [k, n] row-major                        */
  GF_B_NK = 1  /* B = W^T with W stored [n, k] row-major          */
} gf_b_layout;

typedef enum gf_bgrad_mode {
  GF_BGRAD_TWO_PASS = 0, /* per-tile fp32 partial sums, then a fixed-order sum: deterministic */
  GF_BGRAD_ATOMIC = 1    /* one fp32 atomicAdd per column per tile: run-to-run order varies  */
} gf_bgrad_mode;

typedef struct gf_plan gf_plan;

/*
 * Plan one fused GEMM + epilogue: validates the problem, checks that the
 * current CUDA device is an sm_103 GPU, picks the tile configuration and
 * allocates the plan's device workspace (status word; bgrad partial sums for
 * DRELU_BGRAD). Host only; enqueues nothing. Equivalent to
 * gf_matmul_plan_ex(..., GF_B_KN).
 *
 * Source: the plan step of the stateful Matmul ("Fusing Matmul Epilogs with
 * nvmath-python", "Forward-pass capabilities in the source"; nvmath-python /
 * cuBLASLt page, step 2 and "plan reuse").
 *
 * m, n, k   : problem size, 0 <= m, n, k < 2^31; n % 8 == 0 and k % 8 == 0
 *             (16-byte row strides), else GF_ERR_UNSUPPORTED. m, n or k may be
 *             0 (an empty product; k == 0 makes acc = 0).
 * dtype     : element type of A, B, bias and out.
 * epilog    : one of gf_epilog.
 * bias_axis : GF_BIAS_COL or GF_BIAS_ROW; DRELU_BGRAD needs GF_BIAS_COL (its
 *             bias gradient is per column), else GF_ERR_UNSUPPORTED. Ignored by
 *             GF_EPILOG_NONE.
 * Returns a library-owned plan (release with gf_plan_free), or NULL with the
 * reason in gf_last_error().
 *
 * Environment overrides, read when a plan is made (gf_plan_set_option
 * called afterwards wins): GF_KERNEL (as GF_OPT_KERNEL), GF_TILE_N (128 or
 * 256, as GF_OPT_TILE_N), GF_BGRAD_MODE=atomic, GF_WAIT_LIMIT_US (as
 * GF_OPT_WAIT_LIMIT_US); GF_DEBUG prints a nonzero device status word from
 * gf_plan_status on stderr. Out-of-range values are ignored.
 */
GF_API gf_plan* gf_matmul_plan(int64_t m, int64_t n, int64_t k, gf_dtype dtype, gf_epilog epilog,
                               gf_bias_axis bias_axis);

/* gf_matmul_plan with the storage of B given explicitly (see gf_b_layout).
 * The backward of a linear layer multiplies by W^T for the forward weight W
 * ("Backward-pass path shown in the example"): that is GF_B_NK with W. */
GF_API gf_plan* gf_matmul_plan_ex(int64_t m, int64_t n, int64_t k, gf_dtype dtype,
                                  gf_epilog epilog, gf_bias_axis bias_axis,
                                  gf_b_layout b_layout);

/*
 * Enqueue the planned GEMM + epilogue on `stream` and return at once (the
 * nvmath-python / cuBLASLt page, step 3: execution does not block; the
 * caller synchronises). One kernel launch, plus one small finalize launch
 * for DRELU_BGRAD / DGELU_BGRAD in GF_BGRAD_TWO_PASS mode.
 *
 * A       : device [m, k].
 * B       : device [k, n] (GF_B_KN) or [n, k] (GF_B_NK).
 * bias    : device, n (GF_BIAS_COL) or m (GF_BIAS_ROW) elements of dtype.
 *           Required by RELU_BIAS, RELU_AUX_BIAS, BIAS, GELU_BIAS and
 *           GELU_AUX_BIAS; ignored otherwise.
 * out     : device [m, n] of dtype. Always required (when m*n > 0).
 * aux_in  : DRELU_BGRAD: relu_aux words [ceil(m/32), n] from a RELU_AUX_BIAS
 *           forward. DGELU_BGRAD: the pre-activation [m, n] of dtype from a
 *           GELU_AUX_BIAS forward. Required by both; ignored otherwise.
 * aux_out : RELU_AUX_BIAS: relu_aux words [ceil(m/32), n], written in full.
 *           GELU_AUX_BIAS: the pre-activation [m, n] of dtype. Required by
 *           both; ignored otherwise.
 * bgrad   : device fp32 [n], overwritten with the column sums of the fp32
 *           epilogue output (before rounding). Required by DRELU_BGRAD and
 *           DGELU_BGRAD; ignored otherwise.
 * A missing required pointer or a pointer not 16-byte aligned gives
 * GF_ERR_INVALID_VALUE; a failed launch gives GF_ERR_CUDA. The plan's
 * workspace is shared by its calls: use one plan from one stream at a time.
 */
GF_API gf_status gf_matmul_execute(const gf_plan* plan, const void* A, const void* B,
                                   const void* bias, void* out, const void* aux_in,
                                   void* aux_out, float* bgrad, struct CUstream_st* stream);

/*
 * Gate+up SwiGLU forward in one kernel ("gemm_swiglu_mlp_fusion.py" sample,
 * module docstring: silu(x Wg^T) * (x Wu^T) as one fused kernel, the down
 * projection a separate GEMM). Per output tile the kernel keeps two fp32
 * accumulators in tensor memory, g = x Wg^T and u = x Wu^T, and its epilogue
 * writes h = silu(g) * u with silu(g) = g / (1 + e^-g).
 *
 * m = rows of x (tokens), n = I (intermediate width), k = H (model width),
 * same size rules as gf_matmul_plan. save_gu = 1 also stores g and u
 * (rounded to dtype) for the backward ("save" rather than recompute); 0 does
 * not. The down projection out = h Wd^T is a plain
 * gf_matmul_plan_ex(m, H, I, dtype, GF_EPILOG_NONE, GF_BIAS_COL, GF_B_NK).
 */
GF_API gf_plan* gf_swiglu_plan(int64_t m, int64_t n, int64_t k, gf_dtype dtype, int save_gu);

/*
 * x: device [m, k]; Wg, Wu: device [n, k] (nn.Linear weights); h: device
 * [m, n]; g_out, u_out: device [m, n], required when the plan saves them,
 * ignored otherwise. All of dtype, 16-byte aligned. Asynchronous on stream,
 * one kernel launch. Errors as gf_matmul_execute; a plan that is not a
 * SwiGLU plan gives GF_ERR_INVALID_VALUE.
 */
GF_API gf_status gf_swiglu_execute(const gf_plan* plan, const void* x, const void* Wg,
                                   const void* Wu, void* h, void* g_out, void* u_out,
                                   struct CUstream_st* stream);

/*
 * dSwiGLU as the epilogue of dh = dout . Wd ("gemm_swiglu_mlp_fusion.py",
 * module docstring: the backward's dSwiGLU fused as the epilogue of
 * matmul(dout, Wd) -> dh). With the saved g and u:
 *   d_up   = dh * silu(g)
 *   d_gate = dh * u * sigmoid(g) * (1 + g (1 - sigmoid(g)))
 * m = rows, n = I, k = H. dout: device [m, k]; Wd: device [k, n] (the
 * down-projection weight as stored, [H, I]); g, u: device [m, n] from a
 * saving SwiGLU forward; d_gate, d_up: device [m, n]. All of dtype.
 */
GF_API gf_plan* gf_dswiglu_plan(int64_t m, int64_t n, int64_t k, gf_dtype dtype);

GF_API gf_status gf_dswiglu_execute(const gf_plan* plan, const void* dout, const void* Wd,
                                    const void* g, const void* u, void* d_gate, void* d_up,
                                    struct CUstream_st* stream);

/*
 * Synchronise `stream`, then read and clear the plan's device status word.
 * Returns GF_ERR_DEVICE_TIMEOUT if a bounded wait in a kernel of this plan
 * gave up since the last call (the kernel then skipped the rest of its work
 * and returned; its outputs are incomplete), GF_ERR_CUDA if the stream
 * reports an error, else GF_OK. Not on the pages: the library's failure
 * detection.
 */
GF_API gf_status gf_plan_status(const gf_plan* plan, struct CUstream_st* stream);

/*
 * Plan options (not on the pages; tuning and failure-detection knobs).
 * GF_OPT_BGRAD_MODE      : a gf_bgrad_mode (default GF_BGRAD_TWO_PASS).
 * GF_OPT_WAIT_LIMIT_US   : the limit of every bounded wait inside the kernel,
 *                          in microseconds (default 2000000, min 1000).
 * GF_OPT_TILE_N          : output tile width, 128 or 256 (0: the plan's choice).
 * GF_OPT_FAULT_DROP_LOAD : test hook. When v > 0 the producer skips its v-th
 *                          stage load, so the consumer's bounded wait runs
 *                          out; execute then completes with
 *                          GF_ERR_DEVICE_TIMEOUT from gf_plan_status. 0: off.
 * GF_OPT_KERNEL          : 0 the plan's choice (the CTA-pair kernel when its
 *                          256-row tiles fill the resident pairs, with
 *                          256 x 512 tiles when k >= 2048 and their
 *                          schedule -- waves of the resident pairs, with the
 *                          last-wave split of GF_OPT_SPLIT_K -- is no longer
 *                          than the 256 x 256 tiles' weighed by the wide
 *                          tile's gain, 12 % (4 % for the gate+up SwiGLU
 *                          plans); else the single-CTA kernel),
 *                          1 the single-CTA kernel
 *                          (128 x tile_n tiles), 2 the CTA-pair kernel
 *                          (256 x 256 tiles on two SMs, 256 x 128 for the
 *                          gate+up SwiGLU plans; GF_ERR_UNSUPPORTED if it
 *                          cannot be resident on this device), 3 the
 *                          CTA-pair kernel with 256 x 512 tiles (256 x 256
 *                          for the gate+up SwiGLU plans, each output column
 *                          taking a column of both weights: 3/4 of the
 *                          operand traffic per flop, one accumulator whose
 *                          halves are released as soon as the epilogue has
 *                          them in registers).
 * Returns GF_ERR_INVALID_VALUE for an unknown option or value.
 */
typedef enum gf_option {
  GF_OPT_BGRAD_MODE = 0,
  GF_OPT_WAIT_LIMIT_US = 1,
  GF_OPT_TILE_N = 2,
  GF_OPT_FAULT_DROP_LOAD = 3,
  GF_OPT_KERNEL = 4,
  GF_OPT_GROUP_M = 5,
  GF_OPT_L2_HINTS = 6,
  GF_OPT_SCHEDULE = 7,
  GF_OPT_SPLIT_K = 8,
  GF_OPT_PDL = 9,
  GF_OPT_RASTER = 10
} gf_option;
/* GF_OPT_SCHEDULE: how persistent CTAs (or CTA pairs) walk the output tiles,
 * overlapping each tile's epilogue with the next tile's mainloop.
 *   0 the plan's choice: 2 for the CTA-pair kernel, 3 for the single-CTA one;
 *   1 one tile per CTA (pair), launched in raster order by the hardware;
 *   2 dynamic (CTA-pair kernel): each pair takes the next tile from a counter
 *     in the plan's workspace, so the tiles in flight stay a contiguous run of
 *     the raster order and share their operand panels in L2;
 *   3 static: pair (CTA) c takes tiles c, c + grid, c + 2 grid, ... */
/* GF_OPT_L2_HINTS: L2 eviction priority of the operand loads, 10 * a + b with
 * a (for A) and b (for B) each 0 = no hint, 1 = evict first (streamed),
 * 2 = evict last (re-read by the tiles that follow). */
/* GF_OPT_GROUP_M: output tiles are visited in groups of this many row blocks
 * (128 rows, or 256 for the CTA-pair kernel) -- or column blocks, see
 * GF_OPT_RASTER -- so that concurrently running tiles share operand panels
 * in L2. 0: the plan's choice (8, or 4 column blocks for the 256 x 512
 * tiles); 1..4096 otherwise. */
/* GF_OPT_SPLIT_K: the single-CTA kernel shares the k-blocks of each output
 * tile among this many CTAs (one B operand only); so does the CTA-pair kernel
 * with 256 x 256 or 256 x 512 tiles for GF_EPILOG_NONE plans (each of its
 * CTAs then has a partial sum and a counter of its own, and the last to
 * finish for its 128 rows adds them; the plan's choice there splits only the
 * tiles of a last wave that is at most half full, when k has at least 32
 * blocks, or 128 when the tiles fill more than three waves, and it takes the
 * 256 x 512 tiles when their split schedule is the shorter one).
 * Each CTA leaves its fp32 partial sum in the plan's workspace; the last one
 * of a tile to finish adds the partials in split order (the result does not
 * depend on which finishes last) and runs the epilogue, so no CTA waits for
 * another. 0: the plan's choice (a split when k has at least 16 blocks of 64
 * and the tiles fill at most half the SMs: as many splits as the idle SMs
 * take, at most 8 and at most sqrt(k / 128)); 1: no split; 2..64: that many
 * (fewer when k has fewer 64-wide blocks; none when the partial sums would
 * take more than 256 MB). The workspace grows to tiles x splits x 128 x tile_n
 * fp32 plus one counter per tile; GF_ERR_OUT_OF_MEMORY (and no split) when it
 * cannot be allocated. Set options only while no launch of the plan is in
 * flight. */
/* GF_OPT_RASTER: the order of the output tiles. 1: raster groups of
 * GF_OPT_GROUP_M row blocks, column by column within a group (the group's
 * A panels stay in L2 while B streams through); 2: groups of GF_OPT_GROUP_M
 * column blocks, row by row within a group (B panels stay in L2); 0 (default)
 * the plan's choice: 2 with groups of 4 for the 256 x 512 tiles, else 1 with
 * groups of 8. Results are the same in every order. */
/* GF_OPT_PDL: 1 (default) launches the plan's kernels as programmatic
 * dependent launches: a kernel's launch and set-up (barriers, tensor memory,
 * descriptor prefetch) overlap the end of the kernel before it on the stream,
 * and it touches global memory only once that kernel has completed and its
 * writes are visible, so results are the same as with 0 (plain stream
 * order). */

GF_API gf_status gf_plan_set_option(gf_plan* plan, gf_option option, int64_t value);

/*
 * Plan-time autotuning of a gf_matmul plan (the plan-time algorithm search of
 * the nvmath-python / cuBLASLt page, "limitations" paragraph: autotuning
 * through MatmulPlanPreferences; here a search over this library's own
 * kernels). Runs the planned product once per candidate (CTA-pair kernel
 * with 256- or 512-wide tiles, dynamic or static schedule and raster groups
 * of 4, 8 or 16 tile rows; single-CTA kernel with 256- or 128-wide tiles,
 * and with 128-wide tiles k split 1, 2, 4 or 8 ways) on the caller's buffers,
 * `reps` timed launches each after one warm-up, synchronising `stream`, and
 * keeps the fastest in the plan. The outputs hold the result of the last
 * launch. Arguments as gf_matmul_execute; reps in 1..100.
 */
GF_API gf_status gf_matmul_autotune(gf_plan* plan, const void* A, const void* B,
                                    const void* bias, void* out, const void* aux_in,
                                    void* aux_out, float* bgrad, struct CUstream_st* stream,
                                    int32_t reps);

/* Read back the plan's choices: tile_m, tile_n, stages, grid size (CTAs per
 * launch), workspace bytes. Any out-pointer may be NULL. */
GF_API gf_status gf_plan_describe(const gf_plan* plan, int32_t* tile_m, int32_t* tile_n,
                                  int32_t* stages, int32_t* grid, int64_t* workspace_bytes);

/* The number of CTAs that share the k-blocks of one output tile in the
 * plan's current configuration (1: no split). GF_ERR_INVALID_VALUE for a
 * NULL argument. */
GF_API gf_status gf_plan_k_splits(const gf_plan* plan, int32_t* k_splits);

/* The number of kernels one execute of the plan enqueues in its current
 * configuration: 0 for an empty output, else 1, plus 1 for the bias-gradient
 * epilogs in GF_BGRAD_TWO_PASS mode (the finalize kernel that adds the
 * partials; GF_BGRAD_ATOMIC enqueues a memset of bgrad instead).
 * GF_ERR_INVALID_VALUE for a NULL argument. */
GF_API gf_status gf_plan_launches(const gf_plan* plan, int32_t* launches);

/*
 * DRELU_BGRAD that allocates nothing. The pages have no counterpart: this
 * entry point exists for callers that cannot call cudaMalloc (or any
 * allocating routine) -- code that must only use memory handed to it, such
 * as a framework's memory pool, a real-time loop that must not enter the
 * allocator, or a host API that forbids allocation while it runs. A plan
 * (gf_matmul_plan_ex) allocates its workspace; this call does not.
 *
 * It computes exactly what gf_matmul_execute computes for a
 * GF_EPILOG_DRELU_BGRAD plan in GF_BGRAD_TWO_PASS mode (same kernels, same
 * arguments: A, B, out, aux_in, bgrad as documented there) and returns at
 * once after enqueuing on `stream`.
 *
 * Scratch: the per-128-row-block partial sums live in one fixed device array
 * inside the library, GF_NOALLOC_MAX_PARTIALS fp32 values (8 MiB) plus a
 * 256-byte status word. Every GPU that loads the library holds it until the
 * process exits. ceil(m/128) * n must not exceed GF_NOALLOC_MAX_PARTIALS
 * (else GF_ERR_UNSUPPORTED, nothing enqueued).
 *
 * The first call on a device (and the first after its context was torn down
 * and re-created, e.g. by a device reset) looks up the array's device
 * address for that device (cudaGetSymbolAddress; no allocation); make that
 * first call before any stream capture. Every call shares the one array and
 * reuses it as the previous call left it: each call clears the status word on
 * its stream before its kernel starts, and every partial sum the finalize
 * reads is written by that call's kernel; calls that overlap on the GPU
 * (other streams, other threads) race on it and must be serialised by the
 * caller. A bounded wait that gives up inside the kernel is recorded in the
 * array's status word; gf_noalloc_status reports it.
 *
 * Returns GF_OK, GF_ERR_INVALID_VALUE (bad size, enum, NULL or misaligned
 * pointer), GF_ERR_UNSUPPORTED (n or k not a multiple of 8, beyond the
 * scratch limit, not an sm_103 device), GF_ERR_NO_DEVICE or GF_ERR_CUDA.
 */
#define GF_NOALLOC_MAX_PARTIALS 2097152

GF_API gf_status gf_drelu_bgrad_noalloc(int64_t m, int64_t n, int64_t k, gf_dtype dtype,
                                        gf_b_layout b_layout, const void* A, const void* B,
                                        void* out, const void* aux_in, float* bgrad,
                                        struct CUstream_st* stream);

/*
 * The status of gf_drelu_bgrad_noalloc on the calling thread's current
 * device, the counterpart of gf_plan_status for that allocation-free call
 * (it allocates nothing either). Synchronises `stream`, then reads the
 * status word of the library's fixed scratch array: GF_ERR_DEVICE_TIMEOUT
 * (and the word is cleared) if a bounded wait in the most recent call's
 * kernel gave up, whose outputs are then incomplete; GF_ERR_CUDA if the
 * stream reports an error; else GF_OK. GF_ERR_NO_DEVICE / GF_ERR_UNSUPPORTED
 * as gf_drelu_bgrad_noalloc. The pages have no counterpart.
 */
GF_API gf_status gf_noalloc_status(struct CUstream_st* stream);

/* Release the plan and its workspace ("free" on the nvmath-python / cuBLASLt
 * page, step 3). Caller tensors are untouched. NULL is a no-op. Work already
 * enqueued with the plan must have completed. */
GF_API void gf_plan_free(gf_plan* plan);

/* Static text for a status code. */
GF_API const char* gf_status_string(gf_status status);

/* The status of the last failing call on this thread (GF_OK if none). */
GF_API gf_status gf_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GF_H */
