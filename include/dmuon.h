/*
 * dmuon.h -- C ABI of the GB300 batched Gram-space Newton-Schulz Muon step.
 *
 * Subject: "DMuon: Efficient Distributed Muon Training with Near-Adam
 * Overhead" (arXiv 2606.27153), gist.science technical summary (pt/fr),
 * section 2.2 "Gram Newton-Schulz iteration": the owner of a weight matrix
 * runs Newton-Schulz on its momentum-aggregated gradient in the m x m Gram
 * space G = X X^T (m < n), forms G SYRK-style (lower triangle only), and
 * batches matrices of like shape so small ones do not leave the GPU idle.
 * This library is that per-owner compute on one GPU: no ranks, no
 * collectives.
 *
 * One optimizer step, per matrix W (rows x cols) with gradient and momentum
 * of the same shape and dtype:
 *   M' = beta*M + grad;  U = grad + beta*M'       (Nesterov; option: U = M')
 *   X  = U (rows <= cols) or U^T (rows > cols):    m x n, m = min, n = max
 *   X0 = X / (||X||_F + eps)
 *   T Newton-Schulz steps with the quintic (a, b, c):
 *     Gram route:   R = X0 X0^T; per step P = aI + bR + cR^2, Q <- P Q,
 *                   R <- P R P; result Q X0
 *     direct route: per step A = X X^T, B = bA + cA^2, X <- aX + B X
 *   W' = (1 - lr*wd) W - lr*s*O,  O = result in W's orientation,
 *   s = sqrt(max(1, rows/cols)) (option: 0.2*sqrt(max(rows, cols))).
 * The pages fix neither coefficients, eps, momentum form nor update scale;
 * the defaults are the published Muon ones: (3.4445, -4.7750, 2.0315),
 * T = 5, eps = 1e-7, Nesterov, aspect scale.
 *
 * Conventions for every entry point:
 *  - Pointer arrays are HOST arrays of `count` DEVICE pointers, in the order
 *    of the shapes given to dmuon_plan.  Each tensor is row-major,
 *    contiguous, rows x cols elements of the shape's dtype, and starts on a
 *    16-byte boundary (else DMUON_ERR_ALIGN).
 *  - The caller owns params, grads, momenta and the workspace.  The library
 *    owns only host-side plan data.  params and momenta are updated in place;
 *    grads are read only.
 *  - dmuon_step is asynchronous on `stream` (a cudaStream_t passed as void*,
 *    NULL = legacy default stream).  It allocates nothing and never
 *    synchronises the host, except that a change of the pointer set since the
 *    previous step uploads the new pointer table with one pageable copy.
 *    With the same pointer set as the previous call it issues only stream
 *    work (memsets and kernel launches), so such a call can be captured in a
 *    CUDA graph and replayed (timers off).  The tensor-core launches after
 *    the step's first kernel are programmatic dependent launches: each may be
 *    placed while the one before it finishes and touches global memory only
 *    after that one has completed; the step's first kernel waits for the
 *    caller's earlier work in the ordinary way.
 *  - Errors are negative status codes; dmuon_last_error() gives the message
 *    of the calling thread's last failure.  A handle must not be used on two
 *    streams at once.
 *  - Every device-side wait inside the kernels is bounded; on time-out the
 *    kernel records DMUON_ERR_DEVICE_TIMEOUT in the workspace status word and
 *    returns.  dmuon_device_status() reads (and clears) it.
 */
#ifndef DMUON_H
#define DMUON_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* storage dtypes of W, grad and momentum */
#define DMUON_BF16 0
#define DMUON_FP32 1

/* precision modes */
#define DMUON_PREC_BF16 0 /* tcgen05 tensor cores, bf16 operands, fp32 accumulation (default) */
#define DMUON_PREC_FP32 1 /* fp32 FFMA (SIMT) for every product: validation mode */

/* route rules (which Newton-Schulz form a bucket runs) */
#define DMUON_ROUTE_AUTO 0   /* Gram when n >= 3m or m <= small_m, else direct */
#define DMUON_ROUTE_GRAM 1   /* Gram space for every bucket */
#define DMUON_ROUTE_DIRECT 2 /* direct m x n iteration for every bucket */

/* per-bucket route and m x m engine reported by dmuon_plan_bucket */
#define DMUON_BUCKET_GRAM 1
#define DMUON_BUCKET_DIRECT 2
#define DMUON_ENGINE_TC_BF16 0 /* tensor cores, bf16 operands */
#define DMUON_ENGINE_SIMT_FP32 1 /* fp32 FFMA */
#define DMUON_ENGINE_TC_SPLIT 2 /* tensor cores, split-bf16 operands: each m x m operand
                                   x = hi + lo (hi = bf16(x), lo = bf16(x - hi)) and each
                                   product hi*hi + hi*lo + lo*hi; the final product's Q
                                   as hi + lo */

/* tile rules of the tensor-core symmetric products of bf16 buckets with m <= 128
   (larger buckets, and FP32 precision, always run one matrix per tile: SINGLE) */
#define DMUON_TILE_AUTO 0     /* a shape: the plan's rule; the plan: PACKED */
#define DMUON_TILE_PACKED 1   /* 2 (m <= 128) or 4 (m <= 64) matrices per 256 x 256 pair
                                 tile, laid block-diagonally */
#define DMUON_TILE_SINGLE 2   /* one matrix per pair tile */

/* update-scale rules */
#define DMUON_SCALE_ASPECT 0 /* s = sqrt(max(1, rows/cols)) */
#define DMUON_SCALE_RMS 1    /* s = 0.2*sqrt(max(rows, cols)) */

/* status codes */
#define DMUON_OK 0
#define DMUON_ERR_INVALID_ARG -1
#define DMUON_ERR_ALIGN -2
#define DMUON_ERR_NO_WORKSPACE -3
#define DMUON_ERR_UNSUPPORTED_DTYPE -4
#define DMUON_ERR_CUDA -5
#define DMUON_ERR_DEVICE_TIMEOUT -6
#define DMUON_ERR_UNSUPPORTED_DEVICE -7
#define DMUON_ERR_WORKSPACE_TOO_SMALL -8

/* limits checked by dmuon_plan */
#define DMUON_MAX_DIM (1 << 20)      /* rows, cols <= 2^20 */
#define DMUON_MAX_ELEMS (1LL << 31)  /* rows*cols < 2^31 */
#define DMUON_MAX_NS_STEPS 16

typedef struct dmuon_plan_s* dmuon_handle_t;

typedef struct {
    int64_t rows;     /* >= 1 */
    int64_t cols;     /* >= 1 */
    int32_t dtype;    /* DMUON_BF16 | DMUON_FP32 */
    int32_t route;    /* this matrix's route rule: 0 (DMUON_ROUTE_AUTO) = the plan's
                         options->route; DMUON_ROUTE_GRAM or DMUON_ROUTE_DIRECT override it
                         (e.g. from a measured per-bucket choice) */
    int32_t tile;     /* this matrix's tile rule: 0 (DMUON_TILE_AUTO) = the plan's
                         options->tile_rule; DMUON_TILE_PACKED or _SINGLE override it */
    int32_t reserved; /* 0 */
} dmuon_shape_t;

/* Zero-initialised options give the defaults noted on each field. */
typedef struct {
    int32_t precision;      /* DMUON_PREC_*; default DMUON_PREC_BF16 */
    int32_t route;          /* DMUON_ROUTE_*; default AUTO */
    float ns_a, ns_b, ns_c; /* quintic coefficients; all 0 => (3.4445, -4.7750, 2.0315) */
    float eps;              /* normalisation epsilon; 0 => 1e-7 */
    int32_t scale_rule;     /* DMUON_SCALE_*; default ASPECT */
    int32_t no_nesterov;    /* 0 => Nesterov U = grad + beta*M'; 1 => U = M' */
    int32_t small_m;        /* AUTO route and BF16 mode: Gram buckets with m <= small_m run
                               their m x m products on split-bf16 tensor cores
                               (DMUON_ENGINE_TC_SPLIT); 0 => 256; < 0 => none */
    int32_t tile_rule;      /* DMUON_TILE_*; 0 (AUTO) => PACKED */
    uint64_t workspace_budget; /* bytes for one wave of buckets; 0 => everything in one wave */
} dmuon_options_t;

typedef struct {
    int32_t dtype;     /* DMUON_BF16 | DMUON_FP32 */
    int32_t route;     /* DMUON_BUCKET_GRAM | DMUON_BUCKET_DIRECT */
    int32_t mm_engine; /* DMUON_ENGINE_* used for the m x m products */
    int32_t tile;      /* DMUON_TILE_PACKED or DMUON_TILE_SINGLE (the bucket's resolved rule) */
    int64_t m, n;      /* canonical short and long side */
    int64_t count;     /* matrices in the bucket */
    int64_t per_matrix_bytes; /* workspace bytes one matrix of the bucket needs in a wave */
} dmuon_bucket_info_t;

/* ---- planning (host only: no CUDA call, works without a GPU) ---------- */

/* Shape-bucketing planner (DMuon technical summary on gist.science, section
 * 2.2, "batching": matrices of like shape are grouped so that small ones do
 * not leave the GPU idle; the Gram iteration takes the short side m < n).
 * Each shape is canonicalised to (m, n, transposed)
 * with m = min(rows, cols), n = max(rows, cols), transposed = rows > cols
 * (tall matrices are packed transposed), and its route resolved: the shape's
 * own rule, else options->route; AUTO gives Gram when n >= 3m or m <=
 * small_m, else direct; FP32 precision gives Gram unless the rule is DIRECT.
 * Its tile rule likewise: the shape's own, else options->tile_rule, AUTO
 * meaning PACKED; SINGLE wherever packing does not apply (m > 128, FP32).
 * Buckets are keyed (dtype, m, n, route, tile), ordered by that key ascending
 * (DMUON_BUCKET_GRAM before DMUON_BUCKET_DIRECT); matrices keep their input
 * order inside a bucket.  Buckets are then packed, in bucket order, into waves whose
 * workspace fits options->workspace_budget, splitting a bucket where needed.
 * Returns NULL on error (message in dmuon_last_error): count < 1, a NULL
 * pointer, a dimension outside [1, DMUON_MAX_DIM], rows*cols >=
 * DMUON_MAX_ELEMS, an unknown dtype, an unknown shape route or tile rule, a
 * nonzero reserved field, bad options,
 * or a budget smaller than one matrix. */
dmuon_handle_t dmuon_plan(const dmuon_shape_t* shapes, int64_t count);
dmuon_handle_t dmuon_plan_ex(const dmuon_shape_t* shapes, int64_t count,
                             const dmuon_options_t* options);
void dmuon_destroy(dmuon_handle_t h); /* NULL is a no-op */

int64_t dmuon_plan_num_buckets(dmuon_handle_t h);
int dmuon_plan_bucket(dmuon_handle_t h, int64_t bucket, dmuon_bucket_info_t* out);
/* out receives `count` input indices, in bucket order */
int dmuon_plan_bucket_members(dmuon_handle_t h, int64_t bucket, int64_t* out);
int64_t dmuon_plan_num_waves(dmuon_handle_t h);
int64_t dmuon_plan_wave_num_pieces(dmuon_handle_t h, int64_t wave);
/* piece = matrices [start, start+count) of bucket `bucket` (bucket order) */
int dmuon_plan_wave_piece(dmuon_handle_t h, int64_t wave, int64_t piece,
                          int64_t* bucket, int64_t* start, int64_t* count);
/* Algorithmic FLOPs of one step with `ns_steps` iterations (section 2.2,
 * "symmetry": the symmetric products count half): 2 per
 * multiply-add, symmetric outputs counted once (SYRK and the m x m products
 * at half).  Gram bucket: (3 m^2 n + (4T-3) m^3) per matrix; direct bucket:
 * T (3 m^2 n + m^3).  Written to out[0]; out[1] gets the part run on tensor
 * cores.  Returns DMUON_OK. */
int dmuon_plan_flops(dmuon_handle_t h, int32_t ns_steps, double* out);

/* ---- workspace --------------------------------------------------------- */

/* Device bytes the caller must provide (256-byte aligned).  No counterpart
 * in the paper (its module plugs into the training framework and allocates
 * there, section 2 and the abstract); here the caller owns every device byte. */
size_t dmuon_workspace_bytes(dmuon_handle_t h);
/* Binds caller-owned device memory (e.g. a torch uint8 tensor) of at least
 * dmuon_workspace_bytes(h) bytes, 256-byte aligned, on the current device.
 * Builds the TMA tensor maps and launch tables and copies them into the
 * workspace (synchronous).  Needs an sm_103 GPU: DMUON_ERR_UNSUPPORTED_DEVICE
 * otherwise. */
int dmuon_bind_workspace(dmuon_handle_t h, void* dev_ptr, size_t bytes);

/* ---- the step ---------------------------------------------------------- */

/* One Muon step over every planned matrix (formula in the file header):
 * the per-owner compute of section 2.2 -- Newton-Schulz on the
 * momentum-aggregated gradient (section 1) carried in the Gram space, then
 * Muon's update rule, unchanged (section 5).
 * params[i], grads[i], momenta[i]: device pointers of shape i.  lr, wd >= 0,
 * 0 <= beta < 1 (finite), 1 <= ns_steps <= DMUON_MAX_NS_STEPS.  Errors:
 * INVALID_ARG (NULL arrays or pointers, bad scalars), ALIGN,
 * NO_WORKSPACE, CUDA (launch failure). */
int dmuon_step(dmuon_handle_t h, void* const* params, const void* const* grads,
               void* const* momenta, float lr, float beta, float wd,
               int32_t ns_steps, void* stream);

/* No counterpart in the paper (overlap of the caller's parameter copies with
 * the step, in the spirit of section 2.2's overlap of communication and
 * compute).  dmuon_step, with one more ordering point: if params_ready (a cudaEvent_t
 * passed as void*) is not NULL, `stream` waits for it right before the first
 * launch that writes the parameters -- the final product of the first wave;
 * the momentum, normalisation and Newton-Schulz launches before it do not
 * wait.  A caller still reading the previous step's parameters (e.g. copying
 * them to the host on another stream) records params_ready when done and so
 * overlaps that read with this step's earlier phases.  Same return codes as
 * dmuon_step. */
int dmuon_step_ex(dmuon_handle_t h, void* const* params, const void* const* grads, void* const* momenta,
                  float lr, float beta, float wd, int32_t ns_steps, void* stream, void* params_ready);

/* No counterpart in the paper (bounded device waits are this library's).
 * Synchronises `stream`, returns the device status word (DMUON_OK or
 * DMUON_ERR_DEVICE_TIMEOUT) and clears it. */
int dmuon_device_status(dmuon_handle_t h, void* stream);

/* ---- measurement ------------------------------------------------------- */

#define DMUON_TIMER_MOMENTUM 0 /* momentum + pack + sum of squares */
#define DMUON_TIMER_NORM 1     /* per-matrix 1/(||X||+eps) */
#define DMUON_TIMER_SYRK 2     /* first product of every wave: Gram / first A = X X^T */
#define DMUON_TIMER_NS 3       /* the Newton-Schulz polynomial products */
#define DMUON_TIMER_FINAL 4    /* final product fused with the update */
#define DMUON_TIMER_TC 5       /* every tcgen05 GEMM launch (sum) */
#define DMUON_TIMER_SIMT 6     /* every fp32 FFMA GEMM launch (sum) */
#define DMUON_TIMER_COUNT 7

/* Stage timers (the paper reports optimizer-step time per stage of its
 * pipeline, section 4; no API of its own).
 * enable != 0 records a CUDA event pair around every launch of later steps
 * (on the step's stream).  Resets the accumulated times. */
int dmuon_set_timing(dmuon_handle_t h, int32_t enable);
/* Synchronises the recorded events and writes, per DMUON_TIMER_* slot, the
 * accumulated milliseconds to ms[slot] and the number of launches to
 * launches[slot] (either may be NULL).  n = number of slots to write. */
int dmuon_get_timing(dmuon_handle_t h, double* ms, int64_t* launches, int32_t n);

/* ---- errors ------------------------------------------------------------ */

const char* dmuon_last_error(void);       /* thread-local, never NULL */
const char* dmuon_status_string(int status);

/* ---- inspection (tests) ------------------------------------------------ */

#define DMUON_BUF_X 0  /* packed u (and direct-route iterate 0) */
#define DMUON_BUF_RF 1 /* Gram route: fp32 R after the last update; direct: fp32 A.  Held by
                          the fp32 FFMA engine and the split engine (there only its lower
                          triangle is written: it is read only as the next polynomial's b R
                          term); the plain bf16 tensor-core engine has none (the b R term reads
                          the bf16 operand) and the query fails for its buckets. */
#define DMUON_BUF_R_OPERAND 2 /* the operand copy of R / A that the products read
                                 (bf16 on tensor cores, the fp32 buffer otherwise): both
                                 triangles, bitwise symmetric.  With DMUON_ENGINE_TC_SPLIT
                                 each row is [hi | lo], each part ld / 2 elements: hi =
                                 bf16(R), lo = bf16(R - hi) from column ld / 2 on */

/* No counterpart in the paper (test inspection of the symmetric operands of
 * section 2.2).  Byte offset into the bound workspace, leading dimension (elements), batch
 * stride (elements) and element dtype (DMUON_BF16 | DMUON_FP32; may be NULL)
 * of buffer `which` of piece (wave, piece). */
int dmuon_debug_buffer(dmuon_handle_t h, int64_t wave, int64_t piece, int32_t which,
                       uint64_t* offset, int64_t* ld, int64_t* batch_stride, int32_t* elem_type);

/* ---- owner assignment (host only) --------------------------------------
 *
 * DMuon technical summary (gist.science), section 2.3 "compute-aware load
 * balancing": every matrix gets one owner rank, which alone runs its update;
 * the owners minimise the predicted makespan (largest per-rank sum of
 * predicted costs), posed as a mixed-integer program, with a greedy fallback
 * for very large instances.  The single-GPU step has no ranks: this computes
 * the assignment for a multi-rank caller from costs it supplies (e.g. the
 * plan's per-matrix FLOPs below, or measured per-bucket step times).
 *
 * costs:  host array of `count` finite costs >= 0 (any unit).
 * ranks:  number of owner ranks, >= 1.
 * method: DMUON_ASSIGN_GREEDY -- longest processing time first: matrices in
 *         decreasing cost (ties: lower index first), each to the least-loaded
 *         rank so far (ties: lower rank); any count.
 *         DMUON_ASSIGN_EXACT -- the optimum of the makespan program (branch
 *         and bound from the greedy solution); count <= 32, and an instance
 *         whose search exceeds 2e8 nodes returns DMUON_ERR_INVALID_ARG.
 * owner:  host array of `count` ranks in [0, ranks), written.
 * makespan: if not NULL, the largest per-rank sum of the result, each rank's
 *         costs added in increasing matrix index.
 * Returns DMUON_OK or DMUON_ERR_INVALID_ARG (negative / non-finite cost, bad
 * count, ranks or method, NULL array).  No device work. */
#define DMUON_ASSIGN_GREEDY 0
#define DMUON_ASSIGN_EXACT 1
int dmuon_assign_owners(const double* costs, int64_t count, int32_t ranks, int32_t method, int32_t* owner,
                        double* makespan);

/* Per-matrix algorithmic FLOPs of one step at ns_steps, in the order of the
 * plan's shapes (same formulas as dmuon_plan_flops, by each matrix's bucket
 * route; their sum is dmuon_plan_flops' out[0]): a cost model for
 * dmuon_assign_owners.  flops: host array of the plan's count.  Returns
 * DMUON_OK or DMUON_ERR_INVALID_ARG. */
int dmuon_plan_matrix_flops(dmuon_handle_t h, int32_t ns_steps, double* flops);

/* ---- AdamW on the same tensors (comparison step) ------------------------
 *
 * The element-wise optimizer the pages measure DMuon against (technical
 * summary, section 4: "+2 % per-step latency over AdamW"), so that the two
 * optimizer steps can be timed on the same tensors.  Published AdamW with
 * decoupled weight decay and bias correction; per element, in fp32 from the
 * stored values, t = step:
 *   m = beta1*m + (1-beta1)*g,  v = beta2*v + (1-beta2)*g^2
 *   W = (1 - lr*wd)*W - lr/(1-beta1^t) * m / (sqrt(v)/sqrt(1-beta2^t) + eps)
 * and W, m, v are stored back (round to nearest even).
 *
 * params, grads, exp_avgs, exp_avg_sqs: HOST arrays of `count` DEVICE
 * pointers; tensor i holds numels[i] contiguous elements of dtypes[i]
 * (DMUON_BF16 | DMUON_FP32) in all four arrays, each 16-byte aligned.
 * params, exp_avgs and exp_avg_sqs are updated in place; grads are read.
 * Asynchronous on `stream`; allocates nothing (the tensor table is passed as
 * kernel parameters, 256 tensors per launch).  Every wait inside the kernel
 * is bounded; dmuon_adamw_status() reports one that gave up.  Returns DMUON_OK,
 * DMUON_ERR_INVALID_ARG (count, numel, step < 1, betas outside [0, 1),
 * eps <= 0, NULL array), DMUON_ERR_UNSUPPORTED_DTYPE, DMUON_ERR_ALIGN or
 * DMUON_ERR_CUDA. */
int dmuon_adamw_step(void* const* params, const void* const* grads, void* const* exp_avgs,
                     void* const* exp_avg_sqs, const int64_t* numels, const int32_t* dtypes, int64_t count,
                     float lr, float beta1, float beta2, float eps, float wd, int64_t step, void* stream);
/* Synchronous: DMUON_ERR_DEVICE_TIMEOUT if a wait inside an AdamW launch on
 * the current device gave up (about 2 s; its tensors are then only partly
 * updated) since the last call, else DMUON_OK; clears the flag.
 * DMUON_ERR_CUDA if the flag cannot be read. */
int dmuon_adamw_status(void);

/* ---- one small matrix without device allocation ------------------------
 *
 * No counterpart in the paper: an addition for callers that cannot allocate
 * device memory, so cannot give dmuon_step its workspace -- code whose device
 * memory is entirely held by another allocator (a framework's caching pool),
 * or that runs under a fixed memory budget and may not grow device
 * allocations once training started.
 *
 * One Muon step (formula in the file header; defaults only: quintic
 * (3.4445, -4.7750, 2.0315), eps 1e-7, Nesterov, aspect scale) on ONE matrix,
 * in fp32 FFMA arithmetic (the numerics of DMUON_PREC_FP32), in one thread
 * block on `stream`.  param and momentum (device, rows x cols, row-major,
 * dtype DMUON_BF16 | DMUON_FP32, 16-byte aligned) are updated in place; grad
 * is read.  Its scratch is a static device array of 1.3125 MiB that every GPU
 * loading the library holds until exit, which limits the shape to
 * min(rows, cols) <= 128 and rows*cols <= 262144; larger shapes return
 * DMUON_ERR_INVALID_ARG with the limit in dmuon_last_error().  It calls no
 * cudaMalloc, cudaFree or other allocating routine.  The first call on a
 * device (and the first after its context was destroyed and re-created, e.g.
 * by cudaDeviceReset) looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it with the
 * context's unique id; make that first call before any stream capture.
 * All calls on a device share the array: calls that may overlap on the GPU
 * (unordered streams) race on it and must be serialised by the caller.
 * Returns DMUON_OK, DMUON_ERR_INVALID_ARG, DMUON_ERR_ALIGN,
 * DMUON_ERR_UNSUPPORTED_DTYPE or DMUON_ERR_CUDA. */
int dmuon_step_noalloc(void* param, const void* grad, void* momentum, int64_t rows, int64_t cols,
                       int32_t dtype, float lr, float beta, float wd, int32_t ns_steps, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DMUON_H */
