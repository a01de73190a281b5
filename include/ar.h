/*
 * ar.h -- C ABI of the single-GPU allreduce schedule engine (sm_103a).
 *
 * P "virtual ranks" are P buffers of n elements resident in one GPU's HBM.
 * An allreduce combines them elementwise with one associative operator and
 * leaves the result in every buffer ("A Generalization of the Allreduce
 * Operation", introduction: a combination of the processes' vectors that is
 * distributed back to every process).  The call shape follows the in-place,
 * stream-asynchronous, status-returning collective of "All-Reduce, in
 * depth" (The APIs): arguments in, an error code out, work enqueued on a
 * stream.
 *
 * The engine follows a named schedule exactly: it compiles the schedule into
 * rounds of transfers and into each element's reduction tree, then either
 *   - AR_FORM_FUSED: one pass that reads every contribution once, evaluates
 *     the schedule's reduction trees in registers / shared memory and writes
 *     every rank's result (2 P S bytes of HBM traffic, the minimum), or
 *   - AR_FORM_STEP: one kernel launch per round of the schedule, moving and
 *     combining exactly the chunks that round moves.
 * In AR_ORDER_FAITHFUL mode both forms give bit-identical results to the
 * schedule run literally (bf16: every combine rounded to bf16).  In
 * AR_ORDER_FP32ACC mode (fused only) the kernel accumulates all P
 * contributions in fp32 in its own fixed order and rounds once.
 *
 * Conventions common to every function:
 *   - Every function returns ar_status; AR_OK is 0.  Nothing aborts.
 *   - Sizes are element counts unless the name says bytes.
 *   - Pointers named *_bufs are host arrays of P pointers; the pointers are
 *     device (or host, for ar_execute_host) addresses owned by the caller.
 *   - Functions whose comment says "host only" make no CUDA call and may be
 *     used on a machine without a GPU.
 */
#ifndef AR_H
#define AR_H

#if !defined(__CUDACC_RTC__) /* the engine's run-time compiled kernels bring their own */
#include <stddef.h>
#include <stdint.h>
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define AR_MAX_RANKS 64

typedef enum {
    AR_OK = 0,
    AR_ERR_INVALID_ARG = 1, /* null / aliased / overlapping pointers, bad sizes */
    AR_ERR_UNSUPPORTED = 2, /* valid request this engine does not implement   */
    AR_ERR_CUDA = 3,        /* a CUDA runtime call failed                      */
    AR_ERR_NOMEM = 4,       /* host or device allocation failed                */
    AR_ERR_TIMEOUT = 5,     /* a bounded wait inside a kernel gave up          */
    AR_ERR_INTERNAL = 6     /* a kernel met a program kind it does not run, or
                               a guard band around plan scratch was overwritten:
                               an engine fault, never the caller's              */
} ar_status;

typedef enum { AR_INT32 = 0, AR_FLOAT32 = 1, AR_BFLOAT16 = 2 } ar_dtype;

/* Element operations (elementwise operator of "還元演算子" (Reduction operator),
 * binomial-tree section).  The receiving rank's own value is always the left
 * operand.  int32 sum / prod wrap modulo 2^32.  fp32 is IEEE round-to-
 * nearest-even with subnormals.  bf16 widens both operands to fp32, applies
 * the fp32 op and rounds to bf16 (nearest even) after every op.
 * max = a > b ? a : b, min = a < b ? a : b (ties and NaN keep b). */
/* AR_AVG: the sum divided by P, inside the collective ("All-Reduce, in
 * depth", The APIs: ncclAvg divides by the rank count so that no separate
 * scaling pass is needed).  Each result is divided once, where its sum is
 * complete (IEEE fp32 division, round to nearest even; bf16: the bf16 sum
 * widened, divided in fp32, rounded to bf16; FP32ACC: the fp32 sum divided,
 * then rounded).  Float types only: int32 gives AR_ERR_UNSUPPORTED. */
typedef enum { AR_SUM = 0, AR_PROD = 1, AR_MAX = 2, AR_MIN = 3, AR_AVG = 4 } ar_op;

/* Schedules.
 *  AR_RING        ring reduce-scatter + all-gather over P chunks; rank r
 *                 sends to r + 1 ("All-Reduce, in depth", The ring
 *                 algorithm; "A Generalization of the Allreduce Operation",
 *                 ring as the cyclic-group straightforward algorithm, Fig. 5).
 *                 2(P-1) rounds.
 *  AR_BINOMIAL    binomial-tree reduce to rank 0 (x_i <- x_i (+) x_{i+2^k})
 *                 then broadcast ("還元演算子", binomial tree).  2 ceil(log2 P).
 *  AR_RH          recursive halving reduce-scatter + doubling all-gather,
 *                 distance P/2 first; the bandwidth-optimal generalized
 *                 algorithm with the XOR group ("A Generalization ...",
 *                 remark after eq. 25, Table 1.b).  2 log2 P rounds.
 *  AR_RD          recursive doubling, whole vectors, distance 1 first.
 *                 log2 P rounds.
 *  AR_HYBRID      k1 halving rounds, recursive doubling on the block each rank
 *                 then owns, k1 doubling rounds ("A Generalization ...",
 *                 introduction, the classic hybrid).  log2 P + k1 rounds.
 *                 RH, RD and the hybrid take any P: with P' the largest power
 *                 of two <= P, a preparation round folds rank P'+i into rank i,
 *                 the schedule runs on ranks 0..P'-1 and a finalization round
 *                 copies rank i's result to rank P'+i ("A Generalization ...",
 *                 introduction, the workaround for non-power-of-two counts):
 *                 two more rounds; k1 <= log2 P'.
 *  AR_GENERALIZED the group-theoretic generalized allreduce for any P
 *                 ("A Generalization ...", eqs. 17-44): cyclic group (any P)
 *                 or XOR group (P = 2^k); r distribution steps removed,
 *                 0 <= r <= ceil(log2 P); 2 ceil(log2 P) - r rounds.
 *  AR_AHC         asymmetric hierarchical allreduce (AHC, HCCL, Description):
 *                 contiguous groups of the given sizes, LCM x G chunks, ring
 *                 reduce-scatter inside each group, ring allreduce between the
 *                 logical devices with identical IDs, ring all-gather inside
 *                 each group.
 *  AR_PIPELINE    pipelined chain reduce over `blocks` blocks (ceil split):
 *                 in round t unit i passes block t - i to unit i + 1, which
 *                 combines it; the last unit holds every block after
 *                 p + blocks - 2 rounds ("還元演算子" (Reduction operator),
 *                 pipelined algorithm); then the mirror-image pipelined
 *                 broadcast.  2 (p + blocks - 2) rounds. */
typedef enum {
    AR_RING = 0, AR_BINOMIAL = 1, AR_RH = 2, AR_RD = 3,
    AR_HYBRID = 4, AR_GENERALIZED = 5, AR_AHC = 6, AR_PIPELINE = 7
} ar_algo;

enum { AR_FORM_FUSED = 0, AR_FORM_STEP = 1 };
enum { AR_ORDER_FAITHFUL = 0, AR_ORDER_FP32ACC = 1 };
enum { AR_GROUP_CYCLIC = 0, AR_GROUP_XOR = 1 };
/* Which part of the schedule runs ("All-Reduce, in depth", The APIs: FSDP and
 * ZeRO use the reduce-scatter for gradients and the all-gather for
 * parameters).  Available for AR_RING, AR_RH and AR_GENERALIZED with r = 0.
 *  REDUCE_SCATTER: afterwards every chunk's owner holds its full reduction
 *    (ring: chunk k on rank k-1 mod P; RH / generalized: chunk k on rank k;
 *    RH with P not a power of two: ranks 0..P'-1 over P' chunks); the other
 *    chunks of every buffer are unspecified.
 *  ALL_GATHER: the owners' chunks (same ownership) are copied to every rank;
 *    the other chunks' inputs are ignored. */
enum { AR_PHASE_ALLREDUCE = 0, AR_PHASE_REDUCE_SCATTER = 1, AR_PHASE_ALL_GATHER = 2 };

typedef struct {
    int form;               /* AR_FORM_FUSED or AR_FORM_STEP                      */
    int order;              /* AR_ORDER_FAITHFUL or AR_ORDER_FP32ACC (fused only) */
    int group;              /* AR_GENERALIZED: AR_GROUP_CYCLIC or AR_GROUP_XOR    */
    int r;                  /* AR_GENERALIZED: removed distribution steps         */
    int k1;                 /* AR_HYBRID: halving steps, 0..log2 P                */
    int n_groups;           /* AR_AHC: number of groups G                         */
    const int* group_sizes; /* AR_AHC: G sizes adding up to P (copied at create)  */
    int blocks;             /* AR_PIPELINE: blocks m, 1..4096 (0 means 1)         */
    int phase;              /* AR_PHASE_*; 0 = the whole allreduce               */
    int jit;                /* DAG programs as run-time compiled code: AR_JIT_*  */
} ar_params;

/* ar_params.jit.  A plan whose staged launches evaluate DAG programs
 * (rank-specific results, rounds with cyclic transfers) can run them as
 * straight-line code compiled for the plan with NVRTC when the plan is
 * created (bit-identical results; see ar_plan_info.kernels).  AUTO: when
 * those launches move at least 16 MiB and the programs hold at most 4096
 * instruction words; ON: whenever they fit that size; OFF: always
 * interpret.  Without NVRTC on the system the plan interprets. */
enum { AR_JIT_AUTO = 0, AR_JIT_ON = 1, AR_JIT_OFF = -1 };

typedef struct {
    int P;
    int dtype, op, algo, form, order, phase;
    uint64_t n;                  /* elements per rank                              */
    int steps;                   /* rounds of the schedule                         */
    uint64_t sent_bytes_max;     /* max over ranks of bytes sent, all rounds       */
    uint64_t sent_bytes_total;   /* bytes sent by all ranks, all rounds            */
    uint64_t combines;           /* element combines the schedule performs         */
    int max_slots;               /* partials a rank holds per chunk at once (>= 1) */
    int n_segments;              /* element ranges with one reduction tree each    */
    /* Filled for plans (ar_plan_query); zero for schedules. */
    uint64_t hbm_bytes;          /* algorithmic HBM bytes moved by one execute     */
    uint64_t scratch_bytes;      /* device scratch the plan owns                   */
    int launches;                /* kernel launches per execute (aligned buffers)  */
    int tile_bytes;              /* bytes per input tile in the staged kernel      */
    int n_programs;              /* distinct tile programs                         */
    uint64_t n_items;            /* work items over all launches                   */
    int kernels;                 /* kernels the aligned launches use: AR_KERNEL_*  */
    uint64_t messages;           /* transfers over all rounds (one per message)    */
} ar_plan_info;

/* ar_plan_info.kernels bits: the rank-streaming kernel (chains, single trees,
 * fp32 accumulation), the staged kernel (DAG programs), the element-wise
 * kernel (unaligned edges and tiny passes), DAG_JIT when the staged
 * launches run the plan's run-time compiled DAG kernel, WORD_JIT for the
 * run-time compiled word kernel (launches whose DAG programs it runs with
 * one 32-bit word of every input buffer per thread in registers),
 * CHAIN_WORD for the chain word kernel (chains of small and mid-sized
 * passes, the same way), COPY for the copy kernel (fused passes whose
 * programs copy one input to their outputs: the all-gathers), and FEW for the
 * few-input kernel (a CTA per 16 KB item: fused passes of chains and fp32
 * accumulations of 2 to 16 inputs, of more in passes of at least 1.5 GiB,
 * and of single trees of up to 8 leaves that write every rank). */
enum { AR_KERNEL_STREAM = 1, AR_KERNEL_STAGED = 2, AR_KERNEL_ELEMENTWISE = 4, AR_KERNEL_DAG_JIT = 8,
       AR_KERNEL_WORD_JIT = 16, AR_KERNEL_CHAIN_WORD = 32, AR_KERNEL_COPY = 64, AR_KERNEL_FEW = 128 };

typedef struct ar_schedule_s* ar_schedule_t;
typedef struct ar_plan_s* ar_plan_t;

/* ---- schedule compiler (host only) ---------------------------------------
 * ar_schedule_create compiles (P, n, dtype, op, algo, params) into rounds of
 * transfers and per-element reduction trees.  P in 1..AR_MAX_RANKS (larger P:
 * AR_ERR_UNSUPPORTED).  params may be NULL for the defaults (fused, faithful,
 * cyclic, r = 0, k1 = 0).  On success *out owns host memory released by
 * ar_schedule_destroy.  Errors: AR_ERR_INVALID_ARG (P < 1, unknown enum, null
 * out, AHC sizes not adding up to P, r or k1 out of range),
 * AR_ERR_UNSUPPORTED (P > AR_MAX_RANKS, the XOR group with P not a power of
 * two, AHC with more than 4096 chunks, FP32ACC with the step form),
 * AR_ERR_NOMEM. */
ar_status ar_schedule_create(int P, uint64_t n, ar_dtype dtype, ar_op op, ar_algo algo,
                             const ar_params* params, ar_schedule_t* out);
ar_status ar_schedule_destroy(ar_schedule_t s);
/* Counters of the compiled schedule (hbm / plan fields left zero). */
ar_status ar_schedule_query(ar_schedule_t s, ar_plan_info* info);
/* Elements each rank sends in round `step` (0-based): writes P counts to
 * elems_per_rank.  AR_ERR_INVALID_ARG if step is out of range. */
ar_status ar_schedule_step_sent(ar_schedule_t s, int step, uint64_t* elems_per_rank);
/* The reduction tree the schedule leaves in element `elem` of rank `rank`, as
 * text: a leaf is a rank number, "(a+b)" is a combine whose left operand a is
 * the receiver's value.  Writes at most cap bytes including the terminating
 * NUL; *needed receives the full length + 1.  AR_ERR_INVALID_ARG when the
 * buffer is too small (nothing useful written) or indices are out of range. */
ar_status ar_schedule_tree(ar_schedule_t s, int rank, uint64_t elem, char* buf, size_t cap,
                           size_t* needed);

/* ---- cost model and step selection (host only) ----------------------------
 * "A Generalization of the Allreduce Operation", the complexity of the
 * algorithm with r removed distribution steps (eq. 36) and the r that
 * minimises it (eq. 37): every step costs a latency alpha, every byte sent
 * beta, every byte reduced gamma.  On one GPU the messages of all P ranks in
 * a round share the HBM, so for the engine's step form (one launch per
 * round) a schedule costs
 *     alpha * rounds + beta * (bytes sent, all ranks)
 *                    + gamma * (bytes combined, all ranks)
 *                    + delta * (messages, all ranks and rounds)
 * i.e. the page's per-process beta and gamma are P times these.  delta is
 * the engine's own term, not on the page: each message is at least one work
 * item, which costs time however few its bytes (0 gives the page's model;
 * eqs. 36-37 and ar_cost_optimal_r leave it out).  The fused form moves
 * 2 P S bytes in one launch whatever the schedule, so the model selects
 * among step-form schedules only. */
typedef struct {
    double alpha_us;              /* per round (one kernel launch)           */
    double beta_us_per_byte;      /* per byte sent, summed over ranks        */
    double gamma_us_per_byte;     /* per byte combined, summed over ranks    */
    double delta_us_per_message;  /* per message (transfer), summed          */
} ar_cost_model;

/* The step-form model fitted on GB300 (bench.py --costmodel). */
ar_status ar_cost_model_default(ar_cost_model* out);
/* Predicted step-form time of a compiled schedule under the model: from its
 * rounds, bytes sent and combines.  AR_ERR_INVALID_ARG on null arguments. */
ar_status ar_cost_predict(ar_schedule_t s, const ar_cost_model* model, double* us);
/* Eq. (37) for P ranks of bytes_per_rank bytes (m): the real minimiser
 * r* = log2(alpha / (ln 2 * m * (L beta + (2L - 2) gamma))) of eq. (36),
 * L = ceil(log2 P), taken to whichever neighbouring integer eq. (36) rates
 * lower and clamped to 0..L-1 (eq. 36 holds for r < L; the latency-optimal
 * r = L is costed separately on the page, and by ar_cost_select here).
 * P = 1 gives 0.  AR_ERR_INVALID_ARG on P < 1, P > AR_MAX_RANKS, m = 0, a
 * non-positive alpha, negative beta or gamma, or null pointers. */
ar_status ar_cost_optimal_r(int P, uint64_t bytes_per_rank, const ar_cost_model* model, int* r);
/* The step-form schedule with the lowest predicted time among the ring, the
 * binomial tree, RD, RH, the hybrid for every k1 and the cyclic generalized
 * schedule for every r (the page's ring / tree switch and r choice made on
 * exact counters).  Writes the algorithm, its params (step form, faithful)
 * and the prediction; ties keep the earlier candidate in that order.  Errors
 * as ar_schedule_create. */
ar_status ar_cost_select(int P, uint64_t n, ar_dtype dtype, ar_op op, const ar_cost_model* model,
                         ar_algo* algo, ar_params* params, double* us);

/* Host only: compiles, without a GPU, the run-time compiled kernels a plan
 * with these parameters would use with params.jit = AR_JIT_ON (the staged DAG
 * kernel and the word kernel); *cubin_bytes receives their total code size, 0
 * when the plan has no DAG program.  AR_ERR_UNSUPPORTED when NVRTC cannot be
 * loaded, AR_ERR_CUDA when a compilation fails. */
ar_status ar_schedule_dag_kernel(ar_schedule_t s, size_t* cubin_bytes);

/* Host only: the work a plan with these parameters would launch, lowered as
 * ar_plan_create lowers it (no device needed) and checked two ways, each by
 * code apart from the lowering's own:
 *   tiling_ok   every launch set's bulk and edge items tile its element
 *               ranges exactly, program by program (no gap, no overlap), and
 *               every bulk item is 16-byte aligned in offset and length;
 *   windows_ok  the windows of the pipelined host path (ar_execute_host) are
 *               consecutive over [0, n) and every item lies inside its
 *               window's elements (1 when there are no windows).
 * wave_balance: over the rank-streaming launch sets, the largest byte share
 * one of 152 CTAs takes when the items are dealt round robin, over the mean
 * share (1 = even).
 * AR_ERR_INVALID_ARG on null arguments, AR_ERR_NOMEM. */
typedef struct {
    uint64_t items;          /* bulk + edge items over all launch sets          */
    int launch_sets;         /* launch sets (one per round; one when fused)     */
    int windows;             /* windows of the host path; 0: one pass           */
    int tiling_ok;           /* 1 or 0, as above                                */
    int windows_ok;          /* 1 or 0, as above                                */
    double wave_balance;     /* >= 1, as above (1 with no streamed items)       */
    int stream_tile_bytes;   /* rank tile of the rank-streaming kernel          */
    int stream_stages;       /* its pipeline depth                              */
    int staged_tile_bytes;   /* input tile of the staged kernel (DAG programs)  */
    int staged_stages;       /* its pipeline depth                              */
    uint64_t dag_words;      /* instruction words of the staged launches' DAG
                                programs (what a run-time compiled DAG kernel
                                holds)                                          */
    int word_sets;           /* launch sets on the run-time compiled word kernel
                                (as a plan with params.jit would lower them
                                here, NVRTC permitting)                         */
    uint64_t word_kernel_words; /* instruction words of their programs           */
    int stream_tmem;         /* 1: the tree stack lives in tensor memory        */
    int copy_sets;           /* launch sets on the copy kernel                  */
    int few_sets;            /* launch sets on the few-input kernel             */
} ar_lowering_info;
ar_status ar_schedule_lowering(ar_schedule_t s, ar_lowering_info* out);

/* ---- plans (need a CUDA device) -------------------------------------------
 * ar_plan_create compiles the schedule, lowers it to tile programs for the
 * chosen form and uploads them to the current device; it allocates the
 * plan's device tables and, for the step form of schedules that keep two
 * partials per chunk, scratch.  No kernel runs.  Errors as
 * ar_schedule_create plus AR_ERR_CUDA / AR_ERR_NOMEM. */
ar_status ar_plan_create(int P, uint64_t n, ar_dtype dtype, ar_op op, ar_algo algo,
                         const ar_params* params, ar_plan_t* out);
/* Frees the plan's host and device memory.  Synchronises the device first. */
ar_status ar_plan_destroy(ar_plan_t plan);
/* Counters of the schedule and of its lowering. */
ar_status ar_plan_query(ar_plan_t plan, ar_plan_info* info);
/* Checks P rank buffers as ar_execute does, launching nothing: non-null,
 * aligned to the element size, pairwise disjoint, and each one device memory
 * of the plan's device (cudaMalloc'd, from a pool, or managed) whose n
 * elements lie inside the allocation holding it ("All-Reduce, in depth", The
 * APIs: the collective works on device buffers the caller owns).  Pageable or
 * pinned host memory, another device's memory, and a pointer whose n
 * elements run past its allocation give AR_ERR_INVALID_ARG.  (The extent is
 * checked where the driver reports allocation ranges.)  With n = 0: AR_OK. */
ar_status ar_plan_check_buffers(ar_plan_t plan, void* const* rank_bufs);
/* Enqueues the allreduce on `stream` (0 = legacy default stream) and returns.
 * rank_bufs: host array of P device pointers, each to n elements of the
 * plan's dtype on the plan's device, distinct, non-overlapping and aligned
 * to the element size (AR_ERR_INVALID_ARG otherwise, before any launch).
 * Residency and extent are checked as by ar_plan_check_buffers whenever the
 * pointer set differs from the last one this plan accepted (a repeated set
 * is not re-queried: freeing a buffer and passing its pointer again is the
 * caller's error).  With n = 0 the call is a no-op and the pointers are not
 * inspected.  Every buffer is both input and output.
 * 16-byte aligned buffers use the tiled kernels (rank-streaming, staged); any
 * other alignment is valid and takes a slower element-wise path.  Executes of one plan must be
 * ordered on one stream (they share the plan's scratch).  The launch itself
 * is checked (AR_ERR_CUDA); kernel-side failures are reported by
 * ar_plan_check. */
ar_status ar_execute(ar_plan_t plan, void* const* rank_bufs, void* stream);
/* End-to-end variant: copies P host buffers to the P device buffers (checked
 * as ar_execute checks them), runs the
 * allreduce and copies every device buffer back to its host buffer, then
 * synchronises `stream`.  Large fused plans on 16-byte-aligned device buffers
 * are processed in element windows of about 128 MB: the copies in of window
 * w+1 and out of window w-1 run on two internal streams of the plan while
 * window w is reduced on `stream` (every element's result depends only on
 * that element of every rank).  Otherwise: all copies in, the allreduce, all
 * copies out, on `stream`.  One cudaMemcpyAsync per buffer, window and
 * direction.  host_bufs should be pinned for full speed.  Calls on one plan
 * must not overlap (they share the internal streams). */
ar_status ar_execute_host(ar_plan_t plan, void* const* host_bufs, void* const* dev_bufs,
                          void* stream);
/* Self-test of the bounded waits every kernel uses (no plan needed): launches
 * one CTA that waits on an mbarrier nothing ever completes; the wait gives up
 * after timeout_ms (1..10000) exactly as a kernel's wait does after two
 * seconds, records the status bit and returns, so the device stays usable.
 * Synchronises `stream`.  Returns AR_ERR_TIMEOUT when the wait gave up (the
 * expected result), AR_OK if it completed, AR_ERR_INVALID_ARG for a timeout
 * out of range, AR_ERR_CUDA / AR_ERR_NOMEM on failures. */
ar_status ar_selftest_bounded_wait(uint32_t timeout_ms, void* stream);
/* Synchronises the device and reads the plan's device status word and the
 * guard bands around its scratch: AR_OK; AR_ERR_INTERNAL if a kernel met a
 * program kind it does not run or a guard band was overwritten (this takes
 * precedence); AR_ERR_TIMEOUT if a bounded wait in a kernel gave up.  The
 * status word is cleared after a failure is read.  AR_ERR_CUDA if
 * synchronisation fails. */
ar_status ar_plan_check(ar_plan_t plan);

/* Static text for a status code (never NULL). */
const char* ar_status_string(ar_status s);

/* ---- allreduce without device allocation ----------------------------------
 * The pages have no counterpart to this call; it exists for callers that must
 * not allocate device memory: a process whose GPU memory is already reserved
 * in full by another allocator (a framework's caching pool), a service with a
 * device-memory budget fixed at start-up, or a hot path that cannot pay for
 * cudaMalloc / cudaFree's implicit device-wide synchronisation.  Such a caller
 * cannot create a plan, because ar_plan_create allocates the plan's tables,
 * status word and scratch.
 *
 * ar_allreduce_static compiles the schedule on the host (as ar_plan_create
 * does) and runs the same kernels on the same rank buffers (same arguments,
 * layout and result as ar_plan_create + ar_execute), but puts every byte of
 * device scratch -- the status word, the tile-program tables and, for the step
 * form, the second partial of a chunk -- in one file-scope static device array
 * of AR_STATIC_SCRATCH_BYTES that every GPU loading the library holds until the
 * process exits.  It calls no cudaMalloc, cudaFree or other allocating routine;
 * host memory is used only while the schedule is compiled.
 *   - Set-up: the first call made with a given device current resolves the
 *     array's device address (cudaGetSymbolAddress) for that device; make that
 *     first call before any stream capture.  The address is kept for the life
 *     of the process: a cudaDeviceReset after the first call is not supported.
 *   - Limits: AR_ERR_UNSUPPORTED when the schedule's tables need more than
 *     AR_STATIC_TABLE_BYTES or its partial slots more than what is left of the
 *     array (AR_STATIC_SCRATCH_BYTES - AR_STATIC_TABLE_BYTES - 256 bytes).
 *   - Sharing: every call reuses the one array and overwrites the previous
 *     call's contents (the status word is cleared, the tables rewritten, on
 *     `stream`).  Calls that can overlap on the GPU race with each other:
 *     issue them on one stream, or order them with events.
 *   - Errors as ar_plan_create + ar_execute, the rank buffers checked as by
 *     ar_plan_check_buffers on every call.  Kernel-side failures (a bounded
 *     wait that gave up, a program a kernel does not run) land in the array's
 *     status word, which each call clears when it starts: read it with
 *     ar_allreduce_static_check after a call and before the next one. */
#define AR_STATIC_SCRATCH_BYTES (32u << 20)
#define AR_STATIC_TABLE_BYTES (1u << 20)
ar_status ar_allreduce_static(int P, uint64_t n, ar_dtype dtype, ar_op op, ar_algo algo,
                              const ar_params* params, void* const* rank_bufs, void* stream);
/* Synchronises `stream`, then reads and clears the status word the kernels of
 * ar_allreduce_static calls on the current device write: AR_OK (also when no
 * call has run on this device), AR_ERR_INTERNAL if a kernel met a program it
 * does not run, AR_ERR_TIMEOUT if a bounded wait gave up, AR_ERR_CUDA if the
 * copy or the synchronisation fails.  Allocates nothing. */
ar_status ar_allreduce_static_check(void* stream);

#ifdef __cplusplus
}
#endif
#endif /* AR_H */
