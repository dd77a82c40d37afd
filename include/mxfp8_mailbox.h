/*
 * mxfp8_mailbox.h -- C ABI of the MXFP8 low-batch publishing GEMM and its
 * Lamport mailbox (one GPU, sm_103a).
 *
 * The operation (page "vllm.models.deepseek_v41.nvidia.specialized_decode.
 * boundary.publishing_gemm", module description "GEMM structure" and
 * "Ordering"):
 *
 *   C[t][n] = sum_k W[n][k] * x[t][k]        t < m <= 8, n < N, k < K
 *
 * with W and x MXFP8 (E4M3FN elements, one E8M0FNU scale per 32-element K
 * block), FP32 accumulation and a BF16 result.  The GEMM's epilogue publishes
 * every output, rounded to BF16 with negative zero cleared, into generation
 * stage_state[0] of a Lamport mailbox and sets stage_state[1] to that
 * generation.  A consumer (page "vllm.models.deepseek_v41.nvidia.ops.cute_dsl.
 * all_gather", module description steps 2 and 3), launched as the GEMM's
 * programmatic dependent, polls the slots until no word is the sentinel,
 * copies them out, stores the sentinel back and advances the generation.
 *
 * Conventions for every function below:
 *  - Pointers named "device" are device (HBM) addresses owned by the caller;
 *    the library never allocates, frees or retains them beyond what is stated.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Every launch is asynchronous on that stream; calls on one
 *    mailbox must be issued in order on one stream and must not overlap.
 *  - Argument errors are found on the host before any launch; the function
 *    then returns MXFP8_ERR_INVALID or MXFP8_ERR_UNSUPPORTED, launches
 *    nothing, and mxfp8_last_error() describes the problem.
 *  - Device-side waits: every poll of the mailbox and every wait of the
 *    GEMM's pipeline (mbarriers, the split-K exchange) has a time limit
 *    (mailbox_consume's timeout_ns; the descriptor's wait_limit_ms); one that
 *    runs out sets a bit in stage_state[3] (read with mxfp8_mailbox_status)
 *    and the kernel drains instead of hanging.  Two waits have no time limit
 *    in hardware: tcgen05.alloc (tensor-memory columns) and the cluster
 *    barriers of split-K.  They are kept from depending on each other by
 *    construction: a CTA allocates at most half of an SM's tensor memory,
 *    and a clustered launch asks for enough shared memory that at most two
 *    of its CTAs share an SM.
 *  - All functions are thread-compatible; mxfp8_last_error() is per thread.
 */
#ifndef MXFP8_MAILBOX_H
#define MXFP8_MAILBOX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Three generations (all_gather page, module description step 3). */
#define MXFP8_MAILBOX_GENERATIONS 3
/* The Lamport sentinel word, FP32 negative zero / INT32_MIN (all_gather page,
 * module description step 1). */
#define MXFP8_MAILBOX_SENTINEL 0x80000000u
/* At most eight activation rows (publishing_gemm page, PublishingMxfp8Linear.
 * supports: 0 < num_tokens <= min(LOW_BATCH_MAX_ROWS, capacity)). */
#define MXFP8_MAX_ROWS 8

/* Bits of stage_state[3]. */
#define MXFP8_FLAG_POLL_TIMEOUT 0x1 /* the consumer's poll ran out of time   */
#define MXFP8_FLAG_GEMM_TIMEOUT 0x2 /* a GEMM pipeline wait ran out of time  */
#define MXFP8_FLAG_BAD_STATE 0x4    /* a kernel read a generation not in 0..2 */

typedef enum mxfp8_status {
  MXFP8_OK = 0,
  MXFP8_ERR_INVALID = 1,     /* bad argument: NULL, misaligned, bad shape        */
  MXFP8_ERR_UNSUPPORTED = 2, /* well-formed but not taken (m, split_k, stages)   */
  MXFP8_ERR_CUDA = 3,        /* a CUDA runtime call failed                       */
  MXFP8_ERR_TIMEOUT = 4,     /* a device-side wait ran out (mxfp8_mailbox_status) */
  MXFP8_ERR_STATE = 5        /* the state words hold a generation not in 0..2    */
} mxfp8_status;

/* Shape and tactic of one publishing GEMM (the tactic fields follow the
 * publishing_gemm page's (cta_k, ab_stages, sfb_tmem_stages, split_k); the x
 * scales ride in the same ring as the W scales, so there is no separate sfb
 * stage count).  acc_blocks is this library's addition: how many 32-wide K
 * blocks the tensor core sums in one accumulator before the epilogue folds
 * the partial into its compensated (two-float) sum; 1 keeps every output
 * within 2 BF16 ULPs of the exact sum on near-cancelling outputs that a single
 * long FP32 accumulation misses.  Zero in a tactic field asks the library to
 * choose. */
typedef struct mxfp8_gemm_desc {
  int32_t n;          /* output columns N ("hidden"): a positive multiple of 128     */
  int32_t k;          /* reduction length K: a positive multiple of 32, <= 32768     */
  int32_t capacity_m; /* mailbox rows per generation: 1..8                           */
  int32_t split_k;    /* cluster split-K S: 1, 2, 4 (the page's sizes) or 8 (a
                         portable cluster, one token per CTA; measured slower than
                         4 where both fit, so never chosen); 0 = choose among 1, 2,
                         4: the largest with at most two CTAs per SM and >= 2 K
                         tiles per split                                               */
  int32_t cta_k;      /* K per pipeline stage, in units of fold: 128 (0 = 128) or 256.
                         With 256 a stage holds two 128-wide K tiles (128 fold K each)
                         that share one full and one empty barrier and come in one W
                         copy, one W-scale copy and one x load; accumulator and scale
                         slots stay per tile, so the results are bit-identical to
                         128's.  256 takes fold 1, 2 or 4, split_k 1, 2 or 4,
                         acc_blocks 4, the 32x32b read-out, and pipes such that
                         2 x pipes divides the accumulator ring (8 slots; 4 at fold 4,
                         so at most 2 pipes there).  `stages` then counts 256-wide
                         stages.  Measured on GB300: 2-6 % less GEMM time at
                         K = 2048, slower at K >= 4096 (fold 4's 2 pipes, shorter
                         rings), so 0 chooses 128.                                     */
  int32_t stages;     /* shared-memory ring depth: 2..16 (0 = choose)                */
  int32_t acc_blocks; /* K blocks per promoted partial sum: 1 or 4 (0 = 4)           */
  int32_t w_layout;   /* MXFP8_W_IN_PLACE or MXFP8_W_TILED (0 = choose)              */
  int32_t l2_prefetch;/* W stages past the ring each of the grid's later CTAs warms in
                         L2 before its grid wait, so HBM keeps streaming while the
                         previous kernel finishes and the grid wait holds the ring:
                         1..64, -1 = none, 0 = choose (16)                              */
  int32_t pipes;      /* producer lanes and MMA-issuing warps sharing the ring: 1, 2
                         or 4, dividing `stages` (stage i and its ring slots belong to
                         pipe i % pipes).  0 = choose: 4 when the grid has at most one
                         CTA per SM and 4 divides the ring, else 2 on an even ring, else
                         1.  One thread's bulk copies and tensor-core instructions are
                         served one after another, so few-CTA grids need several.     */
  int32_t tmem_load;  /* how the epilogue reads accumulators out of tensor memory:
                         MXFP8_TMEM_LOAD_32X32B (0 = this: thread = output column) or
                         MXFP8_TMEM_LOAD_16X256B (the gemm page's default shape, with
                         column_lanes = 1 being the 32x32b case: a thread holds 4
                         columns x 2 tokens and one warp-local transpose follows the
                         main loop).  The two give identical bits.                     */
  int32_t fold;       /* K pieces stacked in the MMA's 128 rows: 1, 2, 4 or 8.  A CTA then
                         owns 128/fold output columns, its A operand holding fold
                         consecutive 128-wide K pieces of those weight rows and its B
                         operand the matching fold groups of 8 activation columns
                         (N = 8 fold); only the diagonal blocks of the product are
                         kept.  Each stage stays 16 KB of W and 4 MMAs; the grid has
                         fold times more CTAs, for shapes whose N/128 x split_k CTAs
                         leave SMs idle.  fold > 1 takes split_k 1, 2 or 4, acc_blocks
                         4 and the 32x32b read-out; fold 8 takes split_k 1 and at most
                         2 pipes (its accumulator ring holds 2 slots of 64 tensor-memory
                         columns).  0 = choose: the largest fold that keeps the grid
                         within one CTA per SM, pads K no further and leaves every
                         split a stage (fold 8 only unsplit and from 8 stages per CTA;
                         1 when the other fields ask for what folding cannot take).   */
  int32_t l2_prefetch_early;/* W stages past the ring that each of the first 70 % of
                         the grid's CTAs warms in L2 (l2_prefetch covers the rest).
                         Those launch while the previous kernel still streams, and
                         a deep prefetch would take HBM from it: 1..64, -1 = none,
                         0 = choose (an explicit l2_prefetch's value, else 4 with
                         two CTAs per SM and none with one; measured on GB300: the
                         N=7168, K=16384, S=4 chain 21.44 -> 20.25 us per call
                         against 6 stages for every CTA)                              */
  int32_t wait_limit_ms;/* how long one wait of the GEMM's pipeline (a ring slot, an
                         accumulator slot, the split-K exchange) may last before it
                         gives up: it then sets MXFP8_FLAG_GEMM_TIMEOUT in
                         stage_state[3] and the kernel drains its copies in flight
                         and exits (the values it wrote are then meaningless).
                         1..60000, 0 = 2000.  A run that times out takes at most a
                         few such limits before it exits.                             */
} mxfp8_gemm_desc;

/* Where the GEMM streams W from.  IN_PLACE: the caller's [N][K] buffer,
 * through 2-D TMA tiles (the handle borrows w).  TILED: a copy made once at
 * create inside the workspace, laid out stage by stage (128 rows x 128 K
 * bytes; 128/fold rows x fold K pieces when folded), already in the order
 * shared memory holds it, so every pipeline stage is one contiguous 16 KB
 * read; the caller's w is not read after create. */
#define MXFP8_W_IN_PLACE 1
#define MXFP8_W_TILED 2

/* Accumulator read-out shapes (tcgen05.ld), publishing_gemm page,
 * epilog_warp (16x256b, or 32x32b when column_lanes == 1). */
#define MXFP8_TMEM_LOAD_32X32B 1
#define MXFP8_TMEM_LOAD_16X256B 2

typedef struct mxfp8_publish_gemm mxfp8_publish_gemm; /* opaque */

/* Bytes of a mailbox of `capacity_m` rows and `n` columns: 3 generations x
 * capacity_m x n BF16 values, as 16-byte packs (all_gather page, module
 * description: mailbox[generation][rank][pack], here with one rank).  The
 * mailbox is laid out [generation][row][column] BF16, row-major.  Returns 0
 * for an invalid shape (capacity_m not in 1..8, n not a positive multiple of
 * 8). */
size_t mxfp8_mailbox_bytes(int32_t capacity_m, int32_t n);

/* Arm a mailbox (all_gather page, LamportAllGather.__init__: every slot
 * starts as the sentinel, the state is zero).  mailbox: device, 16-byte
 * aligned, mxfp8_mailbox_bytes(capacity_m, n) bytes.  stage_state: device,
 * 16-byte aligned int32[4]: [0] next generation (written by the consumer,
 * read by the GEMM), [1] active generation (written by the GEMM, read by the
 * consumer), [2] zero (unused by this protocol), [3] error flags.  Launches one
 * kernel on `stream`. */
mxfp8_status mxfp8_mailbox_init(void* mailbox, int32_t* stage_state, int32_t capacity_m,
                                int32_t n, void* stream);

/* Device bytes the handle needs: W's scale factors re-laid once at create
 * into the tiled order the tensor-core copy reads (N/128 x ceil(K/128) chunks
 * of 512 bytes), plus, for MXFP8_W_TILED (and for w_layout 0, which chooses
 * it), the tiled copy of W (N x ceil(K/128) x 128 bytes).  With an explicit
 * fold f, K rounds up to a multiple of 128 f instead (N/(128/f) x
 * ceil(K/(128 f)) chunks; N x ceil(K/(128 f)) x 128 f bytes of W); fold 0
 * sizes like 1, as it only chooses folds that pad K no further.  0 for an
 * invalid descriptor. */
size_t mxfp8_publish_gemm_workspace_bytes(const mxfp8_gemm_desc* desc);

/* Build a publishing GEMM for one weight and one mailbox (publishing_gemm
 * page, module description "Addresses": the mailbox, stage-state address,
 * capacity and hidden size are fixed per publisher, whose buffers live as
 * long as it does).
 *  w:          device, 16-byte aligned, [N][K] E4M3FN bytes, K contiguous.
 *  w_scale:    device, [N][K/32] E8M0FNU bytes, row-major.
 *  mailbox:    device, 16-byte aligned, as for mxfp8_mailbox_init.
 *  stage_state:device, 16-byte aligned int32[4].
 *  workspace:  device, 256-byte aligned, >= mxfp8_publish_gemm_workspace_bytes.
 * The handle borrows mailbox, stage_state and workspace until destroy, and w
 * too for MXFP8_W_IN_PLACE (w_scale, and w for MXFP8_W_TILED, are read once,
 * by kernels launched here on `stream`, and not afterwards).  On success *out
 * receives the handle.
 * Ordering: the kernels launched here write the workspace, which every run
 * reads.  The first run (of any kind) on the handle must therefore be ordered
 * after them: issued on the same `stream`, or on a stream made to wait for it
 * (an event, or a synchronisation).  That first run launches with a full
 * stream dependency; later runs overlap their weight loads with the kernel
 * before them (see mxfp8_publish_gemm_run). */
mxfp8_status mxfp8_publish_gemm_create(const mxfp8_gemm_desc* desc, const void* w,
                                       const void* w_scale, void* mailbox,
                                       int32_t* stage_state, void* workspace,
                                       size_t workspace_bytes, void* stream,
                                       mxfp8_publish_gemm** out);

/* The resolved shape and tactic of a handle (split_k, cta_k, stages,
 * acc_blocks filled in), plus the dynamic shared memory, tensor-memory columns and grid size of
 * its launch. */
mxfp8_status mxfp8_publish_gemm_config(const mxfp8_publish_gemm* gemm, mxfp8_gemm_desc* desc,
                                       int32_t* smem_bytes, int32_t* tmem_columns,
                                       int32_t* grid_ctas);

/* The tactic mxfp8_publish_gemm_create would resolve for `desc` on a device
 * with `sms` SMs, `smem_per_sm` bytes of shared memory per SM and
 * `smem_per_block_optin` bytes per CTA at most (GB300: 152, 233472, 232448),
 * with no device, memory or launch involved: the same checks and the same
 * resolution.  *resolved receives the descriptor with every tactic field
 * filled in; the other outputs (each may be NULL) as for
 * mxfp8_publish_gemm_config.  Returns what create would for the descriptor,
 * or MXFP8_ERR_INVALID for non-positive limits. */
mxfp8_status mxfp8_publish_gemm_plan(const mxfp8_gemm_desc* desc, int32_t sms,
                                     int32_t smem_per_sm, int32_t smem_per_block_optin,
                                     mxfp8_gemm_desc* resolved, int32_t* smem_bytes,
                                     int32_t* tmem_columns, int32_t* grid_ctas);

/* Everything a run with m rows needs, done ahead, launching nothing
 * (publishing_gemm page, PublishingMxfp8Linear.precompile: a publish without
 * its consumer would desynchronise the mailbox).  Call before CUDA-graph
 * capture.  Returns MXFP8_ERR_UNSUPPORTED for m not in 1..min(8, capacity_m). */
mxfp8_status mxfp8_publish_gemm_precompile(mxfp8_publish_gemm* gemm, int32_t m);

/* One publishing GEMM (publishing_gemm page, PublishingMxfp8Linear.__call__
 * and PublishingLowLatencyBlockscaledGemmKernel.epilog_warp):
 *  x:       device, 16-byte aligned, [m][K] E4M3FN bytes.
 *  x_scale: device, [m][K/32] E8M0FNU bytes, row-major.
 *  m:       1..min(8, capacity_m), else MXFP8_ERR_UNSUPPORTED.
 *  c:       device, 16-byte aligned, [m][N] BF16, or NULL to skip C.  C keeps
 *           negative zero; the mailbox copy clears it.
 * The device current when the handle was created must be current (else
 * MXFP8_ERR_INVALID); a handle is used by one host thread at a time.
 * Publishes into generation g = stage_state[0] and sets stage_state[1] = g.
 * Launched with programmatic stream serialisation (except the handle's first
 * run, which takes a full dependency on create's kernels): weight loads may
 * start before the previous kernel on `stream` finishes; x, x_scale, alpha
 * and the state are read only after it has.  So the weight (w for
 * MXFP8_W_IN_PLACE) and the workspace must not be written by the kernel
 * right before a run on the stream, nor by one still running when that
 * kernel starts; writes ordered before a kernel launched without
 * programmatic serialisation, or before a synchronisation, are safe.  Every
 * run must be followed, on the same stream, by exactly one mailbox_consume
 * before the next run. */
mxfp8_status mxfp8_publish_gemm_run(mxfp8_publish_gemm* gemm, const void* x,
                                    const void* x_scale, int32_t m, void* c, void* stream);

/* mxfp8_publish_gemm_run with a global scale (publishing_gemm page,
 * epilog_warp with use_scale: the accumulator times mScale[0] before the
 * conversion to BF16): C = alpha * sum_k W x, published as in
 * mxfp8_publish_gemm_run.  alpha: device, 4-byte aligned FP32 scalar, read
 * after the grid wait (so the previous kernel may write it), or NULL for 1.
 * The product is formed on the compensated sum and rounded once. */
mxfp8_status mxfp8_publish_gemm_run_scaled(mxfp8_publish_gemm* gemm, const void* x,
                                           const void* x_scale, int32_t m, const float* alpha,
                                           void* c, void* stream);

/* The same GEMM without the publish (the unfused path of the publishing_gemm
 * page's module description: the plain GEMM writes C, a separate publish
 * kernel reads it back).  c is required. */
mxfp8_status mxfp8_gemm_run_unfused(mxfp8_publish_gemm* gemm, const void* x,
                                    const void* x_scale, int32_t m, void* c, void* stream);

/* The standalone publish kernel of the unfused path: reads C [m][n] BF16
 * (device, 16-byte aligned), writes it with negative zero cleared into
 * generation stage_state[0], then sets stage_state[1].  Its result is bit-
 * identical to the fused epilogue's. */
mxfp8_status mailbox_publish(void* mailbox, int32_t* stage_state, int32_t capacity_m,
                             int32_t n, int32_t m, const void* c, void* stream);

/* The consumer (all_gather page, module description steps 2 and 3, one
 * rank), launched as the previous kernel's programmatic dependent: reads
 * g = stage_state[1]; polls mailbox[g][t][*] for t < m until no 32-bit word
 * is the sentinel; writes out[t][*] (device, 16-byte aligned, [m][n] BF16);
 * stores the sentinel back; one CTA sets stage_state[0] = (g + 1) mod 3 (no
 * CTA of the consumer reads that word; the next publisher reads it after the
 * consumer has completed).  A poll still unsatisfied after
 * timeout_ns nanoseconds (0 = one second) gives up: it sets
 * MXFP8_FLAG_POLL_TIMEOUT, still copies and resets its slot, and the
 * generation still advances, so the stream drains. */
mxfp8_status mailbox_consume(void* mailbox, int32_t* stage_state, int32_t capacity_m,
                             int32_t n, int32_t m, void* out, uint64_t timeout_ns,
                             void* stream);

/* Synchronises `stream`, copies stage_state (device int32[4]) into words
 * (host int32[4]) and reports: MXFP8_ERR_TIMEOUT if a timeout flag is set,
 * MXFP8_ERR_STATE if the bad-state flag is set or a generation word is not in
 * 0..2, else MXFP8_OK. */
mxfp8_status mxfp8_mailbox_status(const int32_t* stage_state, int32_t* words, void* stream);

/* Releases the handle (host memory only; the caller's buffers stay). */
void mxfp8_publish_gemm_destroy(mxfp8_publish_gemm* gemm);

/* ------------------------------------------------------------------------
 * The Lamport all-gather with one rank (page "vllm.models.deepseek_v41.
 * nvidia.ops.cute_dsl.all_gather", module description steps 1-3), on its own
 * mailbox: three generations of `capacity_bytes` (a positive multiple of 16,
 * at most MXFP8_GATHER_MAX_CAPACITY) as 16-byte packs, and state words
 * int32[4]: [0] the call's generation, [1] the arrival count, [2] unused,
 * [3] error flags (the MXFP8_FLAG_* bits; mxfp8_mailbox_status reads them).
 * ------------------------------------------------------------------------ */
#define MXFP8_GATHER_MAX_CAPACITY (64u << 20)

/* Mailbox bytes for a capacity (3 * capacity_bytes), 0 if it is invalid. */
size_t lamport_gather_mailbox_bytes(size_t capacity_bytes);

/* Arm a gather mailbox: every word the sentinel, the state zero
 * (LamportAllGather.__init__).  mailbox: device, 16-byte aligned,
 * lamport_gather_mailbox_bytes(capacity_bytes); state: device, 16-byte
 * aligned int32[4].  One kernel on `stream`. */
mxfp8_status lamport_gather_init(void* mailbox, int32_t* state, size_t capacity_bytes,
                                 void* stream);

/* One gather (_AllGatherKernel): in (device, 16-byte aligned, nbytes = 16 to
 * capacity_bytes, a multiple of 16) is published with every 32-bit word equal
 * to 0x80000000 cleared to 0 (LamportAllGather.__call__: FP32 negative zero
 * arrives as positive zero), polled back from the rank's own slot, written to
 * out (device, 16-byte aligned, nbytes), and the slot reset; the last CTA
 * advances the generation.  Launched with programmatic stream serialisation;
 * it triggers its dependents once it has published.  A poll still unsatisfied
 * after timeout_ns (0 = one second) sets MXFP8_FLAG_POLL_TIMEOUT.  Calls on
 * one mailbox must be ordered on one stream and must not overlap. */
mxfp8_status lamport_all_gather(void* mailbox, int32_t* state, size_t capacity_bytes,
                                const void* in, size_t nbytes, void* out, uint64_t timeout_ns,
                                void* stream);

/* ------------------------------------------------------------------------
 * The tagged-pair mailbox (page "vllm.models.deepseek_v41.amd.mono.common.
 * sync", Mailbox: each 32-bit value stored next to the launch's tag, a
 * consumer polls until every tag matches, nothing is reset), as an
 * alternative protocol for the projection's output.  pairs: device, 16-byte
 * aligned, tagged_mailbox_bytes(capacity_m, n): [capacity_m][n/2] pairs of
 * uint32 (value word holding BF16 columns 2w | 2w+1 << 16, tag).  Tag 0 is the
 * armed state and is refused; the caller gives every call a new tag (an
 * epoch) and calls on one mailbox are ordered on one stream.  The BF16 bits
 * move unchanged (no sentinel, so negative zero is kept).
 * ------------------------------------------------------------------------ */

/* Bytes of a tagged mailbox: capacity_m * n * 4 (0 for an invalid shape:
 * capacity_m not in 1..8, n not a positive multiple of 8). */
size_t tagged_mailbox_bytes(int32_t capacity_m, int32_t n);

/* Arm: every pair zero (tag 0). */
mxfp8_status tagged_mailbox_init(void* pairs, int32_t capacity_m, int32_t n, void* stream);

/* put: C [m][n] BF16 (device, 16-byte aligned) with `tag`, each value in one
 * 16-byte store with its tag.  PDL launch. */
mxfp8_status tagged_publish(void* pairs, int32_t capacity_m, int32_t n, int32_t m,
                            const void* c, uint32_t tag, void* stream);

/* poll: out [m][n] BF16 (device, 16-byte aligned) once every tag of rows
 * t < m equals `tag`; nothing is reset.  A poll unsatisfied after timeout_ns
 * (0 = one second) gives up, copies what is there and, if flags (device
 * int32) is not NULL, sets MXFP8_FLAG_POLL_TIMEOUT in it.  PDL launch. */
mxfp8_status tagged_consume(void* pairs, int32_t capacity_m, int32_t n, int32_t m, uint32_t tag,
                            void* out, uint64_t timeout_ns, int32_t* flags, void* stream);

/* Scratch bytes the library keeps in device memory for
 * mxfp8_publish_gemm_run_noalloc: a static array that every GPU loading the
 * library holds until the process exits. */
#define MXFP8_NOALLOC_SCRATCH_BYTES (4u << 20)

/* The publishing GEMM in one call that allocates nothing.  The source pages
 * have no counterpart: it exists for callers that cannot allocate --
 * runtimes that hand all device memory to a fixed pool at start-up and forbid
 * cudaMalloc afterwards, latency-critical issue paths where an allocation
 * (which may synchronise the device) is not allowed, and plain C hosts
 * without a device allocator of their own.  It needs no handle and no
 * workspace: W is read in place (MXFP8_W_IN_PLACE; w_layout 0 means that
 * here, MXFP8_W_TILED is refused), and W's scale factors are re-laid on every
 * call into the library's static scratch array (MXFP8_NOALLOC_SCRATCH_BYTES),
 * then the same GEMM kernel as mxfp8_publish_gemm_run runs on it.
 *  desc:        as for mxfp8_publish_gemm_create; N/128 * ceil(K/128) * 512
 *               bytes of scale chunks must fit the scratch, else
 *               MXFP8_ERR_UNSUPPORTED (e.g. N = 8192 with K = 16384 fits).
 *  w, w_scale:  device, as for mxfp8_publish_gemm_create (both read per call).
 *  x, x_scale, m, c: as for mxfp8_publish_gemm_run.
 *  mailbox, stage_state: device, as for mxfp8_mailbox_init.
 * The first call on a device resolves the scratch array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  That address is kept for the life of the
 * process: after a cudaDeviceReset of the device it is no longer valid, and
 * this call must not be used there again.  Every call shares the one array
 * and leaves its scale chunks there; calls that overlap on the GPU (on two
 * streams, or two threads) race on it and must not be issued.  The GEMM
 * launches with a full stream dependency (the re-layout right before it
 * writes what it reads first), so it never overlaps the kernel before it.
 * A call that repeats the previous call's device, w and desc reuses that
 * call's tactic and tensor map (and x's map when x and m repeat too): no
 * re-encoding on the host.  As after mxfp8_publish_gemm_run, one
 * mailbox_consume must follow on the stream. */
mxfp8_status mxfp8_publish_gemm_run_noalloc(const mxfp8_gemm_desc* desc, const void* w,
                                            const void* w_scale, const void* x,
                                            const void* x_scale, int32_t m, void* c,
                                            void* mailbox, int32_t* stage_state, void* stream);

/* Text of the calling thread's last error ("" if none). */
const char* mxfp8_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MXFP8_MAILBOX_H */
