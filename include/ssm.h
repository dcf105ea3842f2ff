/*
 * ssm.h: C ABI of the GB300 (sm_103a) selective state-space forward library.
 *
 * Three operations, all forward only, all on one GPU:
 *
 *   ssm_ssd_fwd      Mamba-2 chunked SSD forward, (x, dt, A, B, C, D, h0) -> (y, h_final).
 *                    Definition: "Accelerating Mamba-2 with High-Performance Forward
 *                    Pass Kernels in NVIDIA CUDA Tile", section "Mamba-2 architecture":
 *                        h_t = exp(a_t) h_{t-1} + x_t b_t^T,  a_t = A dt_t,  b_t = dt_t B_t
 *                        y_t = h_t c_t + D x_t
 *                    with the inclusive output reading (y_t reads the state after token
 *                    t, as the post's chunked form and its causal mask i >= j do).  The
 *                    chunked evaluation follows the same section's jump formula
 *                        h_{t+T} = exp(G_last) h_t + X^T (exp(G_last - G) . B)
 *                    and chunk output
 *                        Y = exp(G) C h + (exp(G_i - G_j) . (C B^T) . M) X + D X,
 *                    run as four kernels (chunk cumsum, chunk state, state passing,
 *                    chunk scan; the post's "Kernel 1".."Kernel 3" with the chunk loop of
 *                    Kernel 2 split into a parallel part and a look-back scan).
 *
 *   ssm_ssd_step     the same recurrence for ONE new token per sequence with a carried
 *                    state (decode): (x, dt, A, B, C, D, state) -> (y, state'), one
 *                    streaming kernel over the f32 state.
 *
 *   ssm_linscan_fwd  scalar selective scan h[t] = a[t] h[t-1] + b[t], h[-1] = 0, per row.
 *                    Definition: "Selective-scan CUDA kernels", section "The problem";
 *                    computed as a single-pass decoupled look-back prefix scan under the
 *                    pair combine (a1,b1).(a2,b2) = (a1 a2, a2 b1 + b2) (same page, "The
 *                    five kernels", Level 3c).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library never
 *     allocates, frees or retains them.  Tensors are dense, row-major (C order), with a
 *     16-byte aligned base address.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  The call returns once the kernels are enqueued.
 *   - Host-detectable errors return synchronously, before anything is enqueued.  No
 *     exception crosses the ABI.  Device-side failures of the bounded look-back waits are
 *     recorded in a status word inside the workspace and reported by
 *     ssm_check_device_status().
 *   - Workspace: caller-owned device memory of at least *_workspace_bytes() bytes, 256-byte
 *     aligned, ZERO-FILLED BEFORE ITS FIRST USE (e.g. cudaMemset).  Every call leaves it
 *     ready for the next call.  One workspace must not be used by two calls that can run
 *     concurrently (different streams without ordering).
 *   - Not thread-safe per workspace; different workspaces may be used from different host
 *     threads.
 *   - Every call can be captured into a CUDA graph and replayed (nothing is allocated or
 *     synchronized; the look-back flags carry an epoch kept in the workspace that each launch
 *     advances).  Make one ordinary call per device and shape before capturing, so that
 *     one-time set-up (kernel attributes, the no-alloc scratch address) happens outside the
 *     capture.  ssm_ssd_fwd_tune, ssm_linscan_fwd_tune (the two also allocate, for the
 *     duration of the call, the temporary buffer they flush L2 with) and
 *     ssm_check_device_status synchronize and cannot be captured.
 */
#ifndef SSM_GB300_H
#define SSM_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ssm_stream_t; /* same type as cudaStream_t */

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = 1, /* negative size, NULL required pointer, nheads % ngroups != 0 */
    SSM_ERR_UNSUPPORTED = 2, /* shape outside what the kernels are built for */
    SSM_ERR_ALIGNMENT = 3,   /* a tensor or workspace base is not aligned as required */
    SSM_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than *_workspace_bytes() */
    SSM_ERR_CUDA = 5,        /* a CUDA runtime call failed (launch, attribute, sync) */
    SSM_ERR_TIMEOUT = 6,     /* a bounded look-back wait gave up (device status word) */
    SSM_ERR_BOUNDS = 7       /* a device index check of a debug build (SSM_DEBUG) failed (device status word) */
} ssm_status;

typedef enum {
    SSM_F32 = 0,  /* x, dt, B, C and y are float32 */
    SSM_BF16 = 1  /* x, dt, B, C and y are bfloat16; accumulation stays float32 */
} ssm_dtype;

/* Human-readable name of a status code (static storage; never NULL). */
SSM_API const char *ssm_status_string(ssm_status status);

/* Library version as "major.minor.patch" (static storage). */
SSM_API const char *ssm_version(void);

/*
 * Workspace size in bytes for ssm_ssd_fwd with these sizes (0 when any size is invalid or
 * unsupported; ssm_ssd_fwd reports the reason).  The workspace holds the per-token decay
 * cumsums, the per-chunk states and the look-back flags of the state-passing scan.
 */
SSM_API size_t ssm_ssd_fwd_workspace_bytes(int64_t batch, int64_t seqlen, int nheads, int headdim,
                                   int dstate, int ngroups, int chunk, ssm_dtype dtype);

/*
 * Mamba-2 SSD forward (definition above).
 *
 * Inputs (element type `dtype` unless marked f32):
 *   x   [batch, seqlen, nheads, headdim]
 *   dt  [batch, seqlen, nheads]          time steps, used as given (already positive)
 *   A   [nheads] f32                     per-head decay rate (A < 0 for a stable state)
 *   B   [batch, seqlen, ngroups, dstate] input projection; head h reads group
 *                                        h / (nheads / ngroups)
 *   C   [batch, seqlen, ngroups, dstate] output projection, same grouping
 *   D   [nheads] f32                     skip weight
 *   h0  [batch, nheads, headdim, dstate] f32 initial state, or NULL for zeros
 * Outputs:
 *   y        [batch, seqlen, nheads, headdim], element type `dtype`
 *   h_final  [batch, nheads, headdim, dstate] f32 state after the last token, or NULL
 *            (not written).  It can be passed back as h0 of a call on the next segment.
 * Sizes: batch >= 0, seqlen >= 0 (batch == 0 or seqlen == 0 enqueue only the copy of h0
 *   into h_final), nheads >= 1, ngroups >= 1 dividing nheads, headdim == 64,
 *   dstate in {64, 128}, chunk in {64, 128, 256}.  seqlen need not be a multiple of chunk
 *   (the last chunk is zero-padded, which is exact: dt = 0 gives decay 1 and no input).
 * Errors: SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED, SSM_ERR_ALIGNMENT (any tensor not
 *   16-byte aligned, workspace not 256-byte aligned), SSM_ERR_WORKSPACE, SSM_ERR_CUDA.
 */
SSM_API ssm_status ssm_ssd_fwd(const void *x, const void *dt, const float *A, const void *B, const void *C,
                       const float *D, const float *h0, void *y, float *h_final,
                       int64_t batch, int64_t seqlen, int nheads, int headdim, int dstate,
                       int ngroups, int chunk, ssm_dtype dtype,
                       void *workspace, size_t workspace_bytes, ssm_stream_t stream);

/*
 * Per-shape plans for ssm_ssd_fwd.  "Accelerating Mamba-2 with High-Performance Forward Pass
 * Kernels in NVIDIA CUDA Tile", section "Mamba-2 performance optimization", gets its speed
 * across shapes from an autotuner that searches block sizes per shape; here the choices are
 * discrete plans, picked by measurement:
 *   - the state path: chunk states and the recurrence over chunks in one kernel (bf16, headdim
 *     64, dstate 128, an even number of heads per group), or the two kernels chunk-state then
 *     state-passing, the latter sequential over chunks or a decoupled look-back.  With more
 *     (batch, head pair) chains than SMs the one-kernel pass runs one CTA per SM on equal
 *     ranges of chunks, and a CTA that starts inside a chain waits (bounded) for the state its
 *     predecessor publishes; the CTAs claim their ranges in order, so that predecessor is
 *     always already running and the pass needs no co-residency of its CTAs.  With few long
 *     chains the one-kernel pass can instead split them ("split chains"): one CTA per SM runs
 *     an equal piece of chunks at once, every piece that starts inside a chain from a zero
 *     state, and a light second kernel then adds to each such piece's chunk-initial states the
 *     state it enters with (composed in f32 from the pieces' end states; h_in is then rounded
 *     to bf16 twice);
 *   - the one-kernel pass's shared-memory ring split: X slots (loaded from DRAM) and B slots
 *     (loaded from L2) share a fixed budget: 4 + 3, 3 + 4 or 5 + 2;
 *   - the chunk scan's run of heads per CTA (the tensor-core path).
 * Without a plan, ssm_ssd_fwd picks by fixed rules of thumb.  A plan id packs
 * (fused + 1) | (sequential + 1) << 2 | heads_per_cta << 4 | ring << 20, where fused and
 * sequential are 1 (yes), 0 (no) or -1 (rule of thumb), fused may also be 2 (the one-kernel
 * pass with split chains; the rule takes it for between a sixteenth and a half as many chains
 * as SMs, with at least 32 chunks each), heads_per_cta (0 .. 65535) n > 0 gives
 * every chunk-scan CTA a run of at most n heads (a tile's heads split evenly) and 0 means the
 * split a model of the hardware's CTA dispatch finds fastest (large runs first, small runs
 * last; ssm_debug_scan_schedule shows it; the first call of a shape on a device spends up to
 * ~25 ms of host time on that search, which is cached, makes no CUDA call and so may fall
 * inside a stream capture), and ring is 1 (4 + 3), 2 (3 + 4), 3 (5 + 2) or 0 (the rule: 4 + 3).
 *
 * ssm_ssd_fwd_tune takes exactly ssm_ssd_fwd's arguments and runs every candidate plan for
 * these sizes on the caller's buffers (y and h_final are overwritten; each candidate computes
 * the same result up to rounding): one warm-up and `reps` timed runs each (CUDA events on
 * `stream`), synchronizing the stream.  Before each run, outside the timed events, it writes a
 * temporary device buffer of twice the L2 size (allocated for the call and freed at its end;
 * the runs go back to back if it cannot be allocated), so that every candidate is timed with
 * its inputs out of L2, as after other work.  The plan with the smallest median time is stored for
 * the current device and these sizes in a process-wide table that later ssm_ssd_fwd calls
 * with the same sizes use; *plan_out and *ms_out (either may be NULL) receive it and its time.
 * A device error recorded by a candidate (SSM_ERR_TIMEOUT) is returned and no plan is stored.
 * ssm_ssd_fwd_set_plan stores a given plan (-1 removes the entry), ssm_ssd_fwd_get_plan reads
 * the stored one (-1: none), ssm_ssd_fwd_clear_plans empties the table.  The table is shared
 * by all host threads (guarded by a lock).
 * Errors: as ssm_ssd_fwd, plus SSM_ERR_INVALID_ARG for reps < 1 or an invalid plan id.
 */
SSM_API ssm_status ssm_ssd_fwd_tune(const void *x, const void *dt, const float *A, const void *B, const void *C,
                                    const float *D, const float *h0, void *y, float *h_final, int64_t batch,
                                    int64_t seqlen, int nheads, int headdim, int dstate, int ngroups, int chunk,
                                    ssm_dtype dtype, void *workspace, size_t workspace_bytes, ssm_stream_t stream,
                                    int reps, int *plan_out, float *ms_out);
SSM_API ssm_status ssm_ssd_fwd_set_plan(int64_t batch, int64_t seqlen, int nheads, int headdim, int dstate,
                                        int ngroups, int chunk, ssm_dtype dtype, int plan);
SSM_API ssm_status ssm_ssd_fwd_get_plan(int64_t batch, int64_t seqlen, int nheads, int headdim, int dstate,
                                        int ngroups, int chunk, ssm_dtype dtype, int *plan);
SSM_API void ssm_ssd_fwd_clear_plans(void);

/*
 * Mamba-2 decode step: ONE new token per sequence, with the state carried between calls.
 * Definition: the recurrence above applied to a single token ("Accelerating Mamba-2 with
 * High-Performance Forward Pass Kernels in NVIDIA CUDA Tile", section "Mamba-2
 * architecture": the recurrent form, one state update per token, that the post contrasts
 * with the chunked form; and its note that the final state of one call can start the next,
 * so the h_final of ssm_ssd_fwd over a prompt is the state_in of the first step):
 *     state_out = exp(A dt) state_in + x (dt B)^T      (per head, H x S, S contiguous)
 *     y         = state_out c + D x                     (inclusive reading)
 *
 * Inputs (element type `dtype` unless marked f32):
 *   x         [batch, nheads, headdim]
 *   dt        [batch, nheads]            time steps, used as given (already positive)
 *   A, D      [nheads] f32
 *   B, C      [batch, ngroups, dstate]   head h reads group h / (nheads / ngroups)
 *   state_in  [batch, nheads, headdim, dstate] f32, or NULL for zeros (a first token)
 * Outputs:
 *   state_out [batch, nheads, headdim, dstate] f32.  It may be the same pointer as
 *             state_in (the state is then updated in place); any other overlap of the two
 *             is rejected with SSM_ERR_INVALID_ARG.
 *   y         [batch, nheads, headdim], element type `dtype`
 * Sizes: batch >= 0 (0: nothing is enqueued), nheads >= 1, ngroups >= 1 dividing nheads,
 *   headdim a positive multiple of 16, dstate in {64, 128}.  No workspace.  One kernel is
 *   enqueued on `stream`; it reads and writes the state once (8 * headdim * dstate bytes per
 *   head), so it runs at the HBM rate.
 * Errors: SSM_ERR_INVALID_ARG, SSM_ERR_UNSUPPORTED, SSM_ERR_ALIGNMENT (any tensor not 16-byte
 *   aligned), SSM_ERR_CUDA.
 */
SSM_API ssm_status ssm_ssd_step(const void *x, const void *dt, const float *A, const void *B, const void *C,
                                const float *D, const float *state_in, float *state_out, void *y,
                                int64_t batch, int nheads, int headdim, int dstate, int ngroups,
                                ssm_dtype dtype, ssm_stream_t stream);

/* Workspace size in bytes for ssm_linscan_fwd on rows x len (0 when a size is negative). */
SSM_API size_t ssm_linscan_workspace_bytes(int64_t rows, int64_t len);

/*
 * Scalar selective scan (definition above), independently on each row.
 *   a, b  [rows, len] f32 inputs;  h [rows, len] f32 output (may not alias a or b).
 * rows >= 0, len >= 0 (either 0: nothing is enqueued).  Rows need not be 16-byte aligned
 * individually (len may be odd); only the base pointers must be.
 * Errors: SSM_ERR_INVALID_ARG, SSM_ERR_ALIGNMENT, SSM_ERR_WORKSPACE, SSM_ERR_CUDA.
 */
SSM_API ssm_status ssm_linscan_fwd(const float *a, const float *b, float *h, int64_t rows, int64_t len,
                           void *workspace, size_t workspace_bytes, ssm_stream_t stream);

/*
 * Per-size CTA shapes of ssm_linscan_fwd (the scan counterpart of the SSD plans above, after the
 * block-size and occupancy search of "Accelerating Mamba-2 with High-Performance Forward Pass
 * Kernels in NVIDIA CUDA Tile", section "Mamba-2 performance optimization").  A shape fixes the
 * look-back scan's CTA: its consumer groups (which take the CTA's tiles in turn), the depth of
 * its shared-memory ring and the CTAs resident per SM:
 *   1  two groups, 7 stages, one CTA per SM (the rule for rows of at least 4 tiles)
 *   2  one group, 3 stages, two CTAs per SM (the rule for shorter rows)
 *   3  two groups, 6 stages, one CTA per SM
 *   4  one group, 6 stages, one CTA per SM
 * ssm_linscan_fwd_tune takes ssm_linscan_fwd's arguments, runs every shape on the caller's
 * buffers (h is overwritten with the scan; a warm-up and `reps` timed runs each, CUDA events on
 * `stream`, synchronizing it; each run preceded by the same L2 flush as ssm_ssd_fwd_tune's) and stores the shape with the smallest median time for the current
 * device and these (rows, len) in a process-wide table that later ssm_linscan_fwd calls use;
 * *shape_out and *ms_out (either may be NULL) receive it and its time.  A device error recorded
 * by a candidate (SSM_ERR_TIMEOUT) is returned and nothing is stored.  ssm_linscan_set_shape
 * stores a shape (-1 or 0 removes the entry), ssm_linscan_get_shape reads it (-1: none, the
 * rule applies), ssm_linscan_clear_shapes empties the table.  ssm_linscan_fwd_noalloc always
 * takes the rule.  Errors: as ssm_linscan_fwd, plus SSM_ERR_INVALID_ARG for reps < 1 or a shape
 * outside -1 .. 4.
 */
SSM_API ssm_status ssm_linscan_fwd_tune(const float *a, const float *b, float *h, int64_t rows, int64_t len,
                                        void *workspace, size_t workspace_bytes, ssm_stream_t stream, int reps,
                                        int *shape_out, float *ms_out);
SSM_API ssm_status ssm_linscan_set_shape(int64_t rows, int64_t len, int shape);
SSM_API ssm_status ssm_linscan_get_shape(int64_t rows, int64_t len, int *shape);
SSM_API void ssm_linscan_clear_shapes(void);

/*
 * Scalar selective scan for callers that cannot allocate device memory (the pages have no
 * counterpart; this is a convenience of this library).  Some callers must not allocate once
 * they are running: a framework that reserves its device memory up front and forbids later
 * allocation, a real-time loop that cannot afford the implicit device synchronisation of
 * cudaMalloc / cudaFree, or a host that simply has no allocator to hand out a workspace.
 * This entry point takes the same a, b, h, rows and len as ssm_linscan_fwd (same layout,
 * alignment and results, same kernel) but no workspace: the scan's scratch lives in a fixed
 * device array inside the library, sized for rows * len <= 2^26 elements (67,108,864),
 * 262,400 bytes that every GPU which loads the library keeps until the process exits.
 *   - Larger scans return SSM_ERR_UNSUPPORTED without enqueuing anything; use
 *     ssm_linscan_fwd with a workspace for them.
 *   - It allocates nothing: no cudaMalloc, cudaFree or allocating library routine.  It
 *     enqueues a 16-byte cudaMemsetAsync that clears the scratch header, then the kernel.
 *   - Every call looks up the device address of the scratch array on the current device (the
 *     first call on a device may load the library's device code there); make the first call on
 *     each device before any stream capture.
 *   - All calls share the one scratch array, which keeps the previous call's contents.  Calls
 *     that may overlap on the GPU (different streams without ordering) race and must not be
 *     issued.
 *   - Device-side look-back timeouts (a wait beyond 1 s, which needs a GPU that stopped making
 *     progress) are not reported by this entry point: there is no workspace to pass to
 *     ssm_check_device_status, and the next call clears the scratch's status word.  The
 *     output of such a call is invalid: tiles whose wait ran out hold NaN, and tiles no thread
 *     reached keep whatever h held before the call.
 * Errors: SSM_ERR_INVALID_ARG, SSM_ERR_ALIGNMENT, SSM_ERR_UNSUPPORTED, SSM_ERR_CUDA.
 */
SSM_API ssm_status ssm_linscan_fwd_noalloc(const float *a, const float *b, float *h, int64_t rows, int64_t len,
                                           ssm_stream_t stream);

/*
 * Baseline scans of the same recurrence, kept for measurement: the levels of "Selective-scan
 * CUDA kernels", section "The five kernels" (its traffic-model study compares them), each as
 * that page describes it, without this library's tuning.  ssm_linscan_fwd is the production
 * scan (the page's Level 3c, redesigned); use these only to compare against it.
 *   SSM_SCAN_BLELLOCH          Level 1: one CTA per row, up- and down-sweep in shared memory;
 *                              len <= 2048.  No workspace.
 *   SSM_SCAN_THREE_PASS        Level 2: local tile scans, a spine scan per row, then the
 *                              prefix applied; three launches; len <= 4,194,304 and
 *                              rows <= 65,535.  Workspace: a float per element plus 8 bytes
 *                              per 2048-element tile.
 *   SSM_SCAN_LOOKBACK_SERIAL   Level 3: single-pass decoupled look-back over 256-element tiles,
 *                              one thread walking the predecessors.
 *   SSM_SCAN_LOOKBACK_WARP     Level 3b: the same with a warp inspecting 32 predecessors at once.
 *                              Both look-backs need a zero-filled workspace (left ready for the
 *                              next call) and report timeouts through ssm_check_device_status.
 *   SSM_SCAN_HILLIS_STEELE     the page's PyTorch baseline algorithm (listed there as future
 *                              work in CUDA): ceil(log2 len) full-array passes of the combine at
 *                              doubling distances.  Workspace: four floats per element.
 * Arguments as ssm_linscan_fwd.  Errors: SSM_ERR_INVALID_ARG (unknown algorithm, negative
 * size), SSM_ERR_UNSUPPORTED (a size beyond the algorithm's limit), SSM_ERR_ALIGNMENT,
 * SSM_ERR_WORKSPACE, SSM_ERR_CUDA.
 */
typedef enum {
    SSM_SCAN_BLELLOCH = 1,
    SSM_SCAN_THREE_PASS = 2,
    SSM_SCAN_LOOKBACK_SERIAL = 3,
    SSM_SCAN_LOOKBACK_WARP = 4,
    SSM_SCAN_HILLIS_STEELE = 5
} ssm_scan_algo;
SSM_API size_t ssm_linscan_baseline_workspace_bytes(ssm_scan_algo algo, int64_t rows, int64_t len);
SSM_API ssm_status ssm_linscan_baseline(ssm_scan_algo algo, const float *a, const float *b, float *h, int64_t rows,
                                        int64_t len, void *workspace, size_t workspace_bytes, ssm_stream_t stream);

/*
 * Synchronizes `stream`, reads the device status word at the start of `workspace` (either
 * kind) and returns SSM_OK or the recorded device error (SSM_ERR_TIMEOUT when a bounded wait
 * exceeded its limit; the outputs of that call are then invalid).  After an error it also
 * resets the workspace's claim counters, so the workspace is usable again.
 */
SSM_API ssm_status ssm_check_device_status(void *workspace, ssm_stream_t stream);

/*
 * Test hook for the bounded look-back waits (not needed in normal use).  From the next
 * call on, the look-back tile with claim index `stall_tile` (-1: none) of every look-back
 * kernel skips publishing its aggregate and prefix, and every wait gives up after
 * `spin_limit_ns` nanoseconds (0: the default of 1 s).  The waiting tiles then record
 * SSM_ERR_TIMEOUT in the status word and return; no kernel waits without a limit.
 */
SSM_API void ssm_debug_set_lookback_fault(int64_t stall_tile, uint64_t spin_limit_ns);

/*
 * Debug builds.  The library compiled with -DSSM_DEBUG (libssm_gb300_debug.so, built beside the
 * release library) checks the indexes of its kernels' raw global-memory accesses and of the
 * shared-memory slots they compute: a failed check records SSM_ERR_BOUNDS in the call's
 * status word, which ssm_check_device_status reports, and the access is skipped; nothing traps.
 * This stands in for a memory sanitizer.  ssm_debug_build returns 1 in such a build, else 0.
 *
 * ssm_debug_set_bounds_fault is a test hook of debug builds: from the next ssm_ssd_fwd call on,
 * the chunk-cumsum kernel checks its G and dt^T stores against a bound `shrink` elements short
 * of the real one, so that the stores of the last `shrink` elements fail the check, are skipped
 * and SSM_ERR_BOUNDS is reported (the forward's output is then not valid).  0 turns it off.
 * Release builds: returns SSM_ERR_UNSUPPORTED and changes nothing.
 */
SSM_API int ssm_debug_build(void);
SSM_API ssm_status ssm_debug_set_bounds_fault(int64_t shrink);

/*
 * Test hook for the fused state pass's work split (host only; no GPU call).  For `chains`
 * (batch, head pair) chains of `nchunks` chunks on a GPU with `sms` SMs it lists, in the order
 * each CTA runs them, the segments of every CTA: one row of six int64 per segment, (cta, chain,
 * first chunk, end chunk, starts from the state the previous CTA publishes, publishes its final
 * state for the next CTA).  With `split` nonzero, the split-chains schedule: a segment that
 * starts inside its chain starts from zero instead (its state is added afterwards) and one that
 * ends inside its chain publishes into its CTA's own slot.  Writes at most `cap` rows to `rows`
 * (which may be NULL) and returns the number of segments, or -1 for a negative size or sms < 1.
 */
SSM_API int64_t ssm_debug_fused_schedule(int64_t chains, int64_t nchunks, int sms, int split, int64_t *rows,
                                         int64_t cap);

/*
 * Test hook for the chunk scan's work split (host only; no GPU call).  The chunk scan's CTAs
 * take its `tiles` tiles ((batch, chunk, group, row tile), row tile fastest and the later row tile
 * first; `row_tiles` = 1 for chunk 128, 2 for chunk 256) in order, in three tiers: tier k covers the next out[2k] tiles with
 * out[2k+1] CTAs per tile, the tile's `heads_per_group` heads split evenly between those CTAs.
 * `plan_heads` is the plan's heads per CTA (0: the split a model of the hardware's CTA dispatch
 * on `sms` SMs finds fastest, large runs of heads first and small ones last).  Writes six
 * int64 to `out` (which may be NULL) and returns the number of CTAs, or -1 for invalid sizes.
 */
SSM_API int64_t ssm_debug_scan_schedule(int64_t tiles, int row_tiles, int heads_per_group, int sms, int plan_heads,
                                        int64_t *out);

/*
 * Kernel timing (measurement aid; not needed in normal use).  Between ssm_profile_begin()
 * and ssm_profile_end(), every ssm_ssd_fwd / ssm_ssd_step / ssm_linscan_fwd call records a
 * CUDA event on its own stream before and after each kernel it launches (at most
 * `max_launches` launches are recorded; later ones are counted but not timed).  ssm_profile_end() synchronizes the
 * recorded events and writes, for each kernel id below, the summed device time in
 * milliseconds and the number of launches (arrays of length SSM_PROFILE_KERNELS).
 * Kernel ids: 0 linscan_lookback, 1 ssd_chunk_cumsum, 2 ssd_chunk_state,
 * 3 ssd_state_passing, 4 ssd_chunk_scan, 5 ssd_state_fused (chunk states and state passing in
 * one pass; used instead of 2 and 3 where it applies), 6 ssd_step (ssm_ssd_step),
 * 7 linscan_baseline (ssm_linscan_baseline, all its launches), 8 ssd_state_fixup (the second
 * kernel of the one-kernel state pass with split chains).  Host-side only;
 * process-global; not thread-safe.
 */
#define SSM_PROFILE_KERNELS 9
SSM_API ssm_status ssm_profile_begin(int max_launches);
SSM_API ssm_status ssm_profile_end(double *ms_out, int64_t *launches_out);

#ifdef __cplusplus
}
#endif
#endif /* SSM_GB300_H */
