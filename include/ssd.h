/*
 * ssd.h -- C ABI of the GB300 (sm_103a) Mamba-2 chunked SSD forward pass (and
 * its backward, ssd_backward).
 *
 * Method: "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
 * NVIDIA CUDA Tile", section "Mamba-2 architecture".  Per batch b and head h,
 * with a_t = A[h] dt_t and b_t = dt_t B_t, the layer computes
 *
 *     h_t = exp(a_t) h_{t-1} + x_t (outer) b_t          state, P x S
 *     y_t = h_t c_t + D[h] x_t                          output, P
 *
 * y uses the post-update state h_t: the page's chunked output equation keeps
 * the diagonal of the causal mask (one line of the page writes h_{t-1}; this
 * library follows the chunked equations).  The work is split as on the page
 * (section "three kernels"): an in-chunk cumulative sum of a, the chunk
 * state jump h_{t+T} = exp(G_last) h_t + (exp(G_last - G) b)^T x, a
 * sequential pass over chunks, and the per-chunk output
 * Y = exp(G) C h + ((C B^T) * exp(G_i - G_j) * M) (dt X) + D X.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers to dense row-major arrays in the
 *   layouts listed below; each must be 16-byte aligned.  The caller owns and
 *   allocates every buffer, including the workspace of ssd_forward.  The
 *   library never allocates device memory, frees or synchronises (except
 *   ssd_forward_tune, which times candidates and waits for them, and the
 *   error read-outs).  Launch plans are passed to each call, never stored.
 *   The only state the library keeps between calls is the scratch array of
 *   ssd_forward_noalloc and one library-wide device error word, which only
 *   the calls without a workspace of their own report to (the step-wise
 *   entry points and ssd_forward_noalloc); ssd_forward and the calls built
 *   on it report to a word inside the caller's workspace.
 * - `stream` is a cudaStream_t (NULL = legacy default stream); all work is
 *   enqueued on it and runs asynchronously.
 * - Arguments are validated before anything is launched; a rejected call
 *   returns an error code and enqueues nothing.  A launch failure returns
 *   SSD_ERR_CUDA.  SSD_ERR_TIMEOUT reports that a bounded device-side wait
 *   gave up (the results of that call are then undefined).  Nothing throws.
 * - A debug-bounds build of the library (compiled with SSD_DEBUG_BOUNDS
 *   defined; the release build never is) checks the index of every plain
 *   global load and store of its kernels against the extent of the buffer
 *   it addresses, skips an access that falls outside, and reports it through
 *   the same error words as SSD_ERR_BOUNDS.  The checks cost time and
 *   compile away in the release build.
 * - Preconditions that are documented but not checked: A <= 0 and dt >= 0 (so
 *   every a_t <= 0, the page's stability condition), finite inputs, and
 *   output buffers that do not overlap inputs.  The bf16 output kernels 1
 *   and 2 of the launch plans (below) also need |c_i . b_j| < 2^20 for
 *   every pair of tokens of a chunk (they keep C B^T as fp16 scaled by
 *   2^-4); larger products come out as inf / NaN without an error code.
 *   The other output kernels keep C B^T in fp32 or bf16 and have no such
 *   limit.  Inside the row's own 64-token block, kernels 1 and 2 factor the
 *   decay exp2(G_i - G_j) into exp2(G_i - G_r) exp2(G_r - G_j) about the
 *   block's last token r, which keeps a positive exponent of at most +96
 *   (log2 units) in fp32; blocks whose total decay is steeper than 2^-96 use
 *   the direct exponent instead, so no input makes that factor overflow.
 *
 * Dimensions (ssd_dims): batch b >= 1, seqlen L >= 1, nheads nh >= 1,
 * headdim P, dstate S, ngroups ng (nh % ng == 0; head h reads group
 * h / (nh / ng), as on the page), chunk T.  Supported: P, S multiples of 16
 * with 16 <= P <= 128 and 16 <= S <= 256; T in {64, 128, 256}.  Anything
 * else returns SSD_ERR_UNSUPPORTED.  nc = ceil(L / T); the last chunk may be
 * partial and is treated as zero-padded (dt = 0), which changes nothing.
 *
 * Layouts ("io" = the I/O element type given by ssd_dtype):
 *   x  [b, L, nh, P] io        dt [b, L, nh] io        A [nh] f32
 *   B  [b, L, ng, S] io        C  [b, L, ng, S] io     D [nh] f32
 *   h0, final_state [b, nh, P, S] f32
 *   G  [b, nh, nc*T] f32  -- chunk-local inclusive cumsum of a, times log2(e)
 *   dstates, states [b, nh, nc, P, S] f32
 *   y  [b, L, nh, P] io
 * With SSD_F32 the tensor-core products run in TF32 with fp32 accumulation;
 * with SSD_BF16 they take bf16 operands and accumulate in fp32.
 */
#ifndef SSD_GB300_H
#define SSD_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSD_API __attribute__((visibility("default")))
#else
#define SSD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SSD_OK = 0,
  SSD_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment, nh % ng */
  SSD_ERR_UNSUPPORTED = 2, /* dims outside the supported range */
  SSD_ERR_CUDA = 3,        /* a CUDA call or launch failed */
  SSD_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up */
  SSD_ERR_BOUNDS = 5       /* a debug-bounds build caught an out-of-range access */
} ssd_status;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

typedef struct {
  int64_t batch, seqlen, nheads, headdim, dstate, ngroups, chunk;
} ssd_dims;

/* Launch plan of the bf16 forward path: the knobs that change how fast the
 * kernels run, never what they compute.  No counterpart on the pages beyond
 * their remark that an autotuner picks tile sizes, stages and occupancy per
 * shape; these are this library's knobs:
 *   chunk_state_heads  heads per work item of the chunk-jump kernel (they
 *                      share one load of B; divides nheads / ngroups)
 *   chunk_state_ctas   CTAs per SM of that kernel: 1 (up to 4 heads per
 *                      item) or 2 (up to 2)
 *   scan_kernel        output kernel: 0 = per-(128-row tile, chunk, head
 *                      slice) kernel for every shape; 1 = kernel sharing one
 *                      C B^T of a whole chunk between a slice of heads (P =
 *                      64, S in {64, 128}, T in {128, 256}); 2 = the same
 *                      with one 128-row tile of the chunk per CTA (P = 64,
 *                      S in {64, 128, 256}, T in {128, 256}); 3 = the
 *                      output pass with the decay factored about one anchor
 *                      per chunk, C B^T kept in bf16 without decay and
 *                      shared by the slice's heads (P = 64, S a multiple of
 *                      64 up to 256, T in {128, 256}; the default where it
 *                      applies)
 *   scan_heads         heads per CTA of that output kernel (divides
 *                      nheads / ngroups; at most 4, and heads * P <= 256, for
 *                      kernel 0)
 * A plan is an argument of the calls that take one (NULL = the cost-model
 * default, ssd_forward_default_plan); the library keeps no table of plans.
 * Only SSD_BF16 has plans: an fp32 call must pass NULL. */
typedef struct {
  int32_t chunk_state_heads, chunk_state_ctas, scan_kernel, scan_heads;
} ssd_plan;

/* Bytes at the start of every workspace of ssd_forward, ssd_forward_host and
 * ssd_forward_host_overlapped that hold the call's device error word.  A new
 * workspace must have them zeroed once before its first use (for example
 * cudaMemsetAsync(ws, 0, SSD_WS_HEADER_BYTES, stream)); after that the
 * library writes the word only when a bounded device-side wait gives up, and
 * ssd_workspace_error reads and clears it. */
#define SSD_WS_HEADER_BYTES 256u

/* Human-readable name of a status code (static storage, never NULL). */
SSD_API const char *ssd_status_string(ssd_status s);

/* Bytes of device workspace ssd_forward needs for these dims and dtype,
 * including the SSD_WS_HEADER_BYTES header (0 if the dims are invalid or
 * unsupported). */
SSD_API size_t ssd_forward_workspace_size(const ssd_dims *dims, ssd_dtype dtype);

/* Kernel 1 of the page ("Kernel 1: Computing cumulative sums"):
 *   G[b,h,k*T+i] = log2(e) * sum_{s=0..i} A[h] * dt[b, k*T+s, h]
 * i.e. the inclusive cumsum of a restarted at every chunk, scaled so later
 * steps can use exp2.  Positions past L hold the chunk's last real value.
 * In: dt (io), A.  Out: G. */
SSD_API ssd_status ssd_chunk_cumsum(const ssd_dims *dims, ssd_dtype dtype,
                            const void *dt, const float *A, float *G,
                            void *stream);

/* The jump term of the state update (page section "Mamba-2 architecture",
 * decayed jump formula; the tensor-core product inside fwd_pass_state):
 *   dstates[b,h,k][p][s] = sum_{j in chunk k}
 *        exp2(G_last,k - G_j) * dt_j * x[b,j,h,p] * B[b,j,g,s]
 * i.e. the state chunk k alone would produce from a zero start.
 * In: x, B, dt (io), G (from ssd_chunk_cumsum).  Out: dstates. */
SSD_API ssd_status ssd_chunk_state(const ssd_dims *dims, ssd_dtype dtype,
                           const void *x, const void *B, const void *dt,
                           const float *G, float *dstates, void *stream);

/* The sequential pass over chunks of the page's fwd_pass_state, which stores
 * the state at the start of every chunk:
 *   h = h0 (or 0 if h0 == NULL);  for k in 0..nc-1:
 *       states[b,h,k] = h;   h = exp2(G_last,k) * h + dstates[b,h,k]
 *   final_state = h  (skipped if final_state == NULL).
 * In: dstates, G, h0 (nullable).  Out: states, final_state (nullable). */
SSD_API ssd_status ssd_state_passing(const ssd_dims *dims, const float *dstates,
                             const float *G, const float *h0, float *states,
                             float *final_state, void *stream);

/* The page's compute_out (chunked output equation), per chunk k:
 *   y_i = exp2(G_i) * states[k] c_i
 *       + sum_{j<=i in chunk} (c_i . B_j) exp2(G_i - G_j) dt_j x_j
 *       + D[h] x_i
 * The T x T interaction tile stays on chip.  D == NULL means D = 0.
 * In: x, B, C, dt (io), G, states, D.  Out: y (io). */
SSD_API ssd_status ssd_chunk_scan(const ssd_dims *dims, ssd_dtype dtype,
                          const void *x, const void *B, const void *C,
                          const void *dt, const float *G, const float *states,
                          const float *D, void *y, void *stream);

/* The whole forward pass on one stream: the four steps above (or a fused
 * equivalent) with G and the per-chunk states kept in `workspace`
 * (>= ssd_forward_workspace_size bytes, 256-byte aligned, its first
 * SSD_WS_HEADER_BYTES zeroed before its first use).  h0, D and final_state
 * may be NULL.  Out: y (io), final_state (f32).  Runs the default launch
 * plan (ssd_forward_ex takes one).  A bounded device-side wait that gives up
 * is recorded in the workspace's error word (ssd_workspace_error).
 * The call allocates nothing and never synchronises, so after one eager call
 * on the device (which does the one-time set-up) it can be captured in a CUDA
 * graph and replayed on new inputs written into the same buffers. */
SSD_API ssd_status ssd_forward(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                       const void *dt, const float *A, const void *B,
                       const void *C, const float *D, const float *h0,
                       void *y, float *final_state, void *workspace,
                       size_t ws_bytes, void *stream);

/* ssd_forward with an explicit launch plan (NULL = the default plan; must be
 * NULL for SSD_F32).  A plan that is not one of
 * ssd_forward_plan_candidates(dims, dtype) returns SSD_ERR_INVALID_ARG with
 * nothing enqueued. */
SSD_API ssd_status ssd_forward_ex(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                                  const void *dt, const float *A, const void *B,
                                  const void *C, const float *D, const float *h0,
                                  void *y, float *final_state, void *workspace,
                                  size_t ws_bytes, const ssd_plan *plan, void *stream);

/* Synchronises `stream` and reports whether a kernel of a call that used
 * `workspace` (ssd_forward, ssd_forward_ex, ssd_forward_profiled,
 * ssd_forward_tune, ssd_forward_host, ssd_forward_host_overlapped) gave up a
 * bounded device-side wait since the word was last cleared
 * (SSD_ERR_TIMEOUT; the outputs of that call are undefined) or, in the
 * debug-bounds build, made an out-of-range access (SSD_ERR_BOUNDS), then
 * clears the word.  Each workspace has its own word, so calls on other workspaces
 * or streams neither see nor clear it.  SSD_ERR_INVALID_ARG for a NULL or
 * misaligned workspace; SSD_ERR_CUDA if the synchronisation fails. */
SSD_API ssd_status ssd_workspace_error(void *workspace, void *stream);

/* The same for the library-wide error word, which only the calls without a
 * workspace of their own report to: the step-wise entry points
 * (ssd_chunk_cumsum, ssd_chunk_state, ssd_state_passing, ssd_chunk_scan),
 * ssd_decode_step and ssd_forward_noalloc.  Synchronises `stream`, reports
 * SSD_ERR_TIMEOUT if any of them gave up a bounded wait on this device (or,
 * in the debug-bounds build, SSD_ERR_BOUNDS for an out-of-range access)
 * since the word was last cleared, and clears it. */
SSD_API ssd_status ssd_device_error(void *stream);

/* Self-test of the bounded device-side waits (no counterpart on the pages):
 * enqueues on `stream` one CTA whose wait on a barrier that nothing arrives
 * on gives up after limit_ns nanoseconds (1e3 <= limit_ns <= 1e9, else
 * SSD_ERR_INVALID_ARG) and records the give-up in *err_word -- a 4-byte
 * aligned device int, such as the header of a workspace (read it back with
 * ssd_workspace_error) -- or, with err_word NULL, in the library-wide word
 * (ssd_device_error).  The kernel then returns.  While a word holds a
 * give-up, the bounded waits of later calls reporting to the same word
 * return at once, so read it back before using that word again. */
SSD_API ssd_status ssd_selftest_bounded_wait(uint64_t limit_ns, int *err_word, void *stream);

/* ssd_forward_ex with per-launch timing.  `events` holds n_events
 * cudaEvent_t handles created by the caller; events[0] is recorded on
 * `stream` before the first launch and events[i+1] right after launch i
 * (while i + 1 < n_events).  *n_launches (if not NULL) receives the number
 * of kernel launches the call enqueued.  events may be NULL when n_events is
 * 0 (then nothing is recorded).  Same arguments, results and errors as
 * ssd_forward_ex otherwise. */
SSD_API ssd_status ssd_forward_profiled(const ssd_dims *dims, ssd_dtype dtype,
                                        const void *x, const void *dt, const float *A,
                                        const void *B, const void *C, const float *D,
                                        const float *h0, void *y, float *final_state,
                                        void *workspace, size_t ws_bytes,
                                        const ssd_plan *plan, void *stream,
                                        void *const *events, int n_events,
                                        int *n_launches);

/* Bytes of device workspace ssd_forward_host needs: room for the device copies
 * of every input and output plus the workspace of ssd_forward, which comes
 * first (so the header is this workspace's first SSD_WS_HEADER_BYTES); 0 if
 * the dims are invalid or unsupported. */
SSD_API size_t ssd_forward_host_workspace_size(const ssd_dims *dims, ssd_dtype dtype,
                                               int has_D, int has_h0,
                                               int want_final_state);

/* ssd_forward on HOST buffers: copies x, dt, A, B, C, D, h0 from host memory
 * into `workspace` (device, >= ssd_forward_host_workspace_size bytes, 256-byte
 * aligned, header zeroed before its first use), runs the forward pass there
 * with `plan` (as for ssd_forward_ex), and copies y (and final_state, if
 * not NULL) back to host memory, all enqueued on `stream`.  The host buffers
 * must stay valid until the stream reaches the end of the call; page-locked
 * host memory makes the copies asynchronous.  D, h0 and final_state may be
 * NULL.  Host pointers need no particular alignment. */
SSD_API ssd_status ssd_forward_host(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                                    const void *dt, const float *A, const void *B,
                                    const void *C, const float *D, const float *h0,
                                    void *y, float *final_state, void *workspace,
                                    size_t ws_bytes, const ssd_plan *plan, void *stream);

/* Device workspace of ssd_forward_host_overlapped for these dims and slice
 * count (0 if the dims are invalid or unsupported). */
SSD_API size_t ssd_forward_host_overlapped_workspace_size(const ssd_dims *dims, ssd_dtype dtype,
                                                          int has_D, int has_h0,
                                                          int want_final_state, int n_slices);

/* ssd_forward_host with the copies overlapped with the computation.  The
 * work is cut into up to n_slices slices: along the batch when batch >= 2,
 * else along the tokens in runs of whole chunks, each slice starting from
 * the previous slice's final state (the recurrence resumes exactly from a
 * final state).  Slice i's host->device copies (its x, dt, B and C rows) run
 * on h2d_stream, its forward pass on `stream`, its device->host copies on
 * d2h_stream, so that slice i+1 uploads while slice i computes and slice i-1
 * downloads; x, dt and y buffers in `workspace` are double-buffered.  The
 * ordering between the three streams uses CUDA events that the call creates
 * and releases itself; no memory is allocated.  `stream` waits for both
 * copy streams before the call returns control of it -- also when the call
 * fails after enqueueing some copies -- so work enqueued on `stream`
 * afterwards sees y and final_state in host memory once it runs, and the
 * host buffers and the workspace may be reused once `stream` reaches it.
 * h2d_stream / d2h_stream may be NULL (that direction then runs on
 * `stream`).  `plan` as for ssd_forward_ex (checked against every slice's
 * dims before anything is enqueued).  Other arguments as for
 * ssd_forward_host; workspace >= ssd_forward_host_overlapped_workspace_size
 * bytes, 256-byte aligned, header zeroed before its first use.  The host
 * buffers should be page-locked for the copies to overlap. */
SSD_API ssd_status ssd_forward_host_overlapped(const ssd_dims *dims, ssd_dtype dtype,
                                               const void *x, const void *dt, const float *A,
                                               const void *B, const void *C, const float *D,
                                               const float *h0, void *y, float *final_state,
                                               void *workspace, size_t ws_bytes, int n_slices,
                                               const ssd_plan *plan, void *stream,
                                               void *h2d_stream, void *d2h_stream);

/* One token of the recurrence for every (batch, head) state -- the
 * recurrent form of the page's section "Mamba-2 architecture", the
 * single-token step of sequential inference:
 *   h[b,h]     = exp(A[h] dt[b,h]) h[b,h] + (dt[b,h] x[b,h,:]) (outer) B[b,g,:]
 *   y[b,h,p]   = sum_s h[b,h,p,s] C[b,g,s] + D[h] x[b,h,p]
 * with g = h / (nh / ng) and the output taken from the updated state.
 * dims: batch, nheads, headdim, dstate, ngroups as for ssd_forward; seqlen
 * must be 1; chunk is ignored.
 * Layouts: x, y [b, nh, P] io; dt [b, nh] io; B, C [b, ng, S] io;
 *   A, D [nh] f32; state [b, nh, P, S] f32, read and overwritten in place.
 *   state has the layout of h0 / final_state of ssd_forward, so decoding can
 *   continue from a forward pass's final state.  D may be NULL (D = 0).
 * Supported: any P >= 1; S a multiple of 4, at most 1024; else
 * SSD_ERR_UNSUPPORTED.  Pointers 16-byte aligned (SSD_ERR_INVALID_ARG
 * otherwise).  Enqueued on `stream`; nothing is allocated. */
SSD_API ssd_status ssd_decode_step(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                                   const void *dt, const float *A, const void *B,
                                   const void *C, const float *D, float *state, void *y,
                                   void *stream);

/* Size in bytes of the fixed device scratch array ssd_forward_noalloc uses as
 * its workspace (32 MiB, reserved per device once the library's module is
 * loaded there). */
#define SSD_NOALLOC_SCRATCH_BYTES (32u << 20)

/* ssd_forward with no workspace argument and no allocation.  The page has no
 * counterpart: this is a calling convention, not a step of the method.
 *
 * Who needs it: callers that cannot allocate device memory when they run the
 * layer -- a runtime that has given all free device memory to its own pool
 * up front and must not take more per call; a plain C caller with no
 * allocator of its own to hand out a workspace; a latency-sensitive loop that
 * cannot accept the device-wide synchronisation that cudaFree implies.
 * Instead of a caller-provided workspace it uses a statically sized array
 * inside this library (SSD_NOALLOC_SCRATCH_BYTES per device), so it calls
 * neither cudaMalloc nor cudaFree nor any library routine that allocates.
 *
 * Limit: dims whose ssd_forward_workspace_size(dims, dtype) exceeds
 * SSD_NOALLOC_SCRATCH_BYTES are rejected with SSD_ERR_UNSUPPORTED before
 * anything is enqueued; use ssd_forward with your own workspace for those
 * (for example bf16, b 4, L 2048, nh 24, P 64, S 128, T 256 needs about
 * 25 MB and fits; b 2, L 4096, nh 80 with the same P, S, T needs about 84 MB
 * and does not).  Invalid dims, dtype or pointers return the same codes as
 * ssd_forward, with nothing enqueued; they are checked before the size, so
 * an oversize call with a NULL tensor still returns SSD_ERR_INVALID_ARG.
 *
 * First-call set-up: the first call in each CUDA context (per device, and
 * again after a device reset or with another context current) looks up the
 * array's device address in that context (cudaGetSymbolAddress, which may
 * also load the library's module there) and caches it under a mutex, keyed
 * by (device, context).  Make one call on each device before starting any
 * stream capture or other region that must not see such set-up; later calls
 * in the same context only read the cache.  SSD_ERR_CUDA if the look-up
 * fails.  A bounded device-side wait that gives up is reported to the
 * library-wide error word (ssd_device_error): the array is not the caller's
 * to read.
 *
 * Concurrency: there is ONE array per device, shared by every call on that
 * device.  Calls whose execution overlaps -- on different streams, or from
 * different host threads without stream ordering between them -- race on it
 * and corrupt each other's results.  Calls on one stream are ordered and
 * safe.  Nothing in the array has to start at zero: each call writes every
 * scratch byte it reads before reading it, so no clearing is needed between
 * calls.  Arguments, layouts, outputs and errors are otherwise those of
 * ssd_forward; the outputs are the values ssd_forward computes for the same
 * inputs. */
SSD_API ssd_status ssd_forward_noalloc(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                                       const void *dt, const float *A, const void *B,
                                       const void *C, const float *D, const float *h0,
                                       void *y, float *final_state, void *stream);

/* ------------------------------------------------------------- backward */

/* Bytes of device workspace ssd_backward needs, including the
 * SSD_WS_HEADER_BYTES header (0 if the dims are invalid or the backward
 * does not support them). */
SSD_API size_t ssd_backward_workspace_size(const ssd_dims *dims, ssd_dtype dtype);

/* Gradients of a loss through the forward pass of ssd_forward.  The pages
 * (section "Mamba-2 architecture") name the backward pass without deriving
 * it; this is the adjoint of the recurrence above, g_t = dL/dh_t =
 * gy_t c_t^T + exp(a_{t+1}) g_{t+1} from g = gfinal after the last token,
 * in the chunked form of the forward:
 *   dx_t  = g_t b_t + D[h] gy_t
 *   dB_t  = sum over the group's heads of dt_t g_t^T x_t
 *   dC_t  = sum over the group's heads of h_t^T gy_t
 *   ddt_t = <B_t, g_t^T x_t> + A[h] sum_{t' >= t} <g_{t'}, h_{t'-1}> exp(a_{t'})
 *   dA[h] = sum over b, t of dt_t sum_{t' >= t} <g_{t'}, h_{t'-1}> exp(a_{t'})
 *   dD[h] = sum over b, t of <gy_t, x_t>,   dh0 = exp(a_1) g_1
 * (the inner sums run over the whole sequence; per chunk they become one
 * reverse cumsum within the chunk and the adjoint state R_k carried between
 * chunks).  In: x, dt, A, B, C, D, h0 as for ssd_forward, gy = dL/dy
 * [b, L, nh, P] and gfinal = dL/dfinal_state [b, nh, P, S].  Out: dx, ddt,
 * dA, dB, dC, dD, dh0 in the layouts of x, dt, A, B, C, D, h0.  D, h0 and
 * gfinal may be NULL (zero); dD and dh0 may be NULL (not written).  The
 * forward's intermediates (G, start states, final state) are recomputed in
 * `workspace` (>= ssd_backward_workspace_size bytes, 256-byte aligned, its
 * first SSD_WS_HEADER_BYTES zeroed before its first use).
 * P = 64, S in {64, 128, 256}.  Every product of the backward, and of the
 * forward states it recomputes, runs in fp32 or near it: the in-chunk
 * products on the CUDA cores in fp32, the GEMM-shaped ones (the chunks'
 * jump terms and the state terms of every token) on the tensor cores with
 * each fp32 operand split into two TF32 parts (three products, about 2^-21
 * relative error each).  With
 * SSD_BF16, x, dt, B, C, gy and dx, ddt, dB, dC are bf16 (converted to and
 * from fp32 copies in the workspace, one launch each way); dA, dD, dh0, A,
 * D, h0 and gfinal are fp32 with either dtype.  dB, dC,
 * dA and dD are summed in a fixed order: repeated calls give the same bits.
 * Allocates nothing and never synchronises. */
SSD_API ssd_status ssd_backward(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                                const void *dt, const float *A, const void *B, const void *C,
                                const float *D, const float *h0, const void *gy,
                                const float *gfinal, void *dx, void *ddt, float *dA, void *dB,
                                void *dC, float *dD, float *dh0, void *workspace,
                                size_t ws_bytes, void *stream);

/* ssd_backward recording CUDA events around its launches, as
 * ssd_forward_profiled does: events[0] before the first launch and
 * events[i] after launch i (i < n_events), *n_launches (may be NULL) = the
 * number of launches, 12: the cumsum, the scaled inputs x~ and gy~, the
 * forward jump terms, the state pass, the adjoint's jump terms, the
 * backward state pass, c_i . B_j per chunk and group, the dx and ysm state
 * terms, the per-token kernel, the per-chunk finish, the reduction and the
 * dB and dC state terms (14 with SSD_BF16: the input conversion first, the
 * output conversion last). */
SSD_API ssd_status ssd_backward_profiled(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                                         const void *dt, const float *A, const void *B,
                                         const void *C, const float *D, const float *h0,
                                         const void *gy, const float *gfinal, void *dx,
                                         void *ddt, float *dA, void *dB, void *dC, float *dD,
                                         float *dh0, void *workspace, size_t ws_bytes,
                                         void *stream, void *const *events, int n_events,
                                         int *n_launches);

/* ---------------------------------------------------------------- plans */

/* Every valid plan for these dims: writes up to max_out plans to `out` (may
 * be NULL when max_out is 0) and returns how many there are (0 for SSD_F32,
 * which has no plan, and for invalid or unsupported dims).  Host-only; needs
 * no GPU. */
SSD_API int ssd_forward_plan_candidates(const ssd_dims *dims, ssd_dtype dtype, ssd_plan *out,
                                        int max_out);

/* The cost-model plan (SSD_ERR_UNSUPPORTED for SSD_F32; the usual codes for
 * invalid dims).  Host-only. */
SSD_API ssd_status ssd_forward_default_plan(const ssd_dims *dims, ssd_dtype dtype,
                                            ssd_plan *out);

/* Timing autotuner for these dims on the current device.  Arguments as for
 * ssd_forward (SSD_BF16 only, else SSD_ERR_UNSUPPORTED).  Runs the forward
 * pass once with the default plan, then times every chunk-jump plan and
 * every output-kernel plan on `stream` (one untimed launch, then `reps`
 * timed launches, 1 <= reps <= 1000), picks the fastest of each (the two
 * kernels are independent), runs the forward pass once more with that
 * combination, and waits for the stream.  With flush NULL the `reps`
 * launches run back to back between two CUDA events (a warm L2); with a
 * device buffer `flush` of flush_bytes > 0 bytes -- larger than the L2 (for
 * example 256 MB) -- each launch is timed alone after the buffer has been
 * overwritten, so every candidate is timed from a cold L2, as a forward pass
 * over fresh inputs runs.  On return y and final_state hold that last pass's
 * results and *chosen (required) the plan, which the caller passes to later
 * calls (ssd_forward_ex); nothing is installed or remembered.  Blocks the
 * host and creates and destroys CUDA events: not for use inside a stream
 * capture. */
SSD_API ssd_status ssd_forward_tune(const ssd_dims *dims, ssd_dtype dtype, const void *x,
                                   const void *dt, const float *A, const void *B,
                                   const void *C, const float *D, const float *h0, void *y,
                                   float *final_state, void *workspace, size_t ws_bytes,
                                   int reps, void *flush, size_t flush_bytes, void *stream,
                                   ssd_plan *chosen);

#ifdef __cplusplus
}
#endif

#endif /* SSD_GB300_H */
