/*
 * ssd.h -- C ABI of the GB300 (sm_103a) Mamba-2 SSD chunked forward.
 *
 * The operation is the Mamba-2 layer recurrence of "Accelerating Mamba-2 with
 * High-Performance Forward Pass Kernels in NVIDIA CUDA Tile", section
 * "Mamba-2 architecture":
 *
 *     h_t = exp(A[h] * dt_t) * h_{t-1} + dt_t * x_t (outer) B_t      (P x N state)
 *     y_t = h_t C_t + D[h] * x_t                                        (updated state)
 *
 * evaluated chunk by chunk in four stages (sections "Kernel 1: Computing
 * cumulative sums", "Kernel 2: fwd_pass_state", "Kernel 3: compute_out"):
 * chunk_cumsum, chunk_state, state_passing, chunk_scan.  Head h reads group
 * g = h / (H / G) of B and C.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensors are described by ssd_tensor: a pointer, a dtype, and shape and
 *   strides in ELEMENTS.  The innermost stride must be 1.  Pointers passed
 *   to the compute entry points are DEVICE pointers of the current device.
 * - Shapes (B batch, L seqlen, H nheads, P headdim, N dstate, G ngroups,
 *   Q chunk_size, nc = ceil(L / Q)):
 *     x  [B, L, H, P]  bf16 or f32        dt [B, L, H] f32 (post-softplus, >= 0)
 *     A  [H]           f32 (<= 0)         D  [H] f32, optional (absent = 0)
 *     B  [B, L, G, N]  dtype of x         C  [B, L, G, N] dtype of x
 *     initial_states [B, H, P, N] f32, optional (absent = 0)
 *     y  [B, L, H, P]  dtype of x         final_states [B, H, P, N] f32, optional
 *   The sign conditions on dt and A are the method's premises (every kept
 *   exponent is <= 0); they are documented, not checked.
 * - Supported geometry: P and N in {16, 32, 64, 128}; Q in {64, 128, 256};
 *   H a multiple of G.  Anything else returns SSD_ERR_UNSUPPORTED.
 * - Alignment: every base pointer 16-byte aligned; for x, B, C and y every
 *   outer stride a multiple of 16 bytes.  Violations return SSD_ERR_ALIGNMENT.
 * - Ownership: the caller owns every buffer, workspace included.  The library
 *   never allocates, frees or synchronises; all work is enqueued in order on
 *   `stream` and returns asynchronously.  Inputs must stay alive until the
 *   stream passes this call.  `stream` is a cudaStream_t (NULL = the legacy
 *   default stream).
 * - Errors: every check runs on the host before any launch; on failure the
 *   call returns a status, launches nothing, and ssd_last_error_detail()
 *   names the check and its figures.  A launch failure returns SSD_ERR_CUDA.
 *   No C++ exception crosses this boundary.
 * - Aliasing: outputs must not overlap inputs (checked by address range).
 * - Results are deterministic: repeated calls give bitwise-identical outputs
 *   (no floating-point atomics).
 * - Device state: the library keeps two objects in device memory of its own
 *   (a device error word, and the static scratch array of
 *   ssd_chunked_fwd_static_scratch) and looks up their addresses once per
 *   device, on first use.  cudaDeviceReset discards them, so do not reset a
 *   device the library has been used on in the same process.  The cached
 *   addresses belong to the context current at that first use: call the
 *   library from the device's primary context (what the CUDA runtime uses
 *   by default), not from contexts created with the driver API.
 */
#ifndef SSD_GB300_H
#define SSD_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1, /* null pointer, bad shape, dtype or aliasing  */
    SSD_ERR_UNSUPPORTED = 2, /* valid but outside the supported geometry     */
    SSD_ERR_ALIGNMENT = 3,   /* pointer or stride alignment                  */
    SSD_ERR_WORKSPACE = 4,   /* workspace missing or too small               */
    SSD_ERR_CUDA = 5,        /* a CUDA runtime or launch error               */
    SSD_ERR_TIMEOUT = 6,     /* a device-side bounded wait gave up           */
    SSD_ERR_DEVICE_BOUNDS = 7 /* a device-side bounds check failed (debug
                                 build only: libssd_gb300_debug.so)          */
} ssd_status;

/* SSD_I32 only for the parent and state-slot indices of ssd_state_update_tokens
 * and the conv-state slot indices of ssd_mixer_prologue. */
typedef enum { SSD_F32 = 0, SSD_BF16 = 1, SSD_I32 = 2 } ssd_dtype;

typedef struct {
    void *data;          /* device pointer                                   */
    int32_t dtype;       /* ssd_dtype                                        */
    int32_t ndim;        /* number of valid entries in shape / stride        */
    int64_t shape[5];
    int64_t stride[5];   /* in elements                                      */
} ssd_tensor;

/* Human-readable name of a status code (static storage). */
const char *ssd_status_string(ssd_status status);

/* Text of the last failed check on the calling thread (thread-local storage,
 * valid until the next call on that thread); "" after a successful call. */
const char *ssd_last_error_detail(void);

/* Waits for `stream`, then reports (and clears) the device-side error word of
 * the current device: SSD_ERR_DEVICE_BOUNDS if a kernel of the debug build
 * (compiled with SSD_DEBUG_BOUNDS) found an index, shared-memory offset or
 * tensor-memory column out of range (ssd_last_error_detail names the source
 * file and line of the first one; the access was skipped, not made),
 * SSD_ERR_TIMEOUT if any kernel gave up a bounded wait since the last call
 * (its outputs are then not valid), SSD_OK otherwise, SSD_ERR_CUDA if CUDA
 * itself reports an error.  This is the only entry point that synchronises;
 * call it where a check is wanted. */
ssd_status ssd_device_status(void *stream);

/* Test hook for the failure path above: launches one CTA on `stream` whose
 * bounded wait (on an mbarrier phase nothing completes) gives up after
 * limit_ns (at most 100 ms) and records the timeout in the device error word,
 * the same way every kernel of the library does.  The next ssd_device_status
 * on that stream then returns SSD_ERR_TIMEOUT and clears the word.  Nothing
 * else is in flight in that CTA, so the context stays usable. */
ssd_status ssd_selftest_wait_timeout(uint64_t limit_ns, void *stream);

/* Test hook for the debug build's bounds checks (libssd_gb300_debug.so, built
 * with SSD_DEBUG_BOUNDS; they stand in for a memory checker): launches one
 * thread on `stream` that tests an index out of range by construction.  The
 * check records the failure in the device error word and skips the access
 * (no memory is touched); the next ssd_device_status on that stream returns
 * SSD_ERR_DEVICE_BOUNDS naming ssd_selftest.cu and clears the word.  The
 * normal build returns SSD_ERR_UNSUPPORTED and launches nothing. */
ssd_status ssd_selftest_bounds_check(void *stream);

/* Bytes of device workspace ssd_chunked_fwd needs for this problem, written
 * to *bytes.  x_dtype is the ssd_dtype of x, B, C.  On the four-step path the
 * workspace holds the scaled in-chunk cumulative sums G [B, H, nc*Q] f32, the
 * per-chunk states [B, nc, H, P, N] f32 and the chunk-entering states
 * [B, nc, H, P, N] in the dtype of x; for f32 inputs with P = 64, N = 128 and
 * Q of 128 or 256 (chunk_state and chunk_scan on the tensor cores) it also
 * holds bf16 hi / lo copies of x, B, C and the chunk-entering states.  The
 * fused path needs none, except when the (batch, head) or (batch, head pair)
 * slabs do not fill whole waves of SMs and it splits the remainder by
 * sequence: then it holds each segment's local state, decay and entering
 * state (at most 64 MiB; ssd_describe_plan names the split).  The answer
 * depends on the SM count of the current device.  Returns
 * SSD_ERR_INVALID_ARG / SSD_ERR_UNSUPPORTED for shapes ssd_chunked_fwd would
 * reject. */
ssd_status ssd_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads,
                              int64_t headdim, int64_t dstate, int64_t ngroups,
                              int64_t chunk_size, int32_t x_dtype,
                              size_t *bytes);

/* One line naming the kernels ssd_chunked_fwd would launch for this problem
 * ("fused: ..." for the single-kernel path, "staged: ..." for the four-step
 * path), or the reason it would be rejected.  Thread-local storage, valid
 * until the next call on the thread.  Never launches or touches the GPU. */
const char *ssd_describe_plan(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                              int64_t dstate, int64_t ngroups, int64_t chunk_size,
                              int32_t x_dtype);

/* The SSD chunked forward: y and (optionally) final_states from x, dt, A, B,
 * C, D, initial_states, as defined at the top of this file.  A sequence
 * length that is not a multiple of chunk_size is handled as if zero-padded
 * (dt = x = B = C = 0 on the padding), which changes nothing; only the L real
 * tokens of y are written.  D, initial_states and final_states may be NULL.
 * workspace: device memory of at least ssd_workspace_size() bytes, 256-byte
 * aligned, owned by the caller; its contents on entry are ignored. */
ssd_status ssd_chunked_fwd(const ssd_tensor *x, const ssd_tensor *dt,
                           const ssd_tensor *A, const ssd_tensor *B,
                           const ssd_tensor *C, const ssd_tensor *D,
                           const ssd_tensor *initial_states,
                           int64_t chunk_size, int64_t ngroups,
                           ssd_tensor *y, ssd_tensor *final_states,
                           void *workspace, size_t workspace_bytes,
                           void *stream);

/* The same forward with the mixer's output gate applied to y: "Optimizing
 * Nemotron v3 Super in TensorRT-LLM", section 6.2 (out * silu(z)), here for
 * every token of the prefill:
 *
 *   y[b, t, h, p] = (the ssd_chunked_fwd output) * silu(z[b, t, h, p]),
 *   silu(z) = z / (1 + exp(-z))
 *
 * z [B, L, H, P] in the dtype of x, 16-byte aligned base, outer strides
 * multiples of 16 bytes, overlapping no output.  The gate is one more launch
 * after the scan (on either plan), in place on y: y read and written, z read
 * once.  Everything else as ssd_chunked_fwd (same workspace size). */
ssd_status ssd_chunked_fwd_gated(const ssd_tensor *x, const ssd_tensor *dt,
                                 const ssd_tensor *A, const ssd_tensor *B,
                                 const ssd_tensor *C, const ssd_tensor *D,
                                 const ssd_tensor *z, const ssd_tensor *initial_states,
                                 int64_t chunk_size, int64_t ngroups, ssd_tensor *y,
                                 ssd_tensor *final_states, void *workspace,
                                 size_t workspace_bytes, void *stream);

/* ---- sequence sharding over ranks -------------------------------------------
 * "mamba-metal", "The essence of selective scan": the recurrence
 * h_t = a_t h_{t-1} + b_t over a run of tokens composes into one pair
 * (a, b) = (total decay, state reached from zero), and pairs compose
 * associatively in sequence order, (a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2).
 * A sequence split into contiguous segments, one per rank (rank order =
 * sequence order), is run as: every rank calls ssd_chunked_fwd on its segment
 * with no initial state (its y from zero, its final state b) and
 * ssd_segment_logdecay (log a); the ranks exchange (log a, b); each rank calls
 * ssd_sequence_combine for the state h_in entering its segment and
 * ssd_shard_correct, which adds h_in's contribution to y and turns b into the
 * rank's final state.  The result is the unsplit forward's up to rounding (y
 * is rounded twice in bf16 runs).  The exchange itself is the caller's (the
 * Python binding's chunked_fwd_sequence_sharded uses torch.distributed).
 * Same conventions as ssd_chunked_fwd: device pointers, every check before
 * any launch, work enqueued on `stream`, no allocation. */

/* logdecay[b, h] = A[h] * sum_t dt[b, t, h] (natural log of the segment's
 * total decay).  dt [B, L, H] f32 (innermost stride 1), A [H] f32,
 * logdecay [B, H] f32 contiguous (output). */
ssd_status ssd_segment_logdecay(const ssd_tensor *dt, const ssd_tensor *A,
                                ssd_tensor *logdecay, void *stream);

/* h_in = the composition of the pairs of ranks 0 .. rank - 1, applied to
 * initial_states (or zero): h <- exp(logdecay[q]) h + states[q] for q = 0 ..
 * rank - 1.  logdecay [R, B, H] f32, states [R, B, H, P, N] f32 (the gathered
 * pairs of all R ranks), initial_states [B, H, P, N] f32 or NULL (the state
 * entering the whole sequence), h_in [B, H, P, N] f32 (output), all
 * contiguous; 0 <= rank < R. */
ssd_status ssd_sequence_combine(const ssd_tensor *logdecay_all, const ssd_tensor *states_all,
                                const ssd_tensor *initial_states, int32_t rank,
                                ssd_tensor *h_in, void *stream);

/* In place: y[b, t, h, :] += exp(cum[b, t, h]) * C[b, t, g, :] . h_in[b, h]^T
 * with cum the inclusive prefix over the segment of A[h] dt[b, ., h] and g =
 * h / (H / ngroups), and, if final_states is given, final_states <-
 * exp(logdecay) h_in + final_states.  y [B, L, H, P] (f32 or bf16; innermost
 * stride 1) holds the segment's output from a zero state and C [B, L, G, N]
 * has y's dtype; dt, A as for ssd_chunked_fwd; h_in, final_states
 * [B, H, P, N] f32 and logdecay [B, H] f32, contiguous. */
ssd_status ssd_shard_correct(const ssd_tensor *dt, const ssd_tensor *A, const ssd_tensor *C,
                             const ssd_tensor *h_in, const ssd_tensor *logdecay,
                             int64_t ngroups, ssd_tensor *y, ssd_tensor *final_states,
                             void *stream);

/* ---- allocation-free variant ------------------------------------------------
 * The pages have no counterpart of this call; it exists for callers that
 * cannot hand the library a device workspace: code that runs where no
 * allocator is reachable (a plug-in inside a host program that owns all
 * device memory and exposes no workspace hook), or where calling cudaMalloc
 * is not acceptable (it may synchronise the device and its latency is
 * unbounded, which a fixed-latency loop cannot afford).
 *
 * Same inputs, outputs and results as ssd_chunked_fwd, but its scratch comes
 * from one file-scope __device__ array of SSD_STATIC_SCRATCH_BYTES that every
 * GPU loading this library holds until the process exits.  The call
 * allocates and frees nothing.  Problems whose scratch (ssd_workspace_size)
 * exceeds SSD_STATIC_SCRATCH_BYTES are rejected with SSD_ERR_WORKSPACE before
 * any launch.  The first call on a device (with that device current) looks
 * up the array's device address and caches it; make that first call before
 * any stream capture.  All calls on a device share the one array, which
 * keeps the last call's contents (nothing in it needs to start at zero:
 * every byte a call reads is written earlier in that call), so calls whose
 * execution overlaps on the GPU (different streams, no ordering) race and
 * corrupt each other's results: order them on one stream or with events. */
#define SSD_STATIC_SCRATCH_BYTES ((size_t)64 << 20)

ssd_status ssd_chunked_fwd_static_scratch(const ssd_tensor *x, const ssd_tensor *dt,
                                          const ssd_tensor *A, const ssd_tensor *B,
                                          const ssd_tensor *C, const ssd_tensor *D,
                                          const ssd_tensor *initial_states,
                                          int64_t chunk_size, int64_t ngroups,
                                          ssd_tensor *y, ssd_tensor *final_states,
                                          void *stream);

/* ---- decode step ------------------------------------------------------------ */

/* One decode token of the layer: the selective state update of "Optimizing
 * Nemotron v3 Super in TensorRT-LLM", section 6.1 "The SSU Math", with the
 * dt bias, softplus and z gate of section 6.2's reference.  For every
 * (b, h), with g = h / (H / G):
 *
 *   dt'  = dt[b, h] + dt_bias[h]                    (dt_bias optional, absent = 0)
 *   dt'  = log(1 + exp(dt'))                        (if dt_softplus; dt' above 20
 *                                                    is kept as is, the same in fp32)
 *   state[b, h] = exp(A[h] dt') state[b, h] + dt' x[b, h] (outer) B[b, g]
 *   out[b, h, p] = sum_n state[b, h, p, n] C[b, g, n] + D[h] x[b, h, p]
 *   out *= silu(z[b, h]) = z / (1 + exp(-z))        (if z is given)
 *
 * Shapes, dtypes and layouts:
 *   state [B, H, P, N] f32 or bf16, packed, read and updated in place
 *   x     [B, H, P] bf16 or f32                  z   [B, H, P] dtype of x, optional
 *   dt    [B, H] f32 (post-softplus unless dt_softplus, then raw)
 *   A     [H] f32 (<= 0)                         D, dt_bias [H] f32, optional
 *   B, C  [B, G, N] dtype of x, same strides     out [B, H, P] dtype of x
 * The state is the one ssd_chunked_fwd returns as final_states, so prefill
 * followed by decode steps continues the same recurrence.  A bf16 state is the
 * 16-bit state cache of the same page's section 6.4.3 (the layout it dispatches
 * to on Blackwell): the update and out are computed in fp32 from the stored
 * values, out from the unrounded new state, and the state is stored rounded to
 * nearest even (the state's dtype is the storage format only).  P and N in
 * {16, 32, 64, 128}; H a multiple of G.  Alignment: state, B and C base
 * pointers 16-byte aligned, B and C outer strides multiples of 16 bytes.
 * Aliasing: out must not overlap any input or the state, and the state must
 * not overlap any input.  Errors, ownership and streams as above; the state
 * is modified only if the call returns SSD_OK (nothing is launched on error).
 * One launch, no workspace. */
ssd_status ssd_state_update(ssd_tensor *state, const ssd_tensor *x, const ssd_tensor *dt,
                            const ssd_tensor *A, const ssd_tensor *B, const ssd_tensor *C,
                            const ssd_tensor *D, const ssd_tensor *z,
                            const ssd_tensor *dt_bias, int32_t dt_softplus,
                            int64_t ngroups, ssd_tensor *out, void *stream);

/* T decode tokens per sequence in one call, as in speculative decoding, where
 * the draft tokens of each sequence are checked together: "Optimizing Nemotron
 * v3 Super in TensorRT-LLM", section 10.3 "Stateful SSM Caching for
 * Speculative Decoding" and section 10.4 "Multi-Token State Update Kernel".
 * For every (b, h), with s the running P x N state:
 *
 *   s = state[b, h]
 *   for t = 0 .. T-1:
 *       if parent and t > 0 and 0 <= parent[b, t] < t:
 *           s = intermediate_states[b, parent[b, t], h]     (a tree of drafts)
 *       s = exp(A[h] dt') s + dt' x[b, t, h] (outer) B[b, t, g]   (dt' as above)
 *       intermediate_states[b, t, h] = s                  (if given)
 *       out[b, t, h, p] = (sum_n s[p, n] C[b, t, g, n] + D[h] x[b, t, h, p])
 *                         * silu(z[b, t, h, p])           (z optional)
 *   state[b, h] = s                                       (if update_state != 0)
 *
 * Token t starts from the state after token t - 1, unless parent[b, t] names
 * an earlier token of the same call (0 <= parent[b, t] < t): then it starts
 * from the state after that token.  Other parent values (-1, say) keep the
 * chain; parent[b, 0] is not read.  With update_state = 0 the state is left
 * as it was (a verification pass: the accepted step's intermediate state is
 * promoted by the caller).
 *
 * Continuous batching (the serving kernel's state_batch_idx and pad_slot_id,
 * same section): with state_indices given, the state and intermediate_states
 * are pools of S slots and row b uses slot state_indices[b] of both (the
 * state[b, h] and intermediate_states[b, t, h] above read [state_indices[b],
 * ...]).  A row whose index lies outside [0, S) (a negative pad id, say) is
 * padding: nothing is read or written for it, its out rows included.  Slots
 * of real rows must be distinct (not checked: two rows on one slot race).
 *
 * Shapes, dtypes and layouts (the token axis second):
 *   state [B, H, P, N] f32 or bf16, packed (bf16: rounded as for ssd_state_update,
 *         after every token: the s of the next token is the rounded one);
 *         [S, H, P, N] with state_indices
 *   x, z, out [B, T, H, P] bf16 or f32 (z optional, out the dtype of x)
 *   dt    [B, T, H] f32                          A, D, dt_bias [H] f32
 *   B, C  [B, T, G, N] dtype of x, same strides
 *   intermediate_states [B, T, H, P, N] dtype of the state, packed, optional
 *         (required with parent); [S, T, H, P, N] with state_indices
 *   parent [B, T] SSD_I32, optional
 *   state_indices [B] SSD_I32, contiguous, optional
 * T = 1 without intermediate states or parents is ssd_state_update.  Alignment
 * as for ssd_state_update, plus intermediate_states 16-byte aligned.  Aliasing:
 * out, the state and intermediate_states overlap neither each other nor any
 * input.  Errors, ownership and streams as above.  One launch, no workspace;
 * the state is read and written once whatever T. */
ssd_status ssd_state_update_tokens(ssd_tensor *state, const ssd_tensor *x, const ssd_tensor *dt,
                                   const ssd_tensor *A, const ssd_tensor *B, const ssd_tensor *C,
                                   const ssd_tensor *D, const ssd_tensor *z,
                                   const ssd_tensor *dt_bias, int32_t dt_softplus,
                                   int64_t ngroups, ssd_tensor *out,
                                   ssd_tensor *intermediate_states, const ssd_tensor *parent,
                                   const ssd_tensor *state_indices, int32_t update_state,
                                   void *stream);

/* ---- mixer prologue ----------------------------------------------------------
 * The steps of the Mamba-2 mixer between its input projection and the scan, in
 * one pass: the causal depthwise convolution with SiLU over the xBC channels,
 * the split of its output into x, B and C, and the dt preparation -- "Optimizing
 * Nemotron v3 Super in TensorRT-LLM", sections 6.2 (dt + dt_bias, softplus),
 * 7.1 (the split written directly in the layout the scan reads), 8
 * ("CausalConv1d Optimization") and 10.3 / 10.5 (the conv state and its
 * per-token windows).  With u the inputs of a sequence preceded by conv_state
 * (its last W inputs so far, oldest first; zeros when conv_state is NULL):
 *
 *   xbc[b, t, c] = silu(conv_bias[c] + sum_k conv_weight[c, k] u[b, t - (W-1) + k, c])
 *   x = xbc[..., 0 : H P] as [B, L, H, P]
 *   B = xbc[..., H P : H P + G N] as [B, L, G, N],   C = xbc[..., H P + G N :]
 *   dt_out = dt + dt_bias, then log(1 + exp(.)) if dt_softplus (kept as is above
 *            20, the same in fp32)
 *   conv_state <- the last W inputs of u (in place);
 *   conv_windows[b, t] = the last W inputs up to and including token t
 *
 * Shapes, dtypes and layouts:
 *   xBC [B, L, Dc] bf16 or f32, Dc = H P + 2 G N (H and P from x, N from B)
 *   conv_weight [Dc, W] f32, packed, W in 1..4 (weight[:, W-1] takes the
 *     current token); conv_bias [Dc] f32, optional
 *   conv_state [B, Dc, W] dtype of xBC, packed, optional
 *   conv_windows [B, L, Dc, W] dtype of xBC, packed, optional
 *   conv_state_indices [B] SSD_I32, contiguous, optional (needs conv_state):
 *     the conv_state_indices of section 10.5 -- conv_state and conv_windows
 *     become pools [S, Dc, W] and [S, L, Dc, W] and row b reads and writes
 *     slot conv_state_indices[b] of both; a row whose index lies outside
 *     [0, S) is padding: nothing is read or written for it, its x, B, C and
 *     dt_out rows included.  Real rows must name distinct slots (not checked).
 *   dt, dt_out [B, L, H] f32; dt_bias [H] f32, optional
 *   x [B, L, H, P], B and C [B, L, G, N], dtype of xBC (outputs)
 * The outputs are what ssd_chunked_fwd takes as x, dt, B and C.  Alignment:
 * xBC, x, B, C base pointers 16-byte aligned and their outer strides multiples
 * of 16 bytes.  Aliasing: no output (the conv state included) may overlap an
 * input or another output.  P and N in {16, 32, 64, 128}.  Errors,
 * ownership and streams as above; one launch (two when conv_state is given and
 * a sequence is split over several CTAs, which needs L > 8), no workspace. */
ssd_status ssd_mixer_prologue(const ssd_tensor *xBC, const ssd_tensor *conv_weight,
                              const ssd_tensor *conv_bias, ssd_tensor *conv_state,
                              ssd_tensor *conv_windows, const ssd_tensor *conv_state_indices,
                              const ssd_tensor *dt, const ssd_tensor *dt_bias,
                              int32_t dt_softplus, int64_t ngroups, ssd_tensor *x,
                              ssd_tensor *B, ssd_tensor *C, ssd_tensor *dt_out, void *stream);

/* ---- stage entry points (the four steps of ssd_chunked_fwd, one call each;
 *      same conventions; used to check each step on its own) ---------------- */

/* Step 1, "Kernel 1: Computing cumulative sums": for every chunk c,
 *   G[b, h, c*Q + k] = log2(e) * sum_{k' <= k} A[h] * dt[b, c*Q + k', h]
 * over the zero-padded sequence (so positions past L repeat the chunk's last
 * real value).  G: [B, H, nc*Q] f32, contiguous. */
ssd_status ssd_stage_chunk_cumsum(const ssd_tensor *dt, const ssd_tensor *A,
                                  int64_t chunk_size, ssd_tensor *G,
                                  void *stream);

/* Step 2, the jump formula of "Kernel 2: fwd_pass_state" without the carried
 * state: the state one chunk leaves behind when it starts from zero,
 *   S[b, c, h, p, n] = sum_{j in chunk c} 2^(G_last - G_j) dt_j x_j[p] B_j[n]
 * with G_last = G[b, h, c*Q + Q - 1].  S: [B, nc, H, P, N] f32, contiguous. */
ssd_status ssd_stage_chunk_state(const ssd_tensor *x, const ssd_tensor *B,
                                 const ssd_tensor *dt, const ssd_tensor *G,
                                 int64_t chunk_size, int64_t ngroups,
                                 ssd_tensor *S, void *stream);

/* Step 3, the sequential loop of "Kernel 2: fwd_pass_state": for each (b, h),
 *   h_prev[0] = initial_states (or 0),
 *   h_prev[c+1] = 2^(G_last,c) h_prev[c] + S[c],   final = h_prev[nc]
 * in fp32.  h_prev: [B, nc, H, P, N] f32 or bf16 (stored rounded), contiguous;
 * final_states may be NULL. */
ssd_status ssd_stage_state_passing(const ssd_tensor *S, const ssd_tensor *G,
                                   const ssd_tensor *initial_states,
                                   int64_t chunk_size, ssd_tensor *h_prev,
                                   ssd_tensor *final_states, void *stream);

/* Step 4, "Kernel 3: compute_out": per chunk,
 *   Y = 2^G (C h_prev^T) + (2^(G_i - G_j) (C B^T)_ij [j <= i]) (dt x) + D x
 * with the causal selection taken before any exponent is used.  h_prev must
 * have the dtype of x for bf16 inputs and f32 for f32 inputs. */
ssd_status ssd_stage_chunk_scan(const ssd_tensor *x, const ssd_tensor *dt,
                                const ssd_tensor *G, const ssd_tensor *B,
                                const ssd_tensor *C, const ssd_tensor *D,
                                const ssd_tensor *h_prev, int64_t chunk_size,
                                int64_t ngroups, ssd_tensor *y, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SSD_GB300_H */
