/*
 * ssd.h -- C ABI of libssd_b300.so, the B300 (sm_103a) forward pass of the
 * SSD chunked scan, the sequence-mixing layer of Mamba-2.
 *
 * The operation (Structured State Space Duality, "The recurrence as one
 * matrix"; scalar-times-identity decay as in the same section; the general
 * diagonal decay of "What the duality gives up" and of "On Structured
 * State-Space Duality", abstract, point (i)):
 *
 *   for every batch row bi and head h, with g = h / (H / G):
 *     h_{-1} = init_state[bi,h]                      (zero when NULL)
 *     a_t    = exp(dt[bi,t,h] * A[h])                (scalar A, shape (H))
 *     a_t[n] = exp(dt[bi,t,h] * A[h,n])              (diagonal A, shape (H,N))
 *     h_t    = a_t (.) h_{t-1} + B[bi,t,g,:] x[bi,t,h,:]^T          (N x P)
 *     y[bi,t,h,:] = C[bi,t,g,:]^T h_t + D[h] x[bi,t,h,:]            (D optional)
 *     final_state[bi,h] = h_{T-1}
 *
 * It is evaluated by the chunked algorithm of the same page ("The chunked
 * algorithm takes both"): chunks of Q tokens; inside a chunk the decay-masked
 * quadratic form (C B^T o L) X on tensor cores; across chunks one fp32 state
 * recurrence step per chunk ("When it breaks": decay sums and state in fp32).
 * The result equals the recurrence up to rounding for every Q.
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers to dense row-major arrays in
 *     the layouts given below, owned by the caller.  The library allocates no
 *     memory and keeps no pointer after a call returns.
 *   - Every pointer must be 16-byte aligned (SSD_ERR_ALIGNMENT otherwise),
 *     except in ssd_scan and ssd_decode_step (element alignment).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  The library never synchronises except in
 *     ssd_check_device_status.
 *   - Every function returns an int status (SSD_OK = 0).  All argument checks
 *     run before anything is enqueued; on any argument error nothing is
 *     enqueued (dims beyond a path's launch or index limits are rejected as
 *     SSD_ERR_UNSUPPORTED there).  A CUDA runtime failure while enqueueing
 *     returns SSD_ERR_CUDA and may leave the work enqueued before it.
 *   - Not reentrant on one workspace: two calls that share a workspace must be
 *     ordered on the GPU (same stream or an event between them).
 */
#ifndef SSD_B300_H
#define SSD_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSD_ABI_VERSION 1

#if defined(__GNUC__)
#define SSD_API __attribute__((visibility("default")))
#else
#define SSD_API
#endif

/* ---- status codes ---------------------------------------------------- */
#define SSD_OK              0
#define SSD_ERR_INVALID_ARG 1  /* a size, mode or required pointer is invalid   */
#define SSD_ERR_UNSUPPORTED 2  /* valid, but outside what this build handles    */
#define SSD_ERR_ALIGNMENT   3  /* a pointer is not 16-byte aligned              */
#define SSD_ERR_WORKSPACE   4  /* workspace NULL or smaller than required       */
#define SSD_ERR_CUDA        5  /* a CUDA runtime/driver call or launch failed   */
#define SSD_ERR_TIMEOUT     6  /* device side: a bounded inter-CTA wait expired  */
#define SSD_ERR_DEVICE      7  /* device side: a kernel's own check failed       */
#define SSD_ERR_SCRATCH_LIMIT 8 /* ssd_fwd_noalloc: problem exceeds its scratch  */

/* ---- modes ----------------------------------------------------------- */
#define SSD_A_SCALAR   0       /* A has shape (H): a_t = exp(dt_t A_h) I        */
#define SSD_A_DIAGONAL 1       /* A has shape (H,N): one decay per state dim    */

#define SSD_DTYPE_BF16 0       /* x, B, C, y are bfloat16                       */
#define SSD_DTYPE_F32  1       /* x, B, C, y are float32                        */

#define SSD_PATH_AUTO     0    /* pick the fastest path that supports the dims   */
#define SSD_PATH_GENERIC  1    /* CUDA-core fp32 pipeline (any supported dims)   */
#define SSD_PATH_TCGEN05  2    /* fused tcgen05/TMA kernel (restricted dims)     */

/* Problem description.  Names follow the pages' notation:
 *   b batch, T sequence length, H heads, P head dim, N state dim,
 *   G B/C groups (H % G == 0), Q chunk length.
 * Constraints: b >= 0, T >= 0, H >= 1, G >= 1, H % G == 0,
 *   1 <= P <= 256 and P a power of two, 1 <= N <= 256, N * P <= 16384,
 *   Q in {64, 128, 256}.
 * b == 0 or T == 0 is a valid empty problem: y is empty and final_state is
 * init_state (or zero).  A ragged last chunk (T % Q != 0) is allowed.
 * Domain (not checked on the device): dt >= 0 and A <= 0, all finite.  The
 * tcgen05 paths keep their matrix operands in fp16: when x, B, C, a C B^T entry
 * or a state entry entering a 128-token block leaves the fp16 range
 * (|v| > 65504), the call reports SSD_ERR_DEVICE through
 * ssd_check_device_status and its outputs are invalid; the generic path has
 * no such limit (SSD_PATH_GENERIC computes such inputs in fp32).  Outside the
 * domain (a growing decay) the tcgen05 paths' decay factors can leave fp16 as
 * well, with the same report. */
typedef struct ssd_dims {
    int64_t b, T, H, P, N, G, Q;
    int32_t a_mode;    /* SSD_A_SCALAR or SSD_A_DIAGONAL                       */
    int32_t io_dtype;  /* SSD_DTYPE_BF16 or SSD_DTYPE_F32                      */
    int32_t path;      /* SSD_PATH_*; SSD_PATH_AUTO unless testing a path      */
    int32_t reserved;  /* must be 0                                            */
} ssd_dims;

/* Paths.  SSD_PATH_TCGEN05 is one persistent kernel with TMA loads and tcgen05
 * tensor-core products accumulating in TMEM:
 *  - scalar A: bf16 io, P == 64, N in {128, 256}, Q in {128, 256}; the state
 *    passes block to block through an L2-resident ring;
 *  - diagonal A: bf16 io, P == N == 64, any Q; one CTA per (batch row, head) at
 *    a time keeps the state in TMEM, and every decay is split at a reference
 *    token so that the fp16 operands carry factors <= 1 (the pairs inside one
 *    16-token group are summed in fp32 on the CUDA cores).
 * Both evaluate every chunk as 128-token blocks (the chunked algorithm applied
 * inside the chunk, equal up to rounding).  SSD_PATH_GENERIC (fp32 CUDA-core
 * kernels) takes every dims the ABI accepts.  SSD_PATH_AUTO picks TCGEN05 where
 * it applies.
 *
 * Bytes of device workspace ssd_fwd needs for `dims` (written to *bytes).
 * Host-only; enqueues nothing.  Returns SSD_ERR_INVALID_ARG /
 * SSD_ERR_UNSUPPORTED for dims ssd_fwd would reject. */
SSD_API int ssd_fwd_workspace_size(const ssd_dims *dims, size_t *bytes);

/* The kernel path ssd_fwd would run for `dims` (SSD_PATH_GENERIC or
 * SSD_PATH_TCGEN05), written to *path.  Host-only. */
SSD_API int ssd_fwd_path(const ssd_dims *dims, int32_t *path);

/* Forward pass.  Layouts (all dense, row-major, device memory):
 *   x           (b,T,H,P)  io dtype         read
 *   dt          (b,T,H)    float32          read
 *   A           (H) or (H,N) float32        read (per a_mode)
 *   B, C        (b,T,G,N)  io dtype         read
 *   D           (H)        float32 or NULL  read; NULL = no skip term
 *   init_state  (b,H,N,P)  float32 or NULL  read; NULL = zero state
 *   y           (b,T,H,P)  io dtype         written
 *   final_state (b,H,N,P)  float32 or NULL  written; NULL = not returned
 *   workspace   >= ssd_fwd_workspace_size bytes, device memory, 256-byte
 *               aligned; scratch owned by the caller, contents need no
 *               initialisation and are undefined after the call.
 * y must not alias any input.  Returns after enqueueing the kernels on
 * `stream`; errors found on the device (SSD_ERR_TIMEOUT, SSD_ERR_DEVICE)
 * are reported by ssd_check_device_status. */
SSD_API int ssd_fwd(const ssd_dims *dims,
            const void *x, const float *dt, const float *A,
            const void *B, const void *C, const float *D,
            const float *init_state,
            void *y, float *final_state,
            void *workspace, size_t workspace_bytes,
            void *stream);

/* Synchronises `stream`, then reads the device-side status word that the
 * last ssd_fwd on this workspace left, and clears it.  Returns SSD_OK,
 * SSD_ERR_TIMEOUT (an inter-CTA wait hit its iteration limit; outputs are
 * invalid), SSD_ERR_DEVICE, or SSD_ERR_CUDA if the stream reported an error. */
SSD_API int ssd_check_device_status(void *workspace, size_t workspace_bytes, void *stream);

/* Static English text for a status code (never NULL). */
SSD_API const char *ssd_status_string(int status);

/* SSD_ABI_VERSION of the loaded library. */
SSD_API int ssd_abi_version(void);

/* Test hook for the failure-detection path of the fused kernel.
 * The fused kernel hands the state from one 128-token block of a sequence to
 * the next through global memory; each wait for it is bounded.
 * spin_limit: iteration limit of each such wait (<= 0 restores the default).
 * withhold_chunk: when >= 0, the work items of 128-token block number
 * withhold_chunk never publish their state, so the next block's wait runs out,
 * continues with a zero state, and the call reports SSD_ERR_TIMEOUT through
 * ssd_check_device_status.  Process-wide; not for production use.
 * Returns SSD_OK. */
SSD_API int ssd_debug_set_wait(int64_t spin_limit, int64_t withhold_chunk);

/* Linear form.  The same map as ssd_fwd, same arguments and layouts, no
 * workspace, evaluated by the recurrence itself, token by token, on CUDA
 * cores: one block per (batch row, head) keeps the N x P state in registers
 * for the whole sequence (Structured State Space Duality, "The recurrence as
 * one matrix": the O(T) linear form, against which the pages set the
 * chunked algorithm).  dims->path must be SSD_PATH_AUTO; dims->Q is checked
 * like ssd_fwd's but not used.  Supported: every dims ssd_fwd accepts.
 * init_state and final_state may be the same buffer (the state is then
 * updated in place).  Pointers need only element alignment here (2 bytes
 * for bf16, 4 for float32), not the 16 bytes of ssd_fwd.  Arithmetic in fp32; the result equals ssd_fwd's up to
 * rounding ("When it breaks": the forms are not bit-identical).  Returns
 * after enqueueing one kernel; the linear form has no device-side waits, so
 * the return value is the whole status. */
SSD_API int ssd_scan(const ssd_dims *dims,
            const void *x, const float *dt, const float *A,
            const void *B, const void *C, const float *D,
            const float *init_state,
            void *y, float *final_state,
            void *stream);

/* One decode step: ssd_scan with dims->T == 1 and the state updated in place.
 *   x (b,1,H,P), dt (b,1,H), B and C (b,1,G,N) for the new token; A and D as
 *   in ssd_fwd; state (b,H,N,P) float32, read and overwritten with
 *   h_t = a_t (.) h_{t-1} + B_t x_t^T; y (b,1,H,P) written with
 *   C_t^T h_t + D x_t.
 * A model that ran ssd_fwd over a prompt continues from its final_state with
 * one call per generated token.  SSD_ERR_INVALID_ARG unless dims->T == 1
 * and state is non-NULL. */
SSD_API int ssd_decode_step(const ssd_dims *dims,
            const void *x, const float *dt, const float *A,
            const void *B, const void *C, const float *D,
            float *state, void *y,
            void *stream);

/* Backward pass: the gradients of
 *   L = sum y * dy + sum final_state * dfinal
 * for the map ssd_fwd computes (the chunked algorithm's training cost is
 * what Structured State Space Duality, "The chunked algorithm takes both",
 * weighs; the pages give no backward, so this is the chain rule of the
 * recurrence of "The recurrence as one matrix").  CUDA cores, fp32
 * arithmetic, two paths:
 *  - scalar A with P in {64, 128} and N in {64, 128, 256} (not P = 128 with
 *    N = 256): the chunked algorithm run backwards on Q-token chunks (Q = 64;
 *    32 at N = 256 and at P = N = 128, where the 64-token product kernel's
 *    shared memory would not fit) -- the state entering every chunk (the
 *    generic forward's chunk-state kernels), the adjoint at every chunk's
 *    end (a reverse scan over chunks), then per chunk and head the dense
 *    products of the quadratic form and the rank-N terms;
 *  - every other dims: a forward sweep stores the state at the start of
 *    every 8-token block, and a reverse sweep recomputes each block's states
 *    from it while it runs the adjoint recurrence
 *    g = C_t dy_t^T + a_{t+1} (.) g.
 *
 * Inputs (device memory, layouts of ssd_fwd): x, dt, A, B, C, D (or NULL),
 * init_state (or NULL) as given to the forward call; dy (b,T,H,P) io dtype;
 * dfinal (b,H,N,P) float32 or NULL (zero).  Outputs, all written (none
 * accumulated into):
 *   dx (b,T,H,P) io dtype      ddt (b,T,H) float32    dA like A, float32
 *   dB, dC (b,T,G,N) io dtype (summed over the heads of each group)
 *   dD (H) float32 or NULL (not computed; sum of dy . x per head)
 *   dinit (b,H,N,P) float32 or NULL (not computed)
 * dA and dD are sums over chunks (or token ranges) added with fp32 atomics,
 * so they may differ in the last bits from one call to the next; every other
 * output is reproducible.
 * dims->path must be SSD_PATH_AUTO (the chunked path where it applies, the
 * recurrence elsewhere) or SSD_PATH_GENERIC (the recurrence for every dims);
 * SSD_ERR_UNSUPPORTED otherwise.  The backward takes 4 <= P <= 128.  Every pointer 16-byte
 * aligned; workspace >= ssd_bwd_workspace_size bytes, 256-byte aligned
 * (chunked path, Q as above: two fp32 arrays of b*H*ceil(T/Q)*N*P floats --
 * the states and the adjoints -- plus 2*b*T*H*N floats of per-head dB and dC
 * and b*ceil(T/Q)*G*Q*Q floats of C B^T per chunk and group; the
 * other path: checkpoints b*H*ceil(N/(1024/P))*ceil(T/8)*4 KB plus fp32
 * per-token arrays of 3*b*T*H*N + b*T*H*P floats; each region rounded up to
 * 256 bytes).  Asynchronous on `stream`; on any
 * argument error nothing is enqueued.  b == 0 or T == 0: dA and dD are zero
 * and dinit is dfinal (or zero). */
SSD_API int ssd_bwd_workspace_size(const ssd_dims *dims, size_t *bytes);
SSD_API int ssd_bwd(const ssd_dims *dims,
            const void *x, const float *dt, const float *A,
            const void *B, const void *C, const float *D,
            const float *init_state, const void *dy, const float *dfinal,
            void *dx, float *ddt, float *dA, void *dB, void *dC,
            float *dD, float *dinit,
            void *workspace, size_t workspace_bytes, void *stream);

/* Allocation-free forward pass.  The paper has no counterpart to this entry
 * point; it exists for callers that may not allocate device memory
 * themselves: for example a plug-in inside a host application that owns the
 * whole device-memory budget through its own pool, or a latency-bound loop
 * in which cudaMalloc, which can synchronise the device, is not allowed.
 *
 * Same arguments and layouts as ssd_fwd, minus the workspace: it runs the
 * generic path with its scratch in one fixed array of
 * SSD_NOALLOC_SCRATCH_BYTES (64 MiB) compiled into the library.  Every GPU
 * that loads the library holds that array until the process exits.  A
 * problem whose scratch (256 + align256(4*b*H*nc) + 4*b*H*nc*N*P bytes,
 * nc = ceil(T/Q), align256 rounding up to a multiple of 256) does not fit
 * is rejected with SSD_ERR_SCRATCH_LIMIT before anything is enqueued.  The
 * function calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * The first call on each device looks up that device's address of the array
 * (with the device current); make that first call before any stream capture.
 * The address is cached with the context it belongs to and looked up again
 * when the current context differs (for example after cudaDeviceReset); a
 * call right after such a change does that lookup, so it too should come
 * before any stream capture.
 * All calls in the process share the one array and it keeps the previous
 * call's contents (the status word is cleared by each call), so calls whose
 * executions overlap on the GPU -- on different streams, or from different
 * host threads without ordering -- race on it and give wrong results.
 * The generic path has no device-side waits, so the return value (argument
 * and launch errors) is the whole status of a call. */
#define SSD_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
SSD_API int ssd_fwd_noalloc(const ssd_dims *dims,
            const void *x, const float *dt, const float *A,
            const void *B, const void *C, const float *D,
            const float *init_state,
            void *y, float *final_state,
            void *stream);

/* Measurement hook.  When both handles are non-NULL (cudaEvent_t values
 * created by the caller), every later ssd_fwd records `start_event` on its
 * stream right before it launches its dominant kernel and `stop_event` right
 * after, so the caller can time that kernel alone with cudaEventElapsedTime.
 * Pass NULLs to switch it off.  Process-wide.  Returns SSD_OK. */
SSD_API int ssd_debug_set_kernel_events(void *start_event, void *stop_event);

/* Number of kernels this process has launched through the library so far
 * (written to *count).  Host-side counter; returns SSD_OK. */
SSD_API int ssd_launch_count(uint64_t *count);

/* Text of the last CUDA runtime error a call of this library ran into (the
 * cause behind the most recent SSD_ERR_CUDA), or "no error".  Process-wide,
 * static storage, never NULL. */
SSD_API const char *ssd_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SSD_B300_H */
