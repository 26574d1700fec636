/*
 * ssd.h -- C ABI of libssd, a single-GPU (B300, sm_103a) implementation of the
 * Mamba-2 state-space-duality (SSD) layer's forward scan, and its backward.
 *
 * The layer ("Mamba 模型" §4.1-4.2; "草稿:Mamba2", state space duality) maps
 * per-token inputs x, step sizes dt and projections B, C to outputs y through
 * the selective SSM recurrence, one independent recurrence per
 * (batch, head, headdim row):
 *
 *     h_t = exp(dt_t * A_h) * h_{t-1} + dt_t * x_t (outer) B_t      h in R^{P x N}
 *     y_t = C_t . h_t + D_h * x_t
 *
 * with a scalar A_h and D_h per head, B and C shared by the heads of one group
 * (head h uses group h / (nheads/ngroups)), headdim P and state size N.  The
 * library evaluates it the way the SSD papers describe: the causal
 * semiseparable matrix is split into diagonal blocks of `chunk` tokens,
 * computed as small masked matrix products inside each chunk, and off-diagonal
 * blocks carried by the per-chunk hidden state ("Mamba 模型" §4.1, block
 * decomposition; "Mamba-2架构深度解析" §2.2, the chunked hybrid mode).
 *
 * Conventions shared by every entry point:
 *   - All tensors are dense, row-major, with the layouts given below.
 *   - x, B, C and y have element type `dtype` (fp32 or bf16).  dt, A, D and the
 *     states are always fp32.  y is rounded to nearest-even in bf16 mode.
 *   - Pointers passed to ssd_fwd / ssd_fwd_ws are DEVICE pointers on the
 *     current CUDA device, owned by the caller; the library keeps none of them
 *     after the enqueued work completes.  bf16 tensors must be 16-byte aligned,
 *     fp32 tensors 4-byte aligned.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*, NULL = the
 *     legacy default stream) and the call returns without synchronising.
 *   - Invalid arguments are reported before anything is enqueued.
 *   - y must not overlap any input.  init_state == final_state (an in-place
 *     state carry) is allowed; any other overlap is undefined.
 *   - The library holds no global mutable host state apart from a
 *     thread-local error message, and may be called from several threads.
 */
#ifndef SSD_H
#define SSD_H

#include <stddef.h>

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
    SSD_ERR_INVALID_ARG = 1,  /* NULL required pointer, dimension <= 0, nheads % ngroups != 0,
                                 misaligned pointer, workspace too small, unknown dtype */
    SSD_ERR_UNSUPPORTED = 2,  /* valid but outside what this build handles (see ssd_fwd) */
    SSD_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
    SSD_ERR_NO_MEMORY = 4,    /* device or host allocation failed */
    SSD_ERR_TIMEOUT = 5       /* a bounded device-side wait gave up (ssd_check_device_status) */
} ssd_status_t;

typedef enum {
    SSD_DTYPE_F32 = 0,  /* x, B, C, y in fp32: computed with fp32 FMA (no tensor cores) */
    SSD_DTYPE_BF16 = 1  /* x, B, C, y in bf16: tensor-core contractions, fp32 accumulation */
} ssd_dtype_t;

/* Which kernel family ssd_fwd runs for a problem (see ssd_fwd_path). */
typedef enum {
    SSD_PATH_NONE = -1,     /* the problem is rejected */
    SSD_PATH_SIMT = 0,           /* fp32 FMA chunked kernels (any dtype) */
    SSD_PATH_TCGEN05 = 1,        /* bf16 chunked kernels on tcgen05 tensor cores, TMEM accumulators:
                                    chunk states, state passing, outputs */
    SSD_PATH_TCGEN05_FUSED = 2   /* one bf16 tcgen05 kernel; chunk-to-chunk states resolved by a
                                    decoupled look-back (headdim 64/128, dstate 64/128, blocks of at
                                    most 128 tokens) */
} ssd_path_t;

/*
 * ssd_fwd -- the SSD layer forward scan over a whole batch of sequences.
 *
 *   x           [batch][seqlen][nheads][headdim]  dtype     input
 *   dt          [batch][seqlen][nheads]           fp32      step sizes, taken as given
 *                                                           (no softplus, bias or clamp)
 *   A           [nheads]                          fp32      decay rate per head (normally < 0)
 *   B, C        [batch][seqlen][ngroups][dstate]  dtype     input / output projections
 *   D           [nheads]                          fp32      skip weight; NULL means 0
 *   init_state  [batch][nheads][headdim][dstate]  fp32      state before token 0; NULL means 0
 *   y           [batch][seqlen][nheads][headdim]  dtype     OUT
 *   final_state [batch][nheads][headdim][dstate]  fp32      OUT state after the last token;
 *                                                           NULL skips it
 *   chunk       block length Q of the decomposition, 1..256 (the result does
 *               not depend on it beyond rounding); seqlen need not be a
 *               multiple of it.  Where a fused kernel covers the sizes, a
 *               chunk longer than 128 is evaluated as equal blocks of at most
 *               128 tokens (ssd_fwd_block tells the length used).
 *
 * A device workspace of ssd_fwd_workspace_size() bytes is taken from the
 * stream-ordered allocator (cudaMallocAsync / cudaFreeAsync on `stream`).
 *
 * Returns SSD_OK once the work is enqueued; SSD_ERR_INVALID_ARG as described
 * above; SSD_ERR_UNSUPPORTED for chunk > 256, headdim > 256 or dstate > 256;
 * SSD_ERR_NO_MEMORY if the workspace cannot be allocated; SSD_ERR_CUDA if a
 * launch fails.  Errors raised while the kernels run are reported by
 * ssd_check_device_status().
 */
SSD_API ssd_status_t ssd_fwd(const void *x, const float *dt, const float *A, const void *B, const void *C,
                     const float *D, const float *init_state, void *y, float *final_state,
                     int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                     int chunk, ssd_dtype_t dtype, void *stream);

/*
 * ssd_fwd_workspace_size -- bytes of device workspace ssd_fwd_ws needs for
 * this problem: the per-chunk hidden states of the block decomposition
 * ("Mamba 模型" §4.1, off-diagonal blocks through the hidden state),
 * [batch][nheads][nchunks][headdim][dstate] fp32, plus one fp32 chunk decay
 * per (batch, head, chunk).  Writes the size to *bytes.  Same argument checks
 * as ssd_fwd (no pointers involved).
 */
SSD_API ssd_status_t ssd_fwd_workspace_size(int batch, int seqlen, int nheads, int headdim, int ngroups,
                                    int dstate, int chunk, ssd_dtype_t dtype, size_t *bytes);

/*
 * ssd_fwd_ws -- ssd_fwd with a caller-provided device workspace of at least
 * ssd_fwd_workspace_size() bytes, 256-byte aligned.  Nothing is allocated.
 * The workspace must not be used by anything else until the enqueued work has
 * completed.  SSD_ERR_INVALID_ARG if it is NULL, misaligned or too small.
 */
SSD_API ssd_status_t ssd_fwd_ws(const void *x, const float *dt, const float *A, const void *B, const void *C,
                        const float *D, const float *init_state, void *y, float *final_state,
                        int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                        int chunk, ssd_dtype_t dtype, void *workspace, size_t workspace_bytes,
                        void *stream);

/*
 * ssd_fwd_host -- ssd_fwd on HOST buffers (same layouts and meanings).  The
 * call copies the inputs to the current device, runs the scan on `stream`,
 * copies y (and final_state when non-NULL) back and synchronises the stream
 * before returning.  The work is cut into up to eight parts -- groups of batch
 * elements, or whole-chunk token ranges of each sequence with the state carried
 * from one range to the next -- so that uploads (on a library-owned stream),
 * the scan (on `stream`) and downloads (on a second library-owned stream)
 * overlap.  Device buffers come from a library-owned stream-ordered memory
 * pool (one per device) and go back to it before return; the pool keeps that
 * memory for later calls (about twice the call's input size, the largest call
 * so far) until the process exits, so a loop of calls does not map device
 * memory again each time.  Pinned host memory gives the fastest copies and the
 * overlap; pageable memory works.  Calls on one device are serialised (they
 * share the copy streams).  Same error codes as ssd_fwd; a device-side error is
 * returned directly.
 */
SSD_API ssd_status_t ssd_fwd_host(const void *x, const float *dt, const float *A, const void *B, const void *C,
                          const float *D, const float *init_state, void *y, float *final_state,
                          int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                          int chunk, ssd_dtype_t dtype, void *stream);

/*
 * ssd_fwd_noalloc -- ssd_fwd for callers that may not allocate device memory.
 * This entry point has no counterpart in the SSD papers; it exists for
 * deployment: processes that hand all device memory to a framework-owned pool,
 * plugins hosted by such runtimes, and latency-critical loops that cannot
 * afford an allocator call, which can synchronise the device or fail under
 * memory pressure.
 *
 * Same arguments, layouts and asynchronous behaviour as ssd_fwd.  Instead of a
 * workspace it uses a fixed 32 MiB scratch array compiled into the library,
 * which every device that loads the library holds until the process exits; it
 * calls no allocator at all.  It runs the fused bf16 kernel only (bf16,
 * headdim 64 or 128, dstate 64 or 128; a chunk longer than 128 as equal blocks
 * of at most 128 tokens, which changes the results only in rounding) and returns
 * SSD_ERR_UNSUPPORTED, with the needed and available sizes in
 * ssd_last_error_detail(), for anything else or for a problem whose scratch
 * (ssd_fwd_workspace_size) exceeds 32 MiB.  At dstate 64 the scratch is one
 * state slot per CTA, at most 16 MiB, so every size fits (the 2.7B-shaped
 * layer, batch 2 x 2048 tokens, uses 16 MiB); at dstate 128 it is 128 KiB per
 * (chunk, head block) unit, so at most 255 units fit (the grouped layer of
 * 16 x 4096 tokens, 32 heads x 128, needs 2 GiB and is rejected).
 *
 * The first call on a device looks up the scratch array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any stream
 * capture.  All calls on a device share the one array, and each call clears
 * the parts that must start at zero: calls whose work overlaps on the GPU
 * (different streams, or another thread) race and corrupt each other's
 * results.  Serialise them.
 */
SSD_API ssd_status_t ssd_fwd_noalloc(const void *x, const float *dt, const float *A, const void *B, const void *C,
                                     const float *D, const float *init_state, void *y, float *final_state,
                                     int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                                     int chunk, ssd_dtype_t dtype, void *stream);

/*
 * ssd_fwd_varlen -- ssd_fwd over packed variable-length sequences ("dynamic
 * sequence packing", "Mamba-2架构深度解析" §5): nseq sequences stored back to
 * back along one token dimension, each its own recurrence.  Sequence s owns the
 * packed tokens cu_seqlens[s] .. cu_seqlens[s+1]-1; its state starts from
 * init_state[s] (or zero) at its first token and ends in final_state[s]:
 *
 *     x, y        [total][nheads][headdim]   dtype, total = cu_seqlens[nseq]
 *     dt          [total][nheads]            fp32
 *     B, C        [total][ngroups][dstate]   dtype
 *     init_state, final_state  [nseq][nheads][headdim][dstate] fp32, each may be NULL
 *     cu_seqlens  HOST int32 [nseq + 1]: cu_seqlens[0] = 0, nondecreasing;
 *                 read during the call only (the library builds its chunk table from it)
 *
 * A, D, chunk, dtype, stream, the alignment rules and the asynchrony are those
 * of ssd_fwd; the workspace (the per-chunk states plus the chunk table) comes
 * from the stream-ordered allocator.  Empty sequences are allowed: their
 * final state is their initial state (or zero).  Chunks never straddle two
 * sequences: each sequence is cut into chunks from its own first token, the
 * last one partial.  Every kernel family takes packed sequences: the fused
 * kernels where ssd_fwd would run them (their units walk a chunk table), the
 * multi-kernel tcgen05 and fp32 paths otherwise (one CTA per chunk-table entry,
 * the state passing restarted at each sequence).  SSD_ERR_UNSUPPORTED for the
 * sizes ssd_fwd rejects, or for more than INT32_MAX packed tokens or chunks.
 * SSD_ERR_INVALID_ARG for a NULL cu_seqlens, nseq <= 0, offsets that do not
 * start at 0 or decrease, and the checks of ssd_fwd.
 */
SSD_API ssd_status_t ssd_fwd_varlen(const void *x, const float *dt, const float *A, const void *B, const void *C,
                                    const float *D, const int *cu_seqlens, int nseq, const float *init_state,
                                    void *y, float *final_state, int nheads, int headdim, int ngroups, int dstate,
                                    int chunk, ssd_dtype_t dtype, void *stream);

/* Pre-step flags of ssd_fwd_pre. */
enum { SSD_PRE_SOFTPLUS = 1, SSD_PRE_ZOH = 2 };

/*
 * ssd_fwd_pre -- ssd_fwd with the per-(token, head) pre-step of its scalar
 * inputs applied on the device first.  The discretisation of the pages
 * ("Mamba模型：线性复杂度序列建模的革命性突破" §2.2, "Mamba 模型" §2.3.1: zero-order
 * hold, Abar = exp(dt A), Bbar = (dt A)^-1 (exp(dt A) - 1) dt B; §3.2 of the
 * first page: dt comes out of a softplus) gives, for a scalar A per head:
 *
 *     dt_eff[b][t][h] = softplus(dt + dt_bias[h])   if pre_flags & SSD_PRE_SOFTPLUS
 *                       dt + dt_bias[h]              otherwise (dt_bias NULL => 0)
 *     decay           = exp(dt_eff A[h])
 *     input scale     = expm1(dt_eff A[h]) / A[h]    if pre_flags & SSD_PRE_ZOH (dt_eff when A[h] = 0)
 *                       dt_eff                       otherwise (the SSD layer's dt B)
 *
 *     h_t = decay_t h_{t-1} + scale_t x_t B_t,   y_t = C_t . h_t + D x_t
 *
 * With dt_bias NULL and pre_flags 0 it is ssd_fwd.  dt_bias is [nheads] fp32
 * device memory or NULL; every other argument, layout, ownership rule and error
 * is that of ssd_fwd (the workspace, which also holds dt_eff and the scale,
 * comes from the stream-ordered allocator).  SSD_ERR_INVALID_ARG also for
 * unknown pre_flags bits or a misaligned dt_bias.
 */
SSD_API ssd_status_t ssd_fwd_pre(const void *x, const float *dt, const float *dt_bias, int pre_flags, const float *A,
                                 const void *B, const void *C, const float *D, const float *init_state, void *y,
                                 float *final_state, int batch, int seqlen, int nheads, int headdim, int ngroups,
                                 int dstate, int chunk, ssd_dtype_t dtype, void *stream);

/*
 * ssd_step -- one recurrent step of the layer, the constant-size-state
 * inference form ("深挖-Mamba", Mamba-vs-Transformer comparison table: no KV
 * cache, only the fixed-size hidden state h_t; section "Mamba-2 (2024)":
 * matrix form for training, recurrent form for inference).  For one new token
 * per sequence, for every (b, h, p) with g = h / (nheads / ngroups):
 *
 *     a        = exp(dt[b][h] * A[h])
 *     s[n]     = a * s[n] + dt[b][h] * x[b][h][p] * B[b][g][n]   (state, in place)
 *     y[b][h][p] = sum_n C[b][g][n] * s[n] + D[h] * x[b][h][p]
 *
 * i.e. exactly ssd_fwd for seqlen 1 with init_state = final_state = state, so
 * a chain of steps continues a prefix run by ssd_fwd (its final_state) token by
 * token.  Device pointers:
 *   x      [batch][nheads][headdim]            dtype
 *   dt     [batch][nheads] fp32;  A, D [nheads] fp32 (D may be NULL: no skip)
 *   B, C   [batch][ngroups][dstate]            dtype
 *   state  [batch][nheads][headdim][dstate] fp32, read and overwritten
 *   y      out [batch][nheads][headdim]        dtype (bf16: round to nearest even)
 * y must not overlap state or any input.  The caller owns every buffer; the
 * library keeps no pointer after the enqueued work completes.  Nothing is
 * allocated.  Returns SSD_OK once the kernel is enqueued on `stream`;
 * SSD_ERR_INVALID_ARG for a NULL required pointer, a dimension <= 0,
 * nheads % ngroups != 0, an unknown dtype or a misaligned pointer;
 * SSD_ERR_CUDA if the launch fails.
 */
SSD_API ssd_status_t ssd_step(const void *x, const float *dt, const float *A, const void *B, const void *C,
                              const float *D, float *state, void *y, int batch, int nheads, int headdim,
                              int ngroups, int dstate, ssd_dtype_t dtype, void *stream);

/*
 * ssd_bwd -- backward of ssd_fwd: the gradients of a scalar loss L with
 * respect to every input, given the loss's gradients dy = dL/dy and
 * dfinal_state = dL/d final_state.  By the chain rule through the recurrence
 * above, with lam_t = dL/dh_t (per (batch, head, headdim row), a vector over
 * dstate), lam_{L-1} = dy_{L-1} C_{L-1} + dfinal, lam_t = dy_t C_t + a_{t+1} lam_{t+1},
 * a_t = exp(dt_t A_h):
 *
 *     dx_t    = D_h dy_t + dt_t (B_t . lam_t)
 *     dB_t    = sum over the group's heads and rows of dt_t x_t lam_t
 *     dC_t    = sum over the group's heads and rows of dy_t h_t
 *     ddt_t   = sum over rows of x_t (B_t . lam_t) + A_h a_t (lam_t . h_{t-1})
 *     dA_h    = sum over batch, tokens and rows of dt_t a_t (lam_t . h_{t-1})
 *     dD_h    = sum of dy_t x_t;     dinit = a_0 lam_0
 *
 * The pages ask the backward to recompute the intermediate states rather than
 * store them ("Mamba 模型" §3.4, recomputation); this call keeps nothing from
 * the forward: it recomputes the per-chunk states from the inputs with the
 * same block decomposition ("Mamba 模型" §4.1; its own chunk length, 64 or
 * 128 tokens) and runs the adjoint state recurrence backwards over the chunks.
 *
 *   x, dt, A, B, C, D, init_state   the forward's inputs, as in ssd_fwd (D and
 *                                   init_state may be NULL, meaning 0)
 *   dy           [batch][seqlen][nheads][headdim]  dtype (the type of x)
 *   dfinal_state [batch][nheads][headdim][dstate]  fp32, NULL means 0
 *   dx           OUT [batch][seqlen][nheads][headdim]  fp32
 *   ddt          OUT [batch][seqlen][nheads]           fp32
 *   dA           OUT [nheads]                          fp32
 *   dB, dC       OUT [batch][seqlen][ngroups][dstate]  fp32
 *   dD           OUT [nheads] fp32, NULL skips it (written also when D is NULL)
 *   dinit_state  OUT [batch][nheads][headdim][dstate]  fp32, NULL skips it
 *
 * Every gradient is fp32 whatever dtype is.  For bf16 inputs with headdim 64
 * and dstate 64 (x, dy, B, C 16-byte aligned) the in-chunk products run on
 * tcgen05 tensor cores over 128-token chunks, every fp32 operand split into two
 * bf16 terms so that the products keep fp32-level accuracy; every other size
 * runs on fp32 FMA over 64-token chunks.  The sums over heads, chunks and batch
 * run in a fixed order, so two calls on the same inputs give identical bits.  A_h <= 0 is assumed (every exponent is
 * then <= 0).  Device pointers, alignment, ownership and asynchrony as for
 * ssd_fwd; outputs must not overlap inputs or each other.  A device workspace
 * of ssd_bwd_workspace_size() bytes is taken from the stream-ordered allocator.
 * Returns SSD_OK once the work is enqueued; SSD_ERR_INVALID_ARG for a NULL
 * required pointer, a dimension <= 0, nheads % ngroups != 0, an unknown dtype or
 * a misaligned pointer; SSD_ERR_UNSUPPORTED for headdim > 128 or dstate > 256;
 * SSD_ERR_NO_MEMORY / SSD_ERR_CUDA as for ssd_fwd.
 */
SSD_API ssd_status_t ssd_bwd(const void *x, const float *dt, const float *A, const void *B, const void *C,
                             const float *D, const float *init_state, const void *dy, const float *dfinal_state,
                             float *dx, float *ddt, float *dA, float *dB, float *dC, float *dD, float *dinit_state,
                             int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                             ssd_dtype_t dtype, void *stream);

/*
 * ssd_bwd_workspace_size -- bytes of device workspace one ssd_bwd takes for
 * these sizes: the recomputed chunk states and the adjoint chunk states
 * (2 x [batch][nheads][nchunks][headdim][dstate] fp32, 64-token chunks), chunk
 * decays, per-chunk parts of dA and dD, and, when a group has more than one
 * head, per-head parts of dB and dC (2 x [batch][seqlen][nheads][dstate] fp32).
 * Same argument checks as ssd_bwd (no pointers involved).
 */
SSD_API ssd_status_t ssd_bwd_workspace_size(int batch, int seqlen, int nheads, int headdim, int ngroups,
                                            int dstate, ssd_dtype_t dtype, size_t *bytes);

/*
 * ssd_bwd_kernels -- how many kernels one ssd_bwd launches for these sizes,
 * with their names written comma-separated into `names` as ssd_fwd_kernels
 * does; -1 when the sizes are rejected.  Pure host function.  ssd_profile_events
 * times ssd_bwd's kernels the same way as a forward's.
 */
SSD_API int ssd_bwd_kernels(int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                            ssd_dtype_t dtype, char *names, size_t names_len);

/*
 * ssd_fwd_path -- the kernel family ssd_fwd would run for these sizes
 * (SSD_PATH_NONE when they are rejected).  Pure host function: no CUDA call.
 */
SSD_API ssd_path_t ssd_fwd_path(int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                        int chunk, ssd_dtype_t dtype);

/*
 * ssd_fwd_block -- the chunk length ssd_fwd evaluates for these sizes, or -1
 * when they are rejected.  Pure host function: no CUDA call.  The block
 * decomposition ("Mamba 模型" §4.1) is exact for any chunk length: a requested
 * chunk longer than 128 tokens is evaluated as equal blocks of at most 128
 * (256 -> 128, 200 -> 100) whenever the sizes take a fused kernel (bf16,
 * headdim 64/128, dstate 64/128); the outputs then differ from the requested
 * length only in rounding.  Otherwise the requested chunk itself.  ssd_fwd,
 * ssd_fwd_varlen, ssd_fwd_host, ssd_fwd_pre and the workspace and kernel queries
 * all use this length.
 */
SSD_API int ssd_fwd_block(int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate, int chunk,
                          ssd_dtype_t dtype);

/*
 * ssd_fwd_kernels -- how many kernels one ssd_fwd launches for these sizes,
 * with their names written comma-separated into `names` (when non-NULL,
 * truncated to names_len bytes including the terminator).  Returns -1 when the
 * sizes are rejected.  Pure host function: no CUDA call.
 */
SSD_API int ssd_fwd_kernels(int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                            int chunk, ssd_dtype_t dtype, char *names, size_t names_len);

/*
 * ssd_profile_events -- per-kernel timing hook for benchmarks.  After a call
 * with non-NULL `events` (cudaEvent_t handles passed as void*, owned by the
 * caller, created on the device the forwards run on), every forward issued from
 * this thread records, for its k-th kernel (k = 0, 1, ...), events[2k] on its
 * stream right before the launch -- after the library's host-side set-up for
 * that kernel and any memset it needs -- and events[2k+1] right after it,
 * while 2k+1 < count.  The time between the two is the kernel's own device
 * time.  NULL or count <= 0 switches the hook off; count is at most 16.  The
 * setting is thread-local; the library never creates, destroys or waits on
 * these events.
 */
SSD_API ssd_status_t ssd_profile_events(void *const *events, int count);

/*
 * ssd_test_set_fault -- failure-detection test hook; not for production use.
 * The fused kernels resolve the chunk-to-chunk recurrence by waiting, inside
 * the kernel, for other units' published chunk states ("Mamba 模型" §4.1: the
 * off-diagonal blocks pass through the hidden state).  Every such wait, and
 * every wait on the kernels' own barriers, is bounded; a wait that runs out
 * sets the device error word, the kernel gives up instead of hanging, and
 * ssd_check_device_status() returns SSD_ERR_TIMEOUT.  This hook makes that
 * path testable without any fault: for forwards issued later from the calling
 * thread, every bounded wait of the fused kernels gives up after
 * `wait_limit_ns` nanoseconds (0 restores the default, 2 s), and the unit
 * `withhold_unit` (its index among the fused kernels' units, -1 for none;
 * unit 0 is chunk 0 of the first head block of batch element 0) never
 * publishes its chunk state, so the units after it in its sequence wait for a
 * flag that nothing sets.  The outputs of such a forward are undefined; the
 * kernel still ends and the context stays usable.  Thread-local setting;
 * SSD_ERR_INVALID_ARG for withhold_unit < -1.
 */
SSD_API ssd_status_t ssd_test_set_fault(unsigned long long wait_limit_ns, long long withhold_unit);

/*
 * ssd_check_device_status -- synchronise `stream`, then read and clear the
 * library's device error word on the current device.  Returns SSD_OK,
 * SSD_ERR_TIMEOUT (a bounded wait inside a kernel gave up), SSD_ERR_INVALID_ARG
 * (a kernel-side bounds check failed) or SSD_ERR_CUDA (the stream reported an
 * error).
 */
SSD_API ssd_status_t ssd_check_device_status(void *stream);

/* Static description of a status code. */
SSD_API const char *ssd_status_string(ssd_status_t status);

/* Thread-local detail of the last failing call on this thread ("" if none). */
SSD_API const char *ssd_last_error_detail(void);

/* Library version string. */
SSD_API const char *ssd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSD_H */
