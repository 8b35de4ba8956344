/*
 * ssd_scan.h -- C ABI of the GB300 (sm_103a) Mamba-2 SSD chunked-scan forward.
 *
 * The operation (one independent recurrence per batch row b and head h, with
 * B/C group g = h / (nheads / ngroups)):
 *
 *   dt_t = clamp(softplus(dt_raw[b,t,h] + dt_bias[h]))
 *   h_t  = exp(dt_t * A[h]) * h_{t-1} + dt_t * x[b,t,h,:] (outer) B[b,t,g,:]
 *   y_t  = h_t . C[b,t,g,:] + D[h] * x[b,t,h,:],   out = y_t * silu(z[b,t,h,:])
 *
 * The argument set (dt_bias, dt_limit, D, z with the "silu" activation,
 * initial_states, seq_idx, chunk_size, returned final states) is the one of
 * the mamba_split_conv1d_scan_combined / mamba_chunk_scan_combined calls in
 * the repro script of state-spaces/mamba issue #647.  The layout
 * [batch, seq, head, hidden] of x, z and out is the "mamba2_ssd" layout named
 * in the differences list of fla-org/flash-linear-attention PR #49, which
 * also states that B/C are shared by groups of heads.  Initial and final
 * states give chunked prefill as described in state-spaces/mamba PR #488.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, dense
 *    row-major (C-contiguous) in the layout given, 16-byte aligned (except
 *    in ssd_scan_fwd_host, whose tensors are in host memory).  The library
 *    keeps no pointer after the call returns.
 *  - "x dtype" is the dtype argument: SSD_DTYPE_F32 (float) or
 *    SSD_DTYPE_BF16 (__nv_bfloat16).  dt_bias, A, D, states are float.
 *  - Everything is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *    default stream); no call synchronises the host.  Inputs must stay valid
 *    and unmodified until the work completes on that stream.
 *  - Arguments are validated before anything is launched.  On error nothing
 *    is launched, a negative SSD_ERR_* code is returned and
 *    ssd_last_error() describes it (per host thread).
 *  - Sizes: headdim in {16, 32, 64, 128}; dstate a multiple of 16 in
 *    [16, 256]; chunk_size in {16, 32, 64, 128, 256}; nheads divisible by
 *    ngroups; batch >= 1; seqlen >= 1.
 */
#ifndef SSD_SCAN_H
#define SSD_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSD_ABI_VERSION 3

typedef enum { SSD_DTYPE_F32 = 0, SSD_DTYPE_BF16 = 1 } ssd_dtype_t;

enum {
    SSD_OK = 0,
    SSD_ERR_ARG = -1,          /* bad size, option or dtype                  */
    SSD_ERR_NULL = -2,         /* a required pointer is NULL                 */
    SSD_ERR_ALIGN = -3,        /* a pointer is not 16-byte aligned           */
    SSD_ERR_UNSUPPORTED = -4,  /* valid but outside the supported shapes     */
    SSD_ERR_WORKSPACE = -5,    /* caller workspace too small                 */
    SSD_ERR_CUDA = -6,         /* a CUDA runtime call or launch failed       */
    SSD_ERR_TIMEOUT = -7       /* a launch gave up a bounded wait (ssd_scan_status) */
};

/* Version of this ABI.  New behaviour goes into new symbols; an existing
 * signature is never changed in place (an in-place change of a native fwd
 * signature broke its callers in state-spaces/mamba PR #488).
 *   1  the calls below up to ssd_scan_fwd_host
 *   2  adds SSD_ERR_TIMEOUT, ssd_scan_status, ssd_scan_fwd_strided, the
 *      block calls ssd_causal_conv1d and ssd_group_rmsnorm,
 *      ssd_decode_step and the backward ssd_scan_bwd and ssd_scan_bwd_ex
 *      (with their workspace queries); every version-1 symbol is unchanged
 *   3  adds ssd_scan_workspace_bytes_min: bf16 shapes outside the fused
 *      kernel run the fp32 tensor-core stages on fp32 copies when the
 *      workspace holds them (ssd_scan_workspace_bytes counts the copies; a
 *      workspace of the version-2 size still works, on the stage kernels);
 *      every version-2 symbol is unchanged */
int ssd_abi_version(void);

/* Message for the last error returned on the calling host thread ("" if
 * none).  The string stays valid until the next call on that thread. */
const char *ssd_last_error(void);

/* Status of the work already launched on the current device.  The
 * tensor-core kernel bounds every internal wait (2 s; it should never need
 * more than microseconds).  A wait that gives up ends the launch early: its
 * `out` and `final_states` are then NOT valid although the launching call
 * returned SSD_OK, because the launching call does not synchronise.  The
 * kernel records that in a device-wide status word (sticky across launches
 * and streams until reset), which this call reads.
 *   reset   nonzero: clear the word after reading it
 *   stream  cudaStream_t; the call synchronises it first (so every launch
 *           enqueued on it before has finished) and copies 4 bytes to the
 *           host; it allocates nothing.
 * Returns SSD_OK (no launch gave up), SSD_ERR_TIMEOUT (ssd_last_error()
 * names the wait) or SSD_ERR_CUDA. */
int ssd_scan_status(int reset, void *stream);

/* Bytes of device workspace ssd_scan_fwd needs for these sizes: a control
 * block of (64 + batch*nheads) int32 (work counter, error word, hand-off
 * flags of the fused kernel), processed dt and per-chunk cumsum
 * [batch, nheads, nchunks, chunk_size] float each, per-chunk segment counts
 * [batch, nchunks, chunk_size] int32, and chunk states
 * [batch, nchunks, nheads, headdim, dstate] float (the fused kernel uses the
 * start of this region for its state hand-off slots).  Each piece starts on
 * a 256-byte boundary.  0 on bad sizes.
 *
 * For bf16 inputs with headdim 64, dstate 128, chunk_size 128 or 256 and an
 * even number of heads per group (nheads / ngroups), ssd_scan_fwd runs all
 * four stages in the fused tensor-core kernel of ssd_chunk_fused (which then
 * computes stage 1 itself and leaves the dt / cumsum / segment regions of
 * the workspace unused); otherwise the four stage kernels below.  The fused
 * kernel keeps each head pair's state on chip for a segment of consecutive
 * chunks and hands it on between segments; the segment length is chosen from
 * the shape (the longest that leaves every SM about twelve work items) unless
 * the environment variable SSD_FUSED_SEGMENT_CHUNKS gives one (a tuning /
 * test override; results agree to rounding for every length).
 *
 * fp32 inputs with headdim 64 or 128, dstate a multiple of 32 up to 256 and
 * chunk_size 128 or 256 run chunk_state / chunk_scan on the tensor cores
 * (3xTF32, 128-token stages; the workspace then also holds C B^T per
 * (batch, chunk, group) and B pre-split for the tensor cores).  bf16 inputs
 * of those shapes that the fused kernel does not take run the same way on
 * fp32 copies of x, B, C, z and out in the workspace (the values exactly,
 * out rounded to bf16 once); the size returned here includes the copies. */
size_t ssd_scan_workspace_bytes(int64_t batch, int64_t seqlen, int nheads,
                                int headdim, int dstate, int ngroups,
                                int chunk_size, ssd_dtype_t dtype);

/* The least workspace ssd_scan_fwd (and ssd_scan_fwd_strided) accepts for
 * these sizes: ssd_scan_workspace_bytes without the fp32 copies above.  With
 * a workspace too small for the copies, those bf16 shapes run the bf16 stage
 * kernels instead (slower; the result agrees to rounding).  0 on bad sizes.
 * ssd_scan_fwd_noalloc's static scratch is checked against this size.
 * (ABI version 3.) */
size_t ssd_scan_workspace_bytes_min(int64_t batch, int64_t seqlen, int nheads,
                                    int headdim, int dstate, int ngroups,
                                    int chunk_size, ssd_dtype_t dtype);

/*
 * Full SSD chunked-scan forward.
 *
 *   x              [batch, seqlen, nheads, headdim]   x dtype
 *   dt             [batch, seqlen, nheads]            x dtype (raw, before bias)
 *   dt_bias        [nheads] float, or NULL (= 0)
 *   dt_softplus    nonzero: dt = softplus(dt + dt_bias)
 *   dt_limit_lo/hi clamp of dt after softplus; (0, +inf) means no clamp
 *   A              [nheads] float (negative for a decaying state)
 *   B, C           [batch, seqlen, ngroups, dstate]   x dtype
 *   D              [nheads] float, or NULL (= 0)
 *   z              [batch, seqlen, nheads, headdim]   x dtype, or NULL (no gate)
 *   initial_states [batch, nheads, headdim, dstate] float, or NULL (= 0)
 *   seq_idx        [batch, seqlen] int32, or NULL.  The state is reset to
 *                  zero before token t whenever seq_idx[b,t] != seq_idx[b,t-1]
 *                  (packed documents); initial_states then only reach the
 *                  first document.
 *   chunk_size     chunk length of the chunked algorithm (the result does not
 *                  depend on it beyond rounding)
 *   out            [batch, seqlen, nheads, headdim]   x dtype (written)
 *   final_states   [batch, nheads, headdim, dstate] float, or NULL; the
 *                  state after the last token (written)
 *   workspace      device buffer of >= ssd_scan_workspace_bytes(...) bytes,
 *                  or NULL: the library then takes it from the stream-ordered
 *                  allocator (cudaMallocAsync / cudaFreeAsync on `stream`).
 *   stream         cudaStream_t
 * Returns SSD_OK or a negative SSD_ERR_* code.
 */
int ssd_scan_fwd(const void *x, const void *dt, const float *dt_bias,
                 int dt_softplus, float dt_limit_lo, float dt_limit_hi,
                 const float *A, const void *B, const void *C, const float *D,
                 const void *z, const float *initial_states,
                 const int32_t *seq_idx, int64_t batch, int64_t seqlen,
                 int nheads, int headdim, int dstate, int ngroups,
                 int chunk_size, ssd_dtype_t dtype, void *out,
                 float *final_states, void *workspace, size_t workspace_bytes,
                 void *stream);

/* Element strides of a [batch, seqlen, ...] input whose per-token part is
 * dense: `batch` elements between batch rows, `token` elements between
 * consecutive tokens.  The dense layout of ssd_scan_fwd is
 * {seqlen * row, row} with row = nheads * headdim (x, z), nheads (dt) or
 * ngroups * dstate (B, C). */
typedef struct {
    int64_t batch;
    int64_t token;
} ssd_stride_t;

/*
 * ssd_scan_fwd on strided views of x, dt, B, C and z, such as the slices of
 * the fused input projection `zxbcdt` (z, xBC, dt) and of the convolved xBC
 * (x, B, C) in the block around the scan (the repro script of
 * state-spaces/mamba issue #647 splits one projection into them).  Within a
 * token each input is dense as in ssd_scan_fwd ([nheads, headdim] for x and
 * z, [nheads] for dt, [ngroups, dstate] for B and C); between tokens and
 * batch rows it advances by the given strides (elements, >= 0 and at most
 * 2^40; z_stride is ignored when z is NULL).  out, final_states and the
 * [nheads] / state arguments are dense, every pointer 16-byte aligned, and
 * everything else is as in ssd_scan_fwd.  The tensor-core path takes strides
 * that are multiples of 8 elements for x, z, B, C and even for dt (TMA needs
 * 16-byte strides; dt is read in pairs of heads); other strides run the
 * four stage kernels.  Returns SSD_OK or a negative SSD_ERR_* code.
 */
int ssd_scan_fwd_strided(const void *x, ssd_stride_t x_stride, const void *dt,
                         ssd_stride_t dt_stride, const float *dt_bias,
                         int dt_softplus, float dt_limit_lo, float dt_limit_hi,
                         const float *A, const void *B, ssd_stride_t B_stride,
                         const void *C, ssd_stride_t C_stride, const float *D,
                         const void *z, ssd_stride_t z_stride,
                         const float *initial_states, const int32_t *seq_idx,
                         int64_t batch, int64_t seqlen, int nheads,
                         int headdim, int dstate, int ngroups, int chunk_size,
                         ssd_dtype_t dtype, void *out, float *final_states,
                         void *workspace, size_t workspace_bytes,
                         void *stream);

/* ---------------------------------------------------------------------------
 * The four stages of ssd_scan_fwd, exposed one by one (same conventions).
 * nchunks = ceil(seqlen / chunk_size).  Chunk-major intermediates:
 *   dt_out, dA_cumsum  [batch, nheads, nchunks, chunk_size] float
 *   chunk_seg          [batch, nchunks, chunk_size] int32: for each token,
 *                      the number of seq_idx changes (state resets) from the
 *                      chunk's first token up to and including it; 0 means
 *                      "same document as the token before the chunk".
 *   states             [batch, nchunks, nheads, headdim, dstate] float
 * Positions past seqlen in the last chunk hold dt = 0, the chunk's last
 * cumsum and last segment count.
 * ------------------------------------------------------------------------- */

/* Stage 1: dt preprocessing (bias, softplus, clamp) fused with the
 * inclusive per-chunk cumsum of dt*A.  chunk_seg may be NULL iff seq_idx is
 * NULL. */
int ssd_dt_cumsum(const void *dt, const float *dt_bias, int dt_softplus,
                  float dt_limit_lo, float dt_limit_hi, const float *A,
                  const int32_t *seq_idx, int64_t batch, int64_t seqlen,
                  int nheads, int chunk_size, ssd_dtype_t dtype,
                  float *dt_out, float *dA_cumsum, int32_t *chunk_seg,
                  void *stream);

/* Stage 2: chunk states, for each (b, chunk c, head h) (tensor cores for the
 * bf16 headdim-64 / dstate-128 shapes of ssd_chunk_fused, else CUDA cores):
 *   states[b,c,h,p,n] = sum_{j in c, same segment as the chunk's last token}
 *        exp(cs_last - cs_j) * dt_j * x[b,j,h,p] * B[b,j,g,n]
 * chunk_seg may be NULL (no resets). */
int ssd_chunk_state(const void *x, const void *B, const float *dt_out,
                    const float *dA_cumsum, const int32_t *chunk_seg,
                    int64_t batch, int64_t seqlen, int nheads, int headdim,
                    int dstate, int ngroups, int chunk_size, ssd_dtype_t dtype,
                    float *states, void *stream);

/* Stage 3: inter-chunk state passing, sequential over chunks, in place:
 * on entry states[b,c] holds chunk c's own state S_c; on return it holds the
 * state entering chunk c, H_{c-1}, with H_{-1} = initial_states (or 0) and
 *   H_c = [no reset in chunk c] * exp(cs_last(c)) * H_{c-1} + S_c.
 * final_states (may be NULL) receives H_{nchunks-1}. */
int ssd_state_passing(float *states, const float *dA_cumsum,
                      const int32_t *chunk_seg, const float *initial_states,
                      float *final_states, int64_t batch, int64_t seqlen,
                      int nheads, int headdim, int dstate, int chunk_size,
                      void *stream);

/* Stage 4: outputs (tensor cores, through the fused kernel reading
 * prev_states, for the shapes of ssd_chunk_fused; else CUDA cores).  For
 * token i of chunk c:
 *   y_i = sum_{j<=i in c, same segment} exp(cs_i - cs_j) (C_i . B_j) dt_j x_j
 *       + [no reset since the chunk start] exp(cs_i) * (H_{c-1} . C_i)
 *       + D x_i,            out_i = y_i * silu(z_i)  (z may be NULL)
 * prev_states is stage 3's output. */
int ssd_chunk_scan(const void *x, const void *B, const void *C,
                   const float *dt_out, const float *dA_cumsum,
                   const int32_t *chunk_seg, const float *prev_states,
                   const float *D, const void *z, int64_t batch,
                   int64_t seqlen, int nheads, int headdim, int dstate,
                   int ngroups, int chunk_size, ssd_dtype_t dtype, void *out,
                   void *stream);

/* Stages 2-4 fused into one tensor-core (tcgen05) kernel, for bf16 inputs
 * with headdim 64, dstate 128, chunk_size 128 or 256 and an even number of
 * heads per group (SSD_ERR_UNSUPPORTED otherwise; the kernel takes the heads
 * of a group in pairs that share the B / C tiles).  Inputs are stage 1's dt_out / dA_cumsum / chunk_seg plus x, B,
 * C, D, z, initial_states as in ssd_scan_fwd; writes out and (if not NULL)
 * final_states.  workspace (>= ssd_scan_workspace_bytes) is required: the
 * kernel hands each chunk's final state to the next chunk through it.  If a
 * bounded internal wait gives up (which it should never do), the int32 at
 * byte offset 4 of the workspace is nonzero after the kernel and
 * ssd_scan_status returns SSD_ERR_TIMEOUT; the outputs are then not valid. */
int ssd_chunk_fused(const void *x, const void *B, const void *C,
                    const float *dt_out, const float *dA_cumsum,
                    const int32_t *chunk_seg, const float *D, const void *z,
                    const float *initial_states, int64_t batch, int64_t seqlen,
                    int nheads, int headdim, int dstate, int ngroups,
                    int chunk_size, ssd_dtype_t dtype, void *out,
                    float *final_states, void *workspace,
                    size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Variant of ssd_scan_fwd that allocates nothing.  (The pages have no
 * counterpart of this call; it exists for callers of this library.)
 *
 * Some callers cannot allocate device memory at all: a host application
 * whose own allocator owns the whole device and forbids plug-in code from
 * calling cudaMalloc, or a latency-critical path on which an allocation call,
 * which can synchronise the device or fail under memory pressure, is not
 * acceptable.  For them this call keeps its scratch (processed dt, per-chunk
 * cumsum and reset counts, chunk states) in one static device array of
 * SSD_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU that
 * loads the library holds until the process exits.  It calls no cudaMalloc,
 * cudaFree or other allocating routine; the caller still passes all inputs
 * and outputs, with the arguments and meaning of ssd_scan_fwd.
 *
 *  - Sizes whose scratch (ssd_scan_workspace_bytes) exceeds
 *    SSD_NOALLOC_SCRATCH_BYTES are rejected with SSD_ERR_WORKSPACE before
 *    anything is launched; use ssd_scan_fwd with a workspace for those.
 *  - Every call looks up the array's device address (cudaGetSymbolAddress,
 *    with the calling device current; nothing is cached, so a reset or
 *    re-created context is safe).  The first call on a device may load the
 *    library's module there: make it before any stream capture.
 *  - Like ssd_scan_fwd the call does not synchronise; ssd_scan_status (which
 *    allocates nothing either) tells whether its launch gave up a bounded
 *    internal wait.
 *  - Every call on a device shares the one array, which keeps the last
 *    call's contents; no part of it needs to start at zero.  Calls whose
 *    work overlaps on the GPU (different streams, or other host threads)
 *    race on the array: order them on one stream or serialise them.
 * ------------------------------------------------------------------------- */
#define SSD_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

int ssd_scan_fwd_noalloc(const void *x, const void *dt, const float *dt_bias,
                         int dt_softplus, float dt_limit_lo, float dt_limit_hi,
                         const float *A, const void *B, const void *C,
                         const float *D, const void *z,
                         const float *initial_states, const int32_t *seq_idx,
                         int64_t batch, int64_t seqlen, int nheads, int headdim,
                         int dstate, int ngroups, int chunk_size,
                         ssd_dtype_t dtype, void *out, float *final_states,
                         void *stream);

/* ---------------------------------------------------------------------------
 * The forward with the tensors in HOST memory.  (The pages have no
 * counterpart of this call; it is the library's runtime for callers whose
 * data lives on the host.)  Arguments as in ssd_scan_fwd, except that x, dt,
 * dt_bias, A, B, C, D, z, initial_states, seq_idx are host pointers (read)
 * and out, final_states host pointers (written).  The batch is processed in
 * slices of rows_per_slice batch rows (<= 0: the library picks about an
 * eighth of the batch) through two device staging buffers carved from
 * `workspace` (device memory of >= ssd_scan_host_workspace_bytes(...) bytes,
 * 256-byte aligned): each slice is copied in, scanned by ssd_scan_fwd's
 * kernels and copied out on three internal streams ordered with events, so
 * that the copies of one slice overlap the scan and copies of its
 * neighbours.  The work starts after the caller's earlier work on `stream`,
 * and `stream` waits for the last copy out: to the caller the call behaves
 * like one operation on `stream` (synchronise it before reading out).  Host
 * memory should be page-locked (cudaHostAlloc / cudaHostRegister); pageable
 * memory works, but its copies do not overlap.  The host buffers and the
 * workspace must stay untouched until `stream` has passed the call.  Calls
 * on one device share the internal streams; their enqueueing is serialised
 * by a lock, so calls from several host threads are safe but do not
 * overlap each other.  Returns SSD_OK or a negative SSD_ERR_* code. */
size_t ssd_scan_host_workspace_bytes(int64_t batch, int64_t seqlen, int nheads,
                                     int headdim, int dstate, int ngroups,
                                     int chunk_size, ssd_dtype_t dtype,
                                     int64_t rows_per_slice);

int ssd_scan_fwd_host(const void *x, const void *dt, const float *dt_bias,
                      int dt_softplus, float dt_limit_lo, float dt_limit_hi,
                      const float *A, const void *B, const void *C,
                      const float *D, const void *z,
                      const float *initial_states, const int32_t *seq_idx,
                      int64_t batch, int64_t seqlen, int nheads, int headdim,
                      int dstate, int ngroups, int chunk_size,
                      ssd_dtype_t dtype, void *out, float *final_states,
                      int64_t rows_per_slice, void *workspace,
                      size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * The block around the scan.  The repro script of state-spaces/mamba issue
 * #647 calls mamba_split_conv1d_scan_combined: the input projection zxbcdt
 * is split into z | xBC | dt, xBC goes through a causal depthwise conv1d of
 * width 4 with bias and the "silu" activation and is split into x | B | C,
 * the scan runs, and its gated output (norm_before_gate=False: y * silu(z))
 * is normalised by an RMSNorm over groups of d_inner / ngroups channels
 * (rmsnorm_weight, rmsnorm_eps) before the output projection.  With these two
 * calls and ssd_scan_fwd_strided (which reads x, B, C, z, dt as strided
 * views), everything but the two projections runs in this library.
 * ------------------------------------------------------------------------- */

/* Causal depthwise conv1d over the token axis, one filter per channel:
 *   out[b,t,c] = act(bias[c] + sum_{k<width} weight[c*width + k] x[b, t-width+1+k, c])
 * with act = SiLU if silu != 0 (else identity).  Taps before the sequence
 * start are zero, and so are taps in another document when seq_idx
 * ([batch, seqlen] int32, or NULL) differs from token t's (each packed
 * document is convolved on its own).
 *   x        [batch, seqlen, channels], x dtype, channels dense per token;
 *            x_stride gives the batch / token strides in elements (e.g. the
 *            xBC slice of zxbcdt), multiples of 16 bytes, token >= channels
 *   weight   [channels, width] float;  bias [channels] float or NULL
 *   out      [batch, seqlen, channels] x dtype, dense (written; must not
 *            overlap x)
 * channels a multiple of 8; width 1..8; x, out, bias, seq_idx 16-byte
 * aligned.  Enqueued on `stream`; returns SSD_OK or a negative SSD_ERR_*. */
int ssd_causal_conv1d(const void *x, ssd_stride_t x_stride, const float *weight,
                      const float *bias, const int32_t *seq_idx, int64_t batch,
                      int64_t seqlen, int channels, int width, int silu,
                      ssd_dtype_t dtype, void *out, void *stream);

/* RMSNorm over groups of channels, in place:
 *   y[r, c] = y[r, c] * weight[c] / sqrt(mean_{c' in group(c)} y[r, c']^2 + eps)
 * for rows r < rows (batch * seqlen tokens), channels c < dim (d_inner =
 * nheads * headdim, head-major: channel h * headdim + p), groups of
 * group_size consecutive channels (d_inner / ngroups gives the block's
 * grouped norm; dim gives one norm over all channels).  Applied to
 * ssd_scan_fwd's out (already gated by silu(z)) this is the block's norm
 * with norm_before_gate=False.  y dense [rows, dim] x dtype, 16-byte
 * aligned; weight [dim] float; group_size a multiple of 8 dividing dim.
 * Sums of squares in fp32.  Returns SSD_OK or a negative SSD_ERR_*. */
int ssd_group_rmsnorm(void *y, const float *weight, float eps, int64_t rows,
                      int dim, int group_size, ssd_dtype_t dtype, void *stream);

/* ---------------------------------------------------------------------------
 * One decode step.  The initial / final states of ssd_scan_fwd are what let a
 * prefill be continued (chunked prefill, prefix caching, speculative
 * decoding: state-spaces/mamba PR #488); generating then advances the state
 * one token at a time.  For every batch row, the recurrence at one token:
 *   dt' = clamp(softplus(dt + dt_bias)) (options as in ssd_scan_fwd)
 *   state <- exp(dt' A[h]) state + dt' x[b,h,:] (outer) B[b,g,:]   (in place)
 *   out[b,h,:] = state C[b,g,:] + D[h] x[b,h,:],  times silu(z[b,h,:]) if z
 *   x, z, out  [batch, nheads, headdim]  x dtype (out written)
 *   dt         [batch, nheads]           x dtype
 *   B, C       [batch, ngroups, dstate]  x dtype
 *   state      [batch, nheads, headdim, dstate] float, 16-byte aligned; read
 *              and written (the final_states of a prefill can be passed as is)
 * dstate a multiple of 8 up to 256.  Equal, up to rounding, to ssd_scan_fwd
 * over that one token with initial_states = state and final_states written
 * back.  Enqueued on `stream`; returns SSD_OK or a negative SSD_ERR_*. */
int ssd_decode_step(const void *x, const void *dt, const float *dt_bias,
                    int dt_softplus, float dt_limit_lo, float dt_limit_hi,
                    const float *A, const void *B, const void *C, const float *D,
                    const void *z, float *state, int64_t batch, int nheads,
                    int headdim, int dstate, int ngroups, ssd_dtype_t dtype,
                    void *out, void *stream);

/* ---------------------------------------------------------------------------
 * Backward of ssd_scan_fwd: the gradients of sum(out * dout) with respect to
 * every input.  The flash-linear-attention PR #49 page (fla-org) asks that
 * the chunked kernels' backward be checked as well as their forward; this is
 * that backward for the SSD scan, fp32 only.
 *
 * Method: the adjoint of the recurrence is the recurrence run backwards in
 * time, so the heavy parts are three more chunked scans of the forward's own
 * stage kernels with the operands' roles swapped (dx: time-reversed scan of
 * dy with B and C exchanged; dB: time-reversed scan of C against dy and x;
 * dC: forward scan of B against x and dy, started from the transposed
 * initial states), plus the forward recomputed once for y before the gate.
 * The gradient of the decays a_t = dt_t A is a reverse cumulative sum over
 * the tokens; dt's gradient then goes back through clamp (the gradient
 * passes where lo <= dt' <= hi), softplus and bias.
 *
 * Inputs exactly as for ssd_scan_fwd (dense, fp32, 16-byte aligned; dt the
 * raw dt), plus dout [batch, seqlen, nheads, headdim] float.  Outputs, all
 * dense float, shaped like their inputs and written (not accumulated):
 *   dx, dz          [batch, seqlen, nheads, headdim]  (dz required iff z)
 *   ddt             [batch, seqlen, nheads]   gradient w.r.t. the raw dt
 *   dB, dC          [batch, seqlen, ngroups, dstate]
 *   dA, d_dt_bias, dD  [nheads]   (d_dt_bias, dD may be NULL)
 *   d_initial_states  [batch, nheads, headdim, dstate]  (may be NULL)
 * d_dt_bias is the gradient of the bias whether or not dt_bias was given.
 * headdim and dstate in {16, 32, 64, 128}; chunk_size as for ssd_scan_fwd;
 * ngroups at most 8192.
 * Workspace: device memory of at least ssd_scan_bwd_workspace_bytes (0 for
 * unsupported sizes), used only during the call's stream work.  Enqueued on
 * `stream`; returns SSD_OK or a negative SSD_ERR_* (nothing launched on an
 * argument error). */
size_t ssd_scan_bwd_workspace_bytes(int64_t batch, int64_t seqlen, int nheads,
                                    int headdim, int dstate, int ngroups,
                                    int chunk_size);
int ssd_scan_bwd(const float *x, const float *dt, const float *dt_bias,
                 int dt_softplus, float dt_limit_lo, float dt_limit_hi,
                 const float *A, const float *B, const float *C, const float *D,
                 const float *z, const float *initial_states,
                 const int32_t *seq_idx, const float *dout, int64_t batch,
                 int64_t seqlen, int nheads, int headdim, int dstate,
                 int ngroups, int chunk_size, float *dx, float *ddt,
                 float *d_dt_bias, float *dA, float *dB, float *dC, float *dD,
                 float *dz, float *d_initial_states, void *workspace,
                 size_t workspace_bytes, void *stream);

/* The backward with its element-wise tensors in a given dtype.  dtype
 * SSD_DTYPE_F32 is ssd_scan_bwd.  SSD_DTYPE_BF16: x, dt, B, C, z and dout are
 * bf16 (the inputs and upstream gradient of a bf16 forward, e.g. a bf16
 * training step), and so are the gradients dx, ddt, dB, dC and dz written;
 * A, dt_bias, D, initial_states and their gradients stay float.  The bf16
 * values are converted to fp32 in the workspace, the fp32 backward runs on
 * them, and the fp32 gradients are rounded to bf16 at the end.  Workspace:
 * ssd_scan_bwd_ex_workspace_bytes (0 for unsupported sizes or dtypes).
 * Sizes, layouts, alignment and errors otherwise as for ssd_scan_bwd. */
size_t ssd_scan_bwd_ex_workspace_bytes(int64_t batch, int64_t seqlen,
                                       int nheads, int headdim, int dstate,
                                       int ngroups, int chunk_size,
                                       ssd_dtype_t dtype);
int ssd_scan_bwd_ex(const void *x, const void *dt, const float *dt_bias,
                    int dt_softplus, float dt_limit_lo, float dt_limit_hi,
                    const float *A, const void *B, const void *C,
                    const float *D, const void *z, const float *initial_states,
                    const int32_t *seq_idx, const void *dout, int64_t batch,
                    int64_t seqlen, int nheads, int headdim, int dstate,
                    int ngroups, int chunk_size, ssd_dtype_t dtype, void *dx,
                    void *ddt, float *d_dt_bias, float *dA, void *dB, void *dC,
                    float *dD, void *dz, float *d_initial_states,
                    void *workspace, size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SSD_SCAN_H */
