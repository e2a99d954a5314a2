/*
 * ss_scan: selective scan (S6) forward pass and single-token state update for
 * NVIDIA B300 (sm_103a).
 *
 * C ABI. Plain pointers and sizes; no CUDA or framework types beyond the
 * opaque stream handle, which is a cudaStream_t (pass NULL for the legacy
 * default stream).
 *
 * The operation, by page title and section:
 *  - "Mamba: Linear-Time Sequence Modeling with Selective State Spaces",
 *    section "Method": zero-order-hold discretisation A_bar = exp(Delta A) and
 *    the linear recurrence h_t = A_bar h_{t-1} + B_bar x_t, y_t = C h_t.
 *  - same page, section "The Selection Mechanism (S6)": B_t, C_t (width N,
 *    shared over channels) and Delta_t = softplus(parameter + projection)
 *    depend on the input token.
 *  - soft186.com, "Mamba选择性状态空间机制", section "动态参数化的状态空间":
 *    dt = softplus(projection + delta_bias), dA = exp(dt * A), the state is
 *    multiplied by dA and receives the input times dt * B.
 *  - same Mamba page, sections "Hardware-aware state expansion" and
 *    "Questions": the expanded state (batch, L, dim, N) never goes to device
 *    memory; only the contracted output (batch, dim, L) is written; decoding
 *    keeps a fixed dim x N state per sequence and advances it one token at a
 *    time.
 *
 * Per row (b, d) and time step l the library computes
 *     dt  = softplus(delta[b,d,l] + delta_bias[d])    (or the sum itself)
 *     h_n = exp(dt * A[d,n]) * h_n + dt * B[b,n,l] * u[b,d,l]     n < N
 *     y   = (sum_n C[b,n,l] * h_n + D[d] * u[b,d,l]) * silu(z[b,d,l])
 * with the state h held in fp32 on chip and h_N after the last step
 * optionally written out.
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller, C-contiguous,
 *    16-byte aligned. The library never frees or retains them.
 *  - Calls are asynchronous and stream-ordered on the given stream; they do
 *    not synchronise. Argument errors are detected on the host before any
 *    launch and returned immediately (nothing is enqueued).
 *  - Errors found on the device (a bounded wait that ran out) are recorded in
 *    a per-context error word; read it with ss_get_device_error.
 *  - A context must not be used from two host threads at once. Two streams
 *    may share a context only for ss_state_update calls; a chunked
 *    ss_scan_fwd uses context scratch, so give each concurrent stream its own
 *    context.
 */
#ifndef SS_SCAN_H
#define SS_SCAN_H

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *ss_stream_t; /* == cudaStream_t */

typedef enum { SS_F32 = 0, SS_BF16 = 1 } ss_dtype;

typedef enum {
    SS_OK = 0,
    SS_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or aliasing */
    SS_ERR_UNSUPPORTED = 2,  /* valid but not built (e.g. dstate not in {1,2,4,8,16}) */
    SS_ERR_CUDA = 3,         /* a CUDA runtime call failed */
    SS_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up */
    SS_ERR_DEVICE = 5        /* other device-detected error */
} ss_status;

typedef struct ss_ctx ss_ctx;

/*
 * Create a context bound to CUDA device `device`. It queries the device
 * (SM count, shared memory) and owns a small device buffer holding the error
 * word; chunk-carry scratch is allocated on first need and kept.
 * *out receives the context. Returns SS_OK, SS_ERR_INVALID_ARG (out NULL) or
 * SS_ERR_CUDA.
 */
int ss_create(ss_ctx **out, int device);

/* Free a context and its scratch. NULL is accepted. Synchronises the device. */
int ss_destroy(ss_ctx *ctx);

/*
 * Selective scan forward.
 *   batch, dim, dstate, seqlen : Bt, D (= d_inner), N, L. dim >= 1, batch >= 1,
 *                                dstate in {1,2,4,8,16}, seqlen >= 0.
 *   in_dtype   : dtype of u, delta, z, B, C (SS_F32 or SS_BF16).
 *   out_dtype  : dtype of y (SS_F32 or SS_BF16; bf16 rounds to nearest even).
 *   u, delta, z: (batch, dim, seqlen). z may be NULL: no gate.
 *   A          : (dim, dstate) fp32, real; entries are expected to be negative
 *                (not checked).
 *   B, C       : (batch, dstate, seqlen), input-dependent, shared by all d.
 *   D, delta_bias : (dim) fp32; either may be NULL (treated as zero).
 *   delta_softplus: nonzero -> dt = softplus(delta + bias); zero -> the sum.
 *   h0         : (batch, dim, dstate) fp32 initial state, or NULL for zero.
 *   y          : (batch, dim, seqlen) output. Must not overlap any input.
 *   h_last     : (batch, dim, dstate) fp32 final state, or NULL. May equal h0
 *                (read before written, per row).
 * Returns SS_OK or an error from ss_status. seqlen == 0 writes h_last = h0
 * (or zeros) and nothing else.
 */
typedef struct {
    int batch, dim, dstate;
    long long seqlen;
    int in_dtype, out_dtype;
    const void *u, *delta, *z;
    const float *A;
    const void *B, *C;
    const float *D, *delta_bias;
    int delta_softplus;
    const float *h0;
    void *y;
    float *h_last;
} ss_scan_args;

int ss_scan_fwd(ss_ctx *ctx, const ss_scan_args *args, ss_stream_t stream);

/*
 * Single-token selective state update (decoding).
 *   state  : (batch, dim, dstate) fp32, read and overwritten in place with the
 *            state after this token.
 *   x, dt, z : (batch, dim) in in_dtype; z may be NULL.
 *   A      : (dim, dstate) fp32;  B, C : (batch, dstate) in in_dtype.
 *   D, dt_bias : (dim) fp32 or NULL.  dt_softplus as delta_softplus above.
 *   y      : (batch, dim) in out_dtype; must not overlap the inputs or state.
 * The arithmetic is that of ss_scan_fwd with seqlen = 1 and h0 = h_last = state.
 */
typedef struct {
    int batch, dim, dstate;
    int in_dtype, out_dtype;
    float *state;
    const void *x, *dt, *z;
    const float *A;
    const void *B, *C;
    const float *D, *dt_bias;
    int dt_softplus;
    void *y;
} ss_update_args;

int ss_state_update(ss_ctx *ctx, const ss_update_args *args, ss_stream_t stream);

/*
 * Backward pass of the selective scan: the gradients of a loss with respect to
 * every input of ss_scan_fwd, given dy = dL/dy and optionally dh_last =
 * dL/dh_L. The forward states are recomputed, not stored ("Mamba: Linear-Time
 * Sequence Modeling with Selective State Spaces", section "Hardware-aware
 * state expansion": recomputation in the backward pass); the context keeps a
 * checkpoint of every row's state every 16 steps (batch * ceil(dim/32) * 32 *
 * seqlen/16 * dstate floats of scratch, allocated on first need).
 *   Inputs as for ss_scan_fwd (same shapes, in_dtype for u, delta, z, B, C).
 *   dy     : (batch, dim, seqlen) fp32.   dh_last: (batch, dim, dstate) fp32 or NULL.
 *   Outputs, fp32, overwritten:
 *     du, ddelta : (batch, dim, seqlen);  dz: same, or NULL (skipped; must be
 *                  NULL when z is NULL)
 *     dA         : (dim, dstate);  dB, dC: (batch, dstate, seqlen)
 *     dD, ddelta_bias : (dim) or NULL;  dh0: (batch, dim, dstate) or NULL
 *   The context's SS_OPT_DISCRETIZATION applies: with SS_DISC_ZOH the
 *   gradients are those of the exact zero-order-hold scan (taken on the
 *   one-lane-per-state kernel, which is slower than the simplified form's).
 *   seqlen must be a multiple of 16, else SS_ERR_UNSUPPORTED. Outputs must not
 *   overlap inputs or each other.
 *   dB and dC are sums over channels accumulated with atomic adds, so their
 *   low bits may differ from run to run.
 */
typedef struct {
    int batch, dim, dstate;
    long long seqlen;
    int in_dtype;
    const void *u, *delta, *z;
    const float *A;
    const void *B, *C;
    const float *D, *delta_bias;
    int delta_softplus;
    const float *h0;
    const float *dy, *dh_last;
    float *du, *ddelta, *dz;
    float *dA, *dB, *dC;
    float *dD, *ddelta_bias;
    float *dh0;
} ss_scan_bwd_args;

int ss_scan_bwd(ss_ctx *ctx, const ss_scan_bwd_args *args, ss_stream_t stream);

/*
 * Mamba-2 state space duality (SSD) forward: the selective scan with a scalar
 * decay per head, computed chunk by chunk (64 steps) with matrix products on
 * the tensor cores (soft186.com, "Mamba选择性状态空间机制", section
 * "状态空间对偶性算法突破": Mamba-2 computes the scan through a block
 * decomposition of its semiseparable matrix). Per batch b, head h, channel p:
 *     dt   = softplus(dt_raw[b,l,h] + dt_bias[h])      (or the sum itself)
 *     H_pn = exp(dt A[h]) H_pn + dt x[b,l,h,p] B[b,l,n]
 *     y[b,l,h,p] = sum_n C[b,l,n] H_pn + D[h] x[b,l,h,p]
 * which is ss_scan_fwd with A constant over states and heads' channels, dt
 * shared by a head's channels, and B, C shared by all heads (one group).
 *   x, y   : (batch, seqlen, heads, headdim), x bf16, y fp32 or bf16.
 *   dt     : (batch, seqlen, heads) bf16.   A, D, dt_bias: (heads) fp32 (D,
 *            dt_bias may be NULL).   B, C: (batch, seqlen, dstate) bf16.
 *   h0, h_last: (batch, heads, headdim, dstate) fp32 or NULL (zero start / not
 *            written); h_last may equal h0.
 *   headdim must be 64, dstate 64 or 128, seqlen a multiple of 64 and the
 *   inputs bf16, else SS_ERR_UNSUPPORTED. The products run in bf16 with fp32
 *   accumulation (the state carried between chunks in fp32).
 */
typedef struct {
    int batch, heads, headdim, dstate;
    long long seqlen;
    int in_dtype, out_dtype;
    const void *x, *dt;
    const float *A;
    const void *B, *C;
    const float *D, *dt_bias;
    int dt_softplus;
    const float *h0;
    void *y;
    float *h_last;
} ss_ssd_args;

int ss_ssd_fwd(ss_ctx *ctx, const ss_ssd_args *args, ss_stream_t stream);

/*
 * Causal depthwise 1D convolution: the Mamba block's convolution in front of
 * the selective scan ("Mamba: Linear-Time Sequence Modeling with Selective
 * State Spaces", section "Key terms", the Mamba block; soft186.com,
 * "Mamba选择性状态空间机制", section "基础模型构建": width d_conv = 4 and the
 * causal-conv1d package). Per row (b, d), W = width:
 *     out[l] = bias[d] + sum_{k<W} weight[d,k] * xin(l - (W-1) + k)
 *     xin(j) = x[b,d,j] for j >= 0; init_state[b,d,(W-1)+j] for j < 0
 *              (zero when init_state is NULL)
 *     out[l] = silu(out[l])                  when silu != 0
 *     final_state[b,d,:] = xin(L-(W-1)) .. xin(L-1), the last W-1 inputs
 *   batch, dim >= 1; width in {2, 3, 4} (else SS_ERR_UNSUPPORTED); seqlen >= 0.
 *   x     : (batch, dim, seqlen) in in_dtype.   out : same shape, out_dtype;
 *           must not overlap x.
 *   weight: (dim, width) fp32.   bias: (dim) fp32 or NULL.
 *   init_state, final_state: (batch, dim, width-1) fp32, oldest input first,
 *           or NULL; final_state must not overlap init_state, x or out.
 *   Device pointers, 16-byte aligned, caller-owned. seqlen == 0 writes
 *   final_state = init_state (or zeros) and nothing else.
 */
typedef struct {
    int batch, dim, width;
    long long seqlen;
    int in_dtype, out_dtype;
    const void *x;
    const float *weight, *bias;
    const float *init_state;
    int silu;
    void *out;
    float *final_state;
} ss_conv1d_args;

int ss_conv1d_fwd(ss_ctx *ctx, const ss_conv1d_args *args, ss_stream_t stream);

/*
 * The Mamba block's convolution fused in front of the selective scan: the
 * convolution of ss_conv1d_fwd (its silu applied when conv_silu != 0) gives
 * u, and the scan of ss_scan_fwd runs on that u, in one pass over the inputs
 * ("Mamba: Linear-Time Sequence Modeling with Selective State Spaces",
 * section "Key terms": the block's 1D convolution feeds the selective SSM;
 * same page, section "Hardware-aware state expansion": inputs cross into
 * on-chip memory once). Per row (b, d), W = conv_width:
 *     c[l] = conv_bias[d] + sum_{k<W} conv_weight[d,k] * xin(l-(W-1)+k)
 *     xin(j) = x[b,d,j] for j >= 0; conv_init[b,d,(W-1)+j] for j < 0
 *              (zero when conv_init is NULL)
 *     u[l] = silu(c[l]) when conv_silu != 0, else c[l]
 *     y, h_last: ss_scan_fwd on (u, delta, z, A, B, C, D, delta_bias, h0)
 *   scan           : as for ss_scan_fwd, except that scan.u holds x, the
 *                    convolution's input (batch, dim, seqlen) in in_dtype.
 *                    u is kept in fp32 (never rounded to in_dtype) inside.
 *   conv_width     : 2, 3 or 4 (else SS_ERR_UNSUPPORTED).
 *   conv_weight    : (dim, conv_width) fp32.   conv_bias: (dim) fp32 or NULL.
 *   conv_init      : (batch, dim, conv_width-1) fp32, oldest input first, or NULL.
 *   u_out          : (batch, dim, seqlen) in in_dtype, 32-byte aligned, or
 *                    NULL: receives u rounded to in_dtype (for a backward).
 *   conv_state_out : (batch, dim, conv_width-1) fp32 or NULL: the last
 *                    conv_width-1 inputs, the convolution's decode state.
 * Outputs must not overlap inputs or each other (h_last == h0 is allowed).
 * Only the chained pair-row kernel carries the fusion: dstate 16, seqlen a
 * multiple of 16, u, delta, z, y 32-byte aligned, the simplified input
 * matrix, and variant AUTO, CHUNKED or ROWS with 0 or 2 threads per row;
 * anything else returns SS_ERR_UNSUPPORTED (compose ss_conv1d_fwd and
 * ss_scan_fwd there). seqlen == 0 writes h_last = h0 (or zeros) and
 * conv_state_out = conv_init (or zeros).
 */
typedef struct {
    ss_scan_args scan;
    int conv_width;
    const float *conv_weight, *conv_bias;
    const float *conv_init;
    int conv_silu;
    void *u_out;
    float *conv_state_out;
} ss_conv_scan_args;

int ss_conv_scan_fwd(ss_ctx *ctx, const ss_conv_scan_args *args, ss_stream_t stream);

/*
 * One decode step of the convolution, per row (b, d):
 *     out = bias[d] + sum_{k<W-1} weight[d,k] * state[b,d,k] + weight[d,W-1] * x[b,d]
 *     (then silu when silu != 0); state drops its oldest input and appends x.
 *   state : (batch, dim, width-1) fp32, oldest first, updated in place.
 *   x, out: (batch, dim) in in_dtype / out_dtype; out must not overlap the
 *           inputs or the state.
 * The arithmetic is that of ss_conv1d_fwd with seqlen = 1 and
 * init_state = final_state = state.
 */
typedef struct {
    int batch, dim, width;
    int in_dtype, out_dtype;
    float *state;
    const void *x;
    const float *weight, *bias;
    int silu;
    void *out;
} ss_conv1d_update_args;

int ss_conv1d_update(ss_ctx *ctx, const ss_conv1d_update_args *args, ss_stream_t stream);

/*
 * Selective scan forward without any device allocation. The pages have no
 * counterpart to this entry point: it exists for callers that may not call
 * cudaMalloc at all (inside memory-planned or graph-captured regions, in
 * real-time paths that must not block on the allocator, in plugins whose host
 * owns every allocation). ss_create allocates, so no context is used.
 *   args         : as for ss_scan_fwd; the shape must suit the chained
 *                  pair-row kernel (dstate 16, seqlen a multiple of 16, u,
 *                  delta, z, y 32-byte aligned) and its scratch must fit the
 *                  library's static 8 MiB device array (roughly
 *                  batch * seqlen * 128 B + batch * dim * 64 B + 1 KiB);
 *                  otherwise SS_ERR_UNSUPPORTED and nothing is enqueued.
 *   device_error : caller-owned device int that receives SS_ERR_TIMEOUT if a
 *                  bounded device wait gives up (it is only written then);
 *                  may be NULL.
 * The scratch array is shared by every call on a device and keeps the last
 * call's contents; the call clears what must start at zero. Calls that
 * overlap on the GPU race on it: order them on one stream. Calls from several
 * host threads are serialised by a per-device lock held while the call is
 * numbered and enqueued, so on one stream they run in that order. The first
 * successful call on a device resolves the array's address and clears it
 * synchronously: make it before any stream capture. If that set-up fails the
 * call returns SS_ERR_CUDA and the next call tries it again. Returns SS_OK or
 * an error from ss_status.
 */
int ss_scan_fwd_noalloc(const ss_scan_args *args, int *device_error, ss_stream_t stream);

/*
 * Synchronise `stream`, then return and clear the context's device error
 * word: SS_OK when no device-side check fired since the last read,
 * SS_ERR_TIMEOUT when a bounded wait gave up, SS_ERR_CUDA if the sync failed.
 */
int ss_get_device_error(ss_ctx *ctx, ss_stream_t stream);

/* Static text for a status code. */
const char *ss_status_string(int status);

/*
 * Kernel selection for ss_scan_fwd (default SS_VARIANT_AUTO).
 *   SS_VARIANT_ROWS    : one pass; each row's time axis is walked in order by
 *                        a small group of threads, inputs staged by TMA.
 *   SS_VARIANT_CHUNKED : the time axis is cut into segments scanned in
 *                        parallel from a zero state; per-segment (decay,
 *                        state) pairs are combined along time by a
 *                        warp-shuffle associative scan and the segments are
 *                        scanned again from their carried-in state (dstate
 *                        16, seqlen a multiple of 16). AUTO picks it when there
 *                        are too few row blocks of 32 rows to fill the GPU.
 *   SS_VARIANT_SIMPLE  : one thread per row, plain loads; used for shapes the
 *                        staged kernels cannot take (e.g. seqlen % 8 != 0).
 * Options (ss_set_option):
 *   SS_OPT_VARIANT          one of ss_variant.
 *   SS_OPT_SEGMENTS         time segments per row block for the chunked
 *                           variant (0 = auto).
 *   SS_OPT_THREADS_PER_ROW  how the rows variant splits a row's states over
 *                           threads: 1 = one thread per row (any dstate);
 *                           2 = two threads share a pair of rows, and the
 *                           row blocks' time steps are cut into one equal
 *                           range per persistent warp (a row block split
 *                           between two ranges passes its state through the
 *                           context scratch; dstate 16); 4 = four threads per
 *                           row (dstate 16); 0 = auto (2 for dstate 16, else 1).
 *   SS_OPT_RESIDENT_WARPS   persistent warps per SM for the pair kernel
 *                           (default 8; 0 = as many as fit).
 *   SS_OPT_WAIT_LIMIT       polls before a device-side wait gives up and
 *                           reports SS_ERR_TIMEOUT (default 2^22, roughly a
 *                           second; 1 .. 2^30).
 *   SS_OPT_DISCRETIZATION   input matrix of ss_scan_fwd, ss_scan_bwd and ss_state_update:
 *                           SS_DISC_SIMPLIFIED (default) uses dt * B, the step
 *                           the soft186.com article prints ("动态参数化的状态空间");
 *                           SS_DISC_ZOH uses the exact zero-order hold
 *                           (exp(dt A) - 1) / A * B of the Mamba page's section
 *                           "Method" (dt * B where A = 0). ZOH runs on the
 *                           chained pair-row and chunked kernels (AUTO picks
 *                           them as for the simplified form) and on the
 *                           one-thread-per-row kernels; forcing the 4-thread
 *                           split-row kernel (THREADS_PER_ROW 4) returns
 *                           SS_ERR_UNSUPPORTED, and so does ss_conv_scan_fwd. ss_scan_fwd_noalloc
 *                           always uses the simplified form.
 *   SS_OPT_TEST_DROP_TILE   test hook: the rows kernel never issues the loads
 *                           of this tile index, so its wait runs out and the
 *                           timeout path is exercised (-1 = off, the default).
 *   SS_OPT_SSD_PATH         tensor-core kernel of ss_ssd_fwd:
 *                           SS_SSD_PATH_TCGEN05 runs the tensor-memory kernel
 *                           (tcgen05 products with accumulators in tensor
 *                           memory, 128-step chunks, operands and y moved by
 *                           TMA; headdim 64, dstate 128, seqlen a multiple of
 *                           128, y, B and C 16-byte aligned, else
 *                           SS_ERR_UNSUPPORTED); SS_SSD_PATH_MMA_SYNC runs the
 *                           warp-level mma.sync kernel (64-step chunks, any
 *                           headdim multiple of 16 and dstate 64 or 128);
 *                           SS_SSD_PATH_AUTO (default) takes the tensor-memory
 *                           kernel wherever it applies (the faster of the two
 *                           at the Mamba-2 block shape), else mma.sync.
 * Returns SS_OK or SS_ERR_INVALID_ARG (unknown option or value out of range).
 */
typedef enum {
    SS_VARIANT_AUTO = 0,
    SS_VARIANT_ROWS = 1,
    SS_VARIANT_CHUNKED = 2,
    SS_VARIANT_SIMPLE = 3
} ss_variant;

typedef enum {
    SS_OPT_VARIANT = 0,
    SS_OPT_SEGMENTS = 1,
    SS_OPT_THREADS_PER_ROW = 2,
    SS_OPT_WAIT_LIMIT = 3,
    SS_OPT_TEST_DROP_TILE = 4,
    SS_OPT_RESIDENT_WARPS = 5,
    SS_OPT_DISCRETIZATION = 6,
    SS_OPT_SSD_PATH = 7
} ss_option;

typedef enum {
    SS_SSD_PATH_AUTO = 0,
    SS_SSD_PATH_MMA_SYNC = 1,
    SS_SSD_PATH_TCGEN05 = 2
} ss_ssd_path;

typedef enum { SS_DISC_SIMPLIFIED = 0, SS_DISC_ZOH = 1 } ss_discretization;

int ss_set_option(ss_ctx *ctx, int option, long long value);

/*
 * Describe the last ss_scan_fwd / ss_state_update enqueued on this context:
 * *variant receives the ss_variant that ran, *launches the number of kernels
 * it enqueued. After ss_ssd_fwd, *variant is 1 for the tensor-memory kernel
 * and 0 for the mma.sync kernel. Either pointer may be NULL.
 */
int ss_last_launch(const ss_ctx *ctx, int *variant, int *launches);

#ifdef __cplusplus
}
#endif

#endif /* SS_SCAN_H */
