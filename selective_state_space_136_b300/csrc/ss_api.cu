// C ABI of the ss_scan library: context management, argument validation and
// kernel selection. Every entry point validates on the host and returns an
// ss_status; nothing is enqueued when validation fails.
#include <stdint.h>
#include <string.h>

#include "ss_internal.h"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dtype(int t) { return t == SS_F32 || t == SS_BF16; }

bool valid_dstate(int n) { return n == 1 || n == 2 || n == 4 || n == 8 || n == 16; }

struct Span {
    uintptr_t lo, hi;  // [lo, hi)
};
Span span(const void *p, size_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Span{a, a + bytes};
}
bool overlaps(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

// Grow the context scratch to hold the chained kernel's buffers; zero it when
// (re)allocated (the flags must start below every epoch).
int ensure_pair_scratch(ss_ctx *ctx, const ssh::ScanParams &p, int n_seg, bool chunked,
                        ssh::PairWork *w) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t flags_b = up((size_t)ssh::pair_row_blocks(p) * 8);
    const size_t carry_b = up(ssh::pair_carry_bytes(p));
    const size_t bc_b = up(ssh::pair_bc_bytes(p));
    const size_t agg_b = chunked ? up(ssh::pair_agg_bytes(p, n_seg)) : 0;
    const size_t need = 256 + flags_b + carry_b + bc_b + agg_b;
    if (need > ctx->scratch_bytes) {
        if (ctx->scratch) {
            if (cudaFree(ctx->scratch) != cudaSuccess) return SS_ERR_CUDA;
            ctx->scratch = nullptr;
            ctx->scratch_bytes = 0;
        }
        if (cudaMalloc(&ctx->scratch, need) != cudaSuccess) return SS_ERR_CUDA;
        if (cudaMemset(ctx->scratch, 0, need) != cudaSuccess) return SS_ERR_CUDA;
        ctx->scratch_bytes = need;
    }
    uint8_t *base = static_cast<uint8_t *>(ctx->scratch);
    w->counter = reinterpret_cast<unsigned long long *>(base);
    w->flags = reinterpret_cast<unsigned long long *>(base + 256);
    w->carry = reinterpret_cast<float *>(base + 256 + flags_b);
    w->bc = reinterpret_cast<float *>(base + 256 + flags_b + carry_b);
    w->hagg = chunked ? reinterpret_cast<float *>(base + 256 + flags_b + carry_b + bc_b) : nullptr;
    w->sdt = chunked ? w->hagg + (size_t)ssh::pair_row_blocks(p) * n_seg * 32 * 16 : nullptr;
    w->chunked = chunked;
    return SS_OK;
}

int dispatch_scan(ss_ctx *ctx, const ssh::ScanParams &p, cudaStream_t st);

int set_device(const ss_ctx *ctx) {
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return SS_ERR_CUDA;
    if (cur != ctx->device && cudaSetDevice(ctx->device) != cudaSuccess) return SS_ERR_CUDA;
    return SS_OK;
}

}  // namespace

extern "C" {

const char *ss_status_string(int status) {
    switch (status) {
        case SS_OK: return "ok";
        case SS_ERR_INVALID_ARG: return "invalid argument";
        case SS_ERR_UNSUPPORTED: return "unsupported configuration";
        case SS_ERR_CUDA: return "CUDA runtime error";
        case SS_ERR_TIMEOUT: return "device wait timed out";
        case SS_ERR_DEVICE: return "device-side error";
        default: return "unknown status";
    }
}

int ss_create(ss_ctx **out, int device) {
    if (!out) return SS_ERR_INVALID_ARG;
    *out = nullptr;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
        return SS_ERR_CUDA;
    ss_ctx *c = new ss_ctx();
    c->device = device;
    int prev = 0;
    cudaGetDevice(&prev);
    if (cudaSetDevice(device) != cudaSuccess ||
        cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, device) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&c->max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                               device) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void **>(&c->d_err), sizeof(int)) != cudaSuccess ||
        cudaMemset(c->d_err, 0, sizeof(int)) != cudaSuccess) {
        if (c->d_err) cudaFree(c->d_err);
        delete c;
        cudaSetDevice(prev);
        return SS_ERR_CUDA;
    }
    cudaSetDevice(prev);
    *out = c;
    return SS_OK;
}

int ss_destroy(ss_ctx *ctx) {
    if (!ctx) return SS_OK;
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(ctx->device);
    cudaDeviceSynchronize();
    if (ctx->d_err) cudaFree(ctx->d_err);
    if (ctx->scratch) cudaFree(ctx->scratch);
    if (ctx->bwd_scratch) cudaFree(ctx->bwd_scratch);
    cudaSetDevice(prev);
    delete ctx;
    return SS_OK;
}

int ss_set_option(ss_ctx *ctx, int option, long long value) {
    if (!ctx) return SS_ERR_INVALID_ARG;
    switch (option) {
        case SS_OPT_VARIANT:
            if (value < SS_VARIANT_AUTO || value > SS_VARIANT_SIMPLE) return SS_ERR_INVALID_ARG;
            ctx->variant = (int)value;
            return SS_OK;
        case SS_OPT_SEGMENTS:
            if (value < 0 || value > 65535) return SS_ERR_INVALID_ARG;
            ctx->segments = (int)value;
            return SS_OK;
        case SS_OPT_THREADS_PER_ROW:
            if (value != 0 && value != 1 && value != 2 && value != 4) return SS_ERR_INVALID_ARG;
            ctx->rows_tpr = (int)value;
            return SS_OK;
        case SS_OPT_RESIDENT_WARPS:
            if (value < 0 || value > 64) return SS_ERR_INVALID_ARG;
            ctx->warps_per_sm = (int)value;
            return SS_OK;
        case SS_OPT_DISCRETIZATION:
            if (value != SS_DISC_SIMPLIFIED && value != SS_DISC_ZOH) return SS_ERR_INVALID_ARG;
            ctx->zoh = (int)value;
            return SS_OK;
        case SS_OPT_WAIT_LIMIT:
            if (value < 1 || value > (1LL << 30)) return SS_ERR_INVALID_ARG;
            ctx->wait_limit = (uint32_t)value;
            return SS_OK;
        case SS_OPT_TEST_DROP_TILE:
            if (value < -1 || value > (1LL << 30)) return SS_ERR_INVALID_ARG;
            ctx->drop_tile = (int)value;
            return SS_OK;
        case SS_OPT_SSD_PATH:
            if (value < SS_SSD_PATH_AUTO || value > SS_SSD_PATH_TCGEN05) return SS_ERR_INVALID_ARG;
            ctx->ssd_path = (int)value;
            return SS_OK;
        default: return SS_ERR_INVALID_ARG;
    }
}

int ss_last_launch(const ss_ctx *ctx, int *variant, int *launches) {
    if (!ctx) return SS_ERR_INVALID_ARG;
    if (variant) *variant = ctx->last_variant;
    if (launches) *launches = ctx->last_launches;
    return SS_OK;
}

int ss_get_device_error(ss_ctx *ctx, ss_stream_t stream) {
    if (!ctx) return SS_ERR_INVALID_ARG;
    if (set_device(ctx) != SS_OK) return SS_ERR_CUDA;
    int h = 0;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return SS_ERR_CUDA;
    if (cudaMemcpy(&h, ctx->d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SS_ERR_CUDA;
    if (h != 0 && cudaMemset(ctx->d_err, 0, sizeof(int)) != cudaSuccess) return SS_ERR_CUDA;
    return h;
}

int ss_scan_fwd(ss_ctx *ctx, const ss_scan_args *a, ss_stream_t stream) {
    if (!ctx || !a) return SS_ERR_INVALID_ARG;
    if (a->batch < 1 || a->dim < 1 || a->seqlen < 0) return SS_ERR_INVALID_ARG;
    if (!valid_dtype(a->in_dtype) || !valid_dtype(a->out_dtype)) return SS_ERR_INVALID_ARG;
    if (!valid_dstate(a->dstate)) return SS_ERR_UNSUPPORTED;
    if ((long long)a->batch * a->dim > (1LL << 40) || a->seqlen >= (1LL << 40))
        return SS_ERR_INVALID_ARG;
    const long long rows = (long long)a->batch * a->dim;
    const size_t esz = a->in_dtype == SS_BF16 ? 2 : 4;
    const size_t osz = a->out_dtype == SS_BF16 ? 2 : 4;
    const size_t n_elem = (size_t)rows * (size_t)a->seqlen;
    const size_t n_bc = (size_t)a->batch * a->dstate * (size_t)a->seqlen;
    const size_t n_state = (size_t)rows * a->dstate;
    if (!a->A) return SS_ERR_INVALID_ARG;
    if (a->seqlen > 0 && (!a->u || !a->delta || !a->B || !a->C || !a->y))
        return SS_ERR_INVALID_ARG;
    const void *ptrs[] = {a->u, a->delta, a->z, a->A, a->B, a->C, a->D, a->delta_bias, a->h0,
                          a->y, a->h_last};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return SS_ERR_INVALID_ARG;
    // outputs must not overlap inputs (h_last == h0 is allowed: read then written per row)
    if (a->seqlen > 0) {
        const Span y = span(a->y, n_elem * osz);
        const Span ins[] = {span(a->u, n_elem * esz), span(a->delta, n_elem * esz),
                            span(a->z, a->z ? n_elem * esz : 0), span(a->B, n_bc * esz),
                            span(a->C, n_bc * esz), span(a->A, (size_t)a->dim * a->dstate * 4),
                            span(a->D, a->D ? (size_t)a->dim * 4 : 0),
                            span(a->delta_bias, a->delta_bias ? (size_t)a->dim * 4 : 0),
                            span(a->h0, a->h0 ? n_state * 4 : 0),
                            span(a->h_last, a->h_last ? n_state * 4 : 0)};
        for (const Span &s : ins)
            if (overlaps(y, s)) return SS_ERR_INVALID_ARG;
    }
    if (a->h_last && a->h0 && a->h_last != a->h0 &&
        overlaps(span(a->h_last, n_state * 4), span(a->h0, n_state * 4)))
        return SS_ERR_INVALID_ARG;
    if (a->h_last && a->seqlen > 0) {
        const Span hl = span(a->h_last, n_state * 4);
        const Span ins[] = {span(a->u, n_elem * esz), span(a->delta, n_elem * esz),
                            span(a->z, a->z ? n_elem * esz : 0), span(a->B, n_bc * esz),
                            span(a->C, n_bc * esz)};
        for (const Span &s : ins)
            if (overlaps(hl, s)) return SS_ERR_INVALID_ARG;
    }
    if (set_device(ctx) != SS_OK) return SS_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    ctx->last_launches = 0;

    if (a->seqlen == 0) {
        ctx->last_variant = SS_VARIANT_AUTO;
        if (!a->h_last) return SS_OK;
        cudaError_t e = a->h0 ? (a->h0 == a->h_last
                                     ? cudaSuccess
                                     : cudaMemcpyAsync(a->h_last, a->h0, n_state * 4,
                                                       cudaMemcpyDeviceToDevice, st))
                              : cudaMemsetAsync(a->h_last, 0, n_state * 4, st);
        return e == cudaSuccess ? SS_OK : SS_ERR_CUDA;
    }

    ssh::ScanParams p{a->batch, a->dim, a->dstate, a->seqlen, a->in_dtype, a->out_dtype,
                      a->u, a->delta, a->z, a->A, a->B, a->C, a->D, a->delta_bias,
                      a->delta_softplus, a->h0, a->y, a->h_last, ctx->d_err, ctx->wait_limit,
                      ctx->drop_tile, ctx->zoh};
    return dispatch_scan(ctx, p, st);
}

}  // extern "C"

namespace {

// Launch the chained pair-row kernel (one pass) or its chunked variant (time
// segments scanned in parallel, then combined) for p; the rule is the one
// SS_VARIANT_AUTO uses: chunked when there are fewer than half as many row
// blocks as resident warps.
int run_pair(ss_ctx *ctx, const ssh::ScanParams &p, bool chunked, cudaStream_t st,
             int *launches) {
    int rc;
    if (chunked) {
        const long long resident = (long long)(ctx->warps_per_sm > 0 ? ctx->warps_per_sm : 8) *
                                   ctx->sm_count;
        int req = ctx->segments;
        if (req <= 0) {
            // about one unit per resident warp (one segment fewer when that
            // still fills 95 % of them: the output pass then runs in one wave,
            // not 1.3), and segments of at most 8192 steps so long sequences
            // split into many small balanced units
            const long long rb = ssh::pair_row_blocks(p);
            long long r = (resident + rb - 1) / rb;
            if (r > 2 && rb * (r - 1) * 20 >= resident * 19) --r;
            const long long by_len = (p.seqlen + 8191) / 8192;
            if (by_len > r) r = by_len;
            req = (int)(r < 2 ? 2 : (r > 65535 ? 65535 : r));
        }
        const int n_seg = ssh::pair_segments(p, req);
        ssh::PairWork w{};
        if ((rc = ensure_pair_scratch(ctx, p, n_seg, true, &w)) != SS_OK) return rc;
        w.epoch = ++ctx->epoch;
        w.sm_count = ctx->sm_count;
        w.warps_per_sm = ctx->warps_per_sm;
        w.n_seg = n_seg;
        *launches = n_seg >= 2 ? 4 : 2;
        return ssh::launch_pair(p, w, st);
    }
    ssh::PairWork w{};
    const int n_seg = 1;  // the chained kernel balances by tile ranges, not segments
    if ((rc = ensure_pair_scratch(ctx, p, n_seg, false, &w)) != SS_OK) return rc;
    w.epoch = ++ctx->epoch;
    w.sm_count = ctx->sm_count;
    w.warps_per_sm = ctx->warps_per_sm;
    w.n_seg = n_seg;
    *launches = 2;
    return ssh::launch_pair(p, w, st);
}

bool prefer_chunked(const ss_ctx *ctx, const ssh::ScanParams &p) {
    const long long resident = (long long)(ctx->warps_per_sm > 0 ? ctx->warps_per_sm : 8) *
                               ctx->sm_count;
    return 2LL * ssh::pair_row_blocks(p) < resident;
}

int dispatch_scan(ss_ctx *ctx, const ssh::ScanParams &p, cudaStream_t st) {
    int variant = ctx->variant;
    const bool rows_ok = ssh::rows_supported(p) && ssh::seq_supported(p);
    // the exact zero-order hold runs on the pair-row kernels (chained and
    // chunked) and the one-thread-per-row kernels; not on the 4-thread rows kernel
    const bool pair_ok = ssh::pair_supported(p);
    if (variant == SS_VARIANT_AUTO) {
        // few row blocks for the machine: scan time segments in parallel
        if (pair_ok && prefer_chunked(ctx, p)) variant = SS_VARIANT_CHUNKED;
        else variant = rows_ok ? SS_VARIANT_ROWS : SS_VARIANT_SIMPLE;
    }
    if (variant == SS_VARIANT_ROWS && !rows_ok) return SS_ERR_UNSUPPORTED;
    int rc, launches = 1;
    if (variant == SS_VARIANT_CHUNKED) {
        if (!pair_ok) return SS_ERR_UNSUPPORTED;
        rc = run_pair(ctx, p, true, st, &launches);
    } else if (variant == SS_VARIANT_ROWS) {
        int tpr = ctx->rows_tpr;
        if (tpr == 0) tpr = pair_ok ? 2 : 1;
        if (ctx->zoh && tpr == 4) return SS_ERR_UNSUPPORTED;
        if (tpr == 2) {
            if (!pair_ok) return SS_ERR_UNSUPPORTED;
            rc = run_pair(ctx, p, false, st, &launches);
        } else if (tpr == 1) {
            rc = ssh::launch_seq(p, ctx->max_smem_optin, st);
        } else {
            rc = ssh::launch_rows(p, tpr, ctx->max_smem_optin, st);
        }
    } else {
        rc = ssh::launch_simple(p, st);
    }
    ctx->last_variant = variant;
    ctx->last_launches = rc == SS_OK ? launches : 0;
    return rc;
}

}  // namespace

extern "C" {

int ss_conv_scan_fwd(ss_ctx *ctx, const ss_conv_scan_args *ca, ss_stream_t stream) {
    if (!ctx || !ca) return SS_ERR_INVALID_ARG;
    const ss_scan_args *a = &ca->scan;
    if (a->batch < 1 || a->dim < 1 || a->seqlen < 0) return SS_ERR_INVALID_ARG;
    if (!valid_dtype(a->in_dtype) || !valid_dtype(a->out_dtype)) return SS_ERR_INVALID_ARG;
    if (ca->conv_width < 2 || ca->conv_width > 4) return SS_ERR_UNSUPPORTED;
    if (a->dstate != 16) return SS_ERR_UNSUPPORTED;
    if ((long long)a->batch * a->dim > (1LL << 40) || a->seqlen >= (1LL << 40))
        return SS_ERR_INVALID_ARG;
    if (!a->A || !ca->conv_weight) return SS_ERR_INVALID_ARG;
    if (a->seqlen > 0 && (!a->u || !a->delta || !a->B || !a->C || !a->y))
        return SS_ERR_INVALID_ARG;
    const void *ptrs[] = {a->u, a->delta, a->z, a->A, a->B, a->C, a->D, a->delta_bias, a->h0,
                          a->y, a->h_last, ca->conv_weight, ca->conv_bias, ca->conv_init,
                          ca->u_out, ca->conv_state_out};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return SS_ERR_INVALID_ARG;
    const long long rows = (long long)a->batch * a->dim;
    const size_t esz = a->in_dtype == SS_BF16 ? 2 : 4, osz = a->out_dtype == SS_BF16 ? 2 : 4;
    const size_t n_elem = (size_t)rows * (size_t)a->seqlen;
    const size_t n_bc = (size_t)a->batch * 16 * (size_t)a->seqlen;
    const size_t n_state = (size_t)rows * 16;
    const size_t n_cst = (size_t)rows * (size_t)(ca->conv_width - 1);
    // every output against every input and against the other outputs
    const Span ins[] = {span(a->u, n_elem * esz), span(a->delta, n_elem * esz),
                        span(a->z, a->z ? n_elem * esz : 0), span(a->B, n_bc * esz),
                        span(a->C, n_bc * esz), span(a->A, (size_t)a->dim * 16 * 4),
                        span(a->D, a->D ? (size_t)a->dim * 4 : 0),
                        span(a->delta_bias, a->delta_bias ? (size_t)a->dim * 4 : 0),
                        span(a->h0, a->h0 ? n_state * 4 : 0),
                        span(ca->conv_weight, (size_t)a->dim * ca->conv_width * 4),
                        span(ca->conv_bias, ca->conv_bias ? (size_t)a->dim * 4 : 0),
                        span(ca->conv_init, ca->conv_init ? n_cst * 4 : 0)};
    const Span outs[] = {span(a->y, a->seqlen > 0 ? n_elem * osz : 0),
                         span(a->h_last, a->h_last ? n_state * 4 : 0),
                         span(ca->u_out, ca->u_out ? n_elem * esz : 0),
                         span(ca->conv_state_out, ca->conv_state_out ? n_cst * 4 : 0)};
    const size_t n_out = sizeof(outs) / sizeof(outs[0]);
    for (size_t i = 0; i < n_out; ++i) {
        for (const Span &in : ins) {
            // h_last may be h0 itself (read, then written per row)
            if (i == 1 && a->h0 && a->h_last == a->h0 && in.lo == span(a->h0, 1).lo) continue;
            if (overlaps(outs[i], in)) return SS_ERR_INVALID_ARG;
        }
        for (size_t j = i + 1; j < n_out; ++j)
            if (overlaps(outs[i], outs[j])) return SS_ERR_INVALID_ARG;
    }
    if (set_device(ctx) != SS_OK) return SS_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    ctx->last_launches = 0;
    ctx->last_variant = SS_VARIANT_AUTO;
    if (a->seqlen == 0) {
        if (a->h_last) {
            const cudaError_t e = a->h0 ? (a->h0 == a->h_last ? cudaSuccess
                                                              : cudaMemcpyAsync(a->h_last, a->h0, n_state * 4,
                                                                                cudaMemcpyDeviceToDevice, st))
                                        : cudaMemsetAsync(a->h_last, 0, n_state * 4, st);
            if (e != cudaSuccess) return SS_ERR_CUDA;
        }
        if (ca->conv_state_out) {
            const cudaError_t e = ca->conv_init
                                      ? cudaMemcpyAsync(ca->conv_state_out, ca->conv_init, n_cst * 4,
                                                        cudaMemcpyDeviceToDevice, st)
                                      : cudaMemsetAsync(ca->conv_state_out, 0, n_cst * 4, st);
            if (e != cudaSuccess) return SS_ERR_CUDA;
        }
        return SS_OK;
    }
    ssh::ScanParams p{a->batch, a->dim, a->dstate, a->seqlen, a->in_dtype, a->out_dtype,
                      a->u, a->delta, a->z, a->A, a->B, a->C, a->D, a->delta_bias,
                      a->delta_softplus, a->h0, a->y, a->h_last, ctx->d_err, ctx->wait_limit,
                      ctx->drop_tile, ctx->zoh, ca->conv_width, ca->conv_silu, ca->conv_weight,
                      ca->conv_bias, ca->conv_init, ca->conv_state_out, ca->u_out};
    // the fused convolution lives in the chained pair-row kernel only (its u_out
    // stores whole 32-byte sectors, like y)
    if (!ssh::pair_supported(p) || ctx->zoh) return SS_ERR_UNSUPPORTED;
    if (ca->u_out && (reinterpret_cast<uintptr_t>(ca->u_out) & 31u) != 0) return SS_ERR_UNSUPPORTED;
    bool chunked = prefer_chunked(ctx, p);
    if (ctx->variant == SS_VARIANT_CHUNKED) chunked = true;
    else if (ctx->variant == SS_VARIANT_ROWS && (ctx->rows_tpr == 0 || ctx->rows_tpr == 2)) chunked = false;
    else if (ctx->variant != SS_VARIANT_AUTO) return SS_ERR_UNSUPPORTED;
    int launches = 0;
    const int rc = run_pair(ctx, p, chunked, st, &launches);
    ctx->last_variant = chunked ? SS_VARIANT_CHUNKED : SS_VARIANT_ROWS;
    ctx->last_launches = rc == SS_OK ? launches : 0;
    return rc;
}

int ss_state_update(ss_ctx *ctx, const ss_update_args *a, ss_stream_t stream) {
    if (!ctx || !a) return SS_ERR_INVALID_ARG;
    if (a->batch < 1 || a->dim < 1) return SS_ERR_INVALID_ARG;
    if (!valid_dtype(a->in_dtype) || !valid_dtype(a->out_dtype)) return SS_ERR_INVALID_ARG;
    if (!valid_dstate(a->dstate)) return SS_ERR_UNSUPPORTED;
    if ((long long)a->batch * a->dim > (1LL << 40)) return SS_ERR_INVALID_ARG;
    if (!a->state || !a->x || !a->dt || !a->A || !a->B || !a->C || !a->y)
        return SS_ERR_INVALID_ARG;
    const void *ptrs[] = {a->state, a->x, a->dt, a->z, a->A, a->B, a->C, a->D, a->dt_bias, a->y};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return SS_ERR_INVALID_ARG;
    const size_t rows = (size_t)a->batch * a->dim;
    const size_t esz = a->in_dtype == SS_BF16 ? 2 : 4;
    const size_t osz = a->out_dtype == SS_BF16 ? 2 : 4;
    const Span y = span(a->y, rows * osz);
    const Span stt = span(a->state, rows * a->dstate * 4);
    const Span ins[] = {stt, span(a->x, rows * esz), span(a->dt, rows * esz),
                        span(a->z, a->z ? rows * esz : 0),
                        span(a->A, (size_t)a->dim * a->dstate * 4),
                        span(a->B, (size_t)a->batch * a->dstate * esz),
                        span(a->C, (size_t)a->batch * a->dstate * esz),
                        span(a->D, a->D ? (size_t)a->dim * 4 : 0),
                        span(a->dt_bias, a->dt_bias ? (size_t)a->dim * 4 : 0)};
    for (const Span &s : ins)
        if (overlaps(y, s)) return SS_ERR_INVALID_ARG;
    for (size_t i = 1; i < sizeof(ins) / sizeof(ins[0]); ++i)
        if (overlaps(stt, ins[i])) return SS_ERR_INVALID_ARG;
    if (set_device(ctx) != SS_OK) return SS_ERR_CUDA;
    ssh::UpdateParams p{a->batch, a->dim, a->dstate, a->in_dtype, a->out_dtype, a->state,
                        a->x, a->dt, a->z, a->A, a->B, a->C, a->D, a->dt_bias,
                        a->dt_softplus, a->y, ctx->zoh};
    const int rc = ssh::launch_update(p, reinterpret_cast<cudaStream_t>(stream));
    ctx->last_variant = 0;
    ctx->last_launches = rc == SS_OK ? 1 : 0;
    return rc;
}

int ss_scan_bwd(ss_ctx *ctx, const ss_scan_bwd_args *a, ss_stream_t stream) {
    if (!ctx || !a) return SS_ERR_INVALID_ARG;
    if (a->batch < 1 || a->dim < 1 || a->seqlen < 1) return SS_ERR_INVALID_ARG;
    if (!valid_dtype(a->in_dtype)) return SS_ERR_INVALID_ARG;
    if (!valid_dstate(a->dstate)) return SS_ERR_UNSUPPORTED;
    if ((long long)a->batch * a->dim > (1LL << 40) || a->seqlen >= (1LL << 35))
        return SS_ERR_INVALID_ARG;
    if (!a->u || !a->delta || !a->A || !a->B || !a->C || !a->dy || !a->du || !a->ddelta ||
        !a->dA || !a->dB || !a->dC)
        return SS_ERR_INVALID_ARG;
    if (a->dz && !a->z) return SS_ERR_INVALID_ARG;
    const void *ptrs[] = {a->u,  a->delta, a->z,  a->A,  a->B,  a->C,  a->D,  a->delta_bias,
                          a->h0, a->dy,    a->dh_last, a->du, a->ddelta, a->dz, a->dA,
                          a->dB, a->dC,    a->dD, a->ddelta_bias, a->dh0};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return SS_ERR_INVALID_ARG;
    const size_t rows = (size_t)a->batch * a->dim, L = (size_t)a->seqlen, N = (size_t)a->dstate;
    const size_t esz = a->in_dtype == SS_BF16 ? 2 : 4;
    const Span ins[] = {span(a->u, rows * L * esz), span(a->delta, rows * L * esz),
                        span(a->z, a->z ? rows * L * esz : 0), span(a->A, (size_t)a->dim * N * 4),
                        span(a->B, (size_t)a->batch * N * L * esz),
                        span(a->C, (size_t)a->batch * N * L * esz),
                        span(a->D, a->D ? (size_t)a->dim * 4 : 0),
                        span(a->delta_bias, a->delta_bias ? (size_t)a->dim * 4 : 0),
                        span(a->h0, a->h0 ? rows * N * 4 : 0), span(a->dy, rows * L * 4),
                        span(a->dh_last, a->dh_last ? rows * N * 4 : 0)};
    const Span outs[] = {span(a->du, rows * L * 4), span(a->ddelta, rows * L * 4),
                         span(a->dz, a->dz ? rows * L * 4 : 0), span(a->dA, (size_t)a->dim * N * 4),
                         span(a->dB, (size_t)a->batch * N * L * 4),
                         span(a->dC, (size_t)a->batch * N * L * 4),
                         span(a->dD, a->dD ? (size_t)a->dim * 4 : 0),
                         span(a->ddelta_bias, a->ddelta_bias ? (size_t)a->dim * 4 : 0),
                         span(a->dh0, a->dh0 ? rows * N * 4 : 0)};
    const size_t n_out = sizeof(outs) / sizeof(outs[0]);
    for (size_t i = 0; i < n_out; ++i) {
        for (const Span &s : ins)
            if (overlaps(outs[i], s)) return SS_ERR_INVALID_ARG;
        for (size_t j = i + 1; j < n_out; ++j)
            if (overlaps(outs[i], outs[j])) return SS_ERR_INVALID_ARG;
    }
    ssh::BwdParams p{a->batch, a->dim, a->dstate, a->seqlen, a->in_dtype, a->u, a->delta, a->z,
                     a->A, a->B, a->C, a->D, a->delta_bias, a->delta_softplus, a->h0, a->dy,
                     a->dh_last, a->du, a->ddelta, a->dz, a->dA, a->dB, a->dC, a->dD,
                     a->ddelta_bias, a->dh0, nullptr, ctx->zoh};
    if (!ssh::bwd_supported(p)) return SS_ERR_UNSUPPORTED;
    if (set_device(ctx) != SS_OK) return SS_ERR_CUDA;
    const size_t need = ssh::bwd_ckpt_bytes(p);
    if (need > ctx->bwd_scratch_bytes) {
        if (ctx->bwd_scratch) {
            if (cudaFree(ctx->bwd_scratch) != cudaSuccess) return SS_ERR_CUDA;
            ctx->bwd_scratch = nullptr;
            ctx->bwd_scratch_bytes = 0;
        }
        if (cudaMalloc(&ctx->bwd_scratch, need) != cudaSuccess) return SS_ERR_CUDA;
        ctx->bwd_scratch_bytes = need;
    }
    p.ckpt = static_cast<float *>(ctx->bwd_scratch);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the sums over rows start from zero
    float *sums[] = {a->dA, a->dB, a->dC, a->dD, a->ddelta_bias};
    const size_t sum_b[] = {(size_t)a->dim * N * 4, (size_t)a->batch * N * L * 4,
                            (size_t)a->batch * N * L * 4, (size_t)a->dim * 4, (size_t)a->dim * 4};
    for (int i = 0; i < 5; ++i)
        if (sums[i] && cudaMemsetAsync(sums[i], 0, sum_b[i], st) != cudaSuccess) return SS_ERR_CUDA;
    const int rc = ssh::launch_bwd(p, st);
    ctx->last_variant = 0;
    ctx->last_launches = rc == SS_OK ? 1 : 0;
    return rc;
}

int ss_ssd_fwd(ss_ctx *ctx, const ss_ssd_args *a, ss_stream_t stream) {
    if (!ctx || !a) return SS_ERR_INVALID_ARG;
    if (a->batch < 1 || a->heads < 1 || a->headdim < 1 || a->dstate < 1 || a->seqlen < 1)
        return SS_ERR_INVALID_ARG;
    if (!valid_dtype(a->in_dtype) || !valid_dtype(a->out_dtype)) return SS_ERR_INVALID_ARG;
    if (!a->x || !a->dt || !a->A || !a->B || !a->C || !a->y) return SS_ERR_INVALID_ARG;
    const void *ptrs[] = {a->x, a->dt, a->A, a->B, a->C, a->D, a->dt_bias, a->h0, a->y, a->h_last};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return SS_ERR_INVALID_ARG;
    if ((long long)a->batch * a->heads > (1LL << 30) || a->seqlen >= (1LL << 35))
        return SS_ERR_INVALID_ARG;
    const size_t esz = a->in_dtype == SS_BF16 ? 2 : 4, osz = a->out_dtype == SS_BF16 ? 2 : 4;
    const size_t BL = (size_t)a->batch * (size_t)a->seqlen;
    const size_t nx = BL * a->heads * a->headdim;
    const size_t nst = (size_t)a->batch * a->heads * a->headdim * a->dstate * 4;
    const Span y = span(a->y, nx * osz), hl = span(a->h_last, a->h_last ? nst : 0);
    const Span ins[] = {span(a->x, nx * esz), span(a->dt, BL * a->heads * esz),
                        span(a->A, (size_t)a->heads * 4), span(a->B, BL * a->dstate * esz),
                        span(a->C, BL * a->dstate * esz),
                        span(a->D, a->D ? (size_t)a->heads * 4 : 0),
                        span(a->dt_bias, a->dt_bias ? (size_t)a->heads * 4 : 0)};
    for (const Span &s : ins)
        if (overlaps(y, s) || overlaps(hl, s)) return SS_ERR_INVALID_ARG;
    if (overlaps(y, span(a->h0, a->h0 ? nst : 0)) || overlaps(y, hl)) return SS_ERR_INVALID_ARG;
    if (a->h0 && a->h_last && a->h0 != a->h_last && overlaps(span(a->h0, nst), hl))
        return SS_ERR_INVALID_ARG;
    ssh::SsdParams p{a->batch, a->heads, a->headdim, a->dstate, a->seqlen, a->in_dtype,
                     a->out_dtype, a->x, a->dt, a->A, a->B, a->C, a->D, a->dt_bias,
                     a->dt_softplus, a->h0, a->y, a->h_last, ctx->d_err, ctx->wait_limit};
    // AUTO takes the tensor-memory kernel wherever it applies (the faster one),
    // else the mma.sync kernel
    const bool tc = ctx->ssd_path == SS_SSD_PATH_TCGEN05 ||
                    (ctx->ssd_path == SS_SSD_PATH_AUTO && ssh::ssd_tc_supported(p));
    if (tc ? !ssh::ssd_tc_supported(p) : !ssh::ssd_supported(p)) return SS_ERR_UNSUPPORTED;
    if (set_device(ctx) != SS_OK) return SS_ERR_CUDA;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int rc = tc ? ssh::launch_ssd_tc(p, st) : ssh::launch_ssd(p, st);
    ctx->last_variant = tc ? 1 : 0;
    ctx->last_launches = rc == SS_OK ? 1 : 0;
    return rc;
}

int ss_conv1d_fwd(ss_ctx *ctx, const ss_conv1d_args *a, ss_stream_t stream) {
    if (!ctx || !a) return SS_ERR_INVALID_ARG;
    if (a->batch < 1 || a->dim < 1 || a->seqlen < 0) return SS_ERR_INVALID_ARG;
    if (!valid_dtype(a->in_dtype) || !valid_dtype(a->out_dtype)) return SS_ERR_INVALID_ARG;
    if (a->width < 2 || a->width > 4) return SS_ERR_UNSUPPORTED;
    if ((long long)a->batch * a->dim > (1LL << 40) || a->seqlen >= (1LL << 40))
        return SS_ERR_INVALID_ARG;
    if (!a->weight || (a->seqlen > 0 && (!a->x || !a->out))) return SS_ERR_INVALID_ARG;
    const void *ptrs[] = {a->x, a->weight, a->bias, a->init_state, a->out, a->final_state};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return SS_ERR_INVALID_ARG;
    const size_t rows = (size_t)a->batch * a->dim;
    const size_t n = rows * (size_t)a->seqlen;
    const size_t esz = a->in_dtype == SS_BF16 ? 2 : 4, osz = a->out_dtype == SS_BF16 ? 2 : 4;
    const size_t st_b = rows * (size_t)(a->width - 1) * 4;
    const Span x = span(a->x, n * esz), out = span(a->out, n * osz);
    const Span init = span(a->init_state, a->init_state ? st_b : 0);
    const Span fin = span(a->final_state, a->final_state ? st_b : 0);
    const Span params[] = {span(a->weight, (size_t)a->dim * a->width * 4),
                           span(a->bias, a->bias ? (size_t)a->dim * 4 : 0)};
    if (overlaps(out, x) || overlaps(out, init)) return SS_ERR_INVALID_ARG;
    if (overlaps(fin, init) || overlaps(fin, x) || overlaps(fin, out)) return SS_ERR_INVALID_ARG;
    for (const Span &s : params)
        if (overlaps(out, s) || overlaps(fin, s)) return SS_ERR_INVALID_ARG;
    if (set_device(ctx) != SS_OK) return SS_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    ctx->last_variant = 0;
    if (a->seqlen == 0) {
        ctx->last_launches = 0;
        if (!a->final_state) return SS_OK;
        const cudaError_t e = a->init_state
                                  ? cudaMemcpyAsync(a->final_state, a->init_state, st_b,
                                                    cudaMemcpyDeviceToDevice, st)
                                  : cudaMemsetAsync(a->final_state, 0, st_b, st);
        return e == cudaSuccess ? SS_OK : SS_ERR_CUDA;
    }
    ssh::ConvParams p{a->batch, a->dim, a->width, a->seqlen, a->in_dtype, a->out_dtype, a->x,
                      a->weight, a->bias, a->init_state, a->silu, a->out, a->final_state};
    const int rc = ssh::launch_conv1d(p, st);
    ctx->last_launches = rc == SS_OK ? 1 : 0;
    return rc;
}

int ss_conv1d_update(ss_ctx *ctx, const ss_conv1d_update_args *a, ss_stream_t stream) {
    if (!ctx || !a) return SS_ERR_INVALID_ARG;
    if (a->batch < 1 || a->dim < 1) return SS_ERR_INVALID_ARG;
    if (!valid_dtype(a->in_dtype) || !valid_dtype(a->out_dtype)) return SS_ERR_INVALID_ARG;
    if (a->width < 2 || a->width > 4) return SS_ERR_UNSUPPORTED;
    if ((long long)a->batch * a->dim > (1LL << 40)) return SS_ERR_INVALID_ARG;
    if (!a->state || !a->x || !a->weight || !a->out) return SS_ERR_INVALID_ARG;
    const void *ptrs[] = {a->state, a->x, a->weight, a->bias, a->out};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return SS_ERR_INVALID_ARG;
    const size_t rows = (size_t)a->batch * a->dim;
    const size_t esz = a->in_dtype == SS_BF16 ? 2 : 4, osz = a->out_dtype == SS_BF16 ? 2 : 4;
    const Span out = span(a->out, rows * osz);
    const Span stt = span(a->state, rows * (size_t)(a->width - 1) * 4);
    const Span ins[] = {stt, span(a->x, rows * esz),
                        span(a->weight, (size_t)a->dim * a->width * 4),
                        span(a->bias, a->bias ? (size_t)a->dim * 4 : 0)};
    for (const Span &s : ins)
        if (overlaps(out, s)) return SS_ERR_INVALID_ARG;
    for (size_t i = 1; i < sizeof(ins) / sizeof(ins[0]); ++i)
        if (overlaps(stt, ins[i])) return SS_ERR_INVALID_ARG;
    if (set_device(ctx) != SS_OK) return SS_ERR_CUDA;
    ssh::ConvUpdateParams p{a->batch, a->dim, a->width, a->in_dtype, a->out_dtype, a->state,
                            a->x, a->weight, a->bias, a->silu, a->out};
    const int rc = ssh::launch_conv1d_update(p, reinterpret_cast<cudaStream_t>(stream));
    ctx->last_variant = 0;
    ctx->last_launches = rc == SS_OK ? 1 : 0;
    return rc;
}

}  // extern "C"
