// Host-side internals of the ss_scan library: the context and the launchers
// each kernel file provides. Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ss_scan.h"

struct ss_ctx {
    int device = 0;
    int sm_count = 0;
    int max_smem_optin = 0;
    int *d_err = nullptr;          // device error word (one int)
    void *scratch = nullptr;       // chunk-carry scratch, grown on demand
    size_t scratch_bytes = 0;
    int variant = SS_VARIANT_AUTO;
    int segments = 0;              // 0 = choose automatically
    int rows_tpr = 0;              // threads per row for the rows kernel (0 = auto)
    int warps_per_sm = 8;          // persistent warps per SM for the chained kernel
    unsigned long long epoch = 0;  // calls that used the chained scratch
    uint32_t wait_limit = 1u << 22;  // polls before a device wait gives up
    int drop_tile = -1;            // test hook: a tile whose loads are never issued
    int zoh = 0;                   // SS_DISC_ZOH: exact zero-order-hold input matrix
    int ssd_path = SS_SSD_PATH_AUTO;
    void *bwd_scratch = nullptr;   // backward checkpoints, grown on demand
    size_t bwd_scratch_bytes = 0;
    int last_variant = 0;
    int last_launches = 0;
};

namespace ssh {

// Parameters common to the scan kernels (device pointers).
struct ScanParams {
    int batch, dim, dstate;
    long long seqlen;
    int in_dtype, out_dtype;
    const void *u, *delta, *z;
    const float *A;
    const void *B, *C;
    const float *D, *bias;
    int softplus;
    const float *h0;
    void *y;
    float *h_last;
    int *err;
    uint32_t wait_limit;
    int drop_tile;
    int zoh;  // exact zero-order-hold input matrix (one-thread-per-row kernels only)
    // causal conv1d fused in front of the scan (chained pair-row kernel only):
    // with conv_width > 0, `u` holds the convolution's input x and the scan's
    // u is silu(conv(x)) (conv(x) when conv_silu == 0), formed in registers
    int conv_width;           // 0 (no convolution) or 2..4
    int conv_silu;
    const float *conv_w;      // (dim, conv_width)
    const float *conv_b;      // (dim) or null
    const float *conv_init;   // (batch, dim, conv_width - 1) or null (zeros)
    float *conv_state;        // (batch, dim, conv_width - 1) out, or null
    void *u_out;              // (batch, dim, seqlen) in in_dtype out, or null
};

int launch_simple(const ScanParams &p, cudaStream_t st);
// tpr: threads per row (1, 2 or 4 for dstate 16; ignored otherwise).
int launch_rows(const ScanParams &p, int tpr, int max_smem_optin, cudaStream_t st);
// True when the rows kernel can take these arguments (TMA constraints).
bool rows_supported(const ScanParams &p);
// One thread per row, all states in registers (the default for staged shapes).
int launch_seq(const ScanParams &p, int max_smem_optin, cudaStream_t st);
bool seq_supported(const ScanParams &p);

// Chained pair-row variant (dstate 16): scratch it needs and its launcher.
struct PairWork {
    float *bc;                       // packed fp32 B/C, pair_bc_bytes()
    float *carry;                    // pair_carry_bytes()
    unsigned long long *flags;       // one per row block, zeroed once at allocation
    unsigned long long *counter;     // two work counters, reset by the first kernel of a call
    float *hagg;                     // chunked only: pair_agg_bytes() (end states, then carries)
    float *sdt;                      //   and the summed dt per (row block, segment)
    bool chunked;                    // aggregate + combine + output instead of one chained pass
    unsigned long long epoch;        // strictly increasing per call on this scratch
    int n_seg;                       // time segments per row block
    int warps_per_sm;                // persistent warps per SM (0 = as many as fit)
    int sm_count;
};
size_t pair_bc_bytes(const ScanParams &p);
size_t pair_carry_bytes(const ScanParams &p);
int pair_segments(const ScanParams &p, int requested);  // actual count for a request
size_t pair_agg_bytes(const ScanParams &p, int n_seg);
int pair_row_blocks(const ScanParams &p);
bool pair_supported(const ScanParams &p);
int launch_pair(const ScanParams &p, const PairWork &w, cudaStream_t st);

struct UpdateParams {
    int batch, dim, dstate;
    int in_dtype, out_dtype;
    float *state;
    const void *x, *dt, *z;
    const float *A;
    const void *B, *C;
    const float *D, *bias;
    int softplus;
    void *y;
    int zoh;
};
int launch_update(const UpdateParams &p, cudaStream_t st);

// backward pass (ss_bwd.cu)
struct BwdParams {
    int batch, dim, dstate;
    long long seqlen;
    int in_dtype;
    const void *u, *delta, *z;
    const float *A;
    const void *B, *C;
    const float *D, *bias;
    int softplus;
    const float *h0;
    const float *dy, *dh_last;
    float *du, *ddelta, *dz, *dA, *dB, *dC, *dD, *dbias, *dh0;
    float *ckpt;  // scratch: bwd_ckpt_bytes
    int zoh;      // exact zero-order-hold input matrix (the scalar backward kernel)
};
size_t bwd_ckpt_bytes(const BwdParams &p);
bool bwd_supported(const BwdParams &p);
int launch_bwd(const BwdParams &p, cudaStream_t st);

// Mamba-2 SSD forward (ss_ssd.cu)
struct SsdParams {
    int batch, heads, headdim, dstate;
    long long seqlen;
    int in_dtype, out_dtype;
    const void *x, *dt;
    const float *A;
    const void *B, *C;
    const float *D, *dt_bias;
    int softplus;
    const float *h0;
    void *y;
    float *h_last;
    int *err;             // device error word (SS_ERR_TIMEOUT when a wait gives up)
    uint32_t wait_limit;  // polls before a device-side wait gives up
};
bool ssd_supported(const SsdParams &p);
int launch_ssd(const SsdParams &p, cudaStream_t st);
bool ssd_tc_supported(const SsdParams &p);
int launch_ssd_tc(const SsdParams &p, cudaStream_t st);

// causal depthwise conv1d (ss_conv.cu)
struct ConvParams {
    int batch, dim, width;
    long long seqlen;
    int in_dtype, out_dtype;
    const void *x;
    const float *w, *bias, *init_state;
    int silu;
    void *out;
    float *final_state;
};
int launch_conv1d(const ConvParams &p, cudaStream_t st);
struct ConvUpdateParams {
    int batch, dim, width;
    int in_dtype, out_dtype;
    float *state;
    const void *x;
    const float *w, *bias;
    int silu;
    void *out;
};
int launch_conv1d_update(const ConvUpdateParams &p, cudaStream_t st);

}  // namespace ssh
