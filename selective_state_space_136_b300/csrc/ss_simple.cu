// Selective scan, plain variant: one thread per row (b, d) walks the time
// axis in order with its dstate fp32 states in registers. Plain global loads,
// no alignment needs beyond the element size. It serves shapes the staged
// kernels cannot take (seqlen not a multiple of 8, small problems).
//
// Per step (the recurrence of "Mamba: Linear-Time Sequence Modeling with
// Selective State Spaces", sections "Method" and "The Selection Mechanism
// (S6)"):  dt = softplus(delta + bias);  h_n = exp(dt A_n) h_n + dt u B_n;
//          y = (sum_n C_n h_n + D u) * silu(z).
#include "ss_common.cuh"
#include "ss_internal.h"

namespace {

using namespace ssk;

template <typename Tin, typename Tout, int N>
__global__ void __launch_bounds__(128) scan_simple_kernel(const ssh::ScanParams p) {
    const long long rows = (long long)p.batch * p.dim;
    const long long row = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= rows) return;
    const long long L = p.seqlen;
    const int b = (int)(row / p.dim), d = (int)(row % p.dim);
    float A2[N], h[N];
#pragma unroll
    for (int n = 0; n < N; ++n) {
        A2[n] = p.A[(long long)d * N + n] * kLog2e;
        h[n] = p.h0 ? p.h0[row * N + n] : 0.f;
    }
    const float bias = p.bias ? p.bias[d] : 0.f;
    const float Dd = p.D ? p.D[d] : 0.f;
    const Tin *u = static_cast<const Tin *>(p.u) + row * L;
    const Tin *dl = static_cast<const Tin *>(p.delta) + row * L;
    const Tin *z = p.z ? static_cast<const Tin *>(p.z) + row * L : nullptr;
    const Tin *Bm = static_cast<const Tin *>(p.B) + (long long)b * N * L;
    const Tin *Cm = static_cast<const Tin *>(p.C) + (long long)b * N * L;
    Tout *y = static_cast<Tout *>(p.y) + row * L;
    for (long long l = 0; l < L; ++l) {
        const float uv = to_f32(u[l]);
        const float x = to_f32(dl[l]) + bias;
        const float dt = p.softplus ? softplus(x) : x;
        const float dtu = dt * uv;
        float acc = 0.f;
#pragma unroll
        for (int n = 0; n < N; ++n) {
            const float Bv = to_f32(Bm[(long long)n * L + l]);
            if (p.zoh) {
                float e;
                const float f = zoh_step(dt, p.A[(long long)d * N + n], &e);
                h[n] = fmaf(e, h[n], f * uv * Bv);
            } else {
                const float e = ex2(dt * A2[n]);
                h[n] = fmaf(e, h[n], dtu * Bv);
            }
            acc = fmaf(to_f32(Cm[(long long)n * L + l]), h[n], acc);
        }
        acc = fmaf(Dd, uv, acc);
        if (z) acc *= silu(to_f32(z[l]));
        store_out(y + l, acc);
    }
    if (p.h_last) {
#pragma unroll
        for (int n = 0; n < N; ++n) p.h_last[row * N + n] = h[n];
    }
}

template <typename Tin, typename Tout>
int launch_n(const ssh::ScanParams &p, cudaStream_t st) {
    const long long rows = (long long)p.batch * p.dim;
    const dim3 block(128), grid((unsigned)((rows + 127) / 128));
    switch (p.dstate) {
        case 1: scan_simple_kernel<Tin, Tout, 1><<<grid, block, 0, st>>>(p); break;
        case 2: scan_simple_kernel<Tin, Tout, 2><<<grid, block, 0, st>>>(p); break;
        case 4: scan_simple_kernel<Tin, Tout, 4><<<grid, block, 0, st>>>(p); break;
        case 8: scan_simple_kernel<Tin, Tout, 8><<<grid, block, 0, st>>>(p); break;
        case 16: scan_simple_kernel<Tin, Tout, 16><<<grid, block, 0, st>>>(p); break;
        default: return SS_ERR_UNSUPPORTED;
    }
    return cudaPeekAtLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

}  // namespace

int ssh::launch_simple(const ssh::ScanParams &p, cudaStream_t st) {
    const bool ib = p.in_dtype == SS_BF16, ob = p.out_dtype == SS_BF16;
    if (ib && ob) return launch_n<uint16_t, uint16_t>(p, st);
    if (ib) return launch_n<uint16_t, float>(p, st);
    if (ob) return launch_n<float, uint16_t>(p, st);
    return launch_n<float, float>(p, st);
}
