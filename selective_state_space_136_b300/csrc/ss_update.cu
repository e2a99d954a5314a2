// Single-token selective state update (decoding).
//
// Decoding keeps one fixed dim x N fp32 state per sequence and advances it by
// one token per call, O(1) work per token ("Mamba: Linear-Time Sequence
// Modeling with Selective State Spaces", section "Questions", on generation
// without a KV cache). The arithmetic is one step of the scan recurrence.
//
// Layout of the work: TPR threads per row (b, d), each owning NS = N / TPR
// consecutive states, read and written as 16-byte vectors (a warp's state
// accesses are contiguous). Four threads per row for N = 16 measured fastest:
// fewer threads per row keep fewer loads in flight, more repeat the per-row
// work (dt, softplus) in too many threads. The output sum over states is
// finished with xor-shuffles inside the row's thread group. Bandwidth-bound: the state
// is read and written once (8 B per state element); x, dt, z, y are 2-4 B per
// row and B, C, A, D, bias are shared by many rows (cache hits).
#include "ss_common.cuh"
#include "ss_internal.h"

#ifndef SS_UPD_TPR16
#define SS_UPD_TPR16 4  // threads per row for dstate 16
#endif
#ifndef SS_UPD_RPT
#define SS_UPD_RPT 1  // rows per thread group (2 measured the same, 4 slower)
#endif

namespace {

using namespace ssk;

// NS consecutive fp32 values, 16-byte vectors where NS allows it
template <int NS>
__device__ __forceinline__ void ld_f32(const float *p, float *v) {
    if constexpr (NS % 4 == 0) {
#pragma unroll
        for (int i = 0; i < NS; i += 4) {
            const float4 t = *reinterpret_cast<const float4 *>(p + i);
            v[i] = t.x, v[i + 1] = t.y, v[i + 2] = t.z, v[i + 3] = t.w;
        }
    } else if constexpr (NS == 2) {
        const float2 t = *reinterpret_cast<const float2 *>(p);
        v[0] = t.x, v[1] = t.y;
    } else {
        v[0] = p[0];
    }
}
template <int NS>
__device__ __forceinline__ void st_f32(float *p, const float *v) {
    if constexpr (NS % 4 == 0) {
#pragma unroll
        for (int i = 0; i < NS; i += 4)
            *reinterpret_cast<float4 *>(p + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else if constexpr (NS == 2) {
        *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
    } else {
        p[0] = v[0];
    }
}
// NS consecutive input values (fp32 or bf16) widened to fp32
template <int NS>
__device__ __forceinline__ void ld_in(const float *p, float *v) { ld_f32<NS>(p, v); }
template <int NS>
__device__ __forceinline__ void ld_in(const uint16_t *p, float *v) {
    if constexpr (NS % 8 == 0) {
#pragma unroll
        for (int i = 0; i < NS; i += 8) {
            const uint4 t = *reinterpret_cast<const uint4 *>(p + i);
            const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) v[i + 2 * k] = bf16lo(w[k]), v[i + 2 * k + 1] = bf16hi(w[k]);
        }
    } else if constexpr (NS == 4) {
        const uint2 t = *reinterpret_cast<const uint2 *>(p);
        v[0] = bf16lo(t.x), v[1] = bf16hi(t.x), v[2] = bf16lo(t.y), v[3] = bf16hi(t.y);
    } else {
#pragma unroll
        for (int i = 0; i < NS; ++i) v[i] = to_f32(p[i]);
    }
}

__device__ __forceinline__ float gate(float z, float) { return silu(z); }
__device__ __forceinline__ float gate(float z, uint16_t) {
    // bf16 z: silu through tanh.approx, as in the scan kernel
    const f2 g = silu2_tanh(mk2(z, z));
    return g.x;
}

template <typename Tin, typename Tout, int N, int TPR, int RPT>
__global__ void __launch_bounds__(256) state_update_kernel(const ssh::UpdateParams p) {
    constexpr int NS = N / TPR;
    const uint32_t rows = (uint32_t)p.batch * (uint32_t)p.dim;
    const uint32_t g = blockIdx.x * blockDim.x + threadIdx.x;
    const int q = (int)(g % TPR);
    // RPT rows per thread group, one grid-width of groups apart, so every
    // warp access stays contiguous; all loads of all RPT rows are issued
    // before any arithmetic
    const uint32_t span = gridDim.x * blockDim.x / TPR;
    float st[RPT][NS], A[RPT][NS], Bv[RPT][NS], Cv[RPT][NS], xv[RPT], xr[RPT], zv[RPT], Dd[RPT];
    uint32_t row[RPT];
    bool ok[RPT];
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        const uint32_t rr = g / TPR + k * span;
        ok[k] = rr < rows;
        // threads past the end keep running on row 0 so the shuffles stay full-warp
        row[k] = ok[k] ? rr : 0u;
        const uint32_t bq = row[k] / (uint32_t)p.dim;
        const int b = (int)bq, d = (int)(row[k] - bq * (uint32_t)p.dim);
        ld_f32<NS>(p.state + (long long)row[k] * N + q * NS, st[k]);
        xv[k] = to_f32(static_cast<const Tin *>(p.x)[row[k]]);
        xr[k] = to_f32(static_cast<const Tin *>(p.dt)[row[k]]) + (p.bias ? p.bias[d] : 0.f);
        zv[k] = p.z ? to_f32(static_cast<const Tin *>(p.z)[row[k]]) : 0.f;
        Dd[k] = p.D ? p.D[d] : 0.f;
        ld_f32<NS>(p.A + (long long)d * N + q * NS, A[k]);
        ld_in<NS>(static_cast<const Tin *>(p.B) + (long long)b * N + q * NS, Bv[k]);
        ld_in<NS>(static_cast<const Tin *>(p.C) + (long long)b * N + q * NS, Cv[k]);
    }
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        const float dt = p.softplus ? softplus1(xr[k]) : xr[k];
        const float dtx = dt * xv[k];
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < NS; ++i) {
            if (p.zoh) {
                float e;
                const float f = zoh_step(dt, A[k][i], &e);
                st[k][i] = fmaf(e, st[k][i], f * xv[k] * Bv[k][i]);
            } else {
                const float e = ex2(dt * (A[k][i] * kLog2e));
                st[k][i] = fmaf(e, st[k][i], dtx * Bv[k][i]);
            }
            acc = fmaf(Cv[k][i], st[k][i], acc);
        }
#pragma unroll
        for (int m = TPR / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
        if (ok[k]) {
            st_f32<NS>(p.state + (long long)row[k] * N + q * NS, st[k]);
            if (q == 0) {
                float o = fmaf(Dd[k], xv[k], acc);
                if (p.z) o *= gate(zv[k], Tin());
                store_out(static_cast<Tout *>(p.y) + row[k], o);
            }
        }
    }
}

template <typename Tin, typename Tout>
int launch_n(const ssh::UpdateParams &p, cudaStream_t st) {
    const long long rows = (long long)p.batch * p.dim;
    if (rows * 16 >= (1LL << 31)) return SS_ERR_UNSUPPORTED;
    constexpr int R = SS_UPD_RPT;
    auto go = [&](auto kern, int tpr) {
        const long long groups = (rows + R - 1) / R;
        kern<<<(unsigned)((groups * tpr + 255) / 256), 256, 0, st>>>(p);
    };
    switch (p.dstate) {
        case 1: go(state_update_kernel<Tin, Tout, 1, 1, R>, 1); break;
        case 2: go(state_update_kernel<Tin, Tout, 2, 1, R>, 1); break;
        case 4: go(state_update_kernel<Tin, Tout, 4, 1, R>, 1); break;
        case 8: go(state_update_kernel<Tin, Tout, 8, 2, R>, 2); break;
        case 16: go(state_update_kernel<Tin, Tout, 16, SS_UPD_TPR16, R>, SS_UPD_TPR16); break;
        default: return SS_ERR_UNSUPPORTED;
    }
    return cudaPeekAtLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

}  // namespace

int ssh::launch_update(const ssh::UpdateParams &p, cudaStream_t st) {
    const bool ib = p.in_dtype == SS_BF16, ob = p.out_dtype == SS_BF16;
    if (ib && ob) return launch_n<uint16_t, uint16_t>(p, st);
    if (ib) return launch_n<uint16_t, float>(p, st);
    if (ob) return launch_n<float, uint16_t>(p, st);
    return launch_n<float, float>(p, st);
}
