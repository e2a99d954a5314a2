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

template <typename Tin, typename Tout, int N, int TPR>
__global__ void __launch_bounds__(256) state_update_kernel(const ssh::UpdateParams p) {
    constexpr int NS = N / TPR;
    const long long rows = (long long)p.batch * p.dim;
    const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long row_raw = g / TPR;
    const int q = (int)(g % TPR);
    const bool ok = row_raw < rows;
    // threads past the end keep running on row 0 so the shuffles stay full-warp
    const long long row = ok ? row_raw : 0;
    // 32-bit division (the launcher keeps batch * dim * TPR below 2^31)
    const uint32_t bq = (uint32_t)row / (uint32_t)p.dim;
    const int b = (int)bq, d = (int)((uint32_t)row - bq * (uint32_t)p.dim);

    float st[NS], A[NS], Bv[NS], Cv[NS];
    ld_f32<NS>(p.state + row * N + q * NS, st);
    const float xv = to_f32(static_cast<const Tin *>(p.x)[row]);
    const float xr = to_f32(static_cast<const Tin *>(p.dt)[row]) + (p.bias ? p.bias[d] : 0.f);
    ld_f32<NS>(p.A + (long long)d * N + q * NS, A);
    ld_in<NS>(static_cast<const Tin *>(p.B) + (long long)b * N + q * NS, Bv);
    ld_in<NS>(static_cast<const Tin *>(p.C) + (long long)b * N + q * NS, Cv);
    const float dt = p.softplus ? softplus1(xr) : xr;
    const float dtx = dt * xv;
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        if (p.zoh) {
            float e;
            const float f = zoh_step(dt, A[i], &e);
            st[i] = fmaf(e, st[i], f * xv * Bv[i]);
        } else {
            const float e = ex2(dt * (A[i] * kLog2e));
            st[i] = fmaf(e, st[i], dtx * Bv[i]);
        }
        acc = fmaf(Cv[i], st[i], acc);
    }
#pragma unroll
    for (int m = TPR / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (!ok) return;
    st_f32<NS>(p.state + row * N + q * NS, st);
    if (q == 0) {
        float o = fmaf(p.D ? p.D[d] : 0.f, xv, acc);
        if (p.z) o *= gate(to_f32(static_cast<const Tin *>(p.z)[row]), Tin());
        store_out(static_cast<Tout *>(p.y) + row, o);
    }
}

template <typename Tin, typename Tout>
int launch_n(const ssh::UpdateParams &p, cudaStream_t st) {
    const long long rows = (long long)p.batch * p.dim;
    if (rows * 16 >= (1LL << 31)) return SS_ERR_UNSUPPORTED;
    auto go = [&](auto kern, int tpr) {
        const long long threads = rows * tpr;
        kern<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(p);
    };
    switch (p.dstate) {
        case 1: go(state_update_kernel<Tin, Tout, 1, 1>, 1); break;
        case 2: go(state_update_kernel<Tin, Tout, 2, 1>, 1); break;
        case 4: go(state_update_kernel<Tin, Tout, 4, 1>, 1); break;
        case 8: go(state_update_kernel<Tin, Tout, 8, 2>, 2); break;
        case 16: go(state_update_kernel<Tin, Tout, 16, SS_UPD_TPR16>, SS_UPD_TPR16); break;
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
