// Single-token selective state update (decoding).
//
// Decoding keeps one fixed dim x N fp32 state per sequence and advances it by
// one token per call, O(1) work per token ("Mamba: Linear-Time Sequence
// Modeling with Selective State Spaces", section "Questions", on generation
// without a KV cache). The arithmetic is one step of the scan recurrence.
//
// Layout of the work: TPR = dstate/4 threads per row (b, d) (one for
// dstate <= 4), each owning NS consecutive states, so a warp reads the state
// as contiguous 16-byte vectors. The output sum over states is finished with
// xor-shuffles inside the row's thread group. Purely bandwidth-bound: the
// state is read and written once (8 B per state element), everything else is
// per-row or per-batch.
#include "ss_common.cuh"
#include "ss_internal.h"

namespace {

using namespace ssk;

template <int NS>
struct VecF;
template <>
struct VecF<1> {
    static __device__ __forceinline__ void ld(const float *p, float *v) { v[0] = *p; }
    static __device__ __forceinline__ void st(float *p, const float *v) { *p = v[0]; }
};
template <>
struct VecF<2> {
    static __device__ __forceinline__ void ld(const float *p, float *v) {
        const float2 t = *reinterpret_cast<const float2 *>(p);
        v[0] = t.x, v[1] = t.y;
    }
    static __device__ __forceinline__ void st(float *p, const float *v) {
        *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
    }
};
template <>
struct VecF<4> {
    static __device__ __forceinline__ void ld(const float *p, float *v) {
        const float4 t = *reinterpret_cast<const float4 *>(p);
        v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
    }
    static __device__ __forceinline__ void st(float *p, const float *v) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};

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
    const int b = (int)(row / p.dim), d = (int)(row % p.dim);

    const float xv = to_f32(static_cast<const Tin *>(p.x)[row]);
    const float xr = to_f32(static_cast<const Tin *>(p.dt)[row]) + (p.bias ? p.bias[d] : 0.f);
    const float dt = p.softplus ? softplus(xr) : xr;
    const float dtx = dt * xv;

    float st[NS], A[NS];
    VecF<NS>::ld(p.state + row * N + q * NS, st);
    VecF<NS>::ld(p.A + (long long)d * N + q * NS, A);
    const Tin *Bb = static_cast<const Tin *>(p.B) + (long long)b * N + q * NS;
    const Tin *Cb = static_cast<const Tin *>(p.C) + (long long)b * N + q * NS;
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        const float e = ex2(dt * (A[i] * kLog2e));
        st[i] = fmaf(e, st[i], dtx * to_f32(Bb[i]));
        acc = fmaf(to_f32(Cb[i]), st[i], acc);
    }
#pragma unroll
    for (int m = TPR / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (!ok) return;
    VecF<NS>::st(p.state + row * N + q * NS, st);
    if (q == 0) {
        float o = fmaf(p.D ? p.D[d] : 0.f, xv, acc);
        if (p.z) o *= silu(to_f32(static_cast<const Tin *>(p.z)[row]));
        store_out(static_cast<Tout *>(p.y) + row, o);
    }
}

template <typename Tin, typename Tout>
int launch_n(const ssh::UpdateParams &p, cudaStream_t st) {
    const long long rows = (long long)p.batch * p.dim;
    auto go = [&](auto kern, int tpr) {
        const long long threads = rows * tpr;
        kern<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(p);
    };
    switch (p.dstate) {
        case 1: go(state_update_kernel<Tin, Tout, 1, 1>, 1); break;
        case 2: go(state_update_kernel<Tin, Tout, 2, 1>, 1); break;
        case 4: go(state_update_kernel<Tin, Tout, 4, 1>, 1); break;
        case 8: go(state_update_kernel<Tin, Tout, 8, 2>, 2); break;
        case 16: go(state_update_kernel<Tin, Tout, 16, 4>, 4); break;
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
