// Device helpers shared by the ss_scan kernels (sm_103a).
//
// Inline PTX only for what the C++ front end cannot express: the MUFU base-2
// exponential, packed fp32x2 arithmetic (sm_100+), mbarriers and TMA tensor
// copies. Every spin-wait is bounded and reports through the error word.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ss_scan.h"

namespace ssk {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- element io
// Inputs arrive as fp32 or as bf16 bit patterns; both widen exactly to fp32.
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(uint16_t v) { return __uint_as_float(uint32_t(v) << 16); }
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void store_out(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_out(uint16_t *p, float v) {
    *p = __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// ---------------------------------------------------------------- arithmetic
// 2^x on the MUFU unit; inputs far below -126 flush to zero.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// softplus(x) = log(1 + e^x). Above 20 the correction e^-x < 2.1e-9 is
// below half an ulp of x, so x itself is the fp32 answer.
__device__ __forceinline__ float softplus(float x) {
    return x > 20.f ? x : log1pf(ex2(x * kLog2e));
}

// silu(z) = z * sigmoid(z) = z / (1 + e^-z). For z << 0 the denominator
// overflows to +inf and the quotient is -0, the right limit.
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.f + ex2(-z * kLog2e)); }

// Exact zero-order hold for one state ("Mamba: Linear-Time Sequence Modeling
// with Selective State Spaces", section "Method", diagonal A): the decay
// e = exp(dt a) and the input factor (exp(dt a) - 1) / a (dt at a = 0), with
// exp(dt a) - 1 from expm1f so that small dt a keeps its precision.
__device__ __forceinline__ float zoh_step(float dt, float a, float *e) {
    const float em1 = expm1f(dt * a);
    *e = 1.f + em1;
    return a != 0.f ? em1 / a : dt;
}

// Packed fp32x2 arithmetic (two lanes per instruction on sm_100+).
struct f2 {
    float x, y;
};
__device__ __forceinline__ f2 mk2(float a, float b) { return f2{a, b}; }
__device__ __forceinline__ f2 fmul2(f2 a, f2 b) {
    f2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ f2 ffma2(f2 a, f2 b, f2 c) {
    f2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ f2 fadd2(f2 a, f2 b) {
    f2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log1p(w) / w on [0, 1]: degree-7 polynomial fitted for minimax relative
// error (weighted Chebyshev least squares with Lawson refinement; see
// fit_log1p_poly.py). w * P(w) is within 3.5e-7 relative of log1p(w).
__device__ __forceinline__ f2 log1p_unit2(f2 w) {
    const float c0 = 9.999998212e-01f, c1 = -4.999740422e-01f, c2 = 3.327547908e-01f,
                c3 = -2.449546158e-01f, c4 = 1.774523854e-01f, c5 = -1.076816618e-01f,
                c6 = 4.408959672e-02f, c7 = -8.539198898e-03f;
    f2 p = mk2(c7, c7);
    p = ffma2(p, w, mk2(c6, c6));
    p = ffma2(p, w, mk2(c5, c5));
    p = ffma2(p, w, mk2(c4, c4));
    p = ffma2(p, w, mk2(c3, c3));
    p = ffma2(p, w, mk2(c2, c2));
    p = ffma2(p, w, mk2(c1, c1));
    p = ffma2(p, w, mk2(c0, c0));
    return fmul2(p, w);
}

// log1p(w) on [0, 1] for a single value: w * P6(w), P6 a degree-6 polynomial
// fitted like the degree-7 one above (within 1.4e-6 relative of log1p(w)).
__device__ __forceinline__ float log1p_unit(float w) {
    float p = 1.414100733e-02f;
    p = fmaf(p, w, -6.640174985e-02f);
    p = fmaf(p, w, 1.492238194e-01f);
    p = fmaf(p, w, -2.350385785e-01f);
    p = fmaf(p, w, 3.310944736e-01f);
    p = fmaf(p, w, -4.998696446e-01f);
    p = fmaf(p, w, 9.999987483e-01f);
    return p * w;
}
// softplus(x) = max(x, 0) + log1p(2^(-|x| log2 e)), branch-free (see softplus2).
__device__ __forceinline__ float softplus1(float x) {
    return fmaxf(x, 0.f) + log1p_unit(ex2(fabsf(x) * -kLog2e));
}

// Degree-6 variant of log1p_unit2 (within 1.4e-6 relative of log1p(w)).
__device__ __forceinline__ f2 log1p_unit2_d6(f2 w) {
    f2 p = mk2(1.414100733e-02f, 1.414100733e-02f);
    p = ffma2(p, w, mk2(-6.640174985e-02f, -6.640174985e-02f));
    p = ffma2(p, w, mk2(1.492238194e-01f, 1.492238194e-01f));
    p = ffma2(p, w, mk2(-2.350385785e-01f, -2.350385785e-01f));
    p = ffma2(p, w, mk2(3.310944736e-01f, 3.310944736e-01f));
    p = ffma2(p, w, mk2(-4.998696446e-01f, -4.998696446e-01f));
    p = ffma2(p, w, mk2(9.999987483e-01f, 9.999987483e-01f));
    return fmul2(p, w);
}
// Degree-4 variant (within 5.7e-5 relative of log1p(w)): for bf16 inputs,
// whose own rounding (2^-9 relative) is far coarser.
__device__ __forceinline__ f2 log1p_unit2_d4(f2 w) {
    f2 p = mk2(4.134725779e-02f, 4.134725779e-02f);
    p = ffma2(p, w, mk2(-1.574271172e-01f, -1.574271172e-01f));
    p = ffma2(p, w, mk2(3.063008785e-01f, 3.063008785e-01f));
    p = ffma2(p, w, mk2(-4.969778061e-01f, -4.969778061e-01f));
    p = ffma2(p, w, mk2(9.999432564e-01f, 9.999432564e-01f));
    return fmul2(p, w);
}
__device__ __forceinline__ f2 softplus2_d4(f2 x) {
    const f2 t = fmul2(mk2(fabsf(x.x), fabsf(x.y)), mk2(-kLog2e, -kLog2e));
    const f2 w = mk2(ex2(t.x), ex2(t.y));
    return fadd2(mk2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)), log1p_unit2_d4(w));
}
__device__ __forceinline__ f2 softplus2_d6(f2 x) {
    const f2 t = fmul2(mk2(fabsf(x.x), fabsf(x.y)), mk2(-kLog2e, -kLog2e));
    const f2 w = mk2(ex2(t.x), ex2(t.y));
    return fadd2(mk2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)), log1p_unit2_d6(w));
}

// 256-bit (one 32-byte sector) per-thread global load / store (sm_100+).
struct u8v {
    uint32_t w[8];
};
__device__ __forceinline__ u8v ldg256(const void *p) {
    u8v v;
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]),
                   "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
                 : "l"(p));
    return v;
}
__device__ __forceinline__ void stg256(void *p, const float *f) {
    asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(f[0]),
                 "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7])
                 : "memory");
}

// softplus on a pair: max(x, 0) + log1p(2^(-|x| log2 e)). No branch: for
// x > ~17 the log1p term is below half an ulp of x; for x < -87 the
// exponential flushes to zero and so does the result.
__device__ __forceinline__ f2 softplus2(f2 x) {
    const f2 t = fmul2(mk2(fabsf(x.x), fabsf(x.y)), mk2(-kLog2e, -kLog2e));
    const f2 w = mk2(ex2(t.x), ex2(t.y));
    return fadd2(mk2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)), log1p_unit2(w));
}

// silu on a pair: z / (1 + 2^(-z log2 e)); z << 0 gives rcp(inf) = 0 -> -0.
// silu(z) = z sigmoid(z) = (z/2) (1 + tanh(z/2)): one MUFU.TANH per element.
// tanh.approx.f32 has a relative error near 2^-11, so this form serves the
// bf16-input path only (its tolerance is relative to max |y|).
__device__ __forceinline__ float tanh_approx(float x) {
    float r;
    asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ f2 silu2_tanh(f2 z) {
    const f2 hz = fmul2(z, mk2(0.5f, 0.5f));
    return ffma2(hz, mk2(tanh_approx(hz.x), tanh_approx(hz.y)), hz);
}
// The factor g of silu(x) = x * g(x), i.e. sigmoid(x): (1 + tanh(x/2)) / 2 on
// the tanh unit (bf16-input path), 1 / (1 + 2^(-x log2 e)) otherwise.
__device__ __forceinline__ f2 silu2_gate_tanh(f2 x) {
    const f2 hx = fmul2(x, mk2(0.5f, 0.5f));
    return ffma2(mk2(0.5f, 0.5f), mk2(tanh_approx(hx.x), tanh_approx(hx.y)), mk2(0.5f, 0.5f));
}
__device__ __forceinline__ f2 silu2_gate(f2 x) {
    const f2 t = fmul2(x, mk2(-kLog2e, -kLog2e));
    const f2 d = fadd2(mk2(ex2(t.x), ex2(t.y)), mk2(1.f, 1.f));
    return mk2(rcp_approx(d.x), rcp_approx(d.y));
}
__device__ __forceinline__ f2 silu2(f2 z) {
    const f2 t = fmul2(z, mk2(-kLog2e, -kLog2e));
    const f2 d = fadd2(mk2(ex2(t.x), ex2(t.y)), mk2(1.f, 1.f));
    return fmul2(z, mk2(rcp_approx(d.x), rcp_approx(d.y)));
}

// ---------------------------------------------------------------- cp.async
// 16-byte global -> shared copy; bytes beyond src_bytes (0..16) are zero-filled.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---------------------------------------------------------------- error word
__device__ __forceinline__ void set_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------- mbarrier / TMA
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for phase `parity` of `bar`, giving up after `limit` polls (each poll
// may block in hardware for a short while, then sleeps 256 ns).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (i >= 8) __nanosleep(256);
    }
    return false;
}
// 2D tiled TMA load global -> shared, completion signalled on `bar`.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace ssk
