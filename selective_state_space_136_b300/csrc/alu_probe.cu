// Throughput probes for the two compute units the selective scan leans on:
// the MUFU base-2 exponential and the FP32 FMA pipe (scalar and packed
// fp32x2). Measurement support for the benchmark's compute roofline; not part
// of the scan library.
//
// Each thread runs 8 independent dependency chains so the unit, not latency,
// limits the rate. The mixed probe runs the scan's own ratio, one ex2 to four
// FMA lane-ops (two packed FFMA2), on independent chains: its rate shows
// whether the two units overlap (time of the slower) or not (sum of both). The kernel also records SM cycles (clock64) against the
// global nanosecond timer in one thread, which gives the SM clock the probe
// actually ran at.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void ffma2(float &a0, float &a1, float b0, float b1, float c0,
                                      float c1) {
    asm volatile(
        "{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %3};\n\tmov.b64 rc, {%4, %5};\n\t"
        "fma.rn.f32x2 ra, ra, rb, rc;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int WHICH>
__global__ void __launch_bounds__(256) probe_kernel(float *sink, int iters,
                                                    unsigned long long *clk) {
    float a[8], c[16], acc[8][4] = {};
    const uint32_t fa = 0x3f803f80u + threadIdx.x, fb = 0x3f003f00u;  // bf16 pairs near 1 and 0.5
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = 0.25f + 0.01f * i + 1e-6f * threadIdx.x;
#pragma unroll
    for (int i = 0; i < 16; ++i) c[i] = 0.5f + 0.01f * i + 1e-6f * threadIdx.x;
    uint64_t c0 = 0, t0 = 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) c0 = clock64(), t0 = gtimer();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if constexpr (WHICH == 0) {
#pragma unroll
                for (int i = 0; i < 8; ++i) a[i] = ex2(-a[i]);
            } else if constexpr (WHICH == 1) {
#pragma unroll
                for (int i = 0; i < 8; ++i) a[i] = fmaf(a[i], 0.9990234375f, 0.0009765625f);
            } else if constexpr (WHICH == 4) {
#pragma unroll
                for (int i = 0; i < 8; ++i) mma_bf16(acc[i], fa, fa, fa, fa, fb, fb);
            } else if constexpr (WHICH == 2) {
#pragma unroll
                for (int i = 0; i < 8; i += 2)
                    ffma2(a[i], a[i + 1], 0.9990234375f, 0.9990234375f, 0.0009765625f,
                          0.0009765625f);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    a[i] = ex2(-a[i]);
                    ffma2(c[(2 * i) % 16], c[(2 * i + 1) % 16], 0.9990234375f, 0.9990234375f,
                          0.0009765625f, 0.0009765625f);
                    ffma2(c[(2 * i + 2) % 16], c[(2 * i + 3) % 16], 0.9990234375f,
                          0.9990234375f, 0.0009765625f, 0.0009765625f);
                }
            }
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        clk[0] = clock64() - c0;
        clk[1] = gtimer() - t0;
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += a[i];
#pragma unroll
    for (int i = 0; i < 16; ++i) s += c[i];
#pragma unroll
    for (int i = 0; i < 8; ++i) s += acc[i][0] + acc[i][1] + acc[i][2] + acc[i][3];
    if (s == 1234.5f) sink[threadIdx.x] = s;  // keeps the chains live
}

// The scan's inner step alone, with no global memory traffic: a lane pair
// holds R rows (R/2 of them its own) and 8 of the 16 states of each; per step
// the partner rows' dt and dt*u cross by xor-shuffle, B and C of the step come
// from shared memory as 4 broadcast 16-byte loads, and each row's output sum
// is finished with one more shuffle, as in the chained pair-row scan kernel.
// 16-step tiles are unrolled. Measures how many state elements per clock per
// SM the step sustains for a given number of warps per SM, i.e. what the
// arithmetic reaches at a shape's parallelism before any loads or stores.
template <int R>
__global__ void __launch_bounds__(256) scan_step_kernel(float *sink, int tiles,
                                                        unsigned long long *clk) {
    constexpr int O = R / 2, TL = 16;
    constexpr unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31, q = lane & 1;
    __shared__ float bcs[TL * 32];
    for (int i = threadIdx.x; i < TL * 32; i += blockDim.x) bcs[i] = 0.25f + 1e-3f * (i & 31);
    __syncthreads();
    float A2[R][8], h[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            A2[r][n] = -(8 * q + n + 1) * 1.4426950408889634f * (1.f + 0.01f * r);
            h[r][n] = 0.f;
        }
    const float dt0 = 0.01f + 1e-5f * threadIdx.x;
    float ysum = 0.f;
    uint64_t c0 = 0, t0 = 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) c0 = clock64(), t0 = gtimer();
    for (int it = 0; it < tiles; ++it) {
#pragma unroll
        for (int l = 0; l < TL; ++l) {
            float dts[R], dus[R];
#pragma unroll
            for (int i = 0; i < O; ++i) {
                dts[i] = (dt0 + 1e-3f * l + 1e-7f * it) * (1.f + 0.125f * i);
                dus[i] = 0.5f - 0.01f * l - 0.02f * i;
            }
#pragma unroll
            for (int i = 0; i < O; ++i) {
                dts[O + i] = __shfl_xor_sync(FULL, dts[i], 1);
                dus[O + i] = __shfl_xor_sync(FULL, dus[i], 1);
            }
            const float4 *bl = reinterpret_cast<const float4 *>(bcs + l * 32 + 8 * q);
            const float4 b0 = bl[0], b1 = bl[1], c0v = bl[4], c1 = bl[5];
            const float Bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
            const float Cv[8] = {c0v.x, c0v.y, c0v.z, c0v.w, c1.x, c1.y, c1.z, c1.w};
            float part[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                for (int n = 0; n < 8; n += 2) {
                    float2 hh = make_float2(h[r][n], h[r][n + 1]);
                    ffma2(hh.x, hh.y, ex2(dts[r] * A2[r][n]), ex2(dts[r] * A2[r][n + 1]),
                          dus[r] * Bv[n], dus[r] * Bv[n + 1]);
                    h[r][n] = hh.x, h[r][n + 1] = hh.y;
                    acc0 = fmaf(Cv[n], h[r][n], acc0);
                    acc1 = fmaf(Cv[n + 1], h[r][n + 1], acc1);
                }
                part[r] = acc0 + acc1;
            }
#pragma unroll
            for (int i = 0; i < O; ++i) ysum += part[i] + __shfl_xor_sync(FULL, part[O + i], 1);
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        clk[0] = clock64() - c0;
        clk[1] = gtimer() - t0;
    }
    float sacc = ysum;
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int n = 0; n < 8; ++n) sacc += h[r][n];
    if (sacc == 1234.5f) sink[threadIdx.x] = sacc;
}

}  // namespace

extern "C" {

// The scan's inner step (scan_step_kernel) with rows_per_lane in {2, 4} rows
// per lane pair and warps_per_sm resident warps (one wave): state elements per
// clock per SM, and the SM clock seen. Returns 0 or the CUDA error code.
int ss_probe_scan_step(int rows_per_lane, int warps_per_sm, int device, double *el_per_clk_sm,
                       double *sm_ghz) {
    if ((rows_per_lane != 2 && rows_per_lane != 4) || warps_per_sm < 1 || warps_per_sm > 32)
        return -1;
    cudaError_t e = cudaSetDevice(device);
    if (e != cudaSuccess) return (int)e;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    float *sink = nullptr;
    unsigned long long *clk = nullptr;
    cudaMalloc(&sink, 256 * sizeof(float));
    cudaMalloc(&clk, 2 * sizeof(unsigned long long));
    cudaStream_t st;
    cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    const int threads = warps_per_sm >= 8 ? 256 : 32 * warps_per_sm;
    const int blocks = sms * (warps_per_sm * 32 / threads);
    const int tiles = 1500;
    auto run = [&](int n) {
        if (rows_per_lane == 2) scan_step_kernel<2><<<blocks, threads, 0, st>>>(sink, n, clk);
        else scan_step_kernel<4><<<blocks, threads, 0, st>>>(sink, n, clk);
    };
    run(tiles / 8);
    cudaEventRecord(a, st);
    run(tiles);
    cudaEventRecord(b, st);
    e = cudaEventSynchronize(b);
    float ms = 0.f;
    unsigned long long hc[2] = {0, 0};
    if (e == cudaSuccess) {
        cudaEventElapsedTime(&ms, a, b);
        cudaMemcpy(hc, clk, sizeof(hc), cudaMemcpyDeviceToHost);
        const double g = hc[1] ? (double)hc[0] / (double)hc[1] : 0.0;
        const double elems = (double)blocks * threads * tiles * 16.0 * rows_per_lane * 8.0;
        if (sm_ghz) *sm_ghz = g;
        if (el_per_clk_sm) *el_per_clk_sm = g > 0 ? elems / (ms * 1e-3) / (g * 1e9) / sms : 0.0;
    }
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    cudaStreamDestroy(st);
    cudaFree(sink);
    cudaFree(clk);
    return (int)e;
}

// which: 0 = MUFU ex2, 1 = FFMA, 2 = packed FFMA2 (counted as 2 FMA each),
// 3 = mixed (counted in ex2: each ex2 comes with four FMA lane-ops),
// 4 = legacy tensor-core mma.sync m16n8k16 bf16 with fp32 accumulation (flops).
// Writes the sustained rate in operations per second and the SM clock in GHz
// seen by the probe. Returns 0 on success, the CUDA error code otherwise.
int ss_probe_alu_occ(int which, int device, int warps_per_sm, double *ops_per_s,
                     double *sm_ghz);

int ss_probe_alu(int which, int device, double *ops_per_s, double *sm_ghz) {
    return ss_probe_alu_occ(which, device, 64, ops_per_s, sm_ghz);
}

// The same probes with `warps_per_sm` warps resident per SM (blocks of up to
// 256 threads, one wave): what a scheduler sustains with few warps to pick from.
int ss_probe_alu_occ(int which, int device, int warps_per_sm, double *ops_per_s,
                     double *sm_ghz) {
    if (warps_per_sm < 1 || warps_per_sm > 64 || which < 0 || which > 4) return -1;
    cudaError_t e = cudaSetDevice(device);
    if (e != cudaSuccess) return (int)e;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    float *sink = nullptr;
    unsigned long long *clk = nullptr;
    cudaMalloc(&sink, 256 * sizeof(float));
    cudaMalloc(&clk, 2 * sizeof(unsigned long long));
    cudaStream_t st;
    cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    const int threads = warps_per_sm >= 8 ? 256 : 32 * warps_per_sm;
    const int blocks = sms * (warps_per_sm * 32 / threads);
    const int iters = which == 0 || which == 3 ? 2048 : 8192;
    auto run = [&](int n) {
        if (which == 0) probe_kernel<0><<<blocks, threads, 0, st>>>(sink, n, clk);
        else if (which == 1) probe_kernel<1><<<blocks, threads, 0, st>>>(sink, n, clk);
        else if (which == 2) probe_kernel<2><<<blocks, threads, 0, st>>>(sink, n, clk);
        else if (which == 3) probe_kernel<3><<<blocks, threads, 0, st>>>(sink, n, clk);
        else probe_kernel<4><<<blocks, threads, 0, st>>>(sink, n, clk);
    };
    run(iters / 8);  // warm-up
    cudaEventRecord(a, st);
    run(iters);
    cudaEventRecord(b, st);
    e = cudaEventSynchronize(b);
    float ms = 0.f;
    unsigned long long hc[2] = {0, 0};
    if (e == cudaSuccess) {
        cudaEventElapsedTime(&ms, a, b);
        cudaMemcpy(hc, clk, sizeof(hc), cudaMemcpyDeviceToHost);
        // 4 x 8 operations per thread and iteration; for the mma probe 4 x 8
        // m16n8k16 products of 4096 flops per warp and iteration
        const double ops = which == 4 ? (double)blocks * (threads / 32) * iters * 32.0 * 4096.0
                                      : (double)blocks * threads * iters * 32.0;
        if (ops_per_s) *ops_per_s = ops / (ms * 1e-3);
        if (sm_ghz) *sm_ghz = hc[1] ? (double)hc[0] / (double)hc[1] : 0.0;
    }
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    cudaStreamDestroy(st);
    cudaFree(sink);
    cudaFree(clk);
    return (int)e;
}

}  // extern "C"
