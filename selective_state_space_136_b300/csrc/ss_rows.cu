// Selective scan, staged rows variant (the main one-pass kernel).
//
// What it computes is the selective recurrence of "Mamba: Linear-Time
// Sequence Modeling with Selective State Spaces" (sections "Method" and "The
// Selection Mechanism (S6)") with the dt * B input term of the soft186.com
// article (section "动态参数化的状态空间"), fused as the page's section
// "Hardware-aware state expansion" asks: inputs go from device memory to
// on-chip memory once, the state lives only in registers, and only the
// contracted output y (and the final state) is written back.
//
// Work split. A CTA owns RPB consecutive channels d of one batch b and walks
// the whole time axis in tiles of TL steps. Each row (b, d) is served by TPR
// threads; thread q of a row owns states n in [q*NS, (q+1)*NS), NS = N/TPR.
// Per tile:
//   1. TMA brings u, delta, z (RPB x TL) and B, C (N x TL) of the tile into a
//      ring of S shared-memory stages; one mbarrier per stage.
//   2. Prologue: thread q of a row computes dt = softplus(delta + bias) and
//      dt*u for TL/TPR steps of its row into shared memory (each (row, step)
//      once); all threads widen B, C to fp32 and transpose them to [l][n] so
//      the inner loop reads each step's B, C as broadcast vectors.
//   3. Inner loop over the TL steps, fully unrolled: per state one multiply
//      dt * A*log2(e), one MUFU ex2, one multiply dt*u*B, one FMA for the
//      state, one FMA for the output partial; pairs of states use the packed
//      fp32x2 forms.
//   4. The TPR output partials of a row are summed through shared memory; the
//      thread owning each step adds D*u, multiplies by silu(z) and stores y
//      as contiguous vectors.
// Steps past the end of the sequence get dt = 0, which makes them exact
// no-ops on the state (exp(0) = 1, no input).
#include "ss_common.cuh"
#include "ss_internal.h"

#include <cudaTypedefs.h>

namespace {

using namespace ssk;

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <typename Tin, int N, int TPR, int RPB, int TL, int S>
struct Layout {
    static constexpr int ESZ = (int)sizeof(Tin);
    static constexpr int ROWT = RPB * TL * ESZ;   // one row-tensor tile
    static constexpr int BCT = N * TL * ESZ;      // one B or C tile
    static constexpr int OFF_U = 0;
    static constexpr int OFF_DL = align_up(ROWT, 128);
    static constexpr int OFF_Z = 2 * align_up(ROWT, 128);
    static constexpr int OFF_B = 3 * align_up(ROWT, 128);
    static constexpr int OFF_C = OFF_B + align_up(BCT, 128);
    static constexpr int STAGE = OFF_C + align_up(BCT, 128);
    static constexpr int BSTRIDE = N + 4;          // padded [l][n] rows of Bf, Cf
    static constexpr int OFF_BF = S * STAGE;
    static constexpr int BF_BYTES = align_up(TL * BSTRIDE * 4, 128);
    static constexpr int OFF_CF = OFF_BF + BF_BYTES;
    static constexpr int OFF_DTW = OFF_CF + BF_BYTES;  // [TL][RPB] (dt, dt*u)
    static constexpr int DTW_BYTES = TL * RPB * 8;
    static constexpr int YSTRIDE = TL + 4;              // padded partial rows
    static constexpr int OFF_YP = OFF_DTW + DTW_BYTES;
    static constexpr int YP_BYTES = TPR > 1 ? RPB * TPR * YSTRIDE * 4 : 0;
    static constexpr int OFF_BAR = align_up(OFF_YP + YP_BYTES, 8);
    static constexpr int TOTAL = OFF_BAR + S * 8 + 128;  // + slack to align the base
    static_assert(OFF_DL % 128 == 0 && OFF_Z % 128 == 0 && OFF_B % 128 == 0 &&
                      OFF_C % 128 == 0 && STAGE % 128 == 0,
                  "TMA destinations must be 128-byte aligned");
};

// Load V consecutive elements starting at shared address p (16-byte aligned
// for V * sizeof(T) >= 16) and widen to fp32.
template <int V>
__device__ __forceinline__ void lds_widen(const uint16_t *p, float *v) {
    if constexpr (V % 8 == 0) {
#pragma unroll
        for (int j = 0; j < V / 8; ++j) {
            const uint4 w = reinterpret_cast<const uint4 *>(p)[j];
            v[8 * j + 0] = bf16lo(w.x), v[8 * j + 1] = bf16hi(w.x);
            v[8 * j + 2] = bf16lo(w.y), v[8 * j + 3] = bf16hi(w.y);
            v[8 * j + 4] = bf16lo(w.z), v[8 * j + 5] = bf16hi(w.z);
            v[8 * j + 6] = bf16lo(w.w), v[8 * j + 7] = bf16hi(w.w);
        }
    } else if constexpr (V % 4 == 0) {
#pragma unroll
        for (int j = 0; j < V / 4; ++j) {
            const uint2 w = reinterpret_cast<const uint2 *>(p)[j];
            v[4 * j + 0] = bf16lo(w.x), v[4 * j + 1] = bf16hi(w.x);
            v[4 * j + 2] = bf16lo(w.y), v[4 * j + 3] = bf16hi(w.y);
        }
    } else {
#pragma unroll
        for (int j = 0; j < V; ++j) v[j] = to_f32(p[j]);
    }
}
template <int V>
__device__ __forceinline__ void lds_widen(const float *p, float *v) {
    if constexpr (V % 4 == 0) {
#pragma unroll
        for (int j = 0; j < V / 4; ++j) {
            const float4 w = reinterpret_cast<const float4 *>(p)[j];
            v[4 * j + 0] = w.x, v[4 * j + 1] = w.y, v[4 * j + 2] = w.z, v[4 * j + 3] = w.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < V; ++j) v[j] = p[j];
    }
}

// Read NS consecutive fp32 from shared memory (aligned to NS * 4 bytes, up to 16).
template <int NS>
__device__ __forceinline__ void lds_f32(const float *p, float *v) {
    if constexpr (NS % 4 == 0) {
#pragma unroll
        for (int j = 0; j < NS / 4; ++j) {
            const float4 w = reinterpret_cast<const float4 *>(p)[j];
            v[4 * j] = w.x, v[4 * j + 1] = w.y, v[4 * j + 2] = w.z, v[4 * j + 3] = w.w;
        }
    } else if constexpr (NS == 2) {
        const float2 w = *reinterpret_cast<const float2 *>(p);
        v[0] = w.x, v[1] = w.y;
    } else {
        v[0] = p[0];
    }
}

// Store V consecutive outputs to global memory; vectorised when the whole
// run is in range (the caller guarantees 16-byte alignment then).
template <int V>
__device__ __forceinline__ void store_run(float *dst, const float *v, int valid) {
    if (valid >= V && V % 4 == 0) {
#pragma unroll
        for (int j = 0; j < V / 4; ++j)
            reinterpret_cast<float4 *>(dst)[j] =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    } else {
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < valid) dst[j] = v[j];
    }
}
template <int V>
__device__ __forceinline__ void store_run(uint16_t *dst, const float *v, int valid) {
    if (valid >= V && V % 8 == 0) {
#pragma unroll
        for (int j = 0; j < V / 8; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[8 * j + 2 * k]));
                const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[8 * j + 2 * k + 1]));
                w[k] = lo | (hi << 16);
            }
            reinterpret_cast<uint4 *>(dst)[j] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < V; ++j)
            if (j < valid) store_out(dst + j, v[j]);
    }
}

template <typename Tin, typename Tout, int N, int TPR, int RPB, int TL, int S>
__global__ void __launch_bounds__(RPB *TPR)
    scan_rows_kernel(const __grid_constant__ CUtensorMap tm_u,
                     const __grid_constant__ CUtensorMap tm_dl,
                     const __grid_constant__ CUtensorMap tm_z,
                     const __grid_constant__ CUtensorMap tm_B,
                     const __grid_constant__ CUtensorMap tm_C, const ssh::ScanParams p) {
    using LY = Layout<Tin, N, TPR, RPB, TL, S>;
    constexpr int NS = N / TPR;   // states per thread
    constexpr int LP = TL / TPR;  // steps per thread in prologue/epilogue
    constexpr int NT = RPB * TPR;
    static_assert(N % TPR == 0 && TL % TPR == 0 && 32 % TPR == 0, "bad split");
    static_assert(NS % 2 == 0 || NS == 1, "states are processed in pairs");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + LY::OFF_BAR);
    float *Bf = reinterpret_cast<float *>(smem + LY::OFF_BF);
    float *Cf = reinterpret_cast<float *>(smem + LY::OFF_CF);
    float2 *dtw = reinterpret_cast<float2 *>(smem + LY::OFF_DTW);
    float *yps = reinterpret_cast<float *>(smem + LY::OFF_YP);

    const int tid = threadIdx.x;
    const int r = tid / TPR, q = tid % TPR;
    const int b = blockIdx.y;
    const int d = blockIdx.x * RPB + r;
    const bool row_ok = d < p.dim;
    const int dc = row_ok ? d : p.dim - 1;
    const long long row = (long long)b * p.dim + d;
    const int L = (int)p.seqlen;
    const int n_tiles = (L + TL - 1) / TL;
    const int row0 = b * p.dim + blockIdx.x * RPB;  // first TMA row of this CTA

    // per-thread constants: A * log2(e) for the owned states, the state itself
    f2 A2[(NS + 1) / 2], h[(NS + 1) / 2];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        const float a = p.A[(long long)dc * N + q * NS + i] * kLog2e;
        const float h0 = (p.h0 && row_ok) ? p.h0[row * N + q * NS + i] : 0.f;
        if (i & 1) A2[i / 2].y = a, h[i / 2].y = h0;
        else A2[i / 2].x = a, h[i / 2].x = h0;
    }
    const float bias = p.bias ? p.bias[dc] : 0.f;
    const float Dd = p.D ? p.D[dc] : 0.f;
    const bool has_z = p.z != nullptr;
    const uint32_t stage_bytes = (has_z ? 3u : 2u) * LY::ROWT + 2u * LY::BCT;

    auto issue = [&](int t) {
        if (t == p.drop_tile) return;  // test hook: leave this tile's barrier unarmed
        const int s = t % S;
        uint8_t *st = smem + s * LY::STAGE;
        mbar_expect_tx(&bar[s], stage_bytes);
        const int x = t * TL;
        tma_load_2d(st + LY::OFF_U, &tm_u, x, row0, &bar[s]);
        tma_load_2d(st + LY::OFF_DL, &tm_dl, x, row0, &bar[s]);
        if (has_z) tma_load_2d(st + LY::OFF_Z, &tm_z, x, row0, &bar[s]);
        tma_load_2d(st + LY::OFF_B, &tm_B, x, b * N, &bar[s]);
        tma_load_2d(st + LY::OFF_C, &tm_C, x, b * N, &bar[s]);
    };

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0)
        for (int t = 0; t < S && t < n_tiles; ++t) issue(t);

    for (int k = 0; k < n_tiles; ++k) {
        const int s = k % S;
        const bool ready = mbar_wait_bounded(&bar[s], (uint32_t)(k / S) & 1u, p.wait_limit);
        const uint8_t *st = smem + s * LY::STAGE;
        const Tin *su = reinterpret_cast<const Tin *>(st + LY::OFF_U);
        const Tin *sdl = reinterpret_cast<const Tin *>(st + LY::OFF_DL);
        const Tin *sz = reinterpret_cast<const Tin *>(st + LY::OFF_Z);
        const Tin *sB = reinterpret_cast<const Tin *>(st + LY::OFF_B);
        const Tin *sC = reinterpret_cast<const Tin *>(st + LY::OFF_C);
        const int l0 = k * TL;
        const int nvalid = min(TL, L - l0);

        // ---- prologue: dt and dt*u once per (row, step); B, C to fp32 [l][n]
        {
            float uv[LP], dv[LP];
            lds_widen<LP>(su + r * TL + q * LP, uv);
            lds_widen<LP>(sdl + r * TL + q * LP, dv);
#pragma unroll
            for (int i = 0; i < LP; ++i) {
                const int l = q * LP + i;
                const float x = dv[i] + bias;
                float dt = p.softplus ? softplus(x) : x;
                if (l >= nvalid) dt = 0.f;
                dtw[l * RPB + r] = make_float2(dt, dt * uv[i]);
            }
        }
        for (int i = tid; i < N * TL; i += NT) {
            const int n = i / TL, l = i % TL;
            Bf[l * LY::BSTRIDE + n] = to_f32(sB[i]);
            Cf[l * LY::BSTRIDE + n] = to_f32(sC[i]);
        }
        if (__syncthreads_or(!ready)) {
            // A load never arrived: record it, let the other in-flight loads
            // land (bounded), and leave.
            if (tid == 0) set_error(p.err, SS_ERR_TIMEOUT);
            for (int t = k + 1; t < k + S && t < n_tiles; ++t)
                if (t != p.drop_tile)
                    mbar_wait_bounded(&bar[t % S], (uint32_t)(t / S) & 1u, p.wait_limit);
            return;
        }

        // ---- inner loop over the tile's steps
        float yp[TL];
#pragma unroll
        for (int l = 0; l < TL; ++l) {
            const float2 dd = dtw[l * RPB + r];
            float bv[NS], cv[NS];
            lds_f32<NS>(Bf + l * LY::BSTRIDE + q * NS, bv);
            lds_f32<NS>(Cf + l * LY::BSTRIDE + q * NS, cv);
            if constexpr (NS == 1) {
                const float e = ex2(dd.x * A2[0].x);
                h[0].x = fmaf(e, h[0].x, dd.y * bv[0]);
                yp[l] = cv[0] * h[0].x;
            } else {
                const f2 dt2 = mk2(dd.x, dd.x), du2 = mk2(dd.y, dd.y);
                f2 acc = mk2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < NS / 2; ++j) {
                    const f2 t = fmul2(dt2, A2[j]);
                    const f2 e = mk2(ex2(t.x), ex2(t.y));
                    const f2 bu = fmul2(du2, mk2(bv[2 * j], bv[2 * j + 1]));
                    h[j] = ffma2(e, h[j], bu);
                    acc = j == 0 ? fmul2(mk2(cv[0], cv[1]), h[0])
                                 : ffma2(mk2(cv[2 * j], cv[2 * j + 1]), h[j], acc);
                }
                yp[l] = acc.x + acc.y;
            }
        }

        // ---- sum the TPR partials of each step; thread q keeps steps [q*LP, (q+1)*LP)
        float ys[LP];
        if constexpr (TPR == 1) {
#pragma unroll
            for (int i = 0; i < LP; ++i) ys[i] = yp[i];
        } else {
            float *mine = yps + (r * TPR + q) * LY::YSTRIDE;
#pragma unroll
            for (int j = 0; j < TL / 4; ++j)
                reinterpret_cast<float4 *>(mine)[j] =
                    make_float4(yp[4 * j], yp[4 * j + 1], yp[4 * j + 2], yp[4 * j + 3]);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < LP; ++i) ys[i] = 0.f;
#pragma unroll
            for (int t = 0; t < TPR; ++t) {
                float v[LP];
                lds_widen<LP>(yps + (r * TPR + t) * LY::YSTRIDE + q * LP, v);
#pragma unroll
                for (int i = 0; i < LP; ++i) ys[i] += v[i];
            }
        }

        // ---- epilogue: D skip, silu(z) gate, store y
        if (row_ok) {
            float uv[LP], zv[LP], o[LP];
            lds_widen<LP>(su + r * TL + q * LP, uv);
            if (has_z) lds_widen<LP>(sz + r * TL + q * LP, zv);
#pragma unroll
            for (int i = 0; i < LP; ++i) {
                float v = fmaf(Dd, uv[i], ys[i]);
                if (has_z) v *= silu(zv[i]);
                o[i] = v;
            }
            const int first = l0 + q * LP;
            Tout *dst = static_cast<Tout *>(p.y) + row * (long long)L + first;
            store_run<LP>(dst, o, nvalid - q * LP);
        }
        __syncthreads();
        if (tid == 0 && k + S < n_tiles) issue(k + S);
    }

    if (row_ok && p.h_last) {
#pragma unroll
        for (int i = 0; i < NS; ++i)
            p.h_last[row * N + q * NS + i] = (i & 1) ? h[i / 2].y : h[i / 2].x;
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 2D row-major view [outer][inner] with the given row pitch in bytes.
bool make_map(CUtensorMap *tm, const void *base, bool bf16, uint64_t inner, uint64_t outer,
              uint64_t pitch, uint32_t box_inner, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {pitch};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(tm, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename Tin, typename Tout, int N, int TPR, int RPB, int TL, int S>
int launch_cfg(const ssh::ScanParams &p, int max_smem, cudaStream_t st) {
    using LY = Layout<Tin, N, TPR, RPB, TL, S>;
    auto kern = scan_rows_kernel<Tin, Tout, N, TPR, RPB, TL, S>;
    if (LY::TOTAL > max_smem) return SS_ERR_UNSUPPORTED;
    static bool attr_set[64] = {false};  // per instantiation and device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SS_ERR_CUDA;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::TOTAL) !=
            cudaSuccess)
            return SS_ERR_CUDA;
        attr_set[dev] = true;
    }
    const bool bf = sizeof(Tin) == 2;
    const uint64_t L = (uint64_t)p.seqlen, rows = (uint64_t)p.batch * p.dim;
    const uint64_t pitch = L * sizeof(Tin);
    CUtensorMap tu, tdl, tz, tB, tC;
    if (!make_map(&tu, p.u, bf, L, rows, pitch, TL, RPB) ||
        !make_map(&tdl, p.delta, bf, L, rows, pitch, TL, RPB) ||
        !make_map(&tz, p.z ? p.z : p.u, bf, L, rows, pitch, TL, RPB) ||
        !make_map(&tB, p.B, bf, L, (uint64_t)p.batch * N, pitch, TL, N) ||
        !make_map(&tC, p.C, bf, L, (uint64_t)p.batch * N, pitch, TL, N))
        return SS_ERR_CUDA;
    const dim3 grid((unsigned)((p.dim + RPB - 1) / RPB), (unsigned)p.batch);
    kern<<<grid, RPB * TPR, LY::TOTAL, st>>>(tu, tdl, tz, tB, tC, p);
    return cudaPeekAtLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

template <typename Tin, typename Tout>
int launch_types(const ssh::ScanParams &p, int tpr, int max_smem, cudaStream_t st) {
    constexpr int S = 3;
    switch (p.dstate) {
        case 1: return launch_cfg<Tin, Tout, 1, 1, 128, 32, S>(p, max_smem, st);
        case 2: return launch_cfg<Tin, Tout, 2, 1, 128, 32, S>(p, max_smem, st);
        case 4: return launch_cfg<Tin, Tout, 4, 1, 128, 32, S>(p, max_smem, st);
        case 8: return launch_cfg<Tin, Tout, 8, 2, 64, 32, S>(p, max_smem, st);
        case 16:
            if (tpr == 1) return launch_cfg<Tin, Tout, 16, 1, 32, 16, S>(p, max_smem, st);
            if (tpr == 2) return launch_cfg<Tin, Tout, 16, 2, 32, 32, S>(p, max_smem, st);
            return launch_cfg<Tin, Tout, 16, 4, 32, 32, S>(p, max_smem, st);
        default: return SS_ERR_UNSUPPORTED;
    }
}

}  // namespace

bool ssh::rows_supported(const ssh::ScanParams &p) {
    const int esz = p.in_dtype == SS_BF16 ? 2 : 4;
    const int osz = p.out_dtype == SS_BF16 ? 2 : 4;
    if ((p.seqlen * esz) % 16 != 0 || (p.seqlen * osz) % 16 != 0) return false;
    if (p.seqlen >= (1LL << 31)) return false;
    if (!encode_fn()) return false;
    return true;
}

int ssh::launch_rows(const ssh::ScanParams &p, int tpr, int max_smem, cudaStream_t st) {
    const bool ib = p.in_dtype == SS_BF16, ob = p.out_dtype == SS_BF16;
    if (ib && ob) return launch_types<uint16_t, uint16_t>(p, tpr, max_smem, st);
    if (ib) return launch_types<uint16_t, float>(p, tpr, max_smem, st);
    if (ob) return launch_types<float, uint16_t>(p, tpr, max_smem, st);
    return launch_types<float, float>(p, tpr, max_smem, st);
}
