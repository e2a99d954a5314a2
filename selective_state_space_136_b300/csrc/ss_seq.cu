// Selective scan, sequential-rows variant: one thread owns one row (b, d) and
// all of its dstate fp32 states, and walks the time axis in order.
//
// The arithmetic is the selective recurrence of "Mamba: Linear-Time Sequence
// Modeling with Selective State Spaces" (sections "Method" and "The Selection
// Mechanism (S6)") with the dt * B input term of the soft186.com article
// (section "动态参数化的状态空间"), fused as the Mamba page's section
// "Hardware-aware state expansion" describes: inputs cross from device memory
// to on-chip memory once, the state never leaves registers, and only the
// contracted output y (plus the final state) goes back.
//
// Why one thread per row: every per-(row, step) quantity (dt, dt*u, the D
// skip, the silu(z) gate) is then computed exactly once, in registers, and
// the sum over states needs no cross-thread reduction. Only B and C are
// shared, by all rows of a batch: they are the one thing staged for the whole
// CTA.
//
// Data movement per tile of TL steps:
//  - u, delta, z (private to a row): cp.async 16-byte chunks into a
//    [tensor][chunk][thread] ring, so each thread later reads its own chunks
//    with conflict-free 128-bit shared loads (a warp reads 512 contiguous
//    bytes). Chunks past the end of the sequence are zero-filled.
//  - B, C (shared by the CTA's rows): one TMA box each per tile into a ring
//    of mbarrier-tracked stages, then widened once to fp32 and transposed to
//    [step][n] so the inner loop reads each step's B and C as broadcast
//    vectors.
// Inner loop per step and pair of states (packed fp32x2 forms):
//    t = dt * A log2(e);  e = 2^t (MUFU);  bu = dt*u * B;  h = e * h + bu;
//    acc += C * h
// Steps past the end get dt = 0, an exact no-op on the state.
#include "ss_common.cuh"
#include "ss_internal.h"

#include <cudaTypedefs.h>

namespace {

using namespace ssk;

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

// Tile shape: warps per CTA, steps per tile, pipeline stages (compile-time
// overridable for tuning builds).
#ifndef SS_SEQ_W
#define SS_SEQ_W 4
#endif
#ifndef SS_SEQ_TL
#define SS_SEQ_TL 16
#endif
#ifndef SS_SEQ_S
#define SS_SEQ_S 3
#endif
#ifndef SS_SEQ_MINB
#define SS_SEQ_MINB 3
#endif

template <typename Tin, int N, int W, int TL, int S>
struct SeqLayout {
    static constexpr int NT = 32 * W;
    static constexpr int ESZ = (int)sizeof(Tin);
    static constexpr int CH = TL * ESZ / 16;            // 16-byte chunks per row per tensor
    static constexpr int VPC = 16 / ESZ;                 // values per chunk
    static constexpr int STREAM = 3 * CH * NT * 16;      // one stage of u, delta, z
    static constexpr int BC_TILE = N * TL * ESZ;         // one B or C box
    static constexpr int OFF_C = align_up(BC_TILE, 128); // TMA destinations are 128-byte aligned
    static constexpr int BC_STAGE = align_up(OFF_C + BC_TILE, 128);
    static constexpr int FSTRIDE = N >= 4 ? N + 4 : 4;   // fp32 [step][n] row, 16-byte aligned
    static constexpr int F_TILE = TL * FSTRIDE * 4;      // one widened B or C tile
    static constexpr int OFF_STREAM = 0;
    static constexpr int OFF_BC = S * STREAM;
    static constexpr int OFF_F = OFF_BC + S * BC_STAGE;  // [2 buffers][B, C]
    static constexpr int OFF_BAR = align_up(OFF_F + 4 * F_TILE, 8);
    static constexpr int TOTAL = OFF_BAR + S * 8 + 128;
    static_assert(OFF_BC % 128 == 0 && BC_STAGE % 128 == 0 && OFF_C % 128 == 0,
                  "TMA destinations must be 128-byte aligned");
    static_assert(STREAM % 16 == 0 && OFF_F % 16 == 0 && (FSTRIDE * 4) % 16 == 0,
                  "cp.async chunks and vector loads need 16-byte alignment");
};

template <int V>
__device__ __forceinline__ void lds_vec(const float *p, float *v) {
    if constexpr (V >= 4) {
#pragma unroll
        for (int j = 0; j < V / 4; ++j) {
            const float4 w = reinterpret_cast<const float4 *>(p)[j];
            v[4 * j] = w.x, v[4 * j + 1] = w.y, v[4 * j + 2] = w.z, v[4 * j + 3] = w.w;
        }
    } else if constexpr (V == 2) {
        const float2 w = *reinterpret_cast<const float2 *>(p);
        v[0] = w.x, v[1] = w.y;
    } else {
        v[0] = *p;
    }
}

// Two consecutive inputs of a row from its staged 32-bit words.
__device__ __forceinline__ f2 pair_at(const uint32_t *w, int i, uint16_t) {
    return mk2(bf16lo(w[i]), bf16hi(w[i]));
}
__device__ __forceinline__ f2 pair_at(const uint32_t *w, int i, float) {
    return mk2(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
}

// One recurrence step for all N states of a row; returns sum_n C_n h_n.
template <int N>
__device__ __forceinline__ float step_states(f2 *h, const f2 *A2, float dt, float du,
                                             const float *Bl, const float *Cl, float uv,
                                             bool zoh) {
    if (zoh) {
        // exact zero-order hold, one state at a time (A2 holds A log2(e))
        float acc = 0.f;
#pragma unroll
        for (int n = 0; n < N; ++n) {
            float &hn = (n & 1) ? h[n / 2].y : h[n / 2].x;
            const float a = ((n & 1) ? A2[n / 2].y : A2[n / 2].x) * kLn2;
            float e;
            const float f = zoh_step(dt, a, &e);
            hn = fmaf(e, hn, f * uv * Bl[n]);
            acc = fmaf(Cl[n], hn, acc);
        }
        return acc;
    }
    if constexpr (N == 1) {
        const float e = ex2(dt * A2[0].x);
        h[0].x = fmaf(e, h[0].x, du * Bl[0]);
        return Cl[0] * h[0].x;
    } else {
        float bv[N], cv[N];
        lds_vec<N>(Bl, bv);
        lds_vec<N>(Cl, cv);
        const f2 dd = mk2(dt, dt), uu = mk2(du, du);
        f2 acc0 = mk2(0.f, 0.f), acc1 = mk2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < N / 2; ++j) {
            const f2 t = fmul2(dd, A2[j]);
            const f2 e = mk2(ex2(t.x), ex2(t.y));
            const f2 bu = fmul2(uu, mk2(bv[2 * j], bv[2 * j + 1]));
            h[j] = ffma2(e, h[j], bu);
            const f2 c = mk2(cv[2 * j], cv[2 * j + 1]);
            if (j == 0) acc0 = fmul2(c, h[0]);
            else if (j == 1) acc1 = fmul2(c, h[1]);
            else if (j & 1) acc1 = ffma2(c, h[j], acc1);
            else acc0 = ffma2(c, h[j], acc0);
        }
        if constexpr (N >= 4) acc0 = fadd2(acc0, acc1);
        return acc0.x + acc0.y;
    }
}

template <int V>
__device__ __forceinline__ void store_vals(float *dst, const float *v) {
#pragma unroll
    for (int j = 0; j < V / 4; ++j)
        reinterpret_cast<float4 *>(dst)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2],
                                                         v[4 * j + 3]);
}
template <int V>
__device__ __forceinline__ void store_vals(uint16_t *dst, const float *v) {
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
}

template <typename Tin, typename Tout, int N, int W, int TL, int S>
__global__ void __launch_bounds__(32 * W, SS_SEQ_MINB)
    scan_seq_kernel(const __grid_constant__ CUtensorMap tm_B,
                    const __grid_constant__ CUtensorMap tm_C, const ssh::ScanParams p) {
    using LY = SeqLayout<Tin, N, W, TL, S>;
    constexpr int NT = LY::NT, CH = LY::CH, VPC = LY::VPC;
    constexpr int NP = (N + 1) / 2;  // state pairs
    static_assert(TL % 16 == 0, "tile must hold whole chunks for every dtype");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + LY::OFF_BAR);
    float *F = reinterpret_cast<float *>(smem + LY::OFF_F);

    const int tid = threadIdx.x;
    const int b = blockIdx.y;
    const int d = blockIdx.x * NT + tid;
    const bool row_ok = d < p.dim;
    const int dc = row_ok ? d : p.dim - 1;
    const long long row = (long long)b * p.dim + dc;
    const int L = (int)p.seqlen;
    const int n_tiles = (L + TL - 1) / TL;
    const bool has_z = p.z != nullptr;

    f2 A2[NP], h[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        const int n0 = 2 * j, n1 = 2 * j + 1 < N ? 2 * j + 1 : 2 * j;
        A2[j] = mk2(p.A[(long long)dc * N + n0] * kLog2e, p.A[(long long)dc * N + n1] * kLog2e);
        h[j] = (p.h0 && row_ok) ? mk2(p.h0[row * N + n0], p.h0[row * N + n1]) : mk2(0.f, 0.f);
    }
    const float bias = p.bias ? p.bias[dc] : 0.f;
    const float Dd = p.D ? p.D[dc] : 0.f;

    const Tin *g_u = static_cast<const Tin *>(p.u) + row * L;
    const Tin *g_dl = static_cast<const Tin *>(p.delta) + row * L;
    const Tin *g_z = has_z ? static_cast<const Tin *>(p.z) + row * L : g_u;

    // stage `t` of the per-row streams and of B/C
    auto issue = [&](int t) {
        if (t < n_tiles) {
            const int s = t % S;
            uint8_t *st = smem + LY::OFF_STREAM + s * LY::STREAM;
            const int l0 = t * TL;
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int lc = l0 + c * VPC;
                const int nv = row_ok ? max(0, min(VPC, L - lc)) : 0;
                const uint32_t bytes = (uint32_t)(nv * LY::ESZ);
                const size_t off = nv ? (size_t)lc : 0;
                cp_async16(st + ((0 * CH + c) * NT + tid) * 16, g_u + off, bytes);
                cp_async16(st + ((1 * CH + c) * NT + tid) * 16, g_dl + off, bytes);
                if (has_z) cp_async16(st + ((2 * CH + c) * NT + tid) * 16, g_z + off, bytes);
            }
            if (tid == 0 && t != p.drop_tile) {
                uint8_t *bc = smem + LY::OFF_BC + s * LY::BC_STAGE;
                mbar_expect_tx(&bar[s], 2 * LY::BC_TILE);
                tma_load_2d(bc, &tm_B, l0, b * N, &bar[s]);
                tma_load_2d(bc + LY::OFF_C, &tm_C, l0, b * N, &bar[s]);
            }
        }
        cp_async_commit();  // one group per call, empty past the end: keeps counting uniform
    };
    // widen + transpose tile t's B, C ([n][step] bf16/fp32) into F[buf] ([step][n] fp32)
    auto widen_bc = [&](int t, int buf) {
        const Tin *bc = reinterpret_cast<const Tin *>(smem + LY::OFF_BC + (t % S) * LY::BC_STAGE);
        const Tin *cc = reinterpret_cast<const Tin *>(smem + LY::OFF_BC + (t % S) * LY::BC_STAGE +
                                                      LY::OFF_C);
        float *fB = F + buf * 2 * (LY::F_TILE / 4);
        float *fC = fB + LY::F_TILE / 4;
        for (int i = tid; i < N * TL / 2; i += NT) {
            const int n = (2 * i) / TL, l = (2 * i) % TL;
            const f2 vb = mk2(to_f32(bc[2 * i]), to_f32(bc[2 * i + 1]));
            const f2 vc = mk2(to_f32(cc[2 * i]), to_f32(cc[2 * i + 1]));
            fB[l * LY::FSTRIDE + n] = vb.x;
            fB[(l + 1) * LY::FSTRIDE + n] = vb.y;
            fC[l * LY::FSTRIDE + n] = vc.x;
            fC[(l + 1) * LY::FSTRIDE + n] = vc.y;
        }
    };
    auto bail = [&](int k_waited) {
        // a B/C load never arrived: record it, let the other loads land, leave
        if (tid == 0) set_error(p.err, SS_ERR_TIMEOUT);
        for (int t = k_waited + 1; t <= k_waited + S - 2 && t < n_tiles; ++t)
            if (t != p.drop_tile) mbar_wait_bounded(&bar[t % S], (uint32_t)(t / S) & 1u, p.wait_limit);
        cp_async_wait_all();
    };

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < S - 1; ++t) issue(t);
    {
        const bool ok = n_tiles == 0 || mbar_wait_bounded(&bar[0], 0u, p.wait_limit);
        if (n_tiles > 0) widen_bc(0, 0);
        if (__syncthreads_or(!ok)) {
            bail(0);
            return;
        }
    }

    for (int k = 0; k < n_tiles; ++k) {
        issue(k + S - 1);
        bool ok = true;
        if (k + 1 < n_tiles) {
            ok = mbar_wait_bounded(&bar[(k + 1) % S], (uint32_t)((k + 1) / S) & 1u, p.wait_limit);
            widen_bc(k + 1, (k + 1) & 1);
        }
        cp_async_wait<S - 1>();

        // this thread's u, delta, z for the tile, as 32-bit words
        constexpr int WPT = TL * LY::ESZ / 4;  // words per tensor per tile
        uint32_t uw[WPT], dw[WPT], zw[WPT];
        {
            const uint8_t *st = smem + LY::OFF_STREAM + (k % S) * LY::STREAM;
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const uint4 a = *reinterpret_cast<const uint4 *>(st + ((0 * CH + c) * NT + tid) * 16);
                const uint4 bq = *reinterpret_cast<const uint4 *>(st + ((1 * CH + c) * NT + tid) * 16);
                uw[4 * c] = a.x, uw[4 * c + 1] = a.y, uw[4 * c + 2] = a.z, uw[4 * c + 3] = a.w;
                dw[4 * c] = bq.x, dw[4 * c + 1] = bq.y, dw[4 * c + 2] = bq.z, dw[4 * c + 3] = bq.w;
                if (has_z) {
                    const uint4 zq = *reinterpret_cast<const uint4 *>(st + ((2 * CH + c) * NT + tid) * 16);
                    zw[4 * c] = zq.x, zw[4 * c + 1] = zq.y, zw[4 * c + 2] = zq.z, zw[4 * c + 3] = zq.w;
                } else {
                    zw[4 * c] = zw[4 * c + 1] = zw[4 * c + 2] = zw[4 * c + 3] = 0u;
                }
            }
        }

        const float *fB = F + (k & 1) * 2 * (LY::F_TILE / 4);
        const float *fC = fB + LY::F_TILE / 4;
        const int l0 = k * TL;
        const bool tail = l0 + TL > L;
        // phase 1: dt and dt*u for every step of the tile (independent chains)
        f2 dt[TL / 2], du[TL / 2];
#pragma unroll
        for (int i = 0; i < TL / 2; ++i) {
            const f2 x = fadd2(pair_at(dw, i, Tin()), mk2(bias, bias));
            dt[i] = p.softplus ? softplus2(x) : x;
            if (tail) {
                if (l0 + 2 * i >= L) dt[i].x = 0.f;
                if (l0 + 2 * i + 1 >= L) dt[i].y = 0.f;
            }
            du[i] = fmul2(dt[i], pair_at(uw, i, Tin()));
        }
        // phase 2: the recurrence, step by step
        float out[TL];
#pragma unroll
        for (int i = 0; i < TL / 2; ++i) {
            const f2 uo = pair_at(uw, i, Tin());
            out[2 * i] = step_states<N>(h, A2, dt[i].x, du[i].x, fB + (2 * i) * LY::FSTRIDE,
                                        fC + (2 * i) * LY::FSTRIDE, uo.x, p.zoh);
            out[2 * i + 1] = step_states<N>(h, A2, dt[i].y, du[i].y,
                                            fB + (2 * i + 1) * LY::FSTRIDE,
                                            fC + (2 * i + 1) * LY::FSTRIDE, uo.y, p.zoh);
        }
        // phase 3: D skip and silu(z) gate
#pragma unroll
        for (int i = 0; i < TL / 2; ++i) {
            f2 o = ffma2(mk2(Dd, Dd), pair_at(uw, i, Tin()), mk2(out[2 * i], out[2 * i + 1]));
            if (has_z) o = fmul2(o, silu2(pair_at(zw, i, Tin())));
            out[2 * i] = o.x;
            out[2 * i + 1] = o.y;
        }
        if (row_ok) {
            Tout *dst = static_cast<Tout *>(p.y) + row * (long long)L + l0;
            if (!tail) {
                store_vals<TL>(dst, out);
            } else {
#pragma unroll
                for (int i = 0; i < TL; ++i)
                    if (l0 + i < L) store_out(dst + i, out[i]);
            }
        }
        if (__syncthreads_or(!ok)) {
            bail(k + 1);
            return;
        }
    }

    if (row_ok && p.h_last) {
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            p.h_last[row * N + 2 * j] = h[j].x;
            if (2 * j + 1 < N) p.h_last[row * N + 2 * j + 1] = h[j].y;
        }
    }
}

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

template <typename Tin, typename Tout, int N, int W, int TL, int S>
int launch_cfg(const ssh::ScanParams &p, int max_smem, cudaStream_t st) {
    using LY = SeqLayout<Tin, N, W, TL, S>;
    auto kern = scan_seq_kernel<Tin, Tout, N, W, TL, S>;
    if (LY::TOTAL > max_smem) return SS_ERR_UNSUPPORTED;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SS_ERR_CUDA;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::TOTAL) !=
            cudaSuccess)
            return SS_ERR_CUDA;
        attr_set[dev] = true;
    }
    const bool bf = sizeof(Tin) == 2;
    const uint64_t L = (uint64_t)p.seqlen;
    CUtensorMap tB, tC;
    if (!make_map(&tB, p.B, bf, L, (uint64_t)p.batch * N, L * sizeof(Tin), TL, N) ||
        !make_map(&tC, p.C, bf, L, (uint64_t)p.batch * N, L * sizeof(Tin), TL, N))
        return SS_ERR_CUDA;
    const dim3 grid((unsigned)((p.dim + LY::NT - 1) / LY::NT), (unsigned)p.batch);
    kern<<<grid, LY::NT, LY::TOTAL, st>>>(tB, tC, p);
    return cudaPeekAtLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

template <typename Tin, typename Tout>
int launch_types(const ssh::ScanParams &p, int max_smem, cudaStream_t st) {
    constexpr int W = SS_SEQ_W, TL = SS_SEQ_TL, S = SS_SEQ_S;
    switch (p.dstate) {
        case 1: return launch_cfg<Tin, Tout, 1, W, TL, S>(p, max_smem, st);
        case 2: return launch_cfg<Tin, Tout, 2, W, TL, S>(p, max_smem, st);
        case 4: return launch_cfg<Tin, Tout, 4, W, TL, S>(p, max_smem, st);
        case 8: return launch_cfg<Tin, Tout, 8, W, TL, S>(p, max_smem, st);
        case 16: return launch_cfg<Tin, Tout, 16, W, TL, S>(p, max_smem, st);
        default: return SS_ERR_UNSUPPORTED;
    }
}

}  // namespace

bool ssh::seq_supported(const ssh::ScanParams &p) {
    const int esz = p.in_dtype == SS_BF16 ? 2 : 4;
    const int osz = p.out_dtype == SS_BF16 ? 2 : 4;
    if ((p.seqlen * esz) % 16 != 0 || (p.seqlen * osz) % 16 != 0) return false;
    if (p.seqlen >= (1LL << 31)) return false;
    return encode_fn() != nullptr;
}

int ssh::launch_seq(const ssh::ScanParams &p, int max_smem, cudaStream_t st) {
    const bool ib = p.in_dtype == SS_BF16, ob = p.out_dtype == SS_BF16;
    if (ib && ob) return launch_types<uint16_t, uint16_t>(p, max_smem, st);
    if (ib) return launch_types<uint16_t, float>(p, max_smem, st);
    if (ob) return launch_types<float, uint16_t>(p, max_smem, st);
    return launch_types<float, float>(p, max_smem, st);
}
