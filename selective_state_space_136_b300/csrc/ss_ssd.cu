// Mamba-2 state space duality (SSD): the selective scan with a scalar decay
// per head, computed chunk by chunk with matrix products on the tensor cores.
//
// soft186.com, "Mamba选择性状态空间机制", section "状态空间对偶性算法突破": Mamba-2
// computes the scan through a block decomposition of its semiseparable
// matrix. With A = a_h I per head h, dt shared by the head's P channels and B,
// C shared by all heads, the recurrence per head
//     H(t) = exp(dt_t a) H(t-1) + dt_t x_t B_t^T        (P x N state)
//     y_t  = H(t) C_t + D x_t
// splits, for a chunk of Q steps with cum_t = sum_{r<=t} dt_r a (within the
// chunk) and H_prev the state entering it, into
//     y_t  = sum_{s<=t} (C_t . B_s) exp(cum_t - cum_s) dt_s x_s    (intra-chunk)
//          + exp(cum_t) H_prev C_t + D x_t                          (from the carry)
//     H_new = exp(cum_{Q-1}) H_prev + sum_s exp(cum_{Q-1} - cum_s) dt_s x_s B_s^T
// i.e. four contractions per chunk: G = C B^T (Q x Q over N), (G o decay) X
// (Q x P over Q), C H_prev^T (Q x P over N) and B^T X~ (N x P over Q). They
// run as bf16 mma.sync with fp32 accumulation; the carried state stays in fp32
// accumulators and enters the C H_prev product as two bf16 terms (hi + lo).
//
// One CTA of 4 warps per (batch, head, group of kPC channels) walks the
// chunks in order; warp w owns rows t in [16w, 16w+16) of the chunk products
// and state rows n in [N/4 w, N/4 (w+1)) of the carried state. Splitting a
// head's channels over CTAs repeats the C B^T product in each but halves a
// CTA's shared memory and work, so more CTAs run at once and the grid's last
// wave is less empty.
#include "ss_common.cuh"
#include "ss_internal.h"

namespace {

using namespace ssk;

constexpr int kQ = 64;   // chunk length
constexpr int kP = 64;   // head dimension
#ifndef SS_SSD_PC
#define SS_SSD_PC 32
#endif
constexpr int kPC = SS_SSD_PC;  // channels of the head per CTA
static_assert(kP % kPC == 0 && kPC % 16 == 0, "channel groups of whole 16-column tiles");
constexpr int kPad = 8;  // bf16 padding per smem row (rows 16 bytes apart in banks)

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return a | (b << 16);
}
__device__ __forceinline__ float bf16_round(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
}

__device__ __forceinline__ void store_pair(float *p, float a, float b) {
    *reinterpret_cast<float2 *>(p) = make_float2(a, b);
}
__device__ __forceinline__ void store_pair(uint16_t *p, float a, float b) {
    *reinterpret_cast<uint32_t *>(p) = pack_bf16(a, b);
}

template <int N>
struct SsdSmem {
    uint16_t X[kQ][kPC + kPad];    // x of the chunk, [t][p]
    uint16_t Xs[kQ][kPC + kPad];   // x scaled by exp(cum_last - cum_s) dt_s, [s][p]
    uint16_t Bm[kQ][N + kPad];     // B of the chunk, [s][n]
    uint16_t Cm[kQ][N + kPad];     // C of the chunk, [t][n]
    uint16_t Hh[N][kPC + kPad];    // carried state, high bf16 part, [n][p]
    uint16_t Hl[N][kPC + kPad];    // carried state, low bf16 part (H - hi), [n][p]
    float dt[kQ];                  // dt_t of the chunk
    float cum[kQ];                 // cum_t
};

// 16x16 A-operand tile at (row0, col0) of a row-major bf16 array with `pitch`
// elements per row.
__device__ __forceinline__ void load_a(uint32_t (&a)[4], const uint16_t *base, int pitch,
                                       int row0, int col0, int lane) {
    const int r = row0 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int c = col0 + (lane >> 4) * 8;
    ldsm_x4(a, base + r * pitch + c);
}
// A operand (m x k) read transposed from a row-major [k][m] array: the 16x16
// tile with m in [m0, m0+16), k in [k0, k0+16).
__device__ __forceinline__ void load_a_t(uint32_t (&a)[4], const uint16_t *base, int pitch, int m0,
                                         int k0, int lane) {
    const int mi = lane >> 3;
    const int r = k0 + (lane & 7) + (mi >> 1) * 8;
    const int c = m0 + (mi & 1) * 8;
    ldsm_x4_t(a, base + r * pitch + c);
}
// B operands of two n-tiles (n in [n0, n0+16)) over k in [k0, k0+16), from a
// row-major [n][k] array: b[0], b[1] for n-tile n0, b[2], b[3] for n0 + 8.
__device__ __forceinline__ void load_b_nk(uint32_t (&b)[4], const uint16_t *base, int pitch,
                                          int n0, int k0, int lane) {
    const int r = n0 + (lane & 7) + (lane >> 4) * 8;
    const int c = k0 + ((lane >> 3) & 1) * 8;
    ldsm_x4(b, base + r * pitch + c);
}
// The same from a row-major [k][n] array (read transposed).
__device__ __forceinline__ void load_b_kn(uint32_t (&b)[4], const uint16_t *base, int pitch,
                                          int n0, int k0, int lane) {
    const int r = k0 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int c = n0 + (lane >> 4) * 8;
    ldsm_x4_t(b, base + r * pitch + c);
}

template <typename Tin, typename Tout, int N>
__global__ void __launch_bounds__(128) ssd_fwd_kernel(const ssh::SsdParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SsdSmem<N> &sm = *reinterpret_cast<SsdSmem<N> *>(smem_raw);
    constexpr int NW = N / 4;  // state rows per warp
    constexpr int MT = NW / 16;  // 16-row tiles of the state per warp
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tg = lane & 3;
    constexpr int NG = kP / kPC;  // channel groups per head
    const int b = blockIdx.x / (p.heads * NG), h = (blockIdx.x / NG) % p.heads;
    const int p0 = (blockIdx.x % NG) * kPC;  // first channel of this CTA
    const long long L = p.seqlen;
    const float a = p.A[h] * kLog2e;  // log2 units
    const float bias = p.dt_bias ? p.dt_bias[h] : 0.f;
    const float Dh = p.D ? p.D[h] : 0.f;
    const long long xs_t = (long long)p.heads * kP;  // x / y stride between steps

    // carried state of this warp's rows: Hacc[mt][pt][4] covers n = 16 mt + {g, g+8}
    // (+ NW warp), p = p0 + 8 pt + 2 tg + {0, 1}
    float Hacc[MT][kPC / 8][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int pt = 0; pt < kPC / 8; ++pt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int n = NW * warp + 16 * mt + g + (e >> 1) * 8;
                const int pp = p0 + 8 * pt + 2 * tg + (e & 1);
                Hacc[mt][pt][e] =
                    p.h0 ? p.h0[(((long long)b * p.heads + h) * kP + pp) * N + n] : 0.f;
            }
    auto publish_state = [&]() {  // Hacc -> Hh/Hl (bf16 hi + lo) in smem
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int pt = 0; pt < kPC / 8; ++pt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int n = NW * warp + 16 * mt + g + (e >> 1) * 8;
                    const int pp = 8 * pt + 2 * tg;
                    const float v0 = Hacc[mt][pt][e], v1 = Hacc[mt][pt][e + 1];
                    const float h0 = bf16_round(v0), h1 = bf16_round(v1);
                    *reinterpret_cast<uint32_t *>(&sm.Hh[n][pp]) = pack_bf16(h0, h1);
                    *reinterpret_cast<uint32_t *>(&sm.Hl[n][pp]) = pack_bf16(v0 - h0, v1 - h1);
                }
    };
    publish_state();

    const int n_chunks = (int)(L / kQ);
    for (int c = 0; c < n_chunks; ++c) {
        const long long l0 = (long long)c * kQ;
        __syncthreads();  // the previous chunk is done with X, Xs, B, C, dt, cum
        // ---- load the chunk: x (Q x P), B and C (Q x N) straight into shared
        // memory by asynchronous 16-byte copies (all in flight at once)
        for (int i = tid; i < kQ * kPC / 8; i += 128) {
            const int t = i / (kPC / 8), c8 = (i % (kPC / 8)) * 8;
            const Tin *src = static_cast<const Tin *>(p.x) + ((long long)b * L + l0 + t) * xs_t +
                             (long long)h * kP + p0 + c8;
            cp_async16(&sm.X[t][c8], src, 16);
        }
        for (int i = tid; i < 2 * kQ * N / 8; i += 128) {
            const int which = i / (kQ * N / 8), j = i % (kQ * N / 8);
            const int t = j / (N / 8), c8 = (j % (N / 8)) * 8;
            const Tin *src = static_cast<const Tin *>(which ? p.C : p.B) +
                             ((long long)b * L + l0 + t) * N + c8;
            cp_async16(which ? &sm.Cm[t][c8] : &sm.Bm[t][c8], src, 16);
        }
        cp_async_commit();
        if (warp == 0) {
            // dt_t and the inclusive prefix sum of dt_t a over the chunk (2 steps per lane)
            float d2[2], s2[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int t = 2 * lane + k;
                const float xr =
                    to_f32(static_cast<const Tin *>(p.dt)[((long long)b * L + l0 + t) * p.heads + h]) + bias;
                d2[k] = p.softplus ? softplus1(xr) : xr;
                s2[k] = d2[k] * a;
            }
            float run = s2[0] + s2[1];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, run, off);
                if (lane >= off) run += o;
            }
            const float before = run - (s2[0] + s2[1]);
            sm.dt[2 * lane] = d2[0], sm.dt[2 * lane + 1] = d2[1];
            sm.cum[2 * lane] = before + s2[0];
            sm.cum[2 * lane + 1] = before + s2[0] + s2[1];
        }
        cp_async_wait_all();
        __syncthreads();

        // ---- G = C B^T for rows t in [16 warp, 16 warp + 16), all s
        const int t0 = 16 * warp;
        float G[kQ / 8][4];
#pragma unroll
        for (int j = 0; j < kQ / 8; ++j) G[j][0] = G[j][1] = G[j][2] = G[j][3] = 0.f;
#pragma unroll
        for (int k0 = 0; k0 < N; k0 += 16) {
            uint32_t af[4];
            load_a(af, &sm.Cm[0][0], N + kPad, t0, k0, lane);
#pragma unroll
            for (int j = 0; j < kQ / 8; j += 2) {
                uint32_t bf[4];
                load_b_nk(bf, &sm.Bm[0][0], N + kPad, 8 * j, k0, lane);
                mma16816(G[j], af, bf[0], bf[1]);
                mma16816(G[j + 1], af, bf[2], bf[3]);
            }
        }
        // decay mask: M[t][s] = G exp(cum_t - cum_s) dt_s for s <= t, else 0
        const float cum_r0 = sm.cum[t0 + g], cum_r1 = sm.cum[t0 + g + 8];
#pragma unroll
        for (int j = 0; j < kQ / 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = t0 + g + (e >> 1) * 8, s = 8 * j + 2 * tg + (e & 1);
                const float ct = (e >> 1) ? cum_r1 : cum_r0;
                G[j][e] = s <= t ? G[j][e] * ex2(ct - sm.cum[s]) * sm.dt[s] : 0.f;
            }
        // ---- Y = M X (intra-chunk)
        float Y[kPC / 8][4];
#pragma unroll
        for (int j = 0; j < kPC / 8; ++j) Y[j][0] = Y[j][1] = Y[j][2] = Y[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < kQ / 16; ++kk) {
            // the accumulators of s-tiles 2kk, 2kk+1 are the A fragment of k-step kk
            uint32_t af[4];
            af[0] = pack_bf16(G[2 * kk][0], G[2 * kk][1]);
            af[1] = pack_bf16(G[2 * kk][2], G[2 * kk][3]);
            af[2] = pack_bf16(G[2 * kk + 1][0], G[2 * kk + 1][1]);
            af[3] = pack_bf16(G[2 * kk + 1][2], G[2 * kk + 1][3]);
#pragma unroll
            for (int j = 0; j < kPC / 8; j += 2) {
                uint32_t bf[4];
                load_b_kn(bf, &sm.X[0][0], kPC + kPad, 8 * j, 16 * kk, lane);
                mma16816(Y[j], af, bf[0], bf[1]);
                mma16816(Y[j + 1], af, bf[2], bf[3]);
            }
        }
        // ---- + exp(cum_t) C H_prev^T (state from before the chunk; hi and lo parts)
        {
            float Z[kPC / 8][4];
#pragma unroll
            for (int j = 0; j < kPC / 8; ++j) Z[j][0] = Z[j][1] = Z[j][2] = Z[j][3] = 0.f;
#pragma unroll
            for (int k0 = 0; k0 < N; k0 += 16) {
                uint32_t af[4];
                load_a(af, &sm.Cm[0][0], N + kPad, t0, k0, lane);
#pragma unroll
                for (int j = 0; j < kPC / 8; j += 2) {
                    uint32_t bf[4];
                    load_b_kn(bf, &sm.Hh[0][0], kPC + kPad, 8 * j, k0, lane);
                    mma16816(Z[j], af, bf[0], bf[1]);
                    mma16816(Z[j + 1], af, bf[2], bf[3]);
                    load_b_kn(bf, &sm.Hl[0][0], kPC + kPad, 8 * j, k0, lane);
                    mma16816(Z[j], af, bf[0], bf[1]);
                    mma16816(Z[j + 1], af, bf[2], bf[3]);
                }
            }
            const float f0 = ex2(cum_r0), f1 = ex2(cum_r1);
#pragma unroll
            for (int j = 0; j < kPC / 8; ++j) {
                Y[j][0] = fmaf(f0, Z[j][0], Y[j][0]);
                Y[j][1] = fmaf(f0, Z[j][1], Y[j][1]);
                Y[j][2] = fmaf(f1, Z[j][2], Y[j][2]);
                Y[j][3] = fmaf(f1, Z[j][3], Y[j][3]);
            }
        }
        // ---- + D x, store y
#pragma unroll
        for (int j = 0; j < kPC / 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const int t = t0 + g + (e >> 1) * 8, pp = 8 * j + 2 * tg;
                const uint32_t xw = *reinterpret_cast<const uint32_t *>(&sm.X[t][pp]);
                const float y0 = fmaf(Dh, bf16lo(xw), Y[j][e]);
                const float y1 = fmaf(Dh, bf16hi(xw), Y[j][e + 1]);
                Tout *dst = static_cast<Tout *>(p.y) + ((long long)b * L + l0 + t) * xs_t +
                            (long long)h * kP + p0 + pp;
                store_pair(dst, y0, y1);
            }

        // ---- carry: H = exp(cum_last) H + B^T (x scaled by exp(cum_last - cum_s) dt_s)
        const float cum_last = sm.cum[kQ - 1];
        for (int i = tid; i < kQ * kPC / 2; i += 128) {
            const int s = i / (kPC / 2), pp = (i % (kPC / 2)) * 2;
            const float w = ex2(cum_last - sm.cum[s]) * sm.dt[s];
            const uint32_t xw = *reinterpret_cast<const uint32_t *>(&sm.X[s][pp]);
            *reinterpret_cast<uint32_t *>(&sm.Xs[s][pp]) = pack_bf16(bf16lo(xw) * w, bf16hi(xw) * w);
        }
        __syncthreads();  // Xs ready; every warp is done reading Hh/Hl of the previous state
        const float decay = ex2(cum_last);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int pt = 0; pt < kPC / 8; ++pt)
#pragma unroll
                for (int e = 0; e < 4; ++e) Hacc[mt][pt][e] *= decay;
#pragma unroll
            for (int k0 = 0; k0 < kQ; k0 += 16) {
                uint32_t af[4];
                load_a_t(af, &sm.Bm[0][0], N + kPad, NW * warp + 16 * mt, k0, lane);
#pragma unroll
                for (int pt = 0; pt < kPC / 8; pt += 2) {
                    uint32_t bf[4];
                    load_b_kn(bf, &sm.Xs[0][0], kPC + kPad, 8 * pt, k0, lane);
                    mma16816(Hacc[mt][pt], af, bf[0], bf[1]);
                    mma16816(Hacc[mt][pt + 1], af, bf[2], bf[3]);
                }
            }
        }
        publish_state();
    }

    if (p.h_last) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int pt = 0; pt < kPC / 8; ++pt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int n = NW * warp + 16 * mt + g + (e >> 1) * 8;
                    const int pp = p0 + 8 * pt + 2 * tg + (e & 1);
                    p.h_last[(((long long)b * p.heads + h) * kP + pp) * N + n] = Hacc[mt][pt][e];
                }
    }
}

template <typename Tin, typename Tout, int N>
int ssd_n(const ssh::SsdParams &p, cudaStream_t st) {
    const int smem = (int)sizeof(SsdSmem<N>);
    auto kern = ssd_fwd_kernel<Tin, Tout, N>;
    static bool done[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SS_ERR_CUDA;
    if (!done[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return SS_ERR_CUDA;
        done[dev] = true;
    }
    kern<<<(unsigned)((long long)p.batch * p.heads * (kP / kPC)), 128, smem, st>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

template <typename Tin, typename Tout>
int ssd_t(const ssh::SsdParams &p, cudaStream_t st) {
    switch (p.dstate) {
        case 64: return ssd_n<Tin, Tout, 64>(p, st);
        case 128: return ssd_n<Tin, Tout, 128>(p, st);
        default: return SS_ERR_UNSUPPORTED;
    }
}

}  // namespace

bool ssh::ssd_supported(const ssh::SsdParams &p) {
    return p.in_dtype == SS_BF16 && p.headdim == kP && (p.dstate == 64 || p.dstate == 128) && p.seqlen % kQ == 0 &&
           (long long)p.batch * p.heads * (kP / kPC) < (1LL << 31);
}

int ssh::launch_ssd(const ssh::SsdParams &p, cudaStream_t st) {
    if (p.in_dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
    return p.out_dtype == SS_BF16 ? ssd_t<uint16_t, uint16_t>(p, st) : ssd_t<uint16_t, float>(p, st);
}
