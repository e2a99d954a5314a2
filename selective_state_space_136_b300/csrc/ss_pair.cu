// Selective scan, chained pair-row variant (the default for dstate 16 when
// there are many rows).
//
// What it computes is the selective recurrence of "Mamba: Linear-Time
// Sequence Modeling with Selective State Spaces" (sections "Method" and "The
// Selection Mechanism (S6)") with the dt * B input term of the soft186.com
// article (section "动态参数化的状态空间"), fused as the Mamba page's section
// "Hardware-aware state expansion" describes: inputs cross into on-chip
// memory once, the 16 states of a row stay in registers, only y and the final
// state are written.
//
// Two kernels per call:
//  1. bc_pack: widens B and C ((batch, 16, L), bf16 or fp32) once into fp32
//     rows [batch][L][B0..B15 C0..C15], the layout the scan reads, and resets
//     the work counter of the call.
//  2. scan_pair: persistent one-warp CTAs. A warp serves 32 rows of one batch
//     as 16 row pairs; lane 2g+q owns row 2g+q for the per-row work (dt,
//     dt*u, D skip, gate, loads and stores) and states [8q, 8q+8) of BOTH
//     rows of its pair. Sharing each loaded B/C value between two rows halves
//     the shared-memory bytes per state element; the partner row's dt and
//     dt*u, and the partner's partial output, cross with one xor-shuffle each.
//
// Work is cut into units (time segment s, row block rb) taken from an atomic
// counter in segment-major order, so the units of one row block are started
// in time order. A unit starts from the state the previous segment of its
// row block left in a global carry buffer (published with a release flag and
// read after a bounded acquire wait). Segments only balance the load across
// the machine: nothing is recomputed, and the exact order of the recurrence
// along time is kept. A segment count of 1 gives plain static rows.
//
// Per tile of TL steps: each lane loads its own row's u, delta, z for the
// next tile with one 256-bit load per tensor (whole 32-byte sectors, one tile
// ahead, held in registers) and writes its y as whole sectors; the fp32 B/C
// tile arrives by one TMA box into an mbarrier-tracked ring of S stages.
#include "ss_common.cuh"
#include "ss_internal.h"

#include <cudaTypedefs.h>

#ifndef SS_PAIR_TL
#define SS_PAIR_TL 16
#endif
#ifndef SS_PAIR_S
#define SS_PAIR_S 4
#endif
#ifndef SS_PAIR_MINB
#define SS_PAIR_MINB 8
#endif
#ifndef SS_PAIR_TANH
#define SS_PAIR_TANH 1  // silu through tanh.approx for bf16 inputs
#endif

namespace {

using namespace ssk;

constexpr int kN = 16;  // states per row served by this variant

template <typename Tin, int TL, int S>
struct PairLayout {
    static constexpr int ESZ = (int)sizeof(Tin);
    static constexpr int NV = TL * ESZ / 32;           // 32-byte loads per row per tensor per tile
    static constexpr int BC_BOX = TL * 2 * kN * 4;     // fp32 [TL][B16 C16]
    static constexpr int OFF_BAR = S * BC_BOX;
    static constexpr int OFF_CONV = OFF_BAR + 64;       // fused convolution: 32 lanes x 8 floats
    static constexpr int TOTAL = OFF_CONV + 32 * 8 * 4 + 128;
    static_assert(S * 8 <= 64, "mbarriers fit before the convolution's slots");
    static_assert(BC_BOX % 128 == 0, "TMA destinations 128-byte aligned");
    static_assert(NV >= 1 && TL * ESZ % 32 == 0, "a tile row is whole 32-byte sectors");
};

// ---------------------------------------------------------------- B/C pack

template <typename Tin>
__global__ void __launch_bounds__(256) bc_pack_kernel(const Tin *__restrict__ B,
                                                      const Tin *__restrict__ C, float *BC,
                                                      long long L, int batch,
                                                      unsigned long long *counter) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // (b, l)
    if (i == 0 && counter) counter[0] = counter[1] = 0ull;  // one per scan pass
    if (i >= (long long)batch * L) return;
    const long long b = i / L, l = i % L;
    const Tin *Bb = B + b * kN * L + l;
    const Tin *Cb = C + b * kN * L + l;
    float4 *dst = reinterpret_cast<float4 *>(BC + i * 2 * kN);
#pragma unroll
    for (int n = 0; n < kN; n += 4)
        dst[n / 4] = make_float4(to_f32(Bb[n * L]), to_f32(Bb[(n + 1) * L]),
                                 to_f32(Bb[(n + 2) * L]), to_f32(Bb[(n + 3) * L]));
#pragma unroll
    for (int n = 0; n < kN; n += 4)
        dst[4 + n / 4] = make_float4(to_f32(Cb[n * L]), to_f32(Cb[(n + 1) * L]),
                                     to_f32(Cb[(n + 2) * L]), to_f32(Cb[(n + 3) * L]));
}

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ f2 pair_at(const uint32_t *w, int i, uint16_t) {
    return mk2(bf16lo(w[i]), bf16hi(w[i]));
}
__device__ __forceinline__ f2 pair_at(const uint32_t *w, int i, float) {
    return mk2(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
}

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Store one tile of a row (32-byte aligned) as whole 32-byte sectors.
template <int V>
__device__ __forceinline__ void store_tile(float *dst, const float *v) {
#pragma unroll
    for (int j = 0; j < V / 8; ++j) stg256(dst + 8 * j, v + 8 * j);
}
template <int V>
__device__ __forceinline__ void store_tile(uint16_t *dst, const float *v) {
#pragma unroll
    for (int j = 0; j < V / 16; ++j) {
        float w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[16 * j + 2 * k]));
            const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[16 * j + 2 * k + 1]));
            w[k] = __uint_as_float(lo | (hi << 16));
        }
        stg256(dst + 16 * j, w);
    }
}

// Work of one pass.
//  chained (one pass): the tiles of all row blocks, laid end to end, are cut
//    into `units` equal ranges (one per persistent warp, taken in order from
//    the counter). With at least as many row blocks as ranges, a range spans
//    at most the tail of one row block, whole row blocks, and the head of one
//    more, so each row block is split at most once: its head piece (in one
//    range) hands its end state to its tail piece (in the next range) through
//    the carry buffer. This balances the work to within one tile per warp.
//  chunked passes: units are (segment, row block) in segment-major order.
struct PairSched {
    int rb_per_batch;          // row blocks of 32 rows per batch
    int total_rb;              // batch * rb_per_batch
    int nt;                    // tiles per row
    int n_seg;                 // chunked: time segments per row block
    int seg_len;               // chunked: steps per segment (multiple of TL)
    long long units;           // chained: ranges; chunked: segments x row blocks
    unsigned long long *counter;
    unsigned long long *flags;  // per row block: epoch << 16 | 1 once its head piece is done
    float *carry;               // per row block: 32 rows x 16 states
    const float *BC;            // packed fp32 B/C
    unsigned long long epoch;
    float *hagg;                // [row block][segment][32 rows][16]: end states, then carries
    float *sdt;                 // [row block][segment][32 rows]: summed dt per segment
};

// Chained pass: store the end state of the head piece of row block `rbi`
// (this lane's half of the states of its row pair) and release the row
// block's flag so its tail piece may start from it.
__device__ __forceinline__ void publish_carry(const PairSched &sch, int rbi, int lane, int q,
                                              const f2 (&h)[2][4]) {
    float *c0 = sch.carry + ((long long)rbi * 32 + lane) * kN + 8 * q;
    float *c1 = sch.carry + ((long long)rbi * 32 + (lane ^ 1)) * kN + 8 * q;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        __stcg(c0 + 2 * j, h[0][j].x);
        __stcg(c0 + 2 * j + 1, h[0][j].y);
        __stcg(c1 + 2 * j, h[1][j].x);
        __stcg(c1 + 2 * j + 1, h[1][j].y);
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release(sch.flags + rbi, (sch.epoch << 16) | 1ull);
}

// ---------------------------------------------------------------- cross-segment carry

// One warp per row. Lane g holds segment g's affine map h -> a h + b per state
// (a = 2^(A log2(e) * summed dt), b = end state from zero); an inclusive
// Kogge-Stone scan with up-shuffles composes the maps in time order,
// (a1, b1) then (a2, b2) = (a2 a1, a2 b1 + b2), and applying the prefix to
// the initial state gives the state each segment starts from. Segments are
// taken 32 at a time with the running state carried between rounds. The
// result overwrites the aggregate: slot g then holds the state entering
// segment g + 1.
__global__ void __launch_bounds__(128) carry_combine_kernel(const ssh::ScanParams p,
                                                            const PairSched sch) {
    constexpr unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const long long wrow = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (wrow >= (long long)sch.total_rb * 32) return;  // whole warps exit together
    const int rbi = (int)(wrow / 32), rib = (int)(wrow % 32);
    const int b = rbi / sch.rb_per_batch, blk = rbi % sch.rb_per_batch;
    const int d = blk * 32 + rib;
    const int dc = d < p.dim ? d : p.dim - 1;
    const long long row = (long long)b * p.dim + dc;
    float A2[kN], hc[kN];
#pragma unroll
    for (int n = 0; n < kN; ++n) {
        A2[n] = p.A[(long long)dc * kN + n] * kLog2e;
        hc[n] = p.h0 ? p.h0[row * kN + n] : 0.f;
    }
    const int n_agg = sch.n_seg - 1;
    for (int g0 = 0; g0 < n_agg; g0 += 32) {
        const int g = g0 + lane;
        const bool valid = g < n_agg;
        const long long slot = ((long long)rbi * sch.n_seg + g) * 32 + rib;
        const float sd = valid ? __ldcg(sch.sdt + slot) : 0.f;
        float a[kN], bb[kN];
#pragma unroll
        for (int n = 0; n < kN; ++n) {
            a[n] = valid ? ex2(A2[n] * sd) : 1.f;
            bb[n] = valid ? __ldcg(sch.hagg + slot * kN + n) : 0.f;
        }
#pragma unroll
        for (int off = 1; off < 32; off *= 2) {
#pragma unroll
            for (int n = 0; n < kN; ++n) {
                const float ap = __shfl_up_sync(FULL, a[n], off);
                const float bp = __shfl_up_sync(FULL, bb[n], off);
                if (lane >= off) {
                    bb[n] = fmaf(a[n], bp, bb[n]);
                    a[n] *= ap;
                }
            }
        }
#pragma unroll
        for (int n = 0; n < kN; ++n) {
            const float st = fmaf(a[n], hc[n], bb[n]);  // state after segment g
            if (valid) __stcg(sch.hagg + slot * kN + n, st);
            hc[n] = __shfl_sync(FULL, st, 31);
        }
    }
}


// Input term of one state pair under the exact zero-order hold, for decay
// exponent tt = dt a log2(e) (e = 2^tt), 1 / a and u B: ((e - 1) / a) u B.
// For |dt a| < 1/8 the difference e - 1 cancels, so there the factor is
// dt (1 + x/2 + x^2/6 + x^3/24 + x^4/120), x = dt a (Taylor series of
// (e^x - 1) / x, truncation below x^5/720 < 5e-9 relative); an a of 0 has
// x = 0 and gets dt, the limit.
__device__ __forceinline__ f2 zoh_input(f2 tt, f2 e, f2 ia, f2 dd, f2 ub) {
    const f2 fd = ffma2(e, ia, mk2(-ia.x, -ia.y));
    const f2 x = fmul2(tt, mk2(kLn2, kLn2));
    f2 ph = ffma2(x, mk2(1.f / 120.f, 1.f / 120.f), mk2(1.f / 24.f, 1.f / 24.f));
    ph = ffma2(ph, x, mk2(1.f / 6.f, 1.f / 6.f));
    ph = ffma2(ph, x, mk2(0.5f, 0.5f));
    ph = ffma2(ph, x, mk2(1.f, 1.f));
    const f2 fs = fmul2(dd, ph);
    const f2 f = mk2(fabsf(x.x) < 0.125f ? fs.x : fd.x, fabsf(x.y) < 0.125f ? fs.y : fd.y);
    return fmul2(f, ub);
}

// ---------------------------------------------------------------- the scan

// MODE: kChain  - units chained along time through the carry buffer (one pass);
//       kAgg    - aggregate pass: every segment but the last from a zero state,
//                 no output; stores the end state and the summed dt;
//       kSeg    - output pass: every segment from its carried-in state.
enum { kChain = 0, kAgg = 1, kSeg = 2 };

// what the kernel does besides the plain recurrence:
//  kConv - the causal convolution fused in front (u formed from x in registers)
//  kZoh  - the exact zero-order-hold input factor (exp(dt a) - 1) / a in place of dt
enum { kPlain = 0, kConv = 1, kZoh = 2 };

#ifdef SS_PAIR_MAXNREG
#define SS_PAIR_BOUNDS __maxnreg__(SS_PAIR_MAXNREG)
#else
#define SS_PAIR_BOUNDS __launch_bounds__(32, SS_PAIR_MINB)
#endif

template <typename Tin, typename Tout, int TL, int S, int MODE, int FL>
__global__ void SS_PAIR_BOUNDS
    scan_pair_kernel(const __grid_constant__ CUtensorMap tm_bc, const ssh::ScanParams p,
                     const PairSched sch) {
    constexpr bool OUT = MODE != kAgg;  // produces y
    constexpr bool CV = FL == kConv, ZH = FL == kZoh;
    using LY = PairLayout<Tin, TL, S>;
    constexpr unsigned FULL = 0xffffffffu;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + LY::OFF_BAR);

    const int lane = threadIdx.x;
    const int q = lane & 1;              // which half of the states
    const int L = (int)p.seqlen;
    const bool has_z = p.z != nullptr;

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    long long gt = 0;  // tiles issued by this warp so far, across units (stage/parity clock)
    bool failed = false;

    // chained pass: ranges of the row blocks' tiles laid end to end (see PairSched)
    long long r_begin = 0, r_end = 0, c_cur = -1, c_first = 0;
    for (;;) {
        int seg = 0, rbi = 0, t_begin = 0, t_end = 0;  // the piece: tiles [t_begin, t_end) of row block rbi
        if (MODE == kChain) {
            if (c_cur < c_first) {
                // next range; its pieces go from the last row block it touches
                // to the first, so the head piece a later range waits for is done
                // first and the tail piece that waits on an earlier range is done last
                unsigned long long t = 0;
                if (lane == 0) t = atomicAdd(sch.counter, 1ull);
                t = __shfl_sync(FULL, t, 0);
                if ((long long)t >= sch.units) break;
                const long long total = (long long)sch.total_rb * sch.nt;
                r_begin = total * (long long)t / sch.units;
                r_end = total * ((long long)t + 1) / sch.units;
                if (r_end <= r_begin) continue;
                c_first = r_begin / sch.nt;
                c_cur = (r_end - 1) / sch.nt;
            }
            rbi = (int)c_cur;
            t_begin = (int)(max(r_begin, c_cur * sch.nt) - c_cur * sch.nt);
            t_end = (int)(min(r_end, (c_cur + 1) * sch.nt) - c_cur * sch.nt);
            --c_cur;
        } else {
            unsigned long long t = 0;
            if (lane == 0) t = atomicAdd(sch.counter + (MODE == kSeg ? 1 : 0), 1ull);
            t = __shfl_sync(FULL, t, 0);
            if ((long long)t >= sch.units) break;
            seg = (int)(t / sch.total_rb);
            rbi = (int)(t % sch.total_rb);
            t_begin = seg * (sch.seg_len / TL);
            t_end = min(sch.nt, t_begin + sch.seg_len / TL);
        }
        const int b = rbi / sch.rb_per_batch, blk = rbi % sch.rb_per_batch;
        const int d = blk * 32 + lane;
        const bool row_ok = d < p.dim;
        const int dc = row_ok ? d : p.dim - 1;
        const long long row = (long long)b * p.dim + dc;
        const int dp = __shfl_xor_sync(FULL, dc, 1);  // partner row (same batch)
        const int l_begin = t_begin * TL;
        const int n_tiles = t_end - t_begin;
        // chained: where the piece's state comes from and goes to
        const bool at_start = t_begin == 0, at_end = t_end == sch.nt;

        // states [8q, 8q+8) of [0] the own row and [1] the partner row, as pairs
        f2 A2[2][4], h[2][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = 8 * q + 2 * j;
            A2[0][j] = mk2(p.A[(long long)dc * kN + n] * kLog2e, p.A[(long long)dc * kN + n + 1] * kLog2e);
            A2[1][j] = mk2(p.A[(long long)dp * kN + n] * kLog2e, p.A[(long long)dp * kN + n + 1] * kLog2e);
        }
        // exact zero-order hold: 1 / a per state (an a of 0 is covered by the
        // series form below, which the factor then always selects)
        f2 ia[2][ZH ? 4 : 1];
        if constexpr (ZH) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = 8 * q + 2 * j;
                ia[0][j] = mk2(1.f / p.A[(long long)dc * kN + n], 1.f / p.A[(long long)dc * kN + n + 1]);
                ia[1][j] = mk2(1.f / p.A[(long long)dp * kN + n], 1.f / p.A[(long long)dp * kN + n + 1]);
            }
        }
        // initial state: zero (aggregate pass), h0 (first segment), the
        // carried-in state of the combine pass, or the chained carry
        {
            const float *src0 = nullptr, *src1 = nullptr;
            bool from_carry = false;
            if (MODE == kAgg) {
                // from zero
            } else if (MODE == kSeg && seg > 0) {
                src0 = sch.hagg + (((long long)rbi * sch.n_seg + seg - 1) * 32 + lane) * kN;
                src1 = sch.hagg + (((long long)rbi * sch.n_seg + seg - 1) * 32 + (lane ^ 1)) * kN;
                from_carry = true;
            } else if (MODE == kSeg || at_start) {
                if (p.h0) {
                    src0 = p.h0 + row * kN;
                    src1 = p.h0 + ((long long)b * p.dim + dp) * kN;
                }
            } else {
                // the tail of a split row block: wait for its head's carry. Only
                // this call's flag counts: one left by another call (any other
                // epoch) runs the bounded wait out and reports a timeout.
                const unsigned long long want = (sch.epoch << 16) | 1ull;
                bool ok = true;
                if (lane == 0) {
                    ok = false;
                    for (uint32_t i = 0; i < p.wait_limit; ++i) {
                        if (ld_acquire(sch.flags + rbi) == want) {
                            ok = true;
                            break;
                        }
                        __nanosleep(128);
                    }
                }
                ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
                if (!ok) {
                    if (lane == 0) set_error(p.err, SS_ERR_TIMEOUT);
                    failed = true;
                    break;
                }
                asm volatile("fence.acq_rel.gpu;" ::: "memory");
                src0 = sch.carry + ((long long)rbi * 32 + lane) * kN;
                src1 = sch.carry + ((long long)rbi * 32 + (lane ^ 1)) * kN;
                from_carry = true;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = 8 * q + 2 * j;
                if (src0) {
                    h[0][j] = from_carry ? mk2(__ldcg(src0 + n), __ldcg(src0 + n + 1))
                                         : mk2(src0[n], src0[n + 1]);
                    h[1][j] = from_carry ? mk2(__ldcg(src1 + n), __ldcg(src1 + n + 1))
                                         : mk2(src1[n], src1[n + 1]);
                } else {
                    h[0][j] = h[1][j] = mk2(0.f, 0.f);
                }
            }
        }
        const float bias = p.bias ? p.bias[dc] : 0.f;
        const float Dd = p.D ? p.D[dc] : 0.f;
        const Tin *g_u = static_cast<const Tin *>(p.u) + row * L;  // u, or the conv's x
        const Tin *g_dl = static_cast<const Tin *>(p.delta) + row * L;
        const Tin *g_z = has_z ? static_cast<const Tin *>(p.z) + row * L : g_u;
        float sdt = 0.f, sdt_c = 0.f;  // summed dt of the own row (aggregate pass), compensated

        // fused convolution (own row), kept in this lane's shared-memory slot
        // between tiles (registers are the scan's): the weights right-aligned in
        // 4 taps (a narrower filter has leading zero taps), the bias, and the 3
        // inputs before the next tile (earlier steps of x, else the initial
        // state, else zero)
        float *cslot = reinterpret_cast<float *>(smem + LY::OFF_CONV) + 8 * lane;
        if constexpr (CV) {
            const int W = p.conv_width;
            float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int k = 0; k < W; ++k) v[4 - W + k] = p.conv_w[(long long)dc * W + k];
            v[4] = p.conv_b ? p.conv_b[dc] : 0.f;
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const int idx = l_begin - 3 + j;  // step of x
                const int slot = (W - 1) + idx;   // slot of the initial state when idx < 0
                v[5 + j] = idx >= 0 ? to_f32(g_u[idx])
                                    : ((p.conv_init && slot >= 0)
                                           ? p.conv_init[row * (W - 1) + slot] : 0.f);
            }
            reinterpret_cast<float4 *>(cslot)[0] = make_float4(v[0], v[1], v[2], v[3]);
            reinterpret_cast<float4 *>(cslot)[1] = make_float4(v[4], v[5], v[6], v[7]);
        }

        // B/C tile k of this unit into ring stage (gt + k) % S
        auto issue_bc = [&](int k) {
            if (k < n_tiles && lane == 0 && (int)(gt + k) != p.drop_tile) {
                const int s = (int)((gt + k) % S);
                mbar_expect_tx(&bar[s], LY::BC_BOX);
                tma_load_2d(smem + s * LY::BC_BOX, &tm_bc, 0,
                            (int)((long long)b * L + l_begin + k * TL), &bar[s]);
            }
        };
        // this lane's u, delta, z for tile k: whole 32-byte sectors of its row
        auto load_streams = [&](int k, u8v (&su)[LY::NV], u8v (&sd)[LY::NV], u8v (&sz)[LY::NV]) {
            const long long off = (long long)l_begin + (long long)k * TL;
#pragma unroll
            for (int v = 0; v < LY::NV; ++v) {
                su[v] = ldg256(g_u + off + v * (32 / LY::ESZ));
                sd[v] = ldg256(g_dl + off + v * (32 / LY::ESZ));
                if (OUT && has_z) sz[v] = ldg256(g_z + off + v * (32 / LY::ESZ));
            }
        };

#pragma unroll
        for (int k = 0; k < S - 1; ++k) issue_bc(k);
        u8v nu[LY::NV], nd[LY::NV], nz[LY::NV];
        load_streams(0, nu, nd, nz);

        for (int k = 0; k < n_tiles; ++k) {
            issue_bc(k + S - 1);
            u8v cu[LY::NV], cd[LY::NV], cz[LY::NV];
#pragma unroll
            for (int v = 0; v < LY::NV; ++v) cu[v] = nu[v], cd[v] = nd[v], cz[v] = nz[v];
            if (k + 1 < n_tiles) load_streams(k + 1, nu, nd, nz);
            const uint32_t *uw = cu[0].w, *dw = cd[0].w, *zw = cz[0].w;
            (void)zw;
            // (for fp32 inputs the NV loads of a tensor are consecutive registers)

            // own row: u of the tile; with the fused convolution its output,
            // otherwise the loaded words, widened where they are used
            f2 uv[CV ? TL / 2 : 1] = {};
            auto u_at = [&](int i) -> f2 {
                if constexpr (CV) return uv[i];
                else return pair_at(uw, i, Tin());
            };
            if constexpr (CV) {
                // x of the tile and the 3 inputs before it: c[l] = cb + sum_k cw[k] x[l-3+k]
                const float4 s0 = reinterpret_cast<const float4 *>(cslot)[0];
                const float4 s1 = reinterpret_cast<const float4 *>(cslot)[1];
                const float cw[4] = {s0.x, s0.y, s0.z, s0.w}, cb = s1.x;
                float xv[TL + 3];
                xv[0] = s1.y, xv[1] = s1.z, xv[2] = s1.w;
#pragma unroll
                for (int i = 0; i < TL / 2; ++i) {
                    const f2 w2 = pair_at(uw, i, Tin());
                    xv[3 + 2 * i] = w2.x;
                    xv[3 + 2 * i + 1] = w2.y;
                }
#pragma unroll
                for (int i = 0; i < TL / 2; ++i) {
                    f2 c2 = mk2(cb, cb);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        c2 = ffma2(mk2(cw[k], cw[k]), mk2(xv[2 * i + k], xv[2 * i + 1 + k]), c2);
                    uv[i] = !p.conv_silu ? c2
                                         : ((SS_PAIR_TANH && sizeof(Tin) == 2) ? fmul2(c2, silu2_gate_tanh(c2))
                                                                             : fmul2(c2, silu2_gate(c2)));
                }
                reinterpret_cast<float4 *>(cslot)[1] = make_float4(cb, xv[TL], xv[TL + 1], xv[TL + 2]);
                if (OUT && p.u_out && row_ok) {
                    float uo[TL];
#pragma unroll
                    for (int i = 0; i < TL / 2; ++i) uo[2 * i] = uv[i].x, uo[2 * i + 1] = uv[i].y;
                    store_tile<TL>(static_cast<Tin *>(p.u_out) + row * (long long)L + l_begin + k * TL, uo);
                }
                if (OUT && p.conv_state && row_ok && k + 1 == n_tiles &&
                    (MODE == kSeg ? seg + 1 == sch.n_seg : at_end)) {
                    const int W = p.conv_width;
                    for (int j = 0; j < W - 1; ++j)
                        p.conv_state[row * (W - 1) + j] = xv[TL + 3 - (W - 1) + j];
                }
            }

            // own row: dt and dt*u for the tile (each (row, step) once)
            f2 dt[TL / 2], du[TL / 2];
#pragma unroll
            for (int i = 0; i < TL / 2; ++i) {
                const f2 x = fadd2(pair_at(dw, i, Tin()), mk2(bias, bias));
                // softplus: the degree-4 fit for bf16 inputs, degree 6 for fp32
                dt[i] = p.softplus ? (sizeof(Tin) == 2 ? softplus2_d4(x) : softplus2_d6(x)) : x;
                // the simplified input matrix takes dt * u; the zero-order hold
                // takes u (its factor is formed per state)
                du[i] = ZH ? u_at(i) : fmul2(dt[i], u_at(i));
            }
            if (MODE == kAgg) {
                // pairwise sum of the tile's dt, then a compensated running sum
                f2 s4[TL / 4];
#pragma unroll
                for (int i = 0; i < TL / 4; ++i) s4[i] = fadd2(dt[2 * i], dt[2 * i + 1]);
#pragma unroll
                for (int w = TL / 8; w >= 1; w /= 2)
#pragma unroll
                    for (int i = 0; i < w; ++i) s4[i] = fadd2(s4[i], s4[i + w]);
                const float ts = s4[0].x + s4[0].y;
                const float yk = ts - sdt_c, tk = sdt + yk;
                sdt_c = (tk - sdt) - yk;
                sdt = tk;
            }

            const long long g = gt + k;
            const int s = (int)(g % S);
            const bool ok = mbar_wait_bounded(&bar[s], (uint32_t)(g / S) & 1u, p.wait_limit);
            if (!__all_sync(FULL, ok)) {
                if (lane == 0) set_error(p.err, SS_ERR_TIMEOUT);
                for (int j = k + 1; j < k + S && j < n_tiles; ++j)
                    if ((int)(gt + j) != p.drop_tile)
                        mbar_wait_bounded(&bar[(gt + j) % S], (uint32_t)((gt + j) / S) & 1u,
                                          p.wait_limit);
                failed = true;
                break;
            }
            const float *bc = reinterpret_cast<const float *>(smem + s * LY::BC_BOX);

            // the recurrence for both rows of the pair, this lane's 8 states
            float out[TL];
            if constexpr (!OUT) {
#pragma unroll
                for (int l = 0; l < TL; ++l) {
                    const float dto = (l & 1) ? dt[l / 2].y : dt[l / 2].x;
                    const float duo = (l & 1) ? du[l / 2].y : du[l / 2].x;
                    const float dtp = __shfl_xor_sync(FULL, dto, 1);
                    const float dup = __shfl_xor_sync(FULL, duo, 1);
                    const float4 *bl = reinterpret_cast<const float4 *>(bc + l * 2 * kN + 8 * q);
                    const float4 b0 = bl[0], b1 = bl[1];
                    const f2 Bp[4] = {mk2(b0.x, b0.y), mk2(b0.z, b0.w), mk2(b1.x, b1.y), mk2(b1.z, b1.w)};
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const float dtr = r ? dtp : dto, dur = r ? dup : duo;
                        const f2 dd = mk2(dtr, dtr), uu = mk2(dur, dur);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const f2 tt = fmul2(dd, A2[r][j]);
                            const f2 e = mk2(ex2(tt.x), ex2(tt.y));
                            if constexpr (ZH)
                                h[r][j] = ffma2(e, h[r][j], zoh_input(tt, e, ia[r][j], dd, fmul2(uu, Bp[j])));
                            else
                                h[r][j] = ffma2(e, h[r][j], fmul2(uu, Bp[j]));
                        }
                    }
                }
            } else {
#pragma unroll
            for (int l = 0; l < TL; ++l) {
                const float dto = (l & 1) ? dt[l / 2].y : dt[l / 2].x;
                const float duo = (l & 1) ? du[l / 2].y : du[l / 2].x;
                const float dtp = __shfl_xor_sync(FULL, dto, 1);
                const float dup = __shfl_xor_sync(FULL, duo, 1);
                const float4 *bl = reinterpret_cast<const float4 *>(bc + l * 2 * kN + 8 * q);
                const float4 *cl = reinterpret_cast<const float4 *>(bc + l * 2 * kN + kN + 8 * q);
                const float4 b0 = bl[0], b1 = bl[1], c0 = cl[0], c1 = cl[1];
                const f2 Bp[4] = {mk2(b0.x, b0.y), mk2(b0.z, b0.w), mk2(b1.x, b1.y), mk2(b1.z, b1.w)};
                const f2 Cp[4] = {mk2(c0.x, c0.y), mk2(c0.z, c0.w), mk2(c1.x, c1.y), mk2(c1.z, c1.w)};
                float part[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float dtr = r ? dtp : dto, dur = r ? dup : duo;
                    const f2 dd = mk2(dtr, dtr), uu = mk2(dur, dur);
                    f2 a;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const f2 tt = fmul2(dd, A2[r][j]);
                        const f2 e = mk2(ex2(tt.x), ex2(tt.y));
                        if constexpr (ZH)
                            h[r][j] = ffma2(e, h[r][j], zoh_input(tt, e, ia[r][j], dd, fmul2(uu, Bp[j])));
                        else
                            h[r][j] = ffma2(e, h[r][j], fmul2(uu, Bp[j]));
                        // one accumulator chain over the 4 pairs (even and odd states)
                        a = j == 0 ? fmul2(Cp[0], h[r][0]) : ffma2(Cp[j], h[r][j], a);
                    }
                    part[r] = a.x + a.y;
                }
                // own total = my half of my row + the partner's half of my row
                out[l] = part[0] + __shfl_xor_sync(FULL, part[1], 1);
            }

            // chained head piece: its end state is known now; hand it on before
            // this tile's y stores are issued, so the fence that orders the carry
            // before the flag has no fresh stores to wait for
            if (MODE == kChain && k + 1 == n_tiles && !at_end) publish_carry(sch, rbi, lane, q, h);

            // own row: D skip and silu(z) gate
#pragma unroll
            for (int i = 0; i < TL / 2; ++i) {
                f2 o = ffma2(mk2(Dd, Dd), u_at(i), mk2(out[2 * i], out[2 * i + 1]));
                if (has_z)
                    o = fmul2(o, (SS_PAIR_TANH && sizeof(Tin) == 2) ? silu2_tanh(pair_at(zw, i, Tin()))
                                                                   : silu2(pair_at(zw, i, Tin())));
                out[2 * i] = o.x;
                out[2 * i + 1] = o.y;
            }
            if (row_ok) {
                Tout *dst = static_cast<Tout *>(p.y) + row * (long long)L + l_begin + k * TL;
                store_tile<TL>(dst, out);
            }
            }  // OUT
            __syncwarp();  // every lane is done with B/C stage s before it is refilled
        }
        if (failed) break;
        gt += n_tiles;

        if (MODE == kAgg) {
            // the segment's end state (from zero) and the own row's summed dt
            float *a0 = sch.hagg + (((long long)rbi * sch.n_seg + seg) * 32 + lane) * kN + 8 * q;
            float *a1 = sch.hagg + (((long long)rbi * sch.n_seg + seg) * 32 + (lane ^ 1)) * kN + 8 * q;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                __stcg(a0 + 2 * j, h[0][j].x);
                __stcg(a0 + 2 * j + 1, h[0][j].y);
                __stcg(a1 + 2 * j, h[1][j].x);
                __stcg(a1 + 2 * j + 1, h[1][j].y);
            }
            __stcg(sch.sdt + ((long long)rbi * sch.n_seg + seg) * 32 + lane, sdt);
            continue;
        }
        // the final state, once the row block's last tile is done (a chained
        // head piece handed its state on inside its last tile). Lane q holds
        // states [8q, 8q+8) of its own row and of the partner row.
        const bool last = MODE == kSeg ? seg + 1 == sch.n_seg : at_end;
        if (last && p.h_last) {
            if (row_ok) {
                float *hl = p.h_last + row * kN + 8 * q;
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    reinterpret_cast<float4 *>(hl)[j] = make_float4(
                        h[0][2 * j].x, h[0][2 * j].y, h[0][2 * j + 1].x, h[0][2 * j + 1].y);
            }
            if ((blk * 32 + (lane ^ 1)) < p.dim) {
                float *hp = p.h_last + ((long long)b * p.dim + dp) * kN + 8 * q;
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    reinterpret_cast<float4 *>(hp)[j] = make_float4(
                        h[1][2 * j].x, h[1][2 * j].y, h[1][2 * j + 1].x, h[1][2 * j + 1].y);
            }
        }
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// Per device and instantiation, once: allow the dynamic shared memory and ask
// how many one-warp CTAs of the kernel fit on an SM.
template <typename K>
int resident_ctas(K kern, int smem, int *out) {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SS_ERR_CUDA;
    if (cache[dev] == 0) {
        int per_sm = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32, smem) !=
                cudaSuccess)
            return SS_ERR_CUDA;
        cache[dev] = per_sm < 1 ? 1 : per_sm;
    }
    *out = cache[dev];
    return SS_OK;
}

template <typename Tin, typename Tout, int TL, int S, int MODE, int FL>
int launch_mode(const ssh::ScanParams &p, const ssh::PairWork &w, const PairSched &sch,
                const CUtensorMap &tm, long long units, cudaStream_t st) {
    using LY = PairLayout<Tin, TL, S>;
    auto kern = scan_pair_kernel<Tin, Tout, TL, S, MODE, FL>;
    int per_sm = 0;
    int rc = resident_ctas(kern, LY::TOTAL, &per_sm);
    if (rc != SS_OK) return rc;
    if (w.warps_per_sm > 0 && w.warps_per_sm < per_sm) per_sm = w.warps_per_sm;
    long long grid = (long long)per_sm * w.sm_count;
    if (grid > units) grid = units;
    if (grid < 1) return SS_OK;
    PairSched sc = sch;
    // chained: one range per warp (never more ranges than row blocks)
    sc.units = MODE == kChain ? grid : units;
    kern<<<(unsigned)grid, 32, LY::TOTAL, st>>>(tm, p, sc);
    return cudaPeekAtLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

template <typename Tin, typename Tout, int TL, int S, int FL>
int launch_cfg(const ssh::ScanParams &p, const ssh::PairWork &w, cudaStream_t st) {
    const long long L = p.seqlen;
    // 1. pack B/C, reset the work counters
    {
        const long long n = (long long)p.batch * L;
        bc_pack_kernel<Tin><<<(unsigned)((n + 255) / 256), 256, 0, st>>>(
            static_cast<const Tin *>(p.B), static_cast<const Tin *>(p.C), w.bc, L, p.batch,
            w.counter);
    }
    auto fn = encode_fn();
    if (!fn) return SS_ERR_CUDA;
    CUtensorMap tm;
    const cuuint64_t dims[2] = {(cuuint64_t)(2 * kN), (cuuint64_t)((long long)p.batch * L)};
    const cuuint64_t strides[1] = {(cuuint64_t)(2 * kN * 4)};
    const cuuint32_t box[2] = {(cuuint32_t)(2 * kN), (cuuint32_t)TL};
    const cuuint32_t estr[2] = {1, 1};
    if (fn(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, w.bc, dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return SS_ERR_CUDA;
    PairSched sch{};
    sch.rb_per_batch = (p.dim + 31) / 32;
    sch.total_rb = p.batch * sch.rb_per_batch;
    sch.nt = (int)(L / TL);
    sch.seg_len = (int)(((L + w.n_seg - 1) / w.n_seg + TL - 1) / TL * TL);
    sch.n_seg = (int)((L + sch.seg_len - 1) / sch.seg_len);
    sch.counter = w.counter;
    sch.flags = w.flags;
    sch.carry = w.carry;
    sch.BC = w.bc;
    sch.epoch = w.epoch;
    sch.hagg = w.hagg;
    sch.sdt = w.sdt;
    if (!w.chunked || sch.n_seg < 2) {
        // 2. one chained pass: at most one range per row block
        return launch_mode<Tin, Tout, TL, S, kChain, FL>(p, w, sch, tm, (long long)sch.total_rb, st);
    }
    // 2. aggregate every segment but the last, in parallel
    int rc = launch_mode<Tin, Tout, TL, S, kAgg, FL>(p, w, sch, tm,
                                                 (long long)sch.total_rb * (sch.n_seg - 1), st);
    if (rc != SS_OK) return rc;
    // 3. combine the segment maps along time: the state entering each segment
    {
        const long long warps = (long long)sch.total_rb * 32;
        carry_combine_kernel<<<(unsigned)((warps + 3) / 4), 128, 0, st>>>(p, sch);
        if (cudaPeekAtLastError() != cudaSuccess) return SS_ERR_CUDA;
    }
    // 4. every segment again from its carried-in state, writing y
    return launch_mode<Tin, Tout, TL, S, kSeg, FL>(p, w, sch, tm,
                                               (long long)sch.total_rb * sch.n_seg, st);
}

}  // namespace

size_t ssh::pair_bc_bytes(const ssh::ScanParams &p) {
    return (size_t)p.batch * (size_t)p.seqlen * 2 * kN * sizeof(float);
}
int ssh::pair_segments(const ssh::ScanParams &p, int requested) {
    const long long tl = SS_PAIR_TL;
    const long long seg_len = ((p.seqlen + requested - 1) / requested + tl - 1) / tl * tl;
    return (int)((p.seqlen + seg_len - 1) / seg_len);
}
size_t ssh::pair_agg_bytes(const ssh::ScanParams &p, int n_seg) {
    // end states and summed dt per (row block, segment)
    return (size_t)ssh::pair_row_blocks(p) * (size_t)n_seg * 32 * (kN + 1) * sizeof(float);
}
size_t ssh::pair_carry_bytes(const ssh::ScanParams &p) {
    return (size_t)p.batch * (size_t)((p.dim + 31) / 32) * 32 * kN * sizeof(float);
}
int ssh::pair_row_blocks(const ssh::ScanParams &p) { return p.batch * ((p.dim + 31) / 32); }

bool ssh::pair_supported(const ssh::ScanParams &p) {
    if (p.dstate != kN) return false;
    // whole tiles only: seqlen a multiple of the tile, so every row and every
    // tile of every tensor starts on a 32-byte boundary (given 32-byte aligned
    // base pointers)
    if (p.seqlen % SS_PAIR_TL != 0) return false;
    const void *ptrs[] = {p.u, p.delta, p.z, p.y};
    for (const void *q : ptrs)
        if (q && (reinterpret_cast<uintptr_t>(q) & 31u) != 0) return false;
    if ((long long)p.batch * p.seqlen >= (1LL << 31)) return false;
    return encode_fn() != nullptr;
}

template <int FL>
int launch_pair_t(const ssh::ScanParams &p, const ssh::PairWork &w, cudaStream_t st) {
    constexpr int TL = SS_PAIR_TL, S = SS_PAIR_S;
    const bool ib = p.in_dtype == SS_BF16, ob = p.out_dtype == SS_BF16;
    if (ib && ob) return launch_cfg<uint16_t, uint16_t, TL, S, FL>(p, w, st);
    if (ib) return launch_cfg<uint16_t, float, TL, S, FL>(p, w, st);
    if (ob) return launch_cfg<float, uint16_t, TL, S, FL>(p, w, st);
    return launch_cfg<float, float, TL, S, FL>(p, w, st);
}

int ssh::launch_pair(const ssh::ScanParams &p, const ssh::PairWork &w, cudaStream_t st) {
    if (p.conv_width > 0) {
        // the fused convolution serves the simplified input matrix only
        if (p.conv_width < 2 || p.conv_width > 4 || !p.conv_w || p.zoh) return SS_ERR_UNSUPPORTED;
        return launch_pair_t<kConv>(p, w, st);
    }
    if (p.zoh) return launch_pair_t<kZoh>(p, w, st);
    return launch_pair_t<kPlain>(p, w, st);
}
