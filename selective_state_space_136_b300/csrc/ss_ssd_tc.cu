// Mamba-2 state space duality (SSD) forward on the fifth-generation tensor
// cores: tcgen05 products with operands in shared memory and accumulators in
// tensor memory (TMEM).
//
// The computation is the chunked block decomposition of soft186.com,
// "Mamba选择性状态空间机制", section "状态空间对偶性算法突破" (the selective
// recurrence with A = a_h I per head, dt shared by the head's P channels, B and
// C shared by all heads), the same as the mma.sync kernel in ss_ssd.cu, with
// Q = 128-step chunks so that every product has M = 128 rows (one TMEM lane
// per row). Per chunk, with cum_t the running sum of dt_r a (log2 units):
//   G  = C B^T                                  (t x s over n)      -> TMEM
//   M  = G o exp2(cum_t - cum_s) dt_s, s <= t   (bf16, shared memory)
//   Y  = M X                                    (t x p over s)      -> TMEM
//   Z  = C H_prev                               (t x p over n; H as bf16 hi + lo)
//   y  = Y + exp2(cum_t) Z + D x
//   S  = exp2(cum_last) S + B^T Xs,  Xs[s] = x_s exp2(cum_last - cum_s) dt_s
// where S[n][p] is the carried state, kept in fp32 in TMEM for the whole row
// of chunks and copied to shared memory as bf16 hi + lo for the next Z.
//
// One CTA of 16 warps per (batch, head). Warp w reads TMEM lanes
// [32 (w % 4), 32 (w % 4) + 32) (rows t of G, Y, Z; rows n of S) and takes
// part w / 4 of four of each epilogue's columns. Thread 0 issues the MMAs: G,
// then at once Z (it needs only C and the previous state), S as soon as Xs and
// the rescaled state are in place, and Y after the mask; G and the chunk's
// last product are committed to one mbarrier each, so Z and S run under the
// CUDA-core phases (Xs, rescale, mask) and only Y is waited for at the end.
// Warp 0 forms the next chunk's dt and its prefix sum while Y runs. C and B
// arrive by TMA into two buffers, the next chunk's issued at this one's start;
// the next chunk's x waits in registers.
// y leaves through a 128-byte-swizzled shared tile (the masked tile's buffer,
// free once Y is done) by TMA stores, whole rows at a time. The mask's
// exponentials below the diagonal 32 x 32 band are factored per 16-column
// block with end e: exp2(cum_t - cum_s) = exp2(cum_t - cum_e) exp2(cum_e -
// cum_s), both factors at most 1 (cum falls along the chunk), one exponential
// per row and block plus one per column, instead of one per element. Shared
// operand tiles are stored as 8-row x 16-byte core matrices, column blocks
// fastest, and described to the tensor core without swizzling: K-major tiles
// (C, B, M) with the leading offset between K-adjacent core matrices and the
// stride offset between 8-row groups; MN-major tiles (X, Xs, H, and B read as
// B^T) the other way round.
#include <cudaTypedefs.h>

#include "ss_common.cuh"
#include "ss_internal.h"

namespace {

using namespace ssk;

constexpr int kQ = 128;  // chunk length = MMA rows
constexpr int kP = 64;   // head dimension
constexpr int kN = 128;  // state size
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColG = 0;    // G (128 columns)
constexpr uint32_t kColY = 128;  // Y (64)
constexpr uint32_t kColS = 192;  // carried state S (64)
constexpr uint32_t kColZ = 256;  // Z: C H_hi in 64, C H_lo in 64

struct TcSmem {
    uint16_t C[2][kQ * kN];  // C of the chunk [t][n], K-major for G and Z (two buffers)
    uint16_t B[2][kQ * kN];  // B of the chunk [s][n]: K-major for G, MN-major (B^T) for S
    uint16_t M[kQ * kQ];     // masked G [t][s], K-major for Y
    uint16_t X[kQ * kP];     // x of the chunk [s][p], MN-major for Y
    uint16_t Xs[kQ * kP];    // scaled x [s][p], MN-major for S
    uint16_t H[kN * 2 * kP];  // carried state [n][hi p | lo p]: bf16 high part, then S - hi;
                              // MN-major B of one 128-column Z product
    float dt[kQ];
    float cum[kQ];
    float W[kQ];  // exp2(cum_e - cum_s) dt_s, e the last step of s's 16-column block
    uint64_t bar;      // G of the chunk done
    uint64_t bars;     // Z and S of the chunk done (committed after S)
    uint64_t bary;     // every product of the chunk done (committed after Y)
    uint64_t bardrain; // after a wait that gave up: whatever was issued is done
    uint64_t cbar[2];  // TMA arrival of C and B into buffer 0 / 1
    uint32_t tmem;
};

// Byte offset of element (r, c) of a bf16 tile with `cols` columns stored as
// 8-row x 16-byte core matrices, the column blocks of an 8-row group adjacent.
__device__ __forceinline__ uint32_t cm_off(int r, int c, int cols) {
    return ((((r >> 3) * (cols >> 3)) + (c >> 3)) << 7) + ((r & 7) << 4) + ((c & 7) << 1);
}

// Shared-memory matrix descriptor without swizzling: start address, leading
// and stride byte offsets (all in 16-byte units), descriptor version 1.
__device__ __forceinline__ uint64_t sdesc(const void *p, uint32_t byte_off, uint32_t lbo,
                                          uint32_t sbo) {
    const uint32_t a = smem_u32(p) + byte_off;
    return (uint64_t)((a >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, A/B
// MN-major flags, N >> 3 and M >> 4.
constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kIdG = idesc_bf16(kQ, kQ, 0, 0);  // G: C (K-major) x B (K-major)
constexpr uint32_t kIdY = idesc_bf16(kQ, kP, 0, 1);      // Y: K-major A x MN-major B
constexpr uint32_t kIdZ = idesc_bf16(kQ, 2 * kP, 0, 1);  // Z: C x [H_hi | H_lo]
constexpr uint32_t kIdS = idesc_bf16(kN, kP, 1, 1);  // S: B^T (MN-major) x Xs (MN-major)
// descriptor offsets (bytes)
constexpr uint32_t kKmLbo = 128, kKmSbo = 128 * (kQ / 8);  // K-major 128-column tiles
constexpr uint32_t kKmStep = 256;                          // 16 columns of K
constexpr uint32_t kMn64Lbo = 128 * (kP / 8), kMn64Sbo = 128, kMn64Step = 2 * kMn64Lbo;
constexpr uint32_t kMn128Lbo = 128 * (kN / 8), kMn128Sbo = 128, kMn128Step = 2 * kMn128Lbo;

// A descriptor advanced by `bytes` along its start address (no carry out of
// the 14-bit field: every tile lies within the first 256 KB of shared memory).
__device__ __forceinline__ uint64_t dadv(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t ad, uint64_t bd, uint32_t id,
                                        bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(ad), "l"(bd), "r"(id), "r"((uint32_t)accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 16 consecutive fp32 columns of this thread's TMEM lane; the wait is part of
// the same statement, so the registers are valid when it returns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];\n\ttcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// 2 x 16 fp32 columns of this thread's TMEM lane with one wait for all.
__device__ __forceinline__ void tmem_ld16x2(uint32_t a0, uint32_t a1, float (&v0)[16], float (&v1)[16]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(a0), "r"(a1)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v0[i] = __uint_as_float(r[0 + i]);
#pragma unroll
    for (int i = 0; i < 16; ++i) v1[i] = __uint_as_float(r[16 + i]);
}
// 3 x 16 fp32 columns of this thread's TMEM lane with one wait for all.
__device__ __forceinline__ void tmem_ld16x3(uint32_t a0, uint32_t a1, uint32_t a2, float (&v0)[16],
                                            float (&v1)[16], float (&v2)[16]) {
    uint32_t r[48];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%48];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%49];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%50];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47])
        : "r"(a0), "r"(a1), "r"(a2)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v0[i] = __uint_as_float(r[0 + i]);
#pragma unroll
    for (int i = 0; i < 16; ++i) v1[i] = __uint_as_float(r[16 + i]);
#pragma unroll
    for (int i = 0; i < 16; ++i) v2[i] = __uint_as_float(r[32 + i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 4D tiled TMA load global -> shared, completion signalled on `bar`.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *tm, int c0, int c1,
                                            int c2, int c3, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_u32(bar))
        : "memory");
}

// 2D TMA store shared -> global of one box (bulk group of the issuing thread).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *tm, int x, int y, const void *src) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            reinterpret_cast<uint64_t>(tm)),
        "r"(x), "r"(y), "r"(smem_u32(src))
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// the shared-memory sources of every committed store have been read
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Byte offset of 16-byte piece j of row r in a tile of 128-byte rows stored
// with the 128-byte swizzle (piece index XOR row mod 8).
__device__ __forceinline__ uint32_t sw128(int r, int j) {
    return (uint32_t)(r * 128 + ((j ^ (r & 7)) << 4));
}

// Global loads kept in program order (volatile): issued where written, one
// chunk ahead of their use, rather than moved next to it.
__device__ __forceinline__ uint4 ldg_v4_ordered(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint16_t ldg_u16_ordered(const void *p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return a | (b << 16);
}
__device__ __forceinline__ float round_bf16(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
}

// Row n of the state (16 columns at p0) as bf16 hi and lo parts into the H tile.
__device__ __forceinline__ void put_state16(uint8_t *hs, int n, int p0, const float (&v)[16]) {
    uint32_t wh[8], wl[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float h0 = round_bf16(v[2 * j]), h1 = round_bf16(v[2 * j + 1]);
        wh[j] = pack2(h0, h1);
        wl[j] = pack2(v[2 * j] - h0, v[2 * j + 1] - h1);
    }
    constexpr int W = 2 * kP;
    *reinterpret_cast<uint4 *>(hs + cm_off(n, p0, W)) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
    *reinterpret_cast<uint4 *>(hs + cm_off(n, p0 + 8, W)) = make_uint4(wh[4], wh[5], wh[6], wh[7]);
    *reinterpret_cast<uint4 *>(hs + cm_off(n, kP + p0, W)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
    *reinterpret_cast<uint4 *>(hs + cm_off(n, kP + p0 + 8, W)) = make_uint4(wl[4], wl[5], wl[6], wl[7]);
}

// Bounded wait for an MMA commit: polls mbarrier.try_wait (which itself
// suspends for a while) without sleeping in between.
__device__ __forceinline__ bool mma_wait(uint64_t *bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// 16 y values of row t, channels c .. c + 15 of the head, into the staging
// tile: fp32 output as two boxes of 32 channels (16 KB each), bf16 as one box
// of 64 channels; 128-byte rows, swizzled.
__device__ __forceinline__ void stage16(uint8_t *st, int t, int c, const float (&v)[16], float) {
    uint8_t *box = st + (c >> 5) * (kQ * 128);
    const int j0 = (c & 31) >> 2;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        *reinterpret_cast<float4 *>(box + sw128(t, j0 + j)) =
            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}
__device__ __forceinline__ void stage16(uint8_t *st, int t, int c, const float (&v)[16], uint16_t) {
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = pack2(v[2 * j], v[2 * j + 1]);
    const int j0 = c >> 3;
    *reinterpret_cast<uint4 *>(st + sw128(t, j0)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4 *>(st + sw128(t, j0 + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
}

constexpr int kThreads = 512;  // 16 warps: warp w serves TMEM lanes 32 (w % 4) .. +32 and
                               // column part w / 4 of each epilogue
constexpr int kParts = kThreads / 128;  // warps per TMEM lane quarter
constexpr int kCols = kP / kParts;      // this thread's columns of Y, Z and S

template <typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
    ssd_tc_kernel(const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ CUtensorMap tm_c,
                  const __grid_constant__ CUtensorMap tm_b, const ssh::SsdParams p) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned: the y staging tile (in M) is read with the 128-byte swizzle
    TcSmem &sm = *reinterpret_cast<TcSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sM = reinterpret_cast<uint8_t *>(sm.M), *sX = reinterpret_cast<uint8_t *>(sm.X);
    uint8_t *sXs = reinterpret_cast<uint8_t *>(sm.Xs);
    uint8_t *sH = reinterpret_cast<uint8_t *>(sm.H);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, part = warp >> 2;
    const int r = 32 * quarter + lane;  // this thread's TMEM lane: row t of G, Y, Z; row n of S
    const int b = blockIdx.x / p.heads, h = blockIdx.x % p.heads;
    const long long L = p.seqlen;
    const float a = p.A[h] * kLog2e;  // log2 units
    const float bias = p.dt_bias ? p.dt_bias[h] : 0.f;
    const float Dh = p.D ? p.D[h] : 0.f;
    const long long xs_t = (long long)p.heads * kP;  // x / y stride between steps
    const uint16_t *gx = static_cast<const uint16_t *>(p.x);
    const uint16_t *gdt = static_cast<const uint16_t *>(p.dt);
    const long long st_base = ((long long)b * p.heads + h) * kP * kN;  // h0 / h_last (p, n)
    const int n_chunks = (int)(L / kQ);

    // The 16-byte pieces of a tile moved by one warp instruction: 8 rows (lane
    // mod 8) by 4 adjacent pieces (lane / 8), so the global side reads 8 rows x
    // 64 contiguous bytes (16 whole sectors) and each group of 8 lanes writes 8
    // rows of one core matrix (distinct banks). Block k of warp w is block
    // w + 8 k of the tile's (rows / 8) x (pieces / 4) blocks, pieces fastest.
    auto piece = [&](int k, int blocks_per_row_group, int &row, int &pc) {
        const int blk = warp + (kThreads / 32) * k;
        row = 8 * (blk / blocks_per_row_group) + (lane & 7);
        pc = 4 * (blk % blocks_per_row_group) + (lane >> 3);
    };
    // C and B of chunk c into buffer c & 1 by TMA (thread 0): each tile is a 4D
    // box (n mod 8, t mod 8, n / 8, t / 8) whose shared-memory image is the
    // core-matrix layout of cm_off; one mbarrier per buffer counts the bytes.
    auto issue_cb = [&](int c) {
        uint64_t *cb = &sm.cbar[c & 1];
        mbar_expect_tx(cb, 2u * kQ * kN * 2u);
        const int g8 = (int)(((long long)b * L + (long long)c * kQ) / 8);
        tma_load_4d(sm.C[c & 1], &tm_c, 0, 0, 0, g8, cb);
        tma_load_4d(sm.B[c & 1], &tm_b, 0, 0, 0, g8, cb);
    };
    // x of chunk c: this thread's four 16-byte pieces, into registers
    constexpr int kXPieces = kQ * kP / 8 / kThreads;
    auto load_x = [&](int c, uint4 (&xr)[kXPieces]) {
        const long long l0 = (long long)c * kQ;
#pragma unroll
        for (int k = 0; k < kXPieces; ++k) {
            int s, p8;
            piece(k, kP / 32, s, p8);
            xr[k] = ldg_v4_ordered(gx + ((long long)b * L + l0 + s) * xs_t + (long long)h * kP + 8 * p8);
        }
    };
    // raw dt of chunk c, four steps per lane of warp 0
    auto load_dt = [&](int c, uint16_t (&dr)[4]) {
        const long long l0 = (long long)c * kQ;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            dr[k] = ldg_u16_ordered(gdt + ((long long)b * L + l0 + 4 * lane + k) * p.heads + h);
    };

    // dt, its running sum (times a, log2 units) and the block weights W of a
    // chunk from raw dt, four steps per lane of warp 0, into registers
    auto dt_scan = [&](const uint16_t (&raw)[4], float (&d4)[4], float (&c4)[4], float (&w4)[4]) {
        float run = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float xv = to_f32(raw[k]) + bias;
            d4[k] = p.softplus ? softplus1(xv) : xv;
            run += d4[k] * a;
            c4[k] = run;
        }
        float incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        const float before = incl - run;
#pragma unroll
        for (int k = 0; k < 4; ++k) c4[k] += before;
        // the block of 16 steps is 4 lanes; its last step is lane | 3's fourth
        const float ce = __shfl_sync(0xffffffffu, c4[3], lane | 3);
#pragma unroll
        for (int k = 0; k < 4; ++k) w4[k] = ex2(ce - c4[k]) * d4[k];
    };
    auto dt_put = [&](const float (&d4)[4], const float (&c4)[4], const float (&w4)[4]) {
        *reinterpret_cast<float4 *>(&sm.dt[4 * lane]) = make_float4(d4[0], d4[1], d4[2], d4[3]);
        *reinterpret_cast<float4 *>(&sm.cum[4 * lane]) = make_float4(c4[0], c4[1], c4[2], c4[3]);
        *reinterpret_cast<float4 *>(&sm.W[4 * lane]) = make_float4(w4[0], w4[1], w4[2], w4[3]);
    };

    if (warp == 0) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                smem_u32(&sm.tmem)),
            "r"(kTmemCols)
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        mbar_init(&sm.bars, 1);
        mbar_init(&sm.bary, 1);
        mbar_init(&sm.bardrain, 1);
        mbar_init(&sm.cbar[0], 1);
        mbar_init(&sm.cbar[1], 1);
        fence_mbar_init();
    }
    uint4 xr[kXPieces];
    uint16_t dr[4] = {0, 0, 0, 0};
    float nd[4] = {0.f, 0.f, 0.f, 0.f}, nc[4] = {0.f, 0.f, 0.f, 0.f}, nw[4] = {0.f, 0.f, 0.f, 0.f};
    // chunk c's C/B use buffer c & 1 for the (c / 2)-th time: its arrival is
    // phase c / 2 of that buffer's barrier. Thread 0 tracks the last chunk whose
    // loads it issued and the last it saw arrive.
    int cb_issued = -1, cb_arrived = -1;
    tc_fence_before();
    __syncthreads();  // the barriers are initialised before the first TMA uses one
    tc_fence_after();
    if (n_chunks > 0) {
        if (tid == 0) {
            issue_cb(0);
            cb_issued = 0;
        }
        load_x(0, xr);
        if (warp == 0) {
            load_dt(0, dr);
            dt_scan(dr, nd, nc, nw);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem;
    const uint32_t trow = tmem + ((uint32_t)(32 * quarter) << 16);  // this warp's lanes
    const int c0 = kCols * part;  // this thread's columns of Y, Z and S

    // initial state: row n = r, columns [c0, c0 + kCols) of S (tensor memory) and of H
#pragma unroll
    for (int j = 0; j < kCols / 16; ++j) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            v[i] = p.h0 ? p.h0[st_base + (long long)(c0 + 16 * j + i) * kN + r] : 0.f;
        tmem_st16(trow + kColS + c0 + 16 * j, v);
        put_state16(sH, r, c0 + 16 * j, v);
    }
    tmem_wait_st();

    uint32_t phase = 0;
    bool timed_out = false;
    for (int c = 0; c < n_chunks; ++c) {
        const long long l0 = (long long)c * kQ;
        const uint8_t *sC = reinterpret_cast<const uint8_t *>(sm.C[c & 1]);
        const uint8_t *sB = reinterpret_cast<const uint8_t *>(sm.B[c & 1]);
        __syncthreads();  // every reader of the previous chunk's tiles is done
        // ---- x of the chunk from registers into its tile; dt and its prefix sum
#pragma unroll
        for (int k = 0; k < kXPieces; ++k) {
            int s, p8;
            piece(k, kP / 32, s, p8);
            *reinterpret_cast<uint4 *>(sX + cm_off(s, 8 * p8, kP)) = xr[k];
        }
        if (warp == 0) dt_put(nd, nc, nw);  // formed during the previous chunk
        const bool more = c + 1 < n_chunks;
        bool cb_late = false;
        // ---- the next chunk's operands start moving now
        if (tid == 0) {
            if (more) {  // buffer (c + 1) & 1 was last read by chunk c - 1's products
                issue_cb(c + 1);
                cb_issued = c + 1;
            }
            // this chunk's C and B have landed
            cb_late = !mbar_wait_bounded(&sm.cbar[c & 1], (c >> 1) & 1, p.wait_limit);
            if (!cb_late) cb_arrived = c;
        }
        if (more) {
            load_x(c + 1, xr);
            if (warp == 0) load_dt(c + 1, dr);
        }
        fence_proxy_async();
        tc_fence_before();
        if (__syncthreads_or(cb_late)) {
            if (tid == 0) set_error(p.err, SS_ERR_TIMEOUT);
            timed_out = true;
            break;
        }
        tc_fence_after();

        // ---- G = C B^T into TMEM columns [0, 128). The descriptors are formed by
        // the whole of warp 0 (warp-uniform values) and lane 0 issues.
        if (warp == 0) {
            const uint64_t dC = sdesc(sC, 0, kKmLbo, kKmSbo), dB = sdesc(sB, 0, kKmLbo, kKmSbo);
            const uint64_t dH = sdesc(sH, 0, kMn128Lbo, kMn128Sbo);
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < kN / 16; ++k)
                    mma_f16(tmem + kColG, dadv(dC, k * kKmStep), dadv(dB, k * kKmStep), kIdG, k > 0);
                mma_commit(&sm.bar);
                // Z = C [H_hi | H_lo] (H written by the previous chunk, fenced at the chunk start)
#pragma unroll
                for (int k = 0; k < kN / 16; ++k)
                    mma_f16(tmem + kColZ, dadv(dC, k * kKmStep), dadv(dH, k * kMn128Step), kIdZ, k > 0);
            }
            __syncwarp();
        }
        const float cum_last = sm.cum[kQ - 1];
        // ---- meanwhile: Xs (row s = r, this part's pieces) and S scaled by
        // the chunk's decay in place (row r, this part's columns)
        {
            const int s = r;
            const float w = ex2(cum_last - sm.cum[s]) * sm.dt[s];
#pragma unroll
            for (int k = 0; k < kP / 8 / kParts; ++k) {
                const int p8 = (kP / 8 / kParts) * part + k;
                const uint4 v = *reinterpret_cast<const uint4 *>(sX + cm_off(s, 8 * p8, kP));
                const uint4 o = make_uint4(pack2(bf16lo(v.x) * w, bf16hi(v.x) * w),
                                           pack2(bf16lo(v.y) * w, bf16hi(v.y) * w),
                                           pack2(bf16lo(v.z) * w, bf16hi(v.z) * w),
                                           pack2(bf16lo(v.w) * w, bf16hi(v.w) * w));
                *reinterpret_cast<uint4 *>(sXs + cm_off(s, 8 * p8, kP)) = o;
            }
            const float dec = ex2(cum_last);
#pragma unroll
            for (int j = 0; j < kCols / 16; ++j) {
                float v0[16];
                tmem_ld16(trow + kColS + c0 + 16 * j, v0);
#pragma unroll
                for (int i = 0; i < 16; ++i) v0[i] *= dec;
                tmem_st16(trow + kColS + c0 + 16 * j, v0);
            }
            tmem_wait_st();
        }
        if (tid == 0) bulk_wait_read();  // the previous chunk's y has left the M buffer
        fence_proxy_async();  // Xs is visible to the tensor core
        tc_fence_before();
        if (__syncthreads_or(!mma_wait(&sm.bar, phase, p.wait_limit))) {
            if (tid == 0) set_error(p.err, SS_ERR_TIMEOUT);
            timed_out = true;
            break;
        }
        tc_fence_after();
        // ---- S += B^T Xs (the rescaled state and Xs are in place)
        if (warp == 0) {
            const uint64_t dBt = sdesc(sB, 0, kMn128Lbo, kMn128Sbo);
            const uint64_t dXs = sdesc(sXs, 0, kMn64Lbo, kMn64Sbo);
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < kQ / 16; ++k)
                    mma_f16(tmem + kColS, dadv(dBt, k * kMn128Step), dadv(dXs, k * kMn64Step), kIdS, true);
                mma_commit(&sm.bars);
            }
            __syncwarp();
        }

        // ---- M = G o exp2(cum_t - cum_s) dt_s (s <= t), row t = r; the 16-column
        // pieces left of and on this quarter's band, dealt round the parts
        {
            const int t = r;
            const float ct = sm.cum[t];
            // this warp's pieces j = part, part + kParts, ... below 2 (quarter + 1), two per load
            // pieces left of the band (s0 + 16 <= 32 quarter <= t for every lane of
            // the warp) take the factored form; the band's two pieces the direct one
            auto mask_piece = [&](int s0, const float (&g)[16]) {
                uint32_t w[8];
                if (s0 + 16 <= 32 * quarter) {
                    const float E = ex2(ct - sm.cum[s0 + 15]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int s = s0 + 2 * i;
                        w[i] = pack2(g[2 * i] * E * sm.W[s], g[2 * i + 1] * E * sm.W[s + 1]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int s = s0 + 2 * i;
                        const float m0 = s <= t ? g[2 * i] * ex2(ct - sm.cum[s]) * sm.dt[s] : 0.f;
                        const float m1 = s + 1 <= t
                                             ? g[2 * i + 1] * ex2(ct - sm.cum[s + 1]) * sm.dt[s + 1]
                                             : 0.f;
                        w[i] = pack2(m0, m1);
                    }
                }
                *reinterpret_cast<uint4 *>(sM + cm_off(t, s0, kQ)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(sM + cm_off(t, s0 + 8, kQ)) =
                    make_uint4(w[4], w[5], w[6], w[7]);
            };
            // right of the band s > t: zeros (the buffer held the last chunk's y)
            for (int s8 = 4 * (quarter + 1) + part; s8 < kQ / 8; s8 += kParts)
                *reinterpret_cast<uint4 *>(sM + cm_off(t, 8 * s8, kQ)) = make_uint4(0u, 0u, 0u, 0u);
            const int np = 2 * (quarter + 1);
            for (int j = part; j < np; j += 2 * kParts) {
                const int s0 = 16 * j;
                if (j + kParts < np) {
                    float g0[16], g1[16];
                    tmem_ld16x2(trow + kColG + s0, trow + kColG + s0 + 16 * kParts, g0, g1);
                    mask_piece(s0, g0);
                    mask_piece(s0 + 16 * kParts, g1);
                } else {
                    float g0[16];
                    tmem_ld16(trow + kColG + s0, g0);
                    mask_piece(s0, g0);
                }
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- Y = M X; the commit covers every product of the chunk
        if (warp == 0) {
            const uint64_t dM = sdesc(sM, 0, kKmLbo, kKmSbo), dX = sdesc(sX, 0, kMn64Lbo, kMn64Sbo);
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < kQ / 16; ++k)
                    mma_f16(tmem + kColY, dadv(dM, k * kKmStep), dadv(dX, k * kMn64Step), kIdY, k > 0);
                mma_commit(&sm.bary);
            }
            __syncwarp();
        }
        // meanwhile: the next chunk's dt, running sum and block weights (its raw
        // dt was loaded at this chunk's start)
        if (warp == 0 && more) dt_scan(dr, nd, nc, nw);
        // meanwhile too: the new state's row n = r (this part's columns) into H
        // for the next chunk's Z; Z and S are done (this chunk's Z has read H)
        const bool s_ok = mma_wait(&sm.bars, phase, p.wait_limit);
        if (s_ok) {
            tc_fence_after();
            const int n = r;
#pragma unroll
            for (int j = 0; j < kCols / 16; ++j) {
                float v0[16];
                tmem_ld16(trow + kColS + c0 + 16 * j, v0);
                put_state16(sH, n, c0 + 16 * j, v0);
            }
        }
        if (__syncthreads_or(!s_ok || !mma_wait(&sm.bary, phase, p.wait_limit))) {
            if (tid == 0) set_error(p.err, SS_ERR_TIMEOUT);
            timed_out = true;
            break;
        }
        phase ^= 1u;  // both barriers complete one phase per chunk
        tc_fence_after();

        // ---- y row t = r, this part's channels, into the staging tile (the M
        // buffer) and out by TMA
        {
            const int t = r;
            const float ft = ex2(sm.cum[t]);
            auto finish = [&](int j, float (&yv)[16], const float (&zh)[16], const float (&zl)[16]) {
                const uint4 x0 = *reinterpret_cast<const uint4 *>(sX + cm_off(t, c0 + 16 * j, kP));
                const uint4 x1 = *reinterpret_cast<const uint4 *>(sX + cm_off(t, c0 + 16 * j + 8, kP));
                const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    yv[2 * i] = fmaf(Dh, bf16lo(xw[i]), fmaf(ft, zh[2 * i] + zl[2 * i], yv[2 * i]));
                    yv[2 * i + 1] = fmaf(Dh, bf16hi(xw[i]),
                                         fmaf(ft, zh[2 * i + 1] + zl[2 * i + 1], yv[2 * i + 1]));
                }
                stage16(sM, t, c0 + 16 * j, yv, Tout());
            };
#pragma unroll
            for (int j = 0; j < kCols / 16; ++j) {
                float y0[16], zh0[16], zl0[16];
                tmem_ld16x3(trow + kColY + c0 + 16 * j, trow + kColZ + c0 + 16 * j,
                            trow + kColZ + kP + c0 + 16 * j, y0, zh0, zl0);
                finish(j, y0, zh0, zl0);
            }
        }
        fence_proxy_async();  // the staged y is visible to the TMA unit
        __syncthreads();
        if (tid == 0) {
            const int yrow = (int)((long long)b * L + l0);
            if (sizeof(Tout) == 4) {
                tma_store_2d(&tm_y, h * kP, yrow, sM);
                tma_store_2d(&tm_y, h * kP + 32, yrow, sM + kQ * 128);
            } else {
                tma_store_2d(&tm_y, h * kP, yrow, sM);
            }
            bulk_commit();
        }
    }
    if (tid == 0) {
        bulk_wait_all();  // the y stores have completed
        // after a wait that gave up: C/B loads still in flight land before exit
        for (int k = cb_arrived + 1; k <= cb_issued; ++k)
            if (!mbar_wait_bounded(&sm.cbar[k & 1], (k >> 1) & 1, p.wait_limit)) break;
    }
    // after a wait that gave up: one more commit tracks every product issued so
    // far; give it a bounded wait before their tensor memory is freed
    if (timed_out) {
        if (tid == 0) mma_commit(&sm.bardrain);
        mma_wait(&sm.bardrain, 0, p.wait_limit);
    }

    if (p.h_last) {
#pragma unroll
        for (int j = 0; j < kCols / 16; ++j) {
            float v0[16];
            tmem_ld16(trow + kColS + c0 + 16 * j, v0);
#pragma unroll
            for (int i = 0; i < 16; ++i) p.h_last[st_base + (long long)(c0 + 16 * j + i) * kN + r] = v0[i];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
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

template <typename Tout>
int ssd_tc_t(const ssh::SsdParams &p, cudaStream_t st) {
    const int smem = (int)sizeof(TcSmem) + 1024;
    auto kern = ssd_tc_kernel<Tout>;
    // y as rows of heads * 64 channels, one row per (batch, step); boxes of 128
    // rows by 128 bytes (32 fp32 or 64 bf16 channels), 128-byte swizzle
    auto fn = encode_fn();
    if (!fn) return SS_ERR_UNSUPPORTED;
    CUtensorMap tm;
    const cuuint64_t dims[2] = {(cuuint64_t)p.heads * kP, (cuuint64_t)p.batch * p.seqlen};
    const cuuint64_t strides[1] = {(cuuint64_t)p.heads * kP * sizeof(Tout)};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / sizeof(Tout)), (cuuint32_t)kQ};
    const cuuint32_t estr[2] = {1, 1};
    if (fn(&tm, sizeof(Tout) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
           2, p.y, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return SS_ERR_UNSUPPORTED;
    // C and B (batch, L, N) bf16 as 4D boxes (n mod 8, t mod 8, n / 8, t / 8):
    // strides 2 B, 256 B, 16 B and 2048 B; a box of 8 x 8 x 16 x 16 is one
    // 128 x 128 tile in core-matrix order
    CUtensorMap tc_, tb_;
    {
        const cuuint64_t d4[4] = {8, 8, (cuuint64_t)kN / 8, (cuuint64_t)p.batch * p.seqlen / 8};
        const cuuint64_t s4[3] = {(cuuint64_t)kN * 2, 16, (cuuint64_t)kN * 2 * 8};
        const cuuint32_t b4[4] = {8, 8, (cuuint32_t)kN / 8, (cuuint32_t)kQ / 8};
        const cuuint32_t e4[4] = {1, 1, 1, 1};
        const void *bases[2] = {p.C, p.B};
        CUtensorMap *maps[2] = {&tc_, &tb_};
        for (int i = 0; i < 2; ++i)
            if (fn(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(bases[i]), d4,
                   s4, b4, e4, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return SS_ERR_UNSUPPORTED;
    }
    static bool done[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SS_ERR_CUDA;
    if (!done[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return SS_ERR_CUDA;
        done[dev] = true;
    }
    kern<<<(unsigned)((long long)p.batch * p.heads), kThreads, smem, st>>>(tm, tc_, tb_, p);
    return cudaPeekAtLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

}  // namespace

bool ssh::ssd_tc_supported(const ssh::SsdParams &p) {
    // y, C and B move by TMA: 16-byte aligned bases and (batch, step) rows
    // indexable in 32 bits
    return p.in_dtype == SS_BF16 && p.headdim == kP && p.dstate == kN && p.seqlen % kQ == 0 &&
           (long long)p.batch * p.heads < (1LL << 31) &&
           (long long)p.batch * p.seqlen < (1LL << 31) &&
           ((reinterpret_cast<uintptr_t>(p.y) | reinterpret_cast<uintptr_t>(p.B) |
             reinterpret_cast<uintptr_t>(p.C)) & 15u) == 0 &&
           encode_fn() != nullptr;
}

int ssh::launch_ssd_tc(const ssh::SsdParams &p, cudaStream_t st) {
    if (!ssd_tc_supported(p)) return SS_ERR_UNSUPPORTED;
    return p.out_dtype == SS_BF16 ? ssd_tc_t<uint16_t>(p, st) : ssd_tc_t<float>(p, st);
}
