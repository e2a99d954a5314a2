// Causal depthwise 1D convolution of the Mamba block and its decode step.
//
// "Mamba: Linear-Time Sequence Modeling with Selective State Spaces", section
// "Key terms": the Mamba block puts a 1D convolution in front of the
// selective SSM; soft186.com, "Mamba选择性状态空间机制", section
// "基础模型构建": its width is d_conv = 4, and the convolution is causal (the
// causal-conv1d package). Per row (b, d) with W = width:
//     out[l] = bias[d] + sum_{k<W} w[d,k] * xin(l - (W-1) + k)
// where xin(j < 0) comes from the optional initial state (the W-1 inputs
// before step 0), optionally followed by silu; the final state is the last
// W-1 inputs.
//
// The forward pass is a pure stream (2-4 bytes read and 2-4 written per
// element), so the layout is chosen for coalescing: a chunk is 8 consecutive
// steps of one row and consecutive threads own consecutive chunks, so a warp
// reads and writes whole contiguous lines. The W-1 inputs before a chunk come
// from the previous chunk's last bytes (a cache hit: the neighbouring thread
// loads the same line) or from the initial state.
#include "ss_common.cuh"
#include "ss_internal.h"

namespace {

using namespace ssk;

constexpr int kChunk = 8;  // steps per chunk

#ifndef SS_CONV_CPT
#define SS_CONV_CPT 1  // chunks per thread (more measured slower)
#endif

// 8 consecutive inputs at p (16-byte aligned), widened to fp32
__device__ __forceinline__ void load8(const uint16_t *p, float *v) {
    const uint4 t = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) v[2 * k] = bf16lo(w[k]), v[2 * k + 1] = bf16hi(w[k]);
}
__device__ __forceinline__ void load8(const float *p, float *v) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4);
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
}
// the last 4 of the 8 inputs at p (p 16-byte aligned)
__device__ __forceinline__ void load_tail4(const uint16_t *p, float *v) {
    const uint2 t = *reinterpret_cast<const uint2 *>(p + 4);
    v[0] = bf16lo(t.x), v[1] = bf16hi(t.x), v[2] = bf16lo(t.y), v[3] = bf16hi(t.y);
}
__device__ __forceinline__ void load_tail4(const float *p, float *v) {
    const float4 a = *reinterpret_cast<const float4 *>(p + 4);
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w;
}
__device__ __forceinline__ void store8(uint16_t *p, const float *v) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * k]));
        const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * k + 1]));
        w[k] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void store8(float *p, const float *v) {
    *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// Whole chunks: seqlen a multiple of 8. A block owns 256 * CPT consecutive
// chunks (of all rows laid end to end); thread i takes chunks i, i + 256, ...,
// so every load instruction of a warp covers whole contiguous lines, and all
// of a thread's loads are issued before any arithmetic.
// Index arithmetic is 32-bit (the launcher only takes this kernel when the
// chunk count fits), with a shift when the chunks per row are a power of two.
template <typename Tin, typename Tout, int W, int CPT>
__global__ void __launch_bounds__(256) conv1d_chunk_kernel(const ssh::ConvParams p, int cpr_shift) {
    const long long L = p.seqlen;
    const uint32_t cpr = (uint32_t)(L / kChunk);
    const uint32_t total = (uint32_t)p.batch * (uint32_t)p.dim * cpr;
    const uint32_t t0 = blockIdx.x * (256u * CPT) + threadIdx.x;
    auto split = [&](uint32_t t, uint32_t &r, uint32_t &c) {
        if (cpr_shift >= 0) r = t >> cpr_shift, c = t & (cpr - 1);
        else r = t / cpr, c = t - (t / cpr) * cpr;
    };

    float cur[CPT][kChunk], prev[CPT][4];
#pragma unroll
    for (int u = 0; u < CPT; ++u) {
        const uint32_t t = t0 + u * 256;
        if (t >= total) continue;
        uint32_t r, c;
        split(t, r, c);
        const Tin *xr = static_cast<const Tin *>(p.x) + (long long)r * L;
        load8(xr + (long long)c * kChunk, cur[u]);
        if (c > 0) {
            load_tail4(xr + (long long)(c - 1) * kChunk, prev[u]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // prev[j] is the input 4 - j steps before the chunk: state slot (W-1) - (4 - j)
                const int slot = (W - 1) - (4 - j);
                prev[u][j] = (p.init_state && slot >= 0) ? p.init_state[(long long)r * (W - 1) + slot] : 0.f;
            }
        }
    }
#pragma unroll
    for (int u = 0; u < CPT; ++u) {
        const uint32_t t = t0 + u * 256;
        if (t >= total) continue;
        uint32_t r, c;
        split(t, r, c);
        const int d = (int)(r % (uint32_t)p.dim);
        float w[W];
#pragma unroll
        for (int k = 0; k < W; ++k) w[k] = p.w[(long long)d * W + k];
        const float bias = p.bias ? p.bias[d] : 0.f;
        float o[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            float acc = bias;
#pragma unroll
            for (int k = 0; k < W; ++k) {
                const int j = i - (W - 1) + k;  // input index within the chunk
                acc = fmaf(w[k], j >= 0 ? cur[u][j] : prev[u][4 + j], acc);
            }
            o[i] = acc;
        }
        if (p.silu) {
            // bf16 outputs: silu through one tanh.approx (relative error near
            // 2^-11, below the 2^-9 rounding of the bf16 result); fp32
            // outputs: z / (1 + 2^(-z log2 e))
#pragma unroll
            for (int i = 0; i < kChunk; i += 2) {
                const f2 z2 = mk2(o[i], o[i + 1]);
                const f2 s2 = sizeof(Tout) == 2 ? silu2_tanh(z2) : mk2(silu(o[i]), silu(o[i + 1]));
                o[i] = s2.x, o[i + 1] = s2.y;
            }
        }
        store8(static_cast<Tout *>(p.out) + (long long)r * L + (long long)c * kChunk, o);
        if (p.final_state && c == cpr - 1) {
#pragma unroll
            for (int j = 0; j < W - 1; ++j)
                p.final_state[(long long)r * (W - 1) + j] = cur[u][kChunk - (W - 1) + j];
        }
    }
}

// Any seqlen: one thread per output, plain loads; the thread of the last step
// of a row also writes the row's final state.
template <typename Tin, typename Tout, int W>
__global__ void __launch_bounds__(256) conv1d_any_kernel(const ssh::ConvParams p) {
    const long long L = p.seqlen;
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (long long)p.batch * p.dim * L) return;
    const long long r = t / L, l = t % L;
    const int d = (int)(r % p.dim);
    const Tin *xr = static_cast<const Tin *>(p.x) + r * L;
    auto xin = [&](long long j) -> float {
        if (j >= 0) return to_f32(xr[j]);
        return p.init_state ? p.init_state[r * (W - 1) + (W - 1) + j] : 0.f;
    };
    float acc = p.bias ? p.bias[d] : 0.f;
#pragma unroll
    for (int k = 0; k < W; ++k) acc = fmaf(p.w[(long long)d * W + k], xin(l - (W - 1) + k), acc);
    store_out(static_cast<Tout *>(p.out) + r * L + l, p.silu ? silu(acc) : acc);
    if (p.final_state && l == L - 1) {
        float fs[W - 1];
#pragma unroll
        for (int j = 0; j < W - 1; ++j) fs[j] = xin(L - (W - 1) + j);
#pragma unroll
        for (int j = 0; j < W - 1; ++j) p.final_state[r * (W - 1) + j] = fs[j];
    }
}

// Decode: one thread per row.
template <typename Tin, typename Tout, int W>
__global__ void __launch_bounds__(256) conv1d_update_kernel(const ssh::ConvUpdateParams p) {
    // 32-bit indices (the launcher keeps batch * dim below 2^31)
    const uint32_t r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= (uint32_t)p.batch * (uint32_t)p.dim) return;
    const int d = (int)(r % (uint32_t)p.dim);
    float s[W - 1];
#pragma unroll
    for (int k = 0; k < W - 1; ++k) s[k] = p.state[(long long)r * (W - 1) + k];
    const float xv = to_f32(static_cast<const Tin *>(p.x)[r]);
    float acc = p.bias ? p.bias[d] : 0.f;
#pragma unroll
    for (int k = 0; k < W - 1; ++k) acc = fmaf(p.w[(long long)d * W + k], s[k], acc);
    acc = fmaf(p.w[(long long)d * W + W - 1], xv, acc);
    store_out(static_cast<Tout *>(p.out) + r, p.silu ? silu(acc) : acc);
#pragma unroll
    for (int k = 0; k < W - 2; ++k) p.state[(long long)r * (W - 1) + k] = s[k + 1];
    p.state[(long long)r * (W - 1) + W - 2] = xv;
}

template <typename Tin, typename Tout, int W>
int conv_w(const ssh::ConvParams &p, cudaStream_t st) {
    const long long rows = (long long)p.batch * p.dim;
    const bool chunked = p.seqlen % kChunk == 0;
    const long long chunks = chunked ? rows * (p.seqlen / kChunk) : 0;
    if (chunked && chunks < (1LL << 31)) {
        constexpr int CPT = SS_CONV_CPT;
        const long long cpr = p.seqlen / kChunk;
        const int shift = (cpr & (cpr - 1)) == 0 ? __builtin_ctzll((unsigned long long)cpr) : -1;
        const unsigned blocks = (unsigned)((chunks + 256 * CPT - 1) / (256 * CPT));
        conv1d_chunk_kernel<Tin, Tout, W, CPT><<<blocks, 256, 0, st>>>(p, shift);
    } else {
        const long long threads = rows * p.seqlen;
        conv1d_any_kernel<Tin, Tout, W><<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(p);
    }
    return cudaPeekAtLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

template <typename Tin, typename Tout>
int conv_t(const ssh::ConvParams &p, cudaStream_t st) {
    switch (p.width) {
        case 2: return conv_w<Tin, Tout, 2>(p, st);
        case 3: return conv_w<Tin, Tout, 3>(p, st);
        case 4: return conv_w<Tin, Tout, 4>(p, st);
        default: return SS_ERR_UNSUPPORTED;
    }
}

template <typename Tin, typename Tout>
int conv_update_t(const ssh::ConvUpdateParams &p, cudaStream_t st) {
    const long long rows = (long long)p.batch * p.dim;
    if (rows >= (1LL << 31)) return SS_ERR_UNSUPPORTED;
    const unsigned blocks = (unsigned)((rows + 255) / 256);
    switch (p.width) {
        case 2: conv1d_update_kernel<Tin, Tout, 2><<<blocks, 256, 0, st>>>(p); break;
        case 3: conv1d_update_kernel<Tin, Tout, 3><<<blocks, 256, 0, st>>>(p); break;
        case 4: conv1d_update_kernel<Tin, Tout, 4><<<blocks, 256, 0, st>>>(p); break;
        default: return SS_ERR_UNSUPPORTED;
    }
    return cudaPeekAtLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

}  // namespace

int ssh::launch_conv1d(const ssh::ConvParams &p, cudaStream_t st) {
    const bool ib = p.in_dtype == SS_BF16, ob = p.out_dtype == SS_BF16;
    if (ib && ob) return conv_t<uint16_t, uint16_t>(p, st);
    if (ib) return conv_t<uint16_t, float>(p, st);
    if (ob) return conv_t<float, uint16_t>(p, st);
    return conv_t<float, float>(p, st);
}

int ssh::launch_conv1d_update(const ssh::ConvUpdateParams &p, cudaStream_t st) {
    const bool ib = p.in_dtype == SS_BF16, ob = p.out_dtype == SS_BF16;
    if (ib && ob) return conv_update_t<uint16_t, uint16_t>(p, st);
    if (ib) return conv_update_t<uint16_t, float>(p, st);
    if (ob) return conv_update_t<float, uint16_t>(p, st);
    return conv_update_t<float, float>(p, st);
}
