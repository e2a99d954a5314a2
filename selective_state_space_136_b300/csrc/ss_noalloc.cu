// ss_scan_fwd_noalloc: the selective scan for callers that cannot allocate
// device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits, e.g. inside a
// framework's memory-planned or graph-captured region where a stray
// allocation would break the capture or the planner's accounting, in
// real-time paths that may not block on the allocator, or in plugins whose
// host owns every allocation. ss_create allocates (its error word) and the
// chained kernel's context scratch is allocated on first use, so neither can
// be used there.
//
// What it does instead: the chained pair-row kernel's scratch (work counter,
// per-row-block flags, carry buffer, packed fp32 B/C) lives in one
// file-scope __device__ array of kNoAllocScratchBytes (8 MiB). Every GPU that
// loads this library keeps that array until the process exits. The first
// successful call on a device resolves the array's device address
// (cudaGetSymbolAddress, with that device current) and zeroes the flags once
// with a synchronous cudaMemset; make that first call before any stream
// capture. A set-up that fails is retried by the next call. Later calls only
// enqueue kernels.
//
// Every call on a device shares the one array and leaves its contents behind:
// the work counter is reset by the first kernel of each call and the flags are
// tagged with a per-device call number, so stale contents are never read. The
// call number is drawn and the kernels are enqueued under one per-device lock,
// so calls from several host threads on one stream run in call-number order
// (the calls are serialised on the host). A chained wait accepts only its own
// call's flag: a flag left by any other call makes it give up after its
// bounded wait and report SS_ERR_TIMEOUT instead of reading a foreign carry.
// Two calls that overlap on the GPU (different streams, no ordering between
// them) race on the array and give wrong results; order them on one stream.
#include <mutex>

#include "ss_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct DeviceSlot {
    bool ready = false;  // set-up done (only ever set on success)
    unsigned char *base = nullptr;
    unsigned long long calls = 0;
    int sm_count = 0;
    std::mutex mu;  // guards the set-up, `calls` and the enqueue of a call
};
DeviceSlot g_slots[kMaxDevices];

size_t up256(size_t x) { return (x + 255) / 256 * 256; }


// Layout of the array for one call: [counter][flags][carry][packed B/C].
size_t scratch_need(const ssh::ScanParams &p, size_t *flags_b, size_t *carry_b) {
    *flags_b = up256((size_t)ssh::pair_row_blocks(p) * 8);
    *carry_b = up256(ssh::pair_carry_bytes(p));
    return 256 + *flags_b + *carry_b + up256(ssh::pair_bc_bytes(p));
}

// One-time set-up of a device's slot, called with slot.mu held and the device
// current; on failure the slot stays not ready and the next call tries again.
int setup(int dev, DeviceSlot &slot) {
    void *ptr = nullptr;
    int sms = 0;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return SS_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SS_ERR_CUDA;
    // flags must start below every call number; nothing else needs clearing
    if (cudaMemset(ptr, 0, kNoAllocScratchBytes) != cudaSuccess) return SS_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return SS_ERR_CUDA;
    slot.base = static_cast<unsigned char *>(ptr);
    slot.sm_count = sms;
    slot.ready = true;
    return SS_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int ss_scan_fwd_noalloc(const ss_scan_args *a, int *device_error,
                                   ss_stream_t stream) {
    if (!a) return SS_ERR_INVALID_ARG;
    if (a->batch < 1 || a->dim < 1 || a->seqlen < 1) return SS_ERR_INVALID_ARG;
    if ((a->in_dtype != SS_F32 && a->in_dtype != SS_BF16) ||
        (a->out_dtype != SS_F32 && a->out_dtype != SS_BF16))
        return SS_ERR_INVALID_ARG;
    if (!a->u || !a->delta || !a->A || !a->B || !a->C || !a->y) return SS_ERR_INVALID_ARG;
    const void *ptrs[] = {a->u, a->delta, a->z, a->A, a->B, a->C, a->D, a->delta_bias, a->h0,
                          a->y, a->h_last, device_error};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return SS_ERR_INVALID_ARG;
    if ((long long)a->batch * a->dim > (1LL << 40) || a->seqlen >= (1LL << 31))
        return SS_ERR_INVALID_ARG;
    // outputs must not overlap the inputs (same rule as ss_scan_fwd)
    {
        const size_t rows = (size_t)a->batch * a->dim;
        const size_t esz = a->in_dtype == SS_BF16 ? 2 : 4, osz = a->out_dtype == SS_BF16 ? 2 : 4;
        const size_t n_elem = rows * (size_t)a->seqlen;
        const size_t n_bc = (size_t)a->batch * a->dstate * (size_t)a->seqlen;
        auto lo = [](const void *p) { return reinterpret_cast<uintptr_t>(p); };
        auto hit = [&](const void *p, size_t pb, const void *q, size_t qb) {
            return p && q && pb && qb && lo(p) < lo(q) + qb && lo(q) < lo(p) + pb;
        };
        const void *ins[] = {a->u, a->delta, a->z, a->B, a->C};
        const size_t inb[] = {n_elem * esz, n_elem * esz, n_elem * esz, n_bc * esz, n_bc * esz};
        for (int i = 0; i < 5; ++i)
            if (hit(a->y, n_elem * osz, ins[i], inb[i]) ||
                hit(a->h_last, rows * a->dstate * 4, ins[i], inb[i]))
                return SS_ERR_INVALID_ARG;
    }

    ssh::ScanParams p{a->batch, a->dim, a->dstate, a->seqlen, a->in_dtype, a->out_dtype,
                      a->u, a->delta, a->z, a->A, a->B, a->C, a->D, a->delta_bias,
                      a->delta_softplus, a->h0, a->y, a->h_last, device_error,
                      1u << 22, -1, 0};
    // this entry point serves the chained pair-row kernel only
    if (!ssh::pair_supported(p)) return SS_ERR_UNSUPPORTED;
    size_t flags_b = 0, carry_b = 0;
    if (scratch_need(p, &flags_b, &carry_b) > kNoAllocScratchBytes) return SS_ERR_UNSUPPORTED;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SS_ERR_CUDA;
    DeviceSlot &slot = g_slots[dev];
    // the call number and the enqueue happen under one lock, so the kernels of
    // calls made from several threads reach the stream in call-number order
    std::lock_guard<std::mutex> g(slot.mu);
    if (!slot.ready) {
        const int rc = setup(dev, slot);
        if (rc != SS_OK) return rc;
    }
    ssh::PairWork w{};
    w.counter = reinterpret_cast<unsigned long long *>(slot.base);
    w.flags = reinterpret_cast<unsigned long long *>(slot.base + 256);
    w.carry = reinterpret_cast<float *>(slot.base + 256 + flags_b);
    w.bc = reinterpret_cast<float *>(slot.base + 256 + flags_b + carry_b);
    w.epoch = ++slot.calls;
    w.n_seg = 1;
    w.warps_per_sm = 8;
    w.sm_count = slot.sm_count;
    return ssh::launch_pair(p, w, reinterpret_cast<cudaStream_t>(stream));
}
