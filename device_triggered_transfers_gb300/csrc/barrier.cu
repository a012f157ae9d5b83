// The N-rank notify/wait barrier over virtual ranks (PyPTO, "Barrier: Signals Only").
//
// Every virtual rank is one CTA of one cooperative launch, so the ranks that wait on one
// another are guaranteed to be resident together.  Thread 0 of each CTA does the rank's
// notifies (one release fence, then relaxed atomic adds, gpu scope); thread src waits on the
// cell of source src (relaxed loads, counted polls, then an acquire fence); a CTA barrier then
// hands the result to the other threads.
#include <cstdint>
#include <mutex>
#include <new>

#include "internal.h"

namespace dtt {
namespace {

__device__ __forceinline__ int32_t ld_relaxed_s32(const int32_t* p) {
    int32_t v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_relaxed_add_s32(int32_t* p, int32_t v) {
    asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Notify row `me` of every peer's window, then wait for row src >= gen of my window for every
// src != me.  window(q) returns rank q's window.  Called by every thread of the CTA (needs
// blockDim.x >= P); returns 0 or DTT_ETIMEDOUT in every thread.
//  - notify: thread 0 makes one release fence, cumulative over the CTA's earlier stores (the
//    barrier before the call), then relaxed adds that go out together;
//  - wait: thread src polls cell src with relaxed loads (all sources at once, bounded), then an
//    acquire fence; the closing CTA barrier passes the ordering to the other threads.
template <class Window>
__device__ __forceinline__ int notify_wait(Window window, uint32_t me, uint32_t P, int32_t gen,
                                           uint64_t max_polls) {
    __shared__ int s_rc;
    if (threadIdx.x == 0) {
        s_rc = 0;
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        for (uint32_t peer = 0; peer < P; ++peer)
            if (peer != me) red_relaxed_add_s32(window(peer) + me, 1);
    }
    __syncthreads();
    const uint32_t src = threadIdx.x;
    if (src < P && src != me) {
        const int32_t* cell = window(me) + src;
        uint64_t i = 0;
        uint32_t ns = 0;
        bool ok = true;
        while (ld_relaxed_s32(cell) < gen) {
            if (++i >= max_polls) { ok = false; break; }
            __nanosleep(ns);
            ns = ns < 256 ? ns + 32 : 256;
        }
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        if (!ok) s_rc = DTT_ETIMEDOUT;
    }
    __syncthreads();
    return s_rc;
}

struct HandrolledParams {
    int32_t* signal[DTT_MAX_RANKS];
    int32_t* y[DTT_MAX_RANKS];
    int32_t* status;
    uint32_t P;
    int32_t gen;
    uint64_t max_polls;
};

__global__ void handrolled_kernel(const __grid_constant__ HandrolledParams p) {
    const uint32_t me = blockIdx.x;
    auto window = [&](uint32_t q) { return p.signal[q]; };
    const int rc = notify_wait(window, me, p.P, p.gen, p.max_polls);
    if (threadIdx.x == 0) p.status[me] = rc;
    // the observable: this rank's window, read cell by cell after the waits
    for (uint32_t i = threadIdx.x; i < p.P; i += blockDim.x) p.y[me][i] = ld_relaxed_s32(p.signal[me] + i);
}

struct RevealParams {
    const int32_t* x[DTT_MAX_RANKS];
    int32_t* data[DTT_MAX_RANKS];
    int32_t* y[DTT_MAX_RANKS];
    int32_t* counters;     // P x P internal windows, row-major by rank
    int32_t* status;
    uint32_t P;
    uint32_t size;
    int32_t gen;
    uint64_t max_polls;
};

__global__ void reveal_kernel(const __grid_constant__ RevealParams p) {
    const uint32_t me = blockIdx.x;
    for (uint32_t i = threadIdx.x; i < p.size; i += blockDim.x) p.data[me][i] = p.x[me][i];
    __syncthreads();   // the staged slice precedes thread 0's release notifies
    auto window = [&](uint32_t q) { return p.counters + (uint64_t)q * p.P; };
    const int rc = notify_wait(window, me, p.P, p.gen, p.max_polls);
    if (threadIdx.x == 0) p.status[me] = rc;
    const int32_t* peer = p.data[(me + 1) % p.P];
    for (uint32_t i = threadIdx.x; i < p.size; i += blockDim.x) p.y[me][i] = ld_relaxed_s32(peer + i);
}

}  // namespace

cudaError_t preload_barrier_kernels() {
    cudaError_t e = prepare_kernel(handrolled_kernel);
    if (e == cudaSuccess) e = prepare_kernel(reveal_kernel);
    return e;
}

}  // namespace dtt

struct dtt_barrier {
    uint32_t P = 0;
    int32_t* d_counters = nullptr;
    int32_t gen = 0;
};

using namespace dtt;

extern "C" {

int dtt_barrier_handrolled(int32_t* const* signal, int32_t* const* y, uint32_t P, uint32_t gen,
                           uint64_t max_polls, int32_t* status, cudaStream_t stream) {
    if (!signal || !y || !status || P < 1 || P > DTT_MAX_RANKS || gen < 1 || gen > 0x7FFFFFFFu)
        return fail(DTT_EINVAL, "dtt_barrier_handrolled: bad args");
    HandrolledParams hp{};
    for (uint32_t r = 0; r < P; ++r) {
        if (!signal[r] || !y[r]) return fail(DTT_EINVAL, "dtt_barrier_handrolled: NULL window");
        hp.signal[r] = signal[r];
        hp.y[r] = y[r];
    }
    hp.status = status;
    hp.P = P;
    hp.gen = (int32_t)gen;
    hp.max_polls = max_polls;
    void* args[] = {&hp};
    DTT_CUDA_TRY(cudaLaunchCooperativeKernel((const void*)handrolled_kernel, dim3(P), dim3(32), args, 0, stream));
    return DTT_OK;
}

int dtt_barrier_create(uint32_t P, dtt_barrier** out) {
    if (!out || P < 1 || P > DTT_MAX_RANKS) return fail(DTT_EINVAL, "dtt_barrier_create: bad args");
    const int pre = preload_once();
    if (pre != DTT_OK) return pre;
    dtt_barrier* b = new (std::nothrow) dtt_barrier();
    if (!b) return fail(DTT_ENOMEM, "dtt_barrier_create: out of memory");
    b->P = P;
    cudaError_t e = cudaMalloc(&b->d_counters, (size_t)P * P * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMemset(b->d_counters, 0, (size_t)P * P * sizeof(int32_t));
    if (e != cudaSuccess) {
        cudaFree(b->d_counters);
        delete b;
        return fail(DTT_ECUDA, "dtt_barrier_create: %s", cudaGetErrorString(e));
    }
    *out = b;
    return DTT_OK;
}

void dtt_barrier_destroy(dtt_barrier* b) {
    if (!b) return;
    cudaFree(b->d_counters);
    delete b;
}

int dtt_barrier_reveal(dtt_barrier* b, const int32_t* const* x, int32_t* const* data,
                       int32_t* const* y, uint32_t size, uint64_t max_polls, int32_t* status,
                       cudaStream_t stream) {
    if (!b || !x || !data || !y || !status) return fail(DTT_EINVAL, "dtt_barrier_reveal: bad args");
    if (b->gen == 0x7FFFFFFF) return fail(DTT_EROUNDLIMIT, "dtt_barrier_reveal: generation limit reached");
    RevealParams rp{};
    for (uint32_t r = 0; r < b->P; ++r) {
        if (!x[r] || !data[r] || !y[r]) return fail(DTT_EINVAL, "dtt_barrier_reveal: NULL slice");
        rp.x[r] = x[r];
        rp.data[r] = data[r];
        rp.y[r] = y[r];
    }
    rp.counters = b->d_counters;
    rp.status = status;
    rp.P = b->P;
    rp.size = size;
    rp.gen = b->gen + 1;
    rp.max_polls = max_polls;
    void* args[] = {&rp};
    DTT_CUDA_TRY(cudaLaunchCooperativeKernel((const void*)reveal_kernel, dim3(b->P), dim3(256), args, 0, stream));
    b->gen += 1;
    return DTT_OK;
}

}  // extern "C"

// ---- the reveal without any allocation ------------------------------------------------------
// The builtin barrier's internal counters for dtt_barrier_reveal_noalloc live in this fixed
// array (DTT_NOALLOC_MAX_RANKS^2 int32 = 1 KiB), part of the library's device image: every GPU
// that loads the library holds it until the process exits.  Every call uses the same array.
static __device__ __align__(256) int32_t g_reveal_counters[DTT_NOALLOC_MAX_RANKS * DTT_NOALLOC_MAX_RANKS];

namespace {

std::mutex g_noalloc_mu;
int32_t* g_noalloc_counters[64] = {};   // device address of the array, per device id

// Set-up, once per device with that device current.  In host code the array's name is only a
// host-side stand-in, so its device address must come from cudaGetSymbolAddress.
int noalloc_counters(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(DTT_ECUDA, "dtt_barrier_reveal_noalloc: no CUDA device");
    if (dev < 0 || dev >= 64) return fail(DTT_EINVAL, "dtt_barrier_reveal_noalloc: device id %d not supported", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_counters[dev]) {
        const int pre = preload_once();
        if (pre != DTT_OK) return pre;
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_reveal_counters);
        if (e != cudaSuccess || !p)
            return fail(DTT_ECUDA, "dtt_barrier_reveal_noalloc: cudaGetSymbolAddress failed: %s",
                        cudaGetErrorString(e));
        g_noalloc_counters[dev] = static_cast<int32_t*>(p);
    }
    *out = g_noalloc_counters[dev];
    return DTT_OK;
}

}  // namespace

extern "C" int dtt_barrier_reveal_noalloc(const int32_t* const* x, int32_t* const* data,
                                          int32_t* const* y, uint32_t P, uint32_t size,
                                          uint64_t max_polls, int32_t* status, cudaStream_t stream) {
    if (!x || !data || !y || !status) return fail(DTT_EINVAL, "dtt_barrier_reveal_noalloc: bad args");
    if (P < 1 || P > DTT_NOALLOC_MAX_RANKS)
        return fail(DTT_EINVAL, "dtt_barrier_reveal_noalloc: P = %u is outside 1..%d, the ranks its static counter array holds",
                    P, DTT_NOALLOC_MAX_RANKS);
    RevealParams rp{};
    for (uint32_t r = 0; r < P; ++r) {
        if (!x[r] || !data[r] || !y[r]) return fail(DTT_EINVAL, "dtt_barrier_reveal_noalloc: NULL slice");
        rp.x[r] = x[r];
        rp.data[r] = data[r];
        rp.y[r] = y[r];
    }
    int32_t* counters = nullptr;
    const int rc = noalloc_counters(&counters);
    if (rc != DTT_OK) return rc;
    // the array keeps the previous call's counts: clear the P x P cells this call uses, in
    // stream order, so that this call's barrier is generation 1
    DTT_CUDA_TRY(cudaMemsetAsync(counters, 0, (size_t)P * P * sizeof(int32_t), stream));
    rp.counters = counters;
    rp.status = status;
    rp.P = P;
    rp.size = size;
    rp.gen = 1;
    rp.max_polls = max_polls;
    void* args[] = {&rp};
    DTT_CUDA_TRY(cudaLaunchCooperativeKernel((const void*)reveal_kernel, dim3(P), dim3(256), args, 0, stream));
    return DTT_OK;
}
