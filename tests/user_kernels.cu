// A user's own producer and consumer kernels driving a triggered plan through the public
// device header alone (the peer-kernel side of "Triggered Plans", Model; the kernel author's
// contract).  Built by tests/test_gpu_user_kernels.py into a temporary shared object.
//
// producer: CTA c writes chunk c of the rank's slice (one writer per chunk), then marks it.
// consumer: CTA c waits for chunk c at rank q, then copies it to dst; status[c] = 0 or timeout.
// paced producer: CTA c first waits until chunk c - 1 of its rank is reusable (delivered to
// every peer), the source side of "Triggered SDMA Plans" (API: reusable).
// probe: CTA i records dtt_reusable of chunk first + i.
#include <cstdint>

#include <cuda_runtime.h>

#include "dtt_device.cuh"

namespace {

// The byte a producer stores at slice offset i of `rank` in `round`: any pattern that changes
// with the round, so that a stale copy is caught.
__device__ __forceinline__ uint8_t value_at(uint32_t rank, uint32_t round, uint64_t i) {
    uint32_t x = (uint32_t)i * 2654435761u ^ (rank * 0x9E3779B9u) ^ (round * 0x85EBCA6Bu);
    x ^= x >> 15;
    return (uint8_t)x;
}

__global__ void user_producer(dtt_handle h, uint8_t* slice, uint64_t chunk_bytes) {
    const uint32_t c = blockIdx.x;
    const uint64_t base = (uint64_t)c * chunk_bytes;
    for (uint64_t i = threadIdx.x; i < chunk_bytes; i += blockDim.x)
        slice[base + i] = value_at(h.rank, h.round, base + i);
    dtt_mark_ready(h, h.first_chunk + c);      // the whole CTA, after its stores
}

__global__ void user_consumer(dtt_handle h, const uint8_t* buf, uint8_t* dst, uint64_t chunk_bytes,
                              uint64_t max_polls, int32_t* status) {
    const uint32_t c = blockIdx.x;              // global chunk id; chunk c covers bytes c * chunk_bytes
    const int r = dtt_wait(h, c, max_polls);
    if (threadIdx.x == 0) status[c] = r;
    if (r != 0) return;
    const uint64_t base = (uint64_t)c * chunk_bytes;
    for (uint64_t i = threadIdx.x; i < chunk_bytes; i += blockDim.x) dst[base + i] = buf[base + i];
}

// A producer that waits, before CTA c writes chunk c, until chunk c - 1 of its rank has been
// delivered everywhere (dtt_wait_reusable), and records the wait's result and when it ended.
__global__ void user_producer_paced(dtt_handle h, uint8_t* slice, uint64_t chunk_bytes, uint64_t max_polls,
                                    int32_t* wait_status, uint64_t* wait_end) {
    const uint32_t c = blockIdx.x;
    if (c > 0) {
        const int r = dtt_wait_reusable(h, h.first_chunk + c - 1, max_polls);
        if (threadIdx.x == 0) {
            wait_status[c] = r;
            uint64_t t;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
            wait_end[c] = t;
        }
    }
    const uint64_t base = (uint64_t)c * chunk_bytes;
    for (uint64_t i = threadIdx.x; i < chunk_bytes; i += blockDim.x)
        slice[base + i] = value_at(h.rank, h.round, base + i);
    dtt_mark_ready(h, h.first_chunk + c);
}

// Out-of-order completion ("Triggered Plans", The kernel author's contract, item 1): one CTA
// writes the rank's chunks last to first, marking each after its stores, so chunk 0 -- the
// head of every copier queue of this rank -- opens last.  `spin_ns` of busy time after each mark
// leaves the later chunks open for a while before the head opens.
__global__ void user_producer_reverse(dtt_handle h, uint8_t* slice, uint64_t chunk_bytes, uint64_t spin_ns) {
    for (uint32_t k = h.n_chunks; k-- > 0;) {
        const uint64_t base = (uint64_t)k * chunk_bytes;
        for (uint64_t i = threadIdx.x; i < chunk_bytes; i += blockDim.x)
            slice[base + i] = value_at(h.rank, h.round, base + i);
        dtt_mark_ready(h, h.first_chunk + k);
        if (threadIdx.x == 0 && spin_ns) {
            uint64_t t0, t;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
            do { asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)); } while (t - t0 < spin_ns);
        }
        __syncthreads();
    }
}

// Group consumer ("Triggered Plans", Not supported yet, "Waiting on a group"): CTA g waits ONCE
// on group g (members gids[goff[g] .. goff[g + 1]), global chunk c covering bytes
// [c * chunk_bytes, (c + 1) * chunk_bytes) of every buffer), then copies every member to dst.
__global__ void user_group_consumer(dtt_handle h, const uint8_t* buf, uint8_t* dst, uint64_t chunk_bytes,
                                    const uint32_t* goff, const uint32_t* gids, uint64_t max_polls,
                                    int32_t* status) {
    const uint32_t g = blockIdx.x;
    const int r = dtt_wait_group(h, g, max_polls);
    if (threadIdx.x == 0) status[g] = r;
    if (r != 0) return;
    for (uint32_t i = goff[g]; i < goff[g + 1]; ++i) {
        const uint64_t base = (uint64_t)gids[i] * chunk_bytes;
        for (uint64_t x = threadIdx.x; x < chunk_bytes; x += blockDim.x) dst[base + x] = buf[base + x];
    }
}

// CTA i records dtt_group_arrived of group first + i.
__global__ void user_group_probe(dtt_handle h, uint32_t first, int32_t* out) {
    const bool a = dtt_group_arrived(h, first + blockIdx.x);
    if (threadIdx.x == 0) out[blockIdx.x] = a ? 1 : 0;
}

// CTA i asks dtt_reusable of global chunk first + i.
__global__ void user_probe_reusable(dtt_handle h, uint32_t first, int32_t* out) {
    const bool r = dtt_reusable(h, first + blockIdx.x);
    if (threadIdx.x == 0) out[blockIdx.x] = r ? 1 : 0;
}

// Overlapping rounds: CTA i records dtt_writable of global chunk first + i, then waits for it
// (dtt_wait_writable, at most max_polls polls) and records the wait's result.
__global__ void user_probe_writable(dtt_handle h, uint32_t first, uint64_t max_polls, int32_t* now,
                                    int32_t* waited) {
    const bool w = dtt_writable(h, first + blockIdx.x);
    const int r = dtt_wait_writable(h, first + blockIdx.x, max_polls);
    if (threadIdx.x == 0) {
        now[blockIdx.x] = w ? 1 : 0;
        waited[blockIdx.x] = r;
    }
}

}  // namespace

// What the documented contract asks of a user's kernels before the first round: loaded now,
// and the library's shared-memory carveout.
extern "C" int user_kernels_prepare(void) {
    cudaFuncAttributes a{};
    if (cudaFuncGetAttributes(&a, user_producer) != cudaSuccess) return 1;
    if (cudaFuncGetAttributes(&a, user_consumer) != cudaSuccess) return 1;
    if (cudaFuncSetAttribute(user_producer, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return 1;
    if (cudaFuncSetAttribute(user_consumer, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return 1;
    if (cudaFuncGetAttributes(&a, user_producer_reverse) != cudaSuccess) return 1;
    if (cudaFuncSetAttribute(user_producer_reverse, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return 1;
    if (cudaFuncGetAttributes(&a, user_group_consumer) != cudaSuccess) return 1;
    if (cudaFuncSetAttribute(user_group_consumer, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return 1;
    if (cudaFuncGetAttributes(&a, user_group_probe) != cudaSuccess) return 1;
    if (cudaFuncGetAttributes(&a, user_producer_paced) != cudaSuccess) return 1;
    if (cudaFuncGetAttributes(&a, user_probe_reusable) != cudaSuccess) return 1;
    if (cudaFuncGetAttributes(&a, user_probe_writable) != cudaSuccess) return 1;
    if (cudaFuncSetAttribute(user_producer_paced, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return 1;
    return 0;
}

extern "C" int user_produce(const dtt_handle* h, void* slice, uint64_t chunk_bytes, cudaStream_t s) {
    if (h->n_chunks == 0) return 0;
    user_producer<<<h->n_chunks, 256, 0, s>>>(*h, static_cast<uint8_t*>(slice), chunk_bytes);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

extern "C" int user_consume(const dtt_handle* h, const void* buf, void* dst, uint64_t chunk_bytes,
                            uint64_t max_polls, int32_t* status, cudaStream_t s) {
    user_consumer<<<h->n_global, 256, 0, s>>>(*h, static_cast<const uint8_t*>(buf), static_cast<uint8_t*>(dst),
                                              chunk_bytes, max_polls, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

extern "C" int user_produce_paced(const dtt_handle* h, void* slice, uint64_t chunk_bytes, uint64_t max_polls,
                                  int32_t* wait_status, uint64_t* wait_end, cudaStream_t s) {
    if (h->n_chunks == 0) return 0;
    user_producer_paced<<<h->n_chunks, 256, 0, s>>>(*h, static_cast<uint8_t*>(slice), chunk_bytes, max_polls,
                                                    wait_status, wait_end);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

extern "C" int user_probe(const dtt_handle* h, uint32_t first, uint32_t n, int32_t* out, cudaStream_t s) {
    if (n == 0) return 0;
    user_probe_reusable<<<n, 64, 0, s>>>(*h, first, out);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

extern "C" int user_produce_reverse(const dtt_handle* h, void* slice, uint64_t chunk_bytes, uint64_t spin_ns,
                                    cudaStream_t s) {
    if (h->n_chunks == 0) return 0;
    user_producer_reverse<<<1, 256, 0, s>>>(*h, static_cast<uint8_t*>(slice), chunk_bytes, spin_ns);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

extern "C" int user_group_consume(const dtt_handle* h, uint32_t n_groups, const void* buf, void* dst,
                                  uint64_t chunk_bytes, const uint32_t* goff, const uint32_t* gids,
                                  uint64_t max_polls, int32_t* status, cudaStream_t s) {
    user_group_consumer<<<n_groups, 256, 0, s>>>(*h, static_cast<const uint8_t*>(buf), static_cast<uint8_t*>(dst),
                                                 chunk_bytes, goff, gids, max_polls, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

extern "C" int user_group_probe_launch(const dtt_handle* h, uint32_t first, uint32_t n, int32_t* out,
                                       cudaStream_t s) {
    if (n == 0) return 0;
    user_group_probe<<<n, 64, 0, s>>>(*h, first, out);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

extern "C" int user_probe_writable_launch(const dtt_handle* h, uint32_t first, uint32_t n, uint64_t max_polls,
                                          int32_t* now, int32_t* waited, cudaStream_t s) {
    if (n == 0) return 0;
    user_probe_writable<<<n, 64, 0, s>>>(*h, first, max_polls, now, waited);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}
