/*
 * dtt_device.cuh -- device side of a triggered plan: mark_ready, arrived, wait, reusable,
 * writable and the group waits.
 *
 * Include from producer and consumer kernels; the kernel receives a dtt_handle (include/dtt.h)
 * by value.  Every function here is called by ALL threads of a CTA (dtt_mark_ready_cluster:
 * of a cluster), outside divergent code, the same number of times in every thread ("Triggered
 * Plans", The kernel author's contract, items 2 and 5).  They use __syncthreads internally.
 *
 * Memory ordering ("Triggered Plans", section Memory ordering), restated for one GPU:
 *  - mark_ready: a CTA barrier orders every thread's earlier stores before thread 0, whose
 *    acq_rel atomic add on the chunk's writer counter (gpu scope) is cumulative over them.
 *    The writer whose add completes the round's count then stores ready = round with release
 *    semantics: the copier acquires `ready`, not the counter, and the release keeps every
 *    writer's stores (acquired through the counter's read-modify-write chain) ahead of it.
 *    The pages' copy engine reads behind L2 and needs system scope; every reader here is an SM
 *    of the same GPU, so gpu scope suffices.
 *  - arrived / wait: thread 0 reads the gate with an acquire load (gpu scope); a CTA barrier
 *    passes the result to the other threads, and data they load afterwards is this round's.
 *    Polls are counted, never clock-bounded.
 *  - reusable / writable: thread 0 acquires the chunk's completion word, which the copier bumps
 *    after a release fence once every copy of the chunk has landed (and so after its reads of
 *    it); writable asks for the previous round's count (overlapping rounds).
 *  - groups: the mark that opens a gate, and the copier's arrival signal at a peer, add one to
 *    that rank's counters of the chunk's groups after a release fence; dtt_wait_group acquires
 *    the counter, so data of every member read after it is this round's.
 *  - A producer that writes through the async proxy (TMA stores) must complete those writes
 *    (cp.async.bulk.wait_group 0) and issue fence.proxy.async before calling mark_ready; a
 *    consumer that reads landed bytes through the async proxy (TMA loads) issues
 *    fence.proxy.async.global after its wait, as the library's consumer GEMM does.
 */
#ifndef DTT_DEVICE_CUH
#define DTT_DEVICE_CUH

#include <stdint.h>
#include "dtt.h"

namespace dtt_dev {

__device__ __forceinline__ uint64_t ld_acquire(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t ld_relaxed(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(uint64_t* p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t atom_add_acq_rel(uint64_t* p, uint64_t v) {
    uint64_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;"
                 : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}

__device__ __forceinline__ void red_release_add(uint64_t* p, uint64_t v) {
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void red_relaxed_add(uint64_t* p, uint64_t v) {
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void red_relaxed_max(uint64_t* p, uint64_t v) {
    asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool first_thread() {
    return threadIdx.x == 0 && threadIdx.y == 0 && threadIdx.z == 0;
}

__device__ __forceinline__ uint64_t* gate_row(const dtt_handle& h, uint32_t table, uint32_t chunk) {
    return h.gates + ((uint64_t)table * h.n_global + chunk) * DTT_GATE_WORDS;
}

/* One writer's mark, issued by one thread after the caller's barrier. */
__device__ __forceinline__ void mark_one(const dtt_handle& h, uint32_t chunk) {
    if (chunk < h.first_chunk || chunk >= h.first_chunk + h.n_chunks) {
        atomicOr(h.status, DTT_DEV_EBADCHUNK);
        return;
    }
    uint64_t* row = gate_row(h, h.rank, chunk);
    const uint64_t target = (uint64_t)h.round * h.writers[chunk];
    const uint64_t now = atom_add_acq_rel(row + DTT_GATE_COUNTER, 1) + 1;
    if (now == target) {
        if (h.flags & DTT_HANDLE_TIMESTAMPS) st_relaxed(row + DTT_GATE_T_OPEN, globaltimer());
        if (h.groups.counters) {
            // the chunk is readable at its own rank from now on: it counts in the rank's counter
            // of each of its groups.  The chunk's group ids are read first, then one release
            // fence covers the gate and every counter (each relaxed write after the fence is a
            // release pattern)
            const uint32_t a = h.groups.chunk_off[chunk], b = h.groups.chunk_off[chunk + 1];
            uint64_t* grow = h.groups.counters + (uint64_t)h.rank * h.groups.n_groups;
            fence_acq_rel();
            st_relaxed(row + DTT_GATE_READY, h.round);
            for (uint32_t i = a; i < b; ++i) red_relaxed_add(grow + h.groups.chunk_ids[i], 1);
        } else {
            st_release(row + DTT_GATE_READY, h.round);
        }
        if (h.host_ready) {
            // a copy-engine plan: the host proxy issues the copies once it reads this word, so
            // the chunk's data is made visible at system scope first
            asm volatile("fence.acq_rel.sys;\n\t"
                         "st.relaxed.sys.global.u32 [%0], %1;" ::"l"(h.host_ready + chunk), "r"(h.round) : "memory");
        }
    } else if (now > target) {
        red_relaxed_max(row + DTT_GATE_ERROR, h.round);
    }
}

/* The counter a rank polls for group g and the count that completes this round; null when the
 * plan has no group g (a misuse bit is set). */
__device__ __forceinline__ const uint64_t* group_word(const dtt_handle& h, uint32_t g, uint64_t* target) {
    if (!h.groups.counters || g >= h.groups.n_groups) {
        atomicOr(h.status, DTT_DEV_EBADGROUP);
        return nullptr;
    }
    const uint64_t at = (uint64_t)h.rank * h.groups.n_groups + g;
    *target = (uint64_t)h.round * h.groups.size[at];
    return h.groups.counters + at;
}

/* Ranks a chunk of this rank is copied to: every other rank, or those of its peer mask. */
__device__ __forceinline__ uint32_t receivers(const dtt_handle& h, uint32_t chunk) {
    if (!h.peer_masks) return h.P - 1;
    return (uint32_t)__popc(h.peer_masks[chunk] & ~(1u << h.rank));
}

/* The word a rank polls for `chunk`: its own chunks are local once ready; other ranks' chunks
 * are here once they arrived. */
__device__ __forceinline__ const uint64_t* wait_word(const dtt_handle& h, uint32_t chunk) {
    const uint64_t* row = gate_row(h, h.rank, chunk);
    const bool own = chunk >= h.first_chunk && chunk < h.first_chunk + h.n_chunks;
    return row + (own ? DTT_GATE_READY : DTT_GATE_ARRIVAL);
}

}  // namespace dtt_dev

/* Mark `chunk` (global id, one of this rank's) ready: one of its `writers` marks this round.
 * Call after this CTA's writes to the chunk. */
__device__ __forceinline__ void dtt_mark_ready(const dtt_handle& h, uint32_t chunk) {
    __syncthreads();
    if (dtt_dev::first_thread()) dtt_dev::mark_one(h, chunk);
    __syncthreads();
}

/* Cluster form: every CTA of a thread-block cluster calls it after its writes; a cluster
 * barrier (release / acquire, cluster scope) orders all of them before CTA 0's thread 0,
 * which issues ONE mark.  The cluster counts as one writer. */
__device__ __forceinline__ void dtt_mark_ready_cluster(const dtt_handle& h, uint32_t chunk) {
    __syncthreads();
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
    uint32_t crank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
    if (crank == 0 && dtt_dev::first_thread()) dtt_dev::mark_one(h, chunk);
    __syncthreads();
}

/* One poll: has `chunk` arrived here this round (own chunk: is it ready)? */
__device__ __forceinline__ bool dtt_arrived(const dtt_handle& h, uint32_t chunk) {
    __shared__ int dtt_arrived_flag;
    __syncthreads();
    if (dtt_dev::first_thread())
        dtt_arrived_flag = (uint32_t)dtt_dev::ld_acquire(dtt_dev::wait_word(h, chunk)) >= h.round;
    __syncthreads();
    return dtt_arrived_flag != 0;
}

/* Wait until `chunk` has arrived here this round (own chunk: until it is ready), polling at
 * most max_polls times.  Returns 0, or DTT_ETIMEDOUT if the polls ran out. */
__device__ __forceinline__ int dtt_wait(const dtt_handle& h, uint32_t chunk, uint64_t max_polls) {
    __shared__ int dtt_wait_result;
    __syncthreads();
    if (dtt_dev::first_thread()) {
        const uint64_t* w = dtt_dev::wait_word(h, chunk);
        int r = DTT_ETIMEDOUT;
        uint32_t ns = 0;
        for (uint64_t i = 0; i < max_polls; ++i) {
            if ((uint32_t)dtt_dev::ld_acquire(w) >= h.round) { r = 0; break; }
            __nanosleep(ns);
            ns = ns < 256 ? ns + 32 : 256;
        }
        dtt_wait_result = r;
    }
    __syncthreads();
    return dtt_wait_result;
}

/* One poll of group g ("Triggered Plans", Not supported yet: "Waiting on a group"): has every
 * chunk of the group become readable here this round (other ranks' chunks arrived, this rank's
 * own chunks ready)?  A group the plan does not have sets DTT_DEV_EBADGROUP and reads false. */
__device__ __forceinline__ bool dtt_group_arrived(const dtt_handle& h, uint32_t g) {
    __shared__ int dtt_group_arrived_flag;
    __syncthreads();
    if (dtt_dev::first_thread()) {
        uint64_t target = 0;
        const uint64_t* w = dtt_dev::group_word(h, g, &target);
        dtt_group_arrived_flag = w && dtt_dev::ld_acquire(w) >= target;
    }
    __syncthreads();
    return dtt_group_arrived_flag != 0;
}

/* Wait until dtt_group_arrived(h, g), polling one counter at most max_polls times: one wait
 * covers every chunk of the group, of any source rank.  Returns 0, or DTT_ETIMEDOUT if the polls
 * ran out (or the plan has no group g).  Data read after it is this round's. */
__device__ __forceinline__ int dtt_wait_group(const dtt_handle& h, uint32_t g, uint64_t max_polls) {
    __shared__ int dtt_wait_group_result;
    __syncthreads();
    if (dtt_dev::first_thread()) {
        uint64_t target = 0;
        const uint64_t* w = dtt_dev::group_word(h, g, &target);
        int r = DTT_ETIMEDOUT;
        uint32_t ns = 0;
        for (uint64_t i = 0; w && i < max_polls; ++i) {
            if (dtt_dev::ld_acquire(w) >= target) { r = 0; break; }
            __nanosleep(ns);
            ns = ns < 256 ? ns + 32 : 256;
        }
        dtt_wait_group_result = r;
    }
    __syncthreads();
    return dtt_wait_group_result;
}

/* Source side ("Triggered SDMA Plans", API: the device view's `reusable`; Design notes: the
 * completion word of the gate row): has every copy of this rank's own `chunk` landed at every
 * peer this round, so that the chunk's bytes may be written again?  True when the chunk's
 * completion word has reached round * (its receivers: P - 1 unless it goes to only some peers),
 * the copier's deliveries of it over all rounds.
 * The acquire orders the copier's reads of the chunk before the caller's later writes.  A
 * chunk of another rank sets DTT_DEV_EBADCHUNK in the plan's status word and returns false. */
__device__ __forceinline__ bool dtt_reusable(const dtt_handle& h, uint32_t chunk) {
    __shared__ int dtt_reusable_flag;
    __syncthreads();
    if (dtt_dev::first_thread()) {
        int f = 0;
        if (chunk < h.first_chunk || chunk >= h.first_chunk + h.n_chunks) {
            atomicOr(h.status, DTT_DEV_EBADCHUNK);
        } else {
            const uint64_t* w = dtt_dev::gate_row(h, h.rank, chunk) + DTT_GATE_COMPLETION;
            f = dtt_dev::ld_acquire(w) >= (uint64_t)h.round * dtt_dev::receivers(h, chunk);
        }
        dtt_reusable_flag = f;
    }
    __syncthreads();
    return dtt_reusable_flag != 0;
}

/* Wait until dtt_reusable(h, chunk), polling at most max_polls times.  Returns 0, or
 * DTT_ETIMEDOUT if the polls ran out (or the chunk is not this rank's). */
__device__ __forceinline__ int dtt_wait_reusable(const dtt_handle& h, uint32_t chunk, uint64_t max_polls) {
    __shared__ int dtt_wait_reusable_result;
    __syncthreads();
    if (dtt_dev::first_thread()) {
        int r = DTT_ETIMEDOUT;
        if (chunk < h.first_chunk || chunk >= h.first_chunk + h.n_chunks) {
            atomicOr(h.status, DTT_DEV_EBADCHUNK);
        } else {
            const uint64_t* w = dtt_dev::gate_row(h, h.rank, chunk) + DTT_GATE_COMPLETION;
            const uint64_t target = (uint64_t)h.round * dtt_dev::receivers(h, chunk);
            uint32_t ns = 0;
            for (uint64_t i = 0; i < max_polls; ++i) {
                if (dtt_dev::ld_acquire(w) >= target) { r = 0; break; }
                __nanosleep(ns);
                ns = ns < 256 ? ns + 32 : 256;
            }
        }
        dtt_wait_reusable_result = r;
    }
    __syncthreads();
    return dtt_wait_reusable_result;
}

namespace dtt_dev {

/* The completion count at which rank h.rank's own `chunk` may be written in round h.round:
 * every copy of it made in round h.round - 1 has landed, (round - 1) * receivers deliveries. */
__device__ __forceinline__ const uint64_t* writable_word(const dtt_handle& h, uint32_t chunk, uint64_t* target) {
    if (chunk < h.first_chunk || chunk >= h.first_chunk + h.n_chunks) {
        atomicOr(h.status, DTT_DEV_EBADCHUNK);
        return nullptr;
    }
    *target = (uint64_t)(h.round - 1) * receivers(h, chunk);
    return gate_row(h, h.rank, chunk) + DTT_GATE_COMPLETION;
}

/* One thread: bounded wait until writable (true), or false when the polls ran out. */
__device__ __forceinline__ bool wait_writable_one(const dtt_handle& h, uint32_t chunk, uint64_t max_polls) {
    uint64_t target = 0;
    const uint64_t* w = writable_word(h, chunk, &target);
    if (!w) return false;
    uint32_t ns = 0;
    for (uint64_t i = 0; i < max_polls; ++i) {
        if (ld_acquire(w) >= target) return true;
        __nanosleep(ns);
        ns = ns < 256 ? ns + 32 : 256;
    }
    return false;
}

}  // namespace dtt_dev

/* Overlapping rounds ("Triggered Plans", Not supported yet: "Overlapping rounds"; plans made with
 * opts.overlap): may this rank write its own `chunk` in round h.round -- has every copy of it
 * made in the previous round landed, so that no copier still reads the previous round's bytes?
 * That is the chunk's completion word at (round - 1) * receivers.  Always true when rounds do
 * not overlap (the previous round was checked before this one started).  The acquire orders the
 * copier's reads before the caller's later writes.  A chunk of another rank sets
 * DTT_DEV_EBADCHUNK and reads false. */
__device__ __forceinline__ bool dtt_writable(const dtt_handle& h, uint32_t chunk) {
    __shared__ int dtt_writable_flag;
    __syncthreads();
    if (dtt_dev::first_thread()) {
        uint64_t target = 0;
        const uint64_t* w = dtt_dev::writable_word(h, chunk, &target);
        dtt_writable_flag = w && dtt_dev::ld_acquire(w) >= target;
    }
    __syncthreads();
    return dtt_writable_flag != 0;
}

/* Wait until dtt_writable(h, chunk), polling at most max_polls times; call it before the first
 * write of a chunk in a round.  Returns 0, or DTT_ETIMEDOUT if the polls ran out (or the chunk is
 * not this rank's): the chunk must then be left unwritten. */
__device__ __forceinline__ int dtt_wait_writable(const dtt_handle& h, uint32_t chunk, uint64_t max_polls) {
    __shared__ int dtt_wait_writable_result;
    __syncthreads();
    if (dtt_dev::first_thread())
        dtt_wait_writable_result = dtt_dev::wait_writable_one(h, chunk, max_polls) ? 0 : DTT_ETIMEDOUT;
    __syncthreads();
    return dtt_wait_writable_result;
}

#endif /* DTT_DEVICE_CUH */
