// The persistent copier and the plan's small kernels (completion check, force-open, publish,
// consumer).
//
// The copier stands where the pages' copy engine runs its pre-armed packet chain: wait until a
// chunk's gate is open (ready >= round), copy each region to the same offset in every peer's
// buffer, then add one to the peer's arrival word ("Triggered Plans", introduction and section
// Model; "Triggered SDMA Plans", Design notes).  One launch serves one round.  Its CTAs are
// split among the sending ranks in proportion to their bytes; the CTAs of source s walk s's
// chunks in schedule order, every CTA waiting on every gate in turn, so a chunk completed early
// waits for the chunks before it, as on one copy-engine queue ("Triggered Plans", The kernel
// author's contract, item 1).  A chunk's pieces are dealt round-robin over the source's CTAs,
// continuing from where the previous chunk's pieces stopped; each piece is read ONCE and
// written to all P-1 peers.  The CTA that finishes a chunk's last piece (found with an acq_rel
// counter in the owner's gate row) signals the arrival at every peer with a release add.
#include <cstdint>

#include "dtt_device.cuh"
#include "internal.h"

namespace dtt {
namespace {

constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 ld_cg16(const void* p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_cs16(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                 ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ uint8_t ld_cg8(const uint8_t* p) {
    uint16_t v;
    asm volatile("ld.global.cg.u8 %0, [%1];" : "=h"(v) : "l"(p));
    return (uint8_t)v;
}

// Copy one piece from buffer s to every other buffer: 16-byte vectors, kUnroll loads in
// flight per thread, each value stored to all peers.
__device__ __forceinline__ void copy_piece_vec(const CopierParams& p, uint32_t s,
                                               const PieceDesc& pc) {
    const uint32_t rv = pc.row_bytes >> 4;
    const uint32_t total = rv * pc.rows;
    const char* src = p.bufs[s] + pc.off;
    const uint32_t stride = blockDim.x * kUnroll;
    for (uint32_t v0 = threadIdx.x; v0 < total; v0 += stride) {
        uint4 val[kUnroll];
        uint64_t off[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint32_t v = v0 + u * blockDim.x;
            if (v < total) {
                uint32_t row = 0, col = v;
                if (pc.rows > 1) {
                    row = v / rv;
                    col = v - row * rv;
                }
                off[u] = (uint64_t)row * pc.pitch + ((uint64_t)col << 4);
                val[u] = ld_cg16(src + off[u]);
            }
        }
#pragma unroll 1
        for (uint32_t q = 0; q < p.P; ++q) {
            if (q == s) continue;
            char* dst = p.bufs[q] + pc.off;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const uint32_t v = v0 + u * blockDim.x;
                if (v < total) st_cs16(dst + off[u], val[u]);
            }
        }
    }
}

// Byte-wise copy for pieces that are not 16-byte aligned.
__device__ __forceinline__ void copy_piece_bytes(const CopierParams& p, uint32_t s,
                                                 const PieceDesc& pc) {
    const uint64_t total = (uint64_t)pc.row_bytes * pc.rows;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(p.bufs[s]) + pc.off;
    for (uint64_t b = threadIdx.x; b < total; b += blockDim.x) {
        const uint64_t row = b / pc.row_bytes, col = b - row * pc.row_bytes;
        const uint64_t o = row * pc.pitch + col;
        const uint8_t v = ld_cg8(src + o);
        for (uint32_t q = 0; q < p.P; ++q)
            if (q != s) reinterpret_cast<uint8_t*>(p.bufs[q])[pc.off + o] = v;
    }
}

// Thread 0: poll the gate until its low 32 bits reach `round`; counted polls with a short
// sleep between them.  Returns false when the polls run out.
__device__ __forceinline__ bool poll_gate(const uint64_t* ready, uint32_t round,
                                          uint64_t max_polls) {
    uint32_t ns = 0;
    for (uint64_t i = 0;; ++i) {
        if ((uint32_t)dtt_dev::ld_acquire(ready) >= round) return true;
        if (i >= max_polls) return false;
        __nanosleep(ns);
        ns = ns < 128 ? ns + 16 : 128;
    }
}

__global__ void __launch_bounds__(1024) copier_kernel(const __grid_constant__ CopierParams p) {
    __shared__ int s_go[2];
    const uint32_t b = blockIdx.x;
    uint32_t s = 0;
    while (s + 1 < p.P && b >= p.cta_base[s + 1]) ++s;
    if (b < p.cta_base[s] || b >= p.cta_base[s + 1]) return;   // spare CTA
    const uint32_t G = p.cta_base[s + 1] - p.cta_base[s];
    const uint32_t j = b - p.cta_base[s];
    const uint64_t* table_s = p.gates + (uint64_t)s * p.n_global * DTT_GATE_WORDS;

    for (uint32_t k = 0; k < p.n_chunks[s]; ++k) {
        const uint32_t c = p.first_chunk[s] + k;
        const ChunkDesc cd = p.chunks[c];
        if (threadIdx.x == 0) {
            const bool ok = poll_gate(table_s + (uint64_t)c * DTT_GATE_WORDS + DTT_GATE_READY,
                                      p.round, p.max_polls);
            if (!ok) {
                atomicAdd(&p.status->copier_timeouts, 1u);
                atomicMin(&p.status->timeout_chunk, c);
            }
            s_go[k & 1] = ok;
        }
        __syncthreads();
        if (!s_go[k & 1]) return;
        const uint32_t i0 = (j + G - cd.rot) % G;
        if (i0 >= cd.n_pieces) continue;
        for (uint32_t i = i0; i < cd.n_pieces; i += G) {
            const PieceDesc pc = p.pieces[cd.piece_begin + i];
            if (pc.vec)
                copy_piece_vec(p, s, pc);
            else
                copy_piece_bytes(p, s, pc);
        }
        __syncthreads();   // every thread's stores of this chunk precede thread 0's release
        if (threadIdx.x == 0) {
            uint64_t* row = p.gates + ((uint64_t)s * p.n_global + c) * DTT_GATE_WORDS;
            const uint64_t done = dtt_dev::atom_add_acq_rel(row + DTT_GATE_COPIER, 1) + 1;
            if (done == (uint64_t)p.round * cd.n_part) {
                // last piece of the chunk: signal arrival at every peer
                for (uint32_t q = 0; q < p.P; ++q) {
                    if (q == s) continue;
                    uint64_t* prow = p.gates + ((uint64_t)q * p.n_global + c) * DTT_GATE_WORDS;
                    if (p.flags & DTT_HANDLE_TIMESTAMPS)
                        dtt_dev::st_relaxed(prow + DTT_GATE_T_ARRIVE, dtt_dev::globaltimer());
                    dtt_dev::red_release_add(prow + DTT_GATE_ARRIVAL, 1);
                }
                dtt_dev::red_release_add(row + DTT_GATE_COMPLETION, p.P - 1);
            }
        }
    }
}

// Completion check: flags[c] = 0 delivered, 1 short (marks or an arrival missing), 2 extra.
__global__ void check_kernel(const __grid_constant__ CheckParams p, uint8_t* flags) {
    for (uint32_t c = blockIdx.x * blockDim.x + threadIdx.x; c < p.n_global;
         c += gridDim.x * blockDim.x) {
        const ChunkDesc cd = p.chunks[c];
        const uint64_t* row = p.gates + ((uint64_t)cd.owner * p.n_global + c) * DTT_GATE_WORDS;
        const uint64_t cnt = dtt_dev::ld_acquire(row + DTT_GATE_COUNTER);
        const uint64_t target = (uint64_t)p.round * cd.writers;
        uint8_t f = 0;
        if (cnt > target || dtt_dev::ld_relaxed(row + DTT_GATE_ERROR) != 0) {
            f = 2;
        } else if (cnt < target) {
            f = 1;
        } else {
            for (uint32_t q = 0; q < p.P; ++q) {
                if (q == cd.owner) continue;
                const uint64_t* prow = p.gates + ((uint64_t)q * p.n_global + c) * DTT_GATE_WORDS;
                if (dtt_dev::ld_acquire(prow + DTT_GATE_ARRIVAL) < p.round) f = 1;
            }
        }
        flags[c] = f;
    }
}

// close() in mid-round: open every gate still closed so the copier sends chunks as they stand.
__global__ void force_open_kernel(uint64_t* gates, const ChunkDesc* chunks, uint32_t n_global,
                                  uint32_t round) {
    for (uint32_t c = blockIdx.x * blockDim.x + threadIdx.x; c < n_global;
         c += gridDim.x * blockDim.x) {
        uint64_t* ready = gates + ((uint64_t)chunks[c].owner * n_global + c) * DTT_GATE_WORDS;
        if ((uint32_t)dtt_dev::ld_acquire(ready) < round) dtt_dev::st_release(ready, round);
    }
}

struct PublishParams {
    dtt_handle h[DTT_MAX_RANKS];
    uint32_t P;
    uint32_t first;
    uint32_t marks;
};

// A producer that only marks: CTA i gives chunk first + i its marks (`marks` of them, or the
// chunk's writer count when marks == 0) on behalf of the rank that owns it.  Work queued
// before it on the same stream (host-to-device copies, other kernels) precedes the marks.
__global__ void publish_kernel(const __grid_constant__ PublishParams p) {
    const uint32_t c = p.first + blockIdx.x;
    uint32_t r = 0;
    while (r < p.P && !(c >= p.h[r].first_chunk && c < p.h[r].first_chunk + p.h[r].n_chunks)) ++r;
    if (r >= p.P) return;
    const dtt_handle& h = p.h[r];
    const uint32_t m = p.marks ? p.marks : h.writers[c];
    for (uint32_t i = 0; i < m; ++i) dtt_mark_ready(h, c);
}

// Consumer: wait for every other rank's chunk with the device-side wait, then copy it out of
// the rank's own buffer.  CTA b takes chunks b, b + gridDim.x, ... in global order.
__global__ void consumer_kernel(const __grid_constant__ CopierParams p, dtt_handle h, char* dst,
                                uint64_t max_polls, int32_t* status) {
    for (uint32_t c = blockIdx.x; c < p.n_global; c += gridDim.x) {
        const ChunkDesc cd = p.chunks[c];
        if (cd.owner == h.rank) {
            if (threadIdx.x == 0) status[c] = 0;
            continue;
        }
        const int w = dtt_wait(h, c, max_polls);
        if (threadIdx.x == 0) status[c] = w;
        if (w != 0) continue;
        const char* src = p.bufs[h.rank];
        for (uint32_t i = 0; i < cd.n_pieces; ++i) {
            const PieceDesc pc = p.pieces[cd.piece_begin + i];
            const uint64_t total = (uint64_t)pc.row_bytes * pc.rows;
            for (uint64_t x = threadIdx.x; x < total; x += blockDim.x) {
                const uint64_t row = x / pc.row_bytes, col = x - row * pc.row_bytes;
                const uint64_t o = pc.off + row * pc.pitch + col;
                dst[o] = src[o];
            }
        }
    }
}

}  // namespace

cudaError_t launch_copier(const CopierParams& p, uint32_t ctas, uint32_t threads, uint32_t method,
                          cudaStream_t s) {
    (void)method;
    copier_kernel<<<ctas, threads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_check(const CheckParams& p, uint8_t* flags, cudaStream_t s) {
    const uint32_t threads = 256;
    uint32_t blocks = (p.n_global + threads - 1) / threads;
    if (blocks == 0) blocks = 1;
    if (blocks > 1024) blocks = 1024;
    check_kernel<<<blocks, threads, 0, s>>>(p, flags);
    return cudaGetLastError();
}

cudaError_t launch_force_open(uint64_t* gates, const ChunkDesc* chunks, uint32_t n_global,
                              uint32_t round, cudaStream_t s) {
    uint32_t blocks = (n_global + 255) / 256;
    if (blocks == 0) blocks = 1;
    force_open_kernel<<<blocks, 256, 0, s>>>(gates, chunks, n_global, round);
    return cudaGetLastError();
}

cudaError_t launch_consumer(const CopierParams& p, dtt_handle h, char* dst, uint64_t max_polls,
                            int32_t* status, uint32_t ctas, cudaStream_t s) {
    if (ctas == 0) ctas = 1;
    if (ctas > p.n_global) ctas = p.n_global ? p.n_global : 1;
    consumer_kernel<<<ctas, 256, 0, s>>>(p, h, dst, max_polls, status);
    return cudaGetLastError();
}

cudaError_t preload_copier_kernels() {
    cudaError_t e = prepare_kernel(copier_kernel);
    if (e == cudaSuccess) e = prepare_kernel(check_kernel);
    if (e == cudaSuccess) e = prepare_kernel(force_open_kernel);
    if (e == cudaSuccess) e = prepare_kernel(publish_kernel);
    if (e == cudaSuccess) e = prepare_kernel(consumer_kernel);
    return e;
}

}  // namespace dtt

using namespace dtt;

extern "C" int dtt_publish(const dtt_handle* handles, uint32_t P, uint32_t first_chunk,
                           uint32_t n_chunks, uint32_t marks, cudaStream_t stream) {
    if (!handles || P < 1 || P > DTT_MAX_RANKS) return fail(DTT_EINVAL, "dtt_publish: bad args");
    if (n_chunks == 0) return DTT_OK;
    PublishParams pp{};
    for (uint32_t r = 0; r < P; ++r) pp.h[r] = handles[r];
    pp.P = P;
    pp.first = first_chunk;
    pp.marks = marks;
    publish_kernel<<<n_chunks, 32, 0, stream>>>(pp);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(DTT_ECUDA, "dtt_publish: launch failed: %s", cudaGetErrorString(e));
    return DTT_OK;
}
