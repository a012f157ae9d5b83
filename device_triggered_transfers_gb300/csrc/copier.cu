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

// Tell the host through mapped memory that chunk c has reached every peer this round (the
// gpu-scope arrival adds above it are ordered before this system-scope release).
__device__ __forceinline__ void notify_host(const CopierParams& p, uint32_t c) {
    if (p.host_arrived)
        asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(p.host_arrived + c), "r"(p.round) : "memory");
}

// Chunk c of source s has landed at every peer: per peer its arrival signal (and time stamp) and
// the peer's counters of the chunk's groups, then the source's completion word and the host
// stamp.  The chunk's group ids are read first; then ONE release fence covers every signal (a
// fence followed by relaxed writes is a release pattern in the PTX memory model): it orders
// every copy of the chunk -- this thread's, or those acquired from the CTAs that made them
// through the piece counter -- before each of them.
__device__ __forceinline__ void signal_arrivals(const CopierParams& p, uint32_t s, uint32_t c,
                                                uint32_t peers, uint32_t receivers) {
    constexpr uint32_t kIdsInRegs = 4;
    uint32_t ga = 0, gb = 0, ids[kIdsInRegs];
    if (p.groups.counters) {
        ga = p.groups.chunk_off[c];
        gb = p.groups.chunk_off[c + 1];
#pragma unroll
        for (uint32_t j = 0; j < kIdsInRegs; ++j) ids[j] = ga + j < gb ? p.groups.chunk_ids[ga + j] : 0;
    }
    dtt_dev::fence_acq_rel();
    for (uint32_t q = 0; q < p.P; ++q) {
        if (!((peers >> q) & 1u)) continue;
        uint64_t* prow = p.gates + ((uint64_t)q * p.n_global + c) * DTT_GATE_WORDS;
        if (p.flags & DTT_HANDLE_TIMESTAMPS) dtt_dev::st_relaxed(prow + DTT_GATE_T_ARRIVE, dtt_dev::globaltimer());
        dtt_dev::red_relaxed_add(prow + DTT_GATE_ARRIVAL, 1);
        if (gb > ga) {
            uint64_t* grow = p.groups.counters + (uint64_t)q * p.groups.n_groups;
#pragma unroll
            for (uint32_t j = 0; j < kIdsInRegs; ++j)
                if (ga + j < gb) dtt_dev::red_relaxed_add(grow + ids[j], 1);
            for (uint32_t i = ga + kIdsInRegs; i < gb; ++i) dtt_dev::red_relaxed_add(grow + p.groups.chunk_ids[i], 1);
        }
    }
    uint64_t* row = p.gates + ((uint64_t)s * p.n_global + c) * DTT_GATE_WORDS;
    dtt_dev::red_relaxed_add(row + DTT_GATE_COMPLETION, receivers);
    notify_host(p, c);
}

// The CTA that takes a chunk's first piece stamps, in the owner's gate row, when the copier began
// the chunk this round (the row's arrival-time word, which only peer rows use otherwise): the
// time from the gate's opening to it is the chunk's wait in its queue, the time from it to each
// arrival the transfer's.
__device__ __forceinline__ void stamp_copy_start(const CopierParams& p, uint32_t s, uint32_t c) {
    if (p.flags & DTT_HANDLE_TIMESTAMPS)
        dtt_dev::st_relaxed(p.gates + ((uint64_t)s * p.n_global + c) * DTT_GATE_WORDS + DTT_GATE_T_ARRIVE,
                            dtt_dev::globaltimer());
}

// Copy one piece from buffer s to each receiver's landing place: 16-byte vectors, kUnroll loads
// in flight per thread, each value stored to every receiver (at the piece's destination).
__device__ __forceinline__ void copy_piece_vec(const CopierParams& p, uint32_t s, uint32_t peers,
                                               const PieceDesc& pc) {
    const uint32_t rv = pc.row_bytes >> 4;
    const uint32_t total = rv * pc.rows;
    const char* src = p.bufs[s] + pc.off;
    const uint32_t stride = blockDim.x * kUnroll;
    for (uint32_t v0 = threadIdx.x; v0 < total; v0 += stride) {
        uint4 val[kUnroll];
        uint64_t doff[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint32_t v = v0 + u * blockDim.x;
            if (v < total) {
                uint32_t row = 0, col = v;
                if (pc.rows > 1) {
                    row = v / rv;
                    col = v - row * rv;
                }
                val[u] = ld_cg16(src + (uint64_t)row * pc.pitch + ((uint64_t)col << 4));
                doff[u] = (uint64_t)row * pc.dst_pitch + ((uint64_t)col << 4);
            }
        }
#pragma unroll 1
        for (uint32_t q = 0; q < p.P; ++q) {
            if (!((peers >> q) & 1u)) continue;
            char* dst = p.dst[q] + pc.dst_off;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const uint32_t v = v0 + u * blockDim.x;
                if (v < total) st_cs16(dst + doff[u], val[u]);
            }
        }
    }
}

// Byte-wise copy for pieces that are not 16-byte aligned.
__device__ __forceinline__ void copy_piece_bytes(const CopierParams& p, uint32_t s, uint32_t peers,
                                                 const PieceDesc& pc) {
    const uint64_t total = (uint64_t)pc.row_bytes * pc.rows;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(p.bufs[s]) + pc.off;
    for (uint64_t b = threadIdx.x; b < total; b += blockDim.x) {
        const uint64_t row = b / pc.row_bytes, col = b - row * pc.row_bytes;
        const uint8_t v = ld_cg8(src + row * pc.pitch + col);
        const uint64_t o = pc.dst_off + row * pc.dst_pitch + col;
        for (uint32_t q = 0; q < p.P; ++q)
            if ((peers >> q) & 1u) reinterpret_cast<uint8_t*>(p.dst[q])[o] = v;
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

__device__ __forceinline__ void copier_body(const CopierParams& p) {
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
                atomicMax(&p.status->timeout_inv, 0xFFFFFFFFu - c);
            }
            s_go[k & 1] = ok;
        }
        __syncthreads();
        if (!s_go[k & 1]) return;
        const uint32_t i0 = (j + G - cd.rot) % G;
        if (i0 >= cd.n_pieces) continue;
        if (i0 == 0 && threadIdx.x == 0) stamp_copy_start(p, s, c);
        for (uint32_t i = i0; i < cd.n_pieces; i += G) {
            const PieceDesc pc = p.pieces[cd.piece_begin + i];
            if (pc.vec)
                copy_piece_vec(p, s, cd.peers, pc);
            else
                copy_piece_bytes(p, s, cd.peers, pc);
        }
        __syncthreads();   // every thread's stores of this chunk precede thread 0's release
        if (threadIdx.x == 0) {
            uint64_t* row = p.gates + ((uint64_t)s * p.n_global + c) * DTT_GATE_WORDS;
            const uint64_t done = dtt_dev::atom_add_acq_rel(row + DTT_GATE_COPIER, 1) + 1;
            if (done == (uint64_t)p.round * cd.n_part) signal_arrivals(p, s, c, cd.peers, cd.receivers);   // the chunk's last piece
        }
    }
}

// This round's copier CTAs count themselves out once their work (and every store and arrival
// of it) is done; the check waits for the count instead of following the copier on its stream.
__device__ __forceinline__ void count_out(const CopierParams& p) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&p.status->copier_exit) : "memory");
}

// ---- early launch --------------------------------------------------------------------------------
// A copier that dtt_plan_wait launched for the next round before the host started that round
// (opts.early_copier_us; it queues behind this round's copier on the copy stream, so its launch
// costs the next round nothing -- the pages' "prepare" step arms the copy engine's queue ahead of
// the round in the same way).  CTA 0's thread 0 waits until plan_start claims the round on the
// mapped handshake word, or gives the round up after go_wait_ns with a compare-and-swap of its
// own -- exactly one side wins -- and publishes the decision for the other CTAs.  A copier whose
// round was given up (or aborted by the host) exits without touching a gate or a status word,
// not even the count-out, and plan_start launches a fresh one.

__device__ __forceinline__ uint64_t ld_acquire_sys(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.acquire.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t cas_sys(uint64_t* p, uint64_t cmp, uint64_t val) {
    uint64_t old;
    asm volatile("atom.acq_rel.sys.global.cas.b64 %0, [%1], %2, %3;"
                 : "=l"(old) : "l"(p), "l"(cmp), "l"(val) : "memory");
    return old;
}

// Thread 0 of CTA 0: has the host started this copier's round?  Bounded by go_wait_ns.
__device__ __forceinline__ bool early_decide(const CopierParams& p) {
    const uint64_t start = early_start_value(p.round), stop = early_stop_value(p.round);
    const uint64_t t0 = dtt_dev::globaltimer();
    bool go = false;
    for (;;) {
        const uint64_t v = ld_acquire_sys(p.go_host);
        if (v == start) { go = true; break; }
        if (v != p.go_prior) break;                          // the host aborted the round
        if (dtt_dev::globaltimer() - t0 >= p.go_wait_ns) {
            go = cas_sys(p.go_host, p.go_prior, stop) == start;   // the host may have just claimed it
            break;
        }
        __nanosleep(256);
    }
    dtt_dev::st_release(&p.status->early_go, go ? start : stop);
    return go;
}

// Thread 0 of every other CTA: CTA 0's decision, 1 go / 0 given up, or -1 when it did not come
// within twice CTA 0's bound plus a millisecond (CTA 0's own wait is bounded, so this is a
// safety net that ends the CTA as a copier timeout).
__device__ __forceinline__ int early_follow(const CopierParams& p) {
    const uint64_t start = early_start_value(p.round);
    const uint64_t t0 = dtt_dev::globaltimer(), limit = 2 * p.go_wait_ns + 1000000;
    uint32_t ns = 0;
    for (;;) {
        const uint64_t v = dtt_dev::ld_acquire(&p.status->early_go);
        if (v >= start) return v == start ? 1 : 0;
        if (dtt_dev::globaltimer() - t0 >= limit) return -1;
        __nanosleep(ns);
        ns = ns < 256 ? ns + 32 : 256;
    }
}

// Thread 0: the early handshake of this CTA (1 go, 0 exit silently, -1 exit as a timeout).
__device__ __forceinline__ int early_gate(const CopierParams& p) {
    const int e = blockIdx.x == 0 ? (early_decide(p) ? 1 : 0) : early_follow(p);
    if (e < 0) atomicAdd(&p.status->copier_timeouts, 1u);
    return e;
}

__global__ void __launch_bounds__(1024) copier_kernel(const __grid_constant__ CopierParams p) {
    if (p.go_host) {
        __shared__ int s_early;
        if (threadIdx.x == 0) s_early = early_gate(p);
        __syncthreads();
        const int e = s_early;
        if (e <= 0) {
            if (e < 0 && threadIdx.x == 0) count_out(p);
            return;
        }
    }
    copier_body(p);
    __syncthreads();
    if (threadIdx.x == 0) count_out(p);
}

// ---- bulk-copy (TMA) path ----------------------------------------------------------------------
// One thread per CTA drives the copy engine of its SM: bulk loads (cp.async.bulk, completing on
// an mbarrier) fill a ring of shared-memory stages, and each stage is written back to every peer
// with bulk stores.  Loads of later pieces overlap the stores of earlier ones.  The SM's other
// resources stay free for the producer.  Every piece fits one stage (the plan cuts them so) and
// is 16-byte aligned.  A 2D window of short rows moves as one tensor-map box (one load, one
// store per peer) instead of a bulk copy per row.

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Bounded wait for the phase with the given parity.  Returns false when the polls run out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < (1u << 26); ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done) : "r"(bar), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}

// L2 policy for the copier's own traffic: a source chunk is read once and a peer's copy is not
// read again by the copier, so both are the first lines L2 gives up -- the chunks the producer
// is writing right now stay cached until the copier reads them.
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_load(uint32_t dst_smem, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;"
        ::"r"(dst_smem), "l"(src), "r"(bytes), "r"(bar), "l"(pol) : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, uint32_t src_smem, uint32_t bytes, uint64_t pol) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
                 ::"l"(dst), "r"(src_smem), "r"(bytes), "l"(pol) : "memory");
}

// One box of a 2D window through its tensor map (8-byte elements, no swizzle): a load into a
// shared-memory stage completing on an mbarrier, and a store from the stage.
__device__ __forceinline__ void tensor_load(uint32_t dst_smem, const CUtensorMap* map, uint32_t x, uint32_t y,
                                            uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(dst_smem), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void tensor_store(const CUtensorMap* map, uint32_t x, uint32_t y, uint32_t src_smem,
                                             uint64_t pol) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(src_smem), "l"(pol) : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void copier_bulk_body(const CopierParams& p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t b = blockIdx.x;
    uint32_t s = 0;
    while (s + 1 < p.P && b >= p.cta_base[s + 1]) ++s;
    if (b < p.cta_base[s] || b >= p.cta_base[s + 1]) return;
    const uint32_t G = p.cta_base[s + 1] - p.cta_base[s];
    const uint32_t j = b - p.cta_base[s];
    const uint32_t S = p.stages;
    const uint64_t pol = evict_first_policy();
    uint8_t* stage0 = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)S * p.stage_bytes);
    for (uint32_t i = 0; i < S; ++i) mbar_init(smem_addr(bars + i), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");

    const char* src_base = p.bufs[s];
    const uint64_t* table_s = p.gates + (uint64_t)s * p.n_global * DTT_GATE_WORDS;
    uint64_t it0 = 0;          // items issued so far by this CTA (stage and phase bookkeeping)
    uint64_t loads_hi = 0;     // loads issued: indices [0, loads_hi)
    uint64_t waited_hi = 0;    // loads whose stage has been seen full: indices [0, waited_hi)
    bool failed = false;

    auto load = [&](const PieceDesc& pc, uint64_t idx) {
        const uint32_t st = (uint32_t)(idx % S);
        const uint32_t bar = smem_addr(bars + st);
        const uint32_t dst = smem_addr(stage0 + (size_t)st * p.stage_bytes);
        mbar_expect_tx(bar, pc.row_bytes * pc.rows);
        if (pc.tmap != kNoMap) {
            tensor_load(dst, p.tmaps + (size_t)pc.tmap * p.P + s, pc.x, pc.y, bar, pol);
        } else {
            for (uint32_t r = 0; r < pc.rows; ++r)
                bulk_load(dst + r * pc.row_bytes, src_base + pc.off + (uint64_t)r * pc.pitch, pc.row_bytes, bar, pol);
        }
        loads_hi = idx + 1;
    };
    uint32_t peers = 0;        // receivers of the chunk being copied
    auto store = [&](const PieceDesc& pc, uint64_t idx) {
        const uint32_t st = (uint32_t)(idx % S);
        const uint32_t src = smem_addr(stage0 + (size_t)st * p.stage_bytes);
        for (uint32_t q = 0; q < p.P; ++q) {
            if (!((peers >> q) & 1u)) continue;
            if (pc.tmap != kNoMap) {       // lands at its own offsets: the same map shape
                tensor_store(p.tmaps + (size_t)pc.tmap * p.P + q, pc.x, pc.y, src, pol);
                continue;
            }
            char* dst = p.dst[q] + pc.dst_off;
            for (uint32_t r = 0; r < pc.rows; ++r)
                bulk_store(dst + (uint64_t)r * pc.dst_pitch, src + r * pc.row_bytes, pc.row_bytes, pol);
        }
        bulk_commit();
    };

    for (uint32_t k = 0; k < p.n_chunks[s] && !failed; ++k) {
        const uint32_t c = p.first_chunk[s] + k;
        const ChunkDesc cd = p.chunks[c];
        if (!poll_gate(table_s + (uint64_t)c * DTT_GATE_WORDS + DTT_GATE_READY, p.round, p.max_polls)) {
            atomicAdd(&p.status->copier_timeouts, 1u);
            atomicMax(&p.status->timeout_inv, 0xFFFFFFFFu - c);
            break;
        }
        fence_proxy_async_global();   // the producer's writes, acquired above, precede the bulk loads
        peers = cd.peers;
        const uint32_t i0 = (j + G - cd.rot) % G;
        if (i0 >= cd.n_pieces) continue;
        if (i0 == 0) stamp_copy_start(p, s, c);
        const uint32_t n = (cd.n_pieces - i0 + G - 1) / G;       // my pieces of this chunk
        const PieceDesc* mine = p.pieces + cd.piece_begin + i0;  // stride G
        const uint32_t pre = n < S - 1 ? n : S - 1;
        for (uint32_t t = 0; t < pre; ++t) load(mine[(uint64_t)t * G], it0 + t);
        for (uint32_t t = 0; t < n; ++t) {
            const uint64_t idx = it0 + t;
            if (!mbar_wait(smem_addr(bars + idx % S), (uint32_t)((idx / S) & 1))) {
                atomicAdd(&p.status->bulk_timeouts, 1u);
                failed = true;
                break;
            }
            waited_hi = idx + 1;
            store(mine[(uint64_t)t * G], idx);
            const uint32_t u = t + S - 1;
            if (u < n) {
                if (t >= 1) bulk_wait_read1();    // piece t-1 has left the stage piece u reuses
                load(mine[(uint64_t)u * G], it0 + u);
            }
        }
        bulk_wait_all();              // every store of this chunk has been written
        fence_proxy_async_global();   // ... and is ordered before the generic-proxy release below
        it0 += n;
        if (failed) break;
        uint64_t* row = p.gates + ((uint64_t)s * p.n_global + c) * DTT_GATE_WORDS;
        const uint64_t done = dtt_dev::atom_add_acq_rel(row + DTT_GATE_COPIER, 1) + 1;
        if (done == (uint64_t)p.round * cd.n_part) signal_arrivals(p, s, c, cd.peers, cd.receivers);
    }
    // leave nothing in flight: stores, and (after a failed wait) loads still landing in the ring
    bulk_wait_all();
    for (uint64_t idx = waited_hi + (failed ? 1 : 0); idx < loads_hi; ++idx)
        if (!mbar_wait(smem_addr(bars + idx % S), (uint32_t)((idx / S) & 1))) break;
}

__global__ void __launch_bounds__(32) copier_bulk_kernel(const __grid_constant__ CopierParams p) {
    if (threadIdx.x != 0) return;       // one thread drives the CTA's bulk copies
    if (p.go_host) {
        const int e = early_gate(p);
        if (e <= 0) {
            if (e < 0) count_out(p);
            return;
        }
    }
    copier_bulk_body(p);
    count_out(p);
}

// wait()'s completion check, run after the copier and the producer: one flag per chunk, written
// straight into the mapped host block.  A pending round (overlapping rounds) is checked while the
// next round's marks may already count: a count above round * writers is then no extra mark by
// itself, and only the error word -- set by the mark that passes its own round's count -- is.  The last CTA to finish copies the status words out,
// zeroes them for the next round, and only then stores the sequence number the host polls for.
__global__ void check_kernel(const __grid_constant__ CheckParams p) {
    // launched after the producers on their stream; the copier counts its CTAs out
    if (threadIdx.x == 0) {
        uint32_t late = 0;
        if (p.copier_ctas) {
            late = 1;
            uint32_t ns = 0;
            for (uint64_t i = 0; i < p.max_polls; ++i) {
                uint32_t n;
                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(n) : "l"(&p.status->copier_exit) : "memory");
                if (n >= p.copier_ctas) { late = 0; break; }
                __nanosleep(ns);
                ns = ns < 128 ? ns + 32 : 128;   // a late wake-up delays the whole round
            }
        }
        if (late) atomicExch(&p.status->check_late, 1u);
    }
    // Thread 0's acquire of the copier's count-out (every copier CTA adds to it with a release
    // after its arrival signals) and the barrier order the gate words read below after all of
    // the round's copier writes; the producers finished before this kernel started.  So the
    // reads need no acquire of their own and go out together.
    __syncthreads();
    for (uint32_t c = blockIdx.x * blockDim.x + threadIdx.x; c < p.n_global;
         c += gridDim.x * blockDim.x) {
        const ChunkDesc cd = p.chunks[c];
        const uint64_t* row = p.gates + ((uint64_t)cd.owner * p.n_global + c) * DTT_GATE_WORDS;
        const uint64_t cnt = dtt_dev::ld_relaxed(row + DTT_GATE_COUNTER);
        const uint64_t err = dtt_dev::ld_relaxed(row + DTT_GATE_ERROR);
        bool arrived = true;
        for (uint32_t q = 0; q < p.P; ++q) {
            if (!((cd.peers >> q) & 1u)) continue;
            const uint64_t* prow = p.gates + ((uint64_t)q * p.n_global + c) * DTT_GATE_WORDS;
            arrived &= dtt_dev::ld_relaxed(prow + DTT_GATE_ARRIVAL) >= p.round;
        }
        const uint64_t target = (uint64_t)p.round * cd.writers;
        const bool extra = err != 0 || (!p.pending && cnt > target);
        p.host_flags[c] = extra ? 2 : (cnt < target || !arrived) ? 1 : 0;
    }
    __shared__ uint32_t s_last;
    __syncthreads();                     // the CTA's flag stores, then one release for all of them
    if (threadIdx.x == 0) {
        if (gridDim.x == 1) {
            s_last = 1;                  // the fence before the sequence number covers the flags
        } else {
            uint32_t prev;
            asm volatile("fence.acq_rel.sys;\n\t"
                         "atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                         : "=r"(prev) : "l"(&p.status->check_arrive) : "memory");
            s_last = prev == gridDim.x - 1;
        }
    }
    __syncthreads();
    if (!s_last || threadIdx.x != 0) return;
    DevStatus* d = p.status;
    volatile uint32_t* hs = &p.host->st.misuse;
    hs[0] = d->misuse;
    hs[1] = d->copier_timeouts;
    hs[2] = d->timeout_inv;
    hs[3] = d->bulk_timeouts;
    hs[5] = d->copier_exit;
    hs[6] = d->check_late;
    d->misuse = 0;
    d->copier_timeouts = 0;
    d->timeout_inv = 0;
    d->bulk_timeouts = 0;
    d->check_arrive = 0;
    d->copier_exit = 0;
    d->check_late = 0;
    asm volatile("fence.acq_rel.sys;\n\t"
                 "st.release.sys.global.u32 [%0], %1;" ::"l"(&p.host->done), "r"(p.seq) : "memory");
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

// The copy-engine transport's ATOMIC step: stream-ordered after every copy of the run of chunks
// [c, c_end) to every peer (so those bytes are visible to this kernel), one thread signals each
// chunk of the run, in order, as the SM copier does.
__global__ void ce_signal_kernel(const __grid_constant__ CeSignalParams p) {
    if (threadIdx.x != 0) return;
    dtt_dev::fence_acq_rel();
    for (uint32_t c = p.c; c < p.c_end; ++c) {
        for (uint32_t q = 0; q < p.P; ++q) {
            if (!((p.peers >> q) & 1u)) continue;
            uint64_t* prow = p.gates + ((uint64_t)q * p.n_global + c) * DTT_GATE_WORDS;
            if (p.flags & DTT_HANDLE_TIMESTAMPS) dtt_dev::st_relaxed(prow + DTT_GATE_T_ARRIVE, dtt_dev::globaltimer());
            dtt_dev::red_relaxed_add(prow + DTT_GATE_ARRIVAL, 1);
            if (p.groups.counters) {
                uint64_t* grow = p.groups.counters + (uint64_t)q * p.groups.n_groups;
                for (uint32_t i = p.groups.chunk_off[c]; i < p.groups.chunk_off[c + 1]; ++i)
                    dtt_dev::red_relaxed_add(grow + p.groups.chunk_ids[i], 1);
            }
        }
        uint64_t* row = p.gates + ((uint64_t)p.s * p.n_global + c) * DTT_GATE_WORDS;
        dtt_dev::red_relaxed_add(row + DTT_GATE_COMPLETION, p.receivers);
        if (p.host_arrived)
            asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(p.host_arrived + c), "r"(p.round) : "memory");
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
        if (!((cd.peers >> h.rank) & 1u)) {       // its own chunk, or not addressed to it
            if (threadIdx.x == 0) status[c] = 0;
            continue;
        }
        const int w = dtt_wait(h, c, max_polls);
        if (threadIdx.x == 0) status[c] = w;
        if (w != 0) continue;
        const char* src = p.dst[h.rank];          // where this rank's copies landed
        for (uint32_t i = 0; i < cd.n_pieces; ++i) {
            const PieceDesc pc = p.pieces[cd.piece_begin + i];
            const uint64_t total = (uint64_t)pc.row_bytes * pc.rows;
            for (uint64_t x = threadIdx.x; x < total; x += blockDim.x) {
                const uint64_t row = x / pc.row_bytes, col = x - row * pc.row_bytes;
                const uint64_t o = pc.dst_off + row * pc.dst_pitch + col;
                dst[o] = src[o];
            }
        }
    }
}

}  // namespace

cudaError_t launch_copier(const CopierParams& p, uint32_t ctas, uint32_t threads, uint32_t method,
                          cudaStream_t s) {
    if (method == DTT_COPY_TMA) {
        const size_t smem = bulk_smem_bytes(p.stage_bytes, p.stages);
        copier_bulk_kernel<<<ctas, 32, smem, s>>>(p);
    } else {
        copier_kernel<<<ctas, threads, 0, s>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_check(const CheckParams& p, cudaStream_t s) {
    const uint32_t threads = 256;
    uint32_t blocks = (p.n_global + threads - 1) / threads;
    if (blocks == 0) blocks = 1;
    if (blocks > 1024) blocks = 1024;
    check_kernel<<<blocks, threads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_force_open(uint64_t* gates, const ChunkDesc* chunks, uint32_t n_global,
                              uint32_t round, cudaStream_t s) {
    uint32_t blocks = (n_global + 255) / 256;
    if (blocks == 0) blocks = 1;
    force_open_kernel<<<blocks, 256, 0, s>>>(gates, chunks, n_global, round);
    return cudaGetLastError();
}

cudaError_t launch_ce_signal(const CeSignalParams& p, cudaStream_t s) {
    ce_signal_kernel<<<1, 32, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_consumer(const CopierParams& p, dtt_handle h, char* dst, uint64_t max_polls,
                            int32_t* status, uint32_t ctas, cudaStream_t s) {
    if (ctas == 0) ctas = 1;
    if (ctas > p.n_global) ctas = p.n_global ? p.n_global : 1;
    consumer_kernel<<<ctas, 256, 0, s>>>(p, h, dst, max_polls, status);
    return cudaGetLastError();
}

cudaError_t copier_regs_per_thread(uint32_t method, int* regs) {
    cudaFuncAttributes a{};
    const cudaError_t e = method == DTT_COPY_TMA ? cudaFuncGetAttributes(&a, copier_bulk_kernel)
                                                 : cudaFuncGetAttributes(&a, copier_kernel);
    *regs = a.numRegs;
    return e;
}

cudaError_t copier_static_smem(uint32_t method, size_t* bytes) {
    cudaFuncAttributes a{};
    const cudaError_t e = method == DTT_COPY_TMA ? cudaFuncGetAttributes(&a, copier_bulk_kernel)
                                                 : cudaFuncGetAttributes(&a, copier_kernel);
    *bytes = a.sharedSizeBytes;
    return e;
}

cudaError_t preload_copier_kernels() {
    cudaError_t e = prepare_kernel(copier_kernel);
    if (e == cudaSuccess) e = prepare_kernel(copier_bulk_kernel);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(copier_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kBulkSmemMax);
    if (e == cudaSuccess) e = prepare_kernel(check_kernel);
    if (e == cudaSuccess) e = prepare_kernel(force_open_kernel);
    if (e == cudaSuccess) e = prepare_kernel(publish_kernel);
    if (e == cudaSuccess) e = prepare_kernel(consumer_kernel);
    if (e == cudaSuccess) e = prepare_kernel(ce_signal_kernel);
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
