// The GEMM producer: a persistent tcgen05 / TMEM bf16 GEMM that marks each 128 x 128 tile's
// chunk as soon as the tile is stored ("Triggered Plans", section Model: a tiled producer "such
// as a GEMM"; program p takes steps p, p + num_programs, ... and marks first_chunk + step /
// num_programs).  One launch covers every virtual rank: C_r = A_r . B for r = 0..P-1.
//
// Per CTA (one per SM, 192 threads), warp-specialised:
//   warp 4      TMA: loads 128 x 64 bf16 tiles of A_r and of B^T (K-major, 128-byte swizzle)
//               into a ring of shared-memory stages, completing on mbarriers;
//   warp 5      MMA: one thread issues tcgen05.mma (M = 128, N = TN = 256 when N allows it,
//               else 128, K = 16, fp32 accumulate in TMEM) and commits each stage back to the
//               TMA warp, and each finished block of TN / 128 tiles to the epilogue;
//   warps 0-3   epilogue: tcgen05.ld the accumulator (warp w owns TMEM lanes 32w..32w+31 =
//               tile rows), round to bf16, store to the rank's buffer, then a named barrier
//               over these 128 threads and one mark.
// Two TMEM accumulators (2 x TN columns) let the MMA warp start the next block while the
// epilogue drains the previous one; the epilogue marks each 128 x 128 tile of a block.  Every wait is bounded; on a timeout the CTA records an
// error, lets its copies and MMAs finish (bounded), frees its TMEM and returns.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "dtt_device.cuh"
#include "internal.h"

namespace dtt {
namespace {

constexpr uint32_t BM = 128, BN = 128, BK = 64, UMMA_K = 16;   // BM x BN: the marked tile
constexpr uint32_t A_STAGE = BM * BK * 2;            // 16 KiB
constexpr uint32_t ACC_BUFS = 2;
constexpr uint32_t EPI_THREADS = 128;
constexpr uint32_t THREADS = EPI_THREADS + 64;       // + TMA warp + MMA warp
constexpr uint32_t TMA_WARP = 4, MMA_WARP = 5;
constexpr uint32_t WAIT_LIMIT = 1u << 22;

// One MMA covers TN columns: TN / 128 adjacent marked tiles of one tile row.  TN = 256 halves the
// shared-memory traffic per FLOP for A (the 128 x 128 form needs ~112 B/clk of operand reads per
// SM at full rate, close to what shared memory delivers).
template <uint32_t TN>
struct Cfg {
    static constexpr uint32_t UNIT = TN / BN;                         // tiles per MMA block
    static constexpr uint32_t STAGES = TN == 256 ? 4 : 6;
    static constexpr uint32_t B_STAGE = TN * BK * 2;
    static constexpr uint32_t TMEM_COLS = ACC_BUFS * TN;              // 256 or 512 fp32 columns
    static constexpr uint32_t SMEM_BYTES = 1024 /* alignment slack */ + STAGES * (A_STAGE + B_STAGE) + 256;
    // instruction descriptor (kind::f16): D fp32, A and B bf16, both K-major, N = TN, M = 128
    static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((TN >> 3) << 17) | ((BM >> 4) << 24);
};

struct GemmParams {
    CUtensorMap tmA;     // A, all ranks stacked: [P*M rows, K] bf16, box 64 x 128
    CUtensorMap tmB;     // B^T: [N rows, K] bf16, box 64 x 128
    char* bufs[DTT_MAX_RANKS];
    dtt_handle h[DTT_MAX_RANKS];
    uint64_t slice_off[DTT_MAX_RANKS];
    uint64_t ldc;
    uint32_t P, M, N, K, NP;
    uint32_t* err;
};

__device__ __forceinline__ uint32_t saddr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void bar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void bar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Bounded wait for the phase of the given parity; false when the limit ran out or another role
// already reported an error.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort) {
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done) : "r"(bar), "r"(parity) : "memory");
        if (done) return true;
        if ((i & 255) == 255 && *abort) return false;
    }
    return false;
}

// AND of v over the 128 epilogue threads (named barrier 1), the same result in every thread.
__device__ __forceinline__ bool epi_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"((uint32_t)v), "n"(EPI_THREADS) : "memory");
    return r != 0;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar) : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);          // start address
    d |= (uint64_t)1 << 16;                           // leading byte offset (unused here)
    d |= (uint64_t)(1024u >> 4) << 32;                // stride byte offset
    d |= (uint64_t)1 << 46;                           // descriptor version
    d |= (uint64_t)2 << 61;                           // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(__uint_as_float(hi)), "f"(__uint_as_float(lo)));
    return r;
}

// Overlapping rounds (the handle's DTT_HANDLE_OVERLAP flag): one thread waits until the chunks
// of rank h.rank's tiles [t0, t0 + n) (row-major tile indices) may be written -- the previous
// round's copies of them have landed -- before the epilogue stores them.  False when a wait ran
// out (DTT_DEV_EWRITABLE is set; the caller stops the GEMM).
__device__ __forceinline__ bool unit_writable(const dtt_handle& h, uint32_t t0, uint32_t n, uint32_t NP) {
    if (!(h.flags & DTT_HANDLE_OVERLAP)) return true;
    for (uint32_t c = h.first_chunk + t0 / NP; c <= h.first_chunk + (t0 + n - 1) / NP; ++c)
        if (!dtt_dev::wait_writable_one(h, c, kWritablePolls)) {
            atomicOr(h.status, DTT_DEV_EWRITABLE);
            return false;
        }
    return true;
}

// Work is cut in units of TN / 128 adjacent tiles of one tile row.  Every rank's units form one
// sequence, the ranks taking turns (unit 0 of rank 0, of rank 1, ..., then unit 1 of each), and
// program p takes its places p, p + NP, ..., so no program has more than one unit above the
// mean and every rank's chunks open at the same pace: the copier's CTAs of every source have
// work all along, and the last chunks to open are small ones of every rank, not one rank's
// whole tail.  Tile (tm, tn) is step tm * tiles_n + tn of its rank and, once stored, gets one
// mark on chunk first_chunk + step / NP.
template <uint32_t TN>
__global__ void __launch_bounds__(THREADS, 1) gemm_producer_kernel(const __grid_constant__ GemmParams p) {
    using G = Cfg<TN>;
    constexpr uint32_t STAGES = G::STAGES, B_STAGE = G::B_STAGE, TMEM_COLS = G::TMEM_COLS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_STAGE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_STAGE);
    uint64_t* full = bars;                        // [STAGES]  TMA -> MMA
    uint64_t* empty = bars + STAGES;              // [STAGES]  MMA -> TMA
    uint64_t* acc_full = bars + 2 * STAGES;       // [2]       MMA -> epilogue
    uint64_t* acc_empty = acc_full + ACC_BUFS;    // [2]       epilogue -> MMA
    uint64_t* drain = acc_empty + ACC_BUFS;       // [1]       MMA teardown
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const uint32_t warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (uint32_t i = 0; i < STAGES; ++i) {
            bar_init(saddr(full + i), 1);
            bar_init(saddr(empty + i), 1);
        }
        for (uint32_t i = 0; i < ACC_BUFS; ++i) {
            bar_init(saddr(acc_full + i), 1);
            bar_init(saddr(acc_empty + i), EPI_THREADS);
        }
        bar_init(saddr(drain), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(saddr(tmem_slot)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const uint32_t tiles_n = p.N / BN, units_n = p.N / TN, units = (p.M / BM) * units_n;
    const uint32_t kblocks = p.K / BK;
    auto fail = [&]() {
        *abort_flag = 1;
        atomicAdd(p.err, 1u);
    };

    if (warp == TMA_WARP) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, issued = 0;
            bool ok = true;
            for (uint32_t gu = blockIdx.x; gu < p.P * units && ok; gu += p.NP) {
                    const uint32_t r = gu % p.P, u = gu / p.P;
                    const int32_t row_a = (int32_t)(r * p.M + (u / units_n) * BM);
                    const int32_t row_b = (int32_t)((u % units_n) * TN);
                    for (uint32_t kb = 0; kb < kblocks; ++kb) {
                        if (!bar_wait(saddr(empty + stage), phase ^ 1, abort_flag)) { fail(); ok = false; break; }
                        bar_expect_tx(saddr(full + stage), A_STAGE + B_STAGE);
                        tma_load_2d(saddr(sA + stage * A_STAGE), &p.tmA, (int32_t)(kb * BK), row_a, saddr(full + stage));
                        tma_load_2d(saddr(sB + stage * B_STAGE), &p.tmB, (int32_t)(kb * BK), row_b, saddr(full + stage));
                        ++issued;
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                }
            // the last loads of every stage have landed before the CTA can leave
            volatile uint32_t never = 0;
            for (uint32_t i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
                (void)bar_wait(saddr(full + i % STAGES), (i / STAGES) & 1, &never);
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (uint32_t gu = blockIdx.x; gu < p.P * units && ok; gu += p.NP) {
                    if (!bar_wait(saddr(acc_empty + acc), acc_phase ^ 1, abort_flag)) { fail(); ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + acc * TN;
                    for (uint32_t kb = 0; kb < kblocks; ++kb) {
                        if (!bar_wait(saddr(full + stage), phase, abort_flag)) { fail(); ok = false; break; }
                        tc_fence_after();
                        const uint64_t da = smem_desc(saddr(sA + stage * A_STAGE));
                        const uint64_t db = smem_desc(saddr(sB + stage * B_STAGE));
#pragma unroll
                        for (uint32_t k = 0; k < BK / UMMA_K; ++k)
                            umma(d_tmem, da + 2 * k, db + 2 * k, G::IDESC, (kb | k) != 0);
                        umma_commit(saddr(empty + stage));     // the stage is free once these finish
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    umma_commit(saddr(acc_full + acc));        // the tile is complete in TMEM
                    if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1; }
                }
            // every MMA this thread issued has finished before TMEM is released
            umma_commit(saddr(drain));
            volatile uint32_t never = 0;
            (void)bar_wait(saddr(drain), 0, &never);
        }
    } else {
        // epilogue warps 0..3: thread t of warp w owns row 32w + t of every tile
        uint32_t acc = 0, acc_phase = 0;
        const uint32_t row_in_tile = warp * 32 + lane;
        bool ok = true;
        for (uint32_t gu = blockIdx.x; gu < p.P * units && ok; gu += p.NP) {
                const uint32_t r = gu % p.P, u = gu / p.P;
                const uint32_t tm = u / units_n, tn0 = (u % units_n) * G::UNIT;
                bool mine = bar_wait(saddr(acc_full + acc), acc_phase, abort_flag);
                if (!mine) fail();
                if (threadIdx.x == 0 && mine && !unit_writable(p.h[r], tm * tiles_n + tn0, G::UNIT, p.NP)) {
                    fail();
                    mine = false;
                }
                // one decision for all 128 epilogue threads, so none is left at a barrier
                if (!epi_all(mine && !*abort_flag)) { ok = false; break; }
                tc_fence_after();
                char* crow = p.bufs[r] + p.slice_off[r] + (uint64_t)(tm * BM + row_in_tile) * p.ldc +
                             (uint64_t)tn0 * BN * 2;
                const uint32_t taddr = tmem_base + ((warp * 32u) << 16) + acc * TN;
#pragma unroll 1
                for (uint32_t g = 0; g < TN / 32; ++g) {
                    uint32_t v[32];
                    tmem_ld32(taddr + g * 32, v);
                    uint4* dst = reinterpret_cast<uint4*>(crow + g * 64);
#pragma unroll
                    for (uint32_t q = 0; q < 4; ++q)
                        dst[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                                            pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
                }
                tc_fence_before();
                bar_arrive(saddr(acc_empty + acc));            // TMEM buffer may be overwritten
                // the unit's stores by all 128 threads precede one mark per tile
                asm volatile("bar.sync 1, %0;" ::"n"(EPI_THREADS) : "memory");
                if (threadIdx.x == 0)
                    for (uint32_t k = 0; k < G::UNIT; ++k)
                        dtt_dev::mark_one(p.h[r], p.h[r].first_chunk + (tm * tiles_n + tn0 + k) / p.NP);
                if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1; }
            }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS) : "memory");
}

// ---- the consumer form ----------------------------------------------------------------------
// The peer kernel of a triggered plan ("Triggered Plans", Model: peer kernel wait(chunk); Memory
// ordering, Consumer): D = X_q . W^T over rank q's gathered buffer X_q, loading each 128-row
// block of X_q only once every chunk covering those rows has arrived at q this round (q's own
// chunks: once they are ready), so the GEMM runs while the all-gather is still delivering.
struct ConsumerParams {
    CUtensorMap tmX;     // X_q: [rows, K] bf16, box 64 x 128
    CUtensorMap tmW;     // W^T: [N, K] bf16, box 64 x TN
    dtt_handle h;        // rank q's handle for this round
    const uint32_t* order;   // row blocks in the order they are taken
    const uint32_t* c0;      // per row block: the chunk ids [c0, c1] that cover it
    const uint32_t* c1;
    const uint32_t* order2;  // pair form: pairs of row blocks (2 pb, 2 pb + 1) in the order taken
    const uint32_t* bgroup;  // per row block: its chunk group (one wait), or null: wait per chunk
    char* D;
    uint64_t ldd;
    uint64_t max_polls;
    uint32_t blocks, N, K;
    uint32_t* err;
};

// Bounded wait for every chunk in [c0, c1] at rank h.rank, then order the data read by the
// bulk copies that follow after the acquire.
__device__ __forceinline__ bool wait_chunks(const dtt_handle& h, uint32_t c0, uint32_t c1, uint64_t max_polls,
                                            volatile uint32_t* abort) {
    for (uint32_t c = c0; c <= c1; ++c) {
        const uint64_t* w = dtt_dev::wait_word(h, c);
        uint32_t ns = 0;
        bool ok = false;
        for (uint64_t i = 0; i < max_polls; ++i) {
            if ((uint32_t)dtt_dev::ld_acquire(w) >= h.round) { ok = true; break; }
            if ((i & 63) == 63 && *abort) return false;
            __nanosleep(ns);
            ns = ns < 256 ? ns + 32 : 256;
        }
        if (!ok) return false;
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

// Bounded wait for row block b's chunks: one poll of its group's counter when the plan has block
// groups ("Triggered Plans", Not supported yet, "Waiting on a group"), else every chunk in turn.
__device__ __forceinline__ bool wait_block(const ConsumerParams& p, uint32_t b, volatile uint32_t* abort) {
    if (!p.bgroup) return wait_chunks(p.h, p.c0[b], p.c1[b], p.max_polls, abort);
    const uint32_t g = p.bgroup[b];
    if (g != 0xFFFFFFFFu) {                  // a block no chunk touches has nothing to wait for
        const dtt_group_table& t = p.h.groups;
        const uint64_t* w = t.counters + (uint64_t)p.h.rank * t.n_groups + g;
        const uint64_t target = (uint64_t)p.h.round * t.size[g];
        uint32_t ns = 0;
        bool ok = false;
        for (uint64_t i = 0; i < p.max_polls; ++i) {
            if (dtt_dev::ld_acquire(w) >= target) { ok = true; break; }
            if ((i & 63) == 63 && *abort) return false;
            __nanosleep(ns);
            ns = ns < 256 ? ns + 32 : 256;
        }
        if (!ok) return false;
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

// Shared memory of the consumer with ST stages: a smaller ring lets it sit beside a bulk-copy
// copier's ring on the same SM.
template <uint32_t TN, uint32_t ST>
constexpr uint32_t consumer_smem() { return 1024 + ST * (A_STAGE + Cfg<TN>::B_STAGE) + 256; }

template <uint32_t TN, uint32_t ST>
__global__ void __launch_bounds__(THREADS, 1) gemm_consumer_kernel(const __grid_constant__ ConsumerParams p) {
    using G = Cfg<TN>;
    constexpr uint32_t STAGES = ST, B_STAGE = G::B_STAGE, TMEM_COLS = G::TMEM_COLS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_STAGE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_STAGE);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* acc_full = bars + 2 * STAGES;
    uint64_t* acc_empty = acc_full + ACC_BUFS;
    uint64_t* drain = acc_empty + ACC_BUFS;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const uint32_t warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (uint32_t i = 0; i < STAGES; ++i) {
            bar_init(saddr(full + i), 1);
            bar_init(saddr(empty + i), 1);
        }
        for (uint32_t i = 0; i < ACC_BUFS; ++i) {
            bar_init(saddr(acc_full + i), 1);
            bar_init(saddr(acc_empty + i), EPI_THREADS);
        }
        bar_init(saddr(drain), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(saddr(tmem_slot)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const uint32_t units_n = p.N / TN, units = p.blocks * units_n, kblocks = p.K / BK;
    auto fail = [&]() {
        *abort_flag = 1;
        atomicAdd(p.err, 1u);
    };

    if (warp == TMA_WARP) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, issued = 0;
            bool ok = true;
            for (uint32_t u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const uint32_t b = p.order[u / units_n];
                if (!wait_block(p, b, abort_flag)) { fail(); break; }
                const int32_t row_x = (int32_t)(b * BM), row_w = (int32_t)((u % units_n) * TN);
                for (uint32_t kb = 0; kb < kblocks; ++kb) {
                    if (!bar_wait(saddr(empty + stage), phase ^ 1, abort_flag)) { fail(); ok = false; break; }
                    bar_expect_tx(saddr(full + stage), A_STAGE + B_STAGE);
                    tma_load_2d(saddr(sA + stage * A_STAGE), &p.tmX, (int32_t)(kb * BK), row_x, saddr(full + stage));
                    tma_load_2d(saddr(sB + stage * B_STAGE), &p.tmW, (int32_t)(kb * BK), row_w, saddr(full + stage));
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            volatile uint32_t never = 0;
            for (uint32_t i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
                (void)bar_wait(saddr(full + i % STAGES), (i / STAGES) & 1, &never);
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (uint32_t u = blockIdx.x; u < units && ok; u += gridDim.x) {
                if (!bar_wait(saddr(acc_empty + acc), acc_phase ^ 1, abort_flag)) { fail(); break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * TN;
                for (uint32_t kb = 0; kb < kblocks; ++kb) {
                    if (!bar_wait(saddr(full + stage), phase, abort_flag)) { fail(); ok = false; break; }
                    tc_fence_after();
                    const uint64_t da = smem_desc(saddr(sA + stage * A_STAGE));
                    const uint64_t db = smem_desc(saddr(sB + stage * B_STAGE));
#pragma unroll
                    for (uint32_t k = 0; k < BK / UMMA_K; ++k)
                        umma(d_tmem, da + 2 * k, db + 2 * k, G::IDESC, (kb | k) != 0);
                    umma_commit(saddr(empty + stage));
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                umma_commit(saddr(acc_full + acc));
                if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1; }
            }
            umma_commit(saddr(drain));
            volatile uint32_t never = 0;
            (void)bar_wait(saddr(drain), 0, &never);
        }
    } else {
        uint32_t acc = 0, acc_phase = 0;
        const uint32_t row_in_tile = warp * 32 + lane;
        for (uint32_t u = blockIdx.x; u < units; u += gridDim.x) {
            bool mine = bar_wait(saddr(acc_full + acc), acc_phase, abort_flag);
            if (!mine) fail();
            if (!epi_all(mine && !*abort_flag)) break;
            tc_fence_after();
            const uint32_t b = p.order[u / units_n];
            char* drow = p.D + (uint64_t)(b * BM + row_in_tile) * p.ldd + (uint64_t)(u % units_n) * TN * 2;
            const uint32_t taddr = tmem_base + ((warp * 32u) << 16) + acc * TN;
#pragma unroll 1
            for (uint32_t g = 0; g < TN / 32; ++g) {
                uint32_t v[32];
                tmem_ld32(taddr + g * 32, v);
                uint4* dst = reinterpret_cast<uint4*>(drow + g * 64);
#pragma unroll
                for (uint32_t j = 0; j < 4; ++j)
                    dst[j] = make_uint4(pack_bf16x2(v[8 * j + 0], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                                        pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
            }
            tc_fence_before();
            bar_arrive(saddr(acc_empty + acc));
            if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1; }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS) : "memory");
}

// ---- the 2-CTA form -------------------------------------------------------------------------
// A cluster of two CTAs on two SMs computes 256 x 256 blocks with tcgen05.mma.cta_group::2
// (M = 256, N = 256): each CTA holds its 128 rows of A and its 128 columns of B^T per stage, so a
// CTA moves 32 KiB per k-block instead of the 48 KiB the one-CTA 128 x 256 form needs, and each
// CTA's TMEM receives its own 128 rows of the block.  One thread of the even CTA (the leader)
// issues every MMA; the leader's mbarriers count both CTAs' loads (as bytes) and both
// epilogues, and the MMA's completions are multicast to both CTAs.
constexpr uint32_t G2_TN = 256;                       // block columns (B^T rows) per MMA
constexpr uint32_t G2_BHALF = BN * BK * 2;            // 16 KiB: this CTA's 128 rows of B^T
constexpr uint32_t G2_STAGES = 6;
constexpr uint32_t G2_TMEM_COLS = ACC_BUFS * G2_TN;   // 512 fp32 columns
constexpr uint32_t G2_SMEM = 1024 + G2_STAGES * (A_STAGE + G2_BHALF) + 256;
constexpr uint32_t G2_IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((G2_TN >> 3) << 17) | ((256u >> 4) << 24);

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t at_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void bar_arrive_at(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// A tile load into this CTA's shared memory that completes on the leader's mbarrier.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 uint32_t cluster_bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2 "
        "[%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cluster_bar) : "memory");
}

__device__ __forceinline__ void umma_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrive once on the mbarrier at this offset in both CTAs when the MMAs issued so far finish.
__device__ __forceinline__ void umma_commit_both(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(bar), "h"((uint16_t)0x3) : "memory");
}

__device__ __forceinline__ void umma_commit_local2(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar) : "memory");
}

// A unit is a 256 x 256 block; every rank's units form one sequence, the ranks taking turns as
// in the one-CTA form, and cluster c of NC takes its places c, c + NC, ...; CTA q of the pair
// owns the unit's rows 128 q .. 128 q + 127.  Tile (tm, tn) is step
// tm * tiles_n + tn of its rank and, once stored, gets one mark on chunk first_chunk + step / NP.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
gemm2_producer_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + G2_STAGES * A_STAGE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + G2_STAGES * G2_BHALF);
    uint64_t* full = bars;                        // [STAGES]  leader: both CTAs' loads -> MMA
    uint64_t* empty = bars + G2_STAGES;           // [STAGES]  each CTA: MMA -> its TMA warp
    uint64_t* acc_full = bars + 2 * G2_STAGES;    // [2]       each CTA: MMA -> its epilogue
    uint64_t* acc_empty = acc_full + ACC_BUFS;    // [2]       leader: both epilogues -> MMA
    uint64_t* drain = acc_empty + ACC_BUFS;       // [1]       leader: MMA teardown
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const uint32_t warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t q = cluster_rank();
    const bool leader = q == 0;
    if (threadIdx.x == 0) {
        for (uint32_t i = 0; i < G2_STAGES; ++i) {
            bar_init(saddr(full + i), 1);            // the leader's expect_tx covers both CTAs' bytes
            bar_init(saddr(empty + i), 1);
        }
        for (uint32_t i = 0; i < ACC_BUFS; ++i) {
            bar_init(saddr(acc_full + i), 1);
            bar_init(saddr(acc_empty + i), 2);       // one arrival per CTA's epilogue
        }
        bar_init(saddr(drain), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(saddr(tmem_slot)), "r"(G2_TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync_all();          // both CTAs' barriers exist before either arrives remotely
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const uint32_t tiles_n = p.N / BN, units_n = p.N / G2_TN, units = (p.M / 256) * units_n;
    const uint32_t kblocks = p.K / BK;
    const uint32_t c0 = blockIdx.x / 2, NC = gridDim.x / 2;
    const uint32_t peer_abort = at_rank(saddr(tmem_slot + 1), q ^ 1);
    auto fail = [&]() {
        *abort_flag = 1;
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort), "r"(1u) : "memory");
        atomicAdd(p.err, 1u);
    };

    if (warp == TMA_WARP) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, issued = 0;
            bool ok = true;
            for (uint32_t gu = c0; gu < p.P * units && ok; gu += NC) {
                    const uint32_t r = gu % p.P, u = gu / p.P;
                    const int32_t row_a = (int32_t)(r * p.M + (u / units_n) * 256 + q * BM);
                    const int32_t row_b = (int32_t)((u % units_n) * G2_TN + q * BN);
                    for (uint32_t kb = 0; kb < kblocks; ++kb) {
                        if (!bar_wait(saddr(empty + stage), phase ^ 1, abort_flag)) { fail(); ok = false; break; }
                        // The peer's loads may land before the leader's expect_tx (the barrier's
                        // transaction count goes below zero for a while), but never a phase
                        // early: its stage is free only once the MMA has consumed that stage.
                        const uint32_t fb = at_rank(saddr(full + stage), 0);
                        if (leader) bar_expect_tx(saddr(full + stage), 2 * (A_STAGE + G2_BHALF));
                        tma_load_2d_pair(saddr(sA + stage * A_STAGE), &p.tmA, (int32_t)(kb * BK), row_a, fb);
                        tma_load_2d_pair(saddr(sB + stage * G2_BHALF), &p.tmB, (int32_t)(kb * BK), row_b, fb);
                        ++issued;
                        if (++stage == G2_STAGES) { stage = 0; phase ^= 1; }
                    }
                }
            // the leader's full barriers count both CTAs' loads: once its last phases complete,
            // every load of the pair has landed
            if (leader) {
                volatile uint32_t never = 0;
                for (uint32_t i = issued > G2_STAGES ? issued - G2_STAGES : 0; i < issued; ++i)
                    (void)bar_wait(saddr(full + i % G2_STAGES), (i / G2_STAGES) & 1, &never);
            }
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0 && leader) {
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (uint32_t gu = c0; gu < p.P * units && ok; gu += NC) {
                    if (!bar_wait(saddr(acc_empty + acc), acc_phase ^ 1, abort_flag)) { fail(); ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + acc * G2_TN;
                    for (uint32_t kb = 0; kb < kblocks; ++kb) {
                        if (!bar_wait(saddr(full + stage), phase, abort_flag)) { fail(); ok = false; break; }
                        tc_fence_after();
                        const uint64_t da = smem_desc(saddr(sA + stage * A_STAGE));
                        const uint64_t db = smem_desc(saddr(sB + stage * G2_BHALF));
#pragma unroll
                        for (uint32_t k = 0; k < BK / UMMA_K; ++k)
                            umma_pair(d_tmem, da + 2 * k, db + 2 * k, G2_IDESC, (kb | k) != 0);
                        umma_commit_both(saddr(empty + stage));   // both CTAs' stages are free
                        if (++stage == G2_STAGES) { stage = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                    umma_commit_both(saddr(acc_full + acc));      // the block is in both TMEMs
                    if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1; }
                }
            // every MMA has finished before either CTA releases TMEM or shared memory
            umma_commit_local2(saddr(drain));
            volatile uint32_t never = 0;
            (void)bar_wait(saddr(drain), 0, &never);
        }
    } else {
        // epilogue warps 0..3: thread t of warp w owns row 32w + t of this CTA's 128 rows
        uint32_t acc = 0, acc_phase = 0;
        const uint32_t row_in_tile = warp * 32 + lane;
        bool ok = true;
        for (uint32_t gu = c0; gu < p.P * units && ok; gu += NC) {
                const uint32_t r = gu % p.P, u = gu / p.P;
                const uint32_t tm = (u / units_n) * 2 + q, tn0 = (u % units_n) * (G2_TN / BN);
                bool mine = bar_wait(saddr(acc_full + acc), acc_phase, abort_flag);
                if (!mine) fail();
                if (threadIdx.x == 0 && mine && !unit_writable(p.h[r], tm * tiles_n + tn0, G2_TN / BN, p.NP)) {
                    fail();
                    mine = false;
                }
                if (!epi_all(mine && !*abort_flag)) { ok = false; break; }
                tc_fence_after();
                char* crow = p.bufs[r] + p.slice_off[r] + (uint64_t)(tm * BM + row_in_tile) * p.ldc +
                             (uint64_t)tn0 * BN * 2;
                const uint32_t taddr = tmem_base + ((warp * 32u) << 16) + acc * G2_TN;
#pragma unroll 1
                for (uint32_t g = 0; g < G2_TN / 32; ++g) {
                    uint32_t v[32];
                    tmem_ld32(taddr + g * 32, v);
                    uint4* dst = reinterpret_cast<uint4*>(crow + g * 64);
#pragma unroll
                    for (uint32_t j = 0; j < 4; ++j)
                        dst[j] = make_uint4(pack_bf16x2(v[8 * j + 0], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                                            pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
                }
                tc_fence_before();
                // every TMEM read and store of this CTA's rows precedes one arrival at the leader
                // (the accumulator may be overwritten) and one mark per tile
                asm volatile("bar.sync 1, %0;" ::"n"(EPI_THREADS) : "memory");
                if (threadIdx.x == 0) {
                    bar_arrive_at(at_rank(saddr(acc_empty + acc), 0));
                    for (uint32_t k = 0; k < G2_TN / BN; ++k)
                        dtt_dev::mark_one(p.h[r], p.h[r].first_chunk + (tm * tiles_n + tn0 + k) / p.NP);
                }
                if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1; }
            }
    }
    tc_fence_before();
    cluster_sync_all();          // no CTA leaves while the pair's MMAs or loads may touch it
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(G2_TMEM_COLS)
                     : "memory");
}

// ---- the consumer in the 2-CTA form ----------------------------------------------------------
// D = X . W^T by CTA pairs.  A unit is a 256 x 256 block of D over the pair of 128-row blocks
// (2 pb, 2 pb + 1) of X; CTA q of the pair waits for the chunks of its own row block 2 pb + q
// before it loads it, so each half enters the MMA as soon as it has arrived.  Pair blocks are
// taken in the order their later half opens (order2); cluster c of NC takes units c, c + NC, ...
template <uint32_t ST>
constexpr uint32_t g2c_smem() { return 1024 + ST * (A_STAGE + G2_BHALF) + 256; }

template <uint32_t ST>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
gemm2_consumer_kernel(const __grid_constant__ ConsumerParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + ST * A_STAGE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + ST * G2_BHALF);
    uint64_t* full = bars;                        // [ST]  leader: both CTAs' loads -> MMA
    uint64_t* empty = bars + ST;                  // [ST]  each CTA: MMA -> its TMA warp
    uint64_t* acc_full = bars + 2 * ST;           // [2]   each CTA: MMA -> its epilogue
    uint64_t* acc_empty = acc_full + ACC_BUFS;    // [2]   leader: both epilogues -> MMA
    uint64_t* drain = acc_empty + ACC_BUFS;       // [1]   leader: MMA teardown
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const uint32_t warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t q = cluster_rank();
    const bool leader = q == 0;
    if (threadIdx.x == 0) {
        for (uint32_t i = 0; i < ST; ++i) {
            bar_init(saddr(full + i), 1);
            bar_init(saddr(empty + i), 1);
        }
        for (uint32_t i = 0; i < ACC_BUFS; ++i) {
            bar_init(saddr(acc_full + i), 1);
            bar_init(saddr(acc_empty + i), 2);
        }
        bar_init(saddr(drain), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(saddr(tmem_slot)), "r"(G2_TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const uint32_t units_n = p.N / G2_TN, units = (p.blocks / 2) * units_n, kblocks = p.K / BK;
    const uint32_t c0 = blockIdx.x / 2, NC = gridDim.x / 2;
    const uint32_t peer_abort = at_rank(saddr(tmem_slot + 1), q ^ 1);
    auto fail = [&]() {
        *abort_flag = 1;
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort), "r"(1u) : "memory");
        atomicAdd(p.err, 1u);
    };

    if (warp == TMA_WARP) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, issued = 0;
            bool ok = true;
            for (uint32_t u = c0; u < units && ok; u += NC) {
                const uint32_t b = 2 * p.order2[u / units_n] + q;
                if (!wait_block(p, b, abort_flag)) { fail(); break; }
                const int32_t row_a = (int32_t)(b * BM);
                const int32_t row_b = (int32_t)((u % units_n) * G2_TN + q * BN);
                for (uint32_t kb = 0; kb < kblocks; ++kb) {
                    if (!bar_wait(saddr(empty + stage), phase ^ 1, abort_flag)) { fail(); ok = false; break; }
                    const uint32_t fb = at_rank(saddr(full + stage), 0);
                    if (leader) bar_expect_tx(saddr(full + stage), 2 * (A_STAGE + G2_BHALF));
                    tma_load_2d_pair(saddr(sA + stage * A_STAGE), &p.tmX, (int32_t)(kb * BK), row_a, fb);
                    tma_load_2d_pair(saddr(sB + stage * G2_BHALF), &p.tmW, (int32_t)(kb * BK), row_b, fb);
                    ++issued;
                    if (++stage == ST) { stage = 0; phase ^= 1; }
                }
            }
            if (leader) {
                volatile uint32_t never = 0;
                for (uint32_t i = issued > ST ? issued - ST : 0; i < issued; ++i)
                    (void)bar_wait(saddr(full + i % ST), (i / ST) & 1, &never);
            }
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0 && leader) {
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (uint32_t u = c0; u < units && ok; u += NC) {
                if (!bar_wait(saddr(acc_empty + acc), acc_phase ^ 1, abort_flag)) { fail(); break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * G2_TN;
                for (uint32_t kb = 0; kb < kblocks; ++kb) {
                    if (!bar_wait(saddr(full + stage), phase, abort_flag)) { fail(); ok = false; break; }
                    tc_fence_after();
                    const uint64_t da = smem_desc(saddr(sA + stage * A_STAGE));
                    const uint64_t db = smem_desc(saddr(sB + stage * G2_BHALF));
#pragma unroll
                    for (uint32_t k = 0; k < BK / UMMA_K; ++k)
                        umma_pair(d_tmem, da + 2 * k, db + 2 * k, G2_IDESC, (kb | k) != 0);
                    umma_commit_both(saddr(empty + stage));
                    if (++stage == ST) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                umma_commit_both(saddr(acc_full + acc));
                if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1; }
            }
            umma_commit_local2(saddr(drain));
            volatile uint32_t never = 0;
            (void)bar_wait(saddr(drain), 0, &never);
        }
    } else {
        uint32_t acc = 0, acc_phase = 0;
        const uint32_t row_in_tile = warp * 32 + lane;
        for (uint32_t u = c0; u < units; u += NC) {
            bool mine = bar_wait(saddr(acc_full + acc), acc_phase, abort_flag);
            if (!mine) fail();
            if (!epi_all(mine && !*abort_flag)) break;
            tc_fence_after();
            const uint32_t b = 2 * p.order2[u / units_n] + q;
            char* drow = p.D + (uint64_t)(b * BM + row_in_tile) * p.ldd + (uint64_t)(u % units_n) * G2_TN * 2;
            const uint32_t taddr = tmem_base + ((warp * 32u) << 16) + acc * G2_TN;
#pragma unroll 1
            for (uint32_t g = 0; g < G2_TN / 32; ++g) {
                uint32_t v[32];
                tmem_ld32(taddr + g * 32, v);
                uint4* dst = reinterpret_cast<uint4*>(drow + g * 64);
#pragma unroll
                for (uint32_t j = 0; j < 4; ++j)
                    dst[j] = make_uint4(pack_bf16x2(v[8 * j + 0], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                                        pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
            }
            tc_fence_before();
            // every TMEM read of this CTA's rows precedes one arrival at the leader
            asm volatile("bar.sync 1, %0;" ::"n"(EPI_THREADS) : "memory");
            if (threadIdx.x == 0) bar_arrive_at(at_rank(saddr(acc_empty + acc), 0));
            if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1; }
        }
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(G2_TMEM_COLS)
                     : "memory");
}

// A 2D bf16 K-major operand: rows x K elements, box 64 (K) x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t K, uint32_t box_rows) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K * 2};
    const cuuint32_t box[2] = {BK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The operands' tensor maps depend only on their addresses and shapes, so the last few are kept
// and a repeated launch (every round of a plan) skips the encoding on the host.
struct MapCacheEntry {
    const void* A;
    const void* Bt;
    uint64_t rows_a, N, K;
    uint32_t TN;
    CUtensorMap tmA, tmB;
};
std::mutex g_map_mu;
MapCacheEntry g_map_cache[8];
uint32_t g_map_used = 0, g_map_next = 0;

bool operand_maps(const void* A, const void* Bt, uint64_t rows_a, uint64_t N, uint64_t K, uint32_t TN,
                  CUtensorMap* tmA, CUtensorMap* tmB) {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (uint32_t i = 0; i < g_map_used; ++i) {
        const MapCacheEntry& e = g_map_cache[i];
        if (e.A == A && e.Bt == Bt && e.rows_a == rows_a && e.N == N && e.K == K && e.TN == TN) {
            *tmA = e.tmA;
            *tmB = e.tmB;
            return true;
        }
    }
    MapCacheEntry e{A, Bt, rows_a, N, K, TN, {}, {}};
    if (!make_map(&e.tmA, A, rows_a, K, BM) || !make_map(&e.tmB, Bt, N, K, TN)) return false;
    g_map_cache[g_map_next] = e;
    g_map_next = (g_map_next + 1) % 8;
    if (g_map_used < 8) ++g_map_used;
    *tmA = e.tmA;
    *tmB = e.tmB;
    return true;
}

// How many clusters of a CTA-pair kernel can be resident at once: a property of the kernel,
// its shared memory and the device.  The query costs the host microseconds, so it is asked
// once per (device, kernel) and reused by every later launch.
struct FitEntry {
    int dev;
    const void* kernel;
    int fit;
};
std::mutex g_fit_mu;
FitEntry g_fit[16];
uint32_t g_fit_used = 0;

template <class Kern>
int cluster_fit(Kern kernel, uint32_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const void* key = reinterpret_cast<const void*>(kernel);
    {
        std::lock_guard<std::mutex> lock(g_fit_mu);
        for (uint32_t i = 0; i < g_fit_used; ++i)
            if (g_fit[i].dev == dev && g_fit[i].kernel == key) return g_fit[i].fit;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    int fit = 0;
    if (cudaOccupancyMaxActiveClusters(&fit, kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(g_fit_mu);
    if (g_fit_used < 16) g_fit[g_fit_used++] = FitEntry{dev, key, fit};
    return fit;
}

}  // namespace

template <uint32_t TN>
static cudaError_t prepare_gemm() {
    cudaError_t e = prepare_kernel(gemm_producer_kernel<TN>);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_producer_kernel<TN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)Cfg<TN>::SMEM_BYTES);
    return e;
}

template <uint32_t TN, uint32_t ST>
static cudaError_t prepare_consumer() {
    cudaError_t e = prepare_kernel(gemm_consumer_kernel<TN, ST>);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_consumer_kernel<TN, ST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)consumer_smem<TN, ST>());
    return e;
}

template <uint32_t ST>
static cudaError_t prepare_consumer_pair() {
    cudaError_t e = prepare_kernel(gemm2_consumer_kernel<ST>);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm2_consumer_kernel<ST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)g2c_smem<ST>());
    return e;
}

// The deepest ring (at most the producer form's) whose shared memory fits in `budget` bytes;
// the full ring when none of the smaller ones fits either (the GEMM then waits for room).
template <uint32_t TN, uint32_t ST>
static void launch_consumer_ring(const ConsumerParams& cp, uint32_t ctas, uint64_t budget, cudaStream_t s) {
    if constexpr (ST > 2) {
        if (consumer_smem<TN, ST>() > budget) {
            launch_consumer_ring<TN, ST - 1>(cp, ctas, budget, s);
            return;
        }
    }
    if (consumer_smem<TN, ST>() > budget) {
        gemm_consumer_kernel<TN, Cfg<TN>::STAGES><<<ctas, THREADS, consumer_smem<TN, Cfg<TN>::STAGES>(), s>>>(cp);
        return;
    }
    gemm_consumer_kernel<TN, ST><<<ctas, THREADS, consumer_smem<TN, ST>(), s>>>(cp);
}

// The pair form with the deepest ring (at most 6 stages, at least 3) that fits in `budget`, as
// many clusters as can be resident at once; false when no such launch exists.
template <uint32_t ST>
static bool launch_consumer_pair(const ConsumerParams& cp, uint32_t ctas, uint64_t budget, cudaStream_t s) {
    if constexpr (ST > 3) {
        if (g2c_smem<ST>() > budget) return launch_consumer_pair<ST - 1>(cp, ctas, budget, s);
    }
    if (g2c_smem<ST>() > budget) return false;
    const int fit = cluster_fit(gemm2_consumer_kernel<ST>, g2c_smem<ST>());
    if (fit < 1) return false;
    const uint32_t pairs = std::min<uint32_t>(ctas / 2, (uint32_t)fit);
    gemm2_consumer_kernel<ST><<<2 * pairs, THREADS, g2c_smem<ST>(), s>>>(cp);
    return true;
}

int launch_gemm_consumer(const ConsumerLaunch& cl, cudaStream_t stream) {
    ConsumerParams cp{};
    cp.h = cl.h;
    cp.order = cl.order;
    cp.c0 = cl.c0;
    cp.c1 = cl.c1;
    cp.order2 = cl.order2;
    cp.bgroup = cl.bgroup;
    cp.D = cl.D;
    cp.ldd = cl.ldd;
    cp.max_polls = cl.max_polls;
    cp.blocks = cl.blocks;
    cp.N = cl.N;
    cp.K = cl.K;
    cp.err = cl.err;
    // CTA pairs (M = 256, N = 256 per MMA) when the blocks pair up and the columns tile by 256
    if (cl.order2 && cl.N % 256 == 0 && cl.blocks % 2 == 0 && cl.ctas >= 2) {
        if (!operand_maps(cl.X, cl.Wt, cl.rows, cl.N, cl.K, BN, &cp.tmX, &cp.tmW))
            return fail(DTT_ECUDA, "dtt_gemm_consumer: cannot encode the tensor maps");
        if (launch_consumer_pair<6>(cp, cl.ctas, cl.smem_budget, stream)) {
            const cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return fail(DTT_ECUDA, "dtt_gemm_consumer: launch failed: %s", cudaGetErrorString(e));
            return DTT_OK;
        }
    }
    const uint32_t TN = (cl.N % 256 == 0) ? 256 : 128;
    if (!operand_maps(cl.X, cl.Wt, cl.rows, cl.N, cl.K, TN, &cp.tmX, &cp.tmW))
        return fail(DTT_ECUDA, "dtt_gemm_consumer: cannot encode the tensor maps");
    if (TN == 256)
        launch_consumer_ring<256, Cfg<256>::STAGES>(cp, cl.ctas, cl.smem_budget, stream);
    else
        launch_consumer_ring<128, Cfg<128>::STAGES>(cp, cl.ctas, cl.smem_budget, stream);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(DTT_ECUDA, "dtt_gemm_consumer: launch failed: %s", cudaGetErrorString(e));
    return DTT_OK;
}

cudaError_t preload_gemm_kernels() {
    cudaError_t e = prepare_gemm<128>();
    if (e == cudaSuccess) e = prepare_gemm<256>();
    if (e == cudaSuccess) e = prepare_consumer<128, 6>();
    if (e == cudaSuccess) e = prepare_consumer<128, 5>();
    if (e == cudaSuccess) e = prepare_consumer<128, 4>();
    if (e == cudaSuccess) e = prepare_consumer<128, 3>();
    if (e == cudaSuccess) e = prepare_consumer<128, 2>();
    if (e == cudaSuccess) e = prepare_consumer<256, 4>();
    if (e == cudaSuccess) e = prepare_consumer<256, 3>();
    if (e == cudaSuccess) e = prepare_consumer<256, 2>();
    if (e == cudaSuccess) e = prepare_kernel(gemm2_producer_kernel);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm2_producer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G2_SMEM);
    if (e == cudaSuccess) e = prepare_consumer_pair<6>();
    if (e == cudaSuccess) e = prepare_consumer_pair<5>();
    if (e == cudaSuccess) e = prepare_consumer_pair<4>();
    if (e == cudaSuccess) e = prepare_consumer_pair<3>();
    return e;
}

}  // namespace dtt

using namespace dtt;

extern "C" int dtt_gemm_producer(const void* A, const void* Bt, void* const* bufs, uint32_t P, uint32_t M,
                                 uint32_t N, uint32_t K, uint64_t ldc, const uint64_t* slice_off,
                                 uint32_t num_programs, const dtt_handle* handles, uint32_t* err,
                                 cudaStream_t stream) {
    if (!A || !Bt || !bufs || !slice_off || !handles || !err || P < 1 || P > DTT_MAX_RANKS)
        return fail(DTT_EINVAL, "dtt_gemm_producer: bad args");
    if (M == 0 || N == 0 || K == 0 || M % BM || N % BN || K % BK)
        return fail(DTT_EINVAL, "dtt_gemm_producer: M and N must be multiples of 128 and K of 64");
    if (num_programs == 0 || ldc < (uint64_t)N * 2 || ldc % 16)
        return fail(DTT_EINVAL, "dtt_gemm_producer: bad num_programs or ldc");
    if (reinterpret_cast<uintptr_t>(A) % 16 || reinterpret_cast<uintptr_t>(Bt) % 16)
        return fail(DTT_EINVAL, "dtt_gemm_producer: operands must be 16-byte aligned");
    const uint32_t TN = (N % 256 == 0) ? 256 : 128;   // widest MMA block that tiles N
    // the 2-CTA form when the blocks tile both M and N and the launch can hold a CTA pair
    const bool pair = M % 256 == 0 && N % 256 == 0 && num_programs >= 2;
    GemmParams gp{};
    if (!operand_maps(A, Bt, (uint64_t)P * M, N, K, pair ? BN : TN, &gp.tmA, &gp.tmB))
        return fail(DTT_ECUDA, "dtt_gemm_producer: cannot encode the tensor maps");
    // the producer marks first_chunk + (row-major tile index) / num_programs: every rank's part of
    // the plan must have exactly that many chunks (tile_chunks with tiles_per_chunk = num_programs)
    const uint64_t tiles = (uint64_t)(M / BM) * (N / BN);
    const uint64_t want_chunks = (tiles + num_programs - 1) / num_programs;
    for (uint32_t r = 0; r < P; ++r)
        if (handles[r].n_chunks != want_chunks || handles[r].P != P || handles[r].rank != r)
            return fail(DTT_EINVAL, "dtt_gemm_producer: rank %u's handle has %u chunks; a %u x %u output in "
                                    "128 x 128 tiles over %u programs needs %llu (tile_chunks with "
                                    "tiles_per_chunk = num_programs)", r, handles[r].n_chunks, M, N,
                        num_programs, (unsigned long long)want_chunks);
    for (uint32_t r = 0; r < P; ++r) {
        if (!bufs[r] || (reinterpret_cast<uintptr_t>(bufs[r]) + slice_off[r]) % 16)
            return fail(DTT_EINVAL, "dtt_gemm_producer: rank %u's output is not 16-byte aligned", r);
        gp.bufs[r] = static_cast<char*>(bufs[r]);
        gp.h[r] = handles[r];
        gp.slice_off[r] = slice_off[r];
    }
    gp.ldc = ldc;
    gp.P = P;
    gp.M = M;
    gp.N = N;
    gp.K = K;
    gp.NP = num_programs;
    gp.err = err;
    if (pair) {
        // a persistent grid: no more CTA pairs than can be resident at once
        const int fit = cluster_fit(gemm2_producer_kernel, G2_SMEM);
        if (fit < 1) return fail(DTT_ECUDA, "dtt_gemm_producer: no CTA pair fits on this device");
        const uint32_t pairs = std::min<uint32_t>(num_programs / 2, (uint32_t)fit);
        gemm2_producer_kernel<<<2 * pairs, THREADS, G2_SMEM, stream>>>(gp);
    } else if (TN == 256)
        gemm_producer_kernel<256><<<num_programs, THREADS, Cfg<256>::SMEM_BYTES, stream>>>(gp);
    else
        gemm_producer_kernel<128><<<num_programs, THREADS, Cfg<128>::SMEM_BYTES, stream>>>(gp);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(DTT_ECUDA, "dtt_gemm_producer: launch failed: %s", cudaGetErrorString(e));
    return DTT_OK;
}
