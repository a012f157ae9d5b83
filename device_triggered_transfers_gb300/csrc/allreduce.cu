// The two-shot all-reduce ("Triggered Plans", Not supported yet: reduce-scatter and two-shot
// all-reduce are what other destinations make possible): a reduce-scatter plan whose chunks land
// in staging slots of the block's owner, one kernel that waits for each sub-block's group, adds
// the P parts in f32 in rank order and marks the sum for an in-place all-gather plan.
//
// One launch covers every virtual rank; it walks the sub-blocks (b, j) b-major, the order a
// producer writing its vector row by row completes them.  In each CTA one control thread does
// all the GPU-scope synchronisation -- it polls the sub-blocks' groups ahead of the work, and
// counts the CTA's finished sub-blocks into global counters whose last CTA marks the all-gather
// chunk -- and hands both ends to the compute warps through shared memory.  The compute warps
// only load, add and store, striding over each sub-block as one grid so that at any moment the
// whole GPU reads neighbouring vectors of each part.
#include <cstdint>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include <cuda_bf16.h>

#include "dtt_device.cuh"
#include "internal.h"

namespace dtt {
namespace {

struct ReduceParams {
    char* bufs[DTT_MAX_RANKS];          // rank r's vector, from byte 0
    const char* stage[DTT_MAX_RANKS];   // rank r's staging area (its buffer, or its staging buffer)
    dtt_handle rs[DTT_MAX_RANKS];       // reduce-scatter plan, per rank
    dtt_handle ag[DTT_MAX_RANKS];       // all-gather plan, per rank
    uint64_t pitch;        // bytes between rows
    uint64_t slot_off;     // slot 0 in each staging area
    uint64_t slot_bytes;   // from one slot to the next: block_rows * pitch
    uint64_t Mb, Mj;       // block rows, sub-block rows
    uint64_t max_polls;    // of one group wait
    uint32_t J;            // sub-blocks per block
    uint32_t vrow;         // 16-byte vectors per row
    uint32_t contig;       // rows back to back (pitch == vrow * 16): a sub-block is one range
    uint32_t gather;       // 1: mark each summed sub-block for the all-gather plan (all-reduce)
    uint32_t* counters;    // [P * J]: CTAs done with (b, j) this launch; zero between launches
    uint32_t* err;         // waits that ran out
};

// f32 lanes of a 16-byte vector, and the conversions (bf16 -> f32 is exact; f32 -> bf16 rounds
// to nearest even).
template <int DT> struct Lanes;
template <> struct Lanes<DTT_BF16> {
    static constexpr int n = 8;
    static __device__ __forceinline__ void unpack(const uint4& v, float* f) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    static __device__ __forceinline__ uint4 pack(const float* f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct Lanes<DTT_F32> {
    static constexpr int n = 4;
    static __device__ __forceinline__ void unpack(const uint4& v, float* f) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    static __device__ __forceinline__ uint4 pack(const float* f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};

__device__ __forceinline__ void st16(char* p, const uint4& v) { *reinterpret_cast<uint4*>(p) = v; }

// Threads per reduce CTA at most: a control warp (lane 0 publishes, lane 1 completes) and up
// to 15 compute warps of ~60 registers.
constexpr uint32_t kReduceMaxThreads = 512;

__device__ __forceinline__ uint32_t sm_addr(const void* q) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(q));
}
__device__ __forceinline__ uint32_t ld_acquire_cta(const uint32_t* q) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(sm_addr(q)) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_cta(uint32_t* q, uint32_t v) {
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(sm_addr(q)), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release_cta(uint32_t* q, uint32_t v) {
    asm volatile("red.release.cta.shared::cta.add.u32 [%0], %1;" ::"r"(sm_addr(q)), "r"(v) : "memory");
}
// 16 bytes through L2 only: every part is read once, and no line read before the control
// thread's acquire can be served from L1.
__device__ __forceinline__ uint4 ld_cg(const char* q) {
    return __ldcg(reinterpret_cast<const uint4*>(q));
}

// One compute warp's share of sub-block (b, j): vectors first_t, first_t + stride, ... of it, U
// at a time, the P parts of each loaded together and added in rank order -- part b is the
// owner's rows (own), part s != b slot s (slot0 + s * slot_bytes).  CONTIG: rows back to back,
// so vector t of a part is its t-th 16 bytes (a separate instance: with padded rows the offset
// needs a division).
template <int DT, int P, bool CONTIG>
__device__ __forceinline__ void add_sub_block(const ReduceParams& p, uint32_t b, char* own, const char* slot0,
                                              uint64_t first_t, uint64_t stride, uint64_t per_unit) {
    using E = Lanes<DT>;
    auto part = [&](int s) -> const char* { return (uint32_t)s == b ? own : slot0 + (uint64_t)s * p.slot_bytes; };
    constexpr int U = P <= 2 ? 4 : (P <= 4 ? 2 : 1); // vectors a lane takes at once
    for (uint64_t t0 = first_t; t0 < per_unit; t0 += stride * U) {
        uint64_t off[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint64_t t = t0 + (uint64_t)k * stride;
            off[k] = CONTIG ? t : (t / p.vrow) * (p.pitch / 16) + t % p.vrow;   // in 16-byte vectors
        }
        if constexpr (P <= 8) {
            // every part of the U vectors in flight at once, then each vector added and stored
            // in turn (one accumulator live)
            const char* src[P];
#pragma unroll
            for (int s = 0; s < P; ++s) src[s] = part(s);
            uint4 v[U][P];
#pragma unroll
            for (int k = 0; k < U; ++k)
                if (t0 + (uint64_t)k * stride < per_unit) {
#pragma unroll
                    for (int s = 0; s < P; ++s) v[k][s] = ld_cg(src[s] + off[k] * 16);
                }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                if (t0 + (uint64_t)k * stride >= per_unit) continue;
                float acc[E::n];
#pragma unroll
                for (int s = 0; s < P; ++s) {
                    float f[E::n];
                    E::unpack(v[k][s], f);
#pragma unroll
                    for (int e = 0; e < E::n; ++e) acc[e] = s == 0 ? f[e] : acc[e] + f[e];
                }
                st16(own + off[k] * 16, E::pack(acc));
            }
        } else {
            // P > 8 (one vector at a time): the parts in batches of 8 into one accumulator
            static_assert(U == 1, "one vector a lane above 4 parts");
            float acc[E::n];
#pragma unroll
            for (int s0 = 0; s0 < P; s0 += 8) {
                uint4 v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (s0 + i < P) v[i] = ld_cg(part(s0 + i) + off[0] * 16);   // addresses made here:
                                                                                 // 16 pointers would not
                                                                                 // fit the registers
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (s0 + i >= P) continue;
                    float f[E::n];
                    E::unpack(v[i], f);
#pragma unroll
                    for (int e = 0; e < E::n; ++e) acc[e] = s0 + i == 0 ? f[e] : acc[e] + f[e];
                }
            }
            st16(own + off[0] * 16, E::pack(acc));
        }
    }
}

// Shared memory of a CTA: the sub-blocks published to the compute warps, the abort flag, and
// per sub-block the CTA's compute warps done with it.
enum { kReady = 0, kAbort = 1, kDone = 2 };

// At most 64 registers a thread, so that four 256-thread CTAs fit an SM (the kernel is bound by
// the loads each SM keeps in flight; the compiler alone takes ~85 registers and halves that).
template <int DT, int P, bool CONTIG>
__global__ void __maxnreg__(64) reduce_kernel(const __grid_constant__ ReduceParams p) {
    extern __shared__ __align__(16) uint32_t ctl[];   // [kDone + P * J]
    const uint32_t units = (uint32_t)P * p.J;
    for (uint32_t i = threadIdx.x; i < kDone + units; i += blockDim.x) ctl[i] = 0;
    __syncthreads();
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const uint32_t NCW = (blockDim.x >> 5) - 1;       // compute warps

    if (warp == 0) {
        if (lane == 0) {
            // The publisher.  It reads the counters of up to 8 groups ahead (relaxed, all in
            // flight together) and publishes the ready prefix behind one fence: a relaxed read
            // followed by fence.acq_rel is an acquire, and the release at CTA scope that
            // publishes (ready = n) hands it on to the compute warps, so their loads of a
            // published sub-block follow every copy of it.
            uint32_t nw = 0;
            uint64_t idle = 0;
            uint32_t ns = 0;
            bool bad = false;
            while (nw < units) {
                const uint32_t n = units - nw < 8 ? units - nw : 8;
                uint64_t have[8], want[8];
#pragma unroll
                for (uint32_t i = 0; i < 8; ++i) {
                    if (i >= n) break;
                    const uint32_t g = nw + i;
                    const uint64_t* w = dtt_dev::group_word(p.rs[g / p.J], g, &want[i]);
                    if (!w) { bad = true; break; }
                    have[i] = dtt_dev::ld_relaxed(w);
                }
                if (bad) break;                        // a plan without the group (misuse bit set)
                uint32_t r = 0;
                while (r < n && have[r] >= want[r]) ++r;
                if (r) {
                    dtt_dev::fence_acq_rel();
                    nw += r;
                    st_release_cta(ctl + kReady, nw);
                    idle = 0;
                    ns = 0;
                    continue;
                }
                if (++idle > p.max_polls) break;      // nothing arrived for max_polls polls
                __nanosleep(ns);
                ns = ns < 256 ? ns + 32 : 256;
            }
            if (nw < units) {
                // gave up: the sub-blocks from nw on are never added, so they stay unmarked and
                // the all-gather plan's wait reports them short
                atomicAdd(p.err, 1u);
                st_release_cta(ctl + kAbort, 1);
            }
        } else if (lane == 1) {
            // The completer.  Its acquire of the CTA's count of a sub-block (CTA scope) lets its
            // acq_rel add on the global counter release all of the CTA's stores of it; the CTA
            // whose add completes the count has every CTA's stores, resets the counter for the
            // next launch (stream-ordered after this one) and marks the all-gather chunk.
            uint32_t nd = 0, ns = 0;
            for (uint64_t i = 0; nd < units; ++i) {
                if (ld_acquire_cta(ctl + kDone + nd) == NCW) {
                    uint32_t old;
                    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(p.counters + nd) : "memory");
                    if (old + 1 == gridDim.x) {
                        asm volatile("st.relaxed.gpu.global.u32 [%0], 0;" ::"l"(p.counters + nd) : "memory");
                        const uint32_t b = nd / p.J, j = nd - b * p.J;
                        if (p.gather) dtt_dev::mark_one(p.ag[b], p.ag[b].first_chunk + j);
                    }
                    ++nd;
                    i = 0;
                    ns = 0;
                    continue;
                }
                // the compute warps stop only after an abort; the bound is a backstop.  The
                // back-off grows to ~1 us: a sub-block takes a few microseconds to add, and a
                // faster spin only takes issue slots from the compute warps of its SM
                // sub-partition (every CTA's control warp may share one)
                if (ld_acquire_cta(ctl + kAbort) || i > 4 * p.max_polls + (1u << 20)) break;
                __nanosleep(ns);
                ns = ns < 1024 ? ns + 64 : 1024;
            }
        }
        return;
    }

    // compute warps: each sub-block as one grid of NCW * gridDim.x warps; a warp counts itself
    // done with a sub-block (a release at CTA scope) when it reaches the next one
    const uint64_t per_unit = p.Mj * p.vrow;          // vectors in one sub-block
    const uint64_t stride = (uint64_t)gridDim.x * NCW * 32;
    const uint64_t first_t = ((uint64_t)blockIdx.x * NCW + (warp - 1)) * 32 + lane;
    uint32_t pending = ~0u;                           // the sub-block whose count is still owed
    // the sub-blocks are walked in order, the pointers stepped one sub-block at a time (no
    // division or multiply per sub-block: a warp does its setup between two rounds of loads)
    uint32_t b = 0, j = 0;
    const uint64_t step = p.Mj * p.pitch;
    char* own = p.bufs[0];
    const char* slot0 = p.stage[0] + p.slot_off;
    for (uint32_t u = 0; u < units; ++u) {
        int go = 1;
        if (lane == 0) {
            uint32_t ns = 0;
            for (uint64_t i = 0;; ++i) {
                if (ld_acquire_cta(ctl + kReady) > u) break;
                if (ld_acquire_cta(ctl + kAbort) || i > 4 * p.max_polls + (1u << 20)) { go = 0; break; }
                __nanosleep(ns);
                ns = ns < 128 ? ns + 16 : 128;
            }
        }
        go = __shfl_sync(0xFFFFFFFFu, go, 0);
        if (!go) return;     // (an owed count is left unpaid: nothing after it gets marked)
        __syncwarp();        // the lanes' loads below follow lane 0's acquire
        if (pending != ~0u && lane == 0) red_release_cta(ctl + kDone + pending, 1);
        add_sub_block<DT, P, CONTIG>(p, b, own, slot0, first_t, stride, per_unit);
        __syncwarp();        // the warp's stores before lane 0's release (at the next sub-block)
        pending = u;
        if (++j == p.J) {
            j = 0;
            if (++b < (uint32_t)P) {
                own = p.bufs[b] + (uint64_t)b * p.Mb * p.pitch;
                slot0 = p.stage[b] + p.slot_off;
            }
        } else {
            own += step;
            slot0 += step;
        }
    }
    if (lane == 0) red_release_cta(ctl + kDone + pending, 1);
}

using ReduceFn = void (*)(ReduceParams);

// Sub-blocks of one all-reduce in all: the reduce kernel keeps a shared-memory counter for each.
constexpr uint32_t kMaxUnits = 4096;

// The instance for a dtype, P = 2 .. DTT_MAX_RANKS and rows back to back or padded (a kernel of
// its own each: the padded form's offsets need a division, and one kernel holding both would
// take the registers of the heavier).
template <int DT, bool C>
ReduceFn reduce_for(uint32_t P) {
    static_assert(DTT_MAX_RANKS == 16, "one instance per rank count");
    switch (P) {
        case 2: return reduce_kernel<DT, 2, C>;
        case 3: return reduce_kernel<DT, 3, C>;
        case 4: return reduce_kernel<DT, 4, C>;
        case 5: return reduce_kernel<DT, 5, C>;
        case 6: return reduce_kernel<DT, 6, C>;
        case 7: return reduce_kernel<DT, 7, C>;
        case 8: return reduce_kernel<DT, 8, C>;
        case 9: return reduce_kernel<DT, 9, C>;
        case 10: return reduce_kernel<DT, 10, C>;
        case 11: return reduce_kernel<DT, 11, C>;
        case 12: return reduce_kernel<DT, 12, C>;
        case 13: return reduce_kernel<DT, 13, C>;
        case 14: return reduce_kernel<DT, 14, C>;
        case 15: return reduce_kernel<DT, 15, C>;
        case 16: return reduce_kernel<DT, 16, C>;
        default: return nullptr;
    }
}

ReduceFn reduce_entry(uint32_t dtype, uint32_t P, bool contig) {
    if (dtype == DTT_BF16) return contig ? reduce_for<DTT_BF16, true>(P) : reduce_for<DTT_BF16, false>(P);
    return contig ? reduce_for<DTT_F32, true>(P) : reduce_for<DTT_F32, false>(P);
}

}  // namespace

cudaError_t preload_allreduce_kernels() {
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    for (uint32_t P = 2; P <= DTT_MAX_RANKS && e == cudaSuccess; ++P)
        for (uint32_t dt : {(uint32_t)DTT_BF16, (uint32_t)DTT_F32}) {
            for (bool c : {true, false}) {
                e = prepare_kernel(reduce_entry(dt, P, c));
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(reduce_entry(dt, P, c), cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
                if (e != cudaSuccess) break;
            }
            if (e != cudaSuccess) break;
        }
    return e;
}

}  // namespace dtt

using namespace dtt;

struct dtt_allreduce {
    uint32_t P = 0;
    dtt_allreduce_desc d{};
    uint64_t Mj = 0, rb = 0, pitch = 0, slot_off = 0, slot_bytes = 0;
    char* bufs[DTT_MAX_RANKS] = {};
    char* stage[DTT_MAX_RANKS] = {};
    dtt_plan* rs = nullptr;
    dtt_plan* ag = nullptr;
    uint32_t* d_counters = nullptr;
    uint64_t max_polls = 0;
    size_t smem = 0;                     // the reduce kernel's dynamic shared memory
    bool serial = false;                 // deferred_copier = 1: every kernel after its inputs
    bool gather = true;                  // all-reduce (false: reduce-scatter, no all-gather plan)
    cudaEvent_t ev_rs = nullptr;         // serial: the reduce-scatter copier has finished
    cudaEvent_t ev_reduce = nullptr;     // the reduce has finished (serial; and what a
                                         // reduce-scatter's wait waits for)
    // dtt_allreduce_host (made at its first call): the reduce's stream, and events ordering it
    // and the copies in after the round's start, and the marks after the copies in
    cudaStream_t host_stream = nullptr;
    cudaEvent_t ev_host = nullptr, ev_in = nullptr;
};

namespace {

void release(dtt_allreduce* ar) {
    if (!ar) return;
    if (ar->rs) dtt_plan_close(ar->rs);
    if (ar->ag) dtt_plan_close(ar->ag);
    if (ar->d_counters) cudaFree(ar->d_counters);
    if (ar->ev_rs) cudaEventDestroy(ar->ev_rs);
    if (ar->ev_reduce) cudaEventDestroy(ar->ev_reduce);
    if (ar->ev_host) cudaEventDestroy(ar->ev_host);
    if (ar->ev_in) cudaEventDestroy(ar->ev_in);
    if (ar->host_stream) cudaStreamDestroy(ar->host_stream);
    delete ar;
}

struct ScheduleSet {
    std::vector<dtt_schedule*> s;
    ~ScheduleSet() {
        for (dtt_schedule* x : s) dtt_schedule_free(x);
    }
};

// The bulk-copy copier the all-reduce defaults to: three one-warp CTAs per SM, two 16 KiB
// stages each -- light on registers and threads, so both plans' copiers and the reduce fit an SM
// (the reduce takes almost no shared memory).
dtt_plan_opts default_opts() {
    dtt_plan_opts o;
    dtt_plan_opts_default(&o);
    o.method = DTT_COPY_TMA;
    o.ctas_per_sm = 3;
    o.piece_bytes = 16384;
    o.stages = 2;
    return o;
}

int check_opts(const dtt_plan_opts& o, const char* which) {
    if (o.method == DTT_COPY_ENGINE)
        return fail(DTT_EINVAL, "dtt_allreduce_create: the %s plan cannot use the copy-engine transport", which);
    if (o.deferred_copier > 1 || o.overlap)
        return fail(DTT_EINVAL, "dtt_allreduce_create: the %s plan runs rounds one at a time with its copier "
                                "launched at start or in order (overlap 0, deferred_copier 0 or 1)", which);
    return DTT_OK;
}

// The reduce kernel's CTAs beside both copiers' on one SM (quiet: report no error, only the code).
int check_room(const dtt_allreduce* ar, bool quiet = false) {
    CopierRoom a, b;
    int rc = plan_copier_room(ar->rs, &a);
    if (rc == DTT_OK && ar->ag) rc = plan_copier_room(ar->ag, &b);
    if (rc != DTT_OK) return rc;
    int dev = 0, sms = 0, thr = 0, regs = 0, smem = 0, reserved = 0, blocks = 0;
    cudaFuncAttributes fa{};
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&thr, cudaDevAttrMaxThreadsPerMultiProcessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&regs, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&blocks, cudaDevAttrMaxBlocksPerMultiprocessor, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, reduce_entry(ar->d.dtype, ar->P, ar->pitch == ar->rb)) != cudaSuccess || sms <= 0)
        return fail(DTT_ECUDA, "dtt_allreduce_create: cannot query the device or the reduce kernel");
    const uint64_t per_sm = (ar->d.reduce_ctas + (uint64_t)sms - 1) / (uint64_t)sms;
    const uint64_t r_thr = per_sm * ar->d.reduce_threads;
    const uint64_t r_regs = r_thr * (((uint64_t)fa.numRegs + 7) / 8 * 8);
    const uint64_t r_smem = per_sm * (fa.sharedSizeBytes + ar->smem + (uint64_t)reserved);
    if (a.ctas + b.ctas + per_sm > (uint64_t)blocks || a.threads + b.threads + r_thr > (uint64_t)thr ||
        a.regs + b.regs + r_regs > (uint64_t)regs || a.smem + b.smem + r_smem > (uint64_t)smem) {
        if (quiet) return DTT_EINVAL;
        return fail(DTT_EINVAL,
                    "dtt_allreduce_create: per SM, the two copiers (%u + %u CTAs, %u + %u threads, %llu + %llu "
                    "registers, %llu + %llu bytes of shared memory) and %llu reduce CTA(s) of %u threads x %d "
                    "registers do not fit (%d threads, %d registers, %d bytes): the reduce waits on the copiers, "
                    "so all of them must be resident at once",
                    a.ctas, b.ctas, a.threads, b.threads, (unsigned long long)a.regs, (unsigned long long)b.regs,
                    (unsigned long long)a.smem, (unsigned long long)b.smem, (unsigned long long)per_sm,
                    ar->d.reduce_threads, fa.numRegs, thr, regs, smem);
    }
    return DTT_OK;
}

}  // namespace

extern "C" {

int dtt_allreduce_create(void* const* bufs, uint64_t buf_bytes, void* const* staging, uint64_t staging_bytes,
                         uint32_t P, const dtt_allreduce_desc* desc, const dtt_plan_opts* rs_opts,
                         const dtt_plan_opts* ag_opts, cudaStream_t rs_copy_stream, cudaStream_t ag_copy_stream,
                         dtt_allreduce** out) {
    if (!out) return fail(DTT_EINVAL, "dtt_allreduce_create: out is NULL");
    *out = nullptr;
    if (!bufs || !desc || P < 2 || P > DTT_MAX_RANKS)
        return fail(DTT_EINVAL, "dtt_allreduce_create: need buffers, a descriptor and 2 <= P <= %d", DTT_MAX_RANKS);
    dtt_allreduce_desc d = *desc;
    if (d.dtype != DTT_BF16 && d.dtype != DTT_F32)
        return fail(DTT_EINVAL, "dtt_allreduce_create: dtype must be DTT_BF16 or DTT_F32");
    if (d.sub_blocks == 0) d.sub_blocks = 1;
    // a control warp and 7 compute warps: the reduce alone is as fast with 15, but in the round
    // the copiers then have less of each SM (418 us rounds against 440 on the benchmark's size)
    if (d.reduce_threads == 0) d.reduce_threads = 256;
    const uint64_t eb = d.dtype == DTT_BF16 ? 2 : 4;
    if (d.block_rows == 0 || d.cols == 0 || d.block_rows % d.sub_blocks)
        return fail(DTT_EINVAL, "dtt_allreduce_create: block_rows and cols must be positive, sub_blocks must divide block_rows");
    if (d.cols > (1ull << 40) || d.block_rows > (1ull << 40))
        return fail(DTT_EINVAL, "dtt_allreduce_create: block too large");
    const uint64_t rb = d.cols * eb;
    if (d.pitch == 0) d.pitch = rb;
    if (rb % 16 || d.pitch % 16 || d.pitch < rb)
        return fail(DTT_EINVAL, "dtt_allreduce_create: row bytes and pitch must be multiples of 16, pitch >= row bytes");
    if (d.reduce_threads % 32 || d.reduce_threads < 64 || d.reduce_threads > kReduceMaxThreads)
        return fail(DTT_EINVAL, "dtt_allreduce_create: reduce_threads must be a multiple of 32 in [64, %u] "
                                "(a control warp and compute warps)", kReduceMaxThreads);
    const uint64_t Mj = d.block_rows / d.sub_blocks;
    if (Mj * (rb / 16) >= (1ull << 40) || (uint64_t)P * d.sub_blocks > kMaxUnits)
        return fail(DTT_EINVAL, "dtt_allreduce_create: at most %u sub-blocks in all (P x sub_blocks), "
                                "each under 2^40 vectors", kMaxUnits);
    const uint64_t M = (uint64_t)P * d.block_rows;
    uint64_t vec_span = 0, slots = 0, ends = 0;
    if (__builtin_mul_overflow(M, d.pitch, &vec_span) || __builtin_add_overflow(vec_span, vec_span, &ends))
        return fail(DTT_EINVAL, "dtt_allreduce_create: rows x pitch overflows 64 bits");
    const uint64_t vec_bytes = vec_span - d.pitch + rb;
    slots = vec_span;                                            // the P slots: P x block_rows rows
    const uint64_t slot_off = staging ? 0 : vec_span;
    if (vec_bytes > buf_bytes || (!staging && slot_off + slots > buf_bytes))
        return fail(DTT_EINVAL, "dtt_allreduce_create: a %llu-byte buffer cannot hold the vector%s (%llu bytes)",
                    (unsigned long long)buf_bytes, staging ? "" : " and the P slots after it",
                    (unsigned long long)(staging ? vec_bytes : slot_off + slots));
    if (staging && staging_bytes < slots)
        return fail(DTT_EINVAL, "dtt_allreduce_create: staging buffers need %llu bytes", (unsigned long long)slots);
    for (uint32_t r = 0; r < P; ++r) {
        if (!bufs[r] || reinterpret_cast<uintptr_t>(bufs[r]) % 16 ||
            (staging && (!staging[r] || reinterpret_cast<uintptr_t>(staging[r]) % 16)))
            return fail(DTT_EINVAL, "dtt_allreduce_create: buffers must be non-NULL and 16-byte aligned");
    }
    dtt_plan_opts ro = rs_opts ? *rs_opts : default_opts();
    dtt_plan_opts ao = ag_opts ? *ag_opts : default_opts();
    int rc = check_opts(ro, "reduce-scatter");
    if (rc == DTT_OK && !d.scatter_only) rc = check_opts(ao, "all-gather");
    if (rc == DTT_OK && !d.scatter_only && ro.deferred_copier != ao.deferred_copier)
        rc = fail(DTT_EINVAL, "dtt_allreduce_create: both plans launch their copiers the same way "
                              "(deferred_copier 0 for both, or 1 for both)");
    if (rc == DTT_OK) rc = preload_once();
    if (rc != DTT_OK) return rc;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return fail(DTT_ECUDA, "dtt_allreduce_create: cannot query the device");
    if (d.reduce_ctas == 0) d.reduce_ctas = (uint32_t)sms;

    ro.allgather = 0;
    ao.allgather = 0;
    ro.dst_bufs = staging;
    ro.dst_bytes = staging ? staging_bytes : 0;
    ao.dst_bufs = nullptr;
    ao.dst_bytes = 0;

    dtt_allreduce* ar = new (std::nothrow) dtt_allreduce();
    if (!ar) return fail(DTT_ENOMEM, "dtt_allreduce_create: out of memory");
    ar->P = P;
    ar->d = d;
    ar->Mj = Mj;
    ar->rb = rb;
    ar->pitch = d.pitch;
    ar->slot_off = slot_off;
    ar->slot_bytes = d.block_rows * d.pitch;
    ar->max_polls = ro.max_polls ? ro.max_polls : (1ull << 22);
    ar->serial = ro.deferred_copier == 1;
    ar->gather = d.scatter_only == 0;
    for (uint32_t r = 0; r < P; ++r) {
        ar->bufs[r] = static_cast<char*>(bufs[r]);
        ar->stage[r] = static_cast<char*>(staging ? staging[r] : bufs[r]);
    }

    // a sub-block's rows: one byte range when they are back to back, else a 2D window
    auto rows_region = [&](uint64_t row) {
        dtt_region g{};
        g.offset = row * d.pitch;
        if (d.pitch == rb) {
            g.row_bytes = Mj * rb;
            g.rows = 1;
            g.pitch = Mj * rb;
        } else {
            g.row_bytes = rb;
            g.rows = Mj;
            g.pitch = Mj > 1 ? d.pitch : rb;
        }
        return g;
    };
    ScheduleSet rs_s, ag_s;
    for (uint32_t s = 0; s < P && rc == DTT_OK; ++s) {
        dtt_schedule* sc = nullptr;
        rc = dtt_schedule_empty(&sc);
        if (rc != DTT_OK) break;
        rs_s.s.push_back(sc);
        for (uint32_t b = 0; b < P && rc == DTT_OK; ++b)
            for (uint32_t j = 0; j < d.sub_blocks && rc == DTT_OK; ++j) {
                const dtt_region g = rows_region((uint64_t)b * d.block_rows + (uint64_t)j * Mj);
                dtt_dest dst{};
                dst.offset = slot_off + ((uint64_t)s * d.block_rows + (uint64_t)j * Mj) * d.pitch;
                dst.pitch = g.pitch;
                rc = dtt_schedule_add_chunk_to(sc, &g, &dst, 1, 1, 1u << b);
            }
        dtt_schedule* ac = nullptr;
        if (rc == DTT_OK) rc = dtt_schedule_chunks((uint64_t)s * d.block_rows * d.pitch, d.block_rows, rb, d.pitch,
                                                   d.sub_blocks, &ac);
        if (ac) ag_s.s.push_back(ac);
    }
    if (rc == DTT_OK) rc = dtt_plan_create(bufs, buf_bytes, P, rs_s.s.data(), &ro, rs_copy_stream, &ar->rs);
    if (rc == DTT_OK) {
        // group (b, j) = b * J + j: chunk (s, b, j) of every rank s, rank s's chunks numbered
        // after the P * J of each lower rank
        const uint32_t J = d.sub_blocks, n = P * J;
        std::vector<uint32_t> offs(n + 1), ids((size_t)n * P);
        for (uint32_t g = 0; g <= n; ++g) offs[g] = g * P;
        for (uint32_t b = 0; b < P; ++b)
            for (uint32_t j = 0; j < J; ++j)
                for (uint32_t s = 0; s < P; ++s) ids[(size_t)(b * J + j) * P + s] = s * P * J + b * J + j;
        rc = dtt_plan_define_groups(ar->rs, n, offs.data(), ids.data());
    }
    if (rc == DTT_OK && ar->gather)
        rc = dtt_plan_create(bufs, buf_bytes, P, ag_s.s.data(), &ao, ag_copy_stream, &ar->ag);
    // in order (serial) nothing spins beside the reduce: no room to check
    ar->smem = (2 + (size_t)P * d.sub_blocks) * sizeof(uint32_t);
    if (rc == DTT_OK && !ar->serial) rc = check_room(ar);
    if (rc == DTT_OK &&
        (cudaEventCreateWithFlags(&ar->ev_rs, cudaEventDisableTiming) != cudaSuccess ||
         cudaEventCreateWithFlags(&ar->ev_reduce, cudaEventDisableTiming) != cudaSuccess))
        rc = fail(DTT_ECUDA, "dtt_allreduce_create: cannot create an event");
    if (rc == DTT_OK) {
        const size_t cb = (size_t)P * d.sub_blocks * sizeof(uint32_t);
        if (cudaMalloc(reinterpret_cast<void**>(&ar->d_counters), cb) != cudaSuccess)
            rc = fail(DTT_ENOMEM, "dtt_allreduce_create: cannot allocate the reduce counters");
        else if (cudaMemset(ar->d_counters, 0, cb) != cudaSuccess)
            rc = fail(DTT_ECUDA, "dtt_allreduce_create: cannot clear the reduce counters");
    }
    if (rc != DTT_OK) {
        const std::string msg = dtt_last_error();
        release(ar);
        return fail(rc, "%s", msg.c_str());
    }
    *out = ar;
    return DTT_OK;
}

int dtt_allreduce_plans(const dtt_allreduce* ar, dtt_plan** rs, dtt_plan** ag) {
    if (!ar) return fail(DTT_EINVAL, "dtt_allreduce_plans: NULL all-reduce");
    if (rs) *rs = ar->rs;
    if (ag) *ag = ar->ag;
    return DTT_OK;
}

int dtt_allreduce_start(dtt_allreduce* ar, cudaStream_t producer_stream, dtt_handle* rs_handles) {
    if (!ar) return fail(DTT_EINVAL, "dtt_allreduce_start: NULL all-reduce");
    if (dtt_plan_state(ar->rs) != DTT_PLAN_PREPARED ||
        (ar->ag && (dtt_plan_state(ar->ag) != DTT_PLAN_PREPARED || dtt_plan_round(ar->rs) != dtt_plan_round(ar->ag))))
        return fail(DTT_ESTATE, "dtt_allreduce_start: both plans must be PREPARED for the same round");
    dtt_handle tmp[DTT_MAX_RANKS];
    int rc = dtt_plan_start(ar->rs, producer_stream, rs_handles ? rs_handles : tmp);
    if (rc == DTT_OK && ar->ag) rc = dtt_plan_start(ar->ag, producer_stream, tmp);
    return rc;
}

int dtt_allreduce_reduce(dtt_allreduce* ar, uint32_t* err, cudaStream_t stream) {
    if (!ar || !err) return fail(DTT_EINVAL, "dtt_allreduce_reduce: NULL argument");
    if (dtt_plan_state(ar->rs) != DTT_PLAN_RUNNING ||
        (ar->ag && (dtt_plan_state(ar->ag) != DTT_PLAN_RUNNING || dtt_plan_round(ar->rs) != dtt_plan_round(ar->ag))))
        return fail(DTT_ESTATE, "dtt_allreduce_reduce: both plans must be RUNNING in the same round");
    if (stream == plan_copy_stream(ar->rs) || (ar->ag && stream == plan_copy_stream(ar->ag)))
        return fail(DTT_EINVAL, "dtt_allreduce_reduce: use a stream other than the plans' copy streams");
    ReduceParams p{};
    for (uint32_t r = 0; r < ar->P; ++r) {
        p.bufs[r] = ar->bufs[r];
        p.stage[r] = ar->stage[r];
        int rc = dtt_plan_handle(ar->rs, r, &p.rs[r]);
        if (rc == DTT_OK && ar->ag) rc = dtt_plan_handle(ar->ag, r, &p.ag[r]);
        if (rc != DTT_OK) return rc;
    }
    p.pitch = ar->pitch;
    p.slot_off = ar->slot_off;
    p.slot_bytes = ar->slot_bytes;
    p.Mb = ar->d.block_rows;
    p.Mj = ar->Mj;
    p.max_polls = ar->max_polls;
    p.J = ar->d.sub_blocks;
    p.vrow = (uint32_t)(ar->rb / 16);
    p.contig = ar->pitch == ar->rb ? 1u : 0u;
    p.gather = ar->gather ? 1u : 0u;
    p.counters = ar->d_counters;
    p.err = err;
    if (ar->serial) {
        // the reduce-scatter copier after the producers (on the producer stream so far), the
        // reduce after that copier
        const int rc = dtt_plan_launch_copier(ar->rs);
        if (rc != DTT_OK) return rc;
        DTT_CUDA_TRY(cudaEventRecord(ar->ev_rs, plan_copy_stream(ar->rs)));
        DTT_CUDA_TRY(cudaStreamWaitEvent(stream, ar->ev_rs, 0));
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(ar->d.reduce_ctas, 1, 1);
    cfg.blockDim = dim3(ar->d.reduce_threads, 1, 1);
    cfg.dynamicSmemBytes = ar->smem;
    cfg.stream = stream;
    void* args[] = {&p};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(reduce_entry(ar->d.dtype, ar->P, ar->pitch == ar->rb)), args);
    if (e != cudaSuccess) return fail(DTT_ECUDA, "dtt_allreduce_reduce: launch failed: %s", cudaGetErrorString(e));
    DTT_CUDA_TRY(cudaEventRecord(ar->ev_reduce, stream));
    if (ar->serial && ar->ag) {
        // the all-gather copier after the reduce (and after the producer stream's work)
        DTT_CUDA_TRY(cudaStreamWaitEvent(plan_copy_stream(ar->ag), ar->ev_reduce, 0));
        return dtt_plan_launch_copier(ar->ag);
    }
    return DTT_OK;
}

int dtt_allreduce_wait(dtt_allreduce* ar, dtt_report* rs_report, dtt_report* ag_report) {
    if (!ar) return fail(DTT_EINVAL, "dtt_allreduce_wait: NULL all-reduce");
    const int a = dtt_plan_wait(ar->rs, rs_report);
    const std::string msg = a != DTT_OK ? std::string(dtt_last_error()) : std::string();
    if (!ar->ag) {
        // a reduce-scatter: its result is the reduce kernel's stores (bounded: its waits end)
        if (ag_report) *ag_report = dtt_report{};
        if (a != DTT_OK) return fail(a, "reduce-scatter: %s", msg.c_str());
        DTT_CUDA_TRY(cudaEventSynchronize(ar->ev_reduce));
        return DTT_OK;
    }
    const int b = dtt_plan_wait(ar->ag, ag_report);
    if (a != DTT_OK) return fail(a, "reduce-scatter: %s", msg.c_str());
    if (b != DTT_OK) {
        const std::string m2 = dtt_last_error();
        return fail(b, "all-gather: %s", m2.c_str());
    }
    return DTT_OK;
}

int dtt_allreduce_host(dtt_allreduce* ar, const void* const* host_parts, void* host_out, uint32_t out_rank,
                       uint32_t* err, cudaStream_t stream, dtt_report* rs_report, dtt_report* ag_report) {
    if (!ar || !host_parts || !err) return fail(DTT_EINVAL, "dtt_allreduce_host: NULL argument");
    if (!ar->ag) return fail(DTT_EINVAL, "dtt_allreduce_host: needs an all-reduce (not scatter_only)");
    if (ar->serial)
        return fail(DTT_EINVAL, "dtt_allreduce_host: the reduce runs while the vectors come in: not with "
                                "deferred_copier = 1");
    if (out_rank >= ar->P) return fail(DTT_EINVAL, "dtt_allreduce_host: out_rank out of range");
    PlanHostIo in{}, out{};
    int rc = plan_host_io(ar->rs, &in);
    if (rc == DTT_OK) rc = plan_host_io(ar->ag, &out);
    if (rc != DTT_OK) return rc;
    if ((!ar->host_stream && cudaStreamCreateWithFlags(&ar->host_stream, cudaStreamNonBlocking) != cudaSuccess) ||
        (!ar->ev_host && cudaEventCreateWithFlags(&ar->ev_host, cudaEventDisableTiming) != cudaSuccess) ||
        (!ar->ev_in && cudaEventCreateWithFlags(&ar->ev_in, cudaEventDisableTiming) != cudaSuccess))
        return fail(DTT_ECUDA, "dtt_allreduce_host: cannot create its stream or events");
    const uint32_t P = ar->P, J = ar->d.sub_blocks;
    const uint64_t Mb = ar->d.block_rows, Mj = ar->Mj, rb = ar->rb, pitch = ar->pitch;

    // the all-gather copier stamps each chunk's arrival into mapped host memory for the copy back
    plan_set_host_round(ar->ag, host_out != nullptr, false);
    dtt_handle h[DTT_MAX_RANKS];
    rc = dtt_allreduce_start(ar, stream, h);
    plan_set_host_round(ar->ag, false, false);
    if (rc != DTT_OK) return rc;
    const uint32_t R = dtt_plan_round(ar->ag);

    // The reduce on a stream of its own, after start's work on `stream`: it waits on each
    // sub-block's group while the later rows are still coming in.
    DTT_CUDA_TRY(cudaEventRecord(ar->ev_host, stream));
    DTT_CUDA_TRY(cudaStreamWaitEvent(ar->host_stream, ar->ev_host, 0));
    DTT_CUDA_TRY(cudaStreamWaitEvent(in.h2d, ar->ev_host, 0));
    rc = dtt_allreduce_reduce(ar, err, ar->host_stream);
    if (rc != DTT_OK) return rc;

    // rows [r0, r0 + n) of a vector between the host (rows back to back) and the device (pitch)
    auto rows_copy = [&](char* dst, uint64_t dpitch, const char* src, uint64_t spitch, uint64_t n,
                         cudaMemcpyKind kind, cudaStream_t s) -> cudaError_t {
        if (dpitch == rb && spitch == rb) return cudaMemcpyAsync(dst, src, n * rb, kind, s);
        return cudaMemcpy2DAsync(dst, dpitch, src, spitch, rb, n, kind, s);
    };
    // Copy back: block b of out_rank's result, sub-block by sub-block as the all-gather delivers
    // them (its own block once its chunks have gone out: the reduce wrote them before marking),
    // in copies of at least 8 MiB or the rest of the block.
    std::vector<uint32_t> back(P, 0);
    const uint64_t kBack = 8ull << 20;
    auto poll = [&](bool final) -> int {
        for (uint32_t b = 0; b < P; ++b) {
            uint32_t k = back[b];
            while (k < J && __atomic_load_n(&out.arrived[b * J + k], __ATOMIC_ACQUIRE) == R) ++k;
            if (k == back[b] || !(k == J || final || (k - back[b]) * Mj * rb >= kBack)) continue;
            const uint64_t r0 = b * Mb + back[b] * Mj;
            const cudaError_t e = rows_copy(static_cast<char*>(host_out) + r0 * rb, rb,
                                            ar->bufs[out_rank] + r0 * pitch, pitch, (k - back[b]) * Mj,
                                            cudaMemcpyDeviceToHost, out.d2h);
            if (e != cudaSuccess) return fail(DTT_ECUDA, "dtt_allreduce_host: %s", cudaGetErrorString(e));
            back[b] = k;
        }
        return DTT_OK;
    };

    // Copies in, in the groups' order: sub-blocks [j0, j1) of block b (at least the reduce-scatter
    // plan's host_piece_bytes of a rank, 0: 16 MiB, or the rest of the block) of every rank, then
    // the marks of those reduce-scatter chunks -- rank s's chunk (b, j) is s * P * J + b * J + j --
    // once the copies have landed.  (On the host link of a GB300, copies in of 4 MiB ran at ~190
    // GB/s against ~205 for 16 MiB and ~55 for 1 MiB.)
    const uint64_t kIn = in.piece_bytes ? in.piece_bytes : (16ull << 20);
    for (uint32_t b = 0; b < P; ++b) {
        for (uint32_t j0 = 0; j0 < J;) {
            uint32_t j1 = j0 + 1;
            while (j1 < J && (j1 - j0) * Mj * rb < kIn) ++j1;
            const uint64_t r0 = b * Mb + j0 * Mj, n = (j1 - j0) * Mj;
            bool any = false;
            for (uint32_t s = 0; s < P; ++s) {
                if (!host_parts[s]) continue;
                const cudaError_t e = rows_copy(ar->bufs[s] + r0 * pitch, pitch,
                                                static_cast<const char*>(host_parts[s]) + r0 * rb, rb, n,
                                                cudaMemcpyHostToDevice, in.h2d);
                if (e != cudaSuccess) return fail(DTT_ECUDA, "dtt_allreduce_host: %s", cudaGetErrorString(e));
                any = true;
            }
            if (any) {
                DTT_CUDA_TRY(cudaEventRecord(ar->ev_in, in.h2d));
                DTT_CUDA_TRY(cudaStreamWaitEvent(stream, ar->ev_in, 0));
            }
            for (uint32_t s = 0; s < P; ++s) {
                rc = dtt_publish(h, P, s * P * J + b * J + j0, j1 - j0, 0, stream);
                if (rc != DTT_OK) return rc;
            }
            if (host_out && (rc = poll(false)) != DTT_OK) return rc;
            j0 = j1;
        }
    }
    // the reduce before whatever follows on `stream` (its error word included)
    DTT_CUDA_TRY(cudaStreamWaitEvent(stream, ar->ev_reduce, 0));
    if (host_out) {
        // the rest as it arrives; once the all-gather copier has exited, whatever arrived is final
        for (uint64_t spin = 1;; ++spin) {
            if ((rc = poll(false)) != DTT_OK) return rc;
            bool all = true;
            for (uint32_t b = 0; b < P; ++b) all = all && back[b] == J;
            if (all) break;
            if ((spin & 1023) == 0) {
                const cudaError_t e = cudaEventQuery(out.copier_end);
                if (e == cudaSuccess) break;
                if (e != cudaErrorNotReady) return fail(DTT_ECUDA, "dtt_allreduce_host: %s", cudaGetErrorString(e));
            }
        }
        if ((rc = poll(true)) != DTT_OK) return rc;
    }
    plan_set_host_round(ar->ag, false, true);
    rc = dtt_allreduce_wait(ar, rs_report, ag_report);
    plan_set_host_round(ar->ag, false, false);
    if (rc != DTT_OK) {
        cudaStreamSynchronize(out.d2h);
        return rc;
    }
    if (host_out) {
        DTT_CUDA_TRY(cudaStreamSynchronize(out.d2h));
        for (uint32_t b = 0; b < P; ++b)
            if (back[b] != J) return fail(DTT_ETIMEDOUT, "dtt_allreduce_host: block %u came back short", b);
    }
    return dtt_allreduce_next_round(ar);
}

int dtt_allreduce_next_round(dtt_allreduce* ar) {
    if (!ar) return fail(DTT_EINVAL, "dtt_allreduce_next_round: NULL all-reduce");
    if (dtt_plan_state(ar->rs) != DTT_PLAN_DONE || (ar->ag && dtt_plan_state(ar->ag) != DTT_PLAN_DONE))
        return fail(DTT_ESTATE, "dtt_allreduce_next_round: both plans must be DONE");
    int rc = dtt_plan_next_round(ar->rs);
    if (rc == DTT_OK && ar->ag) rc = dtt_plan_next_round(ar->ag);
    return rc;
}

int dtt_allreduce_destroy(dtt_allreduce* ar) {
    if (!ar) return DTT_OK;
    int rc = DTT_OK;
    if (ar->rs) {
        const int a = dtt_plan_close(ar->rs);
        if (a != DTT_OK) rc = a;
        ar->rs = nullptr;
    }
    if (ar->ag) {
        const int b = dtt_plan_close(ar->ag);
        if (b != DTT_OK && rc == DTT_OK) rc = b;
        ar->ag = nullptr;
    }
    release(ar);
    return rc;
}

}  // extern "C"
