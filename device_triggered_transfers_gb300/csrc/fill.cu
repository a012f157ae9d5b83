// The hashed-fill producer: a persistent tiled producer that writes hash(seed, rank, round,
// row, col) values into each rank's slice and marks chunks as it goes ("Triggered Plans",
// section Model: program p takes steps p, p + num_programs, ..., stores the step's tile and
// marks first_chunk + step / num_programs).  One launch covers every virtual rank
// (blockIdx.y = rank).  A program is one CTA, or a thread-block cluster whose CTAs split each
// tile by rows and mark once per step through dtt_mark_ready_cluster.
#include <cstdint>

#include <cuda_bf16.h>

#include "dtt_device.cuh"
#include "internal.h"
#include "order.h"

namespace dtt {
namespace {

struct FillParams {
    char* bufs[DTT_MAX_RANKS];
    dtt_handle h[DTT_MAX_RANKS];
    uint64_t slice_off[DTT_MAX_RANKS];
    uint64_t M, N, pitch;
    uint32_t seed, BM, BN, NP, TPC;
    uint32_t order_kind, group_m, mark_mode, cluster, rank_mask;
    uint32_t vec;    // 16-byte stores allowed (bases, offsets, pitch and BN*elem aligned)
    uint32_t group;  // CTAs that write one step together and mark it once (counter-based)
    uint32_t* counters;   // group > 1: one per (rank, step), zero between rounds
    uint32_t pace;        // > 0: wait for chunk k - pace to be reusable before chunk k
};

// Polls of the pacing wait: advisory, so it gives up after about a millisecond.
constexpr uint64_t kPacePolls = 4096;

// MurmurHash3's 32-bit finaliser (public-domain hash by Austin Appleby).
__device__ __forceinline__ uint32_t fmix32(uint32_t h) {
    h ^= h >> 16;
    h *= 0x85EBCA6Bu;
    h ^= h >> 13;
    h *= 0xC2B2AE35u;
    h ^= h >> 16;
    return h;
}

// fmix32 after its first xor-shift.
__device__ __forceinline__ uint32_t fmix32_tail(uint32_t h) {
    h *= 0x85EBCA6Bu;
    h ^= h >> 13;
    h *= 0xC2B2AE35u;
    h ^= h >> 16;
    return h;
}

// fmix32((idx + i) ^ salt) for the elements i < 16 of a vector whose first index idx is a
// multiple of 16 / elem_bytes: idx + i = idx ^ i, and i leaves bits 16 and up alone, so the
// salt, the index and the first xor-shift fold into one value per vector, B = X ^ (X >> 16)
// with X = idx ^ salt, and element i hashes to fmix32_tail(B ^ i).
__device__ __forceinline__ uint32_t vec_base(uint32_t idx, uint32_t salt) {
    const uint32_t x = idx ^ salt;
    return x ^ (x >> 16);
}

// ((h >> 8) - 2^23) * 2^-23, an exact float in [-1, 1), built from bits.  With m the mantissa
// bits 8..30 of h, f = 1 + m 2^-23 lies in [1, 2); the result is (f - 1.5) + 0.5 when bit 31 of
// h is set and (f - 1.5) - 0.5 otherwise.  Every step is exact, so this equals the integer form.
__device__ __forceinline__ float uniform(uint32_t h) {
    const float f = __uint_as_float(((h >> 8) & 0x7FFFFFu) | 0x3F800000u);
    const float half = __uint_as_float((~h & 0x80000000u) | 0x3F000000u);   // +-0.5
    return (f - 1.5f) + half;
}

template <int DT> struct Elem;
template <> struct Elem<DTT_BF16> {
    static constexpr int bytes = 2;
    static __device__ __forceinline__ uint4 pack(uint32_t b) {
        uint32_t w[4];
#pragma unroll
        for (uint32_t i = 0; i < 4; ++i) {
            const __nv_bfloat162 v = __floats2bfloat162_rn(uniform(fmix32_tail(b ^ (2 * i))),
                                                           uniform(fmix32_tail(b ^ (2 * i + 1))));
            w[i] = *reinterpret_cast<const uint32_t*>(&v);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    static __device__ __forceinline__ void scalar(char* p, uint32_t salt, uint32_t idx) {
        *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(uniform(fmix32(idx ^ salt)));
    }
};
template <> struct Elem<DTT_F32> {
    static constexpr int bytes = 4;
    static __device__ __forceinline__ uint4 pack(uint32_t b) {
        return make_uint4(__float_as_uint(uniform(fmix32_tail(b))),
                          __float_as_uint(uniform(fmix32_tail(b ^ 1u))),
                          __float_as_uint(uniform(fmix32_tail(b ^ 2u))),
                          __float_as_uint(uniform(fmix32_tail(b ^ 3u))));
    }
    static __device__ __forceinline__ void scalar(char* p, uint32_t salt, uint32_t idx) {
        *reinterpret_cast<float*>(p) = uniform(fmix32(idx ^ salt));
    }
};
// fmix32_tail without its last xor-shift: the low byte of the full hash is the xor of bytes 0
// and 2 of this value.
__device__ __forceinline__ uint32_t fmix32_tail_open(uint32_t h) {
    h *= 0x85EBCA6Bu;
    h ^= h >> 13;
    h *= 0xC2B2AE35u;
    return h;
}

template <> struct Elem<DTT_U8> {
    static constexpr int bytes = 1;
    static __device__ __forceinline__ uint4 pack(uint32_t b) {
        uint32_t w[4];
#pragma unroll
        for (uint32_t i = 0; i < 4; ++i) {
            // the low bytes of four hashes g ^ (g >> 16) in one word: bytes 0 and 2 of each g
            // gathered by two permutes per pair, then one xor for all four
            const uint32_t g0 = fmix32_tail_open(b ^ (4 * i)), g1 = fmix32_tail_open(b ^ (4 * i + 1));
            const uint32_t g2 = fmix32_tail_open(b ^ (4 * i + 2)), g3 = fmix32_tail_open(b ^ (4 * i + 3));
            const uint32_t p = __byte_perm(g0, g1, 0x6240);   // g0.b0 g1.b0 g0.b2 g1.b2
            const uint32_t q = __byte_perm(g2, g3, 0x6240);   // g2.b0 g3.b0 g2.b2 g3.b2
            w[i] = __byte_perm(p, q, 0x5410) ^ __byte_perm(p, q, 0x7632);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    static __device__ __forceinline__ void scalar(char* p, uint32_t salt, uint32_t idx) {
        *reinterpret_cast<uint8_t*>(p) = (uint8_t)(fmix32(idx ^ salt) & 0xFFu);
    }
};

// Write rows [ra, rb) x cols [c0, c0 + cols) of rank r's slice.
template <int DT>
__device__ __forceinline__ void write_block(const FillParams& p, char* base, uint32_t salt,
                                            uint64_t ra, uint64_t rb, uint64_t c0, uint64_t cols) {
    using E = Elem<DT>;
    constexpr uint32_t VPE = 16 / E::bytes;     // elements per 16-byte vector
    if (ra >= rb || cols == 0) return;
    const uint32_t nrows = (uint32_t)(rb - ra);
    if (p.vec && c0 == 0 && cols == p.N && p.pitch == p.N * E::bytes &&
        (uint64_t)nrows * (p.N / VPE) < (1ull << 32)) {
        // whole rows that follow each other: one contiguous range, vector v at byte 16 v of it
        const uint32_t nv = nrows * (uint32_t)(p.N / VPE), step = blockDim.x * VPE;
        uint4* d = reinterpret_cast<uint4*>(base + ra * p.pitch) + threadIdx.x;
        uint32_t idx = (uint32_t)(ra * p.N) + threadIdx.x * VPE;
        for (uint32_t v = threadIdx.x; v < nv; v += blockDim.x, d += blockDim.x, idx += step)
            *d = E::pack(vec_base(idx, salt));
        return;
    }
    uint32_t nvec = 0;
    if (p.vec) {
        // thread t takes vectors t, t + blockDim, ... of the block; (row i, vector k) advances
        // by a fixed quotient and remainder instead of a division per vector
        nvec = (uint32_t)(cols / VPE);
        if (nvec) {
            const uint32_t total = nrows * nvec;
            const uint32_t dq = blockDim.x / nvec, dr = blockDim.x % nvec;
            uint32_t i = threadIdx.x / nvec, k = threadIdx.x % nvec;
            for (uint32_t v = threadIdx.x; v < total; v += blockDim.x) {
                const uint64_t row = ra + i, col = c0 + (uint64_t)k * VPE;
                const uint32_t idx = (uint32_t)(row * p.N + col);
                *reinterpret_cast<uint4*>(base + row * p.pitch + col * E::bytes) = E::pack(vec_base(idx, salt));
                i += dq;
                k += dr;
                if (k >= nvec) { k -= nvec; ++i; }
            }
        }
    }
    const uint32_t done = nvec * VPE, tail = (uint32_t)cols - done;
    if (tail == 0) return;
    const uint32_t total = nrows * tail;
    for (uint32_t v = threadIdx.x; v < total; v += blockDim.x) {
        const uint32_t i = v / tail, k = v - i * tail;
        const uint64_t row = ra + i, col = c0 + done + k;
        E::scalar(base + row * p.pitch + col * E::bytes, salt, (uint32_t)(row * p.N + col));
    }
}

__device__ __forceinline__ void mark(const dtt_handle& h, uint32_t chunk, uint32_t cluster) {
    if (cluster > 1)
        dtt_mark_ready_cluster(h, chunk);
    else
        dtt_mark_ready(h, chunk);
}

// A group of `group` CTAs acting as one writer: each CTA orders its stores before an acq_rel
// add on the step's counter; the CTA whose add completes the group has acquired every other
// CTA's stores, resets the counter for the next round (the next launch is stream-ordered after
// this one) and issues the chunk's one mark.
__device__ __forceinline__ void group_mark(const dtt_handle& h, uint32_t chunk, uint32_t* counter,
                                           uint32_t group) {
    __syncthreads();
    if (dtt_dev::first_thread()) {
        uint32_t old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
        if (old + 1 == group) {
            asm volatile("st.relaxed.gpu.global.u32 [%0], 0;" ::"l"(counter) : "memory");
            dtt_dev::mark_one(h, chunk);
        }
    }
    __syncthreads();
}

// Per-chunk waits of a fill CTA, made when it reaches chunk k of its rank (bits of `waits`):
//  - kWritable (overlapping rounds): the previous round's copies of chunk k must have landed
//    before its bytes change (that round's copier may still be reading them); every CTA of a
//    program asks for itself.  A wait that runs out sets kNoWrite -- the rest of this CTA's
//    writes are left undone, while its marks still go out, so no barrier of a cluster or counter
//    of a group is left waiting -- and DTT_DEV_EWRITABLE, which fails the round.
//  - kPacing: keep the bytes written but not yet delivered within `pace` chunks of this rank,
//    so that the copier reads them from L2; the result does not depend on the outcome.  A wait
//    that runs out means the copier is not keeping up (or not running): the CTA stops pacing, so
//    it stalls at most once per launch.  With overlapping rounds the chunks before this round's
//    first `pace` are the previous round's last ones (its copier runs just before this round's):
//    chunk k < pace waits for the previous round's delivery of chunk n - pace + k.
// The loop carries two words for them: the waits still made, and the current chunk.
constexpr uint32_t kPacing = 1u, kWritable = 2u, kNoWrite = 4u;

__device__ __forceinline__ uint32_t chunk_waits(const dtt_handle& h, uint32_t k, uint32_t waits, uint32_t pace) {
    if ((waits & kWritable) && !(waits & kNoWrite) &&
        dtt_wait_writable(h, h.first_chunk + k, kWritablePolls) != 0) {
        waits |= kNoWrite;
        if (dtt_dev::first_thread()) atomicOr(h.status, DTT_DEV_EWRITABLE);
    }
    if (waits & kPacing) {
        int w = 0;
        if (k >= pace)
            w = dtt_wait_reusable(h, h.first_chunk + (k - pace), kPacePolls);
        else if ((waits & kWritable) && h.n_chunks + k >= pace)
            w = dtt_wait_writable(h, h.first_chunk + (h.n_chunks + k - pace), kPacePolls);
        if (w != 0) waits &= ~kPacing;
    }
    return waits;
}

template <int DT>
__device__ __forceinline__ void fill_body(const FillParams& p) {
    const uint32_t r = blockIdx.y;
    if (!((p.rank_mask >> r) & 1u)) return;
    const dtt_handle& h = p.h[r];
    const uint32_t team = p.cluster * p.group;          // CTAs of one program (one writer)
    const uint32_t prog = blockIdx.x / team, member = blockIdx.x % team;
    const uint64_t tiles_m = (p.M + p.BM - 1) / p.BM, tiles_n = (p.N + p.BN - 1) / p.BN;
    const uint64_t T = tiles_m * tiles_n;
    const uint32_t salt = fmix32(p.seed ^ fmix32(r ^ fmix32(h.round)));
    char* base = p.bufs[r] + p.slice_off[r];
    // the waits a CTA makes when it reaches a new chunk (chunk_waits): bits of kPacing,
    // kWritable and kNoWrite, two words carried through the loop
    uint32_t waits = (p.pace ? kPacing : 0u) | ((h.flags & DTT_HANDLE_OVERLAP) ? kWritable : 0u);
    uint32_t cur = 0xFFFFFFFFu;   // index within the rank of the chunk of the last step
    for (uint64_t step = prog; step < T; step += p.NP) {
        const uint32_t k = p.mark_mode == DTT_MARK_AT_END ? 0u : (uint32_t)step / p.TPC;   // T < 2^31
        if (k != cur) {
            cur = k;
            if (waits & (kPacing | kWritable)) waits = chunk_waits(h, k, waits, p.pace);
        }
        uint32_t tm, tn;
        tile_of(p.order_kind, p.group_m, step, (uint32_t)tiles_m, (uint32_t)tiles_n, &tm, &tn);
        const uint64_t r0 = (uint64_t)tm * p.BM, c0 = (uint64_t)tn * p.BN;
        const uint64_t rows = min((uint64_t)p.BM, p.M - r0), cols = min((uint64_t)p.BN, p.N - c0);
        const uint64_t per = (rows + team - 1) / team;
        const uint64_t ra = r0 + min(rows, member * per), rb = r0 + min(rows, (member + 1) * per);
        if (!(waits & kNoWrite)) write_block<DT>(p, base, salt, ra, rb, c0, cols);
        if (p.mark_mode == DTT_MARK_PER_STEP) {
            const uint32_t chunk = h.first_chunk + k;
            if (p.group > 1)
                group_mark(h, chunk, p.counters + (uint64_t)r * T + step, p.group);
            else
                mark(h, chunk, p.cluster);
        }
    }
    if (p.mark_mode == DTT_MARK_AT_END) mark(h, h.first_chunk, p.cluster);
}

// The fill with up to 64 registers a thread (its fastest inner loop; 1024-thread CTAs still fit
// an SM).  The cap is stated: left to itself the compiler laid one instance out in 32 registers
// with spills.
template <int DT>
__global__ void __maxnreg__(64) fill_kernel(const __grid_constant__ FillParams p) {
    fill_body<DT>(p);
}

// The same fill in at most 56 registers a thread, for paced launches that need several
// producer CTAs of an SM resident at once beside the copier's: eight 128-thread CTAs then leave
// the registers of three copier CTAs free (with 64 registers they would take all of them).
template <int DT>
__global__ void __maxnreg__(56) fill_kernel_lean(const __grid_constant__ FillParams p) {
    fill_body<DT>(p);
}

}  // namespace

template <class K>
static cudaError_t prepare_fill(K kernel) {
    cudaError_t e = prepare_kernel(kernel);
    // clusters of up to 16 CTAs (beyond the portable 8) for one-writer chunks
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

cudaError_t preload_fill_kernels() {
    cudaError_t e = prepare_fill(fill_kernel<DTT_BF16>);
    if (e == cudaSuccess) e = prepare_fill(fill_kernel<DTT_F32>);
    if (e == cudaSuccess) e = prepare_fill(fill_kernel<DTT_U8>);
    if (e == cudaSuccess) e = prepare_fill(fill_kernel_lean<DTT_BF16>);
    if (e == cudaSuccess) e = prepare_fill(fill_kernel_lean<DTT_F32>);
    if (e == cudaSuccess) e = prepare_fill(fill_kernel_lean<DTT_U8>);
    return e;
}

namespace {

// The fill kernel for a dtype, lean (register-capped) or not.
const void* fill_entry(uint32_t dtype, bool lean) {
    if (lean)
        return dtype == DTT_BF16 ? (const void*)fill_kernel_lean<DTT_BF16>
             : dtype == DTT_F32  ? (const void*)fill_kernel_lean<DTT_F32>
                                 : (const void*)fill_kernel_lean<DTT_U8>;
    return dtype == DTT_BF16 ? (const void*)fill_kernel<DTT_BF16>
         : dtype == DTT_F32  ? (const void*)fill_kernel<DTT_F32>
                             : (const void*)fill_kernel<DTT_U8>;
}

}  // namespace

}  // namespace dtt

using namespace dtt;

extern "C" int dtt_fill_producer(void* const* bufs, uint32_t P, const dtt_fill_desc* d,
                                 const dtt_handle* handles, cudaStream_t stream) {
    if (!bufs || !d || !handles || P < 1 || P > DTT_MAX_RANKS)
        return fail(DTT_EINVAL, "dtt_fill_producer: bad args");
    if (d->M == 0 || d->N == 0 || d->BM == 0 || d->BN == 0 || d->num_programs == 0 ||
        d->tiles_per_chunk == 0)
        return fail(DTT_EINVAL, "dtt_fill_producer: sizes must be positive");
    if (d->dtype > DTT_U8 || d->mark_mode > DTT_MARK_AT_END)
        return fail(DTT_EINVAL, "dtt_fill_producer: bad dtype or mark mode");
    const uint32_t cluster = d->cluster ? d->cluster : 1;
    const uint32_t group = d->group ? d->group : 1;
    const uint32_t threads = d->threads ? d->threads : 256;
    if (cluster > 16 || threads % 32 || threads > 1024)
        return fail(DTT_EINVAL, "dtt_fill_producer: cluster <= 16, threads a multiple of 32 <= 1024");
    if ((handles[0].flags & DTT_HANDLE_OVERLAP) && threads > 512)
        // with overlapping rounds the next round's copier is queued behind this round's and may
        // take an SM before this producer's CTAs do: each CTA must fit beside the copier's CTAs
        // (which keep to half an SM), so at most 512 threads of up to 64 registers
        return fail(DTT_EINVAL, "dtt_fill_producer: with overlapping rounds a producer CTA has at most 512 threads "
                                "(it must fit on an SM beside the copier's CTAs)");
    if (group > 1 && (cluster > 1 || d->mark_mode != DTT_MARK_PER_STEP || !d->group_counters))
        return fail(DTT_EINVAL, "dtt_fill_producer: group writers need cluster 1, per-step marks and counters");
    if ((uint64_t)d->num_programs * cluster * group > 0x7FFFFFFFull)
        return fail(DTT_EINVAL, "dtt_fill_producer: grid too large");
    const uint32_t eb = d->dtype == DTT_BF16 ? 2 : d->dtype == DTT_F32 ? 4 : 1;
    if (((d->M + d->BM - 1) / d->BM) * ((d->N + d->BN - 1) / d->BN) >= (1ull << 31))
        return fail(DTT_EINVAL, "dtt_fill_producer: a rank's slice must have fewer than 2^31 tiles");
    if ((uint64_t)d->BM * d->BN >= (1ull << 31))
        return fail(DTT_EINVAL, "dtt_fill_producer: a BM x BN tile must hold fewer than 2^31 elements");
    if (d->M > 1 && d->pitch < d->N * eb) return fail(DTT_EINVAL, "dtt_fill_producer: pitch < row bytes");
    const uint64_t span = (d->M - 1) * d->pitch + d->N * eb;
    for (uint32_t r = 0; r < P; ++r)
        if (((d->rank_mask >> r) & 1u) && (d->slice_off[r] > d->buf_bytes || span > d->buf_bytes - d->slice_off[r]))
            return fail(DTT_EINVAL, "dtt_fill_producer: rank %u's slice runs past its %llu-byte buffer", r,
                        (unsigned long long)d->buf_bytes);
    FillParams p{};
    // 16-byte stores need aligned rows and tile columns; the folded per-vector hash also needs
    // every vector's first element index (row * N + col) to be a multiple of the vector width
    bool vec = (d->pitch % 16 == 0) && ((uint64_t)d->BN * eb % 16 == 0) && (d->N % (16 / eb) == 0);
    for (uint32_t r = 0; r < P; ++r) {
        p.bufs[r] = static_cast<char*>(bufs[r]);
        p.h[r] = handles[r];
        p.slice_off[r] = d->slice_off[r];
        vec = vec && (reinterpret_cast<uintptr_t>(bufs[r]) % 16 == 0) && (d->slice_off[r] % 16 == 0);
    }
    p.M = d->M;
    p.N = d->N;
    p.pitch = d->pitch;
    p.seed = d->seed;
    p.BM = d->BM;
    p.BN = d->BN;
    p.NP = d->num_programs;
    p.TPC = d->tiles_per_chunk;
    p.order_kind = d->order.kind;
    p.group_m = d->order.group_m;
    p.mark_mode = d->mark_mode;
    p.cluster = cluster;
    p.rank_mask = d->rank_mask;
    p.vec = vec ? 1u : 0u;
    p.group = group;
    p.counters = d->group_counters;
    p.pace = d->pace;
    bool lean = false;     // the register-capped fill (paced launches with several CTAs per SM)
    if (p.pace) {
        // a paced program waits for chunks that other programs write: they must all be
        // resident at once, or the waits only run out (the copier's CTAs take room too, so this
        // is a necessary condition, not a sufficient one)
        // Ranks outside rank_mask exit at once and hold no room.  Clusters are placed whole, so
        // for cluster > 1 the count that matters is of clusters the device can hold at once.
        uint32_t producing = 0;
        for (uint32_t r = 0; r < P; ++r) producing += (d->rank_mask >> r) & 1u;
        // several CTAs of an SM must be resident at once beside the copier: the lean fill
        int sms = 0, dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            return fail(DTT_ECUDA, "dtt_fill_producer: cannot query the SM count");
        lean = (uint64_t)d->num_programs * cluster * group * producing > (uint64_t)sms;
        const void* k = fill_entry(d->dtype, lean);
        if (cluster > 1) {
            cudaLaunchConfig_t occ{};
            occ.gridDim = dim3(d->num_programs * cluster * group, P, 1);
            occ.blockDim = dim3(threads, 1, 1);
            cudaLaunchAttribute ca[1];
            ca[0].id = cudaLaunchAttributeClusterDimension;
            ca[0].val.clusterDim.x = cluster;
            ca[0].val.clusterDim.y = 1;
            ca[0].val.clusterDim.z = 1;
            occ.attrs = ca;
            occ.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, k, &occ) != cudaSuccess)
                return fail(DTT_ECUDA, "dtt_fill_producer: cannot query the producer's cluster occupancy");
            const uint64_t need = (uint64_t)d->num_programs * group * producing;
            if (need > (uint64_t)clusters)
                return fail(DTT_EINVAL, "dtt_fill_producer: a paced producer needs all its %llu clusters "
                                        "resident at once (at most %d here)", (unsigned long long)need, clusters);
        } else {
            int per_sm = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, (int)threads, 0) != cudaSuccess)
                return fail(DTT_ECUDA, "dtt_fill_producer: cannot query the producer's occupancy");
            const uint64_t ctas = (uint64_t)d->num_programs * group * producing;
            if (ctas > (uint64_t)per_sm * (uint64_t)sms)
                return fail(DTT_EINVAL, "dtt_fill_producer: a paced producer needs all its %llu CTAs resident "
                                        "at once (at most %d per SM here)", (unsigned long long)ctas, per_sm);
        }
    }

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(d->num_programs * cluster * group, P, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster > 1 ? 1 : 0;
    void* args[] = {&p};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, fill_entry(d->dtype, lean), args);
    if (e != cudaSuccess) return fail(DTT_ECUDA, "dtt_fill_producer: launch failed: %s", cudaGetErrorString(e));
    return DTT_OK;
}
