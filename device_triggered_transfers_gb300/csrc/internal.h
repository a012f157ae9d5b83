// Private declarations shared by the library's translation units: error reporting, the
// copier's descriptor tables and the plan object.  Not part of the C ABI.
#pragma once

#include <cstdint>
#include <cstdio>
#include <string>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "dtt.h"

namespace dtt {

// The driver's tensor-map encoder (cuTensorMapEncodeTiled, through the runtime's entry-point
// query so that the library needs no link against libcuda); nullptr if the driver lacks it.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

// Thread-local message behind dtt_last_error().
void set_error(const char* fmt, ...);
int fail(int code, const char* fmt, ...);

#define DTT_CUDA_TRY(expr)                                                                   \
    do {                                                                                     \
        cudaError_t e_ = (expr);                                                             \
        if (e_ != cudaSuccess)                                                               \
            return ::dtt::fail(DTT_ECUDA, "%s: %s (%s:%d)", #expr, cudaGetErrorString(e_),   \
                               __FILE__, __LINE__);                                          \
    } while (0)

constexpr uint32_t kNoMap = 0xFFFFFFFFu;

// Polls of a library producer's wait for a chunk to become writable (overlapping rounds): about a
// second with the waits' back-off, after which the producer leaves its part of the chunk unwritten
// and sets DTT_DEV_EWRITABLE.
constexpr uint64_t kWritablePolls = 1ull << 22;

// One unit of copier work: a sub-window of a region (rows x row_bytes, pitch apart) at byte
// offset `off` of every buffer.  `vec` = 1 when off, row_bytes and pitch are multiples of 16.
// Bulk-copy path: `tmap` names the tensor-map shape that moves the whole window as one box
// (maps [tmap * P + q] for buffer q), with the box origin at element column x (8-byte elements)
// and row y; kNoMap: one bulk copy per row.
struct PieceDesc {
    uint64_t off;
    uint64_t pitch;
    uint64_t dst_off;           // where it lands (the same as off unless the chunk has destinations)
    uint64_t dst_pitch;
    uint32_t row_bytes;
    uint32_t rows;
    uint32_t vec;
    uint32_t tmap;
    uint32_t x;
    uint32_t y;
};

// Per global chunk: its pieces [piece_begin, piece_begin + n_pieces), the copier CTA of its
// source that takes piece 0 (`rot`), how many CTAs take part (n_part) and the source rank.
struct ChunkDesc {
    uint32_t piece_begin;
    uint32_t n_pieces;
    uint32_t rot;
    uint32_t n_part;
    uint32_t owner;
    uint32_t writers;
    uint64_t bytes;
    uint32_t peers;             // receiving ranks as a bit mask (never the owner)
    uint32_t receivers;         // popcount of peers
};

// Plan-wide device status block.
struct DevStatus {
    uint32_t misuse;            // DTT_DEV_* bits from mark_ready
    uint32_t copier_timeouts;   // copier CTAs that gave up on a gate
    uint32_t timeout_inv;       // 0xFFFFFFFF - (smallest chunk id a copier CTA gave up on); 0: none
    uint32_t bulk_timeouts;     // bulk-copy waits (mbarrier, bulk groups) that gave up
    uint32_t check_arrive;      // check_kernel CTAs done with their chunks (the last one resets it)
    uint32_t copier_exit;       // copier CTAs of this round that have finished
    uint32_t check_late;        // 1: the check gave up waiting for the copier
    uint32_t pad;
    // An early copier's decision for its round R, published by its CTA 0 for the other CTAs:
    // 2R (the host started round R: copy) or 2R + 1 (it expired or was aborted: exit).  Grows
    // with the rounds and is never reset.
    uint64_t early_go;
};

// Values of the early-copier handshake word for round R (HostStatus::go, DevStatus::early_go).
inline __host__ __device__ uint64_t early_start_value(uint32_t round) { return 2ull * round; }
inline __host__ __device__ uint64_t early_stop_value(uint32_t round) { return 2ull * round + 1; }

// A round's outcome in pinned, device-mapped host memory, written by check_kernel itself so that
// wait() needs no device-to-host copy: the status words, then `done` (the sequence number of
// the last check that finished, stored last with a system-scope release), then one flag byte per
// chunk right after the struct (0 complete, 1 short, 2 extra marks).
struct HostStatus {
    DevStatus st;
    uint32_t done;
    uint32_t pad;
    // Early-copier handshake (opts.early_copier_us): a copier launched before its round waits
    // until plan_start moves this word from the value it held at the launch (`go_prior`) to
    // early_start_value(round); if that does not happen in time, the copier moves it to
    // early_stop_value(round) itself and exits.  Both sides use a compare-and-swap at system
    // scope, so exactly one of them decides.  The host also stores the stop value to abort.
    uint64_t go;
    uint64_t pad2[2];
};

struct CopierParams {
    char* bufs[DTT_MAX_RANKS];
    char* dst[DTT_MAX_RANKS];   // where copies land: the buffers, or the destination buffers
    const CUtensorMap* tmaps;   // bulk-copy path: [shape][rank] maps of the 2D windows (or null)
    uint64_t* gates;
    const ChunkDesc* chunks;
    const PieceDesc* pieces;
    DevStatus* status;
    uint32_t cta_base[DTT_MAX_RANKS + 1];
    uint32_t first_chunk[DTT_MAX_RANKS];
    uint32_t n_chunks[DTT_MAX_RANKS];
    uint32_t P;
    uint32_t n_global;
    uint32_t round;
    uint32_t flags;
    uint64_t max_polls;
    uint32_t stage_bytes;       // bulk-copy path: bytes per shared-memory stage (>= a piece, 128-aligned)
    uint32_t stages;            // bulk-copy path: stages in the ring
    uint32_t* host_arrived;     // or null: mapped host words, word c = round once chunk c reached every peer
    // Early launch (null for a launch at plan_start): the device address of HostStatus::go, the
    // value it held when this copier was launched, and how long CTA 0 waits for the host's
    // start of the round (globaltimer ns) before it gives the round up.
    uint64_t* go_host;
    uint64_t go_prior;
    uint64_t go_wait_ns;
    dtt_group_table groups;     // the plan's chunk groups (counters == null: none)
};

struct CheckParams {
    const uint64_t* gates;
    const ChunkDesc* chunks;
    uint32_t P;
    uint32_t n_global;
    uint32_t round;
    uint32_t pending;           // 1: the next round may already be marking (overlapping rounds), so
                                // only the error word reports extra marks
    uint32_t seq;               // stored in host->done once every flag and status word is there
    uint32_t copier_ctas;       // wait until this many copier CTAs have finished (0: no copier)
    uint64_t max_polls;         // bound of that wait
    DevStatus* status;          // the round's device status; the last CTA copies it out and zeroes it
    HostStatus* host;           // device address of the mapped host block
    uint8_t* host_flags;        // device address of its flag bytes
};

// Bulk-copy copier: a ring of `stages` shared-memory stages of stage_bytes, then one mbarrier
// per stage; at most kBulkSmemMax bytes of dynamic shared memory per CTA.
constexpr size_t kBulkSmemMax = 200 * 1024;
// Shared-memory stage of the bulk-copy path: a piece, rounded up to the 128-byte alignment that
// tensor copies need.
inline uint32_t bulk_stage_bytes(uint32_t piece_bytes) { return (piece_bytes + 127u) & ~127u; }

inline size_t bulk_smem_bytes(uint32_t stage_bytes, uint32_t stages) {
    return (size_t)stage_bytes * stages + 8 * (size_t)stages;
}

// Kernel launchers (copier.cu).
cudaError_t launch_copier(const CopierParams& p, uint32_t ctas, uint32_t threads, uint32_t method,
                          cudaStream_t s);
// Completion check: flags[c] = 0 delivered, 1 short, 2 extra marks.
cudaError_t launch_check(const CheckParams& p, cudaStream_t s);
cudaError_t launch_force_open(uint64_t* gates, const ChunkDesc* chunks, uint32_t n_global,
                              uint32_t round, cudaStream_t s);
// Copy-engine transport: after every copy of chunk c (source s) has landed, one warp signals its
// arrival at each peer, the peers' group counters and s's completion word (as the SM copier does).
struct CeSignalParams {
    uint64_t* gates;
    dtt_group_table groups;
    uint32_t* host_arrived;     // or null
    uint32_t P, n_global, s, c, round, flags;
    uint32_t peers, receivers;  // the chunks' receiving ranks
    uint32_t c_end;             // the run of chunks [c, c_end) of source s, copied together
};
cudaError_t launch_ce_signal(const CeSignalParams& p, cudaStream_t s);
cudaError_t launch_consumer(const CopierParams& p, dtt_handle h, char* dst, uint64_t max_polls,
                            int32_t* status, uint32_t ctas, cudaStream_t s);

// An SM runs CTAs of one shared-memory carveout at a time: a kernel whose preferred L1/shared
// split differs from that of the copier CTAs already resident cannot start on those SMs until
// they drain, and with a copier CTA on every SM that is after the copier exits.  Every library
// kernel therefore asks for the same split, the largest shared-memory share.
constexpr int kCarveout = cudaSharedmemCarveoutMaxShared;

// Load a kernel now (lazy module loading would otherwise load it at its first launch, which can
// wait for the device to go idle) and give it the library's carveout.
template <class K>
cudaError_t prepare_kernel(K kernel) {
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, kernel);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, kCarveout);
    return e;
}

// Force-load each translation unit's kernels on the current device (see dtt_preload).
cudaError_t preload_copier_kernels();
cudaError_t copier_regs_per_thread(uint32_t method, int* regs);   // of the copier kernel for `method`
cudaError_t copier_static_smem(uint32_t method, size_t* bytes);  // its static shared memory

// What a plan's copier holds on each SM while it runs (nothing for the copy-engine transport,
// whose copies need no SM): CTAs, threads, registers (per-thread count rounded up to the
// allocation unit of 8) and shared memory including the per-CTA reservation.
struct CopierRoom {
    uint32_t ctas = 0, threads = 0;
    uint64_t regs = 0, smem = 0;
};
int plan_copier_room(const dtt_plan* p, CopierRoom* out);

// Host-buffer rounds driven from outside the plan (the all-reduce's): the plan's streams for
// copies in and out, its mapped arrival words (word c = the round of chunk c's last arrival,
// stamped by a copier launched while notify is on) and the event recorded after such a launch.
struct PlanHostIo {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    const uint32_t* arrived = nullptr;
    cudaEvent_t copier_end = nullptr;
    uint64_t piece_bytes = 0;          // opts.host_piece_bytes (0: the caller's default)
};
int plan_host_io(const dtt_plan* p, PlanHostIo* out);
// notify: the next copier launch stamps the arrival words; quiet: wait() launches no early
// copier for the next round (one launched then would not stamp them).
void plan_set_host_round(dtt_plan* p, bool notify, bool quiet);
cudaStream_t plan_copy_stream(const dtt_plan* p);   // the stream its copier runs on
cudaError_t preload_allreduce_kernels();

// The consumer GEMM (gemm.cu): D = X . W^T over one rank's gathered buffer X [rows, K] bf16,
// each 128-row block loaded once the chunk ids [c0[b], c1[b]] have arrived at that rank.
struct ConsumerLaunch {
    const void* X;
    uint64_t rows;
    const void* Wt;
    uint32_t N, K;
    char* D;
    uint64_t ldd;
    dtt_handle h;
    const uint32_t* order;
    const uint32_t* c0;
    const uint32_t* c1;
    const uint32_t* order2;     // pairs of row blocks in the order they are taken (pair form)
    const uint32_t* bgroup;     // per block: its chunk group id (block groups), or null
    uint32_t blocks;
    uint64_t max_polls;
    uint32_t* err;
    uint32_t ctas;
    uint64_t smem_budget;       // shared memory a consumer CTA can have beside the copier's CTAs
};
int launch_gemm_consumer(const ConsumerLaunch& cl, cudaStream_t stream);
cudaError_t preload_fill_kernels();
cudaError_t preload_barrier_kernels();
cudaError_t preload_gemm_kernels();
// dtt_preload() for library-internal callers: once per device, then a no-op.
int preload_once();

// Host schedule representation (schedule.cpp).
struct HostChunk {
    std::vector<dtt_region> regions;
    uint32_t writers;
    std::vector<dtt_dest> dests;   // empty: every region lands at its own offsets
    uint32_t peers = 0;            // DTT_ALL_PEERS or a bit mask of receiving ranks
};

}  // namespace dtt

struct dtt_schedule {
    std::vector<dtt::HostChunk> chunks;
};
