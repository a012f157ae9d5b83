// The host side of a triggered plan: validation, gate tables, copier descriptor tables, and the
// round state machine start -> wait -> next_round ("Triggered Plans", sections Model, The kernel
// author's contract, Gates and rounds, Requirements and limits; "Triggered SDMA Plans", API and
// Design notes).  One process drives all P virtual ranks, so the collective steps of the pages
// (create, next_round, close) are single calls here.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <cstring>
#include <new>
#include <mutex>
#include <thread>
#include <vector>

#include "internal.h"

using namespace dtt;

namespace {

// A tensor-map shape of the bulk-copy path: boxes of `inner` 8-byte elements by `rows` rows, in
// a buffer seen as rows of `pitch` bytes.  The plan encodes one map per (shape, buffer).
struct MapShape {
    uint32_t inner, rows;
    uint64_t pitch;
    bool operator==(const MapShape& o) const { return inner == o.inner && rows == o.rows && pitch == o.pitch; }
};
constexpr size_t kMaxMapShapes = 256;

// The copy-engine transport (opts.method = DTT_COPY_ENGINE): a proxy thread of the plan stands in
// for the pages' pre-armed copy-engine queues.  start() hands it a round; it polls the mapped gate
// words in each source's schedule order and issues each open chunk's copies on the (source, peer)
// streams, then the chunk's signal kernel after joining them.
struct CeProxy {
    std::thread thread;
    std::mutex mu;
    std::condition_variable cv;
    bool stop = false;
    bool busy = false;                  // issuing `round`
    uint32_t round = 0;
    uint32_t queued = 0;                // overlapping rounds: the round to issue after `round` (0: none)
    uint32_t issued = 0;                // the last round whose chunks were all issued (or given up)
    std::atomic<bool> open_all{false};  // close() in mid-round: every chunk goes as it stands
    int rc_of[2] = {DTT_OK, DTT_OK};    // per round parity; DTT_ETIMEDOUT: a gate stayed closed past the bound
    uint32_t stuck_chunk = 0;
    uint32_t* h_ready = nullptr;        // pinned, mapped: word c = round of chunk c's last opening
    uint32_t* h_ready_dev = nullptr;
    std::vector<cudaStream_t> streams;  // [s * P + q]
    std::vector<cudaEvent_t> ev;        // [s * P + q]
    std::vector<uint32_t> reg_begin;    // chunk c's regions: regs[reg_begin[c] .. reg_begin[c + 1])
    std::vector<dtt_region> regs;
    std::vector<dtt_dest> dests;        // where each region lands
};

}  // namespace

struct dtt_plan {
    uint32_t P = 0;
    uint64_t buf_bytes = 0;
    char* bufs[DTT_MAX_RANKS] = {};
    char* dst[DTT_MAX_RANKS] = {};    // where copies land: bufs, or the separate destination buffers
    uint64_t dst_bytes = 0;
    bool separate_dst = false;
    bool other_dests = false;         // some chunk lands elsewhere or goes to only some peers
    uint32_t* d_peer_masks = nullptr; // per global chunk, when other_dests
    dtt_plan_opts opts{};
    int device = 0;

    uint32_t n_global = 0;
    uint32_t first_chunk[DTT_MAX_RANKS] = {};
    uint32_t n_chunks[DTT_MAX_RANKS] = {};
    std::vector<ChunkDesc> chunks;
    std::vector<PieceDesc> pieces;
    std::vector<uint32_t> writers;
    std::vector<uint32_t> peer_masks; // receivers of each global chunk
    std::vector<MapShape> shapes;     // bulk-copy path: the tensor-map shapes of the 2D windows

    uint32_t copier_ctas = 0;
    uint32_t copier_threads = 0;
    uint32_t cta_base[DTT_MAX_RANKS + 1] = {};

    uint64_t* d_gates = nullptr;
    uint32_t* d_writers = nullptr;
    ChunkDesc* d_chunks = nullptr;
    PieceDesc* d_pieces = nullptr;
    CUtensorMap* d_tmaps = nullptr;   // [shape][rank]
    DevStatus* d_status = nullptr;    // [2]: one block per round parity (status_of), so that a
                                      // pending round's copier and check keep their own words
    HostStatus* h_status = nullptr;   // pinned, mapped: check_kernel writes the round's outcome here
    HostStatus* h_status_dev = nullptr;   // its device address
    uint8_t* h_flags = nullptr;       // the flag bytes right after it
    uint32_t wait_seq = 0;            // sequence number of the last check launched

    // host-buffer rounds (dtt_allgather_host): the copier stamps each chunk's arrival into
    // mapped host words, the host copies the gathered bytes back as they arrive
    uint32_t* h_arrived = nullptr;    // pinned, mapped: [n_global], word c = round of c's last arrival
    uint32_t* h_arrived_dev = nullptr;
    bool notify_host = false;         // the next copier launch stamps h_arrived
    cudaEvent_t ev_copier_end = nullptr;   // after that launch: the copier has exited
    cudaEvent_t ev_h2d = nullptr;
    std::vector<cudaEvent_t> ev_pieces;   // one per host-to-device piece of the output rank's slice
    std::vector<cudaEvent_t> ev_free;     // dtt_allgather_host_rounds: events not in use
    cudaStream_t h2d_stream = nullptr;
    cudaStream_t d2h_stream = nullptr;

    // chunk groups (dtt_plan_define_groups): the device table and its arrays, and the block size
    // when they were defined by position (dtt_plan_define_block_groups; 0 otherwise)
    uint32_t n_groups = 0;
    std::vector<uint32_t> group_size;
    std::vector<uint32_t> block_group;   // block -> group id (UINT32_MAX: no chunk touches it)
    uint64_t group_block_bytes = 0;
    uint64_t* d_group_counters = nullptr;
    uint32_t* d_group_arrays = nullptr;   // size, chunk_off, chunk_ids back to back

    // consumer GEMM: per 128-row block of one rank's buffer seen as [rows, K], the order the
    // blocks are taken in and the chunk ids that cover each block (device, built on first use)
    uint32_t cons_rank = UINT32_MAX, cons_K = 0, cons_blocks = 0, cons_cap = 0;
    bool cons_grouped = false;
    uint32_t* d_cons = nullptr;       // [3][blocks] + [blocks / 2 + 1]: order, c0, c1, order2

    cudaStream_t copy_stream = nullptr;
    bool own_copy_stream = false;
    cudaStream_t aux_stream = nullptr;
    cudaEvent_t ev_producer = nullptr;
    cudaStream_t producer_stream = nullptr;

    int state = DTT_PLAN_PREPARED;
    uint32_t round = 1;
    bool copier_launched = false;   // this round's copier is on the copy stream
    bool live_round = false;        // this round was started and its check has not run yet

    // opts.overlap: the round in flight behind the current one (0: none), whether its copier was
    // launched, and an event after its producers (its check follows that event, not the
    // producers of the round after it)
    uint32_t pending = 0;
    bool pending_copier = false;
    cudaEvent_t ev_pending = nullptr;
    CeProxy* ce = nullptr;          // opts.method == DTT_COPY_ENGINE

    // opts.early_copier_us: wait() launches the next round's copier behind this round's, and
    // start() claims it through HostStatus::go (see CopierParams::go_host).
    bool host_atomics = false;      // the device and the host can share atomics on mapped memory
    bool early_pending = false;     // an early copier for round early_round awaits its claim
    bool early_launched = false;    // an early copier was ever launched (close drains the copy stream)
    bool suppress_early = false;    // inside dtt_allgather_host: its rounds stamp arrivals for the host
    uint32_t early_round = 0;
    uint64_t go_shadow = 0;         // the value HostStatus::go holds (the host sees every change)
    uint64_t early_launches = 0, early_claims = 0, early_expired = 0, early_aborts = 0;

    // Plans sharing a copy stream ("Triggered Plans", The kernel author's contract: CLOSING):
    // the order of this plan's last copier launch among all plans, and an event after that
    // copier, recorded when another plan uses the same stream.
    uint64_t launch_seq = 0;
    cudaEvent_t ev_done = nullptr;
    bool done_valid = false;

    // opts.time_copier: a ring of event pairs around the copier launches, read back lazily (when
    // a pair comes round again, or in dtt_plan_stats) so that timing adds no wait to a round
    static constexpr uint32_t kTimeRing = 64;
    cudaEvent_t ev_copier[kTimeRing][2] = {};
    uint64_t timed_launches = 0, timed_read = 0;
    double copier_ms_total = 0, copier_ms_last = 0;
};

namespace {

struct RegionRef {
    uint64_t lo, hi;     // byte extent [lo, hi)
    uint32_t rank;
    const dtt_region* reg;
};

// Do two regions share a byte?  Both are sorted row sets (pitch > 0 or a single row), so a
// merge over their rows decides it exactly.
bool regions_intersect(const dtt_region& a, const dtt_region& b) {
    uint64_t i = 0, j = 0;
    while (i < a.rows && j < b.rows) {
        const uint64_t alo = a.offset + i * a.pitch, ahi = alo + a.row_bytes;
        const uint64_t blo = b.offset + j * b.pitch, bhi = blo + b.row_bytes;
        if (alo < bhi && blo < ahi) return true;
        if (ahi <= bhi) ++i; else ++j;
    }
    return false;
}

void stop_ce(dtt_plan* p);

void free_device(dtt_plan* p) {
    stop_ce(p);
    cudaFree(p->d_gates);
    cudaFree(p->d_writers);
    cudaFree(p->d_chunks);
    cudaFree(p->d_pieces);
    cudaFree(p->d_tmaps);
    cudaFree(p->d_status);
    cudaFreeHost(p->h_status);
    if (p->ev_producer) cudaEventDestroy(p->ev_producer);
    if (p->ev_pending) cudaEventDestroy(p->ev_pending);
    p->ev_pending = nullptr;
    if (p->ev_done) cudaEventDestroy(p->ev_done);
    p->ev_done = nullptr;
    if (p->ev_copier_end) cudaEventDestroy(p->ev_copier_end);
    if (p->ev_h2d) cudaEventDestroy(p->ev_h2d);
    for (cudaEvent_t e : p->ev_pieces) cudaEventDestroy(e);
    p->ev_pieces.clear();
    for (cudaEvent_t e : p->ev_free) cudaEventDestroy(e);
    p->ev_free.clear();
    if (p->d2h_stream) cudaStreamDestroy(p->d2h_stream);
    if (p->h2d_stream) cudaStreamDestroy(p->h2d_stream);
    p->h2d_stream = nullptr;
    if (p->h_arrived) cudaFreeHost(p->h_arrived);
    if (p->d_cons) cudaFree(p->d_cons);
    p->d_cons = nullptr;
    cudaFree(p->d_group_counters);
    cudaFree(p->d_group_arrays);
    cudaFree(p->d_peer_masks);
    p->d_peer_masks = nullptr;
    p->d_group_counters = nullptr;
    p->d_group_arrays = nullptr;
    p->ev_copier_end = nullptr;
    p->ev_h2d = nullptr;
    p->d2h_stream = nullptr;
    p->h_arrived = nullptr;
    p->h_arrived_dev = nullptr;
    for (auto& pair : p->ev_copier)
        for (cudaEvent_t& e : pair) {
            if (e) cudaEventDestroy(e);
            e = nullptr;
        }
    if (p->aux_stream) cudaStreamDestroy(p->aux_stream);
    if (p->own_copy_stream && p->copy_stream) cudaStreamDestroy(p->copy_stream);
    p->d_gates = nullptr;
    p->d_writers = nullptr;
    p->d_chunks = nullptr;
    p->d_pieces = nullptr;
    p->d_tmaps = nullptr;
    p->d_status = nullptr;
    p->h_flags = nullptr;
    p->h_status = nullptr;
    p->h_status_dev = nullptr;
    p->ev_producer = nullptr;
    p->aux_stream = nullptr;
    p->copy_stream = nullptr;
}

struct CutCtx {
    uint64_t piece_bytes;
    uint64_t buf_bytes;
    bool bases_aligned;
    bool tensor;                      // bulk-copy path: 2D windows as tensor-map boxes
    std::vector<MapShape>* shapes;
};

// The shape index of a box, adding the shape if it is new; kNoMap when the table is full.
uint32_t shape_of(const MapShape& m, std::vector<MapShape>* shapes) {
    for (size_t i = 0; i < shapes->size(); ++i)
        if ((*shapes)[i] == m) return (uint32_t)i;
    if (shapes->size() >= kMaxMapShapes) return kNoMap;
    shapes->push_back(m);
    return (uint32_t)(shapes->size() - 1);
}

// Can this 2D window move as tensor-map boxes?  Rows of 16-byte multiples up to 2 KiB (256
// elements of 8 bytes, the widest box), 16-byte aligned columns (a box's x coordinate must be),
// and every row of the window inside the buffer's whole rows of `pitch` bytes.
bool tensor_window(const dtt_region& r, const CutCtx& cx) {
    if (!cx.tensor || !cx.bases_aligned || r.rows < 2 || r.pitch <= r.row_bytes) return false;
    const uint64_t col = r.offset % r.pitch, row0 = r.offset / r.pitch;
    return r.row_bytes % 16 == 0 && r.row_bytes <= 2048 && r.row_bytes < cx.piece_bytes &&
           r.pitch % 16 == 0 && col % 16 == 0 && col + r.row_bytes <= r.pitch &&
           (row0 + r.rows) * r.pitch <= cx.buf_bytes && r.pitch / 8 <= 0xFFFFFFFFull &&
           cx.buf_bytes / r.pitch <= 0xFFFFFFFFull && (r.pitch >> 40) == 0;
}

// Cut one region into copier pieces of at most piece_bytes: whole rows when a row fits,
// otherwise column pieces of single rows.  Each piece lands at the matching rows and columns of
// the region's destination `d`.  On the bulk-copy path a 2D window's pieces of whole rows (at
// most 256 rows each, the tallest box) are tensor-map boxes when the window allows it and lands
// at its own offsets (a box is stored through the same map shape it was loaded with).
void cut_region(const dtt_region& r, const dtt_dest& d, const CutCtx& cx, std::vector<PieceDesc>* out) {
    const uint64_t piece_bytes = cx.piece_bytes;
    const bool same_place = d.offset == r.offset && (r.rows <= 1 || d.pitch == r.pitch);
    auto push = [&](uint64_t off, uint64_t doff, uint64_t rb, uint64_t rows, uint64_t pitch, uint64_t dpitch,
                    uint32_t tmap) {
        PieceDesc pc{};
        pc.off = off;
        pc.pitch = rows > 1 ? pitch : rb;
        pc.dst_off = doff;
        pc.dst_pitch = rows > 1 ? dpitch : rb;
        pc.row_bytes = (uint32_t)rb;
        pc.rows = (uint32_t)rows;
        pc.vec = cx.bases_aligned && (off % 16 == 0) && (rb % 16 == 0) && (rows <= 1 || pitch % 16 == 0) &&
                 (doff % 16 == 0) && (rows <= 1 || dpitch % 16 == 0);
        pc.tmap = tmap;
        if (tmap != kNoMap) {
            pc.x = (uint32_t)((off % pitch) / 8);
            pc.y = (uint32_t)(off / pitch);
        }
        out->push_back(pc);
    };
    if (r.rows == 0 || r.row_bytes == 0) return;
    if (r.row_bytes >= piece_bytes) {
        for (uint64_t i = 0; i < r.rows; ++i)
            for (uint64_t c = 0; c < r.row_bytes; c += piece_bytes)
                push(r.offset + i * r.pitch + c, d.offset + i * d.pitch + c, std::min(piece_bytes, r.row_bytes - c), 1,
                     0, 0, kNoMap);
    } else {
        const bool tensor = same_place && tensor_window(r, cx);
        uint64_t per = std::max<uint64_t>(1, piece_bytes / r.row_bytes);
        if (tensor) per = std::min<uint64_t>(per, 256);
        for (uint64_t i = 0; i < r.rows; i += per) {
            const uint64_t rows = std::min(per, r.rows - i);
            const uint32_t tmap = tensor && rows > 1
                ? shape_of(MapShape{(uint32_t)(r.row_bytes / 8), (uint32_t)rows, r.pitch}, cx.shapes)
                : kNoMap;
            push(r.offset + i * r.pitch, d.offset + i * d.pitch, r.row_bytes, rows, r.pitch, d.pitch, tmap);
        }
    }
}

CopierParams copier_params(const dtt_plan* p, uint32_t round);

// The device status block of round `round` (rounds of one parity share one; at most two rounds
// are in flight, and a round's check clears its block before the round two later can start).
DevStatus* status_of(const dtt_plan* p, uint32_t round) { return p->d_status + (round & 1u); }

// Add the timed copier launches up to `upto` (in launch order) to the copier statistics.
int read_copier_times(dtt_plan* p, uint64_t upto) {
    for (; p->timed_read < upto; ++p->timed_read) {
        cudaEvent_t* pair = p->ev_copier[p->timed_read % dtt_plan::kTimeRing];
        float ms = 0;
        cudaError_t e = cudaEventElapsedTime(&ms, pair[0], pair[1]);
        if (e == cudaErrorNotReady) {
            DTT_CUDA_TRY(cudaEventSynchronize(pair[1]));
            e = cudaEventElapsedTime(&ms, pair[0], pair[1]);
        }
        DTT_CUDA_TRY(e);
        p->copier_ms_last = ms;
        p->copier_ms_total += ms;
    }
    return DTT_OK;
}

// ---- plans sharing the device -------------------------------------------------------------
// Live plans (created and not yet released by dtt_plan_close) and closed plans whose device
// memory is still held: cudaFree waits for the whole device, so memory is released only while
// no plan's copier can be spinning on a gate (a spinning copier ends only when its producer
// runs or its polls run out).
std::mutex g_plans_mu;
std::vector<dtt_plan*> g_live;
std::vector<dtt_plan*> g_retired;
uint64_t g_launch_seq = 0;

bool may_spin(const dtt_plan* q) {
    return ((q->state == DTT_PLAN_RUNNING || q->state == DTT_PLAN_CLOSING) && q->copier_launched) ||
           q->early_pending || (q->pending && q->pending_copier) || (q->live_round && q->copier_launched);
}

// Is p's copier queued behind an earlier plan's copier on the same stream that has not finished?
bool blocked_behind(const dtt_plan* p) {
    for (const dtt_plan* q : g_live)
        if (q != p && q->copy_stream == p->copy_stream && q->launch_seq < p->launch_seq && may_spin(q) &&
            !(q->done_valid && cudaEventQuery(q->ev_done) == cudaSuccess))
            return true;
    return false;
}

// Free the device memory of retired plans once no copier can be spinning.  Holds g_plans_mu.
void reap_locked() {
    for (const dtt_plan* q : g_live)
        if (may_spin(q)) return;
    for (dtt_plan* q : g_retired) {
        free_device(q);
        delete q;
    }
    g_retired.clear();
}

// Launch this round's copier on the copy stream (bracketed by a pair of timing events when asked).
int launch_round_copier(dtt_plan* p) {
    bool shared = false;
    {
        std::lock_guard<std::mutex> lock(g_plans_mu);
        p->launch_seq = ++g_launch_seq;
        for (dtt_plan* q : g_live) {
            if (q == p || q->copy_stream != p->copy_stream) continue;
            shared = true;
            if (may_spin(q) && !q->done_valid) {     // mark where the earlier copier ends
                DTT_CUDA_TRY(cudaEventRecord(q->ev_done, p->copy_stream));
                q->done_valid = true;
            }
        }
    }
    p->done_valid = false;
    cudaEvent_t* pair = nullptr;
    if (p->opts.time_copier) {
        if (p->timed_launches - p->timed_read == dtt_plan::kTimeRing) {   // the oldest pair is reused
            const int rc = read_copier_times(p, p->timed_read + 1);
            if (rc != DTT_OK) return rc;
        }
        pair = p->ev_copier[p->timed_launches % dtt_plan::kTimeRing];
        DTT_CUDA_TRY(cudaEventRecord(pair[0], p->copy_stream));
    }
    DTT_CUDA_TRY(launch_copier(copier_params(p, p->round), p->copier_ctas, p->copier_threads, p->opts.method,
                               p->copy_stream));
    if (pair) {
        DTT_CUDA_TRY(cudaEventRecord(pair[1], p->copy_stream));
        ++p->timed_launches;
    }
    if (shared) {
        DTT_CUDA_TRY(cudaEventRecord(p->ev_done, p->copy_stream));
        p->done_valid = true;
    }
    if (p->notify_host) DTT_CUDA_TRY(cudaEventRecord(p->ev_copier_end, p->copy_stream));
    p->copier_launched = true;
    return DTT_OK;
}

// The plan's group table with device addresses (all null when it has no groups).
dtt_group_table group_table(const dtt_plan* p) {
    dtt_group_table t{};
    if (!p->n_groups) return t;
    t.counters = p->d_group_counters;
    t.size = p->d_group_arrays;
    t.chunk_off = p->d_group_arrays + (size_t)p->P * p->n_groups;
    t.chunk_ids = p->d_group_arrays + (size_t)p->P * p->n_groups + (p->n_global + 1);
    t.n_groups = p->n_groups;
    return t;
}

dtt_handle make_handle(const dtt_plan* p, uint32_t r) {
    dtt_handle h{};
    h.gates = p->d_gates;
    h.writers = p->d_writers;
    h.status = &status_of(p, p->round)->misuse;
    h.round = p->round;
    h.rank = r;
    h.P = p->P;
    h.n_global = p->n_global;
    h.first_chunk = p->first_chunk[r];
    h.n_chunks = p->n_chunks[r];
    h.flags = (p->opts.timestamps ? DTT_HANDLE_TIMESTAMPS : 0u) | (p->opts.overlap ? DTT_HANDLE_OVERLAP : 0u);
    h.groups = group_table(p);
    h.peer_masks = p->d_peer_masks;
    h.host_ready = p->ce ? p->ce->h_ready_dev : nullptr;
    return h;
}

CopierParams copier_params(const dtt_plan* p, uint32_t round) {
    CopierParams cp{};
    for (uint32_t r = 0; r < p->P; ++r) {
        cp.bufs[r] = p->bufs[r];
        cp.dst[r] = p->dst[r];
        cp.first_chunk[r] = p->first_chunk[r];
        cp.n_chunks[r] = p->n_chunks[r];
    }
    for (uint32_t r = 0; r <= p->P; ++r) cp.cta_base[r] = p->cta_base[r];
    cp.gates = p->d_gates;
    cp.chunks = p->d_chunks;
    cp.pieces = p->d_pieces;
    cp.status = status_of(p, round);
    cp.P = p->P;
    cp.n_global = p->n_global;
    cp.round = round;
    cp.flags = p->opts.timestamps ? DTT_HANDLE_TIMESTAMPS : 0u;
    cp.max_polls = p->opts.max_polls;
    cp.stage_bytes = bulk_stage_bytes(p->opts.piece_bytes);
    cp.tmaps = p->d_tmaps;
    cp.host_arrived = p->notify_host ? p->h_arrived_dev : nullptr;
    cp.stages = p->opts.stages;
    cp.groups = group_table(p);
    return cp;
}

// ---- the early copier (opts.early_copier_us) ------------------------------------------------
// Does another live plan use p's copy stream?  A copier launched early would hold that stream
// until p's next start, so shared streams launch at start as before.
bool stream_shared(const dtt_plan* p) {
    std::lock_guard<std::mutex> lock(g_plans_mu);
    for (const dtt_plan* q : g_live)
        if (q != p && q->copy_stream == p->copy_stream) return true;
    return false;
}

bool early_allowed(const dtt_plan* p) {
    return p->opts.early_copier_us && p->host_atomics && p->n_global && !p->opts.time_copier &&
           p->opts.method != DTT_COPY_ENGINE && !p->opts.overlap &&
           p->opts.deferred_copier != 1 && !p->suppress_early && p->round < 0xFFFFFFFFu &&
           !stream_shared(p);
}

uint64_t* go_word(dtt_plan* p) { return &p->h_status->go; }

bool cas_go(dtt_plan* p, uint64_t* expected, uint64_t desired) {
    return __atomic_compare_exchange_n(go_word(p), expected, desired, false, __ATOMIC_ACQ_REL,
                                       __ATOMIC_ACQUIRE);
}

// Launch round p->round + 1's copier now, on the copy stream behind this round's.
int launch_early(dtt_plan* p) {
    CopierParams cp = copier_params(p, p->round + 1);
    cp.go_host = &p->h_status_dev->go;
    cp.go_prior = p->go_shadow;
    cp.go_wait_ns = (uint64_t)p->opts.early_copier_us * 1000;
    DTT_CUDA_TRY(launch_copier(cp, p->copier_ctas, p->copier_threads, p->opts.method, p->copy_stream));
    p->early_pending = true;
    p->early_launched = true;
    p->early_round = p->round + 1;
    ++p->early_launches;
    return DTT_OK;
}

// Take a pending early copier's round away from it: it exits without copying (if it has not
// already given the round up itself).
void abort_early(dtt_plan* p) {
    if (!p->early_pending) return;
    uint64_t expected = p->go_shadow;
    const uint64_t stop = early_stop_value(p->early_round);
    if (cas_go(p, &expected, stop)) {
        p->go_shadow = stop;
        ++p->early_aborts;
    } else {
        p->go_shadow = expected;      // it had given the round up already
        ++p->early_expired;
    }
    p->early_pending = false;
}

// start(): claim the pending early copier for the current round.  True when it will copy this
// round; false when it had already given the round up (then a fresh copier is needed).
bool claim_early(dtt_plan* p) {
    if (!p->early_pending) return false;
    p->early_pending = false;
    uint64_t expected = p->go_shadow;
    const uint64_t start = early_start_value(p->round);
    if (cas_go(p, &expected, start)) {
        p->go_shadow = start;
        ++p->early_claims;
        return true;
    }
    p->go_shadow = expected;          // early_stop_value(round): it expired
    ++p->early_expired;
    return false;
}

// ---- the copy-engine transport (opts.method = DTT_COPY_ENGINE) -----------------------------------
// Chunk c's bytes as one contiguous range (source offset, destination offset, length), or a zero
// length when its regions are not one contiguous range on both sides.
struct CeRange {
    uint64_t src, dst, len;
};

CeRange ce_range(const CeProxy& ce, uint32_t c) {
    if (ce.reg_begin[c + 1] - ce.reg_begin[c] != 1) return {0, 0, 0};
    const dtt_region& r = ce.regs[ce.reg_begin[c]];
    const dtt_dest& d = ce.dests[ce.reg_begin[c]];
    if (r.rows != 1 && (r.pitch != r.row_bytes || d.pitch != r.row_bytes)) return {0, 0, 0};
    return {r.offset, d.offset, r.rows * r.row_bytes};
}

// Issue the run of chunks [c, c_end) of source s (one chunk, or consecutive chunks whose bytes
// follow each other on both sides, so that one copy per peer moves them all): every region to
// every peer on the (s, q) queue, then -- once all of them have landed (the other queues'
// events joined onto the last one) -- one signal kernel for the run.
int ce_issue(dtt_plan* p, uint32_t s, uint32_t c, uint32_t c_end, uint32_t round) {
    CeProxy& ce = *p->ce;
    const uint32_t P = p->P;
    uint32_t last = UINT32_MAX;
    const uint32_t peers = p->chunks[c].peers;
    CeRange run{0, 0, 0};
    if (c_end > c + 1) {
        run = ce_range(ce, c);
        run.len = ce_range(ce, c_end - 1).src + ce_range(ce, c_end - 1).len - run.src;
    }
    for (uint32_t q = 0; q < P; ++q) {
        if (!((peers >> q) & 1u)) continue;
        cudaStream_t st = ce.streams[s * P + q];
        if (run.len) {
            DTT_CUDA_TRY(cudaMemcpyAsync(p->dst[q] + run.dst, p->bufs[s] + run.src, run.len,
                                         cudaMemcpyDeviceToDevice, st));
        } else {
            for (uint32_t i = ce.reg_begin[c]; i < ce.reg_begin[c_end]; ++i) {
                const dtt_region& r = ce.regs[i];
                const dtt_dest& d = ce.dests[i];
                if (r.rows == 0 || r.row_bytes == 0) continue;
                if (r.rows == 1)
                    DTT_CUDA_TRY(cudaMemcpyAsync(p->dst[q] + d.offset, p->bufs[s] + r.offset, r.row_bytes,
                                                 cudaMemcpyDeviceToDevice, st));
                else
                    DTT_CUDA_TRY(cudaMemcpy2DAsync(p->dst[q] + d.offset, d.pitch, p->bufs[s] + r.offset, r.pitch,
                                                   r.row_bytes, r.rows, cudaMemcpyDeviceToDevice, st));
            }
        }
        last = q;
    }
    if (last == UINT32_MAX) return DTT_OK;        // no receivers: nothing to copy or signal
    cudaStream_t sl = ce.streams[s * P + last];
    for (uint32_t q = 0; q < P; ++q) {
        if (q == last || !((peers >> q) & 1u)) continue;
        DTT_CUDA_TRY(cudaEventRecord(ce.ev[s * P + q], ce.streams[s * P + q]));
        DTT_CUDA_TRY(cudaStreamWaitEvent(sl, ce.ev[s * P + q], 0));
    }
    CeSignalParams sp{};
    sp.gates = p->d_gates;
    sp.groups = group_table(p);
    sp.host_arrived = nullptr;
    sp.P = P;
    sp.n_global = p->n_global;
    sp.s = s;
    sp.c = c;
    sp.c_end = c_end;
    sp.round = round;
    sp.flags = p->opts.timestamps ? DTT_HANDLE_TIMESTAMPS : 0u;
    sp.peers = peers;
    sp.receivers = p->chunks[c].receivers;
    DTT_CUDA_TRY(launch_ce_signal(sp, sl));
    return DTT_OK;
}

// May chunk c join the run ending with chunk c - 1 of the same source: the same receivers, and
// its bytes right after the run's on both sides?  Runs stop at kCeRunBytes, so that the first
// chunk of a run is not signalled too long after it landed.
constexpr uint64_t kCeRunBytes = 64ull << 20;

bool ce_joins(const dtt_plan* p, const CeProxy& ce, uint32_t c, uint64_t run_bytes) {
    if (p->chunks[c].peers != p->chunks[c - 1].peers) return false;
    const CeRange a = ce_range(ce, c - 1), b = ce_range(ce, c);
    return a.len && b.len && b.src == a.src + a.len && b.dst == a.dst + a.len && run_bytes + b.len <= kCeRunBytes;
}

// One round on the proxy thread: every source's chunks in schedule order, each as soon as its
// gate's host word shows the round.  Gives up when no gate has opened for max_polls x 256 ns
// (about a second at the default), leaving the rest unsent for wait() to report.
int ce_run_round(dtt_plan* p, uint32_t round) {
    CeProxy& ce = *p->ce;
    const uint32_t P = p->P;
    uint32_t next[DTT_MAX_RANKS], end[DTT_MAX_RANKS];
    uint64_t remaining = 0;
    for (uint32_t s = 0; s < P; ++s) {
        next[s] = p->first_chunk[s];
        end[s] = p->first_chunk[s] + p->n_chunks[s];
        remaining += p->n_chunks[s];
    }
    const auto bound = std::chrono::nanoseconds(256 * std::max<uint64_t>(p->opts.max_polls, 1));
    auto last_progress = std::chrono::steady_clock::now();
    for (uint64_t spin = 0; remaining; ++spin) {
        bool progress = false;
        for (uint32_t s = 0; s < P; ++s) {
            while (next[s] < end[s]) {
                const uint32_t c = next[s];
                auto is_open = [&](uint32_t x) {
                    return __atomic_load_n(&ce.h_ready[x], __ATOMIC_ACQUIRE) >= round ||
                           ce.open_all.load(std::memory_order_acquire);
                };
                if (!is_open(c)) break;           // head of line: this source's later chunks wait
                // the open chunks right behind it whose bytes follow on go in the same copies
                uint32_t c_end = c + 1;
                uint64_t run_bytes = ce_range(ce, c).len;
                while (c_end < end[s] && is_open(c_end) && ce_joins(p, ce, c_end, run_bytes)) {
                    run_bytes += ce_range(ce, c_end).len;
                    ++c_end;
                }
                const int rc = ce_issue(p, s, c, c_end, round);
                if (rc != DTT_OK) return rc;
                remaining -= c_end - c;
                next[s] = c_end;
                progress = true;
            }
        }
        if (progress) {
            last_progress = std::chrono::steady_clock::now();
        } else if ((spin & 63) == 63) {
            if (std::chrono::steady_clock::now() - last_progress > bound) {
                uint32_t stuck = UINT32_MAX;
                for (uint32_t s = 0; s < P; ++s)
                    if (next[s] < end[s]) stuck = std::min(stuck, next[s]);
                ce.stuck_chunk = stuck;
                return fail(DTT_ETIMEDOUT, "copy-engine proxy: chunk %u's gate stayed closed", stuck);
            }
            std::this_thread::yield();
        }
    }
    return DTT_OK;
}

void ce_main(dtt_plan* p) {
    CeProxy& ce = *p->ce;
    int dev = p->device;
    cudaSetDevice(dev);
    for (;;) {
        uint32_t round;
        {
            std::unique_lock<std::mutex> lock(ce.mu);
            ce.cv.wait(lock, [&] { return ce.stop || ce.busy; });
            if (ce.stop) return;
            round = ce.round;
        }
        const int rc = ce_run_round(p, round);
        {
            std::lock_guard<std::mutex> lock(ce.mu);
            ce.rc_of[round & 1u] = rc;
            ce.issued = round;
            if (ce.queued) {                // the next round was started behind this one
                ce.round = ce.queued;
                ce.queued = 0;
            } else {
                ce.busy = false;
            }
        }
        ce.cv.notify_all();
    }
}

// Set up the proxy: the regions of every chunk, the queues, the mapped gate words and the thread.
int start_ce(dtt_plan* p, const dtt_schedule* const* scheds) {
    p->ce = new (std::nothrow) CeProxy();
    if (!p->ce) return fail(DTT_ENOMEM, "dtt_plan_create: out of memory");
    CeProxy& ce = *p->ce;
    const uint32_t P = p->P;
    ce.reg_begin.push_back(0);
    for (uint32_t r = 0; r < P; ++r) {
        const dtt_schedule* sc = scheds ? scheds[r] : nullptr;
        if (!sc) continue;
        for (const HostChunk& ch : sc->chunks) {
            ce.regs.insert(ce.regs.end(), ch.regions.begin(), ch.regions.end());
            for (size_t i = 0; i < ch.regions.size(); ++i)
                ce.dests.push_back(ch.dests.empty() ? dtt_dest{ch.regions[i].offset, ch.regions[i].pitch} : ch.dests[i]);
            ce.reg_begin.push_back((uint32_t)ce.regs.size());
        }
    }
    const size_t words = std::max<size_t>(1, p->n_global);
    DTT_CUDA_TRY(cudaHostAlloc(&ce.h_ready, words * sizeof(uint32_t), cudaHostAllocMapped | cudaHostAllocPortable));
    for (size_t c = 0; c < words; ++c) ce.h_ready[c] = p->round - 1;   // as after the rounds before
    DTT_CUDA_TRY(cudaHostGetDevicePointer(reinterpret_cast<void**>(&ce.h_ready_dev), ce.h_ready, 0));
    ce.streams.assign((size_t)P * P, nullptr);
    ce.ev.assign((size_t)P * P, nullptr);
    for (uint32_t s = 0; s < P; ++s)
        for (uint32_t q = 0; q < P; ++q) {
            if (q == s) continue;
            DTT_CUDA_TRY(cudaStreamCreateWithFlags(&ce.streams[s * P + q], cudaStreamNonBlocking));
            DTT_CUDA_TRY(cudaEventCreateWithFlags(&ce.ev[s * P + q], cudaEventDisableTiming));
        }
    try {
        ce.thread = std::thread(ce_main, p);
    } catch (...) {
        return fail(DTT_ENOMEM, "dtt_plan_create: cannot start the copy-engine proxy thread");
    }
    return DTT_OK;
}

void stop_ce(dtt_plan* p) {
    if (!p->ce) return;
    CeProxy& ce = *p->ce;
    if (ce.thread.joinable()) {
        {
            std::lock_guard<std::mutex> lock(ce.mu);
            ce.stop = true;
        }
        ce.cv.notify_all();
        ce.thread.join();
    }
    for (cudaStream_t st : ce.streams)
        if (st) cudaStreamDestroy(st);
    for (cudaEvent_t e : ce.ev)
        if (e) cudaEventDestroy(e);
    if (ce.h_ready) cudaFreeHost(ce.h_ready);
    delete p->ce;
    p->ce = nullptr;
}

// Wait until the proxy has issued (or given up on) round `round`'s chunks (0: every round handed
// to it), then order stream `after` after every queue (or, with no stream, wait for them).
// Returns the proxy's status for that round.
int ce_join(dtt_plan* p, cudaStream_t after, uint32_t round) {
    CeProxy& ce = *p->ce;
    int rc;
    {
        std::unique_lock<std::mutex> lock(ce.mu);
        ce.cv.wait(lock, [&] { return !ce.busy || (round && ce.issued >= round); });
        rc = ce.rc_of[(round ? round : ce.issued) & 1u];
    }
    for (uint32_t s = 0; s < p->P; ++s)
        for (uint32_t q = 0; q < p->P; ++q) {
            if (q == s) continue;
            DTT_CUDA_TRY(cudaEventRecord(ce.ev[s * p->P + q], ce.streams[s * p->P + q]));
            if (after) DTT_CUDA_TRY(cudaStreamWaitEvent(after, ce.ev[s * p->P + q], 0));
            else DTT_CUDA_TRY(cudaEventSynchronize(ce.ev[s * p->P + q]));
        }
    return rc;
}

// Does rank q receive a chunk of rank r with peer mask `peers`?
inline bool receives(uint32_t peers, uint32_t r, uint32_t q) {
    return q != r && (peers == 0 || ((peers >> q) & 1u));
}

// Destinations ("Triggered Plans", Not supported yet, "Other destinations", as this library reads
// it): every copy lands inside its receiving buffer, no two copies land on the same bytes of one
// buffer, and in place no copy lands on bytes its receiving rank itself sends.
int validate_destinations(const dtt_plan* p, const dtt_schedule* const* scheds) {
    const uint32_t P = p->P;
    const uint64_t nbytes = p->separate_dst ? p->dst_bytes : p->buf_bytes;
    std::vector<dtt_region> landed;   // one buffer's landed (and, in place, sent) windows
    std::vector<RegionRef> refs;
    for (uint32_t q = 0; q < P; ++q) {
        landed.clear();
        refs.clear();
        std::vector<uint32_t> who;    // rank of each entry: q itself for its sent windows
        if (!p->separate_dst && scheds && scheds[q])
            for (const HostChunk& ch : scheds[q]->chunks)
                for (const dtt_region& reg : ch.regions) {
                    landed.push_back(reg);
                    who.push_back(q);
                }
        for (uint32_t r = 0; r < P; ++r) {
            const dtt_schedule* s = scheds ? scheds[r] : nullptr;
            if (!s) continue;
            for (const HostChunk& ch : s->chunks) {
                if (!receives(ch.peers, r, q)) continue;
                for (size_t i = 0; i < ch.regions.size(); ++i) {
                    const dtt_region& reg = ch.regions[i];
                    dtt_region d = reg;
                    if (!ch.dests.empty()) {
                        d.offset = ch.dests[i].offset;
                        d.pitch = reg.rows > 1 ? ch.dests[i].pitch : reg.row_bytes;
                    }
                    if (d.rows == 0 || d.row_bytes == 0) continue;
                    const uint64_t span = (d.rows - 1) * d.pitch + d.row_bytes;
                    if (d.offset > nbytes || span > nbytes - d.offset)
                        return fail(DTT_EINVAL, "plan: a chunk of rank %u lands outside rank %u's %llu-byte buffer",
                                    r, q, (unsigned long long)nbytes);
                    landed.push_back(d);
                    who.push_back(r);
                }
            }
        }
        for (size_t i = 0; i < landed.size(); ++i) {
            const dtt_region& d = landed[i];
            refs.push_back(RegionRef{d.offset, d.offset + (d.rows - 1) * d.pitch + d.row_bytes, who[i], &landed[i]});
        }
        std::sort(refs.begin(), refs.end(), [](const RegionRef& a, const RegionRef& b) { return a.lo < b.lo; });
        for (size_t i = 0; i < refs.size(); ++i)
            for (size_t k = i + 1; k < refs.size() && refs[k].lo < refs[i].hi; ++k)
                if (regions_intersect(*refs[i].reg, *refs[k].reg))
                    return fail(DTT_EOVERLAP, "plan: copies from ranks %u and %u land on the same bytes of rank %u's buffer",
                                refs[i].rank, refs[k].rank, q);
    }
    return DTT_OK;
}

int validate_plan(dtt_plan* p, const dtt_schedule* const* scheds) {
    const uint32_t P = p->P;
    // ---- validation --------------------------------------------------------------------
    uint64_t S = p->buf_bytes;
    if (p->opts.allgather) {
        if (p->buf_bytes % P) return fail(DTT_EINVAL, "plan: buffer does not split into P equal slices");
        S = p->buf_bytes / P;
    }
    std::vector<RegionRef> refs;
    uint64_t total_regions = 0;
    for (uint32_t r = 0; r < P; ++r) {
        const dtt_schedule* s = scheds ? scheds[r] : nullptr;
        if (!s) continue;
        for (const HostChunk& ch : s->chunks) {
            if (ch.writers == 0) return fail(DTT_EINVAL, "plan: rank %u has a chunk with no writers", r);
            if (!ch.dests.empty() && ch.dests.size() != ch.regions.size())
                return fail(DTT_EINVAL, "plan: rank %u has a chunk with a destination count unlike its regions", r);
            if (P < 32 && (ch.peers >> P))
                return fail(DTT_EINVAL, "plan: rank %u's peer mask names a rank outside the plan", r);
            if (!ch.dests.empty() || ch.peers) p->other_dests = true;
            for (const dtt_region& reg : ch.regions) {
                ++total_regions;
                if (reg.rows == 0 || reg.row_bytes == 0) continue;
                if (reg.rows > 1 && reg.pitch < reg.row_bytes)
                    return fail(DTT_EINVAL, "plan: rank %u region with pitch < row_bytes", r);
                const uint64_t lo = reg.offset;
                const uint64_t span = (reg.rows - 1) * reg.pitch + reg.row_bytes;
                if (lo > p->buf_bytes || span > p->buf_bytes - lo)
                    return fail(DTT_EINVAL, "plan: rank %u region [%llu, +%llu) outside the %llu-byte buffer",
                                r, (unsigned long long)lo, (unsigned long long)span,
                                (unsigned long long)p->buf_bytes);
                const uint64_t hi = lo + span;
                if (p->opts.allgather && (lo < r * S || hi > (uint64_t)(r + 1) * S))
                    return fail(DTT_EOUTOFROWS, "plan: rank %u sends bytes outside its own rows", r);
                if (ch.dests.empty()) refs.push_back(RegionRef{lo, hi, r, &reg});   // lands at its own offsets
            }
        }
    }
    if (p->opts.max_regions && total_regions > p->opts.max_regions)
        return fail(DTT_ECAPACITY, "plan: %llu regions exceed the capacity of %llu",
                    (unsigned long long)total_regions, (unsigned long long)p->opts.max_regions);
    std::sort(refs.begin(), refs.end(), [](const RegionRef& a, const RegionRef& b) { return a.lo < b.lo; });
    for (size_t i = 0; i < refs.size(); ++i)
        for (size_t k = i + 1; k < refs.size() && refs[k].lo < refs[i].hi; ++k)
            if (refs[k].rank != refs[i].rank && regions_intersect(*refs[i].reg, *refs[k].reg))
                return fail(DTT_EOVERLAP, "plan: ranks %u and %u send the same bytes", refs[i].rank,
                            refs[k].rank);
    if (p->other_dests || p->separate_dst) return validate_destinations(p, scheds);
    return DTT_OK;
}

int build_plan(dtt_plan* p, const dtt_schedule* const* scheds) {
    const uint32_t P = p->P;
    // ---- global chunk numbering and copier work ------------------------------------------
    bool bases_aligned = true;
    for (uint32_t r = 0; r < P; ++r)
        bases_aligned &= (reinterpret_cast<uintptr_t>(p->bufs[r]) % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(p->dst[r]) % 16 == 0);
    uint64_t src_bytes[DTT_MAX_RANKS] = {};
    uint32_t n = 0;
    for (uint32_t r = 0; r < P; ++r) {
        const dtt_schedule* s = scheds ? scheds[r] : nullptr;
        p->first_chunk[r] = n;
        p->n_chunks[r] = s ? (uint32_t)s->chunks.size() : 0;
        n += p->n_chunks[r];
        if (s)
            for (const HostChunk& ch : s->chunks)
                for (const dtt_region& reg : ch.regions) src_bytes[r] += reg.rows * reg.row_bytes;
    }
    p->n_global = n;

    // copier CTAs per sending rank, in proportion to its bytes (at least one each)
    uint32_t senders = 0;
    uint64_t all_bytes = 0;
    for (uint32_t r = 0; r < P; ++r) {
        if (p->n_chunks[r]) ++senders;
        all_bytes += src_bytes[r];
    }
    uint32_t C = p->copier_ctas;
    if (C < senders) C = senders;
    uint32_t G[DTT_MAX_RANKS] = {};
    uint32_t given = 0;
    for (uint32_t r = 0; r < P; ++r) {
        if (!p->n_chunks[r]) continue;
        uint64_t g = all_bytes ? (uint64_t)C * src_bytes[r] / all_bytes : C / senders;
        G[r] = (uint32_t)std::max<uint64_t>(1, g);
        given += G[r];
    }
    while (given > C) {   // trim the largest shares
        uint32_t big = 0;
        for (uint32_t r = 1; r < P; ++r) if (G[r] > G[big]) big = r;
        --G[big];
        --given;
    }
    for (uint32_t r = 0; given < C && senders; r = (r + 1) % P)
        if (p->n_chunks[r]) { ++G[r]; ++given; }
    p->cta_base[0] = 0;
    for (uint32_t r = 0; r < P; ++r) p->cta_base[r + 1] = p->cta_base[r] + G[r];
    p->copier_ctas = std::max<uint32_t>(1, p->cta_base[P]);

    const CutCtx cx{p->opts.piece_bytes, p->buf_bytes, bases_aligned, p->opts.method == DTT_COPY_TMA,
                    &p->shapes};
    for (uint32_t r = 0; r < P; ++r) {
        const dtt_schedule* s = scheds ? scheds[r] : nullptr;
        if (!s) continue;
        uint64_t dealt = 0;
        for (const HostChunk& ch : s->chunks) {
            ChunkDesc cd{};
            cd.piece_begin = (uint32_t)p->pieces.size();
            for (size_t i = 0; i < ch.regions.size(); ++i) {
                const dtt_region& reg = ch.regions[i];
                const dtt_dest d = ch.dests.empty() ? dtt_dest{reg.offset, reg.pitch} : ch.dests[i];
                cut_region(reg, d, cx, &p->pieces);
                cd.bytes += reg.rows * reg.row_bytes;
            }
            for (uint32_t q = 0; q < P; ++q)
                if (receives(ch.peers, r, q)) cd.peers |= 1u << q;
            cd.receivers = (uint32_t)__builtin_popcount(cd.peers);
            if (p->pieces.size() == cd.piece_begin) {   // an empty chunk still signals arrival
                PieceDesc empty{};
                empty.tmap = kNoMap;
                p->pieces.push_back(empty);
            }
            cd.n_pieces = (uint32_t)p->pieces.size() - cd.piece_begin;
            cd.rot = (uint32_t)(dealt % G[r]);
            cd.n_part = std::min(cd.n_pieces, G[r]);
            cd.owner = r;
            cd.writers = ch.writers;
            dealt += cd.n_pieces;
            p->chunks.push_back(cd);
            p->writers.push_back(ch.writers);
            p->peer_masks.push_back(cd.peers);
        }
    }
    if (p->pieces.size() > 0xFFFFFFFFull) return fail(DTT_ECAPACITY, "plan: too many copier pieces");
    if (p->opts.method == DTT_COPY_TMA)
        for (const PieceDesc& pc : p->pieces)
            if (pc.rows && !pc.vec)
                return fail(DTT_EINVAL, "plan: the bulk-copy path needs 16-byte aligned regions "
                                        "(offset, row bytes and pitch); use DTT_COPY_VEC16");
    return DTT_OK;
}

int upload(dtt_plan* p) {
    const uint32_t P = p->P, n = p->n_global;
    const uint64_t prior = p->round - 1;    // gates as they stand after `prior` rounds
    std::vector<uint64_t> gates((uint64_t)P * n * DTT_GATE_WORDS, 0);
    for (uint32_t c = 0; c < n; ++c) {
        const ChunkDesc& cd = p->chunks[c];
        uint64_t* own = &gates[((uint64_t)cd.owner * n + c) * DTT_GATE_WORDS];
        own[DTT_GATE_READY] = prior;
        own[DTT_GATE_COUNTER] = prior * cd.writers;
        own[DTT_GATE_COMPLETION] = prior * cd.receivers;
        own[DTT_GATE_COPIER] = prior * cd.n_part;
        for (uint32_t q = 0; q < P; ++q)
            if ((cd.peers >> q) & 1u) gates[((uint64_t)q * n + c) * DTT_GATE_WORDS + DTT_GATE_ARRIVAL] = prior;
    }
    const size_t n_gate_bytes = std::max<size_t>(1, gates.size() * sizeof(uint64_t));
    DTT_CUDA_TRY(cudaMalloc(&p->d_gates, n_gate_bytes));
    DTT_CUDA_TRY(cudaMalloc(&p->d_writers, std::max<size_t>(1, n * sizeof(uint32_t))));
    DTT_CUDA_TRY(cudaMalloc(&p->d_chunks, std::max<size_t>(1, n * sizeof(ChunkDesc))));
    DTT_CUDA_TRY(cudaMalloc(&p->d_pieces, std::max<size_t>(1, p->pieces.size() * sizeof(PieceDesc))));
    // the round's status on the device; its outcome and the per-chunk flags in mapped host memory
    DTT_CUDA_TRY(cudaMalloc(&p->d_status, 2 * sizeof(DevStatus)));
    const size_t host_bytes = sizeof(HostStatus) + std::max<size_t>(1, n);
    DTT_CUDA_TRY(cudaHostAlloc(&p->h_status, host_bytes, cudaHostAllocMapped | cudaHostAllocPortable));
    std::memset(p->h_status, 0, host_bytes);
    DTT_CUDA_TRY(cudaHostGetDevicePointer(reinterpret_cast<void**>(&p->h_status_dev), p->h_status, 0));
    p->h_flags = reinterpret_cast<uint8_t*>(p->h_status + 1);
    const size_t arr_bytes = std::max<size_t>(1, n) * sizeof(uint32_t);
    DTT_CUDA_TRY(cudaHostAlloc(&p->h_arrived, arr_bytes, cudaHostAllocMapped | cudaHostAllocPortable));
    std::memset(p->h_arrived, 0, arr_bytes);
    DTT_CUDA_TRY(cudaHostGetDevicePointer(reinterpret_cast<void**>(&p->h_arrived_dev), p->h_arrived, 0));
    if (p->opts.time_copier) {
        for (auto& pair : p->ev_copier)
            for (cudaEvent_t& e : pair) DTT_CUDA_TRY(cudaEventCreate(&e));
    }
    if (!gates.empty())
        DTT_CUDA_TRY(cudaMemcpy(p->d_gates, gates.data(), gates.size() * sizeof(uint64_t), cudaMemcpyHostToDevice));
    if (n && p->other_dests) {
        DTT_CUDA_TRY(cudaMalloc(&p->d_peer_masks, n * sizeof(uint32_t)));
        DTT_CUDA_TRY(cudaMemcpy(p->d_peer_masks, p->peer_masks.data(), n * sizeof(uint32_t), cudaMemcpyHostToDevice));
    }
    if (n) {
        DTT_CUDA_TRY(cudaMemcpy(p->d_writers, p->writers.data(), n * sizeof(uint32_t), cudaMemcpyHostToDevice));
        DTT_CUDA_TRY(cudaMemcpy(p->d_chunks, p->chunks.data(), n * sizeof(ChunkDesc), cudaMemcpyHostToDevice));
    }
    if (!p->pieces.empty())
        DTT_CUDA_TRY(cudaMemcpy(p->d_pieces, p->pieces.data(), p->pieces.size() * sizeof(PieceDesc),
                                cudaMemcpyHostToDevice));
    if (!p->shapes.empty()) {     // one map per (shape, buffer): 8-byte elements, no swizzle
        auto encode = tensor_map_encoder();
        if (!encode) return fail(DTT_ECUDA, "plan: the driver has no tensor-map encoder");
        std::vector<CUtensorMap> maps(p->shapes.size() * P);
        for (size_t i = 0; i < p->shapes.size(); ++i) {
            const MapShape& m = p->shapes[i];
            const cuuint64_t dims[2] = {m.pitch / 8, p->buf_bytes / m.pitch};
            const cuuint64_t strides[1] = {m.pitch};
            const cuuint32_t box[2] = {m.inner, m.rows};
            const cuuint32_t estr[2] = {1, 1};
            for (uint32_t q = 0; q < P; ++q)
                if (encode(&maps[i * P + q], CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, p->bufs[q], dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                    return fail(DTT_ECUDA, "plan: cannot encode the tensor map of a %u x %u-byte window",
                                m.rows, m.inner * 8);
        }
        DTT_CUDA_TRY(cudaMalloc(&p->d_tmaps, maps.size() * sizeof(CUtensorMap)));
        DTT_CUDA_TRY(cudaMemcpy(p->d_tmaps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice));
    }
    DTT_CUDA_TRY(cudaMemset(p->d_status, 0, 2 * sizeof(DevStatus)));
    return DTT_OK;
}

}  // namespace

namespace dtt {

static std::mutex g_preload_mu;
static uint64_t g_preloaded = 0;     // bit d: device d's kernels are loaded

int preload_once() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(DTT_ECUDA, "dtt_preload: no CUDA device");
    std::lock_guard<std::mutex> lock(g_preload_mu);
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (bit && (g_preloaded & bit)) return DTT_OK;
    cudaError_t e = preload_copier_kernels();
    if (e == cudaSuccess) e = preload_fill_kernels();
    if (e == cudaSuccess) e = preload_barrier_kernels();
    if (e == cudaSuccess) e = preload_gemm_kernels();
    if (e == cudaSuccess) e = preload_allreduce_kernels();
    if (e != cudaSuccess) return fail(DTT_ECUDA, "dtt_preload: %s", cudaGetErrorString(e));
    g_preloaded |= bit;
    return DTT_OK;
}

int plan_copier_room(const dtt_plan* p, CopierRoom* out) {
    *out = CopierRoom{};
    if (p->opts.method == DTT_COPY_ENGINE || p->copier_ctas == 0) return DTT_OK;
    int sms = 0, reserved = 0, regs = 0;
    size_t smem = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess || sms <= 0 ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, p->device) != cudaSuccess ||
        copier_regs_per_thread(p->opts.method, &regs) != cudaSuccess ||
        copier_static_smem(p->opts.method, &smem) != cudaSuccess)
        return fail(DTT_ECUDA, "cannot query the copier kernel or the device");
    const uint32_t per_sm = (p->copier_ctas + (uint32_t)sms - 1) / (uint32_t)sms;
    const uint32_t thr = p->opts.method == DTT_COPY_TMA ? 32 : p->copier_threads;
    const uint64_t cta_smem = p->opts.method == DTT_COPY_TMA
                                  ? bulk_smem_bytes(bulk_stage_bytes(p->opts.piece_bytes), p->opts.stages)
                                  : smem;
    out->ctas = per_sm;
    out->threads = per_sm * thr;
    out->regs = (uint64_t)per_sm * thr * (((uint64_t)regs + 7) / 8 * 8);
    out->smem = (uint64_t)per_sm * (cta_smem + (uint64_t)reserved);
    return DTT_OK;
}

cudaStream_t plan_copy_stream(const dtt_plan* p) { return p->copy_stream; }

int plan_host_io(const dtt_plan* p, PlanHostIo* out) {
    if (p->ce) return fail(DTT_EINVAL, "host-buffer rounds need an SM copier (not DTT_COPY_ENGINE)");
    out->h2d = p->h2d_stream;
    out->d2h = p->d2h_stream;
    out->arrived = p->h_arrived;
    out->copier_end = p->ev_copier_end;
    out->piece_bytes = p->opts.host_piece_bytes;
    return DTT_OK;
}

void plan_set_host_round(dtt_plan* p, bool notify, bool quiet) {
    p->notify_host = notify;
    p->suppress_early = quiet;
}

}  // namespace dtt

extern "C" {

int dtt_preload(void) { return preload_once(); }

void dtt_plan_opts_default(dtt_plan_opts* o) {
    if (!o) return;
    std::memset(o, 0, sizeof(*o));
    o->allgather = 1;
    o->method = DTT_COPY_VEC16;
    o->ctas_per_sm = 1;
    o->copier_threads = 512;
    o->piece_bytes = 65536;
    o->timestamps = 1;
    o->initial_round = 1;
    o->max_polls = 1ull << 22;
}

int dtt_plan_create(void* const* bufs, uint64_t buf_bytes, uint32_t P,
                    const dtt_schedule* const* scheds, const dtt_plan_opts* opts,
                    cudaStream_t copy_stream, dtt_plan** out) {
    if (!out) return fail(DTT_EINVAL, "dtt_plan_create: out is NULL");
    *out = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_plans_mu);
        reap_locked();
    }
    if (!bufs || P < 1 || P > DTT_MAX_RANKS || buf_bytes == 0)
        return fail(DTT_EINVAL, "dtt_plan_create: need 1 <= P <= %d buffers of a positive size", DTT_MAX_RANKS);
    dtt_plan* p = new (std::nothrow) dtt_plan();
    if (!p) return fail(DTT_ENOMEM, "dtt_plan_create: out of memory");
    if (opts) p->opts = *opts; else dtt_plan_opts_default(&p->opts);
    dtt_plan_opts& o = p->opts;
    if (o.initial_round == 0) o.initial_round = 1;
    if (o.max_polls == 0) o.max_polls = 1ull << 22;
    if (o.piece_bytes == 0) o.piece_bytes = 65536;
    if (o.copier_threads == 0) o.copier_threads = 512;
    if (o.ctas_per_sm == 0) o.ctas_per_sm = 1;
    if (o.stages == 0 && o.piece_bytes % 16 == 0)   // as many stages as fit, at most 8
        o.stages = (uint32_t)std::max<size_t>(2, std::min<size_t>(8, kBulkSmemMax / (bulk_stage_bytes(o.piece_bytes) + 8)));
    if (o.piece_bytes % 16 || o.copier_threads % 32 || o.copier_threads > 1024 ||
        (o.method != DTT_COPY_VEC16 && o.method != DTT_COPY_TMA && o.method != DTT_COPY_ENGINE)) {
        delete p;
        return fail(DTT_EINVAL, "dtt_plan_create: bad options (piece_bytes %% 16, threads %% 32 <= 1024, method)");
    }
    if (o.host_piece_bytes % 4096) {
        delete p;
        return fail(DTT_EINVAL, "dtt_plan_create: host_piece_bytes must be a multiple of 4096");
    }
    if (o.deferred_copier > 2) {
        delete p;
        return fail(DTT_EINVAL, "dtt_plan_create: deferred_copier is 0, 1 or 2");
    }
    if (o.overlap > 1 || (o.overlap && o.deferred_copier == 1)) {
        // a round's producers wait for the previous round's copies, so that copier must run
        // beside them, not after them
        delete p;
        return fail(DTT_EINVAL, "dtt_plan_create: overlap is 0 or 1, and overlapping rounds need deferred_copier 0 or 2");
    }
    if (o.early_copier_us > 1000000) {
        delete p;
        return fail(DTT_EINVAL, "dtt_plan_create: early_copier_us is at most 1000000 (one second)");
    }
    if (o.method == DTT_COPY_TMA && o.stages < 2) {      // the ring loads ahead by stages - 1
        delete p;
        return fail(DTT_EINVAL, "dtt_plan_create: the bulk-copy path needs at least 2 stages");
    }
    if (o.method == DTT_COPY_TMA && bulk_smem_bytes(bulk_stage_bytes(o.piece_bytes), o.stages) > kBulkSmemMax) {
        delete p;
        return fail(DTT_EINVAL, "dtt_plan_create: stages x piece_bytes exceeds %zu bytes of shared memory",
                    kBulkSmemMax);
    }
    p->P = P;
    p->buf_bytes = buf_bytes;
    p->round = o.initial_round;
    for (uint32_t r = 0; r < P; ++r) {
        if (!bufs[r]) {
            delete p;
            return fail(DTT_EINVAL, "dtt_plan_create: buffer %u is NULL", r);
        }
        p->bufs[r] = static_cast<char*>(bufs[r]);
        p->dst[r] = p->bufs[r];
    }
    if (o.dst_bufs) {                 // separate destination (staging) buffers
        if (o.dst_bytes == 0) {
            delete p;
            return fail(DTT_EINVAL, "dtt_plan_create: dst_bufs needs dst_bytes > 0");
        }
        for (uint32_t r = 0; r < P; ++r) {
            if (!o.dst_bufs[r]) {
                delete p;
                return fail(DTT_EINVAL, "dtt_plan_create: destination buffer %u is NULL", r);
            }
            p->dst[r] = static_cast<char*>(o.dst_bufs[r]);
        }
        p->separate_dst = true;
        p->dst_bytes = o.dst_bytes;
    }
    o.dst_bufs = nullptr;             // the plan keeps its own copy of the pointers
    int rc = validate_plan(p, scheds);    // host-only checks come first
    if (rc != DTT_OK) {
        delete p;
        return rc;
    }
    int sms = 0;
    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
        delete p;
        return fail(DTT_ECUDA, "dtt_plan_create: no CUDA device");
    }
    rc = preload_once();
    if (rc != DTT_OK) {
        delete p;
        return rc;
    }
    int host_atomics = 0;
    if (cudaDeviceGetAttribute(&host_atomics, cudaDevAttrHostNativeAtomicSupported, p->device) != cudaSuccess)
        host_atomics = 0;
    p->host_atomics = host_atomics != 0;
    p->copier_ctas = o.copier_ctas ? o.copier_ctas : (uint32_t)sms * o.ctas_per_sm;
    p->copier_threads = o.copier_threads;
    if (o.deferred_copier != 1 && o.method != DTT_COPY_ENGINE) {
        // The copier spins while the producer runs, so it must leave an SM room for producer
        // CTAs: at most half of its threads (2048) and half of its registers (64 Ki) per SM.
        int regs = 0;
        if (copier_regs_per_thread(o.method, &regs) != cudaSuccess) {
            delete p;
            return fail(DTT_ECUDA, "dtt_plan_create: cannot query the copier kernel");
        }
        const uint64_t per_sm = (p->copier_ctas + (uint32_t)sms - 1) / (uint32_t)sms;
        const uint64_t thr = o.method == DTT_COPY_TMA ? 32 : o.copier_threads;
        if (per_sm * thr > 1024 || per_sm * thr * (uint64_t)regs > 32768) {
            delete p;
            return fail(DTT_EINVAL,
                        "dtt_plan_create: %llu copier CTA(s) of %llu threads x %d registers per SM leave "
                        "too little room for a producer beside the copier (at most 1024 threads and "
                        "32768 registers per SM)",
                        (unsigned long long)per_sm, (unsigned long long)thr, regs);
        }
        if (o.method == DTT_COPY_TMA) {
            // Every copier CTA must be resident at once: a copier CTA still waiting for shared
            // memory keeps the (lower-priority) producer's CTAs from being scheduled, and the
            // resident copier CTAs then wait for gates that nothing opens until their polls run out.
            int sm_smem = 0, reserved = 0;
            if (cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, p->device) != cudaSuccess ||
                cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, p->device) != cudaSuccess) {
                delete p;
                return fail(DTT_ECUDA, "dtt_plan_create: cannot query the shared memory per SM");
            }
            const uint64_t need = per_sm * (bulk_smem_bytes(bulk_stage_bytes(o.piece_bytes), o.stages) + (uint64_t)reserved);
            if (need > (uint64_t)sm_smem) {
                delete p;
                return fail(DTT_EINVAL,
                            "dtt_plan_create: %llu copier CTA(s) per SM need %llu bytes of shared memory, the SM "
                            "has %d: lower ctas_per_sm, stages or piece_bytes",
                            (unsigned long long)per_sm, (unsigned long long)need, sm_smem);
            }
        }
    }
    rc = build_plan(p, scheds);
    if (rc == DTT_OK) rc = upload(p);
    if (rc == DTT_OK && o.method == DTT_COPY_ENGINE) rc = start_ce(p, scheds);
    if (rc == DTT_OK) {
        if (copy_stream) {
            p->copy_stream = copy_stream;
        } else {
            int lo = 0, hi = 0;
            cudaDeviceGetStreamPriorityRange(&lo, &hi);
            if (cudaStreamCreateWithPriority(&p->copy_stream, cudaStreamNonBlocking, hi) != cudaSuccess)
                rc = fail(DTT_ECUDA, "dtt_plan_create: cannot create the copy stream");
            else
                p->own_copy_stream = true;
        }
    }
    if (rc == DTT_OK && cudaStreamCreateWithFlags(&p->aux_stream, cudaStreamNonBlocking) != cudaSuccess)
        rc = fail(DTT_ECUDA, "dtt_plan_create: cannot create the aux stream");
    if (rc == DTT_OK && (cudaEventCreateWithFlags(&p->ev_producer, cudaEventDisableTiming) != cudaSuccess ||
                         cudaEventCreateWithFlags(&p->ev_done, cudaEventDisableTiming) != cudaSuccess ||
                         cudaEventCreateWithFlags(&p->ev_copier_end, cudaEventDisableTiming) != cudaSuccess ||
                         cudaEventCreateWithFlags(&p->ev_h2d, cudaEventDisableTiming) != cudaSuccess ||
                         cudaEventCreateWithFlags(&p->ev_pending, cudaEventDisableTiming) != cudaSuccess))
        rc = fail(DTT_ECUDA, "dtt_plan_create: cannot create an event");
    if (rc == DTT_OK && (cudaStreamCreateWithFlags(&p->d2h_stream, cudaStreamNonBlocking) != cudaSuccess ||
                         cudaStreamCreateWithFlags(&p->h2d_stream, cudaStreamNonBlocking) != cudaSuccess))
        rc = fail(DTT_ECUDA, "dtt_plan_create: cannot create the host-copy streams");
    if (rc != DTT_OK) {           // all or nothing: free what was prepared
        free_device(p);
        delete p;
        return rc;
    }
    p->state = DTT_PLAN_PREPARED;
    {
        std::lock_guard<std::mutex> lock(g_plans_mu);
        g_live.push_back(p);
    }
    *out = p;
    return DTT_OK;
}

int dtt_plan_start(dtt_plan* p, cudaStream_t producer_stream, dtt_handle* handles) {
    if (!p) return fail(DTT_EINVAL, "dtt_plan_start: NULL plan");
    if (p->state != DTT_PLAN_PREPARED) return fail(DTT_ESTATE, "dtt_plan_start: plan is not PREPARED (state %d)", p->state);
    if (producer_stream == p->copy_stream)
        return fail(DTT_EINVAL, "dtt_plan_start: the producer stream must differ from the copy stream");
    p->copier_launched = false;      // the status words were zeroed by the last check (or upload)
    if (p->early_pending && (p->early_round != p->round || p->notify_host))
        abort_early(p);              // a host-buffer round needs a copier that stamps arrivals
    if (p->ce) {                     // the proxy issues this round's copies as gates open
        {
            std::lock_guard<std::mutex> lock(p->ce->mu);
            p->ce->rc_of[p->round & 1u] = DTT_OK;
            p->ce->open_all.store(false);
            if (p->n_global) {
                if (p->ce->busy) {
                    p->ce->queued = p->round;    // behind the pending round (overlapping rounds)
                } else {
                    p->ce->round = p->round;
                    p->ce->busy = true;
                }
            }
        }
        p->ce->cv.notify_all();
    } else if (claim_early(p)) {
        p->copier_launched = true;   // launched by the last wait(), now claimed for this round
    } else if (p->n_global && !p->opts.deferred_copier) {
        const int rc = launch_round_copier(p);
        if (rc != DTT_OK) return rc;
    }
    p->producer_stream = producer_stream;
    if (handles)
        for (uint32_t r = 0; r < p->P; ++r) handles[r] = make_handle(p, r);
    p->live_round = true;
    p->state = DTT_PLAN_RUNNING;
    return DTT_OK;
}

int dtt_plan_handle(const dtt_plan* p, uint32_t rank, dtt_handle* out) {
    if (!p || !out || rank >= p->P) return fail(DTT_EINVAL, "dtt_plan_handle: bad args");
    *out = make_handle(p, rank);
    return DTT_OK;
}

int dtt_plan_launch_copier(dtt_plan* p) {
    if (!p) return fail(DTT_EINVAL, "dtt_plan_launch_copier: NULL plan");
    if (p->state != DTT_PLAN_RUNNING) return fail(DTT_ESTATE, "dtt_plan_launch_copier: plan is not RUNNING");
    if (p->copier_launched || !p->n_global || p->ce) return DTT_OK;
    if (p->opts.deferred_copier == 1) {   // after the producers: no overlap
        DTT_CUDA_TRY(cudaEventRecord(p->ev_producer, p->producer_stream));
        DTT_CUDA_TRY(cudaStreamWaitEvent(p->copy_stream, p->ev_producer, 0));
    }
    return launch_round_copier(p);
}

namespace {

// Launch round `round`'s completion check on `stream`; it waits on the device for `copier_ctas`
// copier CTAs of that round to count themselves out.  pending: the round after it may already
// be marking, so only the error word reports extra marks.
int launch_round_check(dtt_plan* p, uint32_t round, uint32_t copier_ctas, bool pending, cudaStream_t stream,
                       uint32_t* seq) {
    CheckParams ck{};
    ck.copier_ctas = copier_ctas;
    ck.max_polls = 8 * p->opts.max_polls;
    ck.gates = p->d_gates;
    ck.chunks = p->d_chunks;
    ck.P = p->P;
    ck.n_global = p->n_global;
    ck.round = round;
    ck.pending = pending ? 1u : 0u;
    ck.seq = ++p->wait_seq;
    ck.status = status_of(p, round);
    ck.host = p->h_status_dev;
    ck.host_flags = p->h_status_dev ? reinterpret_cast<uint8_t*>(p->h_status_dev + 1) : nullptr;
    DTT_CUDA_TRY(launch_check(ck, stream));
    *seq = ck.seq;
    return DTT_OK;
}

// Poll the mapped host block until the check with sequence number `seq` has reported.  The check
// stores its sequence number last, after every flag and status word; the stream it runs on is
// asked now and then, so that a failed launch or a dead context ends the wait with the CUDA
// error instead of spinning.
int await_check(dtt_plan* p, uint32_t seq, cudaStream_t stream) {
    const uint32_t* done = &p->h_status->done;
    for (uint64_t spin = 1;; ++spin) {
        if (__atomic_load_n(done, __ATOMIC_ACQUIRE) == seq) return DTT_OK;
        if ((spin & 4095) == 0) {
            const cudaError_t e = cudaStreamQuery(stream);
            if (e == cudaErrorNotReady) continue;
            if (e != cudaSuccess) return fail(DTT_ECUDA, "dtt_plan_wait: %s", cudaGetErrorString(e));
            if (__atomic_load_n(done, __ATOMIC_ACQUIRE) == seq) return DTT_OK;
            return fail(DTT_ECUDA, "dtt_plan_wait: the check kernel finished without reporting");
        }
    }
}

// Turn the reported flags and status words of round `round`'s check into a report and a code.
int read_report(dtt_plan* p, uint32_t round, int ce_rc, dtt_report* report) {
    dtt_report rep{};
    rep.round = round;
    rep.copier_timeouts = p->h_status->st.copier_timeouts + (ce_rc == DTT_ETIMEDOUT ? 1u : 0u);
    rep.device_status = p->h_status->st.misuse;
    const bool late = p->h_status->st.check_late != 0;
    for (uint32_t c = 0; c < p->n_global; ++c) {
        if (p->h_flags[c] == 2) {
            if (rep.n_extra < DTT_REPORT_MAX) rep.extra_chunks[rep.n_extra] = c;
            ++rep.n_extra;
        } else if (p->h_flags[c] == 1) {
            if (rep.n_short < DTT_REPORT_MAX) rep.short_chunks[rep.n_short] = c;
            ++rep.n_short;
        }
    }
    int rc = DTT_OK;
    if (rep.n_extra) {
        rc = fail(DTT_EEXTRA, "dtt_plan_wait: %u chunk(s) got extra marks in round %u (first: %u)",
                  rep.n_extra, round, rep.extra_chunks[0]);
    } else if (rep.device_status) {
        rc = fail(DTT_EINVAL, "dtt_plan_wait: %s",
                  (rep.device_status & DTT_DEV_EBADCHUNK)
                      ? "a kernel marked, or asked reusable or writable of, a chunk its rank does not own"
                  : (rep.device_status & DTT_DEV_EBADGROUP)
                      ? "a kernel waited on a group the plan does not have"
                      : "a producer gave up waiting for a chunk to become writable");
    } else if (rep.n_short) {
        rc = fail(DTT_ETIMEDOUT, "dtt_plan_wait: %u chunk(s) short in round %u (first: %u)",
                  rep.n_short, round, rep.short_chunks[0]);
    } else if (late) {
        rc = fail(DTT_ETIMEDOUT, "dtt_plan_wait: the copier had not finished when the check gave up");
    }
    rep.status = rc;
    if (report) *report = rep;
    return rc;
}

// Overlapping rounds: check the pending round, on the plan's aux stream after the producers
// queued before it became pending (not after the next round's).
int wait_pending(dtt_plan* p, dtt_report* report) {
    const uint32_t R = p->pending;
    int ce_rc = DTT_OK;
    if (p->ce) ce_rc = ce_join(p, p->aux_stream, R);   // the check follows the round's copies
    DTT_CUDA_TRY(cudaStreamWaitEvent(p->aux_stream, p->ev_pending, 0));
    uint32_t seq = 0;
    int rc = launch_round_check(p, R, p->pending_copier ? p->copier_ctas : 0, true, p->aux_stream, &seq);
    if (rc == DTT_OK) rc = await_check(p, seq, p->aux_stream);
    if (rc != DTT_OK) return rc;
    rc = read_report(p, R, ce_rc, report);
    p->pending = 0;
    p->pending_copier = false;
    if (rc != DTT_OK) p->state = DTT_PLAN_FAILED;   // the current round, if started, is closed with the plan
    return rc;
}

}  // namespace

int dtt_plan_wait(dtt_plan* p, dtt_report* report) {
    if (!p) return fail(DTT_EINVAL, "dtt_plan_wait: NULL plan");
    if (p->pending && p->state != DTT_PLAN_FAILED) return wait_pending(p, report);
    if (p->state != DTT_PLAN_RUNNING) return fail(DTT_ESTATE, "dtt_plan_wait: plan is not RUNNING (state %d)", p->state);
    const int lc = dtt_plan_launch_copier(p);    // deferred plans: the copier runs now
    if (lc != DTT_OK) return lc;
    // The check follows the producers on their stream and waits on the device for the copier's
    // CTAs to count themselves out (no event between the streams, no launch gap after the copier).
    int ce_rc = DTT_OK;
    if (p->ce) ce_rc = ce_join(p, p->producer_stream, p->round);   // the check follows every queue
    uint32_t seq = 0;
    int rc = launch_round_check(p, p->round, p->copier_launched ? p->copier_ctas : 0, false, p->producer_stream, &seq);
    if (rc != DTT_OK) return rc;
    // The next round's copier queues behind this one while the host waits: its launch leaves
    // the next round's critical path.  It copies nothing until start() claims it.
    if (early_allowed(p)) {
        const int erc = launch_early(p);
        if (erc != DTT_OK) return erc;
    }
    rc = await_check(p, seq, p->producer_stream);
    if (rc != DTT_OK) {
        abort_early(p);
        return rc;
    }
    p->live_round = false;
    rc = read_report(p, p->round, ce_rc, report);
    p->state = rc == DTT_OK ? DTT_PLAN_DONE : DTT_PLAN_FAILED;
    if (rc != DTT_OK) abort_early(p);    // a failed plan has no next round
    return rc;
}

int dtt_plan_next_round(dtt_plan* p) {
    if (!p) return fail(DTT_EINVAL, "dtt_plan_next_round: NULL plan");
    if (p->opts.overlap && p->state == DTT_PLAN_RUNNING && !p->pending) {
        // overlapping rounds: the running round stays in flight (pending) and the next one is
        // prepared.  Its copier goes on the copy stream now, ahead of the next round's, so every
        // queue serves it first; its check will follow the producers queued so far.
        if (p->round == 0xFFFFFFFFu)
            return fail(DTT_EROUNDLIMIT, "dtt_plan_next_round: a plan is limited to 2^32 - 1 rounds");
        const int lc = dtt_plan_launch_copier(p);
        if (lc != DTT_OK) return lc;
        DTT_CUDA_TRY(cudaEventRecord(p->ev_pending, p->producer_stream));
        p->pending = p->round;
        p->pending_copier = p->copier_launched;
        p->live_round = false;
        p->copier_launched = false;
        ++p->round;
        p->state = DTT_PLAN_PREPARED;
        return DTT_OK;
    }
    if (p->state != DTT_PLAN_DONE) return fail(DTT_ESTATE, "dtt_plan_next_round: plan is not DONE (state %d)", p->state);
    if (p->round == 0xFFFFFFFFu)
        return fail(DTT_EROUNDLIMIT, "dtt_plan_next_round: a plan is limited to 2^32 - 1 rounds");
    ++p->round;
    p->state = DTT_PLAN_PREPARED;
    return DTT_OK;
}

uint32_t dtt_plan_pending_round(const dtt_plan* p) { return p ? p->pending : 0; }

namespace {

// Wait for p's last copier to finish (its gates are open by now).
int drain_copier(dtt_plan* p) {
    if (p->aux_stream && cudaStreamSynchronize(p->aux_stream) != cudaSuccess)
        return fail(DTT_ECUDA, "dtt_plan_close: aux stream failed");
    if (!p->copier_launched && !p->pending_copier) return DTT_OK;
    const cudaError_t e = p->done_valid ? cudaEventSynchronize(p->ev_done) : cudaStreamSynchronize(p->copy_stream);
    return e == cudaSuccess ? DTT_OK : fail(DTT_ECUDA, "dtt_plan_close: copy stream failed: %s", cudaGetErrorString(e));
}

// The user is done with p: drop it from the live list, free it now or when nothing spins.
void release(dtt_plan* p) {
    std::lock_guard<std::mutex> lock(g_plans_mu);
    g_live.erase(std::remove(g_live.begin(), g_live.end(), p), g_live.end());
    g_retired.push_back(p);
    reap_locked();
}

// Finish every CLOSING plan on `stream` that no longer waits behind an earlier copier.  Their
// gates were opened by their own close, so each copier now runs to its end.
int finish_closing(cudaStream_t stream) {
    int rc = DTT_OK;
    for (bool progress = true; progress;) {
        progress = false;
        dtt_plan* next = nullptr;
        {
            std::lock_guard<std::mutex> lock(g_plans_mu);
            for (dtt_plan* q : g_live)
                if (q->state == DTT_PLAN_CLOSING && q->copy_stream == stream && !blocked_behind(q) &&
                    (!next || q->launch_seq < next->launch_seq))
                    next = q;
        }
        if (next) {
            const int r = drain_copier(next);
            if (r != DTT_OK) rc = r;
            next->state = DTT_PLAN_CLOSED;     // released by its owner's next dtt_plan_close
            progress = true;
        }
    }
    return rc;
}

}  // namespace

int dtt_plan_close(dtt_plan* p) {
    if (!p) return DTT_OK;
    if (p->state == DTT_PLAN_CLOSED) {      // finished by the close of the plan it waited behind
        release(p);
        return DTT_OK;
    }
    int rc = DTT_OK;
    abort_early(p);                          // a copier launched for a round that never starts
    if (p->early_launched && p->state != DTT_PLAN_RUNNING && p->state != DTT_PLAN_CLOSING &&
        cudaStreamSynchronize(p->copy_stream) != cudaSuccess)
        rc = fail(DTT_ECUDA, "dtt_plan_close: copy stream failed");
    // Mid-round: a started round whose check has not run, or a pending round (overlapping rounds).
    const bool mid = (p->live_round || p->pending) && p->state != DTT_PLAN_CLOSING;
    if (mid) {
        // what the producers queued so far is written first; then every gate still closed is
        // opened (for the latest round in flight, which opens the pending round's too), so each
        // copier sends its chunks as they stand and exits
        const uint32_t top = p->live_round ? p->round : p->pending;
        if (cudaStreamSynchronize(p->producer_stream) != cudaSuccess)
            rc = fail(DTT_ECUDA, "dtt_plan_close: producer stream failed");
        if (p->n_global && launch_force_open(p->d_gates, p->d_chunks, p->n_global, top, p->aux_stream) != cudaSuccess)
            rc = fail(DTT_ECUDA, "dtt_plan_close: force-open launch failed");
        if (p->ce) {                 // the proxy sends every chunk as it stands, then drains
            p->ce->open_all.store(true);
            const int jr = ce_join(p, nullptr, 0);
            if (jr != DTT_OK && jr != DTT_ETIMEDOUT) rc = jr;
        }
        if (p->live_round && !p->copier_launched && p->n_global && !p->ce) {   // deferred: send the chunks now
            if (cudaStreamSynchronize(p->aux_stream) != cudaSuccess || launch_round_copier(p) != DTT_OK)
                rc = fail(DTT_ECUDA, "dtt_plan_close: copier launch failed");
        }
    }
    if (mid || p->state == DTT_PLAN_CLOSING) {
        bool blocked;
        {
            std::lock_guard<std::mutex> lock(g_plans_mu);
            blocked = blocked_behind(p);
        }
        if (blocked) {                      // queued behind an earlier plan's waiting copier
            p->state = DTT_PLAN_CLOSING;
            return rc == DTT_OK ? DTT_CLOSING : rc;
        }
        const int r = drain_copier(p);
        if (r != DTT_OK) rc = r;
    } else if (p->aux_stream && cudaStreamSynchronize(p->aux_stream) != cudaSuccess) {
        rc = fail(DTT_ECUDA, "dtt_plan_close: aux stream failed");
    }
    p->state = DTT_PLAN_CLOSED;
    const int r = finish_closing(p->copy_stream);
    if (r != DTT_OK) rc = r;
    release(p);
    return rc;
}

int dtt_plan_stats(dtt_plan* p, double* copier_ms_last, double* copier_ms_total,
                   uint64_t* rounds_timed) {
    if (!p) return fail(DTT_EINVAL, "dtt_plan_stats: NULL plan");
    const int rc = read_copier_times(p, p->timed_launches);
    if (rc != DTT_OK) return rc;
    if (copier_ms_last) *copier_ms_last = p->copier_ms_last;
    if (copier_ms_total) *copier_ms_total = p->copier_ms_total;
    if (rounds_timed) *rounds_timed = p->timed_read;
    return DTT_OK;
}

int dtt_plan_define_groups(dtt_plan* p, uint32_t n_groups, const uint32_t* offsets, const uint32_t* chunk_ids) {
    if (!p || !offsets || (!chunk_ids && offsets[n_groups]) || n_groups == 0)
        return fail(DTT_EINVAL, "dtt_plan_define_groups: bad args");
    if (p->opts.overlap)
        return fail(DTT_EINVAL, "dtt_plan_define_groups: a plan with overlapping rounds has no groups (a member's "
                                "next-round arrival would count toward this round's wait)");
    if (p->n_groups) return fail(DTT_ESTATE, "dtt_plan_define_groups: the plan's groups are defined already");
    if (p->state != DTT_PLAN_PREPARED || p->round != p->opts.initial_round || p->wait_seq || p->early_launched)
        return fail(DTT_ESTATE, "dtt_plan_define_groups: groups are defined before the plan's first start");
    if (offsets[0] != 0) return fail(DTT_EINVAL, "dtt_plan_define_groups: offsets[0] must be 0");
    // per group: its members, distinct and in range; per chunk: the groups it belongs to (CSR);
    // per (rank, group): the members that reach the rank (its own, or addressed to it)
    std::vector<uint32_t> size((size_t)p->P * n_groups, 0), chunk_off(p->n_global + 1, 0);
    std::vector<uint32_t> seen(p->n_global, UINT32_MAX);
    for (uint32_t g = 0; g < n_groups; ++g) {
        if (offsets[g + 1] <= offsets[g])
            return fail(DTT_EINVAL, "dtt_plan_define_groups: group %u is empty (or offsets decrease)", g);
        for (uint32_t i = offsets[g]; i < offsets[g + 1]; ++i) {
            const uint32_t c = chunk_ids[i];
            if (c >= p->n_global) return fail(DTT_EINVAL, "dtt_plan_define_groups: chunk id %u out of range", c);
            if (seen[c] == g) return fail(DTT_EINVAL, "dtt_plan_define_groups: chunk %u twice in group %u", c, g);
            seen[c] = g;
            ++chunk_off[c + 1];
            const ChunkDesc& cd = p->chunks[c];
            for (uint32_t q = 0; q < p->P; ++q)
                if (q == cd.owner || ((cd.peers >> q) & 1u)) ++size[(size_t)q * n_groups + g];
        }
    }
    for (uint32_t c = 0; c < p->n_global; ++c) chunk_off[c + 1] += chunk_off[c];
    std::vector<uint32_t> ids(chunk_off[p->n_global]), fill(chunk_off.begin(), chunk_off.end() - 1);
    for (uint32_t g = 0; g < n_groups; ++g)
        for (uint32_t i = offsets[g]; i < offsets[g + 1]; ++i) ids[fill[chunk_ids[i]]++] = g;
    // counters begin as after the rounds before this one
    const uint64_t prior = p->round - 1;
    std::vector<uint64_t> counters((uint64_t)p->P * n_groups);
    for (uint32_t q = 0; q < p->P; ++q)
        for (uint32_t g = 0; g < n_groups; ++g)
            counters[(uint64_t)q * n_groups + g] = prior * size[(size_t)q * n_groups + g];
    std::vector<uint32_t> arrays;
    arrays.reserve(size.size() + chunk_off.size() + ids.size() + 1);
    arrays.insert(arrays.end(), size.begin(), size.end());
    arrays.insert(arrays.end(), chunk_off.begin(), chunk_off.end());
    arrays.insert(arrays.end(), ids.begin(), ids.end());
    arrays.push_back(0);
    // no copier of this plan runs yet; plain allocations and copies are ordered before its first
    // start (on the legacy stream, which the plan's non-blocking streams do not wait for, so
    // the copies are synchronous here)
    DTT_CUDA_TRY(cudaMalloc(&p->d_group_counters, counters.size() * sizeof(uint64_t)));
    DTT_CUDA_TRY(cudaMalloc(&p->d_group_arrays, arrays.size() * sizeof(uint32_t)));
    DTT_CUDA_TRY(cudaMemcpy(p->d_group_counters, counters.data(), counters.size() * sizeof(uint64_t),
                            cudaMemcpyHostToDevice));
    DTT_CUDA_TRY(cudaMemcpy(p->d_group_arrays, arrays.data(), arrays.size() * sizeof(uint32_t),
                            cudaMemcpyHostToDevice));
    p->n_groups = n_groups;
    p->group_size = size;
    return DTT_OK;
}

int dtt_plan_define_block_groups(dtt_plan* p, uint64_t block_bytes, uint32_t* n_groups, uint32_t* block_group) {
    if (!p || block_bytes == 0) return fail(DTT_EINVAL, "dtt_plan_define_block_groups: bad args");
    if (p->other_dests || p->separate_dst)
        return fail(DTT_EINVAL, "dtt_plan_define_block_groups: needs chunks that land at their own offsets");
    const uint64_t nb = (p->buf_bytes + block_bytes - 1) / block_bytes;
    if (nb > 0xFFFFFFF0ull) return fail(DTT_EINVAL, "dtt_plan_define_block_groups: too many blocks");
    // the blocks each chunk touches, from the copier's pieces (every row of every piece)
    std::vector<std::vector<uint32_t>> members(nb);
    for (uint32_t c = 0; c < p->n_global; ++c) {
        const ChunkDesc& cd = p->chunks[c];
        uint64_t last = UINT64_MAX;
        std::vector<uint64_t> touched;
        for (uint32_t i = 0; i < cd.n_pieces; ++i) {
            const PieceDesc& pc = p->pieces[cd.piece_begin + i];
            for (uint32_t r = 0; r < pc.rows; ++r) {
                const uint64_t lo = pc.off + (uint64_t)r * pc.pitch, hi = lo + pc.row_bytes;
                for (uint64_t b = lo / block_bytes; b * block_bytes < hi; ++b)
                    if (b != last) {
                        touched.push_back(b);
                        last = b;
                    }
            }
        }
        std::sort(touched.begin(), touched.end());
        touched.erase(std::unique(touched.begin(), touched.end()), touched.end());
        for (uint64_t b : touched) members[b].push_back(c);
    }
    std::vector<uint32_t> offsets(1, 0), ids, bg(nb, UINT32_MAX);
    for (uint64_t b = 0; b < nb; ++b) {
        if (members[b].empty()) continue;
        bg[b] = (uint32_t)(offsets.size() - 1);
        ids.insert(ids.end(), members[b].begin(), members[b].end());
        offsets.push_back((uint32_t)ids.size());
    }
    if (offsets.size() < 2) return fail(DTT_EINVAL, "dtt_plan_define_block_groups: no chunk touches any block");
    const int rc = dtt_plan_define_groups(p, (uint32_t)(offsets.size() - 1), offsets.data(), ids.data());
    if (rc != DTT_OK) return rc;
    p->group_block_bytes = block_bytes;
    p->block_group = bg;
    if (n_groups) *n_groups = p->n_groups;
    if (block_group) std::copy(bg.begin(), bg.end(), block_group);
    return DTT_OK;
}

int dtt_plan_read_group_counters(dtt_plan* p, uint64_t* host, uint64_t n_words) {
    if (!p || !host) return fail(DTT_EINVAL, "dtt_plan_read_group_counters: bad args");
    if (!p->n_groups) return fail(DTT_EINVAL, "dtt_plan_read_group_counters: the plan has no groups");
    const uint64_t need = (uint64_t)p->P * p->n_groups;
    if (n_words < need)
        return fail(DTT_EINVAL, "dtt_plan_read_group_counters: need %llu words", (unsigned long long)need);
    DTT_CUDA_TRY(cudaMemcpyAsync(host, p->d_group_counters, need * sizeof(uint64_t), cudaMemcpyDeviceToHost,
                                 p->aux_stream));
    DTT_CUDA_TRY(cudaStreamSynchronize(p->aux_stream));
    return DTT_OK;
}

int dtt_plan_early_stats(const dtt_plan* p, uint64_t* launched, uint64_t* claimed, uint64_t* expired,
                         uint64_t* aborted) {
    if (!p) return fail(DTT_EINVAL, "dtt_plan_early_stats: NULL plan");
    if (launched) *launched = p->early_launches;
    if (claimed) *claimed = p->early_claims;
    if (expired) *expired = p->early_expired;
    if (aborted) *aborted = p->early_aborts;
    return DTT_OK;
}

int dtt_plan_state(const dtt_plan* p) { return p ? p->state : DTT_EINVAL; }
uint32_t dtt_plan_round(const dtt_plan* p) { return p ? p->round : 0; }

int dtt_plan_info(const dtt_plan* p, uint32_t* n_global, uint32_t* first_chunk, uint32_t* n_chunks,
                  uint64_t** gates_device) {
    if (!p) return fail(DTT_EINVAL, "dtt_plan_info: NULL plan");
    if (n_global) *n_global = p->n_global;
    for (uint32_t r = 0; r < p->P; ++r) {
        if (first_chunk) first_chunk[r] = p->first_chunk[r];
        if (n_chunks) n_chunks[r] = p->n_chunks[r];
    }
    if (gates_device) *gates_device = p->d_gates;
    return DTT_OK;
}

int dtt_plan_read_gates(dtt_plan* p, uint64_t* host, uint64_t n_words) {
    if (!p || !host) return fail(DTT_EINVAL, "dtt_plan_read_gates: bad args");
    const uint64_t need = (uint64_t)p->P * p->n_global * DTT_GATE_WORDS;
    if (n_words < need) return fail(DTT_EINVAL, "dtt_plan_read_gates: need %llu words", (unsigned long long)need);
    if (need == 0) return DTT_OK;
    // on the plan's own auxiliary stream: a copier launched early for the next round may hold
    // the copy stream until that round starts
    DTT_CUDA_TRY(cudaMemcpyAsync(host, p->d_gates, need * sizeof(uint64_t), cudaMemcpyDeviceToHost, p->aux_stream));
    DTT_CUDA_TRY(cudaStreamSynchronize(p->aux_stream));
    return DTT_OK;
}

namespace {

// The byte extent [lo, hi) of every chunk in the buffers, from the copier's pieces (0, 0 for a
// chunk without bytes).
void chunk_extents(const dtt_plan* p, std::vector<uint64_t>* lo, std::vector<uint64_t>* hi) {
    lo->assign(p->n_global, 0);
    hi->assign(p->n_global, 0);
    for (uint32_t c = 0; c < p->n_global; ++c) {
        const ChunkDesc& cd = p->chunks[c];
        uint64_t a = UINT64_MAX, b = 0;
        for (uint32_t i = 0; i < cd.n_pieces; ++i) {
            const PieceDesc& pc = p->pieces[cd.piece_begin + i];
            if (!pc.rows) continue;
            a = std::min(a, pc.off);
            b = std::max(b, pc.off + (uint64_t)(pc.rows - 1) * pc.pitch + pc.row_bytes);
        }
        if (b) {
            (*lo)[c] = a;
            (*hi)[c] = b;
        }
    }
}

}  // namespace

int dtt_allgather_host(dtt_plan* p, const void* const* host_slices, void* host_out,
                       uint32_t out_rank, cudaStream_t stream, dtt_report* report) {
    if (!p || !host_slices) return fail(DTT_EINVAL, "dtt_allgather_host: bad args");
    if (!p->opts.allgather) return fail(DTT_EINVAL, "dtt_allgather_host: needs an all-gather plan");
    if (p->ce) return fail(DTT_EINVAL, "dtt_allgather_host: needs an SM copier (not DTT_COPY_ENGINE)");
    if (p->other_dests || p->separate_dst)
        return fail(DTT_EINVAL, "dtt_allgather_host: needs chunks that land at their own offsets");
    if (out_rank >= p->P) return fail(DTT_EINVAL, "dtt_allgather_host: out_rank out of range");
    if (p->pending) return fail(DTT_ESTATE, "dtt_allgather_host: round %u is still pending: wait for it first", p->pending);
    const uint32_t P = p->P;
    const uint64_t S = p->buf_bytes / P;
    // the byte extent [lo, hi) of every chunk inside its rank's slice
    std::vector<uint64_t> lo, hi;
    chunk_extents(p, &lo, &hi);
    for (uint32_t c = 0; c < p->n_global; ++c) {
        const uint64_t base = (uint64_t)p->chunks[c].owner * S;
        if (hi[c]) {
            lo[c] -= base;
            hi[c] -= base;
        }
    }
    dtt_handle h[DTT_MAX_RANKS];
    p->notify_host = host_out != nullptr;        // the copier stamps each chunk's arrival
    int rc = dtt_plan_start(p, stream, h);
    if (rc == DTT_OK && p->opts.deferred_copier == 2) rc = dtt_plan_launch_copier(p);   // needed early
    p->notify_host = false;
    if (rc != DTT_OK) return rc;
    const uint32_t round = p->round;

    // Host to device in pieces; a chunk is marked as soon as the bytes it covers have landed, so
    // the copier fans it out while later pieces are still in flight.
    // pieces of a quarter of a slice, at least 4 MiB: the slices already pipeline one behind
    // the other, and every piece boundary costs the copy engine a pause
    const uint64_t kPiece = p->opts.host_piece_bytes
                                ? p->opts.host_piece_bytes
                                : std::max<uint64_t>(4ull << 20, (S / 4 + 4095) & ~uint64_t(4095));
    std::vector<uint64_t> copied(P, 0), back(P, 0);   // bytes copied in / copied back per slice
    std::vector<uint32_t> marked(P);
    for (uint32_t r = 0; r < P; ++r) {
        marked[r] = p->first_chunk[r];
        if (!host_slices[r]) copied[r] = S;
    }
    auto mark_ready_prefix = [&](uint32_t r) -> int {
        const uint32_t end = p->first_chunk[r] + p->n_chunks[r];
        uint32_t k = marked[r];
        while (k < end && hi[k] <= copied[r]) ++k;
        if (k == marked[r]) return DTT_OK;
        const int prc = dtt_publish(h, P, marked[r], k - marked[r], 0, stream);
        marked[r] = k;
        return prc;
    };
    // Device to host: rank out_rank's gathered buffer, each slice as far as every chunk of it
    // has arrived (out_rank's own slice as far as it was copied in).
    auto copy_back = [&](uint32_t r, uint64_t upto) -> int {
        if (upto <= back[r]) return DTT_OK;
        DTT_CUDA_TRY(cudaMemcpyAsync(static_cast<char*>(host_out) + r * S + back[r],
                                     p->bufs[out_rank] + r * S + back[r], upto - back[r],
                                     cudaMemcpyDeviceToHost, p->d2h_stream));
        back[r] = upto;
        return DTT_OK;
    };
    auto arrived_prefix = [&](uint32_t r) -> uint64_t {
        uint64_t x = S;
        for (uint32_t c = p->first_chunk[r]; c < p->first_chunk[r] + p->n_chunks[r]; ++c)
            if (__atomic_load_n(&p->h_arrived[c], __ATOMIC_ACQUIRE) != round) x = std::min(x, lo[c]);
        return x;
    };
    // the output rank's own pieces, each copied back once its copy in has completed (asked of
    // its event on the host, so no copy back queues behind a copy in on the device)
    std::vector<std::pair<size_t, uint64_t>> own;   // (event index, copied prefix)
    size_t own_next = 0;
    auto poll = [&](bool final) -> int {
        while (own_next < own.size()) {
            const cudaError_t e = final ? cudaEventSynchronize(p->ev_pieces[own[own_next].first])
                                        : cudaEventQuery(p->ev_pieces[own[own_next].first]);
            if (e == cudaErrorNotReady) break;
            if (e != cudaSuccess) return fail(DTT_ECUDA, "dtt_allgather_host: %s", cudaGetErrorString(e));
            const int prc = copy_back(out_rank, own[own_next++].second);
            if (prc != DTT_OK) return prc;
        }
        for (uint32_t r = 0; r < P; ++r) {
            if (r == out_rank) continue;
            const uint64_t x = arrived_prefix(r);
            // copies back of at least a host piece (or the slice's rest): on this GB300 a 4 MiB
            // copy out, beside copies in, ran at ~110 GB/s against ~140 GB/s for 8 MiB
            if (x == S || x >= back[r] + kPiece || (final && x > back[r])) {
                const int prc = copy_back(r, x);
                if (prc != DTT_OK) return prc;
            }
        }
        return DTT_OK;
    };
    for (uint32_t r = 0; r < P; ++r) {             // ranks without host data: as they stand
        if (host_slices[r]) continue;
        rc = mark_ready_prefix(r);
        if (rc != DTT_OK) return rc;
    }
    if (host_out && !host_slices[out_rank]) {
        DTT_CUDA_TRY(cudaEventRecord(p->ev_h2d, stream));
        DTT_CUDA_TRY(cudaStreamWaitEvent(p->d2h_stream, p->ev_h2d, 0));
        rc = copy_back(out_rank, S);
        if (rc != DTT_OK) return rc;
    }
    // the copies stream back to back on their own stream; the marks (kernels on `stream`) and
    // the copies back each wait for the piece they depend on
    DTT_CUDA_TRY(cudaEventRecord(p->ev_h2d, stream));       // after plan_start's work on `stream`
    DTT_CUDA_TRY(cudaStreamWaitEvent(p->h2d_stream, p->ev_h2d, 0));
    // slice by slice, so each slice (and the fan-out and copy back behind it) completes as early
    // as it can; pieces within a slice let its chunks open before the whole slice is in
    for (uint32_t r = 0; r < P; ++r) {
        while (copied[r] < S) {
            const uint64_t n = std::min(kPiece, S - copied[r]);
            DTT_CUDA_TRY(cudaMemcpyAsync(p->bufs[r] + r * S + copied[r],
                                         static_cast<const char*>(host_slices[r]) + copied[r], n,
                                         cudaMemcpyHostToDevice, p->h2d_stream));
            copied[r] += n;
            DTT_CUDA_TRY(cudaEventRecord(p->ev_h2d, p->h2d_stream));
            const uint32_t before = marked[r];
            const uint32_t end = p->first_chunk[r] + p->n_chunks[r];
            if (before < end && hi[before] <= copied[r]) {
                DTT_CUDA_TRY(cudaStreamWaitEvent(stream, p->ev_h2d, 0));
                rc = mark_ready_prefix(r);
                if (rc != DTT_OK) return rc;
            }
            if (host_out && r == out_rank) {        // its own bytes go back once they are in
                if (own.size() == p->ev_pieces.size()) {
                    cudaEvent_t e = nullptr;
                    DTT_CUDA_TRY(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
                    p->ev_pieces.push_back(e);
                }
                DTT_CUDA_TRY(cudaEventRecord(p->ev_pieces[own.size()], p->h2d_stream));
                own.emplace_back(own.size(), copied[r]);
            }
            if (host_out && (rc = poll(false)) != DTT_OK) return rc;
        }
    }
    DTT_CUDA_TRY(cudaStreamWaitEvent(stream, p->ev_h2d, 0));   // every copy precedes the check
    if (host_out) {
        // the rest as it arrives; once the copier has exited, whatever arrived is final
        for (uint64_t spin = 1;; ++spin) {
            if ((rc = poll(false)) != DTT_OK) return rc;
            bool all = true;
            for (uint32_t r = 0; r < P; ++r) all = all && back[r] == S;
            if (all) break;
            if ((spin & 1023) == 0) {
                const cudaError_t e = cudaEventQuery(p->ev_copier_end);
                if (e == cudaSuccess) break;
                if (e != cudaErrorNotReady)
                    return fail(DTT_ECUDA, "dtt_allgather_host: %s", cudaGetErrorString(e));
            }
        }
        if ((rc = poll(true)) != DTT_OK) return rc;
    }
    p->suppress_early = true;
    rc = dtt_plan_wait(p, report);
    p->suppress_early = false;
    if (rc != DTT_OK) {
        cudaStreamSynchronize(p->d2h_stream);
        return rc;
    }
    if (host_out) {
        DTT_CUDA_TRY(cudaStreamSynchronize(p->d2h_stream));
        for (uint32_t r = 0; r < P; ++r)
            if (back[r] != S) return fail(DTT_ETIMEDOUT, "dtt_allgather_host: slice %u came back short", r);
    }
    return dtt_plan_next_round(p);
}

namespace {

// One round of dtt_allgather_host_rounds: its host buffers and how far each slice has gone in
// (copied), been marked and come back (back), with the copy-back events later rounds gate on.
struct HostRound {
    uint32_t R = 0;
    bool started = false, checked = false;
    dtt_handle h[DTT_MAX_RANKS];
    const void* const* slices = nullptr;    // P host pointers (NULL: the slice as it stands)
    char* out = nullptr;                    // the output rank's gathered buffer (or NULL)
    uint64_t copied[DTT_MAX_RANKS] = {}, back[DTT_MAX_RANKS] = {};
    uint32_t marked[DTT_MAX_RANKS] = {};
    // per slice: (prefix copied back once the copy is done, event after that copy)
    std::vector<std::pair<uint64_t, cudaEvent_t>> d2h[DTT_MAX_RANKS];
    // the output rank's own pieces: (prefix copied in, event after that copy)
    std::vector<std::pair<uint64_t, cudaEvent_t>> own;
    size_t own_next = 0;
    cudaEvent_t copier_end = nullptr;       // after this round's copier on the copy stream
};

cudaEvent_t take_event(dtt_plan* p) {
    if (!p->ev_free.empty()) {
        cudaEvent_t e = p->ev_free.back();
        p->ev_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    return cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess ? e : nullptr;
}

void give_events(dtt_plan* p, HostRound& x) {
    for (auto& v : x.d2h) {
        for (auto& pe : v) p->ev_free.push_back(pe.second);
        v.clear();
    }
    for (auto& pe : x.own) p->ev_free.push_back(pe.second);
    x.own.clear();
    if (x.copier_end) p->ev_free.push_back(x.copier_end);
    x.copier_end = nullptr;
}

// The event after the first copy back of slice r that reaches `upto`, or nullptr if none has
// been issued yet.
cudaEvent_t back_event(const HostRound& x, uint32_t r, uint64_t upto) {
    for (const auto& pe : x.d2h[r])
        if (pe.first >= upto) return pe.second;
    return nullptr;
}

}  // namespace

int dtt_allgather_host_rounds(dtt_plan* p, uint32_t n_rounds, const void* const* host_slices,
                              void* const* host_outs, uint32_t out_rank, cudaStream_t stream,
                              dtt_report* reports) {
    if (!p || !host_slices) return fail(DTT_EINVAL, "dtt_allgather_host_rounds: bad args");
    if (!p->opts.overlap) return fail(DTT_EINVAL, "dtt_allgather_host_rounds: needs a plan with overlapping rounds");
    if (!p->opts.allgather) return fail(DTT_EINVAL, "dtt_allgather_host_rounds: needs an all-gather plan");
    if (p->ce) return fail(DTT_EINVAL, "dtt_allgather_host_rounds: needs an SM copier (not DTT_COPY_ENGINE)");
    if (p->other_dests || p->separate_dst)
        return fail(DTT_EINVAL, "dtt_allgather_host_rounds: needs chunks that land at their own offsets");
    if (out_rank >= p->P) return fail(DTT_EINVAL, "dtt_allgather_host_rounds: out_rank out of range");
    if (p->state != DTT_PLAN_PREPARED || p->pending)
        return fail(DTT_ESTATE, "dtt_allgather_host_rounds: needs a PREPARED plan with no round pending");
    if (n_rounds == 0) return DTT_OK;
    if ((uint64_t)p->round + n_rounds - 1 > 0xFFFFFFFFull)
        return fail(DTT_EROUNDLIMIT, "dtt_allgather_host_rounds: the rounds would pass 2^32 - 1");
    const uint32_t P = p->P;
    const uint64_t S = p->buf_bytes / P;
    std::vector<uint64_t> lo, hi;            // each chunk's byte extent inside its rank's slice
    chunk_extents(p, &lo, &hi);
    for (uint32_t c = 0; c < p->n_global; ++c) {
        const uint64_t base = (uint64_t)p->chunks[c].owner * S;
        if (hi[c]) {
            lo[c] -= base;
            hi[c] -= base;
        }
    }
    // a whole slice per copy unless asked otherwise: the rounds overlap one another, so a round
    // needs no finer pieces, and larger copies move faster over the host link (c2: 436 GB/s with
    // 8 MiB pieces, 476 GB/s with whole 32 MiB slices)
    const uint64_t kPiece = p->opts.host_piece_bytes ? p->opts.host_piece_bytes
                                                     : std::max<uint64_t>(4ull << 20, (S + 4095) & ~uint64_t(4095));
    std::vector<HostRound> rounds(n_rounds);
    for (uint32_t k = 0; k < n_rounds; ++k) {
        HostRound& x = rounds[k];
        x.slices = host_slices + (size_t)k * P;
        x.out = host_outs ? static_cast<char*>(host_outs[k]) : nullptr;
        for (uint32_t r = 0; r < P; ++r) {
            x.marked[r] = p->first_chunk[r];
            if (!x.slices[r]) x.copied[r] = S;
        }
    }
    int rc = DTT_OK;
    auto fail_all = [&](int code) -> int {
        for (HostRound& x : rounds) give_events(p, x);
        return code;
    };

    // Start round k: its copier (queued behind the round in flight, if any) stamps each chunk's
    // arrival into mapped host memory.
    auto start_round = [&](HostRound& x) -> int {
        p->notify_host = true;
        int src = dtt_plan_start(p, stream, x.h);
        if (src == DTT_OK && p->opts.deferred_copier == 2) src = dtt_plan_launch_copier(p);
        p->notify_host = false;
        if (src != DTT_OK) return src;
        x.R = p->round;
        x.started = true;
        x.copier_end = take_event(p);
        if (!x.copier_end) return fail(DTT_ECUDA, "dtt_allgather_host_rounds: cannot create an event");
        DTT_CUDA_TRY(cudaEventRecord(x.copier_end, p->copy_stream));
        return DTT_OK;
    };
    // Rank r's chunks [marked, k) whose bytes are all in go to the copier.  prev: the round
    // before, still coming back: a chunk's copies land in the output rank's buffer, so they wait
    // (on the device) for that round's copy back of the same bytes.
    auto publish = [&](HostRound& x, const HostRound* prev, uint32_t r) -> int {
        const uint32_t end = p->first_chunk[r] + p->n_chunks[r];
        uint32_t k = x.marked[r];
        while (k < end && hi[k] <= x.copied[r]) ++k;
        if (k == x.marked[r]) return DTT_OK;
        if (prev && prev->out && r != out_rank) {
            uint32_t q = x.marked[r];
            while (q < k) {                       // as far as that round's copies back reach
                cudaEvent_t e = back_event(*prev, r, hi[q]);
                if (!e) break;
                uint32_t q2 = q;
                while (q2 < k && back_event(*prev, r, hi[q2]) == e) ++q2;
                DTT_CUDA_TRY(cudaStreamWaitEvent(stream, e, 0));
                const int prc = dtt_publish(x.h, P, q, q2 - q, 0, stream);
                if (prc != DTT_OK) return prc;
                q = q2;
            }
            x.marked[r] = q;
            return DTT_OK;
        }
        const int prc = dtt_publish(x.h, P, x.marked[r], k - x.marked[r], 0, stream);
        x.marked[r] = k;
        return prc;
    };
    // Copy in the next piece of rank r's slice if it may be overwritten: the round before has
    // delivered every chunk it touches, and (the output rank's own slice) copied those bytes back.
    auto copy_in = [&](HostRound& x, const HostRound* prev, uint32_t r) -> int {
        if (x.copied[r] >= S) return DTT_OK;
        const uint64_t a = x.copied[r], n = std::min(kPiece, S - a), b = a + n;
        if (prev) {
            for (uint32_t c = p->first_chunk[r]; c < p->first_chunk[r] + p->n_chunks[r]; ++c)
                if (hi[c] && lo[c] < b && hi[c] > a &&
                    __atomic_load_n(&p->h_arrived[c], __ATOMIC_ACQUIRE) < prev->R)
                    return DTT_OK;                // still being sent: not yet
            if (prev->out && r == out_rank) {
                cudaEvent_t e = back_event(*prev, r, b);
                if (!e) return DTT_OK;            // not yet copied back
                DTT_CUDA_TRY(cudaStreamWaitEvent(p->h2d_stream, e, 0));
            }
        }
        DTT_CUDA_TRY(cudaMemcpyAsync(p->bufs[r] + r * S + a, static_cast<const char*>(x.slices[r]) + a, n,
                                     cudaMemcpyHostToDevice, p->h2d_stream));
        x.copied[r] = b;
        DTT_CUDA_TRY(cudaEventRecord(p->ev_h2d, p->h2d_stream));
        DTT_CUDA_TRY(cudaStreamWaitEvent(stream, p->ev_h2d, 0));
        if (x.out && r == out_rank) {
            cudaEvent_t e = take_event(p);
            if (!e) return fail(DTT_ECUDA, "dtt_allgather_host_rounds: cannot create an event");
            DTT_CUDA_TRY(cudaEventRecord(e, p->h2d_stream));
            x.own.emplace_back(b, e);
        }
        return publish(x, prev, r);
    };
    // Copy back slice r of the output rank's buffer up to `upto`.
    auto copy_back = [&](HostRound& x, uint32_t r, uint64_t upto) -> int {
        if (upto <= x.back[r]) return DTT_OK;
        DTT_CUDA_TRY(cudaMemcpyAsync(x.out + r * S + x.back[r], p->bufs[out_rank] + r * S + x.back[r],
                                     upto - x.back[r], cudaMemcpyDeviceToHost, p->d2h_stream));
        x.back[r] = upto;
        cudaEvent_t e = take_event(p);
        if (!e) return fail(DTT_ECUDA, "dtt_allgather_host_rounds: cannot create an event");
        DTT_CUDA_TRY(cudaEventRecord(e, p->d2h_stream));
        x.d2h[r].emplace_back(upto, e);
        return DTT_OK;
    };
    // Copies back as far as chunks have arrived (the output rank's own pieces once copied in).
    // final: the round's copier has exited, so whatever arrived is all there is.
    auto come_back = [&](HostRound& x, bool final) -> int {
        if (!x.out) return DTT_OK;
        while (x.own_next < x.own.size()) {
            const cudaError_t e = cudaEventQuery(x.own[x.own_next].second);
            if (e == cudaErrorNotReady) break;
            if (e != cudaSuccess) return fail(DTT_ECUDA, "dtt_allgather_host_rounds: %s", cudaGetErrorString(e));
            const int prc = copy_back(x, out_rank, x.own[x.own_next++].first);
            if (prc != DTT_OK) return prc;
        }
        if (!x.slices[out_rank] && x.back[out_rank] < S) {     // its rows as they stand
            const int prc = copy_back(x, out_rank, S);
            if (prc != DTT_OK) return prc;
        }
        for (uint32_t r = 0; r < P; ++r) {
            if (r == out_rank) continue;
            // a chunk's stamp is the round of its last arrival everywhere: this round's, or (for
            // bytes already copied back) the next round's
            uint64_t upto = S;
            for (uint32_t c = p->first_chunk[r]; c < p->first_chunk[r] + p->n_chunks[r]; ++c)
                if (hi[c] > x.back[r] && __atomic_load_n(&p->h_arrived[c], __ATOMIC_ACQUIRE) < x.R)
                    upto = std::min(upto, lo[c]);
            if (upto == S || upto >= x.back[r] + kPiece || (final && upto > x.back[r])) {
                const int prc = copy_back(x, r, upto);
                if (prc != DTT_OK) return prc;
            }
        }
        return DTT_OK;
    };
    auto all_in = [&](const HostRound& x) {
        for (uint32_t r = 0; r < P; ++r)
            if (x.copied[r] < S || x.marked[r] < p->first_chunk[r] + p->n_chunks[r]) return false;
        return true;
    };
    auto all_back = [&](const HostRound& x) {
        if (!x.out) return true;
        for (uint32_t r = 0; r < P; ++r)
            if (x.back[r] < S) return false;
        return true;
    };

    // Round k's bytes go in, are marked, fanned out and come back while round k + 1's go in
    // behind them; round k is checked (the pending round) once it has come back.
    DTT_CUDA_TRY(cudaEventRecord(p->ev_h2d, stream));      // after the caller's work on `stream`
    DTT_CUDA_TRY(cudaStreamWaitEvent(p->h2d_stream, p->ev_h2d, 0));
    if ((rc = start_round(rounds[0])) != DTT_OK) return fail_all(rc);
    uint32_t cur = 0;                         // the oldest round not yet checked
    for (uint64_t spin = 1; cur < n_rounds; ++spin) {
        HostRound& x = rounds[cur];
        HostRound* y = cur + 1 < n_rounds ? &rounds[cur + 1] : nullptr;
        const HostRound* before = cur > 0 && !rounds[cur - 1].checked ? &rounds[cur - 1] : nullptr;
        for (uint32_t r = 0; r < P && rc == DTT_OK; ++r) {
            while (x.copied[r] < S && rc == DTT_OK) {
                const uint64_t was = x.copied[r];
                rc = copy_in(x, before, r);
                if (x.copied[r] == was) break;
            }
            if (rc == DTT_OK) rc = publish(x, before, r);
        }
        if (rc == DTT_OK) rc = come_back(x, false);
        // the next round starts once this one is all in: this round is left pending
        if (rc == DTT_OK && y && !y->started && all_in(x)) {
            rc = dtt_plan_next_round(p);
            if (rc == DTT_OK) rc = start_round(*y);
        }
        if (rc == DTT_OK && y && y->started) {
            for (uint32_t r = 0; r < P && rc == DTT_OK; ++r) {
                while (y->copied[r] < S && rc == DTT_OK) {
                    const uint64_t was = y->copied[r];
                    rc = copy_in(*y, &x, r);
                    if (y->copied[r] == was) break;
                }
                if (rc == DTT_OK) rc = publish(*y, &x, r);
            }
            if (rc == DTT_OK) rc = come_back(*y, false);
        }
        if (rc != DTT_OK) return fail_all(rc);
        bool done_back = all_in(x) && all_back(x);
        if (!done_back && (spin & 1023) == 0) {
            const cudaError_t e = cudaEventQuery(x.copier_end);
            if (e == cudaSuccess) {               // nothing more will arrive
                if ((rc = come_back(x, true)) != DTT_OK) return fail_all(rc);
                done_back = true;
            } else if (e != cudaErrorNotReady) {
                return fail_all(fail(DTT_ECUDA, "dtt_allgather_host_rounds: %s", cudaGetErrorString(e)));
            }
        }
        if (done_back && all_in(x)) {
            // check round x: the pending one when the next has started, else the current one
            DTT_CUDA_TRY(cudaStreamWaitEvent(stream, p->ev_h2d, 0));   // every copy in precedes the check
            p->suppress_early = true;
            rc = dtt_plan_wait(p, reports ? &reports[cur] : nullptr);
            p->suppress_early = false;
            if (rc != DTT_OK) {
                cudaStreamSynchronize(p->d2h_stream);
                return fail_all(rc);
            }
            x.checked = true;
            if (x.out) {
                DTT_CUDA_TRY(cudaStreamSynchronize(p->d2h_stream));
                for (uint32_t r = 0; r < P; ++r)
                    if (x.back[r] != S)
                        return fail_all(fail(DTT_ETIMEDOUT, "dtt_allgather_host_rounds: round %u's slice %u came back short",
                                             x.R, r));
            }
            if (cur > 0) give_events(p, rounds[cur - 1]);
            ++cur;
            if (cur < n_rounds && !rounds[cur].started) {     // a round of its own: nothing pending
                rc = dtt_plan_next_round(p);
                if (rc == DTT_OK) rc = start_round(rounds[cur]);
                if (rc != DTT_OK) return fail_all(rc);
            }
        }
    }
    give_events(p, rounds[n_rounds - 1]);
    if (n_rounds > 1) give_events(p, rounds[n_rounds - 2]);
    return dtt_plan_next_round(p);
}

int dtt_gemm_consumer(dtt_plan* p, uint32_t rank, const void* Wt, uint32_t N, uint32_t K, void* D,
                      uint64_t ldd, uint32_t num_programs, uint64_t max_polls, uint32_t* err,
                      cudaStream_t stream) {
    if (!p || !Wt || !D || !err || rank >= p->P) return fail(DTT_EINVAL, "dtt_gemm_consumer: bad args");
    if (p->state != DTT_PLAN_RUNNING) return fail(DTT_ESTATE, "dtt_gemm_consumer: plan is not RUNNING");
    if (stream == p->copy_stream) return fail(DTT_EINVAL, "dtt_gemm_consumer: use a stream other than the copy stream");
    if (p->other_dests || p->separate_dst)
        return fail(DTT_EINVAL, "dtt_gemm_consumer: needs chunks that land at their own offsets");
    const uint64_t row_bytes = 2ull * K;
    if (N == 0 || K == 0 || N % 128 || K % 64 || p->buf_bytes % (row_bytes * 128))
        return fail(DTT_EINVAL, "dtt_gemm_consumer: N must be a multiple of 128, K of 64, and the buffer "
                                "a whole number of 128-row blocks of K bf16");
    if (ldd < 2ull * N || ldd % 16 || reinterpret_cast<uintptr_t>(D) % 16 || reinterpret_cast<uintptr_t>(Wt) % 16)
        return fail(DTT_EINVAL, "dtt_gemm_consumer: bad ldd or alignment");
    const uint64_t rows = p->buf_bytes / row_bytes;
    const uint32_t blocks = (uint32_t)(rows / 128);
    // with block groups of this block size, each block is one group wait
    const bool grouped = p->n_groups && p->group_block_bytes == 128 * row_bytes &&
                         p->block_group.size() >= blocks;
    if (!p->d_cons || p->cons_rank != rank || p->cons_K != K || p->cons_grouped != grouped) {
        // which chunks cover each block, and the blocks in the order their chunks open: by the
        // chunk's place in its rank's schedule, then by rank
        std::vector<uint64_t> lo, hi;
        chunk_extents(p, &lo, &hi);
        std::vector<uint32_t> c0(blocks, 1), c1(blocks, 0), key(blocks, UINT32_MAX), order(blocks);
        const uint64_t bb = 128 * row_bytes;
        for (uint32_t c = 0; c < p->n_global; ++c) {
            if (!hi[c]) continue;
            const uint32_t owner = p->chunks[c].owner, local = c - p->first_chunk[owner];
            for (uint64_t b = lo[c] / bb; b < blocks && b * bb < hi[c]; ++b) {
                if (c0[b] > c1[b]) c0[b] = c1[b] = c;
                c0[b] = std::min(c0[b], c);
                c1[b] = std::max(c1[b], c);
                key[b] = std::min(key[b], local * DTT_MAX_RANKS + owner);
            }
        }
        for (uint32_t b = 0; b < blocks; ++b) order[b] = b;
        std::stable_sort(order.begin(), order.end(), [&](uint32_t x, uint32_t y) { return key[x] < key[y]; });
        // pairs of blocks (2 pb, 2 pb + 1) for the pair form, in the order their later half is taken
        std::vector<uint32_t> pos(blocks), order2(blocks / 2), late(blocks / 2);
        for (uint32_t i = 0; i < blocks; ++i) pos[order[i]] = i;
        for (uint32_t pb = 0; pb < blocks / 2; ++pb) {
            order2[pb] = pb;
            late[pb] = std::max(pos[2 * pb], pos[2 * pb + 1]);
        }
        std::stable_sort(order2.begin(), order2.end(), [&](uint32_t x, uint32_t y) { return late[x] < late[y]; });
        std::vector<uint32_t> table;
        table.reserve(4 * (size_t)blocks + blocks / 2 + 1);
        table.insert(table.end(), order.begin(), order.end());
        table.insert(table.end(), c0.begin(), c0.end());
        table.insert(table.end(), c1.begin(), c1.end());
        table.insert(table.end(), order2.begin(), order2.end());
        table.push_back(0);
        if (grouped) table.insert(table.end(), p->block_group.begin(), p->block_group.begin() + blocks);
        else table.insert(table.end(), blocks, 0u);
        if (p->d_cons && p->cons_cap < blocks) {
            DTT_CUDA_TRY(cudaFreeAsync(p->d_cons, stream));
            p->d_cons = nullptr;
        }
        // stream-ordered: no wait for the rest of the device, where a copier may be spinning
        if (!p->d_cons) {
            DTT_CUDA_TRY(cudaMallocAsync(reinterpret_cast<void**>(&p->d_cons), table.size() * sizeof(uint32_t), stream));
            p->cons_cap = blocks;
        }
        p->cons_blocks = blocks;
        DTT_CUDA_TRY(cudaMemcpyAsync(p->d_cons, table.data(), table.size() * sizeof(uint32_t),
                                     cudaMemcpyHostToDevice, stream));
        p->cons_rank = rank;
        p->cons_K = K;
        p->cons_grouped = grouped;
    }
    ConsumerLaunch cl{};
    cl.X = p->bufs[rank];
    cl.rows = rows;
    cl.Wt = Wt;
    cl.N = N;
    cl.K = K;
    cl.D = static_cast<char*>(D);
    cl.ldd = ldd;
    cl.h = make_handle(p, rank);
    cl.order = p->d_cons;
    cl.c0 = p->d_cons + p->cons_blocks;
    cl.c1 = p->d_cons + 2 * (size_t)p->cons_blocks;
    cl.order2 = p->d_cons + 3 * (size_t)p->cons_blocks;
    cl.bgroup = grouped ? p->d_cons + 3 * (size_t)p->cons_blocks + p->cons_blocks / 2 + 1 : nullptr;
    cl.blocks = blocks;
    cl.max_polls = max_polls ? max_polls : p->opts.max_polls;
    cl.err = err;
    cl.ctas = num_programs ? num_programs : 148;
    // room beside the copier: an SM has 228 KiB of shared memory, 1 KiB of it reserved per CTA
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device);
    uint64_t copier_smem = 0;
    if (p->opts.method == DTT_COPY_TMA && sms > 0) {
        const uint64_t per_sm = (p->copier_ctas + (uint32_t)sms - 1) / (uint32_t)sms;
        copier_smem = per_sm * (bulk_smem_bytes(bulk_stage_bytes(p->opts.piece_bytes), p->opts.stages) + 1024);
    }
    cl.smem_budget = copier_smem + 2048 < 228 * 1024 ? 228 * 1024 - copier_smem - 1024 : 0;
    return launch_gemm_consumer(cl, stream);
}

int dtt_consumer_gather(dtt_plan* p, uint32_t rank, void* dst, uint64_t max_polls, int32_t* status,
                        uint32_t ctas, cudaStream_t stream) {
    if (!p || !dst || !status || rank >= p->P) return fail(DTT_EINVAL, "dtt_consumer_gather: bad args");
    if (p->state != DTT_PLAN_RUNNING) return fail(DTT_ESTATE, "dtt_consumer_gather: plan is not RUNNING");
    if (stream == p->copy_stream) return fail(DTT_EINVAL, "dtt_consumer_gather: use a stream other than the copy stream");
    if (!p->n_global) return DTT_OK;
    const CopierParams cp = copier_params(p, p->round);
    DTT_CUDA_TRY(launch_consumer(cp, make_handle(p, rank), static_cast<char*>(dst), max_polls, status, ctas, stream));
    return DTT_OK;
}

}  // extern "C"
