/*
 * dtt.h -- C ABI of the GB300-native triggered-plan library (device-triggered transfers).
 *
 * A triggered plan sends the output of a running producer kernel to every other rank without
 * a host round trip per chunk: the producer marks each chunk of its output ready once it is
 * written, and a copier moves the chunk to the same offsets in every peer's buffer and then
 * signals its arrival there (Iris docs, "Triggered Plans", introduction and section Model;
 * ROCm/iris pull 573, "Triggered SDMA Plans", introduction).  On one GB300 the P ranks are
 * virtual ranks: P buffers of one size in the GPU's own HBM, driven by one process.  The
 * copier is a persistent CUDA kernel that polls the gates (it stands where the pages use a
 * copy engine's poll / copy / atomic packet chain).
 *
 * Conventions shared by every call:
 *  - Return value: DTT_OK (0) or a negative DTT_E* code; dtt_last_error() then gives a message
 *    (thread-local, valid until the next failing call on the same thread).
 *  - Pointers named "device" are CUDA device addresses in the current device's context;
 *    "host" pointers are ordinary (or pinned, where stated) host memory.  Streams are
 *    cudaStream_t handles owned by the caller unless stated.
 *  - Byte offsets inside a buffer are relative to the buffer's first byte.
 *  - Nothing here takes a framework (torch) type.
 */
#ifndef DTT_H
#define DTT_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------------------------------- */
/* Limits and codes                                                                          */
/* ---------------------------------------------------------------------------------------- */

#define DTT_MAX_RANKS 16        /* virtual ranks per plan */
#define DTT_REPORT_MAX 64       /* chunk ids listed in a dtt_report */
#define DTT_LINEAR_MAX (1ull << 30)  /* linear regions are split at 1 GiB ("Triggered Plans",
                                        section Model and section Requirements and limits) */

enum {
    DTT_CLOSING = 1,       /* not an error: dtt_plan_close left the plan CLOSING (see there) */
    DTT_OK = 0,
    DTT_EINVAL = -1,       /* invalid argument */
    DTT_EOUTOFROWS = -2,   /* all-gather: a schedule leaves its rank's own rows
                              ("Triggered Plans", section Model, prepare_all_gather) */
    DTT_EOVERLAP = -3,     /* two ranks send the same bytes
                              ("Triggered Plans", section Requirements and limits) */
    DTT_ECAPACITY = -4,    /* plan larger than its configured capacity */
    DTT_EROUNDLIMIT = -5,  /* round would pass 2^32 - 1 ("Triggered Plans", Gates and rounds) */
    DTT_ESTATE = -6,       /* call not valid in the plan's current state */
    DTT_EEXTRA = -7,       /* a chunk got more marks than its writers
                              ("Triggered Plans", The kernel author's contract, item 2) */
    DTT_ETIMEDOUT = -8,    /* a wait gave up; the report names the short chunks (same item) */
    DTT_ECUDA = -9,        /* a CUDA runtime call failed (message has the CUDA error) */
    DTT_ENOMEM = -10       /* host or device allocation failed */
};

/* Plan states ("Triggered Plans", The kernel author's contract: done / FAILED / CLOSING). */
enum {
    DTT_PLAN_PREPARED = 0, /* created or advanced by next_round; start() is next */
    DTT_PLAN_RUNNING = 1,  /* start() launched this round's copier */
    DTT_PLAN_DONE = 2,     /* wait() found every chunk delivered */
    DTT_PLAN_FAILED = 3,   /* wait() found extra marks or short chunks; only close() is valid */
    DTT_PLAN_CLOSING = 4,  /* close() opened its gates, but its copier waits behind an earlier
                              plan's copier on the same copy stream */
    DTT_PLAN_CLOSED = 5
};

/* Element types of the library's producers. */
enum { DTT_BF16 = 0, DTT_F32 = 1, DTT_U8 = 2 };

/* Copier data paths. */
enum {
    DTT_COPY_VEC16 = 0,    /* 16-byte vector loads and stores, read once, fan out to peers */
    DTT_COPY_TMA = 1,      /* bulk async copies (cp.async.bulk) staged through shared memory */
    DTT_COPY_ENGINE = 2    /* the GPU's copy engines, driven by a host proxy thread of the plan
                              (no copier kernel): the closest CUDA analogue of the pages' copy-engine
                              queues.  The producer's gate-opening mark also stamps the round into
                              a mapped host word; the proxy polls those words in schedule order
                              (POLL_REGMEM), issues one cudaMemcpyAsync / cudaMemcpy2DAsync per
                              region and peer on one stream per (source, peer) queue (COPY), and
                              once the chunk's copies to every peer are done a one-warp kernel adds
                              its arrivals, group counts and completion (ATOMIC).  Consecutive open
                              chunks of a source whose bytes follow each other on both sides (up to
                              64 MiB) go as one copy per peer and one signal kernel.  Each source
                              byte is read once per peer.  dtt_allgather_host needs an SM copier. */
};

/* ---------------------------------------------------------------------------------------- */
/* Regions, chunks and schedules ("Triggered Plans", section Model)                          */
/* ---------------------------------------------------------------------------------------- */

/* One copy: `rows` rows of `row_bytes` bytes, `pitch` bytes apart, starting at byte
 * `offset` of the buffer.  A byte range has rows == 1 and pitch == row_bytes.  The copy lands
 * at the same offset in every peer's buffer. */
typedef struct dtt_region {
    uint64_t offset;
    uint64_t row_bytes;
    uint64_t rows;
    uint64_t pitch;
} dtt_region;

/* A host-side list of chunks (ordered groups of regions, each with its writer count), in
 * the order the producer completes them.  Opaque; owned by the caller, freed with
 * dtt_schedule_free.  A plan copies what it needs at creation. */
typedef struct dtt_schedule dtt_schedule;

/* Producer step-to-tile order shared by the host builder and the library's producers, so
 * the two cannot drift ("Triggered Plans", section Model: pass the kernel's own mapping).
 * kind DTT_ORDER_ROW_MAJOR: step s -> (s / tiles_n, s % tiles_n).
 * kind DTT_ORDER_GROUPED: groups of group_m tile rows swept column by column: with
 *   g = s / (group_m * tiles_n), m0 = g * group_m, h = min(tiles_m - m0, group_m),
 *   w = s % (group_m * tiles_n):  tm = m0 + w % h,  tn = w / h. */
enum { DTT_ORDER_ROW_MAJOR = 0, DTT_ORDER_GROUPED = 1 };
typedef struct dtt_order {
    uint32_t kind;
    uint32_t group_m;
} dtt_order;

/* A caller-supplied step-to-tile map for hand-written producers (host only).  Returns 0 and
 * writes (tm, tn) for `step`. */
typedef int (*dtt_order_fn)(uint64_t step, void* ctx, uint32_t* tm, uint32_t* tn);

/* The builtin order on the host (the same function the library's producers run).
 * Errors: DTT_EINVAL for an unknown kind, group_m == 0 with kind GROUPED, or step >= tiles. */
int dtt_tile_of(const dtt_order* order, uint64_t step, uint32_t tiles_m, uint32_t tiles_n,
                uint32_t* tm, uint32_t* tn);

/* whole(): one chunk holding the block of `rows` rows (row_bytes each, pitch apart) at
 * base_off, marked once by each of `num_programs` programs at their end: writers =
 * num_programs ("Triggered Plans", section Model).  Contiguous rows form one byte range split
 * into 1 GiB pieces, strided rows one 2D region.  Errors: DTT_EINVAL (num_programs == 0,
 * pitch < row_bytes with rows > 1). */
int dtt_schedule_whole(uint64_t base_off, uint64_t rows, uint64_t row_bytes, uint64_t pitch,
                       uint32_t num_programs, dtt_schedule** out);

/* chunks(): row blocks completed in order, one writer each ("Triggered Plans", section Model).
 * Block size is ceil(rows / num_chunks) rows, the last block shorter (so fewer chunks than
 * asked can result when the division is uneven; dtt_schedule_info reports the count).
 * Errors: DTT_EINVAL (num_chunks == 0 or > rows, pitch < row_bytes). */
int dtt_schedule_chunks(uint64_t base_off, uint64_t rows, uint64_t row_bytes, uint64_t pitch,
                        uint32_t num_chunks, dtt_schedule** out);

/* tile_chunks(): consecutive steps of a tiled producer over an M x N slice of elem_bytes
 * elements whose rows are pitch bytes apart, starting at base_off.  Step s stores tile
 * (tm, tn) given by `fn(s, ctx)` when fn is non-NULL, else by the builtin `order` (NULL means
 * row-major).  Each tile is one 2D region clipped at the slice edges; chunk k holds steps
 * [k*tiles_per_chunk, (k+1)*tiles_per_chunk) and has one writer per step ("Triggered Plans",
 * section Model: the producer marks first_chunk + step / num_programs).  Errors: DTT_EINVAL
 * (zero sizes, order not a bijection onto the tiles). */
int dtt_schedule_tile_chunks(uint64_t base_off, uint64_t M, uint64_t N, uint32_t elem_bytes,
                             uint64_t pitch, uint32_t BM, uint32_t BN, uint32_t tiles_per_chunk,
                             const dtt_order* order, dtt_order_fn fn, void* ctx,
                             dtt_schedule** out);

/* An empty schedule: a rank that sends nothing (a broadcast's receivers, "Triggered Plans",
 * section Requirements and limits), or the start of a hand-built schedule. */
int dtt_schedule_empty(dtt_schedule** out);

/* Append one chunk of n regions (copied) with `writers` marks per round.  Byte ranges longer
 * than 1 GiB are split here.  Errors: DTT_EINVAL (writers == 0, n == 0, pitch < row_bytes). */
int dtt_schedule_add_chunk(dtt_schedule* s, const dtt_region* regions, uint32_t n,
                           uint32_t writers);

/* Where a region lands: the same rows of the same width, at byte `offset` of the receiving
 * rank's buffer (or of its destination buffer, dtt_plan_opts.dst_bufs), rows `pitch` apart. */
typedef struct dtt_dest {
    uint64_t offset;
    uint64_t pitch;
} dtt_dest;

/* Other destinations ("Triggered Plans", Not supported yet: a copy could not change offset, pitch
 * or buffer, and a chunk could not go to only some peers; reduce-scatter and two-shot all-reduce
 * need both).  As dtt_schedule_add_chunk, and in addition:
 *  - dests (NULL: every region lands at its own offsets): one destination per region;
 *  - peer_mask: bit q set = rank q receives the chunk (DTT_ALL_PEERS = every other rank); the
 *    owner's bit is ignored.  Only the receivers get arrivals; completion counts them.
 * A byte range is split at 1 GiB together with its destination when both are contiguous.
 * The plan checks destinations at create (see dtt_plan_create).
 * Errors: DTT_EINVAL (as dtt_schedule_add_chunk; a destination pitch below the row bytes). */
#define DTT_ALL_PEERS 0u
int dtt_schedule_add_chunk_to(dtt_schedule* s, const dtt_region* regions, const dtt_dest* dests,
                              uint32_t n, uint32_t writers, uint32_t peer_mask);

/* A chunk's destinations (dests_out: at most cap of them; *n_dests = the chunk's region count,
 * or 0 when its regions land at their own offsets) and its peer mask (DTT_ALL_PEERS or the bits
 * given).  Errors: DTT_EINVAL. */
int dtt_schedule_get_dests(const dtt_schedule* s, uint32_t chunk, dtt_dest* dests_out,
                           uint64_t cap, uint64_t* n_dests, uint32_t* peer_mask);

/* Number of chunks and regions. */
int dtt_schedule_info(const dtt_schedule* s, uint32_t* n_chunks, uint64_t* n_regions);

/* Copy chunk `chunk`'s regions into regions_out (at most cap of them) and its writer count;
 * *n_regions receives the chunk's region count. */
int dtt_schedule_get(const dtt_schedule* s, uint32_t chunk, dtt_region* regions_out,
                     uint64_t cap, uint64_t* n_regions, uint32_t* writers);

void dtt_schedule_free(dtt_schedule* s);

/* ---------------------------------------------------------------------------------------- */
/* Plans ("Triggered Plans", sections Model, The kernel author's contract, Gates and rounds)  */
/* ---------------------------------------------------------------------------------------- */

typedef struct dtt_plan dtt_plan;

typedef struct dtt_plan_opts {
    uint32_t allgather;      /* 1: rank r's regions must lie in bytes [r*S, (r+1)*S), S =
                                buf_bytes / P (prepare_all_gather's check); 0: only bounds */
    uint32_t method;         /* DTT_COPY_VEC16 or DTT_COPY_TMA */
    uint32_t copier_ctas;    /* copier CTAs; 0 = SM count x ctas_per_sm */
    uint32_t ctas_per_sm;    /* used when copier_ctas == 0; 0 = 1 */
    uint32_t copier_threads; /* threads per copier CTA (multiple of 32, <= 1024); 0 = 512 */
    uint32_t piece_bytes;    /* largest unit of copier work (multiple of 16); 0 = 65536 */
    uint32_t timestamps;     /* 1: stamp gate-open and arrival times (globaltimer, ns) */
    uint32_t initial_round;  /* 0 or 1: rounds start at 1; larger: gates begin as if
                                initial_round - 1 rounds had completed (round-limit tests) */
    uint64_t max_polls;      /* copier polls of one gate before it gives up; 0 = 2^22 */
    uint64_t max_regions;    /* capacity: regions in the plan; 0 = unlimited */
    uint32_t deferred_copier;/* 0: start() launches the copier.  1: dtt_plan_launch_copier or
                                wait() launches it after the work queued on the producer
                                stream (no overlap; for profilers that serialise kernels).
                                2: dtt_plan_launch_copier (or wait()) launches it with no
                                dependency, so the caller can launch its producer first and
                                the copier right after it, the two still overlapping */
    uint32_t stages;         /* DTT_COPY_TMA: shared-memory stages per copier CTA, each
                                piece_bytes long (2 <= stages, stages * piece_bytes <= 200 KiB);
                                0 = as many as fit, at most 8 */
    uint32_t time_copier;    /* 1: time every copier launch with CUDA events on the copy
                                stream (read with dtt_plan_stats) */
    uint32_t host_piece_bytes;/* dtt_allgather_host: bytes per host-to-device copy (a multiple
                                of 4096); 0 = a quarter of a slice, at least 4 MiB (rounds back
                                to back, dtt_allgather_host_rounds: 0 = a whole slice).  On an
                                all-reduce's reduce-scatter plan: dtt_allreduce_host's least
                                bytes a rank per copy in (0 = 16 MiB) */
    void* const* dst_bufs;    /* NULL: copies land in the P buffers themselves.  Else a host array
                                 of P device pointers, dst_bytes each: separate destination buffers
                                 (staging buffers) that every copy lands in, at its chunk's
                                 destinations (dtt_schedule_add_chunk_to).  Not with
                                 dtt_allgather_host, dtt_gemm_consumer or block groups. */
    uint64_t dst_bytes;
    uint32_t early_copier_us; /* > 0: dtt_plan_wait launches the NEXT round's copier right after
                                this round's check, queued behind this round's copier, so that
                                the next dtt_plan_start launches nothing (the pages' "prepare":
                                the copy engine's queue is armed before the round).  That copier
                                copies nothing until dtt_plan_start claims it; if no start comes
                                within early_copier_us microseconds of it beginning to wait, it
                                gives the round up and exits, and start launches a fresh copier.
                                The claim and the give-up are one compare-and-swap each on a
                                mapped host word, so exactly one side wins.  A failed wait,
                                dtt_plan_close and dtt_allgather_host abort it.  While it waits it
                                holds the copy stream and its SM resources: a device-wide
                                synchronisation (cudaDeviceSynchronize, cudaFree) made between
                                wait and the next start lasts until it gives up, and so does the
                                first launch of a kernel not yet loaded (lazy module loading
                                waits for the device to idle).  Ignored (the
                                copier is launched at start) with time_copier, deferred_copier
                                = 1, overlap, a copy stream another live plan uses, or a device
                                without host-native atomics.  At most 1000000; 0 = off */
    uint32_t overlap;         /* 1: overlapping rounds ("Triggered Plans", Not supported yet:
                                "Overlapping rounds" -- wait() had to return before next_round()
                                could prepare the next round).  dtt_plan_next_round may then also
                                be called while the round is RUNNING: that round stays in flight
                                (pending) and the next one is PREPARED, so at most two rounds are in
                                flight.  The pending round's copier runs before the next round's on
                                the copy stream, so every (source, peer) queue serves the pending
                                round first.  A producer of round R may write a chunk only once
                                round R-1's copies of it have landed (dtt_writable; the library's
                                producers wait for it on their own), and whatever reads what round
                                R-1 delivered must be done before round R's producers run.
                                dtt_plan_wait checks the pending round first.  Not with
                                deferred_copier = 1 (a round's producers wait for the previous
                                round's copier) or chunk groups (a member's next-round arrival
                                would count toward this round's group wait); the early copier is
                                not used (the next round's copier is queued at its start, behind the
                                pending one).  The next round's copier may take an SM's room before
                                the next round's producer does, so producer CTAs must fit on an SM
                                beside the copier's (which keep to half its threads and registers):
                                the library's fill takes at most 512 threads per CTA on such plans.
                                0 = rounds one at a time */
} dtt_plan_opts;

void dtt_plan_opts_default(dtt_plan_opts* opts);

#define DTT_HANDLE_TIMESTAMPS 1u   /* dtt_handle.flags bit: stamp gate-open times */
#define DTT_HANDLE_OVERLAP 2u      /* dtt_handle.flags bit: the plan overlaps rounds, so a producer
                                      waits for dtt_writable before it writes a chunk */
#define DTT_DEV_EBADCHUNK 1u       /* device status bit: a rank marked (or asked dtt_reusable of)
                                      a chunk it does not own */
#define DTT_DEV_EBADGROUP 2u       /* device status bit: a wait named a group the plan lacks */
#define DTT_DEV_EWRITABLE 4u       /* device status bit: a library producer's wait for a chunk to
                                      become writable (overlapping rounds) ran out; it left its part
                                      of the chunk unwritten, and wait() reports the round failed */

/* A plan's chunk groups (dtt_plan_define_groups): device arrays owned by the plan, their
 * addresses carried by value in every handle.  A group is a set of global chunk ids, of any
 * source ranks.  Each virtual rank q has one counter per group, counters[q * n_groups + g],
 * that goes up by one whenever a member becomes readable at q: the copier adds one when it
 * signals a member's arrival at q, and the mark that opens a member's gate adds one at its own
 * rank.  When chunks go to only some peers, q counts only the members that reach it (its own,
 * or addressed to it): size[q * n_groups + g] of them per round.  So after R rounds every
 * counter holds R * size, and a wait on group g passes at round * size ("Triggered Plans", Not
 * supported yet: "Waiting on a group" -- no single counter covers several chunks or several
 * source ranks). */
typedef struct dtt_group_table {
    uint64_t* counters;          /* [P][n_groups], monotonic, never reset */
    const uint32_t* size;        /* [P][n_groups]: members of group g that reach rank q */
    const uint32_t* chunk_off;   /* [n_global + 1]: chunk c's groups are */
    const uint32_t* chunk_ids;   /*   chunk_ids[chunk_off[c] .. chunk_off[c + 1]) */
    uint32_t n_groups;
    uint32_t reserved;
} dtt_group_table;

/* Device-side view of a plan for one rank and one round, passed by value to producer and
 * consumer kernels (the pages' TriggeredView handle).  Plain data; valid until the next
 * dtt_plan_start of the same plan or its close. */
typedef struct dtt_handle {
    uint64_t* gates;          /* device: P gate tables, [P][n_global][8] uint64 */
    const uint32_t* writers;  /* device: writers per global chunk */
    uint32_t* status;         /* device: plan status word (device-side misuse bits) */
    uint32_t round;
    uint32_t rank;
    uint32_t P;
    uint32_t n_global;        /* chunks in the plan, all ranks */
    uint32_t first_chunk;     /* global id of this rank's first chunk */
    uint32_t n_chunks;        /* this rank's chunk count */
    uint32_t flags;           /* bit 0: timestamps */
    uint32_t reserved;
    dtt_group_table groups;   /* the plan's groups (device arrays); counters == NULL: none */
    const uint32_t* peer_masks; /* device: receivers of each global chunk as a bit mask, or NULL
                                 when every chunk goes to every other rank */
    uint32_t* host_ready;     /* DTT_COPY_ENGINE plans: device address of mapped host words, word c
                                 = the round chunk c's gate last opened in (the mark that opens a
                                 gate stores it after a system-scope fence); NULL otherwise */
} dtt_handle;

/* Gate row: 64 bytes = 8 uint64 words per (rank, global chunk) ("Triggered Plans", Gates and
 * rounds: ready, arrival and a writer counter; "Triggered SDMA Plans", Design notes: ready,
 * arrival, completion, error, contributor counter).  Gates are never reset. */
enum {
    DTT_GATE_READY = 0,       /* owner's row: round of the last gate opening (low 32 bits
                                 are compared with >= round) */
    DTT_GATE_ARRIVAL = 1,     /* peer's row: one per round when the chunk has landed here */
    DTT_GATE_COMPLETION = 2,  /* owner's row: deliveries made, (P-1) per round */
    DTT_GATE_ERROR = 3,       /* owner's row: round of an extra mark, else 0 */
    DTT_GATE_COUNTER = 4,     /* owner's row: writer marks, round*writers after a round */
    DTT_GATE_T_OPEN = 5,      /* owner's row: globaltimer when the gate opened */
    DTT_GATE_T_ARRIVE = 6,    /* peer's row: globaltimer when the arrival was signalled; owner's
                                 row: when the copier began the chunk (SM copiers) */
    DTT_GATE_COPIER = 7,      /* owner's row: copier-internal progress counter */
    DTT_GATE_WORDS = 8
};

/* Result of dtt_plan_wait. */
typedef struct dtt_report {
    int32_t status;           /* DTT_OK, DTT_EEXTRA or DTT_ETIMEDOUT */
    uint32_t n_short;         /* chunks short of marks or of an arrival somewhere */
    uint32_t n_extra;         /* chunks with more marks than writers this round */
    uint32_t copier_timeouts; /* copier CTAs that gave up polling a gate */
    uint32_t device_status;   /* device-side misuse bits (e.g. a mark on a foreign chunk) */
    uint32_t round;
    uint32_t short_chunks[DTT_REPORT_MAX];  /* the first n_short ids, ascending */
    uint32_t extra_chunks[DTT_REPORT_MAX];  /* the first n_extra ids, ascending */
} dtt_report;

/* Create a plan over P symmetric buffers (bufs: host array of P device pointers, each
 * buf_bytes long, 16-byte aligned for the vector path) with one schedule per rank (scheds:
 * host array of P schedules; a NULL entry or empty schedule sends nothing).  Chunk ids are
 * global: rank r's chunks follow those of ranks 0..r-1 ("Triggered Plans", section Model).
 * Validates every region (inside the buffer; inside the rank's rows when opts->allgather;
 * no byte sent by two ranks to the same offsets) and every destination (inside the receiving
 * buffer; no two copies landing on the same bytes of one buffer; in place, no copy landing on
 * bytes its receiving rank sends: DTT_EOVERLAP), allocates the gate tables and the copier's
 * descriptor tables on the device, and leaves the plan PREPARED for round opts->initial_round
 * (1 by default).
 * copy_stream: a non-blocking stream for the copier, or NULL to let the plan create (and
 * own) a high-priority one.  Creation succeeds for every rank or for none: on error nothing
 * stays allocated ("Triggered Plans", The kernel author's contract).
 * Unless opts->deferred_copier is 1, the copier runs beside the producer, so its launch must leave
 * every SM room for producer CTAs: creation fails with DTT_EINVAL when the copier CTAs of one
 * SM would take more than 1024 threads or 32768 registers, or (bulk-copy path) more shared
 * memory than the SM has (a copier CTA left waiting for shared memory would keep the producer
 * from starting).  opts->overlap needs deferred_copier 0 or 2 (DTT_EINVAL otherwise).
 * Errors: DTT_EINVAL, DTT_EOUTOFROWS, DTT_EOVERLAP, DTT_ECAPACITY, DTT_ENOMEM, DTT_ECUDA. */
int dtt_plan_create(void* const* bufs, uint64_t buf_bytes, uint32_t P,
                    const dtt_schedule* const* scheds, const dtt_plan_opts* opts,
                    cudaStream_t copy_stream, dtt_plan** out);

/* Start the current round: launch its copier on the plan's copy stream and fill handles[r]
 * (host array of P) for every rank.  producer_stream is where the producers will run; wait()
 * orders its check after the work queued there.  It must differ from the copy stream.
 * The copier polls each source's gates in schedule order, so chunks completed out of order
 * are correct but wait for earlier ones ("Triggered Plans", The kernel author's contract,
 * item 1).  With a round pending (opts.overlap) the copier queues behind the pending round's on
 * the copy stream.  Errors: DTT_ESTATE (not PREPARED), DTT_EINVAL, DTT_ECUDA. */
int dtt_plan_start(dtt_plan* plan, cudaStream_t producer_stream, dtt_handle* handles);

/* Plans with opts.deferred_copier set: launch this round's copier now on the copy stream --
 * for deferred_copier = 1 ordered after the work queued so far on the producer stream, for
 * deferred_copier = 2 with no such dependency (it runs beside the producer).  A no-op when the
 * copier is already running.  Errors: DTT_ESTATE (not RUNNING), DTT_ECUDA. */
int dtt_plan_launch_copier(dtt_plan* plan);

/* The handle of one rank for the current round.  Errors: DTT_EINVAL. */
int dtt_plan_handle(const dtt_plan* plan, uint32_t rank, dtt_handle* out);

/* Block until the round is complete everywhere, then check it with a kernel: every chunk got
 * exactly writers marks this round and arrived at every peer ("Triggered Plans", Gates and
 * rounds; "Triggered SDMA Plans", Design notes, completion).  The check kernel is queued on
 * the producer stream (after everything the producers queued) and waits on the device, at
 * most 8 x max_polls polls, for the round's copier CTAs to finish; it writes its verdict into
 * mapped host memory, which this call polls.  Fills *report when non-NULL (report->round names
 * the round checked).
 * Overlapping rounds (opts.overlap): while a round is pending, this call checks that round, on an
 * internal stream ordered after the producers queued before its dtt_plan_next_round (not after
 * the next round's); the next round's marks may already count, so a count above writers is not
 * read as an extra mark there -- the gate row's error word, which the mark that passes its own
 * round's count sets, reports extra marks.  On success the plan's state is left as it was
 * (PREPARED or RUNNING, for the next round); on failure the plan is FAILED.
 * Returns DTT_OK (plan DONE, or no longer pending), DTT_EEXTRA or DTT_ETIMEDOUT (plan FAILED; the
 * report names the chunks, or the copier had not finished), DTT_ESTATE (not RUNNING and nothing
 * pending) or DTT_ECUDA. */
int dtt_plan_wait(dtt_plan* plan, dtt_report* report);

/* Advance to the next round: "done reading this round's data" ("Triggered Plans", The kernel
 * author's contract, item 6).  With opts.overlap, also from RUNNING when no round is pending: the
 * running round becomes pending (its copier is launched now if it was deferred, and its check
 * will follow the producers queued so far on the producer stream) and the next round is PREPARED.
 * Errors: DTT_ESTATE (not DONE, nor RUNNING with overlap and nothing pending), DTT_EROUNDLIMIT
 * (the round is already 2^32 - 1; the state is unchanged), DTT_ECUDA. */
int dtt_plan_next_round(dtt_plan* plan);

/* The round in flight behind the current one (opts.overlap: "Triggered Plans", Not supported
 * yet, "Overlapping rounds"), or 0 when none is (and for a NULL plan). */
uint32_t dtt_plan_pending_round(const dtt_plan* plan);

/* Close the plan ("Triggered Plans", The kernel author's contract, close()).  In the middle of
 * a round, the work already queued on the producer stream finishes first, then every gate
 * still closed is opened, so the copier sends each chunk as it stands.
 *
 * Plans may share a copy stream (pass the same copy_stream to dtt_plan_create).  A copier
 * then runs only after every copier launched before it on that stream.  If this plan's
 * copier is queued behind an earlier plan's copier that is still waiting on that plan's gates,
 * the plan cannot finish first: close returns DTT_CLOSING at once and leaves the plan CLOSING.
 * Closing (or waiting on) the earlier plan lets it drain; closing the earlier plan also
 * finishes every CLOSING plan behind it, which then reads CLOSED.  Call dtt_plan_close on a
 * CLOSING or CLOSED plan again to release it.  Plans can be closed in any order.
 *
 * Otherwise the plan's copier is drained and the plan released; the pointer is invalid
 * afterwards.  Device memory is freed at once, or, while another plan's copier may still be
 * spinning on a gate, as soon as none is (cudaFree waits for the whole device).
 * Returns DTT_OK, DTT_CLOSING, or DTT_ECUDA if a CUDA call failed on the way (the plan is
 * released all the same). */
int dtt_plan_close(dtt_plan* plan);

int dtt_plan_state(const dtt_plan* plan);
uint32_t dtt_plan_round(const dtt_plan* plan);

/* Plan layout: n_global chunks; first_chunk / n_chunks per rank (host arrays of P, may be
 * NULL); *gates_device = the gate tables' device address. */
int dtt_plan_info(const dtt_plan* plan, uint32_t* n_global, uint32_t* first_chunk,
                  uint32_t* n_chunks, uint64_t** gates_device);

/* Copier timing of a plan created with opts.time_copier = 1: the device time of the last
 * copier launch and the sum over all launches so far (milliseconds, from CUDA events recorded
 * around each launch on the copy stream), and how many launches were timed.  The events are
 * read here (waiting for the copy stream's launched copiers), not in dtt_plan_wait, so timing
 * adds no synchronisation to a round.  Any pointer may be NULL.  Errors: DTT_EINVAL, DTT_ECUDA. */
int dtt_plan_stats(dtt_plan* plan, double* copier_ms_last, double* copier_ms_total,
                   uint64_t* rounds_timed);

/* Define the plan's chunk groups ("Triggered Plans", Not supported yet: "Waiting on a group";
 * see dtt_group_table): group g holds the global chunk ids chunk_ids[offsets[g] ..
 * offsets[g + 1]) (host arrays; offsets has n_groups + 1 entries, offsets[0] = 0).  A chunk may
 * belong to several groups; within a group ids are distinct.  Kernels then wait once per group
 * with dtt_wait_group.  Allowed once per plan, before its first dtt_plan_start; the counters
 * begin as after the rounds before opts.initial_round.  The tables live on the device until the
 * plan is closed.  Errors: DTT_EINVAL (empty group, id out of range or repeated in a group,
 * n_groups == 0, a plan with opts.overlap), DTT_ESTATE (started already, or groups defined
 * already), DTT_ECUDA. */
int dtt_plan_define_groups(dtt_plan* plan, uint32_t n_groups, const uint32_t* offsets,
                           const uint32_t* chunk_ids);

/* Groups by position: group b holds every chunk with a byte in [b * block_bytes, (b + 1) *
 * block_bytes) of the buffers, b = 0 .. ceil(buf_bytes / block_bytes) - 1 (for example the
 * 128-row blocks a consumer GEMM loads: block_bytes = 128 rows x row bytes).  A block no chunk
 * touches gets no group of its own: *n_groups (may be NULL) receives the count and block_group
 * (host, may be NULL, ceil(buf_bytes / block_bytes) entries) each block's group id, or
 * UINT32_MAX.  Otherwise as dtt_plan_define_groups. */
int dtt_plan_define_block_groups(dtt_plan* plan, uint64_t block_bytes, uint32_t* n_groups,
                                 uint32_t* block_group);

/* Copy the group counters (P * n_groups uint64, rank-major) to host memory and wait for the
 * copy.  Errors: DTT_EINVAL (no groups, n_words short), DTT_ECUDA. */
int dtt_plan_read_group_counters(dtt_plan* plan, uint64_t* host, uint64_t n_words);

/* Counts of a plan's early copiers (opts.early_copier_us) so far: launched by dtt_plan_wait,
 * claimed by the next dtt_plan_start, found by the host to have given their round up (start then
 * launched a fresh copier), and aborted by the host (failed wait, close, host-buffer round).  Any
 * pointer may be NULL.  Errors: DTT_EINVAL. */
int dtt_plan_early_stats(const dtt_plan* plan, uint64_t* launched, uint64_t* claimed,
                         uint64_t* expired, uint64_t* aborted);

/* Copy the P gate tables (P * n_global * 8 uint64, rank-major) to host memory `host`
 * (n_words long), on an internal stream of the plan, and wait for the copy.  Made mid-round it
 * is a snapshot.  Errors: DTT_EINVAL if n_words is short. */
int dtt_plan_read_gates(dtt_plan* plan, uint64_t* host, uint64_t n_words);

/* Host-buffer all-gather, one round end to end: copy each rank's slice (host_slices[r],
 * pinned host memory, S = buf_bytes / P bytes; NULL: the rank's rows as they stand) into its
 * own rows, let the copier fan the chunks out, wait, and copy rank out_rank's gathered buffer
 * (buf_bytes) to host_out (pinned, may be NULL).  Then advances to the next round.
 * The round is pipelined: slices go in rank by rank, in pieces, on a stream of the plan; each
 * chunk is marked (a kernel on `stream`) as soon as the bytes it covers have landed, so the
 * copier fans it out while later pieces are still in flight; the copier stamps each chunk's
 * arrival into pinned, mapped host memory, and the host copies every slice of out_rank's
 * buffer back, on another stream of the plan, as far as its chunks have arrived.  The call
 * returns when everything has landed in host_out.  Needs an all-gather plan in state
 * PREPARED with no round pending (opts.overlap: check the pending round first).  The report
 * is filled as by dtt_plan_wait.  Errors: as start / wait / next_round,
 * DTT_ETIMEDOUT if a slice could not be copied back completely. */
int dtt_allgather_host(dtt_plan* plan, const void* const* host_slices, void* host_out,
                       uint32_t out_rank, cudaStream_t stream, dtt_report* report);

/* Host-buffer all-gather over n_rounds rounds back to back, pipelined across rounds (a plan made
 * with opts.overlap; like dtt_allgather_host, this library's own addition: the pages move device
 * data only, and this call feeds a plan's rounds from host memory): each round as dtt_allgather_host, but round k + 1's slices start going in
 * while round k's gathered buffer is still coming back, so the host link carries both directions
 * nearly all the time.  Round k + 1's bytes of a slice go in only once round k has delivered the
 * chunks they overwrite (the copier's arrival stamps in mapped host memory, polled here) and, in
 * the output rank's own rows, copied them back; a chunk of round k + 1 is marked only once round
 * k's copy back of the bytes its copies will overwrite in the output rank's buffer is done (an
 * event the marking kernel's stream waits on).  Round k is checked (the plan's pending round)
 * once it has come back.
 *  - host_slices: n_rounds * P pinned host pointers, round-major (round k's at [k * P, k * P + P)),
 *    S = buf_bytes / P bytes each; NULL: that slice as it stands.
 *  - host_outs: n_rounds pinned host pointers of buf_bytes each; the array or an entry may be NULL
 *    (that round is not copied back).
 *  - reports: n_rounds reports (may be NULL), filled as by dtt_plan_wait.
 * The call returns when every round has come back and been checked, and leaves the plan PREPARED
 * for the round after them.  Needs an all-gather plan made with opts.overlap, PREPARED with no
 * round pending, an SM copier and chunks that land at their own offsets.
 * Errors: DTT_EINVAL, DTT_ESTATE, DTT_EROUNDLIMIT, those of dtt_plan_wait (the plan is then FAILED),
 * DTT_ETIMEDOUT (a slice came back short), DTT_ECUDA. */
int dtt_allgather_host_rounds(dtt_plan* plan, uint32_t n_rounds, const void* const* host_slices,
                              void* const* host_outs, uint32_t out_rank, cudaStream_t stream,
                              dtt_report* reports);

/* ---------------------------------------------------------------------------------------- */
/* Producers and consumers shipped with the library                                          */
/* ---------------------------------------------------------------------------------------- */

/* Marks of the fill producer. */
enum {
    DTT_MARK_PER_STEP = 0,   /* mark first_chunk + step / tiles_per_chunk after each step */
    DTT_MARK_AT_END = 1      /* each program marks first_chunk once after its last step
                                (whole(): "marked ready once per program at the end") */
};

/* Hashed-fill producer.  Rank r's slice is M x N elements of `dtype` with rows `pitch` bytes
 * apart, starting at byte slice_off[r] of bufs[r].  It is produced as BM x BN tiles by
 * num_programs programs per rank: program p takes steps p, p + num_programs, ... in `order`
 * ("Triggered Plans", section Model, the persistent tiled producer), writes the tile and marks
 * per mark_mode.  A program is one CTA; or a thread-block cluster of `cluster` CTAs that
 * marks once per step after a cluster barrier; or a group of `group` CTAs anywhere on the GPU
 * whose last CTA to finish a step marks it once, after acquiring the others' stores through an
 * acq_rel counter.  Either way the program is one writer.  Element (row, col) of rank r in
 * round R holds hash(seed, r, R, row, col): with fmix32 the MurmurHash3 finaliser,
 * salt = fmix32(seed ^ fmix32(r ^ fmix32(R))), h = fmix32((row*N + col) mod 2^32 ^ salt),
 * u = ((h >> 8) - 2^23) * 2^-23 in [-1, 1); bf16 = u rounded to nearest even, f32 = u,
 * u8 = h & 0xFF.  Only ranks whose bit is set in rank_mask produce. */
typedef struct dtt_fill_desc {
    uint32_t dtype;
    uint32_t seed;
    uint64_t M, N;
    uint64_t pitch;
    uint64_t buf_bytes;      /* size of every buffer: slices must lie inside it */
    uint64_t slice_off[DTT_MAX_RANKS];
    uint32_t BM, BN;
    uint32_t num_programs;
    uint32_t tiles_per_chunk;
    dtt_order order;
    uint32_t mark_mode;
    uint32_t cluster;        /* 1..16 CTAs per program (above 8 needs non-portable clusters) */
    uint32_t rank_mask;
    uint32_t threads;        /* threads per CTA; 0 = 256; at most 512 with overlapping rounds */
    uint32_t group;          /* > 1: a program is `group` CTAs that split each step's rows; the
                                last of them to finish a step issues its one mark (per-step
                                marks only, cluster must be 1) */
    uint32_t pace;           /* > 0: before its first step in chunk k >= pace, a program waits
                                (advisory: at most ~1 ms, then it goes on) until chunk k - pace of
                                its rank is reusable (dtt_reusable: delivered to every peer), so
                                that the bytes written but not yet copied stay within `pace`
                                chunks per rank and the copier reads them from L2.  A CTA whose
                                wait runs out stops pacing for the rest of the launch, so each
                                CTA stalls at most once (~1 ms) per launch when the copier lags.
                                Timing only: the data and marks are the same, and the wait is
                                on a chunk earlier in schedule order whose writers have all
                                marked it, so it cannot hold up any mark.  With overlapping
                                rounds (the handles' DTT_HANDLE_OVERLAP), chunk k < pace waits in
                                the same way for the previous round's delivery of chunk n - pace + k
                                (n: the rank's chunks), whose copier runs just before this round's.
                                Needs the copier running beside the producer (deferred_copier 0 or
                                2) and every producer CTA resident at once (checked: DTT_EINVAL
                                otherwise). */
    uint32_t* group_counters;/* group > 1: device uint32[P * steps per rank], zero before the
                                first round (the producer leaves them zero after each round) */
} dtt_fill_desc;

/* Launch the fill producer for all P ranks on `stream` (handles: host array of P, from
 * dtt_plan_start).  bufs: host array of P device pointers.  Errors: DTT_EINVAL, DTT_ECUDA. */
int dtt_fill_producer(void* const* bufs, uint32_t P, const dtt_fill_desc* desc,
                      const dtt_handle* handles, cudaStream_t stream);

/* GEMM producer (tcgen05 tensor cores, TMEM accumulators, TMA loads): for every rank r,
 * C_r = A_r . B with bf16 inputs, fp32 accumulation and round-to-nearest-even bf16 output,
 * stored at bufs[r] + slice_off[r] as M rows of N elements, ldc bytes apart.  This is the
 * tiled producer "such as a GEMM" of "Triggered Plans" (section Model).
 *  - A: device bf16 [P][M][K], K contiguous.  Bt: device bf16 [N][K] = B transposed, K
 *    contiguous.
 *  - Persistent: num_programs CTAs, each taking 128 x 128 tiles p, p + num_programs, ... of
 *    rank 0, then of rank 1, and so on, in row-major tile order.  After each tile's stores it
 *    marks first_chunk + step / num_programs, so its schedule is
 *    dtt_schedule_tile_chunks(slice_off[r], M, N, 2, ldc, 128, 128, num_programs, row-major).
 *  - err: device uint32, incremented when a bounded internal wait gives up (0 after a clean
 *    run).
 *  - Needs M and N multiples of 128, K a multiple of 64, and 16-byte aligned operands and
 *    outputs.  Every handle must have ceil((M / 128) (N / 128) / num_programs) chunks (the
 *    schedule above), else DTT_EINVAL before anything is launched.  One CTA per SM uses ~194 KiB of shared memory, so it runs beside the vector
 *    copier, not the bulk copier.
 * Errors: DTT_EINVAL, DTT_ECUDA. */
int dtt_gemm_producer(const void* A, const void* Bt, void* const* bufs, uint32_t P, uint32_t M,
                      uint32_t N, uint32_t K, uint64_t ldc, const uint64_t* slice_off,
                      uint32_t num_programs, const dtt_handle* handles, uint32_t* err,
                      cudaStream_t stream);

/* A producer that only marks: chunks [first_chunk, first_chunk + n_chunks) (global ids) each
 * get `marks` marks, or their writer count when marks == 0, from one CTA per chunk launched on
 * `stream`, on behalf of the rank that owns each chunk (handles: host array of P from
 * dtt_plan_start).  Work queued earlier on `stream` -- host-to-device copies of the chunk's
 * data, other kernels -- precedes the marks.  It serves host-fed rounds and lets a caller give
 * a chunk an extra mark or leave one short ("Triggered Plans", The kernel author's contract,
 * item 2, names both).  With overlapping rounds the bytes of a chunk copied in before its marks
 * must not land before the previous round's copies of it have (dtt_writable): the marks
 * themselves do not wait.  Errors: DTT_EINVAL, DTT_ECUDA. */
int dtt_publish(const dtt_handle* handles, uint32_t P, uint32_t first_chunk, uint32_t n_chunks,
                uint32_t marks, cudaStream_t stream);

/* Consumer GEMM, the peer-kernel side of a triggered plan ("Triggered Plans", Model: peer
 * kernel wait(chunk); Memory ordering, Consumer): D = X . W^T, where X is rank `rank`'s buffer
 * seen as [rows = buf_bytes / (2 K), K] bf16 (its gathered output), Wt = W^T [N, K] bf16
 * (K-major, device) and D [rows, N] bf16 (device, rows ldd bytes apart).  Each 128-row block of
 * X is loaded only after every chunk covering it has arrived at `rank` this round (its own
 * chunks: once they are ready), polling at most max_polls times per chunk (0: the plan's), so
 * the GEMM runs while the all-gather is still delivering.  tcgen05 / TMEM, fp32 accumulation,
 * bf16 out, num_programs persistent CTAs (0: 148).  Call after dtt_plan_start, on a stream
 * other than the copy stream.  A wait that runs out adds 1 to *err (device uint32) and the
 * kernel stops.  Requirements: N % 128 == 0, K % 64 == 0, buf_bytes a multiple of 256 K,
 * 16-byte aligned Wt, D and ldd.  When N % 256 == 0, the rows form an even number of 128-row
 * blocks and num_programs >= 2, CTA pairs (tcgen05 cta_group::2, 256 x 256 per MMA) compute it,
 * each CTA waiting for its own row block, with the deepest ring of 6 to 3 stages of 32 KiB
 * that fits beside the plan's copier CTAs on an SM; otherwise single CTAs (128 x 256 or
 * 128 x 128) with up to 4 stages of 48 KiB.  Where no ring fits (a bulk-copy ring of ~200 KiB
 * per SM) the GEMM starts only as the copier's CTAs leave.  The first call for a (rank, K)
 * builds a small table on the device (stream-ordered).
 * Errors: DTT_EINVAL, DTT_ESTATE (plan not RUNNING), DTT_ECUDA. */
int dtt_gemm_consumer(dtt_plan* plan, uint32_t rank, const void* Wt, uint32_t N, uint32_t K, void* D,
                      uint64_t ldd, uint32_t num_programs, uint64_t max_polls, uint32_t* err,
                      cudaStream_t stream);

/* Consumer: rank `rank` waits for every chunk of the other ranks that it receives (in global id
 * order, with the device-side wait, at most max_polls polls each) and copies each chunk's landed
 * bytes from where they landed (the rank's own buffer, or its destination buffer) to the same
 * offsets of `dst` (device, buf_bytes or dst_bytes long) -- data read after the wait is this
 * round's ("Triggered Plans", Memory ordering, Consumer).  Per-chunk results go to status
 * (device int32 [n_global]: 0, or DTT_ETIMEDOUT; 0 for chunks it does not receive).  Launch with at most
 * `ctas` CTAs on `stream` (a third stream, concurrent with producer and copier).
 * Errors: DTT_EINVAL, DTT_ESTATE (plan not RUNNING), DTT_ECUDA. */
int dtt_consumer_gather(dtt_plan* plan, uint32_t rank, void* dst, uint64_t max_polls,
                        int32_t* status, uint32_t ctas, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------- */
/* Two-shot all-reduce and reduce-scatter ("Triggered Plans", Not supported yet: reduce-     */
/* scatter and two-shot all-reduce are what other destinations make possible)                */
/* ---------------------------------------------------------------------------------------- */

/* The pages name the two-shot all-reduce and say nothing more of it; this is the plain
 * reading, built from two plans over the same P buffers and one library kernel between them.
 *  - Data: rank r's vector x_r is M = P * block_rows rows of `cols` elements (bf16 or f32),
 *    rows `pitch` bytes apart from byte 0 of bufs[r].  Every rank ends with
 *    y = x_0 + ... + x_{P-1} there, added in f32 in rank order 0..P-1 (IEEE round to nearest
 *    even after each add) and rounded once to the element type (bf16: nearest even).
 *  - Rank b owns block b, rows [b * block_rows, (b + 1) * block_rows), cut into sub_blocks
 *    chunks of block_rows / sub_blocks rows (Mj).
 *  - Reduce-scatter plan: rank s's chunk b * sub_blocks + j (sub-block j of block b of its
 *    vector) goes to rank b only, into slot s of b's staging area -- the same rows of the block,
 *    from byte slot_off + s * block_rows * pitch.  The staging area is b's own buffer after the
 *    vector (slot_off = M * pitch, so buf_bytes >= 2 M pitch) or, with staging buffers, that
 *    buffer from byte 0 (staging_bytes >= P * block_rows * pitch).  Rank b's own chunks of block
 *    b go nowhere (only b's bit in their peer mask) and its own slot stays unused.  Group
 *    b * sub_blocks + j holds the P chunks (s, b, j): at rank b its own one counts when marked
 *    and the others when they land, so one group wait covers them all.
 *  - dtt_allreduce_reduce: for every (b, j), b-major, waits for that group at rank b, adds rank
 *    b's own rows and the P - 1 slots in rank order, writes the sum over b's own rows and marks
 *    rank b's all-gather chunk j (once: the last of its warps to finish issues the mark).  At
 *    most 4096 sub-blocks in all (P x sub_blocks).
 *  - All-gather plan: rank b's chunk j (sub-block j of block b) goes to every other rank at the
 *    same rows.
 * A round: dtt_allreduce_start, the producers write every rank's vector and mark its
 * reduce-scatter chunks (with the handles start returns), dtt_allreduce_reduce,
 * dtt_allreduce_wait, dtt_allreduce_next_round.  Rounds run one at a time. */
typedef struct dtt_allreduce dtt_allreduce;

typedef struct dtt_allreduce_desc {
    uint32_t dtype;          /* DTT_BF16 or DTT_F32 */
    uint32_t sub_blocks;     /* chunks per block, dividing block_rows; 0 = 1 */
    uint64_t block_rows;     /* rows each rank reduces (its block), >= 1 */
    uint64_t cols;           /* elements per row; cols x element bytes a multiple of 16 */
    uint64_t pitch;          /* bytes between rows, a multiple of 16; 0 = cols x element bytes */
    uint32_t reduce_ctas;    /* CTAs of the reduce kernel; 0 = one per SM */
    uint32_t reduce_threads; /* threads per reduce CTA: one control warp (the group waits, the
                                counts and marks) and the rest compute warps (loads, adds,
                                stores); a multiple of 32 in [64, 512]; 0 = 256 */
    uint32_t scatter_only;   /* 1: a reduce-scatter -- the first shot alone: rank b ends with the
                                sum over its block b and its own partial in its other rows; no
                                all-gather plan (ag_opts ignored, dtt_allreduce_plans gives NULL
                                for it, and dtt_allreduce_wait also waits for the reduce kernel) */
} dtt_allreduce_desc;

/* Build both plans and the reduce kernel's counters.  bufs: host array of P (2..16) device
 * pointers, buf_bytes each, 16-byte aligned; staging: NULL (slots in bufs after the vector) or
 * a host array of P device pointers, staging_bytes each, 16-byte aligned.  rs_opts / ag_opts:
 * the plans' options (NULL: bulk-copy copiers of three 32-thread CTAs per SM with two 16 KiB
 * stages each); the library sets allgather = 0 and the destination buffers itself.  Both
 * copiers spin while the reduce kernel waits on the first one's deliveries, so the two
 * copiers' CTAs and the reduce's must fit on an SM together (threads, registers, shared
 * memory): checked here, DTT_EINVAL otherwise.  deferred_copier = 1 on both plans runs the
 * round in order instead -- the reduce-scatter copier after the producers, the reduce after that
 * copier, the all-gather copier after the reduce (dtt_allreduce_reduce launches all three), so
 * it completes where kernels run one at a time (a profiler that serialises launches); nothing
 * then runs beside the reduce and no room is checked.  Not with the copy-engine transport,
 * overlap, deferred_copier = 2 or the two plans' deferred_copier differing (DTT_EINVAL).  Copy
 * streams: as dtt_plan_create (NULL: each plan makes its own).  The caller owns the buffers;
 * the all-reduce owns its plans.
 * Errors: DTT_EINVAL, DTT_EOVERLAP, DTT_ENOMEM, DTT_ECUDA (nothing stays allocated). */
int dtt_allreduce_create(void* const* bufs, uint64_t buf_bytes, void* const* staging,
                         uint64_t staging_bytes, uint32_t P, const dtt_allreduce_desc* desc,
                         const dtt_plan_opts* rs_opts, const dtt_plan_opts* ag_opts,
                         cudaStream_t rs_copy_stream, cudaStream_t ag_copy_stream,
                         dtt_allreduce** out);

/* The two plans, owned by the all-reduce (for dtt_plan_read_gates, dtt_plan_stats and the
 * like; not to be started, waited on or closed directly).  Either pointer may be NULL.
 * Errors: DTT_EINVAL. */
int dtt_allreduce_plans(const dtt_allreduce* ar, dtt_plan** rs, dtt_plan** ag);

/* Start the current round on both plans (their copiers launch on their copy streams).
 * rs_handles (host array of P, may be NULL) receives the reduce-scatter plan's handles, for
 * the producers' marks.  Errors: as dtt_plan_start (both plans PREPARED). */
int dtt_allreduce_start(dtt_allreduce* ar, cudaStream_t producer_stream, dtt_handle* rs_handles);

/* Launch the reduce kernel on `stream`, normally the producer stream after the producers: its
 * CTAs spin on group waits, so on another stream the producers' CTAs must fit beside it.  In
 * order (deferred_copier = 1) it also launches the reduce-scatter copier before the reduce
 * (ordered after the producer stream's work so far) and the all-gather copier after it.
 * In each CTA one control thread polls the sub-blocks' groups ahead of the work and counts the
 * CTA's finished sub-blocks (the marks); the compute warps only load, add and store.
 * err: device uint32, incremented by a CTA whose control thread saw nothing move for the
 * reduce-scatter plan's max_polls polls; that CTA stops, the all-gather chunks not yet marked
 * stay so and dtt_allreduce_wait fails.  Errors: DTT_ESTATE (a plan not
 * RUNNING), DTT_EINVAL, DTT_ECUDA. */
int dtt_allreduce_reduce(dtt_allreduce* ar, uint32_t* err, cudaStream_t stream);

/* dtt_plan_wait on the reduce-scatter plan, then on the all-gather plan (reports may be NULL).
 * Returns the first error (both plans are waited on either way).  After a failed wait the plans
 * are FAILED (and the reduce kernel's counters may hold a partial count): destroy the
 * all-reduce. */
int dtt_allreduce_wait(dtt_allreduce* ar, dtt_report* rs_report, dtt_report* ag_report);

/* Host-buffer all-reduce, one round end to end (this library's own addition, like
 * dtt_allgather_host: the pages move device data only).  host_parts: host array of P pointers,
 * rank r's vector in pinned host memory as P * block_rows rows of cols elements back to back
 * (a NULL entry: that rank's vector as it stands on the device); host_out: pinned host memory
 * of the same size for rank out_rank's result, or NULL.  The round is pipelined: the vectors go
 * in on a stream of the reduce-scatter plan sub-block by sub-block in the groups' order (every
 * rank's rows of the first sub-blocks of block 0 first, in copies of at least the reduce-scatter
 * plan's host_piece_bytes a rank -- 0: 16 MiB -- or the rest of a block), each reduce-scatter
 * chunk is marked (a kernel on `stream`) once its rows have landed, the reduce kernel runs on
 * a stream of the all-reduce while later rows are still coming in (err as for
 * dtt_allreduce_reduce), and the all-gather copier stamps each chunk's arrival into pinned,
 * mapped host memory so that out_rank's result comes back (on a stream of the all-gather plan)
 * sub-block by sub-block as it is delivered, in copies of at least 8 MiB or the rest of a
 * block.  Then both waits and both
 * next_rounds; the call returns once host_out holds the result and the round is checked.  Only
 * the concurrent form (deferred_copier 0) of an all-reduce (not scatter_only); both plans
 * PREPARED.  The reports are filled as by dtt_allreduce_wait.  Errors: DTT_EINVAL, DTT_ESTATE,
 * those of start, reduce and wait, DTT_ETIMEDOUT if a block of the result could not be copied
 * back, DTT_ECUDA.  After an error other than DTT_EINVAL or DTT_ESTATE, destroy the all-reduce. */
int dtt_allreduce_host(dtt_allreduce* ar, const void* const* host_parts, void* host_out, uint32_t out_rank,
                       uint32_t* err, cudaStream_t stream, dtt_report* rs_report, dtt_report* ag_report);

/* dtt_plan_next_round on both plans.  Errors: as dtt_plan_next_round. */
int dtt_allreduce_next_round(dtt_allreduce* ar);

/* Close both plans (draining their copiers) and free the rest.  Returns the first error of the
 * two closes; the all-reduce is released either way. */
int dtt_allreduce_destroy(dtt_allreduce* ar);

/* ---------------------------------------------------------------------------------------- */
/* N-rank notify/wait barrier (PyPTO, "Barrier: Signals Only")                               */
/* ---------------------------------------------------------------------------------------- */

/* Hand-rolled barrier over P virtual ranks, one CTA each in one cooperative launch.  Rank r
 * adds 1 (atomic, release) to row r of every peer's window signal[peer] (device int32[P]),
 * then waits until row src of its own window is >= gen for every src != r (acquire, at most
 * max_polls polls each), then copies its window to y[r] (device int32[P]) (sections The idea
 * and Walkthrough; counters are monotonic, so the gen-th use of one set of windows passes
 * gen).  status (device int32[P]): 0, or DTT_ETIMEDOUT for a rank whose wait gave up.
 * signal and y are host arrays of P device pointers.  Errors: DTT_EINVAL, DTT_ECUDA. */
int dtt_barrier_handrolled(int32_t* const* signal, int32_t* const* y, uint32_t P, uint32_t gen,
                           uint64_t max_polls, int32_t* status, cudaStream_t stream);

/* The builtin barrier's state: P x P int32 internal counters on the device (zeroed at create)
 * and the host's generation count.  Owned by the caller. */
typedef struct dtt_barrier dtt_barrier;
int dtt_barrier_create(uint32_t P, dtt_barrier** out);
void dtt_barrier_destroy(dtt_barrier* b);

/* The builtin reveal (section Walkthrough, the builtin reveal): every rank stages x[r] into
 * data[r] (size int32 each), passes a barrier on the internal counters (no tally in any user
 * window), then loads the next rank's staged slice: y[r] = data[(r + 1) % P].  x, data, y are
 * host arrays of P device pointers; status as for dtt_barrier_handrolled. */
int dtt_barrier_reveal(dtt_barrier* b, const int32_t* const* x, int32_t* const* data,
                       int32_t* const* y, uint32_t size, uint64_t max_polls, int32_t* status,
                       cudaStream_t stream);

/* The same reveal for callers that cannot allocate device memory when they call it.  The
 * pages have no counterpart: this entry point is this library's own addition.
 * Who needs it: code whose device memory is owned entirely by another allocator (a caching
 * allocator or a fixed arena that a stray cudaMalloc would fail against or fragment), and code
 * that must not pay for an allocation while other work is in flight (cudaFree synchronises the
 * whole device).  dtt_barrier_create allocates the counters with cudaMalloc; this call does
 * not: the internal counters live in a fixed device array inside the library, sized for
 * DTT_NOALLOC_MAX_RANKS ranks (DTT_NOALLOC_MAX_RANKS^2 int32 = 1 KiB), which every GPU that
 * loads the library holds until the process exits.  The call itself calls no cudaMalloc,
 * cudaFree or other allocating routine.
 * Arguments, results and status are those of dtt_barrier_reveal, with P given directly.
 *  - The first call on a device (that device current) looks up the array's device address
 *    and prepares the library's kernels; make that first call before any stream capture.
 *  - Every call clears the P x P counters it uses (stream-ordered, on `stream`) and then runs
 *    one barrier generation on them.
 *  - All calls share the one array: calls that overlap on the GPU (on different streams, or
 *    from several threads) race on it and may pass their barrier early or time out.
 *    Serialise them, for example on one stream.
 * Errors: DTT_EINVAL (P outside 1..DTT_NOALLOC_MAX_RANKS, NULL pointers), DTT_ECUDA. */
#define DTT_NOALLOC_MAX_RANKS 16
int dtt_barrier_reveal_noalloc(const int32_t* const* x, int32_t* const* data, int32_t* const* y,
                               uint32_t P, uint32_t size, uint64_t max_polls, int32_t* status,
                               cudaStream_t stream);

/* ---------------------------------------------------------------------------------------- */
/* Errors                                                                                    */
/* ---------------------------------------------------------------------------------------- */

const char* dtt_last_error(void);

/* Prepare every kernel of the library on the current device: load it now, and give it the
 * library's shared-memory carveout (cudaSharedmemCarveoutMaxShared).
 *  - With lazy module loading (the CUDA default) the first launch of a kernel may wait until
 *    the device is idle, and a copier spinning on a gate keeps it busy until its polls run out.
 *  - An SM runs CTAs of one L1/shared-memory split at a time.  The copier puts a CTA on every
 *    SM, so a kernel whose preferred split differs (the driver derives one from occupancy when
 *    none is set) cannot start until the copier exits.
 * dtt_plan_create and dtt_barrier_create call it (once per device).  A caller's own producer
 * and consumer kernels that run during a round need the same two steps: load them before the
 * first round (cudaFuncGetAttributes) and set cudaFuncAttributePreferredSharedMemoryCarveout
 * to cudaSharedmemCarveoutMaxShared.  Otherwise they start only after the copier gives up.
 * Errors: DTT_ECUDA. */
int dtt_preload(void);

#ifdef __cplusplus
}
#endif

#endif /* DTT_H */
