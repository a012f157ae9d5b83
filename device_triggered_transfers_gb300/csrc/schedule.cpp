// Schedule builders: whole(), chunks(), tile_chunks() and hand-built schedules ("Triggered
// Plans", section Model; "Triggered SDMA Plans", section API).  Host code only.
#include <cstdarg>
#include <cstring>
#include <new>
#include <vector>

#include "internal.h"
#include "order.h"

namespace dtt {

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
}

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

// A block of rows as regions: contiguous rows (or one row) are a byte range cut into pieces of
// at most 1 GiB (a linear copy's 30-bit byte count); strided rows are one 2D sub-window.
static void block_regions(uint64_t off, uint64_t rows, uint64_t row_bytes, uint64_t pitch,
                          std::vector<dtt_region>* out) {
    if (rows == 0 || row_bytes == 0) return;
    if (rows == 1 || pitch == row_bytes) {
        const uint64_t n = rows * row_bytes;
        for (uint64_t pos = 0; pos < n; pos += DTT_LINEAR_MAX) {
            const uint64_t len = (n - pos) < DTT_LINEAR_MAX ? (n - pos) : DTT_LINEAR_MAX;
            out->push_back(dtt_region{off + pos, len, 1, len});
        }
    } else {
        out->push_back(dtt_region{off, row_bytes, rows, pitch});
    }
}

}  // namespace dtt

using namespace dtt;

extern "C" {

const char* dtt_last_error(void) { return g_err; }

int dtt_tile_of(const dtt_order* order, uint64_t step, uint32_t tiles_m, uint32_t tiles_n,
                uint32_t* tm, uint32_t* tn) {
    if (!tm || !tn || tiles_m == 0 || tiles_n == 0) return fail(DTT_EINVAL, "dtt_tile_of: bad args");
    const uint32_t kind = order ? order->kind : (uint32_t)DTT_ORDER_ROW_MAJOR;
    const uint32_t gm = order ? order->group_m : 0;
    if (kind != DTT_ORDER_ROW_MAJOR && kind != DTT_ORDER_GROUPED)
        return fail(DTT_EINVAL, "dtt_tile_of: unknown order kind %u", kind);
    if (kind == DTT_ORDER_GROUPED && gm == 0)
        return fail(DTT_EINVAL, "dtt_tile_of: grouped order needs group_m >= 1");
    if (step >= (uint64_t)tiles_m * tiles_n) return fail(DTT_EINVAL, "dtt_tile_of: step past the tiles");
    tile_of(kind, gm, step, tiles_m, tiles_n, tm, tn);
    return DTT_OK;
}

int dtt_schedule_empty(dtt_schedule** out) {
    if (!out) return fail(DTT_EINVAL, "dtt_schedule_empty: out is NULL");
    *out = new (std::nothrow) dtt_schedule();
    return *out ? DTT_OK : fail(DTT_ENOMEM, "dtt_schedule_empty: out of memory");
}

void dtt_schedule_free(dtt_schedule* s) { delete s; }

int dtt_schedule_add_chunk(dtt_schedule* s, const dtt_region* regions, uint32_t n,
                           uint32_t writers) {
    if (!s || !regions || n == 0) return fail(DTT_EINVAL, "dtt_schedule_add_chunk: no regions");
    if (writers == 0) return fail(DTT_EINVAL, "dtt_schedule_add_chunk: a chunk needs writers >= 1");
    HostChunk ch;
    ch.writers = writers;
    for (uint32_t i = 0; i < n; ++i) {
        const dtt_region& r = regions[i];
        if (r.rows > 1 && r.pitch < r.row_bytes)
            return fail(DTT_EINVAL, "dtt_schedule_add_chunk: region %u has pitch < row_bytes", i);
        if (r.rows == 0 || r.row_bytes == 0) continue;
        if (r.rows == 1 || r.pitch == r.row_bytes)
            block_regions(r.offset, r.rows, r.row_bytes, r.row_bytes, &ch.regions);
        else
            ch.regions.push_back(r);
    }
    s->chunks.push_back(std::move(ch));
    return DTT_OK;
}

int dtt_schedule_add_chunk_to(dtt_schedule* s, const dtt_region* regions, const dtt_dest* dests,
                              uint32_t n, uint32_t writers, uint32_t peer_mask) {
    if (!dests) {
        const int rc = dtt_schedule_add_chunk(s, regions, n, writers);
        if (rc == DTT_OK) s->chunks.back().peers = peer_mask;
        return rc;
    }
    if (!s || !regions || n == 0) return fail(DTT_EINVAL, "dtt_schedule_add_chunk_to: no regions");
    if (writers == 0) return fail(DTT_EINVAL, "dtt_schedule_add_chunk_to: a chunk needs writers >= 1");
    HostChunk ch;
    ch.writers = writers;
    ch.peers = peer_mask;
    for (uint32_t i = 0; i < n; ++i) {
        const dtt_region& r = regions[i];
        const dtt_dest& d = dests[i];
        if (r.rows > 1 && (r.pitch < r.row_bytes || d.pitch < r.row_bytes))
            return fail(DTT_EINVAL, "dtt_schedule_add_chunk_to: region %u has a (destination) pitch below its row bytes", i);
        if (r.rows == 0 || r.row_bytes == 0) continue;
        const bool src_contig = r.rows == 1 || r.pitch == r.row_bytes;
        const bool dst_contig = r.rows == 1 || d.pitch == r.row_bytes;
        if (src_contig && dst_contig) {     // one byte range on both sides, cut at 1 GiB together
            const uint64_t bytes = r.rows * r.row_bytes;
            for (uint64_t pos = 0; pos < bytes; pos += DTT_LINEAR_MAX) {
                const uint64_t len = (bytes - pos) < DTT_LINEAR_MAX ? (bytes - pos) : DTT_LINEAR_MAX;
                ch.regions.push_back(dtt_region{r.offset + pos, len, 1, len});
                ch.dests.push_back(dtt_dest{d.offset + pos, len});
            }
        } else {
            ch.regions.push_back(r);
            ch.dests.push_back(dtt_dest{d.offset, r.rows > 1 ? d.pitch : r.row_bytes});
        }
    }
    s->chunks.push_back(std::move(ch));
    return DTT_OK;
}

int dtt_schedule_get_dests(const dtt_schedule* s, uint32_t chunk, dtt_dest* dests_out, uint64_t cap,
                           uint64_t* n_dests, uint32_t* peer_mask) {
    if (!s || chunk >= s->chunks.size()) return fail(DTT_EINVAL, "dtt_schedule_get_dests: no such chunk");
    const HostChunk& c = s->chunks[chunk];
    if (n_dests) *n_dests = c.dests.size();
    if (peer_mask) *peer_mask = c.peers;
    if (dests_out) {
        const uint64_t n = c.dests.size() < cap ? c.dests.size() : cap;
        if (n) std::memcpy(dests_out, c.dests.data(), n * sizeof(dtt_dest));
    }
    return DTT_OK;
}

int dtt_schedule_whole(uint64_t base_off, uint64_t rows, uint64_t row_bytes, uint64_t pitch,
                       uint32_t num_programs, dtt_schedule** out) {
    if (!out || num_programs == 0) return fail(DTT_EINVAL, "dtt_schedule_whole: num_programs must be >= 1");
    if (rows > 1 && pitch < row_bytes) return fail(DTT_EINVAL, "dtt_schedule_whole: pitch < row_bytes");
    dtt_schedule* s = new (std::nothrow) dtt_schedule();
    if (!s) return fail(DTT_ENOMEM, "dtt_schedule_whole: out of memory");
    HostChunk ch;
    ch.writers = num_programs;
    block_regions(base_off, rows, row_bytes, pitch, &ch.regions);
    s->chunks.push_back(std::move(ch));
    *out = s;
    return DTT_OK;
}

int dtt_schedule_chunks(uint64_t base_off, uint64_t rows, uint64_t row_bytes, uint64_t pitch,
                        uint32_t num_chunks, dtt_schedule** out) {
    if (!out || num_chunks == 0 || num_chunks > rows)
        return fail(DTT_EINVAL, "dtt_schedule_chunks: need 1 <= num_chunks <= rows");
    if (rows > 1 && pitch < row_bytes) return fail(DTT_EINVAL, "dtt_schedule_chunks: pitch < row_bytes");
    dtt_schedule* s = new (std::nothrow) dtt_schedule();
    if (!s) return fail(DTT_ENOMEM, "dtt_schedule_chunks: out of memory");
    const uint64_t block = (rows + num_chunks - 1) / num_chunks;
    for (uint64_t r0 = 0; r0 < rows; r0 += block) {
        const uint64_t nr = (rows - r0) < block ? (rows - r0) : block;
        HostChunk ch;
        ch.writers = 1;
        block_regions(base_off + r0 * pitch, nr, row_bytes, pitch, &ch.regions);
        s->chunks.push_back(std::move(ch));
    }
    *out = s;
    return DTT_OK;
}

int dtt_schedule_tile_chunks(uint64_t base_off, uint64_t M, uint64_t N, uint32_t elem_bytes,
                             uint64_t pitch, uint32_t BM, uint32_t BN, uint32_t tiles_per_chunk,
                             const dtt_order* order, dtt_order_fn fn, void* ctx,
                             dtt_schedule** out) {
    if (!out || M == 0 || N == 0 || elem_bytes == 0 || BM == 0 || BN == 0 || tiles_per_chunk == 0)
        return fail(DTT_EINVAL, "dtt_schedule_tile_chunks: sizes must be positive");
    if (M > 1 && pitch < N * elem_bytes) return fail(DTT_EINVAL, "dtt_schedule_tile_chunks: pitch < row bytes");
    const uint64_t tiles_m64 = (M + BM - 1) / BM, tiles_n64 = (N + BN - 1) / BN;
    if (tiles_m64 > 0xFFFFFFFFull || tiles_n64 > 0xFFFFFFFFull)
        return fail(DTT_EINVAL, "dtt_schedule_tile_chunks: too many tiles");
    const uint32_t tiles_m = (uint32_t)tiles_m64, tiles_n = (uint32_t)tiles_n64;
    const uint64_t T = tiles_m64 * tiles_n64;
    const uint32_t kind = order ? order->kind : (uint32_t)DTT_ORDER_ROW_MAJOR;
    const uint32_t gm = order ? order->group_m : 0;
    if (!fn && kind != DTT_ORDER_ROW_MAJOR && !(kind == DTT_ORDER_GROUPED && gm > 0))
        return fail(DTT_EINVAL, "dtt_schedule_tile_chunks: bad builtin order");
    std::vector<uint8_t> seen(T, 0);
    dtt_schedule* s = new (std::nothrow) dtt_schedule();
    if (!s) return fail(DTT_ENOMEM, "dtt_schedule_tile_chunks: out of memory");
    HostChunk cur;
    cur.writers = 0;
    for (uint64_t step = 0; step < T; ++step) {
        uint32_t tm = 0, tn = 0;
        if (fn) {
            if (fn(step, ctx, &tm, &tn) != 0) {
                delete s;
                return fail(DTT_EINVAL, "dtt_schedule_tile_chunks: order callback failed at step %llu",
                            (unsigned long long)step);
            }
        } else {
            tile_of(kind, gm, step, tiles_m, tiles_n, &tm, &tn);
        }
        if (tm >= tiles_m || tn >= tiles_n || seen[(uint64_t)tm * tiles_n + tn]) {
            delete s;
            return fail(DTT_EINVAL, "dtt_schedule_tile_chunks: order is not a bijection onto the tiles");
        }
        seen[(uint64_t)tm * tiles_n + tn] = 1;
        const uint64_t r0 = (uint64_t)tm * BM, c0 = (uint64_t)tn * BN;
        const uint64_t rows = (M - r0) < BM ? (M - r0) : BM;
        const uint64_t cols = (N - c0) < BN ? (N - c0) : BN;
        cur.regions.push_back(dtt_region{base_off + r0 * pitch + c0 * elem_bytes, cols * elem_bytes,
                                         rows, pitch});
        cur.writers += 1;
        if (cur.writers == tiles_per_chunk || step + 1 == T) {
            s->chunks.push_back(std::move(cur));
            cur = HostChunk();
            cur.writers = 0;
        }
    }
    *out = s;
    return DTT_OK;
}

int dtt_schedule_info(const dtt_schedule* s, uint32_t* n_chunks, uint64_t* n_regions) {
    if (!s) return fail(DTT_EINVAL, "dtt_schedule_info: NULL schedule");
    uint64_t nr = 0;
    for (const auto& c : s->chunks) nr += c.regions.size();
    if (n_chunks) *n_chunks = (uint32_t)s->chunks.size();
    if (n_regions) *n_regions = nr;
    return DTT_OK;
}

int dtt_schedule_get(const dtt_schedule* s, uint32_t chunk, dtt_region* regions_out,
                     uint64_t cap, uint64_t* n_regions, uint32_t* writers) {
    if (!s || chunk >= s->chunks.size()) return fail(DTT_EINVAL, "dtt_schedule_get: no such chunk");
    const HostChunk& c = s->chunks[chunk];
    if (n_regions) *n_regions = c.regions.size();
    if (writers) *writers = c.writers;
    if (regions_out) {
        const uint64_t n = c.regions.size() < cap ? c.regions.size() : cap;
        if (n) std::memcpy(regions_out, c.regions.data(), n * sizeof(dtt_region));
    }
    return DTT_OK;
}

}  // extern "C"
