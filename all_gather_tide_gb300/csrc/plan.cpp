// Group planner: the per-parameter layout of Table 2 of the paper ("The Endgame of FSDP
// Communication", arXiv 2610.38228) and the flat chunk lists the kernels walk.
//
// Layout (abstract; Fig. 1; Table 2): parameter p is split on dim 0 into R pieces of
// m_p = ceil(rows_p / R) rows; a piece is s_p = m_p * L_p elements; the pieces of all parameters
// are packed in parameter order at prefix offsets o_p into each rank's shard of S elements.
// Because dim-0 pieces of a row-major tensor are contiguous, rank d's piece of p is the range
// [d*s_p, d*s_p + v(d,p)*L_p) of the tensor, v(d,p) = clamp(rows_p - d*m_p, 0, m_p).
#include <algorithm>

#include "../../include/tide.h"
#include "tide_internal.h"

namespace tide {

namespace {
bool mul_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }
bool add_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_add_overflow(a, b, out); }
}  // namespace

int64_t valid_rows(int64_t rows_p, int64_t m_p, int64_t d) {
    return std::min(m_p, std::max<int64_t>(0, rows_p - d * m_p));
}

int make_layout(int32_t R, int32_t P, const int64_t* rows, const int64_t* row_len, Plan* out) {
    if (!rows || !row_len || !out || R < 1 || R > TIDE_MAX_RANKS || P < 1) return TIDE_EINVAL;
    Plan pl;
    pl.R = R;
    pl.P = P;
    pl.rows.assign(rows, rows + P);
    pl.row_len.assign(row_len, row_len + P);
    pl.m.resize(P);
    pl.s.resize(P);
    pl.o.resize(P);
    int64_t off = 0, un = 0;
    for (int32_t p = 0; p < P; ++p) {
        if (rows[p] < 1 || row_len[p] < 1) return TIDE_EINVAL;
        const int64_t m = rows[p] / R + (rows[p] % R != 0);
        int64_t s, n, Rm;
        if (!mul_ok(m, row_len[p], &s) || !mul_ok(rows[p], row_len[p], &n) || !mul_ok(m, R, &Rm) ||
            !mul_ok(Rm, row_len[p], &Rm))
            return TIDE_ERANGE;
        pl.m[p] = m;
        pl.s[p] = s;
        pl.o[p] = off;
        if (!add_ok(off, s, &off) || !add_ok(un, n, &un)) return TIDE_ERANGE;
    }
    int64_t total;
    if (!mul_ok(off, R, &total) || !mul_ok(total, 4, &total)) return TIDE_ERANGE;
    pl.S = off;
    pl.U = un;
    *out = std::move(pl);
    return TIDE_OK;
}

void make_work_lists(Plan* pl) {
    // Reduce-scatter: destination-major, parameter order within a shard, so each CTA pass
    // writes a contiguous run of the shard and reads R contiguous runs of gradient p.
    pl->rs.clear();
    pl->rs_piece.clear();
    int64_t chunks = 0;
    for (int32_t d = 0; d < pl->R; ++d) {
        for (int32_t p = 0; p < pl->P; ++p) {
            RsSeg sg{};
            sg.dst_off = pl->o[p];
            sg.src_off = int64_t(d) * pl->s[p];
            sg.valid = valid_rows(pl->rows[p], pl->m[p], d) * pl->row_len[p];
            sg.total = pl->s[p];
            sg.chunk_begin = chunks;
            sg.d = d;
            sg.p = p;
            sg.vec = sg.src_off % 8 == 0;  // 16-byte gradient loads; stores adapt to the shard offset
            const int64_t n = (sg.total + kRsChunk - 1) / kRsChunk;
            chunks += n;
            pl->rs_piece.insert(pl->rs_piece.end(), size_t(n), int32_t(pl->rs.size()));
            pl->rs.push_back(sg);
        }
    }
    pl->rs_chunks = chunks;

    // The same pieces cut into the bulk-copy kernel's larger chunks.
    pl->rs_bulk.clear();
    pl->rs_bulk_piece.clear();
    chunks = 0;
    for (RsSeg sg : pl->rs) {
        sg.chunk_begin = chunks;
        const int64_t n = (sg.total + kBulkChunk - 1) / kBulkChunk;
        chunks += n;
        pl->rs_bulk_piece.insert(pl->rs_bulk_piece.end(), size_t(n), int32_t(pl->rs_bulk.size()));
        pl->rs_bulk.push_back(sg);
    }
    pl->rs_bulk_chunks = chunks;

    // Summing step over staging slots: slot r of destination d holds contributor r's slice d of
    // parameter p at o_p, so a piece reads every slot at o_p; chunk ranges count from 0 for each d.
    pl->rs_slots.clear();
    pl->rs_slot_piece.clear();
    std::vector<int64_t> first(size_t(pl->P));
    chunks = 0;
    for (int32_t p = 0; p < pl->P; ++p) {
        first[size_t(p)] = chunks;
        const int64_t n = (pl->s[p] + kBulkChunk - 1) / kBulkChunk;
        chunks += n;
        pl->rs_slot_piece.insert(pl->rs_slot_piece.end(), size_t(n), p);
    }
    pl->rs_slot_chunks = chunks;
    for (int32_t d = 0; d < pl->R; ++d) {
        for (int32_t p = 0; p < pl->P; ++p) {
            RsSeg sg{};
            sg.dst_off = pl->o[p];
            sg.src_off = pl->o[p];
            sg.valid = valid_rows(pl->rows[p], pl->m[p], d) * pl->row_len[p];
            sg.total = pl->s[p];
            sg.chunk_begin = first[size_t(p)];
            sg.d = 0;
            sg.p = 0;
            sg.vec = sg.src_off % 8 == 0;
            pl->rs_slots.push_back(sg);
        }
    }

    // All-gather placement: source-rank-major runs of valid elements; padding never appears.
    pl->ag.clear();
    pl->ag_run.clear();
    chunks = 0;
    for (int32_t r = 0; r < pl->R; ++r) {
        for (int32_t p = 0; p < pl->P; ++p) {
            const int64_t len = valid_rows(pl->rows[p], pl->m[p], r) * pl->row_len[p];
            if (len == 0) continue;
            AgSeg sg{};
            sg.src_off = pl->o[p];
            sg.dst_off = int64_t(r) * pl->s[p];
            sg.len = len;
            sg.chunk_begin = chunks;
            sg.r = r;
            sg.p = p;
            sg.vec = (sg.src_off % 8 == 0) && (sg.dst_off % 8 == 0);
            const int64_t n = (len + kAgChunk - 1) / kAgChunk;
            chunks += n;
            pl->ag_run.insert(pl->ag_run.end(), size_t(n), int32_t(pl->ag.size()));
            pl->ag.push_back(sg);
        }
    }
    pl->ag_chunks = chunks;

    pl->ag_bulk.clear();
    pl->ag_vec_elems = 0;
    chunks = 0;
    for (AgSeg sg : pl->ag) {
        if (sg.vec) pl->ag_vec_elems += sg.len;
        sg.chunk_begin = chunks;
        chunks += (sg.len + kAgBulkChunk - 1) / kAgBulkChunk;
        pl->ag_bulk.push_back(sg);
    }
    pl->ag_bulk_chunks = chunks;
}

int plan_rs_pieces(int32_t R, int32_t P, const int64_t* rows, const int64_t* row_len, RsSeg* out, size_t cap,
                   int64_t* nchunks) {
    if (!rows || !row_len || !out || !nchunks || R < 1 || R > TIDE_MAX_RANKS || P < 1) return TIDE_EINVAL;
    if (size_t(R) * size_t(P) > cap) return TIDE_ERANGE;
    // pass 1: check every parameter and count the chunks of one destination rank's pieces
    int64_t per_rank = 0, off = 0, total = 0;
    for (int32_t p = 0; p < P; ++p) {
        if (rows[p] < 1 || row_len[p] < 1) return TIDE_EINVAL;
        const int64_t m = rows[p] / R + (rows[p] % R != 0);
        int64_t s, n, Rm;
        if (!mul_ok(m, row_len[p], &s) || !mul_ok(rows[p], row_len[p], &n) || !mul_ok(m, R, &Rm) ||
            !mul_ok(Rm, row_len[p], &Rm) || !add_ok(off, s, &off))
            return TIDE_ERANGE;
        per_rank += (s + kRsChunk - 1) / kRsChunk;
    }
    if (!mul_ok(off, R, &total) || !mul_ok(total, 4, &total) || !mul_ok(per_rank, R, &total)) return TIDE_ERANGE;
    // pass 2: the pieces in make_work_lists' order (destination-major, parameter order within a
    // shard), with their chunk ranges in the flat chunk list
    off = 0;
    int64_t before = 0;  // chunks of parameters 0..p-1 in one rank's list
    for (int32_t p = 0; p < P; ++p) {
        const int64_t m = rows[p] / R + (rows[p] % R != 0);
        const int64_t s = m * row_len[p];
        for (int32_t d = 0; d < R; ++d) {
            RsSeg sg{};
            sg.dst_off = off;
            sg.src_off = int64_t(d) * s;
            sg.valid = valid_rows(rows[p], m, d) * row_len[p];
            sg.total = s;
            sg.chunk_begin = int64_t(d) * per_rank + before;
            sg.d = d;
            sg.p = p;
            sg.vec = sg.src_off % 8 == 0;
            out[size_t(d) * size_t(P) + size_t(p)] = sg;
        }
        off += s;
        before += (s + kRsChunk - 1) / kRsChunk;
    }
    *nchunks = per_rank * R;
    return TIDE_OK;
}

}  // namespace tide
