// sv_layout.h — parameter blocks and workspace layout shared by host and device code.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace sv {

// ---- launch geometry ---------------------------------------------------------------------
constexpr int kThreads = 256;               // threads per streaming block
constexpr int kWarps = kThreads / 32;
constexpr int kTileBytes = 16384;           // one bulk copy (a draw-pass or selection stage per row)
constexpr int kStatsTileBytes = 32768;      // one stage of the statistics pass (two 16 KB halves)
constexpr int kStatsStages = 3;             // pipeline depth of the statistics pass
constexpr int kStatsThreads = kThreads + 32;   // eight consumer warps and one producer warp
constexpr int kUnitTiles = 16;              // aim for (row, chunk) units of about this many tiles
constexpr int kDrawStages = 3;              // pipeline depth of the draw pass (two rows per stage)
constexpr int kDrawUnitSubs = 64;           // draw-pass units: 64 sub-chunks (2 tiles) of a row pair
constexpr int kSubBytes = 512;              // bytes of one row per draw sub-chunk (32 x 16 B)
constexpr int kMaxSplit = 64;               // most chunks per row
constexpr int kUnitTarget = 1024;           // at least about this many (row, chunk) units
constexpr int kExactSplit = 16;             // chunks per row in the float-float tier
constexpr int kExactCap = 2048;             // most queued items per call in the float-float tier
constexpr int kExactGroup = 1;              // draw sub-chunks per warp unit in the float-float tier
constexpr long long kWaitLimitCycles = 4000000000LL;   // ~2 s at 2 GHz: bounded barrier waits
constexpr unsigned kSuspendHintNs = 100000;  // a waiting thread sleeps at most this long per try

// ---- certification constants of the float32 tier ------------------------------------------
// Largest relative error of the fast exponential (ex2.approx.ftz.f32) over every float32
// input in [-125, 1]: 1.4584e-7, measured exhaustively on GB300 (sv_selftest_exp2_all; the
// GPU tests re-check it).  Results below 2^-125 flush to zero, an absolute error far below the
// 1e-12 slack every bound carries.
constexpr double kEx2RelErr = 1.5e-7;
constexpr double kU32 = 5.9604644775390625e-08;        // 2^-24, float32 unit roundoff
constexpr double kLn2 = 0.69314718055994530942;
// Relative error of 2^y per unit |y| from rounding y twice in float32: 2 * 2^-24 * ln 2.
constexpr double kYRound = 2.0 * kU32 * kLn2;

// ---- row descriptors ------------------------------------------------------------------------
// A "row set" is a per-sequence logit tensor: row (b, j) starts at base + (b*rows_per_seq + j)*pitch.
struct RowSet {
    const char *base;
    int64_t pitch_bytes;
    int rows_per_seq;
    int rows_used;        // rows j < rows_used of every sequence are candidates
    int skip_greedy;      // 1: rows of greedy sequences are not streamed
};

// Per-(row, chunk, warp) partial of the statistics pass (float32 only: no FP64 on the hot path).
struct WarpPartial {
    float s_hi, s_lo;   // sum of 2^(x c - r) over the warp's elements, float-float
    float a;            // sum of 2^(x c - r) * |x c - r| (feeds the certified error bound)
    int r;              // integer reference exponent, >= x*c of every element seen; -2^30 if none
    float maxv;         // largest logit seen (NaN-free)
    int argmax;         // its lowest index
    int flags;          // kFlagNaN | kFlagPosInf
    int pad;
};

constexpr int kFlagNaN = 1;
constexpr int kFlagPosInf = 2;
constexpr int kNoRef = -(1 << 30);

// Combined statistics of one row.
struct RowStat {
    float s_hi, s_lo;   // S = sum_v 2^(x_v c - r) as float-float (sampled rows), c = log2(e)/T
    float err;          // certified relative error bound of S (float32 tier)
    float maxv;         // greedy rows: the maximum and its lowest index
    int argmax;
    int r;              // the integer reference exponent r
    int flags;
    float ay;           // sum_v 2^(x_v c - r) |x_v c - r| / S: mean |exponent| under the row
};

// Nucleus (top-p) cut of a row: token v is kept iff x_v > cut_x or (x_v == cut_x and v <= cut_id).
// mass = kept probability mass.  A row without a filter has cut_x = -inf, cut_id = INT32_MAX, mass 1.
struct NucleusCut {
    float cut_x;
    int cut_id;
    double mass;
    double log2_mass;
    int ambiguous;  // the float32 tier could not certify the cut
    float mass_f;   // mass rounded to float32 (for float32 consumers)
};

// Saguaro top-F set of a draft row: v in D iff x_v > top_x or (x_v == top_x and v <= top_id).
struct TopSet {
    float top_x;
    int top_id;
    double p_d;     // probability mass of D (after temperature and top-p) before scaling
    double z;       // normaliser after scaling: 1 - (1 - C) p_d
    double z_err;   // relative error bound of z (float32 tier)
    float z_f;      // z rounded to float32
    float z_err_f;  // z_err rounded up to float32
};

// A row as seen by the draw pass: weight(v) = keep(v) * 2^(x_v c - r) * inv_s * (in_D ? sc_d : 1).
struct DrawRow {
    const char *row;
    float c_hi, c_lo;       // c = log2(e)/T
    float rf;               // reference exponent r (as float)
    float inv_s;            // 1 / (S * nucleus mass * Saguaro normaliser), float32
    float cut_x; int cut_id;
    float top_x; int top_id;
    float sc_d;             // C for tokens in D (1 when no transform)
    float ay;               // bound on sum_v w_v |y_v| for this row's normalised weights w
    float k_lo;             // ln2 c_lo inv_s: weight = 2^(x c_hi - r) (inv_s + x k_lo)
    int pad;
    double norm_err;        // relative error bound of inv_s (normaliser from the stats pass)
};

// One pending draw: t* = inverse CDF of w at u, w = max(q - p, 0) (has_p) or q.
struct DrawItem {
    DrawRow q, p;
    double u;
    int *out;               // where t* is written
    double *dbg_r;          // where R (sum of the weights) is written, or nullptr
    int has_p;
    int filt;               // nucleus cut or top-F set in use
    int seq;
    int k;                  // draw position (accepted count for sv_verify)
    int pad[2];             // a multiple of 16 bytes: the draw pass bulk-copies items
};
static_assert(sizeof(DrawItem) % 16 == 0, "draw items are copied with cp.async.bulk");

// Fuzzy verification: per (pair, chunk) partial of the divergence pass, and per pair its
// float32 divergence, error bound and (when the bound could not settle it) float-float value.
struct DivPart {
    float s_hi, s_lo;       // sum of (q + p) h(d) over the chunk, float-float
    float y;                // sum of (q + p)(|y_q| + |y_p|) (feeds the error bound)
    float pad;
};

struct DivItem {
    double exact;           // float-float divergence (state 2)
    int state;              // 0 float32 only, 1 queued for the float-float pass, 2 done
    int pad;
};

// Exact-tier work item: a draw to redo (draw >= 0) or a sequence whose accept tests must be
// redone (draw < 0).
struct ExactItem {
    int draw;
    int seq;
};

// Counters that each call resets before use (kernel-side).
// Zeroed by the host (one memset) before the statistics pass of every call.
struct Counters {
    int n_draws;
    int n_exact;
    unsigned barrier;       // grid barrier of the exact tier
    int next_unit;          // statistics pass: next (row, chunk) unit to hand out
    int next_draw_unit;     // draw pass: next (item, chunk) unit to hand out
    int q_head;             // lazy verification: next queue position to claim (position 0, then later)
    int q0_tail, q_tail;    // lazy verification: position-0 units / later units queued
    int n_pending;          // lazy verification: sequences not finished yet
    int n_div_exact;        // fuzzy verification: divergences queued for the float-float pass
    int pad[6];
};

inline int div_up(long long a, long long b) { return (int)((a + b - 1) / b); }

// Chunks per row: enough (row, chunk) units to balance ~kUnitTarget of them, chunks >= one tile.
inline int choose_split(long long n_rows, long long row_bytes) {
    const long long row_tiles = row_bytes / kTileBytes;
    long long s = row_tiles / kUnitTiles;                                     // units of ~kUnitTiles tiles
    const long long by_units = (kUnitTarget + n_rows - 1) / (n_rows > 0 ? n_rows : 1);
    if (s < by_units) s = by_units;                                           // small batches: more units
    if (s > row_tiles) s = row_tiles;                                         // but chunks >= one tile
    if (s < 1) s = 1;
    if (s > kMaxSplit) s = kMaxSplit;
    return (int)s;
}

// 16-byte vectors per chunk: whole statistics-pass tiles where the row has them, so only a
// row's last chunk ends in a partial tile.  n_split may shrink; both are returned.
inline void chunk_geometry(long long n_vec, int &n_split, int &chunk_vecs) {
    if (n_vec <= 0) {
        n_split = 1;
        chunk_vecs = 1;
        return;
    }
    const long long tv = kStatsTileBytes / 16;
    long long cv = (n_vec + n_split - 1) / n_split;
    if (cv > tv) cv = (cv + tv - 1) / tv * tv;
    chunk_vecs = (int)cv;
    n_split = (int)((n_vec + cv - 1) / cv);
}

// Sub-chunks of a row in the draw pass: one per 32 16-byte vectors, plus a last one holding the
// (< 16 B) scalar tail of the row.
inline int vec_count(int V, int es) { return (int)(((long long)V * es) / 16); }
inline int sub_chunks(int V, int es) { return div_up(vec_count(V, es), 32) + 1; }
// Draw-pass chunks of a row: kDrawUnitSubs vector sub-chunks each.
inline void draw_geometry(int n_sub, int &d_split, int &d_subs_per_chunk) {
    const int n_vsub = n_sub - 1;
    d_subs_per_chunk = kDrawUnitSubs;
    d_split = n_vsub > 0 ? div_up(n_vsub, kDrawUnitSubs) : 1;
}

// Warp units per item in the float-float tier's row pass: groups of kExactGroup vector
// sub-chunks, plus one for the scalar tail.
inline int exact_groups(int n_sub) { return div_up(n_sub - 1, kExactGroup) + 1; }

// 256-byte aligned bump allocator over the caller's workspace.
struct Carver {
    size_t off = 0;
    template <class T>
    size_t take(size_t count) {
        size_t o = (off + 255) & ~size_t(255);
        off = o + count * sizeof(T);
        return o;
    }
};

}  // namespace sv
