// sv_flow.cu — verification without filters as one cooperative dataflow kernel: the statistics
// pass, the accept tests, the residual / bonus draws and the float-float tier of every
// sequence, each started as soon as what it needs is complete.
//
// ["Speculative Speculative Decoding" notes, §2.2 steps ①-④; "Accelerating LLM Decoding with
//  Speculative Sampling (2023)" notes, §3 (accept s with probability min(1, q(s)/p(s)); the
//  first rejection ends the scan, and the draft tokens to its right decide nothing)]
//
// A queue of work units feeds a persistent grid (every block resident: blocks wait for units
// that other blocks queue).  In each block a producer warp takes units in queue order and
// stages them through a ring of 32 KB shared-memory stages, eight consumer warps work on the
// stages, and a finisher warp takes the per-sequence and per-draw decisions off the consumers'
// path.  The units are:
//   statistics  (row, chunk): the streaming pass of sv_stats.cuh;
//   draw        (draw, chunk): 64 sub-chunks of the draw's q (and p) row, 16 KB of each per stage;
//               one float32 sum per 32-vector sub-chunk (sv_draw.cuh);
//   exact C     (item, group): the float-float row pass of the float-float tier over 32 sub-chunks
//               of an uncertified draw (sign-split sums, normalisers, tokens of uncertain sign);
//   exact A     (item, row, quarter): float-float row sums of a sequence whose accept test the
//               float32 tier could not certify.
// The finisher's requests are:
//   sequence    a sequence's queued rows are complete: row statistics, accept tests (or the greedy
//               match), then the draw item and its draw units, or (lazy mode) the next rows;
//   finish      a draw's units are complete: t* with a certified margin, or exact C units;
//   exact B     an uncertified sequence's exact A units are complete: its accept tests in float64
//               from the exact sums, then its draw and exact C units;
//   exact D     an item's exact C units are complete: exact normalisers, the float-float scan and t*.
// A sequence counts as pending until its last token is written; once none is pending and the
// queue is drained, every block ends.
//
// Eager mode (sv_verify) queues every row of every sequence at once, in sequence order, so that
// the draws and float-float work of early sequences run while later ones stream (their rows
// still in L2).  Lazy mode (sv_verify_lazy) queues position 0 of every sequence, then each
// sequence's next rows only after its accept test passes (positions 0 and 1 one at a time, the
// rest in one batch), so rows after a sequence's first rejection are never read.  Calls with
// top-k, top-p or sigma_{F,C} need selection passes between the statistics and the tests and
// run the staged pipeline of sv_verify.cu instead.
#include <math.h>

#include "sv_accept.cuh"
#include "sv_draw.cuh"
#include "sv_exact.cuh"
#include "sv_exp2_table.h"
#include "sv_host.h"
#include "sv_stats.cuh"

namespace sv {

// ---- geometry ------------------------------------------------------------------------------
constexpr int kFlowThreads = kStatsThreads + 32;   // 8 consumer warps, producer, finisher
constexpr int kFlowRing = 64;                      // finisher requests in flight per block
constexpr int kFlowTCache = 1024;                  // temperatures cached in shared memory
// shared memory: control block (barriers, flags, stage descriptions), finisher ring, the eight
// consumer warps' partials of each stage's unit and their arrival counts, temperatures, exp2 table
constexpr int kFlowOffRing = 1024;
constexpr int kFlowOffPart = kFlowOffRing + kFlowRing * 16;
constexpr int kFlowOffPartCnt = kFlowOffPart + kStatsStages * kWarps * (int)sizeof(WarpPartial);
constexpr int kFlowOffTCache = kFlowOffPartCnt + 64;
constexpr int kFlowOffTab = kFlowOffTCache + kFlowTCache * 4;
constexpr int kFlowCtlBytes = kFlowOffTab + 256 * 8;
constexpr size_t kFlowSmemBytes = (size_t)kFlowCtlBytes + (size_t)kStatsStages * kStatsTileBytes;
static_assert(2 * kStatsStages * 8 + 16 + kStatsStages * (int)sizeof(TileMeta) <= 1024, "control block");
static_assert(kDrawUnitSubs * 32 == 2 * (kTileBytes / 16), "a draw unit is two stages of 16 KB per row");

// Queue words: bit 63 valid, bits 60..62 the unit's type, bits 32..59 its payload, bits 0..31
// its index.  A statistics unit's payload is (cumulative warp count << 8) | (first position << 2)
// | batch kind.
constexpr int kUnitStats = 0, kUnitDraw = 1, kUnitExactC = 2, kUnitExactA = 3;
// Batch kinds of statistics units: one position, every remaining position, or the completing
// rows of a sequence handed to the float-float tier (lazy mode).
constexpr int kBatchOne = 0, kBatchTail = 1, kBatchComplete = 2;
constexpr int kLazyTail = 2;
// Stage flags beyond those of the statistics pass.
constexpr int kTileDraw = 16, kTileExactC = 32, kTileExactA = 64;
// Finisher requests.
constexpr int kReqSeq = 0, kReqFinish = 1, kReqExactB = 2, kReqExactD = 3;

struct FlowArgs {
    StatsArgs st;        // row sets, temperatures, partials, counters, stats
    AcceptArgs acc;      // accept context (no nucleus cuts, no top-F sets)
    unsigned long long *units;   // [cap] the queue
    long long cap;
    long long q1_base;   // units[0, q1_base): written by the init kernel; units[q1_base, cap): appended
    FlowCounters *fc;    // the kernel's counters (one cache line each)
    int *pos_cnt;        // [B] consumer warps done with the sequence's statistics units (cumulative)
    int n_seq;
    int lazy;
    // draws
    int n_vec, n_sub, d_split;
    float *subs;         // [B][n_sub] float32 sum of the weights of each sub-chunk
    int *draw_cnt;       // [B] consumer warps done with the draw's units
    // float-float tier
    int *x_cnt;          // [cap_x] consumer warps done with the item's exact C units
    int *a_cnt;          // [cap_x] consumer warps done with the item's exact A units
    float4 *xsubs;       // [cap_x][n_sub] sign-split float-float sums (A_q, A_p) per sub-chunk
    float4 *xnorm;       // [cap_x][n_sub] float-float normaliser parts (S_q, S_p) per sub-chunk
    int *xunc;           // [cap_x][kExactUncCap] tokens of uncertain sign (the first kFlowUncCap used)
    float2 *xuncw;       // [cap_x][kFlowUncCap] their exact residuals (written in exact D)
    double *xsum;        // [cap_x][max_slots][kFlowSplitA][kWarps] exact row sums (exact A)
    ExactDraw *xdraw;    // [cap_x] the draw of an item whose accept tests were redone
    int cap_x;
    int x_groups;        // exact C units per item
    int max_slots;
};

__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Release / acquire fence at GPU scope: the thread's earlier writes (and those it has observed)
// are visible to any thread that observes its later writes, and it sees what such writers wrote
// before their own release.  Lighter than the sequentially consistent __threadfence().
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ unsigned long long unit_word(int type, unsigned payload, unsigned index) {
    return (1ull << 63) | ((unsigned long long)type << 60) | ((unsigned long long)(payload & 0x0FFFFFFFu) << 32) | index;
}

// Row id -> (sequence, position) in the candidate-row numbering of the statistics pass.
__device__ __forceinline__ void seq_pos(const FlowArgs &F, long long rid, int &b, int &j) {
    const int K = F.acc.K;
    if (rid < F.st.n_rows0) {
        b = (int)(rid / (K + 1));
        j = (int)(rid - (long long)b * (K + 1));
    } else {
        const long long r = rid - F.st.n_rows0;
        b = (int)(r / K);
        j = (int)(r - (long long)b * K);
    }
}

// Claim n slots of the appended region (one thread).  Each unit is queued once, so the region
// is sized for all of them; running out means a bug, reported rather than written past.
__device__ __forceinline__ long long flow_claim(const FlowArgs &F, int n) {
    const long long base = F.q1_base + atomicAdd(&F.fc->q_tail.v, n);
    if (base + n > F.cap) {
        report_error(F.st.stats, SV_ERR_WORKSPACE, -1);
        return -1;
    }
    return base;
}

// Queue rows of sequence b (one thread): target rows j0..j1 and draft rows j0..min(j1, K-1) when
// `with_d`.  `kind` tells the finisher how to treat the batch; `cum` is the sequence's
// cumulative count of consumer warps so far.
__device__ void flow_enqueue_rows(const FlowArgs &F, int b, int j0, int j1, bool with_d, int kind, int cum,
                                  bool initial) {
    const int K = F.acc.K, ns = F.st.n_split;
    const int n_t = j1 - j0 + 1;
    const int n_d = with_d ? max(0, min(j1, K - 1) - j0 + 1) : 0;
    const int n = (n_t + n_d) * ns;
    const unsigned payload = ((unsigned)(cum + n * kWarps) << 8) | ((unsigned)j0 << 2) | (unsigned)kind;
    long long base;
    if (initial) {
        base = atomicAdd(&F.fc->q0_tail.v, n);
        if (base + n > F.q1_base) {
            report_error(F.st.stats, SV_ERR_WORKSPACE, b);
            return;
        }
    } else {
        base = flow_claim(F, n);
        if (base < 0) return;
    }
    int k = 0;
    for (int j = j0; j <= j1; ++j) {
        const long long rid = (long long)b * (K + 1) + j;
        for (int c = 0; c < ns; ++c) st_relaxed_u64(&F.units[base + k++], unit_word(kUnitStats, payload, (unsigned)(rid * ns + c)));
    }
    for (int j = j0; j < j0 + n_d; ++j) {
        const long long rid = F.st.n_rows0 + (long long)b * K + j;
        for (int c = 0; c < ns; ++c) st_relaxed_u64(&F.units[base + k++], unit_word(kUnitStats, payload, (unsigned)(rid * ns + c)));
    }
}

// Queue n units of one type with indices first..first+n-1 (one thread).  The data they refer
// to was written before: the fence orders it before the queue words.
__device__ void flow_enqueue(const FlowArgs &F, int type, long long first, int n) {
    __threadfence();
    const long long base = flow_claim(F, n);
    if (base < 0) return;
    for (int k = 0; k < n; ++k) st_relaxed_u64(&F.units[base + k], unit_word(type, 0, (unsigned)(first + k)));
}

__device__ __forceinline__ void flow_done(const FlowArgs &F) { atomicSub(&F.fc->n_pending.v, 1); }

// One sequence of the init kernel: validate, mark the debug fields undefined, queue its first rows.
__device__ void flow_init_seq(const FlowArgs &F, int b) {
    F.pos_cnt[b] = 0;
    const AcceptArgs &a = F.acc;
    const int K = a.K;
    const float T = a.temperature[b];
    const bool greedy = (T == 0.0f);
    int32_t *outs = a.out_tokens + (size_t)b * (K + 1);
    if (a.debug)
        for (int i = 0; i < (K + 1) * SV_DEBUG_FIELDS; ++i) a.debug[(size_t)b * (K + 1) * SV_DEBUG_FIELDS + i] = NAN;
    auto fail = [&](int code) {
        report_error(a.stats, code, b);
        for (int j = 0; j <= K; ++j) outs[j] = -1;
        a.accept_len[b] = 0;
    };
    if (!(greedy || (T >= 1e-3f && T <= 1e3f))) {
        fail(SV_ERR_INVALID_ARG);
        return;
    }
    for (int j = 0; j < K; ++j) {
        const int s = a.tokens[(size_t)b * K + j];
        if (s < 0 || s >= a.V) {
            fail(SV_ERR_BAD_TOKEN);
            return;
        }
    }
    atomicAdd(&F.fc->n_pending.v, 1);
    const bool with_d = !greedy && K > 0;
    if (!F.lazy || kLazyTail <= 0) flow_enqueue_rows(F, b, 0, K, with_d, kBatchTail, 0, true);
    else flow_enqueue_rows(F, b, 0, 0, with_d, kBatchOne, 0, true);
}

// Every sequence's init (grid-stride over sequences), and the clearing of the appended part of
// the queue and of the per-item counters.
__global__ void __launch_bounds__(kThreads) k_flow_init(const FlowArgs F, int B) {
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long nthr = (long long)gridDim.x * blockDim.x;
    for (long long i = F.q1_base + tid; i < F.cap; i += nthr) F.units[i] = 0ull;
    for (long long i = tid; i < B; i += nthr) F.draw_cnt[i] = 0;
    for (long long i = tid; i < F.cap_x; i += nthr) {
        F.x_cnt[i] = 0;
        F.a_cnt[i] = 0;
        F.acc.exact_unc[i] = 0;
    }
    for (long long bb = tid; bb < B; bb += nthr) flow_init_seq(F, (int)bb);
}

// ------------------------------------------------------------------------------------------
// Finisher: decisions
// ------------------------------------------------------------------------------------------

// Push a float-float item for sequence b (draw >= 0: that draw; else the accept tests) and
// queue its units.  Past the tier's capacity the float32 result stands, counted as unresolved.
__device__ void flow_to_exact(const FlowArgs &F, int draw, int b) {
    const AcceptArgs &a = F.acc;
    stats_add(a.stats, &a.stats->reresolved, 1);
    const int i = atomicAdd(&F.fc->n_exact.v, 1);
    if (i >= F.cap_x) {
        stats_add(a.stats, &a.stats->unresolved, 1);
        flow_done(F);
        return;
    }
    a.exact[i] = {draw, b};
    if (draw >= 0) {
        flow_enqueue(F, kUnitExactC, (long long)i * F.x_groups, F.x_groups);
    } else {
        const int n_rows = 2 * a.K + 1;
        for (int slot = 0; slot < n_rows; ++slot)
            flow_enqueue(F, kUnitExactA, ((long long)i * F.max_slots + slot) * kFlowSplitA, kFlowSplitA);
    }
}

// The draw item of a sampled sequence that accepted k tokens (k < K and a residual: rows k), its
// units queued.
template <int ES>
__device__ void flow_draw(const FlowArgs &F, int b, int k, float T, const RowStat &rq, const RowStat &rp) {
    const AcceptArgs &a = F.acc;
    const int K = a.K;
    DrawItem it;
    const char *qrow = a.tgt.base + ((long long)b * a.tgt.rows_per_seq + k) * a.tgt.pitch_bytes;
    it.q = draw_row(qrow, T, rq, nullptr, nullptr, 1.0f);
    it.has_p = k < K && !a.draw_from_q;
    if (it.has_p) {
        const char *prow = a.drf.base + ((long long)b * a.drf.rows_per_seq + k) * a.drf.pitch_bytes;
        it.p = draw_row(prow, T, rp, nullptr, nullptr, 1.0f);
    } else {
        it.p = {};
        it.p.top_x = INFINITY;
        it.p.cut_x = -INFINITY;
        it.p.cut_id = 0x7FFFFFFF;
    }
    it.filt = 0;
    it.u = a.uniforms[(size_t)b * (K + 1) + K];
    it.out = a.out_tokens + (size_t)b * (K + 1) + k;
    it.dbg_r = a.debug ? a.debug + (size_t)b * (K + 1) * SV_DEBUG_FIELDS + SV_DBG_R : nullptr;
    it.seq = b;
    it.k = k;
    const int d = atomicAdd(&F.fc->n_draws.v, 1);
    a.draws[d] = it;
    flow_enqueue(F, kUnitDraw, (long long)d * F.d_split, F.d_split);
}

// Debug values of position j of a sampled sequence (both rows' statistics known).
template <int ES>
__device__ void flow_debug(const AcceptArgs &a, int b, int j, float T, const RowStat &rq, const RowStat *rp) {
    const int K = a.K;
    double *dbg = a.debug + ((size_t)b * (K + 1) + j) * SV_DEBUG_FIELDS;
    dbg[SV_DBG_LSE_Q] = rs_g(rq) * kLn2;
    dbg[SV_DBG_MASS_Q] = 1.0;
    if (rp == nullptr) return;
    const int s = a.tokens[(size_t)b * K + j];
    const double cd = 1.4426950408889634074 / (double)T;
    const char *trow = a.tgt.base + ((long long)b * a.tgt.rows_per_seq + j) * a.tgt.pitch_bytes;
    const char *drow = a.drf.base + ((long long)b * a.drf.rows_per_seq + j) * a.drf.pitch_bytes;
    const float xt = load_elem<ES>(trow, s), xd = load_elem<ES>(drow, s);
    const double lq = xt == -INFINITY ? -INFINITY : (double)xt * cd - rs_g(rq);
    const double lp = xd == -INFINITY ? -INFINITY : (double)xd * cd - rs_g(*rp);
    dbg[SV_DBG_LSE_P] = rs_g(*rp) * kLn2;
    dbg[SV_DBG_Q_S] = exp2(lq);
    dbg[SV_DBG_P_S] = exp2(lp);
    dbg[SV_DBG_RATIO] = (lp == -INFINITY) ? (lq == -INFINITY ? 0.0 : INFINITY) : exp2(lq - lp);
    dbg[SV_DBG_MASS_P] = 1.0;
}

__device__ __forceinline__ RowStat shfl_rowstat(const RowStat &r, int src) {
    RowStat o;
    o.s_hi = __shfl_sync(0xFFFFFFFFu, r.s_hi, src);
    o.s_lo = __shfl_sync(0xFFFFFFFFu, r.s_lo, src);
    o.err = __shfl_sync(0xFFFFFFFFu, r.err, src);
    o.maxv = __shfl_sync(0xFFFFFFFFu, r.maxv, src);
    o.argmax = __shfl_sync(0xFFFFFFFFu, r.argmax, src);
    o.r = __shfl_sync(0xFFFFFFFFu, r.r, src);
    o.flags = __shfl_sync(0xFFFFFFFFu, r.flags, src);
    o.ay = __shfl_sync(0xFFFFFFFFu, r.ay, src);
    return o;
}

__device__ __forceinline__ bool rowstat_bad(const RowStat &r, bool greedy) {
    return (r.flags != 0) || (greedy ? !isfinite(r.maxv) : !rs_sampled_ok(r));
}

// The batch of rows starting at position j0 of sequence b is complete (one warp).  In eager
// mode the batch is every row of the sequence: all are checked first (a non-finite row anywhere
// fails the sequence, and every position's debug values are written), then the positions are
// walked.  When every row was one unit (large batches), the consumers combined the rows'
// statistics already and lane j loads position j's statistics and the logits of its drafted
// token, all at once; otherwise the rows are combined here from the chunks' partials, one after
// another.  In lazy mode the batch's rows are combined as the walk reaches them.
template <int ES>
__device__ void flow_fin_seq(const FlowArgs &F, int b, int j0, int kind, int cum) {
    const AcceptArgs &a = F.acc;
    const int lane = threadIdx.x & 31;
    const int K = a.K, ns = F.st.n_split;
    const float T = a.temperature[b];
    const int tok_l = lane < K ? a.tokens[(size_t)b * K + lane] : -1;
    const double u_l = lane <= K ? a.uniforms[(size_t)b * (K + 1) + lane] : 0.0;
    const bool greedy = (T == 0.0f);
    const bool all_read = !F.lazy;
    const bool fast = all_read && ns == 1 && K < 32;
    auto token = [&](int j) {
        const int v = __shfl_sync(0xFFFFFFFFu, tok_l, j & 31);
        return j < 32 ? v : a.tokens[(size_t)b * K + j];
    };
    auto outputs = [&](int k, int tstar) {
        int32_t *outs = a.out_tokens + (size_t)b * (K + 1);
        for (int j = lane; j <= K; j += 32)
            outs[j] = j < k ? (j < 32 ? tok_l : a.tokens[(size_t)b * K + j]) : (j == k ? tstar : -1);
        if (lane == 0) a.accept_len[b] = k;
    };
    auto row_t = [&](int j) { return a.tgt.base + ((long long)b * a.tgt.rows_per_seq + j) * a.tgt.pitch_bytes; };
    auto row_d = [&](int j) { return a.drf.base + ((long long)b * a.drf.rows_per_seq + j) * a.drf.pitch_bytes; };
    // a row's statistics (valid in lane 0): read when the consumers combined them, else combined
    // here from the chunks' partials; kept for the float-float tier and checked
    auto combine = [&](long long rid, int &bad) {
        RowStat r{};
        if (ns == 1) {
            if (lane == 0) r = a.rowstat[rid];
        } else {
            r = combine_row(a.part + (size_t)rid * ns * kWarps, ns * kWarps, greedy, T);
        }
        if (lane == 0) {
            if (ns != 1) a.rowstat[rid] = r;
            if (rowstat_bad(r, greedy)) {
                report_error(a.stats, SV_ERR_NONFINITE, (int)rid);
                bad = 1;
            }
        }
        return r;
    };
    // debug values of position j, written by the calling lane (rq, rp: its rows' statistics)
    auto debug_own = [&](int j, const RowStat &rq, const RowStat &rp) {
        if (!a.debug) return;
        if (greedy) {
            a.debug[((size_t)b * (K + 1) + j) * SV_DEBUG_FIELDS + SV_DBG_MASS_Q] = 1.0;
            if (j < K) a.debug[((size_t)b * (K + 1) + j) * SV_DEBUG_FIELDS + SV_DBG_MASS_P] = 1.0;
        } else {
            flow_debug<ES>(a, b, j, T, rq, j < K ? &rp : nullptr);
        }
    };
    // every row of positions j_from..j_to, combined one after another
    auto combine_range = [&](int j_from, int j_to, int &bad) {
        for (int jj = j_from; jj <= j_to; ++jj) {
            const RowStat rq = combine((long long)b * (K + 1) + jj, bad);
            RowStat rp{};
            if (!greedy && jj < K) rp = combine(F.st.n_rows0 + (long long)b * K + jj, bad);
            if (lane == 0) debug_own(jj, rq, rp);
        }
    };
    int bad = 0;
    const int j_last = kind == kBatchOne ? j0 : K;   // rows of positions j0..j_last were read
    if (lane == 0) {
        const int n_d = greedy ? 0 : max(0, min(j_last, K - 1) - j0 + 1);
        stats_add(a.stats, &a.stats->rows, j_last - j0 + 1 + n_d);
    }
    // lane j's position: its rows' statistics and its drafted token's two logits (fast path)
    RowStat rq_l{}, rp_l{};
    float xt_l = 0.f, xd_l = 0.f;
    if (fast) {
        const int j = lane;
        int badl = 0;
        if (j <= K) {
            const long long rid_q = (long long)b * (K + 1) + j, rid_p = F.st.n_rows0 + (long long)b * K + j;
            rq_l = a.rowstat[rid_q];
            if (!greedy && j < K) {
                rp_l = a.rowstat[rid_p];
                xt_l = load_elem<ES>(row_t(j), tok_l);
                xd_l = load_elem<ES>(row_d(j), tok_l);
            }
            if (rowstat_bad(rq_l, greedy)) {
                report_error(a.stats, SV_ERR_NONFINITE, (int)rid_q);
                badl = 1;
            }
            if (!greedy && j < K && rowstat_bad(rp_l, greedy)) {
                report_error(a.stats, SV_ERR_NONFINITE, (int)rid_p);
                badl = 1;
            }
        }
        bad = __any_sync(0xFFFFFFFFu, badl);
        if (bad) {
            outputs(0, -1);
            if (lane == 0) flow_done(F);
            return;
        }
        if (j <= K) debug_own(j, rq_l, rp_l);
    } else if (kind == kBatchComplete || all_read) {
        combine_range(j0, K, bad);
        bad = __shfl_sync(0xFFFFFFFFu, bad, 0);
        if (bad) {
            outputs(0, -1);
            if (lane == 0) flow_done(F);
            return;
        }
        if (kind == kBatchComplete) {
            if (lane == 0) flow_to_exact(F, -1, b);
            return;
        }
    }
    float c_hi = 0.f, c_lo = 0.f;
    if (!greedy) log2e_over(T, c_hi, c_lo);
    for (int j = j0; j <= j_last; ++j) {
        const long long rid_q = (long long)b * (K + 1) + j, rid_p = F.st.n_rows0 + (long long)b * K + j;
        const bool with_p = !greedy && j < K;
        const int s = j < K ? token(j) : -1;   // every lane: token() shuffles
        RowStat rq{}, rp{};
        float xt = 0.f, xd = 0.f;
        if (fast) {
            rq = shfl_rowstat(rq_l, j);
            rp = shfl_rowstat(rp_l, j);
            xt = __shfl_sync(0xFFFFFFFFu, xt_l, j);
            xd = __shfl_sync(0xFFFFFFFFu, xd_l, j);
        } else {
            if (all_read) {
                if (lane == 0) {
                    rq = a.rowstat[rid_q];
                    if (with_p) rp = a.rowstat[rid_p];
                }
            } else {
                rq = combine(rid_q, bad);
                if (with_p) rp = combine(rid_p, bad);
                if (lane == 0) debug_own(j, rq, rp);
            }
            if (with_p && lane == 0) {
                xt = load_elem<ES>(row_t(j), s);
                xd = load_elem<ES>(row_d(j), s);
            }
        }
        const double u_j = __shfl_sync(0xFFFFFFFFu, u_l, j & 31);
        // lane 0 decides: 0 finished (k, tstar), 1 accepted, 2 float-float tier, 3 a draw is queued
        int verdict = 0, k = 0, tstar = -1;
        if (lane == 0) {
            if (bad) {
                k = 0;
            } else if (greedy) {
                if (j < K && s == rq.argmax) {
                    verdict = 1;
                } else {
                    k = j;
                    tstar = rq.argmax;
                }
            } else if (with_p) {
                const AcceptOutcome o = accept_test_x(a, b, j, s, j < 32 ? u_j : a.uniforms[(size_t)b * (K + 1) + j],
                                                      c_hi, c_lo, rq, rp, xt, xd);
                stats_add(a.stats, &a.stats->accept_tests, 1);
                if (o.near) stats_add(a.stats, &a.stats->near_boundary, 1);
                if (o.amb) {
                    verdict = 2;
                    k = j;
                } else if (o.acc) {
                    verdict = 1;
                } else {
                    k = j;
                    verdict = 3;
                }
            } else {
                k = K;
                verdict = 3;   // all K accepted: bonus draw from row K
            }
        }
        verdict = __shfl_sync(0xFFFFFFFFu, verdict, 0);
        k = __shfl_sync(0xFFFFFFFFu, k, 0);
        tstar = __shfl_sync(0xFFFFFFFFu, tstar, 0);
        bad = __shfl_sync(0xFFFFFFFFu, bad, 0);
        if (verdict == 0 || verdict == 3) {
            outputs(k, tstar);   // tstar = -1 for a draw: the finish writes it
            __syncwarp();
            if (lane == 0) {
                if (verdict == 3) flow_draw<ES>(F, b, k, T, rq, rp);
                else flow_done(F);
            }
            return;
        }
        if (verdict == 2) {
            outputs(k, -1);   // placeholders; the float-float tier writes the final outputs
            if (j_last > j && !all_read) combine_range(j + 1, j_last, bad);   // the rest of this batch is read
            if (j_last > j || j + 1 > K) {
                __syncwarp();
                if (lane == 0) flow_to_exact(F, -1, b);
            } else if (lane == 0) {
                flow_enqueue_rows(F, b, j + 1, K, !greedy, kBatchComplete, cum, false);
            }
            return;
        }
        // accepted: the next position is in this batch, or queue it (alone, or with the tail)
        if (j == j_last) {
            if (lane == 0) {
                const int jn = j + 1;
                if (jn >= kLazyTail) flow_enqueue_rows(F, b, jn, K, !greedy && jn < K, kBatchTail, cum, false);
                else flow_enqueue_rows(F, b, jn, jn, !greedy && jn < K, kBatchOne, cum, false);
            }
            return;
        }
    }
}

// A draw's sub-chunk sums are complete: t* with a certified margin (one warp).  The sums are
// scanned in float-float, 16 sub-chunks per lane; the sub-chunk holding u R is rescanned token
// by token exactly as the draw units weighed it; t* stands if u R is farther than the proven
// error bound from both its boundaries, else the draw goes to the float-float tier.
template <int ES>
__device__ void flow_finish(const FlowArgs &F, int d) {
    constexpr int EPV = 16 / ES;
    const AcceptArgs &a = F.acc;
    const int lane = threadIdx.x & 31;
    const DrawItem it = a.draws[d];
    const float *subs = F.subs + (size_t)d * F.n_sub;
    const int n_sub = F.n_sub, n_vsub = n_sub - 1;
    const int per = (n_sub + 31) / 32;
    const int s0 = min(lane * per, n_sub), s1 = min(s0 + per, n_sub);
    ff wsum = {0.f, 0.f};
    int last_pos = -1;
    for (int sb = s0; sb < s1; sb += 8) {   // eight loads in flight, then their sums
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = sb + e < s1 ? subs[sb + e] : 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if (sb + e < s1) {
                wsum = ff_add_f(wsum, v[e]);
                if (v[e] > 0.f) last_pos = sb + e;
            }
        }
    }
    ff incl = wsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float h = __shfl_up_sync(0xFFFFFFFFu, incl.hi, o);
        const float l = __shfl_up_sync(0xFFFFFFFFu, incl.lo, o);
        if (lane >= o) incl = ff_add(incl, {h, l});
    }
    ff excl = {__shfl_up_sync(0xFFFFFFFFu, incl.hi, 1), __shfl_up_sync(0xFFFFFFFFu, incl.lo, 1)};
    if (lane == 0) excl = {0.f, 0.f};
    const ff R = {__shfl_sync(0xFFFFFFFFu, incl.hi, 31), __shfl_sync(0xFFFFFFFFu, incl.lo, 31)};
    const int last_sub = warp_max_i(last_pos);
    float u_hi = 0.f, u_lo = 0.f;
    if (lane == 0) {
        u_hi = __double2float_rn(it.u);
        u_lo = __double2float_rn(it.u - (double)u_hi);
    }
    u_hi = __shfl_sync(0xFFFFFFFFu, u_hi, 0);
    u_lo = __shfl_sync(0xFFFFFFFFu, u_lo, 0);
    const ff thr = ff_mul(R, {u_hi, u_lo});
    // the lane whose range holds thr finds the sub-chunk
    int found = -1;
    ff pre = excl;
    if (wsum.hi > 0.f && ff_diff(thr, excl) >= 0.f && ff_diff(thr, incl) < 0.f) {
        ff run = excl;
        bool done = false;
        for (int sb = s0; sb < s1 && !done; sb += 8) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = sb + e < s1 ? subs[sb + e] : 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (!done && sb + e < s1) {
                    const ff nx = ff_add_f(run, v[e]);
                    if (v[e] > 0.f) {
                        found = sb + e;
                        pre = run;
                        if (ff_diff(thr, nx) < 0.f) done = true;
                    }
                    run = nx;
                }
            }
        }
    }
    const unsigned fm = __ballot_sync(0xFFFFFFFFu, found >= 0);
    int sub;
    bool ambiguous = false;
    if (fm) {
        const int src = __ffs(fm) - 1;
        sub = __shfl_sync(0xFFFFFFFFu, found, src);
        pre = {__shfl_sync(0xFFFFFFFFu, pre.hi, src), __shfl_sync(0xFFFFFFFFu, pre.lo, src)};
    } else {
        // thr at or beyond the last boundary (rounding) or R == 0: the last positive sub-chunk
        sub = last_sub;
        ambiguous = true;
        ff p = {0.f, 0.f};
        for (int s = lane; s < max(sub, 0); s += 32) p = ff_add_f(p, subs[s]);
        pre = warp_sum_ff(p);
    }
    if (sub < 0) {
        // every weight is zero: degenerate; the float-float tier decides
        if (lane == 0) {
            *it.out = -1;
            stats_add(a.stats, &a.stats->draws, 1);
            flow_to_exact(F, d, it.seq);
        }
        return;
    }
    // rescan the sub-chunk token by token (same arithmetic as the draw units)
    float wv[EPV];
    int ntok = 0, tok0 = 0;
    if (sub < n_vsub) {
        const int vi = sub * 32 + lane;
        tok0 = vi * EPV;
        if (vi < F.n_vec) {
            ntok = EPV;
            const uint4 q = __ldg(reinterpret_cast<const uint4 *>(it.q.row) + vi);
            const uint4 p = it.has_p ? __ldg(reinterpret_cast<const uint4 *>(it.p.row) + vi) : q;
            if (it.has_p) vec_weights<ES, true, false>(it, q, p, tok0, wv);
            else vec_weights<ES, false, false>(it, q, p, tok0, wv);
        }
    } else {
        tok0 = F.n_vec * EPV + lane;
        if (tok0 < a.V) {
            ntok = 1;
            wv[0] = draw_scalar<ES>(it, tok0);
        }
    }
    ff lt = {0.f, 0.f};
#pragma unroll
    for (int i = 0; i < EPV; ++i)
        if (i < ntok) lt = ff_add_f(lt, wv[i]);
    ff inc = lt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float h = __shfl_up_sync(0xFFFFFFFFu, inc.hi, o);
        const float l = __shfl_up_sync(0xFFFFFFFFu, inc.lo, o);
        if (lane >= o) inc = ff_add(inc, {h, l});
    }
    ff run = ff_add(pre, ff_sub(inc, lt));
    int hit = -1;
    ff c_prev = run, c_hit = run;
#pragma unroll
    for (int i = 0; i < EPV; ++i) {
        if (i < ntok) {
            const ff nxt = ff_add_f(run, wv[i]);
            if (hit < 0 && wv[i] > 0.f && ff_diff(thr, nxt) < 0.f) {
                hit = i;
                c_prev = run;
                c_hit = nxt;
            }
            run = nxt;
        }
    }
    const unsigned m = __ballot_sync(0xFFFFFFFFu, hit >= 0);
    int tstar;
    float dprev, dhit;
    if (m != 0) {
        const int src = __ffs(m) - 1;
        const int tok = tok0 + (ntok == 1 ? 0 : hit);
        tstar = __shfl_sync(0xFFFFFFFFu, tok, src);
        dprev = __shfl_sync(0xFFFFFFFFu, ff_diff(thr, c_prev), src);
        dhit = __shfl_sync(0xFFFFFFFFu, ff_diff(c_hit, thr), src);
    } else {
        int lastpos = -1;
#pragma unroll
        for (int i = 0; i < EPV; ++i)
            if (i < ntok && wv[i] > 0.f) lastpos = i;
        const unsigned mm = __ballot_sync(0xFFFFFFFFu, lastpos >= 0);
        const int src = mm ? 31 - __clz(mm) : 0;
        const int tok = tok0 + (ntok == 1 ? 0 : max(lastpos, 0));
        tstar = __shfl_sync(0xFFFFFFFFu, tok, src);
        dprev = dhit = 0.f;
        ambiguous = true;
    }
    if (lane == 0) {
        const float A = it.q.ay + (it.has_p ? it.p.ay : 0.f);
        const float E = draw_error_bound(it, R.hi, A, fmaxf(thr.hi + dhit, 0.f) + thr.hi);
        if (dprev <= E || dhit <= E) ambiguous = true;
        const bool near = dprev < 1e-6f * R.hi || dhit < 1e-6f * R.hi;
        *it.out = tstar;
        if (it.dbg_r) *it.dbg_r = (double)R.hi + (double)R.lo;
        stats_add(a.stats, &a.stats->draws, 1);
        if (near) stats_add(a.stats, &a.stats->near_boundary, 1);
        if (ambiguous) flow_to_exact(F, d, it.seq);
        else flow_done(F);
    }
}

// Row `slot` (0..K target, K+1..2K draft) of sequence b for the float-float tier.
__device__ __forceinline__ ExactRow flow_row(const FlowArgs &F, int b, int slot) {
    const AcceptArgs &a = F.acc;
    const int K = a.K;
    ExactRow e;
    const bool is_t = slot <= K;
    const int j = is_t ? slot : slot - K - 1;
    const long long rid = is_t ? (long long)b * (K + 1) + j : F.st.n_rows0 + (long long)b * K + j;
    const RowSet &rs = is_t ? a.tgt : a.drf;
    e.row = rs.base + ((long long)b * rs.rows_per_seq + j) * rs.pitch_bytes;
    log2e_over(a.temperature[b], e.c.hi, e.c.lo);
    e.rf = (float)a.rowstat[rid].r;
    e.cut_x = -INFINITY;
    e.cut_id = 0x7FFFFFFF;
    e.top_x = INFINITY;
    e.top_id = -1;
    e.sc = 1.0f;
    e.valid = 1;
    e.filt = 0;
    return e;
}

// An uncertified sequence's exact row sums are complete: its accept tests in float64 from them,
// then its draw (one warp; the float64 work runs on lane 0).
template <int ES>
__device__ void flow_exact_b(const FlowArgs &F, int i) {
    const AcceptArgs &a = F.acc;
    const int lane = threadIdx.x & 31;
    const int b = a.exact[i].seq, K = a.K;
    const double cc = 1.4426950408889634074 / (double)a.temperature[b];
    auto sum = [&](int slot) {
        double s = 0.0;
        const double *p = F.xsum + ((size_t)i * F.max_slots + slot) * kFlowSplitA * kWarps;
        for (int t = lane; t < kFlowSplitA * kWarps; t += 32) s += p[t];
        return warp_sum_d(s);
    };
    int k = K, unresolved = 0;
    for (int j = 0; j < K; ++j) {
        const double sq = sum(j), sp = sum(K + 1 + j);
        const ExactRow rt = flow_row(F, b, j), rd = flow_row(F, b, K + 1 + j);
        const int s = a.tokens[(size_t)b * K + j];
        const float xt = load_elem<ES>(rt.row, s), xdr = load_elem<ES>(rd.row, s);
        const double lq = xt == -INFINITY ? -INFINITY : (double)xt * cc - (double)rt.rf - log2(sq);
        const double lp = xdr == -INFINITY ? -INFINITY : (double)xdr * cc - (double)rd.rf - log2(sp);
        const double ratio = (lp == -INFINITY) ? (lq == -INFINITY ? 0.0 : INFINITY) : exp2(lq - lp);
        const double r = fmin(1.0, ratio);
        const double uj = a.uniforms[(size_t)b * (K + 1) + j];
        if (fabs(uj - r) < 1e-12) unresolved = 1;
        if (a.debug && lane == 0) {
            double *dbg = a.debug + ((size_t)b * (K + 1) + j) * SV_DEBUG_FIELDS;
            dbg[SV_DBG_LSE_Q] = ((double)rt.rf + log2(sq)) * kLn2;
            dbg[SV_DBG_LSE_P] = ((double)rd.rf + log2(sp)) * kLn2;
            dbg[SV_DBG_Q_S] = exp2(lq);
            dbg[SV_DBG_P_S] = exp2(lp);
            dbg[SV_DBG_RATIO] = ratio;
            dbg[SV_DBG_MASS_Q] = 1.0;
            dbg[SV_DBG_MASS_P] = 1.0;
        }
        if (!(uj < r)) {
            k = j;
            break;
        }
    }
    const double sqk = sum(k);
    double spk = 0.0;
    const bool has_p = k < K && !a.draw_from_q;
    if (has_p) spk = sum(K + 1 + k);
    if (lane == 0) {
        if (unresolved) stats_add(a.stats, &a.stats->unresolved, 1);
        a.accept_len[b] = k;
        for (int j = 0; j <= K; ++j) a.out_tokens[(size_t)b * (K + 1) + j] = j < k ? a.tokens[(size_t)b * K + j] : -1;
        ExactDraw xd;
        xd.q = flow_row(F, b, k);
        xd.inv_q = (float)(1.0 / sqk);
        xd.has_p = has_p;
        xd.p = xd.q;
        xd.inv_p = 0.f;
        if (has_p) {
            xd.p = flow_row(F, b, K + 1 + k);
            xd.inv_p = (float)(1.0 / spk);
        }
        xd.sign_tol = (float)(8.0 * kU32);
        xd.u = a.uniforms[(size_t)b * (K + 1) + K];
        xd.out = a.out_tokens + (size_t)b * (K + 1) + k;
        xd.dbg_r = a.debug ? a.debug + (size_t)b * (K + 1) * SV_DEBUG_FIELDS + SV_DBG_R : nullptr;
        F.xdraw[i] = xd;
        flow_enqueue(F, kUnitExactC, (long long)i * F.x_groups, F.x_groups);
    }
}

__device__ __forceinline__ ExactDraw flow_item_draw(const FlowArgs &F, int i) {
    const ExactItem itm = F.acc.exact[i];
    return itm.draw >= 0 ? exact_draw_from(F.acc.draws[itm.draw]) : F.xdraw[i];
}

// An item's float-float row pass is complete: exact normalisers, the exact residuals of the
// tokens of uncertain sign, a float-float scan of the sub-chunk masses, the sub-chunk holding
// u R rescanned token by token, t* (one warp; float-float throughout).
template <int ES>
__device__ void flow_exact_d(const FlowArgs &F, int i, const float2 *tab) {
    const AcceptArgs &a = F.acc;
    const int lane = threadIdx.x & 31;
    const ExactDraw d = flow_item_draw(F, i);
    const float4 *xs = F.xsubs + (size_t)i * F.n_sub;
    const float4 *xn = F.xnorm + (size_t)i * F.n_sub;
    const int n_sub = F.n_sub, n_vsub = n_sub - 1, n_vec = F.n_vec;
    ff sq = {0.f, 0.f}, sp = {0.f, 0.f};
    for (int s8 = lane; s8 < n_sub; s8 += 8 * 32) {   // eight loads in flight, then their sums
        float4 v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = s8 + e * 32 < n_sub ? xn[s8 + e * 32] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            sq = ff_add(sq, {v[e].x, v[e].y});
            sp = ff_add(sp, {v[e].z, v[e].w});
        }
    }
    sq = warp_sum_ff(sq);
    sp = warp_sum_ff(sp);
    const ff iq = ff_recip(sq), ip = d.has_p ? ff_recip(sp) : ff{0.f, 0.f};
    // exact residuals of the tokens whose sign the float32 test could not settle
    const int n_unc_all = a.exact_unc[i];
    const int n_unc = min(n_unc_all, kFlowUncCap);
    if (lane == 0 && n_unc_all > kFlowUncCap) stats_add(a.stats, &a.stats->unresolved, 1);
    const int *unc = F.xunc + (size_t)i * kExactUncCap;
    float2 *uncw = F.xuncw + (size_t)i * kFlowUncCap;
    for (int k = lane; k < n_unc; k += 32) {
        const int t = unc[k];
        const float xq = load_elem<ES>(d.q.row, t), xp = load_elem<ES>(d.p.row, t);
        const ff w = ff_sub(ff_mul(exact_w(d.q, xq, t, tab), iq), ff_mul(exact_w(d.p, xp, t, tab), ip));
        uncw[k] = w.hi > 0.f ? make_float2(w.hi, w.lo) : make_float2(0.f, 0.f);
    }
    __syncwarp();
    __threadfence_block();
    // W(s) = A_q(s) / S_q - A_p(s) / S_p (+ the exact residuals of its uncertain tokens) for the
    // lane's own sub-chunks, written over the item's sums in place (read back below), so that the
    // uncertain list is walked once per lane
    float4 *xw = F.xsubs + (size_t)i * F.n_sub;
    const int per = (n_sub + 31) / 32;
    const int s0 = min(lane * per, n_sub), s1 = min(s0 + per, n_sub);
    for (int sb = s0; sb < s1; sb += 4) {
        float4 v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = sb + e < s1 ? xs[sb + e] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (sb + e < s1) {
                const ff w = ff_sub(ff_mul({v[e].x, v[e].y}, iq), ff_mul({v[e].z, v[e].w}, ip));
                xw[sb + e] = make_float4(w.hi, w.lo, 0.f, 0.f);
            }
        }
    }
    for (int k = 0; k < n_unc; ++k) {
        const int t = unc[k];
        const int ts = t < n_vec * (16 / ES) ? t / (32 * (16 / ES)) : n_vsub;
        if (ts >= s0 && ts < s1) {
            const float4 v = xw[ts];
            const ff w = ff_add({v.x, v.y}, {uncw[k].x, uncw[k].y});
            xw[ts] = make_float4(w.hi, w.lo, 0.f, 0.f);
        }
    }
    __syncwarp();
    __threadfence_block();   // the fallback below reads other lanes' sub-chunks
    auto W = [&](int s) {
        const float4 v = xw[s];
        return ff{v.x, v.y};
    };
    ff mine = {0.f, 0.f};
    int last_pos = -1;
    for (int sb = s0; sb < s1; sb += 4) {
        ff v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = sb + e < s1 ? W(sb + e) : ff{0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (sb + e < s1) {
                mine = ff_add(mine, v[e]);
                if (v[e].hi > 0.f) last_pos = sb + e;
            }
        }
    }
    ff incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float h = __shfl_up_sync(0xFFFFFFFFu, incl.hi, o);
        const float l = __shfl_up_sync(0xFFFFFFFFu, incl.lo, o);
        if (lane >= o) incl = ff_add(incl, {h, l});
    }
    ff excl = {__shfl_up_sync(0xFFFFFFFFu, incl.hi, 1), __shfl_up_sync(0xFFFFFFFFu, incl.lo, 1)};
    if (lane == 0) excl = {0.f, 0.f};
    const ff R = {__shfl_sync(0xFFFFFFFFu, incl.hi, 31), __shfl_sync(0xFFFFFFFFu, incl.lo, 31)};
    const int last_sub = warp_max_i(last_pos);
    float u_hi = 0.f, u_lo = 0.f;
    if (lane == 0) {
        u_hi = __double2float_rn(d.u);
        u_lo = __double2float_rn(d.u - (double)u_hi);
    }
    u_hi = __shfl_sync(0xFFFFFFFFu, u_hi, 0);
    u_lo = __shfl_sync(0xFFFFFFFFu, u_lo, 0);
    const ff thr = ff_mul(R, {u_hi, u_lo});
    int found = -1;
    ff pre = excl;
    if (mine.hi > 0.f && ff_diff(thr, excl) >= 0.f && ff_diff(thr, incl) < 0.f) {
        ff run = excl;
        bool done = false;
        for (int sb = s0; sb < s1 && !done; sb += 4) {
            ff v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = sb + e < s1 ? W(sb + e) : ff{0.f, 0.f};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (!done && sb + e < s1) {
                    const ff nx = ff_add(run, v[e]);
                    if (v[e].hi > 0.f && ff_diff(thr, nx) < 0.f) {
                        found = sb + e;
                        pre = run;
                        done = true;
                    }
                    run = nx;
                }
            }
        }
    }
    const unsigned fm = __ballot_sync(0xFFFFFFFFu, found >= 0);
    int sub;
    if (fm) {
        const int src = __ffs(fm) - 1;
        sub = __shfl_sync(0xFFFFFFFFu, found, src);
        pre = {__shfl_sync(0xFFFFFFFFu, pre.hi, src), __shfl_sync(0xFFFFFFFFu, pre.lo, src)};
    } else {
        // u R at or past the last boundary through rounding: the last positive sub-chunk
        sub = last_sub;
        ff p = {0.f, 0.f};
        for (int s = lane; s < max(sub, 0); s += 32) p = ff_add(p, W(s));
        pre = warp_sum_ff(p);
    }
    int tstar = -1;
    bool unres = false;
    if (sub >= 0) {
        // rescan the sub-chunk: (32 x tokens per vector) tokens, 16 / ES per lane, float-float scan
        constexpr int EPV = 16 / ES;
        const int t0 = sub < n_vsub ? sub * 32 * EPV : n_vec * EPV;
        const int ntok = sub < n_vsub ? min(32 * EPV, (n_vec - sub * 32) * EPV) : a.V - n_vec * EPV;
        ff wt[EPV];
        float xq[EPV], xp[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e) {   // the lane's logits first, all loads in flight
            const int idx = lane * EPV + e;   // lane-major: the lane's tokens are consecutive
            xq[e] = idx < ntok ? load_elem<ES>(d.q.row, t0 + idx) : -INFINITY;
            xp[e] = (idx < ntok && d.has_p) ? load_elem<ES>(d.p.row, t0 + idx) : -INFINITY;
        }
        ff lt = {0.f, 0.f};
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            const int idx = lane * EPV + e;
            wt[e] = {0.f, 0.f};
            if (idx < ntok) {
                const int t = t0 + idx;
                const ff q = ff_mul(exact_w(d.q, xq[e], t, tab), iq);
                if (d.has_p) {
                    const ff w = ff_sub(q, ff_mul(exact_w(d.p, xp[e], t, tab), ip));
                    wt[e] = w.hi > 0.f ? w : ff{0.f, 0.f};
                } else {
                    wt[e] = q;
                }
            }
            lt = ff_add(lt, wt[e]);
        }
        ff inc = lt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float h = __shfl_up_sync(0xFFFFFFFFu, inc.hi, o);
            const float l = __shfl_up_sync(0xFFFFFFFFu, inc.lo, o);
            if (lane >= o) inc = ff_add(inc, {h, l});
        }
        ff run = ff_add(pre, ff_sub(inc, lt));
        int hit = -1, lastp = -1;
        ff c_prev = run, c_hit = run;
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            const ff nxt = ff_add(run, wt[e]);
            if (wt[e].hi > 0.f) {
                lastp = e;
                if (hit < 0 && ff_diff(thr, nxt) < 0.f) {
                    hit = e;
                    c_prev = run;
                    c_hit = nxt;
                }
            }
            run = nxt;
        }
        // float-float sums over ~V / 256 sub-chunks: worst-case relative error below 2e-11, plus
        // the exponents' low-word rounding, about 2^-48 |x c| <= 2^-48 (|r| + 126)
        const float tol = (2e-11f + 0x1p-46f * (fabsf(d.q.rf) + fabsf(d.p.rf) + 252.0f)) * R.hi;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, hit >= 0);
        if (m) {
            const int src = __ffs(m) - 1;
            tstar = __shfl_sync(0xFFFFFFFFu, t0 + src * EPV + hit, src);
            const bool close = ff_diff(thr, c_prev) < tol || ff_diff(c_hit, thr) < tol;
            unres = __shfl_sync(0xFFFFFFFFu, close, src);
        } else {
            // rounding left u R past the sub-chunk: its last positive token, unresolved
            const unsigned mm = __ballot_sync(0xFFFFFFFFu, lastp >= 0);
            const int src = mm ? 31 - __clz(mm) : 0;
            tstar = mm ? __shfl_sync(0xFFFFFFFFu, t0 + src * EPV + lastp, src) : -1;
            unres = true;
        }
    }
    if (lane == 0) {
        *d.out = tstar;
        if (unres) stats_add(a.stats, &a.stats->unresolved, 1);
        if (d.dbg_r) *d.dbg_r = (double)R.hi + (double)R.lo;
        flow_done(F);
    }
}

// ------------------------------------------------------------------------------------------
// Consumer warps: the float-float work units
// ------------------------------------------------------------------------------------------

// Exact C: sub-chunks g * 32 + warp, + 8, ... of item i: per sub-chunk the sums of the q- and
// p-weights of tokens whose residual q - p is certainly positive (a sign test with the float32
// normalisers and their bound), and the normaliser parts; tokens of uncertain sign are listed.
template <int ES>
__device__ void flow_exact_c(const FlowArgs &F, long long unit, const float2 *tab) {
    constexpr int EPV = 16 / ES;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int i = (int)(unit / F.x_groups), g = (int)(unit - (long long)i * F.x_groups);
    const ExactDraw d = flow_item_draw(F, i);
    const int n_vsub = F.n_sub - 1, n_vec = F.n_vec;
    float4 *xs = F.xsubs + (size_t)i * F.n_sub;
    float4 *xn = F.xnorm + (size_t)i * F.n_sub;
    for (int sb = g * kFlowGroupSubs + warp; sb < min((g + 1) * kFlowGroupSubs, F.n_sub); sb += kWarps) {
        ff nq = {0.f, 0.f}, np = {0.f, 0.f}, aq = {0.f, 0.f}, ap = {0.f, 0.f};
        auto token = [&](float xq, float xp, int v) {
            const ff eq = exact_w(d.q, xq, v, tab);
            nq = ff_add(nq, eq);
            if (!d.has_p) {
                aq = ff_add(aq, eq);
                return;
            }
            const ff ep = exact_w(d.p, xp, v, tab);
            np = ff_add(np, ep);
            const float wq = eq.hi * d.inv_q, wp = ep.hi * d.inv_p;
            const float diff = wq - wp, tol = d.sign_tol * (wq + wp);
            if (diff > tol) {
                aq = ff_add(aq, eq);
                ap = ff_add(ap, ep);
            } else if (diff >= -tol && wq > 0.f) {
                const int slot = atomicAdd(&F.acc.exact_unc[i], 1);
                if (slot < kFlowUncCap) F.xunc[(size_t)i * kExactUncCap + slot] = v;
            }
        };
        if (sb < n_vsub) {
            const int vi = sb * 32 + lane;
            if (vi < n_vec) {
                const uint4 wq = __ldg(reinterpret_cast<const uint4 *>(d.q.row) + vi);
                const uint4 wp = d.has_p ? __ldg(reinterpret_cast<const uint4 *>(d.p.row) + vi) : wq;
#pragma unroll 2
                for (int k = 0; k < EPV; ++k) token(elem_of<ES>(wq, k), elem_of<ES>(wp, k), vi * EPV + k);
            }
        } else {
            const int t = n_vec * EPV + lane;
            if (t < F.acc.V) {
                const float xq = load_elem<ES>(d.q.row, t);
                token(xq, d.has_p ? load_elem<ES>(d.p.row, t) : xq, t);
            }
        }
        aq = warp_sum_ff(aq);
        ap = warp_sum_ff(ap);
        nq = warp_sum_ff(nq);
        np = warp_sum_ff(np);
        if (lane == 0) {
            xs[sb] = make_float4(aq.hi, aq.lo, ap.hi, ap.lo);
            xn[sb] = make_float4(nq.hi, nq.lo, np.hi, np.lo);
        }
    }
}

// Exact A: the float-float sum S = sum_v 2^(x_v c - r) over a quarter of one row of item i's
// sequence; each consumer warp writes its own part.
template <int ES>
__device__ void flow_exact_a(const FlowArgs &F, long long unit, const float2 *tab) {
    constexpr int EPV = 16 / ES;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
    const long long per_item = (long long)F.max_slots * kFlowSplitA;
    const int i = (int)(unit / per_item);
    const int rem = (int)(unit - (long long)i * per_item);
    const int slot = rem / kFlowSplitA, c = rem - slot * kFlowSplitA;
    const ExactRow r = flow_row(F, F.acc.exact[i].seq, slot);
    const int n_vec = F.n_vec;
    const int cv = (n_vec + kFlowSplitA - 1) / kFlowSplitA;
    const int v0 = min(c * cv, n_vec), v1 = min(v0 + cv, n_vec);
    ff s = {0.f, 0.f};
    for (int vi = v0 + tid; vi < v1; vi += kThreads) {
        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(r.row) + vi);
#pragma unroll 1
        for (int k = 0; k < EPV; ++k) {
            const float x = elem_of<ES>(w, k);
            if (x != -INFINITY) s = ff_add(s, ff_exp2_xc(x, r.c, (int)r.rf, tab));
        }
    }
    if (c == kFlowSplitA - 1) {
        const int t = n_vec * EPV + tid;
        if (t < F.acc.V) {
            const float x = load_elem<ES>(r.row, t);
            if (x != -INFINITY) s = ff_add(s, ff_exp2_xc(x, r.c, (int)r.rf, tab));
        }
    }
    s = warp_sum_ff(s);
    if (lane == 0) F.xsum[(((size_t)i * F.max_slots + slot) * kFlowSplitA + c) * kWarps + warp] = ff_to_double(s);
}

// ------------------------------------------------------------------------------------------
// The kernel
// ------------------------------------------------------------------------------------------
template <int ES>
__global__ void __launch_bounds__(kFlowThreads, 2) k_flow(const FlowArgs F) {
    pdl_trigger();   // a dependent launch may be scheduled; it waits for this kernel
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kStatsStages;
    int *abort_flag = reinterpret_cast<int *>(smem + 2 * kStatsStages * 8);
    volatile int *ring_tail = abort_flag + 1;     // requests posted
    volatile int *ring_head = abort_flag + 2;     // requests taken by the finisher warp
    volatile int *cons_done = abort_flag + 3;     // consumer warps that left their loop
    TileMeta *meta = reinterpret_cast<TileMeta *>(smem + 2 * kStatsStages * 8 + 16);
    volatile int4 *ring = reinterpret_cast<volatile int4 *>(smem + kFlowOffRing);   // (x, type << 24 | y, z, slot + 1)
    WarpPartial *s_part = reinterpret_cast<WarpPartial *>(smem + kFlowOffPart);   // [stage][warp]
    int *s_part_cnt = reinterpret_cast<int *>(smem + kFlowOffPartCnt);             // [stage]
    float *t_cache = reinterpret_cast<float *>(smem + kFlowOffTCache);
    float2 *tab = reinterpret_cast<float2 *>(smem + kFlowOffTab);
    unsigned char *tiles = smem + kFlowCtlBytes;
    const StatsArgs &a = F.st;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        for (int s = 0; s < kStatsStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        *abort_flag = 0;
        *ring_tail = 0;
        *ring_head = 0;
        *cons_done = 0;
        for (int st = 0; st < kStatsStages; ++st) s_part_cnt[st] = 0;
        fence_barrier_init();
    }
    const int n_cache = min(kFlowTCache, F.n_seq);
    for (int i = tid; i < n_cache; i += blockDim.x) t_cache[i] = a.temperature[i];
    for (int i = tid; i < 256; i += blockDim.x) tab[i] = kExp2Table[i];
    if (tid < kFlowRing) {
        ring[tid].x = 0;
        ring[tid].y = 0;
        ring[tid].z = 0;
        ring[tid].w = 0;
    }
    __syncthreads();

    if (warp == kWarps + 1) {
        // ---------------- finisher ----------------
        int h = 0;
        long long t0 = clock64();   // start of the current idle wait
        unsigned ns = 64;
        while (true) {
            if (h < *ring_tail) {
                int4 r = make_int4(0, 0, 0, 0);
                bool ok = false;
                for (int spin = 0; spin < (1 << 22); ++spin) {   // the request's fields land just after its slot
                    volatile int4 *v = &ring[h % kFlowRing];
                    if (v->w == h + 1) {
                        __threadfence_block();
                        r = make_int4(v->x, v->y, v->z, v->w);
                        ok = true;
                        break;
                    }
                    __nanosleep(32);
                }
                __syncwarp();
                if (!ok) {
                    if (lane == 0 && atomicExch(abort_flag, 1) == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
                    break;
                }
                __threadfence();   // acquire: the data the request refers to was fenced before it was posted
                const int type = r.y >> 24, y = r.y & 0xFFFFFF;
                if (type == kReqSeq) flow_fin_seq<ES>(F, r.x, y >> 2, y & 3, r.z);
                else if (type == kReqFinish) flow_finish<ES>(F, r.x);
                else if (type == kReqExactB) flow_exact_b<ES>(F, r.x);
                else flow_exact_d<ES>(F, r.x, tab);
                __syncwarp();
                ++h;
                if (lane == 0) *ring_head = h;
                ns = 64;
                t0 = clock64();
            } else {
                const int done = *cons_done;
                __threadfence_block();
                if (done == kWarps && h == *ring_tail) break;
                if (*reinterpret_cast<volatile int *>(abort_flag) || clock64() - t0 > 4 * a.wait_limit) break;
                __nanosleep(ns);
                ns = ns < 512 ? 2 * ns : 512;
            }
        }
        return;
    }

    if (warp == kWarps) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t policy = policy_evict_first();
            long long in_flight[kStatsStages];
            for (int s = 0; s < kStatsStages; ++s) in_flight[s] = -1;
            long long it = 0;
            int st = 0;
            uint32_t epar = 0;
            bool ok = true;
            // Two queues, taken in order: the units the init kernel wrote (every sequence's
            // first rows), then the units appended during the pass (draws, float-float units,
            // lazy mode's later rows), so that the bandwidth-bound row statistics stream without
            // interruption.  Claims are plain atomic increments, which scale to every producer at
            // once.  A producer that drew an appended position past the tail keeps it as a
            // reservation and takes the unit as soon as its word is written; every position below
            // the head is reserved by exactly one producer, so no unit is left unclaimed.
            const int q0_n = *reinterpret_cast<volatile int *>(&F.fc->q0_tail.v);
            volatile int *q_tail_v = reinterpret_cast<volatile int *>(&F.fc->q_tail.v);
            volatile int *q_head1_v = reinterpret_cast<volatile int *>(&F.fc->q_head1.v);
            volatile int *q_head0_v = reinterpret_cast<volatile int *>(&F.fc->q_head.v);
            long long resv = -1;   // a reserved appended position, not yet written
            // 1: a word claimed, 0: nothing available now
            auto claim_word = [&](unsigned long long &wd) -> int {
                if (resv < 0 && *q_head0_v < q0_n) {
                    const int c = atomicAdd(&F.fc->q_head.v, 1);
                    if (c < q0_n) {
                        wd = ld_relaxed_u64(&F.units[c]);
                        return 1;
                    }
                }
                if (resv < 0 && *q_head1_v < *q_tail_v) resv = F.q1_base + atomicAdd(&F.fc->q_head1.v, 1);
                if (resv >= F.cap) resv = -1;   // cannot happen: the queue holds every unit of the call
                if (resv >= 0) {
                    wd = ld_relaxed_u64(&F.units[resv]);
                    if (wd >> 63) {
                        resv = -1;
                        return 1;
                    }
                }
                return 0;
            };
            // stage one: wait for the stage to be free, then describe it
            auto next_stage = [&]() -> bool {
                if (it >= kStatsStages) {
                    if (!mbar_wait_or_abort(&empty[st], epar, abort_flag, a.wait_limit)) {
                        if (atomicExch(abort_flag, 1) == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
                        return false;
                    }
                }
                in_flight[st] = -1;
                return true;
            };
            auto advance = [&]() {
                ++it;
                if (++st == kStatsStages) {
                    st = 0;
                    if (it >= 2 * kStatsStages) epar ^= 1u;   // round r >= 2 waits phase r - 1
                }
            };
            // The next unit is claimed while the current one's last stage waits for a free slot,
            // so the claim's round trips overlap the copies in flight.
            unsigned long long pf = 0;   // a claimed word not yet issued (bit 63 set), or 0
            auto prefetch = [&]() {
                if (pf >> 63) return;
                unsigned long long wd = 0;
                const int got = claim_word(wd);
                if (got > 0) pf = wd;
            };
            while (ok) {
                long long unit = -1;
                unsigned payload = 0;
                int type = 0;
                unsigned long long word = 0;
                unsigned ns = 64;
                int spins = 0;
                const long long t_start = clock64();   // the wait is bounded by its own length
                while (true) {
                    if (pf >> 63) {
                        word = pf;
                        pf = 0;
                        break;
                    }
                    if (claim_word(word) > 0) break;
                    // nothing queued: has every sequence finished?  (read every few tries: every
                    // idle producer polls it; the sleeps grow so idle producers stay quiet)
                    if ((spins++ & 3) == 0 && ld_acquire(&F.fc->n_pending.v) == 0) break;
                    if (*reinterpret_cast<volatile int *>(abort_flag) || clock64() - t_start > a.wait_limit) {
                        if (atomicExch(abort_flag, 1) == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
                        ok = false;
                        break;
                    }
                    __nanosleep(ns);
                    ns = ns < 1024 ? 2 * ns : 1024;
                }
                if (ok && (word >> 63)) {
                    unit = (long long)(unsigned)(word & 0xFFFFFFFFu);
                    type = (int)((word >> 60) & 7u);
                    payload = (unsigned)((word >> 32) & 0x0FFFFFFFu);
                    if (type != kUnitStats) __threadfence();   // acquire: the unit's data was written before it
                }
                const bool have = ok && unit >= 0;
                if (!have) {
                    if (next_stage()) {
                        TileMeta m;
                        m.flags = kTileEnd;
                        meta[st] = m;
                        mbar_arrive(&full[st]);
                    }
                    break;
                }
                if (type == kUnitStats) {
                    const UnitInfo ui = stats_unit<ES>(a, unit, t_cache, n_cache);
                    const int nt = max(unit_tiles(ui), 1);
                    for (int t = 0; t < nt && ok; ++t) {
                        if (t == nt - 1) prefetch();
                        if (!ok || !next_stage()) {
                            ok = false;
                            break;
                        }
                        const int fv = ui.v0 + t * (kStatsTileBytes / 16);
                        const int nv = max(0, min(kStatsTileBytes / 16, ui.v1 - fv));
                        TileMeta m;
                        m.row = ui.row;
                        m.rid = ui.rid;
                        m.c_hi = ui.c_hi;
                        m.c_lo = ui.c_lo;
                        m.chunk = ui.chunk;
                        m.fv = fv;
                        m.nv = nv;
                        m.tail0 = ui.tail0;
                        m.n_tail = ui.n_tail;
                        m.flags = (t == 0 ? kTileFirst : 0) | (t == nt - 1 ? kTileLast : 0) | (ui.greedy ? kTileGreedy : 0);
                        m.aux = (int)payload;
                        meta[st] = m;
                        if (nv > 0) {
                            mbar_arrive_expect_tx(&full[st], (uint32_t)nv * 16u);
                            bulk_load_stream(tiles + st * kStatsTileBytes, ui.row + (size_t)fv * 16, (uint32_t)nv * 16u,
                                             &full[st], policy);
                            in_flight[st] = it;
                        } else {
                            mbar_arrive(&full[st]);
                        }
                        advance();
                    }
                } else if (type == kUnitDraw) {
                    const int d = (int)(unit / F.d_split), c = (int)(unit - (long long)d * F.d_split);
                    const DrawItem *item = F.acc.draws + d;
                    const char *qrow = item->q.row, *prow = item->p.row;
                    const bool has_p = item->has_p != 0;
                    const int n_vsub = F.n_sub - 1;
                    const int sb0 = min(c * kDrawUnitSubs, n_vsub), sb1 = min(sb0 + kDrawUnitSubs, n_vsub);
                    const int v0 = sb0 * 32, v1 = max(v0, min(sb1 * 32, F.n_vec));
                    constexpr int HV = kTileBytes / 16;   // vectors per half stage
                    const int nt = max((v1 - v0 + HV - 1) / HV, 1);
                    for (int t = 0; t < nt && ok; ++t) {
                        if (t == nt - 1) prefetch();
                        if (!ok || !next_stage()) {
                            ok = false;
                            break;
                        }
                        const int fv = v0 + t * HV;
                        const int nv = max(0, min(HV, v1 - fv));
                        TileMeta m;
                        m.rid = d;
                        m.chunk = c;
                        m.fv = fv;
                        m.nv = nv;
                        m.flags = kTileDraw | (t == nt - 1 ? kTileLast : 0);
                        m.aux = 0;
                        meta[st] = m;
                        if (nv > 0) {
                            const uint32_t bytes = (uint32_t)nv * 16u;
                            mbar_arrive_expect_tx(&full[st], has_p ? 2u * bytes : bytes);
                            bulk_load_stream(tiles + st * kStatsTileBytes, qrow + (size_t)fv * 16, bytes, &full[st], policy);
                            if (has_p)
                                bulk_load_stream(tiles + st * kStatsTileBytes + kTileBytes, prow + (size_t)fv * 16, bytes,
                                                 &full[st], policy);
                            in_flight[st] = it;
                        } else {
                            mbar_arrive(&full[st]);
                        }
                        advance();
                    }
                } else {
                    // a float-float unit: no copy, the consumers read the rows themselves
                    if (!next_stage()) {
                        ok = false;
                    } else {
                        TileMeta m;
                        m.rid = unit;
                        m.flags = type == kUnitExactC ? kTileExactC : kTileExactA;
                        m.nv = 0;
                        m.aux = 0;
                        meta[st] = m;
                        mbar_arrive(&full[st]);
                        advance();
                    }
                }
            }
            // after an abort, copies still in flight land before shared memory is released
            if (*reinterpret_cast<volatile int *>(abort_flag)) {
                for (int s = 0; s < kStatsStages; ++s)
                    if (in_flight[s] >= 0)
                        mbar_wait_bounded(&full[s], (uint32_t)((in_flight[s] / kStatsStages) & 1), a.wait_limit / 16);
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    // Post a request to this block's finisher warp (lane 0; bounded wait for ring space).
    auto post = [&](int type, int x, int y, int z) {
        __threadfence();
        const long long t0 = clock64();
        while (*ring_tail - *ring_head >= kFlowRing - kWarps) {
            if (*reinterpret_cast<volatile int *>(abort_flag) || clock64() - t0 > a.wait_limit) {
                if (atomicExch(abort_flag, 1) == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
                return;
            }
            __nanosleep(128);
        }
        const int slot = atomicAdd(reinterpret_cast<int *>(const_cast<int *>(ring_tail)), 1);
        volatile int4 *e = &ring[slot % kFlowRing];
        e->x = x;
        e->y = (type << 24) | y;
        e->z = z;
        __threadfence_block();
        e->w = slot + 1;
    };
    StatAcc A;
    acc_init(A);
    int st = 0;
    uint32_t par = 0;
    int cur_d = -1;
    DrawItem item;
    for (;;) {
        if (!mbar_wait_or_abort(&full[st], par, abort_flag, a.wait_limit)) {
            if (lane == 0 && atomicExch(abort_flag, 1) == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
            break;
        }
        const int flags = meta[st].flags;
        if (flags & kTileEnd) break;
        unsigned char *stage = tiles + st * kStatsTileBytes;
        if (flags & kTileDraw) {
            const int d = (int)meta[st].rid, c = meta[st].chunk, fv = meta[st].fv, nv = meta[st].nv;
            if (d != cur_d) {
                __threadfence();   // acquire: the item was written before its units were queued
                item = F.acc.draws[d];
                cur_d = d;
            }
            float *subs_item = F.subs + (size_t)d * F.n_sub;
            if (item.has_p) draw_tile<ES, true, false>(item, stage, stage + kTileBytes, fv, nv, subs_item);
            else draw_tile<ES, false, false>(item, stage, stage + kTileBytes, fv, nv, subs_item);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            if (flags & kTileLast) {
                if (c == F.d_split - 1 && warp == 0) {
                    // the scalar tail of the row forms the last sub-chunk
                    constexpr int EPV = 16 / ES;
                    const int t0 = F.n_vec * EPV;
                    const float w = t0 + lane < F.acc.V ? draw_scalar<ES>(item, t0 + lane) : 0.f;
                    const float W = warp_sum_f(w);
                    if (lane == 0) subs_item[F.n_sub - 1] = W;
                }
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    if (atomicAdd(&F.draw_cnt[d], 1) == F.d_split * kWarps - 1) {
                        __threadfence();
                        post(kReqFinish, d, 0, 0);
                    }
                }
                __syncwarp();
            }
        } else if (flags & (kTileExactC | kTileExactA)) {
            const long long unit = meta[st].rid;
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);   // no data in the stage: free it at once
            __threadfence();   // acquire: the item's draw was written before its units were queued
            if (flags & kTileExactC) {
                flow_exact_c<ES>(F, unit, tab);
                __syncwarp();
                if (lane == 0) {
                    const int i = (int)(unit / F.x_groups);
                    __threadfence();
                    if (atomicAdd(&F.x_cnt[i], 1) == F.x_groups * kWarps - 1) {
                        __threadfence();
                        post(kReqExactD, i, 0, 0);
                    }
                }
            } else {
                flow_exact_a<ES>(F, unit, tab);
                __syncwarp();
                if (lane == 0) {
                    const int i = (int)(unit / ((long long)F.max_slots * kFlowSplitA));
                    __threadfence();
                    if (atomicAdd(&F.a_cnt[i], 1) == (2 * F.acc.K + 1) * kFlowSplitA * kWarps - 1) {
                        __threadfence();
                        post(kReqExactB, i, 0, 0);
                    }
                }
            }
            __syncwarp();
        } else {
            const TileMeta m = meta[st];
            const bool greedy = (m.flags & kTileGreedy) != 0;
            if (m.flags & kTileFirst) acc_init(A);
            if (m.nv > 0) acc_tile<ES>(A, stage, m.nv, m.fv, greedy, m.c_hi);
            __syncwarp();
            if (m.flags & kTileLast) {
                if (tid < m.n_tail) {
                    const float x = load_elem<ES>(m.row, m.tail0 + tid);
                    acc_scalar(A, x, m.tail0 + tid, greedy, m.c_hi, m.c_lo);
                }
                // The eight warps' partials of the unit meet in shared memory; the last warp to
                // arrive stores all eight and makes them visible with one fence and one count, so
                // a unit costs one global fence, not eight.  The stage is released only after
                // this (its partial slots and count are reused by the stage's next unit).
                acc_store(A, greedy, s_part + st * kWarps + warp);
                __syncwarp();
                int last = 0;
                if (lane == 0) {
                    __threadfence_block();
                    last = atomicAdd(&s_part_cnt[st], 1) == kWarps - 1;
                }
                last = __shfl_sync(0xFFFFFFFFu, last, 0);
                if (last) {
                    __threadfence_block();
                    const uint4 *src = reinterpret_cast<const uint4 *>(s_part + st * kWarps);
                    uint4 *dst = reinterpret_cast<uint4 *>(a.part + ((size_t)m.rid * a.n_split + m.chunk) * kWarps);
                    static_assert(kWarps * sizeof(WarpPartial) == 16 * 16, "one 16-byte word per lane of half a warp");
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (lane < 16) v = src[lane];
                    __syncwarp();
                    // the stage's partial slots are read: free the stage before the fence, so that
                    // the fence's wait holds up this warp only, not the block's pipeline
                    if (lane == 0) {
                        s_part_cnt[st] = 0;
                        mbar_arrive(&empty[st]);
                    }
                    // the batch's last unit hands the sequence to the finisher
                    int b = 0, j = 0;
                    seq_pos(F, m.rid, b, j);
                    if (a.n_split == 1) {
                        // the unit is the whole row: its statistics are combined here, off the
                        // finisher's path (the partials are read from the registers of lanes 0-15)
                        __shared__ __align__(16) WarpPartial s_row[kWarps][kWarps];   // per warp: the 8 partials
                        if (lane < 16) reinterpret_cast<uint4 *>(s_row[warp])[lane] = v;
                        __syncwarp();
                        const float Tb = b < n_cache ? t_cache[b] : F.acc.temperature[b];
                        const RowStat r = combine_row(s_row[warp], kWarps, greedy, Tb);
                        if (lane == 0) F.acc.rowstat[m.rid] = r;
                    } else if (lane < 16) {
                        dst[lane] = v;
                    }
                    __syncwarp();
                    if (lane == 0) {
                        fence_acq_rel_gpu();
                        if (atomicAdd(&F.pos_cnt[b], kWarps) == (m.aux >> 8) - kWarps) {
                            fence_acq_rel_gpu();
                            post(kReqSeq, b, m.aux & 0xFF, m.aux >> 8);
                        }
                    }
                } else if (lane == 0) {
                    mbar_arrive(&empty[st]);
                }
                __syncwarp();
            } else if (lane == 0) {
                mbar_arrive(&empty[st]);
            }
        }
        if (++st == kStatsStages) {
            st = 0;
            par ^= 1u;
        }
    }
    __syncwarp();
    if (lane == 0) atomicAdd(reinterpret_cast<int *>(const_cast<int *>(cons_done)), 1);
}

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------
template <int ES>
static sv_status launch_flow(const VerifyPlan &pl, const AcceptArgs &acc_in, int B, int lazy, void *ws,
                             cudaStream_t stream) {
    DeviceInfo di;
    if (!device_info(di)) return SV_ERR_CUDA;
    char *w = static_cast<char *>(ws);
    Counters *counters = reinterpret_cast<Counters *>(w + pl.off_counters);
    FlowArgs F{};
    F.st.set[0] = acc_in.tgt;
    F.st.set[1] = acc_in.drf;
    F.st.n_sets = 2;
    F.st.V = acc_in.V;
    F.st.temperature = acc_in.temperature;
    F.st.n_split = pl.n_split;
    F.st.chunk_vecs = pl.chunk_vecs;
    F.st.n_rows0 = pl.n_rows0;
    F.st.n_units = (pl.n_rows0 + pl.n_rows1) * pl.n_split;
    F.st.part = reinterpret_cast<WarpPartial *>(w + pl.off_part);
    F.st.counters = counters;
    F.st.stats = acc_in.stats;
    F.st.wait_limit = kWaitLimitCycles;
    F.acc = acc_in;
    F.acc.part = F.st.part;
    F.acc.n_split = pl.n_split;
    F.acc.n_rows0 = pl.n_rows0;
    F.acc.rowstat = reinterpret_cast<RowStat *>(w + pl.off_rowstat);
    F.acc.nuc = nullptr;
    F.acc.top = nullptr;
    F.acc.draws = reinterpret_cast<DrawItem *>(w + pl.off_draws);
    F.acc.exact = reinterpret_cast<ExactItem *>(w + pl.off_exact);
    F.acc.exact_unc = reinterpret_cast<int *>(w + pl.off_xunc_n);
    F.acc.counters = counters;
    F.units = reinterpret_cast<unsigned long long *>(w + pl.off_lz_units);
    F.cap = pl.lz_cap;
    F.q1_base = pl.n_flow_initial;
    F.pos_cnt = reinterpret_cast<int *>(w + pl.off_lz_pos);
    F.n_seq = B;
    F.lazy = lazy;
    F.n_vec = pl.n_vec;
    F.n_sub = pl.n_sub;
    F.d_split = pl.d_split;
    F.subs = reinterpret_cast<float *>(w + pl.off_subs);
    F.draw_cnt = reinterpret_cast<int *>(w + pl.off_draw_cnt);
    F.x_cnt = reinterpret_cast<int *>(w + pl.off_xcnt);
    F.a_cnt = reinterpret_cast<int *>(w + pl.off_acnt);
    F.xsubs = reinterpret_cast<float4 *>(w + pl.off_xsubs);
    F.xnorm = reinterpret_cast<float4 *>(w + pl.off_xnorm);
    F.xunc = reinterpret_cast<int *>(w + pl.off_xunc);
    F.xuncw = reinterpret_cast<float2 *>(w + pl.off_xuncw);
    F.xsum = reinterpret_cast<double *>(w + pl.off_xpart);
    F.xdraw = reinterpret_cast<ExactDraw *>(w + pl.off_xdraw);
    F.cap_x = pl.cap_x;
    F.x_groups = pl.x_groups;
    F.max_slots = pl.max_slots;
    F.fc = reinterpret_cast<FlowCounters *>(w + pl.off_flow_ctr);
    if (cudaMemsetAsync(F.fc, 0, sizeof(FlowCounters), stream) != cudaSuccess) return SV_ERR_CUDA;
    {
        const long long clear = F.cap - F.q1_base;
        long long grid = div_up(B, kThreads);
        const long long want = (clear + kThreads * 16LL - 1) / (kThreads * 16LL);
        if (grid < want) grid = want;
        if (grid > 4LL * di.sms) grid = 4LL * di.sms;
        if (grid < 1) grid = 1;
        k_flow_init<<<(unsigned)grid, kThreads, 0, stream>>>(F, B);
        if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    }
    const int occ = prepare_kernel((const void *)k_flow<ES>, kFlowThreads, kFlowSmemBytes);
    if (occ < 1) return SV_ERR_CUDA;
    // blocks wait for units that other blocks queue, so every block must be resident: a
    // cooperative launch guarantees it (or fails)
    static_assert(sizeof(FlowArgs) < 4096, "kernel parameter block");
    void *args[] = {&F};
    profile_begin(stream);
    const cudaError_t e = cudaLaunchCooperativeKernel((const void *)k_flow<ES>, dim3(di.sms * occ), dim3(kFlowThreads),
                                                      args, kFlowSmemBytes, stream);
    if (e != cudaSuccess) return SV_ERR_CUDA;
    profile_end(stream);
    return SV_OK;
}

sv_status flow_verify(const VerifyPlan &pl, const AcceptArgs &acc, int B, int lazy, void *ws, cudaStream_t stream) {
    if (pl.es == 4) return launch_flow<4>(pl, acc, B, lazy, ws, stream);
    return launch_flow<2>(pl, acc, B, lazy, ws, stream);
}

}  // namespace sv

using namespace sv;

extern "C" sv_status sv_verify_lazy(const void *target_logits, int64_t t_row_pitch, const void *draft_logits,
                                    int64_t d_row_pitch, int d_rows_per_seq, sv_dtype dtype,
                                    const int32_t *draft_tokens, const double *uniforms, int B, int K, int V,
                                    const float *temperature, const float *top_p, const int32_t *top_k,
                                    int saguaro_F, float saguaro_C,
                                    int32_t *accept_len, int32_t *out_tokens, double *debug, sv_stats *stats,
                                    void *workspace, size_t workspace_bytes, sv_stream_t stream) {
    return sv::verify_entry(target_logits, t_row_pitch, draft_logits, d_row_pitch, d_rows_per_seq, dtype, draft_tokens,
                            uniforms, B, K, V, temperature, top_p, top_k, saguaro_F, saguaro_C, 0, 1, accept_len,
                            out_tokens, debug, stats, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}
