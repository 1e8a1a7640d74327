// sv_lazy.cu — sv_verify_lazy: the verification of sv_verify, reading each sequence's rows
// position by position and stopping at its first rejection.
//
// ["Accelerating LLM Decoding with Speculative Sampling (2023)" notes, §3: after the first
//  rejection the draft tokens to its right are discarded, so their rows decide nothing]
//
// The statistics pass of sv_verify reads every candidate row; the accept tests then use only
// the rows up to the first rejection.  Here one persistent kernel does both in order: a
// queue holds (row, chunk) units; position 0 of every sequence is queued first; the
// consumer warp that completes the last unit of a position combines its rows, runs the
// accept test (or the greedy match) and either queues the next position or finishes the
// sequence (outputs, draw item).  The draws and the float-float tier then run as in
// sv_verify.  Outputs are those of sv_verify; debug fields of positions that were never read
// stay NaN and only rows that were read count in stats.rows.  Top-p and sigma_{F,C} need
// per-row selection passes between the statistics and the tests, so calls with either use
// the sv_verify pipeline.
#include <math.h>

#include "sv_accept.cuh"
#include "sv_draw.cuh"
#include "sv_exact.cuh"
#include "sv_host.h"
#include "sv_stats.cuh"

namespace sv {

struct LazyArgs {
    StatsArgs st;     // row sets, temperatures, partials, counters
    AcceptArgs acc;   // accept context (no nucleus cuts, no top-F sets)
    unsigned long long *units;   // [cap] queued units: bit 63 set once written, aux in bits 32..62,
                                 // unit (row * n_split + chunk) in bits 0..31; cleared per call
    int *pos_cnt;     // [B] consumer warps done with the sequence's batches so far (cumulative)
    long long cap;
    long long q1_base;   // units[0, q1_base): position 0, written before the pass;
                         // units[q1_base, cap): later batches, appended during it
    int n_seq;           // B
};

// Batches: one position (the usual case), the tail from kLazyTail on (every remaining position
// at once: deep positions are rare, and one batch instead of one per position shortens the
// serial chain), or the completing batch of a sequence handed to the float-float tier.
constexpr int kBatchOne = 0, kBatchTail = 1, kBatchComplete = 2;
constexpr int kLazyTail = 2;

__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Row id -> (sequence, position) in the candidate-row numbering of the statistics pass.
__device__ __forceinline__ void seq_pos(const LazyArgs &L, long long rid, int &b, int &j) {
    const int K = L.acc.K;
    if (rid < L.st.n_rows0) {
        b = (int)(rid / (K + 1));
        j = (int)(rid - (long long)b * (K + 1));
    } else {
        const long long r = rid - L.st.n_rows0;
        b = (int)(r / K);
        j = (int)(r - (long long)b * K);
    }
}

// Queue rows of sequence b: target rows j0..j1 and draft rows j0..min(j1, K-1) when `with_d`.
// One thread.  `kind` says how the finisher treats the batch (see lazy_finish); `cum` is the
// sequence's cumulative consumer-warp count so far.
__device__ void lazy_enqueue(const LazyArgs &L, int b, int j0, int j1, bool with_d, int kind, int cum) {
    const int K = L.acc.K, ns = L.st.n_split;
    const int n_t = j1 - j0 + 1;
    const int n_d = with_d ? max(0, min(j1, K - 1) - j0 + 1) : 0;
    const int n = (n_t + n_d) * ns;
    // aux: the sequence's cumulative count of consumer warps once this batch is done (its
    // counter is never reset), the batch's first position, its kind
    const int aux = ((cum + n * kWarps) << 8) | (j0 << 2) | kind;
    // one 64-bit store per unit carries the unit and its valid bit, so a reader needs no fence
    const unsigned long long tag = (1ull << 63) | ((unsigned long long)(unsigned)aux << 32);
    const bool first = j0 == 0 && kind != kBatchComplete;   // position 0, queued before the pass
    const long long base = first ? (long long)atomicAdd(&L.st.counters->q0_tail, n)
                                 : L.q1_base + atomicAdd(&L.st.counters->q_tail, n);
    if (base + n > (first ? L.q1_base : L.cap)) {   // cannot happen: each unit is queued once
        report_error(L.st.stats, SV_ERR_WORKSPACE, b);
        return;
    }
    int k = 0;
    for (int j = j0; j <= j1; ++j) {
        const long long rid = (long long)b * (K + 1) + j;
        for (int c = 0; c < ns; ++c) st_relaxed_u64(&L.units[base + k++], tag | (unsigned)(rid * ns + c));
    }
    for (int j = j0; j < j0 + n_d; ++j) {
        const long long rid = L.st.n_rows0 + (long long)b * K + j;
        for (int c = 0; c < ns; ++c) st_relaxed_u64(&L.units[base + k++], tag | (unsigned)(rid * ns + c));
    }
}

// Write a finished sequence's tokens: s_1..s_k, then `tstar` at k (-1 when a draw fills it), -1.
__device__ __forceinline__ void lazy_outputs(const AcceptArgs &a, int b, int k, int tstar) {
    const int K = a.K;
    int32_t *outs = a.out_tokens + (size_t)b * (K + 1);
    for (int j = 0; j <= K; ++j) outs[j] = j < k ? a.tokens[(size_t)b * K + j] : (j == k ? tstar : -1);
    a.accept_len[b] = k;
}

// Per sequence: validate, clear debug fields, queue position 0.
__global__ void __launch_bounds__(kThreads) k_lazy_init(const LazyArgs L, int B) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const AcceptArgs &a = L.acc;
    const int K = a.K;
    const float T = a.temperature[b];
    const bool greedy = (T == 0.0f);
    if (a.debug)
        for (int i = 0; i < (K + 1) * SV_DEBUG_FIELDS; ++i) a.debug[(size_t)b * (K + 1) * SV_DEBUG_FIELDS + i] = NAN;
    if (!(greedy || (T >= 1e-3f && T <= 1e3f))) {
        report_error(a.stats, SV_ERR_INVALID_ARG, b);
        lazy_outputs(a, b, 0, -1);
        return;
    }
    for (int j = 0; j < K; ++j) {
        const int s = a.tokens[(size_t)b * K + j];
        if (s < 0 || s >= a.V) {
            report_error(a.stats, SV_ERR_BAD_TOKEN, b);
            lazy_outputs(a, b, 0, -1);
            return;
        }
    }
    atomicAdd(&L.st.counters->n_pending, 1);
    if (kLazyTail <= 0) lazy_enqueue(L, b, 0, K, !greedy && K > 0, kBatchTail, 0);
    else lazy_enqueue(L, b, 0, 0, !greedy && K > 0, kBatchOne, 0);
}

// Draw item and outputs of a sampled sequence that accepted k tokens (k < K: residual at row k).
template <int ES>
__device__ void lazy_draw(const AcceptArgs &a, int b, int k, float T, const RowStat &rq, const RowStat &rp) {
    const int K = a.K;
    DrawItem it;
    const char *qrow = a.tgt.base + ((long long)b * a.tgt.rows_per_seq + k) * a.tgt.pitch_bytes;
    it.q = draw_row(qrow, T, rq, nullptr, nullptr, 1.0f);
    it.has_p = k < K;
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
    a.draws[atomicAdd(&a.counters->n_draws, 1)] = it;
}

// The finisher warp: the batch of rows (starting at position j0) of sequence b is complete.
// Latency matters here (a sequence's next batch waits for it): the loads it needs are issued
// together up front, both rows' partials are combined in one pass each, and outputs are
// written by all lanes.
template <int ES>
__device__ void lazy_finish(const LazyArgs &L, int b, int j0, int kind, int cum) {
    const AcceptArgs &a = L.acc;
    const int lane = threadIdx.x & 31;
    const int K = a.K, ns = L.st.n_split;
    const float T = a.temperature[b];
    const int tok_l = lane < K ? a.tokens[(size_t)b * K + lane] : -1;                // s_lane
    const double u_l = lane <= K ? a.uniforms[(size_t)b * (K + 1) + lane] : 0.0;    // u_lane
    const bool greedy = (T == 0.0f);
    auto token = [&](int j) {
        const int v = __shfl_sync(0xFFFFFFFFu, tok_l, j & 31);
        return j < 32 ? v : a.tokens[(size_t)b * K + j];
    };
    // s_1..s_k, then tstar (-1: a draw fills it), then -1; accept_len = k
    auto outputs = [&](int k, int tstar) {
        int32_t *outs = a.out_tokens + (size_t)b * (K + 1);
        for (int j = lane; j <= K; j += 32) outs[j] = j < k ? (j < 32 ? tok_l : a.tokens[(size_t)b * K + j]) : (j == k ? tstar : -1);
        if (lane == 0) a.accept_len[b] = k;
    };
    auto combine = [&](long long rid, int &bad) {
        const RowStat r = combine_row(a.part + (size_t)rid * ns * kWarps, ns * kWarps, greedy, T);
        if (lane == 0) {
            a.rowstat[rid] = r;
            if ((r.flags != 0) || (greedy ? !isfinite(r.maxv) : !rs_sampled_ok(r))) {
                report_error(a.stats, SV_ERR_NONFINITE, (int)rid);
                bad = 1;
            }
        }
        return r;
    };
    // statistics of the batch's rows that the walk below did not reach (for the float-float tier)
    auto combine_rest = [&](int j_from, int &bad) {
        for (int jj = j_from; jj <= K; ++jj) combine((long long)b * (K + 1) + jj, bad);
        for (int jj = j_from; jj < K; ++jj) combine(L.st.n_rows0 + (long long)b * K + jj, bad);
    };
    auto done = [&]() {
        if (lane == 0) atomicSub(&L.st.counters->n_pending, 1);
    };
    auto to_exact = [&]() {
        if (lane == 0) {
            stats_add(a.stats, &a.stats->reresolved, 1);
            push_exact(a.counters, a.exact, a.exact_unc, {-1, b}, a.stats);
        }
    };
    int bad = 0;
    if (lane == 0) {   // rows this batch streamed
        const int last = kind == kBatchOne ? j0 : K;
        const int n_d = greedy ? 0 : max(0, min(last, K - 1) - j0 + 1);
        stats_add(a.stats, &a.stats->rows, last - j0 + 1 + n_d);
    }
    if (kind == kBatchComplete) {
        combine_rest(j0, bad);
        bad = __shfl_sync(0xFFFFFFFFu, bad, 0);
        if (bad) outputs(0, -1);
        else to_exact();
        done();
        return;
    }
    const int j_last = kind == kBatchTail ? K : j0;   // rows of positions j0..j_last are read
    float c_hi = 0.f, c_lo = 0.f;
    if (!greedy) log2e_over(T, c_hi, c_lo);
    for (int j = j0; j <= j_last; ++j) {
        const RowStat rq = combine((long long)b * (K + 1) + j, bad);
        const bool with_p = !greedy && j < K;
        RowStat rp{};
        if (with_p) rp = combine(L.st.n_rows0 + (long long)b * K + j, bad);
        const int s = j < K ? token(j) : -1;
        const double u_j = __shfl_sync(0xFFFFFFFFu, u_l, j);
        // lane 0 decides: 0 finished with (k, tstar), 1 accepted, 2 for the float-float tier
        int verdict = 0, k = 0, tstar = -1;
        if (lane == 0) {
            if (bad) {
                k = 0;
            } else if (greedy) {
                if (j < K && s == rq.argmax) verdict = 1;
                else {
                    k = j;
                    tstar = rq.argmax;
                }
            } else {
                if (a.debug) {
                    double *dbg = a.debug + ((size_t)b * (K + 1) + j) * SV_DEBUG_FIELDS;
                    dbg[SV_DBG_LSE_Q] = rs_g(rq) * kLn2;
                    dbg[SV_DBG_MASS_Q] = 1.0;
                    if (with_p) {
                        const double cd = 1.4426950408889634074 / (double)T;
                        const char *trow = a.tgt.base + ((long long)b * a.tgt.rows_per_seq + j) * a.tgt.pitch_bytes;
                        const char *drow = a.drf.base + ((long long)b * a.drf.rows_per_seq + j) * a.drf.pitch_bytes;
                        const float xt = load_elem<ES>(trow, s), xd = load_elem<ES>(drow, s);
                        const double lq = xt == -INFINITY ? -INFINITY : (double)xt * cd - rs_g(rq);
                        const double lp = xd == -INFINITY ? -INFINITY : (double)xd * cd - rs_g(rp);
                        dbg[SV_DBG_LSE_P] = rs_g(rp) * kLn2;
                        dbg[SV_DBG_Q_S] = exp2(lq);
                        dbg[SV_DBG_P_S] = exp2(lp);
                        dbg[SV_DBG_RATIO] = (lp == -INFINITY) ? (lq == -INFINITY ? 0.0 : INFINITY) : exp2(lq - lp);
                        dbg[SV_DBG_MASS_P] = 1.0;
                    }
                }
                if (with_p) {
                    const AcceptOutcome o = accept_test<ES>(a, b, j, s, u_j, c_hi, c_lo, rq, rp);
                    stats_add(a.stats, &a.stats->accept_tests, 1);
                    if (o.near) stats_add(a.stats, &a.stats->near_boundary, 1);
                    if (o.amb) {
                        verdict = 2;
                        k = j;   // placeholder outputs; the float-float tier writes the final ones
                    } else if (o.acc) {
                        verdict = 1;
                    } else {
                        k = j;
                        lazy_draw<ES>(a, b, j, T, rq, rp);
                    }
                } else {
                    k = K;
                    lazy_draw<ES>(a, b, K, T, rq, rp);   // all K accepted: bonus draw from row K
                }
            }
        }
        verdict = __shfl_sync(0xFFFFFFFFu, verdict, 0);
        k = __shfl_sync(0xFFFFFFFFu, k, 0);
        tstar = __shfl_sync(0xFFFFFFFFu, tstar, 0);
        bad = __shfl_sync(0xFFFFFFFFu, bad, 0);
        if (verdict == 0) {
            outputs(k, tstar);
            done();
            return;
        }
        if (verdict == 2) {
            outputs(k, -1);
            if (j_last > j) {
                combine_rest(j + 1, bad);   // the rest of this tail batch is read already
                to_exact();
                done();
            } else if (j + 1 <= K) {
                if (lane == 0) lazy_enqueue(L, b, j + 1, K, !greedy, kBatchComplete, cum);
            } else {
                to_exact();
                done();
            }
            return;
        }
        // accepted: the next position is in this batch, or queue it (alone, or with the tail)
        if (j == j_last) {
            if (lane == 0) {
                const int jn = j + 1;
                if (jn >= kLazyTail) lazy_enqueue(L, b, jn, K, !greedy && jn < K, kBatchTail, cum);
                else lazy_enqueue(L, b, jn, jn, !greedy && jn < K, kBatchOne, cum);
            }
            return;
        }
    }
}

// Loads with acquire semantics at GPU scope (queue flags written by other blocks).
__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Block of the lazy pass: eight consumer warps, the producer warp, and a finisher warp that
// runs the position bookkeeping (row combine, accept test, queueing) off the consumers' path.
constexpr int kLazyThreads = kStatsThreads + 32;
constexpr int kLazyRing = 64;                 // finish requests in flight per block
constexpr int kLazyTCache = 2048;             // temperatures cached in shared memory
constexpr int kLazyCtlBytes = 1024 + kLazyRing * 16 + kLazyTCache * 4;   // + request ring + cache
static_assert(2 * kStatsStages * 8 + 16 + kStatsStages * (int)sizeof(TileMeta) <= 1024, "control block");
constexpr size_t kLazySmemBytes = (size_t)kLazyCtlBytes + (size_t)kStatsStages * kStatsTileBytes;

// The statistics pass of k_stats with a work queue that grows while it runs.
template <int ES>
__global__ void __launch_bounds__(kLazyThreads, 2) k_lazy(const LazyArgs L) {
    pdl_trigger();   // a dependent launch may be scheduled; it waits for this kernel
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kStatsStages;
    int *abort_flag = reinterpret_cast<int *>(smem + 2 * kStatsStages * 8);
    volatile int *ring_tail = abort_flag + 1;     // requests posted
    volatile int *ring_head = abort_flag + 2;     // requests taken by the finisher warp
    volatile int *cons_done = abort_flag + 3;     // consumer warps that left their loop
    TileMeta *meta = reinterpret_cast<TileMeta *>(smem + 2 * kStatsStages * 8 + 16);
    volatile int4 *ring = reinterpret_cast<volatile int4 *>(smem + 1024);   // (b, j0, completing, tag)
    unsigned char *tiles = smem + kLazyCtlBytes;
    const StatsArgs &a = L.st;
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
        fence_barrier_init();
    }
    // temperatures of the first sequences in shared memory (the producer looks one up per unit)
    float *t_cache = reinterpret_cast<float *>(smem + 1024 + kLazyRing * 16);
    const int n_cache = min(kLazyTCache, L.n_seq);
    for (int i = tid; i < n_cache; i += blockDim.x) t_cache[i] = a.temperature[i];
    if (tid < kLazyRing) {
        ring[tid].x = 0;
        ring[tid].y = 0;
        ring[tid].z = 0;
        ring[tid].w = 0;
    }
    __syncthreads();

    if (warp == kWarps + 1) {
        // ---------------- finisher ----------------
        int h = 0;
        const long long t0 = clock64();
        unsigned ns = 64;
        while (true) {
            if (h < *ring_tail) {
                int4 r = make_int4(0, 0, 0, 0);
                bool ok = false;
                for (int spin = 0; spin < (1 << 22); ++spin) {   // the request's fields land just after its slot
                    volatile int4 *v = &ring[h % kLazyRing];
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
                lazy_finish<ES>(L, r.x, r.y >> 2, r.y & 3, r.z);
                __syncwarp();
                ++h;
                if (lane == 0) *ring_head = h;
                ns = 64;
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
            // One FIFO: the position-0 units written before the pass, then the units finishers
            // append during it.  In the bulk of the pass each iteration claims the next slot and
            // starts loading its word before issuing the current unit's copies; near the end it
            // claims only when idle, so that queued units go to idle blocks.
            const long long q0_n = *reinterpret_cast<volatile int *>(&a.counters->q0_tail);
            auto slot_of = [&](long long c) { return c < q0_n ? c : L.q1_base + (c - q0_n); };
            auto load_word = [&](long long c) {
                const long long sl = slot_of(c);
                return sl < L.cap ? ld_relaxed_u64(&L.units[sl]) : 0ull;
            };
            long long claim = atomicAdd(&a.counters->q_head, 1);
            unsigned long long word = load_word(claim);
            const long long t_start = clock64();
            while (ok) {
                long long unit = -1;
                int aux = 0;
                unsigned ns = 32;
                while (slot_of(claim) < L.cap && !(word >> 63)) {
                    if (ld_acquire(&a.counters->n_pending) == 0) break;   // no more work will appear
                    if (*reinterpret_cast<volatile int *>(abort_flag) || clock64() - t_start > a.wait_limit) {
                        if (atomicExch(abort_flag, 1) == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
                        ok = false;
                        break;
                    }
                    __nanosleep(ns);
                    ns = ns < 256 ? 2 * ns : 256;
                    word = load_word(claim);
                }
                if (word >> 63) {
                    unit = (long long)(unsigned)(word & 0xFFFFFFFFu);
                    aux = (int)((word >> 32) & 0x7FFFFFFFu);
                }
                const bool have = ok && unit >= 0;
                long long next = -1;
                unsigned long long next_word = 0;
                if (have && q0_n + *reinterpret_cast<volatile int *>(&a.counters->q_tail) - claim > 2LL * gridDim.x) {
                    next = atomicAdd(&a.counters->q_head, 1);
                    next_word = load_word(next);
                }
                UnitInfo ui;
                if (have) ui = stats_unit<ES>(a, unit, t_cache, n_cache);
                const int nt = have ? max(unit_tiles(ui), 1) : 1;
                for (int t = 0; t < nt; ++t, ++it) {
                    if (it >= kStatsStages) {
                        if (!mbar_wait_or_abort(&empty[st], epar, abort_flag, a.wait_limit)) {
                            if (atomicExch(abort_flag, 1) == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
                            ok = false;
                            break;
                        }
                    }
                    in_flight[st] = -1;
                    TileMeta m;
                    if (!have) {
                        m.flags = kTileEnd;
                        meta[st] = m;
                        mbar_arrive(&full[st]);
                        ok = false;
                        break;
                    }
                    const int fv = ui.v0 + t * (kStatsTileBytes / 16);
                    const int nv = max(0, min(kStatsTileBytes / 16, ui.v1 - fv));
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
                    m.aux = aux;
                    meta[st] = m;
                    if (nv > 0) {
                        mbar_arrive_expect_tx(&full[st], (uint32_t)nv * 16u);
                        bulk_load_stream(tiles + st * kStatsTileBytes, ui.row + (size_t)fv * 16, (uint32_t)nv * 16u,
                                         &full[st], policy);
                        in_flight[st] = it;
                    } else {
                        mbar_arrive(&full[st]);
                    }
                    if (++st == kStatsStages) {
                        st = 0;
                        if (it >= 2 * kStatsStages - 1) epar ^= 1u;
                    }
                }
                if (next >= 0) {
                    claim = next;
                    word = next_word;
                } else {
                    claim = atomicAdd(&a.counters->q_head, 1);
                    word = load_word(claim);
                }
            }
            if (*reinterpret_cast<volatile int *>(abort_flag)) {
                for (int s = 0; s < kStatsStages; ++s)
                    if (in_flight[s] >= 0)
                        mbar_wait_bounded(&full[s], (uint32_t)((in_flight[s] / kStatsStages) & 1), a.wait_limit / 16);
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    StatAcc A;
    acc_init(A);
    int st = 0;
    uint32_t par = 0;
    for (;;) {
        if (!mbar_wait_or_abort(&full[st], par, abort_flag, a.wait_limit)) {
            if (lane == 0 && atomicExch(abort_flag, 1) == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
            break;
        }
        const TileMeta m = meta[st];
        if (m.flags & kTileEnd) break;
        const bool greedy = (m.flags & kTileGreedy) != 0;
        if (m.flags & kTileFirst) acc_init(A);
        if (m.nv > 0) acc_tile<ES>(A, tiles + st * kStatsTileBytes, m.nv, m.fv, greedy, m.c_hi);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        if (m.flags & kTileLast) {
            if (tid < m.n_tail) {
                const float x = load_elem<ES>(m.row, m.tail0 + tid);
                acc_scalar(A, x, m.tail0 + tid, greedy, m.c_hi, m.c_lo);
            }
            acc_store(A, greedy, a.part + ((size_t)m.rid * a.n_split + m.chunk) * kWarps + warp);
            // the warp that completes the batch of rows finishes the position
            int b = 0, j = 0, fin = 0;
            seq_pos(L, m.rid, b, j);
            if (lane == 0) {
                __threadfence();
                fin = atomicAdd(&L.pos_cnt[b], 1) == (m.aux >> 8) - 1;
            }
            fin = __shfl_sync(0xFFFFFFFFu, fin, 0);
            if (fin && lane == 0) {
                // hand the finish to the finisher warp (bounded wait for ring space)
                __threadfence();
                const long long t0 = clock64();
                bool room = true;
                while (*ring_tail - *ring_head >= kLazyRing - kWarps) {
                    if (*reinterpret_cast<volatile int *>(abort_flag) || clock64() - t0 > a.wait_limit) {
                        room = false;
                        if (atomicExch(abort_flag, 1) == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
                        break;
                    }
                    __nanosleep(128);
                }
                if (room) {
                    const int slot = atomicAdd(reinterpret_cast<int *>(const_cast<int *>(ring_tail)), 1);
                    volatile int4 *e = &ring[slot % kLazyRing];
                    e->x = b;
                    e->y = m.aux & 0xFF;        // (first position << 2) | kind
                    e->z = m.aux >> 8;          // cumulative count reached
                    __threadfence_block();
                    e->w = slot + 1;
                }
            }
            __syncwarp();
        }
        if (++st == kStatsStages) {
            st = 0;
            par ^= 1u;
        }
    }
    __syncwarp();
    if (lane == 0) atomicAdd(reinterpret_cast<int *>(const_cast<int *>(cons_done)), 1);
}

template <int ES>
static sv_status launch_lazy(const VerifyPlan &pl, const AcceptArgs &acc_in, int B, void *ws, cudaStream_t stream) {
    DeviceInfo di;
    if (!device_info(di)) return SV_ERR_CUDA;
    char *w = static_cast<char *>(ws);
    Counters *counters = reinterpret_cast<Counters *>(w + pl.off_counters);
    LazyArgs L{};
    L.st.set[0] = acc_in.tgt;
    L.st.set[1] = acc_in.drf;
    L.st.n_sets = 2;
    L.st.V = acc_in.V;
    L.st.temperature = acc_in.temperature;
    L.st.n_split = pl.n_split;
    L.st.chunk_vecs = pl.chunk_vecs;
    L.st.n_rows0 = pl.n_rows0;
    L.st.n_units = (pl.n_rows0 + pl.n_rows1) * pl.n_split;
    L.st.part = reinterpret_cast<WarpPartial *>(w + pl.off_part);
    L.st.counters = counters;
    L.st.stats = acc_in.stats;
    L.st.wait_limit = kWaitLimitCycles;
    L.acc = acc_in;
    L.acc.part = L.st.part;
    L.acc.n_split = pl.n_split;
    L.acc.n_rows0 = pl.n_rows0;
    L.acc.rowstat = reinterpret_cast<RowStat *>(w + pl.off_rowstat);
    L.acc.nuc = nullptr;
    L.acc.top = nullptr;
    L.acc.draws = reinterpret_cast<DrawItem *>(w + pl.off_draws);
    L.acc.exact = reinterpret_cast<ExactItem *>(w + pl.off_exact);
    L.acc.exact_unc = reinterpret_cast<int *>(w + pl.off_xunc_n);
    L.acc.counters = counters;
    L.units = reinterpret_cast<unsigned long long *>(w + pl.off_lz_units);
    L.pos_cnt = reinterpret_cast<int *>(w + pl.off_lz_pos);
    L.cap = pl.lz_cap;
    L.q1_base = (long long)B * pl.n_split * (acc_in.K > 0 ? 2 : 1);
    L.n_seq = B;
    if (cudaMemsetAsync(counters, 0, sizeof(Counters), stream) != cudaSuccess) return SV_ERR_CUDA;
    if (cudaMemsetAsync(L.units, 0, (size_t)pl.lz_cap * sizeof(unsigned long long), stream) != cudaSuccess)
        return SV_ERR_CUDA;
    if (cudaMemsetAsync(L.pos_cnt, 0, (size_t)B * sizeof(int), stream) != cudaSuccess) return SV_ERR_CUDA;
    k_lazy_init<<<(unsigned)div_up(B, kThreads), kThreads, 0, stream>>>(L, B);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    {
        const int occ = prepare_kernel((const void *)k_lazy<ES>, kLazyThreads, kLazySmemBytes);
        if (occ < 1) return SV_ERR_CUDA;
        // blocks wait for units that other blocks queue, so every block must be resident:
        // a cooperative launch guarantees it (or fails)
        static_assert(sizeof(LazyArgs) < 4096, "kernel parameter block");
        void *args[] = {&L};
        profile_begin(stream);
        const cudaError_t e = cudaLaunchCooperativeKernel((const void *)k_lazy<ES>, dim3(di.sms * occ),
                                                          dim3(kLazyThreads), args, kLazySmemBytes, stream);
        if (e != cudaSuccess) return SV_ERR_CUDA;
        profile_end(stream);
    }
    DrawArgs da;
    da.items = L.acc.draws;
    da.counters = counters;
    da.V = acc_in.V;
    da.n_vec = pl.n_vec;
    da.n_sub = pl.n_sub;
    da.n_split = pl.d_split;
    da.subs_per_chunk = pl.d_subs_per_chunk;
    da.subs = reinterpret_cast<float *>(w + pl.off_subs);
    da.exact = L.acc.exact;
    da.exact_unc = L.acc.exact_unc;
    da.stats = acc_in.stats;
    da.wait_limit = kWaitLimitCycles;
    {
        const sv_status st = launch_draws<ES>(da, (long long)B, di, stream);
        if (st != SV_OK) return st;
    }
    ExactArgs xa;
    xa.tgt = acc_in.tgt;
    xa.drf = acc_in.drf;
    xa.K = acc_in.K;
    xa.V = acc_in.V;
    xa.temperature = acc_in.temperature;
    xa.tokens = acc_in.tokens;
    xa.uniforms = acc_in.uniforms;
    xa.accept_len = acc_in.accept_len;
    xa.out_tokens = acc_in.out_tokens;
    xa.debug = acc_in.debug;
    xa.sag_C = acc_in.sag_C;
    xa.sag_on = 0;
    xa.draw_from_q = 0;
    xa.nuc = nullptr;
    xa.top = nullptr;
    xa.rowstat = L.acc.rowstat;
    xa.n_rows0 = pl.n_rows0;
    xa.draws = L.acc.draws;
    xa.items = L.acc.exact;
    xa.counters = counters;
    xa.xpart = reinterpret_cast<double *>(w + pl.off_xpart);
    xa.xdraw = reinterpret_cast<ExactDraw *>(w + pl.off_xdraw);
    xa.xsubs = reinterpret_cast<float4 *>(w + pl.off_xsubs);
    xa.xnorm = reinterpret_cast<float4 *>(w + pl.off_xnorm);
    xa.xunc_n = reinterpret_cast<int *>(w + pl.off_xunc_n);
    xa.xunc = reinterpret_cast<int *>(w + pl.off_xunc);
    xa.n_vec = pl.n_vec;
    xa.n_sub = pl.n_sub;
    xa.xsplit = pl.x_split;
    xa.max_slots = 2 * acc_in.K + 1 > 2 ? 2 * acc_in.K + 1 : 2;
    xa.stats = acc_in.stats;
    xa.wait_limit = kWaitLimitCycles;
    return launch_exact<ES>(xa, di, stream);
}

}  // namespace sv

using namespace sv;

extern "C" sv_status sv_verify_lazy(const void *target_logits, int64_t t_row_pitch, const void *draft_logits,
                                    int64_t d_row_pitch, int d_rows_per_seq, sv_dtype dtype,
                                    const int32_t *draft_tokens, const double *uniforms, int B, int K, int V,
                                    const float *temperature, const float *top_p, const int32_t *top_k,
                                    int saguaro_F, float saguaro_C,
                                    int32_t *accept_len, int32_t *out_tokens, double *debug, sv_stats *stats,
                                    void *workspace, size_t workspace_bytes, sv_stream_t stream_) {
    const bool sag_on = saguaro_F > 0 && saguaro_C != 1.0f;
    if (top_p != nullptr || top_k != nullptr || sag_on)
        return sv_verify(target_logits, t_row_pitch, draft_logits, d_row_pitch, d_rows_per_seq, dtype, draft_tokens,
                         uniforms, B, K, V, temperature, top_p, top_k, saguaro_F, saguaro_C, accept_len, out_tokens, debug,
                         stats, workspace, workspace_bytes, stream_);
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (B < 1 || K < 0 || K > SV_MAX_K || V < 1) return SV_ERR_INVALID_ARG;
    if (!rows_ok(target_logits, t_row_pitch, V, dtype)) return SV_ERR_INVALID_ARG;
    if (K > 0 && (!rows_ok(draft_logits, d_row_pitch, V, dtype) || d_rows_per_seq < K)) return SV_ERR_INVALID_ARG;
    if ((K > 0 && draft_tokens == nullptr) || uniforms == nullptr || temperature == nullptr) return SV_ERR_INVALID_ARG;
    if (accept_len == nullptr || out_tokens == nullptr) return SV_ERR_INVALID_ARG;
    if (saguaro_F < 0 || !(saguaro_C >= 0.0f && saguaro_C <= 1.0f)) return SV_ERR_INVALID_ARG;
    if ((long long)V * B * (2 * K + 1) > (1LL << 46)) return SV_ERR_INVALID_ARG;
    const int es = elem_size(dtype);
    const VerifyPlan pl = plan_verify(B, K, V, es);
    if (pl.lz_cap >= (1LL << 31)) return SV_ERR_INVALID_ARG;
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < pl.bytes) return SV_ERR_WORKSPACE;
    if (!on_current_device(stream, target_logits, K > 0 ? draft_logits : nullptr)) return SV_ERR_INVALID_ARG;
    if (stats && cudaMemsetAsync(stats, 0, sizeof(sv_stats), stream) != cudaSuccess) return SV_ERR_CUDA;
    AcceptArgs acc{};
    acc.tgt = {static_cast<const char *>(target_logits), t_row_pitch * es, K + 1, K + 1, 0};
    acc.drf = {static_cast<const char *>(K > 0 ? draft_logits : target_logits), (K > 0 ? d_row_pitch : t_row_pitch) * es,
               K > 0 ? d_rows_per_seq : 1, K, 1};
    acc.K = K;
    acc.V = V;
    acc.temperature = temperature;
    acc.top_p = nullptr;
    acc.sag_on = 0;
    acc.sag_C = 1.0f;
    acc.tokens = draft_tokens;
    acc.uniforms = uniforms;
    acc.accept_len = accept_len;
    acc.out_tokens = out_tokens;
    acc.debug = debug;
    acc.stats = stats;
    if (es == 4) return launch_lazy<4>(pl, acc, B, workspace, stream);
    return launch_lazy<2>(pl, acc, B, workspace, stream);
}
