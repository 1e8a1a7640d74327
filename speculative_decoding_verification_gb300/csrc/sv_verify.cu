// sv_verify.cu — sv_verify: modified rejection sampling over the vocabulary for B sequences.
//
// ["Speculative Speculative Decoding" notes, §2.2 steps ①-④; "Accelerating LLM Decoding with
//  Speculative Sampling (2023)" notes, §3; "Mirror Speculative Decoding" notes, §2 step 3]
//
// Kernels, in stream order:
//   k_stats        one streaming pass over every needed row: target rows of all sequences, draft
//                  rows of sampled sequences (greedy sequences never read the draft)
//   k_nucleus      (top-p only) the nucleus cut of every sampled row
//   k_topset       (sigma_{F,C} only) the top-F set of every draft row
//   k_accept       per sequence: float64 row normalisers, the accept tests u < min(1, q/p) with a
//                  certified margin, the first rejection k, greedy outputs, and a draw item
//   k_draw_sums    per draw: sub-chunk sums of w = (q_{k+1} - p_{k+1})_+ or q_{K+1}
//   k_draw_finish  per draw: t* with a certified margin
//   k_exact        float-float tier for the decisions the margins could not settle
#include <math.h>

#include "sv_accept.cuh"
#include "sv_draw.cuh"
#include "sv_exact.cuh"
#include "sv_host.h"
#include "sv_select.cuh"
#include "sv_stats.cuh"
#include "sv_tiers.cuh"

namespace sv {

template <int ES>
__global__ void __launch_bounds__(kThreads) k_accept(const AcceptArgs a) {
    __shared__ RowStat rs[2 * SV_MAX_K + 1];
    __shared__ int s_err;
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = a.K, V = a.V;
    const float T = a.temperature[b];
    const bool greedy = (T == 0.0f);
    const bool bad_t = !(greedy || (T >= 1e-3f && T <= 1e3f));
    int32_t *outs = a.out_tokens + (size_t)b * (K + 1);
    if (tid == 0) s_err = 0;
    __syncthreads();
    if (bad_t) {
        if (tid == 0) {
            report_error(a.stats, SV_ERR_INVALID_ARG, b);
            a.accept_len[b] = 0;
        }
        for (int j = tid; j <= K; j += kThreads) outs[j] = -1;
        return;
    }
    const int n_t = K + 1, n_d = greedy ? 0 : K;
    // warp 0 loads its lane's draft token, uniform and the two logits at that token now, so
    // that those loads overlap the row combination below
    int s = -1;
    float xt = 0.f, xd = 0.f;
    double u_acc = 0.0;
    if (warp == 0 && lane < K) {
        s = a.tokens[(size_t)b * K + lane];
        if (!greedy && s >= 0 && s < V) {
            const char *trow = a.tgt.base + ((long long)b * a.tgt.rows_per_seq + lane) * a.tgt.pitch_bytes;
            const char *drow = a.drf.base + ((long long)b * a.drf.rows_per_seq + lane) * a.drf.pitch_bytes;
            xt = load_elem<ES>(trow, s);
            xd = load_elem<ES>(drow, s);
            u_acc = a.uniforms[(size_t)b * (K + 1) + lane];
        }
    }
    for (int i = warp; i < n_t + n_d; i += kWarps) {
        const long long rid = i < n_t ? (long long)b * n_t + i : a.n_rows0 + (long long)b * K + (i - n_t);
        const RowStat r = combine_row(a.part + (size_t)rid * a.n_split * kWarps, a.n_split * kWarps, greedy, T);
        if (lane == 0) {
            rs[i] = r;
            a.rowstat[rid] = r;
            const bool bad = (r.flags != 0) || (greedy ? !isfinite(r.maxv) : !rs_sampled_ok(r));
            if (bad) {
                atomicOr(&s_err, 1);
                report_error(a.stats, SV_ERR_NONFINITE, (int)rid);
            }
        }
    }
    __syncthreads();
    if (warp != 0) return;
    if (lane == 0) stats_add(a.stats, &a.stats->rows, n_t + n_d);
    if (s_err) {
        if (lane == 0) a.accept_len[b] = 0;
        for (int j = lane; j <= K; j += 32) outs[j] = -1;
        return;
    }

    // ---- accept tests (lane j tests position j+1), float32 / float-float only ----
    // ratio = q(s)/p(s) = 2^(y_q - y_p) * (S_p m_p z_p) / (S_q m_q C_s) with y = x c - r, S the
    // row sums, m the nucleus masses, z the Saguaro normaliser and C_s = C on the top-F set.
    // y_q - y_p is formed in float-float; its float32 exponential, the products and the
    // quotient carry kEx2RelErr + 8u, the row sums err_q + err_p, the masses 2(err_q + err_p)
    // and the normaliser z_err; u < ratio is certain outside ratio (1 -+ delta).
    float c_hi = 0.f, c_lo = 0.f;
    if (!greedy) log2e_over(T, c_hi, c_lo);
    bool acc = false, amb = false, near = false, badtok = false;
    bool keep_q = false, keep_p = false, in_top = false;
    float ratio = NAN;
    if (lane < K) {
        badtok = s < 0 || s >= V;
        if (!badtok) {
            if (greedy) {
                acc = (s == rs[lane].argmax);
            } else {
                const AcceptOutcome o = accept_test_x(a, b, lane, s, u_acc, c_hi, c_lo, rs[lane], rs[n_t + lane], xt, xd);
                acc = o.acc;
                amb = o.amb;
                near = o.near;
                keep_q = o.keep_q;
                keep_p = o.keep_p;
                in_top = o.in_top;
                ratio = o.ratio;
            }
        }
    }
    const unsigned lowK = K >= 32 ? 0xFFFFFFFFu : ((1u << K) - 1u);
    const unsigned accm = __ballot_sync(0xFFFFFFFFu, acc) & lowK;
    const unsigned badm = __ballot_sync(0xFFFFFFFFu, badtok) & lowK;
    const unsigned rej = ~accm & lowK;
    const int k = rej ? __ffs(rej) - 1 : K;
    const unsigned scanned = (unsigned)((k < K) ? ((2ull << k) - 1ull) : (unsigned long long)lowK);
    const unsigned ambm = __ballot_sync(0xFFFFFFFFu, amb) & scanned;
    const unsigned nearm = __ballot_sync(0xFFFFFFFFu, near) & scanned;
    if (badm) {
        if (lane == 0) {
            report_error(a.stats, SV_ERR_BAD_TOKEN, b);
            a.accept_len[b] = 0;
        }
        for (int j = lane; j <= K; j += 32) outs[j] = -1;
        return;
    }
    // outputs: s_1..s_k, then t* (greedy now, sampled after the draw), -1 padding
    for (int j = lane; j <= K; j += 32) outs[j] = j < k ? a.tokens[(size_t)b * K + j] : -1;
    __syncwarp();
    if (lane == 0) {
        a.accept_len[b] = k;
        if (greedy) outs[k] = rs[k].argmax;
        if (!greedy) {
            stats_add(a.stats, &a.stats->accept_tests, min(k + 1, K));
            stats_add(a.stats, &a.stats->near_boundary, __popc(nearm));
        }
    }
    if (a.debug) {
        // reference values in float64 (debug output only)
        const double cd = greedy ? 0.0 : 1.4426950408889634074 / (double)T;
        double q_s = NAN, p_s = NAN, rat = NAN;
        if (!greedy && lane < K && !badtok) {
            const long long rid_t = (long long)b * n_t + lane;
            const long long rid_d = a.n_rows0 + (long long)b * K + lane;
            const char *trow = a.tgt.base + ((long long)b * a.tgt.rows_per_seq + lane) * a.tgt.pitch_bytes;
            const char *drow = a.drf.base + ((long long)b * a.drf.rows_per_seq + lane) * a.drf.pitch_bytes;
            const float xt = load_elem<ES>(trow, s), xd = load_elem<ES>(drow, s);
            double lq = keep_q ? (double)xt * cd - rs_g(rs[lane]) : -INFINITY;
            double lp = keep_p ? (double)xd * cd - rs_g(rs[n_t + lane]) : -INFINITY;
            if (a.nuc) {
                lq -= a.nuc[rid_t].log2_mass;
                lp -= a.nuc[rid_d].log2_mass;
            }
            if (a.sag_on && a.top) {
                if (in_top) lp += log2((double)a.sag_C);
                lp -= log2(a.top[rid_d].z);
            }
            q_s = exp2(lq);
            p_s = exp2(lp);
            rat = (lp == -INFINITY) ? (lq == -INFINITY ? 0.0 : INFINITY) : exp2(lq - lp);
        }
        for (int j = lane; j <= K; j += 32) {
            double *dbg = a.debug + ((size_t)b * (K + 1) + j) * SV_DEBUG_FIELDS;
            const long long rid_t = (long long)b * n_t + j;
            dbg[SV_DBG_LSE_Q] = greedy ? NAN : rs_g(rs[j]) * kLn2;
            dbg[SV_DBG_LSE_P] = (greedy || j >= K) ? NAN : rs_g(rs[n_t + j]) * kLn2;
            dbg[SV_DBG_Q_S] = j < K ? q_s : NAN;
            dbg[SV_DBG_P_S] = j < K ? p_s : NAN;
            dbg[SV_DBG_RATIO] = j < K ? rat : NAN;
            dbg[SV_DBG_MASS_Q] = (greedy || !a.nuc) ? 1.0 : a.nuc[rid_t].mass;
            dbg[SV_DBG_MASS_P] = (greedy || !a.nuc || j >= K) ? 1.0 : a.nuc[a.n_rows0 + (long long)b * K + j].mass;
            dbg[SV_DBG_R] = NAN;
        }
    }
    if (greedy || lane != 0) return;
    if (ambm) {
        // an accept test too close to call in float32: the float-float tier redoes the sequence
        stats_add(a.stats, &a.stats->reresolved, 1);
        push_exact(a.counters, a.exact, a.exact_unc, {-1, b}, a.stats);
        return;
    }
    const int d = atomicAdd(&a.counters->n_draws, 1);
    DrawItem it;
    const long long rid_q = (long long)b * n_t + k;
    const char *qrow = a.tgt.base + ((long long)b * a.tgt.rows_per_seq + k) * a.tgt.pitch_bytes;
    it.q = draw_row(qrow, T, rs[k], a.nuc ? a.nuc + rid_q : nullptr, nullptr, 1.0f);
    it.has_p = k < K && !a.draw_from_q;
    if (it.has_p) {
        const long long rid_p = a.n_rows0 + (long long)b * K + k;
        const char *prow = a.drf.base + ((long long)b * a.drf.rows_per_seq + k) * a.drf.pitch_bytes;
        it.p = draw_row(prow, T, rs[n_t + k], a.nuc ? a.nuc + rid_p : nullptr,
                        (a.sag_on && a.top) ? a.top + rid_p : nullptr, a.sag_C);
    } else {
        it.p = {};
        it.p.top_x = INFINITY;
        it.p.cut_x = -INFINITY;
        it.p.cut_id = 0x7FFFFFFF;
    }
    it.filt = (a.nuc != nullptr) || (it.has_p && a.sag_on && a.top != nullptr);
    it.u = a.uniforms[(size_t)b * (K + 1) + K];
    it.out = outs + k;
    it.dbg_r = a.debug ? a.debug + (size_t)b * (K + 1) * SV_DEBUG_FIELDS + SV_DBG_R : nullptr;
    it.seq = b;
    it.k = k;
    a.draws[d] = it;
}

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------
VerifyPlan plan_verify(int B, int K, int V, int es) {
    VerifyPlan p;
    p.es = es;
    p.n_rows0 = (long long)B * (K + 1);
    p.n_rows1 = (long long)B * K;
    const long long n_cand = p.n_rows0 + p.n_rows1;
    const long long row_bytes = (long long)V * es;
    p.n_split = choose_split(n_cand, row_bytes);
    p.n_vec = vec_count(V, es);
    chunk_geometry(p.n_vec, p.n_split, p.chunk_vecs);
    p.n_sub = sub_chunks(V, es);
    draw_geometry(p.n_sub, p.d_split, p.d_subs_per_chunk);
    Carver cv;
    p.off_counters = cv.take<Counters>(1);
    p.off_part = cv.take<WarpPartial>((size_t)n_cand * p.n_split * kWarps);
    p.off_rowstat = cv.take<RowStat>((size_t)n_cand);
    p.off_nuc = cv.take<NucleusCut>((size_t)n_cand);
    p.off_top = cv.take<TopSet>((size_t)n_cand);
    p.off_draws = cv.take<DrawItem>((size_t)B);
    p.off_subs = cv.take<float>((size_t)B * p.n_sub);
    const size_t cap = (size_t)(B < kExactCap ? B : (int)kExactCap);
    p.off_exact = cv.take<ExactItem>(cap);
    const int max_slots = 2 * K + 1 > 2 ? 2 * K + 1 : 2;
    p.off_xpart = cv.take<double>(cap * max_slots * kExactSplit * 3);
    p.off_xdraw = cv.take<ExactDraw>(cap);
    p.x_split = exact_groups(p.n_sub);
    p.off_xsubs = cv.take<float4>(cap * p.n_sub);
    p.off_xnorm = cv.take<float4>(cap * p.x_split);
    p.off_xunc_n = cv.take<int>(cap);
    p.off_xunc = cv.take<int>(cap * kExactUncCap);
    p.lz_cap = n_cand * p.n_split;
    p.off_lz_units = cv.take<unsigned long long>((size_t)p.lz_cap);
    p.off_lz_pos = cv.take<int>((size_t)B);
    const long long n_pairs = (long long)B * K;
    long long want = n_pairs > 0 ? (2LL * kUnitTarget + n_pairs - 1) / n_pairs : 1;
    if (want > kMaxSplit) want = kMaxSplit;
    if (want > p.n_vec) want = p.n_vec > 0 ? p.n_vec : 1;
    p.dv_chunks = (int)(want < 1 ? 1 : want);
    p.dv_words = p.n_vec > 0 ? (p.n_vec + p.dv_chunks - 1) / p.dv_chunks : 1;
    p.off_dpart = cv.take<DivPart>((size_t)(n_pairs > 0 ? n_pairs : 1) * p.dv_chunks);
    p.off_ditem = cv.take<DivItem>((size_t)(n_pairs > 0 ? n_pairs : 1));
    p.off_dq = cv.take<int>((size_t)(n_pairs > 0 ? n_pairs : 1));
    p.off_deferred = cv.take<int>((size_t)B);
    // the float-float divergence pass splits each queued pair over up to kDivExactChunks chunks;
    // the entries are shared by the queued pairs, so fewer chunks each when many are queued
    const long long np1 = n_pairs > 0 ? n_pairs : 1;
    p.dx_cap = (int)(4 * np1 > 4096 ? 4 * np1 : 4096);
    p.off_dxa = cv.take<float4>((size_t)p.dx_cap);
    p.off_dxb = cv.take<float2>((size_t)p.dx_cap);
    p.off_dxcnt = cv.take<int>((size_t)np1);
    p.bytes = cv.off + 256;
    return p;
}

template <int ES>
static sv_status launch_verify(const VerifyPlan &pl, const AcceptArgs &acc_in, const float *top_p,
                               const int32_t *top_k, int F, float C, int B, void *ws, cudaStream_t stream) {
    DeviceInfo di;
    if (!device_info(di)) return SV_ERR_CUDA;
    char *w = static_cast<char *>(ws);
    Counters *counters = reinterpret_cast<Counters *>(w + pl.off_counters);
    WarpPartial *part = reinterpret_cast<WarpPartial *>(w + pl.off_part);
    const long long wait = kWaitLimitCycles;
    AcceptArgs acc = acc_in;

    // 1. statistics pass
    StatsArgs sa;
    sa.set[0] = acc.tgt;
    sa.set[1] = acc.drf;
    sa.n_sets = 2;
    sa.V = acc.V;
    sa.temperature = acc.temperature;
    sa.n_split = pl.n_split;
    sa.chunk_vecs = pl.chunk_vecs;
    sa.n_rows0 = pl.n_rows0;
    sa.n_units = (pl.n_rows0 + pl.n_rows1) * pl.n_split;
    sa.part = part;
    sa.counters = counters;
    sa.stats = acc.stats;
    sa.zero_stats = true;
    sa.wait_limit = wait;
    {
        const sv_status st = launch_stats<ES>(sa, di, stream);
        if (st != SV_OK) return st;
    }
    // 2. top-k / nucleus cuts and top-F sets (only when asked for)
    NucleusCut *nuc = nullptr;
    TopSet *top = nullptr;
    if (top_p || top_k) {
        nuc = reinterpret_cast<NucleusCut *>(w + pl.off_nuc);
        sv_status st = launch_nucleus<ES>(acc.tgt, acc.drf, pl.n_rows0, pl.n_rows1, acc.V, acc.temperature, top_p,
                                          top_k, part, pl.n_split, nuc, acc.stats, stream);
        if (st != SV_OK) return st;
    }
    if (acc.sag_on) {
        top = reinterpret_cast<TopSet *>(w + pl.off_top);
        sv_status st = launch_topset<ES>(acc.drf, pl.n_rows0, B, acc.K, acc.V, acc.temperature, F, C, part,
                                         pl.n_split, nuc, top, acc.stats, di, stream);
        if (st != SV_OK) return st;
    }
    // 3. accept tests
    acc.part = part;
    acc.n_split = pl.n_split;
    acc.n_rows0 = pl.n_rows0;
    acc.rowstat = reinterpret_cast<RowStat *>(w + pl.off_rowstat);
    acc.nuc = nuc;
    acc.top = top;
    acc.draws = reinterpret_cast<DrawItem *>(w + pl.off_draws);
    acc.exact = reinterpret_cast<ExactItem *>(w + pl.off_exact);
    acc.exact_unc = reinterpret_cast<int *>(w + pl.off_xunc_n);
    acc.counters = counters;
    if (launch_pdl(k_accept<ES>, dim3(B), dim3(kThreads), 0, stream, acc) != cudaSuccess) return SV_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    // 4-5. draws and the float-float tier
    return launch_draw_tiers<ES>(pl, acc, nuc, top, w, B, di, stream);
}

}  // namespace sv

using namespace sv;

extern "C" size_t sv_verify_workspace_size(int B, int K, int V) {
    if (B < 1 || K < 0 || K > SV_MAX_K || V < 1) return 0;
    const VerifyPlan a = plan_verify(B, K, V, 4), b = plan_verify(B, K, V, 2);
    return a.bytes > b.bytes ? a.bytes : b.bytes;
}

sv_status sv::verify_entry(const void *target_logits, int64_t t_row_pitch, const void *draft_logits,
                           int64_t d_row_pitch, int d_rows_per_seq, sv_dtype dtype, const int32_t *draft_tokens,
                           const double *uniforms, int B, int K, int V, const float *temperature, const float *top_p,
                           const int32_t *top_k, int saguaro_F, float saguaro_C, int draw_from_q, int32_t *accept_len,
                           int32_t *out_tokens, double *debug, sv_stats *stats, void *workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
    if (B < 1 || K < 0 || K > SV_MAX_K || V < 1) return SV_ERR_INVALID_ARG;
    if (!rows_ok(target_logits, t_row_pitch, V, dtype)) return SV_ERR_INVALID_ARG;
    if (K > 0 && (!rows_ok(draft_logits, d_row_pitch, V, dtype) || d_rows_per_seq < K)) return SV_ERR_INVALID_ARG;
    if ((K > 0 && draft_tokens == nullptr) || uniforms == nullptr || temperature == nullptr) return SV_ERR_INVALID_ARG;
    if (accept_len == nullptr || out_tokens == nullptr) return SV_ERR_INVALID_ARG;
    if (saguaro_F < 0 || !(saguaro_C >= 0.0f && saguaro_C <= 1.0f)) return SV_ERR_INVALID_ARG;
    if ((long long)V * B * (2 * K + 1) > (1LL << 46)) return SV_ERR_INVALID_ARG;
    const int es = elem_size(dtype);
    const VerifyPlan pl = plan_verify(B, K, V, es);
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < pl.bytes) return SV_ERR_WORKSPACE;
    if (!on_current_device(stream, target_logits, K > 0 ? draft_logits : nullptr)) return SV_ERR_INVALID_ARG;
    // stats is cleared by the call's first kernel (launch_stats)

    AcceptArgs acc{};
    acc.tgt = {static_cast<const char *>(target_logits), t_row_pitch * es, K + 1, K + 1, 0};
    acc.drf = {static_cast<const char *>(K > 0 ? draft_logits : target_logits), (K > 0 ? d_row_pitch : t_row_pitch) * es,
               K > 0 ? d_rows_per_seq : 1, K, 1};
    acc.K = K;
    acc.V = V;
    acc.temperature = temperature;
    acc.top_p = top_p;
    acc.sag_on = (saguaro_F > 0 && saguaro_C != 1.0f) ? 1 : 0;
    acc.sag_C = saguaro_C;
    acc.tokens = draft_tokens;
    acc.uniforms = uniforms;
    acc.accept_len = accept_len;
    acc.out_tokens = out_tokens;
    acc.debug = debug;
    acc.stats = stats;
    acc.draw_from_q = draw_from_q;
    if (es == 4) return launch_verify<4>(pl, acc, top_p, top_k, saguaro_F, saguaro_C, B, workspace, stream);
    return launch_verify<2>(pl, acc, top_p, top_k, saguaro_F, saguaro_C, B, workspace, stream);
}

extern "C" sv_status sv_verify(const void *target_logits, int64_t t_row_pitch, const void *draft_logits,
                               int64_t d_row_pitch, int d_rows_per_seq, sv_dtype dtype, const int32_t *draft_tokens,
                               const double *uniforms, int B, int K, int V, const float *temperature,
                               const float *top_p, const int32_t *top_k, int saguaro_F, float saguaro_C,
                               int32_t *accept_len, int32_t *out_tokens, double *debug, sv_stats *stats,
                               void *workspace, size_t workspace_bytes, sv_stream_t stream) {
    return sv::verify_entry(target_logits, t_row_pitch, draft_logits, d_row_pitch, d_rows_per_seq, dtype, draft_tokens,
                            uniforms, B, K, V, temperature, top_p, top_k, saguaro_F, saguaro_C, 0, accept_len,
                            out_tokens, debug, stats, workspace, workspace_bytes,
                            reinterpret_cast<cudaStream_t>(stream));
}
