// sv_sample.cu — sv_saguaro_sample: draft sampling under sigma_{F,C}.
//
// [SSD notes §4.4, Theorems 15 and 19; SSD abstract page, "Method"]: the draft probabilities of the
// top-F tokens (ranked by draft logit) are multiplied by C and the row is renormalised, so the
// residual (q - p')_+ concentrates on those tokens.  Each row is one inverse-CDF draw in token-id
// order; greedy rows (T = 0) take the argmax.
//
// Kernels: k_stats (row normalisers) -> [k_nucleus] -> [k_topset] -> k_sample_items (one draw item
// per sampled row) -> k_draw_sums -> k_draw_finish -> k_exact.
#include "sv_draw.cuh"
#include "sv_exact.cuh"
#include "sv_host.h"
#include "sv_select.cuh"
#include "sv_stats.cuh"

namespace sv {

struct SampleArgs {
    RowSet rows;
    int n_rows, V;
    const float *temperature;
    float C;
    int sag_on;
    const double *uniforms;
    int32_t *tokens;
    double *debug;
    sv_stats *stats;
    const WarpPartial *part;
    int n_split;
    RowStat *rowstat;
    const NucleusCut *nuc;
    const TopSet *top;
    DrawItem *draws;
    Counters *counters;
};

// One warp per row: combine the statistics, then either write the argmax (greedy) or queue a draw.
__global__ void __launch_bounds__(kThreads) k_sample_items(const SampleArgs a, long long total) {
    pdl_trigger();   // a dependent launch may be scheduled; it waits for this kernel
    const int lane = threadIdx.x & 31;
    const long long r = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5;
    if (r >= total) return;
    const long long b = r / a.n_rows, j = r - b * a.n_rows;
    const float T = a.temperature[b];
    const bool greedy = (T == 0.0f);
    if (!(greedy || (T >= 1e-3f && T <= 1e3f))) {
        if (lane == 0) {
            report_error(a.stats, SV_ERR_INVALID_ARG, (int)b);
            a.tokens[r] = -1;
        }
        return;
    }
    // combine partials (same arithmetic as the verify path)
    const RowStat rs = combine_row(a.part + (size_t)r * a.n_split * kWarps, a.n_split * kWarps, greedy, T);
    if (lane != 0) return;
    a.rowstat[r] = rs;
    const bool bad = rs.flags != 0 || (greedy ? !isfinite(rs.maxv) : !rs_sampled_ok(rs));
    if (bad) {
        report_error(a.stats, SV_ERR_NONFINITE, (int)r);
        a.tokens[r] = -1;
        return;
    }
    stats_add(a.stats, &a.stats->rows, 1);
    if (a.debug) {
        double *dbg = a.debug + (size_t)r * 4;
        dbg[0] = greedy ? NAN : rs_g(rs) * kLn2;
        dbg[1] = (a.top && !greedy) ? a.top[r].p_d : 0.0;
        dbg[2] = (a.top && !greedy) ? a.top[r].z : 1.0;
        dbg[3] = (a.nuc && !greedy) ? a.nuc[r].mass : 1.0;
    }
    if (greedy) {
        a.tokens[r] = rs.argmax;
        return;
    }
    const char *row = a.rows.base + (b * a.rows.rows_per_seq + j) * a.rows.pitch_bytes;
    DrawItem it;
    // the sampled row carries both the nucleus cut and the top-F scaling
    {
        DrawRow &d = it.q;
        d.row = row;
        log2e_over(T, d.c_hi, d.c_lo);
        d.rf = (float)rs.r;
        float norm = rs.s_hi;
        double err = rs_err(rs) + 4.0 * kU32;   // S_lo dropped, products, reciprocal
        d.cut_x = -INFINITY;
        d.cut_id = 0x7FFFFFFF;
        d.top_x = INFINITY;
        d.top_id = -1;
        d.sc_d = 1.0f;
        if (a.nuc) {
            d.cut_x = a.nuc[r].cut_x;
            d.cut_id = a.nuc[r].cut_id;
            norm = __fmul_rn(norm, a.nuc[r].mass_f);
            err += 2.0 * rs_err(rs) + kU32 + 1e-12;
        }
        if (a.top) {
            d.top_x = a.top[r].top_x;
            d.top_id = a.top[r].top_id;
            d.sc_d = a.C;
            norm = __fmul_rn(norm, a.top[r].z_f);
            err += (double)a.top[r].z_err_f + kU32;
        }
        d.inv_s = __frcp_rn(norm);
        d.k_lo = __fmul_rn(__fmul_rn(d.c_lo, (float)kLn2), d.inv_s);
        d.pad = 0;
        d.ay = __fdiv_ru(rs.ay * (1.0f + 0x1p-20f), __fdiv_rn(norm, rs.s_hi) * (1.0f - 0x1p-20f));
        d.norm_err = err;
    }
    it.p = {};
    it.p.top_x = INFINITY;
    it.p.cut_x = -INFINITY;
    it.p.cut_id = 0x7FFFFFFF;
    it.has_p = 0;
    it.filt = (a.nuc != nullptr) || (a.top != nullptr);
    it.u = a.uniforms[r];
    it.out = a.tokens + r;
    it.dbg_r = nullptr;
    it.seq = (int)b;
    it.k = (int)j;
    const int d = atomicAdd(&a.counters->n_draws, 1);
    a.draws[d] = it;
}

struct SamplePlan {
    VerifyPlan v;   // geometry of the statistics and draw passes
    size_t bytes;
};

static SamplePlan plan_sample(int B, int n_rows, int V, int es) {
    // A sampling call is a verify-shaped problem with one "target" row set and no draft set;
    // each sampled row is one draw.
    const long long rows = (long long)B * n_rows;
    SamplePlan sp;
    VerifyPlan &p = sp.v;
    p.es = es;
    p.n_rows0 = rows;
    p.n_rows1 = 0;
    p.n_split = choose_split(rows, (long long)V * es);
    p.n_vec = vec_count(V, es);
    chunk_geometry(p.n_vec, p.n_split, p.chunk_vecs);
    p.n_sub = sub_chunks(V, es);
    draw_geometry(p.n_sub, p.d_split, p.d_subs_per_chunk);
    Carver cv;
    p.off_counters = cv.take<Counters>(1);
    p.off_part = cv.take<WarpPartial>((size_t)rows * p.n_split * kWarps);
    p.off_rowstat = cv.take<RowStat>((size_t)rows);
    p.off_nuc = cv.take<NucleusCut>((size_t)rows);
    p.off_top = cv.take<TopSet>((size_t)rows);
    p.off_draws = cv.take<DrawItem>((size_t)rows);
    p.off_subs = cv.take<float>((size_t)rows * p.n_sub);
    const size_t capx = (size_t)(rows < (long long)kExactCap ? rows : (long long)kExactCap);
    p.off_exact = cv.take<ExactItem>(capx);
    p.off_xpart = cv.take<double>(capx * 2 * kExactSplit * 3);
    p.off_xdraw = cv.take<ExactDraw>(capx);
    p.x_split = exact_groups(p.n_sub);
    p.off_xsubs = cv.take<float4>(capx * p.n_sub);
    p.off_xnorm = cv.take<float4>(capx * p.x_split);
    p.off_xunc_n = cv.take<int>(capx);
    p.off_xunc = cv.take<int>(capx * kExactUncCap);
    p.bytes = cv.off + 256;
    sp.bytes = p.bytes;
    return sp;
}

template <int ES>
static sv_status launch_sample(const SamplePlan &sp, const SampleArgs &in, const float *top_p,
                               const int32_t *top_k, int F, int B, void *ws, cudaStream_t stream) {
    const VerifyPlan &pl = sp.v;
    DeviceInfo di;
    if (!device_info(di)) return SV_ERR_CUDA;
    char *w = static_cast<char *>(ws);
    Counters *counters = reinterpret_cast<Counters *>(w + pl.off_counters);
    WarpPartial *part = reinterpret_cast<WarpPartial *>(w + pl.off_part);
    RowStat *rowstat = reinterpret_cast<RowStat *>(w + pl.off_rowstat);
    SampleArgs a = in;
    StatsArgs sa;
    sa.set[0] = a.rows;
    sa.set[1] = a.rows;
    sa.n_sets = 1;
    sa.V = a.V;
    sa.temperature = a.temperature;
    sa.n_split = pl.n_split;
    sa.chunk_vecs = pl.chunk_vecs;
    sa.n_rows0 = pl.n_rows0;
    sa.n_units = pl.n_rows0 * pl.n_split;
    sa.part = part;
    sa.counters = counters;
    sa.stats = a.stats;
    sa.wait_limit = kWaitLimitCycles;
    {
        const sv_status st = launch_stats<ES>(sa, di, stream);
        if (st != SV_OK) return st;
    }
    NucleusCut *nuc = nullptr;
    TopSet *top = nullptr;
    if (top_p || top_k) {
        nuc = reinterpret_cast<NucleusCut *>(w + pl.off_nuc);
        const sv_status st = launch_nucleus<ES>(a.rows, a.rows, pl.n_rows0, 0, a.V, a.temperature, top_p, top_k,
                                                part, pl.n_split, nuc, a.stats, stream);
        if (st != SV_OK) return st;
    }
    if (a.sag_on) {
        top = reinterpret_cast<TopSet *>(w + pl.off_top);
        const sv_status st = launch_topset<ES>(a.rows, 0, B, a.n_rows, a.V, a.temperature, F, a.C, part, pl.n_split,
                                               nuc, top, a.stats, di, stream);
        if (st != SV_OK) return st;
    }
    a.part = part;
    a.n_split = pl.n_split;
    a.rowstat = rowstat;
    a.nuc = nuc;
    a.top = top;
    a.draws = reinterpret_cast<DrawItem *>(w + pl.off_draws);
    a.counters = counters;
    const long long total = pl.n_rows0;
    k_sample_items<<<(unsigned)div_up(total * 32, kThreads), kThreads, 0, stream>>>(a, total);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    DrawArgs da;
    da.items = a.draws;
    da.counters = counters;
    da.V = a.V;
    da.n_vec = pl.n_vec;
    da.n_sub = pl.n_sub;
    da.n_split = pl.d_split;
    da.subs_per_chunk = pl.d_subs_per_chunk;
    da.subs = reinterpret_cast<float *>(w + pl.off_subs);
    da.exact = reinterpret_cast<ExactItem *>(w + pl.off_exact);
    da.exact_unc = reinterpret_cast<int *>(w + pl.off_xunc_n);
    da.stats = a.stats;
    da.wait_limit = kWaitLimitCycles;
    {
        const sv_status st = launch_draws<ES>(da, total, di, stream);
        if (st != SV_OK) return st;
    }
    ExactArgs xa{};
    xa.tgt = a.rows;
    xa.drf = a.rows;
    xa.K = 0;
    xa.V = a.V;
    xa.temperature = a.temperature;
    xa.nuc = nuc;
    xa.top = top;
    xa.rowstat = rowstat;
    xa.n_rows0 = pl.n_rows0;
    xa.draws = a.draws;
    xa.items = da.exact;
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
    xa.max_slots = 2;
    xa.stats = a.stats;
    xa.wait_limit = kWaitLimitCycles;
    return launch_exact<ES>(xa, di, stream);
}

}  // namespace sv

using namespace sv;

extern "C" size_t sv_saguaro_sample_workspace_size(int B, int n_rows, int V) {
    if (B < 1 || n_rows < 1 || V < 1) return 0;
    const SamplePlan a = plan_sample(B, n_rows, V, 4), b = plan_sample(B, n_rows, V, 2);
    return a.bytes > b.bytes ? a.bytes : b.bytes;
}

extern "C" sv_status sv_saguaro_sample(const void *draft_logits, int64_t row_pitch, int rows_per_seq, sv_dtype dtype,
                                       int B, int n_rows, int V, const float *temperature, const float *top_p,
                                       const int32_t *top_k, int F, float C, const double *uniforms, int32_t *tokens, double *debug,
                                       sv_stats *stats, void *workspace, size_t workspace_bytes,
                                       sv_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (B < 1 || n_rows < 1 || V < 1 || rows_per_seq < n_rows) return SV_ERR_INVALID_ARG;
    if (!rows_ok(draft_logits, row_pitch, V, dtype)) return SV_ERR_INVALID_ARG;
    if (temperature == nullptr || uniforms == nullptr || tokens == nullptr) return SV_ERR_INVALID_ARG;
    if (F < 0 || !(C >= 0.0f && C <= 1.0f)) return SV_ERR_INVALID_ARG;
    const int es = elem_size(dtype);
    const SamplePlan sp = plan_sample(B, n_rows, V, es);
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < sp.bytes) return SV_ERR_WORKSPACE;
    if (!on_current_device(stream, draft_logits)) return SV_ERR_INVALID_ARG;
    if (stats && cudaMemsetAsync(stats, 0, sizeof(sv_stats), stream) != cudaSuccess) return SV_ERR_CUDA;
    SampleArgs a{};
    a.rows = {static_cast<const char *>(draft_logits), row_pitch * es, rows_per_seq, n_rows, 0};
    a.n_rows = n_rows;
    a.V = V;
    a.temperature = temperature;
    a.C = C;
    a.sag_on = (F > 0 && C != 1.0f) ? 1 : 0;
    a.uniforms = uniforms;
    a.tokens = tokens;
    a.debug = debug;
    a.stats = stats;
    if (es == 4) return launch_sample<4>(sp, a, top_p, top_k, F, B, workspace, stream);
    return launch_sample<2>(sp, a, top_p, top_k, F, B, workspace, stream);
}
