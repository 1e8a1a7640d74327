// sv_accept.cuh — the accept test of one position and the draw parameters of one row, shared by
// the per-sequence accept kernel and the lazy (position-by-position) verification kernel.
//
// ["Speculative Speculative Decoding" notes, §2.2 ③; "Accelerating LLM Decoding with Speculative
//  Sampling (2023)" notes, §3 (accept s with probability min(1, q(s)/p(s))), §6 (filters first)]
#pragma once

#include "sv_device.cuh"
#include "sv_stats.cuh"

namespace sv {

struct AcceptArgs {
    RowSet tgt, drf;
    int K, V;
    const float *temperature;
    const float *top_p;
    int sag_on;
    float sag_C;
    const int32_t *tokens;
    const double *uniforms;
    int32_t *accept_len;
    int32_t *out_tokens;
    double *debug;
    sv_stats *stats;
    const WarpPartial *part;
    int n_split;
    long long n_rows0;
    RowStat *rowstat;
    const NucleusCut *nuc;
    const TopSet *top;
    DrawItem *draws;
    ExactItem *exact;
    int *exact_unc;
    Counters *counters;
    int draw_from_q;        // 1: a rejection draws from q itself, not from (q - p)+
};

// Draw parameters of one row, float32 only: inv_s = 1 / (S * nucleus mass * Saguaro normaliser).
__device__ __forceinline__ DrawRow draw_row(const char *row, float T, const RowStat &rs, const NucleusCut *nc,
                                            const TopSet *ts, float sag_C) {
    DrawRow d;
    d.row = row;
    log2e_over(T, d.c_hi, d.c_lo);
    d.rf = (float)rs.r;
    float norm = rs.s_hi;
    double err = (double)rs.err + 4.0 * kU32;   // S_lo dropped, products, reciprocal
    d.cut_x = -INFINITY;
    d.cut_id = 0x7FFFFFFF;
    if (nc) {
        d.cut_x = nc->cut_x;
        d.cut_id = nc->cut_id;
        norm = __fmul_rn(norm, nc->mass_f);
        err += 2.0 * (double)rs.err + kU32 + 1e-12;   // the kept mass is a ratio of two sums of the same pass
    }
    d.top_x = INFINITY;
    d.top_id = -1;
    d.sc_d = 1.0f;
    if (ts) {
        d.top_x = ts->top_x;
        d.top_id = ts->top_id;
        d.sc_d = sag_C;
        norm = __fmul_rn(norm, ts->z_f);
        err += (double)ts->z_err_f + kU32;
    }
    d.inv_s = __frcp_rn(norm);
    d.k_lo = __fmul_rn(__fmul_rn(d.c_lo, (float)kLn2), d.inv_s);
    d.pad = 0;
    // mean |y| under the normalised weights: at most the row's, divided by the kept mass and z
    d.ay = __fdiv_ru(rs.ay * (1.0f + 0x1p-20f), __fdiv_rn(norm, rs.s_hi) * (1.0f - 0x1p-20f));
    d.norm_err = err;
    return d;
}

// Outcome of the accept test of position j (0-based) of sequence b.
struct AcceptOutcome {
    bool acc, amb, near;
    bool keep_q, keep_p, in_top;
    float ratio;
};

// Float32 accept test with a certified margin: ratio = q(s)/p(s) = 2^(y_q - y_p) (S_p m_p z)/
// (S_q m_q C_s) with y = x c - r, S the row sums, m the nucleus masses, z the Saguaro normaliser
// and C_s = C on the top-F set; y_q - y_p is formed in float-float.  The exponential, the
// products and the quotient carry kEx2RelErr + 8u, the row sums err_q + err_p, the masses
// 2(err_q + err_p), the normaliser z_err; u < ratio is certain outside ratio (1 -+ delta).
// xt, xd: the target and draft logits of token s at position j (loaded by the caller).
__device__ __forceinline__ AcceptOutcome accept_test_x(const AcceptArgs &a, int b, int j, int s, double u_acc,
                                                       float c_hi, float c_lo, const RowStat &rq, const RowStat &rp,
                                                       float xt, float xd) {
    bool acc = false, amb = false, near = false;
    bool keep_q = false, keep_p = false, in_top = false;
    float ratio = NAN;
    const long long rid_t = (long long)b * (a.K + 1) + j;
    const long long rid_d = a.n_rows0 + (long long)b * a.K + j;
    float num = rp.s_hi, den = rq.s_hi;
    float delta = (float)(kEx2RelErr + 8.0 * kU32 + 1e-10) + rq.err + rp.err;
    keep_q = xt != -INFINITY;
    keep_p = xd != -INFINITY;
    if (a.nuc) {
        const NucleusCut &nq = a.nuc[rid_t], &np = a.nuc[rid_d];
        keep_q = keep_q && (xt > nq.cut_x || (xt == nq.cut_x && s <= nq.cut_id));
        keep_p = keep_p && (xd > np.cut_x || (xd == np.cut_x && s <= np.cut_id));
        num = __fmul_rn(num, np.mass_f);
        den = __fmul_rn(den, nq.mass_f);
        delta += 2.0f * (rq.err + rp.err) + (float)(2.0 * kU32);
    }
    if (a.sag_on && a.top) {
        const TopSet &t = a.top[rid_d];
        in_top = xd > t.top_x || (xd == t.top_x && s <= t.top_id);
        num = __fmul_rn(num, t.z_f);
        if (in_top) den = __fmul_rn(den, a.sag_C);
        delta += t.z_err_f + (float)kU32;
    }
    if (!keep_p) {
        ratio = keep_q ? INFINITY : 0.0f;
    } else if (!keep_q) {
        ratio = 0.0f;
    } else {
        const ff c = {c_hi, c_lo};
        const ff yq = ff_affine(xt, c, {(float)rq.r, 0.f});
        const ff yp = ff_affine(xd, c, {(float)rp.r, 0.f});
        const ff dy = ff_sub(yq, yp);
        delta += 1e-12f * (fabsf(yq.hi) + fabsf(yp.hi));   // float-float y and c
        // dy is about log2(den / num) wherever the test is close, i.e. up to +-log2 V and more:
        // split it into an integer n and a fraction f in [-1/2, 1/2] (exact), so the fast
        // exponential sees only f, inside the range its error bound was measured on, and 2^n
        // scales the quotient exactly (to inf or 0 where it leaves the float32 range).
        const float n = rintf(fminf(fmaxf(dy.hi, -512.0f), 512.0f));
        const float f = __fsub_rn(dy.hi, n);
        const float e = ex2_fast(f) * fmaf(dy.lo, (float)kLn2, 1.0f);
        ratio = ldexpf(e * __fdiv_rn(num, den), (int)n);
    }
    delta *= 1.01f;
    const float rr = fminf(1.0f, ratio);
    const float lo = fminf(1.0f, ratio * (1.0f - delta));
    const float hi = fminf(1.0f, ratio * (1.0f + delta));
    const float u = __double2float_rn(u_acc);
    // u is rounded to float32 (relative error 2^-24, inside delta's 8u); a ratio that
    // underflowed is decided by the float-float tier unless u is clearly above it
    acc = u < rr;
    amb = (u >= lo && u < hi) || (keep_q && keep_p && ratio < 0x1p-100f && u < 0x1p-90f);
    near = fabsf(u - rr) < 1e-6f;
    return {acc, amb, near, keep_q, keep_p, in_top, ratio};
}

// The accept test of position j with the two logits of s loaded here.
template <int ES>
__device__ __forceinline__ AcceptOutcome accept_test(const AcceptArgs &a, int b, int j, int s, double u_acc,
                                                     float c_hi, float c_lo, const RowStat &rq, const RowStat &rp) {
    const RowSet &ts = a.tgt, &ds = a.drf;
    const char *trow = ts.base + ((long long)b * ts.rows_per_seq + j) * ts.pitch_bytes;
    const char *drow = ds.base + ((long long)b * ds.rows_per_seq + j) * ds.pitch_bytes;
    return accept_test_x(a, b, j, s, u_acc, c_hi, c_lo, rq, rp, load_elem<ES>(trow, s), load_elem<ES>(drow, s));
}

}  // namespace sv
