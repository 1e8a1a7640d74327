// sv_exact.cuh — float-float tier for decisions the float32 tier could not certify.
//
// One cooperative kernel works through the queue in phases separated by bounded grid
// barriers:
//   A. (only for queued sequences whose accept tests were too close to call) exact row sums
//      S = sum_v 2^(x_v c - r) of every row of those sequences;
//   B. per item: the accept tests of such sequences again in float64 with the exact sums; then
//      the parameters of the item's draw;
//   C. one float-float pass over the draw rows: per row the normaliser (sum of its weights),
//      per 32-vector sub-chunk the sums of q- and p-weights over tokens whose residual
//      q - p is certainly positive (a sign test with the float32 normalisers and their error
//      bound), and a list of the few tokens whose sign the test cannot settle;
//   D. per item: exact normalisers, sub-chunk masses W = A_q/S_q - A_p/S_p plus the exact
//      residuals of the listed tokens, a float64 scan, the sub-chunk holding u R, a
//      float-float rescan, t*.
// Results agree with a float64 evaluation except when u R lies within 2e-11 relative of a
// boundary; such decisions are counted in sv_stats.unresolved.  Element exponentials use
// Tang's table method in float-float (sv_device.cuh); in phase C the weights of bf16 rows
// without filters come from per-block tables of two exact factors (see tab_w); no float64
// work runs per element.
#pragma once

#include "sv_device.cuh"
#include "sv_exp2_table.h"
#include "sv_draw.cuh"
#include "sv_host.h"

namespace sv {

constexpr int kExactUncCap = 1024;   // uncertain-sign tokens listed per item

struct ExactRow {
    const char *row;
    ff c;
    float rf;
    float cut_x;
    int cut_id;
    float top_x;
    int top_id;
    float sc;       // factor on the top-F set (1: none)
    int valid;
    int filt;       // a nucleus cut or a top-F set is in use
};

struct ExactDraw {
    ExactRow q, p;
    float inv_q, inv_p;     // float32 normalisers for the sign test
    float sign_tol;         // relative tolerance of the sign test
    int has_p;
    double u;
    int *out;
    double *dbg_r;
};

struct ExactArgs {
    // verification context (for sequences whose accept tests are redone)
    RowSet tgt, drf;
    int K, V;
    const float *temperature;
    const int32_t *tokens;
    const double *uniforms;
    int32_t *accept_len;
    int32_t *out_tokens;
    double *debug;
    float sag_C;
    int sag_on;
    const NucleusCut *nuc;   // per candidate row, or nullptr
    const TopSet *top;       // per candidate row, or nullptr
    const RowStat *rowstat;
    long long n_rows0;
    // queue
    const DrawItem *draws;
    const ExactItem *items;
    Counters *counters;
    // workspace
    double *xpart;           // [item][slot][kExactSplit][3]   (phase A)
    ExactDraw *xdraw;        // [item]
    float4 *xsubs;           // [item][n_sub]: A_q (ff), A_p (ff)
    float4 *xnorm;           // [item][xsplit]: S_q (ff), S_p (ff) per unit
    int *xunc_n;             // [item]
    int *xunc;               // [item][kExactUncCap]
    int n_vec, n_sub, xsplit, max_slots;
    sv_stats *stats;
    long long wait_limit;
    int draw_from_q;         // 1: a rejection draws from q itself, not from (q - p)+
};


// Bounded grid-wide barrier for a cooperative launch.  The counter is zeroed earlier in the call.
__device__ __forceinline__ bool grid_barrier(unsigned *ctr, unsigned &target, long long limit) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        target += gridDim.x;
        __threadfence();
        atomicAdd(ctr, 1u);
        const long long t0 = clock64();
        int ok = 1;
        while (true) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
            if (v >= target) break;
            if (clock64() - t0 > limit) {
                ok = 0;
                break;
            }
            __nanosleep(64);
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

__device__ __forceinline__ bool in_cut(float x, int v, float cx, int cid) { return x > cx || (x == cx && v <= cid); }

__device__ __forceinline__ ExactRow exact_row_from_draw(const DrawRow &r) {
    ExactRow e;
    e.row = r.row;
    e.c = {r.c_hi, r.c_lo};
    e.rf = r.rf;
    e.cut_x = r.cut_x;
    e.cut_id = r.cut_id;
    e.top_x = r.top_x;
    e.top_id = r.top_id;
    e.sc = r.sc_d;
    e.valid = r.row != nullptr;
    e.filt = (e.cut_x > -INFINITY) || (e.top_id >= 0);
    return e;
}

// Row `slot` (0..K target, K+1..2K draft) of a queued sequence.
__device__ __forceinline__ ExactRow seq_row(const ExactArgs &a, int b, int slot) {
    const int K = a.K;
    ExactRow e;
    const bool is_t = slot <= K;
    const int j = is_t ? slot : slot - K - 1;
    const long long rid = is_t ? (long long)b * (K + 1) + j : a.n_rows0 + (long long)b * K + j;
    const RowSet &rs = is_t ? a.tgt : a.drf;
    e.row = rs.base + ((long long)b * rs.rows_per_seq + j) * rs.pitch_bytes;
    log2e_over(a.temperature[b], e.c.hi, e.c.lo);
    e.rf = (float)a.rowstat[rid].r;
    e.cut_x = -INFINITY;
    e.cut_id = 0x7FFFFFFF;
    e.top_x = INFINITY;
    e.top_id = -1;
    e.sc = 1.0f;
    if (a.nuc) {
        e.cut_x = a.nuc[rid].cut_x;
        e.cut_id = a.nuc[rid].cut_id;
    }
    if (!is_t && a.top && a.sag_on) {
        e.top_x = a.top[rid].top_x;
        e.top_id = a.top[rid].top_id;
        e.sc = a.sag_C;
    }
    e.valid = 1;
    e.filt = (e.cut_x > -INFINITY) || (e.top_id >= 0);
    return e;
}

// Weight of token v in a row: keep(v) * 2^(x c - r) * (sc on the top-F set), float-float.
__device__ __forceinline__ ff exact_w(const ExactRow &r, float x, int v, const float2 *tab) {
    if (x == -INFINITY || (r.filt && !in_cut(x, v, r.cut_x, r.cut_id))) return {0.f, 0.f};
    ff e = ff_exp2_xc(x, r.c, (int)r.rf, tab);
    if (r.filt && in_cut(x, v, r.top_x, r.top_id)) e = ff_mul(e, {r.sc, 0.f});
    return e;
}

__device__ __forceinline__ ExactDraw exact_draw_from(const DrawItem &d) {
    ExactDraw xd;
    xd.q = exact_row_from_draw(d.q);
    xd.inv_q = d.q.inv_s;
    xd.has_p = d.has_p;
    xd.p = d.has_p ? exact_row_from_draw(d.p) : xd.q;
    xd.inv_p = d.has_p ? d.p.inv_s : 0.f;
    xd.sign_tol = (float)(1.05 * (d.q.norm_err + (d.has_p ? d.p.norm_err : 0.0)) + 4.0 * kU32);
    xd.u = d.u;
    xd.out = d.out;
    xd.dbg_r = d.dbg_r;
    return xd;
}

// Element k of a 16-byte vector, for loops that are not unrolled (no local-memory array).
template <int ES>
__device__ __forceinline__ float elem_of(const uint4 &w, int k) {
    const int j = ES == 4 ? k : (k >> 1);
    const unsigned b = j == 0 ? w.x : j == 1 ? w.y : j == 2 ? w.z : w.w;
    if (ES == 4) return __uint_as_float(b);
    return (k & 1) ? bf16_hi(b) : bf16_lo(b);
}

template <int ES>
__device__ __forceinline__ void load_vec(const char *row, int vi, float (&x)[16 / ES]) {
    const uint4 w = __ldg(reinterpret_cast<const uint4 *>(row) + vi);
    unpack<ES>(w, x);
}

// Adds b to the float-float sum s without renormalising: TwoSum of the high parts, then the
// rounding error and b's low part into s.lo (the cascaded summation of Ogita, Rump and Oishi,
// "Accurate sum and dot product", 2005).  For n nonnegative terms the result is within about
// n^2 u^2 of the sum, far below the tier's 2e-11 tolerance for the n <= 8 terms a lane adds
// per sub-chunk.
__device__ __forceinline__ void ff_acc(ff &s, ff b) {
    const float t = __fadd_rn(s.hi, b.hi);
    const float bb = __fsub_rn(t, s.hi);
    const float e = __fadd_rn(__fsub_rn(s.hi, __fsub_rn(t, bb)), __fsub_rn(b.hi, bb));
    s.lo = __fadd_rn(s.lo, __fadd_rn(e, b.lo));
    s.hi = t;
}

// 2^(x c - r) in float-float for rows whose r satisfies |r| < 2^19, without branches: the same
// steps as ff_exp2_xc, with results below 2^-140 (and -inf logits) selected to zero at the end.
// For such rows every token with x c_hi - r >= -140 has |x c_hi| < 2^20, so ff_exp2_xc's
// wide-argument path is never needed; arguments that select zero are replaced by 0 first, so
// every intermediate stays finite.
__device__ __forceinline__ ff ff_exp2_nf(float x, ff c, int r, float rf, const float2 *tab) {
    const ff p0 = two_prod(x, c.hi);
    const bool zero = !(__fsub_rn(p0.hi, rf) >= -140.0f);
    const float xs = zero ? 0.f : x;
    const float ph = zero ? 0.f : p0.hi, pl = zero ? 0.f : p0.lo;
    const float yl = __fmaf_rn(xs, c.lo, pl);
    const float kf = rintf(__fmul_rn(ph, 256.0f));
    const int k = static_cast<int>(kf);
    const float rh = __fsub_rn(ph, __fmul_rn(kf, 0.00390625f));   // exact
    const float L_HI = 0.693147182464599609375f;
    const float L_LO = -1.9046542999577520e-09f;
    ff s = two_prod(rh, L_HI);
    s.lo = __fmaf_rn(rh, L_LO, __fmaf_rn(yl, L_HI, s.lo));
    s = fast_two_sum(s.hi, s.lo);
    const ff s2 = two_prod(s.hi, s.hi);
    const float half_s2 = __fmul_rn(0.5f, s2.hi);
    const float cubic = __fmul_rn(__fmul_rn(s2.hi, s.hi), __fmaf_rn(s.hi, 1.0f / 24.0f, 1.0f / 6.0f));
    const float small = __fadd_rn(__fmaf_rn(s.hi, s.lo, __fmul_rn(0.5f, s2.lo)), cubic);
    ff t = fast_two_sum(s.hi, half_s2);
    t.lo = __fadd_rn(t.lo, __fadd_rn(s.lo, small));
    const int j = k & 255;
    const int n = (k >> 8) - r;
    const float2 T = tab[j];
    const ff P = two_prod(T.x, t.hi);
    ff e = fast_two_sum(T.x, P.hi);
    const float tail = __fadd_rn(T.y, __fadd_rn(P.lo, __fmaf_rn(T.x, t.lo, __fmul_rn(T.y, t.hi))));
    e = fast_two_sum(e.hi, __fadd_rn(e.lo, tail));
    const float sc = zero ? 0.f : pow2i(n);
    return {__fmul_rn(e.hi, sc), __fmul_rn(e.lo, sc)};
}

// Factored weights for bf16 rows.  A bf16 logit is x = s 2^(E-127) (1 + (8 m_h + m_l)/128),
// m_h its top three and m_l its low four mantissa bits, so 2^(x c - r) = 2^(v1 c - r) 2^(v2 c)
// exactly, with v1 = s 2^(E-127) (1 + m_h/8) and v2 = s 2^(E-127) m_l/128 both floats.  A
// table of the first factor per row over (s, E, m_h) and one of the second per temperature
// over (s, E, m_l), each entry a float-float exponential, turn a token's weight into two
// shared-memory loads and a float-float product: the relative error stays a few times 2^-44,
// like the direct exponential's.  Exponents outside the tables, entries whose factor could
// leave [2^-100, 2^64] (first) or [2^-32, 2^32] (second), and -inf or zero logits take the
// direct exponential, so a product stays in [2^-132, 2^96]: it cannot overflow, and below
// 2^-126, where the direct exponential flushes to zero, the two differ by less than 2^-126
// of a row sum that is at least 1/2.
constexpr int kTabE0 = 118;                   // |x| in [2^-9, 2^7)
constexpr int kTabNE = 16;
constexpr int kTabGroups = 2 * kTabNE;        // (s, E)
constexpr int kTab1 = kTabGroups * 8;         // first-factor entries
constexpr int kTab2 = kTabGroups * 16;        // second-factor entries
constexpr int kTabSlots = 2;                  // items whose tables one block holds
static_assert(kTab1 == kThreads, "one first-factor entry per thread");

__device__ __forceinline__ float tab_scale(int g) {   // s 2^(E-127) of group g
    const float p = __int_as_float((kTabE0 + (g & (kTabNE - 1))) << 23);
    return g >= kTabNE ? -p : p;
}

__device__ __forceinline__ float2 tab_first(float v, const ExactRow &r, const float2 *tab) {
    const float y = __fmaf_rn(v, r.c.hi, -r.rf);
    if (!(y >= -100.0f && y <= 64.0f)) return make_float2(__int_as_float(0x7FC00000), 0.f);
    const ff e = ff_exp2_nf(v, r.c, (int)r.rf, r.rf, tab);
    return make_float2(e.hi, e.lo);
}

__device__ __forceinline__ float2 tab_second(float v, ff c, const float2 *tab) {
    if (!(fabsf(__fmul_rn(v, c.hi)) <= 32.0f)) return make_float2(__int_as_float(0x7FC00000), 0.f);
    const ff e = ff_exp2_nf(v, c, 0, 0.f, tab);
    return make_float2(e.hi, e.lo);
}

// Rows without filters whose r satisfies |r| < 2^19: the unrolled row pass applies.
__device__ __forceinline__ bool nf_rows(const ExactDraw &d) {
    return !d.q.filt && !(d.has_p && d.p.filt) && fabsf(d.q.rf) < 0x1p19f && (!d.has_p || fabsf(d.p.rf) < 0x1p19f);
}

__device__ __forceinline__ bool same_c(const ExactDraw &d) {
    return !d.has_p || (d.q.c.hi == d.p.c.hi && d.q.c.lo == d.p.c.lo);
}

// Tables of one item, by the whole block: t1q / t1p per row, t2q for q's temperature (and
// t2p for p's when it differs).
__device__ __forceinline__ void build_tables(const ExactDraw &d, float2 *t1q, float2 *t1p, float2 *t2q, float2 *t2p,
                                             const float2 *tab, int tid) {
    const float v1 = tab_scale(tid >> 3) * (1.0f + 0.125f * (float)(tid & 7));
    t1q[tid] = tab_first(v1, d.q, tab);
    if (d.has_p) t1p[tid] = tab_first(v1, d.p, tab);
    const bool same = same_c(d);
    for (int j = tid; j < kTab2; j += kThreads) {
        const float v2 = tab_scale(j >> 4) * (0.0078125f * (float)(j & 15));
        t2q[j] = tab_second(v2, d.q.c, tab);
        if (!same) t2p[j] = tab_second(v2, d.p.c, tab);
    }
}

// Weight of the bf16 logit with bit pattern b (16 bits) from the tables; ok is false where
// the tables cannot give it.
__device__ __forceinline__ ff tab_w(uint32_t b, const float2 *t1, const float2 *t2, bool &ok) {
    const int e = (int)((b >> 7) & 0xFFu) - kTabE0;
    const bool inr = (unsigned)e < (unsigned)kTabNE;
    const int g = (inr ? e : 0) + (int)(b >> 15) * kTabNE;
    const float2 f1 = t1[g * 8 + (int)((b >> 4) & 7u)];
    const float2 f2 = t2[g * 16 + (int)(b & 15u)];
    const float h = __fmul_rn(f1.x, f2.x);
    const float l = __fmaf_rn(f1.x, f2.y, __fmaf_rn(f1.y, f2.x, __fmaf_rn(f1.x, f2.x, -h)));
    ok = inr && h >= 0.f;
    return {h, l};
}

// The direct exponential for the few tokens the tables leave out, kept out of line so that
// the unrolled token loop stays small.
static __device__ __noinline__ ff exp2_direct(float x, ff c, int r, float rf, const float2 *tab) {
    return ff_exp2_nf(x, c, r, rf, tab);
}

// Phase C of the float-float tier on vector sub-chunks [g0, g1) of item i when neither row has
// a filter and both rows' r satisfy |r| < 2^19: the same sums as the general path (sign-split
// A_q, A_p per sub-chunk, tokens of uncertain sign listed; the normaliser partial of the whole
// run in unit g0's slot and zero in the others, which phase D adds up all the same), with the
// sub-chunk's tokens unrolled without branches and the next sub-chunk's logits loaded ahead.
template <int ES, bool HAS_P, bool TAB>
__device__ __forceinline__ void exact_run_nf(const ExactArgs &a, const ExactDraw &d, int i, int g0, int g1, int lane,
                                             const float2 *tab, float4 *xs, const float2 *t1q, const float2 *t2q,
                                             const float2 *t1p, const float2 *t2p) {
    static_assert(!TAB || ES == 2, "tables for bf16 rows");
    static_assert(kExactGroup == 1, "one sub-chunk per unit");
    constexpr int EPV = 16 / ES;
    const uint4 *qrow = reinterpret_cast<const uint4 *>(d.q.row);
    const uint4 *prow = reinterpret_cast<const uint4 *>(d.p.row);
    const int rq = (int)d.q.rf, rp = (int)d.p.rf;
    auto load = [&](int sb, uint4 &wq, uint4 &wp) {
        const int vi = sb * 32 + lane;
        wq = wp = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);   // -inf: weight 0
        if (ES == 4) wq = wp = make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
        if (sb < g1 && vi < a.n_vec) {
            wq = __ldg(qrow + vi);
            if (HAS_P) wp = __ldg(prow + vi);
        }
    };
    uint4 nq_w, np_w;
    load(g0, nq_w, np_w);
    // the normaliser partials of the whole run, reduced across the warp once at its end
    ff nq_run = {0.f, 0.f}, np_run = {0.f, 0.f};
    for (int sb = g0; sb < g1; ++sb) {
        const uint4 wq = nq_w, wp = np_w;
        load(sb + 1, nq_w, np_w);
        const int vi = sb * 32 + lane;
        ff nq = {0.f, 0.f}, np = {0.f, 0.f}, aq = {0.f, 0.f}, ap = {0.f, 0.f};
        unsigned unc = 0;   // tokens of this lane whose sign the float32 test cannot settle
        // four tokens at a time (a loop of two for bf16), which keeps the unrolled code small
        // enough for the instruction cache
#pragma unroll 1
        for (int h = 0; h < EPV / 4; ++h) {
            float xq[4], xp[4];
            if constexpr (ES == 2) {
                const uint32_t q0 = h ? wq.z : wq.x, q1 = h ? wq.w : wq.y;
                const uint32_t p0 = h ? wp.z : wp.x, p1 = h ? wp.w : wp.y;
                xq[0] = bf16_lo(q0); xq[1] = bf16_hi(q0); xq[2] = bf16_lo(q1); xq[3] = bf16_hi(q1);
                xp[0] = bf16_lo(p0); xp[1] = bf16_hi(p0); xp[2] = bf16_lo(p1); xp[3] = bf16_hi(p1);
            } else {
                xq[0] = __uint_as_float(wq.x); xq[1] = __uint_as_float(wq.y);
                xq[2] = __uint_as_float(wq.z); xq[3] = __uint_as_float(wq.w);
                xp[0] = __uint_as_float(wp.x); xp[1] = __uint_as_float(wp.y);
                xp[2] = __uint_as_float(wp.z); xp[3] = __uint_as_float(wp.w);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                ff eq, ep;
                if constexpr (TAB) {
                    const uint32_t wq2 = (k < 2) ? (h ? wq.z : wq.x) : (h ? wq.w : wq.y);
                    const uint32_t bq = (k & 1) ? (wq2 >> 16) : (wq2 & 0xFFFFu);
                    bool ok;
                    eq = tab_w(bq, t1q, t2q, ok);
                    if (!ok) eq = exp2_direct(xq[k], d.q.c, rq, d.q.rf, tab);
                    if (HAS_P) {
                        const uint32_t wp2 = (k < 2) ? (h ? wp.z : wp.x) : (h ? wp.w : wp.y);
                        const uint32_t bp = (k & 1) ? (wp2 >> 16) : (wp2 & 0xFFFFu);
                        ep = tab_w(bp, t1p, t2p, ok);
                        if (!ok) ep = exp2_direct(xp[k], d.p.c, rp, d.p.rf, tab);
                    }
                } else {
                    eq = ff_exp2_nf(xq[k], d.q.c, rq, d.q.rf, tab);
                    if (HAS_P) ep = ff_exp2_nf(xp[k], d.p.c, rp, d.p.rf, tab);
                }
                ff_acc(nq, eq);
                if (HAS_P) {
                    ff_acc(np, ep);
                    const float wq1 = eq.hi * d.inv_q, wp1 = ep.hi * d.inv_p;
                    const float diff = wq1 - wp1, tol = d.sign_tol * (wq1 + wp1);
                    const bool pos = diff > tol;
                    unc |= (!pos && diff >= -tol && wq1 > 0.f) ? (1u << (4 * h + k)) : 0u;
                    ff_acc(aq, pos ? eq : ff{0.f, 0.f});
                    ff_acc(ap, pos ? ep : ff{0.f, 0.f});
                } else {
                    ff_acc(aq, eq);
                }
            }
        }
        if (HAS_P && __any_sync(0xFFFFFFFFu, unc != 0)) {
            for (int k = 0; k < EPV; ++k) {
                if (unc & (1u << k)) {
                    const int slot = atomicAdd(&a.xunc_n[i], 1);
                    if (slot < kExactUncCap) a.xunc[(size_t)i * kExactUncCap + slot] = vi * EPV + k;
                }
            }
        }
        nq_run = ff_add(nq_run, fast_two_sum(nq.hi, nq.lo));
        np_run = ff_add(np_run, fast_two_sum(np.hi, np.lo));
        aq = warp_sum_ff(fast_two_sum(aq.hi, aq.lo));
        ap = warp_sum_ff(fast_two_sum(ap.hi, ap.lo));
        if (lane == 0) {
            xs[sb] = make_float4(aq.hi, aq.lo, ap.hi, ap.lo);
            if (sb > g0) a.xnorm[(size_t)i * a.xsplit + sb] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    nq_run = warp_sum_ff(nq_run);
    np_run = warp_sum_ff(np_run);
    if (lane == 0) a.xnorm[(size_t)i * a.xsplit + g0] = make_float4(nq_run.hi, nq_run.lo, np_run.hi, np_run.lo);
}

template <int ES>
__global__ void __launch_bounds__(kThreads, 3) k_exact(const ExactArgs a) {
    constexpr int EPV = 16 / ES;
    pdl_trigger();   // the stream's next kernel may be scheduled; it waits for this one to finish
    __shared__ float2 tab[256];
    __shared__ double s_red[3][kWarps];
    const int n_items = min(*reinterpret_cast<volatile int *>(&a.counters->n_exact), kExactCap);
    if (n_items == 0) return;   // uniform across the grid
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    {
        tab[tid] = kExp2Table[tid];
    }
    int acc_here = 0;
    for (int i = tid; i < n_items; i += kThreads) acc_here |= a.items[i].draw < 0;
    const bool any_accept = __syncthreads_or(acc_here) != 0;
    unsigned bar_target = 0;
    const int n_vsub = a.n_sub - 1;
    const int n_vec = a.n_vec;

    // ---- phase A: exact sums of every row of sequences whose accept tests are redone ------
    if (any_accept) {
        const int chunk_vecs = (n_vec + kExactSplit - 1) / kExactSplit;
        const long long units = (long long)n_items * a.max_slots * kExactSplit;
        for (long long u = blockIdx.x; u < units; u += gridDim.x) {
            const int i = (int)(u / ((long long)a.max_slots * kExactSplit));
            const int rem = (int)(u - (long long)i * a.max_slots * kExactSplit);
            const int slot = rem / kExactSplit, c = rem - slot * kExactSplit;
            const ExactItem it = a.items[i];
            if (it.draw >= 0 || slot > 2 * a.K) continue;   // block-uniform
            const ExactRow r = seq_row(a, it.seq, slot);
            ff sa = {0.f, 0.f}, sk = {0.f, 0.f}, skd = {0.f, 0.f};
            const int v0 = min(c * chunk_vecs, n_vec), v1 = min(v0 + chunk_vecs, n_vec);
            auto add = [&](float x, int v) {
                if (x == -INFINITY) return;
                const ff e = ff_exp2_xc(x, r.c, (int)r.rf, tab);
                sa = ff_add(sa, e);
                if (in_cut(x, v, r.cut_x, r.cut_id)) {
                    sk = ff_add(sk, e);
                    if (in_cut(x, v, r.top_x, r.top_id)) skd = ff_add(skd, e);
                }
            };
            for (int vi = v0 + tid; vi < v1; vi += kThreads) {
                float x[EPV];
                load_vec<ES>(r.row, vi, x);
#pragma unroll
                for (int k = 0; k < EPV; ++k) add(x[k], vi * EPV + k);
            }
            if (c == kExactSplit - 1) {
                const int t0 = n_vec * EPV;
                if (t0 + tid < a.V) add(load_elem<ES>(r.row, t0 + tid), t0 + tid);
            }
            const ff wa = warp_sum_ff(sa), wk = warp_sum_ff(sk), wd = warp_sum_ff(skd);
            if (lane == 0) {
                s_red[0][warp] = ff_to_double(wa);
                s_red[1][warp] = ff_to_double(wk);
                s_red[2][warp] = ff_to_double(wd);
            }
            __syncthreads();
            if (tid < 3) {
                double t = 0.0;
                for (int w = 0; w < kWarps; ++w) t += s_red[tid][w];
                a.xpart[(((size_t)i * a.max_slots + slot) * kExactSplit + c) * 3 + tid] = t;
            }
            __syncthreads();
        }
        if (!grid_barrier(&a.counters->barrier, bar_target, a.wait_limit)) {
            if (tid == 0 && blockIdx.x == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
            return;
        }
    }

    // ---- phase B: the accept tests of queued sequences, then their draw parameters -----------
    const int gwarp = blockIdx.x * kWarps + warp, nwarps = gridDim.x * kWarps;
    for (int i = gwarp; i < n_items && any_accept; i += nwarps) {
        const ExactItem it = a.items[i];
        ExactDraw xd;
        if (it.draw >= 0) {
            continue;   // draw items take their parameters in phase C
        } else {
            const int b = it.seq, K = a.K;
            const double cc = 1.4426950408889634074 / (double)a.temperature[b];
            auto sums = [&](int slot, double &sa, double &sk, double &sd) {
                sa = sk = sd = 0.0;
                for (int c = lane; c < kExactSplit; c += 32) {
                    const double *p = a.xpart + (((size_t)i * a.max_slots + slot) * kExactSplit + c) * 3;
                    sa += p[0];
                    sk += p[1];
                    sd += p[2];
                }
                sa = warp_sum_d(sa);
                sk = warp_sum_d(sk);
                sd = warp_sum_d(sd);
            };
            int k = K, unresolved = 0;
            for (int j = 0; j < K; ++j) {
                const ExactRow rt = seq_row(a, b, j), rd = seq_row(a, b, K + 1 + j);
                double ta, tk, tdd, da, dk, dd;
                sums(j, ta, tk, tdd);
                sums(K + 1 + j, da, dk, dd);
                const int s = a.tokens[(size_t)b * K + j];
                const float xt = load_elem<ES>(rt.row, s), xdr = load_elem<ES>(rd.row, s);
                const double lq = in_cut(xt, s, rt.cut_x, rt.cut_id) ? ((double)xt * cc - (double)rt.rf - log2(tk))
                                                                      : -INFINITY;
                const double zp = a.sag_on ? dk - (1.0 - (double)a.sag_C) * dd : dk;
                double lp = -INFINITY;
                if (in_cut(xdr, s, rd.cut_x, rd.cut_id)) {
                    lp = (double)xdr * cc - (double)rd.rf - log2(zp);
                    if (a.sag_on && in_cut(xdr, s, rd.top_x, rd.top_id)) lp += log2((double)a.sag_C);
                }
                const double ratio = (lp == -INFINITY) ? (lq == -INFINITY ? 0.0 : INFINITY) : exp2(lq - lp);
                const double r = fmin(1.0, ratio);
                const double uj = a.uniforms[(size_t)b * (K + 1) + j];
                if (fabs(uj - r) < 1e-12) unresolved = 1;
                if (a.debug && lane == 0) {
                    double *dbg = a.debug + ((size_t)b * (K + 1) + j) * SV_DEBUG_FIELDS;
                    dbg[SV_DBG_LSE_Q] = ((double)rt.rf + log2(ta)) * kLn2;
                    dbg[SV_DBG_LSE_P] = ((double)rd.rf + log2(da)) * kLn2;
                    dbg[SV_DBG_Q_S] = exp2(lq);
                    dbg[SV_DBG_P_S] = exp2(lp);
                    dbg[SV_DBG_RATIO] = ratio;
                    dbg[SV_DBG_MASS_Q] = tk / ta;
                    dbg[SV_DBG_MASS_P] = dk / da;
                }
                if (!(uj < r)) {
                    k = j;
                    break;
                }
            }
            if (lane == 0) {
                if (unresolved) stats_add(a.stats, &a.stats->unresolved, 1);
                a.accept_len[b] = k;
                for (int j = 0; j <= K; ++j)
                    a.out_tokens[(size_t)b * (K + 1) + j] = j < k ? a.tokens[(size_t)b * K + j] : -1;
            }
            double sa, sk, sd;
            sums(k, sa, sk, sd);
            xd.q = seq_row(a, b, k);
            xd.inv_q = (float)(1.0 / sk);
            xd.has_p = k < K && !a.draw_from_q;
            xd.p = xd.q;
            xd.inv_p = 0.f;
            if (xd.has_p) {
                double pa, pk, pd;
                sums(K + 1 + k, pa, pk, pd);
                xd.p = seq_row(a, b, K + 1 + k);
                xd.inv_p = (float)(1.0 / (a.sag_on ? pk - (1.0 - (double)a.sag_C) * pd : pk));
            }
            xd.sign_tol = (float)(8.0 * kU32);
            xd.u = a.uniforms[(size_t)b * (K + 1) + K];
            xd.out = a.out_tokens + (size_t)b * (K + 1) + k;
            xd.dbg_r = a.debug ? a.debug + (size_t)b * (K + 1) * SV_DEBUG_FIELDS + SV_DBG_R : nullptr;
        }
        if (lane == 0) a.xdraw[i] = xd;
    }
    if (any_accept && !grid_barrier(&a.counters->barrier, bar_target, a.wait_limit)) {
        if (tid == 0 && blockIdx.x == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
        return;
    }

    // ---- phase C: one float-float pass over the draw rows, one warp per unit ----------------
    // A unit is kExactGroup sub-chunks of one item (or its scalar tail): per sub-chunk the
    // sign-split sums (A_q, A_p), per unit the two normaliser partials.  No block barriers.
    // Each warp takes a contiguous range of units, so that an item's parameters are read once
    // per run of its units and the next sub-chunk's logits are in flight while one is summed.
    const int n_grp = a.xsplit;   // exact_groups(n_sub)
    const long long units_c = (long long)n_items * n_grp;
    // balanced ranges: every warp gets floor or ceil of units_c / nwarps
    const long long uc0 = units_c * gwarp / nwarps, uc1 = units_c * (gwarp + 1) / nwarps;
    // bf16: the factored-weight tables of the (at most kTabSlots) items this block's units touch
    __shared__ float2 s_t1[kTabSlots][2][kTab1];
    __shared__ float2 s_t2[kTabSlots][2][kTab2];
    int tab_i0 = 0, tab_n = 0;   // block-uniform
    if constexpr (ES == 2) {
        const long long ub0 = units_c * (blockIdx.x * kWarps) / nwarps;
        const long long ub1 = units_c * ((blockIdx.x + 1) * kWarps) / nwarps;
        if (ub1 > ub0 && (ub1 - 1) / n_grp - ub0 / n_grp < kTabSlots) {
            tab_i0 = (int)(ub0 / n_grp);
            tab_n = (int)((ub1 - 1) / n_grp) - tab_i0 + 1;
            for (int ts = 0; ts < tab_n; ++ts) {
                const ExactItem itm = a.items[tab_i0 + ts];
                const ExactDraw d = itm.draw >= 0 ? exact_draw_from(a.draws[itm.draw]) : a.xdraw[tab_i0 + ts];
                if (nf_rows(d))
                    build_tables(d, s_t1[ts][0], s_t1[ts][1], s_t2[ts][0], s_t2[ts][1], tab, tid);
            }
            __syncthreads();
        }
    }
    for (long long u = uc0; u < uc1;) {
        const int i = (int)(u / n_grp);
        const long long u_end = min(uc1, (long long)(i + 1) * n_grp);
        int g = (int)(u - (long long)i * n_grp);
        const int g_end = (int)(u_end - (long long)i * n_grp);
        u = u_end;
        const ExactItem itm = a.items[i];
        const ExactDraw d = itm.draw >= 0 ? exact_draw_from(a.draws[itm.draw]) : a.xdraw[i];
        float4 *xs = a.xsubs + (size_t)i * a.n_sub;
        const int ts = i - tab_i0;
        if (kExactGroup == 1 && nf_rows(d) && (ES == 4 || (ts >= 0 && ts < tab_n))) {
            // rows without filters: the vector sub-chunks on the unrolled path (bf16: from the tables)
            const int gv_end = min(g_end, n_grp - 1);
            if (g < gv_end) {
                if constexpr (ES == 2) {
                    const float2 *t2p = same_c(d) ? s_t2[ts][0] : s_t2[ts][1];
                    if (d.has_p)
                        exact_run_nf<ES, true, true>(a, d, i, g, gv_end, lane, tab, xs, s_t1[ts][0], s_t2[ts][0],
                                                     s_t1[ts][1], t2p);
                    else
                        exact_run_nf<ES, false, true>(a, d, i, g, gv_end, lane, tab, xs, s_t1[ts][0], s_t2[ts][0],
                                                      nullptr, nullptr);
                } else {
                    if (d.has_p) exact_run_nf<ES, true, false>(a, d, i, g, gv_end, lane, tab, xs, nullptr, nullptr,
                                                              nullptr, nullptr);
                    else exact_run_nf<ES, false, false>(a, d, i, g, gv_end, lane, tab, xs, nullptr, nullptr, nullptr,
                                                        nullptr);
                }
                g = gv_end;
            }
        }
        for (; g < g_end; ++g) {
            ff nq = {0.f, 0.f}, np = {0.f, 0.f};
            // one token: its contributions to the normalisers and, by the sign test, to (A_q, A_p)
            auto token = [&](float xq, float xp, int v, ff &aq, ff &ap) {
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
                    const int slot = atomicAdd(&a.xunc_n[i], 1);
                    if (slot < kExactUncCap) a.xunc[(size_t)i * kExactUncCap + slot] = v;
                }
            };
            if (g < n_grp - 1) {
                const int sb0 = g * kExactGroup, sb1 = min(sb0 + kExactGroup, n_vsub);
                for (int sb = sb0; sb < sb1; ++sb) {
                    const int vi = sb * 32 + lane;
                    ff aq = {0.f, 0.f}, ap = {0.f, 0.f};
                    if (vi < n_vec) {
                        const uint4 wq = __ldg(reinterpret_cast<const uint4 *>(d.q.row) + vi);
                        const uint4 wp = d.has_p ? __ldg(reinterpret_cast<const uint4 *>(d.p.row) + vi) : wq;
#pragma unroll 1
                        for (int k = 0; k < EPV; ++k)
                            token(elem_of<ES>(wq, k), elem_of<ES>(wp, k), vi * EPV + k, aq, ap);
                    }
                    aq = warp_sum_ff(aq);
                    ap = warp_sum_ff(ap);
                    if (lane == 0) xs[sb] = make_float4(aq.hi, aq.lo, ap.hi, ap.lo);
                }
            } else {
                const int t = n_vec * EPV + lane;
                ff aq = {0.f, 0.f}, ap = {0.f, 0.f};
                if (t < a.V) {
                    const float xq = load_elem<ES>(d.q.row, t);
                    token(xq, d.has_p ? load_elem<ES>(d.p.row, t) : xq, t, aq, ap);
                }
                aq = warp_sum_ff(aq);
                ap = warp_sum_ff(ap);
                if (lane == 0) xs[n_vsub] = make_float4(aq.hi, aq.lo, ap.hi, ap.lo);
            }
            nq = warp_sum_ff(nq);
            np = warp_sum_ff(np);
            if (lane == 0) a.xnorm[(size_t)i * n_grp + g] = make_float4(nq.hi, nq.lo, np.hi, np.lo);
        }
    }
    if (!grid_barrier(&a.counters->barrier, bar_target, a.wait_limit)) {
        if (tid == 0 && blockIdx.x == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
        return;
    }

    // ---- phase D: one block per item: exact sub-chunk masses, block scan, t* ----------------
    // Float-float throughout (the float64 pipe of this GPU would set the latency of the block).
    __shared__ float2 s_unc_w[kExactUncCap];
    __shared__ int s_unc_sub[kExactUncCap];
    __shared__ float2 s_scan[kWarps];
    __shared__ float4 s_norm[kWarps];
    __shared__ int s_sub;
    __shared__ float2 s_pre;
    __shared__ int s_last;
    for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
        const ExactItem itm = a.items[i];
        const ExactDraw d = itm.draw >= 0 ? exact_draw_from(a.draws[itm.draw]) : a.xdraw[i];
        const float4 *xs = a.xsubs + (size_t)i * a.n_sub;
        // this thread's contiguous range of sub-chunks; its first two masses are loaded now so
        // that the loads overlap the normaliser reduction
        const int per = (a.n_sub + kThreads - 1) / kThreads;
        const int s0 = min(tid * per, a.n_sub), s1 = min(s0 + per, a.n_sub);
        const float4 xs0 = s0 < s1 ? xs[s0] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 xs1 = s0 + 1 < s1 ? xs[s0 + 1] : make_float4(0.f, 0.f, 0.f, 0.f);
        // normalisers
        ff sq = {0.f, 0.f}, sp = {0.f, 0.f};
        for (int k = tid; k < n_grp; k += kThreads) {
            const float4 v = a.xnorm[(size_t)i * n_grp + k];
            sq = ff_add(sq, {v.x, v.y});
            sp = ff_add(sp, {v.z, v.w});
        }
        sq = warp_sum_ff(sq);
        sp = warp_sum_ff(sp);
        if (lane == 0) s_norm[warp] = make_float4(sq.hi, sq.lo, sp.hi, sp.lo);
        if (tid == 0) {
            s_sub = -1;
            s_last = -1;
        }
        __syncthreads();
        sq = {0.f, 0.f};
        sp = {0.f, 0.f};
        for (int w = 0; w < kWarps; ++w) {
            const float4 v = s_norm[w];
            sq = ff_add(sq, {v.x, v.y});
            sp = ff_add(sp, {v.z, v.w});
        }
        const ff iq = ff_recip(sq), ip = d.has_p ? ff_recip(sp) : ff{0.f, 0.f};
        // exact residuals of the tokens whose sign the float32 test could not settle
        const int n_unc_all = a.xunc_n[i];
        const int n_unc = min(n_unc_all, kExactUncCap);
        if (tid == 0 && n_unc_all > kExactUncCap) stats_add(a.stats, &a.stats->unresolved, 1);
        for (int k = tid; k < n_unc; k += kThreads) {
            const int t = a.xunc[(size_t)i * kExactUncCap + k];
            const float xq = load_elem<ES>(d.q.row, t), xp = load_elem<ES>(d.p.row, t);
            const ff w = ff_sub(ff_mul(exact_w(d.q, xq, t, tab), iq), ff_mul(exact_w(d.p, xp, t, tab), ip));
            s_unc_w[k] = w.hi > 0.f ? make_float2(w.hi, w.lo) : make_float2(0.f, 0.f);
            s_unc_sub[k] = t < n_vec * EPV ? t / (32 * EPV) : n_vsub;
        }
        __syncthreads();
        auto W = [&](int s) {
            const float4 v = s == s0 ? xs0 : s == s0 + 1 ? xs1 : xs[s];
            ff w = ff_sub(ff_mul({v.x, v.y}, iq), ff_mul({v.z, v.w}, ip));
            for (int k = 0; k < n_unc; ++k)
                if (s_unc_sub[k] == s) w = ff_add(w, {s_unc_w[k].x, s_unc_w[k].y});
            return w;
        };
        // block scan of the per-thread range sums
        ff mine = {0.f, 0.f};
        int last_pos = -1;
        for (int s = s0; s < s1; ++s) {
            const ff w = W(s);
            mine = ff_add(mine, w);
            if (w.hi > 0.f) last_pos = s;
        }
        atomicMax(&s_last, last_pos);
        ff incl, excl, R;
        block_scan_ff(mine, incl, excl, R, s_scan);
        const float u_hi = __double2float_rn(d.u);
        const float u_lo = __double2float_rn(d.u - (double)u_hi);
        const ff thr = ff_mul(R, {u_hi, u_lo});
        if (mine.hi > 0.f && ff_diff(thr, excl) >= 0.f && ff_diff(thr, incl) < 0.f) {
            ff run = excl;
            for (int s = s0; s < s1; ++s) {
                const ff w = W(s);
                const ff nx = ff_add(run, w);
                if (w.hi > 0.f && ff_diff(thr, nx) < 0.f) {
                    s_sub = s;
                    s_pre = make_float2(run.hi, run.lo);
                    break;
                }
                run = nx;
            }
        }
        __syncthreads();
        int sub = s_sub;
        ff pre = {s_pre.x, s_pre.y};
        if (sub < 0) {
            // u R at or past the last boundary through rounding: the last positive sub-chunk
            sub = s_last;
            if (tid == 0 && sub >= 0) {
                ff p = {0.f, 0.f};
                for (int s = 0; s < sub; ++s) p = ff_add(p, W(s));
                s_pre = make_float2(p.hi, p.lo);
            }
            __syncthreads();
            pre = {s_pre.x, s_pre.y};
        }
        __syncthreads();   // every thread has read s_sub / s_pre before they are reused below
        // rescan the sub-chunk holding u R: one token per thread, block scan in float-float
        if (sub >= 0) {
            const int t0 = sub < n_vsub ? sub * 32 * EPV : n_vec * EPV;
            const int ntok = sub < n_vsub ? min(32 * EPV, (n_vec - sub * 32) * EPV) : a.V - n_vec * EPV;
            ff wt = {0.f, 0.f};
            if (tid < ntok) {
                const int t = t0 + tid;
                const float xq = load_elem<ES>(d.q.row, t);
                const ff q = ff_mul(exact_w(d.q, xq, t, tab), iq);
                if (d.has_p) {
                    const float xp = load_elem<ES>(d.p.row, t);
                    const ff w = ff_sub(q, ff_mul(exact_w(d.p, xp, t, tab), ip));
                    wt = w.hi > 0.f ? w : ff{0.f, 0.f};
                } else {
                    wt = q;
                }
            }
            ff inc = wt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float h = __shfl_up_sync(0xFFFFFFFFu, inc.hi, o);
                const float l = __shfl_up_sync(0xFFFFFFFFu, inc.lo, o);
                if (lane >= o) inc = ff_add(inc, {h, l});
            }
            if (lane == 31) s_norm[warp] = make_float4(inc.hi, inc.lo, 0.f, 0.f);
            if (tid == 0) {
                s_sub = 0x7FFFFFFF;   // first hit token (thread index)
                s_last = -1;          // last positive token
            }
            __syncthreads();
            ff base = pre;
            for (int w = 0; w < warp; ++w) base = ff_add(base, {s_norm[w].x, s_norm[w].y});
            const ff c_hit = ff_add(base, inc), c_prev = ff_add(base, ff_sub(inc, wt));
            if (wt.hi > 0.f) {
                atomicMax(&s_last, tid);
                if (ff_diff(thr, c_hit) < 0.f) atomicMin(&s_sub, tid);
            }
            __syncthreads();
            const int hit = s_sub;
            // float-float sums over ~V / 256 sub-chunks: worst-case relative error below 2e-11,
            // plus the exponents' low-word rounding, about 2^-48 |x c| <= 2^-48 (|r| + 126)
            const float tol = (2e-11f + 0x1p-46f * (fabsf(d.q.rf) + fabsf(d.p.rf) + 252.0f)) * R.hi;
            if (hit != 0x7FFFFFFF) {
                if (tid == hit) {
                    *d.out = t0 + tid;
                    if (ff_diff(thr, c_prev) < tol || ff_diff(c_hit, thr) < tol)
                        stats_add(a.stats, &a.stats->unresolved, 1);
                }
            } else if (tid == 0) {
                // rounding left u R past the sub-chunk: its last positive token, unresolved
                *d.out = s_last >= 0 ? t0 + s_last : -1;
                stats_add(a.stats, &a.stats->unresolved, 1);
            }
        } else if (tid == 0) {
            *d.out = -1;
        }
        if (tid == 0 && d.dbg_r) *d.dbg_r = (double)R.hi + (double)R.lo;
        __syncthreads();
    }
}

// The float-float tier runs as one cooperative grid (all co-resident blocks) so that its phases
// can be separated by grid barriers.  With an empty queue every block returns at once.
template <int ES>
sv_status launch_exact(const ExactArgs &xa, const DeviceInfo &di, cudaStream_t stream) {
    static_assert(sizeof(ExactArgs) < 4096, "kernel parameter block");
    const int occ = prepare_kernel((const void *)k_exact<ES>, kThreads, 0);
    if (occ < 1) return SV_ERR_CUDA;
    void *args[] = {const_cast<ExactArgs *>(&xa)};
    const cudaError_t e = cudaLaunchCooperativeKernel((const void *)k_exact<ES>, dim3(di.sms * occ), dim3(kThreads),
                                                      args, 0, stream);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace sv
