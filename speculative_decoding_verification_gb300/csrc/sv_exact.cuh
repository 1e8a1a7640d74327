// sv_exact.cuh — float-float tier for decisions the float32 tier could not certify.
//
// One cooperative kernel handles the queue in four phases separated by grid barriers:
//   1. exact row sums  S_all = sum_v 2^(x_v c - r), S_keep (nucleus tokens), S_keepD (and in the
//      Saguaro top-F set), float-float per element (Tang's table method), float64 across threads;
//   2. per item: exact normalisers; for a queued sequence, its accept tests again in float64;
//      then the parameters of its draw;
//   3. exact sub-chunk sums of the draw weights (float-float per element);
//   4. per item: float64 scan, the sub-chunk that holds u R, a float-float rescan, t*.
// Results agree with a float64 evaluation except when u R lies within ~1e-12 relative of a
// boundary; such decisions are counted in sv_stats.unresolved.
#pragma once

#include "sv_device.cuh"
#include "sv_draw.cuh"

namespace sv {

struct ExactRow {
    const char *row;
    ff c;
    float rf;
    float cut_x;
    int cut_id;
    float top_x;
    int top_id;
    int valid;
};

struct ExactDraw {
    ExactRow q, p;
    ff inv_q, inv_p;
    float sc_q, sc_p;       // Saguaro factor C on each row's top-F set (1: none)
    int has_p;
    double u;
    int *out;
    double *dbg_r;
    int active;
    int pad;
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
    double *xpart;           // [item][slot][chunk][3]
    ExactDraw *xdraw;        // [item]
    double *xsubs;           // [item][n_sub]
    int n_vec, n_sub, xsplit, max_slots;
    sv_stats *stats;
    long long wait_limit;
};

__device__ __forceinline__ ff ff_mul(ff a, ff b) {
    ff p = two_prod(a.hi, b.hi);
    p.lo = __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, p.lo));
    return fast_two_sum(p.hi, p.lo);
}

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

__device__ __forceinline__ ExactRow exact_row_from_draw(const DrawRow &r) {
    ExactRow e;
    e.row = r.row;
    e.c = {r.c_hi, r.c_lo};
    e.rf = r.rf;
    e.cut_x = r.cut_x;
    e.cut_id = r.cut_id;
    e.top_x = r.top_x;
    e.top_id = r.top_id;
    e.valid = r.row != nullptr;
    return e;
}

// Row `slot` of exact item i.
__device__ __forceinline__ ExactRow exact_row(const ExactArgs &a, int i, int slot, long long *rid_out) {
    const ExactItem it = a.items[i];
    ExactRow e;
    e.valid = 0;
    *rid_out = -1;
    if (it.draw >= 0) {
        const DrawItem &d = a.draws[it.draw];
        if (slot == 0) e = exact_row_from_draw(d.q);
        else if (slot == 1 && d.has_p) e = exact_row_from_draw(d.p);
        return e;
    }
    const int K = a.K, b = it.seq;
    if (slot > 2 * K) return e;
    const bool is_t = slot <= K;
    const int j = is_t ? slot : slot - K - 1;
    const long long rid = is_t ? (long long)b * (K + 1) + j : a.n_rows0 + (long long)b * K + j;
    const RowSet &rs = is_t ? a.tgt : a.drf;
    const double c = 1.4426950408889634074 / (double)a.temperature[b];
    e.row = rs.base + ((long long)b * rs.rows_per_seq + j) * rs.pitch_bytes;
    e.c = ff_from_double(c);
    e.rf = (float)a.rowstat[rid].r;
    e.cut_x = -INFINITY;
    e.cut_id = 0x7FFFFFFF;
    e.top_x = INFINITY;
    e.top_id = -1;
    if (a.nuc) {
        e.cut_x = a.nuc[rid].cut_x;
        e.cut_id = a.nuc[rid].cut_id;
    }
    if (!is_t && a.top && a.sag_on) {
        e.top_x = a.top[rid].top_x;
        e.top_id = a.top[rid].top_id;
    }
    e.valid = 1;
    *rid_out = rid;
    return e;
}

__device__ __forceinline__ bool in_cut(float x, int v, float cx, int cid) { return x > cx || (x == cx && v <= cid); }

template <int ES>
__device__ __forceinline__ void exact_elem_sums(const ExactRow &r, float x, int v, const float2 *tab, ff &sa, ff &sk,
                                                ff &skd) {
    const ff y = ff_affine(x, r.c, {r.rf, 0.f});
    const ff e = ff_exp2(y.hi, y.lo, tab);
    sa = ff_add(sa, e);
    if (in_cut(x, v, r.cut_x, r.cut_id)) {
        sk = ff_add(sk, e);
        if (in_cut(x, v, r.top_x, r.top_id)) skd = ff_add(skd, e);
    }
}

// Exact draw weight of token v.
__device__ __forceinline__ ff exact_weight(const ExactDraw &d, float xq, float xp, int v, const float2 *tab) {
    ff q = {0.f, 0.f};
    if (in_cut(xq, v, d.q.cut_x, d.q.cut_id)) {
        const ff y = ff_affine(xq, d.q.c, {d.q.rf, 0.f});
        q = ff_mul(ff_exp2(y.hi, y.lo, tab), d.inv_q);
        if (in_cut(xq, v, d.q.top_x, d.q.top_id)) q = ff_mul(q, {d.sc_q, 0.f});
    }
    if (!d.has_p) return q;
    ff p = {0.f, 0.f};
    if (in_cut(xp, v, d.p.cut_x, d.p.cut_id)) {
        const ff y = ff_affine(xp, d.p.c, {d.p.rf, 0.f});
        p = ff_mul(ff_exp2(y.hi, y.lo, tab), d.inv_p);
        if (in_cut(xp, v, d.p.top_x, d.p.top_id)) p = ff_mul(p, {d.sc_p, 0.f});
    }
    ff w = ff_sub(q, p);
    if (!(w.hi > 0.f)) w = {0.f, 0.f};
    return w;
}

template <int ES>
__global__ void __launch_bounds__(kThreads) k_exact(const ExactArgs a) {
    constexpr int EPV = 16 / ES;
    __shared__ float2 tab[256];
    __shared__ double s_red[3][kWarps];
    const int n_items = min(*reinterpret_cast<volatile int *>(&a.counters->n_exact), kExactCap);
    if (n_items == 0) return;   // uniform across the grid
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    {
        const double t = exp2((double)tid / 256.0);
        const float hi = (float)t;
        tab[tid] = make_float2(hi, (float)(t - (double)hi));
    }
    __syncthreads();
    unsigned bar_target = 0;
    const int n_vsub = a.n_sub - 1;
    const int n_vec = a.n_vec;
    const int chunk_vecs = (n_vec + a.xsplit - 1) / a.xsplit;

    // ---- phase 1: exact row sums ---------------------------------------------------------
    const long long units1 = (long long)n_items * a.max_slots * a.xsplit;
    for (long long u = blockIdx.x; u < units1; u += gridDim.x) {
        const int i = (int)(u / ((long long)a.max_slots * a.xsplit));
        const int rem = (int)(u - (long long)i * a.max_slots * a.xsplit);
        const int slot = rem / a.xsplit, c = rem - slot * a.xsplit;
        long long rid;
        const ExactRow r = exact_row(a, i, slot, &rid);
        if (!r.valid) continue;   // block-uniform
        ff sa = {0.f, 0.f}, sk = {0.f, 0.f}, skd = {0.f, 0.f};
        const int v0 = min(c * chunk_vecs, n_vec), v1 = min(v0 + chunk_vecs, n_vec);
        for (int vi = v0 + tid; vi < v1; vi += kThreads) {
            const uint4 w = __ldg(reinterpret_cast<const uint4 *>(r.row) + vi);
            float x[EPV];
            unpack<ES>(w, x);
#pragma unroll
            for (int k = 0; k < EPV; ++k) exact_elem_sums<ES>(r, x[k], vi * EPV + k, tab, sa, sk, skd);
        }
        if (c == a.xsplit - 1) {
            const int t0 = n_vec * EPV;
            if (t0 + tid < a.V) exact_elem_sums<ES>(r, load_elem<ES>(r.row, t0 + tid), t0 + tid, tab, sa, sk, skd);
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
            a.xpart[(((size_t)i * a.max_slots + slot) * a.xsplit + c) * 3 + tid] = t;
        }
        __syncthreads();
    }
    if (!grid_barrier(&a.counters->barrier, bar_target, a.wait_limit)) {
        if (tid == 0 && blockIdx.x == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
        return;
    }

    // ---- phase 2: exact normalisers, accept tests of queued sequences, draw set-up ----------
    const int gwarp = blockIdx.x * kWarps + warp, nwarps = gridDim.x * kWarps;
    for (int i = gwarp; i < n_items; i += nwarps) {
        const ExactItem it = a.items[i];
        auto sums = [&](int slot, double &sa, double &sk, double &sd) {
            sa = sk = sd = 0.0;
            for (int c = lane; c < a.xsplit; c += 32) {
                const double *p = a.xpart + (((size_t)i * a.max_slots + slot) * a.xsplit + c) * 3;
                sa += p[0];
                sk += p[1];
                sd += p[2];
            }
            sa = warp_sum_d(sa);
            sk = warp_sum_d(sk);
            sd = warp_sum_d(sd);
        };
        ExactDraw xd;
        xd.active = 1;
        if (it.draw >= 0) {
            const DrawItem &d = a.draws[it.draw];
            double sa, sk, sd;
            sums(0, sa, sk, sd);
            xd.q = exact_row_from_draw(d.q);
            xd.sc_q = d.q.sc_d;
            xd.sc_p = d.p.sc_d;
            xd.inv_q = ff_from_double(1.0 / (sk - (1.0 - (double)d.q.sc_d) * sd));
            xd.has_p = d.has_p;
            if (d.has_p) {
                double pa, pk, pd;
                sums(1, pa, pk, pd);
                xd.p = exact_row_from_draw(d.p);
                xd.inv_p = ff_from_double(1.0 / (pk - (1.0 - (double)d.p.sc_d) * pd));
            }
            xd.u = d.u;
            xd.out = d.out;
            xd.dbg_r = d.dbg_r;
        } else {
            // redo the accept tests of sequence b in float64 with exact normalisers
            const int b = it.seq, K = a.K;
            const float T = a.temperature[b];
            const double cc = 1.4426950408889634074 / (double)T;
            int k = K;
            int unresolved = 0;
            for (int j = 0; j < K; ++j) {
                long long rid_t, rid_d;
                const ExactRow rt = exact_row(a, i, j, &rid_t);
                const ExactRow rd = exact_row(a, i, K + 1 + j, &rid_d);
                double ta, tk, tdd, da, dk, dd;
                sums(j, ta, tk, tdd);
                sums(K + 1 + j, da, dk, dd);
                const int s = a.tokens[(size_t)b * K + j];
                const float xt = load_elem<ES>(rt.row, s), xdr = load_elem<ES>(rd.row, s);
                double lq = in_cut(xt, s, rt.cut_x, rt.cut_id) ? ((double)xt * cc - (double)rt.rf - log2(tk)) : -INFINITY;
                double zp = a.sag_on ? dk - (1.0 - (double)a.sag_C) * dd : dk;
                double lp = -INFINITY;
                if (in_cut(xdr, s, rd.cut_x, rd.cut_id)) {
                    lp = (double)xdr * cc - (double)rd.rf - log2(zp);
                    if (a.sag_on && in_cut(xdr, s, rd.top_x, rd.top_id)) lp += log2((double)a.sag_C);
                }
                double ratio;
                if (lp == -INFINITY) ratio = lq == -INFINITY ? 0.0 : INFINITY;
                else ratio = exp2(lq - lp);
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
            long long rq, rp;
            double sa, sk, sd;
            sums(k, sa, sk, sd);
            xd.q = exact_row(a, i, k, &rq);
            xd.q.top_x = INFINITY;
            xd.inv_q = ff_from_double(1.0 / sk);
            xd.has_p = k < K;
            xd.sc_q = 1.0f;
            xd.sc_p = a.sag_on ? a.sag_C : 1.0f;
            if (k < K) {
                double pa, pk, pd;
                sums(K + 1 + k, pa, pk, pd);
                xd.p = exact_row(a, i, K + 1 + k, &rp);
                xd.inv_p = ff_from_double(1.0 / (a.sag_on ? pk - (1.0 - (double)a.sag_C) * pd : pk));
            }
            xd.u = a.uniforms[(size_t)b * (K + 1) + K];
            xd.out = a.out_tokens + (size_t)b * (K + 1) + k;
            xd.dbg_r = a.debug ? a.debug + (size_t)b * (K + 1) * SV_DEBUG_FIELDS + SV_DBG_R : nullptr;
        }
        if (lane == 0) a.xdraw[i] = xd;
    }
    if (!grid_barrier(&a.counters->barrier, bar_target, a.wait_limit)) {
        if (tid == 0 && blockIdx.x == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
        return;
    }

    // ---- phase 3: exact sub-chunk sums of the draw weights ----------------------------------
    const int subs_per_chunk = (n_vsub + a.xsplit - 1) / a.xsplit;
    const long long units3 = (long long)n_items * a.xsplit;
    for (long long u = blockIdx.x; u < units3; u += gridDim.x) {
        const int i = (int)(u / a.xsplit), c = (int)(u - (long long)i * a.xsplit);
        const ExactDraw &d = a.xdraw[i];
        double *xs = a.xsubs + (size_t)i * a.n_sub;
        const int sb0 = min(c * subs_per_chunk, n_vsub), sb1 = min(sb0 + subs_per_chunk, n_vsub);
        for (int sb = sb0 + warp; sb < sb1; sb += kWarps) {
            const int vi = sb * 32 + lane;
            ff acc = {0.f, 0.f};
            if (vi < n_vec) {
                const uint4 wq = __ldg(reinterpret_cast<const uint4 *>(d.q.row) + vi);
                const uint4 wp = d.has_p ? __ldg(reinterpret_cast<const uint4 *>(d.p.row) + vi) : wq;
                float xq[EPV], xp[EPV];
                unpack<ES>(wq, xq);
                unpack<ES>(wp, xp);
#pragma unroll
                for (int k = 0; k < EPV; ++k) acc = ff_add(acc, exact_weight(d, xq[k], xp[k], vi * EPV + k, tab));
            }
            acc = warp_sum_ff(acc);
            if (lane == 0) xs[sb] = ff_to_double(acc);
        }
        if (c == a.xsplit - 1 && warp == 0) {
            const int t = n_vec * EPV + lane;
            ff acc = {0.f, 0.f};
            if (t < a.V) {
                const float xq = load_elem<ES>(d.q.row, t);
                const float xp = d.has_p ? load_elem<ES>(d.p.row, t) : xq;
                acc = exact_weight(d, xq, xp, t, tab);
            }
            acc = warp_sum_ff(acc);
            if (lane == 0) xs[n_vsub] = ff_to_double(acc);
        }
    }
    if (!grid_barrier(&a.counters->barrier, bar_target, a.wait_limit)) {
        if (tid == 0 && blockIdx.x == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
        return;
    }

    // ---- phase 4: scan and pick t* (one warp per item) --------------------------------------
    for (int i = gwarp; i < n_items; i += nwarps) {
        const ExactDraw &d = a.xdraw[i];
        const double *xs = a.xsubs + (size_t)i * a.n_sub;
        // warp scan over sub-chunks in blocks of 32
        double R = 0.0;
        for (int s = lane; s < a.n_sub; s += 32) R += xs[s];
        R = warp_sum_d(R);
        const double thr = d.u * R;
        int sub = -1;
        double pre = 0.0, run = 0.0;
        int last_pos = -1;
        double last_pre = 0.0;
        for (int base = 0; base < a.n_sub && sub < 0; base += 32) {
            const int s = base + lane;
            const double v = s < a.n_sub ? xs[s] : 0.0;
            double inc = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                if (lane >= o) inc += t;
            }
            const double ex = run + inc - v;
            const bool hit = v > 0.0 && thr < ex + v;
            const unsigned m = __ballot_sync(0xFFFFFFFFu, hit);
            const unsigned mp = __ballot_sync(0xFFFFFFFFu, v > 0.0);
            if (mp) {
                const int src = 31 - __clz(mp);
                last_pos = base + src;
                last_pre = __shfl_sync(0xFFFFFFFFu, ex, src);
            }
            if (m) {
                const int src = __ffs(m) - 1;
                sub = base + src;
                pre = __shfl_sync(0xFFFFFFFFu, ex, src);
            }
            run = __shfl_sync(0xFFFFFFFFu, run + inc, 31);
        }
        if (sub < 0) {
            sub = last_pos;
            pre = last_pre;
        }
        int tstar = -1;
        if (sub >= 0) {
            ff wv[EPV];
            int ntok = 0, tok0;
            if (sub < n_vsub) {
                const int vi = sub * 32 + lane;
                tok0 = vi * EPV;
                if (vi < n_vec) {
                    ntok = EPV;
                    const uint4 wq = __ldg(reinterpret_cast<const uint4 *>(d.q.row) + vi);
                    const uint4 wp = d.has_p ? __ldg(reinterpret_cast<const uint4 *>(d.p.row) + vi) : wq;
                    float xq[EPV], xp[EPV];
                    unpack<ES>(wq, xq);
                    unpack<ES>(wp, xp);
#pragma unroll
                    for (int k = 0; k < EPV; ++k) wv[k] = exact_weight(d, xq[k], xp[k], tok0 + k, tab);
                }
            } else {
                tok0 = n_vec * EPV + lane;
                if (tok0 < a.V) {
                    ntok = 1;
                    const float xq = load_elem<ES>(d.q.row, tok0);
                    const float xp = d.has_p ? load_elem<ES>(d.p.row, tok0) : xq;
                    wv[0] = exact_weight(d, xq, xp, tok0, tab);
                }
            }
            double lt = 0.0;
            for (int k = 0; k < ntok; ++k) lt += ff_to_double(wv[k]);
            double inc = lt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                if (lane >= o) inc += t;
            }
            double c = pre + inc - lt;
            int hit = -1, lastk = -1;
            double cp = c, ch = c;
            for (int k = 0; k < ntok; ++k) {
                const double wk = ff_to_double(wv[k]);
                const double nx = c + wk;
                if (wk > 0.0) lastk = k;
                if (hit < 0 && wk > 0.0 && thr < nx) {
                    hit = k;
                    cp = c;
                    ch = nx;
                }
                c = nx;
            }
            const unsigned m = __ballot_sync(0xFFFFFFFFu, hit >= 0);
            bool unres = false;
            if (m) {
                const int src = __ffs(m) - 1;
                tstar = __shfl_sync(0xFFFFFFFFu, tok0 + (ntok == 1 ? 0 : hit), src);
                const double c_prev = __shfl_sync(0xFFFFFFFFu, cp, src);
                const double c_hit = __shfl_sync(0xFFFFFFFFu, ch, src);
                unres = (thr - c_prev) < 1e-12 * R || (c_hit - thr) < 1e-12 * R;
            } else {
                const unsigned mm = __ballot_sync(0xFFFFFFFFu, lastk >= 0);
                const int src = mm ? 31 - __clz(mm) : 0;
                tstar = __shfl_sync(0xFFFFFFFFu, tok0 + (ntok == 1 ? 0 : max(lastk, 0)), src);
                unres = true;
            }
            if (lane == 0 && unres) stats_add(a.stats, &a.stats->unresolved, 1);
        }
        if (lane == 0) {
            *d.out = tstar;
            if (d.dbg_r) *d.dbg_r = R;
        }
    }
}

}  // namespace sv

#include "sv_host.h"

namespace sv {

// The float-float tier runs as one cooperative grid (one block per SM) so that its phases can
// be separated by grid barriers.  With an empty queue every block returns at once.
template <int ES>
sv_status launch_exact(const ExactArgs &xa, const DeviceInfo &di, cudaStream_t stream) {
    static_assert(sizeof(ExactArgs) < 4096, "kernel parameter block");
    void *args[] = {const_cast<ExactArgs *>(&xa)};
    const cudaError_t e =
        cudaLaunchCooperativeKernel((const void *)k_exact<ES>, dim3(di.sms), dim3(kThreads), args, 0, stream);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace sv
