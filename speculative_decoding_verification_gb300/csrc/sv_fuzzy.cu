// sv_fuzzy.cu — sv_fuzzy_verify: one verification stage of three-model speculative decoding.
//
// ["3-Model Speculative Decoding (PyramidSD)" notes, "Method": a verifier (the qualifier for the
//  draft model, the target for the qualifier) checks a drafter's tokens position by position;
//  fuzzy acceptance keeps a position while Div(P_verifier, P_drafter) <= tau, assisted acceptance
//  runs the speculative-sampling test and replaces a rejected token by a sample of the
//  verifier's own distribution.]
//
// Div is the Jensen-Shannon divergence in bits, a sum of non-negative per-token terms
//   (q log2(2q/(q+p)) + p log2(2p/(q+p))) / 2 = M g(l),  M = max(q, p), l = |log2(q/p)|,
//   g(l) = ((1 + z)(1 - log2(1 + z)) - l z) / 2, z = 2^-l  (0 at l = 0, 1/2 as l grows),
// with g read from a cubic table (sv_js_table.h) and l taken from the exponents: one
// exponential per token.  The float-float pass (positions too close to tau) evaluates the same
// term as (q + p) h(d) / 4, h(d) = (1 + d) log2(1 + d) + (1 - d) log2(1 - d), d = (q - p)/(q + p),
// by its series for |d| < 1/4 and by float-float logarithms elsewhere.
//
// Kernels, in stream order (divergence mode):
//   k_stats          row statistics of every verifier row and every drafter row
//   k_rowstats       one RowStat per row
//   k_div            per (row pair, chunk): float32 partial sums of s h(d), and of the error weight
//   k_fuzzy_accept   per sequence: divergences with a certified error bound, the first position
//                    above tau; positions too close to tau are queued for...
//   k_div_exact_sums, k_div_exact_terms  ...a float-float evaluation of their divergence, each pair
//                    split into chunks over the grid, after which k_fuzzy_accept runs again for
//                    the deferred sequences
//   k_draw_sums, k_draw_finish, k_exact   the draw from the verifier's row at the first failure
// The assisted mode is the sv_verify pipeline with the residual draw replaced by a draw from q.
#include <math.h>

#include "sv_accept.cuh"
#include "sv_device.cuh"
#include "sv_exp2_table.h"
#include "sv_host.h"
#include "sv_js_table.h"
#include "sv_stats.cuh"
#include "sv_tiers.cuh"

namespace sv {

constexpr int kDivExactChunks = 128;   // most chunks per pair in the float-float divergence pass

struct FuzzyArgs {
    RowSet ver, drf;
    int B, K, V;
    const float *temperature;
    const int32_t *tokens;
    const double *uniforms;
    float tau;
    int32_t *accept_len, *out_tokens;
    double *div_out;           // [B][K] or null
    sv_stats *stats;
    const WarpPartial *part;
    int n_split;
    long long n_rows0, n_rows;
    RowStat *rowstat;
    DivPart *dpart;
    int dv_chunks, dv_words, n_vec;
    DivItem *ditem;
    int *dq;
    float4 *dxa;               // [entry]: a chunk's float-float row sums (S_q, S_p)
    float2 *dxb;               // [entry]: a chunk's float-float divergence sum
    int *dxcnt;                // [queue slot]: chunks done, zeroed when the pair is queued
    int dx_cap;
    int *deferred;
    Counters *counters;
    DrawItem *draws;
};

__device__ __forceinline__ bool fuzzy_t_ok(float T) { return T == 0.0f || (T >= 1e-3f && T <= 1e3f); }

// One RowStat per row (one warp per row).
__global__ void __launch_bounds__(kThreads) k_rowstats(const FuzzyArgs a) {
    const long long rid = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (rid >= a.n_rows) return;
    const long long b = rid < a.n_rows0 ? rid / (a.K + 1) : (rid - a.n_rows0) / a.K;
    const float T = a.temperature[b];
    if (!fuzzy_t_ok(T)) return;
    const RowStat r = combine_row(a.part + (size_t)rid * a.n_split * kWarps, a.n_split * kWarps, T == 0.0f, T);
    if ((threadIdx.x & 31) == 0) a.rowstat[rid] = r;
}

// One token's term of the divergence, M g(l) with M = max(q, p) and l = |log2(q/p)| (the float
// weights of the draw pass), and its error weight M (|y_q| + |y_p|).  l comes from the exponents
// (y_q - y_p + log2(inv_q / inv_p) + (x_q - x_p) c_lo), so one exponential per token suffices; g
// is read from the cubic table in shared memory.
struct JsPair {
    DrawRow Q, P;
    float dL;   // log2(inv_q) - log2(inv_p)
};

__device__ __forceinline__ void js_term(float xq, float xp, const JsPair &J, const float4 *tab, float &f, float &yw) {
    xq = fmaxf(xq, kDrawFloor);
    xp = fmaxf(xp, kDrawFloor);
    const float yq = fmaf(xq, J.Q.c_hi, -J.Q.rf), yp = fmaf(xp, J.P.c_hi, -J.P.rf);
    const float lam = (yq - yp) + fmaf(xq - xp, J.Q.c_lo, J.dL);
    const bool qbig = lam >= 0.f;
    const float M = ex2_fast(qbig ? yq : yp) * fmaf(qbig ? xq : xp, qbig ? J.Q.k_lo : J.P.k_lo, qbig ? J.Q.inv_s : J.P.inv_s);
    const float l = fabsf(lam) * (float)kJsTableN;
    float g = 0.5f;
    if (l < (float)(kJsTableN * kJsTableL)) {
        const int i = (int)l;
        const float t = l - (float)i;
        const float4 e = tab[i];
        g = fmaf(t, fmaf(t, fmaf(t, e.w, e.z), e.y), e.x);
    }
    f = M * g;
    yw = M * (fabsf(yq) + fabsf(yp));
}

__device__ __forceinline__ DrawRow fuzzy_row(const FuzzyArgs &a, bool ver, long long b, int j, float T) {
    const RowSet &rs = ver ? a.ver : a.drf;
    const long long rid = ver ? b * (a.K + 1) + j : a.n_rows0 + b * a.K + j;
    const char *row = rs.base + (b * rs.rows_per_seq + j) * rs.pitch_bytes;
    return draw_row(row, T, a.rowstat[rid], nullptr, nullptr, 1.0f);
}

__device__ __forceinline__ bool row_ok(const RowStat &r, bool greedy) {
    return r.flags == 0 && (greedy ? isfinite(r.maxv) : rs_sampled_ok(r));
}

// Per (row pair, chunk) partial sums of the divergence.
template <int ES>
__global__ void __launch_bounds__(kThreads) k_div(const FuzzyArgs a) {
    constexpr int EPV = 16 / ES;
    __shared__ float s_h[kWarps], s_l[kWarps], s_y[kWarps];
    __shared__ float4 s_js[kJsTableSize];
    const long long unit = blockIdx.x;
    const long long pair = unit / a.dv_chunks;
    const int chunk = (int)(unit - pair * a.dv_chunks);
    const long long b = pair / a.K;
    const int j = (int)(pair - b * a.K);
    const float T = a.temperature[b];
    if (T == 0.0f || !fuzzy_t_ok(T)) return;
    const RowStat rq = a.rowstat[b * (a.K + 1) + j], rp = a.rowstat[a.n_rows0 + b * a.K + j];
    if (!row_ok(rq, false) || !row_ok(rp, false)) return;   // reported by k_fuzzy_accept
    for (int i = threadIdx.x; i < kJsTableSize; i += kThreads) s_js[i] = kJsTable[i];
    __shared__ JsPair s_J;
    if (threadIdx.x == 0) {   // the rows' parameters once per block (their float64 parts are not per thread)
        JsPair J;
        J.Q = fuzzy_row(a, true, b, j, T);
        J.P = fuzzy_row(a, false, b, j, T);
        J.dL = (float)(log2((double)J.Q.inv_s) - log2((double)J.P.inv_s));
        s_J = J;
    }
    __syncthreads();
    const JsPair J = s_J;
    const DrawRow &Q = J.Q, &P = J.P;
    const int w0 = chunk * a.dv_words, w1 = min(a.n_vec, w0 + a.dv_words);
    const uint4 *vq = reinterpret_cast<const uint4 *>(Q.row);
    const uint4 *vp = reinterpret_cast<const uint4 *>(P.row);
    ff acc = {0.f, 0.f};
    float ysum = 0.f;
    for (int wi = w0 + threadIdx.x; wi < w1; wi += kThreads) {
        const uint4 gq = __ldg(vq + wi), gp = __ldg(vp + wi);
        float xq[EPV], xp[EPV];
        if constexpr (ES == 2) {
            xq[0] = bf16_lo(gq.x); xq[1] = bf16_hi(gq.x); xq[2] = bf16_lo(gq.y); xq[3] = bf16_hi(gq.y);
            xq[4] = bf16_lo(gq.z); xq[5] = bf16_hi(gq.z); xq[6] = bf16_lo(gq.w); xq[7] = bf16_hi(gq.w);
            xp[0] = bf16_lo(gp.x); xp[1] = bf16_hi(gp.x); xp[2] = bf16_lo(gp.y); xp[3] = bf16_hi(gp.y);
            xp[4] = bf16_lo(gp.z); xp[5] = bf16_hi(gp.z); xp[6] = bf16_lo(gp.w); xp[7] = bf16_hi(gp.w);
        } else {
            xq[0] = __uint_as_float(gq.x); xq[1] = __uint_as_float(gq.y);
            xq[2] = __uint_as_float(gq.z); xq[3] = __uint_as_float(gq.w);
            xp[0] = __uint_as_float(gp.x); xp[1] = __uint_as_float(gp.y);
            xp[2] = __uint_as_float(gp.z); xp[3] = __uint_as_float(gp.w);
        }
        float fs = 0.f, ys = 0.f;
#pragma unroll
        for (int k = 0; k < EPV; ++k) {
            float f, yw;
            js_term(xq[k], xp[k], J, s_js, f, yw);
            fs += f;
            ys += yw;
        }
        acc = ff_add_f(acc, fs);
        ysum += ys;
    }
    if (chunk == a.dv_chunks - 1) {   // the row's last (< 16 B) elements
        for (int v = a.n_vec * EPV + threadIdx.x; v < a.V; v += kThreads) {
            float f, yw;
            js_term(load_elem<ES>(Q.row, v), load_elem<ES>(P.row, v), J, s_js, f, yw);
            acc = ff_add_f(acc, f);
            ysum += yw;
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        acc = ff_add(acc, {__shfl_xor_sync(0xFFFFFFFFu, acc.hi, o), __shfl_xor_sync(0xFFFFFFFFu, acc.lo, o)});
        ysum += __shfl_xor_sync(0xFFFFFFFFu, ysum, o);
    }
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        s_h[warp] = acc.hi;
        s_l[warp] = acc.lo;
        s_y[warp] = ysum;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        ff t = {0.f, 0.f};
        float y = 0.f;
        for (int w = 0; w < kWarps; ++w) {
            t = ff_add(t, {s_h[w], s_l[w]});
            y += s_y[w];
        }
        a.dpart[unit] = {t.hi, t.lo, y, 0.f};
    }
}

// Float-float log2 of x in (0, 2]: a float32 estimate y0, then log2(x 2^-y0) = log2(1 + t) with
// |t| ~ 2^-22 from its series (t - t^2/2 + t^3/3) / ln 2.
__device__ __forceinline__ ff ff_log2(ff x, const float2 *tab) {
    const float y0 = log2f(x.hi);
    const ff r = ff_mul(x, ff_exp2(-y0, 0.f, tab));
    const ff t = ff_add_f(r, -1.0f);
    const ff t2 = ff_mul(t, t);
    ff ln = ff_sub(t, ff_mul({0.5f, 0.f}, t2));
    ln = ff_add(ln, ff_mul({1.0f / 3.0f, 0.f}, ff_mul(t2, t)));
    const ff inv_ln2 = {1.44269502162933349609375f, 1.925963033500011e-08f};
    return ff_add({y0, 0.f}, ff_mul(ln, inv_ln2));
}

// The divergences of the queued pairs in float-float.  Each pair is split into ch chunks of
// its row pair (ch from the number queued, so that their (pair, chunk) entries fit the
// workspace), and two persistent passes run over all (pair, chunk) units: the first sums the
// chunk's q and p masses, the second takes the pair's exact row sums from those partials, sums
// its chunk's divergence terms, and the last chunk of a pair to finish adds the pair's
// partials and records the divergence.
__device__ __forceinline__ int div_exact_chunks(int n, int cap) {
    const int ch = n > 0 ? cap / n : 1;
    return ch < 1 ? 1 : (ch > kDivExactChunks ? kDivExactChunks : ch);
}

struct DivExactUnit {
    long long pair;
    int slot, chunk, v0, v1;   // tokens [v0, v1) of the pair's rows
};

__device__ __forceinline__ DivExactUnit div_exact_unit(const FuzzyArgs &a, long long u, int ch) {
    DivExactUnit x;
    x.slot = (int)(u / ch);
    x.chunk = (int)(u - (long long)x.slot * ch);
    x.pair = a.dq[x.slot];
    const int per = (a.V + ch - 1) / ch;
    x.v0 = min(x.chunk * per, a.V);
    x.v1 = min(x.v0 + per, a.V);
    return x;
}

// Block sum of two float-float values (every thread of the block calls; s_h.. hold kWarps).
__device__ __forceinline__ void block_ff2(ff u, ff v, ff &U, ff &W, float *s_h, float *s_l, float *s_h2,
                                          float *s_l2) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        u = ff_add(u, {__shfl_xor_sync(0xFFFFFFFFu, u.hi, o), __shfl_xor_sync(0xFFFFFFFFu, u.lo, o)});
        v = ff_add(v, {__shfl_xor_sync(0xFFFFFFFFu, v.hi, o), __shfl_xor_sync(0xFFFFFFFFu, v.lo, o)});
    }
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        s_h[w] = u.hi;
        s_l[w] = u.lo;
        s_h2[w] = v.hi;
        s_l2[w] = v.lo;
    }
    __syncthreads();
    U = {0.f, 0.f};
    W = {0.f, 0.f};
    for (int i = 0; i < kWarps; ++i) {
        U = ff_add(U, {s_h[i], s_l[i]});
        W = ff_add(W, {s_h2[i], s_l2[i]});
    }
    __syncthreads();
}

// Pass 1: per (pair, chunk), the float-float sums of 2^(x c - r) over the chunk's tokens of
// the verifier row (q) and the drafter row (p).
template <int ES>
__global__ void __launch_bounds__(kThreads) k_div_exact_sums(const FuzzyArgs a) {
    __shared__ float2 tab[256];
    __shared__ float s_h[kWarps], s_l[kWarps], s_h2[kWarps], s_l2[kWarps];
    const int n = *reinterpret_cast<volatile int *>(&a.counters->n_div_exact);
    if (n == 0) return;   // uniform across the grid
    const int ch = div_exact_chunks(n, a.dx_cap);
    tab[threadIdx.x] = kExp2Table[threadIdx.x];
    __syncthreads();
    for (long long u = blockIdx.x; u < (long long)n * ch; u += gridDim.x) {
        const DivExactUnit x = div_exact_unit(a, u, ch);
        const long long b = x.pair / a.K;
        const int j = (int)(x.pair - b * a.K);
        const float T = a.temperature[b];
        const RowStat rq = a.rowstat[b * (a.K + 1) + j], rp = a.rowstat[a.n_rows0 + b * a.K + j];
        float c_hi, c_lo;
        log2e_over(T, c_hi, c_lo);
        const ff c = {c_hi, c_lo};
        const char *qrow = a.ver.base + (b * a.ver.rows_per_seq + j) * a.ver.pitch_bytes;
        const char *prow = a.drf.base + (b * a.drf.rows_per_seq + j) * a.drf.pitch_bytes;
        auto mass = [&](float xv, int r) -> ff { return xv == -INFINITY ? ff{0.f, 0.f} : ff_exp2_xc(xv, c, r, tab); };
        ff sq = {0.f, 0.f}, sp = {0.f, 0.f};
        for (int v = x.v0 + threadIdx.x; v < x.v1; v += kThreads) {
            sq = ff_add(sq, mass(load_elem<ES>(qrow, v), rq.r));
            sp = ff_add(sp, mass(load_elem<ES>(prow, v), rp.r));
        }
        ff Sq, Sp;
        block_ff2(sq, sp, Sq, Sp, s_h, s_l, s_h2, s_l2);
        if (threadIdx.x == 0) a.dxa[(size_t)x.slot * ch + x.chunk] = make_float4(Sq.hi, Sq.lo, Sp.hi, Sp.lo);
    }
}

// Pass 2: per (pair, chunk), the float-float divergence terms of the chunk's tokens with the
// pair's exact row sums; the last chunk of a pair adds the partials and records the divergence.
template <int ES>
__global__ void __launch_bounds__(kThreads) k_div_exact_terms(const FuzzyArgs a) {
    __shared__ float2 tab[256];
    __shared__ ff s_c[12];
    __shared__ float s_h[kWarps], s_l[kWarps], s_h2[kWarps], s_l2[kWarps];
    __shared__ ff s_inv[2];
    __shared__ int s_last;
    const int n = *reinterpret_cast<volatile int *>(&a.counters->n_div_exact);
    if (n == 0) return;   // uniform across the grid
    const int ch = div_exact_chunks(n, a.dx_cap);
    tab[threadIdx.x] = kExp2Table[threadIdx.x];
    if (threadIdx.x < 12) {
        const float k = (float)(threadIdx.x + 1);
        s_c[threadIdx.x] = ff_recip({k * (2.0f * k - 1.0f), 0.f});   // 1 / (k (2k - 1))
    }
    __syncthreads();
    const ff inv_ln2 = {1.44269502162933349609375f, 1.925963033500011e-08f};
    for (long long u = blockIdx.x; u < (long long)n * ch; u += gridDim.x) {
        const DivExactUnit x = div_exact_unit(a, u, ch);
        const long long b = x.pair / a.K;
        const int j = (int)(x.pair - b * a.K);
        const float T = a.temperature[b];
        const RowStat rq = a.rowstat[b * (a.K + 1) + j], rp = a.rowstat[a.n_rows0 + b * a.K + j];
        float c_hi, c_lo;
        log2e_over(T, c_hi, c_lo);
        const ff c = {c_hi, c_lo};
        const char *qrow = a.ver.base + (b * a.ver.rows_per_seq + j) * a.ver.pitch_bytes;
        const char *prow = a.drf.base + (b * a.drf.rows_per_seq + j) * a.drf.pitch_bytes;
        auto mass = [&](float xv, int r) -> ff { return xv == -INFINITY ? ff{0.f, 0.f} : ff_exp2_xc(xv, c, r, tab); };
        // the pair's exact row sums from the chunks' partials (one warp)
        if (threadIdx.x < 32) {
            ff sq = {0.f, 0.f}, sp = {0.f, 0.f};
            for (int k = threadIdx.x; k < ch; k += 32) {
                const float4 pv = a.dxa[(size_t)x.slot * ch + k];
                sq = ff_add(sq, {pv.x, pv.y});
                sp = ff_add(sp, {pv.z, pv.w});
            }
            sq = warp_sum_ff(sq);
            sp = warp_sum_ff(sp);
            if (threadIdx.x == 0) {
                s_inv[0] = ff_recip(sq);
                s_inv[1] = ff_recip(sp);
            }
        }
        __syncthreads();
        const ff iq = s_inv[0], ip = s_inv[1];
        ff acc = {0.f, 0.f};
        for (int v = x.v0 + threadIdx.x; v < x.v1; v += kThreads) {
            const ff q = ff_mul(mass(load_elem<ES>(qrow, v), rq.r), iq);
            const ff p = ff_mul(mass(load_elem<ES>(prow, v), rp.r), ip);
            const ff s = ff_add(q, p);
            if (!(s.hi > 0.f)) continue;
            const ff rs = ff_recip(s);
            const ff d = ff_mul(ff_sub(q, p), rs);
            ff h;
            if (fabsf(d.hi) < 0.25f) {
                const ff d2 = ff_mul(d, d);
                ff poly = s_c[11];
                for (int k = 10; k >= 0; --k) poly = ff_add(s_c[k], ff_mul(d2, poly));
                h = ff_mul(ff_mul(d2, poly), inv_ln2);
            } else {
                const ff qa = ff_mul(ff_add(q, q), rs), pb = ff_mul(ff_add(p, p), rs);
                h = {0.f, 0.f};
                if (qa.hi > 0x1p-100f) h = ff_add(h, ff_mul(qa, ff_log2(qa, tab)));
                else if (qa.hi > 0.f) h = ff_add_f(h, qa.hi * log2f(qa.hi));
                if (pb.hi > 0x1p-100f) h = ff_add(h, ff_mul(pb, ff_log2(pb, tab)));
                else if (pb.hi > 0.f) h = ff_add_f(h, pb.hi * log2f(pb.hi));
            }
            acc = ff_add(acc, ff_mul(s, h));
        }
        ff F, unused;
        block_ff2(acc, {0.f, 0.f}, F, unused, s_h, s_l, s_h2, s_l2);
        if (threadIdx.x == 0) {
            a.dxb[(size_t)x.slot * ch + x.chunk] = make_float2(F.hi, F.lo);
            __threadfence();
            s_last = atomicAdd(&a.dxcnt[x.slot], 1) == ch - 1;
        }
        __syncthreads();
        if (s_last && threadIdx.x < 32) {
            __threadfence();
            ff t = {0.f, 0.f};
            for (int k = threadIdx.x; k < ch; k += 32) {
                const float2 pv = __ldcg(&a.dxb[(size_t)x.slot * ch + k]);   // written by other blocks: L2
                t = ff_add(t, {pv.x, pv.y});
            }
            t = warp_sum_ff(t);
            if (threadIdx.x == 0) {
                const double dv = 0.25 * ff_to_double(t);
                a.ditem[x.pair].exact = dv;
                a.ditem[x.pair].state = 2;
                if (fabs(dv - (double)a.tau) < 1e-10) stats_add(a.stats, &a.stats->unresolved, 1);
            }
        }
        __syncthreads();   // s_inv and s_last are rewritten by the next unit
    }
}

// Per sequence (one warp): the divergence of every position with its error bound, the first
// position above tau, outputs and the draw item.  Pass 0 defers a sequence whose decision
// depends on a divergence the bound cannot place; pass 1 finishes the deferred sequences with
// the float-float values.
template <int ES>
__global__ void __launch_bounds__(32) k_fuzzy_accept(const FuzzyArgs a, int pass) {
    const int b = blockIdx.x, lane = threadIdx.x;
    const int K = a.K, V = a.V;
    if (pass == 1 && !a.deferred[b]) return;
    const float T = a.temperature[b];
    const bool greedy = T == 0.0f;
    int32_t *outs = a.out_tokens + (size_t)b * (K + 1);
    if (!fuzzy_t_ok(T)) {
        if (lane == 0) {
            report_error(a.stats, SV_ERR_INVALID_ARG, b);
            a.accept_len[b] = 0;
        }
        for (int j = lane; j <= K; j += 32) outs[j] = -1;
        return;
    }
    // rows: every verifier row and every drafter row must be finite
    bool bad = false;
    for (int j = lane; j <= K; j += 32) bad |= !row_ok(a.rowstat[(long long)b * (K + 1) + j], greedy);
    for (int j = lane; j < K; j += 32) bad |= !row_ok(a.rowstat[a.n_rows0 + (long long)b * K + j], greedy);
    int s = -1;
    bool badtok = false;
    if (lane < K) {
        s = a.tokens[(size_t)b * K + lane];
        badtok = s < 0 || s >= V;
    }
    const bool any_bad = __any_sync(0xFFFFFFFFu, bad), any_badtok = __any_sync(0xFFFFFFFFu, badtok);
    if (any_bad || any_badtok) {
        if (lane == 0) {
            report_error(a.stats, any_bad ? SV_ERR_NONFINITE : SV_ERR_BAD_TOKEN, b);
            a.accept_len[b] = 0;
        }
        for (int j = lane; j <= K; j += 32) outs[j] = -1;
        return;
    }
    double dv = 0.0;
    bool amb = false;
    if (lane < K) {
        const long long pair = (long long)b * K + lane;
        const RowStat rq = a.rowstat[(long long)b * (K + 1) + lane], rp = a.rowstat[a.n_rows0 + pair];
        if (greedy) {
            dv = rq.argmax == rp.argmax ? 0.0 : 1.0;   // one-hot rows
        } else if (a.ditem[pair].state == 2) {
            dv = a.ditem[pair].exact;
        } else {
            ff F = {0.f, 0.f};
            float Y = 0.f;
            for (int c = 0; c < a.dv_chunks; ++c) {
                const DivPart dp = a.dpart[pair * a.dv_chunks + c];
                F = ff_add(F, {dp.s_hi, dp.s_lo});
                Y += dp.y;
            }
            dv = ff_to_double(F);
            // Bound on |dv - JSD|.  Per token the term is M g(l).  M carries the weight's relative
            // error (the normaliser, the exponential, the factor and product roundings, and
            // ln2 u |y| from rounding y once): at most g M (A + ln2 u |y|) with g <= 1/2 and
            // sum M <= 2.  l carries u (|y_q| + |y_p|) from the exponents' roundings plus the
            // normalisers' relative errors / ln2 (through dL); g moves by at most kJsSlopeMax per
            // unit of l.  The table adds kJsTableErr per unit of M, its Horner evaluation 3u, the
            // float32 word sums 8u.  Y = sum M (|y_q| + |y_p|).
            const DrawRow Q = fuzzy_row(a, true, b, lane, T), P = fuzzy_row(a, false, b, lane, T);
            const double rq2 = kLn2 * 0x1p-23 * (fabs((double)Q.rf) + 128.0);
            const double rp2 = kLn2 * 0x1p-23 * (fabs((double)P.rf) + 128.0);
            const double Aq = kEx2RelErr + 4.0 * kU32 + Q.norm_err + rq2 * rq2;
            const double Ap = kEx2RelErr + 4.0 * kU32 + P.norm_err + rp2 * rp2;
            const double E = 1.0002 * (Aq + Ap) + 0.5 * kLn2 * kU32 * 1.01 * 1.001 * (double)Y +
                             kJsSlopeMax * (3.0 * kU32 * 1.001 * (double)Y + 2.0 * 1.4427 * (Q.norm_err + P.norm_err)) +
                             2.0 * kJsTableErr + 8.0 * kU32 + 8.0 * kU32 * dv + 1e-9;
            amb = fabs(dv - (double)a.tau) <= E;
        }
    }
    const bool acc = lane < K && dv <= (double)a.tau;
    const unsigned lowK = K >= 32 ? 0xFFFFFFFFu : ((1u << K) - 1u);
    const unsigned accm = __ballot_sync(0xFFFFFFFFu, acc) & lowK;
    const unsigned rej = ~accm & lowK;
    const int k = rej ? __ffs(rej) - 1 : K;
    // every position the bound cannot place is queued (not only those up to k): once they are
    // settled the first failure may lie further on, and pass 1 must not meet another
    const unsigned ambm = __ballot_sync(0xFFFFFFFFu, amb) & lowK;
    if (ambm) {   // pass 0 only: pass 1 reads float-float values
        if ((ambm >> lane) & 1u) {
            const long long pair = (long long)b * K + lane;
            a.ditem[pair].state = 1;
            const int slot = atomicAdd(&a.counters->n_div_exact, 1);
            a.dxcnt[slot] = 0;
            a.dq[slot] = (int)pair;
        }
        if (lane == 0) {
            a.deferred[b] = 1;
            stats_add(a.stats, &a.stats->reresolved, 1);
        }
        return;
    }
    if (a.div_out && lane < K) a.div_out[(size_t)b * K + lane] = dv;
    for (int j = lane; j <= K; j += 32) outs[j] = j < k ? a.tokens[(size_t)b * K + j] : -1;
    __syncwarp();
    if (lane != 0) return;
    a.accept_len[b] = k;
    stats_add(a.stats, &a.stats->rows, 2 * K + 1);
    if (greedy) {
        outs[k] = a.rowstat[(long long)b * (K + 1) + k].argmax;
        return;
    }
    stats_add(a.stats, &a.stats->accept_tests, min(k + 1, K));
    const int d = atomicAdd(&a.counters->n_draws, 1);
    DrawItem it;
    it.q = fuzzy_row(a, true, b, k, T);
    it.p = {};
    it.p.top_x = INFINITY;
    it.p.cut_x = -INFINITY;
    it.p.cut_id = 0x7FFFFFFF;
    it.has_p = 0;
    it.filt = 0;
    it.u = a.uniforms[(size_t)b * (K + 1) + K];
    it.out = outs + k;
    it.dbg_r = nullptr;
    it.seq = b;
    it.k = k;
    a.draws[d] = it;
}

template <int ES>
static sv_status launch_fuzzy(const VerifyPlan &pl, FuzzyArgs fa, AcceptArgs acc, void *ws, cudaStream_t stream) {
    DeviceInfo di;
    if (!device_info(di)) return SV_ERR_CUDA;
    char *w = static_cast<char *>(ws);
    Counters *counters = reinterpret_cast<Counters *>(w + pl.off_counters);
    WarpPartial *part = reinterpret_cast<WarpPartial *>(w + pl.off_part);
    StatsArgs sa;
    sa.set[0] = fa.ver;
    sa.set[1] = fa.drf;
    sa.n_sets = 2;
    sa.V = fa.V;
    sa.temperature = fa.temperature;
    sa.n_split = pl.n_split;
    sa.chunk_vecs = pl.chunk_vecs;
    sa.n_rows0 = pl.n_rows0;
    sa.n_units = (pl.n_rows0 + pl.n_rows1) * pl.n_split;
    sa.part = part;
    sa.counters = counters;
    sa.stats = fa.stats;
    sa.wait_limit = kWaitLimitCycles;
    {
        const sv_status st = launch_stats<ES>(sa, di, stream);
        if (st != SV_OK) return st;
    }
    fa.part = part;
    fa.n_split = pl.n_split;
    fa.n_rows0 = pl.n_rows0;
    fa.n_rows = pl.n_rows0 + pl.n_rows1;
    fa.rowstat = reinterpret_cast<RowStat *>(w + pl.off_rowstat);
    fa.dpart = reinterpret_cast<DivPart *>(w + pl.off_dpart);
    fa.dv_chunks = pl.dv_chunks;
    fa.dv_words = pl.dv_words;
    fa.n_vec = pl.n_vec;
    fa.ditem = reinterpret_cast<DivItem *>(w + pl.off_ditem);
    fa.dq = reinterpret_cast<int *>(w + pl.off_dq);
    fa.dxa = reinterpret_cast<float4 *>(w + pl.off_dxa);
    fa.dxb = reinterpret_cast<float2 *>(w + pl.off_dxb);
    fa.dxcnt = reinterpret_cast<int *>(w + pl.off_dxcnt);
    fa.dx_cap = pl.dx_cap;
    fa.deferred = reinterpret_cast<int *>(w + pl.off_deferred);
    fa.counters = counters;
    fa.draws = reinterpret_cast<DrawItem *>(w + pl.off_draws);
    const long long n_pairs = (long long)fa.B * fa.K;
    if (n_pairs > 0 && cudaMemsetAsync(fa.ditem, 0, sizeof(DivItem) * n_pairs, stream) != cudaSuccess)
        return SV_ERR_CUDA;
    if (cudaMemsetAsync(fa.deferred, 0, sizeof(int) * fa.B, stream) != cudaSuccess) return SV_ERR_CUDA;
    k_rowstats<<<(unsigned)div_up(fa.n_rows, kWarps), kThreads, 0, stream>>>(fa);
    if (n_pairs > 0) k_div<ES><<<(unsigned)(n_pairs * fa.dv_chunks), kThreads, 0, stream>>>(fa);
    k_fuzzy_accept<ES><<<fa.B, 32, 0, stream>>>(fa, 0);
    if (n_pairs > 0) {
        // persistent passes over the queued pairs' chunks (the queue length is on the device)
        const unsigned gx = (unsigned)(di.sms * 4);
        k_div_exact_sums<ES><<<gx, kThreads, 0, stream>>>(fa);
        k_div_exact_terms<ES><<<gx, kThreads, 0, stream>>>(fa);
        k_fuzzy_accept<ES><<<fa.B, 32, 0, stream>>>(fa, 1);
    }
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    acc.part = part;
    acc.n_split = pl.n_split;
    acc.n_rows0 = pl.n_rows0;
    acc.rowstat = fa.rowstat;
    acc.nuc = nullptr;
    acc.top = nullptr;
    acc.draws = fa.draws;
    acc.exact = reinterpret_cast<ExactItem *>(w + pl.off_exact);
    acc.exact_unc = reinterpret_cast<int *>(w + pl.off_xunc_n);
    acc.counters = counters;
    return launch_draw_tiers<ES>(pl, acc, nullptr, nullptr, w, fa.B, di, stream);
}

}  // namespace sv

using namespace sv;

extern "C" size_t sv_fuzzy_verify_workspace_size(int B, int K, int V) { return sv_verify_workspace_size(B, K, V); }

extern "C" sv_status sv_fuzzy_verify(const void *verifier_logits, int64_t v_row_pitch, const void *drafter_logits,
                                     int64_t d_row_pitch, int d_rows_per_seq, sv_dtype dtype,
                                     const int32_t *draft_tokens, const double *uniforms, int B, int K, int V,
                                     const float *temperature, float tau, int mode, int32_t *accept_len,
                                     int32_t *out_tokens, double *divergence, sv_stats *stats, void *workspace,
                                     size_t workspace_bytes, sv_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (mode == SV_ACCEPT_ASSISTED) {
        if (divergence != nullptr) return SV_ERR_INVALID_ARG;
        return verify_entry(verifier_logits, v_row_pitch, drafter_logits, d_row_pitch, d_rows_per_seq, dtype,
                            draft_tokens, uniforms, B, K, V, temperature, nullptr, nullptr, 0, 1.0f, 1, accept_len,
                            out_tokens, nullptr, stats, workspace, workspace_bytes, stream);
    }
    if (mode != SV_ACCEPT_DIVERGENCE || !isfinite(tau)) return SV_ERR_INVALID_ARG;
    if (B < 1 || K < 0 || K > SV_MAX_K || V < 1) return SV_ERR_INVALID_ARG;
    if (!rows_ok(verifier_logits, v_row_pitch, V, dtype)) return SV_ERR_INVALID_ARG;
    if (K > 0 && (!rows_ok(drafter_logits, d_row_pitch, V, dtype) || d_rows_per_seq < K)) return SV_ERR_INVALID_ARG;
    if ((K > 0 && draft_tokens == nullptr) || uniforms == nullptr || temperature == nullptr) return SV_ERR_INVALID_ARG;
    if (accept_len == nullptr || out_tokens == nullptr) return SV_ERR_INVALID_ARG;
    if ((long long)V * B * (2 * K + 1) > (1LL << 46)) return SV_ERR_INVALID_ARG;
    const int es = elem_size(dtype);
    const VerifyPlan pl = plan_verify(B, K, V, es);
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < pl.bytes) return SV_ERR_WORKSPACE;
    if (!on_current_device(stream, verifier_logits, K > 0 ? drafter_logits : nullptr)) return SV_ERR_INVALID_ARG;
    if (stats && cudaMemsetAsync(stats, 0, sizeof(sv_stats), stream) != cudaSuccess) return SV_ERR_CUDA;
    FuzzyArgs fa{};
    // every row of both models is streamed (greedy sequences compare the two argmaxes)
    fa.ver = {static_cast<const char *>(verifier_logits), v_row_pitch * es, K + 1, K + 1, 0};
    fa.drf = {static_cast<const char *>(K > 0 ? drafter_logits : verifier_logits),
              (K > 0 ? d_row_pitch : v_row_pitch) * es, K > 0 ? d_rows_per_seq : 1, K, 0};
    fa.B = B;
    fa.K = K;
    fa.V = V;
    fa.temperature = temperature;
    fa.tokens = draft_tokens;
    fa.uniforms = uniforms;
    fa.tau = tau;
    fa.accept_len = accept_len;
    fa.out_tokens = out_tokens;
    fa.div_out = divergence;
    fa.stats = stats;
    AcceptArgs acc{};
    acc.tgt = fa.ver;
    acc.drf = fa.drf;
    acc.K = K;
    acc.V = V;
    acc.temperature = temperature;
    acc.tokens = draft_tokens;
    acc.uniforms = uniforms;
    acc.accept_len = accept_len;
    acc.out_tokens = out_tokens;
    acc.stats = stats;
    acc.sag_C = 1.0f;
    acc.draw_from_q = 1;
    if (es == 4) return launch_fuzzy<4>(pl, fa, acc, workspace, stream);
    return launch_fuzzy<2>(pl, fa, acc, workspace, stream);
}
