// sv_tree.cu — sv_tree_verify (a tree of drafted tokens verified in one pass) and sv_tree_reuse.
//
// ["Mirror Speculative Decoding" notes, §1.1 (tree drafts: the target verifies a candidate tree
//  at once), §3.1-§3.3 (branch-complete trees; the committed prefix reuses the tree when it is
//  one of its paths, depth-2 branching included); "Accelerating LLM Decoding with Speculative
//  Sampling (2023)" notes, §3 (the accept test and the residual, applied again after each
//  rejection among a node's children)]
//
// Node i (1..N) holds tokens[i-1] below node parents[i-1] < i; node 0 is the context.  Row i of
// the target and draft logits follows node i.  Greedy sequences follow the first child holding
// the target argmax.  Sampled sequences test a node's children in index order: child i passes
// iff u < min(1, (q(t) - c_i p(t))+ / (R(c_i) p(t))) with R(c) = sum_v (q_v - c p_v)+, c_1 = 0,
// c_(i+1) = c_i + R(c_i) (the residual of the residual, in closed form); when every child fails
// the token is drawn from (q - c p)+ by the inverse CDF in id order.
//
// Kernels: k_stats (every target row; draft rows of sampled sequences), k_tree_rowstats, and
// k_tree_walk, one block per sequence.  The walk takes every decision in float32 with a
// certified margin: the per-token weights carry (kEx2RelErr + 4u + normaliser error + ln2 u |y|)
// relative error, each residual sum R(c) is a block reduction over both rows with that error
// summed, c accumulates the errors of the sums it adds up.  A node whose decision the margin
// cannot settle is redone in float-float (exact row sums, residual sums and draw).
#include <cooperative_groups.h>
#include <math.h>

#include "sv_accept.cuh"
#include "sv_device.cuh"
#include "sv_draw.cuh"
#include "sv_exp2_table.h"
#include "sv_host.h"
#include "sv_stats.cuh"

namespace sv {

struct TreeArgs {
    RowSet tgt, drf;           // rows (b, i), i = 0..N
    int B, N, V;
    const int32_t *parents, *tokens;
    const double *uniforms;    // [B][N+1]: u[b][0] the draw, u[b][i] node i's test
    const float *temperature;
    int32_t *accept_len, *out_tokens, *path;
    sv_stats *stats;
    const WarpPartial *part;
    int n_split;
    long long n_rows0, n_rows;
    RowStat *rowstat;
    int n_vec;
};

__global__ void __launch_bounds__(kThreads) k_tree_rowstats(const TreeArgs a) {
    const long long rid = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (rid >= a.n_rows) return;
    const long long b = (rid < a.n_rows0 ? rid : rid - a.n_rows0) / (a.N + 1);
    const float T = a.temperature[b];
    const bool greedy = T == 0.0f;
    if (!(greedy || (T >= 1e-3f && T <= 1e3f))) return;
    if (rid >= a.n_rows0 && greedy) return;   // draft rows of greedy sequences are not read
    const RowStat r = combine_row(a.part + (size_t)rid * a.n_split * kWarps, a.n_split * kWarps, greedy, T);
    if ((threadIdx.x & 31) == 0) a.rowstat[rid] = r;
}

// ---- cluster-wide helpers (every thread of every block gets the result) ----------------------
// kTreeCluster blocks share one sequence; each streams its slice of every row.
constexpr int kTreeCluster = 8;

struct TreeShared {
    float2 tab[256];
    float s_hi[kWarps], s_lo[kWarps];
    float2 part;               // this block's share of a cluster sum / scan
    int owner;                 // draw: first segment of this block past u R (kThreads: none)
    int result;
    float2 c_at, c_before;     // draw: cumulative sums at t* and before it (owner block)
    DrawRow q, p;              // the current node's rows (set by thread 0)
    int flag;                  // a decision taken by thread 0, read by every thread
};

// Thread 0's value of v for every thread of the block (decisions carry float64 bounds: one
// thread evaluates them, the FP64 pipe is narrow on this GPU).
__device__ __forceinline__ int block_bcast(int v, TreeShared &S) {
    __syncthreads();
    if (threadIdx.x == 0) S.flag = v;
    __syncthreads();
    return S.flag;
}

struct TreeCtx {
    cooperative_groups::cluster_group cl;
    int rank;
    int n_vec, V;
    int w0, w1;                // this block's slice of 16-byte words
    bool tail;                 // this block also takes the row's scalar tail
};

__device__ __forceinline__ ff block_sum_ffv(ff v, TreeShared &S) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
        v = ff_add(v, {__shfl_xor_sync(0xFFFFFFFFu, v.hi, o), __shfl_xor_sync(0xFFFFFFFFu, v.lo, o)});
    const int w = threadIdx.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) {
        S.s_hi[w] = v.hi;
        S.s_lo[w] = v.lo;
    }
    __syncthreads();
    ff t = {0.f, 0.f};
    for (int i = 0; i < kWarps; ++i) t = ff_add(t, {S.s_hi[i], S.s_lo[i]});
    return t;
}

// Sum over the cluster, added in rank order so that every block gets the same value.
__device__ __forceinline__ ff cluster_sum_ff(TreeCtx &X, ff v, TreeShared &S) {
    const ff b = block_sum_ffv(v, S);
    if (threadIdx.x == 0) S.part = make_float2(b.hi, b.lo);
    X.cl.sync();
    ff t = {0.f, 0.f};
    for (int q = 0; q < kTreeCluster; ++q) {
        const float2 pq = *X.cl.map_shared_rank(&S.part, q);
        t = ff_add(t, {pq.x, pq.y});
    }
    X.cl.sync();   // S.part is free again
    return t;
}

// Normalised float32 weight of one token (the draw pass's form).
__device__ __forceinline__ float tw(const DrawRow &R, float x, float &y) {
    x = fmaxf(x, kDrawFloor);
    y = fmaf(x, R.c_hi, -R.rf);
    return ex2_fast(y) * fmaf(x, R.k_lo, R.inv_s);
}

// Float-float weight 2^(x c - r) / S of one token.
__device__ __forceinline__ ff twx(float x, ff c, int r, ff inv_s, const float2 *tab) {
    if (x == -INFINITY) return {0.f, 0.f};
    return ff_mul(ff_exp2_xc(x, c, r, tab), inv_s);
}

// Calls fn(xq, xp, v) for every token of this block's slice of the two rows (16-byte words, then
// the scalar tail in the last block).  Thread t takes words w0 + t, w0 + t + blockDim, ...
template <int ES, class Fn>
__device__ __forceinline__ void for_pair(const TreeCtx &X, const char *rq, const char *rp, Fn fn) {
    constexpr int EPV = 16 / ES;
    for (int wi = X.w0 + threadIdx.x; wi < X.w1; wi += kThreads) {
        const uint4 gq = __ldg(reinterpret_cast<const uint4 *>(rq) + wi);
        const uint4 gp = __ldg(reinterpret_cast<const uint4 *>(rp) + wi);
        float xq[EPV], xp[EPV];
        unpack<ES>(gq, xq);
        unpack<ES>(gp, xp);
#pragma unroll
        for (int k = 0; k < EPV; ++k) fn(xq[k], xp[k], wi * EPV + k);
    }
    if (X.tail)
        for (int v = X.n_vec * EPV + threadIdx.x; v < X.V; v += kThreads) fn(load_elem<ES>(rq, v), load_elem<ES>(rp, v), v);
}

// Per-token relative error of a float32 weight, without the ln2 u |y| part: the exponential,
// the factor and product roundings, the normaliser and the factor's second-order remainder.
__device__ __forceinline__ double base_err(const DrawRow &R) {
    const double r2 = kLn2 * 0x1p-23 * (fabs((double)R.rf) + 128.0);
    return kEx2RelErr + 4.0 * kU32 + R.norm_err + r2 * r2;
}

constexpr double kTreeKappa = kLn2 * kU32 * 1.01;   // relative error per unit |y| (y rounded once)

// Float32 residual sum R(c) = sum_v (q_v - c p_v)+ and a bound on its error.  dc bounds the error
// of c itself.
template <int ES>
__device__ __forceinline__ float tree_R(TreeCtx &X, const DrawRow &Q, const DrawRow &P, float c, double dc,
                                        TreeShared &S, double &err) {
    ff acc = {0.f, 0.f};
    for_pair<ES>(X, Q.row, P.row, [&](float xq, float xp, int) {
        float yq, yp;
        const float wq = tw(Q, xq, yq), wp = tw(P, xp, yp);
        acc = ff_add_f(acc, fmaxf(fmaf(-c, wp, wq), 0.f));
    });
    const ff R = cluster_sum_ff(X, acc, S);
    // the positive part is 1-Lipschitz: sum_v |dq_v| + c |dp_v| + |dc| p_v, plus the sums
    // (evaluated by thread 0 only, which takes the decisions)
    err = 0.0;
    if (threadIdx.x == 0)
        err = (base_err(Q) + kTreeKappa * Q.ay) + (double)c * (base_err(P) + kTreeKappa * P.ay) + dc +
              8.0 * kU32 * (1.0 + (double)c) + 1e-12;
    return R.hi + R.lo;
}

template <int ES>
__device__ __forceinline__ ff tree_R_exact(TreeCtx &X, const char *rq, const char *rp, ff c_, int r_q, int r_p, ff iq,
                                           ff ip, ff c, TreeShared &S) {
    ff acc = {0.f, 0.f};
    for_pair<ES>(X, rq, rp, [&](float xq, float xp, int) {
        const ff d = ff_sub(twx(xq, c_, r_q, iq, S.tab), ff_mul(c, twx(xp, c_, r_p, ip, S.tab)));
        if (d.hi > 0.f) acc = ff_add(acc, d);
    });
    return cluster_sum_ff(X, acc, S);
}

// Inverse-CDF draw over w_v = (q_v - c p_v)+ (c = 0: q) in id order: t* = min{v : C(v) > u R}.
// Segments of contiguous words, one per thread of the cluster in id order; float32 sums into
// float-float per thread, a float-float scan over the cluster; the owning thread rescans its
// segment.  Returns t* and whether the margin certifies it (float32 weights); with EXACT the
// weights are float-float.
template <int ES, bool EXACT>
__device__ __forceinline__ int tree_draw(TreeCtx &X, const DrawRow &Q, const DrawRow &P, float c, double dc,
                                         double u, ff c_, int r_q, int r_p, ff iq, ff ip, ff cx, TreeShared &S,
                                         bool &certain) {
    constexpr int EPV = 16 / ES;
    const int n_vec = X.n_vec, V = X.V;
    const int per = (n_vec + kThreads * kTreeCluster - 1) / (kThreads * kTreeCluster);   // words per segment
    const int g = X.rank * kThreads + (int)threadIdx.x;
    const int w0 = min(n_vec, g * per), w1 = min(n_vec, w0 + per);
    const bool last = g == kThreads * kTreeCluster - 1;
    auto weight = [&](float xq, float xp) -> ff {
        if constexpr (EXACT) {
            const ff d = ff_sub(twx(xq, c_, r_q, iq, S.tab), ff_mul(cx, twx(xp, c_, r_p, ip, S.tab)));
            return d.hi > 0.f ? d : ff{0.f, 0.f};
        } else {
            float yq, yp;
            const float wq = tw(Q, xq, yq), wp = c > 0.f ? tw(P, xp, yp) : 0.f;
            return {fmaxf(fmaf(-c, wp, wq), 0.f), 0.f};
        }
    };
    ff seg = {0.f, 0.f};
    for (int wi = w0; wi < w1; ++wi) {
        const uint4 gq = __ldg(reinterpret_cast<const uint4 *>(Q.row) + wi);
        const uint4 gp = __ldg(reinterpret_cast<const uint4 *>(P.row) + wi);
        float xq[EPV], xp[EPV];
        unpack<ES>(gq, xq);
        unpack<ES>(gp, xp);
        if constexpr (EXACT) {
#pragma unroll
            for (int k = 0; k < EPV; ++k) seg = ff_add(seg, weight(xq[k], xp[k]));
        } else {
            float ws = 0.f;
#pragma unroll
            for (int k = 0; k < EPV; ++k) ws += weight(xq[k], xp[k]).hi;
            seg = ff_add_f(seg, ws);
        }
    }
    if (last)
        for (int v = n_vec * EPV; v < V; ++v) seg = ff_add(seg, weight(load_elem<ES>(Q.row, v), load_elem<ES>(P.row, v)));
    // inclusive scan of the segment sums in thread order, then over the blocks in rank order
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    ff inc = seg;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const ff t = {__shfl_up_sync(0xFFFFFFFFu, inc.hi, o), __shfl_up_sync(0xFFFFFFFFu, inc.lo, o)};
        if (lane >= o) inc = ff_add(t, inc);
    }
    __syncthreads();
    if (lane == 31) {
        S.s_hi[warp] = inc.hi;
        S.s_lo[warp] = inc.lo;
    }
    __syncthreads();
    ff base = {0.f, 0.f}, blk = {0.f, 0.f};
    for (int i = 0; i < kWarps; ++i) {
        if (i < warp) base = ff_add(base, {S.s_hi[i], S.s_lo[i]});
        blk = ff_add(blk, {S.s_hi[i], S.s_lo[i]});
    }
    if (threadIdx.x == 0) {
        S.part = make_float2(blk.hi, blk.lo);
        S.owner = kThreads;
        S.result = -1;
    }
    X.cl.sync();
    ff before_blocks = {0.f, 0.f}, R = {0.f, 0.f};
    for (int q = 0; q < kTreeCluster; ++q) {
        const float2 pq = *X.cl.map_shared_rank(&S.part, q);
        if (q < X.rank) before_blocks = ff_add(before_blocks, {pq.x, pq.y});
        R = ff_add(R, {pq.x, pq.y});
    }
    inc = ff_add(before_blocks, ff_add(base, inc));
    const ff Xu = ff_mul({(float)u, (float)(u - (double)(float)u)}, R);
    const ff excl = ff_sub(inc, seg);
    if (ff_diff(inc, Xu) > 0.f && seg.hi > 0.f) atomicMin(&S.owner, (int)threadIdx.x);
    X.cl.sync();
    int owner_rank = -1, owner_t = kThreads;
    for (int q = 0; q < kTreeCluster && owner_rank < 0; ++q) {
        const int o = *X.cl.map_shared_rank(&S.owner, q);
        if (o < kThreads) {
            owner_rank = q;
            owner_t = o;
        }
    }
    if (X.rank == owner_rank && (int)threadIdx.x == owner_t) {
        ff C = excl;
        int t_star = -1;
        ff before = excl;
        auto step = [&](float xq, float xp, int v) {
            if (t_star >= 0) return;
            const ff w = weight(xq, xp);
            if (!(w.hi > 0.f)) return;
            before = C;
            C = ff_add(C, w);
            if (ff_diff(C, Xu) > 0.f) t_star = v;
        };
        for (int wi = w0; wi < w1 && t_star < 0; ++wi) {
            const uint4 gq = __ldg(reinterpret_cast<const uint4 *>(Q.row) + wi);
            const uint4 gp = __ldg(reinterpret_cast<const uint4 *>(P.row) + wi);
            float xq[EPV], xp[EPV];
            unpack<ES>(gq, xq);
            unpack<ES>(gp, xp);
#pragma unroll
            for (int k = 0; k < EPV; ++k) step(xq[k], xp[k], wi * EPV + k);
        }
        if (last)
            for (int v = n_vec * EPV; v < V && t_star < 0; ++v) step(load_elem<ES>(Q.row, v), load_elem<ES>(P.row, v), v);
        S.result = t_star;
        S.c_at = make_float2(C.hi, C.lo);
        S.c_before = make_float2(before.hi, before.lo);
    }
    X.cl.sync();
    int t_star = -1;
    float2 c_at = make_float2(0.f, 0.f), c_bf = make_float2(0.f, 0.f);
    if (owner_rank >= 0) {
        TreeShared *O = X.cl.map_shared_rank(&S, owner_rank);
        t_star = O->result;
        c_at = O->c_at;
        c_bf = O->c_before;
    }
    X.cl.sync();   // the owner's results are read before any block moves on
    int ok = 0;
    if (threadIdx.x == 0) {
        const double Xd = ff_to_double(Xu), Rd = ff_to_double(R);
        const double ca = (double)c_at.x + c_at.y, cb = (double)c_bf.x + c_bf.y;
        if (owner_rank < 0 || t_star < 0) {   // rounding left u R at or beyond the total
            ok = 0;
        } else if (EXACT) {
            ok = !(fabs(ca - Xd) < 1e-11 * Rd || fabs(Xd - cb) < 1e-11 * Rd);
        } else {
            // max(u, 1-u) times the summed per-token errors, the float32 word sums and the scans
            const double tok = (base_err(Q) + kTreeKappa * Q.ay) + (double)c * (base_err(P) + kTreeKappa * P.ay) + dc;
            const double E = fmax(u, 1.0 - u) * tok + 8.1 * kU32 * (ca + u * Rd) + 1e-9 * Rd + 1e-30;
            ok = (ca - Xd) > E && (Xd - cb) > E;
        }
    }
    certain = block_bcast(ok, S) != 0;
    if (owner_rank < 0) t_star = -1;
    return t_star;
}

// Per sequence: the walk through the tree (one cluster of kTreeCluster blocks; every block takes
// the same decisions from the same values, each streams its slice of the rows).
template <int ES>
__global__ void __cluster_dims__(kTreeCluster, 1, 1) __launch_bounds__(kThreads) k_tree_walk(const TreeArgs a) {
    __shared__ TreeShared S;
    __shared__ int s_first[SV_MAX_TREE + 1], s_next[SV_MAX_TREE + 1], s_tok[SV_MAX_TREE + 1];
    __shared__ int s_err, s_errcode;
    const int b = blockIdx.x / kTreeCluster, N = a.N, V = a.V;
    TreeCtx X{cooperative_groups::this_cluster(), 0, a.n_vec, V, 0, 0, false};
    X.rank = (int)X.cl.block_rank();
    {
        const int per = (a.n_vec + kTreeCluster - 1) / kTreeCluster;
        X.w0 = min(a.n_vec, X.rank * per);
        X.w1 = min(a.n_vec, X.w0 + per);
        X.tail = X.rank == kTreeCluster - 1;
    }
    const float T = a.temperature[b];
    const bool greedy = T == 0.0f;
    int32_t *outs = a.out_tokens + (size_t)b * (N + 1);
    int32_t *pth = a.path ? a.path + (size_t)b * N : nullptr;
    S.tab[threadIdx.x] = kExp2Table[threadIdx.x];
    if (threadIdx.x == 0) {
        s_err = 0;
        s_errcode = 0;
        if (!(greedy || (T >= 1e-3f && T <= 1e3f))) {
            s_err = 1;
            s_errcode = SV_ERR_INVALID_ARG;
        }
        for (int i = 0; i <= N; ++i) s_first[i] = -1;
        for (int i = N; i >= 1 && !s_err; --i) {   // descending: each list ends up ascending
            const int p = a.parents[(size_t)b * N + i - 1], t = a.tokens[(size_t)b * N + i - 1];
            if (p < 0 || p >= i) {
                s_err = 1;
                s_errcode = SV_ERR_INVALID_ARG;
            } else if (t < 0 || t >= V) {
                s_err = 1;
                s_errcode = SV_ERR_BAD_TOKEN;
            } else {
                s_tok[i] = t;
                s_next[i] = s_first[p];
                s_first[p] = i;
            }
        }
        if (!s_err) {   // rows the walk may read must be finite
            for (int i = 0; i <= N && !s_err; ++i) {
                const RowStat rt = a.rowstat[(long long)b * (N + 1) + i];
                bool ok = rt.flags == 0 && (greedy ? isfinite(rt.maxv) : rs_sampled_ok(rt));
                if (!greedy && s_first[i] >= 0) {
                    const RowStat rd = a.rowstat[a.n_rows0 + (long long)b * (N + 1) + i];
                    ok = ok && rd.flags == 0 && rs_sampled_ok(rd);
                }
                if (!ok) {
                    s_err = 1;
                    s_errcode = SV_ERR_NONFINITE;
                }
            }
        }
        if (s_err && X.rank == 0) report_error(a.stats, s_errcode, b);
    }
    __syncthreads();
    if (s_err || (greedy && X.rank != 0)) {   // (greedy: block 0 walks alone; no block reads another's memory)
        if (!s_err) return;
        if (X.rank != 0) return;
        if (threadIdx.x == 0) a.accept_len[b] = 0;
        for (int j = threadIdx.x; j <= N; j += kThreads) outs[j] = -1;
        if (pth)
            for (int j = threadIdx.x; j < N; j += kThreads) pth[j] = -1;
        return;
    }
    int node = 0, k = 0, t_star = -1;
    long long tests = 0;
    int exact_nodes = 0, unresolved = 0;
    if (greedy) {
        if (threadIdx.x == 0) {
            while (true) {
                const int am = a.rowstat[(long long)b * (N + 1) + node].argmax;
                int nxt = -1;
                for (int c = s_first[node]; c >= 0; c = s_next[c])
                    if (s_tok[c] == am) {
                        nxt = c;
                        break;
                    }
                if (nxt < 0) {
                    t_star = am;
                    break;
                }
                if (pth) pth[k] = nxt;
                outs[k++] = s_tok[nxt];
                node = nxt;
            }
        }
    } else {
        const double *ub = a.uniforms + (size_t)b * (N + 1);
        while (true) {
            const long long rt = (long long)b * (N + 1) + node, rd = a.n_rows0 + rt;
            const char *rowq = a.tgt.base + ((long long)b * a.tgt.rows_per_seq + node) * a.tgt.pitch_bytes;
            const char *rowp = a.drf.base + ((long long)b * a.drf.rows_per_seq + node) * a.drf.pitch_bytes;
            const bool has_children = s_first[node] >= 0;
            if (threadIdx.x == 0) {
                S.q = draw_row(rowq, T, a.rowstat[rt], nullptr, nullptr, 1.0f);
                S.p = has_children ? draw_row(rowp, T, a.rowstat[rd], nullptr, nullptr, 1.0f) : S.q;
            }
            __syncthreads();
            const DrawRow Q = S.q, P = S.p;
            // ---- float32 tier ----
            float c = 0.f, R = 1.f;
            double dc = 0.0, dR = 0.0;
            bool exact = false;
            int nxt = -1;
            for (int ch = s_first[node]; ch >= 0 && !exact; ch = s_next[ch]) {
                ++tests;
                // the test, by thread 0: 0 reject, 1 accept, 2 too close to call
                int dec = 0;
                if (threadIdx.x == 0) {
                    const int t = s_tok[ch];
                    const double ut = ub[ch];
                    float yq, yp;
                    const float qt = tw(Q, load_elem<ES>(rowq, t), yq), pt = tw(P, load_elem<ES>(rowp, t), yp);
                    const double eq = base_err(Q) + kTreeKappa * fabsf(yq), ep = base_err(P) + kTreeKappa * fabsf(yp);
                    const double num = (double)qt - (double)c * (double)pt;
                    const double lhs = ut * (double)R * (double)pt;
                    const double E = ut * ((double)R * pt * ep + pt * dR) + qt * eq + (double)c * pt * ep + pt * dc +
                                     4.0 * kU32 * (qt + (double)c * pt + lhs) + 1e-40;
                    const double rhs = fmax(num, 0.0);
                    if (fabs(lhs - rhs) <= E || (pt == 0.f && fabs(num) <= E)) dec = 2;
                    else dec = lhs < rhs ? 1 : 0;
                }
                dec = block_bcast(dec, S);
                if (dec == 2) {
                    exact = true;
                    break;
                }
                if (dec == 1) {
                    nxt = ch;
                    break;
                }
                // rejected: c <- c + R(c); R <- R(c)
                const float c_new = c + R;
                const double dc_new = threadIdx.x == 0 ? dc + dR + kU32 * (double)c_new : 0.0;
                double eR;
                const float R_new = tree_R<ES>(X, Q, P, c_new, dc_new, S, eR);
                if (!block_bcast((double)R_new > eR, S)) {   // cannot tell the residual from empty
                    exact = true;
                    break;
                }
                c = c_new;
                dc = dc_new;
                R = R_new;
                dR = eR;
            }
            if (!exact && nxt < 0) {   // every child failed (or none): the draw
                bool certain = false;
                const int t = tree_draw<ES, false>(X, Q, P, c, dc, ub[0], {0.f, 0.f}, 0, 0, {0.f, 0.f}, {0.f, 0.f},
                                                   {0.f, 0.f}, S, certain);
                if (certain) t_star = t;
                else exact = true;
            }
            // ---- float-float tier: the whole node again ----
            if (exact) {
                ++exact_nodes;
                nxt = -1;
                t_star = -1;
                float c_hi, c_lo;
                log2e_over(T, c_hi, c_lo);
                const ff c_ = {c_hi, c_lo};
                const int r_q = a.rowstat[rt].r, r_p = has_children ? a.rowstat[rd].r : r_q;
                ff sq = {0.f, 0.f}, sp = {0.f, 0.f};
                for_pair<ES>(X, rowq, rowp, [&](float xq, float xp, int) {
                    if (xq != -INFINITY) sq = ff_add(sq, ff_exp2_xc(xq, c_, r_q, S.tab));
                    if (has_children && xp != -INFINITY) sp = ff_add(sp, ff_exp2_xc(xp, c_, r_p, S.tab));
                });
                const ff Sq = cluster_sum_ff(X, sq, S);
                const ff Sp = cluster_sum_ff(X, sp, S);
                const ff iq = ff_recip(Sq), ip = has_children ? ff_recip(Sp) : ff{0.f, 0.f};
                ff cx = {0.f, 0.f}, Rx = {1.f, 0.f};
                for (int ch = s_first[node]; ch >= 0; ch = s_next[ch]) {
                    const int t = s_tok[ch];
                    const ff qt = twx(load_elem<ES>(rowq, t), c_, r_q, iq, S.tab);
                    const ff pt = twx(load_elem<ES>(rowp, t), c_, r_p, ip, S.tab);
                    const double num = ff_to_double(ff_sub(qt, ff_mul(cx, pt)));
                    const double lhs = ub[ch] * ff_to_double(ff_mul(Rx, pt));
                    const double rhs = fmax(num, 0.0);
                    if (fabs(lhs - rhs) < 1e-11 * fmax(ff_to_double(qt), 1e-300)) ++unresolved;
                    if (lhs < rhs) {
                        nxt = ch;
                        break;
                    }
                    const ff c_next = ff_add(cx, Rx);
                    const ff R_next = tree_R_exact<ES>(X, rowq, rowp, c_, r_q, r_p, iq, ip, c_next, S);
                    if (!(R_next.hi > 0.f)) {   // empty residual after rounding: draw from q
                        cx = {0.f, 0.f};
                        Rx = {1.f, 0.f};
                        break;
                    }
                    cx = c_next;
                    Rx = R_next;
                }
                if (nxt < 0) {
                    bool certain = true;
                    const int t = tree_draw<ES, true>(X, Q, P, 0.f, 0.0, ub[0], c_, r_q, r_p, iq, ip, cx, S, certain);
                    if (!certain) ++unresolved;
                    t_star = t >= 0 ? t : a.rowstat[rt].argmax;
                }
            }
            if (nxt < 0) break;
            if (threadIdx.x == 0 && X.rank == 0) {
                if (pth) pth[k] = nxt;
                outs[k] = s_tok[nxt];
            }
            ++k;
            node = nxt;
        }
    }
    __syncthreads();
    if (!greedy) X.cl.sync();   // no block leaves while another may read its shared memory
    if (X.rank != 0) return;
    if (threadIdx.x == 0) {   // (greedy: k and t_star come from thread 0's walk)
        a.accept_len[b] = k;
        outs[k] = t_star;
        for (int j = k + 1; j <= N; ++j) outs[j] = -1;
        if (pth)
            for (int j = k; j < N; ++j) pth[j] = -1;
        stats_add(a.stats, &a.stats->rows, greedy ? N + 1 : 2 * (N + 1));
        if (!greedy) {
            stats_add(a.stats, &a.stats->accept_tests, tests);
            if (exact_nodes) stats_add(a.stats, &a.stats->reresolved, exact_nodes);
            if (unresolved) stats_add(a.stats, &a.stats->unresolved, unresolved);
        }
    }
}

// ---- reuse check ---------------------------------------------------------------------------
__global__ void k_tree_reuse(const int32_t *parents, const int32_t *tokens, int N, const int32_t *accept_len,
                             const int32_t *out_tokens, int K, int B, int32_t *reuse_node) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int kk = accept_len[b];
    int node = 0;
    if (kk < 0 || kk > K) {
        reuse_node[b] = -1;
        return;
    }
    for (int j = 0; j <= kk && node >= 0; ++j) {
        const int t = out_tokens[(size_t)b * (K + 1) + j];
        int nxt = -1;
        for (int i = node + 1; i <= N; ++i)   // children of node, lowest index first
            if (parents[(size_t)b * N + i - 1] == node && tokens[(size_t)b * N + i - 1] == t) {
                nxt = i;
                break;
            }
        node = nxt;
    }
    reuse_node[b] = node > 0 ? node : -1;
}

struct TreePlan {
    int n_split = 1, chunk_vecs = 1, n_vec = 0;
    long long n_rows0 = 0, n_rows1 = 0;
    size_t off_counters = 0, off_part = 0, off_rowstat = 0, bytes = 0;
};

static TreePlan plan_tree(int B, int N, int V, int es) {
    TreePlan p;
    p.n_rows0 = (long long)B * (N + 1);
    p.n_rows1 = p.n_rows0;
    const long long n_rows = p.n_rows0 + p.n_rows1;
    p.n_split = choose_split(n_rows, (long long)V * es);
    p.n_vec = vec_count(V, es);
    chunk_geometry(p.n_vec, p.n_split, p.chunk_vecs);
    Carver cv;
    p.off_counters = cv.take<Counters>(1);
    p.off_part = cv.take<WarpPartial>((size_t)n_rows * p.n_split * kWarps);
    p.off_rowstat = cv.take<RowStat>((size_t)n_rows);
    p.bytes = cv.off + 256;
    return p;
}

template <int ES>
static sv_status launch_tree(const TreePlan &pl, TreeArgs ta, void *ws, cudaStream_t stream) {
    DeviceInfo di;
    if (!device_info(di)) return SV_ERR_CUDA;
    char *w = static_cast<char *>(ws);
    StatsArgs sa;
    sa.set[0] = ta.tgt;
    sa.set[1] = ta.drf;
    sa.n_sets = 2;
    sa.V = ta.V;
    sa.temperature = ta.temperature;
    sa.n_split = pl.n_split;
    sa.chunk_vecs = pl.chunk_vecs;
    sa.n_rows0 = pl.n_rows0;
    sa.n_units = (pl.n_rows0 + pl.n_rows1) * pl.n_split;
    sa.part = reinterpret_cast<WarpPartial *>(w + pl.off_part);
    sa.counters = reinterpret_cast<Counters *>(w + pl.off_counters);
    sa.stats = ta.stats;
    sa.wait_limit = kWaitLimitCycles;
    {
        const sv_status st = launch_stats<ES>(sa, di, stream);
        if (st != SV_OK) return st;
    }
    ta.part = sa.part;
    ta.n_split = pl.n_split;
    ta.n_rows0 = pl.n_rows0;
    ta.n_rows = pl.n_rows0 + pl.n_rows1;
    ta.rowstat = reinterpret_cast<RowStat *>(w + pl.off_rowstat);
    ta.n_vec = pl.n_vec;
    k_tree_rowstats<<<(unsigned)div_up(ta.n_rows, kWarps), kThreads, 0, stream>>>(ta);
    k_tree_walk<ES><<<(unsigned)ta.B * kTreeCluster, kThreads, 0, stream>>>(ta);
    return cuda_status(cudaGetLastError());
}

}  // namespace sv

using namespace sv;

extern "C" size_t sv_tree_verify_workspace_size(int B, int N, int V) {
    if (B < 1 || N < 0 || N > SV_MAX_TREE || V < 1) return 0;
    const TreePlan a = plan_tree(B, N, V, 4), b = plan_tree(B, N, V, 2);
    return a.bytes > b.bytes ? a.bytes : b.bytes;
}

extern "C" sv_status sv_tree_verify(const void *target_logits, int64_t t_row_pitch, const void *draft_logits,
                                    int64_t d_row_pitch, sv_dtype dtype, const int32_t *parents,
                                    const int32_t *tokens, const double *uniforms, int B, int N, int V,
                                    const float *temperature, int32_t *accept_len, int32_t *out_tokens,
                                    int32_t *path, sv_stats *stats, void *workspace, size_t workspace_bytes,
                                    sv_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (B < 1 || N < 0 || N > SV_MAX_TREE || V < 1) return SV_ERR_INVALID_ARG;
    if (!rows_ok(target_logits, t_row_pitch, V, dtype) || !rows_ok(draft_logits, d_row_pitch, V, dtype))
        return SV_ERR_INVALID_ARG;
    if ((N > 0 && (parents == nullptr || tokens == nullptr)) || uniforms == nullptr || temperature == nullptr)
        return SV_ERR_INVALID_ARG;
    if (accept_len == nullptr || out_tokens == nullptr) return SV_ERR_INVALID_ARG;
    if ((long long)V * B * 2 * (N + 1) > (1LL << 46)) return SV_ERR_INVALID_ARG;
    const int es = elem_size(dtype);
    const TreePlan pl = plan_tree(B, N, V, es);
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < pl.bytes) return SV_ERR_WORKSPACE;
    if (!on_current_device(stream, target_logits, draft_logits)) return SV_ERR_INVALID_ARG;
    if (stats && cudaMemsetAsync(stats, 0, sizeof(sv_stats), stream) != cudaSuccess) return SV_ERR_CUDA;
    TreeArgs ta{};
    ta.tgt = {static_cast<const char *>(target_logits), t_row_pitch * es, N + 1, N + 1, 0};
    ta.drf = {static_cast<const char *>(draft_logits), d_row_pitch * es, N + 1, N + 1, 1};
    ta.B = B;
    ta.N = N;
    ta.V = V;
    ta.parents = parents;
    ta.tokens = tokens;
    ta.uniforms = uniforms;
    ta.temperature = temperature;
    ta.accept_len = accept_len;
    ta.out_tokens = out_tokens;
    ta.path = path;
    ta.stats = stats;
    if (es == 4) return launch_tree<4>(pl, ta, workspace, stream);
    return launch_tree<2>(pl, ta, workspace, stream);
}

extern "C" sv_status sv_tree_reuse(const int32_t *parents, const int32_t *tokens, int N, const int32_t *accept_len,
                                   const int32_t *out_tokens, int K, int B, int32_t *reuse_node, sv_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (B < 1 || N < 0 || K < 0 || accept_len == nullptr || out_tokens == nullptr || reuse_node == nullptr)
        return SV_ERR_INVALID_ARG;
    if (N > 0 && (parents == nullptr || tokens == nullptr)) return SV_ERR_INVALID_ARG;
    if (!on_current_device(stream, accept_len, reuse_node)) return SV_ERR_INVALID_ARG;
    k_tree_reuse<<<(unsigned)div_up(B, 128), 128, 0, stream>>>(parents, tokens, N, accept_len, out_tokens, K, B,
                                                               reuse_node);
    return cuda_status(cudaGetLastError());
}
