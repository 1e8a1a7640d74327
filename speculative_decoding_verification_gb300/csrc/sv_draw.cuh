// sv_draw.cuh — inverse-CDF draws in token-id order, float32 tier with a certified error bound.
//
// A draw item names one or two rows and a uniform u.  Its weights are
//     w_v = max(q_v - p_v, 0)   (residual: SSD notes §2.2 ③; SpS notes §3)   or   w_v = q_v  (bonus),
// with q_v = keep_q(v) 2^(x_v c - r_q) inv_q and p_v = keep_p(v) 2^(y_v c - r_p) inv_p (C for v in
// the Saguaro top-F set).  The token is t* = min{v : w_0 + ... + w_v > u R}, R = sum_v w_v.
//
// Pass 1 (k_draw_sums): a persistent grid streams the rows through bulk copies and writes, per
// 32-vector sub-chunk of the row, the float32 sum of w and of the error weights
// q_v |y_q| + p_v |y_p|.  Pass 2 (k_draw_finish): one block per item scans the sub-chunk sums
// in float64, locates the sub-chunk that holds u R, recomputes its tokens' weights exactly as
// pass 1 did, and picks t*.  If u R lies within the proven error bound of either boundary of
// t*, the item is queued for the float-float tier.
#pragma once

#include "sv_device.cuh"
#include "sv_host.h"
#include "sv_stats.cuh"

namespace sv {

struct DrawArgs {
    const DrawItem *items;
    Counters *counters;
    int V, n_vec, n_sub;        // n_sub = vector sub-chunks + 1 tail sub-chunk
    int n_split;                // chunks per row
    int subs_per_chunk;         // vector sub-chunks per chunk
    float *subs;                // [item][n_sub] = float32 sum of w over the sub-chunk
    ExactItem *exact;           // exact-tier queue (may be nullptr: no re-resolution)
    int *exact_unc;             // per queued item: uncertain-token count, zeroed at push
    sv_stats *stats;
    long long wait_limit;
};

// Per-element weight (identical in both passes).  The exponent x c_hi - r is rounded once;
// the low part of c enters as the factor 1 + ln2 c_lo x (first order), folded into the
// normaliser: t = inv_s + x (ln2 c_lo inv_s).  x is clamped below (see the callers), so t is
// finite wherever 2^y > 0.
template <bool HAS_P, bool FILT>
__device__ __forceinline__ float draw_weight(const DrawItem &it, float xq, float xp, int v) {
    float eq = ex2_fast(fmaf(xq, it.q.c_hi, -it.q.rf));
    float tq = fmaf(xq, it.q.k_lo, it.q.inv_s);
    if (FILT) {
        const bool keep = xq > it.q.cut_x || (xq == it.q.cut_x && v <= it.q.cut_id);
        const bool in_d = xq > it.q.top_x || (xq == it.q.top_x && v <= it.q.top_id);
        eq = keep ? eq : 0.0f;
        tq = in_d ? __fmul_rn(tq, it.q.sc_d) : tq;
    }
    if (HAS_P) {
        float ep = ex2_fast(fmaf(xp, it.p.c_hi, -it.p.rf));
        float tp = fmaf(xp, it.p.k_lo, it.p.inv_s);
        if (FILT) {
            const bool keep = xp > it.p.cut_x || (xp == it.p.cut_x && v <= it.p.cut_id);
            const bool in_d = xp > it.p.top_x || (xp == it.p.top_x && v <= it.p.top_id);
            ep = keep ? ep : 0.0f;
            tp = in_d ? __fmul_rn(tp, it.p.sc_d) : tp;
        }
        const float pv = __fmul_rn(ep, tp);
        return fmaxf(__fmaf_rn(eq, tq, -pv), 0.0f);
    }
    return __fmul_rn(eq, tq);
}

// Logits below this weigh exactly 0 at every allowed temperature; clamping them there keeps
// the factor t above finite (a -inf logit would otherwise give 0 * inf).
constexpr uint32_t kDrawFloor2 = 0xF149F149u;   // bf16 pair (-9.95e29, -9.95e29)
constexpr float kDrawFloor = -9.95e29f;

// Weights of one vector (EPV tokens from element e0); returns their tree sum.  bf16 rows
// without filters take the packed path: two tokens per f32x2 instruction, each rounded exactly
// as draw_weight rounds it (fma.rn.f32x2 is two IEEE fmas; x k_lo + inv_s and ep tp are formed
// negated for p, which round-to-nearest mirrors exactly), so both passes see the same weights.
template <int ES, bool HAS_P, bool FILT>
__device__ __forceinline__ float vec_weights(const DrawItem &it, uint4 wq, uint4 wp, int e0, float (&wv)[16 / ES]) {
    constexpr int EPV = 16 / ES;
    if constexpr (ES == 2 && !FILT) {
        const f32x2 chq = f2_pack(it.q.c_hi, it.q.c_hi), nrq = f2_pack(-it.q.rf, -it.q.rf);
        const f32x2 klq = f2_pack(it.q.k_lo, it.q.k_lo), isq = f2_pack(it.q.inv_s, it.q.inv_s);
        const f32x2 chp = f2_pack(it.p.c_hi, it.p.c_hi), nrp = f2_pack(-it.p.rf, -it.p.rf);
        const f32x2 nklp = f2_pack(-it.p.k_lo, -it.p.k_lo), nisp = f2_pack(-it.p.inv_s, -it.p.inv_s);
        const f32x2 zero2 = f2_pack(0.f, 0.f);
        const uint32_t qw[4] = {wq.x, wq.y, wq.z, wq.w};
        const uint32_t pw[4] = {wp.x, wp.y, wp.z, wp.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const f32x2 xq = f2_from_bf16x2(bmax2(qw[h], kDrawFloor2));
            const f32x2 eq = f2_ex2(f2_fma(xq, chq, nrq));
            const f32x2 tq = f2_fma(xq, klq, isq);
            float w0, w1;
            if (HAS_P) {
                const f32x2 xp = f2_from_bf16x2(bmax2(pw[h], kDrawFloor2));
                const f32x2 ep = f2_ex2(f2_fma(xp, chp, nrp));
                const f32x2 ntp = f2_fma(xp, nklp, nisp);   // -(x k_lo + inv_s)
                const f32x2 npv = f2_fma(ep, ntp, zero2);   // -(ep tp)
                f2_unpack(f2_fma(eq, tq, npv), w0, w1);
                w0 = fmaxf(w0, 0.0f);
                w1 = fmaxf(w1, 0.0f);
            } else {
                f2_unpack(f2_fma(eq, tq, zero2), w0, w1);
            }
            wv[2 * h] = w0;
            wv[2 * h + 1] = w1;
        }
        return ((wv[0] + wv[1]) + (wv[2] + wv[3])) + ((wv[4] + wv[5]) + (wv[6] + wv[7]));
    }
    float xq[EPV], xp[EPV];
    if constexpr (ES == 2) {
        unpack<ES>(make_uint4(bmax2(wq.x, kDrawFloor2), bmax2(wq.y, kDrawFloor2), bmax2(wq.z, kDrawFloor2),
                              bmax2(wq.w, kDrawFloor2)), xq);
        if (HAS_P)
            unpack<ES>(make_uint4(bmax2(wp.x, kDrawFloor2), bmax2(wp.y, kDrawFloor2), bmax2(wp.z, kDrawFloor2),
                                  bmax2(wp.w, kDrawFloor2)), xp);
    } else {
        unpack<ES>(wq, xq);
        if (HAS_P) unpack<ES>(wp, xp);
#pragma unroll
        for (int i = 0; i < EPV; ++i) {
            xq[i] = fmaxf(xq[i], kDrawFloor);
            xp[i] = HAS_P ? fmaxf(xp[i], kDrawFloor) : xq[i];
        }
    }
#pragma unroll
    for (int i = 0; i < EPV; ++i) wv[i] = draw_weight<HAS_P, FILT>(it, xq[i], HAS_P ? xp[i] : xq[i], e0 + i);
    if constexpr (EPV == 8) {
        return ((wv[0] + wv[1]) + (wv[2] + wv[3])) + ((wv[4] + wv[5]) + (wv[6] + wv[7]));
    } else {
        return (wv[0] + wv[1]) + (wv[2] + wv[3]);
    }
}

// One consumer warp's share of a tile: 32-vector groups g = warp, warp + kWarps, ...; each
// group is one sub-chunk, whose sum lane 0 writes.
template <int ES, bool HAS_P, bool FILT>
__device__ __forceinline__ void draw_tile(const DrawItem &it, const unsigned char *bq, const unsigned char *bp,
                                          int fv, int nv, float *subs_item) {
    constexpr int EPV = 16 / ES;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll 1
    for (int g = warp; g * 32 < nv; g += kWarps) {
        const int vi = g * 32 + lane;
        float w = 0.f;
        if (vi < nv) {
            const uint4 q = lds128(bq + vi * 16);
            const uint4 p = HAS_P ? lds128(bp + vi * 16) : q;
            float wv[EPV];
            w = vec_weights<ES, HAS_P, FILT>(it, q, p, (fv + vi) * EPV, wv);
        }
        const float W = warp_sum_f(w);
        if (lane == 0) subs_item[(fv + g * 32) / 32] = W;
    }
}

template <int ES>
__device__ __forceinline__ float draw_scalar(const DrawItem &it, int v) {
    const float xq = fmaxf(load_elem<ES>(it.q.row, v), kDrawFloor);
    const float xp = it.has_p ? fmaxf(load_elem<ES>(it.p.row, v), kDrawFloor) : xq;
    if (it.has_p) return it.filt ? draw_weight<true, true>(it, xq, xp, v) : draw_weight<true, false>(it, xq, xp, v);
    return it.filt ? draw_weight<false, true>(it, xq, xp, v) : draw_weight<false, false>(it, xq, xp, v);
}

// One pipeline stage of the draw pass: a q tile and (with a draft row) a p tile of one item.
struct DrawMeta {
    int d;            // item
    int fv, nv;       // first vector of the tile within the row, vectors in the tile
    int flags;        // kTileLast (last tile of the item's last chunk: also the scalar tail) | kTileEnd
};
constexpr int kDrawItemOff = 256;   // per stage: a copy of its item, bulk-copied with the tiles
constexpr int kDrawCtlBytes = 1024;
static_assert(2 * kDrawStages * 8 + 16 + kDrawStages * (int)sizeof(DrawMeta) <= kDrawItemOff, "control block");
static_assert(kDrawItemOff + kDrawStages * (int)sizeof(DrawItem) <= kDrawCtlBytes, "item copies");
constexpr size_t kDrawSmemBytes = (size_t)kDrawCtlBytes + (size_t)2 * kDrawStages * kTileBytes;

// Pass 1, warp-specialised like the statistics pass: the producer warp takes (item, chunk)
// units from a global counter and streams each unit's q and p tiles into shared memory, with a
// copy of the item itself in the same stage; eight consumer warps weight the tokens and write
// one float32 sum per 32-vector sub-chunk.
template <int ES>
__global__ void __launch_bounds__(kStatsThreads, 2) k_draw_sums(const DrawArgs a) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kDrawStages;
    int *abort_flag = reinterpret_cast<int *>(smem + 2 * kDrawStages * 8);
    DrawMeta *meta = reinterpret_cast<DrawMeta *>(smem + 2 * kDrawStages * 8 + 16);
    DrawItem *stage_item = reinterpret_cast<DrawItem *>(smem + kDrawItemOff);
    unsigned char *tiles = smem + kDrawCtlBytes;   // stage s: q tile at 2s, p tile at 2s+1
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int n_items = *reinterpret_cast<volatile int *>(&a.counters->n_draws);
    const int n_vsub = a.n_sub - 1;

    if (tid == 0) {
        for (int s = 0; s < kDrawStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kWarps) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t policy = policy_evict_first();
            const long long n_units = (long long)n_items * a.n_split;
            long long in_flight[kDrawStages];
            for (int s = 0; s < kDrawStages; ++s) in_flight[s] = -1;
            long long it = 0;           // tiles issued
            int st = 0;                 // it % kDrawStages
            uint32_t epar = 0;          // parity of the "empty" phase to wait for at stage st
            bool ok = true;
            // the next unit is claimed as soon as the current one is known, so that the claim's
            // round trip overlaps the current unit's copies
            long long u_next = atomicAdd(&a.counters->next_draw_unit, 1);
            while (ok) {
                const long long u = u_next;
                const bool have = u < n_units;
                if (have) u_next = atomicAdd(&a.counters->next_draw_unit, 1);
                int d = 0, c = 0, v0 = 0, v1 = 0;
                const DrawItem *item = nullptr;
                if (have) {
                    d = (int)(u / a.n_split);
                    c = (int)(u - (long long)d * a.n_split);
                    const int s0 = min(c * a.subs_per_chunk, n_vsub), s1 = min(s0 + a.subs_per_chunk, n_vsub);
                    v0 = s0 * 32;
                    v1 = max(v0, min(s1 * 32, a.n_vec));
                    item = a.items + d;
                }
                const int nt = have ? max((v1 - v0 + kTileBytes / 16 - 1) / (kTileBytes / 16), 1) : 1;
                for (int t = 0; t < nt; ++t, ++it) {
                    if (it >= kDrawStages) {
                        if (!mbar_wait_or_abort(&empty[st], epar, abort_flag, a.wait_limit)) {
                            if (atomicExch(abort_flag, 1) == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
                            ok = false;
                            break;
                        }
                    }
                    in_flight[st] = -1;
                    DrawMeta m;
                    if (!have) {
                        m.flags = kTileEnd;
                        meta[st] = m;
                        mbar_arrive(&full[st]);
                        ok = false;
                        break;
                    }
                    const int fv = v0 + t * (kTileBytes / 16);
                    const int nv = max(0, min(kTileBytes / 16, v1 - fv));
                    m.d = d;
                    m.fv = fv;
                    m.nv = nv;
                    m.flags = (t == nt - 1 && c == a.n_split - 1) ? kTileLast : 0;
                    meta[st] = m;
                    const uint32_t bytes = (uint32_t)nv * 16u;
                    const bool has_p = item->has_p != 0;
                    const uint32_t tile_bytes = nv > 0 ? (has_p ? 2u * bytes : bytes) : 0u;
                    mbar_arrive_expect_tx(&full[st], tile_bytes + (uint32_t)sizeof(DrawItem));
                    bulk_load(stage_item + st, item, (uint32_t)sizeof(DrawItem), &full[st]);
                    if (nv > 0) {
                        bulk_load_stream(tiles + (2 * st) * kTileBytes, item->q.row + (size_t)fv * 16, bytes, &full[st],
                                         policy);
                        if (has_p)
                            bulk_load_stream(tiles + (2 * st + 1) * kTileBytes, item->p.row + (size_t)fv * 16, bytes,
                                             &full[st], policy);
                    }
                    in_flight[st] = it;
                    if (++st == kDrawStages) {
                        st = 0;
                        if (it >= 2 * kDrawStages - 1) epar ^= 1u;   // round r >= 2 waits phase r - 1
                    }
                }
            }
            if (*reinterpret_cast<volatile int *>(abort_flag)) {
                for (int s = 0; s < kDrawStages; ++s)
                    if (in_flight[s] >= 0)
                        mbar_wait_bounded(&full[s], (uint32_t)((in_flight[s] / kDrawStages) & 1), a.wait_limit / 16);
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    int st = 0;
    uint32_t par = 0;
    for (;;) {
        if (!mbar_wait_or_abort(&full[st], par, abort_flag, a.wait_limit)) {
            if (lane == 0 && atomicExch(abort_flag, 1) == 0) report_error(a.stats, SV_ERR_TIMEOUT, -1);
            break;
        }
        const DrawMeta m = meta[st];
        if (m.flags & kTileEnd) break;
        const DrawItem item = stage_item[st];   // read before the stage is released below
        float *subs_item = a.subs + (size_t)m.d * a.n_sub;
        const unsigned char *bq = tiles + (2 * st) * kTileBytes;
        const unsigned char *bp = bq + kTileBytes;
        if (item.has_p) {
            if (item.filt) draw_tile<ES, true, true>(item, bq, bp, m.fv, m.nv, subs_item);
            else draw_tile<ES, true, false>(item, bq, bp, m.fv, m.nv, subs_item);
        } else {
            if (item.filt) draw_tile<ES, false, true>(item, bq, bp, m.fv, m.nv, subs_item);
            else draw_tile<ES, false, false>(item, bq, bp, m.fv, m.nv, subs_item);
        }
        // the scalar tail of the row forms the last sub-chunk
        if ((m.flags & kTileLast) && warp == 0) {
            constexpr int EPV = 16 / ES;
            const int t0 = a.n_vec * EPV;
            const float w = t0 + lane < a.V ? draw_scalar<ES>(item, t0 + lane) : 0.f;
            const float W = warp_sum_f(w);
            if (lane == 0) subs_item[n_vsub] = W;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        if (++st == kDrawStages) {
            st = 0;
            par ^= 1u;
        }
    }
}

// Block-wide scan of one float-float value per thread (kThreads threads, all of them calling):
// inclusive and exclusive prefix sums in thread order and the block total.  Warp scans by
// shuffles, then one warp scans the warp totals: three barriers.  s_w holds kWarps entries.
__device__ __forceinline__ void block_scan_ff(ff v, ff &incl, ff &excl, ff &total, float2 *s_w) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    ff inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float h = __shfl_up_sync(0xFFFFFFFFu, inc.hi, o);
        const float l = __shfl_up_sync(0xFFFFFFFFu, inc.lo, o);
        if (lane >= o) inc = ff_add(inc, {h, l});
    }
    if (lane == 31) s_w[warp] = make_float2(inc.hi, inc.lo);
    __syncthreads();
    if (warp == 0) {
        ff t = lane < kWarps ? ff{s_w[lane].x, s_w[lane].y} : ff{0.f, 0.f};
#pragma unroll
        for (int o = 1; o < kWarps; o <<= 1) {
            const float h = __shfl_up_sync(0xFFFFFFFFu, t.hi, o);
            const float l = __shfl_up_sync(0xFFFFFFFFu, t.lo, o);
            if (lane >= o) t = ff_add(t, {h, l});
        }
        __syncwarp();
        if (lane < kWarps) s_w[lane] = make_float2(t.hi, t.lo);   // inclusive warp prefixes
    }
    __syncthreads();
    const ff base = warp > 0 ? ff{s_w[warp - 1].x, s_w[warp - 1].y} : ff{0.f, 0.f};
    const float ph = __shfl_up_sync(0xFFFFFFFFu, inc.hi, 1), pl = __shfl_up_sync(0xFFFFFFFFu, inc.lo, 1);
    incl = ff_add(base, inc);
    excl = lane > 0 ? ff_add(base, {ph, pl}) : base;
    total = {s_w[kWarps - 1].x, s_w[kWarps - 1].y};
    __syncthreads();   // s_w may be reused by the caller
}

// Bound on |(u R~ - C~(v)) - (u R - C(v))| for any v, where ~ marks the computed prefix sums.
// With per-token errors d_v = |w~_v - w_v| the difference is (1-u) sum_{i<=v} d_i and
// u sum_{i>v} d_i of opposite signs at worst, so it is at most max(u, 1-u) sum_v d_v.  Each
// sub-chunk sum of non-negative terms has 8 float32 rounding levels (3 per 16-byte vector, 5
// across the warp) and the scans over sub-chunks are float-float, so C~(v) and u R~ carry at
// most 8u (C(v) + u R) between them; the caller passes C(v) + u R at the boundary it checks.
// sum_v d_v: the exponent x c_hi - r rounded once (ln2 u per unit |y|, summed as A), the
// exponential (kEx2RelErr), the factor t = inv_s (1 + ln2 c_lo x) (its rounding, and the
// second-order remainder (ln2 (|r| + 128) 2^-23)^2), the products (2u), and the rows'
// normaliser errors; for a bonus draw without filters a common normaliser error cancels.
// The float-float scans add well under 1e-9 R.  Evaluated in float32 and rounded up.
__device__ __forceinline__ float draw_error_bound(const DrawItem &it, float W, float A, float c_sum) {
    const float u = (float)kU32;
    const float ex = (float)kEx2RelErr;
    const float rq = ((float)kLn2 * 0x1p-23f) * (fabsf(it.q.rf) + 128.0f);
    const float rp = ((float)kLn2 * 0x1p-23f) * (fabsf(it.p.rf) + 128.0f);
    float e = (float)(kLn2 * kU32 * 1.01) * A;
    if (it.has_p) {
        e += 1.0001f * (ex + 3.0f * u + rq * rq + (float)it.q.norm_err) +
             1.0001f * (ex + 3.0f * u + rp * rp + (float)it.p.norm_err);
    } else if (it.filt) {
        // tokens inside and outside the scaled set carry different normaliser errors
        e += (ex + 3.0f * u + rq * rq + (float)it.q.norm_err) * W;
    } else {
        e += (ex + 2.0f * u + rq * rq) * W;
    }
    const float uu = (float)fmax(it.u, 1.0 - it.u);
    return (uu * e + 8.1f * u * c_sum + 1e-9f * W + 1e-30f) * (1.0f + 0x1p-18f);
}

// One block per item, float32 / float-float only: the sub-chunk sums are scanned in
// float-float, the sub-chunk holding u R is rescanned token by token, and t* is certified
// against draw_error_bound.
template <int ES>
__global__ void __launch_bounds__(kThreads) k_draw_finish(const DrawArgs a) {
    pdl_wait();
    constexpr int EPV = 16 / ES;
    __shared__ float2 s_w[kWarps];
    __shared__ int s_sub;
    __shared__ float2 s_pre;
    __shared__ int s_last_sub;
    __shared__ float2 s_u;   // u as float-float, split once (float64 on one thread)

    const int d = blockIdx.x;
    const int n_items = *reinterpret_cast<volatile int *>(&a.counters->n_draws);
    if (d >= n_items) return;
    const DrawItem it = a.items[d];
    const float *subs = a.subs + (size_t)d * a.n_sub;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_sub = a.n_sub, n_vsub = n_sub - 1;

    // 1. per-thread contiguous ranges of sub-chunks
    const int per = (n_sub + kThreads - 1) / kThreads;
    const int s0 = min(tid * per, n_sub), s1 = min(s0 + per, n_sub);
    ff wsum = {0.f, 0.f};
    int last_pos = -1;
    for (int s = s0; s < s1; ++s) {
        const float v = subs[s];
        wsum = ff_add_f(wsum, v);
        if (v > 0.f) last_pos = s;
    }
    // 2. block scan of wsum in float-float
    if (tid == 0) {
        s_sub = -1;
        s_last_sub = -1;
        const float u_hi = __double2float_rn(it.u);
        s_u = make_float2(u_hi, __double2float_rn(it.u - (double)u_hi));
    }
    ff incl, excl, R;
    block_scan_ff(wsum, incl, excl, R, s_w);
    atomicMax(&s_last_sub, last_pos);
    __syncthreads();
    // sum_v (q_v |y_q,v| + p_v |y_p,v|) over the normalised rows, from the statistics pass
    const float A = it.q.ay + (it.has_p ? it.p.ay : 0.f);
    const ff thr = ff_mul(R, {s_u.x, s_u.y});
    // 3. the thread whose range holds thr finds the sub-chunk
    if (wsum.hi > 0.f && ff_diff(thr, excl) >= 0.f && ff_diff(thr, incl) < 0.f) {
        ff run = excl, pre = excl;
        int found = -1;
        for (int s = s0; s < s1; ++s) {
            const float wv = subs[s];
            const ff nx = ff_add_f(run, wv);
            if (wv > 0.f) {
                found = s;
                pre = run;
                if (ff_diff(thr, nx) < 0.f) break;
            }
            run = nx;
        }
        s_sub = found;
        s_pre = make_float2(pre.hi, pre.lo);
    }
    __syncthreads();
    int sub = s_sub;
    ff pre = {s_pre.x, s_pre.y};
    bool ambiguous = false;
    if (sub < 0) {
        // thr at or beyond the last boundary (rounding) or R == 0: the last positive weight
        sub = s_last_sub;
        ambiguous = true;
        if (sub >= 0 && tid == 0) {
            ff p = {0.f, 0.f};
            for (int s = 0; s < sub; ++s) p = ff_add_f(p, subs[s]);
            s_pre = make_float2(p.hi, p.lo);
        }
        __syncthreads();
        pre = {s_pre.x, s_pre.y};
    }
    if (warp != 0) return;
    if (sub < 0) {
        // every weight is zero: degenerate; the exact tier decides
        if (lane == 0) {
            *it.out = -1;
            if (a.exact) push_exact(a.counters, a.exact, a.exact_unc, {d, it.seq}, a.stats);
            stats_add(a.stats, &a.stats->reresolved, 1);
            stats_add(a.stats, &a.stats->draws, 1);
        }
        return;
    }
    // 4. rescan the sub-chunk token by token (same arithmetic as pass 1)
    float wv[EPV];
    int ntok = 0, tok0 = 0;
    if (sub < n_vsub) {
        const int vi = sub * 32 + lane;
        tok0 = vi * EPV;
        if (vi < a.n_vec) {
            ntok = EPV;
            const uint4 q = __ldg(reinterpret_cast<const uint4 *>(it.q.row) + vi);
            const uint4 p = it.has_p ? __ldg(reinterpret_cast<const uint4 *>(it.p.row) + vi) : q;
            if (it.has_p) {
                if (it.filt) vec_weights<ES, true, true>(it, q, p, tok0, wv);
                else vec_weights<ES, true, false>(it, q, p, tok0, wv);
            } else {
                if (it.filt) vec_weights<ES, false, true>(it, q, p, tok0, wv);
                else vec_weights<ES, false, false>(it, q, p, tok0, wv);
            }
        }
    } else {
        tok0 = a.n_vec * EPV + lane;
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
    float dprev, dhit;   // thr - C(t*-1) and C(t*) - thr
    if (m != 0) {
        const int src = __ffs(m) - 1;
        const int tok = tok0 + (ntok == 1 ? 0 : hit);
        tstar = __shfl_sync(0xFFFFFFFFu, tok, src);
        const float dp = ff_diff(thr, c_prev), dh = ff_diff(c_hit, thr);
        dprev = __shfl_sync(0xFFFFFFFFu, dp, src);
        dhit = __shfl_sync(0xFFFFFFFFu, dh, src);
    } else {
        // rounding left thr past this sub-chunk: take its last positive weight, flag it
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
        // C(t*) + u R covers both boundaries' prefix and total terms
        const float E = draw_error_bound(it, R.hi, A, fmaxf(thr.hi + dhit, 0.f) + thr.hi);
        if (dprev <= E || dhit <= E) ambiguous = true;
        const bool near = dprev < 1e-6f * R.hi || dhit < 1e-6f * R.hi;
        *it.out = tstar;
        if (it.dbg_r) *it.dbg_r = (double)R.hi + (double)R.lo;
        stats_add(a.stats, &a.stats->draws, 1);
        if (near) stats_add(a.stats, &a.stats->near_boundary, 1);
        if (ambiguous && a.exact) {
            stats_add(a.stats, &a.stats->reresolved, 1);
            push_exact(a.counters, a.exact, a.exact_unc, {d, it.seq}, a.stats);
        }
    }
}

// Host side: both passes of the draws.  The number of items is known only on the device, so
// the pass-1 grid is the persistent size and pass 2 has one block per possible item.
template <int ES>
static sv_status launch_draws(const DrawArgs &da, long long max_items, const DeviceInfo &di, cudaStream_t stream) {
    const int occ = prepare_kernel((const void *)k_draw_sums<ES>, kStatsThreads, kDrawSmemBytes);
    if (occ < 1) return SV_ERR_CUDA;
    long long grid = (long long)di.sms * occ;
    const long long maxu = max_items * da.n_split;
    if (grid > maxu) grid = maxu;
    if (grid < 1) grid = 1;
    if (launch_pdl(k_draw_sums<ES>, dim3((unsigned)grid), dim3(kStatsThreads), kDrawSmemBytes, stream, da) !=
        cudaSuccess)
        return SV_ERR_CUDA;
    if (launch_pdl(k_draw_finish<ES>, dim3((unsigned)max_items), dim3(kThreads), 0, stream, da) != cudaSuccess)
        return SV_ERR_CUDA;
    return SV_OK;
}

}  // namespace sv
