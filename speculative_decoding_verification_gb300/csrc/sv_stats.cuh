// sv_stats.cuh — statistics pass: one streaming read of every needed logit row.
//
// For a sampled row (temperature T > 0, c = log2(e)/T) the pass accumulates
//   S = sum_v 2^(x_v c - r)       with an integer reference r >= max_v x_v c,
//   A = sum_v 2^(x_v c - r) |x_v c - r|    (enters the certified error bound),
// so that log2 sum_v 2^(x_v c) = r + log2 S and LSE = (r + log2 S) ln 2.  For a greedy row
// (T == 0) it finds the maximum and its lowest index.  Both track NaN / +inf.
//
// Work is handed out as (row, chunk) units from a global counter to a persistent grid.  In each
// block a producer warp streams the units' 32 KB tiles into shared memory with 1-D bulk copies
// (cp.async.bulk) and eight consumer warps read them with 128-bit shared loads.  Each consumer
// warp writes one WarpPartial per unit; partials are combined per row by the accept kernel.
#pragma once

#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

struct StatsArgs {
    RowSet set[2];
    int n_sets;
    int V;
    const float *temperature;   // per sequence; nullptr -> T = 1
    int n_split;                // chunks per row
    int chunk_vecs;             // 16-byte vectors per chunk
    long long n_rows0;          // candidate rows in set 0
    long long n_units;          // candidate rows * n_split
    WarpPartial *part;          // [candidate row][chunk][warp]
    Counters *counters;         // zeroed by the host before the pass (work counter; later kernels)
    sv_stats *stats;
    bool zero_stats = false;    // the counter reset also clears *stats (the call's first launch)
    long long wait_limit;
};

struct UnitInfo {
    const char *row;
    long long rid;
    int chunk;
    int v0, v1;           // vector range
    int tail0, n_tail;    // scalar tail elements (last chunk only)
    bool needed;
    bool greedy;
    float c_hi, c_lo;
};

template <int ES>
// t_cache: the temperatures in shared memory (n_cache of them), or nullptr.
__device__ __forceinline__ UnitInfo stats_unit(const StatsArgs &a, long long u, const float *t_cache = nullptr,
                                               int n_cache = 0) {
    UnitInfo ui;
    ui.rid = u / a.n_split;
    ui.chunk = static_cast<int>(u - ui.rid * a.n_split);
    const int s = ui.rid < a.n_rows0 ? 0 : 1;
    const long long lr = s == 0 ? ui.rid : ui.rid - a.n_rows0;
    const RowSet &rs = a.set[s];
    const long long b = lr / rs.rows_used;
    const long long j = lr - b * rs.rows_used;
    const float T = b < n_cache ? t_cache[b] : (a.temperature ? a.temperature[b] : 1.0f);
    ui.greedy = (T == 0.0f);
    ui.needed = !(rs.skip_greedy && ui.greedy);
    ui.row = rs.base + (b * rs.rows_per_seq + j) * rs.pitch_bytes;
    if (ui.greedy) {
        ui.c_hi = ui.c_lo = 0.0f;
    } else {
        log2e_over(T, ui.c_hi, ui.c_lo);
    }
    constexpr int EPV = 16 / ES;
    const int n_vec = (a.V * ES) / 16;
    ui.v0 = min(ui.chunk * a.chunk_vecs, n_vec);
    ui.v1 = min(ui.v0 + a.chunk_vecs, n_vec);
    ui.tail0 = n_vec * EPV;
    ui.n_tail = (ui.chunk == a.n_split - 1) ? (a.V - ui.tail0) : 0;
    return ui;
}

__device__ __forceinline__ int unit_tiles(const UnitInfo &ui) {
    return (ui.v1 - ui.v0 + (kStatsTileBytes / 16) - 1) / (kStatsTileBytes / 16);
}

// Per-thread accumulator.
struct StatAcc {
    int r;
    float rf, thr, s, comp, aerr;
    float m;
    int am;
    int flags;
};

__device__ __forceinline__ float fmax_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

__device__ __forceinline__ void acc_init(StatAcc &A) {
    A.r = kNoRef;
    A.rf = (float)kNoRef;
    A.thr = -INFINITY;
    A.s = 0.f;
    A.comp = 0.f;
    A.aerr = 0.f;
    A.m = -INFINITY;
    A.am = 0x7FFFFFFF;
    A.flags = 0;
}

// Raise the reference exponent so that x*c <= r for x <= vmax (exact power-of-two rescale).
__device__ __forceinline__ void acc_reference(StatAcc &A, float vmax, float c_hi) {
    if (vmax != vmax) {
        A.flags |= kFlagNaN;
        return;
    }
    if (isinf(vmax)) {
        if (vmax > 0.f) A.flags |= kFlagPosInf;
        return;
    }
    float yr = ceilf(vmax * c_hi);
    yr = fminf(fmaxf(yr, -1.0e9f), 1.0e9f);
    const int rn = (int)yr;
    if (rn > A.r) {
        const int d = rn - A.r;
        const float sc = pow2i(-d);
        const float tot = A.s + A.comp;
        A.aerr = (A.aerr + (float)min(d, 1 << 20) * tot) * sc;
        A.s *= sc;
        A.comp *= sc;
        A.r = rn;
        A.rf = (float)rn;
    }
    A.thr = fmaxf(A.rf / c_hi, vmax);
}

__device__ __forceinline__ void acc_add(StatAcc &A, float s8) {
    const float t = __fadd_rn(A.s, s8);
    const float e = (A.s >= s8) ? __fadd_rn(__fsub_rn(A.s, t), s8) : __fadd_rn(__fsub_rn(s8, t), A.s);
    A.comp = __fadd_rn(A.comp, e);
    A.s = t;
}

// Largest finite logit magnitude kept as is; smaller logits (and -inf) have 2^(x c - r) = 0
// for every allowed c, so clamping them there changes no weight and keeps x c - r finite.
constexpr uint32_t kBf16Floor2 = 0xF149F149u;   // bf16 pair (-9.95e29, -9.95e29)
constexpr float kF32Floor = -9.95e29f;

// One element outside the vector stream (row tails).
__device__ __forceinline__ void acc_scalar(StatAcc &A, float x, int idx, bool greedy, float c_hi, float c_lo) {
    if (greedy) {
        if (!(x <= A.m)) {
            if (x != x) {
                A.flags |= kFlagNaN;
            } else {
                A.m = x;
                A.am = idx;
                if (isinf(x)) A.flags |= kFlagPosInf;
            }
        }
        return;
    }
    if (!(x <= A.thr)) acc_reference(A, x, c_hi);
    (void)c_lo;   // applied to the row sum in combine_row
    const float y = fmaf(fmaxf(x, kF32Floor), c_hi, -A.rf);
    const float e = ex2_fast(y);
    A.aerr = fmaf(e, -y, A.aerr);
    acc_add(A, e);
}

// The error weight A = sum 2^y (-y) of a thread's share of a tile with every logit clamped at
// the floor first.  The fast path leaves the clamp out; a -inf logit (a masked token) or one
// whose x c_hi overflows gives y = -inf there, and 2^y y = 0 * inf = NaN, so the tile's weight
// is taken again here.  The row sum needs no second pass: those elements weigh 0 either way.
template <int ES>
__device__ __noinline__ float acc_tile_weight_clamped(const unsigned char *buf, int nv, float c_hi, float rf) {
    constexpr int EPV = 16 / ES;
    constexpr int NV = kTileBytes / 16 / kThreads;
    float a = 0.f;
    for (int i = 0; i < NV; ++i) {
        const int vi = threadIdx.x + i * kThreads;
        if (vi >= nv) break;
        float x[EPV];
        unpack<ES>(lds128(buf + vi * 16), x);
        for (int k = 0; k < EPV; ++k) {
            const float y = fmaf(fmax_nan(x[k], kF32Floor), c_hi, -rf);
            a = fmaf(ex2_fast(y), -y, a);
        }
    }
    return a;
}

// A thread's share of one 16 KB half of a stage: its NV vectors (vi = tid + i * kThreads) are
// loaded together, checked against the reference with one combined maximum, and their
// 8 * NV (bf16) exponentials are independent, so the SFU work overlaps.  Vectors past the
// end of a partial tile hold no element.  Sampled rows accumulate S = sum 2^y and
// A = sum 2^y (-y) with y = x c_hi - r <= 0 rounded once (c = c_hi + c_lo); combine_row
// applies the x c_lo part to the row sum to first order.  One compensated addition per tile.
template <int ES>
__device__ __forceinline__ void acc_half(StatAcc &A, const unsigned char *buf, int nv, int fv, bool greedy, float c_hi) {
    constexpr int EPV = 16 / ES;
    constexpr int NV = kTileBytes / 16 / kThreads;
    // vectors past the end of a partial tile: -inf for greedy rows (they can never hold the
    // argmax), the floor for sampled rows (weight 0, and no -inf to send the tile's error weight
    // down the clamped path)
    const uint32_t ninf = greedy ? (ES == 2 ? 0xFF80FF80u : 0xFF800000u)
                                 : (ES == 2 ? kBf16Floor2 : __float_as_uint(kF32Floor));
    const int tid = threadIdx.x;
    uint4 w[NV];
    if (nv == kTileBytes / 16) {
#pragma unroll
        for (int i = 0; i < NV; ++i) w[i] = lds128(buf + (tid + i * kThreads) * 16);
    } else {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int vi = tid + i * kThreads;
            w[i] = vi < nv ? lds128(buf + vi * 16) : make_uint4(ninf, ninf, ninf, ninf);
        }
    }
    float vmax;
    if constexpr (ES == 2) {
        uint32_t pm = bmax2(bmax2(w[0].x, w[0].y), bmax2(w[0].z, w[0].w));
#pragma unroll
        for (int i = 1; i < NV; ++i) pm = bmax2(pm, bmax2(bmax2(w[i].x, w[i].y), bmax2(w[i].z, w[i].w)));
        vmax = fmax_nan(bf16_lo(pm), bf16_hi(pm));
    } else {
        vmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            vmax = fmax_nan(vmax, fmax_nan(fmax_nan(__uint_as_float(w[i].x), __uint_as_float(w[i].y)),
                                           fmax_nan(__uint_as_float(w[i].z), __uint_as_float(w[i].w))));
    }
    if (greedy) {
        if (!(vmax <= A.m)) {
            if (vmax != vmax) {
                A.flags |= kFlagNaN;
                return;
            }
            // the first index (in this thread's increasing order) holding the new maximum
            int idx = -1;
            for (int i = NV - 1; i >= 0; --i) {
                float x[EPV];
                unpack<ES>(w[i], x);
                for (int k = EPV - 1; k >= 0; --k)
                    if (x[k] == vmax) idx = (fv + tid + i * kThreads) * EPV + k;
            }
            A.m = vmax;
            A.am = idx;
            if (isinf(vmax)) A.flags |= kFlagPosInf;
        }
        return;
    }
    if (!(vmax <= A.thr)) acc_reference(A, vmax, c_hi);
    // Both elements of a pair go through one f32x2 instruction, each rounded as its scalar form:
    // y = x c_hi - r (one rounding), e = 2^y, and the error weight accumulates e y (= -A).  The
    // row sum's tree keeps its depth: two pair additions inside a vector (bf16: 4 pairs; f32: one
    // addition of 2 pairs), two across the tile's vectors, and the final lo + hi, i.e. 3 + 2
    // rounding levels for bf16 (2 + 2 for f32) as the error bound counts them.
    const f32x2 c2 = f2_pack(c_hi, c_hi), nr2 = f2_pack(-A.rf, -A.rf);
    f32x2 sv[NV];
    f32x2 ay2[2] = {0ull, 0ull};
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        constexpr int PPV = 8 / ES;   // pairs per 16-byte vector
        f32x2 e2[PPV];
#pragma unroll
        for (int k = 0; k < PPV; ++k) {
            const uint32_t w0 = k == 0 ? w[i].x : k == 1 ? w[i].y : k == 2 ? w[i].z : w[i].w;
            f32x2 x2;
            if constexpr (ES == 2) {
                x2 = f2_from_bf16x2(w0);
            } else {
                x2 = f2_from_u32x2(k == 0 ? w[i].x : w[i].z, k == 0 ? w[i].y : w[i].w);
            }
            const f32x2 y2 = f2_fma(x2, c2, nr2);
            e2[k] = f2_ex2(y2);
            ay2[i & 1] = f2_fma(e2[k], y2, ay2[i & 1]);
        }
        if constexpr (PPV == 4) {
            sv[i] = f2_add(f2_add(e2[0], e2[1]), f2_add(e2[2], e2[3]));
        } else {
            sv[i] = f2_add(e2[0], e2[1]);
        }
    }
    f32x2 s2;
    if constexpr (NV == 4) {
        s2 = f2_add(f2_add(sv[0], sv[1]), f2_add(sv[2], sv[3]));
    } else {
        s2 = sv[0];
#pragma unroll
        for (int i = 1; i < NV; ++i) s2 = f2_add(s2, sv[i]);
    }
    const float st = f2_sum(s2);
    float at = -f2_sum(f2_add(ay2[0], ay2[1]));
    if (at != at) at = acc_tile_weight_clamped<ES>(buf, nv, c_hi, A.rf);
    acc_add(A, st);
    A.aerr += at;
}

// A thread's share of one 32 KB stage: its two 16 KB halves in order (each with its own maximum
// check, tree sums and compensated addition), so a thread's elements are met in increasing id
// order and the per-stage costs (barrier wait, stage description, release) are paid once.
template <int ES>
__device__ __forceinline__ void acc_tile(StatAcc &A, const unsigned char *buf, int nv, int fv, bool greedy, float c_hi) {
    constexpr int HV = kTileBytes / 16;   // vectors per half
    acc_half<ES>(A, buf, min(nv, HV), fv, greedy, c_hi);
    if (nv > HV) acc_half<ES>(A, buf + kTileBytes, nv - HV, fv + HV, greedy, c_hi);
}

// Warp-combine and store this unit's partial (float32 / float-float arithmetic only).
__device__ __forceinline__ void acc_store(const StatAcc &A0, bool greedy, WarpPartial *dst) {
    StatAcc A = A0;
    const int lane = threadIdx.x & 31;
    WarpPartial p;
    p.flags = warp_or_i(A.flags);
    p.pad = 0;
    if (greedy) {
        warp_argmax(A.m, A.am);
        p.s_hi = p.s_lo = p.a = 0.0f;
        p.r = kNoRef;
        p.maxv = A.m;
        p.argmax = A.am;
    } else {
        const int rw = warp_max_i(A.r);
        const int d = rw - A.r;   // >= 0; scaling by 2^-d is exact
        const float sc = pow2i(-d);
        ff v = fast_two_sum(A.s, A.comp);
        v.hi *= sc;
        v.lo *= sc;
        const float a = (A.aerr + (float)min(d, 1 << 20) * (A.s + A.comp)) * sc;
        v = warp_sum_ff(v);
        p.s_hi = v.hi;
        p.s_lo = v.lo;
        p.a = warp_sum_f(a);
        p.r = rw;
        p.maxv = -INFINITY;
        p.argmax = 0x7FFFFFFF;
    }
    if (lane == 0) *dst = p;
}

// One pipeline stage's description, written by the producer before the stage's copy is issued.
struct TileMeta {
    const char *row;
    long long rid;
    float c_hi, c_lo;
    int chunk;
    int fv, nv;           // first vector of the tile within the row, vectors in the tile
    int tail0, n_tail;    // scalar tail of the row (last tile of a row's last chunk)
    int flags;            // kTileFirst | kTileLast | kTileGreedy | kTileEnd
    int aux;              // lazy verification: (warps expected for the position << 1) | completing
};
constexpr int kTileFirst = 1, kTileLast = 2, kTileGreedy = 4, kTileEnd = 8;

constexpr int kStatsCtlBytes = 1024;   // full[], empty[], abort flag, TileMeta[]
static_assert(2 * kStatsStages * 8 + 16 + kStatsStages * (int)sizeof(TileMeta) <= kStatsCtlBytes, "control block");
constexpr size_t kStatsSmemBytes = (size_t)kStatsCtlBytes + (size_t)kStatsStages * kStatsTileBytes;

// Warp-specialised pipeline.  The producer (lane 0 of the last warp) takes (row, chunk) units
// from a global counter, skips units that are not needed, and streams each unit's tiles into a
// kStatsStages-deep ring of 32 KB shared-memory tiles with 1-D bulk copies; per stage it first
// waits until the eight consumer warps released the stage ("empty"), writes the TileMeta, then
// issues the copy that completes the stage's "full" barrier.  Consumer warps wait on "full",
// accumulate their share of the tile, and release it.  Waits sleep (suspend hint) instead of
// spinning, give up after wait_limit cycles or once another warp has aborted, and on abort the
// producer lets its copies in flight land before the block exits.
template <int ES>
__global__ void __launch_bounds__(kStatsThreads, 2) k_stats(const StatsArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kStatsStages;
    int *abort_flag = reinterpret_cast<int *>(smem + 2 * kStatsStages * 8);
    TileMeta *meta = reinterpret_cast<TileMeta *>(smem + 2 * kStatsStages * 8 + 16);
    unsigned char *tiles = smem + kStatsCtlBytes;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    pdl_wait();      // the counters are zeroed by the kernel before this one
    pdl_trigger();   // the next kernel may be scheduled now; it waits for this one's results

    if (tid == 0) {
        for (int s = 0; s < kStatsStages; ++s) {
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
            long long in_flight[kStatsStages];   // tile number whose copy a stage waits for, or -1
            for (int s = 0; s < kStatsStages; ++s) in_flight[s] = -1;
            long long it = 0;           // tiles issued
            int st = 0;                 // it % kStatsStages
            uint32_t epar = 0;          // parity of the "empty" phase to wait for at stage st
            bool ok = true;
            int u = atomicAdd(&a.counters->next_unit, 1);
            while (ok) {
                // the next needed unit (or the end)
                UnitInfo ui;
                bool have = false;
                while (u < a.n_units) {
                    ui = stats_unit<ES>(a, u);
                    u = atomicAdd(&a.counters->next_unit, 1);   // fetch ahead; used for the next unit
                    if (ui.needed) {
                        have = true;
                        break;
                    }
                }
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
                    m.aux = 0;
                    meta[st] = m;
                    if (nv > 0) {
                        mbar_arrive_expect_tx(&full[st], (uint32_t)nv * 16u);
                        bulk_load_stream(tiles + st * kStatsTileBytes, ui.row + (size_t)fv * 16, (uint32_t)nv * 16u,
                                         &full[st], policy);
                        in_flight[st] = it;
                    } else {
                        mbar_arrive(&full[st]);   // a tail-only unit: nothing to copy
                    }
                    if (++st == kStatsStages) {
                        st = 0;
                        if (it >= 2 * kStatsStages - 1) epar ^= 1u;   // round r >= 2 waits phase r - 1
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
            // the row's last (< 16 B) elements come after every vector, keeping greedy ties on the lowest id
            if (tid < m.n_tail) {
                const float x = load_elem<ES>(m.row, m.tail0 + tid);
                acc_scalar(A, x, m.tail0 + tid, greedy, m.c_hi, m.c_lo);
            }
            acc_store(A, greedy, a.part + ((size_t)m.rid * a.n_split + m.chunk) * kWarps + warp);
        }
        if (++st == kStatsStages) {
            st = 0;
            par ^= 1u;
        }
    }
}

// Host side: clear the call's counters, then run the statistics pass on a persistent grid.
// Zeroes a call's counters (and, when given, its sv_stats block) once the stream's previous
// kernel has finished with them.
static __global__ void k_zero_counters(Counters *c, sv_stats *st) {
    pdl_wait();
    pdl_trigger();
    int *w = reinterpret_cast<int *>(c);
    for (int i = threadIdx.x; i < (int)(sizeof(Counters) / sizeof(int)); i += blockDim.x) w[i] = 0;
    if (st != nullptr) {
        int *v = reinterpret_cast<int *>(st);
        for (int i = threadIdx.x; i < (int)(sizeof(sv_stats) / sizeof(int)); i += blockDim.x) v[i] = 0;
    }
}

template <int ES>
static sv_status launch_stats(const StatsArgs &sa, const DeviceInfo &di, cudaStream_t stream) {
    // the counters are zeroed by a kernel rather than a memset, so that the launches of the
    // whole call (and of the next call) form one chain of programmatic dependent launches
    if (launch_pdl(k_zero_counters, dim3(1), dim3(64), 0, stream, sa.counters, sa.zero_stats ? sa.stats : nullptr) !=
        cudaSuccess)
        return SV_ERR_CUDA;
    const int occ = prepare_kernel((const void *)k_stats<ES>, kStatsThreads, kStatsSmemBytes);
    if (occ < 1) return SV_ERR_CUDA;
    long long grid = (long long)di.sms * occ;
    if (grid > sa.n_units) grid = sa.n_units;
    if (grid < 1) grid = 1;
    profile_begin(stream);
    if (launch_pdl(k_stats<ES>, dim3((unsigned)grid), dim3(kStatsThreads), kStatsSmemBytes, stream, sa) != cudaSuccess)
        return SV_ERR_CUDA;
    profile_end(stream);
    return SV_OK;
}

// Combine a row's warp partials (one warp).  Float-float accumulation; the few float64
// operations happen once per row.
__device__ __forceinline__ RowStat combine_row(const WarpPartial *P, int np, bool greedy, float T) {
    const int lane = threadIdx.x & 31;
    // one pass over the partials: each lane keeps its own reference and raises it (an exact
    // power-of-two rescale; A gains d * S as every -y grows by d), then the lanes agree on one
    ff s = {0.f, 0.f};
    float a = 0.f;
    int rl = kNoRef;
    float m = -INFINITY;
    int am = 0x7FFFFFFF, fl = 0;
    for (int p = lane; p < np; p += 32) {
        const WarpPartial w = P[p];
        fl |= w.flags;
        if (greedy) {
            if (w.maxv > m || (w.maxv == m && w.argmax < am)) {
                m = w.maxv;
                am = w.argmax;
            }
        } else {
            if (w.r > rl) {
                const int d = w.r - rl;
                const float sc = pow2i(-d);
                a = (a + (float)min(d, 1 << 20) * (s.hi + s.lo)) * sc;
                s.hi *= sc;
                s.lo *= sc;
                rl = w.r;
            }
            const int d = rl - w.r;
            const float sc = pow2i(-d);
            s = ff_add(s, {w.s_hi * sc, w.s_lo * sc});
            a += (w.a + (float)min(d, 1 << 20) * (w.s_hi + w.s_lo)) * sc;
        }
    }
    const int rmax = warp_max_i(rl);
    if (!greedy) {
        const int d = rmax - rl;
        const float sc = pow2i(-d);
        a = (a + (float)min(d, 1 << 20) * (s.hi + s.lo)) * sc;
        s.hi *= sc;
        s.lo *= sc;
    }
    s = warp_sum_ff(s);
    a = warp_sum_f(a);
    RowStat r;
    r.flags = warp_or_i(fl);
    warp_argmax(m, am);
    r.maxv = m;
    r.argmax = am;
    r.r = rmax;
    r.ay = 0.f;
    r.s_hi = r.s_lo = r.err = 0.f;
    if (!greedy && lane == 0) {
        float c_hi, c_lo;
        log2e_over(T, c_hi, c_lo);
        // The pass summed e = 2^(x c_hi - r); the true terms are e 2^(x c_lo) = e (1 + k x c_hi + q)
        // with k = ln2 c_lo / c_hi and |q| <= (ln2 |x c_lo|)^2 (|x c_lo| <= 2^-22 here).  Since
        // x c_hi = y + r and sum e (-y) = a:  S = S_pass + k (r S_pass - a).
        const ff S0 = fast_two_sum(s.hi, s.lo);
        const float k = (float)kLn2 * __fdiv_rn(c_lo, c_hi);
        const float corr = k * fmaf((float)rmax, S0.hi, -a);
        const ff S = ff_add(S0, {corr, 0.f});
        r.s_hi = S.hi;
        r.s_lo = S.lo;
        // A counts 2^y (-y); the few y > 0 left by rounding (x c_hi may exceed r by a rounding of
        // the threshold: y <= (|r| + 1) 2^-22, each with 2^y < 2, at most S of them) can lower it
        // by 2 S (|r| + 1) 2^-22 at most.  ay bounds sum q |y| for y = x c_hi - r and, with
        // |x c_lo| <= (|r| + 128) 2^-23 added, for y = x c - r as the draw pass computes it.
        const float rr = (float)(abs(rmax) + 128);
        const float ay = (S0.hi > 0.f ? __fdiv_rn(a, S0.hi) : 0.f) + rr * 0x1p-20f;
        r.ay = ay;
        // exponential + exponent rounded once (ln2 u per unit |y|) + second-order c_lo term +
        // summation (3 + 2 tree levels per tile, compensated running sum, float-float merges) +
        // the correction's own rounding; evaluated in float32 and rounded up by 2^-20
        const float q2 = (float)kLn2 * rr * 0x1p-23f;
        r.err = (float)(kEx2RelErr + 9.0 * kU32 + 1e-12) + (float)(1.02 * kLn2 * kU32) * ay + q2 * q2;
        r.err *= 1.0f + 0x1p-20f;
    }
    return r;   // s_hi, s_lo, err valid in lane 0 (sampled rows)
}

// Double-precision views of a row's statistics, for kernels off the per-sequence hot path.
__device__ __forceinline__ double rs_S(const RowStat &r) { return (double)r.s_hi + (double)r.s_lo; }
__device__ __forceinline__ double rs_g(const RowStat &r) { return (double)r.r + log2(rs_S(r)); }
__device__ __forceinline__ double rs_err(const RowStat &r) { return (double)r.err; }
__device__ __forceinline__ bool rs_sampled_ok(const RowStat &r) { return r.s_hi > 0.f && r.s_hi < INFINITY; }

}  // namespace sv
