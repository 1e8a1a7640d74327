// sv_select.cuh — ranking passes over logit rows, one block per row.
//
//  * top-N selection (cache keys, top-kappa roots, the Saguaro top-F set): a most-significant-
//    digit radix select on order-preserving 32-bit keys (two 8-bit passes for bf16, four for
//    float32) finds the key K* of the N-th token; ties at K* are taken in id order by an ordered
//    block scan, so ranking ties go to the lowest id.
//  * nucleus (top-p) cut [SpS notes §3 and §6: the filter acts on q and on p before the ratio]:
//    the same radix select weighted by probability mass 2^(x c - r) finds the shortest prefix in
//    (probability desc, id asc) order whose mass reaches top_p.  The float32 masses carry a
//    proven error bound; a cut the bound cannot settle is recomputed in float-float in the same
//    block.
#pragma once

#include "sv_device.cuh"
#include "sv_exp2_table.h"
#include "sv_host.h"
#include "sv_stats.cuh"

namespace sv {

constexpr int kMaxTopN = 1024;   // longest sorted top-N list (cache keys, roots)

// ---- element iteration ------------------------------------------------------------------
template <int ES, class Fn>
__device__ __forceinline__ void for_each_elem(const char *row, int V, Fn fn) {
    constexpr int EPV = 16 / ES;
    const int n_vec = (V * ES) / 16;
    for (int vi = threadIdx.x; vi < n_vec; vi += blockDim.x) {
        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(row) + vi);
        float x[EPV];
        if constexpr (ES == 2) {
            x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
            x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
        } else {
            x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
            x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
        }
#pragma unroll
        for (int k = 0; k < EPV; ++k) fn(x[k], vi * EPV + k);
    }
    for (int v = n_vec * EPV + threadIdx.x; v < V; v += blockDim.x) fn(load_elem<ES>(row, v), v);
}

// Block-wide exclusive scan of one int per thread (blockDim == kThreads).
__device__ __forceinline__ int block_excl_scan(int v, int &total, int *s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    int off = 0, tot = 0;
    for (int w = 0; w < kWarps; ++w) {
        const int t = s_warp[w];
        if (w < warp) off += t;
        tot += t;
    }
    __syncthreads();
    total = tot;
    return off + inc - v;
}

// Digit of the current radix pass: the largest bin d with above + sum_{b >= d} h[b] >= need.
// Returns d and the count (or mass) of bins strictly above d; d = -1 if no bin reaches need.
template <class T>
__device__ __forceinline__ void pick_digit(const T *h, T need, int &digit, T &above) {
    const int lane = threadIdx.x & 31;
    T c = 0;
    for (int i = 0; i < 8; ++i) c += h[8 * lane + i];
    T S = c;   // inclusive suffix over lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const T t = __shfl_down_sync(0xFFFFFFFFu, S, o);
        if (lane + o < 32) S += t;
    }
    const unsigned m = __ballot_sync(0xFFFFFFFFu, S >= need);
    digit = -1;
    above = 0;
    if (m == 0) return;
    const int L = 31 - __clz(m);
    int d = -1;
    T acc = 0;
    if (lane == L) {
        acc = S - c;
        for (int b = 8 * L + 7; b >= 8 * L; --b) {
            if (acc + h[b] >= need) {
                d = b;
                break;
            }
            acc += h[b];
        }
    }
    digit = __shfl_sync(0xFFFFFFFFu, d, L);
    above = __shfl_sync(0xFFFFFFFFu, acc, L);
}

// After the 8-bit passes over the top 16 bits, a bf16 key is complete except for its low 16
// bits, which are 0 for positive values and all ones for negative ones (the key of a negative
// float is its complement).
template <int ES>
__device__ __forceinline__ uint32_t complete_key(uint32_t prefix) {
    if (ES == 2 && !(prefix & 0x80000000u)) prefix |= 0xFFFFu;
    return prefix;
}

__device__ __forceinline__ float key_value(uint32_t k) {
    return (k & 0x80000000u) ? __uint_as_float(k & 0x7FFFFFFFu) : __uint_as_float(~k);
}

// Count-weighted radix select: the key K* of the N-th largest element (1 <= N <= V) and the
// number of elements strictly above it.
template <int ES>
__device__ uint32_t radix_select_count(const char *row, int V, int N, int &n_above, unsigned *hist, int *s_dig) {
    uint32_t prefix = 0, mask = 0;
    int need = N;
    constexpr int passes = ES == 2 ? 2 : 4;
    for (int p = 0; p < passes; ++p) {
        const int shift = 24 - 8 * p;
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for_each_elem<ES>(row, V, [&](float x, int) {
            const uint32_t k = f32_key(x);
            if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
        });
        __syncthreads();
        if (threadIdx.x < 32) {
            int d;
            unsigned above;
            pick_digit<unsigned>(hist, (unsigned)need, d, above);
            if (threadIdx.x == 0) {
                s_dig[0] = d < 0 ? 0 : d;
                s_dig[1] = (int)above;
            }
        }
        __syncthreads();
        need -= s_dig[1];
        prefix |= (uint32_t)s_dig[0] << shift;
        mask |= 255u << shift;
        __syncthreads();
    }
    n_above = N - need;
    return complete_key<ES>(prefix);
}

// Ids of the first `want` elements with key == kstar, in increasing id order.  Writes them to
// out (if not null) at out[0..want) and returns the id of the last one (-1 if fewer exist).
template <int ES>
__device__ int ordered_ties(const char *row, int V, uint32_t kstar, int want, int *out, int *s_warp, int *s_last) {
    constexpr int EPV = 16 / ES;
    const int n_vec = (V * ES) / 16;
    const int n_pseudo = n_vec + (V > n_vec * EPV ? 1 : 0);   // the scalar tail as one pseudo-vector
    if (threadIdx.x == 0) *s_last = -1;
    __syncthreads();
    int base = 0;
    for (int vb = 0; vb < n_pseudo && base < want; vb += blockDim.x) {
        const int vi = vb + threadIdx.x;
        float x[EPV];
        int n = 0, e0 = 0;
        if (vi < n_vec) {
            const uint4 w = __ldg(reinterpret_cast<const uint4 *>(row) + vi);
            if constexpr (ES == 2) {
                x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
                x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
            } else {
                x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
                x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
            }
            n = EPV;
            e0 = vi * EPV;
        } else if (vi < n_pseudo) {
            e0 = n_vec * EPV;
            n = V - e0;
            for (int k = 0; k < n; ++k) x[k] = load_elem<ES>(row, e0 + k);
        }
        int cnt = 0;
        for (int k = 0; k < n; ++k) cnt += (f32_key(x[k]) == kstar) ? 1 : 0;
        int total;
        const int excl = block_excl_scan(cnt, total, s_warp);
        if (cnt > 0 && base + excl < want) {
            int r = base + excl;
            for (int k = 0; k < n && r < want; ++k) {
                if (f32_key(x[k]) == kstar) {
                    if (out) out[r] = e0 + k;
                    if (r == want - 1) *s_last = e0 + k;
                    ++r;
                }
            }
        }
        base += total;
    }
    __syncthreads();
    const int last = *s_last;
    __syncthreads();
    return last;
}

// ------------------------------------------------------------------------------------------
// Top-N lists: sorted (logit desc, id asc) ids of each row.
// ------------------------------------------------------------------------------------------
struct TopNArgs {
    const char *base;
    int64_t pitch_bytes;
    int rows_per_seq;
    int rows_used;          // rows j < rows_used of every sequence
    long long n_rows;       // B * rows_used
    int V;
    // per-row N: n_of_j[j] (cache keys) or n_all
    int n_all;
    int n_of_j[SV_MAX_K + 2];
    int32_t *list;          // [row][list_stride] sorted ids (output)
    float *list_x;          // [row][list_stride] their logits (output, may be null)
    int list_stride;
};

template <int ES>
__global__ void __launch_bounds__(kThreads) k_topn(const TopNArgs a) {
    __shared__ unsigned hist[256];
    __shared__ int s_dig[2], s_warp[kWarps], s_last, s_cnt;
    __shared__ uint32_t s_key[kMaxTopN];
    __shared__ int s_id[kMaxTopN];
    const long long r = blockIdx.x;
    if (r >= a.n_rows) return;
    const long long b = r / a.rows_used, j = r - b * a.rows_used;
    const char *row = a.base + (b * a.rows_per_seq + j) * a.pitch_bytes;
    int N = a.n_all > 0 ? a.n_all : a.n_of_j[j];
    if (N > a.V) N = a.V;
    if (N <= 0) return;
    int n_above;
    const uint32_t kstar = radix_select_count<ES>(row, a.V, N, n_above, hist, s_dig);
    if (threadIdx.x == 0) s_cnt = 0;
    __syncthreads();
    for_each_elem<ES>(row, a.V, [&](float x, int v) {
        const uint32_t k = f32_key(x);
        if (k > kstar) {
            const int slot = atomicAdd(&s_cnt, 1);
            if (slot < kMaxTopN) {
                s_key[slot] = k;
                s_id[slot] = v;
            }
        }
    });
    __syncthreads();
    const int na = min(s_cnt, kMaxTopN);
    // rank sort of the strictly-greater entries
    int32_t *out = a.list + (size_t)r * a.list_stride;
    for (int i = threadIdx.x; i < na; i += blockDim.x) {
        const uint32_t ki = s_key[i];
        const int ii = s_id[i];
        int rank = 0;
        for (int q = 0; q < na; ++q) {
            const uint32_t kq = s_key[q];
            rank += (kq > ki || (kq == ki && s_id[q] < ii)) ? 1 : 0;
        }
        out[rank] = ii;
    }
    // the ties at K*, lowest ids first
    ordered_ties<ES>(row, a.V, kstar, N - na, out + na, s_warp, &s_last);
    __syncthreads();
    if (a.list_x) {
        __threadfence_block();
        for (int i = threadIdx.x; i < N; i += blockDim.x) a.list_x[(size_t)r * a.list_stride + i] = load_elem<ES>(row, out[i]);
    }
}

// ------------------------------------------------------------------------------------------
// Nucleus cut of each sampled row.
// ------------------------------------------------------------------------------------------
struct NucleusArgs {
    RowSet set[2];
    long long n_rows0, n_rows;
    int V;
    const float *temperature;
    const float *top_p;
    const WarpPartial *part;
    int n_split;
    NucleusCut *nuc;
    sv_stats *stats;
};

// Float-float mass of one element (exact tier arithmetic).
__device__ __forceinline__ double exact_mass(float x, ff c, float rf, const float2 *tab) {
    if (x == -INFINITY) return 0.0;
    return ff_to_double(ff_exp2_xc(x, c, (int)rf, tab));
}

// Mass-weighted radix select: the key K* at which the running mass from the top, in
// (value desc) order, first reaches `target`; the mass strictly above K*, and the count of
// elements at K*.  mass(x) gives each element's weight; the histogram bins accumulate in
// float64.  When `total` is non-null the first pass also sums every element's mass into it
// (and `target_frac` then scales that total into the target).
template <int ES, class Mass>
__device__ uint32_t radix_select_mass(const char *row, int V, double target_in, double target_frac, Mass mass,
                                      double *hm, unsigned *hc, int *s_dig, double *s_dm, double *s_red,
                                      double &above_out, int &cnt_out, double *total, double *aux_total) {
    uint32_t prefix = 0, mask = 0;
    double above_m = 0.0, target = target_in;
    int cnt_star = 0;
    constexpr int passes = ES == 2 ? 2 : 4;
    for (int p = 0; p < passes; ++p) {
        const int shift = 24 - 8 * p;
        for (int i = threadIdx.x; i < 256; i += blockDim.x) {
            hm[i] = 0.0;
            hc[i] = 0;
        }
        __syncthreads();
        double tsum = 0.0, asum = 0.0;
        for_each_elem<ES>(row, V, [&](float x, int) {
            const uint32_t k = f32_key(x);
            if ((k & mask) == prefix) {
                const double2 m = mass(x);   // (mass, auxiliary error weight)
                const unsigned bin = (k >> shift) & 255u;
                atomicAdd(&hm[bin], m.x);
                atomicAdd(&hc[bin], 1u);
                if (p == 0) {
                    tsum += m.x;
                    asum += m.y;
                }
            }
        });
        if (p == 0 && total) {
            tsum = warp_sum_d(tsum);
            asum = warp_sum_d(asum);
            if ((threadIdx.x & 31) == 0) {
                s_red[threadIdx.x >> 5] = tsum;
                hm[256 + (threadIdx.x >> 5)] = asum;
            }
        }
        __syncthreads();
        if (p == 0 && total) {
            double t = 0.0, at = 0.0;
            for (int w = 0; w < kWarps; ++w) {
                t += s_red[w];
                at += hm[256 + w];
            }
            *total = t;
            if (aux_total) *aux_total = at;
            target = target_frac * t;
        }
        if (threadIdx.x < 32) {
            int d;
            double above;
            pick_digit<double>(hm, target - above_m, d, above);
            if (d < 0) {   // rounding: the rest of the group falls short; keep all of it
                int lo = 0;
                for (int q = 0; q < 256; ++q)
                    if (hc[q]) {
                        lo = q;
                        break;
                    }
                double ab = 0.0;
                for (int q = 255; q > lo; --q) ab += hm[q];
                d = lo;
                above = ab;
            }
            if (threadIdx.x == 0) {
                s_dig[0] = d;
                s_dm[0] = above;
                s_dig[1] = (int)hc[d];
            }
        }
        __syncthreads();
        above_m += s_dm[0];
        prefix |= (uint32_t)s_dig[0] << shift;
        mask |= 255u << shift;
        cnt_star = s_dig[1];
        __syncthreads();
    }
    above_out = above_m;
    cnt_out = cnt_star;
    return complete_key<ES>(prefix);
}

template <int ES>
__global__ void __launch_bounds__(kThreads) k_nucleus(const NucleusArgs a) {
    __shared__ double hm[256 + kWarps];
    __shared__ unsigned hc[256];
    __shared__ int s_dig[2], s_warp[kWarps], s_last;
    __shared__ double s_dm[2];
    __shared__ double s_red[kWarps];
    __shared__ float2 tab[256];
    __shared__ RowStat s_rs;
    const long long rid = blockIdx.x;
    if (rid >= a.n_rows) return;
    const int s = rid < a.n_rows0 ? 0 : 1;
    const long long lr = s == 0 ? rid : rid - a.n_rows0;
    const RowSet &rs = a.set[s];
    const long long b = lr / rs.rows_used, j = lr - b * rs.rows_used;
    const float T = a.temperature[b];
    const float tp = a.top_p[b];
    NucleusCut none;
    none.cut_x = -INFINITY;
    none.cut_id = 0x7FFFFFFF;
    none.mass = 1.0;
    none.log2_mass = 0.0;
    none.ambiguous = 0;
    none.mass_f = 1.0f;
    if (!(tp < 1.0f) || !(T >= 1e-3f && T <= 1e3f)) {   // off, greedy or invalid temperature
        if (threadIdx.x == 0) a.nuc[rid] = none;
        return;
    }
    const char *row = rs.base + (b * rs.rows_per_seq + j) * rs.pitch_bytes;
    if (threadIdx.x < 32) {
        const RowStat st = combine_row(a.part + (size_t)rid * a.n_split * kWarps, a.n_split * kWarps, false, T);
        if (threadIdx.x == 0) s_rs = st;
    }
    __syncthreads();
    const RowStat st = s_rs;
    if (!rs_sampled_ok(st) || st.flags) {   // reported by the accept / sampling kernels
        if (threadIdx.x == 0) a.nuc[rid] = none;
        return;
    }
    float c_hi, c_lo;
    log2e_over(T, c_hi, c_lo);
    const float rf = (float)st.r;

    // ---- float32 tier: masses 2^(x c - r) as in the statistics pass ----
    auto fast_mass = [&](float x) {   // (mass, mass * |y|): the second feeds the error bound
        const float y = fmaf(x, c_lo, fmaf(x, c_hi, -rf));
        const float e = ex2_fast(y);
        return make_double2((double)e, (double)(e * fabsf(y)));
    };
    double above_m, S_fast, A_row;
    int cnt_star;
    const uint32_t kstar = radix_select_mass<ES>(row, a.V, 0.0, (double)tp, fast_mass, hm, hc, s_dig, s_dm, s_red,
                                                 above_m, cnt_star, &S_fast, &A_row);
    const double target = (double)tp * S_fast;
    const float xstar = key_value(kstar);
    const double estar = (double)ex2_fast(fmaf(xstar, c_lo, fmaf(xstar, c_hi, -rf)));
    int jt = (int)ceil((target - above_m) / estar);
    jt = max(1, min(jt, cnt_star));
    // certification: cum and target come from the same per-element masses; the kept set is an
    // upper set, so its error per unit mass is at most the row's (weighted mean of |y|).
    const double cum_hi = above_m + jt * estar, cum_lo = above_m + (jt - 1) * estar;
    const double rel = kEx2RelErr + 1.02 * kYRound * (A_row / S_fast) + 4.0 * kU32 + 1e-12;
    const double E = rel * (cum_hi + (double)tp * S_fast) + 1e-15 * S_fast;
    const bool ambiguous = (target - cum_lo) <= E || (cum_hi - target) <= E;
    NucleusCut out;
    out.ambiguous = ambiguous ? 1 : 0;
    out.mass_f = 1.0f;
    if (!ambiguous) {
        out.cut_x = xstar;
        out.cut_id = ordered_ties<ES>(row, a.V, kstar, jt, nullptr, s_warp, &s_last);
        out.mass = cum_hi / S_fast;
    } else {
        // ---- float-float tier: the same select on exact masses ----
        {
            tab[threadIdx.x] = kExp2Table[threadIdx.x];
        }
        __syncthreads();
        const ff cff = {c_hi, c_lo};
        auto exact = [&](float x) { return make_double2(exact_mass(x, cff, rf, tab), 0.0); };
        double A_x, S_x;
        int cnt_x;
        const uint32_t kx = radix_select_mass<ES>(row, a.V, 0.0, (double)tp, exact, hm, hc, s_dig, s_dm, s_red, A_x,
                                                  cnt_x, &S_x, nullptr);
        const float xx = key_value(kx);
        const double e_x = exact_mass(xx, cff, rf, tab);
        const double tgt = (double)tp * S_x;
        const double jr = (tgt - A_x) / e_x;
        int jx = (int)ceil(jr);
        jx = max(1, min(jx, cnt_x));
        const bool unres = fabs(jr - rint(jr)) < 1e-9 * fmax(1.0, fabs(jr));
        out.cut_x = xx;
        out.cut_id = ordered_ties<ES>(row, a.V, kx, jx, nullptr, s_warp, &s_last);
        out.mass = (A_x + jx * e_x) / S_x;
        if (threadIdx.x == 0) {
            stats_add(a.stats, &a.stats->reresolved, 1);
            if (unres) stats_add(a.stats, &a.stats->unresolved, 1);
        }
    }
    out.log2_mass = log2(out.mass);
    out.mass_f = (float)out.mass;
    if (threadIdx.x == 0) a.nuc[rid] = out;
}

template <int ES>
sv_status launch_nucleus(const RowSet &tgt, const RowSet &drf, long long n_rows0, long long n_rows1, int V,
                         const float *temperature, const float *top_p, const WarpPartial *part, int n_split,
                         RowStat *rowstat, NucleusCut *nuc, sv_stats *stats, const DeviceInfo &di,
                         cudaStream_t stream) {
    (void)rowstat;
    (void)di;
    NucleusArgs a;
    a.set[0] = tgt;
    a.set[1] = drf;
    a.n_rows0 = n_rows0;
    a.n_rows = n_rows0 + n_rows1;
    a.V = V;
    a.temperature = temperature;
    a.top_p = top_p;
    a.part = part;
    a.n_split = n_split;
    a.nuc = nuc;
    a.stats = stats;
    if (a.n_rows < 1) return SV_OK;
    k_nucleus<ES><<<(unsigned)a.n_rows, kThreads, 0, stream>>>(a);
    return cuda_status(cudaGetLastError());
}

// ------------------------------------------------------------------------------------------
// Saguaro top-F set of each draft row and its mass P_D (after temperature and top-p).
// ------------------------------------------------------------------------------------------
struct TopSetArgs {
    RowSet rows;             // draft rows: (b, j) for j < rows.rows_used
    long long rid0;          // candidate-row index of (0, 0)
    long long n_rows;
    int V, F;
    float C;
    const float *temperature;
    const WarpPartial *part;
    int n_split;
    const NucleusCut *nuc;   // indexed by candidate row, or null
    TopSet *top;             // indexed by candidate row
};

template <int ES>
__global__ void __launch_bounds__(kThreads) k_topset(const TopSetArgs a) {
    __shared__ unsigned hist[256];
    __shared__ int s_dig[2], s_warp[kWarps], s_last;
    __shared__ double s_red[kWarps];
    __shared__ RowStat s_rs;
    const long long lr = blockIdx.x;
    if (lr >= a.n_rows) return;
    const long long rid = a.rid0 + lr;
    const long long b = lr / a.rows.rows_used, j = lr - b * a.rows.rows_used;
    const float T = a.temperature[b];
    TopSet none;
    none.top_x = INFINITY;
    none.top_id = -1;
    none.p_d = 0.0;
    none.z = 1.0;
    none.z_err = 0.0;
    none.z_f = 1.0f;
    none.z_err_f = 0.0f;
    if (!(T >= 1e-3f && T <= 1e3f)) {   // greedy or invalid: no transform
        if (threadIdx.x == 0) a.top[rid] = none;
        return;
    }
    const char *row = a.rows.base + (b * a.rows.rows_per_seq + j) * a.rows.pitch_bytes;
    if (threadIdx.x < 32) {
        const RowStat st = combine_row(a.part + (size_t)rid * a.n_split * kWarps, a.n_split * kWarps, false, T);
        if (threadIdx.x == 0) s_rs = st;
    }
    __syncthreads();
    const RowStat st = s_rs;
    if (!rs_sampled_ok(st) || st.flags) {
        if (threadIdx.x == 0) a.top[rid] = none;
        return;
    }
    const int N = min(a.F, a.V);
    int n_above;
    const uint32_t kstar = radix_select_count<ES>(row, a.V, N, n_above, hist, s_dig);
    const int last = ordered_ties<ES>(row, a.V, kstar, N - n_above, nullptr, s_warp, &s_last);
    const float xstar = key_value(kstar);
    // mass of D, restricted to the nucleus when top-p is on
    float c_hi, c_lo;
    log2e_over(T, c_hi, c_lo);
    const float rf = (float)st.r;
    float cut_x = -INFINITY;
    int cut_id = 0x7FFFFFFF;
    double mass_n = 1.0;
    if (a.nuc) {
        cut_x = a.nuc[rid].cut_x;
        cut_id = a.nuc[rid].cut_id;
        mass_n = a.nuc[rid].mass;
    }
    double e_d = 0.0;
    for_each_elem<ES>(row, a.V, [&](float x, int v) {
        const bool in_d = x > xstar || (x == xstar && v <= last);
        const bool keep = x > cut_x || (x == cut_x && v <= cut_id);
        if (in_d && keep) e_d += (double)ex2_fast(fmaf(x, c_lo, fmaf(x, c_hi, -rf)));
    });
    e_d = warp_sum_d(e_d);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = e_d;
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
        for (int w = 0; w < kWarps; ++w) tot += s_red[w];
        TopSet t;
        t.top_x = xstar;
        t.top_id = last;
        t.p_d = fmin(1.0, tot / (rs_S(st) * mass_n));
        t.z = 1.0 - (1.0 - (double)a.C) * t.p_d;
        // p_d is a ratio of two sums of the same pass: relative error <= 2 err (x2 with top-p)
        const double pd_rel = (a.nuc ? 4.04 : 2.02) * rs_err(st);
        t.z_err = t.z > 0.0 ? (1.0 - (double)a.C) * t.p_d * pd_rel / t.z + 1e-12 : 1.0;
        t.z_f = (float)t.z;
        t.z_err_f = (float)t.z_err * (1.0f + 0x1p-20f);
        a.top[rid] = t;
    }
}

template <int ES>
sv_status launch_topset(const RowSet &drf, long long rid0, int B, int rows_used, int V, const float *temperature,
                        int F, float C, const WarpPartial *part, int n_split, const NucleusCut *nuc, TopSet *top,
                        sv_stats *stats, const DeviceInfo &di, cudaStream_t stream) {
    (void)stats;
    (void)di;
    TopSetArgs a;
    a.rows = drf;
    a.rows.rows_used = rows_used;
    a.rid0 = rid0;
    a.n_rows = (long long)B * rows_used;
    a.V = V;
    a.F = F;
    a.C = C;
    a.temperature = temperature;
    a.part = part;
    a.n_split = n_split;
    a.nuc = nuc;
    a.top = top;
    if (a.n_rows < 1) return SV_OK;
    k_topset<ES><<<(unsigned)a.n_rows, kThreads, 0, stream>>>(a);
    return cuda_status(cudaGetLastError());
}

}  // namespace sv
