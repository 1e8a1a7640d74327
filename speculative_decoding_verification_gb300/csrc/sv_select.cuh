// sv_select.cuh — ranking passes over logit rows, one block per row.
//
//  * top-N selection (cache keys, top-kappa roots, the Saguaro top-F set): a most-significant-
//    digit radix select on order-preserving 32-bit keys (two 8-bit passes for bf16, four for
//    float32) finds the key K* of the N-th token; ties at K* are taken in id order by an ordered
//    block scan, so ranking ties go to the lowest id.
//  * top-k and nucleus (top-p) cuts [SpS notes §3 and §6: the filters act on q and on p before
//    the ratio]: the count select finds the k-th token; the same radix select weighted by
//    probability mass 2^(x c - r) finds the shortest prefix in (probability desc, id asc) order
//    whose mass reaches top_p (of the row, or of the top-k set when both are on).  The float32 masses carry a
//    proven error bound; a cut the bound cannot settle is recomputed in float-float in the same
//    block.
#pragma once

#include <cooperative_groups.h>

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
    sv_stats *stats;        // timeouts of the cluster path (may be null)
    int ring_stages;        // cluster path: stages of each block's bulk-copy ring
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
// Top-N of one row by a cluster of S <= 8 blocks (N <= kTopNFast).
//
// Elements are ranked by a 64-bit code: the order key above the complemented id, so that codes
// are distinct and larger codes come first in (key desc, id asc) order.  Each block streams its
// contiguous share of the row through a ring of bulk copies; in a first pass every thread keeps
// the largest key of the vectors it sees.  A key that at least N of those maxima reach is a
// lower bound tau on the row's N-th largest key (N distinct elements reach it), so the row's
// first N are all among the elements of key >= tau.  A second pass over the share (from the
// ring when the share fits in it, else streamed again) marks each thread's group of four
// vectors whose largest key reaches tau, and one warp per marked group turns the elements of
// key >= tau into codes; each block ranks its candidates, and its first N go to
// block 0, which ranks the union: an element of the row's first N has all elements above it in
// the union, so its rank there is its rank in the row.  A block whose candidates overflow
// kTopNCand marks the row, and block 0 then takes it alone by the radix select.
// ------------------------------------------------------------------------------------------
constexpr int kTopNFast = 128;            // largest N of the cluster path
constexpr int kTopNCluster = 8;           // largest cluster
constexpr int kTopNCand = 512;            // candidates one block holds
constexpr int kTopNStageVecs = 1024;      // 16-byte vectors per stage of the bulk-copy ring
constexpr int kTopNStages = 4;            // most ring stages
constexpr size_t kTopNStageBytes = (size_t)kTopNStageVecs * 16;
static_assert(kTopNFast <= kThreads, "one thread per rank of the block's maxima");

__device__ __forceinline__ uint64_t rank_code(uint32_t key, int id) {
    return ((uint64_t)key << 32) | (uint64_t)(~(uint32_t)id);
}
__device__ __forceinline__ uint32_t code_key(uint64_t c) { return (uint32_t)(c >> 32); }
__device__ __forceinline__ int code_id(uint64_t c) { return (int)(~(uint32_t)c); }

// Dynamic shared memory of a row-cluster kernel: the ring (stages x kTopNStageBytes), then
// block 0's gather area (block q's sorted first N at q * N: S * N codes).
inline size_t topn_dyn_bytes(int stages, int S, int n_max) {
    return (size_t)stages * kTopNStageBytes + (size_t)S * n_max * sizeof(uint64_t);
}

struct TopNCl {
    uint64_t cand[kTopNCand];                  // this block's candidates (radix path: keys, ids)
    uint64_t res[kTopNFast];                   // block 0: the row's first N, sorted
    uint32_t mx[2 * kThreads];                 // thread maxima; the marked vectors; radix path: tie ids
    uint32_t taus[kTopNCluster];               // block q's bound, written by block q
    uint32_t tau_b;
    uint64_t bar[kTopNStages];                 // ring stages
    int n_top[kTopNCluster], over[kTopNCluster];
    int n_cand, n_mark, fail;
    uint32_t nth_key;                          // block 0: the row's N-th element
    int nth_id;
    unsigned hist[256];                        // radix path
    int dig[2], warp_tot[kWarps], last, cnt;
};

// Elements g, g + G, ... of the row in 16-byte vectors (four loads in flight per thread), then
// the scalar tail.
template <int ES, class Fn>
__device__ __forceinline__ void for_strided(const char *row, int V, int g, int G, Fn fn) {
    constexpr int EPV = 16 / ES;
    const int n_vec = (V * ES) / 16;
    const uint4 *p = reinterpret_cast<const uint4 *>(row);
    int vi = g;
    for (; vi + 3 * G < n_vec; vi += 4 * G) {
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) w[u] = __ldg(p + vi + u * G);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float x[EPV];
            unpack<ES>(w[u], x);
#pragma unroll
            for (int k = 0; k < EPV; ++k) fn(x[k], (vi + u * G) * EPV + k);
        }
    }
    for (; vi < n_vec; vi += G) {
        float x[EPV];
        unpack<ES>(__ldg(p + vi), x);
#pragma unroll
        for (int k = 0; k < EPV; ++k) fn(x[k], vi * EPV + k);
    }
    for (int v = n_vec * EPV + g; v < V; v += G) fn(load_elem<ES>(row, v), v);
}

// The largest order key of a 16-byte vector, exactly: the maximum ignores NaN (an all-NaN
// result sends the vector to the per-element keys), and -0 shares +0's key.
template <int ES>
__device__ __forceinline__ uint32_t vec_key_max(uint4 w) {
    float m;
    if constexpr (ES == 2) {
        uint32_t h;
        asm("max.bf16x2 %0, %1, %2;" : "=r"(h) : "r"(w.x), "r"(w.y));
        uint32_t h2;
        asm("max.bf16x2 %0, %1, %2;" : "=r"(h2) : "r"(w.z), "r"(w.w));
        asm("max.bf16x2 %0, %1, %2;" : "=r"(h) : "r"(h), "r"(h2));
        asm("max.bf16x2 %0, %1, %2;" : "=r"(h) : "r"(h), "r"(__byte_perm(h, 0u, 0x1032)));
        m = bf16_lo(h);
    } else {
        m = fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)), fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
    uint32_t k = f32_key(m);
    if (__any_sync(__activemask(), m != m)) {   // never on finite rows: a uniform branch
        if (m != m) {                            // every element NaN
            float x[16 / ES];
            unpack<ES>(w, x);
            k = 0u;
#pragma unroll
            for (int i = 0; i < 16 / ES; ++i) k = max(k, f32_key(x[i]));
        }
    }
    return k;
}

// The largest order key of four 16-byte vectors (one packed maximum tree, then one key), exactly
// as vec_key_max.
template <int ES>
__device__ __forceinline__ uint32_t group_key_max(const uint4 (&w)[4]) {
    float m;
    if constexpr (ES == 2) {
        uint32_t a[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t h0, h1;
            asm("max.bf16x2 %0, %1, %2;" : "=r"(h0) : "r"(w[k].x), "r"(w[k].y));
            asm("max.bf16x2 %0, %1, %2;" : "=r"(h1) : "r"(w[k].z), "r"(w[k].w));
            asm("max.bf16x2 %0, %1, %2;" : "=r"(a[k]) : "r"(h0), "r"(h1));
        }
        asm("max.bf16x2 %0, %1, %2;" : "=r"(a[0]) : "r"(a[0]), "r"(a[1]));
        asm("max.bf16x2 %0, %1, %2;" : "=r"(a[2]) : "r"(a[2]), "r"(a[3]));
        asm("max.bf16x2 %0, %1, %2;" : "=r"(a[0]) : "r"(a[0]), "r"(a[2]));
        asm("max.bf16x2 %0, %1, %2;" : "=r"(a[0]) : "r"(a[0]), "r"(__byte_perm(a[0], 0u, 0x1032)));
        m = bf16_lo(a[0]);
    } else {
        float a[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            a[k] = fmaxf(fmaxf(__uint_as_float(w[k].x), __uint_as_float(w[k].y)),
                         fmaxf(__uint_as_float(w[k].z), __uint_as_float(w[k].w)));
        m = fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3]));
    }
    uint32_t k = f32_key(m);
    if (__any_sync(__activemask(), m != m)) {   // never on finite rows: a uniform branch
        if (m != m) {                            // every element NaN
            k = 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float x[16 / ES];
                unpack<ES>(w[j], x);
#pragma unroll
                for (int i = 0; i < 16 / ES; ++i) k = max(k, f32_key(x[i]));
            }
        }
    }
    return k;
}

// The 32 values of a warp in descending order across lanes (bitonic network).
__device__ __forceinline__ uint32_t warp_sort_desc(uint32_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const uint32_t o = __shfl_xor_sync(0xFFFFFFFFu, v, j);
            const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
            v = keep_max ? max(v, o) : min(v, o);
        }
    return v;
}

// Rank of (k, id) among n (key, id) pairs in (key desc, id asc) order.
__device__ __forceinline__ int pair_rank(const uint32_t *keys, const int *ids, int n, uint32_t k, int id) {
    int r = 0;
    for (int j = 0; j < n; ++j) {
        const uint32_t o = keys[j];
        r += (o > k || (o == k && ids[j] < id)) ? 1 : 0;
    }
    return r;
}

// Single-block radix select: the N-th element into nth_key / nth_id and, in list mode
// (N <= kTopNFast), the sorted first N as codes in res.
template <int ES>
__device__ void topn_exact_block(const char *row, int V, int N, bool list, TopNCl &s) {
    uint32_t *xkey = reinterpret_cast<uint32_t *>(s.cand);
    int *xid = reinterpret_cast<int *>(s.cand) + kTopNCand;
    int *tie = reinterpret_cast<int *>(s.mx);
    int n_above;
    const uint32_t kstar = radix_select_count<ES>(row, V, N, n_above, s.hist, s.dig);
    if (!list) {
        const int last = ordered_ties<ES>(row, V, kstar, N - n_above, nullptr, s.warp_tot, &s.last);
        if (threadIdx.x == 0) {
            s.nth_key = kstar;
            s.nth_id = last;
        }
        __syncthreads();
        return;
    }
    if (threadIdx.x == 0) s.cnt = 0;
    __syncthreads();
    for_each_elem<ES>(row, V, [&](float x, int v) {
        const uint32_t k = f32_key(x);
        if (k > kstar) {
            const int slot = atomicAdd(&s.cnt, 1);
            if (slot < kTopNCand) {
                xkey[slot] = k;
                xid[slot] = v;
            }
        }
    });
    __syncthreads();
    const int na = min(s.cnt, kTopNCand);   // = n_above < N
    for (int i = threadIdx.x; i < na; i += blockDim.x)
        s.res[pair_rank(xkey, xid, na, xkey[i], xid[i])] = rank_code(xkey[i], xid[i]);
    ordered_ties<ES>(row, V, kstar, N - na, tie, s.warp_tot, &s.last);
    for (int i = threadIdx.x; i < N - na; i += blockDim.x) s.res[na + i] = rank_code(kstar, tie[i]);
    __syncthreads();
    if (threadIdx.x == 0) {
        s.nth_key = code_key(s.res[N - 1]);
        s.nth_id = code_id(s.res[N - 1]);
    }
    __syncthreads();
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// The cluster part of the top-N of one row, called by every block of the cluster (1 <= N <=
// min(V, kTopNFast)).  Block `rank` takes the contiguous share [v0, v1) of the row's 16-byte
// vectors, streamed by bulk copies through `ring` (`stages` x kTopNStageBytes of dynamic
// shared memory, followed by S * N codes of block 0's gather area); its
// thread tid sees vectors v0 + tid + k kThreads, in increasing order.  `each_vec(w, vi)` sees
// every vector of the share once and `each_elem(x, v)` every scalar-tail element; `publish()`
// runs in every block just before the last barrier (to write per-block results into block 0).
// Returns true in block 0 when the row needs the radix path (a block's candidates overflowed);
// otherwise block 0 holds the row's first N in res and the N-th element in nth_key / nth_id.
// Other blocks return false and must not touch block 0 after.  s.fail is set in a block whose
// copies did not arrive in time (its results are then meaningless; the caller reports it).
template <int ES, class EachVec, class EachElem, class Publish>
__device__ bool cluster_topn(const cooperative_groups::cluster_group &cl, const char *row, int V, int N, TopNCl &s,
                             char *ring, int stages, long long wait_limit, EachVec each_vec, EachElem each_elem,
                             Publish publish) {
    constexpr int EPV = 16 / ES;
    const int S = (int)cl.num_blocks(), rank = (int)cl.block_rank();
    const int tid = threadIdx.x, lane = tid & 31;
    const int g = rank * kThreads + tid, G = S * kThreads;
    const int n_vec = (V * ES) / 16;
    const int per = (n_vec + S - 1) / S;
    const int v0 = min(rank * per, n_vec), v1 = min(v0 + per, n_vec);
    const int n_chunks = (v1 - v0 + kTopNStageVecs - 1) / kTopNStageVecs;
    // the ring carries a sequence of chunks j: the share once (j < n_chunks) and, unless the
    // whole share stays in the ring, once more for the second pass (chunk j - n_chunks of the
    // share)
    uint64_t *gath = reinterpret_cast<uint64_t *>(ring + (size_t)stages * kTopNStageBytes);
    const bool resident = n_chunks <= stages;
    const int total = resident ? n_chunks : 2 * n_chunks;
    auto chunk_vecs = [&](int c) { return min(kTopNStageVecs, v1 - v0 - c * kTopNStageVecs); };
    auto issue = [&](int j) {   // thread 0
        const int c = j < n_chunks ? j : j - n_chunks, st = j % stages;
        const uint32_t bytes = (uint32_t)chunk_vecs(c) * 16u;
        mbar_arrive_expect_tx(&s.bar[st], bytes);
        bulk_load(ring + (size_t)st * kTopNStageBytes, row + (size_t)(v0 + c * kTopNStageVecs) * 16, bytes,
                  &s.bar[st]);
    };
    cluster_arrive_relaxed();   // completes once every block has started (before any DSMEM access)
    if (tid == 0) {
        s.tau_b = 0u;
        s.n_cand = 0;
        s.n_mark = 0;
        s.fail = 0;
        for (int i = 0; i < stages; ++i) mbar_init(&s.bar[i], 1);
        fence_barrier_init();
        for (int j = 0; j < min(stages, total); ++j) issue(j);
    }
    __syncthreads();
    // A thread's vectors of a chunk: tid + k kThreads for k < n (n <= 4, as kTopNStageVecs = 4
    // kThreads); absent ones repeat the first, so a group's maximum is the maximum of its vectors.
    auto group = [&](const char *base, int nv, int vbase, auto fn4) {
        if (tid >= nv) return;
        uint4 w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = tid + k * kThreads;
            w[k] = (k == 0 || i < nv) ? lds128(base + i * 16) : w[0];
        }
        fn4(w, min(4, (nv - tid + kThreads - 1) / kThreads), vbase + tid);
    };
    static_assert(kTopNStageVecs == 4 * kThreads, "a thread's vectors of a chunk form one group");
    // consumes ring chunks j0 .. j1-1 with fn4(w[4], n, vi0); refills each stage once every
    // thread is done with it.  A copy late beyond wait_limit ends the streaming (s.fail) after
    // the copies still in flight have landed (bounded).
    bool failed = false;
    auto stream = [&](int j0, int j1, auto fn) {
        if (failed) return;
        for (int j = j0; j < j1; ++j) {
            const int st = j % stages, c = j < n_chunks ? j : j - n_chunks;
            const bool ok = mbar_wait_bounded(&s.bar[st], (uint32_t)(j / stages) & 1u, wait_limit);
            if (ok) group(ring + (size_t)st * kTopNStageBytes, chunk_vecs(c), v0 + c * kTopNStageVecs, fn);
            if (__syncthreads_or(!ok)) {
                const int issued = min(j + stages, total);
                for (int d = j; d < issued; ++d)
                    mbar_wait_bounded(&s.bar[d % stages], (uint32_t)(d / stages) & 1u, wait_limit);
                if (tid == 0) s.fail = 1;
                failed = true;
                return;
            }
            if (tid == 0 && j + stages < total) issue(j + stages);
        }
    };
    // ---- pass 1: each thread's largest key ----
    uint32_t mk = 0u;
    stream(0, n_chunks, [&](const uint4 (&w)[4], int n, int vi0) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (k < n) each_vec(w[k], vi0 + k * kThreads);
        mk = max(mk, group_key_max<ES>(w));
    });
    for (int v = n_vec * EPV + g; v < V; v += G) {
        const float x = load_elem<ES>(row, v);
        each_elem(x, v);
        mk = max(mk, f32_key(x));
    }
    // the block's bound: the largest key that N thread maxima reach (0: none, below every key)
    if (N <= 32) {
        const uint32_t w = __shfl_sync(0xFFFFFFFFu, warp_sort_desc(mk), N - 1);
        if (lane == 0) atomicMax(&s.tau_b, w);
    } else {
        s.mx[tid] = mk;
        __syncthreads();
        int r = 0;
        for (int j = 0; j < kThreads; ++j) r += s.mx[j] >= mk ? 1 : 0;
        if (r >= N) atomicMax(&s.tau_b, mk);
    }
    __syncthreads();
    cluster_wait();
    if (tid < S) *cl.map_shared_rank(&s.taus[rank], tid) = s.tau_b;
    cl.sync();   // (1) every block's bound is in every block
    uint32_t tau = 0u;
    for (int q = 0; q < S; ++q) tau = max(tau, s.taus[q]);
    // ---- pass 2: the codes of the elements of key >= tau ----
    // A cheap sweep marks the groups whose largest key reaches tau (few); their elements are
    // then expanded, one group per thread.
    auto add = [&](uint64_t c) {
        const int slot = atomicAdd(&s.n_cand, 1);
        if (slot < kTopNCand) s.cand[slot] = c;
    };
    constexpr int kMarkCap = 2 * kThreads;
    auto mark = [&](const uint4 (&w)[4], int, int vi0) {
        if (group_key_max<ES>(w) >= tau) {
            const int slot = atomicAdd(&s.n_mark, 1);
            if (slot < kMarkCap) s.mx[slot] = (uint32_t)vi0;
        }
    };
    if (resident) {
        if (!failed)
            for (int c = 0; c < n_chunks; ++c)
                group(ring + (size_t)c * kTopNStageBytes, chunk_vecs(c), v0 + c * kTopNStageVecs, mark);
    } else {
        stream(n_chunks, total, mark);
    }
    for (int v = n_vec * EPV + g; v < V; v += G) {
        const uint32_t key = f32_key(load_elem<ES>(row, v));
        if (key >= tau) add(rank_code(key, v));
    }
    __syncthreads();
    const int n_mark = s.n_mark;
    if (n_mark > kMarkCap) {
        if (tid == 0) s.n_cand = kTopNCand + 1;   // overflow: the radix path
    } else {
        // one warp per marked group: lane l takes element l % EPV of vector l / EPV of the group
        // (lanes 0 .. 4 EPV - 1)
        const int warp = tid >> 5;
        for (int i = warp; i < n_mark; i += kWarps) {
            const int vi0 = (int)s.mx[i];
            const int c = (vi0 - v0) / kTopNStageVecs;
            const int vend = v0 + c * kTopNStageVecs + chunk_vecs(c);   // end of the group's chunk
            const int vi = vi0 + (lane / EPV) * kThreads, e = vi * EPV + lane % EPV;
            if (lane < 4 * EPV && vi < vend) {
                const float x = resident ? (ES == 2 ? bf16_lo((uint32_t)*reinterpret_cast<const unsigned short *>(
                                                          ring + (size_t)(vi - v0) * 16 + (lane % EPV) * 2))
                                                    : *reinterpret_cast<const float *>(ring + (size_t)(vi - v0) * 16 +
                                                                                       (lane % EPV) * 4))
                                         : load_elem<ES>(row, e);
                const uint32_t key = f32_key(x);
                if (key >= tau) add(rank_code(key, e));
            }
        }
    }
    __syncthreads();
    const int nc = s.n_cand;
    if (nc <= kTopNCand) {
        uint64_t *dst = cl.map_shared_rank(gath, 0) + rank * N;
        for (int i = tid; i < nc; i += kThreads) {
            const uint64_t c = s.cand[i];
            int r = 0;
#pragma unroll 8
            for (int j = 0; j < nc; ++j) r += s.cand[j] > c ? 1 : 0;
            if (r < N) dst[r] = c;
        }
    }
    if (tid == 0) {
        *cl.map_shared_rank(&s.n_top[rank], 0) = min(nc, N);
        *cl.map_shared_rank(&s.over[rank], 0) = nc > kTopNCand ? 1 : 0;
    }
    publish();
    cl.sync();   // (2) every block's list and results are in block 0
    if (rank != 0) return false;
    int over = 0;
    for (int q = 0; q < S; ++q) over |= s.over[q];
    if (over) return true;
    for (int idx = tid; idx < S * N; idx += kThreads) {
        const int q = idx / N, i = idx - q * N;
        if (i >= s.n_top[q]) continue;
        const uint64_t c = gath[idx];
        int r = 0;
        for (int q2 = 0; q2 < S; ++q2) {
            const uint64_t *l = gath + q2 * N;
            const int n = s.n_top[q2];
            for (int j = 0; j < n; ++j) r += l[j] > c ? 1 : 0;
        }
        if (r < N) s.res[r] = c;
    }
    __syncthreads();
    if (tid == 0) {
        s.nth_key = code_key(s.res[N - 1]);
        s.nth_id = code_id(s.res[N - 1]);
    }
    __syncthreads();
    return false;
}

// Top-N lists by clusters: cluster c of the grid takes row c.
template <int ES>
__global__ void __launch_bounds__(kThreads) k_topn_cl(const TopNArgs a) {
    __shared__ TopNCl s;
    extern __shared__ __align__(128) char ring[];
    const cooperative_groups::cluster_group cl = cooperative_groups::this_cluster();
    const long long r = blockIdx.x / cl.num_blocks();
    if (r >= a.n_rows) return;
    const long long b = r / a.rows_used, j = r - b * a.rows_used;
    const char *row = a.base + (b * a.rows_per_seq + j) * a.pitch_bytes;
    int N = a.n_all > 0 ? a.n_all : a.n_of_j[j];
    if (N > a.V) N = a.V;
    if (N <= 0) return;   // the same in every block of the cluster
    const bool radix = cluster_topn<ES>(cl, row, a.V, N, s, ring, a.ring_stages, kWaitLimitCycles, [](uint4, int) {},
                                        [](float, int) {}, [] {});
    if (s.fail && threadIdx.x == 0) report_error(a.stats, SV_ERR_TIMEOUT, (int)r);
    if (cl.block_rank() != 0) return;
    if (radix) topn_exact_block<ES>(row, a.V, N, true, s);
    int32_t *out = a.list + (size_t)r * a.list_stride;
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
        const int id = code_id(s.res[i]);
        out[i] = id;
        if (a.list_x) a.list_x[(size_t)r * a.list_stride + i] = load_elem<ES>(row, id);
    }
}

// Cluster size for n_rows rows: two blocks for every SM when the rows are few (a block of a
// 128256-token bf16 row then keeps its whole 64 KB share in its ring, three blocks to an SM),
// at most kTopNCluster per row.
inline int topn_cluster_size(long long n_rows, int sms) {
    int S = 1;
    while (S < kTopNCluster && n_rows * S < 2LL * sms) S *= 2;
    return S;
}

// Ring stages for shares of a row of n_vec vectors over S blocks: enough to hold a share (then
// the second pass reads shared memory), at most kTopNStages.
inline int topn_ring_stages(int n_vec, int S) {
    const int share = (n_vec + S - 1) / S;
    const int chunks = (share + kTopNStageVecs - 1) / kTopNStageVecs;
    return chunks < 1 ? 1 : (chunks > kTopNStages ? kTopNStages : chunks);
}

// Launch of a row-per-cluster kernel: grid = n_rows * S blocks, clusters of S.
template <class Args>
cudaError_t launch_row_clusters(void (*kern)(Args), const Args &args, long long n_rows, int S, size_t smem,
                                cudaStream_t stream) {
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_rows * S));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

// Top-N lists of TopNArgs rows: the cluster path when every N fits it, else one block per row.
template <int ES>
cudaError_t launch_topn(const TopNArgs &ta_in, int max_n, int sms, cudaStream_t stream) {
    if (ta_in.n_rows < 1) return cudaSuccess;
    if (max_n <= kTopNFast) {
        TopNArgs ta = ta_in;
        const int S = topn_cluster_size(ta.n_rows, sms);
        ta.ring_stages = topn_ring_stages((int)((long long)ta.V * ES / 16), S);
        return launch_row_clusters(k_topn_cl<ES>, ta, ta.n_rows, S, topn_dyn_bytes(ta.ring_stages, S, max_n), stream);
    }
    const TopNArgs &ta = ta_in;
    k_topn<ES><<<(unsigned)ta.n_rows, kThreads, 0, stream>>>(ta);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// Nucleus cut of each sampled row.
// ------------------------------------------------------------------------------------------
struct NucleusArgs {
    RowSet set[2];
    long long n_rows0, n_rows;
    int V;
    const float *temperature;
    const float *top_p;      // [B] or null
    const int32_t *top_k;    // [B] or null
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

// Block sums of three doubles; every thread gets the totals.  s_red holds 3 * kWarps doubles.
__device__ __forceinline__ double3 block_sum_d3(double x, double y, double z, double *s_red) {
    x = warp_sum_d(x);
    y = warp_sum_d(y);
    z = warp_sum_d(z);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        s_red[w] = x;
        s_red[kWarps + w] = y;
        s_red[2 * kWarps + w] = z;
    }
    __syncthreads();
    double3 t = {0.0, 0.0, 0.0};
    for (int i = 0; i < kWarps; ++i) {
        t.x += s_red[i];
        t.y += s_red[kWarps + i];
        t.z += s_red[2 * kWarps + i];
    }
    __syncthreads();
    return t;
}

// The filters of one row as one upper set of the (logit desc, id asc) order.  Top-k keeps
// the first k tokens: a count-weighted select finds the key of the k-th, exactly.  Top-p keeps
// the shortest prefix whose mass reaches top_p times the mass it filters (the whole row, or
// the top-k set when both are on: top-k acts first and the nucleus is that of the
// renormalised top-k distribution, and since both are prefixes of one order the result is
// the shorter of the two).  Masses: float32 with a proven bound, float-float when the bound
// cannot settle the nucleus cut.
template <int ES>
__global__ void __launch_bounds__(kThreads) k_nucleus(const NucleusArgs a) {
    pdl_trigger();   // a dependent launch may be scheduled; it waits for this kernel
    __shared__ double hm[256 + kWarps];
    __shared__ unsigned hc[256];
    __shared__ int s_dig[2], s_warp[kWarps], s_last;
    __shared__ double s_dm[2];
    __shared__ double s_red[3 * kWarps];
    __shared__ float2 tab[256];
    __shared__ RowStat s_rs;
    const long long rid = blockIdx.x;
    if (rid >= a.n_rows) return;
    const int s = rid < a.n_rows0 ? 0 : 1;
    const long long lr = s == 0 ? rid : rid - a.n_rows0;
    const RowSet &rs = a.set[s];
    const long long b = lr / rs.rows_used, j = lr - b * rs.rows_used;
    const float T = a.temperature[b];
    const float tp = a.top_p ? a.top_p[b] : 1.0f;
    const int tk = a.top_k ? a.top_k[b] : 0;
    const bool p_on = tp < 1.0f;
    const bool k_on = tk > 0 && tk < a.V;
    NucleusCut none;
    none.cut_x = -INFINITY;
    none.cut_id = 0x7FFFFFFF;
    none.mass = 1.0;
    none.log2_mass = 0.0;
    none.ambiguous = 0;
    none.mass_f = 1.0f;
    if (!(p_on || k_on) || !(T >= 1e-3f && T <= 1e3f)) {   // off, greedy or invalid temperature
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

    // ---- top-k: the key of the k-th token and how many of its ties are kept ----
    uint32_t kk = 0;
    int k_ties = 0;
    float xk = -INFINITY;
    if (k_on) {
        int n_above;
        kk = radix_select_count<ES>(row, a.V, tk, n_above, hc, s_dig);
        k_ties = tk - n_above;
        xk = key_value(kk);
    }

    // ---- float32 tier: masses 2^(x c - r) as in the statistics pass ----
    auto fast_mass = [&](float x) {   // (mass, mass * |y|): the second feeds the error bound
        const float y = fmaf(x, c_lo, fmaf(x, c_hi, -rf));
        const float e = ex2_fast(y);
        return make_double2((double)e, (double)(e * fabsf(y)));
    };
    double S_fast = 0.0, A_row = 0.0, M_above_k = 0.0, M_k = 0.0, e_k = 0.0;
    if (k_on) {   // row sum, error weight and the top-k mass in one pass
        double ts = 0.0, ta = 0.0, tm = 0.0;
        for_each_elem<ES>(row, a.V, [&](float x, int) {
            const double2 w = fast_mass(x);
            ts += w.x;
            ta += w.y;
            if (f32_key(x) > kk) tm += w.x;
        });
        const double3 t = block_sum_d3(ts, ta, tm, s_red);
        S_fast = t.x;
        A_row = t.y;
        M_above_k = t.z;
        e_k = fast_mass(xk).x;
        M_k = M_above_k + k_ties * e_k;
    }
    uint32_t kstar = kk;
    float xstar = xk;
    double above_m = M_above_k, estar = e_k, target = M_k;
    int jt = k_ties;
    if (p_on) {
        int cnt_star;
        if (k_on) {
            target = (double)tp * M_k;
            kstar = radix_select_mass<ES>(row, a.V, target, 0.0, fast_mass, hm, hc, s_dig, s_dm, s_red, above_m,
                                          cnt_star, nullptr, nullptr);
        } else {
            kstar = radix_select_mass<ES>(row, a.V, 0.0, (double)tp, fast_mass, hm, hc, s_dig, s_dm, s_red, above_m,
                                          cnt_star, &S_fast, &A_row);
            target = (double)tp * S_fast;
        }
        xstar = key_value(kstar);
        estar = fast_mass(xstar).x;
        jt = (int)ceil((target - above_m) / estar);
        jt = max(1, min(jt, cnt_star));
        if (k_on && (kstar < kk || (kstar == kk && jt > k_ties))) {   // past the top-k set
            kstar = kk;
            xstar = xk;
            jt = k_ties;
            estar = e_k;
            above_m = M_above_k;
        }
    }
    // certification: cum and target come from the same per-element masses; the kept set is an
    // upper set, so its error per unit mass is at most the row's (weighted mean of |y|).  A
    // top-k cut alone involves no rounding.
    // the float64 certification by thread 0 alone (this GPU's float64 pipe is narrow)
    __shared__ int s_amb;
    if (threadIdx.x == 0) {
        const double cum_hi = above_m + jt * estar, cum_lo = above_m + (jt - 1) * estar;
        const double rel = kEx2RelErr + 1.02 * kYRound * (A_row / S_fast) + 4.0 * kU32 + 1e-12;
        const double E = rel * (cum_hi + target) + 1e-15 * S_fast;
        s_amb = p_on && ((target - cum_lo) <= E || (cum_hi - target) <= E) ? 1 : 0;
    }
    __syncthreads();
    const bool ambiguous = s_amb != 0;
    double m_num = 0.0, m_den = 1.0;   // the kept mass num / den, formed by thread 0 below
    NucleusCut out;
    out.ambiguous = ambiguous ? 1 : 0;
    out.mass_f = 1.0f;
    if (!ambiguous) {
        out.cut_x = xstar;
        out.cut_id = ordered_ties<ES>(row, a.V, kstar, jt, nullptr, s_warp, &s_last);
        m_num = above_m + jt * estar;
        m_den = S_fast;
    } else {
        // ---- float-float tier: the same selects on exact masses ----
        tab[threadIdx.x] = kExp2Table[threadIdx.x];
        __syncthreads();
        const ff cff = {c_hi, c_lo};
        auto exact = [&](float x) { return make_double2(exact_mass(x, cff, rf, tab), 0.0); };
        double A_x, S_x, tgt, M_above_kx = 0.0, e_kx = 0.0;
        int cnt_x;
        uint32_t kx;
        if (k_on) {
            double ts = 0.0, tm = 0.0;
            for_each_elem<ES>(row, a.V, [&](float x, int) {
                const double m = exact(x).x;
                ts += m;
                if (f32_key(x) > kk) tm += m;
            });
            const double3 t = block_sum_d3(ts, tm, 0.0, s_red);
            S_x = t.x;
            M_above_kx = t.y;
            e_kx = exact(xk).x;
            tgt = (double)tp * (M_above_kx + k_ties * e_kx);
            kx = radix_select_mass<ES>(row, a.V, tgt, 0.0, exact, hm, hc, s_dig, s_dm, s_red, A_x, cnt_x, nullptr,
                                       nullptr);
        } else {
            kx = radix_select_mass<ES>(row, a.V, 0.0, (double)tp, exact, hm, hc, s_dig, s_dm, s_red, A_x, cnt_x, &S_x,
                                       nullptr);
            tgt = (double)tp * S_x;
        }
        float xx = key_value(kx);
        double e_x = exact(xx).x;
        double jr = (tgt - A_x) / e_x;
        int jx = (int)ceil(jr);
        jx = max(1, min(jx, cnt_x));
        if (k_on && (kx < kk || (kx == kk && jx > k_ties))) {
            kx = kk;
            xx = xk;
            e_x = e_kx;
            A_x = M_above_kx;
            jx = k_ties;
            jr = (tgt - A_x) / e_x;
        }
        const bool unres = fabs(jr - rint(jr)) < 1e-9 * fmax(1.0, fabs(jr));
        out.cut_x = xx;
        out.cut_id = ordered_ties<ES>(row, a.V, kx, jx, nullptr, s_warp, &s_last);
        m_num = A_x + jx * e_x;
        m_den = S_x;
        if (threadIdx.x == 0) {
            stats_add(a.stats, &a.stats->reresolved, 1);
            if (unres) stats_add(a.stats, &a.stats->unresolved, 1);
        }
    }
    if (threadIdx.x != 0) return;
    out.mass = m_num / m_den;
    out.log2_mass = log2(out.mass);
    out.mass_f = (float)out.mass;
    a.nuc[rid] = out;
}

// ------------------------------------------------------------------------------------------
// bf16 rows: the filters from a histogram of the row's values.
//
// A bf16 logit takes one of 65536 values and its 16-bit order key is its rank among them.  A
// cluster of kNucSplit blocks shares a row: block q holds one counter per value for the q-th
// quarter of the keys from the top (64 KB of shared memory), and each block reads a quarter of
// the row and adds its tokens to the counters of whichever block holds their values
// (distributed shared memory).  All tokens of one value carry the same mass 2^(x c - r), so the
// mass a value holds is its count times one float-float exponential, and the cumulative count
// and mass in (value desc) order come from scans over the counters rather than the tokens.  The
// k-th token and the nucleus cut follow from float-float masses (relative error ~2^-44 each);
// the position inside the cut's group of equal values is then found in id order.
// ------------------------------------------------------------------------------------------
constexpr int kNucSplit = 4;                                  // blocks per row
constexpr int kNucKeys = 65536 / kNucSplit;                   // values counted per block
constexpr int kNucBins = kNucKeys / kThreads;                 // values per thread segment (64)
constexpr size_t kNucHistBytes = kNucKeys * sizeof(unsigned);
static_assert(kNucBins == 64, "two values per lane per segment");

struct NucXch {   // what one block of the cluster publishes to the others
    ff mass;      // total mass of the block's keys / mass strictly above a located cut
    ff each;      // mass of one token at the cut's value
    int count;    // tokens in the block's keys / tokens of the cut's value
    int key, pos; // a located cut: 16-bit key and how many of its equal values are kept
    int pad;
};

// 16-bit order key of a bf16 bit pattern (-0 ranks with +0).
__device__ __forceinline__ uint32_t bf16_key16(uint32_t bits) {
    if (bits == 0x8000u) bits = 0u;
    return (bits & 0x8000u) ? (0xFFFFu - bits) : (bits | 0x8000u);
}

// The bf16 value of a 16-bit order key.
__device__ __forceinline__ float bf16_key_value(uint32_t k16) {
    const uint32_t bits = (k16 & 0x8000u) ? (k16 & 0x7FFFu) : (0xFFFFu - k16);
    return __uint_as_float(bits << 16);
}

// Float-float mass 2^(x c - r) of one token of the value with key k16.
__device__ __forceinline__ ff key_mass(uint32_t k16, ff c, int r, const float2 *tab) {
    const float x = bf16_key_value(k16);
    if (x == -INFINITY) return {0.f, 0.f};
    return ff_exp2_xc(x, c, r, tab);
}

__device__ __forceinline__ ff ff_shfl_xor(ff v, int o) {
    return {__shfl_xor_sync(0xFFFFFFFFu, v.hi, o), __shfl_xor_sync(0xFFFFFFFFu, v.lo, o)};
}
__device__ __forceinline__ ff ff_shfl_up(ff v, int o) {
    return {__shfl_up_sync(0xFFFFFFFFu, v.hi, o), __shfl_up_sync(0xFFFFFFFFu, v.lo, o)};
}
__device__ __forceinline__ ff ff_shfl(ff v, int l) {
    return {__shfl_sync(0xFFFFFFFFu, v.hi, l), __shfl_sync(0xFFFFFFFFu, v.lo, l)};
}
__device__ __forceinline__ bool ff_ge(ff a, ff b) { return a.hi > b.hi || (a.hi == b.hi && a.lo >= b.lo); }
__device__ __forceinline__ ff ff_times(ff m, unsigned n) { return ff_mul(m, {(float)n, 0.f}); }

// A located cut inside one block's keys, in (value desc) order: the value `key`, of which `pos`
// tokens are kept; `mass` is the mass strictly above it and `each` one token's mass.  Count
// mode: the need-th token from the top of the block.  Mass mode: the first value at which base +
// the cumulative mass reaches target.  Called by the whole block; one warp walks the segment
// that holds the cut and writes *out.
__device__ __forceinline__ void locate_cut(bool by_mass, int need, ff base, ff target, uint32_t kbase,
                                           const unsigned *cnt, const int *exc, const ff *exm, const int *segc,
                                           const ff *segm, ff c, int r, const float2 *tab, int *s_owner, NucXch *out) {
    const int t = threadIdx.x, lane = t & 31;
    if (t == 0) *s_owner = kThreads;
    __syncthreads();
    const bool mine = segc[t] > 0 && (by_mass ? ff_ge(ff_add(base, ff_add(exm[t], segm[t])), target)
                                              : exc[t] + segc[t] >= need);
    if (mine) atomicMin(s_owner, t);
    __syncthreads();
    int owner = *s_owner;
    if (owner == kThreads) {   // rounding left the mass short of target: the last occupied value
        __syncthreads();
        if (t == 0) *s_owner = -1;
        __syncthreads();
        if (segc[t] > 0) atomicMax(s_owner, t);
        __syncthreads();
        owner = *s_owner;
        if (owner < 0 && t == 0) *out = {base, {0.f, 0.f}, 0, (int)kbase, 1, 0};   // an empty block (not reached)
    }
    if (owner >= 0 && (t >> 5) == (owner >> 5)) {
        const int top = kNucKeys - 1 - kNucBins * owner;
        ff cum = ff_add(base, exm[owner]);
        int cc = exc[owner];
        bool done = false;
        int last_lane = -1;
        NucXch last = {};
        for (int g = 0; g < 2 && !done; ++g) {
            const int li = top - (32 * g + lane);
            const unsigned n = cnt[li];
            const uint32_t k16 = kbase + (uint32_t)li;
            const ff m = n ? key_mass(k16, c, r, tab) : ff{0.f, 0.f};
            const ff add = n ? ff_times(m, n) : ff{0.f, 0.f};
            int ci = (int)n;
            ff mi = add;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int tc = __shfl_up_sync(0xFFFFFFFFu, ci, o);
                const ff tm = ff_shfl_up(mi, o);
                if (lane >= o) {
                    ci += tc;
                    mi = ff_add(tm, mi);
                }
            }
            ff ex = ff_shfl_up(mi, 1);
            int cx = __shfl_up_sync(0xFFFFFFFFu, ci, 1);
            if (lane == 0) {
                ex = {0.f, 0.f};
                cx = 0;
            }
            const ff above = ff_add(cum, ex);
            const bool cross = n > 0 && (by_mass ? ff_ge(ff_add(cum, mi), target) : cc + ci >= need);
            const unsigned mask = __ballot_sync(0xFFFFFFFFu, cross);
            const unsigned occ = __ballot_sync(0xFFFFFFFFu, n > 0);
            if (mask) {
                if (lane == __ffs(mask) - 1) {
                    int pos;
                    if (by_mass) {
                        const ff d = ff_sub(target, above);
                        const double md = ff_to_double(m);
                        pos = md > 0.0 ? (int)ceil(ff_to_double(d) / md) : 1;
                    } else {
                        pos = need - (cc + cx);
                    }
                    *out = {above, m, (int)n, (int)k16, max(1, min(pos, (int)n)), 0};
                }
                done = true;
            } else if (occ) {
                const int L = 31 - __clz(occ);
                if (lane == L) last = {above, m, (int)n, (int)k16, (int)n, 0};
                last_lane = L;
            }
            cum = ff_add(cum, ff_shfl(mi, 31));
            cc += __shfl_sync(0xFFFFFFFFu, ci, 31);
        }
        if (!done && lane == last_lane) *out = last;   // not reached by the mass: the last value, all of it
    }
    __syncthreads();
}

// Matches of key k16 among the 8 bf16 tokens of a 16-byte word.
__device__ __forceinline__ int key_matches8(uint4 q, uint32_t k16) {
    const uint32_t a[4] = {q.x, q.y, q.z, q.w};
    int m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m += bf16_key16(a[i] & 0xFFFFu) == k16;
        m += bf16_key16(a[i] >> 16) == k16;
    }
    return m;
}

// Id of the pos-th token (1-based, in id order) whose bf16 key is k16, found by the blocks of the
// cluster together: the row is cut into kNucSplit * kWarps stretches, one per warp; each lane
// keeps the match count of every 16-byte word it reads (4 bits each), so the warp whose stretch
// holds the pos-th match finds its word by scanning those counts and reads that word once more.
// Returns the id in block 0 (-1 if the row has fewer matches).
constexpr int kTieWords = 32;   // words per lane kept (stretches up to 1024 words: V <= 262144)

template <class Cluster>
__device__ int bf16_tie_id(Cluster &cl, int rank, const char *row, int V, uint32_t k16, int pos, int *s_wc,
                           int *s_own, int *s_res) {
    constexpr int kStretches = kNucSplit * kWarps;
    constexpr int kDepth = 8;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, g = rank * kWarps + w;
    const int n_vec = (V * 2) / 16;
    const int per = (n_vec + kStretches - 1) / kStretches;
    const int lo = min(n_vec, g * per), hi = min(n_vec, lo + per);
    const int J = (per + 31) / 32;   // words per lane
    const uint4 *rv = reinterpret_cast<const uint4 *>(row);
    const uint16_t *r16 = reinterpret_cast<const uint16_t *>(row);
    uint32_t nib[kTieWords / 8] = {0u, 0u, 0u, 0u};
    int cnt = 0;
    for (int j0 = 0; j0 < J; j0 += kDepth) {
        uint4 q[kDepth];
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
            const int vi = lo + 32 * (j0 + d) + lane;
            q[d] = (j0 + d < J && vi < hi) ? __ldg(rv + vi) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
            const int j = j0 + d, vi = lo + 32 * j + lane;
            const int m = (j < J && vi < hi) ? key_matches8(q[d], k16) : 0;
            cnt += m;
            if (j < kTieWords) {
#pragma unroll
                for (int x = 0; x < kTieWords / 8; ++x)
                    if ((j >> 3) == x) nib[x] |= (uint32_t)m << (4 * (j & 7));
            }
        }
    }
    if (g == kStretches - 1)
        for (int v = n_vec * 8 + lane; v < V; v += 32) cnt += bf16_key16(r16[v]) == k16;
    cnt = (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)cnt);
    if (lane == 0) s_wc[w] = cnt;
    if (threadIdx.x == 0) *s_res = -1;
    cl.sync();
    static_assert(kStretches == 32, "one stretch per lane of warp 0");
    if (threadIdx.x < 32) {   // the stretch that holds the pos-th match: lane l reads stretch l
        const int cx = cl.map_shared_rank(s_wc, lane / kWarps)[lane % kWarps];
        int inc = cx;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int tt = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= o) inc += tt;
        }
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, inc - cx < pos && pos <= inc);
        const int L = hit ? __ffs(hit) - 1 : -1;
        const int L_off = __shfl_sync(0xFFFFFFFFu, inc - cx, L < 0 ? 0 : L);
        if (lane == 0) {
            s_own[0] = L;
            s_own[1] = L_off;
        }
    }
    __syncthreads();
    const int own = s_own[0];
    if (own == g) {
        int need = pos - s_own[1];
        for (int j = 0; j < J && need > 0; ++j) {
            int m;
            if (j < kTieWords) {
                m = (int)((nib[j >> 3] >> (4 * (j & 7))) & 15u);
            } else {
                const int vi = lo + 32 * j + lane;
                m = vi < hi ? key_matches8(__ldg(rv + vi), k16) : 0;
            }
            int inc = m;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int tt = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                if (lane >= o) inc += tt;
            }
            const int tot = __shfl_sync(0xFFFFFFFFu, inc, 31);
            if (tot >= need) {
                if (inc - m < need && inc >= need) {
                    const int vi = lo + 32 * j + lane;
                    const uint4 qq = __ldg(rv + vi);
                    const uint32_t a4[4] = {qq.x, qq.y, qq.z, qq.w};
                    int k = need - (inc - m);
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t bits = (i & 1) ? (a4[i >> 1] >> 16) : (a4[i >> 1] & 0xFFFFu);
                        if (bf16_key16(bits) == k16 && --k == 0) {
                            *s_res = vi * 8 + i;
                            break;
                        }
                    }
                }
                need = 0;
            } else {
                need -= tot;
            }
        }
        if (need > 0 && g == kStretches - 1 && lane == 0)   // the scalar tail
            for (int v = n_vec * 8; v < V; ++v)
                if (bf16_key16(r16[v]) == k16 && --need == 0) {
                    *s_res = v;
                    break;
                }
    }
    cl.sync();
    return (rank == 0 && own >= 0) ? *cl.map_shared_rank(s_res, own / kWarps) : -1;
}

template <int ES>
__global__ void __cluster_dims__(kNucSplit, 1, 1) __launch_bounds__(kThreads, 3) k_nucleus_hist(const NucleusArgs a) {
    pdl_trigger();   // a dependent launch may be scheduled; it waits for this kernel
    static_assert(ES == 2, "value histogram: bf16 rows only");
    namespace cg = cooperative_groups;
    extern __shared__ __align__(16) unsigned s_cnt[];   // kNucKeys counters
    __shared__ float2 tab[256];
    __shared__ int s_segc[kThreads], s_exc[kThreads];
    __shared__ ff s_segm[kThreads], s_exm[kThreads];
    __shared__ NucXch s_x[3];                           // totals, top-k cut, nucleus cut
    __shared__ int s_owner, s_wc[kWarps], s_own[2], s_res;
    __shared__ RowStat s_rs;
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank();
    const long long rid = blockIdx.x / kNucSplit;
    if (rid >= a.n_rows) return;                        // the whole cluster
    const int s = rid < a.n_rows0 ? 0 : 1;
    const long long lr = s == 0 ? rid : rid - a.n_rows0;
    const RowSet &rs = a.set[s];
    const long long b = lr / rs.rows_used, j = lr - b * rs.rows_used;
    const float T = a.temperature[b];
    const float tp = a.top_p ? a.top_p[b] : 1.0f;
    const int tk = a.top_k ? a.top_k[b] : 0;
    const bool p_on = tp < 1.0f;
    const bool k_on = tk > 0 && tk < a.V;
    NucleusCut none;
    none.cut_x = -INFINITY;
    none.cut_id = 0x7FFFFFFF;
    none.mass = 1.0;
    none.log2_mass = 0.0;
    none.ambiguous = 0;
    none.mass_f = 1.0f;
    if (!(p_on || k_on) || !(T >= 1e-3f && T <= 1e3f)) {   // off, greedy or invalid temperature
        if (threadIdx.x == 0 && rank == 0) a.nuc[rid] = none;
        return;
    }
    const char *row = rs.base + (b * rs.rows_per_seq + j) * rs.pitch_bytes;
    if (threadIdx.x < 32) {
        const RowStat st = combine_row(a.part + (size_t)rid * a.n_split * kWarps, a.n_split * kWarps, false, T);
        if (threadIdx.x == 0) s_rs = st;
    }
    tab[threadIdx.x] = kExp2Table[threadIdx.x];
    for (int i = threadIdx.x; i < kNucKeys / 4; i += kThreads) reinterpret_cast<uint4 *>(s_cnt)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    const RowStat st = s_rs;
    if (!rs_sampled_ok(st) || st.flags) {   // reported by the accept / sampling kernels
        if (threadIdx.x == 0 && rank == 0) a.nuc[rid] = none;
        return;
    }
    float c_hi, c_lo;
    log2e_over(T, c_hi, c_lo);
    const ff c = {c_hi, c_lo};
    const int r = st.r;

    // ---- counts per value: every block reads the whole row and counts the tokens whose values
    //      fall in its quarter of the keys (block q: the q-th quarter from the top).  The quarter
    //      of a bf16 value is fixed by its two top bits; -0 and +0 are counted apart here
    //      (adjacent keys of the same mass) and taken together when a cut falls on them. ----
    const uint32_t kbase = (uint32_t)(kNucSplit - 1 - rank) * (uint32_t)kNucKeys;
    {
        // block 0: bits 0x4000-0x7FFF, 1: 0x0000-0x3FFF (non-negative); 2: 0x8000-0xBFFF,
        // 3: 0xC000-0xFFFF (negative, whose keys run opposite to their bits)
        const uint32_t top2 = rank == 0 ? 0x4000u : rank == 1 ? 0x0000u : rank == 2 ? 0x8000u : 0xC000u;
        const uint32_t flip = rank < 2 ? 0u : 0xFFFFu;
        auto add_tok = [&](uint32_t bits) {
            if ((bits & 0xC000u) == top2) atomicAdd(&s_cnt[(bits ^ flip) & (uint32_t)(kNucKeys - 1)], 1u);
        };
        auto add8 = [&](uint4 wd) {
            add_tok(wd.x & 0xFFFFu);
            add_tok(wd.x >> 16);
            add_tok(wd.y & 0xFFFFu);
            add_tok(wd.y >> 16);
            add_tok(wd.z & 0xFFFFu);
            add_tok(wd.z >> 16);
            add_tok(wd.w & 0xFFFFu);
            add_tok(wd.w >> 16);
        };
        const int n_vec = (a.V * 2) / 16;
        const uint4 *rv = reinterpret_cast<const uint4 *>(row);
        constexpr int kDepth = 8;   // loads in flight per thread
        int vi = threadIdx.x;
        for (; vi + (kDepth - 1) * kThreads < n_vec; vi += kDepth * kThreads) {
            uint4 q[kDepth];
#pragma unroll
            for (int d = 0; d < kDepth; ++d) q[d] = __ldg(rv + vi + d * kThreads);
#pragma unroll
            for (int d = 0; d < kDepth; ++d) add8(q[d]);
        }
        for (; vi < n_vec; vi += kThreads) add8(__ldg(rv + vi));
        const uint16_t *r16 = reinterpret_cast<const uint16_t *>(row);
        for (int v = n_vec * 8 + threadIdx.x; v < a.V; v += kThreads) add_tok(r16[v]);
    }
    cl.sync();   // all counts are in

    // ---- segment sums: a segment is kNucBins adjacent keys (segment t of block q: the values
    //      just below key top(t)); the 4 x 256 segments are dealt round-robin to the blocks so
    //      that a dense stretch of values is shared out; two values per lane ----
    {
        const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
        constexpr int kAhead = 4;   // segments whose counters are loaded together
        for (int q0 = 0; q0 < 32; q0 += kAhead) {
            unsigned n0[kAhead], n1[kAhead];
#pragma unroll
            for (int d = 0; d < kAhead; ++d) {
                const int G = kNucSplit * (32 * w + q0 + d) + rank;
                const unsigned *cnt = cl.map_shared_rank(s_cnt, G / kThreads);
                const int top = kNucKeys - 1 - kNucBins * (G % kThreads);
                n0[d] = cnt[top - lane];
                n1[d] = cnt[top - 32 - lane];
            }
#pragma unroll
            for (int d = 0; d < kAhead; ++d) {
                const int G = kNucSplit * (32 * w + q0 + d) + rank;
                const int owner = G / kThreads, seg = G % kThreads;
                const uint32_t kb = (uint32_t)(kNucSplit - 1 - owner) * (uint32_t)kNucKeys;
                const int top = kNucKeys - 1 - kNucBins * seg;
                int *segc = cl.map_shared_rank(s_segc, owner);
                ff *segm = cl.map_shared_rank(s_segm, owner);
                if (!__any_sync(0xFFFFFFFFu, (n0[d] | n1[d]) != 0)) {
                    if (lane == 0) {
                        segc[seg] = 0;
                        segm[seg] = {0.f, 0.f};
                    }
                    continue;
                }
                ff m = {0.f, 0.f};
                if (n0[d]) m = ff_times(key_mass(kb + (uint32_t)(top - lane), c, r, tab), n0[d]);
                if (n1[d]) m = ff_add(m, ff_times(key_mass(kb + (uint32_t)(top - 32 - lane), c, r, tab), n1[d]));
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) m = ff_add(m, ff_shfl_xor(m, o));
                const int nc = (int)__reduce_add_sync(0xFFFFFFFFu, n0[d] + n1[d]);
                if (lane == 0) {
                    segc[seg] = nc;
                    segm[seg] = m;
                }
            }
        }
    }
    cl.sync();
    if (threadIdx.x < 32) {   // exclusive prefixes over the segments, 8 per lane in order
        const int lane = threadIdx.x;
        int lc = 0;
        ff lm = {0.f, 0.f};
        for (int q = 0; q < 8; ++q) {
            lc += s_segc[8 * lane + q];
            lm = ff_add(lm, s_segm[8 * lane + q]);
        }
        int ic = lc;
        ff im = lm;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int tc = __shfl_up_sync(0xFFFFFFFFu, ic, o);
            const ff tm = ff_shfl_up(im, o);
            if (lane >= o) {
                ic += tc;
                im = ff_add(tm, im);
            }
        }
        int ec = ic - lc;
        ff em = ff_shfl_up(im, 1);
        if (lane == 0) em = {0.f, 0.f};
        for (int q = 0; q < 8; ++q) {
            s_exc[8 * lane + q] = ec;
            s_exm[8 * lane + q] = em;
            ec += s_segc[8 * lane + q];
            em = ff_add(em, s_segm[8 * lane + q]);
        }
        if (lane == 31) {
            s_x[0].count = ec;
            s_x[0].mass = em;
        }
    }
    cl.sync();
    // totals of the blocks above this one, and of the row (the same sums in every block)
    int cnt_above[kNucSplit];
    ff m_above[kNucSplit];
    ff S = {0.f, 0.f};
    int C = 0;
    for (int q = 0; q < kNucSplit; ++q) {
        const NucXch *xq = cl.map_shared_rank(&s_x[0], q);
        cnt_above[q] = C;
        m_above[q] = S;
        C += xq->count;
        S = ff_add(S, xq->mass);
    }

    // ---- top-k: the k-th token from the top (exact counts) ----
    int k_rank = 0;
    if (k_on)
        for (int q = 0; q < kNucSplit; ++q)
            if (tk > cnt_above[q]) k_rank = q;
    if (k_on && rank == k_rank)
        locate_cut(false, tk - cnt_above[rank], m_above[rank], {0.f, 0.f}, kbase, s_cnt, s_exc, s_exm, s_segc,
                   s_segm, c, r, tab, &s_owner, &s_x[1]);
    cl.sync();
    // -0 (key 0x7FFF) and +0 (key 0x8000) are one value: a cut on either becomes a cut on +0
    // with the tokens of both, in id order
    const int n_pz = (int)cl.map_shared_rank(s_cnt, 1)[0];
    const int n_nz = (int)cl.map_shared_rank(s_cnt, 2)[kNucKeys - 1];
    auto fold_zero = [&](NucXch &x) {
        if (x.key == 0x7FFF) {
            x.key = 0x8000;
            x.mass = ff_sub(x.mass, ff_times(x.each, (unsigned)n_pz));
            x.pos += n_pz;
            x.count += n_pz;
        } else if (x.key == 0x8000) {
            x.count += n_nz;
        }
    };
    NucXch kc = {};
    if (k_on) {
        kc = *cl.map_shared_rank(&s_x[1], k_rank);
        fold_zero(kc);
    }
    const ff M_k = k_on ? ff_add(kc.mass, ff_times(kc.each, (unsigned)kc.pos)) : S;

    // ---- top-p: the first value where the mass from the top reaches top_p of M_k ----
    const ff target = ff_mul({tp, 0.f}, M_k);
    int p_rank = 0;
    if (p_on)
        for (int q = 1; q < kNucSplit; ++q)
            if (!ff_ge(m_above[q], target)) p_rank = q;
    if (p_on && rank == p_rank)
        locate_cut(true, 0, m_above[rank], target, kbase, s_cnt, s_exc, s_exm, s_segc, s_segm, c, r, tab, &s_owner,
                   &s_x[2]);
    cl.sync();
    NucXch pc = kc;
    if (p_on) {
        pc = *cl.map_shared_rank(&s_x[2], p_rank);
        fold_zero(pc);
        if (k_on && (pc.key < kc.key || (pc.key == kc.key && pc.pos > kc.pos))) pc = kc;   // past the top-k set
    }
    cl.sync();   // every block has read the cuts before any is overwritten
    // the id of the last kept token of the cut's value (all of them kept: no search)
    const int cut_id = pc.pos >= pc.count ? 0x7FFFFFFF
                                          : bf16_tie_id(cl, rank, row, a.V, (uint32_t)pc.key, pc.pos, s_wc, s_own, &s_res);
    cl.sync();   // no block leaves while another may still read its shared memory
    if (rank != 0 || threadIdx.x != 0) return;   // float64 on one thread: this GPU's float64 pipe is narrow

    const double above = ff_to_double(pc.mass), each = ff_to_double(pc.each), Sd = ff_to_double(S);
    const double cum_hi = above + pc.pos * each;
    NucleusCut out;
    out.ambiguous = 0;
    out.cut_x = bf16_key_value((uint32_t)pc.key);
    out.cut_id = cut_id;
    out.mass = cum_hi / Sd;
    out.log2_mass = log2(out.mass);
    out.mass_f = (float)out.mass;
    if (p_on) {
        // each mass carries ~2^-44 and the float-float sums add ~2^-44 per level
        const double tg = ff_to_double(target), cum_lo = above + (pc.pos - 1) * each;
        const double E = 2e-11 * (cum_hi + tg);
        if ((tg - cum_lo) <= E || (cum_hi - tg) <= E) stats_add(a.stats, &a.stats->unresolved, 1);
    }
    a.nuc[rid] = out;
}

template <int ES>
sv_status launch_nucleus(const RowSet &tgt, const RowSet &drf, long long n_rows0, long long n_rows1, int V,
                         const float *temperature, const float *top_p, const int32_t *top_k, const WarpPartial *part,
                         int n_split, NucleusCut *nuc, sv_stats *stats, cudaStream_t stream) {
    NucleusArgs a;
    a.set[0] = tgt;
    a.set[1] = drf;
    a.n_rows0 = n_rows0;
    a.n_rows = n_rows0 + n_rows1;
    a.V = V;
    a.temperature = temperature;
    a.top_p = top_p;
    a.top_k = top_k;
    a.part = part;
    a.n_split = n_split;
    a.nuc = nuc;
    a.stats = stats;
    if (a.n_rows < 1) return SV_OK;
    if constexpr (ES == 2) {
        if (prepare_kernel(reinterpret_cast<const void *>(&k_nucleus_hist<2>), kThreads, kNucHistBytes) < 1)
            return SV_ERR_CUDA;
        k_nucleus_hist<2><<<(unsigned)(kNucSplit * a.n_rows), kThreads, kNucHistBytes, stream>>>(a);
    } else {
        k_nucleus<ES><<<(unsigned)a.n_rows, kThreads, 0, stream>>>(a);
    }
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
    sv_stats *stats;
    int ring_stages;         // stages of each block's bulk-copy ring
};

// Masses of the kept tokens inside and outside D (the elements at or above (xstar, last) in
// (logit desc, id asc) order), by one block over the whole row: (E, A, count) of each side.
template <int ES, class Kept, class Mass>
__device__ void topset_split_block(const char *row, int V, float xstar, int last, Kept kept, Mass mass, double *s_red,
                                   double3 &t_in, double3 &t_out) {
    ff e_in = {0.f, 0.f}, e_out = {0.f, 0.f};
    float a_in = 0.f, a_out = 0.f;
    int n_in = 0, n_out = 0;
    for_strided<ES>(row, V, threadIdx.x, kThreads, [&](float x, int v) {
        if (!kept(x, v)) return;
        float y;
        const float e = mass(x, y);
        if (x > xstar || (x == xstar && v <= last)) {
            e_in = ff_add_f(e_in, e);
            a_in += e * fabsf(y);
            ++n_in;
        } else {
            e_out = ff_add_f(e_out, e);
            a_out += e * fabsf(y);
            ++n_out;
        }
    });
    t_in = block_sum_d3(ff_to_double(e_in), (double)a_in, (double)n_in, s_red);
    t_out = block_sum_d3(ff_to_double(e_out), (double)a_out, (double)n_out, s_red);
}

// One cluster per row.  The pass of the cluster top-N also sums, per block, the masses of the
// kept tokens (float-float per thread); block 0 takes the F-th element, the masses of the first
// F from its list, and the rest as the row total less those (or, when a block's candidates
// overflowed or that difference is too small to trust, one pass of its own over the row).
template <int ES>
__global__ void __launch_bounds__(kThreads) k_topset(const TopSetArgs a) {
    pdl_trigger();   // a dependent launch may be scheduled; it waits for this kernel
    __shared__ TopNCl s;
    extern __shared__ __align__(128) char ring[];
    __shared__ double s_red[3 * kWarps];
    __shared__ RowStat s_rs;
    __shared__ double s_tot[kTopNCluster][4];   // block 0: each block's (E, A, count) of kept tokens
    __shared__ float4 s_fin[kTopNFast / 32];     // block 0: the first N's (E hi, E lo, A, count) per warp
    __shared__ int s_trust;
    const cooperative_groups::cluster_group cl = cooperative_groups::this_cluster();
    const int S = (int)cl.num_blocks(), rank = (int)cl.block_rank();
    const long long lr = blockIdx.x / S;
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
        if (threadIdx.x == 0 && rank == 0) a.top[rid] = none;
        return;
    }
    const char *row = a.rows.base + (b * a.rows.rows_per_seq + j) * a.rows.pitch_bytes;
    if (threadIdx.x < 32) {
        const RowStat st = combine_row(a.part + (size_t)rid * a.n_split * kWarps, a.n_split * kWarps, false, T);
        if (threadIdx.x == 0) s_rs = st;
    }
    __syncthreads();
    const RowStat st = s_rs;
    if (!rs_sampled_ok(st) || st.flags) {   // the same in every block of the cluster
        if (threadIdx.x == 0 && rank == 0) a.top[rid] = none;
        return;
    }
    const int N = min(a.F, a.V);
    float c_hi, c_lo;
    log2e_over(T, c_hi, c_lo);
    const float rf = (float)st.r;
    float cut_x = -INFINITY;
    int cut_id = 0x7FFFFFFF;
    if (a.nuc) {
        cut_x = a.nuc[rid].cut_x;
        cut_id = a.nuc[rid].cut_id;
    }
    // tokens the top-k / top-p filters keep, and their float32 masses 2^y, y = x c - r
    auto kept = [&](float x, int v) { return x != -INFINITY && (x > cut_x || (x == cut_x && v <= cut_id)); };
    auto mass = [&](float x, float &y) {
        y = fmaf(x, c_lo, fmaf(x, c_hi, -rf));
        return ex2_fast(y);
    };
    double3 t_in, t_out;
    float xstar;
    int last;
    bool direct = true;
    double sub_err = 0.0;   // absolute error of an outside mass taken as a difference
    if (N > kTopNFast) {   // a single-block cluster (the launch sees to it): radix select, split pass
        topn_exact_block<ES>(row, a.V, N, false, s);
        xstar = key_value(s.nth_key);
        last = s.nth_id;
        topset_split_block<ES>(row, a.V, xstar, last, kept, mass, s_red, t_in, t_out);
    } else {
        // rows under a top-k / top-p cut sum their kept masses in the pass; the others take the
        // row total S from the statistics pass (the same masses, with a certified bound)
        const bool filtered = a.nuc != nullptr && !(cut_x == -INFINITY && cut_id == 0x7FFFFFFF);
        ff e_t = {0.f, 0.f};
        float a_t = 0.f;
        int n_t = 0;
        auto add_mass = [&](float x, int v) {
            if (!kept(x, v)) return;
            float y;
            const float e = mass(x, y);
            e_t = ff_add_f(e_t, e);
            a_t = fmaf(e, fabsf(y), a_t);
            ++n_t;
        };
        const bool radix = cluster_topn<ES>(
            cl, row, a.V, N, s, ring, a.ring_stages, kWaitLimitCycles,
            [&](uint4 w, int vi) {
                if (!filtered) return;
                float x[16 / ES];
                unpack<ES>(w, x);
#pragma unroll
                for (int k = 0; k < 16 / ES; ++k) add_mass(x[k], vi * (16 / ES) + k);
            },
            [&](float x, int v) {
                if (filtered) add_mass(x, v);
            },
            [&] {
                if (!filtered) return;
                const double3 t = block_sum_d3(ff_to_double(e_t), (double)a_t, (double)n_t, s_red);
                if (threadIdx.x == 0) {
                    double *d = cl.map_shared_rank(&s_tot[0][0], 0) + 4 * rank;
                    d[0] = t.x;
                    d[1] = t.y;
                    d[2] = t.z;
                }
            });
        if (s.fail && threadIdx.x == 0) report_error(a.stats, SV_ERR_TIMEOUT, (int)b);
        if (rank != 0) return;
        if (radix) topn_exact_block<ES>(row, a.V, N, false, s);
        xstar = key_value(s.nth_key);
        last = s.nth_id;
        if (radix) {
            topset_split_block<ES>(row, a.V, xstar, last, kept, mass, s_red, t_in, t_out);
        } else {
            // the first N (N <= kTopNFast: warps 0-3) in float-float, summed by thread 0
            const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
            ff e_i = {0.f, 0.f};
            float a_i = 0.f;
            int n_i = 0;
            if (threadIdx.x < N) {
                const uint64_t c = s.res[threadIdx.x];
                const float x = key_value(code_key(c));
                const int v = code_id(c);
                if (kept(x, v)) {
                    float y;
                    const float e = mass(x, y);
                    e_i.hi = e;
                    a_i = e * fabsf(y);
                    n_i = 1;
                }
            }
            if (warp * 32 < N) {
                e_i = warp_sum_ff(e_i);
                a_i = warp_sum_f(a_i);
                n_i = __reduce_add_sync(0xFFFFFFFFu, n_i);
                if (lane == 0) s_fin[warp] = make_float4(e_i.hi, e_i.lo, a_i, (float)n_i);
            }
            __syncthreads();
            // thread 0 alone forms the totals in float64 (this GPU's float64 pipe is narrow) and
            // tells the block whether the difference can be trusted
            bool trust = true;
            if (threadIdx.x == 0) {
                {
                    ff E = {0.f, 0.f};
                    float A = 0.f, n = 0.f;
                    for (int w = 0; w * 32 < N; ++w) {
                        E = ff_add(E, {s_fin[w].x, s_fin[w].y});
                        A += s_fin[w].z;
                        n += s_fin[w].w;
                    }
                    t_in = make_double3(ff_to_double(E), (double)A, (double)n);
                }
                direct = false;
                if (filtered) {
                    double E = 0.0, A = 0.0, n = 0.0;
                    for (int q = 0; q < S; ++q) {
                        E += s_tot[q][0];
                        A += s_tot[q][1];
                        n += s_tot[q][2];
                    }
                    // E - E_in: the masses of D cancel exactly (the same float32 values on both
                    // sides); each float-float addition errs by at most 2^-47 of its sum, so a
                    // thread's share of n elements leaves at most n 2^-47 E.  A enters the bound only.
                    t_out.x = E - t_in.x;
                    t_out.y = fmax(A - t_in.y, 0.0) + 1e-4 * A;
                    t_out.z = n - t_in.z;
                    if (t_out.z == 0.0) t_out.x = t_out.y = 0.0;   // nothing kept outside D
                    const double r_rel = (double)(a.V / (S * kThreads) + 16) * 0x1p-46;
                    sub_err = r_rel * E;
                    trust = t_out.z == 0.0 || t_out.x > 0x1p17 * sub_err;
                } else {
                    // S - E_in, off by at most err S + r_in E_in; A S bounds the outside sum of e |y|
                    const double Srow = (double)st.s_hi + (double)st.s_lo;
                    const float fin = (float)t_in.x;
                    const double r_in = (double)((float)(kEx2RelErr + 4.0 * kU32) +
                                                 (float)(1.02 * kYRound) * (fin > 0.f ? __fdiv_ru((float)t_in.y, fin) : 0.f)) *
                                        (1.0 + 0x1p-16);
                    t_out.x = Srow - t_in.x;
                    t_out.y = 1.01 * (double)st.ay * Srow + 1e-30;
                    t_out.z = 1.0;   // a positive outside mass (checked below) means a kept token outside D
                    sub_err = (double)st.err * Srow + r_in * t_in.x;
                    trust = t_out.x > 16.0 * sub_err && t_out.x > 0x1p-4 * Srow;
                }
                s_trust = trust ? 1 : 0;
            }
            __syncthreads();
            if (!s_trust) {   // too small to take as a difference: the block sums both sides
                topset_split_block<ES>(row, a.V, xstar, last, kept, mass, s_red, t_in, t_out);
                direct = true;
            }
        }
    }
    if (threadIdx.x != 0) return;
    const double C = (double)a.C, Ein = t_in.x, Eout = t_out.x;
    const double num = C * Ein + Eout, den = Ein + Eout;
    TopSet t = none;
    if (C == 0.0 && t_out.z == 0.0) {
        // every kept token lies in D and C = 0: no transform (the row is used unchanged)
        t.p_d = 1.0;
    } else if (!(num > 0.0)) {
        // the mass left outside D underflows float32: no transform, reported as unresolved
        stats_add(a.stats, &a.stats->unresolved, 1);
    } else {
        t.top_x = xstar;
        t.top_id = last;
        const double inv_den = 1.0 / den;   // the one float64 quotient (this GPU's float64 is slow)
        t.p_d = Ein * inv_den;
        t.z = num * inv_den;
        // The bound, in float32 with every quotient and product rounded up.  Each part is a sum
        // of float32 masses: relative error kEx2RelErr + ln2 u |y| per token (A / E is the
        // mass-weighted mean |y|; the float32 sums of e |y| are within 1% of it) plus rounding;
        // masses that flush to zero below 2^-126 are at most V 2^-126 in all; an outside mass
        // taken as a difference adds its own error sub_err.
        const float fEin = (float)Ein, fEout = (float)Eout, fnum = (float)num, fden = (float)den, fC = a.C;
        const float base = (float)(kEx2RelErr + 4.0 * kU32), ky = (float)(1.02 * kYRound);
        const float r_in = __fmaf_ru(ky, fEin > 0.f ? __fdiv_ru((float)t_in.y, fEin) : 0.f, base);
        float r_out = __fmaf_ru(ky, fEout > 0.f ? __fdiv_ru((float)t_out.y, fEout) : 0.f, base);
        if (!direct) r_out = __fadd_ru(r_out, fEout > 0.f ? __fdiv_ru((float)sub_err, fEout) : INFINITY);
        const float uf = (float)a.V * 0x1p-126f;
        const float e_in = __fmul_ru(fEin, r_in), e_out = __fmaf_ru(fEout, r_out, uf);
        const float rel_num = __fdiv_ru(__fmaf_ru(fC, e_in, e_out), fnum);
        const float rel_den = __fdiv_ru(__fadd_ru(e_in, e_out), fden);
        t.z_err_f = __fmul_ru(__fadd_ru(__fadd_ru(rel_num, rel_den), 1e-12f), 1.0f + 0x1p-16f);
        t.z_err = (double)t.z_err_f;
        t.z_f = (float)t.z;
    }
    a.top[rid] = t;
}

template <int ES>
sv_status launch_topset(const RowSet &drf, long long rid0, int B, int rows_used, int V, const float *temperature,
                        int F, float C, const WarpPartial *part, int n_split, const NucleusCut *nuc, TopSet *top,
                        sv_stats *stats, const DeviceInfo &di, cudaStream_t stream) {
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
    a.stats = stats;
    if (a.n_rows < 1) return SV_OK;
    const int S = F > kTopNFast ? 1 : topn_cluster_size(a.n_rows, di.sms);
    a.ring_stages = topn_ring_stages((int)((long long)V * ES / 16), S);
    const int n_max = F < V ? F : V;
    return cuda_status(launch_row_clusters(k_topset<ES>, a, a.n_rows, S,
                                           topn_dyn_bytes(a.ring_stages, S, n_max > kTopNFast ? 1 : n_max), stream));
}

}  // namespace sv
