// sv_rank.cu — entry points built on ranking passes: the speculation cache keys and top-kappa rows.
//
// sv_cache_keys  [SSD notes §5.1]: at depth k < K the cache guesses the bonus token among the
//                top-F_k draft tokens of the row that proposed s_{k+1}, leaving s_{k+1} out (it
//                was sent for verification, so it cannot be the bonus token); at depth K among
//                the top-F_K tokens of the draft row at position K+1.
// sv_topk_rows   [Mirror-SD notes §3.1]: the early-exit head's top-kappa tokens and their
//                log-probabilities become the branch roots sent to the draft.
#include "sv_device.cuh"
#include "sv_host.h"
#include "sv_select.cuh"
#include "sv_stats.cuh"

namespace sv {

struct KeysArgs {
    const int32_t *list;     // [B][K+1][stride] sorted top lists
    int stride;
    const int32_t *tokens;   // [B][K]
    int B, K, V;
    int F[SV_MAX_K + 1];
    int off[SV_MAX_K + 2];
    int32_t *keys;           // [B][off[K+1]]
    sv_stats *stats;
};

// One thread per (sequence, depth).
__global__ void k_keys_finish(const KeysArgs a) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= a.B * (a.K + 1)) return;
    const int b = t / (a.K + 1), k = t - b * (a.K + 1);
    const int Fk = a.F[k];
    int32_t *out = a.keys + (size_t)b * a.off[a.K + 1] + a.off[k];
    const int32_t *lst = a.list + ((size_t)b * (a.K + 1) + k) * a.stride;
    int excl = -1;
    if (k < a.K) {
        excl = a.tokens[(size_t)b * a.K + k];
        if (excl < 0 || excl >= a.V) {
            report_error(a.stats, SV_ERR_BAD_TOKEN, b);
            for (int i = 0; i < Fk; ++i) out[i] = -1;
            return;
        }
    }
    const int n = k < a.K ? Fk + 1 : Fk;
    int w = 0;
    for (int i = 0; i < n && w < Fk; ++i) {
        const int id = lst[i];
        if (id != excl) out[w++] = id;
    }
    for (; w < Fk; ++w) out[w] = -1;
}

struct TopKArgs {
    const int32_t *list;
    const float *list_x;
    int stride, kappa;
    long long n_rows;
    const float *temperature;
    const WarpPartial *part;
    int n_split;
    int32_t *ids;
    double *logprobs;
    sv_stats *stats;
};

// One warp per row: normaliser from the statistics pass, then log p = x/T - LSE.
__global__ void __launch_bounds__(kThreads) k_topk_finish(const TopKArgs a) {
    const long long r = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= a.n_rows) return;
    const float T = a.temperature ? a.temperature[r] : 1.0f;
    if (!(T >= 1e-3f && T <= 1e3f)) {
        if (lane == 0) report_error(a.stats, SV_ERR_INVALID_ARG, (int)r);
        for (int i = lane; i < a.kappa; i += 32) {
            a.ids[r * a.kappa + i] = -1;
            if (a.logprobs) a.logprobs[r * a.kappa + i] = NAN;
        }
        return;
    }
    const RowStat st = combine_row(a.part + (size_t)r * a.n_split * kWarps, a.n_split * kWarps, false, T);
    double lse = 0.0;
    int bad = 0;
    if (lane == 0) {
        bad = st.flags != 0 || !rs_sampled_ok(st);
        lse = bad ? 0.0 : rs_g(st) * kLn2;
        if (bad) report_error(a.stats, SV_ERR_NONFINITE, (int)r);
        else stats_add(a.stats, &a.stats->rows, 1);
    }
    lse = __shfl_sync(0xFFFFFFFFu, lse, 0);
    bad = __shfl_sync(0xFFFFFFFFu, bad, 0);
    for (int i = lane; i < a.kappa; i += 32) {
        a.ids[r * a.kappa + i] = bad ? -1 : a.list[r * a.stride + i];
        if (a.logprobs) a.logprobs[r * a.kappa + i] = bad ? NAN : (double)a.list_x[r * a.stride + i] / (double)T - lse;
    }
}

}  // namespace sv

using namespace sv;

static size_t keys_ws(int B, int K, int stride) {
    Carver cv;
    cv.take<int32_t>((size_t)B * (K + 1) * stride);
    return cv.off + 256;
}

extern "C" size_t sv_cache_keys_workspace_size(int B, int K, int V) {
    if (B < 1 || K < 0 || K > SV_MAX_K || V < 1) return 0;
    return keys_ws(B, K, V < kMaxTopN ? V : kMaxTopN);
}

extern "C" sv_status sv_cache_keys(const void *draft_logits, int64_t row_pitch, int rows_per_seq, sv_dtype dtype,
                                   const int32_t *draft_tokens, const int32_t *F_int, int B, int K, int V,
                                   int32_t *keys, sv_stats *stats, void *workspace, size_t workspace_bytes,
                                   sv_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (B < 1 || K < 0 || K > SV_MAX_K || V < 1 || rows_per_seq < K + 1) return SV_ERR_INVALID_ARG;
    if (!rows_ok(draft_logits, row_pitch, V, dtype) || F_int == nullptr || keys == nullptr) return SV_ERR_INVALID_ARG;
    if (K > 0 && draft_tokens == nullptr) return SV_ERR_INVALID_ARG;
    TopNArgs ta{};
    KeysArgs ka{};
    long long tot = 0;
    int stride = 1;
    for (int k = 0; k <= K; ++k) {
        const int f = F_int[k];
        if (f < 0 || (k < K && f > V - 1) || f > V) return SV_ERR_INVALID_ARG;
        const int n = k < K ? f + 1 : f;
        if (n > kMaxTopN) return SV_ERR_INVALID_ARG;
        ta.n_of_j[k] = n;
        ka.F[k] = f;
        ka.off[k] = (int)tot;
        tot += f;
        if (n > stride) stride = n;
    }
    if (tot > (1LL << 30)) return SV_ERR_INVALID_ARG;
    ka.off[K + 1] = (int)tot;
    const int es = elem_size(dtype);
    const size_t need = keys_ws(B, K, stride);
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need) return SV_ERR_WORKSPACE;
    if (!on_current_device(stream, draft_logits, keys)) return SV_ERR_INVALID_ARG;
    if (stats && cudaMemsetAsync(stats, 0, sizeof(sv_stats), stream) != cudaSuccess) return SV_ERR_CUDA;
    int32_t *list = static_cast<int32_t *>(workspace);
    ta.base = static_cast<const char *>(draft_logits);
    ta.pitch_bytes = row_pitch * es;
    ta.rows_per_seq = rows_per_seq;
    ta.rows_used = K + 1;
    ta.n_rows = (long long)B * (K + 1);
    ta.V = V;
    ta.n_all = 0;
    ta.list = list;
    ta.list_x = nullptr;
    ta.list_stride = stride;
    ta.stats = stats;
    DeviceInfo di;
    if (!device_info(di)) return SV_ERR_CUDA;
    if ((es == 4 ? launch_topn<4>(ta, stride, di.sms, stream) : launch_topn<2>(ta, stride, di.sms, stream)) !=
        cudaSuccess)
        return SV_ERR_CUDA;
    ka.list = list;
    ka.stride = stride;
    ka.tokens = draft_tokens;
    ka.B = B;
    ka.K = K;
    ka.V = V;
    ka.keys = keys;
    ka.stats = stats;
    k_keys_finish<<<div_up((long long)B * (K + 1), 256), 256, 0, stream>>>(ka);
    return cuda_status(cudaGetLastError());
}

struct TopKPlan {
    VerifyPlan v;
    size_t off_list = 0, off_list_x = 0, bytes = 0;
};

static TopKPlan plan_topk(int n_rows, int V, int es, int stride) {
    TopKPlan tp;
    VerifyPlan &p = tp.v;
    p.es = es;
    p.n_rows0 = n_rows;
    p.n_split = choose_split(n_rows, (long long)V * es);
    p.n_vec = vec_count(V, es);
    chunk_geometry(p.n_vec, p.n_split, p.chunk_vecs);
    Carver cv;
    p.off_counters = cv.take<Counters>(1);
    p.off_part = cv.take<WarpPartial>((size_t)n_rows * p.n_split * kWarps);
    tp.off_list = cv.take<int32_t>((size_t)n_rows * stride);
    tp.off_list_x = cv.take<float>((size_t)n_rows * stride);
    tp.bytes = cv.off + 256;
    return tp;
}

extern "C" size_t sv_topk_rows_workspace_size(int n_rows, int V) {
    if (n_rows < 1 || V < 1) return 0;
    const int stride = V < kMaxTopN ? V : kMaxTopN;
    const TopKPlan a = plan_topk(n_rows, V, 4, stride), b = plan_topk(n_rows, V, 2, stride);
    return a.bytes > b.bytes ? a.bytes : b.bytes;
}

extern "C" sv_status sv_topk_rows(const void *logits, int64_t row_pitch, sv_dtype dtype, int n_rows, int V, int kappa,
                                  const float *temperature, int32_t *ids, double *logprobs, sv_stats *stats,
                                  void *workspace, size_t workspace_bytes, sv_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (n_rows < 1 || V < 1 || kappa < 1 || kappa > V || kappa > kMaxTopN) return SV_ERR_INVALID_ARG;
    if (!rows_ok(logits, row_pitch, V, dtype) || ids == nullptr) return SV_ERR_INVALID_ARG;
    const int es = elem_size(dtype);
    const TopKPlan tp = plan_topk(n_rows, V, es, kappa);
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < tp.bytes) return SV_ERR_WORKSPACE;
    if (!on_current_device(stream, logits, ids)) return SV_ERR_INVALID_ARG;
    DeviceInfo di;
    if (!device_info(di)) return SV_ERR_CUDA;
    if (stats && cudaMemsetAsync(stats, 0, sizeof(sv_stats), stream) != cudaSuccess) return SV_ERR_CUDA;
    char *w = static_cast<char *>(workspace);
    const VerifyPlan &pl = tp.v;
    StatsArgs sa{};
    sa.set[0] = {static_cast<const char *>(logits), row_pitch * es, 1, 1, 0};
    sa.set[1] = sa.set[0];
    sa.n_sets = 1;
    sa.V = V;
    sa.temperature = temperature;
    sa.n_split = pl.n_split;
    sa.chunk_vecs = pl.chunk_vecs;
    sa.n_rows0 = n_rows;
    sa.n_units = (long long)n_rows * pl.n_split;
    sa.part = reinterpret_cast<WarpPartial *>(w + pl.off_part);
    sa.counters = reinterpret_cast<Counters *>(w + pl.off_counters);
    sa.stats = stats;
    sa.wait_limit = kWaitLimitCycles;
    {
        const sv_status st = es == 4 ? launch_stats<4>(sa, di, stream) : launch_stats<2>(sa, di, stream);
        if (st != SV_OK) return st;
    }
    TopNArgs ta{};
    ta.base = static_cast<const char *>(logits);
    ta.pitch_bytes = row_pitch * es;
    ta.rows_per_seq = 1;
    ta.rows_used = 1;
    ta.n_rows = n_rows;
    ta.V = V;
    ta.n_all = kappa;
    ta.list = reinterpret_cast<int32_t *>(w + tp.off_list);
    ta.list_x = reinterpret_cast<float *>(w + tp.off_list_x);
    ta.list_stride = kappa;
    ta.stats = stats;
    if ((es == 4 ? launch_topn<4>(ta, kappa, di.sms, stream) : launch_topn<2>(ta, kappa, di.sms, stream)) !=
        cudaSuccess)
        return SV_ERR_CUDA;
    TopKArgs ka{};
    ka.list = ta.list;
    ka.list_x = ta.list_x;
    ka.stride = kappa;
    ka.kappa = kappa;
    ka.n_rows = n_rows;
    ka.temperature = temperature;
    ka.part = sa.part;
    ka.n_split = pl.n_split;
    ka.ids = ids;
    ka.logprobs = logprobs;
    ka.stats = stats;
    k_topk_finish<<<(unsigned)div_up((long long)n_rows * 32, kThreads), kThreads, 0, stream>>>(ka);
    return cuda_status(cudaGetLastError());
}
