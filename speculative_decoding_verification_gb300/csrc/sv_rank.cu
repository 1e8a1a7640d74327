// sv_rank.cu — entry points built on ranking passes (top-F / top-kappa selection).
#include "sv_device.cuh"
#include "sv_host.h"

using namespace sv;

extern "C" size_t sv_cache_keys_workspace_size(int B, int K, int V) { return 256; }

extern "C" sv_status sv_cache_keys(const void *, int64_t, int, sv_dtype, const int32_t *, const int32_t *, int, int,
                                   int, int32_t *, sv_stats *, void *, size_t, sv_stream_t) {
    return SV_ERR_INVALID_ARG;
}

extern "C" size_t sv_topk_rows_workspace_size(int n_rows, int V) { return 256; }

extern "C" sv_status sv_topk_rows(const void *, int64_t, sv_dtype, int, int, int, const float *, int32_t *, double *,
                                  sv_stats *, void *, size_t, sv_stream_t) {
    return SV_ERR_INVALID_ARG;
}
