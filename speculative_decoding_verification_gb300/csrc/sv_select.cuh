// sv_select.cuh — ranking passes: nucleus (top-p) cuts and Saguaro top-F sets.
#pragma once

#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

template <int ES>
sv_status launch_nucleus(const RowSet &tgt, const RowSet &drf, long long n_rows0, long long n_rows1, int V,
                         const float *temperature, const float *top_p, const WarpPartial *part, int n_split,
                         RowStat *rowstat, NucleusCut *nuc, sv_stats *stats, const DeviceInfo &di,
                         cudaStream_t stream) {
    return SV_ERR_INVALID_ARG;   // not yet available
}

template <int ES>
sv_status launch_topset(const RowSet &drf, long long n_rows0, int B, int K, int V, const float *temperature, int F,
                        float C, const WarpPartial *part, int n_split, const NucleusCut *nuc, TopSet *top,
                        sv_stats *stats, const DeviceInfo &di, cudaStream_t stream) {
    return SV_ERR_INVALID_ARG;   // not yet available
}

}  // namespace sv
