// sv_cache.cu — cache lookup (SSD abstract page, "Method") and Mirror-SD branch reuse
// (Mirror-SD notes §3.2).  Integer work only: one thread per sequence.
#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

struct KeyOffsets {
    int off[SV_MAX_K + 2];   // off[k] = sum_{i<k} F_i; off[K+1] = total
};

__global__ void k_cache_lookup(const int32_t *accept_len, const int32_t *out_tokens, const int32_t *keys,
                               KeyOffsets ko, int B, int K, uint8_t *hit) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int k = accept_len[b];
    uint8_t h = 0;
    if (k >= 0 && k <= K) {
        const int t = out_tokens[(size_t)b * (K + 1) + k];
        const int32_t *row = keys + (size_t)b * ko.off[K + 1];
        for (int i = ko.off[k]; i < ko.off[k + 1]; ++i)
            if (row[i] == t && t >= 0) h = 1;
    }
    hit[b] = h;
}

__global__ void k_mirror_reuse(const int32_t *branches, const int32_t *accept_len, const int32_t *out_tokens, int B,
                               int kappa, int gamma, uint8_t *reuse) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int k = accept_len[b];
    uint8_t r = 0;
    if (k >= 0 && k < gamma) {
        const int32_t *pre = out_tokens + (size_t)b * (gamma + 1);
        for (int i = 0; i < kappa && !r; ++i) {
            const int32_t *br = branches + ((size_t)b * kappa + i) * gamma;
            bool same = true;
            for (int j = 0; j <= k && same; ++j) same = (br[j] == pre[j]);
            if (same) r = 1;
        }
    }
    reuse[b] = r;
}

}  // namespace sv

using namespace sv;

extern "C" sv_status sv_cache_lookup(const int32_t *accept_len, const int32_t *out_tokens, const int32_t *keys,
                                     const int32_t *F_int, int B, int K, uint8_t *hit, sv_stream_t stream) {
    if (!accept_len || !out_tokens || !keys || !F_int || !hit || B < 1 || K < 0 || K > SV_MAX_K)
        return SV_ERR_INVALID_ARG;
    KeyOffsets ko;
    long long tot = 0;
    for (int k = 0; k <= K; ++k) {
        if (F_int[k] < 0) return SV_ERR_INVALID_ARG;
        ko.off[k] = (int)tot;
        tot += F_int[k];
        if (tot > (1LL << 30)) return SV_ERR_INVALID_ARG;
    }
    ko.off[K + 1] = (int)tot;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!on_current_device(s, keys, hit)) return SV_ERR_INVALID_ARG;
    k_cache_lookup<<<div_up(B, 256), 256, 0, s>>>(accept_len, out_tokens, keys, ko, B, K, hit);
    return cuda_status(cudaGetLastError());
}

extern "C" sv_status sv_mirror_reuse(const int32_t *branches, const int32_t *accept_len, const int32_t *out_tokens,
                                     int B, int kappa, int gamma, uint8_t *reuse, sv_stream_t stream) {
    if (!branches || !accept_len || !out_tokens || !reuse || B < 1 || kappa < 1 || gamma < 1)
        return SV_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!on_current_device(s, branches, reuse)) return SV_ERR_INVALID_ARG;
    k_mirror_reuse<<<div_up(B, 256), 256, 0, s>>>(branches, accept_len, out_tokens, B, kappa, gamma, reuse);
    return cuda_status(cudaGetLastError());
}
