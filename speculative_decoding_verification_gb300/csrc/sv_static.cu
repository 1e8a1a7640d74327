// sv_static.cu — sv_verify_static: the verification call with its scratch in a fixed device
// array of the library instead of a workspace the caller allocates.
//
// Callers that cannot allocate device memory use it: a serving engine that gives (nearly)
// all free HBM to its KV-cache pool at start-up, where a cudaMalloc in the decode loop would
// fail or shrink that pool, and a host program that loads this library as a plug-in and owns
// every device allocation in its process.  Nothing here allocates: the array is part of the
// loaded module, and each call hands its device address to the ordinary verification path.
#include <mutex>

#include "sv_host.h"

// The scratch array.  In host code this name is only a host-side stand-in for the symbol,
// never a device address: its address on a device comes from cudaGetSymbolAddress, with that
// device current.
static __device__ __align__(256) unsigned char sv_static_scratch[SV_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Set-up, once per device: look up the array's device address with that device current.  The
// address is kept for the life of the process; it does not survive a reset of the device's
// context (cudaDeviceReset), after which the module is loaded again elsewhere.
sv_status scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress((void **)&ptr, sv_static_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return SV_ERR_CUDA;
        }
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return SV_OK;
}

}  // namespace

extern "C" sv_status sv_verify_static(const void *target_logits, int64_t t_row_pitch, const void *draft_logits,
                                      int64_t d_row_pitch, int d_rows_per_seq, sv_dtype dtype,
                                      const int32_t *draft_tokens, const double *uniforms, int B, int K, int V,
                                      const float *temperature, const float *top_p, const int32_t *top_k,
                                      int saguaro_F, float saguaro_C,
                                      int32_t *accept_len, int32_t *out_tokens, double *debug, sv_stats *stats,
                                      sv_stream_t stream) {
    if (B < 1 || K < 0 || K > SV_MAX_K || V < 1) return SV_ERR_INVALID_ARG;
    if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
    // Sizes beyond the array are refused before any device work.
    const sv::VerifyPlan plan = sv::plan_verify(B, K, V, sv::elem_size(dtype));
    if (plan.bytes > SV_STATIC_SCRATCH_BYTES) return SV_ERR_WORKSPACE;
    void *scratch = nullptr;
    const sv_status st = scratch_address(&scratch);
    if (st != SV_OK) return st;
    return sv_verify(target_logits, t_row_pitch, draft_logits, d_row_pitch, d_rows_per_seq, dtype, draft_tokens,
                     uniforms, B, K, V, temperature, top_p, top_k, saguaro_F, saguaro_C, accept_len, out_tokens, debug,
                     stats, scratch, SV_STATIC_SCRATCH_BYTES, stream);
}
