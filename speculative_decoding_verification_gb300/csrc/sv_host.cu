// sv_host.cu — host utilities, sv_fanout (Theorem 12), status strings and device self-tests.
#include <math.h>
#include <mutex>
#include <vector>

#include "sv_device.cuh"
#include "sv_exp2_table.h"
#include <string.h>

#include "sv_host.h"

namespace sv {

namespace {
std::mutex g_mu;
std::vector<DeviceInfo> g_dev;   // indexed by device id
}  // namespace

bool device_info(DeviceInfo &out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if ((int)g_dev.size() <= dev) g_dev.resize(dev + 1);
    DeviceInfo &d = g_dev[dev];
    if (d.device != dev) {
        int sms = 0, smem = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
        if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return false;
        d.device = dev;
        d.sms = sms;
        d.max_smem_optin = smem;
    }
    out = d;
    return true;
}

bool on_current_device(cudaStream_t s, const void *p0, const void *p1) {
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) return false;
    // While the stream is being captured into a graph the queries below would end the capture,
    // so they are skipped; the same call made outside a capture is checked.
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    if (cs != cudaStreamCaptureStatusNone) return true;
    if (s != nullptr && s != cudaStreamLegacy && s != cudaStreamPerThread) {
        int sd = -1;
        if (cudaStreamGetDevice(s, &sd) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        if (sd != cur) return false;
    }
    const void *ps[2] = {p0, p1};
    for (const void *p : ps) {
        if (p == nullptr) continue;
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (at.type == cudaMemoryTypeDevice && at.device != cur) return false;
    }
    return true;
}

namespace {
thread_local cudaEvent_t t_prof_begin = nullptr, t_prof_end = nullptr;
}

void profile_begin(cudaStream_t s) {
    if (t_prof_begin) cudaEventRecord(t_prof_begin, s);
}

void profile_end(cudaStream_t s) {
    if (t_prof_end) cudaEventRecord(t_prof_end, s);
}

int prepare_kernel(const void *func, int threads, size_t smem_bytes) {
    if (smem_bytes > 48 * 1024) {
        if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes) != cudaSuccess)
            return 0;
    }
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, func, threads, smem_bytes) != cudaSuccess) return 0;
    return blocks;
}

// ---- self-tests ---------------------------------------------------------------------------
__global__ void k_selftest_timeout(long long limit, sv_stats *stats) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        // expect 16 bytes that no copy will deliver: the phase never completes
        mbar_arrive_expect_tx(&bar, 16);
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(&bar, 0, limit);
    if (__syncthreads_or(!ok) && threadIdx.x == 0) report_error(stats, SV_ERR_TIMEOUT, -1);
}

__global__ void k_selftest_exp2(double lo, double hi, long long n, unsigned long long *out_bits) {
    __shared__ float2 tab[256];
    {
        tab[threadIdx.x] = kExp2Table[threadIdx.x];
    }
    __syncthreads();
    double e_fast = 0.0, e_ff = 0.0;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const double xd = lo + (hi - lo) * ((double)i / (double)(n > 1 ? n - 1 : 1));
        const float x = (float)xd;
        const double ref = exp2((double)x);
        if (ref > 0x1p-125) {
            const double f = (double)ex2_fast(x);
            e_fast = fmax(e_fast, fabs(f - ref) / ref);
            const ff y = {x, 0.0f};
            const ff e = ff_exp2(y.hi, y.lo, tab);
            e_ff = fmax(e_ff, fabs(ff_to_double(e) - ref) / ref);
            // the exponential with an integer offset folded into the exponent, 2^(x * 1 - r)
            const ff e0 = ff_exp2_xc(x, {1.0f, 0.0f}, 0, tab);
            e_ff = fmax(e_ff, fabs(ff_to_double(e0) - ref) / ref);
            if (x >= -60.0f) {
                const ff e5 = ff_exp2_xc(x, {1.0f, 0.0f}, 5, tab);
                const double ref5 = exp2((double)x - 5.0);
                e_ff = fmax(e_ff, fabs(ff_to_double(e5) - ref5) / ref5);
            }
        }
    }
    // non-negative doubles order like their bit patterns
    atomicMax(&out_bits[0], (unsigned long long)__double_as_longlong(e_fast));
    atomicMax(&out_bits[1], (unsigned long long)__double_as_longlong(e_ff));
}

// Every float32 x with key(lo) <= key(x) <= key(hi), key the order-preserving map of the bit
// patterns that host_order_key computes: the same two errors as k_selftest_exp2, over all
// inputs instead of a sample.  The kernel walks the keys and maps each back to its float.
__device__ __forceinline__ float f32_from_order_key(unsigned k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__global__ void k_selftest_exp2_all(unsigned k0, long long count, unsigned long long *out_bits) {
    __shared__ float2 tab[256];
    {
        tab[threadIdx.x] = kExp2Table[threadIdx.x];
    }
    __syncthreads();
    double e_fast = 0.0, e_ff = 0.0;
    unsigned long long n_eval = 0;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < count;
         i += (long long)gridDim.x * blockDim.x) {
        const float x = f32_from_order_key(k0 + (unsigned)i);
        const double ref = exp2((double)x);
        if (ref > 0x1p-125) {
            const double f = (double)ex2_fast(x);
            e_fast = fmax(e_fast, fabs(f - ref) / ref);
            const ff e = ff_exp2(x, 0.0f, tab);
            e_ff = fmax(e_ff, fabs(ff_to_double(e) - ref) / ref);
            ++n_eval;
        }
    }
    const int lane = threadIdx.x & 31;
    for (int o = 16; o > 0; o >>= 1) {
        e_fast = fmax(e_fast, __shfl_xor_sync(0xFFFFFFFFu, e_fast, o));
        e_ff = fmax(e_ff, __shfl_xor_sync(0xFFFFFFFFu, e_ff, o));
        n_eval += __shfl_xor_sync(0xFFFFFFFFu, n_eval, o);
    }
    if (lane == 0) {
        atomicMax(&out_bits[0], (unsigned long long)__double_as_longlong(e_fast));
        atomicMax(&out_bits[1], (unsigned long long)__double_as_longlong(e_ff));
        atomicAdd(reinterpret_cast<double *>(&out_bits[2]), (double)n_eval);
    }
}

}  // namespace sv

using namespace sv;

static unsigned host_order_key(float x) {
    unsigned b;
    memcpy(&b, &x, sizeof(b));
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

extern "C" sv_status sv_selftest_exp2_all(float lo, float hi, double *out, sv_stream_t stream) {
    if (out == nullptr || !(lo <= hi) || lo < -125.0f || hi > 100.0f) return SV_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!on_current_device(s, out)) return SV_ERR_INVALID_ARG;
    if (cudaMemsetAsync(out, 0, 3 * sizeof(double), s) != cudaSuccess) return SV_ERR_CUDA;
    const unsigned k0 = host_order_key(lo), k1 = host_order_key(hi);
    const long long count = (long long)k1 - (long long)k0 + 1;
    k_selftest_exp2_all<<<4096, 256, 0, s>>>(k0, count, reinterpret_cast<unsigned long long *>(out));
    return cuda_status(cudaGetLastError());
}

extern "C" const char *sv_status_string(sv_status s) {
    switch (s) {
        case SV_OK: return "ok";
        case SV_ERR_INVALID_ARG: return "invalid argument";
        case SV_ERR_CUDA: return "CUDA runtime error";
        case SV_ERR_NONFINITE: return "non-finite logits";
        case SV_ERR_TIMEOUT: return "bounded wait timed out";
        case SV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case SV_ERR_BAD_TOKEN: return "token id outside [0, V)";
    }
    return "unknown status";
}

extern "C" int sv_version(void) { return 100; }   // 0.1.0

extern "C" void sv_set_profile_events(void *begin, void *end) {
    t_prof_begin = static_cast<cudaEvent_t>(begin);
    t_prof_end = static_cast<cudaEvent_t>(end);
}

// Theorem 12 (SSD abstract page, "Method"): F_k = F_0 a^(k/(1+r)) for k < K and
// F_K = F_0 a^(K/(1+r)) (1-a)^(-1/(1+r)), scaled so that the F_k sum to the budget.
extern "C" sv_status sv_fanout(double budget, double a, double r, int K, double *F_real, int32_t *F_int) {
    if (F_real == nullptr || F_int == nullptr) return SV_ERR_INVALID_ARG;
    if (!(a > 0.0 && a < 1.0) || !(r > -1.0) || !(budget >= 0.0) || !(budget < 2147483647.0)) return SV_ERR_INVALID_ARG;
    if (K < 0 || K > SV_MAX_K) return SV_ERR_INVALID_ARG;
    const double e = 1.0 / (1.0 + r);
    double shape[SV_MAX_K + 1];
    double total = 0.0;
    for (int k = 0; k < K; ++k) shape[k] = pow(a, k * e);
    shape[K] = pow(a, K * e) * pow(1.0 - a, -e);
    // sum the smallest terms first
    double sorted[SV_MAX_K + 1];
    for (int k = 0; k <= K; ++k) sorted[k] = shape[k];
    for (int i = 1; i <= K; ++i)
        for (int j = i; j > 0 && sorted[j] < sorted[j - 1]; --j) {
            const double t = sorted[j];
            sorted[j] = sorted[j - 1];
            sorted[j - 1] = t;
        }
    for (int k = 0; k <= K; ++k) total += sorted[k];
    const double f0 = budget / total;
    long long floor_sum = 0;
    double rem[SV_MAX_K + 1];
    for (int k = 0; k <= K; ++k) {
        F_real[k] = f0 * shape[k];
        const double fl = floor(F_real[k]);
        F_int[k] = (int32_t)fl;
        rem[k] = F_real[k] - fl;
        floor_sum += F_int[k];
    }
    long long deficit = (long long)floor(budget) - floor_sum;
    bool used[SV_MAX_K + 1] = {false};
    while (deficit > 0) {
        int best = -1;
        for (int k = 0; k <= K; ++k)
            if (!used[k] && (best < 0 || rem[k] > rem[best])) best = k;
        if (best < 0) break;
        used[best] = true;
        F_int[best] += 1;
        --deficit;
    }
    return SV_OK;
}

extern "C" sv_status sv_selftest_timeout(int64_t limit_cycles, sv_stats *stats, sv_stream_t stream) {
    if (stats == nullptr || limit_cycles < 0) return SV_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!on_current_device(s, stats)) return SV_ERR_INVALID_ARG;
    if (cudaMemsetAsync(stats, 0, sizeof(sv_stats), s) != cudaSuccess) return SV_ERR_CUDA;
    k_selftest_timeout<<<1, 64, 0, s>>>(limit_cycles, stats);
    return cuda_status(cudaGetLastError());
}

extern "C" sv_status sv_selftest_exp2(double lo, double hi, int64_t n, double *out, sv_stream_t stream) {
    if (out == nullptr || n < 1 || !(lo <= hi) || lo < -125.0 || hi > 100.0) return SV_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!on_current_device(s, out)) return SV_ERR_INVALID_ARG;
    if (cudaMemsetAsync(out, 0, 2 * sizeof(double), s) != cudaSuccess) return SV_ERR_CUDA;
    k_selftest_exp2<<<1024, 256, 0, s>>>(lo, hi, n, reinterpret_cast<unsigned long long *>(out));
    return cuda_status(cudaGetLastError());
}
