// sv_hostio.cu — sv_verify on inputs in host memory: the rows the verification reads, and its
// small inputs, are copied into staging buffers carved from the workspace; the verification runs
// there; the committed outputs are copied back.  All on the caller's stream.
#include <cstring>

#include "sv_host.h"

using namespace sv;

namespace {

// Copies the first K rows of every sequence with a nonzero temperature from pinned host memory
// (read through its device mapping) into the staging rows: sequence b's row j goes to staging
// row b * K + j.  16-byte words when both sides allow it, else 4-byte words, else bytes; a
// grid-stride loop over (row, word).  One launch replaces one copy per run of rows.
__global__ void k_gather_rows(const char *__restrict__ src, long long src_seq_bytes, long long src_pitch,
                              const float *__restrict__ temperature, int B, int K, char *__restrict__ dst,
                              long long dst_pitch, long long row_bytes, int wb) {
    const long long words = row_bytes / wb;
    const long long total = (long long)B * K * words;
    const long long G = (long long)gridDim.x * blockDim.x;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += G) {
        const long long r = i / words, w = i - r * words;
        const int s = (int)(r / K), j = (int)(r % K);
        if (temperature[s] == 0.0f) continue;   // a greedy sequence's draft rows are never read
        const char *a = src + s * src_seq_bytes + j * src_pitch + w * wb;
        char *d = dst + ((long long)s * K + j) * dst_pitch + w * wb;
        if (wb == 16) *reinterpret_cast<uint4 *>(d) = *reinterpret_cast<const uint4 *>(a);
        else if (wb == 4) *reinterpret_cast<uint32_t *>(d) = *reinterpret_cast<const uint32_t *>(a);
        else *d = *a;
    }
}

struct HostPlan {
    int64_t pitch;   // staging row pitch in elements (16-byte rows)
    size_t off_t, off_d, off_tok, off_u, off_T, off_tp, off_tk, off_al, off_ot, off_ws, ws_bytes, bytes;
};

HostPlan plan_host(int B, int K, int V, int es) {
    HostPlan h;
    const int epv = 16 / es;
    h.pitch = ((int64_t)V + epv - 1) / epv * epv;
    Carver cv;
    h.off_t = cv.take<char>((size_t)B * (K + 1) * h.pitch * es);
    h.off_d = cv.take<char>((size_t)B * (K > 0 ? K : 1) * h.pitch * es);
    h.off_tok = cv.take<int32_t>((size_t)B * (K > 0 ? K : 1));
    h.off_u = cv.take<double>((size_t)B * (K + 1));
    h.off_T = cv.take<float>((size_t)B);
    h.off_tp = cv.take<float>((size_t)B);
    h.off_tk = cv.take<int32_t>((size_t)B);
    h.off_al = cv.take<int32_t>((size_t)B);
    h.off_ot = cv.take<int32_t>((size_t)B * (K + 1));
    h.ws_bytes = sv_verify_workspace_size(B, K, V);
    h.off_ws = cv.take<char>(h.ws_bytes);
    h.bytes = cv.off + 256;
    return h;
}

}  // namespace

extern "C" size_t sv_verify_host_workspace_size(int B, int K, int V, sv_dtype dtype) {
    if (B < 1 || K < 0 || K > SV_MAX_K || V < 1 || (dtype != SV_F32 && dtype != SV_BF16)) return 0;
    return plan_host(B, K, V, elem_size(dtype)).bytes;
}

extern "C" sv_status sv_verify_host(const void *target_logits, int64_t t_row_pitch, const void *draft_logits,
                                    int64_t d_row_pitch, int d_rows_per_seq, sv_dtype dtype,
                                    const int32_t *draft_tokens, const double *uniforms, int B, int K, int V,
                                    const float *temperature, const float *top_p, const int32_t *top_k, int saguaro_F,
                                    float saguaro_C, int32_t *accept_len, int32_t *out_tokens, sv_stats *stats,
                                    void *workspace, size_t workspace_bytes, size_t *h2d_bytes,
                                    sv_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (B < 1 || K < 0 || K > SV_MAX_K || V < 1 || (dtype != SV_F32 && dtype != SV_BF16)) return SV_ERR_INVALID_ARG;
    if (target_logits == nullptr || t_row_pitch < V || uniforms == nullptr || temperature == nullptr ||
        accept_len == nullptr || out_tokens == nullptr)
        return SV_ERR_INVALID_ARG;
    if (K > 0 && (draft_logits == nullptr || draft_tokens == nullptr || d_row_pitch < V || d_rows_per_seq < K))
        return SV_ERR_INVALID_ARG;
    const int es = elem_size(dtype);
    const HostPlan h = plan_host(B, K, V, es);
    if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < h.bytes) return SV_ERR_WORKSPACE;
    if (!on_current_device(stream, workspace)) return SV_ERR_INVALID_ARG;
    char *w = static_cast<char *>(workspace);
    const size_t row_bytes = (size_t)V * es, dst_pitch = (size_t)h.pitch * es;
    size_t moved = 0;
    auto copy_rows = [&](char *dst, const char *src, size_t src_pitch, size_t rows) {
        moved += rows * row_bytes;
        return cudaMemcpy2DAsync(dst, dst_pitch, src, src_pitch, row_bytes, rows, cudaMemcpyHostToDevice, stream) ==
               cudaSuccess;
    };
    auto copy = [&](size_t off, const void *src, size_t bytes) {
        moved += bytes;
        return cudaMemcpyAsync(w + off, src, bytes, cudaMemcpyHostToDevice, stream) == cudaSuccess;
    };
    // the temperatures first: the draft gather below reads them on the device
    if (!copy(h.off_T, temperature, (size_t)B * sizeof(float))) return SV_ERR_CUDA;
    // every target row
    if (!copy_rows(w + h.off_t, static_cast<const char *>(target_logits), (size_t)t_row_pitch * es,
                   (size_t)B * (K + 1)))
        return SV_ERR_CUDA;
    // draft rows j < K of the sampled sequences: from pinned memory one gather launch, else one
    // copy per run of consecutive sequences (one per sequence when the host rows hold more than
    // K rows per sequence)
    if (K > 0) {
        const char *drf = static_cast<const char *>(draft_logits);
        const size_t spitch = (size_t)d_row_pitch * es;
        cudaPointerAttributes pa;
        const bool pinned = cudaPointerGetAttributes(&pa, drf) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
                            pa.devicePointer != nullptr;
        cudaGetLastError();   // a pageable pointer leaves no error behind
        int n_seq = 0;
        for (int b = 0; b < B; ++b) n_seq += temperature[b] != 0.0f ? 1 : 0;
        if (pinned && n_seq > 0) {
            DeviceInfo di;
            if (!device_info(di)) return SV_ERR_CUDA;
            const char *src = static_cast<const char *>(pa.devicePointer);
            const uintptr_t al = (uintptr_t)src | (uintptr_t)spitch | (uintptr_t)row_bytes | (uintptr_t)dst_pitch;
            const int wb = (al % 16 == 0) ? 16 : (al % 4 == 0) ? 4 : 1;
            k_gather_rows<<<(unsigned)(di.sms * 8), 256, 0, stream>>>(
                src, (long long)d_rows_per_seq * spitch, (long long)spitch,
                reinterpret_cast<const float *>(w + h.off_T), B, K, w + h.off_d, (long long)dst_pitch,
                (long long)row_bytes, wb);
            if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
            moved += (size_t)n_seq * K * row_bytes;
        }
        for (int b0 = 0; b0 < B && !pinned;) {
            if (temperature[b0] == 0.0f) {
                ++b0;
                continue;
            }
            int b1 = b0 + 1;
            if (d_rows_per_seq == K)
                while (b1 < B && temperature[b1] != 0.0f) ++b1;
            if (!copy_rows(w + h.off_d + (size_t)b0 * K * dst_pitch, drf + (size_t)b0 * d_rows_per_seq * spitch, spitch,
                           (size_t)(b1 - b0) * K))
                return SV_ERR_CUDA;
            b0 = b1;
        }
        if (!copy(h.off_tok, draft_tokens, (size_t)B * K * sizeof(int32_t))) return SV_ERR_CUDA;
    }
    if (!copy(h.off_u, uniforms, (size_t)B * (K + 1) * sizeof(double))) return SV_ERR_CUDA;
    if (top_p && !copy(h.off_tp, top_p, (size_t)B * sizeof(float))) return SV_ERR_CUDA;
    if (top_k && !copy(h.off_tk, top_k, (size_t)B * sizeof(int32_t))) return SV_ERR_CUDA;
    if (h2d_bytes) *h2d_bytes = moved;
    const sv_status st = verify_entry(
        w + h.off_t, h.pitch, K > 0 ? w + h.off_d : nullptr, h.pitch, K > 0 ? K : 1, dtype,
        K > 0 ? reinterpret_cast<const int32_t *>(w + h.off_tok) : nullptr, reinterpret_cast<const double *>(w + h.off_u),
        B, K, V, reinterpret_cast<const float *>(w + h.off_T), top_p ? reinterpret_cast<const float *>(w + h.off_tp) : nullptr,
        top_k ? reinterpret_cast<const int32_t *>(w + h.off_tk) : nullptr, saguaro_F, saguaro_C, 0,
        reinterpret_cast<int32_t *>(w + h.off_al), reinterpret_cast<int32_t *>(w + h.off_ot), nullptr, stats,
        w + h.off_ws, h.ws_bytes, stream);
    if (st != SV_OK) return st;
    if (cudaMemcpyAsync(accept_len, w + h.off_al, (size_t)B * sizeof(int32_t), cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaMemcpyAsync(out_tokens, w + h.off_ot, (size_t)B * (K + 1) * sizeof(int32_t), cudaMemcpyDeviceToHost,
                        stream) != cudaSuccess)
        return SV_ERR_CUDA;
    return SV_OK;
}
