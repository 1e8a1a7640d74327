// sv_host.h — host-side helpers shared by the entry points: argument checks, device facts,
// launch wrappers and the workspace carving of each call.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "specverify.h"
#include "sv_layout.h"

namespace sv {

struct DeviceInfo {
    int device = -1;
    int sms = 0;
    int max_smem_optin = 0;
};

// Facts about the current device (cached per device id).  Returns false on a CUDA error.
bool device_info(DeviceInfo &out);

// Thread-local profiling events (sv_set_profile_events) around the statistics pass.
void profile_begin(cudaStream_t s);
void profile_end(cudaStream_t s);

// Opt a kernel into `bytes` of dynamic shared memory and return its resident blocks per SM.
int prepare_kernel(const void *func, int threads, size_t smem_bytes);

inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

inline int elem_size(sv_dtype d) { return d == SV_F32 ? 4 : 2; }

// Checks common to every call that streams logit rows.
inline bool rows_ok(const void *base, int64_t pitch, int V, sv_dtype dtype) {
    if (base == nullptr || V < 1 || pitch < V) return false;
    if (dtype != SV_F32 && dtype != SV_BF16) return false;
    const int es = elem_size(dtype);
    if (!aligned(base, 16)) return false;
    if (((int64_t)pitch * es) % 16 != 0) return false;
    return true;
}

// The call's stream and the device arrays p0, p1 (either may be null) belong to the current
// device.  A stream of another device would run the kernels there while the workspace plan and
// the SM count come from the current one, and an array on another device would be read without
// peer access.  Host and managed memory pass.  One stream query and two pointer queries, none
// while the stream is being captured into a CUDA graph (they would end the capture).
bool on_current_device(cudaStream_t s, const void *p0, const void *p1 = nullptr);

inline sv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SV_OK : SV_ERR_CUDA; }

// ---- the verification pipeline (shared by sv_verify and its variants) --------------------
struct VerifyPlan {
    int es = 2;
    long long n_rows0 = 0, n_rows1 = 0;   // candidate target / draft rows
    int n_split = 1, chunk_vecs = 1;       // statistics pass
    int n_vec = 0, n_sub = 0;              // draw pass geometry
    int d_split = 1, d_subs_per_chunk = 1;
    // workspace offsets
    size_t off_part = 0, off_rowstat = 0, off_draws = 0, off_subs = 0, off_exact = 0, off_counters = 0;
    size_t off_nuc = 0, off_top = 0;
    size_t off_xpart = 0, off_xdraw = 0, off_xsubs = 0, off_xnorm = 0, off_xunc_n = 0, off_xunc = 0;
    int x_split = 1;                       // chunks per row in the float-float pass
    size_t off_lz_units = 0, off_lz_pos = 0;   // lazy verification queue
    long long lz_cap = 0;                  // queue capacity: every (row, chunk) unit once
    int dv_chunks = 1, dv_words = 1;       // fuzzy verification: chunks per row pair, words per chunk
    size_t off_dpart = 0, off_ditem = 0, off_dq = 0, off_deferred = 0;
    size_t off_dxa = 0, off_dxb = 0, off_dxcnt = 0;   // float-float divergences: per (queued pair, chunk)
    int dx_cap = 1;                        // (pair, chunk) entries of off_dxa / off_dxb
    size_t bytes = 0;
};

VerifyPlan plan_verify(int B, int K, int V, int es);

// The sv_verify pipeline; draw_from_q = 1 replaces the residual draw after a rejection by a draw
// from the target row itself (the assisted acceptance of three-model speculative decoding).
sv_status verify_entry(const void *target_logits, int64_t t_row_pitch, const void *draft_logits, int64_t d_row_pitch,
                       int d_rows_per_seq, sv_dtype dtype, const int32_t *draft_tokens, const double *uniforms, int B,
                       int K, int V, const float *temperature, const float *top_p, const int32_t *top_k, int saguaro_F,
                       float saguaro_C, int draw_from_q, int32_t *accept_len, int32_t *out_tokens, double *debug,
                       sv_stats *stats, void *workspace, size_t workspace_bytes, cudaStream_t stream);

}  // namespace sv
