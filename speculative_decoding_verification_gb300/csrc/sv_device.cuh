// sv_device.cuh — device helpers for libspecverify (sm_103a).
//
// Inline PTX for the shared-memory barriers and 1-D bulk (TMA) copies that stage logit rows
// into shared memory, the float32 fast exponential, bfloat16 unpacking, order-preserving
// integer keys, float-float arithmetic for the exact tier, and status reporting.
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "specverify.h"
#include "sv_layout.h"

namespace sv {

// ------------------------------------------------------------------------------------------
// Shared-memory barriers and bulk copies
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes barrier initialisation visible to the asynchronous (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: the thread sleeps until the phase completes or about `ns`
// nanoseconds pass, instead of spinning and taking issue slots from working warps.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Waits for the barrier phase with the given parity; gives up after `limit` SM clock cycles.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, kSuspendHintNs)) return true;
        if (clock64() - t0 > limit) return false;
    }
}

// As mbar_wait_bounded, and also gives up once *abort_flag is set by another warp.  Between
// tries the warp backs off (32 ns doubling to 256 ns), so waiting warps leave the issue slots
// to the warps that have work.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity, const int *abort_flag,
                                                   long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    unsigned ns = 32;
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, kSuspendHintNs)) return true;
        if (*reinterpret_cast<const volatile int *>(abort_flag) || clock64() - t0 > limit) return false;
        __nanosleep(ns);
        ns = ns < 256 ? 2 * ns : 256;
    }
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes` on `bar`.
// Both addresses must be 16-byte aligned and bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 1-D bulk copy with an L2 evict-first policy (streamed logits are read once).
__device__ __forceinline__ void bulk_load_stream(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Programmatic dependent launch.  A kernel launched with launch_pdl may start while the
// previous kernel of the stream is still running; pdl_wait() returns once that kernel has
// completed and its results are visible, so it comes before the first read of them.
// pdl_trigger() lets the next kernel (if launched with launch_pdl) start early; its own
// pdl_wait() still waits for this kernel's completion.  Both are no-ops without a dependent.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <class... Params, class... Args>
inline cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

// ------------------------------------------------------------------------------------------
// Element access
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Packed bf16x2 maximum that propagates NaN.
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Unpack one 16-byte vector of ES-byte elements.
template <int ES>
__device__ __forceinline__ void unpack(uint4 w, float (&x)[16 / ES]) {
    if constexpr (ES == 2) {
        x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
        x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
    } else {
        x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
        x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
    }
}

template <int ES>
__device__ __forceinline__ float load_elem(const char *row, int64_t v) {
    if (ES == 4) return __ldg(reinterpret_cast<const float *>(row) + v);
    const uint16_t h = __ldg(reinterpret_cast<const unsigned short *>(row) + v);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// ------------------------------------------------------------------------------------------
// Exponentials
// ------------------------------------------------------------------------------------------
// Fast tier: the SFU base-2 exponential (denormal results flush to zero).  Its largest
// relative error over the arguments the library feeds it is measured by sv_selftest_exp2 and
// bounded by kEx2RelErr in the certification of float32 decisions.
__device__ __forceinline__ float ex2_fast(float y) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
    return r;
}

// ------------------------------------------------------------------------------------------
// Packed float32 pairs: Blackwell's f32x2 add / multiply-add issue one instruction for two
// IEEE round-to-nearest operations, each rounded exactly as its scalar form.  A pair lives in
// one 64-bit register (lo in the low word).
// ------------------------------------------------------------------------------------------
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_pack(float lo, float hi) {
    f32x2 d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}

__device__ __forceinline__ void f2_unpack(f32x2 v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// The two bfloat16 values of a 32-bit word as a float pair (lo element first), exactly.
__device__ __forceinline__ f32x2 f2_from_bf16x2(uint32_t w) {
    f32x2 d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(w << 16), "r"(w & 0xFFFF0000u));
    return d;
}

__device__ __forceinline__ f32x2 f2_from_u32x2(uint32_t lo, uint32_t hi) {
    f32x2 d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}

__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// 2^y of both lanes with the fast exponential.
__device__ __forceinline__ f32x2 f2_ex2(f32x2 y) {
    float lo, hi;
    f2_unpack(y, lo, hi);
    return f2_pack(ex2_fast(lo), ex2_fast(hi));
}

__device__ __forceinline__ float f2_sum(f32x2 v) {
    float lo, hi;
    f2_unpack(v, lo, hi);
    return __fadd_rn(lo, hi);
}

// Exact power of two for an integer exponent (0 below the normal range).
__device__ __forceinline__ float pow2i(int e) {
    if (e < -126) return 0.0f;
    if (e > 127) e = 127;
    return __int_as_float((e + 127) << 23);
}

// ------------------------------------------------------------------------------------------
// Float-float arithmetic (exact tier).  Each value is hi + lo with |lo| <= ulp(hi)/2.
// The _rn intrinsics keep the compiler from contracting the error-free transforms.
// ------------------------------------------------------------------------------------------
struct ff {
    float hi, lo;
};

__device__ __forceinline__ ff two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}

// Requires |a| >= |b| (or a == 0).
__device__ __forceinline__ ff fast_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ ff two_prod(float a, float b) {
    const float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ ff ff_add(ff a, ff b) {
    ff s = two_sum(a.hi, b.hi);
    const float t = __fadd_rn(__fadd_rn(a.lo, b.lo), s.lo);
    return fast_two_sum(s.hi, t);
}

__device__ __forceinline__ ff ff_sub(ff a, ff b) { return ff_add(a, {-b.hi, -b.lo}); }

__device__ __forceinline__ ff ff_mul(ff a, ff b) {
    ff p = two_prod(a.hi, b.hi);
    p.lo = __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, p.lo));
    return fast_two_sum(p.hi, p.lo);
}

// 1 / a in float-float: a float32 reciprocal refined by one Newton step in float-float.
__device__ __forceinline__ ff ff_recip(ff a) {
    const float r0 = __frcp_rn(a.hi);
    const ff e = ff_sub({1.0f, 0.0f}, ff_mul(a, {r0, 0.0f}));   // 1 - a r0, about 2^-24
    return ff_add({r0, 0.0f}, ff_mul({r0, 0.0f}, e));
}

// a + b for a float b.
__device__ __forceinline__ ff ff_add_f(ff a, float b) {
    const ff s = two_sum(a.hi, b);
    return fast_two_sum(s.hi, __fadd_rn(s.lo, a.lo));
}

// a - b as a float (the float-float difference rounded once): its sign is that of a - b.
__device__ __forceinline__ float ff_diff(ff a, ff b) { return ff_sub(a, b).hi; }

__device__ __forceinline__ double ff_to_double(ff a) { return (double)a.hi + (double)a.lo; }

__device__ __forceinline__ ff ff_from_double(double d) {
    const float h = (float)d;
    return {h, (float)(d - (double)h)};
}

// 2^(yh + yl) as float-float, Tang's table-driven method (P. T. P. Tang, "Table-driven
// implementation of the exponential function in IEEE floating-point arithmetic", ACM TOMS
// 15(2), 1989): y = n + j/256 + r with |r| <= 1/512; 2^(j/256) comes from a 256-entry
// float-float table (tab[j] = {hi, lo}); 2^r = e^s with s = r ln 2 is its Taylor series
// to s^4 (the next term is below 4e-17).  Valid for yh in [-200, 120]; results below 2^-126
// flush to zero.
__device__ __forceinline__ ff ff_exp2(float yh, float yl, const float2 *tab) {
    const float kf = rintf(__fmul_rn(yh, 256.0f));
    const int k = static_cast<int>(kf);
    const float rh = __fsub_rn(yh, __fmul_rn(kf, 0.00390625f));   // exact
    // s = (rh + yl) ln2, float-float; ln2 = L_HI + L_LO
    const float L_HI = 0.693147182464599609375f;
    const float L_LO = -1.9046542999577520e-09f;
    ff s = two_prod(rh, L_HI);
    s.lo = __fmaf_rn(rh, L_LO, __fmaf_rn(yl, L_HI, s.lo));
    s = fast_two_sum(s.hi, s.lo);
    // e^s - 1 = s + s^2/2 + s^3/6 + s^4/24
    const ff s2 = two_prod(s.hi, s.hi);
    const float half_s2 = __fmul_rn(0.5f, s2.hi);
    const float cubic = __fmul_rn(__fmul_rn(s2.hi, s.hi), __fmaf_rn(s.hi, 1.0f / 24.0f, 1.0f / 6.0f));
    const float small = __fadd_rn(__fmaf_rn(s.hi, s.lo, __fmul_rn(0.5f, s2.lo)), cubic);
    ff t = fast_two_sum(s.hi, half_s2);
    t.lo = __fadd_rn(t.lo, __fadd_rn(s.lo, small));
    // 2^(j/256) (1 + t)
    const int j = k & 255;
    const int n = k >> 8;
    const float2 T = tab[j];
    const ff P = two_prod(T.x, t.hi);
    ff e = fast_two_sum(T.x, P.hi);
    const float tail = __fadd_rn(T.y, __fadd_rn(P.lo, __fmaf_rn(T.x, t.lo, __fmul_rn(T.y, t.hi))));
    e = fast_two_sum(e.hi, __fadd_rn(e.lo, tail));
    const float sc = pow2i(n);
    return {__fmul_rn(e.hi, sc), __fmul_rn(e.lo, sc)};
}

// c = log2(e) / T as a float-float pair using float32 operations only (the FP64 pipe is far
// slower than FP32 on this GPU).  The quotient is rounded down, so c_lo >= 0: x * c_hi and
// x * c_lo then share a sign and a -inf logit gives -inf (never inf - inf).  The remainder of
// the quotient is exact, so c_hi + c_lo carries about 46 significant bits.
__device__ __forceinline__ void log2e_over(float T, float &c_hi, float &c_lo) {
    const float L2E_HI = 1.44269502162933349609375f;
    const float L2E_LO = 1.925963033500011e-08f;
    c_hi = __fdiv_rd(L2E_HI, T);
    const float rem = __fadd_rn(__fmaf_rn(-c_hi, T, L2E_HI), L2E_LO);
    c_lo = __fdiv_rn(rem, T);
}

// x * c - g as float-float, with c = c.hi + c.lo and g = g.hi + g.lo float-float constants.
// x * c.hi is exact through an FMA; the remaining terms are small.
__device__ __forceinline__ ff ff_affine(float x, ff c, ff g) {
    const ff p = two_prod(x, c.hi);
    ff d = two_sum(p.hi, -g.hi);
    d.lo = __fadd_rn(d.lo, __fadd_rn(__fsub_rn(p.lo, g.lo), __fmul_rn(x, c.lo)));
    return fast_two_sum(d.hi, d.lo);
}

// 2^(x c - r) in float-float for a float x, a float-float c and an integer r.  The product
// x c_hi is exact through two_prod and x c_lo joins its low word; r joins the exponent after
// the table reduction, so no float-float subtraction is needed.  The low word's rounding is
// about 2^-48 |x c| in the exponent.  Outside |x c_hi| < 2^20 it falls back to ff_affine and
// ff_exp2; results below 2^-126 flush to zero.
__device__ __forceinline__ ff ff_exp2_xc(float x, ff c, int r, const float2 *tab) {
    const ff p = two_prod(x, c.hi);
    if (!(fabsf(p.hi) < 0x1p20f)) {
        const ff y = ff_affine(x, c, {(float)r, 0.f});
        return ff_exp2(y.hi, y.lo, tab);
    }
    if (__fsub_rn(p.hi, (float)r) < -140.0f) return {0.f, 0.f};
    const float yl = __fmaf_rn(x, c.lo, p.lo);
    const float kf = rintf(__fmul_rn(p.hi, 256.0f));
    const int k = static_cast<int>(kf);
    const float rh = __fsub_rn(p.hi, __fmul_rn(kf, 0.00390625f));   // exact
    const float L_HI = 0.693147182464599609375f;
    const float L_LO = -1.9046542999577520e-09f;
    ff s = two_prod(rh, L_HI);
    s.lo = __fmaf_rn(rh, L_LO, __fmaf_rn(yl, L_HI, s.lo));
    s = fast_two_sum(s.hi, s.lo);
    const ff s2 = two_prod(s.hi, s.hi);
    const float half_s2 = __fmul_rn(0.5f, s2.hi);
    const float cubic = __fmul_rn(__fmul_rn(s2.hi, s.hi), __fmaf_rn(s.hi, 1.0f / 24.0f, 1.0f / 6.0f));
    const float small = __fadd_rn(__fmaf_rn(s.hi, s.lo, __fmul_rn(0.5f, s2.lo)), cubic);
    ff t = fast_two_sum(s.hi, half_s2);
    t.lo = __fadd_rn(t.lo, __fadd_rn(s.lo, small));
    const int j = k & 255;
    const int n = (k >> 8) - r;
    const float2 T = tab[j];
    const ff P = two_prod(T.x, t.hi);
    ff e = fast_two_sum(T.x, P.hi);
    const float tail = __fadd_rn(T.y, __fadd_rn(P.lo, __fmaf_rn(T.x, t.lo, __fmul_rn(T.y, t.hi))));
    e = fast_two_sum(e.hi, __fadd_rn(e.lo, tail));
    const float sc = pow2i(n);
    return {__fmul_rn(e.hi, sc), __fmul_rn(e.lo, sc)};
}


// ------------------------------------------------------------------------------------------
// Order-preserving keys (larger value -> larger key) for ranking logits.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t f32_key(float x) {
    uint32_t b = __float_as_uint(x);
    if (b == 0x80000000u) b = 0u;   // -0 ranks with +0: equal logits, ordered by id
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// ------------------------------------------------------------------------------------------
// Status reporting into the caller's sv_stats block.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void report_error(sv_stats *st, int code, int index) {
    if (st == nullptr) return;
    if (atomicCAS(&st->status, 0, code) == 0) atomicExch(&st->error_index, index);
}

__device__ __forceinline__ void stats_add(sv_stats *st, int64_t *field_in_stats, long long v) {
    if (st == nullptr || v == 0) return;
    atomicAdd(reinterpret_cast<unsigned long long *>(field_in_stats), static_cast<unsigned long long>(v));
}

// Queue an item for the float-float tier; past the queue's capacity the float32 result stands
// and the decision is counted as unresolved.
__device__ __forceinline__ void push_exact(Counters *ctr, ExactItem *q, int *unc_n, ExactItem item, sv_stats *st) {
    const int e = atomicAdd(&ctr->n_exact, 1);
    if (e < kExactCap) {
        q[e] = item;
        unc_n[e] = 0;
    } else {
        stats_add(st, &st->unresolved, 1);
    }
}

// ------------------------------------------------------------------------------------------
// Warp helpers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

__device__ __forceinline__ int warp_or_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// (value, index) maximum with ties to the lowest index.
__device__ __forceinline__ void warp_argmax(float &v, int &i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, i, o);
        if (ov > v || (ov == v && oi < i)) {
            v = ov;
            i = oi;
        }
    }
}

__device__ __forceinline__ ff warp_sum_ff(ff a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ff b;
        b.hi = __shfl_xor_sync(0xFFFFFFFFu, a.hi, o);
        b.lo = __shfl_xor_sync(0xFFFFFFFFu, a.lo, o);
        a = ff_add(a, b);
    }
    return a;
}

}  // namespace sv
