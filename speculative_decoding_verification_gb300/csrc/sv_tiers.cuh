// sv_tiers.cuh — the draw pass and the float-float tier after an accept kernel: every
// verification entry point ends with these two launches over the draw items it queued.
#pragma once

#include "sv_accept.cuh"
#include "sv_draw.cuh"
#include "sv_exact.cuh"
#include "sv_host.h"

namespace sv {

template <int ES>
sv_status launch_draw_tiers(const VerifyPlan &pl, const AcceptArgs &acc, const NucleusCut *nuc, const TopSet *top,
                            char *w, int B, const DeviceInfo &di, cudaStream_t stream) {
    Counters *counters = reinterpret_cast<Counters *>(w + pl.off_counters);
    const long long wait = kWaitLimitCycles;
    // draws
    DrawArgs da;
    da.items = acc.draws;
    da.counters = counters;
    da.V = acc.V;
    da.n_vec = pl.n_vec;
    da.n_sub = pl.n_sub;
    da.n_split = pl.d_split;
    da.subs_per_chunk = pl.d_subs_per_chunk;
    da.subs = reinterpret_cast<float *>(w + pl.off_subs);
    da.exact = acc.exact;
    da.exact_unc = acc.exact_unc;
    da.stats = acc.stats;
    da.wait_limit = wait;
    {
        const sv_status st = launch_draws<ES>(da, (long long)B, di, stream);
        if (st != SV_OK) return st;
    }
    // float-float tier
    ExactArgs xa;
    xa.tgt = acc.tgt;
    xa.drf = acc.drf;
    xa.K = acc.K;
    xa.V = acc.V;
    xa.temperature = acc.temperature;
    xa.tokens = acc.tokens;
    xa.uniforms = acc.uniforms;
    xa.accept_len = acc.accept_len;
    xa.out_tokens = acc.out_tokens;
    xa.debug = acc.debug;
    xa.sag_C = acc.sag_C;
    xa.sag_on = acc.sag_on;
    xa.nuc = nuc;
    xa.top = top;
    xa.rowstat = acc.rowstat;
    xa.n_rows0 = pl.n_rows0;
    xa.draws = acc.draws;
    xa.items = acc.exact;
    xa.counters = counters;
    xa.xpart = reinterpret_cast<double *>(w + pl.off_xpart);
    xa.xdraw = reinterpret_cast<ExactDraw *>(w + pl.off_xdraw);
    xa.xsubs = reinterpret_cast<float4 *>(w + pl.off_xsubs);
    xa.xnorm = reinterpret_cast<float4 *>(w + pl.off_xnorm);
    xa.xunc_n = reinterpret_cast<int *>(w + pl.off_xunc_n);
    xa.xunc = reinterpret_cast<int *>(w + pl.off_xunc);
    xa.n_vec = pl.n_vec;
    xa.n_sub = pl.n_sub;
    xa.xsplit = pl.x_split;
    xa.max_slots = 2 * acc.K + 1 > 2 ? 2 * acc.K + 1 : 2;
    xa.stats = acc.stats;
    xa.wait_limit = wait;
    xa.draw_from_q = acc.draw_from_q;
    return launch_exact<ES>(xa, di, stream);
}

}  // namespace sv
