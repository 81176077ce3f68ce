// attn.cu -- picks the kernels of the forward and backward attention passes
// and sets up their arguments.
#include "attn.h"

namespace llsa {

size_t fwd_workspace_bytes(const Shape& s) {
    return fwd_grp_supported(s) && !s.raster ? group_workspace_bytes(s) : 0;
}

int launch_fwd(const Shape& s, const void* q, const void* k, const void* v, const float* pyr,
               const int32_t* sel_idx, const int32_t* coarse_idx, void* o, float* lse, void* ws, cudaStream_t st) {
    AttnArgs a = make_attn_args(s);
    a.q = q; a.k = k; a.v = v;
    a.kpyr = pyr + s.slices * a.pyr_stride;
    a.vpyr = pyr + 2 * s.slices * a.pyr_stride;
    a.sel = sel_idx; a.coarse = coarse_idx; a.out_o = o; a.lse = lse;
    // raster-order tokens: the per-query-block tensor-core forward only
    if (s.raster) return fwd_tc_supported(s) ? launch_fwd_tc(s, a, st) : LLSA_ERR_UNSUPPORTED;
    if (fwd_grp_supported(s)) {
        int32_t *order, *gdesc, *ngroups;
        GroupRec* recs;
        carve_group_workspace(s, ws, &order, &gdesc, &ngroups, &recs);
        GroupArgs g;
        g.coarse = coarse_idx;
        g.C = s.C;
        g.Le = s.Le;
        for (int l = 0; l < 4; l++) {
            g.col[l] = l < s.Le ? s.col_off[l + 1] : 0;
            g.n_level[l] = l < s.Le ? s.n_level[l + 1] : 1;
        }
        LLSA_TRY(launch_group(s, sel_idx, g, order, gdesc, ngroups, recs, st));
        // both forwards are launched; each reads the group counts and only one
        // does the work (the other returns at once); for K_1 = 4 there is no
        // per-block tensor-core forward and the grouped one always runs
        LLSA_TRY(launch_fwd_grp(s, a, ngroups, recs, st));
        if (!fwd_tc_supported(s)) return LLSA_OK;  // the grouped forward always runs (K_1 = 4)
        a.ngroups = ngroups;
        a.ngroups_n = s.slices * (long long)group_windows(s);
        return launch_fwd_tc(s, a, st);
    }
    if (fwd_tc_supported(s)) return launch_fwd_tc(s, a, st);
    return launch_fwd_simt(s, a, st);
}

int launch_bwd(const Shape& s, const void* q, const void* k, const void* v, const void* o, const float* lse,
               const void* dout, const float* pyr, const int32_t* sel_idx, const int32_t* coarse_idx,
               const int32_t* col_ptr, const int32_t* row_idx, void* dq, void* dk, void* dv, void* ws,
               cudaStream_t st) {
    if (s.raster && !(bwd_tc_supported(s) && fwd_tc_supported(s))) return LLSA_ERR_UNSUPPORTED;
    AttnArgs a = make_attn_args(s);
    a.q = q; a.k = k; a.v = v; a.o = o; a.dout = dout; a.lse_in = lse;
    a.kpyr = pyr + s.slices * a.pyr_stride;
    a.vpyr = pyr + 2 * s.slices * a.pyr_stride;
    a.sel = sel_idx; a.coarse = coarse_idx; a.col_ptr = col_ptr; a.row_idx = row_idx;
    a.dq = dq; a.dk = dk; a.dv = dv;
    carve_bwd_workspace(s, ws, &a);
    if (bwd_tc_supported(s)) {
        LLSA_TRY(launch_bwd_dq_tc(s, a, st));
        LLSA_TRY(launch_coarse_reduce(s, a, st));
        return launch_bwd_dkv_tc(s, a, st);
    }
    LLSA_TRY(launch_bwd_dq_simt(s, a, st));
    LLSA_TRY(launch_coarse_reduce(s, a, st));
    return launch_bwd_dkv_simt(s, a, st);
}

}  // namespace llsa
