// select.cu -- hierarchical Top-K selection and the enrichment index.
//
// Method: Pith review of arXiv 2512.16615, "Core claim" and "What carries the
// argument": the coarsest level computes full similarities and keeps the K
// best per query; each finer level scores only the K*B children of the blocks
// kept above and carries the indices down (referee comment on Algorithm 1: the
// parent-to-child map is read as contiguous, children of j are jB..jB+B-1).
// Scores are raw dot products of pooled Q and K in fp32; ties go to the lower
// index; stored rows are ascending. The enrichment tokens of level l for
// query block i come from level l's row of i's ancestor floor(i / B^(l-1)):
// its rank-1 choice (TOP1), the ancestor itself (ANCESTOR) or the whole
// ascending row (ALLK), written into level l's columns of i's coarse row.
//
// One launch per level, coarsest first (each level needs the one above). A CTA
// owns up to 16 sibling query rows that share one candidate list: candidate
// key rows are staged through shared memory in tiles of 32*KPL (coalesced
// float4 loads), the 16 warps score the CTA's rows against the tile as KPL
// query rows x 32 candidates each (packed two-wide fp32 FMAs over even/odd
// columns; a candidate row is read once per KPL query rows), and the
// warp then runs K rounds of an arg-max tournament over its row's candidates
// (each lane holding ceil(C/32) of them): scores map to order-preserving
// unsigned keys, so a round is one warp max-reduction of the key and one
// min-reduction of the index among the lanes holding that key. K <= 64 and
// C <= 1024 here, so K rounds cost less than a full sort of the C candidates.
// With 16 or more candidates per lane (K_{l+1} B >= 512) the K-th largest key
// is found instead by a 32-step binary search on the key bits (one warp sum
// per step), and the row keeps every key above it plus the lowest indices
// among the ties.
#include <limits.h>

#include "internal.h"

namespace llsa {
namespace {

constexpr int kMaxRows = 16;  // query rows (warps) per CTA
constexpr int kMaxCand = 1024;
constexpr int kMaxKeep = 64;

struct SelectArgs {
    const float* qpyr;     // Q pyramid of slice 0 (level rows at row_off)
    const float* kpyr;     // K pyramid of slice 0
    long long pyr_stride;  // floats per slice pyramid
    int row_off;           // first pyramid row of this level
    int n_l, d, B;
    const int* parent;     // level l+1 selection of slice 0, or nullptr
    long long parent_stride;
    int Kp;
    int Kl;
    int* out;
    long long out_stride;
    int* coarse;           // [slices][T][ccols]
    int T, ccols, col0;    // coarse row length; this level's first column
    int level, span;       // span = B^(level-1)
    int rows_per_cta;
    int C;                 // candidates per row
    int n_parent;          // rows of the parent level (index check)
    int rule;              // enrichment rule
    int* status;
};

// Order-preserving map of a float to an unsigned key (for non-NaN inputs;
// -0 and +0 map to the same key).
__device__ __forceinline__ unsigned order_key(float v) {
    if (v == 0.f) v = 0.f;
    const unsigned u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// DT: the head dimension as a compile-time constant (64 or 128: divisions
// and the scoring loop resolve at compile time), or 0 for any d
template <int CPL, int KPL, int DT>
__global__ void __launch_bounds__(32 * kMaxRows, CPL <= 8 ? (DT > 0 ? 3 : 4) : 1) select_level_kernel(SelectArgs a) {
    constexpr int kTile = 32 * KPL;  // candidate rows per shared-memory tile
    extern __shared__ float4 smem4[];
    const int d = DT > 0 ? DT : a.d, C = a.C;
    const int ktile_stride = d + 4;
    float* ktile = reinterpret_cast<float*>(smem4);                 // [kTile][d+4]
    float* qrows = ktile + kTile * ktile_stride;                     // [rows][d]
    float* scores = qrows + kMaxRows * d;                            // [rows][C]
    int* cand = reinterpret_cast<int*>(scores + kMaxRows * C);       // [C]
    int* kept = cand + C;                                            // [rows][kMaxKeep]
    int* sorted = kept + kMaxRows * kMaxKeep;                        // [rows][kMaxKeep]

    const long long slice = blockIdx.y;
    const int row0 = blockIdx.x * a.rows_per_cta;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nthreads = blockDim.x;
    const float* qp = a.qpyr + slice * a.pyr_stride + (long long)a.row_off * d;
    const float* kp = a.kpyr + slice * a.pyr_stride + (long long)a.row_off * d;

    // candidate list (ascending token indices)
    if (a.parent) {
        const int* prow = a.parent + slice * a.parent_stride + (long long)(row0 / a.B) * a.Kp;
        for (int c = threadIdx.x; c < C; c += nthreads) {
            int j = prow[c / a.B];
            if (j < 0 || j >= a.n_parent) {
                set_status(a.status, LLSA_ERR_BAD_INDEX);
                j = 0;
            }
            cand[c] = j * a.B + c % a.B;
        }
    } else {
        for (int c = threadIdx.x; c < C; c += nthreads) cand[c] = c;
    }
    // query rows of this CTA
    const int nrows = min(a.rows_per_cta, a.n_l - row0);
    for (int i = threadIdx.x; i < nrows * (d / 4); i += nthreads) {
        const int r = i / (d / 4), c4 = i % (d / 4);
        reinterpret_cast<float4*>(qrows + r * d)[c4] =
            __ldg(reinterpret_cast<const float4*>(qp + (long long)(row0 + r) * d) + c4);
    }

    // scores, tile by tile
    for (int t0 = 0; t0 < C; t0 += kTile) {
        __syncthreads();
        const int tn = min(kTile, C - t0);
        for (int i = threadIdx.x; i < tn * (d / 4); i += nthreads) {
            const int r = i / (d / 4), c4 = i % (d / 4);
            reinterpret_cast<float4*>(ktile + r * ktile_stride)[c4] =
                __ldg(reinterpret_cast<const float4*>(kp + (long long)cand[t0 + r] * d) + c4);
        }
        __syncthreads();
        {
            // warp = (row group, candidate group): KPL query rows against 32
            // candidates, so each candidate row is read once per KPL query
            // rows (query rows are broadcast reads)
            const int rg = warp / KPL, cl = (warp % KPL) * 32 + lane;
            const float* kr = ktile + cl * ktile_stride;
            float2 acc[KPL];
#pragma unroll
            for (int r = 0; r < KPL; r++) acc[r] = make_float2(0.f, 0.f);
            for (int c = 0; c < d; c += 4) {
                const float4 k4 = *reinterpret_cast<const float4*>(kr + c);
                const float2 ka = make_float2(k4.x, k4.y), kb = make_float2(k4.z, k4.w);
#pragma unroll
                for (int r = 0; r < KPL; r++) {
                    const float4 q4 = *reinterpret_cast<const float4*>(qrows + (rg * KPL + r) * d + c);
                    acc[r] = __ffma2_rn(make_float2(q4.x, q4.y), ka, acc[r]);
                    acc[r] = __ffma2_rn(make_float2(q4.z, q4.w), kb, acc[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < KPL; r++)
                if (rg * KPL + r < nrows && cl < tn) scores[(rg * KPL + r) * C + t0 + cl] = acc[r].x + acc[r].y;
        }
    }
    __syncthreads();
    if (warp >= nrows) return;

    // Top-K rounds for row `warp`; a NaN score ranks with -inf
    unsigned key[CPL];
    int idx[CPL];
#pragma unroll
    for (int m = 0; m < CPL; m++) {
        const int c = lane + 32 * m;
        if (c < C) {
            const float v = scores[warp * C + c];
            key[m] = order_key(v != v ? -INFINITY : v);
            idx[m] = cand[c];
        } else {
            key[m] = 0u;  // below every score
            idx[m] = INT_MAX;
        }
    }
    int* krow = kept + warp * kMaxKeep;
    if constexpr (CPL <= 8) {
        // each lane sorts its candidates best first (insertion sort in
        // registers); a round then compares only the lanes' current heads
#pragma unroll
        for (int i = 1; i < CPL; i++)
#pragma unroll
            for (int j = i; j > 0; j--)
                if (key[j] > key[j - 1] || (key[j] == key[j - 1] && idx[j] < idx[j - 1])) {
                    const unsigned tk = key[j]; key[j] = key[j - 1]; key[j - 1] = tk;
                    const int ti = idx[j]; idx[j] = idx[j - 1]; idx[j - 1] = ti;
                }
        int head = 0;
        for (int k = 0; k < a.Kl; k++) {
            unsigned hk = 0u;
            int hi = INT_MAX;
#pragma unroll
            for (int m = 0; m < CPL; m++)
                if (head == m) { hk = key[m]; hi = idx[m]; }
            const unsigned wk = __reduce_max_sync(0xffffffffu, hk);
            const int wi = (int)__reduce_min_sync(0xffffffffu, hk == wk ? (unsigned)hi : 0xffffffffu);
            if (hk == wk && hi == wi) head++;
            if (lane == 0) krow[k] = wi;
        }
    } else {
        // 16 or more candidates per lane: a threshold select instead of K
        // rounds. T = the K-th largest key counted with multiplicity, found
        // bit by bit from the top (the largest T with at least K keys >= T;
        // padding keys are 0, below every score). The kept set is every key
        // above T, then the lowest indices among the keys equal to T: the same
        // set the rounds keep.
        unsigned T = 0u;
        for (int bit = 31; bit >= 0; bit--) {
            const unsigned t = T | (1u << bit);
            unsigned cnt = 0;
#pragma unroll
            for (int m = 0; m < CPL; m++) cnt += key[m] >= t ? 1u : 0u;
            if ((int)__reduce_add_sync(0xffffffffu, cnt) >= a.Kl) T = t;
        }
        bool sel[CPL];
        unsigned above = 0;
#pragma unroll
        for (int m = 0; m < CPL; m++) {
            sel[m] = key[m] > T;
            above += sel[m] ? 1u : 0u;
        }
        for (int need = a.Kl - (int)__reduce_add_sync(0xffffffffu, above); need > 0; need--) {
            unsigned bi = 0xffffffffu;
#pragma unroll
            for (int m = 0; m < CPL; m++)
                if (!sel[m] && key[m] == T && (unsigned)idx[m] < bi) bi = (unsigned)idx[m];
            const unsigned wi = __reduce_min_sync(0xffffffffu, bi);
#pragma unroll
            for (int m = 0; m < CPL; m++)
                if (!sel[m] && key[m] == T && (unsigned)idx[m] == wi) sel[m] = true;
        }
        // rank 1 (the largest key, the lowest index among equal ones; always
        // kept) first, then the others in lane order
        unsigned bk = 0u;
        int bi = INT_MAX;
#pragma unroll
        for (int m = 0; m < CPL; m++)
            if (key[m] > bk || (key[m] == bk && idx[m] < bi)) { bk = key[m]; bi = idx[m]; }
        const unsigned wk = __reduce_max_sync(0xffffffffu, bk);
        const int w1 = (int)__reduce_min_sync(0xffffffffu, bk == wk ? (unsigned)bi : 0xffffffffu);
        int base = 1;
#pragma unroll
        for (int m = 0; m < CPL; m++) {
            const bool put = sel[m] && idx[m] != w1;
            const unsigned bits = __ballot_sync(0xffffffffu, put);
            if (put) krow[base + __popc(bits & ((1u << lane) - 1u))] = idx[m];
            base += __popc(bits);
        }
        if (lane == 0) krow[0] = w1;
    }
    __syncwarp();
    const int row = row0 + warp;
    int* orow = a.out + slice * a.out_stride + (long long)row * a.Kl;
    int* srow = sorted + warp * kMaxKeep;
    for (int k = lane; k < a.Kl; k += 32) {
        const int v = krow[k];
        int rank = 0;
        for (int k2 = 0; k2 < a.Kl; k2++) rank += krow[k2] < v;
        orow[rank] = v;
        srow[rank] = v;
    }
    __syncwarp();
    // enrichment index: every level-1 descendant of this row gets, in this
    // level's columns, the row's rank-1 selection (TOP1), the row itself
    // (ANCESTOR) or the whole ascending row (ALLK)
    int* crow = a.coarse + (slice * a.T + (long long)row * a.span) * a.ccols + a.col0;
    if (a.rule == LLSA_ENRICH_ALLK) {
        for (int x = lane; x < a.span * a.Kl; x += 32)
            crow[(long long)(x / a.Kl) * a.ccols + x % a.Kl] = srow[x % a.Kl];
    } else {
        const int top1 = a.rule == LLSA_ENRICH_ANCESTOR ? row : krow[0];
        for (int q = lane; q < a.span; q += 32) crow[(long long)q * a.ccols] = top1;
    }
}

template <int KPL>
size_t level_smem(const SelectArgs& a) {
    return sizeof(float) * (32 * KPL * (a.d + 4) + kMaxRows * a.d + kMaxRows * a.C) +
           sizeof(int) * (a.C + 2 * kMaxRows * kMaxKeep);
}

template <int CPL, int KPL, int DT>
int launch_level_kpl(const SelectArgs& a, long long slices, cudaStream_t st) {
    const int grid_x = (a.n_l + a.rows_per_cta - 1) / a.rows_per_cta;
    const size_t smem = level_smem<KPL>(a);
    if (smem > 200 * 1024 || slices > 65535) return LLSA_ERR_UNSUPPORTED;
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(select_level_kernel<CPL, KPL, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    LLSA_LAUNCH("select_level", st,
                select_level_kernel<CPL, KPL, DT>
                <<<dim3(grid_x, (unsigned)slices), 32 * kMaxRows, smem, st>>>(a));
    return LLSA_OK;
}

// four candidates per lane per tile where the tile fits, else two; d = 64
// and d = 128 have their own instantiations
template <int CPL>
int launch_level(const SelectArgs& a, long long slices, cudaStream_t st) {
    if (level_smem<4>(a) <= 200 * 1024) {
        if (a.d == 64) return launch_level_kpl<CPL, 4, 64>(a, slices, st);
        if (a.d == 128) return launch_level_kpl<CPL, 4, 128>(a, slices, st);
        return launch_level_kpl<CPL, 4, 0>(a, slices, st);
    }
    return launch_level_kpl<CPL, 2, 0>(a, slices, st);
}

}  // namespace

int launch_select(const Shape& s, const float* pyr, int32_t* sel_idx, int32_t* coarse_idx, int32_t* level_idx,
                  cudaStream_t st) {
    const long long pyr_stride = (long long)s.P * s.d;
    const float* qpyr = pyr;
    const float* kpyr = pyr + s.slices * pyr_stride;
    // rows per CTA: a divisor of B (siblings share a parent) of at most 16
    int rpc = 1;
    for (int r = 1; r <= kMaxRows; r++)
        if (s.B % r == 0) rpc = r;
    long long span = 1;
    for (int l = 1; l < s.L; l++) span *= s.B;
    for (int l = s.L; l >= 1; l--) {
        SelectArgs a;
        a.qpyr = qpyr;
        a.kpyr = kpyr;
        a.pyr_stride = pyr_stride;
        a.row_off = s.row_offset[l];
        a.n_l = s.n_level[l];
        a.d = s.d;
        a.B = s.B;
        a.Kl = s.topk_level[l];
        a.coarse = coarse_idx;
        a.T = s.T;
        a.ccols = s.C;
        a.col0 = s.col_off[l];
        a.level = l;
        a.span = (int)span;
        a.status = status_ptr();
        a.rule = s.rule;
        if (l == s.L) {
            a.parent = nullptr;
            a.parent_stride = 0;
            a.Kp = 0;
            a.C = s.n_level[l];
            a.rows_per_cta = kMaxRows;
            a.n_parent = 0;
        } else {
            a.parent = level_idx + s.level_idx_offset[l + 1];
            a.parent_stride = s.level_idx_per_slice;
            a.Kp = s.topk_level[l + 1];
            a.C = a.Kp * s.B;
            a.rows_per_cta = rpc;
            a.n_parent = s.n_level[l + 1];
        }
        if (l == 1) {
            a.out = sel_idx;
            a.out_stride = (long long)s.T * s.K1;
        } else {
            a.out = level_idx + s.level_idx_offset[l];
            a.out_stride = s.level_idx_per_slice;
        }
        if (a.C > kMaxCand || a.Kl > kMaxKeep) return LLSA_ERR_UNSUPPORTED;
        const int cpl = (a.C + 31) / 32;
        int rc;
        if (cpl <= 1) rc = launch_level<1>(a, s.slices, st);
        else if (cpl <= 2) rc = launch_level<2>(a, s.slices, st);
        else if (cpl <= 4) rc = launch_level<4>(a, s.slices, st);
        else if (cpl <= 8) rc = launch_level<8>(a, s.slices, st);
        else if (cpl <= 16) rc = launch_level<16>(a, s.slices, st);
        else rc = launch_level<32>(a, s.slices, st);
        if (rc != LLSA_OK) return rc;
        span /= s.B;
    }
    return LLSA_OK;
}

}  // namespace llsa
