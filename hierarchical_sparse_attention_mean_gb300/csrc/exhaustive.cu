// exhaustive.cu -- single-level full scoring of the level-1 tokens, the
// reference the hierarchical selection is measured against (routing recall).
//
// Method: Pith review of arXiv 2512.16615, "Core claim" (the hierarchy
// replaces full scoring at the fine level) and the referee's question on
// routing recall: how much of the exhaustive fine-level Top-K the coarse-to-
// fine selection keeps. Here every level-1 query token (a pooled query block)
// scores all T level-1 key tokens with the same raw pooled dot product as the
// selection (fp32, same summation order, so a pair scores identically in both
// kernels) and keeps its K_x = min(K, T) best; ties go to the lower index;
// rows are stored ascending.
//
// A CTA owns 16 query rows (one warp each) and streams all T key rows through
// shared memory in tiles of 128. Each warp keeps its running Top-K in shared
// memory; a tile's candidates are merged only when one of them beats the
// current K-th entry (after the first tiles that is rare), by K rounds of a
// warp max / min reduction over order-preserving keys.
#include <limits.h>

#include <algorithm>

#include "internal.h"

namespace llsa {
namespace {

constexpr int kRowsX = 16;   // query rows (warps) per CTA
constexpr int kKPL = 4;      // candidates per lane per tile
constexpr int kTileX = 32 * kKPL;
constexpr int kKeepX = 64;   // K at most

struct ExArgs {
    const float* qpyr;     // level-1 rows of the Q pyramid of slice 0
    const float* kpyr;     // level-1 rows of the K pyramid of slice 0
    long long pyr_stride;  // floats per slice pyramid
    int T, d, K;
    int* out;              // [slices][T][K]
};

// Order-preserving map of a float to an unsigned key (non-NaN inputs; -0 and
// +0 map to the same key). Key 0 is below every score.
__device__ __forceinline__ unsigned score_key(float v) {
    if (v != v) v = -INFINITY;  // a NaN score ranks with -inf
    if (v == 0.f) v = 0.f;
    const unsigned u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ bool beats(unsigned ka, int ia, unsigned kb, int ib) {
    return ka > kb || (ka == kb && ia < ib);
}

__global__ void __launch_bounds__(32 * kRowsX) exhaustive_kernel(ExArgs a) {
    extern __shared__ float4 smem4[];
    const int d = a.d, T = a.T, K = a.K;
    const int ks = d + 4;
    float* ktile = reinterpret_cast<float*>(smem4);                        // [kTileX][d+4]
    float* qrows = ktile + kTileX * ks;                                     // [kRowsX][d]
    unsigned* bkey = reinterpret_cast<unsigned*>(qrows + kRowsX * d);       // [kRowsX][kKeepX]
    int* bidx = reinterpret_cast<int*>(bkey + kRowsX * kKeepX);             // [kRowsX][kKeepX]

    const long long slice = blockIdx.y;
    const int row0 = blockIdx.x * kRowsX;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nrows = min(kRowsX, T - row0);
    const float* qp = a.qpyr + slice * a.pyr_stride;
    const float* kp = a.kpyr + slice * a.pyr_stride;

    for (int i = threadIdx.x; i < nrows * (d / 4); i += blockDim.x) {
        const int r = i / (d / 4), c4 = i % (d / 4);
        reinterpret_cast<float4*>(qrows + r * d)[c4] =
            __ldg(reinterpret_cast<const float4*>(qp + (long long)(row0 + r) * d) + c4);
    }
    // running Top-K: placeholders (key 0, index INT_MAX) below every candidate
    for (int i = threadIdx.x; i < kRowsX * kKeepX; i += blockDim.x) {
        bkey[i] = 0u;
        bidx[i] = INT_MAX;
    }
    unsigned* mk = bkey + warp * kKeepX;
    int* mi = bidx + warp * kKeepX;

    for (int t0 = 0; t0 < T; t0 += kTileX) {
        __syncthreads();
        const int tn = min(kTileX, T - t0);
        for (int i = threadIdx.x; i < tn * (d / 4); i += blockDim.x) {
            const int r = i / (d / 4), c4 = i % (d / 4);
            reinterpret_cast<float4*>(ktile + r * ks)[c4] =
                __ldg(reinterpret_cast<const float4*>(kp + (long long)(t0 + r) * d) + c4);
        }
        __syncthreads();
        if (warp >= nrows) continue;
        // scores of this lane's candidates: packed two-wide FMAs over even/odd
        // columns, the selection's own arithmetic
        const float* qr = qrows + warp * d;
        float2 acc[kKPL];
#pragma unroll
        for (int j = 0; j < kKPL; j++) acc[j] = make_float2(0.f, 0.f);
        for (int c = 0; c < d; c += 4) {
            const float4 q4 = *reinterpret_cast<const float4*>(qr + c);
            const float2 qa = make_float2(q4.x, q4.y), qb = make_float2(q4.z, q4.w);
#pragma unroll
            for (int j = 0; j < kKPL; j++) {
                const float4 k4 = *reinterpret_cast<const float4*>(ktile + (lane + 32 * j) * ks + c);
                acc[j] = __ffma2_rn(qa, make_float2(k4.x, k4.y), acc[j]);
                acc[j] = __ffma2_rn(qb, make_float2(k4.z, k4.w), acc[j]);
            }
        }
        unsigned ck[kKPL];
        int ci[kKPL];
        bool pass = false;
        const unsigned tk = mk[K - 1];
        const int ti = mi[K - 1];
#pragma unroll
        for (int j = 0; j < kKPL; j++) {
            const int c = lane + 32 * j;
            ck[j] = c < tn ? score_key(acc[j].x + acc[j].y) : 0u;
            ci[j] = c < tn ? t0 + c : INT_MAX;
            pass |= c < tn && beats(ck[j], ci[j], tk, ti);
        }
        if (!__any_sync(0xffffffffu, pass)) continue;
        // merge: the current best (two per lane) and this lane's candidates
        constexpr int E = kKeepX / 32 + kKPL;
        unsigned ek[E];
        int ei[E];
#pragma unroll
        for (int m = 0; m < kKeepX / 32; m++) {
            const int r = lane + 32 * m;
            ek[m] = r < K ? mk[r] : 0u;
            ei[m] = r < K ? mi[r] : INT_MAX;
        }
#pragma unroll
        for (int j = 0; j < kKPL; j++) {
            ek[kKeepX / 32 + j] = ck[j];
            ei[kKeepX / 32 + j] = ci[j];
        }
        __syncwarp();
        unsigned taken = 0;
        for (int r = 0; r < K; r++) {
            unsigned bk = 0u;
            int bi = INT_MAX;
#pragma unroll
            for (int m = 0; m < E; m++)
                if (!(taken >> m & 1u) && beats(ek[m], ei[m], bk, bi)) { bk = ek[m]; bi = ei[m]; }
            const unsigned wk = __reduce_max_sync(0xffffffffu, bk);
            const int wi = (int)__reduce_min_sync(0xffffffffu, bk == wk ? (unsigned)bi : 0xffffffffu);
#pragma unroll
            for (int m = 0; m < E; m++)
                if (ei[m] == wi && ek[m] == wk) taken |= 1u << m;
            if (lane == 0) {
                mk[r] = wk;
                mi[r] = wi;
            }
        }
        __syncwarp();
    }
    __syncthreads();
    if (warp >= nrows) return;
    // the row's indices in ascending order
    int* orow = a.out + (slice * T + row0 + warp) * (long long)K;
    for (int k = lane; k < K; k += 32) {
        const int v = mi[k];
        int rank = 0;
        for (int k2 = 0; k2 < K; k2++) rank += mi[k2] < v;
        orow[rank] = v;
    }
}

}  // namespace

int launch_select_exhaustive(const Shape& s, const float* pyr, int32_t* out, cudaStream_t st) {
    ExArgs a;
    a.pyr_stride = (long long)s.P * s.d;
    a.qpyr = pyr + (long long)s.row_offset[1] * s.d;
    a.kpyr = pyr + s.slices * a.pyr_stride + (long long)s.row_offset[1] * s.d;
    a.T = s.T;
    a.d = s.d;
    a.K = std::min(s.topk, s.T);
    a.out = out;
    if (a.K < 1 || a.K > kKeepX || s.slices > 65535) return LLSA_ERR_UNSUPPORTED;
    const size_t smem = sizeof(float) * ((size_t)kTileX * (s.d + 4) + (size_t)kRowsX * s.d) +
                        (sizeof(unsigned) + sizeof(int)) * kRowsX * kKeepX;
    if (smem > 200 * 1024) return LLSA_ERR_UNSUPPORTED;
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(exhaustive_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const dim3 grid((s.T + kRowsX - 1) / kRowsX, (unsigned)s.slices);
    LLSA_LAUNCH("select_exhaustive", st, exhaustive_kernel<<<grid, 32 * kRowsX, smem, st>>>(a));
    return LLSA_OK;
}

}  // namespace llsa
