// pool.cu -- hierarchical compression: mean pyramids of Q, K and V.
//
// Method: Pith review of arXiv 2512.16615, "Core claim" (Q, K, V mean-pooled
// over log-many levels) and "What carries the argument" (L = floor(log_B N - 1)
// levels of contiguous B-token blocks). Level l row j is the mean of the B rows
// jB..jB+B-1 of level l-1; level 0 is the input.
//
// HBM-bound: every input byte is read once with 128-bit loads; each CTA owns
// a chunk of up to 4096 consecutive tokens of one tensor of one slice, writes
// its level-1 rows, then derives the coarser levels of the chunk from the rows
// it just wrote (L1/L2-resident). Levels whose blocks are longer than a chunk
// (only when B^L > 4096) are finished by a second small kernel. Under
// LLSA_ORDER_RASTER (index reordering, referee comments on Sec. 5.1 and
// Figure 2) the inputs are read in place as 4 x 4 token patches, so the
// pyramid is the one of the reordered tokens without a reordering pass.
#include "internal.h"

namespace llsa {
namespace {

constexpr int kPoolThreads = 256;
constexpr int kMaxChunk = 4096;

struct PoolArgs {
    const void* x[3];
    float* pyr;
    long long slices;
    int n, d, B, P;
    int raster, side;  // inputs in the raster order of a side x side image (B = 16)
    int chunk, levels_in_chunk;
    LevelTable lv;
};

// Mean of B rows of a coarser level (float4 column vv of rows r*B..r*B+B-1
// at row stride d), eight loads in flight, added in row order.
__device__ __forceinline__ float4 mean_rows(const float* prev, long long r, int B, int d, int vv, float inv) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < B; c0 += 8) {
        float4 f[8];
#pragma unroll
        for (int u = 0; u < 8; u++)
            f[u] = c0 + u < B ? *reinterpret_cast<const float4*>(prev + (r * B + c0 + u) * d + vv * 4)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 8; u++)
            if (c0 + u < B) {
                acc.x += f[u].x; acc.y += f[u].y; acc.z += f[u].z; acc.w += f[u].w;
            }
    }
    return make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

template <typename T, bool R>
__global__ void __launch_bounds__(kPoolThreads) pool_chunk_kernel(PoolArgs a) {
    const int tensor = blockIdx.y;
    const int nchunks = a.n / a.chunk;
    const long long slice = blockIdx.x / nchunks;
    const int c = blockIdx.x % nchunks;
    const int d = a.d, B = a.B;
    const T* x = static_cast<const T*>(a.x[tensor]) + (slice * a.n + (long long)c * a.chunk) * d;
    float* ps = a.pyr + ((long long)tensor * a.slices + slice) * a.P * (long long)d;
    const float inv = 1.0f / (float)B;

    // level 1: each item sums B input rows over 8 channels (one 16-byte vector
    // for bf16); consecutive threads take consecutive vectors of a row. Level-1
    // row r of the chunk is block b = c * rows + r of the slice: tokens 16 b ..
    // in tile order, or the block's 4 x 4 patch of the raster image, summed in
    // the same (tile) order.
    {
        const int rows = a.chunk / B;
        const int V = d / 8;
        float* out = ps + ((long long)a.lv.row_offset[1] + (long long)c * rows) * d;
        for (int item = threadIdx.x; item < rows * V; item += kPoolThreads) {
            const int r = item / V, vv = item % V;
            const T* src = x + (long long)r * B * d + vv * 8;
            if constexpr (R)  // block c * rows + r of the slice, from the tensor's base
                src = static_cast<const T*>(a.x[tensor]) + token_row(slice, a.n, 1, a.side, (c * rows + r) * B) * d + vv * 8;
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; i++) acc[i] = 0.f;
            int cc = 0;
            for (; cc + 8 <= B; cc += 8) {
                float f[8][8];
#pragma unroll
                for (int u = 0; u < 8; u++) load8(src + (R ? block_token_offset(cc + u, a.side) : (long long)(cc + u)) * d, f[u]);
#pragma unroll
                for (int u = 0; u < 8; u++)
#pragma unroll
                    for (int i = 0; i < 8; i++) acc[i] += f[u][i];
            }
            for (; cc < B; cc++) {
                float f[8];
                load8(src + (R ? block_token_offset(cc, a.side) : (long long)cc) * d, f);
#pragma unroll
                for (int i = 0; i < 8; i++) acc[i] += f[i];
            }
            float* dst = out + (long long)r * d + vv * 8;
            *reinterpret_cast<float4*>(dst) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
            *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
        }
    }
    // coarser levels inside the chunk, from the rows this CTA just wrote
    int rows_prev = a.chunk / B;
    for (int l = 2; l <= a.levels_in_chunk; l++) {
        __syncthreads();
        const int rows = rows_prev / B;
        const float* prev = ps + ((long long)a.lv.row_offset[l - 1] + (long long)c * rows_prev) * d;
        float* out = ps + ((long long)a.lv.row_offset[l] + (long long)c * rows) * d;
        const int V = d / 4;
        for (int item = threadIdx.x; item < rows * V; item += kPoolThreads) {
            const int r = item / V, vv = item % V;
            *reinterpret_cast<float4*>(out + (long long)r * d + vv * 4) = mean_rows(prev, r, B, d, vv, inv);
        }
        rows_prev = rows;
    }
}

// Levels above the chunk: one CTA per (slice, tensor), level by level.
__global__ void __launch_bounds__(kPoolThreads) pool_upper_kernel(PoolArgs a, int first_level, int L) {
    const int tensor = blockIdx.y;
    const long long slice = blockIdx.x;
    const int d = a.d, B = a.B;
    float* ps = a.pyr + ((long long)tensor * a.slices + slice) * a.P * (long long)d;
    const float inv = 1.0f / (float)B;
    for (int l = first_level; l <= L; l++) {
        __syncthreads();
        const int rows = a.lv.n_level[l];
        const float* prev = ps + (long long)a.lv.row_offset[l - 1] * d;
        float* out = ps + (long long)a.lv.row_offset[l] * d;
        const int V = d / 4;
        for (int item = threadIdx.x; item < rows * V; item += kPoolThreads) {
            const int r = item / V, vv = item % V;
            *reinterpret_cast<float4*>(out + (long long)r * d + vv * 4) = mean_rows(prev, r, B, d, vv, inv);
        }
    }
}

}  // namespace

int launch_pool(const Shape& s, const void* q, const void* k, const void* v, float* pyr, cudaStream_t st) {
    PoolArgs a;
    a.x[0] = q; a.x[1] = k; a.x[2] = v;
    a.pyr = pyr; a.slices = s.slices; a.n = s.n; a.d = s.d; a.B = s.B; a.P = s.P;
    a.raster = s.raster; a.side = s.side;
    a.lv = level_table(s);
    // largest level whose blocks fit in one chunk, then widen the chunk by
    // powers of two while it still divides N
    int lc = 0;
    long long span = 1;
    while (lc < s.L && span * s.B <= kMaxChunk) { span *= s.B; lc++; }
    if (lc == 0) return LLSA_ERR_UNSUPPORTED;
    long long chunk = span;
    while (chunk * 2 <= kMaxChunk && s.n % (chunk * 2) == 0) chunk *= 2;
    a.chunk = (int)chunk;
    a.levels_in_chunk = lc;
    const long long blocks = s.slices * (s.n / chunk);
    if (blocks > 0x7fffffffLL) return LLSA_ERR_UNSUPPORTED;
    dim3 grid((unsigned)blocks, 3);
    // one instance per dtype and token order
    if (s.dtype == LLSA_DTYPE_BF16 && s.raster)
        LLSA_LAUNCH("pool_chunk", st, pool_chunk_kernel<__nv_bfloat16, true><<<grid, kPoolThreads, 0, st>>>(a));
    else if (s.dtype == LLSA_DTYPE_BF16)
        LLSA_LAUNCH("pool_chunk", st, pool_chunk_kernel<__nv_bfloat16, false><<<grid, kPoolThreads, 0, st>>>(a));
    else if (s.raster)
        LLSA_LAUNCH("pool_chunk", st, pool_chunk_kernel<float, true><<<grid, kPoolThreads, 0, st>>>(a));
    else
        LLSA_LAUNCH("pool_chunk", st, pool_chunk_kernel<float, false><<<grid, kPoolThreads, 0, st>>>(a));
    if (lc < s.L)
        LLSA_LAUNCH("pool_upper", st,
                    pool_upper_kernel<<<dim3((unsigned)s.slices, 3), kPoolThreads, 0, st>>>(a, lc + 1, s.L));
    return LLSA_OK;
}

}  // namespace llsa
