// transpose.cu -- sparse index transpose (CSR to CSC).
//
// Method: Pith review of arXiv 2512.16615, "What carries the argument": a
// sparse-index transpose (CSR-to-CSC scan) gives the backward pass, for each
// key block, its query blocks without building a dense N x N mask. The
// counting-sort form follows Gustavson's permuted transposition (reference
// [11] of the paper): count the entries of each column, exclusive-scan the
// counts into column pointers, scatter the row numbers.
//
// Four kernels per call, all slices in one launch each:
//   count   -- 128-bit loads of the CSR entries, one atomic per entry into the
//              column counters (the workspace);
//   scan    -- one CTA per slice: coalesced int4 loads, warp-shuffle prefix
//              scans, CTA-wide carry; writes col_ptr and the scatter cursors;
//   scatter -- 128-bit loads again, an atomic cursor per entry gives its slot;
//   order   -- one warp per column puts its rows in ascending order (warp
//              bitonic sort for up to 32 rows, a shared-memory bitmap of row
//              numbers for longer columns), so the result is deterministic
//              and bit-exact whatever order the atomics took.
#include <limits.h>

#include <algorithm>

#include "internal.h"

namespace llsa {
namespace {

constexpr int kCountThreads = 256;
constexpr int kScanThreads = 1024;
constexpr int kOrderWarps = 8;

// Entries are processed four at a time (one 128-bit load); the last vector
// may be short when the entry count is not a multiple of four.
__device__ __forceinline__ int load_entries(const int* __restrict__ sel, long long v, long long total, int* vals) {
    const long long e0 = v * 4;
    if (e0 + 3 < total) {
        const int4 e = __ldg(reinterpret_cast<const int4*>(sel) + v);
        vals[0] = e.x; vals[1] = e.y; vals[2] = e.z; vals[3] = e.w;
        return 4;
    }
    int m = 0;
    for (; e0 + m < total; m++) vals[m] = sel[e0 + m];
    return m;
}

__global__ void __launch_bounds__(kCountThreads) transpose_count_kernel(const int* __restrict__ sel, long long total,
                                                                         int per_slice, int ncols, int* __restrict__ cnt,
                                                                         int* status) {
    const long long nvec = (total + 3) / 4;
    for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < nvec;
         v += (long long)gridDim.x * blockDim.x) {
        int vals[4];
        const int m = load_entries(sel, v, total, vals);
        for (int u = 0; u < m; u++) {
            const long long slice = (v * 4 + u) / per_slice;
            if (vals[u] >= 0 && vals[u] < ncols) atomicAdd(cnt + slice * ncols + vals[u], 1);
            else set_status(status, LLSA_ERR_BAD_INDEX);
        }
    }
}

// Exclusive scan of one slice's column counts. Each thread owns 4
// consecutive counters of a 4096-wide tile.
__global__ void __launch_bounds__(kScanThreads) transpose_scan_kernel(int* __restrict__ cnt, int ncols,
                                                                       int* __restrict__ col_ptr) {
    __shared__ int warp_tot[kScanThreads / 32];
    __shared__ int carry_s;
    const long long slice = blockIdx.x;
    int* c = cnt + slice * ncols;
    int* cp = col_ptr + slice * (long long)(ncols + 1);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool vec = (ncols % 4) == 0;  // keeps every slice's row 16-byte aligned
    if (threadIdx.x == 0) carry_s = 0;
    __syncthreads();
    for (int base = 0; base < ncols; base += 4 * kScanThreads) {
        const int j = base + 4 * threadIdx.x;
        int v[4] = {0, 0, 0, 0};
        if (vec && j + 3 < ncols) {
            int4 t = *reinterpret_cast<const int4*>(c + j);
            v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
        } else {
            for (int u = 0; u < 4; u++) if (j + u < ncols) v[u] = c[j + u];
        }
        const int local = v[0] + v[1] + v[2] + v[3];
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = warp_tot[lane];
            int wi = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int t = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= o) wi += t;
            }
            warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
        }
        __syncthreads();
        const int carry = carry_s;
        int run = carry + warp_tot[warp] + incl - local;
        int out[4];
        for (int u = 0; u < 4; u++) { out[u] = run; run += v[u]; }
        if (vec && j + 3 < ncols) {
            *reinterpret_cast<int4*>(c + j) = make_int4(out[0], out[1], out[2], out[3]);  // scatter cursors
            for (int u = 0; u < 4; u++) cp[j + u] = out[u];
        } else {
            for (int u = 0; u < 4; u++) if (j + u < ncols) { c[j + u] = out[u]; cp[j + u] = out[u]; }
        }
        __syncthreads();
        if (threadIdx.x == kScanThreads - 1) carry_s = run;
        __syncthreads();
    }
    if (threadIdx.x == 0) cp[ncols] = carry_s;
}

__global__ void __launch_bounds__(kCountThreads) transpose_scatter_kernel(const int* __restrict__ sel,
                                                                           long long total, int per_slice, int K,
                                                                           int ncols, int* __restrict__ cursor,
                                                                           int* __restrict__ row_idx) {
    const long long nvec = (total + 3) / 4;
    for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < nvec;
         v += (long long)gridDim.x * blockDim.x) {
        int vals[4];
        const int m = load_entries(sel, v, total, vals);
        for (int u = 0; u < m; u++) {
            const int j = vals[u];
            if (j < 0 || j >= ncols) continue;
            const long long e = v * 4 + u;
            const long long slice = e / per_slice;
            const int pos = atomicAdd(cursor + slice * ncols + j, 1);
            row_idx[slice * per_slice + pos] = (int)(e - slice * per_slice) / K;
        }
    }
}

__device__ __forceinline__ int bitonic_warp_sort(int x, int lane) {
    // ascending bitonic sort of one value per lane
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const int y = __shfl_xor_sync(0xffffffffu, x, j);
            const bool up = ((lane & k) == 0);
            const bool lower = ((lane & j) == 0);
            x = (lower == up) ? min(x, y) : max(x, y);
        }
    }
    return x;
}

__global__ void __launch_bounds__(32 * kOrderWarps) transpose_order_kernel(const int* __restrict__ col_ptr,
                                                                            long long columns, int ncols,
                                                                            int per_slice, int nrows,
                                                                            int* __restrict__ row_idx) {
    extern __shared__ unsigned bitmap_all[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int words = (nrows + 31) / 32;
    unsigned* bm = bitmap_all + warp * words;
    for (long long col = blockIdx.x * (long long)kOrderWarps + warp; col < columns;
         col += (long long)gridDim.x * kOrderWarps) {
        const long long slice = col / ncols;
        const int j = (int)(col - slice * ncols);
        const int* cp = col_ptr + slice * (long long)(ncols + 1);
        const int beg = cp[j], cnt = cp[j + 1] - beg;
        int* r = row_idx + slice * per_slice + beg;
        if (cnt <= 1) continue;
        if (cnt <= 32) {
            int x = lane < cnt ? r[lane] : INT_MAX;
            x = bitonic_warp_sort(x, lane);
            if (lane < cnt) r[lane] = x;
            continue;
        }
        for (int w = lane; w < words; w += 32) bm[w] = 0u;
        __syncwarp();
        for (int e = lane; e < cnt; e += 32) {
            const int i = r[e];
            if (i >= 0 && i < nrows) atomicOr(bm + (i >> 5), 1u << (i & 31));
        }
        __syncwarp();
        int written = 0;
        for (int w0 = 0; w0 < words; w0 += 32) {
            const int w = w0 + lane;
            unsigned bits = w < words ? bm[w] : 0u;
            const int pc = __popc(bits);
            int incl = pc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            int pos = written + incl - pc;
            while (bits) {
                const int b = __ffs(bits) - 1;
                bits &= bits - 1;
                r[pos++] = w * 32 + b;
            }
            written += __shfl_sync(0xffffffffu, incl, 31);
        }
        __syncwarp();
    }
}

}  // namespace

// sel: [slices][rows][K] with entries in [0, ncols). scratch: [slices][ncols].
int launch_transpose(const Shape& s, const int32_t* sel, int rows, int K, int ncols, int32_t* col_ptr,
                     int32_t* row_idx, int32_t* scratch, cudaStream_t st) {
    const int per_slice = rows * K;
    const long long total = s.slices * (long long)per_slice;
    if (s.slices > 0x7fffffffLL) return LLSA_ERR_UNSUPPORTED;
    int* status = status_ptr();
    if (cudaMemsetAsync(scratch, 0, sizeof(int) * s.slices * (size_t)ncols, st) != cudaSuccess) return LLSA_ERR_CUDA;
    const long long nvec = (total + 3) / 4;
    const int grid = (int)std::max<long long>(1, std::min<long long>((nvec + kCountThreads - 1) / kCountThreads,
                                                                       (long long)sm_count() * 8));
    LLSA_LAUNCH("transpose_count", st,
                transpose_count_kernel<<<grid, kCountThreads, 0, st>>>(sel, total, per_slice, ncols, scratch, status));
    LLSA_LAUNCH("transpose_scan", st,
                transpose_scan_kernel<<<(unsigned)s.slices, kScanThreads, 0, st>>>(scratch, ncols, col_ptr));
    LLSA_LAUNCH("transpose_scatter", st,
                transpose_scatter_kernel<<<grid, kCountThreads, 0, st>>>(sel, total, per_slice, K, ncols, scratch,
                                                                        row_idx));
    const long long columns = s.slices * (long long)ncols;
    const size_t smem = sizeof(unsigned) * kOrderWarps * (size_t)((rows + 31) / 32);
    if (smem > 200 * 1024) return LLSA_ERR_UNSUPPORTED;
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(transpose_order_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const int ogrid = (int)std::min<long long>((columns + kOrderWarps - 1) / kOrderWarps, (long long)sm_count() * 16);
    LLSA_LAUNCH("transpose_order", st,
                transpose_order_kernel<<<ogrid, 32 * kOrderWarps, smem, st>>>(col_ptr, columns, ncols, per_slice,
                                                                              rows, row_idx));
    return LLSA_OK;
}

}  // namespace llsa
