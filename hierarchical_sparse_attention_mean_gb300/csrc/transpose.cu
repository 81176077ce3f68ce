// transpose.cu -- sparse index transpose (CSR to CSC).
//
// Method: Pith review of arXiv 2512.16615, "What carries the argument": a
// sparse-index transpose (CSR-to-CSC scan) gives the backward pass, for each
// key block, its query blocks without building a dense N x N mask. The
// counting-sort form follows Gustavson's permuted transposition (reference
// [11] of the paper): count the entries of each column, exclusive-scan the
// counts into column pointers, scatter the row numbers.
//
// One kernel per call where a slice fits the shared memory of eight CTAs and
// all slices' clusters are resident at once: a cluster of eight CTAs per slice.
//   1. CTA r takes rows [r R, (r+1) R) of the slice: it counts their entries
//      per column in shared memory, scans the counts, and places each row
//      number in its column's run (shared-memory atomics choose the slot);
//      then it sorts each run (a thread per short run, a warp and a bitmap of
//      the CTA's rows per long one).
//   2. Cluster barrier. CTA r owns columns [r C, (r+1) C): it reads every
//      CTA's run length of those columns through distributed shared memory,
//      scans the totals (the CTAs' sums are exchanged the same way) and
//      writes col_ptr.
//   3. CTA r writes the output of its columns, a contiguous range of row_idx:
//      per column, the runs of CTAs 0..7 in that order, each CTA's runs of
//      32 consecutive columns read as one block by consecutive lanes. The
//      CTAs' rows lie in ascending ranges and each run is sorted, so every
//      column comes out ascending and the result is the same whatever order
//      the atomics took.
//   HBM sees the entries read (twice, the second time mostly from L2) and the
//   output written once; no global atomics, no scratch.
//
// Otherwise four kernels, all slices in one launch each:
//   count   -- 128-bit loads of the CSR entries, one atomic per entry into the
//              column counters (the workspace);
//   scan    -- one CTA per slice: coalesced int4 loads, warp-shuffle prefix
//              scans, CTA-wide carry; writes col_ptr and the scatter cursors;
//   scatter -- 128-bit loads again, an atomic cursor per entry gives its slot;
//   order   -- one warp per column puts its rows in ascending order (warp
//              bitonic sort for up to 32 rows, a shared-memory bitmap of row
//              numbers for longer columns), so the result is deterministic
//              and bit-exact whatever order the atomics took.
#include <cooperative_groups.h>
#include <limits.h>

#include <algorithm>
#include <mutex>

#include "internal.h"

namespace cg = cooperative_groups;

namespace llsa {
namespace {

constexpr int kCountThreads = 256;
constexpr int kCluster = 8;           // CTAs per slice in the one-kernel transpose
constexpr int kClThreads = 1024;
constexpr int kClWarps = kClThreads / 32;
constexpr int kShortRun = 16;         // runs up to this length are sorted by one thread
constexpr size_t kClSmemMax = 220 * 1024;
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

// Shared memory of the one-kernel transpose, identical in every CTA of a
// cluster (distributed shared memory addresses it by the same offsets).
struct ClLayout {
    int R, C, words;  // rows per CTA, owned columns per CTA, bitmap words per warp
    size_t off_rows, off_queue, off_bits, off_misc, bytes;
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

__host__ __device__ inline ClLayout cl_layout(int rows, int K, int ncols) {
    ClLayout L;
    L.R = (rows + kCluster - 1) / kCluster;
    L.C = (ncols + kCluster - 1) / kCluster;
    L.words = (L.R + 31) / 32;
    const size_t ent = (size_t)L.R * K;
    L.off_rows = align16(sizeof(int) * ((size_t)ncols + 1));                           // run[ncols + 1]
    L.off_queue = L.off_rows + align16(sizeof(int) * ent);                              // rws[R K]
    L.off_bits = L.off_queue + align16(sizeof(int) * (ent / (kShortRun + 1) + 1));     // queue
    L.off_misc = L.off_bits + align16(sizeof(unsigned) * (size_t)kClWarps * L.words);  // bitmaps
    L.bytes = L.off_misc + align16(sizeof(int) * (64 + (size_t)(L.C + 31) / 32 + 1));  // misc, group sums
    return L;
}

__device__ __forceinline__ int warp_inclusive_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Exclusive scan of one value per thread of the CTA; the CTA's total lands in
// *total, which every thread may read once the call returns.
__device__ __forceinline__ int cta_exclusive_scan(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < kClWarps ? warp_sums[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += t;
        }
        if (lane < kClWarps) warp_sums[lane] = wi - w;
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    const int ex = warp_sums[warp] + incl - v;
    __syncthreads();
    return ex;
}

// The CTA's entries [e0, e1) of the slice, eight loads in flight per thread;
// f(entry index, column) for each.
template <typename F>
__device__ __forceinline__ void for_entries(const int* __restrict__ src, int e0, int e1, F f) {
    for (int eb = e0 + (int)threadIdx.x; eb < e1; eb += 8 * kClThreads) {
        int v[8];
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const int e = eb + u * kClThreads;
            v[u] = e < e1 ? __ldg(src + e) : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const int e = eb + u * kClThreads;
            if (e < e1) f(e, v[u]);
        }
    }
}

// One cluster of kCluster CTAs per slice; every thread reaches every barrier.
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kClThreads, 1)
transpose_cluster_kernel(const int* __restrict__ sel, int rows, int K, int ncols, int* __restrict__ col_ptr,
                         int* __restrict__ row_idx, int* status) {
    extern __shared__ __align__(16) unsigned char cl_smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const ClLayout L = cl_layout(rows, K, ncols);
    // run: counts per column, then first slots, then (after placement) run ends
    int* run = reinterpret_cast<int*>(cl_smem);
    int* rws = reinterpret_cast<int*>(cl_smem + L.off_rows);     // row numbers grouped by column
    int* queue = reinterpret_cast<int*>(cl_smem + L.off_queue);  // columns whose run is long
    unsigned* bits = reinterpret_cast<unsigned*>(cl_smem + L.off_bits);
    int* misc = reinterpret_cast<int*>(cl_smem + L.off_misc);    // [0, 32) warp sums, 32 queue length, 33 total
    const int r = (int)cluster.block_rank();
    const long long slice = blockIdx.x / kCluster;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = min(rows, r * L.R), r1 = min(rows, r0 + L.R);
    const int e0 = r0 * K, e1 = r1 * K;
    const int* src = sel + slice * (long long)rows * K;

    // 1a. entries per column among this CTA's rows
    for (int j = tid; j <= ncols; j += kClThreads) run[j] = 0;
    if (tid == 0) misc[32] = 0;
    __syncthreads();
    for_entries(src, e0, e1, [&](int, int j) {
        if (j >= 0 && j < ncols) atomicAdd(run + j, 1);
        else set_status(status, LLSA_ERR_BAD_INDEX);
    });
    __syncthreads();
    // 1b. first slot of each column's run: each warp scans a contiguous chunk
    // of the counts, consecutive lanes on consecutive words
    {
        const int chunk = (ncols + kClWarps - 1) / kClWarps;
        const int ja = min(ncols, warp * chunk), jb = min(ncols, ja + chunk);
        int sum = 0;
        for (int j = ja + lane; j < jb; j += 32) sum += run[j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        int carry = __shfl_sync(0xffffffffu, cta_exclusive_scan(lane == 0 ? sum : 0, misc, misc + 33), 0);
        for (int j0 = ja; j0 < jb; j0 += 32) {
            const int j = j0 + lane;
            const int c = j < jb ? run[j] : 0;
            const int incl = warp_inclusive_scan(c);
            if (j < jb) run[j] = carry + incl - c;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    __syncthreads();
    // 1c. placement (second read of the entries, mostly from L2); afterwards
    // run[j] is the end of column j's run, i.e. its run is [run[j-1], run[j])
    for_entries(src, e0, e1, [&](int e, int j) {
        if (j >= 0 && j < ncols) rws[atomicAdd(run + j, 1)] = e / K;
    });
    __syncthreads();
    // 1d. each run in ascending row order: insertion sort by one thread for a
    // short run, a warp and a bitmap over the CTA's rows for a long one (a
    // column holds a row at most once, the entries of a row being distinct)
    for (int j = tid; j < ncols; j += kClThreads) {
        const int b = j > 0 ? run[j - 1] : 0, e = run[j];
        if (e - b <= 1) continue;
        if (e - b > kShortRun) {
            queue[atomicAdd(misc + 32, 1)] = j;
            continue;
        }
        for (int x = b + 1; x < e; x++) {
            const int key = rws[x];
            int y = x - 1;
            while (y >= b && rws[y] > key) {
                rws[y + 1] = rws[y];
                y--;
            }
            rws[y + 1] = key;
        }
    }
    __syncthreads();
    {
        const int nq = misc[32];
        unsigned* bm = bits + warp * L.words;
        for (int qi = warp; qi < nq; qi += kClWarps) {
            const int j = queue[qi];
            const int b = j > 0 ? run[j - 1] : 0, e = run[j];
            for (int w = lane; w < L.words; w += 32) bm[w] = 0u;
            __syncwarp();
            for (int x = b + lane; x < e; x += 32) {
                const int i = rws[x] - r0;
                atomicOr(bm + (i >> 5), 1u << (i & 31));
            }
            __syncwarp();
            int written = b;
            for (int w0 = 0; w0 < L.words; w0 += 32) {
                const int w = w0 + lane;
                unsigned m = w < L.words ? bm[w] : 0u;
                const int pc = __popc(m);
                int incl = pc;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                int pos = written + incl - pc;
                while (m) {
                    const int bt = __ffs(m) - 1;
                    m &= m - 1;
                    rws[pos++] = r0 + w * 32 + bt;
                }
                written += __shfl_sync(0xffffffffu, incl, 31);
            }
            __syncwarp();
        }
    }
    // 2. this CTA's columns [c0, c1), in groups of 32 (a column per lane):
    // every CTA's run bounds of a group, read through distributed shared
    // memory by consecutive lanes, give the group's entries; a scan over the
    // groups and over the CTAs' totals gives the output slots
    cluster.sync();
    const int c0 = min(ncols, r * L.C), c1 = min(ncols, c0 + L.C);
    const int ngroups = (c1 - c0 + 31) / 32;
    int* gsum = misc + 64;  // per group: its entries, then its first slot in the CTA's range
    for (int g = warp; g < ngroups; g += kClWarps) {
        const int j = c0 + g * 32 + lane;
        int t = 0;
        if (j < c1)
#pragma unroll
            for (int q = 0; q < kCluster; q++) {
                const int* rq = cluster.map_shared_rank(run, q);
                t += rq[j] - (j > 0 ? rq[j - 1] : 0);
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) gsum[g] = t;
    }
    __syncthreads();
    if (warp == 0) {
        int carry = 0;
        for (int g0 = 0; g0 < ngroups; g0 += 32) {
            const int g = g0 + lane;
            const int v = g < ngroups ? gsum[g] : 0;
            const int incl = warp_inclusive_scan(v);
            if (g < ngroups) gsum[g] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) misc[33] = carry;
    }
    cluster.sync();  // every CTA's total of owned entries is in its misc[33]
    int base = 0;
    for (int q = 0; q < r; q++) base += cluster.map_shared_rank(misc, q)[33];
    int* cp = col_ptr + slice * (long long)(ncols + 1);
    int* out = row_idx + slice * (long long)rows * K;
    // 3. per group: col_ptr, then every CTA's runs of the group's columns. The
    // group's runs in one CTA are one contiguous block of its rows[] (the
    // columns are consecutive); consecutive lanes read it, and each lane finds
    // its entry's column by a binary search over the lanes' run starts; in a
    // column, CTA q's run follows those of CTAs 0..q-1
    for (int g = warp; g < ngroups; g += kClWarps) {
        const int j = c0 + g * 32 + lane;
        const bool act = j < c1;
        const int last = min(31, c1 - c0 - g * 32 - 1);  // lane of the group's last column
        int bq[kCluster], eq[kCluster], t = 0;
#pragma unroll
        for (int q = 0; q < kCluster; q++) {
            const int* rq = cluster.map_shared_rank(run, q);
            bq[q] = act ? (j > 0 ? rq[j - 1] : 0) : INT_MAX;
            eq[q] = act ? rq[j] : INT_MAX;
            t += act ? eq[q] - bq[q] : 0;
        }
        int dst = base + gsum[g] + warp_inclusive_scan(t) - t;  // this column's next output slot
        if (act) cp[j] = dst;
#pragma unroll
        for (int q = 0; q < kCluster; q++) {
            const int* wq = cluster.map_shared_rank(rws, q);
            const int blk0 = __shfl_sync(0xffffffffu, bq[q], 0);
            const int n = __shfl_sync(0xffffffffu, eq[q], last) - blk0;
            const int shift = act ? dst - bq[q] : 0;  // rows[x] of this column goes to out[x + shift]
            for (int k0 = 0; k0 < n; k0 += 32) {
                const int x = blk0 + k0 + lane;
                int c = 0;  // the last lane whose run starts at or before x
#pragma unroll
                for (int st = 16; st > 0; st >>= 1)
                    if (__shfl_sync(0xffffffffu, bq[q], c + st) <= x) c += st;
                const int sh = __shfl_sync(0xffffffffu, shift, c);
                if (k0 + lane < n) out[x + sh] = wq[x];
            }
            if (act) dst += eq[q] - bq[q];
        }
    }
    if (r == kCluster - 1 && tid == 0) cp[ncols] = base + misc[33];
    cluster.sync();  // no CTA leaves while another still reads its shared memory
}

// Whether the one-kernel transpose serves this shape: its shared memory fits
// and every slice's cluster is resident at once. A second wave of clusters
// doubles its time, and then the multi-kernel form, which spreads the entries
// over every SM, is faster (measured at 512x512 tokens: 16 slices, 15
// resident clusters). The resident-cluster count is asked once per size and
// device.
bool cluster_serves(long long slices, int rows, int K, int ncols, size_t* bytes) {
    const ClLayout L = cl_layout(rows, K, ncols);
    *bytes = L.bytes;
    if (L.bytes > kClSmemMax || (long long)rows * K > INT_MAX) return false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    static std::mutex mu;
    static size_t last_bytes = 0;
    static int last_dev = -1, last_clusters = 0;
    std::lock_guard<std::mutex> lk(mu);
    if (L.bytes != last_bytes || dev != last_dev) {
        last_bytes = L.bytes;
        last_dev = dev;
        last_clusters = 0;
        if (cudaFuncSetAttribute(transpose_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kClSmemMax) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kCluster);
        cfg.blockDim = dim3(kClThreads);
        cfg.dynamicSmemBytes = L.bytes;
        if (cudaOccupancyMaxActiveClusters(&last_clusters, transpose_cluster_kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();
            last_clusters = 0;
        }
    }
    return slices <= last_clusters;
}

}  // namespace

// sel: [slices][rows][K] with entries in [0, ncols). scratch: [slices][ncols].
int launch_transpose(const Shape& s, const int32_t* sel, int rows, int K, int ncols, int32_t* col_ptr,
                     int32_t* row_idx, int32_t* scratch, cudaStream_t st) {
    const int per_slice = rows * K;
    const long long total = s.slices * (long long)per_slice;
    if (s.slices > 0x7fffffffLL) return LLSA_ERR_UNSUPPORTED;
    int* status = status_ptr();
    size_t cl_bytes = 0;
    if (cluster_serves(s.slices, rows, K, ncols, &cl_bytes)) {
        LLSA_LAUNCH("transpose", st,
                    transpose_cluster_kernel<<<(unsigned)(s.slices * kCluster), kClThreads, cl_bytes, st>>>(
                        sel, rows, K, ncols, col_ptr, row_idx, status));
        return LLSA_OK;
    }
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
