// group.cu -- groups of query blocks that share their selected key blocks, the
// work units of the grouped tensor-core attention kernels.
//
// The attention of one query block gathers its K_1 selected key blocks. Query
// blocks whose selections overlap can share one gather: the grouped kernels
// stack up to 8 query blocks (M = 128 query rows) against the union of their
// selections. This pass decides which query blocks go together. It changes
// no result (every query row still attends exactly its own key set), only how
// many key blocks are gathered per query block.
//
// Rule, per (batch, head) slice: each query block i gets an anchor, the
// selected key block j of its row whose bit-reversed index is smallest (a
// MinHash of the selection with the bit-reversal permutation as the hash:
// rows that share most of their blocks usually share the anchor, and of
// blocks spaced along the index the one with the most trailing zero bits
// wins, so overlapping windows of blocks agree on it). Query blocks are
// sorted by (anchor, i); each run of equal anchors is cut into groups of at
// most 8 consecutive entries. The result is deterministic.
//
// Output per slice: order[T] (query blocks in sorted order), gdesc[g] =
// start | count << 16 for group g (its query blocks are order[start ..
// start + count)), ngroups (number of groups).
#include <algorithm>

#include "attn.h"

namespace llsa {
namespace {

constexpr int kGrpThreads = 1024;
constexpr int kIdxBits = 14;  // query and key block indices below 2^14

// Exclusive prefix (sum or max) over the block's threads, one value each.
template <bool kMax>
__device__ int block_exclusive(int v, int* warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x = kMax ? max(x, y) : x + y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t = kMax ? max(t, y) : t + y;
        }
        warp_tot[lane] = t;  // inclusive over warps
    }
    __syncthreads();
    const int before = warp == 0 ? (kMax ? -1 : 0) : warp_tot[warp - 1];
    int ex = __shfl_up_sync(0xffffffffu, x, 1);
    if (lane == 0) ex = kMax ? -1 : 0;
    const int r = kMax ? max(before, ex) : before + ex;
    __syncthreads();  // warp_tot is reused by the next call
    return r;
}

__global__ void __launch_bounds__(kGrpThreads)
group_kernel(const int32_t* __restrict__ sel, int T, int K1, int bits, int Tp, int32_t* __restrict__ order,
             int32_t* __restrict__ gdesc, int32_t* __restrict__ ngroups) {
    extern __shared__ int smem_g[];
    int* key = smem_g;        // Tp sort keys: anchor << 14 | i
    int* gst = smem_g + Tp;   // group starts (T + 1)
    __shared__ int warp_tot[32];
    const long long slice = blockIdx.x;
    const int32_t* srow = sel + slice * (long long)T * K1;
    const int tid = threadIdx.x;

    for (int i = tid; i < Tp; i += kGrpThreads) {
        int k = 0x7FFFFFFF;
        if (i < T) {
            unsigned best = 0xFFFFFFFFu;
            int anc = i;  // a row without a valid entry groups by itself
            for (int c = 0; c < K1; c++) {
                const int j = srow[(long long)i * K1 + c];
                if (j < 0 || j >= T) continue;
                const unsigned h = bits > 0 ? (__brev((unsigned)j) >> (32 - bits)) : 0u;
                if (h < best) {
                    best = h;
                    anc = j;
                }
            }
            k = (anc << kIdxBits) | i;
        }
        key[i] = k;
    }
    __syncthreads();
    // bitonic sort, ascending
    for (int k = 2; k <= Tp; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int idx = tid; idx < (Tp >> 1); idx += kGrpThreads) {
                const int lo = (idx / j) * 2 * j + (idx % j), hi = lo + j;
                const bool up = (lo & k) == 0;
                const int a = key[lo], b = key[hi];
                if ((a > b) == up) {
                    key[lo] = b;
                    key[hi] = a;
                }
            }
            __syncthreads();
        }
    // runs of equal anchors, cut every 8 entries: each thread scans a
    // contiguous segment of the sorted order
    const int per = (T + kGrpThreads - 1) / kGrpThreads;
    const int p0 = min(T, tid * per), p1 = min(T, p0 + per);
    int last_start = -1;
    for (int p = p0; p < p1; p++)
        if (p == 0 || (key[p] >> kIdxBits) != (key[p - 1] >> kIdxBits)) last_start = p;
    const int rs0 = block_exclusive<true>(last_start, warp_tot);  // run start carried into the segment
    int rs = rs0, cnt = 0;
    for (int p = p0; p < p1; p++) {
        if (p == 0 || (key[p] >> kIdxBits) != (key[p - 1] >> kIdxBits)) rs = p;
        if (((p - rs) & 7) == 0) cnt++;
    }
    int gid = block_exclusive<false>(cnt, warp_tot);
    rs = rs0;
    for (int p = p0; p < p1; p++) {
        if (p == 0 || (key[p] >> kIdxBits) != (key[p - 1] >> kIdxBits)) rs = p;
        if (((p - rs) & 7) == 0) gst[gid++] = p;
        order[slice * T + p] = key[p] & ((1 << kIdxBits) - 1);
    }
    // the last thread holding entries knows the total
    if (p1 == T && p0 < p1) {
        gst[gid] = T;
        ngroups[slice] = gid;
    }
    if (T == 0 && tid == 0) ngroups[slice] = 0;
    __syncthreads();
    const int ng = ngroups[slice];
    for (int g = tid; g < ng; g += kGrpThreads)
        gdesc[slice * T + g] = gst[g] | ((gst[g + 1] - gst[g]) << 16);
}

}  // namespace

bool group_supported(const Shape& s) { return s.T >= 1 && s.T <= (1 << kIdxBits); }

size_t group_workspace_bytes(const Shape& s) {
    // order [slices][T], gdesc [slices][T], ngroups [slices]
    return align256(sizeof(int32_t) * (size_t)s.slices * s.T) * 2 + align256(sizeof(int32_t) * (size_t)s.slices);
}

void carve_group_workspace(const Shape& s, void* ws, int32_t** order, int32_t** gdesc, int32_t** ngroups) {
    unsigned char* p = static_cast<unsigned char*>(ws);
    const size_t a = align256(sizeof(int32_t) * (size_t)s.slices * s.T);
    *order = reinterpret_cast<int32_t*>(p);
    *gdesc = reinterpret_cast<int32_t*>(p + a);
    *ngroups = reinterpret_cast<int32_t*>(p + 2 * a);
}

int launch_group(const Shape& s, const int32_t* sel, int32_t* order, int32_t* gdesc, int32_t* ngroups,
                 cudaStream_t st) {
    if (!group_supported(s)) return LLSA_ERR_UNSUPPORTED;
    int Tp = 1, bits = 0;
    while (Tp < s.T) {
        Tp <<= 1;
        bits++;
    }
    const size_t smem = sizeof(int) * ((size_t)Tp + s.T + 1);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return LLSA_ERR_CUDA;
    LLSA_LAUNCH("group", st,
                group_kernel<<<(unsigned)s.slices, kGrpThreads, smem, st>>>(sel, s.T, s.K1, bits, Tp, order, gdesc,
                                                                             ngroups));
    return LLSA_OK;
}

}  // namespace llsa
