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
// Rule: each query block i gets an anchor, the selected key block j of its
// row whose bit-reversed index is smallest (a MinHash of the selection with
// the bit-reversal permutation as the hash: rows that share most of their
// blocks usually share the anchor, and of blocks spaced along the index the
// one with the most trailing zero bits wins, so overlapping windows of
// blocks agree on it). Within each window of kGroupWindow consecutive query blocks of
// a slice, the window's blocks are sorted by (anchor, i) and each run of
// equal anchors is cut into groups of at most 8 consecutive entries. The
// result is deterministic. (Windows keep the sort small and the pass wide;
// on the pixel inputs they cost about 1 % more gathered blocks than one sort
// per slice.)
//
// For each group the pass also writes its record (GroupRec): the union of its
// selections, which union blocks each member selected, the members and their
// enrichment tokens, so the grouped kernels copy a group's description as it
// is instead of assembling it on their critical path.
//
// Output, per window u = slice * windows + w covering query blocks
// [w * kGroupWindow, min(T, (w + 1) * kGroupWindow)): order[slice * T + p] for p in that
// range (the window's query blocks in sorted order), gdesc[slice * T + w *
// kGroupWindow + g] = start | count << 16 for its group g (start a position in the
// slice's order), ngroups[u] (number of groups), recs[slice * T + w *
// kGroupWindow + g] (the group's record).
#include <algorithm>

#include "attn.h"

namespace llsa {
namespace {

constexpr int kThr = kGroupWindow < 1024 ? kGroupWindow : 1024;  // threads per grouping CTA
constexpr int kWinE = kGroupWindow / kThr;  // sort keys per thread
constexpr int kIdxBits = 14;  // query and key block indices below 2^14

// Exclusive prefix (sum or max) over the block's threads, one value each.
template <bool kMax>
__device__ int block_exclusive(int v, int* warp_tot) {  // kThr threads
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

// Anchor of query block i: the entry of its selection row with the smallest
// bit-reversed index (invalid entries skipped; none valid: the block itself).
template <int K1>
__device__ __forceinline__ int anchor_of(const int32_t* row, int i, int T, int bits) {
    unsigned best = 0xFFFFFFFFu;
    int anc = i;
    int v[K1];
#pragma unroll
    for (int c = 0; c < K1; c += 4) {
        const int4 q = *reinterpret_cast<const int4*>(row + c);
        v[c] = q.x; v[c + 1] = q.y; v[c + 2] = q.z; v[c + 3] = q.w;
    }
#pragma unroll
    for (int c = 0; c < K1; c++) {
        const int j = v[c];
        if (j < 0 || j >= T) continue;
        const unsigned h = bits > 0 ? (__brev((unsigned)j) >> (32 - bits)) : 0u;
        if (h < best) {
            best = h;
            anc = j;
        }
    }
    return anc;
}

__device__ __forceinline__ int anchor_generic(const int32_t* row, int K1, int i, int T, int bits) {
    unsigned best = 0xFFFFFFFFu;
    int anc = i;
    for (int c = 0; c < K1; c++) {
        const int j = row[c];
        if (j < 0 || j >= T) continue;
        const unsigned h = bits > 0 ? (__brev((unsigned)j) >> (32 - bits)) : 0u;
        if (h < best) {
            best = h;
            anc = j;
        }
    }
    return anc;
}

// Raw loads of one group: its selection entries (element r * 32 + lane of
// the count * KK entries) and enrichment tokens (lane = query block * 4 + level).
template <int KK>
struct RecLoads {
    static constexpr int RR = 8 * KK / 32;
    int g0, count, qb;
    int v[RR];
    int ce;
};

template <int KK>
__device__ __forceinline__ void rec_load(RecLoads<KK>& L, int g, int ng, int lane, const int* gst, const int* key_s,
                                         const int32_t* srow, long long slice, int T, const GroupArgs& ga) {
    L.count = 0;
    if (g >= ng) return;
    L.g0 = gst[g];
    L.count = gst[g + 1] - L.g0;
    L.qb = lane < L.count ? (key_s[L.g0 + lane] & ((1 << kIdxBits) - 1)) : 0;
#pragma unroll
    for (int r = 0; r < RecLoads<KK>::RR; r++) {
        const int e = r * 32 + lane, qs = e / KK, c = e % KK;
        const int qb = __shfl_sync(0xffffffffu, L.qb, qs & 7);
        L.v[r] = qs < L.count ? srow[(long long)qb * KK + c] : -2;
    }
    const int qs = lane >> 2, l = lane & 3;
    const int qb = __shfl_sync(0xffffffffu, L.qb, qs);
    L.ce = (qs < L.count && l < ga.Le) ? ga.coarse[(slice * T + qb) * ga.C + ga.col[l]] : 0;
}

template <int KK>
__device__ void records(int warp, int lane, int ng, const int* gst, const int* key_s, const int32_t* srow,
                        long long slice, int T, int i0, const GroupArgs& ga, GroupRec* recs, int* status,
                        GroupRec& R) {
    constexpr int RR = RecLoads<KK>::RR, NE = RR * 32;
    RecLoads<KK> cur, nxt;
    rec_load<KK>(cur, warp, ng, lane, gst, key_s, srow, slice, T, ga);
    for (int g = warp; g < ng; g += kThr / 32) {
        rec_load<KK>(nxt, g + kThr / 32, ng, lane, gst, key_s, srow, slice, T, ga);
        const int count = cur.count;
        (&R.mask[0][0])[lane] = 0u;
        int v[RR];
#pragma unroll
        for (int r = 0; r < RR; r++) {
            const int qs = (r * 32 + lane) / KK;
            int jb = cur.v[r];
            v[r] = 0x7FFFFFFF;
            if (qs < count) {
                if (jb < 0 || jb >= T) {
                    if (status) atomicCAS(status, 0, LLSA_ERR_BAD_INDEX);
                    jb = 0;
                }
                v[r] = (jb << 3) | qs;
            }
        }
#pragma unroll
        for (int kk = 2; kk <= NE; kk <<= 1)
#pragma unroll
            for (int jj = kk >> 1; jj > 0; jj >>= 1) {
                if (jj >= 32) {
                    const int rj = jj >> 5;
#pragma unroll
                    for (int r = 0; r < RR; r++)
                        if ((r & rj) == 0) {
                            const bool up = ((r * 32 + lane) & kk) == 0;
                            const int x = v[r], y = v[r + rj];
                            if ((x > y) == up) {
                                v[r] = y;
                                v[r + rj] = x;
                            }
                        }
                } else {
#pragma unroll
                    for (int r = 0; r < RR; r++) {
                        const int y = __shfl_xor_sync(0xffffffffu, v[r], jj);
                        const bool lower = (lane & jj) == 0;
                        const bool up = ((r * 32 + lane) & kk) == 0;
                        v[r] = (lower == up) ? min(v[r], y) : max(v[r], y);
                    }
                }
            }
        __syncwarp();
        int base = 0;
#pragma unroll
        for (int r = 0; r < RR; r++) {
            int prev = __shfl_up_sync(0xffffffffu, v[r], 1);
            const int last_prev = __shfl_sync(0xffffffffu, v[r > 0 ? r - 1 : 0], 31);
            if (lane == 0) prev = r > 0 ? last_prev : -1;
            const bool valid = v[r] != 0x7FFFFFFF;
            const bool first = valid && (prev < 0 || (prev >> 3) != (v[r] >> 3));
            const unsigned fm = __ballot_sync(0xffffffffu, first);
            const int slot = base + __popc(fm & (0xFFFFFFFFu >> (31 - lane))) - 1;
            if (first) R.uni[slot] = (unsigned short)(v[r] >> 3);
            if (valid) atomicOr(&R.mask[v[r] & 7][slot >> 5], 1u << (slot & 31));
            base += __popc(fm);
        }
        {
            const int qs = lane >> 2, l = lane & 3;
            int e = cur.ce;
            if (qs < count && l < ga.Le && (e < 0 || e >= ga.n_level[l])) {
                if (status) atomicCAS(status, 0, LLSA_ERR_BAD_INDEX);
                e = 0;
            }
            R.ce[qs][l] = (unsigned short)e;
        }
        if (lane < 8) R.qb[lane] = (unsigned short)cur.qb;
        if (lane == 0) {
            R.count = count;
            R.nslots = base;
            R.slice = (int)slice;
        }
        __syncwarp();
        reinterpret_cast<uint4*>(recs + slice * T + i0 + g)[lane] = reinterpret_cast<const uint4*>(&R)[lane];
        __syncwarp();
        cur = nxt;
    }
}

// One CTA of kThr threads per window of E * kThr query blocks; element e =
// thread * E + r of the window's sort keys sits in register r of a thread.
template <int E>
__global__ void __launch_bounds__(kThr)
group_kernel(const int32_t* __restrict__ sel, int T, int K1, int bits, int windows, GroupArgs gargs,
             int32_t* __restrict__ order, int32_t* __restrict__ gdesc, int32_t* __restrict__ ngroups,
             GroupRec* __restrict__ recs, int* status) {
    constexpr int W = E * kThr;
    __shared__ int key_s[W];
    __shared__ int gst[W + 1];
    __shared__ GroupRec rec_s[kThr / 32];
    __shared__ int warp_tot[32];
    __shared__ int total_s;
    const long long unit = blockIdx.x;
    const long long slice = unit / windows;
    const int i0 = (int)(unit % windows) * W;
    const int nw = min(W, T - i0);
    const int32_t* srow = sel + slice * (long long)T * K1;
    const int tid = threadIdx.x, lane = tid & 31;

    int key[E];
#pragma unroll
    for (int r = 0; r < E; r++) {
        const int e = tid * E + r;
        key[r] = 0x7FFFFFFF;
        if (e < nw) {
            const int i = i0 + e;
            const int32_t* row = srow + (long long)i * K1;
            const int anc = K1 == 4 ? anchor_of<4>(row, i, T, bits)
                            : K1 == 8 ? anchor_of<8>(row, i, T, bits)
                            : K1 == 16 ? anchor_of<16>(row, i, T, bits)
                                       : anchor_generic(row, K1, i, T, bits);
            key[r] = (anc << kIdxBits) | i;
        }
    }
    // bitonic sort, ascending: strides below E inside a thread, below 32 E
    // across lanes, larger ones through shared memory
    for (int k = 2; k <= W; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j < E) {
#pragma unroll
                for (int r = 0; r < E; r++) {
                    const int rp = r ^ j;
                    if (rp > r) {
                        const bool up = ((tid * E + r) & k) == 0;
                        const int x = key[r], y = key[rp];
                        if ((x > y) == up) {
                            key[r] = y;
                            key[rp] = x;
                        }
                    }
                }
            } else if (j < 32 * E) {
                const bool lower = (lane & (j / E)) == 0;
#pragma unroll
                for (int r = 0; r < E; r++) {
                    const bool up = ((tid * E + r) & k) == 0;
                    const int y = __shfl_xor_sync(0xffffffffu, key[r], j / E);
                    key[r] = (lower == up) ? min(key[r], y) : max(key[r], y);
                }
            } else {
#pragma unroll
                for (int r = 0; r < E; r++) key_s[tid * E + r] = key[r];
                __syncthreads();
#pragma unroll
                for (int r = 0; r < E; r++) {
                    const int e = tid * E + r;
                    const bool up = (e & k) == 0, lower = (e & j) == 0;
                    const int y = key_s[e ^ j];
                    key[r] = (lower == up) ? min(key[r], y) : max(key[r], y);
                }
                __syncthreads();
            }
        }
#pragma unroll
    for (int r = 0; r < E; r++) key_s[tid * E + r] = key[r];
    __syncthreads();
    // runs of equal anchors, cut every 8 entries; each thread scans its E
    // positions of the window's sorted order
    const int p0 = min(nw, tid * E), p1 = min(nw, p0 + E);
    int last_start = -1;
    for (int p = p0; p < p1; p++)
        if (p == 0 || (key_s[p] >> kIdxBits) != (key_s[p - 1] >> kIdxBits)) last_start = p;
    const int rs0 = block_exclusive<true>(last_start, warp_tot);  // run start carried into the segment
    int rs = rs0, cnt = 0;
    for (int p = p0; p < p1; p++) {
        if (p == 0 || (key_s[p] >> kIdxBits) != (key_s[p - 1] >> kIdxBits)) rs = p;
        if (((p - rs) & 7) == 0) cnt++;
    }
    int gid = block_exclusive<false>(cnt, warp_tot);
    rs = rs0;
    for (int p = p0; p < p1; p++) {
        if (p == 0 || (key_s[p] >> kIdxBits) != (key_s[p - 1] >> kIdxBits)) rs = p;
        if (((p - rs) & 7) == 0) gst[gid++] = p;
        order[slice * T + i0 + p] = key_s[p] & ((1 << kIdxBits) - 1);
    }
    if (p1 == nw && p0 < p1) {
        gst[gid] = nw;
        total_s = gid;
        ngroups[unit] = gid;
    }
    __syncthreads();
    const int ng = total_s;
    for (int g = tid; g < ng; g += kThr) gdesc[slice * T + i0 + g] = (i0 + gst[g]) | ((gst[g + 1] - gst[g]) << 16);
    // each group's record, one warp per group: the union of its selections
    // (entries value << 3 | query block, sorted; the first of each run of
    // equal blocks is a union block), the masks, the enrichment tokens. The
    // next group's selection rows and tokens are loaded before this one is
    // sorted, so the loads overlap the work.
    const int warp = tid >> 5;
    GroupRec& R = rec_s[warp];
    if (K1 == 4) records<4>(warp, lane, ng, gst, key_s, srow, slice, T, i0, gargs, recs, status, R);
    else if (K1 == 8) records<8>(warp, lane, ng, gst, key_s, srow, slice, T, i0, gargs, recs, status, R);
    else records<16>(warp, lane, ng, gst, key_s, srow, slice, T, i0, gargs, recs, status, R);
}

}  // namespace

bool group_supported(const Shape& s) { return s.T >= 1 && s.T <= (1 << kIdxBits) && (s.K1 == 4 || s.K1 == 8 || s.K1 == 16) && s.Le <= 4; }

size_t group_workspace_bytes(const Shape& s) {
    // order [slices][T], gdesc [slices][T], ngroups [slices][windows], records [slices][T]
    const size_t windows = (size_t)group_windows(s);
    return align256(sizeof(int32_t) * (size_t)s.slices * s.T) * 2 +
           align256(sizeof(int32_t) * (size_t)s.slices * windows) + sizeof(GroupRec) * (size_t)s.slices * s.T;
}

void carve_group_workspace(const Shape& s, void* ws, int32_t** order, int32_t** gdesc, int32_t** ngroups,
                           GroupRec** recs) {
    unsigned char* p = static_cast<unsigned char*>(ws);
    const size_t a = align256(sizeof(int32_t) * (size_t)s.slices * s.T);
    const size_t b = align256(sizeof(int32_t) * (size_t)s.slices * group_windows(s));
    *order = reinterpret_cast<int32_t*>(p);
    *gdesc = reinterpret_cast<int32_t*>(p + a);
    *ngroups = reinterpret_cast<int32_t*>(p + 2 * a);
    *recs = reinterpret_cast<GroupRec*>(p + 2 * a + b);
}

int group_windows(const Shape& s) { return (s.T + kGroupWindow - 1) / kGroupWindow; }

int launch_group(const Shape& s, const int32_t* sel, const GroupArgs& ga, int32_t* order, int32_t* gdesc,
                 int32_t* ngroups, GroupRec* recs, cudaStream_t st) {
    if (!group_supported(s)) return LLSA_ERR_UNSUPPORTED;
    int bits = 0;
    while ((1 << bits) < s.T) bits++;
    const int windows = group_windows(s);
    LLSA_LAUNCH("group", st,
                group_kernel<kWinE><<<(unsigned)(s.slices * windows), kThr, 0, st>>>(
                    sel, s.T, s.K1, bits, windows, ga, order, gdesc, ngroups, recs, status_ptr()));
    return LLSA_OK;
}

}  // namespace llsa
