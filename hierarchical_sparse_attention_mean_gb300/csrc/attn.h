// attn.h -- arguments and helpers shared by the attention kernels (CUDA-core
// path and tensor-core path).
#pragma once

#include "internal.h"

namespace llsa {

struct AttnArgs {
    const void *q, *k, *v, *o, *dout;
    const float *kpyr, *vpyr;  // K and V pyramids of slice 0
    long long pyr_stride;      // floats per slice pyramid (P * d)
    const int *sel, *coarse, *col_ptr, *row_idx;
    void* out_o;
    float* lse;
    const float* lse_in;
    void *dq, *dk, *dv;
    float *Dbuf, *gK, *gV, *dKc, *dVc;  // backward workspace
    long long slices;
    int n, d, B, L, Le, K1, T, P;
    int side;  // image side under LLSA_ORDER_RASTER (the kernels are instantiated per token order)
    float scale, lnB;
    LevelTable lv;
    int* status;
    int spin;        // polls before a bounded wait gives up (kSpinLimit unless a test lowered it)
    int test_flags;  // LLSA_TEST_* switches of llsa_test_set_wait_limit (0 in normal use)
    // set when the grouping pass ran: its group counts per window (the
    // forwards choose between them from these), else nullptr
    const int32_t* ngroups;
    long long ngroups_n;
    int rule;  // enrichment rule
    // enrichment columns: C per coarse row, Lc used (levels 1..Le); column c
    // holds a token of level col_level[c]; level l owns columns
    // col_off[l] .. col_off[l+1]-1
    int C, Lc;
    unsigned char col_level[kMaxCoarse];
    short col_off[LLSA_MAX_LEVELS + 2];
};

AttnArgs make_attn_args(const Shape& s);
size_t align256(size_t x);
void carve_bwd_workspace(const Shape& s, void* ws, AttnArgs* a);

int launch_fwd_simt(const Shape& s, const AttnArgs& a, cudaStream_t st);
int launch_bwd_dq_simt(const Shape& s, const AttnArgs& a, cudaStream_t st);
int launch_coarse_reduce(const Shape& s, const AttnArgs& a, cudaStream_t st);
int launch_bwd_dkv_simt(const Shape& s, const AttnArgs& a, cudaStream_t st);

// groups of query blocks sharing their selected key blocks (group.cu) and the
// grouped tensor-core forward over them (bf16, B = 16, d = 64, K_1 in {4, 8, 16})
bool group_supported(const Shape& s);
constexpr int kGroupWindow = 1024;  // query blocks per grouping window
int group_windows(const Shape& s);    // grouping windows per slice

// Description of one group of query blocks (group.cu writes one per group at
// the group's gdesc position; the grouped kernels copy it as it is): the
// union U of the group's selected key blocks (ascending), which union blocks
// each of its query blocks selected, the query blocks and their enrichment
// tokens. 512 bytes, 16-byte aligned (copied as 16-byte pieces); indices fit
// 16 bits (T <= 2^14).
struct alignas(16) GroupRec {
    uint32_t mask[8][4];        // bit u % 32 of word u / 32: union block u selected by query block q
    unsigned short uni[128];    // union blocks, ascending (K_1 <= 16: at most 128)
    unsigned short qb[8];       // the group's query blocks
    unsigned short ce[8][4];    // enrichment token of query block q at level l + 1 (l < L_e <= 3)
    int count, nslots;          // query blocks, union blocks
    int slice;
    int pad[9];
};
static_assert(sizeof(GroupRec) == 512 && alignof(GroupRec) == 16, "group record");

// What the grouping needs beyond the selection: the enrichment columns.
struct GroupArgs {
    const int32_t* coarse;  // [slices][T][C]
    int C, Le;
    int col[4];             // column of level l + 1
    int n_level[4];         // tokens of level l + 1
};
size_t group_workspace_bytes(const Shape& s);
void carve_group_workspace(const Shape& s, void* ws, int32_t** order, int32_t** gdesc, int32_t** ngroups,
                           GroupRec** recs);
int launch_group(const Shape& s, const int32_t* sel, const GroupArgs& ga, int32_t* order, int32_t* gdesc,
                 int32_t* ngroups, GroupRec* recs, cudaStream_t st);
bool fwd_grp_supported(const Shape& s);

// Which forward runs after the grouping pass. The grouped forward costs about
// four per-query-block forwards per group (measured on GB300 over inputs
// whose groups average 1.9 to 5.5 query blocks), so it runs when the groups
// hold at least 4.5 query blocks on average, unless a test forces one path.
#ifdef __CUDACC__
__device__ __forceinline__ bool grouped_forward(long long groups, long long blocks, int test_flags) {
    if (test_flags & LLSA_TEST_FORCE_GROUPED) return true;
    if (test_flags & LLSA_TEST_FORCE_PER_BLOCK) return false;
    return 2 * blocks >= 9 * groups;
}

// Sum of n group counts, by one whole warp (every lane gets it).
__device__ __forceinline__ long long sum_groups(const int32_t* ngroups, long long n, int lane) {
    long long tot = 0;
    for (long long u = lane; u < n; u += 32) tot += ngroups[u];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    return tot;
}
#endif
int launch_fwd_grp(const Shape& s, const AttnArgs& a, const int32_t* ngroups, const GroupRec* recs,
                   cudaStream_t st);

// per-query-block tensor-core forward (bf16, B = 16, d in {64, 128} with K_1 in
// {8, 16}, d = 64 with K_1 = 32)
bool fwd_tc_supported(const Shape& s);
int launch_fwd_tc(const Shape& s, const AttnArgs& a, cudaStream_t st);
int launch_bwd_dq_tc(const Shape& s, const AttnArgs& a, cudaStream_t st);
// the tensor-core backward (dQ and dK/dV kernels): bf16, B = 16, d in {64, 128},
// K_1 in {4, 8, 16} (and 32 at d = 64), one enrichment column per level
bool bwd_tc_supported(const Shape& s);
bool bwd_dkv_tc_fits(const Shape& s);
int launch_bwd_dkv_tc(const Shape& s, const AttnArgs& a, cudaStream_t st);

// Adds to the fine-key gradients of column chunk c4 of key block j the
// gradients of the pooled tokens above it: the level-l ancestor of block j is
// j / B^(l-1); each of its B^l fine rows receives 1/B^l of its gradient.
__device__ __forceinline__ void add_pooled_grads(const AttnArgs& a, long long slice, int j, int c4, float* kk,
                                                 float* vv) {
    long long span = a.B;
    int anc = j;
    for (int l = 1; l <= a.Le; l++) {
        const long long off = (slice * a.P + a.lv.row_offset[l] + anc) * (long long)a.d + c4 * 4;
        const float4 gk = *reinterpret_cast<const float4*>(a.dKc + off);
        const float4 gv = *reinterpret_cast<const float4*>(a.dVc + off);
        const float inv = 1.0f / (float)span;
        kk[0] += gk.x * inv; kk[1] += gk.y * inv; kk[2] += gk.z * inv; kk[3] += gk.w * inv;
        vv[0] += gv.x * inv; vv[1] += gv.y * inv; vv[2] += gv.z * inv; vv[3] += gv.w * inv;
        span *= a.B;
        anc /= a.B;
    }
}

}  // namespace llsa
