// attn_fwd_tc.cu -- block-sparse attention forward with KV enrichment on the
// tcgen05 tensor cores (bf16 in, fp32 accumulate), for B = 16, d in {64, 128}
// and K_1 in {8, 16} (128 or 256 fine keys per query block), and K_1 = 32 at
// d = 64 (512 keys: four key tiles, one ring stage).
//
// Method: Pith review of arXiv 2512.16615, "Core claim": every query block of
// B tokens attends the B tokens of its K selected blocks plus one pooled K/V
// token per level with weight B^l (logit + ln B^l, KV Reweighting).
//
// A query block has only 16 queries but 128 or 256 keys, so the contraction
// runs key-major: S^T = K_sel Q^T (M = 128 keys per tile, N = 16, K = d) and
// O^T = V_sel^T P^T (M = d, N = 16, K = keys). All keys of a block are in one
// pass, so the softmax is exact (no online rescaling): the max and the sum over
// the block's K*B fine keys and L_e pooled keys are reduced across the 128
// threads of a warpgroup (one key per thread and tile, 16 query columns each).
//
// Warp roles (persistent CTAs, one per SM, query blocks strided over CTAs):
//   warps 0, 2, 3  gather, each for every third block: the Q block and the K_1
//                  selected K and V blocks as 16-row TMA boxes (128-byte
//                  swizzle, the layout the MMA descriptors describe) and the
//                  pooled K/V rows as bulk copies, into a ring of stages;
//   warp 1         TMEM owner and MMA issuer (one thread);
//   warps 4-7,     two softmax/epilogue warpgroups taking alternate query
//   warps 8-11     blocks, each with its own S and O columns in TMEM.
// Every mbarrier wait is bounded; a timeout records LLSA_ERR_TIMEOUT and the
// CTA drains and exits.
//
// Where the grouped forward (attn_fwd_grp.cu) also applies, both are launched
// after the grouping pass and these kernels return at once when the groups
// are large enough for it (AttnArgs::ngroups; the rule is grouped_forward).
//
// Token order: each kernel is built for the tile order and for the raster order
// of a square image (index reordering, referee comments on Sec. 5.1 and
// Figure 2): in the latter a block's tokens come in as one 4 x 4 patch (a 4-D
// TMA box landing in the same swizzled layout) and its output rows go back to
// the patch's pixels; the arithmetic is the same.
#include <algorithm>

#include "attn.h"
#include "tc.cuh"

namespace llsa {
namespace {

using namespace tc;

constexpr int kThreads = 384;
constexpr int kSmemBudget = 215 * 1024;
constexpr float kLog2e = 1.4426950408889634f;

template <int D, int NT>
struct Cfg {
    static constexpr int NF = NT * 128;          // fine keys per query block
    static constexpr int REG = D / 64;           // 64-column regions of a row
    static constexpr int CH = D / 8;             // 16-byte chunks per bf16 row
    static constexpr int Q_BYTES = 16 * D * 2;
    static constexpr int KV_BYTES = NF * D * 2;
    static constexpr int CO_BYTES = 2 * 4 * D * 4;  // pooled K and V rows (fp32), up to 4 levels
    static constexpr int STAGE_BYTES = Q_BYTES + 2 * KV_BYTES + CO_BYTES;
    static constexpr int P_BYTES = 16 * NF * 2;  // per warpgroup
    static constexpr int FIXED = 2 * P_BYTES + 4096;
    static constexpr int STAGES_RAW = (kSmemBudget - FIXED) / STAGE_BYTES;
    // gather warps, each owning SPP stages of its own (so every stage barrier
    // is waited on in order and a parity can never match an older phase)
    static constexpr int NPROD = STAGES_RAW >= 3 ? 3 : (STAGES_RAW >= 2 ? 2 : 1);
    static constexpr int SPP = (STAGES_RAW < 1 ? 1 : (STAGES_RAW > 6 ? 6 : STAGES_RAW)) / NPROD;
    static constexpr int STAGES = NPROD * SPP;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + FIXED;
    // TMEM columns per warpgroup: S at +0 (16 per key tile), O after it
    static constexpr int TM_O = NT <= 2 ? 32 : NT * 16;
    static constexpr int TM_GROUP = NT <= 2 ? 64 : 128;
    static constexpr int TM_ALLOC = 2 * TM_GROUP;
};

// Block bl of a CTA goes to gather warp bl % NPROD; within that warp's
// sequence (k = bl / NPROD) it takes the warp's stage k % SPP for use k / SPP.
template <class C>
__device__ __forceinline__ void stage_of(int bl, int& st, int& u) {
    const int k = bl / C::NPROD;
    st = (bl % C::NPROD) * C::SPP + k % C::SPP;
    u = k / C::SPP;
}

struct Misc {
    float red_max[2][16][4];  // [group][query][warp]
    float red_sum[2][16][4];
    float cs[2][16][4];       // pooled-key scores (scaled, + ln B^l), -inf beyond L_e
    float ecs[2][16][4];      // coarse probabilities exp(cs - lse), 0 beyond L_e
    float mfin[2][16];        // row maximum times log2(e)
    float izfin[2][16];       // 1 / row sum
    uint64_t full[6], empty[6], q_ready[2], s_full[2], p_full[2], o_full[2], s_free[2], o_free[2], drain;
    uint32_t tmem_slot;
    int abort_flag;
};

template <int D, int NT, bool R>
__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
              const __grid_constant__ CUtensorMap mv, AttnArgs a) {
    using C = Cfg<D, NT>;
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned base (128-byte swizzle atoms), derived from the
    // __shared__ array by pointer arithmetic so accesses stay shared-space
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* stages = sm;
    unsigned char* pbuf = stages + C::STAGES * C::STAGE_BYTES;
    Misc* ms = reinterpret_cast<Misc*>(pbuf + 2 * C::P_BYTES);
    volatile int* abort_flag = &ms->abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long total = a.slices * (long long)a.T;
    const int G = gridDim.x;
    const int K1 = NT * 8, Le = a.Le;
    // after a grouping pass, the grouped forward may take this call instead
    if (a.ngroups != nullptr) {
        bool skip = false;
        if (warp == 0) {
            const long long groups = sum_groups(a.ngroups, a.ngroups_n, lane);
            skip = lane == 0 && grouped_forward(groups, total, a.test_flags);
        }
        if (__syncthreads_or(skip)) return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; s++) {
            mbar_init(smem_u32(&ms->full[s]), 1);
            mbar_init(smem_u32(&ms->empty[s]), 1);
        }
        for (int w = 0; w < 2; w++) {
            mbar_init(smem_u32(&ms->q_ready[w]), 1);
            mbar_init(smem_u32(&ms->s_full[w]), 1);
            mbar_init(smem_u32(&ms->p_full[w]), 128);
            mbar_init(smem_u32(&ms->o_full[w]), 1);
            mbar_init(smem_u32(&ms->s_free[w]), 128);
            mbar_init(smem_u32(&ms->o_free[w]), 128);
        }
        mbar_init(smem_u32(&ms->drain), 1);
        ms->abort_flag = 0;
        fence_mbar_init();
    }
    for (int x = threadIdx.x; x < 2 * 16 * 4; x += kThreads) {
        (&ms->cs[0][0][0])[x] = -INFINITY;
        (&ms->ecs[0][0][0])[x] = 0.f;
    }
    if (warp == 1) tmem_alloc(smem_u32(&ms->tmem_slot), C::TM_ALLOC);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = ms->tmem_slot;

    if ((warp == 0 || warp == 2 || warp == 3) && (warp == 0 ? 0 : warp - 1) < C::NPROD) {
        // ----------------------------------------------------------- gather
        // NPROD warps issue the copies, each for every NPROD-th block: the Q
        // block, the K_1 selected K and V blocks (one 16-row TMA box each) and
        // the pooled K/V rows (1D bulk copies). Index rows are loaded two of
        // the warp's blocks ahead so their latency overlaps earlier copies.
        const int pw = warp == 0 ? 0 : warp - 1;
        auto load_idx = [&](int bl, int& jb, int& ce) {
            const long long g = blockIdx.x + (long long)bl * G;
            jb = 0;
            ce = 0;
            if (g >= total) return;
            const long long slice = g / a.T;
            const int i = (int)(g - slice * a.T);
            if (lane < K1) jb = a.sel[(slice * a.T + i) * a.K1 + lane];
            if (lane < Le) ce = a.coarse[(slice * a.T + i) * a.C + lane];
        };
        int jb0, ce0, jb1, ce1;
        load_idx(pw, jb0, ce0);
        load_idx(pw + C::NPROD, jb1, ce1);
        int issued = -1;
        for (int bl = pw;; bl += C::NPROD) {
            const long long g = blockIdx.x + (long long)bl * G;
            if (g >= total || (a.test_flags & LLSA_TEST_NO_COPIES)) break;
            int jb = jb0, e = ce0;
            jb0 = jb1;
            ce0 = ce1;
            load_idx(bl + 2 * C::NPROD, jb1, ce1);
            int st, u;
            stage_of<C>(bl, st, u);
            bool ok = true;
            if (u >= 1 && lane == 0) ok = mbar_wait(smem_u32(&ms->empty[st]), (u - 1) & 1, abort_flag, a.status, a.spin);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0);
            if (!ok) break;
            const long long slice = g / a.T;
            const int i = (int)(g - slice * a.T);
            unsigned char* sQ = stages + st * C::STAGE_BYTES;
            unsigned char* sK = sQ + C::Q_BYTES;
            unsigned char* sV = sK + C::KV_BYTES;
            unsigned char* sC = sV + C::KV_BYTES;
            const uint32_t fb = smem_u32(&ms->full[st]);
            if (lane == 0) mbar_arrive_expect_tx(fb, C::STAGE_BYTES - C::CO_BYTES + 2 * Le * D * 4);
            __syncwarp();
            if (lane == 0) {
                const int yq = (int)(slice * a.n + (long long)i * 16);
                for (int r = 0; r < C::REG; r++) {
                    if constexpr (R) tma_load_block<true>(smem_u32(sQ + r * 16 * 128), &mq, r * 64, slice, i, a.n, fb);
                    else tma_load_2d(smem_u32(sQ + r * 16 * 128), &mq, r * 64, yq, fb);
                }
            }
            if (lane < K1) {
                if (jb < 0 || jb >= a.T) {
                    set_status(a.status, LLSA_ERR_BAD_INDEX);
                    jb = 0;
                }
                const int yk = R ? jb : (int)(slice * a.n + (long long)jb * 16);
                for (int r = 0; r < C::REG; r++) {
                    if constexpr (R) {
                        tma_load_block<true>(smem_u32(sK + r * C::NF * 128 + lane * 2048), &mk, r * 64, slice, yk, a.n, fb);
                        tma_load_block<true>(smem_u32(sV + r * C::NF * 128 + lane * 2048), &mv, r * 64, slice, yk, a.n, fb);
                    } else {
                        tma_load_2d(smem_u32(sK + r * C::NF * 128 + lane * 2048), &mk, r * 64, yk, fb);
                        tma_load_2d(smem_u32(sV + r * C::NF * 128 + lane * 2048), &mv, r * 64, yk, fb);
                    }
                }
            }
            if (lane < Le) {
                if (e < 0 || e >= a.lv.n_level[lane + 1]) {
                    set_status(a.status, LLSA_ERR_BAD_INDEX);
                    e = 0;
                }
                const long long row = slice * a.pyr_stride + (long long)(a.lv.row_offset[lane + 1] + e) * D;
                bulk_load(smem_u32(sC + lane * D * 4), a.kpyr + row, D * 4, fb);
                bulk_load(smem_u32(sC + (4 + lane) * D * 4), a.vpyr + row, D * 4, fb);
            }
            issued = bl;
        }
        // the copies of this warp's last block per stage must land before exit
        if (lane == 0)
            for (int bl = issued; bl >= 0 && bl > issued - C::NPROD * C::SPP; bl -= C::NPROD) {
                int st, u;
                stage_of<C>(bl, st, u);
                for (int it = 0; it < kSpinLimit && !mbar_try(smem_u32(&ms->full[st]), u & 1); it++) {
                }
            }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16(128, 16, 0, 0);
            constexpr uint32_t idPV = idesc_bf16(D, 16, 1, 0);
            // descriptors of the ring's base; operands add (offset >> 4)
            const uint64_t dKQ = desc_sw128(smem_u32(stages), 16, 1024);          // K-major
            const uint64_t dV = desc_sw128(smem_u32(stages), C::NF * 128, 1024);  // MN-major V
            const uint64_t dP = desc_sw128(smem_u32(pbuf), 16, 1024);
            auto issue_S = [&](int bl) -> bool {
                const int w = bl & 1, j = bl >> 1;
                int st, u;
                stage_of<C>(bl, st, u);
                if (!mbar_wait(smem_u32(&ms->full[st]), u & 1, abort_flag, a.status, a.spin)) return false;
                mbar_arrive(smem_u32(&ms->q_ready[w]));  // the group may read Q and pooled rows
                // S columns of this group: free once the group has read its previous S
                if (j >= 1 && !mbar_wait(smem_u32(&ms->s_free[w]), (j - 1) & 1, abort_flag, a.status, a.spin)) return false;
                tc_fence_after();
                const uint32_t q0 = (uint32_t)(st * C::STAGE_BYTES), k0 = q0 + C::Q_BYTES;
#pragma unroll
                for (int t = 0; t < NT; t++)
#pragma unroll
                    for (int ks = 0; ks < D / 16; ks++)
                        mma_bf16(tbase + w * C::TM_GROUP + t * 16,
                                 dKQ + ((k0 + (ks / 4) * C::NF * 128 + t * 128 * 128 + (ks % 4) * 32) >> 4),
                                 dKQ + ((q0 + (ks / 4) * 16 * 128 + (ks % 4) * 32) >> 4), idS, ks > 0);
                mma_commit(smem_u32(&ms->s_full[w]));
                return true;
            };
            auto issue_PV = [&](int bl) -> bool {
                const int w = bl & 1, j = bl >> 1;
                int st, u;
                stage_of<C>(bl, st, u);
                if (!mbar_wait(smem_u32(&ms->p_full[w]), j & 1, abort_flag, a.status, a.spin)) return false;
                if (j >= 1 && !mbar_wait(smem_u32(&ms->o_free[w]), (j - 1) & 1, abort_flag, a.status, a.spin)) return false;
                tc_fence_after();
                const uint32_t v0 = (uint32_t)(st * C::STAGE_BYTES + C::Q_BYTES + C::KV_BYTES);
                const uint32_t p0 = (uint32_t)(w * C::P_BYTES);
#pragma unroll
                for (int ks = 0; ks < C::NF / 16; ks++)
                    mma_bf16(tbase + w * C::TM_GROUP + C::TM_O, dV + ((v0 + ks * 2048) >> 4),
                             dP + ((p0 + (ks / 4) * 2048 + (ks % 4) * 32) >> 4), idPV, ks > 0);
                mma_commit(smem_u32(&ms->o_full[w]));
                mma_commit(smem_u32(&ms->empty[st]));
                return true;
            };
            const long long mine = total > blockIdx.x ? (total - blockIdx.x + G - 1) / G : 0;
            bool ok = true;
            if (C::STAGES >= 2) {
                // S of the next block goes ahead of P V of this one, so the other
                // warpgroup's softmax overlaps this one's
                ok = mine > 0 ? issue_S(0) : true;
                for (long long bl = 0; ok && bl < mine; bl++) {
                    if (bl + 1 < mine) ok = issue_S((int)bl + 1);
                    if (ok) ok = issue_PV((int)bl);
                }
            } else {
                // one stage: the next block's operands arrive only after P V frees it
                for (long long bl = 0; ok && bl < mine; bl++) {
                    ok = issue_S((int)bl);
                    if (ok) ok = issue_PV((int)bl);
                }
            }
            // no MMA may be in flight when TMEM is released
            mma_commit(smem_u32(&ms->drain));
            for (int it = 0; it < kSpinLimit && !mbar_try(smem_u32(&ms->drain), 0); it++) {
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ----------------------------------------- softmax + epilogue groups
        const int w = (warp - 4) >> 2, qr = warp & 3;
        const int tw = threadIdx.x - 128 * (1 + w);
        const uint32_t tS = tbase + w * C::TM_GROUP + ((uint32_t)(qr * 32) << 16);
        const uint32_t tO = tS + C::TM_O;
        const float sc = a.scale, scl2 = a.scale * kLog2e;
        const int dd = D == 64 ? 16 * qr + lane : 32 * qr + lane;  // O^T row this thread reads back
        const bool valid = D == 64 ? lane < 16 : true;
        // pooled-key score pairs: two threads per (query, level)
        const int pi = tw >> 1, half = tw & 1;
        const bool pact = pi < 16 * Le;
        const int pq = pact ? pi / Le : 0, pl = pact ? pi % Le : 0;
        unsigned char* P = pbuf + w * C::P_BYTES;
        for (int bl = w;; bl += 2) {
            const long long g = blockIdx.x + (long long)bl * G;
            if (g >= total) break;
            const int j = bl >> 1;
            int st, u;
            stage_of<C>(bl, st, u);
            const long long slice = g / a.T;
            const int i = (int)(g - slice * a.T);
            const unsigned char* sQ = stages + st * C::STAGE_BYTES;
            const float* sCk = reinterpret_cast<const float*>(sQ + C::Q_BYTES + 2 * C::KV_BYTES);
            // After a timeout every later wait returns at once; the group keeps
            // walking the same barriers so no thread is left waiting on another.
            // q_ready (set by the MMA thread once it has seen the stage full) is
            // per group and in order; waiting on the stage barrier itself could
            // alias an older phase when stages are few.
            mbar_wait(smem_u32(&ms->q_ready[w]), j & 1, abort_flag, a.status, a.spin);
            {
                float acc0 = 0.f, acc1 = 0.f;
                if (pact) {
                    const float* kc = sCk + pl * D;
#pragma unroll
                    for (int c8 = half * C::CH / 2; c8 < (half + 1) * C::CH / 2; c8++) {
                        const uint4 raw = *reinterpret_cast<const uint4*>(sQ + sw128_offset(pq, c8 * 8, 16));
                        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
                        const float4 k0 = *reinterpret_cast<const float4*>(kc + c8 * 8);
                        const float4 k1 = *reinterpret_cast<const float4*>(kc + c8 * 8 + 4);
                        const float2 x0 = __bfloat1622float2(h[0]), x1 = __bfloat1622float2(h[1]);
                        const float2 x2 = __bfloat1622float2(h[2]), x3 = __bfloat1622float2(h[3]);
                        acc0 = fmaf(x0.x, k0.x, acc0); acc1 = fmaf(x0.y, k0.y, acc1);
                        acc0 = fmaf(x1.x, k0.z, acc0); acc1 = fmaf(x1.y, k0.w, acc1);
                        acc0 = fmaf(x2.x, k1.x, acc0); acc1 = fmaf(x2.y, k1.y, acc1);
                        acc0 = fmaf(x3.x, k1.z, acc0); acc1 = fmaf(x3.y, k1.w, acc1);
                    }
                }
                float sum = acc0 + acc1;
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                if (pact && half == 0) ms->cs[w][pq][pl] = sc * sum + (float)(pl + 1) * a.lnB;
            }
            // this thread's column of the pooled V rows, read while the stage is held
            float vc[4];
#pragma unroll
            for (int l = 0; l < 4; l++) vc[l] = (l < Le && valid) ? sCk[(4 + l) * D + dd] : 0.f;

            mbar_wait(smem_u32(&ms->s_full[w]), j & 1, abort_flag, a.status, a.spin);
            tc_fence_after();
            float s[NT][16];
#pragma unroll
            for (int t = 0; t < NT; t++) tmem_ld16(tS + t * 16, s[t]);
            tc_fence_before();
            mbar_arrive(smem_u32(&ms->s_free[w]));
            float x[16];
#pragma unroll
            for (int c = 0; c < 16; c++) {
                x[c] = s[0][c];
#pragma unroll
                for (int t = 1; t < NT; t++) x[c] = fmaxf(x[c], s[t][c]);
            }
            float r = warp_reduce16<true>(x, lane);
            if (!(lane & 1)) ms->red_max[w][lane >> 1][qr] = r;
            named_barrier(1 + w, 128);
            // row maxima over the fine keys (raw scores, then scaled) and the
            // pooled keys, one row per thread of the first 16
            if (tw < 16) {
                const float4 rm = *reinterpret_cast<const float4*>(ms->red_max[w][tw]);
                const float4 cz = *reinterpret_cast<const float4*>(ms->cs[w][tw]);
                ms->mfin[w][tw] = fmaxf(fmaxf(fmaxf(rm.x, rm.y), fmaxf(rm.z, rm.w)) * sc,
                                        fmaxf(fmaxf(cz.x, cz.y), fmaxf(cz.z, cz.w))) * kLog2e;
            }
            named_barrier(1 + w, 128);
            float mo[16];
#pragma unroll
            for (int c = 0; c < 16; c += 4) {
                const float4 v = *reinterpret_cast<const float4*>(&ms->mfin[w][c]);
                mo[c] = v.x; mo[c + 1] = v.y; mo[c + 2] = v.z; mo[c + 3] = v.w;
            }
#pragma unroll
            for (int c = 0; c < 16; c++) {
                x[c] = 0.f;
#pragma unroll
                for (int t = 0; t < NT; t++) {
                    s[t][c] = ex2(fmaf(s[t][c], scl2, -mo[c]));
                    x[c] += s[t][c];
                }
            }
            r = warp_reduce16<false>(x, lane);
            if (!(lane & 1)) ms->red_sum[w][lane >> 1][qr] = r;
            named_barrier(1 + w, 128);
            if (tw < 16) {
                // z >= 1 (the maximum contributes exp(0)), so the approximate
                // reciprocal is safe
                const float4 rs = *reinterpret_cast<const float4*>(ms->red_sum[w][tw]);
                const float4 cz = *reinterpret_cast<const float4*>(ms->cs[w][tw]);
                const float m2 = ms->mfin[w][tw];
                const float e0 = ex2(fmaf(cz.x, kLog2e, -m2)), e1 = ex2(fmaf(cz.y, kLog2e, -m2));
                const float e2 = ex2(fmaf(cz.z, kLog2e, -m2)), e3 = ex2(fmaf(cz.w, kLog2e, -m2));
                const float z = ((rs.x + rs.y) + (rs.z + rs.w)) + ((e0 + e1) + (e2 + e3));
                const float iz = rcp_approx(z);
                ms->izfin[w][tw] = iz;
                *reinterpret_cast<float4*>(ms->ecs[w][tw]) = make_float4(e0 * iz, e1 * iz, e2 * iz, e3 * iz);
                a.lse[slice * a.n + (long long)i * 16 + tw] = m2 * (1.0f / kLog2e) + logf(z);
            }
            named_barrier(1 + w, 128);
            float iz[16];
#pragma unroll
            for (int c = 0; c < 16; c += 4) {
                const float4 v = *reinterpret_cast<const float4*>(&ms->izfin[w][c]);
                iz[c] = v.x; iz[c + 1] = v.y; iz[c + 2] = v.z; iz[c + 3] = v.w;
            }
            // normalised P (bf16) as the [query][key] K-major operand
#pragma unroll
            for (int t = 0; t < NT; t++) {
                const int key = t * 128 + qr * 32 + lane;
                unsigned char* pb = P + (key >> 6) * 2048 + (key & 7) * 2;
                const int chk = (key & 63) >> 3;
#pragma unroll
                for (int c = 0; c < 16; c++)
                    *reinterpret_cast<__nv_bfloat16*>(pb + c * 128 + ((chk ^ (c & 7)) << 4)) =
                        __float2bfloat16_rn(s[t][c] * iz[c]);
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(smem_u32(&ms->p_full[w]));
            // epilogue: O^T from TMEM plus the pooled values, written as bf16 rows
            mbar_wait(smem_u32(&ms->o_full[w]), j & 1, abort_flag, a.status, a.spin);
            tc_fence_after();
            float o[16];
            tmem_ld16(tO, o);
            tc_fence_before();
            mbar_arrive(smem_u32(&ms->o_free[w]));
            if (valid) {
                // the block's rows, contiguous in tile order, a 4 x 4 patch in raster order
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out_o) + (slice * a.n + (long long)i * 16) * D + dd;
                if constexpr (R) dst = static_cast<__nv_bfloat16*>(a.out_o) + token_row(slice, a.n, 1, a.side, i * 16) * D + dd;
#pragma unroll
                for (int c = 0; c < 16; c++) {
                    const float4 pz = *reinterpret_cast<const float4*>(ms->ecs[w][c]);
                    float val = o[c];
                    val = fmaf(pz.x, vc[0], val);
                    val = fmaf(pz.y, vc[1], val);
                    val = fmaf(pz.z, vc[2], val);
                    val = fmaf(pz.w, vc[3], val);
                    if constexpr (R) dst[block_token_offset(c, a.side) * D] = __float2bfloat16_rn(val);
                    else dst[c * D] = __float2bfloat16_rn(val);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, C::TM_ALLOC);
    }
}

// ---------------------------------------------------------------------------
// Pipelined variant, used where shared memory holds at least four stages.
//
// Differences from the kernel above:
//  * S^T of a block is issued up to LA blocks ahead of its P V, into one of
//    two S buffers per group; P and O are double-buffered per group as well,
//    so a group writes P of its block j and then finishes the epilogue of
//    block j-1 while P V of j runs on the tensor cores;
//  * softmax shift: the exponentials subtract the largest pooled-key logit of
//    the query (computed one block ahead, so it is ready with S) instead of
//    the row maximum. Softmax is shift-invariant, so only the range matters:
//    if any fine logit exceeds that shift by more than 2^kShiftSlack, the
//    group redoes the block with the exact row maximum (S stays in TMEM until
//    that decision). The common path has one group barrier per block;
//  * the three gather warps split every block's copies (a warp's copy
//    requests issue one after another), each arriving on the stage barrier
//    with its own byte count;
//  * the MMA warp issues out of order between the S and P V streams (P V
//    first, as it frees a stage), through an election inside the MMA asm so
//    that no divergent branch surrounds the MMA instructions.
constexpr float kShiftSlack = 64.f;  // base-2 exponent range above the shift

template <int D, int NT>
struct PCfg {
    static constexpr int NF = NT * 128;
    static constexpr int REG = D / 64;
    static constexpr int Q_BYTES = 16 * D * 2;
    static constexpr int KV_BYTES = NF * D * 2;
    static constexpr int CO_BYTES = 2 * 4 * D * 4;
    static constexpr int STAGE_BYTES = Q_BYTES + 2 * KV_BYTES + CO_BYTES;
    static constexpr int P_BYTES = 16 * NF * 2;
    static constexpr int FIXED = 4 * P_BYTES + 8192;
    static constexpr int STAGES_RAW = (kSmemBudget - FIXED) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr int LA = STAGES - 1 > 4 ? 4 : STAGES - 1;  // S issued ahead of P V
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + FIXED;
    static constexpr int TM_S = NT * 16;                         // columns of one S buffer
    static constexpr int TM_GROUP = 2 * TM_S + 2 * 16;           // two S and two O buffers
    static constexpr int TM_ALLOC = 2 * TM_GROUP <= 128 ? 128 : 256;
};

// the stage count of PCfg without instantiating it
template <int D, int NT>
constexpr bool pipe_fits() {
    return (kSmemBudget - (4 * 16 * NT * 128 * 2 + 8192)) / (16 * D * 2 + 2 * NT * 128 * D * 2 + 2 * 4 * D * 4) >= 4;
}

struct PMisc {
    float red_sum[2][2][16][4];  // [group][buffer][query][warp]
    float red_max[2][16][4];     // exact-maximum pass
    float cmax[2][3][16];        // [group][coarse buffer][query]: largest pooled logit (base 2)
    float csum[2][3][16];        // sum over levels of 2^(pooled logit - cmax)
    float cs2[2][3][16][4];      // pooled logits (base 2), -inf beyond L_e
    float ecs[2][2][16][4];      // coarse probabilities, read by the epilogue
    float izs[2][2][16];         // 1 / row sum, read by the epilogue
    int flags[2][2][4];          // per warp: a logit left the shift's range
    uint64_t full[8], empty[8];
    uint64_t s_full[2][2], s_free[2][2], p_full[2][2], o_full[2][2], o_free[2][2], drain;
    uint32_t tmem_slot;
    int abort_flag;
};

template <int D, int NT, bool R>
__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_pipe_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, AttnArgs a) {
    using C = PCfg<D, NT>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* stages = sm;
    unsigned char* pbuf = stages + C::STAGES * C::STAGE_BYTES;
    PMisc* ms = reinterpret_cast<PMisc*>(pbuf + 4 * C::P_BYTES);
    volatile int* abort_flag = &ms->abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long total = a.slices * (long long)a.T;
    const int G = gridDim.x;
    const int K1 = NT * 8, Le = a.Le;
    // after a grouping pass, the grouped forward may take this call instead
    if (a.ngroups != nullptr) {
        bool skip = false;
        if (warp == 0) {
            const long long groups = sum_groups(a.ngroups, a.ngroups_n, lane);
            skip = lane == 0 && grouped_forward(groups, total, a.test_flags);
        }
        if (__syncthreads_or(skip)) return;
    }
    const long long mine = total > blockIdx.x ? (total - blockIdx.x + G - 1) / G : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; s++) {
            mbar_init(smem_u32(&ms->full[s]), 3);  // one arrival per gather warp
            mbar_init(smem_u32(&ms->empty[s]), 1);
        }
        for (int w = 0; w < 2; w++)
            for (int b = 0; b < 2; b++) {
                mbar_init(smem_u32(&ms->s_full[w][b]), 1);
                mbar_init(smem_u32(&ms->s_free[w][b]), 128);
                mbar_init(smem_u32(&ms->p_full[w][b]), 128);
                mbar_init(smem_u32(&ms->o_full[w][b]), 1);
                mbar_init(smem_u32(&ms->o_free[w][b]), 128);
            }
        mbar_init(smem_u32(&ms->drain), 1);
        ms->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(&ms->tmem_slot), C::TM_ALLOC);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = ms->tmem_slot;

    if (warp == 0 || warp == 2 || warp == 3) {
        // ----------------------------------------------------------- gather
        // Block bl uses stage bl % STAGES for the (bl / STAGES)-th time. The
        // three gather warps split every block's copies (a warp issues its
        // copies one request at a time): warp 0 the Q block and the K_1 K
        // blocks, warp 2 the V blocks, warp 3 the pooled K/V rows; each
        // arrives on the stage barrier with the bytes of its own copies.
        // Index rows are loaded two blocks ahead.
        const int role = warp == 0 ? 0 : warp - 1;
        auto load_idx = [&](long long bl) -> int {
            if (bl >= mine) return 0;
            const long long g = blockIdx.x + bl * G;
            const long long slice = g / a.T;
            const int i = (int)(g - slice * a.T);
            if (role < 2) return lane < K1 ? a.sel[(slice * a.T + i) * a.K1 + lane] : 0;
            return lane < Le ? a.coarse[(slice * a.T + i) * a.C + lane] : 0;
        };
        const uint32_t my_bytes = role == 0 ? C::Q_BYTES + C::KV_BYTES : role == 1 ? C::KV_BYTES : 2 * Le * D * 4;
        int ix0 = load_idx(0), ix1 = load_idx(1);
        long long issued = -1;
        const long long nb = (a.test_flags & LLSA_TEST_NO_COPIES) ? 0 : mine;  // failure-detection test
        for (long long bl = 0; bl < nb; bl++) {
            int ix = ix0;
            ix0 = ix1;
            ix1 = load_idx(bl + 2);
            const int st = (int)(bl % C::STAGES), u = (int)(bl / C::STAGES);
            bool ok = true;
            if (u >= 1 && lane == 0) ok = mbar_wait(smem_u32(&ms->empty[st]), (u - 1) & 1, abort_flag, a.status, a.spin);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0);
            if (!ok) break;
            const long long g = blockIdx.x + bl * G;
            const long long slice = g / a.T;
            const int i = (int)(g - slice * a.T);
            unsigned char* sQ = stages + st * C::STAGE_BYTES;
            unsigned char* sK = sQ + C::Q_BYTES;
            unsigned char* sV = sK + C::KV_BYTES;
            unsigned char* sC = sV + C::KV_BYTES;
            const uint32_t fb = smem_u32(&ms->full[st]);
            if (lane == 0) mbar_arrive_expect_tx(fb, my_bytes);
            __syncwarp();
            if (role == 0 && lane == 0) {
                const int yq = (int)(slice * a.n + (long long)i * 16);
                for (int r = 0; r < C::REG; r++) {
                    if constexpr (R) tma_load_block<true>(smem_u32(sQ + r * 16 * 128), &mq, r * 64, slice, i, a.n, fb);
                    else tma_load_2d(smem_u32(sQ + r * 16 * 128), &mq, r * 64, yq, fb);
                }
            }
            if (role < 2 && lane < K1) {
                if (ix < 0 || ix >= a.T) {
                    set_status(a.status, LLSA_ERR_BAD_INDEX);
                    ix = 0;
                }
                const int yk = R ? ix : (int)(slice * a.n + (long long)ix * 16);
                for (int r = 0; r < C::REG; r++) {
                    if constexpr (R) {
                        if (role == 0)
                            tma_load_block<true>(smem_u32(sK + r * C::NF * 128 + lane * 2048), &mk, r * 64, slice, yk, a.n, fb);
                        else
                            tma_load_block<true>(smem_u32(sV + r * C::NF * 128 + lane * 2048), &mv, r * 64, slice, yk, a.n, fb);
                    } else {
                        if (role == 0) tma_load_2d(smem_u32(sK + r * C::NF * 128 + lane * 2048), &mk, r * 64, yk, fb);
                        else tma_load_2d(smem_u32(sV + r * C::NF * 128 + lane * 2048), &mv, r * 64, yk, fb);
                    }
                }
            }
            if (role == 2 && lane < Le) {
                if (ix < 0 || ix >= a.lv.n_level[lane + 1]) {
                    set_status(a.status, LLSA_ERR_BAD_INDEX);
                    ix = 0;
                }
                const long long row = slice * a.pyr_stride + (long long)(a.lv.row_offset[lane + 1] + ix) * D;
                bulk_load(smem_u32(sC + lane * D * 4), a.kpyr + row, D * 4, fb);
                bulk_load(smem_u32(sC + (4 + lane) * D * 4), a.vpyr + row, D * 4, fb);
            }
            issued = bl;
        }
        // copies still in flight must land before the CTA exits
        if (lane == 0)
            for (long long bl = issued; bl >= 0 && bl > issued - C::STAGES; bl--) {
                const int st = (int)(bl % C::STAGES), u = (int)(bl / C::STAGES);
                for (int it = 0; it < kSpinLimit && !mbar_try(smem_u32(&ms->full[st]), u & 1); it++) {
                }
            }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        constexpr uint32_t idS = idesc_bf16(128, 16, 0, 0);
        constexpr uint32_t idPV = idesc_bf16(D, 16, 1, 0);
        const uint64_t dKQ = desc_sw128(smem_u32(stages), 16, 1024);          // K-major
        const uint64_t dV = desc_sw128(smem_u32(stages), C::NF * 128, 1024);  // MN-major V
        const uint64_t dP = desc_sw128(smem_u32(pbuf), 16, 1024);
        // block bl: group bl & 1, its j-th block, buffer j & 1 used for the (j >> 1)-th time
        auto s_ready = [&](long long bl) -> bool {
            const int w = (int)(bl & 1), b = (int)((bl >> 1) & 1);
            const uint32_t use = (uint32_t)(bl >> 2);
            const int st = (int)(bl % C::STAGES), u = (int)(bl / C::STAGES);
            return mbar_test(smem_u32(&ms->full[st]), u & 1) &&
                   (use == 0 || mbar_test(smem_u32(&ms->s_free[w][b]), (use - 1) & 1));
        };
        auto pv_ready = [&](long long bl) -> bool {
            const int w = (int)(bl & 1), b = (int)((bl >> 1) & 1);
            const uint32_t use = (uint32_t)(bl >> 2);
            return mbar_test(smem_u32(&ms->p_full[w][b]), use & 1) &&
                   (use == 0 || mbar_test(smem_u32(&ms->o_free[w][b]), (use - 1) & 1));
        };
        auto issue_S = [&](long long bl) {
            const int w = (int)(bl & 1), b = (int)((bl >> 1) & 1);
            const int st = (int)(bl % C::STAGES);
            tc_fence_after();
            const uint32_t q0 = (uint32_t)(st * C::STAGE_BYTES), k0 = q0 + C::Q_BYTES;
            const uint32_t dt = tbase + w * C::TM_GROUP + b * C::TM_S;
#pragma unroll
            for (int t = 0; t < NT; t++)
#pragma unroll
                for (int ks = 0; ks < D / 16; ks++) {
                    const uint64_t da = dKQ + ((k0 + (ks / 4) * C::NF * 128 + t * 128 * 128 + (ks % 4) * 32) >> 4);
                    const uint64_t db = dKQ + ((q0 + (ks / 4) * 16 * 128 + (ks % 4) * 32) >> 4);
                    mma_bf16_warp(dt + t * 16, da, db, idS, ks > 0);
                }
            mma_commit_warp(smem_u32(&ms->s_full[w][b]));
        };
        auto issue_PV = [&](long long bl) {
            const int w = (int)(bl & 1), b = (int)((bl >> 1) & 1);
            const int st = (int)(bl % C::STAGES);
            tc_fence_after();
            const uint32_t v0 = (uint32_t)(st * C::STAGE_BYTES + C::Q_BYTES + C::KV_BYTES);
            const uint32_t p0 = (uint32_t)((w * 2 + b) * C::P_BYTES);
            const uint32_t dt = tbase + w * C::TM_GROUP + 2 * C::TM_S + b * 16;
#pragma unroll
            for (int ks = 0; ks < C::NF / 16; ks++) {
                const uint64_t da = dV + ((v0 + ks * 2048) >> 4);
                const uint64_t db = dP + ((p0 + (ks / 4) * 2048 + (ks % 4) * 32) >> 4);
                mma_bf16_warp(dt, da, db, idPV, ks > 0);
            }
            mma_commit_warp(smem_u32(&ms->o_full[w][b]));
            mma_commit_warp(smem_u32(&ms->empty[st]));
        };
        // Out-of-order issue between the two in-order streams: P V of the
        // oldest block as soon as its P is written (it frees a stage), else
        // S of the next block once its operands have landed, at most LA
        // blocks ahead of P V. Idle polls are bounded like every other wait.
        long long nS = 0, nP = 0;
        int idle = 0;
        while (nP < mine) {
            int act = 0;
            if (lane == 0) {
                if (nP < nS && pv_ready(nP)) act = 2;
                else if (nS < mine && nS < nP + C::LA && s_ready(nS)) act = 1;
            }
            act = __shfl_sync(0xffffffffu, act, 0);
            if (act == 1) {
                issue_S(nS++);
                idle = 0;
            } else if (act == 2) {
                issue_PV(nP++);
                idle = 0;
            } else {
                int stop = 0;
                if (lane == 0) {
                    if (++idle >= a.spin) {
                        *abort_flag = 1;
                        set_status(a.status, LLSA_ERR_TIMEOUT);
                        stop = 1;
                    } else if ((idle & 63) == 0 && *abort_flag) {
                        stop = 1;
                    }
                }
                if (__shfl_sync(0xffffffffu, stop, 0)) break;
            }
        }
        // no MMA may be in flight when TMEM is released
        mma_commit_warp(smem_u32(&ms->drain));
        if (lane == 0)
            for (int it = 0; it < kSpinLimit && !mbar_try(smem_u32(&ms->drain), 0); it++) {
            }
        __syncwarp();
    } else if (warp >= 4) {
        // ----------------------------------------- softmax + epilogue groups
        const int w = (warp - 4) >> 2, qr = warp & 3;
        const int tw = threadIdx.x - 128 * (1 + w);
        const uint32_t lanes = (uint32_t)(qr * 32) << 16;
        const float sc = a.scale, scl2 = a.scale * kLog2e;
        const int dd = D == 64 ? 16 * qr + lane : 32 * qr + lane;  // O^T row this thread reads back
        const bool valid = D == 64 ? lane < 16 : true;
        const long long nblk = mine > w ? (mine - w + 1) / 2 : 0;  // blocks w, w + 2, ...
        const int cq = tw >> 3, cpart = tw & 7;                   // pooled-score role
        // pooled-key logits (base 2, + l ln B) of the group's block j into coarse buffer cb;
        // eight threads per query, each a 16-byte chunk of the row per 64 columns
        auto coarse = [&](long long j, int cb) {
            const long long bl = w + 2 * j;
            const int st = (int)(bl % C::STAGES), u = (int)(bl / C::STAGES);
            mbar_wait(smem_u32(&ms->full[st]), u & 1, abort_flag, a.status, a.spin);
            const unsigned char* sQ = stages + st * C::STAGE_BYTES;
            const float* sCk = reinterpret_cast<const float*>(sQ + C::Q_BYTES + 2 * C::KV_BYTES);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int cc = 0; cc < D / 64; cc++) {
                const int c8 = cpart + 8 * cc;
                const uint4 raw = *reinterpret_cast<const uint4*>(sQ + sw128_offset(cq, c8 * 8, 16));
                const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
                const float2 x0 = __bfloat1622float2(h[0]), x1 = __bfloat1622float2(h[1]);
                const float2 x2 = __bfloat1622float2(h[2]), x3 = __bfloat1622float2(h[3]);
#pragma unroll
                for (int l = 0; l < 4; l++)
                    if (l < Le) {
                        const float4 k0 = *reinterpret_cast<const float4*>(sCk + l * D + c8 * 8);
                        const float4 k1 = *reinterpret_cast<const float4*>(sCk + l * D + c8 * 8 + 4);
                        float t0 = x0.x * k0.x, t1 = x0.y * k0.y;
                        t0 = fmaf(x1.x, k0.z, t0); t1 = fmaf(x1.y, k0.w, t1);
                        t0 = fmaf(x2.x, k1.x, t0); t1 = fmaf(x2.y, k1.y, t1);
                        t0 = fmaf(x3.x, k1.z, t0); t1 = fmaf(x3.y, k1.w, t1);
                        acc[l] += t0 + t1;
                    }
            }
            float cs[4], cm = -INFINITY;
#pragma unroll
            for (int l = 0; l < 4; l++) {
                float v = acc[l];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                cs[l] = l < Le ? (sc * v + (float)(l + 1) * a.lnB) * kLog2e : -INFINITY;
                cm = fmaxf(cm, cs[l]);
            }
            float sum = 0.f;
#pragma unroll
            for (int l = 0; l < 4; l++)
                if (l < Le) sum += ex2(cs[l] - cm);
            if (cpart == 0) {
                ms->cmax[w][cb][cq] = cm;
                ms->csum[w][cb][cq] = sum;
            }
            if (cpart < 4) ms->cs2[w][cb][cq][cpart] = cpart == 0 ? cs[0] : cpart == 1 ? cs[1] : cpart == 2 ? cs[2] : cs[3];
        };
        auto epilogue = [&](long long j, const float* vcp) {
            const long long bl = w + 2 * j;
            const int b = (int)(j & 1);
            const uint32_t use = (uint32_t)(j >> 1);
            const long long g = blockIdx.x + bl * G;
            const long long slice = g / a.T;
            const int i = (int)(g - slice * a.T);
            mbar_wait(smem_u32(&ms->o_full[w][b]), use & 1, abort_flag, a.status, a.spin);
            tc_fence_after();
            float o[16];
            tmem_ld16(tbase + w * C::TM_GROUP + 2 * C::TM_S + b * 16 + lanes, o);
            tc_fence_before();
            mbar_arrive(smem_u32(&ms->o_free[w][b]));
            if (valid) {
                // the block's rows, contiguous in tile order, a 4 x 4 patch in raster order
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out_o) + (slice * a.n + (long long)i * 16) * D + dd;
                if constexpr (R) dst = static_cast<__nv_bfloat16*>(a.out_o) + token_row(slice, a.n, 1, a.side, i * 16) * D + dd;
#pragma unroll
                for (int c = 0; c < 16; c++) {
                    const float4 pz = *reinterpret_cast<const float4*>(ms->ecs[w][b][c]);
                    float val = o[c] * ms->izs[w][b][c];
                    val = fmaf(pz.x, vcp[0], val);
                    val = fmaf(pz.y, vcp[1], val);
                    val = fmaf(pz.z, vcp[2], val);
                    val = fmaf(pz.w, vcp[3], val);
                    if constexpr (R) dst[block_token_offset(c, a.side) * D] = __float2bfloat16_rn(val);
                    else dst[c * D] = __float2bfloat16_rn(val);
                }
            }
        };

        if (nblk > 0) {
            coarse(0, 0);
            named_barrier(1 + w, 128);
        }
        float vc_prev[4] = {0.f, 0.f, 0.f, 0.f};
        int cb = 0;  // coarse buffer of block j: j % 3
        for (long long j = 0; j < nblk; j++) {
            const long long bl = w + 2 * j;
            const int b = (int)(j & 1);
            const uint32_t use = (uint32_t)(j >> 1);
            const int st = (int)(bl % C::STAGES);
            const long long g = blockIdx.x + bl * G;
            const long long slice = g / a.T;
            const int i = (int)(g - slice * a.T);
            const float* sCk = reinterpret_cast<const float*>(stages + st * C::STAGE_BYTES + C::Q_BYTES + 2 * C::KV_BYTES);
            const uint32_t tS = tbase + w * C::TM_GROUP + b * C::TM_S + lanes;
            float m2[16];
#pragma unroll
            for (int c = 0; c < 16; c += 4) {
                const float4 v = *reinterpret_cast<const float4*>(&ms->cmax[w][cb][c]);
                m2[c] = v.x; m2[c + 1] = v.y; m2[c + 2] = v.z; m2[c + 3] = v.w;
            }
            mbar_wait(smem_u32(&ms->s_full[w][b]), use & 1, abort_flag, a.status, a.spin);
            tc_fence_after();
            float s[NT][16];
#pragma unroll
            for (int t = 0; t < NT; t++) tmem_ld16(tS + t * 16, s[t]);
            float x[16], amax = -INFINITY;
#pragma unroll
            for (int c = 0; c < 16; c++) {
                x[c] = 0.f;
#pragma unroll
                for (int t = 0; t < NT; t++) {
                    const float arg = fmaf(s[t][c], scl2, -m2[c]);
                    amax = fmaxf(amax, arg);
                    s[t][c] = ex2(arg);
                    x[c] += s[t][c];
                }
            }
            // the next block's pooled logits, while this block's sums travel
            const int cbn = cb == 2 ? 0 : cb + 1;
            if (j + 1 < nblk) coarse(j + 1, cbn);
            float r = warp_reduce16<false>(x, lane);
            if (!(lane & 1)) ms->red_sum[w][b][lane >> 1][qr] = r;
            const unsigned wide = __ballot_sync(0xffffffffu, !(amax <= kShiftSlack));
            if (lane == 0) ms->flags[w][b][qr] = wide != 0u;
            named_barrier(1 + w, 128);
            const int4 fl = *reinterpret_cast<const int4*>(ms->flags[w][b]);
            float fac[16];  // rescales the pooled sum to the final shift
            if ((fl.x | fl.y | fl.z | fl.w) != 0) {
                // exact row maxima from the raw S, still held in TMEM
#pragma unroll
                for (int t = 0; t < NT; t++) tmem_ld16(tS + t * 16, s[t]);
#pragma unroll
                for (int c = 0; c < 16; c++) {
                    x[c] = s[0][c];
#pragma unroll
                    for (int t = 1; t < NT; t++) x[c] = fmaxf(x[c], s[t][c]);
                }
                r = warp_reduce16<true>(x, lane);
                if (!(lane & 1)) ms->red_max[w][lane >> 1][qr] = r;
                named_barrier(1 + w, 128);
#pragma unroll
                for (int c = 0; c < 16; c++) {
                    const float4 rm = *reinterpret_cast<const float4*>(ms->red_max[w][c]);
                    const float mn = fmaxf(m2[c], fmaxf(fmaxf(rm.x, rm.y), fmaxf(rm.z, rm.w)) * scl2);
                    fac[c] = ex2(m2[c] - mn);
                    m2[c] = mn;
                    x[c] = 0.f;
#pragma unroll
                    for (int t = 0; t < NT; t++) {
                        s[t][c] = ex2(fmaf(s[t][c], scl2, -m2[c]));
                        x[c] += s[t][c];
                    }
                }
                r = warp_reduce16<false>(x, lane);
                if (!(lane & 1)) ms->red_sum[w][b][lane >> 1][qr] = r;
                named_barrier(1 + w, 128);
            } else {
#pragma unroll
                for (int c = 0; c < 16; c++) fac[c] = 1.f;
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&ms->s_free[w][b]));
            // this thread's column of the pooled V rows, read while the stage is held
            float vc[4];
#pragma unroll
            for (int l = 0; l < 4; l++) vc[l] = (l < Le && valid) ? sCk[(4 + l) * D + dd] : 0.f;
            // unnormalised P (bf16, <= 2^kShiftSlack) as the [query][key]
            // K-major operand; O is scaled by 1 / row sum in the epilogue
            unsigned char* P = pbuf + (w * 2 + b) * C::P_BYTES;
#pragma unroll
            for (int t = 0; t < NT; t++) {
                const int key = t * 128 + qr * 32 + lane;
                unsigned char* pb = P + (key >> 6) * 2048 + (key & 7) * 2;
                const int chk = (key & 63) >> 3;
#pragma unroll
                for (int c = 0; c < 16; c++)
                    *reinterpret_cast<__nv_bfloat16*>(pb + c * 128 + ((chk ^ (c & 7)) << 4)) = __float2bfloat16_rn(s[t][c]);
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(smem_u32(&ms->p_full[w][b]));
            // while P V runs: row sums (fine keys + pooled keys), each >= 1
            // because the shift is one of the logits or lies above all of them
            if (tw < 64) {
                const int q = tw >> 2, l = tw & 3;
                float mq = 0.f, fq = 1.f;
#pragma unroll
                for (int c = 0; c < 16; c++)
                    if (c == q) { mq = m2[c]; fq = fac[c]; }
                const float4 rs = *reinterpret_cast<const float4*>(ms->red_sum[w][b][q]);
                const float z = ((rs.x + rs.y) + (rs.z + rs.w)) + ms->csum[w][cb][q] * fq;
                const float iz = rcp_approx(z);
                ms->ecs[w][b][q][l] = ex2(ms->cs2[w][cb][q][l] - mq) * iz;
                if (l == 0) {
                    ms->izs[w][b][q] = iz;
                    a.lse[slice * a.n + (long long)i * 16 + q] = mq * (1.0f / kLog2e) + logf(z);
                }
            }
            if (j >= 1) epilogue(j - 1, vc_prev);
#pragma unroll
            for (int l = 0; l < 4; l++) vc_prev[l] = vc[l];
            cb = cbn;
        }
        if (nblk > 0) epilogue(nblk - 1, vc_prev);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, C::TM_ALLOC);
    }
}

template <int D, int NT, bool R>
int launch_pipe(const Shape& s, const AttnArgs& a, const CUtensorMap& mq, const CUtensorMap& mk,
                const CUtensorMap& mv, cudaStream_t st) {
    using C = PCfg<D, NT>;
    static_assert(C::SMEM <= 227 * 1024 && C::STAGES >= 4, "shared memory budget");
    static_assert(sizeof(PMisc) <= 8192, "misc block");
    cudaFuncSetAttribute(fwd_tc_pipe_kernel<D, NT, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    const long long total = s.slices * (long long)s.T;
    const int grid = (int)std::min<long long>(total, (long long)sm_count());
    LLSA_LAUNCH("fwd_tc", st, fwd_tc_pipe_kernel<D, NT, R><<<grid, kThreads, C::SMEM, st>>>(mq, mk, mv, a));
    return LLSA_OK;
}

template <int D, int NT, bool R>
int launch_cfg(const Shape& s, const AttnArgs& a, const CUtensorMap& mq, const CUtensorMap& mk,
               const CUtensorMap& mv, cudaStream_t st) {
    using C = Cfg<D, NT>;
    static_assert(C::SMEM <= 227 * 1024, "shared memory budget");
    static_assert(sizeof(Misc) <= 4096, "misc block");
    cudaFuncSetAttribute(fwd_tc_kernel<D, NT, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    const long long total = s.slices * (long long)s.T;
    const int grid = (int)std::min<long long>(total, (long long)sm_count());
    LLSA_LAUNCH("fwd_tc", st, fwd_tc_kernel<D, NT, R><<<grid, kThreads, C::SMEM, st>>>(mq, mk, mv, a));
    return LLSA_OK;
}

// the pipelined kernel where four stages fit, else the few-stage one; each
// built once per token order
template <int D, int NT>
int launch_any(const Shape& s, const AttnArgs& a, const CUtensorMap& mq, const CUtensorMap& mk,
               const CUtensorMap& mv, cudaStream_t st) {
    if constexpr (pipe_fits<D, NT>()) {
        return s.raster ? launch_pipe<D, NT, true>(s, a, mq, mk, mv, st) : launch_pipe<D, NT, false>(s, a, mq, mk, mv, st);
    } else {
        return s.raster ? launch_cfg<D, NT, true>(s, a, mq, mk, mv, st) : launch_cfg<D, NT, false>(s, a, mq, mk, mv, st);
    }
}

}  // namespace

bool fwd_tc_supported(const Shape& s) {
    // one enrichment column per level (the pooled keys sit in four row slots)
    // (K_1 = 32 at d = 64: four key tiles, one ring stage)
    return s.dtype == LLSA_DTYPE_BF16 && s.B == 16 && (s.d == 64 || s.d == 128) &&
           (s.K1 == 8 || s.K1 == 16 || (s.K1 == 32 && s.d == 64)) && s.Le <= 4 && s.Lc == s.Le &&
           s.slices * (long long)s.n < (1LL << 31);
}

int launch_fwd_tc(const Shape& s, const AttnArgs& a, cudaStream_t st) {
    CUtensorMap mq, mk, mv;
    LLSA_TRY(make_tmap_tokens(&mq, a.q, s));
    LLSA_TRY(make_tmap_tokens(&mk, a.k, s));
    LLSA_TRY(make_tmap_tokens(&mv, a.v, s));
    if (s.d == 64) {
        if (s.K1 == 32) return launch_any<64, 4>(s, a, mq, mk, mv, st);
        return s.K1 == 8 ? launch_any<64, 1>(s, a, mq, mk, mv, st) : launch_any<64, 2>(s, a, mq, mk, mv, st);
    }
    return s.K1 == 8 ? launch_any<128, 1>(s, a, mq, mk, mv, st) : launch_any<128, 2>(s, a, mq, mk, mv, st);
}

}  // namespace llsa
