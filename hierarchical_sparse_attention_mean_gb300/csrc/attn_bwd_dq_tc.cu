// attn_bwd_dq_tc.cu -- backward, query-major part, on the tcgen05 tensor cores
// (bf16, B = 16, d in {64, 128}, K_1 in {4, 8, 16}, and K_1 = 32 at d = 64):
// dq, D = rowsum(dO o) (stored
// with lse as (lse, D) pairs for the key-major kernel), and
// the per-(query block, level) partial gradients of the pooled keys and values.
//
// Method: Pith review of arXiv 2512.16615, referee comment on Sec. 4.3 and
// Figure 4 (the backward uses only sparse indices) with the forward of "Core
// claim". For token t of query block i and each of its keys x (the K*B fine
// keys and the L_e pooled keys): P = exp(s - lse_t), dP = dO_t . v_x,
// dS = P (dP - D_t), dq_t = scale * sum_x dS k_x; a pooled key also collects
// scale * sum_t dS q_t and sum_t P dO_t for the pooled-level gradients.
//
// Per query block, key-major like the forward: S^T = K_sel Q^T and
// dP^T = V_sel dO^T (M = 128 keys per tile, 64 when K_1 = 4; N = 16 queries), dS^T computed per
// TMEM lane and stored as the K-major operand, then dq^T = K_sel^T dS^T with
// the same K tile read as an MN-major operand (M = d, N = 16, K = keys). The
// softmax needs no reduction here: lse is known.
//
// Pooled keys: eight threads per query compute D_t and the query's dot
// products with the pooled K and V rows (one 16-byte chunk of each row per 64
// columns), so P, dS and D_t of a query are known without a group barrier.
// The pooled-level partial gradients are two more MMAs per block:
// gK^T = Q^T dS_c and gV^T = dO^T P_c (M = d, N = 16 with L_e <= 4 columns
// used, K = the 16 queries), with dS_c and P_c stored as bf16 operands like
// the fine-key dS.
//
// Warp roles: three gather warps split every block's copies (warp 0 the Q, dO
// and o boxes, lse and the pooled rows; warp 2 the K blocks; warp 3 the V
// blocks) into a ring of stages; warp 1 issues the MMAs out of order between
// the S stream and the gradient stream (gradient first, as it frees a stage),
// through an election inside the MMA asm; two warpgroups alternate query
// blocks.
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

template <int D, int NF_>
struct Cfg {
    static constexpr int NF = NF_;                // fine keys per query block (16 K_1)
    static constexpr int NT = NF < 128 ? 1 : NF / 128;  // key tiles (one MMA M each)
    static constexpr int MT = NF < 128 ? NF : 128;      // keys per tile (the MMA's M)
    static constexpr int REG = D / 64;
    static constexpr int Q_BYTES = 16 * D * 2;
    static constexpr int KV_BYTES = NF * D * 2;
    static constexpr int CO_BYTES = 2 * 4 * D * 4;  // pooled K and V rows (fp32)
    // Q, dO, o, K, V, pooled rows, lse (64 B, padded)
    static constexpr int OFF_DO = Q_BYTES, OFF_O = 2 * Q_BYTES, OFF_K = 3 * Q_BYTES;
    static constexpr int OFF_V = OFF_K + KV_BYTES, OFF_C = OFF_V + KV_BYTES, OFF_L = OFF_C + CO_BYTES;
    static constexpr int STAGE_BYTES = OFF_L + 1024;
    static constexpr int DS_BYTES = 16 * NF * 2;  // per warpgroup
    static constexpr int BC_BYTES = 2048;         // per warpgroup and operand: 16 rows x 128 B
    static constexpr int FIXED = 2 * DS_BYTES + 4 * BC_BYTES + 4096;
    static constexpr int STAGES_RAW = (kSmemBudget - FIXED) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 6 ? 6 : STAGES_RAW;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + FIXED;
    // TMEM columns per warpgroup: S +0 and dP (16 per key tile each), then dq,
    // gK, gV (16 each); up to two key tiles S +0, dP +32, dq +64, gK +96, gV +112
    static constexpr int TM_DP = NT <= 2 ? 32 : NT * 16;
    static constexpr int TM_DQ = 2 * TM_DP, TM_GK = TM_DQ + 32, TM_GV = TM_DQ + 48;
    static constexpr int TM_GROUP = NT <= 2 ? 128 : 256;
    static constexpr int TM_ALLOC = 2 * TM_GROUP;
};

struct Misc {
    float dsum[2][16];       // D_t
    float cds[2][2][16][4];  // pooled-key dS, [group][block parity][query][level]
    uint64_t full[6], empty[6], q_ready[2], s_full[2], ds_full[2], g_full[2], s_free[2], o_free[2], drain;
    uint32_t tmem_slot;
    int abort_flag;
};

template <int D, int NF, bool R>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mdo,
                 const __grid_constant__ CUtensorMap mo, const __grid_constant__ CUtensorMap mk,
                 const __grid_constant__ CUtensorMap mv, AttnArgs a) {
    using C = Cfg<D, NF>;
    constexpr int NT = C::NT;
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned base (128-byte swizzle atoms), derived from the
    // __shared__ array by pointer arithmetic so accesses stay shared-space
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* stages = sm;
    unsigned char* dsbuf = stages + C::STAGES * C::STAGE_BYTES;
    unsigned char* bcbuf = dsbuf + 2 * C::DS_BYTES;  // [group][dS_c, P_c]
    Misc* ms = reinterpret_cast<Misc*>(bcbuf + 4 * C::BC_BYTES);
    volatile int* abort_flag = &ms->abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long total = a.slices * (long long)a.T;
    const int G = gridDim.x;
    const int K1 = NF / 16, Le = a.Le;
    const long long mine = total > blockIdx.x ? (total - blockIdx.x + G - 1) / G : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; s++) {
            mbar_init(smem_u32(&ms->full[s]), 3);  // one arrival per gather warp
            mbar_init(smem_u32(&ms->empty[s]), 1);
        }
        for (int w = 0; w < 2; w++) {
            mbar_init(smem_u32(&ms->q_ready[w]), 1);
            mbar_init(smem_u32(&ms->s_full[w]), 1);
            mbar_init(smem_u32(&ms->ds_full[w]), 128);
            mbar_init(smem_u32(&ms->g_full[w]), 1);
            mbar_init(smem_u32(&ms->s_free[w]), 128);
            mbar_init(smem_u32(&ms->o_free[w]), 128);
        }
        mbar_init(smem_u32(&ms->drain), 1);
        ms->abort_flag = 0;
        fence_mbar_init();
    }
    // rows L_e..15 of the pooled operands stay zero
    for (int x = threadIdx.x; x < 4 * C::BC_BYTES / 16; x += kThreads)
        reinterpret_cast<uint4*>(bcbuf)[x] = make_uint4(0u, 0u, 0u, 0u);
    fence_async_smem();
    if (warp == 1) tmem_alloc(smem_u32(&ms->tmem_slot), C::TM_ALLOC);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = ms->tmem_slot;

    if (warp == 0 || warp == 2 || warp == 3) {
        // ----------------------------------------------------------- gather
        // Block bl uses stage bl % STAGES for the (bl / STAGES)-th time; each
        // warp arrives on the stage barrier with the bytes of its own copies.
        const int role = warp == 0 ? 0 : warp - 1;
        auto load_idx = [&](long long bl) -> int {
            if (bl >= mine) return 0;
            const long long g = blockIdx.x + bl * G;  // global query block (slice * T + i)
            if (role == 0) return lane < Le ? a.coarse[g * a.C + lane] : 0;
            return lane < K1 ? a.sel[g * a.K1 + lane] : 0;
        };
        const uint32_t my_bytes = role == 0 ? 3 * C::Q_BYTES + 64 + 2 * Le * D * 4 : C::KV_BYTES;
        int ix0 = load_idx(0), ix1 = load_idx(1);
        long long issued = -1;
        const long long nb = (a.test_flags & LLSA_TEST_NO_COPIES) ? 0 : mine;  // failure-detection test
        // block bl is global query block blockIdx.x + bl * G: block i of
        // slice `slice` (walked, no division per block)
        long long slice = blockIdx.x / a.T;
        int i = (int)(blockIdx.x - slice * a.T);
        for (long long bl = 0; bl < nb; bl++, i += G) {
            while (i >= a.T) {
                i -= a.T;
                slice++;
            }
            int ix = ix0;
            ix0 = ix1;
            ix1 = load_idx(bl + 2);
            const int st = (int)(bl % C::STAGES), u = (int)(bl / C::STAGES);
            bool ok = true;
            if (u >= 1 && lane == 0) ok = mbar_wait(smem_u32(&ms->empty[st]), (u - 1) & 1, abort_flag, a.status, a.spin);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0);
            if (!ok) break;
            unsigned char* sb = stages + st * C::STAGE_BYTES;
            const uint32_t fb = smem_u32(&ms->full[st]);
            if (lane == 0) mbar_arrive_expect_tx(fb, my_bytes);
            __syncwarp();
            const long long tok0 = slice * a.n + (long long)i * 16;
            if (role == 0) {
                if (lane == 0) {
                    for (int r = 0; r < C::REG; r++) {
                        if constexpr (R) {
                            tma_load_block<true>(smem_u32(sb + r * 2048), &mq, r * 64, slice, i, a.n, fb);
                            tma_load_block<true>(smem_u32(sb + C::OFF_DO + r * 2048), &mdo, r * 64, slice, i, a.n, fb);
                            tma_load_block<true>(smem_u32(sb + C::OFF_O + r * 2048), &mo, r * 64, slice, i, a.n, fb);
                        } else {
                            tma_load_2d(smem_u32(sb + r * 2048), &mq, r * 64, (int)tok0, fb);
                            tma_load_2d(smem_u32(sb + C::OFF_DO + r * 2048), &mdo, r * 64, (int)tok0, fb);
                            tma_load_2d(smem_u32(sb + C::OFF_O + r * 2048), &mo, r * 64, (int)tok0, fb);
                        }
                    }
                    bulk_load(smem_u32(sb + C::OFF_L), a.lse_in + tok0, 64, fb);
                }
                if (lane < Le) {
                    if (ix < 0 || ix >= a.lv.n_level[lane + 1]) {
                        set_status(a.status, LLSA_ERR_BAD_INDEX);
                        ix = 0;
                    }
                    const long long row = slice * a.pyr_stride + (long long)(a.lv.row_offset[lane + 1] + ix) * D;
                    bulk_load(smem_u32(sb + C::OFF_C + lane * D * 4), a.kpyr + row, D * 4, fb);
                    bulk_load(smem_u32(sb + C::OFF_C + (4 + lane) * D * 4), a.vpyr + row, D * 4, fb);
                }
            } else if (lane < K1) {
                if (ix < 0 || ix >= a.T) {
                    set_status(a.status, LLSA_ERR_BAD_INDEX);
                    ix = 0;
                }
                const int yk = R ? ix : (int)(slice * a.n + (long long)ix * 16);
                for (int r = 0; r < C::REG; r++) {
                    if constexpr (R) {
                        if (role == 1)
                            tma_load_block<true>(smem_u32(sb + C::OFF_K + r * C::NF * 128 + lane * 2048), &mk, r * 64,
                                                 slice, yk, a.n, fb);
                        else
                            tma_load_block<true>(smem_u32(sb + C::OFF_V + r * C::NF * 128 + lane * 2048), &mv, r * 64,
                                                 slice, yk, a.n, fb);
                    } else {
                        if (role == 1) tma_load_2d(smem_u32(sb + C::OFF_K + r * C::NF * 128 + lane * 2048), &mk, r * 64, yk, fb);
                        else tma_load_2d(smem_u32(sb + C::OFF_V + r * C::NF * 128 + lane * 2048), &mv, r * 64, yk, fb);
                    }
                }
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
        constexpr uint32_t idS = idesc_bf16(C::MT, 16, 0, 0);
        constexpr uint32_t idQ = idesc_bf16(D, 16, 1, 0);
        const uint64_t dKm = desc_sw128(smem_u32(stages), 16, 1024);            // K-major
        const uint64_t dMN = desc_sw128(smem_u32(stages), C::NF * 128, 1024);   // K tile as MN-major
        const uint64_t dQT = desc_sw128(smem_u32(stages), 16 * 128, 1024);      // Q / dO tiles as MN-major
        const uint64_t dDS = desc_sw128(smem_u32(dsbuf), 16, 1024);
        const uint64_t dBC = desc_sw128(smem_u32(bcbuf), 16, 1024);
        // block bl: group bl & 1, its j-th block
        auto s_ready = [&](long long bl) -> bool {
            const int w = (int)(bl & 1);
            const uint32_t j = (uint32_t)(bl >> 1);
            const int st = (int)(bl % C::STAGES), u = (int)(bl / C::STAGES);
            return mbar_test(smem_u32(&ms->full[st]), u & 1) &&
                   (j == 0 || mbar_test(smem_u32(&ms->s_free[w]), (j - 1) & 1));
        };
        auto g_ready = [&](long long bl) -> bool {
            const int w = (int)(bl & 1);
            const uint32_t j = (uint32_t)(bl >> 1);
            return mbar_test(smem_u32(&ms->ds_full[w]), j & 1) &&
                   (j == 0 || mbar_test(smem_u32(&ms->o_free[w]), (j - 1) & 1));
        };
        auto issue_S = [&](long long bl) {
            const int w = (int)(bl & 1);
            const int st = (int)(bl % C::STAGES);
            if (lane == 0) mbar_arrive(smem_u32(&ms->q_ready[w]));  // the group may read the stage
            tc_fence_after();
            const uint32_t s0 = (uint32_t)(st * C::STAGE_BYTES);
#pragma unroll
            for (int t = 0; t < NT; t++)
#pragma unroll
                for (int ks = 0; ks < D / 16; ks++) {
                    const uint32_t koff = (ks / 4) * C::NF * 128 + t * 128 * 128 + (ks % 4) * 32;
                    const uint32_t qoff = (ks / 4) * 2048 + (ks % 4) * 32;
                    mma_bf16_warp(tbase + w * C::TM_GROUP + t * 16, dKm + ((s0 + C::OFF_K + koff) >> 4),
                                  dKm + ((s0 + qoff) >> 4), idS, ks > 0);
                    mma_bf16_warp(tbase + w * C::TM_GROUP + C::TM_DP + t * 16, dKm + ((s0 + C::OFF_V + koff) >> 4),
                                  dKm + ((s0 + C::OFF_DO + qoff) >> 4), idS, ks > 0);
                }
            mma_commit_warp(smem_u32(&ms->s_full[w]));
        };
        auto issue_G = [&](long long bl) {
            const int w = (int)(bl & 1);
            const int st = (int)(bl % C::STAGES);
            tc_fence_after();
            const uint32_t s0 = (uint32_t)(st * C::STAGE_BYTES);
            const uint32_t d0 = (uint32_t)(w * C::DS_BYTES);
            const uint32_t b0 = (uint32_t)(w * 2 * C::BC_BYTES);
            const uint32_t tg = tbase + w * C::TM_GROUP;
#pragma unroll
            for (int ks = 0; ks < C::NF / 16; ks++)
                mma_bf16_warp(tg + C::TM_DQ, dMN + ((s0 + C::OFF_K + ks * 2048) >> 4),
                              dDS + ((d0 + (ks / 4) * 2048 + (ks % 4) * 32) >> 4), idQ, ks > 0);
            mma_bf16_warp(tg + C::TM_GK, dQT + (s0 >> 4), dBC + (b0 >> 4), idQ, 0);
            mma_bf16_warp(tg + C::TM_GV, dQT + ((s0 + C::OFF_DO) >> 4), dBC + ((b0 + C::BC_BYTES) >> 4), idQ, 0);
            mma_commit_warp(smem_u32(&ms->g_full[w]));
            mma_commit_warp(smem_u32(&ms->empty[st]));
        };
        // out of order between the two in-order streams; idle polls bounded
        long long nS = 0, nG = 0;
        int idle = 0;
        while (nG < mine) {
            int act = 0;
            if (lane == 0) {
                if (nG < nS && g_ready(nG)) act = 2;
                else if (nS < mine && s_ready(nS)) act = 1;
            }
            act = __shfl_sync(0xffffffffu, act, 0);
            if (act == 1) {
                issue_S(nS++);
                idle = 0;
            } else if (act == 2) {
                issue_G(nG++);
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
        // --------------------------------------------- elementwise + epilogue
        const int w = (warp - 4) >> 2, qr = warp & 3;
        const int tw = threadIdx.x - 128 * (1 + w);
        const uint32_t tS = tbase + w * C::TM_GROUP + ((uint32_t)(qr * 32) << 16);
        const float sc = a.scale, scl2 = a.scale * kLog2e;
        const int dd = D == 64 ? 16 * qr + lane : 32 * qr + lane;
        const bool valid = D == 64 ? lane < 16 : true;
        const int cq = tw >> 3, cpart = tw & 7;  // pooled role: query, chunk
        unsigned char* DS = dsbuf + w * C::DS_BYTES;
        unsigned char* BCs = bcbuf + w * 2 * C::BC_BYTES;  // dS_c; P_c follows
        for (long long bl = w; bl < mine; bl += 2) {
            const long long g = blockIdx.x + bl * G;
            const uint32_t j = (uint32_t)(bl >> 1);
            const int st = (int)(bl % C::STAGES);
            const long long tok0 = g * 16;  // slice * n + i * B (n = T * B)
            const unsigned char* sb = stages + st * C::STAGE_BYTES;
            const float* sKc = reinterpret_cast<const float*>(sb + C::OFF_C);
            const float* sLse = reinterpret_cast<const float*>(sb + C::OFF_L);
            // waits return at once after a timeout; the group keeps walking the
            // same barriers so that no thread waits on another
            mbar_wait(smem_u32(&ms->q_ready[w]), j & 1, abort_flag, a.status, a.spin);
            // D_t = dO_t . o_t and the pooled-key dots q_t . k_l, dO_t . v_l:
            // eight threads per query, one 16-byte chunk per 64 columns each
            {
                float dsa = 0.f, sa[4] = {0.f, 0.f, 0.f, 0.f}, pa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int cc = 0; cc < D / 64; cc++) {
                    const int c8 = cpart + 8 * cc;
                    const uint32_t off = sw128_offset(cq, c8 * 8, 16);
                    const uint4 q4 = *reinterpret_cast<const uint4*>(sb + off);
                    const uint4 g4 = *reinterpret_cast<const uint4*>(sb + C::OFF_DO + off);
                    const uint4 o4 = *reinterpret_cast<const uint4*>(sb + C::OFF_O + off);
                    const __nv_bfloat162* qh = reinterpret_cast<const __nv_bfloat162*>(&q4);
                    const __nv_bfloat162* gh = reinterpret_cast<const __nv_bfloat162*>(&g4);
                    const __nv_bfloat162* oh = reinterpret_cast<const __nv_bfloat162*>(&o4);
                    float qf[8], gf[8];
#pragma unroll
                    for (int h = 0; h < 4; h++) {
                        const float2 qv = __bfloat1622float2(qh[h]), gv = __bfloat1622float2(gh[h]);
                        const float2 ov = __bfloat1622float2(oh[h]);
                        qf[2 * h] = qv.x; qf[2 * h + 1] = qv.y;
                        gf[2 * h] = gv.x; gf[2 * h + 1] = gv.y;
                        dsa = fmaf(gv.x, ov.x, dsa);
                        dsa = fmaf(gv.y, ov.y, dsa);
                    }
#pragma unroll
                    for (int l = 0; l < 4; l++)
                        if (l < Le) {
                            const float4 k0 = *reinterpret_cast<const float4*>(sKc + l * D + c8 * 8);
                            const float4 k1 = *reinterpret_cast<const float4*>(sKc + l * D + c8 * 8 + 4);
                            const float4 v0 = *reinterpret_cast<const float4*>(sKc + (4 + l) * D + c8 * 8);
                            const float4 v1 = *reinterpret_cast<const float4*>(sKc + (4 + l) * D + c8 * 8 + 4);
                            sa[l] = fmaf(qf[0], k0.x, sa[l]); sa[l] = fmaf(qf[1], k0.y, sa[l]);
                            sa[l] = fmaf(qf[2], k0.z, sa[l]); sa[l] = fmaf(qf[3], k0.w, sa[l]);
                            sa[l] = fmaf(qf[4], k1.x, sa[l]); sa[l] = fmaf(qf[5], k1.y, sa[l]);
                            sa[l] = fmaf(qf[6], k1.z, sa[l]); sa[l] = fmaf(qf[7], k1.w, sa[l]);
                            pa[l] = fmaf(gf[0], v0.x, pa[l]); pa[l] = fmaf(gf[1], v0.y, pa[l]);
                            pa[l] = fmaf(gf[2], v0.z, pa[l]); pa[l] = fmaf(gf[3], v0.w, pa[l]);
                            pa[l] = fmaf(gf[4], v1.x, pa[l]); pa[l] = fmaf(gf[5], v1.y, pa[l]);
                            pa[l] = fmaf(gf[6], v1.z, pa[l]); pa[l] = fmaf(gf[7], v1.w, pa[l]);
                        }
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    dsa += __shfl_xor_sync(0xffffffffu, dsa, o);
#pragma unroll
                    for (int l = 0; l < 4; l++) {
                        sa[l] += __shfl_xor_sync(0xffffffffu, sa[l], o);
                        pa[l] += __shfl_xor_sync(0xffffffffu, pa[l], o);
                    }
                }
                const float lq = sLse[cq];
                float pc = 0.f, dsc = 0.f;  // this thread's level: cpart (< 4)
#pragma unroll
                for (int l = 0; l < 4; l++) {
                    const float s = sc * sa[l] + (float)(l + 1) * a.lnB;
                    const float p = l < Le ? ex2((s - lq) * kLog2e) : 0.f;
                    if (l == cpart) {
                        pc = p;
                        dsc = p * (pa[l] - dsa);
                    }
                }
                if (cpart == 0) {
                    ms->dsum[w][cq] = dsa;
                    // (lse, D) pairs: the key-major kernel fetches both with one copy
                    *reinterpret_cast<float2*>(a.Dbuf + 2 * (tok0 + cq)) = make_float2(lq, dsa);
                }
                if (cpart < 4) {
                    ms->cds[w][j & 1][cq][cpart] = dsc;
                    const uint32_t bo = sw128_offset(cpart, cq, 16);
                    *reinterpret_cast<__nv_bfloat16*>(BCs + bo) = __float2bfloat16_rn(dsc);
                    *reinterpret_cast<__nv_bfloat16*>(BCs + C::BC_BYTES + bo) = __float2bfloat16_rn(pc);
                }
            }
            // this thread's column of the pooled K rows (for dq's pooled term)
            float kc[4];
#pragma unroll
            for (int l = 0; l < 4; l++) kc[l] = (l < Le && valid) ? sKc[l * D + dd] : 0.f;
            named_barrier(1 + w, 128);
            // dS^T for the fine keys from S^T and dP^T
            float lse2[16], dsm[16];
#pragma unroll
            for (int c = 0; c < 16; c += 4) {
                const float4 l4 = *reinterpret_cast<const float4*>(sLse + c);
                const float4 d4 = *reinterpret_cast<const float4*>(&ms->dsum[w][c]);
                lse2[c] = l4.x * kLog2e; lse2[c + 1] = l4.y * kLog2e; lse2[c + 2] = l4.z * kLog2e; lse2[c + 3] = l4.w * kLog2e;
                dsm[c] = d4.x; dsm[c + 1] = d4.y; dsm[c + 2] = d4.z; dsm[c + 3] = d4.w;
            }
            mbar_wait(smem_u32(&ms->s_full[w]), j & 1, abort_flag, a.status, a.spin);
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < NT; t++) {
                float s[16], dp[16];
                tmem_ld16(tS + t * 16, s);
                tmem_ld16(tS + C::TM_DP + t * 16, dp);
                // an M = 128 tile holds key qr * 32 + lane in this thread's TMEM
                // lane; an M = 64 tile (K_1 = 4) holds key 16 qr + lane in lanes
                // 0-15 of each quarter
                const int key = C::MT == 128 ? t * 128 + qr * 32 + lane : 16 * qr + lane;
                if (C::MT != 128 && lane >= 16) continue;
                unsigned char* db = DS + (key >> 6) * 2048 + (key & 7) * 2;
                const int chk = (key & 63) >> 3;
#pragma unroll
                for (int c = 0; c < 16; c++) {
                    const float p = ex2(fmaf(s[c], scl2, -lse2[c]));
                    *reinterpret_cast<__nv_bfloat16*>(db + c * 128 + ((chk ^ (c & 7)) << 4)) =
                        __float2bfloat16_rn(p * (dp[c] - dsm[c]));
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&ms->s_free[w]));
            fence_async_smem();
            mbar_arrive(smem_u32(&ms->ds_full[w]));
            // epilogue: dq^T plus the pooled keys' term, times scale; the
            // pooled-level partial gradients of this block
            mbar_wait(smem_u32(&ms->g_full[w]), j & 1, abort_flag, a.status, a.spin);
            tc_fence_after();
            float q[16], gk[16], gv[16];
            tmem_ld16(tS + C::TM_DQ, q);
            tmem_ld16(tS + C::TM_GK, gk);
            tmem_ld16(tS + C::TM_GV, gv);
            tc_fence_before();
            mbar_arrive(smem_u32(&ms->o_free[w]));
            if (valid) {
                // the block's rows: tok0 .. +15 in tile order, a 4 x 4 patch in raster order
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dq) + tok0 * D + dd;
                if constexpr (R) {
                    const long long sl = g / a.T;
                    dst = static_cast<__nv_bfloat16*>(a.dq) + token_row(sl, a.n, 1, a.side, (int)(tok0 - sl * a.n)) * D + dd;
                }
#pragma unroll
                for (int c = 0; c < 16; c++) {
                    const float4 g4 = *reinterpret_cast<const float4*>(ms->cds[w][j & 1][c]);
                    float val = q[c];
                    val = fmaf(g4.x, kc[0], val);
                    val = fmaf(g4.y, kc[1], val);
                    val = fmaf(g4.z, kc[2], val);
                    val = fmaf(g4.w, kc[3], val);
                    if constexpr (R) dst[block_token_offset(c, a.side) * D] = __float2bfloat16_rn(sc * val);
                    else dst[c * D] = __float2bfloat16_rn(sc * val);
                }
                const long long off = g * (long long)a.Le * D + dd;
#pragma unroll
                for (int l = 0; l < 4; l++)
                    if (l < Le) {
                        a.gK[off + (long long)l * D] = sc * gk[l];
                        a.gV[off + (long long)l * D] = gv[l];
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

template <int D, int NF, bool R>
int launch_one(const Shape& s, const AttnArgs& a, const CUtensorMap* maps, cudaStream_t st) {
    using C = Cfg<D, NF>;
    static_assert(C::SMEM <= 227 * 1024, "shared memory budget");
    static_assert(sizeof(Misc) <= 4096, "misc block");
    static_assert(C::STAGES >= 1, "one stage at least");
    cudaFuncSetAttribute(bwd_dq_tc_kernel<D, NF, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    const long long total = s.slices * (long long)s.T;
    const int grid = (int)std::min<long long>(total, (long long)sm_count());
    LLSA_LAUNCH("bwd_dq_tc", st,
                bwd_dq_tc_kernel<D, NF, R><<<grid, kThreads, C::SMEM, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], a));
    return LLSA_OK;
}

// each built once per token order
template <int D, int NF>
int launch_cfg(const Shape& s, const AttnArgs& a, const CUtensorMap* maps, cudaStream_t st) {
    return s.raster ? launch_one<D, NF, true>(s, a, maps, st) : launch_one<D, NF, false>(s, a, maps, st);
}

}  // namespace

int launch_bwd_dq_tc(const Shape& s, const AttnArgs& a, cudaStream_t st) {
    CUtensorMap maps[5];
    const void* bases[5] = {a.q, a.dout, a.o, a.k, a.v};
    for (int t = 0; t < 5; t++) LLSA_TRY(make_tmap_tokens(&maps[t], bases[t], s));
    if (s.d == 64) {
        if (s.K1 == 4) return launch_cfg<64, 64>(s, a, maps, st);
        if (s.K1 == 32) return launch_cfg<64, 512>(s, a, maps, st);
        return s.K1 == 8 ? launch_cfg<64, 128>(s, a, maps, st) : launch_cfg<64, 256>(s, a, maps, st);
    }
    if (s.K1 == 4) return launch_cfg<128, 64>(s, a, maps, st);
    return s.K1 == 8 ? launch_cfg<128, 128>(s, a, maps, st) : launch_cfg<128, 256>(s, a, maps, st);
}

bool bwd_tc_supported(const Shape& s) {
    return s.dtype == LLSA_DTYPE_BF16 && s.B == 16 && (s.d == 64 || s.d == 128) &&
           (s.K1 == 4 || s.K1 == 8 || s.K1 == 16 || (s.K1 == 32 && s.d == 64)) && s.Le <= 4 && s.Lc == s.Le &&
           s.slices * (long long)s.n < (1LL << 31) && bwd_dkv_tc_fits(s);
}

}  // namespace llsa
