// attn_bwd_dq_tc.cu -- backward, query-major part, on the tcgen05 tensor cores
// (bf16, B = 16, d in {64, 128}, K_1 in {8, 16}): dq, D = rowsum(dO o) (stored
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
// dP^T = V_sel dO^T (M = 128 keys per tile, N = 16 queries), dS^T computed per
// TMEM lane and stored as the K-major operand, then dq^T = K_sel^T dS^T with
// the same K tile read as an MN-major operand (M = d, N = 16, K = keys). The
// softmax needs no reduction here: lse is known.
//
// Warp roles as in the forward: up to three gather warps (TMA boxes for Q, dO,
// o and the selected K and V blocks; bulk copies for pooled rows and lse),
// one MMA thread, two warpgroups alternating query blocks.
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
    static constexpr int NF = NT * 128;
    static constexpr int REG = D / 64;
    static constexpr int CH = D / 8;
    static constexpr int Q_BYTES = 16 * D * 2;
    static constexpr int KV_BYTES = NF * D * 2;
    static constexpr int CO_BYTES = 2 * 4 * D * 4;  // pooled K and V rows (fp32)
    // Q, dO, o, K, V, pooled rows, lse (64 B, padded)
    static constexpr int OFF_DO = Q_BYTES, OFF_O = 2 * Q_BYTES, OFF_K = 3 * Q_BYTES;
    static constexpr int OFF_V = OFF_K + KV_BYTES, OFF_C = OFF_V + KV_BYTES, OFF_L = OFF_C + CO_BYTES;
    static constexpr int STAGE_BYTES = OFF_L + 1024;
    static constexpr int DS_BYTES = 16 * NF * 2;  // per warpgroup
    static constexpr int FIXED = 2 * DS_BYTES + 4096;
    static constexpr int STAGES_RAW = (kSmemBudget - FIXED) / STAGE_BYTES;
    static constexpr int NPROD = STAGES_RAW >= 3 ? 3 : (STAGES_RAW >= 2 ? 2 : 1);
    static constexpr int SPP = (STAGES_RAW < 1 ? 1 : (STAGES_RAW > 6 ? 6 : STAGES_RAW)) / NPROD;
    static constexpr int STAGES = NPROD * SPP;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + FIXED;
    static constexpr int TM_GROUP = 128;  // per warpgroup: S at +0, dP at +32, dq at +64
};

template <class C>
__device__ __forceinline__ void stage_of(int bl, int& st, int& u) {
    const int k = bl / C::NPROD;
    st = (bl % C::NPROD) * C::SPP + k % C::SPP;
    u = k / C::SPP;
}

struct Misc {
    float dsum[2][16];       // D_t
    float cp[2][16][4];      // pooled-key P
    float cds[2][16][4];     // pooled-key dS
    uint64_t full[6], empty[6], q_ready[2], s_full[2], ds_full[2], dq_full[2], s_free[2], o_free[2], drain;
    uint32_t tmem_slot;
    int abort_flag;
};

__device__ __forceinline__ float bf16_at(const unsigned char* tile, int row, int col) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + sw128_offset(row, col, 16)));
}

template <int D, int NT>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mdo,
                 const __grid_constant__ CUtensorMap mo, const __grid_constant__ CUtensorMap mk,
                 const __grid_constant__ CUtensorMap mv, AttnArgs a) {
    using C = Cfg<D, NT>;
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned base (128-byte swizzle atoms), derived from the
    // __shared__ array by pointer arithmetic so accesses stay shared-space
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* stages = sm;
    unsigned char* dsbuf = stages + C::STAGES * C::STAGE_BYTES;
    Misc* ms = reinterpret_cast<Misc*>(dsbuf + 2 * C::DS_BYTES);
    volatile int* abort_flag = &ms->abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long total = a.slices * (long long)a.T;
    const int G = gridDim.x;
    const int K1 = NT * 8, Le = a.Le;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; s++) {
            mbar_init(smem_u32(&ms->full[s]), 1);
            mbar_init(smem_u32(&ms->empty[s]), 1);
        }
        for (int w = 0; w < 2; w++) {
            mbar_init(smem_u32(&ms->q_ready[w]), 1);
            mbar_init(smem_u32(&ms->s_full[w]), 1);
            mbar_init(smem_u32(&ms->ds_full[w]), 128);
            mbar_init(smem_u32(&ms->dq_full[w]), 1);
            mbar_init(smem_u32(&ms->s_free[w]), 128);
            mbar_init(smem_u32(&ms->o_free[w]), 128);
        }
        mbar_init(smem_u32(&ms->drain), 1);
        ms->abort_flag = 0;
        fence_mbar_init();
    }
    for (int x = threadIdx.x; x < 2 * 16 * 4; x += kThreads) {
        (&ms->cp[0][0][0])[x] = 0.f;
        (&ms->cds[0][0][0])[x] = 0.f;
    }
    if (warp == 1) tmem_alloc(smem_u32(&ms->tmem_slot), 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = ms->tmem_slot;

    if ((warp == 0 || warp == 2 || warp == 3) && (warp == 0 ? 0 : warp - 1) < C::NPROD) {
        // ----------------------------------------------------------- gather
        const int pw = warp == 0 ? 0 : warp - 1;
        auto load_idx = [&](int bl, int& jb, int& ce) {
            const long long g = blockIdx.x + (long long)bl * G;
            jb = 0;
            ce = 0;
            if (g >= total) return;
            const long long slice = g / a.T;
            const int i = (int)(g - slice * a.T);
            if (lane < K1) jb = a.sel[(slice * a.T + i) * a.K1 + lane];
            if (lane < Le) ce = a.coarse[(slice * a.T + i) * a.L + lane];
        };
        int jb0, ce0, jb1, ce1;
        load_idx(pw, jb0, ce0);
        load_idx(pw + C::NPROD, jb1, ce1);
        int issued = -1;
        for (int bl = pw;; bl += C::NPROD) {
            const long long g = blockIdx.x + (long long)bl * G;
            if (g >= total) break;
            int jb = jb0, e = ce0;
            jb0 = jb1;
            ce0 = ce1;
            load_idx(bl + 2 * C::NPROD, jb1, ce1);
            int st, u;
            stage_of<C>(bl, st, u);
            bool ok = true;
            if (u >= 1 && lane == 0) ok = mbar_wait(smem_u32(&ms->empty[st]), (u - 1) & 1, abort_flag, a.status);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0);
            if (!ok) break;
            const long long slice = g / a.T;
            const int i = (int)(g - slice * a.T);
            unsigned char* sb = stages + st * C::STAGE_BYTES;
            const uint32_t fb = smem_u32(&ms->full[st]);
            if (lane == 0) mbar_arrive_expect_tx(fb, 3 * C::Q_BYTES + 2 * C::KV_BYTES + 2 * Le * D * 4 + 64);
            __syncwarp();
            const long long tok0 = slice * a.n + (long long)i * 16;
            if (lane == 0) {
                for (int r = 0; r < C::REG; r++) {
                    tma_load_2d(smem_u32(sb + r * 2048), &mq, r * 64, (int)tok0, fb);
                    tma_load_2d(smem_u32(sb + C::OFF_DO + r * 2048), &mdo, r * 64, (int)tok0, fb);
                    tma_load_2d(smem_u32(sb + C::OFF_O + r * 2048), &mo, r * 64, (int)tok0, fb);
                }
                bulk_load(smem_u32(sb + C::OFF_L), a.lse_in + tok0, 64, fb);
            }
            if (lane < K1) {
                if (jb < 0 || jb >= a.T) {
                    set_status(a.status, LLSA_ERR_BAD_INDEX);
                    jb = 0;
                }
                const int yk = (int)(slice * a.n + (long long)jb * 16);
                for (int r = 0; r < C::REG; r++) {
                    tma_load_2d(smem_u32(sb + C::OFF_K + r * C::NF * 128 + lane * 2048), &mk, r * 64, yk, fb);
                    tma_load_2d(smem_u32(sb + C::OFF_V + r * C::NF * 128 + lane * 2048), &mv, r * 64, yk, fb);
                }
            }
            if (lane < Le) {
                if (e < 0 || e >= a.lv.n_level[lane + 1]) {
                    set_status(a.status, LLSA_ERR_BAD_INDEX);
                    e = 0;
                }
                const long long row = slice * a.pyr_stride + (long long)(a.lv.row_offset[lane + 1] + e) * D;
                bulk_load(smem_u32(sb + C::OFF_C + lane * D * 4), a.kpyr + row, D * 4, fb);
                bulk_load(smem_u32(sb + C::OFF_C + (4 + lane) * D * 4), a.vpyr + row, D * 4, fb);
            }
            issued = bl;
        }
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
            constexpr uint32_t idQ = idesc_bf16(D, 16, 1, 0);
            const uint64_t dKm = desc_sw128(smem_u32(stages), 16, 1024);            // K-major
            const uint64_t dMN = desc_sw128(smem_u32(stages), C::NF * 128, 1024);   // K tile as MN-major
            const uint64_t dDS = desc_sw128(smem_u32(dsbuf), 16, 1024);
            auto issue_S = [&](int bl) -> bool {
                const int w = bl & 1, j = bl >> 1;
                int st, u;
                stage_of<C>(bl, st, u);
                if (!mbar_wait(smem_u32(&ms->full[st]), u & 1, abort_flag, a.status)) return false;
                mbar_arrive(smem_u32(&ms->q_ready[w]));
                if (j >= 1 && !mbar_wait(smem_u32(&ms->s_free[w]), (j - 1) & 1, abort_flag, a.status)) return false;
                tc_fence_after();
                const uint32_t s0 = (uint32_t)(st * C::STAGE_BYTES);
#pragma unroll
                for (int t = 0; t < NT; t++)
#pragma unroll
                    for (int ks = 0; ks < D / 16; ks++) {
                        const uint32_t koff = (ks / 4) * C::NF * 128 + t * 128 * 128 + (ks % 4) * 32;
                        const uint32_t qoff = (ks / 4) * 2048 + (ks % 4) * 32;
                        mma_bf16(tbase + w * C::TM_GROUP + t * 16, dKm + ((s0 + C::OFF_K + koff) >> 4),
                                 dKm + ((s0 + qoff) >> 4), idS, ks > 0);
                        mma_bf16(tbase + w * C::TM_GROUP + 32 + t * 16, dKm + ((s0 + C::OFF_V + koff) >> 4),
                                 dKm + ((s0 + C::OFF_DO + qoff) >> 4), idS, ks > 0);
                    }
                mma_commit(smem_u32(&ms->s_full[w]));
                return true;
            };
            auto issue_DQ = [&](int bl) -> bool {
                const int w = bl & 1, j = bl >> 1;
                int st, u;
                stage_of<C>(bl, st, u);
                if (!mbar_wait(smem_u32(&ms->ds_full[w]), j & 1, abort_flag, a.status)) return false;
                if (j >= 1 && !mbar_wait(smem_u32(&ms->o_free[w]), (j - 1) & 1, abort_flag, a.status)) return false;
                tc_fence_after();
                const uint32_t k0 = (uint32_t)(st * C::STAGE_BYTES + C::OFF_K);
                const uint32_t d0 = (uint32_t)(w * C::DS_BYTES);
#pragma unroll
                for (int ks = 0; ks < C::NF / 16; ks++)
                    mma_bf16(tbase + w * C::TM_GROUP + 64, dMN + ((k0 + ks * 2048) >> 4),
                             dDS + ((d0 + (ks / 4) * 2048 + (ks % 4) * 32) >> 4), idQ, ks > 0);
                mma_commit(smem_u32(&ms->dq_full[w]));
                mma_commit(smem_u32(&ms->empty[st]));
                return true;
            };
            const long long mine = total > blockIdx.x ? (total - blockIdx.x + G - 1) / G : 0;
            bool ok = true;
            if (C::STAGES >= 2) {
                ok = mine > 0 ? issue_S(0) : true;
                for (long long bl = 0; ok && bl < mine; bl++) {
                    if (bl + 1 < mine) ok = issue_S((int)bl + 1);
                    if (ok) ok = issue_DQ((int)bl);
                }
            } else {
                for (long long bl = 0; ok && bl < mine; bl++) {
                    ok = issue_S((int)bl);
                    if (ok) ok = issue_DQ((int)bl);
                }
            }
            mma_commit(smem_u32(&ms->drain));
            for (int it = 0; it < kSpinLimit && !mbar_try(smem_u32(&ms->drain), 0); it++) {
            }
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
        const int pi = tw >> 1, half = tw & 1;
        const bool pact = pi < 16 * Le;
        const int pq = pact ? pi / Le : 0, pl = pact ? pi % Le : 0;
        unsigned char* DS = dsbuf + w * C::DS_BYTES;
        for (int bl = w;; bl += 2) {
            const long long g = blockIdx.x + (long long)bl * G;
            if (g >= total) break;
            const int j = bl >> 1;
            int st, u;
            stage_of<C>(bl, st, u);
            const long long slice = g / a.T;
            const int i = (int)(g - slice * a.T);
            const long long tok0 = slice * a.n + (long long)i * 16;
            const unsigned char* sb = stages + st * C::STAGE_BYTES;
            const float* sKc = reinterpret_cast<const float*>(sb + C::OFF_C);
            const float* sLse = reinterpret_cast<const float*>(sb + C::OFF_L);
            // waits return at once after a timeout; the group keeps walking the
            // same barriers so that no thread waits on another
            mbar_wait(smem_u32(&ms->q_ready[w]), j & 1, abort_flag, a.status);
            // D_t = dO_t . o_t: eight threads per row, D/64 chunks of 8 each
            {
                const int row = tw >> 3, part = tw & 7;
                float acc = 0.f;
#pragma unroll
                for (int c8 = part; c8 < C::CH; c8 += 8) {
                    const uint4 g4 = *reinterpret_cast<const uint4*>(sb + C::OFF_DO + sw128_offset(row, c8 * 8, 16));
                    const uint4 o4 = *reinterpret_cast<const uint4*>(sb + C::OFF_O + sw128_offset(row, c8 * 8, 16));
                    const __nv_bfloat162* gh = reinterpret_cast<const __nv_bfloat162*>(&g4);
                    const __nv_bfloat162* oh = reinterpret_cast<const __nv_bfloat162*>(&o4);
#pragma unroll
                    for (int h = 0; h < 4; h++) {
                        const float2 gf = __bfloat1622float2(gh[h]), of = __bfloat1622float2(oh[h]);
                        acc = fmaf(gf.x, of.x, acc);
                        acc = fmaf(gf.y, of.y, acc);
                    }
                }
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                acc += __shfl_xor_sync(0xffffffffu, acc, 4);
                if (part == 0) {
                    ms->dsum[w][row] = acc;
                    // (lse, D) pairs: the key-major kernel fetches both with one copy
                    *reinterpret_cast<float2*>(a.Dbuf + 2 * (tok0 + row)) = make_float2(sLse[row], acc);
                }
            }
            // this thread's column of the pooled K rows (for dq's pooled term)
            float kc[4];
#pragma unroll
            for (int l = 0; l < 4; l++) kc[l] = (l < Le && valid) ? sKc[l * D + dd] : 0.f;
            named_barrier(1 + w, 128);
            // pooled keys: two threads per (query, level)
            {
                float s0 = 0.f, s1 = 0.f, p0 = 0.f, p1 = 0.f;
                if (pact) {
                    const float* kr = sKc + pl * D;
                    const float* vr = sKc + (4 + pl) * D;
#pragma unroll
                    for (int c8 = half * C::CH / 2; c8 < (half + 1) * C::CH / 2; c8++) {
                        const uint4 q4 = *reinterpret_cast<const uint4*>(sb + sw128_offset(pq, c8 * 8, 16));
                        const uint4 g4 = *reinterpret_cast<const uint4*>(sb + C::OFF_DO + sw128_offset(pq, c8 * 8, 16));
                        const __nv_bfloat162* qh = reinterpret_cast<const __nv_bfloat162*>(&q4);
                        const __nv_bfloat162* gh = reinterpret_cast<const __nv_bfloat162*>(&g4);
#pragma unroll
                        for (int h = 0; h < 4; h++) {
                            const float2 qf = __bfloat1622float2(qh[h]), gf = __bfloat1622float2(gh[h]);
                            const float2 kf = *reinterpret_cast<const float2*>(kr + c8 * 8 + 2 * h);
                            const float2 vf = *reinterpret_cast<const float2*>(vr + c8 * 8 + 2 * h);
                            s0 = fmaf(qf.x, kf.x, s0); s1 = fmaf(qf.y, kf.y, s1);
                            p0 = fmaf(gf.x, vf.x, p0); p1 = fmaf(gf.y, vf.y, p1);
                        }
                    }
                }
                float sdot = s0 + s1, pdot = p0 + p1;
                sdot += __shfl_xor_sync(0xffffffffu, sdot, 1);
                pdot += __shfl_xor_sync(0xffffffffu, pdot, 1);
                if (pact && half == 0) {
                    const float s = sc * sdot + (float)(pl + 1) * a.lnB;
                    const float p = ex2((s - sLse[pq]) * kLog2e);
                    ms->cp[w][pq][pl] = p;
                    ms->cds[w][pq][pl] = p * (pdot - ms->dsum[w][pq]);
                }
            }
            named_barrier(1 + w, 128);
            // partial gradients of the pooled keys and values of this block:
            // gK = scale * sum_t dS_t q_t, gV = sum_t P_t dO_t
            for (int it = tw; it < Le * D; it += 128) {
                const int l = it / D, c = it % D;
                float gk = 0.f, gv = 0.f;
#pragma unroll
                for (int t = 0; t < 16; t++) {
                    gk = fmaf(ms->cds[w][t][l], bf16_at(sb, t, c), gk);
                    gv = fmaf(ms->cp[w][t][l], bf16_at(sb + C::OFF_DO, t, c), gv);
                }
                const long long off = ((slice * a.T + i) * a.Le + l) * (long long)D + c;
                a.gK[off] = sc * gk;
                a.gV[off] = gv;
            }
            // dS^T for the fine keys from S^T and dP^T
            float lse2[16], dsm[16];
#pragma unroll
            for (int c = 0; c < 16; c += 4) {
                const float4 l4 = *reinterpret_cast<const float4*>(sLse + c);
                const float4 d4 = *reinterpret_cast<const float4*>(&ms->dsum[w][c]);
                lse2[c] = l4.x * kLog2e; lse2[c + 1] = l4.y * kLog2e; lse2[c + 2] = l4.z * kLog2e; lse2[c + 3] = l4.w * kLog2e;
                dsm[c] = d4.x; dsm[c + 1] = d4.y; dsm[c + 2] = d4.z; dsm[c + 3] = d4.w;
            }
            mbar_wait(smem_u32(&ms->s_full[w]), j & 1, abort_flag, a.status);
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < NT; t++) {
                float s[16], dp[16];
                tmem_ld16(tS + t * 16, s);
                tmem_ld16(tS + 32 + t * 16, dp);
                const int key = t * 128 + qr * 32 + lane;
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
            // epilogue: dq^T from TMEM plus the pooled keys' term, times scale
            mbar_wait(smem_u32(&ms->dq_full[w]), j & 1, abort_flag, a.status);
            tc_fence_after();
            float q[16];
            tmem_ld16(tS + 64, q);
            tc_fence_before();
            mbar_arrive(smem_u32(&ms->o_free[w]));
            if (valid) {
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dq) + tok0 * D + dd;
#pragma unroll
                for (int c = 0; c < 16; c++) {
                    const float4 g4 = *reinterpret_cast<const float4*>(ms->cds[w][c]);
                    float val = q[c];
                    val = fmaf(g4.x, kc[0], val);
                    val = fmaf(g4.y, kc[1], val);
                    val = fmaf(g4.z, kc[2], val);
                    val = fmaf(g4.w, kc[3], val);
                    dst[c * D] = __float2bfloat16_rn(sc * val);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 256);
    }
}

template <int D, int NT>
int launch_cfg(const Shape& s, const AttnArgs& a, const CUtensorMap* maps, cudaStream_t st) {
    using C = Cfg<D, NT>;
    static_assert(C::SMEM <= 227 * 1024, "shared memory budget");
    static_assert(sizeof(Misc) <= 4096, "misc block");
    cudaFuncSetAttribute(bwd_dq_tc_kernel<D, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    const long long total = s.slices * (long long)s.T;
    const int grid = (int)std::min<long long>(total, (long long)sm_count());
    LLSA_LAUNCH("bwd_dq_tc", st,
                bwd_dq_tc_kernel<D, NT><<<grid, kThreads, C::SMEM, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4], a));
    return LLSA_OK;
}

}  // namespace

int launch_bwd_dq_tc(const Shape& s, const AttnArgs& a, cudaStream_t st) {
    CUtensorMap maps[5];
    const long long rows = s.slices * (long long)s.n;
    const void* bases[5] = {a.q, a.dout, a.o, a.k, a.v};
    for (int t = 0; t < 5; t++) LLSA_TRY(make_tmap_bf16(&maps[t], bases[t], rows, s.d, 16));
    if (s.d == 64) return s.K1 == 8 ? launch_cfg<64, 1>(s, a, maps, st) : launch_cfg<64, 2>(s, a, maps, st);
    return s.K1 == 8 ? launch_cfg<128, 1>(s, a, maps, st) : launch_cfg<128, 2>(s, a, maps, st);
}

}  // namespace llsa
