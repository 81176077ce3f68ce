// attn_bwd_dkv_tc.cu -- backward, key-major part, on the tcgen05 tensor cores
// (bf16, B = 16, d in {64, 128}): dk, dv of every fine key block from the
// query blocks that selected it, plus the pooled-level gradients.
//
// Method: Pith review of arXiv 2512.16615, "What carries the argument" (the
// sparse-index transpose gives each key block its query blocks without a
// dense N x N mask) and the referee's Sec. 4.3 / Figure 4 comments (sparse
// key-value backward). For fine key block j and every query block i in CSC
// column j: dv_j += P^T dO_i, dk_j += scale dS^T q_i, with P and dS recomputed
// from q, k, v, dO, lse and D. Then dk_t += sum_l dK^(l)[anc] / B^l (and dv
// likewise) for the pooled tokens above j.
//
// The column's query blocks are stacked eight at a time (M = 128 query rows):
// S = Q_stack K_j^T and dP = dO_stack V_j^T (N = 16 keys), one TMEM lane per
// query row, so P and dS need only that row's lse and D; then the gradients
// accumulate in TMEM across the column's groups, in CSC order (deterministic):
// for d = 64 one MMA per 16 rows computes [Q_stack ; dO_stack]^T [dS | P]
// (M = 128, N = 32) whose diagonal blocks are dk^T and dv^T; for d = 128,
// dk^T += Q_stack^T dS and dv^T += dO_stack^T P (M = d, N = 16). Each (key
// block, group of eight) is one item; items follow the key blocks of the CTA
// in order; the two warpgroups take alternate key blocks.
//
// Warp roles: three gather warps split every item's copies (warp 0 K_j and
// V_j; warp 2 the Q stack; warp 3 the dO stack) into a ring of stages, and
// each softmax thread loads its query row's (lse, D) pair itself, one item
// ahead; warp 1 issues the S stream and warp 12 the gradient stream, each in
// order with blocking waits, through an election inside the MMA asm.
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

constexpr int kThreads = 416;  // 13 warps: 3 gather, 2 MMA issuers, 8 in two warpgroups
constexpr int kSmemBudget = 215 * 1024;
constexpr int kMaxKeyBlocks = 2048;  // key blocks per CTA (counts kept in shared memory)
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct Cfg {
    static constexpr int REG = D / 64;
    static constexpr int QS_BYTES = 128 * D * 2;  // eight stacked 16-row query blocks
    static constexpr int KB_BYTES = 16 * D * 2;
    // Q stack, dO stack, K_j, V_j
    static constexpr int OFF_DO = QS_BYTES, OFF_K = 2 * QS_BYTES, OFF_V = OFF_K + KB_BYTES;
    static constexpr int STAGE_BYTES = OFF_V + KB_BYTES;
    // per warpgroup and buffer: dS^T and P^T of one item as K-major operands,
    // interleaved per 64 rows (dS^T chunk c at c * 4096, P^T chunk c at +2048)
    static constexpr int PG_BYTES = 8192;
    static constexpr int FIXED = 4 * PG_BYTES + 4096 + kMaxKeyBlocks * 12;
    static constexpr int STAGES_RAW = (kSmemBudget - FIXED) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 6 ? 6 : STAGES_RAW;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + FIXED;
    // per warpgroup: two S/dP buffers (+0, +32: S, then dP 16 columns on;
    // alternate items of the group) and two gradient accumulators (+64, +96:
    // 32 columns each, alternate key blocks of the group)
    static constexpr int TM_GROUP = 128;
};

struct Misc {
    // per warpgroup, each used in that group's own item order
    // [group][buffer]: item buffers alternate with the group's items,
    // accumulators with its key blocks
    uint64_t full[6], empty[6];
    uint64_t s_full[2][2], s_free[2][2], p_full[2][2], p_free[2][2];
    uint64_t acc_full[2][2], acc_free[2][2], drain[2];
    uint32_t tmem_slot;
    int abort_flag;
    int n_kb, n_items;
};

// Walks the items of a CTA in order: key block, group (kb & 1), index within
// the key block, per-group item and key-block counters (barrier phases).
struct ItemWalk {
    int n = -1, kb = 0, w = 0, gi = 0, k = 0, kn = 0;
    bool last = false;
    int wk0 = 0, wk1 = 0, wkb0 = 0, wkb1 = 0;  // items / finished key blocks per group
    __device__ __forceinline__ void next(const int* kitem, const int* kcnt, int n_kb) {
        n++;
        while (kb + 1 < n_kb && kitem[kb + 1] <= n) kb++;
        w = kb & 1;
        gi = n - kitem[kb];
        last = 8 * (gi + 1) >= kcnt[kb];
        k = w ? wk1++ : wk0++;
        kn = w ? wkb1 : wkb0;
        if (last) (w ? wkb1 : wkb0)++;
    }
};

template <int D, bool R>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mdo,
                  const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv, AttnArgs a) {
    using C = Cfg<D>;
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned base (128-byte swizzle atoms), derived from the
    // __shared__ array by pointer arithmetic so accesses stay shared-space
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* stages = sm;
    unsigned char* pbuf = stages + C::STAGES * C::STAGE_BYTES;  // [warpgroup][buffer] dS^T / P^T
    Misc* ms = reinterpret_cast<Misc*>(pbuf + 4 * C::PG_BYTES);
    int* kcnt = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(ms) + 4096);  // per key block: column count
    int* kitem = kcnt + kMaxKeyBlocks;                                                  // first item of the key block
    int* kbeg = kitem + kMaxKeyBlocks;                                                  // first CSC entry of the column
    volatile int* abort_flag = &ms->abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long total = a.slices * (long long)a.T;
    const int G = gridDim.x;
    const int n_kb = total > blockIdx.x ? (int)((total - blockIdx.x + G - 1) / G) : 0;

    // stages start zeroed: rows of an item's unused query blocks keep finite
    // values (zeros or an earlier block), so P = dS = 0 there stays exact
    for (int x = threadIdx.x; x < C::STAGES * C::STAGE_BYTES / 16; x += kThreads)
        reinterpret_cast<uint4*>(stages)[x] = make_uint4(0, 0, 0, 0);
    // column counts of this CTA's key blocks and the running item count
    for (int kb = threadIdx.x; kb < n_kb; kb += kThreads) {
        const long long g = blockIdx.x + (long long)kb * G;
        const long long slice = g / a.T;
        const int j = (int)(g - slice * a.T);
        const int* cp = a.col_ptr + slice * (long long)(a.T + 1);
        const int b = cp[j], e = cp[j + 1];
        // a column outside [0, T*K_1] is reported and treated as empty
        const bool good = b >= 0 && e >= b && e <= a.K1 * a.T;
        if (!good) set_status(a.status, LLSA_ERR_BAD_INDEX);
        kcnt[kb] = good ? e - b : 0;
        kbeg[kb] = good ? b : 0;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; s++) {
            mbar_init(smem_u32(&ms->full[s]), 3);  // one arrival per gather warp
            mbar_init(smem_u32(&ms->empty[s]), 1);
        }
        for (int w = 0; w < 2; w++) {
            for (int b = 0; b < 2; b++) {
                mbar_init(smem_u32(&ms->s_full[w][b]), 1);
                mbar_init(smem_u32(&ms->s_free[w][b]), 128);
                mbar_init(smem_u32(&ms->p_full[w][b]), 128);
                mbar_init(smem_u32(&ms->p_free[w][b]), 1);
                mbar_init(smem_u32(&ms->acc_full[w][b]), 1);
                mbar_init(smem_u32(&ms->acc_free[w][b]), 128);
            }
        }
        mbar_init(smem_u32(&ms->drain[0]), 1);
        mbar_init(smem_u32(&ms->drain[1]), 1);
        ms->abort_flag = 0;
        fence_mbar_init();
    }
    fence_async_smem();
    __syncthreads();
    if (warp == 0) {
        // exclusive scan of the item counts (ceil(count / 8)) over key blocks
        int carry = 0;
        for (int base = 0; base < n_kb; base += 32) {
            const int kb = base + lane;
            const int v = kb < n_kb ? (kcnt[kb] + 7) / 8 : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            if (kb < n_kb) kitem[kb] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            ms->n_kb = n_kb;
            ms->n_items = carry;
        }
    }
    if (warp == 1) tmem_alloc(smem_u32(&ms->tmem_slot), 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = ms->tmem_slot;
    const int n_items = ms->n_items;

    if (warp == 0 || warp == 2 || warp == 3) {
        // ----------------------------------------------------------- gather
        // Item n uses stage n % STAGES for the (n / STAGES)-th time. The query
        // blocks of the next item are located while this one is issued.
        const int role = warp == 0 ? 0 : warp - 1;
        // key block kb_walk is global block blockIdx.x + kb_walk * G, i.e.
        // block w_j of slice w_slice (walked, no division per item)
        int kb_walk = 0;
        long long w_slice = blockIdx.x / a.T;
        int w_j = (int)(blockIdx.x - w_slice * a.T);
        auto locate = [&](int n, int& kb, int& nv, int& qb, long long& ksl, int& kj) {
            while (kb_walk + 1 < n_kb && kitem[kb_walk + 1] <= n) {
                kb_walk++;
                w_j += G;
                while (w_j >= a.T) {
                    w_j -= a.T;
                    w_slice++;
                }
            }
            kb = kb_walk;
            ksl = w_slice;
            kj = w_j;
            const int gi = n - kitem[kb];
            nv = min(8, kcnt[kb] - 8 * gi);
            qb = lane < nv ? a.row_idx[w_slice * a.T * a.K1 + kbeg[kb] + 8 * gi + lane] : 0;
        };
        int kb, nv, qb, kb1 = 0, nv1 = 0, qb1 = 0, j, j1 = 0;
        long long slice, slice1 = 0;
        int issued = -1;
        if (n_items > 0) locate(0, kb1, nv1, qb1, slice1, j1);
        const int ni = (a.test_flags & LLSA_TEST_NO_COPIES) ? 0 : n_items;  // failure-detection test
        for (int n = 0; n < ni; n++) {
            kb = kb1; nv = nv1; qb = qb1; slice = slice1; j = j1;
            if (n + 1 < n_items) locate(n + 1, kb1, nv1, qb1, slice1, j1);
            const int st = n % C::STAGES, u = n / C::STAGES;
            bool ok = true;
            if (u >= 1 && lane == 0) ok = mbar_wait(smem_u32(&ms->empty[st]), (u - 1) & 1, abort_flag, a.status, a.spin);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0);
            if (!ok) break;
            if (lane < nv && (qb < 0 || qb >= a.T)) {
                set_status(a.status, LLSA_ERR_BAD_INDEX);
                qb = 0;
            }
            unsigned char* sb = stages + st * C::STAGE_BYTES;
            const uint32_t fb = smem_u32(&ms->full[st]);
            const uint32_t bytes = role == 0 ? 2 * C::KB_BYTES : nv * C::KB_BYTES;
            if (lane == 0) mbar_arrive_expect_tx(fb, bytes);
            __syncwarp();
            const long long tok = slice * a.n + (long long)qb * 16;
            if (role == 0) {
                if (lane == 0) {
                    const int yk = (int)(slice * a.n + (long long)j * 16);
                    for (int r = 0; r < C::REG; r++) {
                        if constexpr (R) {
                            tma_load_block<true>(smem_u32(sb + C::OFF_K + r * 2048), &mk, r * 64, slice, j, a.n, fb);
                            tma_load_block<true>(smem_u32(sb + C::OFF_V + r * 2048), &mv, r * 64, slice, j, a.n, fb);
                        } else {
                            tma_load_2d(smem_u32(sb + C::OFF_K + r * 2048), &mk, r * 64, yk, fb);
                            tma_load_2d(smem_u32(sb + C::OFF_V + r * 2048), &mv, r * 64, yk, fb);
                        }
                    }
                }
            } else if (lane < nv) {
                const int off = role == 1 ? 0 : C::OFF_DO;
                const CUtensorMap* map = role == 1 ? &mq : &mdo;
                for (int r = 0; r < C::REG; r++) {
                    if constexpr (R)
                        tma_load_block<true>(smem_u32(sb + off + r * 128 * 128 + lane * 2048), map, r * 64, slice, qb, a.n, fb);
                    else
                        tma_load_2d(smem_u32(sb + off + r * 128 * 128 + lane * 2048), map, r * 64, (int)tok, fb);
                }
            }
            issued = n;
        }
        // copies still in flight must land before the CTA exits
        if (lane == 0)
            for (int n = issued; n >= 0 && n > issued - C::STAGES; n--) {
                const int st = n % C::STAGES, u = n / C::STAGES;
                for (int it = 0; it < kSpinLimit && !mbar_try(smem_u32(&ms->full[st]), u & 1); it++) {
                }
            }
    } else if (warp == 1 || warp == 12) {
        // ------------------------------------------------------ MMA issuers
        constexpr uint32_t idS = idesc_bf16(128, 16, 0, 0);
        constexpr uint32_t idG = D == 64 ? idesc_bf16(128, 32, 1, 0) : idesc_bf16(D, 16, 1, 0);
        const uint64_t dKm = desc_sw128(smem_u32(stages), 16, 1024);         // K-major
        const uint64_t dMN = desc_sw128(smem_u32(stages), 128 * 128, 1024);  // stacks as MN-major
        const uint64_t dPB = desc_sw128(smem_u32(pbuf), 16, 1024);
        auto issue_S = [&](const ItemWalk& it) {
            const int st = it.n % C::STAGES;
            tc_fence_after();
            const uint32_t s0 = (uint32_t)(st * C::STAGE_BYTES);
            const uint32_t tg = tbase + it.w * C::TM_GROUP + (it.k & 1) * 32;
#pragma unroll
            for (int ks = 0; ks < D / 16; ks++) {
                const uint32_t qoff = (ks / 4) * 128 * 128 + (ks % 4) * 32;
                const uint32_t koff = (ks / 4) * 2048 + (ks % 4) * 32;
                mma_bf16_warp(tg, dKm + ((s0 + qoff) >> 4), dKm + ((s0 + C::OFF_K + koff) >> 4), idS, ks > 0);
                mma_bf16_warp(tg + 16, dKm + ((s0 + C::OFF_DO + qoff) >> 4), dKm + ((s0 + C::OFF_V + koff) >> 4),
                              idS, ks > 0);
            }
            mma_commit_warp(smem_u32(&ms->s_full[it.w][it.k & 1]));
        };
        auto issue_G = [&](const ItemWalk& it) {
            const int st = it.n % C::STAGES;
            tc_fence_after();
            const uint32_t s0 = (uint32_t)(st * C::STAGE_BYTES);
            const uint32_t pg = (uint32_t)((it.w * 2 + (it.k & 1)) * C::PG_BYTES);
            const uint32_t tg = tbase + it.w * C::TM_GROUP + 64 + (it.kn & 1) * 32;
#pragma unroll
            for (int ks = 0; ks < 8; ks++) {
                const uint32_t boff = pg + (ks / 4) * 4096 + (ks % 4) * 32;
                const uint32_t acc = (it.gi > 0 || ks > 0) ? 1u : 0u;
                if (D == 64) {
                    // rows 0-63 Q^T, rows 64-127 dO^T (the dO stack is QS_BYTES on,
                    // the descriptor's M-chunk stride); columns 0-15 dS, 16-31 P
                    mma_bf16_warp(tg, dMN + ((s0 + ks * 2048) >> 4), dPB + (boff >> 4), idG, acc);
                } else {
                    mma_bf16_warp(tg, dMN + ((s0 + ks * 2048) >> 4), dPB + (boff >> 4), idG, acc);
                    mma_bf16_warp(tg + 16, dMN + ((s0 + C::OFF_DO + ks * 2048) >> 4), dPB + ((boff + 2048) >> 4), idG,
                                  acc);
                }
            }
            mma_commit_warp(smem_u32(&ms->p_free[it.w][it.k & 1]));
            mma_commit_warp(smem_u32(&ms->empty[st]));
            if (it.last) mma_commit_warp(smem_u32(&ms->acc_full[it.w][it.kn & 1]));
        };
        // one in-order stream per issuing warp: warp 1 the S stream, warp 12
        // the gradient stream; each waits on its own barriers, lane 0 waiting
        // and broadcasting the outcome
        auto wait1 = [&](uint64_t* bar, uint32_t parity) -> bool {
            int ok = 1;
            if (lane == 0) ok = mbar_wait(smem_u32(bar), parity, abort_flag, a.status, a.spin) ? 1 : 0;
            return __shfl_sync(0xffffffffu, ok, 0) != 0;
        };
        ItemWalk it;
        const bool s_role = warp == 1;
        for (int n = 0; n < n_items; n++) {
            it.next(kitem, kcnt, n_kb);
            const int st = it.n % C::STAGES, u = it.n / C::STAGES;
            if (s_role) {
                if (!wait1(&ms->full[st], u & 1)) break;
                if (it.k >= 2 && !wait1(&ms->s_free[it.w][it.k & 1], ((it.k >> 1) - 1) & 1)) break;
                issue_S(it);
            } else {
                // an accumulator is free once the epilogue of the group's key
                // block before last (its previous user) read it
                if (!wait1(&ms->p_full[it.w][it.k & 1], (it.k >> 1) & 1)) break;
                if (it.gi == 0 && it.kn >= 2 && !wait1(&ms->acc_free[it.w][it.kn & 1], ((it.kn >> 1) - 1) & 1)) break;
                issue_G(it);
            }
        }
        // no MMA of this warp may be in flight when TMEM is released
        mma_commit_warp(smem_u32(&ms->drain[s_role ? 0 : 1]));
        if (lane == 0)
            for (int x = 0; x < kSpinLimit && !mbar_try(smem_u32(&ms->drain[s_role ? 0 : 1]), 0); x++) {
            }
        __syncwarp();
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------ P, dS per query row; epilogue
        const int w = (warp - 4) >> 2, qr = warp & 3;
        const int tq = threadIdx.x - 128 * (1 + w);  // query row of the stack = TMEM lane
        const uint32_t lanes = (uint32_t)(qr * 32) << 16;
        const uint32_t tg = tbase + w * C::TM_GROUP + lanes;
        const float sc = a.scale, scl2 = a.scale * kLog2e;
        // epilogue rows: for d = 64, warps 0-1 of the group hold dk^T rows and
        // warps 2-3 dv^T rows (TMEM lanes 0-63 / 64-127); for d = 128 every
        // warp holds 32 rows of both
        const bool is_k = D == 64 ? qr < 2 : true;
        const int dd = D == 64 ? 32 * (qr & 1) + lane : 32 * qr + lane;
        unsigned char* pb0 = pbuf + w * 2 * C::PG_BYTES + (tq >> 6) * 4096 + (tq & 7) * 2;
        const int chk = (tq & 63) >> 3;
        int kn = 0, k = 0;  // key blocks with items / items of this group so far
        // The epilogue of a key block runs after the first item of the group's
        // next key block (its accumulator is the other one), so its wait on
        // the last gradient MMA and its stores overlap that item.
        bool pend = false, pacc = false;
        long long pslice = 0;
        int pj = 0, pkn = 0;
        float prk[4], prv[4];
        auto epilogue = [&]() {
            // dk = scale * acc + pooled fold, dv = acc + pooled fold
            float kk[16], vv[16];
            if (pacc) {
                mbar_wait(smem_u32(&ms->acc_full[w][pkn & 1]), (pkn >> 1) & 1, abort_flag, a.status, a.spin);
                tc_fence_after();
                const uint32_t ta = tg + 64 + (pkn & 1) * 32;
                if (D == 64) {
                    tmem_ld16(ta + (is_k ? 0 : 16), kk);
#pragma unroll
                    for (int c = 0; c < 16; c++) vv[c] = kk[c];
                } else {
                    tmem_ld16(ta, kk);
                    tmem_ld16(ta + 16, vv);
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&ms->acc_free[w][pkn & 1]));
            } else {
#pragma unroll
                for (int c = 0; c < 16; c++) kk[c] = vv[c] = 0.f;
            }
            float fk = 0.f, fv = 0.f;
            long long span = a.B;  // B^l
#pragma unroll
            for (int l = 0; l < 4; l++) {
                const float inv = 1.0f / (float)span;
                fk = fmaf(prk[l], inv, fk);
                fv = fmaf(prv[l], inv, fv);
                span *= a.B;
            }
            // the block's rows, contiguous in tile order, a 4 x 4 patch in raster order
            long long row0 = (pslice * a.n + (long long)pj * 16) * D + dd;
            if constexpr (R) row0 = token_row(pslice, a.n, 1, a.side, pj * 16) * D + dd;
            if (is_k) {
                __nv_bfloat16* dk = static_cast<__nv_bfloat16*>(a.dk) + row0;
#pragma unroll
                for (int c = 0; c < 16; c++) {
                    if constexpr (R) dk[block_token_offset(c, a.side) * D] = __float2bfloat16_rn(fmaf(sc, kk[c], fk));
                    else dk[c * D] = __float2bfloat16_rn(fmaf(sc, kk[c], fk));
                }
            }
            if (D == 128 || !is_k) {
                __nv_bfloat16* dv = static_cast<__nv_bfloat16*>(a.dv) + row0;
#pragma unroll
                for (int c = 0; c < 16; c++) {
                    if constexpr (R) dv[block_token_offset(c, a.side) * D] = __float2bfloat16_rn(vv[c] + fv);
                    else dv[c * D] = __float2bfloat16_rn(vv[c] + fv);
                }
            }
        };
        // (lse, D) of this thread's query row for one of the group's items,
        // loaded one item ahead of its use, so the two dependent loads (the
        // CSC row, then the pair) hide behind the item before
        auto load_ld = [&](int kb2, int gi2, long long sl2) -> float2 {
            if (kb2 >= n_kb || tq >= 16 * min(8, kcnt[kb2] - 8 * gi2)) return make_float2(0.f, 0.f);
            int qb2 = a.row_idx[sl2 * a.T * a.K1 + kbeg[kb2] + 8 * gi2 + (tq >> 4)];
            if (qb2 < 0 || qb2 >= a.T) qb2 = 0;  // reported by the gather warps
            return *reinterpret_cast<const float2*>(a.Dbuf + 2 * (sl2 * a.n + (long long)qb2 * 16 + (tq & 15)));
        };
        // key block kb of this group is block j of slice `slice`, and its
        // next item's key block kbn block nj of slice nsl (walked by 2 G)
        const long long g0 = blockIdx.x + (long long)w * G;
        long long slice = g0 / a.T, nsl = slice;
        int j = (int)(g0 - slice * a.T), nj = j;
        auto step2 = [&](long long& sl, int& jj) {
            jj += 2 * G;
            while (jj >= a.T) {
                jj -= a.T;
                sl++;
            }
        };
        int kbn = w, gin = 0;  // the group's next item
        while (kbn < n_kb && kcnt[kbn] == 0) {
            kbn += 2;
            step2(nsl, nj);
        }
        float2 ld_next = load_ld(kbn, gin, nsl);
        for (int kb = w; kb < n_kb; kb += 2, step2(slice, j)) {
            const int cnt = kcnt[kb], items = (cnt + 7) / 8;
            // pooled-level gradients above this key block: loaded before its
            // items, combined only in its epilogue so the loads' latency hides
            float rk[4], rv[4];
            {
                int anc = j;
#pragma unroll
                for (int l = 0; l < 4; l++) {
                    rk[l] = rv[l] = 0.f;
                    if (l < a.Le) {
                        const long long off = (slice * a.P + a.lv.row_offset[l + 1] + anc) * (long long)D + dd;
                        if (is_k) rk[l] = a.dKc[off];
                        if (D == 128 || !is_k) rv[l] = a.dVc[off];
                    }
                    anc /= a.B;
                }
            }
            for (int gi = 0; gi < items; gi++, k++) {
                const bool row_ok = tq < 16 * min(8, cnt - 8 * gi);
                // waits return at once after a timeout; the group keeps walking
                const int b = k & 1;
                const uint32_t ph = (uint32_t)(k >> 1) & 1;
                const float2 ld = ld_next;  // (lse, D)
                if (8 * (gin + 1) < kcnt[kbn]) {
                    gin++;
                } else {
                    gin = 0;
                    do {
                        kbn += 2;
                        step2(nsl, nj);
                    } while (kbn < n_kb && kcnt[kbn] == 0);
                }
                ld_next = load_ld(kbn, gin, nsl);
                const float lse2 = ld.x * kLog2e, Dq = ld.y;
                mbar_wait(smem_u32(&ms->s_full[w][b]), ph, abort_flag, a.status, a.spin);
                tc_fence_after();
                float s[16], dp[16];
                tmem_ld16(tg + b * 32, s);
                tmem_ld16(tg + b * 32 + 16, dp);
                tc_fence_before();
                mbar_arrive(smem_u32(&ms->s_free[w][b]));
                // the operands of this group's item before last (same buffer) must be consumed
                if (k >= 2) mbar_wait(smem_u32(&ms->p_free[w][b]), ph ^ 1u, abort_flag, a.status, a.spin);
                unsigned char* pb = pb0 + b * C::PG_BYTES;
#pragma unroll
                for (int c = 0; c < 16; c++) {
                    float pr = ex2(fmaf(s[c], scl2, -lse2));
                    float ds = pr * (dp[c] - Dq);
                    if (!row_ok) {
                        pr = 0.f;
                        ds = 0.f;
                    }
                    const uint32_t off = c * 128 + ((chk ^ (c & 7)) << 4);
                    *reinterpret_cast<__nv_bfloat16*>(pb + off) = __float2bfloat16_rn(ds);
                    *reinterpret_cast<__nv_bfloat16*>(pb + 2048 + off) = __float2bfloat16_rn(pr);
                }
                fence_async_smem();
                mbar_arrive(smem_u32(&ms->p_full[w][b]));
                if (gi == 0 && pend) {
                    epilogue();
                    pend = false;
                }
            }
            if (pend) {  // no item to overlap with
                epilogue();
                pend = false;
            }
            pend = true;
            pacc = items > 0;
            pslice = slice;
            pj = j;
            pkn = kn;
#pragma unroll
            for (int l = 0; l < 4; l++) {
                prk[l] = rk[l];
                prv[l] = rv[l];
            }
            if (items > 0) kn++;
        }
        if (pend) epilogue();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 256);
    }
}

template <int D, bool R>
int launch_one(const Shape& s, const AttnArgs& a, const CUtensorMap* maps, cudaStream_t st) {
    using C = Cfg<D>;
    static_assert(C::SMEM <= 227 * 1024, "shared memory budget");
    static_assert(sizeof(Misc) <= 4096, "misc block");
    static_assert(C::STAGES >= 1, "one stage at least");
    cudaFuncSetAttribute(bwd_dkv_tc_kernel<D, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    const long long total = s.slices * (long long)s.T;
    const int grid = (int)std::min<long long>(total, (long long)sm_count());
    if ((total + grid - 1) / grid > kMaxKeyBlocks) return LLSA_ERR_UNSUPPORTED;
    LLSA_LAUNCH("bwd_dkv_tc", st,
                bwd_dkv_tc_kernel<D, R><<<grid, kThreads, C::SMEM, st>>>(maps[0], maps[1], maps[2], maps[3], a));
    return LLSA_OK;
}

// each built once per token order
template <int D>
int launch_cfg(const Shape& s, const AttnArgs& a, const CUtensorMap* maps, cudaStream_t st) {
    return s.raster ? launch_one<D, true>(s, a, maps, st) : launch_one<D, false>(s, a, maps, st);
}

}  // namespace

bool bwd_dkv_tc_fits(const Shape& s) {
    const long long total = s.slices * (long long)s.T;
    const int grid = (int)std::min<long long>(total, (long long)sm_count());
    return grid > 0 && (total + grid - 1) / grid <= kMaxKeyBlocks;
}

int launch_bwd_dkv_tc(const Shape& s, const AttnArgs& a, cudaStream_t st) {
    CUtensorMap maps[4];
    const void* bases[4] = {a.q, a.dout, a.k, a.v};
    for (int t = 0; t < 4; t++) LLSA_TRY(make_tmap_tokens(&maps[t], bases[t], s));
    return s.d == 64 ? launch_cfg<64>(s, a, maps, st) : launch_cfg<128>(s, a, maps, st);
}

}  // namespace llsa
