// attn_fwd_grp.cu -- block-sparse attention forward with KV enrichment on the
// tcgen05 tensor cores, over groups of query blocks that share their selected
// key blocks (bf16 in, fp32 accumulate; B = 16, d = 64, K_1 in {4, 8, 16},
// L_e <= 3).
//
// Method: Pith review of arXiv 2512.16615, "Core claim": every query block of
// B tokens attends the B tokens of its K selected blocks plus one pooled K/V
// token per level with weight B^l (logit + ln B^l, KV Reweighting).
//
// A group (group.cu) holds up to 8 query blocks; their 128 query rows are the
// M = 128 rows of every product. U, the union of the group's selected key
// blocks in ascending order, is gathered once and processed in tiles of 4
// blocks: S = Q K_U^T (M = 128, N = 16 * blocks in the tile, K = d), then
// O += P V_U (M = 128, N = d, K = 16 keys per step, one union block per step).
// A query row keeps only the union blocks its own block selected; the others
// get probability 0, so each row still attends exactly its key set.
//
// One thread per query row (the row's S, P and O live in its TMEM lane), so
// the softmax needs no exchange between threads:
//   * shift: the row's largest pooled-key logit. Softmax is shift-invariant;
//     when a tile holds logits more than 2^64 (base 2) above the shift, the
//     shift moves to that tile's row maximum and the row's sum and output
//     accumulated so far are rescaled (never the case for the pixel inputs,
//     exercised by a test whose fine logits lie far above the pooled ones);
//   * P (unnormalised, bf16) goes to TMEM and is the A operand of the P V
//     product; O is scaled by 1 / row sum in the epilogue, which also adds the
//     pooled values and writes the row's output and LSE.
// S and P are double-buffered in TMEM, so S of the next tile is computed
// while the softmax works on this one, and P of a tile is written while the
// P V product of the tile before runs.
//
// Warp roles (persistent CTAs, groups strided over CTAs, alternate groups to
// the two softmax warpgroups):
//   warps 0, 2  one per softmax warpgroup: its groups' records (group.cu)
//               into the Q slots, Q boxes, pooled K/V rows (cp.async), K and V
//               boxes of the tiles;
//   warps 1, 3  MMA issuers, one per softmax warpgroup (warp 1 also owns TMEM);
//   warps 4-7,  softmax / epilogue warpgroups, each with two S and two P
//   warps 8-11  buffers and one O accumulator in TMEM, two Q slots and three
//               K/V stages.
// Every mbarrier wait is bounded; a timeout records LLSA_ERR_TIMEOUT and the
// CTA drains and exits.
#include <algorithm>

#include "attn.h"
#include "tc.cuh"

namespace llsa {
namespace {

using namespace tc;

constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSlack = 64.f;  // base-2 range of the logits above the shift
constexpr int kLeMax = 3;       // pooled levels held per group

template <int K1>
struct GCfg {
    static constexpr int D = 64;
    static constexpr int TS = 4;                    // union blocks per tile (N = 64)
    static constexpr int NU = 8 * K1;               // union capacity (8 query blocks)
    static constexpr int MW = NU / 32;              // mask words per query block
    static constexpr int Q_BYTES = 128 * D * 2;     // 8 query blocks x 16 rows
    static constexpr int PK_OFF = Q_BYTES;          // pooled K rows [query block][level][d] fp32
    static constexpr int PV_OFF = PK_OFF + 8 * kLeMax * D * 4;
    static constexpr int META_OFF = PV_OFF + 8 * kLeMax * D * 4;
    static constexpr int QSLOT = (META_OFF + 1024 + 1023) / 1024 * 1024;
    static constexpr int NQW = 2;                   // Q slots per warpgroup
    static constexpr int KTILE = TS * 16 * D * 2;   // 8 KB: the K (or V) blocks of a tile
    static constexpr int NKW = 3;                   // K stages and V stages per warpgroup
    static constexpr int SMEM = 1024 + 2 * NQW * QSLOT + 2 * 2 * NKW * KTILE + 1024;
    // TMEM columns of a warpgroup: S0, S1 (64 each), P0, P1 (32 each, bf16
    // pairs), O (64)
    static constexpr int TM_S = 0, TM_P = 128, TM_O = 192, TM_WG = 256;
};

struct GBar {
    uint64_t q_full[4], q_empty[4], k_full[6], k_empty[6], v_full[6], v_empty[6];
    uint64_t s_full[2][2], s_free[2][2], p_full[2][2], pv_done[2][2], o_free[2], drain[2];
    uint32_t tmem_slot;
    int abort_flag;
    long long total_groups;
};

struct GArgs {
    AttnArgs a;
    const int32_t* ngroups;  // groups per window of query blocks (group.cu)
    const GroupRec* recs;    // group records, at slice * T + window * win + group
    int windows, win;        // windows per slice, query blocks per window
    int always;              // run whatever the group sizes (no per-block tensor-core forward for this shape)
};

__device__ __forceinline__ bool wait_all(uint32_t mbar, uint32_t parity, volatile int* abort_flag, int* status,
                                         int limit) {
    const bool ok = mbar_wait_n(mbar, parity, abort_flag, status, limit);
    return __all_sync(0xffffffffu, ok);
}

// Unnormalised P of one 32-key chunk (two union blocks) with the shift m:
// active blocks (bits h of act2) get 2^(s * scl2 - m), the others 0; adds the
// values to sum and flags a value above kSlack.
__device__ __forceinline__ void chunk_p(const uint32_t* sraw, uint32_t act2, float scl2, float m, float& sum,
                                        bool& over, uint32_t* pk) {
#pragma unroll
    for (int h = 0; h < 2; h++) {
        const bool act = (act2 >> h) & 1u;
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            const float x0 = fmaf(__uint_as_float(sraw[16 * h + i]), scl2, -m);
            const float x1 = fmaf(__uint_as_float(sraw[16 * h + i + 1]), scl2, -m);
            over |= act && fmaxf(x0, x1) > kSlack;
            const float p0 = act ? ex2(x0) : 0.f, p1 = act ? ex2(x1) : 0.f;
            sum += p0 + p1;
            pk[8 * h + i / 2] = pack_bf16x2(p0, p1);
        }
    }
}

// The rare path of a tile, taken by a whole warp when some row of it saw a
// logit more than kSlack above its shift: each such row moves its shift up
// to the tile's row maximum, its sum of earlier tiles and (when earlier tiles
// of the group went into O) its O row are rescaled, and the tile's P is
// written again. S of the tile is still in TMEM. Kept out of line so that
// the common path keeps its registers.
template <int D>
__device__ __noinline__ void shift_up(uint32_t tS, uint32_t tP, uint32_t tO, int nch, uint32_t m4, uint32_t wm4,
                                      float scl2, bool over, bool rescale_o, float sum0, float* m_run, float* sum) {
    float tmax = -INFINITY;
    for (int c = 0; c < nch; c++) {
        if (!((wm4 >> (2 * c)) & 3u)) continue;
        uint32_t sraw[32];
        tmem_ld32_nowait(tS + 32 * c, sraw);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 2; h++)
            if ((m4 >> (2 * c + h)) & 1u)
#pragma unroll
                for (int i = 0; i < 16; i++) tmax = fmaxf(tmax, __uint_as_float(sraw[16 * h + i]));
    }
    const float m_old = *m_run;
    const float m_new = over ? tmax * scl2 : m_old;
    const float f = over ? (m_old == -INFINITY ? 0.f : ex2(m_old - m_new)) : 1.f;
    float s = sum0 * f;
    bool unused = false;
    for (int c = 0; c < nch; c++) {
        if (!((wm4 >> (2 * c)) & 3u)) continue;  // zeros already written
        uint32_t sraw[32], pk[16];
        tmem_ld32_nowait(tS + 32 * c, sraw);
        tmem_wait_ld();
        chunk_p(sraw, (m4 >> (2 * c)) & 3u, scl2, m_new, s, unused, pk);
        tmem_st16(tP + 16 * c, pk);
    }
    if (rescale_o) {
        for (int c = 0; c < D / 32; c++) {
            uint32_t ov[32];
            tmem_ld32_nowait(tO + 32 * c, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; i++) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
            tmem_st16(tO + 32 * c, ov);
            tmem_st16(tO + 32 * c + 16, ov + 16);
        }
    }
    *m_run = m_new;
    *sum = s;
}

template <int K1>
__global__ void __launch_bounds__(kThreads, 1)
fwd_grp_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, GArgs ga) {
    using C = GCfg<K1>;
    using Meta = GroupRec;
    constexpr int D = C::D;
    const AttnArgs& a = ga.a;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* qslots = sm;                       // [2 * NQW][QSLOT]
    unsigned char* kst = sm + 2 * C::NQW * C::QSLOT;  // K stages [2 * NKW][KTILE]
    unsigned char* vst = kst + 2 * C::NKW * C::KTILE;  // V stages [2 * NKW][KTILE]
    GBar* bar = reinterpret_cast<GBar*>(vst + 2 * C::NKW * C::KTILE);
    volatile int* abort_flag = &bar->abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, T = a.T, Le = a.Le;

    if (threadIdx.x == 0) {
        for (int w = 0; w < 2; w++) {
            for (int b = 0; b < 2; b++) {
                mbar_init(smem_u32(&bar->s_full[w][b]), 1);
                mbar_init(smem_u32(&bar->s_free[w][b]), 128);
                mbar_init(smem_u32(&bar->p_full[w][b]), 128);
                mbar_init(smem_u32(&bar->pv_done[w][b]), 1);
            }
            mbar_init(smem_u32(&bar->o_free[w]), 128);
        }
        for (int s = 0; s < 2 * C::NQW; s++) {
            mbar_init(smem_u32(&bar->q_full[s]), 1 + 32);    // Q boxes (tx) + the gather warp's cp.async lanes
            mbar_init(smem_u32(&bar->q_empty[s]), 1 + 128);  // last S of the group + the warpgroup's epilogue
        }
        for (int s = 0; s < 2 * C::NKW; s++) {
            mbar_init(smem_u32(&bar->k_full[s]), 1);   // K boxes (tx)
            mbar_init(smem_u32(&bar->k_empty[s]), 1);  // S of the tile done
            mbar_init(smem_u32(&bar->v_full[s]), 1);   // V boxes (tx)
            mbar_init(smem_u32(&bar->v_empty[s]), 1);  // P V of the tile done
        }
        mbar_init(smem_u32(&bar->drain[0]), 1);
        mbar_init(smem_u32(&bar->drain[1]), 1);
        bar->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        long long tot = 0;
        for (long long u = lane; u < a.slices * ga.windows; u += 32) tot += ga.ngroups[u];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        if (lane == 0) bar->total_groups = tot;
    }
    if (warp == 1) tmem_alloc(smem_u32(&bar->tmem_slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = bar->tmem_slot;
    const long long total = bar->total_groups;
    // the per-query-block forward, launched after this one, takes the call
    // when the groups are too small
    const bool run = ga.always || grouped_forward(total, a.slices * (long long)T, a.test_flags);
    const long long mine = run && total > blockIdx.x ? (total - blockIdx.x + G - 1) / G : 0;
    // groups of warpgroup w: the CTA's groups w, w + 2, ...
    const long long mineW[2] = {(mine + 1) / 2, mine / 2};

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ gather
        // Warp 0 serves warpgroup 0 (the CTA's groups 0, 2, ...), warp 2
        // warpgroup 1 (groups 1, 3, ...).
        const int w = warp >> 1;
        long long cur_slice = 0, cur_base = 0;  // walk of the per-window group counts
        int cur_win = 0;
        long long qissued = 0;                  // groups whose Q slot copies were issued
        constexpr int R = C::NU / 32;
        // The next group's record (group.cu) is loaded one group ahead, one
        // independent 16-byte piece per lane, so the load is in flight while
        // this group's tiles go out.
        uint4 n_rec = make_uint4(0u, 0u, 0u, 0u);
        auto load_next = [&](long long jn) {
            if (jn >= mineW[w]) return;
            const long long gi = blockIdx.x + (2 * jn + w) * G;
            while (cur_slice < a.slices && gi >= cur_base + ga.ngroups[cur_slice * ga.windows + cur_win]) {
                cur_base += ga.ngroups[cur_slice * ga.windows + cur_win];
                if (++cur_win == ga.windows) {
                    cur_win = 0;
                    cur_slice++;
                }
            }
            const GroupRec* rec = ga.recs + cur_slice * T + cur_win * ga.win + (int)(gi - cur_base);
            n_rec = reinterpret_cast<const uint4*>(rec)[lane];
        };
        load_next(0);
        // Set-up of group jn in its Q slot (free by now): the record into the
        // slot, Q boxes, pooled rows; then the next record.
        auto setup = [&](long long jn) {
            const int qsl = w * C::NQW + (int)(jn % C::NQW);
            unsigned char* slot = qslots + qsl * C::QSLOT;
            Meta* meta = reinterpret_cast<Meta*>(slot + C::META_OFF);
            reinterpret_cast<uint4*>(meta)[lane] = n_rec;
            __syncwarp();
            const int count = meta->count;
            const long long slice = meta->slice;
            const int qb_l = lane < count ? meta->qb[lane] : 0;
            // the slot's copies: Q rows (TMA), pooled K and V rows of the
            // group's enrichment tokens (cp.async, 16-byte pieces); the
            // barrier's completion also publishes the record to the consumers
            const uint32_t qf = smem_u32(&bar->q_full[qsl]);
            if (lane == 0) mbar_arrive_expect_tx(qf, (uint32_t)(count * 16 * D * 2));
            __syncwarp();
            if (lane < count)
                tma_load_2d(smem_u32(slot + lane * 2048), &mq, 0, (int)(slice * a.n + (long long)qb_l * 16), qf);
            {
                // row x = (query block * kLeMax + level) * 2 + (0: K, 1: V)
                constexpr int per_row = D * 4 / 16;
                const int items = count * kLeMax * 2 * per_row;
                for (int it0 = 0; it0 < items; it0 += 32) {
                    const int it = it0 + lane;
                    const int row = it / per_row, piece = it % per_row;
                    const int ql = row >> 1, isv = row & 1, qs = ql / kLeMax, l = ql % kLeMax;
                    if (it >= items || l >= Le) continue;
                    const int e = meta->ce[qs][l];
                    const float* src = (isv ? a.vpyr : a.kpyr) + slice * a.pyr_stride +
                                       (long long)(a.lv.row_offset[l + 1] + e) * D + piece * 4;
                    unsigned char* dst = slot + (isv ? C::PV_OFF : C::PK_OFF) + ql * D * 4 + piece * 16;
                    cp_async16(smem_u32(dst), src);
                }
                cp_async_arrive(qf);
            }
            qissued = jn + 1;
            load_next(jn + 1);
        };
        int tk = 0, tv = 0;   // tiles whose K / V boxes were issued
        int v_ns = 0, v_yk = 0;  // the tile whose V boxes are pending
        auto issue_v = [&]() -> bool {
            const int stv = w * C::NKW + tv % C::NKW, use = tv / C::NKW;
            if (use >= 1 && !wait_all(smem_u32(&bar->v_empty[stv]), (uint32_t)((use - 1) & 1), abort_flag, a.status, a.spin))
                return false;
            const uint32_t fb = smem_u32(&bar->v_full[stv]);
            if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)(v_ns * 16 * D * 2));
            __syncwarp();
            if (lane < v_ns) tma_load_2d(smem_u32(vst + stv * C::KTILE + lane * 2048), &mv, 0, v_yk, fb);
            tv++;
            v_ns = 0;
            return true;
        };
        // a failure-detection test can switch the copies off (nothing armed,
        // every consumer's first wait runs out)
        const long long jN = (a.test_flags & LLSA_TEST_NO_COPIES) ? 0 : mineW[w];
        bool ok = true;
        if (jN > 0) setup(0);
        for (long long j = 0; j < jN && ok; j++) {
            const int qsl = w * C::NQW + (int)(j % C::NQW);
            const Meta* meta = reinterpret_cast<const Meta*>(qslots + qsl * C::QSLOT + C::META_OFF);
            const int nslots = meta->nslots;
            const long long slice = meta->slice;
            // K boxes of the group's tiles, each tile's V boxes one tile later
            // (a K stage is free once S of its tile is done, a V stage only
            // once P V is, so K runs ahead)
            const int nt = (nslots + C::TS - 1) / C::TS;
            for (int t = 0; t < nt && ok; t++) {
                const int stk = w * C::NKW + tk % C::NKW, use = tk / C::NKW;
                if (use >= 1 &&
                    !wait_all(smem_u32(&bar->k_empty[stk]), (uint32_t)((use - 1) & 1), abort_flag, a.status, a.spin)) {
                    ok = false;
                    break;
                }
                const int ns = min(C::TS, nslots - t * C::TS);
                const int yk = lane < ns ? (int)(slice * a.n + (long long)meta->uni[t * C::TS + lane] * 16) : 0;
                const uint32_t fb = smem_u32(&bar->k_full[stk]);
                if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)(ns * 16 * D * 2));
                __syncwarp();
                if (lane < ns) tma_load_2d(smem_u32(kst + stk * C::KTILE + lane * 2048), &mk, 0, yk, fb);
                tk++;
                if (v_ns > 0) ok = issue_v();
                v_ns = ns;
                v_yk = yk;
            }
            // the next group, once its Q slot is free
            if (ok && j + 1 < jN) {
                const long long jn = j + 1, qu = jn / C::NQW;
                if (qu >= 1 && !wait_all(smem_u32(&bar->q_empty[w * C::NQW + (int)(jn % C::NQW)]),
                                         (uint32_t)((qu - 1) & 1), abort_flag, a.status, a.spin))
                    ok = false;
                else
                    setup(jn);
            }
        }
        if (ok && v_ns > 0) ok = issue_v();
        asm volatile("cp.async.wait_all;\n" ::: "memory");
        // copies this warp issued must land before the CTA exits (after a
        // normal run every phase below has completed already)
        if (lane == 0) {
            for (int back = 1; back <= C::NKW && back <= tk; back++) {
                const int tau = tk - back;
                const int st = w * C::NKW + tau % C::NKW;
                for (int it = 0; it < kSpinLimit && !mbar_test(smem_u32(&bar->k_full[st]), (tau / C::NKW) & 1);
                     it++) {
                }
            }
            for (int back = 1; back <= C::NKW && back <= tv; back++) {
                const int tau = tv - back;
                const int st = w * C::NKW + tau % C::NKW;
                for (int it = 0; it < kSpinLimit && !mbar_test(smem_u32(&bar->v_full[st]), (tau / C::NKW) & 1);
                     it++) {
                }
            }
            for (long long back = 1; back <= C::NQW && back <= qissued; back++) {
                const long long jj = qissued - back;
                const int qsl = w * C::NQW + (int)(jj % C::NQW);
                for (int it = 0;
                     it < kSpinLimit && !mbar_test(smem_u32(&bar->q_full[qsl]), (uint32_t)((jj / C::NQW) & 1));
                     it++) {
                }
            }
        }
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------------- MMA issuers
        // Warp 1 issues for warpgroup 0, warp 3 for warpgroup 1, each one
        // in-order stream S(0), then S(tau + 1), P V(tau) for tau = 0, 1, ...
        // with blocking waits (at a group boundary P V(tau) comes first). S(tau + 1) needs the softmax to be done with
        // the S buffer of tile tau - 1; P V(tau) needs P of tile tau; neither
        // waits for anything issued later in the stream.
        const int w = warp == 1 ? 0 : 1;
        const uint64_t dK = desc_sw128(smem_u32(kst), 16, 1024);  // K-major Q and K
        const uint64_t dQ = desc_sw128(smem_u32(qslots), 16, 1024);
        const uint64_t dV = desc_sw128(smem_u32(vst), C::TS * 16 * 128, 1024);  // MN-major V
        constexpr uint32_t idPV = idesc_bf16(128, D, 0, 1);
        long long gS = 0, gP = 0;                 // group of the next S / P V
        int tS = 0, tP = 0, tauS = 0, tauP = 0;  // tile within the group / of the warpgroup
        int nsl[4] = {-1, -1, -1, -1};            // union sizes by group mod 4 (S leads P V by one tile)
        auto issue_S = [&]() -> bool {
            const int qsl = w * C::NQW + (int)(gS % C::NQW);
            if (tS == 0) {
                if (!wait_all(smem_u32(&bar->q_full[qsl]), (uint32_t)((gS / C::NQW) & 1), abort_flag, a.status, a.spin))
                    return false;
                nsl[gS & 3] = reinterpret_cast<const Meta*>(qslots + qsl * C::QSLOT + C::META_OFF)->nslots;
            }
            const int nslots = nsl[gS & 3];
            const int st = w * C::NKW + tauS % C::NKW;
            const int b = tauS & 1;
            if (!wait_all(smem_u32(&bar->k_full[st]), (uint32_t)((tauS / C::NKW) & 1), abort_flag, a.status, a.spin))
                return false;
            if (tauS >= 2 &&
                !wait_all(smem_u32(&bar->s_free[w][b]), (uint32_t)(((tauS >> 1) - 1) & 1), abort_flag, a.status, a.spin))
                return false;
            tc_fence_after();
            const int ns = min(C::TS, nslots - tS * C::TS);
            const uint32_t q0 = (uint32_t)(qsl * C::QSLOT), k0 = (uint32_t)(st * C::KTILE);
            const uint32_t idS = idesc_bf16(128, 16 * ns, 0, 0);
            const uint32_t dt = tbase + w * C::TM_WG + C::TM_S + b * 64;
#pragma unroll
            for (int ks = 0; ks < D / 16; ks++)
                mma_bf16_warp(dt, dQ + ((q0 + ks * 32) >> 4), dK + ((k0 + ks * 32) >> 4), idS, ks > 0);
            mma_commit_warp(smem_u32(&bar->s_full[w][b]));
            mma_commit_warp(smem_u32(&bar->k_empty[st]));
            const int nt = (nslots + C::TS - 1) / C::TS;
            if (tS == nt - 1) mma_commit_warp(smem_u32(&bar->q_empty[qsl]));  // done with this Q
            tauS++;
            if (++tS == nt) {
                tS = 0;
                gS++;
            }
            return true;
        };
        auto issue_PV = [&]() -> bool {
            const int b = tauP & 1;
            if (!wait_all(smem_u32(&bar->p_full[w][b]), (uint32_t)((tauP >> 1) & 1), abort_flag, a.status, a.spin))
                return false;
            if (tP == 0 && gP >= 1 &&
                !wait_all(smem_u32(&bar->o_free[w]), (uint32_t)((gP - 1) & 1), abort_flag, a.status, a.spin))
                return false;
            tc_fence_after();
            const int nslots = nsl[gP & 3];
            const int ns = min(C::TS, nslots - tP * C::TS);
            const int st = w * C::NKW + tauP % C::NKW;
            if (!wait_all(smem_u32(&bar->v_full[st]), (uint32_t)((tauP / C::NKW) & 1), abort_flag, a.status, a.spin))
                return false;
            tc_fence_after();
            const uint32_t v0 = (uint32_t)(st * C::KTILE);
            const uint32_t dt = tbase + w * C::TM_WG + C::TM_O;
            const uint32_t pt = tbase + w * C::TM_WG + C::TM_P + b * 32;
            for (int u = 0; u < ns; u++)
                mma_bf16_ts_warp(dt, pt + 8 * u, dV + ((v0 + u * 2048) >> 4), idPV, (tP > 0 || u > 0) ? 1u : 0u);
            mma_commit_warp(smem_u32(&bar->pv_done[w][b]));
            mma_commit_warp(smem_u32(&bar->v_empty[st]));
            const int nt = (nslots + C::TS - 1) / C::TS;
            tauP++;
            if (++tP == nt) {
                tP = 0;
                gP++;
            }
            return true;
        };
        // a group's first S goes after the previous group's last P V, so a
        // late Q of the next group never holds up that P V and the epilogue
        bool ok = mineW[w] > 0 ? issue_S() : true;
        while (ok && gP < mineW[w]) {
            if (gS < mineW[w]) ok = issue_S();
            if (ok) ok = issue_PV();
        }
        // no MMA of this warp may be in flight when TMEM is released
        mma_commit_warp(smem_u32(&bar->drain[w]));
        if (lane == 0)
            for (int it = 0; it < kSpinLimit && !mbar_try(smem_u32(&bar->drain[w]), 0); it++) {
            }
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------------------------------------- softmax / epilogue
        const int w = (warp - 4) >> 2, q4 = warp & 3;
        const int r = q4 * 32 + lane;  // query row of the group
        const int qs = r >> 4;         // query block slot
        const uint32_t lanes = (uint32_t)(q4 * 32) << 16;
        const uint32_t tS0 = tbase + w * C::TM_WG + C::TM_S + lanes;
        const uint32_t tP0 = tbase + w * C::TM_WG + C::TM_P + lanes;
        const uint32_t tO = tbase + w * C::TM_WG + C::TM_O + lanes;
        const float sc = a.scale, scl2 = a.scale * kLog2e;
        int tau = 0;
        for (long long j = 0; j < mineW[w]; j++) {
            const int qsl = w * C::NQW + (int)(j % C::NQW);
            const unsigned char* slot = qslots + qsl * C::QSLOT;
            const Meta* meta = reinterpret_cast<const Meta*>(slot + C::META_OFF);
            if (!wait_all(smem_u32(&bar->q_full[qsl]), (uint32_t)((j / C::NQW) & 1), abort_flag, a.status, a.spin)) break;
            // the group's description, kept in registers
            const int count = meta->count, nslots = meta->nslots;
            const long long slice = meta->slice;
            const bool valid = qs < count;
            const int qb = valid ? meta->qb[qs] : 0;
            uint32_t mw[C::MW];
#pragma unroll
            for (int x = 0; x < C::MW; x++) mw[x] = valid ? meta->mask[qs][x] : 0u;
            // pooled-key logits (base 2, + l ln B) of this row
            float cs2[kLeMax], m_run = -INFINITY;
#pragma unroll
            for (int l = 0; l < kLeMax; l++) cs2[l] = -INFINITY;
            if (valid) {
                const float* pk = reinterpret_cast<const float*>(slot + C::PK_OFF) + qs * kLeMax * D;
                float acc[kLeMax];
#pragma unroll
                for (int l = 0; l < kLeMax; l++) acc[l] = 0.f;
#pragma unroll
                for (int c8 = 0; c8 < D / 8; c8++) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(slot + sw128_offset(r, c8 * 8, 128));
                    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
                    float x[8];
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const float2 f = __bfloat1622float2(h[i]);
                        x[2 * i] = f.x;
                        x[2 * i + 1] = f.y;
                    }
#pragma unroll
                    for (int l = 0; l < kLeMax; l++)
                        if (l < Le) {
                            const float4 k0 = *reinterpret_cast<const float4*>(pk + l * D + c8 * 8);
                            const float4 k1 = *reinterpret_cast<const float4*>(pk + l * D + c8 * 8 + 4);
                            float t0 = x[0] * k0.x, t1 = x[1] * k0.y;
                            t0 = fmaf(x[2], k0.z, t0); t1 = fmaf(x[3], k0.w, t1);
                            t0 = fmaf(x[4], k1.x, t0); t1 = fmaf(x[5], k1.y, t1);
                            t0 = fmaf(x[6], k1.z, t0); t1 = fmaf(x[7], k1.w, t1);
                            acc[l] += t0 + t1;
                        }
                }
#pragma unroll
                for (int l = 0; l < kLeMax; l++)
                    if (l < Le) {
                        cs2[l] = (sc * acc[l] + (float)(l + 1) * a.lnB) * kLog2e;
                        m_run = fmaxf(m_run, cs2[l]);
                    }
            }
            float sum = 0.f;
            const int nt = (nslots + C::TS - 1) / C::TS;
            bool ok = true;
            for (int t = 0; t < nt; t++, tau++) {
                const int b = tau & 1;
                const uint32_t use = (uint32_t)(tau >> 1);
                const uint32_t tS = tS0 + b * 64, tP = tP0 + b * 32;
                if (!wait_all(smem_u32(&bar->s_full[w][b]), use & 1, abort_flag, a.status, a.spin)) {
                    ok = false;
                    break;
                }
                // P buffer b was last read by the P V product two tiles back
                if (use >= 1 && !wait_all(smem_u32(&bar->pv_done[w][b]), (use - 1) & 1, abort_flag, a.status, a.spin)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int sb = t * C::TS;  // first union slot of the tile
                const uint32_t m4 = (mw[sb >> 5] >> (sb & 31)) & 0xFu;
                const uint32_t wm4 = __reduce_or_sync(0xffffffffu, m4);
                const int ns = min(C::TS, nslots - sb);
                const int nch = (ns + 1) >> 1;  // 32-key chunks the P V product reads
                // unnormalised P with the current shift; a logit more than
                // kSlack above it flags the tile
                const float sum0 = sum;
                bool over = false;
                {
                    uint32_t sraw[2][32];
#pragma unroll
                    for (int c = 0; c < 2; c++)
                        if (c < nch && ((wm4 >> (2 * c)) & 3u)) tmem_ld32_nowait(tS + 32 * c, sraw[c]);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 2; c++) {
                        if (c >= nch) break;
                        uint32_t pk[16];
                        if ((wm4 >> (2 * c)) & 3u) {
                            chunk_p(sraw[c], (m4 >> (2 * c)) & 3u, scl2, m_run, sum, over, pk);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; i++) pk[i] = 0u;
                        }
                        tmem_st16(tP + 16 * c, pk);
                    }
                }
                if (__any_sync(0xffffffffu, over)) {
                    // rare: see shift_up; when this group's earlier tiles went
                    // into O, the last of their P V products must be complete
                    if (t > 0) {
                        const int bp = (tau - 1) & 1;
                        if (!wait_all(smem_u32(&bar->pv_done[w][bp]), (uint32_t)(((tau - 1) >> 1) & 1), abort_flag,
                                      a.status, a.spin)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    shift_up<D>(tS, tP, tO, nch, m4, wm4, scl2, over, t > 0, sum0, &m_run, &sum);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(smem_u32(&bar->s_free[w][b]));
                mbar_arrive(smem_u32(&bar->p_full[w][b]));
            }
            if (!ok) break;
            // epilogue: O / row sum + pooled values
            {
                const int bl = (tau - 1) & 1;
                if (!wait_all(smem_u32(&bar->pv_done[w][bl]), (uint32_t)(((tau - 1) >> 1) & 1), abort_flag, a.status, a.spin))
                    break;
            }
            tc_fence_after();
            uint32_t ov[D];
#pragma unroll
            for (int c = 0; c < D / 32; c++) tmem_ld32_nowait(tO + 32 * c, ov + 32 * c);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar->o_free[w]));
            if (valid) {
                float pl[kLeMax];
                float z = sum;
#pragma unroll
                for (int l = 0; l < kLeMax; l++) {
                    pl[l] = l < Le ? ex2(cs2[l] - m_run) : 0.f;
                    z += pl[l];
                }
                const float iz = 1.0f / z;
#pragma unroll
                for (int l = 0; l < kLeMax; l++) pl[l] *= iz;
                const float* pv = reinterpret_cast<const float*>(slot + C::PV_OFF) + qs * kLeMax * D;
                const long long row = slice * a.n + (long long)qb * 16 + (r & 15);
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out_o) + row * D;
#pragma unroll
                for (int c8 = 0; c8 < D / 8; c8++) {
                    float y[8];
#pragma unroll
                    for (int i = 0; i < 8; i++) y[i] = __uint_as_float(ov[8 * c8 + i]) * iz;
#pragma unroll
                    for (int l = 0; l < kLeMax; l++)
                        if (l < Le) {
                            const float4 v0 = *reinterpret_cast<const float4*>(pv + l * D + 8 * c8);
                            const float4 v1 = *reinterpret_cast<const float4*>(pv + l * D + 8 * c8 + 4);
                            y[0] = fmaf(pl[l], v0.x, y[0]); y[1] = fmaf(pl[l], v0.y, y[1]);
                            y[2] = fmaf(pl[l], v0.z, y[2]); y[3] = fmaf(pl[l], v0.w, y[3]);
                            y[4] = fmaf(pl[l], v1.x, y[4]); y[5] = fmaf(pl[l], v1.y, y[5]);
                            y[6] = fmaf(pl[l], v1.z, y[6]); y[7] = fmaf(pl[l], v1.w, y[7]);
                        }
                    *reinterpret_cast<uint4*>(dst + 8 * c8) = make_uint4(
                        pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
                }
                a.lse[row] = m_run * (1.0f / kLog2e) + logf(z);
            }
            // the slot (Q rows, pooled rows, description) is no longer read here
            mbar_arrive(smem_u32(&bar->q_empty[qsl]));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
}

template <int K1>
int launch_k(const Shape& s, const GArgs& ga, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
             cudaStream_t st) {
    using C = GCfg<K1>;
    static_assert(C::SMEM <= 227 * 1024, "shared memory budget");
    static_assert(sizeof(GroupRec) <= 1024, "meta block");
    static_assert(sizeof(GBar) <= 1024, "barrier block");
    if (cudaFuncSetAttribute(fwd_grp_kernel<K1>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
        return LLSA_ERR_CUDA;
    // groups per step are at most the query blocks; one CTA per SM
    const long long upper = s.slices * (long long)s.T;
    const int grid = (int)std::min<long long>(upper, (long long)sm_count());
    LLSA_LAUNCH("fwd_grp", st, fwd_grp_kernel<K1><<<grid, kThreads, C::SMEM, st>>>(mq, mk, mv, ga));
    return LLSA_OK;
}

}  // namespace

bool fwd_grp_supported(const Shape& s) {
    return s.dtype == LLSA_DTYPE_BF16 && s.B == 16 && s.d == 64 && (s.K1 == 4 || s.K1 == 8 || s.K1 == 16) &&
           s.Le <= kLeMax &&
           s.Lc == s.Le && group_supported(s) && s.slices * (long long)s.n < (1LL << 31);
}

int launch_fwd_grp(const Shape& s, const AttnArgs& a, const int32_t* ngroups, const GroupRec* recs,
                   cudaStream_t st) {
    CUtensorMap mq, mk, mv;
    const long long rows = s.slices * (long long)s.n;
    LLSA_TRY(make_tmap_bf16(&mq, a.q, rows, s.d, 16));
    LLSA_TRY(make_tmap_bf16(&mk, a.k, rows, s.d, 16));
    LLSA_TRY(make_tmap_bf16(&mv, a.v, rows, s.d, 16));
    GArgs ga;
    ga.a = a;
    ga.ngroups = ngroups;
    ga.recs = recs;
    ga.windows = group_windows(s);
    ga.win = kGroupWindow;
    ga.always = fwd_tc_supported(s) ? 0 : 1;
    if (s.K1 == 4) return launch_k<4>(s, ga, mq, mk, mv, st);
    return s.K1 == 8 ? launch_k<8>(s, ga, mq, mk, mv, st) : launch_k<16>(s, ga, mq, mk, mv, st);
}

}  // namespace llsa
