// tc.cuh -- sm_103a building blocks for the tensor-core kernels: tcgen05 MMA
// with operands in shared memory and accumulators in tensor memory (TMEM), TMA
// tile loads, mbarriers with bounded waits.
//
// Encodings (checked on a GB300 before use):
//   shared-memory matrix descriptor: start >> 4 in bits 0-13, leading byte
//   offset >> 4 in 16-29, stride byte offset >> 4 in 32-45, version 1 at bit 46,
//   layout 2 (128-byte swizzle) in bits 61-63. With 128-byte rows the swizzle
//   atom is 8 rows = 1024 B: K-major operands use SBO = 1024 and step along K by
//   moving the start address 32 B per 16 bf16; MN-major operands store rows of
//   64 MN-elements per K index, SBO = 1024 (8 K rows), LBO = the distance
//   between 64-wide MN regions, and step along K by 16 rows (2048 B).
//   instruction descriptor (kind::f16): D f32 (bit 4), A, B bf16 (bits 7, 10),
//   A / B MN-major flags (bits 15, 16), N >> 3 (bits 17-22), M >> 4 (24-28).
//   TMEM accumulator of an M = 128 MMA: row r in lane r; of an M = 64 MMA: row
//   r in lane 32 * (r / 16) + r % 16 (the first 16 lanes of each quarter).
#pragma once

#include <cuda.h>

#include "internal.h"

namespace llsa {
namespace tc {

constexpr int kSpinLimit = 1 << 22;  // bounded waits: ~ seconds, then LLSA_ERR_TIMEOUT

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (TMEM) (+)= A (smem) * B (smem); one thread issues.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// Whole (converged) warp: one elected lane issues the MMA. The election sits
// inside the asm so no divergent branch surrounds the MMA instruction.
__device__ __forceinline__ void mma_bf16_warp(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n.reg .pred p, e;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// Whole (converged) warp: the elected lane commits (the same lane that
// mma_bf16_warp elects, so it tracks that lane's MMAs).
__device__ __forceinline__ void mma_commit_warp(uint32_t mbar) {
    asm volatile("{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n"
                 :: "r"(mbar) : "memory");
}

// Arrives on the mbarrier once every MMA issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n"
                 :: "r"(mbar) : "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" :: "r"(mbar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" :: "r"(mbar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" :: "r"(mbar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t mbar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok) : "r"(mbar), "r"(parity) : "memory");
    return ok != 0;
}

// Non-blocking test of the phase of the given parity.
__device__ __forceinline__ bool mbar_test(uint32_t mbar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok) : "r"(mbar), "r"(parity) : "memory");
    return ok != 0;
}

// Waits for the phase of the given parity to complete. Gives up, recording
// LLSA_ERR_TIMEOUT, after `limit` polls (the library's wait limit: kSpinLimit
// unless a failure-detection test lowered it), or as soon as another thread
// of the CTA gave up (abort flag); returns false then. The loop bound is the
// compile-time kSpinLimit and `limit` is read only on the failing path, which
// keeps the waiting code of the hot loops as it compiles without a test limit.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, volatile int* abort_flag, int* status,
                                          int limit) {
    for (int it = 0; it < kSpinLimit; it++) {
        if (mbar_try(mbar, parity)) return true;
        if ((it & 7) == 7 && (*abort_flag || it >= limit)) {
            if (!*abort_flag) {
                *abort_flag = 1;
                set_status(status, LLSA_ERR_TIMEOUT);
            }
            return false;
        }
    }
    *abort_flag = 1;
    set_status(status, LLSA_ERR_TIMEOUT);
    return false;
}

// The same wait with the poll count itself as the loop bound (the grouped
// forward kernel's waits compile better this way).
__device__ __forceinline__ bool mbar_wait_n(uint32_t mbar, uint32_t parity, volatile int* abort_flag, int* status,
                                            int limit) {
    for (int it = 0; it < limit; it++) {
        if (mbar_try(mbar, parity)) return true;
        if ((it & 7) == 7 && *abort_flag) return false;
    }
    *abort_flag = 1;
    set_status(status, LLSA_ERR_TIMEOUT);
    return false;
}

// 2D tiled TMA load (box from the tensor map) into shared memory, completing
// bytes on the mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t mbar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n"
                 :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar) : "memory");
}

// 4D tiled TMA load (box from the tensor map), completing bytes on the mbarrier.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];\n"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(mbar) : "memory");
}

// Block b (16 tokens) of slice `slice` of a token tensor, columns col ..
// col + 63, through a map from make_tmap_tokens: rows slice * n + 16 b ..
// +15 in tile order, or (RASTER) the block's 4 x 4 patch of the raster image.
// Both land as 16 rows of 128 bytes in the same swizzled layout. The order is
// a compile-time choice: each kernel is built once per order, so the tile
// order's copies carry no raster code.
template <bool RASTER>
__device__ __forceinline__ void tma_load_block(uint32_t dst, const CUtensorMap* map, int col, long long slice, int b,
                                               int n, uint32_t mbar) {
    if constexpr (RASTER) {
        int px, py;
        block_patch(b, px, py);
        tma_load_4d(dst, map, col, 4 * px, 4 * py, (int)slice, mbar);
    } else {
        tma_load_2d(dst, map, col, (int)(slice * n + (long long)b * 16), mbar);
    }
}

// 1D bulk copy global -> shared (16-byte aligned addresses, size a multiple
// of 16), completing bytes on the mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
                 :: "r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(mbar) : "memory");
}

// 16-byte asynchronous copy global -> shared through L2 (not L1).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" :: "r"(dst), "l"(src) : "memory");
}

// Arrives on the mbarrier once every cp.async issued so far by this thread
// has landed (the arrival is counted in the barrier's initial count).
__device__ __forceinline__ void cp_async_arrive(uint32_t mbar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" :: "r"(mbar) : "memory");
}

// 2^x with the hardware approximation (relative error about 2^-22).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// 1/x with the hardware approximation (relative error about 2^-23).
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// Whole warp: allocate ncols TMEM columns, address written to smem slot.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" :: "r"(slot), "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" :: "r"(taddr), "r"(ncols));
}

// 32 lanes x 16 consecutive 32-bit columns; lane i of the warp reads TMEM
// lane (taddr.lane + i). Includes the wait for completion.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

// D (TMEM) (+)= A (TMEM) * B (smem), whole (converged) warp, the elected lane
// issues. A is M x 16 bf16 held in TMEM: row m in lane m, elements 2c and 2c+1
// packed in column c (low half first), 8 columns per 16-element K step.
__device__ __forceinline__ void mma_bf16_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                 uint32_t acc) {
    asm volatile("{\n.reg .pred p, e;\nsetp.ne.b32 p, %4, 0;\nelect.sync _|e, 0xffffffff;\n"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
                 :: "r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

// 32 lanes x 32 consecutive 32-bit columns, without the completion wait (pair
// with tmem_wait_ld before the registers are used).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t* r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

// 32 lanes x 16 consecutive 32-bit columns from registers; pair with
// tmem_wait_st before the columns are read by an MMA or another thread.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16};\n"
                 :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                    "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
                    "r"(v[15])
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// Two floats as one word of bf16 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;\n" :: "r"(id), "r"(nthreads) : "memory");
}

// Byte offset of element (row, col) of a tile stored as 128-byte swizzled
// rows of 64 bf16, with regions of `region_rows` rows per 64 columns.
__device__ __forceinline__ uint32_t sw128_offset(int row, int col, int region_rows) {
    const int region = col >> 6, c = col & 63;
    return (uint32_t)(region * region_rows * 128 + row * 128 + ((((c >> 3) ^ (row & 7))) << 4) + ((c & 7) << 1));
}

// Reduces 16 values per lane across the warp so that lanes 2c and 2c+1 end up
// holding the reduction of column c (16 shuffles instead of 80).
template <bool kMax>
__device__ __forceinline__ float warp_reduce16(const float* v, int lane) {
    auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
    float w8[8], w4[4], w2[2];
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const float send = b4 ? v[i] : v[i + 8];
        const float keep = b4 ? v[i + 8] : v[i];
        w8[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float send = b3 ? w8[i] : w8[i + 4];
        const float keep = b3 ? w8[i + 4] : w8[i];
        w4[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
#pragma unroll
    for (int i = 0; i < 2; i++) {
        const float send = b2 ? w4[i] : w4[i + 2];
        const float keep = b2 ? w4[i + 2] : w4[i];
        w2[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
    const float send = b1 ? w2[0] : w2[1];
    const float keep = b1 ? w2[1] : w2[0];
    float r = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
    return op(r, __shfl_xor_sync(0xffffffffu, r, 1));
}

}  // namespace tc

// Host: a 2D bf16 tensor map over a row-major [rows, cols] matrix with a box
// of 16 rows x 64 columns and 128-byte swizzle (the layout the descriptors
// above describe). Returns LLSA_OK or LLSA_ERR_CUDA.
int make_tmap_bf16(CUtensorMap* map, const void* base, long long rows, int cols, int box_rows);

// Host: the tensor map of a bf16 token tensor [slices][n][d] for
// tma_load_block: the 2D map above (16-row boxes) in tile order, or under
// LLSA_ORDER_RASTER a 4D map [slices][side][side][d] with 4 x 4 token boxes
// of 64 columns and the same swizzle.
int make_tmap_tokens(CUtensorMap* map, const void* base, const Shape& s);

}  // namespace llsa
