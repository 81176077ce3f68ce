// internal.h -- helpers shared by the translation units of the LLSA CUDA
// library (not installed; the public boundary is include/llsa.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "llsa.h"

namespace llsa {

// ---------------------------------------------------------------- shapes --

// Everything a launcher needs, derived once from llsa_params.
struct Shape {
    long long slices;  // batch * heads
    int n, d, B, L, Le, K1, T, P;
    int dtype;
    float scale;
    int rule;  // enrichment rule (LLSA_ENRICH_*)
    int topk;  // K as requested (before the per-level clamp)
    int raster, side;  // token tensors in the raster order of a side x side image (LLSA_ORDER_RASTER)
    // enrichment columns: C per coarse_idx row (levels 1..L), Lc of them used
    // (levels 1..L_e, a prefix); level l owns columns col_off[l] .. col_off[l+1]-1
    int C, Lc;
    int col_off[LLSA_MAX_LEVELS + 2];
    int n_level[LLSA_MAX_LEVELS + 1];
    int topk_level[LLSA_MAX_LEVELS + 1];
    int row_offset[LLSA_MAX_LEVELS + 1];
    long long level_idx_offset[LLSA_MAX_LEVELS + 1];
    long long level_idx_per_slice;
};

constexpr int kMaxCoarse = 64;  // coarse keys per query (ALLK)

// Level tables passed by value to kernels.
struct LevelTable {
    int row_offset[LLSA_MAX_LEVELS + 1];
    int n_level[LLSA_MAX_LEVELS + 1];
};

inline LevelTable level_table(const Shape& s) {
    LevelTable t;
    for (int l = 0; l <= LLSA_MAX_LEVELS; l++) {
        t.row_offset[l] = s.row_offset[l];
        t.n_level[l] = s.n_level[l];
    }
    return t;
}

// ----------------------------------------------------------- token order --

// The kernels work in the hierarchical tile order. With B = 16 the blocks of
// 16 consecutive tokens are 4 x 4 patches of the image: block b's base-16
// digits (finest first) are row digit * 4 + column digit of its patch, so the
// patch's top-left pixel is (4 py, 4 px), and token w of the block is pixel
// (4 py + w / 4, 4 px + w % 4). Under LLSA_ORDER_RASTER the token tensors are
// addressed through these two maps instead of being permuted first.
__host__ __device__ __forceinline__ void block_patch(int b, int& px, int& py) {
    px = 0;
    py = 0;
#pragma unroll
    for (int k = 0; k < 8; k++) {
        px |= ((b >> (4 * k)) & 3) << (2 * k);
        py |= ((b >> (4 * k + 2)) & 3) << (2 * k);
    }
}

// Row (in [slices * n]) of the token at tile position t of slice `slice`.
__host__ __device__ __forceinline__ long long token_row(long long slice, int n, int raster, int side, int t) {
    if (!raster) return slice * n + t;
    int px, py;
    block_patch(t >> 4, px, py);
    return slice * n + (long long)(4 * py + ((t >> 2) & 3)) * side + 4 * px + (t & 3);
}

// Rows from a block's first token to its token w: w in tile order
// (row_stride 4), or row w / 4 and column w % 4 of the block's patch in raster
// order (row_stride = the image side).
__host__ __device__ __forceinline__ long long block_token_offset(int w, int row_stride) {
    return (long long)(w >> 2) * row_stride + (w & 3);
}

// ------------------------------------------------------------ launching --

// Called around every kernel launch: profiling events, launch count and the
// launch error check. `end` returns LLSA_OK or LLSA_ERR_CUDA.
void launch_begin(const char* name, cudaStream_t st);
int launch_end(const char* name, cudaStream_t st);

#define LLSA_LAUNCH(name, stream, ...)                          \
    do {                                                        \
        ::llsa::launch_begin(name, stream);                     \
        __VA_ARGS__;                                            \
        int _llsa_rc = ::llsa::launch_end(name, stream);        \
        if (_llsa_rc != LLSA_OK) return _llsa_rc;               \
    } while (0)

#define LLSA_TRY(expr)                                          \
    do {                                                        \
        int _llsa_rc = (expr);                                  \
        if (_llsa_rc != LLSA_OK) return _llsa_rc;               \
    } while (0)

// Device status word of the current device (LLSA_ERR_* codes, first wins).
int* status_ptr();

// Number of SMs of the current device.
int sm_count();

// Polls before a bounded device wait gives up, and the test switches, as set
// by llsa_test_set_wait_limit (defaults: the kernels' own limit, no switch).
int wait_limit();
int test_flags();

// LLSA_OK when the current device is a GB300 (compute capability 10.3); also
// sets up the per-device status word on first use.
int device_ready();

// ---------------------------------------------------------------- launchers

int launch_pool(const Shape& s, const void* q, const void* k, const void* v, float* pyr, cudaStream_t st);
int launch_select(const Shape& s, const float* pyr, int32_t* sel_idx, int32_t* coarse_idx, int32_t* level_idx,
                  cudaStream_t st);
size_t fwd_workspace_bytes(const Shape& s);
int launch_fwd(const Shape& s, const void* q, const void* k, const void* v, const float* pyr,
               const int32_t* sel_idx, const int32_t* coarse_idx, void* o, float* lse, void* ws, cudaStream_t st);
int launch_select_exhaustive(const Shape& s, const float* pyr, int32_t* out, cudaStream_t st);
int launch_reorder(const Shape& s, int side, int root, int digits, const void* in, void* out, int inverse,
                   cudaStream_t st);
int launch_transpose(const Shape& s, const int32_t* sel, int rows, int K, int ncols, int32_t* col_ptr,
                     int32_t* row_idx, int32_t* scratch, cudaStream_t st);
size_t bwd_workspace_bytes(const Shape& s);
int launch_bwd(const Shape& s, const void* q, const void* k, const void* v, const void* o, const float* lse,
               const void* dout, const float* pyr, const int32_t* sel_idx, const int32_t* coarse_idx,
               const int32_t* col_ptr, const int32_t* row_idx, void* dq, void* dk, void* dv, void* ws,
               cudaStream_t st);

// ------------------------------------------------------- device helpers --

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* f) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ void load8(const float* p, float* f) {
    float4 a = __ldg(reinterpret_cast<const float4*>(p));
    float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ void store4(__nv_bfloat16* p, const float* f) {
    __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]);
    __nv_bfloat162 b = __floats2bfloat162_rn(f[2], f[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ void store4(float* p, const float* f) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Records the first error code into the status word.
__device__ __forceinline__ void set_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

}  // namespace llsa
