// reorder.cu -- hierarchical tile order of the tokens of a square image.
//
// Method: Pith review of arXiv 2512.16615, referee comments on Sec. 5.1 and
// Figure 2 (index reordering): tokens are reordered so that contiguous
// B-token blocks are compact in the image. Reading (the page gives no
// formula): with B = s^2 and an s^m x s^m raster image, every run of B^l
// consecutive positions in the new order is an s^l x s^l square of pixels,
// recursively. Pixel (r, c) with base-s digits r_k, c_k goes to position
// sum_k (r_k * s + c_k) * B^k.
//
// The kernel is a permutation of [slices][N][d] rows: one thread per 16-byte
// vector of an output row; a row (d * element bytes, a multiple of 16) is
// read from its source position as consecutive 16-byte vectors, so every
// access is a whole, aligned sector run. HBM-bound: it reads and writes
// slices * N * d elements once.
#include <algorithm>

#include "internal.h"

namespace llsa {
namespace {

struct ReorderArgs {
    const uint4* in;
    uint4* out;
    long long slices;
    int n, vec_per_row, s, m, width;
    int inverse;  // 0: raster -> tile order; 1: tile order -> raster
};

// tile position of raster token t
__device__ __forceinline__ int tile_pos(int t, int width, int s, int m) {
    int r = t / width, c = t - r * width;
    int p = 0, mult = 1;
    for (int k = 0; k < m; k++) {
        const int rk = r % s, ck = c % s;
        r /= s;
        c /= s;
        p += (rk * s + ck) * mult;
        mult *= s * s;
    }
    return p;
}

// raster token of tile position p
__device__ __forceinline__ int raster_pos(int p, int width, int s, int m) {
    int r = 0, c = 0, mult = 1;
    const int B = s * s;
    for (int k = 0; k < m; k++) {
        const int dk = p % B;
        p /= B;
        r += (dk / s) * mult;
        c += (dk % s) * mult;
        mult *= s;
    }
    return r * width + c;
}

__global__ void __launch_bounds__(256) reorder_kernel(ReorderArgs a) {
    const long long per_slice = (long long)a.n * a.vec_per_row;
    const long long total = a.slices * per_slice;
    for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
         g += (long long)gridDim.x * blockDim.x) {
        const long long slice = g / per_slice;
        const long long rem = g - slice * per_slice;
        const int o = (int)(rem / a.vec_per_row), v = (int)(rem - (long long)o * a.vec_per_row);
        // forward: out[tile_pos(t)] = in[t], so output position o reads raster_pos(o)
        const int src = a.inverse ? tile_pos(o, a.width, a.s, a.m) : raster_pos(o, a.width, a.s, a.m);
        a.out[g] = __ldcs(a.in + (slice * a.n + src) * (long long)a.vec_per_row + v);
    }
}

}  // namespace

int launch_reorder(const Shape& s, int side, int root, int digits, const void* in, void* out, int inverse,
                   cudaStream_t st) {
    ReorderArgs a;
    a.in = static_cast<const uint4*>(in);
    a.out = static_cast<uint4*>(out);
    a.slices = s.slices;
    a.n = s.n;
    a.vec_per_row = s.d * (s.dtype == LLSA_DTYPE_BF16 ? 2 : 4) / 16;
    a.s = root;
    a.m = digits;
    a.width = side;
    a.inverse = inverse;
    const long long total = a.slices * (long long)a.n * a.vec_per_row;
    const int grid = (int)std::min<long long>((total + 255) / 256, (long long)sm_count() * 16);
    LLSA_LAUNCH("reorder", st, reorder_kernel<<<grid, 256, 0, st>>>(a));
    return LLSA_OK;
}

}  // namespace llsa
