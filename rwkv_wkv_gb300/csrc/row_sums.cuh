// Row reductions of the decode kernels' thread mapping: a 64-wide row of the
// state sits in the 16 lanes of a half-warp, each lane holding 4 columns of 4
// rows (v[m]: this lane's partial of row m).
#pragma once

#include <cuda_runtime.h>

namespace wkv7 {

// The four row sums as a reduce-scatter: lane l of each half-warp ends with the
// sum of row (l >> 2) & 3.  The pairwise additions (partners at xor 8, 4, 2, 1,
// in that order) are those of a butterfly over each row, so the sums equal the
// butterfly's bit for bit, in 5 shuffles instead of 16.
__device__ __forceinline__ float reduce_scatter4(const float (&v)[4], int hl) {
    const bool b3 = (hl & 8) != 0, b2 = (hl & 4) != 0;
    const float t0 = (b3 ? v[2] : v[0]) + __shfl_xor_sync(0xffffffffu, b3 ? v[0] : v[2], 8);
    const float t1 = (b3 ? v[3] : v[1]) + __shfl_xor_sync(0xffffffffu, b3 ? v[1] : v[3], 8);
    float u = (b2 ? t1 : t0) + __shfl_xor_sync(0xffffffffu, b2 ? t0 : t1, 4);
    u += __shfl_xor_sync(0xffffffffu, u, 2);
    u += __shfl_xor_sync(0xffffffffu, u, 1);
    return u;
}

// All four row sums in every lane: the reduce-scatter, then a broadcast.
__device__ __forceinline__ void row_sums4(float (&v)[4], int lane) {
    const float u = reduce_scatter4(v, lane & 15);
#pragma unroll
    for (int m = 0; m < 4; ++m) v[m] = __shfl_sync(0xffffffffu, u, (lane & 16) | (4 * m));
}

}  // namespace wkv7
