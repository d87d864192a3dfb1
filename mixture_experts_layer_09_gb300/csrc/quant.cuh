// quant.cuh -- int16 activation groups for the integer dot products of the GEMV arm.
#pragma once

#include "common.cuh"

namespace moe {

// position of column j (0..7) of an 8-column word in the dp2a operand order
// [c0 c2 c4 c6 c1 c3 c5 c7]
__device__ __forceinline__ int dp2a_pos(int j) { return (j & 1) ? 4 + (j >> 1) : (j >> 1); }

// Position of column `col` of an activation row in its stored order.  A row is stored in
// slices of `kc` columns (the width the GEMV kernel stages at once); inside a slice, the
// 16-byte pieces (8 columns) are ordered [chunk / 8][piece in chunk][chunk % 8] so that the 8
// pieces a warp reads with one instruction are contiguous; inside a piece, columns are in
// dp2a order.
__device__ __forceinline__ int act_pos(int col, int kc) {
    const int sl = col / kc, cin = col % kc;
    const int c = cin >> 5, qq = (cin >> 3) & 3, w = cin & 7;
    return sl * kc + ((((c >> 3) * 4 + qq) * 8 + (c & 7)) << 3) + dp2a_pos(w);
}

// Quantise the 32 values held by a warp (one per lane) to int16 with a power-of-two scale.
// Writes the values into row `row_q` (group `grp`, stored order of slice width kc) and the
// group's {scale bits, integer sum} pair.
__device__ __forceinline__ void quantize_group(float v, int lane, int16_t* row_q, int grp, int kc, int2* meta) {
    const float amax = warp_max(fabsf(v));
    int q = 0;
    float scale = 1.f;
    if (amax > 0.f && amax <= 3.0e38f) {
        int ex;
        frexpf(amax, &ex);  // amax = m * 2^ex, m in [0.5, 1): |v| * 2^(15 - ex) < 2^15
        q = __float2int_rn(ldexpf(v, 15 - ex));
        q = max(-32767, min(32767, q));
        scale = ldexpf(1.f, ex - 15);
    }
    row_q[act_pos(grp * 32 + lane, kc)] = static_cast<int16_t>(q);
    const int qs = __reduce_add_sync(0xffffffffu, q);
    if (lane == 0) *meta = make_int2(__float_as_int(scale), qs);
}

// Stored row length of an activation of K columns: a multiple of 256 columns, so that every
// slice's pieces are whole groups of 8 chunks.
__host__ __device__ constexpr inline int act_row(int K) { return (K + 255) / 256 * 256; }

// Slice widths of the GEMV kernels: gate/up stages 512 columns of x, down 1024 columns of h.
constexpr int kSliceX = 512;
constexpr int kSliceH = 1024;

}  // namespace moe
