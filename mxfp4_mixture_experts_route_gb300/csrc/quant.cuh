// Token rows of the expert GEMMs (the token gather kernel's arithmetic).
//
// For a valid pick of token t at sorted position r: rows 2r and 2r + 1 of xq hold
// hi = e4m3(x[t] / 2^s) and lo = e4m3(x[t] / 2^s - hi) for every 32-element
// block, and the scale table xs holds the block's e8m0 byte s + 127, chosen so
// that the block's largest magnitude divided by 2^s lies in [128, 256)
// (clamped to bytes 1..247).  For a bf16 x the two rows add up to x / 2^s
// exactly, but for elements more than 2^9 below the block maximum (there the
// error is below 2^-17 of it).  The unused bytes of the last stage's scale
// rows of xs and hs (K / 32 not a multiple of 8) are set to 127 (scale 1), as
// their codes are zero.
#pragma once

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {

// Eight consecutive elements of one token row, quantised: four consecutive
// threads hold one 32-element block (its scale byte `e` is the same in all
// four).
struct QuantChunk {
    uint2 hi, lo;
    int e;
};

// Eight bf16 elements v of one row (a thread's chunk).  All 32 lanes of the
// warp call it (the block maximum is taken across lanes); lanes past the row
// pass zeros (whole blocks of four threads, d / 8 being a multiple of 16).
__device__ __forceinline__ QuantChunk quantize_vals(const uint4 v) {
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        f[2 * j] = __uint_as_float(wv[j] << 16);
        f[2 * j + 1] = __uint_as_float(wv[j] & 0xFFFF0000u);
    }
    uint32_t amax = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = max(amax, __float_as_uint(fabsf(f[j])));
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int e = (int)((amax >> 23) & 0xFFu) - 7;
    e = e < 1 ? 1 : (e > 247 ? 247 : e);
    const float mult = __uint_as_float((uint32_t)(254 - e) << 23);   // 2^-(e - 127)
    uint32_t hw[2] = {0, 0}, lw[2] = {0, 0};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float a0 = f[2 * j] * mult, a1 = f[2 * j + 1] * mult;
        const uint32_t h2 = ptx::cvt_e4m3x2(a0, a1);
        float b0, b1;
        ptx::e4m3x2_to_f32(h2, b0, b1);
        const uint32_t l2 = ptx::cvt_e4m3x2(a0 - b0, a1 - b1);
        hw[j >> 1] |= h2 << (16 * (j & 1));
        lw[j >> 1] |= l2 << (16 * (j & 1));
    }
    QuantChunk q;
    q.hi = make_uint2(hw[0], hw[1]);
    q.lo = make_uint2(lw[0], lw[1]);
    q.e = e;
    return q;
}

// Elements 8c .. 8c+7 of the row `in` (d / 8 chunks; act = c < d / 8), an
// input of the call (read through the read-only path)
__device__ __forceinline__ QuantChunk quantize_chunk(const uint4* __restrict__ in, int c, bool act) {
    return quantize_vals(act ? __ldg(in + c) : make_uint4(0, 0, 0, 0));
}

// The same for a row an earlier kernel of the call wrote (read through L2)
__device__ __forceinline__ QuantChunk quantize_chunk_dep(const uint4* in, int c, bool act) {
    return quantize_vals(act ? ld_dep(in + c) : make_uint4(0, 0, 0, 0));
}

// Chunk c of pick row r: its hi and lo bytes, and (first thread of the block)
// the block's scale byte in row r of the scale table.
__device__ __forceinline__ void store_chunk(const QuantChunk& q, int c, int r, int d, size_t table_rows,
                                            uint8_t* __restrict__ xq, uint8_t* __restrict__ xs) {
    uint8_t* hi_row = xq + (size_t)(2 * r) * d;
    *reinterpret_cast<uint2*>(hi_row + 8 * c) = q.hi;
    *reinterpret_cast<uint2*>(hi_row + d + 8 * c) = q.lo;
    if ((c & 3) == 0) {
        const int blk = c >> 2;
        xs[((size_t)(blk >> 3) * table_rows + r) * TOKEN_SCALE_ROW + (blk & 7)] = (uint8_t)q.e;
    }
}

// The unused bytes of row r's last scale rows in xs and hs (by threads 0-7).
__device__ __forceinline__ void pad_scale_rows(int r, int d, int I, size_t table_rows, uint8_t* __restrict__ xs,
                                               uint8_t* __restrict__ hs, int tid) {
    if (tid < 8) {
        const int j = tid;
        const int nbx = d / 32, nbh = I / 32;
        if ((nbx & 7) && j >= (nbx & 7)) xs[((size_t)(nbx >> 3) * table_rows + r) * TOKEN_SCALE_ROW + j] = 127;
        if ((nbh & 7) && j >= (nbh & 7)) hs[((size_t)(nbh >> 3) * table_rows + r) * TOKEN_SCALE_ROW + j] = 127;
    }
}

}  // namespace moe
