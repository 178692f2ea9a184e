// Blocked inverse of a 64 x 64 unit lower-triangular matrix on CUDA cores (fp32), shared by
// the tensor-core chunk kernel and the chunked backward.
#pragma once

#include "ptx.cuh"

namespace efla {

// T~ = (I + A~)^{-1} for a 64 x 64 unit lower-triangular I + A~, in place in At (fp32, row
// stride LD, a multiple of 4), by 256 threads (index pi) that meet at named barrier BAR.  The
// scratch Y of the products lives in the upper-right 32x32 block of At, which the inverse
// never reads.
// Each step applies
//   [[L1, 0], [B, L2]]^{-1} = [[L1^{-1}, 0], [-L2^{-1} B L1^{-1}, L2^{-1}]]
// for unit lower-triangular L1, L2:
//   1. the eight diagonal 8x8 blocks by column substitution: warps 0 and 1 of the
//      256 threads, four blocks per warp, one lane per column holding the whole column in
//      registers (no shuffles; the other warps wait at the barrier);
//   2. the off-diagonal 8x8 block of each diagonal 16x16 block, one output per thread;
//   3. blocks (1,0) and (3,2) of 16:  T~_IJ = -T~_II (A~_IJ T~_JJ);
//   4. the lower-left 32x32 block:    T~_21 = -T~_22 (A~_21 T~_11)  (32x32 blocks).
// Steps 3 and 4 are register-tiled fp32 products.
template <int BAR, int LD>
__device__ __forceinline__ void invert_unit_lower(float *At, int pi) {
    float *Y = At + 32;  // [32][LD] rows 0-31, columns 32-63
    const int lane = pi & 31, pw = pi >> 5;
    if (pw < 2) {  // 1. the eight diagonal 8x8 blocks, one lane per column
        const int B0 = 8 * (4 * pw + (lane >> 3)), c = lane & 7;
        float col[8];  // col[s] = T~[B0 + s][B0 + c]
#pragma unroll
        for (int s = 0; s < 8; ++s) col[s] = s == c ? 1.f : 0.f;
#pragma unroll
        for (int t = 1; t < 8; ++t) {
            const float4 r0 = *reinterpret_cast<const float4 *>(At + (B0 + t) * LD + B0);
            const float4 r1 = *reinterpret_cast<const float4 *>(At + (B0 + t) * LD + B0 + 4);
            const float a[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
            float a0 = 0.f, a1 = 0.f;  // A~[t][s] for s < t; col[s] = 0 for s < c
#pragma unroll
            for (int s = 0; s < 8; s += 2) {
                if (s < t) a0 = fmaf(a[s], col[s], a0);
                if (s + 1 < t) a1 = fmaf(a[s + 1], col[s + 1], a1);
            }
            col[t] = t > c ? -(a0 + a1) : col[t];
        }
        __syncwarp();  // the four blocks of this warp have been read
#pragma unroll
        for (int s = 0; s < 8; ++s) At[(B0 + s) * LD + B0 + c] = col[s];
    }
    ptx::named_bar(BAR, 256);
    {  // 2. 8 -> 16 within each diagonal 16x16 block: T~_21 = -T~_22 (A~_21 T~_11), 8x8 blocks;
       //    one output per thread, the intermediate in the unused upper-right block
        const int q = pi >> 6, r = (pi >> 3) & 7, cc = pi & 7;
        const int R0 = 16 * q;
        const float *arow = At + (R0 + 8 + r) * LD + R0;  // A~_21 row r
        float y = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) y = fmaf(arow[k], At[(R0 + k) * LD + R0 + cc], y);
        At[(8 * q + r) * LD + 32 + cc] = y;
        ptx::named_bar(BAR, 256);
        const float *trow = At + (R0 + 8 + r) * LD + R0 + 8;  // T~_22 row r
        float z = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) z = fmaf(trow[k], At[(8 * q + k) * LD + 32 + cc], z);
        At[(R0 + 8 + r) * LD + R0 + cc] = -z;
    }
    ptx::named_bar(BAR, 256);
    {
        const int q = pi >> 7, tt = pi & 127;
        const int I = 2 * q + 1, J = 2 * q;
        const int r = tt >> 3, c0 = (tt & 7) * 2;
        float *yq = Y + q * (16 * LD);  // [16][LD]
        float y0 = 0.f, y1 = 0.f;
        const float *arow = At + (16 * I + r) * LD + 16 * J;
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(arow + k4);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 bv = *reinterpret_cast<const float2 *>(At + (16 * J + k4 + e) * LD + 16 * J + c0);
                y0 = fmaf(av[e], bv.x, y0);
                y1 = fmaf(av[e], bv.y, y1);
            }
        }
        *reinterpret_cast<float2 *>(yq + r * LD + c0) = make_float2(y0, y1);
        ptx::named_bar(BAR, 256);
        float z0 = 0.f, z1 = 0.f;
        const float *trow = At + (16 * I + r) * LD + 16 * I;  // T~_II row r (zeros above the diagonal)
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {
            const float4 tq = *reinterpret_cast<const float4 *>(trow + k4);
            const float tv[4] = {tq.x, tq.y, tq.z, tq.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 yv = *reinterpret_cast<const float2 *>(yq + (k4 + e) * LD + c0);
                z0 = fmaf(tv[e], yv.x, z0);
                z1 = fmaf(tv[e], yv.y, z1);
            }
        }
        // nobody reads block (I, J) in this phase: write it at once
        *reinterpret_cast<float2 *>(At + (16 * I + r) * LD + 16 * J + c0) = make_float2(-z0, -z1);
        ptx::named_bar(BAR, 256);
    }
    {
        const int r0 = 2 * (pi >> 4), c0 = 2 * (pi & 15);
        float x00 = 0.f, x01 = 0.f, x10 = 0.f, x11 = 0.f;
        const float *a0 = At + (32 + r0) * LD, *a1 = a0 + LD;
#pragma unroll 2
        for (int k4 = 0; k4 < 32; k4 += 4) {
            const float4 p0 = *reinterpret_cast<const float4 *>(a0 + k4);
            const float4 p1 = *reinterpret_cast<const float4 *>(a1 + k4);
            const float va0[4] = {p0.x, p0.y, p0.z, p0.w}, va1[4] = {p1.x, p1.y, p1.z, p1.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 bv = *reinterpret_cast<const float2 *>(At + (k4 + e) * LD + c0);  // T~_11
                x00 = fmaf(va0[e], bv.x, x00);
                x01 = fmaf(va0[e], bv.y, x01);
                x10 = fmaf(va1[e], bv.x, x10);
                x11 = fmaf(va1[e], bv.y, x11);
            }
        }
        *reinterpret_cast<float2 *>(Y + r0 * LD + c0) = make_float2(x00, x01);
        *reinterpret_cast<float2 *>(Y + (r0 + 1) * LD + c0) = make_float2(x10, x11);
        ptx::named_bar(BAR, 256);
        float z00 = 0.f, z01 = 0.f, z10 = 0.f, z11 = 0.f;
        const float *t0 = At + (32 + r0) * LD + 32, *t1 = t0 + LD;  // T~_22 rows
#pragma unroll 2
        for (int k4 = 0; k4 < 32; k4 += 4) {
            const float4 p0 = *reinterpret_cast<const float4 *>(t0 + k4);
            const float4 p1 = *reinterpret_cast<const float4 *>(t1 + k4);
            const float tv0[4] = {p0.x, p0.y, p0.z, p0.w}, tv1[4] = {p1.x, p1.y, p1.z, p1.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 xv = *reinterpret_cast<const float2 *>(Y + (k4 + e) * LD + c0);
                z00 = fmaf(tv0[e], xv.x, z00);
                z01 = fmaf(tv0[e], xv.y, z01);
                z10 = fmaf(tv1[e], xv.x, z10);
                z11 = fmaf(tv1[e], xv.y, z11);
            }
        }
        // nobody reads the lower-left block in this phase: write it at once
        *reinterpret_cast<float2 *>(At + (32 + r0) * LD + c0) = make_float2(-z00, -z01);
        *reinterpret_cast<float2 *>(At + (33 + r0) * LD + c0) = make_float2(-z10, -z11);
        ptx::named_bar(BAR, 256);
    }
}

}  // namespace efla
