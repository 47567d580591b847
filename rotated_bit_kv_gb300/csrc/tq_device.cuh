// Device helpers shared by the write-side and read-side kernels.
//
// Vector convention: a 128-dim vector is held by one warp, four consecutive
// coordinates per lane (lane l holds coordinates 4l .. 4l+3).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tq_internal.h"

#define TQ_FULL_MASK 0xffffffffu

namespace tq {

__device__ __forceinline__ void load4(const void* base, size_t elem, int dtype, float v[4]) {
    if (dtype == TQ_F32) {
        float4 x = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else if (dtype == TQ_F16) {
        uint2 u = *reinterpret_cast<const uint2*>(static_cast<const __half*>(base) + elem);
        float2 a = __half22float2(*reinterpret_cast<__half2*>(&u.x));
        float2 b = __half22float2(*reinterpret_cast<__half2*>(&u.y));
        v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    } else {
        uint2 u = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + elem);
        v[0] = __uint_as_float(u.x << 16);
        v[1] = __uint_as_float(u.x & 0xffff0000u);
        v[2] = __uint_as_float(u.y << 16);
        v[3] = __uint_as_float(u.y & 0xffff0000u);
    }
}

// Unnormalised Walsh-Hadamard butterflies over the low `log2(lanes*4)` index
// bits: two in-lane stages (strides 1, 2) then shuffle stages over lane bits
// 1 .. lanes/2 (strides 4 .. 2*lanes).  Natural (Sylvester) order.
template <int LANES>
__device__ __forceinline__ void wht_warp(float v[4]) {
    float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2; v[1] = a1 + a3; v[2] = a0 - a2; v[3] = a1 - a3;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int m = 1; m < LANES; m <<= 1) {
        // upper lane: o - v, lower lane: v + o; one fma with an exact +-1 factor
        const float sgn = (lane & m) ? -1.f : 1.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float o = __shfl_xor_sync(TQ_FULL_MASK, v[i], m);
            v[i] = fmaf(sgn, v[i], o);
        }
    }
}

// Hamilton product of quaternions (w, x, y, z).
__device__ __forceinline__ void qmul(const float p[4], const float q[4], float r[4]) {
    r[0] = p[0] * q[0] - p[1] * q[1] - p[2] * q[2] - p[3] * q[3];
    r[1] = p[0] * q[1] + p[1] * q[0] + p[2] * q[3] - p[3] * q[2];
    r[2] = p[0] * q[2] - p[1] * q[3] + p[2] * q[0] + p[3] * q[1];
    r[3] = p[0] * q[3] + p[1] * q[2] - p[2] * q[1] + p[3] * q[0];
}

// v -> q_L v conj(q_R) on this lane's 4-dim block  [RotaryQuant, Key design 2]
__device__ __forceinline__ void so4_forward(const float* quat8, float v[4]) {
    float qL[4] = {quat8[0], quat8[1], quat8[2], quat8[3]};
    float qRc[4] = {quat8[4], -quat8[5], -quat8[6], -quat8[7]};
    float t[4];
    qmul(qL, v, t);
    qmul(t, qRc, v);
}

// transpose of the block map: v -> conj(q_L) v q_R (its inverse for unit quaternions)
__device__ __forceinline__ void so4_transpose(const float* quat8, float v[4]) {
    float qLc[4] = {quat8[0], -quat8[1], -quat8[2], -quat8[3]};
    float qR[4] = {quat8[4], quat8[5], quat8[6], quat8[7]};
    float t[4];
    qmul(qLc, v, t);
    qmul(t, qR, v);
}

// rotated = R x for the uniform rotation kinds (this lane's 4 coordinates).
__device__ __forceinline__ void rotate_forward(int rot, const tq_head_params& P, float v[4]) {
    const int lane = threadIdx.x & 31;
    if (rot == TQ_ROT_WHT128) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] *= P.signs[4 * lane + i];
        wht_warp<32>(v);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] *= 0.08838834764831845f;   // 1/sqrt(128)
    } else if (rot == TQ_ROT_WHT32) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] *= P.signs[4 * lane + i];
        wht_warp<8>(v);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] *= 0.17677669529663687f;   // 1/sqrt(32)
    } else {
        wht_warp<32>(v);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] *= 0.08838834764831845f;
        so4_forward(P.quat[lane], v);
    }
}

// x = R^T rotated for the uniform rotation kinds.
__device__ __forceinline__ void rotate_inverse(int rot, const tq_head_params& P, float v[4]) {
    const int lane = threadIdx.x & 31;
    if (rot == TQ_ROT_WHT128) {
        wht_warp<32>(v);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] *= 0.08838834764831845f * P.signs[4 * lane + i];
    } else if (rot == TQ_ROT_WHT32) {
        wht_warp<8>(v);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] *= 0.17677669529663687f * P.signs[4 * lane + i];
    } else {
        so4_transpose(P.quat[lane], v);
        wht_warp<32>(v);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] *= 0.08838834764831845f;
    }
}

// Mixed-rate keys: rotated[r] = sum over the columns of r's segment of
// kmat[r][c] * x[gcoord[c]]; `xs` is the warp's staged copy of x (128 floats).
__device__ __forceinline__ void rotate_forward_dense(const tq_head_params& P, const float* kmat,
                                                     const float* xs, float v[4]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = 4 * lane + i;
        int s = 0;
        while (s < 3 && r >= P.k_seg_start[s + 1]) ++s;
        const int c0 = P.k_seg_start[s], c1 = P.k_seg_start[s + 1];
        const float* row = kmat + (size_t)r * 128;
        float acc = 0.f;
        for (int c = c0; c < c1; ++c) acc = fmaf(row[c], xs[P.k_gcoord[c]], acc);
        v[i] = acc;
    }
}

// v = rows 4l .. 4l+3 of M xs for a 128 x 128 matrix stored transposed (MT,
// row-major: MT[c][j] = M[j][c], 16-byte aligned) and the warp's staged vector
// xs (128 floats, shared memory): per column one coalesced 16-byte load per lane
// and a broadcast of x_c.
__device__ __forceinline__ void dense_rows_t(const float* MT, const float* xs, float v[4]) {
    const int lane = threadIdx.x & 31;
    const float4* col = reinterpret_cast<const float4*>(MT) + lane;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
    for (int c = 0; c < 128; ++c) {
        const float4 m = __ldg(col + 32 * c);
        const float x = xs[c];
        a0 = fmaf(m.x, x, a0);
        a1 = fmaf(m.y, x, a1);
        a2 = fmaf(m.z, x, a2);
        a3 = fmaf(m.w, x, a3);
    }
    v[0] = a0; v[1] = a1; v[2] = a2; v[3] = a3;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m; m >>= 1) x += __shfl_xor_sync(TQ_FULL_MASK, x, m);
    return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int m = 16; m; m >>= 1) x = fmaxf(x, __shfl_xor_sync(TQ_FULL_MASK, x, m));
    return x;
}

__device__ __forceinline__ float load_norm(const void* base, size_t i, int norm_f16) {
    return norm_f16 ? __half2float(static_cast<const __half*>(base)[i]) : static_cast<const float*>(base)[i];
}

}  // namespace tq
