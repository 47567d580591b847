// Register-level helpers of the tensor-core kernels (decode on the tile layout,
// the unquantised-token prefix kernel): the legacy warp-level MMA, byte
// permutes, the 8x8 transpose, fp16 packing with the rounding remainder, 2^x,
// streaming loads, compile-time unrolling.  Internal linkage: included by one
// translation unit per kernel family.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <utility>

namespace {

__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// the same MMA with bf16 operands (A and B both bf16)
__device__ __forceinline__ void mma16816_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ float ex2(float x) {   // hardware 2^x (ftz); 2^-inf = 0
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint4 ldg_stream4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg_stream2(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg_u64(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ldg_u128(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

template <class Fn, int... I>
__device__ __forceinline__ void unroll_seq(Fn&& f, std::integer_sequence<int, I...>) {
    (f(std::integral_constant<int, I>{}), ...);
}
template <int N, class Fn>
__device__ __forceinline__ void unroll(Fn&& f) {
    unroll_seq(f, std::make_integer_sequence<int, N>{});
}

// bf16 pair of (x, y) (lo = false) or of what its bf16 rounding leaves (lo = true)
__device__ __forceinline__ uint32_t pack_part_bf(float x, float y, bool lo) {
    const uint32_t h = pack_bf2(x, y);
    if (!lo) return h;
    return pack_bf2(x - __uint_as_float(h << 16), y - __uint_as_float(h & 0xffff0000u));
}

// fp16 pair of (x, y) (lo = false) or of what the fp16 rounding of (x, y)
// leaves (lo = true)
__device__ __forceinline__ uint32_t pack_part(float x, float y, bool lo) {
    const uint32_t h = pack_h2(x, y);
    if (!lo) return h;
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
    return pack_h2(x - f.x, y - f.y);
}

__device__ __forceinline__ float h_lo(uint32_t x) { return __half2float(__ushort_as_half((unsigned short)(x & 0xFFFFu))); }
__device__ __forceinline__ float h_hi(uint32_t x) { return __half2float(__ushort_as_half((unsigned short)(x >> 16))); }

// Online-softmax state of one warp for NT groups of four heads; lane (r, c) holds
// head 4j + c: o~ at coordinates 32 mt + 2r + {0, 1, 16, 17} (unnormalised), the
// running base m (log2 units) and its part of the running sum l.
template <int NT>
struct WState {
    float o[NT][4][4];
    float m[NT], l[NT];
    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            m[j] = -INFINITY;
            l[j] = 0.f;
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) o[j][mt][0] = o[j][mt][1] = o[j][mt][2] = o[j][mt][3] = 0.f;
        }
    }
};


// Online softmax of one 16-token tile: scores (log2 units) s0 / s8 of tokens r and
// r + 8 for head 4j + c (lane (r, c)).  The base m moves only when a score passes
// m + 4, so every weight 2^(s - m) <= 16 and rescales of (l, o) are rare; the tile
// maximum (over the 8 lanes of a head) is formed only then.
template <int NT>
__device__ __forceinline__ void tile_softmax(const float (&s0)[NT], const float (&s8)[NT], WState<NT>& ws) {
    bool move = false;
#pragma unroll
    for (int j = 0; j < NT; ++j) move = move || s0[j] > ws.m[j] + 4.f || s8[j] > ws.m[j] + 4.f;
    if (__any_sync(0xffffffffu, move)) {
        float mn[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            float mt = fmaxf(s0[j], s8[j]);
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
            mn[j] = mt > ws.m[j] + 4.f ? mt : ws.m[j];
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const float cf = ex2(ws.m[j] - mn[j]);   // 0 on the first tile (m = -inf)
            ws.l[j] *= cf;
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                ws.o[j][mt][0] *= cf; ws.o[j][mt][1] *= cf; ws.o[j][mt][2] *= cf; ws.o[j][mt][3] *= cf;
            }
            ws.m[j] = mn[j];
        }
    }
}

// The PV operand B of one head group from the weights p0 / p8 of tokens r and
// r + 8 (lane (r, c), head 4j + c): after the 8x8 transposes lane (r, c) holds, for
// head r/2, tokens 2c, 2c+1 (k step 0: b0, b1) and 2c+8, 2c+9 (k step 1), each
// weight in the column of its parity (selectors sel_lo / sel_hi of the lane).
__device__ __forceinline__ void p_operand_words(uint32_t w0, uint32_t w8, uint32_t sel_lo, uint32_t sel_hi,
                                                uint32_t (&bp)[2][2]) {
    const uint32_t t0 = movtrans(w0), t1 = movtrans(w8);
    bp[0][0] = prmt(t0, 0u, sel_lo);
    bp[0][1] = prmt(t0, 0u, sel_hi);
    bp[1][0] = prmt(t1, 0u, sel_lo);
    bp[1][1] = prmt(t1, 0u, sel_hi);
}

__device__ __forceinline__ void p_operand(float p0, float p8, uint32_t sel_lo, uint32_t sel_hi, uint32_t (&bp)[2][2]) {
    const uint32_t t0 = movtrans(pack_h2(p0, p0)), t1 = movtrans(pack_h2(p8, p8));
    bp[0][0] = prmt(t0, 0u, sel_lo);
    bp[0][1] = prmt(t0, 0u, sel_hi);
    bp[1][0] = prmt(t1, 0u, sel_lo);
    bp[1][1] = prmt(t1, 0u, sel_hi);
}

}  // namespace
