// Tensor-core decode attention on 3-bit packed codes (one 128-wide rotation
// segment: WHT128 or SO(4) o WHT128) for up to 8 query heads per KV head.
//
// [RotaryQuant] Key design 3 and [TQ-MNN] §3.3: the QK dot products and the V
// accumulation run in the rotated domain directly on the packed codes; q is
// rotated once, the output once.  [Block-GTQ]: dequantised fp16 operands with
// fp32 accumulation on tensor cores, key-axis split with log-sum-exp merge.
//
// Each warp streams its own 16-token tiles (cp.async ring, 4 stages) and runs
//   QK:  S[16 tok x 8 heads] = K~[16 tok x 128] . q~[128 x 8]      (8 mma m16n8k16)
//   PV:  O[128 x 8 heads]   += V~^T[128 x 16 tok] . P[16 tok x 8]  (8 mma m16n8k16)
// with an online softmax between them.  K~ and V~ never exist in memory: the
// A operands are built in registers from the 3-bit codes by byte permutes:
// two codes at the same bit offset in two bytes of a token and the same two
// bytes of a second token form one selector of four 3-bit indices, and two
// PRMT lookups into 8-entry byte tables (low and high bytes of the fp16
// codebook) give four fp16 values.  The order in which a lane meets the 128
// coordinates is a fixed permutation; q~ (QK operand B) and the output
// dimensions (PV rows) follow the same permutation.
#include <stddef.h>

#include "tq_decode_common.cuh"

namespace {

constexpr int kTile = 16;
constexpr int kStages = 4;
constexpr int kRec = 48;   // bytes of one 3-bit record

// In a 48-bit window (two 24-bit groups, 16 codes), code pairs (PP[i], QQ[i])
// sit at the same bit offset in two bytes three bytes apart.
__host__ __device__ constexpr int pp_of(int i) { return i < 2 ? i : i < 4 ? i + 1 : i < 6 ? i + 2 : i == 6 ? 2 : 5; }
__host__ __device__ constexpr int qq_of(int i) { return pp_of(i) + 8; }

struct alignas(16) TcStage {
    uint8_t k[kTile * kRec];
    uint8_t v[kTile * kRec];
    uint8_t kn[kTile * 4];
    uint8_t vn[kTile * 4];
};

struct TcFinal {
    float wo[4][8][128];
    float wm[4][8];
    float wl[4][8];
    float ot[8][128];
};

struct TcSmem {
    union {
        TcStage ring[4][kStages];
        TcFinal fin;
    };
    alignas(16) float qts[8][128];
    int is_last;
};

struct Pools { uint32_t lo0, lo1, hi0, hi1; };

// Byte tables of the fp16 codebook scaled by s (chosen on the host so that s * c
// rounds almost exactly to fp16); 1/s is applied to the fp32 norm factors.
__device__ __forceinline__ Pools make_pools(const float* cent, float sc) {
    uint32_t u[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) u[i] = __half_as_ushort(__float2half_rn(sc * cent[i]));
    Pools p;
    p.lo0 = (u[0] & 255u) | ((u[1] & 255u) << 8) | ((u[2] & 255u) << 16) | ((u[3] & 255u) << 24);
    p.lo1 = (u[4] & 255u) | ((u[5] & 255u) << 8) | ((u[6] & 255u) << 16) | ((u[7] & 255u) << 24);
    p.hi0 = (u[0] >> 8) | ((u[1] >> 8) << 8) | ((u[2] >> 8) << 16) | ((u[3] >> 8) << 24);
    p.hi1 = (u[4] >> 8) | ((u[5] >> 8) << 8) | ((u[6] >> 8) << 16) | ((u[7] >> 8) << 24);
    return p;
}

// Five views of a token's 48-bit window held in two words (wa, wb); the window
// starts at bit 0 of wa (even window) or bit 16 (odd window).
struct Win { uint32_t b, f8, f16, s0, s8; };

__device__ __forceinline__ Win make_win(uint32_t wa, uint32_t wb, int base) {
    Win w;
    w.b = __funnelshift_rc(wa, wb, base);        // window bytes 0-3
    w.f8 = __funnelshift_rc(wa, wb, base + 8);   // bytes 1-4
    w.f16 = __funnelshift_rc(wa, wb, base + 16); // bytes 2-5
    w.s0 = __funnelshift_rc(wa, wb, base + 2);   // window >> 2: codes 2, 10 byte-aligned
    w.s8 = __funnelshift_rc(wa, wb, base + 10);  // window >> 10: codes 5, 13
    return w;
}

// Selector of four 3-bit indices from H = [A.bi, A.bj, B.bi, B.bj] at in-byte
// offset O, then the two byte-table lookups.  Nibbles: (A@p, B@p, A@q, B@q).
template <int O>
__device__ __forceinline__ void lookup4(uint32_t H, const Pools& pl, uint32_t& rlo, uint32_t& rhi) {
    const uint32_t t = (O ? __umulhi(H, 1u << (32 - O)) : H) & 0x07070707u;   // shift on the FMA pipe
    uint32_t sel;
    asm("mad.hi.u32 %0, %1, 1048576, %1;" : "=r"(sel) : "r"(t));   // t + (t >> 12)
    rlo = __byte_perm(pl.lo0, pl.lo1, sel);
    rhi = __byte_perm(pl.hi0, pl.hi1, sel);
}

__device__ __forceinline__ uint32_t view(const Win& w, int which) {
    return which == 0 ? w.b : which == 1 ? w.f8 : which == 2 ? w.f16 : which == 3 ? w.s0 : w.s8;
}

// Pattern i of a window pair: (view, in-byte offset) of code pair (PP[i], QQ[i]).
template <int I>
__device__ __forceinline__ void pattern(const Win& A, const Win& B, const Pools& pl, uint32_t& rlo, uint32_t& rhi) {
    constexpr int V = I < 2 ? 0 : I < 4 ? 1 : I < 6 ? 2 : I == 6 ? 3 : 4;
    constexpr int O = I == 0 ? 0 : I == 1 ? 3 : I == 2 ? 1 : I == 3 ? 4 : I == 4 ? 2 : I == 5 ? 5 : I == 6 ? 4 : 5;
    const uint32_t H = __byte_perm(view(A, V), view(B, V), 0x7430);
    lookup4<O>(H, pl, rlo, rhi);
}

__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma1688(float* d, uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(b0));
}

__device__ __forceinline__ void cp_async16s(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes));
}

__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

__device__ __forceinline__ float ldnorm(const uint8_t* p, int i, int f16) {
    return f16 ? __half2float(reinterpret_cast<const __half*>(p)[i]) : reinterpret_cast<const float*>(p)[i];
}

template <int GPE>
__global__ void __launch_bounds__(kThreads, 4) decode_tc3(DecodeArgs a) {
    __shared__ TcSmem S;
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = lane >> 2, c = lane & 3;
    const tq_head_params& P = a.params[h];
    const int L = clamp_len(a, b);
    const int t0 = s * a.split_len;
    const int t1 = min(t0 + a.split_len, L);
    const int ntiles = t1 > t0 ? (t1 - t0 + kTile - 1) / kTile : 0;
    const size_t head_tok = ((size_t)b * a.Hkv + h) * a.Tcap;
    const int nb = a.norm_f16 ? 2 : 4;
    TcStage* ring = S.ring[warp];

    // per-lane copy plan: chunk `lane` (and `lane + 32` for lanes < 16) of the
    // 768-byte K and V tiles, one 16-byte chunk of a norm tile for lanes 0..7
    const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(S.ring[warp]);
    const uint8_t* gk = a.k_codes + (head_tok + t0) * kRec + 16 * lane;
    const uint8_t* gv = a.v_codes + (head_tok + t0) * kRec + 16 * lane;
    const int nch = lane & 3;
    const bool has_n = lane < 8 && 16 * nch < kTile * nb;
    const uint8_t* gn = static_cast<const uint8_t*>(lane < 4 ? a.k_norms : a.v_norms) + (head_tok + t0) * nb + 16 * nch;
    const uint32_t on = (uint32_t)(lane < 4 ? offsetof(TcStage, kn) : offsetof(TcStage, vn)) + 16 * nch;
    const int nsec = t1 - t0;

    auto issue = [&](int tl, int st) {
        const uint32_t dst = ring_s + st * (uint32_t)sizeof(TcStage);
        const size_t co = (size_t)tl * (kTile * kRec);
        const int rem = nsec - tl * kTile;
        if (rem >= kTile) {
            cp_async16s(dst + offsetof(TcStage, k) + 16 * lane, gk + co, 16);
            cp_async16s(dst + offsetof(TcStage, v) + 16 * lane, gv + co, 16);
            if (lane < 16) {
                cp_async16s(dst + offsetof(TcStage, k) + 512 + 16 * lane, gk + co + 512, 16);
                cp_async16s(dst + offsetof(TcStage, v) + 512 + 16 * lane, gv + co + 512, 16);
            }
            if (has_n) cp_async16s(dst + on, gn + (size_t)tl * kTile * nb, 16);
        } else {
            const int cb = rem * kRec;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int ch = lane + 32 * k;
                if (ch < 48) {
                    const int n = min(16, max(0, cb - 16 * ch));
                    const size_t off = n ? co + 32 * 16 * k : 0;
                    cp_async16s(dst + offsetof(TcStage, k) + 16 * ch, n ? gk + off : gk - 16 * lane, n);
                    cp_async16s(dst + offsetof(TcStage, v) + 16 * ch, n ? gv + off : gv - 16 * lane, n);
                }
            }
            if (has_n) {
                const int n = min(16, max(0, rem * nb - 16 * nch));
                cp_async16s(dst + on, n ? gn + (size_t)tl * kTile * nb : gn - 16 * nch, n);
            }
        }
    };

    // start the stream before the prologue's q rotation
#pragma unroll
    for (int k = 0; k < kStages - 1; ++k) {
        const int tl = warp + 4 * k;
        if (tl < ntiles) issue(tl, k);
        cp_async_commit();
    }

    // q~ = R_K q for the (up to) 8 query heads, scaled to log2 units
    for (int g = warp; g < 8; g += 4) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (g < a.G) {
            const size_t elem = ((size_t)b * a.Hq + (size_t)h * a.G + g) * 128 + 4 * lane;
            tq::load4(a.q, elem, a.q_dtype, v);
            tq::rotate_forward(a.rot, P, v);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) S.qts[g][4 * lane + i] = v[i] * (kLog2e * kInvSqrtD);
    }
    const Pools pk = make_pools(P.k_cent[0], P.k_h_scale[0]);
    const Pools pv = make_pools(P.v_cent[0], P.v_h_scale[0]);
    const float kinv = 1.0f / P.k_h_scale[0], vinv = 1.0f / P.v_h_scale[0];
    __syncthreads();
    // QK operand B: lane (r, c) holds head r at the coordinates its A operand meets
    uint32_t bq[8][2];
#pragma unroll
    for (int st = 0; st < 8; ++st) {
        const int base = 32 * c + 16 * (st >> 2);
        const int i0 = 2 * (st & 3), i1 = i0 + 1;
        bq[st][0] = pack_h2(S.qts[r][base + pp_of(i0)], S.qts[r][base + qq_of(i0)]);
        bq[st][1] = pack_h2(S.qts[r][base + pp_of(i1)], S.qts[r][base + qq_of(i1)]);
    }

    float o[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const int vw = (3 * r) >> 1;          // first word of this lane row's V window
    const int vbase = (r & 1) ? 16 : 0;

    for (int it = 0;; ++it) {
        const int tl = warp + 4 * it;
        if (tl >= ntiles) break;
        {
            const int tn = warp + 4 * (it + kStages - 1);
            if (tn < ntiles) issue(tn, (it + kStages - 1) % kStages);
            cp_async_commit();
        }
        cp_async_wait<kStages - 1>();
        __syncwarp();
        const TcStage& sg = ring[it % kStages];
        const int nval = min(kTile, t1 - (t0 + tl * kTile));

        // ---- QK on tensor cores
        const uint32_t* kA = reinterpret_cast<const uint32_t*>(sg.k + r * kRec) + 3 * c;
        const uint32_t* kB = reinterpret_cast<const uint32_t*>(sg.k + (r + 8) * kRec) + 3 * c;
        const uint32_t a0 = kA[0], a1 = kA[1], a2 = kA[2];
        const uint32_t b0 = kB[0], b1 = kB[1], b2 = kB[2];
        float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ws = 0; ws < 2; ++ws) {
            const Win A = ws == 0 ? make_win(a0, a1, 0) : make_win(a1, a2, 16);
            const Win B = ws == 0 ? make_win(b0, b1, 0) : make_win(b1, b2, 16);
            uint32_t rl, rh, rl2, rh2;
            pattern<0>(A, B, pk, rl, rh);
            pattern<1>(A, B, pk, rl2, rh2);
            mma16816(d, __byte_perm(rl, rh, 0x6240), __byte_perm(rl, rh, 0x7351), __byte_perm(rl2, rh2, 0x6240),
                     __byte_perm(rl2, rh2, 0x7351), bq[4 * ws][0], bq[4 * ws][1]);
            pattern<2>(A, B, pk, rl, rh);
            pattern<3>(A, B, pk, rl2, rh2);
            mma16816(e, __byte_perm(rl, rh, 0x6240), __byte_perm(rl, rh, 0x7351), __byte_perm(rl2, rh2, 0x6240),
                     __byte_perm(rl2, rh2, 0x7351), bq[4 * ws + 1][0], bq[4 * ws + 1][1]);
            pattern<4>(A, B, pk, rl, rh);
            pattern<5>(A, B, pk, rl2, rh2);
            mma16816(d, __byte_perm(rl, rh, 0x6240), __byte_perm(rl, rh, 0x7351), __byte_perm(rl2, rh2, 0x6240),
                     __byte_perm(rl2, rh2, 0x7351), bq[4 * ws + 2][0], bq[4 * ws + 2][1]);
            pattern<6>(A, B, pk, rl, rh);
            pattern<7>(A, B, pk, rl2, rh2);
            mma16816(e, __byte_perm(rl, rh, 0x6240), __byte_perm(rl, rh, 0x7351), __byte_perm(rl2, rh2, 0x6240),
                     __byte_perm(rl2, rh2, 0x7351), bq[4 * ws + 3][0], bq[4 * ws + 3][1]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i] += e[i];

        // ---- online softmax (log2 units); lane holds tokens r, r+8 x heads 2c, 2c+1
        const bool vr0 = r < nval, vr8 = r + 8 < nval;
        const float kn0 = ldnorm(sg.kn, r, a.norm_f16) * kinv, kn8 = ldnorm(sg.kn, r + 8, a.norm_f16) * kinv;
        const float sc0 = vr0 ? d[0] * kn0 : -INFINITY;
        const float sc1 = vr0 ? d[1] * kn0 : -INFINITY;
        const float sc2 = vr8 ? d[2] * kn8 : -INFINITY;
        const float sc3 = vr8 ? d[3] * kn8 : -INFINITY;
        float mt0 = fmaxf(sc0, sc2), mt1 = fmaxf(sc1, sc3);
#pragma unroll
        for (int msk = 4; msk < 32; msk <<= 1) {
            mt0 = fmaxf(mt0, __shfl_xor_sync(TQ_FULL_MASK, mt0, msk));
            mt1 = fmaxf(mt1, __shfl_xor_sync(TQ_FULL_MASK, mt1, msk));
        }
        // the exponent base moves only when the tile max exceeds it by more than
        // 4 (log2 units): p <= 16 otherwise, and the accumulators are rescaled rarely
        const float mn0 = mt0 > m0 + 4.f ? mt0 : m0, mn1 = mt1 > m1 + 4.f ? mt1 : m1;
        const float c0 = m0 == -INFINITY ? 0.f : exp2f(m0 - mn0);
        const float c1 = m1 == -INFINITY ? 0.f : exp2f(m1 - mn1);
        const float p0 = exp2f(sc0 - mn0), p1 = exp2f(sc1 - mn1);
        const float p2 = exp2f(sc2 - mn0), p3 = exp2f(sc3 - mn1);
        if (!__all_sync(TQ_FULL_MASK, mn0 == m0 && mn1 == m1)) {
            l0 *= c0;
            l1 *= c1;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                o[i][0] *= c0; o[i][1] *= c1; o[i][2] *= c0; o[i][3] *= c1;
            }
        }
        l0 += p0 + p2;
        l1 += p1 + p3;
        m0 = mn0;
        m1 = mn1;
        const float vn0 = ldnorm(sg.vn, r, a.norm_f16) * vinv, vn8 = ldnorm(sg.vn, r + 8, a.norm_f16) * vinv;
        const uint32_t pb0 = movtrans(pack_h2(p0 * vn0, p1 * vn0));
        const uint32_t pb1 = movtrans(pack_h2(p2 * vn8, p3 * vn8));

        // ---- PV on tensor cores: rows = this lane row's window of the V record
        const uint32_t* v0 = reinterpret_cast<const uint32_t*>(sg.v + (2 * c) * kRec) + vw;
        const uint32_t* v1 = reinterpret_cast<const uint32_t*>(sg.v + (2 * c + 1) * kRec) + vw;
        const uint32_t* v2 = reinterpret_cast<const uint32_t*>(sg.v + (2 * c + 8) * kRec) + vw;
        const uint32_t* v3 = reinterpret_cast<const uint32_t*>(sg.v + (2 * c + 9) * kRec) + vw;
        {
            // tokens (2c, 2c+1) -> k-slots 0..7 of the tile, then (2c+8, 2c+9)
            const Win V0 = make_win(v0[0], v0[1], vbase), V1 = make_win(v1[0], v1[1], vbase);
            uint32_t rl, rh;
#define TQ_PV_HALF(I, VA, VB, PB)                                                                  \
    pattern<I>(VA, VB, pv, rl, rh);                                                                \
    mma1688(o[I], __byte_perm(rl, rh, 0x5140), __byte_perm(rl, rh, 0x7362), PB);
            TQ_PV_HALF(0, V0, V1, pb0) TQ_PV_HALF(1, V0, V1, pb0) TQ_PV_HALF(2, V0, V1, pb0)
            TQ_PV_HALF(3, V0, V1, pb0) TQ_PV_HALF(4, V0, V1, pb0) TQ_PV_HALF(5, V0, V1, pb0)
            TQ_PV_HALF(6, V0, V1, pb0) TQ_PV_HALF(7, V0, V1, pb0)
        }
        {
            const Win V2 = make_win(v2[0], v2[1], vbase), V3 = make_win(v3[0], v3[1], vbase);
            uint32_t rl, rh;
            TQ_PV_HALF(0, V2, V3, pb1) TQ_PV_HALF(1, V2, V3, pb1) TQ_PV_HALF(2, V2, V3, pb1)
            TQ_PV_HALF(3, V2, V3, pb1) TQ_PV_HALF(4, V2, V3, pb1) TQ_PV_HALF(5, V2, V3, pb1)
            TQ_PV_HALF(6, V2, V3, pb1) TQ_PV_HALF(7, V2, V3, pb1)
#undef TQ_PV_HALF
        }
        __syncwarp();
    }
    cp_async_wait<0>();

    // ---- per-warp state -> CTA state
#pragma unroll
    for (int msk = 4; msk < 32; msk <<= 1) {
        l0 += __shfl_xor_sync(TQ_FULL_MASK, l0, msk);
        l1 += __shfl_xor_sync(TQ_FULL_MASK, l1, msk);
    }
    __syncthreads();   // every warp is done with its ring before it is reused
    TcFinal& F = S.fin;
    if (r == 0) {
        F.wm[warp][2 * c] = m0; F.wm[warp][2 * c + 1] = m1;
        F.wl[warp][2 * c] = l0; F.wl[warp][2 * c + 1] = l1;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int dp = 16 * r + pp_of(i), dq = 16 * r + qq_of(i);
        F.wo[warp][2 * c][dp] = o[i][0];
        F.wo[warp][2 * c + 1][dp] = o[i][1];
        F.wo[warp][2 * c][dq] = o[i][2];
        F.wo[warp][2 * c + 1][dq] = o[i][3];
    }
    __syncthreads();
    float mm[GPE], ll[GPE];
#pragma unroll
    for (int g = 0; g < GPE; ++g) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, F.wm[w][g]);
        float Lt = 0.f, ov = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float wt = (M == -INFINITY || F.wm[w][g] == -INFINITY) ? 0.f : exp2f(F.wm[w][g] - M);
            Lt = fmaf(wt, F.wl[w][g], Lt);
            ov = fmaf(wt, F.wo[w][g][tid], ov);
        }
        mm[g] = M;
        ll[g] = Lt;
        F.ot[g][tid] = ov;
    }
    __syncthreads();
    epilogue<GPE>(a, P, F.ot, mm, ll, &S.is_last, b, h, s);
}

}  // namespace

bool tq_decode_tc_supported(const tq_cache_desc* d) {
    if (d->k_mixed || d->rot == TQ_ROT_WHT32) return false;
    if (d->k_bits != 3 || d->v_bits != 3 || d->group > 8) return false;
    // tile starts of the norm arrays must be 16-byte aligned
    return ((int64_t)d->t_capacity * d->norm_bytes) % 16 == 0;
}

int tq_decode_tc_split_align() { return kTile; }

cudaError_t tq_decode_tc_launch(const tq_cache_desc* d, const tq::DecodeArgs& a, int splits, cudaStream_t stream) {
    dim3 grid(splits, d->n_kv_heads, d->batch);
    if (d->group <= 1) decode_tc3<1><<<grid, kThreads, 0, stream>>>(a);
    else if (d->group <= 4) decode_tc3<4><<<grid, kThreads, 0, stream>>>(a);
    else decode_tc3<8><<<grid, kThreads, 0, stream>>>(a);
    return cudaPeekAtLastError();
}
