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

#include <utility>

#include "tq_decode_common.cuh"

namespace {

// keys through the code-pair table (1) or through byte-permute lookups (0)
#ifndef TQ_TC_KEY_TABLE
#define TQ_TC_KEY_TABLE 1
#endif

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
    alignas(16) uint32_t tab[64 * 32];
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
__device__ __forceinline__ void lookup4(uint32_t H, const Pools& pl, uint32_t fm, uint32_t& rlo, uint32_t& rhi) {
    const uint32_t t = (O ? __umulhi(H, 1u << (32 - O)) : H) & 0x07070707u;   // shift on the FMA pipe
    uint32_t sel;
    asm("mad.hi.u32 %0, %1, %2, %1;" : "=r"(sel) : "r"(t), "r"(fm));   // t + (t >> 12), fm = 1 << 20
    rlo = __byte_perm(pl.lo0, pl.lo1, sel);
    rhi = __byte_perm(pl.hi0, pl.hi1, sel);
}

template <int V>
__device__ __forceinline__ uint32_t view(const Win& w) {
    return V == 0 ? w.b : V == 1 ? w.f8 : V == 2 ? w.f16 : V == 3 ? w.s0 : w.s8;
}

// Pattern i of a window pair: (view, in-byte offset) of code pair (PP[i], QQ[i]).
template <int I>
__device__ __forceinline__ void pattern(const Win& A, const Win& B, const Pools& pl, uint32_t fm, uint32_t& rlo,
                                        uint32_t& rhi) {
    constexpr int V = I < 2 ? 0 : I < 4 ? 1 : I < 6 ? 2 : I == 6 ? 3 : 4;
    constexpr int O = I == 0 ? 0 : I == 1 ? 3 : I == 2 ? 1 : I == 3 ? 4 : I == 4 ? 2 : I == 5 ? 5 : I == 6 ? 4 : 5;
    const uint32_t H = __byte_perm(view<V>(A), view<V>(B), 0x7430);
    lookup4<O>(H, pl, fm, rlo, rhi);
}

__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

// PRMT in its generic mode: a selector nibble with bit 3 set replicates the sign
// bit of the chosen byte (the __byte_perm intrinsic keeps only bits 0-2)
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ float ex2(float x) {   // hardware 2^x (ftz); 2^-inf = 0
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float ldnorm(const uint8_t* p, int i, int f16) {
    return f16 ? __half2float(reinterpret_cast<const __half*>(p)[i]) : reinterpret_cast<const float*>(p)[i];
}

// ---- shared-memory table route
//
// tab[e][lane] = fp16x2 (s c[e & 7], s c[e >> 3]) for the 64 values e of a 6-bit
// field (two consecutive 3-bit codes, the lower one in the low half).  Every lane
// reads its own copy (bank = lane), so a warp's 32 lookups take one pass.

// the word for a field that `t` carries at bits 7..12 (other bits of t arbitrary)
__device__ __forceinline__ uint32_t tab_lk(const uint32_t* tab, uint32_t t, uint32_t lane4) {
    return *reinterpret_cast<const uint32_t*>(reinterpret_cast<const char*>(tab) + ((t & 0x1F80u) | lane4));
}

// the 6-bit field at bit P of w, moved to bits 7..12
template <int P>
__device__ __forceinline__ uint32_t at7(uint32_t w) {
    if constexpr (P < 7) return w * (1u << (7 - P));
    else if constexpr (P > 7) return __umulhi(w, 1u << (39 - P));
    else return w;
}

// field F (bits 6F .. 6F+5) of a 96-bit key chunk (w0, w1, w2), moved to bits 7..12
template <int F>
__device__ __forceinline__ uint32_t kfield7(uint32_t w0, uint32_t w1, uint32_t w2) {
    if constexpr (F < 5) return at7<6 * F>(w0);
    else if constexpr (F == 5) return __funnelshift_r(w0, w1, 23);
    else if constexpr (F < 10) return at7<6 * F - 32>(w1);
    else if constexpr (F == 10) return __funnelshift_r(w1, w2, 21);
    else return at7<6 * F - 64>(w2);
}

// field I of a 48-bit value window held as L (bits 0..31) and H (bits 32..47 at 0..15)
template <int I>
__device__ __forceinline__ uint32_t vfield7(uint32_t L, uint32_t H) {
    if constexpr (I < 5) return at7<6 * I>(L);
    else if constexpr (I == 5) return __funnelshift_r(L, H, 23);
    else return at7<6 * I - 32>(H);
}

template <class Fn, int... I>
__device__ __forceinline__ void unroll_seq(Fn&& f, std::integer_sequence<int, I...>) {
    (f(std::integral_constant<int, I>{}), ...);
}
template <int N, class Fn>
__device__ __forceinline__ void unroll(Fn&& f) {
    unroll_seq(f, std::make_integer_sequence<int, N>{});
}

// GPE: query heads computed per KV head (4 or 8, two MMA columns each);
// EP: heads kept by the epilogue (padded group); KLDS: keys through the table
// (else through byte-permute lookups).
template <int GPE, int EP, bool KLDS>
__global__ void __launch_bounds__(kThreads, GPE <= 4 ? 5 : 4) decode_tc4(DecodeArgs a) {
    constexpr int NT = GPE / 4;   // groups of four heads: n tiles of both products
    constexpr int NC = 4 / NT;    // independent QK accumulators per n tile
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

    // start the stream before the prologue
#pragma unroll
    for (int k = 0; k < kStages - 1; ++k) {
        const int tl = warp + 4 * k;
        if (tl < ntiles) issue(tl, k);
        cp_async_commit();
    }

    // code-pair table (keys and values share it: both are 3-bit codes of one
    // 128-coordinate segment, so their codebooks and fp16 scales coincide)
    {
        const float sv = P.v_h_scale[0];
        for (int i = tid; i < 64 * 32; i += kThreads) {
            const int e = i >> 5;
            S.tab[i] = pack_h2(sv * P.v_cent[0][e & 7], sv * P.v_cent[0][e >> 3]);
        }
    }
    // q~ = R_K q for the computed heads, scaled to log2 units
    for (int g = warp; g < GPE; g += 4) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (g < a.G) {
            const size_t elem = ((size_t)b * a.Hq + (size_t)h * a.G + g) * 128 + 4 * lane;
            tq::load4(a.q, elem, a.q_dtype, v);
            tq::rotate_forward(a.rot, P, v);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) S.qts[g][4 * lane + i] = v[i] * (kLog2e * kInvSqrtD);
    }
    Pools pk{};
    if constexpr (!KLDS) pk = make_pools(P.k_cent[0], P.k_h_scale[0]);
    const float kinv = 1.0f / P.k_h_scale[0], vinv = 1.0f / P.v_h_scale[0];
    const uint32_t fm = a.fold_mul;
    __syncthreads();

    // QK operand B: column r of n tile j is head 4j + r/2; lane c's k slots of
    // step st are the coordinates its A registers carry
    uint32_t bq[NT][8][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const float* qh = S.qts[4 * j + (r >> 1)];
#pragma unroll
        for (int st = 0; st < 8; ++st) {
            if constexpr (KLDS) {
                const int d0 = 32 * c + 2 * st, d1 = 32 * c + 2 * (st + 8);
                bq[j][st][0] = pack_h2(qh[d0], qh[d0 + 1]);
                bq[j][st][1] = pack_h2(qh[d1], qh[d1 + 1]);
            } else {
                const int base = 32 * c + 16 * (st >> 2);
                const int i0 = 2 * (st & 3), i1 = i0 + 1;
                bq[j][st][0] = pack_h2(qh[base + pp_of(i0)], qh[base + qq_of(i0)]);
                bq[j][st][1] = pack_h2(qh[base + pp_of(i1)], qh[base + qq_of(i1)]);
            }
        }
    }

    float o[NT][4][4];
    float m_[NT], l_[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        m_[j] = -INFINITY;
        l_[j] = 0.f;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) o[j][mt][0] = o[j][mt][1] = o[j][mt][2] = o[j][mt][3] = 0.f;
    }
    const uint32_t lane4 = 4u * lane;
    const uint32_t* tab = S.tab;
    const int vw = (3 * r) >> 1;                 // first word of this lane row's 48-bit value window
    const uint32_t vsh = (r & 1) ? 16u : 0u;     // its bit offset in that word
    // PV operand B: bytes 0-3 = (x_r, x_r+8) of this lane, 4-7 = those of lane row
    // r ^ 1; nibble 9 gives a zero byte (sign fill of a non-negative fp16)
    const bool odd = r & 1;
    const uint32_t selA0 = odd ? 0x5499u : 0x9910u, selB0 = odd ? 0x1099u : 0x9954u;
    const uint32_t selA1 = odd ? 0x7699u : 0x9932u, selB1 = odd ? 0x3299u : 0x9976u;

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

        // ---- QK: rows = tokens r, r + 8; lane c owns coordinates 32c .. 32c+31
        const uint32_t* kA = reinterpret_cast<const uint32_t*>(sg.k + r * kRec) + 3 * c;
        const uint32_t* kB = reinterpret_cast<const uint32_t*>(sg.k + (r + 8) * kRec) + 3 * c;
        const uint32_t x0 = kA[0], x1 = kA[1], x2 = kA[2];
        const uint32_t y0 = kB[0], y1 = kB[1], y2 = kB[2];
        float acc[NT][NC][4];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int q = 0; q < NC; ++q) acc[j][q][0] = acc[j][q][1] = acc[j][q][2] = acc[j][q][3] = 0.f;
        unroll<8>([&](auto st_) {
            constexpr int st = decltype(st_)::value;
            uint32_t a0, a1, a2, a3;
            if constexpr (KLDS) {
                a0 = tab_lk(tab, kfield7<st>(x0, x1, x2), lane4);
                a1 = tab_lk(tab, kfield7<st>(y0, y1, y2), lane4);
                a2 = tab_lk(tab, kfield7<st + 8>(x0, x1, x2), lane4);
                a3 = tab_lk(tab, kfield7<st + 8>(y0, y1, y2), lane4);
            } else {
                const Win A = (st >> 2) == 0 ? make_win(x0, x1, 0) : make_win(x1, x2, 16);
                const Win B = (st >> 2) == 0 ? make_win(y0, y1, 0) : make_win(y1, y2, 16);
                uint32_t rl, rh, rl2, rh2;
                pattern<2 * (st & 3)>(A, B, pk, fm, rl, rh);
                pattern<2 * (st & 3) + 1>(A, B, pk, fm, rl2, rh2);
                a0 = __byte_perm(rl, rh, 0x6240);
                a1 = __byte_perm(rl, rh, 0x7351);
                a2 = __byte_perm(rl2, rh2, 0x6240);
                a3 = __byte_perm(rl2, rh2, 0x7351);
            }
#pragma unroll
            for (int j = 0; j < NT; ++j) mma16816(acc[j][st % NC], a0, a1, a2, a3, bq[j][st][0], bq[j][st][1]);
        });

        // ---- online softmax (log2 units); lane holds head 4j + c for tokens r, r + 8
        const float kn0 = ldnorm(sg.kn, r, a.norm_f16) * kinv, kn8 = ldnorm(sg.kn, r + 8, a.norm_f16) * kinv;
        const float vn0 = ldnorm(sg.vn, r, a.norm_f16), vn8 = ldnorm(sg.vn, r + 8, a.norm_f16);
        float mn[NT], cf[NT], p0[NT], p8[NT];
        bool same = true;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            float s0 = acc[j][0][0], s8 = acc[j][0][2];
#pragma unroll
            for (int q = 1; q < NC; ++q) {
                s0 += acc[j][q][0];
                s8 += acc[j][q][2];
            }
            s0 *= kn0;
            s8 *= kn8;
            if (nval < kTile) {   // partial last tile: tokens past the section take no weight
                if (r >= nval) s0 = -INFINITY;
                if (r + 8 >= nval) s8 = -INFINITY;
            }
            float mt = fmaxf(s0, s8);
            mt = fmaxf(mt, __shfl_xor_sync(TQ_FULL_MASK, mt, 4));
            mt = fmaxf(mt, __shfl_xor_sync(TQ_FULL_MASK, mt, 8));
            mt = fmaxf(mt, __shfl_xor_sync(TQ_FULL_MASK, mt, 16));
            // the exponent base moves only when the tile max exceeds it by more
            // than 4 (log2 units): p <= 16 otherwise, and rescales are rare
            mn[j] = mt > m_[j] + 4.f ? mt : m_[j];
            cf[j] = ex2(m_[j] - mn[j]);   // 0 on the first tile (m = -inf)
            p0[j] = ex2(s0 - mn[j]);
            p8[j] = ex2(s8 - mn[j]);
            same = same && mn[j] == m_[j];
        }
        if (!__all_sync(TQ_FULL_MASK, same)) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                l_[j] *= cf[j];
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    o[j][mt][0] *= cf[j]; o[j][mt][1] *= cf[j]; o[j][mt][2] *= cf[j]; o[j][mt][3] *= cf[j];
                }
            }
        }
        // PV operand B for k steps u = 0 (tokens 0..7) and 1 (8..15): slot s < 4
        // holds token 8u + 2s, slot s >= 4 token 8u + 2(s - 4) + 1
        uint32_t bp[NT][2][2];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            l_[j] += p0[j] + p8[j];
            m_[j] = mn[j];
            const uint32_t X = pack_h2(p0[j] * vn0, p8[j] * vn8);
            const uint32_t Y = __shfl_xor_sync(TQ_FULL_MASK, X, 4);
            bp[j][0][0] = movtrans(prmt(X, Y, selA0));
            bp[j][0][1] = movtrans(prmt(X, Y, selB0));
            bp[j][1][0] = movtrans(prmt(X, Y, selA1));
            bp[j][1][1] = movtrans(prmt(X, Y, selB1));
        }

        // ---- PV (coordinate-pair form): row r / r + 8 of m tile mt = pair
        // 8r + 2mt / 8r + 2mt + 1, i.e. fields 2mt / 2mt + 1 of the lane row's window
        unroll<2>([&](auto u_) {
            constexpr int u = decltype(u_)::value;
            const int ta = 8 * u + 2 * c;
            const uint32_t* va = reinterpret_cast<const uint32_t*>(sg.v + ta * kRec) + vw;
            const uint32_t* vb = reinterpret_cast<const uint32_t*>(sg.v + (ta + 1) * kRec) + vw;
            const uint32_t LA = __funnelshift_r(va[0], va[1], vsh), HA = va[1] >> vsh;
            const uint32_t LB = __funnelshift_r(vb[0], vb[1], vsh), HB = vb[1] >> vsh;
            unroll<4>([&](auto mt_) {
                constexpr int mt = decltype(mt_)::value;
                const uint32_t a0 = tab_lk(tab, vfield7<2 * mt>(LA, HA), lane4);
                const uint32_t a1 = tab_lk(tab, vfield7<2 * mt + 1>(LA, HA), lane4);
                const uint32_t a2 = tab_lk(tab, vfield7<2 * mt>(LB, HB), lane4);
                const uint32_t a3 = tab_lk(tab, vfield7<2 * mt + 1>(LB, HB), lane4);
#pragma unroll
                for (int j = 0; j < NT; ++j) mma16816(o[j][mt], a0, a1, a2, a3, bp[j][u][0], bp[j][u][1]);
            });
        });
        __syncwarp();
    }
    cp_async_wait<0>();

    // ---- per-warp state -> CTA state; lane (r, c) holds o~ of head 4j + c at
    // coordinates 16r .. 16r + 15
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int msk = 4; msk < 32; msk <<= 1) l_[j] += __shfl_xor_sync(TQ_FULL_MASK, l_[j], msk);
    __syncthreads();   // every warp is done with its ring before it is reused
    TcFinal& F = S.fin;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        if (r == 0) {
            F.wm[warp][4 * j + c] = m_[j];
            F.wl[warp][4 * j + c] = l_[j];
        }
        float4* dst = reinterpret_cast<float4*>(&F.wo[warp][4 * j + c][16 * r]);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) dst[mt] = make_float4(o[j][mt][0], o[j][mt][1], o[j][mt][2], o[j][mt][3]);
    }
    __syncthreads();
    float mm[EP], ll[EP];
#pragma unroll
    for (int g = 0; g < EP; ++g) {
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
        F.ot[g][tid] = ov * vinv;   // the value table carried the scale s_V
    }
    __syncthreads();
    epilogue<EP>(a, P, F.ot, mm, ll, &S.is_last, b, h, s);
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
    constexpr bool klds = TQ_TC_KEY_TABLE != 0;
    dim3 grid(splits, d->n_kv_heads, d->batch);
    if (d->group <= 1) decode_tc4<4, 1, klds><<<grid, kThreads, 0, stream>>>(a);
    else if (d->group <= 4) decode_tc4<4, 4, klds><<<grid, kThreads, 0, stream>>>(a);
    else decode_tc4<8, 8, klds><<<grid, kThreads, 0, stream>>>(a);
    return cudaPeekAtLastError();
}
