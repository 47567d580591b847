// Tensor-core decode attention on 3-bit packed codes (one 128-wide rotation
// segment: WHT128 or SO(4) o WHT128) for up to 8 query heads per KV head.
//
// [RotaryQuant] Key design 3 and [TQ-MNN] §3.3: the QK dot products and the V
// accumulation run in the rotated domain directly on the packed codes; q is
// rotated once, the output once.  [Block-GTQ]: dequantised fp16 operands with
// fp32 accumulation on tensor cores, key-axis split with log-sum-exp merge.
//
// Each warp streams its own 16-token tiles (cp.async ring) and runs, per group
// of four query heads,
//   QK:  S[16 tok x 8] = K~[16 tok x 128] . B_q[128 x 8]          (8 mma m16n8k16)
//   PV:  O[64 pairs x 8] += V~[64 pairs x 32] . B_p[32 x 8]       (8 mma m16n8k16)
// Column n of both products is head n/2 of the group: in QK the two columns of
// a head are equal, in PV they hold the even and odd coordinate of each
// coordinate pair (coordinate-pair form: a PV row is a coordinate pair, its k
// index a (token, parity) pair, and B_p[(t, j)][(g, j')] = p_g(t) n_V(t) [j == j']).
// Every operand register holds two fp16 codebook values of one token, read from
// a 64-entry table of code pairs in shared memory (one copy per lane, so the 32
// lanes of a warp never share a bank) indexed by 6 consecutive bits of the
// record.  The order in which a lane meets the coordinates is a fixed
// permutation; q~ and the output coordinates follow it.
//
// Work split.  With an explicit split count every CTA takes one section of one
// (batch, KV head) pair.  Otherwise (stream-K) one wave of CTAs, as many as fit
// on the GPU at once, divides all 16-token tiles of all pairs evenly in pair
// order: a CTA's range covers the end of one pair, whole pairs and the start of
// another; each piece is a segment with its own softmax state, published as a
// partial and merged by the last CTA to finish a pair.
#include <stddef.h>

#include <mutex>
#include <utility>

#include "tq_decode_common.cuh"

namespace {

// warps of a stream-K CTA (one CTA per SM) for up to four heads per KV head
#ifndef TQ_TC_SK_WARPS
#define TQ_TC_SK_WARPS 16
#endif
// section kernel: two tiles per softmax step (1) or one (0)
#ifndef TQ_TC_TWO_TILES
#define TQ_TC_TWO_TILES 0
#endif
// value operands through byte-permute lookups (1) or the shared-memory table (0)
#ifndef TQ_TC_V_PRMT
#define TQ_TC_V_PRMT 0
#endif

constexpr int kTile = 16;
#ifndef TQ_TC_STAGES
#define TQ_TC_STAGES 3
#endif
#ifndef TQ_TC_MIN_BLOCKS
#define TQ_TC_MIN_BLOCKS (TQ_TC_TWO_TILES ? 4 : 5)
#endif

constexpr int kStages = TQ_TC_STAGES;   // cp.async ring depth per warp
constexpr int kRec = 48;                // bytes of one 3-bit record
constexpr int kSkMaxGrid = 152 * 8;     // bound on stream-K CTAs (sizes the partial slots)
constexpr int kSkSegs = 8;              // segments handled per round of a stream-K CTA

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
    float mm[8], ll[8];
};

struct TcSmem {
    union {
        TcStage ring[4][4];   // 4 stages per warp: two tiles processed, two in flight
        TcFinal fin;
    };
    alignas(16) float qts[8][128];
    alignas(16) uint32_t tab[64 * 32];
    int is_last;
};

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

// predicated 16-byte copy (no branch)
__device__ __forceinline__ void cp_async16p(uint32_t dst, const void* src, bool pred) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %2, 0;\n @p cp.async.cg.shared.global [%0], [%1], 16;\n}\n" ::"r"(dst),
        "l"(src), "r"((int)pred));
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

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

// ---- code-pair table
//
// tab[e][lane] = fp16x2 (s c[e & 7], s c[e >> 3]) for the 64 values e of a 6-bit
// field (two consecutive 3-bit codes, the lower one in the low half); s is the
// host-chosen scale that makes s c round almost exactly to fp16.

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

// tiles of one (batch, KV head) pair for batch b (length clamped, flags raised when asked)
__device__ __forceinline__ int pair_tiles(const DecodeArgs& a, int b, bool report) {
    int L = a.seq_lens[b];
    int flags = 0;
    if (L > a.Tcap) { flags |= TQ_DEV_SEQ_OVER_CAPACITY; L = a.Tcap; }
    if (L > a.max_seq) { flags |= TQ_DEV_SEQ_OVER_MAX; L = a.max_seq; }
    if (L < 0) L = 0;
    if (report && flags && a.status) atomicOr(a.status, flags);
    return (L + kTile - 1) / kTile;
}

__device__ __forceinline__ int pair_len(const DecodeArgs& a, int b) {
    return min(max(a.seq_lens[b], 0), min(a.Tcap, a.max_seq));
}

// A segment: tiles [t_lo, t_hi) of pair (b, h) whose sequence has L tokens.  Its
// partial goes to slot `slot`; the pair's partials are slots [first, first + parts).
// `off`: position of its first tile within a stream-K round.
struct Seg {
    int b, h, L, t_lo, t_hi, slot, first, parts, off;
};

// ---- byte-permute route (integer pipe instead of shared memory)
//
// Two 8-byte pools hold the low and the high bytes of the fp16 codebook (scaled
// as the table).  In a 48-bit window of 16 codes, code pairs (PP[i], QQ[i]) sit
// at the same bit offset of two bytes three bytes apart; the same two bytes of a
// second token's window complete a selector of four 3-bit indices, and two PRMT
// lookups plus two byte merges give (A@PP, A@QQ) and (B@PP, B@QQ) as fp16x2.
__host__ __device__ constexpr int pp_of(int i) { return i < 2 ? i : i < 4 ? i + 1 : i < 6 ? i + 2 : i == 6 ? 2 : 5; }
__host__ __device__ constexpr int qq_of(int i) { return pp_of(i) + 8; }

struct Pools {
    uint32_t lo0, lo1, hi0, hi1;
};

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

// Five byte-offset views of a 48-bit window starting at bit `base` of (wa, wb).
struct Win {
    uint32_t b, f8, f16, s0, s8;
};

__device__ __forceinline__ Win make_win(uint32_t wa, uint32_t wb, uint32_t base) {
    Win w;
    w.b = __funnelshift_rc(wa, wb, base);         // window bytes 0-3
    w.f8 = __funnelshift_rc(wa, wb, base + 8);    // bytes 1-4
    w.f16 = __funnelshift_rc(wa, wb, base + 16);  // bytes 2-5
    w.s0 = __funnelshift_rc(wa, wb, base + 2);    // window >> 2: codes 2, 10 byte-aligned
    w.s8 = __funnelshift_rc(wa, wb, base + 10);   // window >> 10: codes 5, 13
    return w;
}

template <int V>
__device__ __forceinline__ uint32_t view(const Win& w) {
    return V == 0 ? w.b : V == 1 ? w.f8 : V == 2 ? w.f16 : V == 3 ? w.s0 : w.s8;
}

// pattern I of a window pair: X = (A@PP[I], A@QQ[I]), Y = (B@PP[I], B@QQ[I])
template <int I>
__device__ __forceinline__ void pattern(const Win& A, const Win& B, const Pools& pl, uint32_t fm, uint32_t& X,
                                        uint32_t& Y) {
    constexpr int V = I < 2 ? 0 : I < 4 ? 1 : I < 6 ? 2 : I == 6 ? 3 : 4;
    constexpr int O = I == 0 ? 0 : I == 1 ? 3 : I == 2 ? 1 : I == 3 ? 4 : I == 4 ? 2 : I == 5 ? 5 : I == 6 ? 4 : 5;
    const uint32_t H = __byte_perm(view<V>(A), view<V>(B), 0x7430);   // [A.bi, A.bj, B.bi, B.bj]
    const uint32_t t = (O ? __umulhi(H, 1u << (32 - O)) : H) & 0x07070707u;
    uint32_t sel;
    asm("mad.hi.u32 %0, %1, %2, %1;" : "=r"(sel) : "r"(t), "r"(fm));   // t + (t >> 12): nibbles (A@p, B@p, A@q, B@q)
    const uint32_t rl = __byte_perm(pl.lo0, pl.lo1, sel), rh = __byte_perm(pl.hi0, pl.hi1, sel);
    X = __byte_perm(rl, rh, 0x6240);
    Y = __byte_perm(rl, rh, 0x7351);
}

// ---- one 16-token tile of one warp

struct LaneCtx {
    uint32_t lane4;                       // 4 x lane: the lane's column of the code-pair table
    int r, c;                             // mma fragment row group and column pair
    int vw;                               // first word of the lane row's 48-bit value window
    uint32_t vsh;                         // its bit offset in that word
    uint32_t selA0, selB0, selA1, selB1;  // PRMT selectors building the PV operand B
    Pools pv;                             // value codebook byte pools (byte-permute route)
    uint32_t fm;                          // 1 << 20
};

__device__ __forceinline__ LaneCtx lane_ctx(const DecodeArgs& a) {
    LaneCtx lc;
    lc.pv = make_pools(a.params[0].v_cent[0], a.params[0].v_h_scale[0]);
    lc.fm = a.fold_mul;
    const int lane = threadIdx.x & 31;
    lc.lane4 = 4u * lane;
    lc.r = lane >> 2;
    lc.c = lane & 3;
    lc.vw = (3 * lc.r) >> 1;
    lc.vsh = (lc.r & 1) ? 16u : 0u;
    // bytes 0-3 = (x_r, x_r+8) of this lane, 4-7 = those of lane row r ^ 1;
    // nibble 9 gives a zero byte (sign fill of a non-negative fp16)
    const bool odd = lc.r & 1;
    lc.selA0 = odd ? 0x5499u : 0x9910u;
    lc.selB0 = odd ? 0x1099u : 0x9954u;
    lc.selA1 = odd ? 0x7699u : 0x9932u;
    lc.selB1 = odd ? 0x3299u : 0x9976u;
    return lc;
}

// Online-softmax state of one warp for NT groups of four heads; lane (r, c)
// holds head 4j + c: o~ at coordinates 16r .. 16r + 15 (unnormalised), the
// running max m (log2 units) and its part of the running sum l.
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

// QK operand B from q~ ([GPE][128] floats in shared memory): column r of n tile
// j is head 4j + r/2; k step st of lane c carries coordinates 32c + 2st, +1 (a0,
// a1) and 32c + 2(st + 8), +1 (a2, a3)
template <int NT>
__device__ __forceinline__ void load_bq(const float (*qts)[128], const LaneCtx& lc, uint32_t (&bq)[NT][8][2]) {
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const float* qh = qts[4 * j + (lc.r >> 1)];
#pragma unroll
        for (int st = 0; st < 8; ++st) {
            const int d0 = 32 * lc.c + 2 * st, d1 = 32 * lc.c + 2 * (st + 8);
            bq[j][st][0] = pack_h2(qh[d0], qh[d0 + 1]);
            bq[j][st][1] = pack_h2(qh[d1], qh[d1 + 1]);
        }
    }
}

// PV for one staged tile with operand B `bp` (k steps u = 0, 1).  Row r / r + 8
// of m tile mt is a coordinate pair of the lane row's 48-bit window: with the
// table, fields 2mt / 2mt + 1 (coordinates 16r + 4mt + {0, 1} / {2, 3}); with
// byte permutes, patterns 2mt / 2mt + 1 (coordinates 16r + PP, QQ of each).
template <int NT>
__device__ __forceinline__ void pv_tile(const TcStage& sg, const uint32_t (&bp)[NT][2][2], const uint32_t* tab,
                                        const LaneCtx& lc, WState<NT>& ws) {
    const int c = lc.c;
    unroll<2>([&](auto u_c) {
        constexpr int u = decltype(u_c)::value;
        const int ta = 8 * u + 2 * c;
        const uint32_t* va = reinterpret_cast<const uint32_t*>(sg.v + ta * kRec) + lc.vw;
        const uint32_t* vb = reinterpret_cast<const uint32_t*>(sg.v + (ta + 1) * kRec) + lc.vw;
        if constexpr (TQ_TC_V_PRMT) {
            const Win A = make_win(va[0], va[1], lc.vsh), B = make_win(vb[0], vb[1], lc.vsh);
            unroll<4>([&](auto mt_c) {
                constexpr int mt = decltype(mt_c)::value;
                uint32_t a0, a1, a2, a3;
                pattern<2 * mt>(A, B, lc.pv, lc.fm, a0, a2);
                pattern<2 * mt + 1>(A, B, lc.pv, lc.fm, a1, a3);
#pragma unroll
                for (int j = 0; j < NT; ++j) mma16816(ws.o[j][mt], a0, a1, a2, a3, bp[j][u][0], bp[j][u][1]);
            });
        } else {
            const uint32_t LA = __funnelshift_r(va[0], va[1], lc.vsh), HA = va[1] >> lc.vsh;
            const uint32_t LB = __funnelshift_r(vb[0], vb[1], lc.vsh), HB = vb[1] >> lc.vsh;
            unroll<4>([&](auto mt_c) {
                constexpr int mt = decltype(mt_c)::value;
                const uint32_t a0 = tab_lk(tab, vfield7<2 * mt>(LA, HA), lc.lane4);
                const uint32_t a1 = tab_lk(tab, vfield7<2 * mt + 1>(LA, HA), lc.lane4);
                const uint32_t a2 = tab_lk(tab, vfield7<2 * mt>(LB, HB), lc.lane4);
                const uint32_t a3 = tab_lk(tab, vfield7<2 * mt + 1>(LB, HB), lc.lane4);
#pragma unroll
                for (int j = 0; j < NT; ++j) mma16816(ws.o[j][mt], a0, a1, a2, a3, bp[j][u][0], bp[j][u][1]);
            });
        }
    });
}

// output coordinate (within the lane row's 16) of o[mt][q]
__device__ __forceinline__ constexpr int pv_coord(int mt, int q) {
    return TQ_TC_V_PRMT ? ((q & 1) ? qq_of(2 * mt + (q >> 1)) : pp_of(2 * mt + (q >> 1))) : 4 * mt + q;
}

// QK, online softmax and PV for one staged tile of `nval` valid tokens.
template <int NT>
__device__ __forceinline__ void tile_step(const TcStage& sg, int nval, const uint32_t (&bq)[NT][8][2],
                                          const uint32_t* tab, const LaneCtx& lc, float kinv, int norm_f16,
                                          WState<NT>& ws) {
    constexpr int NC = 4 / NT;   // independent QK accumulators per n tile
    const int r = lc.r, c = lc.c;
    const uint32_t lane4 = lc.lane4;

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
    unroll<8>([&](auto st_c) {
        constexpr int st = decltype(st_c)::value;
        const uint32_t a0 = tab_lk(tab, kfield7<st>(x0, x1, x2), lane4);
        const uint32_t a1 = tab_lk(tab, kfield7<st>(y0, y1, y2), lane4);
        const uint32_t a2 = tab_lk(tab, kfield7<st + 8>(x0, x1, x2), lane4);
        const uint32_t a3 = tab_lk(tab, kfield7<st + 8>(y0, y1, y2), lane4);
#pragma unroll
        for (int j = 0; j < NT; ++j) mma16816(acc[j][st % NC], a0, a1, a2, a3, bq[j][st][0], bq[j][st][1]);
    });

    // ---- online softmax (log2 units); lane holds head 4j + c for tokens r, r + 8
    const float kn0 = ldnorm(sg.kn, r, norm_f16) * kinv, kn8 = ldnorm(sg.kn, r + 8, norm_f16) * kinv;
    const float vn0 = ldnorm(sg.vn, r, norm_f16), vn8 = ldnorm(sg.vn, r + 8, norm_f16);
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
        if (nval < kTile) {   // ragged last tile: tokens past the end take no weight
            if (r >= nval) s0 = -INFINITY;
            if (r + 8 >= nval) s8 = -INFINITY;
        }
        float mt = fmaxf(s0, s8);
        mt = fmaxf(mt, __shfl_xor_sync(TQ_FULL_MASK, mt, 4));
        mt = fmaxf(mt, __shfl_xor_sync(TQ_FULL_MASK, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(TQ_FULL_MASK, mt, 16));
        // the exponent base moves only when the tile max exceeds it by more
        // than 4 (log2 units): p <= 16 otherwise, and rescales are rare
        mn[j] = mt > ws.m[j] + 4.f ? mt : ws.m[j];
        cf[j] = ex2(ws.m[j] - mn[j]);   // 0 on the first tile (m = -inf)
        p0[j] = ex2(s0 - mn[j]);
        p8[j] = ex2(s8 - mn[j]);
        same = same && mn[j] == ws.m[j];
    }
    (void)same;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        ws.l[j] *= cf[j];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            ws.o[j][mt][0] *= cf[j]; ws.o[j][mt][1] *= cf[j]; ws.o[j][mt][2] *= cf[j]; ws.o[j][mt][3] *= cf[j];
        }
    }
    // PV operand B for k steps u = 0 (tokens 0..7) and 1 (8..15): slot s < 4
    // holds token 8u + 2s, slot s >= 4 token 8u + 2(s - 4) + 1
    uint32_t bp[NT][2][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        ws.l[j] += p0[j] + p8[j];
        ws.m[j] = mn[j];
        const uint32_t X = pack_h2(p0[j] * vn0, p8[j] * vn8);
        const uint32_t Y = __shfl_xor_sync(TQ_FULL_MASK, X, 4);
        bp[j][0][0] = movtrans(prmt(X, Y, lc.selA0));
        bp[j][0][1] = movtrans(prmt(X, Y, lc.selB0));
        bp[j][1][0] = movtrans(prmt(X, Y, lc.selA1));
        bp[j][1][1] = movtrans(prmt(X, Y, lc.selB1));
    }

    pv_tile<NT>(sg, bp, tab, lc, ws);
}

// Two full tiles at once: the same products, one softmax step over their 32
// tokens (one max reduction, one rescale), and twice the independent work in
// flight for the warp.
template <int NT>
__device__ __forceinline__ void tile_step2(const TcStage& sa, const TcStage& sb, const uint32_t (&bq)[NT][8][2],
                                           const uint32_t* tab, const LaneCtx& lc, float kinv, int norm_f16,
                                           WState<NT>& ws) {
    constexpr int NC = 4 / NT;
    const int r = lc.r, c = lc.c;
    const uint32_t lane4 = lc.lane4;
    const TcStage* sg[2] = {&sa, &sb};

    // ---- QK for both tiles
    uint32_t x[2][3], y[2][3];
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) {
        const uint32_t* kA = reinterpret_cast<const uint32_t*>(sg[tt]->k + r * kRec) + 3 * c;
        const uint32_t* kB = reinterpret_cast<const uint32_t*>(sg[tt]->k + (r + 8) * kRec) + 3 * c;
        x[tt][0] = kA[0]; x[tt][1] = kA[1]; x[tt][2] = kA[2];
        y[tt][0] = kB[0]; y[tt][1] = kB[1]; y[tt][2] = kB[2];
    }
    float acc[2][NT][NC][4];
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int q = 0; q < NC; ++q) acc[tt][j][q][0] = acc[tt][j][q][1] = acc[tt][j][q][2] = acc[tt][j][q][3] = 0.f;
    unroll<8>([&](auto st_c) {
        constexpr int st = decltype(st_c)::value;
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
            const uint32_t a0 = tab_lk(tab, kfield7<st>(x[tt][0], x[tt][1], x[tt][2]), lane4);
            const uint32_t a1 = tab_lk(tab, kfield7<st>(y[tt][0], y[tt][1], y[tt][2]), lane4);
            const uint32_t a2 = tab_lk(tab, kfield7<st + 8>(x[tt][0], x[tt][1], x[tt][2]), lane4);
            const uint32_t a3 = tab_lk(tab, kfield7<st + 8>(y[tt][0], y[tt][1], y[tt][2]), lane4);
#pragma unroll
            for (int j = 0; j < NT; ++j)
                mma16816(acc[tt][j][st % NC], a0, a1, a2, a3, bq[j][st][0], bq[j][st][1]);
        }
    });

    // ---- one online-softmax step over both tiles (log2 units)
    float kn[2][2], vn[2][2];
#pragma unroll
    for (int tt = 0; tt < 2; ++tt) {
        kn[tt][0] = ldnorm(sg[tt]->kn, r, norm_f16) * kinv;
        kn[tt][1] = ldnorm(sg[tt]->kn, r + 8, norm_f16) * kinv;
        vn[tt][0] = ldnorm(sg[tt]->vn, r, norm_f16);
        vn[tt][1] = ldnorm(sg[tt]->vn, r + 8, norm_f16);
    }
    uint32_t bp[2][NT][2][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        float sc[2][2];
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
            float s0 = acc[tt][j][0][0], s8 = acc[tt][j][0][2];
#pragma unroll
            for (int q = 1; q < NC; ++q) {
                s0 += acc[tt][j][q][0];
                s8 += acc[tt][j][q][2];
            }
            sc[tt][0] = s0 * kn[tt][0];
            sc[tt][1] = s8 * kn[tt][1];
        }
        float mt = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        mt = fmaxf(mt, __shfl_xor_sync(TQ_FULL_MASK, mt, 4));
        mt = fmaxf(mt, __shfl_xor_sync(TQ_FULL_MASK, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(TQ_FULL_MASK, mt, 16));
        const float mn = mt > ws.m[j] + 4.f ? mt : ws.m[j];
        const float cf = ex2(ws.m[j] - mn);
        ws.m[j] = mn;
        float lsum = 0.f;
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
            const float p0 = ex2(sc[tt][0] - mn), p8 = ex2(sc[tt][1] - mn);
            lsum += p0 + p8;
            const uint32_t X = pack_h2(p0 * vn[tt][0], p8 * vn[tt][1]);
            const uint32_t Y = __shfl_xor_sync(TQ_FULL_MASK, X, 4);
            bp[tt][j][0][0] = movtrans(prmt(X, Y, lc.selA0));
            bp[tt][j][0][1] = movtrans(prmt(X, Y, lc.selB0));
            bp[tt][j][1][0] = movtrans(prmt(X, Y, lc.selA1));
            bp[tt][j][1][1] = movtrans(prmt(X, Y, lc.selB1));
        }
        ws.l[j] = fmaf(ws.l[j], cf, lsum);
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
            ws.o[j][m4][0] *= cf; ws.o[j][m4][1] *= cf; ws.o[j][m4][2] *= cf; ws.o[j][m4][3] *= cf;
        }
    }

    // ---- PV for both tiles
    uint32_t bpa[NT][2][2], bpb[NT][2][2];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            bpa[j][u][0] = bp[0][j][u][0]; bpa[j][u][1] = bp[0][j][u][1];
            bpb[j][u][0] = bp[1][j][u][0]; bpb[j][u][1] = bp[1][j][u][1];
        }
    pv_tile<NT>(sa, bpa, tab, lc, ws);
    pv_tile<NT>(sb, bpb, tab, lc, ws);
}

// A warp's state into its merge slot: wo[g][128], wm[g], wl[g] for its heads.
template <int NT>
__device__ __forceinline__ void warp_state_out(WState<NT>& ws, const LaneCtx& lc, float (*wo)[128], float* wm,
                                               float* wl) {
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int msk = 4; msk < 32; msk <<= 1) ws.l[j] += __shfl_xor_sync(TQ_FULL_MASK, ws.l[j], msk);
        if (lc.r == 0) {
            wm[4 * j + lc.c] = ws.m[j];
            wl[4 * j + lc.c] = ws.l[j];
        }
        float* dst = &wo[4 * j + lc.c][16 * lc.r];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[pv_coord(mt, q)] = ws.o[j][mt][q];
    }
}

// Merge NW warp states (wo[w][g][128] at stride `wstride` floats, wm/wl[w][8]) into
// ot[g][128] (scaled by vinv) and mm/ll[g]; NTHR threads.
template <int EP, int NTHR>
__device__ __forceinline__ void merge_warps(int nw, const float* wo, int wstride, const float (*wm)[8],
                                            const float (*wl)[8], float vinv, float (*ot)[128], float* mm, float* ll) {
    for (int i = threadIdx.x; i < EP * 128; i += NTHR) {
        const int g = i >> 7, d = i & 127;
        float M = -INFINITY;
        for (int w = 0; w < nw; ++w) M = fmaxf(M, wm[w][g]);
        float Lt = 0.f, ov = 0.f;
        for (int w = 0; w < nw; ++w) {
            const float wt = (M == -INFINITY || wm[w][g] == -INFINITY) ? 0.f : exp2f(wm[w][g] - M);
            Lt = fmaf(wt, wl[w][g], Lt);
            ov = fmaf(wt, wo[(size_t)w * wstride + g * 128 + d], ov);
        }
        ot[g][d] = ov * vinv;   // the value table carried the scale s_V
        if (d == 0) {
            mm[g] = M;
            ll[g] = Lt;
        }
    }
}

// Finish a segment: ot[g][c] holds its unnormalised o~, (mm[g], ll[g]) its
// softmax state (shared memory).  One part: normalise and write; else publish
// the partial and let the last CTA of the pair merge all of them.  NTHR threads.
template <int GP, int NTHR>
__device__ void finish_segment(const DecodeArgs& a, const tq_head_params& P, float (*ot)[128], const float* mm,
                               const float* ll, int* is_last, const Seg& sg) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int pair = sg.b * a.Hkv + sg.h;
    if (sg.parts > 1) {
        float* part = a.ws_part + (size_t)sg.slot * GP * kPartStride;
        for (int i = tid; i < GP * 128; i += NTHR) part[(i >> 7) * kPartStride + (i & 127)] = ot[i >> 7][i & 127];
        if (tid < GP) {
            part[tid * kPartStride + 128] = mm[tid];
            part[tid * kPartStride + 129] = ll[tid];
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const int ticket = atomicAdd(a.tickets + pair, 1);
            *is_last = ticket == sg.parts - 1;
        }
        __syncthreads();
        if (!*is_last) return;
        __threadfence();
        // log-sum-exp merge over the pair's parts  [Block-GTQ]
        merge_parts<GP, NTHR>(a.ws_part + (size_t)sg.first * GP * kPartStride, sg.parts, ot);
        if (tid == 0) a.tickets[pair] = 0;   // ready for the next call
        __syncthreads();
    } else {
        for (int i = tid; i < GP * 128; i += NTHR) {
            const int g = i >> 7;
            ot[g][i & 127] = ll[g] > 0.f ? ot[g][i & 127] / ll[g] : 0.f;
        }
        __syncthreads();
    }
    // o = R_V^T o~, once per query head  [RotaryQuant Key design 3, Kernel D]
    for (int g = warp; g < a.G; g += NTHR / 32) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = ot[g][4 * lane + i];
        tq::rotate_inverse(a.rot, P, v);
        float4* o4 = reinterpret_cast<float4*>(a.out + ((size_t)sg.b * a.Hq + (size_t)sg.h * a.G + g) * 128) + lane;
        *o4 = make_float4(v[0], v[1], v[2], v[3]);
    }
}

// code-pair table (keys and values share it: both are 3-bit codes of one
// 128-coordinate segment, so their codebooks and fp16 scales coincide)
template <int NTHR>
__device__ __forceinline__ void build_table(const DecodeArgs& a, uint32_t* tab) {
    const tq_head_params& P0 = a.params[0];
    const float sv = P0.v_h_scale[0];
    for (int i = threadIdx.x; i < 64 * 32; i += NTHR) {
        const int e = i >> 5;
        tab[i] = pack_h2(sv * P0.v_cent[0][e & 7], sv * P0.v_cent[0][e >> 3]);
    }
}

// q~ = R_K q of head g of pair (b, h) into dst[128] (log2 units); one warp
__device__ __forceinline__ void rotate_q(const DecodeArgs& a, const tq_head_params& P, int b, int h, int g,
                                         float* dst) {
    const int lane = threadIdx.x & 31;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (g < a.G) {
        const size_t elem = ((size_t)b * a.Hq + (size_t)h * a.G + g) * 128 + 4 * lane;
        tq::load4(a.q, elem, a.q_dtype, v);
        tq::rotate_forward(a.rot, P, v);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[4 * lane + i] = v[i] * (kLog2e * kInvSqrtD);
}

// Copy plan of one lane: chunk `lane` (and `lane + 32` for lanes < 16) of the
// 768-byte K and V tiles, one 16-byte chunk of a norm tile for lanes 0..7.
__device__ __forceinline__ void issue_tile(const DecodeArgs& a, uint32_t dst, int b, int h, int L, int t) {
    const int lane = threadIdx.x & 31;
    const int nb = a.norm_f16 ? 2 : 4;
    const size_t head_tok = ((size_t)b * a.Hkv + h) * a.Tcap;
    const uint8_t* gk = a.k_codes + head_tok * kRec + 16 * lane;
    const uint8_t* gv = a.v_codes + head_tok * kRec + 16 * lane;
    const int nch = lane & 3;
    const bool has_n = lane < 8 && 16 * nch < kTile * nb;
    const uint8_t* gn = static_cast<const uint8_t*>(lane < 4 ? a.k_norms : a.v_norms) + head_tok * nb + 16 * nch;
    const uint32_t on = (uint32_t)(lane < 4 ? offsetof(TcStage, kn) : offsetof(TcStage, vn)) + 16 * nch;
    const size_t co = (size_t)t * (kTile * kRec);
    const int rem = L - t * kTile;
    if (rem >= kTile) {
        cp_async16s(dst + offsetof(TcStage, k) + 16 * lane, gk + co, 16);
        cp_async16s(dst + offsetof(TcStage, v) + 16 * lane, gv + co, 16);
        cp_async16p(dst + offsetof(TcStage, k) + 512 + 16 * lane, gk + co + 512, lane < 16);
        cp_async16p(dst + offsetof(TcStage, v) + 512 + 16 * lane, gv + co + 512, lane < 16);
        cp_async16p(dst + on, gn + (size_t)t * kTile * nb, has_n);
    } else {   // ragged last tile of the sequence: zero-fill past its end
        const int cb = rem * kRec;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int ch = lane + 32 * k;
            if (ch < 48) {
                const int n = min(16, max(0, cb - 16 * ch));
                const size_t off = n ? co + 32 * 16 * k : 0;
                cp_async16s(dst + offsetof(TcStage, k) + 16 * ch, gk + off, n);
                cp_async16s(dst + offsetof(TcStage, v) + 16 * ch, gv + off, n);
            }
        }
        if (has_n) {
            const int n = min(16, max(0, rem * nb - 16 * nch));
            cp_async16s(dst + on, gn + (n ? (size_t)t * kTile * nb : 0), n);
        }
    }
}

// The lane's part of the copies of one pair's tiles, set up once per segment.
struct CopyPlan {
    const uint8_t* gk;   // this lane's 16-byte chunk of tile 0 of the keys
    const uint8_t* gv;
    const uint8_t* gn;   // its 16-byte chunk of norm tile 0 (lanes 0..7)
    uint32_t on;         // stage offset of that norm chunk
    int nb;              // bytes per norm
    bool has_n;
};

__device__ __forceinline__ CopyPlan copy_plan(const DecodeArgs& a, int b, int h) {
    const int lane = threadIdx.x & 31;
    CopyPlan cp;
    cp.nb = a.norm_f16 ? 2 : 4;
    const size_t head_tok = ((size_t)b * a.Hkv + h) * a.Tcap;
    cp.gk = a.k_codes + head_tok * kRec + 16 * lane;
    cp.gv = a.v_codes + head_tok * kRec + 16 * lane;
    const int nch = lane & 3;
    cp.has_n = lane < 8 && 16 * nch < kTile * cp.nb;
    cp.gn = static_cast<const uint8_t*>(lane < 4 ? a.k_norms : a.v_norms) + head_tok * cp.nb + 16 * nch;
    cp.on = (uint32_t)(lane < 4 ? offsetof(TcStage, kn) : offsetof(TcStage, vn)) + 16 * nch;
    return cp;
}

// Tile t (of a sequence of L tokens) into the stage at dst; full tiles take no branch.
__device__ __forceinline__ void issue_planned(const CopyPlan& cp, uint32_t dst, int L, int t) {
    const int lane = threadIdx.x & 31;
    const size_t co = (size_t)t * (kTile * kRec);
    const int rem = L - t * kTile;
    if (rem >= kTile) {
        cp_async16s(dst + offsetof(TcStage, k) + 16 * lane, cp.gk + co, 16);
        cp_async16s(dst + offsetof(TcStage, v) + 16 * lane, cp.gv + co, 16);
        cp_async16p(dst + offsetof(TcStage, k) + 512 + 16 * lane, cp.gk + co + 512, lane < 16);
        cp_async16p(dst + offsetof(TcStage, v) + 512 + 16 * lane, cp.gv + co + 512, lane < 16);
        cp_async16p(dst + cp.on, cp.gn + (size_t)t * kTile * cp.nb, cp.has_n);
    } else {   // ragged last tile of the sequence: zero-fill past its end
        const int cb = rem * kRec;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int ch = lane + 32 * k;
            if (ch < 48) {
                const int n = min(16, max(0, cb - 16 * ch));
                const size_t off = n ? co + 32 * 16 * k : 0;
                cp_async16s(dst + offsetof(TcStage, k) + 16 * ch, cp.gk + off, n);
                cp_async16s(dst + offsetof(TcStage, v) + 16 * ch, cp.gv + off, n);
            }
        }
        if (cp.has_n) {
            const int n = min(16, max(0, rem * cp.nb - 16 * (lane & 3)));
            cp_async16s(dst + cp.on, cp.gn + (n ? (size_t)t * kTile * cp.nb : 0), n);
        }
    }
}

// ---- explicit splits: one CTA of 4 warps per (section, KV head, batch); its
// warps take the section's tiles round-robin
template <int GPE, int EP>
__global__ void __launch_bounds__(kThreads, GPE <= 4 ? TQ_TC_MIN_BLOCKS : 3) decode_tc(DecodeArgs a) {
    constexpr int NT = GPE / 4;
    __shared__ TcSmem S;
    // launched as a programmatic dependent of the previous kernel in the stream:
    // nothing is read before that kernel has completed and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    build_table<kThreads>(a, S.tab);
    const int L = clamp_len(a, b);
    const int t0 = s * a.split_len;   // a multiple of the tile
    const int t1 = min(t0 + a.split_len, L);
    Seg sg;
    sg.b = b;
    sg.h = h;
    sg.L = L;
    sg.t_lo = t0 / kTile;
    sg.t_hi = t1 > t0 ? (t1 + kTile - 1) / kTile : sg.t_lo;
    sg.first = (b * a.Hkv + h) * a.n_splits;
    sg.slot = sg.first + s;
    sg.parts = a.n_splits;
    sg.off = 0;
    const tq_head_params& P = a.params[h];
    const int nseg = sg.t_hi - sg.t_lo;
    const int nmine = nseg > warp ? (nseg - warp + 3) / 4 : 0;   // this warp: tiles t_lo + warp + 4i
    const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(S.ring[warp]);
    constexpr uint32_t kStageBytes = (uint32_t)sizeof(TcStage);
    auto tile_of = [&](int i) { return sg.t_lo + warp + 4 * i; };
    const CopyPlan cpl = copy_plan(a, b, h);
    constexpr int kAhead = TQ_TC_TWO_TILES ? 2 : 3;   // tiles in flight beyond those being processed
#pragma unroll
    for (int k = 0; k < kAhead; ++k) {   // start the stream before the q rotation
        if (k < nmine) issue_planned(cpl, ring_s + k * kStageBytes, L, tile_of(k));
        cp_async_commit();
    }
    for (int g = warp; g < GPE; g += 4) rotate_q(a, P, b, h, g, S.qts[g]);
    const float kinv = 1.0f / P.k_h_scale[0], vinv = 1.0f / P.v_h_scale[0];
    __syncthreads();
    const LaneCtx lc = lane_ctx(a);
    uint32_t bq[NT][8][2];
    load_bq<NT>(S.qts, lc, bq);
    WState<NT> ws;
    ws.reset();
    if constexpr (TQ_TC_TWO_TILES) {
        for (int i = 0; i < nmine; i += 2) {
#pragma unroll
            for (int k = 2; k < 4; ++k) {
                if (i + k < nmine) issue_planned(cpl, ring_s + ((i + k) % 4) * kStageBytes, L, tile_of(i + k));
                cp_async_commit();
            }
            cp_async_wait<2>();
            __syncwarp();
            const int nva = min(kTile, L - tile_of(i) * kTile);
            const TcStage& sa = S.ring[warp][i % 4];
            if (i + 1 < nmine) {
                const int nvb = min(kTile, L - tile_of(i + 1) * kTile);
                const TcStage& sb = S.ring[warp][(i + 1) % 4];
                if (nva == kTile && nvb == kTile) {
                    tile_step2<NT>(sa, sb, bq, S.tab, lc, kinv, a.norm_f16, ws);
                } else {
                    tile_step<NT>(sa, nva, bq, S.tab, lc, kinv, a.norm_f16, ws);
                    tile_step<NT>(sb, nvb, bq, S.tab, lc, kinv, a.norm_f16, ws);
                }
            } else {
                tile_step<NT>(sa, nva, bq, S.tab, lc, kinv, a.norm_f16, ws);
            }
            __syncwarp();
        }
    } else {
        for (int i = 0; i < nmine; ++i) {
            if (i + 3 < nmine) issue_planned(cpl, ring_s + ((i + 3) % 4) * kStageBytes, L, tile_of(i + 3));
            cp_async_commit();
            cp_async_wait<3>();
            __syncwarp();
            tile_step<NT>(S.ring[warp][i % 4], min(kTile, L - tile_of(i) * kTile), bq, S.tab, lc, kinv, a.norm_f16,
                          ws);
            __syncwarp();
        }
    }
    cp_async_wait<0>();
    __syncthreads();   // every warp is done with its ring before it is reused
    TcFinal& F = S.fin;
    warp_state_out<NT>(ws, lc, F.wo[warp], F.wm[warp], F.wl[warp]);
    __syncthreads();
    merge_warps<EP, kThreads>(4, &F.wo[0][0][0], 8 * 128, F.wm, F.wl, vinv, F.ot, F.mm, F.ll);
    __syncthreads();
    finish_segment<EP, kThreads>(a, P, F.ot, F.mm, F.ll, &S.is_last, sg);
}

// ---- stream-K: one persistent CTA of NW warps per SM
//
// The CTA's warps claim the tiles of its range one at a time, in order, so that
// a warp that runs ahead takes more of them; at the end of a segment the CTA
// merges its warps' states (the ring keeps streaming the next segment's tiles).
template <int GPE>
constexpr int sk_warps() { return GPE <= 4 ? TQ_TC_SK_WARPS : 8; }

template <int GPE>
struct SkSmem {
    static constexpr int NW = sk_warps<GPE>();
    TcStage ring[NW][kStages];
    float wo[NW][GPE][128];
    float wm[NW][8];
    float wl[NW][8];
    float ot[8][128];
    float mm[8], ll[8];
    float qts[kSkSegs][GPE][128];
    uint32_t tab[64 * 32];
    Seg seg[kSkSegs + 1];
    long long scan[NW];
    long long b_base, next_pos, cur_base;
    int b_first, cur_b, nseg, round_tiles, claim, is_last;
};

template <int GPE>
constexpr size_t sk_smem_bytes() { return sizeof(SkSmem<GPE>); }

template <int GPE, int EP>
__global__ void __launch_bounds__(sk_warps<GPE>() * 32, 1) decode_sk(DecodeArgs a) {
    constexpr int NT = GPE / 4;
    constexpr int NW = sk_warps<GPE>();
    constexpr int NTHR = NW * 32;
    extern __shared__ __align__(128) unsigned char sk_raw[];
    SkSmem<GPE>& S = *reinterpret_cast<SkSmem<GPE>*>(sk_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    build_table<NTHR>(a, S.tab);

    // ---- the CTA's range of tile positions: all tiles of all pairs in pair order
    const int per = (a.B + NTHR - 1) / NTHR;   // batches summed by each thread, in order
    const int bt0 = min(a.B, tid * per), bt1 = min(a.B, bt0 + per);
    long long loc = 0;
    for (int bb = bt0; bb < bt1; ++bb) loc += pair_tiles(a, bb, blockIdx.x == 0);
    long long inc = loc;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const long long y = __shfl_up_sync(TQ_FULL_MASK, inc, d);
        if (lane >= d) inc += y;
    }
    if (lane == 31) S.scan[warp] = inc;
    if (tid == 0) S.b_first = -1;
    __syncthreads();
    long long before = 0, total = 0;
    for (int w = 0; w < NW; ++w) {
        before += w < warp ? S.scan[w] : 0;
        total += S.scan[w];
    }
    const long long pre = before + inc - loc;   // tiles per head of batches < bt0
    const long long tiles_all = total * a.Hkv;
    const long long W = (tiles_all + gridDim.x - 1) / gridDim.x;
    const long long lo = (long long)blockIdx.x * W, hi = min(lo + W, tiles_all);
    if (lo < hi && (long long)a.Hkv * pre <= lo && lo < (long long)a.Hkv * (pre + loc)) {
        long long p = (long long)a.Hkv * pre;
        for (int bb = bt0; bb < bt1; ++bb) {
            const long long n = (long long)a.Hkv * pair_tiles(a, bb, false);
            if (lo < p + n) { S.b_first = bb; S.b_base = p; break; }
            p += n;
        }
    }
    // batches with no tokens get zero output (no tile of theirs exists)
    for (int bb = blockIdx.x; bb < a.B; bb += gridDim.x) {
        if (pair_len(a, bb) == 0) {
            float* ob = a.out + (size_t)bb * a.Hq * 128;
            for (int i = tid; i < a.Hq * 128; i += NTHR) ob[i] = 0.f;
        }
    }
    __syncthreads();
    if (lo >= hi || S.b_first < 0) return;
    if (tid == 0) {
        S.next_pos = lo;
        S.cur_b = S.b_first;
        S.cur_base = S.b_base;
    }
    const LaneCtx lc = lane_ctx(a);
    const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(S.ring[warp]);
    constexpr uint32_t kStageBytes = (uint32_t)sizeof(TcStage);

    for (;;) {
        // ---- next round: up to kSkSegs segments from next_pos (thread 0)
        __syncthreads();
        if (tid == 0) {
            long long p = S.next_pos, base = S.cur_base;
            int b = S.cur_b, n = 0, off = 0;
            while (p < hi && n < kSkSegs && b < a.B) {
                const int L = pair_len(a, b);
                const int nt = (L + kTile - 1) / kTile;
                if (nt == 0 || p >= base + (long long)a.Hkv * nt) {
                    base += (long long)a.Hkv * nt;
                    ++b;
                    continue;
                }
                const long long rel = p - base;
                const int h = (int)(rel / nt);
                const int t = (int)(rel - (long long)h * nt);
                const long long pstart = base + (long long)h * nt;
                const int take = (int)min((long long)(nt - t), hi - p);
                const long long fc = pstart / W, lc_ = (pstart + nt - 1) / W;
                const int pair = b * a.Hkv + h;
                Seg& sg = S.seg[n];
                sg.b = b;
                sg.h = h;
                sg.L = L;
                sg.t_lo = t;
                sg.t_hi = t + take;
                sg.first = (int)fc + pair;   // slot of CTA c for pair p: c + p (unique along the tile order)
                sg.slot = (int)blockIdx.x + pair;
                sg.parts = (int)(lc_ - fc + 1);
                sg.off = off;
                off += take;
                p += take;
                ++n;
            }
            S.seg[n].off = off;
            S.nseg = n;
            S.round_tiles = off;
            S.claim = 0;
            S.next_pos = p;
            S.cur_b = b;
            S.cur_base = base;
        }
        __syncthreads();
        const int nseg = S.nseg, round_tiles = S.round_tiles;
        if (nseg == 0) break;
        // q~ of every segment's heads
        for (int i = warp; i < nseg * GPE; i += NW) {
            const Seg& sg = S.seg[i / GPE];
            rotate_q(a, a.params[sg.h], sg.b, sg.h, i % GPE, S.qts[i / GPE][i % GPE]);
        }

        // ---- claims: each warp takes the round's tiles one at a time in order;
        // claim n of a warp goes to ring stage n % kStages
        int q[kStages];   // claimed positions, oldest first (-1: none)
        int nclaim = 0;
        auto claim = [&]() -> int {
            int g = 0;
            if (lane == 0) g = atomicAdd(&S.claim, 1);
            g = __shfl_sync(TQ_FULL_MASK, g, 0);
            if (g >= round_tiles) g = -1;
            if (g >= 0) {
                int k = 0;
                while (k + 1 < nseg && S.seg[k + 1].off <= g) ++k;
                const Seg& sg = S.seg[k];
                issue_tile(a, ring_s + (nclaim % kStages) * kStageBytes, sg.b, sg.h, sg.L, sg.t_lo + g - sg.off);
            }
            ++nclaim;
            cp_async_commit();
            return g;
        };
        __syncthreads();   // q~ ready; claim counter reset seen by all
#pragma unroll
        for (int k = 0; k < kStages - 1; ++k) q[k] = claim();
        int head = 0;      // ring stage of q[0]

        for (int k = 0; k < nseg; ++k) {
            const Seg sg = S.seg[k];
            const int end = S.seg[k + 1].off;
            const tq_head_params& P = a.params[sg.h];
            const float kinv = 1.0f / P.k_h_scale[0], vinv = 1.0f / P.v_h_scale[0];
            uint32_t bq[NT][8][2];
            load_bq<NT>(S.qts[k], lc, bq);
            WState<NT> ws;
            ws.reset();
            while (q[0] >= 0 && q[0] < end) {
                q[kStages - 1] = claim();
                cp_async_wait<kStages - 1>();
                __syncwarp();
                const int t = sg.t_lo + q[0] - sg.off;
                const int nval = min(kTile, sg.L - t * kTile);
                tile_step<NT>(S.ring[warp][head], nval, bq, S.tab, lc, kinv, a.norm_f16, ws);
#pragma unroll
                for (int i = 0; i + 1 < kStages; ++i) q[i] = q[i + 1];
                head = head + 1 == kStages ? 0 : head + 1;
                __syncwarp();
            }
            warp_state_out<NT>(ws, lc, S.wo[warp], S.wm[warp], S.wl[warp]);
            __syncthreads();
            merge_warps<EP, NTHR>(NW, &S.wo[0][0][0], GPE * 128, S.wm, S.wl, vinv, S.ot, S.mm, S.ll);
            __syncthreads();
            finish_segment<EP, NTHR>(a, P, S.ot, S.mm, S.ll, &S.is_last, sg);
            __syncthreads();
        }
        cp_async_wait<0>();
    }
}

// occupancy of the stream-K kernels (CTAs per SM x SMs), looked up once per device
template <int GPE, int EP>
int sk_capacity(int dev) {
    const size_t smem = sk_smem_bytes<GPE>();
    if (cudaFuncSetAttribute(decode_sk<GPE, EP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_sk<GPE, EP>, sk_warps<GPE>() * 32, smem) !=
            cudaSuccess ||
        n < 1)
        return 0;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) return 0;
    return n * sms;
}

int sk_grid_cap(int group) {
    static std::mutex mu;
    static int cache[64][3];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const int which = group <= 1 ? 0 : group <= 4 ? 1 : 2;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev][which]) {
        const int v = which == 0 ? sk_capacity<4, 1>(dev) : which == 1 ? sk_capacity<4, 4>(dev) : sk_capacity<8, 8>(dev);
        if (v <= 0) return 0;
        cache[dev][which] = v;
    }
    return cache[dev][which];
}

}  // namespace

bool tq_decode_tc_supported(const tq_cache_desc* d) {
    if (d->k_mixed || d->rot == TQ_ROT_WHT32) return false;
    if (d->k_bits != 3 || d->v_bits != 3 || d->group > 8) return false;
    // tile starts of the norm arrays must be 16-byte aligned
    return ((int64_t)d->t_capacity * d->norm_bytes) % 16 == 0;
}

int tq_decode_tc_split_align() { return kTile; }

int tq_decode_tc_sk_slots(const tq_cache_desc* d) { return kSkMaxGrid + d->batch * d->n_kv_heads; }

int tq_decode_tc_sk_grid(const tq_cache_desc* d, int max_seq_len) {
    const int cap = sk_grid_cap(d->group);
    if (cap <= 0) return 0;
    // at least 64 tiles (4 per warp) per CTA on average
    const long long tiles = (long long)d->batch * d->n_kv_heads * ((max_seq_len + kTile - 1) / kTile);
    long long g = (tiles + 63) / 64;
    if (g > cap) g = cap;
    if (g > kSkMaxGrid) g = kSkMaxGrid;
    return g < 1 ? 1 : (int)g;
}

cudaError_t tq_decode_tc_launch(const tq_cache_desc* d, const tq::DecodeArgs& a, int splits, int sk_grid,
                                cudaStream_t stream) {
    if (sk_grid > 0) {
        if (d->group <= 1) decode_sk<4, 1><<<sk_grid, sk_warps<4>() * 32, sk_smem_bytes<4>(), stream>>>(a);
        else if (d->group <= 4) decode_sk<4, 4><<<sk_grid, sk_warps<4>() * 32, sk_smem_bytes<4>(), stream>>>(a);
        else decode_sk<8, 8><<<sk_grid, sk_warps<8>() * 32, sk_smem_bytes<8>(), stream>>>(a);
        return cudaPeekAtLastError();
    }
    // programmatic dependent launch: the CTAs are placed while the previous kernel
    // (typically the token append) finishes, and wait for it on the device
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(splits, d->n_kv_heads, d->batch);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (d->group <= 1) return cudaLaunchKernelEx(&cfg, decode_tc<4, 1>, a);
    if (d->group <= 4) return cudaLaunchKernelEx(&cfg, decode_tc<4, 4>, a);
    return cudaLaunchKernelEx(&cfg, decode_tc<8, 8>, a);
}
