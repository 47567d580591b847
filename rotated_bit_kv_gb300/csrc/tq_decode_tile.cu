// Tensor-core decode attention on the 16-token tile layout (tq_tile.cuh): 3- or
// 4-bit codes, one 128-wide rotation segment (WHT128, SO(4) o WHT128) or four
// 32-wide blocks with a norm each (WHT32), or mixed-rate keys (up to four
// same-width groups with a norm each) over uniform values; up to 8 query heads
// per KV head.
//
// [RotaryQuant] Key design 3 and [TQ-MNN] §3.3: the QK dot products and the V
// accumulation run in the rotated domain directly on the packed codes; q is
// rotated once, the output once.  [Block-GTQ]: dequantised fp16 operands with
// fp32 accumulation on tensor cores; key-axis split with log-sum-exp merge.
//
// Each warp takes whole tiles.  A lane loads its 48 (3-bit) or 64 (4-bit) bytes
// of a tile's keys and values with two coalesced global loads each, straight into
// registers, and turns every byte of them into an mma operand register with one
// byte permute (the byte, placed above the lane's column, is the address) and one
// shared-memory load from a table of code pairs: row e of the table holds, in
// every lane's column, the fp16 pair (s c[lo(e)], s c[hi(e)]) of the field in
// byte e, so the 32 lanes of a warp never share a bank.  Per group of four query
// heads and per tile:
//   QK:  S[16 tok x 8] = K~[16 x 128] . B_q[128 x 8]          (8 mma m16n8k16)
//   PV:  O[64 pairs x 8] += V~[64 pairs x 32] . B_p[32 x 8]    (8 mma m16n8k16)
// In QK column 2g of B_q holds head g's rotated query rounded to fp16 and column
// 2g + 1 its rounding error, so that their sum carries the query to about 2^-22;
// for the WHT32 format each 32-wide block accumulates in its own chain, which the
// block's norm weighs.
// In PV a row is a coordinate pair, a k index a (token, parity) pair and
// B_p[(t, j)][(g, j')] = p_g(t) n_V(t) [j == j'], so that every operand register is
// one field of one token for keys and values alike.
//
// Work split (stream-K): all tiles of all (batch, KV head) pairs, in pair order,
// are divided evenly over a grid of persistent CTAs; a CTA's range is a sequence
// of pieces of pairs.  The CTA's warps take a piece's tiles round-robin, merge
// their softmax states in shared memory, and publish the piece's (m, l, o~); the
// last CTA to finish a pair merges its pieces by log-sum-exp and applies R_V^T.
#include <stddef.h>

#include <mutex>
#include <type_traits>
#include <utility>

#include "tq_decode_common.cuh"
#include "tq_mma.cuh"
#include "tq_tile.cuh"

namespace {

using tqtile::kTok;

#ifndef TQ_TILE_WARPS
#define TQ_TILE_WARPS 8
#endif
constexpr int kNW = TQ_TILE_WARPS;       // warps per CTA
constexpr int kNThr = kNW * 32;
constexpr int kMaxGrid = 152 * 8;        // bound on CTAs (sizes the partial slots)
// The code-pair table is the first member of the dynamic shared memory, which
// starts after the 1 KB the CUDA runtime reserves per block: its shared address
// is this constant, folded into every lookup's immediate offset (the kernel
// checks it at entry).
constexpr uint32_t kTabShared = 1024;
#ifndef TQ_TILE_QKCH
#define TQ_TILE_QKCH 2   // QK accumulator chains of the one-norm formats (2 or 4)
#endif

template <int GPE, bool KMIX>
constexpr int pieces_per_round() { return (GPE <= 4 && !KMIX) ? 8 : 2; }

// A piece: tiles [t_lo, t_hi) of pair (b, h) whose sequence has L tokens.  Its
// partial goes to slot `slot`; the pair's partials are slots [first, first + parts).
struct Seg {
    int b, h, L, t_lo, t_hi, slot, first, parts;
};

template <int GPE, bool KMIX>
struct TileSmem {
    static constexpr int NP = pieces_per_round<GPE, KMIX>();
    static constexpr int NT = GPE / 4;
    uint32_t tab[256 * 64];      // row e: 32 lane columns of table X, then 32 of table Y
    // mixed-rate keys: the key tables (KX: the 1..3-bit groups, KY: the 4-bit
    // group), 64 KB above the value tables; the QK operand B of each (k step,
    // group) of the current piece; the groups each k step touches (bit 4 st + s)
    uint32_t ktab[KMIX ? 256 * 64 : 1];
    std::conditional_t<KMIX, uint2[1][8][4][NT][32], uint2[1]> bm;
    uint32_t kmask[1];
    alignas(16) float qts[NP][GPE][128];     // rotated queries of the round's pieces (log2 units)
    alignas(16) float wo[kNW][GPE][128];     // warp states (float2 stores)
    float wm[kNW][8], wl[kNW][8];
    alignas(16) float ot[8][128];
    float mm[8], ll[8];
    Seg seg[NP + 1];
    long long scan[kNW];
    long long b_base, next_pos, cur_base;
    int b_first, cur_b, nseg;
    int last[NP];                // this CTA published the last partial of piece k's pair
};

// the key tables sit 64 KB above the value tables (the lookups put the block in
// address byte 2); float2 / float4 accesses need the 16-byte alignment
using SmemMix1 = TileSmem<4, true>;
using SmemMix2 = TileSmem<8, true>;
using SmemUni1 = TileSmem<4, false>;
static_assert(offsetof(SmemMix1, ktab) == 65536 && offsetof(SmemMix2, ktab) == 65536,
              "key tables must follow the value tables");
static_assert(offsetof(SmemUni1, wo) % 16 == 0 && offsetof(SmemMix2, wo) % 16 == 0,
              "warp state rows must be 16-byte aligned");

// ---- code-pair table and lookups

// Table row e: columns 0..31 = X(e), 32..63 = Y(e), each value in all 32 columns.
// 3-bit: X(e) = (s c[e & 7], s c[(e >> 3) & 7]) (field in byte bits 0-5);
// Y(e) reads the field from byte bits 0-1 and 4-7 (the middle word of a group).
// 4-bit: X(e) = (s c[e & 15], s c[e >> 4]).  s: the codebook's fp16 scale.
template <int BITS>
__device__ __forceinline__ void build_table(const tq_head_params& P0, uint32_t* tab) {
    const float sc = P0.v_h_scale[0];
    const float* cb = P0.v_cent[0];
    for (int i = threadIdx.x; i < 256 * 16; i += kNThr) {
        const int e = i >> 4, part = i & 15;
        int lo, hi;
        if (BITS == 4) {
            lo = e & 15;
            hi = e >> 4;
        } else if (part < 8) {
            lo = e & 7;
            hi = (e >> 3) & 7;
        } else {
            const int f = (e & 3) | ((e >> 4) << 2);
            lo = f & 7;
            hi = f >> 3;
        }
        const uint32_t v = pack_h2(sc * cb[lo], sc * cb[hi]);
        reinterpret_cast<uint4*>(tab)[i] = make_uint4(v, v, v, v);
    }
}

// table word at byte offset `addr` of the table
__device__ __forceinline__ uint32_t lk(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1+1024];" : "=r"(v) : "r"(addr));
    return v;
}

// table word of byte K of w: the byte goes to bits 8-15, the lane's column
// offset (4 lane, + 128 for table Y) comes from byte 0 of `col` and the table
// block (0: values, 1: mixed-rate keys, 64 KB above) from byte 2
template <int K>
__device__ __forceinline__ uint32_t lkb(uint32_t w, uint32_t col) {
    return lk(prmt(w, col, 0x7604u | (K << 4)));
}

// Key tables of mixed-rate keys, for the head whose parameters are P.  In the
// tile layout a b-bit code c of the 1..3-bit groups is stored as c + 2^b, so the
// two nibbles of a byte tell its width: 2-3 (1 bit), 4-7 (2 bits), 8-15 (3
// bits).  Row e of KX holds (s_g c_g[lo], s_g c_g[hi]) for the group g both
// nibbles name; KY holds the pairs of the 4-bit group (codes stored as is).
__device__ __forceinline__ void build_ktable(const tq_head_params& P, uint32_t* ktab) {
    for (int i = threadIdx.x; i < 256 * 16; i += kNThr) {
        const int e = i >> 4, part = i & 15;
        const int lo = e & 15, hi = e >> 4;
        uint32_t v = 0u;
        if (part >= 8) {
            v = pack_h2(P.k_h_scale[3] * P.k_cent[3][lo], P.k_h_scale[3] * P.k_cent[3][hi]);
        } else {
            const int g = lo >= 8 ? 2 : lo >= 4 ? 1 : lo >= 2 ? 0 : -1;
            const int gh = hi >= 8 ? 2 : hi >= 4 ? 1 : hi >= 2 ? 0 : -1;
            if (g >= 0 && g == gh) {
                const int off = 2 << g;
                v = pack_h2(P.k_h_scale[g] * P.k_cent[g][lo - off], P.k_h_scale[g] * P.k_cent[g][hi - off]);
            }
        }
        reinterpret_cast<uint4*>(ktab)[i] = make_uint4(v, v, v, v);
    }
}

// Table words of a three-word group of 3-bit codes: o[4 w + k] for byte k of word
// w, o[12 + g] for the field spread over byte lane g of the three words.
__device__ __forceinline__ void group3(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t cx, uint32_t cy,
                                       uint32_t (&o)[16]) {
    unroll<4>([&](auto k_c) {
        constexpr int k = decltype(k_c)::value;
        o[k] = lkb<k>(w0, cx);
        o[4 + k] = lkb<k>(w1, cy);
        o[8 + k] = lkb<k>(w2, cx);
    });
    const uint32_t m1 = 0x03030303u, m2 = 0x0F0F0F0Fu;
    const uint32_t s1 = ((w0 >> 6) & m1) | (w1 & ~m1);
    const uint32_t s2 = (s1 & m2) | ((w2 >> 2) & ~m2);
    unroll<4>([&](auto g_c) {
        constexpr int g = decltype(g_c)::value;
        o[12 + g] = lkb<g>(s2, cx);
    });
}

// ... of a four-word group of 4-bit codes: o[4 w + k] for byte k of word w.
__device__ __forceinline__ void group4(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3, uint32_t cx,
                                       uint32_t (&o)[16]) {
    unroll<4>([&](auto k_c) {
        constexpr int k = decltype(k_c)::value;
        o[k] = lkb<k>(w0, cx);
        o[4 + k] = lkb<k>(w1, cx);
        o[8 + k] = lkb<k>(w2, cx);
        o[12 + k] = lkb<k>(w3, cx);
    });
}

// ... of a four-word group of mixed-rate key codes, field f through column col[f]
__device__ __forceinline__ void group4m(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                        const uint32_t (&col)[16], uint32_t (&o)[16]) {
    unroll<4>([&](auto k_c) {
        constexpr int k = decltype(k_c)::value;
        o[k] = lkb<k>(w0, col[k]);
        o[4 + k] = lkb<k>(w1, col[4 + k]);
        o[8 + k] = lkb<k>(w2, col[8 + k]);
        o[12 + k] = lkb<k>(w3, col[12 + k]);
    });
}

// index into a value group's table words of field q of the low-half token (A) and
// of the high-half token (B)
template <int BITS>
__host__ __device__ constexpr int vA(int q) {
    return (BITS == 4 || q < 6) ? 4 * (q >> 1) + (q & 1) : 12 + (q - 6);
}
template <int BITS>
__host__ __device__ constexpr int vB(int q) {
    return (BITS == 4 || q < 6) ? 4 * (q >> 1) + 2 + (q & 1) : 14 + (q - 6);
}

// ---- per-lane context and tile registers

struct Lane {
    int r, c;
    uint32_t cx, cy;           // table column offsets (X, Y) in byte 0
    uint32_t sel_lo, sel_hi;   // P operand selectors (parity e = r & 1)
    uint32_t sw_a, sw_b;       // value-norm pair selectors for the A and B token of a pair
};

__device__ __forceinline__ Lane lane_ctx() {
    Lane l;
    const int lane = threadIdx.x & 31;
    l.r = lane >> 2;
    l.c = lane & 3;
    l.cx = 4u * lane;
    l.cy = 4u * lane + 128u;
    const bool e = l.r & 1;
    // (x, 0) for parity 0, (0, x) for parity 1, x = low / high half of the source
    l.sel_lo = e ? 0x1044u : 0x4410u;
    l.sel_hi = e ? 0x3244u : 0x4432u;
    l.sw_a = e ? 0x1032u : 0x3210u;
    l.sw_b = e ? 0x3210u : 0x1032u;
    return l;
}

// A lane's part of one tile: key words and norms (KRegs), value words and norms
// (VRegs); loaded separately so that a warp can keep two tiles in flight in two
// register sets.
template <int BITS, int NSEG>
struct KRegs {
    static constexpr int W = tqtile::group_words(BITS);
    uint32_t k[2 * W];
    uint32_t kn[NSEG == 1 ? 2 : 4];   // one slot: (n_r, n_r+8) as fp16 pair or two fp32
};
template <int BITS, int NSEG>
struct VRegs {
    static constexpr int W = tqtile::group_words(BITS);
    uint32_t v[2 * W];
    uint32_t vn[NSEG == 1 ? 2 : 8];
};

// Base pointers of one (batch, KV head) pair.
struct PairPtr {
    const uint8_t* k;
    const uint8_t* v;
    const uint8_t* kn;
    const uint8_t* vn;
};

// KB / KN: key code bits (4 for the nibble containers of mixed-rate keys) and
// key norm slots; VB / VN: the same for the values.
template <int KB, int KN, int VB, int VN>
__device__ __forceinline__ PairPtr pair_ptr(const DecodeArgs& a, int b, int h) {
    const size_t pair = (size_t)b * a.Hkv + h;
    const size_t tiles = (size_t)(a.Tcap / kTok);   // Tcap here is the allocated (tile-rounded) length
    const int nb = a.norm_f16 ? 2 : 4;
    PairPtr p;
    p.k = a.k_codes + pair * tiles * tqtile::tile_bytes(KB);
    p.v = a.v_codes + pair * tiles * tqtile::tile_bytes(VB);
    p.kn = static_cast<const uint8_t*>(a.k_norms) + pair * tiles * kTok * KN * nb;
    p.vn = static_cast<const uint8_t*>(a.v_norms) + pair * tiles * kTok * VN * nb;
    return p;
}

template <int BITS, int NSEG>
__device__ __forceinline__ void load_k(KRegs<BITS, NSEG>& td, const PairPtr& pp, int t, const Lane& ln, bool f16n) {
    const int lane = threadIdx.x & 31;
    const uint8_t* kt = pp.k + (size_t)t * tqtile::tile_bytes(BITS);
    const uint4 k0 = ldg_stream4(kt + 16 * lane);
    td.k[0] = k0.x; td.k[1] = k0.y; td.k[2] = k0.z; td.k[3] = k0.w;
    if constexpr (BITS == 3) {
        const uint2 k1 = ldg_stream2(kt + 512 + 8 * lane);
        td.k[4] = k1.x; td.k[5] = k1.y;
    } else {
        const uint4 k1 = ldg_stream4(kt + 512 + 16 * lane);
        td.k[4] = k1.x; td.k[5] = k1.y; td.k[6] = k1.z; td.k[7] = k1.w;
    }
    if constexpr (NSEG == 1) {
        if (f16n) {
            td.kn[0] = ldg_u32(pp.kn + ((size_t)t * kTok + 2 * ln.r) * 2);
            td.kn[1] = 0;
        } else {
            const uint2 kk = ldg_u64(pp.kn + ((size_t)t * kTok + 2 * ln.r) * 4);
            td.kn[0] = kk.x; td.kn[1] = kk.y;
        }
    } else {   // fp16 block norms of tokens r, r + 8
        const uint4 kk = ldg_u128(pp.kn + ((size_t)t * kTok * 4 + 8 * ln.r) * 2);
        td.kn[0] = kk.x; td.kn[1] = kk.y; td.kn[2] = kk.z; td.kn[3] = kk.w;
    }
}

template <int BITS, int NSEG>
__device__ __forceinline__ void load_v(VRegs<BITS, NSEG>& td, const PairPtr& pp, int t, const Lane& ln, bool f16n) {
    const int lane = threadIdx.x & 31;
    const uint8_t* vt = pp.v + (size_t)t * tqtile::tile_bytes(BITS);
    const uint4 v0 = ldg_stream4(vt + 16 * lane);
    td.v[0] = v0.x; td.v[1] = v0.y; td.v[2] = v0.z; td.v[3] = v0.w;
    if constexpr (BITS == 3) {
        const uint2 v1 = ldg_stream2(vt + 512 + 8 * lane);
        td.v[4] = v1.x; td.v[5] = v1.y;
    } else {
        const uint4 v1 = ldg_stream4(vt + 512 + 16 * lane);
        td.v[4] = v1.x; td.v[5] = v1.y; td.v[6] = v1.z; td.v[7] = v1.w;
    }
    if constexpr (NSEG == 1) {
        if (f16n) {
            td.vn[0] = ldg_u32(pp.vn + ((size_t)t * kTok + 2 * ln.r) * 2);
            td.vn[1] = 0;
        } else {
            const uint2 vv = ldg_u64(pp.vn + ((size_t)t * kTok + 2 * ln.r) * 4);
            td.vn[0] = vv.x; td.vn[1] = vv.y;
        }
    } else {   // fp16 block norms of tokens 2c, 2c+1, 2c+8, 2c+9
        const uint4 v0n = ldg_u128(pp.vn + ((size_t)t * kTok * 4 + 16 * ln.c) * 2);
        const uint4 v1n = ldg_u128(pp.vn + ((size_t)t * kTok * 4 + 16 * ln.c + 8) * 2);
        td.vn[0] = v0n.x; td.vn[1] = v0n.y; td.vn[2] = v0n.z; td.vn[3] = v0n.w;
        td.vn[4] = v1n.x; td.vn[5] = v1n.y; td.vn[6] = v1n.z; td.vn[7] = v1n.w;
    }
}

// The QK operand B of a lane (uniform-rate keys), in registers.
template <int NT>
struct BqT {
    uint32_t r[NT][8][2];
    __device__ __forceinline__ uint2 get(int j, int st) const { return make_uint2(r[j][st][0], r[j][st][1]); }
};

// QK operand B from q~ ([GPE][128] floats, log2 units) times kinv: lane (r, c), head
// 4j + r/2; k step st holds coordinates 16 st + 2c, +1 (b0) and 16 st + 2c + 8, +9
// (b1).  Column parity r & 1 carries the fp16 rounding of q~ (0) or its rounding
// error (1), so that the two columns add up to q~ to about 2^-22.
template <int NT>
__device__ __forceinline__ void load_bq(const float (*qts)[128], const Lane& ln, float kinv,
                                        uint32_t (&bq)[NT][8][2]) {
    const bool odd = ln.r & 1;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const float* qh = qts[4 * j + (ln.r >> 1)];
#pragma unroll
        for (int st = 0; st < 8; ++st) {
            const int d0 = 16 * st + 2 * ln.c, d1 = d0 + 8;
            bq[j][st][0] = pack_part(qh[d0] * kinv, qh[d0 + 1] * kinv, odd);
            bq[j][st][1] = pack_part(qh[d1] * kinv, qh[d1 + 1] * kinv, odd);
        }
    }
}

// QK of one tile: scores (log2 units) s0 / s8 of tokens r and r + 8 for head 4j + c.
template <int NT, int BITS, int NSEG>
__device__ __forceinline__ void qk_phase(const KRegs<BITS, NSEG>& kd, const Lane& ln, const BqT<NT>& bq,
                                         bool f16n, float (&s0)[NT], float (&s8)[NT]) {
    // ---- QK: rows = tokens r (kr) and r + 8 (k8); accumulator chains: k steps of
    // even / odd index (one norm) or one chain per 32-wide block (k steps 2b, 2b+1)
    constexpr int CH = NSEG == 1 ? TQ_TILE_QKCH : 4;
    float acc[NT][CH][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int q = 0; q < CH; ++q) acc[j][q][0] = acc[j][q][1] = acc[j][q][2] = acc[j][q][3] = 0.f;
    {
        uint32_t kr[16], k8[16];
        if constexpr (BITS == 3) {
            group3(kd.k[0], kd.k[1], kd.k[2], ln.cx, ln.cy, kr);
            group3(kd.k[3], kd.k[4], kd.k[5], ln.cx, ln.cy, k8);
        } else {
            group4(kd.k[0], kd.k[1], kd.k[2], kd.k[3], ln.cx, kr);
            group4(kd.k[4], kd.k[5], kd.k[6], kd.k[7], ln.cx, k8);
        }
#pragma unroll
        for (int st = 0; st < 8; ++st) {
            const int ch = NSEG == 1 ? (st & (CH - 1)) : (st >> 1);
#pragma unroll
            for (int j = 0; j < NT; ++j)
            {
                const uint2 b = bq.get(j, st);
                mma16816(acc[j][ch], kr[2 * st], k8[2 * st], kr[2 * st + 1], k8[2 * st + 1], b.x, b.y);
            }
        }
    }

    // ---- scores (log2 units) of tokens r and r + 8 for head 4j + c
    if constexpr (NSEG == 1) {
        const float kn0 = f16n ? h_lo(kd.kn[0]) : __uint_as_float(kd.kn[0]);
        const float kn8 = f16n ? h_hi(kd.kn[0]) : __uint_as_float(kd.kn[1]);
#pragma unroll
        for (int j = 0; j < NT; ++j) {   // both columns (rounded q~ and its remainder), every chain
            float a0 = acc[j][0][0] + acc[j][0][1], a8 = acc[j][0][2] + acc[j][0][3];
#pragma unroll
            for (int q = 1; q < CH; ++q) {
                a0 += acc[j][q][0] + acc[j][q][1];
                a8 += acc[j][q][2] + acc[j][q][3];
            }
            s0[j] = a0 * kn0;
            s8[j] = a8 * kn8;
        }
    } else {
        float n0[4], n8[4];
        n0[0] = h_lo(kd.kn[0]); n0[1] = h_hi(kd.kn[0]); n0[2] = h_lo(kd.kn[1]); n0[3] = h_hi(kd.kn[1]);
        n8[0] = h_lo(kd.kn[2]); n8[1] = h_hi(kd.kn[2]); n8[2] = h_lo(kd.kn[3]); n8[3] = h_hi(kd.kn[3]);
#pragma unroll
        for (int j = 0; j < NT; ++j) {   // per block: rounded q~ and its remainder, then the block's norm
            float a0 = n0[0] * (acc[j][0][0] + acc[j][0][1]), a8 = n8[0] * (acc[j][0][2] + acc[j][0][3]);
#pragma unroll
            for (int b = 1; b < 4; ++b) {
                a0 = fmaf(n0[b], acc[j][b][0] + acc[j][b][1], a0);
                a8 = fmaf(n8[b], acc[j][b][2] + acc[j][b][3], a8);
            }
            s0[j] = a0;
            s8[j] = a8;
        }
    }
}

// QK of one tile of mixed-rate keys.  Group s of the head (the 2^(s+1)-level
// codes) accumulates in chain s over the k steps it touches (bit 4 st + s of
// `mask`); the operand B of (k step st, group s) holds q~ on the group's
// coordinates over the group's table scale, zero elsewhere (bm: this lane's
// entry of [st][s][head group j] for the piece).  Each chain is weighed by the
// token's norm of its group [Block-GTQ, per-group norms].  colpack: the lane's
// key-table column per field (byte f & 3 of word f >> 2; + 128 for table KY).
template <int NT>
__device__ __forceinline__ void qk_phase_mix(const KRegs<4, 4>& kd, const uint32_t (&colpack)[4], const uint2* bm,
                                             uint32_t mask, float (&s0)[NT], float (&s8)[NT]) {
    float acc[NT][4][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[j][q][0] = acc[j][q][1] = acc[j][q][2] = acc[j][q][3] = 0.f;
    {
        uint32_t col[16];
        unroll<16>([&](auto f_c) {
            constexpr int f = decltype(f_c)::value;
            // byte f & 3 of the field's word, key-table block 1 in byte 2
            col[f] = prmt(colpack[f >> 2], 0x00010000u, 0x7640u | (f & 3));
        });
        uint32_t kr[16], k8[16];
        group4m(kd.k[0], kd.k[1], kd.k[2], kd.k[3], col, kr);
        group4m(kd.k[4], kd.k[5], kd.k[6], kd.k[7], col, k8);
        unroll<8>([&](auto st_c) {
            constexpr int st = decltype(st_c)::value;
            unroll<4>([&](auto g_c) {
                constexpr int g = decltype(g_c)::value;
                if (mask & (1u << (4 * st + g))) {
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const uint2 b = bm[((st * 4 + g) * NT + j) * 32];
                        mma16816(acc[j][g], kr[2 * st], k8[2 * st], kr[2 * st + 1], k8[2 * st + 1], b.x, b.y);
                    }
                }
            });
        });
    }
    float n0[4], n8[4];
    n0[0] = h_lo(kd.kn[0]); n0[1] = h_hi(kd.kn[0]); n0[2] = h_lo(kd.kn[1]); n0[3] = h_hi(kd.kn[1]);
    n8[0] = h_lo(kd.kn[2]); n8[1] = h_hi(kd.kn[2]); n8[2] = h_lo(kd.kn[3]); n8[3] = h_hi(kd.kn[3]);
#pragma unroll
    for (int j = 0; j < NT; ++j) {   // per group: rounded q~ and its remainder, then the group's norm
        float a0 = n0[0] * (acc[j][0][0] + acc[j][0][1]), a8 = n8[0] * (acc[j][0][2] + acc[j][0][3]);
#pragma unroll
        for (int g = 1; g < 4; ++g) {
            a0 = fmaf(n0[g], acc[j][g][0] + acc[j][g][1], a0);
            a8 = fmaf(n8[g], acc[j][g][2] + acc[j][g][3], a8);
        }
        s0[j] = a0;
        s8[j] = a8;
    }
}

// Online softmax and PV of one tile of `nval` valid tokens (past-the-end tokens of
// a short last tile take no weight), from its scores.
template <int NT, int BITS, int NSEG>
__device__ __forceinline__ void pv_phase(const VRegs<BITS, NSEG>& td, float (&s0)[NT], float (&s8)[NT], int nval,
                                         const Lane& ln, bool f16n, WState<NT>& ws) {
    const int r = ln.r;
    constexpr int W = tqtile::group_words(BITS);
    uint32_t vg[2][16];
    auto vlookups = [&](auto u_c) {
        constexpr int u = decltype(u_c)::value;
        if constexpr (BITS == 3) group3(td.v[W * u], td.v[W * u + 1], td.v[W * u + 2], ln.cx, ln.cy, vg[u]);
        else group4(td.v[W * u], td.v[W * u + 1], td.v[W * u + 2], td.v[W * u + 3], ln.cx, vg[u]);
    };
    const bool in0 = r < nval, in8 = r + 8 < nval;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        s0[j] = in0 ? s0[j] : -INFINITY;
        s8[j] = in8 ? s8[j] : -INFINITY;
    }

    // ---- online softmax (lazy base: p <= 16, rare rescales)
    tile_softmax<NT>(s0, s8, ws);

    // ---- P operand (k = token-parity pairs, columns = head-parity pairs)
    // After the transposes lane (r, c) holds, for head r/2 (+4j), tokens 2c, 2c+1
    // (T0) and 2c+8, 2c+9 (T1); k step u = 0 takes tokens 2c (b0) and 2c+1 (b1),
    // u = 1 tokens 2c+8 and 2c+9.
    uint32_t bp[NT][2][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        float p0 = ex2(s0[j] - ws.m[j]), p8 = ex2(s8[j] - ws.m[j]);
        ws.l[j] += p0 + p8;
        if constexpr (NSEG == 1) {
            float vn0 = f16n ? h_lo(td.vn[0]) : __uint_as_float(td.vn[0]);
            float vn8 = f16n ? h_hi(td.vn[0]) : __uint_as_float(td.vn[1]);
            vn0 = in0 ? vn0 : 0.f;   // past the end: zero weight even if the stored norm is not finite
            vn8 = in8 ? vn8 : 0.f;
            p0 *= vn0;
            p8 *= vn8;
        }
        p_operand(p0, p8, ln.sel_lo, ln.sel_hi, bp[j]);
    }

    // ---- PV: group u of the values holds tokens 2c + 8u (A) and 2c + 1 + 8u (B)
    unroll<2>([&](auto u_c) {
        constexpr int u = decltype(u_c)::value;
        vlookups(u_c);
        // four blocks: each m tile is one block; its value norms scale the P operand
        uint32_t wa[4] = {0u, 0u, 0u, 0u}, wb[4] = {0u, 0u, 0u, 0u};
        (void)wa;
        (void)wb;
        if constexpr (NSEG == 4) {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                uint32_t w = td.vn[4 * u + b];   // (n_b(2c + 8u), n_b(2c + 1 + 8u))
                const int ta = 2 * ln.c + 8 * u;
                w = (ta < nval ? (w & 0xFFFFu) : 0u) | (ta + 1 < nval ? (w & 0xFFFF0000u) : 0u);
                wa[b] = prmt(w, w, ln.sw_a);
                wb[b] = prmt(w, w, ln.sw_b);
            }
        }
        unroll<4>([&](auto mt_c) {
            constexpr int mt = decltype(mt_c)::value;
            const uint32_t a0 = vg[u][vA<BITS>(2 * mt)], a1 = vg[u][vA<BITS>(2 * mt + 1)];
            const uint32_t a2 = vg[u][vB<BITS>(2 * mt)], a3 = vg[u][vB<BITS>(2 * mt + 1)];
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                if constexpr (NSEG == 1) {
                    mma16816(ws.o[j][mt], a0, a1, a2, a3, bp[j][u][0], bp[j][u][1]);
                } else {
                    mma16816(ws.o[j][mt], a0, a1, a2, a3, hmul2(bp[j][u][0], wa[mt]), hmul2(bp[j][u][1], wb[mt]));
                }
            }
        });
    });
}

// A warp's state into its merge slot: wo[g][128], wm[g], wl[g] for its heads.
template <int NT>
__device__ __forceinline__ void warp_state_out(WState<NT>& ws, const Lane& ln, float (*wo)[128], float* wm,
                                               float* wl) {
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int msk = 4; msk < 32; msk <<= 1) ws.l[j] += __shfl_xor_sync(TQ_FULL_MASK, ws.l[j], msk);
        if (ln.r == 0) {
            wm[4 * j + ln.c] = ws.m[j];
            wl[4 * j + ln.c] = ws.l[j];
        }
        float* dst = wo[4 * j + ln.c];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            const int d = 32 * mt + 2 * ln.r;
            *reinterpret_cast<float2*>(dst + d) = make_float2(ws.o[j][mt][0], ws.o[j][mt][1]);
            *reinterpret_cast<float2*>(dst + d + 16) = make_float2(ws.o[j][mt][2], ws.o[j][mt][3]);
        }
    }
}

// Merge the kNW warp states into ot[g][128] (scaled by vinv) and mm/ll[g].
template <int EP, int GPE>
__device__ __forceinline__ void merge_warps(const float (*wo)[GPE][128], const float (*wm)[8], const float (*wl)[8],
                                            float vinv, float (*ot)[128], float* mm, float* ll) {
    for (int i = threadIdx.x; i < EP * 128; i += kNThr) {
        const int g = i >> 7, d = i & 127;
        float M = -INFINITY;
        for (int w = 0; w < kNW; ++w) M = fmaxf(M, wm[w][g]);
        float Lt = 0.f, ov = 0.f;
        for (int w = 0; w < kNW; ++w) {
            const float wt = (M == -INFINITY || wm[w][g] == -INFINITY) ? 0.f : exp2f(wm[w][g] - M);
            Lt = fmaf(wt, wl[w][g], Lt);
            ov = fmaf(wt, wo[w][g][d], ov);
        }
        ot[g][d] = ov * vinv;   // the table carried the scale s
        if (d == 0) {
            mm[g] = M;
            ll[g] = Lt;
        }
    }
}

// Log-sum-exp merge of `parts` published partials (rows [part t][head g] of
// kPartStride floats: o~[128], m, l) into ot[g][0..127], normalised  [Block-GTQ].
// The partials sit in L2, a round trip away, so the merge is one online sweep:
// thread (g, d4) takes four coordinates of head g and, per batch of MB parts,
// issues all of the batch's loads (m_t, l_t and its o~ quadruple) at once, then
// moves its running maximum M to the batch's and folds the batch in:
//   acc = 2^(M_old - M) acc + sum_t 2^(m_t - M) o~_t,  L likewise with l_t.
// Empty parts (m = -inf) weigh 0; a pair with no tokens gives 0.  The merged
// (M, L) of head g go to mo[g], lo[g] (shared).
template <int GP>
__device__ __forceinline__ void merge_pieces(const float* base, int parts, float (*ot)[128], float* mo, float* lo) {
    static_assert(GP * 32 <= kNThr, "one coordinate quadruple per thread");
    constexpr int MB = GP <= 4 ? 8 : 16;   // parts in flight (the 4-head kernels' register budget)
    const int tid = threadIdx.x, g = tid >> 5, d4 = tid & 31;
    if (g >= GP) return;
    const float* pr = base + (size_t)g * kPartStride;
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int t = 0; t < parts; t += MB) {
        float4 v[MB];
        float2 ml[MB];
#pragma unroll
        for (int u = 0; u < MB; ++u) {
            const float* row = pr + (size_t)(t + u) * GP * kPartStride;
            const bool in = t + u < parts;
            v[u] = in ? __ldcg(reinterpret_cast<const float4*>(row) + d4) : make_float4(0.f, 0.f, 0.f, 0.f);
            ml[u] = in ? __ldcg(reinterpret_cast<const float2*>(row + 128)) : make_float2(-INFINITY, 0.f);
        }
        float Mb = M;
#pragma unroll
        for (int u = 0; u < MB; ++u) Mb = fmaxf(Mb, ml[u].x);
        if (Mb == -INFINITY) continue;   // nothing but empty parts so far
        const float cf = M == -INFINITY ? 0.f : exp2f(M - Mb);
        L *= cf;
        acc.x *= cf; acc.y *= cf; acc.z *= cf; acc.w *= cf;
#pragma unroll
        for (int u = 0; u < MB; ++u) {
            const float w = ml[u].x == -INFINITY ? 0.f : exp2f(ml[u].x - Mb);
            L = fmaf(w, ml[u].y, L);
            acc.x = fmaf(w, v[u].x, acc.x);
            acc.y = fmaf(w, v[u].y, acc.y);
            acc.z = fmaf(w, v[u].z, acc.z);
            acc.w = fmaf(w, v[u].w, acc.w);
        }
        M = Mb;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    if (d4 == 0) {
        mo[g] = M;
        lo[g] = L;
    }
    ot[g][4 * d4] = acc.x * inv;
    ot[g][4 * d4 + 1] = acc.y * inv;
    ot[g][4 * d4 + 2] = acc.z * inv;
    ot[g][4 * d4 + 3] = acc.w * inv;
}

// o = R_V^T o~ for the pair's query heads from ot (normalised), into out
// [RotaryQuant Key design 3, Kernel D]; with a.lse, each head's log2-sum-exp
// m + log2 l from its softmax state (mm, ll)
__device__ __forceinline__ void store_out(const DecodeArgs& a, const tq_head_params& P, float (*ot)[128],
                                          const float* mm, const float* ll, const Seg& sg) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (a.lse && threadIdx.x < a.G)
        a.lse[(size_t)sg.b * a.Hq + (size_t)sg.h * a.G + threadIdx.x] =
            ll[threadIdx.x] > 0.f ? mm[threadIdx.x] + log2f(ll[threadIdx.x]) : -INFINITY;
    for (int g = warp; g < a.G; g += kNW) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = ot[g][4 * lane + i];
        tq::rotate_inverse(a.rot, P, v);
        float4* o4 = reinterpret_cast<float4*>(a.out + ((size_t)sg.b * a.Hq + (size_t)sg.h * a.G + g) * 128) + lane;
        *o4 = make_float4(v[0], v[1], v[2], v[3]);
    }
}

// Finish a piece: ot[g][c] holds its unnormalised o~, (mm[g], ll[g]) its softmax
// state (shared memory).  One part: normalise, rotate back and write.  Else
// publish the partial and take a ticket; *last tells whether this CTA's partial
// was the pair's last (its merge comes after the CTA's other pieces of the round).
template <int GP>
__device__ void finish_piece(const DecodeArgs& a, const tq_head_params& P, float (*ot)[128], const float* mm,
                             const float* ll, int* last, const Seg& sg) {
    const int tid = threadIdx.x;
    if (sg.parts > 1) {
        float* part = a.ws_part + (size_t)sg.slot * GP * kPartStride;
        for (int i = tid; i < GP * 128; i += kNThr) part[(i >> 7) * kPartStride + (i & 127)] = ot[i >> 7][i & 127];
        if (tid < GP) {
            part[tid * kPartStride + 128] = mm[tid];
            part[tid * kPartStride + 129] = ll[tid];
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const int ticket = atomicAdd(a.tickets + sg.b * a.Hkv + sg.h, 1);
            *last = ticket == sg.parts - 1;
        }
    } else {
        for (int i = tid; i < GP * 128; i += kNThr) {
            const int g = i >> 7;
            ot[g][i & 127] = ll[g] > 0.f ? ot[g][i & 127] / ll[g] : 0.f;
        }
        __syncthreads();
        store_out(a, P, ot, mm, ll, sg);
        if (tid == 0) *last = 0;
    }
}

// The merge of a pair whose last partial this CTA published: all partials by
// log-sum-exp, the ticket reset for the next call, then R_V^T and the write.
template <int GP>
__device__ void merge_pair(const DecodeArgs& a, const tq_head_params& P, float (*ot)[128], float* mm, float* ll,
                           const Seg& sg) {
    __threadfence();
    merge_pieces<GP>(a.ws_part + (size_t)sg.first * GP * kPartStride, sg.parts, ot, mm, ll);
    if (threadIdx.x == 0) a.tickets[sg.b * a.Hkv + sg.h] = 0;   // ready for the next call
    __syncthreads();
    store_out(a, P, ot, mm, ll, sg);
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

// Mixed-rate keys: q~ = R_K q for every query head of the round's nseg pieces,
// R_K the head's block-diagonal matrix of group rotations over the grouped
// coordinates [Block-GTQ, physical encoding and grouping]:
//   q~[r] = sum over c in r's group of kmat[r][c] q[gcoord[c]].
// The whole CTA.  One round trip of loads: the raw queries into qts, each piece's
// gcoord into gco, the first piece's matrix (16 float4 per thread) staged
// transposed in kt (kt[c][r]: conflict-free reads).  Then the queries gathered
// into group order in xg ([piece][c][head]), and row r of each piece formed by
// two threads, each over half of r's group.
template <int GPE>
__device__ __forceinline__ void stage_kmat(const DecodeArgs& a, int h, float* kt) {
    const int tid = threadIdx.x;
    const float4* km = reinterpret_cast<const float4*>(a.kmat + (size_t)h * 128 * 128);
    constexpr int PER = 128 * 32 / kNThr;
    float4 v[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int i = tid + u * kNThr;
        v[u] = __ldg(km + (size_t)(i & 127) * 32 + (i >> 7));   // row i & 127, columns 4 (i >> 7) ..
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int i = tid + u * kNThr, r = i & 127, c4 = i >> 7;
        kt[(4 * c4) * 128 + r] = v[u].x;
        kt[(4 * c4 + 1) * 128 + r] = v[u].y;
        kt[(4 * c4 + 2) * 128 + r] = v[u].z;
        kt[(4 * c4 + 3) * 128 + r] = v[u].w;
    }
}

template <int GPE>
__device__ __forceinline__ void rotate_q_mix(const DecodeArgs& a, const Seg* seg, int nseg, float (*qts)[GPE][128],
                                             float* xg, int* gco, float* kt) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = warp; i < nseg * GPE; i += kNW) {
        const Seg& sg = seg[i / GPE];
        const int g = i % GPE;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (g < a.G) tq::load4(a.q, ((size_t)sg.b * a.Hq + (size_t)sg.h * a.G + g) * 128 + 4 * lane, a.q_dtype, v);
#pragma unroll
        for (int e = 0; e < 4; ++e) qts[i / GPE][g][4 * lane + e] = v[e];
    }
    for (int i = tid; i < nseg * 128; i += kNThr) gco[i] = a.params[seg[i >> 7].h].k_gcoord[i & 127];
    stage_kmat<GPE>(a, seg[0].h, kt);
    int staged = seg[0].h;
    __syncthreads();
    for (int i = tid; i < nseg * 128 * GPE; i += kNThr) {
        const int g = i % GPE, c = (i / GPE) & 127, kk = i / (GPE * 128);
        xg[i] = qts[kk][g][gco[kk * 128 + c]];
    }
    __syncthreads();
    for (int kk = 0; kk < nseg; ++kk) {
        const int h = seg[kk].h;
        const tq_head_params& P = a.params[h];
        if (h != staged) {
            stage_kmat<GPE>(a, h, kt);
            staged = h;
            __syncthreads();
        }
        const int r = tid & 127, half = tid >> 7;   // kNThr = 256: two threads per row
        int sr = 0;
        while (sr < 3 && r >= P.k_seg_start[sr + 1]) ++sr;
        const int g0 = P.k_seg_start[sr], g1 = P.k_seg_start[sr + 1];
        const int mid = g0 + ((g1 - g0) >> 1);
        const int c0 = half ? mid : g0, c1 = half ? g1 : mid;
        float acc[GPE];
#pragma unroll
        for (int g = 0; g < GPE; ++g) acc[g] = 0.f;
        for (int c = c0; c < c1; ++c) {
            const float kv = kt[c * 128 + r];
            const float* x0 = xg + ((size_t)kk * 128 + c) * GPE;
#pragma unroll
            for (int g = 0; g < GPE; ++g) acc[g] = fmaf(kv, x0[g], acc[g]);
        }
        if (half) {
#pragma unroll
            for (int g = 0; g < GPE; ++g) qts[kk][g][r] = acc[g];
        }
        __syncthreads();
        if (!half) {
#pragma unroll
            for (int g = 0; g < GPE; ++g) qts[kk][g][r] = (acc[g] + qts[kk][g][r]) * (kLog2e * kInvSqrtD);
        }
        __syncthreads();   // the rows of this piece are complete; kt may be restaged
    }
}

// clamped length of batch b's sequences (flags raised when asked)
__device__ __forceinline__ int seq_len_of(const DecodeArgs& a, int b, bool report) {
    int L = a.seq_lens[b];
    int flags = 0;
    if (L > a.t_cap) { flags |= TQ_DEV_SEQ_OVER_CAPACITY; L = a.t_cap; }
    if (L > a.max_seq) { flags |= TQ_DEV_SEQ_OVER_MAX; L = a.max_seq; }
    if (L < 0) L = 0;
    if (report && flags && a.status) atomicOr(a.status, flags);
    return L;
}

#ifndef TQ_TILE_MINB
#define TQ_TILE_MINB 2
#endif
#ifdef TQ_TILE_MAXNREG
#define TQ_TILE_BOUNDS __maxnreg__(TQ_TILE_MAXNREG)
#else
// two CTAs per SM for four heads and one norm per vector (128 registers); one for
// eight heads, for four 32-wide blocks (their four block norms and chains spill
// at 128 registers: one CTA with all registers measured 8 % faster) and for
// mixed-rate keys (shared memory)
#define TQ_TILE_BOUNDS __launch_bounds__(kNThr, (NT == 1 && !KMIX && NSEG == 1) ? TQ_TILE_MINB : 1)
#endif
// NT: groups of four query heads; BITS, NSEG: code width and norm segments of the
// values (and of the keys unless KMIX: mixed-rate keys in nibble containers with
// four group norms).
template <int NT, int BITS, int NSEG, bool KMIX>
__global__ void TQ_TILE_BOUNDS decode_tile(DecodeArgs a) {
    constexpr int GPE = 4 * NT;
    using Smem = TileSmem<GPE, KMIX>;
    constexpr int NP = Smem::NP;
    constexpr int KB = KMIX ? 4 : BITS, KN = KMIX ? 4 : NSEG;
#ifndef TQ_TILE_DEPTH2
#define TQ_TILE_DEPTH2 1
#endif
    // tiles in flight ahead of the one processed: two where one CTA runs per SM and
    // registers are left (8 heads, or four 32-wide blocks), else one
    constexpr int DEPTH = (TQ_TILE_DEPTH2 && !KMIX && (NT == 2 || NSEG == 4)) ? 2 : 1;
    extern __shared__ __align__(128) unsigned char tile_smem_raw[];
    Smem& S = *reinterpret_cast<Smem*>(tile_smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // launched as a programmatic dependent of the previous kernel in the stream:
    // nothing is read before that kernel has completed and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the lookups address the table at a fixed shared offset: check it (no static
    // shared memory in this kernel, so the dynamic block starts after the
    // reserved 1 KB); on a mismatch nothing is read or written but the flag
    if ((uint32_t)__cvta_generic_to_shared(S.tab) != kTabShared ||
        (KMIX && (uint32_t)__cvta_generic_to_shared(S.ktab) != kTabShared + 65536u)) {
        if (tid == 0 && blockIdx.x == 0 && a.status) atomicOr(a.status, TQ_DEV_INTERNAL);
        return;
    }
    const bool f16n = a.norm_f16 != 0;

    // ---- the CTA's range of tile positions: all tiles of all pairs in pair order
    // (the lengths are read before the table is built, so that both loads overlap)
    const int per = (a.B + kNThr - 1) / kNThr;   // batches summed by each thread, in order
    const int bt0 = min(a.B, tid * per), bt1 = min(a.B, bt0 + per);
    long long loc = 0;
    for (int bb = bt0; bb < bt1; ++bb) loc += (seq_len_of(a, bb, blockIdx.x == 0) + kTok - 1) / kTok;
    build_table<BITS>(a.params[0], S.tab);
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
    for (int w = 0; w < kNW; ++w) {
        before += w < warp ? S.scan[w] : 0;
        total += S.scan[w];
    }
    const long long pre = before + inc - loc;   // tiles per head of batches < bt0
    const long long tiles_all = total * a.Hkv;
    const long long Wd = (tiles_all + gridDim.x - 1) / gridDim.x;
    const long long lo = (long long)blockIdx.x * Wd, hi = min(lo + Wd, tiles_all);
    if (lo < hi && (long long)a.Hkv * pre <= lo && lo < (long long)a.Hkv * (pre + loc)) {
        long long p = (long long)a.Hkv * pre;
        for (int bb = bt0; bb < bt1; ++bb) {
            const long long n = (long long)a.Hkv * ((seq_len_of(a, bb, false) + kTok - 1) / kTok);
            if (lo < p + n) { S.b_first = bb; S.b_base = p; break; }
            p += n;
        }
    }
    // batches with no tokens get zero output (no tile of theirs exists)
    for (int bb = blockIdx.x; bb < a.B; bb += gridDim.x) {
        if (seq_len_of(a, bb, false) == 0) {
            float* ob = a.out + (size_t)bb * a.Hq * 128;
            for (int i = tid; i < a.Hq * 128; i += kNThr) ob[i] = 0.f;
            if (a.lse)
                for (int i = tid; i < a.Hq; i += kNThr) a.lse[(size_t)bb * a.Hq + i] = -INFINITY;
        }
    }
    __syncthreads();
    if (lo >= hi || S.b_first < 0) return;
    if (tid == 0) {
        S.next_pos = lo;
        S.cur_b = S.b_first;
        S.cur_base = S.b_base;
    }
    const Lane ln = lane_ctx();
    const float kinv = 1.0f / a.params[0].k_h_scale[0], vinv = 1.0f / a.params[0].v_h_scale[0];

    for (;;) {
        // ---- next round: up to NP pieces from next_pos (thread 0)
        __syncthreads();
        if (tid == 0) {
            long long p = S.next_pos, base = S.cur_base;
            int b = S.cur_b, n = 0;
            while (p < hi && n < NP && b < a.B) {
                const int L = seq_len_of(a, b, false);
                const int nt = (L + kTok - 1) / kTok;
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
                const long long fc = pstart / Wd, lc = (pstart + nt - 1) / Wd;
                const int pair = b * a.Hkv + h;
                Seg& sg = S.seg[n];
                sg.b = b;
                sg.h = h;
                sg.L = L;
                sg.t_lo = t;
                sg.t_hi = t + take;
                sg.first = (int)fc + pair;   // slot of CTA c for pair p: c + p (unique along the tile order)
                sg.slot = (int)blockIdx.x + pair;
                sg.parts = (int)(lc - fc + 1);
                p += take;
                ++n;
            }
            S.nseg = n;
            S.next_pos = p;
            S.cur_b = b;
            S.cur_base = base;
        }
        __syncthreads();
        const int nseg = S.nseg;
        if (nseg == 0) break;

        // the round's first tile, in flight while the queries are rotated
        KRegs<KB, KN> kA, kB;
        VRegs<BITS, NSEG> vA, vB;
        PairPtr pp = pair_ptr<KB, KN, BITS, NSEG>(a, S.seg[0].b, S.seg[0].h);
        bool first_loaded = false;
        if (S.seg[0].t_lo + warp < S.seg[0].t_hi) {
            load_k(kA, pp, S.seg[0].t_lo + warp, ln, f16n);
            load_v(vA, pp, S.seg[0].t_lo + warp, ln, f16n);
            first_loaded = true;
        }
        if constexpr (!KMIX) {
            for (int i = warp; i < nseg * GPE; i += kNW) {
                const Seg& sg = S.seg[i / GPE];
                rotate_q(a, a.params[sg.h], sg.b, sg.h, i % GPE, S.qts[i / GPE][i % GPE]);
            }
            __syncthreads();
        }

        for (int k = 0; k < nseg; ++k) {
            const Seg sg = S.seg[k];
            const tq_head_params& P = a.params[sg.h];
            BqT<NT> bq;
            uint32_t colpack[4];
            uint32_t kmask = 0u;
            const uint2* bmp = nullptr;
            if constexpr (KMIX) {
                // per piece (so that a CTA's second piece never delays its first):
                // q~ of the piece's heads, staging the group rotations in the key
                // tables' space; the k steps each group touches (warp 0, lane
                // 4 st + g); operand B of every (k step, group, head group, lane);
                // then the key tables of the piece's head
                static_assert(kNThr == 256, "two threads per rotated row");
                static_assert(kNW * GPE * 128 >= 128 * GPE + 128, "scratch for the gathered queries and gcoord");
                float* xg = &S.wo[0][0][0];
                rotate_q_mix<GPE>(a, &S.seg[k], 1, S.qts, xg, reinterpret_cast<int*>(xg + 128 * GPE),
                                  reinterpret_cast<float*>(S.ktab));
                if (warp == 0) {
                    const int st = lane >> 2, g = lane & 3;
                    const int glo = P.k_seg_start[g] >> 1, ghi = P.k_seg_start[g + 1] >> 1;
                    const bool touch = ghi > glo && glo < 8 * st + 8 && ghi > 8 * st;
                    const uint32_t m = __ballot_sync(TQ_FULL_MASK, touch);
                    if (lane == 0) S.kmask[0] = m;
                }
                // lane (r, c) holds head 4j + r/2, coordinates of pairs 8 st + c (b0)
                // and 8 st + c + 4 (b1) when they lie in group g, as the rounded q~
                // (r even) or its rounding remainder (r odd), over the group's
                // table scale
                for (int i = tid; i < 8 * 4 * NT * 32; i += kNThr) {
                    const int L = i & 31;
                    int rest = i >> 5;
                    const int j = rest % NT;
                    rest /= NT;
                    const int g = rest & 3, st = rest >> 2;
                    const int glo = P.k_seg_start[g] >> 1, ghi = P.k_seg_start[g + 1] >> 1;
                    const int r = L >> 2, c = L & 3;
                    const float* qh = S.qts[0][4 * j + (r >> 1)];
                    const int p0 = 8 * st + c, p1 = p0 + 4;
                    uint32_t b0 = 0u, b1 = 0u;
                    if (ghi > glo) {
                        const float ki = 1.0f / P.k_h_scale[g];
                        if (p0 >= glo && p0 < ghi) b0 = pack_part(qh[2 * p0] * ki, qh[2 * p0 + 1] * ki, r & 1);
                        if (p1 >= glo && p1 < ghi) b1 = pack_part(qh[2 * p1] * ki, qh[2 * p1 + 1] * ki, r & 1);
                    }
                    S.bm[0][st][g][j][L] = make_uint2(b0, b1);
                }
                build_ktable(P, S.ktab);   // rotate_q_mix ended with a barrier: the staging is done
                __syncthreads();
                const int p4 = P.k_seg_start[3] >> 1;   // first pair of the 4-bit group
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t x = 0u;
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb) {
                        const int pr = tqtile::k_pair(ln.c, 4 * w + kb);
                        x |= (4u * lane + (pr >= p4 ? 128u : 0u)) << (8 * kb);
                    }
                    colpack[w] = x;
                }
                kmask = S.kmask[0];
                bmp = &S.bm[0][0][0][0][lane];
            } else {
                load_bq<NT>(S.qts[k], ln, kinv, bq.r);
            }
            (void)colpack;
            (void)kmask;
            (void)bmp;
            WState<NT> ws;
            ws.reset();
            // this warp's tiles of the piece: t_lo + warp + kNW i
            const int n = sg.t_hi - sg.t_lo > warp ? (sg.t_hi - sg.t_lo - warp + kNW - 1) / kNW : 0;
            auto tile_at = [&](int i) { return sg.t_lo + warp + kNW * i; };
            auto nval_at = [&](int i) { return min(kTok, sg.L - tile_at(i) * kTok); };
            auto step = [&](const KRegs<KB, KN>& kd, const VRegs<BITS, NSEG>& vd, int nv) {
                float s0[NT], s8[NT];
                if constexpr (KMIX) qk_phase_mix<NT>(kd, colpack, bmp, kmask, s0, s8);
                else qk_phase<NT, BITS, NSEG>(kd, ln, bq, f16n, s0, s8);
                pv_phase<NT, BITS, NSEG>(vd, s0, s8, nv, ln, f16n, ws);
            };
            if (n > 0 && !first_loaded) {
                load_k(kA, pp, tile_at(0), ln, f16n);
                load_v(vA, pp, tile_at(0), ln, f16n);
            }
            if constexpr (DEPTH == 2) {
                // tiles i + 1 and i + 2 in flight while tile i is processed
                KRegs<KB, KN> kC;
                VRegs<BITS, NSEG> vC;
                if (n > 1) {
                    load_k(kB, pp, tile_at(1), ln, f16n);
                    load_v(vB, pp, tile_at(1), ln, f16n);
                }
                for (int i = 0; i < n; i += 3) {
                    if (i + 2 < n) {
                        load_k(kC, pp, tile_at(i + 2), ln, f16n);
                        load_v(vC, pp, tile_at(i + 2), ln, f16n);
                    }
                    step(kA, vA, nval_at(i));
                    if (i + 1 >= n) break;
                    if (i + 3 < n) {
                        load_k(kA, pp, tile_at(i + 3), ln, f16n);
                        load_v(vA, pp, tile_at(i + 3), ln, f16n);
                    }
                    step(kB, vB, nval_at(i + 1));
                    if (i + 2 >= n) break;
                    if (i + 4 < n) {
                        load_k(kB, pp, tile_at(i + 4), ln, f16n);
                        load_v(vB, pp, tile_at(i + 4), ln, f16n);
                    }
                    step(kC, vC, nval_at(i + 2));
                }
            } else {
                // tile i + 1 in flight while tile i is processed
                for (int i = 0; i < n; i += 2) {
                    if (i + 1 < n) {
                        load_k(kB, pp, tile_at(i + 1), ln, f16n);
                        load_v(vB, pp, tile_at(i + 1), ln, f16n);
                    }
                    step(kA, vA, nval_at(i));
                    if (i + 1 >= n) break;
                    if (i + 2 < n) {
                        load_k(kA, pp, tile_at(i + 2), ln, f16n);
                        load_v(vA, pp, tile_at(i + 2), ln, f16n);
                    }
                    step(kB, vB, nval_at(i + 1));
                }
            }
            // the next piece's first tile, in flight during the merge
            first_loaded = false;
            if (k + 1 < nseg) {
                const Seg& sn = S.seg[k + 1];
                pp = pair_ptr<KB, KN, BITS, NSEG>(a, sn.b, sn.h);
                if (sn.t_lo + warp < sn.t_hi) {
                    load_k(kA, pp, sn.t_lo + warp, ln, f16n);
                    load_v(vA, pp, sn.t_lo + warp, ln, f16n);
                    first_loaded = true;
                }
            }
            warp_state_out<NT>(ws, ln, S.wo[warp], S.wm[warp], S.wl[warp]);
            __syncthreads();
            merge_warps<GPE, GPE>(S.wo, S.wm, S.wl, vinv, S.ot, S.mm, S.ll);
            __syncthreads();
            finish_piece<GPE>(a, P, S.ot, S.mm, S.ll, &S.last[k], sg);
            __syncthreads();
        }
        // merges of the pairs whose last partial this CTA published, after all of
        // the round's tiles (a merge never delays the CTA's own partial of a pair)
        for (int k = 0; k < nseg; ++k) {
            if (!S.last[k]) continue;
            const Seg sg = S.seg[k];
            merge_pair<GPE>(a, a.params[sg.h], S.ot, S.mm, S.ll, sg);
            __syncthreads();
        }
    }
}

using KernelPtr = void (*)(DecodeArgs);

template <int NT, int BITS, int NSEG, bool KMIX>
KernelPtr kernel_of(size_t* smem) {
    *smem = sizeof(TileSmem<4 * NT, KMIX>);
    return decode_tile<NT, BITS, NSEG, KMIX>;
}

template <int NT>
KernelPtr pick_nt(const tq_cache_desc* d, size_t* smem) {
    const bool v4 = d->v_bits == 4;
    if (d->k_mixed) return v4 ? kernel_of<NT, 4, 1, true>(smem) : kernel_of<NT, 3, 1, true>(smem);
    if (d->rot == TQ_ROT_WHT32) return v4 ? kernel_of<NT, 4, 4, false>(smem) : kernel_of<NT, 3, 4, false>(smem);
    return v4 ? kernel_of<NT, 4, 1, false>(smem) : kernel_of<NT, 3, 1, false>(smem);
}

KernelPtr pick(const tq_cache_desc* d, size_t* smem) {
    return d->group <= 4 ? pick_nt<1>(d, smem) : pick_nt<2>(d, smem);
}

// resident CTAs of the kernel for this format (CTAs per SM x SMs), looked up once
// per device and kernel
int grid_cap(const tq_cache_desc* d) {
    static std::mutex mu;
    static int cache[64][16];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const int which = (d->group <= 4 ? 0 : 8) + (d->v_bits == 4 ? 4 : 0) + (d->rot == TQ_ROT_WHT32 ? 2 : 0) +
                      (d->k_mixed ? 1 : 0);
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev][which]) {
        size_t smem = 0;
        KernelPtr fn = pick(d, &smem);
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kNThr, smem) != cudaSuccess || n < 1) return 0;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) return 0;
        cache[dev][which] = n * sms;
    }
    return cache[dev][which];
}

}  // namespace

bool tq_decode_tc_supported(const tq_cache_desc* d) { return d->layout == TQ_LAYOUT_TILE16; }

int tq_decode_tc_sk_slots(const tq_cache_desc* d) { return kMaxGrid + d->batch * d->n_kv_heads; }

int tq_decode_tc_max_grid() { return kMaxGrid; }

int tq_decode_tc_sk_grid(const tq_cache_desc* d, int max_seq_len) {
    // resident CTAs on this device; without one, the design's: 2 (4 query heads
    // per KV head, one norm per vector) or 1 CTAs per SM on 152 SMs
    int cap = grid_cap(d);
    if (cap <= 0) cap = (d->group <= 4 && !d->k_mixed && d->rot != TQ_ROT_WHT32 ? TQ_TILE_MINB : 1) * 152;
    // one wave of resident CTAs, each warp with at least one tile
    const long long tiles = (long long)d->batch * d->n_kv_heads * ((max_seq_len + kTok - 1) / kTok);
    long long g = (tiles + kNW - 1) / kNW;
    if (g > cap) g = cap;
    if (g > kMaxGrid) g = kMaxGrid;
    return g < 1 ? 1 : (int)g;
}

cudaError_t tq_decode_tc_launch(const tq_cache_desc* d, const tq::DecodeArgs& a, int grid, cudaStream_t stream) {
    // sets the kernel's dynamic shared-memory limit on this device (once)
    if (grid_cap(d) <= 0) return cudaErrorInvalidConfiguration;
    size_t smem = 0;
    KernelPtr fn = pick(d, &smem);
    // programmatic dependent launch: the CTAs are placed while the previous kernel
    // (typically the token append) finishes, and wait for it on the device
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kNThr);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, a);
}
