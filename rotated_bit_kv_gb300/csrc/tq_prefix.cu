// Decode attention over a block of unquantised tokens plus the packed cache.
//
// [RotaryQuant] deferred prefill: the prompt's K and V stay in fp16 and only the
// tokens generated while decoding are quantised; [Block-GTQ] recent-token
// buffer: the newest tokens are kept unquantised.  Either way a query attends
// to the union of two parts of its keys.  The packed part runs through the
// compressed-domain decode (tq_decode.cu / tq_decode_tile.cu), which leaves the
// normalised output and each head's log2-sum-exp (lse); this file attends to the
// unquantised part in the original domain and merges the two by log-sum-exp
// [Block-GTQ, key-axis split]:
//   M = max(lse_p, m_f),  o = (2^(lse_p - M) o_p + 2^(m_f - M) o~_f) / (2^(lse_p - M) + 2^(m_f - M) l_f)
// with (m_f, l_f, o~_f) the unquantised part's running max, sum and unnormalised
// output (scores in log2 units: q log2(e) / sqrt(d)).
//
// Kernel: grid (splits, n_kv, batch), 4 warps.  A CTA takes a section of the
// sequence's unquantised tokens; each warp takes every fourth token of it, one
// token per step: lane l holds coordinates 4l .. 4l+3 of K, V, of every query
// head's q (registers) and of its output.  The G per-lane partial dot products
// are summed across the warp by a reduce-scatter (each lane ends with the score
// of one head) and the G weights are broadcast back for the V accumulation.
// The warps' states are merged in shared memory; with one section the CTA
// merges with the packed part and writes the output, else it publishes its
// partial and the last CTA of the (batch, KV head) merges all of them.
#include <stddef.h>

#include "tq_decode_common.cuh"
#include "tq_mma.cuh"

namespace {

constexpr int kPW = 4;                  // warps per CTA
constexpr int kPThr = kPW * 32;

struct PrefixArgs {
    const void* k;          // [B][cap][Hkv][128]
    const void* v;
    const void* q;          // [B][Hq][128]
    const int32_t* lens;    // [B]
    const float* lse_p;     // [B][Hq] of the packed part, or null (no packed part)
    float* out;             // [B][Hq][128]: the packed part's output in, the merged output out
    float* ws_part;         // [B * Hkv][splits][GP] rows of kPartStride floats
    int32_t* tickets;       // [B * Hkv]
    int32_t* status;
    const uint8_t* k_meta;  // ZipFusion pages: [B * Hkv][pages] x 8 bytes each, else null
    const uint8_t* v_meta;
    int B, Hq, Hkv, G, cap, max_len, splits, split_len, dtype, q_dtype;
};

__device__ __forceinline__ float ex2f(float x) {   // hardware 2^x; 2^-inf = 0
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Sum x[0 .. GP-1] over the warp, scattered: afterwards lane l holds the full sum
// of head (l >> (5 - log2 GP)) in x[0] (halving exchanges, then whole-value sums
// over the remaining lane bits).
template <int GP>
__device__ __forceinline__ float reduce_scatter(float (&x)[GP], int lane) {
#pragma unroll
    for (int m = 16, n = GP; m >= 1; m >>= 1) {
        if (n > 1) {
            const int half = n >> 1;
            const bool upper = lane & m;
#pragma unroll
            for (int i = 0; i < GP / 2; ++i) {
                if (i < half) {
                    const float send = upper ? x[i] : x[i + half];
                    const float keep = upper ? x[i + half] : x[i];
                    x[i] = keep + __shfl_xor_sync(TQ_FULL_MASK, send, m);
                }
            }
            n = half;
        } else {
            x[0] += __shfl_xor_sync(TQ_FULL_MASK, x[0], m);
        }
    }
    return x[0];
}

template <int GP>
constexpr int log2_gp() { return GP == 1 ? 0 : GP == 2 ? 1 : GP == 4 ? 2 : GP == 8 ? 3 : 4; }

// clamped prefix length of batch b (flags raised when asked)
__device__ __forceinline__ int prefix_len(const PrefixArgs& a, int b, bool report) {
    int L = a.lens[b];
    int flags = 0;
    if (L > a.cap) { flags |= TQ_DEV_SEQ_OVER_CAPACITY; L = a.cap; }
    if (L > a.max_len) { flags |= TQ_DEV_SEQ_OVER_MAX; L = a.max_len; }
    if (L < 0) L = 0;
    if (report && flags && a.status) atomicOr(a.status, flags);
    return L;
}

// The end of a prefix CTA: ot[g][0..127] (flat, unnormalised) and (sM, sL) hold
// its section's state.  Sections: publish, the last CTA of the (batch, KV head)
// merges them all (normalised into ot, (M, L) in sM, sL); one section:
// normalise.  Then the merge with the packed part:
//   o = (w_p o_p + w_f L_f o_f) / (w_p + w_f L_f).
template <int GP, int NTHR>
__device__ __forceinline__ void prefix_finish(const PrefixArgs& a, float* ot, float* sM, float* sL, int* is_last,
                                              int b, int h, int s) {
    const int tid = threadIdx.x;
    if (a.splits > 1) {
        float* part = a.ws_part + ((((size_t)b * a.Hkv + h) * a.splits + s) * GP) * kPartStride;
        for (int i = tid; i < GP * 128; i += NTHR) part[(i >> 7) * kPartStride + (i & 127)] = ot[i];
        if (tid < GP) {
            part[tid * kPartStride + 128] = sM[tid];
            part[tid * kPartStride + 129] = sL[tid];
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const int ticket = atomicAdd(a.tickets + (size_t)b * a.Hkv + h, 1);
            *is_last = ticket == a.splits - 1;
        }
        __syncthreads();
        if (!*is_last) return;
        __threadfence();
        merge_parts<GP, NTHR>(a.ws_part + (((size_t)b * a.Hkv + h) * a.splits * GP) * kPartStride, a.splits,
                              reinterpret_cast<float(*)[128]>(ot), sM, sL);
        if (tid == 0) a.tickets[(size_t)b * a.Hkv + h] = 0;   // ready for the next call
        __syncthreads();
    } else {
        for (int i = tid; i < GP * 128; i += NTHR) {
            const int g = i >> 7;
            ot[i] = sL[g] > 0.f ? ot[i] / sL[g] : 0.f;
        }
        __syncthreads();
    }
    for (int i = tid; i < a.G * 128; i += NTHR) {
        const int g = i >> 7;
        float* dst = a.out + ((size_t)b * a.Hq + (size_t)h * a.G + g) * 128 + (i & 127);
        const float lp = a.lse_p ? a.lse_p[(size_t)b * a.Hq + (size_t)h * a.G + g] : -INFINITY;
        const float Mf = sM[g], Lf = sL[g];
        const float M = fmaxf(lp, Mf);
        const float wp = lp == -INFINITY ? 0.f : ex2f(lp - M);
        const float wf = (Mf == -INFINITY || !(Lf > 0.f)) ? 0.f : ex2f(Mf - M) * Lf;
        const float den = wp + wf;
        const float op = wp > 0.f ? *dst : 0.f;   // the packed output is read only when it weighs
        *dst = den > 0.f ? (wp * op + wf * ot[i]) / den : 0.f;
    }
}

template <int GP>
__global__ void __launch_bounds__(kPThr) prefix_attend(PrefixArgs a) {
    __shared__ __align__(16) float wo[kPW][GP][128];
    __shared__ float wm[kPW][GP], wl[kPW][GP];
    __shared__ float sM[GP], sL[GP];
    __shared__ int is_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    // programmatic dependent of the packed decode: its output and lse are read after this
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int L = prefix_len(a, b, s == 0 && h == 0);
    const int t0 = s * a.split_len, t1 = min(L, t0 + a.split_len);

    // this lane's four coordinates of every head's query, in log2 units
    float qv[GP][4];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (g < a.G) tq::load4(a.q, ((size_t)b * a.Hq + (size_t)h * a.G + g) * 128 + 4 * lane, a.q_dtype, v);
#pragma unroll
        for (int i = 0; i < 4; ++i) qv[g][i] = v[i] * (kLog2e * kInvSqrtD);
    }
    constexpr int LG = log2_gp<GP>();
    const int myg = lane >> (5 - LG);        // head whose score this lane ends with
    float m = -INFINITY, l = 0.f;            // of head myg (identical in its lanes)
    float o[GP][4];
#pragma unroll
    for (int g = 0; g < GP; ++g) o[g][0] = o[g][1] = o[g][2] = o[g][3] = 0.f;

    const size_t row = (size_t)a.Hkv * 128;   // elements per token position
    const size_t base = ((size_t)b * a.cap * a.Hkv + h) * 128 + 4 * lane;
    for (int t = t0 + warp; t < t1; t += kPW) {
        float kx[4], vx[4];
        tq::load4(a.k, base + (size_t)t * row, a.dtype, kx);
        tq::load4(a.v, base + (size_t)t * row, a.dtype, vx);
        float part[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g)
            part[g] = fmaf(qv[g][0], kx[0], fmaf(qv[g][1], kx[1], fmaf(qv[g][2], kx[2], qv[g][3] * kx[3])));
        const float sc = reduce_scatter<GP>(part, lane);
        // online softmax of head myg; the base moves only past m + 4 (weights <= 16)
        const bool move = sc > m + 4.f;
        const float mn = move ? sc : m;
        const float c = ex2f(m - mn);         // 1 unless the base moved (0 on the first token)
        const float p = ex2f(sc - mn);
        l = fmaf(l, c, p);
        m = mn;
        if (__any_sync(TQ_FULL_MASK, move)) {
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                const float cg = __shfl_sync(TQ_FULL_MASK, c, g << (5 - LG));
                o[g][0] *= cg; o[g][1] *= cg; o[g][2] *= cg; o[g][3] *= cg;
            }
        }
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            const float pg = __shfl_sync(TQ_FULL_MASK, p, g << (5 - LG));
#pragma unroll
            for (int i = 0; i < 4; ++i) o[g][i] = fmaf(pg, vx[i], o[g][i]);
        }
    }

    // ---- the warps' states into one (m, l, o~) per head
#pragma unroll
    for (int g = 0; g < GP; ++g)
        *reinterpret_cast<float4*>(&wo[warp][g][4 * lane]) = make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
    if ((lane & ((32 >> LG) - 1)) == 0) {
        wm[warp][myg] = m;
        wl[warp][myg] = l;
    }
    __syncthreads();
    float* ot = &wo[0][0][0];   // merged in place into warp 0's rows
    for (int i = tid; i < GP * 128; i += kPThr) {
        const int g = i >> 7, d = i & 127;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kPW; ++w) M = fmaxf(M, wm[w][g]);
        float Lt = 0.f, ov = 0.f;
#pragma unroll
        for (int w = 0; w < kPW; ++w) {
            const float wt = (M == -INFINITY || wm[w][g] == -INFINITY) ? 0.f : ex2f(wm[w][g] - M);
            Lt = fmaf(wt, wl[w][g], Lt);
            ov = fmaf(wt, wo[w][g][d], ov);
        }
        ot[i] = ov;   // wo[0][g][d]: this thread alone reads and writes column (g, d)
        if (d == 0) {
            sM[g] = M;
            sL[g] = Lt;
        }
    }
    __syncthreads();

    prefix_finish<GP, kPThr>(a, ot, sM, sL, &is_last, b, h, s);
}

// ---- tensor-core kernel for up to 8 query heads per KV head
//
// Each warp takes whole 16-token tiles of its CTA's section, on the legacy
// warp-level MMA with fp16 operands and fp32 accumulation, in the coordinate-pair
// form of the packed-cache kernel with the operands read straight from the
// unquantised rows:
//   QK: S[16 tok x 8] = K[16 x 128] . B_q[128 x 8], lane (r, c) holding pairs
//       16c .. 16c+15 of tokens r and r + 8 (64 contiguous bytes each) and B_q the
//       query (rounded to fp16, and its rounding remainder, in the two columns of
//       a head) at the same pairs;
//   PV: O[64 pairs x 8] += V[pairs x (token, parity)] . B_p, m tile mt holding
//       pairs 8r + 2mt (rows r) and 8r + 2mt + 1 (rows r + 8), so that lane (r, c)
//       reads pairs 8r .. 8r+7 (32 contiguous bytes) of tokens 2c, 2c+1, 2c+8,
//       2c+9 and ends with coordinates 16r .. 16r+15 of its head.
// bf16 rows run bf16 MMAs as they are (the query and the weights split into their
// bf16 rounding and its remainder); fp32 rows are rounded to fp16 on load.
constexpr int kTW = 8;
constexpr int kTThr = kTW * 32;

// N 16-bit pair words (2N elements) of the input from element `elem` (16-byte
// aligned): fp32 rounded to fp16 pairs; fp16 and bf16 words as they are
template <int DT, int N>
__device__ __forceinline__ void load_words(const void* base, size_t elem, uint32_t (&w)[N]) {
    if constexpr (DT == TQ_F32) {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem);
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float4 x = __ldg(p + i);
            w[2 * i] = pack_h2(x.x, x.y);
            w[2 * i + 1] = pack_h2(x.z, x.w);
        }
    } else {
        const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem);
#pragma unroll
        for (int i = 0; i < N / 4; ++i) {
            const uint4 x = __ldg(p + i);
            w[4 * i] = x.x; w[4 * i + 1] = x.y; w[4 * i + 2] = x.z; w[4 * i + 3] = x.w;
        }
    }
}

// Operand sources of the tile kernel.  A lane (r, c) needs, per 16-token tile:
// keys, pairs 16c .. 16c+15 (coordinates 32c .. 32c+31) of tokens r and r + 8, as
// 16 fp16 pair words each; values, pairs 8r .. 8r+7 (coordinates 16r .. 16r+15) of
// tokens 2c, 2c+1, 2c+8, 2c+9, 8 words each.

// Unquantised rows [B][cap][Hkv][128] of DT.
template <int DT>
struct RowSrc {
    static constexpr bool kLaunch2 = DT != TQ_F32;   // two CTAs per SM fit its registers
    static constexpr bool kBf16 = DT == TQ_BF16;     // bf16 words go to bf16 MMAs as they are
    static constexpr int kLoad = DT == TQ_BF16 ? TQ_F16 : DT;   // 16-bit words: copied
    const void* k;
    const void* v;
    size_t base, row;
    int t1;
    __device__ __forceinline__ RowSrc(const PrefixArgs& a, int b, int h, int t1_)
        : k(a.k), v(a.v), base(((size_t)b * a.cap * a.Hkv + h) * 128), row((size_t)a.Hkv * 128), t1(t1_) {}
    __device__ __forceinline__ size_t tok(int tb, int i) const { return (size_t)min(tb + i, t1 - 1); }
    __device__ __forceinline__ void prefetch(int) {}
    __device__ __forceinline__ void finish_k(uint32_t (&)[16], uint32_t (&)[16]) const {}
    __device__ __forceinline__ void finish_v(uint32_t (&)[8], uint32_t (&)[8], uint32_t (&)[8], uint32_t (&)[8]) const {}
    __device__ __forceinline__ void load_k(int tb, int r, int c, uint32_t (&kr)[16], uint32_t (&k8)[16]) const {
        load_words<kLoad>(k, base + tok(tb, r) * row + 32 * c, kr);
        load_words<kLoad>(k, base + tok(tb, r + 8) * row + 32 * c, k8);
    }
    __device__ __forceinline__ void load_v(int tb, int r, int c, uint32_t (&va0)[8], uint32_t (&vb0)[8],
                                           uint32_t (&va1)[8], uint32_t (&vb1)[8]) const {
        load_words<kLoad>(v, base + tok(tb, 2 * c) * row + 16 * r, va0);
        load_words<kLoad>(v, base + tok(tb, 2 * c + 1) * row + 16 * r, vb0);
        load_words<kLoad>(v, base + tok(tb, 2 * c + 8) * row + 16 * r, va1);
        load_words<kLoad>(v, base + tok(tb, 2 * c + 9) * row + 16 * r, vb1);
    }
};

// ---- ZipFusion pages [ZipFusion, compression format, register restore]
//
// A page is 16 tokens of one (batch, KV head) and of K or V: four 512-value blocks
// of 64 groups of 8 values, each block either compressed (512 low bytes, then 256
// code bytes: 768 B) or raw (1024 B of bf16), stored one after another from the
// page's offset.  A block holds the groups that lane L = 4r + c of a warp reads at
// one step, groups 2L and 2L + 1 side by side (so a block's mode is warp-uniform
// and a lane's part of it is one 16-byte and one 8-byte piece):
//   K block q: tokens r and r + 8, coordinates 32c + 8q .. +7;
//   V block 2e + q: tokens 2c + 8e and 2c + 8e + 1, coordinates 16r + 8q .. +7.
// Metadata, 8 bytes per page: the offset of block 0 in 256-byte units from the
// pool base (uint32), then one byte per block: b/2 (compressed) or kZipRaw.
constexpr uint32_t kZipRaw = 0xFF;

// Eight bf16 values of a compressed group, as four bf16 pair words, from their low
// bytes (l0: values 0-3, l1: 4-7) and code word w: high bytes 128 s + b/2 + d in
// one add for values 0-3 (sign bit 7, d bits 0-2) and one for 4-7 (sign bit 6,
// d bits 3-5; moved into the same places).
__device__ __forceinline__ void zip_group(uint32_t l0, uint32_t l1, uint32_t w, uint32_t hb4, uint32_t* out) {
    const uint32_t hi_a = (w & 0x87878787u) + hb4;
    const uint32_t hi_b = (((w >> 3) & 0x07070707u) | ((w << 1) & 0x80808080u)) + hb4;
    out[0] = prmt(l0, hi_a, 0x5140u);
    out[1] = prmt(l0, hi_a, 0x7362u);
    out[2] = prmt(l1, hi_b, 0x5140u);
    out[3] = prmt(l1, hi_b, 0x7362u);
}

struct ZipSrc {
    static constexpr bool kLaunch2 = true;
    static constexpr bool kBf16 = true;
    const uint8_t* kpool;
    const uint8_t* vpool;
    const uint8_t* kmeta;   // this (batch, KV head)'s pages
    const uint8_t* vmeta;
    uint32_t lim;           // pool size in 256-byte units: a page's offset must stay below lim - 16
    int32_t* status;
    int t1;
    uint2 km, vm;           // metadata of the next tile to load, fetched a tile ahead
    __device__ __forceinline__ ZipSrc(const PrefixArgs& a, int b, int h, int t1_)
        : kpool(static_cast<const uint8_t*>(a.k)), vpool(static_cast<const uint8_t*>(a.v)),
          kmeta(a.k_meta + ((size_t)b * a.Hkv + h) * (a.cap / 16) * 8),
          vmeta(a.v_meta + ((size_t)b * a.Hkv + h) * (a.cap / 16) * 8),
          lim((uint32_t)((size_t)a.B * a.Hkv * (a.cap / 16) * 16)), status(a.status), t1(t1_),
          km(make_uint2(0u, 0u)), vm(make_uint2(0u, 0u)) {}
    // the metadata of tile tb (the next one load_k / load_v will take): its data
    // loads then need no dependent metadata round trip
    __device__ __forceinline__ void prefetch(int tb) {
        if (tb < t1) {
            km = __ldg(reinterpret_cast<const uint2*>(kmeta + (size_t)(tb >> 4) * 8));
            vm = __ldg(reinterpret_cast<const uint2*>(vmeta + (size_t)(tb >> 4) * 8));
        }
    }
    // a page's metadata; an offset outside the pool reads page 0 and raises a flag
    __device__ __forceinline__ uint2 checked(uint2 m) const {
        if (m.x > lim - 16) {
            if (status) atomicOr(status, TQ_DEV_BAD_METADATA);
            m.x = 0;
        }
        return m;
    }
    // The lane's two groups (2L, 2L + 1) of every block of a page, loaded into w0 / w1
    // as they are stored (the decode waits for use, so the loads' latency overlaps
    // the current tile): block j raw: w0[4j..] and w1[4j..] its 32 bytes; compressed:
    // w0[4j..4j+3] the 16 low bytes, w1[4j], w1[4j+1] the 8 code bytes.
    __device__ __forceinline__ static void load_page(const uint8_t* pool, uint2 m, int lane, uint32_t (&w0)[16],
                                                     uint32_t (&w1)[16]) {
        const uint8_t* blk = pool + (size_t)m.x * 256;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t mark = (m.y >> (8 * j)) & 0xFFu;   // warp-uniform
            if (mark == kZipRaw) {
                const uint4* p = reinterpret_cast<const uint4*>(blk + 32 * lane);
                const uint4 x = __ldg(p), y = __ldg(p + 1);
                w0[4 * j] = x.x; w0[4 * j + 1] = x.y; w0[4 * j + 2] = x.z; w0[4 * j + 3] = x.w;
                w1[4 * j] = y.x; w1[4 * j + 1] = y.y; w1[4 * j + 2] = y.z; w1[4 * j + 3] = y.w;
                blk += 1024;
            } else {
                const uint4 lo = __ldg(reinterpret_cast<const uint4*>(blk + 16 * lane));
                const uint2 cw = __ldg(reinterpret_cast<const uint2*>(blk + 512 + 8 * lane));
                w0[4 * j] = lo.x; w0[4 * j + 1] = lo.y; w0[4 * j + 2] = lo.z; w0[4 * j + 3] = lo.w;
                w1[4 * j] = cw.x; w1[4 * j + 1] = cw.y;
                blk += 768;
            }
        }
    }
    // ... and restored in place to bf16 pair words: w0[4j ..] group 2L, w1[4j ..] 2L + 1
    __device__ __forceinline__ static void restore_page(uint32_t marks, uint32_t (&w0)[16], uint32_t (&w1)[16]) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t mark = (marks >> (8 * j)) & 0xFFu;
            if (mark != kZipRaw) {
                const uint32_t hb4 = mark * 0x01010101u;
                const uint32_t c0 = w1[4 * j], c1 = w1[4 * j + 1];
                zip_group(w0[4 * j + 2], w0[4 * j + 3], c1, hb4, &w1[4 * j]);
                zip_group(w0[4 * j], w0[4 * j + 1], c0, hb4, &w0[4 * j]);
            }
        }
    }
    uint32_t kmarks = 0, vmarks = 0;   // block marks of the tile last loaded
    __device__ __forceinline__ void load_k(int, int r, int c, uint32_t (&kr)[16], uint32_t (&k8)[16]) {
        const uint2 m = checked(km);
        kmarks = m.y;
        load_page(kpool, m, 4 * r + c, kr, k8);   // block q: pairs 16c + 4q .. +3
    }
    __device__ __forceinline__ void finish_k(uint32_t (&kr)[16], uint32_t (&k8)[16]) const {
        restore_page(kmarks, kr, k8);
    }
    // values: block 2e + q holds tokens 2c + 8e (w0) and 2c + 8e + 1 (w1), pairs
    // 8r + 4q ..; va0 / vb0 are blocks 0, 1 and va1 / vb1 blocks 2, 3 of w0 / w1
    __device__ __forceinline__ void load_v(int, int r, int c, uint32_t (&va0)[8], uint32_t (&vb0)[8],
                                           uint32_t (&va1)[8], uint32_t (&vb1)[8]) {
        const uint2 m = checked(vm);
        vmarks = m.y;
        uint32_t w0[16], w1[16];
        load_page(vpool, m, 4 * r + c, w0, w1);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            va0[i] = w0[i];
            vb0[i] = w1[i];
            va1[i] = w0[8 + i];
            vb1[i] = w1[8 + i];
        }
    }
    __device__ __forceinline__ void finish_v(uint32_t (&va0)[8], uint32_t (&vb0)[8], uint32_t (&va1)[8],
                                             uint32_t (&vb1)[8]) const {
        uint32_t w0[16], w1[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            w0[i] = va0[i];
            w1[i] = vb0[i];
            w0[8 + i] = va1[i];
            w1[8 + i] = vb1[i];
        }
        restore_page(vmarks, w0, w1);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            va0[i] = w0[i];
            vb0[i] = w1[i];
            va1[i] = w0[8 + i];
            vb1[i] = w1[8 + i];
        }
    }
};

template <int NT, class Src>
__global__ void __launch_bounds__(kTThr, (NT == 1 && Src::kLaunch2) ? 2 : 1) prefix_tile(PrefixArgs a) {
    constexpr int GPE = 4 * NT;
    __shared__ __align__(16) float qf[GPE][128];
    __shared__ __align__(16) float wo[kTW][GPE][128];
    __shared__ float wm[kTW][GPE], wl[kTW][GPE];
    __shared__ float sM[GPE], sL[GPE];
    __shared__ int is_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int L = prefix_len(a, b, s == 0 && h == 0);
    const int t0 = s * a.split_len, t1 = min(L, t0 + a.split_len);
    for (int g = warp; g < GPE; g += kTW) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (g < a.G) tq::load4(a.q, ((size_t)b * a.Hq + (size_t)h * a.G + g) * 128 + 4 * lane, a.q_dtype, v);
#pragma unroll
        for (int i = 0; i < 4; ++i) qf[g][4 * lane + i] = v[i] * (kLog2e * kInvSqrtD);
    }
    __syncthreads();
    constexpr bool BF = Src::kBf16;   // bf16 operands (P split into its bf16 rounding and remainder)
    const int r = lane >> 2, c = lane & 3;
    const bool odd = r & 1;
    uint32_t bq[NT][8][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const float* qh = qf[4 * j + (r >> 1)];
#pragma unroll
        for (int st = 0; st < 8; ++st) {
            const int d0 = 2 * (16 * c + 2 * st);
            bq[j][st][0] = BF ? pack_part_bf(qh[d0], qh[d0 + 1], odd) : pack_part(qh[d0], qh[d0 + 1], odd);
            bq[j][st][1] = BF ? pack_part_bf(qh[d0 + 2], qh[d0 + 3], odd) : pack_part(qh[d0 + 2], qh[d0 + 3], odd);
        }
    }
    auto mma = [](float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
        if constexpr (BF) mma16816_bf16(d, a0, a1, a2, a3, b0, b1);
        else mma16816(d, a0, a1, a2, a3, b0, b1);
    };
    const uint32_t sel_lo = odd ? 0x1044u : 0x4410u, sel_hi = odd ? 0x3244u : 0x4432u;
    WState<NT> ws;
    ws.reset();

    const int ntile = t1 > t0 ? (t1 - t0 + 15) / 16 : 0;
    Src src(a, b, h, t1);   // past the end of a tile: rows that exist, weight 0
    uint32_t kr[16], k8[16], va0[8], vb0[8], va1[8], vb1[8];
    auto load_k = [&](int tb) { src.load_k(tb, r, c, kr, k8); };
    auto load_v = [&](int tb) { src.load_v(tb, r, c, va0, vb0, va1, vb1); };
    if (warp < ntile) {
        src.prefetch(t0 + 16 * warp);
        load_k(t0 + 16 * warp);
        load_v(t0 + 16 * warp);
        src.prefetch(t0 + 16 * (warp + kTW));
    }
    for (int i = warp; i < ntile; i += kTW) {
        const int tb = t0 + 16 * i, nval = min(16, t1 - tb);
        src.finish_k(kr, k8);   // restore the stored form (ZipFusion pages) now that it is needed
        float acc[NT][2][4];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int q = 0; q < 2; ++q) acc[j][q][0] = acc[j][q][1] = acc[j][q][2] = acc[j][q][3] = 0.f;
#pragma unroll
        for (int st = 0; st < 8; ++st)
#pragma unroll
            for (int j = 0; j < NT; ++j)
                mma(acc[j][st & 1], kr[2 * st], k8[2 * st], kr[2 * st + 1], k8[2 * st + 1], bq[j][st][0],
                    bq[j][st][1]);
        float s0[NT], s8[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {   // both columns (rounded q and its remainder), both chains
            s0[j] = r < nval ? (acc[j][0][0] + acc[j][0][1]) + (acc[j][1][0] + acc[j][1][1]) : -INFINITY;
            s8[j] = r + 8 < nval ? (acc[j][0][2] + acc[j][0][3]) + (acc[j][1][2] + acc[j][1][3]) : -INFINITY;
        }
        if (i + kTW < ntile) load_k(tb + 16 * kTW);   // the key registers are free
        tile_softmax<NT>(s0, s8, ws);
        src.finish_v(va0, vb0, va1, vb1);
        uint32_t bp[NT][2][2], bl[NT][2][2];   // bl: bf16 remainders of P (BF only)
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const float p0 = ex2(s0[j] - ws.m[j]), p8 = ex2(s8[j] - ws.m[j]);
            ws.l[j] += p0 + p8;
            if constexpr (BF) {
                p_operand_words(pack_part_bf(p0, p0, false), pack_part_bf(p8, p8, false), sel_lo, sel_hi, bp[j]);
                p_operand_words(pack_part_bf(p0, p0, true), pack_part_bf(p8, p8, true), sel_lo, sel_hi, bl[j]);
            } else {
                p_operand(p0, p8, sel_lo, sel_hi, bp[j]);
            }
        }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                mma(ws.o[j][mt], va0[2 * mt], va0[2 * mt + 1], vb0[2 * mt], vb0[2 * mt + 1], bp[j][0][0], bp[j][0][1]);
                mma(ws.o[j][mt], va1[2 * mt], va1[2 * mt + 1], vb1[2 * mt], vb1[2 * mt + 1], bp[j][1][0], bp[j][1][1]);
                if constexpr (BF) {
                    mma(ws.o[j][mt], va0[2 * mt], va0[2 * mt + 1], vb0[2 * mt], vb0[2 * mt + 1], bl[j][0][0],
                        bl[j][0][1]);
                    mma(ws.o[j][mt], va1[2 * mt], va1[2 * mt + 1], vb1[2 * mt], vb1[2 * mt + 1], bl[j][1][0],
                        bl[j][1][1]);
                }
            }
        if (i + kTW < ntile) load_v(tb + 16 * kTW);
        src.prefetch(tb + 32 * kTW);   // the tile after next
    }

    // ---- the warps' states into one (m, l, o~) per head (flat in wo[0])
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int msk = 4; msk < 32; msk <<= 1) ws.l[j] += __shfl_xor_sync(TQ_FULL_MASK, ws.l[j], msk);
        if (r == 0) {
            wm[warp][4 * j + c] = ws.m[j];
            wl[warp][4 * j + c] = ws.l[j];
        }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
            *reinterpret_cast<float4*>(&wo[warp][4 * j + c][16 * r + 4 * mt]) =
                make_float4(ws.o[j][mt][0], ws.o[j][mt][1], ws.o[j][mt][2], ws.o[j][mt][3]);
    }
    __syncthreads();
    float* ot = &wo[0][0][0];
    for (int i = tid; i < GPE * 128; i += kTThr) {
        const int g = i >> 7, d = i & 127;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kTW; ++w) M = fmaxf(M, wm[w][g]);
        float Lt = 0.f, ov = 0.f;
#pragma unroll
        for (int w = 0; w < kTW; ++w) {
            const float wt = (M == -INFINITY || wm[w][g] == -INFINITY) ? 0.f : ex2f(wm[w][g] - M);
            Lt = fmaf(wt, wl[w][g], Lt);
            ov = fmaf(wt, wo[w][g][d], ov);
        }
        ot[i] = ov;   // wo[0][g][d]: this thread alone reads and writes column (g, d)
        if (d == 0) {
            sM[g] = M;
            sL[g] = Lt;
        }
    }
    __syncthreads();
    prefix_finish<GPE, kTThr>(a, ot, sM, sL, &is_last, b, h, s);
}

using PrefixFn = void (*)(PrefixArgs);

// Up to 8 query heads per KV head: the tensor-core kernel (*tc set); more: the
// CUDA-core kernel.
PrefixFn pick_prefix(int G, int dtype, bool* tc) {
    *tc = G <= 8;
    if (G <= 4)
        return dtype == TQ_F16 ? prefix_tile<1, RowSrc<TQ_F16>>
                               : dtype == TQ_BF16 ? prefix_tile<1, RowSrc<TQ_BF16>> : prefix_tile<1, RowSrc<TQ_F32>>;
    if (G <= 8)
        return dtype == TQ_F16 ? prefix_tile<2, RowSrc<TQ_F16>>
                               : dtype == TQ_BF16 ? prefix_tile<2, RowSrc<TQ_BF16>> : prefix_tile<2, RowSrc<TQ_F32>>;
    return prefix_attend<16>;
}

// heads per partial row group: the tensor-core kernel's 4 or 8, the CUDA-core kernel's 16
int gp_of(int G) { return G <= 4 ? 4 : G <= 8 ? 8 : 16; }

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t up256(size_t n) { return (n + 255) & ~(size_t)255; }

// Sections of the tensor-core kernel: 304 CTAs of 8 warps (one wave at two per
// SM, the fp16 four-head kernel; two waves of the others), sections of at least
// 128 tokens (a tile per warp), whole tiles.
int tile_splits(const tq_cache_desc* d, int max_prefix_len) {
    const long long pairs = (long long)d->batch * d->n_kv_heads;
    const long long want = (152LL * 2 + pairs - 1) / pairs;
    long long sp = (max_prefix_len + 127) / 128;
    if (sp > want) sp = want;
    if (sp > TQ_MAX_SPLITS) sp = TQ_MAX_SPLITS;
    return sp < 1 ? 1 : (int)sp;
}

// Sections of the CUDA-core kernel: enough CTAs to fill the GPU about eight
// times over (4-warp CTAs), sections of at least 64 tokens.  Never fewer than
// the tensor-core kernel's, so the workspace sized by these fits both.
int prefix_splits(const tq_cache_desc* d, int max_prefix_len) {
    const long long pairs = (long long)d->batch * d->n_kv_heads;
    const long long want = (152LL * 8 + pairs - 1) / pairs;
    long long sp = (max_prefix_len + 63) / 64;
    if (sp > want) sp = want;
    if (sp > TQ_MAX_SPLITS) sp = TQ_MAX_SPLITS;
    return sp < 1 ? 1 : (int)sp;
}

// Workspace of the packed part (the automatic plan's largest need)
size_t packed_ws_bytes(const tq_cache_desc* d) { return up256(tq_decode_workspace_bytes(d, 128)); }

}  // namespace

extern "C" {

size_t tq_decode_prefix_workspace_bytes(const tq_cache_desc* d, int32_t max_prefix_len) {
    if (!d || d->head_dim != TQ_HEAD_DIM || max_prefix_len < 0) return 0;
    const size_t pairs = (size_t)d->batch * d->n_kv_heads;
    const int sp = prefix_splits(d, max_prefix_len);
    return packed_ws_bytes(d) + up256((size_t)d->batch * d->n_q_heads * sizeof(float)) +
           up256(pairs * sizeof(int32_t)) + pairs * (size_t)sp * gp_of(d->group) * kPartStride * sizeof(float);
}

tq_status tq_decode_attention_prefix(const tq_cache_desc* d, const tq_cache_ptrs* c, const void* q, int32_t q_dtype,
                                     const int32_t* d_seq_lens, int32_t max_seq_len, const void* k_prefix,
                                     const void* v_prefix, int32_t prefix_dtype, int32_t prefix_capacity,
                                     const int32_t* d_prefix_lens, int32_t max_prefix_len, float* out,
                                     void* workspace, size_t workspace_bytes, int32_t* d_status, void* stream) {
    if (!d || d->head_dim != TQ_HEAD_DIM || !q || !out || !d_prefix_lens) return TQ_ERR_INVALID_ARG;
    if (q_dtype != TQ_F32 && q_dtype != TQ_F16 && q_dtype != TQ_BF16) return TQ_ERR_INVALID_ARG;
    if (prefix_dtype != TQ_F32 && prefix_dtype != TQ_F16 && prefix_dtype != TQ_BF16) return TQ_ERR_INVALID_ARG;
    if (max_seq_len < 0 || max_prefix_len < 0 || prefix_capacity < 0 || max_prefix_len > prefix_capacity)
        return TQ_ERR_INVALID_ARG;
    if (max_prefix_len > 0 && (!k_prefix || !v_prefix)) return TQ_ERR_INVALID_ARG;
    const size_t qa = q_dtype == TQ_F32 ? 16 : 8;   // the unquantised rows are read in 16-byte pieces
    if (!aligned_to(k_prefix, 16) || !aligned_to(v_prefix, 16) || !aligned_to(q, qa) || !aligned_to(out, 16))
        return TQ_ERR_INVALID_ARG;
    const size_t need = tq_decode_prefix_workspace_bytes(d, max_prefix_len);
    if (!workspace || workspace_bytes < need || !aligned_to(workspace, 256)) return TQ_ERR_WORKSPACE;
    if (d->batch > 65535 || d->n_kv_heads > 65535) return TQ_ERR_INVALID_ARG;

    char* ws = static_cast<char*>(workspace);
    const size_t pbytes = packed_ws_bytes(d);
    float* lse = reinterpret_cast<float*>(ws + pbytes);
    int32_t* tickets = reinterpret_cast<int32_t*>(ws + pbytes + up256((size_t)d->batch * d->n_q_heads * sizeof(float)));
    float* part = reinterpret_cast<float*>(reinterpret_cast<char*>(tickets) +
                                           up256((size_t)d->batch * d->n_kv_heads * sizeof(int32_t)));
    // the packed part: output and log2-sum-exp
    if (max_seq_len > 0) {
        tq_status st = tq_decode_run(d, c, q, q_dtype, d_seq_lens, max_seq_len, out, ws, pbytes, d_status, stream,
                                     TQ_VMODE_AUTO, 0, lse);
        if (st != TQ_OK) return st;
        if (max_prefix_len == 0) return TQ_OK;   // nothing unquantised to add
    }
    PrefixArgs a;
    a.k = k_prefix;
    a.v = v_prefix;
    a.q = q;
    a.lens = d_prefix_lens;
    a.lse_p = max_seq_len > 0 ? lse : nullptr;
    a.out = out;
    a.ws_part = part;
    a.tickets = tickets;
    a.status = d_status;
    a.k_meta = a.v_meta = nullptr;
    a.B = d->batch;
    a.Hq = d->n_q_heads;
    a.Hkv = d->n_kv_heads;
    a.G = d->group;
    a.cap = prefix_capacity;
    a.max_len = max_prefix_len;
    bool tc = false;
    PrefixFn fn = pick_prefix(d->group, prefix_dtype, &tc);
    a.splits = tc ? tile_splits(d, max_prefix_len) : prefix_splits(d, max_prefix_len);
    a.split_len = (max_prefix_len + a.splits - 1) / a.splits;
    if (tc) a.split_len = (a.split_len + 15) / 16 * 16;   // whole tiles per section
    a.dtype = prefix_dtype;
    a.q_dtype = q_dtype;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.splits, d->n_kv_heads, d->batch);
    cfg.blockDim = dim3(tc ? kTThr : kPThr);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, a) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// ZipFusion pages: store and attention  [ZipFusion]
namespace {

constexpr int kZipPage = 4096;   // bytes of one page's slot (its uncompressed size)

struct ZipStoreArgs {
    const uint16_t* src[2];   // K, V: [B][n_tokens][Hkv][128] bf16
    uint8_t* pool[2];
    uint8_t* meta[2];
    const int32_t* lens;
    int32_t* status;
    int B, Hkv, n_tokens, cap, pages;
};

// One CTA per (page, part, KV head, batch): blockIdx.x = 2 page + part (0 K, 1 V).
// Warp j encodes block j of the page; lane L = 4r + c holds its groups 2L and
// 2L + 1 (the page layout above).  A full page's block compresses when its
// exponents fit [b, b + 15]; a partial page (the sequence's last) is stored raw
// with zeros past the end.
__global__ void __launch_bounds__(128) zip_store(ZipStoreArgs z) {
    __shared__ uint32_t marks[4];
    const int tid = threadIdx.x, lane = tid & 31, j = tid >> 5;
    const int p = blockIdx.x >> 1, part = blockIdx.x & 1, h = blockIdx.y, b = blockIdx.z;
    int L = z.lens[b];
    if (L > z.cap || L > z.n_tokens) {
        if (tid == 0 && p == 0 && part == 0 && h == 0 && z.status) atomicOr(z.status, TQ_DEV_SEQ_OVER_CAPACITY);
        L = min(L, min(z.cap, z.n_tokens));
    }
    if (16 * p >= L) return;   // no token of this page (uniform)
    const bool full = 16 * p + 16 <= L;
    const int r = lane >> 2, c = lane & 3;
    uint32_t w[8];   // groups 2L (w[0..3]) and 2L + 1 (w[4..7]): 16 bf16 values
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        int t, d0;
        if (part == 0) {
            t = r + 8 * u;
            d0 = 32 * c + 8 * j;
        } else {
            t = 8 * (j >> 1) + 2 * c + u;
            d0 = 16 * r + 8 * (j & 1);
        }
        t += 16 * p;
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (t < L) x = __ldg(reinterpret_cast<const uint4*>(z.src[part] + (((size_t)b * z.n_tokens + t) * z.Hkv + h) * 128 + d0));
        w[4 * u] = x.x; w[4 * u + 1] = x.y; w[4 * u + 2] = x.z; w[4 * u + 3] = x.w;
    }
    int emin = 255, emax = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int e = (int)((w[i >> 1] >> (16 * (i & 1) + 7)) & 0xFFu);
        emin = min(emin, e);
        emax = max(emax, e);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        emin = min(emin, __shfl_xor_sync(TQ_FULL_MASK, emin, o));
        emax = max(emax, __shfl_xor_sync(TQ_FULL_MASK, emax, o));
    }
    const int base = emin & ~1;
    const bool comp = full && emax <= base + 15;
    if (lane == 0) marks[j] = comp ? (uint32_t)(base >> 1) : kZipRaw;
    __syncthreads();
    const size_t slot = ((size_t)b * z.Hkv + h) * z.pages + p;
    int off = 0;
    for (int i = 0; i < j; ++i) off += marks[i] == kZipRaw ? 1024 : 768;
    uint8_t* blk = z.pool[part] + slot * kZipPage + off;
    if (comp) {
        uint32_t lo[4] = {0u, 0u, 0u, 0u}, code[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t v = (w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
            lo[i >> 2] |= (v & 0xFFu) << (8 * (i & 3));
            const uint32_t sgn = v >> 15, d = (((v >> 7) & 0xFFu) - (uint32_t)base) >> 1;
            const int q = i >> 3, k = i & 7;
            code[q] |= (k < 4 ? ((sgn << 7) | d) : ((sgn << 6) | (d << 3))) << (8 * (k & 3));
        }
        *reinterpret_cast<uint4*>(blk + 16 * lane) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        *reinterpret_cast<uint2*>(blk + 512 + 8 * lane) = make_uint2(code[0], code[1]);
    } else {
        uint4* d4 = reinterpret_cast<uint4*>(blk + 32 * lane);
        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    if (tid == 0) {
        const uint32_t off256 = (uint32_t)(slot * (kZipPage / 256));
        *reinterpret_cast<uint2*>(z.meta[part] + slot * 8) =
            make_uint2(off256, marks[0] | (marks[1] << 8) | (marks[2] << 16) | (marks[3] << 24));
    }
}

bool zip_shape_ok(int32_t batch, int32_t n_kv_heads, int32_t t_capacity) {
    return batch > 0 && batch <= 65535 && n_kv_heads > 0 && n_kv_heads <= 65535 && t_capacity > 0 &&
           t_capacity % 16 == 0 && (long long)batch * n_kv_heads * (t_capacity / 16) * (kZipPage / 256) < (1LL << 32);
}

int zip_splits(int32_t batch, int32_t n_kv_heads, int32_t max_seq_len) {
    const long long pairs = (long long)batch * n_kv_heads;
    const long long want = (152LL * 2 + pairs - 1) / pairs;
    long long sp = (max_seq_len + 127) / 128;
    if (sp > want) sp = want;
    if (sp > TQ_MAX_SPLITS) sp = TQ_MAX_SPLITS;
    return sp < 1 ? 1 : (int)sp;
}

}  // namespace

extern "C" {

size_t tq_zip_pool_bytes(int32_t batch, int32_t n_kv_heads, int32_t t_capacity) {
    if (!zip_shape_ok(batch, n_kv_heads, t_capacity)) return 0;
    return (size_t)batch * n_kv_heads * (t_capacity / 16) * kZipPage;
}

size_t tq_zip_meta_bytes(int32_t batch, int32_t n_kv_heads, int32_t t_capacity) {
    if (!zip_shape_ok(batch, n_kv_heads, t_capacity)) return 0;
    return (size_t)batch * n_kv_heads * (t_capacity / 16) * 8;
}

tq_status tq_zip_store(const void* K, const void* V, int32_t batch, int32_t n_kv_heads, int32_t n_tokens,
                       int32_t t_capacity, const int32_t* d_lens, void* k_pool, void* v_pool, void* k_meta,
                       void* v_meta, int32_t* d_status, void* stream) {
    if (!K || !V || !d_lens || !k_pool || !v_pool || !k_meta || !v_meta || n_tokens < 1) return TQ_ERR_INVALID_ARG;
    if (!zip_shape_ok(batch, n_kv_heads, t_capacity)) return TQ_ERR_INVALID_ARG;
    if (!aligned_to(K, 16) || !aligned_to(V, 16) || !aligned_to(k_pool, 256) || !aligned_to(v_pool, 256) ||
        !aligned_to(k_meta, 8) || !aligned_to(v_meta, 8))
        return TQ_ERR_INVALID_ARG;
    ZipStoreArgs z;
    z.src[0] = static_cast<const uint16_t*>(K);
    z.src[1] = static_cast<const uint16_t*>(V);
    z.pool[0] = static_cast<uint8_t*>(k_pool);
    z.pool[1] = static_cast<uint8_t*>(v_pool);
    z.meta[0] = static_cast<uint8_t*>(k_meta);
    z.meta[1] = static_cast<uint8_t*>(v_meta);
    z.lens = d_lens;
    z.status = d_status;
    z.B = batch;
    z.Hkv = n_kv_heads;
    z.n_tokens = n_tokens;
    z.cap = t_capacity;
    z.pages = t_capacity / 16;
    const int pages_used = (min(n_tokens, t_capacity) + 15) / 16;
    dim3 grid(2 * pages_used, n_kv_heads, batch);
    zip_store<<<grid, 128, 0, (cudaStream_t)stream>>>(z);
    return cudaPeekAtLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

size_t tq_zip_workspace_bytes(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads, int32_t max_seq_len) {
    if (batch < 1 || n_kv_heads < 1 || n_q_heads < 1 || n_q_heads % n_kv_heads || max_seq_len < 0) return 0;
    const int G = n_q_heads / n_kv_heads;
    if (G > 8) return 0;
    const size_t pairs = (size_t)batch * n_kv_heads;
    const int sp = zip_splits(batch, n_kv_heads, max_seq_len);
    return up256(pairs * sizeof(int32_t)) + pairs * (size_t)sp * gp_of(G) * kPartStride * sizeof(float);
}

tq_status tq_zip_decode_attention(const void* q, int32_t q_dtype, int32_t batch, int32_t n_q_heads,
                                  int32_t n_kv_heads, int32_t t_capacity, const void* k_pool, const void* v_pool,
                                  const void* k_meta, const void* v_meta, const int32_t* d_seq_lens,
                                  int32_t max_seq_len, float* out, void* workspace, size_t workspace_bytes,
                                  int32_t* d_status, void* stream) {
    if (!q || !k_pool || !v_pool || !k_meta || !v_meta || !d_seq_lens || !out) return TQ_ERR_INVALID_ARG;
    if (q_dtype != TQ_F32 && q_dtype != TQ_F16 && q_dtype != TQ_BF16) return TQ_ERR_INVALID_ARG;
    if (!zip_shape_ok(batch, n_kv_heads, t_capacity) || n_q_heads < 1 || n_q_heads % n_kv_heads)
        return TQ_ERR_INVALID_ARG;
    if (max_seq_len < 1 || max_seq_len > t_capacity) return TQ_ERR_INVALID_ARG;
    if (n_q_heads / n_kv_heads > 8) return TQ_ERR_UNSUPPORTED;
    const size_t qa = q_dtype == TQ_F32 ? 16 : 8;
    if (!aligned_to(q, qa) || !aligned_to(out, 16) || !aligned_to(k_pool, 256) || !aligned_to(v_pool, 256) ||
        !aligned_to(k_meta, 8) || !aligned_to(v_meta, 8))
        return TQ_ERR_INVALID_ARG;
    const size_t need = tq_zip_workspace_bytes(batch, n_q_heads, n_kv_heads, max_seq_len);
    if (!workspace || workspace_bytes < need || !aligned_to(workspace, 256)) return TQ_ERR_WORKSPACE;
    PrefixArgs a;
    a.k = k_pool;
    a.v = v_pool;
    a.q = q;
    a.lens = d_seq_lens;
    a.lse_p = nullptr;   // no second part: the merge leaves the pages' attention as is
    a.out = out;
    a.tickets = static_cast<int32_t*>(workspace);
    a.ws_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                         up256((size_t)batch * n_kv_heads * sizeof(int32_t)));
    a.status = d_status;
    a.k_meta = static_cast<const uint8_t*>(k_meta);
    a.v_meta = static_cast<const uint8_t*>(v_meta);
    a.B = batch;
    a.Hq = n_q_heads;
    a.Hkv = n_kv_heads;
    a.G = n_q_heads / n_kv_heads;
    a.cap = t_capacity;
    a.max_len = max_seq_len;
    a.splits = zip_splits(batch, n_kv_heads, max_seq_len);
    a.split_len = ((max_seq_len + a.splits - 1) / a.splits + 15) / 16 * 16;   // whole pages per section
    a.dtype = TQ_BF16;
    a.q_dtype = q_dtype;
    PrefixFn fn = a.G <= 4 ? prefix_tile<1, ZipSrc> : prefix_tile<2, ZipSrc>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.splits, n_kv_heads, batch);
    cfg.blockDim = dim3(kTThr);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, a) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // extern "C"
