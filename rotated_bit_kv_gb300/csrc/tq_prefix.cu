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
// bf16 and fp32 inputs are rounded to fp16 on load (values must lie in fp16 range).
constexpr int kTW = 8;
constexpr int kTThr = kTW * 32;

__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t x) {
    return pack_h2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}

// N fp16 words (2N elements) of the input from element `elem` (16-byte aligned)
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
        if constexpr (DT == TQ_BF16) {
#pragma unroll
            for (int i = 0; i < N; ++i) w[i] = bf2_to_h2(w[i]);
        }
    }
}

template <int NT, int DT>
__global__ void __launch_bounds__(kTThr, (NT == 1 && DT == TQ_F16) ? 2 : 1) prefix_tile(PrefixArgs a) {
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
    const int r = lane >> 2, c = lane & 3;
    const bool odd = r & 1;
    uint32_t bq[NT][8][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const float* qh = qf[4 * j + (r >> 1)];
#pragma unroll
        for (int st = 0; st < 8; ++st) {
            const int d0 = 2 * (16 * c + 2 * st);
            bq[j][st][0] = pack_part(qh[d0], qh[d0 + 1], odd);
            bq[j][st][1] = pack_part(qh[d0 + 2], qh[d0 + 3], odd);
        }
    }
    const uint32_t sel_lo = odd ? 0x1044u : 0x4410u, sel_hi = odd ? 0x3244u : 0x4432u;
    WState<NT> ws;
    ws.reset();

    const int ntile = t1 > t0 ? (t1 - t0 + 15) / 16 : 0;
    const size_t row = (size_t)a.Hkv * 128;
    const size_t base = ((size_t)b * a.cap * a.Hkv + h) * 128;
    auto tok = [&](int tb, int i) { return (size_t)min(tb + i, t1 - 1); };   // past the end: a valid row, weight 0
    uint32_t kr[16], k8[16], va0[8], vb0[8], va1[8], vb1[8];
    auto load_k = [&](int tb) {
        load_words<DT>(a.k, base + tok(tb, r) * row + 32 * c, kr);
        load_words<DT>(a.k, base + tok(tb, r + 8) * row + 32 * c, k8);
    };
    auto load_v = [&](int tb) {
        load_words<DT>(a.v, base + tok(tb, 2 * c) * row + 16 * r, va0);
        load_words<DT>(a.v, base + tok(tb, 2 * c + 1) * row + 16 * r, vb0);
        load_words<DT>(a.v, base + tok(tb, 2 * c + 8) * row + 16 * r, va1);
        load_words<DT>(a.v, base + tok(tb, 2 * c + 9) * row + 16 * r, vb1);
    };
    if (warp < ntile) {
        load_k(t0 + 16 * warp);
        load_v(t0 + 16 * warp);
    }
    for (int i = warp; i < ntile; i += kTW) {
        const int tb = t0 + 16 * i, nval = min(16, t1 - tb);
        float acc[NT][2][4];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int q = 0; q < 2; ++q) acc[j][q][0] = acc[j][q][1] = acc[j][q][2] = acc[j][q][3] = 0.f;
#pragma unroll
        for (int st = 0; st < 8; ++st)
#pragma unroll
            for (int j = 0; j < NT; ++j)
                mma16816(acc[j][st & 1], kr[2 * st], k8[2 * st], kr[2 * st + 1], k8[2 * st + 1], bq[j][st][0],
                         bq[j][st][1]);
        float s0[NT], s8[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {   // both columns (rounded q and its remainder), both chains
            s0[j] = r < nval ? (acc[j][0][0] + acc[j][0][1]) + (acc[j][1][0] + acc[j][1][1]) : -INFINITY;
            s8[j] = r + 8 < nval ? (acc[j][0][2] + acc[j][0][3]) + (acc[j][1][2] + acc[j][1][3]) : -INFINITY;
        }
        if (i + kTW < ntile) load_k(tb + 16 * kTW);   // the key registers are free
        tile_softmax<NT>(s0, s8, ws);
        uint32_t bp[NT][2][2];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const float p0 = ex2(s0[j] - ws.m[j]), p8 = ex2(s8[j] - ws.m[j]);
            ws.l[j] += p0 + p8;
            p_operand(p0, p8, sel_lo, sel_hi, bp[j]);
        }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                mma16816(ws.o[j][mt], va0[2 * mt], va0[2 * mt + 1], vb0[2 * mt], vb0[2 * mt + 1], bp[j][0][0],
                         bp[j][0][1]);
                mma16816(ws.o[j][mt], va1[2 * mt], va1[2 * mt + 1], vb1[2 * mt], vb1[2 * mt + 1], bp[j][1][0],
                         bp[j][1][1]);
            }
        if (i + kTW < ntile) load_v(tb + 16 * kTW);
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
    if (G <= 4) return dtype == TQ_F16 ? prefix_tile<1, TQ_F16> : dtype == TQ_BF16 ? prefix_tile<1, TQ_BF16>
                                                                                     : prefix_tile<1, TQ_F32>;
    if (G <= 8) return dtype == TQ_F16 ? prefix_tile<2, TQ_F16> : dtype == TQ_BF16 ? prefix_tile<2, TQ_BF16>
                                                                                     : prefix_tile<2, TQ_F32>;
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
