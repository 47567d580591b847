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

    // ---- sections: publish, the last CTA merges (normalised into ot, (M, L) in sM, sL)
    if (a.splits > 1) {
        float* part = a.ws_part + ((((size_t)b * a.Hkv + h) * a.splits + s) * GP) * kPartStride;
        for (int i = tid; i < GP * 128; i += kPThr) part[(i >> 7) * kPartStride + (i & 127)] = ot[i];
        if (tid < GP) {
            part[tid * kPartStride + 128] = sM[tid];
            part[tid * kPartStride + 129] = sL[tid];
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const int ticket = atomicAdd(a.tickets + (size_t)b * a.Hkv + h, 1);
            is_last = ticket == a.splits - 1;
        }
        __syncthreads();
        if (!is_last) return;
        __threadfence();
        merge_parts<GP, kPThr>(a.ws_part + (((size_t)b * a.Hkv + h) * a.splits * GP) * kPartStride, a.splits,
                               reinterpret_cast<float(*)[128]>(ot), sM, sL);
        if (tid == 0) a.tickets[(size_t)b * a.Hkv + h] = 0;   // ready for the next call
        __syncthreads();
    } else {
        for (int i = tid; i < GP * 128; i += kPThr) {
            const int g = i >> 7;
            ot[i] = sL[g] > 0.f ? ot[i] / sL[g] : 0.f;
        }
        __syncthreads();
    }

    // ---- merge with the packed part: o = (w_p o_p + w_f L_f o_f) / (w_p + w_f L_f)
    for (int i = tid; i < a.G * 128; i += kPThr) {
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

using PrefixFn = void (*)(PrefixArgs);

PrefixFn pick_prefix(int G) {
    if (G <= 1) return prefix_attend<1>;
    if (G <= 4) return prefix_attend<4>;
    if (G <= 8) return prefix_attend<8>;
    return prefix_attend<16>;
}

int gp_of(int G) { return G <= 1 ? 1 : G <= 4 ? 4 : G <= 8 ? 8 : 16; }

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t up256(size_t n) { return (n + 255) & ~(size_t)255; }

// Sections of the unquantised tokens: enough CTAs to fill the GPU about eight
// times over (4-warp CTAs), sections of at least 64 tokens.
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
    const size_t pa = prefix_dtype == TQ_F32 ? 16 : 8, qa = q_dtype == TQ_F32 ? 16 : 8;
    if (!aligned_to(k_prefix, pa) || !aligned_to(v_prefix, pa) || !aligned_to(q, qa) || !aligned_to(out, 16))
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
    a.splits = prefix_splits(d, max_prefix_len);
    a.split_len = (max_prefix_len + a.splits - 1) / a.splits;
    a.dtype = prefix_dtype;
    a.q_dtype = q_dtype;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.splits, d->n_kv_heads, d->batch);
    cfg.blockDim = dim3(kPThr);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pick_prefix(d->group), a) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // extern "C"
