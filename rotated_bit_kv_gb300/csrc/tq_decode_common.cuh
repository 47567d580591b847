// Device code shared by the decode kernels (CUDA-core and tensor-core variants):
// launch arguments, record/norm loads, q rotation prologue, sequence-length
// clamping and the split epilogue (log-sum-exp merge by the last CTA of a
// (batch, KV head), then one inverse rotation).  Included by one translation
// unit per kernel family; everything here has internal linkage.
#pragma once
#include "tq_device.cuh"

namespace tq {
// Launch arguments of every decode kernel.
struct DecodeArgs {
    const uint8_t* k_codes;
    const void* k_norms;
    const uint8_t* v_codes;
    const void* v_norms;
    const tq_head_params* params;
    const float* kmat;
    const void* q;
    const int32_t* seq_lens;
    float* out;
    float* lse;         // optional [B][Hq]: log2-sum-exp of each head's scores (log2 units), or null
    float* ws_part;
    int32_t* tickets;
    int32_t* status;
    // Tcap: positions per (batch, KV head) in the arrays (t_alloc); t_cap: the
    // logical capacity (t_capacity)
    int B, Hq, Hkv, G, Tcap, t_cap, max_seq, n_splits, split_len, q_dtype, norm_f16, rot, k_mixed;
    uint32_t fold_mul;   // 1 << 20 (a runtime operand keeps the selector fold on the FMA pipe)
};
}  // namespace tq

namespace {

constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kInvSqrtD = 0.08838834764831845f;   // 1/sqrt(128)
constexpr int kPartStride = 132;                      // 128 (o~) + m + l, 16-byte rows
constexpr float kQjlScale = 0.009791516697777346f;    // sqrt(pi/2) / 128 (two-stage keys)

using DecodeArgs = tq::DecodeArgs;

template <int F> struct Fmt {
    static constexpr bool three = (F == TQ_FMT_ONE3 || F == TQ_FMT_BLK3);
    // two-stage keys: `mse_words` words of 1-bit codes, then 4 words of signs
    static constexpr bool qjl = (F == TQ_FMT_QJ1 || F == TQ_FMT_QJ2);
    static constexpr int mse_words = F == TQ_FMT_QJ2 ? 4 : 0;
    // mixed-rate keys in tight records (codes at their groups' widths)
    static constexpr bool tight = (F == TQ_FMT_MXT2 || F == TQ_FMT_MXT3);
    static constexpr int bytes = qjl ? 4 * (mse_words + 4) : tight ? (F == TQ_FMT_MXT2 ? 32 : 48) : three ? 48 : 64;
    static constexpr int words = bytes / 4;
    static constexpr int nslots = qjl ? 2 : (F == TQ_FMT_ONE3 || F == TQ_FMT_ONE4) ? 1 : 4;
    static constexpr bool blk = (F == TQ_FMT_BLK3 || F == TQ_FMT_BLK4);
    static constexpr bool mix = (F == TQ_FMT_MIX4 || tight);
};

// index of code c (compile-time in unrolled loops) from a record in registers
template <bool THREE>
__device__ __forceinline__ uint32_t code_at(const uint32_t* w, int c) {
    if (THREE) {
        const int bit = 3 * c, wi = bit >> 5, sh = bit & 31;
        if (sh <= 29) return (w[wi] >> sh) & 7u;
        return __funnelshift_r(w[wi], w[wi + 1], sh) & 7u;
    }
    return (w[c >> 3] >> (4 * (c & 7))) & 15u;
}

template <int F>
__device__ __forceinline__ void load_record(const uint8_t* base, size_t tok, uint32_t* w) {
    const uint4* p = reinterpret_cast<const uint4*>(base + tok * Fmt<F>::bytes);
#pragma unroll
    for (int i = 0; i < Fmt<F>::words / 4; ++i) {
        uint4 u = __ldg(p + i);
        w[4 * i] = u.x; w[4 * i + 1] = u.y; w[4 * i + 2] = u.z; w[4 * i + 3] = u.w;
    }
}

template <int F>
__device__ __forceinline__ void load_norms(const void* base, size_t tok, int norm_f16, float* n) {
    if (Fmt<F>::nslots == 1) {
        n[0] = tq::load_norm(base, tok, norm_f16);
    } else if (Fmt<F>::nslots == 2) {
        if (norm_f16) {
            const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(static_cast<const __half*>(base) + tok * 2));
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u));
            n[0] = a.x; n[1] = a.y;
        } else {
            const float2 f = __ldg(reinterpret_cast<const float2*>(static_cast<const float*>(base) + tok * 2));
            n[0] = f.x; n[1] = f.y;
        }
    } else if (norm_f16) {
        uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const __half*>(base) + tok * 4));
        float2 a = __half22float2(*reinterpret_cast<__half2*>(&u.x));
        float2 b = __half22float2(*reinterpret_cast<__half2*>(&u.y));
        n[0] = a.x; n[1] = a.y; n[2] = b.x; n[3] = b.y;
    } else {
        float4 f = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + tok * 4));
        n[0] = f.x; n[1] = f.y; n[2] = f.z; n[3] = f.w;
    }
}

template <int GP>
__device__ __forceinline__ void load_row(const float* row, float* q) {
    if (GP % 4 == 0) {
#pragma unroll
        for (int i = 0; i < GP / 4; ++i) {
            float4 v = reinterpret_cast<const float4*>(row)[i];
            q[4 * i] = v.x; q[4 * i + 1] = v.y; q[4 * i + 2] = v.z; q[4 * i + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < GP; ++i) q[i] = row[i];
    }
}

// s_g = sum over segments of n_seg * sum_c q~_g[c] C_seg[idx_c]   (log2 units:
// q~ already carries log2(e) / sqrt(d)).  Two-stage keys [TQ-MNN §2.4]:
// s_g = n <q~_g, C[idx]> + n rho <u_g, 2 sign - 1> with u_g = S q~_g sqrt(pi/2) / d
// (in ut, same units); nrm = (n, n rho).
//
// Tight mixed-rate records: the record goes to this thread's staging words
// (kst[i * kstride]) and the groups are walked in ascending width, the code at
// position p read from bit offset sum_{p' < p} b_p' (funnel shift of two staged
// words); kseg_start holds the groups' first positions.
template <int GP, int KF>
__device__ __forceinline__ void qk_token(const uint32_t* rec, const float* nrm, const float (*qt)[GP],
                                         const float (*ut)[GP], const float (*kcb)[16], const uint8_t* kseg_of,
                                         float* sc, uint32_t* kst = nullptr, int kstride = 0,
                                         const int* kseg_start = nullptr) {
    using K = Fmt<KF>;
#pragma unroll
    for (int g = 0; g < GP; ++g) sc[g] = 0.f;
    if constexpr (K::tight) {
#pragma unroll
        for (int i = 0; i < K::words; ++i) kst[i * kstride] = rec[i];
        int off = 0;
#pragma unroll 1
        for (int s = 0; s < 4; ++s) {
            const int p1 = kseg_start[s + 1];
            const uint32_t mask = (2u << s) - 1u;   // width s + 1
            float part[GP];
#pragma unroll
            for (int g = 0; g < GP; ++g) part[g] = 0.f;
#pragma unroll 2
            for (int p = kseg_start[s]; p < p1; ++p, off += s + 1) {
                const int wi = off >> 5;
                const uint32_t lo = kst[wi * kstride];
                const uint32_t hi = kst[min(wi + 1, K::words - 1) * kstride];
                const float v = kcb[s][__funnelshift_r(lo, hi, off & 31) & mask];
                float q[GP];
                load_row<GP>(qt[p], q);
#pragma unroll
                for (int g = 0; g < GP; ++g) part[g] = fmaf(v, q[g], part[g]);
            }
#pragma unroll
            for (int g = 0; g < GP; ++g) sc[g] = fmaf(nrm[s], part[g], sc[g]);
        }
    } else if constexpr (K::qjl) {
        float ms[GP], sg[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) { ms[g] = 0.f; sg[g] = 0.f; }
        if constexpr (K::mse_words > 0) {
            const float c0 = kcb[0][0], c1 = kcb[0][1];
#pragma unroll
            for (int c = 0; c < 128; ++c) {
                const float v = ((rec[c >> 5] >> (c & 31)) & 1u) ? c1 : c0;
                float q[GP];
                load_row<GP>(qt[c], q);
#pragma unroll
                for (int g = 0; g < GP; ++g) ms[g] = fmaf(v, q[g], ms[g]);
            }
        }
#pragma unroll
        for (int j = 0; j < 128; ++j) {
            const float sgn = ((rec[K::mse_words + (j >> 5)] >> (j & 31)) & 1u) ? 1.f : -1.f;
            float u[GP];
            load_row<GP>(ut[j], u);
#pragma unroll
            for (int g = 0; g < GP; ++g) sg[g] = fmaf(sgn, u[g], sg[g]);
        }
#pragma unroll
        for (int g = 0; g < GP; ++g) sc[g] = fmaf(nrm[0], ms[g], nrm[1] * sg[g]);
    } else if (K::mix) {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
            const int s = kseg_of[c];
            float n = nrm[0];
            n = s == 1 ? nrm[1] : n;
            n = s == 2 ? nrm[2] : n;
            n = s == 3 ? nrm[3] : n;
            const float v = kcb[s][code_at<false>(rec, c)] * n;
            float q[GP];
            load_row<GP>(qt[c], q);
#pragma unroll
            for (int g = 0; g < GP; ++g) sc[g] = fmaf(v, q[g], sc[g]);
        }
    } else {
        constexpr int nseg = K::blk ? 4 : 1;
        constexpr int len = 128 / nseg;
#pragma unroll
        for (int s = 0; s < nseg; ++s) {
            float part[GP];
#pragma unroll
            for (int g = 0; g < GP; ++g) part[g] = 0.f;
#pragma unroll
            for (int cc = 0; cc < len; ++cc) {
                const int c = s * len + cc;
                const float v = kcb[s][code_at<K::three>(rec, c)];
                float q[GP];
                load_row<GP>(qt[c], q);
#pragma unroll
                for (int g = 0; g < GP; ++g) part[g] = fmaf(v, q[g], part[g]);
            }
#pragma unroll
            for (int g = 0; g < GP; ++g) sc[g] = fmaf(nrm[s], part[g], sc[g]);
        }
    }
}

template <int GP, int KF, int VF>
struct Smem {
    alignas(16) float qt[128][GP];
    alignas(16) float kcb[4][16];
    alignas(16) float vcb[4][16];
    alignas(16) float xs[4][128];     // per-warp staging for the dense key rotation of q
    alignas(16) float red[4][GP];
    alignas(16) float red2[4][GP];
    alignas(16) uint8_t kseg_of[128];
    alignas(16) float ut[Fmt<KF>::qjl ? 128 : 1][GP];   // two-stage keys: S q~ sqrt(pi/2) / d
    int kseg_start[5];                                  // mixed-rate keys: the groups' first positions
    int is_last;
};

// Prologue shared by both modes: codebooks, q~ = R_K q (scaled to log2 units).
template <int GP, int KF, int VF>
__device__ __forceinline__ void prologue(const DecodeArgs& a, const tq_head_params& P, Smem<GP, KF, VF>& S,
                                         int b, int h) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < 64) {
        S.kcb[tid >> 4][tid & 15] = P.k_cent[tid >> 4][tid & 15];
        S.vcb[tid >> 4][tid & 15] = P.v_cent[tid >> 4][tid & 15];
    }
    if (Fmt<KF>::mix) {
        int s = 0;
        while (s < 3 && tid >= P.k_seg_start[s + 1]) ++s;
        S.kseg_of[tid] = (uint8_t)s;
        if (tid < 5) S.kseg_start[tid] = P.k_seg_start[tid];
    }
    for (int g = warp; g < GP; g += 4) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (g < a.G) {
            const size_t elem = ((size_t)b * a.Hq + (size_t)h * a.G + g) * 128 + 4 * lane;
            tq::load4(a.q, elem, a.q_dtype, v);
            if (Fmt<KF>::mix) {
                float* xs = S.xs[warp];
#pragma unroll
                for (int i = 0; i < 4; ++i) xs[4 * lane + i] = v[i];
                __syncwarp();
                tq::rotate_forward_dense(P, a.kmat + (size_t)h * 128 * 128, xs, v);
                __syncwarp();
            } else {
                tq::rotate_forward(a.rot, P, v);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) S.qt[4 * lane + i][g] = v[i] * (kLog2e * kInvSqrtD);
        if constexpr (Fmt<KF>::qjl) {
            // u = S q~, once per query head [TQ-MNN §2.4]; the projection sits
            // where mixed-rate keys keep their matrices
            float* xs = S.xs[warp];
#pragma unroll
            for (int i = 0; i < 4; ++i) xs[4 * lane + i] = v[i];
            __syncwarp();
            float u[4];
            tq::dense_rows_t(a.kmat + (size_t)h * 128 * 128, xs, u);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) S.ut[4 * lane + i][g] = u[i] * (kLog2e * kInvSqrtD * kQjlScale);
        }
    }
}

// Clamp the sequence length and flag what was clamped.
__device__ __forceinline__ int clamp_len(const DecodeArgs& a, int b) {
    int L = a.seq_lens[b];
    int flags = 0;
    if (L > a.t_cap) { flags |= TQ_DEV_SEQ_OVER_CAPACITY; L = a.t_cap; }
    if (L > a.max_seq) { flags |= TQ_DEV_SEQ_OVER_MAX; L = a.max_seq; }
    if (L < 0) L = 0;
    if (flags && a.status && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(a.status, flags);  // once per batch
    return L;
}

// Log-sum-exp merge of `parts` published partials (rows [part t][head g] of
// kPartStride floats: o~[128], m, l) into ot[g][0..127], normalised  [Block-GTQ].
// A warp per head finds M_g = max_t m_t and L_g = sum_t 2^(m_t - M_g) l_t; then each
// thread accumulates four coordinates of one head over the parts, its loads
// independent of each other so that their latencies overlap.  Empty parts
// (m = -inf) weigh 0; a pair with no tokens gives 0.  NTHR threads; M_g and L_g
// stay in sM, sL (shared).
template <int GP, int NTHR>
__device__ __forceinline__ void merge_parts(const float* base, int parts, float (*ot)[128], float* sM, float* sL) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int g = warp; g < GP; g += NTHR / 32) {
        float M = -INFINITY;
        for (int t = lane; t < parts; t += 32) M = fmaxf(M, __ldcg(base + ((size_t)t * GP + g) * kPartStride + 128));
#pragma unroll
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(TQ_FULL_MASK, M, o));
        float L = 0.f;
        for (int t = lane; t < parts; t += 32) {
            const float* pr = base + ((size_t)t * GP + g) * kPartStride;
            const float mt = __ldcg(pr + 128);
            L = fmaf(mt == -INFINITY ? 0.f : exp2f(mt - M), __ldcg(pr + 129), L);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(TQ_FULL_MASK, L, o);
        if (lane == 0) {
            sM[g] = M;
            sL[g] = L;
        }
    }
    __syncthreads();
    for (int i = tid; i < GP * 32; i += NTHR) {
        const int g = i >> 5, d4 = i & 31;
        const float M = sM[g];
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int t = 0; t < parts; ++t) {
            const float* pr = base + ((size_t)t * GP + g) * kPartStride;
            const float mt = __ldcg(pr + 128);
            const float4 v = __ldcg(reinterpret_cast<const float4*>(pr) + d4);
            const float w = mt == -INFINITY ? 0.f : exp2f(mt - M);
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
        const float L = sL[g];
        const float inv = L > 0.f ? 1.f / L : 0.f;
        ot[g][4 * d4] = acc.x * inv;
        ot[g][4 * d4 + 1] = acc.y * inv;
        ot[g][4 * d4 + 2] = acc.z * inv;
        ot[g][4 * d4 + 3] = acc.w * inv;
    }
}

// Epilogue: `ot[g][c]` holds this CTA's unnormalised o~, (m[g], l[g]) its
// softmax state (identical in every thread).  Either finalise directly (one
// split) or publish the partial and let the last CTA merge; the finalising CTA
// also writes each head's log2-sum-exp when asked (a.lse).
template <int GP>
__device__ void epilogue(const DecodeArgs& a, const tq_head_params& P, float (*ot)[128], const float* m,
                         const float* l, int* is_last, int b, int h, int s) {
    __shared__ float sM[GP], sL[GP];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (a.n_splits > 1) {
        float* part = a.ws_part + ((((size_t)b * a.Hkv + h) * a.n_splits + s) * GP) * kPartStride;
        for (int i = tid; i < GP * 128; i += kThreads) part[(i >> 7) * kPartStride + (i & 127)] = ot[i >> 7][i & 127];
        if (tid < GP) {
            part[tid * kPartStride + 128] = m[tid];
            part[tid * kPartStride + 129] = l[tid];
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const int ticket = atomicAdd(a.tickets + (size_t)b * a.Hkv + h, 1);
            *is_last = ticket == a.n_splits - 1;
        }
        __syncthreads();
        if (!*is_last) return;
        __threadfence();
        // log-sum-exp merge over the splits  [Block-GTQ]
        merge_parts<GP, kThreads>(a.ws_part + (((size_t)b * a.Hkv + h) * a.n_splits * GP) * kPartStride,
                                  a.n_splits, ot, sM, sL);
        if (tid == 0) a.tickets[(size_t)b * a.Hkv + h] = 0;   // ready for the next call
        __syncthreads();
    } else {
        for (int i = tid; i < GP * 128; i += kThreads) {
            const int g = i >> 7;
            ot[g][i & 127] = l[g] > 0.f ? ot[g][i & 127] / l[g] : 0.f;
        }
        if (tid < GP) {
            sM[tid] = m[tid];
            sL[tid] = l[tid];
        }
        __syncthreads();
    }
    if (a.lse && tid < a.G)   // the softmax mass, for a later merge with other keys
        a.lse[(size_t)b * a.Hq + (size_t)h * a.G + tid] = sL[tid] > 0.f ? sM[tid] + log2f(sL[tid]) : -INFINITY;
    // o = R_V^T o~, once per query head  [RotaryQuant Key design 3, Kernel D]
    for (int g = warp; g < a.G; g += 4) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = ot[g][4 * lane + i];
        tq::rotate_inverse(a.rot, P, v);
        float4* o4 = reinterpret_cast<float4*>(a.out + ((size_t)b * a.Hq + (size_t)h * a.G + g) * 128) + lane;
        *o4 = make_float4(v[0], v[1], v[2], v[3]);
    }
}

}  // namespace

// Tensor-core decode on the tile layout (tq_decode_tile.cu).  Supported: every
// TQ_LAYOUT_TILE16 cache.
bool tq_decode_tc_supported(const tq_cache_desc* d);
// partial slots the workspace must hold, and the automatic grid (CTAs; 0 when the
// occupancy cannot be read)
int tq_decode_tc_sk_slots(const tq_cache_desc* d);
int tq_decode_tc_sk_grid(const tq_cache_desc* d, int max_seq_len);
int tq_decode_tc_max_grid();
cudaError_t tq_decode_tc_launch(const tq_cache_desc* d, const tq::DecodeArgs& a, int grid, cudaStream_t stream);
