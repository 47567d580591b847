// CUDA-core decode kernels on the natural layout (one record per token):
// dimension-parallel (decode_dp) and token-parallel (decode_tp) V accumulation
// [RotaryQuant, Key design 3], templated on the query heads per KV head (padded:
// 1, 4, 8, 16) and the key and value code formats.  Included by the translation
// units that instantiate them (tq_decode.cu: one-stage formats;
// tq_decode_two_stage.cu: two-stage keys [TQ-MNN §2.4]); everything here has
// internal linkage.
//
// Grid: (split, KV head, batch); 128 threads.  Each CTA rotates the G query
// heads of its KV head into shared memory, streams its section of the cache,
// and leaves a partial (m, l, o~) per query head.  The last CTA of a (batch,
// KV head) to finish -- found with an atomic ticket, no spinning -- merges the
// sections and applies R_V^T.
#pragma once
#include "tq_decode_common.cuh"

namespace {
// ---------------------------------------------------------------------------
// Dimension-parallel V accumulation: per tile of 128 tokens, thread t computes
// the logits of token t (token parallel QK); the tile's V codes are staged in
// shared memory and thread c accumulates dimension c of o~ for every head.
template <int GP, int KF, int VF>
struct SmemDP {
    Smem<GP, KF, VF> s;
    alignas(16) float psm[128][GP];
    alignas(16) float vns[128][4];
    alignas(16) uint32_t vtile[128 * Fmt<VF>::words];
    alignas(16) float ot[GP][128];
};

template <int GP, int KF, int VF>
__global__ void __launch_bounds__(kThreads) decode_dp(DecodeArgs a) {
    using KFm = Fmt<KF>;
    using VFm = Fmt<VF>;
    static_assert(!KFm::tight || KFm::words <= VFm::words, "tight key records are staged in the V tile");
    __shared__ __align__(16) SmemDP<GP, KF, VF> S;
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const tq_head_params& P = a.params[h];
    const int L = clamp_len(a, b);
    const int t0 = s * a.split_len;
    const int t1 = min(t0 + a.split_len, L);
    prologue<GP, KF, VF>(a, P, S.s, b, h);
    __syncthreads();

    const size_t head_tok = ((size_t)b * a.Hkv + h) * a.Tcap;
    float m_run[GP], l_part[GP], acc[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) { m_run[g] = -INFINITY; l_part[g] = 0.f; acc[g] = 0.f; }
    const int c = tid;
    const int vseg = VFm::blk ? (c >> 5) : 0;
    const int vbit = VFm::three ? 3 * c : 4 * c;
    const int vwi = vbit >> 5, vsh = vbit & 31;
    const int vwi1 = vwi + 1 < VFm::words ? vwi + 1 : vwi;

    for (int tile = t0; tile < t1; tile += kThreads) {
        const int nvalid = min(kThreads, t1 - tile);
        const int j = tile + tid;
        const bool valid = tid < nvalid;
        float sc[GP];
        float vn[4] = {1.f, 1.f, 1.f, 1.f};
        if (valid) {
            uint32_t rec[KFm::words];
            float kn[4];
            load_record<KF>(a.k_codes, head_tok + j, rec);
            load_norms<KF>(a.k_norms, head_tok + j, a.norm_f16, kn);
            // tight key records are staged in the V tile's words (column tid),
            // which the V copy below overwrites after the barrier
            qk_token<GP, KF>(rec, kn, S.s.qt, S.s.ut, S.s.kcb, S.s.kseg_of, sc, S.vtile + tid, kThreads,
                             S.s.kseg_start);
            load_norms<VF>(a.v_norms, head_tok + j, a.norm_f16, vn);
        } else {
#pragma unroll
            for (int g = 0; g < GP; ++g) sc[g] = -INFINITY;
        }
        if constexpr (KFm::tight) __syncthreads();
        // stage the tile's V codes (contiguous records), 16-byte copies
        {
            const uint4* src = reinterpret_cast<const uint4*>(a.v_codes + (head_tok + tile) * VFm::bytes);
            uint4* dst = reinterpret_cast<uint4*>(S.vtile);
            const int n16 = nvalid * (VFm::bytes / 16);
            for (int i = tid; i < n16; i += kThreads) dst[i] = __ldg(src + i);
        }
        // tile max per head
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            const float wm = tq::warp_max(sc[g]);
            if (lane == 0) S.s.red[warp][g] = wm;
        }
        __syncthreads();
        float corr[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            const float tm = fmaxf(fmaxf(S.s.red[0][g], S.s.red[1][g]), fmaxf(S.s.red[2][g], S.s.red[3][g]));
            const float mn = fmaxf(m_run[g], tm);
            corr[g] = m_run[g] == -INFINITY ? 0.f : exp2f(m_run[g] - mn);
            const float p = valid ? exp2f(sc[g] - mn) : 0.f;
            l_part[g] = fmaf(l_part[g], corr[g], p);
            m_run[g] = mn;
            S.psm[tid][g] = VFm::nslots == 1 ? p * vn[0] : p;
        }
        if (VFm::nslots == 4) {
#pragma unroll
            for (int k = 0; k < 4; ++k) S.vns[tid][k] = vn[k];
        }
        __syncthreads();
#pragma unroll
        for (int g = 0; g < GP; ++g) acc[g] *= corr[g];
        const float* cb = S.s.vcb[vseg];
        for (int jj = 0; jj < nvalid; ++jj) {
            const uint32_t* vr = S.vtile + jj * VFm::words;
            uint32_t idx;
            if (VFm::three) idx = __funnelshift_r(vr[vwi], vr[vwi1], vsh) & 7u;
            else idx = (vr[vwi] >> vsh) & 15u;
            float v = cb[idx];
            if (VFm::nslots == 4) v *= S.vns[jj][vseg];
            float p[GP];
            load_row<GP>(S.psm[jj], p);
#pragma unroll
            for (int g = 0; g < GP; ++g) acc[g] = fmaf(p[g], v, acc[g]);
        }
        __syncthreads();
    }
    // l = sum over threads of l_part
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        const float ws = tq::warp_sum(l_part[g]);
        if (lane == 0) S.s.red2[warp][g] = ws;
    }
#pragma unroll
    for (int g = 0; g < GP; ++g) S.ot[g][c] = acc[g];
    __syncthreads();
    float lt[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) lt[g] = S.s.red2[0][g] + S.s.red2[1][g] + S.s.red2[2][g] + S.s.red2[3][g];
    epilogue<GP>(a, P, S.ot, m_run, lt, &S.s.is_last, b, h, s);
}

// ---------------------------------------------------------------------------
// Token-parallel V accumulation: each warp streams its own tokens (token j of
// the section goes to warp (j / 32) % 4, lane j % 32) with its own online
// softmax state; lane t adds p * v~ of its token into the warp's accumulator
// at positions staggered by lane (conflict-free, no atomics).  Warps merge by
// log-sum-exp once, at the end.  No CTA-wide barrier inside the loop.
template <int GP, int VF>
struct VRow { static constexpr int stride = (Fmt<VF>::words + 4) | 1; };

template <int GP, int KF, int VF>
struct SmemTP {
    Smem<GP, KF, VF> s;
    alignas(16) uint32_t vrec[4][32][VRow<GP, VF>::stride];
    alignas(16) float oacc[4][128][GP];
    alignas(16) float wm[4][GP];
    alignas(16) float wl[4][GP];
    alignas(16) float ot[GP][128];
};

template <int GP, int KF, int VF>
__global__ void __launch_bounds__(kThreads) decode_tp(DecodeArgs a) {
    using KFm = Fmt<KF>;
    using VFm = Fmt<VF>;
    static_assert(!KFm::tight || KFm::words <= VRow<GP, VF>::stride, "tight key records are staged in the V rows");
    __shared__ __align__(16) SmemTP<GP, KF, VF> S;
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const tq_head_params& P = a.params[h];
    const int L = clamp_len(a, b);
    const int t0 = s * a.split_len;
    const int t1 = min(t0 + a.split_len, L);
    prologue<GP, KF, VF>(a, P, S.s, b, h);
    for (int i = lane; i < 128 * GP; i += 32) (&S.oacc[warp][0][0])[i] = 0.f;
    __syncthreads();

    const size_t head_tok = ((size_t)b * a.Hkv + h) * a.Tcap;
    float m_run[GP], l_part[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) { m_run[g] = -INFINITY; l_part[g] = 0.f; }
    uint32_t* myrow = S.vrec[warp][lane];
    float(*oacc)[GP] = S.oacc[warp];

    for (int base = t0 + warp * 32; base < t1; base += 4 * 32) {
        const int j = base + lane;
        const bool valid = j < t1;
        float sc[GP];
        if (valid) {
            uint32_t rec[KFm::words];
            float kn[4];
            load_record<KF>(a.k_codes, head_tok + j, rec);
            load_norms<KF>(a.k_norms, head_tok + j, a.norm_f16, kn);
            // tight key records are staged in this lane's V row before its V record
            qk_token<GP, KF>(rec, kn, S.s.qt, S.s.ut, S.s.kcb, S.s.kseg_of, sc, myrow, 1, S.s.kseg_start);
            uint32_t vr[VFm::words];
            float vn[4] = {1.f, 1.f, 1.f, 1.f};
            load_record<VF>(a.v_codes, head_tok + j, vr);
            load_norms<VF>(a.v_norms, head_tok + j, a.norm_f16, vn);
#pragma unroll
            for (int i = 0; i < VFm::words; ++i) myrow[i] = vr[i];
#pragma unroll
            for (int k = 0; k < 4; ++k) myrow[VFm::words + k] = __float_as_uint(vn[k]);
        } else {
#pragma unroll
            for (int g = 0; g < GP; ++g) sc[g] = -INFINITY;
            // an idle lane contributes exact zeros (code 0 times norm 0, p = 0)
#pragma unroll
            for (int i = 0; i < VFm::words + 4; ++i) myrow[i] = 0u;
        }
        float p[GP], corr[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            const float mn = fmaxf(m_run[g], tq::warp_max(sc[g]));
            corr[g] = m_run[g] == -INFINITY ? 0.f : exp2f(m_run[g] - mn);
            p[g] = valid ? exp2f(sc[g] - mn) : 0.f;
            l_part[g] = fmaf(l_part[g], corr[g], p[g]);
            m_run[g] = mn;
        }
        __syncwarp();
        // rescale this warp's accumulator (lane-strided rows)
        for (int r = lane; r < 128; r += 32) {
#pragma unroll
            for (int g = 0; g < GP; ++g) oacc[r][g] *= corr[g];
        }
        __syncwarp();
        {
            // every lane runs the same 128 steps; at step k lane l updates row
            // (k + l) mod 128, so the 32 rows touched in one step are distinct
            // and the barrier per step keeps steps from overlapping
            const float vn0 = __uint_as_float(myrow[VFm::words]);
            float pv[GP];
#pragma unroll
            for (int g = 0; g < GP; ++g) pv[g] = VFm::nslots == 1 ? p[g] * vn0 : p[g];
            for (int k = 0; k < 128; ++k) {
                const int cpos = (k + lane) & 127;
                uint32_t idx;
                if (VFm::three) {
                    const int bit = 3 * cpos, wi = bit >> 5, sh = bit & 31;
                    const int wi1 = wi + 1 < VFm::words ? wi + 1 : wi;
                    idx = __funnelshift_r(myrow[wi], myrow[wi1], sh) & 7u;
                } else {
                    idx = (myrow[cpos >> 3] >> (4 * (cpos & 7))) & 15u;
                }
                const int sg = VFm::blk ? (cpos >> 5) : 0;
                float v = S.s.vcb[sg][idx];
                if (VFm::nslots == 4) v *= __uint_as_float(myrow[VFm::words + sg]);
                float o[GP];
                load_row<GP>(oacc[cpos], o);
#pragma unroll
                for (int g = 0; g < GP; ++g) o[g] = fmaf(pv[g], v, o[g]);
                if (GP % 4 == 0) {
#pragma unroll
                    for (int i = 0; i < GP / 4; ++i)
                        reinterpret_cast<float4*>(oacc[cpos])[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                } else {
#pragma unroll
                    for (int g = 0; g < GP; ++g) oacc[cpos][g] = o[g];
                }
                __syncwarp();
            }
        }
        __syncwarp();
    }
    // warp states -> CTA state (log-sum-exp over the four warps)
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        const float lw = tq::warp_sum(l_part[g]);
        if (lane == 0) { S.wm[warp][g] = m_run[g]; S.wl[warp][g] = lw; }
    }
    __syncthreads();
    float M[GP], Lt[GP], w[4][GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        M[g] = fmaxf(fmaxf(S.wm[0][g], S.wm[1][g]), fmaxf(S.wm[2][g], S.wm[3][g]));
        Lt[g] = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            w[k][g] = (M[g] == -INFINITY || S.wm[k][g] == -INFINITY) ? 0.f : exp2f(S.wm[k][g] - M[g]);
            Lt[g] = fmaf(w[k][g], S.wl[k][g], Lt[g]);
        }
    }
    const int c = tid;
#pragma unroll
    for (int g = 0; g < GP; ++g)
        S.ot[g][c] = w[0][g] * S.oacc[0][c][g] + w[1][g] * S.oacc[1][c][g] + w[2][g] * S.oacc[2][c][g] +
                     w[3][g] * S.oacc[3][c][g];
    __syncthreads();
    epilogue<GP>(a, P, S.ot, M, Lt, &S.s.is_last, b, h, s);
}

// ---------------------------------------------------------------------------
typedef void (*KernelFn)(DecodeArgs);

template <int GP, int KF, int VF>
KernelFn pick_mode(int mode) {
    if constexpr (GP <= 8) {
        if (mode == TQ_VMODE_TOKEN_PARALLEL) return decode_tp<GP, KF, VF>;
    }
    return decode_dp<GP, KF, VF>;
}
}  // namespace
