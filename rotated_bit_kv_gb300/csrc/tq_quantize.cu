// Write side: quantise-and-append of K and V vectors into the packed cache.
//
// [TQ-MNN] §2.1 (norm -> rotate -> per-coordinate codebook search), §3.1
// (sign-flipped WHT, 32-wide blocks with their own norm), §3.3 (8 three-bit
// indices in 3 bytes, two four-bit indices per byte; quantised in place at
// write time), §3.4 (search as a count of strict boundary comparisons);
// [RotaryQuant] Key design 2 (SO(4) o WHT); [Block-GTQ] mixed-rate keys with
// same-width groups, nibble containers, a whole prompt per call.
//
// One warp encodes one vector (lane l owns coordinates 4l..4l+3): 16-byte or
// 8-byte coalesced loads, warp-shuffle norm and butterflies, per-lane search,
// shuffle assembly of the packed words, coalesced 4-byte stores.
#include "tq_device.cuh"

namespace {

struct QuantArgs {
    const void* src[2];          // K, V: [B][n_new][Hkv][128]
    uint8_t* codes[2];
    void* norms[2];
    const tq_head_params* params;
    const float* kmat;           // mixed-rate keys only
    const int32_t* start_pos;
    int32_t* status;
    int B, n_new, Hkv, Tcap, in_dtype, norm_f16, rot, k_mixed;
    int code_bytes[2], norm_slots[2];
};

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) tq_quantize_kernel(QuantArgs a) {
    __shared__ float xs_all[kWarps][128];
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const long long warp = (long long)blockIdx.x * kWarps + wib;
    const long long total = 2LL * a.B * a.n_new * a.Hkv;
    if (warp >= total) return;
    const int which = (int)(warp & 1);          // 0 = K, 1 = V
    const long long v = warp >> 1;
    const int h = (int)(v % a.Hkv);
    const int t = (int)((v / a.Hkv) % a.n_new);
    const int b = (int)(v / ((long long)a.Hkv * a.n_new));
    const int slot = a.start_pos[b] + t;
    if (slot < 0 || slot >= a.Tcap) {
        if (lane == 0 && a.status) atomicOr(a.status, TQ_DEV_BAD_POSITION);
        return;
    }
    const tq_head_params& P = a.params[h];
    const size_t elem = (((size_t)b * a.n_new + t) * a.Hkv + h) * 128 + 4 * lane;
    float x[4];
    tq::load4(a.src[which], elem, a.in_dtype, x);

    const bool mixed = which == 0 && a.k_mixed;
    const int32_t* seg_start = which == 0 ? P.k_seg_start : P.v_seg_start;
    const float(*bound)[16] = which == 0 ? P.k_bound : P.v_bound;
    const int32_t* seg_bits = which == 0 ? P.k_seg_bits : P.v_seg_bits;

    float y[4];
    float nrm[4] = {0.f, 0.f, 0.f, 0.f};   // per segment
    int segi[4];                           // segment of each of this lane's positions
    if (!mixed) {
#pragma unroll
        for (int i = 0; i < 4; ++i) y[i] = x[i];
        float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
        tq::rotate_forward(a.rot, P, y);
        if (a.rot == TQ_ROT_WHT32) {
            // one norm per 32-dim block = 8 lanes
#pragma unroll
            for (int m = 1; m < 8; m <<= 1) ss += __shfl_xor_sync(TQ_FULL_MASK, ss, m);
            const int s = lane >> 3;
            float n = sqrtf(ss);
            float inv = n > 0.f ? 1.f / n : 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) { y[i] *= inv; segi[i] = s; }
            // gather the four block norms into every lane
#pragma unroll
            for (int k = 0; k < 4; ++k) nrm[k] = __shfl_sync(TQ_FULL_MASK, n, 8 * k);
        } else {
            ss = tq::warp_sum(ss);
            float n = sqrtf(ss);
            float inv = n > 0.f ? 1.f / n : 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) { y[i] *= inv; segi[i] = 0; }
            nrm[0] = n;
        }
    } else {
        float* xs = xs_all[wib];
#pragma unroll
        for (int i = 0; i < 4; ++i) xs[4 * lane + i] = x[i];
        __syncwarp();
        tq::rotate_forward_dense(P, a.kmat + (size_t)h * 128 * 128, xs, y);
        // norm of each group over its original coordinates
        float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 4 * lane + i;
            int s = 0;
            while (s < 3 && r >= seg_start[s + 1]) ++s;
            segi[i] = s;
            const float xv = xs[P.k_gcoord[r]];
#pragma unroll
            for (int k = 0; k < 4; ++k) part[k] += (k == s) ? xv * xv : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) nrm[k] = sqrtf(tq::warp_sum(part[k]));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float n = nrm[0];
#pragma unroll
            for (int k = 1; k < 4; ++k) n = segi[i] == k ? nrm[k] : n;
            y[i] = n > 0.f ? y[i] / n : 0.f;
        }
    }

    // codebook search: idx = #{k : y > boundary_k}
    uint32_t idx[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int s = segi[i];
        const int nb = (1 << seg_bits[s]) - 1;
        uint32_t c = 0;
        for (int k = 0; k < nb; ++k) c += y[i] > bound[s][k] ? 1u : 0u;
        idx[i] = c;
    }

    // pack and store
    uint8_t* rec = a.codes[which] + ((((size_t)b * a.Hkv + h) * a.Tcap) + slot) * a.code_bytes[which];
    const bool nib = mixed || seg_bits[0] == 4;
    if (nib) {
        const uint32_t v16 = idx[0] | (idx[1] << 4) | (idx[2] << 8) | (idx[3] << 12);
        const uint32_t lo = __shfl_sync(TQ_FULL_MASK, v16, (2 * lane) & 31);
        const uint32_t hi = __shfl_sync(TQ_FULL_MASK, v16, (2 * lane + 1) & 31);
        if (lane < 16) reinterpret_cast<uint32_t*>(rec)[lane] = lo | (hi << 16);
    } else {
        // lane l holds 12 bits at bit offset 12 l; word w takes lanes
        // floor(32 w / 12) .. +3
        const uint32_t v12 = idx[0] | (idx[1] << 3) | (idx[2] << 6) | (idx[3] << 9);
        const int w = lane;
        const int L0 = (32 * w) / 12;
        uint32_t word = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int L = L0 + k;
            const uint32_t val = __shfl_sync(TQ_FULL_MASK, v12, L < 32 ? L : 31);
            const int off = 12 * L - 32 * w;
            if (L < 32 && off > -12 && off < 32) word |= off >= 0 ? (val << off) : (val >> (-off));
        }
        if (lane < 12) reinterpret_cast<uint32_t*>(rec)[lane] = word;
    }
    const int slots = a.norm_slots[which];
    if (lane < slots) {
        const size_t ni = ((((size_t)b * a.Hkv + h) * a.Tcap) + slot) * slots + lane;
        float n = nrm[0];
#pragma unroll
        for (int k = 1; k < 4; ++k) n = lane == k ? nrm[k] : n;
        if (a.norm_f16) static_cast<__half*>(a.norms[which])[ni] = __float2half_rn(n);
        else static_cast<float*>(a.norms[which])[ni] = n;
    }
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

extern "C" tq_status tq_quantize_append(const tq_cache_desc* d, const tq_cache_ptrs* c, const void* K,
                                        const void* V, int32_t in_dtype, const int32_t* d_start_pos,
                                        int32_t n_new, int32_t* d_status, void* stream) {
    if (!d || !c || d->head_dim != TQ_HEAD_DIM) return TQ_ERR_INVALID_ARG;
    if (n_new < 0) return TQ_ERR_INVALID_ARG;
    if (n_new == 0) return TQ_OK;
    if (!K || !V || !d_start_pos || !c->k_codes || !c->k_norms || !c->v_codes || !c->v_norms || !c->params)
        return TQ_ERR_INVALID_ARG;
    if (in_dtype != TQ_F32 && in_dtype != TQ_F16 && in_dtype != TQ_BF16) return TQ_ERR_INVALID_ARG;
    const size_t ea = in_dtype == TQ_F32 ? 16 : 8;
    if (!aligned(K, ea) || !aligned(V, ea) || !aligned(c->k_codes, 4) || !aligned(c->v_codes, 4) ||
        !aligned(c->params, 16) || !aligned(c->k_norms, d->norm_bytes) || !aligned(c->v_norms, d->norm_bytes))
        return TQ_ERR_INVALID_ARG;
    QuantArgs a;
    a.src[0] = K;
    a.src[1] = V;
    a.codes[0] = static_cast<uint8_t*>(c->k_codes);
    a.codes[1] = static_cast<uint8_t*>(c->v_codes);
    a.norms[0] = c->k_norms;
    a.norms[1] = c->v_norms;
    a.params = static_cast<const tq_head_params*>(c->params);
    a.kmat = reinterpret_cast<const float*>(static_cast<const char*>(c->params) +
                                            (size_t)d->n_kv_heads * sizeof(tq_head_params));
    a.start_pos = d_start_pos;
    a.status = d_status;
    a.B = d->batch;
    a.n_new = n_new;
    a.Hkv = d->n_kv_heads;
    a.Tcap = d->t_capacity;
    a.in_dtype = in_dtype;
    a.norm_f16 = d->norm_dtype == TQ_F16;
    a.rot = d->rot;
    a.k_mixed = d->k_mixed;
    a.code_bytes[0] = d->k_code_bytes;
    a.code_bytes[1] = d->v_code_bytes;
    a.norm_slots[0] = d->k_norm_slots;
    a.norm_slots[1] = d->v_norm_slots;
    const long long warps = 2LL * d->batch * n_new * d->n_kv_heads;
    const long long blocks = (warps + kWarps - 1) / kWarps;
    if (blocks > 0x7fffffffLL) return TQ_ERR_INVALID_ARG;
    tq_quantize_kernel<<<(unsigned)blocks, kWarps * 32, 0, (cudaStream_t)stream>>>(a);
    return cudaPeekAtLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
