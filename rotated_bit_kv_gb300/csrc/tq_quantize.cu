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
#include <numeric>

#include "tq_device.cuh"
#include "tq_tile.cuh"

namespace {

struct QuantArgs {
    const void* src[2];          // K, V: [B][n_new][Hkv][128]
    uint8_t* codes[2];
    void* norms[2];
    const tq_head_params* params;
    const float* kmat;           // mixed-rate keys only
    const int32_t* start_pos;
    int32_t* status;
    // Tcap: the capacity (valid positions); t_alloc: positions per (batch, KV
    // head) in the arrays; tiled: TQ_LAYOUT_TILE16 (tq_tile.cuh) else one record
    // per position
    int B, n_new, Hkv, Tcap, t_alloc, tiled, in_dtype, norm_f16, rot, k_mixed;
    int k_two;                   // two-stage keys: k_bits (1 or 2), else 0
    int k_tight;                 // mixed-rate keys in tight records (natural layout)
    int code_bytes[2], norm_slots[2];
};

// Element index of norm slot k of the vector at position `pos` = pair * t_alloc +
// slot (which: 0 keys, 1 values).
__device__ __forceinline__ size_t norm_index(const QuantArgs& a, int which, size_t pos, int slots, int k) {
    if (!a.tiled) return pos * slots + k;
    const size_t base = (pos & ~(size_t)15) * slots;
    const int t = (int)(pos & 15);
    if (slots == 1) return base + tqtile::norm_pos1(t);
    return base + (which == 0 ? tqtile::norm_pos4_k(t, k) : tqtile::norm_pos4_v(t, k));
}

// Scatter the packed record `rec` (shared memory, visible to the whole warp) of
// the vector at position `pos` into its tile; every lane of the warp calls this.
__device__ __forceinline__ void store_tiled(const QuantArgs& a, int which, size_t pos, const uint32_t* rec,
                                            int bits, int lane) {
    uint8_t* codes = which ? a.codes[1] : a.codes[0];
    const int t = (int)(pos & 15);
    if (bits == 3) {
        uint8_t* tile = codes + (pos >> 4) * tqtile::tile_bytes(3);
        if (which == 0) tqtile::store_key<3>(tile, rec, t, lane);
        else tqtile::store_value<3>(tile, rec, t, lane);
    } else {
        uint8_t* tile = codes + (pos >> 4) * tqtile::tile_bytes(4);
        if (which == 0) tqtile::store_key<4>(tile, rec, t, lane);
        else tqtile::store_value<4>(tile, rec, t, lane);
    }
}

constexpr int kWarps = 8;
constexpr long long kMaxBlocks = 152LL * 8 * 4;   // four waves of 8 resident CTAs per SM

// Vector index (warp-uniform): K and V alternate, then KV head, token, batch.
struct VecId {
    int which, h, t, b;
};

__device__ __forceinline__ VecId vec_id(const QuantArgs& a, uint32_t v_all) {
    VecId id;
    id.which = (int)(v_all & 1u);
    const uint32_t v = v_all >> 1;
    const uint32_t q = v / (uint32_t)a.Hkv;
    id.h = (int)(v - q * (uint32_t)a.Hkv);
    const uint32_t bb = q / (uint32_t)a.n_new;
    id.t = (int)(q - bb * (uint32_t)a.n_new);
    id.b = (int)bb;
    return id;
}

// input [B][n_new][Hkv][128] in the vector order: element offset (v >> 1) * 128
__device__ __forceinline__ size_t input_elem(uint32_t v_all) {
    return (size_t)(v_all >> 1) * 128 + 4 * (threadIdx.x & 31);
}

// Encode one vector; xin holds this lane's 4 input values.
__device__ __forceinline__ void encode_vector(const QuantArgs& a, const VecId& id, const float* xin, float* xs) {
    const int lane = threadIdx.x & 31;
    const int which = id.which, h = id.h, t = id.t, b = id.b;
    const int slot = a.start_pos[b] + t;
    if (slot < 0 || slot >= a.Tcap) {
        if (lane == 0 && a.status) atomicOr(a.status, TQ_DEV_BAD_POSITION);
        return;
    }
    const tq_head_params& P = a.params[h];
    float x[4] = {xin[0], xin[1], xin[2], xin[3]};

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
    if (!mixed && seg_bits[segi[0]] <= 4) {
        // one segment per lane: its boundaries in registers, an unrolled count
        const int s = segi[0];
        const int nb = (1 << seg_bits[s]) - 1;
        float bd[15];
#pragma unroll
        for (int k = 0; k < 15; ++k) bd[k] = k < nb ? bound[s][k] : INFINITY;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t c = 0;
#pragma unroll
            for (int k = 0; k < 15; ++k) c += y[i] > bd[k] ? 1u : 0u;
            idx[i] = c;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int s = segi[i];
            const int nb = (1 << seg_bits[s]) - 1;
            uint32_t c = 0;
            for (int k = 0; k < nb; ++k) c += y[i] > bound[s][k] ? 1u : 0u;
            idx[i] = c;
        }
    }

    // tile layout: a b-bit code of mixed-rate keys' 1..3-bit groups is stored as
    // code + 2^b, so that its nibble names its group
    if (mixed && a.tiled) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int bw = seg_bits[segi[i]];
            idx[i] += bw < 4 ? (1u << bw) : 0u;
        }
    }
    // pack and store (tile layout: the record goes through the warp's staging
    // buffer, once every lane is done reading the staged input)
    if (mixed && a.k_tight) {
        // tight record [Block-GTQ, packed cache]: the lane's four codes at their
        // widths (at most 16 bits) at the bit offset of position 4l, the
        // exclusive prefix of the lanes' widths; OR-ed into a zeroed staging copy
        int sh = 0;
        uint32_t v = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v |= idx[i] << sh;
            sh += seg_bits[segi[i]];
        }
        int off = sh;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const int o = __shfl_up_sync(TQ_FULL_MASK, off, m);
            if (lane >= m) off += o;
        }
        off -= sh;
        uint32_t* st = reinterpret_cast<uint32_t*>(xs);
        __syncwarp();   // every lane is done with the staged input
        if (lane < 16) st[lane] = 0u;
        __syncwarp();
        const int wi = off >> 5, bs = off & 31;
        atomicOr(st + wi, v << bs);
        if (bs + sh > 32) atomicOr(st + wi + 1, v >> (32 - bs));
        __syncwarp();
        const size_t pos = (((size_t)b * a.Hkv + h) * a.t_alloc) + slot;
        uint32_t* out = reinterpret_cast<uint32_t*>(a.codes[0] + pos * a.code_bytes[0]);
        if (lane < (a.code_bytes[0] >> 2)) out[lane] = st[lane];
        if (lane < 4) {
            const size_t ni = pos * 4 + lane;
            float n = nrm[0];
#pragma unroll
            for (int k = 1; k < 4; ++k) n = lane == k ? nrm[k] : n;
            if (a.norm_f16) static_cast<__half*>(a.norms[0])[ni] = __float2half_rn(n);
            else static_cast<float*>(a.norms[0])[ni] = n;
        }
        return;
    }
    if (a.tiled) __syncwarp();
    const size_t pos = (((size_t)b * a.Hkv + h) * a.t_alloc) + slot;
    uint8_t* rec = a.tiled ? reinterpret_cast<uint8_t*>(xs)
                           : (which ? a.codes[1] : a.codes[0]) + pos * (which ? a.code_bytes[1] : a.code_bytes[0]);
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
    if (a.tiled) {
        __syncwarp();
        store_tiled(a, which, pos, reinterpret_cast<const uint32_t*>(rec), nib ? 4 : 3, lane);
    }
    const int slots = (which ? a.norm_slots[1] : a.norm_slots[0]);
    if (lane < slots) {
        const size_t ni = norm_index(a, which, pos, slots, lane);
        float n = nrm[0];
#pragma unroll
        for (int k = 1; k < 4; ++k) n = lane == k ? nrm[k] : n;
        if (a.norm_f16) static_cast<__half*>((which ? a.norms[1] : a.norms[0]))[ni] = __float2half_rn(n);
        else static_cast<float*>((which ? a.norms[1] : a.norms[0]))[ni] = n;
    }
}

// Two-stage key code [TQ-MNN §2.4]: y = R x / n on the (k_bits - 1)-bit codebook
// (one boundary; no code for k_bits = 1), residual r = y - C[idx], z = S r (fp32,
// the transposed projection in the blob's matrix slot), sign bits z_j >= 0;
// norms n and n ||r||.  Natural layout: the record is (k_bits - 1) * 4 words of
// codes then 4 words of signs, bit j of the stream for coordinate j.
__device__ __forceinline__ void encode_two_stage(const QuantArgs& a, const VecId& id, const float* xin, float* xs) {
    const int lane = threadIdx.x & 31;
    const int h = id.h, t = id.t, b = id.b;
    const int slot = a.start_pos[b] + t;
    if (slot < 0 || slot >= a.Tcap) {
        if (lane == 0 && a.status) atomicOr(a.status, TQ_DEV_BAD_POSITION);
        return;
    }
    const tq_head_params& P = a.params[h];
    float y[4] = {xin[0], xin[1], xin[2], xin[3]};
    const float ss = y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3];
    tq::rotate_forward(a.rot, P, y);
    const float n = sqrtf(tq::warp_sum(ss));
    const float inv = n > 0.f ? 1.f / n : 0.f;
    uint32_t code4 = 0;
    float r[4];
    if (a.k_two == 2) {
        const float bd = P.k_bound[0][0], c0 = P.k_cent[0][0], c1 = P.k_cent[0][1];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float yi = y[i] * inv;
            const bool up = yi > bd;
            code4 |= (up ? 1u : 0u) << i;
            r[i] = yi - (up ? c1 : c0);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) r[i] = y[i] * inv;
    }
    const float rho = sqrtf(tq::warp_sum(r[0] * r[0] + r[1] * r[1] + r[2] * r[2] + r[3] * r[3]));
#pragma unroll
    for (int i = 0; i < 4; ++i) xs[4 * lane + i] = r[i];
    __syncwarp();
    float z[4];
    tq::dense_rows_t(a.kmat + (size_t)h * 128 * 128, xs, z);
    __syncwarp();   // xs is the next vector's staging buffer
    uint32_t sgn4 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) sgn4 |= (z[i] >= 0.f ? 1u : 0u) << i;
    // word w of a 1-bit stream = the 4-bit groups of lanes 8w .. 8w+7
    const int src = 8 * (lane & 3);
    uint32_t wc = 0, wsg = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        wc |= __shfl_sync(TQ_FULL_MASK, code4, src + k) << (4 * k);
        wsg |= __shfl_sync(TQ_FULL_MASK, sgn4, src + k) << (4 * k);
    }
    const size_t pos = (((size_t)b * a.Hkv + h) * a.t_alloc) + slot;
    uint32_t* rec = reinterpret_cast<uint32_t*>(a.codes[0] + pos * a.code_bytes[0]);
    const int mw = 4 * (a.k_two - 1);
    if (lane < 4) {
        if (mw) rec[lane] = wc;
        rec[mw + lane] = wsg;
    }
    if (lane < 2) {
        const float nv = lane == 0 ? n : n * rho;
        const size_t ni = pos * 2 + lane;
        if (a.norm_f16) static_cast<__half*>(a.norms[0])[ni] = __float2half_rn(nv);
        else static_cast<float*>(a.norms[0])[ni] = nv;
    }
}

// Encode one vector of a cache without mixed-rate keys: the rotation kind is a
// template parameter, the boundaries of the lane's segment come in as float4s and
// the count is unrolled.  Same steps and results as encode_vector.
template <int BITS>
__device__ __forceinline__ void search_pack(const QuantArgs& a, const float* bnd, const float y[4], uint8_t* rec) {
    const int lane = threadIdx.x & 31;
    constexpr int NB = (1 << BITS) - 1;
    float bd[NB + 1];
#pragma unroll
    for (int k = 0; k < (NB + 1) / 4; ++k) {
        const float4 f = reinterpret_cast<const float4*>(bnd)[k];
        bd[4 * k] = f.x; bd[4 * k + 1] = f.y; bd[4 * k + 2] = f.z; bd[4 * k + 3] = f.w;
    }
    uint32_t idx[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t c = 0;
#pragma unroll
        for (int k = 0; k < NB; ++k) c += y[i] > bd[k] ? 1u : 0u;
        idx[i] = c;
    }
    if (BITS == 4) {
        const uint32_t v16 = idx[0] | (idx[1] << 4) | (idx[2] << 8) | (idx[3] << 12);
        const uint32_t lo = __shfl_sync(TQ_FULL_MASK, v16, (2 * lane) & 31);
        const uint32_t hi = __shfl_sync(TQ_FULL_MASK, v16, (2 * lane + 1) & 31);
        if (lane < 16) reinterpret_cast<uint32_t*>(rec)[lane] = lo | (hi << 16);
    } else {
        // lane l holds 12 bits at bit offset 12 l; word w takes lanes
        // floor(32 w / 12) .. +3
        const uint32_t v12 = idx[0] | (idx[1] << 3) | (idx[2] << 6) | (idx[3] << 9);
        const int L0 = (32 * lane) / 12;
        uint32_t word = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int L = L0 + k;
            const uint32_t val = __shfl_sync(TQ_FULL_MASK, v12, L < 32 ? L : 31);
            const int off = 12 * L - 32 * lane;
            if (L < 32 && off > -12 && off < 32) word |= off >= 0 ? (val << off) : (val >> (-off));
        }
        if (lane < 12) reinterpret_cast<uint32_t*>(rec)[lane] = word;
    }
}

template <int ROT>
__device__ __forceinline__ void encode_fast(const QuantArgs& a, const VecId& id, const float* xin, float* xs) {
    const int lane = threadIdx.x & 31;
    const int which = id.which, h = id.h, t = id.t, b = id.b;
    const int slot = a.start_pos[b] + t;
    if (slot < 0 || slot >= a.Tcap) {
        if (lane == 0 && a.status) atomicOr(a.status, TQ_DEV_BAD_POSITION);
        return;
    }
    const tq_head_params& P = a.params[h];
    float y[4] = {xin[0], xin[1], xin[2], xin[3]};
    float ss = y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3];
    tq::rotate_forward(ROT, P, y);
    float n;
    if (ROT == TQ_ROT_WHT32) {   // one norm per 32-dim block = 8 lanes
#pragma unroll
        for (int m = 1; m < 8; m <<= 1) ss += __shfl_xor_sync(TQ_FULL_MASK, ss, m);
        n = sqrtf(ss);
    } else {
        n = sqrtf(tq::warp_sum(ss));
    }
    const float inv = n > 0.f ? 1.f / n : 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i] *= inv;
    const int s = ROT == TQ_ROT_WHT32 ? lane >> 3 : 0;
    const int bits = which == 0 ? P.k_seg_bits[s] : P.v_seg_bits[s];
    const float* bnd = which == 0 ? P.k_bound[s] : P.v_bound[s];
    const size_t pos = (((size_t)b * a.Hkv + h) * a.t_alloc) + slot;
    uint8_t* rec = a.tiled ? reinterpret_cast<uint8_t*>(xs)
                           : (which ? a.codes[1] : a.codes[0]) + pos * (which ? a.code_bytes[1] : a.code_bytes[0]);
    if (bits == 4) search_pack<4>(a, bnd, y, rec);
    else search_pack<3>(a, bnd, y, rec);
    if (a.tiled) {
        __syncwarp();
        store_tiled(a, which, pos, reinterpret_cast<const uint32_t*>(rec), bits, lane);
    }
    // norms: one per vector, or one per 32-dim block (lanes 0, 8, 16, 24 hold them)
    const int slots = (which ? a.norm_slots[1] : a.norm_slots[0]);
    const float nv = ROT == TQ_ROT_WHT32 ? __shfl_sync(TQ_FULL_MASK, n, 8 * (lane & 3)) : n;
    if (lane < slots) {
        const size_t ni = norm_index(a, which, pos, slots, lane);
        if (a.norm_f16) static_cast<__half*>((which ? a.norms[1] : a.norms[0]))[ni] = __float2half_rn(nv);
        else static_cast<float*>((which ? a.norms[1] : a.norms[0]))[ni] = nv;
    }
}

// Each warp encodes vectors warp, warp + nwarps, ... (K and V alternate), the
// next vector's input loaded while the current one is encoded.  Vector indices
// fit in 32 bits (checked on the host).
// ROT < 0: any rotation, mixed-rate keys allowed (encode_vector); else the
// specialised path for that rotation kind.
template <int ROT>
__global__ void __launch_bounds__(kWarps * 32) tq_quantize_kernel(QuantArgs a) {
    __shared__ float xs_all[kWarps][128];
    const int wib = threadIdx.x >> 5;
    const uint32_t nwarps = gridDim.x * kWarps;
    const uint32_t total = 2u * (uint32_t)a.B * (uint32_t)a.n_new * (uint32_t)a.Hkv;
    uint32_t v = blockIdx.x * kWarps + wib;
    if (v >= total) return;
    VecId id = vec_id(a, v);
    float x[4];
    tq::load4((id.which ? a.src[1] : a.src[0]), input_elem(v), a.in_dtype, x);
    for (;;) {
        const uint32_t vn = v + nwarps;
        const bool more = vn < total && vn > v;
        VecId idn = id;
        float xn[4] = {0.f, 0.f, 0.f, 0.f};
        if (more) {
            idn = vec_id(a, vn);
            tq::load4((idn.which ? a.src[1] : a.src[0]), input_elem(vn), a.in_dtype, xn);
        }
        if constexpr (ROT < 0) {
            if (id.which == 0 && a.k_two) encode_two_stage(a, id, x, xs_all[wib]);
            else encode_vector(a, id, x, xs_all[wib]);
        } else {
            encode_fast<ROT>(a, id, x, xs_all[wib]);
        }
        if (!more) break;
        __syncwarp();
        v = vn;
        id = idn;
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = xn[i];
    }
}

// ---- half-warp path: caches without mixed-rate keys, K and V of the same width.
//
// A warp takes one (batch, token, KV head): lanes 0-15 encode its K vector,
// lanes 16-31 its V vector; lane j of a half holds coordinates 8j .. 8j+7.  The
// three butterfly stages of strides 1, 2, 4 stay in the lane, the four of
// strides 8 .. 64 cross lanes of the half; 3-bit codes of four lanes are the
// three words of a 32-coordinate group.  Same steps and results as encode_vector.

// Walsh-Hadamard butterflies over 8 * LANES coordinates held 8 per lane
template <int LANES>
__device__ __forceinline__ void wht8(float v[8]) {
#pragma unroll
    for (int st = 1; st < 8; st <<= 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i & st) continue;
            const float x = v[i], y = v[i + st];
            v[i] = x + y;
            v[i + st] = x - y;
        }
    }
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int m = 1; m < LANES; m <<= 1) {
        const float sgn = (lane & m) ? -1.f : 1.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float o = __shfl_xor_sync(TQ_FULL_MASK, v[i], m);
            v[i] = fmaf(sgn, v[i], o);
        }
    }
}

// #{k : y > bd[k]} over the 2^BITS - 1 ascending boundaries, as a binary search:
// each comparison settles one bit of the index, the next threshold is selected by
// the bits above it (same strict comparisons, same result as the count)  [TQ-MNN] §3.4
template <int BITS>
__device__ __forceinline__ uint32_t search_bits(float y, const float* bd) {
    if constexpr (BITS == 3) {
        const bool g2 = y > bd[3];
        const bool g1 = y > (g2 ? bd[5] : bd[1]);
        const bool g0 = y > (g2 ? (g1 ? bd[6] : bd[4]) : (g1 ? bd[2] : bd[0]));
        return (g2 ? 4u : 0u) | (g1 ? 2u : 0u) | (g0 ? 1u : 0u);
    } else {
        const bool g3 = y > bd[7];
        const bool g2 = y > (g3 ? bd[11] : bd[3]);
        const bool g1 = y > (g3 ? (g2 ? bd[13] : bd[9]) : (g2 ? bd[5] : bd[1]));
        const float t0 = g3 ? (g2 ? (g1 ? bd[14] : bd[12]) : (g1 ? bd[10] : bd[8]))
                            : (g2 ? (g1 ? bd[6] : bd[4]) : (g1 ? bd[2] : bd[0]));
        const bool g0 = y > t0;
        return (g3 ? 8u : 0u) | (g2 ? 4u : 0u) | (g1 ? 2u : 0u) | (g0 ? 1u : 0u);
    }
}

// input element type fixed at compile time (DT: TQ_F32, TQ_F16 or TQ_BF16)
template <int DT>
__device__ __forceinline__ void load8t(const void* base, size_t elem, float v[8]) {
    if constexpr (DT == TQ_F32) {
        const float4 x = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem);
        const float4 y = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem + 4);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w; v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
    } else {
        const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (DT == TQ_F16) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
                v[2 * i] = f.x;
                v[2 * i + 1] = f.y;
            } else {
                v[2 * i] = __uint_as_float(w[i] << 16);
                v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            }
        }
    }
}

// What one half-warp lane needs of its KV head's parameters: the signs (WHT
// kinds) or the two quaternion pairs (SO(4)) of its 8 coordinates, and the
// boundaries of its codebook.
template <int ROT, int BITS>
struct HalfParams {
    float s[8];
    float qa[8], qb[8];
    float bd[1 << BITS];
};

template <int ROT, int BITS>
__device__ __forceinline__ void load_half_params(const tq_head_params& P, int hv, int j, HalfParams<ROT, BITS>& hp) {
    if constexpr (ROT == TQ_ROT_SO4_WHT128) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            hp.qa[i] = P.quat[2 * j][i];
            hp.qb[i] = P.quat[2 * j + 1][i];
        }
    } else {
        const float4 s0 = reinterpret_cast<const float4*>(P.signs + 8 * j)[0];
        const float4 s1 = reinterpret_cast<const float4*>(P.signs + 8 * j)[1];
        hp.s[0] = s0.x; hp.s[1] = s0.y; hp.s[2] = s0.z; hp.s[3] = s0.w;
        hp.s[4] = s1.x; hp.s[5] = s1.y; hp.s[6] = s1.z; hp.s[7] = s1.w;
    }
    const int sgi = ROT == TQ_ROT_WHT32 ? j >> 2 : 0;
    const float* bnd = hv ? P.v_bound[sgi] : P.k_bound[sgi];
#pragma unroll
    for (int k = 0; k < (1 << BITS) / 4; ++k) {
        const float4 f = reinterpret_cast<const float4*>(bnd)[k];
        hp.bd[4 * k] = f.x; hp.bd[4 * k + 1] = f.y; hp.bd[4 * k + 2] = f.z; hp.bd[4 * k + 3] = f.w;
    }
}

template <int ROT, int BITS, int DT>
__global__ void __launch_bounds__(kWarps * 32) tq_quantize_half(QuantArgs a) {
    // a programmatic dependent launched after this kernel (decode) may be placed now;
    // it still waits for this grid's completion before it reads anything
    asm volatile("griddepcontrol.launch_dependents;");
    __shared__ __align__(16) uint32_t recbuf[kWarps][2][16];   // tile layout: the K and V records
    const int lane = threadIdx.x & 31, hv = lane >> 4, j = lane & 15;
    const uint32_t nwarps = gridDim.x * kWarps;
    const uint32_t total = (uint32_t)a.B * (uint32_t)a.n_new * (uint32_t)a.Hkv;   // (b, t, h) pairs
    uint32_t p = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (p >= total) return;
    const void* src = hv ? a.src[1] : a.src[0];
    uint8_t* const cbase = hv ? a.codes[1] : a.codes[0];
    const int cbytes = hv ? a.code_bytes[1] : a.code_bytes[0];
    void* const nbase = hv ? a.norms[1] : a.norms[0];
    const int slots = hv ? a.norm_slots[1] : a.norm_slots[0];
    const int Hkv = a.Hkv, n_new = a.n_new, Tcap = a.Tcap;
    float x[8];
    load8t<DT>(src, (size_t)p * 128 + 8 * j, x);
    // p = (b * n_new + t) * Hkv + h, carried forward by nwarps per pass without a division
    int h, t, b;
    {
        const uint32_t q = p / (uint32_t)Hkv;
        h = (int)(p - q * (uint32_t)Hkv);
        b = (int)(q / (uint32_t)n_new);
        t = (int)(q - (uint32_t)b * (uint32_t)n_new);
    }
    const uint32_t sq = nwarps / (uint32_t)Hkv;
    const int sh = (int)(nwarps - sq * (uint32_t)Hkv);
    const int sb = (int)(sq / (uint32_t)n_new);
    const int st = (int)(sq - (uint32_t)sb * (uint32_t)n_new);
    // the head's parameters, reloaded only when the head changes (never, when the
    // launch makes the warp count a multiple of the head count)
    HalfParams<ROT, BITS> hp;
    int h_loaded = -1;
    for (;;) {
        const uint32_t pn = p + nwarps;
        const bool more = pn < total && pn > p;
        float xn[8];
        load8t<DT>(src, (size_t)(more ? pn : p) * 128 + 8 * j, xn);   // next pass (or this one again)

        if (h != h_loaded) {
            load_half_params<ROT, BITS>(a.params[h], hv, j, hp);
            h_loaded = h;
        }
        const int slot = a.start_pos[b] + t;
        if (slot < 0 || slot >= Tcap) {
            if (lane == 0 && a.status) atomicOr(a.status, TQ_DEV_BAD_POSITION);
        } else {
            float y[8];
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = ROT == TQ_ROT_SO4_WHT128 ? x[i] : x[i] * hp.s[i];
            float n;
            if (ROT == TQ_ROT_WHT32) {   // four 32-dim blocks of 4 lanes, one norm each
                wht8<4>(y);
#pragma unroll
                for (int i = 0; i < 8; ++i) y[i] *= 0.17677669529663687f;   // 1/sqrt(32)
#pragma unroll
                for (int m = 1; m < 4; m <<= 1) ss += __shfl_xor_sync(TQ_FULL_MASK, ss, m);
            } else {
                wht8<16>(y);
#pragma unroll
                for (int i = 0; i < 8; ++i) y[i] *= 0.08838834764831845f;   // 1/sqrt(128)
                if (ROT == TQ_ROT_SO4_WHT128) {
                    tq::so4_forward(hp.qa, y);
                    tq::so4_forward(hp.qb, y + 4);
                }
#pragma unroll
                for (int m = 1; m < 16; m <<= 1) ss += __shfl_xor_sync(TQ_FULL_MASK, ss, m);
            }
            n = sqrtf(ss);
            const float inv = n > 0.f ? 1.f / n : 0.f;
            uint32_t code = 0;   // 8 indices of BITS bits, coordinate 8j + i at bit BITS * i
#pragma unroll
            for (int i = 0; i < 8; ++i) code |= search_bits<BITS>(y[i] * inv, hp.bd) << (BITS * i);
            const size_t rec_i = (((size_t)b * Hkv + h) * a.t_alloc) + slot;
            uint32_t* const rb = recbuf[threadIdx.x >> 5][hv];
            uint32_t* rec = a.tiled ? rb : reinterpret_cast<uint32_t*>(cbase + rec_i * cbytes);
            if (BITS == 4) {
                rec[j] = code;
            } else {
                // lanes 4m .. 4m+3 hold 96 bits = words 3m .. 3m+2
                const uint32_t nxt = __shfl_down_sync(TQ_FULL_MASK, code, 1);
                const int r = j & 3, m4 = j >> 2;
                if (r < 3) rec[3 * m4 + r] = (code >> (8 * r)) | (nxt << (24 - 8 * r));
            }
            if (a.tiled) {   // both records through shared memory, then the whole warp scatters each
                __syncwarp();
                store_tiled(a, 0, rec_i, recbuf[threadIdx.x >> 5][0], BITS, lane);
                store_tiled(a, 1, rec_i, recbuf[threadIdx.x >> 5][1], BITS, lane);
                __syncwarp();
            }
            const float nv = ROT == TQ_ROT_WHT32 ? __shfl_sync(TQ_FULL_MASK, n, 16 * hv + 4 * (j & 3)) : n;
            if (j < slots) {
                const size_t ni = norm_index(a, hv, rec_i, slots, j);
                if (a.norm_f16) static_cast<__half*>(nbase)[ni] = __float2half_rn(nv);
                else static_cast<float*>(nbase)[ni] = nv;
            }
        }
        if (!more) break;
        p = pn;
        h += sh;
        const int cq = h >= Hkv ? 1 : 0;
        h -= cq ? Hkv : 0;
        t += st + cq;
        const int cb = t >= n_new ? 1 : 0;
        t -= cb ? n_new : 0;
        b += sb + cb;
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = xn[i];
    }
}

// ---- tensor-core rotation (sign-flipped WHT128, 3-bit codes, fp16/bf16 input)
//
// A warp encodes 16 vectors at once: the K (rows 0-7) and V (rows 8-15) vectors of
// 8 consecutive (batch, token, KV head) triples.  With i = 16 s + i' and
// j = 16 u + j', the Sylvester matrix factors as H128[i][j] = H8[s][u] H16[i'][j'],
// so for each half e of the 16-column block
//   P_s = A_s . B_e        (A_s: columns 16s .. 16s+15 of the sign-flipped input,
//                           B_e: 8 columns of H16; one mma m16n8k16 each)
//   C_u = sum_s H8[s][u] P_s   (an 8-point butterfly on the fp32 accumulators).
// Products of 16-bit inputs and +-1 are exact and accumulate in fp32, so the
// result is the rotated vector times sqrt(128) up to fp32 rounding.  The squared
// norms come from the same fragments: x_m . x_n is an mma of the tile with itself,
// its diagonal the 16 norms.  [TQ-MNN] §3.1 (sign-flipped WHT), §3.4 (search).
//
// Column orders: A column k of step s is coordinate 16s + pi(k) with
// pi(2c + b) = 4c + b, pi(2c + 8 + b) = 4c + 2 + b, so that lane c's operand is one
// 8-byte load; output column n of half e is coordinate 16u + 4c + 2e + b for
// n = 2c + b, so that lane c ends with coordinates 16u + 4c .. 16u + 4c + 3.

template <int DT>
__device__ __forceinline__ void mma_16816_x(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1) {
    if constexpr (DT == TQ_BF16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__host__ __device__ constexpr int popc4(int x) { return (x & 1) + ((x >> 1) & 1) + ((x >> 2) & 1) + ((x >> 3) & 1); }

// +-1 in the 16-bit input format, packed for two k rows (lower k in the low half)
template <int DT>
__device__ __forceinline__ uint32_t pm1_pair(int neg_lo, int neg_hi) {
    constexpr uint32_t one = DT == TQ_BF16 ? 0x3F80u : 0x3C00u;
    return (one | (neg_lo ? 0x8000u : 0u)) | ((one | (neg_hi ? 0x8000u : 0u)) << 16);
}

constexpr int kTcWarps = 4;
constexpr int kTcRow = 288;   // bytes per staged row: 256 + 32, so that the 8-byte operand reads share no bank
constexpr int kCells = 128;                // cells of 1/32 over [-2, 2)
constexpr float kCellMagic = 1572928.f;   // 64 + 1.5 * 2^20: the sum's unit in the last place is 1/8
constexpr long long kTcMinTriples = 4096;   // smaller appends (decode steps) take the half-warp path
constexpr long long kTcMaxBlocks = 152LL * 4 * 4;   // four waves of 4 resident CTAs per SM

// The tile loop of one warp; TAB: codebook search through the cell table `tab`
// (one table for every head, K and V), else a binary search on the head's boundaries.
template <int DT, bool TAB>
__device__ __forceinline__ void qtc_loop(const QuantArgs& a, const float2* tab, uint8_t (*stage)[48],
                                         uint8_t (*ring)[16][kTcRow]) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const uint32_t nwarps = gridDim.x * kTcWarps;
    // a tile = 8 consecutive tokens of one (batch, KV head): tile = (b Hkv + h) ntt + tt
    // holds tokens 8 tt .. 8 tt + 7 (those past n_new are loaded clamped, not stored),
    // so its records fill one half of a 16-token cache tile (consecutive positions)
    const uint32_t ntt = ((uint32_t)a.n_new + 7) / 8;
    const uint32_t tiles = (uint32_t)a.B * (uint32_t)a.Hkv * ntt;
    uint32_t tile = blockIdx.x * kTcWarps + (threadIdx.x >> 5);
    if (tile >= tiles) return;
    const int Hkv = a.Hkv, n_new = a.n_new, Tcap = a.Tcap;
    const uint16_t* Ksrc = static_cast<const uint16_t*>(a.src[0]);
    const uint16_t* Vsrc = static_cast<const uint16_t*>(a.src[1]);

    // H16 columns of each half e as mma operand B (lane: rows 2c, 2c+1 / 2c+8, 2c+9, column g)
    uint32_t hb[2][2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int j = 4 * (g >> 1) + 2 * e + (g & 1);
        hb[e][0] = pm1_pair<DT>(popc4((4 * c) & j) & 1, popc4((4 * c + 1) & j) & 1);
        hb[e][1] = pm1_pair<DT>(popc4((4 * c + 2) & j) & 1, popc4((4 * c + 3) & j) & 1);
    }

    // this lane's (batch, token, KV head): token 8 tt + g of the tile
    int h, t, b, t8;
    auto locate = [&](uint32_t tl_) {
        const uint32_t bh = tl_ / ntt;
        t8 = 8 * (int)(tl_ - bh * ntt);
        b = (int)(bh / (uint32_t)Hkv);
        h = (int)(bh - (uint32_t)b * (uint32_t)Hkv);
        t = t8 + g;
    };
    locate(tile);

    // the head's sign masks (coordinates 16s + 4c .. +3) and K / V boundaries
    uint32_t msk[8][2];
    float kb[8], vb[8];
    int h_loaded = -1;
    auto load_head = [&](int hh) {   // hh is a valid head index for every lane
        const tq_head_params& P = a.params[hh];
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const float4 sg = *reinterpret_cast<const float4*>(P.signs + 16 * s + 4 * c);
            msk[s][0] = (sg.x < 0.f ? 0x8000u : 0u) | (sg.y < 0.f ? 0x80000000u : 0u);
            msk[s][1] = (sg.z < 0.f ? 0x8000u : 0u) | (sg.w < 0.f ? 0x80000000u : 0u);
        }
#pragma unroll
        for (int k = 0; k < 2 && !TAB; ++k) {
            const float4 f = reinterpret_cast<const float4*>(P.k_bound[0])[k];
            const float4 v = reinterpret_cast<const float4*>(P.v_bound[0])[k];
            kb[4 * k] = f.x; kb[4 * k + 1] = f.y; kb[4 * k + 2] = f.z; kb[4 * k + 3] = f.w;
            vb[4 * k] = v.x; vb[4 * k + 1] = v.y; vb[4 * k + 2] = v.z; vb[4 * k + 3] = v.w;
        }
    };

    // The warp's tiles stream through a two-stage ring in shared memory (cp.async,
    // 16 bytes a lane): rows 0-7 = K, 8-15 = V of the tile's 8 tokens (rows past the
    // last token repeat it)
    auto issue = [&](uint32_t tl_, int stg) {
        const uint32_t bh = tl_ / ntt;
        const int tt8 = 8 * (int)(tl_ - bh * ntt);
        const uint32_t bb = bh / (uint32_t)Hkv, hh = bh - bb * (uint32_t)Hkv;
        const size_t row0 = (size_t)bb * n_new * Hkv + hh;   // input row of (bb, token 0, hh)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = lane + 32 * k, row = i >> 4, col = i & 15;
            const int tk = min(tt8 + (row & 7), n_new - 1);
            const uint16_t* src = (k < 4 ? Ksrc : Vsrc) + (row0 + (size_t)tk * Hkv) * 128 + col * 8;
            const uint32_t dst = (uint32_t)__cvta_generic_to_shared(&ring[stg][row][col * 16]);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src));
        }
    };
    uint32_t ax[8][4];   // operand A of the tile: row g = K of triple p, row g + 8 = V of triple p
    uint32_t tl = tile;
    int stg = 0;
    issue(tl, 0);
    asm volatile("cp.async.commit_group;");
    if (tl + nwarps < tiles && tl + nwarps > tl) issue(tl + nwarps, 1);
    asm volatile("cp.async.commit_group;");

    for (;;) {
        const bool valid = t < n_new;
        if (h != h_loaded) {
            load_head(h);
            h_loaded = h;
        }
        asm volatile("cp.async.wait_group 1;" ::: "memory");
        __syncwarp();
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint2 k2 = *reinterpret_cast<const uint2*>(&ring[stg][g][32 * s + 8 * c]);
            const uint2 v2 = *reinterpret_cast<const uint2*>(&ring[stg][g + 8][32 * s + 8 * c]);
            ax[s][0] = k2.x; ax[s][2] = k2.y; ax[s][1] = v2.x; ax[s][3] = v2.y;
        }
        __syncwarp();
        {   // refill the stage with the tile after next
            const uint32_t t2 = tl + 2 * nwarps;
            if (t2 < tiles && t2 > tl) issue(t2, stg);
            asm volatile("cp.async.commit_group;");
        }
        // squared norms: x_m . x_n over the tile; row g's K norm is entry (g, g), its V norm (g + 8, g)
        float n1[4] = {0.f, 0.f, 0.f, 0.f}, n2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            mma_16816_x<DT>(n1, ax[s][0], ax[s][1], ax[s][2], ax[s][3], ax[s][0], ax[s][2]);
            mma_16816_x<DT>(n2, ax[s][0], ax[s][1], ax[s][2], ax[s][3], ax[s][1], ax[s][3]);
        }
        // D x: flip the signs of the coordinates whose sign is -1
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            ax[s][0] ^= msk[s][0]; ax[s][1] ^= msk[s][0];
            ax[s][2] ^= msk[s][1]; ax[s][3] ^= msk[s][1];
        }
        const int src_lane = 4 * g + (g >> 1);
        float kss = (g & 1) ? n1[1] : n1[0], vss = (g & 1) ? n2[3] : n2[2];
        kss = __shfl_sync(TQ_FULL_MASK, kss, src_lane);
        vss = __shfl_sync(TQ_FULL_MASK, vss, src_lane);
        const float kn = sqrtf(kss), vn = sqrtf(vss);
        // y = H D x / (sqrt(128) |x|): one multiplier per vector
        const float km = kn > 0.f ? 0.08838834764831845f * __frcp_rn(kn) : 0.f;
        const float vm = vn > 0.f ? 0.08838834764831845f * __frcp_rn(vn) : 0.f;

        uint32_t pc[8];   // codes of coordinates 16u + 4c .. +3: K at bits 0-11, V at 12-23
#pragma unroll
        for (int u = 0; u < 8; ++u) pc[u] = 0;
        const bool more = tl + nwarps < tiles && tl + nwarps > tl;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float acc[8][4];
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                acc[s][0] = acc[s][1] = acc[s][2] = acc[s][3] = 0.f;
                mma_16816_x<DT>(acc[s], ax[s][0], ax[s][1], ax[s][2], ax[s][3], hb[e][0], hb[e][1]);
            }
#pragma unroll
            for (int hs = 1; hs < 8; hs <<= 1) {
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    if (s & hs) continue;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float x = acc[s][i], y = acc[s + hs][i];
                        acc[s][i] = x + y;
                        acc[s + hs][i] = x - y;
                    }
                }
            }
            auto code_of = [&](float yn, const float* bd) -> uint32_t {
                if constexpr (TAB) {
                    // cell of yn: bits 3..9 of yn * 32 + 64 + 1.5 * 2^20 (steps of 1/8)
                    const float f = fmaf(yn, 32.f, kCellMagic);
                    const float2 en = tab[(__float_as_uint(f) & 0x3F8u) >> 3];
                    return __float_as_uint(en.y) + (yn > en.x ? 1u : 0u);
                } else {
                    return search_bits<3>(yn, bd);
                }
            };
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t k0 = code_of(acc[u][0] * km, kb), k1 = code_of(acc[u][1] * km, kb);
                const uint32_t v0 = code_of(acc[u][2] * vm, vb), v1 = code_of(acc[u][3] * vm, vb);
                pc[u] += ((k0 + (k1 << 3)) + ((v0 + (v1 << 3)) << 12)) << (6 * e);
            }
        }

        // records: lane pair (2m, 2m+1) holds 24 bits of K (the even lane writes
        // them) and of V (the odd lane) at record bytes 6u + 3m .. +2; the 16 records
        // of the tile are assembled in shared memory and leave as 16-byte stores
        int slot = -1;
        if (valid) {
            slot = a.start_pos[b] + t;
            if (slot < 0 || slot >= Tcap) {
                if (c == 0 && a.status) atomicOr(a.status, TQ_DEV_BAD_POSITION);
                slot = -1;
            }
        }
        if (!a.tiled) {   // the natural layout's records, assembled in shared memory
            const bool odd = c & 1;
            uint8_t* sr = &stage[2 * g + (odd ? 1 : 0)][3 * (c >> 1)];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t o = __shfl_xor_sync(TQ_FULL_MASK, pc[u], 1);
                const uint32_t w = odd ? ((o >> 12) & 0xFFFu) | (pc[u] & 0xFFF000u) : (pc[u] & 0xFFFu) | ((o & 0xFFFu) << 12);
                uint8_t* r = sr + 6 * u;
                if (c < 2) {
                    *reinterpret_cast<uint16_t*>(r) = (uint16_t)w;
                    r[2] = (uint8_t)(w >> 16);
                } else {
                    r[0] = (uint8_t)w;
                    *reinterpret_cast<uint16_t*>(r + 1) = (uint16_t)(w >> 8);
                }
            }
        }
        const size_t rec_i = (((size_t)b * Hkv + h) * a.t_alloc) + (slot < 0 ? 0 : slot);
        __syncwarp();
        if (a.tiled) {
            // Tile layout, from the codes in registers.  Lane (g, c) holds, for u = 0..7 and
            // e = 0, 1, the key and value fields of pairs 8u + 2c + e (pc[u] bits 6e.. and
            // 12 + 6e..).  Keys: such a field is slot 2u + (c >> 1) of lane column
            // 2 (c & 1) + e, so a key word holds fields of lanes c and c ^ 2: each builds
            // its bytes, one shuffle merges them, lane c stores column 2 (c & 1) + (c >> 1).
            // Values: the field is slot u of lane row 2c + e, so lane (g, c) builds the
            // whole value halves of rows 2c and 2c + 1.
            const int t = (int)(rec_i & 15);
            const size_t tile = rec_i >> 4;
            const int ch = c >> 1;
            uint32_t kw[2][3];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
#pragma unroll
                for (int w = 0; w < 3; ++w) {
                    uint32_t x = 0;
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const uint32_t f = (pc[2 * w + kk] >> (6 * e)) & 63u;
                        const uint32_t F = (pc[6 + kk] >> (6 * e)) & 63u;
                        x |= (tqtile::byte3(f, w) | tqtile::piece3(F, w)) << (8 * (ch + 2 * kk));
                    }
                    kw[e][w] = x;
                }
            }
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int w = 0; w < 3; ++w) kw[e][w] |= __shfl_xor_sync(TQ_FULL_MASK, kw[e][w], 2);
            if (slot >= 0) {
                uint8_t* kt = a.codes[0] + tile * tqtile::tile_bytes(3);
                const int L = 4 * (t & 7) + 2 * (c & 1) + ch;
#pragma unroll
                for (int w = 0; w < 3; ++w)
                    *reinterpret_cast<uint32_t*>(kt + tqtile::word_off(3, L, 3 * (t >> 3) + w)) = ch ? kw[1][w] : kw[0][w];
                uint8_t* vt = a.codes[1] + tile * tqtile::tile_bytes(3);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int Lv = 4 * (2 * c + e) + ((t & 7) >> 1);
#pragma unroll
                    for (int w = 0; w < 3; ++w) {
                        uint32_t x = 0;
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const uint32_t f = (pc[2 * w + j] >> (12 + 6 * e)) & 63u;
                            const uint32_t F = (pc[6 + j] >> (12 + 6 * e)) & 63u;
                            x |= (tqtile::byte3(f, w) | tqtile::piece3(F, w)) << (8 * j);
                        }
                        *reinterpret_cast<uint16_t*>(vt + tqtile::word_off(3, Lv, 3 * (t >> 3) + w) + 2 * (t & 1)) =
                            (uint16_t)x;
                    }
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < 2; ++k) {   // 48 chunks of 16 bytes: record q / 3, part q % 3
                const int q = lane + 32 * k;
                const int rr = (q < 48 ? q : 47) / 3, part = q - 3 * (q / 3);
                const int src = 4 * (rr >> 1);
                const int slot_r = __shfl_sync(TQ_FULL_MASK, slot, src);
                const unsigned long long ri = __shfl_sync(TQ_FULL_MASK, (unsigned long long)rec_i, src);
                if (q < 48 && slot_r >= 0) {
                    const uint4 v = *reinterpret_cast<const uint4*>(&stage[rr][16 * part]);
                    *reinterpret_cast<uint4*>(((rr & 1) ? a.codes[1] : a.codes[0]) + ri * 48 + 16 * part) = v;
                }
            }
        }
        __syncwarp();
        if (slot >= 0 && c < 2)
            static_cast<__half*>(c ? a.norms[1] : a.norms[0])[norm_index(a, c, rec_i, 1, 0)] =
                __float2half_rn(c ? vn : kn);

        if (!more) break;
        tl += nwarps;
        stg ^= 1;
        locate(tl);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Cell table of the codebook search: cell c holds yn with yn * 32 + 64 in
// [c - 1/8, c + 1] (the cell of the rounded value, widened by the rounding);
// entry c = (the boundary inside that interval or +inf, the number of boundaries
// below it).  Exact when no interval holds two boundaries: then
// #{k : yn > b_k} = idx0 + (yn > inner boundary).

template <int DT>
__global__ void __launch_bounds__(kTcWarps * 32, 4) tq_quantize_tc(QuantArgs a) {
    __shared__ __align__(16) uint8_t stage[kTcWarps][16][48];   // the tile's records: 2g K, 2g + 1 V
    __shared__ __align__(16) uint8_t ring[kTcWarps][2][16][kTcRow];
    __shared__ __align__(16) float2 tab[kCells];
    __shared__ int use_tab;
    const uint32_t tiles = (uint32_t)a.B * (uint32_t)a.Hkv * (((uint32_t)a.n_new + 7) / 8);
    if ((uint32_t)blockIdx.x * kTcWarps >= tiles) return;   // no tile for this CTA (uniform)
    if (threadIdx.x == 0) use_tab = 1;
    __syncthreads();
    // one table serves all heads when every head's K and V boundaries equal head 0's K boundaries
    const float* b0 = a.params[0].k_bound[0];
    for (int i = threadIdx.x; i < a.Hkv * 14; i += blockDim.x) {
        const tq_head_params& P = a.params[i / 14];
        const int k = i % 14;
        if ((k < 7 ? P.k_bound[0][k] : P.v_bound[0][k - 7]) != b0[k % 7]) use_tab = 0;
    }
    for (int cc = threadIdx.x; cc < kCells; cc += blockDim.x) {
        const float lo = ((float)cc - 64.125f) * 0.03125f, hi = ((float)cc - 63.f) * 0.03125f;
        int below = 0, inside = 0;
        float bnd = INFINITY;
        for (int k = 0; k < 7; ++k) {
            const float bk = b0[k];
            if (bk < lo) ++below;
            else if (bk <= hi) { ++inside; bnd = bk; }
        }
        if (inside > 1) use_tab = 0;
        tab[cc] = make_float2(bnd, __uint_as_float((uint32_t)below));
    }
    __syncthreads();
    const int w = threadIdx.x >> 5;
    if (use_tab) qtc_loop<DT, true>(a, tab, stage[w], ring[w]);
    else qtc_loop<DT, false>(a, tab, stage[w], ring[w]);
}

template <int ROT, int BITS>
void launch_half(unsigned g, cudaStream_t st, const QuantArgs& a) {
    if (a.in_dtype == TQ_F32) tq_quantize_half<ROT, BITS, TQ_F32><<<g, kWarps * 32, 0, st>>>(a);
    else if (a.in_dtype == TQ_F16) tq_quantize_half<ROT, BITS, TQ_F16><<<g, kWarps * 32, 0, st>>>(a);
    else tq_quantize_half<ROT, BITS, TQ_BF16><<<g, kWarps * 32, 0, st>>>(a);
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
    a.t_alloc = d->t_alloc;
    a.tiled = d->layout == TQ_LAYOUT_TILE16;
    a.in_dtype = in_dtype;
    a.norm_f16 = d->norm_dtype == TQ_F16;
    a.rot = d->rot;
    a.k_mixed = d->k_mixed;
    a.k_two = tq_two_stage(d) ? d->k_bits : 0;
    a.k_tight = d->k_mixed == 2;
    a.code_bytes[0] = d->k_code_bytes;
    a.code_bytes[1] = d->v_code_bytes;
    a.norm_slots[0] = d->k_norm_slots;
    a.norm_slots[1] = d->v_norm_slots;
    const long long warps = 2LL * d->batch * n_new * d->n_kv_heads;
    if (warps > 0x7fffffffLL) return TQ_ERR_INVALID_ARG;   // vector indices are 32-bit in the kernel
    long long blocks = (warps + kWarps - 1) / kWarps;
    if (blocks > kMaxBlocks) blocks = kMaxBlocks;   // warps loop over the rest
    const cudaStream_t st = (cudaStream_t)stream;
    const long long triples = warps / 2;
    if (!d->k_mixed && d->rot == TQ_ROT_WHT128 && d->k_bits == 3 && d->v_bits == 3 && d->norm_dtype == TQ_F16 &&
        d->k_norm_slots == 1 && d->v_norm_slots == 1 && (in_dtype == TQ_BF16 || in_dtype == TQ_F16) &&
        aligned(K, 16) && aligned(V, 16) && aligned(c->k_codes, 16) && aligned(c->v_codes, 16) &&
        triples >= kTcMinTriples && n_new >= 8) {
        // whole prompts: 16 vectors (K and V of 8 consecutive tokens of one head) per
        // warp through the tensor cores; warps loop over the tiles past one grid
        const long long ttiles = (long long)d->batch * d->n_kv_heads * ((n_new + 7) / 8);
        long long tb = (ttiles + kTcWarps - 1) / kTcWarps;
        if (tb > kTcMaxBlocks) tb = kTcMaxBlocks;
        if (in_dtype == TQ_BF16) tq_quantize_tc<TQ_BF16><<<(unsigned)tb, kTcWarps * 32, 0, st>>>(a);
        else tq_quantize_tc<TQ_F16><<<(unsigned)tb, kTcWarps * 32, 0, st>>>(a);
        return cudaPeekAtLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
    }
    if (!d->k_mixed && d->k_bits == d->v_bits && aligned(K, 16) && aligned(V, 16)) {
        const long long pairs = triples;   // one warp per (batch, token, KV head)
        long long hb = (pairs + kWarps - 1) / kWarps;
        if (hb > kMaxBlocks) {
            // warps loop over the rest; a warp count that is a multiple of the head
            // count keeps each warp on one KV head (its parameters load once)
            hb = kMaxBlocks;
            const int m = d->n_kv_heads / std::gcd(d->n_kv_heads, kWarps);
            if (hb >= m) hb -= hb % m;
        }
        const unsigned g = (unsigned)hb;
        const bool b4 = d->k_bits == 4;
        if (d->rot == TQ_ROT_WHT128) {
            if (b4) launch_half<TQ_ROT_WHT128, 4>(g, st, a);
            else launch_half<TQ_ROT_WHT128, 3>(g, st, a);
        } else if (d->rot == TQ_ROT_WHT32) {
            if (b4) launch_half<TQ_ROT_WHT32, 4>(g, st, a);
            else launch_half<TQ_ROT_WHT32, 3>(g, st, a);
        } else {
            if (b4) launch_half<TQ_ROT_SO4_WHT128, 4>(g, st, a);
            else launch_half<TQ_ROT_SO4_WHT128, 3>(g, st, a);
        }
        return cudaPeekAtLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
    }
    if (d->k_mixed || a.k_two) tq_quantize_kernel<-1><<<(unsigned)blocks, kWarps * 32, 0, st>>>(a);
    else if (d->rot == TQ_ROT_WHT128) tq_quantize_kernel<TQ_ROT_WHT128><<<(unsigned)blocks, kWarps * 32, 0, st>>>(a);
    else if (d->rot == TQ_ROT_WHT32) tq_quantize_kernel<TQ_ROT_WHT32><<<(unsigned)blocks, kWarps * 32, 0, st>>>(a);
    else if (d->rot == TQ_ROT_SO4_WHT128)
        tq_quantize_kernel<TQ_ROT_SO4_WHT128><<<(unsigned)blocks, kWarps * 32, 0, st>>>(a);
    else tq_quantize_kernel<-1><<<(unsigned)blocks, kWarps * 32, 0, st>>>(a);
    return cudaPeekAtLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
