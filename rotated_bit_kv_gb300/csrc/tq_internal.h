// Internal layout shared by the host code and the kernels (not part of the ABI).
#pragma once
#include <stdint.h>

#include "tq.h"

// Per-KV-head parameter record of the blob built by tq_params_build.
// A "segment" is a run of rotated coordinates [start, start + len) of a code
// record that shares one stored norm (slot = segment index) and one codebook.
//   WHT128 / SO4_WHT128 : 1 segment of 128 (codebook for d = 128)
//   WHT32               : 4 segments of 32 (codebook for d = 32)
//   mixed-rate keys     : segment s = bit width s + 1, length n_b (possibly 0),
//                         codebook for d = n_b
//   two-stage keys      : 1 segment of 128 with k_bits - 1 bits (0: no MSE code)
struct alignas(16) tq_head_params {
    float signs[128];         // +-1 of the sign-flipped WHT
    float quat[32][8];        // per 4-dim block: q_L (w,x,y,z), q_R (w,x,y,z)
    int32_t k_seg_start[5];   // k_seg_start[4] == 128
    int32_t k_seg_bits[4];
    int32_t k_nseg;
    int32_t v_seg_start[5];
    int32_t v_seg_bits[4];
    int32_t v_nseg;
    float k_h_scale[4];       // fp16 table scale of segment s (see tq_params_build)
    float v_h_scale[4];
    int32_t pad0[4];
    float k_cent[4][16];      // ascending centroids of segment s
    float k_bound[4][16];     // 2^bits - 1 boundaries of segment s
    float v_cent[4][16];
    float v_bound[4][16];
    int32_t k_gcoord[128];    // mixed-rate keys: original coordinate feeding
                              // concatenated input position p of the groups
};
static_assert(sizeof(tq_head_params) % 16 == 0, "params record must stay 16-byte aligned");

// For mixed-rate keys the blob continues with float k_mat[n_kv][128][128]:
// rotated[r] = sum_c k_mat[r][c] * x[k_gcoord[c]], block diagonal (segment s
// occupies rows and columns [k_seg_start[s], k_seg_start[s+1])).  For two-stage
// keys the same place holds the QJL projections transposed: ST[n_kv][128][128]
// with ST[c][j] = S[j][c] (S's row j gives sign bit j).
static inline int64_t tq_params_blob_bytes(int n_kv, int has_kmat) {
    return (int64_t)n_kv * (int64_t)sizeof(tq_head_params) +
           (has_kmat ? (int64_t)n_kv * 128 * 128 * 4 : 0);
}

// Two-stage keys: a (k_bits - 1)-bit MSE code plus a 1-bit QJL code.
static inline bool tq_two_stage(const tq_cache_desc* d) {
    return !d->k_mixed && (d->k_bits == 1 || d->k_bits == 2);
}

// Key/value code formats used to select kernels.
enum tq_fmt : int {
    TQ_FMT_ONE3 = 0,   // one 128-wide segment, 3-bit codes (48 B)
    TQ_FMT_ONE4 = 1,   // one 128-wide segment, 4-bit codes (64 B)
    TQ_FMT_BLK3 = 2,   // four 32-wide segments, 3-bit codes (48 B)
    TQ_FMT_BLK4 = 3,   // four 32-wide segments, 4-bit codes (64 B)
    TQ_FMT_MIX4 = 4,   // runtime segments, one code per nibble (64 B)
    TQ_FMT_QJ1 = 5,    // two-stage keys, k_bits 1: 128 sign bits (16 B)
    TQ_FMT_QJ2 = 6,    // two-stage keys, k_bits 2: 128 one-bit codes + 128 sign bits (32 B)
    TQ_FMT_MXT2 = 7,   // mixed-rate keys, tight records, 2 bits on average (32 B)
    TQ_FMT_MXT3 = 8,   // mixed-rate keys, tight records, 3 bits on average (48 B)
};

static inline int tq_k_fmt(const tq_cache_desc* d) {
    if (d->k_mixed == 2) return d->k_bits == 2 ? TQ_FMT_MXT2 : TQ_FMT_MXT3;
    if (d->k_mixed) return TQ_FMT_MIX4;
    if (tq_two_stage(d)) return d->k_bits == 1 ? TQ_FMT_QJ1 : TQ_FMT_QJ2;
    if (d->rot == TQ_ROT_WHT32) return d->k_bits == 3 ? TQ_FMT_BLK3 : TQ_FMT_BLK4;
    return d->k_bits == 3 ? TQ_FMT_ONE3 : TQ_FMT_ONE4;
}
static inline int tq_v_fmt(const tq_cache_desc* d) {
    if (d->rot == TQ_ROT_WHT32) return d->v_bits == 3 ? TQ_FMT_BLK3 : TQ_FMT_BLK4;
    return d->v_bits == 3 ? TQ_FMT_ONE3 : TQ_FMT_ONE4;
}

// Host helpers implemented in tq_host.cpp.
#ifdef __cplusplus
extern "C" {
#endif
int tq_v_crossover(const tq_cache_desc* d);   // V-mode crossover length of a natural-layout
                                              // format (TQ_V_CROSSOVER env overrides)
#ifdef __cplusplus
}
#endif

// Decode attention with an optional per-head log2-sum-exp output (lse: device fp32
// [batch][n_q_heads], log2 units of q log2(e) / sqrt(d), or NULL); implemented in
// tq_decode.cu, used by tq_decode_attention_ex and the prefix entry point.
tq_status tq_decode_run(const tq_cache_desc* d, const tq_cache_ptrs* c, const void* q, int32_t q_dtype,
                        const int32_t* d_seq_lens, int32_t max_seq_len, float* out, void* workspace,
                        size_t workspace_bytes, int32_t* d_status, void* stream, int32_t v_mode, int32_t n_splits,
                        float* lse);
