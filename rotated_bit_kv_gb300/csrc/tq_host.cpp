// Host side of the library: Lloyd-Max codebook solver (fp64), RoPE block
// energies and greedy bit allocation, cache descriptor, parameter blob.
//
// Sources (page titles): [TQ-MNN] "TurboQuant: ... MNN runs it on the phone";
// [Block-GTQ] "RoPE-Aware Bit Allocation for KV-Cache Quantization";
// [RotaryQuant] "RotaryQuant: Fitting 120B MoE Models on Consumer Hardware via
// Fused Compressed-Space Attention".
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <vector>

#include "tq_internal.h"

namespace {

// ---------------------------------------------------------------------------
// Gauss-Legendre nodes on [-1, 1] by Newton iteration on P_n (three-term
// recurrence), computed once per call site (no global state).
struct GaussLegendre {
    static constexpr int N = 16;
    double x[N], w[N];
    GaussLegendre() {
        for (int i = 0; i < N; ++i) {
            double z = cos(M_PI * (i + 0.75) / (N + 0.5));
            for (int it = 0; it < 100; ++it) {
                double p0 = 1.0, p1 = z;
                for (int k = 2; k <= N; ++k) {
                    double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
                    p0 = p1;
                    p1 = p2;
                }
                double dp = N * (z * p1 - p0) / (z * z - 1.0);
                double dz = p1 / dp;
                z -= dz;
                if (fabs(dz) < 1e-17) break;
            }
            double p0 = 1.0, p1 = z;
            for (int k = 2; k <= N; ++k) {
                double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
                p0 = p1;
                p1 = p2;
            }
            double dp = N * (z * p1 - p0) / (z * z - 1.0);
            x[i] = z;
            w[i] = 2.0 / ((1.0 - z * z) * dp * dp);
        }
    }
};

// Moments of the unnormalised coordinate density (1 - t^2)^a over (lo, hi]
// [TQ-MNN §2.2, a = (d-3)/2].  With t = sin(th): dt (1-t^2)^a = cos^(2a+1) th dth,
// which is smooth on [-pi/2, pi/2] for a >= -1/2 (every d >= 2).  Composite
// Gauss-Legendre on panels narrower than the density's width in th.
struct Moments { double m0, m1; };

Moments cell_moments(const GaussLegendre& gl, double a, double lo, double hi) {
    double th0 = asin(lo), th1 = asin(hi);
    double e = 2.0 * a + 1.0;
    double h = 0.2 / sqrt(e + 1.0);
    int panels = (int)ceil((th1 - th0) / h);
    if (panels < 1) panels = 1;
    double ph = (th1 - th0) / panels;
    Moments m{0.0, 0.0};
    for (int p = 0; p < panels; ++p) {
        double c = th0 + (p + 0.5) * ph, r = 0.5 * ph;
        for (int i = 0; i < GaussLegendre::N; ++i) {
            double th = c + r * gl.x[i];
            double cs = cos(th);
            double f = (e == 0.0) ? 1.0 : pow(cs > 0.0 ? cs : 0.0, e);
            m.m0 += r * gl.w[i] * f;
            m.m1 += r * gl.w[i] * f * sin(th);
        }
    }
    return m;
}

// Standard normal quantile by bisection on erfc (initial guess only).
double normal_quantile(double p) {
    double lo = -40.0, hi = 40.0;
    for (int i = 0; i < 200; ++i) {
        double mid = 0.5 * (lo + hi);
        if (0.5 * erfc(-mid / sqrt(2.0)) < p) lo = mid; else hi = mid;
    }
    return 0.5 * (lo + hi);
}

// fp64 Lloyd-Max iteration [TQ-MNN §2.3]: boundaries are midpoints of the
// centroids; each centroid is the conditional mean of its cell.
tq_status lloyd_max(int d, int bits, double* c) {
    const int K = 1 << bits;
    const double a = (d - 3) / 2.0;
    GaussLegendre gl;
    for (int k = 0; k < K; ++k) {
        double g = normal_quantile((k + 0.5) / K) / sqrt((double)d);
        c[k] = fmax(-0.95, fmin(0.95, g));
    }
    std::vector<double> nc(K);
    for (int it = 0; it < 200000; ++it) {
        double delta = 0.0;
        for (int k = 0; k < K; ++k) {
            double lo = k == 0 ? -1.0 : 0.5 * (c[k - 1] + c[k]);
            double hi = k == K - 1 ? 1.0 : 0.5 * (c[k] + c[k + 1]);
            Moments m = cell_moments(gl, a, lo, hi);
            nc[k] = m.m1 / m.m0;
        }
        // f is even, so the fixed point is odd-symmetric: mirror the halves so
        // that the middle boundary is exactly 0 and c_k = -c_(K-1-k) exactly.
        for (int k = 0; k < K / 2; ++k) {
            const double s = 0.5 * (nc[K - 1 - k] - nc[k]);
            nc[k] = -s;
            nc[K - 1 - k] = s;
        }
        for (int k = 0; k < K; ++k) {
            delta = fmax(delta, fabs(nc[k] - c[k]));
            c[k] = nc[k];
        }
        if (delta < 1e-15) return TQ_OK;
    }
    return TQ_ERR_NO_CONVERGENCE;
}

// fp16 round-to-nearest-even of a positive normal value (11 significant bits).
double round_half(double x) {
    int e;
    const double m = frexp(x, &e);                 // [0.5, 1)
    return ldexp(nearbyint(ldexp(m, 11)), e - 11);
}

// Scale s in [1, 2) for which the fp16 roundings of s * c_k (via fp32, as the
// kernels compute them) have the smallest worst relative error.  Tensor-core
// kernels keep the codebook as fp16 and fold 1/s into their fp32 norm factors,
// so the codebook itself enters the products almost exactly.
float fp16_table_scale(const float* cent, int K) {
    double best_err = 1e30;
    float best = 1.0f;
    for (int i = 0; i < (1 << 16); ++i) {
        const float sc = (float)(1.0 + i / 65536.0);
        double err = 0.0;
        for (int k = 0; k < K; ++k) {
            const double v = fabs((double)(sc * cent[k]));
            if (v == 0.0) continue;
            err = fmax(err, fabs(round_half(v) - v) / v);
        }
        if (err < best_err) { best_err = err; best = sc; }
    }
    return best;
}

// Codebooks solved during one tq_params_build call, keyed by (d, bits).
struct CodebookMemo {
    struct Entry { int d, bits; float cent[16], bound[16], hscale; };
    std::vector<Entry> e;
    tq_status get(int d, int bits, const float** cent, const float** bound, float* hscale = nullptr) {
        for (auto& x : e)
            if (x.d == d && x.bits == bits) {
                *cent = x.cent; *bound = x.bound;
                if (hscale) *hscale = x.hscale;
                return TQ_OK;
            }
        Entry n{};
        n.d = d;
        n.bits = bits;
        tq_status st = tq_codebook(d, bits, n.cent, n.bound);
        if (st != TQ_OK) return st;
        n.hscale = fp16_table_scale(n.cent, 1 << bits);
        e.push_back(n);
        *cent = e.back().cent;
        *bound = e.back().bound;
        if (hscale) *hscale = e.back().hscale;
        return TQ_OK;
    }
};

}  // namespace

extern "C" {

const char* tq_status_string(tq_status s) {
    switch (s) {
        case TQ_OK: return "TQ_OK";
        case TQ_ERR_INVALID_ARG: return "TQ_ERR_INVALID_ARG";
        case TQ_ERR_UNSUPPORTED: return "TQ_ERR_UNSUPPORTED";
        case TQ_ERR_CUDA: return "TQ_ERR_CUDA";
        case TQ_ERR_NO_CONVERGENCE: return "TQ_ERR_NO_CONVERGENCE";
        case TQ_ERR_WORKSPACE: return "TQ_ERR_WORKSPACE";
        default: return "TQ_ERR_UNKNOWN";
    }
}

int tq_v_crossover(const tq_cache_desc* d) {
    const char* s = getenv("TQ_V_CROSSOVER");
    if (s && *s) {
        long v = strtol(s, nullptr, 10);
        if (v >= 0 && v < (1L << 30)) return (int)v;
    }
    // Measured on GB300 for each natural-layout format (16 query heads per KV
    // head; fp32 norms with 32-wide blocks; fp32 norms with mixed-rate keys; tight
    // mixed-rate records; two-stage keys) over T = 64 .. 4096: dimension-parallel
    // accumulation is as fast or faster at every length (the pages' T = 512 crossover comes from a GPU without the
    // key-axis split), so the crossover is 0 for all of them.
    (void)d;
    return 0;
}

tq_status tq_codebook(int32_t block_dim, int32_t bits, float* centroids, float* boundaries) {
    if (!centroids || !boundaries || block_dim < 2 || block_dim > 4096 || bits < 1 || bits > 4)
        return TQ_ERR_INVALID_ARG;
    double c[16];
    tq_status st = lloyd_max(block_dim, bits, c);
    if (st != TQ_OK) return st;
    const int K = 1 << bits;
    for (int k = 0; k < K; ++k) centroids[k] = (float)c[k];
    for (int k = 0; k + 1 < K; ++k) boundaries[k] = (float)(0.5 * (c[k] + c[k + 1]));
    return TQ_OK;
}

tq_status tq_block_energy(const float* q_cal, const float* k_cal, int32_t T, int32_t G,
                          int32_t head_dim, double* s_out) {
    if (!q_cal || !k_cal || !s_out || T < 1 || G < 1 || head_dim < 2 || (head_dim & 1))
        return TQ_ERR_INVALID_ARG;
    const int L = head_dim / 2;
    std::vector<double> sq(L, 0.0), sk(L, 0.0);
    for (int t = 0; t < T; ++t) {
        for (int g = 0; g < G; ++g) {
            const float* q = q_cal + ((size_t)t * G + g) * head_dim;
            for (int i = 0; i < L; ++i) {
                double a = q[2 * i], b = q[2 * i + 1];
                sq[i] += a * a + b * b;
            }
        }
        const float* k = k_cal + (size_t)t * head_dim;
        for (int i = 0; i < L; ++i) {
            double a = k[2 * i], b = k[2 * i + 1];
            sk[i] += a * a + b * b;
        }
    }
    for (int i = 0; i < L; ++i) s_out[i] = 0.5 * (sq[i] / ((double)T * G) + sk[i] / (double)T);
    return TQ_OK;
}

tq_status tq_block_bit_alloc(const double* s, int32_t L, int32_t b_min, int32_t b_max,
                             int32_t B_total, int32_t* b_out) {
    if (!s || !b_out || L < 1 || b_min < 0 || b_min > b_max || b_max > 30) return TQ_ERR_INVALID_ARG;
    if ((int64_t)B_total < (int64_t)L * b_min || (int64_t)B_total > (int64_t)L * b_max)
        return TQ_ERR_INVALID_ARG;
    for (int i = 0; i < L; ++i) {
        if (!(s[i] >= 0.0)) return TQ_ERR_INVALID_ARG;
        b_out[i] = b_min;
    }
    // Delta_i = (3/4) s_i 4^(-b_i): the decrease of J when block i gets one
    // more bit; it falls by 4x after each bit, so the greedy order is optimal.
    for (int64_t extra = (int64_t)B_total - (int64_t)L * b_min; extra > 0; --extra) {
        int best = -1;
        double best_gain = -1.0;
        for (int i = 0; i < L; ++i) {
            if (b_out[i] >= b_max) continue;
            double gain = 0.75 * s[i] * ldexp(1.0, -2 * b_out[i]);
            if (gain > best_gain) { best = i; best_gain = gain; }
        }
        b_out[best] += 1;
    }
    return TQ_OK;
}

tq_status tq_cache_desc_init(tq_cache_desc* d, int32_t head_dim, int32_t n_q_heads,
                             int32_t n_kv_heads, int32_t batch, int32_t t_capacity, int32_t rot,
                             int32_t k_bits, int32_t v_bits, int32_t norm_dtype, int32_t k_mixed) {
    if (!d) return TQ_ERR_INVALID_ARG;
    memset(d, 0, sizeof(*d));
    if (head_dim <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || batch <= 0 || t_capacity <= 0)
        return TQ_ERR_INVALID_ARG;
    if (n_q_heads % n_kv_heads) return TQ_ERR_INVALID_ARG;
    if (rot != TQ_ROT_WHT128 && rot != TQ_ROT_WHT32 && rot != TQ_ROT_SO4_WHT128) return TQ_ERR_INVALID_ARG;
    if (norm_dtype != TQ_F16 && norm_dtype != TQ_F32) return TQ_ERR_INVALID_ARG;
    if (k_mixed < 0 || k_mixed > 2) return TQ_ERR_INVALID_ARG;
    if (head_dim != TQ_HEAD_DIM) return TQ_ERR_UNSUPPORTED;
    if (n_q_heads / n_kv_heads > TQ_MAX_GROUP) return TQ_ERR_UNSUPPORTED;
    if (v_bits != 3 && v_bits != 4) return TQ_ERR_UNSUPPORTED;
    // two-stage keys [TQ-MNN §2.4]: (k_bits - 1)-bit MSE code + 1-bit QJL code
    const bool two = !k_mixed && (k_bits == 1 || k_bits == 2);
    if (!k_mixed && !two && k_bits != 3 && k_bits != 4) return TQ_ERR_UNSUPPORTED;
    if (!k_mixed && !two && k_bits != v_bits) return TQ_ERR_UNSUPPORTED;   // one kernel per shared width
    if ((k_mixed || two) && rot == TQ_ROT_WHT32) return TQ_ERR_UNSUPPORTED;
    // tight mixed-rate records: k_bits is the average bits per coordinate
    const bool tight = k_mixed == 2;
    if (tight && k_bits != 2 && k_bits != 3) return TQ_ERR_UNSUPPORTED;
    if ((int64_t)batch * n_kv_heads * t_capacity > (int64_t)1 << 40) return TQ_ERR_INVALID_ARG;
    d->head_dim = head_dim;
    d->n_q_heads = n_q_heads;
    d->n_kv_heads = n_kv_heads;
    d->batch = batch;
    d->t_capacity = t_capacity;
    d->rot = rot;
    d->k_bits = k_mixed == 1 ? 0 : k_bits;
    d->v_bits = v_bits;
    d->norm_dtype = norm_dtype;
    d->k_mixed = k_mixed;
    d->group = n_q_heads / n_kv_heads;
    d->k_code_bytes = tight ? 16 * k_bits : k_mixed ? 64 : two ? 16 * k_bits : (k_bits == 3 ? 48 : 64);
    d->v_code_bytes = v_bits == 3 ? 48 : 64;
    d->k_norm_slots = (k_mixed || rot == TQ_ROT_WHT32) ? 4 : two ? 2 : 1;
    d->v_norm_slots = rot == TQ_ROT_WHT32 ? 4 : 1;
    d->norm_bytes = norm_dtype == TQ_F16 ? 2 : 4;
    // the tile layout (read by the tensor-core decode kernel) for every format it
    // covers: at most 8 query heads per KV head, fp16 norms where a vector has
    // four (the 32-wide blocks, mixed-rate keys), not two-stage keys or tight records
    const bool tile = d->group <= 8 && !two && !tight && !((rot == TQ_ROT_WHT32 || k_mixed) && norm_dtype != TQ_F16);
    d->layout = tile ? TQ_LAYOUT_TILE16 : TQ_LAYOUT_NATURAL;
    const int64_t alloc = tile ? ((int64_t)t_capacity + 15) / 16 * 16 : t_capacity;
    if (alloc > 0x7fffffff) return TQ_ERR_INVALID_ARG;
    d->t_alloc = (int32_t)alloc;
    d->params_bytes = tq_params_blob_bytes(n_kv_heads, k_mixed || two);
    return TQ_OK;
}

size_t tq_cache_bytes(const tq_cache_desc* d, int32_t part) {
    if (!d || d->head_dim != TQ_HEAD_DIM) return 0;
    size_t vecs = (size_t)d->batch * d->n_kv_heads * d->t_alloc;
    switch (part) {
        case TQ_PART_K_CODES: return vecs * d->k_code_bytes;
        case TQ_PART_K_NORMS: return vecs * d->k_norm_slots * d->norm_bytes;
        case TQ_PART_V_CODES: return vecs * d->v_code_bytes;
        case TQ_PART_V_NORMS: return vecs * d->v_norm_slots * d->norm_bytes;
        case TQ_PART_PARAMS: return (size_t)d->params_bytes;
        default: return 0;
    }
}

tq_status tq_params_build(const tq_cache_desc* d, const float* signs, const float* quats,
                          const int32_t* k_block_bits, const float* k_group_mats, void* host_blob) {
    if (!d || !host_blob || d->head_dim != TQ_HEAD_DIM) return TQ_ERR_INVALID_ARG;
    const bool need_signs = d->rot == TQ_ROT_WHT128 || d->rot == TQ_ROT_WHT32;
    if (need_signs && !signs) return TQ_ERR_INVALID_ARG;
    if (d->rot == TQ_ROT_SO4_WHT128 && !quats) return TQ_ERR_INVALID_ARG;
    if (d->k_mixed && (!k_block_bits || !k_group_mats)) return TQ_ERR_INVALID_ARG;
    const bool two = tq_two_stage(d);
    if (two && !k_group_mats) return TQ_ERR_INVALID_ARG;
    memset(host_blob, 0, (size_t)d->params_bytes);
    tq_head_params* hp = (tq_head_params*)host_blob;
    float* kmat_all = (float*)((char*)host_blob + (size_t)d->n_kv_heads * sizeof(tq_head_params));
    CodebookMemo memo;
    const float* mats = k_group_mats;
    for (int h = 0; h < d->n_kv_heads; ++h) {
        tq_head_params& p = hp[h];
        for (int i = 0; i < 128; ++i) p.signs[i] = signs ? signs[h * 128 + i] : 1.0f;
        if (quats)
            for (int b = 0; b < 32; ++b)
                for (int j = 0; j < 8; ++j) p.quat[b][j] = quats[((size_t)h * 32 + b) * 8 + j];
        // V segments
        const int vseg = d->rot == TQ_ROT_WHT32 ? 4 : 1;
        const int vlen = 128 / vseg;
        p.v_nseg = vseg;
        for (int s = 0; s <= 4; ++s) p.v_seg_start[s] = s < vseg ? s * vlen : 128;
        for (int s = 0; s < vseg; ++s) {
            const float *c, *bd;
            tq_status st = memo.get(vlen, d->v_bits, &c, &bd, &p.v_h_scale[s]);
            if (st != TQ_OK) return st;
            p.v_seg_bits[s] = d->v_bits;
            memcpy(p.v_cent[s], c, sizeof(float) * 16);
            memcpy(p.v_bound[s], bd, sizeof(float) * 16);
        }
        if (two) {
            // one 128-wide segment with the (k_bits - 1)-bit codebook (none for
            // k_bits = 1); the projection S goes where mixed-rate keys keep k_mat
            p.k_nseg = 1;
            for (int s = 0; s <= 4; ++s) p.k_seg_start[s] = s < 1 ? 0 : 128;
            p.k_seg_bits[0] = d->k_bits - 1;
            if (d->k_bits == 2) {
                const float *c, *bd;
                tq_status st = memo.get(128, 1, &c, &bd, &p.k_h_scale[0]);
                if (st != TQ_OK) return st;
                memcpy(p.k_cent[0], c, sizeof(float) * 16);
                memcpy(p.k_bound[0], bd, sizeof(float) * 16);
            }
            for (int i = 0; i < 128; ++i) p.k_gcoord[i] = i;
            // stored transposed (column c of S contiguous) for coalesced reads
            float* st = kmat_all + (size_t)h * 128 * 128;
            const float* sm = k_group_mats + (size_t)h * 128 * 128;
            for (int j = 0; j < 128; ++j)
                for (int c = 0; c < 128; ++c) st[(size_t)c * 128 + j] = sm[(size_t)j * 128 + c];
        } else if (!d->k_mixed) {
            const int kseg = d->rot == TQ_ROT_WHT32 ? 4 : 1;
            const int klen = 128 / kseg;
            p.k_nseg = kseg;
            for (int s = 0; s <= 4; ++s) p.k_seg_start[s] = s < kseg ? s * klen : 128;
            for (int s = 0; s < kseg; ++s) {
                const float *c, *bd;
                tq_status st = memo.get(klen, d->k_bits, &c, &bd, &p.k_h_scale[s]);
                if (st != TQ_OK) return st;
                p.k_seg_bits[s] = d->k_bits;
                memcpy(p.k_cent[s], c, sizeof(float) * 16);
                memcpy(p.k_bound[s], bd, sizeof(float) * 16);
            }
            for (int i = 0; i < 128; ++i) p.k_gcoord[i] = i;
        } else {
            // same-width groups in ascending width [Block-GTQ]; block i is
            // coordinates (2i, 2i+1)
            const int32_t* bb = k_block_bits + (size_t)h * 64;
            int spent = 0;
            for (int i = 0; i < 64; ++i) {
                if (bb[i] < 1 || bb[i] > 4) return TQ_ERR_INVALID_ARG;
                spent += bb[i];
            }
            if (d->k_mixed == 2 && spent != 64 * d->k_bits) return TQ_ERR_INVALID_ARG;   // fills the tight record
            float* kmat = kmat_all + (size_t)h * 128 * 128;
            int pos = 0;
            p.k_nseg = 4;
            for (int b = 1; b <= 4; ++b) {
                const int s = b - 1;
                p.k_seg_start[s] = pos;
                p.k_seg_bits[s] = b;
                int n = 0;
                for (int i = 0; i < 64; ++i)
                    if (bb[i] == b) {
                        p.k_gcoord[pos + n] = 2 * i;
                        p.k_gcoord[pos + n + 1] = 2 * i + 1;
                        n += 2;
                    }
                if (n) {
                    const float *c, *bd;
                    tq_status st = memo.get(n, b, &c, &bd, &p.k_h_scale[s]);
                    if (st != TQ_OK) return st;
                    memcpy(p.k_cent[s], c, sizeof(float) * 16);
                    memcpy(p.k_bound[s], bd, sizeof(float) * 16);
                    for (int r = 0; r < n; ++r)
                        for (int cc = 0; cc < n; ++cc) kmat[(size_t)(pos + r) * 128 + pos + cc] = mats[(size_t)r * n + cc];
                    mats += (size_t)n * n;
                }
                pos += n;
            }
            p.k_seg_start[4] = pos;   // == 128
        }
    }
    return TQ_OK;
}

}  // extern "C"
