/*
 * tq.h -- C ABI of the GB300 (sm_103a) rotation-quantised KV cache library.
 *
 * The library implements one data-parallel hot path, in two halves:
 *
 *   write side  (tq_quantize_append): per K/V vector, L2 norm -> orthogonal
 *               rotation -> per-coordinate Lloyd-Max codebook search -> 3/4-bit
 *               packing into a caller-owned device cache;
 *   read side   (tq_decode_attention): rotate q once, QK dot products on the
 *               packed codes by codebook lookup, online softmax, V accumulation
 *               in the rotated domain, log-sum-exp merge of key-axis splits, one
 *               inverse rotation of the output.
 *
 * Sources, by page title (sections as printed on each page):
 *   [TQ-MNN]      "TurboQuant: ... MNN runs it on the phone" (zhaode.wang blog)
 *   [RotaryQuant] "RotaryQuant: Fitting 120B MoE Models on Consumer Hardware via
 *                 Fused Compressed-Space Attention" (papernotes.org)
 *   [Block-GTQ]   "RoPE-Aware Bit Allocation for KV-Cache Quantization" (aitrends.kr)
 *
 * Conventions shared by every entry point
 *   - head_dim is 128.  q head g reads KV head g / (n_q_heads / n_kv_heads).
 *   - Every pointer named d_* (and every pointer inside tq_cache_ptrs, q, out,
 *     workspace) is DEVICE memory owned by the caller; the library never
 *     allocates, frees or retains a pointer past the call.  Host pointers are
 *     read during the call only.
 *   - Device entry points are asynchronous and stream ordered on `stream` (a
 *     cudaStream_t passed as void*; NULL = the legacy default stream).  They
 *     return TQ_OK after a successful launch; argument errors that the host can
 *     see are returned before anything is launched.  Conditions only the device
 *     can see (a sequence length above the cache capacity, a write position
 *     outside the cache) are clamped or skipped, never trapped, and OR a
 *     TQ_DEV_* bit into *d_status when d_status is not NULL.
 *   - Apart from tq_decode_attention_noalloc (a fixed scratch array shared by
 *     all its calls, which must therefore be ordered on one stream) the library
 *     keeps no global mutable state: calls on different streams with disjoint
 *     buffers are independent.
 *   - The tensor-core decode kernel is launched as a programmatic dependent of
 *     the kernel before it on the stream: its blocks may be placed while that
 *     kernel finishes, and wait on the device for its completion before they
 *     read anything.  The order the caller sees is the plain stream order.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */
typedef int32_t tq_status;
#define TQ_OK                  0
#define TQ_ERR_INVALID_ARG     1  /* bad shape, pointer, enum or size          */
#define TQ_ERR_UNSUPPORTED     2  /* valid but not built (e.g. head_dim != 128) */
#define TQ_ERR_CUDA            3  /* a CUDA runtime call or launch failed       */
#define TQ_ERR_NO_CONVERGENCE  4  /* the Lloyd-Max iteration did not converge   */
#define TQ_ERR_WORKSPACE       5  /* workspace missing or smaller than required */

/* bits OR-ed into the caller's device status word */
#define TQ_DEV_SEQ_OVER_CAPACITY  1  /* seq_len > t_capacity: clamped          */
#define TQ_DEV_SEQ_OVER_MAX       2  /* seq_len > max_seq_len: clamped         */
#define TQ_DEV_BAD_POSITION       4  /* append position outside [0, capacity): skipped */
#define TQ_DEV_INTERNAL           8  /* a kernel's own layout check failed: output not written */
#define TQ_DEV_BAD_METADATA      16  /* a ZipFusion page offset outside its pool: page 0 read instead */

/* ---------------------------------------------------------------- enums */
#define TQ_F32   0
#define TQ_F16   1
#define TQ_BF16  2

/* Rotation kinds.  R is orthogonal; rotated = R x.
 *   WHT128      R = H_128 D, D = diag(+-1 signs)      [TQ-MNN §3.1]
 *   WHT32       R = diag(H_32 D_k), k = 0..3, each block with its own norm
 *                                                      [TQ-MNN §3.1, block_size = 32]
 *   SO4_WHT128  R = S H_128, S = diag of 32 maps v -> q_L v conj(q_R)
 *                                                      [RotaryQuant, Key design 2]
 * Mixed-rate keys (k_mixed = 1) replace K's rotation by one random orthogonal
 * matrix per same-width group of RoPE blocks [Block-GTQ, physical encoding and
 * grouping]; V keeps `rot`.
 * Two-stage keys (k_bits 1 or 2) [TQ-MNN §2.4]: K keeps `rot` for a
 * (k_bits - 1)-bit MSE code of y = R x / ||x|| and adds a 1-bit QJL code of its
 * residual r = y - C[idx]: the signs of S r for a caller-drawn Gaussian
 * projection S, from which <q~, r> is estimated without bias as
 * ||r|| sqrt(pi/2) / 128 <S q~, sign(S r)>. */
#define TQ_ROT_WHT128      0
#define TQ_ROT_WHT32       1
#define TQ_ROT_SO4_WHT128  2

/* parts of the cache, for tq_cache_bytes */
#define TQ_PART_K_CODES  0
#define TQ_PART_K_NORMS  1
#define TQ_PART_V_CODES  2
#define TQ_PART_V_NORMS  3
#define TQ_PART_PARAMS   4

/* V-accumulation strategies of the decode kernel [RotaryQuant, Key design 3:
 * token ("word") parallel below a crossover length, dimension parallel above] */
#define TQ_VMODE_AUTO            -1
#define TQ_VMODE_TOKEN_PARALLEL   0
#define TQ_VMODE_DIM_PARALLEL     1
#define TQ_VMODE_TENSOR           2  /* dimension parallel on tensor cores (tile layout) */
#define TQ_VMODE_TENSOR_STREAMK   3  /* same kernel as TQ_VMODE_TENSOR (kept as an alias) */

/* Cache layouts (tq_cache_desc.layout, chosen by tq_cache_desc_init) */
#define TQ_LAYOUT_NATURAL  0  /* one packed record per token, token-major             */
#define TQ_LAYOUT_TILE16   1  /* 16-token tiles in the order the decode kernel reads */

#define TQ_HEAD_DIM     128
#define TQ_MAX_GROUP     16   /* maximum n_q_heads / n_kv_heads */
#define TQ_MAX_SPLITS  1024   /* maximum key-axis splits per (batch, KV head) */

/* ---------------------------------------------------------------- layout */
/* Cache descriptor.  Filled by tq_cache_desc_init; treat as read-only.
 *
 * Code records.  The record of one vector holds its 128 indices in rotated-
 * coordinate order: 3-bit indices LSB first (index i at bits [3i, 3i+3) of the
 * little-endian byte stream: 8 indices per 3 bytes, 48 B) or 4-bit indices two
 * per byte (index 2j in the low nibble of byte j, 64 B) [TQ-MNN §3.3].  Mixed-
 * rate keys use the 4-bit container for every width (one index per nibble) with
 * the groups in ascending bit width [Block-GTQ, packed cache].  A "field" is the
 * pair of indices of coordinates (2i, 2i+1): bits [6i, 6i+6) (3-bit) or byte i
 * (4-bit) of the record.  Norm slots: 1 (WHT128, SO4_WHT128), 4 (WHT32: one per
 * 32-dim block) or 4 (mixed-rate keys: slot b-1 holds the norm of the b-bit
 * group, 0 if empty).
 *
 * Tight mixed-rate keys (k_mixed = 2): each code at its group's width b, the
 * groups in ascending width as above, concatenated LSB first (position p at bit
 * offset sum_{p' < p} b_p'), k_bits * 16 bytes for an average of k_bits (2 or 3)
 * bits per coordinate [Block-GTQ, packed cache]; four norm slots as above.
 *
 * Two-stage keys (k_bits 1 or 2): (k_bits - 1) * 16 bytes of 1-bit MSE codes
 * (index i at bit i, LSB first; none for k_bits = 1), then 16 bytes of signs
 * (bit j = 1 iff (S r)_j >= 0): 16 or 32 B.  Two norm slots: ||x|| and
 * ||x|| * ||r||.
 *
 * Positions per (batch, KV head): t_alloc = t_capacity rounded up to a multiple
 * of 16 (TQ_LAYOUT_TILE16) or t_capacity (TQ_LAYOUT_NATURAL).  Every array is
 * [batch][n_kv_heads][t_alloc positions] of per-position data:
 *   k_codes, v_codes  k_code_bytes / v_code_bytes per position, uint8
 *   k_norms, v_norms  k_norm_slots / v_norm_slots per position, norm_dtype
 *
 * TQ_LAYOUT_NATURAL (more than 8 query heads per KV head, fp32 norms with four
 * slots: WHT32 or mixed-rate keys, tight mixed-rate keys, or two-stage keys):
 * position t holds the record and norms of token t.
 *
 * TQ_LAYOUT_TILE16 (every other cache): positions come in tiles of 16; tile j of
 * a (batch, KV head) holds tokens 16j .. 16j+15 in 16 * code_bytes bytes of codes
 * and 16 * slots norms, arranged as the decode kernel's 32 lanes read them.
 * Lane L = 4r + c (r = 0..7, c = 0..3) owns 2W words of a code tile (W = 3 for
 * 3-bit, 4 for 4-bit): words 0..3 at byte 16L, words 4..2W-1 at byte
 * 512 + 8(W-2)L.
 *   keys:   words 0..W-1 hold token r, words W..2W-1 token r+8; a token's W
 *           words in lane L hold its fields s = 0..15 of pairs
 *           i = 8(s>>1) + c + 4(s&1).
 *   values: words 0..W-1 hold token 2c in their low 16-bit halves and token
 *           2c+1 in their high halves, words W..2W-1 tokens 2c+8 and 2c+9; a
 *           token's W halves in lane L hold its fields q = 0..7 of pairs
 *           16(q>>1) + r + 8(q&1).
 *   4-bit: key field s is byte s&3 of word s>>2; value field q is byte q&1 of
 *           half q>>1.
 *   3-bit: key fields 0..11 and value fields 0..5 have a byte each (key: byte
 *           s&3 of word s>>2; value: byte q&1 of half q>>1); in the bytes of the
 *           token's first and third word the field is bits 0-5, in those of its
 *           second word field bits 0-1 are byte bits 0-1 and field bits 2-5 byte
 *           bits 4-7.  Key fields 12..15 (value fields 6, 7) are spread over byte
 *           lane g = s-12 (q-6) of the token's three words: field bits 0-1 in
 *           bits 6-7 of the first word's byte, bits 2-3 in bits 2-3 of the
 *           second's, bits 4-5 in bits 6-7 of the third's.
 *   mixed-rate keys: the 4-bit key layout, with a b-bit code c of a group of
 *           width b < 4 stored as c + 2^b (so its nibble, 2-3, 4-7 or 8-15,
 *           names its width); codes of the 4-bit group are stored as they are.
 *   norms:  one slot: token t at element 2(t&7) + (t>>3) of the tile; four
 *           slots: keys (2(t&7) + (t>>3))*4 + b, values
 *           ((((t&7)>>1)*2 + (t>>3))*4 + b)*2 + (t&1).
 * Each key word and each value half belongs to one token, so appends of single
 * tokens never rewrite another token's bytes. */
typedef struct tq_cache_desc {
    int32_t head_dim;
    int32_t n_q_heads;
    int32_t n_kv_heads;
    int32_t batch;
    int32_t t_capacity;
    int32_t rot;            /* TQ_ROT_* */
    int32_t k_bits;         /* 3 or 4; 1 or 2: two-stage keys (ignored when k_mixed) */
    int32_t v_bits;         /* 3 or 4 */
    int32_t norm_dtype;     /* TQ_F16 or TQ_F32 */
    int32_t k_mixed;        /* 0; 1: nibble records; 2: tight records (k_bits = average bits) */
    /* derived */
    int32_t group;          /* n_q_heads / n_kv_heads */
    int32_t k_code_bytes;
    int32_t v_code_bytes;
    int32_t k_norm_slots;
    int32_t v_norm_slots;
    int32_t norm_bytes;     /* 2 or 4 */
    int32_t layout;         /* TQ_LAYOUT_* */
    int32_t t_alloc;        /* positions per (batch, KV head) (see above) */
    int64_t params_bytes;   /* size of the parameter blob (tq_params_build) */
} tq_cache_desc;

/* Device pointers of one cache (caller owned; see layout above).  `params` is
 * a device copy of the blob written by tq_params_build; it must be 16-byte
 * aligned. */
typedef struct tq_cache_ptrs {
    void* k_codes;
    void* k_norms;
    void* v_codes;
    void* v_norms;
    const void* params;
} tq_cache_ptrs;

/* ---------------------------------------------------------------- host API */

/* Human-readable name of a status code (static string, never NULL). */
const char* tq_status_string(tq_status s);

/* Lloyd-Max codebook for one coordinate of a uniformly random point on the unit
 * sphere in R^block_dim, density f(t) ~ (1 - t^2)^((block_dim-3)/2) on [-1, 1]
 * [TQ-MNN §2.2], with 2^bits cells: each centroid is the conditional mean of
 * its cell, each boundary the midpoint of its neighbours [TQ-MNN §2.3].
 * Solved in fp64 on the host, returned rounded to fp32.
 *   block_dim   2..4096 (128, 32, or a mixed-rate group width)
 *   bits        1..4
 *   centroids   host, 2^bits floats, ascending
 *   boundaries  host, 2^bits - 1 floats (midpoints of the fp64 centroids)
 * Errors: TQ_ERR_INVALID_ARG (range, NULL), TQ_ERR_NO_CONVERGENCE. */
tq_status tq_codebook(int32_t block_dim, int32_t bits, float* centroids, float* boundaries);

/* Block energy of each two-dimensional RoPE block i (coordinates 2i, 2i+1) for
 * one KV head [Block-GTQ, block energy]:
 *   s_i = 1/2 ( mean_{t, g} ||q_{g,t}^(i)||^2 + mean_t ||k_t^(i)||^2 ),
 * over a calibration prefix of T tokens; g runs over the G query heads that
 * read this KV head.
 *   q_cal  host fp32 [T][G][head_dim];  k_cal host fp32 [T][head_dim]
 *   s_out  host fp64 [head_dim / 2]
 * Errors: TQ_ERR_INVALID_ARG. */
tq_status tq_block_energy(const float* q_cal, const float* k_cal, int32_t T, int32_t G,
                          int32_t head_dim, double* s_out);

/* Greedy integer bit allocation [Block-GTQ, greedy allocation]: minimise
 * J(b) = sum_i s_i 4^(-b_i) subject to b_min <= b_i <= b_max and
 * sum_i b_i = B_total.  Every block starts at b_min; each remaining bit goes to
 * the block with the largest marginal gain (3/4) s_i 4^(-b_i) among blocks below
 * b_max (ties to the lowest index).
 *   s      host fp64 [L] (s_i >= 0);  b_out host int32 [L]
 * Errors: TQ_ERR_INVALID_ARG (NULL, L < 1, b_min > b_max, infeasible B_total). */
tq_status tq_block_bit_alloc(const double* s, int32_t L, int32_t b_min, int32_t b_max,
                             int32_t B_total, int32_t* b_out);

/* Fill a cache descriptor and validate the shape.
 *   k_bits  3 or 4 (the same as v_bits), or 1 or 2 for two-stage keys
 *           (WHT128 or SO4_WHT128, any v_bits); ignored when k_mixed = 1; the
 *           average bits per coordinate (2 or 3) when k_mixed = 2
 *   v_bits  3 or 4
 *   k_mixed 0: uniform keys; 1: mixed-rate keys in nibble records; 2: mixed-rate
 *           keys in tight records (the allocation must spend k_bits * 64 block
 *           bits per KV head)
 * Errors: TQ_ERR_INVALID_ARG (non-positive sizes, n_q_heads not a multiple of
 * n_kv_heads, bad enum), TQ_ERR_UNSUPPORTED (head_dim != 128, group >
 * TQ_MAX_GROUP, bits outside the sets above, k_bits 3/4 different from v_bits,
 * WHT32 combined with k_mixed or with two-stage keys). */
tq_status tq_cache_desc_init(tq_cache_desc* desc, int32_t head_dim, int32_t n_q_heads,
                             int32_t n_kv_heads, int32_t batch, int32_t t_capacity,
                             int32_t rot, int32_t k_bits, int32_t v_bits,
                             int32_t norm_dtype, int32_t k_mixed);

/* Bytes of one part of the cache (TQ_PART_*); 0 for an unknown part. */
size_t tq_cache_bytes(const tq_cache_desc* desc, int32_t part);

/* Build the parameter blob (rotation parameters and codebooks, per KV head)
 * into host memory of desc->params_bytes bytes; the caller copies it to a
 * 16-byte aligned device buffer and passes it as tq_cache_ptrs.params.  The
 * random quantities of the method are inputs, drawn by the caller:
 *   signs        host fp32 [n_kv][128], each +1 or -1 (WHT128, WHT32, and the
 *                V rotation of mixed-rate caches); may be NULL for SO4_WHT128
 *   quats        host fp32 [n_kv][32][2][4]: (q_L, q_R) unit quaternions
 *                (w, x, y, z) per 4-dim block; required for SO4_WHT128
 *   k_block_bits host int32 [n_kv][64]: bits of each RoPE block, 1..4; required
 *                iff k_mixed
 *   k_group_mats host fp32: for each KV head, for each width b = 1..4 whose
 *                group is non-empty (n_b = 2 * #blocks), the n_b x n_b
 *                row-major orthogonal matrix Pi_b, concatenated; required iff
 *                k_mixed.  With k_mixed = 2 every head's k_block_bits must sum to
 *                k_bits * 64 (TQ_ERR_INVALID_ARG otherwise).  For two-stage keys (k_bits 1 or 2): the QJL
 *                projections S, [n_kv][128][128] row-major (row j gives sign
 *                bit j), entries i.i.d. N(0, 1) drawn by the caller; required
 * Codebooks are solved here (tq_codebook) for every (width, bits) in use.
 * Errors: TQ_ERR_INVALID_ARG, TQ_ERR_NO_CONVERGENCE. */
tq_status tq_params_build(const tq_cache_desc* desc, const float* signs, const float* quats,
                          const int32_t* k_block_bits, const float* k_group_mats,
                          void* host_blob);

/* ---------------------------------------------------------------- device API */

/* Quantise and append n_new tokens of K and V per sequence [TQ-MNN §2.1 and
 * §3.3 "in-place quantisation on write"; Block-GTQ: a whole prompt in one
 * call].  For every (b, t, h) and both K and V: n = ||x|| per norm segment,
 * y = R x / n, idx = #{k : y > boundary_k} (fp32 compares, ties to the lower
 * cell) [TQ-MNN §3.4], pack, store the norm rounded to norm_dtype.
 * Two-stage keys [TQ-MNN §2.4]: the same on the (k_bits - 1)-bit codebook (no
 * search for k_bits = 1), then r = y - C[idx], z = S r in fp32, sign bits
 * z_j >= 0, norms ||x|| and ||x|| * ||r||.
 *   K, V         device [batch][n_new][n_kv_heads][128] of in_dtype
 *   in_dtype     TQ_F32, TQ_F16 or TQ_BF16
 *   d_start_pos  device int32 [batch]: token t goes to slot d_start_pos[b] + t;
 *                slots outside [0, t_capacity) are skipped and flagged
 *   n_new        >= 0 (0 is a no-op)
 *   d_status     device int32 or NULL
 * Errors: TQ_ERR_INVALID_ARG (NULL, misaligned, bad dtype), TQ_ERR_CUDA. */
tq_status tq_quantize_append(const tq_cache_desc* desc, const tq_cache_ptrs* cache,
                             const void* K, const void* V, int32_t in_dtype,
                             const int32_t* d_start_pos, int32_t n_new,
                             int32_t* d_status, void* stream);

/* Workspace bytes tq_decode_attention needs for at most max_splits key-axis
 * splits: partial (m, l, o~) per (batch, q head, split) plus one ticket per
 * (batch, KV head).  For TQ_LAYOUT_TILE16 caches it also covers the tensor-core
 * kernel's partials (one per CTA and piece of a pair: at most 1216 + batch *
 * n_kv_heads slots), so max_splits = 1 is enough for the automatic plan.  The
 * ticket words must be zero before the first call on a workspace (e.g. a
 * cudaMemset of the whole buffer); every call leaves them zero again. */
size_t tq_decode_workspace_bytes(const tq_cache_desc* desc, int32_t max_splits);

/* One decode step of attention on the packed cache [RotaryQuant, Key design 3;
 * TQ-MNN §3.3 K path and V path; Block-GTQ key-axis split with log-sum-exp
 * merge].  For each batch b and q head g of KV head h:
 *   q~ = R_K q;  s_j = sum_seg n_{j,seg} <q~_seg, C_seg[idx_{j,seg}]> / sqrt(128)
 *   a = softmax(s) over j < seq_len_b;  o~ = sum_j a_j v~_j;  o = R_V^T o~.
 * Two-stage keys [TQ-MNN §2.4]: s_j = (n_j <q~, C[idx_j]> + n_j rho_j
 * sqrt(pi/2) / 128 <S q~, 2 sign_j - 1>) / sqrt(128), with S q~ formed once per
 * query head.
 *   q            device [batch][n_q_heads][128] of q_dtype (TQ_F32/F16/BF16)
 *   d_seq_lens   device int32 [batch]; clamped to [0, min(t_capacity,
 *                max_seq_len)] with TQ_DEV_* flags; seq_len 0 gives o = 0
 *   max_seq_len  host upper bound of d_seq_lens, 1..t_capacity; sizes the
 *                key-axis splits and picks the V-accumulation mode
 *   out          device fp32 [batch][n_q_heads][128]
 *   workspace    device, >= tq_decode_workspace_bytes(desc, splits used); the
 *                splits used are at most TQ_MAX_SPLITS and at most
 *                ceil(max_seq_len / 64) (1 for TQ_LAYOUT_TILE16 caches)
 *   d_status     device int32 or NULL
 * Errors: TQ_ERR_INVALID_ARG, TQ_ERR_WORKSPACE, TQ_ERR_CUDA. */
tq_status tq_decode_attention(const tq_cache_desc* desc, const tq_cache_ptrs* cache,
                              const void* q, int32_t q_dtype, const int32_t* d_seq_lens,
                              int32_t max_seq_len, float* out, void* workspace,
                              size_t workspace_bytes, int32_t* d_status, void* stream);

/* tq_decode_attention with explicit choices, for tests and tuning:
 *   v_mode    TQ_VMODE_*.  TQ_LAYOUT_TILE16 caches run the tensor-core kernel
 *             (AUTO, TENSOR or TENSOR_STREAMK); TQ_LAYOUT_NATURAL caches run
 *             the CUDA-core kernels (AUTO: token parallel below the format's
 *             crossover length, dimension parallel from it on; the crossover
 *             measured on GB300 is 0 for every natural-layout format, so AUTO
 *             is dimension parallel; the environment variable TQ_V_CROSSOVER
 *             overrides it; or either kernel explicitly).
 *   n_splits  0 for the automatic choice; else, CUDA-core kernels: key-axis
 *             splits per (batch, KV head), 1..TQ_MAX_SPLITS; tensor-core
 *             kernel: the number of CTAs the tiles of all pairs are divided
 *             over, 1..1216
 * Errors: as tq_decode_attention; TQ_ERR_UNSUPPORTED if v_mode asks for a
 * kernel that does not read the cache's layout. */
tq_status tq_decode_attention_ex(const tq_cache_desc* desc, const tq_cache_ptrs* cache,
                                 const void* q, int32_t q_dtype, const int32_t* d_seq_lens,
                                 int32_t max_seq_len, float* out, void* workspace,
                                 size_t workspace_bytes, int32_t* d_status, void* stream,
                                 int32_t v_mode, int32_t n_splits);

/* tq_decode_attention for callers that cannot allocate device memory.  The
 * pages have no counterpart to this entry point; it exists for callers that
 * must not call cudaMalloc: code running inside another framework's memory
 * pool, plugins that are given only their input and output buffers, and paths
 * where an allocation would synchronise the device.  The split-K scratch (the
 * per-split partials and the per-(batch, KV head) tickets) is a fixed 8 MiB
 * array inside the library's device image, held by every GPU that loads the
 * library until the process exits; nothing is allocated or freed.
 *   Arguments as tq_decode_attention, without the workspace; the plan is the
 *   automatic one (same splits and V mode as tq_decode_attention).
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any
 *   stream capture.
 *   Every call zeroes the ticket words on `stream` before the kernel; the
 *   partials are overwritten.  All calls share the one array, so calls whose
 *   kernels can overlap on the GPU (concurrent streams, several host threads)
 *   race and corrupt each other: order them on one stream.
 * Errors: as tq_decode_attention; TQ_ERR_WORKSPACE when the plan needs more
 * scratch than tq_decode_noalloc_max_scratch_bytes() (reduce batch * KV heads
 * or use tq_decode_attention with a workspace). */
tq_status tq_decode_attention_noalloc(const tq_cache_desc* desc, const tq_cache_ptrs* cache,
                                      const void* q, int32_t q_dtype, const int32_t* d_seq_lens,
                                      int32_t max_seq_len, float* out, int32_t* d_status,
                                      void* stream);

/* Size in bytes of the fixed scratch array behind tq_decode_attention_noalloc. */
size_t tq_decode_noalloc_max_scratch_bytes(void);

/* Decode attention over two parts of each sequence's keys: a block of
 * unquantised tokens (the prompt's K and V kept in fp16/bf16: deferred prefill
 * [RotaryQuant, IsoQuant decode flow]; or the recent-token buffer [Block-GTQ,
 * limitations]) and the packed cache.  The set of keys attended is the union of
 * the two parts: the first d_prefix_lens[b] unquantised tokens and the first
 * d_seq_lens[b] packed tokens of batch b.  The packed part is attended as by
 * tq_decode_attention (automatic plan), which also leaves each head's log2-sum-
 * exp in the workspace; the unquantised part is attended in the original domain
 * (scores q k / sqrt(d) in fp32 from the stored values) and the two are merged
 * by log-sum-exp [Block-GTQ, key-axis split with log-sum-exp merge].
 *   k_prefix, v_prefix  device, 16-byte aligned, [batch][prefix_capacity]
 *                [n_kv_heads][128] of prefix_dtype (TQ_F32, TQ_F16 or TQ_BF16),
 *                the layout of tq_quantize_append's input; may be NULL when
 *                max_prefix_len = 0.  Up to 8 query heads per KV head the
 *                scores and the value sum run on tensor cores with fp16
 *                operands (bf16 / fp32 values are rounded to fp16: they must
 *                lie in fp16 range) and fp32 accumulation; above 8, in fp32
 *   d_prefix_lens  device int32 [batch]; values above prefix_capacity or
 *                max_prefix_len are clamped (TQ_DEV_SEQ_OVER_CAPACITY /
 *                TQ_DEV_SEQ_OVER_MAX); 0 = no unquantised token
 *   max_seq_len  0 (no packed token: cache and d_seq_lens are not read) up to
 *                t_capacity
 *   max_prefix_len  0 .. prefix_capacity
 *   workspace    device, 256-byte aligned, at least
 *                tq_decode_prefix_workspace_bytes(desc, max_prefix_len) bytes,
 *                zero-filled before its first use; every call leaves it so
 *   out          device fp32 [batch][n_q_heads][128]; a head with no key at all
 *                gets zeros
 * Two kernels on `stream` (the second a programmatic dependent of the first).
 * Errors: TQ_ERR_INVALID_ARG (NULL, misaligned, range), TQ_ERR_WORKSPACE, the
 * errors of tq_decode_attention, TQ_ERR_CUDA. */
tq_status tq_decode_attention_prefix(const tq_cache_desc* desc, const tq_cache_ptrs* cache,
                                     const void* q, int32_t q_dtype,
                                     const int32_t* d_seq_lens, int32_t max_seq_len,
                                     const void* k_prefix, const void* v_prefix,
                                     int32_t prefix_dtype, int32_t prefix_capacity,
                                     const int32_t* d_prefix_lens, int32_t max_prefix_len,
                                     float* out, void* workspace, size_t workspace_bytes,
                                     int32_t* d_status, void* stream);

/* ---------------------------------------------------------------- ZipFusion
 * A lossless store of bf16 K/V and decode attention on it [ZipFusion:
 * compression format; register restore; attention kernel].
 *
 * Pages of 16 tokens of one (batch, KV head), for K and V separately; a page's
 * 2048 values are four 512-value blocks (block j = tokens 4j .. 4j+3, values in
 * (token, coordinate) order).  A block whose exponent fields all lie in
 * [b, b + 15], b = their minimum rounded down to even, is compressed to 768 B:
 * its 512 low bytes (7 mantissa bits and the exponent's lowest bit), then 256
 * code bytes, one byte per pair of values of a group of 8 (values g8+k and g8+k+4,
 * k = 0..3): sign of the first in bit 7 and d = (e - b) >> 1 in bits 0-2, sign of
 * the second in bit 6 and its d in bits 3-5; restore: high byte = 128 sign + b/2
 * + d.  Other blocks, and every block of a page that is not full, stay raw (1024 B
 * of bf16).  Blocks follow one another from the page's offset.  Metadata, 8 bytes
 * per page: uint32 offset of block 0 from the pool base in 256-byte units, then
 * one byte per block: b/2, or 0xFF for raw.
 * Pools hold one 4096-byte slot per page (page (b, h, p) at slot
 * (b * n_kv_heads + h) * (t_capacity / 16) + p); the metadata offset lets a
 * memory manager place pages elsewhere (not part of this library). */

/* Bytes of one pool (K or V) and of one metadata array for a store of
 * t_capacity tokens (a multiple of 16) per (batch, KV head); 0 on bad sizes. */
size_t tq_zip_pool_bytes(int32_t batch, int32_t n_kv_heads, int32_t t_capacity);
size_t tq_zip_meta_bytes(int32_t batch, int32_t n_kv_heads, int32_t t_capacity);

/* Store the first d_lens[b] tokens of K and V of every sequence as pages.
 *   K, V        device bf16 [batch][n_tokens][n_kv_heads][128], 16-byte aligned
 *   d_lens      device int32 [batch]; values above t_capacity or n_tokens are
 *               clamped (TQ_DEV_SEQ_OVER_CAPACITY)
 *   k_pool, v_pool  device, 256-byte aligned, tq_zip_pool_bytes each
 *   k_meta, v_meta  device, 8-byte aligned, tq_zip_meta_bytes each; pages past
 *               a sequence's length are not written
 * Errors: TQ_ERR_INVALID_ARG (NULL, misaligned, sizes), TQ_ERR_CUDA. */
tq_status tq_zip_store(const void* K, const void* V, int32_t batch, int32_t n_kv_heads, int32_t n_tokens,
                       int32_t t_capacity, const int32_t* d_lens, void* k_pool, void* v_pool, void* k_meta,
                       void* v_meta, int32_t* d_status, void* stream);

/* Workspace of tq_zip_decode_attention (0: unsupported shape). */
size_t tq_zip_workspace_bytes(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads, int32_t max_seq_len);

/* Decode attention over stored pages: softmax(q K^T / sqrt(128)) V over the first
 * d_seq_lens[b] tokens, the blocks restored in registers and fed to the tensor
 * cores (fp16 operands, fp32 accumulation; bf16 values must lie in fp16 range).
 *   q           device [batch][n_q_heads][128] of q_dtype; at most 8 query heads
 *               per KV head (else TQ_ERR_UNSUPPORTED)
 *   d_seq_lens  device int32 [batch] (clamped to max_seq_len and t_capacity; the
 *               pages read must have been stored); max_seq_len 1 .. t_capacity
 *   workspace   tq_zip_workspace_bytes, 256-byte aligned, zero-filled before its
 *               first use (every call leaves it so)
 *   out         device fp32 [batch][n_q_heads][128]
 * A page offset outside its pool reads page 0 and ORs TQ_DEV_BAD_METADATA.
 * Errors: TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_WORKSPACE, TQ_ERR_CUDA. */
tq_status tq_zip_decode_attention(const void* q, int32_t q_dtype, int32_t batch, int32_t n_q_heads,
                                  int32_t n_kv_heads, int32_t t_capacity, const void* k_pool,
                                  const void* v_pool, const void* k_meta, const void* v_meta,
                                  const int32_t* d_seq_lens, int32_t max_seq_len, float* out,
                                  void* workspace, size_t workspace_bytes, int32_t* d_status,
                                  void* stream);

/* Workspace bytes of tq_decode_attention_prefix for at most max_prefix_len
 * unquantised tokens per sequence (0 on a bad descriptor). */
size_t tq_decode_prefix_workspace_bytes(const tq_cache_desc* desc, int32_t max_prefix_len);

/* The splits and V mode tq_decode_attention would use (host only).  For the
 * tensor-core kernel *splits_out is the number of CTAs (the 16-token tiles of
 * all (batch, KV head) pairs, in pair order, are divided evenly over them; the
 * pieces of a pair are merged by the last CTA to finish it), 0 when the
 * device's occupancy is not known yet (no call has run on it). */
tq_status tq_decode_plan(const tq_cache_desc* desc, int32_t max_seq_len, int32_t v_mode,
                         int32_t n_splits, int32_t* splits_out, int32_t* v_mode_out);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H_ */
