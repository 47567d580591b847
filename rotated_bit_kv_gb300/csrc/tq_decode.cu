// Read side: decode attention computed on the packed codes.
//
// [RotaryQuant] Key design 3: rotate q once (<Rq, Rk> = q^T k), QK dot products
// and V accumulation on the packed codes in on-chip registers, one inverse
// rotation of the output (o~ = R o); V accumulation token ("word") parallel for
// short contexts, dimension parallel for long ones.  [TQ-MNN] §3.3: K path in
// the rotated domain (q rotated once per head, unpack + codebook lookup +
// multiply-add per key), V path accumulated in the rotated domain with one
// inverse WHT.  [Block-GTQ]: long contexts split along the key axis, sections
// merged by log-sum-exp.
//
// Grid: (split, KV head, batch); 128 threads.  Each CTA rotates the G query
// heads of its KV head into shared memory, streams its section of the cache,
// and leaves a partial (m, l, o~) per query head.  The last CTA of a (batch,
// KV head) to finish -- found with an atomic ticket, no spinning -- merges the
// sections and applies R_V^T.
#include <stdlib.h>


#include "tq_decode_cc.cuh"

// Two-stage keys (tq_decode_two_stage.cu) and tight mixed-rate key records
// (tq_decode_tight.cu): the kernel for (padded group, key format, value format,
// V mode), or null.
KernelFn tq_two_stage_kernel(int GP, int kf, int vf, int mode);
KernelFn tq_tight_kernel(int GP, int kf, int vf, int mode);

namespace {
template <int GP>
KernelFn pick_fmt(int kf, int vf, int mode) {
    if (kf == TQ_FMT_ONE3 && vf == TQ_FMT_ONE3) return pick_mode<GP, TQ_FMT_ONE3, TQ_FMT_ONE3>(mode);
    if (kf == TQ_FMT_ONE4 && vf == TQ_FMT_ONE4) return pick_mode<GP, TQ_FMT_ONE4, TQ_FMT_ONE4>(mode);
    if (kf == TQ_FMT_BLK3 && vf == TQ_FMT_BLK3) return pick_mode<GP, TQ_FMT_BLK3, TQ_FMT_BLK3>(mode);
    if (kf == TQ_FMT_BLK4 && vf == TQ_FMT_BLK4) return pick_mode<GP, TQ_FMT_BLK4, TQ_FMT_BLK4>(mode);
    if (kf == TQ_FMT_MIX4 && vf == TQ_FMT_ONE3) return pick_mode<GP, TQ_FMT_MIX4, TQ_FMT_ONE3>(mode);
    if (kf == TQ_FMT_MIX4 && vf == TQ_FMT_ONE4) return pick_mode<GP, TQ_FMT_MIX4, TQ_FMT_ONE4>(mode);
    return nullptr;
}

KernelFn pick_kernel(int G, int kf, int vf, int mode, int* GP) {
    if (kf == TQ_FMT_QJ1 || kf == TQ_FMT_QJ2) {
        *GP = G <= 1 ? 1 : G <= 4 ? 4 : G <= 8 ? 8 : 16;
        return tq_two_stage_kernel(*GP, kf, vf, mode);
    }
    if (kf == TQ_FMT_MXT2 || kf == TQ_FMT_MXT3) {
        *GP = G <= 1 ? 1 : G <= 4 ? 4 : G <= 8 ? 8 : 16;
        return tq_tight_kernel(*GP, kf, vf, mode);
    }
    if (G <= 1) { *GP = 1; return pick_fmt<1>(kf, vf, mode); }
    if (G <= 4) { *GP = 4; return pick_fmt<4>(kf, vf, mode); }
    if (G <= 8) { *GP = 8; return pick_fmt<8>(kf, vf, mode); }
    *GP = 16;
    return pick_fmt<16>(kf, vf, mode);
}

int padded_group(int G) { return G <= 1 ? 1 : G <= 4 ? 4 : G <= 8 ? 8 : 16; }

bool aligned(const void* p, size_t n) { return ((uintptr_t)p % n) == 0; }

constexpr int kSMs = 152;

}  // namespace

extern "C" {

size_t tq_decode_workspace_bytes(const tq_cache_desc* d, int32_t max_splits) {
    if (!d || d->head_dim != TQ_HEAD_DIM || max_splits < 1) return 0;
    if (max_splits > TQ_MAX_SPLITS) max_splits = TQ_MAX_SPLITS;
    const size_t pairs = (size_t)d->batch * d->n_kv_heads;
    size_t slots = pairs * (size_t)max_splits;
    if (tq_decode_tc_supported(d)) {   // room for the tensor-core kernel's stream-K partials
        const size_t sk = (size_t)tq_decode_tc_sk_slots(d);
        if (sk > slots) slots = sk;
    }
    // the tensor-core kernel's partials hold 4 or 8 heads (its head groups)
    const int gp = tq_decode_tc_supported(d) ? (d->group <= 4 ? 4 : 8) : padded_group(d->group);
    const size_t part = slots * (size_t)gp * kPartStride * sizeof(float);
    const size_t tick = ((pairs * sizeof(int32_t)) + 255) & ~(size_t)255;
    return tick + part;
}

tq_status tq_decode_plan(const tq_cache_desc* d, int32_t max_seq_len, int32_t v_mode, int32_t n_splits,
                         int32_t* splits_out, int32_t* v_mode_out) {
    if (!d || d->head_dim != TQ_HEAD_DIM || max_seq_len < 1 || max_seq_len > d->t_capacity) return TQ_ERR_INVALID_ARG;
    if (v_mode < TQ_VMODE_AUTO || v_mode > TQ_VMODE_TENSOR_STREAMK) return TQ_ERR_INVALID_ARG;
    if (n_splits < 0 || n_splits > TQ_MAX_SPLITS) return TQ_ERR_INVALID_ARG;
    int mode = v_mode == TQ_VMODE_TENSOR_STREAMK ? TQ_VMODE_TENSOR : v_mode;
    if (tq_decode_tc_supported(d)) {
        // tile layout: the tensor-core kernel, at every length (measured faster than
        // the token-parallel kernel down to T = 128)
        if (mode == TQ_VMODE_AUTO) mode = TQ_VMODE_TENSOR;
        if (mode != TQ_VMODE_TENSOR) return TQ_ERR_UNSUPPORTED;
        if (n_splits > tq_decode_tc_max_grid()) return TQ_ERR_INVALID_ARG;
        if (splits_out) *splits_out = n_splits > 0 ? n_splits : tq_decode_tc_sk_grid(d, max_seq_len);
        if (v_mode_out) *v_mode_out = mode;
        return TQ_OK;
    }
    // natural layout: token-parallel below the format's measured crossover,
    // dimension-parallel from it on
    if (mode == TQ_VMODE_TENSOR) return TQ_ERR_UNSUPPORTED;
    if (mode == TQ_VMODE_AUTO) mode = max_seq_len < tq_v_crossover(d) ? TQ_VMODE_TOKEN_PARALLEL : TQ_VMODE_DIM_PARALLEL;
    int splits = n_splits;
    const long long pairs = (long long)d->batch * d->n_kv_heads;
    if (splits == 0) {
        // about 1.6 times the sections that fill the GPU once (four resident
        // 128-thread CTAs per SM), at most 128 partials per pair (the last CTA
        // merges them after the rest: past ~128 the merge costs more than the
        // shorter sections save, as measured on the dimension-parallel kernel),
        // sections of at least 64 tokens
        const long long fill = (4LL * kSMs + pairs - 1) / pairs;
        long long sp = (fill * 8 + 4) / 5;
        if (sp > 128) sp = 128;
        const long long cap = (max_seq_len + 63) / 64;
        if (sp > cap) sp = cap;
        if (sp < 1) sp = 1;
        if (sp > TQ_MAX_SPLITS) sp = TQ_MAX_SPLITS;
        splits = (int)sp;
    }
    if (splits_out) *splits_out = splits;
    if (v_mode_out) *v_mode_out = mode;
    return TQ_OK;
}

}  // extern "C"

// Decode attention with an optional per-head log2-sum-exp output (lse, [batch][n_q]
// fp32 device or null), shared by tq_decode_attention_ex and the prefix entry.
tq_status tq_decode_run(const tq_cache_desc* d, const tq_cache_ptrs* c, const void* q, int32_t q_dtype,
                        const int32_t* d_seq_lens, int32_t max_seq_len, float* out, void* workspace,
                        size_t workspace_bytes, int32_t* d_status, void* stream, int32_t v_mode, int32_t n_splits,
                        float* lse) {
    if (!d || !c || d->head_dim != TQ_HEAD_DIM) return TQ_ERR_INVALID_ARG;
    if (!q || !d_seq_lens || !out || !c->k_codes || !c->k_norms || !c->v_codes || !c->v_norms || !c->params)
        return TQ_ERR_INVALID_ARG;
    if (q_dtype != TQ_F32 && q_dtype != TQ_F16 && q_dtype != TQ_BF16) return TQ_ERR_INVALID_ARG;
    const size_t qa = q_dtype == TQ_F32 ? 16 : 8;
    if (!aligned(q, qa) || !aligned(out, 16) || !aligned(c->k_codes, 16) || !aligned(c->v_codes, 16) ||
        !aligned(c->params, 16) || !aligned(c->k_norms, 16) || !aligned(c->v_norms, 16))
        return TQ_ERR_INVALID_ARG;
    int splits = 0, mode = 0;
    tq_status st = tq_decode_plan(d, max_seq_len, v_mode, n_splits, &splits, &mode);
    if (st != TQ_OK) return st;
    const bool tc = mode == TQ_VMODE_TENSOR;
    if (tc && splits < 1) return TQ_ERR_CUDA;   // the device's occupancy could not be read
    const int kf = tq_k_fmt(d), vf = tq_v_fmt(d);
    int GP = 1;
    KernelFn fn = nullptr;
    if (!tc) {
        fn = pick_kernel(d->group, kf, vf, mode, &GP);
        if (!fn) return TQ_ERR_UNSUPPORTED;
    }
    DecodeArgs a;
    a.k_codes = static_cast<const uint8_t*>(c->k_codes);
    a.k_norms = c->k_norms;
    a.v_codes = static_cast<const uint8_t*>(c->v_codes);
    a.v_norms = c->v_norms;
    a.params = static_cast<const tq_head_params*>(c->params);
    a.kmat = reinterpret_cast<const float*>(static_cast<const char*>(c->params) +
                                            (size_t)d->n_kv_heads * sizeof(tq_head_params));
    a.q = q;
    a.seq_lens = d_seq_lens;
    a.out = out;
    a.lse = lse;
    a.status = d_status;
    a.tickets = nullptr;
    a.ws_part = nullptr;
    if (splits > 1) {   // tensor core: several CTAs may share a pair
        const size_t need = tq_decode_workspace_bytes(d, tc ? 1 : splits);
        if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return TQ_ERR_WORKSPACE;
        const size_t pairs = (size_t)d->batch * d->n_kv_heads;
        const size_t tick = ((pairs * sizeof(int32_t)) + 255) & ~(size_t)255;
        a.tickets = static_cast<int32_t*>(workspace);
        a.ws_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + tick);
    }
    a.B = d->batch;
    a.Hq = d->n_q_heads;
    a.Hkv = d->n_kv_heads;
    a.G = d->group;
    a.Tcap = d->t_alloc;
    a.t_cap = d->t_capacity;
    a.max_seq = max_seq_len;
    a.n_splits = tc ? 0 : splits;
    a.split_len = tc ? 0 : (max_seq_len + splits - 1) / splits;
    a.q_dtype = q_dtype;
    a.norm_f16 = d->norm_dtype == TQ_F16;
    a.rot = d->rot;
    a.k_mixed = d->k_mixed;
    a.fold_mul = 1u << 20;
    if (d->batch > 65535 || d->n_kv_heads > 65535) return TQ_ERR_INVALID_ARG;
    if (tc) return tq_decode_tc_launch(d, a, splits, (cudaStream_t)stream) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
    dim3 grid(splits, d->n_kv_heads, d->batch);
    fn<<<grid, kThreads, 0, (cudaStream_t)stream>>>(a);
    return cudaPeekAtLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

extern "C" {

tq_status tq_decode_attention_ex(const tq_cache_desc* d, const tq_cache_ptrs* c, const void* q, int32_t q_dtype,
                                 const int32_t* d_seq_lens, int32_t max_seq_len, float* out, void* workspace,
                                 size_t workspace_bytes, int32_t* d_status, void* stream, int32_t v_mode,
                                 int32_t n_splits) {
    return tq_decode_run(d, c, q, q_dtype, d_seq_lens, max_seq_len, out, workspace, workspace_bytes, d_status,
                         stream, v_mode, n_splits, nullptr);
}

tq_status tq_decode_attention(const tq_cache_desc* d, const tq_cache_ptrs* c, const void* q, int32_t q_dtype,
                              const int32_t* d_seq_lens, int32_t max_seq_len, float* out, void* workspace,
                              size_t workspace_bytes, int32_t* d_status, void* stream) {
    return tq_decode_attention_ex(d, c, q, q_dtype, d_seq_lens, max_seq_len, out, workspace, workspace_bytes,
                                  d_status, stream, TQ_VMODE_AUTO, 0);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs inside another
// framework's memory pool or allocator (and must not allocate behind its
// back), plugins handed only fixed input/output buffers, and paths where an
// allocation would synchronise the device.  For them the split-K scratch (the
// per-split partials and the per-(batch, KV head) tickets) lives in a fixed
// array in this library's device image instead of a caller-provided buffer.
// Every GPU that loads the library holds this array until the process exits.
#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;   // 8 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device, looked up once per
// device.  In host code the array's name only stands in for the symbol; only
// the address returned here may be handed to a kernel.
tq_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return TQ_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return TQ_OK;
}

}  // namespace

extern "C" size_t tq_decode_noalloc_max_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" tq_status tq_decode_attention_noalloc(const tq_cache_desc* d, const tq_cache_ptrs* c, const void* q,
                                                 int32_t q_dtype, const int32_t* d_seq_lens, int32_t max_seq_len,
                                                 float* out, int32_t* d_status, void* stream) {
    int32_t splits = 0, mode = 0;
    tq_status st = tq_decode_plan(d, max_seq_len, TQ_VMODE_AUTO, 0, &splits, &mode);
    if (st != TQ_OK) return st;
    if (splits < 1) return TQ_ERR_CUDA;
    if (splits == 1) return tq_decode_attention_ex(d, c, q, q_dtype, d_seq_lens, max_seq_len, out, nullptr, 0,
                                                   d_status, stream, TQ_VMODE_AUTO, 1);
    const size_t need = tq_decode_workspace_bytes(d, mode == TQ_VMODE_TENSOR ? 1 : splits);
    if (need == 0 || need > kNoAllocScratchBytes) return TQ_ERR_WORKSPACE;
    void* scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != TQ_OK) return st;
    // the tickets must start at zero; the array keeps whatever the last call left
    const size_t pairs = (size_t)d->batch * d->n_kv_heads;
    if (cudaMemsetAsync(scratch, 0, pairs * sizeof(int32_t), (cudaStream_t)stream) != cudaSuccess) return TQ_ERR_CUDA;
    return tq_decode_attention_ex(d, c, q, q_dtype, d_seq_lens, max_seq_len, out, scratch, kNoAllocScratchBytes,
                                  d_status, stream, TQ_VMODE_AUTO, splits);
}
