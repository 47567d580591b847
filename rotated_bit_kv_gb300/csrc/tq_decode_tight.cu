// Decode attention on caches whose mixed-rate keys are packed tightly: each code
// at its group's width, the groups' codes concatenated [Block-GTQ, packed cache],
// 32 or 48 bytes per key for 2 or 3 bits per coordinate on average (against 64
// in nibbles).  Read by the CUDA-core kernels of tq_decode_cc.cuh (natural
// layout): a thread stages its key's record in shared memory and walks the
// groups in ascending width with a running bit offset.  Values are the one-stage
// 3- or 4-bit codes.  Its own translation unit so that it compiles beside
// tq_decode.cu.
#include "tq_decode_cc.cuh"

namespace {
template <int GP>
KernelFn tight_fmt(int kf, int vf, int mode) {
    if (kf == TQ_FMT_MXT2 && vf == TQ_FMT_ONE3) return pick_mode<GP, TQ_FMT_MXT2, TQ_FMT_ONE3>(mode);
    if (kf == TQ_FMT_MXT2 && vf == TQ_FMT_ONE4) return pick_mode<GP, TQ_FMT_MXT2, TQ_FMT_ONE4>(mode);
    if (kf == TQ_FMT_MXT3 && vf == TQ_FMT_ONE3) return pick_mode<GP, TQ_FMT_MXT3, TQ_FMT_ONE3>(mode);
    if (kf == TQ_FMT_MXT3 && vf == TQ_FMT_ONE4) return pick_mode<GP, TQ_FMT_MXT3, TQ_FMT_ONE4>(mode);
    return nullptr;
}
}  // namespace

// The kernel for (padded group GP, key format, value format, V mode), or null.
KernelFn tq_tight_kernel(int GP, int kf, int vf, int mode) {
    switch (GP) {
        case 1: return tight_fmt<1>(kf, vf, mode);
        case 4: return tight_fmt<4>(kf, vf, mode);
        case 8: return tight_fmt<8>(kf, vf, mode);
        case 16: return tight_fmt<16>(kf, vf, mode);
        default: return nullptr;
    }
}
