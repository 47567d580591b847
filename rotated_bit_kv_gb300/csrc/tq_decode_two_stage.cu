// Decode attention on caches with two-stage keys [TQ-MNN §2.4]: a (b-1)-bit MSE
// code and a 1-bit QJL code of its residual per key, read by the CUDA-core
// kernels of tq_decode_cc.cuh (natural layout).  Each key's score is
//   n <q~, C[idx]> + n rho sqrt(pi/2) / 128 <S q~, 2 sign - 1>,
// the unbiased sign-projection estimate of <q~, r> added to the MSE term; S q~ is
// formed once per query head in the prologue.  Values are the one-stage 3- or
// 4-bit codes.  Its own translation unit so that it compiles beside tq_decode.cu.
#include "tq_decode_cc.cuh"

namespace {
template <int GP>
KernelFn two_stage_fmt(int kf, int vf, int mode) {
    if (kf == TQ_FMT_QJ1 && vf == TQ_FMT_ONE3) return pick_mode<GP, TQ_FMT_QJ1, TQ_FMT_ONE3>(mode);
    if (kf == TQ_FMT_QJ1 && vf == TQ_FMT_ONE4) return pick_mode<GP, TQ_FMT_QJ1, TQ_FMT_ONE4>(mode);
    if (kf == TQ_FMT_QJ2 && vf == TQ_FMT_ONE3) return pick_mode<GP, TQ_FMT_QJ2, TQ_FMT_ONE3>(mode);
    if (kf == TQ_FMT_QJ2 && vf == TQ_FMT_ONE4) return pick_mode<GP, TQ_FMT_QJ2, TQ_FMT_ONE4>(mode);
    return nullptr;
}
}  // namespace

// The kernel for (padded group GP, key format, value format, V mode), or null.
KernelFn tq_two_stage_kernel(int GP, int kf, int vf, int mode) {
    switch (GP) {
        case 1: return two_stage_fmt<1>(kf, vf, mode);
        case 4: return two_stage_fmt<4>(kf, vf, mode);
        case 8: return two_stage_fmt<8>(kf, vf, mode);
        case 16: return two_stage_fmt<16>(kf, vf, mode);
        default: return nullptr;
    }
}
