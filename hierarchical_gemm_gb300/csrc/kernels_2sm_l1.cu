// kernels_2sm_l1.cu -- instantiations of the CTA-pair kernel for the
// RCR operand layout: every tile width and output format, one pair
// per cluster, and (256-wide tiles) two pairs per cluster sharing A.
#include "gemm_sm103_2sm.cuh"
#include "kernels.h"

namespace tsg {

namespace {
template <int BN, int kPairs>
const void* pick(int out) {
    switch (out) {
        case kOutF16: return reinterpret_cast<const void*>(&gemm_sm103_2sm<BN, kOutF16, 1, false, kPairs>);
        case kOutBF16: return reinterpret_cast<const void*>(&gemm_sm103_2sm<BN, kOutBF16, 1, false, kPairs>);
        case kOutF32: return reinterpret_cast<const void*>(&gemm_sm103_2sm<BN, kOutF32, 1, false, kPairs>);
        default: return nullptr;
    }
}
}  // namespace

const void* kernel_2sm_layout1(int block_n, int out_kind, int pairs) {
    if (pairs == 2) return block_n == 256 ? pick<256, 2>(out_kind) : nullptr;
    if (pairs != 1) return nullptr;
    switch (block_n) {
        case 128: return pick<128, 1>(out_kind);
        case 256: return pick<256, 1>(out_kind);
        default: return nullptr;
    }
}

}  // namespace tsg
