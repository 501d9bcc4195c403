// kernels_2sm_f8.cu -- instantiations of the CTA-pair kernel for 8-bit float
// inputs (E4M3 / E5M2) in the RCR layout: every tile width and output
// format, one pair per cluster.
#include "gemm_sm103_2sm.cuh"
#include "kernels.h"

namespace tsg {

namespace {
template <int BN>
const void* pick(int out) {
    switch (out) {
        case kOutF16: return reinterpret_cast<const void*>(&gemm_sm103_2sm<BN, kOutF16, 1, true>);
        case kOutBF16: return reinterpret_cast<const void*>(&gemm_sm103_2sm<BN, kOutBF16, 1, true>);
        case kOutF32: return reinterpret_cast<const void*>(&gemm_sm103_2sm<BN, kOutF32, 1, true>);
        default: return nullptr;
    }
}
}  // namespace

const void* kernel_2sm_f8(int block_n, int out_kind) {
    switch (block_n) {
        case 128: return pick<128>(out_kind);
        case 256: return pick<256>(out_kind);
        case 512: return pick<512>(out_kind);
        default: return nullptr;
    }
}

}  // namespace tsg
