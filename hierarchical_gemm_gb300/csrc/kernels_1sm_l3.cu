// kernels_1sm_l3.cu -- instantiations of the one-SM kernel for the
// CCR operand layout, every tile width and output format.
#include "gemm_sm103.cuh"
#include "kernels.h"

namespace tsg {

namespace {
template <int BN>
const void* pick(int out) {
    switch (out) {
        case kOutF16: return reinterpret_cast<const void*>(&gemm_sm103_1sm<BN, kOutF16, 3>);
        case kOutBF16: return reinterpret_cast<const void*>(&gemm_sm103_1sm<BN, kOutBF16, 3>);
        case kOutF32: return reinterpret_cast<const void*>(&gemm_sm103_1sm<BN, kOutF32, 3>);
        default: return nullptr;
    }
}
}  // namespace

const void* kernel_1sm_layout3(int block_n, int out_kind) {
    switch (block_n) {
        case 64: return pick<64>(out_kind);
        case 128: return pick<128>(out_kind);
        case 192: return pick<192>(out_kind);
        case 256: return pick<256>(out_kind);
        default: return nullptr;
    }
}

}  // namespace tsg
