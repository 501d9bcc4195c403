// kernels_1sm_cs.cu -- instantiations of the one-SM kernel in its
// cluster-split form (2 x 1 clusters splitting each tile's K range,
// partials exchanged through distributed shared memory), RRR layout with
// 16-bit inputs, every tile width and output format.
#include "gemm_sm103.cuh"
#include "kernels.h"

namespace tsg {

namespace {
template <int BN>
const void* pick(int out) {
    switch (out) {
        case kOutF16: return reinterpret_cast<const void*>(&gemm_sm103_1sm<BN, kOutF16, 0, false, true>);
        case kOutBF16: return reinterpret_cast<const void*>(&gemm_sm103_1sm<BN, kOutBF16, 0, false, true>);
        case kOutF32: return reinterpret_cast<const void*>(&gemm_sm103_1sm<BN, kOutF32, 0, false, true>);
        default: return nullptr;
    }
}
}  // namespace

const void* kernel_1sm_cs(int block_n, int out_kind) {
    switch (block_n) {
        case 64: return pick<64>(out_kind);
        case 128: return pick<128>(out_kind);
        case 192: return pick<192>(out_kind);
        case 256: return pick<256>(out_kind);
        default: return nullptr;
    }
}

}  // namespace tsg
