// kernels_1sm.cu -- the host-side lookup of the one-SM kernel's
// instantiations (by tile width, output format, operand layout, input width
// and cluster split) and of the shared memory each needs.
#include "gemm_sm103.cuh"
#include "kernels.h"

#include <type_traits>

namespace tsg {

const void* kernel_1sm(int block_n, int out_kind, int layout, bool in8, int cs) {
    if (cs >= 2) return layout == 0 && !in8 ? kernel_1sm_cs(block_n, out_kind) : nullptr;
    if (cs > 1) return nullptr;
    if (in8) return layout == 1 ? kernel_1sm_f8(block_n, out_kind) : nullptr;
    switch (layout) {
        case 0: return kernel_1sm_layout0(block_n, out_kind);
        case 1: return kernel_1sm_layout1(block_n, out_kind);
        case 2: return kernel_1sm_layout2(block_n, out_kind);
        case 3: return kernel_1sm_layout3(block_n, out_kind);
        default: return nullptr;
    }
}

int64_t kernel_1sm_smem_bytes(int block_n, int out_kind, int stages, int cs) {
    auto pick = [&](auto bn) -> int64_t {
        constexpr int BN = decltype(bn)::value;
        if (cs >= 2) {
            switch (out_kind) {
                case kOutF16: return smem_bytes_1sm<BN, kOutF16, true>(stages);
                case kOutBF16: return smem_bytes_1sm<BN, kOutBF16, true>(stages);
                case kOutF32: return smem_bytes_1sm<BN, kOutF32, true>(stages);
                default: return -1;
            }
        }
        switch (out_kind) {
            case kOutF16: return smem_bytes_1sm<BN, kOutF16>(stages);
            case kOutBF16: return smem_bytes_1sm<BN, kOutBF16>(stages);
            case kOutF32: return smem_bytes_1sm<BN, kOutF32>(stages);
            default: return -1;
        }
    };
    switch (block_n) {
        case 64: return pick(std::integral_constant<int, 64>{});
        case 128: return pick(std::integral_constant<int, 128>{});
        case 192: return pick(std::integral_constant<int, 192>{});
        case 256: return pick(std::integral_constant<int, 256>{});
        default: return -1;
    }
}

}  // namespace tsg
