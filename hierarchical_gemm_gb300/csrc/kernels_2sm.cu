// kernels_2sm.cu -- the host-side lookup of the CTA-pair kernel's
// instantiations (by tile width, output format, operand layout and input
// width) and of the shared memory each needs.
#include "gemm_sm103_2sm.cuh"
#include "kernels.h"

#include <type_traits>

namespace tsg {

const void* kernel_2sm(int block_n, int out_kind, int layout, bool in8) {
    if (in8) return layout == 1 ? kernel_2sm_f8(block_n, out_kind) : nullptr;
    switch (layout) {
        case 0: return kernel_2sm_layout0(block_n, out_kind);
        case 1: return kernel_2sm_layout1(block_n, out_kind);
        case 2: return kernel_2sm_layout2(block_n, out_kind);
        case 3: return kernel_2sm_layout3(block_n, out_kind);
        default: return nullptr;
    }
}

int64_t kernel_2sm_smem_bytes(int block_n, int out_kind, int stages) {
    auto pick = [&](auto bn) -> int64_t {
        constexpr int BN = decltype(bn)::value;
        switch (out_kind) {
            case kOutF16: return smem_bytes_2sm<BN, kOutF16>(stages);
            case kOutBF16: return smem_bytes_2sm<BN, kOutBF16>(stages);
            case kOutF32: return smem_bytes_2sm<BN, kOutF32>(stages);
            default: return -1;
        }
    };
    switch (block_n) {
        case 128: return pick(std::integral_constant<int, 128>{});
        case 256: return pick(std::integral_constant<int, 256>{});
        case 512: return pick(std::integral_constant<int, 512>{});
        default: return -1;
    }
}

}  // namespace tsg
