// kernels_2sm.cu -- instantiations of the CTA-pair kernel (256 x 128 and
// 256 x 256 tiles) for every output format.
#include "gemm_sm103_2sm.cuh"
#include "kernels.h"

#include <type_traits>

namespace tsg {

namespace {
template <int BN>
const void* pick_out_2sm(int out) {
    switch (out) {
        case kOutF16: return reinterpret_cast<const void*>(&gemm_sm103_2sm<BN, kOutF16>);
        case kOutBF16: return reinterpret_cast<const void*>(&gemm_sm103_2sm<BN, kOutBF16>);
        case kOutF32: return reinterpret_cast<const void*>(&gemm_sm103_2sm<BN, kOutF32>);
        default: return nullptr;
    }
}
}  // namespace

const void* kernel_2sm(int block_n, int out_kind) {
    switch (block_n) {
        case 128: return pick_out_2sm<128>(out_kind);
        case 256: return pick_out_2sm<256>(out_kind);
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
        default: return -1;
    }
}

}  // namespace tsg
