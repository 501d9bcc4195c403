// kernels_1sm.cu -- instantiations of the one-SM-per-tile kernel for every
// tile width and output format, and the lookup the host API uses.
#include "gemm_sm103.cuh"
#include "kernels.h"

#include <type_traits>

namespace tsg {

namespace {
template <int BN>
const void* pick_out(int out) {
    switch (out) {
        case kOutF16: return reinterpret_cast<const void*>(&gemm_sm103_1sm<BN, kOutF16>);
        case kOutBF16: return reinterpret_cast<const void*>(&gemm_sm103_1sm<BN, kOutBF16>);
        case kOutF32: return reinterpret_cast<const void*>(&gemm_sm103_1sm<BN, kOutF32>);
        default: return nullptr;
    }
}
}  // namespace

const void* kernel_1sm(int block_n, int out_kind) {
    switch (block_n) {
        case 64: return pick_out<64>(out_kind);
        case 128: return pick_out<128>(out_kind);
        case 192: return pick_out<192>(out_kind);
        case 256: return pick_out<256>(out_kind);
        default: return nullptr;
    }
}

int64_t kernel_1sm_smem_bytes(int block_n, int out_kind, int stages) {
    auto pick = [&](auto bn) -> int64_t {
        constexpr int BN = decltype(bn)::value;
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
