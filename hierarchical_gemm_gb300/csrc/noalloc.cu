// noalloc.cu -- the split-K GEMM for callers that cannot allocate device
// memory (see tsgemm_run_splitk_noalloc in include/tsgemm.h).
//
// The split-K kernel needs scratch memory: an fp32 partial tile per split,
// arrival counters per split tile (one per 32-column chunk and 32-row lane
// quarter) and a status word.  tsgemm_plan allocates
// these with cudaMalloc; this entry point instead carves them out of one
// file-scope device array of fixed size, which every GPU that loads the
// library holds until the process exits.  Nothing here calls cudaMalloc,
// cudaFree or any other allocating routine.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gemm_sm103.cuh"
#include "kernels.h"
#include "planner.h"
#include "tsgemm.h"

namespace {

// Layout of the scratch array:
//   [0, 256)                       status word (int) when the caller passes none
//   [256, 256 + 128 * max tiles)   arrival counters, 32 per split tile at most
//                                  (block_n / 32 chunks x 4 lane quarters)
//   [kWsOffset, end)               fp32 split-K partials
constexpr size_t kScratchBytes = TSGEMM_NOALLOC_SCRATCH_BYTES;
constexpr size_t kCounterOffset = 256;
constexpr size_t kMaxTiles = TSGEMM_NOALLOC_MAX_TILES;
constexpr size_t kCountersPerTile = 32;
constexpr size_t kWsOffset = kCounterOffset + kMaxTiles * kCountersPerTile * sizeof(int);
static_assert(kWsOffset % 256 == 0, "scratch layout");
static_assert(kScratchBytes - kWsOffset >= TSGEMM_NOALLOC_WS_BYTES, "workspace capacity");

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool done = false;
    unsigned char* scratch = nullptr;  // device address of g_scratch
    bool cc_ok = false;
    int num_sms = 0;
};

std::mutex g_mu;
DeviceSetup g_setup[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

// tcgen05 kind::f16 instruction descriptor: fp32 accumulator, A and B of the
// input format, A K-major, B MN-major, M = 128, N = block_n.
uint32_t idesc_for(int dtype_in, int block_n) {
    const uint32_t fmt = dtype_in == TSGEMM_BF16 ? 1u : 0u;
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (1u << 16) | (static_cast<uint32_t>(block_n >> 3) << 17) |
           (static_cast<uint32_t>(128 >> 4) << 24);
}

bool is_device_memory(const void* p, int dev) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeManaged) return true;
    return a.type == cudaMemoryTypeDevice && a.device == dev;
}

bool overlap(const void* a, int64_t na, const void* b, int64_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
}

// Per-device set-up, done by the first call on each device with that device
// current: check the device, look up the device address of the scratch
// array, and raise the shared-memory limit of every kernel this entry point
// can launch (the one-SM kernel for 16-bit inputs in the RRR layout, every
// tile width and output format), so that no later call does one-time
// work.  Returns null on failure.
DeviceSetup* setup_device(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    DeviceSetup& s = g_setup[dev];
    if (s.done) return &s;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    s.cc_ok = (major == 10 && minor == 3);
    s.num_sms = sms;
    if (s.cc_ok) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            (void)cudaGetLastError();
            return nullptr;
        }
        s.scratch = static_cast<unsigned char*>(ptr);
        for (int bn = 64; bn <= 256; bn += 64) {
            for (int out = tsg::kOutF16; out <= tsg::kOutF32; ++out) {
                const void* kern = tsg::kernel_1sm(bn, out, TSGEMM_LAYOUT_RRR, false, 1);
                if (!kern || cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  static_cast<int>(tsg::kSmemPerCtaMax)) != cudaSuccess) {
                    (void)cudaGetLastError();
                    return nullptr;
                }
            }
        }
    }
    s.done = true;
    return &s;
}

}  // namespace

extern "C" tsgemm_status_t tsgemm_run_splitk_noalloc(int64_t M, int64_t N, int64_t K,
                                                     tsgemm_dtype_t dtype_in, tsgemm_dtype_t dtype_out,
                                                     int32_t splits, const void* A, const void* B,
                                                     void* C, int* status, void* stream) {
    tsgemm_status_t st = tsg::validate_problem(M, N, K, dtype_in, dtype_out, TSGEMM_LAYOUT_RRR);
    if (st != TSGEMM_OK) return st;
    if (splits < 0) return TSGEMM_ERR_INVALID_ARG;
    if (!A || !B || !C) return TSGEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) & 15u)
        return TSGEMM_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(status) & 3u) return TSGEMM_ERR_ALIGNMENT;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceSetup* ds = setup_device(dev);
    if (!ds) return TSGEMM_ERR_CUDA;
    if (!ds->cc_ok) return TSGEMM_ERR_UNSUPPORTED;
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return TSGEMM_ERR_CUDA;

    tsgemm_config_t force{};
    force.splits = splits;
    force.block_m = 128;  // the one-SM kernel
    force.stream_k_tiles = -1;  // split mode only
    tsgemm_config_t cfg{};
    st = tsg::choose_config(M, N, K, dtype_in, dtype_out, TSGEMM_LAYOUT_RRR, ds->num_sms, &force, &cfg);
    if (st != TSGEMM_OK) return st;

    const int64_t tiles = ((M + 127) / 128) * ((N + cfg.block_n - 1) / cfg.block_n);
    if (static_cast<size_t>(tiles) > kMaxTiles ||
        static_cast<size_t>(cfg.workspace_bytes) > kScratchBytes - kWsOffset)
        return TSGEMM_ERR_SCRATCH_LIMIT;

    const int64_t a_bytes = M * K * 2, b_bytes = K * N * 2;
    const int64_t c_bytes = M * N * (dtype_out == TSGEMM_F32 ? 4 : 2);
    if (overlap(C, c_bytes, A, a_bytes) || overlap(C, c_bytes, B, b_bytes)) return TSGEMM_ERR_INVALID_ARG;
    if (!is_device_memory(A, dev) || !is_device_memory(B, dev) || !is_device_memory(C, dev))
        return TSGEMM_ERR_INVALID_ARG;
    if (status && !is_device_memory(status, dev)) {
        // mapped pinned host memory is also acceptable for the status word
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, status) != cudaSuccess || a.type != cudaMemoryTypeHost ||
            a.devicePointer == nullptr) {
            (void)cudaGetLastError();
            return TSGEMM_ERR_INVALID_ARG;
        }
        status = static_cast<int*>(a.devicePointer);
    }

    const int out_kind = dtype_out == TSGEMM_F16 ? tsg::kOutF16 : (dtype_out == TSGEMM_BF16 ? tsg::kOutBF16 : tsg::kOutF32);
    const void* kern = tsg::kernel_1sm(cfg.block_n, out_kind, TSGEMM_LAYOUT_RRR, false, 1);
    const int64_t need = tsg::kernel_1sm_smem_bytes(cfg.block_n, out_kind, cfg.stages, 1);
    if (!kern || need > tsg::kSmemPerCtaMax) return TSGEMM_ERR_UNSUPPORTED;
    const int64_t smem = need > tsg::kSmemPerCtaMax / 2 + 1024 ? need : tsg::kSmemPerCtaMax / 2 + 1024;

    CUtensorMap tmA;  // the type carries the alignment the encoder requires
    CUtensorMap tmB;
    CUtensorMap tmC;
    const CUtensorMapDataType dt =
        dtype_in == TSGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint32_t estr[2] = {1, 1};
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        const cuuint32_t box[2] = {64, 128};
        if (enc(&tmA, dt, 2, const_cast<void*>(A), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return TSGEMM_ERR_CUDA;
    }
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 2};
        const cuuint32_t box[2] = {64, 64};
        if (enc(&tmB, dt, 2, const_cast<void*>(B), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return TSGEMM_ERR_CUDA;
    }

    {
        const CUtensorMapDataType dc = dtype_out == TSGEMM_F32
                                           ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                           : (dtype_out == TSGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N * (dtype_out == TSGEMM_F32 ? 4 : 2))};
        const cuuint32_t box[2] = {32, 32};
        const bool dtype_out_is_f32 = dtype_out == TSGEMM_F32;
        if (enc(&tmC, dc, 2, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            (dtype_out_is_f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B),
                CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return TSGEMM_ERR_CUDA;
    }

    int* counters = reinterpret_cast<int*>(ds->scratch + kCounterOffset);
    int* own_status = reinterpret_cast<int*>(ds->scratch);
    float* ws = reinterpret_cast<float*>(ds->scratch + kWsOffset);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents: the split tiles'
    // counters (and the status word this call reports into) must start at
    // zero.
    const size_t ncounters = static_cast<size_t>(cfg.split_tiles) * (cfg.block_n / 32) * 4;
    if ((ncounters > 0 && cudaMemsetAsync(counters, 0, ncounters * sizeof(int), s) != cudaSuccess) ||
        cudaMemsetAsync(status ? status : own_status, 0, sizeof(int), s) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }

    tsg::GemmParams gp{};
    gp.M = static_cast<int32_t>(M);
    gp.N = static_cast<int32_t>(N);
    gp.K = static_cast<int32_t>(K);
    gp.tiles_m = static_cast<int32_t>((M + 127) / 128);
    gp.tiles_n = static_cast<int32_t>((N + cfg.block_n - 1) / cfg.block_n);
    gp.splits = cfg.splits;
    gp.kblocks = static_cast<int32_t>((K + 63) / 64);
    gp.group_m = cfg.group_m;
    gp.stages = cfg.stages;
    gp.debug_flags = 0;
    gp.units = cfg.units;
    gp.full_tiles = tiles - cfg.split_tiles;
    gp.idesc = idesc_for(dtype_in, cfg.block_n);
    gp.csplit = 1;
    gp.C = C;
    gp.ws = ws;
    gp.ws_own = nullptr;  // (stream-K only)
    gp.counters = counters;
    gp.status = status ? status : own_status;
    gp.timeout_ns = static_cast<uint64_t>(cfg.timeout_ms) * 1000000ull;

    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>(cfg.grid), 1, 1);
    lc.blockDim = dim3(tsg::kThreads, 1, 1);
    lc.dynamicSmemBytes = static_cast<size_t>(smem);
    lc.stream = s;
    void* args[4] = {&tmA, &tmB, &tmC, &gp};
    if (cudaLaunchKernelExC(&lc, kern, args) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }
    return TSGEMM_OK;
}
