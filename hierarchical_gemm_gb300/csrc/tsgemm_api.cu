// tsgemm_api.cu -- the C ABI: plans, operand descriptors (TMA tensor maps),
// launches and the device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "gemm_sm103.cuh"
#include "kernels.h"
#include "planner.h"
#include "tsgemm.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the installed driver, looked up through the
// runtime so that the library does not link libcuda directly.
EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

// tcgen05 instruction descriptor, kind::f16 and kind::f8f6f4:
//   bits  4-5  accumulator format (1 = fp32)
//   bits  7-9  A format (kind::f16: 0 = fp16, 1 = bf16;
//              kind::f8f6f4: 0 = E4M3, 1 = E5M2)
//   bits 10-12 B format
//   bit  15    A major (0 = K-major: A stored M x K; 1 = MN-major: stored K x M)
//   bit  16    B major (0 = K-major: B stored N x K; 1 = MN-major: stored K x N)
//   bits 17-22 N >> 3
//   bits 24-28 M >> 4
uint32_t make_idesc(int dtype_in, int m, int n, int layout) {
    const uint32_t fmt = (dtype_in == TSGEMM_BF16 || dtype_in == TSGEMM_E5M2) ? 1u : 0u;
    const uint32_t a_mn = tsg::a_kmajor(layout) ? 0u : 1u;
    const uint32_t b_mn = tsg::b_kmajor(layout) ? 0u : 1u;
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (a_mn << 15) | (b_mn << 16) |
           (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

int out_kind(int dtype_out) {
    return dtype_out == TSGEMM_F16 ? tsg::kOutF16 : (dtype_out == TSGEMM_BF16 ? tsg::kOutBF16 : tsg::kOutF32);
}

int64_t elem_bytes(int dt) { return dt == TSGEMM_F32 ? 4 : (tsg::is_8bit(dt) ? 1 : 2); }

}  // namespace

struct tsgemm_plan_s {
    int64_t M, N, K;
    int dtype_in, dtype_out;
    int layout;
    tsgemm_config_t cfg;
    int device;
    const void* kernel;
    int64_t smem;
    int* status_d;
    float* ws;
    int* counters;
    int64_t num_tiles;
    const void* last_a;
    const void* last_b;
    const void* last_c;
    CUtensorMap tmA;  // the type carries the alignment the encoder requires
    CUtensorMap tmB;
    CUtensorMap tmC;
    tsg::GemmParams params;
};

static void plan_free(tsgemm_plan_s* p) {
    if (!p) return;
    if (p->status_d) cudaFree(p->status_d);
    if (p->ws) cudaFree(p->ws);
    if (p->counters) cudaFree(p->counters);
    delete p;
}

extern "C" {

const char* tsgemm_status_string(tsgemm_status_t s) {
    switch (s) {
        case TSGEMM_OK: return "success";
        case TSGEMM_ERR_INVALID_ARG: return "invalid argument";
        case TSGEMM_ERR_UNSUPPORTED: return "unsupported problem, configuration or device";
        case TSGEMM_ERR_ALIGNMENT: return "pointer or row stride not 16-byte aligned";
        case TSGEMM_ERR_CUDA: return "CUDA call failed";
        case TSGEMM_ERR_TIMEOUT: return "a bounded device wait expired";
        case TSGEMM_ERR_OOM: return "out of device memory";
        case TSGEMM_ERR_SCRATCH_LIMIT: return "problem exceeds the fixed scratch of the no-allocation entry point";
        default: return "unknown status";
    }
}

tsgemm_status_t tsgemm_choose_config(int64_t M, int64_t N, int64_t K, tsgemm_dtype_t dtype_in,
                                     tsgemm_dtype_t dtype_out, tsgemm_layout_t layout,
                                     int32_t num_sms, const tsgemm_config_t* force,
                                     tsgemm_config_t* out) {
    return tsg::choose_config(M, N, K, dtype_in, dtype_out, layout, num_sms, force, out);
}

tsgemm_status_t tsgemm_plan_ex(tsgemm_plan_t* out, int64_t M, int64_t N, int64_t K,
                               tsgemm_dtype_t dtype_in, tsgemm_dtype_t dtype_out,
                               tsgemm_layout_t layout, const tsgemm_config_t* force) {
    if (!out) return TSGEMM_ERR_INVALID_ARG;
    *out = nullptr;
    tsgemm_status_t st = tsg::validate_problem(M, N, K, dtype_in, dtype_out, layout);
    if (st != TSGEMM_OK) return st;

    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return TSGEMM_ERR_UNSUPPORTED;
    if (!encode_fn()) return TSGEMM_ERR_CUDA;

    tsgemm_config_t cfg{};
    st = tsg::choose_config(M, N, K, dtype_in, dtype_out, layout, sms, force, &cfg);
    if (st != TSGEMM_OK) return st;

    const bool pair = cfg.block_m == 256;
    const bool in8 = tsg::is_8bit(dtype_in);
    const int cs = cfg.cluster_split >= 2 ? cfg.cluster_split : 1;
    const void* kern = pair ? tsg::kernel_2sm(cfg.block_n, out_kind(dtype_out), layout, in8)
                            : tsg::kernel_1sm(cfg.block_n, out_kind(dtype_out), layout, in8, cs);
    const int64_t need = pair ? tsg::kernel_2sm_smem_bytes(cfg.block_n, out_kind(dtype_out), cfg.stages)
                              : tsg::kernel_1sm_smem_bytes(cfg.block_n, out_kind(dtype_out), cfg.stages, cs);
    if (!kern || need != tsg::smem_bytes_for(cfg.block_m, cfg.block_n, dtype_out, cfg.stages, cs) ||
        need > tsg::kSmemPerCtaMax)
        return TSGEMM_ERR_UNSUPPORTED;
    // Ask for more than half the SM's shared memory even when the ring is
    // shallow, so one CTA owns each SM and its tensor memory.
    const int64_t smem = need > tsg::kSmemPerCtaMax / 2 + 1024 ? need : tsg::kSmemPerCtaMax / 2 + 1024;
    // The attribute is per kernel, shared by every plan that uses it: set it
    // to the largest size any launch asks for, never lower.
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(tsg::kSmemPerCtaMax)) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }
    if (pair || cs >= 2) {
        // Persistent clusters: launch no more than can be resident at once
        // (a cluster's CTAs must share a GPC).
        const int per_cluster = pair ? 2 : cs;
        cudaLaunchConfig_t lc{};
        lc.gridDim = dim3(static_cast<unsigned>(cfg.grid), 1, 1);
        lc.blockDim = dim3(tsg::kThreads, 1, 1);
        lc.dynamicSmemBytes = static_cast<size_t>(smem);
        // the cluster-split kernel takes its cs x 1 cluster shape at launch
        cudaLaunchAttribute cattr{};
        cattr.id = cudaLaunchAttributeClusterDimension;
        cattr.val.clusterDim.x = static_cast<unsigned>(per_cluster);
        cattr.val.clusterDim.y = 1;
        cattr.val.clusterDim.z = 1;
        if (!pair) {
            lc.attrs = &cattr;
            lc.numAttrs = 1;
        }
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &lc) != cudaSuccess || clusters < 1) {
            (void)cudaGetLastError();
            return TSGEMM_ERR_UNSUPPORTED;
        }
        // (a smaller grid only makes each slot's stream-K range longer; the
        // workspace sized for the larger one still covers it)
        if (cfg.grid > per_cluster * clusters) cfg.grid = per_cluster * clusters;
    }

    // value-initialised; operator new honours the 64-byte alignment the
    // tensor maps need
    tsgemm_plan_s* p = new (std::nothrow) tsgemm_plan_s();
    if (!p) return TSGEMM_ERR_OOM;
    p->M = M;
    p->N = N;
    p->K = K;
    p->dtype_in = dtype_in;
    p->dtype_out = dtype_out;
    p->layout = layout;
    p->cfg = cfg;
    p->device = dev;
    p->kernel = kern;
    p->smem = smem;
    // split-K (stream-K) counters: per 128-row half of each split (stream-K)
    // tile (pairs reduce halves), one per 32-column chunk and lane quarter
    p->num_tiles = (cfg.stream_k_tiles > 0 ? cfg.stream_k_tiles : cfg.split_tiles) * (cfg.block_m / 128) *
                   (cfg.block_n / 32) * 4;

    if (cudaMalloc(&p->status_d, sizeof(int)) != cudaSuccess) {
        (void)cudaGetLastError();
        plan_free(p);
        return TSGEMM_ERR_OOM;
    }
    if (cudaMemset(p->status_d, 0, sizeof(int)) != cudaSuccess) {
        (void)cudaGetLastError();
        plan_free(p);
        return TSGEMM_ERR_CUDA;
    }
    if (cfg.splits > 1 || cfg.stream_k_tiles > 0) {
        if (cudaMalloc(&p->ws, static_cast<size_t>(cfg.workspace_bytes)) != cudaSuccess ||
            cudaMalloc(&p->counters, static_cast<size_t>(p->num_tiles) * sizeof(int)) != cudaSuccess) {
            (void)cudaGetLastError();
            plan_free(p);
            return TSGEMM_ERR_OOM;
        }
        if (cudaMemset(p->counters, 0, static_cast<size_t>(p->num_tiles) * sizeof(int)) != cudaSuccess) {
            (void)cudaGetLastError();
            plan_free(p);
            return TSGEMM_ERR_CUDA;
        }
    }

    tsg::GemmParams& gp = p->params;
    gp.M = static_cast<int32_t>(M);
    gp.N = static_cast<int32_t>(N);
    gp.K = static_cast<int32_t>(K);
    gp.tiles_m = static_cast<int32_t>((M + cfg.block_m - 1) / cfg.block_m);
    gp.tiles_n = static_cast<int32_t>((N + cfg.block_n - 1) / cfg.block_n);
    gp.splits = cfg.splits;
    gp.kblocks = static_cast<int32_t>((K + tsg::slice_k(dtype_in) - 1) / tsg::slice_k(dtype_in));
    gp.group_m = cfg.group_m;
    gp.stages = cfg.stages;
    gp.debug_flags = cfg.debug_flags;
    gp.units = cfg.units;
    gp.full_tiles = ((M + cfg.block_m - 1) / cfg.block_m) * gp.tiles_n - cfg.split_tiles - cfg.stream_k_tiles;
    gp.sk_tiles = cfg.stream_k_tiles;
    gp.sk_work = cfg.stream_k_tiles * gp.kblocks;
    // (a 256 x 512 pair tile is two N = 256 MMAs per K step)
    gp.idesc = make_idesc(dtype_in, cfg.block_m, cfg.block_n == 512 ? 256 : cfg.block_n, layout);
    gp.csplit = cs;
    gp.C = nullptr;
    gp.ws = p->ws;
    // stream-K: the owners' partials follow the contributors' (one 128 x
    // block_n fp32 slot per CTA each)
    gp.ws_own = (cfg.stream_k_tiles > 0 && p->ws) ? p->ws + static_cast<int64_t>(cfg.grid) * 128 * cfg.block_n
                                                  : nullptr;
    gp.counters = p->counters;
    gp.status = p->status_d;
    gp.timeout_ns = static_cast<uint64_t>(cfg.timeout_ms) * 1000000ull;
    *out = p;
    return TSGEMM_OK;
}

tsgemm_status_t tsgemm_plan(tsgemm_plan_t* out, int64_t M, int64_t N, int64_t K,
                            tsgemm_dtype_t dtype_in, tsgemm_dtype_t dtype_out,
                            tsgemm_layout_t layout) {
    return tsgemm_plan_ex(out, M, N, K, dtype_in, dtype_out, layout, nullptr);
}

tsgemm_status_t tsgemm_get_config(tsgemm_plan_t plan, tsgemm_config_t* out) {
    if (!plan || !out) return TSGEMM_ERR_INVALID_ARG;
    *out = plan->cfg;
    return TSGEMM_OK;
}

static tsgemm_status_t check_device_ptr(const void* ptr, int device) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_INVALID_ARG;
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return TSGEMM_ERR_INVALID_ARG;
    if (a.type == cudaMemoryTypeDevice && a.device != device) return TSGEMM_ERR_INVALID_ARG;
    return TSGEMM_OK;
}

static bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
}

static tsgemm_status_t encode_maps(tsgemm_plan_s* p, const void* A, const void* B) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return TSGEMM_ERR_CUDA;
    const bool in8 = tsg::is_8bit(p->dtype_in);
    const CUtensorMapDataType dt = in8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : (p->dtype_in == TSGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    const int64_t eb = in8 ? 1 : 2;
    const cuuint32_t estr[2] = {1, 1};
    // L2 fill size of the operand loads: the one-SM kernel (the HBM-bound
    // skinny shapes) streams its operands and gains from 256-byte fills;
    // the CTA-pair kernel takes plain sector fills (same box, alternating
    // builds: 4096^3 bf16 86.7 us in 6 of 6 runs against 86.7-88.7 with
    // 256-byte fills, 16384 x 16384 x 8192 2155-2158 against 2167 us, the
    // E4M3 and long-K shapes alike; the skinny 128 x 28672 x 8192 shape
    // 78.0-78.5 against 76.5-77.0 us with plain fills)
    const CUtensorMapL2promotion prom =
        p->cfg.block_m == 256 ? CU_TENSOR_MAP_L2_PROMOTION_NONE : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
    auto tile_map = [&](CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, cuuint32_t box_inner,
                        cuuint32_t box_outer) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner * eb)};
        const cuuint32_t box[2] = {box_inner, box_outer};
        return enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, prom, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    // Every box is 128 bytes (one swizzle row) along the contiguous
    // dimension: 64 16-bit or 128 8-bit elements.
    //   A stored M x K: 128 B (K) x 128 (M) boxes;  A stored K x M: 64 (M) x 64 (K)
    //   B stored K x N: 64 (N) x 64 (K) boxes;      B stored N x K: 128 B (K) x
    //   the CTA's columns (N) -- block_n, or block_n / 2 for a CTA pair, or
    //   128 for a 256 x 512 pair tile (two pieces, one per MMA half)
    // (8-bit operands are always stored K-major, the first form of each).
    const cuuint32_t kbox = static_cast<cuuint32_t>(128 / eb);
    const bool ak = tsg::a_kmajor(p->layout), bk = tsg::b_kmajor(p->layout);
    const cuuint32_t b_cols = static_cast<cuuint32_t>(
        p->cfg.block_m == 256 ? (p->cfg.block_n == 512 ? 128 : p->cfg.block_n / 2) : p->cfg.block_n);
    const bool ok_a = ak ? tile_map(&p->tmA, A, p->K, p->M, kbox, 128) : tile_map(&p->tmA, A, p->M, p->K, 64, 64);
    const bool ok_b = bk ? tile_map(&p->tmB, B, p->K, p->N, kbox, b_cols) : tile_map(&p->tmB, B, p->N, p->K, 64, 64);
    return ok_a && ok_b ? TSGEMM_OK : TSGEMM_ERR_CUDA;
}

// C: inner dimension N, outer M; box 32 x 32 (the block one epilogue warp
// stores at a time), in the swizzle the kernel writes its staging buffer in
// (16-bit outputs; fp32 outputs are stored from registers and the map goes
// unused).
static tsgemm_status_t encode_c(tsgemm_plan_s* p, void* C) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return TSGEMM_ERR_CUDA;
    const CUtensorMapDataType dt = p->dtype_out == TSGEMM_F32
                                       ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : (p->dtype_out == TSGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p->N), static_cast<cuuint64_t>(p->M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p->N * elem_bytes(p->dtype_out))};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    const bool dtype_out_is_f32 = p->dtype_out == TSGEMM_F32;
    if (enc(&p->tmC, dt, 2, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            (dtype_out_is_f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B),
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return TSGEMM_ERR_CUDA;
    return TSGEMM_OK;
}

tsgemm_status_t tsgemm_run(tsgemm_plan_t plan, const void* A, const void* B, void* C, void* stream) {
    if (!plan || !A || !B || !C) return TSGEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) & 15u)
        return TSGEMM_ERR_ALIGNMENT;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }
    if (dev != plan->device) return TSGEMM_ERR_INVALID_ARG;
    const int64_t a_bytes = plan->M * plan->K * elem_bytes(plan->dtype_in);
    const int64_t b_bytes = plan->K * plan->N * elem_bytes(plan->dtype_in);
    const int64_t c_bytes = plan->M * plan->N * elem_bytes(plan->dtype_out);
    if (overlaps(C, c_bytes, A, a_bytes) || overlaps(C, c_bytes, B, b_bytes)) return TSGEMM_ERR_INVALID_ARG;

    if (A != plan->last_a || B != plan->last_b) {
        tsgemm_status_t st = check_device_ptr(A, plan->device);
        if (st == TSGEMM_OK) st = check_device_ptr(B, plan->device);
        if (st != TSGEMM_OK) return st;
        plan->last_a = nullptr;
        plan->last_b = nullptr;
        st = encode_maps(plan, A, B);
        if (st != TSGEMM_OK) return st;
        plan->last_a = A;
        plan->last_b = B;
    }
    if (C != plan->last_c) {
        tsgemm_status_t st = check_device_ptr(C, plan->device);
        if (st != TSGEMM_OK) return st;
        plan->last_c = nullptr;
        st = encode_c(plan, C);
        if (st != TSGEMM_OK) return st;
        plan->last_c = C;
    }
    plan->params.C = C;

    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>(plan->cfg.grid), 1, 1);
    lc.blockDim = dim3(tsg::kThreads, 1, 1);
    lc.dynamicSmemBytes = static_cast<size_t>(plan->smem);
    lc.stream = static_cast<cudaStream_t>(stream);
    lc.attrs = nullptr;
    lc.numAttrs = 0;
    cudaLaunchAttribute cattr{};
    if (plan->cfg.cluster_split >= 2) {
        cattr.id = cudaLaunchAttributeClusterDimension;
        cattr.val.clusterDim.x = static_cast<unsigned>(plan->cfg.cluster_split);
        cattr.val.clusterDim.y = 1;
        cattr.val.clusterDim.z = 1;
        lc.attrs = &cattr;
        lc.numAttrs = 1;
    }
    void* args[4] = {&plan->tmA, &plan->tmB, &plan->tmC, &plan->params};
    if (cudaLaunchKernelExC(&lc, plan->kernel, args) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }
    return TSGEMM_OK;
}

tsgemm_status_t tsgemm_status(tsgemm_plan_t plan) {
    if (!plan) return TSGEMM_ERR_INVALID_ARG;
    int word = 0;
    if (cudaMemcpy(&word, plan->status_d, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }
    if (word == TSGEMM_OK) return TSGEMM_OK;
    // A run gave up: clear the word and the split-K tile counters it may
    // have left behind, so the plan can run again.
    if (cudaMemset(plan->status_d, 0, sizeof(int)) != cudaSuccess ||
        (plan->counters &&
         cudaMemset(plan->counters, 0, static_cast<size_t>(plan->num_tiles) * sizeof(int)) != cudaSuccess) ||
        cudaDeviceSynchronize() != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }
    return static_cast<tsgemm_status_t>(word);
}

tsgemm_status_t tsgemm_destroy(tsgemm_plan_t plan) {
    plan_free(plan);
    return TSGEMM_OK;
}

}  // extern "C"
