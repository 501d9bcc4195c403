// gemm_sm103.cuh -- the persistent, warp-specialised tcgen05 GEMM kernel.
//
// C = A * B, A (M x K) and B (K x N) row-major 16-bit floats, fp32
// accumulation in tensor memory, C (M x N) row-major fp16/bf16/fp32.
//
// This is the tile-level GEMM of the TileLang skeleton ("TileScale 与
// TileLang比较", section 核心抽象与编程模型对比): per output tile, clear an
// accumulator, add the product of every BK-slice pair of A and B tiles staged
// in shared memory, then copy the tile out.  The pieces map as follows.
//   * shared-memory tiles A_s[BM, BK], B_s[BK, BN]  -> a ring of `stages`
//     slots filled by TMA tile copies (128-byte swizzle), each guarded by a
//     full/empty mbarrier pair (the software pipeline of T.Pipelined with
//     num_stages);
//   * fragment accumulator C_r[BM, BN]             -> fp32 columns of tensor
//     memory, double buffered so the epilogue of one tile overlaps the
//     main loop of the next;
//   * T.gemm                                        -> tcgen05.mma kind::f16
//     issued by a single thread, BK / 16 instructions per slice;
//   * T.copy(C_r, C)                                -> tcgen05.ld by an
//     epilogue warpgroup, fp32 -> output conversion, global stores;
//   * warp(group) specialisation by rank (TileScale README, T.Scale
//     "warpgroup" example): warp 0 produces, warp 1 issues MMAs, warps 2-5
//     drain the accumulator;
//   * persistent thread blocks (TileScale roadmap, resource control): every
//     CTA walks a static list of work units;
//   * the K split with a reduction (TileScale README, "Example of GEMM",
//     warpgroups split along K and reduce): work units may cover a K range
//     of a tile; partial tiles go to an fp32 workspace and the CTA that
//     finishes a tile last adds the partials in split order 0..S-1.
//
// Every wait is bounded in time (see WaitCtl); a CTA that gives up records a
// timeout in the status word, lets its in-flight copies and MMAs finish,
// frees tensor memory and returns.
#pragma once

#include "ptx.cuh"

namespace tsg {

constexpr int kBM = 128;        // accumulator rows = TMEM lanes
constexpr int kBK = 64;         // K per slice: one 128-byte swizzle row of 16-bit data
constexpr int kUmmaK = 16;      // K per tcgen05.mma kind::f16
constexpr int kThreads = 192;   // 6 warps
constexpr int kEpiThreads = 128;
constexpr int kMaxStages = 16;

enum OutKind { kOutF16 = 0, kOutBF16 = 1, kOutF32 = 2 };

struct GemmParams {
    int32_t M, N, K;
    int32_t tiles_m, tiles_n;
    int32_t splits;       // S
    int32_t kblocks;      // ceil(K / kBK)
    int32_t group_m;      // raster group height in tiles
    int32_t stages;
    int32_t debug_flags;
    int64_t units;        // tiles_m * tiles_n * S
    uint32_t idesc;       // tcgen05 instruction descriptor
    uint32_t pad_;
    void* C;
    float* ws;            // [tile][split][kBM][BN] fp32 partials (S > 1)
    int* counters;        // [tile] arrival counters, zero between launches
    int* status;          // plan status word
    uint64_t timeout_ns;
};

// Work unit u -> (tile row tm, tile column tn, split, linear tile).  Units
// of one tile are adjacent so its splits run at the same time; tiles are
// rastered in groups of `group_m` tile rows so that concurrently running
// CTAs share B panels (and A panels) in L2.
__device__ __forceinline__ void unit_coords(const GemmParams& p, int64_t u, int& tm, int& tn,
                                            int& split, int64_t& tile) {
    tile = u / p.splits;
    split = static_cast<int>(u - tile * p.splits);
    const int64_t span = static_cast<int64_t>(p.group_m) * p.tiles_n;
    const int64_t group = tile / span;
    const int first_m = static_cast<int>(group * p.group_m);
    const int gm = min(p.tiles_m - first_m, p.group_m);
    const int64_t r = tile - group * span;
    tm = first_m + static_cast<int>(r % gm);
    tn = static_cast<int>(r / gm);
}

__device__ __forceinline__ void split_range(const GemmParams& p, int split, int& kb0, int& kb1) {
    kb0 = static_cast<int>(static_cast<int64_t>(split) * p.kblocks / p.splits);
    kb1 = static_cast<int>(static_cast<int64_t>(split + 1) * p.kblocks / p.splits);
}

// Store 32 consecutive fp32 accumulator columns of one row of C, starting at
// column col0, converted to the output format.  Columns at or past N are
// skipped 16 bytes at a time (N * 2 is a multiple of 16, so a 16-byte vector
// is either wholly inside the row or wholly outside).
template <int kOut>
__device__ __forceinline__ void store_row32(const GemmParams& p, int row, int col0,
                                            const uint32_t (&r)[32]) {
    if (row >= p.M) return;
    if constexpr (kOut == kOutF32) {
        float* dst = static_cast<float*>(p.C) + static_cast<int64_t>(row) * p.N + col0;
#pragma unroll
        for (int v = 0; v < 8; ++v)
            if (col0 + 4 * v < p.N) st_global_v4(dst + 4 * v, r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
    } else {
        uint16_t* dst = static_cast<uint16_t*>(p.C) + static_cast<int64_t>(row) * p.N + col0;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            if (col0 + 8 * v < p.N) {
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float lo = __uint_as_float(r[8 * v + 2 * i]);
                    const float hi = __uint_as_float(r[8 * v + 2 * i + 1]);
                    w[i] = kOut == kOutBF16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
                }
                st_global_v4(dst + 8 * v, w[0], w[1], w[2], w[3]);
            }
        }
    }
}

template <int BN>
struct TileShape {
    static constexpr uint32_t kABytes = kBM * kBK * 2;   // 16 KiB
    static constexpr uint32_t kBBytes = BN * kBK * 2;    // BN / 64 boxes of 8 KiB
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    // TMEM column stride between the two accumulators and the allocation
    static constexpr uint32_t kAccCols = BN <= 64 ? 64 : (BN <= 128 ? 128 : 256);
    static constexpr uint32_t kTmemCols = 2 * kAccCols;
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN must be 64, 128, 192 or 256");
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
};

// Bytes of dynamic shared memory the kernel needs for `stages` slots.
template <int BN>
__host__ __device__ constexpr uint32_t smem_bytes_1sm(int stages) {
    return 1024u /* alignment slack */ + stages * TileShape<BN>::kStageBytes +
           8u * (2 * stages + 6) /* barriers */ + 16u /* tmem holder, flags */;
}

template <int BN, int kOut>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_sm103_1sm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
    using TS = TileShape<BN>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const int S = p.stages;

    const uint32_t bars = base + S * TS::kStageBytes;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
    auto tfull_bar = [&](int a) { return bars + 8u * (2 * S + a); };
    auto tempty_bar = [&](int a) { return bars + 8u * (2 * S + 2 + a); };
    const uint32_t drain_bar = bars + 8u * (2 * S + 4);
    const uint32_t epi_bar = bars + 8u * (2 * S + 5);
    uint8_t* misc = base_ptr + S * TS::kStageBytes + 8u * (2 * S + 6);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
    volatile int* last_flag = reinterpret_cast<volatile int*>(misc + 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), kEpiThreads);
        }
        mbar_init(drain_bar, 1);
        mbar_init(epi_bar, kEpiThreads / 32);
        *abort_flag = 0;
        *last_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) tmem_alloc<1>(smem_u32(tmem_holder), TS::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t outstanding = 0, out_parity = 0;  // loads not yet seen complete
            bool skip = (p.debug_flags & 1) && blockIdx.x == 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
                int tm, tn, split;
                int64_t tile;
                unit_coords(p, u, tm, tn, split, tile);
                int kb0, kb1;
                split_range(p, split, kb0, kb1);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, ctl)) {
                        ok = false;
                        break;
                    }
                    if (skip) {
                        skip = false;  // leave this slot's full barrier unsignalled
                    } else {
                        const uint32_t a_dst = base + stage * TS::kStageBytes;
                        mbar_arrive_expect_tx(full_bar(stage), TS::kStageBytes);
                        tma_load_2d(a_dst, &tmA, full_bar(stage), kb * kBK, tm * kBM);
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j)
                            tma_load_2d(a_dst + TS::kABytes + j * 8192u, &tmB, full_bar(stage),
                                        tn * BN + j * 64, kb * kBK);
                        outstanding |= 1u << stage;
                        out_parity = (out_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Let every copy this thread started land before the CTA exits.
            for (int s = 0; s < S; ++s)
                if (outstanding & (1u << s)) wait_bounded(full_bar(s), (out_parity >> s) & 1u, ctl, false);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
                int tm, tn, split;
                int64_t tile;
                unit_coords(p, u, tm, tn, split, tile);
                int kb0, kb1;
                split_range(p, split, kb0, kb1);
                if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, ctl)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * TS::kAccCols;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded(full_bar(stage), phase, ctl)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = base + stage * TS::kStageBytes;
                    const uint32_t b_addr = a_addr + TS::kABytes;
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        // A: K-major, rows 128 B apart, 8-row groups 1024 B apart;
                        //    the k-th 16-element step is 32 B along the row.
                        // B: MN-major, 64-column boxes 8 KiB apart (LBO), 8-row
                        //    groups 1024 B apart (SBO); the k-th step is 16 rows.
                        const uint64_t ad = smem_desc_sw128(a_addr + k * 32u, 16u, 1024u);
                        const uint64_t bd = smem_desc_sw128(b_addr + k * 2048u, 8192u, 1024u);
                        umma_f16<1>(d_tmem, ad, bd, p.idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit(empty_bar(stage));  // slot free once these MMAs have read it
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(tfull_bar(acc));  // accumulator complete
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // Every MMA issued above completes before tensor memory is freed.
            umma_commit(drain_bar);
            wait_bounded(drain_bar, 0u, ctl, false);
        }
        __syncwarp();
    } else {
        // --------------------------------------------------- epilogue --
        const int q = warp & 3;              // TMEM lane quarter of this warp
        const int etid = threadIdx.x - 64;   // 0..127
        const int row_local = q * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t epi_phase = 0;
        // Bounded barrier of the four epilogue warps (an mbarrier with one
        // arrival per warp), so that no epilogue warp can wait forever on a
        // warp that gave up.
        auto epi_sync = [&]() -> bool {
            __syncwarp();
            int good = 1;
            if (lane == 0) {
                mbar_arrive(epi_bar);
                good = wait_bounded(epi_bar, epi_phase, ctl) ? 1 : 0;
            }
            good = __shfl_sync(0xffffffffu, good, 0);
            epi_phase ^= 1u;
            return good != 0;
        };
        for (int64_t u = blockIdx.x; u < p.units; u += gridDim.x) {
            int tm, tn, split;
            int64_t tile;
            unit_coords(p, u, tm, tn, split, tile);
            int ok = 1;
            if (lane == 0) ok = wait_bounded(tfull_bar(acc), acc_phase, ctl) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            __syncwarp();
            tc_fence_after();
            const int row = tm * kBM + row_local;
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * TS::kAccCols;
            if (p.splits == 1) {
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tbase + c, r);
                    tmem_ld_wait();
                    store_row32<kOut>(p, row, tn * BN + c, r);
                }
                tc_fence_before();
                mbar_arrive(tempty_bar(acc));
            } else {
                float* wsp = p.ws + (tile * p.splits + split) * (kBM * BN) + row_local * BN;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tbase + c, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        st_global_v4(wsp + c + 4 * v, r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
                }
                tc_fence_before();
                mbar_arrive(tempty_bar(acc));
                // Publish the partial, then count arrivals for this tile.
                __threadfence();
                if (!epi_sync()) break;
                if (etid == 0) {
                    const int old = atomicAdd(p.counters + tile, 1);
                    *last_flag = (old == p.splits - 1) ? 1 : 0;
                }
                if (!epi_sync()) break;
                if (*last_flag) {
                    // Last CTA of this tile: C = p_0 + p_1 + ... + p_{S-1}.
                    __threadfence();
                    const float* t0 = p.ws + tile * p.splits * (kBM * BN) + row_local * BN;
#pragma unroll 1
                    for (int c = 0; c < BN; c += 32) {
                        uint32_t r[32];
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
                            for (int s = 0; s < p.splits; ++s) {
                                const float4 x = ld_global_cg_f4(t0 + static_cast<int64_t>(s) * (kBM * BN) + c + 4 * v);
                                a4.x += x.x;
                                a4.y += x.y;
                                a4.z += x.z;
                                a4.w += x.w;
                            }
                            r[4 * v] = __float_as_uint(a4.x);
                            r[4 * v + 1] = __float_as_uint(a4.y);
                            r[4 * v + 2] = __float_as_uint(a4.z);
                            r[4 * v + 3] = __float_as_uint(a4.w);
                        }
                        store_row32<kOut>(p, row, tn * BN + c, r);
                    }
                    if (etid == 0) p.counters[tile] = 0;  // ready for the next launch
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    // ------------------------------------------------------------ exit --
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc<1>(tmem_base, TS::kTmemCols);
    }
}

}  // namespace tsg
