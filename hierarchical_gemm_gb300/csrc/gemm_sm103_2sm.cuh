// gemm_sm103_2sm.cuh -- the CTA-pair form of the persistent GEMM kernel.
//
// The TileScale README (section on T.Scale) describes the Blackwell
// cluster-level GEMM as a distributed GEMM running on two SMs, and names a
// cluster-scale GEMM primitive built on distributed shared memory.  Here two
// CTAs of a 2 x 1 cluster compute one 256 x BN output tile together:
//   * CTA r of the pair loads rows [128 r, 128 r + 128) of the tile's A
//     panel and columns [r BN/2, (r + 1) BN/2) of its B panel into its own
//     shared memory (so each SM fetches half the B bytes it would for a
//     128 x BN tile of its own);
//   * the pair's leader (r = 0) issues tcgen05.mma.cta_group::2 with M = 256:
//     the tensor cores of both SMs read the A rows and B columns held by
//     both CTAs' shared memory -- the on-chip "network" of the cluster --
//     and each CTA's tensor memory receives its own 128 rows of the result;
//   * both CTAs' TMA loads complete on the leader's full barrier, which
//     expects the bytes of both; the leader's commits arrive on the empty
//     and accumulator-full barriers of both CTAs (one commit addressed to
//     both);
//   * each CTA's epilogue warpgroup drains its own 128 rows and tells the
//     leader (remote mbarrier arrive) when the accumulator is free again.
// Everything else -- the persistent schedule over work units, the split-K
// workspace reduction, the bounded waits -- is the one-SM kernel's.
//
// The pair is the only cluster shape: no operand tile is multicast.
#pragma once

#include "gemm_sm103.cuh"

namespace tsg {

// BN = 512 (a "wide" tile): the tile's two 256-column halves are the two
// accumulators of tensor memory (so one tile fills it and is not
// double-buffered), each K slice's A feeds two N = 256 MMAs, and each CTA
// holds two 128-column pieces of B, one per half.
template <int BN>
struct PairShape {
    static_assert(BN == 128 || BN == 256 || BN == 512, "pair tiles are 256 x 128, 256 x 256 or 256 x 512");
    static constexpr bool kWide = BN == 512;
    static constexpr uint32_t kABytes = kBM * kBK * 2;      // this CTA's 128 rows: 16 KiB
    static constexpr uint32_t kBCols = BN / 2;              // this CTA's B columns
    static constexpr uint32_t kPieceCols = kWide ? 128 : kBCols;  // B columns of one MMA's half
    static constexpr uint32_t kBBytes = kBCols * kBK * 2;   // kBCols / 64 boxes of 8 KiB
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kAccCols = BN <= 128 ? 128 : 256;
    static constexpr uint32_t kTmemCols = kWide ? 512 : 2 * kAccCols;
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
};

template <int BN, int kOut>
__host__ __device__ constexpr uint32_t smem_bytes_2sm(int stages) {
    return 1024u + stages * PairShape<BN>::kStageBytes + epi_smem_bytes<kOut>() + 8u * (2 * stages + 5) + 16u;
}

template <int BN, int kOut, int kLayout, bool kF8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_sm103_2sm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
    using PS = PairShape<BN>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const int S = p.stages;

    const uint32_t epi_smem = base + S * PS::kStageBytes;  // output staging
    const uint32_t bars = epi_smem + epi_smem_bytes<kOut>();
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
    auto tfull_bar = [&](int a) { return bars + 8u * (2 * S + a); };
    auto tempty_bar = [&](int a) { return bars + 8u * (2 * S + 2 + a); };
    const uint32_t drain_bar = bars + 8u * (2 * S + 4);
    uint8_t* misc = base_ptr + S * PS::kStageBytes + epi_smem_bytes<kOut>() + 8u * (2 * S + 5);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t half = cluster_ctarank();  // 0: the pair's leader, 1: its peer
    const bool leader = half == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);   // the leader's producer arrives once
            mbar_init(empty_bar(s), 1);  // the leader's commit, which arrives in both CTAs
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);                    // the leader's commit
            // every epilogue warp of the pair (wide tiles: accumulator a is
            // drained by warpgroup a of each CTA)
            mbar_init(tempty_bar(a), PS::kWide ? kEpiWarps : 2 * kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmC);
    }
    if (warp == 1) tmem_alloc<2>(smem_u32(tmem_holder), PS::kTmemCols);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // barriers of every CTA initialised before any uses them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
    ctl.peer_abort[ctl.npeers++] = mapa_shared(smem_u32(const_cast<int*>(abort_flag)), half ^ 1u);

    const int64_t cluster_id = blockIdx.x / 2;
    const int64_t nclusters = gridDim.x / 2;

    if (warp == 0) {
        // ------------------------------------------- TMA producer (both) --
        // (lane 0 alone runs the loop; the warp reconverges below)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t outstanding = 0, out_parity = 0;
            // tests only: the first pair's leader leaves its first slot
            // unannounced, so the MMA issuer's bounded wait runs out
            bool skip = (p.debug_flags & 1) && cluster_id == 0 && leader;
            bool ok = true;
            for (int64_t j = 0; ok; ++j) {
                Unit un;
                if (!unit_at(p, cluster_id, nclusters, j, un)) break;
                // Whole tiles of odd rounds walk K backwards: a round then starts on
                // the panel slices the round before ended on, which are still in L2
                // (16384 x 16384 x 8192: up to 6 % fewer DRAM reads).  The MMA issuer
                // needs no change: it takes the slices in ring order.
                const bool rev = un.nsplit == 1 && (j & 1);
                for (int kq = un.kb0; kq < un.kb1; ++kq) {
                    const int kb = rev ? un.kb0 + un.kb1 - 1 - kq : kq;
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, ctl)) {
                        ok = false;
                        break;
                    }
                    if (skip) {
                        skip = false;
                    } else {
                        const uint32_t a_dst = base + stage * PS::kStageBytes;
                        const int32_t arow = un.tm * (2 * kBM) + static_cast<int32_t>(half) * kBM;
                        // (wide tiles: this CTA's piece of each 256-column half)
                        const int32_t bcol = un.tn * BN + static_cast<int32_t>(half) * PS::kPieceCols;
                        constexpr uint32_t kPieceBytes = PS::kPieceCols * kBK * 2;
                        if (leader) {
                            mbar_arrive_expect_tx(full_bar(stage), 2u * PS::kStageBytes);
                            load_slice<kLayout, PS::kPieceCols, false, kF8>(a_dst, a_dst + PS::kABytes, &tmA, &tmB,
                                                                            full_bar(stage), kb, arow, bcol);
                            if constexpr (PS::kWide)
                                load_b<kLayout, PS::kPieceCols, false, kF8>(a_dst + PS::kABytes + kPieceBytes, &tmB,
                                                                            full_bar(stage), kb, bcol + 256);
                        } else {
                            const uint32_t fb = mapa_shared(full_bar(stage), 0u);
                            load_slice<kLayout, PS::kPieceCols, true, kF8>(a_dst, a_dst + PS::kABytes, &tmA, &tmB,
                                                                           fb, kb, arow, bcol);
                            if constexpr (PS::kWide)
                                load_b<kLayout, PS::kPieceCols, true, kF8>(a_dst + PS::kABytes + kPieceBytes, &tmB,
                                                                           fb, kb, bcol + 256);
                        }
                        outstanding |= 1u << stage;
                        out_parity = (out_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < S; ++s) {
                if (!(outstanding & (1u << s))) continue;
                const uint32_t par = (out_parity >> s) & 1u;
                wait_bounded(leader ? full_bar(s) : empty_bar(s), par, ctl, false);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------ MMA issuer (leader) --
        if (leader && lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int64_t j = 0; ok; ++j) {
                Unit un;
                if (!unit_at(p, cluster_id, nclusters, j, un)) break;
                // a wide tile takes both accumulators, whose halves the two
                // epilogue warpgroups free separately
                if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, ctl)) break;
                if (PS::kWide && !wait_bounded(tempty_bar(1), acc_phase ^ 1u, ctl)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * PS::kAccCols;
                for (int kb = un.kb0; kb < un.kb1; ++kb) {
                    if (!wait_bounded(full_bar(stage), phase, ctl)) {
                        ok = false;
                        break;
                    }
                    // (TMA-written operands are visible to the MMA once the
                    // full barrier completes; no tcgen05 fence is needed.)
                    {
                        const uint32_t a_addr = base + stage * PS::kStageBytes;
                        mma_slice<kLayout, 2, kF8>(d_tmem, a_addr, a_addr + PS::kABytes, p.idesc,
                                              kb > un.kb0 ? 1u : 0u);
                        if constexpr (PS::kWide)  // the tile's second 256 columns
                            mma_slice<kLayout, 2, kF8>(d_tmem + 256u, a_addr,
                                                       a_addr + PS::kABytes + PS::kPieceCols * kBK * 2, p.idesc,
                                                       kb > un.kb0 ? 1u : 0u);
                        // slot free in both CTAs, whose slots these MMAs read
                        umma_commit_pair(empty_bar(stage), 0x3u);
                    }
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair(tfull_bar(acc), 0x3u);
                if (PS::kWide) {
                    acc_phase ^= 1u;  // (acc stays 0: one tile at a time)
                } else if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            umma_commit_pair(drain_bar, 0x1u);
            wait_bounded(drain_bar, 0u, ctl, false);
        }
        __syncwarp();
    } else {
        // ----------------------------------------------- epilogue (both) --
        const int q = warp & 3;                   // TMEM lane quarter of this warp
        const int e = warp - 2;                   // epilogue warp 0..7
        const int c_begin = (e >> 2) * (BN / 2);  // warpgroup e/4 drains this half of the columns
        const int etid = threadIdx.x - 64;
        const int row_local = q * 32 + lane;
        CStager<kOut> out{epi_smem + static_cast<uint32_t>(e) * 2u * epi_buf_bytes<kOut>(), 0u, lane};
        int acc = 0;
        uint32_t acc_phase = 0;
        // Release accumulator `a` to the leader's MMA issuer.
        auto release_acc = [&](int a) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    mbar_arrive(tempty_bar(a));
                else
                    mbar_arrive_cluster(tempty_bar(a), 0u);
            }
        };
        const EpiAux aux{cluster_id * 2 + half, 2};
        for (int64_t j = 0;; ++j) {
            Unit un;
            if (!unit_at(p, cluster_id, nclusters, j, un)) break;
            const int tm = un.tm;
            prefetch_sk_partials<BN>(p, un, aux, etid);
            int ok = 1;
            if (lane == 0) ok = wait_bounded(tfull_bar(acc), acc_phase, ctl) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            __syncwarp();
            tc_fence_after();
            const int row0 = tm * (2 * kBM) + static_cast<int>(half) * kBM + q * 32;
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * PS::kAccCols;
            // workspace tile and counter of this CTA's 128-row half
            const int64_t wh = un.slot * 2 + half;
            // (wide tiles: warpgroup e/4 drains accumulator e/4, the tile's
            // columns [256 (e/4), 256 (e/4) + 256), which are TMEM columns
            // of the same numbers)
            const int a_now = PS::kWide ? (e >> 2) : acc;
            drain_unit<BN, kOut>(p, &tmC, out, un, tbase, row0, row_local, wh, aux, c_begin,
                                 [&]() { release_acc(a_now); });
            if (PS::kWide) {
                acc_phase ^= 1u;
            } else if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        out.drain();  // this warp's output stores have read shared memory
    }

    // ------------------------------------------------------------ exit --
    // No CTA leaves while another may still read or write its shared memory
    // or signal its barriers; tensor memory of a pair is freed together.
    // The barriers here are the non-aligned forms, which count threads one
    // by one, so warps whose lane 0 ran a role loop alone may arrive in any
    // convergence state.
    tc_fence_before();
    cta_barrier_any();
    cluster_barrier_any();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc<2>(tmem_base, PS::kTmemCols);
    }
}

}  // namespace tsg
