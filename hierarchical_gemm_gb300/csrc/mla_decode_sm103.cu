// mla_decode_sm103.cu -- the MLA decode shape of the attention block
// (tsattn_mla_decode in tsattn.h) on tcgen05, on CTA pairs.
//
// The FlashMLA example of the TileScale README (section "Example of
// FlashMLA") decodes one query token per sequence: per batch b and block of
// query heads, scores acc_s = Q KV^T + Q_pe K_pe^T over the latent (512)
// and rotary (64) parts, a running row maximum and row sums, weights
// exp2(scale s - scale m) cast to the input format, acc_o = acc_o * scale +
// P KV -- the latent KV is also the value -- and acc_o / logsum at the end.
// Per head that is O = softmax(scale [Q Q_pe] [KV K_pe]^T) KV with 576-deep
// scores and 512-wide values.
//
// A 128 x 512 fp32 output accumulator would take all of one SM's tensor
// memory, so a cluster of two CTAs shares each (batch, 128 heads):
//   * CTA r keeps the output columns [256 r, 256 r + 256) in tensor memory
//     (256 columns) and multiplies by the value columns it needs, the same
//     latent columns of each key block that it loads for the scores;
//   * the scores' 576-deep contraction is split between the pair: CTA 0 over
//     latent dims [0, 256), CTA 1 over latent dims [256, 512) and the 64
//     rotary dims; each holds only its part of every key block in shared
//     memory, and its latent part of Q in tensor memory (the A operand of
//     the score MMAs, written there once by the softmax threads, a row
//     each); CTA 1's rotary part of Q stays in shared memory;
//   * each CTA's softmax warpgroup (a thread per query head) reads its fp32
//     partial scores from tensor memory, writes them into the partner's
//     shared memory (distributed shared memory, st.shared::cluster), and adds
//     the partner's partial to its own: both CTAs then hold the same full
//     scores (the addition is commutative, so the sums agree bit for bit),
//     keep the same running maximum and row sums, and form the same weights
//     P, which each writes into its own shared memory (128-byte swizzle) as
//     the A operand of its P V;
//   * the exchange has a warpgroup of its own, a thread per head: it reads
//     each block's partial from tensor memory and writes it into the
//     partner's exchange buffer (two buffers) while the softmax warpgroup
//     is still on an earlier block, so the exchange and the softmax overlap;
//     the tensor cores compute block j + 2's partial scores as soon as both
//     warpgroups have read block j's (two score buffers).
// Warps 0-3 run the softmax and epilogue and warps 4-7 the exchange (warp w
// reads tensor-memory lanes 32 (w mod 4) .. +31), warp 8 lane 0 loads CTA
// 1's rotary part of Q once and streams key blocks through a three-slot
// ring (optionally asking for later blocks in L2 ahead), warp 9 lane 0
// issues the MMAs, and warp 10 lane 0 relays to the partner that the
// softmax warps have read its partial (the one cross-CTA release of the
// exchange).  Every wait is
// bounded in time; a CTA that gives up records a timeout, sets its
// partner's abort flag, lets its copies and MMAs finish, frees tensor
// memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "attn_common.h"
#include "ptx.cuh"
#include "tsattn.h"

namespace tsg {
namespace mla {

constexpr int kH = 128;                 // query heads per CTA pair (TMEM lanes)
constexpr int kN = 64;                  // keys per block
constexpr int kDL = 512;                // latent (= value) dims
constexpr int kDR = 64;                 // rotary dims
constexpr int kVHalf = kDL / 2;         // value columns per CTA
constexpr int kThreads = 352;           // warps 0-3 softmax, 4-7 exchange, 8 loads, 9 MMAs, 10 relay
constexpr int kWarpSend = 4, kWarpLoad = 8, kWarpMma = 9, kWarpRelay = 10;
constexpr int kSlots = 3;               // key block ring depth
// a 64-dim column of the 128-byte swizzle: 128 heads or 64 keys x 128 bytes
constexpr uint32_t kQAtom = kH * 128u;  // 16 KiB
constexpr uint32_t kKAtom = kN * 128u;  // 8 KiB
constexpr int kMaxAtoms = 5;            // CTA 0: 4 latent atoms; CTA 1: 4 latent + 1 rotary
constexpr uint32_t kSlotBytes = kMaxAtoms * kKAtom;          // 40 KiB
constexpr uint32_t kXBytes = kH * kN * 4u;                   // a partner's fp32 partial scores
constexpr uint32_t kQOff = 0;                                // CTA 1: the rotary part of Q
constexpr uint32_t kPOff = kQOff + kQAtom;                   // the weights P (128 x 64, 16 KiB)
constexpr uint32_t kKOff = kPOff + kQAtom;
constexpr uint32_t kXOff = kKOff + kSlots * kSlotBytes;      // two exchange buffers
constexpr uint32_t kBarOff = kXOff + 2 * kXBytes;
// barriers: q_full, qt_full, kv_full[3], kv_empty[3], s_full[2], s_free[2],
// p_full, pv_done, x_full[2], x_free[2], drain, x_read[2]
constexpr int kNumBars = 2 + 2 * kSlots + 4 + 2 + 4 + 1 + 2;
constexpr uint32_t kMiscOff = kBarOff + 8u * kNumBars;
constexpr uint32_t kSmemBytes = 1024u + kMiscOff + 16u;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kTmemCols = 512;     // O at 0 (256 columns), score buffer i at 256 + 64 i,
constexpr uint32_t kSCol = 256;         // the latent part of Q at 384 (two elements per column)
constexpr uint32_t kQCol = 384;
constexpr float kRescaleLog2 = 8.0f;    // lazy-rescale threshold (base-2 units)
constexpr int kDefaultPrefetch = 0;     // key blocks asked for in L2 ahead of the ring

struct MlaParams {
    const void* Q;        // [B][H][512]: each softmax thread copies its head's part into tensor memory
    int32_t B, H, Skv;
    int32_t nblk;         // key blocks: ceil(Skv / 64)
    float scale_log2;     // scale * log2(e)
    int32_t prefetch;     // key blocks asked for in L2 ahead of the one loaded (0: none)
    int32_t debug_flags;
    void* O;
    int* status;
    uint64_t timeout_ns;
};

// tcgen05 instruction descriptor, kind::f16, fp32 accumulator, M = 128;
// A K-major; B K-major (keys as N) or N-major (value columns as N).
__host__ __device__ constexpr uint32_t idesc(bool f16, uint32_t n, bool b_nmajor) {
    return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) | ((b_nmajor ? 1u : 0u) << 16) |
           ((n >> 3) << 17) | ((128u >> 4) << 24);
}

struct Bars {
    uint32_t b;
    __device__ uint32_t q_full() const { return b; }                                   // rotary Q (TMA)
    __device__ uint32_t qt_full() const { return b + 8u; }                             // latent Q in tensor memory
    __device__ uint32_t kv_full(int s) const { return b + 8u * (2 + s); }
    __device__ uint32_t kv_empty(int s) const { return b + 8u * (2 + kSlots + s); }
    __device__ uint32_t s_full(int i) const { return b + 8u * (2 + 2 * kSlots + i); }  // partial scores ready
    __device__ uint32_t s_free(int i) const { return b + 8u * (4 + 2 * kSlots + i); }  // ... read by both warpgroups
    __device__ uint32_t p_full() const { return b + 8u * (6 + 2 * kSlots); }           // P written
    __device__ uint32_t pv_done() const { return b + 8u * (7 + 2 * kSlots); }          // a P V complete
    __device__ uint32_t x_full(int i) const { return b + 8u * (8 + 2 * kSlots + i); }  // partner's partial here
    __device__ uint32_t x_free(int i) const { return b + 8u * (10 + 2 * kSlots + i); } // partner read ours
    __device__ uint32_t drain() const { return b + 8u * (12 + 2 * kSlots); }
    __device__ uint32_t x_read(int i) const { return b + 8u * (13 + 2 * kSlots + i); } // we read the partner's
};

// One softmax thread: query head row r = 32 quarter + lane of the CTA's 128
// heads.
template <bool kF16>
__device__ __forceinline__ void softmax_rows(const MlaParams& p, const Bars& bar, uint32_t tmem, uint32_t base,
                                             uint32_t peer, int b, int h0, int quarter, int lane,
                                             const WaitCtl& ctl) {
    const int r = quarter * 32 + lane;  // head within the block
    const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c2 = p.scale_log2;
    // every thread waits itself: each then reads or overwrites only its own
    // row, after the barrier's acquire
    auto wait_cluster = [&](uint32_t bb, uint32_t parity) { return wait_bounded<true>(bb, parity, ctl); };
    auto warp_wait = [&](uint32_t bb, uint32_t parity) -> bool {
        int good = 1;
        if (lane == 0) good = wait_bounded(bb, parity, ctl) ? 1 : 0;
        return __shfl_sync(0xffffffffu, good, 0) != 0;
    };
    // exchange buffer i, row r: 16-byte chunk c at + c * 2 KiB
    auto xaddr = [&](int i) { return base + kXOff + static_cast<uint32_t>(i) * kXBytes + static_cast<uint32_t>(r) * 16u; };
    // This head's latent part of Q (256 dims, two per 32-bit column, as
    // they lie in memory) into tensor memory, the score MMAs' A operand;
    // heads past H are zero.
    {
        const uint32_t rank = cluster_ctarank();
        const int head = h0 + r;
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.Q) +
                               ((static_cast<int64_t>(b) * p.H + head) * kDL + rank * kVHalf) / 2;
#pragma unroll 1
        for (int c = 0; c < kVHalf / 2; c += 32) {
            uint32_t v[32];
#pragma unroll
            for (int q = 0; q < 32; q += 4) {
                uint4 x4 = make_uint4(0u, 0u, 0u, 0u);
                if (head < p.H) x4 = __ldg(reinterpret_cast<const uint4*>(qrow + c + q));
                v[q] = x4.x;
                v[q + 1] = x4.y;
                v[q + 2] = x4.z;
                v[q + 3] = x4.w;
            }
            tmem_st_32x32b_x32(trow + kQCol + c, v);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.qt_full());
    }
    // x_full(i) completes once the partner's kXBytes of block j (i = j & 1)
    // have landed and this CTA has armed it for that block: blocks 0 and 1
    // now, block j + 2 once block j has been read out of the buffer
    if (r == 0) {
        mbar_arrive_expect_tx(bar.x_full(0), kXBytes);
        if (p.nblk > 1) mbar_arrive_expect_tx(bar.x_full(1), kXBytes);
    }
    float m_used = -INFINITY;  // base-2 maximum the weights are taken against
    float l = 0.0f;
    bool ok = true;
    // the weights' row in the 128-byte swizzle: 16-byte chunk c of row r at
    // r * 128 + ((c ^ (r mod 8)) * 16)
    const uint32_t prow = base + kPOff + static_cast<uint32_t>(r) * 128u;
    for (int j = 0; ok && j < p.nblk; ++j) {
        const int i = j & 1;
        // this block's own partial (the exchange warpgroup reads it too),
        // then the partner's, added in
        if (!warp_wait(bar.s_full(i), static_cast<uint32_t>(j >> 1) & 1u)) {
            ok = false;
            break;
        }
        tc_fence_after();
        uint32_t own[64];
        tmem_ld_32x32b_x32(trow + kSCol + 64u * i, *reinterpret_cast<uint32_t(*)[32]>(own));
        tmem_ld_32x32b_x32(trow + kSCol + 64u * i + 32u, *reinterpret_cast<uint32_t(*)[32]>(own + 32));
        tmem_ld_wait();
        float f[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) f[c] = __uint_as_float(own[c]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.s_free(i));
        if (!wait_cluster(bar.x_full(i), static_cast<uint32_t>(j >> 1) & 1u)) {
            ok = false;
            break;
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const float4 v = ld_shared_f4(xaddr(i) + c * 2048u);
            f[4 * c] += v.x;
            f[4 * c + 1] += v.y;
            f[4 * c + 2] += v.z;
            f[4 * c + 3] += v.w;
        }
        if (r == 0 && j + 2 < p.nblk) mbar_arrive_expect_tx(bar.x_full(i), kXBytes);  // for block j + 2
        // this warp has read the partner's partial: the relay thread tells
        // the partner, which may then write block j + 2 here
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.x_read(i));
        // keys past Skv weigh nothing
        const int k0 = j * kN;
        if (k0 + kN > p.Skv) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
                if (k0 + c >= p.Skv) f[c] = -INFINITY;
        }
        float mx[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) mx[q] = f[q];
#pragma unroll
        for (int c = 4; c < 64; c += 8) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                asm("max.f32 %0, %1, %2, %3;" : "=f"(mx[q]) : "f"(mx[q]), "f"(f[c + q]), "f"(f[c + 4 + q]));
        }
        const float mb = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        const float m_new = fmaxf(m_used, mb * c2);  // (c2 > 0)
        const bool need = m_used == -INFINITY ? m_new > -INFINITY : m_new > m_used + kRescaleLog2;
        // P V of block j - 1 complete: its weights may be overwritten, and the
        // output accumulator holds P_0 V + ... + P_{j-1} V
        if (j >= 1 && !warp_wait(bar.pv_done(), static_cast<uint32_t>(j - 1) & 1u)) {
            ok = false;
            break;
        }
        if (__any_sync(0xffffffffu, need)) {
            // every lane of the warp moves to its own new maximum
            const float alpha = m_used == -INFINITY ? 0.0f : ex2_approx(m_used - m_new);
            if (m_new > -INFINITY) m_used = m_new;
            l *= alpha;
            if (j >= 1) {
                tc_fence_after();
                const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
                for (int c = 0; c < kVHalf; c += 32) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(trow + c, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 32; q += 2) {
                        const float2 v = mul2(make_float2(__uint_as_float(o[q]), __uint_as_float(o[q + 1])), a2);
                        o[q] = __float_as_uint(v.x);
                        o[q + 1] = __float_as_uint(v.y);
                    }
                    tmem_st_32x32b_x32(trow + c, o);
                }
                tmem_st_wait();
                tc_fence_before();
            }
        }
        // p = 2^(c2 s - m), two weights per packed fused multiply-add, into
        // this row of P in shared memory
        const float mneg = m_used == -INFINITY ? -INFINITY : -m_used;
        const float2 c22 = make_float2(c2, c2), mn2 = make_float2(mneg, mneg);
        float2 rsum[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) rsum[q] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e = 8 * c + 2 * q;
                const float2 x = fma2(make_float2(f[e], f[e + 1]), c22, mn2);
                const float2 pw = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                rsum[q] = add2(rsum[q], pw);
                w[q] = kF16 ? pack_f16x2(pw.x, pw.y) : pack_bf16x2(pw.x, pw.y);
            }
            st_shared_v4(prow + ((static_cast<uint32_t>(c) ^ (static_cast<uint32_t>(r) & 7u)) << 4), w[0], w[1], w[2],
                         w[3]);
        }
        l += ((rsum[0].x + rsum[0].y) + (rsum[1].x + rsum[1].y)) + ((rsum[2].x + rsum[2].y) + (rsum[3].x + rsum[3].y));
        fence_proxy_async_shared();  // the MMA reads P through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.p_full());
    }
    // ---------------------------------------------------- epilogue --
    if (ok && !warp_wait(bar.pv_done(), static_cast<uint32_t>(p.nblk - 1) & 1u)) ok = false;
    if (!ok) return;
    tc_fence_after();
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    const int head = h0 + r;
    const uint32_t rank = cluster_ctarank();
    uint16_t* orow = static_cast<uint16_t*>(p.O) + (static_cast<int64_t>(b) * p.H + head) * kDL + rank * kVHalf;
#pragma unroll 1
    for (int c = 0; c < kVHalf; c += 32) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(trow + c, o);
        tmem_ld_wait();
        uint32_t wv[16];
        const float2 inv2 = make_float2(inv, inv);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float2 v = mul2(make_float2(__uint_as_float(o[2 * q]), __uint_as_float(o[2 * q + 1])), inv2);
            wv[q] = kF16 ? pack_f16x2(v.x, v.y) : pack_bf16x2(v.x, v.y);
        }
        if (head < p.H) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
                st_global_v4(orow + c + 8 * v, wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
        }
    }
}

// One exchange thread, head row r = 32 quarter + lane: block j's partial
// scores from score buffer j & 1 into the partner's exchange buffer j & 1,
// once the partner's softmax has read block j - 2 there.  The stores are
// asynchronous and complete as transaction bytes on the partner's x_full
// barrier, which the partner arms (expects kXBytes) once per block.
__device__ __forceinline__ void send_rows(const MlaParams& p, const Bars& bar, uint32_t tmem, uint32_t base,
                                          uint32_t peer, int quarter, int lane, const WaitCtl& ctl) {
    const int r = quarter * 32 + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    // exchange buffer i, row r: 16-byte chunk c at + c * 2 KiB
    const uint32_t xrow = base + kXOff + static_cast<uint32_t>(r) * 16u;
    for (int j = 0; j < p.nblk; ++j) {
        const int i = j & 1;
        int good = 1;
        if (lane == 0) good = wait_bounded(bar.s_full(i), static_cast<uint32_t>(j >> 1) & 1u, ctl) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, good, 0)) return;
        tc_fence_after();
        uint32_t v[64];
        tmem_ld_32x32b_x32(trow + kSCol + 64u * i, *reinterpret_cast<uint32_t(*)[32]>(v));
        tmem_ld_32x32b_x32(trow + kSCol + 64u * i + 32u, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.s_free(i));
        // every thread waits itself: it then overwrites only its own row
        if (j >= 2 && !wait_bounded<true>(bar.x_free(i), static_cast<uint32_t>((j - 2) >> 1) & 1u, ctl)) return;
        // asynchronous stores that complete as transaction bytes on the
        // partner's x_full barrier, which the partner arms for every block
        const uint32_t dst = mapa_shared(xrow + static_cast<uint32_t>(i) * kXBytes, peer);
        const uint32_t fb = mapa_shared(bar.x_full(i), peer);
#pragma unroll
        for (int c = 0; c < 16; ++c) st_async_v4(dst + c * 2048u, v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3], fb);
    }
}

template <bool kF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_sm103(const __grid_constant__ CUtensorMap tmQpe, const __grid_constant__ CUtensorMap tmKV,
                     const __grid_constant__ CUtensorMap tmKpe, const MlaParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const Bars bar{base + kBarOff};
    uint8_t* misc = base_ptr + kMiscOff;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();   // 0: latent dims [0, 256); 1: [256, 512) and the rotary dims
    const uint32_t peer = rank ^ 1u;
    const int cluster = static_cast<int>(blockIdx.x >> 1);
    const int hblocks = (p.H + kH - 1) / kH;
    const int b = cluster / hblocks;
    const int h0 = (cluster % hblocks) * kH;
    const int natoms = rank == 0 ? 4 : 5;       // 64-dim columns of this CTA's part of the scores

    if (threadIdx.x == 0) {
        mbar_init(bar.q_full(), 1);
        mbar_init(bar.qt_full(), 4);  // every softmax warp
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(bar.kv_full(s), 1);
            mbar_init(bar.kv_empty(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar.s_full(i), 1);
            mbar_init(bar.s_free(i), 8);    // every softmax and exchange warp
            mbar_init(bar.x_full(i), 1);    // armed by this CTA; the partner's bytes complete it
            mbar_init(bar.x_free(i), 1);    // the partner's relay thread
            mbar_init(bar.x_read(i), 4);    // every softmax warp
        }
        mbar_init(bar.p_full(), 4);
        mbar_init(bar.pv_done(), 1);
        mbar_init(bar.drain(), 1);
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tmQpe);
        prefetch_tmap(&tmKV);
        prefetch_tmap(&tmKpe);
    }
    if (warp == kWarpMma) tmem_alloc<1>(smem_u32(tmem_holder), kTmemCols);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers initialised before either uses them
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
    ctl.peer_abort[ctl.npeers++] = mapa_shared(smem_u32(const_cast<int*>(abort_flag)), peer);

    if (warp < kWarpSend) {
        // ---------------------------------------- softmax and epilogue --
        softmax_rows<kF16>(p, bar, tmem, base, peer, b, h0, warp, lane, ctl);
    } else if (warp < kWarpLoad) {
        // ---------------------------------------------------- exchange --
        send_rows(p, bar, tmem, base, peer, warp - kWarpSend, lane, ctl);
    } else if (warp == kWarpRelay) {
        // ----------------------------------------------------- relay --
        // A cluster-scope release arrive costs its thread about a
        // microsecond; one thread here takes it for the softmax warps,
        // which only arrive on the local x_read barrier.  Their reads of
        // the partner's partial happen before this thread's release, which
        // covers them.
        if (lane == 0) {
            for (int j = 0; j < p.nblk; ++j) {
                const int i = j & 1;
                if (!wait_bounded(bar.x_read(i), static_cast<uint32_t>(j >> 1) & 1u, ctl)) break;
                mbar_arrive_cluster(bar.x_free(i), peer);
            }
        }
        __syncwarp();
    } else if (warp == kWarpLoad) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            // CTA r's columns of a key block: latent dims 256 r + 64 a for
            // a < 4; CTA 1's fifth column is the rotary part
            auto atom_map = [&](int a) -> const CUtensorMap* { return a < 4 ? &tmKV : &tmKpe; };
            auto atom_x = [&](int a) { return a < 4 ? static_cast<int32_t>(rank) * kVHalf + 64 * a : 0; };
            if (rank == 1) {
                mbar_arrive_expect_tx(bar.q_full(), kQAtom);
                tma_load_3d(base + kQOff, &tmQpe, bar.q_full(), 0, h0, b);
            } else {
                mbar_arrive(bar.q_full());
            }
            for (int j = kSlots; j < p.prefetch && j < p.nblk; ++j)
                for (int a = 0; a < natoms; ++a) tma_prefetch_3d(atom_map(a), atom_x(a), j * kN, b);
            uint32_t outstanding = 0, out_par = 0;
            for (int j = 0; j < p.nblk; ++j) {
                const int st = j % kSlots;
                const uint32_t ph = static_cast<uint32_t>(j / kSlots) & 1u;
                if (!wait_bounded(bar.kv_empty(st), ph ^ 1u, ctl)) break;
                if (p.prefetch > 0 && j + p.prefetch < p.nblk)
                    for (int a = 0; a < natoms; ++a)
                        tma_prefetch_3d(atom_map(a), atom_x(a), (j + p.prefetch) * kN, b);
                // tests only: the first pair's first CTA leaves its first block unloaded
                if ((p.debug_flags & 1) && cluster == 0 && rank == 0 && j == 0) continue;
                const uint32_t dst = base + kKOff + st * kSlotBytes;
                mbar_arrive_expect_tx(bar.kv_full(st), natoms * kKAtom);
                for (int a = 0; a < natoms; ++a)
                    tma_load_3d(dst + a * kKAtom, atom_map(a), bar.kv_full(st), atom_x(a), j * kN, b);
                outstanding |= 1u << st;
                out_par = (out_par & ~(1u << st)) | (ph << st);
            }
            // every copy this thread started lands before the CTA exits
            wait_bounded(bar.q_full(), 0u, ctl, false);
            for (int s = 0; s < kSlots; ++s)
                if (outstanding & (1u << s)) wait_bounded(bar.kv_full(s), (out_par >> s) & 1u, ctl, false);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc(kF16, kN, false), kIdPV = idesc(kF16, kVHalf, true);
            bool ok = wait_bounded(bar.q_full(), 0u, ctl) && wait_bounded(bar.qt_full(), 0u, ctl);
            // partial S_j = Q_r K_{j,r}^T into score buffer j & 1, 16 dims
            // per step: the latent part with Q from tensor memory (8
            // columns a step), CTA 1's rotary part with Q from shared
            // memory; K K-major (32 bytes along a row of a 64-dim column a
            // step).  For j >= 2 the softmax has read block j - 2 out of the
            // buffer first.
            auto issue_s = [&](int j) -> bool {
                const int st = j % kSlots;
                if (j >= 2 && !wait_bounded(bar.s_free(j & 1), static_cast<uint32_t>((j - 2) >> 1) & 1u, ctl))
                    return false;
                if (!wait_bounded(bar.kv_full(st), static_cast<uint32_t>(j / kSlots) & 1u, ctl)) return false;
                tc_fence_after();
                const uint32_t ks = base + kKOff + st * kSlotBytes;
                const uint32_t d = tmem + kSCol + 64u * (j & 1);
                for (int k = 0; k < 16; ++k) {
                    const uint64_t bd = smem_desc_sw128(ks + (k >> 2) * kKAtom + (k & 3) * 32u, 16u, 1024u);
                    umma_f16_ta(d, tmem + kQCol + 8u * k, bd, kIdS, k > 0 ? 1u : 0u);
                }
                if (natoms == 5) {
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t ad = smem_desc_sw128(base + kQOff + k * 32u, 16u, 1024u);
                        const uint64_t bd = smem_desc_sw128(ks + 4 * kKAtom + k * 32u, 16u, 1024u);
                        umma_f16<1>(d, ad, bd, kIdS, 1u);
                    }
                }
                umma_commit(bar.s_full(j & 1));
                return true;
            };
            // O_r += P_j V_{j,r}: P (128 heads x 64 keys, K-major in the
            // 128-byte swizzle) from shared memory; V the N-major B operand
            // over the CTA's four latent columns of the block (64-dim
            // columns 8 KiB apart, 8-key groups 1 KiB apart, the k-th 16-key
            // step 2 KiB on).
            auto issue_pv = [&](int j) -> bool {
                if (!wait_bounded(bar.p_full(), static_cast<uint32_t>(j) & 1u, ctl)) return false;
                tc_fence_after();
                const uint32_t vs = base + kKOff + (j % kSlots) * kSlotBytes;
#pragma unroll
                for (int k = 0; k < kN / 16; ++k) {
                    const uint64_t ad = smem_desc_sw128(base + kPOff + k * 32u, 16u, 1024u);
                    const uint64_t bd = smem_desc_sw128(vs + k * 2048u, kKAtom, 1024u);
                    umma_f16<1>(tmem, ad, bd, kIdPV, (j > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit(bar.pv_done());
                umma_commit(bar.kv_empty(j % kSlots));  // the block's scores and values are read
                return true;
            };
            // S_0, S_1; then per block j: P V_j (once the softmax has written
            // P_j), which frees the block's ring slot for block j + 3, then
            // S_{j+2} (once both warpgroups have read S_j and block j + 2 is
            // in) -- P V_j never waits for a later block's copy
            if (ok) ok = issue_s(0);
            if (ok && p.nblk > 1) ok = issue_s(1);
            for (int j = 0; ok && j < p.nblk; ++j) {
                ok = issue_pv(j);
                if (ok && j + 2 < p.nblk) ok = issue_s(j + 2);
            }
            // every MMA issued above completes before tensor memory is freed
            umma_commit(bar.drain());
            wait_bounded(bar.drain(), 0u, ctl, false);
        }
        __syncwarp();
    }

    // ------------------------------------------------------------ exit --
    // neither CTA leaves while the partner may still write into its shared
    // memory or arrive on its barriers (non-aligned barriers: warps whose
    // lane 0 ran a role loop alone may arrive in any convergence state)
    tc_fence_before();
    cta_barrier_any();
    cluster_barrier_any();
    if (warp == kWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc<1>(tmem, kTmemCols);
    }
}

// --------------------------------------------------------------- host --

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

constexpr int kMaxDevices = 64;
std::mutex g_mu;
bool g_attr[kMaxDevices][2];

}  // namespace mla
}  // namespace tsg

extern "C" tsgemm_status_t tsattn_mla_decode_ex(int64_t B, int64_t H, int64_t Skv, int32_t dim, int32_t pe_dim,
                                                 tsgemm_dtype_t dtype, float scale, const void* Q, const void* Q_pe,
                                                 const void* KV, const void* K_pe, void* O, int* status, void* stream,
                                                 int32_t debug_flags, int32_t timeout_ms, int32_t prefetch_blocks) {
    using namespace tsg::mla;
    if (B < 1 || H < 1 || Skv < 1 || !Q || !Q_pe || !KV || !K_pe || !O || timeout_ms < 0 || prefetch_blocks < 0 ||
        prefetch_blocks > 64)
        return TSGEMM_ERR_INVALID_ARG;
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return TSGEMM_ERR_INVALID_ARG;
    if (dtype != TSGEMM_F16 && dtype != TSGEMM_BF16) return TSGEMM_ERR_UNSUPPORTED;
    if (dim != kDL || pe_dim != kDR) return TSGEMM_ERR_UNSUPPORTED;
    const int64_t lim = (int64_t{1} << 31) - 1;
    const int64_t hblocks = (H + kH - 1) / kH;
    if (B > lim || H > lim || Skv > lim || 2 * B * hblocks > lim) return TSGEMM_ERR_UNSUPPORTED;
    const uintptr_t all = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(Q_pe) |
                          reinterpret_cast<uintptr_t>(KV) | reinterpret_cast<uintptr_t>(K_pe) |
                          reinterpret_cast<uintptr_t>(O);
    if (all & 15u) return TSGEMM_ERR_ALIGNMENT;
    const int64_t o_bytes = B * H * kDL * 2;
    const int64_t in_bytes[4] = {B * H * kDL * 2, B * H * kDR * 2, B * Skv * kDL * 2, B * Skv * kDR * 2};
    const void* ins[4] = {Q, Q_pe, KV, K_pe};
    for (int i = 0; i < 4; ++i) {
        const uintptr_t x = reinterpret_cast<uintptr_t>(O), y = reinterpret_cast<uintptr_t>(ins[i]);
        if (x < y + static_cast<uintptr_t>(in_bytes[i]) && y < x + static_cast<uintptr_t>(o_bytes))
            return TSGEMM_ERR_INVALID_ARG;
    }

    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return TSGEMM_ERR_UNSUPPORTED;
    if (dev < 0 || dev >= kMaxDevices) return TSGEMM_ERR_UNSUPPORTED;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return TSGEMM_ERR_CUDA;
    const bool f16 = dtype == TSGEMM_F16;
    const void* kern = f16 ? reinterpret_cast<const void*>(&mla_decode_sm103<true>)
                           : reinterpret_cast<const void*>(&mla_decode_sm103<false>);
    int* st = status;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_attr[dev][f16 ? 1 : 0]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kSmemBytes)) != cudaSuccess) {
                (void)cudaGetLastError();
                return TSGEMM_ERR_CUDA;
            }
            g_attr[dev][f16 ? 1 : 0] = true;
        }
    }
    if (!st) st = tsg::attn::library_status_word(dev);
    if (!st) return TSGEMM_ERR_CUDA;

    // [B][rows][cols] as 3-D tensors: a box of 64 columns never crosses into
    // another batch; rows past H (or Skv) read as zeros
    const CUtensorMapDataType dt = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    auto map3 = [&](CUtensorMap* m, const void* ptr, int64_t cols, int64_t rows, cuuint32_t box_rows) {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                                    static_cast<cuuint64_t>(B)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, static_cast<cuuint64_t>(rows * cols) * 2};
        const cuuint32_t box[3] = {64, box_rows, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        return enc(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    alignas(64) CUtensorMap tmQpe, tmKV, tmKpe;
    if (!map3(&tmQpe, Q_pe, kDR, H, kH) || !map3(&tmKV, KV, kDL, Skv, kN) ||
        !map3(&tmKpe, K_pe, kDR, Skv, kN))
        return TSGEMM_ERR_CUDA;

    MlaParams prm{};
    prm.Q = Q;
    prm.B = static_cast<int32_t>(B);
    prm.H = static_cast<int32_t>(H);
    prm.Skv = static_cast<int32_t>(Skv);
    prm.nblk = static_cast<int32_t>((Skv + kN - 1) / kN);
    prm.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
    prm.prefetch = prefetch_blocks;
    prm.debug_flags = debug_flags;
    prm.O = O;
    prm.status = st;
    prm.timeout_ns = static_cast<uint64_t>(timeout_ms ? timeout_ms : 1000) * 1000000ull;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(st, 0, sizeof(int), s) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>(2 * B * hblocks), 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = kSmemBytes;
    lc.stream = s;
    void* args[4] = {&tmQpe, &tmKV, &tmKpe, &prm};
    if (cudaLaunchKernelExC(&lc, kern, args) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }
    return TSGEMM_OK;
}

extern "C" tsgemm_status_t tsattn_mla_decode(int64_t B, int64_t H, int64_t Skv, int32_t dim, int32_t pe_dim,
                                              tsgemm_dtype_t dtype, float scale, const void* Q, const void* Q_pe,
                                              const void* KV, const void* K_pe, void* O, int* status, void* stream) {
    return tsattn_mla_decode_ex(B, H, Skv, dim, pe_dim, dtype, scale, Q, Q_pe, KV, K_pe, O, status, stream, 0, 0,
                                tsg::mla::kDefaultPrefetch);
}
