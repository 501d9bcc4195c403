// attention_sm103.cu -- the attention block (softmax(scale Q K^T) V) on
// tcgen05, and its C ABI (tsattn.h).
//
// It is the per-device block of the FlashMLA example of the TileScale
// README (section "Example of FlashMLA"), laid out for sm_103a:
//   * a CTA owns one tile of 128 query rows of one (batch, head); its Q is
//     loaded once by TMA into shared memory (128-byte swizzle);
//   * key and value blocks of 128 rows stream through rings of their own;
//   * S_j = Q K_j^T is computed by tcgen05.mma into one of two
//     tensor-memory score buffers (acc_s of the example), block j into
//     buffer j mod 2, so that S_{j+1} is ready while the softmax of block j
//     runs;
//   * as in the example, two warpgroups share the tile's score rows: each
//     owns one half of every block's 128 keys (a thread per query row and
//     half).  A warpgroup reads its half of the row of S_j, keeps its own
//     running maximum (scores_max) and row sum (logsum) in base-2 units,
//     and writes P_j = 2^(t - m) rounded to the 16-bit input format
//     (acc_s_cast) over the scores it has read, two weights per 32-bit
//     column;
//   * each half has an output accumulator of its own in tensor memory
//     (acc_o): O_h += P_j[:, half h] V_j[half h, :] by tcgen05.mma, P read
//     from tensor memory (A operand), V from shared memory.  Instead of the
//     example's all-gather of the block maximum, the halves keep separate
//     maxima and combine once, at the end: with m = max(m_0, m_1),
//     O = (2^(m_0 - m) O_0 + 2^(m_1 - m) O_1) / (2^(m_0 - m) l_0 + 2^(m_1 - m) l_1),
//     the same softmax, and no exchange between the warpgroups per block;
//   * each softmax warp writes its 32 rows x 64 columns of O, rounded to the
//     input format, into the key ring (free once every MMA is complete) and
//     sends them to global memory with one tiled TMA store.
// With two score buffers the tensor cores compute S_{j+2} and the P V of
// block j while the softmax of block j + 1 runs: a warpgroup's next block
// never waits for its own P V.
// The rescale is lazy: a half keeps its old maximum until the new one
// exceeds it by 2^8, so its output accumulator is read and rewritten only
// when a row's scores jump; the weights then stay below 2^8, well inside
// the 16-bit formats.
//
// Warp roles: warps 0-3 run the first key half's softmax, warps 4-7 the
// second's (warp w reads tensor-memory lanes 32 (w mod 4) .. +31); warp 8
// lane 0 loads Q and the key blocks, warp 9 lane 0 issues the MMAs, warp 10
// lane 0 loads the value blocks and warp 11 idles.  Every wait is bounded in
// time (WaitCtl); a CTA that gives up records a timeout, lets its copies and
// MMAs finish, frees tensor memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "attn_common.h"
#include "ptx.cuh"
#include "tsattn.h"

namespace tsg {
namespace attn {

constexpr int kBQ = 128;                // query rows per tile (TMEM lanes)
constexpr int kBKV = 128;               // keys per block
constexpr int kHalf = kBKV / 2;         // keys per softmax warpgroup
constexpr int kD = 128;                 // head dimension
constexpr int kThreads = 384;           // two softmax warpgroups; producers and MMA issuer
constexpr int kWarpK = 8, kWarpMma = 9, kWarpV = 10;
constexpr uint32_t kAtom = 128u * 128u; // 128 rows x 128 bytes: one swizzle atom column
constexpr uint32_t kTile = 2u * kAtom;  // 128 rows x 128 16-bit elements
constexpr int kKSlots = 2;              // key ring depth (one slot per score buffer)
constexpr int kVSlots = 2;              // value ring depth
constexpr uint32_t kQOff = 0;
constexpr uint32_t kKOff = kTile;
constexpr uint32_t kVOff = kKOff + kKSlots * kTile;
constexpr uint32_t kBarOff = kVOff + kVSlots * kTile;
// barriers: q_full, k_full[2], v_full[2], v_empty[2], s_full[2],
// p_full[2], o_final, drain
constexpr int kNumBars = 1 + kKSlots + 2 * kVSlots + 2 + 2 + 2;
constexpr uint32_t kMiscOff = kBarOff + 8u * kNumBars;
constexpr uint32_t kSmemBytes = 1024u + kMiscOff + 16u;
constexpr uint32_t kTmemCols = 512;     // S buffers at columns 0 and 128, O_0 at 256, O_1 at 384
constexpr uint32_t kOCol = 256;
constexpr float kRescaleLog2 = 8.0f;    // lazy-rescale threshold (base-2 units)
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct AttnParams {
    int32_t B, H, Sq, Sk;
    int32_t nq;           // CTAs (query tiles) per (batch, head)
    int32_t group;        // causal: (batch, head)s per chunk of the launch order
    int32_t causal;
    float scale_log2;     // scale * log2(e): scores to base-2 exponent units
    int32_t debug_flags;
    int* status;
    uint64_t timeout_ns;
};

// Key / value blocks the query tile starting at row q0 has to visit.
__device__ __forceinline__ int kv_blocks(const AttnParams& p, int q0) {
    if (q0 >= p.Sq) return 0;  // a tile wholly past the last query row
    const int nk = (p.Sk + kBKV - 1) / kBKV;
    if (!p.causal) return nk;
    const int last_q = min(q0 + kBQ - 1, p.Sq - 1);
    const int last_k = last_q + p.Sk - p.Sq;  // the last key that tile's last row sees
    if (last_k < 0) return 0;
    return min(nk, last_k / kBKV + 1);
}

// tcgen05 instruction descriptor, kind::f16, fp32 accumulator, M = N = 128;
// A K-major; B K-major (K^T: rows of K are the N index) or N-major (V).
__host__ __device__ constexpr uint32_t idesc(bool f16, bool b_nmajor) {
    return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) | ((b_nmajor ? 1u : 0u) << 16) |
           ((128u >> 3) << 17) | ((128u >> 4) << 24);
}

// Barrier addresses (8 bytes each, from `b`).
// Block j uses score buffer, key slot and value slot j mod 2.  Few
// barriers on purpose: each commit or wait the MMA issuer makes between
// its MMAs holds up the tensor cores for tens of cycles.
struct Bars {
    uint32_t b;
    __device__ uint32_t q_full() const { return b; }
    __device__ uint32_t k_full(int s) const { return b + 8u * (1 + s); }
    __device__ uint32_t v_full(int s) const { return b + 8u * (1 + kKSlots + s); }
    // P V of the block in value slot s complete (both halves): the slot is
    // free, and the output accumulators hold that block
    __device__ uint32_t v_empty(int s) const { return b + 8u * (1 + kKSlots + kVSlots + s); }
    static constexpr int kS = 1 + kKSlots + 2 * kVSlots;
    // S_j complete in buffer s = j mod 2; key slot s is free again
    __device__ uint32_t s_full(int s) const { return b + 8u * (kS + s); }
    // both halves' weights of the block in buffer s written
    __device__ uint32_t p_full(int s) const { return b + 8u * (kS + 2 + s); }
    // every MMA of the tile complete
    __device__ uint32_t o_final() const { return b + 8u * (kS + 4); }
    __device__ uint32_t drain() const { return b + 8u * (kS + 5); }
};

// A bounded wait that first tests the phase without blocking (the common
// case on the MMA issuer's path: the phase is already complete).
__device__ __forceinline__ bool wait_quick(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
    return mbar_test_wait(bar, parity) || wait_bounded(bar, parity, ctl);
}

// Named barrier of the two warps (one per half) that read the same 32
// tensor-memory lanes; ids 1-4 (0 is the CTA barrier).
__device__ __forceinline__ void pair_sync(int quarter) {
    asm volatile("barrier.sync %0, 64;" ::"r"(1 + quarter) : "memory");
}

// One softmax thread: query row r (TMEM lane quarter q, lane l) of the tile,
// keys [64 h, 64 h + 64) of every block.  `xch` is shared memory for the
// final exchange of (m, l) with the other half, `stage` 4 KiB of shared
// memory (1024-byte aligned) for the warp's part of the output tile; both
// are free once every MMA of the tile is complete.
template <bool kF16>
__device__ __forceinline__ void softmax_half(const AttnParams& p, const Bars& bar, uint32_t tmem, int h, int q0,
                                             int bh, int nkv, int quarter, int lane, float* xch, uint32_t stage,
                                             const CUtensorMap* tmO, const WaitCtl& ctl) {
    const int r = quarter * 32 + lane;  // row within the tile
    const int qrow = q0 + r;
    const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t hcol = static_cast<uint32_t>(kHalf * h);  // this half's columns of a score buffer
    const uint32_t ocol = kOCol + 128u * h;                   // this half's output accumulator
    const int kv_last = p.causal ? qrow + p.Sk - p.Sq : p.Sk - 1;  // last key this row sees
    const float c2 = p.scale_log2;
    // a bounded wait taken by lane 0 for the whole warp
    auto warp_wait = [&](uint32_t b, uint32_t parity) -> bool {
        int good = 1;
        if (lane == 0) good = wait_bounded(b, parity, ctl) ? 1 : 0;
        return __shfl_sync(0xffffffffu, good, 0) != 0;
    };
    float m_used = -INFINITY;  // base-2 maximum this half's weights are taken against
    float l = 0.0f;            // sum of this half's weights
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
        const int sb = j & 1;
        const uint32_t scol = 128u * static_cast<uint32_t>(sb) + hcol;
        // S_j complete.  S_j was issued after both halves' P V of block
        // j - 2, so that is complete too; P V of block j - 1 may still run.
        if (!warp_wait(bar.s_full(sb), static_cast<uint32_t>(j >> 1) & 1u)) {
            ok = false;
            break;
        }
        tc_fence_after();
        uint32_t s[kHalf];
        tmem_ld_32x32b_x32(trow + scol, *reinterpret_cast<uint32_t(*)[32]>(s));
        tmem_ld_32x32b_x32(trow + scol + 32u, *reinterpret_cast<uint32_t(*)[32]>(s + 32));
        tmem_ld_wait();
        // keys past Sk or past the causal limit weigh nothing
        const int k0 = j * kBKV + kHalf * h;
        if (!(k0 + kHalf - 1 <= kv_last && k0 + kHalf <= p.Sk)) {
#pragma unroll
            for (int c = 0; c < kHalf; ++c)
                if (k0 + c > kv_last || k0 + c >= p.Sk) s[c] = __float_as_uint(-INFINITY);
        }
        // maximum of the 64 scores: eight independent chains of
        // three-input maxima, then a tree
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(s[i]);
#pragma unroll
        for (int c = 8; c < 56; c += 16) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                asm("max.f32 %0, %1, %2, %3;"
                    : "=f"(mx[i])
                    : "f"(mx[i]), "f"(__uint_as_float(s[c + i])), "f"(__uint_as_float(s[c + 8 + i])));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], __uint_as_float(s[56 + i]));
        const float mb = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        const float m_new = fmaxf(m_used, mb * c2);  // (c2 > 0)
        const bool need = m_used == -INFINITY ? m_new > -INFINITY : m_new > m_used + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
            // every lane of the warp moves to its own new maximum
            const float alpha = m_used == -INFINITY ? 0.0f : ex2_approx(m_used - m_new);
            if (m_new > -INFINITY) m_used = m_new;
            l *= alpha;
            if (j >= 1) {
                // O_h holds P V of blocks 0 .. j-1 once P V of block j - 1
                // is complete (that of j - 2 is, see above, so the parity
                // names one completion of the slot's barrier)
                if (!warp_wait(bar.v_empty((j - 1) & 1), static_cast<uint32_t>((j - 1) >> 1) & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
                for (int c = 0; c < 128; c += 32) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(trow + ocol + c, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float2 v = mul2(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2);
                        o[i] = __float_as_uint(v.x);
                        o[i + 1] = __float_as_uint(v.y);
                    }
                    tmem_st_32x32b_x32(trow + ocol + c, o);
                }
                tmem_st_wait();
            }
        }
        // p = 2^(c2 s - m): one fused multiply-add per weight, two weights
        // per packed instruction; before any visible key, m = +inf makes
        // every weight 0.  The 64 weights go back over the first 32 of the
        // scores just read, two weights per column.
        const float mneg = m_used == -INFINITY ? -INFINITY : -m_used;
        const float2 c22 = make_float2(c2, c2), mn2 = make_float2(mneg, mneg);
        float2 rsum[4];  // eight independent partial sums, added in a fixed order
#pragma unroll
        for (int i = 0; i < 4; ++i) rsum[i] = make_float2(0.0f, 0.0f);
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float2 x = fma2(make_float2(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), c22, mn2);
            const float2 pw = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            rsum[i & 3] = add2(rsum[i & 3], pw);
            w[i] = kF16 ? pack_f16x2(pw.x, pw.y) : pack_bf16x2(pw.x, pw.y);
        }
        tmem_st_32x32b_x32(trow + scol, w);
        l += ((rsum[0].x + rsum[0].y) + (rsum[1].x + rsum[1].y)) + ((rsum[2].x + rsum[2].y) + (rsum[3].x + rsum[3].y));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.p_full(sb));
    }
    // ---------------------------------------------------- epilogue --
    // The two warps of this lane quarter swap (m, l) through shared memory
    // while P V of the last block still runs: `xch` lies in the Q tile,
    // which no MMA reads once the loop above has seen every block's scores.
    // Both warps pass the pair barrier exactly once, whatever their status,
    // so that neither waits for the other forever.
    xch[2 * (128 * h + r)] = m_used;
    xch[2 * (128 * h + r) + 1] = l;
    pair_sync(quarter);
    const float m_o = xch[2 * (128 * (h ^ 1) + r)], l_o = xch[2 * (128 * (h ^ 1) + r) + 1];
    const float m = fmaxf(m_used, m_o);
    const float f_me = m_used == -INFINITY ? 0.0f : ex2_approx(m_used - m);
    const float f_ot = m_o == -INFINITY ? 0.0f : ex2_approx(m_o - m);
    const float lsum = l * f_me + l_o * f_ot;
    const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
    // this warp writes output columns [64 h, 64 h + 64) of its row, from
    // both halves' accumulators
    const float f0 = (h == 0 ? f_me : f_ot) * inv, f1 = (h == 0 ? f_ot : f_me) * inv;
    const float2 f02 = make_float2(f0, f0), f12 = make_float2(f1, f1);
    // every MMA of the tile complete (P V of both halves, every block)
    if (ok && nkv > 0 && !warp_wait(bar.o_final(), 0u)) ok = false;
    if (!ok) return;
    tc_fence_after();
    // Both halves' 64 columns in one round trip to tensor memory: o[2 c + g]
    // holds O_g's columns 64 h + 32 c .. +31.
    uint32_t o[4][32];
    if (nkv > 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            tmem_ld_32x32b_x32(trow + kOCol + 128u * static_cast<uint32_t>(k & 1) + hcol + 32u * static_cast<uint32_t>(k >> 1), o[k]);
        tmem_ld_wait();
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int i = 0; i < 32; ++i) o[k][i] = 0u;
    }
    // The warp's 32 rows x 64 columns go to shared memory in the 128-byte
    // swizzled layout of the output map (row `lane` at 128 lane bytes, its
    // 16-byte chunk c at chunk c ^ (lane mod 8): a warp's stores then
    // touch every bank four times) and leave in one tiled store.
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float2 a = mul2(make_float2(__uint_as_float(o[2 * c][2 * i]), __uint_as_float(o[2 * c][2 * i + 1])), f02);
            const float2 v = fma2(make_float2(__uint_as_float(o[2 * c + 1][2 * i]), __uint_as_float(o[2 * c + 1][2 * i + 1])), f12, a);
            w[i] = kF16 ? pack_f16x2(v.x, v.y) : pack_bf16x2(v.x, v.y);
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint32_t chunk = static_cast<uint32_t>(4 * c + v);
            st_shared_v4(stage + 128u * static_cast<uint32_t>(lane) + ((chunk ^ (static_cast<uint32_t>(lane) & 7u)) << 4),
                         w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
    }
    // rows past Sq are clipped by the store; a box wholly past it is skipped
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0 && q0 + 32 * quarter < p.Sq) {
        tma_store_3d(tmO, stage, kHalf * h, q0 + 32 * quarter, bh);
        bulk_commit_group();
        bulk_wait_group_read<0>();  // shared memory stays valid until the store has read it
    }
}

template <bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_sm103(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   const AttnParams p) {
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
    // Launch order.  Non-causal: (batch, head) by (batch, head), all CTAs
    // of one alike.  Causal: chunks of p.group (batch, head)s whose K and V
    // fit in L2 together; within a chunk the longest query tiles first, one
    // per (batch, head), so the launch ends on the shortest CTAs.
    int bh, qb;
    if (p.causal) {
        const int span = p.group * p.nq;
        const int chunk = static_cast<int>(blockIdx.x) / span;
        const int gc = min(p.group, p.B * p.H - chunk * p.group);  // (batch, head)s in this chunk
        const int idx = static_cast<int>(blockIdx.x) - chunk * span;
        qb = p.nq - 1 - idx / gc;
        bh = chunk * p.group + idx % gc;
    } else {
        bh = blockIdx.x / p.nq;
        qb = p.nq - 1 - static_cast<int>(blockIdx.x % p.nq);
    }
    const int q0 = qb * kBQ;
    const int nkv = kv_blocks(p, q0);  // key / value blocks the tile visits

    if (threadIdx.x == 0) {
        mbar_init(bar.q_full(), 1);
        for (int s = 0; s < kKSlots; ++s) mbar_init(bar.k_full(s), 1);
        for (int s = 0; s < kVSlots; ++s) {
            mbar_init(bar.v_full(s), 1);
            mbar_init(bar.v_empty(s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar.s_full(s), 1);
            mbar_init(bar.p_full(s), 8);  // every softmax warp of both halves
        }
        mbar_init(bar.o_final(), 1);
        mbar_init(bar.drain(), 1);
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmO);
        // The first copies leave before tensor memory is allocated and the
        // CTA synchronises: Q and the first key and value blocks (the
        // producers take over from the second block).
        if (nkv > 0) {
            mbar_arrive_expect_tx(bar.q_full(), kTile);
            tma_load_3d(base + kQOff, &tmQ, bar.q_full(), 0, q0, bh);
            tma_load_3d(base + kQOff + kAtom, &tmQ, bar.q_full(), 64, q0, bh);
            // tests only: the first CTA leaves its first key block unloaded
            if (!((p.debug_flags & 1) && blockIdx.x == 0)) {
                mbar_arrive_expect_tx(bar.k_full(0), kTile);
                tma_load_3d(base + kKOff, &tmK, bar.k_full(0), 0, 0, bh);
                tma_load_3d(base + kKOff + kAtom, &tmK, bar.k_full(0), 64, 0, bh);
            }
            mbar_arrive_expect_tx(bar.v_full(0), kTile);
            tma_load_3d(base + kVOff, &tmV, bar.v_full(0), 0, 0, bh);
            tma_load_3d(base + kVOff + kAtom, &tmV, bar.v_full(0), 64, 0, bh);
        }
    }
    if (warp == kWarpMma) tmem_alloc<1>(smem_u32(tmem_holder), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
    if (warp < kWarpK) {
        // ---------------------------------------- softmax and epilogue --
        // the output tile is staged in the key ring: box half h (16 KiB),
        // rows of lane quarter q (4 KiB)
        softmax_half<kF16>(p, bar, tmem, warp >> 2, q0, bh, nkv, warp & 3, lane,
                           reinterpret_cast<float*>(base_ptr + kQOff),
                           base + kKOff + 16384u * static_cast<uint32_t>(warp >> 2) + 4096u * static_cast<uint32_t>(warp & 3),
                           &tmO, ctl);
    } else if (warp == kWarpK || warp == kWarpV) {
        // --------------------------------- TMA producers: Q and K / V --
        const bool is_k = warp == kWarpK;
        if (lane == 0 && nkv > 0) {
            // block 0 (and Q) left with the CTA's first thread; its copies
            // count as this thread's for the wait before exit
            const bool skipped0 = is_k && (p.debug_flags & 1) && blockIdx.x == 0;
            uint32_t outstanding = skipped0 ? 0u : 1u, out_par = 0;  // loads per slot
            const int slots = is_k ? kKSlots : kVSlots;
            const CUtensorMap* map = is_k ? &tmK : &tmV;
            for (int j = 1; j < nkv; ++j) {
                const int st = j % slots;
                const uint32_t ph = static_cast<uint32_t>(j / slots) & 1u;
                const uint32_t dst = base + (is_k ? kKOff : kVOff) + st * kTile;
                const uint32_t full = is_k ? bar.k_full(st) : bar.v_full(st);
                // a key slot is free once S of its previous block is complete
                if (!wait_bounded(is_k ? bar.s_full(st) : bar.v_empty(st), ph ^ 1u, ctl)) break;
                mbar_arrive_expect_tx(full, kTile);
                tma_load_3d(dst, map, full, 0, j * kBKV, bh);
                tma_load_3d(dst + kAtom, map, full, 64, j * kBKV, bh);
                outstanding |= 1u << st;
                out_par = (out_par & ~(1u << st)) | (ph << st);
            }
            // every copy this thread started lands before the CTA exits
            if (is_k) wait_bounded(bar.q_full(), 0u, ctl, false);
            for (int s = 0; s < slots; ++s)
                if (outstanding & (1u << s))
                    wait_bounded(is_k ? bar.k_full(s) : bar.v_full(s), (out_par >> s) & 1u, ctl, false);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0 && nkv > 0) {
            constexpr uint32_t kIdS = idesc(kF16, false), kIdPV = idesc(kF16, true);
            static_assert(kKSlots == 2 && kVSlots == 2, "block j uses score buffer, key slot and value slot j mod 2");
            using C0 = std::integral_constant<int, 0>;
            using C1 = std::integral_constant<int, 1>;
            // Every shared-memory descriptor the loop uses is formed here,
            // once, and every slot and buffer index below is a constant: an
            // MMA whose descriptors are computed just before it issues only
            // about every 120 cycles, against 64 for the tensor cores to run
            // one of these 128 x 128 x 16 steps.
            // S = Q K^T: both operands K-major, two 64-wide swizzle columns
            // of D, the k-th 16-deep step 32 bytes along a row.  P V: V (128
            // keys x 128 columns, columns contiguous) is the N-major B
            // operand: 64-column boxes 16 KiB apart, 8-key groups 1 KiB
            // apart, the k-th 16-key step 2 KiB on.
            uint64_t qd[8], kd[kKSlots][8], vd[kVSlots][8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t c = (k >> 2) * kAtom + (k & 3) * 32u;
                qd[k] = smem_desc_sw128(base + kQOff + c, 16u, 1024u);
#pragma unroll
                for (int s = 0; s < kKSlots; ++s) kd[s][k] = smem_desc_sw128(base + kKOff + s * kTile + c, 16u, 1024u);
#pragma unroll
                for (int s = 0; s < kVSlots; ++s)
                    vd[s][k] = smem_desc_sw128(base + kVOff + s * kTile + k * 2048u, kAtom, 1024u);
            }
            bool ok = wait_bounded(bar.q_full(), 0u, ctl);
            // S_j = Q K_j^T into score buffer b = j mod 2, from key slot b.
            // The buffer held the weights of block j - 2, which both halves'
            // P V (issued before) read.
            auto issue_s = [&](auto bc, int j) -> bool {
                constexpr int b = decltype(bc)::value;
                if (!wait_quick(bar.k_full(b), static_cast<uint32_t>(j >> 1) & 1u, ctl)) return false;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) umma_f16<1>(tmem + 128u * b, qd[k], kd[b][k], kIdS, k > 0 ? 1u : 0u);
                umma_commit(bar.s_full(b));  // (K_j read, too)
                return true;
            };
            // O_h += P_j[:, half h] V_j[half h, :]: half h's 64 weights (two
            // per 32-bit column) are the tensor-memory A operand at column
            // 64 h of score buffer b; half h takes V's 16-key steps 4 h ..
            // 4 h + 3.  Block j (b = j mod 2): P V of both halves once both
            // halves' weights are written, then S(j + 2) into the buffer
            // they have read.
            auto block = [&](auto bc, int j) -> bool {
                constexpr int b = decltype(bc)::value;
                if (!wait_quick(bar.v_full(b), static_cast<uint32_t>(j >> 1) & 1u, ctl) ||
                    !wait_quick(bar.p_full(b), static_cast<uint32_t>(j >> 1) & 1u, ctl))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_f16_ta(tmem + kOCol + 128u * h, tmem + 128u * b + 64u * h + 8u * k, vd[b][4 * h + k],
                                    kIdPV, (j > 0 || k > 0) ? 1u : 0u);
                umma_commit(bar.v_empty(b));  // V_j read; O holds block j
                return j + 2 >= nkv || issue_s(bc, j + 2);
            };
            ok = ok && issue_s(C0{}, 0) && (nkv < 2 || issue_s(C1{}, 1));
            for (int j = 0; ok && j < nkv; j += 2) ok = block(C0{}, j) && (j + 1 >= nkv || block(C1{}, j + 1));
            if (ok) umma_commit(bar.o_final());
            // every MMA issued above completes before tensor memory is freed
            umma_commit(bar.drain());
            wait_bounded(bar.drain(), 0u, ctl, false);
        }
        __syncwarp();
    }

    // ------------------------------------------------------------ exit --
    tc_fence_before();
    cta_barrier_any();
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

// The library's status word (one per device that loads the library), used
// when the caller passes no status pointer; the attention block and the MLA
// decode kernel share it.
__device__ int g_attn_status;

struct DeviceState {
    bool ready = false;
    int* status = nullptr;
    bool attr[2] = {false, false};
};
constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

// Device address of the status word on device `dev` (current), looked up
// once per device; null on failure.  Call with g_mu held.
int* status_word_locked(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    DeviceState& ds = g_dev[dev];
    if (!ds.ready) {
        void* sym = nullptr;
        if (cudaGetSymbolAddress(&sym, g_attn_status) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        ds.status = static_cast<int*>(sym);
        ds.ready = true;
    }
    return ds.status;
}

int* library_status_word(int dev) {
    std::lock_guard<std::mutex> lock(g_mu);
    return status_word_locked(dev);
}

}  // namespace attn
}  // namespace tsg

extern "C" {

tsgemm_status_t tsattn_forward_ex(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int32_t D, tsgemm_dtype_t dtype,
                                  float scale, int32_t causal, const void* Q, const void* K, const void* V, void* O,
                                  int* status, void* stream, int32_t debug_flags, int32_t timeout_ms) {
    using namespace tsg::attn;
    if (B < 1 || H < 1 || Sq < 1 || Sk < 1 || !Q || !K || !V || !O || timeout_ms < 0) return TSGEMM_ERR_INVALID_ARG;
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return TSGEMM_ERR_INVALID_ARG;
    if (dtype != TSGEMM_F16 && dtype != TSGEMM_BF16) return TSGEMM_ERR_UNSUPPORTED;
    if (D != kD) return TSGEMM_ERR_UNSUPPORTED;
    const int64_t lim = (int64_t{1} << 31) - 1;
    if (B * H > lim || Sq > lim || Sk > lim || B * H * ((Sq + kBQ - 1) / kBQ) > lim) return TSGEMM_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V) |
         reinterpret_cast<uintptr_t>(O)) &
        15u)
        return TSGEMM_ERR_ALIGNMENT;
    const int64_t qbytes = B * H * Sq * D * 2, kvbytes = B * H * Sk * D * 2;
    auto overlaps = [](const void* a, int64_t na, const void* b, int64_t nb) {
        const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
        return x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
    };
    if (overlaps(O, qbytes, Q, qbytes) || overlaps(O, qbytes, K, kvbytes) || overlaps(O, qbytes, V, kvbytes))
        return TSGEMM_ERR_INVALID_ARG;

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
    const void* kern = f16 ? reinterpret_cast<const void*>(&attn_fwd_sm103<true>)
                           : reinterpret_cast<const void*>(&attn_fwd_sm103<false>);
    {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceState& ds = g_dev[dev];
        if (!status_word_locked(dev)) return TSGEMM_ERR_CUDA;
        if (!ds.attr[f16 ? 1 : 0]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kSmemBytes)) != cudaSuccess) {
                (void)cudaGetLastError();
                return TSGEMM_ERR_CUDA;
            }
            ds.attr[f16 ? 1 : 0] = true;
        }
    }
    int* st = status ? status : g_dev[dev].status;

    // [B*H][S][D] as a 3-D tensor: a 64 (D) x 128 (rows) box never crosses
    // into another (batch, head); rows past S read as zeros.  O is stored
    // in 64 x 32 boxes (one per softmax warp), rows past Sq not written.
    const CUtensorMapDataType dt = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    auto map3 = [&](CUtensorMap* m, const void* ptr, int64_t S, cuuint32_t box_rows) {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                                    static_cast<cuuint64_t>(B * H)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(S * D) * 2};
        const cuuint32_t box[3] = {64, box_rows, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        return enc(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    alignas(64) CUtensorMap tmQ, tmK, tmV, tmO;
    if (!map3(&tmQ, Q, Sq, 128) || !map3(&tmK, K, Sk, 128) || !map3(&tmV, V, Sk, 128) || !map3(&tmO, O, Sq, 32))
        return TSGEMM_ERR_CUDA;

    AttnParams prm{};
    prm.B = static_cast<int32_t>(B);
    prm.H = static_cast<int32_t>(H);
    prm.Sq = static_cast<int32_t>(Sq);
    prm.Sk = static_cast<int32_t>(Sk);
    prm.nq = static_cast<int32_t>((Sq + kBQ - 1) / kBQ);
    // about 8 MiB of K and V per chunk of the causal launch order (four
    // heads at S = 4096, D = 128): the CTAs that run together then share
    // few heads' key blocks in L2.  Same box, alternating builds, causal
    // B 4 H 32 S 4096: 462.5 us against 464.5-466.6 for 16 MiB, 466.6 for
    // 4 MiB, 469.1 for 64 MiB and 506 for 128 MiB
    const int64_t kv_head_bytes = 2 * Sk * static_cast<int64_t>(D) * 2;
    prm.group = static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(B * H, (8ll << 20) / kv_head_bytes)));
    prm.causal = causal ? 1 : 0;
    prm.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
    prm.debug_flags = debug_flags;
    prm.status = st;
    prm.timeout_ns = static_cast<uint64_t>(timeout_ms ? timeout_ms : 1000) * 1000000ull;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(st, 0, sizeof(int), s) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>(B * H * prm.nq), 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = kSmemBytes;
    lc.stream = s;
    void* args[5] = {&tmQ, &tmK, &tmV, &tmO, &prm};
    if (cudaLaunchKernelExC(&lc, kern, args) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }
    return TSGEMM_OK;
}

tsgemm_status_t tsattn_forward(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int32_t D, tsgemm_dtype_t dtype,
                               float scale, int32_t causal, const void* Q, const void* K, const void* V, void* O,
                               int* status, void* stream) {
    return tsattn_forward_ex(B, H, Sq, Sk, D, dtype, scale, causal, Q, K, V, O, status, stream, 0, 0);
}

tsgemm_status_t tsattn_status(void) {
    using namespace tsg::attn;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }
    int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_attn_status, sizeof(int)) != cudaSuccess) {
        (void)cudaGetLastError();
        return TSGEMM_ERR_CUDA;
    }
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(int)) != cudaSuccess) {
            (void)cudaGetLastError();
            return TSGEMM_ERR_CUDA;
        }
    }
    return static_cast<tsgemm_status_t>(word);
}

}  // extern "C"
