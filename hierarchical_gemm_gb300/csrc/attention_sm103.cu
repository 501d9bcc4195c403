// attention_sm103.cu -- the attention block (softmax(scale Q K^T) V) on
// tcgen05, and its C ABI (tsattn.h).
//
// It is the per-device block of the FlashMLA example of the TileScale
// README (section "Example of FlashMLA"), laid out for sm_103a:
//   * a CTA owns two tiles of 128 query rows (A and B) of one (batch, head);
//     their Q is loaded once by TMA into shared memory (128-byte swizzle);
//   * key and value blocks of 128 rows stream through rings of their own: a
//     K slot is free once both tiles' S = Q K^T have read it, a V slot once
//     both tiles' O += P V have;
//   * per tile, S_j = Q K_j^T is computed by tcgen05.mma into the tile's
//     tensor-memory score buffer (acc_s of the example); one warpgroup per
//     tile, a thread per query row, reads its row of S_j, keeps the running
//     maximum (scores_max) and row sum (logsum) in base-2 units, writes
//     P_j = 2^(t - m) rounded to the 16-bit input format (acc_s_cast) back
//     into the score buffer, two weights per 32-bit column, and, when its
//     maximum has grown, rescales its row of the output accumulator
//     (scores_scale);
//   * O += P_j V_j is computed by tcgen05.mma with P read from tensor memory
//     (A operand) and V from shared memory into the tile's tensor-memory
//     accumulator (acc_o); at the end each thread divides its row by the row
//     sum and stores it.
// The two tiles ping-pong: while one tile's warpgroup computes its softmax,
// the tensor cores run the other tile's P V and next S, so neither the
// tensor cores nor the exponential units wait for each other.  (The
// example splits one tile's acc_s between two warpgroups and all-gathers
// it; two tiles need no exchange between the warpgroups at all.)
// The rescale is lazy: a row keeps its old maximum until the new one exceeds
// it by 2^8, so the output accumulator is read and rewritten only when a
// row's scores jump; the weights then stay below 2^8, well inside the
// 16-bit formats, and the final division uses the same maximum as every
// weight, so the result is the same softmax.
//
// Warp roles, in three warpgroups: warps 0-3 run tile A's softmax and
// epilogue, warps 4-7 tile B's (warp w reads tensor-memory lanes
// 32 (w mod 4) .. +31); in the third, warp 8 lane 0 loads Q and the key
// blocks, warp 9 lane 0 issues the MMAs, warp 10 lane 0 loads the value
// blocks and warp 11 idles.  The third warpgroup gives most of its
// registers to the other two (setmaxnreg): a softmax thread holds its whole
// row of 128 scores.  Every wait is bounded in time (WaitCtl); a CTA that
// gives up records a timeout, lets its copies and MMAs finish, frees tensor
// memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "attn_common.h"
#include "ptx.cuh"
#include "tsattn.h"

namespace tsg {
namespace attn {

constexpr int kBQ = 128;                // query rows per tile (TMEM lanes)
constexpr int kTiles = 2;               // query tiles per CTA
constexpr int kBKV = 128;               // keys per block
constexpr int kD = 128;                 // head dimension
constexpr int kThreads = 384;           // two softmax warpgroups; producers and MMA issuer
constexpr int kWarpK = 8, kWarpMma = 9, kWarpV = 10;
// registers per thread after the split: 256 softmax threads at kRegsSoftmax
// and 128 others at kRegsOther may not exceed what the CTA was launched with
// (384 x the kernel's register count; the host checks this before a launch)
constexpr int kRegsSoftmax = 208, kRegsOther = 64;
constexpr int kRegPool = 256 * kRegsSoftmax + 128 * kRegsOther;
constexpr uint32_t kAtom = 128u * 128u; // 128 rows x 128 bytes: one swizzle atom column
constexpr uint32_t kTile = 2u * kAtom;  // 128 rows x 128 16-bit elements
constexpr int kKSlots = 3;              // key ring depth
constexpr int kVSlots = 2;              // value ring depth
constexpr uint32_t kQOff = 0;           // Q of tile A, then tile B
constexpr uint32_t kKOff = kTiles * kTile;
constexpr uint32_t kVOff = kKOff + kKSlots * kTile;
constexpr uint32_t kBarOff = kVOff + kVSlots * kTile;
// barriers: q_full, k_full[3], k_empty[3], v_full[2], v_empty[2], and per
// tile s_full, p_full, p_free; drain
constexpr int kNumBars = 1 + 2 * kKSlots + 2 * kVSlots + 3 * kTiles + 1;
constexpr uint32_t kMiscOff = kBarOff + 8u * kNumBars;
constexpr uint32_t kSmemBytes = 1024u + kMiscOff + 16u;
constexpr uint32_t kTmemCols = 512;     // S of tile t at columns 128 t, O of tile t at 256 + 128 t
constexpr uint32_t kOCol = 256;
constexpr float kRescaleLog2 = 8.0f;    // lazy-rescale threshold (base-2 units)
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct AttnParams {
    int32_t B, H, Sq, Sk;
    int32_t nq;           // CTAs (pairs of query tiles) per (batch, head)
    int32_t group;        // causal: (batch, head)s per chunk of the launch order
    int32_t causal;
    float scale_log2;     // scale * log2(e): scores to base-2 exponent units
    int32_t debug_flags;
    void* O;
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
struct Bars {
    uint32_t b;
    __device__ uint32_t q_full() const { return b; }
    __device__ uint32_t k_full(int s) const { return b + 8u * (1 + s); }
    __device__ uint32_t k_empty(int s) const { return b + 8u * (1 + kKSlots + s); }
    __device__ uint32_t v_full(int s) const { return b + 8u * (1 + 2 * kKSlots + s); }
    __device__ uint32_t v_empty(int s) const { return b + 8u * (1 + 2 * kKSlots + kVSlots + s); }
    __device__ uint32_t s_full(int t) const { return b + 8u * (1 + 2 * kKSlots + 2 * kVSlots + t); }
    __device__ uint32_t p_full(int t) const { return b + 8u * (1 + 2 * kKSlots + 2 * kVSlots + kTiles + t); }
    // P V of tile t complete
    __device__ uint32_t p_free(int t) const { return b + 8u * (1 + 2 * kKSlots + 2 * kVSlots + 2 * kTiles + t); }
    __device__ uint32_t drain() const { return b + 8u * (1 + 2 * kKSlots + 2 * kVSlots + 3 * kTiles); }
};

// One softmax thread: query row r of tile t (TMEM lane quarter q, lane l).
template <bool kF16>
__device__ __forceinline__ void softmax_row(const AttnParams& p, const Bars& bar, uint32_t tmem, int t, int q0,
                                            int bh, int nkv, int quarter, int lane, const WaitCtl& ctl) {
    const int r = quarter * 32 + lane;  // row within the tile
    const int qrow = q0 + r;
    const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t scol = 128u * t, ocol = kOCol + 128u * t;
    const int kv_last = p.causal ? qrow + p.Sk - p.Sq : p.Sk - 1;  // last key this row sees
    const float c2 = p.scale_log2;
    // a bounded wait taken by lane 0 for the whole warp
    auto warp_wait = [&](uint32_t b, uint32_t parity) -> bool {
        int good = 1;
        if (lane == 0) good = wait_bounded(b, parity, ctl) ? 1 : 0;
        return __shfl_sync(0xffffffffu, good, 0) != 0;
    };
    float m_used = -INFINITY;  // base-2 maximum the weights are taken against
    float l = 0.0f;            // sum of this row's weights
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
        // S_j complete: every MMA issued before it is complete too (a
        // commit covers all of them), in particular P V of block j - 1
        if (!warp_wait(bar.s_full(t), static_cast<uint32_t>(j) & 1u)) {
            ok = false;
            break;
        }
        tc_fence_after();
        uint32_t s[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t (&part)[32] = *reinterpret_cast<uint32_t(*)[32]>(s + 32 * c);
            tmem_ld_32x32b_x32(trow + scol + 32u * c, part);
        }
        tmem_ld_wait();
        // keys past Sk or past the causal limit weigh nothing
        const int k0 = j * kBKV;
        if (!(k0 + kBKV - 1 <= kv_last && k0 + kBKV <= p.Sk)) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
                if (k0 + c > kv_last || k0 + c >= p.Sk) s[c] = __float_as_uint(-INFINITY);
        }
        // row maximum: eight independent chains of three-input maxima, then
        // a tree
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(s[i]);
#pragma unroll
        for (int c = 8; c < 128; c += 16) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                asm("max.f32 %0, %1, %2, %3;"
                    : "=f"(mx[i])
                    : "f"(mx[i]), "f"(__uint_as_float(s[c + i])), "f"(__uint_as_float(s[c + 8 + i])));
        }
        const float mb = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        const float m_new = fmaxf(m_used, mb * c2);  // (c2 > 0)
        const bool need = m_used == -INFINITY ? m_new > -INFINITY : m_new > m_used + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
            // every lane of the warp moves to its own new maximum; O holds
            // P_0 V_0 + ... + P_{j-1} V_{j-1}, complete (see above)
            const float alpha = m_used == -INFINITY ? 0.0f : ex2_approx(m_used - m_new);
            if (m_new > -INFINITY) m_used = m_new;
            l *= alpha;
            if (j >= 1) {
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
        // every weight 0.  P_j goes back into the first 64 columns of the
        // score buffer, two weights per column, 32 columns at a time.
        const float mneg = m_used == -INFINITY ? -INFINITY : -m_used;
        const float2 c22 = make_float2(c2, c2), mn2 = make_float2(mneg, mneg);
        float2 rsum[4];  // eight independent partial sums, added in a fixed order
#pragma unroll
        for (int i = 0; i < 4; ++i) rsum[i] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int c = 64 * h + 2 * i;
                const float2 x = fma2(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), c22, mn2);
                const float2 pw = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                rsum[i & 3] = add2(rsum[i & 3], pw);
                w[i] = kF16 ? pack_f16x2(pw.x, pw.y) : pack_bf16x2(pw.x, pw.y);
            }
            tmem_st_32x32b_x32(trow + scol + 32u * h, w);
        }
        l += ((rsum[0].x + rsum[0].y) + (rsum[1].x + rsum[1].y)) + ((rsum[2].x + rsum[2].y) + (rsum[3].x + rsum[3].y));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar.p_full(t));
    }
    // ---------------------------------------------------- epilogue --
    // (S of the last block complete implies P V of the block before it is:
    // the wait for the last P V below cannot be confused with an earlier one)
    if (ok && nkv > 0 && !warp_wait(bar.p_free(t), static_cast<uint32_t>(nkv - 1) & 1u)) ok = false;
    if (!ok) return;
    tc_fence_after();
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    uint16_t* orow = static_cast<uint16_t*>(p.O) + (static_cast<int64_t>(bh) * p.Sq + qrow) * kD;
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
        uint32_t o[32];
        if (nkv > 0) {
            tmem_ld_32x32b_x32(trow + ocol + c, o);
            tmem_ld_wait();
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        uint32_t w[16];
        const float2 inv2 = make_float2(inv, inv);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float2 v = mul2(make_float2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), inv2);
            w[i] = kF16 ? pack_f16x2(v.x, v.y) : pack_bf16x2(v.x, v.y);
        }
        if (qrow < p.Sq) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
                st_global_v4(orow + c + 8 * v, w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
    }
}

template <bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_sm103(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
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
    // fit in L2 together; within a chunk the longest query pairs first, one
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
    const int q0 = qb * kTiles * kBQ;                                // first query row of tile A
    const int n_a = kv_blocks(p, q0), n_b = kv_blocks(p, q0 + kBQ);  // blocks tiles A and B visit
    const int nkv = max(n_a, n_b);                                   // blocks the CTA loads
    auto n_t = [&](int t) { return t == 0 ? n_a : n_b; };

    if (threadIdx.x == 0) {
        mbar_init(bar.q_full(), 1);
        for (int s = 0; s < kKSlots; ++s) {
            mbar_init(bar.k_full(s), 1);
            mbar_init(bar.k_empty(s), 1);
        }
        for (int s = 0; s < kVSlots; ++s) {
            mbar_init(bar.v_full(s), 1);
            mbar_init(bar.v_empty(s), 1);
        }
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(bar.s_full(t), 1);
            mbar_init(bar.p_full(t), 4);  // every softmax warp of the tile
            mbar_init(bar.p_free(t), 1);
        }
        mbar_init(bar.drain(), 1);
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    if (warp == kWarpMma) tmem_alloc<1>(smem_u32(tmem_holder), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
    // (each role's code sits in the branch of its register budget)
    if (warp < kWarpK) {
        // ---------------------------------------- softmax and epilogue --
        setmaxnreg_inc<kRegsSoftmax>();
        const int t = warp >> 2;
        softmax_row<kF16>(p, bar, tmem, t, q0 + t * kBQ, bh, n_t(t), warp & 3, lane, ctl);
    } else {
    setmaxnreg_dec<kRegsOther>();
    if (warp == kWarpK || warp == kWarpV) {
        // --------------------------------- TMA producers: Q and K / V --
        const bool is_k = warp == kWarpK;
        if (lane == 0 && nkv > 0) {
            uint32_t outstanding = 0, out_par = 0;  // loads per slot
            if (is_k) {
                mbar_arrive_expect_tx(bar.q_full(), kTiles * kTile);
                for (int t = 0; t < kTiles; ++t) {
                    const uint32_t qs = base + kQOff + t * kTile;
                    tma_load_3d(qs, &tmQ, bar.q_full(), 0, q0 + t * kBQ, bh);
                    tma_load_3d(qs + kAtom, &tmQ, bar.q_full(), 64, q0 + t * kBQ, bh);
                }
            }
            const int slots = is_k ? kKSlots : kVSlots;
            const CUtensorMap* map = is_k ? &tmK : &tmV;
            for (int j = 0; j < nkv; ++j) {
                const int st = j % slots;
                const uint32_t ph = static_cast<uint32_t>(j / slots) & 1u;
                const uint32_t dst = base + (is_k ? kKOff : kVOff) + st * kTile;
                const uint32_t full = is_k ? bar.k_full(st) : bar.v_full(st);
                if (!wait_bounded(is_k ? bar.k_empty(st) : bar.v_empty(st), ph ^ 1u, ctl)) break;
                // tests only: the first CTA leaves its first key block unloaded
                if (is_k && (p.debug_flags & 1) && blockIdx.x == 0 && j == 0) continue;
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
            bool ok = wait_bounded(bar.q_full(), 0u, ctl);
            // S_t(j) = Q_t K_j^T into tile t's score buffer: both operands
            // K-major, two 64-wide swizzle columns of D, the k-th 16-deep
            // step 32 bytes along a row.  The buffer held P_t(j-1), which
            // P V of tile t (issued before) has read.
            auto issue_s = [&](int t, int j) -> bool {
                const int st = j % kKSlots;
                if (!wait_bounded(bar.k_full(st), static_cast<uint32_t>(j / kKSlots) & 1u, ctl)) return false;
                tc_fence_after();
                const uint32_t qs = base + kQOff + t * kTile, ks = base + kKOff + st * kTile;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t ad = smem_desc_sw128(qs + (k >> 2) * kAtom + (k & 3) * 32u, 16u, 1024u);
                    const uint64_t bd = smem_desc_sw128(ks + (k >> 2) * kAtom + (k & 3) * 32u, 16u, 1024u);
                    umma_f16<1>(tmem + 128u * t, ad, bd, kIdS, k > 0 ? 1u : 0u);
                }
                umma_commit(bar.s_full(t));
                return true;
            };
            // O_t += P_t(j) V_j: P (128 rows x 128 keys, two per 32-bit
            // column) is the tensor-memory A operand in the first 64 columns
            // of tile t's score buffer; V (128 keys x 128 columns, columns
            // contiguous) the N-major B operand: 64-column boxes 16 KiB
            // apart, 8-key groups 1 KiB apart, the k-th 16-key step 2 KiB on.
            auto issue_pv = [&](int t, int j) -> bool {
                const int vs_slot = j % kVSlots;
                if (!wait_bounded(bar.v_full(vs_slot), static_cast<uint32_t>(j / kVSlots) & 1u, ctl) ||
                    !wait_bounded(bar.p_full(t), static_cast<uint32_t>(j) & 1u, ctl))
                    return false;
                tc_fence_after();
                const uint32_t vs = base + kVOff + vs_slot * kTile;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t bd = smem_desc_sw128(vs + k * 2048u, kAtom, 1024u);
                    umma_f16_ta(tmem + kOCol + 128u * t, tmem + 128u * t + 8u * k, bd, kIdPV,
                                (j > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit(bar.p_free(t));
                return true;
            };
            // order: S_A(0), S_B(0); then per block j: P V_A(j), S_A(j+1),
            // P V_B(j), S_B(j+1) -- while one tile's softmax runs, the
            // tensor cores work on the other tile
            for (int t = 0; ok && t < kTiles; ++t)
                if (n_t(t) > 0) ok = issue_s(t, 0);
            if (ok) umma_commit(bar.k_empty(0));
            for (int j = 0; ok && j < nkv; ++j) {
                for (int t = 0; ok && t < kTiles; ++t) {
                    if (j >= n_t(t)) continue;
                    ok = issue_pv(t, j);
                    if (ok && j + 1 < n_t(t)) ok = issue_s(t, j + 1);
                }
                if (!ok) break;
                umma_commit(bar.v_empty(j % kVSlots));                     // V_j read by both tiles
                if (j + 1 < nkv) umma_commit(bar.k_empty((j + 1) % kKSlots));  // K_{j+1} too
            }
            // every MMA issued above completes before tensor memory is freed
            umma_commit(bar.drain());
            wait_bounded(bar.drain(), 0u, ctl, false);
        }
        __syncwarp();
    }
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
            // the warpgroups' register split must fit in what the CTA is
            // launched with, or the softmax warps would wait for registers
            // forever
            cudaFuncAttributes fa{};
            if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) {
                (void)cudaGetLastError();
                return TSGEMM_ERR_CUDA;
            }
            if (fa.numRegs * kThreads < kRegPool) return TSGEMM_ERR_UNSUPPORTED;
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
    // into another (batch, head); rows past S read as zeros
    const CUtensorMapDataType dt = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    auto map3 = [&](CUtensorMap* m, const void* ptr, int64_t S) {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                                    static_cast<cuuint64_t>(B * H)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(S * D) * 2};
        const cuuint32_t box[3] = {64, 128, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        return enc(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    alignas(64) CUtensorMap tmQ, tmK, tmV;
    if (!map3(&tmQ, Q, Sq) || !map3(&tmK, K, Sk) || !map3(&tmV, V, Sk)) return TSGEMM_ERR_CUDA;

    AttnParams prm{};
    prm.B = static_cast<int32_t>(B);
    prm.H = static_cast<int32_t>(H);
    prm.Sq = static_cast<int32_t>(Sq);
    prm.Sk = static_cast<int32_t>(Sk);
    prm.nq = static_cast<int32_t>((Sq + kTiles * kBQ - 1) / (kTiles * kBQ));
    // about 64 MB of K and V per chunk of the causal launch order
    const int64_t kv_head_bytes = 2 * Sk * static_cast<int64_t>(D) * 2;
    prm.group = static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(B * H, (64ll << 20) / kv_head_bytes)));
    prm.causal = causal ? 1 : 0;
    prm.scale_log2 = scale * 1.4426950408889634f;  // log2(e)
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
    lc.gridDim = dim3(static_cast<unsigned>(B * H * prm.nq), 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = kSmemBytes;
    lc.stream = s;
    void* args[4] = {&tmQ, &tmK, &tmV, &prm};
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
