// planner.cpp -- host-side problem validation and the choice of tile width,
// K split, pipeline depth and grid for the persistent kernel.
//
// The choice minimises a simple per-SM time model, in SM clock cycles:
//   * a K-slice (128 bytes of K: 64 16-bit or 128 8-bit elements) of a
//     128 x BN tile costs max(MMA, operand load):
//     MMA   = 128 * BN * 64 / 4096 cycles (4096 bf16 MACs per SM per cycle,
//             twice as many 8-bit MACs, so the same cycles per slice),
//     load  = (A slice + B slice bytes) / kL2BytesPerCycle;
//   * a CTA runs ceil(units / grid) units back to back (wave quantisation);
//   * a split tile adds the reduction: every part writes (S - 1) / S of its
//     fp32 partial and reads as much of the others';
//   * the whole job can go no faster than its HBM traffic allows.
// The model only ranks candidates; the tile widths it picks are the
// measured-best ones on the shapes this library is tuned for.
#include "planner.h"

#include <algorithm>
#include <cmath>

namespace tsg {

bool is_8bit(int dtype) { return dtype == TSGEMM_E4M3 || dtype == TSGEMM_E5M2; }

int64_t in_bytes(int dtype_in) { return is_8bit(dtype_in) ? 1 : 2; }

int slice_k(int dtype_in) { return is_8bit(dtype_in) ? 128 : 64; }

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int64_t kEpiWarps = 8;  // epilogue warps, each staging two 32 x 32 output blocks
constexpr double kMacsPerCycle = 4096.0;
constexpr double kL2BytesPerCycle = 72.0;     // operand feed per SM (measured ballpark)
constexpr double kHbmBytesPerCycle = 3500.0;  // whole GPU (model)
constexpr double kReduceBytesPerCycle = 14.0; // split-K partial writes + reads per SM (measured)
constexpr double kUnitOverhead = 600.0;       // pipeline fill / drain per unit (model)
constexpr bool kAutoStreamK = true;          // the planner proposes stream-K itself
constexpr double kFixupCycles = 11000.0;      // stream-K: segment hand-overs and the final add (measured)
// the same when a whole tile follows: the owner's add from global memory
// and its slowdown of the mainloop beside it (measured ~10 us), less the
// part that tile's mainloop hides, but at least kHiddenFixupCycles
constexpr double kMidFixupCycles = 27000.0;
constexpr double kHiddenFixupCycles = 1500.0;
constexpr int kMaxSplits = 32;
constexpr int kDefaultTimeoutMs = 1000;

bool dtype_pair_ok(int din, int dout) {
    if (din == TSGEMM_F16) return dout == TSGEMM_F16 || dout == TSGEMM_F32;
    if (din == TSGEMM_BF16) return dout == TSGEMM_BF16 || dout == TSGEMM_F32;
    if (din == TSGEMM_E4M3 || din == TSGEMM_E5M2)
        return dout == TSGEMM_F16 || dout == TSGEMM_BF16 || dout == TSGEMM_F32;
    return false;
}

int64_t out_bytes(int dout) { return dout == TSGEMM_F32 ? 4 : 2; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// True when the S parts of some split unit fall into two consecutive rounds
// of the static schedule (units u run in round u / slots).  That is
// correct, but the parts in the earlier round then wait for a whole
// mainloop of the later one, so the planner does not choose it.
bool parts_straddle(int64_t full, int64_t split_tiles, int splits, int64_t slots) {
    if (splits <= 1) return false;
    for (int64_t t = 0; t < split_tiles; ++t) {
        const int64_t first = full + t * splits;
        if (first / slots != (first + splits - 1) / slots) return true;
    }
    return false;
}

struct Estimate {
    double cycles;
    double compute;
};

// bm = 128: one CTA per 128 x bn tile; bm = 256: a CTA pair per 256 x bn
// tile, each SM computing 128 rows and loading half of the B slice.  The
// last `split_tiles` tiles of the schedule are split into `splits` K parts
// (all of them, or only the tail wave's, or none).
Estimate estimate(int64_t M, int64_t N, int64_t K, int din, int dout, int bm, int bn, int splits,
                  int64_t split_tiles, int num_sms) {
    const int64_t tiles = ceil_div(M, bm) * ceil_div(N, bn);
    const int64_t full = tiles - split_tiles;
    const int64_t units = full + split_tiles * splits;
    const int64_t slots = std::max(1, num_sms / (bm / kBM));
    const int64_t grid = std::min<int64_t>(units, slots);
    const int64_t kblocks = ceil_div(K, slice_k(din));
    const double kb_split = std::ceil(static_cast<double>(kblocks) / splits);
    const double mma = kBM * bn * static_cast<double>(kBK) / kMacsPerCycle;
    const double b_bytes = (bm == 256 ? bn / 2 : bn) * kBK * 2.0;
    const double load = (kBM * kBK * 2.0 + b_bytes) / kL2BytesPerCycle;
    const double per_kb = std::max(mma, load);
    // round-robin over `grid` slots: whole tiles first, then split parts
    const double whole_rounds = static_cast<double>(ceil_div(full, grid));
    const double split_rounds = static_cast<double>(ceil_div(split_tiles * splits, grid));
    double compute = whole_rounds * (kblocks * per_kb + kUnitOverhead) +
                     split_rounds * (kb_split * per_kb + kUnitOverhead);
    double bytes = static_cast<double>(in_bytes(din)) * (M * K + K * N) +
                   static_cast<double>(out_bytes(dout)) * M * N;
    if (splits > 1 && split_tiles > 0) {
        // each part writes the (S - 1) / S of its fp32 partial it does not
        // own and reads the others' partials of the chunks it owns
        // (in every round of split units)
        compute += split_rounds * 2.0 * (splits - 1) / splits * static_cast<double>(kBM) * bn * 4.0 /
                   kReduceBytesPerCycle;
        const double ws = 2.0 * 4.0 * (splits - 1) * static_cast<double>(split_tiles) * bm * bn;
        bytes += ws;
    }
    const double hbm = bytes / kHbmBytesPerCycle;
    return {std::max(compute, hbm) + 0.05 * compute, compute};
}

// Stream-K: the last `sk` tiles' K slices spread evenly over the slots,
// run before the last of ceil((tiles - sk) / slots) rounds of whole tiles.
// A tile cut between slots costs its later parts a partial write and its
// first part's CTA the final add, both hidden behind the next mainloop;
// with no whole tiles the add comes at the very end.
Estimate estimate_sk(int64_t M, int64_t N, int64_t K, int din, int dout, int bm, int bn, int64_t sk,
                     int num_sms) {
    const int64_t tiles = ceil_div(M, bm) * ceil_div(N, bn);
    const int64_t slots = std::max(1, num_sms / (bm / kBM));
    const int64_t kblocks = ceil_div(K, slice_k(din));
    const double mma = kBM * bn * static_cast<double>(kBK) / kMacsPerCycle;
    const double b_bytes = (bm == 256 ? bn / 2 : bn) * kBK * 2.0;
    const double load = (kBM * kBK * 2.0 + b_bytes) / kL2BytesPerCycle;
    const double per_kb = std::max(mma, load);
    const double dp_rounds = static_cast<double>(ceil_div(tiles - sk, slots));
    const double sk_slices = std::ceil(static_cast<double>(sk) * kblocks / slots);
    // contributors per owner, whose partials the owner reads from global
    // memory at the split-K rate
    const double owners_parts = std::ceil(kblocks / std::max(1.0, sk_slices));
    const double half_bytes = kBM * bn * 4.0;
    const double fetch = owners_parts * half_bytes / kReduceBytesPerCycle;
    const double tail = dp_rounds >= 1 ? std::max(kHiddenFixupCycles, kMidFixupCycles - kblocks * per_kb)
                                       : kFixupCycles + fetch;
    double compute = dp_rounds * (kblocks * per_kb + kUnitOverhead) + sk_slices * per_kb + 2 * kUnitOverhead + tail;
    double bytes = static_cast<double>(in_bytes(din)) * (M * K + K * N) +
                   static_cast<double>(out_bytes(dout)) * M * N +
                   3.0 * 4.0 * static_cast<double>(slots) * bm * bn;
    const double hbm = bytes / kHbmBytesPerCycle;
    return {std::max(compute, hbm) + 0.05 * compute, compute};
}

}  // namespace

int64_t smem_bytes_for(int block_m, int block_n, int dtype_out, int stages, int cluster_split) {
    const int64_t b_cols = block_m == 256 ? block_n / 2 : block_n;
    const int64_t stage = static_cast<int64_t>(kBM) * kBK * 2 + b_cols * kBK * 2;
    // output staging: 8 epilogue warps x 2 buffers of one 32 x 32 16-bit
    // block (fp32 outputs are stored from registers)
    const int64_t staging = dtype_out == TSGEMM_F32 ? 0 : kEpiWarps * 2 * 32 * 32 * out_bytes(dtype_out);
    // cluster split: a 128 x 32 fp32 exchange chunk per epilogue warpgroup
    // and four barriers
    const int64_t exchange = cluster_split >= 2 ? 2 * 128 * 32 * 4 + 4 * 8 : 0;
    return 1024 + stages * stage + staging + exchange + 8 * (2 * stages + 5) + 16;
}

int max_stages_for(int block_m, int block_n, int dtype_out, int cluster_split) {
    int s = 1;
    while (s < 16 && smem_bytes_for(block_m, block_n, dtype_out, s + 1, cluster_split) <= kSmemPerCtaMax) ++s;
    return s;
}

tsgemm_status_t validate_problem(int64_t M, int64_t N, int64_t K, int dtype_in, int dtype_out,
                                 int layout) {
    if (M < 1 || N < 1 || K < 1) return TSGEMM_ERR_INVALID_ARG;
    if (dtype_in < TSGEMM_F16 || dtype_in > TSGEMM_E5M2) return TSGEMM_ERR_INVALID_ARG;
    if (dtype_out < TSGEMM_F16 || dtype_out > TSGEMM_E5M2) return TSGEMM_ERR_INVALID_ARG;
    if (layout < TSGEMM_LAYOUT_RRR || layout > TSGEMM_LAYOUT_CCR) return TSGEMM_ERR_INVALID_ARG;
    if (!dtype_pair_ok(dtype_in, dtype_out)) return TSGEMM_ERR_UNSUPPORTED;
    // 8-bit operands are read K-major only: A stored M x K, B stored N x K.
    if (is_8bit(dtype_in) && layout != TSGEMM_LAYOUT_RCR) return TSGEMM_ERR_UNSUPPORTED;
    // Tensor-map coordinates and the kernel's tile indices are 32-bit.
    const int64_t lim = (int64_t{1} << 31) - 1;
    if (M > lim || N > lim || K > lim) return TSGEMM_ERR_UNSUPPORTED;
    // Stored row strides of A, B and C must be multiples of 16 bytes (TMA).
    const int64_t a_row = (layout & 2) ? M : K;  // A stored K x M, or M x K
    const int64_t b_row = (layout & 1) ? K : N;  // B stored N x K, or K x N
    const int64_t eb = in_bytes(dtype_in);
    if ((a_row * eb) % 16 != 0 || (b_row * eb) % 16 != 0 || (N * out_bytes(dtype_out)) % 16 != 0)
        return TSGEMM_ERR_ALIGNMENT;
    return TSGEMM_OK;
}

// The DSMEM cluster-split plan (forced by cluster_split = 2, 4 or 8):
// one-SM tiles of the widest width up to N, every tile's K range split
// between the cs CTAs of a cs x 1 cluster, one tile per cluster at a time.
static tsgemm_status_t choose_cluster_split(int64_t M, int64_t N, int num_sms, const tsgemm_config_t& f,
                                            int dtype_out, tsgemm_config_t* out) {
    const int cs = f.cluster_split;
    const int64_t n_pad = ceil_div(N, 64) * 64;
    int bn = f.block_n;
    if (!bn) bn = n_pad >= 256 ? 256 : (n_pad >= 192 ? 192 : (n_pad >= 128 ? 128 : 64));
    tsgemm_config_t c{};
    c.block_m = 128;
    c.block_n = bn;
    c.splits = 1;
    const int smax_fit = max_stages_for(128, bn, dtype_out, cs);
    if (f.stages > smax_fit || (f.stages != 0 && f.stages < 2)) return TSGEMM_ERR_UNSUPPORTED;
    c.stages = f.stages ? f.stages : smax_fit;
    c.group_m = f.group_m ? f.group_m : 8;
    c.cluster_split = cs;
    const int64_t tiles = ceil_div(M, 128) * ceil_div(N, bn);
    c.units = tiles;
    const int64_t slots = (f.grid ? f.grid : num_sms) / cs;
    if (slots < 1) return TSGEMM_ERR_UNSUPPORTED;
    c.grid = static_cast<int32_t>(std::min<int64_t>(tiles, slots) * cs);
    c.timeout_ms = f.timeout_ms ? f.timeout_ms : kDefaultTimeoutMs;
    c.debug_flags = f.debug_flags;
    *out = c;
    return TSGEMM_OK;
}

tsgemm_status_t choose_config(int64_t M, int64_t N, int64_t K, int dtype_in, int dtype_out,
                              int layout, int num_sms, const tsgemm_config_t* force,
                              tsgemm_config_t* out) {
    if (!out) return TSGEMM_ERR_INVALID_ARG;
    tsgemm_status_t st = validate_problem(M, N, K, dtype_in, dtype_out, layout);
    if (st != TSGEMM_OK) return st;
    if (num_sms < 1) return TSGEMM_ERR_INVALID_ARG;
    tsgemm_config_t f{};
    if (force) f = *force;
    if (f.block_m != 0 && f.block_m != 128 && f.block_m != 256) return TSGEMM_ERR_UNSUPPORTED;
    // (block_n 512: the 256 x 512 pair tile, forced only, whole tiles only)
    const bool wide = f.block_n == 512;
    if (f.block_n != 0 && !wide && (f.block_n % 64 != 0 || f.block_n < 64 || f.block_n > 256))
        return TSGEMM_ERR_UNSUPPORTED;
    if (f.block_m == 256 && f.block_n != 0 && f.block_n != 128 && f.block_n != 256 && !wide)
        return TSGEMM_ERR_UNSUPPORTED;
    if (wide && (f.block_m != 256 || f.splits > 1 || f.split_tiles > 0 || f.cluster_split > 1))
        return TSGEMM_ERR_UNSUPPORTED;
    if (f.block_m == 256 && num_sms < 2) return TSGEMM_ERR_UNSUPPORTED;
    if (f.splits < 0 || f.stages < 0 || f.group_m < 0 || f.grid < 0 || f.timeout_ms < 0)
        return TSGEMM_ERR_INVALID_ARG;
    if (f.units != 0 || f.workspace_bytes != 0) return TSGEMM_ERR_INVALID_ARG;  // derived fields
    if (f.split_tiles < 0 || (f.split_tiles > 0 && f.splits < 2)) return TSGEMM_ERR_INVALID_ARG;
    if (f.stream_k_tiles < -1) return TSGEMM_ERR_INVALID_ARG;
    if (f.cluster_split < 0 || f.cluster_split > 8 || (f.cluster_split > 2 && f.cluster_split != 4 &&
                                                        f.cluster_split != 8))
        return TSGEMM_ERR_UNSUPPORTED;
    const bool csplit = f.cluster_split >= 2;
    if (csplit) {
        // the DSMEM K split: one-SM tiles, each split into cs parts between
        // the CTAs of a cs x 1 cluster; RRR layout and 16-bit inputs
        if (f.block_m == 256 || f.splits > 1 || f.split_tiles > 0 || f.stream_k_tiles > 0)
            return TSGEMM_ERR_INVALID_ARG;
        if (layout != TSGEMM_LAYOUT_RRR || is_8bit(dtype_in) || num_sms < f.cluster_split)
            return TSGEMM_ERR_UNSUPPORTED;
    }
    if (f.stream_k_tiles > 0 && (f.splits > 1 || f.split_tiles > 0)) return TSGEMM_ERR_INVALID_ARG;

    const int64_t kblocks = ceil_div(K, slice_k(dtype_in));
    if (f.splits > kblocks || f.splits > 4096) return TSGEMM_ERR_UNSUPPORTED;
    if (csplit) {
        if (kblocks < f.cluster_split) return TSGEMM_ERR_UNSUPPORTED;  // every CTA needs a K slice
        return choose_cluster_split(M, N, num_sms, f, dtype_out, out);
    }

    // Candidate tile widths: never wider than N rounded up to 64.
    const int64_t n_pad = ceil_div(N, 64) * 64;
    int best_bm = 0, best_bn = 0, best_s = 0;
    int64_t best_st = 0, best_sk = 0;
    double best = 0;
    const int bms[2] = {256, 128};  // pairs first: ties go to the pair
    const int bns[5] = {512, 256, 192, 128, 64};
    for (int bm : bms) {
        if (f.block_m && bm != f.block_m) continue;
        if (bm == 256 && num_sms < 2) continue;
        for (int bn : bns) {
            if (bn == 512 && !wide) continue;
            if (bm == 256 && bn != 128 && bn != 256 && bn != 512) continue;
            if (f.block_n && bn != f.block_n) continue;
            if (!f.block_n && bn > n_pad && bn != 64 && !(bm == 256 && bn == 128)) continue;
            const int64_t slots = num_sms / (bm / kBM);
            const int64_t tiles = ceil_div(M, bm) * ceil_div(N, bn);
            const int smax = f.splits ? f.splits
                                      : static_cast<int>(std::min<int64_t>(
                                            std::min<int64_t>(kMaxSplits, slots), std::max<int64_t>(1, kblocks / 4)));
            const int smin = f.splits ? f.splits : 1;
            if (bn == 512) {
                // whole tiles (no split), stream-K only when forced
                const int64_t sk = f.stream_k_tiles > 0 ? f.stream_k_tiles : 0;
                if (sk > tiles || (sk > 0 && sk * kblocks < slots)) return TSGEMM_ERR_UNSUPPORTED;
                const Estimate e = sk ? estimate_sk(M, N, K, dtype_in, dtype_out, bm, bn, sk, num_sms)
                                      : estimate(M, N, K, dtype_in, dtype_out, bm, bn, 1, 0, num_sms);
                best = e.cycles;
                best_bm = bm;
                best_bn = bn;
                best_s = 1;
                best_st = 0;
                best_sk = sk;
                continue;
            }
            // stream-K: the tail wave, or the tail and one full wave before it
            // (so that whole-tile rounds stay whole), or a forced count
            if (f.stream_k_tiles != -1 && smin == 1 && !f.split_tiles) {
                int64_t sk_opts[2] = {-1, -1};
                if (f.stream_k_tiles > 0) {
                    sk_opts[0] = f.stream_k_tiles;
                } else if (kAutoStreamK && (tiles % slots != 0 || tiles < slots)) {
                    sk_opts[0] = tiles % slots;
                    if (tiles > slots) sk_opts[1] = tiles % slots + slots;
                }
                for (int64_t sk : sk_opts) {
                    // every slot needs at least one K slice, so that the
                    // slots sharing a tile are consecutive
                    if (sk <= 0 || sk > tiles || sk * kblocks < slots) continue;
                    const Estimate e = estimate_sk(M, N, K, dtype_in, dtype_out, bm, bn, sk, num_sms);
                    if (best_bn == 0 || e.cycles < best * 0.999) {
                        best = e.cycles;
                        best_bm = bm;
                        best_bn = bn;
                        best_s = 1;
                        best_st = 0;
                        best_sk = sk;
                    }
                }
            }
            for (int s = smin; s <= smax; ++s) {
                if (f.stream_k_tiles > 0) break;
                // which tiles are split: none (s = 1), a forced count, every
                // tile, or only the tiles of the last, partial wave
                int64_t options[2] = {0, -1};
                if (s > 1) {
                    if (f.split_tiles) {
                        options[0] = f.split_tiles;
                    } else {
                        options[0] = tiles;
                        if (!f.splits && tiles > slots && tiles % slots != 0) options[1] = tiles % slots;
                    }
                }
                for (int64_t st : options) {
                    if (st < 0 || st > tiles) continue;
                    if (!f.splits && parts_straddle(tiles - st, st, s, slots)) continue;
                    const Estimate e = estimate(M, N, K, dtype_in, dtype_out, bm, bn, s, st, num_sms);
                    // strict improvement required: ties keep the earlier candidate
                    if (best_bn == 0 || e.cycles < best * 0.999) {
                        best = e.cycles;
                        best_bm = bm;
                        best_bn = bn;
                        best_s = s;
                        best_st = st;
                        best_sk = 0;
                    }
                }
            }
        }
    }
    if (best_bn == 0) return TSGEMM_ERR_UNSUPPORTED;

    // 256 x 512 pair tiles when the whole-tile schedule of them has at
    // least four rounds and a last round at least two thirds full: a K
    // slice's A then feeds two N = 256 MMAs (a quarter fewer operand bytes
    // per flop), which pays while the tile's epilogue, no longer overlapped
    // with the next tile, is a small part of a round and no stream-K is
    // needed (a stream-K reduction of 256 x 512 partials costs more than
    // it balances).  RRR and RCR layouts, as the planner's own choice only.
    if (!f.block_m && !f.block_n && !f.splits && !f.split_tiles && f.stream_k_tiles <= 0 && best_bm == 256 &&
        (layout == TSGEMM_LAYOUT_RRR || layout == TSGEMM_LAYOUT_RCR) && N >= 512 &&
        (!f.stages || f.stages <= max_stages_for(256, 512, dtype_out))) {
        const int64_t wide_tiles = ceil_div(M, 256) * ceil_div(N, 512);
        const int64_t wide_slots = (f.grid ? f.grid : num_sms) / 2;
        const int64_t rounds = wide_slots > 0 ? wide_tiles / wide_slots : 0;
        const int64_t rem = wide_slots > 0 ? wide_tiles % wide_slots : 0;
        if (rounds >= 4 && (rem == 0 || 3 * rem >= 2 * wide_slots)) {
            best_bn = 512;
            best_s = 1;
            best_st = 0;
            best_sk = 0;
        }
    }

    tsgemm_config_t c{};
    c.block_m = best_bm;
    c.block_n = best_bn;
    c.splits = best_s;
    const int smax_fit = max_stages_for(best_bm, best_bn, dtype_out);
    if (f.stages > smax_fit || (f.stages != 0 && f.stages < 2)) return TSGEMM_ERR_UNSUPPORTED;
    c.stages = f.stages ? f.stages : smax_fit;
    // raster groups of 16 tile rows when stream-K is on or the tiles are
    // 256 x 512 (same box, alternating plans: 4096^3 bf16 89.1 against
    // 90.5 us, mean of five; 6144^3 260.7 against 261.8; 16384 x 16384 x
    // 8192 bf16 2251-2264 against 2285-2304 us, E4M3 1177-1182 against
    // 1193-1197, 1000 steps under the power cap 2444-2450 against
    // 2470-2473 us with a quarter less DRAM traffic; 8192^3 alike); 8
    // otherwise
    c.group_m = f.group_m ? f.group_m : ((best_sk > 0 || best_bn == 512) ? 16 : 8);
    c.cluster_split = 1;
    const int64_t tiles = ceil_div(M, best_bm) * ceil_div(N, best_bn);
    c.split_tiles = best_s > 1 ? best_st : 0;
    c.stream_k_tiles = best_sk;
    c.units = (tiles - c.split_tiles) + c.split_tiles * best_s;
    // a pair kernel launches two CTAs per unit slot
    const int64_t ctas_per_slot = best_bm / kBM;
    int64_t slots = (f.grid ? f.grid : num_sms) / ctas_per_slot;
    if (slots < 1) return TSGEMM_ERR_UNSUPPORTED;
    if (best_sk > 0) {
        // every slot takes part in the stream-K ranges; units = whole tiles
        // + stream-K segments (one per tile a slot's range touches)
        const int64_t w = best_sk * kblocks;
        int64_t segs = 0;
        for (int64_t g = 0; g < slots; ++g) {
            const int64_t a = g * w / slots, b = (g + 1) * w / slots;
            if (b > a) segs += (b - 1) / kblocks - a / kblocks + 1;
        }
        c.units = tiles - best_sk + segs;
        c.grid = static_cast<int32_t>(slots * ctas_per_slot);
        // two fp32 partial slots per CTA half of each slot: one for the
        // segment that continues a tile, one for the owner of a tile (which
        // writes its partial when a contributor is still to come)
        c.workspace_bytes = 2 * slots * best_bm * static_cast<int64_t>(best_bn) * 4;
        c.timeout_ms = f.timeout_ms ? f.timeout_ms : kDefaultTimeoutMs;
        c.debug_flags = f.debug_flags;
        *out = c;
        return TSGEMM_OK;
    }
    // (the parts of a split tile never wait for one another, so S may
    // exceed the grid's slots: the parts then run one after another)
    c.grid = static_cast<int32_t>(std::min<int64_t>(c.units, slots) * ctas_per_slot);
    // S fp32 partial slots per split tile; each part fills the chunks it
    // does not own
    c.workspace_bytes = c.split_tiles * best_s * best_bm * static_cast<int64_t>(best_bn) * 4;
    c.timeout_ms = f.timeout_ms ? f.timeout_ms : kDefaultTimeoutMs;
    c.debug_flags = f.debug_flags;
    *out = c;
    return TSGEMM_OK;
}

}  // namespace tsg
