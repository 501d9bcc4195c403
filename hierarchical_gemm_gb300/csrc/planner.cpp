// planner.cpp -- host-side problem validation and the choice of tile width,
// K split, pipeline depth and grid for the persistent kernel.
//
// The choice minimises a simple per-SM time model, in SM clock cycles:
//   * a K-slice (BK = 64) of a 128 x BN tile costs max(MMA, operand load):
//     MMA   = 128 * BN * 64 / 4096 cycles (4096 bf16 MACs per SM per cycle),
//     load  = (A slice + B slice bytes) / kL2BytesPerCycle;
//   * a CTA runs ceil(units / grid) units back to back (wave quantisation);
//   * a split tile adds the last CTA's read of S fp32 partial tiles;
//   * the whole job can go no faster than its HBM traffic allows.
// The model only ranks candidates; the tile widths it picks are the
// measured-best ones on the shapes this library is tuned for.
#include "planner.h"

#include <algorithm>
#include <cmath>

namespace tsg {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr double kMacsPerCycle = 4096.0;
constexpr double kL2BytesPerCycle = 96.0;     // operand feed per SM (model)
constexpr double kHbmBytesPerCycle = 3500.0;  // whole GPU (model)
constexpr double kReduceBytesPerCycle = 64.0; // split-K partial reads per SM (model)
constexpr double kUnitOverhead = 600.0;       // pipeline fill / drain per unit (model)
constexpr int kMaxSplits = 32;
constexpr int kDefaultTimeoutMs = 1000;

bool dtype_pair_ok(int din, int dout) {
    if (din == TSGEMM_F16) return dout == TSGEMM_F16 || dout == TSGEMM_F32;
    if (din == TSGEMM_BF16) return dout == TSGEMM_BF16 || dout == TSGEMM_F32;
    return false;
}

int64_t out_bytes(int dout) { return dout == TSGEMM_F32 ? 4 : 2; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Estimate {
    double cycles;
    double compute;
};

Estimate estimate(int64_t M, int64_t N, int64_t K, int dout, int bn, int splits, int num_sms) {
    const int64_t tiles = ceil_div(M, kBM) * ceil_div(N, bn);
    const int64_t units = tiles * splits;
    const int64_t grid = std::min<int64_t>(units, num_sms);
    const int64_t waves = ceil_div(units, grid);
    const int64_t kblocks = ceil_div(K, kBK);
    const double kb_per_unit = std::ceil(static_cast<double>(kblocks) / splits);
    const double mma = kBM * bn * static_cast<double>(kBK) / kMacsPerCycle;
    const double load = (kBM * kBK * 2.0 + bn * kBK * 2.0) / kL2BytesPerCycle;
    const double per_unit = kb_per_unit * std::max(mma, load) + kUnitOverhead;
    double compute = waves * per_unit;
    if (splits > 1) compute += splits * static_cast<double>(kBM) * bn * 4.0 / kReduceBytesPerCycle;
    double bytes = 2.0 * (M * K + K * N) + static_cast<double>(out_bytes(dout)) * M * N;
    if (splits > 1) {
        // partials are written and read back once: charged both to the HBM
        // floor and, since the reduction is not fully hidden, to the time
        const double ws = 2.0 * 4.0 * splits * static_cast<double>(tiles) * kBM * bn;
        bytes += ws;
        compute += ws / kHbmBytesPerCycle;
    }
    const double hbm = bytes / kHbmBytesPerCycle;
    return {std::max(compute, hbm) + 0.05 * compute, compute};
}

}  // namespace

int64_t smem_bytes_for(int block_n, int stages) {
    const int64_t stage = static_cast<int64_t>(kBM) * kBK * 2 + static_cast<int64_t>(block_n) * kBK * 2;
    return 1024 + stages * stage + 8 * (2 * stages + 6) + 16;
}

int max_stages_for(int block_n) {
    int s = 1;
    while (s < 16 && smem_bytes_for(block_n, s + 1) <= kSmemPerCtaMax) ++s;
    return s;
}

tsgemm_status_t validate_problem(int64_t M, int64_t N, int64_t K, int dtype_in, int dtype_out,
                                 int layout) {
    if (M < 1 || N < 1 || K < 1) return TSGEMM_ERR_INVALID_ARG;
    if (dtype_in < TSGEMM_F16 || dtype_in > TSGEMM_F32) return TSGEMM_ERR_INVALID_ARG;
    if (dtype_out < TSGEMM_F16 || dtype_out > TSGEMM_F32) return TSGEMM_ERR_INVALID_ARG;
    if (layout != TSGEMM_LAYOUT_RRR) return layout < 0 ? TSGEMM_ERR_INVALID_ARG : TSGEMM_ERR_UNSUPPORTED;
    if (!dtype_pair_ok(dtype_in, dtype_out)) return TSGEMM_ERR_UNSUPPORTED;
    // Tensor-map coordinates and the kernel's tile indices are 32-bit.
    const int64_t lim = (int64_t{1} << 31) - 1;
    if (M > lim || N > lim || K > lim) return TSGEMM_ERR_UNSUPPORTED;
    // Row strides of A (K * 2), B (N * 2) and C (N * out) must be multiples
    // of 16 bytes for TMA and for the 16-byte vector stores.
    if ((K * 2) % 16 != 0 || (N * 2) % 16 != 0 || (N * out_bytes(dtype_out)) % 16 != 0)
        return TSGEMM_ERR_ALIGNMENT;
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
    if (f.block_m != 0 && f.block_m != kBM) return TSGEMM_ERR_UNSUPPORTED;
    if (f.block_n != 0 && (f.block_n % 64 != 0 || f.block_n < 64 || f.block_n > 256))
        return TSGEMM_ERR_UNSUPPORTED;
    if (f.splits < 0 || f.stages < 0 || f.group_m < 0 || f.grid < 0 || f.timeout_ms < 0)
        return TSGEMM_ERR_INVALID_ARG;
    if (f.units != 0 || f.workspace_bytes != 0) return TSGEMM_ERR_INVALID_ARG;  // derived fields

    const int64_t kblocks = ceil_div(K, kBK);
    if (f.splits > kblocks || f.splits > 4096) return TSGEMM_ERR_UNSUPPORTED;

    // Candidate tile widths: never wider than N rounded up to 64.
    const int64_t n_pad = ceil_div(N, 64) * 64;
    int best_bn = 0, best_s = 0;
    double best = 0;
    const int bns[4] = {256, 192, 128, 64};
    for (int bn : bns) {
        if (f.block_n && bn != f.block_n) continue;
        if (!f.block_n && bn > n_pad && bn != 64) continue;
        const int smax = f.splits ? f.splits : static_cast<int>(std::min<int64_t>(kMaxSplits, std::max<int64_t>(1, kblocks / 4)));
        const int smin = f.splits ? f.splits : 1;
        for (int s = smin; s <= smax; ++s) {
            const Estimate e = estimate(M, N, K, dtype_out, bn, s, num_sms);
            // strict improvement required: ties keep the wider tile / fewer splits
            if (best_bn == 0 || e.cycles < best * 0.999) {
                best = e.cycles;
                best_bn = bn;
                best_s = s;
            }
        }
    }
    if (best_bn == 0) return TSGEMM_ERR_UNSUPPORTED;

    tsgemm_config_t c{};
    c.block_m = kBM;
    c.block_n = best_bn;
    c.splits = best_s;
    const int smax_fit = max_stages_for(best_bn);
    if (f.stages > smax_fit || (f.stages != 0 && f.stages < 2)) return TSGEMM_ERR_UNSUPPORTED;
    c.stages = f.stages ? f.stages : smax_fit;
    c.group_m = f.group_m ? f.group_m : 8;
    const int64_t tiles = ceil_div(M, kBM) * ceil_div(N, best_bn);
    c.units = tiles * best_s;
    c.grid = static_cast<int32_t>(std::min<int64_t>(c.units, f.grid ? f.grid : num_sms));
    c.workspace_bytes = best_s > 1 ? tiles * best_s * kBM * static_cast<int64_t>(best_bn) * 4 : 0;
    c.timeout_ms = f.timeout_ms ? f.timeout_ms : kDefaultTimeoutMs;
    c.debug_flags = f.debug_flags;
    *out = c;
    return TSGEMM_OK;
}

}  // namespace tsg
