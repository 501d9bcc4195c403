// gemm_sm103.cuh -- the persistent, warp-specialised tcgen05 GEMM kernel.
//
// C = A * B, A (M x K) and B (K x N) 16-bit floats in any of the four
// row/column-major layouts, or 8-bit floats (E4M3 / E5M2) with both operands
// K-major; fp32 accumulation in tensor memory, C (M x N) row-major
// fp16/bf16/fp32.
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
//     (kind::f8f6f4 for 8-bit inputs) issued by a single thread, four
//     instructions per 128-byte slice;
//   * T.copy(C_r, C)                                -> tcgen05.ld by an
//     epilogue warpgroup, fp32 -> output conversion, global stores;
//   * warp(group) specialisation by rank (TileScale README, T.Scale
//     "warpgroup" example): warp 0 produces, warp 1 issues MMAs, warps 2-9
//     (two warpgroups, each taking half of the tile's columns) drain the
//     accumulator;
//   * persistent thread blocks (TileScale roadmap, resource control): every
//     CTA walks a static list of work units;
//   * the K split with a reduction (TileScale README, "Example of GEMM",
//     warpgroups split along K and reduce): a work unit may cover a K range
//     of a tile (all tiles, or only those of the last, partial wave);
//     partial tiles go to an fp32 workspace and are added in split order;
//   * stream-K: the K slices of the schedule's last tiles are spread evenly
//     over all CTAs, so every CTA ends at the same time; the partials of a
//     tile cut between CTAs are added, in K order, by whichever CTA
//     completes the set (usually the one holding its first K slices).
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
constexpr int kEpiWarps = 8;    // two epilogue warpgroups
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 64 + kEpiThreads;  // producer warp, MMA warp, epilogue
constexpr int kMaxStages = 16;

enum OutKind { kOutF16 = 0, kOutBF16 = 1, kOutF32 = 2 };

// K-elements per ring slice: one 128-byte swizzle row of the operand, 64
// 16-bit or 128 8-bit elements.  The shared-memory tiles have the same
// bytes either way; only the MMA kind and the TMA K coordinate differ.
template <bool kF8>
__host__ __device__ constexpr int slice_k() { return kF8 ? 128 : kBK; }

// Operand layouts (the tsgemm_layout_t values): bit 1 set = A stored K x M
// (column-major A, M contiguous); bit 0 set = B stored N x K (column-major
// B, K contiguous -- the transpose_B form).  C is always M x N row-major.
__host__ __device__ constexpr bool a_kmajor(int layout) { return (layout & 2) == 0; }
__host__ __device__ constexpr bool b_kmajor(int layout) { return (layout & 1) != 0; }

// Shared-memory operand tiles use the 128-byte swizzle either way:
//   K-major (rows of 64 K-elements, 128 B): 8-row groups 1024 B apart, the
//     k-th 16-deep MMA step is 32 B along the row (+2 in the descriptor's
//     16-byte address field);
//   MN-major (64 M/N-elements per 128-B row, one row per k): 64-wide boxes
//     8 KiB apart (LBO), 8-row groups 1024 B apart (SBO), the k-th step is
//     16 rows, 2048 B (+128).
__host__ __device__ constexpr uint32_t op_lbo(bool kmajor) { return kmajor ? 16u : 8192u; }
__host__ __device__ constexpr uint64_t op_kstep(bool kmajor) { return kmajor ? 2u : 128u; }

struct GemmParams {
    int32_t M, N, K;
    int32_t tiles_m, tiles_n;
    int32_t splits;       // S: K parts of each split tile
    int32_t kblocks;      // ceil(K / K-elements per slice)
    int32_t group_m;      // raster group height in tiles
    int32_t stages;
    int32_t debug_flags;
    int64_t full_tiles;   // tiles [0, full_tiles) of the schedule are not split
    int64_t units;        // full_tiles + (tiles - full_tiles) * S (split mode)
    int64_t sk_tiles;     // stream-K mode: the last sk_tiles tiles (0: split mode)
    int64_t sk_work;      // sk_tiles * kblocks K slices, spread over the slots
    uint32_t idesc;       // tcgen05 instruction descriptor
    int32_t csplit;       // cluster split: CTAs of a cluster sharing each
                          // tile's K range (2, 4 or 8), else 1
    void* C;
    float* ws;            // fp32 partials of the split tiles (S > 1), or of the
                          // stream-K segments that continue a tile (one per slot)
    float* ws_own;        // stream-K: the partials of tile owners (one per slot)
    int* counters;        // arrival counters per split (stream-K) tile half,
                          // 32-column chunk and lane quarter; zero between launches
    int* status;          // plan status word
    uint64_t timeout_ns;
};

// One work unit: a whole tile, one of the S K-parts of a split tile, or a
// stream-K segment of a tile.
struct Unit {
    int tm, tn;      // tile row and column
    int split;       // place of this unit's partial in the tile's part order
    int nsplit;      // 1: the whole tile; else the tile's parts (S, or a
                     // stream-K owner and its contributors)
    int kb0, kb1;    // K-slices [kb0, kb1)
    int64_t slot;    // index of the tile among the split (or stream-K) tiles
    int sk;          // 0: not stream-K; 1: a later K range of a tile (a
                     // contributor); 2: the tile's first K range (its owner,
                     // part 0)
};

// Tile row and column of linear tile `tile`: tiles are rastered in groups
// of `group_m` tile rows so that concurrently running CTAs share A and B
// panels in L2.
__device__ __forceinline__ void tile_coords(const GemmParams& p, int64_t tile, int& tm, int& tn) {
    const int64_t span = static_cast<int64_t>(p.group_m) * p.tiles_n;
    const int64_t group = tile / span;
    const int first_m = static_cast<int>(group * p.group_m);
    const int gm = min(p.tiles_m - first_m, p.group_m);
    const int64_t rr = tile - group * span;
    tm = first_m + static_cast<int>(rr % gm);
    tn = static_cast<int>(rr / gm);
}

// Work unit u of the static schedule (split mode).  The first full_tiles
// units are whole tiles; after them come the split tiles, their S parts
// adjacent so that they run at the same time (the split tiles are the
// schedule's last, so splitting fills the last, partial wave of tiles).
__device__ __forceinline__ Unit decode_unit(const GemmParams& p, int64_t u) {
    Unit r;
    int64_t tile;
    if (u < p.full_tiles || p.splits == 1) {
        tile = u;
        r.split = 0;
        r.nsplit = 1;
        r.slot = -1;
    } else {
        const int64_t v = u - p.full_tiles;
        const int64_t t = v / p.splits;
        tile = p.full_tiles + t;
        r.split = static_cast<int>(v - t * p.splits);
        r.nsplit = p.splits;
        r.slot = t;
    }
    tile_coords(p, tile, r.tm, r.tn);
    r.kb0 = static_cast<int>(static_cast<int64_t>(r.split) * p.kblocks / r.nsplit);
    r.kb1 = static_cast<int>(static_cast<int64_t>(r.split + 1) * p.kblocks / r.nsplit);
    r.sk = 0;
    return r;
}

// Stream-K mode: the sk_work K slices of the last sk_tiles tiles (tile by
// tile, k ascending) are cut into G equal ranges; slot g takes slices
// [g W / G, (g + 1) W / G).  sk_slot_of(x) is the slot whose range holds
// slice x.
__device__ __forceinline__ int64_t sk_begin(const GemmParams& p, int64_t g, int64_t G) { return g * p.sk_work / G; }
__device__ __forceinline__ int64_t sk_slot_of(const GemmParams& p, int64_t x, int64_t G) {
    return ((x + 1) * G - 1) / p.sk_work;
}

// The j-th work unit of slot g of the G slots (CTAs, or CTA clusters);
// false past the slot's last.  Split mode: units g, g + G, g + 2G, ...
// Stream-K mode: the slot's whole tiles (g, g + G, ... below full_tiles)
// but the last, then the segments of its stream-K range, one per tile it
// touches, then its last whole tile.  A range that starts inside a tile
// contributes that tile's later K slices (sk = 1) and is the first
// segment; one that ends inside a tile holds its first K slices (sk = 2),
// the last segment, which usually finds the others' partials ready and
// adds them while its tensor cores already work on the last whole tile.
// (With no whole tiles the stream-K segments are all there is.)
__device__ __forceinline__ bool unit_at(const GemmParams& p, int64_t g, int64_t G, int64_t j, Unit& r) {
    if (p.sk_tiles == 0) {
        const int64_t u = g + j * G;
        if (u >= p.units) return false;
        r = decode_unit(p, u);
        return true;
    }
    r.split = 0;
    r.nsplit = 1;
    r.slot = -1;
    r.sk = 0;
    const int64_t ndp = g < p.full_tiles ? (p.full_tiles - 1 - g) / G + 1 : 0;
    const int64_t kb = p.kblocks;
    const int64_t a = sk_begin(p, g, G), b = sk_begin(p, g + 1, G);
    const int64_t nsk = b > a ? (b - 1) / kb - a / kb + 1 : 0;  // stream-K segments of the slot
    const int64_t first_dp = ndp > 0 ? ndp - 1 : 0;              // whole tiles before them
    if (j < first_dp || (ndp > 0 && j == first_dp + nsk)) {
        const int64_t d = j < first_dp ? j : ndp - 1;
        tile_coords(p, g + d * G, r.tm, r.tn);
        r.kb0 = 0;
        r.kb1 = p.kblocks;
        return true;
    }
    const int64_t jj = j - first_dp;
    if (jj >= nsk) return false;
    const int64_t start = jj == 0 ? a : (a / kb + jj) * kb;
    const int64_t t = start / kb;
    const int64_t end = min(b, (t + 1) * kb);
    tile_coords(p, p.full_tiles + t, r.tm, r.tn);
    r.kb0 = static_cast<int>(start - t * kb);
    r.kb1 = static_cast<int>(end - t * kb);
    if (r.kb0 > 0 || r.kb1 < kb) {
        // the tile is cut between slots g_o (its owner) .. g_l, consecutive
        const int64_t g_o = sk_slot_of(p, t * kb, G), g_l = sk_slot_of(p, (t + 1) * kb - 1, G);
        r.sk = r.kb0 > 0 ? 1 : 2;
        r.slot = t;
        r.split = static_cast<int>(g - g_o);
        r.nsplit = 1 + static_cast<int>(g_l - g_o);
    }
    return true;
}

// Output path.  16-bit outputs are staged in shared memory: each epilogue
// warp owns two buffers of one 32 x 32 block (rows = its 32 accumulator
// lanes, 32 columns), filled from registers and written to C by a TMA
// tensor store, so that global writes are whole lines and rows or columns
// past the edge of C are clipped by the copy engine.  The block is laid out
// in the tensor map's 64-byte swizzle; buffers are 1024-byte aligned, as
// the swizzle requires.  fp32 outputs go straight from registers to C (each
// thread writes its row's 128 contiguous bytes): their staging would take
// 64 KiB, two slots of the operand ring, and the deeper ring is worth more
// (measured on the 1024 x 1024 x 65536 shape).
template <int kOut>
__host__ __device__ constexpr uint32_t epi_buf_bytes() {
    return kOut == kOutF32 ? 0u : 32u * 32u * 2u;  // one 32 x 32 16-bit block
}
template <int kOut>
__host__ __device__ constexpr uint32_t epi_smem_bytes() {
    return kEpiWarps * 2u * epi_buf_bytes<kOut>();  // 32 KiB (16-bit), none (fp32)
}

template <int kOut>
struct CStager {
    uint32_t buf0;   // this warp's first buffer; the second follows it
    uint32_t which;  // buffer to fill next
    int lane;

    // Convert 32 fp32 values (this lane's row, 32 consecutive columns) and
    // store the warp's 32 x 32 block at (row0, col0) of C.
    __device__ __forceinline__ void put(const GemmParams& p, const CUtensorMap* tmC, int row0, int col0,
                                        const uint32_t (&r)[32]) {
        if constexpr (kOut == kOutF32) {
            // straight to C: this lane's row, 8 16-byte vectors; N is a
            // multiple of 4, so a vector is wholly inside C or outside
            const int row = row0 + lane;
            if (row < p.M) {
                float* dst = static_cast<float*>(p.C) + static_cast<int64_t>(row) * p.N + col0;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (col0 + 4 * j < p.N) st_global_v4(dst + 4 * j, r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
            }
        } else {
            const uint32_t buf = buf0 + which * epi_buf_bytes<kOut>();
            if (lane == 0) bulk_wait_group_read<1>();  // the store that used `buf` last has read it
            __syncwarp();
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float lo = __uint_as_float(r[2 * i]), hi = __uint_as_float(r[2 * i + 1]);
                w[i] = kOut == kOutBF16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
            }
            // 64-byte rows in the TMA 64-byte swizzle: chunk j of row l sits
            // at chunk position j ^ ((l / 2) mod 4)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                st_shared_v4(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2],
                             w[4 * j + 3]);
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
                if (row0 < p.M && col0 < p.N) tma_store_2d(tmC, buf, col0, row0);
                bulk_commit_group();  // (an empty group when the block is wholly outside C)
            }
            which ^= 1u;
        }
    }

    // All of this warp's stores have read their staging buffers, so the
    // CTA may leave: the writes to C complete on their own, before the
    // grid is done (nothing in the kernel reads C back).
    __device__ __forceinline__ void drain() {
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
    }
};

// Drain one work unit's accumulator (128 rows x BN columns of tensor memory
// at `tbase`; this thread holds row `row_local`, and its warp's 32 rows
// start at row `row0` of C).
//   * A whole tile is converted and stored to C.
//   * A unit that holds part of a tile's K range -- one of the S parts of a
//     split tile, or a stream-K segment of a tile cut between slots -- adds
//     its fp32 partial to the others' in a fixed part order (K order):
//     0 + p_0 + p_1 + ... + p_{n-1}.  Part 0 of a stream-K tile is the
//     segment holding the tile's first K slices (its owner), parts 1..n-1
//     the later ranges.  The bits do not depend on which part adds or when.
//     Each epilogue warp works on its 32 rows one 32-column chunk at a time,
//     on its own: if the other n - 1 parts have already counted that chunk
//     in, it adds their partials now; otherwise it writes its partial to the
//     workspace and counts itself in, and the part whose count completes
//     the chunk adds.  No part ever waits for another, so the parts need
//     not run at the same time: a plan stays correct when its CTAs run one
//     after another (more parts than CTAs, or SMs held by other work).
// `h` indexes the split (stream-K) tile's 128-row half: its counters and,
// in split mode, its workspace slots.
struct EpiAux {
    int64_t wsi;          // stream-K: this slot's workspace index (128 x BN fp32 each)
    int64_t wstride;      // stream-K: workspace index step from one slot to the next
};

// Layout of one 128-row x 32-column fp32 partial chunk in the workspace, in
// the order the epilogue warps hold it: [4 lane quarters][8 float4][32
// lanes], so that every warp access is 512 contiguous bytes.
constexpr int kChunkFloats = 4 * 8 * 128;

// Where part s of the unit's tile keeps the partial of 32-column chunk
// `chunk`, at this lane's first float of lane quarter q.
//   split mode: S slots per tile half, [h][part][BN / 32 chunks];
//   stream-K: part 0 (the owner) in the owner area of its slot, part s >= 1
//   in the area of its own slot (the slots of a cut tile are consecutive).
template <int BN>
__device__ __forceinline__ float* part_chunk(const GemmParams& p, const Unit& un, const EpiAux& aux, int64_t h,
                                             int s, int chunk, int q, int lane) {
    const int64_t off = static_cast<int64_t>(chunk) * kChunkFloats + q * (8 * 128) + lane * 4;
    if (un.sk == 0) return p.ws + ((h * un.nsplit + s) * (BN / 32)) * kChunkFloats + off;
    const int64_t idx = aux.wsi + static_cast<int64_t>(s - un.split) * aux.wstride;
    return (s == 0 ? p.ws_own : p.ws) + idx * (kBM * BN) + off;
}

// Counter of (tile half h, chunk, lane quarter q): how many parts have
// written that partial; reset to zero by the part that adds.
template <int BN>
__device__ __forceinline__ int* part_counter(const GemmParams& p, int64_t h, int chunk, int q) {
    return p.counters + (h * (BN / 32) + chunk) * 4 + q;
}

// A stream-K owner segment asks for its contributors' partials in L2 before
// its own accumulator is ready (the contributors, first segments of their
// slots, are usually long done by then).
template <int BN>
__device__ __forceinline__ void prefetch_sk_partials(const GemmParams& p, const Unit& un, const EpiAux& aux,
                                                     int etid) {
    if (un.sk != 2 || etid != 0) return;
    constexpr uint32_t kChunkBytes = kChunkFloats * 4u;
    for (int s = 1; s < un.nsplit; ++s)
        for (int c = 0; c < BN; c += 32)
            bulk_prefetch_l2(p.ws + (aux.wsi + s * aux.wstride) * (kBM * BN) + (c >> 5) * kChunkFloats,
                             kChunkBytes);
}

template <int BN, int kOut, class Release>
__device__ __forceinline__ void drain_parts(const GemmParams& p, const CUtensorMap* tmC, CStager<kOut>& out,
                                            const Unit& un, uint32_t tbase, int row0, int row_local, int64_t h,
                                            const EpiAux& aux, int c_begin, Release&& release) {
    const int n = un.nsplit, me = un.split;
    const int q = row_local >> 5, lane = row_local & 31;
    const int col0 = un.tn * BN;
    constexpr int kNc = BN / 64;  // 32-column chunks in this warpgroup's half
    // Parts start at different chunks, so that (when they run side by side)
    // each completes, and adds, about 1/n of the chunks, at its end.
    const int first = me * kNc / n;
#pragma unroll 1
    for (int k = 0; k < kNc; ++k) {
        int cl = first + k;
        if (cl >= kNc) cl -= kNc;
        const int c = c_begin + cl * 32;
        const int chunk = c >> 5;
        uint32_t r[32];
        tmem_ld_32x32b_x32(tbase + c, r);
        tmem_ld_wait();
        if (k == kNc - 1) release();  // this thread's accumulator part is in registers
        int* cnt = part_counter<BN>(p, h, chunk, q);
        int last = 0;
        if (lane == 0) last = ld_acquire_gpu(cnt) == n - 1 ? 1 : 0;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last) {
            float* dst = part_chunk<BN>(p, un, aux, h, me, chunk, q, lane);
#pragma unroll
            for (int v = 0; v < 8; ++v)
                st_global_v4(dst + v * 128, r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]);
            __threadfence();  // the partial is visible before it is counted
            __syncwarp();
            if (lane == 0) last = atom_acq_rel_gpu_add(cnt, 1) == n - 1 ? 1 : 0;
            last = __shfl_sync(0xffffffffu, last, 0);
            if (!last) continue;
        }
        __threadfence();  // the other parts' partials, counted in, are read after the count
        // 0 + p_0 + ... + p_{n-1}: the others' partials come two loads ahead
        // of the add; this part's own term (in registers) at its place
        auto other = [&](int i) { return i < me ? i : i + 1; };
        auto fetch = [&](int i, float4 (&dst)[8]) {
            if (i < n - 1) {
                const float* src = part_chunk<BN>(p, un, aux, h, other(i), chunk, q, lane);
#pragma unroll
                for (int v = 0; v < 8; ++v) dst[v] = ld_global_cg_f4(src + v * 128);
            }
        };
        float acc[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = 0.0f;
        auto add_own = [&]() {
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = __fadd_rn(acc[j], __uint_as_float(r[j]));
        };
        auto add = [&](const float4 (&src)[8]) {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                acc[4 * v] = __fadd_rn(acc[4 * v], src[v].x);
                acc[4 * v + 1] = __fadd_rn(acc[4 * v + 1], src[v].y);
                acc[4 * v + 2] = __fadd_rn(acc[4 * v + 2], src[v].z);
                acc[4 * v + 3] = __fadd_rn(acc[4 * v + 3], src[v].w);
            }
        };
        float4 pa[8], pb[8];
        fetch(0, pa);
        fetch(1, pb);
#pragma unroll 1
        for (int i = 0; i < n - 1; i += 2) {
            if (i == me) add_own();
            add(pa);
            fetch(i + 2, pa);
            if (i + 1 < n - 1) {
                if (i + 1 == me) add_own();
                add(pb);
                fetch(i + 3, pb);
            }
        }
        if (me == n - 1) add_own();
        uint32_t w[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) w[j] = __float_as_uint(acc[j]);
        out.put(p, tmC, row0, col0 + c, w);
        if (lane == 0) *reinterpret_cast<volatile int*>(cnt) = 0;  // ready for the next launch
    }
}

template <int BN, int kOut, class Release>
__device__ __forceinline__ void drain_unit(const GemmParams& p, const CUtensorMap* tmC, CStager<kOut>& out,
                                           const Unit& un, uint32_t tbase, int row0, int row_local, int64_t h,
                                           const EpiAux& aux, int c_begin, Release&& release) {
    if (un.nsplit > 1) {
        drain_parts<BN, kOut>(p, tmC, out, un, tbase, row0, row_local, h, aux, c_begin, release);
        return;
    }
    const int col0 = un.tn * BN;
    const int c_end = c_begin + BN / 2;  // this warpgroup's half of the columns
#pragma unroll 1
    for (int c = c_begin; c < c_end; c += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tbase + c, r);
        tmem_ld_wait();
        if (c + 32 >= c_end) release();  // this thread's accumulator part is in registers
        out.put(p, tmC, row0, col0 + c, r);
    }
}

// TMA loads of K-slice kb into a ring slot: A rows [row, row + 128) at
// a_dst, B columns [col, col + kBCols) at b_dst, in the layout's operand
// order.  kRemote: the completion goes to a barrier of the peer CTA (the
// pair's leader), which needs the cta_group::2 form of the copy.
template <bool kRemote>
__device__ __forceinline__ void tma_ld(uint32_t dst, const CUtensorMap* m, uint32_t bar, int32_t c0, int32_t c1) {
    if constexpr (kRemote)
        tma_load_2d_pair(dst, m, bar, c0, c1);
    else
        tma_load_2d(dst, m, bar, c0, c1);
}
template <int kLayout, int kBCols, bool kRemote, bool kF8 = false>
__device__ __forceinline__ void load_b(uint32_t b_dst, const CUtensorMap* tmB, uint32_t bar, int kb, int32_t col) {
    static_assert(!kF8 || b_kmajor(kLayout), "8-bit operands are K-major");
    constexpr int kSK = slice_k<kF8>();
    if constexpr (b_kmajor(kLayout)) {
        tma_ld<kRemote>(b_dst, tmB, bar, kb * kSK, col);  // one 128-byte (K) x kBCols (N) box
    } else {
#pragma unroll
        for (int j = 0; j < kBCols / 64; ++j) tma_ld<kRemote>(b_dst + j * 8192u, tmB, bar, col + j * 64, kb * kBK);
    }
}
template <int kLayout, int kBCols, bool kRemote, bool kF8 = false>
__device__ __forceinline__ void load_slice(uint32_t a_dst, uint32_t b_dst, const CUtensorMap* tmA,
                                           const CUtensorMap* tmB, uint32_t bar, int kb, int32_t row,
                                           int32_t col) {
    static_assert(!kF8 || (a_kmajor(kLayout) && b_kmajor(kLayout)), "8-bit operands are K-major");
    constexpr int kSK = slice_k<kF8>();
    if constexpr (a_kmajor(kLayout)) {
        tma_ld<kRemote>(a_dst, tmA, bar, kb * kSK, row);  // one 128-byte (K) x 128 (M) box
    } else {
        tma_ld<kRemote>(a_dst, tmA, bar, row, kb * kBK);  // two 64 (M) x 64 (K) boxes
        tma_ld<kRemote>(a_dst + 8192u, tmA, bar, row + 64, kb * kBK);
    }
    load_b<kLayout, kBCols, kRemote, kF8>(b_dst, tmB, bar, kb, col);
}

// The four MMAs of one K-slice held at a_addr / b_addr: 16-deep kind::f16
// steps, or 32-deep kind::f8f6f4 steps for 8-bit operands (32 bytes of a
// K-major row either way, so the descriptor steps are the same).
template <int kLayout, int kCtaGroup, bool kF8 = false>
__device__ __forceinline__ void mma_slice(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr, uint32_t idesc,
                                          uint32_t accumulate) {
    constexpr bool ak = a_kmajor(kLayout), bk = b_kmajor(kLayout);
    const uint64_t ad = smem_desc_sw128(a_addr, op_lbo(ak), 1024u);
    const uint64_t bd = smem_desc_sw128(b_addr, op_lbo(bk), 1024u);
    constexpr uint64_t as = op_kstep(ak), bs = op_kstep(bk);
    auto mma = [&](uint64_t a, uint64_t b, uint32_t acc) {
        if constexpr (kF8)
            umma_f8<kCtaGroup>(d_tmem, a, b, idesc, acc);
        else
            umma_f16<kCtaGroup>(d_tmem, a, b, idesc, acc);
    };
    mma(ad, bd, accumulate);
    mma(ad + as, bd + bs, 1u);
    mma(ad + 2 * as, bd + 2 * bs, 1u);
    mma(ad + 3 * as, bd + 3 * bs, 1u);
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

// The cluster-split form's exchange area: one 128-row x 32-column fp32
// chunk per epilogue warpgroup, and its full / empty barriers.
constexpr uint32_t kCsBufBytes = 2u * kBM * 32u * 4u;
constexpr uint32_t kCsBytes = kCsBufBytes + 4u * 8u;

// Bytes of dynamic shared memory the kernel needs for `stages` slots.
template <int BN, int kOut, bool kCS = false>
__host__ __device__ constexpr uint32_t smem_bytes_1sm(int stages) {
    return 1024u /* alignment slack */ + stages * TileShape<BN>::kStageBytes + epi_smem_bytes<kOut>() +
           (kCS ? kCsBytes : 0u) + 8u * (2 * stages + 5) /* barriers */ + 16u /* tmem holder, abort flag */;
}

// Cluster split (a cs x 1 cluster of one-SM CTAs per tile, cs = 2, 4 or
// 8): CTA r computes the r-th of cs consecutive parts of the tile's K
// range, and the partial sums travel down the cluster as a chain: CTA r
// receives 0 + p_0 + ... + p_{r-1} from CTA r - 1 through distributed
// shared memory, adds its own p_r (so the parts are summed in K order) and
// passes the sum to CTA r + 1; the last CTA stores C.  Per epilogue warp
// and 32-column chunk: a sender waits until its successor's buffer is free
// (the successor arrives on the sender's empty barrier), writes its 32 rows
// there with st.shared::cluster and arrives (release, cluster scope) on
// the successor's full barrier; a receiver waits for that (acquire), adds,
// and arrives on its predecessor's empty barrier.  Every lane arrives, so
// each lane's own writes (reads) are ordered before its arrival.  `buf` is
// this warp's 4 KiB of its warpgroup's receive buffer; `phase` counts
// chunks.  No CTA waits for one outside its cluster, whose CTAs the
// hardware runs together.
template <int BN, int kOut, class Release>
__device__ __forceinline__ bool drain_cs(const GemmParams& p, const CUtensorMap* tmC, CStager<kOut>& out,
                                         const Unit& un, uint32_t tbase, int row0, int lane, int c_begin,
                                         uint32_t rank, uint32_t buf, uint32_t full_bar, uint32_t empty_bar,
                                         uint32_t& phase, const WaitCtl& ctl, Release&& release) {
    const int col0 = un.tn * BN;
    const int c_end = c_begin + BN / 2;
    const uint32_t last = static_cast<uint32_t>(p.csplit) - 1u;
#pragma unroll 1
    for (int c = c_begin; c < c_end; c += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tbase + c, r);
        tmem_ld_wait();
        if (c + 32 >= c_end) release();
        float acc[32];
        if (rank == 0) {
            // the sum starts from a cleared (+0) accumulator
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = __fadd_rn(0.0f, __uint_as_float(r[j]));
        } else {
            if (!wait_bounded<true>(full_bar, phase, ctl)) return false;
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const float4 x = ld_shared_f4(buf + lane * 16u + v * 512u);
                acc[4 * v] = __fadd_rn(x.x, __uint_as_float(r[4 * v]));
                acc[4 * v + 1] = __fadd_rn(x.y, __uint_as_float(r[4 * v + 1]));
                acc[4 * v + 2] = __fadd_rn(x.z, __uint_as_float(r[4 * v + 2]));
                acc[4 * v + 3] = __fadd_rn(x.w, __uint_as_float(r[4 * v + 3]));
            }
            mbar_arrive_cluster(empty_bar, rank - 1u);  // the predecessor may refill this buffer
        }
        if (rank < last) {
            if (!wait_bounded<true>(empty_bar, phase ^ 1u, ctl)) return false;  // the successor read the last chunk
            const uint32_t dst = mapa_shared(buf + lane * 16u, rank + 1u);
#pragma unroll
            for (int v = 0; v < 8; ++v)
                st_shared_cluster_v4(dst + v * 512u, __float_as_uint(acc[4 * v]), __float_as_uint(acc[4 * v + 1]),
                                     __float_as_uint(acc[4 * v + 2]), __float_as_uint(acc[4 * v + 3]));
            mbar_arrive_cluster(full_bar, rank + 1u);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(acc[j]);
            out.put(p, tmC, row0, col0 + c, r);
        }
        phase ^= 1u;
    }
    return true;
}

// kCS: launched as cs x 1 clusters (a runtime launch attribute, cs =
// p.csplit), the CTAs of a cluster splitting each tile's K range and
// chaining their partial sums through distributed shared memory
// (drain_cs).
template <int BN, int kOut, int kLayout, bool kF8 = false, bool kCS = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_sm103_1sm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
    using TS = TileShape<BN>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const int S = p.stages;

    const uint32_t epi_smem = base + S * TS::kStageBytes;  // output staging
    const uint32_t cs_buf = epi_smem + epi_smem_bytes<kOut>();  // cluster-split exchange
    const uint32_t cs_bars = cs_buf + kCsBufBytes;
    const uint32_t bars = cs_buf + (kCS ? kCsBytes : 0u);
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
    auto tfull_bar = [&](int a) { return bars + 8u * (2 * S + a); };
    auto tempty_bar = [&](int a) { return bars + 8u * (2 * S + 2 + a); };
    const uint32_t drain_bar = bars + 8u * (2 * S + 4);
    uint8_t* misc = base_ptr + (bars - base) + 8u * (2 * S + 5);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

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
        if constexpr (kCS) {
            for (int w = 0; w < 4; ++w) mbar_init(cs_bars + 8u * w, 128);  // every lane of a warpgroup
        }
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmC);
    }
    if (warp == 1) tmem_alloc<1>(smem_u32(tmem_holder), TS::kTmemCols);
    tc_fence_before();
    __syncthreads();
    if constexpr (kCS) cluster_sync();  // every CTA's barriers initialised before any uses them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
    // work slot and, for the cluster split, this CTA's half of every tile's K
    const uint32_t cs_rank = kCS ? cluster_ctarank() : 0u;
    const int cs = kCS ? p.csplit : 1;
    if constexpr (kCS) {
        // a CTA that gives up sets its chain neighbours' abort flags
        const uint32_t me = smem_u32(const_cast<int*>(abort_flag));
        const bool has_prev = cs_rank > 0, has_next = static_cast<int>(cs_rank) + 1 < cs;
        const uint32_t next = has_next ? mapa_shared(me, cs_rank + 1u) : 0u;
        ctl.peer_abort[0] = has_prev ? mapa_shared(me, cs_rank - 1u) : next;
        ctl.peer_abort[1] = next;
        ctl.npeers = (has_prev ? 1 : 0) + (has_next ? 1 : 0);
    }
    const int64_t slot = blockIdx.x / cs;
    const int64_t nslots = gridDim.x / cs;
    auto next_unit = [&](int64_t j, Unit& un) -> bool {
        if (!unit_at(p, slot, nslots, j, un)) return false;
        if constexpr (kCS) {
            un.kb0 = static_cast<int>(static_cast<int64_t>(cs_rank) * p.kblocks / cs);
            un.kb1 = static_cast<int>(static_cast<int64_t>(cs_rank + 1) * p.kblocks / cs);
        }
        return true;
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        // (lane 0 alone runs the loop; the warp reconverges below)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t outstanding = 0, out_parity = 0;  // loads issued, per slot
            bool skip = (p.debug_flags & 1) && blockIdx.x == 0;
            bool ok = true;
            for (int64_t j = 0; ok; ++j) {
                Unit un;
                if (!next_unit(j, un)) break;
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
                        skip = false;  // leave this slot's full barrier unsignalled
                    } else {
                        const uint32_t a_dst = base + stage * TS::kStageBytes;
                        mbar_arrive_expect_tx(full_bar(stage), TS::kStageBytes);
                        load_slice<kLayout, BN, false, kF8>(a_dst, a_dst + TS::kABytes, &tmA, &tmB, full_bar(stage), kb,
                                                       un.tm * kBM, un.tn * BN);
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
            for (int64_t j = 0; ok; ++j) {
                Unit un;
                if (!next_unit(j, un)) break;
                if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, ctl)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * TS::kAccCols;
                for (int kb = un.kb0; kb < un.kb1; ++kb) {
                    if (!wait_bounded(full_bar(stage), phase, ctl)) {
                        ok = false;
                        break;
                    }
                    // (TMA-written operands are visible to the MMA once the
                    // full barrier completes; no tcgen05 fence is needed.)
                    const uint32_t a_addr = base + stage * TS::kStageBytes;
                    mma_slice<kLayout, 1, kF8>(d_tmem, a_addr, a_addr + TS::kABytes, p.idesc, kb > un.kb0 ? 1u : 0u);
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
        const int e = warp - 2;              // epilogue warp 0..7
        const int c_begin = (e >> 2) * (BN / 2);  // warpgroup e/4 drains this half of the columns
        const int etid = threadIdx.x - 64;   // 0..255
        const int row_local = q * 32 + lane;
        CStager<kOut> out{epi_smem + static_cast<uint32_t>(e) * 2u * epi_buf_bytes<kOut>(), 0u, lane};
        int acc = 0;
        uint32_t acc_phase = 0;
        const EpiAux aux{static_cast<int64_t>(blockIdx.x), 1};
        const int wg = e >> 2;
        const uint32_t cs_mine = cs_buf + static_cast<uint32_t>(wg) * (kCsBufBytes / 2) + static_cast<uint32_t>(q) * 4096u;
        uint32_t cs_phase = 0;
        for (int64_t j = 0;; ++j) {
            Unit un;
            if (!next_unit(j, un)) break;
            const int tm = un.tm;
            prefetch_sk_partials<BN>(p, un, aux, etid);
            int ok = 1;
            if (lane == 0) ok = wait_bounded(tfull_bar(acc), acc_phase, ctl) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            __syncwarp();
            tc_fence_after();
            const int row0 = tm * kBM + q * 32;
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * TS::kAccCols;
            auto release = [&]() {
                tc_fence_before();
                mbar_arrive(tempty_bar(acc));
            };
            if constexpr (kCS) {
                if (!drain_cs<BN, kOut>(p, &tmC, out, un, tbase, row0, lane, c_begin, cs_rank, cs_mine,
                                        cs_bars + 8u * wg, cs_bars + 8u * (2 + wg), cs_phase, ctl, release))
                    break;
            } else {
                drain_unit<BN, kOut>(p, &tmC, out, un, tbase, row0, row_local, un.slot, aux, c_begin, release);
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        out.drain();  // this warp's output stores have read shared memory
    }

    // ------------------------------------------------------------ exit --
    // A non-aligned barrier: it counts threads one by one, so warps whose
    // lane 0 ran a role loop alone may arrive in any convergence state.
    tc_fence_before();
    cta_barrier_any();
    // (cluster split: no CTA leaves while another may still write into or
    // read its shared memory)
    if constexpr (kCS) cluster_barrier_any();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc<1>(tmem_base, TS::kTmemCols);
    }
}

}  // namespace tsg
