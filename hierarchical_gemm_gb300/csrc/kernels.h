// kernels.h -- host-visible handles to the compiled GEMM kernels.
#pragma once

#include <stdint.h>

namespace tsg {

// Kernel entry for a tile width (64/128/192/256), output kind (0 fp16,
// 1 bf16, 2 fp32), operand layout (tsgemm_layout_t), input width (in8:
// 8-bit float inputs, RCR layout only) and cluster split (cs = 2, 4 or 8:
// launched as cs x 1 clusters splitting each tile's K; RRR, 16-bit
// inputs); null for an unsupported combination.
const void* kernel_1sm(int block_n, int out_kind, int layout, bool in8, int cs);

// Dynamic shared memory the kernel above uses with `stages` ring slots.
int64_t kernel_1sm_smem_bytes(int block_n, int out_kind, int stages, int cs);

// The CTA-pair kernel (256 x block_n tiles, block_n 128 or 256), launched
// as 2 x 1 clusters; null for an unsupported combination.
const void* kernel_2sm(int block_n, int out_kind, int layout, bool in8);

// Dynamic shared memory per CTA of the pair kernel with `stages` slots.
int64_t kernel_2sm_smem_bytes(int block_n, int out_kind, int stages);

// Per-layout tables (one translation unit each).
const void* kernel_1sm_layout0(int block_n, int out_kind);
const void* kernel_1sm_layout1(int block_n, int out_kind);
const void* kernel_1sm_layout2(int block_n, int out_kind);
const void* kernel_1sm_layout3(int block_n, int out_kind);
const void* kernel_2sm_layout0(int block_n, int out_kind);
const void* kernel_2sm_layout1(int block_n, int out_kind);
const void* kernel_2sm_layout2(int block_n, int out_kind);
const void* kernel_2sm_layout3(int block_n, int out_kind);
const void* kernel_1sm_f8(int block_n, int out_kind);
const void* kernel_1sm_cs(int block_n, int out_kind);
const void* kernel_2sm_f8(int block_n, int out_kind);

}  // namespace tsg
