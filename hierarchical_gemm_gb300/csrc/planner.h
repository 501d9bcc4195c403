// planner.h -- host-side validation and configuration choice for a GEMM
// problem (tile width, split factor, pipeline depth, raster group, grid).
#pragma once

#include <stdint.h>

#include "tsgemm.h"

namespace tsg {

// Shared-memory budget of one CTA on sm_103a (227 KiB opt-in maximum).
constexpr int64_t kSmemPerCtaMax = 232448;

// 8-bit float input formats (E4M3, E5M2).
bool is_8bit(int dtype);

// Bytes per input element (1 or 2).
int64_t in_bytes(int dtype_in);

// K-elements per 128-byte ring slice: 64 (16-bit inputs) or 128 (8-bit).
int slice_k(int dtype_in);

// Validate a problem description without touching a GPU.
tsgemm_status_t validate_problem(int64_t M, int64_t N, int64_t K, int dtype_in, int dtype_out,
                                 int layout);

// Fill *out with the configuration for the problem on a device with
// `num_sms` SMs, honouring every non-zero field of `force` (may be null).
tsgemm_status_t choose_config(int64_t M, int64_t N, int64_t K, int dtype_in, int dtype_out,
                              int layout, int num_sms, const tsgemm_config_t* force,
                              tsgemm_config_t* out);

// Dynamic shared memory per CTA of the kernel for this tile shape (block_m
// 128: one SM per tile; 256: a CTA pair per tile), output type, ring depth
// and cluster split (2: the exchange area of the DSMEM K split).
int64_t smem_bytes_for(int block_m, int block_n, int dtype_out, int stages, int cluster_split = 1);

// Deepest ring that fits the shared-memory budget for this tile shape and
// output type.
int max_stages_for(int block_m, int block_n, int dtype_out, int cluster_split = 1);

}  // namespace tsg
