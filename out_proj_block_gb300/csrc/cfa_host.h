// cfa_host.h -- host-side declarations shared between the translation units of
// the library (not part of the public ABI, which is include/cfa.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "cfa.h"

namespace cfa {

// Kernel entry points (cfa_gemv.cu).
const void *gemv_kernel(int mode, int maxb, bool wide);
const void *gemv_mma_kernel_ptr(int mode);
const void *rmsnorm_kernel_ptr();
const void *advance_kernel_ptr();
const void *mla_kernel_ptr(int heads_per_cluster);  // cfa_mla.cu

// The attention plan, seen from the layer stack (cfa_api.cu).
cfa_status plan_encode_layer(const cfa_plan *pl, const void *W_qkv, const void *W_o,
                             CUtensorMap *tm_wqkv, CUtensorMap *tm_wo);
cfa_status plan_encode_input(const cfa_plan *pl, const void *x, CUtensorMap *tm_x);
cfa_status plan_launch_layer(cfa_plan *pl, const CUtensorMap *tm_wqkv, const CUtensorMap *tm_wo,
                             const CUtensorMap *tm_x, const void *x, void *k_cache,
                             void *v_cache, const int *lens_dev, double rope_theta,
                             const void *resid, void *out, cudaStream_t stream);
unsigned *plan_status_word(cfa_plan *pl);
int plan_launches_per_step(const cfa_plan *pl);  // 1, or 2 with the separate head merge

// Tensor map of a row-major bf16 matrix [rows][cols] with [box_rows x
// box_cols] boxes, no swizzle (cfa_api.cu).
cfa_status encode_bf16_2d(CUtensorMap *tm, const void *base, uint64_t cols, uint64_t rows,
                          uint32_t box_cols, uint32_t box_rows);
// Same with an explicit row stride (elements) and optional 128-byte swizzle.
cfa_status encode_bf16_2d_ex(CUtensorMap *tm, const void *base, uint64_t cols, uint64_t rows,
                             uint64_t row_stride, uint32_t box_cols, uint32_t box_rows,
                             bool swizzle128);

// Records s as the calling thread's last error and returns it.
cfa_status set_last_error(cfa_status s);

}  // namespace cfa
