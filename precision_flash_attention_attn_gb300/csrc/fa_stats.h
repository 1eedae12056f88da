// Launch interface of the statistics kernel (pv_err, delta_err), shared by the
// C-ABI layer and fa_stats.cu.
#pragma once

#include "fa_internal.h"

namespace fa {

struct StatsArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* o;     // BF16 or FP32 (mode 2)
    float* pv_err;     // [BH, N]
    const void* dout;  // BF16 [BH, N, d]; read only when delta_err is set
    float* delta_err;  // nullable: [BH, N]
    int BH, N, d, causal, mode;
    float scale;
    int* status;
};

cudaError_t launch_pv_err(const StatsArgs& a, cudaStream_t stream);

struct SplitArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* o;     // BF16 or FP32 (mode 2)
    const void* dout;  // BF16
    float* err_one;    // [BH, N] each
    float* err_rest;
    float* err_out;
    int BH, N, d, causal, mode;
    float scale, beta, eps;
};

cudaError_t launch_delta_split(const SplitArgs& a, cudaStream_t stream);

}  // namespace fa
