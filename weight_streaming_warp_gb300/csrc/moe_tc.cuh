// moe_tc.cuh -- the tensor-core form of the grouped q8_0 MoE mat-vec (moe_tc.cu), used
// by wsw_moe_gemv_q8_0 for problems with many rows.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace wsw {

struct MoeTcArgs {
    const int8_t *Wq;
    const uint16_t *Wd;
    int64_t E, Mo, K;
    const int8_t *xq;
    const uint16_t *xd;
    const int32_t *ids;
    int64_t R;
    float *y;
    int32_t *err;
};

// Whether the tensor-core path can take this problem.
bool moe_q8_tc_supported(int64_t E, int64_t Mo, int64_t K, int64_t R, const void *Wq, const void *Wd,
                         const void *xq, const void *xd);

// Launch it (one persistent CTA per SM); returns a wsw_status.
int moe_q8_tc_launch(const MoeTcArgs &a, int sm_count, cudaStream_t s, bool pdl);

}  // namespace wsw
