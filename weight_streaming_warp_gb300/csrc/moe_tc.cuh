// moe_tc.cuh -- the forms of the grouped q8_0 MoE mat-vec that wsw_moe_gemv_q8_0 (moe_cc.cu)
// dispatches to besides its own: the tensor-core form (moe_tc.cu) for many routed rows
// and the gathered dense form (gemv_q8_0.cu) for a few.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

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
    void *ws;         // caller workspace (the prepass's sorted activations), or NULL
    size_t ws_bytes;
};

// Workspace bytes of the tensor-core form for these sizes.
size_t moe_q8_tc_workspace_bytes(int64_t E, int64_t K, int64_t R);

// Whether the tensor-core path can take this problem (it needs the workspace).
bool moe_q8_tc_supported(const MoeTcArgs &a);

// Launch it (a prepass, then one persistent CTA per SM); returns a wsw_status.
int moe_q8_tc_launch(const MoeTcArgs &a, int sm_count, cudaStream_t s, bool pdl);

// The form for a few routed rows (gemv_q8_0.cu): a dense mat-vec over R * Mo gathered
// rows, each bit-identical to wsw_gemv_q8_0 on its expert.
bool moe_q8_gather_takes(int64_t R);
int moe_q8_gather_launch(const int8_t *Wq, const uint16_t *Wd, int64_t E, int64_t Mo, int64_t K, const int8_t *xq,
                         const uint16_t *xd, const int32_t *ids, int64_t R, float *y, int32_t *err, const Opts &o,
                         const DeviceInfo &di, cudaStream_t s);

}  // namespace wsw
