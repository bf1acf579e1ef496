// gs_project_variants.h -- launchers of the projection and its chain rule for
// SH coefficients stored as bfloat16 (gs_project_sh16, gs_project_bwd_sh16),
// and of the chain rule fused with an Adam step (gs_project_bwd_adam).  Not
// part of the C ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gs_internal.h"

namespace gs {

cudaError_t launch_project_sh16(const CamParams& cam, int64_t n, int sh_degree, const float* means,
                                const float* scales, const float* quats, const float* opacities,
                                const uint16_t* sh, float* splats, float* depths, int32_t* radii,
                                int32_t* tiles_touched, cudaStream_t st);
cudaError_t launch_project_bwd_sh16(const CamParams& cam, int64_t n, int sh_degree,
                                    const float* means, const float* scales, const float* quats,
                                    const float* opacities, const uint16_t* sh,
                                    const int32_t* tiles_touched, const float* grad2d,
                                    const uint8_t* touched, float* dmeans, float* dscales,
                                    float* dquats, float* dopacities, float* dsh, cudaStream_t st);

// One Adam step on the raw parameters, fused into the chain rule: p[] are
// updated in place, m[] / v[] are the moments (same layouts as the parameters:
// means, log-scales, quaternions, opacity logits, SH).  c1 = 1 / (1 - beta1^t),
// c2 = 1 / (1 - beta2^t).  act_scales / act_opacities, when set, receive the
// activated values of the updated parameters (the next forward's inputs).
struct AdamArgs {
    float* p[5];
    float* m[5];
    float* v[5];
    float lr[6];  // means, scales, quaternions, opacities, SH band 0, SH bands 1-3
    float b1, b2, eps, c1, c2;
    float* act_scales;     // optional: exp(log-scales) after the step
    float* act_opacities;  // optional: sigmoid(logits) after the step
};

cudaError_t launch_project_bwd_adam(const CamParams& cam, int64_t n, int sh_degree,
                                    const int32_t* tiles_touched, const float* grad2d,
                                    const uint8_t* touched, const AdamArgs& adam, cudaStream_t st);

}  // namespace gs
