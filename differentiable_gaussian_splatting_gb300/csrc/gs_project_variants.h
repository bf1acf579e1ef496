// gs_sh16.h -- launchers of the projection and its chain rule for SH
// coefficients stored as bfloat16 (gs_project_sh16, gs_project_bwd_sh16).
// Not part of the C ABI.
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

}  // namespace gs
