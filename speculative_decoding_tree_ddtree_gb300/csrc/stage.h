// stage.h -- host entry point of the host-resident page staging.
#pragma once

#include <cuda_runtime.h>

#include "lucetree.h"

namespace lucetree {

// host_k_dev / host_v_dev: the device-visible addresses of the page-locked host pools
cudaError_t launch_stage_pages(const lucetree_stage_args& a, const void* host_k_dev, const void* host_v_dev,
                               cudaStream_t stream);

}  // namespace lucetree
