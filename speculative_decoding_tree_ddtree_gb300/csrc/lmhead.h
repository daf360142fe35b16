// lmhead.h -- host entry points of the fused lm_head projection + argmax.
#pragma once

#include <cuda_runtime.h>

#include "lucetree.h"

namespace lucetree {

int lmhead_padded_rows(int rows);  // -1 when rows exceeds the largest instantiation (256)
size_t lmhead_workspace_bytes(int rows);
cudaError_t launch_lmhead(const lucetree_lmhead_args& a, void* ws, cudaStream_t stream);

}  // namespace lucetree
