// delta.h -- host entry points of the tree-aware recurrent-state (delta rule) step.
#pragma once

#include <cuda_runtime.h>

#include "lucetree.h"

namespace lucetree {

size_t delta_tree_smem_bytes(int N);  // dynamic shared memory of the tree pass
cudaError_t launch_delta_tree(const lucetree_delta_args& a, cudaStream_t stream);
cudaError_t launch_delta_commit(const lucetree_delta_args& a, cudaStream_t stream);

}  // namespace lucetree
