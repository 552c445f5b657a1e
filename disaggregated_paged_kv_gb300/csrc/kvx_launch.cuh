// kvx_launch.cuh -- the launch used for every libkvx kernel that runs behind another.
#pragma once

#include <cuda_runtime.h>

namespace kvx {

// Launches fn (smem bytes of dynamic shared memory) with programmatic stream serialization:
// the kernel may start while its predecessor on the stream drains, and orders itself after it
// with griddepcontrol.wait.  Where the attribute is refused, the kernel is launched in plain
// stream order.
cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, void **args, cudaStream_t s,
                       size_t smem = 0);

}  // namespace kvx
