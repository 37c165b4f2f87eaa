// gsample.h -- launch-side view of the one-pass Gumbel-max draft-sampling
// kernel (stream_kernels.cu): its entry point per dtype (0 float32, 1
// bf16), threads per CTA, largest cluster and dynamic shared-memory bytes.
#pragma once

#include <cstdint>

namespace mtp {

const void *gsample_kernel(int dtype);
int gsample_threads();
int gsample_max_cluster();
uint32_t gsample_smem_bytes();

}  // namespace mtp
