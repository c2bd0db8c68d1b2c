// host_util.h -- host-side helpers shared by the libdspark translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

constexpr size_t kMaxSmem = 227 * 1024;  // opt-in dynamic shared memory per block on sm_103a

cudaError_t device_sm_count(int* sms);  // multiprocessors of the current device (cached)
// Raises the kernel's dynamic shared-memory limit to `smem` (once per device and kernel) and
// returns its co-resident blocks per SM at (threads, smem); both cached per device.
cudaError_t prepare_kernel(const void* fn, size_t smem, int threads, int* per_sm);
// Co-resident clusters of `cs` blocks of (threads, smem) for `fn` (its shared-memory limit must
// already be raised); cached per device.  *n = 0 when the shape cannot launch.
cudaError_t max_active_clusters(const void* fn, int cs, int threads, size_t smem, int* n);
uint64_t wait_limit_ns();               // bound of every grid-wide wait

dspark_status validate_sample_params(const dspark_sample_params* p);
size_t sample_workspace_bytes(const dspark_sample_params* p);
bool markov_use_mma(const dspark_sample_params* p);

}  // namespace dspark
