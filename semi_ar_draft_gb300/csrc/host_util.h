// host_util.h -- host-side helpers shared by the libdspark translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

constexpr size_t kMaxSmem = 227 * 1024;  // opt-in dynamic shared memory per block on sm_103a

cudaError_t device_sm_count(int* sms);  // multiprocessors of the current device (cached)
uint64_t wait_limit_ns();               // bound of every grid-wide wait

dspark_status validate_sample_params(const dspark_sample_params* p);
size_t sample_workspace_bytes(const dspark_sample_params* p);
bool markov_use_mma(const dspark_sample_params* p);

}  // namespace dspark
