// Host interface of the bounded-wait self-test (selftest.cu).
#pragma once

#include <cuda_runtime.h>

namespace attn {
namespace selftest {

cudaError_t launch_wait(int complete, cudaStream_t s);
int status_exchange(cudaStream_t s, int* host_bits);

}  // namespace selftest
}  // namespace attn
