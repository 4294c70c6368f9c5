// Host interface of the pipelined host-buffer forward (host_io.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>

namespace attn {
namespace hostio {

// Validated arguments; every pointer is host memory.
struct Args {
    const void* q;
    const void* k;
    const void* v;
    const float* sink;
    const int32_t* cu_q;  // (batch+1), host
    const int32_t* cu_k;
    void* out;
    float* lse;
    int batch, total_q, total_k, hq, hkv, head_dim, win_first, win_last, causal;
    float scale;
};

size_t scratch_bytes(const Args& a);
cudaError_t run(const Args& a, void* dev_buf, cudaStream_t caller, std::string* what);

}  // namespace hostio
}  // namespace attn
