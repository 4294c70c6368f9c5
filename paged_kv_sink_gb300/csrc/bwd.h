// Host interface of the backward kernels (bwd.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>

namespace attn {
namespace bwd {

// Validated arguments of attn_sink_bwd.
struct Args {
    const void* q;
    const void* k;
    const void* v;
    const float* sink;
    const void* out;
    const float* lse;
    const void* dout;
    const int32_t* cu_q;
    const int32_t* cu_k;
    void* dq;
    void* dk;
    void* dv;
    float* dsink;
    int batch, total_q, total_k, hq, hkv, head_dim, max_seqlen_q, max_seqlen_k, win_first, win_last, causal;
    float scale;
    // Row strides in elements of q, k, v (inputs) and dq, dk, dv (outputs); 0 means
    // contiguous rows (heads * 64).  With any output stride set, dk/dv rows past
    // cu_seqlens_k[batch] are left untouched instead of zeroed.
    long long q_rs = 0, k_rs = 0, v_rs = 0, dq_rs = 0, dk_rs = 0, dv_rs = 0;
};

size_t workspace_bytes(const Args& a);
cudaError_t launch(const Args& a, void* workspace, size_t ws_bytes, cudaStream_t s, std::string* what);
int status_exchange(cudaStream_t s, int* host_bits);

}  // namespace bwd
}  // namespace attn
