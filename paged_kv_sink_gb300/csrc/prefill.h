// Host interface of the varlen forward kernel (prefill_fwd.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

namespace attn {
namespace prefill {

// Validated arguments of attn_sink_fwd.
struct FwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* sink;
    const int32_t* cu_q;
    const int32_t* cu_k;
    void* out;
    float* lse;
    int batch, total_q, total_k, hq, hkv, head_dim, max_seqlen_q, max_seqlen_k, win_first, win_last, causal;
    float scale;
    // Paged K/V (page_table != nullptr): k / v are the caches (num_pages, page_size,
    // hkv, d), request b's keys are its first seqlens_k[b] cached tokens and cu_k /
    // total_k are unused.  page_size is a power of two >= 8.
    const int32_t* page_table = nullptr;
    const int32_t* seqlens_k = nullptr;
    int max_pages = 0, page_size = 0, num_pages = 0;
    // Row strides of q, k, v in elements (0: contiguous rows of heads * 64).
    long long q_rs = 0, k_rs = 0, v_rs = 0;
};

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t s, std::string* what);
int status_exchange(cudaStream_t s, int* host_bits);

}  // namespace prefill
}  // namespace attn
