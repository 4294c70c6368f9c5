// Host interface of the paged-cache append kernel (kv_append.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {
namespace kvappend {

struct Args {
    const void* k_new;          // (rows, hkv, d) bf16
    const void* v_new;
    const int32_t* cu_new;      // (batch+1) device; nullptr: one new row per request (row b)
    const int32_t* seqlens;     // (batch) device, cache length including the new rows
    const int32_t* page_table;  // (batch, max_pages) device
    void* k_cache;              // (num_pages, page_size, hkv, d) bf16
    void* v_cache;
    int max_pages, batch, hkv, head_dim, page_size, num_pages;
    int max_new;                // host bound on the new rows of one request
};

cudaError_t launch(const Args& a, cudaStream_t s);
int status_exchange(cudaStream_t s, int* host_bits);

}  // namespace kvappend
}  // namespace attn
