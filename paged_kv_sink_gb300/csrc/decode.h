// Host/device interface of the paged decode kernels (decode.cu).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include "attn_sink.h"

namespace attn {
namespace decode {

// Kernel parameters of the split and combine kernels.
struct SplitParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k_cache;
    const __nv_bfloat16* v_cache;
    const int32_t* page_table;
    const int32_t* seqlens;
    float* part_o;    // (batch, hq, max_splits, head_dim) fp32, un-normalised
    float2* part_ml;  // (batch, hq, max_splits): (running max in log2 units, sum)
    int max_pages, hq, hkv, page_size, num_pages, win_first, win_last;
    int split_tokens, max_splits, hblocks, group;
    int page_shift;    // log2(page_size) when it is a power of two, else -1
    float scale_log2;  // softmax scale * log2(e)
};

// Validated arguments of attn_sink_decode_paged.
struct Args {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* page_table;
    const int32_t* seqlens;
    const float* sink;
    void* out;
    float* lse;
    int max_pages, batch, hq, hkv, head_dim, page_size, num_pages, win_first, win_last, group;
    float scale;
};

// Split-KV work decomposition and scratch sizes.
struct Plan {
    int nt;            // 8-head groups per CTA (1 or 2)
    int hblocks;       // CTAs per KV head along the query-head axis
    int split_tokens;  // visible tokens per split
    int max_splits;    // splits of the longest possible request
    long long nvis_max;  // visible tokens of the longest possible request
    size_t part_o_bytes, part_ml_bytes;
};

Plan make_plan(const Args& a);
cudaError_t launch(const Args& a, const Plan& pl, float* part_o, float2* part_ml, cudaStream_t s);
cudaError_t launch_visible_ranges(const int32_t* seqlens, int batch, int win_first, int win_last,
                                  int32_t* ranges, cudaStream_t s);
cudaError_t launch_visible_slots(const int32_t* seqlens, const int32_t* page_table, int max_pages,
                                 int batch, int page_size, int num_pages, int win_first, int win_last,
                                 int32_t* slots, int max_visible, cudaStream_t s);
int status_exchange(cudaStream_t s, int* host_bits);

}  // namespace decode

void record_error(const char* msg);

// Argument checks of the paged decode entry points (api.cu); `who` prefixes the
// error text.  Returns an ATTN_SINK_* status and records the error text.
int validate_decode(const char* who, const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache,
                    const int32_t* page_table, int max_pages, const int32_t* seqlens, int batch, int hq,
                    int hkv, int head_dim, int page_size, int num_pages, int win_first, attn_bf16* out);
// The softmax scale: `scale` if positive, else 1/sqrt(head_dim).
float resolve_scale(float scale, int head_dim);

}  // namespace attn
