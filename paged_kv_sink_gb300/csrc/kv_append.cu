// Writes new tokens' K/V rows into a paged cache (sm_103a).
//
// What it computes: the cache update that precedes attention when the cache is
// paged (flash-attention PR "feat: Implement Sink Attention", Description: the
// KV-cache decode path with a sink; sglang PR "To implement attention-sink",
// suggested code: a request's tokens are reached through its page-table row).
// Request b has n_b new rows and seqlens[b] counts them, so they are its logical
// tokens L_b - n_b .. L_b - 1; token t lives at physical slot
// page_table[b][t / page_size] * page_size + t % page_size.
//
// One block per (request, 8 new rows); each row (Hkv * d bf16) is moved with
// 16-byte loads and stores.  A slot outside the cache or a request with fewer
// tokens than new rows raises a device status bit and skips the row, and so
// does a request with more new rows than the grid covers (max_new).
#include "common.cuh"
#include "kv_append.h"

namespace attn {
namespace kvappend {

constexpr int kRowsPerBlock = 8;
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) kv_append_kernel(const uint4* __restrict__ k_new,
                                                             const uint4* __restrict__ v_new,
                                                             const int32_t* __restrict__ cu_new,
                                                             const int32_t* __restrict__ seqlens,
                                                             const int32_t* __restrict__ page_table, int max_pages,
                                                             int page_size, int num_pages, int vec_per_row,
                                                             uint4* __restrict__ k_cache, uint4* __restrict__ v_cache) {
    const int b = blockIdx.y;
    const int n0 = cu_new ? cu_new[b] : b;
    const int n = cu_new ? cu_new[b + 1] - n0 : 1;
    const int L = seqlens[b];
    const int r_begin = blockIdx.x * kRowsPerBlock;
    // The grid covers max_new rows per request; a request with more new rows
    // than that would leave rows unwritten: flag it.
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0 && n > (int)gridDim.x * kRowsPerBlock)
        raise_status(ATTN_SINK_DEV_SEQLEN_OOB);
    for (int idx = threadIdx.x; idx < kRowsPerBlock * vec_per_row; idx += kThreads) {
        const int r = r_begin + idx / vec_per_row;
        const int c = idx % vec_per_row;
        if (r >= n) break;
        const int t = L - n + r;
        if (t < 0 || t / page_size >= max_pages) {
            if (c == 0) raise_status(ATTN_SINK_DEV_SEQLEN_OOB);
            continue;
        }
        const int pg = page_table[(size_t)b * max_pages + t / page_size];
        if (pg < 0 || pg >= num_pages) {
            if (c == 0) raise_status(ATTN_SINK_DEV_PAGE_OOB);
            continue;
        }
        const size_t dst = ((size_t)pg * page_size + t % page_size) * vec_per_row + c;
        const size_t src = (size_t)(n0 + r) * vec_per_row + c;
        k_cache[dst] = k_new[src];
        v_cache[dst] = v_new[src];
    }
}

cudaError_t launch(const Args& a, cudaStream_t s) {
    if (a.batch == 0 || a.max_new <= 0) return cudaSuccess;
    const int vec = a.hkv * a.head_dim / 8;
    dim3 grid((a.max_new + kRowsPerBlock - 1) / kRowsPerBlock, a.batch);
    kv_append_kernel<<<grid, kThreads, 0, s>>>(
        static_cast<const uint4*>(a.k_new), static_cast<const uint4*>(a.v_new), a.cu_new, a.seqlens, a.page_table,
        a.max_pages, a.page_size, a.num_pages, vec, static_cast<uint4*>(a.k_cache), static_cast<uint4*>(a.v_cache));
    return cudaGetLastError();
}

ATTN_DEFINE_STATUS_ACCESSOR(status_exchange)

}  // namespace kvappend
}  // namespace attn
