// Allocation-free variant of paged decode.
//
// attn_sink_decode_paged takes its split-KV scratch (per-split partial
// outputs and softmax statistics) from a stream-ordered memory pool.  Some
// callers cannot allocate device memory at call time: a serving engine that
// reserved the whole device up front and forbids further cudaMalloc, code
// that must not take the allocator's locks or implicit synchronisation on a
// latency-critical path, or an embedding that only hands the library
// pre-existing buffers.  For them, attn_sink_decode_paged_noalloc runs the
// same decode kernels with the scratch placed in one fixed device array that
// lives as long as the library is loaded.
#include <math.h>
#include <stdio.h>

#include <algorithm>
#include <mutex>
#include <string>

#include "attn_sink.h"
#include "common.cuh"
#include "decode.h"

namespace {

// 32 MiB of scratch.  A GPU holds it from the moment this library's module is
// loaded on it (at the latest, this entry point's first call there) until
// the process exits.
constexpr size_t kScratchBytes = 32ull << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device, looked up once
// per device (the host-side symbol is only a stand-in, never a device address).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

int attn_sink_decode_paged_noalloc(const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache,
                                   const int32_t* page_table, int max_pages, const int32_t* seqlens,
                                   int batch, int hq, int hkv, int head_dim, int page_size, int num_pages,
                                   const float* sink, int win_first, int win_last, float scale,
                                   attn_bf16* out, float* lse, void* stream) {
    attn::record_error("");
    auto fail = [](int code, const char* msg) {
        attn::record_error(msg);
        return code;
    };
    int rc = attn::validate_decode("decode_noalloc", q, k_cache, v_cache, page_table, max_pages, seqlens, batch, hq,
                                   hkv, head_dim, page_size, num_pages, win_first, out);
    if (rc != ATTN_SINK_OK || batch == 0) return rc;

    attn::decode::Args a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.page_table = page_table;
    a.seqlens = seqlens;
    a.sink = sink;
    a.out = out;
    a.lse = lse;
    a.max_pages = max_pages;
    a.batch = batch;
    a.hq = hq;
    a.hkv = hkv;
    a.head_dim = head_dim;
    a.page_size = page_size;
    a.num_pages = num_pages;
    a.win_first = win_first;
    a.win_last = win_last;
    a.group = hq / hkv;
    a.scale = attn::resolve_scale(scale, head_dim);

    // Same work split as the allocating entry point; when its partials do not
    // fit, use fewer, longer splits (the result differs only by rounding).
    attn::decode::Plan pl = attn::decode::make_plan(a);
    auto need = [&](const attn::decode::Plan& p) {
        const size_t o = (p.part_o_bytes + 255) & ~size_t(255);
        return o + p.part_ml_bytes;
    };
    // Longer splits: double the split length, but never past the longest request
    // (rounded to whole 64-token chunks, and kept below 2^31 tokens).
    const long long cap = std::min((pl.nvis_max + 63) / 64 * 64, (1LL << 31) - 64);
    while (need(pl) > kScratchBytes && pl.max_splits > 1) {
        const long long st = std::min(2LL * pl.split_tokens, cap);
        if (st == pl.split_tokens) break;  // already one split per request (or at the cap)
        pl.split_tokens = (int)st;
        pl.max_splits = (int)((pl.nvis_max + st - 1) / st);
        pl.part_o_bytes = (size_t)batch * hq * pl.max_splits * head_dim * sizeof(float);
        pl.part_ml_bytes = (size_t)batch * hq * pl.max_splits * sizeof(float2);
    }
    char msg[256];
    if (need(pl) > kScratchBytes) {
        snprintf(msg, sizeof(msg),
                 "decode_noalloc: batch*hq*head_dim needs %zu bytes of scratch, more than the %zu-byte "
                 "static array; use attn_sink_decode_paged",
                 need(pl), kScratchBytes);
        return fail(ATTN_SINK_ERR_UNSUPPORTED, msg);
    }
    void* base = nullptr;
    cudaError_t e = scratch_address(&base);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof(msg), "decode_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        return fail(ATTN_SINK_ERR_CUDA, msg);
    }
    float* part_o = static_cast<float*>(base);
    float2* part_ml =
        reinterpret_cast<float2*>(static_cast<unsigned char*>(base) + ((pl.part_o_bytes + 255) & ~size_t(255)));
    e = attn::decode::launch(a, pl, part_o, part_ml, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        snprintf(msg, sizeof(msg), "decode_noalloc: launch: %s", cudaGetErrorString(e));
        return fail(ATTN_SINK_ERR_CUDA, msg);
    }
    return ATTN_SINK_OK;
}

}  // extern "C"
