// Shared device helpers for the attention-with-sink kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "attn_sink.h"

#define ATTN_LOG2E 1.4426950408889634f
#define ATTN_LN2 0.6931471805599453f

namespace attn {

// Sticky device status word (ATTN_SINK_DEV_* bits).  Each translation unit
// has its own copy (no relocatable device code is needed); the host side ORs
// them together through the accessor each unit defines with
// ATTN_DEFINE_STATUS_ACCESSOR.
static __device__ int g_dev_status;

__device__ __forceinline__ void raise_status(int bits) { atomicOr(&g_dev_status, bits); }

// Defines `int fn(cudaStream_t s, int* bits)`: adds this unit's status bits
// to *bits and clears them (stream-ordered; the caller synchronises).
#define ATTN_DEFINE_STATUS_ACCESSOR(fn)                                              \
    int fn(cudaStream_t s, int* host_bits) {                                         \
        int v = 0;                                                                   \
        cudaError_t e = cudaMemcpyFromSymbolAsync(&v, attn::g_dev_status, sizeof(int), 0, \
                                                  cudaMemcpyDeviceToHost, s);       \
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);                          \
        if (e != cudaSuccess) return (int)e;                                         \
        *host_bits |= v;                                                             \
        int zero = 0;                                                                \
        e = cudaMemcpyToSymbolAsync(attn::g_dev_status, &zero, sizeof(int), 0,       \
                                    cudaMemcpyHostToDevice, s);                      \
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);                          \
        return (int)e;                                                               \
    }

// Nanosecond wall clock of the GPU.
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Every spin-wait in this library gives up after this long and raises
// ATTN_SINK_DEV_TIMEOUT instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Visible key set of a query at absolute position `pos` (sglang PR "To
// implement attention-sink": first window [0, F) and last window [p+1-W, p+1),
// per sequence).  Returns the two disjoint increasing ranges [a0,b0), [a1,b1).
// win_last <= 0: plain causal, [0, pos+1).
struct Ranges {
    int a0, b0, a1, b1;
};

__host__ __device__ __forceinline__ Ranges visible_ranges(int pos, int win_first, int win_last) {
    Ranges r;
    int n = pos + 1 > 0 ? pos + 1 : 0;  // tokens at positions <= pos
    r.a0 = 0;
    if (win_last <= 0) {
        r.b0 = n;
        r.a1 = n;
        r.b1 = n;
        return r;
    }
    int first_end = win_first < n ? win_first : n;
    if (first_end < 0) first_end = 0;
    int last_begin = n - win_last;
    if (last_begin < first_end) last_begin = first_end;
    r.b0 = first_end;
    r.a1 = last_begin;
    r.b1 = n;
    return r;
}

// Maps the v-th visible token (0-based, in increasing position order) to its
// logical position.
__host__ __device__ __forceinline__ int visible_token(const Ranges& r, int v) {
    int n0 = r.b0 - r.a0;
    return v < n0 ? r.a0 + v : r.a1 + (v - n0);
}

__host__ __device__ __forceinline__ int visible_count(const Ranges& r) {
    return (r.b0 - r.a0) + (r.b1 - r.a1);
}

}  // namespace attn
