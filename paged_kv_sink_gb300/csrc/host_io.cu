// Forward attention on host-resident tensors with the transfers pipelined
// against the kernels (a native runtime piece around the forward kernel).
//
// The batch is processed request by request on library-owned streams:
//   copy-in stream   host -> device rows of request r (q, k, v)
//   compute streams  the forward kernel of request r (two streams, alternating,
//                    so that the grids of consecutive requests overlap)
//   copy-out stream  device -> host rows of out and lse of request r
// chained with events, so the copies of request r + 1 and of request r - 1
// overlap the kernel of request r.  Everything is asynchronous; the caller's
// stream waits for the last copy.  Host buffers should be page-locked
// (cudaHostAlloc / cudaHostRegister): copies from pageable memory are
// synchronous with the host and do not overlap.
#include <mutex>
#include <string>
#include <vector>

#include "attn_sink.h"
#include "common.cuh"
#include "host_io.h"
#include "prefill.h"

namespace attn {
namespace hostio {

namespace {

constexpr int kMaxDevices = 64;

struct Streams {
    cudaStream_t in = nullptr, out = nullptr, comp[2] = {nullptr, nullptr};
};

std::mutex g_mu;
Streams g_streams[kMaxDevices];

cudaError_t device_streams(Streams* s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    Streams& st = g_streams[dev];
    if (!st.in) {
        cudaStream_t t[4];
        for (int i = 0; i < 4; ++i)
            if ((e = cudaStreamCreateWithFlags(&t[i], cudaStreamNonBlocking)) != cudaSuccess) return e;
        st.in = t[0];
        st.out = t[1];
        st.comp[0] = t[2];
        st.comp[1] = t[3];
    }
    *s = st;
    return cudaSuccess;
}

// Events created for one call; destroyed when the call has queued its work
// (a destroyed event that is still pending is released once it completes).
struct Events {
    std::vector<cudaEvent_t> ev;
    cudaError_t make(cudaEvent_t* e) {
        cudaError_t r = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
        if (r == cudaSuccess) ev.push_back(*e);
        return r;
    }
    ~Events() {
        for (cudaEvent_t e : ev) cudaEventDestroy(e);
    }
};

}  // namespace

cudaError_t run(const Args& a, void* dev_buf, cudaStream_t caller, std::string* what) {
    Streams st;
    cudaError_t e = device_streams(&st);
    if (e != cudaSuccess) {
        *what = "streams";
        return e;
    }
    const size_t q_row = (size_t)a.hq * a.head_dim * 2, kv_row = (size_t)a.hkv * a.head_dim * 2;
    char* p = static_cast<char*>(dev_buf);
    auto carve = [&](size_t bytes) {
        char* r = p;
        p += (bytes + 255) & ~size_t(255);
        return r;
    };
    char* dq = carve((size_t)a.total_q * q_row);
    char* dk = carve((size_t)a.total_k * kv_row);
    char* dv = carve((size_t)a.total_k * kv_row);
    char* dout = carve((size_t)a.total_q * q_row);
    float* dlse = reinterpret_cast<float*>(carve((size_t)a.hq * a.total_q * 4));
    float* dsink = a.sink ? reinterpret_cast<float*>(carve((size_t)a.hq * 4)) : nullptr;
    int32_t* dcu_q = reinterpret_cast<int32_t*>(carve((size_t)(a.batch + 1) * 4));
    int32_t* dcu_k = reinterpret_cast<int32_t*>(carve((size_t)(a.batch + 1) * 4));

    Events evs;
    cudaEvent_t ready, meta;
    if ((e = evs.make(&ready)) != cudaSuccess || (e = evs.make(&meta)) != cudaSuccess) {
        *what = "events";
        return e;
    }
    // The scratch was allocated on the caller's stream: every internal stream starts after it.
    if ((e = cudaEventRecord(ready, caller)) != cudaSuccess) return e;
    for (cudaStream_t s : {st.in, st.out, st.comp[0], st.comp[1]})
        if ((e = cudaStreamWaitEvent(s, ready, 0)) != cudaSuccess) return e;

    const char* hq_ = static_cast<const char*>(a.q);
    const char* hk_ = static_cast<const char*>(a.k);
    const char* hv_ = static_cast<const char*>(a.v);
    char* hout = static_cast<char*>(a.out);
    *what = "copy-in";
    if ((e = cudaMemcpyAsync(dcu_q, a.cu_q, (size_t)(a.batch + 1) * 4, cudaMemcpyHostToDevice, st.in)) != cudaSuccess ||
        (e = cudaMemcpyAsync(dcu_k, a.cu_k, (size_t)(a.batch + 1) * 4, cudaMemcpyHostToDevice, st.in)) != cudaSuccess)
        return e;
    if (a.sink && (e = cudaMemcpyAsync(dsink, a.sink, (size_t)a.hq * 4, cudaMemcpyHostToDevice, st.in)) != cudaSuccess)
        return e;
    if ((e = cudaEventRecord(meta, st.in)) != cudaSuccess) return e;

    int launched = 0;
    for (int r = 0; r < a.batch; ++r) {
        const int q0 = a.cu_q[r], q1 = a.cu_q[r + 1], k0 = a.cu_k[r], k1 = a.cu_k[r + 1];
        const int Lq = q1 - q0, Lk = k1 - k0;
        if (Lq <= 0) continue;
        *what = "copy-in";
        if ((e = cudaMemcpyAsync(dq + (size_t)q0 * q_row, hq_ + (size_t)q0 * q_row, (size_t)Lq * q_row,
                                 cudaMemcpyHostToDevice, st.in)) != cudaSuccess)
            return e;
        if (Lk > 0 && ((e = cudaMemcpyAsync(dk + (size_t)k0 * kv_row, hk_ + (size_t)k0 * kv_row, (size_t)Lk * kv_row,
                                            cudaMemcpyHostToDevice, st.in)) != cudaSuccess ||
                       (e = cudaMemcpyAsync(dv + (size_t)k0 * kv_row, hv_ + (size_t)k0 * kv_row, (size_t)Lk * kv_row,
                                            cudaMemcpyHostToDevice, st.in)) != cudaSuccess))
            return e;
        cudaEvent_t in_done, comp_done;
        if ((e = evs.make(&in_done)) != cudaSuccess || (e = evs.make(&comp_done)) != cudaSuccess) {
            *what = "events";
            return e;
        }
        if ((e = cudaEventRecord(in_done, st.in)) != cudaSuccess) return e;
        cudaStream_t cs = st.comp[launched & 1];
        ++launched;
        if ((e = cudaStreamWaitEvent(cs, meta, 0)) != cudaSuccess || (e = cudaStreamWaitEvent(cs, in_done, 0)) != cudaSuccess)
            return e;
        prefill::FwdArgs f = {};
        f.q = dq;
        f.k = dk;
        f.v = dv;
        f.sink = dsink;
        f.cu_q = dcu_q + r;  // this request alone: cu[r], cu[r + 1] are absolute row offsets
        f.cu_k = dcu_k + r;
        f.out = dout;
        f.lse = a.lse ? dlse : nullptr;
        f.batch = 1;
        f.total_q = a.total_q;  // also the lse head stride
        // K/V rows past this request are out of the tensor for this launch (the
        // copy engine may still be writing them): the tail tile reads zeros.
        f.total_k = k1;
        f.hq = a.hq;
        f.hkv = a.hkv;
        f.head_dim = a.head_dim;
        f.max_seqlen_q = Lq;
        f.max_seqlen_k = Lk;
        f.win_first = a.win_first;
        f.win_last = a.win_last;
        f.causal = a.causal;
        f.scale = a.scale;
        if ((e = prefill::launch_fwd(f, cs, what)) != cudaSuccess) return e;
        if ((e = cudaEventRecord(comp_done, cs)) != cudaSuccess) return e;
        *what = "copy-out";
        if ((e = cudaStreamWaitEvent(st.out, comp_done, 0)) != cudaSuccess) return e;
        if ((e = cudaMemcpyAsync(hout + (size_t)q0 * q_row, dout + (size_t)q0 * q_row, (size_t)Lq * q_row,
                                 cudaMemcpyDeviceToHost, st.out)) != cudaSuccess)
            return e;
        if (a.lse && (e = cudaMemcpy2DAsync(a.lse + q0, (size_t)a.total_q * 4, dlse + q0, (size_t)a.total_q * 4,
                                            (size_t)Lq * 4, a.hq, cudaMemcpyDeviceToHost, st.out)) != cudaSuccess)
            return e;
    }
    // The caller's stream (and the release of the scratch on it) waits for every copy.
    *what = "join";
    for (cudaStream_t s : {st.in, st.out, st.comp[0], st.comp[1]}) {
        cudaEvent_t j;
        if ((e = evs.make(&j)) != cudaSuccess) return e;
        if ((e = cudaEventRecord(j, s)) != cudaSuccess || (e = cudaStreamWaitEvent(caller, j, 0)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

size_t scratch_bytes(const Args& a) {
    auto r = [](size_t b) { return (b + 255) & ~size_t(255); };
    const size_t q_row = (size_t)a.hq * a.head_dim * 2, kv_row = (size_t)a.hkv * a.head_dim * 2;
    return 2 * r((size_t)a.total_q * q_row) + 2 * r((size_t)a.total_k * kv_row) + r((size_t)a.hq * a.total_q * 4) +
           r((size_t)a.hq * 4) + 2 * r((size_t)(a.batch + 1) * 4);
}

}  // namespace hostio
}  // namespace attn
