// Forward attention on host-resident tensors with the transfers pipelined
// against the kernels (a native runtime piece around the forward kernel).
//
// The batch is processed in chunks of up to 1024 query rows on library-owned
// streams.  A chunk of rows i0 .. i1 of a request sees only the keys before
// off + i1 (off = Lk - Lq, bottom-right causal alignment), so it runs as a
// one-request forward over those rows and that key prefix, with the same
// alignment, and only the K/V rows its prefix adds have to arrive first:
//   copy-in stream   host -> device: the chunk's q rows and its new k, v rows
//   compute streams  the forward kernel of the chunk (two streams, alternating,
//                    so that the grids of consecutive chunks overlap)
//   copy-out stream  device -> host rows of out and lse of the chunk
// chained with events, so the copies of the next and of the previous chunk
// overlap the kernel of this one, and the first kernel starts after one
// chunk's rows instead of a whole request's.  Requests go in the order
// Johnson's rule gives for the two-stage flow shop copy-in -> kernel (first
// those whose copy-in is shorter than their kernel, by increasing copy-in
// time, then the others by decreasing kernel time).  Everything is
// asynchronous; the caller's stream waits for the last copy.  Host buffers
// should be page-locked (cudaHostAlloc / cudaHostRegister): copies from
// pageable memory are synchronous with the host and do not overlap.
#include <algorithm>
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
constexpr int kChunkRows = 1024;

// One chunk: query rows [qb, qe) and keys [kb, ke) (absolute row offsets).
struct Chunk {
    int qb, qe, kb, ke;
};

// The chunks in processing order (see the file comment).
std::vector<Chunk> plan_chunks(const Args& a) {
    const size_t q_row = (size_t)a.hq * a.head_dim * 2, kv_row = (size_t)a.hkv * a.head_dim * 2;
    // Stage times, estimated from the bytes a request moves in (at ~200 GB/s) and
    // the (query, key) pairs its kernel visits (at ~1.1 PFLOP/s); only their
    // ratios and order matter.
    struct Job {
        int r;
        double in, comp;
    };
    std::vector<Job> jobs;
    for (int r = 0; r < a.batch; ++r) {
        const long long Lq = a.cu_q[r + 1] - a.cu_q[r], Lk = std::max(0, a.cu_k[r + 1] - a.cu_k[r]);
        if (Lq <= 0) continue;
        double pairs = (double)Lq * (double)Lk;
        if (a.causal) {
            const long long off = Lk - Lq;
            pairs = 0.0;
            for (long long i = 0; i < Lq; i += 64) {  // rows i .. i + 63 see about min(Lk, off + i + 32) keys
                const long long n = std::min(64LL, Lq - i);
                pairs += (double)n * (double)std::max(0LL, std::min(Lk, off + i + 32));
            }
        }
        if (a.win_last > 0) pairs = std::min(pairs, (double)Lq * (double)(a.win_first + a.win_last));
        const double bytes_in = (double)Lq * q_row + 2.0 * (double)Lk * kv_row;
        jobs.push_back({r, bytes_in / 200e9, pairs * a.hq * 4.0 * a.head_dim / 1.1e15});
    }
    std::stable_sort(jobs.begin(), jobs.end(), [](const Job& x, const Job& y) {
        const bool fx = x.in <= x.comp, fy = y.in <= y.comp;
        if (fx != fy) return fx;
        return fx ? x.in < y.in : x.comp > y.comp;
    });
    std::vector<Chunk> chunks;
    for (const Job& job : jobs) {
        const int q0 = a.cu_q[job.r], Lq = a.cu_q[job.r + 1] - q0;
        const int k0 = a.cu_k[job.r], Lk = std::max(0, a.cu_k[job.r + 1] - k0);
        for (int i0 = 0; i0 < Lq; i0 += kChunkRows) {
            const int i1 = std::min(Lq, i0 + kChunkRows);
            const int need = a.causal ? std::max(0, std::min(Lk, Lk - Lq + i1)) : Lk;
            chunks.push_back({q0 + i0, q0 + i1, k0, k0 + need});
        }
    }
    return chunks;
}

int count_chunks(const Args& a) {
    int n = 0;
    for (int r = 0; r < a.batch; ++r) {
        const int Lq = a.cu_q[r + 1] - a.cu_q[r];
        if (Lq > 0) n += (Lq + kChunkRows - 1) / kChunkRows;
    }
    return n;
}

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
    const std::vector<Chunk> chunks = plan_chunks(a);
    const int n_chunks = (int)chunks.size();
    // per chunk {q begin, q end, k begin, k end}: the cu_seqlens of its one-request launch
    int32_t* dmeta = reinterpret_cast<int32_t*>(carve((size_t)std::max(1, n_chunks) * 16));

    Events evs;
    cudaEvent_t ready, meta_in;
    if ((e = evs.make(&ready)) != cudaSuccess || (e = evs.make(&meta_in)) != cudaSuccess) {
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
    if (n_chunks > 0 && (e = cudaMemcpyAsync(dmeta, chunks.data(), (size_t)n_chunks * 16, cudaMemcpyHostToDevice,
                                             st.in)) != cudaSuccess)
        return e;
    if (a.sink && (e = cudaMemcpyAsync(dsink, a.sink, (size_t)a.hq * 4, cudaMemcpyHostToDevice, st.in)) != cudaSuccess)
        return e;
    if ((e = cudaEventRecord(meta_in, st.in)) != cudaSuccess) return e;

    int k_have = -1;  // K/V rows of the current request on the device: [kb, k_have)
    for (int c = 0; c < n_chunks; ++c) {
        const Chunk& ch = chunks[c];
        if (c == 0 || chunks[c - 1].kb != ch.kb || chunks[c - 1].qe != ch.qb) k_have = ch.kb;  // a new request
        *what = "copy-in";
        if ((e = cudaMemcpyAsync(dq + (size_t)ch.qb * q_row, hq_ + (size_t)ch.qb * q_row,
                                 (size_t)(ch.qe - ch.qb) * q_row, cudaMemcpyHostToDevice, st.in)) != cudaSuccess)
            return e;
        if (ch.ke > k_have &&
            ((e = cudaMemcpyAsync(dk + (size_t)k_have * kv_row, hk_ + (size_t)k_have * kv_row,
                                  (size_t)(ch.ke - k_have) * kv_row, cudaMemcpyHostToDevice, st.in)) != cudaSuccess ||
             (e = cudaMemcpyAsync(dv + (size_t)k_have * kv_row, hv_ + (size_t)k_have * kv_row,
                                  (size_t)(ch.ke - k_have) * kv_row, cudaMemcpyHostToDevice, st.in)) != cudaSuccess))
            return e;
        k_have = std::max(k_have, ch.ke);
        cudaEvent_t in_done, comp_done;
        if ((e = evs.make(&in_done)) != cudaSuccess || (e = evs.make(&comp_done)) != cudaSuccess) {
            *what = "events";
            return e;
        }
        if ((e = cudaEventRecord(in_done, st.in)) != cudaSuccess) return e;
        cudaStream_t cs = st.comp[c & 1];
        if ((e = cudaStreamWaitEvent(cs, meta_in, 0)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(cs, in_done, 0)) != cudaSuccess)
            return e;
        prefill::FwdArgs f = {};
        f.q = dq;
        f.k = dk;
        f.v = dv;
        f.sink = dsink;
        f.cu_q = dmeta + 4 * c;  // this chunk alone: absolute row offsets
        f.cu_k = dmeta + 4 * c + 2;
        f.out = dout;
        f.lse = a.lse ? dlse : nullptr;
        f.batch = 1;
        f.total_q = a.total_q;  // also the lse head stride
        // K/V rows past the chunk's keys are out of the tensor for this launch (the
        // copy engine may still be writing them): the tail tile reads zeros.
        f.total_k = ch.ke;
        f.hq = a.hq;
        f.hkv = a.hkv;
        f.head_dim = a.head_dim;
        f.max_seqlen_q = ch.qe - ch.qb;
        f.max_seqlen_k = ch.ke - ch.kb;
        f.win_first = a.win_first;
        f.win_last = a.win_last;
        f.causal = a.causal;
        f.scale = a.scale;
        if ((e = prefill::launch_fwd(f, cs, what)) != cudaSuccess) return e;
        if ((e = cudaEventRecord(comp_done, cs)) != cudaSuccess) return e;
        *what = "copy-out";
        if ((e = cudaStreamWaitEvent(st.out, comp_done, 0)) != cudaSuccess) return e;
        if ((e = cudaMemcpyAsync(hout + (size_t)ch.qb * q_row, dout + (size_t)ch.qb * q_row,
                                 (size_t)(ch.qe - ch.qb) * q_row, cudaMemcpyDeviceToHost, st.out)) != cudaSuccess)
            return e;
        if (a.lse && (e = cudaMemcpy2DAsync(a.lse + ch.qb, (size_t)a.total_q * 4, dlse + ch.qb, (size_t)a.total_q * 4,
                                            (size_t)(ch.qe - ch.qb) * 4, a.hq, cudaMemcpyDeviceToHost, st.out)) !=
                          cudaSuccess)
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
           r((size_t)a.hq * 4) + r((size_t)std::max(1, count_chunks(a)) * 16);
}

}  // namespace hostio
}  // namespace attn
