// C ABI of the attention-with-sink library: argument validation, scratch
// memory and kernel launches.  Every entry point is asynchronous on the
// caller's stream and returns an ATTN_SINK_* status.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <mutex>
#include <string>

#include "attn_sink.h"
#include "bwd.h"
#include "common.cuh"
#include "decode.h"
#include "host_io.h"
#include "kv_append.h"
#include "selftest.h"
#include "prefill.h"

namespace {

thread_local std::string t_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(ATTN_SINK_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

// The forward, decode and append grids give the request index a grid dimension
// of at most 65535 blocks, and the forward its 128-row query tiles another.
constexpr int kMaxGridDim = 65535;

int check_grid(const char* who, int batch, int max_seqlen_q) {
    if (batch > kMaxGridDim)
        return fail(ATTN_SINK_ERR_UNSUPPORTED, "%s: batch %d above %d requests per call", who, batch, kMaxGridDim);
    if (max_seqlen_q > 0 && (max_seqlen_q + 127) / 128 > kMaxGridDim)
        return fail(ATTN_SINK_ERR_UNSUPPORTED, "%s: max_seqlen_q %d above %d query rows per request", who,
                    max_seqlen_q, kMaxGridDim * 128);
    return ATTN_SINK_OK;
}

// One library-owned stream-ordered memory pool per device.  Freed blocks are
// kept (release threshold = max) so that steady-state calls do not go back to
// the driver.
constexpr int kMaxDevices = 64;
std::mutex g_pool_mu;
cudaMemPool_t g_pools[kMaxDevices] = {};

cudaError_t device_pool(cudaMemPool_t* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_pool_mu);
    if (!g_pools[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool;
        e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess) return e;
        uint64_t thr = ~0ull;
        e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
        if (e != cudaSuccess) return e;
        g_pools[dev] = pool;
    }
    *out = g_pools[dev];
    return cudaSuccess;
}

// Stream-ordered scratch block, returned to the pool on the same stream.
struct Scratch {
    void* ptr = nullptr;
    cudaStream_t stream = nullptr;
    cudaError_t alloc(size_t bytes, cudaStream_t s) {
        stream = s;
        if (bytes == 0) return cudaSuccess;
        cudaMemPool_t pool;
        cudaError_t e = device_pool(&pool);
        if (e != cudaSuccess) return e;
        return cudaMallocFromPoolAsync(&ptr, bytes, pool, s);
    }
    ~Scratch() {
        if (ptr) cudaFreeAsync(ptr, stream);
    }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace attn {
float resolve_scale(float scale, int head_dim) {
    return scale > 0.f ? scale : 1.0f / sqrtf((float)head_dim);
}

// Sets the calling thread's last-error text (used by entry points defined in
// other translation units).
void record_error(const char* msg) { t_last_error = msg; }
}  // namespace attn

extern "C" {

const char* attn_sink_last_error(void) { return t_last_error.c_str(); }

const char* attn_sink_version(void) { return "attn_sink_gb300 0.1 (sm_103a)"; }

}  // extern "C"

namespace attn {

int validate_decode(const char* who, const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache,
                    const int32_t* page_table, int max_pages, const int32_t* seqlens, int batch, int hq,
                    int hkv, int head_dim, int page_size, int num_pages, int win_first, attn_bf16* out) {
    if (batch < 0 || hq <= 0 || hkv <= 0 || max_pages <= 0 || page_size <= 0 || num_pages <= 0)
        return fail(ATTN_SINK_ERR_INVALID, "%s: sizes must be positive (batch may be 0)", who);
    if (win_first < 0) return fail(ATTN_SINK_ERR_INVALID, "%s: win_first must be >= 0", who);
    if (head_dim != 64 && head_dim != 128)
        return fail(ATTN_SINK_ERR_UNSUPPORTED, "%s: head_dim %d not supported (64, 128)", who, head_dim);
    if (hq % hkv) return fail(ATTN_SINK_ERR_UNSUPPORTED, "%s: hq %% hkv != 0", who);
    if (batch == 0) return ATTN_SINK_OK;
    if (!q || !k_cache || !v_cache || !page_table || !seqlens || !out)
        return fail(ATTN_SINK_ERR_INVALID, "%s: NULL tensor pointer", who);
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q) || !aligned16(out))
        return fail(ATTN_SINK_ERR_INVALID, "%s: q, caches and out must be 16-byte aligned", who);
    if ((long long)num_pages * page_size >= (1LL << 31) || (long long)max_pages * page_size >= (1LL << 31))
        return fail(ATTN_SINK_ERR_UNSUPPORTED, "%s: cache slots must fit in int32", who);
    return check_grid(who, batch, 0);
}

}  // namespace attn

namespace {

int run_decode(const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache, const int32_t* page_table,
               int max_pages, const int32_t* seqlens, int batch, int hq, int hkv, int head_dim, int page_size,
               int num_pages, const float* sink, int win_first, int win_last, float scale, attn_bf16* out,
               float* lse, cudaStream_t s) {
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
    attn::decode::Plan pl = attn::decode::make_plan(a);
    Scratch ws;
    cudaError_t e = ws.alloc(pl.part_o_bytes + pl.part_ml_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode: scratch allocation");
    float* part_o = static_cast<float*>(ws.ptr);
    float2* part_ml = reinterpret_cast<float2*>(static_cast<char*>(ws.ptr) + pl.part_o_bytes);
    e = attn::decode::launch(a, pl, part_o, part_ml, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode: launch");
    return ATTN_SINK_OK;
}

int run_append(const attn_bf16* k_new, const attn_bf16* v_new, const int32_t* cu_new, const int32_t* seqlens,
               const int32_t* page_table, int max_pages, int batch, int hkv, int head_dim, int page_size,
               int num_pages, int max_new, attn_bf16* k_cache, attn_bf16* v_cache, cudaStream_t s) {
    attn::kvappend::Args a;
    a.k_new = k_new;
    a.v_new = v_new;
    a.cu_new = cu_new;
    a.seqlens = seqlens;
    a.page_table = page_table;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.max_pages = max_pages;
    a.batch = batch;
    a.hkv = hkv;
    a.head_dim = head_dim;
    a.page_size = page_size;
    a.num_pages = num_pages;
    a.max_new = max_new;
    cudaError_t e = attn::kvappend::launch(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "kv_append: launch");
    return ATTN_SINK_OK;
}

}  // namespace

extern "C" {

int attn_sink_decode_paged(const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache,
                           const int32_t* page_table, int max_pages, const int32_t* seqlens,
                           int batch, int hq, int hkv, int head_dim, int page_size, int num_pages,
                           const float* sink, int win_first, int win_last, float scale,
                           attn_bf16* out, float* lse, void* stream) {
    t_last_error.clear();
    int rc = attn::validate_decode("decode", q, k_cache, v_cache, page_table, max_pages, seqlens, batch, hq, hkv, head_dim,
                             page_size, num_pages, win_first, out);
    if (rc != ATTN_SINK_OK || batch == 0) return rc;
    return run_decode(q, k_cache, v_cache, page_table, max_pages, seqlens, batch, hq, hkv, head_dim, page_size,
                      num_pages, sink, win_first, win_last, scale, out, lse, static_cast<cudaStream_t>(stream));
}

int attn_sink_kv_append(const attn_bf16* k_new, const attn_bf16* v_new, const int32_t* cu_new,
                        const int32_t* seqlens, const int32_t* page_table, int max_pages, int batch, int hkv,
                        int head_dim, int page_size, int num_pages, int max_new, attn_bf16* k_cache,
                        attn_bf16* v_cache, void* stream) {
    t_last_error.clear();
    if (batch < 0 || hkv <= 0 || max_pages <= 0 || page_size <= 0 || num_pages <= 0 || max_new < 0)
        return fail(ATTN_SINK_ERR_INVALID, "kv_append: sizes must be positive (batch, max_new may be 0)");
    if (head_dim != 64 && head_dim != 128)
        return fail(ATTN_SINK_ERR_UNSUPPORTED, "kv_append: head_dim %d not supported (64, 128)", head_dim);
    if ((long long)num_pages * page_size >= (1LL << 31) || (long long)max_pages * page_size >= (1LL << 31))
        return fail(ATTN_SINK_ERR_UNSUPPORTED, "kv_append: cache slots must fit in int32");
    if (batch == 0 || max_new == 0) return ATTN_SINK_OK;
    if (!k_new || !v_new || !seqlens || !page_table || !k_cache || !v_cache)
        return fail(ATTN_SINK_ERR_INVALID, "kv_append: NULL tensor pointer");
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(ATTN_SINK_ERR_INVALID, "kv_append: tensors must be 16-byte aligned");
    if (!cu_new && max_new != 1)
        return fail(ATTN_SINK_ERR_INVALID, "kv_append: without cu_new every request appends one row (max_new 1)");
    if (int rc = check_grid("kv_append", batch, 0)) return rc;
    return run_append(k_new, v_new, cu_new, seqlens, page_table, max_pages, batch, hkv, head_dim, page_size,
                      num_pages, max_new, k_cache, v_cache, static_cast<cudaStream_t>(stream));
}

int attn_sink_decode_paged_append(const attn_bf16* q, const attn_bf16* k_new, const attn_bf16* v_new,
                                  attn_bf16* k_cache, attn_bf16* v_cache, const int32_t* page_table,
                                  int max_pages, const int32_t* seqlens, int batch, int hq, int hkv, int head_dim,
                                  int page_size, int num_pages, const float* sink, int win_first, int win_last,
                                  float scale, attn_bf16* out, float* lse, void* stream) {
    t_last_error.clear();
    int rc = attn::validate_decode("decode", q, k_cache, v_cache, page_table, max_pages, seqlens, batch, hq, hkv, head_dim,
                             page_size, num_pages, win_first, out);
    if (rc != ATTN_SINK_OK || batch == 0) return rc;
    if (!k_new || !v_new) return fail(ATTN_SINK_ERR_INVALID, "decode_append: NULL k_new / v_new");
    if (!aligned16(k_new) || !aligned16(v_new))
        return fail(ATTN_SINK_ERR_INVALID, "decode_append: k_new, v_new must be 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = run_append(k_new, v_new, nullptr, seqlens, page_table, max_pages, batch, hkv, head_dim, page_size,
                    num_pages, 1, k_cache, v_cache, s);
    if (rc != ATTN_SINK_OK) return rc;
    return run_decode(q, k_cache, v_cache, page_table, max_pages, seqlens, batch, hq, hkv, head_dim, page_size,
                      num_pages, sink, win_first, win_last, scale, out, lse, s);
}

int attn_sink_visible_ranges(const int32_t* seqlens, int batch, int win_first, int win_last,
                             int32_t* ranges, void* stream) {
    t_last_error.clear();
    if (batch < 0 || win_first < 0) return fail(ATTN_SINK_ERR_INVALID, "visible_ranges: bad sizes");
    if (batch == 0) return ATTN_SINK_OK;
    if (!seqlens || !ranges) return fail(ATTN_SINK_ERR_INVALID, "visible_ranges: NULL pointer");
    cudaError_t e = attn::decode::launch_visible_ranges(seqlens, batch, win_first, win_last, ranges,
                                                        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "visible_ranges: launch");
    return ATTN_SINK_OK;
}

int attn_sink_visible_slots(const int32_t* seqlens, const int32_t* page_table, int max_pages,
                            int batch, int page_size, int num_pages, int win_first, int win_last,
                            int32_t* slots, int max_visible, void* stream) {
    t_last_error.clear();
    if (batch < 0 || max_pages <= 0 || page_size <= 0 || num_pages <= 0 || max_visible < 0 || win_first < 0)
        return fail(ATTN_SINK_ERR_INVALID, "visible_slots: bad sizes");
    if ((long long)num_pages * page_size >= (1LL << 31))
        return fail(ATTN_SINK_ERR_UNSUPPORTED, "visible_slots: cache slots must fit in int32");
    if (batch == 0 || max_visible == 0) return ATTN_SINK_OK;
    if (!seqlens || !page_table || !slots) return fail(ATTN_SINK_ERR_INVALID, "visible_slots: NULL pointer");
    cudaError_t e = attn::decode::launch_visible_slots(seqlens, page_table, max_pages, batch, page_size,
                                                       num_pages, win_first, win_last, slots, max_visible,
                                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "visible_slots: launch");
    return ATTN_SINK_OK;
}

static int validate_varlen(const char* who, const void* q, const void* k, const void* v,
                           const int32_t* cu_q, const int32_t* cu_k, int batch, int total_q,
                           int total_k, int hq, int hkv,
                           int head_dim, int max_seqlen_q, int max_seqlen_k, int win_first,
                           int win_last, int causal, bool allow_d128) {
    if (batch < 0 || total_q < 0 || total_k < 0 || hq <= 0 || hkv <= 0 || max_seqlen_q < 0 ||
        max_seqlen_k < 0 || win_first < 0)
        return fail(ATTN_SINK_ERR_INVALID, "%s: sizes must be non-negative (heads positive)", who);
    if (win_last > 0 && !causal)
        return fail(ATTN_SINK_ERR_INVALID, "%s: first/last-window selection needs causal attention", who);
    if (head_dim != 64 && !(allow_d128 && head_dim == 128))
        return fail(ATTN_SINK_ERR_UNSUPPORTED, "%s: head_dim %d not supported (%s)", who, head_dim,
                    allow_d128 ? "64, 128" : "64");
    if (hq % hkv) return fail(ATTN_SINK_ERR_UNSUPPORTED, "%s: hq %% hkv != 0", who);
    if (batch == 0) return ATTN_SINK_OK;
    if (!q || !k || !v || !cu_q || !cu_k) return fail(ATTN_SINK_ERR_INVALID, "%s: NULL tensor pointer", who);
    if (!aligned16(q) || !aligned16(k) || !aligned16(v))
        return fail(ATTN_SINK_ERR_INVALID, "%s: q, k, v must be 16-byte aligned", who);
    return ATTN_SINK_OK;
}

}  // extern "C"

namespace {

// A row stride (elements) is 0 (contiguous) or covers the row's heads and keeps
// every row 16-byte aligned.
int check_stride(const char* who, const char* name, long long rs, int heads, int head_dim) {
    if (rs == 0) return ATTN_SINK_OK;
    if (rs < (long long)heads * head_dim || rs % 8)
        return fail(ATTN_SINK_ERR_INVALID,
                    "%s: %s row stride %lld must be 0 or >= heads*head_dim and a multiple of 8", who, name, rs);
    return ATTN_SINK_OK;
}

int fwd_impl(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, long long q_rs, long long k_rs,
             long long v_rs, const float* sink, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch,
             int total_q, int total_k, int hq, int hkv, int head_dim, int max_seqlen_q, int max_seqlen_k,
             int win_first, int win_last, int causal, float scale, attn_bf16* out, float* lse, void* stream) {
    int rc = validate_varlen("fwd", q, k, v, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, hq, hkv, head_dim,
                             max_seqlen_q, max_seqlen_k, win_first, win_last, causal, true);
    if (rc != ATTN_SINK_OK || batch == 0 || max_seqlen_q == 0 || total_q == 0) return rc;
    if ((rc = check_grid("fwd", batch, max_seqlen_q)) != ATTN_SINK_OK) return rc;
    if (!out) return fail(ATTN_SINK_ERR_INVALID, "fwd: NULL out");
    if (!aligned16(out)) return fail(ATTN_SINK_ERR_INVALID, "fwd: out must be 16-byte aligned");
    attn::prefill::FwdArgs a = {};
    a.q = q;
    a.k = k;
    a.v = v;
    a.sink = sink;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.out = out;
    a.lse = lse;
    a.batch = batch;
    a.total_q = total_q;
    a.total_k = total_k;
    a.hq = hq;
    a.hkv = hkv;
    a.head_dim = head_dim;
    a.max_seqlen_q = max_seqlen_q;
    a.max_seqlen_k = max_seqlen_k;
    a.win_first = win_first;
    a.win_last = win_last;
    a.causal = causal ? 1 : 0;
    a.scale = attn::resolve_scale(scale, head_dim);
    a.q_rs = q_rs;
    a.k_rs = k_rs;
    a.v_rs = v_rs;
    std::string err;
    cudaError_t e = attn::prefill::launch_fwd(a, static_cast<cudaStream_t>(stream), &err);
    if (e != cudaSuccess) return fail(ATTN_SINK_ERR_CUDA, "fwd: %s: %s", err.c_str(), cudaGetErrorString(e));
    return ATTN_SINK_OK;
}

}  // namespace

extern "C" {

int attn_sink_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, const float* sink,
                  const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch, int total_q,
                  int total_k, int hq, int hkv, int head_dim, int max_seqlen_q, int max_seqlen_k,
                  int win_first, int win_last, int causal, float scale, attn_bf16* out, float* lse,
                  void* stream) {
    t_last_error.clear();
    return fwd_impl(q, k, v, 0, 0, 0, sink, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, hq, hkv, head_dim,
                    max_seqlen_q, max_seqlen_k, win_first, win_last, causal, scale, out, lse, stream);
}

int attn_sink_fwd_strided(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, long long q_row_stride,
                          long long k_row_stride, long long v_row_stride, const float* sink,
                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch, int total_q,
                          int total_k, int hq, int hkv, int head_dim, int max_seqlen_q, int max_seqlen_k,
                          int win_first, int win_last, int causal, float scale, attn_bf16* out, float* lse,
                          void* stream) {
    t_last_error.clear();
    int rc;
    if ((rc = check_stride("fwd_strided", "q", q_row_stride, hq, head_dim)) != ATTN_SINK_OK ||
        (rc = check_stride("fwd_strided", "k", k_row_stride, hkv, head_dim)) != ATTN_SINK_OK ||
        (rc = check_stride("fwd_strided", "v", v_row_stride, hkv, head_dim)) != ATTN_SINK_OK)
        return rc;
    return fwd_impl(q, k, v, q_row_stride, k_row_stride, v_row_stride, sink, cu_seqlens_q, cu_seqlens_k, batch,
                    total_q, total_k, hq, hkv, head_dim, max_seqlen_q, max_seqlen_k, win_first, win_last, causal,
                    scale, out, lse, stream);
}

int attn_sink_fwd_host(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, const float* sink,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch, int hq, int hkv,
                       int head_dim, int win_first, int win_last, int causal, float scale, attn_bf16* out,
                       float* lse, void* stream) {
    t_last_error.clear();
    if (batch < 0 || hq <= 0 || hkv <= 0 || win_first < 0)
        return fail(ATTN_SINK_ERR_INVALID, "fwd_host: sizes must be non-negative (heads positive)");
    if (win_last > 0 && !causal)
        return fail(ATTN_SINK_ERR_INVALID, "fwd_host: first/last-window selection needs causal attention");
    if (head_dim != 64 && head_dim != 128)
        return fail(ATTN_SINK_ERR_UNSUPPORTED, "fwd_host: head_dim %d not supported (64, 128)", head_dim);
    if (hq % hkv) return fail(ATTN_SINK_ERR_UNSUPPORTED, "fwd_host: hq %% hkv != 0");
    if (batch == 0) return ATTN_SINK_OK;
    if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !out)
        return fail(ATTN_SINK_ERR_INVALID, "fwd_host: NULL pointer");
    if (cu_seqlens_q[0] != 0 || cu_seqlens_k[0] != 0)
        return fail(ATTN_SINK_ERR_INVALID, "fwd_host: cu_seqlens must start at 0");
    for (int b = 0; b < batch; ++b)
        if (cu_seqlens_q[b + 1] < cu_seqlens_q[b] || cu_seqlens_k[b + 1] < cu_seqlens_k[b])
            return fail(ATTN_SINK_ERR_INVALID, "fwd_host: cu_seqlens must be non-decreasing");
    attn::hostio::Args a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.sink = sink;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.out = out;
    a.lse = lse;
    a.batch = batch;
    a.total_q = cu_seqlens_q[batch];
    a.total_k = cu_seqlens_k[batch];
    a.hq = hq;
    a.hkv = hkv;
    a.head_dim = head_dim;
    a.win_first = win_first;
    a.win_last = win_last;
    a.causal = causal ? 1 : 0;
    a.scale = attn::resolve_scale(scale, head_dim);
    if (a.total_q == 0) return ATTN_SINK_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Scratch ws;
    cudaError_t e = ws.alloc(attn::hostio::scratch_bytes(a), s);
    if (e != cudaSuccess) return cuda_fail(e, "fwd_host: scratch allocation");
    std::string err;
    e = attn::hostio::run(a, ws.ptr, s, &err);
    if (e != cudaSuccess) return fail(ATTN_SINK_ERR_CUDA, "fwd_host: %s: %s", err.c_str(), cudaGetErrorString(e));
    return ATTN_SINK_OK;
}

int attn_sink_fwd_paged(const attn_bf16* q, const attn_bf16* k_new, const attn_bf16* v_new, attn_bf16* k_cache,
                        attn_bf16* v_cache, const int32_t* page_table, int max_pages,
                        const int32_t* cu_seqlens_q, const int32_t* seqlens_k, int batch, int total_q, int hq,
                        int hkv, int head_dim, int page_size, int num_pages, int max_seqlen_q, int max_seqlen_k,
                        const float* sink, int win_first, int win_last, int causal, float scale,
                        attn_bf16* out, float* lse, void* stream) {
    t_last_error.clear();
    if (batch < 0 || total_q < 0 || hq <= 0 || hkv <= 0 || max_pages <= 0 || page_size <= 0 || num_pages <= 0 ||
        max_seqlen_q < 0 || max_seqlen_k < 0 || win_first < 0)
        return fail(ATTN_SINK_ERR_INVALID, "fwd_paged: sizes must be non-negative (heads, pages positive)");
    if (win_last > 0 && !causal)
        return fail(ATTN_SINK_ERR_INVALID, "fwd_paged: first/last-window selection needs causal attention");
    if (head_dim != 64 && head_dim != 128)
        return fail(ATTN_SINK_ERR_UNSUPPORTED, "fwd_paged: head_dim %d not supported (64, 128)", head_dim);
    if (hq % hkv) return fail(ATTN_SINK_ERR_UNSUPPORTED, "fwd_paged: hq %% hkv != 0");
    if (page_size < 8 || (page_size & (page_size - 1)))
        return fail(ATTN_SINK_ERR_UNSUPPORTED, "fwd_paged: page_size %d not supported (a power of two >= 8)",
                    page_size);
    if ((long long)num_pages * page_size >= (1LL << 31) || (long long)max_pages * page_size >= (1LL << 31))
        return fail(ATTN_SINK_ERR_UNSUPPORTED, "fwd_paged: cache slots must fit in int32");
    if ((k_new == nullptr) != (v_new == nullptr))
        return fail(ATTN_SINK_ERR_INVALID, "fwd_paged: k_new and v_new are given together or not at all");
    if (batch == 0 || total_q == 0 || max_seqlen_q == 0) return ATTN_SINK_OK;
    if (!q || !k_cache || !v_cache || !page_table || !cu_seqlens_q || !seqlens_k || !out)
        return fail(ATTN_SINK_ERR_INVALID, "fwd_paged: NULL tensor pointer");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (k_new && (!aligned16(k_new) || !aligned16(v_new))))
        return fail(ATTN_SINK_ERR_INVALID, "fwd_paged: tensors must be 16-byte aligned");
    if (int rc = check_grid("fwd_paged", batch, max_seqlen_q)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (k_new) {
        int rc = run_append(k_new, v_new, cu_seqlens_q, seqlens_k, page_table, max_pages, batch, hkv, head_dim,
                            page_size, num_pages, max_seqlen_q, k_cache, v_cache, s);
        if (rc != ATTN_SINK_OK) return rc;
    }
    attn::prefill::FwdArgs a = {};
    a.q = q;
    a.k = k_cache;
    a.v = v_cache;
    a.sink = sink;
    a.cu_q = cu_seqlens_q;
    a.cu_k = nullptr;
    a.out = out;
    a.lse = lse;
    a.batch = batch;
    a.total_q = total_q;
    a.total_k = 0;
    a.hq = hq;
    a.hkv = hkv;
    a.head_dim = head_dim;
    a.max_seqlen_q = max_seqlen_q;
    a.max_seqlen_k = max_seqlen_k;
    a.win_first = win_first;
    a.win_last = win_last;
    a.causal = causal ? 1 : 0;
    a.scale = attn::resolve_scale(scale, head_dim);
    a.page_table = page_table;
    a.seqlens_k = seqlens_k;
    a.max_pages = max_pages;
    a.page_size = page_size;
    a.num_pages = num_pages;
    std::string err;
    cudaError_t e = attn::prefill::launch_fwd(a, s, &err);
    if (e != cudaSuccess) return fail(ATTN_SINK_ERR_CUDA, "fwd_paged: %s: %s", err.c_str(), cudaGetErrorString(e));
    return ATTN_SINK_OK;
}

}  // extern "C"

namespace {

int bwd_impl(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, const long long* rs, const float* sink,
             const attn_bf16* out, const float* lse, const attn_bf16* dout, const int32_t* cu_seqlens_q,
             const int32_t* cu_seqlens_k, int batch, int total_q, int total_k, int hq, int hkv, int head_dim,
             int max_seqlen_q, int max_seqlen_k, int win_first, int win_last, int causal, float scale,
             attn_bf16* dq, attn_bf16* dk, attn_bf16* dv, float* dsink, void* stream) {
    int rc = validate_varlen("bwd", q, k, v, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, hq, hkv, head_dim,
                             max_seqlen_q, max_seqlen_k, win_first, win_last, causal, true);
    if (rc != ATTN_SINK_OK) return rc;
    if ((sink == nullptr) != (dsink == nullptr))
        return fail(ATTN_SINK_ERR_INVALID, "bwd: dsink must be given exactly when sink is");
    if (batch == 0) return ATTN_SINK_OK;
    if (!out || !lse || !dout || !dq || !dk || !dv)
        return fail(ATTN_SINK_ERR_INVALID, "bwd: NULL tensor pointer");
    if (!aligned16(out) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return fail(ATTN_SINK_ERR_INVALID, "bwd: tensors must be 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    attn::bwd::Args a = {};
    a.q = q;
    a.k = k;
    a.v = v;
    a.sink = sink;
    a.out = out;
    a.lse = lse;
    a.dout = dout;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.dsink = dsink;
    a.batch = batch;
    a.total_q = total_q;
    a.total_k = total_k;
    a.hq = hq;
    a.hkv = hkv;
    a.head_dim = head_dim;
    a.max_seqlen_q = max_seqlen_q;
    a.max_seqlen_k = max_seqlen_k;
    a.win_first = win_first;
    a.win_last = win_last;
    a.causal = causal ? 1 : 0;
    a.scale = attn::resolve_scale(scale, head_dim);
    a.q_rs = rs[0];
    a.k_rs = rs[1];
    a.v_rs = rs[2];
    a.dq_rs = rs[3];
    a.dk_rs = rs[4];
    a.dv_rs = rs[5];
    size_t ws_bytes = attn::bwd::workspace_bytes(a);
    Scratch ws;
    cudaError_t e = ws.alloc(ws_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "bwd: scratch allocation");
    std::string err;
    e = attn::bwd::launch(a, ws.ptr, ws_bytes, s, &err);
    if (e != cudaSuccess) return fail(ATTN_SINK_ERR_CUDA, "bwd: %s: %s", err.c_str(), cudaGetErrorString(e));
    return ATTN_SINK_OK;
}

}  // namespace

extern "C" {

int attn_sink_bwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, const float* sink,
                  const attn_bf16* out, const float* lse, const attn_bf16* dout,
                  const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch, int total_q,
                  int total_k, int hq, int hkv, int head_dim, int max_seqlen_q, int max_seqlen_k,
                  int win_first, int win_last, int causal, float scale, attn_bf16* dq, attn_bf16* dk,
                  attn_bf16* dv, float* dsink, void* stream) {
    t_last_error.clear();
    const long long rs[6] = {0, 0, 0, 0, 0, 0};
    return bwd_impl(q, k, v, rs, sink, out, lse, dout, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, hq,
                    hkv, head_dim, max_seqlen_q, max_seqlen_k, win_first, win_last, causal, scale, dq, dk, dv,
                    dsink, stream);
}

int attn_sink_bwd_strided(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, long long q_row_stride,
                          long long k_row_stride, long long v_row_stride, const float* sink,
                          const attn_bf16* out, const float* lse, const attn_bf16* dout,
                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int batch, int total_q,
                          int total_k, int hq, int hkv, int head_dim, int max_seqlen_q, int max_seqlen_k,
                          int win_first, int win_last, int causal, float scale, attn_bf16* dq, attn_bf16* dk,
                          attn_bf16* dv, long long dq_row_stride, long long dk_row_stride,
                          long long dv_row_stride, float* dsink, void* stream) {
    t_last_error.clear();
    int rc;
    const long long rs[6] = {q_row_stride, k_row_stride, v_row_stride, dq_row_stride, dk_row_stride,
                             dv_row_stride};
    const char* names[6] = {"q", "k", "v", "dq", "dk", "dv"};
    for (int i = 0; i < 6; ++i)
        if ((rc = check_stride("bwd_strided", names[i], rs[i], (i % 3) == 0 ? hq : hkv, head_dim)) != ATTN_SINK_OK) return rc;
    return bwd_impl(q, k, v, rs, sink, out, lse, dout, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, hq,
                    hkv, head_dim, max_seqlen_q, max_seqlen_k, win_first, win_last, causal, scale, dq, dk, dv,
                    dsink, stream);
}

int attn_sink_device_status(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int bits = 0;
    int e = attn::decode::status_exchange(s, &bits);
    if (!e) e = attn::prefill::status_exchange(s, &bits);
    if (!e) e = attn::bwd::status_exchange(s, &bits);
    if (!e) e = attn::kvappend::status_exchange(s, &bits);
    if (!e) e = attn::selftest::status_exchange(s, &bits);
    if (e) return cuda_fail(static_cast<cudaError_t>(e), "device_status");
    return bits;
}

int attn_sink_selftest_wait(int complete, void* stream) {
    t_last_error.clear();
    cudaError_t e = attn::selftest::launch_wait(complete, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "selftest_wait: launch");
    return ATTN_SINK_OK;
}

}  // extern "C"
