// Paged single-token decode with an attention sink and first/last-window KV
// selection (split-KV "flash-decoding" form).
//
// What it computes (sglang PR "openai oss attention sink support with
// trtllm-gen backend", Highlights: the decode path takes a per-head sink;
// sglang PR "To implement attention-sink", suggested code: the first 1024 and
// the last 7168 cached tokens, per sequence):
//     O = sum_{t in V} e^{s_t - M} v_t / (e^{sink - M} + sum_{t in V} e^{s_t - M})
// over the visible tokens V of each request, read through its page table.
//
// Structure:
//  * decode_split_kernel -- one CTA per (split of visible tokens, KV head,
//    request).  16-byte cp.async gathers stage 64-token chunks of K and V in
//    shared memory (a multi-stage ring); each warp owns 16 tokens of a chunk.
//    The G query heads of the KV head are the N dimension of two small
//    tensor-core products per chunk: S^T = K q^T (tokens x heads) and
//    O^T += V^T P^T (head_dim x heads), so a group of 8 heads wastes no MMA
//    rows.  Each split writes an un-normalised partial (m, l, o) without the
//    sink.
//  * decode_combine_kernel -- merges the partials of a (request, head) in the
//    log-sum-exp sense and folds the sink in exactly once (flash-attention PR
//    "feat: Implement Sink Attention": a user reports wrong decode results with
//    the sink through the KV-cache API; adding the sink per split would count
//    it once per split).
// Decode is HBM-bound: the products run on mma.sync only so that the FMA
// pipes never limit the gather rate.
#include "common.cuh"
#include "decode.h"

#include <math.h>

namespace attn {
namespace decode {

constexpr int kChunk = 64;     // tokens per pipeline stage
constexpr int kThreads = 128;  // 4 warps x 16 tokens per chunk

// ---------------------------------------------------------------------------
// Warp-level PTX helpers.

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Transpose of an 8x8 b16 matrix held one row pair per thread.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float warp_max_g(float x) {  // over lanes with equal lane%4
    x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
    x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 8));
    x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 16));
    return x;
}
__device__ __forceinline__ float warp_sum_g(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 8);
    x += __shfl_xor_sync(0xffffffffu, x, 16);
    return x;
}

// Byte offset of 16-byte segment `col` of token row `row` in a staged chunk:
// rows of D bf16, segments XOR-swizzled by row so that ldmatrix is conflict-free.
template <int D>
__device__ __forceinline__ uint32_t chunk_off(int row, int col) {
    return row * (D * 2) + ((col ^ (row & 7)) << 4);
}

// Visible-token ranges of request b (decode query at position L-1), with L
// clamped to the page table's capacity.
__device__ __forceinline__ Ranges request_ranges(const SplitParams& p, int b, bool report) {
    int L = p.seqlens[b];
    int cap = p.max_pages * p.page_size;
    if (L > cap) {
        if (report) raise_status(ATTN_SINK_DEV_SEQLEN_OOB);
        L = cap;
    }
    if (L < 0) L = 0;
    return visible_ranges(L - 1, p.win_first, p.win_last);
}

template <int D, int NT, int NSTAGE>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const SplitParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    // Per staged token row: 1 if it holds a visible token read through a valid
    // page, 0 if it was zero-filled (past the split, or an out-of-range page id);
    // invalid rows get a score of -inf, so they take no weight in the softmax.
    __shared__ uint8_t row_ok[NSTAGE][kChunk];
    constexpr int kStageBytes = 2 * kChunk * D * 2;
    constexpr int kSegs = D / 8;                        // 16-byte segments per row
    // The combine kernel is launched as a programmatic dependent of this grid:
    // once every CTA of this grid has started, its CTAs may be scheduled, and
    // they wait (griddepcontrol.wait) for this grid to finish before reading
    // the partials.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int split = blockIdx.x;
    const int kvh = blockIdx.y / p.hblocks;
    const int hb = blockIdx.y % p.hblocks;
    const int b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const Ranges r = request_ranges(p, b, tid == 0 && split == 0 && blockIdx.y == 0);
    const int nvis = visible_count(r);
    const long long v0l = (long long)split * p.split_tokens;
    if (v0l >= nvis) return;
    const int v0 = (int)v0l;
    const int v1 = (int)min((long long)nvis, v0l + p.split_tokens);
    const int nchunks = (v1 - v0 + kChunk - 1) / kChunk;

    const int h_base = kvh * p.group + hb * 8 * NT;
    const int nheads = min(8 * NT, p.group - hb * 8 * NT);

    // q^T fragments (B operand of S^T = K q^T): head lane/4, dims 2(lane%4)+{0,1}, +8.
    uint32_t qf[NT][D / 16][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int head = nt * 8 + (lane >> 2);
        const bool ok = head < nheads;
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + ((size_t)b * p.hq + h_base + (ok ? head : 0)) * D);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qf[nt][kk][0] = ok ? qrow[8 * kk + (lane & 3)] : 0u;
            qf[nt][kk][1] = ok ? qrow[8 * kk + 4 + (lane & 3)] : 0u;
        }
    }

    // Loading: every warp instruction copies whole contiguous token rows
    // (32 x 16 B = 512 B: four 128-byte rows at d 64, two 256-byte rows at
    // d 128).  A warp stages 16 of the chunk's 64 rows; lanes 0..15 look up
    // one row's physical slot each (one page-table read per row and chunk) and
    // the copies fetch it by shuffle.
    constexpr int kRowsPerInst = 32 / kSegs;          // rows per warp instruction
    constexpr int kInsts = 16 / kRowsPerInst;         // instructions per warp and chunk
    const int my_seg = lane % kSegs, my_sub = lane / kSegs;
    auto load_chunk = [&](int c, int stage) {
        uint8_t* sK = smem + stage * kStageBytes;
        uint8_t* sV = sK + kChunk * D * 2;
        // slot of the warp's (lane)-th row; rows of instruction i: (i*4 + warp) * kRowsPerInst + sub
        int slot = -1;
        if (lane < 16) {
            const int row = ((lane / kRowsPerInst) * 4 + warp) * kRowsPerInst + (lane % kRowsPerInst);
            row_ok[stage][row] = 0;
            const int v = v0 + c * kChunk + row;
            if (v < v1) {
                const int t = visible_token(r, v);
                int pg, in_pg;
                if (p.page_shift >= 0) {
                    pg = t >> p.page_shift;
                    in_pg = t & ((1 << p.page_shift) - 1);
                } else {
                    pg = t / p.page_size;
                    in_pg = t - pg * p.page_size;
                }
                const int page = p.page_table[(size_t)b * p.max_pages + pg];
                if ((unsigned)page < (unsigned)p.num_pages) {
                    slot = page * p.page_size + in_pg;
                    row_ok[stage][row] = 1;
                } else {
                    raise_status(ATTN_SINK_DEV_PAGE_OOB);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kInsts; ++i) {
            const int sl = __shfl_sync(0xffffffffu, slot, i * kRowsPerInst + my_sub);
            const int row = (i * 4 + warp) * kRowsPerInst + my_sub;
            const size_t off = sl >= 0 ? ((size_t)sl * p.hkv + kvh) * D + my_seg * 8 : 0;
            const int bytes = sl >= 0 ? 16 : 0;  // 0: zero fill
            const uint32_t so = chunk_off<D>(row, my_seg);
            cp_async_16(smem_u32(sK + so), p.k_cache + off, bytes);
            cp_async_16(smem_u32(sV + so), p.v_cache + off, bytes);
        }
    };

    float m_run[NT][2], l_run[NT][2];
    float o[D / 16][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m_run[nt][0] = m_run[nt][1] = -INFINITY;
        l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) o[mt][nt][i] = 0.f;
    }

#pragma unroll
    for (int s = 0; s < NSTAGE - 1; ++s) {
        if (s < nchunks) load_chunk(s, s);
        cp_async_commit();
    }

    for (int c = 0; c < nchunks; ++c) {
        cp_async_wait<NSTAGE - 2>();
        __syncthreads();
        {
            const int cn = c + NSTAGE - 1;
            if (cn < nchunks) load_chunk(cn, cn % NSTAGE);
            cp_async_commit();
        }
        const uint8_t* sK = smem + (c % NSTAGE) * kStageBytes;
        const uint8_t* sV = sK + kChunk * D * 2;

        // S^T (16 tokens x 8*NT heads) = K_rows q^T
        float sacc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) sacc[nt][i] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a[4];
            const int row = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int col = 2 * kk + (lane >> 4);
            ldsm_x4(a, smem_u32(sK + chunk_off<D>(row, col)));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_16816(sacc[nt], a, qf[nt][kk]);
        }

        const int crow = warp * 16 + (lane >> 2);
        const bool ok0 = row_ok[c % NSTAGE][crow] != 0, ok1 = row_ok[c % NSTAGE][crow + 8] != 0;
        uint32_t pf[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const float x0 = ok0 ? sacc[nt][0] * p.scale_log2 : -INFINITY;
            const float x1 = ok0 ? sacc[nt][1] * p.scale_log2 : -INFINITY;
            const float x2 = ok1 ? sacc[nt][2] * p.scale_log2 : -INFINITY;
            const float x3 = ok1 ? sacc[nt][3] * p.scale_log2 : -INFINITY;
            const float mx0 = warp_max_g(fmaxf(x0, x2));
            const float mx1 = warp_max_g(fmaxf(x1, x3));
            const float mn0 = fmaxf(m_run[nt][0], mx0);
            const float mn1 = fmaxf(m_run[nt][1], mx1);
            const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
            const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = fast_exp2(m_run[nt][0] - ref0);
            const float al1 = fast_exp2(m_run[nt][1] - ref1);
            const float p0 = fast_exp2(x0 - ref0), p2 = fast_exp2(x2 - ref0);
            const float p1 = fast_exp2(x1 - ref1), p3 = fast_exp2(x3 - ref1);
            l_run[nt][0] = l_run[nt][0] * al0 + (p0 + p2);
            l_run[nt][1] = l_run[nt][1] * al1 + (p1 + p3);
            m_run[nt][0] = mn0;
            m_run[nt][1] = mn1;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                o[mt][nt][0] *= al0;
                o[mt][nt][1] *= al1;
                o[mt][nt][2] *= al0;
                o[mt][nt][3] *= al1;
            }
            // P^T (tokens x heads) in accumulator layout -> B operand (tokens x heads).
            pf[nt][0] = movmatrix_trans(pack_bf16x2(p0, p1));
            pf[nt][1] = movmatrix_trans(pack_bf16x2(p2, p3));
        }

        // O^T (D x heads) += V^T (D x 16 tokens) P^T (16 tokens x heads)
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            uint32_t a[4];
            const int row = warp * 16 + (lane & 7) + (lane >> 4) * 8;
            const int col = 2 * mt + ((lane >> 3) & 1);
            ldsm_x4_trans(a, smem_u32(sV + chunk_off<D>(row, col)));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_16816(o[mt][nt], a, pf[nt]);
        }
    }
    cp_async_wait<0>();
    __syncthreads();

    // Merge the four warps' partial states through shared memory.
    constexpr int H = 8 * NT;
    float* sm_m = reinterpret_cast<float*>(smem);  // [4][H]
    float* sm_l = sm_m + 4 * H;                     // [4][H]
    float* sm_o = sm_l + 4 * H;                     // [4][H][D]
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const float l0 = warp_sum_g(l_run[nt][0]);
        const float l1 = warp_sum_g(l_run[nt][1]);
        const int j0 = nt * 8 + 2 * (lane & 3);
        if (lane < 4) {
            sm_m[warp * H + j0] = m_run[nt][0];
            sm_m[warp * H + j0 + 1] = m_run[nt][1];
            sm_l[warp * H + j0] = l0;
            sm_l[warp * H + j0 + 1] = l1;
        }
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            const int d0 = mt * 16 + (lane >> 2);
            sm_o[(warp * H + j0) * D + d0] = o[mt][nt][0];
            sm_o[(warp * H + j0 + 1) * D + d0] = o[mt][nt][1];
            sm_o[(warp * H + j0) * D + d0 + 8] = o[mt][nt][2];
            sm_o[(warp * H + j0 + 1) * D + d0 + 8] = o[mt][nt][3];
        }
    }
    __syncthreads();
    for (int e = tid; e < nheads * D; e += kThreads) {
        const int j = e / D, dd = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_m[w * H + j]);
        const float ref = M == -INFINITY ? 0.f : M;
        float acc = 0.f, l = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float f = fast_exp2(sm_m[w * H + j] - ref);
            acc += sm_o[(w * H + j) * D + dd] * f;
            l += sm_l[w * H + j] * f;
        }
        const size_t slot = ((size_t)b * p.hq + h_base + j) * p.max_splits + split;
        p.part_o[slot * D + dd] = acc;
        if (dd == 0) p.part_ml[slot] = make_float2(M, l);
    }
}

template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const SplitParams p, const float* __restrict__ sink,
                                                          __nv_bfloat16* __restrict__ out,
                                                          float* __restrict__ lse) {
    const int h = blockIdx.x, b = blockIdx.y, dd = threadIdx.x;
    const Ranges r = request_ranges(p, b, false);
    const int nvis = visible_count(r);
    const int nsplit = (int)(((long long)nvis + p.split_tokens - 1) / p.split_tokens);
    const size_t base = ((size_t)b * p.hq + h) * p.max_splits;
    const float sg = sink ? sink[h] * ATTN_LOG2E : -INFINITY;
    // the split grid (this launch's programmatic predecessor) has completed and
    // its partials are visible past this point
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float M = sg;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, p.part_ml[base + s].x);
    float o = 0.f, lse_v;
    if (M == -INFINITY || M == INFINITY) {
        // nothing visible and no sink, or an infinite sink taking all the mass
        lse_v = M;
    } else {
        float Z = fast_exp2(sg - M), acc = 0.f;
        for (int s = 0; s < nsplit; ++s) {
            const float2 ml = p.part_ml[base + s];
            const float f = fast_exp2(ml.x - M);
            Z += ml.y * f;
            acc += p.part_o[(base + s) * D + dd] * f;
        }
        o = acc / Z;
        lse_v = (M + log2f(Z)) * ATTN_LN2;
    }
    out[((size_t)b * p.hq + h) * D + dd] = __float2bfloat16_rn(o);
    if (lse && dd == 0) lse[(size_t)b * p.hq + h] = lse_v;
}

// Test hooks: the visible ranges and slots exactly as the split kernel derives them.
__global__ void visible_ranges_kernel(const int32_t* seqlens, int batch, int win_first, int win_last,
                                      int32_t* ranges) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch) return;
    int L = seqlens[b];
    if (L < 0) L = 0;
    const Ranges r = visible_ranges(L - 1, win_first, win_last);
    ranges[4 * b + 0] = r.a0;
    ranges[4 * b + 1] = r.b0;
    ranges[4 * b + 2] = r.a1;
    ranges[4 * b + 3] = r.b1;
}

__global__ void visible_slots_kernel(SplitParams p, int32_t* slots, int max_visible) {
    const int b = blockIdx.y;
    const Ranges r = request_ranges(p, b, threadIdx.x == 0 && blockIdx.x == 0);
    const int nvis = visible_count(r);
    for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < max_visible; v += gridDim.x * blockDim.x) {
        int32_t out = -1;
        if (v < nvis) {
            const int t = visible_token(r, v);
            const int page = p.page_table[(size_t)b * p.max_pages + t / p.page_size];
            if ((unsigned)page < (unsigned)p.num_pages)
                out = page * p.page_size + t % p.page_size;
            else
                raise_status(ATTN_SINK_DEV_PAGE_OOB);
        }
        slots[(size_t)b * max_visible + v] = out;
    }
}

// ---------------------------------------------------------------------------
// Host side.

static int num_sms_cached() {
    static int sms[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 152;
    if (!sms[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        sms[dev] = v > 0 ? v : 152;
    }
    return sms[dev];
}

Plan make_plan(const Args& a) {
    Plan pl;
    pl.nt = a.group <= 8 ? 1 : 2;
    pl.hblocks = (a.group + 8 * pl.nt - 1) / (8 * pl.nt);
    long long cap = (long long)a.max_pages * a.page_size;
    long long nvis_max = cap;
    if (a.win_last > 0) {
        long long w = (long long)(a.win_first > 0 ? a.win_first : 0) + a.win_last;
        nvis_max = w < cap ? w : cap;
    }
    if (nvis_max < 1) nvis_max = 1;
    const long long units = (long long)a.batch * a.hkv * pl.hblocks;
    // Split size: aim at about two waves of resident CTAs (the shared-memory
    // ring allows 4 CTAs per SM at d 64, 2 at d 128), then clamp so that a
    // split streams at least 256 tokens (the ring's fill and drain amortised)
    // and at most 256 KB of K per split (2048 tokens at d 64, 1024 at d 128):
    // longer splits leave too few CTAs, shorter ones are latency-bound waves.
    const long long slots = (long long)num_sms_cached() * (a.head_dim == 64 ? 4 : 2);
    const long long per_unit = (2 * slots + units - 1) / units;  // splits wanted per (request, head block)
    long long sp = (nvis_max + per_unit - 1) / per_unit;
    sp = (sp + kChunk - 1) / kChunk * kChunk;
    const long long sp_max = 2048LL * 64 / a.head_dim;
    if (sp > sp_max) sp = sp_max;
    if (sp < 256) sp = 256;
    const int split = (int)sp;
    pl.split_tokens = split;
    pl.max_splits = (int)((nvis_max + split - 1) / split);
    pl.nvis_max = nvis_max;
    pl.part_o_bytes = (size_t)a.batch * a.hq * pl.max_splits * a.head_dim * sizeof(float);
    pl.part_ml_bytes = (size_t)a.batch * a.hq * pl.max_splits * sizeof(float2);
    return pl;
}

template <int D, int NT, int NSTAGE>
static cudaError_t launch_split(const SplitParams& sp, const Plan& pl, int batch, int hkv, cudaStream_t s) {
    const int smem = NSTAGE * 2 * kChunk * D * 2;
    auto kern = decode_split_kernel<D, NT, NSTAGE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(pl.max_splits, hkv * pl.hblocks, batch);
    kern<<<grid, kThreads, smem, s>>>(sp);
    return cudaGetLastError();
}

cudaError_t launch(const Args& a, const Plan& pl, float* part_o, float2* part_ml, cudaStream_t s) {
    SplitParams sp;
    sp.q = reinterpret_cast<const __nv_bfloat16*>(a.q);
    sp.k_cache = reinterpret_cast<const __nv_bfloat16*>(a.k_cache);
    sp.v_cache = reinterpret_cast<const __nv_bfloat16*>(a.v_cache);
    sp.page_table = a.page_table;
    sp.seqlens = a.seqlens;
    sp.part_o = part_o;
    sp.part_ml = part_ml;
    sp.max_pages = a.max_pages;
    sp.hq = a.hq;
    sp.hkv = a.hkv;
    sp.page_size = a.page_size;
    sp.num_pages = a.num_pages;
    sp.win_first = a.win_first;
    sp.win_last = a.win_last;
    sp.split_tokens = pl.split_tokens;
    sp.max_splits = pl.max_splits;
    sp.hblocks = pl.hblocks;
    sp.group = a.group;
    sp.scale_log2 = a.scale * ATTN_LOG2E;
    sp.page_shift = -1;
    for (int sh = 0; sh < 31; ++sh)
        if ((1 << sh) == a.page_size) sp.page_shift = sh;
    if (a.batch == 0) return cudaSuccess;
    cudaError_t e;
    if (a.head_dim == 64)
        e = pl.nt == 1 ? launch_split<64, 1, 3>(sp, pl, a.batch, a.hkv, s)
                       : launch_split<64, 2, 3>(sp, pl, a.batch, a.hkv, s);
    else
        e = pl.nt == 1 ? launch_split<128, 1, 3>(sp, pl, a.batch, a.hkv, s)
                       : launch_split<128, 2, 3>(sp, pl, a.batch, a.hkv, s);
    if (e != cudaSuccess) return e;
    // The combine starts as a programmatic dependent of the split grid: its
    // launch and CTA set-up overlap the split kernel's last wave.
    auto* out = reinterpret_cast<__nv_bfloat16*>(a.out);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.hq, a.batch);
    cfg.blockDim = dim3(a.head_dim == 64 ? 64 : 128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float* sink = a.sink;
    float* lse = a.lse;
    if (a.head_dim == 64)
        e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<64>, sp, sink, out, lse);
    else
        e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<128>, sp, sink, out, lse);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_visible_ranges(const int32_t* seqlens, int batch, int win_first, int win_last,
                                  int32_t* ranges, cudaStream_t s) {
    if (batch == 0) return cudaSuccess;
    visible_ranges_kernel<<<(batch + 127) / 128, 128, 0, s>>>(seqlens, batch, win_first, win_last, ranges);
    return cudaGetLastError();
}

cudaError_t launch_visible_slots(const int32_t* seqlens, const int32_t* page_table, int max_pages,
                                 int batch, int page_size, int num_pages, int win_first, int win_last,
                                 int32_t* slots, int max_visible, cudaStream_t s) {
    if (batch == 0 || max_visible == 0) return cudaSuccess;
    SplitParams sp = {};
    sp.page_table = page_table;
    sp.seqlens = seqlens;
    sp.max_pages = max_pages;
    sp.page_size = page_size;
    sp.page_shift = -1;
    sp.num_pages = num_pages;
    sp.win_first = win_first;
    sp.win_last = win_last;
    int bx = (max_visible + 255) / 256;
    if (bx > 1024) bx = 1024;
    visible_slots_kernel<<<dim3(bx, batch), 256, 0, s>>>(sp, slots, max_visible);
    return cudaGetLastError();
}

ATTN_DEFINE_STATUS_ACCESSOR(status_exchange)

}  // namespace decode
}  // namespace attn
