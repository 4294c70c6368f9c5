// Varlen forward attention with a learnable sink and first/last-window
// selection, on tcgen05 tensor cores (sm_103a).
//
// What it computes (flash-attention PR "feat: Implement Sink Attention",
// Description and Key Changes; sglang PR "openai oss attention sink support
// with trtllm-gen backend", extend path):
//     O_i = sum_j e^{s_ij - m_i} v_j / (e^{sink - m_i} + sum_j e^{s_ij - m_i})
// over the keys j visible to query row i (bottom-right causal, optionally the
// first/last window of sglang PR "To implement attention-sink"), together with
// LSE_i = m_i + ln(...) including the sink.
//
// One CTA = 128 query rows x (two query heads of one KV group, or one head
// when the group size is odd); the two heads share every K/V tile.
//   warp 0      TMA producer: Q once, then K/V tiles into a 3-stage ring
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer:
//               S_h = Q_h K^T (128x128, fp32 in TMEM), O_h += P_h V (128x64)
//   warps 2,3   idle (complete warpgroup 0 for the register split)
//   warps 4..11 two softmax warpgroups, one per head; thread = query row.
// The online softmax starts from m = sink, l = 1 (the sink costs nothing per
// tile).  The running reference max is only moved when a tile's max exceeds
// it by more than 2^8 (then O in TMEM is rescaled in place), which keeps every
// P value <= 256 and leaves the result exact.  P is written to shared memory
// in the 128-byte-swizzled K-major layout the PV product reads.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "prefill.h"
#include "sm103.cuh"

namespace attn {
namespace prefill {

using namespace sm103;

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int D = 64;
constexpr int NSTAGE = 3;
constexpr int kThreads = 384;
// Register split (setmaxnreg): warpgroup 0 (TMA + MMA) gives registers to the
// two softmax warpgroups.  128*56 + 256*224 = 64512 = 384 threads * 168, the
// registers the block is launched with.
constexpr int kRegsCtrl = 56;
constexpr int kRegsSoftmax = 224;
constexpr uint32_t kTile = 128 * 128;  // 128 rows x 128 bytes
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct __align__(1024) Smem {
    uint8_t q[2][kTile];
    uint8_t k[NSTAGE][kTile];
    uint8_t v[NSTAGE][kTile];
    uint8_t p[2][2 * kTile];
    uint64_t q_full;
    uint64_t kv_full[NSTAGE];
    uint64_t kv_empty[NSTAGE];
    uint64_t s_full[2], s_free[2], p_full[2], o_done[2];
    uint64_t final_bar;
    uint32_t tmem_base;
    int abort;
};

struct Params {
    const float* sink;
    const int32_t* cu_q;
    const int32_t* cu_k;
    __nv_bfloat16* out;
    float* lse;
    int hq, group, nslot, n_rt, total_q, total_k;
    int win_first, win_last, causal;
    float scale_log2;
};

// Waits that ignore the abort flag (used only to drain work already in flight
// before shared memory / TMEM are released); still bounded in time.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    int dummy = 0;
    mbar_wait(bar, parity, &dummy);
}

__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hu = blockIdx.x;
    const int rt = p.n_rt - 1 - (int)blockIdx.y;  // heaviest row tiles first
    const int b = blockIdx.z;

    const int q_start = p.cu_q[b];
    int Lq = p.cu_q[b + 1] - q_start;
    const int k_start = p.cu_k[b];
    int Lk = p.cu_k[b + 1] - k_start;
    if (q_start + Lq > p.total_q || k_start + Lk > p.total_k || Lq < 0 || Lk < 0) {
        if (threadIdx.x == 0 && rt == 0 && hu == 0) raise_status(ATTN_SINK_DEV_SEQLEN_OOB);
        Lq = max(0, min(Lq, p.total_q - q_start));
        Lk = max(0, min(Lk, p.total_k - k_start));
    }
    const int qs = rt * BM;
    if (qs >= Lq) return;

    const int nslot = p.nslot;
    const int h0 = hu * nslot;
    const int kvh = h0 / p.group;

    // Tiles of keys visible to at least one valid row of this tile.
    const int off = Lk - Lq;
    const int rows_valid = min(BM, Lq - qs);
    const int P0 = off + qs, P1 = off + qs + rows_valid - 1;
    int n_hi = p.causal ? min(P1 + 1, Lk) : Lk;
    if (n_hi < 0) n_hi = 0;
    const int t_end = (n_hi + BN - 1) / BN;
    int ta = t_end, tb = t_end;
    if (p.win_last > 0) {
        const int f = min(p.win_first, n_hi);
        ta = (f + BN - 1) / BN;
        int lo = P0 + 1 - p.win_last;
        if (lo < 0) lo = 0;
        tb = max(ta, lo / BN);
        if (tb > t_end) tb = t_end;
    }
    const int ntiles = ta + (t_end - tb);

    if (threadIdx.x == 0) {
        mbar_init(&S.q_full, 1);
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&S.kv_full[s], 1);
            mbar_init(&S.kv_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&S.s_full[s], 1);
            mbar_init(&S.s_free[s], 128);
            mbar_init(&S.p_full[s], 128);
            mbar_init(&S.o_done[s], 1);
        }
        mbar_init(&S.final_bar, 1);
        S.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&S.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    volatile int* abort = &S.abort;

    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtrl));
      if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            mbar_expect_tx(&S.q_full, nslot * kTile);
            for (int s = 0; s < nslot; ++s) tma_load_3d(S.q[s], &tm_q, &S.q_full, 0, h0 + s, q_start + qs);
            int it = 0;
            for (; it < ntiles; ++it) {
                const int st = it % NSTAGE;
                if (it >= NSTAGE && !mbar_wait(&S.kv_empty[st], ((it / NSTAGE) - 1) & 1, abort)) break;
                const int t = it < ta ? it : tb + (it - ta);
                mbar_expect_tx(&S.kv_full[st], 2 * kTile);
                tma_load_3d(S.k[st], &tm_k, &S.kv_full[st], 0, kvh, k_start + t * BN);
                tma_load_3d(S.v[st], &tm_v, &S.kv_full[st], 0, kvh, k_start + t * BN);
            }
            // Drain: every copy issued must have landed before the CTA exits.
            drain_wait(&S.q_full, 0);
            for (int st = 0; st < NSTAGE; ++st) {
                const int n = it > st ? (it - st + NSTAGE - 1) / NSTAGE : 0;
                if (n > 0) drain_wait(&S.kv_full[st], (n - 1) & 1);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && ntiles > 0) {
            constexpr uint32_t idS = idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t idO = idesc_bf16_f32(BM, D, false, true);
            const uint32_t sq = smem_u32(S.q[0]), sk = smem_u32(S.k[0]), sv = smem_u32(S.v[0]);
            const uint32_t sp = smem_u32(S.p[0]);
            auto issue_S = [&](int it, int slot) {
                const uint32_t kb = sk + (it % NSTAGE) * kTile;
                const uint32_t qb = sq + slot * kTile;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma_ss(tmem + slot * BN, sdesc_sw128(qb + kk * 32, 16, 1024), sdesc_sw128(kb + kk * 32, 16, 1024),
                            idS, kk > 0);
                umma_commit(&S.s_full[slot]);
            };
            auto issue_PV = [&](int it, int slot) {
                const uint32_t vb = sv + (it % NSTAGE) * kTile;
                const uint32_t pb = sp + slot * 2 * kTile;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    umma_ss(tmem + 2 * BN + slot * D,
                            sdesc_sw128(pb + (kk >> 2) * kTile + (kk & 3) * 32, 16, 1024),
                            sdesc_sw128(vb + kk * 2048, 8192, 1024), idO, (it > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&S.o_done[slot]);
            };
            bool ok = mbar_wait(&S.q_full, 0, abort) && mbar_wait(&S.kv_full[0], 0, abort);
            if (ok) {
                tc_fence_after();
                for (int s = 0; s < nslot; ++s) issue_S(0, s);
            }
            for (int it = 0; ok && it < ntiles; ++it) {
                const int nx = it + 1;
                // Both heads' next S as soon as their softmax has read this S
                // (it runs on the tensor core while the softmax works) ...
                if (nx < ntiles) {
                    if (!(ok = mbar_wait(&S.kv_full[nx % NSTAGE], (nx / NSTAGE) & 1, abort))) break;
                    for (int s = 0; s < nslot && ok; ++s) {
                        if (!(ok = mbar_wait(&S.s_free[s], it & 1, abort))) break;
                        tc_fence_after();
                        issue_S(nx, s);
                    }
                    if (!ok) break;
                }
                // ... then each head's P V once its P is in shared memory.
                for (int s = 0; s < nslot && ok; ++s) {
                    if (!(ok = mbar_wait(&S.p_full[s], it & 1, abort))) break;
                    tc_fence_after();
                    issue_PV(it, s);
                }
                if (ok) umma_commit(&S.kv_empty[it % NSTAGE]);
            }
            // Every MMA issued must be complete before TMEM is released.
            umma_commit(&S.final_bar);
            drain_wait(&S.final_bar, 0);
        }
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ------------------------------------------------------------ softmax
        const int slot = (warp - 4) >> 2;
        if (slot < nslot) {
            const int q4 = warp & 3;
            const int r = q4 * 32 + lane;
            const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
            const uint32_t tS = tmem + lane_base + slot * BN;
            const uint32_t tO = tmem + lane_base + 2 * BN + slot * D;
            const int h = h0 + slot;
            const float sg = p.sink ? p.sink[h] * ATTN_LOG2E : -INFINITY;
            const float sl2 = p.scale_log2;
            float m_ref = sg;
            float l = sg == -INFINITY ? 0.f : 1.f;
            const int pos = off + qs + r;
            uint8_t* prow = S.p[slot];
            bool ok = true;
            for (int it = 0; it < ntiles; ++it) {
                const int t = it < ta ? it : tb + (it - ta);
                const int j0 = t * BN;
                ok = mbar_wait(&S.s_full[slot], it & 1, abort);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t s[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, s[c]);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&S.s_free[slot]);

                const int jmax = j0 + BN - 1;
                const bool full = (!p.causal || jmax <= P0) && (jmax < Lk) &&
                                  (p.win_last <= 0 || jmax < p.win_first || j0 >= P1 + 1 - p.win_last);
                if (!full) {
                    int c_hi = p.causal ? pos - j0 + 1 : BN;
                    c_hi = min(c_hi, Lk - j0);
                    const int f_hi = p.win_last > 0 ? p.win_first - j0 : BN;
                    const int w_lo = p.win_last > 0 ? pos + 1 - p.win_last - j0 : 0;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int cc = c * 32 + i;
                            const bool vis = cc < c_hi && (cc < f_hi || cc >= w_lo);
                            if (!vis) s[c][i] = __float_as_uint(-INFINITY);
                        }
                }
                // Row max: eight independent 3-input max chains of 16 values.
                float mc[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t* v = &s[k >> 1][(k & 1) * 16];
                    float m = max3f(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
#pragma unroll
                    for (int i = 3; i < 15; i += 2) m = max3f(m, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
                    mc[k] = fmaxf(m, __uint_as_float(v[15]));
                }
                const float mx =
                    max3f(max3f(mc[0], mc[1], mc[2]), max3f(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
                const float m_new = fmaxf(m_ref, mx * sl2);
                const bool resc = m_new > m_ref + kRescaleThreshold;
                const float alpha = resc ? fast_exp2(m_ref - m_new) : 1.f;
                bool waited = false;
                if (it > 0 && __any_sync(0xffffffffu, resc)) {
                    // O holds PV of earlier tiles: wait for the last one, then rescale in TMEM.
                    ok = mbar_wait(&S.o_done[slot], (it - 1) & 1, abort);
                    if (!__all_sync(0xffffffffu, ok)) {
                        ok = false;
                        break;
                    }
                    waited = true;
                    tc_fence_after();
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t o[32];
                        tmem_ld32(tO + half * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + half * 32, o);
                    }
                    tmem_st_wait();
                }
                if (resc) {
                    l *= alpha;
                    m_ref = m_new;
                }
                const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
                if (it > 0 && !waited) {
                    // the previous PV must be done reading this head's P buffer
                    ok = mbar_wait(&S.o_done[slot], (it - 1) & 1, abort);
                    if (!__all_sync(0xffffffffu, ok)) {
                        ok = false;
                        break;
                    }
                }
                // P = 2^(s*scale*log2e - m): packed fp32x2 FMA, MUFU ex2, packed partial sums.
                const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(-m_use, -m_use);
                uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int cc = 0; cc < 16; ++cc) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i0 = cc * 8 + 2 * e;
                        const uint64_t y = f2_fma(f2_pack(__uint_as_float(s[i0 >> 5][i0 & 31]),
                                                          __uint_as_float(s[(i0 + 1) >> 5][(i0 + 1) & 31])),
                                                  sc2, nm2);
                        float y0, y1;
                        f2_unpack(y, y0, y1);
                        const float x0 = fast_exp2(y0), x1 = fast_exp2(y1);
                        acc2[e] = f2_add(acc2[e], f2_pack(x0, x1));
                        w[e] = pack_bf16x2(x0, x1);
                    }
                    uint8_t* dst = prow + (cc >> 3) * kTile + sw128_off(r, cc & 7);
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(smem_u32(dst)), "r"(w[0]),
                                 "r"(w[1]), "r"(w[2]), "r"(w[3])
                                 : "memory");
                }
                float rs = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float lo, hi;
                    f2_unpack(acc2[e], lo, hi);
                    rs += lo + hi;
                }
                l += rs;
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&S.p_full[slot]);
            }

            // ---------------------------------------------------------- epilogue
            if (ok && ntiles > 0) ok = mbar_wait(&S.o_done[slot], (ntiles - 1) & 1, abort);
            ok = __all_sync(0xffffffffu, ok);
            const bool have = ok && ntiles > 0;
            if (have) tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int row = q_start + qs + r;
            const bool store = r < rows_valid && ok;
            uint4* dst = reinterpret_cast<uint4*>(p.out + ((size_t)row * p.hq + h) * D);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t u[32];
                if (have) {  // warp-uniform: every lane takes part in the collective load
                    tmem_ld32(tO + half * 32, u);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) u[i] = 0u;
                }
                if (store) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(u[8 * c + 0]) * inv, __uint_as_float(u[8 * c + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(u[8 * c + 2]) * inv, __uint_as_float(u[8 * c + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(u[8 * c + 4]) * inv, __uint_as_float(u[8 * c + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(u[8 * c + 6]) * inv, __uint_as_float(u[8 * c + 7]) * inv);
                        dst[half * 4 + c] = w;
                    }
                }
            }
            if (store && p.lse) p.lse[(size_t)h * p.total_q + row] = l > 0.f ? (m_ref + log2f(l)) * ATTN_LN2 : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// (rows, heads, 64) bf16 tensor viewed as a 3-D map {d, head, row}; box {64, 1, box_rows}.
cudaError_t make_map(CUtensorMap* m, const void* base, int heads, long long rows, int box_rows,
                     std::string* what) {
    auto fn = encode_fn();
    if (!fn) {
        *what = "cuTensorMapEncodeTiled unavailable";
        return cudaErrorNotSupported;
    }
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * 2 * heads};
    cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *what = "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")";
        return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t s, std::string* what) {
    if (a.total_q == 0) return cudaSuccess;
    CUtensorMap tq, tk, tv;
    cudaError_t e;
    if ((e = make_map(&tq, a.q, a.hq, a.total_q, BM, what)) != cudaSuccess) return e;
    if ((e = make_map(&tk, a.k, a.hkv, a.total_k, BN, what)) != cudaSuccess) return e;
    if ((e = make_map(&tv, a.v, a.hkv, a.total_k, BN, what)) != cudaSuccess) return e;
    Params p;
    p.sink = a.sink;
    p.cu_q = a.cu_q;
    p.cu_k = a.cu_k;
    p.out = reinterpret_cast<__nv_bfloat16*>(a.out);
    p.lse = a.lse;
    p.hq = a.hq;
    p.group = a.hq / a.hkv;
    p.nslot = (p.group % 2 == 0) ? 2 : 1;
    p.n_rt = (a.max_seqlen_q + BM - 1) / BM;
    p.total_q = a.total_q;
    p.total_k = a.total_k;
    p.win_first = a.win_first;
    p.win_last = a.win_last;
    p.causal = a.causal;
    p.scale_log2 = a.scale * ATTN_LOG2E;
    const size_t smem = sizeof(Smem) + 1024;
    e = cudaFuncSetAttribute(fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
        *what = "smem attribute";
        return e;
    }
    dim3 grid(a.hq / p.nslot, p.n_rt, a.batch);
    fwd_kernel<<<grid, kThreads, smem, s>>>(tq, tk, tv, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) *what = "launch";
    return e;
}

ATTN_DEFINE_STATUS_ACCESSOR(status_exchange)

}  // namespace prefill
}  // namespace attn
