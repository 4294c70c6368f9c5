// Backward of varlen attention with a learnable sink (sm_103a).
//
// What it computes (flash-attention PR "feat: Implement Sink Attention", Key
// Changes: the backward pass returns the gradient of the learnable sink):
// with P_ij = e^{s_ij - LSE_i} over the visible keys and D_i = rowsum(dO_i o O_i)
//     dS = P o (dO V^T - D),  dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO,
//     dsink_h = -sum_i e^{sink_h - LSE_i} D_i
// (the sink carries no value vector, so dO_i . dO/dsink = -p_sink,i D_i).
//
// Three kernels:
//  * bwd_preprocess_kernel: D_i per (row, head) and dsink (warp shuffles, one
//    fp32 atomic per block and head).
//  * bwd_main_kernel (tcgen05): one CTA per (128-key tile, KV head, request);
//    it loops over the query heads of the KV group and the 128-row query tiles
//    that see its keys.  Per step five tcgen05 GEMMs:
//        S = Q K^T, dP = dO V^T              (TMEM, 128 x 128 fp32 each)
//        dV += P^T dO, dK += dS^T Q          (TMEM accumulators over the whole loop)
//        dQ  = dS K                          (TMEM; A = dS read from TMEM)
//    Two warpgroups share the elementwise work: thread = (query row, half of the
//    128 key columns), so the row's LSE and D are per-thread scalars.  They
//    write P and scale dS to shared memory in the 128-byte-swizzled layout (read
//    MN-major as P^T / dS^T for dV / dK and K-major for dQ), and add the
//    previous step's dQ tile to an fp32 accumulator with TMA bulk tensor
//    reduce-adds.  dK/dV are summed over the group in TMEM (no atomics).
//  * bwd_dq_convert_kernel: fp32 dQ accumulator -> bf16.
#include <cudaTypedefs.h>

#include "bwd.h"
#include "common.cuh"
#include "sm103.cuh"

namespace attn {
namespace bwd {

using namespace sm103;

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per CTA
constexpr int DH = 64;   // output columns of dQ / dK / dV per main-kernel pass
constexpr int kThreads = 384;
constexpr int kRegsCtrl = 104;
constexpr int kRegsWork = 200;  // 128*104 + 256*200 = 64512 = 384 * 168
constexpr int kWork = 256;      // elementwise threads: warps 4..11
constexpr uint32_t kTile = 128 * 128;  // one 128-byte-swizzled atom: 128 rows x 128 bytes
// Head-dim dependent sizes.  A 128-row operand tile of Q, dO, K or V is D / 64
// atoms (atom a: elements 64a .. 64a + 63 of every row, at byte offset
// a * kTile).  At d 128 the products S and dP run over both atoms, and the main
// kernel runs twice, each pass producing one 64-column half of dQ, dK and dV
// (the TMEM budget -- S, dP, dV, dK, dQ and dS -- fits 64 output columns); the
// Q / dO ring then has one stage to fit shared memory.
template <int D>
struct Cfg {
    static constexpr int kAtoms = D / 64;
    static constexpr uint32_t kOp = kTile * kAtoms;
    static constexpr int kQStages = D == 64 ? 3 : 1;
};
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S, dP (fp32), dV, dK (fp32 accumulators over the whole loop),
// dQ (fp32, one step) and dS (bf16 pairs: column c holds keys 2c and 2c+1), the
// A operand of dQ = dS K read straight from TMEM.
constexpr uint32_t cS = 0, cDP = 128, cDV = 256, cDK = 320, cDQ = 384, cDS = 448;

template <int D>
struct __align__(1024) Smem {
    static constexpr int kQStages = Cfg<D>::kQStages;
    uint8_t k[Cfg<D>::kOp];
    uint8_t v[Cfg<D>::kOp];
    uint8_t q[kQStages][Cfg<D>::kOp];
    uint8_t dout[kQStages][Cfg<D>::kOp];
    uint8_t pb[2 * kTile];   // P  (128 queries x 128 keys): two 64-key atoms of 128-byte rows
    uint8_t dsb[2 * kTile];  // dS (same layout)
    uint8_t dq_stage[2][kTile];  // dQ tile staging: two 32-column fp32 halves, 128-byte swizzled rows
    uint64_t kv_full;
    uint64_t kv_ready;  // K / V rows past the request's last key zeroed (tail key tiles only)
    uint64_t qdo_tail;  // a head's last query tile reaching past the request lands here first
    uint64_t qdo_full[kQStages], qdo_empty[kQStages];
    uint64_t sdp_full, sdp_free, pds_full, mma2_done;  // per step
    uint64_t dq_staged;     // all elementwise threads wrote their part of the dQ tile
    uint64_t dq_stage_free; // the bulk reduce has finished reading the staging buffer
    uint64_t final_bar;  // dV / dK / dQ issuer done
    uint64_t final_sdp;  // S / dP issuer done
    uint32_t tmem_base;
    int abort;
};

struct MainParams {
    const int32_t* cu_q;
    const int32_t* cu_k;
    const float* lse;      // (hq, total_q)
    const float* dvec;     // (hq, total_q)
    float* dq_accum;       // (total_q, hq, d) fp32
    __nv_bfloat16* dk;     // (total_k, hkv, d), rows dk_rs elements apart
    __nv_bfloat16* dv;     // rows dv_rs elements apart
    long long dk_rs, dv_rs;
    int hq, hkv, group, total_q, total_k;
    int win_first, win_last, causal;
    float scale, scale_log2;
    int dhalf;  // output columns 64 * dhalf .. + 63 of dQ, dK, dV (d 128: two passes)
};

// Loads one 128-row operand tile (D / 64 atoms) starting at `row`.
template <int D>
__device__ __forceinline__ void tma_tile(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int head, int row) {
#pragma unroll
    for (int a = 0; a < Cfg<D>::kAtoms; ++a) tma_load_3d(dst + a * kTile, m, bar, 64 * a, head, row);
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    int dummy = 0;
    mbar_wait(bar, parity, &dummy);
}

// Query tiles of one head that see at least one key of [j0, j0 + BN).
struct QRange {
    int lo, hi;  // tile indices [lo, hi)
};

__device__ __forceinline__ QRange query_tiles(int j0, int Lq, int Lk, int causal, int F, int W) {
    QRange r;
    const int nqt = (Lq + BM - 1) / BM;
    const int off = Lk - Lq;
    int row_lo = 0, row_hi = Lq;  // query rows [row_lo, row_hi)
    if (causal) row_lo = max(0, j0 - off);  // pos >= j0
    if (W > 0 && j0 >= F) {
        // keys all past the first window: pos + 1 - W <= j0 + BN - 1
        row_hi = min(Lq, j0 + BN - 1 + W - off);
    }
    if (j0 >= Lk || row_lo >= row_hi) {
        r.lo = r.hi = 0;
        return r;
    }
    r.lo = row_lo / BM;
    r.hi = min(nqt, (row_hi + BM - 1) / BM);
    return r;
}

// P = 2^(S scale log2(e) - LSE log2(e)) and dS = P (dP - D) for 32 key columns of
// one query row, packed to bf16 pairs; kMask zeroes the keys the row does not see
// (c > c_last, or c_first_end <= c < c_win).
template <bool kMask>
__device__ __forceinline__ void p_ds_half(const uint32_t (&sr)[32], const uint32_t (&dr)[32], int col, uint64_t sc2,
                                          uint64_t nl2x2, uint64_t scx2, uint64_t ndx2, int c_last, int c_first_end,
                                          int c_win, uint32_t* pw, uint32_t* dw) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
        const int c = col + e;
        float y0, y1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sc2, nl2x2), y0, y1);
        float p0 = fast_exp2(y0), p1 = fast_exp2(y1);
        if (kMask) {
            if (c > c_last || (c >= c_first_end && c < c_win)) p0 = 0.f;
            if (c + 1 > c_last || (c + 1 >= c_first_end && c + 1 < c_win)) p1 = 0.f;
        }
        const uint64_t ds = f2_mul(f2_pack(p0, p1),
                                   f2_fma(f2_pack(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])), scx2, ndx2));
        float d0, d1;
        f2_unpack(ds, d0, d1);
        pw[e >> 1] = pack_bf16x2(p0, p1);
        dw[e >> 1] = pack_bf16x2(d0, d1);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const MainParams p) {
    using C = Cfg<D>;
    constexpr int kQStages = C::kQStages;
    constexpr uint32_t kOp = C::kOp;
    extern __shared__ uint8_t smem_raw[];
    Smem<D>& S = *reinterpret_cast<Smem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Grid (KV head, request, key tile) with the key tile slowest: causal key
    // tile 0 is seen by every query tile, so launching tiles in increasing order
    // starts the longest CTAs first and leaves short ones for the tail.
    const int kvh = blockIdx.x, b = blockIdx.y, kt = blockIdx.z;

    const int q_start = p.cu_q[b];
    int Lq = p.cu_q[b + 1] - q_start;
    const int k_start = p.cu_k[b];
    int Lk = p.cu_k[b + 1] - k_start;
    if (q_start + Lq > p.total_q || k_start + Lk > p.total_k || Lq < 0 || Lk < 0) {
        if (threadIdx.x == 0 && kt == 0 && kvh == 0) raise_status(ATTN_SINK_DEV_SEQLEN_OOB);
        Lq = max(0, min(Lq, p.total_q - q_start));
        Lk = max(0, min(Lk, p.total_k - k_start));
    }
    const int j0 = kt * BN;
    if (j0 >= Lk) return;
    const int off = Lk - Lq;
    const QRange qr = query_tiles(j0, Lq, Lk, p.causal, p.win_first, p.win_last);
    const int nqt = qr.hi - qr.lo;
    const int T = nqt * p.group;  // steps: (head g, query tile)
    const bool kv_tail = j0 + BN > Lk;  // the key tile reaches past the request's last key

    if (threadIdx.x == 0) {
        mbar_init(&S.kv_full, 1);
        mbar_init(&S.kv_ready, 1);
        mbar_init(&S.qdo_tail, 1);
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(&S.qdo_full[s], 1);
            mbar_init(&S.qdo_empty[s], 1);
        }
        mbar_init(&S.sdp_full, 1);
        mbar_init(&S.sdp_free, kWork);
        mbar_init(&S.pds_full, kWork);
        mbar_init(&S.mma2_done, 1);
        mbar_init(&S.dq_staged, kWork);
        mbar_init(&S.dq_stage_free, 1);
        mbar_init(&S.final_bar, 1);
        mbar_init(&S.final_sdp, 1);
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
            // -------------------------------------------------------- producer
            // (converged warp: every lane waits, lane 0 issues the copies)
            // Rows a tile covers past the request's own rows (another request's, or
            // past the end of the buffers, zero-filled by TMA) enter the products
            // with zero weight, but 0 times a NaN or an infinity would not vanish:
            // the K / V rows past the last key and the Q / dO rows past the last
            // query are zeroed in shared memory before the tensor core reads them
            // (key row r and query row r are the 128 bytes at r * 128, so they
            // form one contiguous range whatever the swizzle).
            auto zero_rows = [&](uint8_t* tile, int r0) {
#pragma unroll
                for (int a = 0; a < C::kAtoms; ++a) {
                    uint4* t4 = reinterpret_cast<uint4*>(tile + a * kTile);
                    for (int c = r0 * 8 + lane; c < BM * 8; c += 32) t4[c] = make_uint4(0u, 0u, 0u, 0u);
                }
            };
            if (lane == 0) {
                prefetch_tmap(&tm_q);
                prefetch_tmap(&tm_k);
                prefetch_tmap(&tm_v);
                prefetch_tmap(&tm_do);
                mbar_expect_tx(&S.kv_full, 2 * kOp);
                tma_tile<D>(S.k, &tm_k, &S.kv_full, kvh, k_start + j0);
                tma_tile<D>(S.v, &tm_v, &S.kv_full, kvh, k_start + j0);
            }
            bool ok = true;
            if (kv_tail) {
                ok = __all_sync(0xffffffffu, mbar_wait(&S.kv_full, 0, abort));
                if (ok) {
                    zero_rows(S.k, Lk - j0);
                    zero_rows(S.v, Lk - j0);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&S.kv_ready);
                }
            }
            int t = 0, g_c = 0, qt_c = 0, tails = 0;
            bool tail_pending = false;
            for (; ok && t < T; ++t) {
                const int st = t % kQStages;
                if (t >= kQStages &&
                    !__all_sync(0xffffffffu, mbar_wait(&S.qdo_empty[st], (t / kQStages - 1) & 1, abort)))
                    break;
                const int h = kvh * p.group + g_c;
                const int q0 = (qr.lo + qt_c) * BM;
                const bool tail = q0 + BM > Lq;
                uint64_t* bar = tail ? &S.qdo_tail : &S.qdo_full[st];
                if (lane == 0) {
                    mbar_expect_tx(bar, 2 * kOp);
                    tma_tile<D>(S.q[st], &tm_q, bar, h, q_start + q0);
                    tma_tile<D>(S.dout[st], &tm_do, bar, h, q_start + q0);
                }
                if (tail) {
                    tail_pending = true;
                    if (!__all_sync(0xffffffffu, mbar_wait(&S.qdo_tail, tails & 1, abort))) break;
                    tail_pending = false;
                    ++tails;
                    zero_rows(S.q[st], Lq - q0);
                    zero_rows(S.dout[st], Lq - q0);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&S.qdo_full[st]);
                }
                if (++qt_c == nqt) {
                    qt_c = 0;
                    ++g_c;
                }
            }
            if (lane == 0) {
                drain_wait(&S.kv_full, 0);
                if (tail_pending) drain_wait(&S.qdo_tail, tails & 1);
                for (int st = 0; st < kQStages; ++st) {
                    const int n = t > st ? (t - st + kQStages - 1) / kQStages : 0;  // loads issued into stage st
                    if (n > 0) drain_wait(&S.qdo_full[st], (n - 1) & 1);
                }
            }
            __syncwarp();
        } else if (warp == 2 && T > 0) {
            // -------------------------------------------------------- dQ reducer
            // (converged warp: every lane waits, lane 0 issues the reduce-adds)
            // Adds each staged dQ tile (two 32-column fp32 halves) to the fp32
            // accumulator with TMA bulk tensor reduce-adds, then frees the stage.
            int g_c = 0, qt_c = 0;
            for (int tt = 0; tt < T; ++tt) {
                if (!__all_sync(0xffffffffu, mbar_wait(&S.dq_staged, tt & 1, abort))) break;
                if (lane == 0) {
                    const int hh = kvh * p.group + g_c;
                    const int qq0 = (qr.lo + qt_c) * BM;
                    tma_reduce_add_3d(&tm_dq, S.dq_stage[0], p.dhalf * DH, hh, q_start + qq0);
                    tma_reduce_add_3d(&tm_dq, S.dq_stage[1], p.dhalf * DH + 32, hh, q_start + qq0);
                    bulk_commit_group();
                    bulk_wait_read_all();
                    mbar_arrive(&S.dq_stage_free);
                }
                __syncwarp();
                if (++qt_c == nqt) {
                    qt_c = 0;
                    ++g_c;
                }
            }
            if (lane == 0) bulk_wait_all();  // the reduce-adds have landed before the CTA exits
            __syncwarp();
        } else if ((warp == 1 || warp == 3) && T > 0) {
            // -------------------------------------------------------- MMA issuers
            // Two issuing warps feed the tensor core independent instruction
            // streams: warp 1 issues each step's S / dP as soon as the
            // elementwise warps have read the previous ones; warp 3 issues the
            // step's dV / dK / dQ once P and dS are in shared memory.  Both run
            // converged (every lane waits; elect.sync picks the issuing lane),
            // and within a stream the independent accumulator chains are
            // interleaved k-step by k-step.
            constexpr uint32_t idSS = idesc_bf16_f32(BM, BN, false, false);  // S, dP: both K-major
            constexpr uint32_t idKV = idesc_bf16_f32(BN, DH, true, true);    // dV, dK: A (P^T, dS^T) MN-major
            constexpr uint32_t idQ = idesc_bf16_f32(BM, DH, false, true);    // dQ: A (dS) K-major, B (K) MN-major
            const uint32_t half_off = (uint32_t)p.dhalf * (kTile >> 4);      // this pass's 64-column atom
            // Descriptor bases; a k-step adds its byte offset / 16 to the address field.
            const uint64_t dk_k = sdesc_sw128(smem_u32(S.k), 16, 1024);        // K, K-major (B of S)
            const uint64_t dv_k = sdesc_sw128(smem_u32(S.v), 16, 1024);        // V, K-major (B of dP)
            const uint64_t dk_mn = sdesc_sw128(smem_u32(S.k), 8192, 1024) + half_off;  // K, MN-major (B of dQ)
            const uint64_t dp_mn = sdesc_sw128(smem_u32(S.pb), kTile, 1024);   // P^T, MN-major (A of dV)
            const uint64_t ds_mn = sdesc_sw128(smem_u32(S.dsb), kTile, 1024);  // dS^T, MN-major (A of dK)
            auto wait_all = [&](uint64_t* bar, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
            };
            bool ok = wait_all(kv_tail ? &S.kv_ready : &S.kv_full, 0);
            if (warp == 1) {
                for (int t = 0; ok && t < T; ++t) {
                    const int st = t % kQStages;
                    if (!(ok = wait_all(&S.qdo_full[st], (t / kQStages) & 1))) break;
                    if (t > 0 && !(ok = wait_all(&S.sdp_free, (t - 1) & 1))) break;
                    tc_fence_after();
                    const uint64_t dq_k = sdesc_sw128(smem_u32(S.q[st]), 16, 1024);
                    const uint64_t ddo_k = sdesc_sw128(smem_u32(S.dout[st]), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {  // 16 head-dim elements = 32 bytes per k-step
                        const uint32_t o = (kk >> 2) * (kTile >> 4) + (kk & 3) * 2;  // atom kk / 4
                        umma_ss_e(tmem + cS, dq_k + o, dk_k + o, idSS, kk > 0);
                        umma_ss_e(tmem + cDP, ddo_k + o, dv_k + o, idSS, kk > 0);
                    }
                    umma_commit_e(&S.sdp_full);
                }
                // Every MMA this warp issued must be complete before TMEM is released.
                umma_commit_e(&S.final_sdp);
                drain_wait(&S.final_sdp, 0);
            } else {
                for (int t = 0; ok && t < T; ++t) {
                    const int st = t % kQStages;
                    // pds_full also means the previous dQ has been read out of TMEM
                    if (!(ok = wait_all(&S.pds_full, t & 1))) break;
                    tc_fence_after();
                    const uint64_t dq_mn = sdesc_sw128(smem_u32(S.q[st]), 8192, 1024) + half_off;
                    const uint64_t ddo_mn = sdesc_sw128(smem_u32(S.dout[st]), 8192, 1024) + half_off;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        // dV / dK: k-step kk runs over query rows 16 kk .. 16 kk + 15 of P / dS
                        // (2048 bytes into the MN-major A and B alike)
                        const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
                        umma_ss_e(tmem + cDV, dp_mn + 128 * kk, ddo_mn + 128 * kk, idKV, acc);
                        umma_ss_e(tmem + cDK, ds_mn + 128 * kk, dq_mn + 128 * kk, idKV, acc);
                        // dQ: k-step kk runs over keys 16 kk .. 16 kk + 15 (dS in TMEM: 8 columns
                        // per step; MN-major K: 2048 bytes per step)
                        umma_ts_e(tmem + cDQ, tmem + cDS + kk * 8, dk_mn + 128 * kk, idQ, kk > 0);
                    }
                    umma_commit_e(&S.mma2_done);
                    umma_commit_e(&S.qdo_empty[st]);
                }
                umma_commit_e(&S.final_bar);
                drain_wait(&S.final_bar, 0);
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsWork));
        // ------------------------------------------------------------ elementwise
        // Lane = query row i of the tile (TMEM lanes of S, dP and dQ) and key row
        // i of the CTA (TMEM lanes of dK, dV); column half ch = keys [64 ch, 64 ch + 64).
        const int q4 = warp & 3;
        const int ch = (warp - 4) >> 2;
        const int i = q4 * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
        const uint64_t scx2 = f2_pack(p.scale, p.scale);
        const int F = p.win_first, W = p.win_last;
        bool ok = true;

        // The dQ tile of step tt (its GEMMs complete) leaves through shared memory:
        // this lane's query row, 32 columns (half ch), is loaded from TMEM while the
        // step's P / dS are stored, then staged; warp 2 adds the staged tile to the
        // fp32 accumulator with TMA bulk reduce-adds.  dS carries the softmax scale,
        // so the values go out as they are.
        uint32_t* const stage_row = reinterpret_cast<uint32_t*>(S.dq_stage[ch] + i * 128);
        // Query rows past the request's end (another request's rows) are staged as
        // zeros: their dS is zero, but times a non-finite key it would not be.
        auto stage_dq = [&](uint32_t (&u)[32], int q0_row) {
            if (q0_row + i >= Lq) {
#pragma unroll
                for (int c = 0; c < 32; ++c) u[c] = 0u;
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(smem_u32(stage_row) + (((c ^ (i & 7))) << 4)),
                             "r"(u[4 * c]), "r"(u[4 * c + 1]), "r"(u[4 * c + 2]), "r"(u[4 * c + 3])
                             : "memory");
            }
        };
        // LSE and D of this lane's query row for head g of the group and query tile
        // qt (+inf / 0 past the request's end and past the last step)
        auto load_row = [&](int g, int qt, float& lse, float& dd) {
            const int row = (qr.lo + qt) * BM + i;
            lse = INFINITY;
            dd = 0.f;
            if (g < p.group && row < Lq) {
                const size_t at = (size_t)(kvh * p.group + g) * p.total_q + q_start + row;
                lse = __ldg(p.lse + at);
                dd = __ldg(p.dvec + at);
            }
        };

        // step t = g_c * nqt + qt_c (head g_c of the group, query tile qt_c)
        int g_c = 0, qt_c = 0;
        int q0_prev = 0;  // first query row of the previous step's tile
        float lse_cur, d_cur;
        load_row(0, 0, lse_cur, d_cur);
        for (int t = 0; t < T; ++t) {
            const int q0 = (qr.lo + qt_c) * BM;
            int g_n = g_c, qt_n = qt_c + 1;
            if (qt_n == nqt) {
                qt_n = 0;
                ++g_n;
            }
            float lse_nxt, d_nxt;
            load_row(g_n, qt_n, lse_nxt, d_nxt);  // in flight while this step computes
            ok = mbar_wait(&S.sdp_full, t & 1, abort);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int rows_valid = min(BM, Lq - q0);
            const int P0 = off + q0, P1 = off + q0 + rows_valid - 1;
            const int jmax = j0 + BN - 1;
            const bool full = (!p.causal || jmax <= P0) && (jmax < Lk) &&
                              (W <= 0 || jmax < F || j0 >= P1 + 1 - W);
            // visible key columns of this query: c <= c_last and (c < c_first_end or c >= c_win)
            const int qpos = off + q0 + i;
            const int c_last = min(Lk - 1, p.causal ? qpos : Lk - 1) - j0;
            const int c_first_end = W > 0 ? F - j0 : BN;
            const int c_win = W > 0 ? qpos + 1 - W - j0 : 0;
            const float nl2 = -lse_cur * ATTN_LOG2E;  // -inf past the end: P = 0 there
            const uint64_t nl2x2 = f2_pack(nl2, nl2);
            const uint64_t ndx2 = f2_pack(-d_cur * p.scale, -d_cur * p.scale);
            uint32_t pw[32], dw[32];  // packed bf16 P and dS of this query row, 64 key columns
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t sr[32], dr[32];
                const uint32_t col = ch * 64 + half * 32;
                tmem_ld32(tmem + lane_base + cS + col, sr);
                tmem_ld32(tmem + lane_base + cDP + col, dr);
                tmem_ld_wait();
                if (half == 1) {  // S / dP fully read: the next step may overwrite them
                    tc_fence_before();
                    mbar_arrive(&S.sdp_free);
                }
                if (full)
                    p_ds_half<false>(sr, dr, col, sc2, nl2x2, scx2, ndx2, c_last, c_first_end, c_win,
                                     pw + half * 16, dw + half * 16);
                else
                    p_ds_half<true>(sr, dr, col, sc2, nl2x2, scx2, ndx2, c_last, c_first_end, c_win,
                                    pw + half * 16, dw + half * 16);
            }
            uint32_t u[32];  // dQ of step t - 1
            if (t > 0) {  // the previous step's GEMMs must be done reading P / dS
                ok = mbar_wait(&S.mma2_done, (t - 1) & 1, abort);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_ld32(tmem + lane_base + cDQ + ch * 32, u);
            }
            // dS of this row's 64 keys into TMEM for dQ = dS K
            tmem_st32(tmem + lane_base + cDS + ch * 32, *reinterpret_cast<uint32_t(*)[32]>(&dw[0]));
            // 64 key columns = atom ch, chunks 0..7 of 16 bytes
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const uint32_t o = ch * kTile + sw128_off(i, cc);
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(smem_u32(S.pb + o)), "r"(pw[4 * cc]),
                             "r"(pw[4 * cc + 1]), "r"(pw[4 * cc + 2]), "r"(pw[4 * cc + 3])
                             : "memory");
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(smem_u32(S.dsb + o)), "r"(dw[4 * cc]),
                             "r"(dw[4 * cc + 1]), "r"(dw[4 * cc + 2]), "r"(dw[4 * cc + 3])
                             : "memory");
            }
            fence_proxy_async_smem();
            tmem_st_wait();
            if (t > 0) tmem_ld_wait();  // dQ of step t - 1 is out of TMEM before the next dQ GEMM
            tc_fence_before();
            mbar_arrive(&S.pds_full);
            if (t > 0) {
                // the bulk reduce of step t - 2 has finished reading the stage
                ok = t == 1 || mbar_wait(&S.dq_stage_free, (t - 2) & 1, abort);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                stage_dq(u, q0_prev);
                fence_proxy_async_smem();
                mbar_arrive(&S.dq_staged);
            }
            q0_prev = q0;
            lse_cur = lse_nxt;
            d_cur = d_nxt;
            g_c = g_n;
            qt_c = qt_n;
        }
        // last step's dQ, then dK (column half 0) / dV (column half 1)
        if (ok && T > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&S.mma2_done, (T - 1) & 1, abort));
            if (ok) {
                tc_fence_after();
                uint32_t u[32];
                tmem_ld32(tmem + lane_base + cDQ + ch * 32, u);
                tmem_ld_wait();
                ok = __all_sync(0xffffffffu, T == 1 || mbar_wait(&S.dq_stage_free, (T - 2) & 1, abort));
                if (ok) {
                    stage_dq(u, q0_prev);
                    fence_proxy_async_smem();
                    mbar_arrive(&S.dq_staged);
                }
            }
        }
        if (ok && T > 0) ok = mbar_wait(&S.final_bar, 0, abort);
        ok = __all_sync(0xffffffffu, ok);
        const bool have = ok && T > 0;
        if (have) tc_fence_after();
        const int kpos = j0 + i;
        const size_t rowoff =
            (size_t)(k_start + kpos) * (size_t)(ch == 0 ? p.dk_rs : p.dv_rs) + (size_t)kvh * D + p.dhalf * DH;
        const uint32_t col = ch == 0 ? cDK : cDV;
        const float f = 1.f;  // dK: the scale rides on dS
        __nv_bfloat16* outp = ch == 0 ? p.dk : p.dv;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t u[32];
            if (have) {  // warp-uniform: every lane takes part in the collective loads
                tmem_ld32(tmem + lane_base + col + half * 32, u);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) u[e] = 0u;
            }
            if (kpos < Lk) {
                uint4* dst = reinterpret_cast<uint4*>(outp + rowoff + half * 32);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(u[8 * c + 0]) * f, __uint_as_float(u[8 * c + 1]) * f);
                    w.y = pack_bf16x2(__uint_as_float(u[8 * c + 2]) * f, __uint_as_float(u[8 * c + 3]) * f);
                    w.z = pack_bf16x2(__uint_as_float(u[8 * c + 4]) * f, __uint_as_float(u[8 * c + 5]) * f);
                    w.w = pack_bf16x2(__uint_as_float(u[8 * c + 6]) * f, __uint_as_float(u[8 * c + 7]) * f);
                    dst[c] = w;
                }
            }
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
// D_i = rowsum(dO_i o O_i) and dsink.  Block: 256 threads, 64 rows of one head;
// 8 threads per row, 16 bytes each.

template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ out,
                                                             const __nv_bfloat16* __restrict__ dout,
                                                             const float* __restrict__ lse,
                                                             const float* __restrict__ sink, float* __restrict__ dvec,
                                                             float* __restrict__ dsink, int total_q, int hq,
                                                             const int32_t* __restrict__ cu_q, int batch) {
    const int h = blockIdx.y;
    // Rows past the last request (cu_q[batch] <= row < total_q) belong to no
    // request: D = 0 and no sink term, whatever the buffers hold there.
    const int rows = min(total_q, max(0, cu_q[batch]));
    const int tid = threadIdx.x;
    const int sub = tid & 7;
    const float sg = sink ? sink[h] : -INFINITY;
    float acc_sink = 0.f;
    for (int rr = 0; rr < 2; ++rr) {
        const int row = blockIdx.x * 64 + rr * 32 + (tid >> 3);
        float d = 0.f;
        if (row < rows) {
            // eight threads per row, D / 8 elements each (16-byte loads)
#pragma unroll
            for (int j = 0; j < D / 64; ++j) {
                const size_t base = ((size_t)row * hq + h) * D + j * 64 + sub * 8;
                const uint4 o = *reinterpret_cast<const uint4*>(out + base);
                const uint4 g = *reinterpret_cast<const uint4*>(dout + base);
                d += bf16_lo(o.x) * bf16_lo(g.x) + bf16_hi(o.x) * bf16_hi(g.x) + bf16_lo(o.y) * bf16_lo(g.y) +
                     bf16_hi(o.y) * bf16_hi(g.y) + bf16_lo(o.z) * bf16_lo(g.z) + bf16_hi(o.z) * bf16_hi(g.z) +
                     bf16_lo(o.w) * bf16_lo(g.w) + bf16_hi(o.w) * bf16_hi(g.w);
            }
        }
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        d += __shfl_xor_sync(0xffffffffu, d, 4);
        if (row < total_q && sub == 0) {
            dvec[(size_t)h * total_q + row] = d;
            if (sink && row < rows) {
                const float l = lse[(size_t)h * total_q + row];
                // probability mass on the sink, e^{sink - LSE}
                float ps;
                if (sg == -INFINITY)
                    ps = 0.f;
                else if (l == INFINITY)
                    ps = 1.f;
                else
                    ps = __expf(sg - l);
                acc_sink += -ps * d;
            }
        }
    }
    if (!sink) return;
    for (int o = 16; o > 0; o >>= 1) acc_sink += __shfl_xor_sync(0xffffffffu, acc_sink, o);
    __shared__ float red[8];
    if ((tid & 31) == 0) red[tid >> 5] = acc_sink;
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int w = 0; w < 8; ++w) s += red[w];
        atomicAdd(dsink + h, s);
    }
}

// acc holds rows of row4 float4 (hq * 64 / 4); dq rows are dq_rs4 uint2 apart.
__global__ void bwd_dq_convert_kernel(const float4* __restrict__ acc, uint2* __restrict__ dq, size_t n4,
                                      int row4, long long dq_rs4) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 v = acc[i];
        const size_t row = i / (size_t)row4, c = i - row * (size_t)row4;
        dq[row * (size_t)dq_rs4 + c] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    }
}

// ---------------------------------------------------------------------------
// Host side

cudaError_t make_map(CUtensorMap* m, const void* base, int d, int heads, long long rows, std::string* what,
                     long long row_stride = 0);
cudaError_t make_map_dq(CUtensorMap* m, const float* base, int d, int heads, long long rows, std::string* what);

size_t workspace_bytes(const Args& a) {
    const size_t acc = (size_t)a.total_q * a.hq * a.head_dim * sizeof(float);
    const size_t dv = (size_t)a.hq * a.total_q * sizeof(float);
    return ((acc + 255) & ~size_t(255)) + dv;
}

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

// (rows, heads, d) bf16 tensor as {d, head, row}; box {64, 1, 128}: one
// 128-byte-swizzled atom per copy.
cudaError_t make_map(CUtensorMap* m, const void* base, int D, int heads, long long rows, std::string* what,
                     long long row_stride) {
    auto fn = encode_fn();
    if (!fn) {
        *what = "cuTensorMapEncodeTiled unavailable";
        return cudaErrorNotSupported;
    }
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)(row_stride > 0 ? row_stride : (long long)D * heads) * 2};
    cuuint32_t box[3] = {64u, 1, 128};
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

// (rows, heads, d) fp32 dQ accumulator as {d, head, row}; box {32, 1, 128}, 128-byte swizzle.
cudaError_t make_map_dq(CUtensorMap* m, const float* base, int D, int heads, long long rows, std::string* what) {
    auto fn = encode_fn();
    if (!fn) {
        *what = "cuTensorMapEncodeTiled unavailable";
        return cudaErrorNotSupported;
    }
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)D * 4 * heads};
    cuuint32_t box[3] = {32, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *what = "cuTensorMapEncodeTiled (dQ) failed (" + std::to_string((int)r) + ")";
        return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

template <int D>
static cudaError_t launch_d(const Args& a, void* workspace, cudaStream_t s, std::string* what) {
    cudaError_t e;
    const size_t acc_bytes = (size_t)a.total_q * a.hq * D * sizeof(float);
    float* dq_accum = static_cast<float*>(workspace);
    float* dvec = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((acc_bytes + 255) & ~size_t(255)));
    if (a.dsink && (e = cudaMemsetAsync(a.dsink, 0, sizeof(float) * a.hq, s)) != cudaSuccess) {
        *what = "memset dsink";
        return e;
    }
    // dK/dV rows of keys no CTA visits (past every request's end) are zero
    // (contiguous outputs only: a strided output shares its rows with other tensors).
    const bool dkv_contig = a.dk_rs <= 0 && a.dv_rs <= 0;
    if (dkv_contig && ((e = cudaMemsetAsync(a.dk, 0, (size_t)a.total_k * a.hkv * D * 2, s)) != cudaSuccess ||
                       (e = cudaMemsetAsync(a.dv, 0, (size_t)a.total_k * a.hkv * D * 2, s)) != cudaSuccess)) {
        *what = "memset dk/dv";
        return e;
    }
    if (a.total_q > 0) {
        if ((e = cudaMemsetAsync(dq_accum, 0, acc_bytes, s)) != cudaSuccess) {
            *what = "memset dq accumulator";
            return e;
        }
        dim3 g1((a.total_q + 63) / 64, a.hq);
        bwd_preprocess_kernel<D><<<g1, 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(a.out),
                                                 reinterpret_cast<const __nv_bfloat16*>(a.dout), a.lse, a.sink,
                                                 dvec, a.dsink, a.total_q, a.hq, a.cu_q, a.batch);
        if ((e = cudaGetLastError()) != cudaSuccess) {
            *what = "preprocess launch";
            return e;
        }
    }
    if (a.total_q > 0 && a.total_k > 0 && a.max_seqlen_k > 0) {
        CUtensorMap tq, tk, tv, tdo, tdq;
        if ((e = make_map(&tq, a.q, D, a.hq, a.total_q, what, a.q_rs)) != cudaSuccess) return e;
        if ((e = make_map(&tk, a.k, D, a.hkv, a.total_k, what, a.k_rs)) != cudaSuccess) return e;
        if ((e = make_map(&tv, a.v, D, a.hkv, a.total_k, what, a.v_rs)) != cudaSuccess) return e;
        if ((e = make_map(&tdo, a.dout, D, a.hq, a.total_q, what)) != cudaSuccess) return e;
        if ((e = make_map_dq(&tdq, dq_accum, D, a.hq, a.total_q, what)) != cudaSuccess) return e;
        MainParams p;
        p.cu_q = a.cu_q;
        p.cu_k = a.cu_k;
        p.lse = a.lse;
        p.dvec = dvec;
        p.dq_accum = dq_accum;
        p.dk = reinterpret_cast<__nv_bfloat16*>(a.dk);
        p.dv = reinterpret_cast<__nv_bfloat16*>(a.dv);
        p.dk_rs = a.dk_rs > 0 ? a.dk_rs : (long long)a.hkv * D;
        p.dv_rs = a.dv_rs > 0 ? a.dv_rs : (long long)a.hkv * D;
        p.hq = a.hq;
        p.hkv = a.hkv;
        p.group = a.hq / a.hkv;
        p.total_q = a.total_q;
        p.total_k = a.total_k;
        p.win_first = a.win_first;
        p.win_last = a.win_last;
        p.causal = a.causal;
        p.scale = a.scale;
        p.scale_log2 = a.scale * ATTN_LOG2E;
        const size_t smem = sizeof(Smem<D>) + 1024;
        if ((e = cudaFuncSetAttribute(bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem)) != cudaSuccess) {
            *what = "smem attribute";
            return e;
        }
        dim3 g2(a.hkv, a.batch, (a.max_seqlen_k + BN - 1) / BN);
        for (int half = 0; half < D / DH; ++half) {  // one pass per 64 output columns
            p.dhalf = half;
            bwd_main_kernel<D><<<g2, kThreads, smem, s>>>(tq, tk, tv, tdo, tdq, p);
            if ((e = cudaGetLastError()) != cudaSuccess) {
                *what = "main launch";
                return e;
            }
        }
    }
    if (a.total_q > 0) {
        const size_t n4 = (size_t)a.total_q * a.hq * D / 4;
        int blocks = (int)((n4 + 255) / 256);
        if (blocks > 152 * 16) blocks = 152 * 16;
        const long long dq_rs = a.dq_rs > 0 ? a.dq_rs : (long long)a.hq * D;
        bwd_dq_convert_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(dq_accum),
                                                    reinterpret_cast<uint2*>(a.dq), n4, a.hq * D / 4, dq_rs / 4);
        if ((e = cudaGetLastError()) != cudaSuccess) {
            *what = "dq convert launch";
            return e;
        }
    }
    return cudaSuccess;
}

cudaError_t launch(const Args& a, void* workspace, size_t ws_bytes, cudaStream_t s, std::string* what) {
    if (a.total_q == 0 && a.total_k == 0) return cudaSuccess;
    if (ws_bytes < workspace_bytes(a)) {
        *what = "workspace too small";
        return cudaErrorInvalidValue;
    }
    return a.head_dim == 128 ? launch_d<128>(a, workspace, s, what) : launch_d<64>(a, workspace, s, what);
}

ATTN_DEFINE_STATUS_ACCESSOR(status_exchange)

}  // namespace bwd
}  // namespace attn
