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
//    fp32 atomic per block and head); it writes each row's -LSE / scale and -D
//    as a 32-byte record of bf16 parts for the main kernel, and clears the
//    fp32 dQ accumulator.
//  * bwd_main_kernel (tcgen05): one CTA per (128-key tile, KV head, request);
//    it loops over the query heads of the KV group and the 128-row query tiles
//    that see its keys.  Per step five tcgen05 GEMMs, in the key-major
//    orientation (a TMEM lane is a key):
//        S^T = K Q^T, dP^T = V dO^T          (TMEM, 128 keys x 128 queries, fp32)
//        dV += P^T dO, dK += dS^T Q          (A = P^T / dS^T read from TMEM;
//                                             accumulated over the whole loop)
//        dQ  = dS K                          (A = dS from shared memory)
//    The per-query terms ride in the GEMMs: one more 16-wide k-step multiplies
//    a block of ones (keys x 16) by the tile's 128 records (TMA-loaded with Q
//    and dO), each holding -LSE / scale and -D of a query split into three bf16
//    parts, so S^T comes out as S - LSE / scale and dP^T as dP - D.  Sixteen
//    warps: a producer, two MMA issuers and a dQ reducer; two warpgroups for
//    the elementwise work (thread = key x half of the 128 query columns, no
//    per-query data to fetch), which write P^T and dS^T to TMEM as bf16 pairs
//    and dS to shared memory once (the MN-major A of dQ); and one warpgroup
//    that moves each dQ tile from TMEM to a staging buffer, from where TMA
//    bulk tensor reduce-adds add it to an fp32 accumulator.  dK / dV are summed
//    over the group in TMEM (no atomics); dS leaves out the softmax scale,
//    which dK and dQ take on their way out.  Head dim 64 runs
//    bwd_main_kernel (128-row query steps), head dim 128 bwd_main128_kernel
//    (64-row query steps, so that every product fits TMEM at full width).
//  * bwd_dq_convert_kernel: fp32 dQ accumulator times the softmax scale -> bf16.
#include <cudaTypedefs.h>

#include "bwd.h"
#include "common.cuh"
#include "sm103.cuh"

namespace attn {
namespace bwd {

using namespace sm103;

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per CTA
constexpr int DH = 64;   // head dim of bwd_main_kernel (bwd_main128_kernel takes 128)
constexpr int kThreads = 512;
// Registers per thread after the role split (the launch gives 128 to each of the
// 512 threads): 128 * 136 + 256 * 160 + 128 * 56 = 65536.
constexpr int kRegsCtrl = 136;   // warps 0..3: producer, MMA issuers, dQ reducer
constexpr int kRegsWork = 160;   // warps 4..11: elementwise
constexpr int kRegsStage = 56;   // warps 12..15: dQ stagers
constexpr int kWork = 256;       // elementwise threads
constexpr int kStage = 128;      // dQ stager threads
constexpr uint32_t kTile = 128 * 128;  // one 128-byte-swizzled atom: 128 rows x 128 bytes
// Sizes of bwd_main_kernel (head dim 64): a 128-row operand tile of Q, dO, K or
// V is one 128-byte-swizzled atom; the Q / dO ring has three stages.
template <int D>
struct Cfg {
    static_assert(D == 64, "bwd_main_kernel is the head-dim-64 kernel");
    static constexpr int kAtoms = 1;
    static constexpr uint32_t kOp = kTile;
    static constexpr int kQStages = 3;
};
constexpr uint32_t kTmemCols = 512;
// TMEM columns.  Lane = key for S^T, dP^T (fp32, column = query), dV, dK (fp32
// accumulators over the whole loop) and dS^T (bf16 pairs: column c holds
// queries 2c and 2c + 1); lane = query for dQ (fp32, one step).  P^T (bf16
// pairs) is written over the dP^T columns its thread has already read: the
// query half h at cDP + 64 h, 32 columns.  So the next S^T waits only for the
// elementwise warps to read this one, and the next dP^T for dV, which leaves
// it a whole P computation of slack.
constexpr uint32_t cS = 0, cDP = 128, cDV = 256, cDK = 320, cDQ = 384, cDS = 448;
// One 128-row K-major operand of a single k-step (16 bf16 = 32 bytes per row) in
// the 32-byte-swizzled layout.
constexpr uint32_t kAug = 128 * 32;
// Per-query record (the B of the extra k-step): bf16 elements 0..2 hold
// -LSE / scale as h1 + h2 + h3 (x - h1 and its remainder are exact in fp32; an
// infinite value is stored as +-1e30), elements 8..10 hold -D the same way, the
// rest are zero.
constexpr int kRec = 16;

template <int D>
struct __align__(1024) Smem {
    static constexpr int kQStages = Cfg<D>::kQStages;
    uint8_t k[Cfg<D>::kOp];
    uint8_t v[Cfg<D>::kOp];
    uint8_t q[kQStages][Cfg<D>::kOp];
    uint8_t dout[kQStages][Cfg<D>::kOp];
    uint8_t dsb[2 * kTile];       // dS: 128 key rows x 128 queries (two 64-query atoms), the MN-major A of dQ
    uint8_t dq_stage[2][kTile];   // dQ tile staging: two 32-column fp32 halves, 128-byte swizzled rows
    // The extra k-step of S^T and dP^T: A = ones_lse (1 in elements 0..2 of
    // every key row) or ones_d (1 in elements 8..10), B = rec (the tile's
    // per-query records).
    uint8_t ones_lse[kAug];
    uint8_t ones_d[kAug];
    uint8_t rec[kQStages][kAug];
    uint64_t kv_full;
    uint64_t kv_ready;  // K / V rows past the request's last key zeroed (tail key tiles only)
    uint64_t qdo_tail;  // a head's last query tile reaching past the request lands here first
    uint64_t qdo_full[kQStages], qdo_empty[kQStages];
    uint64_t s_full, dp_full;     // per step: S^T / dP^T in TMEM
    uint64_t s_free, p_full;      // S^T read out; dP^T read out and P^T written over it
    uint64_t pv_done;             // dV has read P^T (the dP^T columns are free again)
    uint64_t ds_full, mma2_done;  // dS^T / dS written; dK and dQ done
    uint64_t dq_read;             // the stagers have read dQ out of TMEM
    uint64_t dq_staged;           // the stagers have written the dQ tile
    uint64_t dq_stage_free;       // the bulk reduce has finished reading the staging buffer
    uint64_t final_bar;  // dV / dK / dQ issuer done
    uint64_t final_sdp;  // S^T / dP^T issuer done
    uint32_t tmem_base;
    int abort;
};

struct MainParams {
    const int32_t* cu_q;
    const int32_t* cu_k;
    __nv_bfloat16* dk;     // (total_k, hkv, d), rows dk_rs elements apart
    __nv_bfloat16* dv;     // rows dv_rs elements apart
    long long dk_rs, dv_rs;
    int hq, hkv, group, total_q, total_k;
    int batch, n_kt;  // requests; key tiles of the longest request
    int win_first, win_last, causal;
    float scale, scale_log2;
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

// Query tiles (of `rows` rows) of one head that see at least one key of [j0, j0 + BN).
// Launch order of the key-tile CTAs (a 1-D grid of hkv * batch * n_kt).  Under
// causal masking key tile 0 is seen by every query tile and the last one by
// few, so the long CTAs must start first: tile-major order (key tile slowest)
// does that.  The CTAs of one (KV head, request) also re-read the same Q / dO
// tiles and add into the same dQ rows, which stay in L2 only while those CTAs
// run close together in time; kBand > 0 keeps them together with bands of
// kBand key tiles taken in increasing order, each band walking the (KV head,
// request) pairs with the band's key tiles of one pair adjacent, and the last
// kBand key tiles (the shortest CTAs) tile-major for the tail.  Measured on
// the B 2 x 8192 causal step: bands of 16 cut the d 64 kernel's DRAM traffic
// from 3.8 to 3.0 GB but cost it 4 % in time, and gain the d 128 kernel about
// 1 %, so bwd_main_kernel runs tile-major and bwd_main128_kernel in bands.
struct CtaTile {
    int kvh, b, kt;
};
template <int kBand>
__device__ __forceinline__ CtaTile cta_tile(int i, int hkv, int batch, int n_kt) {
    const int n_grp = hkv * batch;
    const int tail_from = (kBand > 0 && n_kt > 2 * kBand) ? n_kt - kBand : 0;
    const int head = tail_from * n_grp;
    int grp, kt;
    if (i < head) {
        const int band = i / (kBand * n_grp);
        const int wb = min(kBand, tail_from - band * kBand);
        const int r = i - band * kBand * n_grp;
        grp = r / wb;
        kt = band * kBand + r % wb;
    } else {
        const int r = i - head;
        kt = tail_from + r / n_grp;
        grp = r % n_grp;
    }
    return {grp % hkv, grp / hkv, kt};
}

struct QRange {
    int lo, hi;  // tile indices [lo, hi)
};

__device__ __forceinline__ QRange query_tiles(int j0, int Lq, int Lk, int causal, int F, int W, int rows = BM) {
    QRange r;
    const int nqt = (Lq + rows - 1) / rows;
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
    r.lo = row_lo / rows;
    r.hi = min(nqt, (row_hi + rows - 1) / rows);
    return r;
}

// P = 2^((S - LSE / scale) scale log2(e)) for the 32 query columns c0 .. c0 + 31
// of one key (in place: pr holds the shifted S^T on entry, P in fp32 on exit)
// and its bf16 pairs into pw[c0 / 2 ..]; kMask zeroes the columns e outside
// [lo, hi] (a select: their shifted S may be anything).
template <bool kMask, int c0>
__device__ __forceinline__ void p_cols(uint32_t (&pr)[32], uint64_t sc2, int lo, int hi, uint32_t (&pw)[32]) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
        float y0, y1;
        f2_unpack(f2_mul(f2_pack(__uint_as_float(pr[e]), __uint_as_float(pr[e + 1])), sc2), y0, y1);
        float p0 = fast_exp2(y0), p1 = fast_exp2(y1);
        if (kMask) {
            if (c0 + e < lo || c0 + e > hi) p0 = 0.f;
            if (c0 + e + 1 < lo || c0 + e + 1 > hi) p1 = 0.f;
        }
        pr[e] = __float_as_uint(p0);
        pr[e + 1] = __float_as_uint(p1);
        pw[(c0 + e) >> 1] = pack_bf16x2(p0, p1);
    }
}

// dS / scale = P (dP - D) for the 32 query columns c0 .. c0 + 31 of one key (pr:
// their P, dr: their shifted dP^T), as bf16 pairs into dw[c0 / 2 ..]; kMask
// zeroes the columns e outside [lo, hi] (whose dP - D may be anything).
template <bool kMask, int c0>
__device__ __forceinline__ void ds_cols(const uint32_t (&pr)[32], const uint32_t (&dr)[32], int lo, int hi,
                                        uint32_t (&dw)[32]) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
        float a0, a1;
        f2_unpack(f2_mul(f2_pack(__uint_as_float(pr[e]), __uint_as_float(pr[e + 1])),
                         f2_pack(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1]))),
                  a0, a1);
        if (kMask) {
            if (c0 + e < lo || c0 + e > hi) a0 = 0.f;
            if (c0 + e + 1 < lo || c0 + e + 1 > hi) a1 = 0.f;
        }
        dw[(c0 + e) >> 1] = pack_bf16x2(a0, a1);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_rec,
                    const MainParams p) {
    using C = Cfg<D>;
    constexpr int kQStages = C::kQStages;
    constexpr uint32_t kOp = C::kOp;
    extern __shared__ uint8_t smem_raw[];
    Smem<D>& S = *reinterpret_cast<Smem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const CtaTile ct = cta_tile<0>(blockIdx.x, p.hkv, p.batch, p.n_kt);
    const int kvh = ct.kvh, b = ct.b, kt = ct.kt;

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
        mbar_init(&S.s_full, 1);
        mbar_init(&S.dp_full, 1);
        // the elementwise and stager warps arrive once per warp
        mbar_init(&S.s_free, kWork / 32);
        mbar_init(&S.p_full, kWork / 32);
        mbar_init(&S.pv_done, 1);
        mbar_init(&S.ds_full, kWork / 32);
        mbar_init(&S.mma2_done, 1);
        mbar_init(&S.dq_read, kStage / 32);
        mbar_init(&S.dq_staged, kStage / 32);
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
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsCtrl));
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
                prefetch_tmap(&tm_rec);
                mbar_expect_tx(&S.kv_full, 2 * kOp);
                tma_tile<D>(S.k, &tm_k, &S.kv_full, kvh, k_start + j0);
                tma_tile<D>(S.v, &tm_v, &S.kv_full, kvh, k_start + j0);
            }
            {
                // The two ones blocks.  Row j is 32 bytes at j * 32; the 32-byte
                // swizzle stores its 16-byte half c at half c ^ (bit 2 of j).  They
                // are read only by MMAs that wait on a barrier this warp's lane 0
                // arrives on after the fence below.
                const uint4 one = make_uint4(0x3F803F80u, 0x00003F80u, 0u, 0u);  // bf16 1, 1, 1, 0 ...
                const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
                for (int c = lane; c < (int)(kAug / 16); c += 32) {
                    const int j = c >> 1, half = (c & 1) ^ ((j >> 2) & 1);  // logical half stored here
                    reinterpret_cast<uint4*>(S.ones_lse)[c] = half == 0 ? one : zero;
                    reinterpret_cast<uint4*>(S.ones_d)[c] = half == 1 ? one : zero;
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            bool ok = true;
            if (kv_tail) {
                ok = mbar_wait_warp(&S.kv_full, 0, abort);
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
            uint32_t tail_last = 0;  // bit st: the last load into stage st went through qdo_tail
            for (; ok && t < T; ++t) {
                const int st = t % kQStages;
                if (t >= kQStages &&
                    !mbar_wait_warp(&S.qdo_empty[st], (t / kQStages - 1) & 1, abort))
                    break;
                const int h = kvh * p.group + g_c;
                const int q0 = (qr.lo + qt_c) * BM;
                const bool tail = q0 + BM > Lq;
                uint64_t* bar = tail ? &S.qdo_tail : &S.qdo_full[st];
                if (lane == 0) {
                    mbar_expect_tx(bar, 2 * kOp + kAug);
                    tma_tile<D>(S.q[st], &tm_q, bar, h, q_start + q0);
                    tma_tile<D>(S.dout[st], &tm_do, bar, h, q_start + q0);
                    tma_load_3d(S.rec[st], &tm_rec, bar, 0, h, q_start + q0);
                }
                tail_last = tail ? (tail_last | (1u << st)) : (tail_last & ~(1u << st));
                if (tail) {
                    tail_pending = true;
                    if (!mbar_wait_warp(&S.qdo_tail, tails & 1, abort)) break;
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
                // the copies in flight land before the CTA exits
                drain_wait(&S.kv_full, 0);
                if (tail_pending) drain_wait(&S.qdo_tail, tails & 1);
                for (int st = 0; st < kQStages; ++st) {
                    const int n = t > st ? (t - st + kQStages - 1) / kQStages : 0;  // loads issued into stage st
                    if (n > 0 && !((tail_last >> st) & 1u)) drain_wait(&S.qdo_full[st], (n - 1) & 1);
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
                if (!mbar_wait_warp(&S.dq_staged, tt & 1, abort)) break;
                if (lane == 0) {
                    const int hh = kvh * p.group + g_c;
                    const int qq0 = (qr.lo + qt_c) * BM;
                    tma_reduce_add_3d(&tm_dq, S.dq_stage[0], 0, hh, q_start + qq0);
                    tma_reduce_add_3d(&tm_dq, S.dq_stage[1], 32, hh, q_start + qq0);
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
            // streams: warp 1 issues each step's S^T once the elementwise warps
            // have read the previous one, and dP^T once dV has read the previous
            // P^T (written over the dP^T columns); warp 3 issues dV once P^T is in
            // TMEM, then dK / dQ once dS^T / dS are written and the stagers have
            // read the previous dQ.  Both run converged (every lane waits;
            // elect.sync picks the issuing lane), and dK / dQ are interleaved
            // k-step by k-step.
            constexpr uint32_t idSS = idesc_bf16_f32(BN, BM, false, false);  // S^T, dP^T: both K-major
            constexpr uint32_t idKV = idesc_bf16_f32(BN, DH, false, true);   // dV, dK: A in TMEM, B (dO, Q) MN-major
            constexpr uint32_t idQ = idesc_bf16_f32(BM, DH, true, true);     // dQ: A (dS) and B (K) MN-major
            // Descriptor bases; a k-step adds its byte offset / 16 to the address field.
            const uint64_t dk_k = sdesc_sw128(smem_u32(S.k), 16, 1024);        // K, K-major (A of S^T)
            const uint64_t dv_k = sdesc_sw128(smem_u32(S.v), 16, 1024);        // V, K-major (A of dP^T)
            const uint64_t d_ones_lse = sdesc_sw32(smem_u32(S.ones_lse));      // A of the extra k-step of S^T
            const uint64_t d_ones_d = sdesc_sw32(smem_u32(S.ones_d));          // ... and of dP^T
            const uint64_t dk_mn = sdesc_sw128(smem_u32(S.k), 8192, 1024);     // K, MN-major (B of dQ)
            const uint64_t ds_mn = sdesc_sw128(smem_u32(S.dsb), kTile, 1024);  // dS, MN-major (A of dQ)
            auto wait_all = [&](uint64_t* bar, uint32_t parity) { return mbar_wait_warp(bar, parity, abort); };
            bool ok = wait_all(kv_tail ? &S.kv_ready : &S.kv_full, 0);
            if (warp == 1) {
                for (int t = 0; ok && t < T; ++t) {
                    const int st = t % kQStages;
                    if (!(ok = wait_all(&S.qdo_full[st], (t / kQStages) & 1))) break;
                    if (t > 0 && !(ok = wait_all(&S.s_free, (t - 1) & 1))) break;
                    tc_fence_after();
                    const uint64_t dq_k = sdesc_sw128(smem_u32(S.q[st]), 16, 1024);
                    const uint64_t ddo_k = sdesc_sw128(smem_u32(S.dout[st]), 16, 1024);
                    const uint64_t drec = sdesc_sw32(smem_u32(S.rec[st]));
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {  // 16 head-dim elements = 32 bytes per k-step
                        const uint32_t o = (kk >> 2) * (kTile >> 4) + (kk & 3) * 2;  // atom kk / 4
                        umma_ss_e(tmem + cS, dk_k + o, dq_k + o, idSS, kk > 0);
                    }
                    umma_ss_e(tmem + cS, d_ones_lse, drec, idSS, 1u);  // - LSE / scale
                    umma_commit_e(&S.s_full);
                    if (t > 0 && !(ok = wait_all(&S.pv_done, (t - 1) & 1))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t o = (kk >> 2) * (kTile >> 4) + (kk & 3) * 2;
                        umma_ss_e(tmem + cDP, dv_k + o, ddo_k + o, idSS, kk > 0);
                    }
                    umma_ss_e(tmem + cDP, d_ones_d, drec, idSS, 1u);  // - D
                    umma_commit_e(&S.dp_full);
                }
                // Every MMA this warp issued must be complete before TMEM is released.
                umma_commit_e(&S.final_sdp);
                drain_wait(&S.final_sdp, 0);
            } else {
                for (int t = 0; ok && t < T; ++t) {
                    const int st = t % kQStages;
                    if (!(ok = wait_all(&S.p_full, t & 1))) break;
                    tc_fence_after();
                    const uint64_t ddo_mn = sdesc_sw128(smem_u32(S.dout[st]), 8192, 1024);
                    // dV: k-step kk runs over queries 16 kk .. 16 kk + 15 (P^T of query
                    // half kk / 4 sits at cDP + 64 (kk / 4), 8 columns per step;
                    // MN-major dO: 2048 bytes per step)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t a_p = tmem + cDP + 64 * (kk >> 2) + 8 * (kk & 3);
                        umma_ts_e(tmem + cDV, a_p, ddo_mn + 128 * kk, idKV, (t > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit_e(&S.pv_done);
                    if (!(ok = wait_all(&S.ds_full, t & 1))) break;
                    if (t > 0 && !(ok = wait_all(&S.dq_read, (t - 1) & 1))) break;
                    tc_fence_after();
                    const uint64_t dq_mn = sdesc_sw128(smem_u32(S.q[st]), 8192, 1024);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        // dK: queries 16 kk .. 16 kk + 15 (dS^T: 8 columns per step)
                        umma_ts_e(tmem + cDK, tmem + cDS + 8 * kk, dq_mn + 128 * kk, idKV, (t > 0 || kk > 0) ? 1u : 0u);
                        // dQ: keys 16 kk .. 16 kk + 15 (2048 bytes into the MN-major dS and K alike)
                        umma_ss_e(tmem + cDQ, ds_mn + 128 * kk, dk_mn + 128 * kk, idQ, kk > 0);
                    }
                    umma_commit_e(&S.mma2_done);
                    umma_commit_e(&S.qdo_empty[st]);
                }
                umma_commit_e(&S.final_bar);
                drain_wait(&S.final_bar, 0);
            }
        }
    } else if (warp >= 12) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsStage));
        // ------------------------------------------------------------ dQ stagers
        // Lane = query row r of the tile (TMEM lane of dQ).  Each step's dQ tile
        // (its GEMM complete) is read out of TMEM 16 columns at a time and
        // written to the staging buffer (two 32-column fp32 halves, 128-byte
        // swizzled rows); warp 2 adds it to the fp32 accumulator with TMA bulk
        // reduce-adds.  Query rows past the request's end (another request's
        // rows) are staged as zeros: their dS is zero, but times a non-finite key
        // it would not be.  The softmax scale is applied when the accumulator is
        // converted.
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        int g_c = 0, qt_c = 0;
        for (int t = 0; t < T; ++t) {
            const int q0 = (qr.lo + qt_c) * BM;
            bool ok = mbar_wait_warp(&S.mma2_done, t & 1, abort);
            // the bulk reduce of step t - 1 has finished reading the stage
            ok = ok && (t == 0 || mbar_wait_warp(&S.dq_stage_free, (t - 1) & 1, abort));
            if (!ok) break;
            tc_fence_after();
            const bool valid = q0 + r < Lq;
#pragma unroll
            for (int c16 = 0; c16 < 4; ++c16) {  // columns 16 c16 .. 16 c16 + 15
                uint32_t u[16];
                tmem_ld16(tmem + lane_base + cDQ + 16 * c16, u);
                tmem_ld_wait();
                if (c16 == 3) {  // dQ is out of TMEM: the next step's dQ GEMM may overwrite it
                    tc_fence_before();
                    mbar_arrive_warp(&S.dq_read);
                }
                uint8_t* row = S.dq_stage[c16 >> 1] + r * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int chunk = (c16 & 1) * 4 + c;  // 16-byte chunk of the 128-byte row
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(smem_u32(row) + ((chunk ^ (r & 7)) << 4)),
                                 "r"(valid ? u[4 * c] : 0u), "r"(valid ? u[4 * c + 1] : 0u),
                                 "r"(valid ? u[4 * c + 2] : 0u), "r"(valid ? u[4 * c + 3] : 0u)
                                 : "memory");
                }
            }
            fence_proxy_async_smem();
            mbar_arrive_warp(&S.dq_staged);
            if (++qt_c == nqt) {
                qt_c = 0;
                ++g_c;
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsWork));
        // ------------------------------------------------------------ elementwise
        // Lane = key r of the CTA (TMEM lane of S^T, dP^T, P^T, dS^T, dV, dK); hh =
        // query half: columns 64 hh .. 64 hh + 63 of S^T / dP^T.
        const int q4 = warp & 3;
        const int hh = (warp - 4) >> 2;
        const int r = q4 * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
        const int F = p.win_first, W = p.win_last;
        const int kpos = j0 + r;
        bool ok = true;

        // step t = g_c * nqt + qt_c (head g_c of the group, query tile qt_c)
        int g_c = 0, qt_c = 0;
        for (int t = 0; t < T; ++t) {
            const int q0 = (qr.lo + qt_c) * BM;
            if (!(ok = mbar_wait_warp(&S.s_full, t & 1, abort))) break;
            tc_fence_after();
            uint32_t pa[32], pb[32];  // S^T, then P (fp32), of this key's queries 0..31 / 32..63 of the half
            tmem_ld32(tmem + lane_base + cS + 64 * hh, pa);
            tmem_ld32(tmem + lane_base + cS + 64 * hh + 32, pb);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive_warp(&S.s_free);  // S^T read: the next step's S^T may overwrite it
            // Columns e (queries q0 + 64 hh + e) that see this key: lo <= e <= hi.
            // Query position pos sees key kpos iff kpos < Lk, kpos <= pos (causal)
            // and (kpos < F or kpos >= pos + 1 - W) (window); the columns past the
            // request's last query (another request's records) are out too.
            const long long base = (long long)off + q0 + 64 * hh;  // position of column 0
            int lo = 0;
            long long hi_ll = (long long)Lq - 1 - q0 - 64 * hh;
            if (kpos >= Lk) {
                lo = 64;
            } else {
                if (p.causal) lo = (int)max(0LL, min(64LL, (long long)kpos - base));
                if (W > 0 && kpos >= F) hi_ll = min(hi_ll, (long long)kpos + W - 1 - base);
            }
            const int hi = (int)max(-1LL, min(63LL, hi_ll));
            const bool full = __all_sync(0xffffffffu, lo == 0 && hi == 63);
            uint32_t pw[32];
            if (full) {
                p_cols<false, 0>(pa, sc2, lo, hi, pw);
                p_cols<false, 32>(pb, sc2, lo, hi, pw);
            } else {
                p_cols<true, 0>(pa, sc2, lo, hi, pw);
                p_cols<true, 32>(pb, sc2, lo, hi, pw);
            }
            if (!(ok = mbar_wait_warp(&S.dp_full, t & 1, abort))) break;
            tc_fence_after();
            uint32_t dw[32];  // dS / scale of this key's 64 queries, bf16 pairs
            {
                uint32_t dr[32];
                tmem_ld32(tmem + lane_base + cDP + 64 * hh, dr);
                tmem_ld_wait();
                if (full)
                    ds_cols<false, 0>(pa, dr, lo, hi, dw);
                else
                    ds_cols<true, 0>(pa, dr, lo, hi, dw);
                tmem_ld32(tmem + lane_base + cDP + 64 * hh + 32, dr);
                tmem_ld_wait();
                // P^T over this thread's dP^T columns (all read now): the A of dV
                tmem_st32(tmem + lane_base + cDP + 64 * hh, pw);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive_warp(&S.p_full);
                if (full)
                    ds_cols<false, 32>(pb, dr, lo, hi, dw);
                else
                    ds_cols<true, 32>(pb, dr, lo, hi, dw);
            }
            if (t > 0) {  // dK and dQ of the previous step are done with dS^T and dS
                if (!(ok = mbar_wait_warp(&S.mma2_done, (t - 1) & 1, abort))) break;
                tc_fence_after();
            }
            // dS^T: the A of dK
            tmem_st32(tmem + lane_base + cDS + 32 * hh, dw);
            // dS row r (64 queries = atom hh, chunks 0..7 of 16 bytes): the A of dQ
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const uint32_t o = hh * kTile + sw128_off(r, cc);
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(smem_u32(S.dsb + o)), "r"(dw[4 * cc]),
                             "r"(dw[4 * cc + 1]), "r"(dw[4 * cc + 2]), "r"(dw[4 * cc + 3])
                             : "memory");
            }
            fence_proxy_async_smem();
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(&S.ds_full);
            if (++qt_c == nqt) {
                qt_c = 0;
                ++g_c;
            }
        }
        // dK (query half 0) / dV (query half 1)
        if (ok && T > 0) ok = mbar_wait_warp(&S.final_bar, 0, abort);
        const bool have = ok && T > 0;
        if (have) tc_fence_after();
        const size_t rowoff =
            (size_t)(k_start + kpos) * (size_t)(hh == 0 ? p.dk_rs : p.dv_rs) + (size_t)kvh * D;
        const uint32_t col = hh == 0 ? cDK : cDV;
        __nv_bfloat16* outp = hh == 0 ? p.dk : p.dv;
        const float f = hh == 0 ? p.scale : 1.f;  // dK takes the softmax scale that dS left out
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
// Head dim 128 in one pass: bwd_main128_kernel.  The same roles, barriers and
// per-query k-step as bwd_main_kernel, with steps of 64 query rows so that
// TMEM holds every product at full width: S^T 64 columns, dP^T 64 (P^T written
// over it), dV 128, dK 128, dS^T 32 and dQ^T = K^T dS^T 64 (lane = head dim,
// column = query), 480 of 512.  dQ^T leaves through the staging buffer by
// transposed stores (lane = head dim, so a warp writes one 128-byte query row
// per store).
namespace d128 {
constexpr int BQ = 64;                      // query rows per step
constexpr int kQS = 3;                      // Q / dO / record stages
constexpr uint32_t kQAtom = BQ * 128;       // 64 rows x 128 bytes (64 head dims)
constexpr uint32_t kQTile = 2 * kQAtom;     // 64 rows x 128 head dims
constexpr uint32_t kKTile = 2 * kTile;      // 128 keys x 128 head dims
constexpr uint32_t kDqBox = BQ * 128;       // 64 query rows x 32 head dims fp32
constexpr uint32_t kRecTile = BQ * 32;      // 64 records
// TMEM columns: lane = key for S^T, dP^T, dV, dK, dS^T; lane = head dim for dQ^T.
constexpr uint32_t cS = 0, cDP = 64, cDV = 128, cDK = 256, cDS = 384, cDQ = 448;

struct __align__(1024) Smem {
    uint8_t k[kKTile];
    uint8_t v[kKTile];
    uint8_t q[kQS][kQTile];
    uint8_t dout[kQS][kQTile];
    uint8_t dsb[kTile];             // dS: 128 key rows x 64 queries (one atom), the MN-major B of dQ^T
    uint8_t dq_stage[4][kDqBox];    // dQ tile: four 32-dim boxes of 64 query rows, 128-byte swizzled
    uint8_t ones_lse[kAug];
    uint8_t ones_d[kAug];
    uint8_t rec[kQS][kRecTile];
    uint64_t kv_full, kv_ready, qdo_tail;
    uint64_t qdo_full[kQS], qdo_empty[kQS];
    uint64_t s_full, dp_full, s_free, p_full, pv_done, ds_full, mma2_done;
    uint64_t dq_read, dq_staged, dq_stage_free;
    uint64_t final_bar, final_sdp;
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void tma_q(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int head, int row) {
    tma_load_3d(dst, m, bar, 0, head, row);
    tma_load_3d(dst + kQAtom, m, bar, 64, head, row);
}
__device__ __forceinline__ void tma_k(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int head, int row) {
    tma_load_3d(dst, m, bar, 0, head, row);
    tma_load_3d(dst + kTile, m, bar, 64, head, row);
}
}  // namespace d128

__global__ void __launch_bounds__(kThreads, 1)
    bwd_main128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_rec,
                       const MainParams p) {
    using d128::BQ;
    using d128::kQS;
    using d128::kQAtom;
    using d128::kQTile;
    using d128::kKTile;
    using d128::kRecTile;
    using d128::tma_q;
    using d128::tma_k;
    constexpr uint32_t cS = d128::cS, cDP = d128::cDP, cDV = d128::cDV, cDK = d128::cDK, cDS = d128::cDS,
                       cDQ = d128::cDQ;
    constexpr int D = 128;
    extern __shared__ uint8_t smem_raw[];
    d128::Smem& S = *reinterpret_cast<d128::Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const CtaTile ct = cta_tile<16>(blockIdx.x, p.hkv, p.batch, p.n_kt);
    const int kvh = ct.kvh, b = ct.b, kt = ct.kt;

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
    const QRange qr = query_tiles(j0, Lq, Lk, p.causal, p.win_first, p.win_last, BQ);
    const int nqt = qr.hi - qr.lo;
    const int T = nqt * p.group;  // steps: (head g, 64-row query tile)
    const bool kv_tail = j0 + BN > Lk;

    if (threadIdx.x == 0) {
        mbar_init(&S.kv_full, 1);
        mbar_init(&S.kv_ready, 1);
        mbar_init(&S.qdo_tail, 1);
        for (int s = 0; s < kQS; ++s) {
            mbar_init(&S.qdo_full[s], 1);
            mbar_init(&S.qdo_empty[s], 1);
        }
        mbar_init(&S.s_full, 1);
        mbar_init(&S.dp_full, 1);
        mbar_init(&S.s_free, kWork / 32);
        mbar_init(&S.p_full, kWork / 32);
        mbar_init(&S.pv_done, 1);
        mbar_init(&S.ds_full, kWork / 32);
        mbar_init(&S.mma2_done, 1);
        mbar_init(&S.dq_read, kStage / 32);
        mbar_init(&S.dq_staged, kStage / 32);
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
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsCtrl));
        if (warp == 0) {
            // -------------------------------------------------------- producer
            // As in bwd_main_kernel: K / V once, then each step's Q, dO and
            // records; rows past the request's keys / queries are zeroed in shared
            // memory before the tensor core reads them.
            auto zero_rows = [&](uint8_t* atom, int r0, int nrows) {
                uint4* t4 = reinterpret_cast<uint4*>(atom);
                for (int c = r0 * 8 + lane; c < nrows * 8; c += 32) t4[c] = make_uint4(0u, 0u, 0u, 0u);
            };
            if (lane == 0) {
                prefetch_tmap(&tm_q);
                prefetch_tmap(&tm_k);
                prefetch_tmap(&tm_v);
                prefetch_tmap(&tm_do);
                prefetch_tmap(&tm_rec);
                mbar_expect_tx(&S.kv_full, 2 * kKTile);
                tma_k(S.k, &tm_k, &S.kv_full, kvh, k_start + j0);
                tma_k(S.v, &tm_v, &S.kv_full, kvh, k_start + j0);
            }
            {
                // the two ones blocks (see bwd_main_kernel)
                const uint4 one = make_uint4(0x3F803F80u, 0x00003F80u, 0u, 0u);
                const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
                for (int c = lane; c < (int)(kAug / 16); c += 32) {
                    const int j = c >> 1, half = (c & 1) ^ ((j >> 2) & 1);
                    reinterpret_cast<uint4*>(S.ones_lse)[c] = half == 0 ? one : zero;
                    reinterpret_cast<uint4*>(S.ones_d)[c] = half == 1 ? one : zero;
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            bool ok = true;
            if (kv_tail) {
                ok = mbar_wait_warp(&S.kv_full, 0, abort);
                if (ok) {
                    for (int a = 0; a < 2; ++a) {
                        zero_rows(S.k + a * kTile, Lk - j0, BN);
                        zero_rows(S.v + a * kTile, Lk - j0, BN);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&S.kv_ready);
                }
            }
            int t = 0, g_c = 0, qt_c = 0, tails = 0;
            bool tail_pending = false;
            uint32_t tail_last = 0;
            for (; ok && t < T; ++t) {
                const int st = t % kQS;
                if (t >= kQS && !mbar_wait_warp(&S.qdo_empty[st], (t / kQS - 1) & 1, abort)) break;
                const int h = kvh * p.group + g_c;
                const int q0 = (qr.lo + qt_c) * BQ;
                const bool tail = q0 + BQ > Lq;
                uint64_t* bar = tail ? &S.qdo_tail : &S.qdo_full[st];
                if (lane == 0) {
                    mbar_expect_tx(bar, 2 * kQTile + kRecTile);
                    tma_q(S.q[st], &tm_q, bar, h, q_start + q0);
                    tma_q(S.dout[st], &tm_do, bar, h, q_start + q0);
                    tma_load_3d(S.rec[st], &tm_rec, bar, 0, h, q_start + q0);
                }
                tail_last = tail ? (tail_last | (1u << st)) : (tail_last & ~(1u << st));
                if (tail) {
                    tail_pending = true;
                    if (!mbar_wait_warp(&S.qdo_tail, tails & 1, abort)) break;
                    tail_pending = false;
                    ++tails;
                    for (int a = 0; a < 2; ++a) {
                        zero_rows(S.q[st] + a * kQAtom, Lq - q0, BQ);
                        zero_rows(S.dout[st] + a * kQAtom, Lq - q0, BQ);
                    }
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
                for (int st = 0; st < kQS; ++st) {
                    const int n = t > st ? (t - st + kQS - 1) / kQS : 0;
                    if (n > 0 && !((tail_last >> st) & 1u)) drain_wait(&S.qdo_full[st], (n - 1) & 1);
                }
            }
            __syncwarp();
        } else if (warp == 2 && T > 0) {
            // -------------------------------------------------------- dQ reducer
            int g_c = 0, qt_c = 0;
            for (int tt = 0; tt < T; ++tt) {
                if (!mbar_wait_warp(&S.dq_staged, tt & 1, abort)) break;
                if (lane == 0) {
                    const int hh = kvh * p.group + g_c;
                    const int qq0 = (qr.lo + qt_c) * BQ;
#pragma unroll
                    for (int bx = 0; bx < 4; ++bx) tma_reduce_add_3d(&tm_dq, S.dq_stage[bx], 32 * bx, hh, q_start + qq0);
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
            if (lane == 0) bulk_wait_all();
            __syncwarp();
        } else if ((warp == 1 || warp == 3) && T > 0) {
            // -------------------------------------------------------- MMA issuers
            constexpr uint32_t idS = idesc_bf16_f32(BN, BQ, false, false);  // S^T, dP^T: M 128 keys, N 64 queries
            constexpr uint32_t idKV = idesc_bf16_f32(BN, D, false, true);   // dV, dK: A in TMEM, B MN-major, N 128
            constexpr uint32_t idQ = idesc_bf16_f32(D, BQ, true, true);     // dQ^T: A (K^T) and B (dS) MN-major
            const uint64_t dk_k = sdesc_sw128(smem_u32(S.k), 16, 1024);
            const uint64_t dv_k = sdesc_sw128(smem_u32(S.v), 16, 1024);
            const uint64_t d_ones_lse = sdesc_sw32(smem_u32(S.ones_lse));
            const uint64_t d_ones_d = sdesc_sw32(smem_u32(S.ones_d));
            const uint64_t dkT = sdesc_sw128(smem_u32(S.k), kTile, 1024);  // K as the MN-major A of dQ^T (M = head dims)
            const uint64_t ds_mn = sdesc_sw128(smem_u32(S.dsb), kTile, 1024);
            bool ok = mbar_wait_warp(kv_tail ? &S.kv_ready : &S.kv_full, 0, abort);
            if (warp == 1) {
                for (int t = 0; ok && t < T; ++t) {
                    const int st = t % kQS;
                    if (!(ok = mbar_wait_warp(&S.qdo_full[st], (t / kQS) & 1, abort))) break;
                    if (t > 0 && !(ok = mbar_wait_warp(&S.s_free, (t - 1) & 1, abort))) break;
                    tc_fence_after();
                    const uint64_t dq_k = sdesc_sw128(smem_u32(S.q[st]), 16, 1024);
                    const uint64_t ddo_k = sdesc_sw128(smem_u32(S.dout[st]), 16, 1024);
                    const uint64_t drec = sdesc_sw32(smem_u32(S.rec[st]));
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {  // 16 head dims per k-step; atom kk / 4
                        const uint32_t ok_ = (kk >> 2) * (kTile >> 4) + (kk & 3) * 2;
                        const uint32_t oq = (kk >> 2) * (kQAtom >> 4) + (kk & 3) * 2;
                        umma_ss_e(tmem + cS, dk_k + ok_, dq_k + oq, idS, kk > 0);
                    }
                    umma_ss_e(tmem + cS, d_ones_lse, drec, idS, 1u);  // - LSE / scale
                    umma_commit_e(&S.s_full);
                    // P^T of the previous step sits in the dP^T columns until dV has read it
                    if (t > 0 && !(ok = mbar_wait_warp(&S.pv_done, (t - 1) & 1, abort))) break;
                    // and once dK / dQ^T of the previous step are done: the elementwise warps
                    // then learn that from dp_full (no wait of their own before they write
                    // dS^T / dS over it).  Measured 1 % faster here, 3 % slower at d 64.
                    if (t > 0 && !(ok = mbar_wait_warp(&S.mma2_done, (t - 1) & 1, abort))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t ok_ = (kk >> 2) * (kTile >> 4) + (kk & 3) * 2;
                        const uint32_t oq = (kk >> 2) * (kQAtom >> 4) + (kk & 3) * 2;
                        umma_ss_e(tmem + cDP, dv_k + ok_, ddo_k + oq, idS, kk > 0);
                    }
                    umma_ss_e(tmem + cDP, d_ones_d, drec, idS, 1u);  // - D
                    umma_commit_e(&S.dp_full);
                }
                umma_commit_e(&S.final_sdp);
                drain_wait(&S.final_sdp, 0);
            } else {
                for (int t = 0; ok && t < T; ++t) {
                    const int st = t % kQS;
                    if (!(ok = mbar_wait_warp(&S.p_full, t & 1, abort))) break;
                    tc_fence_after();
                    // dO / Q as MN-major B: N = 128 head dims in two atoms kQAtom apart;
                    // a k-step (16 queries) is 2048 bytes on
                    const uint64_t ddo_mn = sdesc_sw128(smem_u32(S.dout[st]), kQAtom, 1024);
#pragma unroll
                    for (int kk = 0; kk < BQ / 16; ++kk)  // P^T of query half kk / 2: cDP + 32 (kk / 2), 8 columns per step
                        umma_ts_e(tmem + cDV, tmem + cDP + 32 * (kk >> 1) + 8 * (kk & 1), ddo_mn + 128 * kk, idKV,
                                  (t > 0 || kk > 0) ? 1u : 0u);
                    umma_commit_e(&S.pv_done);
                    if (!(ok = mbar_wait_warp(&S.ds_full, t & 1, abort))) break;
                    if (t > 0 && !(ok = mbar_wait_warp(&S.dq_read, (t - 1) & 1, abort))) break;
                    tc_fence_after();
                    const uint64_t dq_mn = sdesc_sw128(smem_u32(S.q[st]), kQAtom, 1024);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        // dQ^T: keys 16 kk .. 16 kk + 15 (2048 bytes into K and dS alike)
                        umma_ss_e(tmem + cDQ, dkT + 128 * kk, ds_mn + 128 * kk, idQ, kk > 0);
                        // dK: queries 16 (kk / 2) .. (dS^T 8 columns per step), every other k-step
                        if ((kk & 1) == 1)
                            umma_ts_e(tmem + cDK, tmem + cDS + 8 * (kk >> 1), dq_mn + 128 * (kk >> 1), idKV,
                                      (t > 0 || kk > 1) ? 1u : 0u);
                    }
                    umma_commit_e(&S.mma2_done);
                    umma_commit_e(&S.qdo_empty[st]);
                }
                umma_commit_e(&S.final_bar);
                drain_wait(&S.final_bar, 0);
            }
        }
    } else if (warp >= 12) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsStage));
        // ------------------------------------------------------------ dQ stagers
        // Lane = head dim 32 (warp & 3) + lane of dQ^T (TMEM lanes); 16 query
        // columns at a time, each stored into the query's row of box warp & 3 (a
        // warp writes one 128-byte row per store).  Queries past the request's end
        // are staged as zeros.
        const int box = warp & 3;
        const uint32_t lane_base = (uint32_t)(box * 32) << 16;
        uint8_t* const stage = S.dq_stage[box];
        const uint32_t col = ((uint32_t)(lane >> 2) << 4) | ((uint32_t)(lane & 3) << 2);  // byte in the 128-byte row
        int g_c = 0, qt_c = 0;
        for (int t = 0; t < T; ++t) {
            const int q0 = (qr.lo + qt_c) * BQ;
            bool ok = mbar_wait_warp(&S.mma2_done, t & 1, abort);
            ok = ok && (t == 0 || mbar_wait_warp(&S.dq_stage_free, (t - 1) & 1, abort));
            if (!ok) break;
            tc_fence_after();
            const int nvalid = min(BQ, Lq - q0);
#pragma unroll
            for (int c16 = 0; c16 < BQ / 16; ++c16) {
                uint32_t u[16];
                tmem_ld16(tmem + lane_base + cDQ + 16 * c16, u);
                tmem_ld_wait();
                if (c16 == BQ / 16 - 1) {
                    tc_fence_before();
                    mbar_arrive_warp(&S.dq_read);
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c = 16 * c16 + i;  // query row of the box
                    const uint32_t addr = smem_u32(stage) + c * 128 + (col ^ ((uint32_t)(c & 7) << 4));
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(c < nvalid ? u[i] : 0u) : "memory");
                }
            }
            fence_proxy_async_smem();
            mbar_arrive_warp(&S.dq_staged);
            if (++qt_c == nqt) {
                qt_c = 0;
                ++g_c;
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsWork));
        // ------------------------------------------------------------ elementwise
        // Lane = key r; hh = query half: columns 32 hh .. 32 hh + 31 of the step's
        // 64 queries.
        const int q4 = warp & 3;
        const int hh = (warp - 4) >> 2;
        const int r = q4 * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
        const int F = p.win_first, W = p.win_last;
        const int kpos = j0 + r;
        bool ok = true;
        int g_c = 0, qt_c = 0;
        for (int t = 0; t < T; ++t) {
            const int q0 = (qr.lo + qt_c) * BQ;
            if (!(ok = mbar_wait_warp(&S.s_full, t & 1, abort))) break;
            tc_fence_after();
            uint32_t pa[32];  // S^T, then P (fp32), of this key's 32 queries
            tmem_ld32(tmem + lane_base + cS + 32 * hh, pa);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive_warp(&S.s_free);
            // columns e (queries q0 + 32 hh + e) that see this key: lo <= e <= hi
            const long long base = (long long)off + q0 + 32 * hh;
            int lo = 0;
            long long hi_ll = (long long)Lq - 1 - q0 - 32 * hh;
            if (kpos >= Lk) {
                lo = 32;
            } else {
                if (p.causal) lo = (int)max(0LL, min(32LL, (long long)kpos - base));
                if (W > 0 && kpos >= F) hi_ll = min(hi_ll, (long long)kpos + W - 1 - base);
            }
            const int hi = (int)max(-1LL, min(31LL, hi_ll));
            const bool full = __all_sync(0xffffffffu, lo == 0 && hi == 31);
            uint32_t pw[32];
            if (full)
                p_cols<false, 0>(pa, sc2, lo, hi, pw);
            else
                p_cols<true, 0>(pa, sc2, lo, hi, pw);
            if (!(ok = mbar_wait_warp(&S.dp_full, t & 1, abort))) break;
            tc_fence_after();
            uint32_t dw[32];
            {
                uint32_t dr[32];
                tmem_ld32(tmem + lane_base + cDP + 32 * hh, dr);
                tmem_ld_wait();
                // P^T over this thread's dP^T columns (read): the A of dV
                tmem_st16(tmem + lane_base + cDP + 32 * hh, pw);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive_warp(&S.p_full);
                if (full)
                    ds_cols<false, 0>(pa, dr, lo, hi, dw);
                else
                    ds_cols<true, 0>(pa, dr, lo, hi, dw);
            }
            // dK and dQ^T of the previous step are done with dS^T and dS: dP^T of this step
            // (waited above) was issued after them.
            tmem_st16(tmem + lane_base + cDS + 16 * hh, dw);  // dS^T: the A of dK
            // dS row r, queries 32 hh .. 32 hh + 31 = 16-byte chunks 4 hh .. 4 hh + 3: the B of dQ^T
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const uint32_t o = sw128_off(r, 4 * hh + cc);
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(smem_u32(S.dsb + o)), "r"(dw[4 * cc]),
                             "r"(dw[4 * cc + 1]), "r"(dw[4 * cc + 2]), "r"(dw[4 * cc + 3])
                             : "memory");
            }
            fence_proxy_async_smem();
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(&S.ds_full);
            if (++qt_c == nqt) {
                qt_c = 0;
                ++g_c;
            }
        }
        // dK (query half 0) / dV (query half 1): 128 head dims of key r
        if (ok && T > 0) ok = mbar_wait_warp(&S.final_bar, 0, abort);
        const bool have = ok && T > 0;
        if (have) tc_fence_after();
        const size_t rowoff = (size_t)(k_start + kpos) * (size_t)(hh == 0 ? p.dk_rs : p.dv_rs) + (size_t)kvh * D;
        const uint32_t cbase = hh == 0 ? cDK : cDV;
        __nv_bfloat16* outp = hh == 0 ? p.dk : p.dv;
        const float f = hh == 0 ? p.scale : 1.f;  // dK takes the softmax scale that dS left out
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t u[32];
            if (have) {
                tmem_ld32(tmem + lane_base + cbase + ch * 32, u);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) u[e] = 0u;
            }
            if (kpos < Lk) {
                uint4* dst = reinterpret_cast<uint4*>(outp + rowoff + ch * 32);
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
// D_i = rowsum(dO_i o O_i), the per-query records and dsink.  Block: 256
// threads, 64 rows of one head; 8 threads per row, 16 bytes each.

// x as three bf16 (h1 = x rounded, h2 = the remainder rounded, h3 = what is left
// rounded: x - h1 and x - h1 - h2 are exact in fp32), elements 0..2 of a 16-byte
// half-record.  An infinite x is stored as +-1e30: the k-step multiplies the
// other half of the record by zeros, and 0 times an infinity would be NaN;
// +-1e30 still drives P to 0 (or the column is masked anyway).
__device__ __forceinline__ uint4 split3_bf16(float x) {
    if (isinf(x)) x = copysignf(1e30f, x);
    const float h1 = __bfloat162float(__float2bfloat16_rn(x));
    float r = x - h1;
    const float h2 = __bfloat162float(__float2bfloat16_rn(r));
    r -= h2;
    return make_uint4(pack_bf16x2(h1, h2), pack_bf16x2(r, 0.f), 0u, 0u);
}

// Per block: 64 rows of one query head (the head is the fastest grid index, so
// the blocks in flight read whole rows of O and dO).  Besides D, the records
// and dsink it clears the block's rows of the fp32 dQ accumulator, and (kv_zero)
// the whole grid clears the dK / dV rows past the last request's keys.
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ out,
                                                             const __nv_bfloat16* __restrict__ dout,
                                                             const float* __restrict__ lse,
                                                             const float* __restrict__ sink, uint4* __restrict__ rec,
                                                             float* __restrict__ dsink, float4* __restrict__ dq_acc,
                                                             int total_q, int hq, float scale,
                                                             const int32_t* __restrict__ cu_q,
                                                             const int32_t* __restrict__ cu_k, int batch,
                                                             uint4* __restrict__ dk, uint4* __restrict__ dv,
                                                             int total_k, int hkv, int kv_zero) {
    const int h = blockIdx.x;
    const int n_rb = (total_q + 63) / 64;
    // Rows past the last request (cu_q[batch] <= row < total_q) belong to no
    // request: D = 0, a zero record and no sink term, whatever the buffers hold
    // there.
    const int rows = min(total_q, max(0, cu_q[batch]));
    const int tid = threadIdx.x;
    const int sub = tid & 7;
    const float sg = sink ? sink[h] : -INFINITY;
    float acc_sink = 0.f;
    for (int rb = blockIdx.y; rb < n_rb; rb += gridDim.y) {
        for (int rr = 0; rr < 2; ++rr) {
            const int row = rb * 64 + rr * 32 + (tid >> 3);
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
            if (row < total_q) {
                // this row's D fp32 accumulator values: D / 8 per thread
                float4* a = dq_acc + ((size_t)row * hq + h) * (D / 4) + sub * (D / 32);
#pragma unroll
                for (int j = 0; j < D / 32; ++j) a[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            d += __shfl_xor_sync(0xffffffffu, d, 1);
            d += __shfl_xor_sync(0xffffffffu, d, 2);
            d += __shfl_xor_sync(0xffffffffu, d, 4);
            if (row < total_q && sub < 2) {
                // record (row, h): two 16-byte halves, -LSE / scale (sub 0) and -D (sub 1)
                const float l = (sub == 0 && row < rows) ? lse[(size_t)h * total_q + row] : 0.f;
                rec[((size_t)row * hq + h) * 2 + sub] = split3_bf16(sub == 0 ? -l / scale : -d);
                if (sub == 0 && sink && row < rows) {
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
    }
    if (kv_zero) {
        // dK / dV rows cu_k[batch] .. total_k - 1 belong to no request and no
        // CTA of the main kernel writes them.
        const int k0 = min(total_k, max(0, cu_k[batch]));
        const size_t n16 = (size_t)(total_k - k0) * hkv * (D / 8);
        const size_t first = (size_t)k0 * hkv * (D / 8);
        const size_t nthreads = (size_t)gridDim.x * gridDim.y * blockDim.x;
        for (size_t i = ((size_t)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + tid; i < n16; i += nthreads) {
            dk[first + i] = make_uint4(0u, 0u, 0u, 0u);
            dv[first + i] = make_uint4(0u, 0u, 0u, 0u);
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

// acc holds rows of row4 float4 (hq * d / 4); dq rows are dq_rs4 uint2 apart.  The
// accumulator holds sum dS K with dS short of the softmax scale.
__global__ void bwd_dq_convert_kernel(const float4* __restrict__ acc, uint2* __restrict__ dq, size_t n4,
                                      int row4, long long dq_rs4, float scale) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 v = acc[i];
        const size_t row = i / (size_t)row4, c = i - row * (size_t)row4;
        dq[row * (size_t)dq_rs4 + c] =
            make_uint2(pack_bf16x2(v.x * scale, v.y * scale), pack_bf16x2(v.z * scale, v.w * scale));
    }
}

// ---------------------------------------------------------------------------
// Host side

cudaError_t make_map(CUtensorMap* m, const void* base, int d, int heads, long long rows, std::string* what,
                     long long row_stride = 0, int box_rows = 128);
cudaError_t make_map_dq(CUtensorMap* m, const float* base, int d, int heads, long long rows, std::string* what,
                        int box_rows = 128);
cudaError_t make_map_rec(CUtensorMap* m, const void* base, int heads, long long rows, std::string* what,
                         int box_rows = 128);

// The fp32 dQ accumulator, then the per-query records (32 bytes per row and head).
size_t workspace_bytes(const Args& a) {
    const size_t acc = (size_t)a.total_q * a.hq * a.head_dim * sizeof(float);
    const size_t rec = (size_t)a.total_q * a.hq * kRec * 2;
    return ((acc + 255) & ~size_t(255)) + rec;
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

// (rows, heads, d) bf16 tensor as {d, head, row}; box {64, 1, box_rows}: one
// 128-byte-swizzled atom per copy.
cudaError_t make_map(CUtensorMap* m, const void* base, int D, int heads, long long rows, std::string* what,
                     long long row_stride, int box_rows) {
    auto fn = encode_fn();
    if (!fn) {
        *what = "cuTensorMapEncodeTiled unavailable";
        return cudaErrorNotSupported;
    }
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)(row_stride > 0 ? row_stride : (long long)D * heads) * 2};
    cuuint32_t box[3] = {64u, 1, (cuuint32_t)box_rows};
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

// (rows, heads, d) fp32 dQ accumulator as {d, head, row}; box {32, 1, box_rows}, 128-byte swizzle.
cudaError_t make_map_dq(CUtensorMap* m, const float* base, int D, int heads, long long rows, std::string* what,
                        int box_rows) {
    auto fn = encode_fn();
    if (!fn) {
        *what = "cuTensorMapEncodeTiled unavailable";
        return cudaErrorNotSupported;
    }
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)D * 4 * heads};
    cuuint32_t box[3] = {32, 1, (cuuint32_t)box_rows};
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

// (rows, heads, 16) bf16 per-query records as {16, head, row}; box {16, 1,
// box_rows}, 32-byte swizzle (the layout of the extra k-step's B operand).
cudaError_t make_map_rec(CUtensorMap* m, const void* base, int heads, long long rows, std::string* what,
                         int box_rows) {
    auto fn = encode_fn();
    if (!fn) {
        *what = "cuTensorMapEncodeTiled unavailable";
        return cudaErrorNotSupported;
    }
    cuuint64_t dims[3] = {(cuuint64_t)kRec, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)kRec * 2, (cuuint64_t)kRec * 2 * heads};
    cuuint32_t box[3] = {(cuuint32_t)kRec, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *what = "cuTensorMapEncodeTiled (records) failed (" + std::to_string((int)r) + ")";
        return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

template <int D>
static cudaError_t launch_d(const Args& a, void* workspace, cudaStream_t s, std::string* what) {
    cudaError_t e;
    const size_t acc_bytes = (size_t)a.total_q * a.hq * D * sizeof(float);
    float* dq_accum = static_cast<float*>(workspace);
    uint4* rec = reinterpret_cast<uint4*>(static_cast<char*>(workspace) + ((acc_bytes + 255) & ~size_t(255)));
    if (a.dsink && (e = cudaMemsetAsync(a.dsink, 0, sizeof(float) * a.hq, s)) != cudaSuccess) {
        *what = "memset dsink";
        return e;
    }
    // dK/dV rows of keys no CTA visits (past every request's end) are zero
    // (contiguous outputs only: a strided output shares its rows with other
    // tensors); the preprocess kernel clears them, or a memset when it does
    // not run.
    const bool dkv_contig = a.dk_rs <= 0 && a.dv_rs <= 0;
    if (a.total_q == 0 && dkv_contig && a.total_k > 0 &&
        ((e = cudaMemsetAsync(a.dk, 0, (size_t)a.total_k * a.hkv * D * 2, s)) != cudaSuccess ||
         (e = cudaMemsetAsync(a.dv, 0, (size_t)a.total_k * a.hkv * D * 2, s)) != cudaSuccess)) {
        *what = "memset dk/dv";
        return e;
    }
    if (a.total_q > 0) {
        const int n_rb = (a.total_q + 63) / 64;
        dim3 g1(a.hq, n_rb < 65535 ? n_rb : 65535);
        bwd_preprocess_kernel<D><<<g1, 256, 0, s>>>(
            reinterpret_cast<const __nv_bfloat16*>(a.out), reinterpret_cast<const __nv_bfloat16*>(a.dout), a.lse,
            a.sink, rec, a.dsink, reinterpret_cast<float4*>(dq_accum), a.total_q, a.hq, a.scale, a.cu_q, a.cu_k,
            a.batch, reinterpret_cast<uint4*>(a.dk), reinterpret_cast<uint4*>(a.dv), a.total_k, a.hkv,
            dkv_contig ? 1 : 0);
        if ((e = cudaGetLastError()) != cudaSuccess) {
            *what = "preprocess launch";
            return e;
        }
    }
    if (a.total_q > 0 && a.total_k > 0 && a.max_seqlen_k > 0) {
        // query-side boxes: 128 rows per step at d 64, 64 at d 128
        const int qbox = D == 128 ? d128::BQ : BM;
        CUtensorMap tq, tk, tv, tdo, tdq, trec;
        if ((e = make_map(&tq, a.q, D, a.hq, a.total_q, what, a.q_rs, qbox)) != cudaSuccess) return e;
        if ((e = make_map(&tk, a.k, D, a.hkv, a.total_k, what, a.k_rs)) != cudaSuccess) return e;
        if ((e = make_map(&tv, a.v, D, a.hkv, a.total_k, what, a.v_rs)) != cudaSuccess) return e;
        if ((e = make_map(&tdo, a.dout, D, a.hq, a.total_q, what, 0, qbox)) != cudaSuccess) return e;
        if ((e = make_map_dq(&tdq, dq_accum, D, a.hq, a.total_q, what, qbox)) != cudaSuccess) return e;
        if ((e = make_map_rec(&trec, rec, a.hq, a.total_q, what, qbox)) != cudaSuccess) return e;
        MainParams p;
        p.cu_q = a.cu_q;
        p.cu_k = a.cu_k;
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
        p.batch = a.batch;
        p.n_kt = (a.max_seqlen_k + BN - 1) / BN;
        const long long n_cta = (long long)a.hkv * a.batch * p.n_kt;
        if (n_cta > 0x7fffffffLL) {
            *what = "too many key tiles for one launch";
            return cudaErrorInvalidValue;
        }
        dim3 g2((unsigned)n_cta);
        if constexpr (D == 128) {
            const size_t smem = sizeof(d128::Smem) + 1024;
            static_assert(sizeof(d128::Smem) + 1024 <= 227 * 1024, "shared memory of the d 128 main kernel");
            if ((e = cudaFuncSetAttribute(bwd_main128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)smem)) != cudaSuccess) {
                *what = "smem attribute";
                return e;
            }
            bwd_main128_kernel<<<g2, kThreads, smem, s>>>(tq, tk, tv, tdo, tdq, trec, p);
        } else {
            const size_t smem = sizeof(Smem<D>) + 1024;
            static_assert(sizeof(Smem<D>) + 1024 <= 227 * 1024, "shared memory of the main kernel");
            if ((e = cudaFuncSetAttribute(bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)smem)) != cudaSuccess) {
                *what = "smem attribute";
                return e;
            }
            bwd_main_kernel<D><<<g2, kThreads, smem, s>>>(tq, tk, tv, tdo, tdq, trec, p);
        }
        if ((e = cudaGetLastError()) != cudaSuccess) {
            *what = "main launch";
            return e;
        }
    }
    if (a.total_q > 0) {
        const size_t n4 = (size_t)a.total_q * a.hq * D / 4;
        int blocks = (int)((n4 + 255) / 256);
        if (blocks > 152 * 16) blocks = 152 * 16;
        const long long dq_rs = a.dq_rs > 0 ? a.dq_rs : (long long)a.hq * D;
        bwd_dq_convert_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(dq_accum),
                                                    reinterpret_cast<uint2*>(a.dq), n4, a.hq * D / 4, dq_rs / 4,
                                                    a.scale);
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
