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
// One CTA = 128 query rows of one query head; two CTAs share an SM, so the
// tensor core interleaves two independent pipelines.
//   warp 0      TMA producer: Q once, then the K tiles (3-stage ring)
//   warp 1      TMEM allocator and tcgen05.mma issuer (converged warp, elect.sync):
//               S = Q K^T (128x128 fp32, A and B from shared memory),
//               O += P V  (128x64 fp32, A = P from TMEM, B = V from shared memory)
//   warp 2      TMA producer of the V tiles (3-stage ring)
// With a paged cache the producers fetch each tile as page segments through
// the page table (one TMA copy per segment).
//   warp 3      tcgen05.mma issuer of O += P V (warp 1 then issues S only)
//   warps 4..7  softmax warpgroup; thread = query row.
// TMEM (256 columns): S at 0, O at 128, P (bf16 pairs) at 192.
// The online softmax starts from m = sink, l = 1 (the sink costs nothing per
// tile).  Each tile is first exponentiated against the running reference max
// without computing its row max; only when the row sum shows a value above
// 2^64 (or no reference exists yet) is the row max taken and, if it exceeds
// the reference by more than 2^64, O in TMEM rescaled in place.  P values stay
// below 2^64, far inside fp32/bf16 range, so the result is exact.
#include <cudaTypedefs.h>

#include <type_traits>

#include "common.cuh"
#include "prefill.h"
#include "sm103.cuh"

namespace attn {
namespace prefill {

using namespace sm103;

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int KSTAGE = 3;
constexpr int VSTAGE = 3;
constexpr int kThreads = 256;
// Two CTAs per SM: 128 registers per thread at launch.  setmaxnreg moves them
// from warpgroup 0 (TMA + MMA) to the softmax warpgroup:
// 128*40 + 128*216 = 32768 = 256 threads * 128.
constexpr int kRegsCtrl = 40;
constexpr int kRegsSoftmax = 216;
constexpr uint32_t kAtom = 128 * 128;  // one 128-byte-swizzled atom column: 128 rows x 64 bf16
// Head-dim dependent sizes.  An operand tile of 128 rows is D / 64 atoms, atom a
// holding elements 64a .. 64a + 63 of every row at byte offset a * kAtom.
// TMEM: S at column 0 (128 fp32), O at 128 (D fp32), P at 128 + D (64 columns
// of bf16 pairs); d 64 fits two CTAs per SM (256 columns each), d 128 takes
// one CTA and all 512 columns.
template <int D>
struct Cfg {
    static constexpr int kAtoms = D / 64;
    static constexpr uint32_t kTile = kAtom * kAtoms;
    static constexpr uint32_t kTmemCols = D == 64 ? 256 : 512;
    static constexpr uint32_t cS = 0, cO = 128, cP = 128 + D;
    static constexpr bool kTwoPerSm = D == 64;
};
// The running reference max only moves when a row's max exceeds it by more
// than 2^64 (log2 units below); every P value stays below 2^64 and every sum
// far below fp32's range, so the stale reference costs no accuracy.
constexpr float kRescaleThreshold = 64.0f;
constexpr float kFastSumLimit = 1.8446744e19f;  // 2^64

template <int D>
struct __align__(1024) Smem {
    uint8_t q[Cfg<D>::kTile];
    uint8_t k[KSTAGE][Cfg<D>::kTile];
    uint8_t v[VSTAGE][Cfg<D>::kTile];
    uint64_t q_full;
    uint64_t k_full[KSTAGE], k_empty[KSTAGE];
    uint64_t v_full[VSTAGE], v_empty[VSTAGE];
    uint64_t s_full, s_free, p_full, o_done;  // one phase per key tile
    uint64_t final_bar, final_pv;  // the S issuer's / the P V issuer's MMAs all complete
    uint64_t v_tail;  // the V tile that holds the request's last key lands here first
    uint32_t tmem_base;
    int abort;
};

struct Params {
    const float* sink;
    const int32_t* cu_q;
    const int32_t* cu_k;
    __nv_bfloat16* out;
    float* lse;
    int hq, group, n_rt, total_q, total_k;
    int win_first, win_last, causal;
    float scale_log2;
    // Paged K/V (page_table != nullptr): keys of request b are its first
    // seqlens_k[b] cache tokens; token t sits at slot
    // page_table[b][t >> page_shift] << page_shift | (t & (page_size - 1)).
    const int32_t* page_table;
    const int32_t* seqlens_k;
    int max_pages, page_shift, seg_shift, num_pages;  // a tile is 128 >> seg_shift page segments
};

// Waits that ignore the abort flag (used only to drain work already in flight
// before shared memory / TMEM are released); still bounded in time.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    int dummy = 0;
    mbar_wait(bar, parity, &dummy);
}

// Loads one 128-row operand tile (D / 64 atoms) of a (rows, heads, D) tensor
// starting at `row`, completing on `bar`.
template <int D>
__device__ __forceinline__ void tma_tile(uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int head, int row) {
#pragma unroll
    for (int a = 0; a < Cfg<D>::kAtoms; ++a) tma_load_3d(dst + a * kAtom, m, bar, 64 * a, head, row);
}

// kPaged: launched with a page table (the paged instantiation issues a tile's
// page-segment copies from parallel lanes; the contiguous one never runs that
// branch).
template <int D, bool kPaged>
__global__ void __launch_bounds__(kThreads, 2)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const Params p) {
    using C = Cfg<D>;
    constexpr uint32_t kTile = C::kTile;
    constexpr uint32_t cS = C::cS, cO = C::cO, cP = C::cP;
    extern __shared__ uint8_t smem_raw[];
    // Two CTAs per SM (d 64) only fit without alignment slack: the dynamic
    // shared base (after the 1 KB the hardware reserves per CTA) must already
    // be 1024-aligned for the 128-byte swizzle atoms -- checked, never assumed.
    // At d 128 (one CTA per SM) the base is rounded up inside 1 KB of slack.
    uint8_t* smem_al = C::kTwoPerSm ? smem_raw
                                    : reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                                 ~uintptr_t(1023));
    Smem<D>& S = *reinterpret_cast<Smem<D>*>(smem_al);
    if (smem_u32(smem_al) & 1023u) {
        if (threadIdx.x == 0) raise_status(ATTN_SINK_DEV_LAYOUT);
        return;
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Grid (head, row tile, request): the CTAs in flight share one request's K/V
    // (it stays in L2); within a request the last row tiles (the most key tiles
    // under causal masking) are launched first.
    const int h = blockIdx.x;
    const int rt = p.n_rt - 1 - (int)blockIdx.y;
    const int b = blockIdx.z;

    const int q_start = p.cu_q[b];
    int Lq = p.cu_q[b + 1] - q_start;
    const bool paged = p.page_table != nullptr;
    const int k_start = paged ? 0 : p.cu_k[b];
    int Lk = paged ? p.seqlens_k[b] : p.cu_k[b + 1] - k_start;
    const long long k_cap = paged ? ((long long)p.max_pages << p.page_shift) : (long long)p.total_k - k_start;
    if (q_start + Lq > p.total_q || Lk > k_cap || Lq < 0 || Lk < 0) {
        if (threadIdx.x == 0 && rt == 0 && h == 0) raise_status(ATTN_SINK_DEV_SEQLEN_OOB);
        Lq = max(0, min(Lq, p.total_q - q_start));
        Lk = (int)max(0LL, min((long long)Lk, k_cap));
    }
    const int qs = rt * BM;
    if (qs >= Lq) return;
    const int kvh = h / p.group;

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
        for (int s = 0; s < KSTAGE; ++s) {
            mbar_init(&S.k_full[s], 1);
            mbar_init(&S.k_empty[s], 1);
        }
        for (int s = 0; s < VSTAGE; ++s) {
            mbar_init(&S.v_full[s], 1);
            mbar_init(&S.v_empty[s], 1);
        }
        mbar_init(&S.s_full, 1);
        mbar_init(&S.s_free, 128);
        mbar_init(&S.p_full, 128);
        mbar_init(&S.o_done, 1);
        mbar_init(&S.final_bar, 1);
        mbar_init(&S.final_pv, 1);
        mbar_init(&S.v_tail, 1);
        S.abort = 0;
        fence_mbar_init();
        // Contiguous K / V: Q and the first ring's worth of K and V tiles are
        // requested now, so they load while TMEM is allocated and the CTA
        // synchronises (about a third of a CTA's fixed start-up time); the
        // producer warps take over from the next tile on.
        if constexpr (!kPaged) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            mbar_expect_tx(&S.q_full, kTile);
            tma_tile<D>(S.q, &tm_q, &S.q_full, h, q_start + qs);
            for (int it = 0; it < ntiles && it < KSTAGE; ++it) {
                const int t = it < ta ? it : tb + (it - ta);
                mbar_expect_tx(&S.k_full[it], kTile);
                tma_tile<D>(S.k[it], &tm_k, &S.k_full[it], kvh, k_start + t * BN);
            }
            for (int it = 0; it < ntiles && it < VSTAGE; ++it) {
                const int t = it < ta ? it : tb + (it - ta);
                uint64_t* bar = (t + 1) * BN > Lk ? &S.v_tail : &S.v_full[it];
                mbar_expect_tx(bar, kTile);
                tma_tile<D>(S.v[it], &tm_v, bar, kvh, k_start + t * BN);
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(&S.tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    volatile int* abort = &S.abort;

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtrl));
        if (warp == 0 || warp == 2) {
            // -------------------------------------------------------- producers
            // The warp runs the loop converged: lane 0 waits and issues the TMA
            // copies; with a paged cache lane i first resolves the physical slot
            // of the tile's i-th page segment.
            const bool is_k = warp == 0;
            const int nst = is_k ? KSTAGE : VSTAGE;
            uint64_t* full = is_k ? S.k_full : S.v_full;
            uint64_t* empty = is_k ? S.k_empty : S.v_empty;
            uint8_t* dst0 = is_k ? S.k[0] : S.v[0];
            const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
            const int nseg = BN >> p.seg_shift;
            if (paged && lane == 0) {
                prefetch_tmap(tm);
                if (is_k) {
                    prefetch_tmap(&tm_q);
                    mbar_expect_tx(&S.q_full, kTile);
                    tma_tile<D>(S.q, &tm_q, &S.q_full, h, q_start + qs);
                }
            }
            // The one V tile that reaches past the request's last key (rows of the
            // next request, of no request, or unwritten cache slots) lands on v_tail;
            // this warp then zeroes those rows before it releases the stage, so they
            // enter P V as exact zeros whatever the memory held (a masked P of 0
            // times a NaN or an infinity would not vanish).
            bool tail_issued = false;
            int it = 0;
            for (; it < ntiles; ++it) {
                const int st = it % nst;
                if (it >= nst && !__all_sync(0xffffffffu, mbar_wait(&empty[st], ((it / nst) - 1) & 1, abort)))
                    break;
                const int t = it < ta ? it : tb + (it - ta);
                const bool tail = !is_k && (t + 1) * BN > Lk;
                uint64_t* bar = tail ? &S.v_tail : &full[st];
                if (!paged) {
                    if (lane == 0 && it >= nst) {  // the first nst were issued at start-up
                        mbar_expect_tx(bar, kTile);
                        tma_tile<D>(dst0 + st * kTile, tm, bar, kvh, k_start + t * BN);
                    }
                } else {
                    // Segment `lane` covers keys j .. j + (1 << seg_shift) - 1, inside one page.
                    // Keys past the request's end (masked later) read slot 0.
                    int slot = 0;
                    const int j = t * BN + (lane << p.seg_shift);
                    if (lane < nseg && j < Lk) {
                        const int pg = __ldg(p.page_table + (size_t)b * p.max_pages + (j >> p.page_shift));
                        if (pg >= 0 && pg < p.num_pages)
                            slot = (pg << p.page_shift) | (j & ((1 << p.page_shift) - 1));
                        else
                            raise_status(ATTN_SINK_DEV_PAGE_OOB);
                    }
                    if (lane == 0) mbar_expect_tx(bar, kTile);
                    if constexpr (kPaged) {
                        // lane i issues the copy of segment i
                        __syncwarp();
                        if (lane < nseg)
                            tma_tile<D>(dst0 + st * kTile + ((uint32_t)lane << p.seg_shift) * 128u, tm, bar, kvh,
                                        slot);
                    } else {
                        for (int sg = 0; sg < nseg; ++sg) {
                            const int sl = __shfl_sync(0xffffffffu, slot, sg);
                            if (lane == 0)
                                tma_tile<D>(dst0 + st * kTile + ((uint32_t)sg << p.seg_shift) * 128u, tm, bar, kvh,
                                            sl);
                        }
                    }
                }
                if (tail) {
                    // Used once per CTA (one tile holds the last key): parity 0.
                    tail_issued = true;
                    if (!__all_sync(0xffffffffu, mbar_wait(&S.v_tail, 0, abort))) break;
                    // Key row r of an atom is the 128 bytes at r * 128 (the swizzle
                    // permutes 16-byte chunks within a row), so rows Lk - t*BN .. BN - 1
                    // are one contiguous range per atom.
#pragma unroll
                    for (int a = 0; a < C::kAtoms; ++a) {
                        uint4* vt = reinterpret_cast<uint4*>(dst0 + st * kTile + a * kAtom);
                        for (int c = (Lk - t * BN) * 8 + lane; c < BN * 8; c += 32) vt[c] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();  // the tensor core reads the zeros through the async proxy
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full[st]);
                }
            }
            // Drain: every copy issued must have landed before the CTA exits.
            if (lane == 0) {
                if (is_k) drain_wait(&S.q_full, 0);
                if (tail_issued) drain_wait(&S.v_tail, 0);
                for (int st = 0; st < nst; ++st) {
                    const int n = it > st ? (it - st + nst - 1) / nst : 0;
                    if (n > 0) drain_wait(&full[st], (n - 1) & 1);
                }
            }
            __syncwarp();
        } else if ((warp == 1 || warp == 3) && ntiles > 0) {
            // -------------------------------------------------------- MMA issuers
            // Warp 1 issues S = Q K^T, warp 3 O += P V: the tensor core gets two
            // independent instruction streams, and the issue stalls of a blocked
            // tcgen05.mma fall on two SM sub-partitions (warp w runs on
            // sub-partition w % 4), each slowing one softmax warp, instead of one.
            // Both warps run their loop converged (every lane waits; elect.sync
            // picks the issuing lane).
            constexpr uint32_t idS = idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t idO = idesc_bf16_f32(BM, D, false, true);
            // Descriptor bases; a k-step adds its byte offset / 16 to the address field.
            const uint64_t dq = sdesc_sw128(smem_u32(S.q), 16, 1024);
            const uint64_t dk0 = sdesc_sw128(smem_u32(S.k[0]), 16, 1024);
            const uint64_t dv0 = sdesc_sw128(smem_u32(S.v[0]), kAtom, 1024);  // MN atoms kAtom apart
            auto wait_all = [&](uint64_t* bar, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
            };
            bool ok = true;
            if (warp == 1) {
                ok = wait_all(&S.q_full, 0);
                for (int it = 0; ok && it < ntiles; ++it) {
                    // S of tile it as soon as its K is in and the softmax has read the
                    // previous S (it runs on the tensor core while the softmax works)
                    if (!(ok = wait_all(&S.k_full[it % KSTAGE], (it / KSTAGE) & 1))) break;
                    if (it > 0 && !(ok = wait_all(&S.s_free, (it - 1) & 1))) break;
                    tc_fence_after();
                    const uint64_t dk = dk0 + (it % KSTAGE) * (kTile >> 4);
                    // 16 head-dim elements = 32 bytes per k-step; atom kk / 4
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t o = (kk >> 2) * (kAtom >> 4) + (kk & 3) * 2;
                        umma_ss_e(tmem + cS, dq + o, dk + o, idS, kk > 0);
                    }
                    umma_commit_e(&S.s_full);
                    umma_commit_e(&S.k_empty[it % KSTAGE]);
                }
                // Every MMA issued must be complete before TMEM is released.
                umma_commit_e(&S.final_bar);
                drain_wait(&S.final_bar, 0);
            } else {
                for (int it = 0; ok && it < ntiles; ++it) {
                    // O += P V once P is in TMEM (8 columns of bf16 pairs per 16 keys;
                    // V rows 2048 bytes on per 16 keys)
                    if (!(ok = wait_all(&S.v_full[it % VSTAGE], (it / VSTAGE) & 1))) break;
                    if (!(ok = wait_all(&S.p_full, it & 1))) break;
                    tc_fence_after();
                    const uint64_t dv = dv0 + (it % VSTAGE) * (kTile >> 4);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        umma_ts_e(tmem + cO, tmem + cP + kk * 8, dv + 128 * kk, idO, (it > 0 || kk > 0) ? 1u : 0u);
                    umma_commit_e(&S.o_done);
                    umma_commit_e(&S.v_empty[it % VSTAGE]);
                }
                umma_commit_e(&S.final_pv);
                drain_wait(&S.final_pv, 0);
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ------------------------------------------------------------ softmax
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        const uint32_t tS = tmem + lane_base + cS;
        const uint32_t tO = tmem + lane_base + cO;
        const uint32_t tP = tmem + lane_base + cP;
        const float sg = p.sink ? p.sink[h] * ATTN_LOG2E : -INFINITY;
        const float sl2 = p.scale_log2;
        float m_ref = sg;
        float l = sg == -INFINITY ? 0.f : 1.f;
        const int pos = off + qs + r;
        bool ok = true;
        for (int it = 0; it < ntiles; ++it) {
            const int t = it < ta ? it : tb + (it - ta);
            const int j0 = t * BN;
            ok = mbar_wait(&S.s_full, it & 1, abort);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // S is read into registers and released as soon as all of it is in: the
            // second half is still loading while the first half is exponentiated, and
            // the next S runs on the tensor core during the rest of the exp2 phase.  P
            // is computed and stored in two halves, the first half's TMEM store
            // overlapping the second half's exp2 work.
            uint32_t s[4][32];
            tmem_ld32(tS, s[0]);
            tmem_ld32(tS + 32, s[1]);
            tmem_ld_wait();
            tmem_ld32(tS + 64, s[2]);
            tmem_ld32(tS + 96, s[3]);
            bool s_in = false;
            auto finish_s_load = [&]() {
                if (s_in) return;
                s_in = true;
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&S.s_free);
            };

            const int jmax = j0 + BN - 1;
            const bool full = (!p.causal || jmax <= P0) && (jmax < Lk) &&
                              (p.win_last <= 0 || jmax < p.win_first || j0 >= P1 + 1 - p.win_last);
            int c_hi = BN, f_hi = BN, w_lo = 0;
            if (!full) {
                c_hi = p.causal ? pos - j0 + 1 : BN;
                c_hi = min(c_hi, Lk - j0);
                f_hi = p.win_last > 0 ? p.win_first - j0 : BN;
                w_lo = p.win_last > 0 ? pos + 1 - p.win_last - j0 : 0;
            }
            // Hidden keys of columns 64*hf .. 64*hf + 63 become -inf.
            auto mask_half = [&](auto hfc) {
                constexpr int hf = decltype(hfc)::value;
#pragma unroll
                for (int c = 2 * hf; c < 2 * hf + 2; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int cc = c * 32 + i;
                        const bool vis = cc < c_hi && (cc < f_hi || cc >= w_lo);
                        if (!vis) s[c][i] = __float_as_uint(-INFINITY);
                    }
            };
            // P = 2^(s*scale*log2e - m_use) of one half into w[32*hf ..] (packed fp32x2
            // FMA, MUFU ex2, packed partial sums); returns the half's row sum.
            uint32_t w[64];
            auto exps_half = [&](auto hfc, float m_use) -> float {
                constexpr int hf = decltype(hfc)::value;
                const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(-m_use, -m_use);
                uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int e = 32 * hf; e < 32 * hf + 32; ++e) {
                    const int i0 = 2 * e;
                    const uint64_t y = f2_fma(f2_pack(__uint_as_float(s[i0 >> 5][i0 & 31]),
                                                      __uint_as_float(s[(i0 + 1) >> 5][(i0 + 1) & 31])),
                                              sc2, nm2);
                    float y0, y1;
                    f2_unpack(y, y0, y1);
                    const float x0 = fast_exp2(y0), x1 = fast_exp2(y1);
                    acc2[e & 3] = f2_add(acc2[e & 3], f2_pack(x0, x1));
                    w[e] = pack_bf16x2(x0, x1);
                }
                float sum = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float lo, hi;
                    f2_unpack(acc2[e], lo, hi);
                    sum += lo + hi;
                }
                return sum;
            };
            using H0 = std::integral_constant<int, 0>;
            using H1 = std::integral_constant<int, 1>;
            // The previous P V must be complete before P is overwritten or O
            // rescaled; it normally finished while this tile's S was computed.
            auto wait_prev_pv = [&]() -> bool {
                if (it == 0) return true;
                const bool done = __all_sync(0xffffffffu, mbar_wait(&S.o_done, (it - 1) & 1, abort));
                if (done) tc_fence_after();
                return done;
            };
            // Fast path: exponentiate against the current reference without the row
            // max.  Every value is then <= 2^64 unless a half's row sum exceeds 2^64
            // (or overflowed), in which case the exact pass redoes the tile.
            bool slow = __any_sync(0xffffffffu, m_ref == -INFINITY);
            bool stored0 = false;
            float rs = 0.f;
            if (!slow) {
                if (!full) mask_half(H0{});
                const float rs0 = exps_half(H0{}, m_ref);
                finish_s_load();
                const bool ok0 = !__any_sync(0xffffffffu, !(rs0 <= kFastSumLimit));
                if (!(ok = wait_prev_pv())) break;
                if (ok0) {
                    tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&w[0]));
                    stored0 = true;
                }
                if (!full) mask_half(H1{});
                const float rs1 = exps_half(H1{}, m_ref);
                const bool ok1 = !__any_sync(0xffffffffu, !(rs1 <= kFastSumLimit));
                if (ok0 && ok1) {
                    rs = rs0 + rs1;
                    tmem_st32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&w[32]));
                } else {
                    slow = true;
                }
            } else {
                finish_s_load();
                if (!full) {
                    mask_half(H0{});
                    mask_half(H1{});
                }
                if (!(ok = wait_prev_pv())) break;
            }
            if (slow) {
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
                const float mx = max3f(max3f(mc[0], mc[1], mc[2]), max3f(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
                const float m_new = fmaxf(m_ref, mx * sl2);
                const bool resc = m_new > m_ref + kRescaleThreshold;
                const float alpha = resc ? fast_exp2(m_ref - m_new) : 1.f;
                if (resc) {
                    l *= alpha;
                    m_ref = m_new;
                }
                const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
                rs = exps_half(H0{}, m_use) + exps_half(H1{}, m_use);
                if (it > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t o[32];
                        tmem_ld32(tO + ch * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + ch * 32, o);
                    }
                }
                if (stored0) tmem_st_wait();  // the first half's earlier store lands before its rewrite
                // P as bf16 pairs: TMEM column c holds keys 2c (low half) and 2c+1.
                tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&w[0]));
                tmem_st32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&w[32]));
            }
            l += rs;
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&S.p_full);
        }

        // -------------------------------------------------------------- epilogue
        if (ok && ntiles > 0) ok = mbar_wait(&S.o_done, (ntiles - 1) & 1, abort);
        ok = __all_sync(0xffffffffu, ok);
        const bool have = ok && ntiles > 0;
        if (have) tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int row = q_start + qs + r;
        const bool store = r < rows_valid && ok;
        uint4* dst = reinterpret_cast<uint4*>(p.out + ((size_t)row * p.hq + h) * D);
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t u[32];
            if (have) {  // warp-uniform: every lane takes part in the collective load
                tmem_ld32(tO + ch * 32, u);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) u[i] = 0u;
            }
            if (store) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 wv;
                    wv.x = pack_bf16x2(__uint_as_float(u[8 * c + 0]) * inv, __uint_as_float(u[8 * c + 1]) * inv);
                    wv.y = pack_bf16x2(__uint_as_float(u[8 * c + 2]) * inv, __uint_as_float(u[8 * c + 3]) * inv);
                    wv.z = pack_bf16x2(__uint_as_float(u[8 * c + 4]) * inv, __uint_as_float(u[8 * c + 5]) * inv);
                    wv.w = pack_bf16x2(__uint_as_float(u[8 * c + 6]) * inv, __uint_as_float(u[8 * c + 7]) * inv);
                    dst[ch * 4 + c] = wv;
                }
            }
        }
        if (store && p.lse) p.lse[(size_t)h * p.total_q + row] = l > 0.f ? (m_ref + log2f(l)) * ATTN_LN2 : -INFINITY;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}


// ---------------------------------------------------------------------------
// Head dim 128, two query heads of a KV group per CTA: fwd2_kernel.  One CTA
// per SM holds the same 128 query rows of heads 2 hp and 2 hp + 1 (tiles A and
// B), which share every K / V tile.  Each tile has its own softmax warpgroup
// and its own MMA-issuing warp; P is written over the S columns it came from
// (TMEM: S_A, O_A, S_B, O_B, 128 columns each), so a tile's next S is issued
// only once its P V has read P, and the softmax never waits for P V.  Tile B's
// chain starts after tile A's first P: the two softmax phases alternate, one
// warpgroup exponentiating while the tensor core runs the other tile's P V and
// S, which a single 128-row tile per SM leaves idle.
namespace x2 {
constexpr int kThreads = 384;   // warps 0-3 control, 4-7 softmax A, 8-11 softmax B
constexpr int kRegsCtrl = 72;   // 128 * 72 + 256 * 216 = 64512 = 384 * 168 (launch)
constexpr int kRegsSoftmax = 216;
// K / V ring stages: 2 at head dim 128 (192 KB in all with the two Q tiles).
template <int D>
constexpr int kStagesFor = D == 64 ? 3 : 2;

template <int D>
struct __align__(1024) Smem {
    static constexpr int kStages = kStagesFor<D>;
    static constexpr uint32_t kTile = Cfg<D>::kTile;
    uint8_t q[2][kTile];
    uint8_t k[kStages][kTile];
    uint8_t v[kStages][kTile];
    uint64_t q_full;
    uint64_t k_full[kStages], k_empty[kStages];
    uint64_t v_full[kStages], v_empty[kStages];
    uint64_t s_full[2], p_full[2], o_done[2];  // per tile: one phase per key tile
    uint64_t final_bar[2];
    uint64_t v_tail;
    uint32_t tmem_base;
    int abort;
};
}  // namespace x2

template <int D, bool kPaged>
__global__ void __launch_bounds__(x2::kThreads, 1)
    fwd2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const Params p) {
    using C = Cfg<D>;
    constexpr int kStages = x2::kStagesFor<D>;
    constexpr uint32_t kTile = C::kTile;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem_al =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    x2::Smem<D>& S = *reinterpret_cast<x2::Smem<D>*>(smem_al);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Grid (head pair, row tile, request), as fwd_kernel with head pairs.
    const int hp = blockIdx.x;
    const int rt = p.n_rt - 1 - (int)blockIdx.y;
    const int b = blockIdx.z;

    const int q_start = p.cu_q[b];
    int Lq = p.cu_q[b + 1] - q_start;
    const bool paged = kPaged;
    const int k_start = paged ? 0 : p.cu_k[b];
    int Lk = paged ? p.seqlens_k[b] : p.cu_k[b + 1] - k_start;
    const long long k_cap = paged ? ((long long)p.max_pages << p.page_shift) : (long long)p.total_k - k_start;
    if (q_start + Lq > p.total_q || Lk > k_cap || Lq < 0 || Lk < 0) {
        if (threadIdx.x == 0 && rt == 0 && hp == 0) raise_status(ATTN_SINK_DEV_SEQLEN_OOB);
        Lq = max(0, min(Lq, p.total_q - q_start));
        Lk = (int)max(0LL, min((long long)Lk, k_cap));
    }
    const int qs = rt * BM;
    if (qs >= Lq) return;
    const int kvh = (2 * hp) / p.group;

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
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&S.k_full[s], 1);
            mbar_init(&S.k_empty[s], 2);  // both tiles' S products
            mbar_init(&S.v_full[s], 1);
            mbar_init(&S.v_empty[s], 2);  // both tiles' P V products
        }
        for (int w = 0; w < 2; ++w) {
            mbar_init(&S.s_full[w], 1);
            mbar_init(&S.p_full[w], 128);
            mbar_init(&S.o_done[w], 1);
            mbar_init(&S.final_bar[w], 1);
        }
        mbar_init(&S.v_tail, 1);
        S.abort = 0;
        fence_mbar_init();
        // Contiguous K / V: Q and the first ring's worth of K and V tiles are
        // requested while TMEM is allocated and the CTA synchronises.
        if constexpr (!kPaged) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            mbar_expect_tx(&S.q_full, 2 * kTile);
            tma_tile<D>(S.q[0], &tm_q, &S.q_full, 2 * hp, q_start + qs);
            tma_tile<D>(S.q[1], &tm_q, &S.q_full, 2 * hp + 1, q_start + qs);
            for (int it = 0; it < ntiles && it < kStages; ++it) {
                const int t = it < ta ? it : tb + (it - ta);
                mbar_expect_tx(&S.k_full[it], kTile);
                tma_tile<D>(S.k[it], &tm_k, &S.k_full[it], kvh, k_start + t * BN);
                uint64_t* bar = (t + 1) * BN > Lk ? &S.v_tail : &S.v_full[it];
                mbar_expect_tx(bar, kTile);
                tma_tile<D>(S.v[it], &tm_v, bar, kvh, k_start + t * BN);
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(&S.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    volatile int* abort = &S.abort;

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(x2::kRegsCtrl));
        if (warp == 0 || warp == 2) {
            // -------------------------------------------------------- producers
            // As in fwd_kernel: warp 0 streams K (and, paged, the two Q tiles),
            // warp 2 streams V; a stage is free once both tiles' products have
            // read it.
            const bool is_k = warp == 0;
            uint64_t* full = is_k ? S.k_full : S.v_full;
            uint64_t* empty = is_k ? S.k_empty : S.v_empty;
            uint8_t* dst0 = is_k ? S.k[0] : S.v[0];
            const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
            const int nseg = BN >> p.seg_shift;
            if (paged && lane == 0) {
                prefetch_tmap(tm);
                if (is_k) {
                    prefetch_tmap(&tm_q);
                    mbar_expect_tx(&S.q_full, 2 * kTile);
                    tma_tile<D>(S.q[0], &tm_q, &S.q_full, 2 * hp, q_start + qs);
                    tma_tile<D>(S.q[1], &tm_q, &S.q_full, 2 * hp + 1, q_start + qs);
                }
            }
            bool tail_issued = false;
            int it = 0;
            for (; it < ntiles; ++it) {
                const int st = it % kStages;
                if (it >= kStages &&
                    !__all_sync(0xffffffffu, mbar_wait(&empty[st], ((it / kStages) - 1) & 1, abort)))
                    break;
                const int t = it < ta ? it : tb + (it - ta);
                const bool tail = !is_k && (t + 1) * BN > Lk;
                uint64_t* bar = tail ? &S.v_tail : &full[st];
                if constexpr (!kPaged) {
                    if (lane == 0 && it >= kStages) {  // the first kStages were issued at start-up
                        mbar_expect_tx(bar, kTile);
                        tma_tile<D>(dst0 + st * kTile, tm, bar, kvh, k_start + t * BN);
                    }
                } else {
                    int slot = 0;
                    const int j = t * BN + (lane << p.seg_shift);
                    if (lane < nseg && j < Lk) {
                        const int pg = __ldg(p.page_table + (size_t)b * p.max_pages + (j >> p.page_shift));
                        if (pg >= 0 && pg < p.num_pages)
                            slot = (pg << p.page_shift) | (j & ((1 << p.page_shift) - 1));
                        else
                            raise_status(ATTN_SINK_DEV_PAGE_OOB);
                    }
                    if (lane == 0) mbar_expect_tx(bar, kTile);
                    __syncwarp();
                    if (lane < nseg)
                        tma_tile<D>(dst0 + st * kTile + ((uint32_t)lane << p.seg_shift) * 128u, tm, bar, kvh, slot);
                }
                if (tail) {
                    // Used once per CTA (one tile holds the last key): parity 0.  The rows
                    // at or past the last key are zeroed before the stage is released.
                    tail_issued = true;
                    if (!__all_sync(0xffffffffu, mbar_wait(&S.v_tail, 0, abort))) break;
#pragma unroll
                    for (int a = 0; a < C::kAtoms; ++a) {
                        uint4* vt = reinterpret_cast<uint4*>(dst0 + st * kTile + a * kAtom);
                        for (int c = (Lk - t * BN) * 8 + lane; c < BN * 8; c += 32) vt[c] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full[st]);
                }
            }
            if (lane == 0) {
                if (is_k) drain_wait(&S.q_full, 0);
                if (tail_issued) drain_wait(&S.v_tail, 0);
                for (int st = 0; st < kStages; ++st) {
                    const int n = it > st ? (it - st + kStages - 1) / kStages : 0;
                    if (n > 0) drain_wait(&full[st], (n - 1) & 1);
                }
            }
            __syncwarp();
        } else if (ntiles > 0) {
            // -------------------------------------------------------- MMA issuers
            // Warp 1 issues tile A's S and P V, warp 3 tile B's.  A tile's S(it)
            // overwrites the P it made at it - 1, so it waits for that P V; tile B's
            // first S waits for tile A's first P, which puts the two chains half a
            // period apart.
            const int wgt = warp == 1 ? 0 : 1;
            const uint32_t cS = (uint32_t)wgt * 256, cO = cS + 128;
            constexpr uint32_t idS = idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t idO = idesc_bf16_f32(BM, D, false, true);
            const uint64_t dq = sdesc_sw128(smem_u32(S.q[wgt]), 16, 1024);
            const uint64_t dk0 = sdesc_sw128(smem_u32(S.k[0]), 16, 1024);
            const uint64_t dv0 = sdesc_sw128(smem_u32(S.v[0]), kAtom, 1024);  // MN atoms kAtom apart
            auto wait_all = [&](uint64_t* bar, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
            };
            bool ok = wait_all(&S.q_full, 0);
            if (ok && wgt == 1) ok = wait_all(&S.p_full[0], 0);
            for (int it = 0; ok && it < ntiles; ++it) {
                const int st = it % kStages;
                if (!(ok = wait_all(&S.k_full[st], (it / kStages) & 1))) break;
                if (it > 0 && !(ok = wait_all(&S.o_done[wgt], (it - 1) & 1))) break;
                tc_fence_after();
                const uint64_t dk = dk0 + st * (kTile >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t o = (kk >> 2) * (kAtom >> 4) + (kk & 3) * 2;
                    umma_ss_e(tmem + cS, dq + o, dk + o, idS, kk > 0);
                }
                umma_commit_e(&S.s_full[wgt]);
                umma_commit_e(&S.k_empty[st]);
                if (!(ok = wait_all(&S.v_full[st], (it / kStages) & 1))) break;
                if (!(ok = wait_all(&S.p_full[wgt], it & 1))) break;
                tc_fence_after();
                const uint64_t dv = dv0 + st * (kTile >> 4);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    umma_ts_e(tmem + cO, tmem + cS + kk * 8, dv + 128 * kk, idO, (it > 0 || kk > 0) ? 1u : 0u);
                umma_commit_e(&S.o_done[wgt]);
                umma_commit_e(&S.v_empty[st]);
            }
            umma_commit_e(&S.final_bar[wgt]);
            drain_wait(&S.final_bar[wgt], 0);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(x2::kRegsSoftmax));
        // ------------------------------------------------------------ softmax
        // Warpgroup wg (tile wg, head 2 hp + wg), as in fwd_kernel with P written
        // over the S columns of its tile.
        const int wg = (warp - 4) >> 2;
        const int h = 2 * hp + wg;
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        const uint32_t tS = tmem + lane_base + (uint32_t)wg * 256;
        const uint32_t tO = tS + 128;
        const uint32_t tP = tS;
        const float sg = p.sink ? p.sink[h] * ATTN_LOG2E : -INFINITY;
        const float sl2 = p.scale_log2;
        float m_ref = sg;
        float l = sg == -INFINITY ? 0.f : 1.f;
        const int pos = off + qs + r;
        bool ok = true;
        for (int it = 0; it < ntiles; ++it) {
            const int t = it < ta ? it : tb + (it - ta);
            const int j0 = t * BN;
            ok = mbar_wait(&S.s_full[wg], it & 1, abort);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // S is read into registers; P is computed and stored over it in two
            // halves, the first half's TMEM store overlapping the second half's exp2
            // work.  This tile's next S is issued once its P V has read P, and in the
            // meantime the tensor core runs the other tile's products.
            uint32_t s[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, s[c]);
            tmem_ld_wait();

            const int jmax = j0 + BN - 1;
            const bool full = (!p.causal || jmax <= P0) && (jmax < Lk) &&
                              (p.win_last <= 0 || jmax < p.win_first || j0 >= P1 + 1 - p.win_last);
            int c_hi = BN, f_hi = BN, w_lo = 0;
            if (!full) {
                c_hi = p.causal ? pos - j0 + 1 : BN;
                c_hi = min(c_hi, Lk - j0);
                f_hi = p.win_last > 0 ? p.win_first - j0 : BN;
                w_lo = p.win_last > 0 ? pos + 1 - p.win_last - j0 : 0;
            }
            // Hidden keys of columns 64*hf .. 64*hf + 63 become -inf.
            auto mask_half = [&](auto hfc) {
                constexpr int hf = decltype(hfc)::value;
#pragma unroll
                for (int c = 2 * hf; c < 2 * hf + 2; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int cc = c * 32 + i;
                        const bool vis = cc < c_hi && (cc < f_hi || cc >= w_lo);
                        if (!vis) s[c][i] = __float_as_uint(-INFINITY);
                    }
            };
            // P = 2^(s*scale*log2e - m_use) of one half into w[32*hf ..] (packed fp32x2
            // FMA, MUFU ex2, packed partial sums); returns the half's row sum.
            uint32_t w[64];
            auto exps_half = [&](auto hfc, float m_use) -> float {
                constexpr int hf = decltype(hfc)::value;
                const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(-m_use, -m_use);
                uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int e = 32 * hf; e < 32 * hf + 32; ++e) {
                    const int i0 = 2 * e;
                    const uint64_t y = f2_fma(f2_pack(__uint_as_float(s[i0 >> 5][i0 & 31]),
                                                      __uint_as_float(s[(i0 + 1) >> 5][(i0 + 1) & 31])),
                                              sc2, nm2);
                    float y0, y1;
                    f2_unpack(y, y0, y1);
                    const float x0 = fast_exp2(y0), x1 = fast_exp2(y1);
                    acc2[e & 3] = f2_add(acc2[e & 3], f2_pack(x0, x1));
                    w[e] = pack_bf16x2(x0, x1);
                }
                float sum = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float lo, hi;
                    f2_unpack(acc2[e], lo, hi);
                    sum += lo + hi;
                }
                return sum;
            };
            using H0 = std::integral_constant<int, 0>;
            using H1 = std::integral_constant<int, 1>;
            // The previous P V must be complete before P is overwritten or O
            // rescaled; it normally finished while this tile's S was computed.
            // (P overwrites this tile's S columns, and O may be rescaled, only after the
            // previous P V: this S was issued after that completed, so no wait here.)
            // Fast path: exponentiate against the current reference without the row
            // max.  Every value is then <= 2^64 unless a half's row sum exceeds 2^64
            // (or overflowed), in which case the exact pass redoes the tile.
            bool slow = __any_sync(0xffffffffu, m_ref == -INFINITY);
            bool stored0 = false;
            float rs = 0.f;
            if (!slow) {
                if (!full) mask_half(H0{});
                const float rs0 = exps_half(H0{}, m_ref);
                const bool ok0 = !__any_sync(0xffffffffu, !(rs0 <= kFastSumLimit));
                if (ok0) {
                    tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&w[0]));
                    stored0 = true;
                }
                if (!full) mask_half(H1{});
                const float rs1 = exps_half(H1{}, m_ref);
                const bool ok1 = !__any_sync(0xffffffffu, !(rs1 <= kFastSumLimit));
                if (ok0 && ok1) {
                    rs = rs0 + rs1;
                    tmem_st32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&w[32]));
                } else {
                    slow = true;
                }
            } else {
                if (!full) {
                    mask_half(H0{});
                    mask_half(H1{});
                }
            }
            if (slow) {
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
                const float mx = max3f(max3f(mc[0], mc[1], mc[2]), max3f(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
                const float m_new = fmaxf(m_ref, mx * sl2);
                const bool resc = m_new > m_ref + kRescaleThreshold;
                const float alpha = resc ? fast_exp2(m_ref - m_new) : 1.f;
                if (resc) {
                    l *= alpha;
                    m_ref = m_new;
                }
                const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
                rs = exps_half(H0{}, m_use) + exps_half(H1{}, m_use);
                if (it > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t o[32];
                        tmem_ld32(tO + ch * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + ch * 32, o);
                    }
                }
                if (stored0) tmem_st_wait();  // the first half's earlier store lands before its rewrite
                // P as bf16 pairs: TMEM column c holds keys 2c (low half) and 2c+1.
                tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&w[0]));
                tmem_st32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&w[32]));
            }
            l += rs;
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&S.p_full[wg]);
        }


        // -------------------------------------------------------------- epilogue
        if (ok && ntiles > 0) ok = mbar_wait(&S.o_done[wg], (ntiles - 1) & 1, abort);
        ok = __all_sync(0xffffffffu, ok);
        const bool have = ok && ntiles > 0;
        if (have) tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int row = q_start + qs + r;
        const bool store = r < rows_valid && ok;
        uint4* dst = reinterpret_cast<uint4*>(p.out + ((size_t)row * p.hq + h) * D);
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t u[32];
            if (have) {  // warp-uniform: every lane takes part in the collective load
                tmem_ld32(tO + ch * 32, u);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) u[i] = 0u;
            }
            if (store) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 wv;
                    wv.x = pack_bf16x2(__uint_as_float(u[8 * c + 0]) * inv, __uint_as_float(u[8 * c + 1]) * inv);
                    wv.y = pack_bf16x2(__uint_as_float(u[8 * c + 2]) * inv, __uint_as_float(u[8 * c + 3]) * inv);
                    wv.z = pack_bf16x2(__uint_as_float(u[8 * c + 4]) * inv, __uint_as_float(u[8 * c + 5]) * inv);
                    wv.w = pack_bf16x2(__uint_as_float(u[8 * c + 6]) * inv, __uint_as_float(u[8 * c + 7]) * inv);
                    dst[ch * 4 + c] = wv;
                }
            }
        }
        if (store && p.lse) p.lse[(size_t)h * p.total_q + row] = l > 0.f ? (m_ref + log2f(l)) * ATTN_LN2 : -INFINITY;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
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

// (rows, heads, d) bf16 tensor viewed as a 3-D map {d, head, row}; box {64, 1,
// box_rows}: one 128-byte-swizzled atom per copy (d / 64 copies per tile).
// Rows are row_stride elements apart (0: heads * d, i.e. contiguous).
cudaError_t make_map(CUtensorMap* m, const void* base, int d, int heads, long long rows, int box_rows,
                     std::string* what, long long row_stride = 0) {
    const int D = d;
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

// Head dim 128 runs two query heads per CTA (fwd2_kernel) when the group is even.
// At head dim 64 the same kernel measured 833 against 1158 TFLOP/s on the varlen
// extend: there two independent CTAs per SM (fwd_kernel) keep the tensor core
// busier than one CTA whose two chains wait for each P V before the next S.
template <int D>
constexpr bool kTwoHeadsFor = D == 128;

template <int D>
static cudaError_t launch_fwd_d(const FwdArgs& a, cudaStream_t s, std::string* what) {
    constexpr bool kTwoHeads = kTwoHeadsFor<D>;
    CUtensorMap tq, tk, tv;
    cudaError_t e;
    const bool paged = a.page_table != nullptr;
    int page_shift = 0, seg_shift = 7;
    if (paged) {
        while ((1 << page_shift) < a.page_size) ++page_shift;
        seg_shift = page_shift < 7 ? page_shift : 7;  // segments of min(page_size, 128) rows
    }
    const long long krows = paged ? (long long)a.num_pages * a.page_size : a.total_k;
    if ((e = make_map(&tq, a.q, D, a.hq, a.total_q, BM, what, a.q_rs)) != cudaSuccess) return e;
    if ((e = make_map(&tk, a.k, D, a.hkv, krows, 1 << seg_shift, what, a.k_rs)) != cudaSuccess) return e;
    if ((e = make_map(&tv, a.v, D, a.hkv, krows, 1 << seg_shift, what, a.v_rs)) != cudaSuccess) return e;
    Params p;
    p.page_table = a.page_table;
    p.seqlens_k = a.seqlens_k;
    p.max_pages = a.max_pages;
    p.page_shift = page_shift;
    p.seg_shift = seg_shift;
    p.num_pages = a.num_pages;
    p.sink = a.sink;
    p.cu_q = a.cu_q;
    p.cu_k = a.cu_k;
    p.out = reinterpret_cast<__nv_bfloat16*>(a.out);
    p.lse = a.lse;
    p.hq = a.hq;
    p.group = a.hq / a.hkv;
    p.n_rt = (a.max_seqlen_q + BM - 1) / BM;
    p.total_q = a.total_q;
    p.total_k = a.total_k;
    p.win_first = a.win_first;
    p.win_last = a.win_last;
    p.causal = a.causal;
    p.scale_log2 = a.scale * ATTN_LOG2E;
    const size_t smem = sizeof(Smem<D>) + (Cfg<D>::kTwoPerSm ? 0 : 1024);
    if constexpr (kTwoHeads) if (p.group % 2 == 0) {
        // an even query-head group: two heads per CTA (fwd2_kernel)
        const size_t smem2 = sizeof(x2::Smem<D>) + 1024;
        static_assert(sizeof(x2::Smem<D>) + 1024 <= 227 * 1024, "shared memory of fwd2_kernel");
        auto kernel2 = paged ? fwd2_kernel<D, true> : fwd2_kernel<D, false>;
        e = cudaFuncSetAttribute(kernel2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
        if (e != cudaSuccess) {
            *what = "smem attribute";
            return e;
        }
        dim3 grid2(a.hq / 2, p.n_rt, a.batch);
        kernel2<<<grid2, x2::kThreads, smem2, s>>>(tq, tk, tv, p);
        e = cudaGetLastError();
        if (e != cudaSuccess) *what = "launch";
        return e;
    }
    auto kernel = paged ? fwd_kernel<D, true> : fwd_kernel<D, false>;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
        *what = "smem attribute";
        return e;
    }
    dim3 grid(a.hq, p.n_rt, a.batch);
    kernel<<<grid, kThreads, smem, s>>>(tq, tk, tv, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) *what = "launch";
    return e;
}

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t s, std::string* what) {
    if (a.total_q == 0) return cudaSuccess;
    if (a.head_dim == 128) return launch_fwd_d<128>(a, s, what);
    return launch_fwd_d<64>(a, s, what);
}

ATTN_DEFINE_STATUS_ACCESSOR(status_exchange)

}  // namespace prefill
}  // namespace attn
