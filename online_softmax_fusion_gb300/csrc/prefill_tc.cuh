// Warp-specialised tcgen05 prefill: the Rolling Update form of attention on
// the 5th-generation tensor cores.
//
// Rolling Update (Neptune论文浅读 (gentlecold.top) §5) streams K/V tiles past
// resident Q tiles and repairs the running sum and output with
// exp(m_old - m_new) whenever the row max grows (§3-§4). The warp roles follow
// the Blackwell schedule the Twill review (xllm-io) re-derives in §七 /
// Figure 9: variable-latency loads in one warp, tensor-core GEMMs in another,
// the softmax of two Q sub-tiles in two separate warp groups. That page puts
// the accumulator rescaling in a third group because TMEM reads block; here
// the rescale is conditional (it runs only when a row max grows by more than
// 2^8, which after the first KV tile is rare) and the softmax group does it.
//
// Two CTA forms (template parameter NT, the Q tiles per CTA):
//  * NT = 2, one CTA per SM: two 128-row Q tiles that share one KV head,
//    either two consecutive row blocks of one head (MHA) or the same row
//    block of two query heads of a GQA group. Tensor memory (512 columns):
//    S_0, S_1 (128 fp32 columns each), O_0, O_1 (d columns each). The two
//    tiles alternate on the tensor core.
//  * NT = 1, two CTAs per SM: one 128-row Q tile, half the shared memory
//    (a 2-slot K/V ring for head dim 128) and half the tensor memory (S, O).
//    The two resident CTAs alternate on the tensor core instead, and one
//    CTA's start (Q load, first products) and end (epilogue) overlap the
//    other's steady state; twice the CTAs also fill the SMs at short lengths.
// P_t (bf16, two keys per column) is written over the upper half of S_t, and
// the PV product reads it straight from tensor memory, so per KV step shared
// memory only carries Q K^T's operands, V and the TMA writes.
//
// Per KV step j, for each tile t (the two tiles alternate on the tensor core):
//   TMA warp : K_j, V_j -> 5-slot shared-memory ring (128-byte swizzle)
//   MMA warp : O_t += P_t V_j (A from TMEM), then S_t = Q_t K_j'^T for the
//              tile j' scanned next
//   softmax t: S_t (TMEM) -> registers, row max, p = 2^(x - m), row sum,
//              P_t (bf16) -> TMEM, O_t rescale in TMEM if needed
// The commit that signals S_t for j' also covers the PV product issued
// before it, so when the softmax sees it, O_t is final for step j. One thread
// owns one query row (TMEM lane = row): row reductions need no shuffles.
// KV tiles are scanned in ascending order, or diagonal-first under causal
// ALiBi (the bias then peaks on the first tile) and causal windows. SoftCap
// evaluates tanh as a polynomial on the FMA pipe where |score / cap| allows
// it. O leaves through each tile's Q buffer as bulk tensor stores in the
// paired-head and capped forms, as direct row stores elsewhere.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace attn {

namespace {

// NT = 2: 12 warps = 3 warpgroups (warp 0 TMA, warp 1 MMA, warps 4..7 the
// softmax of tile 0, 8..11 of tile 1). NT = 1: 6 warps (warp 0 TMA, warp 1
// MMA, warps 2..5 the softmax; their TMEM lane quadrants are warp % 4).
template <int NT> constexpr int tc_threads() { return NT == 2 ? 384 : 192; }
template <int NT> constexpr int softmax_warp0() { return NT == 2 ? 4 : 2; }
// Register split of the NT = 2 form (setmaxnreg, per warpgroup): launch
// 168 x 384 = 64512; producer/MMA group 96 x 128 + two softmax groups
// 192 x 256 = 61440 for head dim 128, 80 x 128 (59392) for head dim 64:
// chosen from the compiler's spill report (no spills in any variant). The
// NT = 1 form runs two CTAs of 192 threads at 168 registers each.
template <int D, bool EXTRA>
constexpr int regs_ctl() { return D == 128 ? 96 : 80; }
constexpr int kRegsSoftmax = 192;
constexpr float kRescaleThreshold = 8.0f;       // log2 units: rescale when max grows > 2^8
constexpr uint32_t kTileBytes = 128 * 128;      // one 128-row x 128-byte swizzled box

template <int D, int NT>
struct TcCfg {
    static constexpr int kBoxes = D / 64;                   // 64-element boxes per row
    // K/V ring slots: ~160 KB of ring with one CTA per SM, ~64-80 KB with two
    static constexpr int kStages = NT == 2 ? (D == 128 ? 5 : 10) : (D == 128 ? 2 : 5);
    static constexpr uint32_t kSlotBytes = kBoxes * kTileBytes;
    static constexpr uint32_t kTmemCols = NT == 2 ? 512 : 256;
    static constexpr uint32_t kOCol = NT * 128;              // O_0 after the S tiles
};

template <int D, int NT>
struct TcSmem {
    alignas(1024) uint8_t q[NT][TcCfg<D, NT>::kBoxes][kTileBytes];
    alignas(1024) uint8_t kv[TcCfg<D, NT>::kStages][TcCfg<D, NT>::kBoxes][kTileBytes];
    uint64_t bar_q;
    uint64_t kv_full[TcCfg<D, NT>::kStages];
    uint64_t kv_empty[TcCfg<D, NT>::kStages];
    uint64_t s_full[NT];
    uint64_t p_full[NT];
    uint64_t o_done[NT];
    uint64_t mma_fin;
    uint32_t tmem_base;
    int abort;
};
// dynamic shared memory per CTA is at most 227 KB (plus 1 KB of alignment slack)
static_assert(sizeof(TcSmem<128, 2>) + 1024 <= 232448, "shared memory of the two-tile form");
static_assert(sizeof(TcSmem<64, 2>) + 1024 <= 232448, "shared memory of the two-tile form");
// two CTAs per SM: 228 KB per SM, 1 KB of it reserved per CTA
static_assert(2 * (sizeof(TcSmem<128, 1>) + 1024 + 1024) <= 233472, "two one-tile CTAs per SM");
static_assert(2 * (sizeof(TcSmem<64, 1>) + 1024 + 1024) <= 233472, "two one-tile CTAs per SM");

// tanh(y) ~ y (1 + a3 y^2 + a5 y^4) for |y| <= 0.4: a near-minimax fit of
// the absolute error (Lawson-reweighted least squares on [0, 0.4], max error
// 2.0e-6); tests/test_tanh_fit.py repeats the fit and checks it.
constexpr float kTanhRange = 0.4f;
constexpr float kTanhA3 = -3.326916256e-01f;
constexpr float kTanhA5 = 1.214116698e-01f;

// KV tiles [lo, hi) that the 128 query rows starting at row0 can see.
struct KvRange {
    int lo, hi;
};

__device__ __forceinline__ KvRange kv_range_for(int row0, const PrefillParams& p, bool causal) {
    KvRange r{0, 0};
    if (row0 >= p.Lq) return r;
    const int off = p.Lk - p.Lq;
    const int last = min(row0 + 127, p.Lq - 1);
    int kend = p.Lk;
    if (causal) kend = min(kend, last + off + 1);
    if (p.window_right >= 0) kend = min(kend, last + off + p.window_right + 1);
    int kbeg = 0;
    if (p.window_left >= 0) kbeg = max(0, row0 + off - p.window_left);
    if (kend <= kbeg) return r;
    r.lo = kbeg / 128;
    r.hi = (kend + 127) / 128;
    return r;
}

}  // namespace

// MODE 0: plain. 1: a sliding window (masked tiles take the per-element
// path). 2: SoftCap (cap * tanh(score / cap) on every score, window allowed).
// SoftCap has a variant of its own so that the plain and window code keep
// their register allocation. (Computing 1 / (1 + u) for the tanh on the FMA
// pipe instead of the special-function unit measured slower: 524 against
// 582 TFLOP/s on causal MHA at cap 30.)
template <int D, bool CAUSAL, bool ALIBI, int MODE, int NT>
__global__ void __launch_bounds__(tc_threads<NT>(), NT == 2 ? 1 : 2)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmO, PrefillParams p) {
    constexpr bool EXTRA = MODE != 0;
    constexpr bool CAPPED = MODE == 2;
    // KV tiles in descending order (diagonal first) under causal ALiBi: the
    // bias grows toward the diagonal, so an ascending scan raises the row
    // maximum on nearly every tile (81 % of the steps of the GQA + ALiBi 4k
    // sweep rescaled O, 13 % of the softmax cycles); scanned downward the
    // maximum is set by the first tile. The online softmax is order-free.
    // The window form also measured faster this way (causal, left 1024:
    // 258.6 against 269.3 us); plain causal and capped forms did not (MHA 4k
    // 399.7 against 397.8, 1k 17.5 against 16.7).
    constexpr bool REV = CAUSAL && (ALIBI || MODE == 1);
    using Cfg = TcCfg<D, NT>;
    constexpr int NS = Cfg::kStages;
    constexpr int kSoftmaxWarp0 = softmax_warp0<NT>();
    extern __shared__ uint8_t smem_raw[];
    TcSmem<D, NT>& sm = *reinterpret_cast<TcSmem<D, NT>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int off = p.Lk - p.Lq;

    // ---- work item: NT Q tiles sharing one KV head, heaviest rows first
    const int pair_heads = NT == 2 ? p.pair_heads : 0;
    const int n_hb = pair_heads ? p.Hq / 2 : p.Hq;
    const int rows_per_item = (NT == 1 || pair_heads) ? 128 : 256;
    const int n_rb = (p.Lq + rows_per_item - 1) / rows_per_item;
    const int rb = n_rb - 1 - int(blockIdx.x) / n_hb;
    const int hb = int(blockIdx.x) % n_hb;
    const int head0 = pair_heads ? 2 * hb : hb;
    const int head1 = pair_heads ? 2 * hb + 1 : hb;
    const int row00 = rb * rows_per_item;
    const int row01 = pair_heads ? row00 : row00 + 128;
    KvRange rg0 = kv_range_for(row00, p, CAUSAL);
    KvRange rg1 = NT == 2 ? kv_range_for(row01, p, CAUSAL) : KvRange{0, 0};
    if (p.splits > 1) {
        // split-KV: this CTA takes chunk blockIdx.z of the union of its two
        // tiles' KV ranges and writes fp32 partials for a combine
        const bool f0 = rg0.hi <= rg0.lo, f1 = rg1.hi <= rg1.lo;
        if (!(f0 && f1)) {
            const int ulo = f0 ? rg1.lo : (f1 ? rg0.lo : min(rg0.lo, rg1.lo));
            const int uhi = f0 ? rg1.hi : (f1 ? rg0.hi : max(rg0.hi, rg1.hi));
            const int chunk = (uhi - ulo + p.splits - 1) / p.splits;
            const int s0 = ulo + int(blockIdx.z) * chunk;
            const int s1 = min(uhi, s0 + chunk);
            rg0.lo = max(rg0.lo, s0);
            rg0.hi = min(rg0.hi, s1);
            rg1.lo = max(rg1.lo, s0);
            rg1.hi = min(rg1.hi, s1);
        }
    }
    const int kvh = head0 / p.G;
    // the CTA streams the union of its tiles' KV ranges
    const bool e0 = rg0.hi <= rg0.lo, e1 = rg1.hi <= rg1.lo;
    const int jlo = e0 ? rg1.lo : (e1 ? rg0.lo : min(rg0.lo, rg1.lo));
    const int jhi = e0 ? rg1.hi : (e1 ? rg0.hi : max(rg0.hi, rg1.hi));
    const int n = (e0 && e1) ? 0 : jhi - jlo;

    if (threadIdx.x == 0) {
        mbar_init(&sm.bar_q, 1);
        for (int i = 0; i < NS; ++i) {
            mbar_init(&sm.kv_full[i], 1);
            mbar_init(&sm.kv_empty[i], 1);
        }
        for (int t = 0; t < NT; ++t) {
            mbar_init(&sm.s_full[t], 1);
            mbar_init(&sm.p_full[t], 4);
            mbar_init(&sm.o_done[t], 1);
        }
        mbar_init(&sm.mma_fin, 1);
        sm.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&sm.tmem_base, Cfg::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = sm.tmem_base;
    volatile int* abort = &sm.abort;
    const unsigned long long wlim = p.wait_ns ? p.wait_ns : kWaitLimitNs;
    int issued = 0;   // ring entries issued (producer thread)
    // failure-detection self-test: the first CTA's producer stops before this
    // ring entry, so the MMA warp's wait on it must run out and the CTA must
    // wind down
    const int skip = (p.selftest_skip > 0 && blockIdx.x == 0 && blockIdx.y == 0 &&
                      blockIdx.z == 0) ? p.selftest_skip - 1 : -1;

    if (warp < kSoftmaxWarp0) {
      // control warps: TMA producer (warp 0) and MMA issuer (warp 1)
      if constexpr (NT == 2)
          asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(regs_ctl<D, EXTRA>()));
      if (warp == 0) {
        // ============================================== TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            mbar_arrive_expect_tx(&sm.bar_q, uint32_t(NT) * Cfg::kBoxes * kTileBytes);
#pragma unroll
            for (int bx = 0; bx < Cfg::kBoxes; ++bx) {
                tma_load_3d(sm.q[0][bx], &tmQ, &sm.bar_q, bx * 64, row00, b * p.Hq + head0);
                if constexpr (NT == 2)
                    tma_load_3d(sm.q[NT - 1][bx], &tmQ, &sm.bar_q, bx * 64, row01,
                                b * p.Hq + head1);
            }
            const int z = b * p.Hkv + kvh;
            // ring order = consumption order: K_0, V_0, K_1, V_1, ...
            for (int u = 0; u < 2 * n; ++u) {
                const int slot = u % NS;
                if (u >= NS &&
                    !mbar_wait_limit(&sm.kv_empty[slot], ((u / NS) - 1) & 1, abort, p.status, wlim))
                    break;
                if (u == skip) break;   // self-test: this entry and the rest never come
                mbar_arrive_expect_tx(&sm.kv_full[slot], Cfg::kSlotBytes);
                const CUtensorMap* map = (u & 1) ? &tmV : &tmK;
#pragma unroll
                for (int bx = 0; bx < Cfg::kBoxes; ++bx)
                    tma_load_3d(sm.kv[slot][bx], map, &sm.kv_full[slot], bx * 64,
                                (REV ? jhi - 1 - (u >> 1) : jlo + (u >> 1)) * 128, z);
                issued = u + 1;
            }
        }
    } else if (warp == 1) {
        // ============================================== MMA issuer
        // The whole warp runs the loop; one elected lane issues. A wait that
        // fails (time limit, or another warp's abort) does not end a lane's
        // loop on its own: the lane marks itself bad and keeps step with the
        // others for the rest of the KV step (the products it helps issue
        // then read stale tiles, which is harmless), so every lane reaches
        // every elect.sync. At the next step boundary a vote sees any bad
        // lane and the warp leaves the loop as a whole. The vote sits where
        // the warp would wait for the softmax anyway, off the issue path.
        {
            constexpr uint32_t idS = tc::idesc_bf16(128, 128, 0);
            constexpr uint32_t idO = tc::idesc_bf16(128, D, 1);
            bool bad = !mbar_wait_limit(&sm.bar_q, 0, abort, p.status, wlim);
            tc::fence_after_sync();
            int u = 0;   // next ring entry to consume
            auto acquire = [&]() {
                const int slot = u % NS;
                bad |= !mbar_wait_limit(&sm.kv_full[slot], (u / NS) & 1, abort, p.status, wlim);
                tc::fence_after_sync();
                return slot;
            };
            auto release = [&](int slot) {
                tc::commit_warp(&sm.kv_empty[slot]);
                ++u;
            };
            // Descriptors are built once; a K-step or ring slot only moves the
            // start-address field (16-byte units, 14 bits: every shared
            // address here is below 256 KB, so the field cannot overflow).
            const uint64_t qdesc0 = tc::sdesc_sw128(smem_u32(sm.q[0][0]), 16, 1024);
            const uint64_t qdesc1 = tc::sdesc_sw128(smem_u32(sm.q[NT - 1][0]), 16, 1024);
            const uint64_t kdesc0 = tc::sdesc_sw128(smem_u32(sm.kv[0][0]), 16, 1024);
            const uint64_t vdesc0 = tc::sdesc_sw128(smem_u32(sm.kv[0][0]), kTileBytes, 1024);
            constexpr uint32_t kSlotStep = Cfg::kSlotBytes >> 4;
            auto issue_s = [&](int t, int slot) {
                const uint64_t a0 = t ? qdesc1 : qdesc0;
                const uint64_t b0 = kdesc0 + uint64_t(uint32_t(slot) * kSlotStep);
                const uint32_t d = tbase + t * 128;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t o = ((kk >> 2) * kTileBytes + (kk & 3) * 32) >> 4;
                    tc::mma_bf16_ss_warp(d, a0 + o, b0 + o, idS, kk > 0);
                }
            };
            auto issue_pv = [&](int t, int slot, bool first) {
                const uint64_t b0 = vdesc0 + uint64_t(uint32_t(slot) * kSlotStep);
                const uint32_t tP = tbase + t * 128 + 64;
                const uint32_t d = tbase + Cfg::kOCol + t * D;
                const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_bf16_ts_warp(d, tP + kk * 8, b0 + uint32_t(kk * (2048 >> 4)), idO,
                                    kk > 0 ? 1u : acc0);
            };
            const KvRange rg[2] = {rg0, rg1};
            int pf[2] = {0, 0};   // softmax steps consumed per tile (p_full phases)
            if (!__any_sync(0xffffffffu, bad) && n > 0) {
                const int ks = acquire();           // K of the first tile scanned
                for (int t = 0; t < NT; ++t)
                    if ((REV ? rg[t].hi == jhi : rg[t].lo == jlo) && rg[t].hi > rg[t].lo) {
                        issue_s(t, ks);
                        tc::commit_warp(&sm.s_full[t]);
                    }
                release(ks);
            }
            for (int jj = 0; jj < n; ++jj) {
                if (__any_sync(0xffffffffu, bad)) break;   // the warp leaves as a whole
                const int j = REV ? jhi - 1 - jj : jlo + jj;
                const int jn = REV ? j - 1 : j + 1;  // the tile scanned next
                const int vs = acquire();           // V_j
                int ks = -1;
                auto get_k = [&]() {                // K_jn follows V_j in the ring
                    if (ks < 0) {
                        ++u;
                        ks = acquire();
                        --u;
                    }
                };
                for (int t = 0; t < NT; ++t) {
                    const bool active = j >= rg[t].lo && j < rg[t].hi;
                    if (active) {
                        bad |= !mbar_wait_limit(&sm.p_full[t], pf[t] & 1, abort, p.status, wlim);
                        ++pf[t];
                        tc::fence_after_sync();
                        issue_pv(t, vs, j == (REV ? rg[t].hi - 1 : rg[t].lo));
                    }
                    const bool next_s = (active && jn >= rg[t].lo && jn < rg[t].hi) ||
                                        (jn == (REV ? rg[t].hi - 1 : rg[t].lo) &&
                                         rg[t].hi > rg[t].lo);
                    if (next_s) {
                        get_k();
                        issue_s(t, ks);
                        tc::commit_warp(&sm.s_full[t]);
                    } else if (active) {
                        tc::commit_warp(&sm.o_done[t]);
                    }
                }
                release(vs);
                if (jj + 1 < n) {
                    // every tile that needs K_jn has consumed it by now
                    get_k();
                    release(ks);
                }
            }
            // every MMA this thread issued completes before the CTA ends
            tc::commit_warp(&sm.mma_fin);
            volatile int never = 0;
            mbar_wait_limit(&sm.mma_fin, 0, &never, p.status, wlim);
        }
      }
    } else {
        if constexpr (NT == 2)
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ============================================== softmax groups
        const int t = NT == 2 ? (warp - kSoftmaxWarp0) >> 2 : 0;
        const int q4 = warp & 3;                  // TMEM lane quadrant of this warp
        const int r = q4 * 32 + lane;             // row within the tile
        const int head = t ? head1 : head0;
        const int row0 = t ? row01 : row00;
        const KvRange rgt = t ? rg1 : rg0;
        const int ntile = rgt.hi > rgt.lo ? rgt.hi - rgt.lo : 0;
        const int row = row0 + r;
        const int i_al = row + off;               // bottom-right aligned row index
        const uint32_t lane_off = uint32_t(q4 * 32) << 16;
        const uint32_t tS = tbase + t * 128 + lane_off;
        const uint32_t tP = tS + 64;
        const uint32_t tO = tbase + Cfg::kOCol + t * D + lane_off;
        const float sl2 = p.scale_log2;
        // softcap in the natural-log domain: score / cap, then * cap * log2(e)
        const float sc_div = CAPPED ? (sl2 / kLog2e) / p.softcap : 0.f;
        const float cap_l2 = CAPPED ? p.softcap * kLog2e : 0.f;
        const float slope_l2 = ALIBI ? p.slopes[head] * kLog2e : 0.f;

        float m = -INFINITY;   // reference max (log2 domain)
        float l = 0.f;
        bool ok = true;
        for (int jt = 0; jt < ntile; ++jt) {
            const int j = REV ? rgt.hi - 1 - jt : rgt.lo + jt;
            // warp-uniform wait: the TMEM load below is warp-collective
            ok = mbar_wait_warp_limit(&sm.s_full[t], jt & 1, abort, p.status, wlim);
            if (!ok) break;
            tc::fence_after_sync();
            float s[128];
            {
                uint32_t rr[128];
                tc::tmem_ld_32x32b_x128(tS, rr);
#pragma unroll
                for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(rr[i]);
            }
            const int k0 = j * 128;
            // aligned index of this warp's first row: the warp's 32 rows need
            // per-key masks only on tiles that cross the key length, the
            // causal diagonal or a window edge (warp-uniform)
            const int w_al = row0 + q4 * 32 + off;
            bool need_mask = (k0 + 128 > p.Lk) || (CAUSAL && k0 + 127 > w_al);
            if (EXTRA) {
                if (p.window_left >= 0 && k0 < w_al + 31 - p.window_left) need_mask = true;
                if (p.window_right >= 0 && k0 + 127 > w_al + p.window_right) need_mask = true;
            }
            constexpr bool cap = CAPPED;
            // x = s * scale (log2 domain) + bias, masked; without bias or
            // cap the scale is folded into the exp's FMA below (masked keys
            // hold -inf, which the positive scale keeps)
            const bool fast = !ALIBI && !cap && sl2 > 0.f;
            // the part of every score of this tile that is left out of s[]
            // and carried in the reference max instead (ALiBi row offset)
            float rel = 0.f;
            // causal ALiBi tile whose maximum provably cannot move the
            // reference: the bias is applied in the exponential pass instead
            bool lazy = false;
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (fast && !need_mask) {
#pragma unroll
                for (int c = 0; c < 128; c += 8) {
                    mx4[0] = max3(mx4[0], s[c], s[c + 1]);
                    mx4[1] = max3(mx4[1], s[c + 2], s[c + 3]);
                    mx4[2] = max3(mx4[2], s[c + 4], s[c + 5]);
                    mx4[3] = max3(mx4[3], s[c + 6], s[c + 7]);
                }
            } else if (fast) {
                // masked tile without bias or cap: this row's visible keys
                // are one interval [klo, khi] (key length, causal, window);
                // the raw scores outside it become -inf
                int khi = p.Lk - 1;
                if (CAUSAL) khi = min(khi, i_al);
                int klo = 0;
                if (EXTRA) {
                    if (p.window_left >= 0) klo = max(klo, i_al - p.window_left);
                    if (p.window_right >= 0) khi = min(khi, i_al + p.window_right);
                }
                const int clo = klo - k0, chi = khi - k0;
#pragma unroll
                for (int c = 0; c < 128; c += 2) {
                    if (c < clo || c > chi) s[c] = -INFINITY;
                    if (c + 1 < clo || c + 1 > chi) s[c + 1] = -INFINITY;
                    mx4[(c >> 1) & 3] = max3(mx4[(c >> 1) & 3], s[c], s[c + 1]);
                }
            } else if (ALIBI && CAUSAL && need_mask && !cap && !EXTRA) {
                // a causal ALiBi tile that crosses the diagonal or the key
                // length: the unmasked form below plus one interval test per
                // key (this row sees keys k0 .. k0 + chi of the tile)
                const int chi = min(p.Lk - 1, i_al) - k0;
                const uint64_t sc2 = f2_pack(sl2, sl2);
                const uint64_t step2 = f2_pack(8.f * slope_l2, 8.f * slope_l2);
                uint64_t o2[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    o2[q] = f2_pack(slope_l2 * float(2 * q), slope_l2 * float(2 * q + 1));
#pragma unroll
                for (int c = 0; c < 128; c += 2) {
                    const int q = (c >> 1) & 3;
                    f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sc2, o2[q]), s[c], s[c + 1]);
                    o2[q] = f2_add(o2[q], step2);
                    if (c > chi) s[c] = -INFINITY;
                    if (c + 1 > chi) s[c + 1] = -INFINITY;
                    mx4[q] = max3(mx4[q], s[c], s[c + 1]);
                }
                rel = slope_l2 * float(k0 - i_al);
            } else if (ALIBI && CAUSAL && !need_mask && !cap) {
                // Bound first: every score of the tile is at most max(s) *
                // scale + slope * 127 + slope * (k0 - i'). Scanned diagonal-
                // first, the tiles after the first sit far enough below the
                // reference that this bound already rules out a repair; then
                // the exact maximum is not needed (the kept reference stays
                // exact for O and l alike). Two-tile form only: in the one-tile
                // form (168 registers) it spilled and measured slower.
                if constexpr (NT == 2) {
#pragma unroll
                    for (int c = 0; c < 128; c += 8) {
                        mx4[0] = max3(mx4[0], s[c], s[c + 1]);
                        mx4[1] = max3(mx4[1], s[c + 2], s[c + 3]);
                        mx4[2] = max3(mx4[2], s[c + 4], s[c + 5]);
                        mx4[3] = max3(mx4[3], s[c + 6], s[c + 7]);
                    }
                    const float smax = max3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
                    const float bound = smax * sl2 + slope_l2 * float(k0 + 127 - i_al);
                    lazy = __all_sync(0xffffffffu, sl2 > 0.f && m != -INFINITY &&
                                                       bound <= m + kRescaleThreshold);
#pragma unroll
                    for (int q = 0; q < 4; ++q) mx4[q] = -INFINITY;
                }
                if (!lazy) {
                    // every key of this tile is at or before every row of the
                    // warp: bias = slope * (key - i') = slope * c + b0 with
                    // b0 = slope * (k0 - i'). The row part b0 moves into the
                    // reference max: y = s * scale + slope * c here, and the
                    // exponent below is y - (m - b0), the same value as x - m
                    // with x = y + b0. The column offsets slope * c come from
                    // four packed chains that step 8 columns per add (one add
                    // per key pair; 15 adds of rounding, < 2e-4 in log2 units).
                    const uint64_t sc2 = f2_pack(sl2, sl2);
                    const uint64_t step2 = f2_pack(8.f * slope_l2, 8.f * slope_l2);
                    uint64_t o2[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        o2[q] = f2_pack(slope_l2 * float(2 * q), slope_l2 * float(2 * q + 1));
#pragma unroll
                    for (int c = 0; c < 128; c += 2) {
                        const int q = (c >> 1) & 3;
                        f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sc2, o2[q]), s[c], s[c + 1]);
                        o2[q] = f2_add(o2[q], step2);
                        mx4[q] = max3(mx4[q], s[c], s[c + 1]);
                    }
                }
                rel = slope_l2 * float(k0 - i_al);
            } else if (cap && !need_mask && !ALIBI) {
                // unmasked tile with the cap: x = cap * tanh(y), y = score / cap.
                // When every |y| of the warp's rows is at most 1/2, tanh is an
                // odd polynomial of degree 9 on the FMA pipe in packed pairs: a
                // near-minimax fit on [0, 1/2] (Lawson-reweighted least
                // squares, absolute error 4.3e-9, against 3.9e-6 for the
                // Taylor series through y^9; degree 7 measured slower here).
                // Otherwise the exponential form of the general path below (two
                // special-function operations per score).
                float amax = 0.f;
#pragma unroll
                for (int c = 0; c < 128; c += 2) amax = max3(amax, fabsf(s[c]), fabsf(s[c + 1]));
                if (__all_sync(0xffffffffu, amax * fabsf(sc_div) <= kTanhRange)) {
                    // x = s * Q(s^2) with the scalings folded into Q's
                    // coefficients: x = k y (1 + a3 y^2 + ...), y = u s, so
                    // Q(w) = k u (1 + a3 u^2 w + a5 u^4 w^2 + ...), w = s^2
                    const float u2 = sc_div * sc_div;
                    const float k1 = sc_div * cap_l2;
                    const float k3 = k1 * kTanhA3 * u2;
                    const float k5 = k1 * kTanhA5 * u2 * u2;
                    const uint64_t q5 = f2_pack(k5, k5), q3 = f2_pack(k3, k3);
                    const uint64_t q1 = f2_pack(k1, k1);
#pragma unroll
                    for (int c = 0; c < 128; c += 2) {
                        const uint64_t s2 = f2_pack(s[c], s[c + 1]);
                        const uint64_t w2 = f2_mul(s2, s2);
                        uint64_t q2 = f2_fma(q5, w2, q3);
                        q2 = f2_fma(q2, w2, q1);
                        f2_unpack(f2_mul(s2, q2), s[c], s[c + 1]);
                        mx4[(c >> 1) & 3] = max3(mx4[(c >> 1) & 3], s[c], s[c + 1]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 128; c += 2) {
                        const float y0 = fminf(fmaxf(s[c] * sc_div, -15.f), 15.f);
                        const float y1 = fminf(fmaxf(s[c + 1] * sc_div, -15.f), 15.f);
                        const float e0 = ex2(y0 * (2.f * kLog2e));
                        const float e1 = ex2(y1 * (2.f * kLog2e));
                        s[c] = cap_l2 * ((e0 - 1.f) * rcp_approx(e0 + 1.f));
                        s[c + 1] = cap_l2 * ((e1 - 1.f) * rcp_approx(e1 + 1.f));
                        mx4[(c >> 1) & 3] = max3(mx4[(c >> 1) & 3], s[c], s[c + 1]);
                    }
                }
            } else {
                // general tile: this row's visible keys form one interval
                // [klo, khi] (key length, causal, window), computed once per
                // tile; per key only the transform, the bias and one range test
                int khi = p.Lk - 1;
                if (CAUSAL) khi = min(khi, i_al);
                int klo = 0;
                if (EXTRA) {
                    if (p.window_left >= 0) klo = max(klo, i_al - p.window_left);
                    if (p.window_right >= 0) khi = min(khi, i_al + p.window_right);
                }
                const int clo = klo - k0, chi = khi - k0;
                if (cap) {
#pragma unroll
                    for (int c = 0; c < 128; ++c) {
                        // cap * tanh(score / cap), tanh(y) = (e - 1) / (e + 1)
                        // with e = 2^(2 y log2 e); |y| <= 15 keeps e finite
                        // and tanh(15) rounds to 1 in fp32
                        const float y = fminf(fmaxf(s[c] * sc_div, -15.f), 15.f);
                        const float e = ex2(y * (2.f * kLog2e));
                        float x = cap_l2 * ((e - 1.f) * rcp_approx(e + 1.f));
                        if (ALIBI) {
                            const float dist = float(i_al - (k0 + c));
                            x -= slope_l2 * (CAUSAL ? dist : fabsf(dist));
                        }
                        if (c < clo || c > chi) x = -INFINITY;
                        s[c] = x;
                        mx4[c & 3] = fmaxf(mx4[c & 3], x);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 128; ++c) {
                        float x = s[c] * sl2;
                        if (ALIBI) {
                            const float dist = float(i_al - (k0 + c));
                            x -= slope_l2 * (CAUSAL ? dist : fabsf(dist));
                        }
                        if (c < clo || c > chi) x = -INFINITY;
                        s[c] = x;
                        mx4[c & 3] = fmaxf(mx4[c & 3], x);
                    }
                }
            }
            float mx = max3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
            if (fast) mx *= sl2;
            mx += rel;
            // conditional repair: move the reference max only when the row max
            // exceeds it by more than the threshold (or it is still unset)
            float m_new = m;
            if (mx > m + kRescaleThreshold || (m == -INFINITY && mx != -INFINITY)) m_new = mx;
            const bool rescale = (jt > 0) && (m != -INFINITY) && (m_new != m);
            const float corr = rescale ? ex2(m - m_new) : 1.f;
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            // p = 2^(x - m) as one packed FMA per key pair (x = s * scale on
            // the fast path; s already holds x otherwise, times exactly 1),
            // row sum with packed adds, and P_t (bf16) over the upper half of
            // S_t in tensor memory, 64 keys at a time (S_t is in registers)
            const float mul = fast ? sl2 : 1.f;
            const uint64_t mul2 = f2_pack(mul, mul);
            const uint64_t neg2 = f2_pack(rel - m_use, rel - m_use);
            uint64_t sum2[2] = {0ull, 0ull};
            // the one-tile form runs at 168 registers: P goes out in quarters
            // so fewer packed values are live beside S
            constexpr int kPW = NT == 2 ? 32 : 16;   // packed columns per store
            if (ALIBI && NT == 2 && lazy) {
                // x - m = s * scale + slope * c + slope * (k0 - i') - m, the
                // column and row parts from four packed chains started at
                // slope * (k0 - i') - m
                const uint64_t sc2 = f2_pack(sl2, sl2);
                const uint64_t step2 = f2_pack(8.f * slope_l2, 8.f * slope_l2);
                const float b0 = slope_l2 * float(k0 - i_al) - m_use;
                uint64_t a2[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    a2[q] = f2_pack(fmaf(slope_l2, float(2 * q), b0),
                                    fmaf(slope_l2, float(2 * q + 1), b0));
#pragma unroll
                for (int h = 0; h < 64 / kPW; ++h) {
                    uint32_t pk[kPW];
#pragma unroll
                    for (int c2 = 0; c2 < kPW; ++c2) {
                        const int c = h * 2 * kPW + 2 * c2;
                        const int q = (c >> 1) & 3;
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sc2, a2[q]), x0, x1);
                        a2[q] = f2_add(a2[q], step2);
                        const float p0 = ex2(x0);
                        const float p1 = ex2(x1);
                        sum2[c2 & 1] = f2_add(sum2[c2 & 1], f2_pack(p0, p1));
                        pk[c2] = pack_bf16(p0, p1);
                    }
                    if constexpr (NT == 2)
                        tc::tmem_st_32x32b_x32(tP + h * kPW, pk);
                    else
                        tc::tmem_st_32x32b_x16(tP + h * kPW, pk);
                }
            } else {
#pragma unroll
                for (int h = 0; h < 64 / kPW; ++h) {
                    uint32_t pk[kPW];
#pragma unroll
                    for (int c2 = 0; c2 < kPW; ++c2) {
                        const int c = h * 2 * kPW + 2 * c2;
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), mul2, neg2), x0, x1);
                        const float p0 = ex2(x0);
                        const float p1 = ex2(x1);
                        sum2[c2 & 1] = f2_add(sum2[c2 & 1], f2_pack(p0, p1));
                        pk[c2] = pack_bf16(p0, p1);
                    }
                    if constexpr (NT == 2)
                        tc::tmem_st_32x32b_x32(tP + h * kPW, pk);
                    else
                        tc::tmem_st_32x32b_x16(tP + h * kPW, pk);
                }
            }
            float sa, sb, sc, sd;
            f2_unpack(sum2[0], sa, sb);
            f2_unpack(sum2[1], sc, sd);
            l = l * corr + ((sa + sb) + (sc + sd));
            m = m_new;
            // O_t holds step j-1's result (the commit that signalled S_t^j
            // covers the PV issued before it): repair it if the max moved
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t rr[32];
                    tc::tmem_ld_32x32b_x32(tO + c * 32, rr);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        rr[i] = __float_as_uint(__uint_as_float(rr[i]) * corr);
                    tc::tmem_st_32x32b_x32(tO + c * 32, rr);
                }
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.p_full[t]);
        }

        // ---------------------------------------------------- epilogue
        if (ok && ntile > 0) {
            ok = mbar_wait_warp_limit(&sm.o_done[t], 0, abort, p.status, wlim);
            tc::fence_after_sync();
        }
        bool stored = false;   // this lane committed a bulk store
        if (ok && !*abort) {
            const bool valid = row < p.Lq;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            // O_t goes out through this tile's Q buffer, free now (the commit
            // behind o_done covers every product that read Q_t): each warp
            // writes its 32 rows in the tensor map's 128-byte swizzled layout
            // and stores them with one bulk tensor copy per 64-column box;
            // rows past Lq fall outside the map and are not written. Used
            // where it measured faster: two-tile CTAs whose tiles are two
            // heads of one row block (they finish together), and the capped
            // forms; the staggered tiles of unpaired causal CTAs and the
            // one-tile form store rows straight to global memory (graph
            // replay, us: paired GQA + ALiBi 2k 40.0 against 41.7 and 4k
            // 125.9 against 129.1; one-tile cap 30 860 against 899; causal
            // MHA 4k 413 against 405 and one-tile GQA 1k 20.8 against 20.1
            // when staged, and 415 against 405 even unused: the staged code
            // is compiled into the capped and ALiBi variants only)
            constexpr bool kStageO = CAPPED || ALIBI;
            const bool staged = kStageO && p.splits <= 1 && (CAPPED || (NT == 2 && pair_heads));
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t rr[32];
                if (ntile > 0) {
                    tc::tmem_ld_32x32b_x32(tO + c * 32, rr);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) rr[i] = 0u;
                }
                if (staged) {
                    uint8_t* srow = sm.q[t][c >> 1] + r * 128;
#pragma unroll
                    for (int v8 = 0; v8 < 4; ++v8) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(rr[v8 * 8 + 0]) * inv,
                                        __uint_as_float(rr[v8 * 8 + 1]) * inv);
                        w.y = pack_bf16(__uint_as_float(rr[v8 * 8 + 2]) * inv,
                                        __uint_as_float(rr[v8 * 8 + 3]) * inv);
                        w.z = pack_bf16(__uint_as_float(rr[v8 * 8 + 4]) * inv,
                                        __uint_as_float(rr[v8 * 8 + 5]) * inv);
                        w.w = pack_bf16(__uint_as_float(rr[v8 * 8 + 6]) * inv,
                                        __uint_as_float(rr[v8 * 8 + 7]) * inv);
                        const int chunk = (c & 1) * 4 + v8;   // 16-byte chunk of the 128-byte row
                        *reinterpret_cast<uint4*>(srow + ((chunk ^ (r & 7)) << 4)) = w;
                    }
                } else if (valid && p.splits <= 1) {
                    __nv_bfloat16* orow = p.O + ((size_t(b) * p.Hq + head) * p.Lq + row) * D;
#pragma unroll
                    for (int v8 = 0; v8 < 4; ++v8) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(rr[v8 * 8 + 0]) * inv,
                                        __uint_as_float(rr[v8 * 8 + 1]) * inv);
                        w.y = pack_bf16(__uint_as_float(rr[v8 * 8 + 2]) * inv,
                                        __uint_as_float(rr[v8 * 8 + 3]) * inv);
                        w.z = pack_bf16(__uint_as_float(rr[v8 * 8 + 4]) * inv,
                                        __uint_as_float(rr[v8 * 8 + 5]) * inv);
                        w.w = pack_bf16(__uint_as_float(rr[v8 * 8 + 6]) * inv,
                                        __uint_as_float(rr[v8 * 8 + 7]) * inv);
                        *reinterpret_cast<uint4*>(orow + c * 32 + v8 * 8) = w;
                    }
                } else if (valid) {
                    // split-KV partial: O / l in fp32, [B, Hq, Lq, splits, D]
                    float* prow = p.O_part +
                                  ((((size_t(b) * p.Hq + head) * p.Lq + row) * p.splits) +
                                   blockIdx.z) * D + c * 32;
#pragma unroll
                    for (int v4 = 0; v4 < 8; ++v4)
                        *reinterpret_cast<float4*>(prow + v4 * 4) =
                            make_float4(__uint_as_float(rr[v4 * 4 + 0]) * inv,
                                        __uint_as_float(rr[v4 * 4 + 1]) * inv,
                                        __uint_as_float(rr[v4 * 4 + 2]) * inv,
                                        __uint_as_float(rr[v4 * 4 + 3]) * inv);
                }
            }
            if (staged) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
#pragma unroll
                    for (int bx = 0; bx < D / 64; ++bx)
                        tma_store_3d(&tmO, sm.q[t][bx] + q4 * 32 * 128, bx * 64,
                                     row0 + q4 * 32, b * p.Hq + head);
                    bulk_commit_group();
                    stored = true;
                }
            }
            const float lse_row = l > 0.f ? (m + lg2(l)) * kLn2 : -INFINITY;
            if (valid && p.splits > 1)
                p.LSE_part[((size_t(b) * p.Hq + head) * p.Lq + row) * p.splits + blockIdx.z] = lse_row;
            else if (valid && p.LSE)
                p.LSE[(size_t(b) * p.Hq + head) * p.Lq + row] = lse_row;
        }
        // the Q buffer stays allocated until the stores have read it
        if (stored) bulk_wait_read_all();
        tc::fence_before_sync();
    }

    __syncwarp();
    __syncthreads();
    if (warp == 0 && lane == 0 && *abort) {
        // let this CTA's copies in flight land before its shared memory is released
        volatile int never = 0;
        mbar_wait_limit(&sm.bar_q, 0, &never, p.status, wlim);
        for (int s = 0; s < NS; ++s) {
            int last = -1;
            for (int u = s; u < issued; u += NS) last = u;
            if (last >= 0) mbar_wait_limit(&sm.kv_full[s], (last / NS) & 1, &never, p.status, wlim);
        }
    }
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tbase, Cfg::kTmemCols);
    }
}

namespace {

template <int D, bool CAUSAL, bool ALIBI, int MODE, int NT>
int launch_tc_t(const PrefillLaunch& L, cudaStream_t stream) {
    const size_t smem = sizeof(TcSmem<D, NT>) + 1024;
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(prefill_tc_kernel<D, CAUSAL, ALIBI, MODE, NT>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem)) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set[dev] = true;
    }
    const bool pair = NT == 2 && L.p.pair_heads;
    const int rows_per_item = (NT == 1 || pair) ? 128 : 256;
    const int n_hb = pair ? L.p.Hq / 2 : L.p.Hq;
    const long long items = (long long)((L.p.Lq + rows_per_item - 1) / rows_per_item) * n_hb;
    if (items > 0x7fffffffLL) return ATTN_ERR_SHAPE;
    dim3 grid(unsigned(items), L.p.B, unsigned(L.p.splits > 1 ? L.p.splits : 1));
    prefill_tc_kernel<D, CAUSAL, ALIBI, MODE, NT>
        <<<grid, tc_threads<NT>(), smem, stream>>>(L.tmQ, L.tmK, L.tmV, L.tmO, L.p);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int D, int MODE, int NT>
int launch_tc_e(const PrefillLaunch& L, cudaStream_t stream) {
    const bool alibi = L.p.slopes != nullptr;
    if (L.p.causal)
        return alibi ? launch_tc_t<D, true, true, MODE, NT>(L, stream)
                     : launch_tc_t<D, true, false, MODE, NT>(L, stream);
    return alibi ? launch_tc_t<D, false, true, MODE, NT>(L, stream)
                 : launch_tc_t<D, false, false, MODE, NT>(L, stream);
}

template <int D, int NT>
int launch_tc_d(const PrefillLaunch& L, cudaStream_t stream) {
    if (L.p.softcap > 0.f) return launch_tc_e<D, 2, NT>(L, stream);
    const bool window = L.p.window_left >= 0 || L.p.window_right >= 0;
    return window ? launch_tc_e<D, 1, NT>(L, stream) : launch_tc_e<D, 0, NT>(L, stream);
}

// Launches the form with NT Q tiles per CTA for head dim d.
template <int NT>
int launch_tc_nt(const PrefillLaunch& L, int d, cudaStream_t stream) {
    if (d == 64) return launch_tc_d<64, NT>(L, stream);
    if (d == 128) return launch_tc_d<128, NT>(L, stream);
    return ATTN_ERR_UNSUPPORTED;
}

}  // namespace

}  // namespace attn
