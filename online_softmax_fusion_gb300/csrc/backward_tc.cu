// Attention backward on the 5th-generation tensor cores (head dim 128).
//
// The single-pass algorithm of the Twill review (xllm-io) §七 7.2: each CTA
// owns one block of 128 keys, recomputes P from the forward's log-sum-exp,
// runs the five products and adds its share of dQ to a global fp32
// accumulator. With s the softmax scale and x = s q.k (+ bias):
//   P^T  = exp(x - LSE)                   dP^T = V dO^T
//   dS^T = P^T (dP^T - D),  D_i = dO_i . O_i
//   dV  += P^T dO          dK += dS^T Q    (scaled by s at the end)
//   dQ^T = K^T dS^T        (added to the accumulator, scaled by s later)
// Every product is 128 x 128 with M = 128: the key block (S^T, dP^T, dV, dK)
// or the head dimension (dQ, produced transposed). A step covers 128 query
// rows: a tcgen05 MMA of M = 128 costs the same issue time for any N up to
// 128, so the full width halves the instruction count per FLOP against
// 64-row steps.
//
// CTA roles (512 threads):
//   warp 0      TMA: K, V once; per step the Q tile (128 rows) into a 3-slot
//               ring and the dO tile into a 2-slot ring, with LSE and D of the
//               128 rows beside them
//   warp 1      TMEM allocation; tcgen05.mma issue (one elected lane)
//   warps 4-11  two warpgroups, one thread per key (TMEM lane), each taking
//               64 of the step's 128 query columns: P^T from S^T, P^T (bf16)
//               back into TMEM for dV; dS^T from dP^T into shared memory
//               (bf16, over the step's dO tile once dV has read it) for dK
//               and dQ^T; at the end dK (warps 4-7) and dV (warps 8-11)
//   warps 12-15 the dQ drain: dQ^T (TMEM lane = head dimension) copied to
//               registers as soon as it is complete, which frees its columns,
//               then added to the fp32 accumulator with global reductions
//               while the next step runs (the reductions are bound by the L2,
//               so they need their own warps to overlap everything else)
// Tensor memory (512 columns): S^T (128; P^T bf16 is written over S^T
// columns its group has read), dP^T (128, reused by dQ^T once dS^T is
// formed), dV (128), dK (128). Shared memory (227 KB): K and V resident
// (128-byte swizzle), 3 Q slots, 2 dO slots. The Q ring is one deeper than
// the dO ring because S_{i+1} is issued early in step i, while dP_{i+1} comes
// at its end: both loads get about one step of lead over the L2 traffic of
// the reductions.
//
// Issue order of the tensor core per step i:
//   (P_i) dV_i, S_{i+1} | (dS_i) dK_i, dQ^T_i | (dQ^T_i copied out) dP_{i+1}
// The parenthesised names are the hand-offs each group waits for. S_{i+1}
// goes in ahead of dK_i and dQ^T_i so that the P/dS warps can form P_{i+1}
// directly after dS_i.
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace attn {

namespace {

constexpr int kBtThreads = 512;               // 4 warpgroups
// Register split (setmaxnreg, per warpgroup) of the 128 x 512 = 65536 launch
// registers: control 104 x 128, two P/dS groups 128 x 256, drain 152 x 128
// (65536 in all).
constexpr int kRegsCtl = 104;
constexpr int kRegsSoftmax = 128;
constexpr int kRegsDrain = 152;
static_assert(kRegsCtl * 128 + kRegsSoftmax * 256 + kRegsDrain * 128 <= 65536,
              "register split exceeds the launch budget");
constexpr int kBtKeys = 128;                  // keys per CTA
constexpr int kBtRows = 128;                  // query rows per step
constexpr int kQStages = 3;                   // Q ring slots
constexpr int kOStages = 2;                   // dO ring slots (dS^T reuses them)
constexpr uint32_t kKVBox = 128 * 128;        // 128 keys x 64 dims (bf16, 128 B rows)
constexpr uint32_t kQBox = 128 * 128;         // 128 rows x 64 dims
// TMEM columns
constexpr uint32_t kColS = 0;
constexpr uint32_t kColDP = 128;              // dP^T, then dQ^T of the same step
constexpr uint32_t kColDV = 256;
constexpr uint32_t kColDK = 384;

struct BtSmem {
    alignas(1024) uint8_t k[2][kKVBox];                     // K block, dims 0-63 / 64-127
    alignas(1024) uint8_t v[2][kKVBox];
    alignas(1024) uint8_t q[kQStages][2][kQBox];            // Q tiles (2 boxes each)
    // dO tiles; once dV of the step has read one, its two boxes hold dS^T
    // [key][queries 0-63 | 64-127] (bf16, swizzled)
    alignas(1024) uint8_t dout[kOStages][2][kQBox];
    float lse2[kQStages][kBtRows];                          // LSE * log2(e); +inf = no weight
    float dsum[kOStages][kBtRows];                          // D_i
    uint64_t kv_full;
    uint64_t qfull[kQStages];
    uint64_t qempty[kQStages];
    uint64_t ofull[kOStages];
    uint64_t oempty[kOStages];
    uint64_t s_full;
    uint64_t dp_full;
    uint64_t p_full;
    uint64_t dv_done;
    uint64_t ds_full;
    uint64_t dq_full;
    uint64_t dq_free;
    uint64_t acc_done;
    uint32_t tmem_base;
    int abort;
};
// The layout fills shared memory to within a few hundred bytes, so it is
// used from the 1024-aligned start of the dynamic region without padding.
static_assert(sizeof(BtSmem) <= 232448, "backward tile layout exceeds shared memory");

// Stores 32 lanes x 16 consecutive 32-bit columns (no wait).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :
        : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
          "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
          "r"(r[14]), "r"(r[15])
        : "memory");
}

}  // namespace

template <bool CAUSAL, bool ALIBI>
__global__ void __launch_bounds__(kBtThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  BwdParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 128-byte swizzle needs 1024-aligned tiles and the layout has no
    // room for padding: a misaligned dynamic region is an error, not a hang
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) record_status(p.status, ATTN_ERR_ALIGN);
        return;
    }
    BtSmem& sm = *reinterpret_cast<BtSmem*>(smem_raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work item: key block, KV head, batch (key blocks of a head
    //      consecutive, heaviest first, so concurrent CTAs share dQ rows)
    const int nkb = (p.Lk + kBtKeys - 1) / kBtKeys;
    const int kb = int(blockIdx.x) % nkb;
    const int kvh = (int(blockIdx.x) / nkb) % p.Hkv;
    const int b = int(blockIdx.x) / (nkb * p.Hkv);
    const int k0 = kb * kBtKeys;
    const int off = p.Lk - p.Lq;
    const int n_qb = (p.Lq + kBtRows - 1) / kBtRows;
    const int qb0 = CAUSAL ? min(n_qb, max(0, k0 - off) / kBtRows) : 0;
    const int nq = n_qb - qb0;                    // Q blocks per query head
    const int n = nq * p.G;                       // steps
    auto step_rows = [&](int i, int& h, int& q0) {
        h = kvh * p.G + i / nq;
        q0 = (qb0 + i % nq) * kBtRows;
    };

    if (threadIdx.x == 0) {
        mbar_init(&sm.kv_full, 1);
        // a slot is full once its TMA bytes have landed and its row values
        // (LSE or D) have been written: two arrivals
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(&sm.qfull[s], 2);
            mbar_init(&sm.qempty[s], 1);
        }
        for (int s = 0; s < kOStages; ++s) {
            mbar_init(&sm.ofull[s], 2);
            mbar_init(&sm.oempty[s], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.dp_full, 1);
        mbar_init(&sm.p_full, 8);
        mbar_init(&sm.dv_done, 1);
        mbar_init(&sm.ds_full, 8);
        mbar_init(&sm.dq_full, 1);
        mbar_init(&sm.dq_free, 4);
        mbar_init(&sm.acc_done, 1);
        sm.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&sm.tmem_base, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = sm.tmem_base;
    volatile int* abort = &sm.abort;
    int issued_q = 0, issued_o = 0;   // steps whose Q / dO loads were issued (producer, lane 0)

    if (warp < 4) {
        // control warpgroup: TMA producer (warp 0) and MMA issuer (warp 1)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
        if (warp == 0) {
            // ================================================== TMA producer
            if (lane == 0) {
                tma_prefetch_desc(&tmQ);
                tma_prefetch_desc(&tmK);
                tma_prefetch_desc(&tmV);
                tma_prefetch_desc(&tmdO);
                mbar_arrive_expect_tx(&sm.kv_full, 4 * kKVBox);
                const int zkv = b * p.Hkv + kvh;
                for (int bx = 0; bx < 2; ++bx) {
                    tma_load_3d(sm.k[bx], &tmK, &sm.kv_full, bx * 64, k0, zkv);
                    tma_load_3d(sm.v[bx], &tmV, &sm.kv_full, bx * 64, k0, zkv);
                }
            }
            // Q_j then dO_j; Q has one slot more than dO so that S_{j+1}
            // (issued early in step j) finds its tile loaded
            for (int j = 0; j < n; ++j) {
                const int qs = j % kQStages, os = j % kOStages;
                int h, q0;
                step_rows(j, h, q0);
                const int z = b * p.Hq + h;
                bool ok = true;
                if (j >= kQStages)
                    ok = mbar_wait(&sm.qempty[qs], ((j / kQStages) - 1) & 1, abort, p.status);
                if (__any_sync(0xffffffffu, !ok)) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sm.qfull[qs], 2 * kQBox);
                    for (int bx = 0; bx < 2; ++bx)
                        tma_load_3d(sm.q[qs][bx], &tmQ, &sm.qfull[qs], bx * 64, q0, z);
                    issued_q = j + 1;
                }
                if (j >= kOStages)
                    ok = mbar_wait(&sm.oempty[os], ((j / kOStages) - 1) & 1, abort, p.status);
                if (__any_sync(0xffffffffu, !ok)) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sm.ofull[os], 2 * kQBox);
                    for (int bx = 0; bx < 2; ++bx)
                        tma_load_3d(sm.dout[os][bx], &tmdO, &sm.ofull[os], bx * 64, q0, z);
                    issued_o = j + 1;
                }
            }
        } else if (warp >= 2) {
            // ============================================== row values
            // warp 2: LSE * log2(e) of each step's rows (+inf where a row has
            // no weight) beside the Q ring; warp 3: D beside the dO ring. Each
            // runs ahead through its ring on its own, so the latency of these
            // loads overlaps the tile copies instead of adding to them.
            const bool lse_side = warp == 2;
            const int stages = lse_side ? kQStages : kOStages;
            for (int j = 0; j < n; ++j) {
                const int st = j % stages;
                bool ok = true;
                if (j >= stages)
                    ok = mbar_wait(lse_side ? &sm.qempty[st] : &sm.oempty[st],
                                   ((j / stages) - 1) & 1, abort, p.status);
                if (__any_sync(0xffffffffu, !ok)) break;
                int h, q0;
                step_rows(j, h, q0);
                const size_t rb = (size_t(b) * p.Hq + h) * p.Lq;
                const float* src = lse_side ? p.LSE : p.Dsum;
                float val[kBtRows / 32];
#pragma unroll
                for (int u = 0; u < kBtRows / 32; ++u) {
                    const int row = q0 + lane + 32 * u;
                    val[u] = row < p.Lq ? src[rb + row] : (lse_side ? -INFINITY : 0.f);
                }
                float* dst = lse_side ? sm.lse2[st] : sm.dsum[st];
#pragma unroll
                for (int u = 0; u < kBtRows / 32; ++u)
                    dst[lane + 32 * u] =
                        lse_side ? (val[u] == -INFINITY ? INFINITY : val[u] * kLog2e) : val[u];
                __syncwarp();
                if (lane == 0) mbar_arrive(lse_side ? &sm.qfull[st] : &sm.ofull[st]);
            }
        } else if (warp == 1) {
            // ============================================== MMA issuer
            // (the whole warp runs the loop; one elected lane issues)
            constexpr uint32_t idS = tc::idesc_bf16_ab(128, 128, 0, 0);    // S^T, dP^T
            constexpr uint32_t idD = tc::idesc_bf16_ab(128, 128, 0, 1);    // dV (A TMEM), dK
            constexpr uint32_t idQ = tc::idesc_bf16_ab(128, 128, 1, 1);    // dQ^T
            const uint64_t dk_ = tc::sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);          // K, K-major
            const uint64_t dv_ = tc::sdesc_sw128(smem_u32(sm.v[0]), 16, 1024);
            const uint64_t dkT = tc::sdesc_sw128(smem_u32(sm.k[0]), kKVBox, 1024);      // K^T, MN-major
            const uint64_t dq0 = tc::sdesc_sw128(smem_u32(sm.q[0][0]), 16, 1024);       // Q K-major
            const uint64_t dqm = tc::sdesc_sw128(smem_u32(sm.q[0][0]), kQBox, 1024);    // Q MN-major
            const uint64_t do0 = tc::sdesc_sw128(smem_u32(sm.dout[0][0]), 16, 1024);    // dO K-major
            const uint64_t dom = tc::sdesc_sw128(smem_u32(sm.dout[0][0]), kQBox, 1024); // dO MN-major
            // dS^T over the dO slot: K-major for dK, MN-major for dQ^T
            const uint64_t dsk = do0;
            const uint64_t dsm = dom;
            constexpr uint32_t kSlot = (2 * kQBox) >> 4;     // slot stride of both rings (16-byte units)
            // 16-wide K step kk inside a K-major operand of 64-element boxes
            auto kmaj = [](int kk, uint32_t box) -> uint32_t {
                return ((kk >> 2) * box + (kk & 3) * 32) >> 4;
            };
            // A x B^T over the 128 head dims (S^T = K Q^T, dP^T = V dO^T)
            auto issue_qk = [&](uint64_t a0, uint64_t b0, uint32_t d) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_bf16_ss_warp(d, a0 + kmaj(kk, kKVBox), b0 + kmaj(kk, kQBox), idS, kk > 0);
            };
            auto qslot = [](int i) -> uint32_t { return uint32_t(i % kQStages) * kSlot; };
            auto oslot = [](int i) -> uint32_t { return uint32_t(i % kOStages) * kSlot; };
            bool ok = mbar_wait_warp(&sm.kv_full, 0, abort, p.status);
            tc::fence_after_sync();
            if (ok && n > 0) {
                ok = mbar_wait_warp(&sm.qfull[0], 0, abort, p.status);
                tc::fence_after_sync();
                if (ok) {
                    issue_qk(dk_, dq0, tbase + kColS);
                    tc::commit_warp(&sm.s_full);
                }
                ok = ok && mbar_wait_warp(&sm.ofull[0], 0, abort, p.status);
                tc::fence_after_sync();
                if (ok) {
                    issue_qk(dv_, do0, tbase + kColDP);
                    tc::commit_warp(&sm.dp_full);
                }
            }
            for (int i = 0; ok && i < n; ++i) {
                const uint32_t sq = qslot(i), so = oslot(i);
                // dV += P^T dO (P^T bf16 in TMEM: queries 0-63 at columns
                // 0-31, queries 64-127 at columns 96-127)
                ok = mbar_wait_warp(&sm.p_full, i & 1, abort, p.status);
                if (!ok) break;
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_bf16_ts_warp(tbase + kColDV, tbase + kColS + (kk < 4 ? kk * 8 : 64 + kk * 8),
                                         dom + so + uint32_t(kk * (2048 >> 4)), idD,
                                         (i > 0 || kk > 0) ? 1u : 0u);
                tc::commit_warp(&sm.dv_done);
                // S^T_{i+1} right away (P^T_i in its columns is read by dV_i,
                // issued before it), so P_{i+1} can follow dS_i directly
                if (i + 1 < n) {
                    ok = mbar_wait_warp(&sm.qfull[(i + 1) % kQStages], ((i + 1) / kQStages) & 1,
                                        abort, p.status);
                    if (!ok) break;
                    tc::fence_after_sync();
                    issue_qk(dk_, dq0 + qslot(i + 1), tbase + kColS);
                    tc::commit_warp(&sm.s_full);
                }
                // dS^T of step i is in the slot (and dP^T_i has been read)
                ok = mbar_wait_warp(&sm.ds_full, i & 1, abort, p.status);
                if (!ok) break;
                tc::fence_after_sync();
                // dK += dS^T Q
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_bf16_ss_warp(tbase + kColDK, dsk + so + kmaj(kk, kQBox),
                                         dqm + sq + uint32_t(kk * (2048 >> 4)), idD,
                                         (i > 0 || kk > 0) ? 1u : 0u);
                // dQ^T = K^T dS^T into the dP^T columns
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_bf16_ss_warp(tbase + kColDP, dkT + uint32_t(kk * (2048 >> 4)),
                                         dsm + so + uint32_t(kk * (2048 >> 4)), idQ, kk > 0);
                tc::commit_warp(&sm.dq_full);
                tc::commit_warp(&sm.qempty[i % kQStages]);
                tc::commit_warp(&sm.oempty[i % kOStages]);
                // dP^T_{i+1} once the drain group has copied dQ^T_i out
                if (i + 1 < n) {
                    ok = mbar_wait_warp(&sm.dq_free, i & 1, abort, p.status);
                    ok = ok && mbar_wait_warp(&sm.ofull[(i + 1) % kOStages], ((i + 1) / kOStages) & 1,
                                              abort, p.status);
                    if (!ok) break;
                    tc::fence_after_sync();
                    issue_qk(dv_, do0 + oslot(i + 1), tbase + kColDP);
                    tc::commit_warp(&sm.dp_full);
                }
            }
            // covers every MMA issued above; the epilogue and TMEM release wait on it
            tc::commit_warp(&sm.acc_done);
        }

    } else if (warp < 12) {
        // (at the launch count, 128, there is nothing to raise)
        if constexpr (kRegsSoftmax > 128)
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ===================== P^T and dS^T (one key per thread)
        // Two warpgroups split the 128 query columns of a step: warps 4-7
        // take columns 0-63, warps 8-11 columns 64-127 (same TMEM lanes).
        const int half = warp >= 8 ? 1 : 0;
        const int co = half * 64;                     // first query column of this group
        const int q4 = warp & 3;
        const int kl = q4 * 32 + lane;                // key within the block (TMEM lane)
        const int key = k0 + kl;
        const bool key_ok = key < p.Lk;
        const uint32_t lane_off = uint32_t(q4 * 32) << 16;
        // P^T (bf16) of this group's 64 queries goes over S^T columns this
        // group has read and the other group never reads: columns 0-31
        // (group 0) and 96-127 (group 1)
        const uint32_t p_col = half ? 96u : 0u;
        bool ok = true;
        for (int i = 0; i < n; ++i) {
            const int qs = i % kQStages, os = i % kOStages;
            int h, q0;
            step_rows(i, h, q0);
            const float slope_l2 = ALIBI ? p.slopes[h] * kLog2e : 0.f;
            ok = mbar_wait_warp(&sm.s_full, i & 1, abort, p.status);
            ok = ok && mbar_wait_warp(&sm.qfull[qs], (i / kQStages) & 1, abort, p.status);
            if (!ok) break;
            tc::fence_after_sync();
            const uint32_t tS = tbase + lane_off + kColS + co;
            // rows of this step that some key of the block cannot see
            const bool diag = CAUSAL && (q0 + off < k0 + kBtKeys - 1);
            const float* l2 = sm.lse2[qs] + co;
            const int rq = q0 + co + off;             // aligned row of column 0
            float x[64];
#pragma unroll
            for (int h32 = 0; h32 < 2; ++h32) {
                uint32_t r[32];
                tc::tmem_ld_32x32b_x32(tS + 32 * h32, r);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int cc = 32 * h32 + c;
                    float t = __uint_as_float(r[c]) * p.scale_log2;
                    if (ALIBI) t -= slope_l2 * fabsf(float(rq + cc - key));
                    float pr = ex2(t - l2[cc]);
                    if (!key_ok || (diag && key > rq + cc)) pr = 0.f;
                    x[cc] = pr;
                }
            }
#pragma unroll
            for (int h16 = 0; h16 < 2; ++h16) {
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    pk[c] = pack_bf16(x[32 * h16 + 2 * c], x[32 * h16 + 2 * c + 1]);
                tmem_st16(tbase + lane_off + kColS + p_col + 16 * h16, pk);
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.p_full);
            // dS^T = P^T (dP^T - D)
            ok = mbar_wait_warp(&sm.dp_full, i & 1, abort, p.status);
            ok = ok && mbar_wait_warp(&sm.ofull[os], (i / kOStages) & 1, abort, p.status);
            if (!ok) break;
            tc::fence_after_sync();
            {
                const float* dd = sm.dsum[os] + co;
#pragma unroll
                for (int h32 = 0; h32 < 2; ++h32) {
                    uint32_t r[32];
                    tc::tmem_ld_32x32b_x32(tbase + lane_off + kColDP + co + 32 * h32, r);
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        x[32 * h32 + c] *= __uint_as_float(r[c]) - dd[32 * h32 + c];
                }
            }
            tc::fence_before_sync();
            // dS^T goes over the slot's dO tile once dV_i has read it
            ok = mbar_wait_warp(&sm.dv_done, i & 1, abort, p.status);
            if (!ok) break;
            uint8_t* row = sm.dout[os][half] + kl * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint4 w;
                w.x = pack_bf16(x[8 * j + 0], x[8 * j + 1]);
                w.y = pack_bf16(x[8 * j + 2], x[8 * j + 3]);
                w.z = pack_bf16(x[8 * j + 4], x[8 * j + 5]);
                w.w = pack_bf16(x[8 * j + 6], x[8 * j + 7]);
                *reinterpret_cast<uint4*>(row + ((uint32_t(j) ^ (uint32_t(kl) & 7u)) << 4)) = w;
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.ds_full);
        }

        // ---- dK (times the scale, group 0) or dV (group 1) of this block's
        //      keys; the TMEM loads are warp-collective, so only the stores
        //      depend on the lane's key
        if (ok) ok = mbar_wait_warp(&sm.acc_done, 0, abort, p.status);
        tc::fence_after_sync();
        if (__all_sync(0xffffffffu, ok && !*abort)) {
            const float mul = half ? 1.f : p.scale;
            __nv_bfloat16* dst = (half ? p.dV : p.dK) +
                                 ((size_t(b) * p.Hkv + kvh) * p.Lk + (key_ok ? key : 0)) * 128;
            const uint32_t col = half ? kColDV : kColDK;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                if (n > 0) {
                    tc::tmem_ld_32x32b_x32(tbase + lane_off + col + c * 32, r);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = 0u;
                }
#pragma unroll
                for (int v8 = 0; v8 < 4; ++v8) {
                    uint4 w;
                    w.x = pack_bf16(__uint_as_float(r[v8 * 8 + 0]) * mul,
                                    __uint_as_float(r[v8 * 8 + 1]) * mul);
                    w.y = pack_bf16(__uint_as_float(r[v8 * 8 + 2]) * mul,
                                    __uint_as_float(r[v8 * 8 + 3]) * mul);
                    w.z = pack_bf16(__uint_as_float(r[v8 * 8 + 4]) * mul,
                                    __uint_as_float(r[v8 * 8 + 5]) * mul);
                    w.w = pack_bf16(__uint_as_float(r[v8 * 8 + 6]) * mul,
                                    __uint_as_float(r[v8 * 8 + 7]) * mul);
                    if (key_ok) *reinterpret_cast<uint4*>(dst + c * 32 + v8 * 8) = w;
                }
            }
        }
        tc::fence_before_sync();
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsDrain));
        // ===================== dQ drain (warps 12-15, one head dim per thread)
        // Copies all 128 columns of dQ^T_i out of tensor memory at once, so
        // dP^T_{i+1} can reuse them, then adds them to the accumulator while
        // the next step runs.
        const int q4 = warp & 3;
        const int dl = q4 * 32 + lane;                // head dimension (TMEM lane)
        const uint32_t lane_off = uint32_t(q4 * 32) << 16;
        for (int i = 0; i < n; ++i) {
            if (!mbar_wait_warp(&sm.dq_full, i & 1, abort, p.status)) break;
            tc::fence_after_sync();
            float v[128];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t r[32];
                tc::tmem_ld_32x32b_x32(tbase + lane_off + kColDP + 32 * j, r);
#pragma unroll
                for (int c = 0; c < 32; ++c) v[32 * j + c] = __uint_as_float(r[c]);
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.dq_free);
            int h, q0;
            step_rows(i, h, q0);
            float* dst = p.dQacc + ((size_t(b) * p.Hq + h) * p.Lq + q0) * 128 + dl;
            const int rows = min(kBtRows, p.Lq - q0);
#pragma unroll
            for (int c = 0; c < 128; ++c)
                if (c < rows) atomicAdd(dst + size_t(c) * 128, v[c]);
        }
    }

    __syncwarp();
    __syncthreads();
    if (warp == 0 && lane == 0 && *abort) {
        // let this CTA's copies in flight land before its shared memory is released
        volatile int never = 0;
        mbar_wait(&sm.kv_full, 0, &never, p.status);
        for (int s = 0; s < kQStages; ++s) {
            int last = -1;
            for (int u = s; u < issued_q; u += kQStages) last = u;
            if (last >= 0) mbar_wait(&sm.qfull[s], (last / kQStages) & 1, &never, p.status);
        }
        for (int s = 0; s < kOStages; ++s) {
            int last = -1;
            for (int u = s; u < issued_o; u += kOStages) last = u;
            if (last >= 0) mbar_wait(&sm.ofull[s], (last / kOStages) & 1, &never, p.status);
        }
    }
    if (warp == 1) {
        volatile int never = 0;
        mbar_wait(&sm.acc_done, 0, &never, p.status);
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tbase, 512);
    }
}

namespace {

template <bool CAUSAL, bool ALIBI>
int launch_tc_t(const BwdTcLaunch& L, cudaStream_t stream) {
    const size_t smem = sizeof(BtSmem);   // used from the aligned start, no padding
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ERR_CUDA;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(bwd_tc_kernel<CAUSAL, ALIBI>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem)) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set[dev] = true;
    }
    const long long ctas = (long long)((L.p.Lk + kBtKeys - 1) / kBtKeys) * L.p.Hkv * L.p.B;
    if (ctas > 0x7fffffffLL) return ATTN_ERR_SHAPE;
    bwd_tc_kernel<CAUSAL, ALIBI><<<unsigned(ctas), kBtThreads, smem, stream>>>(
        L.tmQ, L.tmK, L.tmV, L.tmdO, L.p);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

int launch_backward_tc_main(const BwdTcLaunch& L, cudaStream_t stream) {
    const bool alibi = L.p.slopes != nullptr;
    if (L.p.causal)
        return alibi ? launch_tc_t<true, true>(L, stream) : launch_tc_t<true, false>(L, stream);
    return alibi ? launch_tc_t<false, true>(L, stream) : launch_tc_t<false, false>(L, stream);
}

}  // namespace attn
