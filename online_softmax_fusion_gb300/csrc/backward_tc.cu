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
// Every product has the key block (or the head dimension) as its M = 128
// side: S^T and dP^T are 128 x 64 (keys x queries), dV and dK 128 x 128,
// and dQ is produced transposed (128 head-dim rows x 64 queries) so that it
// too has M = 128.
//
// CTA roles (384 threads):
//   warp 0      TMA: K, V once; per step the Q and dO tiles (64 rows) into a
//               4-slot ring, LSE and D of the 64 rows into the same slot
//   warp 1      TMEM allocation; tcgen05.mma issue (one elected lane)
//   warps 4-11  two warpgroups, one thread per key (TMEM lane), each taking
//               32 of the step's 64 query columns: P^T from S^T, P^T (bf16)
//               back into TMEM for dV; dS^T from dP^T into shared memory
//               (bf16) for dK and dQ^T; the previous step's dQ^T columns
//               (TMEM lane = head dimension) added to the fp32 accumulator
//               while dP^T is computed; at the end dK (warps 4-7) and dV
//               (warps 8-11)
// Tensor memory (512 columns): S^T double-buffered (2 x 64; P^T bf16 is
// written over S^T columns its group has read), dP^T (64), dQ^T (64), dV (128),
// dK (128). S^T of the next step is computed while P^T of this step is
// formed. Shared memory: K and V (resident, 128-byte swizzle), the ring and
// one dS^T tile.
//
// Issue order of the tensor core per step i:
//   S_{i+1} | (P_i) dV_i | (dS_i) dP_{i+1}, dK_i, (dQ drained) dQ^T_i
// The parenthesised names are the hand-offs each product waits for.
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace attn {

namespace {

constexpr int kBtThreads = 384;
constexpr int kBtKeys = 128;                  // keys per CTA
constexpr int kBtRows = 64;                   // query rows per step
constexpr int kBtStages = 4;                  // Q / dO ring slots
constexpr uint32_t kKVBox = 128 * 128;        // 128 keys x 64 dims (bf16, 128 B rows)
constexpr uint32_t kQBox = 64 * 128;          // 64 rows x 64 dims
// TMEM columns
constexpr uint32_t kColS = 0;                 // S^T buffers at 0 and 64
constexpr uint32_t kColDP = 128;
constexpr uint32_t kColDQ = 192;
constexpr uint32_t kColDV = 256;
constexpr uint32_t kColDK = 384;

struct BtSmem {
    alignas(1024) uint8_t k[2][kKVBox];                     // K block, dims 0-63 / 64-127
    alignas(1024) uint8_t v[2][kKVBox];
    alignas(1024) uint8_t qd[kBtStages][4][kQBox];          // per slot: Q (2 boxes), dO (2 boxes)
    alignas(1024) uint8_t ds[kBtKeys * 128];                // dS^T [key][64 queries] bf16
    float lse2[kBtStages][kBtRows];                         // LSE * log2(e); +inf = no weight
    float dsum[kBtStages][kBtRows];                         // D_i
    uint64_t kv_full;
    uint64_t full[kBtStages];
    uint64_t empty[kBtStages];
    uint64_t s_full[2];
    uint64_t dp_full;
    uint64_t p_full;
    uint64_t ds_full;
    uint64_t ds_free;
    uint64_t dq_full;
    uint64_t dq_free;
    uint64_t acc_done;
    uint32_t tmem_base;
    int abort;
};

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

// 32 lanes x 64 consecutive 32-bit columns, then wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
    uint32_t a[32], b[32];
    tc::tmem_ld_32x32b_x32(taddr, a);
    tc::tmem_ld_32x32b_x32(taddr + 32u, b);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        v[i] = __uint_as_float(a[i]);
        v[32 + i] = __uint_as_float(b[i]);
    }
}

}  // namespace

template <bool CAUSAL, bool ALIBI>
__global__ void __launch_bounds__(kBtThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    BtSmem& sm = *reinterpret_cast<BtSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
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
        for (int s = 0; s < kBtStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int c = 0; c < 2; ++c) mbar_init(&sm.s_full[c], 1);
        mbar_init(&sm.ds_full, 8);
        mbar_init(&sm.ds_free, 1);
        mbar_init(&sm.dp_full, 1);
        mbar_init(&sm.p_full, 8);
        mbar_init(&sm.dq_full, 1);
        mbar_init(&sm.dq_free, 8);
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
    int issued = 0;   // steps whose Q / dO loads were issued (producer, lane 0)

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
        for (int i = 0; i < n; ++i) {
            const int s = i % kBtStages;
            bool ok = true;
            if (i >= kBtStages)
                ok = mbar_wait(&sm.empty[s], ((i / kBtStages) - 1) & 1, abort, p.status);
            if (__any_sync(0xffffffffu, !ok)) break;
            int h, q0;
            step_rows(i, h, q0);
            const size_t rb = (size_t(b) * p.Hq + h) * p.Lq;
            for (int r = lane; r < kBtRows; r += 32) {
                const int row = q0 + r;
                float l2 = INFINITY, dd = 0.f;
                if (row < p.Lq) {
                    const float l = p.LSE[rb + row];
                    if (l != -INFINITY) l2 = l * kLog2e;
                    dd = p.Dsum[rb + row];
                }
                sm.lse2[s][r] = l2;
                sm.dsum[s][r] = dd;
            }
            __syncwarp();
            if (lane == 0) {
                const int z = b * p.Hq + h;
                mbar_arrive_expect_tx(&sm.full[s], 4 * kQBox);
                for (int bx = 0; bx < 2; ++bx) {
                    tma_load_3d(sm.qd[s][bx], &tmQ, &sm.full[s], bx * 64, q0, z);
                    tma_load_3d(sm.qd[s][2 + bx], &tmdO, &sm.full[s], bx * 64, q0, z);
                }
                issued = i + 1;
            }
        }
    } else if (warp == 1) {
        // ================================================== MMA issuer
        // (the whole warp runs the loop; one elected lane issues)
        constexpr uint32_t idS = tc::idesc_bf16_ab(128, 64, 0, 0);     // S^T, dP^T
        constexpr uint32_t idD = tc::idesc_bf16_ab(128, 128, 0, 1);    // dV (A TMEM), dK
        constexpr uint32_t idQ = tc::idesc_bf16_ab(128, 64, 1, 1);     // dQ^T
        const uint64_t dk_ = tc::sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);          // K, K-major
        const uint64_t dv_ = tc::sdesc_sw128(smem_u32(sm.v[0]), 16, 1024);
        const uint64_t dkT = tc::sdesc_sw128(smem_u32(sm.k[0]), kKVBox, 1024);      // K^T, MN-major
        const uint64_t dq0 = tc::sdesc_sw128(smem_u32(sm.qd[0][0]), 16, 1024);      // Q / dO K-major
        const uint64_t dqm = tc::sdesc_sw128(smem_u32(sm.qd[0][0]), kQBox, 1024);   // Q / dO MN-major
        const uint64_t dsk = tc::sdesc_sw128(smem_u32(sm.ds), 16, 1024);            // dS^T K-major
        const uint64_t dsm = tc::sdesc_sw128(smem_u32(sm.ds), 16384, 1024);         // dS^T MN-major
        constexpr uint32_t kSlot = (4 * kQBox) >> 4;     // ring slot stride (16-byte units)
        constexpr uint32_t kDO = (2 * kQBox) >> 4;       // dO after Q in a slot
        // A x B over K = 128 dims: 8 steps of 16, box switch after 4
        auto issue_qk = [&](uint64_t a0, uint64_t b0, uint32_t d) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t oa = ((kk >> 2) * kKVBox + (kk & 3) * 32) >> 4;
                const uint32_t ob = ((kk >> 2) * kQBox + (kk & 3) * 32) >> 4;
                tc::mma_bf16_ss_warp(d, a0 + oa, b0 + ob, idS, kk > 0);
            }
        };
        bool ok = mbar_wait_warp(&sm.kv_full, 0, abort, p.status);
        tc::fence_after_sync();
        auto wait_full = [&](int i) {
            ok = ok && mbar_wait_warp(&sm.full[i % kBtStages], (i / kBtStages) & 1, abort, p.status);
            tc::fence_after_sync();
        };
        if (ok && n > 0) {
            wait_full(0);
            if (ok) {
                issue_qk(dk_, dq0, tbase + kColS);
                tc::commit_warp(&sm.s_full[0]);
                issue_qk(dv_, dq0 + kDO, tbase + kColDP);
                tc::commit_warp(&sm.dp_full);
            }
        }
        for (int i = 0; ok && i < n; ++i) {
            const int s = i % kBtStages;
            const uint32_t so = uint32_t(s) * kSlot;
            if (i + 1 < n) {
                wait_full(i + 1);
                if (!ok) break;
                const uint32_t s1 = uint32_t((i + 1) % kBtStages) * kSlot;
                issue_qk(dk_, dq0 + s1, tbase + kColS + ((i + 1) & 1) * 64);
                tc::commit_warp(&sm.s_full[(i + 1) & 1]);
            }
            // dV += P^T dO (P^T bf16 in TMEM over the upper half of S^T)
            ok = mbar_wait_warp(&sm.p_full, i & 1, abort, p.status);
            if (!ok) break;
            tc::fence_after_sync();
            {
                const uint32_t tP = tbase + kColS + (i & 1) * 64;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_bf16_ts_warp(tbase + kColDV, tP + (kk < 2 ? kk * 8 : 48 + (kk - 2) * 8),
                                         dqm + so + kDO + uint32_t(kk * (2048 >> 4)), idD,
                                         (i > 0 || kk > 0) ? 1u : 0u);
            }
            // dS^T of step i is in shared memory (and dP^T has been read)
            ok = mbar_wait_warp(&sm.ds_full, i & 1, abort, p.status);
            if (!ok) break;
            tc::fence_after_sync();
            if (i + 1 < n) {
                const uint32_t s1 = uint32_t((i + 1) % kBtStages) * kSlot;
                issue_qk(dv_, dq0 + s1 + kDO, tbase + kColDP);
                tc::commit_warp(&sm.dp_full);
            }
            // dK += dS^T Q
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc::mma_bf16_ss_warp(tbase + kColDK, dsk + uint32_t(kk * 2),
                                     dqm + so + uint32_t(kk * (2048 >> 4)), idD,
                                     (i > 0 || kk > 0) ? 1u : 0u);
            // dQ^T = K^T dS^T once the previous dQ^T has been drained
            if (i > 0) {
                ok = mbar_wait_warp(&sm.dq_free, (i - 1) & 1, abort, p.status);
                if (!ok) break;
                tc::fence_after_sync();
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::mma_bf16_ss_warp(tbase + kColDQ, dkT + uint32_t(kk * (2048 >> 4)),
                                     dsm + uint32_t(kk * (2048 >> 4)), idQ, kk > 0);
            tc::commit_warp(&sm.dq_full);
            tc::commit_warp(&sm.empty[s]);
            tc::commit_warp(&sm.ds_free);
        }
        // covers every MMA issued above; the epilogue and TMEM release wait on it
        tc::commit_warp(&sm.acc_done);
    } else if (warp >= 4) {
        // ===================== P^T, dS^T and the dQ drain (one key per thread)
        // Two warpgroups split the 64 query columns of a step: warps 4-7
        // take columns 0-31, warps 8-11 columns 32-63 (same TMEM lanes).
        const int half = warp >= 8 ? 1 : 0;
        const int co = half * 32;                     // first query column of this group
        const int q4 = warp & 3;
        const int kl = q4 * 32 + lane;                // key within the block (TMEM lane)
        const int key = k0 + kl;
        const bool key_ok = key < p.Lk;
        const uint32_t lane_off = uint32_t(q4 * 32) << 16;
        // P^T (bf16) of this group's 32 queries goes over S^T columns this
        // group has read and the other group never reads: columns 0-15
        // (group 0) and 48-63 (group 1) of the step's S^T buffer
        const uint32_t p_col = half ? 48u : 0u;
        bool ok = true;
        // adds the dQ^T columns of this group for step j to the accumulator
        // (TMEM lane = head dimension here)
        auto drain_dq = [&](int j) -> bool {
            if (!mbar_wait_warp(&sm.dq_full, j & 1, abort, p.status)) return false;
            tc::fence_after_sync();
            uint32_t v[32];
            tc::tmem_ld_32x32b_x32(tbase + lane_off + kColDQ + co, v);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.dq_free);
            int h, q0;
            step_rows(j, h, q0);
            float* dst = p.dQacc + ((size_t(b) * p.Hq + h) * p.Lq + q0 + co) * 128 + kl;
            const int rows = min(32, p.Lq - q0 - co);
#pragma unroll
            for (int c = 0; c < 32; ++c)
                if (c < rows) atomicAdd(dst + size_t(c) * 128, __uint_as_float(v[c]));
            return true;
        };
        for (int i = 0; i < n; ++i) {
            const int s = i % kBtStages;
            int h, q0;
            step_rows(i, h, q0);
            const float slope_l2 = ALIBI ? p.slopes[h] * kLog2e : 0.f;
            ok = mbar_wait_warp(&sm.s_full[i & 1], (i >> 1) & 1, abort, p.status);
            ok = ok && mbar_wait_warp(&sm.full[s], (i / kBtStages) & 1, abort, p.status);
            if (!ok) break;
            tc::fence_after_sync();
            const uint32_t tS = tbase + lane_off + kColS + (i & 1) * 64;
            float x[32];
            {
                uint32_t r[32];
                tc::tmem_ld_32x32b_x32(tS + co, r);
#pragma unroll
                for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(r[c]);
            }
            // rows of this step that some key of the block cannot see
            const bool diag = CAUSAL && (q0 + off < k0 + kBtKeys - 1);
            const float* l2 = sm.lse2[s] + co;
            const int rq = q0 + co + off;             // aligned row of column 0
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                float t = x[c] * p.scale_log2;
                if (ALIBI) t -= slope_l2 * fabsf(float(rq + c - key));
                float pr = ex2(t - l2[c]);
                if (!key_ok || (diag && key > rq + c)) pr = 0.f;
                x[c] = pr;
            }
            {
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) pk[c] = pack_bf16(x[2 * c], x[2 * c + 1]);
                tmem_st16(tS + p_col, pk);
                tc::tmem_wait_st();
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.p_full);
            // the previous step's dQ^T, while dP^T of this step is computed
            if (i > 0 && !drain_dq(i - 1)) { ok = false; break; }
            // dS^T = P^T (dP^T - D)
            ok = mbar_wait_warp(&sm.dp_full, i & 1, abort, p.status);
            if (!ok) break;
            tc::fence_after_sync();
            {
                uint32_t r[32];
                tc::tmem_ld_32x32b_x32(tbase + lane_off + kColDP + co, r);
                const float* dd = sm.dsum[s] + co;
#pragma unroll
                for (int c = 0; c < 32; ++c) x[c] = x[c] * (__uint_as_float(r[c]) - dd[c]);
            }
            // the single dS^T buffer: dK and dQ^T of the previous step have
            // completed (the dQ^T drain above already waited for them)
            if (i >= 1) {
                ok = mbar_wait_warp(&sm.ds_free, (i - 1) & 1, abort, p.status);
                if (!ok) break;
            }
            uint8_t* row = sm.ds + kl * 128;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint4 w;
                w.x = pack_bf16(x[8 * j + 0], x[8 * j + 1]);
                w.y = pack_bf16(x[8 * j + 2], x[8 * j + 3]);
                w.z = pack_bf16(x[8 * j + 4], x[8 * j + 5]);
                w.w = pack_bf16(x[8 * j + 6], x[8 * j + 7]);
                const uint32_t chunk = uint32_t(half * 4 + j);
                *reinterpret_cast<uint4*>(row + ((chunk ^ (uint32_t(kl) & 7u)) << 4)) = w;
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.ds_full);
        }
        if (ok && n > 0) ok = drain_dq(n - 1);
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
    }

    __syncwarp();
    __syncthreads();
    if (warp == 0 && lane == 0 && *abort) {
        // let this CTA's copies in flight land before its shared memory is released
        volatile int never = 0;
        mbar_wait(&sm.kv_full, 0, &never, p.status);
        for (int s = 0; s < kBtStages; ++s) {
            int last = -1;
            for (int u = s; u < issued; u += kBtStages) last = u;
            if (last >= 0) mbar_wait(&sm.full[s], (last / kBtStages) & 1, &never, p.status);
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
    const size_t smem = sizeof(BtSmem) + 1024;
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
