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
// 2^8) and is done by the softmax group itself, so a third group would idle.
//
// CTA = two 128-row Q tiles that share one KV head: either two consecutive
// row blocks of one head (MHA) or the same row block of two query heads of a
// GQA group. Per KV step j:
//   TMA warp : K_j, V_j -> 3-slot shared-memory ring (128-byte swizzle)
//   MMA warp : S_t = Q_t K_j^T into TMEM (t = 0, 1), then O_t += P_t V_j
//   softmax t: S_t (TMEM) -> registers, row max, p = 2^(x - m), row sum,
//              P_t as bf16 into shared memory, O_t rescale in TMEM if needed
// One thread owns one query row (TMEM lane = row), so row reductions need no
// shuffles. Tensor memory: S_0, S_1 (128 fp32 columns each), O_0, O_1
// (d columns each) out of 512.
#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace attn {

namespace {

constexpr int kTcThreads = 384;                 // 12 warps
constexpr int kSoftmaxWarp0 = 4;                // warps 4..7: tile 0, 8..11: tile 1
constexpr float kRescaleThreshold = 8.0f;       // log2 units: rescale when max grows > 2^8
constexpr uint32_t kTileBytes = 128 * 128;      // one 128-row x 128-byte swizzled box

template <int D>
struct TcCfg {
    static constexpr int kBoxes = D / 64;                   // 64-element boxes per row
    static constexpr int kStages = D == 128 ? 3 : 6;        // K/V ring slots
    static constexpr uint32_t kSlotBytes = kBoxes * kTileBytes;
};

template <int D>
struct TcSmem {
    alignas(1024) uint8_t q[2][TcCfg<D>::kBoxes][kTileBytes];
    alignas(1024) uint8_t kv[TcCfg<D>::kStages][TcCfg<D>::kBoxes][kTileBytes];
    alignas(1024) uint8_t p[2][2][kTileBytes];   // P_t: keys 0..63, 64..127
    uint64_t bar_q;
    uint64_t kv_full[TcCfg<D>::kStages];
    uint64_t kv_empty[TcCfg<D>::kStages];
    uint64_t s_full[2];
    uint64_t s_free[2];
    uint64_t p_full[2];
    uint64_t o_done[2];
    uint64_t mma_fin;
    uint32_t tmem_base;
    int abort;
};

struct TileInfo {
    int head;    // query head
    int row0;    // first query row
    int n;       // KV tiles this Q tile needs
};

__device__ __forceinline__ int kv_tiles_for(int row0, int Lq, int Lk, int causal) {
    if (row0 >= Lq) return 0;
    int kend = Lk;
    if (causal) {
        const int last = min(row0 + 127, Lq - 1);
        kend = min(Lk, last + (Lk - Lq) + 1);
    }
    return kend > 0 ? (kend + 127) / 128 : 0;
}

}  // namespace

template <int D, bool CAUSAL, bool ALIBI>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, PrefillParams p) {
    using Cfg = TcCfg<D>;
    constexpr int NS = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    TcSmem<D>& sm = *reinterpret_cast<TcSmem<D>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int off = p.Lk - p.Lq;

    // ---- work item: two Q tiles sharing one KV head, heaviest rows first
    const int pair_heads = p.pair_heads;
    const int n_hb = pair_heads ? p.Hq / 2 : p.Hq;
    const int rows_per_item = pair_heads ? 128 : 256;
    const int n_rb = (p.Lq + rows_per_item - 1) / rows_per_item;
    const int rb = n_rb - 1 - int(blockIdx.x) / n_hb;
    const int hb = int(blockIdx.x) % n_hb;
    TileInfo tile[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        tile[t].head = pair_heads ? 2 * hb + t : hb;
        tile[t].row0 = pair_heads ? rb * 128 : rb * 256 + t * 128;
        tile[t].n = kv_tiles_for(tile[t].row0, p.Lq, p.Lk, CAUSAL);
    }
    const int kvh = tile[0].head / p.G;
    const int n = max(tile[0].n, tile[1].n);

    if (threadIdx.x == 0) {
        mbar_init(&sm.bar_q, 1);
        for (int i = 0; i < NS; ++i) {
            mbar_init(&sm.kv_full[i], 1);
            mbar_init(&sm.kv_empty[i], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&sm.s_full[t], 1);
            mbar_init(&sm.s_free[t], 4);
            mbar_init(&sm.p_full[t], 4);
            mbar_init(&sm.o_done[t], 1);
        }
        mbar_init(&sm.mma_fin, 1);
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
    int issued = 0;   // TMA loads issued (producer thread)

    if (warp == 0) {
        // ============================================== TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            mbar_arrive_expect_tx(&sm.bar_q, 2u * Cfg::kBoxes * kTileBytes);
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int bx = 0; bx < Cfg::kBoxes; ++bx)
                    tma_load_3d(sm.q[t][bx], &tmQ, &sm.bar_q, bx * 64, tile[t].row0,
                                b * p.Hq + tile[t].head);
            const int z = b * p.Hkv + kvh;
            int u = 0;
            bool ok = true;
            auto load = [&](int j, bool is_k) {
                const int slot = u % NS;
                if (u >= NS && !mbar_wait(&sm.kv_empty[slot], ((u / NS) - 1) & 1, abort, p.status))
                    return false;
                mbar_arrive_expect_tx(&sm.kv_full[slot], Cfg::kSlotBytes);
#pragma unroll
                for (int bx = 0; bx < Cfg::kBoxes; ++bx)
                    tma_load_3d(sm.kv[slot][bx], is_k ? &tmK : &tmV, &sm.kv_full[slot], bx * 64,
                                j * 128, z);
                ++u;
                issued = u;
                return true;
            };
            if (n > 0) ok = load(0, true);
            for (int j = 0; ok && j < n; ++j) {
                if (j + 1 < n) ok = load(j + 1, true);
                if (ok) ok = load(j, false);
            }
        }
    } else if (warp == 1) {
        // ============================================== MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_bf16(128, 128, 0);
            constexpr uint32_t idO = tc::idesc_bf16(128, D, 1);
            const uint32_t tS[2] = {tbase, tbase + 128};
            const uint32_t tO[2] = {tbase + 256, tbase + 256 + D};
            bool ok = mbar_wait(&sm.bar_q, 0, abort, p.status);
            tc::fence_after_sync();
            int u = 0;
            auto acquire = [&](int& slot) {
                slot = u % NS;
                if (!mbar_wait(&sm.kv_full[slot], (u / NS) & 1, abort, p.status)) return false;
                tc::fence_after_sync();
                return true;
            };
            auto release = [&](int slot) {
                tc::commit(&sm.kv_empty[slot]);
                ++u;
            };
            auto issue_s = [&](int t, int slot) {
                const uint32_t qa = smem_u32(sm.q[t][0]);
                const uint32_t ka = smem_u32(sm.kv[slot][0]);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t offb = (kk >> 2) * kTileBytes + (kk & 3) * 32;
                    tc::mma_bf16_ss(tS[t], tc::sdesc_sw128(qa + offb, 16, 1024),
                                    tc::sdesc_sw128(ka + offb, 16, 1024), idS, kk > 0);
                }
                tc::commit(&sm.s_full[t]);
            };
            auto issue_pv = [&](int t, int slot, int j) {
                const uint32_t pa = smem_u32(sm.p[t][0]);
                const uint32_t va = smem_u32(sm.kv[slot][0]);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t offa = (kk >> 2) * kTileBytes + (kk & 3) * 32;
                    tc::mma_bf16_ss(tO[t], tc::sdesc_sw128(pa + offa, 16, 1024),
                                    tc::sdesc_sw128(va + kk * 2048, kTileBytes, 1024), idO,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc::commit(&sm.o_done[t]);
            };
            int slot = 0;
            if (ok && n > 0) {
                ok = acquire(slot);
                if (ok) {
                    for (int t = 0; t < 2; ++t)
                        if (tile[t].n > 0) issue_s(t, slot);
                    release(slot);
                }
            }
            for (int j = 0; ok && j < n; ++j) {
                if (j + 1 < n) {
                    ok = acquire(slot);
                    if (!ok) break;
                    for (int t = 0; ok && t < 2; ++t) {
                        if (j + 1 < tile[t].n) {
                            ok = mbar_wait(&sm.s_free[t], j & 1, abort, p.status);
                            tc::fence_after_sync();
                            if (ok) issue_s(t, slot);
                        }
                    }
                    if (!ok) break;
                    release(slot);
                }
                ok = acquire(slot);
                if (!ok) break;
                for (int t = 0; ok && t < 2; ++t) {
                    if (j < tile[t].n) {
                        ok = mbar_wait(&sm.p_full[t], j & 1, abort, p.status);
                        tc::fence_after_sync();
                        if (ok) issue_pv(t, slot, j);
                    }
                }
                if (!ok) break;
                release(slot);
            }
            // every MMA this thread issued completes before the CTA ends
            tc::commit(&sm.mma_fin);
            volatile int never = 0;
            mbar_wait(&sm.mma_fin, 0, &never, p.status);
        }
    } else if (warp >= kSoftmaxWarp0) {
        // ============================================== softmax groups
        const int t = (warp - kSoftmaxWarp0) >> 2;
        const int q4 = warp & 3;                  // TMEM lane quadrant of this warp
        const int r = q4 * 32 + lane;             // row within the tile
        const TileInfo ti = tile[t];
        const int row = ti.row0 + r;
        const int i_al = row + off;               // bottom-right aligned row index
        const uint32_t lane_off = uint32_t(q4 * 32) << 16;
        const uint32_t tS = tbase + t * 128 + lane_off;
        const uint32_t tO = tbase + 256 + t * D + lane_off;
        const float sl2 = p.scale_log2;
        const float slope_l2 = ALIBI ? p.slopes[ti.head] * kLog2e : 0.f;
        uint8_t* prow = &sm.p[t][0][0];

        float m = -INFINITY;   // reference max (log2 domain)
        float l = 0.f;
        bool ok = true;
        for (int j = 0; j < ti.n; ++j) {
            ok = mbar_wait(&sm.s_full[t], j & 1, abort, p.status);
            if (!ok) break;
            tc::fence_after_sync();
            float s[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t rr[32];
                tc::tmem_ld_32x32b_x32(tS + c * 32, rr);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(rr[i]);
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.s_free[t]);

            const int k0 = j * 128;
            const bool need_mask =
                (k0 + 128 > p.Lk) || (CAUSAL && k0 + 127 > ti.row0 + q4 * 32 + off);
            // x = s * scale (log2 domain) + bias, masked; on unmasked tiles
            // without bias the scale is folded into the exp's FMA below
            const bool fast = !need_mask && !ALIBI && sl2 > 0.f;
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (fast) {
#pragma unroll
                for (int c = 0; c < 128; ++c) mx4[c & 3] = fmaxf(mx4[c & 3], s[c]);
            } else {
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    const int key = k0 + c;
                    float x = s[c] * sl2;
                    if (ALIBI) {
                        const float dist = float(i_al - key);
                        x -= slope_l2 * (CAUSAL ? dist : fabsf(dist));
                    }
                    if (need_mask && (key >= p.Lk || (CAUSAL && key > i_al))) x = -INFINITY;
                    s[c] = x;
                    mx4[c & 3] = fmaxf(mx4[c & 3], x);
                }
            }
            float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            if (fast) mx *= sl2;
            // conditional repair: move the reference max only when the row max
            // exceeds it by more than the threshold (or it is still unset)
            float m_new = m;
            if (mx > m + kRescaleThreshold || (m == -INFINITY && mx != -INFINITY)) m_new = mx;
            const bool rescale = (j > 0) && (m != -INFINITY) && (m_new != m);
            const float corr = rescale ? ex2(m - m_new) : 1.f;
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            float rs4[4] = {0.f, 0.f, 0.f, 0.f};
            if (fast) {
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    const float pv = ex2(fmaf(s[c], sl2, -m_use));
                    s[c] = pv;
                    rs4[c & 3] += pv;
                }
            } else {
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    const float pv = ex2(s[c] - m_use);
                    s[c] = pv;
                    rs4[c & 3] += pv;
                }
            }
            const float rs = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
            l = l * corr + rs;
            m = m_new;

            // P_t and O_t are free once PV of the previous step is done
            if (j > 0) {
                ok = mbar_wait(&sm.o_done[t], (j - 1) & 1, abort, p.status);
                if (!ok) break;
                tc::fence_after_sync();
            }
#pragma unroll
            for (int c16 = 0; c16 < 16; ++c16) {
                uint4 w;
                w.x = pack_bf16(s[c16 * 8 + 0], s[c16 * 8 + 1]);
                w.y = pack_bf16(s[c16 * 8 + 2], s[c16 * 8 + 3]);
                w.z = pack_bf16(s[c16 * 8 + 4], s[c16 * 8 + 5]);
                w.w = pack_bf16(s[c16 * 8 + 6], s[c16 * 8 + 7]);
                *reinterpret_cast<uint4*>(prow + (c16 >> 3) * kTileBytes +
                                          sw128_off(r, c16 & 7)) = w;
            }
            fence_proxy_async_smem();
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t rr[32];
                    tc::tmem_ld_32x32b_x32(tO + c * 32, rr);
#pragma unroll
                    for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * corr);
                    tc::tmem_st_32x32b_x32(tO + c * 32, rr);
                }
                tc::tmem_wait_st();
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.p_full[t]);
        }

        // ---------------------------------------------------- epilogue
        if (ok && ti.n > 0) {
            ok = mbar_wait(&sm.o_done[t], (ti.n - 1) & 1, abort, p.status);
            tc::fence_after_sync();
        }
        if (ok && !*abort) {
            const bool valid = row < p.Lq;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16* orow = p.O + ((size_t(b) * p.Hq + ti.head) * p.Lq + (valid ? row : 0)) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t rr[32];
                if (ti.n > 0) {
                    tc::tmem_ld_32x32b_x32(tO + c * 32, rr);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) rr[i] = 0u;
                }
                if (valid) {
#pragma unroll
                    for (int v8 = 0; v8 < 4; ++v8) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(rr[v8 * 8 + 0]) * inv, __uint_as_float(rr[v8 * 8 + 1]) * inv);
                        w.y = pack_bf16(__uint_as_float(rr[v8 * 8 + 2]) * inv, __uint_as_float(rr[v8 * 8 + 3]) * inv);
                        w.z = pack_bf16(__uint_as_float(rr[v8 * 8 + 4]) * inv, __uint_as_float(rr[v8 * 8 + 5]) * inv);
                        w.w = pack_bf16(__uint_as_float(rr[v8 * 8 + 6]) * inv, __uint_as_float(rr[v8 * 8 + 7]) * inv);
                        *reinterpret_cast<uint4*>(orow + c * 32 + v8 * 8) = w;
                    }
                }
            }
            if (valid && p.LSE)
                p.LSE[(size_t(b) * p.Hq + ti.head) * p.Lq + row] =
                    l > 0.f ? (m + lg2(l)) * kLn2 : -INFINITY;
        }
        tc::fence_before_sync();
    }

    __syncwarp();
    __syncthreads();
    if (warp == 0 && lane == 0 && *abort) {
        // let this CTA's copies in flight land before its shared memory is released
        volatile int never = 0;
        mbar_wait(&sm.bar_q, 0, &never, p.status);
        for (int s = 0; s < NS; ++s) {
            int last = -1;
            for (int u = s; u < issued; u += NS) last = u;
            if (last >= 0) mbar_wait(&sm.kv_full[s], (last / NS) & 1, &never, p.status);
        }
    }
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tbase, 512);
    }
}

namespace {

template <int D, bool CAUSAL, bool ALIBI>
int launch_tc_t(const PrefillLaunch& L, cudaStream_t stream) {
    const size_t smem = sizeof(TcSmem<D>) + 1024;
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(prefill_tc_kernel<D, CAUSAL, ALIBI>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem)) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set[dev] = true;
    }
    const int rows_per_item = L.p.pair_heads ? 128 : 256;
    const int n_hb = L.p.pair_heads ? L.p.Hq / 2 : L.p.Hq;
    const long long items = (long long)((L.p.Lq + rows_per_item - 1) / rows_per_item) * n_hb;
    if (items > 0x7fffffffLL) return ATTN_ERR_SHAPE;
    dim3 grid(unsigned(items), L.p.B);
    prefill_tc_kernel<D, CAUSAL, ALIBI><<<grid, kTcThreads, smem, stream>>>(L.tmQ, L.tmK, L.tmV,
                                                                           L.p);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int D>
int launch_tc_d(const PrefillLaunch& L, cudaStream_t stream) {
    const bool alibi = L.p.slopes != nullptr;
    if (L.p.causal)
        return alibi ? launch_tc_t<D, true, true>(L, stream) : launch_tc_t<D, true, false>(L, stream);
    return alibi ? launch_tc_t<D, false, true>(L, stream) : launch_tc_t<D, false, false>(L, stream);
}

}  // namespace

int launch_prefill_tc(const PrefillLaunch& L, int d, cudaStream_t stream) {
    if (d == 64) return launch_tc_d<64>(L, stream);
    if (d == 128) return launch_tc_d<128>(L, stream);
    return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
