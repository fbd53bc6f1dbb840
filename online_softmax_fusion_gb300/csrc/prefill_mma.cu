// Register-tile prefill (mma.sync), the Rolling Update form of attention.
//
// Rolling Update (Neptune论文浅读 (gentlecold.top) §5): the loop over K/V
// blocks carries the previous and current row max; every step repairs the
// running sum and output with exp(m_old - m_new) (§3-§4) before adding the
// new block. Structure: the three-level loop of the CANN FlashAttention blog
// (ai6s.net), section "ops-transformer在昇腾NPU上的工程处理": one CTA per Q
// block, an inner loop over K/V blocks, QK^T then the online softmax update
// then PV, with the next K/V block's copy overlapping the current compute.
//
// This is the portable tensor-core path (warp-level mma.sync on registers),
// kept as a cross-check for the tcgen05 kernel and as the path for shapes
// that kernel does not take. CTA: 8 consumer warps x 16 query rows plus one
// TMA producer warp; K/V tiles of 64 keys in a 2-stage ring.
#include "common.cuh"
#include "kernels.h"

namespace attn {

constexpr int kMmaWarps = 8;
constexpr int kMmaThreads = (kMmaWarps + 1) * 32;
constexpr int kMmaStages = 2;

template <int D>
struct MmaSmem {
    alignas(1024) uint8_t q[D / 64][kMmaBM * 128];
    alignas(1024) uint8_t kv[kMmaStages][2][D / 64][kMmaBN * 128];
    uint64_t qfull;
    uint64_t full[kMmaStages];
    uint64_t empty[kMmaStages];
    int abort;
};

template <int D, bool CAUSAL, bool ALIBI>
__global__ void __launch_bounds__(kMmaThreads)
    prefill_mma_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    MmaSmem<D>& sm = *reinterpret_cast<MmaSmem<D>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    // Causal: launch the longest rows first.
    const int qt = CAUSAL ? int(gridDim.x - 1 - blockIdx.x) : int(blockIdx.x);
    const int h = blockIdx.y;
    const int b = blockIdx.z;
    const int kvh = h / p.G;
    const int q0 = qt * kMmaBM;
    const int off = p.Lk - p.Lq;   // bottom-right alignment of the causal mask
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    int kend = p.Lk;
    if (CAUSAL) kend = min(p.Lk, q0 + kMmaBM + off);
    const int ntiles = kend > 0 ? (kend + kMmaBN - 1) / kMmaBN : 0;

    if (threadIdx.x == 0) {
        mbar_init(&sm.qfull, 1);
        for (int i = 0; i < kMmaStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], kMmaWarps);
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    volatile int* abort = &sm.abort;

    int issued = 0;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    if (warp == kMmaWarps) {
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            mbar_arrive_expect_tx(&sm.qfull, (D / 64) * kMmaBM * 128);
#pragma unroll
            for (int bx = 0; bx < D / 64; ++bx)
                tma_load_3d(sm.q[bx], &tmQ, &sm.qfull, bx * 64, q0, b * p.Hq + h);
            const int z = b * p.Hkv + kvh;
            for (int it = 0; it < ntiles; ++it) {
                const int st = it % kMmaStages;
                if (it >= kMmaStages &&
                    !mbar_wait(&sm.empty[st], ((it / kMmaStages) - 1) & 1, abort, p.status))
                    break;
                mbar_arrive_expect_tx(&sm.full[st], 2u * (D / 64) * kMmaBN * 128);
#pragma unroll
                for (int bx = 0; bx < D / 64; ++bx) {
                    tma_load_3d(sm.kv[st][0][bx], &tmK, &sm.full[st], bx * 64, it * kMmaBN, z);
                    tma_load_3d(sm.kv[st][1][bx], &tmV, &sm.full[st], bx * 64, it * kMmaBN, z);
                }
                issued = it + 1;
            }
        }
    } else if (mbar_wait_warp(&sm.qfull, 0, abort, p.status)) {
        const int g = lane >> 2, t4 = lane & 3;
        uint32_t qa[D / 16][4];
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int r = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int c16 = 2 * kk + (lane >> 4);
            ldsm_x4(smem_u32(&sm.q[c16 / 8][sw128_off(r, c16 % 8)]), qa[kk][0], qa[kk][1],
                    qa[kk][2], qa[kk][3]);
        }
        const int row_al[2] = {q0 + 16 * warp + g + off, q0 + 16 * warp + g + 8 + off};
        const float slope_l2 = ALIBI ? p.slopes[h] * kLog2e : 0.f;

        for (int it = 0; it < ntiles; ++it) {
            const int st = it % kMmaStages;
            if (!mbar_wait_warp(&sm.full[st], (it / kMmaStages) & 1, abort, p.status)) break;
            const uint8_t* kt = &sm.kv[st][0][0][0];
            const uint8_t* vt = &sm.kv[st][1][0][0];

            float sc[kMmaBN / 8][4];
#pragma unroll
            for (int i = 0; i < kMmaBN / 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
                for (int np = 0; np < kMmaBN / 16; ++np) {
                    const int key = 16 * np + (lane & 7) + ((lane >> 4) & 1) * 8;
                    const int c16 = 2 * kk + ((lane >> 3) & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(smem_u32(kt + (c16 / 8) * kMmaBN * 128 + sw128_off(key, c16 % 8)), b0,
                            b1, b2, b3);
                    mma_bf16_16816(sc[2 * np], qa[kk], b0, b1);
                    mma_bf16_16816(sc[2 * np + 1], qa[kk], b2, b3);
                }
            const int k0 = it * kMmaBN;
            const bool need_mask =
                (k0 + kMmaBN > p.Lk) || (CAUSAL && k0 + kMmaBN - 1 > q0 + 16 * warp + off);
#pragma unroll
            for (int nt = 0; nt < kMmaBN / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = k0 + nt * 8 + 2 * t4 + (e & 1);
                    const int r = e >> 1;
                    float x = sc[nt][e] * p.scale_log2;
                    if (ALIBI) x -= slope_l2 * fabsf(float(row_al[r] - j));
                    if (need_mask && (j >= p.Lk || (CAUSAL && j > row_al[r]))) x = -INFINITY;
                    sc[nt][e] = x;
                }
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float mx = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < kMmaBN / 8; ++nt)
                    mx = fmaxf(mx, fmaxf(sc[nt][2 * r], sc[nt][2 * r + 1]));
                mx = shfl_xor_max(mx, 1);
                mx = shfl_xor_max(mx, 2);
                const float m_new = fmaxf(m_run[r], mx);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                const float corr = ex2(m_run[r] - m_use);
                m_run[r] = m_new;
                float ps = 0.f;
#pragma unroll
                for (int nt = 0; nt < kMmaBN / 8; ++nt)
#pragma unroll
                    for (int e = 2 * r; e < 2 * r + 2; ++e) {
                        const float pv = ex2(sc[nt][e] - m_use);
                        sc[nt][e] = pv;
                        ps += pv;
                    }
                l_run[r] = l_run[r] * corr + ps;
#pragma unroll
                for (int dn = 0; dn < D / 8; ++dn) {
                    o[dn][2 * r] *= corr;
                    o[dn][2 * r + 1] *= corr;
                }
            }
#pragma unroll
            for (int k2 = 0; k2 < kMmaBN / 16; ++k2) {
                const uint32_t pa[4] = {
                    pack_bf16(sc[2 * k2][0], sc[2 * k2][1]), pack_bf16(sc[2 * k2][2], sc[2 * k2][3]),
                    pack_bf16(sc[2 * k2 + 1][0], sc[2 * k2 + 1][1]),
                    pack_bf16(sc[2 * k2 + 1][2], sc[2 * k2 + 1][3])};
#pragma unroll
                for (int dn2 = 0; dn2 < D / 16; ++dn2) {
                    const int key = 16 * k2 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int c16 = 2 * dn2 + (lane >> 4);
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_t(smem_u32(vt + (c16 / 8) * kMmaBN * 128 + sw128_off(key, c16 % 8)),
                              v0, v1, v2, v3);
                    mma_bf16_16816(o[2 * dn2], pa, v0, v1);
                    mma_bf16_16816(o[2 * dn2 + 1], pa, v2, v3);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[st]);
        }

        if (!*abort) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
                l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
                const int i = q0 + 16 * warp + g + 8 * r;
                if (i < p.Lq) {
                    const float inv = l_run[r] > 0.f ? 1.f / l_run[r] : 0.f;
                    __nv_bfloat16* orow = p.O + ((size_t(b) * p.Hq + h) * p.Lq + i) * D;
#pragma unroll
                    for (int dn = 0; dn < D / 8; ++dn) {
                        const __nv_bfloat162 v =
                            __floats2bfloat162_rn(o[dn][2 * r] * inv, o[dn][2 * r + 1] * inv);
                        *reinterpret_cast<__nv_bfloat162*>(orow + dn * 8 + 2 * t4) = v;
                    }
                    if (t4 == 0 && p.LSE)
                        p.LSE[(size_t(b) * p.Hq + h) * p.Lq + i] =
                            l_run[r] > 0.f ? (m_run[r] + lg2(l_run[r])) * kLn2 : -INFINITY;
                }
            }
        }
    }
    __syncthreads();
    if (*abort && warp == kMmaWarps && lane == 0) {
        volatile int never = 0;
        mbar_wait(&sm.qfull, 0, &never, p.status);
        for (int st = 0; st < kMmaStages; ++st) {
            int last = -1;
            for (int it = st; it < issued; it += kMmaStages) last = it;
            if (last >= 0) mbar_wait(&sm.full[st], (last / kMmaStages) & 1, &never, p.status);
        }
    }
}

template <int D, bool CAUSAL, bool ALIBI>
static int launch_mma_t(const PrefillLaunch& L, cudaStream_t stream) {
    const size_t smem = sizeof(MmaSmem<D>) + 1024;
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(prefill_mma_kernel<D, CAUSAL, ALIBI>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem)) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set[dev] = true;
    }
    dim3 grid((L.p.Lq + kMmaBM - 1) / kMmaBM, L.p.Hq, L.p.B);
    prefill_mma_kernel<D, CAUSAL, ALIBI><<<grid, kMmaThreads, smem, stream>>>(L.tmQ, L.tmK, L.tmV,
                                                                             L.p);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int D>
static int launch_mma_d(const PrefillLaunch& L, cudaStream_t stream) {
    const bool alibi = L.p.slopes != nullptr;
    if (L.p.causal)
        return alibi ? launch_mma_t<D, true, true>(L, stream) : launch_mma_t<D, true, false>(L, stream);
    return alibi ? launch_mma_t<D, false, true>(L, stream) : launch_mma_t<D, false, false>(L, stream);
}

int launch_prefill_mma(const PrefillLaunch& L, int d, cudaStream_t stream) {
    if (d == 64) return launch_mma_d<64>(L, stream);
    if (d == 128) return launch_mma_d<128>(L, stream);
    return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
