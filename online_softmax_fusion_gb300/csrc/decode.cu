// Split-K decode and its log-sum-exp combine.
//
// Split-K Update (Neptune论文浅读 (gentlecold.top) §6): the key axis is cut
// into splits that are reduced independently (a local max, sum and output
// each), then a global reduction repairs every split with the global max.
// Work decomposition follows the grouped-query decode of CMU 15-779 第 11 讲
// §7.1: one CTA per (batch, KV head, split), the G query heads of the group
// stacked as the rows of one matrix product so every K/V row is read from
// HBM once per KV head.
//
// Data path per CTA: a producer warp streams 64-key K and V tiles with TMA
// (128-byte swizzle) into a 3-stage shared-memory ring guarded by
// mbarriers; four consumer warps each take 16 keys of every tile, compute
// S = Q K^T and O += P V with mma.sync (G heads padded to 16 rows), and keep
// a running max / sum / output per row with the exp(m_old - m_new) repair.
// The four warps' partial states are merged in shared memory at the end.
#include "common.cuh"
#include "kernels.h"

namespace attn {

constexpr int kDecTile = 64;        // keys per tile
constexpr int kDecStages = 3;       // ring depth
constexpr int kDecWarps = 4;        // consumer warps
constexpr int kDecThreads = (kDecWarps + 1) * 32;

template <int D>
struct DecodeSmem {
    // Per stage: K then V, each D/64 boxes of [64 keys][128 B], swizzled.
    alignas(1024) uint8_t kv[kDecStages][2][D / 64][kDecTile * 128];
    alignas(1024) uint8_t q[D / 64][16 * 128];   // 16 query rows, swizzled
    uint64_t full[kDecStages];
    uint64_t empty[kDecStages];
    int abort;
};

template <int D>
__global__ void __launch_bounds__(kDecThreads)
    decode_splitk_kernel(const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    DecodeSmem<D>& sm = *reinterpret_cast<DecodeSmem<D>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int s = blockIdx.x;
    const int kvh = blockIdx.y / p.nrg;
    const int rg = blockIdx.y % p.nrg;
    const int b = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    int kv_len = p.kv_lens ? p.kv_lens[b] : p.Lk_max;
    kv_len = min(max(kv_len, 0), p.Lk_max);
    const int lo = s * p.C;
    const int hi = min(lo + p.C, kv_len);
    const int h0 = kvh * p.G + rg * p.rows;
    const int nrows = min(p.rows, p.G - rg * p.rows);

    if (hi <= lo) {  // empty split: weight zero in the combine
        for (int i = threadIdx.x; i < nrows * D; i += blockDim.x) {
            const int r = i / D, c = i % D;
            p.O_part[((size_t(b) * p.Hq + h0 + r) * p.S + s) * D + c] = 0.f;
        }
        if (threadIdx.x < nrows)
            p.LSE_part[(size_t(b) * p.Hq + h0 + threadIdx.x) * p.S + s] = -INFINITY;
        return;
    }
    const int ntiles = (hi - lo + kDecTile - 1) / kDecTile;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kDecStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], kDecWarps);
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    // Query rows of the group (padded to 16 with zeros), swizzled like K.
    for (int i = threadIdx.x; i < 16 * (D / 8); i += blockDim.x) {
        const int r = i / (D / 8), c16 = i % (D / 8);
        uint4 val = make_uint4(0, 0, 0, 0);
        if (r < nrows)
            val = *reinterpret_cast<const uint4*>(p.Q + (size_t(b) * p.Hq + h0 + r) * D + c16 * 8);
        *reinterpret_cast<uint4*>(&sm.q[c16 / 8][sw128_off(r, c16 % 8)]) = val;
    }
    __syncthreads();

    volatile int* abort = &sm.abort;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    int issued = 0;
    if (warp == kDecWarps) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            const int z = b * p.Hkv + kvh;
            for (int it = 0; it < ntiles; ++it) {
                const int st = it % kDecStages;
                if (it >= kDecStages &&
                    !mbar_wait(&sm.empty[st], ((it / kDecStages) - 1) & 1, abort, p.status))
                    break;
                mbar_arrive_expect_tx(&sm.full[st], 2u * (D / 64) * kDecTile * 128);
                const int key0 = lo + it * kDecTile;
#pragma unroll
                for (int bx = 0; bx < D / 64; ++bx) {
                    tma_load_3d(sm.kv[st][0][bx], &tmK, &sm.full[st], bx * 64, key0, z);
                    tma_load_3d(sm.kv[st][1][bx], &tmV, &sm.full[st], bx * 64, key0, z);
                }
                issued = it + 1;
            }
        }
    } else {
        // ------------------------------------------------------ consumers
        uint32_t qa[D / 16][4];
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int c16 = 2 * kk + (lane >> 4);
            ldsm_x4(smem_u32(&sm.q[c16 / 8][sw128_off(r, c16 % 8)]), qa[kk][0], qa[kk][1],
                    qa[kk][2], qa[kk][3]);
        }
        const int t4 = lane & 3;
        for (int it = 0; it < ntiles; ++it) {
            const int st = it % kDecStages;
            if (!mbar_wait_warp(&sm.full[st], (it / kDecStages) & 1, abort, p.status)) break;
            const uint8_t* kt = &sm.kv[st][0][0][0];
            const uint8_t* vt = &sm.kv[st][1][0][0];

            float sc[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int key = 16 * warp + (lane & 7) + ((lane >> 4) & 1) * 8;
                const int c16 = 2 * kk + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(smem_u32(kt + (c16 / 8) * kDecTile * 128 + sw128_off(key, c16 % 8)), b0,
                        b1, b2, b3);
                mma_bf16_16816(sc[0], qa[kk], b0, b1);
                mma_bf16_16816(sc[1], qa[kk], b2, b3);
            }
            // scale into the log2 domain and mask keys >= hi
            const int kb = lo + it * kDecTile + 16 * warp;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = kb + nt * 8 + 2 * t4 + (e & 1);
                    const float x = sc[nt][e] * p.scale_log2;
                    sc[nt][e] = key < hi ? x : -INFINITY;
                }
            // online softmax update per row (r = 0: row g, r = 1: row g + 8)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float mx = fmaxf(fmaxf(sc[0][2 * r], sc[0][2 * r + 1]),
                                 fmaxf(sc[1][2 * r], sc[1][2 * r + 1]));
                mx = shfl_xor_max(mx, 1);
                mx = shfl_xor_max(mx, 2);
                const float m_new = fmaxf(m_run[r], mx);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                const float corr = ex2(m_run[r] - m_use);
                m_run[r] = m_new;
                float ps = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
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
            uint32_t pa[4] = {pack_bf16(sc[0][0], sc[0][1]), pack_bf16(sc[0][2], sc[0][3]),
                              pack_bf16(sc[1][0], sc[1][1]), pack_bf16(sc[1][2], sc[1][3])};
            // keys of this warp beyond hi: zero their V entries (padding may hold anything)
            const int nvalid = hi - kb;
#pragma unroll
            for (int dn2 = 0; dn2 < D / 16; ++dn2) {
                const int key = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c16 = 2 * dn2 + (lane >> 4);
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(smem_u32(vt + (c16 / 8) * kDecTile * 128 + sw128_off(key, c16 % 8)), v0,
                          v1, v2, v3);
                if (nvalid < 16) {
                    const int k0 = 2 * t4, k1 = 2 * t4 + 8;
                    const uint32_t mlo0 = (k0 < nvalid ? 0x0000ffffu : 0u) |
                                          (k0 + 1 < nvalid ? 0xffff0000u : 0u);
                    const uint32_t mlo1 = (k1 < nvalid ? 0x0000ffffu : 0u) |
                                          (k1 + 1 < nvalid ? 0xffff0000u : 0u);
                    v0 &= mlo0;
                    v2 &= mlo0;
                    v1 &= mlo1;
                    v3 &= mlo1;
                }
                mma_bf16_16816(o[2 * dn2], pa, v0, v1);
                mma_bf16_16816(o[2 * dn2 + 1], pa, v2, v3);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[st]);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
            l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
        }
    }
    __syncthreads();
    // the combine grid may start launching now; it waits for this grid's
    // completion (griddepcontrol.wait) before reading any partial
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (*abort) {
        // Let every copy this CTA issued land before the CTA's shared memory
        // is released (bounded; the status word already holds the error).
        if (warp == kDecWarps && lane == 0) {
            volatile int never = 0;
            for (int st = 0; st < kDecStages; ++st) {
                int last = -1;
                for (int it = st; it < issued; it += kDecStages) last = it;
                if (last >= 0) mbar_wait(&sm.full[st], (last / kDecStages) & 1, &never, p.status);
            }
        }
        return;
    }

    // ---------------------------------------------- merge the warps' states
    float* mo = reinterpret_cast<float*>(&sm.kv[0][0][0][0]);   // [warps][16][D]
    float* mm = mo + kDecWarps * 16 * D;                         // [warps][16]
    float* ml = mm + kDecWarps * 16;                             // [warps][16]
    if (warp < kDecWarps) {
        const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
            const int c = dn * 8 + 2 * t4;
            *reinterpret_cast<float2*>(&mo[(warp * 16 + g) * D + c]) = make_float2(o[dn][0], o[dn][1]);
            *reinterpret_cast<float2*>(&mo[(warp * 16 + g + 8) * D + c]) =
                make_float2(o[dn][2], o[dn][3]);
        }
        if (t4 == 0) {
            mm[warp * 16 + g] = m_run[0];
            mm[warp * 16 + g + 8] = m_run[1];
            ml[warp * 16 + g] = l_run[0];
            ml[warp * 16 + g + 8] = l_run[1];
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nrows * D; i += blockDim.x) {
        const int r = i / D, c = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, mm[w * 16 + r]);
        float lsum = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
            const float wt = ex2(mm[w * 16 + r] - M);
            lsum += wt * ml[w * 16 + r];
            acc += wt * mo[(w * 16 + r) * D + c];
        }
        const size_t row = size_t(b) * p.Hq + h0 + r;
        p.O_part[(row * p.S + s) * D + c] = acc / lsum;
        if (c == 0) p.LSE_part[row * p.S + s] = (M + lg2(lsum)) * kLn2;
    }
}

// One CTA per (batch, query head); thread c owns output column c.
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ O_part,
                                                      const float* __restrict__ LSE_part, int S,
                                                      __nv_bfloat16* __restrict__ O,
                                                      float* __restrict__ LSE) {
    extern __shared__ float wts[];   // [S]
    __shared__ float red[4];
    // launched as a programmatic dependent of the decode: wait until that
    // grid has completed and its partials are visible (no-op otherwise)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t bh = blockIdx.x;
    const float* lp = LSE_part + bh * S;
    const int tid = threadIdx.x;

    float mx = -INFINITY;
    for (int s = tid; s < S; s += blockDim.x) mx = fmaxf(mx, lp[s]);
    for (int m = 16; m > 0; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();

    float sum = 0.f;
    for (int s = tid; s < S; s += blockDim.x) {
        const float l = lp[s];
        const float w = (mx == -INFINITY || l == -INFINITY) ? 0.f : ex2((l - mx) * kLog2e);
        wts[s] = w;
        sum += w;
    }
    for (int m = 16; m > 0; m >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, m);
    if ((tid & 31) == 0) red[tid >> 5] = sum;
    __syncthreads();
    sum = red[0] + red[1] + red[2] + red[3];

    if (tid < D) {
        const float* op = O_part + bh * S * D + tid;
        float acc = 0.f;
        for (int s = 0; s < S; ++s) {
            const float w = wts[s];
            if (w != 0.f) acc += w * op[size_t(s) * D];
        }
        O[bh * D + tid] = __float2bfloat16_rn(sum > 0.f ? acc / sum : 0.f);
    }
    if (tid == 0 && LSE) LSE[bh] = sum > 0.f ? mx + logf(sum) : -INFINITY;
}

template <int D>
static int launch_decode_d(const DecodeLaunch& L, cudaStream_t stream) {
    const size_t smem = sizeof(DecodeSmem<D>) + 1024;
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(decode_splitk_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem)) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set[dev] = true;
    }
    dim3 grid(L.p.S, L.p.Hkv * L.p.nrg, L.p.B);
    decode_splitk_kernel<D><<<grid, kDecThreads, smem, stream>>>(L.tmK, L.tmV, L.p);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int launch_decode(const DecodeLaunch& L, int d, cudaStream_t stream) {
    if (d == 64) return launch_decode_d<64>(L, stream);
    if (d == 128) return launch_decode_d<128>(L, stream);
    return ATTN_ERR_UNSUPPORTED;
}

int launch_combine(const float* O_part, const float* LSE_part, int B, int Hq, int S, int d,
                   void* O, float* LSE, cudaStream_t stream) {
    const size_t smem = size_t(S) * sizeof(float);
    if (smem > 48 * 1024) return ATTN_ERR_WORKSPACE;
    // programmatic stream serialisation: the combine's launch may overlap the
    // tail of a preceding decode grid (which signals launch_dependents)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(B) * unsigned(Hq));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    __nv_bfloat16* Ob = static_cast<__nv_bfloat16*>(O);
    cudaError_t e;
    if (d == 64)
        e = cudaLaunchKernelEx(&cfg, combine_kernel<64>, O_part, LSE_part, S, Ob, LSE);
    else if (d == 128)
        e = cudaLaunchKernelEx(&cfg, combine_kernel<128>, O_part, LSE_part, S, Ob, LSE);
    else
        return ATTN_ERR_UNSUPPORTED;
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn
