// Attention backward, single pass per KV block (the FA3-style single-pass
// algorithm the Twill review (xllm-io) describes in §七 7.2: five GEMMs, one
// exp, and a global-memory atomic reduction for dQ).
//
// With P recomputed from the forward's log-sum-exp (P = exp(x - LSE)):
//   dV_j  = sum_i P_ij dO_i          dP_ij = dO_i . v_j
//   D_i   = dO_i . O_i               dS_ij = P_ij (dP_ij - D_i)
//   dQ_i  = s sum_j dS_ij k_j        dK_j  = s sum_i dS_ij q_i
//
// Kernels:
//   bwd_prep   : D_i = dO_i . O_i (fp32) and a zeroed fp32 dQ accumulator
//   bwd_main   : one CTA per (64-key block, KV head, batch); it keeps K, V of
//                its keys in shared memory and loops over the query heads of
//                the GQA group and the 64-row Q blocks that see its keys:
//                S^T = K Q^T, P^T, dP^T = V dO^T, dS^T, then dV += P^T dO and
//                dK += dS^T Q in registers, and dQ += dS K added to the fp32
//                accumulator with atomics. dK and dV of the block are complete
//                when the loop ends (no atomics for them).
//   bwd_convert: dQ = s * accumulator -> bf16
// Tensor cores through warp-level mma.sync (m16n8k16, bf16 in, fp32 acc).
#include "common.cuh"
#include "kernels.h"

namespace attn {

namespace {

constexpr int kBwdRows = 64;     // query rows per Q block
constexpr int kBwdKeys = 64;     // keys per CTA
constexpr int kBwdWarps = 4;     // warp w owns keys [16w, 16w + 16) of the block
constexpr int kBwdThreads = kBwdWarps * 32;

template <int D>
struct BwdSmem {
    alignas(1024) uint8_t k[D / 64][kBwdKeys * 128];
    alignas(1024) uint8_t v[D / 64][kBwdKeys * 128];
    alignas(1024) uint8_t q[D / 64][kBwdRows * 128];
    alignas(1024) uint8_t dout[D / 64][kBwdRows * 128];
    alignas(1024) uint8_t dst[kBwdKeys * 128];     // dS^T [key][row] bf16
    float lse2[kBwdRows];                          // LSE * log2(e), or -inf
    float dsum[kBwdRows];                          // D_i
};

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// 64 rows x D bf16 from a row-major [rows, D] matrix into the 128-byte
// swizzled layout [D/64 boxes][64 rows][128 B]; rows >= nvalid read as zero.
template <int D>
__device__ __forceinline__ void load_rows(uint8_t (*dst)[64 * 128], const __nv_bfloat16* src,
                                          int row0, int nvalid) {
    for (int i = threadIdx.x; i < 64 * (D / 8); i += blockDim.x) {
        const int r = i / (D / 8), c16 = i % (D / 8);
        const bool ok = r < nvalid;
        const __nv_bfloat16* g = src + size_t(ok ? row0 + r : row0) * D + c16 * 8;
        cp_async_16(smem_u32(&dst[c16 / 8][sw128_off(r, c16 % 8)]), g, ok);
    }
}

__global__ void __launch_bounds__(128) bwd_prep_kernel(const __nv_bfloat16* __restrict__ O,
                                                       const __nv_bfloat16* __restrict__ dO,
                                                       float* __restrict__ Dsum,
                                                       float* __restrict__ dQacc, long long rows,
                                                       int d) {
    const long long r = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const __nv_bfloat16* o = O + r * d;
    const __nv_bfloat16* g = dO + r * d;
    float acc = 0.f;
    for (int c = lane * 2; c < d; c += 64) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(o + c));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(g + c));
        acc += a.x * b.x + a.y * b.y;
        *reinterpret_cast<float2*>(dQacc + r * d + c) = make_float2(0.f, 0.f);
    }
    for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (lane == 0) Dsum[r] = acc;
}

__global__ void __launch_bounds__(256) bwd_convert_kernel(const float* __restrict__ dQacc,
                                                          __nv_bfloat16* __restrict__ dQ,
                                                          long long n2, float scale) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n2;
         i += (long long)gridDim.x * blockDim.x) {
        const float2 a = reinterpret_cast<const float2*>(dQacc)[i];
        reinterpret_cast<__nv_bfloat162*>(dQ)[i] = __floats2bfloat162_rn(a.x * scale, a.y * scale);
    }
}

template <int D, bool CAUSAL, bool ALIBI>
__global__ void __launch_bounds__(kBwdThreads) bwd_main_kernel(BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int k0 = blockIdx.x * kBwdKeys;
    const int kvh = blockIdx.y;
    const int b = blockIdx.z;
    const int off = p.Lk - p.Lq;
    const int kvalid = min(kBwdKeys, p.Lk - k0);

    const size_t kv_base = (size_t(b) * p.Hkv + kvh) * p.Lk;
    load_rows<D>(sm.k, p.K + kv_base * D, k0, kvalid);
    load_rows<D>(sm.v, p.V + kv_base * D, k0, kvalid);
    cp_async_wait_all();

    float dv[D / 8][4], dk[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) dv[i][e] = dk[i][e] = 0.f;

    // Q blocks that can see a key of this block (causal: aligned row >= k0)
    const int n_qb = (p.Lq + kBwdRows - 1) / kBwdRows;
    const int qb0 = CAUSAL ? max(0, k0 - off) / kBwdRows : 0;
    const int key_w = k0 + 16 * warp;   // first key of this warp

    for (int hg = 0; hg < p.G; ++hg) {
        const int h = kvh * p.G + hg;
        const size_t q_base = (size_t(b) * p.Hq + h) * p.Lq;
        const float slope_l2 = ALIBI ? p.slopes[h] * kLog2e : 0.f;
        for (int qb = qb0; qb < n_qb; ++qb) {
            const int q0 = qb * kBwdRows;
            const int qvalid = min(kBwdRows, p.Lq - q0);
            __syncthreads();   // previous block done with q / dout / dst
            load_rows<D>(sm.q, p.Q + q_base * D, q0, qvalid);
            load_rows<D>(sm.dout, p.dO + q_base * D, q0, qvalid);
            for (int r = threadIdx.x; r < kBwdRows; r += blockDim.x) {
                const bool ok = r < qvalid;
                const float l = ok ? p.LSE[q_base + q0 + r] : -INFINITY;
                sm.lse2[r] = l * kLog2e;
                sm.dsum[r] = ok ? p.Dsum[q_base + q0 + r] : 0.f;
            }
            cp_async_wait_all();
            __syncthreads();

            // ---- S^T = K Q^T and dP^T = V dO^T (16 keys x 64 rows per warp)
            float st[8][4], dpt[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) st[i][e] = dpt[i][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int ra = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int ca = 2 * kk + (lane >> 4);
                uint32_t ak[4], av[4];
                ldsm_x4(smem_u32(&sm.k[ca / 8][sw128_off(ra, ca % 8)]), ak[0], ak[1], ak[2], ak[3]);
                ldsm_x4(smem_u32(&sm.v[ca / 8][sw128_off(ra, ca % 8)]), av[0], av[1], av[2], av[3]);
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    const int rb = 16 * np + (lane & 7) + ((lane >> 4) & 1) * 8;
                    const int cb = 2 * kk + ((lane >> 3) & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(smem_u32(&sm.q[cb / 8][sw128_off(rb, cb % 8)]), b0, b1, b2, b3);
                    mma_bf16_16816(st[2 * np], ak, b0, b1);
                    mma_bf16_16816(st[2 * np + 1], ak, b2, b3);
                    ldsm_x4(smem_u32(&sm.dout[cb / 8][sw128_off(rb, cb % 8)]), b0, b1, b2, b3);
                    mma_bf16_16816(dpt[2 * np], av, b0, b1);
                    mma_bf16_16816(dpt[2 * np + 1], av, b2, b3);
                }
            }
            // ---- P^T = exp(x - LSE) (0 where masked), dS^T = P^T (dP^T - D)
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = key_w + g + 8 * (e >> 1);
                    const int rl = nt * 8 + 2 * t4 + (e & 1);
                    const int row = q0 + rl;
                    const float l2 = sm.lse2[rl];
                    float x = st[nt][e] * p.scale_log2;
                    if (ALIBI) x -= slope_l2 * fabsf(float(row + off - key));
                    const bool vis = key < p.Lk && row < p.Lq && l2 != -INFINITY &&
                                     !(CAUSAL && key > row + off);
                    const float pr = vis ? ex2(x - l2) : 0.f;
                    st[nt][e] = pr;
                    dpt[nt][e] = pr * (dpt[nt][e] - sm.dsum[rl]);
                }
            // ---- dV += P^T dO, dK += dS^T Q (K-steps over the 64 rows)
#pragma unroll
            for (int kr = 0; kr < 4; ++kr) {
                const uint32_t pa[4] = {
                    pack_bf16(st[2 * kr][0], st[2 * kr][1]), pack_bf16(st[2 * kr][2], st[2 * kr][3]),
                    pack_bf16(st[2 * kr + 1][0], st[2 * kr + 1][1]),
                    pack_bf16(st[2 * kr + 1][2], st[2 * kr + 1][3])};
                const uint32_t da[4] = {
                    pack_bf16(dpt[2 * kr][0], dpt[2 * kr][1]),
                    pack_bf16(dpt[2 * kr][2], dpt[2 * kr][3]),
                    pack_bf16(dpt[2 * kr + 1][0], dpt[2 * kr + 1][1]),
                    pack_bf16(dpt[2 * kr + 1][2], dpt[2 * kr + 1][3])};
#pragma unroll
                for (int dn2 = 0; dn2 < D / 16; ++dn2) {
                    const int rr = 16 * kr + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int cc = 2 * dn2 + (lane >> 4);
                    uint32_t x0, x1, x2, x3;
                    ldsm_x4_t(smem_u32(&sm.dout[cc / 8][sw128_off(rr, cc % 8)]), x0, x1, x2, x3);
                    mma_bf16_16816(dv[2 * dn2], pa, x0, x1);
                    mma_bf16_16816(dv[2 * dn2 + 1], pa, x2, x3);
                    ldsm_x4_t(smem_u32(&sm.q[cc / 8][sw128_off(rr, cc % 8)]), x0, x1, x2, x3);
                    mma_bf16_16816(dk[2 * dn2], da, x0, x1);
                    mma_bf16_16816(dk[2 * dn2 + 1], da, x2, x3);
                }
            }
            // ---- dS^T to shared memory (bf16) for dQ
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int r2 = 0; r2 < 2; ++r2) {
                    const int kl = 16 * warp + g + 8 * r2;
                    const int rl = nt * 8 + 2 * t4;
                    *reinterpret_cast<uint32_t*>(&sm.dst[sw128_off(kl, rl >> 3) + (rl & 7) * 2]) =
                        pack_bf16(dpt[nt][2 * r2], dpt[nt][2 * r2 + 1]);
                }
            __syncthreads();
            // ---- dQ rows [16w, 16w + 16) of the block += dS K, added to the
            //      fp32 accumulator
            float dq[D / 8][4];
#pragma unroll
            for (int i = 0; i < D / 8; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int ka = 16 * kk + (lane & 7) + ((lane >> 4) & 1) * 8;
                const int ch = 2 * warp + ((lane >> 3) & 1);
                uint32_t a[4];
                ldsm_x4_t(smem_u32(&sm.dst[sw128_off(ka, ch)]), a[0], a[1], a[2], a[3]);
#pragma unroll
                for (int dn2 = 0; dn2 < D / 16; ++dn2) {
                    const int kb = 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int cc = 2 * dn2 + (lane >> 4);
                    uint32_t x0, x1, x2, x3;
                    ldsm_x4_t(smem_u32(&sm.k[cc / 8][sw128_off(kb, cc % 8)]), x0, x1, x2, x3);
                    mma_bf16_16816(dq[2 * dn2], a, x0, x1);
                    mma_bf16_16816(dq[2 * dn2 + 1], a, x2, x3);
                }
            }
#pragma unroll
            for (int r2 = 0; r2 < 2; ++r2) {
                const int row = q0 + 16 * warp + g + 8 * r2;
                if (row < p.Lq) {
                    float* dst = p.dQacc + (q_base + row) * D + 2 * t4;
#pragma unroll
                    for (int dn = 0; dn < D / 8; ++dn)
                        atomicAdd(reinterpret_cast<float2*>(dst + dn * 8),
                                  make_float2(dq[dn][2 * r2], dq[dn][2 * r2 + 1]));
                }
            }
        }
    }
    // ---- dK (times the scale) and dV of this block's keys
#pragma unroll
    for (int r2 = 0; r2 < 2; ++r2) {
        const int key = key_w + g + 8 * r2;
        if (key < p.Lk) {
            __nv_bfloat16* dkr = p.dK + (kv_base + key) * D + 2 * t4;
            __nv_bfloat16* dvr = p.dV + (kv_base + key) * D + 2 * t4;
#pragma unroll
            for (int dn = 0; dn < D / 8; ++dn) {
                *reinterpret_cast<__nv_bfloat162*>(dkr + dn * 8) = __floats2bfloat162_rn(
                    dk[dn][2 * r2] * p.scale, dk[dn][2 * r2 + 1] * p.scale);
                *reinterpret_cast<__nv_bfloat162*>(dvr + dn * 8) =
                    __floats2bfloat162_rn(dv[dn][2 * r2], dv[dn][2 * r2 + 1]);
            }
        }
    }
}

template <int D, bool CAUSAL, bool ALIBI>
int launch_main_t(const BwdParams& p, cudaStream_t stream) {
    const size_t smem = sizeof(BwdSmem<D>) + 1024;
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(bwd_main_kernel<D, CAUSAL, ALIBI>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem)) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attr_set[dev] = true;
    }
    dim3 grid((p.Lk + kBwdKeys - 1) / kBwdKeys, p.Hkv, p.B);
    bwd_main_kernel<D, CAUSAL, ALIBI><<<grid, kBwdThreads, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int D>
int launch_main_d(const BwdParams& p, cudaStream_t stream) {
    const bool alibi = p.slopes != nullptr;
    if (p.causal)
        return alibi ? launch_main_t<D, true, true>(p, stream) : launch_main_t<D, true, false>(p, stream);
    return alibi ? launch_main_t<D, false, true>(p, stream) : launch_main_t<D, false, false>(p, stream);
}

}  // namespace

int launch_backward_prep(const BwdParams& p, int d, cudaStream_t stream) {
    const long long rows = (long long)p.B * p.Hq * p.Lq;
    bwd_prep_kernel<<<unsigned((rows + 3) / 4), 128, 0, stream>>>(p.O, p.dO, p.Dsum, p.dQacc, rows,
                                                                  d);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int launch_backward_convert(const BwdParams& p, int d, cudaStream_t stream) {
    const long long n2 = (long long)p.B * p.Hq * p.Lq * d / 2;
    const long long want = (n2 + 255) / 256;
    const unsigned blocks = unsigned(want < 152LL * 32 ? want : 152LL * 32);
    bwd_convert_kernel<<<blocks, 256, 0, stream>>>(p.dQacc, p.dQ, n2, p.scale);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int launch_backward(const BwdParams& p, int d, cudaStream_t stream) {
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    int st = launch_backward_prep(p, d, stream);
    if (st) return st;
    st = d == 64 ? launch_main_d<64>(p, stream) : launch_main_d<128>(p, stream);
    if (st) return st;
    return launch_backward_convert(p, d, stream);
}

}  // namespace attn
