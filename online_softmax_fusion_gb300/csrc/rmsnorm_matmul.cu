// Fused RMSNorm + matrix product on the 5th-generation tensor cores:
//
//   O = ((X ⊙ G) W) / RMS(X),   RMS(X)_i = sqrt(mean_j X_ij^2 + eps)
//
// 第 11 讲 · 高级 ML 编译 (CMU 15-779) §3 describes the fusion: the division
// by RMS commutes with the product, so it moves after it, and the two
// reductions along the hidden dimension (sum of squares, and the product)
// run in the same loop with their partial sums kept on chip; the scalar tail
// (constant, square root, division) is element-wise work in registers.
//
// The sum of squares is the numerically stable one with the repair that
// Neptune论文浅读 (gentlecold.top) §4 derives for the L2 norm: each row keeps
// a reference 2^E above its largest |x| and the sum s of (x 2^-E)^2; when a
// tile raises E, s is repaired by 2^(2 (E_old - E_new)). With power-of-two
// references the scaling and the repair are exact, and no x^2 is formed, so
// inputs far beyond sqrt(FLT_MAX) keep a finite RMS. Across the K split the
// partial (E, s) of each CTA merge against the largest E (§6's pattern).
//
// Shapes: X [B, H] and O [B, D] row-major, G [H], W [H, D] row-major (O = Y W
// as the page writes it), all bf16. The product is computed transposed:
// O^T tile (128 output features x NB batch rows) = W^T tile x (X ⊙ G)^T, so
// the W tile is the 128-row A operand (MN-major straight from W's layout) and
// the batch is the MMA's N (16..256). That keeps the tensor core's M at 128
// for any batch, and W -- the large operand -- is streamed once.
//
// CTA roles (384 threads), two rings with their own depths:
//   warp 0      TMA of W: per 64-wide K step two 64 x 64 boxes (128-byte
//               swizzle) into the W ring
//   warp 2      TMA of X (64 x NB box) and a bulk copy of G's 64 entries into
//               the X ring
//   warp 1      TMEM allocation; tcgen05.mma issue (one elected lane)
//   warps 4-11  per K step: X -> X ⊙ G in place (bf16) and the repaired
//               sum of squares of X; after the loop, the epilogue
// W needs no conversion, so a W slot's round trip is load -> MMA -> free,
// and the W ring is deep; X slots are converted ahead of the MMA.
// Grid: (output-feature tiles of 128, batch tiles of NB, splits); the
// `splits` CTAs that share an output tile form one thread-block cluster and
// each reduces a contiguous range of K steps. Each CTA then pushes its fp32
// partial tile, slice by slice, and its (E, s) pairs into the other CTAs'
// shared memory (distributed shared memory stores); after one cluster
// barrier each CTA sums its slice of output features from its own shared
// memory, scales it and stores bf16.
//
// Two-pass form (large batch tiles): a conversion pass writes X ⊙ G and
// the whole rows' (E, s) to a workspace; the product kernel then loads the
// converted X straight into the MMA operand ring, its converter warps only
// turn the row statistics into scales while the product runs, and the
// epilogue exchanges partial tiles alone.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace attn {

namespace {

constexpr int kCvtWarp0 = 4;                  // warps 4.. convert and finish
// 8 converter warps (384 threads, two CTAs per SM) or 16 (640 threads, one
// CTA per SM; large batch tiles convert two or more K steps at once)
template <int CVT>
constexpr int rm_threads() { return (kCvtWarp0 + CVT) * 32; }
constexpr uint32_t kWBox = 64 * 128;          // 64 K rows x 64 features (128 B)
constexpr uint32_t kWStageBytes = 2 * kWBox;  // 128 features
constexpr int kEmptyExp = -1000;              // row exponent before any nonzero value
constexpr int kMinExp = -100;                 // references below 2^-100 are raised to it

struct RmsSmem {
    uint64_t wfull[kRmsMaxWStages];   // W tile landed
    uint64_t wempty[kRmsMaxWStages];  // MMAs that read the W slot completed
    uint64_t xfull[kRmsMaxXStages];   // X tile and G chunk landed
    uint64_t xready[kRmsMaxXStages];  // X ⊙ G written (one arrive per converter warp)
    uint64_t xempty[kRmsMaxXStages];  // MMAs that read the X slot completed
    uint64_t acc_full;                // every MMA of this CTA completed
    uint32_t tmem_base;
    int abort;
    alignas(128) uint16_t gbuf[kRmsMaxXStages][64];  // G chunk of each X slot
    int part_e[512];                  // per converter group: partial (E, s) per batch row
    float part_s[512];
    int row_e[256];                   // this CTA's partial (E, s) per batch row
    float row_s[256];
    float row_p[256];                 // 2^-E of the merged row
    float row_c[256];                 // 1 / sqrt(s / H + eps 2^-2E) of the merged row
};

// Untiled bulk copy global -> shared (16-byte aligned, size a multiple of 16),
// completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Barrier over the converter warps only (named barrier 1).
template <int CVT>
__device__ __forceinline__ void converter_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(CVT * 32) : "memory");
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    __nv_bfloat162 r = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&a),
                               *reinterpret_cast<const __nv_bfloat162*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// Per 16-bit half: max(|a|, |b|) (the sign bit is the XOR of the inputs' and
// is cleared by the caller).
__device__ __forceinline__ uint32_t bf16x2_maxabs(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 2^k for k <= 127 (exact), 0 below the normal range: the repair's factor
// 2^(2 (E_part - E_max)) only shrinks, and a part that small next to the
// largest one (whose scaled sum is >= 1/4) is below fp32 resolution anyway.
__device__ __forceinline__ float pow2i(int k) {
    return k < -126 ? 0.f : __int_as_float((127 + min(k, 127)) << 23);
}

// The scalar tail for references far from 1 (|E| > 40), in fp64; kept out
// of line so that the common path's code stays short.
__device__ __noinline__ void row_scale_wide(int em, float t, float eps, float* cf, float* rms) {
    const double td = double(t);
    *cf = float(1.0 / sqrt(td + ldexp(double(eps), -2 * em)));
    *rms = float(sqrt(ldexp(td, 2 * em) + double(eps)));
}

// The scalar tail of one row from its merged (E, s): O = acc * pf * cf with
// pf = 2^-E and cf = 1 / sqrt(s / H + eps 2^-2E); rms = sqrt(s 2^2E / H + eps).
__device__ __forceinline__ void row_scale(int em, float ss, int H, float eps, float& pf, float& cf,
                                          float& rms) {
    pf = 0.f;
    cf = 0.f;
    rms = sqrtf(eps);
    if (ss > 0.f) {
        const float t = ss / float(H);
        pf = ldexpf(1.f, -em);      // subnormal for E > 126 (inputs near the bf16 maximum)
        if (em >= -40 && em <= 40) {
            cf = rsqrtf(t + eps * pow2i(-2 * em));
            rms = sqrtf(t * pow2i(2 * em) + eps);
        } else {
            row_scale_wide(em, t, eps, &cf, &rms);
        }
    }
}

// sum of (x * sc)^2 over the two bf16 values of a word
__device__ __forceinline__ float sq2(uint32_t w, float sc, float acc) {
    const float lo = __uint_as_float(w << 16) * sc;
    const float hi = __uint_as_float(w & 0xffff0000u) * sc;
    return fmaf(hi, hi, fmaf(lo, lo, acc));
}

}  // namespace

// A converter group of cvt_warps = ceil(NB / 32) warps handles one K step
// (one thread per batch row); cvt_groups groups take the K steps in turn, so
// several steps are converted at once.
template <int CVT>
__global__ void __launch_bounds__(rm_threads<CVT>(), CVT == 8 ? 2 : 1)
    rmsnorm_matmul_kernel(const __grid_constant__ CUtensorMap tmX,
                          const __grid_constant__ CUtensorMap tmW, RmsParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ RmsSmem sm;
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int NB = p.NB;
    const int NW = p.w_stages;
    const int NX = p.x_stages;
    const uint32_t xbytes = uint32_t(NB) * 128u;
    uint8_t* wring = ring;
    uint8_t* xring = ring + size_t(NW) * kWStageBytes;
    const int n0 = blockIdx.x * 128;
    const int b0 = blockIdx.y * NB;
    const uint32_t rank = cluster_rank();
    const int S = p.splits;
    // k_tiles * S < 2^31 (the host bounds H): 32-bit division
    const int kt0 = int(rank) * p.k_tiles / S;
    const int kt1 = (int(rank) + 1) * p.k_tiles / S;
    const int nk = kt1 - kt0;
    uint32_t ncols = 32;
    while (ncols < uint32_t(NB)) ncols <<= 1;

    auto issue_w = [&](int i) {
        const int s = i % NW;
        uint8_t* st = wring + size_t(s) * kWStageBytes;
        const int k = (kt0 + i) * 64;
        mbar_arrive_expect_tx(&sm.wfull[s], kWStageBytes);
        tma_load_3d(st, &tmW, &sm.wfull[s], n0, k, 0);
        tma_load_3d(st + kWBox, &tmW, &sm.wfull[s], n0 + 64, k, 0);
    };
    auto issue_x = [&](int i) {
        const int s = i % NX;
        const int k = (kt0 + i) * 64;
        if (p.pre) {
            // X ⊙ G was formed by the conversion pass: the tile goes straight
            // to the product
            mbar_arrive_expect_tx(&sm.xfull[s], xbytes);
        } else {
            const uint32_t gbytes = uint32_t(min(64, p.H - k)) * 2u;
            mbar_arrive_expect_tx(&sm.xfull[s], xbytes + gbytes);
            bulk_load(sm.gbuf[s], p.G + k, gbytes, &sm.xfull[s]);
        }
        tma_load_3d(xring + size_t(s) * xbytes, &tmX, &sm.xfull[s], k, b0, 0);
    };
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
        for (int i = 0; i < NW; ++i) {
            mbar_init(&sm.wfull[i], 1);
            mbar_init(&sm.wempty[i], 1);
        }
        for (int i = 0; i < NX; ++i) {
            mbar_init(&sm.xfull[i], 1);
            mbar_init(&sm.xready[i], p.cvt_warps);
            mbar_init(&sm.xempty[i], 1);
        }
        mbar_init(&sm.acc_full, 1);
        sm.abort = 0;
        fence_mbar_init();
    }
    // the first fill of both rings goes out while TMEM is being allocated:
    // lanes 0.. of warp 0 issue W slots, lanes 16.. issue X slots
    const int w_first = min(NW, nk), x_first = min(NX, nk);
    if (p.chained && threadIdx.x == 0) {
        // the next call on the stream may start its own W stream now
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    if (warp == 0) {
        __syncwarp();
        if (lane < w_first) issue_w(lane);
        // chained: X (and G) may be written by the kernel before this one on
        // the stream, which may still run; W is not (the caller's promise)
        if (p.chained && lane >= 16) asm volatile("griddepcontrol.wait;" ::: "memory");
        if (lane >= 16 && lane - 16 < x_first) issue_x(lane - 16);
    }
    if (warp == 1) {
        tc::tmem_alloc(&sm.tmem_base, ncols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tacc = sm.tmem_base;
    volatile int* abort = &sm.abort;

    int w_issued = w_first, x_issued = x_first;   // loads issued (producer threads)
    if (warp == 0) {
        // ============================================== TMA producer of W
        if (lane == 0) {
            for (int i = NW; i < nk; ++i) {
                const int st = i % NW;
                if (!mbar_wait(&sm.wempty[st], ((i / NW) - 1) & 1, abort, p.status)) break;
                issue_w(i);
                w_issued = i + 1;
            }
        }
    } else if (warp == 2) {
        // ======================================== TMA producer of X and G
        if (lane == 0) {
            if (p.chained) asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int i = NX; i < nk; ++i) {
                const int st = i % NX;
                if (!mbar_wait(&sm.xempty[st], ((i / NX) - 1) & 1, abort, p.status)) break;
                issue_x(i);
                x_issued = i + 1;
            }
        }
    } else if (warp == 1) {
        // ================================================= MMA issuer
        const uint32_t idesc = tc::idesc_bf16_ab(128, NB, 1, 0);
        const uint64_t a0 = tc::sdesc_sw128(smem_u32(wring), kWBox, 1024);
        const uint64_t b0d = tc::sdesc_sw128(smem_u32(xring), 16, 1024);
        for (int i = 0; i < nk; ++i) {
            const int sw = i % NW, sx = i % NX;
            if (!mbar_wait_warp(p.pre ? &sm.xfull[sx] : &sm.xready[sx], (i / NX) & 1, abort,
                                p.status))
                break;
            if (!mbar_wait_warp(&sm.wfull[sw], (i / NW) & 1, abort, p.status)) break;
            tc::fence_after_sync();
            const uint64_t wo = uint64_t((uint32_t(sw) * kWStageBytes) >> 4);
            const uint64_t xo = uint64_t((uint32_t(sx) * xbytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc::mma_bf16_ss_warp(tacc, a0 + wo + uint64_t(kk * (2048 >> 4)),
                                     b0d + xo + uint64_t(kk * (32 >> 4)), idesc,
                                     (i | kk) != 0 ? 1u : 0u);
            tc::commit_warp(&sm.wempty[sw]);
            tc::commit_warp(&sm.xempty[sx]);
        }
        // covers every MMA issued above (and arrives at once if none was)
        tc::commit_warp(&sm.acc_full);
    } else if (warp >= kCvtWarp0) {
        // ================================== X ⊙ G and the sum of squares
        // One thread per batch row of the tile: the row's eight 16-byte chunks
        // sit in one 128-byte swizzled row, and eight consecutive rows put a
        // given chunk in eight different bank groups, so the loads are
        // conflict-free and the row reductions need no shuffles.
        // Group q converts the K steps of X slots s with s % ngroups == q
        // (ngroups divides the X ring depth), so each slot has one owner that
        // waits on the slot's phases in order: a parity wait is only
        // unambiguous one phase ahead of the barrier.
        const int cw = warp - kCvtWarp0;                // 0..7
        const int gw = p.cvt_warps;                     // warps per group
        const int ngroups = p.cvt_groups;
        const int grp = cw / gw;
        const int r = (cw % gw) * 32 + lane;            // batch row of the tile
        if (p.pre) {
            // the conversion pass gives (E, s) of whole rows: the row scales
            // are final while the product still runs, and nothing is merged
            if (p.chained) asm volatile("griddepcontrol.wait;" ::: "memory");
            for (int rr = cw * 32 + lane; rr < NB; rr += CVT * 32) {
                const bool in = b0 + rr < p.B;
                float pf, cf, rms;
                row_scale(in ? p.stats_e[b0 + rr] : kEmptyExp, in ? p.stats_s[b0 + rr] : 0.f,
                          p.H, p.eps, pf, cf, rms);
                sm.row_p[rr] = pf;
                sm.row_c[rr] = cf;
                if (p.rms && blockIdx.x == 0 && rank == 0 && in) p.rms[b0 + rr] = rms;
            }
        } else if (grp < ngroups) {
            int E = kEmptyExp;      // reference exponent: |x| < 2^E for every x seen
            float Ssum = 0.f;       // sum of (x 2^-E)^2
            float SC2 = 0.f;        // 2^-2E, set whenever E changes
            for (int i = grp; i < nk; i += ngroups) {
                const int s = i % NX;
                if (!mbar_wait_warp(&sm.xfull[s], (i / NX) & 1, abort, p.status)) break;
                if (r < NB) {
                    uint8_t* row = xring + size_t(s) * xbytes + r * 128;
                    const uint32_t sw = uint32_t(r) & 7u;
                    uint4 v[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        v[j] = *reinterpret_cast<const uint4*>(row + ((uint32_t(j) ^ sw) << 4));
                    // largest |x| of the row's 64 values (chunk j holds k = 8j .. 8j + 7)
                    uint32_t m4[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        m4[j] = bf16x2_maxabs(bf16x2_maxabs(v[j].x, v[j].y),
                                              bf16x2_maxabs(v[j].z, v[j].w));
                    uint32_t mm = bf16x2_maxabs(
                        bf16x2_maxabs(bf16x2_maxabs(m4[0], m4[1]), bf16x2_maxabs(m4[2], m4[3])),
                        bf16x2_maxabs(bf16x2_maxabs(m4[4], m4[5]), bf16x2_maxabs(m4[6], m4[7])));
                    mm &= 0x7fff7fffu;
                    const uint32_t mb = max(mm & 0xffffu, mm >> 16);
                    if (mb != 0u) {
                        // |x| < 2^(e_biased - 126) for every x of the tile row
                        const int et = max(int(mb >> 7) - 126, kMinExp);
                        if (et > E) {
                            Ssum = ldexpf(Ssum, 2 * (E - et));   // the repair
                            E = et;
                            SC2 = ldexpf(1.f, -2 * E);
                        }
                        if (et >= -60 && et <= 60) {
                            // squares of the tile neither overflow nor lose
                            // anything that matters: sum them unscaled, then
                            // rescale the tile's sum once
                            uint64_t a0 = 0, a1 = 0;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                                for (int h = 0; h < 4; h += 2) {
                                    const uint64_t p0 = f2_pack(__uint_as_float(w[h] << 16),
                                                                __uint_as_float(w[h] & 0xffff0000u));
                                    const uint64_t p1 =
                                        f2_pack(__uint_as_float(w[h + 1] << 16),
                                                __uint_as_float(w[h + 1] & 0xffff0000u));
                                    a0 = f2_fma(p0, p0, a0);
                                    a1 = f2_fma(p1, p1, a1);
                                }
                            }
                            float x0, x1, y0, y1;
                            f2_unpack(a0, x0, x1);
                            f2_unpack(a1, y0, y1);
                            Ssum = fmaf((x0 + x1) + (y0 + y1), SC2, Ssum);
                        } else {
                            const float sc = ldexpf(1.f, -E);
                            float a = Ssum;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                a = sq2(v[j].x, sc, a);
                                a = sq2(v[j].y, sc, a);
                                a = sq2(v[j].z, sc, a);
                                a = sq2(v[j].w, sc, a);
                            }
                            Ssum = a;
                        }
                    }
                    // X ⊙ G in place
                    const uint4* gv = reinterpret_cast<const uint4*>(sm.gbuf[s]);
                    const bool gfull = (kt0 + i) * 64 + 64 <= p.H;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint4 g = make_uint4(0u, 0u, 0u, 0u);
                        if (gfull || (kt0 + i) * 64 + j * 8 < p.H) g = gv[j];
                        uint4 x = v[j];
                        x.x = bf16x2_mul(x.x, g.x);
                        x.y = bf16x2_mul(x.y, g.y);
                        x.z = bf16x2_mul(x.z, g.z);
                        x.w = bf16x2_mul(x.w, g.w);
                        *reinterpret_cast<uint4*>(row + ((uint32_t(j) ^ sw) << 4)) = x;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.xready[s]);
            }
            if (r < NB) {
                sm.part_e[grp * NB + r] = E;
                sm.part_s[grp * NB + r] = Ssum;
            }
        }
        converter_sync<CVT>();
        // merge the groups (the split form of the repair, inside the CTA)
        for (int r = cw * 32 + lane; r < NB && !p.pre; r += CVT * 32) {
            int em = kEmptyExp;
            for (int q = 0; q < ngroups; ++q) em = max(em, sm.part_e[q * NB + r]);
            float ss = 0.f;
            for (int q = 0; q < ngroups; ++q)
                ss += sm.part_s[q * NB + r] * pow2i(2 * (sm.part_e[q * NB + r] - em));
            sm.row_e[r] = em;
            sm.row_s[r] = ss;
        }

        tc::fence_before_sync();
    }

    // ================================================================ epilogue
    // Each CTA pushes its fp32 partial tile, split into `S` slices of
    // 128 / S output features, into the slice owners' shared memory, and its
    // per-row (E, s) into every CTA's; after one cluster barrier every CTA
    // merges and reduces from its own shared memory only. The receive area
    // sits after the rings when it fits there; otherwise it reuses the rings,
    // and a first cluster barrier makes sure every CTA's rings are idle.
    __syncwarp();
    bool ok = true;
    if (warp >= kCvtWarp0) {
        ok = mbar_wait_warp(&sm.acc_full, 0, abort, p.status);
        tc::fence_after_sync();
    }
    __syncthreads();                          // this CTA's (E, s) rows are in sm.row_e / row_s
    if (!p.recv_separate) cluster_sync_all();
    const int wd = 128 / S;                   // output features per slice
    uint8_t* recv = ring + (p.recv_separate ? size_t(NW) * kWStageBytes + size_t(NX) * xbytes : 0);
    const uint32_t recv_a = smem_u32(recv);
    const uint32_t tile_bytes = uint32_t(NB) * 128u * 4u;           // [S][NB][wd] fp32
    const uint32_t e_off = tile_bytes;                               // [S][NB] int
    const uint32_t s_off = tile_bytes + uint32_t(S * NB) * 4u;       // [S][NB] fp32
    if (warp >= kCvtWarp0 && warp < kCvtWarp0 + 8 && ok) {
        const int q4 = warp & 3;                          // TMEM lanes 32 q4 ..
        const int half = (warp - kCvtWarp0) >> 2;         // column half
        const int n = q4 * 32 + lane;                     // output feature in the tile
        const int owner = n / wd;
        const uint32_t dst = map_rank(recv_a, uint32_t(owner)) +
                             uint32_t((int(rank) * NB * wd + (n - owner * wd)) * 4);
        const int c0 = half * (NB / 2);
        for (int cc = 0; cc < NB / 2; cc += 8) {
            uint32_t v[8];
            tc::tmem_ld_32x32b_x8(tacc + (uint32_t(q4 * 32) << 16) + uint32_t(c0 + cc), v);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                st_cluster_u32(dst + uint32_t((c0 + cc + j) * wd * 4), v[j]);
        }
    }
    for (int idx = threadIdx.x; idx < S * NB && !p.pre; idx += rm_threads<CVT>()) {
        const int q = idx / NB, r = idx - (idx / NB) * NB;
        const uint32_t o = uint32_t((int(rank) * NB + r) * 4);
        const uint32_t base = map_rank(recv_a, uint32_t(q));
        st_cluster_u32(base + e_off + o, uint32_t(sm.row_e[r]));
        st_cluster_u32(base + s_off + o, __float_as_uint(sm.row_s[r]));
    }
    tc::fence_before_sync();
    cluster_sync_all();   // every push of every CTA of the cluster has landed
    // chained: O and RMS may be read or written by the kernel before this
    // one on the stream; it has finished once this wait returns
    if (p.chained) asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- merge the per-row statistics of the cluster (local)
    const int* re = reinterpret_cast<const int*>(recv + e_off);
    const float* rs = reinterpret_cast<const float*>(recv + s_off);
    for (int r = threadIdx.x; r < NB && !p.pre; r += rm_threads<CVT>()) {
        int em = kEmptyExp;
        for (int q = 0; q < S; ++q) em = max(em, re[q * NB + r]);
        float ss = 0.f;
        for (int q = 0; q < S; ++q) ss += rs[q * NB + r] * pow2i(2 * (re[q * NB + r] - em));   // the repair
        float pf, cf, rms;
        row_scale(em, ss, p.H, p.eps, pf, cf, rms);
        sm.row_p[r] = pf;
        sm.row_c[r] = cf;
        if (p.rms && blockIdx.x == 0 && rank == 0 && b0 + r < p.B) p.rms[b0 + r] = rms;
    }
    __syncthreads();

    // ---- this CTA's slice of output features, summed over the cluster (local)
    {
        const int q4n = wd / 4;
        const int nlo = int(rank) * wd;
        const float* rt = reinterpret_cast<const float*>(recv);
        for (int u = threadIdx.x; u < NB * q4n; u += rm_threads<CVT>()) {
            const int r = u / q4n;
            const int nl = (u - r * q4n) * 4;
            float4 acc = *reinterpret_cast<const float4*>(rt + r * wd + nl);
            for (int q = 1; q < S; ++q) {
                const float4 v = *reinterpret_cast<const float4*>(rt + (q * NB + r) * wd + nl);
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            const int gb = b0 + r, gn = n0 + nlo + nl;
            if (gb < p.B && gn < p.D && !*abort) {
                const float pf = sm.row_p[r], cf = sm.row_c[r];
                uint2 w;
                w.x = pack_bf16(acc.x * pf * cf, acc.y * pf * cf);
                w.y = pack_bf16(acc.z * pf * cf, acc.w * pf * cf);
                *reinterpret_cast<uint2*>(p.O + size_t(gb) * p.D + gn) = w;
            }
        }
    }

    if (*abort && lane == 0 && (warp == 0 || warp == 2)) {
        // let this CTA's copies in flight land before its shared memory is released
        volatile int never = 0;
        const int nst = warp == 0 ? NW : NX;
        const int iss = warp == 0 ? w_issued : x_issued;
        uint64_t* full = warp == 0 ? sm.wfull : sm.xfull;
        for (int s = 0; s < nst; ++s) {
            int last = -1;
            for (int u = s; u < iss; u += nst) last = u;
            if (last >= 0) mbar_wait(&full[s], (last / nst) & 1, &never, p.status);
        }
    }
    if (warp == 1) {
        volatile int never = 0;
        mbar_wait(&sm.acc_full, 0, &never, p.status);
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tacc, ncols);
    }
}

// The conversion pass of the two-kernel form: X ⊙ G rounded to bf16 (the
// product's operand, the same rounding as the fused converter) and, per row,
// the reference exponent E (2^E above the row's largest |x|) and the sum s of
// (x 2^-E)^2 (exact power-of-two scaling: no square can overflow). One CTA
// of 256 threads per row (one warp per row on B / 8 CTAs measured ~10 us at
// batch 256, most of it before the product could start); the row is read
// twice, the second time from L1.
constexpr int kPrepThreads = 256;

__global__ void __launch_bounds__(kPrepThreads) rms_prep_kernel(
    const __nv_bfloat16* __restrict__ X, const __nv_bfloat16* __restrict__ G,
    __nv_bfloat16* __restrict__ Xg, int* __restrict__ e_out, float* __restrict__ s_out, int B,
    int H, int chained) {
    // the product kernel, launched as this kernel's dependent, may start
    // streaming W now; it waits for this grid before reading Xg or (E, s)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // chained: X may be written, and the workspace still read, by the kernel
    // before this one on the stream; it has finished once this returns
    if (chained) asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ uint32_t red_u[kPrepThreads / 32];
    __shared__ float red_f[kPrepThreads / 32];
    const int row = int(blockIdx.x);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const uint4* x = reinterpret_cast<const uint4*>(X + size_t(row) * H);
    const uint4* g = reinterpret_cast<const uint4*>(G);
    uint4* xg = reinterpret_cast<uint4*>(Xg + size_t(row) * H);
    const int nc = H / 8;
    uint32_t mm = 0u;
    for (int c = threadIdx.x; c < nc; c += kPrepThreads) {
        const uint4 v = x[c];
        mm = bf16x2_maxabs(mm, bf16x2_maxabs(bf16x2_maxabs(v.x, v.y), bf16x2_maxabs(v.z, v.w)));
    }
    mm &= 0x7fff7fffu;
    uint32_t mb = max(mm & 0xffffu, mm >> 16);
    for (int o = 16; o > 0; o >>= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    if (lane == 0) red_u[wid] = mb;
    __syncthreads();
    mb = red_u[0];
#pragma unroll
    for (int w = 1; w < kPrepThreads / 32; ++w) mb = max(mb, red_u[w]);
    const int E = mb != 0u ? max(int(mb >> 7) - 126, kMinExp) : kEmptyExp;
    const float sc = mb != 0u ? ldexpf(1.f, -E) : 0.f;
    float acc = 0.f;
    for (int c = threadIdx.x; c < nc; c += kPrepThreads) {
        uint4 v = x[c];
        acc = sq2(v.x, sc, acc);
        acc = sq2(v.y, sc, acc);
        acc = sq2(v.z, sc, acc);
        acc = sq2(v.w, sc, acc);
        const uint4 gg = g[c];
        v.x = bf16x2_mul(v.x, gg.x);
        v.y = bf16x2_mul(v.y, gg.y);
        v.z = bf16x2_mul(v.z, gg.z);
        v.w = bf16x2_mul(v.w, gg.w);
        xg[c] = v;
    }
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) red_f[wid] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = red_f[0];
#pragma unroll
        for (int w = 1; w < kPrepThreads / 32; ++w) t += red_f[w];
        e_out[row] = E;
        s_out[row] = t;
    }
}

int launch_rmsnorm_prep(const __nv_bfloat16* X, const __nv_bfloat16* G, __nv_bfloat16* Xg,
                        int* e_out, float* s_out, int B, int H, int chained,
                        cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(B));
    cfg.blockDim = dim3(kPrepThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = chained ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, rms_prep_kernel, X, G, Xg, e_out, s_out, B, H, chained) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

namespace {

constexpr int kMaxDev = 64;

size_t smem_bytes(const RmsParams& p) {
    const size_t rings = size_t(p.w_stages) * kWStageBytes + size_t(p.x_stages) * size_t(p.NB) * 128u;
    const size_t recv = size_t(p.NB) * 512u + size_t(8 * p.splits * p.NB);
    return (p.recv_separate ? rings + recv : std::max(rings, recv)) + 1024;
}

// Raises the kernel's dynamic shared-memory limit on the current device to at
// least `smem` (never lowers it).
template <int CVT>
bool ensure_smem_attr(int dev, size_t smem) {
    static size_t attr_set[kMaxDev] = {0};
    if (attr_set[dev] >= smem) return true;
    if (cudaFuncSetAttribute(rmsnorm_matmul_kernel<CVT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
        return false;
    attr_set[dev] = smem;
    return true;
}

template <int CVT>
int launch_t(const RmsLaunch& L, int dev, cudaStream_t stream) {
    const RmsParams& p = L.p;
    const size_t smem = smem_bytes(p);
    if (!ensure_smem_attr<CVT>(dev, smem)) return ATTN_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned((p.D + 127) / 128), unsigned((p.B + p.NB - 1) / p.NB),
                       unsigned(p.splits));
    cfg.blockDim = dim3(rm_threads<CVT>());
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = unsigned(p.splits);
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.chained ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, rmsnorm_matmul_kernel<CVT>, L.tmX, L.tmW, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
}

}  // namespace

int launch_rmsnorm_matmul(const RmsLaunch& L, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return ATTN_ERR_CUDA;
    if (L.p.cvt_all == 16) return launch_t<16>(L, dev, stream);
    if (L.p.cvt_all == 8) return launch_t<8>(L, dev, stream);
    return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
