// Launch descriptors shared between the C-ABI layer (api.cu) and the kernel
// translation units. Host-side only types plus the plain parameter structs
// passed by value to the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace attn {

struct DecodeParams {
    const __nv_bfloat16* Q;   // [B, Hq, d]
    const int* kv_lens;       // [B] or nullptr
    float* O_part;            // [B, Hq, S, d]
    float* LSE_part;          // [B, Hq, S]
    int B, Hq, Hkv, Lk_max;
    int S;                    // splits
    int C;                    // keys per split (multiple of 64)
    int G;                    // query heads per KV head
    int rows;                 // query heads per CTA (<= 16)
    int nrg;                  // CTAs per KV head along the heads (ceil(G / rows))
    float scale_log2;         // softmax scale * log2(e)
    int* status;              // device status word
};

struct DecodeLaunch {
    CUtensorMap tmK;          // K as (d, Lk_max, B*Hkv), box (64, 64, 1), 128 B swizzle
    CUtensorMap tmV;
    DecodeParams p;
};

struct PrefillParams {
    __nv_bfloat16* O;         // [B, Hq, Lq, d]
    float* LSE;               // [B, Hq, Lq] or nullptr
    const float* slopes;      // [Hq] or nullptr (ALiBi)
    int B, Hq, Hkv, Lq, Lk, G;
    float scale_log2;         // softmax scale * log2(e)
    int causal;
    float softcap;            // > 0: scores -> softcap * tanh(score / softcap)
    int window_left;          // >= 0: keys before i' - window_left are masked
    int window_right;         // >= 0: keys after i' + window_right are masked
    int pair_heads;           // tcgen05 kernel: a CTA's two Q tiles are two query
                              // heads of one KV group (1) or two row blocks (0)
    int splits;               // > 1 (tcgen05 kernel): split-KV, grid z = split,
    float* O_part;            //   fp32 partials [B, Hq, Lq, splits, d] instead of O
    float* LSE_part;          //   and [B, Hq, Lq, splits] instead of LSE
    int* status;
    unsigned long long wait_ns;   // tcgen05 kernel: time limit of every device wait
                                  // (0 = the library default)
    int selftest_skip;        // failure-detection self-test only (0 = off): the first
                              // CTA's producer stops before K/V ring entry selftest_skip - 1
};

struct PrefillLaunch {
    CUtensorMap tmQ;          // Q as (d, Lq, B*Hq), box (64, BM, 1), 128 B swizzle
    CUtensorMap tmK;          // K as (d, Lk, B*Hkv), box (64, BN, 1)
    CUtensorMap tmV;
    CUtensorMap tmO;          // O as (d, Lq, B*Hq), box (64, 32, 1): one softmax warp's rows
    PrefillParams p;
};

struct BwdParams {
    const __nv_bfloat16 *Q, *K, *V, *O, *dO;   // forward tensors and dO (layouts as forward)
    const float* LSE;                         // [B, Hq, Lq] natural-log LSE of the forward
    __nv_bfloat16 *dQ, *dK, *dV;              // gradients (dK, dV per KV head)
    float* dQacc;                             // fp32 [B, Hq, Lq, d] accumulator (workspace)
    float* Dsum;                              // fp32 [B, Hq, Lq] rowsum(dO * O) (workspace)
    const float* slopes;                      // [Hq] or nullptr (ALiBi)
    int B, Hq, Hkv, Lq, Lk, G;
    float scale, scale_log2;
    int causal;
    int* status;                              // device status word (tcgen05 form)
};

int launch_backward(const BwdParams& p, int d, cudaStream_t stream);   // mma.sync form
// The pieces around the main kernel: D and a zeroed dQ accumulator; dQ from
// the accumulator.
int launch_backward_prep(const BwdParams& p, int d, cudaStream_t stream);
int launch_backward_convert(const BwdParams& p, int d, cudaStream_t stream);

// tcgen05 backward main kernel (head dim 128): Q / dO maps with 64-row boxes,
// K / V maps with 128-row boxes (bf16, 128-byte swizzle), and the fp32 dQ
// accumulator [B * Hq, Lq, 128] with a (128, 64) box, no swizzle.
struct BwdTcLaunch {
    CUtensorMap tmQ, tmK, tmV, tmdO;
    BwdParams p;
};
int launch_backward_tc_main(const BwdTcLaunch& L, cudaStream_t stream);

int launch_decode(const DecodeLaunch& L, int d, cudaStream_t stream);
int launch_combine(const float* O_part, const float* LSE_part, int B, int Hq, int S, int d,
                   void* O, float* LSE, cudaStream_t stream);

// Register-tile (mma.sync) prefill: Q tile rows and K/V tile keys it expects
// in the tensor-map boxes.
constexpr int kMmaBM = 128;
constexpr int kMmaBN = 64;
int launch_prefill_mma(const PrefillLaunch& L, int d, cudaStream_t stream);

// tcgen05 prefill: box rows for Q and K/V.
constexpr int kTcBM = 128;
constexpr int kTcBN = 128;
int launch_prefill_tc(const PrefillLaunch& L, int d, cudaStream_t stream);    // 2 Q tiles / CTA
int launch_prefill_tc1(const PrefillLaunch& L, int d, cudaStream_t stream);   // 1 Q tile / CTA

// Fused RMSNorm + matrix product: X [B, H], G [H], W [H, D] -> O [B, D].
struct RmsParams {
    __nv_bfloat16* O;                         // [B, D]
    float* rms;                               // [B] or nullptr
    const __nv_bfloat16* G;                   // [H]
    int B, H, D;
    int NB;                                   // batch rows per CTA (multiple of 16, <= 256)
    int splits;                               // CTAs of a cluster sharing one output tile (K split)
    int k_tiles;                              // ceil(H / 64)
    int w_stages;                             // W ring depth
    int x_stages;                             // X ring depth
    int cvt_all;                              // converter warps of the launch: 8 or 16
    int cvt_warps;                            // converter warps per K step (<= 8)
    int cvt_groups;                           // groups taking K steps in turn; divides x_stages
    int recv_separate;                        // the epilogue's receive area follows the rings
    int pre;                                  // X arrives as X ⊙ G (workspace) with each row's
    const int* stats_e;                       //   reference exponent E and sum s of (x 2^-E)^2
    const float* stats_s;                     //   from the conversion pass: no converter work
    int chained;                              // launched as a programmatic dependent of the
                                              // kernel before it: W streams in at once, X and
                                              // the outputs wait for that kernel
    float eps;
    int* status;
};

struct RmsLaunch {
    CUtensorMap tmX, tmW;
    RmsParams p;
};

constexpr int kRmsMaxWStages = 12;
constexpr int kRmsMaxXStages = 8;
int launch_rmsnorm_matmul(const RmsLaunch& L, cudaStream_t stream);
// The conversion pass: Xg = X ⊙ G (bf16) and per row (E, s), one CTA per row;
// chained: launched as a programmatic dependent of the kernel before it.
int launch_rmsnorm_prep(const __nv_bfloat16* X, const __nv_bfloat16* G, __nv_bfloat16* Xg,
                        int* e_out, float* s_out, int B, int H, int chained,
                        cudaStream_t stream);

}  // namespace attn
