/*
 * attn.h - C ABI of the fused online-softmax attention library (libattn.so).
 *
 * The library computes O = softmax(s * Q K^T + bias + mask) V in one pass over
 * the keys, keeping a running row max m, a running sum l and an output
 * accumulator that is rescaled by exp(m_old - m_new) whenever the max grows
 * (the repaired online softmax of Neptune论文浅读 (gentlecold.top) §3-§4).
 * Two forms are exposed:
 *   - prefill, the Rolling Update form (same page, §5): one kernel streams
 *     K/V tiles past resident Q tiles;
 *   - decode, the Split-K Update form (same page, §6): the key axis is split
 *     into independent local reductions whose partial results are merged by
 *     a separate combine call that repairs them with the global max.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers of the current CUDA device,
 *     except the host buffers of attn_prefill_host.
 *   - bf16 tensors are row-major and contiguous, innermost dimension last:
 *       Q [B, Hq, Lq, d]   K, V [B, Hkv, Lk, d]   O [B, Hq, Lq, d]
 *     LSE is fp32 [B, Hq, Lq] and holds the natural-log log-sum-exp of each
 *     row's scaled, biased, masked scores (m + ln l).
 *   - GQA: query head h reads KV head h / (Hq / Hkv) (consecutive groups; the
 *     stacked-heads layout of CMU 15-779 第 11 讲 §7.1). Hq must be a
 *     multiple of Hkv.
 *   - Ownership: the caller allocates and owns every buffer. The library
 *     allocates no device or host memory, never frees, and never
 *     synchronises except inside attn_device_status(). (attn_prefill_host
 *     creates two copy streams and a ring of events per device on first
 *     use and keeps them.)
 *   - Streams: every launch is asynchronous on the given stream
 *     (cudaStream_t passed as void*, NULL = legacy default stream).
 *   - Errors: arguments are validated before anything is launched; an
 *     invalid call launches nothing and returns a non-zero attn_status.
 *     A launch failure returns ATTN_ERR_CUDA. Kernels never trap: a device
 *     wait that exceeds its time limit records ATTN_ERR_TIMEOUT in a device
 *     status word and the kernel returns; attn_device_status() reads it.
 *   - Supported head dims: d in {64, 128}. Pointers must be 16-byte aligned.
 *   - Device lifetime: the library looks up the device addresses of its own
 *     __device__ variables (the status word, the no-alloc decode's array)
 *     once per device and keeps them. Do not call it on a device again after
 *     cudaDeviceReset of that device in the same process.
 */
#ifndef ATTN_H
#define ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_NULL = 1,          /* a required pointer is NULL               */
    ATTN_ERR_SHAPE = 2,         /* a size is <= 0, or Hq % Hkv != 0, ...    */
    ATTN_ERR_UNSUPPORTED = 3,   /* head dim or implementation not built     */
    ATTN_ERR_WORKSPACE = 4,     /* split count out of range                  */
    ATTN_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed         */
    ATTN_ERR_TIMEOUT = 6,       /* a device wait hit its time limit          */
    ATTN_ERR_ALIGN = 7,         /* pointer not 16-byte aligned               */
    ATTN_ERR_VALUE = 8          /* scale not finite, or similar              */
} attn_status;

/* Prefill implementations selectable through attn_prefill_ex. */
enum {
    ATTN_IMPL_AUTO = 0,         /* the fastest built kernel for the shape    */
    ATTN_IMPL_TCGEN05 = 1,      /* warp-specialised tcgen05/TMEM/TMA kernel,
                                   two Q tiles per CTA, one CTA per SM       */
    ATTN_IMPL_MMA_SYNC = 2,     /* register-tile mma.sync kernel             */
    ATTN_IMPL_TCGEN05_1TILE = 3 /* the tcgen05 kernel with one Q tile per
                                   CTA and two CTAs per SM                   */
};

/*
 * attn_prefill - fused attention forward, Rolling Update form.
 *
 * Defines: the attention chain QK^T -> score/mask/bias -> softmax -> .V of
 * Neptune论文浅读 §2, fused along the key axis as in its §5 and in the
 * three-level loop of the CANN FlashAttention blog (ai6s.net), section
 * "ops-transformer在昇腾NPU上的工程处理": an outer loop over Q blocks, an
 * inner loop over K/V blocks with the online softmax state updated per block.
 *
 *   Q      bf16 [B, Hq, Lq, d]      (device, read)
 *   K, V   bf16 [B, Hkv, Lk, d]     (device, read)
 *   O      bf16 [B, Hq, Lq, d]      (device, written; rounded to nearest even)
 *   LSE    fp32 [B, Hq, Lq] or NULL (device, written when non-NULL)
 *   causal non-zero: query row i sees keys j <= i + (Lk - Lq) (bottom-right
 *          aligned); rows that see no key get O = 0, LSE = -inf.
 *   scale  softmax scale s applied to Q K^T (must be finite).
 *   alibi_slopes  NULL, or fp32 [Hq] on the device: adds
 *          -slope[h] * |i + (Lk - Lq) - j| to the scaled score (not scaled).
 *   stream cudaStream_t.
 * Returns ATTN_OK or an attn_status error code.
 */
int attn_prefill(const void* Q, const void* K, const void* V,
                 void* O, float* LSE,
                 int B, int Hq, int Hkv, int Lq, int Lk, int d,
                 int causal, float scale, const float* alibi_slopes,
                 void* stream);

/* As attn_prefill, with an explicit implementation (ATTN_IMPL_*).
 * Returns ATTN_ERR_UNSUPPORTED when that implementation cannot run the shape. */
int attn_prefill_ex(const void* Q, const void* K, const void* V,
                    void* O, float* LSE,
                    int B, int Hq, int Hkv, int Lq, int Lk, int d,
                    int causal, float scale, const float* alibi_slopes,
                    int impl, void* stream);

/*
 * Options of attn_prefill_opts: the attention variants Neptune论文浅读 §9
 * evaluates (Global, Causal, ALiBi, GQA, SoftCap, Window). The page names
 * SoftCap and Window without defining them; this library reads them as:
 *   softcap > 0  the scaled score x becomes softcap * tanh(x / softcap)
 *                (before the ALiBi bias and the masks); 0 = off;
 *   window_left  >= 0: query row i sees no key j < i' - window_left;
 *   window_right >= 0: query row i sees no key j > i' + window_right;
 *                < 0 = unlimited; i' = i + (Lk - Lq) as for the causal mask.
 * KV tiles wholly outside a window are skipped, not just masked.
 */
typedef struct {
    int causal;                  /* as attn_prefill                          */
    float scale;                 /* softmax scale (finite)                   */
    const float* alibi_slopes;   /* NULL or device fp32 [Hq]                 */
    float softcap;               /* >= 0, finite; 0 = off                    */
    int window_left;             /* < 0 = unlimited                          */
    int window_right;            /* < 0 = unlimited                          */
    int impl;                    /* ATTN_IMPL_*; softcap / window need the
                                    tcgen05 kernel (mma.sync: UNSUPPORTED)  */
} attn_prefill_options;

/* attn_prefill with the variants above (same tensors and layouts). */
int attn_prefill_opts(const void* Q, const void* K, const void* V,
                      void* O, float* LSE,
                      int B, int Hq, int Hkv, int Lq, int Lk, int d,
                      const attn_prefill_options* opts, void* stream);

/*
 * attn_prefill_host - attn_prefill_opts on HOST buffers, with the copies
 * pipelined against the kernels. The problem is cut into chunks of KV-head
 * units (one KV head and its Hq/Hkv query heads), contiguous in the
 * [B, H, L, d] layouts; a chunk is either part of one batch item's heads or
 * whole batch items. Per chunk: Q, K, V are copied host -> device on a copy
 * stream of the library, the fused prefill runs on `stream` once they have
 * landed, and O, LSE are copied device -> host on a second copy stream. The
 * stages of consecutive chunks overlap.
 *
 *   Qh, Kh, Vh  bf16 host [B,Hq,Lq,d] / [B,Hkv,Lk,d]           (read)
 *   Oh          bf16 host [B,Hq,Lq,d]                          (written)
 *   LSEh        fp32 host [B,Hq,Lq], or NULL                   (written)
 *               Page-locked host memory lets the copies overlap; with
 *               pageable memory the result is the same, the copies are not
 *               asynchronous.
 *   opts        as attn_prefill_opts (alibi_slopes stays a DEVICE pointer).
 *   chunk_kv_heads  KV-head units per chunk; <= 0: automatic (about 8
 *               chunks); values above Hkv are rounded up to whole batch items.
 *               attn_prefill_host_chunks() gives the resulting chunk count.
 *   workspace   device, attn_prefill_host_workspace_bytes() bytes, 16-byte
 *               aligned, owned by the caller: device copies of Q, K, V, O,
 *               LSE (each region 256-byte aligned).
 *
 * Asynchronous: the call queues everything and returns; the host buffers
 * must stay valid (and the inputs unchanged) until `stream` has passed this
 * call, and O / LSE are complete once it has. Work queued on `stream` before
 * the call finishes before the first copy starts; work queued after it starts
 * after the last copy. Errors: as attn_prefill_opts, all checked before any
 * copy is queued, plus ATTN_ERR_WORKSPACE for a short workspace.
 */
size_t attn_prefill_host_workspace_bytes(int B, int Hq, int Hkv, int Lq, int Lk, int d);
int attn_prefill_host_chunks(int B, int Hkv, int chunk_kv_heads);
int attn_prefill_host(const void* Qh, const void* Kh, const void* Vh, void* Oh, float* LSEh,
                      int B, int Hq, int Hkv, int Lq, int Lk, int d,
                      const attn_prefill_options* opts, int chunk_kv_heads,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_backward - gradients of attn_prefill (causal / ALiBi / GQA variants).
 *
 * The single-pass backward the Twill review (xllm-io) describes in §七 7.2:
 * per K/V block, recompute P = exp(x - LSE) from the forward's LSE, then
 *   dV = P^T dO,  dP = dO V^T,  dS = P (dP - rowsum(dO * O)),
 *   dQ = s dS K (accumulated across K/V blocks with fp32 atomics),
 *   dK = s dS^T Q;  dK and dV are summed over the query heads of a GQA group.
 *
 *   Q, O, dO bf16 [B, Hq, Lq, d]; K, V bf16 [B, Hkv, Lk, d]   (device, read)
 *   LSE      fp32 [B, Hq, Lq] from attn_prefill               (device, read)
 *   dQ       bf16 [B, Hq, Lq, d]; dK, dV bf16 [B, Hkv, Lk, d] (device, written)
 *   causal, scale, alibi_slopes as in attn_prefill (softcap / window: not
 *            supported here).
 *   workspace  device scratch of attn_backward_workspace_bytes(B, Hq, Lq, d)
 *            bytes, 16-byte aligned, owned by the caller (fp32 dQ accumulator
 *            and the row sums); its contents on entry do not matter.
 */
size_t attn_backward_workspace_bytes(int B, int Hq, int Lq, int d);

int attn_backward(const void* Q, const void* K, const void* V,
                  const void* O, const void* dO, const float* LSE,
                  void* dQ, void* dK, void* dV,
                  int B, int Hq, int Hkv, int Lq, int Lk, int d,
                  int causal, float scale, const float* alibi_slopes,
                  void* workspace, size_t workspace_bytes, void* stream);

/* attn_backward with the implementation chosen: ATTN_IMPL_TCGEN05 (head dim
 * 128 only: one CTA per 128-key block, the five products on tcgen05 with
 * S^T, dP^T, dQ^T, dV and dK in tensor memory, dQ added to the workspace
 * accumulator with fp32 atomics), ATTN_IMPL_MMA_SYNC (register-tile form,
 * head dims 64 and 128, dQ added with atomics), or ATTN_IMPL_AUTO (tcgen05
 * for head dim 128, else mma.sync). ATTN_ERR_UNSUPPORTED for any other impl
 * or for tcgen05 with head dim 64. attn_backward is this with AUTO. */
int attn_backward_ex(const void* Q, const void* K, const void* V,
                     const void* O, const void* dO, const float* LSE,
                     void* dQ, void* dK, void* dV,
                     int B, int Hq, int Hkv, int Lq, int Lk, int d,
                     int causal, float scale, const float* alibi_slopes,
                     void* workspace, size_t workspace_bytes, int impl, void* stream);

/*
 * attn_prefill_splitkv - the tcgen05 prefill with each CTA's KV range split
 * into num_splits chunks (grid z), each writing the split-K partials of
 * Neptune论文浅读 §6 (O_s = o / l in fp32 and LSE_s = m + ln l), merged by the
 * log-sum-exp combine of attn_combine with query rows in the role of heads.
 * For low-occupancy shapes (few rows x heads). Causal / ALiBi / GQA as in
 * attn_prefill; no softcap or window. num_splits 1 is attn_prefill itself;
 * 2..16 need a workspace of attn_prefill_splitkv_workspace_bytes() (fp32
 * [B, Hq, Lq, S, d] then [B, Hq, Lq, S], 16-byte aligned). ATTN_ERR_WORKSPACE
 * for num_splits outside 1..16 or a short workspace; other errors as
 * attn_prefill.
 */
size_t attn_prefill_splitkv_workspace_bytes(int B, int Hq, int Lq, int d, int num_splits);
int attn_prefill_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE,
                         int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal, float scale,
                         const float* alibi_slopes, int num_splits, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * attn_rmsnorm_matmul - RMSNorm followed by a matrix product, fused into one
 * kernel.
 *
 *   O = RMSNorm(X; G) W = ((X ⊙ G) W) / RMS(X),
 *   RMS(X)_i = sqrt( (1/H) sum_j X_ij^2 + eps )
 *
 * 第 11 讲 · 高级 ML 编译 (CMU 15-779) §3: the division by RMS commutes with
 * the product and moves after it, and the two reductions over the hidden
 * dimension (sum of squares, product) run in one loop. The sum of squares is
 * the numerically stable one (Neptune论文浅读 §4's repair for the L2 norm:
 * a running power-of-two reference above max |x| and the sum of the scaled
 * squares, repaired when the reference grows), so rows far beyond
 * sqrt(FLT_MAX) in magnitude keep a finite RMS.
 *
 *   X    bf16 [B, H] row-major                 (device, read)
 *   G    bf16 [H]                              (device, read)
 *   W    bf16 [H, D] row-major                 (device, read)
 *   O    bf16 [B, D] row-major                 (device, written)
 *   rms  fp32 [B] RMS(X) per row, or NULL      (device, written)
 *   eps  >= 0 and finite; the page's RMS has none (pass 0 for it)
 *   splits  CTAs that split the hidden dimension for one output tile and
 *           reduce through distributed shared memory (a thread-block
 *           cluster): 1, 2, 4 or 8, at most ceil(H / 64); 0 lets the library
 *           choose (attn_rmsnorm_matmul_splits).
 * A row whose RMS is 0 (all zeros, eps = 0) gives a zero output row.
 * Requirements: H and D multiples of 8 (16-byte row strides); X, G, W, O
 * 16-byte aligned. Errors: ATTN_ERR_NULL (X, G, W or O NULL), ATTN_ERR_SHAPE
 * (a size <= 0 or too large), ATTN_ERR_UNSUPPORTED (H or D not a multiple of
 * 8), ATTN_ERR_VALUE (eps negative or not finite, bad split count),
 * ATTN_ERR_ALIGN; nothing is launched then. Asynchronous on `stream`;
 * allocates nothing.
 */
int attn_rmsnorm_matmul(const void* X, const void* G, const void* W, void* O, float* rms,
                        int B, int H, int D, float eps, int splits, void* stream);

/* The same with the batch tile chosen by the caller: batch_tile rows of X per
 * CTA (a multiple of 16, at most 256; 0 = the library's choice, one tile when
 * B <= 256). Smaller tiles give more CTAs without a K split; larger tiles
 * stream W fewer times. ATTN_ERR_VALUE for any other batch_tile. */
int attn_rmsnorm_matmul_tiled(const void* X, const void* G, const void* W, void* O, float* rms,
                              int B, int H, int D, float eps, int batch_tile, int splits,
                              void* stream);

/*
 * attn_rmsnorm_matmul_chained - attn_rmsnorm_matmul for calls that follow one
 * another on a stream with constant weights (no counterpart in the pages: a
 * launch option of this library).
 *
 * The kernel is launched as a programmatic dependent of whatever kernel
 * precedes it on the stream: it may start while that kernel is finishing,
 * sets up and streams W at once, and waits for that kernel to complete
 * before it reads X or G and before it writes O or RMS. Back-to-back calls
 * (a stack of layers) thus overlap each call's start-up and first W tiles
 * with the end of the call before.
 *   Caller's promise: W is not written by the kernel that precedes this call
 *   on the stream (it may still be running when W is read). X, G, O and RMS
 *   carry no such restriction.
 * Arguments, results and errors as attn_rmsnorm_matmul (automatic batch tile
 * and K split).
 */
int attn_rmsnorm_matmul_chained(const void* X, const void* G, const void* W, void* O, float* rms,
                                int B, int H, int D, float eps, void* stream);

/*
 * attn_rmsnorm_matmul_ws - attn_rmsnorm_matmul with a workspace, which lets
 * large batches take a two-pass form (no counterpart in the pages: the same
 * operation, O = ((X ⊙ G) W) / RMS(X), split into two launches).
 *
 * Forms:
 *   ATTN_RMS_FORM_FUSED     the single kernel of attn_rmsnorm_matmul, which
 *                           converts X ⊙ G and sums squares inside the
 *                           product loop (workspace unused, may be NULL)
 *   ATTN_RMS_FORM_TWO_PASS  a conversion pass writes X ⊙ G (bf16) and each
 *                           row's repaired sum of squares (E, s) to the
 *                           workspace; the product kernel follows it as a
 *                           programmatic dependent and runs with no converter
 *                           stage. Same operands to the tensor core as the
 *                           fused form (X ⊙ G rounded to bf16 once); RMS may
 *                           differ from the fused form's in the last bits
 *                           (another summation order)
 *   ATTN_RMS_FORM_AUTO      the two-pass form (measured faster than the fused
 *                           kernel at batches 16 to 256 at H = D = 4096)
 *   workspace        device, >= attn_rmsnorm_matmul_ws_bytes(B, H) bytes,
 *                    16-byte aligned, caller-owned; contents are scratch
 * Other arguments, results and errors as attn_rmsnorm_matmul (automatic
 * batch tile and K split); ATTN_ERR_WORKSPACE if the workspace is too small,
 * ATTN_ERR_VALUE for an unknown form.
 */
enum { ATTN_RMS_FORM_AUTO = 0, ATTN_RMS_FORM_FUSED = 1, ATTN_RMS_FORM_TWO_PASS = 2 };
size_t attn_rmsnorm_matmul_ws_bytes(int B, int H);
int attn_rmsnorm_matmul_ws(const void* X, const void* G, const void* W, void* O, float* rms,
                           int B, int H, int D, float eps, int form, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * attn_rmsnorm_matmul_ws_chained - attn_rmsnorm_matmul_ws for calls that
 * follow one another on a stream with constant weights (no counterpart in
 * the pages: a launch option of this library, as attn_rmsnorm_matmul_chained).
 * The first kernel of the call (the conversion pass, or the fused kernel) is
 * launched as a programmatic dependent of the kernel before it on the stream
 * and waits for that kernel before it reads X or the workspace; in the
 * two-pass form the product kernel follows the pass as before. Caller's
 * promise: W is not written by the kernel that precedes the call. Arguments,
 * results and errors as attn_rmsnorm_matmul_ws.
 */
int attn_rmsnorm_matmul_ws_chained(const void* X, const void* G, const void* W, void* O,
                                   float* rms, int B, int H, int D, float eps, int form,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* The split count attn_rmsnorm_matmul chooses when given 0 (negative status on
 * invalid sizes). */
int attn_rmsnorm_matmul_splits(int B, int H, int D);

/*
 * Split-K decode (Neptune论文浅读 §6; the split-KV decode of CMU 15-779
 * 第 11 讲 §7.1, which parallelises over batch x KV head x KV sequence and
 * stacks the G = Hq / Hkv query heads of a group as rows so that each K/V row
 * is read once per KV head).
 *
 * Split geometry: with S splits and padded length Lk_max, every split covers
 * C = attn_decode_split_len(Lk_max, S) keys: split s covers keys
 * [s*C, (s+1)*C) clipped to [0, kv_len[b]). Splits beyond a sequence's
 * length are empty and produce LSE_part = -inf, O_part = 0.
 */

/* Resolves a requested split count: requested > 0 is returned unchanged
 * (clipped to [1, Lk_max]); 0 picks a count for this shape and device.
 * Returns the count, or a negative attn_status on invalid sizes. */
int attn_decode_num_splits(int B, int Hkv, int Lk_max, int d, int requested);

/* Keys per split: ceil(ceil(Lk_max / S) / 64) * 64, or a negative
 * attn_status on invalid sizes. */
int attn_decode_split_len(int Lk_max, int num_splits);

/* Bytes of the two partial buffers together: fp32 O_part [B, Hq, S, d] plus
 * fp32 LSE_part [B, Hq, S]. Returns 0 on invalid sizes. */
size_t attn_decode_workspace_bytes(int B, int Hq, int num_splits, int d);

/*
 * attn_decode_splitk - local reductions of the Split-K form.
 *
 *   Q        bf16 [B, Hq, d]                 (device, read; one query token)
 *   K, V     bf16 [B, Hkv, Lk_max, d]        (device, read; padded KV cache)
 *   kv_lens  int32 [B] on the device, each in [0, Lk_max], or NULL (= Lk_max)
 *   scale    softmax scale (finite)
 *   num_splits  S as resolved by attn_decode_num_splits (0 = auto); the
 *            count actually used is written to *out_splits when non-NULL.
 *   O_part   fp32 [B, Hq, S, d]  (device, written): each split's normalised
 *            output o_s / l_s
 *   LSE_part fp32 [B, Hq, S]     (device, written): m_s + ln l_s, or -inf
 * The caller sizes O_part / LSE_part for the resolved S.
 */
int attn_decode_splitk(const void* Q, const void* K, const void* V,
                       const int* kv_lens,
                       int B, int Hq, int Hkv, int Lk_max, int d, float scale,
                       int num_splits, int* out_splits,
                       float* O_part, float* LSE_part, void* stream);

/*
 * attn_combine - global reduction of the Split-K form (Neptune论文浅读 §6:
 * every split's local sum and output is repaired with the global max, then
 * summed). With M = max_s LSE_s and w_s = exp(LSE_s - M):
 *   O = sum_s w_s O_s / sum_s w_s,   LSE = M + ln sum_s w_s.
 * Splits with LSE_s = -inf weigh 0; if all are -inf, O = 0 and LSE = -inf.
 *
 *   O_part fp32 [B, Hq, S, d], LSE_part fp32 [B, Hq, S]  (device, read)
 *   O      bf16 [B, Hq, d]                                (device, written)
 *   LSE    fp32 [B, Hq] or NULL                           (device, written)
 */
int attn_combine(const float* O_part, const float* LSE_part,
                 int B, int Hq, int S, int d,
                 void* O, float* LSE, void* stream);

/* Convenience: attn_decode_splitk followed by attn_combine on one stream,
 * with caller-provided partial buffers sized for the resolved S. */
int attn_decode(const void* Q, const void* K, const void* V, const int* kv_lens,
                int B, int Hq, int Hkv, int Lk_max, int d, float scale,
                int num_splits, float* O_part, float* LSE_part,
                void* O, float* LSE, void* stream);

/*
 * attn_decode_noalloc - attn_decode for callers that cannot allocate.
 *
 * No counterpart in the pages: this is a convenience of this library. It is
 * for callers that have no way to provide the partial buffers attn_decode
 * needs: a serving runtime or plugin host that owns all device memory
 * through its own fixed pool, a latency-critical token loop in which a
 * cudaMalloc / cudaFree could block and synchronise the device, or plain C
 * code that holds only the tensors it was handed.
 *
 * Same arguments and results as attn_decode minus O_part / LSE_part: the
 * partials live in a fixed 32 MiB array inside the library (8 Mi floats),
 * held on every GPU that loads the library until the process exits. The call
 * allocates and frees nothing.
 *   - Limit: B*Hq*S*(d + 1) floats must fit in 8 Mi floats (S the resolved
 *     split count); larger calls return ATTN_ERR_WORKSPACE and launch nothing.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - All calls on a device share the array; calls whose kernels overlap on
 *     the GPU (unordered streams) race on it. Nothing in it needs clearing:
 *     each call writes every partial it reads.
 *   - The looked-up address is kept for the life of the process. After
 *     cudaDeviceReset on a device the array lives at a new address, so do not
 *     call this entry point (nor any other of this library, whose status word
 *     is looked up the same way) on that device again in the same process.
 */
int attn_decode_noalloc(const void* Q, const void* K, const void* V, const int* kv_lens,
                        int B, int Hq, int Hkv, int Lk_max, int d, float scale,
                        int num_splits, void* O, float* LSE, void* stream);

/* Static text for a status code (never NULL). */
const char* attn_status_string(int status);

/* Synchronises `stream`, then returns and clears the device status word of
 * the current device (ATTN_OK when no kernel recorded an error), or
 * ATTN_ERR_CUDA when synchronisation itself failed. */
int attn_device_status(void* stream);

/* Self-test of the library's failure detection (no counterpart in the pages):
 * launches a one-thread kernel that waits on a barrier nothing signals, with
 * a time limit of limit_ms (1..10000), through the same bounded-wait code all
 * kernels use. The kernel records ATTN_ERR_TIMEOUT in the device status word
 * and returns; the context stays usable. Returns the launch status. */
int attn_selftest_wait_timeout(int limit_ms, void* stream);

/* Self-test of failure detection inside the tcgen05 prefill kernel (no
 * counterpart in the pages). Runs attn_prefill (no ALiBi) with the tcgen05
 * form impl (ATTN_IMPL_TCGEN05 or ATTN_IMPL_TCGEN05_1TILE) and two changes:
 * every device wait has a time limit of limit_ms (1..10000), and the first
 * CTA's K/V producer stops before ring entry skip_entry (entries are
 * consumed in the order K_0, V_0, K_1, V_1, ...), so that CTA's MMA warp must
 * give up waiting, record ATTN_ERR_TIMEOUT in the device status word and
 * wind the CTA down: the other warps leave their waits, the copies already
 * in flight land, the issued products complete and the tensor memory is
 * freed before the kernel returns. The other CTAs run normally. Arguments as
 * attn_prefill; returns the launch status. The first CTA's rows of O and LSE
 * are left unwritten when it needed the missing entries. */
int attn_selftest_prefill_abort(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal,
                                float scale, int skip_entry, int limit_ms, int impl,
                                void* stream);

/* Library ABI version (major * 100 + minor). */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H */
