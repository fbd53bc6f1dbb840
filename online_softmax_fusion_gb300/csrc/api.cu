// C-ABI layer of libattn.so: argument validation, TMA descriptor encoding,
// split-count policy, launch dispatch and the device status word.
// The entry points are declared and documented in include/attn.h.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace attn {

// First error recorded by any kernel of this library on this device.
__device__ int g_status_word = 0;

namespace {

constexpr int kMaxDevices = 64;

int* status_ptr() {
    static int* ptrs[kMaxDevices] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int*>(p);
    }
    return ptrs[dev];
}

int sm_count() {
    static int counts[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
    if (!counts[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        counts[dev] = n;
    }
    return counts[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// bf16 tensor [outer, L, d] (d innermost) as a 3-D tensor map with a
// (64, box_rows, 1) box and the 128-byte swizzle; rows past L read as zero.
int make_map(CUtensorMap* m, const void* base, int d, int L, long long outer, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return ATTN_ERR_CUDA;
    cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(L), cuuint64_t(outer)};
    cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(L) * cuuint64_t(d) * 2};
    cuuint32_t box[3] = {64, cuuint32_t(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(int B, int Hq, int Hkv, int d, float scale) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0) return ATTN_ERR_SHAPE;
    if (Hq % Hkv != 0) return ATTN_ERR_SHAPE;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return ATTN_ERR_VALUE;
    if (B > 65535 || Hq > 65535) return ATTN_ERR_SHAPE;
    return ATTN_OK;
}

int ceil_div(long long a, long long b) { return int((a + b - 1) / b); }

// Tile geometry of the fused RMSNorm + product.
//  * batch rows per CTA: one tile when B <= 256 (or the caller's tile), else
//    equal tiles of at most 256;
//  * K split: the largest power of two <= 8 that keeps the whole grid
//    resident (one CTA per SM; two for batch tiles <= 32) and gives each CTA
//    at least one 64-wide K step;
//  * shared memory: ~200 KB per CTA when the grid is one CTA per SM, else
//    ~100 KB (two per SM), less the epilogue's receive area when that gets
//    its own space (small batch tiles; larger ones reuse the rings); the X
//    ring takes a third (half for batch tiles >= 128) in 2..8 slots, a
//    multiple of the converter groups, the W ring the rest (2..12 slots);
//  * converter warps: one thread per batch row and K step. A grid of one
//    CTA per SM with batch tiles >= 128 launches 16 converter warps, so
//    that two or more groups convert K steps at once (a single group's
//    conversion, latency-bound, otherwise paces the loop); its X ring holds
//    two slots per group and the W ring keeps at least 4.
struct RmsGeometry {
    int NB, w_stages, x_stages, splits, k_tiles, cvt_all, cvt_warps, cvt_groups, recv_separate;
};

RmsGeometry rms_geometry(int B, int H, int D, int splits_req, int tile_req) {
    RmsGeometry g;
    const int tile_max = tile_req > 0 ? tile_req : 256;
    const int b_tiles = ceil_div(B, tile_max);
    g.NB = ceil_div(ceil_div(B, b_tiles), 16) * 16;
    g.k_tiles = ceil_div(H, 64);
    const long long base = (long long)ceil_div(D, 128) * ceil_div(B, g.NB);
    const long long sms = sm_count();
    // small batch tiles run two CTAs per SM (their rings fit in ~100 KB)
    const long long slots = g.NB <= 32 ? 2 * sms : sms;
    if (splits_req > 0) {
        g.splits = splits_req;
    } else {
        g.splits = 1;
        while (g.splits * 2 <= 8 && g.splits * 2 <= g.k_tiles && base * g.splits * 2 <= slots)
            g.splits *= 2;
    }
    const int xslot = g.NB * 128;
    const int wslot = 16384;
    int budget = base * g.splits <= sms ? 200 * 1024 : 100 * 1024;
    // the epilogue's receive area: fp32 tile + (E, s) per row and split; it
    // gets its own space when small, else it reuses the rings
    const int recv = g.NB * 512 + 8 * g.splits * g.NB;
    g.recv_separate = recv <= 32 * 1024 + 8 * 8 * 64 ? 1 : 0;
    if (g.recv_separate) budget -= recv;
    budget = std::max(budget, recv + wslot);
    // converter warps per K step: one thread per batch row; the X ring gets a
    // third of the space (half for large batch tiles, whose X slots are big)
    g.cvt_warps = ceil_div(g.NB, 32);
    g.cvt_all = (base * g.splits <= sms && g.NB >= 128) ? 16 : 8;
    if (g.cvt_all == 16) {
        const int groups = 16 / g.cvt_warps;
        const int fit = std::max(groups, (budget - 4 * wslot) / xslot);
        g.x_stages = std::min({kRmsMaxXStages, 2 * groups, fit});
        g.cvt_groups = std::min(groups, g.x_stages);
    } else {
        const int x_share = g.NB >= 128 ? budget / 2 : budget / 3;
        g.x_stages = std::max(2, std::min(kRmsMaxXStages, x_share / xslot));
        g.cvt_groups = std::min(8 / g.cvt_warps, g.x_stages);
    }
    g.x_stages = std::max(g.cvt_groups, g.x_stages / g.cvt_groups * g.cvt_groups);
    g.w_stages = std::max(2, std::min(kRmsMaxWStages, (budget - g.x_stages * xslot) / wslot));
    while (!g.recv_separate && g.w_stages < kRmsMaxWStages &&
           g.w_stages * wslot + g.x_stages * xslot < recv)
        ++g.w_stages;
    return g;
}

}  // namespace

// One thread waits on a barrier that nothing arrives on, with a short limit:
// the bounded-wait path of every kernel, run to its end on purpose.
__global__ void wait_timeout_selftest_kernel(unsigned long long limit_ns, int* status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
        mbar_wait_limit(&bar, 0, &abort_flag, status, limit_ns);
    }
}

}  // namespace attn

using namespace attn;

extern "C" {

int attn_version(void) { return 100; }

const char* attn_status_string(int status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_NULL: return "a required pointer is NULL";
        case ATTN_ERR_SHAPE: return "invalid sizes (non-positive, Hq not a multiple of Hkv, or too large)";
        case ATTN_ERR_UNSUPPORTED: return "unsupported head dim or implementation";
        case ATTN_ERR_WORKSPACE: return "split count out of range";
        case ATTN_ERR_CUDA: return "a CUDA call failed";
        case ATTN_ERR_TIMEOUT: return "a device wait exceeded its time limit";
        case ATTN_ERR_ALIGN: return "pointer not 16-byte aligned";
        case ATTN_ERR_VALUE: return "invalid value (non-finite scale or eps, or a bad split count)";
        default: return "unknown status";
    }
}

int attn_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
    }
    return v;
}

int attn_selftest_wait_timeout(int limit_ms, void* stream) {
    if (limit_ms <= 0 || limit_ms > 10000) return ATTN_ERR_VALUE;
    int* st = status_ptr();
    if (!st) return ATTN_ERR_CUDA;
    wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        (unsigned long long)limit_ms * 1000000ull, st);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"

namespace {

// Automatic choice between the two tcgen05 CTA forms (two Q tiles per CTA,
// one CTA per SM; or one Q tile per CTA, two CTAs per SM), from measurements
// on GB300: the one-tile form wins when the two-tile grid cannot fill the
// SMs once (causal GQA + ALiBi at L = 512 and 1024: 1.2x and 1.14x), and
// with SoftCap, whose softmax is bound by the special-function unit (two
// CTAs per SM interleave it better, 1.06x); the two-tile form wins
// everywhere else (L >= 2048: 1.08-1.1x).
bool prefer_one_tile(const PrefillParams& p, int d) {
    (void)d;
    if (p.softcap > 0.f) return true;
    const bool pair = p.pair_heads != 0;
    const long long rows_per_item = pair ? 128 : 256;
    const long long items = (p.Lq + rows_per_item - 1) / rows_per_item *
                            (long long)(pair ? p.Hq / 2 : p.Hq) * p.B;
    return items < sm_count();
}

int prefill_impl(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int Hq,
                 int Hkv, int Lq, int Lk, int d, int causal, float scale,
                 const float* alibi_slopes, float softcap, int window_left, int window_right,
                 int impl, void* stream, int selftest_skip = 0,
                 unsigned long long wait_ns = 0) {
    if (!Q || !K || !V || !O) return ATTN_ERR_NULL;
    int st = check_common(B, Hq, Hkv, d, scale);
    if (st) return st;
    if (Lq <= 0 || Lk <= 0) return ATTN_ERR_SHAPE;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return ATTN_ERR_ALIGN;
    if ((LSE && (reinterpret_cast<uintptr_t>(LSE) & 3u)) ||
        (alibi_slopes && (reinterpret_cast<uintptr_t>(alibi_slopes) & 3u)))
        return ATTN_ERR_ALIGN;
    if (impl < ATTN_IMPL_AUTO || impl > ATTN_IMPL_TCGEN05_1TILE) return ATTN_ERR_UNSUPPORTED;
    if (!std::isfinite(softcap) || softcap < 0.f) return ATTN_ERR_VALUE;
    const bool extra = softcap > 0.f || window_left >= 0 || window_right >= 0;

    PrefillLaunch L;
    std::memset(&L, 0, sizeof(L));
    L.p.O = static_cast<__nv_bfloat16*>(O);
    L.p.LSE = LSE;
    L.p.slopes = alibi_slopes;
    L.p.B = B;
    L.p.Hq = Hq;
    L.p.Hkv = Hkv;
    L.p.Lq = Lq;
    L.p.Lk = Lk;
    L.p.G = Hq / Hkv;
    L.p.scale_log2 = scale * kLog2e;
    L.p.causal = causal ? 1 : 0;
    L.p.softcap = softcap;
    L.p.window_left = window_left < 0 ? -1 : window_left;
    L.p.window_right = window_right < 0 ? -1 : window_right;
    L.p.pair_heads = (L.p.G % 2 == 0) ? 1 : 0;
    L.p.status = status_ptr();
    if (!L.p.status) return ATTN_ERR_CUDA;
    L.p.selftest_skip = selftest_skip;
    L.p.wait_ns = wait_ns;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const bool want_tc = impl == ATTN_IMPL_TCGEN05 || impl == ATTN_IMPL_TCGEN05_1TILE ||
                         impl == ATTN_IMPL_AUTO;
    if (want_tc) {
        if ((st = make_map(&L.tmQ, Q, d, Lq, (long long)B * Hq, kTcBM))) return st;
        if ((st = make_map(&L.tmK, K, d, Lk, (long long)B * Hkv, kTcBN))) return st;
        if ((st = make_map(&L.tmV, V, d, Lk, (long long)B * Hkv, kTcBN))) return st;
        if ((st = make_map(&L.tmO, O, d, Lq, (long long)B * Hq, 32))) return st;
        const bool one_tile = impl == ATTN_IMPL_TCGEN05_1TILE ||
                              (impl == ATTN_IMPL_AUTO && prefer_one_tile(L.p, d));
        st = one_tile ? launch_prefill_tc1(L, d, s) : launch_prefill_tc(L, d, s);
        if (st != ATTN_ERR_UNSUPPORTED || impl != ATTN_IMPL_AUTO) return st;
    }
    // the register-tile kernel has no softcap / window variants
    if (extra) return ATTN_ERR_UNSUPPORTED;
    if ((st = make_map(&L.tmQ, Q, d, Lq, (long long)B * Hq, kMmaBM))) return st;
    if ((st = make_map(&L.tmK, K, d, Lk, (long long)B * Hkv, kMmaBN))) return st;
    if ((st = make_map(&L.tmV, V, d, Lk, (long long)B * Hkv, kMmaBN))) return st;
    return launch_prefill_mma(L, d, s);
}

}  // namespace

extern "C" {

size_t attn_prefill_splitkv_workspace_bytes(int B, int Hq, int Lq, int d, int num_splits) {
    if (B <= 0 || Hq <= 0 || Lq <= 0 || d <= 0 || num_splits <= 1) return 0;
    return size_t(B) * Hq * Lq * size_t(num_splits) * size_t(d + 1) * sizeof(float);
}

int attn_prefill_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                         int Hq, int Hkv, int Lq, int Lk, int d, int causal, float scale,
                         const float* alibi_slopes, int num_splits, void* workspace,
                         size_t workspace_bytes, void* stream) {
    if (num_splits < 1 || num_splits > 16) return ATTN_ERR_WORKSPACE;
    if (num_splits == 1)
        return prefill_impl(Q, K, V, O, LSE, B, Hq, Hkv, Lq, Lk, d, causal, scale, alibi_slopes,
                            0.f, -1, -1, ATTN_IMPL_TCGEN05, stream);
    if (!Q || !K || !V || !O || !workspace) return ATTN_ERR_NULL;
    int st = check_common(B, Hq, Hkv, d, scale);
    if (st) return st;
    if (Lq <= 0 || Lk <= 0) return ATTN_ERR_SHAPE;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(workspace))
        return ATTN_ERR_ALIGN;
    if ((LSE && (reinterpret_cast<uintptr_t>(LSE) & 3u)) ||
        (alibi_slopes && (reinterpret_cast<uintptr_t>(alibi_slopes) & 3u)))
        return ATTN_ERR_ALIGN;
    if (workspace_bytes < attn_prefill_splitkv_workspace_bytes(B, Hq, Lq, d, num_splits))
        return ATTN_ERR_WORKSPACE;
    PrefillLaunch L;
    std::memset(&L, 0, sizeof(L));
    L.p.O = static_cast<__nv_bfloat16*>(O);
    L.p.LSE = LSE;
    L.p.slopes = alibi_slopes;
    L.p.B = B;
    L.p.Hq = Hq;
    L.p.Hkv = Hkv;
    L.p.Lq = Lq;
    L.p.Lk = Lk;
    L.p.G = Hq / Hkv;
    L.p.scale_log2 = scale * kLog2e;
    L.p.causal = causal ? 1 : 0;
    L.p.softcap = 0.f;
    L.p.window_left = -1;
    L.p.window_right = -1;
    L.p.pair_heads = (L.p.G % 2 == 0) ? 1 : 0;
    L.p.splits = num_splits;
    L.p.O_part = static_cast<float*>(workspace);
    L.p.LSE_part = L.p.O_part + size_t(B) * Hq * Lq * size_t(num_splits) * d;
    L.p.status = status_ptr();
    if (!L.p.status) return ATTN_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = make_map(&L.tmQ, Q, d, Lq, (long long)B * Hq, kTcBM))) return st;
    if ((st = make_map(&L.tmK, K, d, Lk, (long long)B * Hkv, kTcBN))) return st;
    if ((st = make_map(&L.tmV, V, d, Lk, (long long)B * Hkv, kTcBN))) return st;
    L.tmO = L.tmQ;   // not read: split partials are written in fp32 without it
    if ((st = launch_prefill_tc(L, d, s))) return st;
    // the partials of each row merged with the split-K combine (rows act as heads)
    if ((long long)B * Hq > 0x7fffffffLL / Lq) return ATTN_ERR_SHAPE;
    return launch_combine(L.p.O_part, L.p.LSE_part, B * Hq, Lq, num_splits, d, O, LSE, s);
}

int attn_prefill_ex(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int Hq,
                    int Hkv, int Lq, int Lk, int d, int causal, float scale,
                    const float* alibi_slopes, int impl, void* stream) {
    return prefill_impl(Q, K, V, O, LSE, B, Hq, Hkv, Lq, Lk, d, causal, scale, alibi_slopes, 0.f,
                        -1, -1, impl, stream);
}

int attn_prefill_opts(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                      int Hq, int Hkv, int Lq, int Lk, int d, const attn_prefill_options* opts,
                      void* stream) {
    if (!opts) return ATTN_ERR_NULL;
    return prefill_impl(Q, K, V, O, LSE, B, Hq, Hkv, Lq, Lk, d, opts->causal, opts->scale,
                        opts->alibi_slopes, opts->softcap, opts->window_left, opts->window_right,
                        opts->impl, stream);
}

int attn_prefill(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int Hq,
                 int Hkv, int Lq, int Lk, int d, int causal, float scale, const float* alibi_slopes,
                 void* stream) {
    return attn_prefill_ex(Q, K, V, O, LSE, B, Hq, Hkv, Lq, Lk, d, causal, scale, alibi_slopes,
                           ATTN_IMPL_AUTO, stream);
}

int attn_selftest_prefill_abort(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                int B, int Hq, int Hkv, int Lq, int Lk, int d, int causal,
                                float scale, int skip_entry, int limit_ms, int impl,
                                void* stream) {
    if (skip_entry < 0 || limit_ms <= 0 || limit_ms > 10000) return ATTN_ERR_VALUE;
    if (impl != ATTN_IMPL_TCGEN05 && impl != ATTN_IMPL_TCGEN05_1TILE) return ATTN_ERR_UNSUPPORTED;
    return prefill_impl(Q, K, V, O, LSE, B, Hq, Hkv, Lq, Lk, d, causal, scale, nullptr, 0.f, -1,
                        -1, impl, stream, skip_entry + 1,
                        (unsigned long long)limit_ms * 1000000ull);
}

size_t attn_backward_workspace_bytes(int B, int Hq, int Lq, int d) {
    if (B <= 0 || Hq <= 0 || Lq <= 0 || d <= 0) return 0;
    const size_t rows = size_t(B) * size_t(Hq) * size_t(Lq);
    return rows * size_t(d) * sizeof(float) + rows * sizeof(float);
}

int attn_backward(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                  const float* LSE, void* dQ, void* dK, void* dV, int B, int Hq, int Hkv, int Lq,
                  int Lk, int d, int causal, float scale, const float* alibi_slopes,
                  void* workspace, size_t workspace_bytes, void* stream) {
    return attn_backward_ex(Q, K, V, O, dO, LSE, dQ, dK, dV, B, Hq, Hkv, Lq, Lk, d, causal, scale,
                            alibi_slopes, workspace, workspace_bytes, ATTN_IMPL_AUTO, stream);
}

int attn_backward_ex(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* LSE, void* dQ, void* dK, void* dV, int B, int Hq, int Hkv,
                     int Lq, int Lk, int d, int causal, float scale, const float* alibi_slopes,
                     void* workspace, size_t workspace_bytes, int impl, void* stream) {
    if (impl != ATTN_IMPL_AUTO && impl != ATTN_IMPL_TCGEN05 && impl != ATTN_IMPL_MMA_SYNC)
        return ATTN_ERR_UNSUPPORTED;
    if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV || !workspace)
        return ATTN_ERR_NULL;
    int st = check_common(B, Hq, Hkv, d, scale);
    if (st) return st;
    if (Lq <= 0 || Lk <= 0) return ATTN_ERR_SHAPE;
    const void* ptrs[] = {Q, K, V, O, dO, dQ, dK, dV, workspace};
    for (const void* p : ptrs)
        if (!aligned16(p)) return ATTN_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(LSE) & 3u) ||
        (alibi_slopes && (reinterpret_cast<uintptr_t>(alibi_slopes) & 3u)))
        return ATTN_ERR_ALIGN;
    if (workspace_bytes < attn_backward_workspace_bytes(B, Hq, Lq, d)) return ATTN_ERR_WORKSPACE;
    BwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.Q = static_cast<const __nv_bfloat16*>(Q);
    p.K = static_cast<const __nv_bfloat16*>(K);
    p.V = static_cast<const __nv_bfloat16*>(V);
    p.O = static_cast<const __nv_bfloat16*>(O);
    p.dO = static_cast<const __nv_bfloat16*>(dO);
    p.LSE = LSE;
    p.dQ = static_cast<__nv_bfloat16*>(dQ);
    p.dK = static_cast<__nv_bfloat16*>(dK);
    p.dV = static_cast<__nv_bfloat16*>(dV);
    p.dQacc = static_cast<float*>(workspace);
    p.Dsum = p.dQacc + size_t(B) * Hq * Lq * d;
    p.slopes = alibi_slopes;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Lq = Lq;
    p.Lk = Lk;
    p.G = Hq / Hkv;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.causal = causal ? 1 : 0;
    if ((long long)(Lk + 63) / 64 > 0x7fffffffLL || Hkv > 65535) return ATTN_ERR_SHAPE;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const bool tc = impl == ATTN_IMPL_TCGEN05 || (impl == ATTN_IMPL_AUTO && d == 128);
    if (!tc) return launch_backward(p, d, cs);
    if (d != 128) return ATTN_ERR_UNSUPPORTED;
    BwdTcLaunch L;
    std::memset(&L, 0, sizeof(L));
    L.p = p;
    L.p.status = status_ptr();
    if ((st = make_map(&L.tmQ, Q, d, Lq, (long long)B * Hq, 128))) return st;
    if ((st = make_map(&L.tmdO, dO, d, Lq, (long long)B * Hq, 128))) return st;
    if ((st = make_map(&L.tmK, K, d, Lk, (long long)B * Hkv, 128))) return st;
    if ((st = make_map(&L.tmV, V, d, Lk, (long long)B * Hkv, 128))) return st;
    if ((st = launch_backward_prep(p, d, cs))) return st;
    if ((st = launch_backward_tc_main(L, cs))) return st;
    return launch_backward_convert(p, d, cs);
}

int attn_rmsnorm_matmul_splits(int B, int H, int D) {
    if (B <= 0 || H <= 0 || D <= 0) return -ATTN_ERR_SHAPE;
    return rms_geometry(B, H, D, 0, 0).splits;
}

int attn_rmsnorm_matmul(const void* X, const void* G, const void* W, void* O, float* rms, int B,
                        int H, int D, float eps, int splits, void* stream) {
    return attn_rmsnorm_matmul_tiled(X, G, W, O, rms, B, H, D, eps, 0, splits, stream);
}

}  // extern "C"

namespace {
int rmsnorm_matmul_impl(const void* X, const void* G, const void* W, void* O, float* rms,
                        int B, int H, int D, float eps, int batch_tile, int splits, int chained,
                        void* stream, void* workspace = nullptr);

// workspace of the two-pass form: Xg [B, H] bf16, then E [B] int, then s [B] fp32
size_t rms_ws_xg_bytes(int B, int H) { return (size_t(B) * size_t(H) * 2u + 255u) & ~size_t(255); }
size_t rms_ws_vec_bytes(int B) { return (size_t(B) * 4u + 255u) & ~size_t(255); }
}  // namespace

extern "C" {

int attn_rmsnorm_matmul_tiled(const void* X, const void* G, const void* W, void* O, float* rms,
                              int B, int H, int D, float eps, int batch_tile, int splits,
                              void* stream) {
    return rmsnorm_matmul_impl(X, G, W, O, rms, B, H, D, eps, batch_tile, splits, 0, stream);
}

int attn_rmsnorm_matmul_chained(const void* X, const void* G, const void* W, void* O, float* rms,
                                int B, int H, int D, float eps, void* stream) {
    return rmsnorm_matmul_impl(X, G, W, O, rms, B, H, D, eps, 0, 0, 1, stream);
}

size_t attn_rmsnorm_matmul_ws_bytes(int B, int H) {
    if (B <= 0 || H <= 0) return 0;
    return rms_ws_xg_bytes(B, H) + 2 * rms_ws_vec_bytes(B);
}

}  // extern "C"

namespace {
int rmsnorm_ws_impl(const void* X, const void* G, const void* W, void* O, float* rms, int B,
                    int H, int D, float eps, int form, void* workspace, size_t workspace_bytes,
                    int chained, void* stream);
}  // namespace

extern "C" {

int attn_rmsnorm_matmul_ws(const void* X, const void* G, const void* W, void* O, float* rms,
                           int B, int H, int D, float eps, int form, void* workspace,
                           size_t workspace_bytes, void* stream) {
    return rmsnorm_ws_impl(X, G, W, O, rms, B, H, D, eps, form, workspace, workspace_bytes, 0,
                           stream);
}

int attn_rmsnorm_matmul_ws_chained(const void* X, const void* G, const void* W, void* O,
                                   float* rms, int B, int H, int D, float eps, int form,
                                   void* workspace, size_t workspace_bytes, void* stream) {
    return rmsnorm_ws_impl(X, G, W, O, rms, B, H, D, eps, form, workspace, workspace_bytes, 1,
                           stream);
}

}  // extern "C"

namespace {

int rmsnorm_ws_impl(const void* X, const void* G, const void* W, void* O, float* rms, int B,
                    int H, int D, float eps, int form, void* workspace, size_t workspace_bytes,
                    int chained, void* stream) {
    if (form < ATTN_RMS_FORM_AUTO || form > ATTN_RMS_FORM_TWO_PASS) return ATTN_ERR_VALUE;
    if (form == ATTN_RMS_FORM_AUTO) {
        if (B <= 0 || H <= 0 || D <= 0) return ATTN_ERR_SHAPE;
        // measured faster than the fused kernel at every batch tried
        // (16 ... 256 rows at H = D = 4096)
        form = ATTN_RMS_FORM_TWO_PASS;
    }
    if (form == ATTN_RMS_FORM_FUSED)
        return rmsnorm_matmul_impl(X, G, W, O, rms, B, H, D, eps, 0, 0, chained, stream);
    if (!workspace) return ATTN_ERR_NULL;
    if (B > 0 && H > 0 && workspace_bytes < attn_rmsnorm_matmul_ws_bytes(B, H))
        return ATTN_ERR_WORKSPACE;
    return rmsnorm_matmul_impl(X, G, W, O, rms, B, H, D, eps, 0, 0, chained, stream, workspace);
}

}  // namespace

namespace {

int rmsnorm_matmul_impl(const void* X, const void* G, const void* W, void* O, float* rms,
                        int B, int H, int D, float eps, int batch_tile, int splits, int chained,
                        void* stream, void* workspace) {
    if (!X || !G || !W || !O) return ATTN_ERR_NULL;
    if (B <= 0 || H <= 0 || D <= 0) return ATTN_ERR_SHAPE;
    if (B > 65535 * 256 || H > (1 << 30) || D > (1 << 30)) return ATTN_ERR_SHAPE;
    if (H % 8 != 0 || D % 8 != 0) return ATTN_ERR_UNSUPPORTED;
    if (!std::isfinite(eps) || eps < 0.f) return ATTN_ERR_VALUE;
    if (!(splits == 0 || splits == 1 || splits == 2 || splits == 4 || splits == 8))
        return ATTN_ERR_VALUE;
    if (splits > 0 && splits > ceil_div(H, 64)) return ATTN_ERR_VALUE;
    if (batch_tile < 0 || batch_tile > 256 || batch_tile % 16) return ATTN_ERR_VALUE;
    const void* ptrs[] = {X, G, W, O};
    for (const void* p : ptrs)
        if (!aligned16(p)) return ATTN_ERR_ALIGN;
    if (rms && (reinterpret_cast<uintptr_t>(rms) & 3u)) return ATTN_ERR_ALIGN;
    if (workspace && !aligned16(workspace)) return ATTN_ERR_ALIGN;
    // chained calls take the same geometry as plain ones (same result, bit
    // for bit); a grid of one CTA per SM, leaving the second slot to the next
    // call, measured slower (13.1 against 10.7 us at batch 16)
    const RmsGeometry g = rms_geometry(B, H, D, splits, batch_tile);
    RmsLaunch L;
    std::memset(&L, 0, sizeof(L));
    L.p.O = static_cast<__nv_bfloat16*>(O);
    L.p.rms = rms;
    L.p.G = static_cast<const __nv_bfloat16*>(G);
    L.p.B = B;
    L.p.H = H;
    L.p.D = D;
    L.p.NB = g.NB;
    L.p.splits = g.splits;
    L.p.k_tiles = g.k_tiles;
    L.p.w_stages = g.w_stages;
    L.p.x_stages = g.x_stages;
    L.p.cvt_all = g.cvt_all;
    L.p.cvt_warps = g.cvt_warps;
    L.p.cvt_groups = g.cvt_groups;
    L.p.recv_separate = g.recv_separate;
    L.p.chained = chained;
    L.p.eps = eps;
    L.p.status = status_ptr();
    int st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (workspace) {
        // two-pass form: the conversion pass writes X ⊙ G and the per-row
        // (E, s); the product kernel follows it as a programmatic dependent
        // (W streams in while the pass runs) and reads the converted X
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        auto* xg = reinterpret_cast<__nv_bfloat16*>(ws);
        auto* e = reinterpret_cast<int*>(ws + rms_ws_xg_bytes(B, H));
        auto* sq = reinterpret_cast<float*>(ws + rms_ws_xg_bytes(B, H) + rms_ws_vec_bytes(B));
        if ((st = make_map(&L.tmX, xg, H, B, 1, g.NB))) return st;
        if ((st = make_map(&L.tmW, W, D, H, 1, 64))) return st;
        if ((st = launch_rmsnorm_prep(static_cast<const __nv_bfloat16*>(X),
                                      static_cast<const __nv_bfloat16*>(G), xg, e, sq, B, H,
                                      chained, cs)))
            return st;
        L.p.pre = 1;
        L.p.stats_e = e;
        L.p.stats_s = sq;
        L.p.chained = 1;
        return launch_rmsnorm_matmul(L, cs);
    }
    if ((st = make_map(&L.tmX, X, H, B, 1, g.NB))) return st;
    if ((st = make_map(&L.tmW, W, D, H, 1, 64))) return st;
    return launch_rmsnorm_matmul(L, cs);
}

}  // namespace

extern "C" {

int attn_decode_split_len(int Lk_max, int num_splits) {
    if (Lk_max <= 0) return -ATTN_ERR_SHAPE;
    if (num_splits <= 0) return -ATTN_ERR_WORKSPACE;
    const int per = ceil_div(Lk_max, num_splits);
    return ceil_div(per, 64) * 64;
}

int attn_decode_num_splits(int B, int Hkv, int Lk_max, int d, int requested) {
    if (B <= 0 || Hkv <= 0 || Lk_max <= 0) return -ATTN_ERR_SHAPE;
    if (d != 64 && d != 128) return -ATTN_ERR_UNSUPPORTED;
    if (requested < 0) return -ATTN_ERR_WORKSPACE;
    if (requested > 0) return requested < Lk_max ? requested : Lk_max;
    // Splits of about 2048 keys keep CTA work uniform across variable lengths;
    // small batches split finer until there are ~8 CTAs per SM.
    const int max_splits = ceil_div(Lk_max, 64);
    int S = ceil_div(Lk_max, 2048);
    const long long pairs = (long long)B * Hkv;
    const long long target = 8LL * sm_count();
    while (S < max_splits && pairs * S < target) S *= 2;
    if (S > max_splits) S = max_splits;
    return S;
}

size_t attn_decode_workspace_bytes(int B, int Hq, int num_splits, int d) {
    if (B <= 0 || Hq <= 0 || num_splits <= 0 || d <= 0) return 0;
    const size_t rows = size_t(B) * size_t(Hq) * size_t(num_splits);
    return rows * size_t(d) * sizeof(float) + rows * sizeof(float);
}

int attn_decode_splitk(const void* Q, const void* K, const void* V, const int* kv_lens, int B,
                       int Hq, int Hkv, int Lk_max, int d, float scale, int num_splits,
                       int* out_splits, float* O_part, float* LSE_part, void* stream) {
    if (!Q || !K || !V || !O_part || !LSE_part) return ATTN_ERR_NULL;
    int st = check_common(B, Hq, Hkv, d, scale);
    if (st) return st;
    if (Lk_max <= 0) return ATTN_ERR_SHAPE;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O_part) ||
        (reinterpret_cast<uintptr_t>(LSE_part) & 3u) ||
        (kv_lens && (reinterpret_cast<uintptr_t>(kv_lens) & 3u)))
        return ATTN_ERR_ALIGN;
    const int S = attn_decode_num_splits(B, Hkv, Lk_max, d, num_splits);
    if (S <= 0) return -S;
    if (S > 12288) return ATTN_ERR_WORKSPACE;
    const int G = Hq / Hkv;

    DecodeLaunch L;
    std::memset(&L, 0, sizeof(L));
    L.p.Q = static_cast<const __nv_bfloat16*>(Q);
    L.p.kv_lens = kv_lens;
    L.p.O_part = O_part;
    L.p.LSE_part = LSE_part;
    L.p.B = B;
    L.p.Hq = Hq;
    L.p.Hkv = Hkv;
    L.p.Lk_max = Lk_max;
    L.p.S = S;
    L.p.C = attn_decode_split_len(Lk_max, S);
    L.p.G = G;
    L.p.nrg = ceil_div(G, 16);
    L.p.rows = ceil_div(G, L.p.nrg);
    L.p.scale_log2 = scale * kLog2e;
    L.p.status = status_ptr();
    if (!L.p.status) return ATTN_ERR_CUDA;
    if ((long long)Hkv * L.p.nrg > 65535) return ATTN_ERR_SHAPE;
    if ((st = make_map(&L.tmK, K, d, Lk_max, (long long)B * Hkv, 64))) return st;
    if ((st = make_map(&L.tmV, V, d, Lk_max, (long long)B * Hkv, 64))) return st;
    if (out_splits) *out_splits = S;
    return launch_decode(L, d, static_cast<cudaStream_t>(stream));
}

int attn_combine(const float* O_part, const float* LSE_part, int B, int Hq, int S, int d, void* O,
                 float* LSE, void* stream) {
    if (!O_part || !LSE_part || !O) return ATTN_ERR_NULL;
    if (B <= 0 || Hq <= 0) return ATTN_ERR_SHAPE;
    if (S <= 0 || S > 12288) return ATTN_ERR_WORKSPACE;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(O_part) & 3u) || (reinterpret_cast<uintptr_t>(LSE_part) & 3u) ||
        (reinterpret_cast<uintptr_t>(O) & 1u) || (LSE && (reinterpret_cast<uintptr_t>(LSE) & 3u)))
        return ATTN_ERR_ALIGN;
    return launch_combine(O_part, LSE_part, B, Hq, S, d, O, LSE, static_cast<cudaStream_t>(stream));
}

int attn_decode(const void* Q, const void* K, const void* V, const int* kv_lens, int B, int Hq,
                int Hkv, int Lk_max, int d, float scale, int num_splits, float* O_part,
                float* LSE_part, void* O, float* LSE, void* stream) {
    if (!O) return ATTN_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(O) & 1u) || (LSE && (reinterpret_cast<uintptr_t>(LSE) & 3u)))
        return ATTN_ERR_ALIGN;
    int S = 0;
    int st = attn_decode_splitk(Q, K, V, kv_lens, B, Hq, Hkv, Lk_max, d, scale, num_splits, &S,
                                O_part, LSE_part, stream);
    if (st) return st;
    return attn_combine(O_part, LSE_part, B, Hq, S, d, O, LSE, stream);
}

}  // extern "C"
