// Prefill from host buffers: the problem is cut into chunks of whole KV-head
// units (one KV head with its query heads), which are contiguous in the
// [B, H, L, d] layouts, and each chunk goes through three stages on three
// streams:
//   copy stream A : Q, K, V of the chunk, host -> device workspace
//   caller stream : the fused prefill of the chunk (attn_prefill_opts)
//   copy stream B : O, LSE of the chunk, device workspace -> host
// The stages of consecutive chunks overlap, so the step costs about the
// host link's time for all bytes plus one chunk's kernel and read-back,
// instead of the sum of the three. The copy streams and an event ring are
// created once per device and kept; calls on a device are serialised by a
// mutex around the enqueue.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "attn.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kEventRing = 256;      // reused round-robin; see enqueue order below
// Automatic chunking aims at this many chunks. Fewer chunks lengthen the
// pipeline's fill and drain; more serialise more kernels on the caller's
// stream, each at least as long as its longest causal row.
constexpr int kTargetChunks = 8;
constexpr size_t kRegionAlign = 256;

struct PipeCtx {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t ev[kEventRing] = {};
    int next = 0;
    std::mutex mu;
    bool ready = false;
};

PipeCtx g_ctx[kMaxDevices];
std::mutex g_init_mu;

// The per-device streams and events, created on first use.
PipeCtx* pipe_ctx() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    PipeCtx& c = g_ctx[dev];
    std::lock_guard<std::mutex> lk(g_init_mu);
    if (!c.ready) {
        if (cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
        if (cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
        for (int i = 0; i < kEventRing; ++i)
            if (cudaEventCreateWithFlags(&c.ev[i], cudaEventDisableTiming) != cudaSuccess)
                return nullptr;
        c.ready = true;
    }
    return &c;
}

size_t round_up(size_t x) { return (x + kRegionAlign - 1) / kRegionAlign * kRegionAlign; }

struct Regions {
    size_t q, kv, o, lse, total;   // byte sizes (q, kv, o, lse) and the workspace total
};

Regions regions(int B, int Hq, int Hkv, int Lq, int Lk, int d) {
    Regions r;
    r.q = size_t(B) * Hq * Lq * d * 2;
    r.kv = size_t(B) * Hkv * Lk * d * 2;
    r.o = r.q;
    r.lse = size_t(B) * Hq * Lq * 4;
    r.total = round_up(r.q) + 2 * round_up(r.kv) + round_up(r.o) + round_up(r.lse);
    return r;
}

// KV-head units per chunk: within one batch item (n <= Hkv) or whole batch
// items (a multiple of Hkv), so that ALiBi slopes keep a plain head offset.
long long units_per_chunk(int B, int Hkv, int requested) {
    const long long U = (long long)B * Hkv;
    long long n = requested > 0 ? requested : (U + kTargetChunks - 1) / kTargetChunks;
    if (n > Hkv) n = (n + Hkv - 1) / Hkv * Hkv;
    return n < 1 ? 1 : n;
}

}  // namespace

extern "C" {

size_t attn_prefill_host_workspace_bytes(int B, int Hq, int Hkv, int Lq, int Lk, int d) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lk <= 0 || d <= 0) return 0;
    return regions(B, Hq, Hkv, Lq, Lk, d).total;
}

int attn_prefill_host_chunks(int B, int Hkv, int chunk_kv_heads) {
    if (B <= 0 || Hkv <= 0) return 0;
    const long long n = units_per_chunk(B, Hkv, chunk_kv_heads);
    if (n >= Hkv) {
        const long long items = n / Hkv;
        return int((B + items - 1) / items);
    }
    return int((long long)B * ((Hkv + n - 1) / n));
}

int attn_prefill_host(const void* Qh, const void* Kh, const void* Vh, void* Oh, float* LSEh,
                      int B, int Hq, int Hkv, int Lq, int Lk, int d,
                      const attn_prefill_options* opts, int chunk_kv_heads, void* workspace,
                      size_t workspace_bytes, void* stream) {
    // everything the chunks' own validation would reject is rejected here,
    // before any copy is queued
    if (!Qh || !Kh || !Vh || !Oh || !opts || !workspace) return ATTN_ERR_NULL;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lk <= 0 || Hq % Hkv != 0) return ATTN_ERR_SHAPE;
    if (B > 65535 || Hq > 65535) return ATTN_ERR_SHAPE;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (opts->impl < ATTN_IMPL_AUTO || opts->impl > ATTN_IMPL_MMA_SYNC) return ATTN_ERR_UNSUPPORTED;
    if (!std::isfinite(opts->scale) || !std::isfinite(opts->softcap) || opts->softcap < 0.f)
        return ATTN_ERR_VALUE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u) ||
        (opts->alibi_slopes && (reinterpret_cast<uintptr_t>(opts->alibi_slopes) & 3u)))
        return ATTN_ERR_ALIGN;
    const Regions r = regions(B, Hq, Hkv, Lq, Lk, d);
    if (workspace_bytes < r.total) return ATTN_ERR_WORKSPACE;
    PipeCtx* c = pipe_ctx();
    if (!c) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(c->mu);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* dQ = static_cast<char*>(workspace);
    char* dK = dQ + round_up(r.q);
    char* dV = dK + round_up(r.kv);
    char* dO = dV + round_up(r.kv);
    char* dL = dO + round_up(r.o);
    const char* hQ = static_cast<const char*>(Qh);
    const char* hK = static_cast<const char*>(Kh);
    const char* hV = static_cast<const char*>(Vh);
    char* hO = static_cast<char*>(Oh);
    char* hL = reinterpret_cast<char*>(LSEh);
    const int G = Hq / Hkv;
    // bytes of one KV-head unit: its G query heads of Q (and of O), its K (and
    // V) head, its G rows of LSE
    const size_t q_unit = size_t(G) * Lq * d * 2;
    const size_t kv_unit = size_t(Lk) * d * 2;
    const size_t l_unit = size_t(G) * Lq * 4;
    auto next_event = [c]() {
        cudaEvent_t e = c->ev[c->next];
        c->next = (c->next + 1) % kEventRing;
        return e;
    };
    // Each event is waited on right after it is recorded, so reusing it
    // kEventRing records later cannot disturb a wait already queued.
    auto hand_over = [&](cudaStream_t from, cudaStream_t to) -> int {
        cudaEvent_t e = next_event();
        if (cudaEventRecord(e, from) != cudaSuccess) return ATTN_ERR_CUDA;
        return cudaStreamWaitEvent(to, e, 0) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    };

    // one chunk: Bc batch items from unit u0, hkv KV heads each
    auto run_chunk = [&](long long u0, int Bc, int hkv, int slope_off) -> int {
        const size_t nu = size_t(Bc) * hkv;
        const size_t qo = size_t(u0) * q_unit, ko = size_t(u0) * kv_unit, lo = size_t(u0) * l_unit;
        if (cudaMemcpyAsync(dQ + qo, hQ + qo, nu * q_unit, cudaMemcpyDefault, c->h2d) != cudaSuccess ||
            cudaMemcpyAsync(dK + ko, hK + ko, nu * kv_unit, cudaMemcpyDefault, c->h2d) != cudaSuccess ||
            cudaMemcpyAsync(dV + ko, hV + ko, nu * kv_unit, cudaMemcpyDefault, c->h2d) != cudaSuccess)
            return ATTN_ERR_CUDA;
        int st = hand_over(c->h2d, s);
        if (st) return st;
        attn_prefill_options o = *opts;
        if (o.alibi_slopes) o.alibi_slopes += slope_off;
        st = attn_prefill_opts(dQ + qo, dK + ko, dV + ko, dO + qo,
                               hL ? reinterpret_cast<float*>(dL + lo) : nullptr, Bc, hkv * G, hkv,
                               Lq, Lk, d, &o, stream);
        if (st) return st;
        if ((st = hand_over(s, c->d2h))) return st;
        if (cudaMemcpyAsync(hO + qo, dO + qo, nu * q_unit, cudaMemcpyDefault, c->d2h) != cudaSuccess)
            return ATTN_ERR_CUDA;
        if (hL && cudaMemcpyAsync(hL + lo, dL + lo, nu * l_unit, cudaMemcpyDefault, c->d2h) != cudaSuccess)
            return ATTN_ERR_CUDA;
        return ATTN_OK;
    };

    // both copy streams start after the work already queued on the caller's stream
    int st = hand_over(s, c->h2d);
    if (!st) st = hand_over(s, c->d2h);
    if (st) return st;
    const long long n = units_per_chunk(B, Hkv, chunk_kv_heads);
    if (n >= Hkv) {
        const int items = int(n / Hkv);
        for (int b = 0; b < B && !st; b += items)
            st = run_chunk((long long)b * Hkv, b + items <= B ? items : B - b, Hkv, 0);
    } else {
        for (int b = 0; b < B && !st; ++b)
            for (int h0 = 0; h0 < Hkv && !st; h0 += int(n))
                st = run_chunk((long long)b * Hkv + h0, 1, h0 + n <= Hkv ? int(n) : Hkv - h0,
                               h0 * G);
    }
    // the caller's stream resumes after both copy streams, also after an error
    const int j1 = hand_over(c->h2d, s);
    const int j2 = hand_over(c->d2h, s);
    return st ? st : (j1 ? j1 : j2);
}

}  // extern "C"
