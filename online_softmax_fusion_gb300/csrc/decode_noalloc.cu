// Split-K decode for callers that cannot allocate device memory.
//
// The ordinary decode (attn_decode) needs two caller-provided partial
// buffers. Some callers have no way to provide them: a serving runtime or
// plugin host that owns every device allocation through its own fixed pool
// and forbids allocations outside it, a latency-critical token loop where a
// cudaMalloc / cudaFree could block and synchronise the device, or plain C
// code that holds only the tensors it was handed and no allocator. For them
// attn_decode_noalloc keeps the partials in a fixed array that lives in the
// library itself, so the call allocates nothing.
//
// The array is a file-scope __device__ variable of kNoAllocScratchFloats
// floats (32 MiB). Every GPU that loads the library holds it until the
// process exits. All calls on a device share it and it keeps the last call's
// contents; nothing in it needs to start at zero, because the decode kernel
// writes every partial (empty splits included) that the combine then reads.
// Two calls whose kernels overlap on the GPU (different streams without
// ordering between them) race on the array.
#include <cstddef>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

// O_part [B, Hq, S, d] followed by LSE_part [B, Hq, S], fp32.
constexpr size_t kNoAllocScratchFloats = size_t(8) << 20;
static __device__ __align__(256) float g_decode_scratch[kNoAllocScratchFloats];

constexpr int kMaxDevices = 64;

// Device address of the array on the current device. In host code the
// symbol itself is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
float* scratch_on_current_device() {
    static float* ptrs[kMaxDevices] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
            return nullptr;
        ptrs[dev] = static_cast<float*>(p);
    }
    return ptrs[dev];
}

}  // namespace
}  // namespace attn

extern "C" int attn_decode_noalloc(const void* Q, const void* K, const void* V,
                                   const int* kv_lens, int B, int Hq, int Hkv, int Lk_max, int d,
                                   float scale, int num_splits, void* O, float* LSE,
                                   void* stream) {
    if (!Q || !K || !V || !O) return ATTN_ERR_NULL;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lk_max <= 0) return ATTN_ERR_SHAPE;
    const int S = attn_decode_num_splits(B, Hkv, Lk_max, d, num_splits);
    if (S <= 0) return -S;
    const size_t rows = size_t(B) * size_t(Hq) * size_t(S);
    const size_t need = rows * size_t(d) + rows;
    if (need > attn::kNoAllocScratchFloats) return ATTN_ERR_WORKSPACE;
    float* base = attn::scratch_on_current_device();
    if (!base) return ATTN_ERR_CUDA;
    float* O_part = base;
    float* LSE_part = base + rows * size_t(d);
    return attn_decode(Q, K, V, kv_lens, B, Hq, Hkv, Lk_max, d, scale, S, O_part, LSE_part, O,
                       LSE, stream);
}
