// The tcgen05 prefill with two Q tiles per CTA (one CTA per SM); the kernel
// itself is in prefill_tc.cuh.
#include "prefill_tc.cuh"

namespace attn {

int launch_prefill_tc(const PrefillLaunch& L, int d, cudaStream_t stream) {
    return launch_tc_nt<2>(L, d, stream);
}

}  // namespace attn
