// The tcgen05 prefill with one Q tile per CTA (two CTAs per SM); the kernel
// itself is in prefill_tc.cuh.
#include "prefill_tc.cuh"

namespace attn {

int launch_prefill_tc1(const PrefillLaunch& L, int d, cudaStream_t stream) {
    return launch_tc_nt<1>(L, d, stream);
}

}  // namespace attn
