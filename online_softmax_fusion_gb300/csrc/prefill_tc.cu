// tcgen05 prefill: not built yet; every call reports ATTN_ERR_UNSUPPORTED so
// the dispatcher takes the mma.sync kernel.
#include "common.cuh"
#include "kernels.h"

namespace attn {
int launch_prefill_tc(const PrefillLaunch&, int, cudaStream_t) { return ATTN_ERR_UNSUPPORTED; }
}  // namespace attn
