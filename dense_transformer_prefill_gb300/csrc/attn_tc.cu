// tcgen05 flash attention (causal GQA).  Kernel lands in the next step; the
// dispatcher reports it unsupported until then.
#include "internal.h"
#include "ptx.cuh"

namespace dtp {

static __device__ unsigned g_attn_err = 0;

unsigned read_clear_attn_errors() {
    unsigned v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_attn_err, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_attn_err, &z, sizeof(z));
    return v;
}

bool attn_tc_supported(int, int, int) { return false; }

cudaError_t launch_attn_tc(const __nv_bfloat16*, const __nv_bfloat16*, const __nv_bfloat16*,
                           long long, __nv_bfloat16*, int, int, int, int, float, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace dtp
