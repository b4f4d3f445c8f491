// Allocation-free variant of the bf16 causal GQA attention entry point.
//
// Some callers cannot allocate device memory at the point where they need
// attention: code running inside a stream-ordered region it does not own,
// plug-ins handed only the tensors of one op, or runtimes that forbid
// cudaMalloc after start-up (it synchronises the device and can fail under
// memory pressure).  dtp_sdpa_causal_gqa needs a caller-provided workspace for
// the transposed V operand; this variant keeps that scratch in a fixed
// device-resident array instead, so the caller passes only q, k, v and out.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits.  Host code
// may not use the array's name as a device address (it is a host-side
// stand-in), so the device address is looked up once per device with
// cudaGetSymbolAddress on the first call made with that device current.
#include <mutex>

#include "internal.h"

namespace dtp {

// 8 MiB: room for v^T of n_head_kv * head_dim * round_up(T, 8) two-byte values
// (f16 copies of the bf16 v), e.g. 8 kv heads x 128 dims x 4096 tokens.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once).
int scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(DTP_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(DTP_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(DTP_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return DTP_OK;
}

}  // namespace
}  // namespace dtp

using namespace dtp;

extern "C" int dtp_sdpa_causal_gqa_noalloc(const void* q, const void* k, const void* v, void* out,
                                           int T, int n_head, int n_head_kv, int head_dim,
                                           float scale, dtp_stream_t stream) {
    if (!q || !k || !v || !out) return fail(DTP_ERR_INVALID_ARG, "NULL pointer");
    if (T <= 0 || n_head <= 0 || n_head_kv <= 0 || head_dim <= 0)
        return fail(DTP_ERR_INVALID_ARG, "sizes must be >= 1");
    if (n_head % n_head_kv) return fail(DTP_ERR_INVALID_ARG, "n_head %% n_head_kv != 0");
    if (!attn_tc_supported(n_head, n_head_kv, head_dim))
        return fail(DTP_ERR_UNSUPPORTED,
                    "bf16 attention: head_dim must be 64 or 128 and n_head/n_head_kv even");
    if (!aligned16(q) || !aligned16(k) || !aligned16(out))
        return fail(DTP_ERR_INVALID_ARG, "q, k and out must be 16-byte aligned");
    const long long ldvt = (long long)align_up(T, 8);
    const size_t need = (size_t)n_head_kv * head_dim * (size_t)ldvt * 2;
    if (need > kNoAllocScratchBytes)
        return fail(DTP_ERR_WORKSPACE,
                    "attention needs %zu bytes of scratch for v^T (n_head_kv*head_dim*T rounded "
                    "up to 8, 2 bytes each) but the allocation-free variant has a fixed %zu bytes; use "
                    "dtp_sdpa_causal_gqa with a workspace",
                    need, kNoAllocScratchBytes);
    void* scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    __half* vt = (__half*)scratch;
    DTP_CUDA_CHECK(launch_transpose_v((const __nv_bfloat16*)v, vt, T, n_head_kv * head_dim,
                                      (int)ldvt, s));
    DTP_CUDA_CHECK(launch_attn_tc((const __nv_bfloat16*)q, (const __nv_bfloat16*)k, vt, ldvt,
                                  (__nv_bfloat16*)out, T, n_head, n_head_kv, head_dim, scale, s));
    return DTP_OK;
}
