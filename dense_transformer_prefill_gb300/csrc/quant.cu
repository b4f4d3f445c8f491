// Per-row e4m3 quantisation of GEMM operands (the quantised-weight variant of
// the prefill pass): a row y gets the float32 scale s = max|y| / 448 and the
// OCP FP8 E4M3 codes q_j = e4m3(y_j * (448 / max|y|)) (nearest-even,
// saturating at +-448; a zero row gets s = 0 and q = 0).  A GEMM of two such
// operands is s_a[m] s_b[n] (q_a q_b^T)[m, n]: the row scales of the activation
// (per token) and of the weight (per output channel) factor out of every dot
// product, so the tcgen05 kind::f8f6f4 GEMM applies them in its epilogue.
//
//   rmsnorm_e4m3   forward.rs, the RMSNorm step, written straight as e4m3 codes
//   quant_rows     bf16 rows (attention output, SwiGLU act) -> e4m3 codes
//   pack_e4m3      float32 weight rows -> e4m3 codes (+ the gate/up interleave)
#include <cuda_fp8.h>
#include <math.h>

#include "internal.h"

namespace dtp {

namespace {

__device__ __forceinline__ uint8_t to_e4m3(float v) {
    return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// Block-wide reduction in a fixed order; `red` holds one slot per warp.
template <bool MAX>
__device__ float block_reduce(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float u = __shfl_xor_sync(0xffffffffu, v, o);
        v = MAX ? fmaxf(v, u) : v + u;
    }
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < nw; ++i) t = MAX ? fmaxf(t, red[i]) : t + red[i];
    return t;
}

// 448 / amax and amax / 448 (both 0 for a zero row).
__device__ __forceinline__ void row_scale(float amax, float& inv, float& s) {
    inv = amax > 0.f ? 448.0f / amax : 0.f;
    s = amax / 448.0f;
}

__device__ __forceinline__ uint32_t pack4(float a, float b, float c, float d, float inv) {
    return (uint32_t)to_e4m3(a * inv) | ((uint32_t)to_e4m3(b * inv) << 8) |
           ((uint32_t)to_e4m3(c * inv) << 16) | ((uint32_t)to_e4m3(d * inv) << 24);
}

// One block per row, the row held in registers (cols % 4 == 0, cols <= 16 * blockDim).
// y = x * rstd * w exactly as the float32 RMSNorm kernel forms it, then quantised.
__global__ void rmsnorm_e4m3_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                    uint8_t* __restrict__ q, float* __restrict__ scale, int cols,
                                    float eps, const int* __restrict__ row_idx) {
    __shared__ float red[32];
    const size_t r = blockIdx.x;
    const float4* xr =
        reinterpret_cast<const float4*>(x + (size_t)(row_idx ? row_idx[r] : r) * cols);
    const int n4 = cols >> 2;
    float4 v[4];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c4 = threadIdx.x + i * blockDim.x;
        if (c4 < n4) {
            v[i] = xr[c4];
            ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
        }
    }
    ss = block_reduce<false>(ss, red);
    const float rstd = 1.0f / sqrtf(ss / (float)cols + eps);
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c4 = threadIdx.x + i * blockDim.x;
        if (c4 < n4) {
            const float4 g = reinterpret_cast<const float4*>(w)[c4];
            v[i] = make_float4(v[i].x * rstd * g.x, v[i].y * rstd * g.y, v[i].z * rstd * g.z,
                               v[i].w * rstd * g.w);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)),
                                     fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
        }
    }
    amax = block_reduce<true>(amax, red);
    float inv, s;
    row_scale(amax, inv, s);
    uint32_t* qr = reinterpret_cast<uint32_t*>(q + r * cols);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c4 = threadIdx.x + i * blockDim.x;
        if (c4 < n4) qr[c4] = pack4(v[i].x, v[i].y, v[i].z, v[i].w, inv);
    }
    if (threadIdx.x == 0) scale[r] = s;
}

// One block per row of bf16 x [rows, ldx]: cols % 8 == 0, 16-byte aligned rows.
// Rows of up to 8 * 8 * blockDim elements are read once and held in registers
// (8 16-byte chunks per thread); longer rows are read a second time.
__global__ void quant_rows_kernel(const __nv_bfloat16* __restrict__ x, int ldx, int cols,
                                  uint8_t* __restrict__ q, float* __restrict__ scale) {
    __shared__ float red[32];
    const size_t r = blockIdx.x;
    const uint4* xr = reinterpret_cast<const uint4*>(x + r * ldx);
    const int n8 = cols >> 3;
    constexpr int KEEP = 8;
    uint4 held[KEEP];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < KEEP; ++i) {
        const int c8 = threadIdx.x + i * blockDim.x;
        if (c8 < n8) {
            held[i] = xr[c8];
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&held[i]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = __bfloat1622float2(h[j]);
                amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
    }
    for (int c8 = threadIdx.x + KEEP * blockDim.x; c8 < n8; c8 += blockDim.x) {
        const uint4 u = xr[c8];
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(h[j]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
    amax = block_reduce<true>(amax, red);
    float inv, s;
    row_scale(amax, inv, s);
    uint2* qr = reinterpret_cast<uint2*>(q + r * cols);
    auto put = [&](int c8, const uint4& u) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
        const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]),
                     c = __bfloat1622float2(h[2]), d = __bfloat1622float2(h[3]);
        qr[c8] = make_uint2(pack4(a.x, a.y, b.x, b.y, inv), pack4(c.x, c.y, d.x, d.y, inv));
    };
#pragma unroll
    for (int i = 0; i < KEEP; ++i) {
        const int c8 = threadIdx.x + i * blockDim.x;
        if (c8 < n8) put(c8, held[i]);
    }
    for (int c8 = threadIdx.x + KEEP * blockDim.x; c8 < n8; c8 += blockDim.x) put(c8, xr[c8]);
    if (threadIdx.x == 0) scale[r] = s;
}

// One block per source row of a float32 weight [rows, cols]; destination row as
// in pack_matrix (mode 1 / 2: the gate / up half of a 128-row interleave block).
__global__ void pack_e4m3_kernel(const float* __restrict__ src, int cols, uint8_t* __restrict__ dst,
                                 float* __restrict__ dst_scale, int mode) {
    __shared__ float red[32];
    const int r = blockIdx.x;
    const float* sr = src + (size_t)r * cols;
    float amax = 0.f;
    for (int c = threadIdx.x; c < cols; c += blockDim.x) amax = fmaxf(amax, fabsf(sr[c]));
    amax = block_reduce<true>(amax, red);
    float inv, s;
    row_scale(amax, inv, s);
    int dr = r;
    if (mode == 1) dr = 128 * (r / 64) + (r % 64);
    if (mode == 2) dr = 128 * (r / 64) + 64 + (r % 64);
    uint8_t* dq = dst + (size_t)dr * cols;
    for (int c = threadIdx.x; c < cols; c += blockDim.x) dq[c] = to_e4m3(sr[c] * inv);
    if (threadIdx.x == 0) dst_scale[dr] = s;
}

}  // namespace

cudaError_t launch_rmsnorm_e4m3(const float* x, const float* w, uint8_t* q, float* scale,
                                int rows, int cols, float eps, cudaStream_t s,
                                const int* row_idx) {
    LaunchScope ls(DTP_K_RMSNORM, s);
    if (cols % 4 || cols > 16 * 1024) return cudaErrorInvalidValue;
    int threads = ((cols + 15) / 16 + 31) / 32 * 32;       // threads * 16 >= cols
    if (threads < 32) threads = 32;
    rmsnorm_e4m3_kernel<<<rows, threads, 0, s>>>(x, w, q, scale, cols, eps, row_idx);
    return cudaGetLastError();
}

cudaError_t launch_quant_rows_e4m3(const __nv_bfloat16* x, int ldx, int rows, int cols,
                                   uint8_t* q, float* scale, cudaStream_t s) {
    LaunchScope ls(DTP_K_OTHER, s);
    if (cols % 8 || ldx % 8) return cudaErrorInvalidValue;
    quant_rows_kernel<<<rows, 256, 0, s>>>(x, ldx, cols, q, scale);
    return cudaGetLastError();
}

cudaError_t launch_pack_e4m3(const float* src, int rows, int cols, uint8_t* dst, float* dst_scale,
                             int mode, cudaStream_t s) {
    LaunchScope ls(DTP_K_OTHER, s);
    pack_e4m3_kernel<<<rows, 256, 0, s>>>(src, cols, dst, dst_scale, mode);
    return cudaGetLastError();
}

}  // namespace dtp
