// SIMT kernels of the prefill pass: embedding gather, RMSNorm, per-head
// QK-norm + NeoX RoPE, the RoPE angle table, SwiGLU, the float32 GEMM and the
// float32/bf16 causal GQA attention used by the exact (float32) path, and the
// weight-packing conversions.
//
// Steps follow "docs.rs memra-engine 0.130.0, src/forward.rs", Model::forward.
#include <math.h>

#include "internal.h"

namespace dtp {

static __device__ unsigned g_simt_err = 0;

unsigned read_clear_simt_errors() {
    unsigned v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_simt_err, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_simt_err, &z, sizeof(z));
    return v;
}

__device__ __forceinline__ float ld_elt(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_elt(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st_elt(float* p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_elt(__nv_bfloat16* p, size_t i, float v) {
    p[i] = __float2bfloat16_rn(v);
}

// Round a float32 to TensorFloat-32 (keep 10 fraction bits), nearest with ties
// to even: add half of the 13 dropped bits' range, minus one unless the kept
// last bit is odd, then clear them.  Finite inputs only.
__device__ __forceinline__ float round_tf32(float x) {
    uint32_t u = __float_as_uint(x);
    u += 0xFFFu + ((u >> 13) & 1u);
    return __uint_as_float(u & ~0x1FFFu);
}
// float32 storage of tf32 values (DTP_TF32): stores round, loads are plain.
struct tf32_t {
    float v;
};
__device__ __forceinline__ float ld_elt(const tf32_t* p, size_t i) { return p[i].v; }
__device__ __forceinline__ void st_elt(tf32_t* p, size_t i, float v) { p[i].v = round_tf32(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Block-wide sum in a fixed order (deterministic).
__device__ float block_sum(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < nw; ++i) t += red[i];
    return t;
}

// ----------------------------------------------------------------------------- embedding
// forward.rs, Model::forward, the embedding step -- row t of x is row tokens[t]
// of the embedding table.  An id >= V raises the token-range error bit and
// leaves a zero row.  With xb, also the bf16 copy of the row and its sum of
// squares ss[t] (the first layer's fused RMSNorm input, one partial per row).
// A bf16 table with d % 8 == 0 moves 8 elements per thread and step (one
// 16-byte load, two 16-byte float stores, one 16-byte bf16 store).
template <typename Tt>
__global__ void embed_kernel(const uint32_t* __restrict__ tokens, int V, int d,
                             const Tt* __restrict__ table, float* __restrict__ x,
                             __nv_bfloat16* __restrict__ xb, float* __restrict__ ss_out) {
    __shared__ float red[32];
    const int t = blockIdx.x;
    const uint32_t id = tokens[t];
    float* xr = x + (size_t)t * d;
    const bool bad = id >= (uint32_t)V;
    if (bad && threadIdx.x == 0) atomicOr(&g_simt_err, ERRBIT_TOKEN_RANGE);
    const Tt* src = table + (size_t)(bad ? 0 : id) * d;
    float ss = 0.f;
    if constexpr (sizeof(Tt) == 2) {
        if ((d & 7) == 0) {
            for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
                const uint4 u = bad ? make_uint4(0, 0, 0, 0)
                                    : *reinterpret_cast<const uint4*>(src + c);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                float v[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[2 * j] = __uint_as_float(w[j] << 16);
                    v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
                }
                *reinterpret_cast<float4*>(xr + c) = make_float4(v[0], v[1], v[2], v[3]);
                *reinterpret_cast<float4*>(xr + c + 4) = make_float4(v[4], v[5], v[6], v[7]);
                if (xb) {
                    *reinterpret_cast<uint4*>(xb + (size_t)t * d + c) = u;   // already bf16
#pragma unroll
                    for (int j = 0; j < 8; ++j) ss = fmaf(v[j], v[j], ss);
                }
            }
            if (ss_out) {
                ss = block_sum(ss, red);
                if (threadIdx.x == 0) ss_out[t] = ss;
            }
            return;
        }
    }
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        const float v = bad ? 0.f : ld_elt(src, c);
        xr[c] = v;
        if (xb) {
            xb[(size_t)t * d + c] = __float2bfloat16_rn(v);
            ss = fmaf(v, v, ss);
        }
    }
    if (ss_out) {
        ss = block_sum(ss, red);
        if (threadIdx.x == 0) ss_out[t] = ss;
    }
}

cudaError_t launch_embed(const uint32_t* tokens, int T, int V, int d, const void* table,
                         int table_dtype, float* x, cudaStream_t s, __nv_bfloat16* xb,
                         float* ss_out) {
    LaunchScope ls(DTP_K_EMBED, s);
    int threads = d >= 256 ? 256 : 64;
    if (table_dtype == DTP_BF16)
        embed_kernel<<<T, threads, 0, s>>>(tokens, V, d, (const __nv_bfloat16*)table, x, xb,
                                           ss_out);
    else
        embed_kernel<<<T, threads, 0, s>>>(tokens, V, d, (const float*)table, x, xb, ss_out);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------- RMSNorm
// forward.rs, Model::forward: the row RMSNorm step (nrows rows of ncols) -- one block per row.
template <typename To>
__global__ void rmsnorm_kernel(const float* __restrict__ x, const float* __restrict__ w,
                               To* __restrict__ y, int cols, float eps,
                               const int* __restrict__ row_idx) {
    __shared__ float red[32];
    const size_t r = blockIdx.x;
    const float* xr = x + (size_t)(row_idx ? row_idx[r] : r) * cols;
    To* yr = y + r * cols;
    float ss = 0.f;
    const bool vec = (cols & 3) == 0;
    if (vec) {
        for (int c = threadIdx.x * 4; c < cols; c += blockDim.x * 4) {
            float4 v = *reinterpret_cast<const float4*>(xr + c);
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
    } else {
        for (int c = threadIdx.x; c < cols; c += blockDim.x) ss += xr[c] * xr[c];
    }
    ss = block_sum(ss, red);
    const float rstd = 1.0f / sqrtf(ss / (float)cols + eps);
    if (vec) {
        for (int c = threadIdx.x * 4; c < cols; c += blockDim.x * 4) {
            float4 v = *reinterpret_cast<const float4*>(xr + c);
            float4 g = *reinterpret_cast<const float4*>(w + c);
            st_elt(yr, c + 0, v.x * rstd * g.x);
            st_elt(yr, c + 1, v.y * rstd * g.y);
            st_elt(yr, c + 2, v.z * rstd * g.z);
            st_elt(yr, c + 3, v.w * rstd * g.w);
        }
    } else {
        for (int c = threadIdx.x; c < cols; c += blockDim.x) st_elt(yr, c, xr[c] * rstd * w[c]);
    }
}

// Register-resident variant for cols % 4 == 0 and cols <= 16 * blockDim: each
// thread holds up to 4 float4 of the row, so x is read from memory once.
template <typename To>
__device__ __forceinline__ void store4(To* y, int c, float a, float b, float cc, float d) {
    st_elt(y, c + 0, a);
    st_elt(y, c + 1, b);
    st_elt(y, c + 2, cc);
    st_elt(y, c + 3, d);
}
template <>
__device__ __forceinline__ void store4(__nv_bfloat16* y, int c, float a, float b, float cc,
                                       float d) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(cc, d);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(y + c) = u;
}

template <typename To>
__global__ void rmsnorm_reg_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                   To* __restrict__ y, int cols, float eps,
                                   const int* __restrict__ row_idx) {
    __shared__ float red[32];
    const size_t r = blockIdx.x;
    const float4* xr =
        reinterpret_cast<const float4*>(x + (size_t)(row_idx ? row_idx[r] : r) * cols);
    To* yr = y + r * cols;
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
    ss = block_sum(ss, red);
    const float rstd = 1.0f / sqrtf(ss / (float)cols + eps);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c4 = threadIdx.x + i * blockDim.x;
        if (c4 < n4) {
            const float4 g = reinterpret_cast<const float4*>(w)[c4];
            store4(yr, 4 * c4, v[i].x * rstd * g.x, v[i].y * rstd * g.y, v[i].z * rstd * g.z,
                   v[i].w * rstd * g.w);
        }
    }
}

cudaError_t launch_rmsnorm(const float* x, const float* w, void* y, int y_dtype, int rows,
                           int cols, float eps, cudaStream_t s, const int* row_idx) {
    LaunchScope ls(DTP_K_RMSNORM, s);
    const bool vec_ok = (cols % 4 == 0) && cols <= 16 * 1024;
    if (vec_ok) {
        int threads = ((cols + 15) / 16 + 31) / 32 * 32;     // threads * 16 >= cols
        if (threads < 32) threads = 32;
        if (y_dtype == DTP_BF16)
            rmsnorm_reg_kernel<<<rows, threads, 0, s>>>(x, w, (__nv_bfloat16*)y, cols, eps,
                                                        row_idx);
        else if (y_dtype == DTP_TF32)
            rmsnorm_reg_kernel<<<rows, threads, 0, s>>>(x, w, (tf32_t*)y, cols, eps, row_idx);
        else
            rmsnorm_reg_kernel<<<rows, threads, 0, s>>>(x, w, (float*)y, cols, eps, row_idx);
        return cudaGetLastError();
    }
    int threads = cols >= 1024 ? 256 : (cols >= 256 ? 128 : 32);
    if (y_dtype == DTP_BF16)
        rmsnorm_kernel<<<rows, threads, 0, s>>>(x, w, (__nv_bfloat16*)y, cols, eps, row_idx);
    else if (y_dtype == DTP_TF32)
        rmsnorm_kernel<<<rows, threads, 0, s>>>(x, w, (tf32_t*)y, cols, eps, row_idx);
    else
        rmsnorm_kernel<<<rows, threads, 0, s>>>(x, w, (float*)y, cols, eps, row_idx);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------- RoPE angles
// cos/sin of angle = pos * base^(-2i/r), computed in float64 and rounded to
// float32 (forward.rs, the NeoX RoPE step: rope_dim_count rotated dims, base freq_base,
// frequency scale 1).
__device__ __forceinline__ float2 rope_cs(double pos, int i, int rope_dims, double base) {
    const double theta = pow(base, -2.0 * (double)i / (double)rope_dims);
    double sn, cs;
    sincos(pos * theta, &sn, &cs);
    return make_float2((float)cs, (float)sn);
}

// row t of the table holds position pos0 + t
__global__ void rope_table_kernel(float2* tab, int T, int half, int rope_dims, double base,
                                  int pos0) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= T * half) return;
    const int t = idx / half, i = idx % half;
    tab[idx] = rope_cs((double)(pos0 + t), i, rope_dims, base);
}

cudaError_t launch_rope_table(float2* tab, int T, int rope_dims, float freq_base,
                              cudaStream_t s, int pos0) {
    LaunchScope ls(DTP_K_OTHER, s);
    const int half = rope_dims / 2, n = T * half;
    rope_table_kernel<<<(n + 255) / 256, 256, 0, s>>>(tab, T, half, rope_dims, (double)freq_base,
                                                      pos0);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------- QK-norm + RoPE
// One block per token; one warp per (token, head) row.  forward.rs: q/k
// `rms_norm(ncols = head_dim, nrows = heads*T)` then `rope_neox`.
template <typename Tx>
__global__ void qk_norm_rope_kernel(Tx* __restrict__ x, int ld, const float* __restrict__ w,
                                    const int32_t* __restrict__ pos, int n_heads, int hd,
                                    int rope_dims, double base, float eps, int head_stride,
                                    int pos0) {
    extern __shared__ float sm[];
    const int t = blockIdx.x, half = rope_dims / 2;
    float2* cs = reinterpret_cast<float2*>(sm);                 // [half]
    float* rowbuf = sm + 2 * half;                              // [warps][hd]
    const double p = pos ? (double)pos[t] : (double)(pos0 + t);
    for (int i = threadIdx.x; i < half; i += blockDim.x) cs[i] = rope_cs(p, i, rope_dims, base);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    float* rb = rowbuf + warp * hd;
    for (int h = warp; h < n_heads; h += nw) {
        Tx* row = x + (size_t)t * ld + (size_t)h * head_stride;
        float ss = 0.f;
        for (int e = lane; e < hd; e += 32) {
            float v = ld_elt(row, e);
            rb[e] = v;
            ss += v * v;
        }
        ss = warp_sum(ss);
        const float rstd = w ? 1.0f / sqrtf(ss / (float)hd + eps) : 1.0f;
        __syncwarp();
        for (int e = lane; e < hd; e += 32) rb[e] = w ? rb[e] * rstd * w[e] : rb[e];
        __syncwarp();
        for (int e = lane; e < hd; e += 32) {
            float y;
            if (e < half) {
                const float2 c = cs[e];
                y = rb[e] * c.x - rb[e + half] * c.y;
            } else if (e < rope_dims) {
                const float2 c = cs[e - half];
                y = rb[e - half] * c.y + rb[e] * c.x;
            } else {
                y = rb[e];
            }
            st_elt(row, e, y);
        }
        __syncwarp();
    }
}

cudaError_t launch_qk_norm_rope(void* x, int dtype, int ld, const float* w_norm,
                                const int32_t* pos, int T, int n_heads, int head_dim,
                                int rope_dims, float freq_base, float eps, cudaStream_t s,
                                int head_stride, int pos0) {
    LaunchScope ls(DTP_K_OTHER, s);
    if (head_stride <= 0) head_stride = head_dim;
    int warps = n_heads < 8 ? n_heads : 8;
    size_t smem = (size_t)(rope_dims + warps * head_dim) * sizeof(float);
    if (dtype == DTP_BF16)
        qk_norm_rope_kernel<<<T, warps * 32, smem, s>>>((__nv_bfloat16*)x, ld, w_norm, pos,
                                                        n_heads, head_dim, rope_dims,
                                                        (double)freq_base, eps, head_stride, pos0);
    else if (dtype == DTP_TF32)     // float32 storage, results rounded to tf32
        qk_norm_rope_kernel<<<T, warps * 32, smem, s>>>((tf32_t*)x, ld, w_norm, pos, n_heads,
                                                        head_dim, rope_dims, (double)freq_base,
                                                        eps, head_stride, pos0);
    else
        qk_norm_rope_kernel<<<T, warps * 32, smem, s>>>((float*)x, ld, w_norm, pos, n_heads,
                                                        head_dim, rope_dims, (double)freq_base,
                                                        eps, head_stride, pos0);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------- SwiGLU
// forward.rs, the FFN activation: act = silu(gate) * up, silu(x) = x / (1 + e^-x).
__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

template <typename T>
__global__ void swiglu_kernel(const T* __restrict__ g, const T* __restrict__ u, T* __restrict__ o,
                              size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        st_elt(o, i, silu_f(ld_elt(g, i)) * ld_elt(u, i));
}

cudaError_t launch_swiglu(const void* gate, const void* up, void* out, int dtype, size_t n,
                          cudaStream_t s) {
    LaunchScope ls(DTP_K_OTHER, s);
    size_t blocks = (n + 255) / 256;
    if (blocks > 65535 * 8) blocks = 65535 * 8;
    if (dtype == DTP_BF16)
        swiglu_kernel<<<(unsigned)blocks, 256, 0, s>>>((const __nv_bfloat16*)gate,
                                                       (const __nv_bfloat16*)up,
                                                       (__nv_bfloat16*)out, n);
    else
        swiglu_kernel<<<(unsigned)blocks, 256, 0, s>>>((const float*)gate, (const float*)up,
                                                       (float*)out, n);
    return cudaGetLastError();
}

// gu [T, 2F] holds gate/up interleaved in 64-column blocks (block b: gate
// columns 64b..64b+63 then up columns 64b..64b+63); act [T, F] (float32, or
// float32 rounded to tf32 when To is tf32_t).
template <typename To>
__global__ void swiglu_interleaved64_kernel(const float* __restrict__ gu, To* __restrict__ act,
                                            int T, int F) {
    const size_t n = (size_t)T * F;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t t = i / F;
        const int f = (int)(i % F);
        const size_t base = t * 2 * F + (size_t)(f / 64) * 128 + (f % 64);
        st_elt(act, i, silu_f(gu[base]) * gu[base + 64]);
    }
}

cudaError_t launch_swiglu_interleaved64(const float* gu, float* act, int T, int F,
                                        cudaStream_t s, int act_dtype) {
    LaunchScope ls(DTP_K_OTHER, s);
    size_t n = (size_t)T * F, blocks = (n + 255) / 256;
    if (blocks > 65535 * 8) blocks = 65535 * 8;
    if (act_dtype == DTP_TF32)
        swiglu_interleaved64_kernel<<<(unsigned)blocks, 256, 0, s>>>(gu, (tf32_t*)act, T, F);
    else
        swiglu_interleaved64_kernel<<<(unsigned)blocks, 256, 0, s>>>(gu, act, T, F);
    return cudaGetLastError();
}

// x[i] = round_tf32(x[i]) in place (float32 storage).
__global__ void round_tf32_kernel(float* __restrict__ x, size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        x[i] = round_tf32(x[i]);
}

cudaError_t launch_round_tf32(float* x, size_t n, cudaStream_t s) {
    LaunchScope ls(DTP_K_OTHER, s);
    size_t blocks = (n + 255) / 256;
    if (blocks > 65535 * 8) blocks = 65535 * 8;
    round_tf32_kernel<<<(unsigned)blocks, 256, 0, s>>>(x, n);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------- f32 GEMM
// y[M, N] = x[M, K] W[N, K]^T (+ residual): 64x64 tile per block, 256 threads,
// 4x4 outputs per thread, K in steps of 16; accumulation order k = 0..K-1.
constexpr int SG_BM = 64, SG_BN = 64, SG_BK = 16;

template <typename To>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const float* __restrict__ x, int ldx,
                                                        const float* __restrict__ W,
                                                        To* __restrict__ y, int ldy, int M, int N,
                                                        int K, const float* residual) {
    __shared__ float As[SG_BK][SG_BM + 4];
    __shared__ float Bs[SG_BK][SG_BN + 4];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int m0 = blockIdx.y * SG_BM, n0 = blockIdx.x * SG_BN;
    // Two-level sum: each run of 4 * SG_BK = 64 products is summed on its own
    // and the runs' sums are added to acc, so rounding grows with sqrt(64) +
    // sqrt(K / 64) rather than sqrt(K) (K reaches 12288 in the down projection).
    float acc[4][4] = {}, part[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += SG_BK) {
        for (int i = threadIdx.x; i < SG_BM * SG_BK; i += 256) {
            const int r = i / SG_BK, c = i % SG_BK;
            const int gm = m0 + r, gk = k0 + c;
            As[c][r] = (gm < M && gk < K) ? x[(size_t)gm * ldx + gk] : 0.f;
            const int gn = n0 + r;
            Bs[c][r] = (gn < N && gk < K) ? W[(size_t)gn * K + gk] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < SG_BK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) part[i][j] = fmaf(a[i], b[j], part[i][j]);
        }
        __syncthreads();
        if ((k0 / SG_BK) % 4 == 3 || k0 + SG_BK >= K) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i][j] += part[i][j];
                    part[i][j] = 0.f;
                }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int gm = m0 + ty * 4 + i;
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int gn = n0 + tx * 4 + j;
            if (gn >= N) continue;
            float v = acc[i][j];
            if (residual) v += residual[(size_t)gm * ldy + gn];
            st_elt(y, (size_t)gm * ldy + gn, v);
        }
    }
}

cudaError_t launch_gemm_simt(const float* x, int ldx, const float* W, void* y, int y_dtype,
                             int ldy, int M, int N, int K, const float* residual,
                             cudaStream_t s, int kind) {
    LaunchScope ls(kind, s);
    dim3 grid((N + SG_BN - 1) / SG_BN, (M + SG_BM - 1) / SG_BM);
    if (y_dtype == DTP_BF16)
        gemm_simt_kernel<<<grid, 256, 0, s>>>(x, ldx, W, (__nv_bfloat16*)y, ldy, M, N, K,
                                              residual);
    else
        gemm_simt_kernel<<<grid, 256, 0, s>>>(x, ldx, W, (float*)y, ldy, M, N, K, residual);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------- SIMT attention
// forward.rs, Model::forward, the causal attention step over all T keys with
// scale 1/sqrt(head_dim): one warp per (query t, head i); keys in chunks of 32 (one
// per lane), online softmax in float32 with expf.  kv head = i / (h / g).
// Query row t sees keys k0 .. t + q_pos0: k0 = t - tok_pos[t] for packed
// sequences, else 0; q_pos0 > 0 when the queries follow q_pos0 earlier keys
// held in k / v (chunked prefill).
template <typename T, bool VT>
__global__ void attn_simt_kernel(const T* __restrict__ q, int ldq, const T* __restrict__ k,
                                 int ldk, const T* __restrict__ v, int ldv, T* __restrict__ out,
                                 int ldo, int Tn, int n_head, int n_head_kv, int hd, float scale,
                                 const int* __restrict__ tok_pos, int q_head_stride, int q_pos0) {
    extern __shared__ float sm[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x * (blockDim.x >> 5) + warp;
    const int head = blockIdx.y;
    const int kvh = head / (n_head / n_head_kv);
    float* qs = sm + warp * hd;
    if (t >= Tn) return;
    for (int e = lane; e < hd; e += 32)
        qs[e] = ld_elt(q, (size_t)t * ldq + (size_t)head * q_head_stride + e);
    __syncwarp();
    constexpr int MAXD = 8;                 // hd <= 256
    float acc[MAXD];
#pragma unroll
    for (int j = 0; j < MAXD; ++j) acc[j] = 0.f;
    float m = -INFINITY, l = 0.f;
    const int k0 = tok_pos ? t - tok_pos[t] : 0;       // first key of this query's sequence
    const int kl = tok_pos ? t : t + q_pos0;            // last key it sees
    for (int s0 = k0; s0 <= kl; s0 += 32) {
        const int s = s0 + lane;
        float sc = -INFINITY;
        if (s <= kl) {
            const T* kr = k + (size_t)s * ldk + (size_t)kvh * hd;
            float dot = 0.f;
            for (int e = 0; e < hd; ++e) dot = fmaf(qs[e], ld_elt(kr, e), dot);
            sc = dot * scale;
        }
        const float mc = warp_max(sc);
        const float mn = fmaxf(m, mc);
        const float alpha = expf(m - mn);     // m = -inf on the first chunk -> 0
        const float p = (s <= kl) ? expf(sc - mn) : 0.f;
        l = l * alpha + warp_sum(p);
        // this chunk's sum of p v on its own, then folded into the rescaled total
        // (a two-level sum: rounding grows with sqrt(32) + sqrt(T / 32), not sqrt(T))
        float cacc[MAXD];
#pragma unroll
        for (int j = 0; j < MAXD; ++j) cacc[j] = 0.f;
        const int nk = min(32, kl - s0 + 1);
        for (int jj = 0; jj < nk; ++jj) {
            const float pj = __shfl_sync(0xffffffffu, p, jj);
            const int sk = s0 + jj;
#pragma unroll
            for (int j = 0; j < MAXD; ++j) {
                const int e = lane + 32 * j;
                if (e < hd) {
                    const float vv = VT ? ld_elt(v, (size_t)(kvh * hd + e) * ldv + sk)
                                        : ld_elt(v, (size_t)sk * ldv + (size_t)kvh * hd + e);
                    cacc[j] = fmaf(pj, vv, cacc[j]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < MAXD; ++j) acc[j] = fmaf(acc[j], alpha, cacc[j]);
        m = mn;
    }
    const float inv = 1.0f / l;
#pragma unroll
    for (int j = 0; j < MAXD; ++j) {
        const int e = lane + 32 * j;
        if (e < hd) st_elt(out, (size_t)t * ldo + (size_t)head * hd + e, acc[j] * inv);
    }
}

cudaError_t launch_attn_simt(const void* q, int ldq, const void* k, int ldk, const void* v,
                             int ldv, int v_t, void* out, int ldo, int dtype, int T,
                             int n_head, int n_head_kv, int head_dim, float scale,
                             cudaStream_t s, const int* tok_pos, int q_head_stride,
                             int q_pos0) {
    LaunchScope ls(DTP_K_ATTN, s);
    if (q_head_stride <= 0) q_head_stride = head_dim;
    const int warps = 4;
    dim3 grid((T + warps - 1) / warps, n_head);
    size_t smem = (size_t)warps * head_dim * sizeof(float);
    if (dtype == DTP_BF16) {
        using B = __nv_bfloat16;
        if (v_t)
            attn_simt_kernel<B, true><<<grid, warps * 32, smem, s>>>(
                (const B*)q, ldq, (const B*)k, ldk, (const B*)v, ldv, (B*)out, ldo, T, n_head,
                n_head_kv, head_dim, scale, tok_pos, q_head_stride, q_pos0);
        else
            attn_simt_kernel<B, false><<<grid, warps * 32, smem, s>>>(
                (const B*)q, ldq, (const B*)k, ldk, (const B*)v, ldv, (B*)out, ldo, T, n_head,
                n_head_kv, head_dim, scale, tok_pos, q_head_stride, q_pos0);
    } else {
        if (v_t)
            attn_simt_kernel<float, true><<<grid, warps * 32, smem, s>>>(
                (const float*)q, ldq, (const float*)k, ldk, (const float*)v, ldv, (float*)out,
                ldo, T, n_head, n_head_kv, head_dim, scale, tok_pos, q_head_stride, q_pos0);
        else
            attn_simt_kernel<float, false><<<grid, warps * 32, smem, s>>>(
                (const float*)q, ldq, (const float*)k, ldk, (const float*)v, ldv, (float*)out,
                ldo, T, n_head, n_head_kv, head_dim, scale, tok_pos, q_head_stride, q_pos0);
    }
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------- v transpose
// v [T, width] -> vt [width, ldt] (key index contiguous), 32x32 tiles via smem.
template <typename E>
__global__ void transpose_v_kernel(const E* __restrict__ v, int ldv, E* __restrict__ vt, int T,
                                   int width, int ldt) {
    __shared__ E tile[32][33];
    const int t0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int t = t0 + i, c = c0 + threadIdx.x;
        tile[i][threadIdx.x] = (t < T && c < width) ? v[(size_t)t * ldv + c] : E(0.f);
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int c = c0 + i, t = t0 + threadIdx.x;
        if (c < width && t < T) vt[(size_t)c * ldt + t] = tile[threadIdx.x][i];
    }
}

// bf16 v [T, width] -> f16 v^T [width, ldt]: each bf16 value converted to f16
// (exact from 2^-14 up to 65504; the bf16 attention's P V^T MMA takes f16
// operands); a value beyond the f16 range raises ERRBIT_VRANGE.
__global__ void transpose_v_f16_kernel(const __nv_bfloat16* __restrict__ v, int ldv,
                                       __half* __restrict__ vt, int T, int width, int ldt) {
    __shared__ float tile[32][33];
    const int t0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int t = t0 + i, c = c0 + threadIdx.x;
        tile[i][threadIdx.x] = (t < T && c < width) ? __bfloat162float(v[(size_t)t * ldv + c]) : 0.f;
    }
    __syncthreads();
    bool over = false;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int c = c0 + i, t = t0 + threadIdx.x;
        if (c < width && t < T) {
            const float x = tile[threadIdx.x][i];
            over |= !(fabsf(x) <= 65504.0f);
            vt[(size_t)c * ldt + t] = __float2half_rn(x);
        }
    }
    if (over) atomicOr(&g_simt_err, ERRBIT_VRANGE);
}

cudaError_t launch_transpose_v(const __nv_bfloat16* v, __half* vt, int T, int width,
                               int ldt, cudaStream_t s) {
    LaunchScope ls(DTP_K_OTHER, s);
    dim3 grid((T + 31) / 32, (width + 31) / 32), block(32, 8);
    transpose_v_f16_kernel<<<grid, block, 0, s>>>(v, width, vt, T, width, ldt);
    return cudaGetLastError();
}

cudaError_t launch_transpose_v_f32(const float* v, int ldv, float* vt, int T, int width, int ldt,
                                   cudaStream_t s) {
    LaunchScope ls(DTP_K_OTHER, s);
    dim3 grid((T + 31) / 32, (width + 31) / 32), block(32, 8);
    transpose_v_kernel<<<grid, block, 0, s>>>(v, ldv, vt, T, width, ldt);
    return cudaGetLastError();
}

// x[r, c] = round_tf32(x[r, c]) for r < rows, c < cols (row stride ld).
__global__ void round_tf32_rows_kernel(float* __restrict__ x, int ld, int rows, int cols) {
    const size_t n = (size_t)rows * cols;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        float* e = x + (i / cols) * ld + (i % cols);
        *e = round_tf32(*e);
    }
}

cudaError_t launch_round_tf32_rows(float* x, int ld, int rows, int cols, cudaStream_t s) {
    LaunchScope ls(DTP_K_OTHER, s);
    size_t n = (size_t)rows * cols, blocks = (n + 255) / 256;
    if (blocks > 65535 * 8) blocks = 65535 * 8;
    round_tf32_rows_kernel<<<(unsigned)blocks, 256, 0, s>>>(x, ld, rows, cols);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------- packing
// dst row for source row r: mode 0 -> r; mode 1 (gate) -> 128*(r/64) + r%64;
// mode 2 (up) -> 128*(r/64) + 64 + r%64.
// col_scale (optional, [cols]): dst = src * col_scale[c], rounded once (a norm
// weight folded into the matrix that follows the norm).
template <typename To>
__global__ void pack_matrix_kernel(const float* __restrict__ src, int rows, int cols,
                                   To* __restrict__ dst, int mode,
                                   const float* __restrict__ col_scale) {
    const size_t n = (size_t)rows * cols;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const int r = (int)(i / cols), c = (int)(i % cols);
        int dr = r;
        if (mode == 1) dr = 128 * (r / 64) + (r % 64);
        if (mode == 2) dr = 128 * (r / 64) + 64 + (r % 64);
        st_elt(dst, (size_t)dr * cols + c, col_scale ? src[i] * col_scale[c] : src[i]);
    }
}

cudaError_t launch_pack_matrix(const float* src, int rows, int cols, void* dst, int to_dtype,
                               int mode, cudaStream_t s, const float* col_scale) {
    LaunchScope ls(DTP_K_OTHER, s);
    size_t n = (size_t)rows * cols, blocks = (n + 255) / 256;
    if (blocks > 65535 * 16) blocks = 65535 * 16;
    if (to_dtype == DTP_BF16)
        pack_matrix_kernel<<<(unsigned)blocks, 256, 0, s>>>(src, rows, cols, (__nv_bfloat16*)dst,
                                                            mode, col_scale);
    else if (to_dtype == DTP_TF32)
        pack_matrix_kernel<<<(unsigned)blocks, 256, 0, s>>>(src, rows, cols, (tf32_t*)dst, mode,
                                                            col_scale);
    else
        pack_matrix_kernel<<<(unsigned)blocks, 256, 0, s>>>(src, rows, cols, (float*)dst, mode,
                                                            col_scale);
    return cudaGetLastError();
}

__global__ void copy_f32_kernel(const float* __restrict__ a, float* __restrict__ b, size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        b[i] = a[i];
}

cudaError_t launch_copy_f32(const float* src, float* dst, size_t n, cudaStream_t s) {
    LaunchScope ls(DTP_K_OTHER, s);
    size_t blocks = (n + 255) / 256;
    if (blocks > 65535 * 8) blocks = 65535 * 8;
    copy_f32_kernel<<<(unsigned)blocks, 256, 0, s>>>(src, dst, n);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------- packed sequences
// One block: checks cu_seqlens (cu[0] = 0, non-decreasing, cu[n] = total) and
// writes the exclusive prefixes tile_start (ceil(len/128)) and vcol_start
// (len rounded up to 8, so every sequence's v^T block starts on a 16-byte
// boundary), and last_row[b] = cu[b+1] - 1 (clamped to >= 0).  On invalid input
// it raises ERRBIT_SEQLENS and writes an empty schedule (all zeros).
__global__ void seq_meta_kernel(const int* __restrict__ cu, int n, int total,
                                int* __restrict__ tile_start, int* __restrict__ vcol_start,
                                int* __restrict__ last_row, int* __restrict__ bad_flag) {
    __shared__ int s_tiles[1024], s_cols[1024];
    __shared__ int s_bad;
    const int tid = threadIdx.x, nt = blockDim.x;
    if (tid == 0) s_bad = (cu[0] != 0 || cu[n] != total);
    __syncthreads();
    const int per = (n + nt - 1) / nt, b0 = tid * per, b1 = min(n, b0 + per);
    int tiles = 0, cols = 0, bad = 0;
    for (int b = b0; b < b1; ++b) {
        const int len = cu[b + 1] - cu[b];
        if (len < 0) bad = 1;
        const int L = len < 0 ? 0 : len;
        tiles += (L + 127) / 128;
        cols += (L + 7) / 8 * 8;
    }
    if (bad) atomicOr(&s_bad, 1);
    s_tiles[tid] = tiles;
    s_cols[tid] = cols;
    __syncthreads();
    if (tid == 0) {            // exclusive scan of the per-thread sums (nt <= 1024)
        int a = 0, c = 0;
        for (int i = 0; i < nt; ++i) {
            const int ta = s_tiles[i], tc = s_cols[i];
            s_tiles[i] = a;
            s_cols[i] = c;
            a += ta;
            c += tc;
        }
    }
    __syncthreads();
    const int badall = s_bad;
    int a = badall ? 0 : s_tiles[tid], c = badall ? 0 : s_cols[tid];
    for (int b = b0; b < b1; ++b) {
        tile_start[b] = a;
        vcol_start[b] = c;
        last_row[b] = badall ? 0 : max(cu[b + 1] - 1, 0);
        if (!badall) {
            const int L = cu[b + 1] - cu[b];
            a += (L + 127) / 128;
            c += (L + 7) / 8 * 8;
        }
    }
    if (b0 < b1 && b1 == n) tile_start[n] = a;      // the thread whose range ends at n
    if (tid == 0) {
        *bad_flag = badall;
        if (badall) {
            tile_start[n] = 0;
            atomicOr(&g_simt_err, ERRBIT_SEQLENS);
        }
    }
}

// Per token t of sequence b: tok_pos = t - cu[b], tok_vcol = vcol_start[b] + tok_pos,
// both clamped in bounds; with an invalid schedule every token maps to itself.
__global__ void tok_meta_kernel(const int* __restrict__ cu, const int* __restrict__ vcol_start,
                                const int* __restrict__ bad_flag, int n, int total,
                                long long vt_cols, int* __restrict__ tok_pos,
                                int* __restrict__ tok_vcol) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= total) return;
    int pos = t, col = t;
    if (!*bad_flag) {
        int lo = 0, hi = n - 1;            // last b with cu[b] <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cu[mid] <= t) lo = mid;
            else hi = mid - 1;
        }
        pos = t - cu[lo];
        col = vcol_start[lo] + pos;
    }
    tok_pos[t] = min(max(pos, 0), total - 1);
    tok_vcol[t] = (int)min((long long)max(col, 0), vt_cols - 1);
}

cudaError_t launch_seq_meta(const int* cu_seqlens, int n_seq, int total, int* tile_start,
                            int* vcol_start, int* last_row, int* tok_pos, int* tok_vcol,
                            long long vt_cols, cudaStream_t s) {
    LaunchScope ls(DTP_K_OTHER, s);
    // the flag shares tile_start's allocation tail: tile_start has n_seq + 2 slots
    int* bad = tile_start + n_seq + 1;
    int threads = n_seq < 1024 ? ((n_seq + 31) / 32) * 32 : 1024;
    if (threads < 32) threads = 32;
    seq_meta_kernel<<<1, threads, 0, s>>>(cu_seqlens, n_seq, total, tile_start, vcol_start,
                                          last_row, bad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    LaunchScope ls2(DTP_K_OTHER, s);
    tok_meta_kernel<<<(total + 255) / 256, 256, 0, s>>>(cu_seqlens, vcol_start, bad, n_seq, total,
                                                         vt_cols, tok_pos, tok_vcol);
    return cudaGetLastError();
}

// gated attention (f32 path): attn *= sigmoid(gate), gate head blocks gstride apart
__global__ void gate_mul_f32_kernel(float* __restrict__ attn, int lda, const float* __restrict__ gate,
                                    int ldg, int gstride, int T, int n_head, int hd) {
    const size_t n = (size_t)T * n_head * hd;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t t = i / ((size_t)n_head * hd);
        const int r = (int)(i % ((size_t)n_head * hd)), h = r / hd, e = r % hd;
        const float g = gate[t * ldg + (size_t)h * gstride + e];
        attn[t * lda + r] = attn[t * lda + r] / (1.0f + expf(-g));
    }
}

cudaError_t launch_gate_mul_f32(float* attn, int lda, const float* gate, int ldg, int gstride,
                                int T, int n_head, int head_dim, cudaStream_t s) {
    LaunchScope ls(DTP_K_OTHER, s);
    size_t n = (size_t)T * n_head * head_dim, blocks = (n + 255) / 256;
    if (blocks > 65535 * 8) blocks = 65535 * 8;
    gate_mul_f32_kernel<<<(unsigned)blocks, 256, 0, s>>>(attn, lda, gate, ldg, gstride, T, n_head,
                                                         head_dim);
    return cudaGetLastError();
}

__global__ void copy_rows_f32_kernel(const float* __restrict__ a, int lda, float* __restrict__ b,
                                     int ldb, int rows, int cols) {
    const size_t n = (size_t)rows * cols;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t r = i / cols, c = i % cols;
        b[r * ldb + c] = a[r * lda + c];
    }
}

cudaError_t launch_copy_rows_f32(const float* src, int lds, float* dst, int ldd, int rows,
                                 int cols, cudaStream_t s) {
    LaunchScope ls(DTP_K_OTHER, s);
    size_t n = (size_t)rows * cols, blocks = (n + 255) / 256;
    if (blocks > 65535 * 8) blocks = 65535 * 8;
    copy_rows_f32_kernel<<<(unsigned)blocks, 256, 0, s>>>(src, lds, dst, ldd, rows, cols);
    return cudaGetLastError();
}

}  // namespace dtp
