// tcgen05 tensor-core GEMM for the projections, the FFN and the lm_head
// (forward.rs, Model::forward: every projection matmul of the layer and the head), with the
// neighbouring elementwise steps fused into the epilogue:
//   EPI_STORE   y = x W^T (+ residual)      -- O / down projections (residual adds,
//                                              forward.rs, the residual adds) and the lm_head
//   EPI_QKV     per-head QK-RMSNorm + NeoX RoPE on q and k, v stored transposed
//   EPI_SWIGLU  silu(gate) * up on the interleaved gate/up product (the FFN activation)
//
// D[M, N] = A[M, K] B[N, K]^T with A = activations, B = weights, both
// K-contiguous and of one operand kind:
//   OP_BF16  bf16 (kind::f16)
//   OP_TF32  float32 holding tf32 values (kind::tf32; EPI_STORE only)
//   OP_E4M3  e4m3 with a float32 scale per A row and per B row (kind::f8f6f4):
//            the epilogue reads s_a[m] * s_b[n] * acc[m, n]
// A stage holds 128 bytes of K per row (64 bf16, 32 tf32, 128 e4m3).  One
// persistent CTA per SM; the CTAs run in clusters of two, and a pair walks
// 256 x BN output tiles (CTA rank r: rows 128r..128r+127 of the tile):
//   warp 0      TMA producer: the CTA's 128-row A box and its BN/2-row half of
//               the B box (128-byte swizzle) into a STAGES-deep shared-memory
//               ring; both CTAs count their bytes on the even CTA's full
//               barrier, and each waits on its own empty barrier
//   warp 1      (even CTA) one thread issues tcgen05.mma.cta_group::2 (M=256,
//               N=BN, K=16): A from both CTAs' rings, B split between them, D
//               rows of each CTA in its own TMEM; two accumulators (2*BN
//               columns) so the epilogue of tile i overlaps the main loop of
//               tile i+1; its commits arrive on the barriers of both CTAs
//   warps 2..5  epilogue (both CTAs): tcgen05.ld (TMEM lane = output row),
//               fused math, global stores
// A pair holds one B tile between two SMs, so a stage is 32 KB instead of 48
// and the ring 6 deep instead of 4 (BN = 256).
#include <math.h>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace dtp {

// Every wait of these kernels lets try_wait suspend the thread (up to 1 ms, or
// until the phase completes): the producer, MMA and epilogue threads wait for
// long stretches, and looping on short suspensions took issue slots and power
// from the rest of the SM.  Against the short default, alternated on the 8B
// forward (ms per step): gate/up 16.00 vs 16.42, down 9.23 vs 9.82, QKV 4.93
// vs 5.09, O 3.97 vs 4.02; the whole step 97.5k vs 95.2k tokens/s.  (The
// attention kernel keeps the short default: its softmax/MMA hand-offs are
// latency-bound, and the long suspension made it 4% slower.)
constexpr bool kSuspendWaits = true;

static __device__ unsigned g_gemm_err = 0;

unsigned read_clear_gemm_errors() {
    unsigned v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_err, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_gemm_err, &z, sizeof(z));
    return v;
}

// One thread waits on an mbarrier nothing arrives at: the bounded wait gives up,
// raises the error word and the kernel returns.
__global__ void selftest_wait_kernel() {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::wait_bounded<kSuspendWaits>(&bar, 0, &abort_flag, &g_gemm_err, ERRBIT_TIMEOUT);
    }
}

cudaError_t launch_selftest_wait(cudaStream_t s) {
    LaunchScope ls(DTP_K_OTHER, s);
    selftest_wait_kernel<<<1, 32, 0, s>>>();
    return cudaGetLastError();
}

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 192;
// CTAs per cluster: every GEMM runs as CTA pairs with cta_group::2 MMAs
// (kernel parameter CL = 2).  Against single CTAs (CL = 1) on the 8B forward,
// alternated in one process: gate/up 16.5 vs 17.4 ms per step, down 9.7 vs
// 10.0, QKV 5.2 vs 5.4, O 4.0 vs 4.2, lm_head 2.6 vs 3.0.
constexpr int kCluster = 2;

constexpr int kSmemLimit = 232448;   // dynamic shared memory one CTA may use (227 KB)


// CL = 2: a CTA pair computes a 256 x BN tile with cta_group::2 MMAs; each CTA
// holds its 128 A rows and half of the B rows, so a stage is smaller and the
// ring deeper.
template <int BN, int CL = 1>
struct Cfg {
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = (BN / CL) * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // The 224-wide tile gives the epilogue staging to the pipeline (the main
    // loop is latency-bound: its depth matters more than store efficiency
    // there) and stores directly from registers.
    static constexpr bool TMA_OUT = BN != 224;
    // two accumulators; the second starts at a 256-column boundary when BN > 128
    static constexpr int ACC_STRIDE = BN <= 128 ? 128 : 256;
    static constexpr int TMEM_COLS = 2 * ACC_STRIDE;
    // epilogue staging: per epilogue warp two 32-row x 128-byte boxes (4 KB each)
    static constexpr int EPI_BUF = 4096;
    static constexpr int EPI_BYTES = TMA_OUT ? 4 * 2 * EPI_BUF : 0;
    static constexpr int BAR_BYTES = 256;
    // as many stages as fit: 6 / 5 / 4 for BN = 128 / 224 / 256, 8 / 7 / 6 in pairs
    static constexpr int STAGES_FIT = (kSmemLimit - 1024 - BAR_BYTES - EPI_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
    static_assert((2 * STAGES + 13) * 8 + 8 <= BAR_BYTES, "barrier area");
    static_assert(SMEM_BYTES <= kSmemLimit, "shared memory");
};

struct Params {
    int M, N, K;
    int tiles_m, tiles_n, num_kb;
    int vec_ok;     // y row stride / base allow 16-byte vector stores
    int tma_out;    // outputs go through shared-memory staging and TMA stores
    GemmEpiArgs ea;
};

// Per-epilogue-warp staging state: two 32-row x 128-byte boxes in the
// 128-byte-swizzle layout TMA expects (16-byte chunk j of row r at
// r*128 + ((j ^ (r & 7)) << 4)), their residual-load barriers, and a running
// buffer counter.  Lane 0 issues every bulk copy.
struct EpiStage {
    uint8_t* buf[2];
    uint64_t* rbar[2];
    uint32_t rphase[2];
    uint32_t pending[2];    // a residual load into buf[b] not yet waited for
    uint32_t cnt;
    int lane;
    int row0;           // global row of this warp's lane 0
};

__device__ __forceinline__ void stage_put16(uint8_t* buf, int lane, int chunk, uint4 v) {
    *reinterpret_cast<uint4*>(buf + lane * 128 + ((chunk ^ (lane & 7)) << 4)) = v;
}
__device__ __forceinline__ uint4 stage_get16(const uint8_t* buf, int lane, int chunk) {
    return *reinterpret_cast<const uint4*>(buf + lane * 128 + ((chunk ^ (lane & 7)) << 4));
}

__device__ __forceinline__ float f32(uint32_t u) { return __uint_as_float(u); }

// Accumulator columns taddr .. taddr+31 of this thread's row (TMEM address
// taddr = tbase + column offset in the tile), scaled by s_a[row] * s_b[col]
// when the operands carry scales (SC: OP_E4M3).  Whole warp.
template <bool SC>
__device__ __forceinline__ void acc_ld32(const Params& p, uint32_t tbase, uint32_t taddr, int grow,
                                         int n0, uint32_t (&r)[32], float rowmul = 1.f) {
    ptx::tmem_ld32(taddr, r);
    if constexpr (!SC) {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(f32(r[j]) * rowmul);
    } else {
        const int col = n0 + (int)(taddr - tbase);
        const float sa = (grow < p.M ? p.ea.a_scale[grow] : 0.f) * rowmul;
        float sb[32];
        if (col + 32 <= p.N && (reinterpret_cast<uintptr_t>(p.ea.b_scale + col) & 15) == 0) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {      // the same 32 scales in every lane
                const float4 v = *reinterpret_cast<const float4*>(p.ea.b_scale + col + j);
                sb[j] = v.x;
                sb[j + 1] = v.y;
                sb[j + 2] = v.z;
                sb[j + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) sb[j] = col + j < p.N ? p.ea.b_scale[col + j] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(f32(r[j]) * (sa * sb[j]));
    }
}

// Store 32 consecutive floats (as float or bf16) to dst (16-byte aligned when vec).
__device__ __forceinline__ void store_row32(float* dst, const float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
}
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
        uint4 u;
        u.x = ptx::pack_bf16x2(v[j + 0], v[j + 1]);
        u.y = ptx::pack_bf16x2(v[j + 2], v[j + 3]);
        u.z = ptx::pack_bf16x2(v[j + 4], v[j + 5]);
        u.w = ptx::pack_bf16x2(v[j + 6], v[j + 7]);
        *reinterpret_cast<uint4*>(dst + j) = u;
    }
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// 32 values of one v^T column run (stride ld): v is rounded to bf16, as every
// attention operand of the bf16 path, and stored as f16 (the P V^T MMA takes
// f16 operands), which holds the bf16 value exactly from 2^-14 up to 65504 and
// smaller ones on its subnormal grid.  A value beyond the f16 range raises
// ERRBIT_VRANGE.
__device__ __forceinline__ void store_vt32(__half* dst, long long ld, const uint32_t (&r)[32]) {
    bool over = false;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float vb = __bfloat162float(__float2bfloat16_rn(__uint_as_float(r[j])));
        over |= !(fabsf(vb) <= 65504.0f);
        dst[(size_t)j * ld] = __float2half_rn(vb);
    }
    if (over) atomicOr(&g_gemm_err, ERRBIT_VRANGE);
}

// The fused RMSNorm's row scale 1 / sqrt(mean(x^2) + eps) from the producer's
// per-tile partial sums (summed in tile order), or 1 when the GEMM has none.
__device__ __forceinline__ float row_rstd(const GemmEpiArgs& ea, int grow, int M) {
    if (!ea.ss_in || grow >= M) return 1.f;
    float ss = 0.f;
    for (int t = 0; t < ea.n_ss; ++t) ss += ea.ss_in[(size_t)t * ea.ld_ss + grow];
    return 1.0f / sqrtf(ss / (float)ea.norm_cols + ea.norm_eps);
}

// ----------------------------------------------------------------------------- epilogues
template <int BN, bool SC>
__device__ __forceinline__ void epi_store(const Params& p, uint32_t tbase, int grow, int n0) {
    const GemmEpiArgs& ea = p.ea;
    float ss = 0.f;                                  // fused RMSNorm: this tile's sum of y^2
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
        uint32_t r[32];
        __syncwarp();
        acc_ld32<SC>(p, tbase, tbase + c, grow, n0, r);
        const int col0 = n0 + c;
        if (col0 >= p.N) break;                     // warp-uniform
        if (grow >= p.M) continue;                  // the next tcgen05.ld reconverges below
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = f32(r[j]);
        const size_t off = (size_t)grow * ea.ldy + col0;
        if (p.vec_ok && col0 + 32 <= p.N) {
            if (ea.residual) {
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    float4 a = *reinterpret_cast<const float4*>(ea.residual + off + j);
                    v[j] += a.x; v[j + 1] += a.y; v[j + 2] += a.z; v[j + 3] += a.w;
                }
            }
            if (ea.y_dtype == DTP_F32)
                store_row32(reinterpret_cast<float*>(ea.y) + off, v);
            else
                store_row32(reinterpret_cast<__nv_bfloat16*>(ea.y) + off, v);
            if (ea.xb) {
#pragma unroll
                for (int j = 0; j < 32; ++j) ss = fmaf(v[j], v[j], ss);
                store_row32(ea.xb + off, v);
            }
        } else {
            for (int j = 0; j < 32 && col0 + j < p.N; ++j) {
                float x = v[j];
                if (ea.residual) x += ea.residual[off + j];
                if (ea.y_dtype == DTP_F32)
                    reinterpret_cast<float*>(ea.y)[off + j] = x;
                else
                    reinterpret_cast<__nv_bfloat16*>(ea.y)[off + j] = __float2bfloat16_rn(x);
                if (ea.xb) {
                    ss = fmaf(x, x, ss);
                    ea.xb[off + j] = __float2bfloat16_rn(x);
                }
            }
        }
    }
    if (ea.ss_out && grow < p.M) ea.ss_out[(size_t)(n0 / BN) * ea.ld_ss + grow] = ss;
}

// q/k heads: RMSNorm over head_dim with q_norm/k_norm, then NeoX RoPE from the
// cos/sin table; v heads: stored transposed (key index contiguous).
template <int BN, bool SC>
__device__ __forceinline__ void epi_qkv(const Params& p, uint32_t tbase, int grow, int n0) {
    const GemmEpiArgs& ea = p.ea;
    const float rsc = row_rstd(ea, grow, p.M);     // fused RMSNorm row scale (or 1)
    const int hd = ea.head_dim, half = ea.rope_dims / 2;
    const int nq = ea.n_head * hd, nk = ea.n_head_kv * hd;
    const bool live = grow < p.M;
    const int nqc = ea.q_gated ? 2 * nq : nq;      // q region (with the gate rows)
#pragma unroll 1
    for (int h0 = 0; h0 < BN; h0 += hd) {
        const int col = n0 + h0;
        if (col >= p.N) break;
        const uint32_t th = tbase + h0;
        const int blk = col / hd;
        if (ea.q_gated && col < nqc && (blk & 1)) {
            // gate block of head blk/2: stored raw (bf16) for the attention output
#pragma unroll 1
            for (int c = 0; c < hd; c += 32) {
                uint32_t r[32];
                __syncwarp();
                acc_ld32<SC>(p, tbase, th + c, grow, n0, r, rsc);
                if (live) {
                    float y[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) y[j] = f32(r[j]);
                    store_row32(ea.gate + (size_t)grow * nq + (blk >> 1) * hd + c, y);
                }
            }
            continue;
        }
        if (col < nqc + nk) {
            const bool isq = col < nqc;
            const int qcol = ea.q_gated ? (blk >> 1) * hd : col;    // column in q
            const float* w = isq ? ea.q_norm : ea.k_norm;
            float ss = 0.f;
#pragma unroll 1
            for (int c = 0; c < hd; c += 32) {
                uint32_t r[32];
                __syncwarp();
                acc_ld32<SC>(p, tbase, th + c, grow, n0, r, rsc);
#pragma unroll
                for (int j = 0; j < 32; ++j) ss = fmaf(f32(r[j]), f32(r[j]), ss);
            }
            const float rstd = 1.0f / sqrtf(ss / (float)hd + ea.eps);
            __nv_bfloat16* dst = isq ? ea.q + (size_t)grow * nq + qcol
                                     : ea.k + (size_t)grow * nk + (col - nqc);
#pragma unroll 1
            for (int i0 = 0; i0 < half; i0 += 32) {
                uint32_t ra[32], rb[32];
                __syncwarp();
                acc_ld32<SC>(p, tbase, th + i0, grow, n0, ra, rsc);
                acc_ld32<SC>(p, tbase, th + half + i0, grow, n0, rb, rsc);
                if (live) {
                    const int pos = ea.tok_pos ? ea.tok_pos[grow] : grow;
                    // (cos, sin) pairs j, j+1 in one 16-byte load: rows of the table
                    // and i0 are multiples of 32 pairs
                    const float4* cs = reinterpret_cast<const float4*>(ea.rope + (size_t)pos * half + i0);
                    float ya[32], yb[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float a = f32(ra[j]) * rstd * w[i0 + j];
                        const float b = f32(rb[j]) * rstd * w[half + i0 + j];
                        const float4 c4 = cs[j >> 1];
                        const float2 c = (j & 1) ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y);
                        ya[j] = a * c.x - b * c.y;
                        yb[j] = a * c.y + b * c.x;
                    }
                    store_row32(dst + i0, ya);
                    store_row32(dst + half + i0, yb);
                }
            }
#pragma unroll 1
            for (int c = ea.rope_dims; c < hd; c += 32) {
                uint32_t r[32];
                __syncwarp();
                acc_ld32<SC>(p, tbase, th + c, grow, n0, r, rsc);
                if (live) {
                    float y[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) y[j] = f32(r[j]) * rstd * w[c + j];
                    store_row32(dst + c, y);
                }
            }
        } else {
            const int vcol = col - nqc - nk;
#pragma unroll 1
            for (int c = 0; c < hd; c += 32) {
                uint32_t r[32];
                __syncwarp();
                acc_ld32<SC>(p, tbase, th + c, grow, n0, r, rsc);
                if (live) {
                    const int tcol = ea.tok_vcol ? ea.tok_vcol[grow] : grow;
                    __half* dst = ea.vt + (size_t)(vcol + c) * ea.ldvt + tcol;
                    store_vt32(dst, ea.ldvt, r);
                    if (ea.v_rows) {            // token-major copy (a decode KV cache)
                        float y[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) y[j] = f32(r[j]);
                        store_row32(ea.v_rows + (size_t)grow * nk + vcol + c, y);
                    }
                }
            }
        }
    }
}

// gate/up interleaved in 64-column blocks: block b of the product holds gate
// columns 64b..64b+63 then up columns 64b..64b+63; act[:, 64b + j] = silu(g) * u.
template <int BN, bool SC>
__device__ __forceinline__ void epi_swiglu(const Params& p, uint32_t tbase, int grow, int n0) {
    const GemmEpiArgs& ea = p.ea;
    const float rsc = row_rstd(ea, grow, p.M);     // fused RMSNorm row scale (or 1)
    const int F = p.N / 2;
#pragma unroll 1
    for (int b = 0; b < BN; b += 128) {
        const int colblk = n0 + b;
        if (colblk >= p.N) break;
        const int f0 = colblk / 2;
#pragma unroll 1
        for (int c = 0; c < 64; c += 32) {
            uint32_t rg[32], ru[32];
            __syncwarp();
            acc_ld32<SC>(p, tbase, tbase + b + c, grow, n0, rg, rsc);
            acc_ld32<SC>(p, tbase, tbase + b + 64 + c, grow, n0, ru, rsc);
            if (grow < p.M) {
                float a[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) a[j] = silu_f(f32(rg[j])) * f32(ru[j]);
                store_row32(ea.act + (size_t)grow * F + f0 + c, a);
            }
        }
    }
}

// ----------------------------------------------------------------------------- TMA-store epilogues
__device__ __forceinline__ uint4 pack8_bf16(const float* v) {
    uint4 u;
    u.x = ptx::pack_bf16x2(v[0], v[1]);
    u.y = ptx::pack_bf16x2(v[2], v[3]);
    u.z = ptx::pack_bf16x2(v[4], v[5]);
    u.w = ptx::pack_bf16x2(v[6], v[7]);
    return u;
}

// Hand the staged box to TMA (lane 0) after every lane's writes are visible to it.
__device__ __forceinline__ void stage_flush(EpiStage& st, int b, const CUtensorMap* map, int x) {
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (st.lane == 0) {
        ptx::tma_store_2d(map, st.buf[b], x, st.row0);
        ptx::bulk_commit();
    }
}

// Before writing buffer b: the bulk store issued from it two flushes ago has
// finished reading it.
__device__ __forceinline__ void stage_claim(EpiStage& st) {
    if (st.lane == 0) ptx::bulk_wait_read<1>();
    __syncwarp();
}

// Residual chunk (f32 32x32 box) for the chunk at column x into buffer b.
__device__ __forceinline__ void stage_prefetch(EpiStage& st, int b, const CUtensorMap* tmR, int x) {
    if (st.lane == 0) {
        ptx::bulk_wait_read<0>();
        ptx::mbar_arrive_expect_tx(st.rbar[b], 32 * 128);
        ptx::tma_load_2d(tmR, st.rbar[b], st.buf[b], x, st.row0);
    }
    st.pending[b] = 1;
    __syncwarp();
}

// y = acc (+ residual): float32 chunks of 32 columns or bf16 chunks of 64.
// BN must be a multiple of the chunk width (32 for float32, 64 for bf16 output).
template <int BN, bool SC>
__device__ __forceinline__ bool epi_store_tma(const Params& p, EpiStage& st, uint32_t tbase, int n0,
                                              const CUtensorMap* tmY, const CUtensorMap* tmR,
                                              volatile int* abort_flag) {
    const GemmEpiArgs& ea = p.ea;
    const bool f32out = ea.y_dtype == DTP_F32;
    const bool resid = ea.residual != nullptr;
    const int CW = f32out ? 32 : 64;
    const int grow = st.row0 + st.lane;
    float ss = 0.f;                                  // fused RMSNorm: this tile's sum of y^2
#pragma unroll 1
    for (int c = 0; c < BN; c += CW) {
        const int col0 = n0 + c;
        if (col0 >= p.N) break;
        const int b = st.cnt & 1;
        if (resid) {
            // buf[b] already holds (or is receiving) this chunk's residual; the
            // first chunk of a tile was prefetched before the accumulator wait
            if (c + CW < BN && col0 + CW < p.N) stage_prefetch(st, b ^ 1, tmR, col0 + CW);
        } else {
            stage_claim(st);
        }
        float v[64];
        uint32_t r[32];
        __syncwarp();
        acc_ld32<SC>(p, tbase, tbase + c, grow, n0, r);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = f32(r[j]);
        if (!f32out) {
            __syncwarp();
            acc_ld32<SC>(p, tbase, tbase + c + 32, grow, n0, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[32 + j] = f32(r[j]);
        }
        if (resid) {
            const bool ok = ptx::wait_bounded<kSuspendWaits>(st.rbar[b], st.rphase[b], abort_flag, &g_gemm_err,
                                              ERRBIT_TIMEOUT);
            if (!__all_sync(0xffffffffu, ok)) return false;
            st.rphase[b] ^= 1;
            st.pending[b] = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 u = stage_get16(st.buf[b], st.lane, j);
                v[4 * j + 0] += __uint_as_float(u.x);
                v[4 * j + 1] += __uint_as_float(u.y);
                v[4 * j + 2] += __uint_as_float(u.z);
                v[4 * j + 3] += __uint_as_float(u.w);
            }
        }
        if (f32out) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                stage_put16(st.buf[b], st.lane, j,
                            make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                       __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3])));
            if (ea.xb && grow < p.M) {
                float vv[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    vv[j] = v[j];
                    ss = col0 + j < p.N ? fmaf(v[j], v[j], ss) : ss;
                }
                if (col0 + 32 <= p.N) {
                    store_row32(ea.xb + (size_t)grow * ea.ldy + col0, vv);
                } else {
                    for (int j = 0; j < 32 && col0 + j < p.N; ++j)
                        ea.xb[(size_t)grow * ea.ldy + col0 + j] = __float2bfloat16_rn(vv[j]);
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) stage_put16(st.buf[b], st.lane, j, pack8_bf16(v + 8 * j));
        }
        stage_flush(st, b, tmY, col0);
        ++st.cnt;
    }
    if (ea.ss_out && grow < p.M) ea.ss_out[(size_t)(n0 / BN) * ea.ld_ss + grow] = ss;
    return true;
}

// gate/up (interleaved 64-column blocks) -> act = silu(g) * u, bf16 boxes of 64 columns.
template <int BN, bool SC>
__device__ __forceinline__ void epi_swiglu_tma(const Params& p, EpiStage& st, uint32_t tbase,
                                               int n0, const CUtensorMap* tmY) {
    const int grow = st.row0 + st.lane;
    const float rsc = row_rstd(p.ea, grow, p.M);   // fused RMSNorm row scale (or 1)
#pragma unroll 1
    for (int b = 0; b < BN; b += 128) {
        const int colblk = n0 + b;
        if (colblk >= p.N) break;
        const int bb = st.cnt & 1;
        stage_claim(st);
#pragma unroll 1
        for (int c = 0; c < 64; c += 32) {
            uint32_t rg[32], ru[32];
            __syncwarp();
            acc_ld32<SC>(p, tbase, tbase + b + c, grow, n0, rg, rsc);
            acc_ld32<SC>(p, tbase, tbase + b + 64 + c, grow, n0, ru, rsc);
            float a[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) a[j] = silu_f(f32(rg[j])) * f32(ru[j]);
#pragma unroll
            for (int j = 0; j < 4; ++j) stage_put16(st.buf[bb], st.lane, c / 8 + j, pack8_bf16(a + 8 * j));
        }
        stage_flush(st, bb, tmY, colblk / 2);
        ++st.cnt;
    }
}

// QKV: q/k heads normalised and rotated, staged as 64-column bf16 boxes (one or
// two per head); v heads (transposed) and gate blocks stored directly.
template <int BN, bool SC>
__device__ __forceinline__ void epi_qkv_tma(const Params& p, EpiStage& st, uint32_t tbase,
                                            int grow, int n0, const CUtensorMap* tmQ,
                                            const CUtensorMap* tmK) {
    const GemmEpiArgs& ea = p.ea;
    const float rsc = row_rstd(ea, grow, p.M);     // fused RMSNorm row scale (or 1)
    const int hd = ea.head_dim, half = ea.rope_dims / 2;
    const int nq = ea.n_head * hd, nk = ea.n_head_kv * hd;
    const bool live = grow < p.M;
    const int nqc = ea.q_gated ? 2 * nq : nq;
#pragma unroll 1
    for (int h0 = 0; h0 < BN; h0 += hd) {
        const int col = n0 + h0;
        if (col >= p.N) break;
        const uint32_t th = tbase + h0;
        const int blk = col / hd;
        if (ea.q_gated && col < nqc && (blk & 1)) {
#pragma unroll 1
            for (int c = 0; c < hd; c += 32) {
                uint32_t r[32];
                __syncwarp();
                acc_ld32<SC>(p, tbase, th + c, grow, n0, r, rsc);
                if (live) {
                    float y[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) y[j] = f32(r[j]);
                    store_row32(ea.gate + (size_t)grow * nq + (blk >> 1) * hd + c, y);
                }
            }
            continue;
        }
        if (col < nqc + nk) {
            const bool isq = col < nqc;
            const int ocol = isq ? (ea.q_gated ? (blk >> 1) * hd : col) : col - nqc;
            const float* w = isq ? ea.q_norm : ea.k_norm;
            float ss = 0.f;
#pragma unroll 1
            for (int c = 0; c < hd; c += 32) {
                uint32_t r[32];
                __syncwarp();
                acc_ld32<SC>(p, tbase, th + c, grow, n0, r, rsc);
#pragma unroll
                for (int j = 0; j < 32; ++j) ss = fmaf(f32(r[j]), f32(r[j]), ss);
            }
            const float rstd = 1.0f / sqrtf(ss / (float)hd + ea.eps);
            // both staging buffers may be needed (head_dim 128): wait for all reads
            if (st.lane == 0) ptx::bulk_wait_read<0>();
            __syncwarp();
            const int pos = ea.tok_pos ? ea.tok_pos[live ? grow : 0] : grow;
#pragma unroll 1
            for (int i0 = 0; i0 < half; i0 += 32) {
                uint32_t ra[32], rb[32];
                __syncwarp();
                acc_ld32<SC>(p, tbase, th + i0, grow, n0, ra, rsc);
                acc_ld32<SC>(p, tbase, th + half + i0, grow, n0, rb, rsc);
                // (cos, sin) pairs j, j+1 in one 16-byte load: rows of the table
                // and i0 are multiples of 32 pairs
                const float4* cs =
                    reinterpret_cast<const float4*>(ea.rope + (size_t)(live ? pos : 0) * half + i0);
                float ya[32], yb[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float a = f32(ra[j]) * rstd * w[i0 + j];
                    const float bv = f32(rb[j]) * rstd * w[half + i0 + j];
                    const float4 c4 = cs[j >> 1];
                    const float2 c2 = (j & 1) ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y);
                    ya[j] = a * c2.x - bv * c2.y;
                    yb[j] = a * c2.y + bv * c2.x;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    stage_put16(st.buf[(i0 >> 6)], st.lane, ((i0 & 63) >> 3) + j, pack8_bf16(ya + 8 * j));
                    const int cb = half + i0;
                    stage_put16(st.buf[(cb >> 6)], st.lane, ((cb & 63) >> 3) + j, pack8_bf16(yb + 8 * j));
                }
            }
#pragma unroll 1
            for (int c = ea.rope_dims; c < hd; c += 32) {
                uint32_t r[32];
                __syncwarp();
                acc_ld32<SC>(p, tbase, th + c, grow, n0, r, rsc);
                float y[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) y[j] = f32(r[j]) * rstd * w[c + j];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    stage_put16(st.buf[(c >> 6)], st.lane, ((c & 63) >> 3) + j, pack8_bf16(y + 8 * j));
            }
            const CUtensorMap* map = isq ? tmQ : tmK;
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (st.lane == 0) {
                for (int a = 0; a < hd / 64; ++a) ptx::tma_store_2d(map, st.buf[a], ocol + 64 * a, st.row0);
                ptx::bulk_commit();
            }
        } else {
            const int vcol = col - nqc - nk;
#pragma unroll 1
            for (int c = 0; c < hd; c += 32) {
                uint32_t r[32];
                __syncwarp();
                acc_ld32<SC>(p, tbase, th + c, grow, n0, r, rsc);
                if (live) {
                    const int tcol = ea.tok_vcol ? ea.tok_vcol[grow] : grow;
                    __half* dst = ea.vt + (size_t)(vcol + c) * ea.ldvt + tcol;
                    store_vt32(dst, ea.ldvt, r);
                    if (ea.v_rows) {
                        float y[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) y[j] = f32(r[j]);
                        store_row32(ea.v_rows + (size_t)grow * nk + vcol + c, y);
                    }
                }
            }
        }
    }
}

// ----------------------------------------------------------------------------- kernel
enum { OP_BF16 = 0, OP_TF32 = 1, OP_E4M3 = 2 };

// CL = 2: clusters of two CTAs compute 256 x BN tiles with cta_group::2 MMAs.
// The even CTA (rank 0) takes M block 2j, the odd one 2j + 1, of the same N
// block.  Each CTA's producer loads its 128 A rows and its half of the B rows
// (rank r: rows r*BN/2 ..) into its own shared memory; both count their bytes
// on the even CTA's full barrier.  The even CTA's MMA thread issues the pair
// MMAs and commits to the empty and accumulator-full barriers of both CTAs.
// Each CTA's epilogue reads its own TMEM rows; its warps release the
// accumulator on the even CTA's accumulator-empty barrier.
template <int BN, int EPI, int OPK = OP_BF16, int CL = 1>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmY2,
                   const __grid_constant__ CUtensorMap tmR, const Params p) {
    using C = Cfg<BN, CL>;
    static_assert(CL == 1 || CL == 2, "single CTAs or pairs");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + C::STAGES * C::A_BYTES;
    uint8_t* sEpi = smem + C::STAGES * C::STAGE_BYTES;          // 1024-byte aligned
    uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + C::EPI_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* tfull = bars + 2 * C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* rbars = drain + 1;                                 // [4 warps][2]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(rbars + 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = CL > 1 ? ptx::cluster_ctarank() : 0u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&tfull[b], 1);
            // single: every epilogue thread arrives; pairs: lane 0 of the 4
            // epilogue warps of both CTAs
            ptx::mbar_init(&tempty[b], CL == 1 ? 128 : 8);
        }
        ptx::mbar_init(drain, 1);
        for (int i = 0; i < 8; ++i) ptx::mbar_init(&rbars[i], 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    // the warp-collective TMEM allocation and the barriers below are .aligned:
    // every warp arrives converged (thread 0 ran the set-up alone)
    __syncwarp();
    if (warp == 0) {
        if constexpr (CL == 1) {
            ptx::tmem_alloc(tmem_holder, C::TMEM_COLS);
            ptx::tmem_relinquish();
        } else {
            ptx::tmem_alloc_pair(tmem_holder, C::TMEM_COLS);
            ptx::tmem_relinquish_pair();
        }
    }
    if (warp == 1 && lane == 0) {
        ptx::tma_prefetch_desc(&tmA);
        ptx::tma_prefetch_desc(&tmB);
        if (C::TMA_OUT && p.tma_out) {
            ptx::tma_prefetch_desc(&tmY);
            ptx::tma_prefetch_desc(&tmY2);
            ptx::tma_prefetch_desc(&tmR);
        }
    }
    __syncwarp();
    ptx::tc_fence_before();
    if constexpr (CL > 1)
        ptx::cluster_sync();      // the peer's barriers exist before anything arrives on them
    else
        __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const int num_tiles = p.tiles_m * p.tiles_n;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            // pairs: the even CTA's full barriers count both CTAs' bytes
            const uint32_t full_cl = CL > 1 ? ptx::mapa(ptx::smem_u32(full), 0) : 0u;
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                const int mb = tile % p.tiles_m, nb = tile / p.tiles_m;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!ptx::wait_bounded<kSuspendWaits>(&empty[stage], phase ^ 1, abort_flag, &g_gemm_err,
                                           ERRBIT_TIMEOUT))
                        goto producer_done;
                    // a stage holds 128 bytes of K per row: 64 bf16, 32 tf32, 128 e4m3
                    const int k0 = kb * (OPK == OP_TF32 ? BK / 2 : OPK == OP_E4M3 ? 2 * BK : BK);
                    if constexpr (CL == 1) {
                        ptx::mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                        ptx::tma_load_2d(&tmA, &full[stage], sA + stage * C::A_BYTES, k0, mb * BM);
                        ptx::tma_load_2d(&tmB, &full[stage], sB + stage * C::B_BYTES, k0, nb * BN);
                    } else {
                        if (crank == 0) ptx::mbar_arrive_expect_tx(&full[stage], CL * C::STAGE_BYTES);
                        const uint32_t fb = full_cl + stage * 8u;
                        ptx::tma_load_2d_pair(&tmA, fb, sA + stage * C::A_BYTES, k0, mb * BM);
                        ptx::tma_load_2d_pair(&tmB, fb, sB + stage * C::B_BYTES, k0,
                                              nb * BN + (int)crank * (BN / CL));
                    }
                    ++issued;
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if constexpr (CL > 1) {
                // the even CTA's last commits arrive on this CTA's empty barriers:
                // see every stage released once more before the CTA may exit
                for (int i = 0; i < C::STAGES; ++i) {
                    if (!ptx::wait_bounded<kSuspendWaits>(&empty[stage], phase ^ 1, abort_flag, &g_gemm_err,
                                           ERRBIT_TIMEOUT))
                        break;
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        producer_done:
            // pairs: only the even CTA's full barriers count loads
            if (*abort_flag && crank == 0) {
                // let every load still in flight land before the CTA can exit
                int s = stage;
                uint32_t ph = phase;
                for (int i = 0; i < C::STAGES && i < issued; ++i) {
                    if (--s < 0) {
                        s = C::STAGES - 1;
                        ph ^= 1;
                    }
                    volatile int never = 0;
                    ptx::wait_bounded<kSuspendWaits>(&full[s], ph, &never, &g_gemm_err, ERRBIT_TIMEOUT);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && crank == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr int MM = CL * BM;
            const uint32_t idesc = OPK == OP_TF32   ? ptx::idesc_tf32_f32(MM, BN)
                                   : OPK == OP_E4M3 ? ptx::idesc_e4m3_f32(MM, BN)
                                                    : ptx::idesc_bf16_f32(MM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                if (!ptx::wait_bounded<kSuspendWaits>(&tempty[acc], acc_phase ^ 1, abort_flag, &g_gemm_err,
                                       ERRBIT_TIMEOUT))
                    break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * C::ACC_STRIDE;
                bool ok = true;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!ptx::wait_bounded<kSuspendWaits>(&full[stage], phase, abort_flag, &g_gemm_err,
                                           ERRBIT_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint64_t adesc = ptx::sdesc_sw128(ptx::smem_u32(sA + stage * C::A_BYTES));
                    const uint64_t bdesc = ptx::sdesc_sw128(ptx::smem_u32(sB + stage * C::B_BYTES));
                    // four MMAs per stage, each 32 bytes further along K (+2 in
                    // the descriptor's 16-byte address units)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        if constexpr (CL == 2)
                            ptx::umma_pair_ss<OPK>(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc,
                                                   (kb > 0 || kk > 0) ? 1u : 0u);
                        else if constexpr (OPK == OP_TF32)
                            ptx::umma_tf32_ss(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc,
                                              (kb > 0 || kk > 0) ? 1u : 0u);
                        else if constexpr (OPK == OP_E4M3)
                            ptx::umma_e4m3_ss(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc,
                                              (kb > 0 || kk > 0) ? 1u : 0u);
                        else
                            ptx::umma_bf16_ss(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc,
                                              (kb > 0 || kk > 0) ? 1u : 0u);
                    }
                    if constexpr (CL == 1)
                        ptx::umma_commit(&empty[stage]);
                    else
                        ptx::umma_commit_pair(&empty[stage], 3);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                if constexpr (CL == 1)
                    ptx::umma_commit(&tfull[acc]);
                else
                    ptx::umma_commit_pair(&tfull[acc], 3);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            // every MMA issued above completes before TMEM can be released
            if constexpr (CL == 1)
                ptx::umma_commit(drain);
            else
                ptx::umma_commit_pair(drain, 1);
            volatile int never = 0;
            ptx::wait_bounded<kSuspendWaits>(drain, 0, &never, &g_gemm_err, ERRBIT_TIMEOUT);
        }
    } else {
        // ---------------------------------------------------- epilogue warps 2..5
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        EpiStage st;
        st.buf[0] = sEpi + (warp - 2) * 2 * C::EPI_BUF;
        st.buf[1] = st.buf[0] + C::EPI_BUF;
        st.rbar[0] = &rbars[(warp - 2) * 2];
        st.rbar[1] = &rbars[(warp - 2) * 2 + 1];
        st.rphase[0] = st.rphase[1] = 0;
        st.pending[0] = st.pending[1] = 0;
        st.cnt = 0;
        st.lane = lane;
        const bool tma_out = C::TMA_OUT && p.tma_out;
        const bool resid_tma = EPI == EPI_STORE && tma_out && p.ea.residual != nullptr;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const int mb = tile % p.tiles_m, nb = tile / p.tiles_m;
            const int grow = mb * BM + row, n0 = nb * BN;
            st.row0 = mb * BM + quarter * 32;
            // the first residual chunk of the tile loads while the main loop runs
            if (resid_tma) stage_prefetch(st, st.cnt & 1, &tmR, n0);
            const bool ok = ptx::wait_bounded<kSuspendWaits>(&tfull[acc], acc_phase, abort_flag, &g_gemm_err,
                                              ERRBIT_TIMEOUT);
            if (!__all_sync(0xffffffffu, ok)) break;
            ptx::tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * C::ACC_STRIDE;
            bool eok = true;
            if (tma_out) {
                if (EPI == EPI_STORE)
                    eok = epi_store_tma<BN, OPK == OP_E4M3>(p, st, tbase, n0, &tmY, &tmR, abort_flag);
                if (EPI == EPI_QKV) epi_qkv_tma<BN, OPK == OP_E4M3>(p, st, tbase, grow, n0, &tmY, &tmY2);
                if (EPI == EPI_SWIGLU) epi_swiglu_tma<BN, OPK == OP_E4M3>(p, st, tbase, n0, &tmY);
            } else {
                if (EPI == EPI_STORE) epi_store<BN, OPK == OP_E4M3>(p, tbase, grow, n0);
                if (EPI == EPI_QKV) epi_qkv<BN, OPK == OP_E4M3>(p, tbase, grow, n0);
                if (EPI == EPI_SWIGLU) epi_swiglu<BN, OPK == OP_E4M3>(p, tbase, grow, n0);
            }
            __syncwarp();
            ptx::tc_fence_before();
            if constexpr (CL == 1) {
                ptx::mbar_arrive(&tempty[acc]);
            } else {
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(&tempty[acc]), 0));
            }
            if (!eok) break;
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
        // every staged box is written out, and every residual load that was
        // issued but not consumed (only after an abort) has landed, before the
        // CTA and its shared memory go away
        if (lane == 0) {
            ptx::bulk_wait<0>();
            volatile int never = 0;
            for (int b = 0; b < 2; ++b)
                if (st.pending[b])
                    ptx::wait_bounded<kSuspendWaits>(st.rbar[b], st.rphase[b], &never, &g_gemm_err, ERRBIT_TIMEOUT);
        }
        __syncwarp();
    }

    // warps 0 and 1 ran their roles on one lane: converge each warp before the
    // CTA and cluster barriers, which count whole warps
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    // pairs: both CTAs are done with TMEM and every arrival on the other's
    // barriers has landed before either frees anything
    if constexpr (CL > 1) ptx::cluster_sync();
    if (warp == 0) {
        __syncwarp();
        ptx::tc_fence_after();
        if constexpr (CL == 1)
            ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
        else
            ptx::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

template <int BN, int EPI, int OPK = OP_BF16, int CL = 1>
cudaError_t launch_impl(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty,
                        const CUtensorMap& ty2, const CUtensorMap& tr, const Params& p,
                        cudaStream_t s) {
    using C = Cfg<BN, CL>;
    auto kern = gemm_tc_kernel<BN, EPI, OPK, CL>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int max_ctas = 0;      // persistent CTAs that can be resident at once
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        C::SMEM_BYTES);
        max_ctas = num_sms();
        if (attr_err == cudaSuccess && CL > 1) {
            // clusters are placed whole: on a GPU whose SMs do not pair up evenly
            // fewer than num_sms / CL of them fit at once
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = CL;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(num_sms() / CL * CL);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = C::SMEM_BYTES;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int clusters = 0;
            attr_err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
            if (attr_err == cudaSuccess && clusters < 1) attr_err = cudaErrorInvalidConfiguration;
            max_ctas = clusters * CL < num_sms() ? clusters * CL : num_sms() / CL * CL;
        }
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int tiles = p.tiles_m * p.tiles_n;
    const int grid = tiles < max_ctas ? tiles : max_ctas;
    if constexpr (CL == 1) {
        kern<<<grid, kThreads, C::SMEM_BYTES, s>>>(ta, tb, ty, ty2, tr, p);
    } else {
        // pairs of CTAs 2c, 2c+1 take tiles 2c + i*grid and 2c+1 + i*grid: with
        // tiles_m and grid even these are the same N block, M blocks 2j and 2j+1
        if (p.tiles_m % CL != 0 || grid % CL != 0) return cudaErrorInvalidConfiguration;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = CL;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.stream = s;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb, ty, ty2, tr, p);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace

// Tile width: the fused QKV and SwiGLU epilogues need 256 (whole heads / whole
// 128-column gate-up blocks).  A plain store picks the width whose persistent
// schedule finishes first: waves(BN) * BN, waves = ceil(tiles / SMs); 224 only
// with float32 output (its epilogue chunks are 32 columns; bf16 chunks are 64).
static int pick_bn(int M, int N, GemmEpi epi, int y_dtype) {
    if (epi != EPI_STORE) return 256;
    if (N <= 128) return 128;
    if (y_dtype != DTP_F32) return 256;
    // 256 stores through TMA; 224 only when it saves at least 5% of the schedule
    const long long tm = (M + BM - 1) / BM, sms = num_sms();
    auto cost = [&](long long bn) { return (tm * ((N + bn - 1) / bn) + sms - 1) / sms * bn; };
    return 20 * cost(224) < 19 * cost(256) ? 224 : 256;
}

static cudaError_t launch_gemm(const void* x, const void* W, int opk, int M, int N, int K,
                               GemmEpi epi, const GemmEpiArgs& ea, cudaStream_t s, int kind) {
    const bool tf32 = opk == OP_TF32, e4m3 = opk == OP_E4M3;
    int BN = pick_bn(M, N, epi, ea.y_dtype);
    if (tf32 && BN == 224) BN = 256;         // tf32 instantiates the 256 and 128 tiles only
    // operand boxes: 128 bytes of K per row (64 bf16, 32 float32 or 128 e4m3)
    const int bke = tf32 ? BK / 2 : e4m3 ? 2 * BK : BK;
    const CUtensorMapDataType odt = tf32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                    : e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int oeb = tf32 ? 4 : e4m3 ? 1 : 2;
    CUtensorMap ta, tb;
    if (!make_tmap_2d(&ta, x, odt, oeb, M, K, K, BM, bke)) return cudaErrorInvalidValue;
    // B boxes of BN/2 rows: each CTA of a pair holds half of the B tile
    const int cl = kCluster;
    if (!make_tmap_2d(&tb, W, odt, oeb, N, K, K, BN / cl, bke)) return cudaErrorInvalidValue;
    Params p;
    p.M = M;
    p.N = N;
    p.K = K;
    // an even number of M blocks, so the CTAs of a pair share N blocks; a
    // last block past M (odd M/128) reads zeros and stores nothing
    p.tiles_m = ((M + BM - 1) / BM + cl - 1) / cl * cl;
    p.tiles_n = (N + BN - 1) / BN;
    p.num_kb = (K + bke - 1) / bke;
    p.ea = ea;
    p.vec_ok = 1;
    p.tma_out = 0;
    // output (and residual) tensor maps: 32-row boxes of 128 bytes, 128-byte swizzle
    CUtensorMap ty = ta, ty2 = ta, tr = ta;
    auto al16 = [](const void* q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; };
    if (epi == EPI_STORE) {
        const int eb = ea.y_dtype == DTP_F32 ? 4 : 2;
        if ((ea.ldy * eb) % 16 != 0 || !al16(ea.y) || (ea.residual && !al16(ea.residual)))
            p.vec_ok = 0;
        const CUtensorMapDataType dt =
            ea.y_dtype == DTP_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        if (p.vec_ok && make_tmap_2d(&ty, ea.y, dt, eb, M, N, ea.ldy, 32, 128 / eb) &&
            (!ea.residual || make_tmap_2d(&tr, ea.residual, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, M, N,
                                          ea.ldy, 32, 32)))
            p.tma_out = 1;
    } else if (epi == EPI_SWIGLU) {
        p.tma_out = al16(ea.act) &&
                    make_tmap_2d(&ty, ea.act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, N / 2, N / 2, 32, 64);
    } else if (epi == EPI_QKV) {
        const int nq = ea.n_head * ea.head_dim, nk = ea.n_head_kv * ea.head_dim;
        p.tma_out = al16(ea.q) && al16(ea.k) &&
                    make_tmap_2d(&ty, ea.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, nq, nq, 32, 64) &&
                    make_tmap_2d(&ty2, ea.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, nk, nk, 32, 64);
    }
    if (BN == 224) p.tma_out = 0;
    if (!p.tma_out) ty = ty2 = tr = ta;
    LaunchScope ls(kind, s);
    if (tf32) {
        if (epi != EPI_STORE) return cudaErrorNotSupported;
        if (BN == 256) return launch_impl<256, EPI_STORE, OP_TF32, kCluster>(ta, tb, ty, ty2, tr, p, s);
        return launch_impl<128, EPI_STORE, OP_TF32, kCluster>(ta, tb, ty, ty2, tr, p, s);
    }
    if (e4m3) {
        if (BN == 256) {
            if (epi == EPI_QKV) return launch_impl<256, EPI_QKV, OP_E4M3, kCluster>(ta, tb, ty, ty2, tr, p, s);
            if (epi == EPI_SWIGLU)
                return launch_impl<256, EPI_SWIGLU, OP_E4M3, kCluster>(ta, tb, ty, ty2, tr, p, s);
            return launch_impl<256, EPI_STORE, OP_E4M3, kCluster>(ta, tb, ty, ty2, tr, p, s);
        }
        if (BN == 224) return launch_impl<224, EPI_STORE, OP_E4M3, kCluster>(ta, tb, ty, ty2, tr, p, s);
        return launch_impl<128, EPI_STORE, OP_E4M3, kCluster>(ta, tb, ty, ty2, tr, p, s);
    }
    if (BN == 256) {
        if (epi == EPI_QKV) return launch_impl<256, EPI_QKV, OP_BF16, kCluster>(ta, tb, ty, ty2, tr, p, s);
        if (epi == EPI_SWIGLU) return launch_impl<256, EPI_SWIGLU, OP_BF16, kCluster>(ta, tb, ty, ty2, tr, p, s);
        return launch_impl<256, EPI_STORE, OP_BF16, kCluster>(ta, tb, ty, ty2, tr, p, s);
    }
    if (BN == 224) return launch_impl<224, EPI_STORE, OP_BF16, kCluster>(ta, tb, ty, ty2, tr, p, s);
    return launch_impl<128, EPI_STORE, OP_BF16, kCluster>(ta, tb, ty, ty2, tr, p, s);
}

int gemm_tc_tiles_n(int M, int N) {
    const int bn = pick_bn(M, N, EPI_STORE, DTP_F32);
    return (N + bn - 1) / bn;
}

cudaError_t launch_gemm_tc(const __nv_bfloat16* x, const __nv_bfloat16* W, int M, int N, int K,
                           GemmEpi epi, const GemmEpiArgs& ea, cudaStream_t s, int kind) {
    GemmEpiArgs e = ea;
    e.a_scale = e.b_scale = nullptr;
    return launch_gemm(x, W, OP_BF16, M, N, K, epi, e, s, kind);
}

cudaError_t launch_gemm_tc_tf32(const float* x, const float* W, int M, int N, int K,
                                const GemmEpiArgs& ea, cudaStream_t s, int kind) {
    GemmEpiArgs e = ea;
    e.a_scale = e.b_scale = nullptr;
    return launch_gemm(x, W, OP_TF32, M, N, K, EPI_STORE, e, s, kind);
}

cudaError_t launch_gemm_tc_e4m3(const uint8_t* x, const uint8_t* W, int M, int N, int K,
                                GemmEpi epi, const GemmEpiArgs& ea, cudaStream_t s, int kind) {
    if (!ea.a_scale || !ea.b_scale) return cudaErrorInvalidValue;
    return launch_gemm(x, W, OP_E4M3, M, N, K, epi, ea, s, kind);
}

}  // namespace dtp
