// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dtp.h"

namespace dtp {

// ----------------------------------------------------------------------------- errors
int fail(int code, const char* fmt, ...);      // records the message, returns code
void clear_error();

#define DTP_CUDA_CHECK(expr)                                                                   \
    do {                                                                                       \
        cudaError_t e_ = (expr);                                                               \
        if (e_ != cudaSuccess)                                                                 \
            return ::dtp::fail(DTP_ERR_CUDA, "%s: %s (%s:%d)", #expr, cudaGetErrorString(e_),  \
                               __FILE__, __LINE__);                                            \
    } while (0)

// Device error word bits (each kernel family keeps its own word).
enum : unsigned { ERRBIT_TOKEN_RANGE = 1u, ERRBIT_TIMEOUT = 2u, ERRBIT_SEQLENS = 4u,
                  ERRBIT_VRANGE = 8u };

// Read and clear the error words of every kernel family on the current device.
unsigned read_clear_simt_errors();
unsigned read_clear_gemm_errors();
unsigned read_clear_attn_errors();

// ----------------------------------------------------------------------------- timing
// Brackets one kernel launch with the timer events of `kind` (if enabled) and
// counts the launch.  counts = false brackets a span that is not one kernel
// (a whole prompt's pass, a copy): timed, not counted as a launch.
struct LaunchScope {
    LaunchScope(int kind, cudaStream_t s, bool counts = true);
    ~LaunchScope();
    int kind;
    cudaStream_t stream;
    int slot;
};

int num_sms();
size_t align_up(size_t x, size_t a);

// ----------------------------------------------------------------------------- tensor maps
// 2-D row-major tensor [rows, cols] (cols contiguous, row stride ld elements),
// box [box_rows, box_cols], 128-byte swizzle.  Returns false on failure.
bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elt_bytes,
                  uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows, uint32_t box_cols);

// ----------------------------------------------------------------------------- SIMT kernels
cudaError_t launch_embed(const uint32_t* tokens, int T, int V, int d, const void* table,
                         int table_dtype, float* x, cudaStream_t s, __nv_bfloat16* xb = nullptr,
                         float* ss_out = nullptr);
cudaError_t launch_rmsnorm(const float* x, const float* w, void* y, int y_dtype, int rows,
                           int cols, float eps, cudaStream_t s, const int* row_idx = nullptr);
cudaError_t launch_qk_norm_rope(void* x, int dtype, int ld, const float* w_norm,
                                const int32_t* pos, int T, int n_heads, int head_dim,
                                int rope_dims, float freq_base, float eps, cudaStream_t s,
                                int head_stride = 0, int pos0 = 0);
// attn[t, h*hd + e] *= sigmoid(gate[t * ldg + h*gstride + e]) (float32)
cudaError_t launch_gate_mul_f32(float* attn, int lda, const float* gate, int ldg, int gstride,
                                int T, int n_head, int head_dim, cudaStream_t s);
cudaError_t launch_rope_table(float2* tab, int T, int rope_dims, float freq_base,
                              cudaStream_t s, int pos0 = 0);
cudaError_t launch_swiglu(const void* gate, const void* up, void* out, int dtype, size_t n,
                          cudaStream_t s);
cudaError_t launch_swiglu_interleaved64(const float* gu, float* act, int T, int F,
                                        cudaStream_t s, int act_dtype = DTP_F32);
cudaError_t launch_round_tf32(float* x, size_t n, cudaStream_t s);
cudaError_t launch_round_tf32_rows(float* x, int ld, int rows, int cols, cudaStream_t s);
// v [T, ldv] float32 -> vt [width, ldt] (key index contiguous)
cudaError_t launch_transpose_v_f32(const float* v, int ldv, float* vt, int T, int width, int ldt,
                                   cudaStream_t s);
// Per-row e4m3 quantisation (quant.cu): codes q [rows, cols] (row-major, no
// padding) and scale [rows] = max|row| / 448.
cudaError_t launch_rmsnorm_e4m3(const float* x, const float* w, uint8_t* q, float* scale,
                                int rows, int cols, float eps, cudaStream_t s,
                                const int* row_idx = nullptr);
cudaError_t launch_quant_rows_e4m3(const __nv_bfloat16* x, int ldx, int rows, int cols,
                                   uint8_t* q, float* scale, cudaStream_t s);
cudaError_t launch_pack_e4m3(const float* src, int rows, int cols, uint8_t* dst, float* dst_scale,
                             int mode, cudaStream_t s);
cudaError_t launch_gemm_simt(const float* x, int ldx, const float* W, void* y, int y_dtype,
                             int ldy, int M, int N, int K, const float* residual,
                             cudaStream_t s, int kind);
// Causal GQA attention on SIMT cores.  dtype of q/k/v/out: DTP_F32 or DTP_BF16.
// v_t != 0: v is stored transposed [n_head_kv*head_dim, ldv_t] (key index contiguous).
// tok_pos (optional): position of each query within its sequence; the keys of
// query t are then t - tok_pos[t] .. t (sequences packed along the token axis).
cudaError_t launch_attn_simt(const void* q, int ldq, const void* k, int ldk, const void* v,
                             int ldv, int v_t, void* out, int ldo, int dtype, int T,
                             int n_head, int n_head_kv, int head_dim, float scale,
                             cudaStream_t s, const int* tok_pos = nullptr,
                             int q_head_stride = 0, int q_pos0 = 0);
// Per-sequence schedule for packed sequences: tile_start [n_seq+1] (prefix of
// ceil(len/128)), vcol_start [n_seq] (prefix of len rounded up to 8),
// last_row [n_seq] (cu[b+1]-1); then per-token tok_pos / tok_vcol [total].
// Invalid cu_seqlens raise ERRBIT_SEQLENS and leave an empty, in-bounds schedule.
cudaError_t launch_seq_meta(const int* cu_seqlens, int n_seq, int total, int* tile_start,
                            int* vcol_start, int* last_row, int* tok_pos, int* tok_vcol,
                            long long vt_cols, cudaStream_t s);
// v [T, width] bf16 -> vt [width, ldt] f16 (key index contiguous), each value
// converted to f16 (exact from 2^-14 up to 65504); a |v| beyond the f16 range
// raises ERRBIT_VRANGE.
cudaError_t launch_transpose_v(const __nv_bfloat16* v, __half* vt, int T, int width,
                               int ldt, cudaStream_t s);
// to_dtype: DTP_F32, DTP_BF16 or DTP_TF32 (float32 rounded to tf32)
cudaError_t launch_pack_matrix(const float* src, int rows, int cols, void* dst, int to_dtype,
                               int mode, cudaStream_t s, const float* col_scale = nullptr);
cudaError_t launch_copy_f32(const float* src, float* dst, size_t n, cudaStream_t s);
// dst[r, 0:cols] = src[r, 0:cols] for r < rows (float32, row strides lds / ldd)
cudaError_t launch_copy_rows_f32(const float* src, int lds, float* dst, int ldd, int rows,
                                 int cols, cudaStream_t s);

// ----------------------------------------------------------------------------- tcgen05 GEMM
enum GemmEpi {
    EPI_STORE = 0,    // y = acc (+ residual), y f32 or bf16
    EPI_QKV = 1,      // q/k: per-head RMSNorm + NeoX RoPE -> bf16; v -> transposed f16 of bf16(v)
    EPI_SWIGLU = 2,   // gate/up interleaved in 64-column blocks -> silu(g)*u bf16
};

struct GemmEpiArgs {
    // e4m3 operands: y = a_scale[m] * b_scale[n] * (A B^T)[m, n] before the epilogue
    const float* a_scale = nullptr;   // [M]
    const float* b_scale = nullptr;   // [N]
    // EPI_STORE
    void* y = nullptr;
    int y_dtype = DTP_F32;
    long long ldy = 0;
    const float* residual = nullptr;    // f32 [M, ldy] (may alias y)
    // EPI_QKV
    __nv_bfloat16* q = nullptr;         // [M, n_head*hd]
    __nv_bfloat16* k = nullptr;         // [M, n_head_kv*hd]
    __half* vt = nullptr;               // [n_head_kv*hd, ldvt]: f16 copies of bf16(v)
    long long ldvt = 0;
    __nv_bfloat16* v_rows = nullptr;    // optional token-major v [M, n_head_kv*hd]
    const int* tok_pos = nullptr;       // optional per-row RoPE position (default: the row)
    const int* tok_vcol = nullptr;      // optional per-row v^T column (default: the row)
    int q_gated = 0;                    // q region holds [q | gate] per head
    __nv_bfloat16* gate = nullptr;      // [M, n_head*hd] raw gate values (when q_gated)
    const float* q_norm = nullptr;
    const float* k_norm = nullptr;
    const float2* rope = nullptr;       // [M, rope_dims/2] (cos, sin)
    int n_head = 0, n_head_kv = 0, head_dim = 0, rope_dims = 0;
    float eps = 0.f;
    // EPI_SWIGLU
    __nv_bfloat16* act = nullptr;       // [M, N/2]
    // RMSNorm fused across GEMMs (bf16 path).  Producer (EPI_STORE, f32 y): also
    // writes xb = bf16(y) and, per row, the sum of y^2 over each BN-wide tile into
    // ss_out[tile_n * ld_ss + row].  Consumer (EPI_QKV / EPI_SWIGLU, A = xb, the
    // weights pre-multiplied by the norm weights): every row is scaled by
    // 1 / sqrt(sum_t ss_in[t * ld_ss + row] / norm_cols + norm_eps) first.
    __nv_bfloat16* xb = nullptr;
    float* ss_out = nullptr;
    const float* ss_in = nullptr;
    int n_ss = 0, ld_ss = 0, norm_cols = 0;
    float norm_eps = 0.f;
};
// N-tiles of one row that launch_gemm_tc's EPI_STORE with float32 output uses
// (the number of ss_out partials it writes per row).
int gemm_tc_tiles_n(int M, int N);

// y-side work of one GEMM: x [M, K] bf16 (row stride K), W [N, K] bf16.
cudaError_t launch_gemm_tc(const __nv_bfloat16* x, const __nv_bfloat16* W, int M, int N, int K,
                           GemmEpi epi, const GemmEpiArgs& ea, cudaStream_t s, int kind);
// The same GEMM on float32 operands holding tf32 values (tcgen05 kind::tf32),
// EPI_STORE epilogue (float32 y, optional residual); K a multiple of 4.
cudaError_t launch_gemm_tc_tf32(const float* x, const float* W, int M, int N, int K,
                                const GemmEpiArgs& ea, cudaStream_t s, int kind);
// The same GEMM on e4m3 operands (tcgen05 kind::f8f6f4) with a float32 scale per
// row of x (ea.a_scale, [M]) and per row of W (ea.b_scale, [N]); K % 16 == 0.
cudaError_t launch_gemm_tc_e4m3(const uint8_t* x, const uint8_t* W, int M, int N, int K,
                                GemmEpi epi, const GemmEpiArgs& ea, cudaStream_t s, int kind);

cudaError_t launch_selftest_wait(cudaStream_t s);

// ----------------------------------------------------------------------------- tcgen05 attention
// q [T, n_head*hd] bf16, k [T, n_head_kv*hd] bf16, vt [n_head_kv*hd, ldvt] f16
// (f16 of the bf16 values), out [T, n_head*hd] bf16.  S = Q K^T on bf16 operands;
// P (f16) V^T (f16) on f16 operands.
cudaError_t launch_attn_tc(const __nv_bfloat16* q, const __nv_bfloat16* k,
                           const __half* vt, long long ldvt, __nv_bfloat16* out, int T,
                           int n_head, int n_head_kv, int head_dim, float scale, cudaStream_t s);
// Several sequences packed along the token axis (see seq_meta in simt.cu).
struct AttnVarlen {
    const __nv_bfloat16* gate = nullptr;   // optional [T, n_head*hd]: out *= sigmoid(gate)
    // one sequence: the T queries sit at positions p0 .. p0+T-1 and k / v^T hold
    // keys 0 .. p0+T-1 (chunked prefill against a KV state)
    int p0 = 0;
    int n_seq = 0;
    const int* cu_seqlens = nullptr;   // [n_seq + 1]
    const int* tile_start = nullptr;   // [n_seq + 1]
    const int* vcol_start = nullptr;   // [n_seq]
};
cudaError_t launch_attn_tc_varlen(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                  const __half* vt, long long ldvt, long long vt_cols,
                                  __nv_bfloat16* out, int T, int n_head, int n_head_kv,
                                  int head_dim, float scale, const AttnVarlen& vl,
                                  cudaStream_t s);
// The same flash attention on float32 q / k / v^T holding tf32 values (kind::tf32,
// P rounded to tf32, float32 output; no gate): q [T, ldq] with head h at column
// h * q_head_stride, k [rows, ldk], v^T [n_head_kv * hd, ldvt]; ldq, ldk, ldvt
// multiples of 4, 16-byte aligned bases.
cudaError_t launch_attn_tc_f32(const float* q, long long ldq, int q_head_stride, const float* k,
                               long long ldk, const float* vt, long long ldvt, long long vt_cols,
                               float* out, int T, int n_head, int n_head_kv, int head_dim,
                               float scale, const AttnVarlen& vl, cudaStream_t s);
bool attn_tc_supported(int n_head, int n_head_kv, int head_dim);

}  // namespace dtp
