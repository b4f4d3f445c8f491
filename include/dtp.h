/*
 * dtp.h -- C ABI of the GB300 (sm_103a) dense-transformer prefill library.
 *
 * The library computes the whole-sequence (prefill) forward pass of a
 * Qwen3-style dense decoder stack as stated on the page "docs.rs memra-engine
 * 0.130.0, src/forward.rs" (`Model::forward`):
 *
 *   x = tok_embd[tokens]                                  [T, n_embd]
 *   per layer:
 *     h    = rms_norm(x) * attn_norm
 *     q,k,v = h Wq^T, h Wk^T, h Wv^T                      [T, heads*head_dim]
 *     q,k  = rms_norm over each head_dim row * q_norm / k_norm
 *     q,k  = NeoX RoPE at positions 0..T-1 (rope_dim_count, rope_freq_base)
 *     attn = causal GQA softmax(q k^T / sqrt(head_dim)) v
 *     x    = x + attn Wo^T
 *     z    = rms_norm(x) * ffn_norm
 *     x    = x + (silu(z Wg^T) * (z Wu^T)) Wd^T
 *   logits = (rms_norm(x) * output_norm) Wout^T           [T, n_vocab] float32
 *
 * Conventions for every entry point:
 *   - Pointers documented "device" point to device memory of the current CUDA
 *     device; "host" pointers to host memory.  The caller allocates and owns
 *     every buffer; the library never frees caller memory and allocates no
 *     device memory on the forward path.
 *   - Matrices are row-major.  Activations are token-major [T, features]; a
 *     weight is [out_features, in_features] and a projection is y = x W^T.
 *   - Work is enqueued asynchronously on `stream` (NULL = the legacy default
 *     stream).  The return value reports argument validation and launch
 *     errors only; faults detected on the device (a token id out of range, a
 *     bounded pipeline wait that gave up) raise a device error word that
 *     dtp_check() reports after synchronising the stream.
 *   - Every function returns DTP_OK (0) or a negative DTP_ERR_* code and, on
 *     error, sets a message readable with dtp_last_error() (per thread).
 *   - Execution resources: the tensor-core GEMMs launch thread-block clusters
 *     of two CTAs, one CTA per SM, and take as many clusters as can be
 *     resident at once.  A context in which no two-CTA cluster of that size
 *     fits gets DTP_ERR_CUDA from the first GEMM.  The tensor-core attention
 *     launches one CTA of 320 threads per (query tile, head pair).
 */
#ifndef DTP_H
#define DTP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* dtp_stream_t;

enum {
    DTP_OK = 0,
    DTP_ERR_INVALID_ARG = -1,    /* null pointer, non-positive size, inconsistent shape       */
    DTP_ERR_UNSUPPORTED = -2,    /* valid shape that this build's kernels do not tile         */
    DTP_ERR_TOKEN_RANGE = -3,    /* a token id >= n_vocab                                     */
    DTP_ERR_WORKSPACE = -4,      /* workspace or packed buffer smaller than required          */
    DTP_ERR_CUDA = -5,           /* a CUDA runtime/driver call failed                         */
    DTP_ERR_DEVICE_TIMEOUT = -6, /* a kernel's bounded wait gave up (reported by dtp_check)   */
    DTP_ERR_VALUE_RANGE = -7     /* bf16 attention met a v value outside the f16 range or not
                                    finite (reported by dtp_check; see dtp_sdpa_causal_gqa)  */
};

/* Element type of an activation buffer.  DTP_TF32 is float32 storage whose
 * values are TensorFloat-32 (10-bit fraction; producers round to nearest,
 * ties to even): the operand type of the kind::tf32 tensor-core GEMM. */
enum { DTP_F32 = 0, DTP_BF16 = 1, DTP_TF32 = 2 };

/* Arithmetic of the forward pass.
 *   DTP_PREC_F32:  float32 everywhere (SIMT kernels; the pages' "all f32" stage).
 *   DTP_PREC_TF32: every GEMM on tcgen05 tensor cores with tf32 operands (the
 *                  weights and each GEMM input rounded to tf32) and float32
 *                  accumulation; attention on the tcgen05 flash-attention kernel
 *                  (kind::tf32: q/k/v and P rounded to tf32, float32 scores,
 *                  softmax and output; packed sequences and head_dim other than
 *                  64 / 128 use the float32 SIMT kernel on the same tf32 values);
 *                  residual stream, norms, QK-norm/RoPE, SwiGLU and logits in
 *                  float32.
 *   DTP_PREC_BF16: bf16 GEMM/attention operands, float32 accumulation, float32
 *                  residual stream, norms, softmax and logits (tcgen05 tensor cores).
 *   DTP_PREC_E4M3: quantised weights and GEMM inputs: every GEMM operand is OCP
 *                  FP8 E4M3 with one float32 scale per row (weights per output
 *                  channel, activations per token; scale = max|row| / 448, codes
 *                  nearest-even), tcgen05 kind::f8f6f4 with float32 accumulation
 *                  and the two scales applied in the epilogue; embedding, attention
 *                  (q/k/v, P) and the SwiGLU / attention outputs before their
 *                  quantisation are bf16, as in DTP_PREC_BF16. */
enum { DTP_PREC_F32 = 0, DTP_PREC_TF32 = 1, DTP_PREC_BF16 = 2, DTP_PREC_E4M3 = 3 };

typedef struct dtp_config {
    int n_layer;          /* decoder layers                                         */
    int n_embd;           /* model width d                                          */
    int n_head;           /* query heads h                                          */
    int n_head_kv;        /* key/value heads g; h % g == 0 (GQA group = h / g)      */
    int head_dim;         /* per-head width hd (even)                               */
    int rope_dim_count;   /* rotated dims r per head, even, r <= hd                 */
    int n_ff;             /* SwiGLU hidden width F                                  */
    int n_vocab;          /* vocabulary V                                           */
    float rope_freq_base; /* RoPE base; theta_i = base^(-2i/r)                      */
    float rms_eps;        /* epsilon inside every RMSNorm's square root             */
    int precision;        /* DTP_PREC_F32, _TF32, _BF16 or _E4M3                    */
    int attn_gate;        /* 1: gated attention -- the Q projection also yields, per head,
                             head_dim gate values after its head_dim q values, and the
                             attention output is multiplied by sigmoid(gate) before the
                             O projection (memra-engine spec.rs, `q_gate_split`); 0: none */
} dtp_config;

/* One layer's source weights: device float32, the pages' layouts. */
typedef struct dtp_layer_src {
    const float* attn_norm; /* [n_embd]                       */
    const float* wq;        /* [n_head*head_dim, n_embd]; with attn_gate
                               [n_head*2*head_dim, n_embd]: per head, head_dim q rows
                               then head_dim gate rows                            */
    const float* wk;        /* [n_head_kv*head_dim, n_embd]   */
    const float* wv;        /* [n_head_kv*head_dim, n_embd]   */
    const float* q_norm;    /* [head_dim]                     */
    const float* k_norm;    /* [head_dim]                     */
    const float* wo;        /* [n_embd, n_head*head_dim]      */
    const float* ffn_norm;  /* [n_embd]                       */
    const float* w_gate;    /* [n_ff, n_embd]                 */
    const float* w_up;      /* [n_ff, n_embd]                 */
    const float* w_down;    /* [n_embd, n_ff]                 */
} dtp_layer_src;

/* ------------------------------------------------------------------------------------
 * Model weights: packing
 *
 * The forward pass reads weights from one caller-owned device buffer in the
 * library's packed format: per layer Wq;Wk;Wv concatenated into one [(h+2g)hd, d]
 * matrix, Wgate and Wup interleaved in blocks of 64 rows into one [2F, d] matrix,
 * Wo, Wdown, and the four norm vectors; then tok_embd [V, d], output_norm [d]
 * and the lm_head [V, d].  Matrices are stored as bf16 (round to nearest even)
 * under DTP_PREC_BF16, float32 under DTP_PREC_F32, and float32 rounded to tf32
 * (nearest even) under DTP_PREC_TF32, except tok_embd, which stays float32.
 * Under DTP_PREC_BF16 the RMSNorm before the QKV and gate/up projections is
 * fused into them: Wq;Wk;Wv are stored multiplied column-wise by attn_norm and
 * Wgate/Wup by ffn_norm (rounded once, after the product).
 * Under DTP_PREC_E4M3 the matrices are e4m3 codes, each followed by its float32
 * row scales, and tok_embd is bf16.  Norm vectors are float32.
 * ------------------------------------------------------------------------------------ */

/* Bytes of the packed buffer for `cfg` (0 if cfg is invalid). */
size_t dtp_packed_size(const dtp_config* cfg);

/* Convert and write layer `layer` (0 <= layer < n_layer) from `src` (device
 * float32, all 11 pointers non-null) into `packed` (device, packed_bytes >=
 * dtp_packed_size(cfg)).  Asynchronous on `stream`; `src` must stay valid until
 * the stream reaches this point. */
int dtp_pack_layer(const dtp_config* cfg, int layer, const dtp_layer_src* src, void* packed,
                   size_t packed_bytes, dtp_stream_t stream);

/* Write the token embedding tok_embd [V, d], output_norm [d] and the lm_head
 * output [V, d] (device float32) into `packed`. */
int dtp_pack_globals(const dtp_config* cfg, const float* tok_embd, const float* output_norm,
                     const float* output, void* packed, size_t packed_bytes, dtp_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Forward pass  (forward.rs, `Model::forward`)
 * ------------------------------------------------------------------------------------ */

/* Bytes of device workspace dtp_fwd_prefill needs for T tokens (0 if invalid). */
size_t dtp_workspace_size(const dtp_config* cfg, int T);

/* Prefill forward over T >= 1 tokens at positions 0..T-1.
 *   tokens   device uint32 [T], each < n_vocab (checked on the device: an id out
 *            of range raises DTP_ERR_TOKEN_RANGE in dtp_check and its row is zero).
 *   logits   device float32 [T, n_vocab], written.
 *   hidden   device float32 [n_layer + 1, T, n_embd] or NULL; if given, hidden[l]
 *            is the residual stream entering layer l and hidden[n_layer] the
 *            stream entering output_norm.
 *   workspace device, >= dtp_workspace_size(cfg, T) bytes, 256-byte aligned,
 *            owned by the caller; contents on entry are ignored.
 * Buffers may not overlap. */
int dtp_fwd_prefill(const dtp_config* cfg, const void* packed, size_t packed_bytes,
                    const uint32_t* tokens, int T, float* logits, float* hidden, void* workspace,
                    size_t ws_bytes, dtp_stream_t stream);

/* Outputs of dtp_fwd_prefill_ex; every pointer may be NULL (at least one given). */
typedef struct dtp_fwd_outputs {
    float* logits;   /* device float32 [T, n_vocab], or [1, n_vocab] with last_only;
                        NULL skips the output norm and the lm_head                        */
    int last_only;   /* nonzero: logits of position T-1 only (forward.rs `forward_last`) */
    float* hidden;   /* device float32 [n_layer + 1, T, n_embd], as in dtp_fwd_prefill      */
    void* k_cache;   /* device [n_layer, T, n_head_kv*head_dim]: every layer's keys after
                        QK-norm and RoPE (what attention consumed), token-major; bf16 under
                        DTP_PREC_BF16 / _E4M3, float32 otherwise -- a decode KV cache      */
    void* v_cache;   /* device [n_layer, T, n_head_kv*head_dim]: every layer's values, same
                        dtype and layout as k_cache                                         */
} dtp_fwd_outputs;

/* dtp_fwd_prefill with a choice of outputs: last-position logits only
 * (forward.rs `forward_last`), and/or the per-layer K/V a decode step continues
 * from.  Same workspace as dtp_fwd_prefill. */
int dtp_fwd_prefill_ex(const dtp_config* cfg, const void* packed, size_t packed_bytes,
                       const uint32_t* tokens, int T, const dtp_fwd_outputs* out, void* workspace,
                       size_t ws_bytes, dtp_stream_t stream);

/* Several independent sequences in one pass ("varlen" prefill).  Sequence b
 * holds tokens[cu_seqlens[b] .. cu_seqlens[b+1]) at positions 0..len_b-1 and
 * attends only to itself; the projections, norms and FFN run over all `total`
 * tokens at once.
 *   tokens      device uint32 [total]
 *   cu_seqlens  device int32 [n_seq + 1], 0 = cu[0] <= cu[1] <= ... <= cu[n_seq] =
 *               total (checked on the device: otherwise dtp_check reports
 *               DTP_ERR_INVALID_ARG and no attention is computed)
 *   out         as for dtp_fwd_prefill_ex over the `total` packed tokens, except
 *               that last_only gives logits [n_seq, n_vocab], one row per
 *               sequence (an empty sequence's row is unspecified)
 *   workspace   >= dtp_workspace_size_varlen(cfg, total, n_seq) bytes. */
size_t dtp_workspace_size_varlen(const dtp_config* cfg, int total, int n_seq);
int dtp_fwd_prefill_varlen(const dtp_config* cfg, const void* packed, size_t packed_bytes,
                           const uint32_t* tokens, const int32_t* cu_seqlens, int n_seq, int total,
                           const dtp_fwd_outputs* out, void* workspace, size_t ws_bytes,
                           dtp_stream_t stream);

/* Chunked prefill of one sequence against a growing KV state.  The forward.rs
 * `Model::forward` pass is causal, so positions p0 .. p0+C-1 depend on the
 * earlier positions only through every layer's keys and values (after QK-norm
 * and RoPE).  A call processes the C tokens at those positions, reading the
 * keys and values of positions 0 .. p0-1 from `kv_state` (left there by the
 * earlier calls) and writing its own; the chunks' logits, concatenated, equal
 * the logits of one dtp_fwd_prefill over the whole sequence.
 *
 * KV state (device, caller-owned, 256-byte aligned, dtp_kv_state_size bytes
 * for up to max_T positions; nk = n_head_kv*head_dim): per layer l, at byte
 * offset l * S with S the per-layer stride below,
 *   DTP_PREC_BF16 / DTP_PREC_E4M3:
 *                  K  bf16 [max_T, nk] token-major, then (256-byte aligned)
 *                  V^T f16 [nk, ldvt], ldvt = max_T rounded up to 8: f16 copies
 *                  of the bf16 values (exact; the attention's P V^T product takes
 *                  f16 operands)
 *   DTP_PREC_TF32: the same with float32 elements (with a head_dim other than 64
 *                  or 128, or an odd n_head / n_head_kv, V is token-major
 *                  [max_T, nk] inside the V^T region instead)
 *   DTP_PREC_F32:  K  f32 [max_T, nk], then (256-byte aligned) V f32 [max_T, nk]
 * Positions >= p0 + C are neither read nor written.  Calls on one state run
 * in position order (the stream orders them).
 *   tokens     device uint32 [C]
 *   p0, C      p0 >= 0, C >= 1, p0 + C <= max_T
 *   out        logits ([C, n_vocab], or the last position's with last_only) and
 *              hidden ([n_layer + 1, C, n_embd]); k_cache / v_cache must be NULL
 *              (the state holds them)
 *   workspace  >= dtp_workspace_size(cfg, C) bytes
 * Errors: DTP_ERR_INVALID_ARG for a range or pointer problem, DTP_ERR_WORKSPACE
 * for a short state or workspace; nothing is enqueued then. */
size_t dtp_kv_state_size(const dtp_config* cfg, int max_T);
int dtp_fwd_prefill_chunk(const dtp_config* cfg, const void* packed, size_t packed_bytes,
                          const uint32_t* tokens, int C, int p0, void* kv_state,
                          size_t state_bytes, int max_T, const dtp_fwd_outputs* out,
                          void* workspace, size_t ws_bytes, dtp_stream_t stream);

/* Bytes of device workspace dtp_fwd_prefill_host needs (the forward workspace
 * plus device staging for the tokens and logits). */
size_t dtp_workspace_size_host(const dtp_config* cfg, int T);

/* The same pass with HOST tokens (uint32 [T]) and HOST logits (float32
 * [T, n_vocab]): copies the tokens in, runs dtp_fwd_prefill, copies the
 * logits out, all enqueued on `stream`; the caller synchronises the stream
 * before reading `logits_host`.  Token ids are range-checked on the host
 * before anything is enqueued.  Page-locked host buffers make the copies
 * asynchronous. */
int dtp_fwd_prefill_host(const dtp_config* cfg, const void* packed, size_t packed_bytes,
                         const uint32_t* tokens_host, int T, float* logits_host, void* workspace,
                         size_t ws_bytes, dtp_stream_t stream);

/* n prompts of T tokens each, host to host, in order: prompt j's tokens are
 * copied in, its forward pass runs on `stream`, and its logits are copied out to
 * logits_host[j] on a device-to-host stream of the library's own, so that the
 * copy of prompt j overlaps the forward pass of prompt j + 1.  The passes write
 * nb device logit buffers in turn (prompt j: buffer j % nb), and a pass waits
 * for the copy that last used its buffer, so a slow copy holds the passes back
 * only once the other nb - 1 buffers are full.  nb is the largest count from
 * 2 to 8 whose workspace fits in ws_bytes.  Everything is enqueued before the
 * call returns; `stream` completes only after the last copy has landed, so
 * synchronising `stream` makes every logits_host[j] readable.
 *   tokens_host  n host pointers to uint32 [T] (range-checked on the host first)
 *   logits_host  n host pointers to float32 [T, n_vocab] (page-locked memory makes
 *                the copies asynchronous)
 *   workspace    >= dtp_workspace_size_host_batch(cfg, T) bytes (two logit
 *                buffers); dtp_workspace_size_host_batch_n(cfg, T, nb) bytes
 *                for nb of them (each adds T * n_vocab * 4 bytes)
 * One call at a time per device: the library's copy stream is shared.
 * dtp_workspace_size_host_batch_n returns 0 for nb outside 2..8. */
size_t dtp_workspace_size_host_batch(const dtp_config* cfg, int T);
size_t dtp_workspace_size_host_batch_n(const dtp_config* cfg, int T, int n_buffers);
int dtp_fwd_prefill_host_batch(const dtp_config* cfg, const void* packed, size_t packed_bytes,
                               const uint32_t* const* tokens_host, int n, int T,
                               float* const* logits_host, void* workspace, size_t ws_bytes,
                               dtp_stream_t stream);

/* Synchronise `stream`, then report and clear the device error words raised
 * by this library's kernels since the last call: DTP_OK,
 * DTP_ERR_TOKEN_RANGE, DTP_ERR_DEVICE_TIMEOUT, DTP_ERR_VALUE_RANGE,
 * DTP_ERR_INVALID_ARG (packed-sequence offsets), or DTP_ERR_CUDA (a sticky
 * CUDA error). */
int dtp_check(dtp_stream_t stream);

/* Message for the last error raised on the calling thread ("" if none). */
const char* dtp_last_error(void);

/* ------------------------------------------------------------------------------------
 * Per-op entry points (the steps of forward.rs `Model::forward`)
 * ------------------------------------------------------------------------------------ */

/* RMSNorm (forward.rs, Model::forward: the engine's row RMSNorm step over
 * nrows rows of ncols values with a weight vector and eps):
 * y[r, c] = x[r, c] / sqrt(mean_c(x[r, :]^2) + eps) * w[c].
 * x device float32 [rows, cols]; w device float32 [cols]; y device [rows, cols]
 * of y_dtype (DTP_F32, DTP_BF16 or DTP_TF32; bf16 / tf32 rounded to nearest
 * even).  y may alias x when y_dtype is DTP_F32 or DTP_TF32. */
int dtp_rms_norm(const float* x, const float* w, void* y, int y_dtype, int rows, int cols,
                 float eps, dtp_stream_t stream);

/* Per-head QK-RMSNorm then NeoX RoPE, in place (forward.rs, Model::forward:
 * the QK-norm step, an RMSNorm over rows of head_dim values, heads*T rows,
 * then the NeoX rotation of rope_dim_count dims per head at the token
 * positions, base freq_base, frequency scale 1).
 * x device [T, n_heads*head_dim] of dtype (DTP_F32 or DTP_BF16);
 * w_norm device float32 [head_dim], or NULL to apply RoPE only;
 * pos device int32 [T] positions, or NULL for 0..T-1.
 * For each (token t, head) row: y = rms_norm(row) * w_norm, then for
 * i < r/2 the pair (i, i + r/2) is rotated by angle pos[t] * base^(-2i/r);
 * dims >= r are unchanged.  Arithmetic in float32 (angles in float64). */
int dtp_qk_norm_rope_neox(void* x, int dtype, const float* w_norm, const int32_t* pos, int T,
                          int n_heads, int head_dim, int rope_dim_count, float freq_base,
                          float eps, dtp_stream_t stream);

/* Device workspace dtp_sdpa_causal_gqa needs (0 for DTP_F32). */
size_t dtp_sdpa_workspace_size(int T, int n_head_kv, int head_dim, int dtype);

/* Causal grouped-query attention (forward.rs, Model::forward: the attention
 * step, causal, with as many keys as queries and the caller's scale):
 * out[t, i] = sum_{s<=t} softmax_s(scale * q[t,i].k[s,j]) v[s,j],
 * j = i / (n_head / n_head_kv).
 * q, out device [T, n_head*head_dim]; k, v device [T, n_head_kv*head_dim];
 * all of dtype.  DTP_F32: float32 SIMT kernel.  DTP_BF16: tcgen05 flash
 * attention: q k^T on bf16 operands, float32 scores/softmax/accumulation, and
 * the PV product on f16 operands (P rounded to f16; v converted to f16, which
 * holds every bf16 value exactly from 2^-14 up to 65504 and rounds smaller
 * magnitudes to its subnormal grid, an absolute error of at most 2^-25; every
 * |v| must be at most 65504 -- otherwise dtp_check reports
 * DTP_ERR_VALUE_RANGE and the output is not meaningful).  DTP_TF32: the same on float32 buffers holding tf32
 * values (kind::tf32, P rounded to tf32, float32 output).  The tensor-core
 * kinds require head_dim 64 or 128 and an even group size n_head / n_head_kv,
 * and a workspace of dtp_sdpa_workspace_size bytes (device, 256-byte aligned). */
int dtp_sdpa_causal_gqa(const void* q, const void* k, const void* v, void* out, int dtype, int T,
                        int n_head, int n_head_kv, int head_dim, float scale, void* workspace,
                        size_t ws_bytes, dtp_stream_t stream);

/* Allocation-free variant of dtp_sdpa_causal_gqa for dtype DTP_BF16.  The
 * paper has no counterpart: this entry point exists for callers that cannot
 * allocate device memory where they call attention -- an op handed only its
 * input and output tensors, code running inside a stream-ordered region it
 * does not own, or a runtime that forbids cudaMalloc after start-up.
 * Same arguments, layouts and result as dtp_sdpa_causal_gqa with dtype
 * DTP_BF16, minus the workspace: the transposed-V scratch lives in a fixed
 * 8 MiB device array inside the library (held on every GPU that loads the
 * library until the process exits).
 *   - Limit: n_head_kv * head_dim * (T rounded up to 8) * 2 bytes must not
 *     exceed 8 MiB (e.g. 8 kv heads x 128 dims x 4096 tokens); larger calls
 *     return DTP_ERR_WORKSPACE without launching anything.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address once; make that first call before any stream
 *     capture.
 *   - All calls share the one array: calls that overlap on the GPU (for
 *     example on two streams at once) race on it.  Each call rewrites every
 *     scratch element it reads, so nothing needs clearing between calls.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
int dtp_sdpa_causal_gqa_noalloc(const void* q, const void* k, const void* v, void* out, int T,
                                int n_head, int n_head_kv, int head_dim, float scale,
                                dtp_stream_t stream);

/* SwiGLU (forward.rs, Model::forward: the FFN activation of the dense arm;
 * the T-parallel page names the same step silu_mul):
 * out[i] = silu(gate[i]) * up[i], silu(x) = x / (1 + e^-x); n elements of
 * dtype, arithmetic in float32.  out may alias gate or up. */
int dtp_swiglu(const void* gate, const void* up, void* out, int dtype, size_t n,
               dtp_stream_t stream);

/* Linear (forward.rs, Model::forward: a projection matmul, plus the residual
 * add when a residual is given): y[M, N] = x[M, K] W[N, K]^T
 * (+ residual[M, N]).
 * x, W device, both of dtype: DTP_F32 -> float32 SIMT kernel; DTP_BF16 ->
 * tcgen05 tensor cores with float32 accumulation (K % 8 == 0); DTP_TF32 ->
 * tcgen05 kind::tf32 with float32 accumulation (K % 4 == 0, y_dtype DTP_F32;
 * x and W hold tf32 values -- float32 with the low 13 fraction bits zero).
 * y device of y_dtype (DTP_F32 or DTP_BF16).  residual: device float32
 * [M, N] or NULL; when given, y_dtype must be DTP_F32 and y = residual + x W^T;
 * residual may alias y (in-place residual add). */
int dtp_linear(const void* x, const void* W, void* y, int dtype, int y_dtype, int M, int N, int K,
               const float* residual, dtp_stream_t stream);

/* Per-row e4m3 quantisation of a GEMM operand (the DTP_PREC_E4M3 arithmetic; the
 * pages' T-parallel path quantises each activation row to 8 bits before its
 * matmul, `quantize_q8_1`): for each row r of x, scale[r] = max|x[r]| / 448 and
 * q[r, c] = e4m3(x[r, c] * (448 / max|x[r]|)), nearest-even, saturating; a zero
 * row gives scale 0 and zero codes.
 *   x      device [rows, cols] of dtype DTP_F32 or DTP_BF16 (cols % 8 == 0 for bf16)
 *   q      device uint8 [rows, cols] (e4m3 codes, row-major)
 *   scale  device float32 [rows] */
int dtp_quantize_rows_e4m3(const void* x, int dtype, int rows, int cols, uint8_t* q, float* scale,
                           dtp_stream_t stream);

/* rms_norm written as per-row e4m3 codes: y = rms_norm(x) * w as in dtp_rms_norm
 * (float32), then quantised as in dtp_quantize_rows_e4m3 (q [rows, cols], scale
 * [rows]); cols % 4 == 0 and cols <= 16384, x and w 16-byte aligned. */
int dtp_rms_norm_e4m3(const float* x, const float* w, uint8_t* q, float* scale, int rows, int cols,
                      float eps, dtp_stream_t stream);

/* Linear on e4m3 operands: y[M, N] = x_scale[m] * w_scale[n] * (xq wq^T)[m, n]
 * (+ residual), tcgen05 kind::f8f6f4 with float32 accumulation.
 *   xq [M, K], wq [N, K]  device e4m3 codes (dtp_quantize_rows_e4m3), K % 16 == 0,
 *                         16-byte aligned
 *   x_scale [M], w_scale [N]  device float32 row scales
 *   y      device float32 [M, N]; residual as for dtp_linear (may alias y) */
int dtp_linear_e4m3(const uint8_t* xq, const float* x_scale, const uint8_t* wq,
                    const float* w_scale, float* y, int M, int N, int K, const float* residual,
                    dtp_stream_t stream);

/* Fused QKV projection with per-head QK-RMSNorm and NeoX RoPE: the bf16 path's
 * first GEMM of a layer (forward.rs, Model::forward: the three Q/K/V
 * projections, the QK-norm over head_dim rows and the NeoX rotation, as one tcgen05 GEMM whose
 * epilogue normalises and rotates each head at positions 0..T-1).
 *   h      device bf16 [T, d] (the normed layer input)
 *   w_qkv  device bf16 [(n_head + 2 n_head_kv) * head_dim, d]: Wq rows, then Wk, then Wv
 *   q_norm, k_norm  device float32 [head_dim]
 *   q      device bf16 [T, n_head*head_dim]     (written)
 *   k      device bf16 [T, n_head_kv*head_dim]  (written)
 *   vt     device f16 [n_head_kv*head_dim, ldvt], v transposed, each value
 *          f16(bf16(v)): exact from 2^-14 up to 65504, smaller magnitudes on
 *          f16's subnormal grid (written; columns T..ldvt-1 untouched);
 *          ldvt >= T, ldvt % 8 == 0.  A |v| beyond 65504 (the f16 range) raises
 *          DTP_ERR_VALUE_RANGE in dtp_check.
 *   workspace  device, >= dtp_qkv_norm_rope_workspace_size(T, rope_dim_count)
 *          bytes, 16-byte aligned (the cos/sin table).
 * Requires d % 8 == 0, head_dim 64 or 128, (rope_dim_count/2) % 32 == 0 and
 * (head_dim - rope_dim_count) % 32 == 0. */
size_t dtp_qkv_norm_rope_workspace_size(int T, int rope_dim_count);
int dtp_qkv_norm_rope(const void* h, const void* w_qkv, const float* q_norm, const float* k_norm,
                      void* q, void* k, void* vt, int ldvt, int T, int d, int n_head,
                      int n_head_kv, int head_dim, int rope_dim_count, float freq_base, float eps,
                      void* workspace, size_t ws_bytes, dtp_stream_t stream);

/* Fused gate/up projection and SwiGLU: the bf16 path's FFN GEMM (forward.rs:
 * the gate and up projections and the FFN activation).
 *   z      device bf16 [T, d]
 *   w_gu   device bf16 [2*n_ff, d]: gate and up rows interleaved in blocks of 64
 *          (rows 128b..128b+63 = gate rows 64b..64b+63, rows 128b+64..128b+127 =
 *          up rows 64b..64b+63), the layout dtp_pack_layer writes
 *   act    device bf16 [T, n_ff]: act = silu(z Wgate^T) * (z Wup^T)  (written)
 * Requires d % 8 == 0 and n_ff % 64 == 0. */
int dtp_gate_up_swiglu(const void* z, const void* w_gu, void* act, int T, int d, int n_ff,
                       dtp_stream_t stream);

/* Failure-detection self-test.  Launches one CTA whose thread waits, through
 * the same bounded wait every pipeline kernel uses, on an mbarrier that nothing
 * arrives at.  After about one second the wait gives up, raises the device
 * error word and the kernel returns; dtp_check then reports
 * DTP_ERR_DEVICE_TIMEOUT and the CUDA context stays usable.  Returns the
 * launch status. */
int dtp_selftest_wait_timeout(dtp_stream_t stream);

/* ------------------------------------------------------------------------------------
 * Kernel timing (measurement aid; off by default)
 * ------------------------------------------------------------------------------------ */

/* Kernel kinds of the forward pass. */
enum {
    DTP_K_EMBED = 0, DTP_K_RMSNORM = 1, DTP_K_GEMM_QKV = 2, DTP_K_ATTN = 3, DTP_K_GEMM_O = 4,
    DTP_K_GEMM_GATEUP = 5, DTP_K_GEMM_DOWN = 6, DTP_K_GEMM_LMHEAD = 7, DTP_K_OTHER = 8,
    /* spans of dtp_fwd_prefill_host_batch, not single kernels (not counted by
     * dtp_launch_count): one prompt's whole pass on the caller's stream, and
     * one prompt's logits copy on the library's copy stream */
    DTP_K_PROMPT = 9, DTP_K_D2H = 10,
    DTP_K_COUNT = 11
};

/* Start recording a CUDA event pair around each launch of every kernel kind
 * in `kind_mask` (bit k = kind k), up to `capacity` launches per kind.  Creates
 * the events (no device memory).  Replaces any earlier recording. */
int dtp_timer_enable(unsigned kind_mask, int capacity);

/* Stop recording and destroy the events. */
int dtp_timer_disable(void);

/* After the recorded work has completed: number of recorded launches of
 * `kind` and their summed duration in milliseconds. */
int dtp_timer_read(int kind, int* count, float* total_ms);

/* After the recorded work has completed: start and end of each recorded launch
 * (or span) of `kind`, in milliseconds after the start of the first recorded
 * launch of `ref_kind` (negative if earlier), for the first `cap` of them;
 * *count = the number recorded.  start_ms / end_ms: host float [cap]. */
int dtp_timer_spans(int kind, int ref_kind, int cap, float* start_ms, float* end_ms, int* count);

/* Launch counter: kernels this library has launched on the calling process
 * since the last reset (every kernel of every entry point). */
long long dtp_launch_count(int reset);

#ifdef __cplusplus
}
#endif
#endif /* DTP_H */
