// C ABI of the prefill library: argument validation, the packed-weight and
// workspace layouts, the forward-pass orchestration ("docs.rs memra-engine
// 0.130.0, src/forward.rs", Model::forward), per-op entry points, tensor-map
// encoding, kernel timers and the device error words.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"

namespace dtp {

// ----------------------------------------------------------------------------- errors
static thread_local char t_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof(t_err), fmt, ap);
    va_end(ap);
    return code;
}
void clear_error() { t_err[0] = 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 148;
    }
    return cached[dev];
}

// ----------------------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elt_bytes,
                  uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows,
                  uint32_t box_cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * (uint64_t)elt_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ----------------------------------------------------------------------------- timers
struct TimerState {
    std::mutex mu;
    unsigned mask = 0;
    int capacity = 0;
    std::vector<cudaEvent_t> ev[DTP_K_COUNT][2];
    int used[DTP_K_COUNT] = {0};
};
static TimerState g_timer;
static std::atomic<long long> g_launches{0};

LaunchScope::LaunchScope(int k, cudaStream_t s, bool counts) : kind(k), stream(s), slot(-1) {
    if (counts) g_launches.fetch_add(1, std::memory_order_relaxed);
    if (!g_timer.mask) return;
    std::lock_guard<std::mutex> lk(g_timer.mu);
    if (!(g_timer.mask & (1u << kind)) || g_timer.used[kind] >= g_timer.capacity) return;
    slot = g_timer.used[kind]++;
    cudaEventRecord(g_timer.ev[kind][0][slot], stream);
}
LaunchScope::~LaunchScope() {
    if (slot >= 0) cudaEventRecord(g_timer.ev[kind][1][slot], stream);
}

static void timer_destroy() {
    for (int k = 0; k < DTP_K_COUNT; ++k) {
        for (int j = 0; j < 2; ++j) {
            for (cudaEvent_t e : g_timer.ev[k][j]) cudaEventDestroy(e);
            g_timer.ev[k][j].clear();
        }
        g_timer.used[k] = 0;
    }
    g_timer.mask = 0;
    g_timer.capacity = 0;
}

// ----------------------------------------------------------------------------- layouts
static int validate_config(const dtp_config* c) {
    if (!c) return fail(DTP_ERR_INVALID_ARG, "config is NULL");
    if (c->n_layer < 0 || c->n_embd <= 0 || c->n_head <= 0 || c->n_head_kv <= 0 ||
        c->head_dim <= 0 || c->n_ff <= 0 || c->n_vocab <= 0)
        return fail(DTP_ERR_INVALID_ARG, "config sizes must be positive");
    if (c->n_head % c->n_head_kv)
        return fail(DTP_ERR_INVALID_ARG, "n_head (%d) is not a multiple of n_head_kv (%d)",
                    c->n_head, c->n_head_kv);
    if (c->head_dim % 2 || c->rope_dim_count <= 0 || c->rope_dim_count % 2 ||
        c->rope_dim_count > c->head_dim)
        return fail(DTP_ERR_INVALID_ARG, "rope_dim_count must be even and in [2, head_dim]");
    if (!(c->rms_eps >= 0.f) || !(c->rope_freq_base > 0.f))
        return fail(DTP_ERR_INVALID_ARG, "rms_eps must be >= 0 and rope_freq_base > 0");
    if (c->precision != DTP_PREC_F32 && c->precision != DTP_PREC_TF32 &&
        c->precision != DTP_PREC_BF16 && c->precision != DTP_PREC_E4M3)
        return fail(DTP_ERR_INVALID_ARG, "unknown precision %d", c->precision);
    if (c->attn_gate != 0 && c->attn_gate != 1)
        return fail(DTP_ERR_INVALID_ARG, "attn_gate must be 0 or 1");
    if (c->n_embd % 8 || c->n_ff % 64)
        return fail(DTP_ERR_UNSUPPORTED, "n_embd must be a multiple of 8 and n_ff of 64");
    if (c->precision == DTP_PREC_TF32 && (c->n_head * c->head_dim) % 4)
        return fail(DTP_ERR_UNSUPPORTED, "tf32 path: n_head*head_dim must be a multiple of 4");
    if (c->precision == DTP_PREC_E4M3 &&
        ((c->n_head * c->head_dim) % 16 || c->n_embd % 16 || c->n_embd > 16384))
        return fail(DTP_ERR_UNSUPPORTED,
                    "e4m3 path: n_embd and n_head*head_dim must be multiples of 16, n_embd <= 16384");
    if (c->precision == DTP_PREC_BF16 || c->precision == DTP_PREC_E4M3) {
        if (c->head_dim != 64 && c->head_dim != 128)
            return fail(DTP_ERR_UNSUPPORTED, "bf16 path: head_dim must be 64 or 128");
        if ((c->rope_dim_count / 2) % 32 || (c->head_dim - c->rope_dim_count) % 32)
            return fail(DTP_ERR_UNSUPPORTED,
                        "bf16 path: rope_dim_count/2 and head_dim-rope_dim_count must be "
                        "multiples of 32");
    }
    return DTP_OK;
}

struct PackedLayout {
    size_t elt = 4;         // bytes per matrix element (1 for e4m3)
    size_t emb_elt = 4;     // bytes per tok_embd element
    size_t attn_norm, w_qkv, q_norm, k_norm, wo, ffn_norm, w_gu, w_down;   // within a layer
    size_t w_qkv_s = 0, wo_s = 0, w_gu_s = 0, w_down_s = 0;               // e4m3 row scales
    size_t layer_bytes;
    size_t tok_embd, output_norm, output, output_s = 0;                   // absolute
    size_t total;
};

static PackedLayout packed_layout(const dtp_config* c) {
    PackedLayout L;
    const bool e4 = c->precision == DTP_PREC_E4M3;
    L.elt = c->precision == DTP_PREC_BF16 ? 2 : (e4 ? 1 : 4);
    L.emb_elt = (c->precision == DTP_PREC_BF16 || e4) ? 2 : 4;
    const size_t d = c->n_embd, hd = c->head_dim, nq = (size_t)c->n_head * hd,
                 nqkv = (size_t)(c->n_head * (1 + c->attn_gate) + 2 * c->n_head_kv) * hd,
                 F = c->n_ff;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.w_qkv = take(nqkv * d * L.elt);
    L.wo = take(d * nq * L.elt);
    L.w_gu = take(2 * F * d * L.elt);
    L.w_down = take(d * F * L.elt);
    if (e4) {       // one float32 scale per weight row (output channel)
        L.w_qkv_s = take(nqkv * 4);
        L.wo_s = take(d * 4);
        L.w_gu_s = take(2 * F * 4);
        L.w_down_s = take(d * 4);
    }
    L.attn_norm = take(d * 4);
    L.q_norm = take(hd * 4);
    L.k_norm = take(hd * 4);
    L.ffn_norm = take(d * 4);
    L.layer_bytes = o;
    o = L.layer_bytes * c->n_layer;
    L.tok_embd = take((size_t)c->n_vocab * d * L.emb_elt);
    L.output = take((size_t)c->n_vocab * d * L.elt);
    if (e4) L.output_s = take((size_t)c->n_vocab * 4);
    L.output_norm = take(d * 4);
    L.total = o;
    return L;
}

struct Workspace {
    size_t x, h, qkv, attn, gu, act;            // f32 path
    size_t q, k, vt, rope, gate;                 // bf16 path
    long long ldvt;
    size_t q8, s8;                               // e4m3 GEMM operand + row scales
    size_t ssp;                                  // bf16: fused RMSNorm partial sums [tiles][T]
    size_t tokens, logits, logits_more;          // _host staging (logits_more: the batch's
                                                 // further logit buffers)
    size_t tile_start, vcol_start, last_row, tok_pos, tok_vcol;   // packed sequences
    size_t total;
};

// Device logit buffers of dtp_fwd_prefill_host_batch: with nb buffers, prompt
// j's pass writes buffer j % nb, which is free again once prompt j - nb's
// logits copy has landed, so a slow copy stalls the passes only after the
// other nb - 1 buffers fill up.  nb is what the caller's workspace holds,
// between 2 and kMaxBatchBuffers.
constexpr int kMinBatchBuffers = 2;
constexpr int kMaxBatchBuffers = 8;

// Workspace for T tokens; n_seq > 0 adds the packed-sequence schedule and pads
// each sequence's v^T block to a multiple of 8 columns; host adds the token and
// logit staging (batch_buffers logit buffers with a batch).
static Workspace workspace_layout(const dtp_config* c, int T, bool host, int n_seq = 0,
                                  int batch_buffers = 0) {
    Workspace W = {};
    const size_t d = c->n_embd, hd = c->head_dim, nq = (size_t)c->n_head * hd,
                 nk = (size_t)c->n_head_kv * hd, F = c->n_ff;
    const bool e4 = c->precision == DTP_PREC_E4M3;
    const bool bf = c->precision == DTP_PREC_BF16 || e4;    // e4m3 runs the bf16 path
    const size_t e = bf ? 2 : 4;
    size_t o = 256;     // first 256 bytes reserved
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    W.x = take((size_t)T * d * 4);
    W.h = take((size_t)T * d * e);
    W.attn = take((size_t)T * nq * e);
    W.act = take((size_t)T * F * e);
    if (bf) {
        W.ldvt = (long long)align_up((size_t)T + (n_seq > 0 ? 7 * (size_t)n_seq : 0), 8);
        W.q = take((size_t)T * nq * 2);
        W.k = take((size_t)T * nk * 2);
        W.vt = take(nk * (size_t)W.ldvt * 2);
        W.rope = take((size_t)T * (c->rope_dim_count / 2) * sizeof(float2));
        if (c->attn_gate) W.gate = take((size_t)T * nq * 2);
        if (e4) {       // one operand buffer, reused by each GEMM in turn
            W.q8 = take((size_t)T * std::max(std::max(d, nq), F));
            W.s8 = take(align_up((size_t)T, 128) * 4);
        } else {        // one partial per 128 columns at most (the narrowest tile)
            W.ssp = take(((d + 127) / 128) * (size_t)T * 4);
        }
    } else {
        W.qkv = take((size_t)T * (nq * (1 + c->attn_gate) + 2 * nk) * 4);
        W.gu = take((size_t)T * 2 * F * 4);
        if (c->precision == DTP_PREC_TF32) {     // v^T for the tcgen05 tf32 attention
            W.ldvt = (long long)align_up((size_t)T, 8);
            W.vt = take(nk * (size_t)W.ldvt * 4);
        }
    }
    if (host) {
        W.tokens = take((size_t)T * 4);
        W.logits = take((size_t)T * c->n_vocab * 4);
        if (batch_buffers > 1)
            W.logits_more = take((size_t)(batch_buffers - 1) * T * c->n_vocab * 4);
    }
    if (n_seq > 0) {
        W.tile_start = take(((size_t)n_seq + 2) * 4);
        W.vcol_start = take((size_t)n_seq * 4);
        W.last_row = take((size_t)n_seq * 4);
        W.tok_pos = take((size_t)T * 4);
        W.tok_vcol = take((size_t)T * 4);
    }
    W.total = o;
    return W;
}

// Packed-sequence context of one forward call (n_seq == 0: a single sequence).
struct VarlenCtx {
    int n_seq = 0;
    const int* cu = nullptr;
    int* tile_start = nullptr;
    int* vcol_start = nullptr;
    int* last_row = nullptr;
    int* tok_pos = nullptr;
    int* tok_vcol = nullptr;
};

static VarlenCtx varlen_ctx(const Workspace& W, uint8_t* ws, int n_seq, const int* cu) {
    VarlenCtx V;
    if (n_seq <= 0) return V;
    V.n_seq = n_seq;
    V.cu = cu;
    V.tile_start = (int*)(ws + W.tile_start);
    V.vcol_start = (int*)(ws + W.vcol_start);
    V.last_row = (int*)(ws + W.last_row);
    V.tok_pos = (int*)(ws + W.tok_pos);
    V.tok_vcol = (int*)(ws + W.tok_vcol);
    return V;
}

static bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// KV state of a chunked prefill: per layer K (token-major), then V^T (bf16) or
// V (f32), each 256-byte aligned.
struct KvState {
    uint8_t* base = nullptr;    // nullptr: an ordinary (unchunked) pass
    int p0 = 0;
    long long ldvt = 0;         // bf16: V^T row stride (max_T rounded up to 8)
    size_t v_off = 0, layer_bytes = 0;
    uint8_t* k(int l) const { return base + (size_t)l * layer_bytes; }
    uint8_t* v(int l) const { return base + (size_t)l * layer_bytes + v_off; }
};

static KvState kv_state_layout(const dtp_config* c, int max_T) {
    KvState S;
    const size_t nk = (size_t)c->n_head_kv * c->head_dim;
    if (c->precision == DTP_PREC_BF16 || c->precision == DTP_PREC_E4M3 ||
        c->precision == DTP_PREC_TF32) {       // K, then V^T (what the tcgen05 attention reads)
        const size_t eb = c->precision == DTP_PREC_TF32 ? 4 : 2;
        S.ldvt = (long long)align_up((size_t)max_T, 8);
        S.v_off = align_up((size_t)max_T * nk * eb, 256);
        S.layer_bytes = S.v_off + align_up(nk * (size_t)S.ldvt * eb, 256);
    } else {
        S.v_off = align_up((size_t)max_T * nk * 4, 256);
        S.layer_bytes = 2 * S.v_off;
    }
    return S;
}

// ----------------------------------------------------------------------------- forward
static int fwd_f32(const dtp_config* c, const uint8_t* P, const PackedLayout& L,
                   const uint32_t* tokens, int T, const dtp_fwd_outputs& o, uint8_t* ws,
                   const Workspace& W, const VarlenCtx& V, const KvState& S, cudaStream_t s) {
    float* logits = o.logits;
    float* hidden = o.hidden;
    const int d = c->n_embd, hd = c->head_dim, h = c->n_head, g = c->n_head_kv, F = c->n_ff;
    const int nq = h * hd, nk = g * hd;
    const int nqc = nq * (1 + c->attn_gate);            // q region, with the gate rows
    const int nqkv = nqc + 2 * nk;
    const int qstride = c->attn_gate ? 2 * hd : hd;     // q head stride within the q region
    float* x = (float*)(ws + W.x);
    float* hb = (float*)(ws + W.h);
    float* qkv = (float*)(ws + W.qkv);
    float* attn = (float*)(ws + W.attn);
    float* gu = (float*)(ws + W.gu);
    float* act = (float*)(ws + W.act);
    const float scale = 1.0f / sqrtf((float)hd);
    // DTP_PREC_TF32: the GEMMs run on tcgen05 (kind::tf32) and each GEMM input is
    // rounded to tf32 by the kernel that writes it; otherwise the SIMT GEMM
    const bool tc = c->precision == DTP_PREC_TF32;
    const int opd = tc ? DTP_TF32 : DTP_F32;
    // the tcgen05 tf32 attention covers a single sequence (packed sequences and
    // chunks run the float32 SIMT attention on the same tf32 values)
    const bool tca = tc && !V.n_seq && attn_tc_supported(h, g, hd) && aligned(qkv, 16) &&
                     nqkv % 4 == 0 && nqc % 4 == 0;
    auto gemm = [&](const float* a, const float* w, float* y, int M, int N, int K,
                    const float* res, int kind) -> cudaError_t {
        if (!tc) return launch_gemm_simt(a, K, w, y, DTP_F32, N, M, N, K, res, s, kind);
        GemmEpiArgs e;
        e.y = y;
        e.y_dtype = DTP_F32;
        e.ldy = N;
        e.residual = res;
        return launch_gemm_tc_tf32(a, w, M, N, K, e, s, kind);
    };
    if (V.n_seq)
        DTP_CUDA_CHECK(launch_seq_meta(V.cu, V.n_seq, T, V.tile_start, V.vcol_start, V.last_row,
                                       V.tok_pos, V.tok_vcol, T, s));
    DTP_CUDA_CHECK(launch_embed(tokens, T, c->n_vocab, d, P + L.tok_embd, DTP_F32, x, s));
    for (int l = 0; l < c->n_layer; ++l) {
        const uint8_t* lp = P + (size_t)l * L.layer_bytes;
        if (hidden)
            DTP_CUDA_CHECK(launch_copy_f32(x, hidden + (size_t)l * T * d, (size_t)T * d, s));
        DTP_CUDA_CHECK(launch_rmsnorm(x, (const float*)(lp + L.attn_norm), hb, opd, T, d,
                                      c->rms_eps, s));
        DTP_CUDA_CHECK(gemm(hb, (const float*)(lp + L.w_qkv), qkv, T, nqkv, d, nullptr,
                            DTP_K_GEMM_QKV));
        // tf32 mode: q, k and v are rounded to tf32 here (the tensor-core
        // attention's operands); the other attention paths see the same values
        DTP_CUDA_CHECK(launch_qk_norm_rope(qkv, opd, nqkv, (const float*)(lp + L.q_norm),
                                           V.tok_pos, T, h, hd, c->rope_dim_count,
                                           c->rope_freq_base, c->rms_eps, s, qstride, S.p0));
        DTP_CUDA_CHECK(launch_qk_norm_rope(qkv + nqc, opd, nqkv, (const float*)(lp + L.k_norm),
                                           V.tok_pos, T, g, hd, c->rope_dim_count,
                                           c->rope_freq_base, c->rms_eps, s, 0, S.p0));
        if (tc) DTP_CUDA_CHECK(launch_round_tf32_rows(qkv + nqc + nk, nqkv, T, nk, s));
        if (o.k_cache)
            DTP_CUDA_CHECK(launch_copy_rows_f32(qkv + nqc, nqkv,
                                                (float*)o.k_cache + (size_t)l * T * nk, nk, T, nk, s));
        if (o.v_cache)
            DTP_CUDA_CHECK(launch_copy_rows_f32(qkv + nqc + nk, nqkv,
                                                (float*)o.v_cache + (size_t)l * T * nk, nk, T, nk, s));
        if (S.base && tca) {    // chunked, tf32: K rows and V^T columns at p0, tcgen05 attention
            float* ks = (float*)S.k(l);
            float* vts = (float*)S.v(l);
            DTP_CUDA_CHECK(launch_copy_rows_f32(qkv + nqc, nqkv, ks + (size_t)S.p0 * nk, nk, T,
                                                nk, s));
            DTP_CUDA_CHECK(launch_transpose_v_f32(qkv + nqc + nk, nqkv, vts + S.p0, T, nk,
                                                  (int)S.ldvt, s));
            AttnVarlen vl;
            vl.p0 = S.p0;
            DTP_CUDA_CHECK(launch_attn_tc_f32(qkv, nqkv, qstride, ks, nk, vts, S.ldvt, S.p0 + T,
                                              attn, T, h, g, hd, scale, vl, s));
        } else if (S.base) {    // chunked: append this chunk's keys and values to the state
            float* ks = (float*)S.k(l);
            float* vs = (float*)S.v(l);
            DTP_CUDA_CHECK(launch_copy_rows_f32(qkv + nqc, nqkv, ks + (size_t)S.p0 * nk, nk, T,
                                                nk, s));
            DTP_CUDA_CHECK(launch_copy_rows_f32(qkv + nqc + nk, nqkv, vs + (size_t)S.p0 * nk, nk,
                                                T, nk, s));
            DTP_CUDA_CHECK(launch_attn_simt(qkv, nqkv, ks, nk, vs, nk, 0, attn, nq, DTP_F32, T, h,
                                            g, hd, scale, s, nullptr, qstride, S.p0));
        } else if (tca) {
            // one sequence: the tcgen05 attention on tf32 q / k / v^T
            float* vt = (float*)(ws + W.vt);
            DTP_CUDA_CHECK(launch_transpose_v_f32(qkv + nqc + nk, nqkv, vt, T, nk, (int)W.ldvt, s));
            AttnVarlen none;
            DTP_CUDA_CHECK(launch_attn_tc_f32(qkv, nqkv, qstride, qkv + nqc, nqkv, vt, W.ldvt, T,
                                              attn, T, h, g, hd, scale, none, s));
        } else {
            DTP_CUDA_CHECK(launch_attn_simt(qkv, nqkv, qkv + nqc, nqkv, qkv + nqc + nk, nqkv, 0,
                                            attn, nq, DTP_F32, T, h, g, hd, scale, s, V.tok_pos,
                                            qstride));
        }
        if (c->attn_gate)
            DTP_CUDA_CHECK(launch_gate_mul_f32(attn, nq, qkv + hd, nqkv, 2 * hd, T, h, hd, s));
        if (tc) DTP_CUDA_CHECK(launch_round_tf32(attn, (size_t)T * nq, s));
        DTP_CUDA_CHECK(gemm(attn, (const float*)(lp + L.wo), x, T, d, nq, x, DTP_K_GEMM_O));
        DTP_CUDA_CHECK(launch_rmsnorm(x, (const float*)(lp + L.ffn_norm), hb, opd, T, d,
                                      c->rms_eps, s));
        DTP_CUDA_CHECK(gemm(hb, (const float*)(lp + L.w_gu), gu, T, 2 * F, d, nullptr,
                            DTP_K_GEMM_GATEUP));
        DTP_CUDA_CHECK(launch_swiglu_interleaved64(gu, act, T, F, s, opd));
        DTP_CUDA_CHECK(gemm(act, (const float*)(lp + L.w_down), x, T, d, F, x, DTP_K_GEMM_DOWN));
    }
    if (hidden)
        DTP_CUDA_CHECK(
            launch_copy_f32(x, hidden + (size_t)c->n_layer * T * d, (size_t)T * d, s));
    if (!logits) return DTP_OK;
    if (o.last_only && V.n_seq) {            // the last position of every sequence
        DTP_CUDA_CHECK(launch_rmsnorm(x, (const float*)(P + L.output_norm), hb, opd, V.n_seq,
                                      d, c->rms_eps, s, V.last_row));
        DTP_CUDA_CHECK(gemm(hb, (const float*)(P + L.output), logits, V.n_seq, c->n_vocab, d,
                            nullptr, DTP_K_GEMM_LMHEAD));
        return DTP_OK;
    }
    const int rows = o.last_only ? 1 : T;
    const float* xf = x + (size_t)(T - rows) * d;
    DTP_CUDA_CHECK(launch_rmsnorm(xf, (const float*)(P + L.output_norm), hb, opd, rows, d,
                                  c->rms_eps, s));
    DTP_CUDA_CHECK(gemm(hb, (const float*)(P + L.output), logits, rows, c->n_vocab, d, nullptr,
                        DTP_K_GEMM_LMHEAD));
    return DTP_OK;
}

static int fwd_bf16(const dtp_config* c, const uint8_t* P, const PackedLayout& L,
                    const uint32_t* tokens, int T, const dtp_fwd_outputs& o, uint8_t* ws,
                    const Workspace& W, const VarlenCtx& V, const KvState& S, cudaStream_t s) {
    float* logits = o.logits;
    float* hidden = o.hidden;
    typedef __nv_bfloat16 bf;
    const int d = c->n_embd, hd = c->head_dim, h = c->n_head, g = c->n_head_kv, F = c->n_ff;
    const int nq = h * hd, nk = g * hd, nqkv = nq * (1 + c->attn_gate) + 2 * nk;
    float* x = (float*)(ws + W.x);
    bf* hb = (bf*)(ws + W.h);
    bf* gate = c->attn_gate ? (bf*)(ws + W.gate) : nullptr;
    bf* q = (bf*)(ws + W.q);
    bf* k = (bf*)(ws + W.k);
    __half* vt = (__half*)(ws + W.vt);      // f16 copies of bf16(v), key index contiguous
    bf* attn = (bf*)(ws + W.attn);
    bf* act = (bf*)(ws + W.act);
    float2* rope = (float2*)(ws + W.rope);
    const float scale = 1.0f / sqrtf((float)hd);
    const bool fa = attn_tc_supported(h, g, hd);
    // DTP_PREC_E4M3: every GEMM input is quantised per row to e4m3 (q8, scales s8)
    // and every weight is e4m3 with per-row scales; attention stays bf16
    const bool e4 = c->precision == DTP_PREC_E4M3;
    uint8_t* q8 = e4 ? ws + W.q8 : nullptr;
    float* s8 = e4 ? (float*)(ws + W.s8) : nullptr;
    // the GEMM A operand: bf16 `a`, or its e4m3 codes in q8 (b_scale: the weight's
    // row scales)
    auto gemm = [&](const bf* a, const uint8_t* w, const float* w_scale, int M, int N, int K,
                    GemmEpi epi, GemmEpiArgs e, int kind) -> cudaError_t {
        if (!e4) return launch_gemm_tc(a, (const bf*)w, M, N, K, epi, e, s, kind);
        e.a_scale = s8;
        e.b_scale = w_scale;
        return launch_gemm_tc_e4m3(q8, w, M, N, K, epi, e, s, kind);
    };
    // RMSNorm straight to the next GEMM's operand (bf16 h, or e4m3 codes + scales)
    auto norm = [&](const float* xin, const float* w, int rows, const int* row_idx) {
        if (e4) return launch_rmsnorm_e4m3(xin, w, q8, s8, rows, d, c->rms_eps, s, row_idx);
        return launch_rmsnorm(xin, w, hb, DTP_BF16, rows, d, c->rms_eps, s, row_idx);
    };
    // packed sequences: v^T blocks start on 8-column boundaries; the padding
    // columns between them are read by attention (with P = 0), so they are zeroed
    long long vt_cols = T;
    AttnVarlen vl;
    vl.gate = gate;
    if (V.n_seq) {
        vt_cols = W.ldvt;
        DTP_CUDA_CHECK(cudaMemsetAsync(vt, 0, (size_t)nk * W.ldvt * 2, s));
        DTP_CUDA_CHECK(launch_seq_meta(V.cu, V.n_seq, T, V.tile_start, V.vcol_start, V.last_row,
                                       V.tok_pos, V.tok_vcol, vt_cols, s));
        vl.n_seq = V.n_seq;
        vl.cu_seqlens = V.cu;
        vl.tile_start = V.tile_start;
        vl.vcol_start = V.vcol_start;
    }
    long long ldvt = W.ldvt;
    if (S.base) {               // chunked: keys 0 .. p0+T-1 of the state
        vl.p0 = S.p0;
        vt_cols = S.p0 + T;
        ldvt = S.ldvt;
    }
    // row t of the table holds position p0 + t
    DTP_CUDA_CHECK(launch_rope_table(rope, T, c->rope_dim_count, c->rope_freq_base, s, S.p0));
    // bf16: the RMSNorm before the QKV and gate/up GEMMs is fused (GemmEpiArgs,
    // "RMSNorm fused across GEMMs"): whoever writes x -- the embedding, the O and
    // down epilogues -- also writes hb = bf16(x) and per-tile row sums of x^2 into
    // ssp; the next GEMM multiplies its rows by 1/rms, the norm weight being folded
    // into its packed matrix.  e4m3 mode keeps the RMSNorm kernel (its codes need
    // the normalised row's max).
    const bool fused = !e4;
    float* ssp = fused ? (float*)(ws + W.ssp) : nullptr;
    int n_ss = 1;                                    // partials per row in ssp
    auto norm_args = [&](GemmEpiArgs& a) {
        a.ss_in = ssp;
        a.n_ss = n_ss;
        a.ld_ss = T;
        a.norm_cols = d;
        a.norm_eps = c->rms_eps;
    };
    auto norm_out = [&](GemmEpiArgs& a) {
        a.xb = hb;
        a.ss_out = ssp;
        a.ld_ss = T;
    };
    DTP_CUDA_CHECK(launch_embed(tokens, T, c->n_vocab, d, P + L.tok_embd, DTP_BF16, x, s,
                                fused ? hb : nullptr, ssp));
    for (int l = 0; l < c->n_layer; ++l) {
        const uint8_t* lp = P + (size_t)l * L.layer_bytes;
        if (hidden)
            DTP_CUDA_CHECK(launch_copy_f32(x, hidden + (size_t)l * T * d, (size_t)T * d, s));
        if (!fused) DTP_CUDA_CHECK(norm(x, (const float*)(lp + L.attn_norm), T, nullptr));
        GemmEpiArgs e;
        if (fused) norm_args(e);
        // with a KV cache the keys are written straight into it (attention reads them
        // there); a chunk writes its keys and values into the state at position p0
        bf* kl = o.k_cache ? (bf*)o.k_cache + (size_t)l * T * nk : k;
        __half* vtl = vt;
        if (S.base) {
            kl = (bf*)S.k(l);
            vtl = (__half*)S.v(l);
        }
        e.q = q;
        e.k = kl + (size_t)S.p0 * nk;
        e.vt = vtl + S.p0;
        e.ldvt = ldvt;
        e.v_rows = o.v_cache ? (bf*)o.v_cache + (size_t)l * T * nk : nullptr;
        e.tok_pos = V.tok_pos;
        e.tok_vcol = V.tok_vcol;
        e.q_gated = c->attn_gate;
        e.gate = gate;
        e.q_norm = (const float*)(lp + L.q_norm);
        e.k_norm = (const float*)(lp + L.k_norm);
        e.rope = rope;
        e.n_head = h;
        e.n_head_kv = g;
        e.head_dim = hd;
        e.rope_dims = c->rope_dim_count;
        e.eps = c->rms_eps;
        DTP_CUDA_CHECK(gemm(hb, lp + L.w_qkv, (const float*)(lp + L.w_qkv_s), T, nqkv, d, EPI_QKV,
                            e, DTP_K_GEMM_QKV));
        if (fa)
            DTP_CUDA_CHECK(launch_attn_tc_varlen(q, kl, vtl, ldvt, vt_cols, attn, T, h, g, hd,
                                                 scale, vl, s));
        else
            return fail(DTP_ERR_UNSUPPORTED,
                        "bf16 path: attention needs an even n_head/n_head_kv group");
        GemmEpiArgs eo;
        eo.y = x;
        eo.y_dtype = DTP_F32;
        eo.ldy = d;
        eo.residual = x;
        if (fused) norm_out(eo);
        if (e4) DTP_CUDA_CHECK(launch_quant_rows_e4m3(attn, nq, T, nq, q8, s8, s));
        DTP_CUDA_CHECK(gemm(attn, lp + L.wo, (const float*)(lp + L.wo_s), T, d, nq, EPI_STORE, eo,
                            DTP_K_GEMM_O));
        n_ss = gemm_tc_tiles_n(T, d);
        if (!fused) DTP_CUDA_CHECK(norm(x, (const float*)(lp + L.ffn_norm), T, nullptr));
        GemmEpiArgs eg;
        eg.act = act;
        if (fused) norm_args(eg);
        DTP_CUDA_CHECK(gemm(hb, lp + L.w_gu, (const float*)(lp + L.w_gu_s), T, 2 * F, d, EPI_SWIGLU,
                            eg, DTP_K_GEMM_GATEUP));
        if (e4) DTP_CUDA_CHECK(launch_quant_rows_e4m3(act, F, T, F, q8, s8, s));
        DTP_CUDA_CHECK(gemm(act, lp + L.w_down, (const float*)(lp + L.w_down_s), T, d, F, EPI_STORE,
                            eo, DTP_K_GEMM_DOWN));
        n_ss = gemm_tc_tiles_n(T, d);
    }
    if (hidden)
        DTP_CUDA_CHECK(
            launch_copy_f32(x, hidden + (size_t)c->n_layer * T * d, (size_t)T * d, s));
    if (!logits) return DTP_OK;
    // forward.rs `forward_last`: only the last position's logits (of every sequence)
    int rows = o.last_only ? 1 : T;
    if (o.last_only && V.n_seq) {
        rows = V.n_seq;
        DTP_CUDA_CHECK(norm(x, (const float*)(P + L.output_norm), rows, V.last_row));
    } else {
        DTP_CUDA_CHECK(norm(x + (size_t)(T - rows) * d, (const float*)(P + L.output_norm), rows,
                            nullptr));
    }
    GemmEpiArgs el;
    el.y = logits;
    el.y_dtype = DTP_F32;
    el.ldy = c->n_vocab;
    DTP_CUDA_CHECK(gemm(hb, P + L.output, (const float*)(P + L.output_s), rows, c->n_vocab, d,
                        EPI_STORE, el, DTP_K_GEMM_LMHEAD));
    return DTP_OK;
}

}  // namespace dtp

using namespace dtp;

// ================================================================================ C ABI
extern "C" {

const char* dtp_last_error(void) { return t_err; }

long long dtp_launch_count(int reset) {
    return reset ? g_launches.exchange(0) : g_launches.load();
}

size_t dtp_packed_size(const dtp_config* cfg) {
    if (validate_config(cfg) != DTP_OK) return 0;
    return packed_layout(cfg).total;
}

int dtp_pack_layer(const dtp_config* cfg, int layer, const dtp_layer_src* src, void* packed,
                   size_t packed_bytes, dtp_stream_t stream) {
    int rc = validate_config(cfg);
    if (rc) return rc;
    if (!src || !packed) return fail(DTP_ERR_INVALID_ARG, "NULL src or packed");
    if (layer < 0 || layer >= cfg->n_layer)
        return fail(DTP_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, cfg->n_layer);
    const float* ptrs[] = {src->attn_norm, src->wq, src->wk, src->wv, src->q_norm, src->k_norm,
                           src->wo, src->ffn_norm, src->w_gate, src->w_up, src->w_down};
    for (const float* p : ptrs)
        if (!p) return fail(DTP_ERR_INVALID_ARG, "a layer source pointer is NULL");
    PackedLayout L = packed_layout(cfg);
    if (packed_bytes < L.total)
        return fail(DTP_ERR_WORKSPACE, "packed buffer %zu < %zu bytes", packed_bytes, L.total);
    if (!aligned(packed, 256)) return fail(DTP_ERR_INVALID_ARG, "packed must be 256-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    uint8_t* lp = (uint8_t*)packed + (size_t)layer * L.layer_bytes;
    // matrix storage type: bf16, float32, or float32 rounded to tf32
    const int bf = cfg->precision == DTP_PREC_BF16   ? DTP_BF16
                   : cfg->precision == DTP_PREC_TF32 ? DTP_TF32
                                                     : DTP_F32;
    const int d = cfg->n_embd, hd = cfg->head_dim, nq = cfg->n_head * hd,
              nk = cfg->n_head_kv * hd, F = cfg->n_ff;
    const int nqc = nq * (1 + cfg->attn_gate);      // q rows (with the per-head gate rows)
    if (cfg->precision == DTP_PREC_E4M3) {
        // e4m3 codes with one float32 scale per row; same row order as below
        uint8_t* qkv = lp + L.w_qkv;
        float* qkv_s = (float*)(lp + L.w_qkv_s);
        DTP_CUDA_CHECK(launch_pack_e4m3(src->wq, nqc, d, qkv, qkv_s, 0, s));
        DTP_CUDA_CHECK(launch_pack_e4m3(src->wk, nk, d, qkv + (size_t)nqc * d, qkv_s + nqc, 0, s));
        DTP_CUDA_CHECK(launch_pack_e4m3(src->wv, nk, d, qkv + (size_t)(nqc + nk) * d,
                                        qkv_s + nqc + nk, 0, s));
        DTP_CUDA_CHECK(launch_pack_e4m3(src->wo, d, nq, lp + L.wo, (float*)(lp + L.wo_s), 0, s));
        DTP_CUDA_CHECK(launch_pack_e4m3(src->w_gate, F, d, lp + L.w_gu, (float*)(lp + L.w_gu_s),
                                        1, s));
        DTP_CUDA_CHECK(launch_pack_e4m3(src->w_up, F, d, lp + L.w_gu, (float*)(lp + L.w_gu_s), 2,
                                        s));
        DTP_CUDA_CHECK(launch_pack_e4m3(src->w_down, d, F, lp + L.w_down,
                                        (float*)(lp + L.w_down_s), 0, s));
    } else {
    // bf16: the RMSNorm that precedes the QKV and gate/up GEMMs is fused into them
    // (its weight multiplies the matrix's columns here, its 1/rms scales the
    // GEMM's rows in the epilogue)
    const float* an = bf == DTP_BF16 ? src->attn_norm : nullptr;
    const float* fn = bf == DTP_BF16 ? src->ffn_norm : nullptr;
    DTP_CUDA_CHECK(launch_pack_matrix(src->wq, nqc, d, lp + L.w_qkv, bf, 0, s, an));
    DTP_CUDA_CHECK(launch_pack_matrix(src->wk, nk, d, lp + L.w_qkv + (size_t)nqc * d * L.elt, bf, 0,
                                      s, an));
    DTP_CUDA_CHECK(launch_pack_matrix(src->wv, nk, d, lp + L.w_qkv + (size_t)(nqc + nk) * d * L.elt,
                                      bf, 0, s, an));
    DTP_CUDA_CHECK(launch_pack_matrix(src->wo, d, nq, lp + L.wo, bf, 0, s));
    DTP_CUDA_CHECK(launch_pack_matrix(src->w_gate, F, d, lp + L.w_gu, bf, 1, s, fn));
    DTP_CUDA_CHECK(launch_pack_matrix(src->w_up, F, d, lp + L.w_gu, bf, 2, s, fn));
    DTP_CUDA_CHECK(launch_pack_matrix(src->w_down, d, F, lp + L.w_down, bf, 0, s));
    }
    DTP_CUDA_CHECK(launch_pack_matrix(src->attn_norm, 1, d, lp + L.attn_norm, 0, 0, s));
    DTP_CUDA_CHECK(launch_pack_matrix(src->q_norm, 1, hd, lp + L.q_norm, 0, 0, s));
    DTP_CUDA_CHECK(launch_pack_matrix(src->k_norm, 1, hd, lp + L.k_norm, 0, 0, s));
    DTP_CUDA_CHECK(launch_pack_matrix(src->ffn_norm, 1, d, lp + L.ffn_norm, 0, 0, s));
    return DTP_OK;
}

int dtp_pack_globals(const dtp_config* cfg, const float* tok_embd, const float* output_norm,
                     const float* output, void* packed, size_t packed_bytes,
                     dtp_stream_t stream) {
    int rc = validate_config(cfg);
    if (rc) return rc;
    if (!tok_embd || !output_norm || !output || !packed)
        return fail(DTP_ERR_INVALID_ARG, "NULL pointer");
    PackedLayout L = packed_layout(cfg);
    if (packed_bytes < L.total)
        return fail(DTP_ERR_WORKSPACE, "packed buffer %zu < %zu bytes", packed_bytes, L.total);
    if (!aligned(packed, 256)) return fail(DTP_ERR_INVALID_ARG, "packed must be 256-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    uint8_t* P = (uint8_t*)packed;
    const bool e4 = cfg->precision == DTP_PREC_E4M3;
    const int bf = (cfg->precision == DTP_PREC_BF16 || e4) ? DTP_BF16 : DTP_F32;
    const int mat = cfg->precision == DTP_PREC_TF32 ? DTP_TF32 : bf;    // tok_embd is no GEMM operand
    DTP_CUDA_CHECK(launch_pack_matrix(tok_embd, cfg->n_vocab, cfg->n_embd, P + L.tok_embd, bf, 0, s));
    if (e4)
        DTP_CUDA_CHECK(launch_pack_e4m3(output, cfg->n_vocab, cfg->n_embd, P + L.output,
                                        (float*)(P + L.output_s), 0, s));
    else
        DTP_CUDA_CHECK(launch_pack_matrix(output, cfg->n_vocab, cfg->n_embd, P + L.output, mat, 0, s));
    DTP_CUDA_CHECK(launch_pack_matrix(output_norm, 1, cfg->n_embd, P + L.output_norm, 0, 0, s));
    return DTP_OK;
}

size_t dtp_workspace_size(const dtp_config* cfg, int T) {
    if (validate_config(cfg) != DTP_OK || T <= 0) return 0;
    return workspace_layout(cfg, T, false).total;
}

size_t dtp_workspace_size_host(const dtp_config* cfg, int T) {
    if (validate_config(cfg) != DTP_OK || T <= 0) return 0;
    return workspace_layout(cfg, T, true).total;
}

static int fwd_checked(const dtp_config* cfg, const void* packed, size_t packed_bytes,
                       const uint32_t* tokens, int T, const dtp_fwd_outputs& out,
                       void* workspace, size_t ws_bytes, bool host_layout, dtp_stream_t stream,
                       int n_seq = 0, const int* cu_seqlens = nullptr,
                       const KvState& S = KvState()) {
    float* logits = out.logits;
    float* hidden = out.hidden;
    int rc = validate_config(cfg);
    if (rc) return rc;
    if (T <= 0) return fail(DTP_ERR_INVALID_ARG, "T must be >= 1 (got %d)", T);
    if (!packed || !tokens || !workspace)
        return fail(DTP_ERR_INVALID_ARG, "NULL packed, tokens or workspace");
    // (a chunk may only extend its KV state)
    if (!S.base && !logits && !hidden && !out.k_cache && !out.v_cache)
        return fail(DTP_ERR_INVALID_ARG, "no output requested");
    PackedLayout L = packed_layout(cfg);
    if (packed_bytes < L.total)
        return fail(DTP_ERR_WORKSPACE, "packed buffer %zu < %zu bytes", packed_bytes, L.total);
    Workspace W = workspace_layout(cfg, T, host_layout, n_seq);
    if (ws_bytes < W.total)
        return fail(DTP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, W.total);
    const bool tc_path = cfg->precision == DTP_PREC_BF16 || cfg->precision == DTP_PREC_E4M3;
    if (tc_path && !attn_tc_supported(cfg->n_head, cfg->n_head_kv, cfg->head_dim))
        return fail(DTP_ERR_UNSUPPORTED, "bf16 path: n_head / n_head_kv must be even");
    if (!aligned(workspace, 256) || !aligned(packed, 256) || (logits && !aligned(logits, 16)) ||
        (hidden && !aligned(hidden, 16)) || (out.k_cache && !aligned(out.k_cache, 16)) ||
        (out.v_cache && !aligned(out.v_cache, 16)))
        return fail(DTP_ERR_INVALID_ARG,
                    "workspace/packed must be 256-byte aligned, outputs 16-byte aligned");
    if (tc_path && (cfg->n_vocab % 4))
        return fail(DTP_ERR_UNSUPPORTED, "bf16 path: n_vocab must be a multiple of 4");
    cudaStream_t s = (cudaStream_t)stream;
    const VarlenCtx V = varlen_ctx(W, (uint8_t*)workspace, n_seq, cu_seqlens);
    if (tc_path)
        return fwd_bf16(cfg, (const uint8_t*)packed, L, tokens, T, out, (uint8_t*)workspace, W, V,
                        S, s);
    return fwd_f32(cfg, (const uint8_t*)packed, L, tokens, T, out, (uint8_t*)workspace, W, V, S,
                   s);
}

int dtp_fwd_prefill(const dtp_config* cfg, const void* packed, size_t packed_bytes,
                    const uint32_t* tokens, int T, float* logits, float* hidden, void* workspace,
                    size_t ws_bytes, dtp_stream_t stream) {
    if (!logits) return fail(DTP_ERR_INVALID_ARG, "NULL logits");
    dtp_fwd_outputs o = {};
    o.logits = logits;
    o.hidden = hidden;
    return fwd_checked(cfg, packed, packed_bytes, tokens, T, o, workspace, ws_bytes, false, stream);
}

int dtp_fwd_prefill_ex(const dtp_config* cfg, const void* packed, size_t packed_bytes,
                       const uint32_t* tokens, int T, const dtp_fwd_outputs* out, void* workspace,
                       size_t ws_bytes, dtp_stream_t stream) {
    if (!out) return fail(DTP_ERR_INVALID_ARG, "NULL outputs");
    return fwd_checked(cfg, packed, packed_bytes, tokens, T, *out, workspace, ws_bytes, false,
                       stream);
}

size_t dtp_workspace_size_varlen(const dtp_config* cfg, int total, int n_seq) {
    if (validate_config(cfg) != DTP_OK || total <= 0 || n_seq <= 0) return 0;
    return workspace_layout(cfg, total, false, n_seq).total;
}

int dtp_fwd_prefill_varlen(const dtp_config* cfg, const void* packed, size_t packed_bytes,
                           const uint32_t* tokens, const int32_t* cu_seqlens, int n_seq, int total,
                           const dtp_fwd_outputs* out, void* workspace, size_t ws_bytes,
                           dtp_stream_t stream) {
    if (!out) return fail(DTP_ERR_INVALID_ARG, "NULL outputs");
    if (!cu_seqlens || n_seq <= 0)
        return fail(DTP_ERR_INVALID_ARG, "cu_seqlens must be given with n_seq >= 1");
    if (n_seq > (1 << 20)) return fail(DTP_ERR_UNSUPPORTED, "n_seq > 2^20");
    return fwd_checked(cfg, packed, packed_bytes, tokens, total, *out, workspace, ws_bytes, false,
                       stream, n_seq, cu_seqlens);
}

size_t dtp_kv_state_size(const dtp_config* cfg, int max_T) {
    if (validate_config(cfg) != DTP_OK || max_T <= 0) return 0;
    return kv_state_layout(cfg, max_T).layer_bytes * (size_t)cfg->n_layer;
}

int dtp_fwd_prefill_chunk(const dtp_config* cfg, const void* packed, size_t packed_bytes,
                          const uint32_t* tokens, int C, int p0, void* kv_state,
                          size_t state_bytes, int max_T, const dtp_fwd_outputs* out,
                          void* workspace, size_t ws_bytes, dtp_stream_t stream) {
    int rc = validate_config(cfg);
    if (rc) return rc;
    if (!out) return fail(DTP_ERR_INVALID_ARG, "NULL outputs");
    if (!kv_state) return fail(DTP_ERR_INVALID_ARG, "NULL kv_state");
    if (out->k_cache || out->v_cache)
        return fail(DTP_ERR_INVALID_ARG, "chunked prefill: k_cache/v_cache must be NULL");
    if (C <= 0 || p0 < 0 || max_T <= 0 || (long long)p0 + C > max_T)
        return fail(DTP_ERR_INVALID_ARG, "chunk [%d, %d + %d) outside 0..max_T = %d", p0, p0, C,
                    max_T);
    if (!aligned(kv_state, 256)) return fail(DTP_ERR_INVALID_ARG, "kv_state must be 256-byte aligned");
    KvState S = kv_state_layout(cfg, max_T);
    const size_t need = S.layer_bytes * (size_t)cfg->n_layer;
    if (state_bytes < need)
        return fail(DTP_ERR_WORKSPACE, "kv_state %zu < %zu bytes", state_bytes, need);
    S.base = (uint8_t*)kv_state;
    S.p0 = p0;
    return fwd_checked(cfg, packed, packed_bytes, tokens, C, *out, workspace, ws_bytes, false,
                       stream, 0, nullptr, S);
}

int dtp_fwd_prefill_host(const dtp_config* cfg, const void* packed, size_t packed_bytes,
                         const uint32_t* tokens_host, int T, float* logits_host, void* workspace,
                         size_t ws_bytes, dtp_stream_t stream) {
    int rc = validate_config(cfg);
    if (rc) return rc;
    if (T <= 0) return fail(DTP_ERR_INVALID_ARG, "T must be >= 1 (got %d)", T);
    if (!tokens_host || !logits_host || !workspace)
        return fail(DTP_ERR_INVALID_ARG, "NULL tokens_host, logits_host or workspace");
    for (int t = 0; t < T; ++t)
        if (tokens_host[t] >= (uint32_t)cfg->n_vocab)
            return fail(DTP_ERR_TOKEN_RANGE, "token %u at position %d >= n_vocab %d",
                        tokens_host[t], t, cfg->n_vocab);
    Workspace W = workspace_layout(cfg, T, true);
    if (ws_bytes < W.total)
        return fail(DTP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, W.total);
    if (!aligned(workspace, 256)) return fail(DTP_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    uint8_t* ws = (uint8_t*)workspace;
    uint32_t* tok_d = (uint32_t*)(ws + W.tokens);
    float* logit_d = (float*)(ws + W.logits);
    DTP_CUDA_CHECK(cudaMemcpyAsync(tok_d, tokens_host, (size_t)T * 4, cudaMemcpyHostToDevice, s));
    dtp_fwd_outputs o = {};
    o.logits = logit_d;
    rc = fwd_checked(cfg, packed, packed_bytes, tok_d, T, o, workspace, ws_bytes, true, stream);
    if (rc) return rc;
    DTP_CUDA_CHECK(cudaMemcpyAsync(logits_host, logit_d, (size_t)T * cfg->n_vocab * 4,
                                   cudaMemcpyDeviceToHost, s));
    return DTP_OK;
}

size_t dtp_workspace_size_host_batch_n(const dtp_config* cfg, int T, int n_buffers) {
    if (validate_config(cfg) != DTP_OK || T <= 0 || n_buffers < kMinBatchBuffers ||
        n_buffers > kMaxBatchBuffers)
        return 0;
    return workspace_layout(cfg, T, true, 0, n_buffers).total;
}

size_t dtp_workspace_size_host_batch(const dtp_config* cfg, int T) {
    return dtp_workspace_size_host_batch_n(cfg, T, kMinBatchBuffers);
}

// The library's device-to-host copy stream of the current device (created once).
static cudaStream_t copy_stream() {
    static std::mutex mu;
    static cudaStream_t streams[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!streams[dev] && cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking) != cudaSuccess)
        streams[dev] = nullptr;
    return streams[dev];
}

int dtp_fwd_prefill_host_batch(const dtp_config* cfg, const void* packed, size_t packed_bytes,
                               const uint32_t* const* tokens_host, int n, int T,
                               float* const* logits_host, void* workspace, size_t ws_bytes,
                               dtp_stream_t stream) {
    int rc = validate_config(cfg);
    if (rc) return rc;
    if (n <= 0 || T <= 0) return fail(DTP_ERR_INVALID_ARG, "n and T must be >= 1");
    if (!tokens_host || !logits_host || !workspace)
        return fail(DTP_ERR_INVALID_ARG, "NULL tokens_host, logits_host or workspace");
    for (int j = 0; j < n; ++j) {
        if (!tokens_host[j] || !logits_host[j])
            return fail(DTP_ERR_INVALID_ARG, "NULL host buffer for prompt %d", j);
        for (int t = 0; t < T; ++t)
            if (tokens_host[j][t] >= (uint32_t)cfg->n_vocab)
                return fail(DTP_ERR_TOKEN_RANGE, "prompt %d: token %u at position %d >= n_vocab %d",
                            j, tokens_host[j][t], t, cfg->n_vocab);
    }
    // as many logit buffers as the workspace holds
    int nb = kMinBatchBuffers;
    Workspace W = workspace_layout(cfg, T, true, 0, nb);
    if (ws_bytes < W.total)
        return fail(DTP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, W.total);
    while (nb < kMaxBatchBuffers) {
        const Workspace W2 = workspace_layout(cfg, T, true, 0, nb + 1);
        if (W2.total > ws_bytes) break;
        W = W2;
        ++nb;
    }
    if (!aligned(workspace, 256)) return fail(DTP_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    cudaStream_t k = copy_stream();
    if (!k) return fail(DTP_ERR_CUDA, "could not create the copy stream");
    uint8_t* ws = (uint8_t*)workspace;
    uint32_t* tok_d = (uint32_t*)(ws + W.tokens);
    const size_t lbytes = (size_t)T * cfg->n_vocab * 4;
    float* buf[kMaxBatchBuffers];
    buf[0] = (float*)(ws + W.logits);
    for (int b = 1; b < nb; ++b) buf[b] = (float*)(ws + W.logits_more + (b - 1) * lbytes);
    // ready[j]: prompt j's logits are on the device; copied[b]: buffer b is free again
    std::vector<cudaEvent_t> ev;
    auto new_event = [&](cudaEvent_t* e) {
        if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return false;
        ev.push_back(*e);
        return true;
    };
    cudaEvent_t copied[kMaxBatchBuffers] = {};
    rc = DTP_OK;
    for (int j = 0; j < n && rc == DTP_OK; ++j) {
        const int b = j % nb;
        cudaError_t e = cudaSuccess;
        if (copied[b]) e = cudaStreamWaitEvent(s, copied[b], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(tok_d, tokens_host[j], (size_t)T * 4, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) {
            rc = fail(DTP_ERR_CUDA, "%s", cudaGetErrorString(e));
            break;
        }
        dtp_fwd_outputs o = {};
        o.logits = buf[b];
        {
            LaunchScope span(DTP_K_PROMPT, s, false);
            rc = fwd_checked(cfg, packed, packed_bytes, tok_d, T, o, workspace, ws_bytes, true,
                             stream);
        }
        if (rc) break;
        cudaEvent_t ready, done;
        if (!new_event(&ready) || !new_event(&done)) {
            rc = fail(DTP_ERR_CUDA, "cudaEventCreate failed");
            break;
        }
        // the copy of prompt j overlaps the forward of prompt j + 1
        if ((e = cudaEventRecord(ready, s)) == cudaSuccess &&
            (e = cudaStreamWaitEvent(k, ready, 0)) == cudaSuccess) {
            LaunchScope span(DTP_K_D2H, k, false);
            e = cudaMemcpyAsync(logits_host[j], buf[b], lbytes, cudaMemcpyDeviceToHost, k);
        }
        if (e == cudaSuccess) e = cudaEventRecord(done, k);
        if (e != cudaSuccess) {
            rc = fail(DTP_ERR_CUDA, "%s", cudaGetErrorString(e));
            break;
        }
        copied[b] = done;
    }
    // `stream` completes only after every copy has landed
    for (int b = 0; b < nb; ++b)
        if (copied[b]) cudaStreamWaitEvent(s, copied[b], 0);
    for (cudaEvent_t e : ev) cudaEventDestroy(e);      // released once they complete
    return rc;
}

int dtp_check(dtp_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return fail(DTP_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
    unsigned bits = read_clear_simt_errors() | read_clear_gemm_errors() | read_clear_attn_errors();
    if (bits & ERRBIT_TIMEOUT)
        return fail(DTP_ERR_DEVICE_TIMEOUT, "a kernel's bounded pipeline wait gave up");
    if (bits & ERRBIT_VRANGE)
        return fail(DTP_ERR_VALUE_RANGE,
                    "a value v entering bf16 attention was beyond the f16 range (|v| > 65504) "
                    "or not finite");
    if (bits & ERRBIT_SEQLENS)
        return fail(DTP_ERR_INVALID_ARG,
                    "cu_seqlens was not 0 = cu[0] <= cu[1] <= ... <= cu[n_seq] = total (no "
                    "attention was computed)");
    if (bits & ERRBIT_TOKEN_RANGE)
        return fail(DTP_ERR_TOKEN_RANGE, "a token id was >= n_vocab (its row was zeroed)");
    return DTP_OK;
}

// ------------------------------------------------------------------------- per-op entry points
int dtp_rms_norm(const float* x, const float* w, void* y, int y_dtype, int rows, int cols,
                 float eps, dtp_stream_t stream) {
    if (!x || !w || !y) return fail(DTP_ERR_INVALID_ARG, "NULL pointer");
    if (rows <= 0 || cols <= 0) return fail(DTP_ERR_INVALID_ARG, "rows and cols must be >= 1");
    if (y_dtype != DTP_F32 && y_dtype != DTP_BF16 && y_dtype != DTP_TF32)
        return fail(DTP_ERR_INVALID_ARG, "bad y_dtype");
    if (!(eps >= 0.f)) return fail(DTP_ERR_INVALID_ARG, "eps must be >= 0");
    if ((cols % 4 == 0) && (!aligned(x, 16) || !aligned(w, 16)))
        return fail(DTP_ERR_INVALID_ARG, "x and w must be 16-byte aligned");
    DTP_CUDA_CHECK(launch_rmsnorm(x, w, y, y_dtype, rows, cols, eps, (cudaStream_t)stream));
    return DTP_OK;
}

int dtp_qk_norm_rope_neox(void* x, int dtype, const float* w_norm, const int32_t* pos, int T,
                          int n_heads, int head_dim, int rope_dim_count, float freq_base,
                          float eps, dtp_stream_t stream) {
    if (!x) return fail(DTP_ERR_INVALID_ARG, "NULL x");
    if (dtype != DTP_F32 && dtype != DTP_BF16) return fail(DTP_ERR_INVALID_ARG, "bad dtype");
    if (T <= 0 || n_heads <= 0 || head_dim <= 0 || head_dim % 2)
        return fail(DTP_ERR_INVALID_ARG, "T, n_heads must be >= 1 and head_dim even");
    if (rope_dim_count <= 0 || rope_dim_count % 2 || rope_dim_count > head_dim)
        return fail(DTP_ERR_INVALID_ARG, "rope_dim_count must be even and in [2, head_dim]");
    if (head_dim > 1024) return fail(DTP_ERR_UNSUPPORTED, "head_dim > 1024");
    if (!(freq_base > 0.f) || !(eps >= 0.f))
        return fail(DTP_ERR_INVALID_ARG, "freq_base must be > 0 and eps >= 0");
    DTP_CUDA_CHECK(launch_qk_norm_rope(x, dtype, n_heads * head_dim, w_norm, pos, T, n_heads,
                                       head_dim, rope_dim_count, freq_base, eps,
                                       (cudaStream_t)stream));
    return DTP_OK;
}

size_t dtp_sdpa_workspace_size(int T, int n_head_kv, int head_dim, int dtype) {
    if (T <= 0 || n_head_kv <= 0 || head_dim <= 0 || (dtype != DTP_BF16 && dtype != DTP_TF32))
        return 0;
    const size_t eb = dtype == DTP_TF32 ? 4 : 2;
    return align_up((size_t)n_head_kv * head_dim * align_up(T, 8) * eb, 256);
}

int dtp_sdpa_causal_gqa(const void* q, const void* k, const void* v, void* out, int dtype, int T,
                        int n_head, int n_head_kv, int head_dim, float scale, void* workspace,
                        size_t ws_bytes, dtp_stream_t stream) {
    if (!q || !k || !v || !out) return fail(DTP_ERR_INVALID_ARG, "NULL pointer");
    if (dtype != DTP_F32 && dtype != DTP_BF16 && dtype != DTP_TF32)
        return fail(DTP_ERR_INVALID_ARG, "bad dtype");
    if (T <= 0 || n_head <= 0 || n_head_kv <= 0 || head_dim <= 0)
        return fail(DTP_ERR_INVALID_ARG, "sizes must be >= 1");
    if (n_head % n_head_kv) return fail(DTP_ERR_INVALID_ARG, "n_head %% n_head_kv != 0");
    if (head_dim > 256) return fail(DTP_ERR_UNSUPPORTED, "head_dim > 256");
    cudaStream_t s = (cudaStream_t)stream;
    if (dtype == DTP_F32) {
        DTP_CUDA_CHECK(launch_attn_simt(q, n_head * head_dim, k, n_head_kv * head_dim, v,
                                        n_head_kv * head_dim, 0, out, n_head * head_dim, DTP_F32,
                                        T, n_head, n_head_kv, head_dim, scale, s));
        return DTP_OK;
    }
    if (!attn_tc_supported(n_head, n_head_kv, head_dim))
        return fail(DTP_ERR_UNSUPPORTED,
                    "tensor-core attention: head_dim must be 64 or 128 and n_head/n_head_kv even");
    const size_t need = dtp_sdpa_workspace_size(T, n_head_kv, head_dim, dtype);
    if (!workspace || ws_bytes < need)
        return fail(DTP_ERR_WORKSPACE, "sdpa workspace %zu < %zu bytes", ws_bytes, need);
    if (!aligned(workspace, 256) || !aligned(q, 16) || !aligned(k, 16) || !aligned(out, 16))
        return fail(DTP_ERR_INVALID_ARG, "q, k, out must be 16-byte and workspace 256-byte aligned");
    const long long ldvt = (long long)align_up(T, 8);
    if (dtype == DTP_TF32) {
        const int nq = n_head * head_dim, nk = n_head_kv * head_dim;
        float* vt32 = (float*)workspace;
        DTP_CUDA_CHECK(launch_transpose_v_f32((const float*)v, nk, vt32, T, nk, (int)ldvt, s));
        AttnVarlen none;
        DTP_CUDA_CHECK(launch_attn_tc_f32((const float*)q, nq, head_dim, (const float*)k, nk, vt32,
                                          ldvt, T, (float*)out, T, n_head, n_head_kv, head_dim,
                                          scale, none, s));
        return DTP_OK;
    }
    __half* vt = (__half*)workspace;
    DTP_CUDA_CHECK(launch_transpose_v((const __nv_bfloat16*)v, vt, T, n_head_kv * head_dim,
                                      (int)ldvt, s));
    DTP_CUDA_CHECK(launch_attn_tc((const __nv_bfloat16*)q, (const __nv_bfloat16*)k, vt, ldvt,
                                  (__nv_bfloat16*)out, T, n_head, n_head_kv, head_dim, scale, s));
    return DTP_OK;
}

int dtp_swiglu(const void* gate, const void* up, void* out, int dtype, size_t n,
               dtp_stream_t stream) {
    if (!gate || !up || !out) return fail(DTP_ERR_INVALID_ARG, "NULL pointer");
    if (dtype != DTP_F32 && dtype != DTP_BF16) return fail(DTP_ERR_INVALID_ARG, "bad dtype");
    if (n == 0) return DTP_OK;
    DTP_CUDA_CHECK(launch_swiglu(gate, up, out, dtype, n, (cudaStream_t)stream));
    return DTP_OK;
}

int dtp_linear(const void* x, const void* W, void* y, int dtype, int y_dtype, int M, int N, int K,
               const float* residual, dtp_stream_t stream) {
    if (!x || !W || !y) return fail(DTP_ERR_INVALID_ARG, "NULL pointer");
    if (M <= 0 || N <= 0 || K <= 0) return fail(DTP_ERR_INVALID_ARG, "M, N, K must be >= 1");
    if ((dtype != DTP_F32 && dtype != DTP_BF16 && dtype != DTP_TF32) ||
        (y_dtype != DTP_F32 && y_dtype != DTP_BF16))
        return fail(DTP_ERR_INVALID_ARG, "bad dtype");
    if (residual && y_dtype != DTP_F32)
        return fail(DTP_ERR_INVALID_ARG, "a residual needs a float32 output");
    cudaStream_t s = (cudaStream_t)stream;
    if (dtype == DTP_TF32) {
        if (y_dtype != DTP_F32) return fail(DTP_ERR_INVALID_ARG, "tf32 linear: y must be float32");
        if (K % 4) return fail(DTP_ERR_UNSUPPORTED, "tf32 linear: K must be a multiple of 4");
        if (!aligned(x, 16) || !aligned(W, 16))
            return fail(DTP_ERR_INVALID_ARG, "tf32 linear: x and W must be 16-byte aligned");
        GemmEpiArgs e;
        e.y = y;
        e.y_dtype = DTP_F32;
        e.ldy = N;
        e.residual = residual;
        DTP_CUDA_CHECK(launch_gemm_tc_tf32((const float*)x, (const float*)W, M, N, K, e, s,
                                           DTP_K_OTHER));
        return DTP_OK;
    }
    if (dtype == DTP_F32) {
        DTP_CUDA_CHECK(launch_gemm_simt((const float*)x, K, (const float*)W, y, y_dtype, N, M, N, K,
                                        residual, s, DTP_K_OTHER));
        return DTP_OK;
    }
    if (K % 8) return fail(DTP_ERR_UNSUPPORTED, "bf16 linear: K must be a multiple of 8");
    if (!aligned(x, 16) || !aligned(W, 16))
        return fail(DTP_ERR_INVALID_ARG, "bf16 linear: x and W must be 16-byte aligned");
    GemmEpiArgs e;
    e.y = y;
    e.y_dtype = y_dtype;
    e.ldy = N;
    e.residual = residual;
    DTP_CUDA_CHECK(launch_gemm_tc((const __nv_bfloat16*)x, (const __nv_bfloat16*)W, M, N, K,
                                  EPI_STORE, e, s, DTP_K_OTHER));
    return DTP_OK;
}

int dtp_quantize_rows_e4m3(const void* x, int dtype, int rows, int cols, uint8_t* q, float* scale,
                           dtp_stream_t stream) {
    if (!x || !q || !scale) return fail(DTP_ERR_INVALID_ARG, "NULL pointer");
    if (rows <= 0 || cols <= 0) return fail(DTP_ERR_INVALID_ARG, "rows and cols must be >= 1");
    cudaStream_t s = (cudaStream_t)stream;
    if (dtype == DTP_F32) {      // the weight-packing kernel quantises float32 rows
        DTP_CUDA_CHECK(launch_pack_e4m3((const float*)x, rows, cols, q, scale, 0, s));
        return DTP_OK;
    }
    if (dtype != DTP_BF16) return fail(DTP_ERR_INVALID_ARG, "bad dtype");
    if (cols % 8 || !aligned(x, 16) || !aligned(q, 8))
        return fail(DTP_ERR_UNSUPPORTED, "bf16 rows: cols %% 8 == 0, x 16- and q 8-byte aligned");
    DTP_CUDA_CHECK(launch_quant_rows_e4m3((const __nv_bfloat16*)x, cols, rows, cols, q, scale, s));
    return DTP_OK;
}

int dtp_rms_norm_e4m3(const float* x, const float* w, uint8_t* q, float* scale, int rows, int cols,
                      float eps, dtp_stream_t stream) {
    if (!x || !w || !q || !scale) return fail(DTP_ERR_INVALID_ARG, "NULL pointer");
    if (rows <= 0 || cols <= 0) return fail(DTP_ERR_INVALID_ARG, "rows and cols must be >= 1");
    if (!(eps >= 0.f)) return fail(DTP_ERR_INVALID_ARG, "eps must be >= 0");
    if (cols % 4 || cols > 16384 || !aligned(x, 16) || !aligned(w, 16) || !aligned(q, 4))
        return fail(DTP_ERR_UNSUPPORTED,
                    "cols %% 4 == 0 and <= 16384, x/w 16-byte and q 4-byte aligned");
    DTP_CUDA_CHECK(launch_rmsnorm_e4m3(x, w, q, scale, rows, cols, eps, (cudaStream_t)stream));
    return DTP_OK;
}

int dtp_linear_e4m3(const uint8_t* xq, const float* x_scale, const uint8_t* wq,
                    const float* w_scale, float* y, int M, int N, int K, const float* residual,
                    dtp_stream_t stream) {
    if (!xq || !x_scale || !wq || !w_scale || !y) return fail(DTP_ERR_INVALID_ARG, "NULL pointer");
    if (M <= 0 || N <= 0 || K <= 0) return fail(DTP_ERR_INVALID_ARG, "M, N, K must be >= 1");
    if (K % 16) return fail(DTP_ERR_UNSUPPORTED, "e4m3 linear: K must be a multiple of 16");
    if (!aligned(xq, 16) || !aligned(wq, 16))
        return fail(DTP_ERR_INVALID_ARG, "e4m3 linear: xq and wq must be 16-byte aligned");
    GemmEpiArgs e;
    e.y = y;
    e.y_dtype = DTP_F32;
    e.ldy = N;
    e.residual = residual;
    e.a_scale = x_scale;
    e.b_scale = w_scale;
    DTP_CUDA_CHECK(launch_gemm_tc_e4m3(xq, wq, M, N, K, EPI_STORE, e, (cudaStream_t)stream,
                                       DTP_K_OTHER));
    return DTP_OK;
}

size_t dtp_qkv_norm_rope_workspace_size(int T, int rope_dim_count) {
    if (T <= 0 || rope_dim_count <= 0 || rope_dim_count % 2) return 0;
    return align_up((size_t)T * (rope_dim_count / 2) * sizeof(float2), 256);
}

int dtp_qkv_norm_rope(const void* h, const void* w_qkv, const float* q_norm, const float* k_norm,
                      void* q, void* k, void* vt, int ldvt, int T, int d, int n_head,
                      int n_head_kv, int head_dim, int rope_dim_count, float freq_base, float eps,
                      void* workspace, size_t ws_bytes, dtp_stream_t stream) {
    if (!h || !w_qkv || !q_norm || !k_norm || !q || !k || !vt || !workspace)
        return fail(DTP_ERR_INVALID_ARG, "NULL pointer");
    if (T <= 0 || d <= 0 || n_head <= 0 || n_head_kv <= 0 || n_head % n_head_kv)
        return fail(DTP_ERR_INVALID_ARG, "bad sizes (T, d, n_head, n_head_kv)");
    if (rope_dim_count <= 0 || rope_dim_count % 2 || rope_dim_count > head_dim)
        return fail(DTP_ERR_INVALID_ARG, "rope_dim_count must be even and in [2, head_dim]");
    if (!(freq_base > 0.f) || !(eps >= 0.f))
        return fail(DTP_ERR_INVALID_ARG, "freq_base must be > 0 and eps >= 0");
    if (ldvt < T || ldvt % 8) return fail(DTP_ERR_INVALID_ARG, "ldvt must be >= T and a multiple of 8");
    if (d % 8 || (head_dim != 64 && head_dim != 128) || (rope_dim_count / 2) % 32 ||
        (head_dim - rope_dim_count) % 32)
        return fail(DTP_ERR_UNSUPPORTED,
                    "needs d %% 8 == 0, head_dim 64 or 128, rope_dim_count/2 and "
                    "head_dim-rope_dim_count multiples of 32");
    if (ws_bytes < dtp_qkv_norm_rope_workspace_size(T, rope_dim_count))
        return fail(DTP_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes,
                    dtp_qkv_norm_rope_workspace_size(T, rope_dim_count));
    if (!aligned(h, 16) || !aligned(w_qkv, 16) || !aligned(q, 16) || !aligned(k, 16) ||
        !aligned(workspace, 16))
        return fail(DTP_ERR_INVALID_ARG, "h, w_qkv, q, k and workspace must be 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    float2* rope = (float2*)workspace;
    DTP_CUDA_CHECK(launch_rope_table(rope, T, rope_dim_count, freq_base, s));
    GemmEpiArgs e;
    e.q = (__nv_bfloat16*)q;
    e.k = (__nv_bfloat16*)k;
    e.vt = (__half*)vt;
    e.ldvt = ldvt;
    e.q_norm = q_norm;
    e.k_norm = k_norm;
    e.rope = rope;
    e.n_head = n_head;
    e.n_head_kv = n_head_kv;
    e.head_dim = head_dim;
    e.rope_dims = rope_dim_count;
    e.eps = eps;
    const int nqkv = (n_head + 2 * n_head_kv) * head_dim;
    DTP_CUDA_CHECK(launch_gemm_tc((const __nv_bfloat16*)h, (const __nv_bfloat16*)w_qkv, T, nqkv,
                                  d, EPI_QKV, e, s, DTP_K_GEMM_QKV));
    return DTP_OK;
}

int dtp_gate_up_swiglu(const void* z, const void* w_gu, void* act, int T, int d, int n_ff,
                       dtp_stream_t stream) {
    if (!z || !w_gu || !act) return fail(DTP_ERR_INVALID_ARG, "NULL pointer");
    if (T <= 0 || d <= 0 || n_ff <= 0) return fail(DTP_ERR_INVALID_ARG, "sizes must be >= 1");
    if (d % 8 || n_ff % 64)
        return fail(DTP_ERR_UNSUPPORTED, "needs d %% 8 == 0 and n_ff %% 64 == 0");
    if (!aligned(z, 16) || !aligned(w_gu, 16) || !aligned(act, 16))
        return fail(DTP_ERR_INVALID_ARG, "z, w_gu and act must be 16-byte aligned");
    GemmEpiArgs e;
    e.act = (__nv_bfloat16*)act;
    DTP_CUDA_CHECK(launch_gemm_tc((const __nv_bfloat16*)z, (const __nv_bfloat16*)w_gu, T, 2 * n_ff,
                                  d, EPI_SWIGLU, e, (cudaStream_t)stream, DTP_K_GEMM_GATEUP));
    return DTP_OK;
}

int dtp_selftest_wait_timeout(dtp_stream_t stream) {
    DTP_CUDA_CHECK(launch_selftest_wait((cudaStream_t)stream));
    return DTP_OK;
}

// ------------------------------------------------------------------------- timers
int dtp_timer_enable(unsigned kind_mask, int capacity) {
    if (capacity <= 0 || capacity > 1 << 20) return fail(DTP_ERR_INVALID_ARG, "bad capacity");
    std::lock_guard<std::mutex> lk(g_timer.mu);
    timer_destroy();
    for (int k = 0; k < DTP_K_COUNT; ++k) {
        if (!(kind_mask & (1u << k))) continue;
        for (int j = 0; j < 2; ++j) {
            g_timer.ev[k][j].resize(capacity);
            for (int i = 0; i < capacity; ++i) {
                cudaError_t e = cudaEventCreate(&g_timer.ev[k][j][i]);
                if (e != cudaSuccess) {
                    g_timer.ev[k][j].resize(i);
                    timer_destroy();
                    return fail(DTP_ERR_CUDA, "cudaEventCreate: %s", cudaGetErrorString(e));
                }
            }
        }
    }
    g_timer.capacity = capacity;
    g_timer.mask = kind_mask;
    return DTP_OK;
}

int dtp_timer_disable(void) {
    std::lock_guard<std::mutex> lk(g_timer.mu);
    timer_destroy();
    return DTP_OK;
}

int dtp_timer_spans(int kind, int ref_kind, int cap, float* start_ms, float* end_ms, int* count) {
    if (kind < 0 || kind >= DTP_K_COUNT || ref_kind < 0 || ref_kind >= DTP_K_COUNT || cap < 0 ||
        !count || (cap > 0 && (!start_ms || !end_ms)))
        return fail(DTP_ERR_INVALID_ARG, "bad kind, capacity or NULL output");
    std::lock_guard<std::mutex> lk(g_timer.mu);
    const int n = g_timer.used[kind];
    if (n > 0 && g_timer.used[ref_kind] == 0)
        return fail(DTP_ERR_INVALID_ARG, "no span of the reference kind was recorded");
    for (int i = 0; i < n && i < cap; ++i) {
        cudaEvent_t origin = g_timer.ev[ref_kind][0][0];
        cudaError_t e = cudaEventElapsedTime(&start_ms[i], origin, g_timer.ev[kind][0][i]);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&end_ms[i], origin, g_timer.ev[kind][1][i]);
        if (e != cudaSuccess)
            return fail(DTP_ERR_CUDA, "cudaEventElapsedTime: %s", cudaGetErrorString(e));
    }
    *count = n;
    return DTP_OK;
}

int dtp_timer_read(int kind, int* count, float* total_ms) {
    if (kind < 0 || kind >= DTP_K_COUNT || !count || !total_ms)
        return fail(DTP_ERR_INVALID_ARG, "bad kind or NULL output");
    std::lock_guard<std::mutex> lk(g_timer.mu);
    float tot = 0.f;
    const int n = g_timer.used[kind];
    for (int i = 0; i < n; ++i) {
        float ms = 0.f;
        cudaError_t e = cudaEventElapsedTime(&ms, g_timer.ev[kind][0][i], g_timer.ev[kind][1][i]);
        if (e != cudaSuccess) return fail(DTP_ERR_CUDA, "cudaEventElapsedTime: %s", cudaGetErrorString(e));
        tot += ms;
    }
    *count = n;
    *total_ms = tot;
    return DTP_OK;
}

}  // extern "C"
