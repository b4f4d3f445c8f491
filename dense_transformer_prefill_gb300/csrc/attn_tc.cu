// tcgen05 causal grouped-query flash attention (docs.rs memra-engine 0.130.0,
// src/forward.rs, Model::forward: the attention step, causal, over all T keys,
// scaled by 1/sqrt(head_dim); restated as an online-softmax tiled kernel, the
// pages' naive kernel being prior art only).
//
// One CTA = one 128-token query tile of TWO query heads of the same GQA group,
// so every K/V tile brought into shared memory serves 256 query rows.
//   warp 0      TMA: Q tiles of both heads once, then per 128-key tile K_j
//               (one stage) and V_j^T (two stages; v is stored transposed,
//               key index contiguous, so both MMAs read K-major operands)
//   warp 1      one thread issues S_i = Q_i K_j^T (M=128, N=128 keys) into TMEM
//               and O_i += P_i V_j (M=128, N=head_dim) into TMEM, ordered
//               S0 S1 | PV0 S0' | PV1 S1' | ... so each head's softmax
//               overlaps the other head's MMAs
//   warps 2-5   softmax of head 0; warps 6-9 softmax of head 1: TMEM lane =
//               query row; scores scaled into log2 units, running max kept
//               unless it grows by more than 8 (then O is rescaled in TMEM),
//               P = 2^(s - m) rounded to f16 into 128-byte-swizzled shared
//               memory, row sums in float32
// Q K^T runs on bf16 operands; P V on f16 operands (P <= 2^8 under the
// rescale rule, and v^T holds f16 copies of the bf16 values, exact from 2^-14
// up to the f16 range, smaller ones within 2^-25), so P keeps 11 significant
// bits, not 8.
// The same kernel runs on float32 operands holding tf32 values (F32: kind::tf32,
// 32-key tiles so that both heads' float32 Q tiles fit in shared memory, P
// rounded to tf32, float32 output).
// Causality: key tiles up to the one holding the tile's last query position;
// tiles that reach past the first query position mask key > query.  Queries may
// start at a position p0 > 0 (chunked prefill against earlier keys).
// Persistent: one CTA per SM walks work items (a query tile of a head pair),
// longest first, in rounds of one item per CTA whose direction alternates;
// TMEM, barriers and the pipeline carry over from item to item, so the next
// item's Q/K loads and first Q K^T overlap the previous item's last softmax
// and epilogue.
#include <math.h>
#include <mutex>

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

bool attn_tc_supported(int n_head, int n_head_kv, int head_dim) {
    return (head_dim == 64 || head_dim == 128) && n_head_kv > 0 && n_head % n_head_kv == 0 &&
           (n_head / n_head_kv) % 2 == 0;
}

namespace {

constexpr int BQ = 128;          // query rows per tile
constexpr int kThreads = 320;    // 10 warps
constexpr float kRescaleLog2 = 8.0f;
constexpr float kRescaleSum = 256.0f;   // 2^kRescaleLog2

// F32: tf32 operands in float32 storage.  A 128-byte shared-memory row holds
// AE elements (64 bf16 or 32 float32); one MMA consumes 32 bytes of K per row.
template <int HD, bool F32>
struct ACfg {
    static constexpr int EB = F32 ? 4 : 2;
    static constexpr int AE = 128 / EB;
    static constexpr int KSTEP = 32 / EB;
    static constexpr int BKV = F32 ? 32 : 128;       // keys per tile
    static constexpr int Q_BYTES = BQ * HD * EB;
    static constexpr int K_BYTES = BKV * HD * EB;
    static constexpr int V_BYTES = HD * BKV * EB;
    static constexpr int P_BYTES = BQ * BKV * EB;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
    static constexpr int OFF_V = OFF_K + K_BYTES;
    static constexpr int OFF_P = OFF_V + 2 * V_BYTES;
    static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
    static constexpr int SMEM_BYTES = 1024 + OFF_BAR + 256;
    static constexpr int TMEM_COLS = 512;
    static constexpr uint32_t S_COL0 = 0, O_COL0 = 2 * BKV;
};

struct AParams {
    int T, n_head, n_head_kv, n_qt;   // n_qt: query tiles in the schedule (an upper bound for varlen)
    float scale_log2;
    void* out;                        // bf16, or float32 with F32
    int ldo;
    int q_head_stride;                // Q tile column of head h = h * q_head_stride
    // several sequences packed along the token axis (n_seq == 0: one sequence of T tokens)
    int n_seq;
    const int* cu_seqlens;   // [n_seq + 1] token offsets
    const int* tile_start;   // [n_seq + 1] prefix of ceil(len / 128)
    const int* vcol_start;   // [n_seq] first v^T column of each sequence (multiple of 8)
    const __nv_bfloat16* gate;   // optional [T, n_head*hd]: out *= sigmoid(gate) (bf16 only)
    // one sequence (n_seq == 0): queries sit at positions p0 .. p0+T-1 and see
    // keys 0 .. p0+T-1 (kv_len = p0 + T)
    int p0, kv_len;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Max of the unmasked scores of this thread's row of a bf16-mode score tile in
// TMEM (64 columns per load).  DIAG masks keys past the query: key column col
// is hidden from this row when col > row + dof (dof = first query position of
// the tile - first key position).
template <bool DIAG, int BKV>
__device__ __forceinline__ void row_max_bf16(uint32_t tS, int row, int dof, float& mx) {
#pragma unroll
    for (int c = 0; c < BKV; c += 64) {
        uint32_t r[64];
        __syncwarp();
        ptx::tmem_ld64(tS + c, r);
#pragma unroll
        for (int t = 0; t < 64; ++t) {
            const bool masked = DIAG && c + t > row + dof;
            mx = masked ? mx : fmaxf(mx, __uint_as_float(r[t]));
        }
    }
}

// P = 2^(s*sl2 - m_ref) of this thread's row, rounded to f16 into the row's
// 128-byte-swizzled shared-memory slots; rs += sum(P).  The scale-and-shift and
// the row sum run on packed float pairs (two lanes of work per instruction).
template <bool DIAG, int BKV>
__device__ __forceinline__ void row_exp_bf16(uint32_t tS, uint8_t* Prow, int sw, int row, int dof,
                                             float sl2, float m_ref, float& rs) {
    const float2 k2 = make_float2(sl2, sl2), b2 = make_float2(-m_ref, -m_ref);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < BKV; c += 64) {
        uint32_t r[64];
        __syncwarp();
        ptx::tmem_ld64(tS + c, r);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
            float e[8];
#pragma unroll
            for (int t = 0; t < 8; t += 2) {
                const int col = c + c8 * 8 + t;
                const float2 x = __ffma2_rn(
                    make_float2(__uint_as_float(r[c8 * 8 + t]), __uint_as_float(r[c8 * 8 + t + 1])),
                    k2, b2);
                float2 ev = make_float2(ex2(x.x), ex2(x.y));
                if (DIAG) {
                    ev.x = col > row + dof ? 0.f : ev.x;
                    ev.y = col + 1 > row + dof ? 0.f : ev.y;
                }
                acc = __fadd2_rn(acc, ev);
                e[t] = ev.x;
                e[t + 1] = ev.y;
            }
            uint4 u;
            u.x = ptx::pack_f16x2(e[0], e[1]);
            u.y = ptx::pack_f16x2(e[2], e[3]);
            u.z = ptx::pack_f16x2(e[4], e[5]);
            u.w = ptx::pack_f16x2(e[6], e[7]);
            const int chunk_all = (c >> 3) + c8;          // 16-byte chunk index 0..15
            const int atom = chunk_all >> 3, chunk = chunk_all & 7;
            *reinterpret_cast<uint4*>(Prow + atom * BQ * 128 + ((chunk ^ sw) << 4)) = u;
        }
    }
    rs += acc.x + acc.y;
}

// Round a float32 to tf32 (10 fraction bits), nearest with ties to even.
__device__ __forceinline__ float tf32_rne(float x) {
    uint32_t u = __float_as_uint(x);
    u += 0xFFFu + ((u >> 13) & 1u);
    return __uint_as_float(u & ~0x1FFFu);
}

// The same pass on a 32-key tile with P as tf32 in float32 storage (one
// 128-byte row per query: 16-byte chunk c/4 holds keys c .. c+3).
template <bool DIAG, bool WRITE>
__device__ __forceinline__ void tile_pass_f32(uint32_t tS, uint8_t* Prow, int sw, int row, int dof,
                                              float sl2, float m_ref, float& mx, float& rs) {
    uint32_t r[32];
    __syncwarp();
    ptx::tmem_ld32(tS, r);
#pragma unroll
    for (int c4 = 0; c4 < 8; ++c4) {
        float e[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int col = c4 * 4 + t;
            const float sv = __uint_as_float(r[col]);
            const bool masked = DIAG && col > row + dof;
            mx = masked ? mx : fmaxf(mx, sv);
            if (WRITE) {
                e[t] = masked ? 0.f : tf32_rne(ex2(fmaf(sv, sl2, -m_ref)));
                rs += e[t];
            }
        }
        if (WRITE)
            *reinterpret_cast<uint4*>(Prow + ((c4 ^ sw) << 4)) =
                make_uint4(__float_as_uint(e[0]), __float_as_uint(e[1]), __float_as_uint(e[2]),
                           __float_as_uint(e[3]));
    }
}

// The row's tile max (row_max) and its P with row sum (row_exp), bf16 or tf32.
template <bool DIAG, bool F32, int BKV>
__device__ __forceinline__ void row_max(uint32_t tS, int row, int dof, float& mx) {
    if constexpr (F32) {
        float unused = 0.f;
        tile_pass_f32<DIAG, false>(tS, nullptr, 0, row, dof, 0.f, 0.f, mx, unused);
    } else {
        row_max_bf16<DIAG, BKV>(tS, row, dof, mx);
    }
}
template <bool DIAG, bool F32, int BKV>
__device__ __forceinline__ void row_exp(uint32_t tS, uint8_t* Prow, int sw, int row, int dof,
                                        float sl2, float m_ref, float& rs) {
    if constexpr (F32) {
        float unused = -INFINITY;
        tile_pass_f32<DIAG, true>(tS, Prow, sw, row, dof, sl2, m_ref, unused, rs);
    } else {
        row_exp_bf16<DIAG, BKV>(tS, Prow, sw, row, dof, sl2, m_ref, rs);
    }
}

// One work item: a 128-row query tile of a head pair.  Items are numbered
// longest first (the query tile with the most key tiles first); item w -> its
// query tile, kv head g and first query head h0, the sequence it belongs to,
// the position of its first query and its number of key tiles.  Returns false
// for an item beyond a packed-sequence schedule.
struct AItem {
    int qt, g, h0, seq_start, seq_len, vstart, qpos0, n_kv;
};
__device__ __forceinline__ bool attn_item(const AParams& p, int w, int bkv, AItem& it) {
    const int G = p.n_head / p.n_head_kv, pairs = G / 2;
    const int items_per_qt = p.n_head_kv * pairs;
    const int tile_idx = p.n_qt - 1 - w / items_per_qt;
    const int rem = w % items_per_qt;
    it.g = rem / pairs;
    it.h0 = it.g * G + 2 * (rem % pairs);
    it.qt = tile_idx;
    it.seq_start = 0;
    it.seq_len = p.T;
    it.vstart = 0;
    it.qpos0 = p.p0;
    int kv_len = p.kv_len;
    if (p.n_seq > 0) {
        if (tile_idx >= p.tile_start[p.n_seq]) return false;
        int lo = 0, hi = p.n_seq - 1;                        // last b with tile_start[b] <= tile_idx
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.tile_start[mid] <= tile_idx) lo = mid;
            else hi = mid - 1;
        }
        it.qt = tile_idx - p.tile_start[lo];
        it.seq_start = p.cu_seqlens[lo];
        it.seq_len = p.cu_seqlens[lo + 1] - it.seq_start;
        it.vstart = p.vcol_start[lo];
        it.qpos0 = 0;
        kv_len = it.seq_len;
    }
    it.qpos0 += it.qt * BQ;                 // position of the tile's first query
    // key tiles up to the one holding the tile's last query position
    const int kv_tiles = (kv_len + bkv - 1) / bkv, need_tiles = (it.qpos0 + BQ - 1) / bkv + 1;
    it.n_kv = kv_tiles < need_tiles ? kv_tiles : need_tiles;
    return true;
}

// The r-th item of CTA b among `nb` persistent CTAs: rounds of nb items, the
// direction alternating round by round (longest items spread evenly).  -1 when
// the CTA has no r-th item.
__device__ __forceinline__ int attn_item_index(int r, int b, int nb, int n_items) {
    const int w = r * nb + ((r & 1) ? nb - 1 - b : b);
    return w < n_items ? w : -1;
}

template <int HD, bool F32>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AParams p) {
    using C = ACfg<HD, F32>;
    constexpr int BKV = C::BKV, AE = C::AE, KSTEP = C::KSTEP;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem + C::OFF_Q;
    uint8_t* sK = smem + C::OFF_K;
    uint8_t* sV = smem + C::OFF_V;
    uint8_t* sP = smem + C::OFF_P;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* q_full = bars + 0;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = bars + 2;
    uint64_t* v_full = bars + 3;      // [2]
    uint64_t* v_empty = bars + 5;     // [2]
    uint64_t* s_full = bars + 7;      // [2]
    uint64_t* p_full = bars + 9;      // [2]
    uint64_t* o_done = bars + 11;     // [2]
    uint64_t* drain = bars + 13;
    uint64_t* q_empty = bars + 14;    // the item's last Q K^T is done: Q may be replaced
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 15);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // persistent: this CTA takes items b, then (rounds alternating direction)
    // one per round of gridDim.x items, until they run out
    const int n_items = p.n_qt * p.n_head_kv * (p.n_head / p.n_head_kv / 2);
    const int b = (int)blockIdx.x, nb = (int)gridDim.x;

    if (threadIdx.x == 0) {
        ptx::mbar_init(q_full, 1);
        ptx::mbar_init(k_full, 1);
        ptx::mbar_init(k_empty, 1);
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&v_full[i], 1);
            ptx::mbar_init(&v_empty[i], 1);
            ptx::mbar_init(&s_full[i], 1);
            ptx::mbar_init(&p_full[i], 4);     // lane 0 of each softmax warp of head i
            ptx::mbar_init(&o_done[i], 1);
        }
        ptx::mbar_init(drain, 1);
        ptx::mbar_init(q_empty, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    // the warp-collective TMEM allocation and the CTA barrier below are
    // .aligned: every warp arrives converged (thread 0 ran the set-up alone)
    __syncwarp();
    if (warp == 0) {
        ptx::tmem_alloc(tmem_holder, C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            ptx::tma_prefetch_desc(&tmQ);
            ptx::tma_prefetch_desc(&tmK);
            ptx::tma_prefetch_desc(&tmV);
            // loads so far (they index the barriers' phases across items)
            int q_issued = 0, k_issued = 0, v_issued[2] = {0, 0}, kv_loads = 0;
            for (int r = 0; !*abort_flag; ++r) {
                const int w = attn_item_index(r, b, nb, n_items);
                if (w < 0) break;
                AItem it;
                if (!attn_item(p, w, BKV, it)) continue;
                // the previous item's last Q K^T has read Q
                if (q_issued > 0 && !ptx::wait_bounded(q_empty, (q_issued - 1) & 1, abort_flag,
                                                       &g_attn_err, ERRBIT_TIMEOUT))
                    break;
                ptx::mbar_arrive_expect_tx(q_full, 2 * C::Q_BYTES);
                for (int i = 0; i < 2; ++i)
                    for (int a = 0; a < HD / AE; ++a)
                        ptx::tma_load_2d(&tmQ, q_full, sQ + i * C::Q_BYTES + a * BQ * 128,
                                         (it.h0 + i) * p.q_head_stride + a * AE,
                                         it.seq_start + it.qt * BQ);
                ++q_issued;
                for (int j = 0; j < it.n_kv; ++j) {
                    if (!ptx::wait_bounded(k_empty, (k_issued & 1) ^ 1, abort_flag, &g_attn_err,
                                           ERRBIT_TIMEOUT))
                        break;
                    ptx::mbar_arrive_expect_tx(k_full, C::K_BYTES);
                    for (int a = 0; a < HD / AE; ++a)
                        ptx::tma_load_2d(&tmK, k_full, sK + a * BKV * 128, it.g * HD + a * AE,
                                         it.seq_start + j * BKV);
                    ++k_issued;
                    const int vs = kv_loads & 1;
                    if (!ptx::wait_bounded(&v_empty[vs], ((kv_loads >> 1) & 1) ^ 1, abort_flag,
                                           &g_attn_err, ERRBIT_TIMEOUT))
                        break;
                    ptx::mbar_arrive_expect_tx(&v_full[vs], C::V_BYTES);
                    for (int a = 0; a < BKV / AE; ++a)
                        ptx::tma_load_2d(&tmV, &v_full[vs], sV + vs * C::V_BYTES + a * HD * 128,
                                         it.vstart + j * BKV + a * AE, it.g * HD);
                    ++v_issued[vs];
                    ++kv_loads;
                }
            }
            if (*abort_flag) {
                // let the loads still in flight land before the CTA can exit: the
                // latest phase of each barrier completes when its bytes arrive
                volatile int never = 0;
                if (q_issued)
                    ptx::wait_bounded(q_full, (q_issued - 1) & 1, &never, &g_attn_err,
                                      ERRBIT_TIMEOUT);
                if (k_issued)
                    ptx::wait_bounded(k_full, (k_issued - 1) & 1, &never, &g_attn_err,
                                      ERRBIT_TIMEOUT);
                for (int vs = 0; vs < 2; ++vs)
                    if (v_issued[vs])
                        ptx::wait_bounded(&v_full[vs], (v_issued[vs] - 1) & 1, &never, &g_attn_err,
                                          ERRBIT_TIMEOUT);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            const uint32_t idS = F32 ? ptx::idesc_tf32_f32(BQ, BKV) : ptx::idesc_bf16_f32(BQ, BKV);
            // P V^T: f16 A and B (the kind::f16 MMA reads the operand types from
            // the descriptor; both operands of one MMA share a type)
            const uint32_t idO = F32 ? ptx::idesc_tf32_f32(BQ, HD) : ptx::idesc_f16_f32(BQ, HD);
            auto mma = [&](uint32_t d, uint64_t da, uint64_t db, uint32_t id, uint32_t acc) {
                if constexpr (F32) ptx::umma_tf32_ss(d, da, db, id, acc);
                else ptx::umma_bf16_ss(d, da, db, id, acc);
            };
            auto issue_S = [&](int i) {
                const uint32_t d = tmem_base + C::S_COL0 + i * BKV;
#pragma unroll
                for (int kk = 0; kk < HD / KSTEP; ++kk) {
                    const int a = kk / 4, off = (kk % 4) * 32;
                    const uint64_t da =
                        ptx::sdesc_sw128(ptx::smem_u32(sQ + i * C::Q_BYTES + a * BQ * 128 + off));
                    const uint64_t db = ptx::sdesc_sw128(ptx::smem_u32(sK + a * BKV * 128 + off));
                    mma(d, da, db, idS, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_PV = [&](int i, int vs, int j) {
                const uint32_t d = tmem_base + C::O_COL0 + i * HD;
#pragma unroll
                for (int kk = 0; kk < BKV / KSTEP; ++kk) {
                    const int a = kk / 4, off = (kk % 4) * 32;
                    const uint64_t da =
                        ptx::sdesc_sw128(ptx::smem_u32(sP + i * C::P_BYTES + a * BQ * 128 + off));
                    const uint64_t db = ptx::sdesc_sw128(
                        ptx::smem_u32(sV + vs * C::V_BYTES + a * HD * 128 + off));
                    mma(d, da, db, idO, (j > 0 || kk > 0) ? 1u : 0u);
                }
            };
            auto W = [&](uint64_t* b, uint32_t par) {
                return ptx::wait_bounded(b, par, abort_flag, &g_attn_err, ERRBIT_TIMEOUT);
            };
            // consumed so far, across items (they index the barriers' phases)
            int items = 0, k_used = 0, kv_used = 0, tiles = 0;
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int w = attn_item_index(r, b, nb, n_items);
                if (w < 0) break;
                AItem it;
                if (!attn_item(p, w, BKV, it)) continue;
                const int n_kv = it.n_kv;
                ok = W(q_full, items & 1) && W(k_full, k_used & 1);
                if (!ok) break;
                ptx::tc_fence_after();
                issue_S(0);
                ptx::umma_commit(&s_full[0]);
                issue_S(1);
                ptx::umma_commit(&s_full[1]);
                ptx::umma_commit(k_empty);
                ++k_used;
                if (n_kv == 1) ptx::umma_commit(q_empty);    // the item's last use of Q
                // the softmax of this item's tile 0 follows the previous item's
                // epilogue in the same warps, so p_full(tile 0) also means that
                // epilogue has read O: PV(0) may overwrite it
                for (int j = 0; ok && j < n_kv; ++j) {
                    const int vs = kv_used & 1, t = tiles + j;
                    if (!(W(&v_full[vs], (kv_used >> 1) & 1) && W(&p_full[0], t & 1))) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    issue_PV(0, vs, j);
                    ptx::umma_commit(&o_done[0]);
                    const bool more = j + 1 < n_kv;
                    if (more) {
                        if (!W(k_full, k_used & 1)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        issue_S(0);
                        ptx::umma_commit(&s_full[0]);
                    }
                    if (!W(&p_full[1], t & 1)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    issue_PV(1, vs, j);
                    ptx::umma_commit(&o_done[1]);
                    ptx::umma_commit(&v_empty[vs]);
                    ++kv_used;
                    if (more) {
                        issue_S(1);
                        ptx::umma_commit(&s_full[1]);
                        ptx::umma_commit(k_empty);
                        ++k_used;
                        if (j + 2 == n_kv) ptx::umma_commit(q_empty);
                    }
                }
                tiles += n_kv;
                ++items;
            }
            ptx::umma_commit(drain);
            volatile int never = 0;
            ptx::wait_bounded(drain, 0, &never, &g_attn_err, ERRBIT_TIMEOUT);
        }
    } else {
        // ---------------------------------------------------------------- softmax warps
        const int i = (warp - 2) / 4;            // which head of the pair
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem_base + lane_off + C::S_COL0 + i * BKV;
        const uint32_t tO = tmem_base + lane_off + C::O_COL0 + i * HD;
        uint8_t* Prow = sP + i * C::P_BYTES + row * 128;
        const int sw = row & 7;
        bool ok = true;
        int tiles = 0;                           // key tiles so far, across items
        for (int r = 0; ok; ++r) {
            const int w = attn_item_index(r, b, nb, n_items);
            if (w < 0) break;
            AItem it;
            if (!attn_item(p, w, BKV, it)) continue;
            const int n_kv = it.n_kv, qpos0 = it.qpos0, h0 = it.h0, seq_len = it.seq_len;
            const int qrel = it.qt * BQ + row;                   // position within the sequence
            const int qrow = it.seq_start + qrel;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < n_kv; ++j) {
                const int t = tiles + j;
                ok = ptx::wait_bounded(&s_full[i], t & 1, abort_flag, &g_attn_err, ERRBIT_TIMEOUT);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                // P_i and O_i are free once PV_i(j-1) has completed (it precedes
                // S_i(j) on the tensor pipe, so this wait normally returns at once);
                // at j = 0 the previous item's epilogue waited for its last PV
                if (j > 0) {
                    ok = ptx::wait_bounded(&o_done[i], (t - 1) & 1, abort_flag, &g_attn_err,
                                           ERRBIT_TIMEOUT);
                    if (!__all_sync(0xffffffffu, ok)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                }
                const int dof = qpos0 - j * BKV;           // key col c hidden iff c > row + dof
                const bool diag = dof < BKV - 1;
                const float sl2 = p.scale_log2;
                // Speculative single pass: P against the running max m.  A score more
                // than 2^8 above m makes its P, and so the row sum, exceed 2^8; only
                // then is the tile max taken, and if it does raise the row's max by more
                // than 2^8 that row takes the new max, l and O are rescaled and the warp
                // redoes the pass.  The first tile takes its max before the pass.
                float rs = 0.f;
                if (j == 0) {
                    float mx = -INFINITY;
                    if (diag) row_max<true, F32, BKV>(tS, row, dof, mx);
                    else row_max<false, F32, BKV>(tS, row, dof, mx);
                    m = mx * sl2;                   // key 0 is never masked on the first tile
                    if (diag) row_exp<true, F32, BKV>(tS, Prow, sw, row, dof, sl2, m, rs);
                    else row_exp<false, F32, BKV>(tS, Prow, sw, row, dof, sl2, m, rs);
                } else {
                    if (diag) row_exp<true, F32, BKV>(tS, Prow, sw, row, dof, sl2, m, rs);
                    else row_exp<false, F32, BKV>(tS, Prow, sw, row, dof, sl2, m, rs);
                    const bool suspect = !(rs <= kRescaleSum);
                    if (__any_sync(0xffffffffu, suspect)) {
                        float mx = -INFINITY;
                        if (diag) row_max<true, F32, BKV>(tS, row, dof, mx);
                        else row_max<false, F32, BKV>(tS, row, dof, mx);
                        const float m_tile = mx * sl2;
                        const bool need = m_tile > m + kRescaleLog2;
                        if (__any_sync(0xffffffffu, need)) {
                            float alpha = 1.f;
                            if (need) {
                                alpha = ex2(m - m_tile);
                                m = m_tile;
                                l *= alpha;
                            }
#pragma unroll 1
                            for (int c = 0; c < HD; c += 32) {
                                uint32_t r[32];
                                __syncwarp();
                                ptx::tmem_ld32(tO + c, r);
#pragma unroll
                                for (int t = 0; t < 32; ++t)
                                    r[t] = __float_as_uint(__uint_as_float(r[t]) * alpha);
                                ptx::tmem_st32(tO + c, r);
                            }
                            rs = 0.f;
                            if (diag) row_exp<true, F32, BKV>(tS, Prow, sw, row, dof, sl2, m, rs);
                            else row_exp<false, F32, BKV>(tS, Prow, sw, row, dof, sl2, m, rs);
                        }
                    }
                }
                l += rs;
                // every lane's P row is visible to the tensor core before lane 0
                // releases the warp's quarter of P_i
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&p_full[i]);
            }
            if (!ok) break;
            ok = ptx::wait_bounded(&o_done[i], (tiles + n_kv - 1) & 1, abort_flag, &g_attn_err,
                                   ERRBIT_TIMEOUT);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                {   // the epilogue: O / l, and the gate, to the output rows
                    ptx::tc_fence_after();
                    const float inv = 1.0f / l;
                    const size_t obase = (size_t)qrow * p.ldo + (size_t)(h0 + i) * HD;
                    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + obase;
                    float* orow32 = reinterpret_cast<float*>(p.out) + obase;
#pragma unroll 1
                    for (int c = 0; c < HD; c += 32) {
                        uint32_t r[32];
                        __syncwarp();
                        ptx::tmem_ld32(tO + c, r);
                        if (F32 && qrel < seq_len && qrow < p.T) {
#pragma unroll
                            for (int t = 0; t < 32; t += 4)
                                *reinterpret_cast<float4*>(orow32 + c + t) =
                                    make_float4(__uint_as_float(r[t]) * inv, __uint_as_float(r[t + 1]) * inv,
                                                __uint_as_float(r[t + 2]) * inv,
                                                __uint_as_float(r[t + 3]) * inv);
                        } else if (qrel < seq_len && qrow < p.T) {
#pragma unroll
                            for (int t = 0; t < 32; t += 8) {
                                float o[8];
#pragma unroll
                                for (int e = 0; e < 8; ++e) o[e] = __uint_as_float(r[t + e]) * inv;
                                if (p.gate) {      // gated attention: out *= sigmoid(gate)
                                    const uint4 gv = *reinterpret_cast<const uint4*>(
                                        p.gate + (size_t)qrow * p.ldo + (size_t)(h0 + i) * HD + c + t);
                                    const __nv_bfloat16* gb = reinterpret_cast<const __nv_bfloat16*>(&gv);
#pragma unroll
                                    for (int e = 0; e < 8; ++e)
                                        o[e] = o[e] / (1.0f + expf(-__bfloat162float(gb[e])));
                                }
                                uint4 u;
                                u.x = ptx::pack_bf16x2(o[0], o[1]);
                                u.y = ptx::pack_bf16x2(o[2], o[3]);
                                u.z = ptx::pack_bf16x2(o[4], o[5]);
                                u.w = ptx::pack_bf16x2(o[6], o[7]);
                                *reinterpret_cast<uint4*>(orow + c + t) = u;
                            }
                        }
                    }
                }
            }
            tiles += n_kv;
        }
    }

    // Warps 0 and 1 ran their roles on one lane: converge each warp before the
    // CTA barrier, which counts whole warps.  Without this, a GB300 probe saw
    // the producer's lane leave the barrier while the softmax warps still ran.
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int HD, bool F32>
cudaError_t launch_hd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const AParams& p, cudaStream_t s) {
    using C = ACfg<HD, F32>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(attn_tc_kernel<HD, F32>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return attr_err;
    // persistent CTAs, one per SM (the shared memory allows no second), each
    // taking its share of the work items
    const int G = p.n_head / p.n_head_kv;
    const int n_items = p.n_qt * p.n_head_kv * (G / 2);
    const int grid = n_items < num_sms() ? n_items : num_sms();
    attn_tc_kernel<HD, F32><<<grid, kThreads, C::SMEM_BYTES, s>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

// q [T, ldq] (head h at column h * q_head_stride), k [kv rows, ldk], v^T
// [n_head_kv * hd, ldvt] (vt_cols columns), out [T, n_head * hd].
template <bool F32>
cudaError_t launch_attn(const void* q, long long ldq, int q_head_stride, const void* k,
                        long long ldk, const void* vt, long long ldvt, long long vt_cols, void* out,
                        int T, int n_head, int n_head_kv, int head_dim, float scale,
                        const AttnVarlen& vl, cudaStream_t s) {
    if (!attn_tc_supported(n_head, n_head_kv, head_dim)) return cudaErrorNotSupported;
    if (F32 && vl.gate) return cudaErrorNotSupported;
    using C = ACfg<128, F32>;     // element geometry does not depend on HD
    const CUtensorMapDataType dt =
        F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapDataType dtv =
        F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tq, tk, tv;
    const int hd = head_dim;
    // keys: T rows, or p0 + T rows of a KV state (the map ends there, so keys past
    // the last query read zeros, never stale state)
    const int kv_len = vl.n_seq > 0 ? T : vl.p0 + T;
    if (!make_tmap_2d(&tq, q, dt, C::EB, T, (uint64_t)n_head * q_head_stride, (uint64_t)ldq, BQ,
                      C::AE) ||
        !make_tmap_2d(&tk, k, dt, C::EB, kv_len, (uint64_t)n_head_kv * hd, (uint64_t)ldk, C::BKV,
                      C::AE) ||
        !make_tmap_2d(&tv, vt, dtv, C::EB, (uint64_t)n_head_kv * hd, (uint64_t)vt_cols,
                      (uint64_t)ldvt, hd, C::AE))
        return cudaErrorInvalidValue;
    AParams p;
    p.T = T;
    p.n_head = n_head;
    p.n_head_kv = n_head_kv;
    p.n_qt = vl.n_seq > 0 ? (T + BQ - 1) / BQ + vl.n_seq : (T + BQ - 1) / BQ;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = out;
    p.ldo = n_head * hd;
    p.q_head_stride = q_head_stride;
    p.n_seq = vl.n_seq;
    p.cu_seqlens = vl.cu_seqlens;
    p.tile_start = vl.tile_start;
    p.vcol_start = vl.vcol_start;
    p.gate = vl.gate;
    p.p0 = vl.n_seq > 0 ? 0 : vl.p0;
    p.kv_len = kv_len;
    LaunchScope ls(DTP_K_ATTN, s);
    if (hd == 128) return launch_hd<128, F32>(tq, tk, tv, p, s);
    return launch_hd<64, F32>(tq, tk, tv, p, s);
}

}  // namespace

cudaError_t launch_attn_tc(const __nv_bfloat16* q, const __nv_bfloat16* k,
                           const __half* vt, long long ldvt, __nv_bfloat16* out, int T,
                           int n_head, int n_head_kv, int head_dim, float scale, cudaStream_t s) {
    AttnVarlen none;
    return launch_attn_tc_varlen(q, k, vt, ldvt, T, out, T, n_head, n_head_kv, head_dim, scale,
                                 none, s);
}

cudaError_t launch_attn_tc_varlen(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                  const __half* vt, long long ldvt, long long vt_cols,
                                  __nv_bfloat16* out, int T, int n_head, int n_head_kv,
                                  int head_dim, float scale, const AttnVarlen& vl,
                                  cudaStream_t s) {
    const long long nq = (long long)n_head * head_dim, nk = (long long)n_head_kv * head_dim;
    return launch_attn<false>(q, nq, head_dim, k, nk, vt, ldvt, vt_cols, out, T, n_head,
                              n_head_kv, head_dim, scale, vl, s);
}

cudaError_t launch_attn_tc_f32(const float* q, long long ldq, int q_head_stride, const float* k,
                               long long ldk, const float* vt, long long ldvt, long long vt_cols,
                               float* out, int T, int n_head, int n_head_kv, int head_dim,
                               float scale, const AttnVarlen& vl, cudaStream_t s) {
    return launch_attn<true>(q, ldq, q_head_stride, k, ldk, vt, ldvt, vt_cols, out, T, n_head,
                             n_head_kv, head_dim, scale, vl, s);
}

}  // namespace dtp
