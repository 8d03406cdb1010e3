// prefill_bf16.cu -- 16-bit (bf16, or fp16 with the F16 flag) attention
// forward on tcgen05 tensor cores (sm_103a), dense [B, H, S, D] problems or
// packed variable-length sequences (the VARLEN flag).
//
// Computes the tiled online-softmax recurrence of "gfx942 unified attention,
// from the math up", section 3 (running max m, denominator l, rescale
// alpha = 2^(m_old - m_new) in base 2, final o / l) for the operation of
// attention.fkc.md, attention_naive: scale, softcap, ALiBi, causal / window /
// per-row mask, GQA, fully-masked row -> zeros.
//
// Structure (one persistent CTA per SM, 16 warps in four warpgroups):
//   WG0 (warps 0-3)    softmax for query slot 0: thread r owns query row r,
//                      which is TMEM lane r of the slot's S and O tiles
//   WG1 (warps 4-7)    softmax for query slot 1
//   WG2 (warps 8-11)   epilogue for both slots: O / l -> 16-bit rows, lse
//   WG3 warp 12        TMA producer: decodes each work item once and publishes
//                      it to the other roles, loads Q tiles once per item and
//                      K/V tiles through an NS-stage shared-memory ring
//                      (128-byte swizzle)
//   WG3 warp 13        MMA issuer (the whole warp runs the loop, one elected
//                      lane issues): S = Q K^T with both operands in shared
//                      memory, O += P V with P in TMEM and V in shared memory,
//                      fp32 accumulators in TMEM
//   WG3 warps 14-15    idle
// Registers move to the softmax warpgroups with setmaxnreg:
// 2 x 128 x SOFTMAX_REGS + 128 x (EPI_REGS + CONTROL_REGS) <= 512 x LAUNCH_REGS,
// and the host refuses to launch if the compiled launch allocation is smaller.
//
// Two query slots ping-pong on the tensor core: while softmax works on one
// slot's scores, the MMA thread runs the other slot's P V and next Q K^T.  A
// work item is two 128-row query tiles that share one K/V stream: two heads of
// one GQA group at the same rows (Hq / Hkv even), or two consecutive row tiles
// of one head (otherwise).  Items are dealt to CTAs heaviest first in a
// boustrophedon order, so causal work evens out across SMs.
//
// TMEM columns (512 allocated): S/P of slot x at 128 x, O of slot x at
// 256 + D x.  P (16-bit, two per 32-bit column) overwrites the first 64 columns of
// its S tile; the next Q K^T into that tile is issued after the P V that reads
// it, and tcgen05 operations issued by one thread execute in order.
//
// Causal and window tile skipping ("gfx942 unified attention", section 4): a
// slot visits only the key tiles that intersect the union of its rows'
// admissible ranges, the last tile first with ALiBi and the first tile first
// otherwise; element masks are applied only on tiles that cut a row's range.  Lazy rescaling: O and l are rescaled only when the running max grows
// by more than 8 (base-2 units); otherwise the stale max stays the reference,
// which keeps every p <= 2^8 and leaves o / l exact.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int BM = 128;  // query rows per slot
constexpr int BN = 128;  // keys per K/V tile
constexpr int NUM_WARPS = 16;
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int WARP_PRODUCER = 12;
constexpr int WARP_MMA = 13;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float RESCALE_THRESHOLD = 8.0f;  // base-2 units
constexpr int LAUNCH_REGS = 128;          // 65536 / 512
// K/V tiles move through the shared-memory slots in the order the MMA thread
// reads them: per item K_first, then (V_u, K_next) for each tile u but the
// last, V_last last (first_tile / last_tile below give the order).
// Each of these groups is one MMA step and has one full barrier (the TMA
// transaction count of its one or two tiles) and one empty barrier (one
// commit after the step's MMAs), so a step costs the MMA thread one wait and
// one commit.  NG group barriers cycle; a slot is refilled only after the
// group that last used it was released, at most NS groups back, so NG >= NS.
constexpr int NG = 8;
// Work items are decoded once, by the producer warp, and published through a
// ring of NI entries in shared memory (one full and one empty barrier each);
// every thread of the MMA warp, the softmax and the epilogue warpgroups
// releases an entry after copying it.
constexpr int NI = 4;
constexpr int ITEM_READERS = 32 + 2 * 128 + 128;
// K + V bytes of the packed sequences whose items run together: about a fifth
// of the 126 MB L2, so that a band's K and V survive the Q and O streams that
// pass through L2 between two reads of the same key tile (on GB300, 24 MB bands
// beat 16 and 48 MB ones on packed-sequence prefill).  Dense problems run as
// one band: banding them measured 5-7 % slower (heaviest-first over the whole
// list balances the SMs better, and their K / V re-reads cost little time).
constexpr double L2_BAND_BYTES = 24.0 * 1024 * 1024;

template <int D>
struct Cfg {
    static constexpr int HALVES = D / 64;             // 128-byte swizzle slabs per row
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int Q_SLAB = BM * 128;           // bytes of one 64-column slab of a Q tile
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int KV_SLAB = BN * 128;
    static constexpr int NS = (D == 128) ? 4 : 6;     // K/V ring stages
    static constexpr int STAGE_O = BM * 128;          // output staging: 128 rows x 64 columns bf16
    static constexpr int SMEM_BYTES = 2 * Q_BYTES + NS * KV_BYTES + STAGE_O + 1024;  // + alignment slack
    static constexpr int O_COL = 256;
    // setmaxnreg budgets per warpgroup (multiples of 8); this split leaves ptxas
    // spilling at most a few bytes in any variant, the 184/64/80 split spilled
    // the epilogue and control loops
    static constexpr int SOFTMAX_REGS = 176;
    static constexpr int EPI_REGS = 80;
    static constexpr int CONTROL_REGS = 80;
    static_assert(2 * 128 * SOFTMAX_REGS + 128 * EPI_REGS + 128 * CONTROL_REGS <= NUM_THREADS * LAUNCH_REGS,
                  "register split");
};

struct Params {
    uint16_t* out;     // bf16 or fp16 bits
    float* lse;
    const float* slopes;
    const int2* rowb;
    unsigned int* status;
    unsigned long long timeout_ns;
    int B, Hq, Hkv, Sq, Sk, G;
    int causal, wl, wr;
    float scale_log2;  // softmax_scale * log2(e)
    float cap_in;      // softmax_scale / softcap
    float cap_out;     // softcap * log2(e)
    int n_qt;          // query tiles per head (packed sequences: per sequence, at most)
    int pair_heads;    // 1: slots are heads (2p, 2p+1) at one row tile; 0: row tiles (2t, 2t+1) of one head
    int band;          // sequences per band: work items run band by band (all of B for dense problems)
    int n_items;
    // Packed variable-length sequences ("gfx942 unified attention", sections
    // 4-5): q / out [total_q, Hq, D], k / v [total_k, Hkv, D]; sequence b's
    // queries are rows cu_q[b] .. cu_q[b+1]-1, its live keys the first
    // used_k[b] (or all) of rows cu_k[b] .. cu_k[b+1]-1; positions are aligned
    // bottom-right (query i sits at k_len - q_len + i).
    int varlen;
    const int* cu_q;
    const int* cu_k;
    const int* used_k;
    int total_q, total_k;
};

struct Slot {
    int b, h, t;     // t < 0: slot unused in this item
    int lo, hi;      // key-tile range, lo > hi: no admissible key for any row
    int q0, q_len;   // the sequence's first query row (packed layout) and its queries
    int k0, k_len;   // its first key row (packed layout) and its live keys
};

// Position of query row i of a slot's sequence: i (dense problems, top-left)
// or k_len - q_len + i (packed sequences, bottom-right).
template <bool VARLEN>
__device__ __forceinline__ int query_pos(const Slot& s, int i) {
    return VARLEN ? s.k_len - s.q_len + i : i;
}
// Queries and keys of the slot's sequence.
template <bool VARLEN>
__device__ __forceinline__ int seq_q_len(const Params& p, const Slot& s) { return VARLEN ? s.q_len : p.Sq; }
template <bool VARLEN>
__device__ __forceinline__ int seq_k_len(const Params& p, const Slot& s) { return VARLEN ? s.k_len : p.Sk; }

// Admissible key interval [a, e] of query row i of the slot's sequence (a > e when empty).
template <bool VARLEN>
__device__ __forceinline__ void row_interval(const Params& p, const Slot& s, int i, int& a, int& e) {
    const int pos = query_pos<VARLEN>(s, i);
    a = 0;
    e = seq_k_len<VARLEN>(p, s) - 1;
    if (p.causal) e = min(e, pos);
    if (p.wl >= 0) a = max(a, pos - p.wl);
    if (p.wr >= 0) e = min(e, pos + p.wr);
    if (p.rowb) {
        int2 r = __ldg(p.rowb + (size_t)s.b * p.Sq + i);
        a = max(a, r.x);
        e = min(e, r.y);
    }
}

// Item -> (b, h, t) of both slots, the sequence's geometry, and each slot's
// key-tile range.  Called by a whole warp (the range is a warp reduction over
// the slot's rows).  Returns false when neither slot has a query tile (a row
// tile past a packed sequence's end).
template <bool VARLEN>
__device__ __forceinline__ bool decode_item(const Params& p, int item, Slot (&s)[2]) {
    const int lane = threadIdx.x & 31;
    // Items run band by band (p.band sequences each, so a band's K and V stay
    // in L2 while its items run), heaviest row tiles first within a band.
    const int hp = p.pair_heads ? p.Hq / 2 : p.Hq;         // slot pairs per (sequence, row rank)
    const int n_r = p.pair_heads ? p.n_qt : (p.n_qt + 1) / 2;  // row ranks
    const int per_band = n_r * p.band * hp;
    const int band = item / per_band, w = item % per_band;
    const int tr = w / (p.band * hp), rest = w % (p.band * hp);
    const int b = band * p.band + rest / hp, pr = rest % hp;
    if (b >= p.B) return false;
    if (p.pair_heads) {
        int t = p.causal ? (p.n_qt - 1 - tr) : tr;
        s[0] = Slot{b, 2 * pr, t, 0, -1, 0, p.Sq, 0, p.Sk};
        s[1] = Slot{b, 2 * pr + 1, t, 0, -1, 0, p.Sq, 0, p.Sk};
    } else {
        int tp = p.causal ? (n_r - 1 - tr) : tr;
        s[0] = Slot{b, pr, 2 * tp, 0, -1, 0, p.Sq, 0, p.Sk};
        s[1] = Slot{b, pr, (2 * tp + 1 < p.n_qt) ? 2 * tp + 1 : -1, 0, -1, 0, p.Sq, 0, p.Sk};
    }
    if (VARLEN) {
        // the sequence's rows; offsets or lengths outside the tensors are
        // clamped and reported in the status word
        const int b = s[0].b;
        int q0 = __ldg(p.cu_q + b), q1 = __ldg(p.cu_q + b + 1);
        int k0 = __ldg(p.cu_k + b), k1 = __ldg(p.cu_k + b + 1);
        int kl = p.used_k ? __ldg(p.used_k + b) : k1 - k0;
        bool bad = q0 < 0 || q1 < q0 || q1 > p.total_q || k0 < 0 || k1 < k0 || k1 > p.total_k || kl < 0 ||
                   kl > k1 - k0 || q1 - q0 > p.n_qt * BM;
        if (bad) {
            q0 = min(max(q0, 0), p.total_q);
            q1 = min(max(q1, q0), min(p.total_q, q0 + p.n_qt * BM));
            k0 = min(max(k0, 0), p.total_k);
            k1 = min(max(k1, k0), p.total_k);
            kl = min(max(kl, 0), k1 - k0);
            if (lane == 0) atomicOr(p.status, ST_PREFILL_VARLEN_RANGE);
        }
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            s[x].q0 = q0;
            s[x].q_len = q1 - q0;
            s[x].k0 = k0;
            s[x].k_len = kl;
            if (s[x].t * BM >= s[x].q_len) s[x].t = -1;
        }
    }
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        if (s[x].t < 0) continue;
        int kmin = 0x7fffffff, kmax = -1;
        const int q0 = s[x].t * BM;
        for (int r = lane; r < BM; r += 32) {
            int qi = q0 + r;
            if (qi >= seq_q_len<VARLEN>(p, s[x])) break;
            int a, e;
            row_interval<VARLEN>(p, s[x], qi, a, e);
            if (a <= e) {
                kmin = min(kmin, a);
                kmax = max(kmax, e);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
            kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
        }
        if (kmin <= kmax) {
            s[x].lo = kmin / BN;
            s[x].hi = kmax / BN;
        }
    }
    return s[0].t >= 0 || s[1].t >= 0;
}

// Column indices (j, j + 1) of the key pairs of a tile, for the packed ALiBi bias.
__constant__ float2 c_key_pairs[BN / 2] = {
#define GBATTN_KP(i) {2.f * (i), 2.f * (i) + 1.f}
    GBATTN_KP(0),  GBATTN_KP(1),  GBATTN_KP(2),  GBATTN_KP(3),  GBATTN_KP(4),  GBATTN_KP(5),  GBATTN_KP(6),
    GBATTN_KP(7),  GBATTN_KP(8),  GBATTN_KP(9),  GBATTN_KP(10), GBATTN_KP(11), GBATTN_KP(12), GBATTN_KP(13),
    GBATTN_KP(14), GBATTN_KP(15), GBATTN_KP(16), GBATTN_KP(17), GBATTN_KP(18), GBATTN_KP(19), GBATTN_KP(20),
    GBATTN_KP(21), GBATTN_KP(22), GBATTN_KP(23), GBATTN_KP(24), GBATTN_KP(25), GBATTN_KP(26), GBATTN_KP(27),
    GBATTN_KP(28), GBATTN_KP(29), GBATTN_KP(30), GBATTN_KP(31), GBATTN_KP(32), GBATTN_KP(33), GBATTN_KP(34),
    GBATTN_KP(35), GBATTN_KP(36), GBATTN_KP(37), GBATTN_KP(38), GBATTN_KP(39), GBATTN_KP(40), GBATTN_KP(41),
    GBATTN_KP(42), GBATTN_KP(43), GBATTN_KP(44), GBATTN_KP(45), GBATTN_KP(46), GBATTN_KP(47), GBATTN_KP(48),
    GBATTN_KP(49), GBATTN_KP(50), GBATTN_KP(51), GBATTN_KP(52), GBATTN_KP(53), GBATTN_KP(54), GBATTN_KP(55),
    GBATTN_KP(56), GBATTN_KP(57), GBATTN_KP(58), GBATTN_KP(59), GBATTN_KP(60), GBATTN_KP(61), GBATTN_KP(62),
    GBATTN_KP(63)};
#undef GBATTN_KP

__device__ __forceinline__ int item_of(int k, int cta, int grid) {
    return k * grid + ((k & 1) ? (grid - 1 - cta) : cta);
}

__device__ __forceinline__ bool slot_live(const Slot& s) { return s.t >= 0 && s.lo <= s.hi; }

// Order of a slot's key tiles: from the last one down (DOWN) or from the
// first one up.  The recurrence's order is free.  With ALiBi the largest
// scores sit at the diagonal, so visiting it first settles the running max at
// once (no rescales); otherwise an item starts on an unmasked tile, whose
// softmax is the short one, and the masked diagonal tile comes last.
template <bool DOWN>
__device__ __forceinline__ int first_tile(const Slot& s) { return DOWN ? s.hi : s.lo; }
template <bool DOWN>
__device__ __forceinline__ int last_tile(const Slot& s) { return DOWN ? s.lo : s.hi; }
__device__ __forceinline__ bool in_range(const Slot& s, int u) { return s.t >= 0 && u >= s.lo && u <= s.hi; }

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct Smem {
    uint64_t q_full[2], q_empty[2];
    uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
    // l_full[e][x]: entry e of slot x's (l, m) hand-off is written.  One barrier
    // per entry: a slot whose next item has a single key tile finishes that
    // item's softmax without waiting for any P V, so it can publish item n + 1
    // before the epilogue has waited for item n; with one barrier per slot the
    // barrier would then be two phases ahead of the epilogue's parity wait.
    uint64_t l_full[2][2];
    uint64_t grp_full[NG], grp_empty[NG];  // one per step group of K/V tiles
    uint64_t item_full[NI], item_empty[NI];
    uint64_t drain;
    Slot item_slot[NI][2];
    int item_end[NI];       // 1: no item left (the ring's last entry)
    float l_buf[2][2][BM];  // [item parity][slot][row]: softmax denominator l
    float m_buf[2][2][BM];  // running max (base 2) for lse
    uint32_t tmem_base;
    int abort_flag;
};

// The k-th work item of this CTA as published by the producer warp.  Returns
// 1 with the item's slots, 0 when no item is left, -1 if the wait gave up.
// The entry is released as soon as it is copied.
__device__ __forceinline__ int read_item(Smem& sm, int k, const WaitCtl& wc, uint32_t site, Slot (&s)[2]) {
    const int i = k % NI;
    if (!mbar_wait(&sm.item_full[i], (uint32_t)(k / NI) & 1u, wc, site)) return -1;
    const int end = sm.item_end[i];
    s[0] = sm.item_slot[i][0];
    s[1] = sm.item_slot[i][1];
    mbar_arrive(&sm.item_empty[i]);
    return end ? 0 : 1;
}

// ---------------------------------------------------------------------------- softmax role
template <int D, bool SOFTCAP, bool ALIBI, bool VARLEN, bool F16>
__device__ __forceinline__ void softmax_role(const Params& p, Smem& sm, uint32_t tmem, const WaitCtl& wc,
                                             int warp) {
    using C = Cfg<D>;
    const int x = warp >> 2;
    const int r = threadIdx.x & (BM - 1);
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + 128u * x;
    const uint32_t tO = tmem + lane_off + C::O_COL + D * x;
    uint32_t s_cnt = 0, l_cnt = 0;
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    for (int k = 0;; ++k) {
        Slot s[2];
        const int got = read_item(sm, k, wc, ST_PREFILL_SOFTMAX, s);
        if (!__all_sync(0xffffffffu, got >= 0)) return;
        if (got == 0) break;
        const Slot sl = s[x];
        if (!slot_live(sl)) continue;  // unused or fully-masked tile: the epilogue writes zeros
        const int i_row = sl.t * BM + r;            // query row within the sequence
        const int qi = query_pos<VARLEN>(sl, i_row);  // its position (ALiBi)
        int ra = 1, rb = 0;
        if (i_row < seq_q_len<VARLEN>(p, sl)) row_interval<VARLEN>(p, sl, i_row, ra, rb);
        float slope_l2 = 0.f;
        if (ALIBI) slope_l2 = __ldg(p.slopes + sl.h) * LOG2E;
        // A row with no admissible key (or past the sequence) takes +inf as its
        // reference max: every p of the row is then exactly 0 (l = 0, O = 0)
        // without masking its elements on each tile.
        const bool row_live = ra <= rb;
        float m_used = row_live ? -INFINITY : INFINITY, l = 0.f;
        constexpr bool DOWN = ALIBI;
        for (int u = first_tile<DOWN>(sl);; u += DOWN ? -1 : 1) {
            if (DOWN ? u < sl.lo : u > sl.hi) break;
            const bool ok = mbar_wait(&sm.s_full[x], s_cnt & 1, wc, ST_PREFILL_SOFTMAX);
            ++s_cnt;
            if (!__all_sync(0xffffffffu, ok)) return;
            tc_fence_after();
            float sv[BN];
            tmem_ld64_async(tS, &sv[0]);
            tmem_ld64_async(tS + 64, &sv[64]);
            tmem_wait_ld128(sv);
            const int k0 = u * BN;
            if (SOFTCAP || ALIBI) {
                // base-2 logits: cap * tanh(scale s / cap) [+ slope (kj - qi)], times log2(e).
                // tanh is the hardware approximation (relative error about 2^-11,
                // far below the bf16 rounding of P); the ALiBi bias of key k0 + j is
                // base + slope * j with one conversion per tile.
                // Column pairs go through packed FP32 operations; the bias of keys
                // (j, j + 1) is one FFMA2 against their indices in constant memory.
                const float abase = ALIBI ? slope_l2 * (float)(k0 - qi) : 0.f;
                const float2 ab2 = make_float2(abase, abase), sl2b = make_float2(slope_l2, slope_l2);
                const float2 ci2 = make_float2(p.cap_in, p.cap_in), co2 = make_float2(p.cap_out, p.cap_out);
#pragma unroll
                for (int j = 0; j < BN; j += 2) {
                    float2 t = make_float2(sv[j], sv[j + 1]);
                    if (SOFTCAP) {
                        t = __fmul2_rn(t, ci2);
                        t = make_float2(tanh_approx(t.x), tanh_approx(t.y));
                        t = ALIBI ? __ffma2_rn(t, co2, __ffma2_rn(sl2b, c_key_pairs[j >> 1], ab2)) : __fmul2_rn(t, co2);
                    } else {
                        t = __ffma2_rn(t, sl2, __ffma2_rn(sl2b, c_key_pairs[j >> 1], ab2));
                    }
                    sv[j] = t.x;
                    sv[j + 1] = t.y;
                }
            }
            // admissible keys of the tile: lo <= j <= hi; rows with none are
            // not masked (their reference max is +inf).  With no lower bound in
            // the tile for any live row of the warp (causal masks) one compare
            // per key suffices.  The vote is taken by the whole warp, before the
            // per-row branch.
            const int lo = ra - k0, hi = rb - k0;
            const bool no_lower = __all_sync(0xffffffffu, !row_live || lo <= 0);
            if (row_live && (k0 < ra || k0 + BN - 1 > rb)) {
                if (no_lower) {
#pragma unroll
                    for (int j = 0; j < BN; ++j) sv[j] = (j > hi) ? -INFINITY : sv[j];
                } else {
#pragma unroll
                    for (int j = 0; j < BN; ++j) sv[j] = (j < lo || j > hi) ? -INFINITY : sv[j];
                }
            }
            // row max over the tile: 8 independent chains of three-input max
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = max3(sv[i], sv[8 + i], sv[16 + i]);
#pragma unroll
            for (int j = 24; j + 16 <= BN; j += 16) {
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = max3(mx[i], sv[j + i], sv[j + 8 + i]);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], sv[BN - 8 + i]);
            float m_tile = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
            if (!(SOFTCAP || ALIBI)) m_tile *= p.scale_log2;  // scale > 0: max commutes with scaling
            const float m_new = fmaxf(m_used, m_tile);
            float alpha = 1.f;
            if (m_new > m_used + RESCALE_THRESHOLD) {
                if (m_used != -INFINITY) alpha = ex2_approx(m_used - m_new);
                m_used = m_new;
            }
            const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
            const float2 nm = make_float2(-m_ref, -m_ref);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
            uint32_t pw[BN / 2];
#pragma unroll
            for (int j = 0; j < BN; j += 2) {
                float2 y = make_float2(sv[j], sv[j + 1]);
                y = (SOFTCAP || ALIBI) ? __fadd2_rn(y, nm) : __ffma2_rn(y, sl2, nm);
                const float2 pp = make_float2(ex2_approx(y.x), ex2_approx(y.y));
                acc[(j >> 1) & 3] = __fadd2_rn(acc[(j >> 1) & 3], pp);
                pw[j >> 1] = pack16x2<F16>(pp.x, pp.y);
            }
            const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
            const float2 a = __fadd2_rn(a01, a23);
            l = fmaf(l, alpha, a.x + a.y);
            tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pw[0]));
            tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pw[32]));
            // Rescale O when any row of the warp moved its reference max.  The
            // P V of the previous tile has completed: it was issued before this
            // tile's Q K^T, whose completion we waited for.
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    float ov[32];
                    tmem_ld32(tO + c, ov);
                    uint32_t w[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(ov[i] * alpha);
                    tmem_st32(tO + c, w);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&sm.p_full[x]);
        }
        // hand l and the reference max to the epilogue
        const int par = l_cnt & 1;
        sm.l_buf[par][x][r] = l;
        sm.m_buf[par][x][r] = m_used;
        ++l_cnt;
        mbar_arrive(&sm.l_full[par][x]);
    }
}

// ---------------------------------------------------------------------------- epilogue role
template <int D, bool VARLEN, bool F16>
__device__ __forceinline__ void epilogue_role(const Params& p, Smem& sm, uint32_t tmem, const WaitCtl& wc,
                                              int warp, uint8_t* stage, const CUtensorMap* tmO) {
    // Output rows go through a 128-row x 64-column bf16 staging tile in shared
    // memory (128-byte swizzle: thread r writes row r without bank conflicts)
    // and leave by TMA tensor stores, which write whole lines and clip the rows
    // past Sq.  One elected thread issues the stores and waits for their reads
    // of the staging tile before it is refilled.
    using C = Cfg<D>;
    const int r = threadIdx.x & (BM - 1);
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool issuer = (threadIdx.x & (BM - 1)) == 0;
    uint8_t* srow = stage + r * 128;
    uint32_t cnt[2] = {0, 0};
    for (int k = 0;; ++k) {
        Slot s[2];
        const int got = read_item(sm, k, wc, ST_PREFILL_EPILOGUE, s);
        if (!__all_sync(0xffffffffu, got >= 0)) return;
        if (got == 0) break;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const Slot sl = s[x];
            if (sl.t < 0) continue;
            const int qi = sl.t * BM + r;  // query row within the sequence
            const bool live = qi < seq_q_len<VARLEN>(p, sl);
            // output row of this thread and its lse entry: dense [B, Hq, Sq, D] and
            // [B, Hq, Sq], or packed [total_q, Hq, D] and [Hq, total_q]
            const size_t orow = VARLEN ? (size_t)(sl.q0 + qi) * p.Hq + sl.h : ((size_t)sl.b * p.Hq + sl.h) * p.Sq + qi;
            const size_t lrow = VARLEN ? (size_t)sl.h * p.total_q + sl.q0 + qi : orow;
            // a packed tile that ends inside its sequence is written row by row: a
            // tensor store would also write the next sequence's rows
            const bool ragged = VARLEN && sl.t * BM + BM > sl.q_len;
            if (sl.lo > sl.hi) {
                // No admissible key for any row of the tile: zero rows.
                if (live) {
                    uint4* dst = reinterpret_cast<uint4*>(p.out + orow * D);
#pragma unroll
                    for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
                    if (p.lse) p.lse[lrow] = -INFINITY;
                }
                continue;
            }
            const int par = cnt[x] & 1;
            bool ok = mbar_wait(&sm.l_full[par][x], (cnt[x] >> 1) & 1, wc, ST_PREFILL_EPILOGUE);
            ok = ok && mbar_wait(&sm.o_full[x], cnt[x] & 1, wc, ST_PREFILL_EPILOGUE);
            ++cnt[x];
            if (!__all_sync(0xffffffffu, ok)) return;
            tc_fence_after();
            const float l = sm.l_buf[par][x][r];
            const float m = sm.m_buf[par][x][r];
            const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
            const uint32_t tO = tmem + lane_off + C::O_COL + D * x;
#pragma unroll
            for (int hf = 0; hf < C::HALVES; ++hf) {
                // the staging tile is free once the previous store has read it
                if (!ragged) {
                    if (issuer) bulk_wait_group_read0();
                    asm volatile("bar.sync 1, %0;" ::"n"(BM) : "memory");
                }
#pragma unroll
                for (int c32 = 0; c32 < 2; ++c32) {
                    float ov[32];
                    tmem_ld32(tO + hf * 64 + c32 * 32, ov);
                    if (hf == C::HALVES - 1 && c32 == 1) {
                        // all of O_x has been read: the next item may overwrite it
                        tc_fence_before();
                        mbar_arrive(&sm.o_empty[x]);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int c = c32 * 4 + i;  // 16-byte chunk of the 128-byte staging row
                        uint4 w;
                        w.x = pack16x2<F16>(ov[8 * i + 0] * inv_l, ov[8 * i + 1] * inv_l);
                        w.y = pack16x2<F16>(ov[8 * i + 2] * inv_l, ov[8 * i + 3] * inv_l);
                        w.z = pack16x2<F16>(ov[8 * i + 4] * inv_l, ov[8 * i + 5] * inv_l);
                        w.w = pack16x2<F16>(ov[8 * i + 6] * inv_l, ov[8 * i + 7] * inv_l);
                        if (ragged) {
                            if (live) reinterpret_cast<uint4*>(p.out + orow * D + hf * 64)[c] = w;
                        } else {
                            *reinterpret_cast<uint4*>(srow + ((c ^ (r & 7)) << 4)) = w;
                        }
                    }
                }
                if (!ragged) {
                    fence_proxy_async_smem();
                    asm volatile("bar.sync 1, %0;" ::"n"(BM) : "memory");
                    if (issuer) {
                        if (VARLEN)
                            tma_store_3d(tmO, stage, hf * 64, sl.h, sl.q0 + sl.t * BM);
                        else
                            tma_store_3d(tmO, stage, hf * 64, sl.t * BM, sl.b * p.Hq + sl.h);
                        bulk_commit_group();
                    }
                }
            }
            if (live && p.lse) p.lse[lrow] = (l > 0.f) ? (m + log2f(l)) * LN2 : -INFINITY;
        }
    }
    if (issuer) bulk_wait_group0();
}

template <int D, bool SOFTCAP, bool ALIBI, bool VARLEN, bool F16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                        const Params p) {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t dyn_smem[];
    __shared__ Smem sm;

    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ[2] = {base, base + C::Q_BYTES};
    uint8_t* sKV = base + 2 * C::Q_BYTES;
    uint8_t* sStage = sKV + C::NS * C::KV_BYTES;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            mbar_init(&sm.q_full[x], 1);
            mbar_init(&sm.q_empty[x], 1);
            mbar_init(&sm.s_full[x], 1);
            mbar_init(&sm.p_full[x], BM);
            mbar_init(&sm.o_full[x], 1);
            mbar_init(&sm.o_empty[x], BM);
            mbar_init(&sm.l_full[0][x], BM);
            mbar_init(&sm.l_full[1][x], BM);
        }
        for (int i = 0; i < NG; ++i) {
            mbar_init(&sm.grp_full[i], 1);
            mbar_init(&sm.grp_empty[i], 1);
        }
        for (int i = 0; i < NI; ++i) {
            mbar_init(&sm.item_full[i], 1);
            mbar_init(&sm.item_empty[i], ITEM_READERS);
        }
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_PRODUCER) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    WaitCtl wc{&sm.abort_flag, p.status, p.timeout_ns};
    const int grid = gridDim.x, cta = blockIdx.x;

    // Each warpgroup executes one setmaxnreg, at one program point, before its roles split.
    if (warp < 8) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::SOFTMAX_REGS));
        softmax_role<D, SOFTCAP, ALIBI, VARLEN, F16>(p, sm, tmem, wc, warp);
    } else if (warp < 12) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::EPI_REGS));
        epilogue_role<D, VARLEN, F16>(p, sm, tmem, wc, warp, sStage, &tmO);
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::CONTROL_REGS));
        if (warp == WARP_PRODUCER) {
            // -------------------------------------------------------- TMA producer
            if (lane == 0) {
                tma_prefetch_desc(&tmQ);
                tma_prefetch_desc(&tmK);
                tma_prefetch_desc(&tmV);
            }
            uint32_t ld_cnt = 0, grp_cnt = 0, q_cnt[2] = {0, 0};
            // L2 policies of packed sequences: Q read once, K / V read again by the band's other items
            const uint64_t pol_first = createpolicy_evict_first(), pol_last = createpolicy_evict_last();
            int slot_grp[C::NS];  // group that last filled each slot (-1: none)
#pragma unroll
            for (int i = 0; i < C::NS; ++i) slot_grp[i] = -1;
            bool ok = true;
            int pk = 0;  // items published so far (row tiles past a packed sequence's end are skipped)
            for (int k = 0;; ++k) {
                const int item = item_of(k, cta, grid);
                const bool more = item < p.n_items;
                Slot s[2];
                if (more && !decode_item<VARLEN>(p, item, s)) continue;
                {
                    // publish the item (or the end of the list) to the other roles
                    const int i = pk % NI;
                    const bool free_entry =
                        pk < NI || mbar_wait(&sm.item_empty[i], (uint32_t)(pk / NI - 1) & 1u, wc, ST_PREFILL_PRODUCER);
                    ++pk;
                    if (!__all_sync(0xffffffffu, free_entry)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        if (more) {
                            sm.item_slot[i][0] = s[0];
                            sm.item_slot[i][1] = s[1];
                        }
                        sm.item_end[i] = more ? 0 : 1;
                        mbar_arrive(&sm.item_full[i]);
                    }
                }
                if (!more) break;
                if (lane == 0) {
                    const int hkv = s[0].h / p.G;
#pragma unroll
                    for (int x = 0; x < 2 && ok; ++x) {
                        if (!slot_live(s[x])) continue;
                        ok = mbar_wait(&sm.q_empty[x], (q_cnt[x] & 1) ^ 1, wc, ST_PREFILL_PRODUCER);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&sm.q_full[x], C::Q_BYTES);
#pragma unroll
                        for (int hf = 0; hf < C::HALVES; ++hf) {
                            if (VARLEN)  // packed [total_q][Hq][D]; each Q tile is read once
                                tma_load_3d_hint(sQ[x] + hf * C::Q_SLAB, &tmQ, &sm.q_full[x], hf * 64, s[x].h,
                                                 s[x].q0 + s[x].t * BM, pol_first);
                            else
                                tma_load_3d(sQ[x] + hf * C::Q_SLAB, &tmQ, &sm.q_full[x], hf * 64, s[x].t * BM,
                                            s[x].b * p.Hq + s[x].h);
                        }
                        ++q_cnt[x];
                    }
                    int ulo = 0x7fffffff, uhi = -1;
#pragma unroll
                    for (int x = 0; x < 2; ++x)
                        if (slot_live(s[x])) {
                            ulo = min(ulo, s[x].lo);
                            uhi = max(uhi, s[x].hi);
                        }
                    // Key tiles in the order first_tile / last_tile give (down from
                    // uhi with ALiBi, else up from ulo); groups: (K_first), then
                    // (V_u, K_next) for every tile u but the last, then (V_last)
                    constexpr bool DOWN = ALIBI;
                    const int nt = uhi - ulo + 1;
                    for (int i = -1; i < nt && ok; ++i) {
                        const int u = DOWN ? uhi - i : ulo + i;  // V tile of this group
                        const int un = DOWN ? u - 1 : u + 1;     // its K tile
                        const bool has_v = i >= 0, has_k = i < nt - 1;
                        const int nl = (has_v ? 1 : 0) + (has_k ? 1 : 0);
                        // both slots must have been released by the groups that last used them
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            if (i >= nl) break;
                            const int g_prev = slot_grp[(ld_cnt + i) % C::NS];
                            if (g_prev >= 0)
                                ok = ok && mbar_wait(&sm.grp_empty[g_prev % NG], (g_prev / NG) & 1, wc,
                                                     ST_PREFILL_PRODUCER);
                        }
                        if (!ok) break;
                        uint64_t* fb = &sm.grp_full[grp_cnt % NG];
                        mbar_arrive_expect_tx(fb, nl * C::KV_BYTES);
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            if (i >= nl) break;
                            const bool is_v = has_v && i == 0;
                            const int st = (ld_cnt + i) % C::NS;
                            uint8_t* dst = sKV + st * C::KV_BYTES;
                            const int key = (is_v ? u : un) * BN;
#pragma unroll
                            for (int hf = 0; hf < C::HALVES; ++hf) {
                                if (VARLEN)  // packed [total_k][Hkv][D]; the band's other items read it again
                                    tma_load_3d_hint(dst + hf * C::KV_SLAB, is_v ? &tmV : &tmK, fb, hf * 64, hkv,
                                                     s[0].k0 + key, pol_last);
                                else
                                    tma_load_3d(dst + hf * C::KV_SLAB, is_v ? &tmV : &tmK, fb, hf * 64, key,
                                                s[0].b * p.Hkv + hkv);
                            }
                            slot_grp[st] = (int)grp_cnt;
                        }
                        ld_cnt += nl;
                        ++grp_cnt;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
            }
            if (!ok && lane == 0) {
                // Let the copies already issued land before the CTA leaves.
                const uint32_t n = grp_cnt < (uint32_t)NG ? grp_cnt : (uint32_t)NG;
                for (uint32_t i = grp_cnt - n; i < grp_cnt; ++i)
                    mbar_drain(&sm.grp_full[i % NG], (i / NG) & 1, 100000000ull);
#pragma unroll
                for (int x = 0; x < 2; ++x)
                    if (q_cnt[x]) mbar_drain(&sm.q_full[x], (q_cnt[x] - 1) & 1, 100000000ull);
            }
        } else if (warp == WARP_MMA) {
            // -------------------------------------------------------- MMA issuer
            // The whole warp runs the loop and one elected lane issues each MMA and
            // commit (warp-collective forms keep the operands in uniform registers;
            // a single thread can issue a tcgen05.mma only every ~40 cycles while an
            // M=128 N=128 K=16 MMA takes 64).  Waits are warp votes, so the warp
            // stays converged.
            auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, wc, ST_PREFILL_MMA));
            };
            constexpr bool DOWN = ALIBI;  // key-tile order, as in the producer and softmax roles
            constexpr uint32_t IDESC_S = F16 ? idesc_f16_f32(BM, BN, 0) : idesc_bf16_f32(BM, BN, 0);
            constexpr uint32_t IDESC_O = F16 ? idesc_f16_f32(BM, D, 1) : idesc_bf16_f32(BM, D, 1);
            uint32_t ld_cnt = 0, grp_cnt = 0, q_cnt[2] = {0, 0}, p_cnt[2] = {0, 0}, o_cnt[2] = {0, 0};
            bool ok = true;
            const uint32_t sQa[2] = {smem_u32(sQ[0]), smem_u32(sQ[1])};
            const uint32_t sKVa = smem_u32(sKV);
            for (int k = 0;; ++k) {
                Slot s[2];
                const int got = read_item(sm, k, wc, ST_PREFILL_MMA, s);
                if (!__all_sync(0xffffffffu, got >= 0)) {
                    ok = false;
                    break;
                }
                if (got == 0) break;
                {
                    int ulo = 0x7fffffff, uhi = -1;
#pragma unroll
                    for (int x = 0; x < 2; ++x)
                        if (slot_live(s[x])) {
                            ulo = min(ulo, s[x].lo);
                            uhi = max(uhi, s[x].hi);
                        }
                    bool q_ready[2] = {false, false};
                    // S_x(ut) = Q_x K_ut^T; after the slot's last tile Q_x is released
                    // at once, so the next item's Q load overlaps this item's tail.
                    auto issue_s = [&](int x, uint32_t kst, int ut) -> bool {
                        if (!q_ready[x]) {
                            if (!wwait(&sm.q_full[x], q_cnt[x] & 1)) return false;
                            ++q_cnt[x];
                            q_ready[x] = true;
                            tc_fence_after();
                        }
                        const uint32_t qlo = sdesc_lo(sQa[x], 16);
                        const uint32_t klo = sdesc_lo(sKVa + kst * C::KV_BYTES, 16);
                        const uint32_t dS = tmem + 128u * x;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = ((kk >> 2) * C::Q_SLAB + (kk & 3) * 32) >> 4;
                            const uint32_t koff = ((kk >> 2) * C::KV_SLAB + (kk & 3) * 32) >> 4;
                            umma_ss_lo_elect(dS, qlo + off, klo + koff, IDESC_S, kk > 0);
                        }
                        umma_commit_elect(&sm.s_full[x]);
                        if (ut == last_tile<DOWN>(s[x])) umma_commit_elect(&sm.q_empty[x]);
                        return true;
                    };
                    if (ulo <= uhi) {
                        const int nt = uhi - ulo + 1;
                        const int ufirst = DOWN ? uhi : ulo;
                        // prologue step: group (K_first)
                        uint32_t gb = grp_cnt % NG;
                        ok = wwait(&sm.grp_full[gb], (grp_cnt / NG) & 1);
                        ++grp_cnt;
                        uint32_t kst = ld_cnt % C::NS;
                        ld_cnt += 1;
#pragma unroll
                        for (int x = 0; x < 2 && ok; ++x)
                            if (in_range(s[x], ufirst)) ok = issue_s(x, kst, ufirst);
                        if (ok) umma_commit_elect(&sm.grp_empty[gb]);
                        for (int i = 0; i < nt && ok; ++i) {
                            // step u: group (V_u, K_next); each slot's P V and next
                            // Q K^T then go to the tensor pipe as one run
                            const int u = DOWN ? uhi - i : ulo + i;
                            const int un = DOWN ? u - 1 : u + 1;
                            const bool has_next = i < nt - 1;
                            gb = grp_cnt % NG;
                            ok = wwait(&sm.grp_full[gb], (grp_cnt / NG) & 1);
                            ++grp_cnt;
                            if (!ok) break;
                            const uint32_t vst = ld_cnt % C::NS;
                            kst = (ld_cnt + 1) % C::NS;
                            ld_cnt += has_next ? 2 : 1;
#pragma unroll
                            for (int x = 0; x < 2 && ok; ++x) {
                                if (in_range(s[x], u)) {
                                    ok = wwait(&sm.p_full[x], p_cnt[x] & 1);
                                    ++p_cnt[x];
                                    if (ok && u == first_tile<DOWN>(s[x])) {
                                        ok = wwait(&sm.o_empty[x], (o_cnt[x] & 1) ^ 1);
                                        ++o_cnt[x];
                                    }
                                    if (!ok) break;
                                    tc_fence_after();
                                    const uint32_t vlo = sdesc_lo(sKVa + vst * C::KV_BYTES, C::KV_SLAB);
                                    const uint32_t dO = tmem + C::O_COL + D * x, aP = tmem + 128u * x;
                                    const uint32_t acc0 = (u != first_tile<DOWN>(s[x])) ? 1u : 0u;
#pragma unroll
                                    for (int kk = 0; kk < BN / 16; ++kk)
                                        umma_ts_lo_elect(dO, aP + 8u * kk, vlo + ((kk * 16 * 128) >> 4), IDESC_O,
                                                         kk > 0 ? 1u : acc0);
                                    if (u == last_tile<DOWN>(s[x])) umma_commit_elect(&sm.o_full[x]);
                                }
                                if (has_next && in_range(s[x], un)) ok = issue_s(x, kst, un);
                            }
                            if (!ok) break;
                            umma_commit_elect(&sm.grp_empty[gb]);
                        }
                    }
                }
                if (!ok) break;
            }
            if (lane == 0) {
                // Every MMA issued must finish before TMEM is released.
                umma_commit(&sm.drain);
                mbar_drain(&sm.drain, 0, 100000000ull);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == WARP_PRODUCER) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool SOFTCAP, bool ALIBI, bool VARLEN, bool F16>
cudaError_t launch_variant(const Params& prm, int grid, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t stream) {
    auto kern = prefill_bf16_kernel<D, SOFTCAP, ALIBI, VARLEN, F16>;
    const int smem = Cfg<D>::SMEM_BYTES;
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    // The warpgroups' register split must fit in what the launch allocates,
    // or setmaxnreg.inc would wait forever.
    if (fa.numRegs < LAUNCH_REGS) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, NUM_THREADS, smem, stream>>>(tq, tk, tv, to, prm);
    return cudaGetLastError();
}

template <bool VARLEN, bool F16>
cudaError_t launch_flags(const Params& p, int grid, int D, bool cap, bool ali, const CUtensorMap& tq,
                         const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t stream) {
    if (D == 128) {
        if (cap) return ali ? launch_variant<128, true, true, VARLEN, F16>(p, grid, tq, tk, tv, to, stream)
                            : launch_variant<128, true, false, VARLEN, F16>(p, grid, tq, tk, tv, to, stream);
        return ali ? launch_variant<128, false, true, VARLEN, F16>(p, grid, tq, tk, tv, to, stream)
                   : launch_variant<128, false, false, VARLEN, F16>(p, grid, tq, tk, tv, to, stream);
    }
    if (cap) return ali ? launch_variant<64, true, true, VARLEN, F16>(p, grid, tq, tk, tv, to, stream)
                        : launch_variant<64, true, false, VARLEN, F16>(p, grid, tq, tk, tv, to, stream);
    return ali ? launch_variant<64, false, true, VARLEN, F16>(p, grid, tq, tk, tv, to, stream)
               : launch_variant<64, false, false, VARLEN, F16>(p, grid, tq, tk, tv, to, stream);
}

}  // namespace

cudaError_t launch_prefill_bf16(const FwdProblem& f, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t stream) {
    Params p{};
    p.out = static_cast<uint16_t*>(f.out);
    p.lse = f.lse;
    p.slopes = f.slopes;
    p.rowb = reinterpret_cast<const int2*>(f.row_bounds);
    p.status = f.status;
    p.timeout_ns = f.timeout_ns;
    p.B = f.B;
    p.Hq = f.Hq;
    p.Hkv = f.Hkv;
    p.Sq = f.Sq;
    p.Sk = f.Sk;
    p.G = f.Hq / f.Hkv;
    p.causal = f.causal;
    p.wl = f.wl;
    p.wr = f.wr;
    p.scale_log2 = f.scale * LOG2E;
    p.cap_in = f.softcap > 0.f ? f.scale / f.softcap : 0.f;
    p.cap_out = f.softcap * LOG2E;
    p.varlen = f.varlen;
    p.cu_q = f.cu_q;
    p.cu_k = f.cu_k;
    p.used_k = f.used_k;
    p.total_q = f.total_q;
    p.total_k = f.total_k;
    p.n_qt = (f.Sq + BM - 1) / BM;
    p.pair_heads = (p.G % 2 == 0) ? 1 : 0;
    // Packed sequences: bands of sequences whose K and V (at the average length)
    // fill about L2_BAND_BYTES, so that the items running at one time re-read K
    // and V from L2 rather than DRAM.  Dense problems run as one band.
    p.band = f.B;
    if (f.varlen) {
        const double kv_all = (double)f.total_k * f.Hkv * f.D * 2.0 * 2.0;
        const double nb = kv_all > 0 ? L2_BAND_BYTES * f.B / kv_all : f.B;
        p.band = nb < 1.0 ? 1 : (nb > f.B ? f.B : (int)nb);
    }
    const long long n_bands = (f.B + p.band - 1) / p.band;
    const long long n_r = p.pair_heads ? p.n_qt : (p.n_qt + 1) / 2;
    const long long n_items = n_bands * n_r * p.band * (p.pair_heads ? f.Hq / 2 : f.Hq);
    if (n_items > 0x7fffffffLL) return cudaErrorInvalidValue;
    p.n_items = (int)n_items;
    const int grid = p.n_items < f.num_sms ? p.n_items : f.num_sms;
    const bool cap = f.softcap > 0.f, ali = f.slopes != nullptr;
    if (p.varlen)
        return f.f16 ? launch_flags<true, true>(p, grid, f.D, cap, ali, tq, tk, tv, to, stream)
                     : launch_flags<true, false>(p, grid, f.D, cap, ali, tq, tk, tv, to, stream);
    return f.f16 ? launch_flags<false, true>(p, grid, f.D, cap, ali, tq, tk, tv, to, stream)
                 : launch_flags<false, false>(p, grid, f.D, cap, ali, tq, tk, tv, to, stream);
}

}  // namespace gbattn
