// prefill_bf16.cu -- bf16 attention forward on tcgen05 tensor cores (sm_103a).
//
// Computes the tiled online-softmax recurrence of "gfx942 unified attention,
// from the math up", section 3 (running max m, denominator l, rescale
// alpha = 2^(m_old - m_new) in base 2, final o / l) for the operation of
// attention.fkc.md, attention_naive: scale, softcap, ALiBi, causal / window /
// per-row mask, GQA, fully-masked row -> zeros.
//
// Structure (one persistent CTA per SM, 12 warps in three warpgroups):
//   warps 0-3  softmax for query slot 0 (thread r owns query row r = TMEM lane r)
//   warps 4-7  softmax for query slot 1
//   warp  8    TMA producer: Q tiles once per item, K/V tiles through an
//              NS-stage shared-memory ring (128-byte swizzle)
//   warp  9    MMA issuer (one thread): S = Q K^T (both operands from shared
//              memory) and O += P V (P from TMEM, V from shared memory),
//              fp32 accumulators in TMEM
//   warps 10-11 idle
// The control warpgroup gives registers to the softmax warpgroups
// (setmaxnreg): 2 x 128 x SOFTMAX_REGS + 128 x CONTROL_REGS must not exceed
// the launch allocation of 384 x LAUNCH_REGS, which the host checks.
// Two query slots ping-pong on the tensor core: while softmax works on slot 0's
// scores the MMA thread runs slot 1's P V and its next Q K^T, and vice versa.
// A work item is two 128-row query tiles that share one K/V stream: two heads of
// one GQA group at the same rows (Hq / Hkv even), or two consecutive row tiles of
// one head (otherwise).  Items are dealt to CTAs heaviest first in a
// boustrophedon order, so causal work evens out.
//
// TMEM columns (512 allocated): S/P of slot x at 128 x, O of slot x at
// 256 + D x.  P (bf16, two per 32-bit column) overwrites the first 64 columns of
// its S tile; the next Q K^T into that tile is issued after the P V that reads
// it, and tcgen05 operations of one thread execute in order.
//
// Causal and window tile skipping ("gfx942 unified attention", section 4): a
// slot visits only the key tiles that intersect the union of its rows'
// admissible ranges; element masks are applied only on tiles that cut a row's
// range.  Lazy rescaling: O and l are rescaled only when the running max grows
// by more than 8 (base-2 units); the stale max is used as the reference
// otherwise, which keeps every p <= 2^8 and leaves o / l exact.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int BM = 128;  // query rows per slot
constexpr int BN = 128;  // keys per K/V tile
constexpr int NUM_WARPS = 12;
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int WARP_PRODUCER = 8;
constexpr int WARP_MMA = 9;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float RESCALE_THRESHOLD = 8.0f;  // base-2 units
constexpr int LAUNCH_REGS = 168;          // 65536 / 384, rounded down to a multiple of 8
constexpr int SOFTMAX_REGS = 208;
constexpr int CONTROL_REGS = 88;
static_assert(2 * 128 * SOFTMAX_REGS + 128 * CONTROL_REGS <= NUM_THREADS * LAUNCH_REGS, "register split");

template <int D>
struct Cfg {
    static constexpr int HALVES = D / 64;             // 128-byte swizzle slabs per row
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int Q_SLAB = BM * 128;           // bytes of one 64-column slab of a Q tile
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int KV_SLAB = BN * 128;
    static constexpr int NS = (D == 128) ? 4 : 6;     // K/V ring stages
    static constexpr int SMEM_BYTES = 2 * Q_BYTES + NS * KV_BYTES + 1024;  // + alignment slack
    static constexpr int O_COL = 256;
};

struct Params {
    __nv_bfloat16* out;
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
    int n_qt;          // query tiles per head
    int pair_heads;    // 1: slots are heads (2p, 2p+1) at one row tile; 0: row tiles (2t, 2t+1) of one head
    int n_items;
};

struct Slot {
    int b, h, t;  // t < 0: slot unused in this item
    int lo, hi;   // key-tile range, lo > hi: no admissible key for any row
};

// Admissible key interval [a, b] of query row qi (a > b when empty).
__device__ __forceinline__ void row_interval(const Params& p, int b, int qi, int& a, int& e) {
    a = 0;
    e = p.Sk - 1;
    if (p.causal) e = min(e, qi);
    if (p.wl >= 0) a = max(a, qi - p.wl);
    if (p.wr >= 0) e = min(e, qi + p.wr);
    if (p.rowb) {
        int2 r = __ldg(p.rowb + (size_t)b * p.Sq + qi);
        a = max(a, r.x);
        e = min(e, r.y);
    }
}

// Item -> (b, h, t) of both slots, and each slot's key-tile range.  Called by
// a whole warp (the range is a warp reduction over the slot's rows).
__device__ __forceinline__ void decode_item(const Params& p, int item, Slot (&s)[2]) {
    const int lane = threadIdx.x & 31;
    if (p.pair_heads) {
        const int per_t = p.B * (p.Hq / 2);
        int tr = item / per_t, rest = item % per_t;
        int t = p.causal ? (p.n_qt - 1 - tr) : tr;
        int b = rest / (p.Hq / 2), pr = rest % (p.Hq / 2);
        s[0] = Slot{b, 2 * pr, t, 0, -1};
        s[1] = Slot{b, 2 * pr + 1, t, 0, -1};
    } else {
        const int n_tp = (p.n_qt + 1) / 2;
        const int per_t = p.B * p.Hq;
        int tr = item / per_t, rest = item % per_t;
        int tp = p.causal ? (n_tp - 1 - tr) : tr;
        int b = rest / p.Hq, h = rest % p.Hq;
        s[0] = Slot{b, h, 2 * tp, 0, -1};
        s[1] = Slot{b, h, (2 * tp + 1 < p.n_qt) ? 2 * tp + 1 : -1, 0, -1};
    }
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        if (s[x].t < 0) continue;
        int kmin = 0x7fffffff, kmax = -1;
        const int q0 = s[x].t * BM;
        for (int r = lane; r < BM; r += 32) {
            int qi = q0 + r;
            if (qi >= p.Sq) break;
            int a, e;
            row_interval(p, s[x].b, qi, a, e);
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
}

__device__ __forceinline__ int item_of(int k, int cta, int grid) {
    return k * grid + ((k & 1) ? (grid - 1 - cta) : cta);
}

__device__ __forceinline__ bool slot_live(const Slot& s) { return s.t >= 0 && s.lo <= s.hi; }
__device__ __forceinline__ bool in_range(const Slot& s, int u) { return s.t >= 0 && u >= s.lo && u <= s.hi; }

struct Smem {
    uint64_t q_full[2], q_empty[2];
    uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
    uint64_t kv_full[8], kv_empty[8];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

template <int D, bool SOFTCAP, bool ALIBI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const Params p) {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t dyn_smem[];
    __shared__ Smem sm;

    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ[2] = {base, base + C::Q_BYTES};
    uint8_t* sKV = base + 2 * C::Q_BYTES;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int x = 0; x < 2; ++x) {
            mbar_init(&sm.q_full[x], 1);
            mbar_init(&sm.q_empty[x], 1);
            mbar_init(&sm.s_full[x], 1);
            mbar_init(&sm.p_full[x], BM);
            mbar_init(&sm.o_full[x], 1);
            mbar_init(&sm.o_empty[x], BM);
        }
        for (int i = 0; i < C::NS; ++i) {
            mbar_init(&sm.kv_full[i], 1);
            mbar_init(&sm.kv_empty[i], 1);
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

    if (warp >= 8) {
    // Each warpgroup executes one setmaxnreg, at one program point, before its roles split.
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(CONTROL_REGS));
    if (warp == WARP_PRODUCER) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
        uint32_t kv_cnt = 0, q_cnt[2] = {0, 0};
        bool ok = true;
        for (int k = 0;; ++k) {
            const int item = item_of(k, cta, grid);
            if (item >= p.n_items) break;
            Slot s[2];
            decode_item(p, item, s);
            if (lane == 0) {
                const int hkv = s[0].h / p.G;
                for (int x = 0; x < 2 && ok; ++x) {
                    if (!slot_live(s[x])) continue;
                    ok = mbar_wait(&sm.q_empty[x], (q_cnt[x] & 1) ^ 1, wc, ST_PREFILL_PRODUCER);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&sm.q_full[x], C::Q_BYTES);
#pragma unroll
                    for (int hf = 0; hf < C::HALVES; ++hf)
                        tma_load_3d(sQ[x] + hf * C::Q_SLAB, &tmQ, &sm.q_full[x], hf * 64, s[x].t * BM,
                                    s[x].b * p.Hq + s[x].h);
                    ++q_cnt[x];
                }
                int ulo = 0x7fffffff, uhi = -1;
                for (int x = 0; x < 2; ++x)
                    if (slot_live(s[x])) {
                        ulo = min(ulo, s[x].lo);
                        uhi = max(uhi, s[x].hi);
                    }
                for (int u = ulo; u <= uhi && ok; ++u) {
#pragma unroll
                    for (int kv = 0; kv < 2; ++kv) {
                        const int st = kv_cnt % C::NS;
                        ok = mbar_wait(&sm.kv_empty[st], ((kv_cnt / C::NS) & 1) ^ 1, wc, ST_PREFILL_PRODUCER);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&sm.kv_full[st], C::KV_BYTES);
                        uint8_t* dst = sKV + st * C::KV_BYTES;
#pragma unroll
                        for (int hf = 0; hf < C::HALVES; ++hf)
                            tma_load_3d(dst + hf * C::KV_SLAB, kv ? &tmV : &tmK, &sm.kv_full[st], hf * 64, u * BN,
                                        s[0].b * p.Hkv + hkv);
                        ++kv_cnt;
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
        }
        if (!ok && lane == 0) {
            // Let the copies already issued land before the CTA leaves.
            const uint32_t n = kv_cnt < (uint32_t)C::NS ? kv_cnt : (uint32_t)C::NS;
            for (uint32_t i = kv_cnt - n; i < kv_cnt; ++i)
                mbar_drain(&sm.kv_full[i % C::NS], (i / C::NS) & 1, 100000000ull);
            for (int x = 0; x < 2; ++x)
                if (q_cnt[x]) mbar_drain(&sm.q_full[x], (q_cnt[x] - 1) & 1, 100000000ull);
        }
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0);
        constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, 1);
        uint32_t kv_cnt = 0, q_cnt[2] = {0, 0}, p_cnt[2] = {0, 0}, o_cnt[2] = {0, 0};
        bool ok = true;
        const uint32_t sQa[2] = {smem_u32(sQ[0]), smem_u32(sQ[1])};
        const uint32_t sKVa = smem_u32(sKV);
        for (int k = 0;; ++k) {
            const int item = item_of(k, cta, grid);
            if (item >= p.n_items) break;
            Slot s[2];
            decode_item(p, item, s);
            if (lane == 0) {
                int ulo = 0x7fffffff, uhi = -1;
                for (int x = 0; x < 2; ++x)
                    if (slot_live(s[x])) {
                        ulo = min(ulo, s[x].lo);
                        uhi = max(uhi, s[x].hi);
                    }
                bool q_ready[2] = {false, false};
                auto issue_s = [&](int x, uint32_t kst) -> bool {
                    if (!q_ready[x]) {
                        if (!mbar_wait(&sm.q_full[x], q_cnt[x] & 1, wc, ST_PREFILL_MMA)) return false;
                        ++q_cnt[x];
                        q_ready[x] = true;
                        tc_fence_after();
                    }
                    const uint32_t qa = sQa[x], ka = sKVa + kst * C::KV_BYTES;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * C::Q_SLAB + (kk & 3) * 32;
                        const uint32_t koff = (kk >> 2) * C::KV_SLAB + (kk & 3) * 32;
                        umma_ss(tmem + 128u * x, sdesc_sw128(qa + off, 16), sdesc_sw128(ka + koff, 16), IDESC_S,
                                kk > 0);
                    }
                    umma_commit(&sm.s_full[x]);
                    return true;
                };
                if (ulo <= uhi) {
                    // prologue: K of the first tile
                    uint32_t kst = kv_cnt % C::NS;
                    ok = mbar_wait(&sm.kv_full[kst], (kv_cnt / C::NS) & 1, wc, ST_PREFILL_MMA);
                    ++kv_cnt;
                    if (ok) tc_fence_after();
                    for (int x = 0; x < 2 && ok; ++x)
                        if (in_range(s[x], ulo)) ok = issue_s(x, kst);
                    if (ok) umma_commit(&sm.kv_empty[kst]);
                    for (int u = ulo; u <= uhi && ok; ++u) {
                        const uint32_t vst = kv_cnt % C::NS;
                        ok = mbar_wait(&sm.kv_full[vst], (kv_cnt / C::NS) & 1, wc, ST_PREFILL_MMA);
                        ++kv_cnt;
                        if (!ok) break;
                        tc_fence_after();
                        const bool has_next = u < uhi;
                        for (int x = 0; x < 2 && ok; ++x) {
                            if (in_range(s[x], u)) {
                                ok = mbar_wait(&sm.p_full[x], p_cnt[x] & 1, wc, ST_PREFILL_MMA);
                                ++p_cnt[x];
                                if (ok && u == s[x].lo) {
                                    ok = mbar_wait(&sm.o_empty[x], (o_cnt[x] & 1) ^ 1, wc, ST_PREFILL_MMA);
                                    ++o_cnt[x];
                                }
                                if (!ok) break;
                                tc_fence_after();
                                const uint32_t va = sKVa + vst * C::KV_BYTES;
#pragma unroll
                                for (int kk = 0; kk < BN / 16; ++kk) {
                                    umma_ts(tmem + C::O_COL + D * x, tmem + 128u * x + 8u * kk,
                                            sdesc_sw128(va + kk * 16 * 128, C::KV_SLAB), IDESC_O,
                                            (u > s[x].lo || kk > 0) ? 1u : 0u);
                                }
                                if (u == s[x].hi) umma_commit(&sm.o_full[x]);
                            }
                            if (has_next) {
                                if (x == 0) {
                                    kst = kv_cnt % C::NS;
                                    ok = mbar_wait(&sm.kv_full[kst], (kv_cnt / C::NS) & 1, wc, ST_PREFILL_MMA);
                                    ++kv_cnt;
                                    if (!ok) break;
                                    tc_fence_after();
                                }
                                if (in_range(s[x], u + 1)) ok = issue_s(x, kst);
                            }
                        }
                        if (!ok) break;
                        umma_commit(&sm.kv_empty[vst]);
                        if (has_next) umma_commit(&sm.kv_empty[kst]);
                    }
                    for (int x = 0; x < 2 && ok; ++x)
                        if (slot_live(s[x])) umma_commit(&sm.q_empty[x]);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
        }
        if (lane == 0) {
            // Every MMA issued must finish before TMEM is released.
            umma_commit(&sm.drain);
            mbar_drain(&sm.drain, 0, 100000000ull);
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(SOFTMAX_REGS));
        // ------------------------------------------------------------ softmax / epilogue
        const int x = warp >> 2;
        const int r = threadIdx.x & (BM - 1);
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + 128u * x;
        const uint32_t tO = tmem + lane_off + C::O_COL + D * x;
        uint32_t s_cnt = 0, o_cnt = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int item = item_of(k, cta, grid);
            if (item >= p.n_items) break;
            Slot s[2];
            decode_item(p, item, s);
            const Slot sl = s[x];
            if (sl.t < 0) continue;
            const int qi = sl.t * BM + r;
            const bool live = qi < p.Sq;
            int ra = 1, rb = 0;
            if (live) row_interval(p, sl.b, qi, ra, rb);
            const size_t row = ((size_t)sl.b * p.Hq + sl.h) * p.Sq + qi;
            if (sl.lo > sl.hi) {
                // No admissible key for any row of this tile: zero rows.
                if (live) {
                    uint4 z = make_uint4(0, 0, 0, 0);
                    uint4* dst = reinterpret_cast<uint4*>(p.out + row * D);
#pragma unroll
                    for (int i = 0; i < D / 8; ++i) dst[i] = z;
                    if (p.lse) p.lse[row] = -INFINITY;
                }
                continue;
            }
            float slope_l2 = 0.f;
            if (ALIBI) slope_l2 = __ldg(p.slopes + sl.h) * LOG2E;
            float m_used = -INFINITY, l = 0.f;
            for (int u = sl.lo; u <= sl.hi; ++u) {
                ok = mbar_wait(&sm.s_full[x], s_cnt & 1, wc, ST_PREFILL_SOFTMAX);
                ++s_cnt;
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float sv[BN];
                tmem_ld64(tS, *reinterpret_cast<float(*)[64]>(&sv[0]));
                tmem_ld64(tS + 64, *reinterpret_cast<float(*)[64]>(&sv[64]));
                const int k0 = u * BN;
                // base-2 logits
#pragma unroll
                for (int j = 0; j < BN; ++j) {
                    float t;
                    if (SOFTCAP) {
                        t = p.cap_out * tanhf(sv[j] * p.cap_in);
                    } else {
                        t = sv[j] * p.scale_log2;
                    }
                    if (ALIBI) t = fmaf(slope_l2, (float)(k0 + j - qi), t);
                    sv[j] = t;
                }
                if (k0 < ra || k0 + BN - 1 > rb) {
#pragma unroll
                    for (int j = 0; j < BN; ++j) {
                        const int kj = k0 + j;
                        if (kj < ra || kj > rb) sv[j] = -INFINITY;
                    }
                }
                float mx[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = sv[i];
#pragma unroll
                for (int j = 8; j < BN; ++j) mx[j & 7] = fmaxf(mx[j & 7], sv[j]);
                const float m_tile = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                           fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                const float m_new = fmaxf(m_used, m_tile);
                float alpha = 1.f;
                const bool grow = m_new > m_used + RESCALE_THRESHOLD;
                if (grow) {
                    if (m_used != -INFINITY) alpha = ex2_approx(m_used - m_new);
                    m_used = m_new;
                }
                // O rescale (warp-collective TMEM traffic if any row of the warp needs it).
                // A row's earlier P V completed before this tile's scores (in-order tcgen05).
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
                    l *= alpha;
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
                const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
                float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                uint32_t pw[BN / 2];
#pragma unroll
                for (int j = 0; j < BN; j += 2) {
                    const float p0 = ex2_approx(sv[j] - m_ref);
                    const float p1 = ex2_approx(sv[j + 1] - m_ref);
                    ls[(j >> 1) & 7] += p0 + p1;
                    pw[j >> 1] = pack_bf16x2(p0, p1);
                }
                l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
                tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pw[0]));
                tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pw[32]));
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sm.p_full[x]);
            }
            if (!ok) break;
            // epilogue: O = o / l (zero row if l == 0), bf16, straight from registers.
            ok = mbar_wait(&sm.o_full[x], o_cnt & 1, wc, ST_PREFILL_EPILOGUE);
            ++o_cnt;
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                float ov[32];
                tmem_ld32(tO + c, ov);
                if (live) {
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(ov[2 * i] * inv_l, ov[2 * i + 1] * inv_l);
                    uint4* dst = reinterpret_cast<uint4*>(p.out + row * D + c);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                }
            }
            if (live && p.lse) p.lse[row] = (l > 0.f) ? (m_used + log2f(l)) * LN2 : -INFINITY;
            tc_fence_before();
            mbar_arrive(&sm.o_empty[x]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == WARP_PRODUCER) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool SOFTCAP, bool ALIBI>
cudaError_t launch_variant(const Params& prm, int grid, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, cudaStream_t stream) {
    auto kern = prefill_bf16_kernel<D, SOFTCAP, ALIBI>;
    const int smem = Cfg<D>::SMEM_BYTES;
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    // The warpgroups' register split must fit in what the launch allocates,
    // or setmaxnreg.inc would wait forever.
    if (fa.numRegs < LAUNCH_REGS) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, NUM_THREADS, smem, stream>>>(tq, tk, tv, prm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_bf16(const FwdProblem& f, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, cudaStream_t stream) {
    Params p{};
    p.out = static_cast<__nv_bfloat16*>(f.out);
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
    p.n_qt = (f.Sq + BM - 1) / BM;
    p.pair_heads = (p.G % 2 == 0) ? 1 : 0;
    if (p.pair_heads)
        p.n_items = p.n_qt * f.B * (f.Hq / 2);
    else
        p.n_items = ((p.n_qt + 1) / 2) * f.B * f.Hq;
    const int grid = p.n_items < f.num_sms ? p.n_items : f.num_sms;
    const bool cap = f.softcap > 0.f, ali = f.slopes != nullptr;
    if (f.D == 128) {
        if (cap) return ali ? launch_variant<128, true, true>(p, grid, tq, tk, tv, stream)
                            : launch_variant<128, true, false>(p, grid, tq, tk, tv, stream);
        return ali ? launch_variant<128, false, true>(p, grid, tq, tk, tv, stream)
                   : launch_variant<128, false, false>(p, grid, tq, tk, tv, stream);
    }
    if (cap) return ali ? launch_variant<64, true, true>(p, grid, tq, tk, tv, stream)
                        : launch_variant<64, true, false>(p, grid, tq, tk, tv, stream);
    return ali ? launch_variant<64, false, true>(p, grid, tq, tk, tv, stream)
               : launch_variant<64, false, false>(p, grid, tq, tk, tv, stream);
}

}  // namespace gbattn
