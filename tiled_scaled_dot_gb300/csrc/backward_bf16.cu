// backward_bf16.cu -- attention backward by recompute on tcgen05 tensor cores
// (sm_103a), 16-bit inputs (bf16, or fp16 with the F16 flag), dense
// [B, H, S, D] problems.
//
// Computes the gradients of attention.fkc.md, "attention_flash_backward":
// with P the forward's softmax recomputed from Q, K and the forward's lse,
//   dV_j = sum_i P_ij dO_i,   dP_ij = dO_i . V_j,
//   dS_ij = P_ij (dP_ij - Delta_i) [* (1 - tanh^2(s_pre / c)) with softcap],
//   dQ_i = scale sum_j dS_ij K_j,   dK_j = scale sum_i dS_ij Q_i,
// where Delta_i = sum_j P_ij dP_ij = dO_i . O_i (O the forward output), and
// dK / dV of a kv head sum over the query heads of its GQA group.
//
// Three launches, all deterministic (no atomics, fixed summation order):
//   bwd_rows_kernel    per query row its admissible key interval [a, e]
//                      (causal, window, row bounds, Sk) and per 128-row query
//                      tile a summary: the span of its live rows' intervals
//                      and the tightest interval common to all its rows;
//   bwd_kernel<DQ=1>   one work item per (b, head, 128-row query tile): S =
//                      Q K^T, dP = dO V^T for every admissible key tile,
//                      dQ += dS K accumulated in TMEM.  The item's O tile
//                      comes through the streamed-tile ring ahead of its first
//                      K tile; each row's Delta = dO . O is formed from it and
//                      written with the row's base-2 lse (+inf for a row with
//                      no admissible key, so P = 0) for the next launch;
//   bwd_kernel<DQ=0>   one work item per (b, kv head, 128-key tile): S^T =
//                      K Q^T and dP^T = V dO^T for every admissible 128-row
//                      query tile of every head of the group, dV += P^T dO
//                      and dK += dS^T Q accumulated in TMEM.
// The two main launches are one template: a pair of "fixed" tiles per item
// (K, V or Q, dO) stays in shared memory while pairs of "streamed" tiles
// (Q, dO or K, V) move one tile at a time through a ring of NSLOT shared-memory
// slots (each with its own full and empty barrier, so a tile is released as
// soon as its last reader has been issued and the next tiles land early);
// both products S and dP take the fixed tile as A (M = 128 lanes) and the
// streamed tile as B (N = 128).
//
// Structure (10 warps, one persistent CTA per SM):
//   WG0, WG1 (warps 0-7)   element-wise: thread (g, r) owns TMEM lane r and
//                          columns 64 g .. 64 g + 63 of S and dP; writes P
//                          (DQ = 0) and dS as 16-bit into TMEM; at the end of
//                          an item reads the accumulators out (scale, round,
//                          store)
//   warp 8                 TMA producer
//   warp 9                 MMA issuer (one elected lane issues)
// TMEM (512 columns): S / P at 0, dP / dS at 128, accumulators at 256
// (dV or dQ) and 256 + D (dK).  Packed 16-bit P and dS of group g sit at
// columns 64 g .. 64 g + 31 of their tile, so neither group overwrites
// fp32 values the other has not read yet.
//
// MMA order, DQ = 0 (item with steps 0 .. J-1):
//   S_0, dP_0, then per step j: [P_j] dV += P_j dO_j, S_{j+1},
//   [dS_j] dK += dS_j Q_j, dP_{j+1}
// DQ = 1:
//   S_0, dP_0, then per step j: [S_j read] S_{j+1}, [dS_j] dQ += dS_j K_j, dP_{j+1}
// ([x] = wait for the element-wise warps).  P and dS are handed over in two
// halves of each group's columns, each with its own barrier; the MMAs reading
// a half go out as soon as it is in TMEM.  tcgen05 operations issued by one
// thread execute in order, so an MMA that overwrites a TMEM tile is issued
// after the MMA that reads the tile's previous contents.
//
// Item boundaries: the producer fetches an item's first streamed tiles before
// its fixed tiles (which wait until the previous item's MMAs are done with
// theirs) and prefetches the next item's fixed tiles into L2.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int TR = 128;  // rows of every tile (query rows or keys)
constexpr int NUM_WARPS = 10;
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int EW_THREADS = 256;
constexpr int WARP_PRODUCER = 8;
constexpr int WARP_MMA = 9;
constexpr float LOG2E = 1.4426950408889634f;
constexpr int EXTRA_BYTES = 2048;  // per T1 slot (DQ = 0): lse2[128], delta[128], rows int2[128]
constexpr int MAX_SLOTS = 10;

template <int D, bool DQ>
struct BCfg {
    static constexpr int HALVES = D / 64;
    static constexpr int TILE_BYTES = TR * D * 2;
    static constexpr int SLAB = TR * 128;  // one 64-column slab of a tile
    // streamed-tile slots: a step fills two (T1, then T2); as many as fit
    // beside the fixed tiles in 227 KB
    static constexpr int NSLOT = DQ ? (D == 128 ? 5 : 10) : (D == 128 ? 4 : 8);
    static constexpr int SMEM_BYTES = 2 * TILE_BYTES + NSLOT * TILE_BYTES + (DQ ? 0 : NSLOT * EXTRA_BYTES) + 1024;
    static_assert(NSLOT <= MAX_SLOTS && SMEM_BYTES <= 232448 - 1536, "shared memory");
    static constexpr uint32_t ACC1 = 256;      // dV (DQ = 0) or dQ (DQ = 1)
    static constexpr uint32_t ACC2 = 256 + D;  // dK (DQ = 0)
};

struct BParams {
    uint16_t* dq;  // [B, Hq, Sq, D]
    uint16_t* dk;  // [B, Hkv, Sk, D]
    uint16_t* dv;  // [B, Hkv, Sk, D]
    const float* lse2;   // [B * Hq][Sq_pad] base-2 lse (+inf: no admissible key, or padding)
    const float* delta;  // [B * Hq][Sq_pad]
    float* lse2_w;       // the same arrays, written by the DQ = 1 launch
    float* delta_w;
    const float* lse;    // [B, Hq, Sq] natural-log lse of the forward
    const int2* rows;    // [B][Sq_pad] admissible key interval of each query row
    const int4* summ;    // [B][n_qt] per query tile: (lo_live, hi_live, a_max, e_min)
    const float* slopes;
    unsigned int* status;
    unsigned long long timeout_ns;
    int B, Hq, Hkv, Sq, Sk, G, Sq_pad, n_qt, n_kt;
    int causal;
    float scale;       // softmax_scale (dQ, dK)
    float scale_log2;  // softmax_scale * log2(e)
    float cap_in;      // softmax_scale / softcap
    float cap_out;     // softcap * log2(e)
    int n_items;
    int wide_store;    // dq, dk, dv are 32-byte aligned: 32-byte stores
};

__device__ __forceinline__ int item_of(int k, int cta, int grid) {
    return k * grid + ((k & 1) ? (grid - 1 - cta) : cta);
}

__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Fetch one box of a tensor map into L2 ahead of its TMA load.
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* m, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// One 32-byte global store; the address must be 32-byte aligned.
__device__ __forceinline__ void st_global_32b(void* p, const uint32_t* r) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(r[0]), "r"(r[1]),
                 "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

template <bool F16>
__device__ __forceinline__ float widen16(uint16_t x) {
    return F16 ? __half2float(__ushort_as_half(x)) : __uint_as_float(static_cast<uint32_t>(x) << 16);
}

// ---------------------------------------------------------------------------- row intervals
// Grid (n_qt, B), 128 threads: thread r handles query row m * 128 + r.
__global__ void __launch_bounds__(TR) bwd_rows_kernel(const int2* __restrict__ rowb, int2* __restrict__ rows,
                                                      int4* __restrict__ summ, int Sq, int Sk, int Sq_pad,
                                                      int n_qt, int causal, int wl, int wr) {
    const int m = blockIdx.x, b = blockIdx.y, r = threadIdx.x;
    const int i = m * TR + r;
    long long a = 0, e = Sk - 1;
    if (causal) e = e < i ? e : i;
    if (wl >= 0) a = a > (long long)i - wl ? a : (long long)i - wl;
    if (wr >= 0) e = e < (long long)i + wr ? e : (long long)i + wr;
    if (i < Sq && rowb) {
        const int2 rb = rowb[(size_t)b * Sq + i];
        a = a > rb.x ? a : rb.x;
        e = e < rb.y ? e : rb.y;
    }
    const bool live = i < Sq && a <= e;
    if (!live) {
        a = 1;
        e = 0;
    }
    rows[(size_t)b * Sq_pad + i] = make_int2((int)a, (int)e);
    int lo = live ? (int)a : 0x7fffffff, hi = live ? (int)e : -1;
    int amax = live ? (int)a : 0x7fffffff, emin = live ? (int)e : -1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        emin = min(emin, __shfl_xor_sync(0xffffffffu, emin, o));
    }
    __shared__ int4 red[TR / 32];
    if ((r & 31) == 0) red[r >> 5] = make_int4(lo, hi, amax, emin);
    __syncthreads();
    if (r == 0) {
        int4 s = red[0];
        for (int w = 1; w < TR / 32; ++w) {
            s.x = min(s.x, red[w].x);
            s.y = max(s.y, red[w].y);
            s.z = max(s.z, red[w].z);
            s.w = min(s.w, red[w].w);
        }
        summ[(size_t)b * n_qt + m] = s;
    }
}

// ---------------------------------------------------------------------------- work items
// DQ = 0: item -> (b, kv head, key tile n), lowest n first (under a top-left
// causal mask the first key tiles meet the most query tiles).
// DQ = 1: item -> (b, query head, query tile m), last m first under causal.
struct BItem {
    int b, hd, t;
};

template <bool DQ>
__device__ __forceinline__ BItem bwd_item(const BParams& p, int item) {
    const int heads = DQ ? p.Hq : p.Hkv;
    const int per = p.B * heads;
    const int tr = item / per, rest = item - tr * per;
    BItem it;
    it.b = rest / heads;
    it.hd = rest - it.b * heads;
    it.t = (DQ && p.causal) ? (p.n_qt - 1 - tr) : tr;
    return it;
}

// DQ = 0: does query tile m hold a row whose interval meets keys [k0, k1]?
__device__ __forceinline__ bool tile_meets(const int4& s, int k0, int k1) { return s.x <= k1 && s.y >= k0; }

// DQ = 0: range [m_lo, m_hi] of query tiles that meet the key tile (m_lo > m_hi: none).
__device__ __forceinline__ void q_tile_range(const BParams& p, int b, int k0, int k1, int& m_lo, int& m_hi) {
    m_lo = 0x7fffffff;
    m_hi = -1;
    const int4* s = p.summ + (size_t)b * p.n_qt;
    for (int m = 0; m < p.n_qt; ++m) {
        if (tile_meets(__ldg(s + m), k0, k1)) {
            m_lo = min(m_lo, m);
            m_hi = m;
        }
    }
}

// DQ = 1: range [n_lo, n_hi] of key tiles of query tile m (n_lo > n_hi: none).
__device__ __forceinline__ void k_tile_range(const BParams& p, int b, int m, int& n_lo, int& n_hi) {
    const int4 s = __ldg(p.summ + (size_t)b * p.n_qt + m);
    if (s.x <= s.y) {
        n_lo = s.x / TR;
        n_hi = s.y / TR;
    } else {
        n_lo = 0;
        n_hi = -1;
    }
}

struct BSmem {
    uint64_t fix_full, fix_empty;
    uint64_t slot_full[MAX_SLOTS], slot_empty[MAX_SLOTS];
    uint64_t s_full, dp_full, s_free, acc_full, acc_empty;
    uint64_t p_half[2], ds_half[2];  // P / dS of columns 64 g + 32 h .. + 31 of both groups are in TMEM
    uint64_t drain;
    uint64_t delta_bar;  // DQ = 1: both column groups' Delta halves are written
    uint32_t tmem_base;
    int abort_flag;
    float dpart[2][TR];  // DQ = 1: Delta halves per column group and row
};

// The steps of an item, enumerated the same way by every role.
//   DQ = 0: for each head of the group, each query tile in [m_lo, m_hi] that
//           meets the key tile; f(h, m).
//   DQ = 1: each key tile n in [n_lo, n_hi]; f(n).
// f returns false to stop.
template <bool DQ, typename F>
__device__ __forceinline__ bool for_steps(const BParams& p, const BItem& it, F&& f) {
    if (DQ) {
        int n_lo, n_hi;
        k_tile_range(p, it.b, it.t, n_lo, n_hi);
        for (int n = n_lo; n <= n_hi; ++n)
            if (!f(it.hd, n)) return false;
    } else {
        const int k0 = it.t * TR, k1 = min(k0 + TR - 1, p.Sk - 1);
        int m_lo, m_hi;
        q_tile_range(p, it.b, k0, k1, m_lo, m_hi);
        const int4* s = p.summ + (size_t)it.b * p.n_qt;
        for (int hh = 0; hh < p.G; ++hh)
            for (int m = m_lo; m <= m_hi; ++m)
                if (tile_meets(__ldg(s + m), k0, k1) && !f(it.hd * p.G + hh, m)) return false;
    }
    return true;
}

template <bool DQ>
__device__ __forceinline__ int count_steps(const BParams& p, const BItem& it) {
    int n = 0;
    for_steps<DQ>(p, it, [&](int, int) {
        ++n;
        return true;
    });
    return n;
}

// ---------------------------------------------------------------------------- element-wise role
// 32 lanes x 32 bits, 16 consecutive columns per thread (no wait).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Store 32 fp32 accumulator values (times f) of one output row as 16-bit:
// two 32-byte stores when `wide` (dst 32-byte aligned), else four 16-byte ones.
template <bool F16>
__device__ __forceinline__ void store_row32(uint16_t* dst, const float (&v)[32], float f, bool wide) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack16x2<F16>(v[2 * i] * f, v[2 * i + 1] * f);
    if (wide) {
        st_global_32b(dst, w);
        st_global_32b(dst + 16, w + 8);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            reinterpret_cast<uint4*>(dst)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
}

// This column group's half of dO_i . O_i in fp32: D / 2 dimensions of row r
// of two 128 x D tiles in shared memory (64-column slabs, 128-byte swizzle);
// group g takes slab g (D = 128) or chunks 4 g .. 4 g + 3 of the one slab
// (D = 64).  Two accumulators over even and odd dimensions, fixed order.
template <int D, bool F16>
__device__ __forceinline__ float half_row_dot(const uint8_t* a, const uint8_t* o, int g, int r) {
    constexpr int CH = D / 16;
    const int slab = D == 128 ? g : 0, cb = D == 128 ? 0 : 4 * g;
    const uint8_t* pa = a + slab * (TR * 128) + r * 128;
    const uint8_t* po = o + slab * (TR * 128) + r * 128;
    float d0 = 0.f, d1 = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const int off = ((cb + c) ^ (r & 7)) << 4;
        const uint4 x = *reinterpret_cast<const uint4*>(pa + off);
        const uint4 y = *reinterpret_cast<const uint4*>(po + off);
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            d0 = fmaf(widen16<F16>((uint16_t)(xw[t] & 0xffffu)), widen16<F16>((uint16_t)(yw[t] & 0xffffu)), d0);
            d1 = fmaf(widen16<F16>((uint16_t)(xw[t] >> 16)), widen16<F16>((uint16_t)(yw[t] >> 16)), d1);
        }
    }
    return d0 + d1;
}

__device__ __forceinline__ void zero_row(uint16_t* dst, int n) {
    for (int i = 0; i < n / 8; ++i) reinterpret_cast<uint4*>(dst)[i] = make_uint4(0, 0, 0, 0);
}

template <int D, bool DQ, bool SOFTCAP, bool ALIBI, bool F16>
__device__ __forceinline__ void ew_role(const BParams& p, BSmem& sm, uint32_t tmem, const WaitCtl& wc, int warp,
                                        const uint8_t* sX, const uint8_t* sF2, const uint8_t* sT) {
    using C = BCfg<D, DQ>;
    const int g = warp >> 2;          // column group: columns 64 g .. 64 g + 63
    const int r = threadIdx.x & (TR - 1);  // TMEM lane
    const int c0 = 64 * g;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + c0;         // S; packed P at its first 32 columns
    const uint32_t tDP = tmem + lane_off + 128 + c0;  // dP; packed dS at its first 32 columns
    const int grid = gridDim.x, cta = blockIdx.x;
    uint32_t step = 0, acc_cnt = 0, stg = 0;
    uint32_t nlive = 0, dcnt = 0;  // items with steps so far; Delta exchanges so far (DQ = 1)
    for (int k = 0;; ++k) {
        const int item = item_of(k, cta, grid);
        if (item >= p.n_items) break;
        const BItem it = bwd_item<DQ>(p, item);
        const int J = count_steps<DQ>(p, it);
        if (J == 0) {
            // no admissible (row, key) pair touches the item: zero gradient rows
            if (DQ) {
                const int i = it.t * TR + r;
                if (i < p.Sq) zero_row(p.dq + ((size_t)(it.b * p.Hq + it.hd) * p.Sq + i) * D + g * (D / 2), D / 2);
                if (g == 0) {
                    const size_t prow = (size_t)(it.b * p.Hq + it.hd) * p.Sq_pad + i;
                    p.lse2_w[prow] = INFINITY;
                    p.delta_w[prow] = 0.f;
                }
            } else {
                const int key = it.t * TR + r;
                if (key < p.Sk) zero_row((g ? p.dk : p.dv) + ((size_t)(it.b * p.Hkv + it.hd) * p.Sk + key) * D, D);
            }
            continue;
        }
        // DQ = 1: this thread's query row, fixed over the item
        int ra = 1, rb = 0;
        float lse2_i = INFINITY, delta_i = 0.f;
        if (DQ) {
            const int i = it.t * TR + r;  // < Sq_pad
            const int2 iv = __ldg(p.rows + (size_t)it.b * p.Sq_pad + i);
            ra = iv.x;
            rb = iv.y;
            if (i < p.Sq) {
                const float lv = __ldg(p.lse + (size_t)(it.b * p.Hq + it.hd) * p.Sq + i);
                lse2_i = (lv == -INFINITY) ? INFINITY : lv * LOG2E;
            }
        }
        // DQ = 1: fill index of the item's O tile (the producer loads it into the
        // ring ahead of the item's first K tile), and the item's fixed-tile phase
        const uint32_t f_o = 2 * stg + nlive;
        const uint32_t fix_par = nlive & 1u;
        ++nlive;
        bool first = true;
        const bool ok = for_steps<DQ>(p, it, [&](int h, int u) -> bool {
            const uint32_t f1 = 2 * stg;  // fill index of the step's T1 tile (its extras sit beside it)
            const int st = (int)(f1 % C::NSLOT);
            const uint32_t sp = (f1 / C::NSLOT) & 1u;
            ++stg;
            bool w = true;
            // DQ = 0: admissible columns of this thread's key as a bit mask, from
            // the stage's row intervals (all ones when every row admits the tile)
            uint64_t adm = ~0ull;
            if (!DQ) {
                w = mbar_wait(&sm.slot_full[st], sp, wc, ST_BWD_EW);
                const int k0 = it.t * TR, kj = k0 + r;
                const int4 su = __ldg(p.summ + (size_t)it.b * p.n_qt + u);
                if (w && !(su.z <= k0 && su.w >= k0 + TR - 1)) {
                    const int4* xr = reinterpret_cast<const int4*>(sX + st * EXTRA_BYTES + 1024) + c0 / 2;
                    adm = 0ull;
#pragma unroll 8
                    for (int c = 0; c < 64; c += 2) {
                        const int4 iv = xr[c >> 1];  // intervals of columns c, c + 1
                        const uint64_t two = (uint64_t)(kj >= iv.x && kj <= iv.y) | ((uint64_t)(kj >= iv.z && kj <= iv.w) << 1);
                        adm |= two << c;
                    }
                }
            }
            w = w && mbar_wait(&sm.s_full, step & 1u, wc, ST_BWD_EW);
            if (!__all_sync(0xffffffffu, w)) return false;
            // DQ = 0: does any lane of the warp have a masked column?
            const bool warp_masked = !DQ && __any_sync(0xffffffffu, adm != ~0ull);
            tc_fence_after();
            float sv[64];
            tmem_ld64(tS, sv);
            if (DQ) {
                // S is in registers: the next S may overwrite the tile
                tc_fence_before();
                mbar_arrive(&sm.s_free);
            }
            const float slope_l2 = ALIBI ? __ldg(p.slopes + h) * LOG2E : 0.f;
            uint32_t pw[32];
            if (!DQ) {
                // thread = key kj, columns = query rows i = m * 128 + c0 + c
                const float* xl = reinterpret_cast<const float*>(sX + st * EXTRA_BYTES) + c0;  // lse2
                const int kj = it.t * TR + r;
                const float abase = ALIBI ? slope_l2 * (float)(kj - u * TR - c0) : 0.f;
                const uint32_t adm_lo = (uint32_t)adm, adm_hi = (uint32_t)(adm >> 32);
                // the column loop, with or without the per-column mask (a warp-uniform choice)
                // Each 32-column half is packed, stored and announced on its own,
                // so the MMA warp starts dV on the first half while the second
                // is computed.  Packed half h lands on columns 16 h .. 16 h + 15
                // of the group's tile, which hold first-half S values already in
                // registers.
                auto p_loop = [&](auto masked) {
#pragma unroll
                    for (int c = 0; c < 64; c += 2) {
                        float z[2], f[2] = {1.f, 1.f};
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int cc = c + e;
                            if (SOFTCAP) {
                                const float t = tanh_approx(sv[cc] * p.cap_in);
                                z[e] = fmaf(p.cap_out, t, -xl[cc]);
                                f[e] = fmaf(-t, t, 1.f);
                            } else {
                                z[e] = fmaf(sv[cc], p.scale_log2, -xl[cc]);
                            }
                            if (ALIBI) z[e] += fmaf(-slope_l2, (float)cc, abase);
                            float pe = ex2_approx(z[e]);
                            if (decltype(masked)::value) {
                                const uint32_t word = cc < 32 ? adm_lo : adm_hi;
                                pe = ((int)(word << (31 - (cc & 31))) < 0) ? pe : 0.f;
                            }
                            z[e] = pe;
                        }
                        pw[c >> 1] = pack16x2<F16>(z[0], z[1]);
                        sv[c] = z[0] * f[0];
                        sv[c + 1] = z[1] * f[1];
                        if (c == 30 || c == 62) {
                            const int hf = c >> 5;
                            tmem_st16(tS + 16 * hf, *reinterpret_cast<const uint32_t(*)[16]>(&pw[16 * hf]));
                            tmem_wait_st();
                            tc_fence_before();
                            mbar_arrive(&sm.p_half[hf]);
                        }
                    }
                };
                if (warp_masked)
                    p_loop(std::true_type{});
                else
                    p_loop(std::false_type{});
            } else {
                // thread = query row i, columns = keys k0 + c0 + c
                const int i = it.t * TR + r;
                const int kb = u * TR + c0;
                const int lo = ra - kb, hi = rb - kb;
                // the vote is taken by the converged warp, outside any per-lane branch
                const bool need = __any_sync(0xffffffffu, kb < ra || kb + 63 > rb);
                const float abase = ALIBI ? slope_l2 * (float)(kb - i) : 0.f;
                auto p_loop = [&](auto masked) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        float z, f = 1.f;
                        if (SOFTCAP) {
                            const float t = tanh_approx(sv[c] * p.cap_in);
                            z = fmaf(p.cap_out, t, -lse2_i);
                            f = fmaf(-t, t, 1.f);
                        } else {
                            z = fmaf(sv[c], p.scale_log2, -lse2_i);
                        }
                        if (ALIBI) z += fmaf(slope_l2, (float)c, abase);
                        float pe = ex2_approx(z);
                        if (decltype(masked)::value) pe = (c < lo || c > hi) ? 0.f : pe;
                        sv[c] = pe * f;
                    }
                };
                if (need)
                    p_loop(std::true_type{});
                else
                    p_loop(std::false_type{});
            }
            if (DQ && first) {
                // Delta_i = dO_i . O_i: each column group takes half of the
                // dimensions from the fixed dO tile and the item's O tile, and
                // the halves meet in shared memory.  The exchange buffer is
                // rewritten one item later, after every thread has passed this
                // item's first dS hand-off (which needs Delta).
                const int so = (int)(f_o % C::NSLOT);
                bool w2 = mbar_wait(&sm.fix_full, fix_par, wc, ST_BWD_EW);
                w2 = w2 && mbar_wait(&sm.slot_full[so], (f_o / C::NSLOT) & 1u, wc, ST_BWD_EW);
                sm.dpart[g][r] = w2 ? half_row_dot<D, F16>(sF2, sT + so * C::TILE_BYTES, g, r) : 0.f;
                mbar_arrive(&sm.delta_bar);
                w2 = w2 && mbar_wait(&sm.delta_bar, dcnt & 1u, wc, ST_BWD_EW);
                ++dcnt;
                if (!__all_sync(0xffffffffu, w2)) return false;
                const int i = it.t * TR + r;
                delta_i = i < p.Sq ? sm.dpart[0][r] + sm.dpart[1][r] : 0.f;
                if (g == 0) {
                    const size_t prow = (size_t)(it.b * p.Hq + it.hd) * p.Sq_pad + i;
                    p.lse2_w[prow] = lse2_i;
                    p.delta_w[prow] = delta_i;
                }
            }
            first = false;
            w = mbar_wait(&sm.dp_full, step & 1u, wc, ST_BWD_EW);
            if (!__all_sync(0xffffffffu, w)) return false;
            tc_fence_after();
            // dS in two 32-column halves, each stored and announced on its own:
            // packed half h goes to columns 16 h .. 16 h + 15 of the group's
            // tile, which hold first-half dP values already read
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float dp[32];
                tmem_ld32(tDP + 32 * hf, dp);
                if (!DQ) {
                    const float* xd = reinterpret_cast<const float*>(sX + st * EXTRA_BYTES + 512) + c0 + 32 * hf;
#pragma unroll
                    for (int c = 0; c < 32; c += 2)
                        pw[16 * hf + (c >> 1)] = pack16x2<F16>(sv[32 * hf + c] * (dp[c] - xd[c]),
                                                               sv[32 * hf + c + 1] * (dp[c + 1] - xd[c + 1]));
                } else {
#pragma unroll
                    for (int c = 0; c < 32; c += 2)
                        pw[16 * hf + (c >> 1)] = pack16x2<F16>(sv[32 * hf + c] * (dp[c] - delta_i),
                                                               sv[32 * hf + c + 1] * (dp[c + 1] - delta_i));
                }
                tmem_st16(tDP + 16 * hf, *reinterpret_cast<const uint32_t(*)[16]>(&pw[16 * hf]));
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sm.ds_half[hf]);
            }
            ++step;
            return true;
        });
        if (!ok) return;
        // the item's accumulators: read, scale, round, store
        const bool w = mbar_wait(&sm.acc_full, acc_cnt & 1u, wc, ST_BWD_EW);
        ++acc_cnt;
        if (!__all_sync(0xffffffffu, w)) return;
        tc_fence_after();
        if (DQ) {
            const int i = it.t * TR + r;
            uint16_t* dst = p.dq + ((size_t)(it.b * p.Hq + it.hd) * p.Sq + i) * D + g * (D / 2);
#pragma unroll
            for (int c = 0; c < D / 2; c += 32) {
                float v[32];
                tmem_ld32(tmem + lane_off + C::ACC1 + g * (D / 2) + c, v);
                if (i < p.Sq) store_row32<F16>(dst + c, v, p.scale, p.wide_store != 0);
            }
        } else {
            const int key = it.t * TR + r;
            uint16_t* dst = (g ? p.dk : p.dv) + ((size_t)(it.b * p.Hkv + it.hd) * p.Sk + key) * D;
            const uint32_t acc = g ? C::ACC2 : C::ACC1;
            const float f = g ? p.scale : 1.f;
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                float v[32];
                tmem_ld32(tmem + lane_off + acc + c, v);
                if (key < p.Sk) store_row32<F16>(dst + c, v, f, p.wide_store != 0);
            }
        }
        tc_fence_before();
        mbar_arrive(&sm.acc_empty);
    }
}

// ---------------------------------------------------------------------------- kernel
template <int D, bool DQ, bool SOFTCAP, bool ALIBI, bool F16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __grid_constant__ CUtensorMap tmO, const BParams p) {
    using C = BCfg<D, DQ>;
    extern __shared__ __align__(1024) uint8_t dyn_smem[];
    __shared__ BSmem sm;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    uint8_t* sF1 = base;                        // K (DQ = 0) or Q (DQ = 1)
    uint8_t* sF2 = base + C::TILE_BYTES;        // V or dO
    uint8_t* sT = base + 2 * C::TILE_BYTES;     // streamed-tile slots
    uint8_t* sX = sT + C::NSLOT * C::TILE_BYTES;  // per-slot extras (DQ = 0)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&sm.fix_full, 1);
        mbar_init(&sm.fix_empty, 1);
        for (int i = 0; i < C::NSLOT; ++i) {
            mbar_init(&sm.slot_full[i], 1);
            mbar_init(&sm.slot_empty[i], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.dp_full, 1);
        mbar_init(&sm.p_half[0], EW_THREADS);
        mbar_init(&sm.p_half[1], EW_THREADS);
        mbar_init(&sm.s_free, EW_THREADS);
        mbar_init(&sm.ds_half[0], EW_THREADS);
        mbar_init(&sm.ds_half[1], EW_THREADS);
        mbar_init(&sm.acc_full, 1);
        mbar_init(&sm.acc_empty, EW_THREADS);
        mbar_init(&sm.drain, 1);
        mbar_init(&sm.delta_bar, EW_THREADS);
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

    if (warp < 8) {
        ew_role<D, DQ, SOFTCAP, ALIBI, F16>(p, sm, tmem, wc, warp, sX, sF2, sT);
    } else if (warp == WARP_PRODUCER) {
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmDO);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            if (DQ) tma_prefetch_desc(&tmO);
            uint32_t fix_cnt = 0, fills = 0;  // fills: streamed tiles loaded so far (two per step)
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int item = item_of(k, cta, grid);
                if (item >= p.n_items) break;
                const BItem it = bwd_item<DQ>(p, item);
                const int J = count_steps<DQ>(p, it);
                if (J == 0) continue;
                const int hkv = DQ ? it.hd / p.G : it.hd;
                // Streamed tiles of the item's steps [lo, hi): T1 then T2 of each.
                auto fill_steps = [&](int lo, int hi) -> bool {
                    int j = 0;
                    return for_steps<DQ>(p, it, [&](int h, int u) -> bool {
                        const int jj = j++;
                        if (jj < lo) return true;
                        if (jj >= hi) return false;
#pragma unroll
                        for (int x = 0; x < 2; ++x) {  // x = 0: T1 (Q or K), x = 1: T2 (dO or V)
                            const int sl = (int)(fills % C::NSLOT);
                            if (!mbar_wait(&sm.slot_empty[sl], ((fills / C::NSLOT) & 1u) ^ 1u, wc, ST_BWD_PRODUCER))
                                return ok = false;
                            uint64_t* fb = &sm.slot_full[sl];
                            const bool extras = !DQ && x == 0;
                            mbar_arrive_expect_tx(fb, C::TILE_BYTES + (extras ? EXTRA_BYTES : 0));
                            uint8_t* dst = sT + sl * C::TILE_BYTES;
                            const CUtensorMap* m = DQ ? (x ? &tmV : &tmK) : (x ? &tmDO : &tmQ);
                            const int plane = DQ ? it.b * p.Hkv + hkv : it.b * p.Hq + h;
#pragma unroll
                            for (int hf = 0; hf < C::HALVES; ++hf)
                                tma_load_3d(dst + hf * C::SLAB, m, fb, hf * 64, u * TR, plane);
                            if (extras) {
                                const size_t row = (size_t)(it.b * p.Hq + h) * p.Sq_pad + (size_t)u * TR;
                                uint8_t* xb = sX + sl * EXTRA_BYTES;
                                bulk_load(xb, p.lse2 + row, 512, fb);
                                bulk_load(xb + 512, p.delta + row, 512, fb);
                                bulk_load(xb + 1024, p.rows + (size_t)it.b * p.Sq_pad + (size_t)u * TR, 1024, fb);
                            }
                            ++fills;
                        }
                        return true;
                    });
                };
                if (DQ) {
                    // the item's O tile (for Delta) ahead of its streamed tiles; the
                    // element-wise warps read it and the MMA warp releases it
                    const int sl = (int)(fills % C::NSLOT);
                    if (!(ok = mbar_wait(&sm.slot_empty[sl], ((fills / C::NSLOT) & 1u) ^ 1u, wc, ST_BWD_PRODUCER)))
                        break;
                    mbar_arrive_expect_tx(&sm.slot_full[sl], C::TILE_BYTES);
#pragma unroll
                    for (int hf = 0; hf < C::HALVES; ++hf)
                        tma_load_3d(sT + sl * C::TILE_BYTES + hf * C::SLAB, &tmO, &sm.slot_full[sl], hf * 64,
                                    it.t * TR, it.b * p.Hq + it.hd);
                    ++fills;
                }
                // The first steps' tiles go out before the fixed tiles, which wait
                // until the previous item's MMAs are done with theirs; the ring
                // holds them (and the O tile), so this never waits on this item's
                // own MMAs.
                constexpr int PRE = DQ ? (C::NSLOT - 1) / 2 : C::NSLOT / 2;
                const int pre = J < PRE ? J : PRE;
                fill_steps(0, pre);
                if (!ok) break;
                ok = mbar_wait(&sm.fix_empty, (fix_cnt & 1u) ^ 1u, wc, ST_BWD_PRODUCER);
                if (!ok) break;
                mbar_arrive_expect_tx(&sm.fix_full, 2 * C::TILE_BYTES);
#pragma unroll
                for (int hf = 0; hf < C::HALVES; ++hf) {
                    if (DQ) {
                        tma_load_3d(sF1 + hf * C::SLAB, &tmQ, &sm.fix_full, hf * 64, it.t * TR, it.b * p.Hq + it.hd);
                        tma_load_3d(sF2 + hf * C::SLAB, &tmDO, &sm.fix_full, hf * 64, it.t * TR, it.b * p.Hq + it.hd);
                    } else {
                        tma_load_3d(sF1 + hf * C::SLAB, &tmK, &sm.fix_full, hf * 64, it.t * TR, it.b * p.Hkv + hkv);
                        tma_load_3d(sF2 + hf * C::SLAB, &tmV, &sm.fix_full, hf * 64, it.t * TR, it.b * p.Hkv + hkv);
                    }
                }
                ++fix_cnt;
                {
                    // the next item's fixed tiles, into L2 while this item runs
                    const int nx = item_of(k + 1, cta, grid);
                    if (nx < p.n_items) {
                        const BItem in = bwd_item<DQ>(p, nx);
#pragma unroll
                        for (int hf = 0; hf < C::HALVES; ++hf) {
                            if (DQ) {
                                tma_prefetch_l2_3d(&tmQ, hf * 64, in.t * TR, in.b * p.Hq + in.hd);
                                tma_prefetch_l2_3d(&tmDO, hf * 64, in.t * TR, in.b * p.Hq + in.hd);
                            } else {
                                tma_prefetch_l2_3d(&tmK, hf * 64, in.t * TR, in.b * p.Hkv + in.hd);
                                tma_prefetch_l2_3d(&tmV, hf * 64, in.t * TR, in.b * p.Hkv + in.hd);
                            }
                        }
                    }
                }
                fill_steps(pre, J);
            }
            if (!ok) {
                // let the copies already issued land before the CTA leaves
                const uint32_t n = fills < (uint32_t)C::NSLOT ? fills : (uint32_t)C::NSLOT;
                for (uint32_t i = fills - n; i < fills; ++i)
                    mbar_drain(&sm.slot_full[i % C::NSLOT], (i / C::NSLOT) & 1u, 100000000ull);
                if (fix_cnt) mbar_drain(&sm.fix_full, (fix_cnt - 1) & 1u, 100000000ull);
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // The whole warp runs the loop; one elected lane issues each MMA and
        // commit.  Waits are warp votes, so the warp stays converged.
        auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, wc, ST_BWD_MMA));
        };
        constexpr uint32_t IDESC_S = F16 ? idesc_f16_f32(TR, TR, 0) : idesc_bf16_f32(TR, TR, 0);
        constexpr uint32_t IDESC_A = F16 ? idesc_f16_f32(TR, D, 1) : idesc_bf16_f32(TR, D, 1);
        const uint32_t aF1 = smem_u32(sF1), aF2 = smem_u32(sF2), aT = smem_u32(sT);
        // streamed tile of fill index f: its slot address, its wait, its release
        auto tile_of = [&](uint32_t f) { return aT + (f % C::NSLOT) * C::TILE_BYTES; };
        auto wfill = [&](uint32_t f) { return wwait(&sm.slot_full[f % C::NSLOT], (f / C::NSLOT) & 1u); };
        auto release = [&](uint32_t f) { umma_commit_elect(&sm.slot_empty[f % C::NSLOT]); };
        // D[col] = A B^T over K = D: both operands K-major 128 x D tiles
        auto mma_ss = [&](uint32_t col, uint32_t a, uint32_t b) {
            const uint32_t alo = sdesc_lo(a, 16), blo = sdesc_lo(b, 16);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * C::SLAB + (kk & 3) * 32) >> 4;
                umma_ss_lo_elect(tmem + col, alo + off, blo + off, IDESC_S, kk > 0 ? 1u : 0u);
            }
        };
        // D[col] (+)= A[TMEM, packed 16-bit at acol] B over K = 128 rows of the
        // MN-major 128 x D tile b, in two calls by half of the packed columns.
        // The same for half hf of the packed columns: K chunks 2 hf, 2 hf + 1 of
        // each group's 64 columns (P or dS handed over per half); the step's
        // first MMA (half 0, chunk 0) takes `acc`
        auto mma_ts_half = [&](uint32_t col, uint32_t acol, uint32_t b, uint32_t acc, int hf) {
            const uint32_t blo = sdesc_lo(b, C::SLAB);
#pragma unroll
            for (int gi = 0; gi < 2; ++gi)
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int kk = 4 * gi + 2 * hf + i;
                    const uint32_t a = tmem + acol + 64u * gi + 8u * (2 * hf + i);
                    const uint32_t first = (hf == 0 && gi == 0 && i == 0) ? acc : 1u;
                    umma_ts_lo_elect(tmem + col, a, blo + ((kk * 16 * 128) >> 4), IDESC_A, first);
                }
        };
        uint32_t fix_cnt = 0, stg = 0, step = 0, acc_cnt = 0;
        bool ok = true;
        // fills: DQ = 1 items load their O tile first, so fix_cnt (items with
        // steps so far, this one included) fills precede this item's steps on
        // top of two per step
        for (int k = 0; ok; ++k) {
            const int item = item_of(k, cta, grid);
            if (item >= p.n_items) break;
            const BItem it = bwd_item<DQ>(p, item);
            const int J = count_steps<DQ>(p, it);
            if (J == 0) continue;
            ok = wwait(&sm.fix_full, fix_cnt & 1u);
            ++fix_cnt;
            const uint32_t f0 = 2 * stg + (DQ ? fix_cnt : 0u);  // step j: T1 = f0 + 2 j, T2 = f0 + 2 j + 1
            ok = ok && wfill(f0);
            if (!ok) break;
            tc_fence_after();
            mma_ss(0, aF1, tile_of(f0));
            umma_commit_elect(&sm.s_full);
            if (!(ok = wfill(f0 + 1))) break;
            tc_fence_after();
            mma_ss(128, aF2, tile_of(f0 + 1));
            umma_commit_elect(&sm.dp_full);
            if (DQ) release(f0 + 1);  // V_0 has no other reader
            for (int j = 0; j < J && ok; ++j, ++step) {
                const uint32_t t1 = f0 + 2 * j, t2 = t1 + 1, n1 = t1 + 2, n2 = t1 + 3;
                const bool more = j + 1 < J;
                if (!DQ) {
                    ok = wwait(&sm.p_half[0], step & 1u);
                    if (ok && j == 0) ok = wwait(&sm.acc_empty, (acc_cnt & 1u) ^ 1u);
                    if (!ok) break;
                    tc_fence_after();
                    mma_ts_half(C::ACC1, 0, tile_of(t2), j > 0 ? 1u : 0u, 0);  // dV += P^T dO
                    if (!(ok = wwait(&sm.p_half[1], step & 1u))) break;
                    tc_fence_after();
                    mma_ts_half(C::ACC1, 0, tile_of(t2), 1u, 1);
                    release(t2);  // dO_j: read by dP_j and dV_j
                    if (more) {
                        if (!(ok = wfill(n1))) break;
                        tc_fence_after();
                        mma_ss(0, aF1, tile_of(n1));
                        umma_commit_elect(&sm.s_full);
                    }
                    if (!(ok = wwait(&sm.ds_half[0], step & 1u))) break;
                    tc_fence_after();
                    mma_ts_half(C::ACC2, 128, tile_of(t1), j > 0 ? 1u : 0u, 0);  // dK += dS^T Q
                    if (!(ok = wwait(&sm.ds_half[1], step & 1u))) break;
                    tc_fence_after();
                    mma_ts_half(C::ACC2, 128, tile_of(t1), 1u, 1);
                    release(t1);  // Q_j and its extras: read by S_j, dK_j and the element-wise warps
                    if (more) {
                        if (!(ok = wfill(n2))) break;
                        tc_fence_after();
                        mma_ss(128, aF2, tile_of(n2));
                        umma_commit_elect(&sm.dp_full);
                    }
                } else {
                    if (more) {
                        ok = wwait(&sm.s_free, step & 1u);
                        ok = ok && wfill(n1);
                        if (!ok) break;
                        tc_fence_after();
                        mma_ss(0, aF1, tile_of(n1));
                        umma_commit_elect(&sm.s_full);
                    }
                    ok = wwait(&sm.ds_half[0], step & 1u);
                    if (ok && j == 0) ok = wwait(&sm.acc_empty, (acc_cnt & 1u) ^ 1u);
                    if (!ok) break;
                    // every element-wise thread has formed Delta: the O tile is read
                    if (j == 0) release(f0 - 1);
                    tc_fence_after();
                    mma_ts_half(C::ACC1, 128, tile_of(t1), j > 0 ? 1u : 0u, 0);  // dQ += dS K
                    if (!(ok = wwait(&sm.ds_half[1], step & 1u))) break;
                    tc_fence_after();
                    mma_ts_half(C::ACC1, 128, tile_of(t1), 1u, 1);
                    release(t1);                                          // K_j: read by S_j and dQ_j
                    if (more) {
                        if (!(ok = wfill(n2))) break;
                        tc_fence_after();
                        mma_ss(128, aF2, tile_of(n2));
                        umma_commit_elect(&sm.dp_full);
                        release(n2);  // V_{j+1}: read by dP_{j+1} only
                    }
                }
            }
            if (!ok) break;
            stg += J;
            umma_commit_elect(&sm.acc_full);
            umma_commit_elect(&sm.fix_empty);
            ++acc_cnt;
        }
        if (lane == 0) {
            // every MMA issued must finish before TMEM is released
            umma_commit(&sm.drain);
            mbar_drain(&sm.drain, 0, 100000000ull);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == WARP_PRODUCER) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool DQ, bool SOFTCAP, bool ALIBI, bool F16>
cudaError_t launch_main(const BParams& prm, int grid, const CUtensorMap& tq, const CUtensorMap& tdo,
                        const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t stream) {
    auto kern = bwd_kernel<D, DQ, SOFTCAP, ALIBI, F16>;
    const int smem = BCfg<D, DQ>::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, NUM_THREADS, smem, stream>>>(tq, tdo, tk, tv, to, prm);
    return cudaGetLastError();
}

template <int D, bool F16>
cudaError_t launch_flags(const BParams& prm, int grid_a, int grid_b, bool cap, bool ali, const CUtensorMap& tq,
                         const CUtensorMap& tdo, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& to, cudaStream_t stream,
                         cudaEvent_t* ev) {
    BParams pa = prm, pb = prm;
    pa.n_items = prm.n_kt * prm.B * prm.Hkv;
    pb.n_items = prm.n_qt * prm.B * prm.Hq;
    cudaError_t e;
    // dQ first: it writes the Delta and base-2 lse that dK / dV reads
#define GBATTN_BWD_PAIR(CAP, ALI)                                                              \
    e = launch_main<D, true, CAP, ALI, F16>(pb, grid_b, tq, tdo, tk, tv, to, stream);           \
    if (e != cudaSuccess) return e;                                                             \
    if (ev && (e = cudaEventRecord(ev[2], stream)) != cudaSuccess) return e;                    \
    e = launch_main<D, false, CAP, ALI, F16>(pa, grid_a, tq, tdo, tk, tv, to, stream);          \
    if (e != cudaSuccess) return e;                                                             \
    return ev ? cudaEventRecord(ev[3], stream) : cudaSuccess;
    if (cap) {
        if (ali) {
            GBATTN_BWD_PAIR(true, true)
        } else {
            GBATTN_BWD_PAIR(true, false)
        }
    } else {
        if (ali) {
            GBATTN_BWD_PAIR(false, true)
        } else {
            GBATTN_BWD_PAIR(false, false)
        }
    }
#undef GBATTN_BWD_PAIR
}

}  // namespace

size_t backward_sq_pad(int Sq) { return ((size_t)Sq + TR - 1) / TR * TR; }

cudaError_t launch_backward_rows(const BwdProblem& b, cudaStream_t stream) {
    const int Sq_pad = (int)backward_sq_pad(b.Sq), n_qt = (b.Sq + TR - 1) / TR;
    bwd_rows_kernel<<<dim3(n_qt, b.B), TR, 0, stream>>>(reinterpret_cast<const int2*>(b.row_bounds),
                                                        reinterpret_cast<int2*>(b.ws_rows),
                                                        reinterpret_cast<int4*>(b.ws_summ), b.Sq, b.Sk, Sq_pad, n_qt,
                                                        b.causal, b.wl, b.wr);
    return cudaGetLastError();
}

cudaError_t launch_backward_bf16(const BwdProblem& b, const CUtensorMap& tq, const CUtensorMap& tdo,
                                 const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                                 cudaStream_t stream, cudaEvent_t* ev) {
    BParams p{};
    p.dq = static_cast<uint16_t*>(b.dq);
    p.dk = static_cast<uint16_t*>(b.dk);
    p.dv = static_cast<uint16_t*>(b.dv);
    p.lse2 = b.ws_lse2;
    p.delta = b.ws_delta;
    p.lse2_w = b.ws_lse2;
    p.delta_w = b.ws_delta;
    p.lse = b.lse;
    p.rows = reinterpret_cast<const int2*>(b.ws_rows);
    p.summ = reinterpret_cast<const int4*>(b.ws_summ);
    p.slopes = b.slopes;
    p.status = b.status;
    p.timeout_ns = b.timeout_ns;
    p.B = b.B;
    p.Hq = b.Hq;
    p.Hkv = b.Hkv;
    p.Sq = b.Sq;
    p.Sk = b.Sk;
    p.G = b.Hq / b.Hkv;
    p.Sq_pad = (int)backward_sq_pad(b.Sq);
    p.n_qt = (b.Sq + TR - 1) / TR;
    p.n_kt = (b.Sk + TR - 1) / TR;
    p.causal = b.causal;
    p.scale = b.scale;
    p.scale_log2 = b.scale * LOG2E;
    p.cap_in = b.softcap > 0.f ? b.scale / b.softcap : 0.f;
    p.cap_out = b.softcap * LOG2E;
    p.wide_store = ((reinterpret_cast<uintptr_t>(b.dq) | reinterpret_cast<uintptr_t>(b.dk) |
                     reinterpret_cast<uintptr_t>(b.dv)) & 31u) == 0;

    cudaError_t e;
    if (ev && (e = cudaEventRecord(ev[0], stream)) != cudaSuccess) return e;
    if ((e = launch_backward_rows(b, stream)) != cudaSuccess) return e;
    if (ev && (e = cudaEventRecord(ev[1], stream)) != cudaSuccess) return e;

    const int items_a = p.n_kt * b.B * b.Hkv, items_b = p.n_qt * b.B * b.Hq;
    const int grid_a = items_a < b.num_sms ? items_a : b.num_sms;
    const int grid_b = items_b < b.num_sms ? items_b : b.num_sms;
    const bool cap = b.softcap > 0.f, ali = b.slopes != nullptr;
    if (b.D == 128)
        return b.f16 ? launch_flags<128, true>(p, grid_a, grid_b, cap, ali, tq, tdo, tk, tv, to, stream, ev)
                     : launch_flags<128, false>(p, grid_a, grid_b, cap, ali, tq, tdo, tk, tv, to, stream, ev);
    return b.f16 ? launch_flags<64, true>(p, grid_a, grid_b, cap, ali, tq, tdo, tk, tv, to, stream, ev)
                 : launch_flags<64, false>(p, grid_a, grid_b, cap, ali, tq, tdo, tk, tv, to, stream, ev);
}

}  // namespace gbattn
