// decode_bf16.cu -- split-KV decode (one query row per head), the split
// plan, and the launches of the decode kernels and of the log-sum-exp combine.
//
// The path is bound by HBM reads of K and V, so it runs on the SIMT pipes:
//   * one CTA per (batch, kv head, head chunk, split) in this file's kernel
//     (fixed splits: an explicit split count, or a plan of one split); the
//     balanced kernel (decode_balanced.cu) serves automatic multi-split plans
//     with equal shares of all streams' tiles per CTA; all query heads of a
//     GQA group (up to GC of them) are served from one read of each key;
//   * a producer warp streams 64-key K and V tiles with TMA into a 3-stage
//     shared-memory ring (128-byte swizzle, so the consumers' row reads are
//     free of bank conflicts);
//   * four consumer warps take 16 keys of each tile each and keep their own
//     running (m, l, o) per head, merged once at the end of the split.
// Scores: lane (key kq, dimension group dq) dots D/8 dimensions against every
// head with packed FFMA2 and a shuffle reduce-scatter sums the groups.  P V:
// lane owns D/32 output dimensions; probabilities reach it through a small
// per-warp shared buffer.
//
// Template flags: PAGED reads K and V through a block table from a pool
// [num_blocks, block_size, Hkv, D] (attention.fkc.md, "attention_paged_naive"),
// with per-sequence context lengths; F16 reads and writes fp16 instead of bf16.
#include "decode_common.cuh"

namespace gbattn {
namespace {

using namespace dec;

template <int D, int GC, bool SOFTCAP, bool ALIBI, bool PAGED, bool F16>
__global__ void __launch_bounds__(DEC_THREADS, 2)
    decode_bf16_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const DecParams p) {
    using C = DCfg<D>;
    constexpr int DV = D / 32;   // dims per lane in P V
    extern __shared__ __align__(1024) uint8_t dyn_smem[];
    __shared__ uint64_t full_bar[NSTG], empty_bar[NSTG];
    __shared__ int abort_flag;
    __shared__ __align__(16) float2 p_s[CONSUMERS][16][GC];  // (p, p) per key and head
    __shared__ __align__(16) float2 a_s[CONSUMERS][GC];      // (alpha, alpha) per head
    __shared__ float red_m[CONSUMERS][GC], red_l[CONSUMERS][GC];
    __shared__ __align__(16) float red_o[CONSUMERS][GC][D];

    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // blockIdx.x -> (b, hkv, chunk, split)
    int rem = blockIdx.x;
    const int split = rem % p.num_splits;
    rem /= p.num_splits;
    const int hc = rem % p.n_chunks;
    rem /= p.n_chunks;
    const int hkv = rem % p.Hkv;
    const int b = rem / p.Hkv;
    // Keys of this sequence: all Sk, or (paged cache) its context length,
    // capped at what the block table can hold.  The query is the newest token,
    // at position len - 1: the ALiBi term is slope (j - (len - 1)) and a left
    // window admits keys j >= len - 1 - wl.  The splits cover the 64-key tiles
    // from the window's first key to the last key.
    int len = p.Sk;
    if (PAGED) {
        const uint32_t c = __ldg(p.context_lens + b);
        len = c > (uint32_t)p.Sk ? p.Sk : (int)c;
        if (c > (uint32_t)p.Sk && threadIdx.x == 0 && split == 0 && hc == 0) atomicOr(p.status, ST_DECODE_PAGED_RANGE);
    }
    const int k_first = p.wl >= 0 ? max(0, len - 1 - p.wl) : 0;  // first admitted key
    const int t_begin = k_first / TILE + split * p.chunk_tiles;
    const int t_end = min(PAGED ? (len + TILE - 1) / TILE : p.n_tiles, t_begin + p.chunk_tiles);
    const int h0 = hkv * p.G + hc * GC;                     // first query head of this chunk
    const int n_heads = min(GC, p.G - hc * GC);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTG; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], CONSUMERS);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // the combine (a programmatic dependent launch) may be scheduled once every
    // CTA of this grid has started; it waits on the device for this grid's end
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    WaitCtl wc{&abort_flag, p.status, p.timeout_ns};

    if (warp == CONSUMERS) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            uint32_t cnt = 0;
            bool ok = true;
            const int plane = b * p.Hkv + hkv;
            for (int t = t_begin; t < t_end; ++t, ++cnt) {
                const int st = cnt % NSTG;
                ok = mbar_wait(&empty_bar[st], ((cnt / NSTG) & 1) ^ 1, wc, ST_DECODE_PRODUCER);
                if (!ok) break;
                mbar_arrive_expect_tx(&full_bar[st], C::STAGE_BYTES);
                uint8_t* ks = ring + st * C::STAGE_BYTES;
                uint8_t* vs = ks + C::TILE_BYTES;
                if (PAGED) {
                    // one load per block (block_size < 64) or per 64 rows of a block;
                    // keys past the context and bad block indices load from past the
                    // pool's end, which reads zeros (the keys are masked anyway)
                    const int rpl = min(1 << p.bs_log2, TILE);
                    for (int i = 0; i < TILE / rpl; ++i) {
                        const int kp = t * TILE + i * rpl;
                        int z = p.num_blocks << p.bs_log2;
                        if (kp < len) {
                            const uint32_t blk = __ldg(p.block_table + (size_t)b * p.max_blocks + (kp >> p.bs_log2));
                            if (blk < (uint32_t)p.num_blocks)
                                z = ((int)blk << p.bs_log2) + (kp & ((1 << p.bs_log2) - 1));
                            else
                                atomicOr(p.status, ST_DECODE_PAGED_RANGE);
                        }
#pragma unroll
                        for (int sl = 0; sl < C::SLABS; ++sl) {
                            tma_load_3d(ks + sl * C::SLAB + i * rpl * 128, &tmK, &full_bar[st], sl * 64, hkv, z);
                            tma_load_3d(vs + sl * C::SLAB + i * rpl * 128, &tmV, &full_bar[st], sl * 64, hkv, z);
                        }
                    }
                } else {
#pragma unroll
                    for (int sl = 0; sl < C::SLABS; ++sl) {
                        tma_load_3d(ks + sl * C::SLAB, &tmK, &full_bar[st], sl * 64, t * TILE, plane);
                        tma_load_3d(vs + sl * C::SLAB, &tmV, &full_bar[st], sl * 64, t * TILE, plane);
                    }
                }
            }
            if (!ok) {
                const uint32_t n = cnt < (uint32_t)NSTG ? cnt : (uint32_t)NSTG;
                for (uint32_t i = cnt - n; i < cnt; ++i) mbar_drain(&full_bar[i % NSTG], (i / NSTG) & 1, 100000000ull);
            }
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    // Scores: lane = (key kq in 0..3, dimension group dq in 0..7).  A lane dots
    // D/8 dimensions of one key against every head of the chunk (packed FFMA2),
    // then a reduce-scatter over the 8 dimension-group lanes leaves one head's
    // full score in each lane (head hsel, duplicated in the 8/GC lanes that
    // differ only in dq's low bits).  P V: lane owns D/32 output dimensions of
    // every head; probabilities and rescale factors reach it through shared memory.
    constexpr int DQ = D / 8;
    constexpr int DUP = 8 / GC;  // lanes holding the same head after the reduce-scatter
    const int kq = lane >> 3, dq = lane & 7;
    int hsel = 0;
    if (GC >= 2) hsel += ((dq >> 2) & 1) * (GC / 2);
    if (GC >= 4) hsel += ((dq >> 1) & 1) * (GC / 4);
    if (GC >= 8) hsel += (dq & 1);
    const bool writer = (dq & (DUP - 1)) == 0;

    float2 q2[GC][DQ / 2];
#pragma unroll
    for (int h = 0; h < GC; ++h) {
        const bool hv = h < n_heads;
        const uint16_t* qp = p.q + (size_t)(b * p.Hq + h0 + (hv ? h : 0)) * D + dq * DQ;
#pragma unroll
        for (int d = 0; d < DQ; d += 8) {
            const uint4 w = hv ? *reinterpret_cast<const uint4*>(qp + d) : make_uint4(0, 0, 0, 0);
            q2[h][d / 2 + 0] = make_float2(lo16<F16>(w.x) * p.qscale, hi16<F16>(w.x) * p.qscale);
            q2[h][d / 2 + 1] = make_float2(lo16<F16>(w.y) * p.qscale, hi16<F16>(w.y) * p.qscale);
            q2[h][d / 2 + 2] = make_float2(lo16<F16>(w.z) * p.qscale, hi16<F16>(w.z) * p.qscale);
            q2[h][d / 2 + 3] = make_float2(lo16<F16>(w.w) * p.qscale, hi16<F16>(w.w) * p.qscale);
        }
    }
    const float slope_l2 = (ALIBI && hsel < n_heads) ? p.slopes[h0 + hsel] * LOG2E : 0.f;

    float m_h = -INFINITY, l_h = 0.f;  // running max / partial sum of this lane's head and keys
    float2 o2[GC][DV / 2];
#pragma unroll
    for (int h = 0; h < GC; ++h)
#pragma unroll
        for (int c = 0; c < DV / 2; ++c) o2[h][c] = make_float2(0.f, 0.f);

    uint32_t cnt = 0;
    bool ok = true;
    for (int t = t_begin; t < t_end; ++t, ++cnt) {
        const int st = cnt % NSTG;
        ok = mbar_wait(&full_bar[st], (cnt / NSTG) & 1, wc, ST_DECODE_CONSUMER);
        if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
        }
        const uint8_t* ks = ring + st * C::STAGE_BYTES;
        const uint8_t* vs = ks + C::TILE_BYTES;

        // ---- scores: 4 passes of 4 keys, key r = 16 warp + 4 pass + kq
        float sv[4];
#pragma unroll
        for (int ps = 0; ps < 4; ++ps) {
            const int r = warp * 16 + ps * 4 + kq;
            float2 acc[GC];
#pragma unroll
            for (int h = 0; h < GC; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c8 = 0; c8 < DQ / 8; ++c8) {
                const int dim = dq * DQ + c8 * 8;
                const int slab = dim >> 6, chunk = (dim & 63) >> 3;
                const uint4 w = *reinterpret_cast<const uint4*>(ks + slab * C::SLAB + swz(r, chunk));
                const float2 k2[4] = {make_float2(lo16<F16>(w.x), hi16<F16>(w.x)),
                                      make_float2(lo16<F16>(w.y), hi16<F16>(w.y)),
                                      make_float2(lo16<F16>(w.z), hi16<F16>(w.z)),
                                      make_float2(lo16<F16>(w.w), hi16<F16>(w.w))};
#pragma unroll
                for (int h = 0; h < GC; ++h)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[h] = __ffma2_rn(q2[h][c8 * 4 + i], k2[i], acc[h]);
            }
            float v[GC];
#pragma unroll
            for (int h = 0; h < GC; ++h) v[h] = acc[h].x + acc[h].y;
            // reduce-scatter over the 8 dimension-group lanes (xor 4, 2, 1)
            int n = GC;
#pragma unroll
            for (int lv = 0; lv < 3; ++lv) {
                const int mask = 4 >> lv;
                if (n >= 2) {
                    const bool up = (dq & mask) != 0;
                    const int half = n / 2;
#pragma unroll
                    for (int i = 0; i < GC / 2; ++i) {
                        if (i < half) {
                            const float send = up ? v[i] : v[half + i];
                            const float keep = up ? v[half + i] : v[i];
                            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
                        }
                    }
                    n = half;
                } else {
                    v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
                }
            }
            sv[ps] = v[0];
        }
        // ---- logits (base 2), mask, running max of this lane's head over the warp's 16 keys
        float mt = -INFINITY;
#pragma unroll
        for (int ps = 0; ps < 4; ++ps) {
            const int kj = t * TILE + warp * 16 + ps * 4 + kq;
            float x = sv[ps];
            if (SOFTCAP) {
                // cap * tanh(y) with tanh(y) = 1 - 2 / (e^{2y} + 1), y = score / cap, times log2(e)
                const float e = ex2_approx(x * (2.f * LOG2E / p.softcap));
                x = p.softcap * LOG2E * (1.f - 2.f / (e + 1.f));
            }
            if (ALIBI) x = fmaf(slope_l2, (float)(kj - (len - 1)), x);
            if (kj >= len || kj < k_first) x = -INFINITY;
            sv[ps] = x;
            mt = fmaxf(mt, x);
        }
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
        const float m_new = fmaxf(m_h, mt);
        const float alpha = (m_h == -INFINITY) ? 0.f : ex2_approx(m_h - m_new);
        const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;
        float psum = 0.f;
#pragma unroll
        for (int ps = 0; ps < 4; ++ps) {
            const float pv = ex2_approx(sv[ps] - m_ref);
            psum += pv;
            if (writer) p_s[warp][ps * 4 + kq][hsel] = make_float2(pv, pv);
        }
        if (m_new != -INFINITY) {
            l_h = fmaf(l_h, alpha, psum);
            m_h = m_new;
        }
        if (writer && kq == 0) a_s[warp][hsel] = (m_new != -INFINITY) ? make_float2(alpha, alpha) : make_float2(1.f, 1.f);
        __syncwarp();
        // ---- rescale and P V over the warp's 16 keys; lane owns dims [lane*DV, lane*DV + DV)
#pragma unroll
        for (int h = 0; h < GC; ++h) {
            const float2 a2 = a_s[warp][h];
#pragma unroll
            for (int c = 0; c < DV / 2; ++c) o2[h][c] = __fmul2_rn(o2[h][c], a2);
        }
        {
            const int dim = lane * DV;
            const int slab = dim >> 6, chunk = (dim & 63) >> 3, within = (dim & 7) * 2;  // bytes
#pragma unroll 4
            for (int j = 0; j < 16; ++j) {
                const int r = warp * 16 + j;
                const uint8_t* vp = vs + slab * C::SLAB + swz(r, chunk) + within;
                float2 v2[DV / 2];
                if (DV == 4) {
                    const uint2 w = *reinterpret_cast<const uint2*>(vp);
                    v2[0] = make_float2(lo16<F16>(w.x), hi16<F16>(w.x));
                    v2[DV / 2 - 1] = make_float2(lo16<F16>(w.y), hi16<F16>(w.y));
                } else {
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(vp);
                    v2[0] = make_float2(lo16<F16>(w), hi16<F16>(w));
                }
#pragma unroll
                for (int h = 0; h < GC; ++h) {
                    const float2 pp = p_s[warp][j][h];
#pragma unroll
                    for (int c = 0; c < DV / 2; ++c) o2[h][c] = __ffma2_rn(pp, v2[c], o2[h][c]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[st]);
    }

    // ---- merge the four warps' states (fixed order), then write
    l_h += __shfl_xor_sync(0xffffffffu, l_h, 8);
    l_h += __shfl_xor_sync(0xffffffffu, l_h, 16);
    if (writer && kq == 0) {
        red_m[warp][hsel] = m_h;
        red_l[warp][hsel] = l_h;
    }
#pragma unroll
    for (int h = 0; h < GC; ++h)
#pragma unroll
        for (int c = 0; c < DV / 2; ++c)
            *reinterpret_cast<float2*>(&red_o[warp][h][lane * DV + 2 * c]) = o2[h][c];
    asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS * 32) : "memory");
    if (!ok || abort_flag) return;

    const int tid = threadIdx.x;  // 0 .. 127
    for (int i = tid; i < n_heads * D; i += CONSUMERS * 32) {
        const int h = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < CONSUMERS; ++w) M = fmaxf(M, red_m[w][h]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < CONSUMERS; ++w) {
                const float f = (red_m[w][h] == -INFINITY) ? 0.f : ex2_approx(red_m[w][h] - M);
                L += red_l[w][h] * f;
                O += red_o[w][h][d] * f;
            }
        }
        const float val = (L > 0.f) ? O / L : 0.f;
        const float lse2 = (L > 0.f) ? M + log2f(L) : -INFINITY;  // base 2
        const int head = h0 + h;
        const size_t row = (size_t)b * p.Hq + head;
        if (p.num_splits == 1) {
            p.out[row * D + d] = to16<F16>(val);
            if (p.lse && d == 0) p.lse[row] = lse2 * LN2;
        } else {
            const size_t prow = row * p.num_splits + split;
            p.ws_o[prow * D + d] = val;
            if (d == 0) p.ws_lse[prow] = lse2;
        }
    }
}

template <int D, int GC, bool SOFTCAP, bool ALIBI, bool PAGED, bool F16>
cudaError_t launch_dec(const DecParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
    auto kern = decode_bf16_kernel<D, GC, SOFTCAP, ALIBI, PAGED, F16>;
    const int smem = DCfg<D>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long grid = (long long)p.B * p.Hkv * p.n_chunks * p.num_splits;
    kern<<<(unsigned)grid, DEC_THREADS, smem, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

template <int D, int GC, bool PAGED, bool F16>
cudaError_t launch_dec_caps(const DecParams& p, bool cap, bool ali, const CUtensorMap& tk, const CUtensorMap& tv,
                            cudaStream_t s) {
    if (cap)
        return ali ? launch_dec<D, GC, true, true, PAGED, F16>(p, tk, tv, s)
                   : launch_dec<D, GC, true, false, PAGED, F16>(p, tk, tv, s);
    return ali ? launch_dec<D, GC, false, true, PAGED, F16>(p, tk, tv, s)
               : launch_dec<D, GC, false, false, PAGED, F16>(p, tk, tv, s);
}

template <int D, int GC>
cudaError_t launch_dec_flags(const DecParams& p, bool cap, bool ali, bool paged, bool f16, const CUtensorMap& tk,
                             const CUtensorMap& tv, cudaStream_t s) {
    if (f16)
        return paged ? launch_dec_caps<D, GC, true, true>(p, cap, ali, tk, tv, s)
                     : launch_dec_caps<D, GC, false, true>(p, cap, ali, tk, tv, s);
    return paged ? launch_dec_caps<D, GC, true, false>(p, cap, ali, tk, tv, s)
                 : launch_dec_caps<D, GC, false, false>(p, cap, ali, tk, tv, s);
}

}  // namespace

void decode_split_plan(int B, int Hkv, int Sk, int num_sms, int requested, int* num_splits, int* chunk) {
    const int tiles = (Sk + TILE - 1) / TILE;
    int s_best = 1;
    if (requested > 0) {
        s_best = requested < tiles ? requested : tiles;
    } else {
        // Time of a split count s, in tiles streamed by one CTA: waves of
        // resident CTAs (2 per SM) times (tiles per split + a fixed cost of about
        // three tiles per CTA: loading q, merging the warps, writing the partial,
        // and its share of the combine), as measured on GB300 decode shapes.
        // With fewer than about three waves of CTAs in flight the per-CTA
        // streaming rate, not HBM, bounds the decode, so s starts there.
        const long long rows = (long long)B * Hkv;
        const long long slots = (long long)(num_sms > 0 ? num_sms : 1) * 2;
        const int s_cap = tiles < 256 ? tiles : 256;
        long long s_min = (3 * slots + rows - 1) / rows;
        if (s_min > s_cap) s_min = s_cap;
        if (s_min < 1) s_min = 1;
        long long best = -1;
        for (int s = (int)s_min; s <= s_cap; ++s) {
            const int ct = (tiles + s - 1) / s;
            if ((tiles + ct - 1) / ct != s) continue;  // same chunking as a smaller s
            const long long waves = (rows * s + slots - 1) / slots;
            const long long cost = waves * (ct + 3);
            if (best < 0 || cost < best) {
                best = cost;
                s_best = s;
            }
        }
    }
    const int ct = (tiles + s_best - 1) / s_best;
    *num_splits = (tiles + ct - 1) / ct;
    *chunk = ct * TILE;
}

cudaError_t launch_decode_bf16(const DecodeProblem& f, const CUtensorMap& tk, const CUtensorMap& tv,
                               cudaStream_t stream) {
    DecParams p{};
    p.q = static_cast<const uint16_t*>(f.q);
    p.out = static_cast<uint16_t*>(f.out);
    p.lse = f.lse;
    p.slopes = f.slopes;
    p.ws_o = f.ws_o;
    p.ws_lse = f.ws_lse;
    p.status = f.status;
    p.timeout_ns = f.timeout_ns;
    p.B = f.B;
    p.Hq = f.Hq;
    p.Hkv = f.Hkv;
    p.Sk = f.Sk;
    p.G = f.Hq / f.Hkv;
    p.num_splits = f.num_splits;
    p.wl = f.wl;
    p.chunk_tiles = f.chunk / TILE;
    p.n_tiles = (f.Sk + TILE - 1) / TILE;
    p.softcap = f.softcap;
    const bool paged = f.paged != 0;
    if (paged) {
        p.block_table = f.block_table;
        p.context_lens = f.context_lens;
        p.max_blocks = f.max_blocks;
        p.num_blocks = f.num_blocks;
        int lg = 0;
        while ((1 << lg) < f.block_size) ++lg;
        p.bs_log2 = lg;
    }
    const bool cap = f.softcap > 0.f, ali = f.slopes != nullptr;
    p.qscale = cap ? f.scale : f.scale * LOG2E;
    const int G = p.G;
    const int GC = f.D == 128 ? (G >= 3 ? 4 : (G == 2 ? 2 : 1)) : (G >= 5 ? 8 : (G >= 3 ? 4 : (G == 2 ? 2 : 1)));
    p.n_chunks = (G + GC - 1) / GC;
    const bool f16 = f.f16 != 0;
    cudaError_t e;
    // An automatic multi-split plan runs balanced when the fixed splits would
    // leave SMs idle at the end: the CTAs (two per SM) take equal shares of all
    // streams' tiles laid end to end.  That pays for uneven paged contexts and
    // for fixed-split grids of under four waves (a partial last wave weighs a
    // quarter or more); with more waves the fixed-split kernel is as fast (on
    // GB300: B64 Hkv8 Sk8192, 6.7 waves: 6450 GB/s fixed against 6296 balanced;
    // B16, 3.4 waves: 5162 against 5422; paged with contexts 4096..8192: 5819
    // against 6018).
    const int slots = 2 * (f.num_sms > 0 ? f.num_sms : 1);
    const long long fixed_ctas = (long long)f.B * f.Hkv * p.n_chunks * f.num_splits;
    if (f.auto_splits && f.num_splits >= 2 && (paged || fixed_ctas < 4LL * slots)) {
        p.grid_balanced = slots;
        e = launch_balanced(p, f.D, GC, cap, ali, paged, f16, tk, tv, stream);
    } else if (f.D == 128) {
        e = GC == 4   ? launch_dec_flags<128, 4>(p, cap, ali, paged, f16, tk, tv, stream)
            : GC == 2 ? launch_dec_flags<128, 2>(p, cap, ali, paged, f16, tk, tv, stream)
                      : launch_dec_flags<128, 1>(p, cap, ali, paged, f16, tk, tv, stream);
    } else {
        e = GC == 8   ? launch_dec_flags<64, 8>(p, cap, ali, paged, f16, tk, tv, stream)
            : GC == 4 ? launch_dec_flags<64, 4>(p, cap, ali, paged, f16, tk, tv, stream)
            : GC == 2 ? launch_dec_flags<64, 2>(p, cap, ali, paged, f16, tk, tv, stream)
                      : launch_dec_flags<64, 1>(p, cap, ali, paged, f16, tk, tv, stream);
    }
    if (e != cudaSuccess || p.num_splits == 1) return e;
    // every partial lse is in base 2 (logits carry the log2(e) factor).  The
    // combine is a programmatic dependent launch: its blocks are scheduled
    // while the decode kernel drains and wait for its completion on the device.
    const uint32_t* lens = paged ? p.context_lens : nullptr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.B * p.Hq));
    cfg.blockDim = dim3((unsigned)f.D);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float* wo = p.ws_o;
    const float* wl = p.ws_lse;
    if (f.D == 128)
        return f16 ? cudaLaunchKernelEx(&cfg, decode_combine_kernel<128, true>, wo, wl, p.out, p.lse, p.num_splits, LN2,
                                        lens, p.Hq)
                   : cudaLaunchKernelEx(&cfg, decode_combine_kernel<128, false>, wo, wl, p.out, p.lse, p.num_splits,
                                        LN2, lens, p.Hq);
    return f16 ? cudaLaunchKernelEx(&cfg, decode_combine_kernel<64, true>, wo, wl, p.out, p.lse, p.num_splits, LN2, lens,
                                    p.Hq)
               : cudaLaunchKernelEx(&cfg, decode_combine_kernel<64, false>, wo, wl, p.out, p.lse, p.num_splits, LN2, lens,
                                    p.Hq);
}

}  // namespace gbattn
