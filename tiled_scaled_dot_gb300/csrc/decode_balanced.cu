// decode_balanced.cu -- the split-KV decode kernel of automatic multi-split
// plans: a persistent-style grid (two CTAs per SM) in which each CTA takes an
// equal share of all (sequence, kv head, head chunk) streams' 64-key tiles laid
// end to end, producing one partial (o / l, base-2 lse) per run of a stream
// for the fixed-order combine.  The tile loop is the one of decode_bf16.cu's
// kernel: a producer warp streams K and V tiles by TMA into a 3-stage ring,
// four consumer warps score 16 keys of each tile against every query head of
// the GQA group and keep running (m, l, o), merged at the end of each run.
#include "decode_common.cuh"

#include <algorithm>

namespace gbattn {
namespace {

using namespace dec;

template <int D, int GC, bool SOFTCAP, bool ALIBI, bool PAGED, bool F16>
__global__ void __launch_bounds__(DEC_THREADS, 2)
    decode_balanced_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const DecParams p) {
    using C = DCfg<D>;
    constexpr int DV = D / 32;   // dims per lane in P V
    extern __shared__ __align__(1024) uint8_t dyn_smem[];
    __shared__ uint64_t full_bar[NSTG], empty_bar[NSTG];
    __shared__ uint64_t merge_in, merge_out;  // the warps' states are in red_* / have been read
    __shared__ int abort_flag;
    __shared__ int w_start[6];                // balanced mode: b0, its first position, share, r0, t0, has work
    __shared__ Walker<PAGED> c_walk;          // the consumers' walk
    __shared__ Seg c_seg[2];                  // the consumers' current and next run
    __shared__ int c_has[2];
    __shared__ __align__(16) float2 p_s[CONSUMERS][16][GC];  // (p, p) per key and head
    __shared__ __align__(16) float2 a_s[CONSUMERS][GC];      // (alpha, alpha) per head
    __shared__ float red_m[CONSUMERS][GC], red_l[CONSUMERS][GC];
    __shared__ __align__(16) float red_o[CONSUMERS][GC][D];

    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTG; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], CONSUMERS);
        }
        mbar_init(&merge_in, CONSUMERS * 32);
        mbar_init(&merge_out, CONSUMERS * 32);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (PAGED && warp == 0) {
        // Total tiles over all streams, the longest stream, this CTA's share and
        // where it starts.
        const int R = p.Hkv * p.n_chunks;
        long long tot = 0;
        int n_max = 0;
        bool over = false;
        for (int i = lane; i < p.B; i += 32) {
            const int n = seq_tiles<PAGED>(p, i).n;
            tot += n;
            n_max = max(n_max, n);
            over |= __ldg(p.context_lens + i) > (uint32_t)p.Sk;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            tot += __shfl_xor_sync(0xffffffffu, tot, o);
            n_max = max(n_max, __shfl_xor_sync(0xffffffffu, n_max, o));
        }
        if (blockIdx.x == 0 && __any_sync(0xffffffffu, over) && lane == 0) atomicOr(p.status, ST_DECODE_PAGED_RANGE);
        const long long total = tot * R;
        const long long share = balanced_share(total, n_max, p.num_splits, (int)gridDim.x);
        const long long st = (long long)blockIdx.x * share;
        int has = st < total, found = 0;
        long long base = 0, pb0 = 0;
        int b0 = 0;
        for (int i0 = 0; has && i0 < p.B; i0 += 32) {
            const long long v = (i0 + lane < p.B) ? (long long)R * seq_tiles<PAGED>(p, i0 + lane).n : 0;
            long long inc = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            const unsigned m = __ballot_sync(0xffffffffu, base + inc > st);
            if (m) {
                const int L = __ffs(m) - 1;
                b0 = i0 + L;
                pb0 = base + __shfl_sync(0xffffffffu, inc - v, L);
                found = 1;
                break;
            }
            base += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) {
            int r0 = 0, t0 = 0;
            const int n = found ? seq_tiles<PAGED>(p, b0).n : 0;  // > 0: position st falls inside sequence b0
            has = has && n > 0;
            if (has) {
                r0 = (int)((st - pb0) / n);
                t0 = (int)((st - pb0) - (long long)r0 * n);
            }
            w_start[0] = b0;
            w_start[1] = (int)pb0;
            w_start[2] = (int)share;
            w_start[3] = r0;
            w_start[4] = t0;
            w_start[5] = has;
        }
    }
    __syncthreads();
    // the combine (a programmatic dependent launch) may be scheduled once every
    // CTA of this grid has started; it waits on the device for this grid's end
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    WaitCtl wc{&abort_flag, p.status, p.timeout_ns};

    // Every role walks the same runs.  Contiguous: each thread keeps its own
    // walker, started by arithmetic on the launch parameters (every sequence has
    // the same tiles), so its values are the same in every lane.  Paged: the
    // start comes from warp 0's scan; the consumers share one walker in shared
    // memory that thread 0 advances, handing each run over in a two-entry
    // descriptor ring.
    auto init_walker = [&](Walker<PAGED>& wk) {
        wk.c = blockIdx.x;
        wk.done = false;
        wk.b = wk.r = wk.t = wk.pb = wk.share = 0;
        wk.pos = wk.end = 0;
        if (PAGED) {
            wk.b = w_start[0];
            wk.pb = w_start[1];
            wk.share = w_start[2];
            wk.r = w_start[3];
            wk.t = w_start[4];
            wk.done = !w_start[5];
        } else {
            // the walk keeps only pos (Walker::next derives the rest)
            const int per_b = p.Hkv * p.n_chunks * seq_tiles<PAGED>(p, 0).n;  // >= 1
            wk.share = dense_share<PAGED>(p);
            wk.done = (long long)blockIdx.x * wk.share >= (long long)p.B * per_b;
        }
        if (!wk.done) {
            wk.pos = (int)blockIdx.x * wk.share;  // < total tiles (this CTA has work)
            wk.end = wk.pos + wk.share;           // the walk also stops after the last sequence
            wk.sq = seq_tiles<PAGED>(p, wk.b);
        }
    };
    if (PAGED && threadIdx.x == 0) {
        init_walker(c_walk);
        c_has[0] = c_walk.next(p, c_seg[0]);
    }
    __syncthreads();

    if (warp == CONSUMERS) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            uint32_t cnt = 0;
            bool ok = true;
            Walker<PAGED> wk;
            init_walker(wk);
            Seg g;
            while (ok && wk.next(p, g)) {
                const int plane = g.b * p.Hkv + g.hkv;
                for (int t = g.t0; t < g.t1; ++t, ++cnt) {
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
                            if (kp < g.sq.len) {
                                const uint32_t blk =
                                    __ldg(p.block_table + (size_t)g.b * p.max_blocks + (kp >> p.bs_log2));
                                if (blk < (uint32_t)p.num_blocks)
                                    z = ((int)blk << p.bs_log2) + (kp & ((1 << p.bs_log2) - 1));
                                else
                                    atomicOr(p.status, ST_DECODE_PAGED_RANGE);
                            }
#pragma unroll
                            for (int sl = 0; sl < C::SLABS; ++sl) {
                                tma_load_3d(ks + sl * C::SLAB + i * rpl * 128, &tmK, &full_bar[st], sl * 64, g.hkv, z);
                                tma_load_3d(vs + sl * C::SLAB + i * rpl * 128, &tmV, &full_bar[st], sl * 64, g.hkv, z);
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

    uint32_t cnt = 0;
    bool ok = true;
    // One run: its tiles, then the merge of the four warps' states and its
    // result.  Returns false when a wait gave up.
    auto run_seg = [&](const Seg& g, const uint32_t nseg) -> bool {
        const int x = nseg & 1;
        const int len = g.sq.len, k_first = g.sq.k_first;
        const int t0 = g.t0, t1 = g.t1, gb = g.b;
        const int h0 = g.hkv * p.G + g.hc * GC;  // first query head of this chunk
        const int n_heads = min(GC, p.G - g.hc * GC);
        float2 q2[GC][DQ / 2];
#pragma unroll
        for (int h = 0; h < GC; ++h) {
            const bool hv = h < n_heads;
            const uint16_t* qp = p.q + (size_t)(gb * p.Hq + h0 + (hv ? h : 0)) * D + dq * DQ;
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

        for (int t = t0; t < t1; ++t, ++cnt) {
            const int st = cnt % NSTG;
            ok = mbar_wait(&full_bar[st], (cnt / NSTG) & 1, wc, ST_DECODE_CONSUMER);
            if (!__all_sync(0xffffffffu, ok)) return false;
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
            if (writer && kq == 0)
                a_s[warp][hsel] = (m_new != -INFINITY) ? make_float2(alpha, alpha) : make_float2(1.f, 1.f);
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
        if (!ok) return false;

        // ---- merge the four warps' states (fixed order), then write the run's result
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
        mbar_arrive(&merge_in);
        ok = mbar_wait(&merge_in, nseg & 1u, wc, ST_DECODE_CONSUMER);
        if (!__all_sync(0xffffffffu, ok && !abort_flag)) return false;
        // paged: the next run, into the other descriptor (last read before this run's start)
        if (PAGED && threadIdx.x == 0) c_has[x ^ 1] = c_walk.next(p, c_seg[x ^ 1]);
        const int gk = c_seg[x].k, gb2 = c_seg[x].b;
        const bool glast = c_seg[x].last;
        const int h02 = c_seg[x].hkv * p.G + c_seg[x].hc * GC;
        const int n_heads2 = min(GC, p.G - c_seg[x].hc * GC);

        const int tid = threadIdx.x;  // 0 .. 127
        for (int i = tid; i < n_heads2 * D; i += CONSUMERS * 32) {
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
            const size_t row = (size_t)gb2 * p.Hq + h02 + h;
            if (p.num_splits == 1) {
                p.out[row * D + d] = to16<F16>(val);
                if (p.lse && d == 0) p.lse[row] = lse2 * LN2;
            } else if (gk < p.num_splits) {
                const size_t prow = row * p.num_splits + gk;
                p.ws_o[prow * D + d] = val;
                if (d == 0) {
                    p.ws_lse[prow] = lse2;
                    // the stream's unused slots
                    if (glast)
                        for (int k2 = gk + 1; k2 < p.num_splits; ++k2) p.ws_lse[row * p.num_splits + k2] = -INFINITY;
                }
            }
        }
        // red_* may be rewritten, and the next run's descriptor read, once
        // every consumer thread is here
        mbar_arrive(&merge_out);
        ok = mbar_wait(&merge_out, nseg & 1u, wc, ST_DECODE_CONSUMER);
        return __all_sync(0xffffffffu, ok);
    };
    // The next run: paged from the shared descriptor ring, contiguous from the
    // thread's own walker (thread 0 also publishes it for the write-out).
    Walker<PAGED> wk;  // contiguous only
    if (!PAGED) init_walker(wk);
    auto next_seg = [&](Seg& g, const uint32_t nseg) -> bool {
        const int x = nseg & 1;
        if (PAGED) {
            if (!c_has[x]) return false;
            g.b = c_seg[x].b;
            g.hkv = c_seg[x].hkv;
            g.hc = c_seg[x].hc;
            g.t0 = c_seg[x].t0;
            g.t1 = c_seg[x].t1;
            g.sq.len = c_seg[x].sq.len;
            g.sq.k_first = c_seg[x].sq.k_first;
            return true;
        }
        if (!wk.next(p, g)) return false;
        if (threadIdx.x == 0) c_seg[x] = g;  // read back after the tiles, behind merge_in
        return true;
    };
    Seg g;
    for (uint32_t nseg = 0; next_seg(g, nseg); ++nseg)
        if (!run_seg(g, nseg)) break;
}

template <int D, int GC, bool SOFTCAP, bool ALIBI, bool PAGED, bool F16>
cudaError_t launch_dec(const DecParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
    auto kern = decode_balanced_kernel<D, GC, SOFTCAP, ALIBI, PAGED, F16>;
    const int smem = DCfg<D>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)p.grid_balanced, DEC_THREADS, smem, stream>>>(tk, tv, p);
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

namespace dec {

cudaError_t launch_balanced(const DecParams& p, int D, int GC, bool cap, bool ali, bool paged, bool f16,
                            const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
    if (D == 128) {
        if (GC == 4) return launch_dec_flags<128, 4>(p, cap, ali, paged, f16, tk, tv, stream);
        if (GC == 2) return launch_dec_flags<128, 2>(p, cap, ali, paged, f16, tk, tv, stream);
        return launch_dec_flags<128, 1>(p, cap, ali, paged, f16, tk, tv, stream);
    }
    if (GC == 8) return launch_dec_flags<64, 8>(p, cap, ali, paged, f16, tk, tv, stream);
    if (GC == 4) return launch_dec_flags<64, 4>(p, cap, ali, paged, f16, tk, tv, stream);
    if (GC == 2) return launch_dec_flags<64, 2>(p, cap, ali, paged, f16, tk, tv, stream);
    return launch_dec_flags<64, 1>(p, cap, ali, paged, f16, tk, tv, stream);
}

}  // namespace dec
}  // namespace gbattn
