// decode_common.cuh -- pieces shared by the split-KV decode kernels: launch
// parameters, 16-bit helpers, the shared-memory tile layout, the per-sequence
// tile range, the balanced launch's work walk and the log-sum-exp combine.
//
// "gfx942 unified attention, from the math up", section 8: with one query
// row, parallelism comes from splitting the keys across thread blocks and
// combining the partial softmax-weighted outputs.  The combine is the online
// recurrence of section 3 applied across splits: LSE = log sum_s e^{lse_s},
// O = sum_s e^{lse_s - LSE} O_s, evaluated in a fixed split order.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {
namespace dec {

constexpr int TILE = 64;     // keys per tile
constexpr int NSTG = 3;      // ring stages
constexpr int CONSUMERS = 4; // consumer warps
constexpr int DEC_THREADS = (CONSUMERS + 1) * 32;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

struct DecParams {
    const uint16_t* q;   // bf16 or fp16 bits
    uint16_t* out;
    float* lse;
    const float* slopes;
    float* ws_o;
    float* ws_lse;
    unsigned int* status;
    unsigned long long timeout_ns;
    int B, Hq, Hkv, Sk, G;
    int n_chunks;       // head chunks per kv head
    int num_splits;
    int chunk_tiles;    // tiles per split
    int n_tiles;        // tiles over Sk
    float qscale;       // multiplies q: scale * log2(e) (no softcap) or scale (softcap)
    float softcap;
    int wl;             // left window (-1: none): keys j >= len - 1 - wl
    // balanced launch: the CTAs split the concatenated tile streams evenly
    int grid_balanced;  // CTAs of a balanced launch (two per SM)
    // paged cache: tile t of sequence b gathers keys [64 t, 64 t + 64) block by block
    const uint32_t* block_table;   // [B, max_blocks]
    const uint32_t* context_lens;  // [B]
    int max_blocks, bs_log2, num_blocks;
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// low / high 16-bit element of a packed pair, bf16 or fp16
template <bool F16>
__device__ __forceinline__ float lo16(uint32_t w) {
    return F16 ? __half2float(__ushort_as_half((unsigned short)(w & 0xffffu))) : bf16lo(w);
}
template <bool F16>
__device__ __forceinline__ float hi16(uint32_t w) {
    return F16 ? __half2float(__ushort_as_half((unsigned short)(w >> 16))) : bf16hi(w);
}
// fp32 -> the 16-bit storage type (round to nearest even), as bits
template <bool F16>
__device__ __forceinline__ uint16_t to16(float v) {
    return F16 ? __half_as_ushort(__float2half_rn(v)) : __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

template <int D>
struct DCfg {
    static constexpr int SLABS = D / 64;
    static constexpr int SLAB = TILE * 128;           // bytes of one 64-wide slab of a tile
    static constexpr int TILE_BYTES = TILE * D * 2;   // K or V tile
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int SMEM = NSTG * STAGE_BYTES + 1024;
};

// Byte offset of 16-byte chunk `c` (0..7) of row `r` inside a 128-byte-swizzled slab.
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// The keys of sequence b: all Sk, or (paged cache) its context length capped at
// what the block table holds.  The query is the newest token, at position
// len - 1: a left window admits keys j >= len - 1 - wl.  Its tiles run from the
// one holding the first admitted key to the last.
struct SeqTiles {
    int len, k_first, t_first, n;  // n: tiles to visit
};
template <bool PAGED>
__device__ __forceinline__ SeqTiles seq_tiles(const DecParams& p, int b) {
    SeqTiles q;
    q.len = p.Sk;
    if (PAGED) {
        const uint32_t c = __ldg(p.context_lens + b);
        q.len = c > (uint32_t)p.Sk ? p.Sk : (int)c;
    }
    q.k_first = p.wl >= 0 ? max(0, q.len - 1 - p.wl) : 0;
    q.t_first = q.k_first / TILE;
    q.n = max(0, (q.len + TILE - 1) / TILE - q.t_first);
    return q;
}

// Tiles per CTA of a balanced launch: an even share of all streams' tiles,
// but no fewer than a longest stream of n_max tiles can be cut into with at
// most num_splits pieces (a run of n tiles meets at most
// ceil((n - 1) / share) + 1 shares).
__device__ __forceinline__ long long balanced_share(long long total, int n_max, int num_splits, int grid) {
    const long long per = (total + grid - 1) / grid;
    const long long floor_ = (n_max + num_splits - 2) / (num_splits - 1);
    return per > floor_ ? per : floor_;
}
// Contiguous: every sequence has the same tiles, so the share follows from the
// launch parameters alone.
template <bool PAGED>
__device__ __forceinline__ int dense_share(const DecParams& p) {
    const int n = seq_tiles<PAGED>(p, 0).n;
    return (int)balanced_share((long long)p.B * p.Hkv * p.n_chunks * n, n, p.num_splits, (int)gridDim.x);
}

// A run of tiles of one stream (b, kv head, head chunk), and the partial it
// produces: slot k of the stream's num_splits slots.
struct Seg {
    int b, hkv, hc;
    int t0, t1;  // tiles [t0, t1)
    int k;
    bool last;   // the stream's last run: slots after k are unused
    SeqTiles sq;
};

// The runs a CTA of a balanced launch works through, enumerated the same way
// by every role: the streams (b-major, then kv head, then head chunk) laid end
// to end; CTA c takes positions [c * share, (c + 1) * share), which start at
// stream position (b0, r0, t) with sequence b0's first stream at global
// position pb0 (found by the CTA's scan over the context lengths, paged) or
// by arithmetic (contiguous: the walk keeps only pos).
template <bool PAGED>
struct Walker {
    int b, r, t;
    int pos, end, pb, share;  // tile positions: below 2^31 (B Hq Sk < 2^31 and 64-key tiles)
    int c;
    bool done;
    SeqTiles sq;
    __device__ __forceinline__ bool next(const DecParams& q, Seg& g) {
        const DecParams* p = &q;
        if (done) return false;
        const int R = p->Hkv * p->n_chunks;
        if (!PAGED) {
            // every sequence has the same tiles: the run follows from pos alone
            const int shr = dense_share<PAGED>(*p), stop = ((int)blockIdx.x + 1) * shr;
            if (pos >= stop) {
                done = true;
                return false;
            }
            const SeqTiles q1 = seq_tiles<PAGED>(*p, 0);
            const int per_b = R * q1.n;
            const int bb = pos / per_b, rem = pos - bb * per_b, rr = rem / q1.n, tt = rem - rr * q1.n;
            if (bb >= p->B) {
                done = true;
                return false;
            }
            const int n = min(q1.n - tt, stop - pos);
            g.b = bb;
            g.hkv = rr / p->n_chunks;
            g.hc = rr % p->n_chunks;
            g.sq = q1;
            g.t0 = q1.t_first + tt;
            g.t1 = g.t0 + n;
            g.k = pos / shr - (bb * per_b + rr * q1.n) / shr;
            g.last = tt + n == q1.n;
            pos += n;
            return true;
        }
        while (pos < end && b < p->B) {
            if (t == 0 && r == 0) sq = seq_tiles<PAGED>(*p, b);
            if (sq.n == 0) {
                ++b;
                continue;
            }
            const int o = pb + r * sq.n;  // the stream's first position
            const int n = min(sq.n - t, end - pos);
            g.b = b;
            g.hkv = r / p->n_chunks;
            g.hc = r % p->n_chunks;
            g.sq = sq;
            g.t0 = sq.t_first + t;
            g.t1 = g.t0 + n;
            g.k = pos / share - o / share;
            g.last = t + n == sq.n;
            pos += n;
            t += n;
            if (t == sq.n) {
                t = 0;
                if (++r == R) {
                    r = 0;
                    pb += R * sq.n;
                    ++b;
                }
            }
            return true;
        }
        done = true;
        return false;
    }
};

// Combine: one block per (b, h) row, one thread per output dimension.  A
// row whose sequence has no key to visit (an empty paged context) has no
// partials: its output is the zero row.  Slots with lse -inf carry no weight
// and their o is not read.
template <int D, bool F16>
__global__ void __launch_bounds__(D) decode_combine_kernel(const float* __restrict__ ws_o,
                                                           const float* __restrict__ ws_lse,
                                                           uint16_t* __restrict__ out, float* __restrict__ lse,
                                                           int num_splits, float lse_to_natural,
                                                           const uint32_t* __restrict__ context_lens, int Hq) {
    const size_t row = blockIdx.x;
    const int d = threadIdx.x;
    const bool empty = context_lens && __ldg(context_lens + row / Hq) == 0u;
    // launched as a programmatic dependent of the decode kernel: its partials
    // are complete and visible after this wait
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float* ls = ws_lse + row * num_splits;
    float M = -INFINITY;
    if (!empty)
        for (int s = 0; s < num_splits; ++s) M = fmaxf(M, ls[s]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < num_splits; ++s) {
            if (ls[s] == -INFINITY) continue;
            const float w = ex2_approx(ls[s] - M);
            L += w;
            O += w * ws_o[(row * num_splits + s) * D + d];
        }
    }
    out[row * D + d] = to16<F16>(L > 0.f ? O / L : 0.f);
    if (lse && d == 0) lse[row] = (L > 0.f) ? (M + log2f(L)) * lse_to_natural : -INFINITY;
}

// The balanced kernel's launch (decode_balanced.cu); the combine follows it
// in launch_decode_bf16.
cudaError_t launch_balanced(const DecParams& p, int D, int GC, bool cap, bool ali, bool paged, bool f16,
                            const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream);

}  // namespace dec
}  // namespace gbattn
