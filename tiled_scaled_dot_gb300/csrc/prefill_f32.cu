// prefill_f32.cu -- fp32 attention forward with SIMT FFMA (no TF32: its 10-bit
// mantissa cannot meet a 1e-4 max-abs bar).
//
// The tiled online-softmax recurrence of "gfx942 unified attention", section 3,
// per query row, over key tiles of 32 staged in shared memory; the operation
// is attention.fkc.md, attention_naive (scale, softcap, ALiBi, causal /
// window / per-row mask, GQA, fully-masked row -> zeros).  Every tile
// rescales exactly (alpha = 2^(m_old - m_new)), in fp32.
//
// Block: 128 threads; D / 64 threads per query row, each holding 64 of the
// row's dimensions of q and of the running output in registers.
#include "kernels.h"

namespace gbattn {
namespace {

constexpr int KT = 32;  // keys per shared-memory tile
constexpr float LOG2E_F = 1.4426950408889634f;
constexpr float LN2_F = 0.6931471805599453f;

struct Params32 {
    const float* q;
    const float* k;
    const float* v;
    float* out;
    float* lse;
    const float* slopes;
    const int2* rowb;
    int B, Hq, Hkv, Sq, Sk, G;
    int causal, wl, wr;
    float scale;
    float softcap;
};

template <int D, bool SOFTCAP, bool ALIBI>
__global__ void __launch_bounds__(128) prefill_f32_kernel(const Params32 p) {
    constexpr int TPR = D / 64;            // threads per row
    constexpr int ROWS = 128 / TPR;        // rows per block
    constexpr int HALF_STRIDE = 64 + 4;    // floats per 64-wide half row in smem (skewed)
    constexpr int ROW_STRIDE = TPR * HALF_STRIDE;
    __shared__ __align__(16) float Ks[KT * ROW_STRIDE];
    __shared__ __align__(16) float Vs[KT * ROW_STRIDE];
    __shared__ int s_kmin, s_kmax;

    const int tid = threadIdx.x;
    const int rloc = tid / TPR, part = tid % TPR;
    const int nrb = (p.Sq + ROWS - 1) / ROWS;
    const int bh = blockIdx.x / nrb;       // b * Hq + h
    const int b = bh / p.Hq, h = bh % p.Hq;
    const int g = h / p.G;
    const int qi = (blockIdx.x % nrb) * ROWS + rloc;
    const bool live = qi < p.Sq;

    int ra = 1, re = 0;
    if (live) {
        ra = 0;
        re = p.Sk - 1;
        if (p.causal) re = min(re, qi);
        if (p.wl >= 0) ra = max(ra, qi - p.wl);
        if (p.wr >= 0) re = min(re, qi + p.wr);
        if (p.rowb) {
            int2 r = p.rowb[(size_t)b * p.Sq + qi];
            ra = max(ra, r.x);
            re = min(re, r.y);
        }
    }
    if (tid == 0) {
        s_kmin = 0x7fffffff;
        s_kmax = -1;
    }
    __syncthreads();
    if (ra <= re) {
        atomicMin(&s_kmin, ra);
        atomicMax(&s_kmax, re);
    }
    __syncthreads();
    const int kmin = s_kmin, kmax = s_kmax;

    float qv[64], o[64];
    const float* qrow = p.q + (((size_t)b * p.Hq + h) * p.Sq + (live ? qi : 0)) * D + part * 64;
#pragma unroll
    for (int d = 0; d < 64; d += 4) {
        float4 t = live ? *reinterpret_cast<const float4*>(qrow + d) : make_float4(0.f, 0.f, 0.f, 0.f);
        qv[d] = t.x;
        qv[d + 1] = t.y;
        qv[d + 2] = t.z;
        qv[d + 3] = t.w;
        o[d] = o[d + 1] = o[d + 2] = o[d + 3] = 0.f;
    }
    float m = -INFINITY, l = 0.f;  // base-2 units
    const float slope_l2 = ALIBI ? p.slopes[h] * LOG2E_F : 0.f;
    const float* kbase = p.k + ((size_t)b * p.Hkv + g) * p.Sk * D;
    const float* vbase = p.v + ((size_t)b * p.Hkv + g) * p.Sk * D;

    if (kmin <= kmax) {
        for (int k0 = (kmin / KT) * KT; k0 <= kmax; k0 += KT) {
            __syncthreads();
            for (int i = tid; i < KT * D / 4; i += 128) {
                const int j = i / (D / 4), c = (i % (D / 4)) * 4;
                const int kj = k0 + j;
                float4 kv4 = make_float4(0.f, 0.f, 0.f, 0.f), vv4 = kv4;
                if (kj < p.Sk) {
                    kv4 = *reinterpret_cast<const float4*>(kbase + (size_t)kj * D + c);
                    vv4 = *reinterpret_cast<const float4*>(vbase + (size_t)kj * D + c);
                }
                const int so = j * ROW_STRIDE + (c / 64) * HALF_STRIDE + (c % 64);
                *reinterpret_cast<float4*>(Ks + so) = kv4;
                *reinterpret_cast<float4*>(Vs + so) = vv4;
            }
            __syncthreads();
            float t[KT];
            float tmax = -INFINITY;
#pragma unroll 4
            for (int j = 0; j < KT; ++j) {
                const float* kr = Ks + j * ROW_STRIDE + part * HALF_STRIDE;
                float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                for (int d = 0; d < 64; d += 4) {
                    float4 kk = *reinterpret_cast<const float4*>(kr + d);
                    acc0 = fmaf(qv[d], kk.x, acc0);
                    acc1 = fmaf(qv[d + 1], kk.y, acc1);
                    acc0 = fmaf(qv[d + 2], kk.z, acc0);
                    acc1 = fmaf(qv[d + 3], kk.w, acc1);
                }
                float dot = acc0 + acc1;
                if (TPR == 2) dot += __shfl_xor_sync(0xffffffffu, dot, 1);
                float u = p.scale * dot;
                if (SOFTCAP) u = p.softcap * tanhf(u / p.softcap);
                const int kj = k0 + j;
                float tj = u * LOG2E_F;
                if (ALIBI) tj = fmaf(slope_l2, (float)(kj - qi), tj);
                if (kj < ra || kj > re) tj = -INFINITY;
                t[j] = tj;
                tmax = fmaxf(tmax, tj);
            }
            const float m_new = fmaxf(m, tmax);
            if (m_new == -INFINITY) continue;  // nothing admissible so far
            const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - m_new);
            l *= alpha;
#pragma unroll
            for (int d = 0; d < 64; ++d) o[d] *= alpha;
            m = m_new;
#pragma unroll 2
            for (int j = 0; j < KT; ++j) {
                const float pj = exp2f(t[j] - m);
                l += pj;
                const float* vr = Vs + j * ROW_STRIDE + part * HALF_STRIDE;
#pragma unroll
                for (int d = 0; d < 64; d += 4) {
                    float4 vv = *reinterpret_cast<const float4*>(vr + d);
                    o[d] = fmaf(pj, vv.x, o[d]);
                    o[d + 1] = fmaf(pj, vv.y, o[d + 1]);
                    o[d + 2] = fmaf(pj, vv.z, o[d + 2]);
                    o[d + 3] = fmaf(pj, vv.w, o[d + 3]);
                }
            }
        }
    }
    if (!live) return;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float* orow = p.out + (((size_t)b * p.Hq + h) * p.Sq + qi) * D + part * 64;
#pragma unroll
    for (int d = 0; d < 64; d += 4)
        *reinterpret_cast<float4*>(orow + d) = make_float4(o[d] * inv, o[d + 1] * inv, o[d + 2] * inv, o[d + 3] * inv);
    if (p.lse && part == 0) p.lse[((size_t)b * p.Hq + h) * p.Sq + qi] = l > 0.f ? (m + log2f(l)) * LN2_F : -INFINITY;
}

template <int D, bool SOFTCAP, bool ALIBI>
cudaError_t launch32(const Params32& p, cudaStream_t stream) {
    constexpr int ROWS = 128 / (D / 64);
    const long long grid = (long long)((p.Sq + ROWS - 1) / ROWS) * p.B * p.Hq;
    prefill_f32_kernel<D, SOFTCAP, ALIBI><<<(unsigned)grid, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_f32(const FwdProblem& f, cudaStream_t stream) {
    Params32 p{};
    p.q = static_cast<const float*>(f.q);
    p.k = static_cast<const float*>(f.k);
    p.v = static_cast<const float*>(f.v);
    p.out = static_cast<float*>(f.out);
    p.lse = f.lse;
    p.slopes = f.slopes;
    p.rowb = reinterpret_cast<const int2*>(f.row_bounds);
    p.B = f.B;
    p.Hq = f.Hq;
    p.Hkv = f.Hkv;
    p.Sq = f.Sq;
    p.Sk = f.Sk;
    p.G = f.Hq / f.Hkv;
    p.causal = f.causal;
    p.wl = f.wl;
    p.wr = f.wr;
    p.scale = f.scale;
    p.softcap = f.softcap;
    const bool cap = f.softcap > 0.f, ali = f.slopes != nullptr;
    if (f.D == 128) {
        if (cap) return ali ? launch32<128, true, true>(p, stream) : launch32<128, true, false>(p, stream);
        return ali ? launch32<128, false, true>(p, stream) : launch32<128, false, false>(p, stream);
    }
    if (cap) return ali ? launch32<64, true, true>(p, stream) : launch32<64, true, false>(p, stream);
    return ali ? launch32<64, false, true>(p, stream) : launch32<64, false, false>(p, stream);
}

}  // namespace gbattn
