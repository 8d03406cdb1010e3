// backward_f32.cu -- fp32 attention backward with SIMT FFMA (no TF32), for
// the fp32 storage type; the gradients of attention.fkc.md,
// "attention_flash_backward", as in backward_bf16.cu:
//   P_ij = 2^(s_ij log2(e) - lse_i log2(e)),  dP_ij = dO_i . V_j,
//   dS_ij = P_ij (dP_ij - Delta_i) [* (1 - tanh^2(s_pre / c))],
//   dQ_i = scale sum_j dS_ij K_j,  dK_j = scale sum_{h in group, i} dS_ij Q_i,
//   dV_j = sum_{h in group, i} P_ij dO_i,  Delta_i = dO_i . O_i.
// The scores are formed exactly as the fp32 forward forms them (tanhf,
// exp2f), so P matches that forward's lse.  Row intervals come from the shared
// prep launch (bwd_rows_kernel); fixed summation order, no atomics.
//
// Threads: D / 32 per row (query row in the dQ kernel, key in the dK / dV
// kernel), each holding 32 of the row's dimensions; dot products are reduced
// across the row's threads with shuffles.  Operand rows stream through
// shared memory in tiles of 32.
#include "kernels.h"

namespace gbattn {
namespace {

constexpr int T32 = 32;  // rows per shared-memory tile
constexpr float LOG2E_32 = 1.4426950408889634f;

struct B32 {
    const float* q;
    const float* k;
    const float* v;
    const float* dout;
    const float* lse2;   // [B * Hq][Sq_pad]
    const float* delta;  // [B * Hq][Sq_pad]
    const int2* rows;    // [B][Sq_pad]
    const float* slopes;
    float* dq;
    float* dk;
    float* dv;
    int B, Hq, Hkv, Sq, Sk, G, Sq_pad;
    float scale, softcap;
};

// Sum over the TPR consecutive threads of one row.
template <int TPR>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// P and the softcap factor of one (row, key) pair from its raw dot product:
// the fp32 forward's score (scale, softcap, ALiBi in base 2) minus lse2.
template <bool SOFTCAP, bool ALIBI>
__device__ __forceinline__ float prob(const B32& p, float dot, float slope_l2, int kj, int qi, float lse2,
                                      float& f) {
    float u = p.scale * dot;
    f = 1.f;
    if (SOFTCAP) {
        const float t = tanhf(u / p.softcap);
        u = p.softcap * t;
        f = 1.f - t * t;
    }
    float z = u * LOG2E_32;
    if (ALIBI) z = fmaf(slope_l2, (float)(kj - qi), z);
    return exp2f(z - lse2);
}

// One warp per padded row: Delta = dO . O and the base-2 lse.
template <int D>
__global__ void __launch_bounds__(256) bwd_delta32_kernel(const float* __restrict__ dout,
                                                          const float* __restrict__ out,
                                                          const float* __restrict__ lse, float* __restrict__ lse2,
                                                          float* __restrict__ delta, long long n_rows, int Sq,
                                                          int Sq_pad) {
    const int lane = threadIdx.x & 31;
    const long long w0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long row = w0; row < n_rows; row += nw) {
        const long long bh = row / Sq_pad;
        const int i = (int)(row - bh * Sq_pad);
        float d = 0.f, l2 = INFINITY;
        if (i < Sq) {
            const size_t off = ((size_t)bh * Sq + i) * D;
            for (int c = lane; c < D; c += 32) d = fmaf(dout[off + c], out[off + c], d);
            const float lv = lse[(size_t)bh * Sq + i];
            l2 = (lv == -INFINITY) ? INFINITY : lv * LOG2E_32;
        }
        d = row_sum<32>(d);
        if (lane == 0) {
            lse2[row] = l2;
            delta[row] = d;
        }
    }
}

// dQ: a block holds 128 / TPR query rows of one (b, h) and streams the key
// tiles that meet their admissible ranges.
template <int D, bool SOFTCAP, bool ALIBI>
__global__ void __launch_bounds__(128) bwd_dq32_kernel(const B32 p) {
    constexpr int TPR = D / 32, ROWS = 128 / TPR, RS = D + 4;  // skewed smem rows
    __shared__ __align__(16) float Ks[T32 * RS];
    __shared__ __align__(16) float Vs[T32 * RS];
    __shared__ int s_kmin, s_kmax;
    const int tid = threadIdx.x, rloc = tid / TPR, part = tid % TPR;
    const int nrb = (p.Sq + ROWS - 1) / ROWS;
    const int bh = blockIdx.x / nrb, b = bh / p.Hq, h = bh % p.Hq, g = h / p.G;
    const int qi = (blockIdx.x % nrb) * ROWS + rloc;
    const bool live = qi < p.Sq;
    int2 iv = make_int2(1, 0);
    float lse2 = INFINITY, dl = 0.f;
    if (live) {
        iv = p.rows[(size_t)b * p.Sq_pad + qi];
        lse2 = p.lse2[(size_t)bh * p.Sq_pad + qi];
        dl = p.delta[(size_t)bh * p.Sq_pad + qi];
    }
    if (tid == 0) {
        s_kmin = 0x7fffffff;
        s_kmax = -1;
    }
    __syncthreads();
    if (part == 0 && iv.x <= iv.y) {
        atomicMin(&s_kmin, iv.x);
        atomicMax(&s_kmax, iv.y);
    }
    __syncthreads();
    const int kmin = s_kmin, kmax = s_kmax;
    float qv[32], dov[32], acc[32];
    const size_t roff = ((size_t)bh * p.Sq + (live ? qi : 0)) * D + part * 32;
#pragma unroll
    for (int d = 0; d < 32; ++d) {
        qv[d] = live ? p.q[roff + d] : 0.f;
        dov[d] = live ? p.dout[roff + d] : 0.f;
        acc[d] = 0.f;
    }
    const float slope_l2 = ALIBI ? p.slopes[h] * LOG2E_32 : 0.f;
    const float* kb = p.k + ((size_t)b * p.Hkv + g) * p.Sk * D;
    const float* vb = p.v + ((size_t)b * p.Hkv + g) * p.Sk * D;
    for (int k0 = kmin <= kmax ? (kmin / T32) * T32 : 0; k0 <= kmax; k0 += T32) {
        __syncthreads();
        for (int x = tid; x < T32 * D / 4; x += 128) {
            const int j = x / (D / 4), c = (x % (D / 4)) * 4;
            float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), vv = kk;
            if (k0 + j < p.Sk) {
                kk = *reinterpret_cast<const float4*>(kb + (size_t)(k0 + j) * D + c);
                vv = *reinterpret_cast<const float4*>(vb + (size_t)(k0 + j) * D + c);
            }
            *reinterpret_cast<float4*>(Ks + j * RS + c) = kk;
            *reinterpret_cast<float4*>(Vs + j * RS + c) = vv;
        }
        __syncthreads();
        for (int j = 0; j < T32; ++j) {
            const float* kr = Ks + j * RS + part * 32;
            const float* vr = Vs + j * RS + part * 32;
            float s = 0.f, dp = 0.f;
#pragma unroll
            for (int d = 0; d < 32; ++d) {
                s = fmaf(qv[d], kr[d], s);
                dp = fmaf(dov[d], vr[d], dp);
            }
            s = row_sum<TPR>(s);
            dp = row_sum<TPR>(dp);
            const int kj = k0 + j;
            float f;
            float pr = prob<SOFTCAP, ALIBI>(p, s, slope_l2, kj, qi, lse2, f);
            if (kj < iv.x || kj > iv.y) pr = 0.f;
            const float ds = pr * f * (dp - dl);
#pragma unroll
            for (int d = 0; d < 32; ++d) acc[d] = fmaf(ds, kr[d], acc[d]);
        }
    }
    if (!live) return;
    float* dst = p.dq + roff;
#pragma unroll
    for (int d = 0; d < 32; ++d) dst[d] = acc[d] * p.scale;
}

// dK, dV: a block holds 128 / TPR keys of one (b, kv head) and streams every
// query tile of every head of the group.
template <int D, bool SOFTCAP, bool ALIBI>
__global__ void __launch_bounds__(128) bwd_dkdv32_kernel(const B32 p) {
    constexpr int TPR = D / 32, ROWS = 128 / TPR, RS = D + 4;
    __shared__ __align__(16) float Qs[T32 * RS];
    __shared__ __align__(16) float Os[T32 * RS];  // dO
    __shared__ float Ls[T32], Ds[T32];
    __shared__ int2 Is[T32];
    const int tid = threadIdx.x, rloc = tid / TPR, part = tid % TPR;
    const int nkb = (p.Sk + ROWS - 1) / ROWS;
    const int bg = blockIdx.x / nkb, b = bg / p.Hkv, g = bg % p.Hkv;
    const int kj = (blockIdx.x % nkb) * ROWS + rloc;
    const bool live = kj < p.Sk;
    float kv[32], vv[32], dk[32], dv[32];
    const size_t koff = ((size_t)bg * p.Sk + (live ? kj : 0)) * D + part * 32;
#pragma unroll
    for (int d = 0; d < 32; ++d) {
        kv[d] = live ? p.k[koff + d] : 0.f;
        vv[d] = live ? p.v[koff + d] : 0.f;
        dk[d] = dv[d] = 0.f;
    }
    for (int hh = 0; hh < p.G; ++hh) {
        const int h = g * p.G + hh, bh = b * p.Hq + h;
        const float slope_l2 = ALIBI ? p.slopes[h] * LOG2E_32 : 0.f;
        for (int i0 = 0; i0 < p.Sq; i0 += T32) {
            __syncthreads();
            for (int x = tid; x < T32 * D / 4; x += 128) {
                const int r = x / (D / 4), c = (x % (D / 4)) * 4;
                float4 qq = make_float4(0.f, 0.f, 0.f, 0.f), oo = qq;
                if (i0 + r < p.Sq) {
                    qq = *reinterpret_cast<const float4*>(p.q + ((size_t)bh * p.Sq + i0 + r) * D + c);
                    oo = *reinterpret_cast<const float4*>(p.dout + ((size_t)bh * p.Sq + i0 + r) * D + c);
                }
                *reinterpret_cast<float4*>(Qs + r * RS + c) = qq;
                *reinterpret_cast<float4*>(Os + r * RS + c) = oo;
            }
            if (tid < T32) {
                // padded rows (i >= Sq) carry lse2 = +inf and an empty interval
                Ls[tid] = p.lse2[(size_t)bh * p.Sq_pad + i0 + tid];
                Ds[tid] = p.delta[(size_t)bh * p.Sq_pad + i0 + tid];
                Is[tid] = p.rows[(size_t)b * p.Sq_pad + i0 + tid];
            }
            __syncthreads();
            for (int r = 0; r < T32; ++r) {
                const float* qr = Qs + r * RS + part * 32;
                const float* orow = Os + r * RS + part * 32;
                float s = 0.f, dp = 0.f;
#pragma unroll
                for (int d = 0; d < 32; ++d) {
                    s = fmaf(qr[d], kv[d], s);
                    dp = fmaf(orow[d], vv[d], dp);
                }
                s = row_sum<TPR>(s);
                dp = row_sum<TPR>(dp);
                const int2 iv = Is[r];
                float f;
                float pr = prob<SOFTCAP, ALIBI>(p, s, slope_l2, kj, i0 + r, Ls[r], f);
                if (kj < iv.x || kj > iv.y) pr = 0.f;
                const float ds = pr * f * (dp - Ds[r]);
#pragma unroll
                for (int d = 0; d < 32; ++d) {
                    dv[d] = fmaf(pr, orow[d], dv[d]);
                    dk[d] = fmaf(ds, qr[d], dk[d]);
                }
            }
        }
    }
    if (!live) return;
#pragma unroll
    for (int d = 0; d < 32; ++d) {
        p.dk[koff + d] = dk[d] * p.scale;
        p.dv[koff + d] = dv[d];
    }
}

template <int D, bool SOFTCAP, bool ALIBI>
cudaError_t launch_main32(const B32& p, cudaStream_t stream, cudaEvent_t* ev) {
    constexpr int ROWS = 128 / (D / 32);
    cudaError_t e;
    const long long grid_kv = (long long)((p.Sk + ROWS - 1) / ROWS) * p.B * p.Hkv;
    bwd_dkdv32_kernel<D, SOFTCAP, ALIBI><<<(unsigned)grid_kv, 128, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (ev && (e = cudaEventRecord(ev[2], stream)) != cudaSuccess) return e;
    const long long grid_q = (long long)((p.Sq + ROWS - 1) / ROWS) * p.B * p.Hq;
    bwd_dq32_kernel<D, SOFTCAP, ALIBI><<<(unsigned)grid_q, 128, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return ev ? cudaEventRecord(ev[3], stream) : cudaSuccess;
}

}  // namespace

cudaError_t launch_backward_f32(const BwdProblem& b, cudaStream_t stream, cudaEvent_t* ev) {
    B32 p{};
    p.q = static_cast<const float*>(b.q);
    p.k = static_cast<const float*>(b.k);
    p.v = static_cast<const float*>(b.v);
    p.dout = static_cast<const float*>(b.dout);
    p.lse2 = b.ws_lse2;
    p.delta = b.ws_delta;
    p.rows = reinterpret_cast<const int2*>(b.ws_rows);
    p.slopes = b.slopes;
    p.dq = static_cast<float*>(b.dq);
    p.dk = static_cast<float*>(b.dk);
    p.dv = static_cast<float*>(b.dv);
    p.B = b.B;
    p.Hq = b.Hq;
    p.Hkv = b.Hkv;
    p.Sq = b.Sq;
    p.Sk = b.Sk;
    p.G = b.Hq / b.Hkv;
    p.Sq_pad = (int)backward_sq_pad(b.Sq);
    p.scale = b.scale;
    p.softcap = b.softcap;
    cudaError_t e;
    if (ev && (e = cudaEventRecord(ev[0], stream)) != cudaSuccess) return e;
    if ((e = launch_backward_rows(b, stream)) != cudaSuccess) return e;
    const long long n_rows = (long long)b.B * b.Hq * p.Sq_pad;
    long long blocks = (n_rows * 32 + 255) / 256;
    if (blocks > (long long)b.num_sms * 16) blocks = (long long)b.num_sms * 16;
    const float* out = static_cast<const float*>(b.out);
    if (b.D == 128)
        bwd_delta32_kernel<128><<<(int)blocks, 256, 0, stream>>>(p.dout, out, b.lse, b.ws_lse2, b.ws_delta, n_rows,
                                                                 b.Sq, p.Sq_pad);
    else
        bwd_delta32_kernel<64><<<(int)blocks, 256, 0, stream>>>(p.dout, out, b.lse, b.ws_lse2, b.ws_delta, n_rows,
                                                                b.Sq, p.Sq_pad);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (ev && (e = cudaEventRecord(ev[1], stream)) != cudaSuccess) return e;
    const bool cap = b.softcap > 0.f, ali = b.slopes != nullptr;
    if (b.D == 128) {
        if (cap) return ali ? launch_main32<128, true, true>(p, stream, ev) : launch_main32<128, true, false>(p, stream, ev);
        return ali ? launch_main32<128, false, true>(p, stream, ev) : launch_main32<128, false, false>(p, stream, ev);
    }
    if (cap) return ali ? launch_main32<64, true, true>(p, stream, ev) : launch_main32<64, true, false>(p, stream, ev);
    return ali ? launch_main32<64, false, true>(p, stream, ev) : launch_main32<64, false, false>(p, stream, ev);
}

}  // namespace gbattn
