// diag.cu -- one tcgen05 tile product through the attention kernels' layouts
// (see include/gbattn_diag.h).  Used by the tests to pin the descriptor and
// TMEM conventions independently of the attention arithmetic.
#include <cuda_bf16.h>

#include "../../include/gbattn.h"
#include "../../include/gbattn_diag.h"
#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {


namespace {

template <int N, int MODE>
__global__ void __launch_bounds__(128, 1)
    diag_umma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __nv_bfloat16* a_glob, float* c, unsigned int* status,
                     unsigned long long timeout_ns) {
    constexpr int A_BYTES = 128 * 128 * 2;
    constexpr int B_BYTES = 128 * N * 2;
    extern __shared__ __align__(1024) uint8_t dyn_smem[];
    __shared__ uint64_t load_bar, mma_bar;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = base;
    uint8_t* sB = base + A_BYTES;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&load_bar, 1);
        mbar_init(&mma_bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    WaitCtl wc{&abort_flag, status, timeout_ns};

    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&load_bar, A_BYTES + B_BYTES);
        for (int h = 0; h < 2; ++h) tma_load_3d(sA + h * 128 * 128, &tmA, &load_bar, h * 64, 0, 0);
        if (MODE == 0) {
            for (int h = 0; h < 2; ++h) tma_load_3d(sB + h * N * 128, &tmB, &load_bar, h * 64, 0, 0);
        } else {
            for (int h = 0; h < N / 64; ++h) tma_load_3d(sB + h * 128 * 128, &tmB, &load_bar, h * 64, 0, 0);
        }
    }
    if (MODE == 2) {
        // Row r of A (128 bf16) into TMEM lane r, columns 256 .. 319, two per column.
        const int r = threadIdx.x;
        const __nv_bfloat16* ar = a_glob + r * 128;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16) + 256;
        uint32_t w[32];
        for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int k = half * 64 + 2 * i;
                const uint16_t lo = reinterpret_cast<const uint16_t*>(ar)[k];
                const uint16_t hi = reinterpret_cast<const uint16_t*>(ar)[k + 1];
                w[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            }
            tmem_st32(taddr + half * 32, w);
        }
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    bool ok = true;
    if (threadIdx.x == 0) {
        ok = mbar_wait(&load_bar, 0, wc, ST_DIAG);
        if (ok) {
            tc_fence_after();
            const uint32_t aa = smem_u32(sA), ba = smem_u32(sB);
            const uint32_t idesc = idesc_bf16_f32(128, N, MODE == 0 ? 0 : 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                if (MODE == 0) {
                    umma_ss(tmem, sdesc_sw128(aa + (kk >> 2) * 16384 + (kk & 3) * 32, 16),
                            sdesc_sw128(ba + (kk >> 2) * N * 128 + (kk & 3) * 32, 16), idesc, kk > 0);
                } else if (MODE == 1) {
                    umma_ss(tmem, sdesc_sw128(aa + (kk >> 2) * 16384 + (kk & 3) * 32, 16),
                            sdesc_sw128(ba + kk * 16 * 128, 128 * 128), idesc, kk > 0);
                } else {
                    umma_ts(tmem, tmem + 256 + 8 * kk, sdesc_sw128(ba + kk * 16 * 128, 128 * 128), idesc, kk > 0);
                }
            }
            umma_commit(&mma_bar);
        }
    }
    __syncthreads();
    ok = mbar_wait(&mma_bar, 0, wc, ST_DIAG);
    if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const int r = threadIdx.x;
#pragma unroll
        for (int c0 = 0; c0 < N; c0 += 32) {
            float v[32];
            tmem_ld32(taddr + c0, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) c[r * N + c0 + i] = v[i];
        }
    }
    (void)lane;
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int N, int MODE>
cudaError_t run_diag(const CUtensorMap& ta, const CUtensorMap& tb, const void* a, float* c, unsigned int* status,
                     cudaStream_t s) {
    auto k = diag_umma_kernel<N, MODE>;
    const int smem = 128 * 128 * 2 + 128 * N * 2 + 1024;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k<<<1, 128, smem, s>>>(ta, tb, static_cast<const __nv_bfloat16*>(a), c, status, 2000000000ull);
    return cudaGetLastError();
}

// A wait that nothing satisfies: thread 0 waits, with the kernels' bounded
// wait, on an mbarrier that no thread or copy ever arrives at.  When
// timeout_ns has passed the wait sets ST_DIAG in the device status word and
// the kernel returns; nothing else is touched.
__global__ void __launch_bounds__(32, 1) diag_wait_kernel(unsigned int* status, unsigned long long timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        WaitCtl wc{&abort_flag, status, timeout_ns};
        (void)mbar_wait(&bar, 0, wc, ST_DIAG);
    }
}

}  // namespace
}  // namespace gbattn

using namespace gbattn;

extern "C" int gbattn_diag_umma(int mode, const void* a, const void* b, float* c, int n, void* stream) {
    if (!a || !b || !c || (n != 64 && n != 128) || mode < 0 || mode > 2) return GBATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15u) return GBATTN_ERR_INVALID_ARG;
    CUtensorMap ta, tb;
    if (!encode_map_bf16_3d(&ta, a, 128, 128, 1, 128)) return GBATTN_ERR_CUDA;
    const bool ok = mode == 0 ? encode_map_bf16_3d(&tb, b, 128, n, 1, n) : encode_map_bf16_3d(&tb, b, n, 128, 1, 128);
    if (!ok) return GBATTN_ERR_CUDA;
    unsigned int* st = nullptr;
    int sms = 0;
    if (!device_facts(&st, &sms)) return GBATTN_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (n == 128) {
        e = mode == 0 ? run_diag<128, 0>(ta, tb, a, c, st, s)
                      : (mode == 1 ? run_diag<128, 1>(ta, tb, a, c, st, s) : run_diag<128, 2>(ta, tb, a, c, st, s));
    } else {
        e = mode == 0 ? run_diag<64, 0>(ta, tb, a, c, st, s)
                      : (mode == 1 ? run_diag<64, 1>(ta, tb, a, c, st, s) : run_diag<64, 2>(ta, tb, a, c, st, s));
    }
    return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

extern "C" int gbattn_diag_wait_timeout(unsigned long long timeout_ns, void* stream) {
    if (timeout_ns == 0 || timeout_ns > 10000000000ull) return GBATTN_ERR_INVALID_ARG;
    unsigned int* st = nullptr;
    int sms = 0;
    if (!device_facts(&st, &sms)) return GBATTN_ERR_CUDA;
    diag_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(st, timeout_ns);
    return cudaGetLastError() == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}
