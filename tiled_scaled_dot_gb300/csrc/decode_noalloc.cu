// decode_noalloc.cu -- attn_decode_noalloc: the split-KV decode for callers
// that may not allocate device memory themselves.
//
// Some callers cannot hand the library a workspace: an engine that owns every
// byte of device memory through its own pool and forbids other allocations, or
// a latency-critical serving loop where a cudaMalloc (which can synchronise the
// device) is not acceptable.  This entry point takes the decode's scratch from
// a fixed array in device memory that is part of the library's own module, so
// the caller passes only inputs and outputs and nothing is allocated per call.
//
// The array is GBATTN_NOALLOC_SCRATCH_BYTES (32 MiB).  It occupies device
// memory on each GPU where this file's module has been loaded -- under CUDA's
// default lazy loading, where attn_decode_noalloc has been called -- until the
// process exits.  Its device address is looked up once per device and kept, so
// the entry must not be used on a device after a cudaDeviceReset (the module
// may be reloaded elsewhere).  Every call shares the array: a call that
// overlaps another on the GPU (two streams, or two host threads) races on it.
// Nothing in it needs to start at zero: each call writes every partial result
// its combine step reads before reading it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gbattn.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GBATTN_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
constexpr int kMaxDev = 64;
void* g_noalloc_ptr[kMaxDev] = {};

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return GBATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GBATTN_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return GBATTN_OK;
}

}  // namespace

extern "C" int attn_decode_noalloc(const void* q, const void* k, const void* v, const float* alibi_slopes,
                                   void* out, float* lse_out, int B, int Hq, int Hkv, int Sk, int D,
                                   float softmax_scale, float softcap, int num_splits, int dtype, void* stream) {
    const size_t need = attn_decode_workspace_size(B, Hq, Hkv, Sk, D, num_splits);
    if (need > (size_t)GBATTN_NOALLOC_SCRATCH_BYTES) return GBATTN_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != GBATTN_OK) return rc;
    return attn_decode(q, k, v, alibi_slopes, out, lse_out, B, Hq, Hkv, Sk, D, softmax_scale, softcap, -1, -1,
                       num_splits, scratch, (size_t)GBATTN_NOALLOC_SCRATCH_BYTES, dtype, stream);
}
