// api.cu -- the C ABI of libgbattn: argument validation, TMA descriptor
// encoding (with a small cache), kernel dispatch, device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/gbattn.h"
#include "kernels.h"

namespace gbattn {

// Status word written by kernels whose bounded waits give up.
__device__ unsigned int g_status_word;

namespace {

std::mutex g_mu;
uint64_t g_timeout_ns = [] {
    const char* e = std::getenv("GBATTN_WAIT_TIMEOUT_MS");
    if (e && *e) {
        long long ms = std::atoll(e);
        if (ms > 0) return static_cast<uint64_t>(ms) * static_cast<uint64_t>(1000000);
    }
    return static_cast<uint64_t>(2000000000ull);
}();

constexpr int kMaxDevices = 64;
unsigned int* g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Per-device facts (current device): status word address and SM count.

// Small cache of encoded tensor maps keyed by (device, pointer, extents, box).
struct MapKey {
    int dev;
    int kind;  // 0: [planes][rows][cols] tiles, 1: paged pool [planes = tokens][rows = heads][cols]
    int f16;   // element type: 0 bf16, 1 fp16
    const void* base;
    uint64_t cols, rows, planes;
    uint32_t box_rows;
    bool operator==(const MapKey& o) const {
        return dev == o.dev && kind == o.kind && f16 == o.f16 && base == o.base && cols == o.cols && rows == o.rows &&
               planes == o.planes && box_rows == o.box_rows;
    }
};
constexpr int kCache = 32;
MapKey g_keys[kCache];
CUtensorMap g_maps[kCache];
int g_used = 0, g_next = 0;

bool cached_map(CUtensorMap* out, const void* base, uint64_t cols, uint64_t rows, uint64_t planes,
                uint32_t box_rows, int kind = 0, bool f16 = false) {
    int dev = 0;
    cudaGetDevice(&dev);
    MapKey key{dev, kind, f16 ? 1 : 0, base, cols, rows, planes, box_rows};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (int i = 0; i < g_used; ++i)
            if (g_keys[i] == key) {
                *out = g_maps[i];
                return true;
            }
    }
    CUtensorMap m;
    const bool ok = kind == 0 ? encode_map_bf16_3d(&m, base, cols, rows, planes, box_rows, f16)
                              : encode_map_pool_bf16(&m, base, cols, rows, planes, box_rows, f16);
    if (!ok) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    int slot = g_used < kCache ? g_used++ : (g_next++ % kCache);
    g_keys[slot] = key;
    g_maps[slot] = m;
    *out = m;
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b) return false;
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int check_common(int B, int Hq, int Hkv, int S, int Sk, int D, float scale, float softcap, int dtype) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || S <= 0 || Sk <= 0 || D <= 0) return GBATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return GBATTN_ERR_INVALID_ARG;
    if (!(std::isfinite(scale) && scale > 0.f)) return GBATTN_ERR_INVALID_ARG;
    if (!(std::isfinite(softcap) && softcap >= 0.f)) return GBATTN_ERR_INVALID_ARG;
    if (dtype != GBATTN_BF16 && dtype != GBATTN_F32 && dtype != GBATTN_F16) return GBATTN_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return GBATTN_ERR_UNSUPPORTED;
    // 32-bit index limits of the kernels' grids and rows.
    if ((long long)B * Hq * S > 0x7fffffffLL || (long long)B * Hkv * Sk > 0x7fffffffLL) return GBATTN_ERR_UNSUPPORTED;
    return GBATTN_OK;
}

}  // namespace

bool device_facts(unsigned int** status, int* num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return false;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
        g_status_ptr[dev] = static_cast<unsigned int*>(p);
        g_num_sms[dev] = sms;
    }
    *status = g_status_ptr[dev];
    *num_sms = g_num_sms[dev];
    return true;
}

bool encode_map_bf16_3d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t planes,
                        uint32_t box_rows, bool f16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {cols, rows, planes};
    cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType ty = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    return fn(map, ty, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_map_pool_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t heads, uint64_t rows,
                          uint32_t box_rows, bool f16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {cols, heads, rows};
    cuuint64_t strides[2] = {cols * 2, cols * heads * 2};
    cuuint32_t box[3] = {64, 1, box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType ty = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    return fn(map, ty, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gbattn

using namespace gbattn;

extern "C" {

int attn_fwd_ex(const gbattn_fwd_params* a) {
    if (!a) return GBATTN_ERR_INVALID_ARG;
    int rc = check_common(a->B, a->Hq, a->Hkv, a->Sq, a->Sk, a->D, a->softmax_scale, a->softcap, a->dtype);
    if (rc) return rc;
    if (!a->q || !a->k || !a->v || !a->out) return GBATTN_ERR_INVALID_ARG;
    if (a->causal != 0 && a->causal != 1) return GBATTN_ERR_INVALID_ARG;
    if (a->window_left < -1 || a->window_right < -1) return GBATTN_ERR_INVALID_ARG;
    if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->out)) return GBATTN_ERR_INVALID_ARG;
    if (a->row_kv_bounds && (reinterpret_cast<uintptr_t>(a->row_kv_bounds) & 7u)) return GBATTN_ERR_INVALID_ARG;
    if (a->lse_out && (reinterpret_cast<uintptr_t>(a->lse_out) & 3u)) return GBATTN_ERR_INVALID_ARG;
    if (a->alibi_slopes && (reinterpret_cast<uintptr_t>(a->alibi_slopes) & 3u)) return GBATTN_ERR_INVALID_ARG;
    const size_t esz = a->dtype == GBATTN_F32 ? 4 : 2;
    const size_t nq = (size_t)a->B * a->Hq * a->Sq * a->D * esz;
    const size_t nkv = (size_t)a->B * a->Hkv * a->Sk * a->D * esz;
    if (overlaps(a->out, nq, a->q, nq) || overlaps(a->out, nq, a->k, nkv) || overlaps(a->out, nq, a->v, nkv))
        return GBATTN_ERR_INVALID_ARG;

    FwdProblem f{};
    f.q = a->q;
    f.k = a->k;
    f.v = a->v;
    f.slopes = a->alibi_slopes;
    f.row_bounds = a->row_kv_bounds;
    f.out = a->out;
    f.lse = a->lse_out;
    f.B = a->B;
    f.Hq = a->Hq;
    f.Hkv = a->Hkv;
    f.Sq = a->Sq;
    f.Sk = a->Sk;
    f.D = a->D;
    f.scale = a->softmax_scale;
    f.causal = a->causal;
    f.wl = a->window_left;
    f.wr = a->window_right;
    f.softcap = a->softcap;
    f.timeout_ns = g_timeout_ns;
    f.f16 = a->dtype == GBATTN_F16;
    if (!device_facts(&f.status, &f.num_sms)) return GBATTN_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(a->stream);
    cudaError_t e;
    if (a->dtype == GBATTN_F32) {
        e = launch_prefill_f32(f, st);
    } else {
        const bool h = f.f16 != 0;
        CUtensorMap tq, tk, tv, to;
        if (!cached_map(&tq, a->q, a->D, a->Sq, (uint64_t)a->B * a->Hq, 128, 0, h) ||
            !cached_map(&tk, a->k, a->D, a->Sk, (uint64_t)a->B * a->Hkv, 128, 0, h) ||
            !cached_map(&tv, a->v, a->D, a->Sk, (uint64_t)a->B * a->Hkv, 128, 0, h) ||
            !cached_map(&to, a->out, a->D, a->Sq, (uint64_t)a->B * a->Hq, 128, 0, h))
            return GBATTN_ERR_CUDA;
        e = launch_prefill_bf16(f, tq, tk, tv, to, st);
    }
    return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

int attn_fwd(const void* q, const void* k, const void* v, const float* alibi_slopes, void* out, int B, int Hq,
             int Hkv, int Sq, int Sk, int D, float softmax_scale, int causal, int window_left, int window_right,
             float softcap, int dtype, void* stream) {
    gbattn_fwd_params a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.alibi_slopes = alibi_slopes;
    a.out = out;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.Sq = Sq;
    a.Sk = Sk;
    a.D = D;
    a.softmax_scale = softmax_scale;
    a.causal = causal;
    a.window_left = window_left;
    a.window_right = window_right;
    a.softcap = softcap;
    a.dtype = dtype;
    a.stream = stream;
    return attn_fwd_ex(&a);
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                    const int32_t* cu_seqlens_k, const int32_t* seqused_k, const float* alibi_slopes, void* out,
                    float* lse_out, int B, int Hq, int Hkv, int D, int total_q, int total_k, int max_seqlen_q,
                    float softmax_scale, int causal, int window_left, int window_right, float softcap, int dtype,
                    void* stream) {
    if (total_q <= 0 || total_k <= 0 || max_seqlen_q <= 0) return GBATTN_ERR_INVALID_ARG;
    int rc = check_common(B, Hq, Hkv, max_seqlen_q, 1, D, softmax_scale, softcap, dtype);
    if (rc) return rc;
    if ((long long)total_q * Hq > 0x7fffffffLL || (long long)total_k * Hkv > 0x7fffffffLL)
        return GBATTN_ERR_UNSUPPORTED;
    if (dtype == GBATTN_F32) return GBATTN_ERR_UNSUPPORTED;
    if (!q || !k || !v || !out || !cu_seqlens_q || !cu_seqlens_k) return GBATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return GBATTN_ERR_INVALID_ARG;
    if (window_left < -1 || window_right < -1) return GBATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return GBATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) | reinterpret_cast<uintptr_t>(cu_seqlens_k) |
         reinterpret_cast<uintptr_t>(seqused_k)) & 3u)
        return GBATTN_ERR_INVALID_ARG;
    if (lse_out && (reinterpret_cast<uintptr_t>(lse_out) & 3u)) return GBATTN_ERR_INVALID_ARG;
    if (alibi_slopes && (reinterpret_cast<uintptr_t>(alibi_slopes) & 3u)) return GBATTN_ERR_INVALID_ARG;
    const size_t nq = (size_t)total_q * Hq * D * 2, nkv = (size_t)total_k * Hkv * D * 2;
    if (overlaps(out, nq, q, nq) || overlaps(out, nq, k, nkv) || overlaps(out, nq, v, nkv))
        return GBATTN_ERR_INVALID_ARG;

    FwdProblem f{};
    f.q = q;
    f.k = k;
    f.v = v;
    f.slopes = alibi_slopes;
    f.out = out;
    f.lse = lse_out;
    f.B = B;
    f.Hq = Hq;
    f.Hkv = Hkv;
    f.Sq = max_seqlen_q;
    f.Sk = 0;
    f.D = D;
    f.scale = softmax_scale;
    f.causal = causal;
    f.wl = window_left;
    f.wr = window_right;
    f.softcap = softcap;
    f.timeout_ns = g_timeout_ns;
    f.varlen = 1;
    f.f16 = dtype == GBATTN_F16;
    f.cu_q = cu_seqlens_q;
    f.cu_k = cu_seqlens_k;
    f.used_k = seqused_k;
    f.total_q = total_q;
    f.total_k = total_k;
    if (!device_facts(&f.status, &f.num_sms)) return GBATTN_ERR_CUDA;
    CUtensorMap tq, tk, tv, to;
    const bool h = f.f16 != 0;
    if (!cached_map(&tq, q, D, Hq, total_q, 128, 1, h) || !cached_map(&tk, k, D, Hkv, total_k, 128, 1, h) ||
        !cached_map(&tv, v, D, Hkv, total_k, 128, 1, h) || !cached_map(&to, out, D, Hq, total_q, 128, 1, h))
        return GBATTN_ERR_CUDA;
    cudaError_t e = launch_prefill_bf16(f, tq, tk, tv, to, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

// Backward workspace: base-2 lse and Delta per padded query row, row
// intervals and tile summaries, then (recompute only) the forward's lse and
// output.  Every region starts on a 256-byte boundary.
struct BwdLayout {
    size_t lse2, delta, rows, summ, lse, out, total;
};
static BwdLayout bwd_layout(int B, int Hq, int Sq, int D, bool recompute, size_t esz) {
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t sp = backward_sq_pad(Sq), nqt = ((size_t)Sq + 127) / 128;
    BwdLayout L{};
    size_t o = 0;
    L.lse2 = o;
    o += up((size_t)B * Hq * sp * 4);
    L.delta = o;
    o += up((size_t)B * Hq * sp * 4);
    L.rows = o;
    o += up((size_t)B * sp * 8);
    L.summ = o;
    o += up((size_t)B * nqt * 16);
    if (recompute) {
        L.lse = o;
        o += up((size_t)B * Hq * Sq * 4);
        L.out = o;
        o += up((size_t)B * Hq * Sq * D * esz);
    }
    L.total = o;
    return L;
}

size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int Sq, int Sk, int D, int dtype, int recompute) {
    if (check_common(B, Hq, Hkv, Sq, Sk, D, 1.f, 0.f, dtype)) return 0;
    return bwd_layout(B, Hq, Sq, D, recompute != 0, dtype == GBATTN_F32 ? 4 : 2).total;
}

// attn_bwd, with optional events (5): before the forward recompute, then
// those of launch_backward_bf16.
static int bwd_run(const gbattn_bwd_params* a, cudaEvent_t* ev) {
    if (!a) return GBATTN_ERR_INVALID_ARG;
    int rc = check_common(a->B, a->Hq, a->Hkv, a->Sq, a->Sk, a->D, a->softmax_scale, a->softcap, a->dtype);
    if (rc) return rc;
    if (a->B > 65535) return GBATTN_ERR_UNSUPPORTED;  // batch is a grid dimension of the row-interval launch
    if (!a->q || !a->k || !a->v || !a->dout || !a->dq || !a->dk || !a->dv || !a->workspace)
        return GBATTN_ERR_INVALID_ARG;
    if ((a->out == nullptr) != (a->lse == nullptr)) return GBATTN_ERR_INVALID_ARG;
    if (a->causal != 0 && a->causal != 1) return GBATTN_ERR_INVALID_ARG;
    if (a->window_left < -1 || a->window_right < -1) return GBATTN_ERR_INVALID_ARG;
    if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->dout) ||
        (a->out && !aligned16(a->out)) || !aligned16(a->dq) || !aligned16(a->dk) || !aligned16(a->dv))
        return GBATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(a->workspace) & 255u) return GBATTN_ERR_INVALID_ARG;
    if (a->row_kv_bounds && (reinterpret_cast<uintptr_t>(a->row_kv_bounds) & 7u)) return GBATTN_ERR_INVALID_ARG;
    if (a->lse && (reinterpret_cast<uintptr_t>(a->lse) & 3u)) return GBATTN_ERR_INVALID_ARG;
    if (a->alibi_slopes && (reinterpret_cast<uintptr_t>(a->alibi_slopes) & 3u)) return GBATTN_ERR_INVALID_ARG;
    const bool rec = a->out == nullptr;
    const size_t esz = a->dtype == GBATTN_F32 ? 4 : 2;
    const BwdLayout L = bwd_layout(a->B, a->Hq, a->Sq, a->D, rec, esz);
    if (a->workspace_bytes < L.total) return GBATTN_ERR_INVALID_ARG;
    const size_t nq = (size_t)a->B * a->Hq * a->Sq * a->D * esz;
    const size_t nkv = (size_t)a->B * a->Hkv * a->Sk * a->D * esz;
    const void* ins[5] = {a->q, a->k, a->v, a->dout, a->out};
    const size_t ins_n[5] = {nq, nkv, nkv, nq, nq};
    void* grads[3] = {a->dq, a->dk, a->dv};
    const size_t grads_n[3] = {nq, nkv, nkv};
    for (int g = 0; g < 3; ++g) {
        for (int i = 0; i < 5; ++i)
            if (overlaps(grads[g], grads_n[g], ins[i], ins_n[i])) return GBATTN_ERR_INVALID_ARG;
        for (int h = g + 1; h < 3; ++h)
            if (overlaps(grads[g], grads_n[g], grads[h], grads_n[h])) return GBATTN_ERR_INVALID_ARG;
        if (overlaps(grads[g], grads_n[g], a->workspace, L.total)) return GBATTN_ERR_INVALID_ARG;
    }

    BwdProblem b{};
    if (!device_facts(&b.status, &b.num_sms)) return GBATTN_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(a->workspace);
    const void* out = a->out;
    const float* lse = a->lse;
    if (ev && cudaEventRecord(ev[0], static_cast<cudaStream_t>(a->stream)) != cudaSuccess) return GBATTN_ERR_CUDA;
    if (rec) {
        // recompute the forward's output and lse into the workspace
        gbattn_fwd_params f{};
        f.q = a->q;
        f.k = a->k;
        f.v = a->v;
        f.alibi_slopes = a->alibi_slopes;
        f.row_kv_bounds = a->row_kv_bounds;
        f.out = ws + L.out;
        f.lse_out = reinterpret_cast<float*>(ws + L.lse);
        f.B = a->B;
        f.Hq = a->Hq;
        f.Hkv = a->Hkv;
        f.Sq = a->Sq;
        f.Sk = a->Sk;
        f.D = a->D;
        f.softmax_scale = a->softmax_scale;
        f.causal = a->causal;
        f.window_left = a->window_left;
        f.window_right = a->window_right;
        f.softcap = a->softcap;
        f.dtype = a->dtype;
        f.stream = a->stream;
        rc = attn_fwd_ex(&f);
        if (rc) return rc;
        out = f.out;
        lse = f.lse_out;
    }
    b.q = a->q;
    b.k = a->k;
    b.v = a->v;
    b.out = out;
    b.lse = lse;
    b.dout = a->dout;
    b.slopes = a->alibi_slopes;
    b.row_bounds = a->row_kv_bounds;
    b.dq = a->dq;
    b.dk = a->dk;
    b.dv = a->dv;
    b.B = a->B;
    b.Hq = a->Hq;
    b.Hkv = a->Hkv;
    b.Sq = a->Sq;
    b.Sk = a->Sk;
    b.D = a->D;
    b.scale = a->softmax_scale;
    b.causal = a->causal;
    b.wl = a->window_left;
    b.wr = a->window_right;
    b.softcap = a->softcap;
    b.f16 = a->dtype == GBATTN_F16;
    b.ws_lse2 = reinterpret_cast<float*>(ws + L.lse2);
    b.ws_delta = reinterpret_cast<float*>(ws + L.delta);
    b.ws_rows = reinterpret_cast<int32_t*>(ws + L.rows);
    b.ws_summ = reinterpret_cast<int32_t*>(ws + L.summ);
    b.timeout_ns = g_timeout_ns;
    if (a->dtype == GBATTN_F32) {
        cudaError_t e = launch_backward_f32(b, static_cast<cudaStream_t>(a->stream), ev ? ev + 1 : nullptr);
        return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
    }
    const bool h = b.f16 != 0;
    CUtensorMap tq, tdo, tk, tv, to;
    if (!cached_map(&tq, a->q, a->D, a->Sq, (uint64_t)a->B * a->Hq, 128, 0, h) ||
        !cached_map(&tdo, a->dout, a->D, a->Sq, (uint64_t)a->B * a->Hq, 128, 0, h) ||
        !cached_map(&tk, a->k, a->D, a->Sk, (uint64_t)a->B * a->Hkv, 128, 0, h) ||
        !cached_map(&tv, a->v, a->D, a->Sk, (uint64_t)a->B * a->Hkv, 128, 0, h) ||
        !cached_map(&to, out, a->D, a->Sq, (uint64_t)a->B * a->Hq, 128, 0, h))
        return GBATTN_ERR_CUDA;
    cudaError_t e = launch_backward_bf16(b, tq, tdo, tk, tv, to, static_cast<cudaStream_t>(a->stream),
                                         ev ? ev + 1 : nullptr);
    return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

int attn_bwd(const gbattn_bwd_params* a) { return bwd_run(a, nullptr); }

int attn_bwd_phase_times(const gbattn_bwd_params* a, int reps, float* phase_ms) {
    if (!a || !phase_ms || reps <= 0 || reps > 100000) return GBATTN_ERR_INVALID_ARG;
    cudaEvent_t ev[5] = {};
    for (int i = 0; i < 5; ++i)
        if (cudaEventCreate(&ev[i]) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
            return GBATTN_ERR_CUDA;
        }
    double acc[4] = {0, 0, 0, 0};
    int rc = GBATTN_OK;
    for (int r = 0; r < reps && rc == GBATTN_OK; ++r) {
        rc = bwd_run(a, ev);
        if (rc == GBATTN_OK && cudaEventSynchronize(ev[4]) != cudaSuccess) rc = GBATTN_ERR_CUDA;
        for (int i = 0; i < 4 && rc == GBATTN_OK; ++i) {
            float ms = 0.f;
            if (cudaEventElapsedTime(&ms, ev[i], ev[i + 1]) != cudaSuccess) rc = GBATTN_ERR_CUDA;
            acc[i] += ms;
        }
    }
    for (int i = 0; i < 5; ++i) cudaEventDestroy(ev[i]);
    if (rc == GBATTN_OK) {
        for (int i = 0; i < 4; ++i) phase_ms[i] = (float)(acc[i] / reps);
        if (a->dtype != GBATTN_F32) {
            // the 16-bit path launches dQ before dK / dV
            phase_ms[2] = (float)(acc[3] / reps);
            phase_ms[3] = (float)(acc[2] / reps);
        }
    }
    return rc;
}

static int decode_plan(int B, int Hq, int Hkv, int Sk, int D, int num_splits, int* splits, int* chunk) {
    if (check_common(B, Hq, Hkv, 1, Sk, D, 1.f, 0.f, GBATTN_BF16)) return -1;
    if (num_splits < 0) return -1;
    unsigned int* st = nullptr;
    int sms = 0;
    if (!device_facts(&st, &sms)) sms = 148;
    decode_split_plan(B, Hkv, Sk, sms, num_splits, splits, chunk);
    return 0;
}

// Split plan of a decode whose query admits only the keys of a left window
// (window_left >= 0): the plan over the 64-key tiles such a window can touch,
// with no more splits than the plan over all Sk keys, which sizes the
// caller's workspace.
static void decode_plan_window(int B, int Hkv, int Sk, int wl, int sms, int requested, int* splits, int* chunk) {
    decode_split_plan(B, Hkv, Sk, sms, requested, splits, chunk);
    if (wl < 0) return;
    const long long keys = wl + 1LL < (long long)Sk ? wl + 1LL : (long long)Sk;  // admitted keys, at most
    const long long all_tiles = (Sk + 63LL) / 64;
    const long long span = (keys + 62) / 64 + 1;  // 64-key tiles a range of `keys` keys can touch
    if (span >= all_tiles) return;
    int s2 = 0, c2 = 0;
    decode_split_plan(B, Hkv, (int)(span * 64), sms, requested, &s2, &c2);
    if (s2 > *splits) decode_split_plan(B, Hkv, (int)(span * 64), sms, *splits, &s2, &c2);
    *splits = s2;
    *chunk = c2;
}

size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int Sk, int D, int num_splits) {
    int splits = 0, chunk = 0;
    if (decode_plan(B, Hq, Hkv, Sk, D, num_splits, &splits, &chunk)) return 0;
    if (splits <= 1) return 0;
    const size_t rows = (size_t)B * Hq * splits;
    const size_t o_bytes = rows * D * sizeof(float);
    return o_bytes + ((rows * sizeof(float) + 15) & ~size_t(15));
}

int attn_decode(const void* q, const void* k, const void* v, const float* alibi_slopes, void* out, float* lse_out,
                int B, int Hq, int Hkv, int Sk, int D, float softmax_scale, float softcap, int window_left,
                int window_right, int num_splits, void* workspace, size_t workspace_bytes, int dtype, void* stream) {
    int rc = check_common(B, Hq, Hkv, 1, Sk, D, softmax_scale, softcap, dtype);
    if (rc) return rc;
    if (dtype == GBATTN_F32) return GBATTN_ERR_UNSUPPORTED;
    if (!q || !k || !v || !out || num_splits < 0) return GBATTN_ERR_INVALID_ARG;
    if (window_left < -1 || window_right < -1) return GBATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return GBATTN_ERR_INVALID_ARG;
    if (lse_out && (reinterpret_cast<uintptr_t>(lse_out) & 3u)) return GBATTN_ERR_INVALID_ARG;
    if (alibi_slopes && (reinterpret_cast<uintptr_t>(alibi_slopes) & 3u)) return GBATTN_ERR_INVALID_ARG;
    const size_t nq = (size_t)B * Hq * D * 2, nkv = (size_t)B * Hkv * Sk * D * 2;
    if (overlaps(out, nq, q, nq) || overlaps(out, nq, k, nkv) || overlaps(out, nq, v, nkv))
        return GBATTN_ERR_INVALID_ARG;

    DecodeProblem f{};
    if (!device_facts(&f.status, &f.num_sms)) return GBATTN_ERR_CUDA;
    decode_plan_window(B, Hkv, Sk, window_left, f.num_sms, num_splits, &f.num_splits, &f.chunk);
    const size_t need = f.num_splits > 1 ? (size_t)B * Hq * f.num_splits * D * 4 +
                                               (((size_t)B * Hq * f.num_splits * 4 + 15) & ~size_t(15))
                                         : 0;
    if (need > 0) {
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) return GBATTN_ERR_INVALID_ARG;
        if (overlaps(workspace, need, out, nq) || overlaps(workspace, need, q, nq) ||
            overlaps(workspace, need, k, nkv) || overlaps(workspace, need, v, nkv))
            return GBATTN_ERR_INVALID_ARG;
        f.ws_o = static_cast<float*>(workspace);
        f.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + (size_t)B * Hq * f.num_splits * D * 4);
    }
    f.q = q;
    f.k = k;
    f.v = v;
    f.slopes = alibi_slopes;
    f.out = out;
    f.lse = lse_out;
    f.B = B;
    f.Hq = Hq;
    f.Hkv = Hkv;
    f.Sk = Sk;
    f.D = D;
    f.scale = softmax_scale;
    f.softcap = softcap;
    f.wl = window_left;
    f.auto_splits = num_splits == 0;
    f.timeout_ns = g_timeout_ns;
    f.f16 = dtype == GBATTN_F16;
    CUtensorMap tk, tv;
    if (!cached_map(&tk, k, D, Sk, (uint64_t)B * Hkv, 64, 0, f.f16 != 0) ||
        !cached_map(&tv, v, D, Sk, (uint64_t)B * Hkv, 64, 0, f.f16 != 0))
        return GBATTN_ERR_CUDA;
    cudaError_t e = launch_decode_bf16(f, tk, tv, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

static bool paged_geometry(int block_size, int max_blocks, int num_blocks, int* max_ctx) {
    if (block_size < 16 || block_size > 1024 || (block_size & (block_size - 1))) return false;
    if (max_blocks <= 0 || num_blocks <= 0) return false;
    const long long mc = (long long)max_blocks * block_size, pool = (long long)num_blocks * block_size;
    if (mc > 0x7fffffffLL || pool >= 0x7fffffffLL) return false;
    *max_ctx = (int)mc;
    return true;
}

size_t attn_decode_paged_workspace_size(int B, int Hq, int Hkv, int max_blocks_per_seq, int block_size, int D,
                                        int num_splits) {
    int max_ctx = 0;
    if (!paged_geometry(block_size, max_blocks_per_seq, 1, &max_ctx)) return 0;
    return attn_decode_workspace_size(B, Hq, Hkv, max_ctx, D, num_splits);
}

int attn_decode_paged(const void* q, const void* k_cache, const void* v_cache, const uint32_t* block_table,
                      const uint32_t* context_lens, const float* alibi_slopes, void* out, float* lse_out, int B,
                      int Hq, int Hkv, int D, int num_blocks, int block_size, int max_blocks_per_seq,
                      float softmax_scale, float softcap, int window_left, int window_right, int num_splits,
                      void* workspace, size_t workspace_bytes, int dtype, void* stream) {
    int max_ctx = 0;
    if (!paged_geometry(block_size, max_blocks_per_seq, num_blocks, &max_ctx)) return GBATTN_ERR_INVALID_ARG;
    int rc = check_common(B, Hq, Hkv, 1, max_ctx, D, softmax_scale, softcap, dtype);
    if (rc) return rc;
    if (dtype == GBATTN_F32) return GBATTN_ERR_UNSUPPORTED;
    if (!q || !k_cache || !v_cache || !block_table || !context_lens || !out || num_splits < 0)
        return GBATTN_ERR_INVALID_ARG;
    if (window_left < -1 || window_right < -1) return GBATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return GBATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(block_table) | reinterpret_cast<uintptr_t>(context_lens)) & 3u)
        return GBATTN_ERR_INVALID_ARG;
    if (lse_out && (reinterpret_cast<uintptr_t>(lse_out) & 3u)) return GBATTN_ERR_INVALID_ARG;
    if (alibi_slopes && (reinterpret_cast<uintptr_t>(alibi_slopes) & 3u)) return GBATTN_ERR_INVALID_ARG;
    const size_t nq = (size_t)B * Hq * D * 2, npool = (size_t)num_blocks * block_size * Hkv * D * 2;
    if (overlaps(out, nq, q, nq) || overlaps(out, nq, k_cache, npool) || overlaps(out, nq, v_cache, npool))
        return GBATTN_ERR_INVALID_ARG;

    DecodeProblem f{};
    if (!device_facts(&f.status, &f.num_sms)) return GBATTN_ERR_CUDA;
    decode_plan_window(B, Hkv, max_ctx, window_left, f.num_sms, num_splits, &f.num_splits, &f.chunk);
    const size_t need = f.num_splits > 1 ? (size_t)B * Hq * f.num_splits * D * 4 +
                                               (((size_t)B * Hq * f.num_splits * 4 + 15) & ~size_t(15))
                                         : 0;
    if (need > 0) {
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) return GBATTN_ERR_INVALID_ARG;
        if (overlaps(workspace, need, out, nq) || overlaps(workspace, need, q, nq) ||
            overlaps(workspace, need, k_cache, npool) || overlaps(workspace, need, v_cache, npool))
            return GBATTN_ERR_INVALID_ARG;
        f.ws_o = static_cast<float*>(workspace);
        f.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + (size_t)B * Hq * f.num_splits * D * 4);
    }
    f.q = q;
    f.k = k_cache;
    f.v = v_cache;
    f.slopes = alibi_slopes;
    f.out = out;
    f.lse = lse_out;
    f.B = B;
    f.Hq = Hq;
    f.Hkv = Hkv;
    f.Sk = max_ctx;
    f.D = D;
    f.scale = softmax_scale;
    f.softcap = softcap;
    f.wl = window_left;
    f.auto_splits = num_splits == 0;
    f.timeout_ns = g_timeout_ns;
    f.paged = 1;
    f.block_table = block_table;
    f.context_lens = context_lens;
    f.max_blocks = max_blocks_per_seq;
    f.block_size = block_size;
    f.num_blocks = num_blocks;
    f.f16 = dtype == GBATTN_F16;
    const uint32_t box = block_size < 64 ? (uint32_t)block_size : 64u;
    const uint64_t rows = (uint64_t)num_blocks * block_size;
    CUtensorMap tk, tv;
    if (!cached_map(&tk, k_cache, D, Hkv, rows, box, 1, f.f16 != 0) ||
        !cached_map(&tv, v_cache, D, Hkv, rows, box, 1, f.f16 != 0))
        return GBATTN_ERR_CUDA;
    cudaError_t e = launch_decode_bf16(f, tk, tv, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_CUDA;
}

const char* gbattn_status_string(int status) {
    switch (status) {
        case GBATTN_OK: return "ok";
        case GBATTN_ERR_INVALID_ARG: return "invalid argument";
        case GBATTN_ERR_UNSUPPORTED: return "unsupported problem";
        case GBATTN_ERR_CUDA: return "CUDA error";
        case GBATTN_ERR_DEVICE: return "device status word set (a bounded wait ran out)";
        default: return "unknown status";
    }
}

unsigned int gbattn_device_status(void* stream, int clear) {
    unsigned int* st = nullptr;
    int sms = 0;
    if (!device_facts(&st, &sms)) return ~0u;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int v = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return ~0u;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof v) != cudaSuccess) return ~0u;
    if (clear) {
        unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_status_word, &z, sizeof z) != cudaSuccess) return ~0u;
    }
    return v;
}

uint64_t gbattn_set_wait_timeout_ns(uint64_t ns) {
    std::lock_guard<std::mutex> lk(g_mu);
    uint64_t old = g_timeout_ns;
    g_timeout_ns = ns;
    return old;
}

int gbattn_version(void) { return 100; }

}  // extern "C"
