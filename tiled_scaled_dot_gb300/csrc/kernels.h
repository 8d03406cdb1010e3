// kernels.h -- internal interface between the C ABI layer (api.cu) and the
// kernel translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gbattn {

// A validated forward problem (sizes checked, pointers non-null where required).
struct FwdProblem {
    const void* q;
    const void* k;
    const void* v;
    const float* slopes;        // [Hq] or nullptr
    const int32_t* row_bounds;  // [B, Sq, 2] or nullptr
    void* out;
    float* lse;                 // [B, Hq, Sq] or nullptr
    int B, Hq, Hkv, Sq, Sk, D;
    float scale;
    int causal;
    int wl, wr;                 // -1 = unbounded
    float softcap;              // 0 = none
    unsigned int* status;       // device status word
    unsigned long long timeout_ns;
    int num_sms;
    // packed variable-length sequences (q / out [total_q, Hq, D], k / v
    // [total_k, Hkv, D]); Sq is then the longest sequence's query count
    int f16;                    // 16-bit inputs are fp16 (else bf16)
    int varlen;
    const int* cu_q;            // [B + 1]
    const int* cu_k;            // [B + 1]
    const int* used_k;          // [B] or nullptr
    int total_q, total_k;
};

struct DecodeProblem {
    const void* q;
    const void* k;
    const void* v;
    const float* slopes;
    void* out;
    float* lse;
    int B, Hq, Hkv, Sk, D;
    float scale;
    float softcap;
    int wl;                     // left window at the query's position (the last key); -1 = none
    int num_splits;             // resolved (>= 1)
    int auto_splits;            // num_splits came from the automatic plan (the caller asked for 0)
    int chunk;                  // keys per split, multiple of 64
    float* ws_o;                // [B, Hq, num_splits, D] fp32 (num_splits > 1)
    float* ws_lse;              // [B, Hq, num_splits] fp32 (num_splits > 1)
    unsigned int* status;
    unsigned long long timeout_ns;
    int num_sms;
    // paged cache (k, v are pools [num_blocks, block_size, Hkv, D]); Sk is the
    // longest context the block table can hold (max_blocks * block_size)
    int f16;                       // fp16 inputs / output (else bf16)
    int paged;
    const uint32_t* block_table;   // [B, max_blocks]
    const uint32_t* context_lens;  // [B]
    int max_blocks, block_size, num_blocks;
};

// A validated backward problem.  The forward's out and lse are given or were
// recomputed into the workspace before the launch.
struct BwdProblem {
    const void* q;
    const void* k;
    const void* v;
    const void* out;            // [B, Hq, Sq, D]
    const float* lse;           // [B, Hq, Sq]
    const void* dout;           // [B, Hq, Sq, D]
    const float* slopes;        // [Hq] or nullptr
    const int32_t* row_bounds;  // [B, Sq, 2] or nullptr
    void* dq;                   // [B, Hq, Sq, D]
    void* dk;                   // [B, Hkv, Sk, D]
    void* dv;                   // [B, Hkv, Sk, D]
    int B, Hq, Hkv, Sq, Sk, D;
    float scale;
    int causal;
    int wl, wr;
    float softcap;
    int f16;
    // workspace regions (Sq_pad = Sq rounded up to 128)
    float* ws_lse2;             // [B * Hq * Sq_pad]
    float* ws_delta;            // [B * Hq * Sq_pad]
    int32_t* ws_rows;           // [B * Sq_pad * 2]
    int32_t* ws_summ;           // [B * ceil(Sq / 128) * 4]
    unsigned int* status;
    unsigned long long timeout_ns;
    int num_sms;
};

// Bits of the device status word: which wait gave up.
enum : unsigned int {
    ST_PREFILL_PRODUCER = 1u << 0,
    ST_PREFILL_MMA = 1u << 1,
    ST_PREFILL_SOFTMAX = 1u << 2,
    ST_PREFILL_EPILOGUE = 1u << 3,
    ST_PREFILL_VARLEN_RANGE = 1u << 4,  // packed-sequence offsets / lengths outside the tensors
    ST_DECODE_PRODUCER = 1u << 8,
    ST_DECODE_CONSUMER = 1u << 9,
    ST_DECODE_PAGED_RANGE = 1u << 10,  // a physical block index >= num_blocks, or a context past the table
    ST_BWD_PRODUCER = 1u << 12,
    ST_BWD_MMA = 1u << 13,
    ST_BWD_EW = 1u << 14,
    ST_DIAG = 1u << 16,
};

// 3-D 16-bit (bf16, or fp16 when f16) tensor map over a contiguous
// [planes][rows][cols] array with a {64, box_rows, 1} box and 128-byte
// swizzle; out-of-range rows read as 0.
bool encode_map_bf16_3d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t planes,
                        uint32_t box_rows, bool f16 = false);

// 3-D bf16 tensor map over a paged pool [rows][heads][cols] (rows = num_blocks *
// block_size tokens) with a {64, 1, box_rows} box and 128-byte swizzle: one
// box is box_rows consecutive tokens of one head; rows past the pool read as 0.
bool encode_map_pool_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t heads, uint64_t rows,
                          uint32_t box_rows, bool f16 = false);

// Kernel launchers.  Each returns the launch's cudaError_t.
cudaError_t launch_prefill_bf16(const FwdProblem& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& to, cudaStream_t stream);
cudaError_t launch_prefill_f32(const FwdProblem& p, cudaStream_t stream);
cudaError_t launch_decode_bf16(const DecodeProblem& p, const CUtensorMap& tk, const CUtensorMap& tv,
                               cudaStream_t stream);

// to maps the forward output O (read for Delta).  ev (optional, 4 events) is
// recorded before the prep launch, before the dQ launch, before the dK / dV
// launch and after it.
cudaError_t launch_backward_bf16(const BwdProblem& p, const CUtensorMap& tq, const CUtensorMap& tdo,
                                 const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                                 cudaStream_t stream, cudaEvent_t* ev = nullptr);
// The same for fp32 inputs (SIMT).
cudaError_t launch_backward_f32(const BwdProblem& p, cudaStream_t stream, cudaEvent_t* ev = nullptr);
// The backward's first launch (both storage types): each query row's admissible
// key interval and the 128-row tile summaries, into the workspace.
cudaError_t launch_backward_rows(const BwdProblem& p, cudaStream_t stream);
// Rows of the backward's per-row workspace arrays: Sq rounded up to 128.
size_t backward_sq_pad(int Sq);

// Device address of the library's status word and the SM count of the current
// device (looked up once per device).  False if the CUDA runtime fails.
bool device_facts(unsigned int** status, int* num_sms);

// Decode split choice shared by attn_decode and attn_decode_workspace_size.
void decode_split_plan(int B, int Hkv, int Sk, int num_sms, int requested, int* num_splits, int* chunk);

}  // namespace gbattn
