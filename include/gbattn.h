/*
 * gbattn.h -- C ABI of the GB300 (sm_103a) tiled scaled-dot-product attention
 * library (libgbattn.so).
 *
 * Operation (attention.fkc.md, "attention_naive" and "attention_flash";
 * "gfx942 unified attention, from the math up", sections 1-4): for every batch
 * b, query head h and query row i, with kv head g = h / (Hq / Hkv) (the GQA
 * broadcast stated in the header of attention.fkc.md),
 *
 *     s_j = softmax_scale * (Q[b,h,i,:] . K[b,g,j,:])
 *     s_j = softcap * tanh(s_j / softcap)        when softcap > 0
 *     s_j = s_j + alibi_slopes[h] * (j - i)      when alibi_slopes != NULL
 *     s_j = -inf                                 when key j is not admissible
 *     O[b,h,i,:] = sum_j softmax(s)_j V[b,g,j,:] and lse = log sum_j exp(s_j)
 *
 * Admissible (attention.fkc.md, header: position_admissible): not (causal and
 * j > i), not (window_left >= 0 and j + window_left < i), not (window_right
 * >= 0 and j > i + window_right), and, in attn_fwd_ex only, lo <= j <= hi for
 * the row's entry of row_kv_bounds.  A row with no admissible key is the
 * all-zero row, with lse = -inf (attention.fkc.md, attention_naive).  Causal
 * alignment is top-left (key j is in the future of query i when j > i), as in
 * position_admissible.
 *
 * The result is computed by the tiled online-softmax recurrence ("gfx942
 * unified attention", section 3): running max m, denominator l, rescale
 * alpha = exp(m_old - m_new), final O = o / l.
 *
 * Layout (attention.fkc.md, header): every tensor is contiguous, row-major,
 * zero offset, batch first then heads: q [B, Hq, Sq, D], k and v
 * [B, Hkv, Sk, D], out [B, Hq, Sq, D], lse [B, Hq, Sq].
 *
 * Ownership: the caller owns every buffer.  All pointers are device pointers
 * of the current CUDA device, 16-byte aligned.  The library allocates no device
 * memory in any call; it keeps a small host cache of TMA descriptors.  Calls
 * enqueue work on `stream` (a cudaStream_t; NULL = the legacy default stream)
 * and return without synchronising.  `out` must not overlap any input.
 * The library looks up the device addresses of its own module variables (the
 * status word, the scratch array of attn_decode_noalloc) once per device and
 * keeps them: a cudaDeviceReset may move them, so a process must not call the
 * library on a device after resetting it.
 *
 * Errors: every call returns a status code and never aborts the process.
 * Argument errors are detected on the host before anything is launched.
 * GBATTN_ERR_CUDA carries a launch failure (the CUDA error is left in
 * cudaGetLastError).  A kernel that meets a bounded-wait timeout records it in
 * a device status word which gbattn_device_status() reads.
 */
#ifndef GBATTN_H_
#define GBATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of q, k, v and out. */
typedef enum {
    GBATTN_BF16 = 0, /* bfloat16 storage, fp32 accumulation, bf16 output (RNE)   */
    GBATTN_F32 = 1,  /* float32 storage and arithmetic (SIMT FFMA, no TF32)       */
    GBATTN_F16 = 2   /* float16 storage, fp32 accumulation, fp16 output (RNE)     */
} gbattn_dtype;

enum {
    GBATTN_OK = 0,
    GBATTN_ERR_INVALID_ARG = 1, /* null pointer, bad size, Hq % Hkv != 0, ...        */
    GBATTN_ERR_UNSUPPORTED = 2, /* valid problem outside what the kernels implement  */
    GBATTN_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed              */
    GBATTN_ERR_DEVICE = 4       /* the device status word is set (bounded wait ran out) */
};

/*
 * attn_fwd -- multi-head SDPA forward (prefill).
 * attention.fkc.md, attention_naive / attention_flash (operation and
 * AttentionParams: softmax_scale, causal, window_size_left/right, softcap,
 * optional ALiBi slopes [Hq]).
 *
 *  q, k, v        device, layout above, element type `dtype`.
 *  alibi_slopes   device fp32 [Hq] or NULL (no ALiBi).
 *  out            device [B, Hq, Sq, D], element type `dtype`, written fully.
 *  B, Hq, Hkv, Sq, Sk, D   sizes, all > 0; Hq % Hkv == 0.
 *                 D must be 64 or 128 (else GBATTN_ERR_UNSUPPORTED).
 *  softmax_scale  finite and > 0 (usually 1/sqrt(D)).
 *  causal         0 or 1.
 *  window_left, window_right   -1 = unbounded (None), else >= 0.
 *  softcap        0 = none, else finite and > 0.
 *  dtype          GBATTN_BF16, GBATTN_F16 (tensor cores, fp32 accumulation)
 *                 or GBATTN_F32 (SIMT).
 *  stream         cudaStream_t.
 */
int attn_fwd(const void* q, const void* k, const void* v, const float* alibi_slopes, void* out, int B, int Hq,
             int Hkv, int Sq, int Sk, int D, float softmax_scale, int causal, int window_left, int window_right,
             float softcap, int dtype, void* stream);

/*
 * attn_fwd_ex -- attn_fwd with two optional extras:
 *  lse_out        device fp32 [B, Hq, Sq] or NULL: natural-log sum of exp of
 *                 the admissible scores; -inf for a row with none.  The
 *                 online recurrence's m + ln(l) ("gfx942 unified attention",
 *                 section 3).
 *  row_kv_bounds  device int32 [B, Sq, 2] or NULL: inclusive key range
 *                 [lo, hi] admitted for query row (b, i) in addition to the
 *                 mask above; lo > hi admits no key, so the row is zero.
 *                 (Reading of the pages' "window that masks all keys" for
 *                 single rows; the same bounds apply to every head.)
 */
typedef struct {
    const void* q;
    const void* k;
    const void* v;
    const float* alibi_slopes;
    const int32_t* row_kv_bounds;
    void* out;
    float* lse_out;
    int B, Hq, Hkv, Sq, Sk, D;
    float softmax_scale;
    int causal;
    int window_left, window_right;
    float softcap;
    int dtype;
    void* stream;
} gbattn_fwd_params;

int attn_fwd_ex(const gbattn_fwd_params* p);

/*
 * attn_fwd_varlen -- attention over packed variable-length sequences
 * ("gfx942 unified attention", section 5: queries packed [total_q, heads, D]
 * with a cu_seqlens_q prefix sum, seqused_k carrying each sequence's KV
 * length; section 4: the causal mask aligned bottom-right).  Sequence b
 * (0 <= b < B) has queries q[cu_seqlens_q[b] .. cu_seqlens_q[b+1]) and keys
 * k, v[cu_seqlens_k[b] .. cu_seqlens_k[b+1]), of which the first
 * seqused_k[b] are live (all of them when seqused_k is NULL).  With q_len
 * queries and kv_len live keys, query i sits at position kv_len - q_len + i:
 * causal admits keys j <= that position, window_left / window_right (-1 =
 * none) bound j to [pos - window_left, pos + window_right], and ALiBi adds
 * slope_h * (j - pos).  Rows with no admissible key are zero (lse -inf).
 * Softcap and scale as in attn_fwd.
 *
 *  q, out         device [total_q, Hq, D]; k, v device [total_k, Hkv, D]; all of
 *                 type `dtype`.
 *  cu_seqlens_q, cu_seqlens_k  device int32 [B + 1], non-decreasing, from 0;
 *                 cu_seqlens_q[B] = total_q, cu_seqlens_k[B] <= total_k.
 *  seqused_k      device int32 [B] or NULL.
 *  lse_out        device fp32 [Hq, total_q] (natural log) or NULL.
 *  max_seqlen_q   at least every sequence's query count (sizes the work list).
 *  dtype          GBATTN_BF16 or GBATTN_F16 (tensor cores, fp32 accumulation;
 *                 GBATTN_F32 returns GBATTN_ERR_UNSUPPORTED); D 64 or 128.
 * Offsets or lengths outside the tensors (or a sequence longer than
 * max_seqlen_q) are clamped on the device and set bit 4 of the device status
 * word; the output is then unspecified.
 */
int attn_fwd_varlen(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                    const int32_t* cu_seqlens_k, const int32_t* seqused_k, const float* alibi_slopes, void* out,
                    float* lse_out, int B, int Hq, int Hkv, int D, int total_q, int total_k, int max_seqlen_q,
                    float softmax_scale, int causal, int window_left, int window_right, float softcap, int dtype,
                    void* stream);

/*
 * attn_decode_workspace_size -- bytes of device workspace attn_decode needs
 * for this problem and split count (num_splits = 0 picks the split count
 * attn_decode picks, for the current device).  Returns 0 for invalid sizes.
 */
size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int Sk, int D, int num_splits);

/*
 * attn_decode -- decode step: one query row per (b, h), the newest token of
 * its sequence, against the Sk keys before it.
 * "gfx942 unified attention", section 4 (decode runs non-causal: the single
 * query sees every key) and section 8 (split-KV: the keys are split across
 * thread blocks and the partial softmax-weighted outputs combined).  The
 * combine is the online recurrence of section 3 applied across splits, in a
 * fixed split order, so reruns are bitwise identical.
 *
 * The query sits at position Sk - 1, the last key (the alignment under which a
 * non-causal single row is the causal one, and the decode position of
 * attention.fkc.md, attention_paged_naive): the ALiBi term is
 * alibi_slopes[h] * (j - (Sk - 1)), and the window of the dense contract
 * (attention.fkc.md, header: window_size_left/right) admits keys
 * j >= Sk - 1 - window_left; no key lies after the query, so window_right
 * admits every key.  Tiles before the window are not read.
 *
 *  q              device [B, Hq, 1, D]; k, v device [B, Hkv, Sk, D].
 *  alibi_slopes   device fp32 [Hq] or NULL.
 *  out            device [B, Hq, 1, D]; lse_out device fp32 [B, Hq] or NULL.
 *  softcap        0 = none, else > 0.
 *  window_left, window_right   -1 = unbounded (None), else >= 0.
 *  num_splits     0 = automatic; else the number of key chunks (each chunk is a
 *                 multiple of 64 keys; chunks past the end are empty).  With a
 *                 left window the chunks cover the window's keys only.
 *  workspace      device scratch of at least
 *                 attn_decode_workspace_size(B, Hq, Hkv, Sk, D, num_splits)
 *                 bytes, 16-byte aligned (may be NULL when that size is 0).
 *                 Its contents need no initialisation and are not preserved.
 *  dtype          GBATTN_BF16 or GBATTN_F16 (GBATTN_F32 returns GBATTN_ERR_UNSUPPORTED).
 *  D              64 or 128.
 */
int attn_decode(const void* q, const void* k, const void* v, const float* alibi_slopes, void* out, float* lse_out,
                int B, int Hq, int Hkv, int Sk, int D, float softmax_scale, float softcap, int window_left,
                int window_right, int num_splits, void* workspace, size_t workspace_bytes, int dtype, void* stream);

/*
 * attn_decode_noalloc -- attn_decode without a caller-provided workspace.
 * The pages have no counterpart to this entry point: it exists for callers
 * that cannot allocate device memory themselves (an engine whose own pool owns
 * all device memory, or a latency-critical loop that must not call cudaMalloc,
 * which can synchronise the device).  Same arguments and results as
 * attn_decode without a window, minus workspace / workspace_bytes.
 *
 * The split partials go to a fixed scratch array of GBATTN_NOALLOC_SCRATCH_BYTES
 * in the library's own device module.  Under CUDA's default lazy module
 * loading the array occupies device memory on each GPU where this entry has
 * been called (its module loads on first use); with eager loading
 * (CUDA_MODULE_LOADING=EAGER) on each GPU where the library is loaded.  It is
 * held until the process exits.  Nothing is allocated by this call.  A problem whose
 * workspace (attn_decode_workspace_size) exceeds that size returns
 * GBATTN_ERR_UNSUPPORTED; use attn_decode with your own workspace then.
 * All calls share the one array and it keeps the last call's contents, so
 * calls that overlap on the GPU (different streams or host threads) race;
 * serialise them.  The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture begins.
 */
#define GBATTN_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int attn_decode_noalloc(const void* q, const void* k, const void* v, const float* alibi_slopes, void* out,
                        float* lse_out, int B, int Hq, int Hkv, int Sk, int D, float softmax_scale, float softcap,
                        int num_splits, int dtype, void* stream);

/*
 * attn_decode_paged -- decode step over a paged KV cache (attention.fkc.md,
 * "attention_paged_naive": a per-sequence block table over a blocked pool,
 * per-sequence context lengths, the causal mask implicit at the query's
 * absolute position).  One query row per (b, h) (Sq = 1): its keys are the
 * logical positions k_pos = 0 .. context_lens[b] - 1, key k_pos living in pool
 * block block_table[b, k_pos / block_size], row k_pos % block_size.  The query
 * sits at abs_pos = context_lens[b] - 1, so every key of the context is
 * admissible and the ALiBi term is slope_h * (k_pos - abs_pos).  An optional
 * left window (the dense contract's window_size_left at abs_pos) admits only
 * keys k_pos >= abs_pos - window_left; window_right admits every key.  A
 * sequence with context length 0 outputs the zero row (lse -inf).  Split-KV
 * over keys and the log-sum-exp combine as in attn_decode.
 *
 *  q              device [B, Hq, 1, D] (bf16 or fp16, see dtype).
 *  k_cache, v_cache  device pools [num_blocks, block_size, Hkv, D], same type.
 *  block_table    device uint32 [B, max_blocks_per_seq]; only the entries of
 *                 blocks that hold keys of the context are read.
 *  context_lens   device uint32 [B].
 *  alibi_slopes   device fp32 [Hq] or NULL.
 *  out            device [B, Hq, 1, D]; lse_out device fp32 [B, Hq] or NULL.
 *  block_size     a power of two, 16 .. 1024.
 *  num_splits, workspace  as in attn_decode, sized by
 *                 attn_decode_paged_workspace_size (for the longest context
 *                 the table can hold, max_blocks_per_seq * block_size).
 *  dtype          GBATTN_BF16 or GBATTN_F16 (q, pools and out alike); D 64 or 128.
 * The contract's bounds check of physical block indices happens on the device:
 * an index >= num_blocks, or a context length above max_blocks_per_seq *
 * block_size, sets bit 10 of the device status word (gbattn_device_status);
 * the output is then unspecified.  Such keys are never read from outside the
 * pool.
 */
size_t attn_decode_paged_workspace_size(int B, int Hq, int Hkv, int max_blocks_per_seq, int block_size, int D,
                                        int num_splits);
int attn_decode_paged(const void* q, const void* k_cache, const void* v_cache, const uint32_t* block_table,
                      const uint32_t* context_lens, const float* alibi_slopes, void* out, float* lse_out, int B,
                      int Hq, int Hkv, int D, int num_blocks, int block_size, int max_blocks_per_seq,
                      float softmax_scale, float softcap, int window_left, int window_right, int num_splits,
                      void* workspace, size_t workspace_bytes, int dtype, void* stream);

/*
 * attn_bwd -- attention backward by recompute (attention.fkc.md,
 * "attention_flash_backward"): given dO, the gradients of the forward above
 * (same flags, same causal / window / row-bound mask, same softcap and ALiBi),
 *
 *     P      = the forward's softmax, recomputed per row from q, k and lse
 *     dV_j   = sum_i P_ij dO_i                       (summed over the GQA group)
 *     dS_ij  = P_ij (dO_i . V_j - dO_i . O_i)        times 1 - tanh^2(s_pre / c)
 *                                                    with softcap c, s_pre the
 *                                                    scaled score before capping
 *     dQ_i   = softmax_scale sum_j dS_ij K_j
 *     dK_j   = softmax_scale sum_i dS_ij Q_i         (summed over the GQA group)
 *
 * A row with no admissible key contributes nothing (its dQ row is zero).  The
 * result is deterministic: no atomics, a fixed summation order.
 *
 *  q, k, v, dout   device, [B, Hq, Sq, D], [B, Hkv, Sk, D] x 2, [B, Hq, Sq, D].
 *  out, lse        the forward's output [B, Hq, Sq, D] and lse [B, Hq, Sq]
 *                  (attn_fwd_ex with lse_out), both given or both NULL; when
 *                  NULL the forward is recomputed into the workspace first.
 *  alibi_slopes, row_kv_bounds, softmax_scale, causal, window_left,
 *  window_right, softcap   as in attn_fwd_ex.
 *  dq              device [B, Hq, Sq, D], written fully.
 *  dk, dv          device [B, Hkv, Sk, D], written fully.
 *  dtype           GBATTN_BF16 or GBATTN_F16 (tensor cores, fp32
 *                  accumulation) or GBATTN_F32 (SIMT FFMA) for q, k, v, dout,
 *                  out, dq, dk, dv alike; D 64 or 128.
 *  workspace       device, 256-byte aligned, at least
 *                  attn_bwd_workspace_size(..., dtype, recompute) bytes
 *                  (recompute = 1 when out and lse are NULL); the caller owns
 *                  it; its contents are scratch.
 *  Errors: GBATTN_ERR_INVALID_ARG also for a gradient buffer that overlaps an
 *  input, another gradient or the workspace.
 */
typedef struct {
    const void* q;
    const void* k;
    const void* v;
    const void* out;
    const float* lse;
    const void* dout;
    const float* alibi_slopes;
    const int32_t* row_kv_bounds;
    void* dq;
    void* dk;
    void* dv;
    int B, Hq, Hkv, Sq, Sk, D;
    float softmax_scale;
    int causal;
    int window_left, window_right;
    float softcap;
    int dtype;
    void* workspace;
    size_t workspace_bytes;
    void* stream;
} gbattn_bwd_params;

size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int Sq, int Sk, int D, int dtype, int recompute);
int attn_bwd(const gbattn_bwd_params* p);

/*
 * attn_bwd_phase_times -- profiling form of attn_bwd: runs it `reps` times
 * (1 .. 100000) with CUDA events recorded on p->stream between its launches,
 * waits for each run, and writes the mean milliseconds of its four phases to
 * phase_ms[4]: the forward recompute (0 when out and lse are given), the prep
 * launches (row intervals; for fp32 also Delta = dO . O), the dK / dV launch and
 * the dQ launch.  For bf16 / fp16 the dQ launch runs before the dK / dV launch
 * and also forms Delta and the base-2 lse.  The
 * gradients are written as by attn_bwd.  Synchronous; creates and destroys its
 * own events.
 */
int attn_bwd_phase_times(const gbattn_bwd_params* p, int reps, float* phase_ms);

/* Human-readable text of a status code (static storage). */
const char* gbattn_status_string(int status);

/*
 * gbattn_device_status -- synchronise `stream`, then return the device status
 * word of the current device (0 = no kernel met a timeout or bounds fault;
 * otherwise a bitmask of the wait sites that gave up) and clear it when
 * `clear` is non-zero.  Returns (unsigned)-1 if the synchronisation failed.
 */
unsigned int gbattn_device_status(void* stream, int clear);

/*
 * gbattn_set_wait_timeout_ns -- limit of every bounded wait inside the
 * kernels (default 2e9 ns; the environment variable GBATTN_WAIT_TIMEOUT_MS
 * overrides the default at load time).  Returns the previous value.
 */
uint64_t gbattn_set_wait_timeout_ns(uint64_t ns);

/* Library version, e.g. 100 for 0.1.0. */
int gbattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_H_ */
