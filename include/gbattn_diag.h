/*
 * gbattn_diag.h -- diagnostic entry of libgbattn (no counterpart in the pages;
 * it is a self-test of the library's own tensor-core plumbing).
 *
 * gbattn_diag_umma runs ONE 128 x N x 128 bf16 tile product on the tcgen05
 * tensor cores through exactly the shared-memory layouts, descriptors and
 * TMEM paths the attention kernels use, so a test can compare it with a CPU
 * matrix product and tell a layout error from an attention error:
 *
 *   mode 0:  C = A B^T, A [128][128], B [N][128]   both operands K-major
 *            (the layout of S = Q K^T)
 *   mode 1:  C = A B,   A [128][128], B [128][N]   B MN-major
 *            (the layout of O = P V with P in shared memory)
 *   mode 2:  as mode 1 with A moved into TMEM first (the layout of O = P V
 *            with P in TMEM)
 *
 * a, b: device bf16, row-major, 16-byte aligned; c: device fp32 [128][N].
 * n: 64 or 128.  Runs one CTA on `stream` (a cudaStream_t).  Returns a
 * GBATTN_* status (gbattn.h); a wait that gives up sets bit 16 of the device
 * status word (gbattn_device_status).
 */
#ifndef GBATTN_DIAG_H_
#define GBATTN_DIAG_H_

#ifdef __cplusplus
extern "C" {
#endif

int gbattn_diag_umma(int mode, const void* a, const void* b, float* c, int n, void* stream);

/*
 * gbattn_diag_wait_timeout launches one 32-thread block on `stream` (a
 * cudaStream_t) whose thread 0 waits, through the same bounded mbarrier wait
 * the attention kernels use, on a barrier that nothing ever completes.  After
 * timeout_ns nanoseconds (0 < timeout_ns <= 10 s) the wait gives up, sets bit
 * 16 (the diagnostic site) in the device status word read by
 * gbattn_device_status, and the kernel exits normally: the CUDA context stays
 * usable.  It tests the failure path of the bounded waits without a fault.
 * Returns GBATTN_OK once launched, GBATTN_ERR_INVALID_ARG for a timeout out
 * of range, GBATTN_ERR_CUDA if the launch fails.
 */
int gbattn_diag_wait_timeout(unsigned long long timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_DIAG_H_ */
