/*
 * Test-only entry point of the GB300 attention library (not part of the
 * attention API in fa.h; the pages define no counterpart).
 *
 * fa_selftest_mma runs one 128 x N x 128 bf16 GEMM with fp32 accumulation on
 * the tensor cores through the same TMA boxes, shared-memory descriptors and
 * TMEM paths the attention kernels use, so a layout mistake shows up in a
 * plain GEMM rather than inside attention. A and B are bf16 row-major device
 * arrays (16-byte aligned), D an fp32 row-major [128 x N] device array:
 *   mode 0  D = A B^T,  A [128 x 128], B [128 x 128]   (both K-major)
 *   mode 1  D = A B,    A [128 x 128], B [128 x 128]   (B MN-major)
 *   mode 2  D = A B,    as mode 1 but A read from tensor memory
 *   mode 3  D = A^T B,  A [128 x 128], B [128 x  64]   (both MN-major), N = 64
 *   mode 4  D = A B^T,  A [128 x 128], B [ 64 x 128]   (both K-major),  N = 64
 * Queued on `stream` (a cudaStream_t). Returns 0, -1 (bad mode or null
 * pointer), -3 (misaligned), -4 (device is not compute capability 10.3) or
 * -6 (CUDA error).
 */
#ifndef FA_GB300_SELFTEST_H
#define FA_GB300_SELFTEST_H

#if defined(__GNUC__)
#define FA_SELFTEST_API __attribute__((visibility("default")))
#else
#define FA_SELFTEST_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

FA_SELFTEST_API int fa_selftest_mma(int mode, const void* A, const void* B, float* D, void* stream);

/*
 * Exercises the failure path of the library's bounded barrier waits without a
 * fault (the pages have no counterpart; it backs the device status word that
 * fa_get_device_status() reports). One CTA of two warps holds 32 TMEM columns
 * and waits on two shared-memory barriers that nothing ever completes: warp 0
 * with a limit of `limit_cycles` SM clock cycles, warp 1 with the limit the
 * attention kernels use (about two seconds). Warp 0 gives up first, raises the
 * CTA's abort flag and records the timeout bit; warp 1 must then give up at
 * once. The CTA frees its TMEM and returns; no copy or tensor-core operation is
 * ever issued, so none is in flight when the waits end.
 *   out            device int[2], 4-byte aligned: out[w] = 1 if warp w's wait
 *                  succeeded, 0 if it gave up (both 0 after a correct run)
 *   limit_cycles   1000 .. 1e9 (about 0.5 ms at 2 GHz is 1e6)
 * Queued on `stream`; afterwards fa_get_device_status() reports
 * FA_ERR_DEVICE_TIMEOUT once. Returns 0, -1 (null `out` or limit out of
 * range), -3 (misaligned), -4 (not compute capability 10.3) or -6 (CUDA error).
 */
FA_SELFTEST_API int fa_selftest_wait_timeout(long long limit_cycles, int* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_SELFTEST_H */
