// Test-only unit GEMM through the same TMA boxes, shared-memory descriptors,
// instruction descriptors and TMEM paths the attention kernels use. Each mode
// is one 128 x N x 128 product (8 MMAs of K = 16) in one CTA:
//   0  D[128x128] = A (K-major)  * B^T, B [128 x 128] K-major      (S = Q K^T)
//   1  D[128x128] = A (K-major)  * B,   B [128 x 128] MN-major     (dK = dS^T Q)
//   2  D[128x128] = A (in TMEM)  * B,   B [128 x 128] MN-major     (O += P V)
//   3  D[128x 64] = A^T          * B,   A [128 x 128] given K x M (MN-major),
//                                       B [128 x  64] MN-major     (dQ^T = K^T dS^T)
//   4  D[128x 64] = A (K-major)  * B^T, B [ 64 x 128] K-major      (S^T = K Q^T)
// A and B are bf16 row-major device arrays, D is fp32 row-major [128 x N].
#include "fa_internal.h"
#include "fa_selftest.h"
#include "sm103.cuh"

namespace fa {

__device__ unsigned int g_selftest_status;

namespace {

constexpr int kChunk = 128 * 128;

__global__ void __launch_bounds__(128, 1)
    selftest_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __nv_bfloat16* __restrict__ A_raw, float* __restrict__ Dout, int mode) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;                 // 32 KB
  uint8_t* sB = smem + 2 * kChunk;    // 32 KB
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 4 * kChunk);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 2);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wc{abort_flag, &g_selftest_status};
  const int t = threadIdx.x, warp = t >> 5;
  const int N = (mode >= 3) ? 64 : 128;
  const int b_rows = (mode == 4) ? 64 : 128;

  if (t == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  constexpr uint32_t kColA = 128;

  if (mode == 2) {  // A row t -> TMEM lane t, bf16 pairs packed per column
    uint32_t r[64];
    const uint32_t* src = reinterpret_cast<const uint32_t*>(A_raw + (size_t)t * 128);
#pragma unroll
    for (int c = 0; c < 64; ++c) r[c] = src[c];
    tmem_st32(lane_base + kColA, r);
    tmem_st32(lane_base + kColA + 32, r + 32);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (t == 0) {
    const int a_bytes = (mode == 2) ? 0 : 2 * kChunk;
    const int b_bytes = (mode >= 3) ? kChunk : 2 * kChunk;
    mbar_arrive_expect_tx(&bar[0], a_bytes + b_bytes);
    if (mode != 2) {
      tma_load_3d(sA, &tmA, &bar[0], 0, 0, 0);
      tma_load_3d(sA + kChunk, &tmA, &bar[0], 64, 0, 0);
    }
    if (mode == 3) {
      tma_load_3d(sB, &tmB, &bar[0], 0, 0, 0);
    } else if (mode == 4) {
      tma_load_3d(sB, &tmB, &bar[0], 0, 0, 0);                // 64 rows x 128 B
      tma_load_3d(sB + b_rows * 128, &tmB, &bar[0], 64, 0, 0);
    } else {
      tma_load_3d(sB, &tmB, &bar[0], 0, 0, 0);
      tma_load_3d(sB + kChunk, &tmB, &bar[0], 64, 0, 0);
    }
    if (mbar_wait(&bar[0], 0, wc)) {
      tc_fence_after();
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
#pragma unroll 1
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t kmaj = (kk >> 2) * kChunk + (kk & 3) * 32;
        const uint32_t acc = kk > 0;
        switch (mode) {
          case 0:
            umma_ss(tmem, sdesc_sw128(a0 + kmaj, 16, 1024), sdesc_sw128(b0 + kmaj, 16, 1024),
                    idesc_bf16_f32(128, 128, false, false), acc);
            break;
          case 1:
            umma_ss(tmem, sdesc_sw128(a0 + kmaj, 16, 1024),
                    sdesc_sw128(b0 + kk * 2048, kChunk, 1024),
                    idesc_bf16_f32(128, 128, false, true), acc);
            break;
          case 2:
            umma_ts(tmem, tmem + kColA + kk * 8, sdesc_sw128(b0 + kk * 2048, kChunk, 1024),
                    idesc_bf16_f32(128, 128, false, true), acc);
            break;
          case 3:
            umma_ss(tmem, sdesc_sw128(a0 + kk * 2048, kChunk, 1024),
                    sdesc_sw128(b0 + kk * 2048, kChunk, 1024),
                    idesc_bf16_f32(128, 64, true, true), acc);
            break;
          default:
            umma_ss(tmem, sdesc_sw128(a0 + kmaj, 16, 1024),
                    sdesc_sw128(b0 + (kk >> 2) * (b_rows * 128) + (kk & 3) * 32, 16, 1024),
                    idesc_bf16_f32(128, 64, false, false), acc);
            break;
        }
      }
    }
    umma_commit(&bar[1]);
  }
  if (mbar_wait(&bar[1], 0, wc)) {
    tc_fence_after();
    for (int c = 0; c < N; c += 32) {
      uint32_t r[32];
      tmem_ld32(lane_base + c, r);
      tmem_ld_wait();
      reg_fence32(r);
#pragma unroll
      for (int e = 0; e < 32; ++e) Dout[(size_t)t * N + c + e] = __uint_as_float(r[e]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// The failure path of the bounded waits, exercised without a fault: nothing ever
// arrives on either barrier. Warp 0 waits on the first with `limit_cycles`, runs
// out, raises the CTA abort flag and records kDeviceTimeoutBit; warp 1 waits on
// the second with the kernels' own limit (about two seconds) and must give up as
// soon as it sees the abort flag. The CTA holds TMEM during the waits (the
// attention kernels' situation) and frees it on the way out. No copy and no MMA is
// ever issued, so nothing is in flight when the waits give up. out[w] = 1 if warp
// w's wait succeeded, 0 if it gave up.
__global__ void __launch_bounds__(64, 1)
    selftest_timeout_kernel(long long limit_cycles, int* __restrict__ out) {
  __shared__ uint64_t bar[2];
  __shared__ uint32_t tmem_slot;
  __shared__ uint32_t abort_word;
  const WaitCtx wc{&abort_word, &g_selftest_status};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    abort_word = 0u;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const bool ok = warp == 0 ? warp_wait(&bar[0], 0, wc, limit_cycles) : warp_wait(&bar[1], 0, wc);
  if (lane == 0) out[warp] = ok ? 1 : 0;
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
  if (threadIdx.x == 0) {
    mbar_inval(&bar[0]);
    mbar_inval(&bar[1]);
  }
}

}  // namespace

cudaError_t selftest_read_status(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_selftest_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_selftest_status, &zero, sizeof(unsigned int));
}

cudaError_t launch_selftest_mma(int mode, const void* A, const void* B, float* D,
                                cudaStream_t s) {
  CUtensorMap ma, mb;
  const int a_rows = 128, a_cols = 128;
  const int b_rows = (mode == 4) ? 64 : 128, b_cols = (mode == 3) ? 64 : 128;
  if (make_bf16_head_map(&ma, A, 1, a_rows, a_cols, a_rows) != CUDA_SUCCESS ||
      make_bf16_head_map(&mb, B, 1, b_rows, b_cols, b_rows) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const int smem = 4 * kChunk + 64 + 1024;
  cudaError_t e =
      cudaFuncSetAttribute(selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  selftest_kernel<<<1, 128, smem, s>>>(ma, mb, static_cast<const __nv_bfloat16*>(A), D, mode);
  return cudaGetLastError();
}

}  // namespace fa

extern "C" int fa_selftest_mma(int mode, const void* A, const void* B, float* D, void* stream) {
  if (mode < 0 || mode > 4 || !A || !B || !D) return -1;
  if ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15)) return -3;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return -6;
  if (major != 10 || minor != 3) return -4;
  return fa::launch_selftest_mma(mode, A, B, D, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? 0
             : -6;
}

extern "C" int fa_selftest_wait_timeout(long long limit_cycles, int* out, void* stream) {
  if (!out || limit_cycles < 1000 || limit_cycles > fa::kWaitMaxCycles / 4) return -1;
  if (reinterpret_cast<uintptr_t>(out) & 3) return -3;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return -6;
  if (major != 10 || minor != 3) return -4;
  fa::selftest_timeout_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(limit_cycles, out);
  return cudaGetLastError() == cudaSuccess ? 0 : -6;
}
