// Online softmax statistics of fp32 rows ("05_flash_attention.py",
// online_softmax_stats; "Flash Attention" notes, section 1.1): for each row x of
// a row-major matrix, m = max_j x_j and l = sum_j exp(x_j - m), in one pass that
// keeps a running maximum and a sum taken relative to it, rescaled when the
// maximum moves. m + log l is the row's logsumexp and exp(x_j - m) / l its
// softmax.
//
// Memory bound: every element is read once (16-byte loads when the rows allow).
// Each thread keeps its own (m, l) over a strided share of the row; the shares
// are merged as (m1, l1) + (m2, l2) = (M, l1 exp(m1 - M) + l2 exp(m2 - M)) with
// M = max(m1, m2), first across the lanes of a warp, then across the warps of
// the block. Rows of 32768 or more elements get a 256-thread block each, shorter
// rows a warp each; every thread keeps four 16-byte loads in flight (streaming
// loads: the rows are read once).
#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.44269504088896340736f;

struct Stats {
  float m;  // running maximum (-inf before the first element)
  float l;  // sum of exp(x - m) over the elements seen
};

__device__ __forceinline__ float exp_e(float d) { return ex2(d * kLog2e); }

__device__ __forceinline__ Stats merge(Stats a, Stats b) {
  const float M = fmaxf(a.m, b.m);
  if (M == -INFINITY) return {M, 0.f};
  return {M, a.l * exp_e(a.m - M) + b.l * exp_e(b.m - M)};
}

// Adds elements x0..x3 to s (values may be -inf).
__device__ __forceinline__ void add4(Stats& s, float x0, float x1, float x2, float x3) {
  const float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
  if (mx > s.m) {
    s.l = (s.m == -INFINITY) ? 0.f : s.l * exp_e(s.m - mx);
    s.m = mx;
  }
  if (s.m == -INFINITY) return;  // every element so far is -inf
  s.l += (exp_e(x0 - s.m) + exp_e(x1 - s.m)) + (exp_e(x2 - s.m) + exp_e(x3 - s.m));
}

__device__ __forceinline__ void add1(Stats& s, float x) {
  if (x > s.m) {
    s.l = (s.m == -INFINITY) ? 0.f : s.l * exp_e(s.m - x);
    s.m = x;
  }
  if (s.m != -INFINITY) s.l += exp_e(x - s.m);
}

__device__ __forceinline__ Stats warp_merge(Stats s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Stats t;
    t.m = __shfl_xor_sync(0xffffffffu, s.m, o);
    t.l = __shfl_xor_sync(0xffffffffu, s.l, o);
    s = merge(s, t);
  }
  return s;
}

// The share of row `row` that thread `t` of `nt` threads handles.
__device__ __forceinline__ Stats row_share(const float* __restrict__ row, long long cols, bool vec,
                                           int t, int nt) {
  Stats s{-INFINITY, 0.f};
  if (vec) {  // 16-byte aligned row, cols % 4 == 0
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const long long n4 = cols >> 2;
    long long i = t;
    // four 16-byte loads in flight per thread before any arithmetic
    for (; i + 3LL * nt < n4; i += 4LL * nt) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcs(r4 + i + u * nt);
#pragma unroll
      for (int u = 0; u < 4; ++u) add4(s, v[u].x, v[u].y, v[u].z, v[u].w);
    }
    for (; i < n4; i += nt) {
      const float4 v = __ldcs(r4 + i);
      add4(s, v.x, v.y, v.z, v.w);
    }
  } else {
    for (long long i = t; i < cols; i += nt) add1(s, row[i]);
  }
  return s;
}

__global__ void __launch_bounds__(256) softmax_stats_block_kernel(const float* __restrict__ x,
                                                                  long long rows, long long cols,
                                                                  bool vec, float* __restrict__ m,
                                                                  float* __restrict__ l) {
  __shared__ float pm[8], pl[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    Stats s = warp_merge(row_share(x + r * cols, cols, vec, threadIdx.x, blockDim.x));
    if (lane == 0) {
      pm[warp] = s.m;
      pl[warp] = s.l;
    }
    __syncthreads();
    if (warp == 0) {
      Stats t = lane < 8 ? Stats{pm[lane], pl[lane]} : Stats{-INFINITY, 0.f};
      t = warp_merge(t);
      if (lane == 0) {
        m[r] = t.m;
        l[r] = t.l;
      }
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(256) softmax_stats_warp_kernel(const float* __restrict__ x,
                                                                 long long rows, long long cols,
                                                                 bool vec, float* __restrict__ m,
                                                                 float* __restrict__ l) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    const Stats s = warp_merge(row_share(x + r * cols, cols, vec, lane, 32));
    if (lane == 0) {
      m[r] = s.m;
      l[r] = s.l;
    }
  }
}

}  // namespace

cudaError_t launch_softmax_stats(const float* x, long long rows, long long cols, float* m,
                                 float* l, cudaStream_t stream) {
  const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (cols & 3) == 0;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cols >= 32768) {
    const long long grid = rows < 8LL * sms ? rows : 8LL * sms;  // 8 blocks of 256 per SM
    softmax_stats_block_kernel<<<(unsigned)grid, 256, 0, stream>>>(x, rows, cols, vec, m, l);
  } else {
    const long long blocks = (rows + 7) / 8;
    const long long grid = blocks < 8LL * sms ? blocks : 8LL * sms;
    softmax_stats_warp_kernel<<<(unsigned)grid, 256, 0, stream>>>(x, rows, cols, vec, m, l);
  }
  return cudaGetLastError();
}

}  // namespace fa
