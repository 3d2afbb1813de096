// Standard (materialised) attention, the baseline of the pages' IO comparison
// ("05_flash_attention.py", standard_attention and demo_memory): the whole
// score matrix goes through HBM.
//   scores   S = scale * Q K^T for every (query, key) pair, rounded to bf16 and
//            written to S [BH, n, m_pad] (tensor cores, fp32 accumulation)
//   softmax  per row of S: mask (causal: key k visible from query q iff k <= q;
//            columns past m), P = exp(S - max) / sum, rounded to bf16 and written
//            to P [BH, n, m_pad]; L = max + log(sum) of the row (fp32)
//   pv       O = P V (tensor cores, fp32 accumulation), rounded to bf16
// This is the computation the pages contrast with the tiled method: the same
// formulas, but S and P (2 * n * m bf16 values per head) are written to and read
// back from memory instead of staying on chip. Causal masking does not skip any
// work here: S is computed in full and the mask is applied by the softmax, as
// the pages' standard_attention does. m_pad = m rounded up to a multiple of 64;
// P is 0 in the padding columns, so the PV product may run over them.
#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

__device__ unsigned int g_std_status;

namespace {

constexpr int kChunk = 128 * 128;  // bytes of one 64-column chunk of a 128-row bf16 tile

// ------------------------------------------------------------------ scores
// CTA = one 128-row query tile x kScoreTiles consecutive 128-column key tiles of
// one head. Warp 4 (one lane) loads Q once and the key tiles through a two-slot
// ring, and issues S_t = Q K_t^T into one of two TMEM accumulators; warps 0..3
// (TMEM lane quarters) write S_t out (x scale, bf16, staged TMA stores) while the
// next product runs.
constexpr int kScoreTiles = 4;

template <int D>
struct ScoreCfg {
  static constexpr int KCH = D / 64;
  static constexpr int TILE = KCH * kChunk;       // 128 rows x D bf16
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = TILE;              // two slots
  static constexpr int OFF_EPI = 3 * TILE;        // staging, one area per epilogue warp
  static constexpr int OFF_BAR = OFF_EPI + 4 * kStoreStageBytes;
  // barriers: Q landed, K slot full (2), K slot free (2), accumulator full (2),
  // accumulator free (2, 128 arrivals), every product done (drain)
  static constexpr int B_Q = 0, B_KF = 1, B_KE = 3, B_AF = 5, B_AE = 7, B_DRAIN = 9, NBAR = 10;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
};

template <int D>
__global__ void __launch_bounds__(160, 1)
    std_scores_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmS, int n, int m_pad, float scale) {
  using C = ScoreCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + C::NBAR);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wc{abort_flag, &g_std_status};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.y * 128, bh = blockIdx.z;
  const int col_first = blockIdx.x * kScoreTiles * 128;
  const int ntiles = min(kScoreTiles, (m_pad - col_first + 127) / 128);

  if (threadIdx.x == 0) {
    for (int b = 0; b < C::NBAR; ++b)
      mbar_init(&bar[b], (b == C::B_AE || b == C::B_AE + 1) ? 128 : 1);
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

  if (warp == 4) {
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      mbar_arrive_expect_tx(&bar[C::B_Q], C::TILE);
      for (int c = 0; c < C::KCH; ++c)
        tma_load_3d(smem + C::OFF_Q + c * kChunk, &tmQ, &bar[C::B_Q], c * 64, row0, bh);
      auto load_k = [&](int t) {
        const int s = t & 1;
        mbar_arrive_expect_tx(&bar[C::B_KF + s], C::TILE);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(smem + C::OFF_K + s * C::TILE + c * kChunk, &tmK, &bar[C::B_KF + s], c * 64,
                      col_first + t * 128, bh);
      };
      int loaded = min(2, ntiles), consumed = 0;  // K tiles loaded, K tiles waited for
      for (int t = 0; t < loaded; ++t) load_k(t);
      constexpr uint32_t kIdesc = idesc_bf16_f32(128, 128, false, false);
      const bool q_ok = mbar_wait(&bar[C::B_Q], 0, wc);
      for (int t = 0; q_ok && t < ntiles; ++t) {
        const int s = t & 1;
        if (!mbar_wait(&bar[C::B_KF + s], (t >> 1) & 1, wc)) break;
        consumed = t + 1;
        // accumulator s was last read out for tile t - 2
        if (t >= 2 && !mbar_wait(&bar[C::B_AE + s], ((t - 2) >> 1) & 1, wc)) break;
        tc_fence_after();
        const uint32_t qa = smem_u32(smem + C::OFF_Q), kb = smem_u32(smem + C::OFF_K + s * C::TILE);
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunk + (kk & 3) * 32;
          umma_ss(tmem + 128u * s, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                  kIdesc, kk > 0);
        }
        umma_commit(&bar[C::B_AF + s]);
        umma_commit(&bar[C::B_KE + s]);
        if (t + 2 < ntiles) {
          if (!mbar_wait(&bar[C::B_KE + s], (t >> 1) & 1, wc)) break;  // the product read slot s
          load_k(t + 2);
          loaded = t + 3;
        }
      }
      // Let every product and copy issued land before the CTA can exit (bounded
      // waits that ignore the abort flag; on the normal path they pass at once).
      umma_commit(&bar[C::B_DRAIN]);
      const long long t0 = clock64();
      while (!mbar_try_wait(&bar[C::B_DRAIN], 0) && clock64() - t0 < kWaitMaxCycles / 4) {
      }
      if (!q_ok)
        while (!mbar_try_wait(&bar[C::B_Q], 0) && clock64() - t0 < kWaitMaxCycles / 4) {
        }
      for (int t = consumed; t < loaded; ++t)
        while (!mbar_try_wait(&bar[C::B_KF + (t & 1)], (t >> 1) & 1) &&
               clock64() - t0 < kWaitMaxCycles / 4) {
        }
    }
  } else {
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    uint8_t* stage = smem + C::OFF_EPI + warp * kStoreStageBytes;
    for (int t = 0; t < ntiles; ++t) {
      const int s = t & 1;
      if (!warp_wait(&bar[C::B_AF + s], (t >> 1) & 1, wc)) break;
      tc_fence_after();
      const int col0 = col_first + t * 128;
      tmem_rows_store<128>(lane_base + 128u * s, scale, stage, &tmS, col0, row0 + warp * 32, n, bh,
                           m_pad - col0);
      tc_fence_before();
      mbar_arrive(&bar[C::B_AE + s]);
    }
    if (lane == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ------------------------------------------------------------------ softmax
// One block of 256 threads per row of S: pass 1 keeps a running (max, sum) per
// thread over its 8-column pieces (base 2), merges them across the block; pass 2
// reads the row again (from L2: the block has just read it) and writes P.
constexpr int kSoftmaxThreads = 256;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ void merge_stats(float& mx, float& sum, float omx, float osum) {
  const float nm = fmaxf(mx, omx);
  if (nm == -INFINITY) return;  // both empty
  sum = sum * ex2(mx - nm) + osum * ex2(omx - nm);
  mx = nm;
}

__global__ void __launch_bounds__(kSoftmaxThreads)
    std_softmax_kernel(const __nv_bfloat16* __restrict__ S, __nv_bfloat16* __restrict__ P,
                       float* __restrict__ L, int n, int m, int m_pad, int causal) {
  const int q = blockIdx.x;
  const long long row = (long long)blockIdx.y * n + q;
  const uint4* src = reinterpret_cast<const uint4*>(S + row * m_pad);
  uint4* dst = reinterpret_cast<uint4*>(P + row * m_pad);
  const int lim = causal ? min(m, q + 1) : m;  // columns [0, lim) are visible
  const int pieces = m_pad / 8;
  float mx = -INFINITY, sum = 0.f;
  for (int c = threadIdx.x; c < pieces; c += kSoftmaxThreads) {
    if (8 * c >= lim) break;
    const uint4 v = src[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float x[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = bf16_lo(w[e]) * kLog2e;
      x[2 * e + 1] = bf16_hi(w[e]) * kLog2e;
    }
    float cm = -INFINITY;
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (8 * c + e < lim) cm = fmaxf(cm, x[e]);
    float cs = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (8 * c + e < lim) cs += ex2(x[e] - cm);
    merge_stats(mx, sum, cm, cs);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float omx = __shfl_xor_sync(0xffffffffu, mx, o);
    const float osum = __shfl_xor_sync(0xffffffffu, sum, o);
    merge_stats(mx, sum, omx, osum);
  }
  __shared__ float s_mx[kSoftmaxThreads / 32], s_sum[kSoftmaxThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s_mx[warp] = mx;
    s_sum[warp] = sum;
  }
  __syncthreads();
  mx = s_mx[0];
  sum = s_sum[0];
  for (int w = 1; w < kSoftmaxThreads / 32; ++w) merge_stats(mx, sum, s_mx[w], s_sum[w]);
  const float inv = 1.f / sum;
  if (threadIdx.x == 0) L[row] = (mx + lg2(sum)) * kLn2;
  for (int c = threadIdx.x; c < pieces; c += kSoftmaxThreads) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (8 * c < lim) {
      const uint4 v = src[c];
      const uint32_t r[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k = 8 * c + 2 * e;
        const float p0 = k < lim ? ex2(bf16_lo(r[e]) * kLog2e - mx) * inv : 0.f;
        const float p1 = k + 1 < lim ? ex2(bf16_hi(r[e]) * kLog2e - mx) * inv : 0.f;
        w[e] = pack_bf16(p0, p1);
      }
    }
    dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ------------------------------------------------------------------ pv
// CTA = one 128-row query tile of one head: O = P V over the keys in steps of 64.
// Warp 4 (one lane) streams P [128 x 64] and V [64 x D] through a ring and issues
// the products (A = P K-major, B = V MN-major, fp32 in TMEM); warps 0..3 write O.
template <int D>
struct PvCfg {
  static constexpr int KCH = D / 64;
  static constexpr int P_BYTES = kChunk;           // 128 rows x 64 bf16
  static constexpr int V_CHUNK = 64 * 128;         // 64 rows x 64 bf16
  static constexpr int V_BYTES = KCH * V_CHUNK;
  static constexpr int SLOT = P_BYTES + V_BYTES;
  static constexpr int STAGES = 4;
  static constexpr int OFF_EPI = STAGES * SLOT;
  static constexpr int OFF_BAR = OFF_EPI + 4 * kStoreStageBytes;
  // barriers: slot full, slot free (one per slot), every product done
  static constexpr int B_F = 0, B_E = STAGES, B_DONE = 2 * STAGES, NBAR = 2 * STAGES + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
};

template <int D>
__global__ void __launch_bounds__(160, 1)
    std_pv_kernel(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmO, int n, int m_pad, int d) {
  using C = PvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + C::NBAR);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wc{abort_flag, &g_std_status};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * 128, bh = blockIdx.y;
  const int nk = m_pad / 64;

  if (threadIdx.x == 0) {
    for (int b = 0; b < C::NBAR; ++b) mbar_init(&bar[b], 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    if (lane == 0) {
      tma_prefetch_map(&tmP);
      tma_prefetch_map(&tmV);
      auto load = [&](int t) {
        const int s = t % C::STAGES;
        uint8_t* slot = smem + s * C::SLOT;
        mbar_arrive_expect_tx(&bar[C::B_F + s], C::SLOT);
        tma_load_3d(slot, &tmP, &bar[C::B_F + s], t * 64, row0, bh);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(slot + C::P_BYTES + c * C::V_CHUNK, &tmV, &bar[C::B_F + s], c * 64, t * 64, bh);
      };
      int loaded = min(C::STAGES, nk), consumed = 0;  // chunks loaded, chunks waited for
      for (int t = 0; t < loaded; ++t) load(t);
      constexpr uint32_t kIdesc = idesc_bf16_f32(128, D, false, true);
      for (int t = 0; t < nk; ++t) {
        const int s = t % C::STAGES;
        if (!mbar_wait(&bar[C::B_F + s], (t / C::STAGES) & 1, wc)) break;
        consumed = t + 1;
        tc_fence_after();
        const uint32_t pa = smem_u32(smem + s * C::SLOT);
        const uint32_t vb = pa + C::P_BYTES;
        for (int kk = 0; kk < 4; ++kk)
          umma_ss(tmem, sdesc_sw128(pa + kk * 32, 16, 1024),
                  sdesc_sw128(vb + kk * 2048, C::V_CHUNK, 1024), kIdesc, (t > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bar[C::B_E + s]);
        if (t + C::STAGES < nk) {
          if (!mbar_wait(&bar[C::B_E + s], (t / C::STAGES) & 1, wc)) break;
          load(t + C::STAGES);
          loaded = t + C::STAGES + 1;
        }
      }
      umma_commit(&bar[C::B_DONE]);
      // Let every product and copy issued land before the CTA can exit (bounded
      // waits that ignore the abort flag; on the normal path they pass at once).
      const long long t0 = clock64();
      while (!mbar_try_wait(&bar[C::B_DONE], 0) && clock64() - t0 < kWaitMaxCycles / 4) {
      }
      for (int t = consumed; t < loaded; ++t)
        while (!mbar_try_wait(&bar[C::B_F + t % C::STAGES], (t / C::STAGES) & 1) &&
               clock64() - t0 < kWaitMaxCycles / 4) {
        }
    }
  } else {
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    if (warp_wait(&bar[C::B_DONE], 0, wc)) {
      tc_fence_after();
      tmem_rows_store<D>(lane_base, 1.f, smem + C::OFF_EPI + warp * kStoreStageBytes, &tmO, 0,
                         row0 + warp * 32, n, bh, d);
    }
    if (lane == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

template <int D>
cudaError_t launch_standard_d(const StdArgs& a, cudaStream_t stream) {
  using SC = ScoreCfg<D>;
  using PC = PvCfg<D>;
  CUtensorMap mq, mk, ms_st, mp_ld, mv, mo;
  if (make_bf16_head_map(&mq, a.Q, a.BH, a.n, a.d, 128) != CUDA_SUCCESS ||
      make_bf16_head_map(&mk, a.K, a.BH, a.m, a.d, 128) != CUDA_SUCCESS ||
      make_bf16_store_map(&ms_st, a.S, a.BH, a.n, a.m_pad) != CUDA_SUCCESS ||
      make_bf16_head_map(&mp_ld, a.P, a.BH, a.n, a.m_pad, 128) != CUDA_SUCCESS ||
      make_bf16_head_map(&mv, a.V, a.BH, a.m, a.d, 64) != CUDA_SUCCESS ||
      make_bf16_store_map(&mo, a.O, a.BH, a.n, a.d) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(std_scores_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SC::SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(std_pv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, PC::SMEM);
  if (e != cudaSuccess) return e;
  const dim3 g1((unsigned)ceil_div(a.m_pad, kScoreTiles * 128), (unsigned)ceil_div(a.n, 128),
                (unsigned)a.BH);
  std_scores_kernel<D><<<g1, 160, SC::SMEM, stream>>>(mq, mk, ms_st, a.n, a.m_pad, a.scale);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  std_softmax_kernel<<<dim3((unsigned)a.n, (unsigned)a.BH), kSoftmaxThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(a.S), static_cast<__nv_bfloat16*>(a.P), a.L, a.n, a.m,
      a.m_pad, a.causal);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  std_pv_kernel<D><<<dim3((unsigned)ceil_div(a.n, 128), (unsigned)a.BH), 160, PC::SMEM, stream>>>(
      mp_ld, mv, mo, a.n, a.m_pad, a.d);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_standard(const StdArgs& a, cudaStream_t s) {
  return a.d > 64 ? launch_standard_d<128>(a, s) : launch_standard_d<64>(a, s);
}

cudaError_t standard_read_status(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_std_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_std_status, &zero, sizeof(unsigned int));
}

}  // namespace fa
