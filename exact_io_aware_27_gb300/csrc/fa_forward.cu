// Forward pass of exact attention: O = softmax(Q K^T * scale) V and the
// natural-log logsumexp L, one 128-row query tile per CTA.
//
// Method: "05_flash_attention.py", flash_attention_forward. For each query
// tile the key/value blocks are visited left to right; per row the kernel
// keeps the running maximum m and the rescaled exponential sum l, forms
// P = exp(S - m_new), rescales the output accumulator by exp(m_old - m_new)
// and adds P V. At the end O = O / l and L = m + log l. Under causal masking
// key blocks wholly to the right of the tile's last query are never visited,
// and the diagonal block masks k > q.
//
// GB300 mapping (one CTA per (query tile, head), 256 threads):
//   warp 0      TMA producer: Q once, then K_j and V_j into a STAGES-deep ring
//   warp 1      MMA issuer: S_j = Q K_j^T (SS form) into TMEM buffer j % 2,
//               then O += P_{j-1} V_{j-1} (TS form, P read from TMEM)
//   warps 4..7  softmax: thread r owns query row r (= TMEM lane r); reads S
//               with tcgen05.ld, masks, updates (m, l) in base 2 (exp2 via
//               ex2.approx), writes P as bf16 into TMEM, rescales the O row
//               when its maximum moved, and runs the epilogue.
// TMEM (512 columns): S0 [0,128) S1 [128,256) P0 [256,320) P1 [320,384)
// O [384, 384+d). Scores, probabilities and the accumulator never leave the SM.
#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

__device__ unsigned int g_fwd_status;

namespace {

constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct FwdCfg {
  static constexpr int BM = 128;                 // query rows per CTA = TMEM lanes
  static constexpr int BN = 128;                 // keys per block
  static constexpr int KCH = D / 64;             // 128-byte column chunks per row
  static constexpr int CHUNK = 128 * 128;        // bytes of one chunk of a 128-row tile
  static constexpr int TILE = KCH * CHUNK;       // bytes of a Q, K or V tile
  static constexpr int STAGES = (D == 128) ? 2 : 4;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE;
  static constexpr int OFF_V = OFF_K + STAGES * TILE;
  static constexpr int OFF_BAR = OFF_V + STAGES * TILE;
  // barrier slots
  static constexpr int B_Q = 0;
  static constexpr int B_KF = 1;
  static constexpr int B_KE = B_KF + STAGES;
  static constexpr int B_VF = B_KE + STAGES;
  static constexpr int B_VE = B_VF + STAGES;
  static constexpr int B_SF = B_VE + STAGES;  // 2
  static constexpr int B_PF = B_SF + 2;       // 2
  static constexpr int B_OD = B_PF + 2;
  static constexpr int B_DRAIN = B_OD + 1;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
  static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_P0 = 256, COL_P1 = 320,
                            COL_O = 384, TMEM_COLS = 512;
  static constexpr int THREADS = 256;
  static_assert(COL_O + D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct FwdParams {
  __nv_bfloat16* O;
  float* L;
  int n, m, BH, causal, num_q_tiles, group;
  float scale_log2;  // scale * log2(e)
};

// Bounded wait that ignores the abort flag: used only to let copies or MMAs
// already in flight land before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitMaxCycles / 4) break;
  }
}

template <int D>
__global__ void __launch_bounds__(256, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + C::NBAR);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wc{abort_flag, &g_fwd_status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Heads a group at a time (their K/V stay in L2 while the group runs); inside
  // a group the heaviest tiles (the last ones, under causal masking) go first.
  int tile, bh;
  grouped_tile(blockIdx.x, p.BH, p.num_q_tiles, p.group, tile, bh);
  if (p.causal) tile = p.num_q_tiles - 1 - tile;
  const int qs = tile * C::BM;
  int nkb = (p.m + C::BN - 1) / C::BN;
  if (p.causal) {
    const int qmax = min(qs + C::BM, p.n) - 1;  // top-left mask: keys k <= q
    nkb = min(nkb, qmax / C::BN + 1);
  }

  if (threadIdx.x == 0) {
    mbar_init(&bar[C::B_Q], 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bar[C::B_KF + s], 1);
      mbar_init(&bar[C::B_KE + s], 1);
      mbar_init(&bar[C::B_VF + s], 1);
      mbar_init(&bar[C::B_VE + s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar[C::B_SF + b], 1);
      mbar_init(&bar[C::B_PF + b], 128);
    }
    mbar_init(&bar[C::B_OD], 1);
    mbar_init(&bar[C::B_DRAIN], 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      mbar_arrive_expect_tx(&bar[C::B_Q], C::TILE);
#pragma unroll
      for (int c = 0; c < C::KCH; ++c)
        tma_load_3d(smem + C::OFF_Q + c * C::CHUNK, &tmQ, &bar[C::B_Q], c * 64, qs, bh);
      int nk = 0, nv = 0;  // loads issued
      for (int j = 0; j < nkb; ++j) {
        const int s = j % C::STAGES;
        const uint32_t ph = (j / C::STAGES) & 1;
        if (j >= C::STAGES && !mbar_wait(&bar[C::B_KE + s], ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(&bar[C::B_KF + s], C::TILE);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(smem + C::OFF_K + s * C::TILE + c * C::CHUNK, &tmK, &bar[C::B_KF + s],
                      c * 64, j * C::BN, bh);
        nk = j + 1;
        if (j >= C::STAGES && !mbar_wait(&bar[C::B_VE + s], ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(&bar[C::B_VF + s], C::TILE);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(smem + C::OFF_V + s * C::TILE + c * C::CHUNK, &tmV, &bar[C::B_VF + s],
                      c * 64, j * C::BN, bh);
        nv = j + 1;
      }
      // Let every copy this thread issued land before the CTA can exit.
      drain_wait(&bar[C::B_Q], 0);
      for (int j = max(0, nk - C::STAGES); j < nk; ++j)
        drain_wait(&bar[C::B_KF + j % C::STAGES], (j / C::STAGES) & 1);
      for (int j = max(0, nv - C::STAGES); j < nv; ++j)
        drain_wait(&bar[C::B_VF + j % C::STAGES], (j / C::STAGES) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (operands stay warp-uniform); elect.sync picks
    // the issuing lane. Descriptors are built once per buffer and advanced by
    // compile-time byte offsets.
    {
      constexpr uint32_t kIdescS = idesc_bf16_f32(128, C::BN, false, false);
      constexpr uint32_t kIdescO = idesc_bf16_f32(128, D, false, true);
      const uint64_t dQ_k = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
      bool ok = warp_wait(&bar[C::B_Q], 0, wc);
      for (int j = 0; ok && j <= nkb; ++j) {
        if (j < nkb) {
          const int s = j % C::STAGES;
          const int sb = j & 1;
          if (!warp_wait(&bar[C::B_KF + s], (j / C::STAGES) & 1, wc)) break;
          // S buffer sb was last read by the softmax of block j - 2.
          if (j >= 2 && !warp_wait(&bar[C::B_PF + sb], ((j - 2) >> 1) & 1, wc)) break;
          tc_fence_after();
          const uint64_t dK_k = sdesc_sw128(smem_u32(smem + C::OFF_K + s * C::TILE), 16, 1024);
          const uint32_t dS = tmem + (sb ? C::COL_S1 : C::COL_S0);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
            umma_ss_w(dS, sdesc_add(dQ_k, off), sdesc_add(dK_k, off), kIdescS, kk > 0);
          }
          umma_commit_w(&bar[C::B_SF + sb]);
          umma_commit_w(&bar[C::B_KE + s]);
        }
        if (j >= 1) {
          const int jj = j - 1;
          const int s = jj % C::STAGES;
          const int pb = jj & 1;
          if (!warp_wait(&bar[C::B_PF + pb], (jj >> 1) & 1, wc)) break;
          if (!warp_wait(&bar[C::B_VF + s], (jj / C::STAGES) & 1, wc)) break;
          tc_fence_after();
          const uint64_t dV_mn =
              sdesc_sw128(smem_u32(smem + C::OFF_V + s * C::TILE), C::CHUNK, 1024);
          const uint32_t aP = tmem + (pb ? C::COL_P1 : C::COL_P0);
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk)
            umma_ts_w(tmem + C::COL_O, aP + kk * 8, sdesc_add(dV_mn, kk * 2048), kIdescO,
                      (jj > 0 || kk > 0) ? 1u : 0u);
          umma_commit_w(&bar[C::B_OD]);
          umma_commit_w(&bar[C::B_VE + s]);
        }
      }
      umma_commit_w(&bar[C::B_DRAIN]);
      drain_wait(&bar[C::B_DRAIN], 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int row = (warp - 4) * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int qg = qs + row;
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY;  // running max of S * scale * log2(e)
    float l_run = 0.f;        // running sum of exp2(S * scale * log2(e) - m_run)
    bool ok = true;
    for (int j = 0; j < nkb; ++j) {
      const int sb = j & 1;
      if (!warp_wait(&bar[C::B_SF + sb], (j >> 1) & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[128];
      const uint32_t scol = lane_base + (sb ? C::COL_S1 : C::COL_S0);
      tmem_ld32(scol + 0, sr);
      tmem_ld32(scol + 32, sr + 32);
      tmem_ld32(scol + 64, sr + 64);
      tmem_ld32(scol + 96, sr + 96);
      tmem_ld_wait();
      reg_fence32(sr);
      reg_fence32(sr + 32);
      reg_fence32(sr + 64);
      reg_fence32(sr + 96);

      // Last visible column of this block for this row (ragged m, causal k <= q).
      const int ks = j * C::BN;
      int lim = p.m - 1 - ks;
      if (p.causal) lim = min(lim, qg - ks);
      if (lim < C::BN - 1) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > lim) sr[c] = __float_as_uint(-INFINITY);
      }
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
        mx0 = fmaxf(mx0, __uint_as_float(sr[c]));
        mx1 = fmaxf(mx1, __uint_as_float(sr[c + 1]));
      }
      const float m_new = fmaxf(m_run, fmaxf(mx0, mx1) * sl2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // no (-inf) - (-inf)
      const float corr = ex2(m_run - m_use);
      float sum0 = 0.f, sum1 = 0.f;
      uint32_t pp[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = ex2(fmaf(__uint_as_float(sr[2 * c]), sl2, -m_use));
        const float p1 = ex2(fmaf(__uint_as_float(sr[2 * c + 1]), sl2, -m_use));
        sum0 += p0;
        sum1 += p1;
        pp[c] = pack_bf16(p0, p1);
      }
      l_run = l_run * corr + (sum0 + sum1);
      m_run = m_new;

      // P buffer sb and the O accumulator are free once P_{j-1} V_{j-1} is done.
      if (j >= 1) {
        if (!warp_wait(&bar[C::B_OD], (j - 1) & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      const uint32_t pcol = lane_base + (sb ? C::COL_P1 : C::COL_P0);
      tmem_st32(pcol, pp);
      tmem_st32(pcol + 32, pp + 32);
      if (j >= 1 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + C::COL_O + 32 * c, o);
          tmem_ld_wait();
          reg_fence32(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
          tmem_st32(lane_base + C::COL_O + 32 * c, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar[C::B_PF + sb]);
    }

    // ------------------------------------------------------------ epilogue
    if (ok && warp_wait(&bar[C::B_OD], (nkb - 1) & 1, wc)) {
      tc_fence_after();
      const float inv_l = 1.f / l_run;
      __nv_bfloat16* orow = p.O + ((size_t)bh * p.n + qg) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_base + C::COL_O + 32 * c, o);
        tmem_ld_wait();
        reg_fence32(o);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
        if (qg < p.n) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
          dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
        }
      }
      if (qg < p.n) p.L[(size_t)bh * p.n + qg] = (m_run + lg2(l_run)) * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_fwd_d(const FwdArgs& a, cudaStream_t stream) {
  using C = FwdCfg<D>;
  CUtensorMap mq, mk, mv;
  if (make_bf16_head_map(&mq, a.Q, a.BH, a.n, D, C::BM) != CUDA_SUCCESS ||
      make_bf16_head_map(&mk, a.K, a.BH, a.m, D, C::BN) != CUDA_SUCCESS ||
      make_bf16_head_map(&mv, a.V, a.BH, a.m, D, C::BN) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  FwdParams p;
  p.O = static_cast<__nv_bfloat16*>(a.O);
  p.L = a.L;
  p.n = a.n;
  p.m = a.m;
  p.BH = a.BH;
  p.causal = a.causal;
  p.num_q_tiles = ceil_div(a.n, C::BM);
  p.group = heads_per_group(a.BH, p.num_q_tiles);
  p.scale_log2 = a.scale * 1.44269504088896340736f;
  cudaError_t e =
      cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)p.num_q_tiles * (unsigned)a.BH;
  fwd_kernel<D><<<grid, C::THREADS, C::SMEM, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward(const FwdArgs& a, cudaStream_t s) {
  return a.d == 128 ? launch_fwd_d<128>(a, s) : launch_fwd_d<64>(a, s);
}

cudaError_t forward_read_status(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_fwd_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_fwd_status, &zero, sizeof(unsigned int));
}

}  // namespace fa
