// Backward pass of exact attention, FlashAttention-2 recompute form
// ("05_flash_attention.py", flash_attention_backward):
//   D = rowsum(dO o O); for each key block (outer) and query block (inner,
//   skipping blocks wholly above the diagonal under causal masking):
//   P = exp(S - L), dV += P^T dO, dP = dO V^T, dS = P o (dP - D),
//   dQ += dS K * scale, dK += dS^T Q * scale.
//
// Three kernels on one stream:
//   preprocess  D, L * log2(e) (+inf past n) and a zeroed fp32 dQ accumulator
//               in the workspace; memory bound.
//   dkdv        one CTA per (key block of 128, head). The key block's K and V
//               tiles stay in shared memory; dK and dV accumulate in TMEM over
//               the query loop and are written once. The transposed products
//               are formed directly so the key index is the TMEM lane:
//                 S^T  = K Q_i^T        dP^T = V dO_i^T         (SS MMAs)
//                 dV  += P^T dO_i       (TS MMA, P^T written to TMEM as bf16)
//                 dK  += dS^T Q_i       (SS MMA, dS^T staged in shared memory)
//               and this block's share of dQ_i,
//                 d = 128: dQ_i^T = K^T dS^T  (M = d = 128 lanes, N = 64 queries)
//                 d =  64: dQ_i   = dS K      (M = 128 query lanes, N = d = 64)
//               is added into the fp32 accumulator with global atomics.
//   dq          dQ = bf16(accumulator * scale).
//
// dkdv roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer, warps 4..7
// compute P^T and dS^T (thread = key row), warps 8..11 drain dQ from TMEM and
// add it to global memory.
#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

__device__ unsigned int g_bwd_status;

namespace {

constexpr float kLog2e = 1.44269504088896340736f;

template <int D>
struct BwdCfg {
  static constexpr int BN = 128;                    // keys per CTA = TMEM lanes
  static constexpr int BQ = (D == 128) ? 64 : 128;  // queries per inner step
  static constexpr int KCH = D / 64;
  static constexpr int KV_CHUNK = 128 * 128;        // one 64-column chunk of K or V
  static constexpr int KV_TILE = KCH * KV_CHUNK;
  static constexpr int Q_CHUNK = BQ * 128;          // one 64-column chunk of Q_i or dO_i
  static constexpr int Q_TILE = KCH * Q_CHUNK;
  static constexpr int DS_CHUNK = BN * 128;         // 64 queries x 128 keys of dS^T (bf16)
  static constexpr int DS_TILE = (BQ / 64) * DS_CHUNK;
  static constexpr int STAGES = 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_TILE;
  static constexpr int OFF_Q = OFF_V + KV_TILE;
  static constexpr int OFF_DO = OFF_Q + STAGES * Q_TILE;
  static constexpr int OFF_DS = OFF_DO + STAGES * Q_TILE;
  static constexpr int OFF_LSE = OFF_DS + DS_TILE;          // [STAGES][BQ] fp32
  static constexpr int OFF_DD = OFF_LSE + STAGES * BQ * 4;  // [STAGES][BQ] fp32
  static constexpr int OFF_BAR = OFF_DD + STAGES * BQ * 4;
  // barrier slots
  static constexpr int B_KV = 0;
  static constexpr int B_QF = 1;   // + stage
  static constexpr int B_QE = 3;   // + stage
  static constexpr int B_OF = 5;   // + stage
  static constexpr int B_OE = 7;   // + stage
  static constexpr int B_SF = 9;
  static constexpr int B_SFREE = 10;
  static constexpr int B_PF = 11;
  static constexpr int B_DVD = 12;
  static constexpr int B_DSF = 13;
  static constexpr int B_DSD = 14;
  static constexpr int B_DQE = 15;
  static constexpr int B_ACC = 16;
  static constexpr int B_DRAIN = 17;
  static constexpr int NBAR = 18;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
  // TMEM columns
  static constexpr uint32_t COL_S = 0;
  static constexpr uint32_t COL_DP = BQ;
  static constexpr uint32_t COL_P = 2 * BQ;
  static constexpr uint32_t COL_DV = 2 * BQ + BQ / 2;
  static constexpr uint32_t COL_DK = COL_DV + D;
  static constexpr uint32_t COL_DQ = COL_DK + D;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int THREADS = 384;
  static_assert(COL_DQ + 64 <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct BwdParams {
  __nv_bfloat16 *dK, *dV;
  float* ws_dQ;
  int n, m, n_pad, BH, causal;
  float scale, scale_log2;
};

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitMaxCycles / 4) break;
  }
}

template <int D>
__global__ void __launch_bounds__(384, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const __grid_constant__ CUtensorMap tmL2, const __grid_constant__ CUtensorMap tmD,
                const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + C::NBAR);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wc{abort_flag, &g_bwd_status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ktile = blockIdx.x / p.BH;  // key blocks near 0 carry the most work
  const int bh = blockIdx.x % p.BH;
  const int ks = ktile * C::BN;
  const int nqb = (p.n + C::BQ - 1) / C::BQ;
  const int i_start = p.causal ? ks / C::BQ : 0;  // first block with a query q >= ks
  const int nq = max(0, nqb - i_start);

  if (threadIdx.x == 0) {
    mbar_init(&bar[C::B_KV], 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bar[C::B_QF + s], 1);
      mbar_init(&bar[C::B_QE + s], 1);
      mbar_init(&bar[C::B_OF + s], 1);
      mbar_init(&bar[C::B_OE + s], 1);
    }
    mbar_init(&bar[C::B_SF], 1);
    mbar_init(&bar[C::B_SFREE], 128);
    mbar_init(&bar[C::B_PF], 128);
    mbar_init(&bar[C::B_DVD], 1);
    mbar_init(&bar[C::B_DSF], 128);
    mbar_init(&bar[C::B_DSD], 1);
    mbar_init(&bar[C::B_DQE], 128);
    mbar_init(&bar[C::B_ACC], 1);
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
    if (lane == 0 && nq > 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      tma_prefetch_map(&tmdO);
      mbar_arrive_expect_tx(&bar[C::B_KV], 2 * C::KV_TILE);
#pragma unroll
      for (int c = 0; c < C::KCH; ++c) {
        tma_load_3d(smem + C::OFF_K + c * C::KV_CHUNK, &tmK, &bar[C::B_KV], c * 64, ks, bh);
        tma_load_3d(smem + C::OFF_V + c * C::KV_CHUNK, &tmV, &bar[C::B_KV], c * 64, ks, bh);
      }
      int nqi = 0, noi = 0;
      for (int i = 0; i < nq; ++i) {
        const int s = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        const int q0 = (i_start + i) * C::BQ;
        if (i >= C::STAGES && !mbar_wait(&bar[C::B_QE + s], ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(&bar[C::B_QF + s], C::Q_TILE + 2 * C::BQ * 4);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(smem + C::OFF_Q + s * C::Q_TILE + c * C::Q_CHUNK, &tmQ, &bar[C::B_QF + s],
                      c * 64, q0, bh);
        tma_load_2d(smem + C::OFF_LSE + s * C::BQ * 4, &tmL2, &bar[C::B_QF + s], q0, bh);
        tma_load_2d(smem + C::OFF_DD + s * C::BQ * 4, &tmD, &bar[C::B_QF + s], q0, bh);
        nqi = i + 1;
        if (i >= C::STAGES && !mbar_wait(&bar[C::B_OE + s], ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(&bar[C::B_OF + s], C::Q_TILE);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(smem + C::OFF_DO + s * C::Q_TILE + c * C::Q_CHUNK, &tmdO,
                      &bar[C::B_OF + s], c * 64, q0, bh);
        noi = i + 1;
      }
      drain_wait(&bar[C::B_KV], 0);
      for (int i = max(0, nqi - C::STAGES); i < nqi; ++i)
        drain_wait(&bar[C::B_QF + (i & 1)], (i >> 1) & 1);
      for (int i = max(0, noi - C::STAGES); i < noi; ++i)
        drain_wait(&bar[C::B_OF + (i & 1)], (i >> 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nq > 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(128, C::BQ, false, false);
      constexpr uint32_t kIdescDV = idesc_bf16_f32(128, D, false, true);
      constexpr uint32_t kIdescDK = idesc_bf16_f32(128, D, false, true);
      constexpr uint32_t kIdescDQ = (D == 128) ? idesc_bf16_f32(128, C::BQ, true, true)
                                               : idesc_bf16_f32(128, D, true, true);
      const uint32_t sK = smem_u32(smem + C::OFF_K);
      const uint32_t sV = smem_u32(smem + C::OFF_V);
      const uint32_t sDS = smem_u32(smem + C::OFF_DS);
      bool ok = mbar_wait(&bar[C::B_KV], 0, wc);
      for (int i = 0; ok && i <= nq; ++i) {
        if (i < nq) {
          // S^T = K Q_i^T and dP^T = V dO_i^T
          const int s = i & 1;
          const uint32_t ph = (i >> 1) & 1;
          if (!mbar_wait(&bar[C::B_QF + s], ph, wc)) break;
          if (!mbar_wait(&bar[C::B_OF + s], ph, wc)) break;
          if (i >= 1 && !mbar_wait(&bar[C::B_SFREE], (i - 1) & 1, wc)) break;
          tc_fence_after();
          const uint32_t sQ = smem_u32(smem + C::OFF_Q + s * C::Q_TILE);
          const uint32_t sO = smem_u32(smem + C::OFF_DO + s * C::Q_TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32;
            const uint32_t kb = (kk >> 2) * C::Q_CHUNK + (kk & 3) * 32;
            umma_ss(tmem + C::COL_S, sdesc_sw128(sK + ka, 16, 1024),
                    sdesc_sw128(sQ + kb, 16, 1024), kIdescS, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32;
            const uint32_t kb = (kk >> 2) * C::Q_CHUNK + (kk & 3) * 32;
            umma_ss(tmem + C::COL_DP, sdesc_sw128(sV + ka, 16, 1024),
                    sdesc_sw128(sO + kb, 16, 1024), kIdescS, kk > 0);
          }
          umma_commit(&bar[C::B_SF]);
        }
        if (i >= 1) {
          // dK += dS^T Q_{i-1} and this block's share of dQ_{i-1}
          const int ii = i - 1;
          const int s = ii & 1;
          if (!mbar_wait(&bar[C::B_DSF], ii & 1, wc)) break;
          if (ii >= 1 && !mbar_wait(&bar[C::B_DQE], (ii - 1) & 1, wc)) break;
          tc_fence_after();
          const uint32_t sQ = smem_u32(smem + C::OFF_Q + s * C::Q_TILE);
#pragma unroll
          for (int kk = 0; kk < C::BQ / 16; ++kk) {
            const uint32_t ka = (kk >> 2) * C::DS_CHUNK + (kk & 3) * 32;
            umma_ss(tmem + C::COL_DK, sdesc_sw128(sDS + ka, 16, 1024),
                    sdesc_sw128(sQ + kk * 2048, C::Q_CHUNK, 1024), kIdescDK,
                    (ii > 0 || kk > 0) ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk) {
            if (D == 128) {
              umma_ss(tmem + C::COL_DQ, sdesc_sw128(sK + kk * 2048, C::KV_CHUNK, 1024),
                      sdesc_sw128(sDS + kk * 2048, C::DS_CHUNK, 1024), kIdescDQ, kk > 0);
            } else {
              umma_ss(tmem + C::COL_DQ, sdesc_sw128(sDS + kk * 2048, C::DS_CHUNK, 1024),
                      sdesc_sw128(sK + kk * 2048, C::KV_CHUNK, 1024), kIdescDQ, kk > 0);
            }
          }
          umma_commit(&bar[C::B_DSD]);
          umma_commit(&bar[C::B_QE + s]);
        }
        if (i < nq) {
          // dV += P^T dO_i
          const int s = i & 1;
          if (!mbar_wait(&bar[C::B_PF], i & 1, wc)) break;
          tc_fence_after();
          const uint32_t sO = smem_u32(smem + C::OFF_DO + s * C::Q_TILE);
#pragma unroll
          for (int kk = 0; kk < C::BQ / 16; ++kk) {
            umma_ts(tmem + C::COL_DV, tmem + C::COL_P + kk * 8,
                    sdesc_sw128(sO + kk * 2048, C::Q_CHUNK, 1024), kIdescDV,
                    (i > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&bar[C::B_DVD]);
          umma_commit(&bar[C::B_OE + s]);
        }
      }
      umma_commit(&bar[C::B_ACC]);
      umma_commit(&bar[C::B_DRAIN]);
      drain_wait(&bar[C::B_DRAIN], 0);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ P^T, dS^T
    const int krow = (warp - 4) * 32 + lane;
    const int kg = ks + krow;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float sl2 = p.scale_log2;
    const bool key_ok = kg < p.m;
    const uint32_t sDS = smem_u32(smem + C::OFF_DS);
    bool ok = true;
    for (int i = 0; i < nq; ++i) {
      const int s = i & 1;
      const int q0 = (i_start + i) * C::BQ;
      if (!mbar_wait(&bar[C::B_QF + s], (i >> 1) & 1, wc)) { ok = false; break; }
      if (!mbar_wait(&bar[C::B_SF], i & 1, wc)) { ok = false; break; }
      tc_fence_after();
      const float* lse = reinterpret_cast<const float*>(smem + C::OFF_LSE + s * C::BQ * 4);
      const float* dd = reinterpret_cast<const float*>(smem + C::OFF_DD + s * C::BQ * 4);
      // Causal: key kg is hidden from query q when kg > q.
      const bool need_mask = p.causal && (ks + C::BN - 1 > q0);
      const int qlim = kg - q0;  // columns c < qlim are hidden under causal masking

      uint32_t pp[C::BQ / 2];
#pragma unroll
      for (int c = 0; c < C::BQ / 32; ++c) {
        uint32_t sr[32];
        tmem_ld32(lane_base + C::COL_S + 32 * c, sr);
        tmem_ld_wait();
        reg_fence32(sr);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int q = 32 * c + e;
          float p0 = ex2(fmaf(__uint_as_float(sr[e]), sl2, -lse[q]));
          float p1 = ex2(fmaf(__uint_as_float(sr[e + 1]), sl2, -lse[q + 1]));
          if (need_mask) {
            if (q < qlim) p0 = 0.f;
            if (q + 1 < qlim) p1 = 0.f;
          }
          if (!key_ok) p0 = p1 = 0.f;
          pp[16 * c + e / 2] = pack_bf16(p0, p1);
        }
      }
      if (i >= 1) {  // P^T columns are free once dV_{i-1} is done
        if (!mbar_wait(&bar[C::B_DVD], (i - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
      }
#pragma unroll
      for (int c = 0; c < C::BQ / 32; ++c) tmem_st16(lane_base + C::COL_P + 16 * c, pp + 16 * c);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar[C::B_PF]);

      if (i >= 1) {  // dS^T staging is free once dK_{i-1}, dQ_{i-1} are done
        if (!mbar_wait(&bar[C::B_DSD], (i - 1) & 1, wc)) { ok = false; break; }
      }
#pragma unroll
      for (int c = 0; c < C::BQ / 32; ++c) {
        uint32_t dr[32];
        tmem_ld32(lane_base + C::COL_DP + 32 * c, dr);
        tmem_ld_wait();
        reg_fence32(dr);
        if (c == C::BQ / 32 - 1) {  // S^T and dP^T fully read
          tc_fence_before();
          mbar_arrive(&bar[C::B_SFREE]);
        }
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int q = 32 * c + e;
          const uint32_t pv = pp[16 * c + e / 2];
          const float ds0 = bf16_lo(pv) * (__uint_as_float(dr[e]) - dd[q]);
          const float ds1 = bf16_hi(pv) * (__uint_as_float(dr[e + 1]) - dd[q + 1]);
          w[e / 2] = pack_bf16(ds0, ds1);
        }
        // Row krow of dS^T, queries [32c, 32c+32): four 16-byte chunks in the
        // 128-byte-swizzled layout (chunk index XOR row % 8).
        const uint32_t rowbase = sDS + (c >> 1) * C::DS_CHUNK + krow * 128;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t chunk = (uint32_t)(((c & 1) * 4 + t) ^ (krow & 7));
          st_shared_v4(rowbase + chunk * 16, w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bar[C::B_DSF]);
    }

    // ------------------------------------------------------------ dK, dV out
    if (ok) {
      __nv_bfloat16* dv_row = p.dV + ((size_t)bh * p.m + kg) * D;
      __nv_bfloat16* dk_row = p.dK + ((size_t)bh * p.m + kg) * D;
      if (nq == 0) {
        if (key_ok) {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) {
            reinterpret_cast<uint4*>(dv_row)[c] = z;
            reinterpret_cast<uint4*>(dk_row)[c] = z;
          }
        }
      } else if (mbar_wait(&bar[C::B_ACC], 0, wc)) {
        tc_fence_after();
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const uint32_t col = which == 0 ? C::COL_DV : C::COL_DK;
          const float mul = which == 0 ? 1.f : p.scale;
          __nv_bfloat16* dst_row = which == 0 ? dv_row : dk_row;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_base + col + 32 * c, o);
            tmem_ld_wait();
            reg_fence32(o);
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w[e] = pack_bf16(__uint_as_float(o[2 * e]) * mul, __uint_as_float(o[2 * e + 1]) * mul);
            if (key_ok) {
              uint4* dst = reinterpret_cast<uint4*>(dst_row + 32 * c);
              dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
              dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
              dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
              dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
            }
          }
        }
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ drain
    const int t = (warp - 8) * 32 + lane;  // TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    for (int i = 0; i < nq; ++i) {
      const int q0 = (i_start + i) * C::BQ;
      if (!mbar_wait(&bar[C::B_DSD], i & 1, wc)) break;
      tc_fence_after();
      uint32_t v[64];
      tmem_ld32(lane_base + C::COL_DQ, v);
      tmem_ld32(lane_base + C::COL_DQ + 32, v + 32);
      tmem_ld_wait();
      reg_fence32(v);
      reg_fence32(v + 32);
      tc_fence_before();
      mbar_arrive(&bar[C::B_DQE]);
      if (D == 128) {
        // lane t = feature index, column = query
        float* base = p.ws_dQ + ((size_t)bh * p.n_pad + q0) * D + t;
#pragma unroll
        for (int q = 0; q < 64; ++q) atomicAdd(base + (size_t)q * D, __uint_as_float(v[q]));
      } else {
        // lane t = query, column = feature index
        float4* base = reinterpret_cast<float4*>(p.ws_dQ + ((size_t)bh * p.n_pad + q0 + t) * D);
#pragma unroll
        for (int c = 0; c < 16; ++c)
          atomicAdd(base + c, make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                                          __uint_as_float(v[4 * c + 2]),
                                          __uint_as_float(v[4 * c + 3])));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ preprocess
// One warp per workspace row (head bh, query q < n_pad): D = sum_c dO*O,
// L2 = L * log2(e), and the dQ accumulator row cleared. Rows q >= n get
// D = 0 and L2 = +inf so that recomputed probabilities there are exactly 0.
template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const __nv_bfloat16* __restrict__ O,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         const float* __restrict__ L,
                                                         float* __restrict__ ws_D,
                                                         float* __restrict__ ws_L2,
                                                         float* __restrict__ ws_dQ, int n,
                                                         int n_pad, long long rows) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    const long long bh = r / n_pad;
    const int q = (int)(r - bh * n_pad);
    float acc = 0.f;
    if (q < n) {
      const size_t off = ((size_t)bh * n + q) * D;
      if (D == 128) {
        const uint2 a = reinterpret_cast<const uint2*>(O + off)[lane];
        const uint2 b = reinterpret_cast<const uint2*>(dO + off)[lane];
        acc = bf16_lo(a.x) * bf16_lo(b.x) + bf16_hi(a.x) * bf16_hi(b.x) +
              bf16_lo(a.y) * bf16_lo(b.y) + bf16_hi(a.y) * bf16_hi(b.y);
      } else {
        const uint32_t a = reinterpret_cast<const uint32_t*>(O + off)[lane];
        const uint32_t b = reinterpret_cast<const uint32_t*>(dO + off)[lane];
        acc = bf16_lo(a) * bf16_lo(b) + bf16_hi(a) * bf16_hi(b);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    }
    if (lane == 0) {
      ws_D[r] = acc;
      ws_L2[r] = (q < n) ? L[(size_t)bh * n + q] * kLog2e : INFINITY;
    }
    float* drow = ws_dQ + (size_t)r * D;
    if (D == 128) {
      reinterpret_cast<float4*>(drow)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      reinterpret_cast<float2*>(drow)[lane] = make_float2(0.f, 0.f);
    }
  }
}

// ------------------------------------------------------------------ dQ convert
// dQ[bh, q, :] = bf16(accumulator[bh, q, :] * scale) for q < n; 8 values per thread.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ ws_dQ,
                                                         __nv_bfloat16* __restrict__ dQ, int n,
                                                         int n_pad, int d, float scale,
                                                         long long groups) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const int gpr = d / 8;  // groups of 8 per row
  for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += stride) {
    const long long row = g / gpr;  // over BH * n
    const int c8 = (int)(g - row * gpr);
    const long long bh = row / n;
    const int q = (int)(row - bh * n);
    const float4* src =
        reinterpret_cast<const float4*>(ws_dQ + ((size_t)bh * n_pad + q) * d) + 2 * c8;
    const float4 a = src[0], b = src[1];
    reinterpret_cast<uint4*>(dQ + (size_t)row * d)[c8] =
        make_uint4(pack_bf16(a.x * scale, a.y * scale), pack_bf16(a.z * scale, a.w * scale),
                   pack_bf16(b.x * scale, b.y * scale), pack_bf16(b.z * scale, b.w * scale));
  }
}

template <int D>
cudaError_t launch_dkdv_d(const BwdArgs& a, cudaStream_t stream) {
  using C = BwdCfg<D>;
  CUtensorMap mq, mk, mv, mdo, ml2, md;
  if (make_bf16_head_map(&mq, a.Q, a.BH, a.n, D, C::BQ) != CUDA_SUCCESS ||
      make_bf16_head_map(&mk, a.K, a.BH, a.m, D, C::BN) != CUDA_SUCCESS ||
      make_bf16_head_map(&mv, a.V, a.BH, a.m, D, C::BN) != CUDA_SUCCESS ||
      make_bf16_head_map(&mdo, a.dO, a.BH, a.n, D, C::BQ) != CUDA_SUCCESS ||
      make_f32_row_map(&ml2, a.ws_L2, a.BH, a.n_pad, C::BQ) != CUDA_SUCCESS ||
      make_f32_row_map(&md, a.ws_D, a.BH, a.n_pad, C::BQ) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  BwdParams p;
  p.dK = static_cast<__nv_bfloat16*>(a.dK);
  p.dV = static_cast<__nv_bfloat16*>(a.dV);
  p.ws_dQ = a.ws_dQ;
  p.n = a.n;
  p.m = a.m;
  p.n_pad = a.n_pad;
  p.BH = a.BH;
  p.causal = a.causal;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  cudaError_t e =
      cudaFuncSetAttribute(dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)ceil_div(a.m, C::BN) * (unsigned)a.BH;
  dkdv_kernel<D><<<grid, C::THREADS, C::SMEM, stream>>>(mq, mk, mv, mdo, ml2, md, p);
  return cudaGetLastError();
}

int grid_for(long long work_items, int per_block) {
  long long b = (work_items + per_block - 1) / per_block;
  const long long cap = 152LL * 16;  // a few waves over the SMs; grid-stride beyond
  if (b > cap) b = cap;
  return (int)(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t s) {
  const long long rows = (long long)a.BH * a.n_pad;
  const int grid = grid_for(rows, 8);
  if (a.d == 128)
    preprocess_kernel<128><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(a.O), static_cast<const __nv_bfloat16*>(a.dO), a.L,
        a.ws_D, a.ws_L2, a.ws_dQ, a.n, a.n_pad, rows);
  else
    preprocess_kernel<64><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(a.O), static_cast<const __nv_bfloat16*>(a.dO), a.L,
        a.ws_D, a.ws_L2, a.ws_dQ, a.n, a.n_pad, rows);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const BwdArgs& a, cudaStream_t s) {
  return a.d == 128 ? launch_dkdv_d<128>(a, s) : launch_dkdv_d<64>(a, s);
}

cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t s) {
  const long long groups = (long long)a.BH * a.n * (a.d / 8);
  dq_convert_kernel<<<grid_for(groups, 256), 256, 0, s>>>(
      a.ws_dQ, static_cast<__nv_bfloat16*>(a.dQ), a.n, a.n_pad, a.d, a.scale, groups);
  return cudaGetLastError();
}

cudaError_t bwd_read_status(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_bwd_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(unsigned int));
}

}  // namespace fa
