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
// dkdv roles (512 threads): warp 0 TMA producer, warp 1 MMA issuer, warps 4..11
// compute P^T and dS^T (two warpgroups, each owning half of the query columns;
// thread = key row), warps 12..15 drain dQ from TMEM into global memory. The
// MMA issue order is software-pipelined: S^T_i and dP^T_i are issued as soon as
// the compute groups have read block i-1's, ahead of dV_{i-1}, dK_{i-1}, dQ_{i-1}.
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
  static constexpr int CW = BQ / 2;                 // query columns per compute warpgroup
  static constexpr int KCH = D / 64;
  static constexpr int KV_CHUNK = 128 * 128;        // one 64-column chunk of K or V
  static constexpr int KV_TILE = KCH * KV_CHUNK;
  static constexpr int Q_CHUNK = BQ * 128;          // one 64-column chunk of Q_i or dO_i
  static constexpr int Q_TILE = KCH * Q_CHUNK;
  static constexpr int DS_CHUNK = BN * 128;         // 64 queries x 128 keys of dS^T (bf16)
  static constexpr int DS_TILE = (BQ / 64) * DS_CHUNK;
  static constexpr int STAGES = 3;
  // dK reads dS^T from TMEM (the TS form) instead of shared memory; needs BQ/2
  // spare TMEM columns, which only the d = 128 layout has.
  static constexpr bool kDsInTmem = (D == 128);
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
  static constexpr int B_QF = 1;                // + stage: Q_i, dO_i, L_i, D_i landed
  static constexpr int B_QE = B_QF + STAGES;    // + stage: the stage may be refilled
  static constexpr int B_SF = B_QE + STAGES;
  static constexpr int B_SFREE = B_SF + 1;
  static constexpr int B_PF = B_SF + 2;
  static constexpr int B_DVD = B_SF + 3;
  static constexpr int B_DSF = B_SF + 4;
  static constexpr int B_DSD = B_SF + 5;
  static constexpr int B_DQE = B_SF + 6;
  static constexpr int B_ACC = B_SF + 7;
  static constexpr int B_DRAIN = B_SF + 8;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
  // TMEM columns
  static constexpr uint32_t COL_S = 0;
  static constexpr uint32_t COL_DP = BQ;
  static constexpr uint32_t COL_P = 2 * BQ;
  static constexpr uint32_t COL_DV = 2 * BQ + BQ / 2;
  static constexpr uint32_t COL_DK = COL_DV + D;
  static constexpr uint32_t COL_DQ = COL_DK + D;
  static constexpr uint32_t COL_DST = COL_DQ + 64;  // dS^T as bf16 pairs (kDsInTmem)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int THREADS = 512;
  static constexpr int COMPUTE_THREADS = 256;
  static_assert(COL_DST + (kDsInTmem ? BQ / 2 : 0) <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct BwdParams {
  __nv_bfloat16 *dK, *dV;
  float* ws_dQ;
  int n, m, n_pad, BH, causal, ktiles, group;
  float scale, scale_log2;
};

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitMaxCycles / 4) break;
  }
}

template <int D>
__global__ void __launch_bounds__(512, 1)
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
  // Key blocks near 0 carry the most work under causal masking: rank 0 first,
  // heads taken a group at a time so the blocks in flight share L2.
  int ktile, bh;
  grouped_tile(blockIdx.x, p.BH, p.ktiles, p.group, ktile, bh);
  const int ks = ktile * C::BN;
  const int nqb = (p.n + C::BQ - 1) / C::BQ;
  const int i_start = p.causal ? ks / C::BQ : 0;  // first block with a query q >= ks
  const int nq = max(0, nqb - i_start);

  if (threadIdx.x == 0) {
    mbar_init(&bar[C::B_KV], 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bar[C::B_QF + s], 1);
      mbar_init(&bar[C::B_QE + s], 1);
    }
    mbar_init(&bar[C::B_SF], 1);
    mbar_init(&bar[C::B_SFREE], C::COMPUTE_THREADS);
    mbar_init(&bar[C::B_PF], C::COMPUTE_THREADS);
    mbar_init(&bar[C::B_DVD], 1);
    mbar_init(&bar[C::B_DSF], C::COMPUTE_THREADS);
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
      int nqi = 0;
      for (int i = 0; i < nq; ++i) {
        const int s = i % C::STAGES;
        const uint32_t ph = (i / C::STAGES) & 1;
        const int q0 = (i_start + i) * C::BQ;
        if (i >= C::STAGES && !mbar_wait(&bar[C::B_QE + s], ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(&bar[C::B_QF + s], 2 * C::Q_TILE + 2 * C::BQ * 4);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(smem + C::OFF_Q + s * C::Q_TILE + c * C::Q_CHUNK, &tmQ, &bar[C::B_QF + s],
                      c * 64, q0, bh);
        tma_load_2d(smem + C::OFF_LSE + s * C::BQ * 4, &tmL2, &bar[C::B_QF + s], q0, bh);
        tma_load_2d(smem + C::OFF_DD + s * C::BQ * 4, &tmD, &bar[C::B_QF + s], q0, bh);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(smem + C::OFF_DO + s * C::Q_TILE + c * C::Q_CHUNK, &tmdO,
                      &bar[C::B_QF + s], c * 64, q0, bh);
        nqi = i + 1;
      }
      drain_wait(&bar[C::B_KV], 0);
      for (int i = max(0, nqi - C::STAGES); i < nqi; ++i)
        drain_wait(&bar[C::B_QF + i % C::STAGES], (i / C::STAGES) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (operands stay warp-uniform); elect.sync
    // picks the lane that issues each tcgen05 instruction. Descriptors are built
    // once per operand buffer and advanced by compile-time byte offsets.
    if (nq > 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(128, C::BQ, false, false);
      constexpr uint32_t kIdescDV = idesc_bf16_f32(128, D, false, true);
      constexpr uint32_t kIdescDK = idesc_bf16_f32(128, D, false, true);
      constexpr uint32_t kIdescDQ = (D == 128) ? idesc_bf16_f32(128, C::BQ, true, true)
                                               : idesc_bf16_f32(128, D, true, true);
      const uint64_t dK_k = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);  // K, K-major
      const uint64_t dV_k = sdesc_sw128(smem_u32(smem + C::OFF_V), 16, 1024);  // V, K-major
      const uint64_t dK_mn = sdesc_sw128(smem_u32(smem + C::OFF_K), C::KV_CHUNK, 1024);
      const uint64_t dS_k = sdesc_sw128(smem_u32(smem + C::OFF_DS), 16, 1024);   // dS^T rows
      const uint64_t dS_mn = sdesc_sw128(smem_u32(smem + C::OFF_DS), C::DS_CHUNK, 1024);
      bool ok = warp_wait(&bar[C::B_KV], 0, wc);
      for (int i = 0; ok && i <= nq; ++i) {
        if (i < nq) {
          // S^T = K Q_i^T and dP^T = V dO_i^T, as soon as block i-1's are read
          const int s = i % C::STAGES;
          const uint32_t ph = (i / C::STAGES) & 1;
          if (!warp_wait(&bar[C::B_QF + s], ph, wc)) break;
          if (i >= 1 && !warp_wait(&bar[C::B_SFREE], (i - 1) & 1, wc)) break;
          tc_fence_after();
          const uint64_t dQ_k = sdesc_sw128(smem_u32(smem + C::OFF_Q + s * C::Q_TILE), 16, 1024);
          const uint64_t dO_k = sdesc_sw128(smem_u32(smem + C::OFF_DO + s * C::Q_TILE), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32;
            const uint32_t kb = (kk >> 2) * C::Q_CHUNK + (kk & 3) * 32;
            umma_ss_w(tmem + C::COL_S, sdesc_add(dK_k, ka), sdesc_add(dQ_k, kb), kIdescS, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32;
            const uint32_t kb = (kk >> 2) * C::Q_CHUNK + (kk & 3) * 32;
            umma_ss_w(tmem + C::COL_DP, sdesc_add(dV_k, ka), sdesc_add(dO_k, kb), kIdescS, kk > 0);
          }
          umma_commit_w(&bar[C::B_SF]);
        }
        if (i >= 1) {
          const int ii = i - 1;
          const int s = ii % C::STAGES;
          // dV += P^T dO_{i-1}
          if (!warp_wait(&bar[C::B_PF], ii & 1, wc)) break;
          tc_fence_after();
          const uint64_t dO_mn =
              sdesc_sw128(smem_u32(smem + C::OFF_DO + s * C::Q_TILE), C::Q_CHUNK, 1024);
#pragma unroll
          for (int kk = 0; kk < C::BQ / 16; ++kk)
            umma_ts_w(tmem + C::COL_DV, tmem + C::COL_P + kk * 8, sdesc_add(dO_mn, kk * 2048),
                      kIdescDV, (ii > 0 || kk > 0) ? 1u : 0u);
          umma_commit_w(&bar[C::B_DVD]);
          // dK += dS^T Q_{i-1} and this block's share of dQ_{i-1}
          if (!warp_wait(&bar[C::B_DSF], ii & 1, wc)) break;
          if (ii >= 1 && !warp_wait(&bar[C::B_DQE], (ii - 1) & 1, wc)) break;
          tc_fence_after();
          const uint64_t dQ_mn =
              sdesc_sw128(smem_u32(smem + C::OFF_Q + s * C::Q_TILE), C::Q_CHUNK, 1024);
#pragma unroll
          for (int kk = 0; kk < C::BQ / 16; ++kk) {
            const uint32_t ka = (kk >> 2) * C::DS_CHUNK + (kk & 3) * 32;
            if (C::kDsInTmem)
              umma_ts_w(tmem + C::COL_DK, tmem + C::COL_DST + kk * 8, sdesc_add(dQ_mn, kk * 2048),
                        kIdescDK, (ii > 0 || kk > 0) ? 1u : 0u);
            else
              umma_ss_w(tmem + C::COL_DK, sdesc_add(dS_k, ka), sdesc_add(dQ_mn, kk * 2048),
                        kIdescDK, (ii > 0 || kk > 0) ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk) {
            if (D == 128)
              umma_ss_w(tmem + C::COL_DQ, sdesc_add(dK_mn, kk * 2048), sdesc_add(dS_mn, kk * 2048),
                        kIdescDQ, kk > 0);
            else
              umma_ss_w(tmem + C::COL_DQ, sdesc_add(dS_mn, kk * 2048), sdesc_add(dK_mn, kk * 2048),
                        kIdescDQ, kk > 0);
          }
          umma_commit_w(&bar[C::B_DSD]);
          umma_commit_w(&bar[C::B_QE + s]);
        }
      }
      umma_commit_w(&bar[C::B_ACC]);
      umma_commit_w(&bar[C::B_DRAIN]);
      drain_wait(&bar[C::B_DRAIN], 0);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ P^T, dS^T
    const int half = (warp - 4) >> 2;              // which half of the query columns
    const int krow = ((warp - 4) & 3) * 32 + lane;  // key row = TMEM lane
    const int kg = ks + krow;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int c0 = half * C::CW;                   // first query column of this group
    const float sl2 = p.scale_log2;
    const bool key_ok = kg < p.m;
    const uint32_t sDS = smem_u32(smem + C::OFF_DS);
    bool ok = true;
    for (int i = 0; i < nq; ++i) {
      const int s = i % C::STAGES;
      const int q0 = (i_start + i) * C::BQ;
      if (!warp_wait(&bar[C::B_QF + s], (i / C::STAGES) & 1, wc)) { ok = false; break; }
      if (!warp_wait(&bar[C::B_SF], i & 1, wc)) { ok = false; break; }
      tc_fence_after();
      const float* lse = reinterpret_cast<const float*>(smem + C::OFF_LSE + s * C::BQ * 4) + c0;
      const float* dd = reinterpret_cast<const float*>(smem + C::OFF_DD + s * C::BQ * 4) + c0;
      // Causal: key kg is hidden from query q0 + c when c < kg - q0.
      const bool need_mask = p.causal && (ks + C::BN - 1 > q0 + c0);
      const int qlim = kg - q0 - c0;  // in this group's column numbering

      uint32_t pp[C::CW / 2];
      if (C::CW == 32) {
        // Read this group's S^T and dP^T columns, then release them at once so
        // that the next block's S^T / dP^T products overlap this arithmetic.
        uint32_t sr[32], dr[32];
        tmem_ld32(lane_base + C::COL_S + c0, sr);
        tmem_ld32(lane_base + C::COL_DP + c0, dr);
        tmem_ld_wait();
        reg_fence32(sr);
        reg_fence32(dr);
        tc_fence_before();
        mbar_arrive(&bar[C::B_SFREE]);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 l2 = *reinterpret_cast<const float2*>(lse + e);
          float p0 = ex2(fmaf(__uint_as_float(sr[e]), sl2, -l2.x));
          float p1 = ex2(fmaf(__uint_as_float(sr[e + 1]), sl2, -l2.y));
          if (need_mask) {
            if (e < qlim) p0 = 0.f;
            if (e + 1 < qlim) p1 = 0.f;
          }
          if (!key_ok) p0 = p1 = 0.f;
          pp[e / 2] = pack_bf16(p0, p1);
        }
        if (i >= 1) {  // P^T columns are free once dV_{i-1} is done
          if (!warp_wait(&bar[C::B_DVD], (i - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
        }
        tmem_st16(lane_base + C::COL_P + c0 / 2, pp);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar[C::B_PF]);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 d2 = *reinterpret_cast<const float2*>(dd + e);
          const uint32_t pv = pp[e / 2];
          w[e / 2] = pack_bf16(bf16_lo(pv) * (__uint_as_float(dr[e]) - d2.x),
                               bf16_hi(pv) * (__uint_as_float(dr[e + 1]) - d2.y));
        }
        if (i >= 1) {  // dS^T staging is free once dK_{i-1}, dQ_{i-1} are done
          if (!warp_wait(&bar[C::B_DSD], (i - 1) & 1, wc)) { ok = false; break; }
        }
        if (C::kDsInTmem) tmem_st16(lane_base + C::COL_DST + c0 / 2, w);
        // Row krow of dS^T, queries [c0, c0 + 32): four 16-byte chunks of the
        // 128-byte row in the swizzled layout (chunk index XOR row % 8).
        const uint32_t rowbase = sDS + krow * 128;
#pragma unroll
        for (int t = 0; t < 4; ++t)
          st_shared_v4(rowbase + (uint32_t)(((c0 / 8 + t) ^ (krow & 7)) * 16), w[4 * t],
                       w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
        if (C::kDsInTmem) {
          tmem_st_wait();
          tc_fence_before();
        }
      } else {
        // 64 columns per group, in chunks of 32 (registers do not hold both
        // S^T and dP^T at once); S^T / dP^T are released after the last chunk.
#pragma unroll
        for (int c = 0; c < C::CW / 32; ++c) {
          uint32_t sr[32];
          tmem_ld32(lane_base + C::COL_S + c0 + 32 * c, sr);
          tmem_ld_wait();
          reg_fence32(sr);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int q = 32 * c + e;
            const float2 l2 = *reinterpret_cast<const float2*>(lse + q);
            float p0 = ex2(fmaf(__uint_as_float(sr[e]), sl2, -l2.x));
            float p1 = ex2(fmaf(__uint_as_float(sr[e + 1]), sl2, -l2.y));
            if (need_mask) {
              if (q < qlim) p0 = 0.f;
              if (q + 1 < qlim) p1 = 0.f;
            }
            if (!key_ok) p0 = p1 = 0.f;
            pp[16 * c + e / 2] = pack_bf16(p0, p1);
          }
        }
        if (i >= 1) {
          if (!warp_wait(&bar[C::B_DVD], (i - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
        }
#pragma unroll
        for (int c = 0; c < C::CW / 32; ++c)
          tmem_st16(lane_base + C::COL_P + c0 / 2 + 16 * c, pp + 16 * c);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar[C::B_PF]);
        if (i >= 1) {
          if (!warp_wait(&bar[C::B_DSD], (i - 1) & 1, wc)) { ok = false; break; }
        }
#pragma unroll
        for (int c = 0; c < C::CW / 32; ++c) {
          uint32_t dr[32];
          tmem_ld32(lane_base + C::COL_DP + c0 + 32 * c, dr);
          tmem_ld_wait();
          reg_fence32(dr);
          if (c == C::CW / 32 - 1) {  // this group's S^T and dP^T fully read
            tc_fence_before();
            mbar_arrive(&bar[C::B_SFREE]);
          }
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int q = 32 * c + e;
            const float2 d2 = *reinterpret_cast<const float2*>(dd + q);
            const uint32_t pv = pp[16 * c + e / 2];
            w[e / 2] = pack_bf16(bf16_lo(pv) * (__uint_as_float(dr[e]) - d2.x),
                                 bf16_hi(pv) * (__uint_as_float(dr[e + 1]) - d2.y));
          }
          // 64-query chunk (c0 + 32c) / 64 of dS^T, 16-byte chunks ((c0+32c) % 64) / 8 + t
          const int qc = c0 + 32 * c;
          const uint32_t rowbase = sDS + (qc >> 6) * C::DS_CHUNK + krow * 128;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint32_t chunk = (uint32_t)((((qc & 63) >> 3) + t) ^ (krow & 7));
            st_shared_v4(rowbase + chunk * 16, w[4 * t], w[4 * t + 1], w[4 * t + 2],
                         w[4 * t + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bar[C::B_DSF]);
    }

    // ------------------------------------------------------------ dK, dV out
    // Group 0 writes dV, group 1 writes dK (each all D columns of its rows).
    if (ok) {
      __nv_bfloat16* dv_row = p.dV + ((size_t)bh * p.m + kg) * D;
      __nv_bfloat16* dk_row = p.dK + ((size_t)bh * p.m + kg) * D;
      const uint32_t col = half == 0 ? C::COL_DV : C::COL_DK;
      const float mul = half == 0 ? 1.f : p.scale;
      __nv_bfloat16* dst_row = half == 0 ? dv_row : dk_row;
      if (nq == 0) {
        if (key_ok) {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(dst_row)[c] = z;
        }
      } else if (warp_wait(&bar[C::B_ACC], 0, wc)) {
        tc_fence_after();
        {
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
  } else if (warp >= 12) {
    // ------------------------------------------------------------ dQ drain
    const int t = (warp - 12) * 32 + lane;  // TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    bool ok = true;
    for (int i = 0; i < nq; ++i) {
      const int q0 = (i_start + i) * C::BQ;
      if (ok) ok = warp_wait(&bar[C::B_DSD], i & 1, wc);
      uint32_t v[64];
      if (ok) {
        tc_fence_after();
        tmem_ld32(lane_base + C::COL_DQ, v);
        tmem_ld32(lane_base + C::COL_DQ + 32, v + 32);
        tmem_ld_wait();
        reg_fence32(v);
        reg_fence32(v + 32);
        tc_fence_before();
        mbar_arrive(&bar[C::B_DQE]);
      }
      if (D == 128 && ok) {
        // lane t = feature index, column = query: each warp adds 32 consecutive
        // floats of one accumulator row per instruction.
        float* base = p.ws_dQ + ((size_t)bh * p.n_pad + q0) * D + t;
#pragma unroll
        for (int q = 0; q < 64; ++q) atomicAdd(base + (size_t)q * D, __uint_as_float(v[q]));
      } else if (ok) {
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
// Each warp step covers RPW consecutive workspace rows (head bh, query q <
// n_pad), LPR lanes per row, one 16-byte load of O and of dO per lane:
// D = sum_c dO*O, L2 = L * log2(e), and the rows' dQ accumulator cleared. Rows
// q >= n get D = 0 and L2 = +inf so that recomputed probabilities there are
// exactly 0.
template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const __nv_bfloat16* __restrict__ O,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         const float* __restrict__ L,
                                                         float* __restrict__ ws_D,
                                                         float* __restrict__ ws_L2,
                                                         float* __restrict__ ws_dQ, int n,
                                                         int n_pad, long long rows) {
  constexpr int LPR = D / 8;       // lanes per row (8 bf16 per lane)
  constexpr int RPW = 32 / LPR;    // rows per warp step
  const int lane = threadIdx.x & 31;
  const int sub = lane % LPR;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long base = ((long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RPW;
       base < rows; base += warps * RPW) {
    const long long r = base + lane / LPR;  // rows is a multiple of RPW (n_pad % 128 == 0)
    const long long bh = r / n_pad;
    const int q = (int)(r - bh * n_pad);
    float acc = 0.f;
    if (q < n) {
      const size_t off = ((size_t)bh * n + q) * D;
      const uint4 a = reinterpret_cast<const uint4*>(O + off)[sub];
      const uint4 b = reinterpret_cast<const uint4*>(dO + off)[sub];
      acc = bf16_lo(a.x) * bf16_lo(b.x) + bf16_hi(a.x) * bf16_hi(b.x) +
            bf16_lo(a.y) * bf16_lo(b.y) + bf16_hi(a.y) * bf16_hi(b.y) +
            bf16_lo(a.z) * bf16_lo(b.z) + bf16_hi(a.z) * bf16_hi(b.z) +
            bf16_lo(a.w) * bf16_lo(b.w) + bf16_hi(a.w) * bf16_hi(b.w);
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (sub == 0) {
      ws_D[r] = acc;
      ws_L2[r] = (q < n) ? L[(size_t)bh * n + q] * kLog2e : INFINITY;
    }
    // the RPW rows' accumulator (RPW * D floats = 1 KB): two float4 per lane
    float4* drow = reinterpret_cast<float4*>(ws_dQ + (size_t)base * D);
    drow[2 * lane] = make_float4(0.f, 0.f, 0.f, 0.f);
    drow[2 * lane + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ------------------------------------------------------------------ dQ convert
// dQ[bh, q, :] = bf16(accumulator[bh, q, :] * scale) for q < n; 16 values per thread.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ ws_dQ,
                                                         __nv_bfloat16* __restrict__ dQ, int n,
                                                         int n_pad, int d, float scale,
                                                         long long groups) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const int gpr = d / 16;  // groups of 16 per row
  for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += stride) {
    const long long row = g / gpr;  // over BH * n
    const int c16 = (int)(g - row * gpr);
    const long long bh = row / n;
    const int q = (int)(row - bh * n);
    const float4* src =
        reinterpret_cast<const float4*>(ws_dQ + ((size_t)bh * n_pad + q) * d) + 4 * c16;
    const float4 a = src[0], b = src[1], c = src[2], e = src[3];
    uint4* dst = reinterpret_cast<uint4*>(dQ + (size_t)row * d) + 2 * c16;
    dst[0] = make_uint4(pack_bf16(a.x * scale, a.y * scale), pack_bf16(a.z * scale, a.w * scale),
                        pack_bf16(b.x * scale, b.y * scale), pack_bf16(b.z * scale, b.w * scale));
    dst[1] = make_uint4(pack_bf16(c.x * scale, c.y * scale), pack_bf16(c.z * scale, c.w * scale),
                        pack_bf16(e.x * scale, e.y * scale), pack_bf16(e.z * scale, e.w * scale));
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
  p.ktiles = ceil_div(a.m, C::BN);
  p.group = heads_per_group(a.BH, p.ktiles);
  cudaError_t e =
      cudaFuncSetAttribute(dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)p.ktiles * (unsigned)a.BH;
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
  const int grid = grid_for(rows / (a.d == 128 ? 2 : 4), 8);  // warp steps, 8 warps a block
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
  const long long groups = (long long)a.BH * a.n * (a.d / 16);
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
