// Backward pass of exact attention, FlashAttention-2 recompute form
// ("05_flash_attention.py", flash_attention_backward):
//   D = rowsum(dO o O); P = exp(S - L) rebuilt from the saved L;
//   dV = P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = dS K * scale,
//   dK = dS^T Q * scale; blocks wholly above the diagonal are skipped under
//   causal masking.
//
// Three kernels on one stream:
//   preprocess  -D and -L * log2(e) (-inf past n) into the workspace; memory bound.
//   dkdv        one CTA per (key block of 128, head), looping over query blocks
//               of 128. The key block's K and V stay in shared memory; dK and dV
//               accumulate in TMEM and are written once. The transposed
//               products put the key index on the TMEM lane:
//                 S^T  = K Q_i^T       dP^T = V dO_i^T     (SS MMAs)
//                 dV  += P^T dO_i      dK  += dS^T Q_i     (TS MMAs: P^T and dS^T
//                                                           are written to TMEM)
//   dq          one CTA per (query block of 128, head), looping over key blocks
//               of 128, with Q and dO held in TMEM:
//                 S = Q K_j^T, dP = dO V_j^T, dQ += dS K_j  (TS MMAs)
//               dQ accumulates in TMEM and is written once, scaled, as bf16.
//
// The pages' loop adds each block's dS K into dQ in memory from inside the key
// loop. Here dQ is its own pass that recomputes S and dP for its query block:
// two more products of the same size, against an fp32 read-modify-write of dQ
// per (query block, key block) pair. On GB300 those reductions (64 KiB per pair,
// 2.2 GB at n = 4096, 64 heads) are bound by the L2 reduction rate (about
// 6 TB/s) and would cap the backward pass; the recompute runs on tensor cores
// that have room for it, needs no zeroed accumulator or conversion pass, and
// makes dQ deterministic.
//
// Roles (384 threads in both kernels): warp 0 TMA producer, warp 1 MMA issuer
// (whole warp, one elected lane issues), warps 4..11 two compute warpgroups,
// each owning half (64) of the columns of a 128 x 128 score block; thread =
// TMEM lane (key row in dkdv, query row in dq). The products of each half are
// formed separately (N = 64) and the two halves are interleaved, so that one
// group computes probabilities while the tensor cores work for the other.
#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

__device__ unsigned int g_bwd_status;

namespace {

constexpr float kLog2e = 1.44269504088896340736f;

// Bounded wait that ignores the abort flag: used only to let copies or MMAs
// already in flight land before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitMaxCycles / 4) break;
  }
}

// Probabilities for W consecutive columns: s[c] <- exp2(s[c] * sl2 + nl2[c]), 0 for
// c < hide when `masked`; pp[c/2] <- bf16 pairs (skipped when pp is null). nl2 is
// -L * log2(e) per column (dkdv: one per query) or a broadcast scalar (dq).
template <int W, bool kColumnL>
__device__ __forceinline__ void probabilities(uint32_t* s, uint32_t* pp, float sl2,
                                              const float* nl2_cols, float nl2_row, int hide,
                                              bool masked) {
  const uint64_t sl2x2 = f2pack(sl2, sl2);
#pragma unroll
  for (int e = 0; e < W; e += 4) {
    uint64_t b0, b1;
    if (kColumnL) {
      const float4 l = *reinterpret_cast<const float4*>(nl2_cols + e);
      b0 = f2pack(l.x, l.y);
      b1 = f2pack(l.z, l.w);
    } else {
      b0 = b1 = f2pack(nl2_row, nl2_row);
    }
    float x0, x1, x2, x3;
    f2unpack(ffma2(f2pack(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), sl2x2, b0), x0, x1);
    f2unpack(ffma2(f2pack(__uint_as_float(s[e + 2]), __uint_as_float(s[e + 3])), sl2x2, b1), x2,
             x3);
    float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
    if (masked) {
      if (e < hide) p0 = 0.f;
      if (e + 1 < hide) p1 = 0.f;
      if (e + 2 < hide) p2 = 0.f;
      if (e + 3 < hide) p3 = 0.f;
    }
    s[e] = __float_as_uint(p0);
    s[e + 1] = __float_as_uint(p1);
    s[e + 2] = __float_as_uint(p2);
    s[e + 3] = __float_as_uint(p3);
    if (pp) {
      pp[e / 2] = pack_bf16(p0, p1);
      pp[e / 2 + 1] = pack_bf16(p2, p3);
    }
  }
}
template <bool kColumnL>
__device__ __forceinline__ void probabilities32(uint32_t* s, uint32_t* pp, float sl2,
                                                const float* nl2_cols, float nl2_row, int hide,
                                                bool masked) {
  probabilities<32, kColumnL>(s, pp, sl2, nl2_cols, nl2_row, hide, masked);
}
template <bool kColumnL>
__device__ __forceinline__ void probabilities64(uint32_t* s, uint32_t* pp, float sl2,
                                                const float* nl2_cols, float nl2_row, int hide,
                                                bool masked) {
  probabilities<64, kColumnL>(s, pp, sl2, nl2_cols, nl2_row, hide, masked);
}

// dS for 32 columns: w[c/2] <- bf16 pairs of p[c] * (dp[c] + nd[c]).
template <bool kColumnD>
__device__ __forceinline__ void dscores32(const uint32_t* p, const uint32_t* dp, uint32_t* w,
                                          const float* nd_cols, float nd_row) {
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    uint64_t n0, n1;
    if (kColumnD) {
      const float4 v = *reinterpret_cast<const float4*>(nd_cols + e);
      n0 = f2pack(v.x, v.y);
      n1 = f2pack(v.z, v.w);
    } else {
      n0 = n1 = f2pack(nd_row, nd_row);
    }
    const uint64_t t0 = fadd2(f2pack(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), n0);
    const uint64_t t1 = fadd2(f2pack(__uint_as_float(dp[e + 2]), __uint_as_float(dp[e + 3])), n1);
    float a0, a1, a2, a3;
    f2unpack(fmul2(f2pack(__uint_as_float(p[e]), __uint_as_float(p[e + 1])), t0), a0, a1);
    f2unpack(fmul2(f2pack(__uint_as_float(p[e + 2]), __uint_as_float(p[e + 3])), t1), a2, a3);
    w[e / 2] = pack_bf16(a0, a1);
    w[e / 2 + 1] = pack_bf16(a2, a3);
  }
}

// ================================================================== dK, dV
// K of the key block is moved into TMEM once (the A operand of S^T); V stays in
// shared memory. Each query block is taken in two halves of 64 queries and both
// compute groups work on every half (32 queries each). S^T of consecutive halves
// alternates between two TMEM regions and dP^T has a region of its own, so S^T
// of half u+2 is formed while half u is still being processed:
//   S^T_0 dP^T_0 S^T_1 | dV_0 dP^T_1 dK_0 S^T_2 | dV_1 dP^T_2 dK_1 S^T_3 | ...
template <int D>
struct KvCfg {
  static constexpr int BN = 128;      // keys per CTA = TMEM lanes
  static constexpr int BQ = 128;      // queries per block (two halves of 64)
  static constexpr int KCH = D / 64;  // 128-byte column chunks of a row
  static constexpr int CHUNK = 128 * 128;
  static constexpr int TILE = KCH * CHUNK;       // 128 rows of Q, dO, K or V
  static constexpr int HALF_ROWS = 64 * 128;     // bytes of 64 rows of one chunk
  static constexpr int STAGES = (D == 128) ? 2 : 4;
  static constexpr int K_STAGE = STAGES - 1;     // its Q buffer holds K until K is in TMEM
  static constexpr int OFF_V = 0;
  static constexpr int OFF_Q = TILE;
  static constexpr int OFF_DO = OFF_Q + STAGES * TILE;
  static constexpr int OFF_NL2 = OFF_DO + STAGES * TILE;     // [STAGES][BQ] fp32
  static constexpr int OFF_ND = OFF_NL2 + STAGES * BQ * 4;   // [STAGES][BQ] fp32
  static constexpr int OFF_BAR = OFF_ND + STAGES * BQ * 4;
  // barrier slots
  static constexpr int B_KV = 0;              // K, V landed in shared memory
  static constexpr int B_IN = 1;              // K in TMEM (256 arrivals)
  static constexpr int B_QF = 2;              // + stage: Q_i, dO_i, -L2_i, -D_i landed
  static constexpr int B_QE = B_QF + STAGES;  // + stage: the block's products done
  static constexpr int B_SF = B_QE + STAGES;  // + region: S^T in that region done
  static constexpr int B_DPF = B_SF + 2;      // dP^T of the current half done
  // + (u & 1): P^T of half u in TMEM (256 arrivals). Two slots: P^T of half u+1
  // needs only S^T_{u+1}, which is issued before the MMA warp waits for P^T_u,
  // so one barrier could complete twice before that wait and hide its phase.
  static constexpr int B_PF = B_SF + 3;
  static constexpr int B_DSF = B_SF + 5;      // dS^T in TMEM (256 arrivals)
  static constexpr int B_ACC = B_SF + 6;      // dK, dV final
  static constexpr int B_DRAIN = B_SF + 7;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
  // TMEM columns: K as bf16 pairs, two 64-column S^T regions, the dP^T region,
  // dV, dK. Group w keeps P^T over [32w, 32w + 16) and dS^T over
  // [32w + 16, 32w + 32) of the half's S^T region.
  static constexpr uint32_t COL_K = 0;
  static constexpr uint32_t COL_S = 64;   // regions at 64 and 128
  static constexpr uint32_t COL_DP = 192;
  static constexpr uint32_t COL_DV = 256;
  static constexpr uint32_t COL_DK = 256 + D;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int THREADS = 384;
  static constexpr int COMPUTE_THREADS = 256;
  static_assert(COL_DK + D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct KvParams {
  __nv_bfloat16 *dK, *dV;
  int n, m, n_pad, BH, causal, ktiles, group;
  float scale, scale_log2;
};

// TMEM column of k-step kk (16 queries) of the P^T (part 0) or dS^T (part 1)
// operand of a half stored in region `reg`.
__device__ __forceinline__ uint32_t half_operand_col(uint32_t reg, int part, int kk) {
  return reg + (uint32_t)((kk >> 1) * 32 + part * 16 + (kk & 1) * 8);
}

// One CTA of the dK, dV pass: key block `lin` in launch order.
template <int D>
__device__ __forceinline__ void dkdv_cta(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                         const CUtensorMap& tmV, const CUtensorMap& tmdO,
                                         const CUtensorMap& tmNL2, const CUtensorMap& tmND,
                                         const KvParams& p, int lin) {
  using C = KvCfg<D>;
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
  grouped_tile(lin, p.BH, p.ktiles, p.group, ktile, bh);
  const int ks = ktile * C::BN;
  const int nqb = (p.n + C::BQ - 1) / C::BQ;
  const int i_start = p.causal ? ks / C::BQ : 0;  // first block with a query q >= ks
  const int nq = max(0, nqb - i_start);
  const int nu = 2 * nq;                          // halves

  if (threadIdx.x == 0) {
    mbar_init(&bar[C::B_KV], 1);
    mbar_init(&bar[C::B_IN], C::COMPUTE_THREADS);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bar[C::B_QF + s], 1);
      mbar_init(&bar[C::B_QE + s], 1);
    }
    mbar_init(&bar[C::B_SF], 1);
    mbar_init(&bar[C::B_SF + 1], 1);
    mbar_init(&bar[C::B_DPF], 1);
    mbar_init(&bar[C::B_PF], C::COMPUTE_THREADS);
    mbar_init(&bar[C::B_PF + 1], C::COMPUTE_THREADS);
    mbar_init(&bar[C::B_DSF], C::COMPUTE_THREADS);
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
      mbar_arrive_expect_tx(&bar[C::B_KV], 2 * C::TILE);
#pragma unroll
      for (int c = 0; c < C::KCH; ++c) {
        tma_load_3d(smem + C::OFF_Q + C::K_STAGE * C::TILE + c * C::CHUNK, &tmK, &bar[C::B_KV],
                    c * 64, ks, bh);
        tma_load_3d(smem + C::OFF_V + c * C::CHUNK, &tmV, &bar[C::B_KV], c * 64, ks, bh);
      }
      int issued = 0;
      for (int i = 0; i < nq; ++i) {
        const int s = i % C::STAGES;
        const int q0 = (i_start + i) * C::BQ;
        if (i >= C::STAGES && !mbar_wait(&bar[C::B_QE + s], ((i / C::STAGES) & 1) ^ 1, wc)) break;
        if (i == C::K_STAGE && !mbar_wait(&bar[C::B_IN], 0, wc)) break;
        uint64_t* f = &bar[C::B_QF + s];
        mbar_arrive_expect_tx(f, 2 * C::TILE + 2 * C::BQ * 4);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(smem + C::OFF_Q + s * C::TILE + c * C::CHUNK, &tmQ, f, c * 64, q0, bh);
        tma_load_2d(smem + C::OFF_NL2 + s * C::BQ * 4, &tmNL2, f, q0, bh);
        tma_load_2d(smem + C::OFF_ND + s * C::BQ * 4, &tmND, f, q0, bh);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(smem + C::OFF_DO + s * C::TILE + c * C::CHUNK, &tmdO, f, c * 64, q0, bh);
        issued = i + 1;
      }
      drain_wait(&bar[C::B_KV], 0);
      for (int i = max(0, issued - C::STAGES); i < issued; ++i)
        drain_wait(&bar[C::B_QF + i % C::STAGES], (i / C::STAGES) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (nq > 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t kIdescG = idesc_bf16_f32(128, D, false, true);
      const uint64_t v_k = sdesc_sw128(smem_u32(smem + C::OFF_V), 16, 1024);  // V, K-major
      auto sreg = [&](int u) { return tmem + C::COL_S + 64u * (uint32_t)(u & 1); };
      // B operand rows of half u in the Q or dO buffer of its block
      auto half_rows = [&](int base, int u) {
        return smem_u32(smem + base + ((u >> 1) % C::STAGES) * C::TILE + (u & 1) * C::HALF_ROWS);
      };
      // S^T_u = K Q_u^T (TS, N = 64) into its region. The region still holds
      // P^T / dS^T of half u-2, read by dV / dK of that half, which this thread
      // issued earlier: tcgen05.mma instructions of one thread execute in order.
      auto scores = [&](int u) {
        const uint64_t b_k = sdesc_sw128(half_rows(C::OFF_Q, u), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
          umma_ts_w(sreg(u), tmem + C::COL_K + kk * 8, sdesc_add(b_k, off), kIdescS, kk > 0);
        }
        umma_commit_w(&bar[C::B_SF + (u & 1)]);
      };
      // dP^T_u = V dO_u^T (SS, N = 64). The compute groups read dP^T_{u-1}
      // before signalling dS^T_{u-1}.
      auto dscores = [&](int u) {
        const uint64_t b_k = sdesc_sw128(half_rows(C::OFF_DO, u), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
          umma_ss_w(tmem + C::COL_DP, sdesc_add(v_k, off), sdesc_add(b_k, off), kIdescS, kk > 0);
        }
        umma_commit_w(&bar[C::B_DPF]);
      };
      // dV += P^T_u dO_u (part 0) or dK += dS^T_u Q_u (part 1), TS
      auto grads = [&](int u, int part) {
        const uint64_t b_mn =
            sdesc_sw128(half_rows(part == 0 ? C::OFF_DO : C::OFF_Q, u), C::CHUNK, 1024);
        const uint32_t dcol = tmem + (part == 0 ? C::COL_DV : C::COL_DK);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_ts_w(dcol, half_operand_col(sreg(u), part, kk), sdesc_add(b_mn, kk * 2048),
                    kIdescG, (u > 0 || kk > 0) ? 1u : 0u);
      };
      bool ok = warp_wait(&bar[C::B_IN], 0, wc) && warp_wait(&bar[C::B_KV], 0, wc) &&
                warp_wait(&bar[C::B_QF], 0, wc);
      if (ok) {
        tc_fence_after();
        scores(0);
        dscores(0);
        if (nu > 1) scores(1);
      }
      for (int u = 0; ok && u < nu; ++u) {
        if (!warp_wait(&bar[C::B_PF + (u & 1)], (u >> 1) & 1, wc)) break;
        tc_fence_after();
        grads(u, 0);
        if (!warp_wait(&bar[C::B_DSF], u & 1, wc)) break;
        tc_fence_after();
        if (u + 1 < nu) dscores(u + 1);
        grads(u, 1);
        if (u & 1) umma_commit_w(&bar[C::B_QE + (u >> 1) % C::STAGES]);  // block's last reader
        if (u + 2 < nu) {
          if (((u + 2) & 1) == 0) {
            const int i2 = (u + 2) >> 1;
            if (!warp_wait(&bar[C::B_QF + i2 % C::STAGES], (i2 / C::STAGES) & 1, wc)) break;
            tc_fence_after();
          }
          scores(u + 2);
        }
      }
      umma_commit_w(&bar[C::B_ACC]);
      umma_commit_w(&bar[C::B_DRAIN]);
      drain_wait(&bar[C::B_DRAIN], 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ P^T, dS^T
    const int w = (warp - 4) >> 2;               // compute group
    const int krow = (warp & 3) * 32 + lane;     // key row = TMEM lane
    const int kg = ks + krow;
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float sl2 = p.scale_log2;
    const bool key_ok = kg < p.m;
    bool ok = true;
    if (nq > 0) {
      // Group 0 moves key row krow of K into TMEM: the row's 16-byte pieces in
      // the 128-byte-swizzled tile (piece j of a chunk row at j ^ (row % 8)).
      if (w == 0) {
        ok = warp_wait(&bar[C::B_KV], 0, wc);
        if (ok) {
          const uint8_t* tile = smem + C::OFF_Q + C::K_STAGE * C::TILE;
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            uint32_t v[32];
            const uint8_t* row = tile + c * C::CHUNK + krow * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint4 x = *reinterpret_cast<const uint4*>(row + ((j ^ (krow & 7)) << 4));
              v[4 * j] = x.x;
              v[4 * j + 1] = x.y;
              v[4 * j + 2] = x.z;
              v[4 * j + 3] = x.w;
            }
            tmem_st32(tl + C::COL_K + 32 * c, v);
          }
          tmem_st_wait();
          tc_fence_before();
        }
      }
      mbar_arrive(&bar[C::B_IN]);
    }
    for (int u = 0; ok && u < nu; ++u) {
      const int i = u >> 1, h = u & 1;
      const int s = i % C::STAGES;
      const int c0 = 64 * h + 32 * w;              // first query column of this group
      const int q0 = (i_start + i) * C::BQ;
      if (h == 0 && !warp_wait(&bar[C::B_QF + s], (i / C::STAGES) & 1, wc)) { ok = false; break; }
      if (!warp_wait(&bar[C::B_SF + h], (u >> 1) & 1, wc)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sr_col = tl + C::COL_S + 64u * (uint32_t)h + 32u * (uint32_t)w;
      const float* nl2 = reinterpret_cast<const float*>(smem + C::OFF_NL2 + s * C::BQ * 4) + c0;
      const float* nd = reinterpret_cast<const float*>(smem + C::OFF_ND + s * C::BQ * 4) + c0;
      // Columns c < hide are masked: query q0 + c0 + c < key kg under causal
      // masking, or all of them for a key past m.
      const int hide = key_ok ? (p.causal ? kg - q0 - c0 : 0) : 32;
      const bool masked = __any_sync(0xffffffffu, hide > 0);
      uint32_t sr[32], pp[16];
      tmem_ld32(sr_col, sr);
      tmem_ld_wait();
      reg_fence32(sr);
      if (masked)
        probabilities32<true>(sr, pp, sl2, nl2, 0.f, hide, true);
      else
        probabilities32<true>(sr, pp, sl2, nl2, 0.f, 0, false);
      // P^T (bf16) over the first 16 of this group's 32 S^T columns, already read.
      tmem_st16(sr_col, pp);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar[C::B_PF + h]);
      if (!warp_wait(&bar[C::B_DPF], u & 1, wc)) { ok = false; break; }
      tc_fence_after();
      uint32_t dr[32], ws[16];
      tmem_ld32(tl + C::COL_DP + 32u * (uint32_t)w, dr);
      tmem_ld_wait();
      reg_fence32(dr);
      dscores32<true>(sr, dr, ws, nd, 0.f);
      tmem_st16(sr_col + 16, ws);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar[C::B_DSF]);
    }

    // ------------------------------------------------------------ dK, dV out
    // Group 0 writes dV, group 1 writes dK (each all D columns of its rows).
    if (ok) {
      const uint32_t col = w == 0 ? C::COL_DV : C::COL_DK;
      const float mul = w == 0 ? 1.f : p.scale;
      __nv_bfloat16* dst_row = (w == 0 ? p.dV : p.dK) + ((size_t)bh * p.m + kg) * D;
      if (nq == 0) {
        if (key_ok) {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(dst_row)[c] = z;
        }
      } else if (warp_wait(&bar[C::B_ACC], 0, wc)) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tl + col + 32 * c, o);
          tmem_ld_wait();
          reg_fence32(o);
          uint32_t wv[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            wv[e] = pack_bf16(__uint_as_float(o[2 * e]) * mul, __uint_as_float(o[2 * e + 1]) * mul);
          if (key_ok) {
            uint4* dst = reinterpret_cast<uint4*>(dst_row + 32 * c);
            dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            dst[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
            dst[2] = make_uint4(wv[8], wv[9], wv[10], wv[11]);
            dst[3] = make_uint4(wv[12], wv[13], wv[14], wv[15]);
          }
        }
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

// ================================================================== dQ
template <int D>
struct QCfg {
  static constexpr int BM = 128;      // queries per CTA = TMEM lanes
  static constexpr int BN = 128;      // keys per step
  static constexpr int KCH = D / 64;
  static constexpr int CHUNK = 128 * 128;
  static constexpr int TILE = KCH * CHUNK;
  static constexpr int STAGES = (D == 128) ? 3 : 4;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = STAGES * TILE;
  static constexpr int OFF_BAR = 2 * STAGES * TILE;
  // Q and dO of the block are copied into the last stage's K and V buffers
  // first; the compute groups move them into TMEM, then the stage holds K, V.
  static constexpr int QDO_STAGE = STAGES - 1;
  static constexpr int B_QDO = 0;              // Q and dO landed in shared memory
  static constexpr int B_IN = 1;               // Q and dO rows in TMEM (256 arrivals)
  static constexpr int B_KVF = 2;              // + stage: K_j, V_j landed
  static constexpr int B_KVE = B_KVF + STAGES;  // + stage: dQ_j done, refill
  // Per half h of the key block (two slots each):
  static constexpr int B_SF = B_KVE + STAGES;  // + h: S_h done
  static constexpr int B_DPF = B_SF + 2;       // + h: dP_h done
  static constexpr int B_DSF = B_SF + 4;       // + h: dS_h in TMEM (128 arrivals)
  static constexpr int B_ACC = B_SF + 6;
  static constexpr int B_DRAIN = B_SF + 7;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
  // TMEM columns: Q and dO as bf16 pairs (the A operands of S and dP); for half h
  // of the key block S_h at COL_S + 64h (then dS_h as bf16 pairs over its first
  // 32 columns) and dP_h at COL_DP + 64h; dQ.
  static constexpr uint32_t COL_Q = 0;
  static constexpr uint32_t COL_DO = D / 2;
  static constexpr uint32_t COL_S = D;
  static constexpr uint32_t COL_DP = D + 128;
  static constexpr uint32_t COL_DQ = D + 256;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int THREADS = 384;
  static constexpr int COMPUTE_THREADS = 256;
  static constexpr int GROUP_THREADS = 128;
  static constexpr int HALF_ROWS = 64 * 128;  // bytes of 64 rows of one 128-byte chunk
  static_assert(COL_DQ + D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct DqParams {
  __nv_bfloat16* dQ;
  const float *nD, *nL2;
  int n, m, n_pad, BH, causal, qtiles, group;
  float scale, scale_log2;
};

// One CTA of the dQ pass: query block `lin` in launch order.
template <int D>
__device__ __forceinline__ void dq_cta(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                       const CUtensorMap& tmV, const CUtensorMap& tmdO,
                                       const DqParams& p, int lin) {
  using C = QCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + C::NBAR);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wc{abort_flag, &g_bwd_status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Under causal masking the last query blocks see the most keys: they go first.
  int rank, bh;
  grouped_tile(lin, p.BH, p.qtiles, p.group, rank, bh);
  const int qtile = p.causal ? p.qtiles - 1 - rank : rank;
  const int q0 = qtile * C::BM;
  int nkb = (p.m + C::BN - 1) / C::BN;
  if (p.causal) nkb = min(nkb, min(q0 + C::BM - 1, p.n - 1) / C::BN + 1);  // keys k <= q

  if (threadIdx.x == 0) {
    mbar_init(&bar[C::B_QDO], 1);
    mbar_init(&bar[C::B_IN], C::COMPUTE_THREADS);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bar[C::B_KVF + s], 1);
      mbar_init(&bar[C::B_KVE + s], 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&bar[C::B_SF + h], 1);
      mbar_init(&bar[C::B_DPF + h], 1);
      mbar_init(&bar[C::B_DSF + h], C::GROUP_THREADS);
    }
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
    if (lane == 0 && nkb > 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      tma_prefetch_map(&tmdO);
      {
        uint64_t* f = &bar[C::B_QDO];
        mbar_arrive_expect_tx(f, 2 * C::TILE);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c) {
          tma_load_3d(smem + C::OFF_K + C::QDO_STAGE * C::TILE + c * C::CHUNK, &tmQ, f, c * 64,
                      q0, bh);
          tma_load_3d(smem + C::OFF_V + C::QDO_STAGE * C::TILE + c * C::CHUNK, &tmdO, f, c * 64,
                      q0, bh);
        }
      }
      int issued = 0;
      for (int j = 0; j < nkb; ++j) {
        const int s = j % C::STAGES;
        if (j >= C::STAGES && !mbar_wait(&bar[C::B_KVE + s], ((j / C::STAGES) & 1) ^ 1, wc))
          break;
        // the last stage holds Q and dO until they are in TMEM
        if (j == C::QDO_STAGE && !mbar_wait(&bar[C::B_IN], 0, wc)) break;
        uint64_t* f = &bar[C::B_KVF + s];
        mbar_arrive_expect_tx(f, 2 * C::TILE);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c) {
          tma_load_3d(smem + C::OFF_K + s * C::TILE + c * C::CHUNK, &tmK, f, c * 64, j * C::BN, bh);
          tma_load_3d(smem + C::OFF_V + s * C::TILE + c * C::CHUNK, &tmV, f, c * 64, j * C::BN, bh);
        }
        issued = j + 1;
      }
      drain_wait(&bar[C::B_QDO], 0);
      for (int j = max(0, issued - C::STAGES); j < issued; ++j)
        drain_wait(&bar[C::B_KVF + j % C::STAGES], (j / C::STAGES) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Halves of each key block (64 keys, one per compute group) interleaved:
    //   S_0 dP_0 S_1 dP_1 | dQ_0 S_0' dP_0' dQ_1 S_1' dP_1' | ...  (' = next block)
    if (nkb > 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t kIdescQ = idesc_bf16_f32(128, D, false, true);
      // S_h = Q K_h^T and dP_h = dO V_h^T for half h of key block j (N = 64). The
      // S_h columns still hold dS_h of block j-1, read by dQ of block j-1 that
      // this thread issued earlier (in-order execution); group h signalled dS_h
      // of block j-1 only after reading S_h and dP_h of it.
      auto scores = [&](int j, int h) {
        const int s = j % C::STAGES;
        const uint64_t k_k =
            sdesc_sw128(smem_u32(smem + C::OFF_K + s * C::TILE + h * C::HALF_ROWS), 16, 1024);
        const uint64_t v_k =
            sdesc_sw128(smem_u32(smem + C::OFF_V + s * C::TILE + h * C::HALF_ROWS), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
          umma_ts_w(tmem + C::COL_S + 64 * h, tmem + C::COL_Q + kk * 8, sdesc_add(k_k, off),
                    kIdescS, kk > 0);
        }
        umma_commit_w(&bar[C::B_SF + h]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
          umma_ts_w(tmem + C::COL_DP + 64 * h, tmem + C::COL_DO + kk * 8, sdesc_add(v_k, off),
                    kIdescS, kk > 0);
        }
        umma_commit_w(&bar[C::B_DPF + h]);
      };
      bool ok = warp_wait(&bar[C::B_IN], 0, wc) && warp_wait(&bar[C::B_KVF], 0, wc);
      if (ok) {
        tc_fence_after();
        scores(0, 0);
        scores(0, 1);
      }
      for (int j = 0; ok && j < nkb; ++j) {
        const int s = j % C::STAGES;
        for (int h = 0; ok && h < 2; ++h) {
          // dQ += dS_h K_h
          if (!warp_wait(&bar[C::B_DSF + h], j & 1, wc)) { ok = false; break; }
          tc_fence_after();
          const uint64_t k_mn = sdesc_sw128(
              smem_u32(smem + C::OFF_K + s * C::TILE + h * C::HALF_ROWS), C::CHUNK, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ts_w(tmem + C::COL_DQ, tmem + C::COL_S + 64 * h + kk * 8,
                      sdesc_add(k_mn, kk * 2048), kIdescQ, (j > 0 || h > 0 || kk > 0) ? 1u : 0u);
          if (h == 1) umma_commit_w(&bar[C::B_KVE + s]);  // last reader of K_j, V_j
          if (j + 1 < nkb) {
            if (h == 0 &&
                !warp_wait(&bar[C::B_KVF + (j + 1) % C::STAGES], ((j + 1) / C::STAGES) & 1, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
            scores(j + 1, h);
          }
        }
      }
      umma_commit_w(&bar[C::B_ACC]);
      umma_commit_w(&bar[C::B_DRAIN]);
      drain_wait(&bar[C::B_DRAIN], 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ P, dS
    const int h = (warp - 4) >> 2;            // which half of the key columns
    const int r = (warp & 3) * 32 + lane;     // query row = TMEM lane
    const int q = q0 + r;
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const bool row_ok = q < p.n;
    const size_t ws_row = (size_t)bh * p.n_pad + q;  // q < n_pad always
    const float nl2 = p.nL2[ws_row];
    const float nd = p.nD[ws_row];
    const float sl2 = p.scale_log2;
    bool ok = nkb == 0 || warp_wait(&bar[C::B_QDO], 0, wc);
    if (ok && nkb > 0) {
      // Group 0 moves row r of Q into TMEM, group 1 row r of dO: the row's 16-byte
      // pieces in the 128-byte-swizzled tile (piece j of a chunk row at j ^ (r % 8)).
      const uint8_t* tile = smem + (h == 0 ? C::OFF_K : C::OFF_V) + C::QDO_STAGE * C::TILE;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v[32];
        const uint8_t* row = tile + c * C::CHUNK + r * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 x = *reinterpret_cast<const uint4*>(row + ((j ^ (r & 7)) << 4));
          v[4 * j] = x.x;
          v[4 * j + 1] = x.y;
          v[4 * j + 2] = x.z;
          v[4 * j + 3] = x.w;
        }
        tmem_st32(tl + (h == 0 ? C::COL_Q : C::COL_DO) + 32 * c, v);
      }
      tmem_st_wait();
      tc_fence_before();
    }
    mbar_arrive(&bar[C::B_IN]);
    for (int j = 0; j < nkb; ++j) {
      if (!warp_wait(&bar[C::B_SF + h], j & 1, wc)) { ok = false; break; }
      tc_fence_after();
      const int k0 = j * C::BN + 64 * h;  // key of this group's column 0
      // Columns c >= vis are masked: past m, or key k0 + c > q under causal masking.
      int vis = p.m - k0;
      if (p.causal) vis = min(vis, q - k0 + 1);
      const bool masked = __any_sync(0xffffffffu, vis < 64);
      uint32_t sr[64];
      tmem_ld32(tl + C::COL_S + 64 * h, sr);
      tmem_ld32(tl + C::COL_S + 64 * h + 32, sr + 32);
      tmem_ld_wait();
      reg_fence32(sr);
      reg_fence32(sr + 32);
      probabilities64<false>(sr, nullptr, sl2, nullptr, nl2, 0, false);
      if (masked) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= vis) sr[c] = 0u;
      }
      if (!warp_wait(&bar[C::B_DPF + h], j & 1, wc)) { ok = false; break; }
      tc_fence_after();
      uint32_t w[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t dr[32];
        tmem_ld32(tl + C::COL_DP + 64 * h + 32 * half, dr);
        tmem_ld_wait();
        reg_fence32(dr);
        dscores32<false>(sr + 32 * half, dr, w + 16 * half, nullptr, nd);
      }
      // dS (bf16) over this group's first 32 S columns, already read.
      tmem_st32(tl + C::COL_S + 64 * h, w);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar[C::B_DSF + h]);
    }

    // ------------------------------------------------------------ dQ out
    // Group h writes columns [h D/2, (h + 1) D/2) of its row.
    if (ok && (nkb == 0 || warp_wait(&bar[C::B_ACC], 0, wc))) {
      tc_fence_after();
      __nv_bfloat16* dst_row = p.dQ + ((size_t)bh * p.n + q) * D + h * (D / 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t o[32];
        if (nkb > 0) {
          tmem_ld32(tl + C::COL_DQ + h * (D / 2) + 32 * c, o);
          tmem_ld_wait();
          reg_fence32(o);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack_bf16(__uint_as_float(o[2 * e]) * p.scale,
                           __uint_as_float(o[2 * e + 1]) * p.scale);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(dst_row + 32 * c);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
          dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
        }
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

// ================================================================== preprocess
// Each warp step covers RPW consecutive workspace rows (head bh, query q <
// n_pad), LPR lanes per row, one 16-byte load of O and of dO per lane:
// -D = -sum_c dO*O and -L * log2(e). Rows q >= n get -D = 0 and -inf, so that
// recomputed probabilities there are exactly 0.
template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const __nv_bfloat16* __restrict__ O,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         const float* __restrict__ L,
                                                         float* __restrict__ ws_nD,
                                                         float* __restrict__ ws_nL2, int n,
                                                         int n_pad, long long rows) {
  constexpr int LPR = D / 8;     // lanes per row (8 bf16 per lane)
  constexpr int RPW = 32 / LPR;  // rows per warp step
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
      ws_nD[r] = -acc;
      ws_nL2[r] = (q < n) ? -L[(size_t)bh * n + q] * kLog2e : -INFINITY;
    }
  }
}

// The dK, dV and dQ passes in one launch: n_kv CTAs of the first, then n_dq of
// the second, whose heavy blocks fill the SMs the first pass's tail leaves idle.
template <int D>
__global__ void __launch_bounds__(384, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
               const __grid_constant__ CUtensorMap tmNL2, const __grid_constant__ CUtensorMap tmND,
               const KvParams kp, const DqParams qp, int n_kv, int n_dq) {
  const int b = blockIdx.x;
  if (b < n_kv)
    dkdv_cta<D>(tmQ, tmK, tmV, tmdO, tmNL2, tmND, kp, b);
  else
    dq_cta<D>(tmQ, tmK, tmV, tmdO, qp, b - n_kv);
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs& a, bool with_kv, bool with_dq, cudaStream_t stream) {
  using KC = KvCfg<D>;
  using QC = QCfg<D>;
  static_assert(KC::BQ == QC::BM && KC::BN == QC::BN, "the passes share the tensor maps");
  CUtensorMap mq, mk, mv, mdo, ml2, md;
  if (make_bf16_head_map(&mq, a.Q, a.BH, a.n, D, KC::BQ) != CUDA_SUCCESS ||
      make_bf16_head_map(&mk, a.K, a.BH, a.m, D, KC::BN) != CUDA_SUCCESS ||
      make_bf16_head_map(&mv, a.V, a.BH, a.m, D, KC::BN) != CUDA_SUCCESS ||
      make_bf16_head_map(&mdo, a.dO, a.BH, a.n, D, KC::BQ) != CUDA_SUCCESS ||
      make_f32_row_map(&ml2, a.ws_nL2, a.BH, a.n_pad, KC::BQ) != CUDA_SUCCESS ||
      make_f32_row_map(&md, a.ws_nD, a.BH, a.n_pad, KC::BQ) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  KvParams kp;
  kp.dK = static_cast<__nv_bfloat16*>(a.dK);
  kp.dV = static_cast<__nv_bfloat16*>(a.dV);
  kp.n = a.n;
  kp.m = a.m;
  kp.n_pad = a.n_pad;
  kp.BH = a.BH;
  kp.causal = a.causal;
  kp.scale = a.scale;
  kp.scale_log2 = a.scale * kLog2e;
  kp.ktiles = ceil_div(a.m, KC::BN);
  kp.group = heads_per_group(a.BH, kp.ktiles);
  DqParams qp;
  qp.dQ = static_cast<__nv_bfloat16*>(a.dQ);
  qp.nD = a.ws_nD;
  qp.nL2 = a.ws_nL2;
  qp.n = a.n;
  qp.m = a.m;
  qp.n_pad = a.n_pad;
  qp.BH = a.BH;
  qp.causal = a.causal;
  qp.scale = a.scale;
  qp.scale_log2 = a.scale * kLog2e;
  qp.qtiles = ceil_div(a.n, QC::BM);
  qp.group = heads_per_group(a.BH, qp.qtiles);
  const int n_kv = with_kv ? kp.ktiles * a.BH : 0;
  const int n_dq = with_dq ? qp.qtiles * a.BH : 0;
  constexpr int smem = KC::SMEM > QC::SMEM ? KC::SMEM : QC::SMEM;
  cudaError_t e =
      cudaFuncSetAttribute(bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  bwd_kernel<D><<<(unsigned)(n_kv + n_dq), KC::THREADS, smem, stream>>>(mq, mk, mv, mdo, ml2, md,
                                                                        kp, qp, n_kv, n_dq);
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
        a.ws_nD, a.ws_nL2, a.n, a.n_pad, rows);
  else
    preprocess_kernel<64><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(a.O), static_cast<const __nv_bfloat16*>(a.dO), a.L,
        a.ws_nD, a.ws_nL2, a.n, a.n_pad, rows);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const BwdArgs& a, cudaStream_t s) {
  return a.d == 128 ? launch_bwd_d<128>(a, true, false, s) : launch_bwd_d<64>(a, true, false, s);
}

cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t s) {
  return a.d == 128 ? launch_bwd_d<128>(a, false, true, s) : launch_bwd_d<64>(a, false, true, s);
}

cudaError_t launch_bwd_main(const BwdArgs& a, cudaStream_t s) {
  return a.d == 128 ? launch_bwd_d<128>(a, true, true, s) : launch_bwd_d<64>(a, true, true, s);
}

cudaError_t bwd_read_status(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_bwd_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(unsigned int));
}

}  // namespace fa
