// Backward pass of exact attention, FlashAttention-2 recompute form
// ("05_flash_attention.py", flash_attention_backward):
//   D = rowsum(dO o O); P = exp(S - L) rebuilt from the saved L;
//   dV = P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = dS K * scale,
//   dK = dS^T Q * scale; blocks wholly above the diagonal are skipped under
//   causal masking.
//
// Two kernels on one stream:
//   preprocess  -D and -L * log2(e) (-inf past n) into the workspace; memory bound.
//   bwd_kernel  the gradients, persistent: one CTA per SM runs its share of the
//               dK/dV pass (blocks = (128-key block, head)) and then of the dQ pass
//               (blocks = (128-query block, head)); the blocks are dealt in
//               snake order over lists that put the heaviest blocks first within
//               a group of heads.
//   dK/dV pass  K is moved into TMEM (the A operand of S^T); V stays in shared
//               memory (two buffers); Q, dO, -L2 and -D of 64 queries at a time
//               stream through a ring of half-block slots, which also carries the
//               next block's K. Per 64-query half u (key index on the TMEM lane):
//                 S^T = K Q_u^T (TS)       dP^T = V dO_u^T (SS)
//                 dV += P^T dO_u (TS)      dK  += dS^T Q_u (TS)
//               with P^T and dS^T written by the compute warps as bf16 over the
//               S^T columns they have read; S^T alternates between two TMEM regions
//               so S^T of half u+2 forms while half u is processed. dK and dV
//               accumulate in TMEM and are written once per block.
//   dQ pass     Q and dO are moved into TMEM (A operands of S and dP); K and V
//               stream through a ring. Each 128-key block is taken in halves of 64
//               keys, one per compute group (ping-pong):
//                 S_h = Q K_h^T, dP_h = dO V_h^T, dQ += dS_h K_h   (TS)
//               dQ accumulates in TMEM and is written once, scaled, as bf16.
//   Epilogues leave TMEM through per-warp swizzled staging in shared memory and
//   one TMA store per 32 x 32 piece, while the next block's first products run.
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
// Roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer (whole warp, one
// elected lane issues), warps 4..11 two compute warpgroups; thread = TMEM lane
// (key row in the dK/dV pass, query row in the dQ pass).
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
// One CTA walks a list of key blocks (persistent). For each block, K is moved into
// TMEM (the A operand of S^T) and V stays in shared memory (two buffers,
// alternating between blocks). The query loop runs in halves of 64 queries; both
// compute groups work on every half (32 queries each). S^T of consecutive halves
// alternates between two TMEM regions and dP^T has a region of its own, so S^T of
// half u+2 is formed while half u is processed:
//   S^T_0 dP^T_0 S^T_1 | dV_0 dP^T_1 dK_0 S^T_2 | dV_1 dP^T_2 dK_1 S^T_3 | ...
// Q, dO, -L2 and -D stream through a ring of half-block slots (64 queries each);
// the next key block's K comes through the same ring (one slot) and its V into the
// other V buffer while the current block runs; dK, dV are written out while the
// next block's first products run.
template <int D>
struct KvCfg {
  static constexpr int BN = 128;      // keys per block = TMEM lanes
  static constexpr int BQ = 128;      // queries per block (two halves of 64)
  static constexpr int KCH = D / 64;  // 128-byte column chunks of a row
  static constexpr int CHUNK = 128 * 128;
  static constexpr int TILE = KCH * CHUNK;       // 128 rows of K or V
  static constexpr int HCHUNK = 64 * 128;        // one chunk of a 64-row tile
  static constexpr int HTILE = KCH * HCHUNK;     // 64 rows of Q or dO
  // Ring of half-block slots: Q (HTILE) then dO (HTILE) of 64 queries, or the next
  // key block's K (TILE = 2 HTILE) in one slot.
  static constexpr int SLOT = 2 * HTILE;
  static constexpr int STAGES = (D == 128) ? 4 : 8;
  static constexpr int OFF_V = 0;                // two V buffers
  static constexpr int OFF_R = 2 * TILE;         // the ring
  static constexpr int OFF_NL2 = OFF_R + STAGES * SLOT;      // [STAGES][64] fp32
  static constexpr int OFF_ND = OFF_NL2 + STAGES * 64 * 4;   // [STAGES][64] fp32
  // dK / dV staging for the TMA stores, one area per compute warp
  static constexpr int OFF_EPI = (OFF_ND + STAGES * 64 * 4 + 1023) / 1024 * 1024;
  static constexpr int OFF_BAR = OFF_EPI + 8 * kStoreStageBytes;
  // barrier slots
  static constexpr int B_QF = 0;              // + slot: the slot's copies landed
  static constexpr int B_QE = STAGES;         // + slot: the slot may be refilled
  static constexpr int B_VF = 2 * STAGES;     // + buffer: V landed
  static constexpr int B_IN = B_VF + 2;       // K in TMEM (256 arrivals)
  static constexpr int B_SF = B_IN + 1;       // + region: S^T in that region done
  static constexpr int B_DPF = B_SF + 2;      // dP^T of the current half done
  // + (u & 1): P^T of half u in TMEM (256 arrivals). Two slots: P^T of half u+1
  // needs only S^T_{u+1}, which is issued before the MMA warp waits for P^T_u,
  // so one barrier could complete twice before that wait and hide its phase.
  static constexpr int B_PF = B_SF + 3;
  static constexpr int B_DSF = B_SF + 5;      // dS^T in TMEM (256 arrivals)
  static constexpr int B_ACC = B_SF + 6;      // + (block & 1): dK, dV final
  static constexpr int B_EPI = B_SF + 8;      // dK, dV read out of TMEM (256 arrivals)
  static constexpr int B_DRAIN = B_SF + 9;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8;
  // TMEM columns: K as bf16 pairs, two 64-column S^T regions, the dP^T region,
  // dV, dK. Group w keeps P^T over [32w, 32w + 16) and dS^T over
  // [32w + 16, 32w + 32) of the half's S^T region.
  static constexpr uint32_t COL_K = 0;
  static constexpr uint32_t COL_S = 64;   // regions at 64 and 128
  static constexpr uint32_t COL_DP = 192;
  static constexpr uint32_t COL_DV = 256;
  static constexpr uint32_t COL_DK = 256 + D;
  static constexpr int THREADS = 384;
  static constexpr int COMPUTE_THREADS = 256;
  static_assert(COL_DK + D <= 512, "TMEM budget");
  static_assert(SMEM <= 232448 - 64, "shared memory budget");
  static_assert(SLOT == TILE, "a slot holds one K tile");
};

struct KvParams {
  __nv_bfloat16 *dK, *dV;
  int n, m, n_pad, BH, causal, ktiles, group;
  int d;  // head dimension (<= D; the tiles' columns past d are zero)
  float scale, scale_log2;
};


// TMEM column of k-step kk (16 queries) of the P^T (part 0) or dS^T (part 1)
// operand of a half stored in region `reg`.
__device__ __forceinline__ uint32_t half_operand_col(uint32_t reg, int part, int kk) {
  return reg + (uint32_t)((kk >> 1) * 32 + part * 16 + (kk & 1) * 8);
}

// Copies row `r` of a 128-row, 128-byte-swizzled bf16 tile (D / 64 chunks) into
// TMEM columns [col, col + D/2) of this thread's lane: piece j of a chunk row sits
// at j ^ (r % 8).
template <int D>
__device__ __forceinline__ void tile_row_to_tmem(const uint8_t* tile, int r, uint32_t col) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    uint32_t v[32];
    const uint8_t* row = tile + c * (128 * 128) + r * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint4 x = *reinterpret_cast<const uint4*>(row + ((j ^ (r & 7)) << 4));
      v[4 * j] = x.x;
      v[4 * j + 1] = x.y;
      v[4 * j + 2] = x.z;
      v[4 * j + 3] = x.w;
    }
    tmem_st32(col + 32 * c, v);
  }
  tmem_st_wait();
}

// Key blocks snake_item(r0 + t, c, P) (t < count) in launch order, by CTA c.
template <int D>
__device__ __forceinline__ void dkdv_run(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                         const CUtensorMap& tmV, const CUtensorMap& tmdO,
                                         const CUtensorMap& tmNL2, const CUtensorMap& tmND,
                                         const CUtensorMap& tmdK, const CUtensorMap& tmdV,
                                         const KvParams& p, uint8_t* smem, uint32_t tmem,
                                         int r0, int c, int P, int count, const WaitCtx& wc) {
  using C = KvCfg<D>;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bar[C::B_QF + s], 1);
      mbar_init(&bar[C::B_QE + s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar[C::B_VF + b], 1);
      mbar_init(&bar[C::B_SF + b], 1);
      mbar_init(&bar[C::B_PF + b], C::COMPUTE_THREADS);
      mbar_init(&bar[C::B_ACC + b], 1);
    }
    mbar_init(&bar[C::B_IN], C::COMPUTE_THREADS);
    mbar_init(&bar[C::B_DPF], 1);
    mbar_init(&bar[C::B_DSF], C::COMPUTE_THREADS);
    mbar_init(&bar[C::B_EPI], C::COMPUTE_THREADS);
    mbar_init(&bar[C::B_DRAIN], 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Block t: first key, head, first query block and number of query blocks. Key
  // blocks near 0 carry the most work under causal masking: the launch order puts
  // rank 0 first, heads a group at a time so that the blocks in flight share L2.
  auto block = [&](int t, int& ks, int& bh, int& i0, int& nq) {
    int ktile;
    grouped_tile(snake_item(r0 + t, c, P), p.BH, p.ktiles, p.group, ktile, bh);
    ks = ktile * C::BN;
    i0 = p.causal ? ks / C::BQ : 0;  // first query block with a query q >= ks
    nq = max(0, (p.n + C::BQ - 1) / C::BQ - i0);
  };
  // Ring uses: per block one for its K, then one per query block. `ru` counts them,
  // `hu` the halves and `at` the blocks with work, identically in every role.

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      tma_prefetch_map(&tmdO);
      int ru = 0, at = 0;
      bool ok = true;
      for (int t = 0; ok && t < count; ++t) {
        int ks, bh, i0, nq;
        block(t, ks, bh, i0, nq);
        if (nq == 0) continue;
        // V into buffer at % 2, free once block at-2's products are done
        const int vb = at & 1;
        if (at >= 2 && !mbar_wait(&bar[C::B_ACC + vb], ((at >> 1) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(&bar[C::B_VF + vb], C::TILE);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(smem + C::OFF_V + vb * C::TILE + c * C::CHUNK, &tmV, &bar[C::B_VF + vb],
                      c * 64, ks, bh);
        for (int u = -1; u < 2 * nq; ++u, ++ru) {
          const int s = ru % C::STAGES;
          if (ru >= C::STAGES &&
              !mbar_wait(&bar[C::B_QE + s], ((ru / C::STAGES) & 1) ^ 1, wc)) {
            ok = false;
            break;
          }
          uint64_t* f = &bar[C::B_QF + s];
          uint8_t* slot = smem + C::OFF_R + s * C::SLOT;
          if (u < 0) {  // this block's K
            mbar_arrive_expect_tx(f, C::TILE);
#pragma unroll
            for (int c = 0; c < C::KCH; ++c)
              tma_load_3d(slot + c * C::CHUNK, &tmK, f, c * 64, ks, bh);
          } else {  // queries [q, q + 64) of half u: Q, dO, -L2, -D
            const int q = (i0 + (u >> 1)) * C::BQ + 64 * (u & 1);
            mbar_arrive_expect_tx(f, 2 * C::HTILE + 2 * 64 * 4);
#pragma unroll
            for (int c = 0; c < C::KCH; ++c) {
              tma_load_3d(slot + c * C::HCHUNK, &tmQ, f, c * 64, q, bh);
              tma_load_3d(slot + C::HTILE + c * C::HCHUNK, &tmdO, f, c * 64, q, bh);
            }
            tma_load_2d(smem + C::OFF_NL2 + s * 64 * 4, &tmNL2, f, q, bh);
            tma_load_2d(smem + C::OFF_ND + s * 64 * 4, &tmND, f, q, bh);
          }
        }
        if (ok) ++at;
      }
      // Let every copy this thread issued land before the run ends.
      for (int r = max(0, ru - C::STAGES); r < ru; ++r)
        drain_wait(&bar[C::B_QF + r % C::STAGES], (r / C::STAGES) & 1);
      for (int a = max(0, at - 2); a < at; ++a) drain_wait(&bar[C::B_VF + (a & 1)], (a >> 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false, false);
    constexpr uint32_t kIdescG = idesc_bf16_f32(128, D, false, true);
    auto sreg = [&](int u) { return tmem + C::COL_S + 64u * (uint32_t)(u & 1); };
    int ru = 0, hu = 0, at = 0;
    bool ok = true;
    for (int t = 0; ok && t < count; ++t) {
      int ks, bh, i0, nq;
      block(t, ks, bh, i0, nq);
      if (nq == 0) continue;
      const int nu = 2 * nq;
      const int rb = ru + 1;  // ring use of half 0
      // K is in TMEM (its slot may be refilled), V landed, halves 0 and 1 landed
      if (!warp_wait(&bar[C::B_IN], at & 1, wc)) break;
      if (lane == 0) mbar_arrive(&bar[C::B_QE + ru % C::STAGES]);
      if (!warp_wait(&bar[C::B_VF + (at & 1)], (at >> 1) & 1, wc)) break;
      if (!warp_wait(&bar[C::B_QF + rb % C::STAGES], (rb / C::STAGES) & 1, wc)) break;
      if (!warp_wait(&bar[C::B_QF + (rb + 1) % C::STAGES], ((rb + 1) / C::STAGES) & 1, wc)) break;
      tc_fence_after();
      const uint64_t v_k = sdesc_sw128(smem_u32(smem + C::OFF_V + (at & 1) * C::TILE), 16, 1024);
      // Q (part 0) or dO (part 1) of half u in its slot
      auto half_rows = [&](int part, int u) {
        return smem_u32(smem + C::OFF_R + ((rb + u) % C::STAGES) * C::SLOT + part * C::HTILE);
      };
      // S^T_u = K Q_u^T (TS, N = 64) into its region. The region still holds
      // P^T / dS^T of half u-2, read by dV / dK of that half, which this thread
      // issued earlier: tcgen05.mma instructions of one thread execute in order.
      auto scores = [&](int u) {
        const uint64_t b_k = sdesc_sw128(half_rows(0, u), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::HCHUNK + (kk & 3) * 32;
          umma_ts_w(sreg(u), tmem + C::COL_K + kk * 8, sdesc_add(b_k, off), kIdescS, kk > 0);
        }
        umma_commit_w(&bar[C::B_SF + (u & 1)]);
      };
      // dP^T_u = V dO_u^T (SS, N = 64). The compute groups read dP^T_{u-1}
      // before signalling dS^T_{u-1}.
      auto dscores = [&](int u) {
        const uint64_t b_k = sdesc_sw128(half_rows(1, u), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          umma_ss_w(tmem + C::COL_DP, sdesc_add(v_k, (kk >> 2) * C::CHUNK + (kk & 3) * 32),
                    sdesc_add(b_k, (kk >> 2) * C::HCHUNK + (kk & 3) * 32), kIdescS, kk > 0);
        }
        umma_commit_w(&bar[C::B_DPF]);
      };
      // dV += P^T_u dO_u (part 0) or dK += dS^T_u Q_u (part 1), TS
      auto grads = [&](int u, int part) {
        const uint64_t b_mn = sdesc_sw128(half_rows(part == 0 ? 1 : 0, u), C::HCHUNK, 1024);
        const uint32_t dcol = tmem + (part == 0 ? C::COL_DV : C::COL_DK);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_ts_w(dcol, half_operand_col(sreg(u), part, kk), sdesc_add(b_mn, kk * 2048),
                    kIdescG, (u > 0 || kk > 0) ? 1u : 0u);
      };
      scores(0);
      dscores(0);
      scores(1);
      for (int u = 0; ok && u < nu; ++u) {
        if (!warp_wait(&bar[C::B_PF + (u & 1)], ((hu >> 1) + (u >> 1)) & 1, wc)) { ok = false; break; }
        // the previous block's dK, dV have been read out of TMEM
        if (u == 0 && at >= 1 && !warp_wait(&bar[C::B_EPI], (at - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        grads(u, 0);
        if (!warp_wait(&bar[C::B_DSF], (hu + u) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        if (u + 1 < nu) dscores(u + 1);
        grads(u, 1);
        umma_commit_w(&bar[C::B_QE + (rb + u) % C::STAGES]);  // last reader of half u's slot
        if (u + 2 < nu) {
          const int r2 = rb + u + 2;
          if (!warp_wait(&bar[C::B_QF + r2 % C::STAGES], (r2 / C::STAGES) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          scores(u + 2);
        }
      }
      if (!ok) break;
      umma_commit_w(&bar[C::B_ACC + (at & 1)]);
      ru += 1 + 2 * nq;
      hu += nu;
      ++at;
    }
    umma_commit_w(&bar[C::B_DRAIN]);
    drain_wait(&bar[C::B_DRAIN], 0);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ P^T, dS^T
    const int w = (warp - 4) >> 2;               // compute group
    const int krow = (warp & 3) * 32 + lane;     // key row = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float sl2 = p.scale_log2;
    // Group 0 writes dV rows, group 1 dK rows (all D columns of its key row).
    const uint32_t acc_col = tl + (w == 0 ? C::COL_DV : C::COL_DK);
    const float acc_mul = w == 0 ? 1.f : p.scale;
    __nv_bfloat16* const out = w == 0 ? p.dV : p.dK;
    const CUtensorMap* const out_map = w == 0 ? &tmdV : &tmdK;
    uint8_t* const stage = smem + C::OFF_EPI + (warp - 4) * kStoreStageBytes;
    int ru = 0, hu = 0, at = 0;
    int prev_bh = 0, prev_ks = 0;
    bool ok = true;
    // dK / dV of block a (head pbh, keys from pks) out of TMEM
    auto epilogue = [&](int a, int pbh, int pks) {
      if (!warp_wait(&bar[C::B_ACC + (a & 1)], (a >> 1) & 1, wc)) return false;
      tc_fence_after();
      tmem_rows_store<D>(acc_col, acc_mul, stage, out_map, 0, pks + (warp & 3) * 32, p.m, pbh,
                         p.d);
      tc_fence_before();
      mbar_arrive(&bar[C::B_EPI]);
      return true;
    };
    for (int t = 0; ok && t < count; ++t) {
      int ks, bh, i0, nq;
      block(t, ks, bh, i0, nq);
      const int kg = ks + krow;
      const bool key_ok = kg < p.m;
      if (nq == 0) {  // no query sees these keys: dK = dV = 0
        if (key_ok) {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int c = 0; c < D / 8; ++c)
            if (8 * c < p.d) reinterpret_cast<uint4*>(out + ((size_t)bh * p.m + kg) * p.d)[c] = z;
        }
        continue;
      }
      // K of this block into TMEM. The previous block's S^T products, the only
      // readers of these columns, are complete: both groups waited for all of them.
      if (w == 0) {
        const int s = ru % C::STAGES;
        if (!warp_wait(&bar[C::B_QF + s], (ru / C::STAGES) & 1, wc)) { ok = false; break; }
        tile_row_to_tmem<D>(smem + C::OFF_R + s * C::SLOT, krow, tl + C::COL_K);
        tc_fence_before();
      }
      mbar_arrive(&bar[C::B_IN]);
      // The previous block's dK, dV leave TMEM while this block's first products run.
      if (at >= 1 && !epilogue(at - 1, prev_bh, prev_ks)) { ok = false; break; }
      const int rb = ru + 1;
      for (int u = 0; ok && u < 2 * nq; ++u) {
        const int i = u >> 1, h = u & 1;
        const int s = (rb + u) % C::STAGES;
        const int c0 = 64 * h + 32 * w;            // first query column of this group
        const int q0 = (i0 + i) * C::BQ;
        if (!warp_wait(&bar[C::B_QF + s], ((rb + u) / C::STAGES) & 1, wc)) { ok = false; break; }
        if (!warp_wait(&bar[C::B_SF + h], ((hu >> 1) + (u >> 1)) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sr_col = tl + C::COL_S + 64u * (uint32_t)h + 32u * (uint32_t)w;
        const float* nl2 = reinterpret_cast<const float*>(smem + C::OFF_NL2 + s * 64 * 4) + 32 * w;
        const float* nd = reinterpret_cast<const float*>(smem + C::OFF_ND + s * 64 * 4) + 32 * w;
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
        if (!warp_wait(&bar[C::B_DPF], (hu + u) & 1, wc)) { ok = false; break; }
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
      prev_bh = bh;
      prev_ks = ks;
      ru += 1 + 2 * nq;
      hu += 2 * nq;
      ++at;
    }
    if (ok && at >= 1) epilogue(at - 1, prev_bh, prev_ks);
    if (lane == 0) bulk_wait_all();  // the stores have read their staging buffers
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0)
    for (int b = 0; b < C::NBAR; ++b) mbar_inval(&bar[b]);
}

// ================================================================== dQ
// One CTA walks a list of query blocks (persistent). For each block, Q and dO come
// through the K/V ring (one slot) and are moved into TMEM (the A operands of
// S = Q K^T and dP = dO V^T); K and V stream through the ring. Each 128-key block
// is taken in halves of 64 keys, one per compute group:
//   S_0 dP_0 S_1 dP_1 | dQ_0 S_0' dP_0' dQ_1 S_1' dP_1' | ...  (' = next key block)
// dQ accumulates in TMEM and is written once, scaled, as bf16, while the next query
// block's first products run.
template <int D>
struct QCfg {
  static constexpr int BM = 128;      // queries per block = TMEM lanes
  static constexpr int BN = 128;      // keys per step
  static constexpr int KCH = D / 64;
  static constexpr int CHUNK = 128 * 128;
  static constexpr int TILE = KCH * CHUNK;
  static constexpr int HALF_ROWS = 64 * 128;  // bytes of 64 rows of one 128-byte chunk
  static constexpr int STAGES = (D == 128) ? 3 : 4;
  static constexpr int OFF_K = 0;              // ring: K_j (or the next block's Q)
  static constexpr int OFF_V = STAGES * TILE;  // ring: V_j (or the next block's dO)
  static constexpr int OFF_EPI = 2 * STAGES * TILE;  // dQ staging, one area per compute warp
  static constexpr int OFF_BAR = OFF_EPI + 8 * kStoreStageBytes;
  static constexpr int B_KVF = 0;              // + slot: the slot's copies landed
  static constexpr int B_KVE = STAGES;         // + slot: the slot may be refilled
  static constexpr int B_IN = 2 * STAGES;      // Q and dO rows in TMEM (256 arrivals)
  // Per half h of the key block (two slots each):
  static constexpr int B_SF = B_IN + 1;        // + h: S_h done
  static constexpr int B_DPF = B_SF + 2;       // + h: dP_h done
  static constexpr int B_DSF = B_SF + 4;       // + h: dS_h in TMEM (128 arrivals)
  static constexpr int B_ACC = B_SF + 6;       // dQ final
  static constexpr int B_EPI = B_SF + 7;       // dQ read out of TMEM (256 arrivals)
  static constexpr int B_DRAIN = B_SF + 8;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8;
  // TMEM columns: Q and dO as bf16 pairs; for half h of the key block S_h at
  // COL_S + 64h (then dS_h as bf16 pairs over its first 32 columns) and dP_h at
  // COL_DP + 64h; dQ.
  static constexpr uint32_t COL_Q = 0;
  static constexpr uint32_t COL_DO = D / 2;
  static constexpr uint32_t COL_S = D;
  static constexpr uint32_t COL_DP = D + 128;
  static constexpr uint32_t COL_DQ = D + 256;
  static constexpr int THREADS = 384;
  static constexpr int COMPUTE_THREADS = 256;
  static constexpr int GROUP_THREADS = 128;
  static_assert(COL_DQ + D <= 512, "TMEM budget");
  static_assert(SMEM <= 232448 - 64, "shared memory budget");
};

struct DqParams {
  __nv_bfloat16* dQ;
  const float *nD, *nL2;
  int n, m, n_pad, BH, causal, qtiles, group;
  int d;  // head dimension (<= D; the tiles' columns past d are zero)
  float scale, scale_log2;
};

// Query blocks snake_item(r0 + t, c, P) - skip (t < count) in launch order, by CTA c.
template <int D>
__device__ __forceinline__ void dq_run(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                       const CUtensorMap& tmV, const CUtensorMap& tmdO,
                                       const CUtensorMap& tmdQ, const DqParams& p, uint8_t* smem,
                                       uint32_t tmem, int r0,
                                       int c, int P, int skip, int count, const WaitCtx& wc) {
  using C = QCfg<D>;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bar[C::B_KVF + s], 1);
      mbar_init(&bar[C::B_KVE + s], 1);
    }
    mbar_init(&bar[C::B_IN], C::COMPUTE_THREADS);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&bar[C::B_SF + h], 1);
      mbar_init(&bar[C::B_DPF + h], 1);
      mbar_init(&bar[C::B_DSF + h], C::GROUP_THREADS);
    }
    mbar_init(&bar[C::B_ACC], 1);
    mbar_init(&bar[C::B_EPI], C::COMPUTE_THREADS);
    mbar_init(&bar[C::B_DRAIN], 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Block t: head, first query, number of key blocks. Under causal masking the last
  // query blocks see the most keys: the launch order puts them first.
  auto block = [&](int t, int& bh, int& q0, int& nkb) {
    int rank;
    grouped_tile(snake_item(r0 + t, c, P) - skip, p.BH, p.qtiles, p.group, rank, bh);
    q0 = (p.causal ? p.qtiles - 1 - rank : rank) * C::BM;
    nkb = (p.m + C::BN - 1) / C::BN;
    if (p.causal) nkb = min(nkb, min(q0 + C::BM - 1, p.n - 1) / C::BN + 1);  // keys k <= q
  };
  // Ring uses: per block one for its Q and dO, then one per key block. `ru` counts
  // them, `gb` the key blocks and `at` the query blocks with work, in every role.

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      tma_prefetch_map(&tmdO);
      int ru = 0;
      bool ok = true;
      for (int t = 0; ok && t < count; ++t) {
        int bh, q0, nkb;
        block(t, bh, q0, nkb);
        if (nkb == 0) continue;
        for (int j = -1; j < nkb; ++j, ++ru) {
          const int s = ru % C::STAGES;
          if (ru >= C::STAGES &&
              !mbar_wait(&bar[C::B_KVE + s], ((ru / C::STAGES) & 1) ^ 1, wc)) {
            ok = false;
            break;
          }
          uint64_t* f = &bar[C::B_KVF + s];
          mbar_arrive_expect_tx(f, 2 * C::TILE);
          uint8_t* kb = smem + C::OFF_K + s * C::TILE;
          uint8_t* vb = smem + C::OFF_V + s * C::TILE;
#pragma unroll
          for (int c = 0; c < C::KCH; ++c) {
            if (j < 0) {  // this block's Q and dO (64-row boxes: rows q0 and q0 + 64)
              tma_load_3d(kb + c * C::CHUNK, &tmQ, f, c * 64, q0, bh);
              tma_load_3d(kb + c * C::CHUNK + C::HALF_ROWS, &tmQ, f, c * 64, q0 + 64, bh);
              tma_load_3d(vb + c * C::CHUNK, &tmdO, f, c * 64, q0, bh);
              tma_load_3d(vb + c * C::CHUNK + C::HALF_ROWS, &tmdO, f, c * 64, q0 + 64, bh);
            } else {
              tma_load_3d(kb + c * C::CHUNK, &tmK, f, c * 64, j * C::BN, bh);
              tma_load_3d(vb + c * C::CHUNK, &tmV, f, c * 64, j * C::BN, bh);
            }
          }
        }
      }
      for (int r = max(0, ru - C::STAGES); r < ru; ++r)
        drain_wait(&bar[C::B_KVF + r % C::STAGES], (r / C::STAGES) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false, false);
    constexpr uint32_t kIdescQ = idesc_bf16_f32(128, D, false, true);
    int ru = 0, gb = 0, at = 0;
    bool ok = true;
    for (int t = 0; ok && t < count; ++t) {
      int bh, q0, nkb;
      block(t, bh, q0, nkb);
      if (nkb == 0) continue;
      const int rb = ru + 1;  // ring use of key block 0
      // S_h = Q K_h^T and dP_h = dO V_h^T for half h of key block j (N = 64). The
      // S_h columns still hold dS_h of block j-1, read by dQ of block j-1 that
      // this thread issued earlier (in-order execution); group h signalled dS_h
      // of block j-1 only after reading S_h and dP_h of it.
      auto scores = [&](int j, int h) {
        const int s = (rb + j) % C::STAGES;
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
      // Q and dO are in TMEM (their slot may be refilled); key block 0 landed
      if (!warp_wait(&bar[C::B_IN], at & 1, wc)) break;
      if (lane == 0) mbar_arrive(&bar[C::B_KVE + ru % C::STAGES]);
      if (!warp_wait(&bar[C::B_KVF + rb % C::STAGES], (rb / C::STAGES) & 1, wc)) break;
      tc_fence_after();
      scores(0, 0);
      scores(0, 1);
      for (int j = 0; ok && j < nkb; ++j) {
        const int s = (rb + j) % C::STAGES;
        for (int h = 0; ok && h < 2; ++h) {
          // dQ += dS_h K_h
          if (!warp_wait(&bar[C::B_DSF + h], (gb + j) & 1, wc)) { ok = false; break; }
          // the previous query block's dQ has been read out of TMEM
          if (j == 0 && h == 0 && at >= 1 && !warp_wait(&bar[C::B_EPI], (at - 1) & 1, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t k_mn = sdesc_sw128(
              smem_u32(smem + C::OFF_K + s * C::TILE + h * C::HALF_ROWS), C::CHUNK, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ts_w(tmem + C::COL_DQ, tmem + C::COL_S + 64 * h + kk * 8,
                      sdesc_add(k_mn, kk * 2048), kIdescQ, (j > 0 || h > 0 || kk > 0) ? 1u : 0u);
          if (h == 1) umma_commit_w(&bar[C::B_KVE + s]);  // last reader of K_j, V_j
          if (j + 1 < nkb) {
            if (h == 0 && !warp_wait(&bar[C::B_KVF + (rb + j + 1) % C::STAGES],
                                     ((rb + j + 1) / C::STAGES) & 1, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
            scores(j + 1, h);
          }
        }
      }
      if (!ok) break;
      umma_commit_w(&bar[C::B_ACC]);
      ru += 1 + nkb;
      gb += nkb;
      ++at;
    }
    umma_commit_w(&bar[C::B_DRAIN]);
    drain_wait(&bar[C::B_DRAIN], 0);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ P, dS
    const int h = (warp - 4) >> 2;            // which half of the key columns
    const int r = (warp & 3) * 32 + lane;     // query row = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float sl2 = p.scale_log2;
    int ru = 0, gb = 0, at = 0;
    int prev_q = 0, prev_bh = 0;
    bool ok = true;
    uint8_t* const stage = smem + C::OFF_EPI + (warp - 4) * kStoreStageBytes;
    // dQ of block a (head pbh, first query pq0): group h writes columns
    // [h D/2, (h+1) D/2) of the warp's 32 rows
    auto epilogue = [&](int a, int pbh, int pq0) {
      if (!warp_wait(&bar[C::B_ACC], a & 1, wc)) return false;
      tc_fence_after();
      tmem_rows_store<D / 2>(tl + C::COL_DQ + h * (D / 2), p.scale, stage, &tmdQ, h * (D / 2),
                             pq0 + (warp & 3) * 32, p.n, pbh, p.d - h * (D / 2));
      tc_fence_before();
      mbar_arrive(&bar[C::B_EPI]);
      return true;
    };
    for (int t = 0; ok && t < count; ++t) {
      int bh, q0, nkb;
      block(t, bh, q0, nkb);
      const int q = q0 + r;
      if (nkb == 0) {  // no key visible (not reached for m >= 1): dQ = 0
        if (q < p.n) {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int c = 0; c < D / 16; ++c)
            if (h * (D / 2) + 8 * c < p.d)
              reinterpret_cast<uint4*>(p.dQ + ((size_t)bh * p.n + q) * p.d + h * (D / 2))[c] = z;
        }
        continue;
      }
      const size_t ws_row = (size_t)bh * p.n_pad + q;  // q < n_pad always
      const float nl2 = p.nL2[ws_row];
      const float nd = p.nD[ws_row];
      // Group 0 moves row r of Q into TMEM, group 1 row r of dO. The previous
      // block's S and dP products are the only readers of these columns. Group 1
      // has seen the last of them complete (dP_1 of the last key block). Group 0 has
      // seen its own, but Q is also read by S_1 of the last key block, issued after
      // a dQ product that waits for group 1: group 0 waits for that S_1 as well.
      {
        const int s = ru % C::STAGES;
        if (h == 0 && at >= 1) {
          if (!warp_wait(&bar[C::B_SF + 1], (gb - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after();
        }
        if (!warp_wait(&bar[C::B_KVF + s], (ru / C::STAGES) & 1, wc)) { ok = false; break; }
        tile_row_to_tmem<D>(smem + (h == 0 ? C::OFF_K : C::OFF_V) + s * C::TILE, r,
                            tl + (h == 0 ? C::COL_Q : C::COL_DO));
        tc_fence_before();
      }
      mbar_arrive(&bar[C::B_IN]);
      // The previous block's dQ leaves TMEM while this block's first products run.
      if (at >= 1 && !epilogue(at - 1, prev_bh, prev_q)) { ok = false; break; }
      for (int j = 0; j < nkb; ++j) {
        if (!warp_wait(&bar[C::B_SF + h], (gb + j) & 1, wc)) { ok = false; break; }
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
        if (!warp_wait(&bar[C::B_DPF + h], (gb + j) & 1, wc)) { ok = false; break; }
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
      prev_q = q0;
      prev_bh = bh;
      ru += 1 + nkb;
      gb += nkb;
      ++at;
    }
    if (ok && at >= 1) epilogue(at - 1, prev_bh, prev_q);
    if (lane == 0) bulk_wait_all();  // the stores have read their staging buffers
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0)
    for (int b = 0; b < C::NBAR; ++b) mbar_inval(&bar[b]);
}

// ================================================================== preprocess
// Each warp step covers RPW consecutive workspace rows (head bh, query q <
// n_pad), LPR lanes per row, one 16-byte load of O and of dO per lane:
// -D = -sum_c dO*O and -L * log2(e). Rows q >= n get -D = 0 and -inf, so that
// recomputed probabilities there are exactly 0. A warp takes U steps at a time
// and issues all their loads before any arithmetic (memory-level parallelism:
// the kernel is bound by reading O and dO from HBM).
template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const __nv_bfloat16* __restrict__ O,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         const float* __restrict__ L,
                                                         float* __restrict__ ws_nD,
                                                         float* __restrict__ ws_nL2, int n,
                                                         int n_pad, int d, long long rows) {
  constexpr int LPR = D / 8;     // lanes per row (8 bf16 per lane)
  constexpr int RPW = 32 / LPR;  // rows per warp step
  constexpr int U = 4;           // warp steps in flight
  const int lane = threadIdx.x & 31;
  const int sub = lane % LPR;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long base = ((long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RPW * U;
       base < rows; base += warps * RPW * U) {
    // base is a multiple of RPW * U, which divides n_pad: the U * RPW rows of this
    // iteration are queries q0 .. q0 + U * RPW - 1 of one head
    const long long bh = base / n_pad;
    const int q0 = (int)(base - bh * n_pad) + lane / LPR;
    const __nv_bfloat16* o_head = O + (size_t)bh * n * d;
    const __nv_bfloat16* do_head = dO + (size_t)bh * n * d;
    uint4 a[U], b[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = q0 + u * RPW;
      a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);  // zero products for rows and lanes past the data
      if (q < n && 8 * sub < d) {
        a[u] = reinterpret_cast<const uint4*>(o_head + (size_t)q * d)[sub];
        b[u] = reinterpret_cast<const uint4*>(do_head + (size_t)q * d)[sub];
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = q0 + u * RPW;
      float acc = bf16_lo(a[u].x) * bf16_lo(b[u].x) + bf16_hi(a[u].x) * bf16_hi(b[u].x) +
                  bf16_lo(a[u].y) * bf16_lo(b[u].y) + bf16_hi(a[u].y) * bf16_hi(b[u].y) +
                  bf16_lo(a[u].z) * bf16_lo(b[u].z) + bf16_hi(a[u].z) * bf16_hi(b[u].z) +
                  bf16_lo(a[u].w) * bf16_lo(b[u].w) + bf16_hi(a[u].w) * bf16_hi(b[u].w);
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (sub == 0) {
        const size_t r = (size_t)bh * n_pad + q;
        ws_nD[r] = -acc;
        ws_nL2[r] = (q < n) ? -L[(size_t)bh * n + q] * kLog2e : -INFINITY;
      }
    }
  }
}

// Shared memory of the gradient kernel: the larger of the two passes' layouts,
// then the TMEM address slot and the abort word.
template <int D>
struct BwdSmem {
  static constexpr int PASSES = KvCfg<D>::SMEM > QCfg<D>::SMEM ? KvCfg<D>::SMEM : QCfg<D>::SMEM;
  static constexpr int CTL = (PASSES + 7) / 8 * 8;
  static constexpr int BYTES = CTL + 8;
  static_assert(BYTES <= 232448, "shared memory budget");
};

// The gradient kernel: one CTA per SM (persistent). The n_kv key blocks and then
// the n_dq query blocks are dealt out in rounds of P = grid size items (CTA c takes
// snake_item(r, c, P) of round r), so that each CTA runs its share of the dK/dV
// pass and then of the dQ pass; the lists are in launch order (heaviest blocks
// first within a group of heads).
template <int D>
__global__ void __launch_bounds__(384, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
               const __grid_constant__ CUtensorMap tmNL2, const __grid_constant__ CUtensorMap tmND,
               const __grid_constant__ CUtensorMap tmdQ, const __grid_constant__ CUtensorMap tmdK,
               const __grid_constant__ CUtensorMap tmdV, const KvParams kp, const DqParams qp,
               int n_kv, int n_dq) {
  // No static shared memory: the dynamic region then starts on a 1024-byte
  // boundary, which the 128-byte swizzle of the tiles needs and which the layouts
  // assume (they leave no room to align by hand). A kernel that finds another
  // placement reports it and does nothing.
  extern __shared__ uint8_t smem_dyn[];
  if ((smem_u32(smem_dyn) & 1023u) != 0u) {
    if (threadIdx.x == 0) atomicOr(&g_bwd_status, kDeviceLayoutBit);
    return;
  }
  // align1024 is the identity here; it makes the base a run-time value. With the
  // base known at compile time the generated code ran about 10% slower on GB300.
  uint8_t* smem = align1024(smem_dyn);
  constexpr int kCtl = BwdSmem<D>::CTL;  // two words after both passes' layouts
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kCtl);
  uint32_t* abort_word = tmem_slot + 1;
  const WaitCtx wc{abort_word, &g_bwd_status};
  if (threadIdx.x == 0) *abort_word = 0u;
  if ((threadIdx.x >> 5) == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int P = gridDim.x, c = blockIdx.x;
  // Each list is dealt separately; the query blocks in reverse CTA order, so that
  // the CTAs left with one key block more get no query block more.
  int kv_rounds = 0, dq_rounds = 0;
  while (snake_item(kv_rounds, c, P) < n_kv) ++kv_rounds;
  while (snake_item(dq_rounds, P - 1 - c, P) < n_dq) ++dq_rounds;
  if (kv_rounds > 0)
    dkdv_run<D>(tmQ, tmK, tmV, tmdO, tmNL2, tmND, tmdK, tmdV, kp, smem, tmem, 0, c, P, kv_rounds, wc);
  if (dq_rounds > 0)
    dq_run<D>(tmQ, tmK, tmV, tmdO, tmdQ, qp, smem, tmem, 0, P - 1 - c, P, 0, dq_rounds, wc);

  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs& a, bool with_kv, bool with_dq, cudaStream_t stream) {
  using KC = KvCfg<D>;
  using QC = QCfg<D>;
  static_assert(KC::BQ == QC::BM && KC::BN == QC::BN, "the passes share the tensor maps");
  static_assert(KC::THREADS == QC::THREADS, "the passes share the launch");
  CUtensorMap mq, mk, mv, mdo, ml2, md, mdq, mdk, mdv;
  // Q and dO, -L2 and -D travel in 64-row pieces; K and V in 128-row tiles.
  // Rows of d values; the 64-column boxes read zeros past d.
  if (make_bf16_head_map(&mq, a.Q, a.BH, a.n, a.d, 64) != CUDA_SUCCESS ||
      make_bf16_head_map(&mk, a.K, a.BH, a.m, a.d, KC::BN) != CUDA_SUCCESS ||
      make_bf16_head_map(&mv, a.V, a.BH, a.m, a.d, KC::BN) != CUDA_SUCCESS ||
      make_bf16_head_map(&mdo, a.dO, a.BH, a.n, a.d, 64) != CUDA_SUCCESS ||
      make_f32_row_map(&ml2, a.ws_nL2, a.BH, a.n_pad, 64) != CUDA_SUCCESS ||
      make_f32_row_map(&md, a.ws_nD, a.BH, a.n_pad, 64) != CUDA_SUCCESS ||
      make_bf16_store_map(&mdq, a.dQ, a.BH, a.n, a.d) != CUDA_SUCCESS ||
      make_bf16_store_map(&mdk, a.dK, a.BH, a.m, a.d) != CUDA_SUCCESS ||
      make_bf16_store_map(&mdv, a.dV, a.BH, a.m, a.d) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  KvParams kp;
  kp.dK = static_cast<__nv_bfloat16*>(a.dK);
  kp.dV = static_cast<__nv_bfloat16*>(a.dV);
  kp.n = a.n;
  kp.m = a.m;
  kp.n_pad = a.n_pad;
  kp.BH = a.BH;
  kp.causal = a.causal;
  kp.d = a.d;
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
  qp.d = a.d;
  qp.scale = a.scale;
  qp.scale_log2 = a.scale * kLog2e;
  qp.qtiles = ceil_div(a.n, QC::BM);
  qp.group = heads_per_group(a.BH, qp.qtiles);
  const int n_kv = with_kv ? kp.ktiles * a.BH : 0;
  const int n_dq = with_dq ? qp.qtiles * a.BH : 0;
  constexpr int smem = BwdSmem<D>::BYTES;
  cudaError_t e =
      cudaFuncSetAttribute(bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = n_kv + n_dq < sms ? n_kv + n_dq : sms;
  bwd_kernel<D><<<(unsigned)grid, KC::THREADS, smem, stream>>>(mq, mk, mv, mdo, ml2, md, mdq, mdk,
                                                               mdv, kp, qp, n_kv, n_dq);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t s) {
  const long long rows = (long long)a.BH * a.n_pad;
  const bool wide = a.d > 64;
  // 4 warp steps of 2 (d > 64) or 4 rows per warp, 8 warps a block, at most one
  // full-occupancy wave (8 blocks of 256 threads per SM); grid-stride beyond.
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long rows_per_block = (wide ? 2 : 4) * 4 * 8;
  long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  if (blocks > 8LL * sms) blocks = 8LL * sms;
  const int grid = (int)(blocks < 1 ? 1 : blocks);
  if (wide)
    preprocess_kernel<128><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(a.O), static_cast<const __nv_bfloat16*>(a.dO), a.L,
        a.ws_nD, a.ws_nL2, a.n, a.n_pad, a.d, rows);
  else
    preprocess_kernel<64><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(a.O), static_cast<const __nv_bfloat16*>(a.dO), a.L,
        a.ws_nD, a.ws_nL2, a.n, a.n_pad, a.d, rows);
  return cudaGetLastError();
}

// Head dimensions up to 64 run the 64-column kernels, larger ones the 128-column
// kernels (columns past d read as zeros).
cudaError_t launch_bwd_dkdv(const BwdArgs& a, cudaStream_t s) {
  return a.d > 64 ? launch_bwd_d<128>(a, true, false, s) : launch_bwd_d<64>(a, true, false, s);
}

cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t s) {
  return a.d > 64 ? launch_bwd_d<128>(a, false, true, s) : launch_bwd_d<64>(a, false, true, s);
}

cudaError_t launch_bwd_main(const BwdArgs& a, cudaStream_t s) {
  return a.d > 64 ? launch_bwd_d<128>(a, true, true, s) : launch_bwd_d<64>(a, true, true, s);
}

cudaError_t bwd_read_status(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_bwd_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(unsigned int));
}

}  // namespace fa
