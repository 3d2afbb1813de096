// Forward pass of exact attention: O = softmax(Q K^T * scale) V and the
// natural-log logsumexp L, two 128-row query tiles per CTA.
//
// Method: "05_flash_attention.py", flash_attention_forward. For each query
// tile the key/value blocks are visited left to right; per row the kernel
// keeps a reference maximum m and the exponential sum l taken relative to it,
// forms P = exp(S - m), and adds P V to the output accumulator; whenever m
// moves, O and l are rescaled by exp(m_old - m_new). At the end O = O / l and
// L = m + log l. Under causal masking key blocks wholly to the right of a
// tile's last query are never visited, and the diagonal block masks k > q.
// The reference maximum is moved only when a row maximum exceeds it by more
// than 8 (base 2): until then P stays below 2^8 and O, l keep their common
// reference, so the result is the same up to rounding while most blocks need
// no rescaling of O.
//
// GB300 mapping (one persistent CTA per SM, 384 threads). The work items are
// (pair of 128-row query tiles, head); CTA c takes items c, 2P - 1 - c, 2P + c, ...
// of the launch-order list (P CTAs, heaviest items first within a group of heads).
//   warp 0       TMA producer: per item both Q tiles (one ring slot), then K_j
//                and V_j (128 keys each) into a ring shared by the two tiles; the
//                ring runs on across items, so the next item's Q and first blocks
//                arrive while the current item finishes
//   warp 1       MMA issuer (whole warp, one elected lane issues). Keys are
//                taken in steps of 64 (half a loaded block): S_t = Q_t K^T (TS:
//                Q_t read from TMEM) and O_t += P_t V (TS: P_t read from TMEM),
//                the two tiles alternating; S_t of step k+1 is issued right
//                after O_t += P_t V of step k, over the same columns
//   warps 4..7   softmax of tile 0, warps 8..11 softmax of tile 1: thread r
//                first moves row r of Q_t into TMEM, then owns query row r of its
//                tile (= TMEM lane r): reads the 64 S columns of a step with
//                tcgen05.ld, masks, updates (m, l) in base 2 (exp2 via
//                ex2.approx), writes P as bf16 over the first 32 of them,
//                rescales its O row when m moved, moves row r of the next
//                item's Q_t into TMEM and then runs the epilogue (O_t leaves
//                TMEM while the next item's first S_t is formed). While one
//                tile's softmax runs, the tensor cores work on the other.
// TMEM (512 columns at d = 128): Q0, Q1 (d/2 each, bf16 pairs), S0, S1 (64
// each), O0, O1 (d each). Scores, probabilities and the accumulators never
// leave the SM.
#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

__device__ unsigned int g_fwd_status;

namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;  // base-2 units: P stays below 2^8

template <int D>
struct FwdCfg {
  static constexpr int BM = 128;                 // query rows per tile = TMEM lanes
  // Query tiles per CTA. TMEM would hold a third at d = 64, but with the deal's
  // wave quantization at the d = 64 workload sizes three tiles ran slower.
  static constexpr int TILES = 2;
  static constexpr int QUSES = (TILES + 1) / 2;  // ring uses holding an item's Q tiles
  static constexpr int SOFT0 = (TILES == 3) ? 2 : 4;  // first softmax warp
  static constexpr int BN = 128;                 // keys per loaded block (two halves of 64)
  static constexpr int KCH = D / 64;             // 128-byte column chunks per row
  static constexpr int CHUNK = 128 * 128;        // bytes of one chunk of a 128-row tile
  static constexpr int TILE = KCH * CHUNK;       // bytes of a Q, K or V tile
  static constexpr int HALF_ROWS = 64 * 128;     // bytes of 64 rows of one chunk
  // Ring of K/V blocks; its first use holds the two Q tiles until they are in TMEM.
  static constexpr int STAGES = (D == 128) ? 3 : 6;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = STAGES * TILE;
  static constexpr int OFF_EPI = 2 * STAGES * TILE;  // O staging, one area per softmax warp
  static constexpr int OFF_BAR = OFF_EPI + 4 * TILES * kStoreStageBytes;
  // barrier slots
  static constexpr int B_KVF = 0;                // + slot: the slot's copies landed
  static constexpr int B_KVE = STAGES;           // + slot: the slot may be refilled
  static constexpr int B_IN = 2 * STAGES;        // Q tiles in TMEM (256 arrivals)
  static constexpr int B_SF = B_IN + 1;          // + tile: S_t of the current step done
  static constexpr int B_PF = B_SF + TILES;      // + tile: P_t written (128 arrivals)
  static constexpr int B_PVD = B_PF + TILES;     // + tile: the tile's last O += P V done
                                                 // (for a tile with no steps: the item's
                                                 // products done)
  static constexpr int B_DRAIN = B_PVD + TILES;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
  // TMEM columns: Q_t as bf16 pairs (the A operand of S_t = Q_t K^T), S_t of one
  // 64-key step (then P_t as bf16 pairs over its first 32 columns), O_t.
  static constexpr uint32_t COL_Q = 0;           // + (D / 2) * tile
  static constexpr uint32_t COL_S = 128;         // + 64 * tile
  static constexpr uint32_t COL_O = 128 + 64 * TILES;  // + D * tile
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int THREADS = 32 * (SOFT0 + 4 * TILES);
  static_assert(COL_O + TILES * D <= TMEM_COLS, "TMEM budget");
  static_assert((D / 2) * TILES <= COL_S, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct FwdParams {
  __nv_bfloat16* O;
  float* L;
  int n, m, BH, causal, num_pairs, group;
  int d;             // head dimension (<= D; the tiles' columns past d are zero)
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

// 64-key steps a tile of rows [q0, q0 + 128) visits (0 if the tile is past n).
__device__ __forceinline__ int tile_steps(int q0, int n, int m, int causal) {
  if (q0 >= n) return 0;
  int nh = (m + 63) / 64;
  if (causal) nh = min(nh, (min(q0 + 127, n - 1)) / 64 + 1);  // keys k <= q
  return nh;
}

template <int D>
__global__ void __launch_bounds__(FwdCfg<D>::THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
               const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + C::NBAR);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const WaitCtx wc{abort_flag, &g_fwd_status};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Persistent: CTA c takes items snake_item(j, c, P), j = 0, 1, ... of the list of
  // (tile pair, head) items in launch order: heads a group at a time (their K/V
  // stay in L2 while the group runs), inside a group the heaviest tile pairs (the
  // last ones, under causal masking) first.
  const int P = gridDim.x, cta = blockIdx.x;
  const int n_items = p.num_pairs * p.BH;
  int n_mine = 0;
  while (snake_item(n_mine, cta, P) < n_items) ++n_mine;
  // Item j: first query, head and 64-key steps of each tile (tile 0 always has
  // some); returns the steps of the longest tile.
  auto item = [&](int j, int& qs, int& bh, int (&nht)[C::TILES]) {
    int grp;
    grouped_tile(snake_item(j, cta, P), p.BH, p.num_pairs, p.group, grp, bh);
    if (p.causal) grp = p.num_pairs - 1 - grp;
    qs = grp * (C::TILES * C::BM);
    int nh = 0;
#pragma unroll
    for (int t = 0; t < C::TILES; ++t) {
      nht[t] = tile_steps(qs + t * C::BM, p.n, p.m, p.causal);
      nh = max(nh, nht[t]);
    }
    return nh;
  };
  // Ring uses of item j: QUSES for its Q tiles (tiles 2u and 2u + 1 in the K and V
  // buffers of use u), then one per 128-key block of K, V. Every role counts them
  // (`ru`) and the steps of each tile identically.

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bar[C::B_KVF + s], 1);
      mbar_init(&bar[C::B_KVE + s], 1);
    }
    mbar_init(&bar[C::B_IN], 128 * C::TILES);
    for (int t = 0; t < C::TILES; ++t) {
      mbar_init(&bar[C::B_SF + t], 1);
      mbar_init(&bar[C::B_PF + t], 128);
      mbar_init(&bar[C::B_PVD + t], 1);
    }
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
    // Per item: the two Q tiles into the K and V buffers of one ring slot, then
    // K_j, V_j per block. The ring runs on across items, so the next item's Q and
    // first blocks load while the current item finishes.
    if (lane == 0 && n_mine > 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      int ru = 0;
      bool ok = true;
      for (int j = 0; ok && j < n_mine; ++j) {
        int qs, bh, nht[C::TILES];
        const int nkb = (item(j, qs, bh, nht) + 1) / 2;  // 128-key blocks
        for (int u = 0; u < C::QUSES + nkb; ++u, ++ru) {
          const int s = ru % C::STAGES;
          if (ru >= C::STAGES &&
              !mbar_wait(&bar[C::B_KVE + s], ((ru / C::STAGES) & 1) ^ 1, wc)) {
            ok = false;
            break;
          }
          uint64_t* f = &bar[C::B_KVF + s];
          // Q tiles 2u, 2u + 1 (the second only if the CTA has it), or K and V
          const bool q_use = u < C::QUSES;
          const bool two = !q_use || 2 * u + 1 < C::TILES;
          mbar_arrive_expect_tx(f, (two ? 2 : 1) * C::TILE);
#pragma unroll
          for (int c = 0; c < C::KCH; ++c) {
            uint8_t* kdst = smem + C::OFF_K + s * C::TILE + c * C::CHUNK;
            uint8_t* vdst = smem + C::OFF_V + s * C::TILE + c * C::CHUNK;
            if (q_use) {
              tma_load_3d(kdst, &tmQ, f, c * 64, qs + 2 * u * C::BM, bh);
              if (two) tma_load_3d(vdst, &tmQ, f, c * 64, qs + (2 * u + 1) * C::BM, bh);
            } else {
              tma_load_3d(kdst, &tmK, f, c * 64, (u - C::QUSES) * C::BN, bh);
              tma_load_3d(vdst, &tmV, f, c * 64, (u - C::QUSES) * C::BN, bh);
            }
          }
        }
      }
      // Let every copy this thread issued land before the CTA can exit.
      for (int r = max(0, ru - C::STAGES); r < ru; ++r)
        drain_wait(&bar[C::B_KVF + r % C::STAGES], (r / C::STAGES) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Keys in steps of 64 (half a loaded block); the two tiles alternate:
    //   S_0(0) S_1(0) | O_0 += P_0(0) V, S_0(1), O_1 += P_1(0) V, S_1(1) | ...
    // S_t(k+1) overwrites P_t(k), read by the O_t product issued just before it
    // (tcgen05.mma instructions of one thread execute in order).
    if (n_mine > 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t kIdescO = idesc_bf16_f32(128, D, false, true);
      int ru = 0;                 // ring uses of earlier items
      int base[C::TILES] = {};    // each tile's steps in earlier items
      bool ok = true;
      for (int j = 0; ok && j < n_mine; ++j) {
        int qs, bh, nht[C::TILES];
        const int nh = item(j, qs, bh, nht), nkb = (nh + 1) / 2;
        auto use_of = [&](int k) { return ru + C::QUSES + (k >> 1); };  // ring use of step k's block
        auto scores = [&](int t, int k) {
          const uint64_t b_k = sdesc_sw128(
              smem_u32(smem + C::OFF_K + (use_of(k) % C::STAGES) * C::TILE + (k & 1) * C::HALF_ROWS),
              16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
            umma_ts_w(tmem + C::COL_S + 64 * t, tmem + C::COL_Q + (D / 2) * t + kk * 8,
                      sdesc_add(b_k, off), kIdescS, kk > 0);
          }
          umma_commit_w(&bar[C::B_SF + t]);
        };
        auto pv = [&](int t, int k) {
          const uint64_t b_mn = sdesc_sw128(
              smem_u32(smem + C::OFF_V + (use_of(k) % C::STAGES) * C::TILE + (k & 1) * C::HALF_ROWS),
              C::CHUNK, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ts_w(tmem + C::COL_O + D * t, tmem + C::COL_S + 64 * t + kk * 8,
                      sdesc_add(b_mn, kk * 2048), kIdescO, (k > 0 || kk > 0) ? 1u : 0u);
        };
        // Q_0, Q_1 in TMEM. (O_t of the previous item may still be being read out:
        // the O_t += P_t V product that overwrites it waits for P_t, which its
        // softmax warps write only after that.)
        if (!warp_wait(&bar[C::B_IN], j & 1, wc)) { ok = false; break; }
        if (lane == 0)  // the Q slots are free
          for (int u = 0; u < C::QUSES; ++u) mbar_arrive(&bar[C::B_KVE + (ru + u) % C::STAGES]);
        const int u1 = use_of(0);
        if (!warp_wait(&bar[C::B_KVF + u1 % C::STAGES], (u1 / C::STAGES) & 1, wc)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < C::TILES; ++t)
          if (nht[t] > 0) scores(t, 0);
        for (int k = 0; ok && k < nh; ++k) {
          if (k + 1 < nh && ((k + 1) & 1) == 0) {  // step k+1 opens block (k+1)/2
            const int u = use_of(k + 1);
            if (!warp_wait(&bar[C::B_KVF + u % C::STAGES], (u / C::STAGES) & 1, wc)) { ok = false; break; }
          }
#pragma unroll
          for (int t = 0; t < C::TILES; ++t) {
            if (k >= nht[t]) continue;
            if (!warp_wait(&bar[C::B_PF + t], (base[t] + k) & 1, wc)) { ok = false; break; }
            tc_fence_after();
            pv(t, k);
            if (k + 1 < nht[t])
              scores(t, k + 1);
            else
              umma_commit_w(&bar[C::B_PVD + t]);
          }
          // both tiles are done with block k/2 once its second step is issued
          if (ok && ((k & 1) || k + 1 == nh))
            umma_commit_w(&bar[C::B_KVE + use_of(k) % C::STAGES]);
        }
        // A tile with no steps (the second tile of a head's last pair when n mod 256
        // <= 128) is signalled once the item's products are done, so that its
        // softmax warps wait for the item's blocks to be consumed before they wait
        // for the next item's Q slot (whose earlier fill is one of those blocks).
#pragma unroll
        for (int t = 0; t < C::TILES; ++t)
          if (ok && nht[t] == 0) umma_commit_w(&bar[C::B_PVD + t]);
        ru += C::QUSES + nkb;
#pragma unroll
        for (int t = 0; t < C::TILES; ++t) base[t] += nht[t];
      }
      umma_commit_w(&bar[C::B_DRAIN]);
      drain_wait(&bar[C::B_DRAIN], 0);
    }
  } else if (warp >= C::SOFT0) {
    // ------------------------------------------------------------ softmax
    const int t = (warp - C::SOFT0) >> 2;          // query tile of this warpgroup
    const int row = (warp & 3) * 32 + lane;        // row in the tile = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t scol = lane_base + C::COL_S + 64 * t;
    const uint32_t ocol = lane_base + C::COL_O + D * t;
    const float sl2 = p.scale_log2;
    int ru = 0, base_t = 0, pvd_t = 0;  // ring uses, steps and finished items of tile t
    // Row `row` of Q_t of the item whose Q tiles are ring use `rq` into TMEM: the
    // row's 16-byte pieces in the 128-byte-swizzled tile (piece j of a chunk row at
    // j ^ (row % 8)). The previous item's S_t products, the only readers of these
    // columns, are complete: this warp waited for each of them.
    auto move_q = [&](int rq) {
      const int uq = rq + (t >> 1);  // the ring use holding Q_t
      const int s = uq % C::STAGES;
      if (!warp_wait(&bar[C::B_KVF + s], (uq / C::STAGES) & 1, wc)) return false;
      const uint8_t* tile = smem + ((t & 1) == 0 ? C::OFF_K : C::OFF_V) + s * C::TILE;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v[32];
        const uint8_t* src = tile + c * C::CHUNK + row * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 x = *reinterpret_cast<const uint4*>(src + ((q ^ (row & 7)) << 4));
          v[4 * q] = x.x;
          v[4 * q + 1] = x.y;
          v[4 * q + 2] = x.z;
          v[4 * q + 3] = x.w;
        }
        tmem_st32(lane_base + C::COL_Q + (D / 2) * t + 32 * c, v);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar[C::B_IN]);
      return true;
    };
    bool ok = n_mine == 0 || move_q(0);
    for (int j = 0; ok && j < n_mine; ++j) {
      int qs, bh, nht[C::TILES];
      const int nkb = (item(j, qs, bh, nht) + 1) / 2;
      const int nh_t = nht[t];
      const int qg = qs + t * C::BM + row;
      float m_ref = -INFINITY;  // reference maximum of S * scale * log2(e)
      float l_run = 0.f;        // sum of exp2(S * scale * log2(e) - m_ref)
      for (int k = 0; ok && k < nh_t; ++k) {
        if (!warp_wait(&bar[C::B_SF + t], (base_t + k) & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld32(scol, sr);
        tmem_ld32(scol + 32, sr + 32);
        tmem_ld_wait();
        reg_fence32(sr);
        reg_fence32(sr + 32);

        // Last visible column of this step for this row (ragged m, causal k <= q).
        const int ks = 64 * k;
        int lim = p.m - 1 - ks;
        if (p.causal) lim = min(lim, qg - ks);
        if (lim < 63) {
  #pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c > lim) sr[c] = __float_as_uint(-INFINITY);
        }
        // Row maximum: eight chains of three-input maxima.
        float mx[8];
  #pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = __uint_as_float(sr[e]);
  #pragma unroll
        for (int c = 8; c < 64; c += 16)
  #pragma unroll
          for (int e = 0; e < 8; ++e)
            mx[e] = max3f(mx[e], __uint_as_float(sr[c + e]), __uint_as_float(sr[c + 8 + e]));
        const float rmax = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]),
                                 fmaxf(mx[6], mx[7])) * sl2;
        // Move the reference only when the row maximum passed it by the threshold.
        const bool move = rmax > m_ref + kRescaleThreshold;
        const float m_new = move ? rmax : m_ref;
        const float corr = move ? ex2(m_ref - m_new) : 1.f;  // 0 on the first step
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // no (-inf) - (-inf)
        m_ref = m_new;
        // P = exp2(S * scale * log2(e) - m) as bf16 pairs over this row's own S
        // columns.
        const uint64_t sl2x2 = f2pack(sl2, sl2);
        const uint64_t negm2 = f2pack(-m_use, -m_use);
        uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
        uint32_t pp[32];
  #pragma unroll
        for (int c = 0; c < 32; ++c) {
          const uint64_t x2 = ffma2(
              f2pack(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sl2x2, negm2);
          float x0, x1;
          f2unpack(x2, x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          acc2[c & 3] = fadd2(acc2[c & 3], f2pack(p0, p1));
          pp[c] = pack_bf16(p0, p1);
        }
        // S_t(k) completing implies O_t += P_t(k-1) V completed (issued before it),
        // so the O row may be rescaled before this step's product is signalled.
        if (k >= 1 && __any_sync(0xffffffffu, move)) {
  #pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(ocol + 32 * c, o);
            tmem_ld_wait();
            reg_fence32(o);
  #pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
            tmem_st32(ocol + 32 * c, o);
          }
        }
        tmem_st32(scol, pp);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar[C::B_PF + t]);
        float s0, s1, s2, s3, s4, s5, s6, s7;
        f2unpack(acc2[0], s0, s1);
        f2unpack(acc2[1], s2, s3);
        f2unpack(acc2[2], s4, s5);
        f2unpack(acc2[3], s6, s7);
        l_run = l_run * corr + (((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7)));
      }

      // A tile with no steps waits for the end of the item's products first: only
      // then has the earlier fill of the next item's Q slot surely landed, so that
      // the slot's barrier is at most one phase behind the wait in move_q.
      if (ok && nh_t == 0) {
        if (!warp_wait(&bar[C::B_PVD + t], pvd_t & 1, wc)) { ok = false; break; }
        ++pvd_t;
      }
      // The next item's Q_t goes in before this item's O_t comes out, so that the
      // next item's first S products run while the O rows are written.
      if (ok && j + 1 < n_mine && !move_q(ru + C::QUSES + nkb)) ok = false;
      // ---------------------------------------------------------- epilogue
      if (ok && nh_t > 0) {
        if (!warp_wait(&bar[C::B_PVD + t], pvd_t & 1, wc)) { ok = false; break; }
        tc_fence_after();
        // O / l as bf16 through the warp's staging area and TMA (rows past n and
        // the zero columns past d are not written)
        tmem_rows_store<D>(ocol, 1.f / l_run,
                           smem + C::OFF_EPI + (warp - C::SOFT0) * kStoreStageBytes, &tmO, 0,
                           qs + t * C::BM + (warp & 3) * 32, p.n, bh, p.d);
        if (qg < p.n) p.L[(size_t)bh * p.n + qg] = (m_ref + lg2(l_run)) * kLn2;
        tc_fence_before();  // O_t read out before the next item's products overwrite it
        ++pvd_t;
      }
      ru += C::QUSES + nkb;
      base_t += nh_t;
    }
    if (lane == 0) bulk_wait_all();  // the stores have read the staging buffers
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
  CUtensorMap mq, mk, mv, mo;
  // Rows of d values; the 64-column boxes read zeros past d.
  if (make_bf16_head_map(&mq, a.Q, a.BH, a.n, a.d, C::BM) != CUDA_SUCCESS ||
      make_bf16_head_map(&mk, a.K, a.BH, a.m, a.d, C::BN) != CUDA_SUCCESS ||
      make_bf16_head_map(&mv, a.V, a.BH, a.m, a.d, C::BN) != CUDA_SUCCESS ||
      make_bf16_store_map(&mo, a.O, a.BH, a.n, a.d) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  FwdParams p;
  p.O = static_cast<__nv_bfloat16*>(a.O);
  p.L = a.L;
  p.n = a.n;
  p.m = a.m;
  p.BH = a.BH;
  p.causal = a.causal;
  p.d = a.d;
  p.num_pairs = ceil_div(a.n, C::TILES * C::BM);
  p.group = heads_per_group(a.BH, p.num_pairs);
  p.scale_log2 = a.scale * 1.44269504088896340736f;
  cudaError_t e =
      cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  // One CTA per SM (persistent), fewer when there are fewer items.
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long items = (long long)p.num_pairs * a.BH;
  const unsigned grid = (unsigned)(items < sms ? items : sms);
  fwd_kernel<D><<<grid, C::THREADS, C::SMEM, stream>>>(mq, mk, mv, mo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward(const FwdArgs& a, cudaStream_t s) {
  return a.d > 64 ? launch_fwd_d<128>(a, s) : launch_fwd_d<64>(a, s);
}

cudaError_t forward_read_status(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_fwd_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_fwd_status, &zero, sizeof(unsigned int));
}

}  // namespace fa
