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
// GB300 mapping (one CTA per (pair of query tiles, head), 384 threads):
//   warp 0       TMA producer: Q of both tiles once, then K_j and V_j into a
//                STAGES-deep ring shared by the two tiles
//   warp 1       MMA issuer (whole warp, one elected lane issues):
//                S0 = Q0 K_j^T, S1 = Q1 K_j^T, then O0 += P0 V_j, O1 += P1 V_j
//                (P read from TMEM); S_t of block j+1 waits for O_t += P_t V_j
//   warps 4..7   softmax of tile 0, warps 8..11 softmax of tile 1: thread r
//                owns query row r of its tile (= TMEM lane r); reads the S row
//                with tcgen05.ld, masks, updates (m, l) in base 2 (exp2 via
//                ex2.approx), writes P as bf16 over the first 64 columns of
//                its own S row, rescales its O row when m moved, and runs the
//                epilogue. While one tile's softmax runs, the tensor cores work
//                on the other tile.
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256, 256+d) O1 [256+d, 256+2d).
// Scores, probabilities and the accumulators never leave the SM.
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
  static constexpr int TILES = 2;                // query tiles per CTA
  static constexpr int BN = 128;                 // keys per block
  static constexpr int KCH = D / 64;             // 128-byte column chunks per row
  static constexpr int CHUNK = 128 * 128;        // bytes of one chunk of a 128-row tile
  static constexpr int TILE = KCH * CHUNK;       // bytes of a Q, K or V tile
  static constexpr int STAGES = (D == 128) ? 2 : 4;
  static constexpr int OFF_Q = 0;                // TILES query tiles
  static constexpr int OFF_K = OFF_Q + TILES * TILE;
  static constexpr int OFF_V = OFF_K + STAGES * TILE;
  static constexpr int OFF_BAR = OFF_V + STAGES * TILE;
  // barrier slots
  static constexpr int B_Q = 0;
  static constexpr int B_KF = 1;
  static constexpr int B_KE = B_KF + STAGES;
  static constexpr int B_VF = B_KE + STAGES;
  static constexpr int B_VE = B_VF + STAGES;
  static constexpr int B_SF = B_VE + STAGES;    // + tile: S_t ready
  static constexpr int B_PF = B_SF + TILES;     // + 2 tile + half: half of P_t written
  static constexpr int B_PVD = B_PF + 2 * TILES;  // + tile: O_t += P_t V done
  static constexpr int B_DRAIN = B_PVD + TILES;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
  static constexpr uint32_t COL_S = 0;           // + 128 * tile
  static constexpr uint32_t COL_O = 256;         // + D * tile
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int THREADS = 384;
  static_assert(COL_O + TILES * D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct FwdParams {
  __nv_bfloat16* O;
  float* L;
  int n, m, BH, causal, num_pairs, group;
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

// Key blocks a tile of rows [q0, q0 + 128) visits (0 if the tile is past n).
__device__ __forceinline__ int tile_blocks(int q0, int n, int m, int causal) {
  if (q0 >= n) return 0;
  int nkb = (m + 127) / 128;
  if (causal) nkb = min(nkb, (min(q0 + 127, n - 1)) / 128 + 1);  // keys k <= q
  return nkb;
}

template <int D>
__global__ void __launch_bounds__(384, 1)
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
  // a group the heaviest tile pairs (the last ones, under causal masking) go first.
  int pair, bh;
  grouped_tile(blockIdx.x, p.BH, p.num_pairs, p.group, pair, bh);
  if (p.causal) pair = p.num_pairs - 1 - pair;
  const int qs = pair * (C::TILES * C::BM);
  const int nkb0 = tile_blocks(qs, p.n, p.m, p.causal);
  const int nkb1 = tile_blocks(qs + C::BM, p.n, p.m, p.causal);
  const int nkb = max(nkb0, nkb1);

  if (threadIdx.x == 0) {
    mbar_init(&bar[C::B_Q], 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bar[C::B_KF + s], 1);
      mbar_init(&bar[C::B_KE + s], 1);
      mbar_init(&bar[C::B_VF + s], 1);
      mbar_init(&bar[C::B_VE + s], 1);
    }
    for (int t = 0; t < C::TILES; ++t) {
      mbar_init(&bar[C::B_SF + t], 1);
      mbar_init(&bar[C::B_PF + 2 * t], 128);
      mbar_init(&bar[C::B_PF + 2 * t + 1], 128);
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
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      mbar_arrive_expect_tx(&bar[C::B_Q], C::TILES * C::TILE);
#pragma unroll
      for (int t = 0; t < C::TILES; ++t)
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(smem + C::OFF_Q + t * C::TILE + c * C::CHUNK, &tmQ, &bar[C::B_Q], c * 64,
                      qs + t * C::BM, bh);
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
    constexpr uint32_t kIdescS = idesc_bf16_f32(128, C::BN, false, false);
    constexpr uint32_t kIdescO = idesc_bf16_f32(128, D, false, true);
    bool ok = warp_wait(&bar[C::B_Q], 0, wc);
    for (int j = 0; ok && j < nkb; ++j) {
      const int s = j % C::STAGES;
      const uint32_t ph = (j / C::STAGES) & 1;
      if (!warp_wait(&bar[C::B_KF + s], ph, wc)) break;
      const uint64_t dK_k = sdesc_sw128(smem_u32(smem + C::OFF_K + s * C::TILE), 16, 1024);
#pragma unroll
      for (int t = 0; t < C::TILES; ++t) {
        if (j >= (t == 0 ? nkb0 : nkb1)) continue;
        // S_t's columns hold P_t of block j-1 until O_t += P_t V_{j-1} is done.
        if (j >= 1 && !warp_wait(&bar[C::B_PVD + t], (j - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint64_t dQ_k = sdesc_sw128(smem_u32(smem + C::OFF_Q + t * C::TILE), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
          umma_ss_w(tmem + C::COL_S + 128 * t, sdesc_add(dQ_k, off), sdesc_add(dK_k, off),
                    kIdescS, kk > 0);
        }
        umma_commit_w(&bar[C::B_SF + t]);
      }
      if (!ok) break;
      umma_commit_w(&bar[C::B_KE + s]);
      if (!warp_wait(&bar[C::B_VF + s], ph, wc)) break;
      const uint64_t dV_mn = sdesc_sw128(smem_u32(smem + C::OFF_V + s * C::TILE), C::CHUNK, 1024);
#pragma unroll
      for (int t = 0; t < C::TILES; ++t) {
        if (j >= (t == 0 ? nkb0 : nkb1)) continue;
        const uint32_t aP = tmem + C::COL_S + 128 * t;  // P_t: first 64 columns of S_t
        // Keys 0..63 as soon as their P is written, then keys 64..127.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!warp_wait(&bar[C::B_PF + 2 * t + h], j & 1, wc)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
            umma_ts_w(tmem + C::COL_O + D * t, aP + kk * 8, sdesc_add(dV_mn, kk * 2048), kIdescO,
                      (j > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        umma_commit_w(&bar[C::B_PVD + t]);
      }
      if (!ok) break;
      umma_commit_w(&bar[C::B_VE + s]);
    }
    umma_commit_w(&bar[C::B_DRAIN]);
    drain_wait(&bar[C::B_DRAIN], 0);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;                 // query tile of this warpgroup
    const int row = ((warp - 4) & 3) * 32 + lane;  // row in the tile = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t scol = lane_base + C::COL_S + 128 * t;
    const uint32_t ocol = lane_base + C::COL_O + D * t;
    const int qg = qs + t * C::BM + row;
    const int nkb_t = t == 0 ? nkb0 : nkb1;
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY;  // reference maximum of S * scale * log2(e)
    float l_run = 0.f;        // sum of exp2(S * scale * log2(e) - m_ref)
    bool ok = true;
    for (int j = 0; j < nkb_t; ++j) {
      if (!warp_wait(&bar[C::B_SF + t], j & 1, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[128];
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
      // Row maximum: eight chains of three-input maxima.
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = __uint_as_float(sr[k]);
#pragma unroll
      for (int c = 8; c < 128; c += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mx[k] = max3f(mx[k], __uint_as_float(sr[c + k]), __uint_as_float(sr[c + 8 + k]));
      const float rmax = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]),
                               fmaxf(mx[6], mx[7])) * sl2;
      // Move the reference only when the row maximum passed it by the threshold.
      const bool move = rmax > m_ref + kRescaleThreshold;
      const float m_new = move ? rmax : m_ref;
      const float corr = move ? ex2(m_ref - m_new) : 1.f;  // 0 on the first block
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // no (-inf) - (-inf)
      m_ref = m_new;
      // S_t(j) completing implies O_t += P_t V_{j-1} completed (issued before
      // it), so the O row may be rescaled before this block's products start.
      // When no row of the warp moved its reference (the common case) each half
      // of P is signalled as soon as it is written; otherwise both halves are
      // signalled after the rescale.
      const bool rescale = j >= 1 && __any_sync(0xffffffffu, move);
      // P = exp2(S * scale * log2(e) - m) in two halves of 64 keys, written as
      // bf16 pairs over this row's own S columns.
      const uint64_t sl2x2 = f2pack(sl2, sl2);
      const uint64_t negm2 = f2pack(-m_use, -m_use);
      uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pp[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int e = 64 * h + 2 * c;
          const uint64_t x2 =
              ffma2(f2pack(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sl2x2, negm2);
          float x0, x1;
          f2unpack(x2, x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          acc2[c & 3] = fadd2(acc2[c & 3], f2pack(p0, p1));
          pp[c] = pack_bf16(p0, p1);
        }
        tmem_st32(scol + 32 * h, pp);
        if (!rescale) {
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bar[C::B_PF + 2 * t + h]);
        }
      }
      if (rescale) {
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
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bar[C::B_PF + 2 * t]);
        mbar_arrive(&bar[C::B_PF + 2 * t + 1]);
      }
      float s0, s1, s2, s3, s4, s5, s6, s7;
      f2unpack(acc2[0], s0, s1);
      f2unpack(acc2[1], s2, s3);
      f2unpack(acc2[2], s4, s5);
      f2unpack(acc2[3], s6, s7);
      l_run = l_run * corr + (((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7)));
    }

    // ------------------------------------------------------------ epilogue
    if (ok && nkb_t > 0 && warp_wait(&bar[C::B_PVD + t], (nkb_t - 1) & 1, wc)) {
      tc_fence_after();
      const float inv_l = 1.f / l_run;
      __nv_bfloat16* orow = p.O + ((size_t)bh * p.n + qg) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(ocol + 32 * c, o);
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
      if (qg < p.n) p.L[(size_t)bh * p.n + qg] = (m_ref + lg2(l_run)) * kLn2;
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
  p.num_pairs = ceil_div(a.n, C::TILES * C::BM);
  p.group = heads_per_group(a.BH, p.num_pairs);
  p.scale_log2 = a.scale * 1.44269504088896340736f;
  cudaError_t e =
      cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)p.num_pairs * (unsigned)a.BH;
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
