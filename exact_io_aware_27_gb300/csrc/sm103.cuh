// Inline-PTX building blocks for sm_103a: mbarrier, TMA bulk tensor copies,
// tcgen05 MMA / tensor memory (TMEM), and a few arithmetic helpers.
//
// Every wait on an mbarrier is bounded: after about two seconds (or 2^28
// polls) the waiting thread raises the CTA's abort flag, records
// kDeviceTimeoutBit in the translation unit's device status word and returns
// false, so the kernel can unwind instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace fa {

#define FA_DEV __device__ __forceinline__

constexpr unsigned int kDeviceTimeoutBit = 1u;
// Set by a kernel that found its dynamic shared memory at an address its layout
// does not allow (it then returns before touching anything).
constexpr unsigned int kDeviceLayoutBit = 2u;
constexpr long long kWaitMaxCycles = 4000000000ll;  // ~2 s at 2 GHz
constexpr uint32_t kWaitMaxPolls = 1u << 28;

FA_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
FA_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
FA_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
// Returns an mbarrier's shared memory to ordinary use (before it is initialised again).
FA_DEV void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

FA_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
FA_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
FA_DEV uint32_t mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok;
}

// Shared state every bounded wait consults: the CTA-wide abort flag (shared
// memory) and the translation unit's device status word (global memory).
struct WaitCtx {
  volatile uint32_t* abort_flag;
  unsigned int* status;
};

// Waits until the phase with the given parity of `bar` has completed.
// Returns false (after raising the abort flag) if it gave up: after
// `max_cycles` of clock64 or kWaitMaxPolls polls, or at once when another
// thread of the CTA has raised the abort flag.
FA_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w,
                      long long max_cycles = kWaitMaxCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
#pragma unroll 1
  for (uint32_t it = 1; it < kWaitMaxPolls; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*w.abort_flag) return false;
      if (clock64() - t0 > max_cycles) break;
    }
  }
  *w.abort_flag = 1u;
  atomicOr(w.status, kDeviceTimeoutBit);
  return false;
}

// mbar_wait for a whole warp: every lane polls, and the result is agreed
// across the warp so that warp-collective instructions (tcgen05.ld/st) that
// follow are reached by all lanes or by none.
FA_DEV bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w,
                      long long max_cycles = kWaitMaxCycles) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, w, max_cycles));
}

// Linear block index -> (tile rank within a head, head). Heads are taken in
// groups of `group`; inside a group, rank 0 of every head comes first, then
// rank 1, and so on, so that the blocks in flight share a few heads' data in L2.
FA_DEV void grouped_tile(int lin, int BH, int tiles, int group, int& rank, int& bh) {
  const int per_group = group * tiles;
  const int g = lin / per_group;
  const int base = g * group;
  const int gsize = min(group, BH - base);
  const int r = lin - g * per_group;
  rank = r / gsize;
  bh = base + r % gsize;
}

// Item of round r for CTA c of P in a persistent schedule: rounds alternate their
// direction so that, with the items in heaviest-first order, every CTA gets about
// the same total work.
FA_DEV int snake_item(int r, int c, int P) { return r * P + ((r & 1) ? P - 1 - c : c); }

// ---------------------------------------------------------------- TMA
FA_DEV void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Tiled 3-D load; c0 is the innermost coordinate (elements), must be a
// multiple of 16 bytes' worth of elements.
FA_DEV void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                        int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Tiled 3-D store from shared memory, as a bulk async-group of the calling
// thread. Rows and columns outside the tensor are not written. c0 follows the
// load's alignment rule; no coordinate may be negative.
FA_DEV void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
FA_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's bulk groups still read shared memory.
template <int N>
FA_DEV void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until all of this thread's bulk groups are complete.
FA_DEV void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
FA_DEV void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
// Makes this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor-core operand reads, TMA stores).
FA_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
FA_DEV void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
FA_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
FA_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
FA_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
FA_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrives once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
FA_DEV void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]
FA_DEV void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]
FA_DEV void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Warp-collective forms: every lane of a full warp executes the call (so the
// operands stay warp-uniform) and one lane chosen by elect.sync issues it.
FA_DEV void umma_ss_w(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                      uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
FA_DEV void umma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                      uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
FA_DEV void umma_commit_w(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Instruction descriptor for kind::f16 with bf16 A and B and an fp32
// accumulator. a_mn / b_mn select the MN-major (transposed) operand layout.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                       // D format: f32
         | (1u << 7)                     // A format: bf16
         | (1u << 10)                    // B format: bf16
         | ((a_mn ? 1u : 0u) << 15)      // A major-ness
         | ((b_mn ? 1u : 0u) << 16)      // B major-ness
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle. `saddr` is the shared
// address of the operand start; `lbo` / `sbo` are the leading / stride byte
// offsets of the canonical layout:
//   K-major : rows of 128 B (64 bf16 along K), 8-row groups SBO apart; LBO unused.
//   MN-major: 128 B (64 bf16) along MN per row, one row per K index; 8-row K
//             groups SBO apart, 64-wide MN chunks LBO apart.
FA_DEV uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// A descriptor advanced by `bytes` (a multiple of 16) along its start address.
// Valid while the address stays below 256 KB (the 14-bit field does not carry).
FA_DEV uint64_t sdesc_add(uint64_t desc, uint32_t bytes) { return desc + (uint64_t)(bytes >> 4); }

#define FA_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                 "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define FA_P8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), \
                 "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])
#define FA_I8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                 "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// 32 consecutive 32-bit TMEM columns of this thread's lane -> r[0..31].
// Not complete until tmem_ld_wait(); call reg_fence on the registers after it.
FA_DEV void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24)
      : "r"(taddr));
}
FA_DEV void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : FA_R8(0), FA_R8(8)
      : "r"(taddr));
}
FA_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Keeps the compiler from moving uses of r[] above a preceding tmem_ld_wait().
FA_DEV void reg_fence32(uint32_t* r) {
  asm volatile("" : FA_P8(0), FA_P8(8), FA_P8(16), FA_P8(24));
}
FA_DEV void reg_fence16(uint32_t* r) { asm volatile("" : FA_P8(0), FA_P8(8)); }

FA_DEV void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      FA_I8(0), FA_I8(8), FA_I8(16), FA_I8(24)
      : "memory");
}
FA_DEV void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      FA_I8(0), FA_I8(8)
      : "memory");
}
FA_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

#undef FA_R8
#undef FA_P8
#undef FA_I8

// ---------------------------------------------------------------- arithmetic
FA_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
FA_DEV float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Three-input maximum.
FA_DEV float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Packed pairs of fp32 (two lanes in one 64-bit register) for the f32x2 forms.
FA_DEV uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
FA_DEV void f2unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
FA_DEV uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
FA_DEV uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
FA_DEV uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Two floats -> packed bf16 pair (round to nearest even); `lo` in bits 0..15.
FA_DEV uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
FA_DEV float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
FA_DEV float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

FA_DEV void st_shared_v4(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Rounds a shared-memory pointer up so that its shared-space address is a
// multiple of 1024 (the 128-byte swizzle pattern repeats every 1024 bytes and
// is computed from shared-address bits).
FA_DEV uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

// ------------------------------------------------------------------ epilogue stores
// Bytes of one warp's staging area for tmem_rows_store (two buffers of 32 rows x
// 32 bf16); the area must start on a 1024-byte boundary.
constexpr int kStoreStageBytes = 2 * 2048;

// Stores columns [0, NCOL) of this warp's 32 TMEM lanes (an fp32 accumulator at
// `tcol`, times this lane's `mul`, rounded to bf16) to rows row0 .. row0 + 31 of
// head bh and columns col0 + [0, NCOL) of a bf16 [BH, rows, d] tensor, through
// `map` (boxes of 32 columns x 32 rows, 64-byte swizzle). Only the first
// `valid_cols` columns are stored, and nothing when row0 >= nrows (the tensor's
// rows). Each 32-column piece is written to one of the
// warp's two staging buffers in `stage`, with the swizzle the map expects
// (16-byte chunk k of row r at chunk k ^ ((r >> 1) & 3)), and lane 0 stores it
// with one TMA copy; TMA leaves rows and columns outside the tensor untouched.
// Lane 0 owns the copies: before `stage` holds anything else it must call
// bulk_wait_read<0>() (or bulk_wait_all()).
template <int NCOL>
FA_DEV void tmem_rows_store(uint32_t tcol, float mul, uint8_t* stage, const CUtensorMap* map,
                            int col0, int row0, int nrows, int bh, int valid_cols) {
  if (row0 >= nrows) return;  // warp-uniform
  const int lane = threadIdx.x & 31;
  if (lane == 0) bulk_wait_read<0>();  // copies of an earlier call
  __syncwarp();
#pragma unroll
  for (int c = 0; c < NCOL / 32; ++c) {
    if (32 * c >= valid_cols) break;  // warp-uniform
    uint32_t o[32];
    tmem_ld32(tcol + 32 * c, o);
    tmem_ld_wait();
    reg_fence32(o);
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      w[e] = pack_bf16(__uint_as_float(o[2 * e]) * mul, __uint_as_float(o[2 * e + 1]) * mul);
    uint8_t* buf = stage + (c & 1) * 2048;
    if (c >= 2) {  // the copy of piece c - 2 has read this buffer
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
    }
    const uint32_t row = smem_u32(buf) + lane * 64;
    const uint32_t sw = (uint32_t)((lane >> 1) & 3);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      st_shared_v4(row + (((uint32_t)k ^ sw) << 4), w[4 * k], w[4 * k + 1], w[4 * k + 2],
                   w[4 * k + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(map, buf, col0 + 32 * c, row0, bh);
      bulk_commit();
    }
  }
}

}  // namespace fa
