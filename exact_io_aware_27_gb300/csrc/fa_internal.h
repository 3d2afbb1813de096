// Declarations shared by the library's translation units (not installed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fa {

// Rows of the fp32 workspace arrays (-D and -L * log2(e)) per head: n rounded
// up to a multiple of this, so that every tile the kernels touch is in bounds
// and every row stride is a multiple of 16 bytes.
constexpr int kWorkspaceRowAlign = 128;

inline int round_up(int x, int a) { return (x + a - 1) / a * a; }
inline int ceil_div(int x, int a) { return (x + a - 1) / a; }

// Heads per launch-order group (see grouped_tile): enough blocks for about eight
// waves over the SMs. Smaller groups keep fewer heads' data in flight (less L2
// traffic); larger ones let the heavy causal blocks of later heads start
// earlier (a shorter tail). Eight waves measured best on GB300 for both kernels.
int heads_per_group(int BH, int tiles_per_head);

// The size rules every entry point applies (FA_OK or the fa_status they return).
int validate_sizes(int B, int H, int n, int m, int d);

// cuTensorMapEncodeTiled, fetched from the driver at first use.
CUresult encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, cuuint32_t rank,
                           void* base, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                           const cuuint32_t* box, CUtensorMapSwizzle swizzle);

// bf16 [BH, rows, d] viewed as a 3-D tensor (d innermost), boxes of
// 64 columns x box_rows rows with 128-byte swizzle; reads past `rows` in a
// head are zero-filled.
CUresult make_bf16_head_map(CUtensorMap* map, const void* base, int BH, int rows, int d,
                            int box_rows);
// bf16 [BH, rows, d] for the epilogues' stores: boxes of 32 columns x 32 rows
// with 64-byte swizzle; rows and columns past the tensor are not written.
CUresult make_bf16_store_map(CUtensorMap* map, void* base, int BH, int rows, int d);
// fp32 [BH, cols] as a 2-D tensor, boxes of box_cols x 1, no swizzle.
CUresult make_f32_row_map(CUtensorMap* map, const void* base, int BH, int cols, int box_cols);

struct FwdArgs {
  const void *Q, *K, *V;
  void* O;
  float* L;
  int BH, n, m, d, causal;
  float scale;
};
struct BwdArgs {
  const void *Q, *K, *V, *O, *dO;
  const float* L;
  void *dQ, *dK, *dV;
  float* ws_nD;   // [BH, n_pad] fp32, -D; 0 in the padding
  float* ws_nL2;  // [BH, n_pad] fp32, -L * log2(e); -inf in the padding
  int BH, n, m, d, n_pad, causal;
  float scale;
};

// Materialised standard attention (the baseline of the IO comparison): S and P
// are bf16 [BH, n, m_pad] matrices in memory, m_pad = m rounded up to 64.
constexpr int kStdColAlign = 64;
struct StdArgs {
  const void *Q, *K, *V;
  void *S, *P, *O;
  float* L;
  int BH, n, m, m_pad, d, causal;
  float scale;
};

// Kernel launches (return the launch's cudaError_t).
cudaError_t launch_standard(const StdArgs& a, cudaStream_t s);
cudaError_t launch_forward(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_dkdv(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t s);
// dK, dV and dQ in one persistent launch (each CTA: its dK/dV blocks, then its dQ blocks).
cudaError_t launch_bwd_main(const BwdArgs& a, cudaStream_t s);

// Online softmax statistics of fp32 rows (m, l per row).
cudaError_t launch_softmax_stats(const float* x, long long rows, long long cols, float* m,
                                 float* l, cudaStream_t s);

// Read-and-clear of each translation unit's device status word.
cudaError_t forward_read_status(unsigned int* out);
cudaError_t bwd_read_status(unsigned int* out);
cudaError_t selftest_read_status(unsigned int* out);
cudaError_t standard_read_status(unsigned int* out);

// Test-only: one tcgen05 GEMM through the same TMA / descriptor paths the
// attention kernels use (see fa_selftest.h).
cudaError_t launch_selftest_mma(int mode, const void* A, const void* B, float* D,
                                cudaStream_t s);

}  // namespace fa
