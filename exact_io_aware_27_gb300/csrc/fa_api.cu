// Host side of the C-ABI declared in include/fa.h: argument validation,
// workspace layout, TMA tensor-map construction and kernel launches.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

// Compute capability 10.3 check, cached per device ordinal.
constexpr int kMaxDevices = 64;
int g_device_ok[kMaxDevices];  // 0 unknown, 1 ok, -1 unsupported
std::mutex g_device_mu;

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED_DEVICE;
  {
    std::lock_guard<std::mutex> lk(g_device_mu);
    if (g_device_ok[dev] == 0) {
      int major = 0, minor = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return FA_ERR_CUDA;
      g_device_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    return g_device_ok[dev] == 1 ? FA_OK : FA_ERR_UNSUPPORTED_DEVICE;
  }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Range {
  uintptr_t lo, hi;
};
Range range_of(const void* p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return {a, a + bytes};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

constexpr int kMaxSeq = 1 << 24;

int check_sizes(int B, int H, int n, int m, int d) {
  if (B < 1 || H < 1 || n < 1 || m < 1) return FA_ERR_INVALID_ARG;
  if (n > kMaxSeq || m > kMaxSeq) return FA_ERR_INVALID_ARG;
  if ((long long)B * H > 65535) return FA_ERR_INVALID_ARG;
  if (d < 8 || d > 128 || d % 8 != 0) return FA_ERR_UNSUPPORTED_HEAD_DIM;
  return FA_OK;
}

int check_scale(float scale) {
  return (std::isfinite(scale) && scale > 0.f) ? FA_OK : FA_ERR_INVALID_ARG;
}

struct Workspace {
  float* nD;
  float* nL2;
  size_t bytes;
  int n_pad;
};

Workspace workspace_layout(void* base, int B, int H, int n) {
  Workspace w;
  w.n_pad = round_up(n, kWorkspaceRowAlign);
  const size_t rows = (size_t)B * H * w.n_pad;
  float* f = static_cast<float*>(base);
  w.nD = f;
  w.nL2 = f + rows;
  w.bytes = rows * 2 * sizeof(float);
  return w;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

// Shared validation of the backward family. Fills `a` on success.
int prepare_backward(const void* Q, const void* K, const void* V, const void* O, const float* L,
                     const void* dO, int B, int H, int n, int m, int d, int causal, float scale,
                     void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                     bool need_inputs, bool need_outputs, BwdArgs* a) {
  int rc = check_sizes(B, H, n, m, d);
  if (rc != FA_OK) return rc;
  if ((rc = check_scale(scale)) != FA_OK) return rc;
  if (!workspace) return FA_ERR_INVALID_ARG;
  if (need_inputs && (!Q || !K || !V || !O || !L || !dO)) return FA_ERR_INVALID_ARG;
  if (need_outputs && (!dQ || !dK || !dV)) return FA_ERR_INVALID_ARG;
  const void* bf16s[] = {Q, K, V, O, dO, dQ, dK, dV, workspace};
  for (const void* ptr : bf16s)
    if (ptr && !aligned(ptr, 16)) return FA_ERR_MISALIGNED;
  if (L && !aligned(L, 4)) return FA_ERR_MISALIGNED;
  const Workspace w = workspace_layout(workspace, B, H, n);
  if (workspace_bytes < w.bytes) return FA_ERR_WORKSPACE_TOO_SMALL;
  const size_t qn = (size_t)B * H * n * d * 2, km = (size_t)B * H * m * d * 2;
  const Range ins[] = {Q ? range_of(Q, qn) : Range{0, 0},  K ? range_of(K, km) : Range{0, 0},
                       V ? range_of(V, km) : Range{0, 0},  O ? range_of(O, qn) : Range{0, 0},
                       dO ? range_of(dO, qn) : Range{0, 0},
                       L ? range_of(L, (size_t)B * H * n * 4) : Range{0, 0}};
  const Range outs[] = {dQ ? range_of(dQ, qn) : Range{0, 0}, dK ? range_of(dK, km) : Range{0, 0},
                        dV ? range_of(dV, km) : Range{0, 0}, range_of(workspace, w.bytes)};
  for (const Range& o : outs) {
    if (o.lo == o.hi) continue;
    for (const Range& i : ins)
      if (i.lo != i.hi && overlap(o, i)) return FA_ERR_INVALID_ARG;
  }
  for (int x = 0; x < 4; ++x)
    for (int y = x + 1; y < 4; ++y)
      if (outs[x].lo != outs[x].hi && outs[y].lo != outs[y].hi && overlap(outs[x], outs[y]))
        return FA_ERR_INVALID_ARG;
  if ((rc = check_device()) != FA_OK) return rc;
  a->Q = Q;
  a->K = K;
  a->V = V;
  a->O = O;
  a->dO = dO;
  a->L = L;
  a->dQ = dQ;
  a->dK = dK;
  a->dV = dV;
  a->ws_nD = w.nD;
  a->ws_nL2 = w.nL2;
  a->BH = B * H;
  a->n = n;
  a->m = m;
  a->d = d;
  a->n_pad = w.n_pad;
  a->causal = causal ? 1 : 0;
  a->scale = scale;
  return FA_OK;
}

}  // namespace

int validate_sizes(int B, int H, int n, int m, int d) { return check_sizes(B, H, n, m, d); }

int heads_per_group(int BH, int tiles_per_head) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int g = ceil_div(8 * sms, tiles_per_head > 0 ? tiles_per_head : 1);
  return g < 1 ? 1 : (g > BH ? BH : g);
}

CUresult encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, cuuint32_t rank,
                           void* base, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                           const cuuint32_t* box, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = get_encode();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  const cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  return fn(map, dtype, rank, base, dims, strides_bytes, box, elem_strides,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult make_bf16_head_map(CUtensorMap* map, const void* base, int BH, int rows, int d,
                            int box_rows) {
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  return encode_tensor_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
                           dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

CUresult make_bf16_store_map(CUtensorMap* map, void* base, int BH, int rows, int d) {
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * d * 2};
  const cuuint32_t box[3] = {32, 32, 1};
  return encode_tensor_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_64B);
}

CUresult make_f32_row_map(CUtensorMap* map, const void* base, int BH, int cols, int box_cols) {
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)BH};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, 1};
  return encode_tensor_map(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims,
                           strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace fa

using namespace fa;

extern "C" {

int fa_version(void) { return 100; }

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED_HEAD_DIM: return "unsupported head dimension (need a multiple of 8 from 8 to 128)";
    case FA_ERR_MISALIGNED: return "misaligned pointer";
    case FA_ERR_UNSUPPORTED_DEVICE: return "unsupported device (need compute capability 10.3)";
    case FA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_DEVICE_TIMEOUT: return "device barrier wait timed out";
    default: return "unknown status";
  }
}

int fa_forward(const void* Q, const void* K, const void* V, int B, int H, int n, int m, int d,
               int causal, float scale, void* O, float* L, void* stream) {
  int rc = check_sizes(B, H, n, m, d);
  if (rc != FA_OK) return rc;
  if ((rc = check_scale(scale)) != FA_OK) return rc;
  if (!Q || !K || !V || !O || !L) return FA_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(L, 4))
    return FA_ERR_MISALIGNED;
  const size_t qn = (size_t)B * H * n * d * 2, km = (size_t)B * H * m * d * 2;
  const Range ro = range_of(O, qn), rl = range_of(L, (size_t)B * H * n * 4);
  const Range ins[] = {range_of(Q, qn), range_of(K, km), range_of(V, km)};
  for (const Range& i : ins)
    if (overlap(ro, i) || overlap(rl, i)) return FA_ERR_INVALID_ARG;
  if (overlap(ro, rl)) return FA_ERR_INVALID_ARG;
  if ((rc = check_device()) != FA_OK) return rc;
  FwdArgs a;
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.O = O;
  a.L = L;
  a.BH = B * H;
  a.n = n;
  a.m = m;
  a.d = d;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  return from_cuda(launch_forward(a, static_cast<cudaStream_t>(stream)));
}

size_t fa_backward_workspace_size(int B, int H, int n, int m, int d) {
  if (check_sizes(B, H, n, m, d) != FA_OK) return 0;
  return workspace_layout(nullptr, B, H, n).bytes;
}

int fa_backward_preprocess(const void* O, const void* dO, const float* L, int B, int H, int n,
                           int d, void* workspace, size_t workspace_bytes, void* stream) {
  if (!O || !dO || !L) return FA_ERR_INVALID_ARG;
  BwdArgs a;
  const int rc = prepare_backward(nullptr, nullptr, nullptr, O, L, dO, B, H, n, 1, d, 0,
                                  1.0f, nullptr, nullptr, nullptr, workspace, workspace_bytes,
                                  false, false, &a);
  if (rc != FA_OK) return rc;
  return from_cuda(launch_bwd_preprocess(a, static_cast<cudaStream_t>(stream)));
}

int fa_backward_dkdv(const void* Q, const void* K, const void* V, const void* dO, int B, int H,
                     int n, int m, int d, int causal, float scale, void* dK, void* dV,
                     void* workspace, size_t workspace_bytes, void* stream) {
  if (!Q || !K || !V || !dO || !dK || !dV) return FA_ERR_INVALID_ARG;
  BwdArgs a;
  const int rc = prepare_backward(Q, K, V, nullptr, nullptr, dO, B, H, n, m, d, causal, scale,
                                  nullptr, dK, dV, workspace, workspace_bytes, false, false, &a);
  if (rc != FA_OK) return rc;
  return from_cuda(launch_bwd_dkdv(a, static_cast<cudaStream_t>(stream)));
}

int fa_backward_dq(const void* Q, const void* K, const void* V, const void* dO, int B, int H,
                   int n, int m, int d, int causal, float scale, void* dQ, void* workspace,
                   size_t workspace_bytes, void* stream) {
  if (!Q || !K || !V || !dO || !dQ) return FA_ERR_INVALID_ARG;
  BwdArgs a;
  const int rc = prepare_backward(Q, K, V, nullptr, nullptr, dO, B, H, n, m, d, causal, scale,
                                  dQ, nullptr, nullptr, workspace, workspace_bytes, false, false,
                                  &a);
  if (rc != FA_OK) return rc;
  return from_cuda(launch_bwd_dq(a, static_cast<cudaStream_t>(stream)));
}

int fa_backward_grads(const void* Q, const void* K, const void* V, const void* dO, int B, int H,
                      int n, int m, int d, int causal, float scale, void* dQ, void* dK, void* dV,
                      void* workspace, size_t workspace_bytes, void* stream) {
  if (!Q || !K || !V || !dO || !dQ || !dK || !dV) return FA_ERR_INVALID_ARG;
  BwdArgs a;
  const int rc = prepare_backward(Q, K, V, nullptr, nullptr, dO, B, H, n, m, d, causal, scale,
                                  dQ, dK, dV, workspace, workspace_bytes, false, false, &a);
  if (rc != FA_OK) return rc;
  return from_cuda(launch_bwd_main(a, static_cast<cudaStream_t>(stream)));
}

int fa_backward(const void* Q, const void* K, const void* V, const void* O, const float* L,
                const void* dO, int B, int H, int n, int m, int d, int causal, float scale,
                void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                void* stream) {
  BwdArgs a;
  int rc = prepare_backward(Q, K, V, O, L, dO, B, H, n, m, d, causal, scale, dQ, dK, dV,
                            workspace, workspace_bytes, true, true, &a);
  if (rc != FA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_bwd_preprocess(a, s);
  if (e == cudaSuccess) e = launch_bwd_main(a, s);
  return from_cuda(e);
}

int fa_online_softmax_stats(const float* x, long long rows, long long cols, float* m, float* l,
                            void* stream) {
  if (!x || !m || !l || rows < 1 || cols < 1) return FA_ERR_INVALID_ARG;
  if (rows > (1LL << 40) || cols > (1LL << 40)) return FA_ERR_INVALID_ARG;
  if (!aligned(x, 4) || !aligned(m, 4) || !aligned(l, 4)) return FA_ERR_MISALIGNED;
  const Range rx = range_of(x, (size_t)rows * (size_t)cols * 4);
  const Range rm = range_of(m, (size_t)rows * 4), rl = range_of(l, (size_t)rows * 4);
  if (overlap(rx, rm) || overlap(rx, rl) || overlap(rm, rl)) return FA_ERR_INVALID_ARG;
  int rc = check_device();
  if (rc != FA_OK) return rc;
  return from_cuda(launch_softmax_stats(x, rows, cols, m, l, static_cast<cudaStream_t>(stream)));
}

size_t fa_standard_matrix_bytes(int B, int H, int n, int m) {
  if (B < 1 || H < 1 || n < 1 || m < 1 || n > kMaxSeq || m > kMaxSeq) return 0;
  return (size_t)B * H * n * round_up(m, kStdColAlign) * 2;
}

int fa_standard_forward(const void* Q, const void* K, const void* V, int B, int H, int n, int m,
                        int d, int causal, float scale, void* S, void* P, void* O, float* L,
                        void* stream) {
  int rc = check_sizes(B, H, n, m, d);
  if (rc != FA_OK) return rc;
  if ((rc = check_scale(scale)) != FA_OK) return rc;
  if (!Q || !K || !V || !S || !P || !O || !L) return FA_ERR_INVALID_ARG;
  if (ceil_div(n, 128) > 65535) return FA_ERR_INVALID_ARG;  // query tiles: one grid row each
  const void* bf16s[] = {Q, K, V, S, P, O};
  for (const void* ptr : bf16s)
    if (!aligned(ptr, 16)) return FA_ERR_MISALIGNED;
  if (!aligned(L, 4)) return FA_ERR_MISALIGNED;
  const size_t qn = (size_t)B * H * n * d * 2, km = (size_t)B * H * m * d * 2;
  const size_t sp = fa_standard_matrix_bytes(B, H, n, m);
  const Range ins[] = {range_of(Q, qn), range_of(K, km), range_of(V, km)};
  const Range outs[] = {range_of(S, sp), range_of(P, sp), range_of(O, qn),
                        range_of(L, (size_t)B * H * n * 4)};
  for (const Range& o : outs)
    for (const Range& i : ins)
      if (overlap(o, i)) return FA_ERR_INVALID_ARG;
  for (int x = 0; x < 4; ++x)
    for (int y = x + 1; y < 4; ++y)
      if (overlap(outs[x], outs[y])) return FA_ERR_INVALID_ARG;
  if ((rc = check_device()) != FA_OK) return rc;
  StdArgs a;
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.S = S;
  a.P = P;
  a.O = O;
  a.L = L;
  a.BH = B * H;
  a.n = n;
  a.m = m;
  a.m_pad = round_up(m, kStdColAlign);
  a.d = d;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  return from_cuda(launch_standard(a, static_cast<cudaStream_t>(stream)));
}

int fa_get_device_status(int* status_out) {
  if (!status_out) return FA_ERR_INVALID_ARG;
  unsigned int f = 0, b = 0, t = 0, sd = 0;
  if (forward_read_status(&f) != cudaSuccess || bwd_read_status(&b) != cudaSuccess ||
      selftest_read_status(&t) != cudaSuccess || standard_read_status(&sd) != cudaSuccess)
    return FA_ERR_CUDA;
  const unsigned int bits = f | b | t | sd;
  *status_out = (bits & kDeviceTimeoutBit)  ? FA_ERR_DEVICE_TIMEOUT
                : (bits & kDeviceLayoutBit) ? FA_ERR_UNSUPPORTED_DEVICE
                                            : FA_OK;
  return FA_OK;
}

}  // extern "C"
