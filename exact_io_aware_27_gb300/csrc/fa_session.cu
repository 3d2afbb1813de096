// Host-buffer sessions (see include/fa.h): one forward + backward step whose
// inputs and outputs live in host memory, pipelined over chunks of heads.
//
// Heads are independent in both passes, so a step splits B*H into chunks of at
// most `chunk_heads` heads (the first and the last of half that size, which
// shortens the pipeline's fill and drain) and runs three streams: copies in (Q, K, V, dO of chunk c),
// kernels (fa_forward then fa_backward on chunk c) and copies out (O, L, dQ, dK,
// dV of chunk c). Chunk c uses buffer set c % 4; events order each stage after
// the previous stage of its chunk and the copies in of chunk c + 4 after the
// copies out of chunk c, so the copies of one chunk overlap the kernels of its
// neighbours and host <-> device traffic in both directions runs at once. The
// chunks are numbered across steps: a step submitted before the previous one has
// finished continues the same pipeline, so its copies in run while the previous
// step's last copies out still do.
#include <cmath>
#include <cstdint>
#include <new>

#include "fa.h"
#include "fa_internal.h"

namespace fa {
// Buffer sets: chunk c uses set c % kSessionSets. With steps submitted back to back
// four sets measured 9 % faster than three at the benchmark shape (the copies in
// may run one more chunk ahead of the copies out); five or six added under 1 %.
constexpr int kSessionSets = 4;
}  // namespace fa

struct fa_session {
  int B, H, n, m, d, chunk, device;
  long long chunks;  // chunks submitted so far (chunk c uses buffer set c % 4)
  cudaStream_t in, comp, out;
  cudaEvent_t ev_in[fa::kSessionSets], ev_comp[fa::kSessionSets], ev_out[fa::kSessionSets];
  void *Q[fa::kSessionSets], *K[fa::kSessionSets], *V[fa::kSessionSets], *dO[fa::kSessionSets];
  void *O[fa::kSessionSets], *dQ[fa::kSessionSets], *dK[fa::kSessionSets], *dV[fa::kSessionSets];
  float* L[fa::kSessionSets];
  void* ws;
  size_t ws_bytes;
};

namespace fa {
namespace {

constexpr int kSets = kSessionSets;

void release(fa_session* s) {
  if (!s) return;
  for (cudaStream_t st : {s->in, s->comp, s->out})
    if (st) cudaStreamSynchronize(st);
  for (int i = 0; i < kSets; ++i) {
    for (void* p : {s->Q[i], s->K[i], s->V[i], s->dO[i], s->O[i], s->dQ[i], s->dK[i], s->dV[i],
                    static_cast<void*>(s->L[i])})
      if (p) cudaFree(p);
    for (cudaEvent_t e : {s->ev_in[i], s->ev_comp[i], s->ev_out[i]})
      if (e) cudaEventDestroy(e);
  }
  if (s->ws) cudaFree(s->ws);
  for (cudaStream_t st : {s->in, s->comp, s->out})
    if (st) cudaStreamDestroy(st);
  delete s;
}

int copy_in(void* dst, const void* src, size_t bytes, cudaStream_t st) {
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, st) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}
int copy_out(void* dst, const void* src, size_t bytes, cudaStream_t st) {
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, st) == cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

int fa_session_create(int B, int H, int n, int m, int d, int chunk_heads, fa_session** out) {
  if (!out) return FA_ERR_INVALID_ARG;
  *out = nullptr;
  const int rc = validate_sizes(B, H, n, m, d);
  if (rc != FA_OK) return rc;
  if (chunk_heads < 1 || chunk_heads > B * H) return FA_ERR_INVALID_ARG;
  fa_session* s = new (std::nothrow) fa_session{};
  if (!s) return FA_ERR_CUDA;
  s->B = B;
  s->H = H;
  s->n = n;
  s->m = m;
  s->d = d;
  s->chunk = chunk_heads;
  if (cudaGetDevice(&s->device) != cudaSuccess) {
    delete s;
    return FA_ERR_CUDA;
  }
  const size_t qn = (size_t)chunk_heads * n * d * 2, km = (size_t)chunk_heads * m * d * 2;
  bool ok = cudaStreamCreateWithFlags(&s->in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&s->comp, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&s->out, cudaStreamNonBlocking) == cudaSuccess;
  for (int i = 0; ok && i < kSets; ++i) {
    ok = cudaEventCreateWithFlags(&s->ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&s->ev_comp[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&s->ev_out[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaMalloc(&s->Q[i], qn) == cudaSuccess && cudaMalloc(&s->dO[i], qn) == cudaSuccess &&
         cudaMalloc(&s->O[i], qn) == cudaSuccess && cudaMalloc(&s->dQ[i], qn) == cudaSuccess &&
         cudaMalloc(&s->K[i], km) == cudaSuccess && cudaMalloc(&s->V[i], km) == cudaSuccess &&
         cudaMalloc(&s->dK[i], km) == cudaSuccess && cudaMalloc(&s->dV[i], km) == cudaSuccess &&
         cudaMalloc(reinterpret_cast<void**>(&s->L[i]), (size_t)chunk_heads * n * 4) ==
             cudaSuccess;
  }
  if (ok) {
    s->ws_bytes = fa_backward_workspace_size(1, chunk_heads, n, m, d);
    ok = cudaMalloc(&s->ws, s->ws_bytes) == cudaSuccess;
  }
  if (!ok) {
    cudaGetLastError();  // clear the failed call's error
    release(s);
    return FA_ERR_CUDA;
  }
  *out = s;
  return FA_OK;
}

void fa_session_destroy(fa_session* s) { release(s); }

int fa_session_submit(fa_session* s, const void* Q, const void* K, const void* V,
                      const void* dO, int causal, float scale, void* O, float* L, void* dQ,
                      void* dK, void* dV) {
  if (!s || !Q || !K || !V || !dO || !O || !L || !dQ || !dK || !dV) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev != s->device) return FA_ERR_INVALID_ARG;
  const int BH = s->B * s->H, n = s->n, m = s->m, d = s->d;
  // chunk sizes: half, full, ..., full, then the rest as two halves when it is a
  // full chunk (all at most s->chunk heads)
  const int half = (s->chunk + 1) / 2;
  const auto* hq = static_cast<const uint8_t*>(Q);
  const auto* hk = static_cast<const uint8_t*>(K);
  const auto* hv = static_cast<const uint8_t*>(V);
  const auto* hdo = static_cast<const uint8_t*>(dO);
  auto* ho = static_cast<uint8_t*>(O);
  auto* hdq = static_cast<uint8_t*>(dQ);
  auto* hdk = static_cast<uint8_t*>(dK);
  auto* hdv = static_cast<uint8_t*>(dV);
  int rc = FA_OK;
  for (int c = 0, h0 = 0; rc == FA_OK && h0 < BH; ++c) {
    const long long cg = s->chunks++;  // the chunk's number across steps
    const int i = (int)(cg % kSets);
    const int left = BH - h0;
    int hc = c == 0 ? half : s->chunk;
    if (left <= s->chunk) hc = (left > half && c > 0) ? left - half : left;  // end with a half chunk
    if (hc > left) hc = left;
    const size_t qoff = (size_t)h0 * n * d * 2, koff = (size_t)h0 * m * d * 2;
    const size_t qn = (size_t)hc * n * d * 2, km = (size_t)hc * m * d * 2;
    // copies in, once the copies out of the chunk that last used this set are done
    if (cg >= kSets && cudaStreamWaitEvent(s->in, s->ev_out[i], 0) != cudaSuccess) rc = FA_ERR_CUDA;
    if (rc == FA_OK) rc = copy_in(s->Q[i], hq + qoff, qn, s->in);
    if (rc == FA_OK) rc = copy_in(s->K[i], hk + koff, km, s->in);
    if (rc == FA_OK) rc = copy_in(s->V[i], hv + koff, km, s->in);
    if (rc == FA_OK) rc = copy_in(s->dO[i], hdo + qoff, qn, s->in);
    if (rc == FA_OK && cudaEventRecord(s->ev_in[i], s->in) != cudaSuccess) rc = FA_ERR_CUDA;
    // kernels
    if (rc == FA_OK && cudaStreamWaitEvent(s->comp, s->ev_in[i], 0) != cudaSuccess)
      rc = FA_ERR_CUDA;
    if (rc == FA_OK)
      rc = fa_forward(s->Q[i], s->K[i], s->V[i], 1, hc, n, m, d, causal, scale, s->O[i], s->L[i],
                      s->comp);
    if (rc == FA_OK)
      rc = fa_backward(s->Q[i], s->K[i], s->V[i], s->O[i], s->L[i], s->dO[i], 1, hc, n, m, d,
                       causal, scale, s->dQ[i], s->dK[i], s->dV[i], s->ws, s->ws_bytes, s->comp);
    if (rc == FA_OK && cudaEventRecord(s->ev_comp[i], s->comp) != cudaSuccess) rc = FA_ERR_CUDA;
    // copies out
    if (rc == FA_OK && cudaStreamWaitEvent(s->out, s->ev_comp[i], 0) != cudaSuccess)
      rc = FA_ERR_CUDA;
    if (rc == FA_OK) rc = copy_out(ho + qoff, s->O[i], qn, s->out);
    if (rc == FA_OK) rc = copy_out(L + (size_t)h0 * n, s->L[i], (size_t)hc * n * 4, s->out);
    if (rc == FA_OK) rc = copy_out(hdq + qoff, s->dQ[i], qn, s->out);
    if (rc == FA_OK) rc = copy_out(hdk + koff, s->dK[i], km, s->out);
    if (rc == FA_OK) rc = copy_out(hdv + koff, s->dV[i], km, s->out);
    if (rc == FA_OK && cudaEventRecord(s->ev_out[i], s->out) != cudaSuccess) rc = FA_ERR_CUDA;
    h0 += hc;
  }
  return rc;
}

int fa_session_sync(fa_session* s) {
  if (!s) return FA_ERR_INVALID_ARG;
  const bool synced = cudaStreamSynchronize(s->in) == cudaSuccess &&
                      cudaStreamSynchronize(s->comp) == cudaSuccess &&
                      cudaStreamSynchronize(s->out) == cudaSuccess;
  return synced ? FA_OK : FA_ERR_CUDA;
}

int fa_session_step(fa_session* s, const void* Q, const void* K, const void* V, const void* dO,
                    int causal, float scale, void* O, float* L, void* dQ, void* dK, void* dV) {
  int rc = fa_session_submit(s, Q, K, V, dO, causal, scale, O, L, dQ, dK, dV);
  // whatever was queued finishes before the call returns (the host buffers are the caller's)
  if (s) {
    const int rs = fa_session_sync(s);
    if (rc == FA_OK) rc = rs;
  }
  return rc;
}

}  // extern "C"
