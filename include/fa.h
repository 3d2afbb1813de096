/*
 * Exact, IO-aware softmax attention for NVIDIA GB300 (sm_103a): C-ABI boundary.
 *
 * Operation (from "05_flash_attention.py", standard_attention and
 * flash_attention_forward / flash_attention_backward, and the "Flash
 * Attention" notes, sections 1.1 and 1.5):
 *
 *   forward   S = Q K^T * scale            (score tile, never written to memory)
 *             causal: key k is visible from query q only when k <= q (top-left)
 *             P = softmax(S) row-wise,  O = P V
 *             L = m + log(l)               natural-log logsumexp of each score row
 *   backward  for the loss gradient dO = dLoss/dO:
 *             D = rowsum(dO o O),  P rebuilt as exp(S - L)
 *             dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D)
 *             dQ = dS K * scale,  dK = dS^T Q * scale
 *
 * Layouts. Every tensor is dense and row-major ("contiguous"):
 *   Q, dO, O, dQ : bf16 [B, H, n, d]        K, V, dK, dV : bf16 [B, H, m, d]
 *   L            : fp32 [B, H, n]           (natural log)
 * d is a multiple of 8 from 8 to 128 (64 and 128 are the tuned cases; other
 * values run the next larger of the two with the extra columns read as zeros,
 * which changes no result). n, m, B, H >= 1; B*H <= 65535 and n, m <= 2^24.
 * scale must be finite and > 0 (1/sqrt(d) is the usual choice).
 * All arithmetic accumulates in fp32; O, dQ, dK, dV are rounded to bf16
 * (round to nearest even).
 *
 * Pointers. Every pointer is a device pointer the caller owns (for example
 * memory from torch). bf16 tensors and the workspace must be 16-byte aligned;
 * L must be 4-byte aligned. Outputs must not overlap inputs. The library keeps
 * no pointer after a call returns, allocates no device memory and does not
 * synchronise: work is queued on `stream` (a cudaStream_t; NULL = the legacy
 * default stream) and the call returns once it is queued.
 *
 * Errors. Argument errors are reported before anything is queued and leave the
 * outputs untouched. A launch error maps to FA_ERR_CUDA. The kernels bound
 * every wait on an on-chip barrier; a wait that runs out (about two seconds)
 * makes the kernel stop early and record FA_ERR_DEVICE_TIMEOUT in a device
 * status word, readable with fa_get_device_status() once the stream is
 * synchronised. The outputs of such a call are undefined.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

/* Symbols of this header are the library's only exports. */
#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1,          /* null pointer, bad size, bad scale, overlap */
  FA_ERR_UNSUPPORTED_HEAD_DIM = -2, /* d not a multiple of 8 in [8, 128] */
  FA_ERR_MISALIGNED = -3,           /* a pointer breaks the alignment rules above */
  FA_ERR_UNSUPPORTED_DEVICE = -4,   /* current device is not compute capability 10.3 */
  FA_ERR_WORKSPACE_TOO_SMALL = -5,  /* workspace_bytes < fa_backward_workspace_size() */
  FA_ERR_CUDA = -6,                 /* a CUDA runtime / driver call failed */
  FA_ERR_DEVICE_TIMEOUT = -7        /* a kernel gave up waiting on a barrier */
} fa_status;

/*
 * Forward pass ("05_flash_attention.py", flash_attention_forward; the
 * FlashAttention autograd wrapper's forward saves Q, K, V, O, L).
 * Inputs Q [B,H,n,d], K and V [B,H,m,d] (bf16). Outputs O [B,H,n,d] (bf16) and
 * L [B,H,n] (fp32, natural log). One kernel launch on `stream`.
 * Returns FA_OK or a negative fa_status.
 */
FA_API int fa_forward(const void* Q, const void* K, const void* V, int B, int H, int n, int m,
               int d, int causal, float scale, void* O, float* L, void* stream);

/*
 * Bytes of device workspace fa_backward needs: -D and -L * log2(e) (fp32
 * [B, H, n_pad] each, n_pad = n rounded up to a multiple of 128), 8 bytes per
 * padded query row. m and d are checked but do not change the size. Returns 0
 * for invalid sizes.
 */
FA_API size_t fa_backward_workspace_size(int B, int H, int n, int m, int d);

/*
 * Backward pass ("05_flash_attention.py", flash_attention_backward: the
 * FlashAttention-2 recompute form). Inputs Q, K, V, the forward's O and L, and
 * dO. Outputs dQ [B,H,n,d], dK and dV [B,H,m,d] (bf16). `workspace` is caller
 * owned device memory of at least fa_backward_workspace_size() bytes; its
 * contents on entry do not matter. Queues fa_backward_preprocess and
 * fa_backward_grads on `stream`, in that order.
 */
FA_API int fa_backward(const void* Q, const void* K, const void* V, const void* O, const float* L,
                const void* dO, int B, int H, int n, int m, int d, int causal, float scale,
                void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                void* stream);

/*
 * The three stages of fa_backward, callable one by one (same arguments and
 * rules as fa_backward). fa_backward_dkdv and fa_backward_dq read the workspace
 * fa_backward_preprocess wrote and do not modify it, so they may run in either
 * order once it is complete.
 *
 * fa_backward_preprocess: D = rowsum(dO o O) per query row (the first line of
 *   flash_attention_backward) and L * log2(e) for the recompute, stored
 *   negated, into the workspace. Memory bound.
 * fa_backward_dkdv: per key block, loop over query blocks; rebuild P from L,
 *   accumulate dV = P^T dO and dK = dS^T Q * scale on chip and write them once.
 * fa_backward_dq: per query block, loop over key blocks; rebuild P and dP,
 *   accumulate dQ = dS K * scale on chip and write it once (the pages add dS K
 *   into dQ from inside the key loop; this computes the same sum as its own
 *   pass, with no read-modify-write of dQ in memory).
 * fa_backward_grads: fa_backward_dkdv and fa_backward_dq as one kernel launch
 *   (persistent: each thread block runs its share of the dK/dV blocks, then of
 *   the dQ blocks); what fa_backward queues after the preprocess stage. Results
 *   are bitwise identical to the two separate calls.
 */
FA_API int fa_backward_preprocess(const void* O, const void* dO, const float* L, int B, int H, int n,
                           int d, void* workspace, size_t workspace_bytes, void* stream);
FA_API int fa_backward_dkdv(const void* Q, const void* K, const void* V, const void* dO, int B, int H,
                     int n, int m, int d, int causal, float scale, void* dK, void* dV,
                     void* workspace, size_t workspace_bytes, void* stream);
FA_API int fa_backward_dq(const void* Q, const void* K, const void* V, const void* dO, int B, int H,
                   int n, int m, int d, int causal, float scale, void* dQ, void* workspace,
                   size_t workspace_bytes, void* stream);
FA_API int fa_backward_grads(const void* Q, const void* K, const void* V, const void* dO, int B,
                             int H, int n, int m, int d, int causal, float scale, void* dQ,
                             void* dK, void* dV, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * Backward pass without a caller-supplied workspace (the pages have no
 * counterpart: this entry point exists only for callers that cannot allocate
 * device memory). Same arguments, results and rules as fa_backward, minus
 * `workspace` / `workspace_bytes`.
 *
 * Who needs it: code that owns no device allocator -- for example a plugin or
 * custom operator loaded into a host program that keeps every byte of device
 * memory to itself and offers no allocation hook, or a latency-critical caller
 * that must not call cudaMalloc / cudaFree because they can synchronise the
 * whole device. Such callers still pass their own inputs and outputs.
 *
 * Instead of a caller buffer it uses one statically sized array in device
 * global memory inside this library: FA_NOALLOC_WORKSPACE_BYTES (1 MiB), held
 * on every GPU that loads the library until the process exits. Problems whose
 * workspace (fa_backward_workspace_size, 8 bytes per padded query row) exceeds
 * it are rejected with FA_ERR_WORKSPACE_TOO_SMALL before anything is queued;
 * for example B*H = 64 heads of n = 2048 fit, but B*H = 64 heads of n = 4096
 * do not. This call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 *
 * The first call on a device looks up the array's device address on that
 * device (one cudaGetSymbolAddress, with the device current) and caches it;
 * make that first call before any stream capture. All calls share the one
 * array, which keeps the previous call's contents; every call rewrites or
 * clears all of it that it reads. Calls whose work overlaps on the GPU (for
 * example on two streams without ordering between them) race on the array
 * and give undefined results: order them on one stream or with events.
 */
#define FA_NOALLOC_WORKSPACE_BYTES (1024u * 1024u)
FA_API int fa_backward_noalloc(const void* Q, const void* K, const void* V, const void* O,
                               const float* L, const void* dO, int B, int H, int n, int m, int d,
                               int causal, float scale, void* dQ, void* dK, void* dV,
                               void* stream);

/*
 * Standard (materialised) attention, the baseline of the pages' IO comparison
 * ("05_flash_attention.py", standard_attention and demo_memory): the same O and
 * L as fa_forward, computed the way the pages' standard implementation does it,
 * with the n x m score and probability matrices written to memory.
 *   S = scale * Q K^T  for every (query, key) pair, fp32 accumulation, rounded
 *                      to bf16 and stored to S
 *   P = softmax(S)     per row of the stored S, with the causal mask (key k
 *                      visible from query q iff k <= q, top-left) applied here;
 *                      computed in fp32, rounded to bf16 and stored to P;
 *                      L = logsumexp of the row (natural log, fp32)
 *   O = P V            fp32 accumulation, rounded to bf16
 * Causal masking skips no work: S is computed and stored in full. Q, K, V, O and
 * L are laid out as for fa_forward. S and P are caller-owned device buffers of
 * fa_standard_matrix_bytes(B, H, n, m) bytes each, bf16 [B, H, n, m_pad] with
 * m_pad = m rounded up to a multiple of 64; columns past m hold 0 in P (and in
 * S), and their contents on entry do not matter. Because S and P are rounded to
 * bf16, O and L carry the extra error of those roundings (up to 2^-8 of each
 * score and weight). Same size, alignment (16 bytes; L 4 bytes), aliasing
 * (no output may overlap an input or another output) and device rules as
 * fa_forward; three kernel launches on `stream`. Returns FA_OK or a negative
 * fa_status.
 */
FA_API size_t fa_standard_matrix_bytes(int B, int H, int n, int m);
FA_API int fa_standard_forward(const void* Q, const void* K, const void* V, int B, int H, int n,
                               int m, int d, int causal, float scale, void* S, void* P, void* O,
                               float* L, void* stream);

/*
 * Online softmax statistics ("05_flash_attention.py", online_softmax_stats;
 * "Flash Attention" notes, section 1.1), the building block of the forward pass
 * on its own: for each row of the row-major fp32 matrix x [rows, cols] (device
 * memory), m[r] = max_j x[r, j] and l[r] = sum_j exp(x[r, j] - m[r]), computed in
 * one pass over x with a running maximum and a rescaled sum. m[r] + log l[r] is
 * the row's logsumexp and exp(x[r, j] - m[r]) / l[r] its softmax. Entries may be
 * -inf; a row of -inf only gives m = -inf, l = 0. m and l are fp32 [rows]
 * (device memory, caller owned, not overlapping x or each other); x is read
 * once (16-byte loads when x is 16-byte aligned and cols % 4 == 0). Requires
 * rows, cols >= 1 and 4-byte aligned pointers. The pages' block size only fixes
 * the order of the updates, not the result, so it is not an argument here. One
 * kernel launch on `stream`. Returns FA_OK or a negative fa_status.
 */
FA_API int fa_online_softmax_stats(const float* x, long long rows, long long cols, float* m,
                                   float* l, void* stream);

/*
 * Host-buffer sessions: one forward + backward step whose inputs and outputs are
 * in host memory, for callers that keep their tensors on the host. A session owns
 * device buffers for `chunk_heads` heads at a time (four sets), a backward
 * workspace for one chunk and three CUDA streams (copies in, kernels, copies out)
 * on the device current when it is created.
 *
 * fa_session_step splits the B*H heads into chunks of at most chunk_heads (the
 * first and the last of about half that size, which shortens the pipeline's fill
 * and drain); for each chunk it copies Q, K, V, dO in, runs fa_forward and
 * fa_backward on it, and copies O, L, dQ, dK, dV out, so that the copies of one
 * chunk overlap the kernels of its neighbours and both copy directions run at
 * once. Results equal those of fa_forward + fa_backward on the whole batch (the
 * heads are independent). It returns once every output is in host memory. Host
 * buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for the copies
 * to run asynchronously; pageable buffers work but serialise.
 *
 * fa_session_create: shapes and rules as fa_forward, 1 <= chunk_heads <= B*H.
 * It allocates device memory (the only entry point that does): four sets of
 * chunk_heads x (4 n d + 4 m d) bf16 values and chunk_heads x n fp32, plus one
 * workspace. Returns FA_OK and *out, or a negative fa_status (FA_ERR_CUDA if an
 * allocation fails; nothing is left allocated then).
 * fa_session_destroy: waits for the session's streams and frees everything;
 * NULL is a no-op.
 * fa_session_step: host pointers; inputs Q, dO [B,H,n,d] and K, V [B,H,m,d]
 * bf16; outputs O, dQ [B,H,n,d], dK, dV [B,H,m,d] bf16 and L [B,H,n] fp32. Scale
 * rules as fa_forward. The session's device must be current. Returns FA_OK or
 * the first error; kernel timeouts are reported by fa_get_device_status().
 * The host buffers are the caller's and must hold the sizes above: the library
 * sees only their addresses. A session serves one thread at a time (its streams
 * and buffer sets are not shared safely by concurrent steps); separate sessions
 * may run concurrently.
 * fa_session_submit: the same step, arguments and rules as fa_session_step, but
 * it returns once the step's copies and kernels are queued. Steps submitted one
 * after another continue one pipeline, so a step's copies in run while the
 * previous step's copies out still do, and the link is busy in both directions
 * across step boundaries. Until fa_session_sync returns, the caller must leave
 * the step's input buffers unchanged and must not read or reuse its output
 * buffers for anything else (two submitted steps may share input buffers, and
 * may share output buffers when the caller reads only the last step's results:
 * the copies out run in submission order). Host buffers must be page-locked for
 * the call to return before the copies finish. Returns FA_OK or the first error
 * while queuing; kernel timeouts are reported by fa_get_device_status().
 * fa_session_sync: waits until every step submitted on the session has its
 * outputs in host memory. Returns FA_OK, FA_ERR_INVALID_ARG for a NULL session,
 * or FA_ERR_CUDA. fa_session_step is fa_session_submit followed by
 * fa_session_sync.
 */
typedef struct fa_session fa_session;
FA_API int fa_session_create(int B, int H, int n, int m, int d, int chunk_heads,
                             fa_session** out);
FA_API void fa_session_destroy(fa_session* s);
FA_API int fa_session_step(fa_session* s, const void* Q, const void* K, const void* V,
                           const void* dO, int causal, float scale, void* O, float* L,
                           void* dQ, void* dK, void* dV);
FA_API int fa_session_submit(fa_session* s, const void* Q, const void* K, const void* V,
                             const void* dO, int causal, float scale, void* O, float* L,
                             void* dQ, void* dK, void* dV);
FA_API int fa_session_sync(fa_session* s);

/* A static, human-readable name for a status code. Never NULL. */
FA_API const char* fa_status_string(int status);

/*
 * Reads the device status word of the current device into *status_out
 * (FA_OK; FA_ERR_DEVICE_TIMEOUT if a kernel gave up waiting since the last
 * read; FA_ERR_UNSUPPORTED_DEVICE if a kernel found its shared memory placed
 * other than on a 1024-byte boundary and returned without work) and clears it.
 * Synchronises with the device. Returns FA_OK or FA_ERR_CUDA /
 * FA_ERR_INVALID_ARG.
 */
FA_API int fa_get_device_status(int* status_out);

/* Library version, major * 10000 + minor * 100 + patch. */
FA_API int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
