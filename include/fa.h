/*
 * fa.h — exact scaled-dot-product attention for training on sm_103a (GB300).
 *
 * C ABI of libfa_gb300.so: a forward pass that caches the per-row log-sum-exp
 * (LSE), and its vector-Jacobian product (VJP) split into a D-vector
 * preprocess, a dK/dV kernel and a dQ kernel that recompute P per tile from
 * the cached LSE.
 *
 * The operation (page "mlx-bun 0.0.4: package/src/model/flash-attention.ts",
 * forward shader and backward passes 1-3; page "[Metal] Add Flash Attention
 * VJP for training", Implementation Notes):
 *
 *   S[i,j] = scale * Q[b,h,i,:] . K[b,g,j,:]          g = h / (Hq / Hkv)
 *   a key j is hidden from query i when
 *       (causal && j > i)  or  (window > 0 && i >= j && i - j >= window)
 *   LSE[i] = ln sum_{j visible} exp(S[i,j]);   P[i,j] = exp(S[i,j] - LSE[i])
 *   O[i,:] = sum_j P[i,j] V[b,g,j,:]
 *   D[i]   = sum_d dO[i,d] O[i,d]
 *   dS     = P o (dO V^T - D)
 *   dQ = scale * dS K;  dK = scale * sum_{h in group} dS^T Q;  dV = sum_{h in group} P^T dO
 *
 * Conventions shared by every entry point:
 *  - Q, O, dO, dQ are [B, Hq, Tq, D]; K, V, dK, dV are [B, Hkv, Tkv, D];
 *    LSE is [B, Hq, Tq]. All are dense row-major (innermost index last) device
 *    buffers in HBM, owned by the caller, 16-byte aligned.
 *  - Element type: fp16 or bf16 (fa_dtype) for Q, K, V, O, dO, dQ, dK, dV;
 *    LSE is fp32 in natural log. Arithmetic: fp32 accumulation on the tensor
 *    cores, fp32 softmax statistics, round-to-nearest-even on every store.
 *  - Grouped-query attention: Hq must be a multiple of Hkv; consecutive query
 *    heads share a KV head (g = h / (Hq / Hkv)).
 *  - causal is 0 or 1; with Tq != Tkv the causal mask is aligned at the top
 *    left (query i sees keys 0..i), as in page "R/ag_flash_attn.R" (ggmlR),
 *    mask builder. window >= 0 (0 = no window): the window hides only past
 *    keys, so a query sees `window` keys of its past including its own
 *    position; without causal, future keys stay visible.
 *  - A query row that sees no key at all (only possible with a window and
 *    Tq > Tkv) gets O = 0, LSE = -inf, dQ = 0 and adds nothing to dK/dV.
 *  - head_dim D is one of 64, 96, 128, 256. scale must be finite and > 0.
 *  - Outputs are fully overwritten; the caller need not zero them. Outputs
 *    must not overlap inputs or each other.
 *  - The library never allocates or frees memory. Calls are asynchronous on
 *    `stream` (0 = the legacy default stream); results are ready when the
 *    stream reaches the point after the call.
 *  - Arguments are validated before anything is launched; a bad argument
 *    returns an error code and launches nothing. A launch failure returns
 *    FA_ERR_LAUNCH. Errors never abort the process.
 *  - Every wait inside the kernels is bounded (default 4 s, environment
 *    variable FA_WAIT_TIMEOUT_MS overrides). A wait that gives up sets a bit
 *    in a device status word, the kernel runs to its exit without further
 *    waiting, and fa_device_status() reports FA_ERR_TIMEOUT.
 */
#ifndef FA_GB300_H_
#define FA_GB300_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,          /* null pointer, bad size, overlap, bad scale/mask */
  FA_ERR_UNSUPPORTED_HEAD_DIM = 2, /* D not in {64, 96, 128, 256} */
  FA_ERR_UNSUPPORTED_DTYPE = 3,    /* dtype not FA_FP16 / FA_BF16 */
  FA_ERR_MISALIGNED = 4,           /* a buffer is not 16-byte aligned */
  FA_ERR_LAUNCH = 5,               /* a CUDA launch or driver call failed */
  FA_ERR_TIMEOUT = 6               /* a bounded device wait gave up */
} fa_status;

typedef enum { FA_FP16 = 0, FA_BF16 = 1 } fa_dtype;

/* Forward pass (page "mlx-bun 0.0.4: package/src/model/flash-attention.ts",
 * forward shader; online softmax that never materialises S).
 *   q [B,Hq,Tq,D], k/v [B,Hkv,Tkv,D]   inputs, dtype `dt`
 *   o [B,Hq,Tq,D]                      output, dtype `dt`
 *   lse [B,Hq,Tq]                      output, fp32 natural-log LSE (kept for fa_bwd)
 * Sizes: B, Hq, Hkv, Tq, Tkv >= 1; Tq, Tkv <= 2^22; B * Hq <= 2^24.
 * One kernel launch. Tq <= 8 (decode-shaped calls) runs a split-key kernel
 * that launches thread-block clusters of up to 8 CTAs; longer query blocks run
 * the tensor-core tile kernel. Both compute the same result; which one runs
 * changes only the rounding of the fp32 sums.
 * The kernel is launched with programmatic stream serialisation: its launch
 * and set-up overlap the end of the previous kernel in `stream`, and it
 * waits for that kernel to complete before it reads or writes global memory.
 * So stream order is what the caller sees.
 * Returns FA_OK or an error code (nothing launched on error). */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int Hq, int Hkv, int Tq, int Tkv, int D, float scale,
                 int causal, int window, fa_dtype dt, cudaStream_t stream);

/* Bytes of device workspace fa_bwd needs: the fp32 D-vector [B,Hq,Tq]
 * rounded up to 256 bytes. Returns 0 for non-positive sizes. */
size_t fa_bwd_workspace_size(int B, int Hq, int Tq);

/* Backward pass / VJP (page "mlx-bun 0.0.4: package/src/model/
 * flash-attention.ts", backward passes 1-3; page "[Metal] Add Flash Attention
 * VJP for training", Implementation Notes: two kernels, KV-row ownership so
 * grouped heads reduce without atomics). Launches, in order on `stream`:
 *   1. D-vector preprocess  D = rowsum(dO o O)   (from the stored O)
 *   2. dK/dV kernel (one CTA, or a cluster of CTAs sharing the tiles, owns a
 *      block of KV rows and loops over every query head of its group and
 *      every query tile that can see it; Tq <= 8: a kernel that sums over
 *      every query row of the group in fp32 per key row, any mask)
 *   3. dQ kernel (one CTA owns a block of query rows, loops over KV tiles;
 *      Tq <= 8: a split-key kernel over thread-block clusters of up to 8 CTAs)
 * Which kernels run changes only the rounding order of the fp32 sums.
 * Ordering: as for fa_fwd, each kernel is launched to overlap the end of the
 * previous kernel in `stream` (programmatic stream serialisation). It waits
 * for that kernel before it reads or writes global memory, so stream order
 * holds for the caller. On causal, windowed and Tq <= 8 calls, the dQ kernel
 * starts without waiting for the dK/dV kernel: it needs only the D-vector.
 * It waits for dK/dV before it completes, so work queued after fa_bwd on
 * `stream` still sees all three outputs written.
 *   q, k, v, o, dO, lse       inputs (o and lse as written by fa_fwd)
 *   dq [B,Hq,Tq,D], dk/dv [B,Hkv,Tkv,D]  outputs, dtype `dt`
 *   workspace                 caller-owned device scratch of at least
 *                             fa_bwd_workspace_size(B,Hq,Tq) bytes, 16-byte
 *                             aligned; its contents are overwritten.
 * The gradient with respect to LSE is not an input: it is taken as zero.
 * Returns FA_OK or an error code (nothing launched on error). */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                 const float* lse, void* dq, void* dk, void* dv,
                 int B, int Hq, int Hkv, int Tq, int Tkv, int D, float scale,
                 int causal, int window, fa_dtype dt, void* workspace, size_t workspace_bytes,
                 cudaStream_t stream);

/* The three launches of fa_bwd as separate calls, for callers that schedule
 * them themselves (e.g. dK/dV and dQ on two streams once the D-vector is
 * ready) or time them one by one. `dvec` is the D-vector workspace:
 * [B,Hq,Tq] fp32, 16-byte aligned, at least fa_bwd_workspace_size bytes.
 * fa_bwd_preprocess (backward pass 1 of the mlx-bun flash-attention.ts page):
 *   dvec[i] = sum_d dO[i,d] O[i,d]   (fp32 accumulation of the stored O)
 * fa_bwd_dkv (backward pass 2): dk, dv from q, k, v, dO, lse, dvec.
 * fa_bwd_dq  (backward pass 3): dq from q, k, v, dO, lse, dvec.
 * Same argument rules and error behaviour as fa_bwd. */
fa_status fa_bwd_preprocess(const void* o, const void* dO, float* dvec, int B, int Hq, int Tq,
                            int D, fa_dtype dt, cudaStream_t stream);
fa_status fa_bwd_dkv(const void* q, const void* k, const void* v, const void* dO,
                     const float* lse, const float* dvec, void* dk, void* dv,
                     int B, int Hq, int Hkv, int Tq, int Tkv, int D, float scale,
                     int causal, int window, fa_dtype dt, cudaStream_t stream);
fa_status fa_bwd_dq(const void* q, const void* k, const void* v, const void* dO,
                    const float* lse, const float* dvec, void* dq,
                    int B, int Hq, int Hkv, int Tq, int Tkv, int D, float scale,
                    int causal, int window, fa_dtype dt, cudaStream_t stream);

/* fa_bwd without a workspace argument, for callers that cannot allocate any
 * device memory: a plug-in inside a host program that owns every device
 * allocation, or a loop that may not call the allocator (which can
 * synchronise the device) once it runs. The pages have no counterpart of
 * this call; it exists for such callers only.
 * The D-vector goes to a fixed 4 MiB array inside the library instead of a
 * caller buffer: B * Hq * Tq must not exceed fa_bwd_noalloc_max_rows()
 * (2^20), else FA_ERR_INVALID_ARG and nothing is launched. Every other
 * argument, layout and error rule is that of fa_bwd.
 * The array is one per device, shared by every call on that device and kept
 * until the process exits; it holds the last call's D-vector. Calls whose
 * launches overlap on the GPU (two streams, or two host threads) race on it:
 * keep them ordered on one stream. The first call on a device (with that
 * device current) looks up the array's device address, which is set-up work:
 * make that first call before any stream capture. The address belongs to the
 * device's CUDA context; after cudaDeviceReset() the next call finds a new
 * context and looks the address up again (so, after a reset, that call is
 * again a first call). Nothing in the array has to start at zero: each call
 * rewrites the part it uses before reading it. */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const void* dO, const float* lse, void* dq, void* dk, void* dv,
                         int B, int Hq, int Hkv, int Tq, int Tkv, int D, float scale,
                         int causal, int window, fa_dtype dt, cudaStream_t stream);

/* Largest B * Hq * Tq that fa_bwd_noalloc accepts. */
size_t fa_bwd_noalloc_max_rows(void);

/* Human-readable name of a status code (static storage; never NULL). */
const char* fa_status_string(fa_status s);

/* Read the device status word on the current device after synchronising
 * `stream`. *bits receives the raw word (bit 0: a bounded wait gave up); when
 * `clear` is non-zero the word is reset to 0 afterwards. Returns FA_OK when
 * the word is 0, FA_ERR_TIMEOUT when a wait gave up, FA_ERR_LAUNCH when the
 * read itself failed. */
fa_status fa_device_status(unsigned int* bits, int clear, cudaStream_t stream);

/* Self-test of the bounded waits (a library check; the pages have no
 * counterpart). Launches one small kernel on `stream` in which one warp waits
 * on an mbarrier that can never complete, with a limit of `timeout_ms`
 * milliseconds, and a second warp waits on another such barrier with four
 * times that limit. The first wait gives up, sets FA_ERR_TIMEOUT's bit in the
 * device status word and raises the kernel's abort flag, which lets the second
 * warp leave at once; the kernel then exits normally and the context stays
 * usable. Read the result with fa_device_status(). Returns FA_OK once the
 * kernel is launched, FA_ERR_INVALID_ARG for timeout_ms outside 1..10000,
 * FA_ERR_LAUNCH on a launch failure. */
fa_status fa_selftest_wait_timeout(unsigned int timeout_ms, cudaStream_t stream);

/* Bound, in SM clock cycles, of the ordinary waits of every kernel launched
 * after this call by any host thread of the process (a library diagnostic for
 * tests of the give-up path; the pages have no counterpart). 0 restores the
 * default (FA_WAIT_TIMEOUT_MS, else 4 s). With a bound of a few cycles the
 * first wait of each kernel gives up: the kernel sets FA_ERR_TIMEOUT's bit in
 * the device status word and runs to its exit. The waits at exit that let
 * copies and MMAs already in flight finish keep the default bound, so no CTA
 * leaves with work outstanding; outputs of such a call are undefined. Calls
 * made after restoring the default compute normally. Always returns FA_OK. */
fa_status fa_set_wait_limit_cycles(unsigned long long cycles);

/* Version of this ABI (major * 100 + minor). */
int fa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H_ */
