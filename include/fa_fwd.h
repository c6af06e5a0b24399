/* fa_fwd.h -- C ABI of libfa: exact fused attention forward on one GB300 (sm_103a).
 *
 * The operation (per batch b, head h, query row i):
 *     s_ij = scale * <Q[b,h,i,:], K[b,h,j,:]>            for key j in [0, Nk)
 *     s_ij = -inf  if causal and j > i                  (top-left aligned mask)
 *     O[b,h,i,:] = sum_j softmax_j(s_i.) V[b,h,j,:]
 *     L[b,h,i]   = ln sum_j exp(s_ij)                   (natural-log logsumexp)
 * as defined on the CS336 lecture 5 page "05_flash_attention.py", part 2
 * ("FlashAttention 前向": standard_attention and flash_attention_forward, which
 * returns (O, L) with L = m + log(l)), with the scale tau of Algorithm 2 on the
 * "Flash Attention" page (blog.cyberangel.work). The kernel evaluates it tile by
 * tile with the online-softmax statistics (m, l) and an unnormalised output
 * accumulator; the Nq x Nk scores and probabilities never reach global memory.
 *
 * Precision: Q, K, V, O are fp16 or bf16; products are accumulated in fp32; the
 * probabilities fed to the second product are rounded to the input type; L is fp32.
 */
#ifndef FA_FWD_H
#define FA_FWD_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of Q, K, V and O. */
typedef enum { FA_F16 = 0, FA_BF16 = 1 } fa_dtype;

/* Status codes. 0 = success; every error is negative. */
enum {
  FA_OK = 0,
  FA_ERR_NULL = -1,        /* a required pointer is NULL                                  */
  FA_ERR_HEAD_DIM = -2,    /* d is not 64 or 128                                          */
  FA_ERR_SHAPE = -3,       /* B, H, Nq or Nk negative, or B*H*N too large                  */
  FA_ERR_EMPTY_KEYS = -4,  /* Nk == 0 while there are query rows: softmax of an empty row */
  FA_ERR_SCALE = -5,       /* scale is negative, NaN or infinite                          */
  FA_ERR_ALIGN = -6,       /* Q, K, V or O not 16-byte aligned, or L not 4-byte aligned   */
  FA_ERR_DTYPE = -7,       /* dtype is not FA_F16 or FA_BF16                              */
  FA_ERR_CUDA = -8,        /* a CUDA runtime call or the kernel launch failed             */
  FA_ERR_TENSOR_MAP = -9,  /* the driver rejected a TMA tensor map for these arguments    */
  FA_ERR_DEVICE = -10,     /* the current device is not an sm_103 GPU                     */
  FA_ERR_TIMEOUT = -11,    /* device-side: a pipeline wait exceeded its time limit        */
  FA_ERR_WORKSPACE = -12,  /* fa_fwd_ws: workspace missing or too small                   */
  FA_ERR_SCRATCH_LIMIT = -13, /* fa_fwd_noalloc: needs more than FA_NOALLOC_SCRATCH_BYTES  */
  FA_ERR_DROPOUT = -14,    /* dropout probability negative, not finite or too close to 1  */
  FA_ERR_RANGE = -15,      /* an argument outside its documented range                    */
  FA_ERR_BOUNDS = -16      /* device-side, debug builds only (FA_DEBUG): a workspace index
                              outside its layout; the access was skipped                  */
};

/* Limits of fa_set_wait_limit_us, in microseconds: the default (2 s), the smallest and the
 * largest accepted value (100 us and one hour). */
#define FA_WAIT_LIMIT_DEFAULT_US 2000000ull
#define FA_WAIT_LIMIT_MIN_US 100ull
#define FA_WAIT_LIMIT_MAX_US 3600000000ull

/* Size of the fixed device scratch array behind fa_fwd_noalloc (48 MiB). */
#define FA_NOALLOC_SCRATCH_BYTES (48u << 20)

/* fa_fwd -- launch the attention forward pass on `stream`.
 *
 * Arguments (all pointers are DEVICE pointers owned by the caller):
 *   Q      [B, H, Nq, d]  dense row-major, element type `dtype`, 16-byte aligned
 *   K, V   [B, H, Nk, d]  dense row-major, element type `dtype`, 16-byte aligned
 *   O      [B, H, Nq, d]  output, dense row-major, `dtype`, 16-byte aligned
 *   L      [B, H, Nq]     output, fp32, natural-log logsumexp of each score row
 *   d      head dimension, 64 or 128
 *   scale  multiplies Q K^T before the softmax (1/sqrt(d) in the usual use); >= 0
 *   causal non-zero: query i sees key j iff j <= i (top-left aligned when Nq != Nk,
 *          so every query row sees at least key 0)
 *   stream a cudaStream_t (NULL = the legacy default stream)
 *
 * Layout: no padding; row i of head (b, h) of Q starts at element ((b*H + h)*Nq + i)*d.
 * Ownership: calls allocate no device memory and keep no pointer after return. (Every
 *   device that loads the library does hold one fixed array of FA_NOALLOC_SCRATCH_BYTES,
 *   the scratch of fa_fwd_noalloc, until the process exits; fa_fwd never touches it.)
 * Timing: asynchronous. Returns FA_OK once the launch is queued; O and L are valid
 *   after `stream` is synchronised. Calls on different streams that write the same
 *   O/L race.
 * Errors: argument checks happen on the host before any CUDA call and return the
 *   FA_ERR_* code without touching the device. B == 0, H == 0 or Nq == 0 is a no-op
 *   that returns FA_OK (pointers are not inspected). A failed CUDA call returns
 *   FA_ERR_CUDA (the CUDA error is then readable with cudaGetLastError). Device-side
 *   failures (a wait timeout) are reported by fa_last_status().
 */
int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* L,
           int B, int H, int Nq, int Nk, int d, float scale, int causal,
           fa_dtype dtype, void* stream);

/* fa_fwd_workspace_bytes -- size in bytes of the workspace fa_fwd_ws needs for these
 * sizes on the CURRENT device (it depends on the device's SM count), or 0 when the call
 * needs none (causal attention, item counts that fill whole waves of SMs, or invalid
 * sizes). No device memory is touched.
 *
 * fa_fwd_ws -- fa_fwd with a caller-provided device workspace that lets full (non-causal)
 * attention split the key range of work items across CTAs so that every SM gets the same
 * number of K/V tiles ("stream-K"): a CTA that covers only part of an item's keys stores
 * the item rows' partial state (m, l, unnormalised O) in the workspace; the CTA that
 * completes a query tile's key range merges the partial states with the associative
 * combine of the online softmax ("Flash Attention" page, section "平行化") and writes O and
 * L. The partial states are combined in a fixed order, so results do not depend on which
 * CTA finishes last.
 * Same arguments, layout and results as fa_fwd (up to rounding order), plus:
 *   workspace       device pointer, 256-byte aligned, at least fa_fwd_workspace_bytes()
 *                   bytes, ZERO-FILLED before its first use; every completed call leaves
 *                   it zero-filled again (re-zero it after a call that failed on the
 *                   device, e.g. FA_ERR_TIMEOUT). NULL is allowed when the size is 0.
 *   workspace_bytes its size.
 * Calls that share a workspace must not overlap on the GPU. Returns FA_ERR_WORKSPACE when
 * the workspace is missing or too small, FA_ERR_ALIGN when it is misaligned. */
size_t fa_fwd_workspace_bytes(int B, int H, int Nq, int Nk, int d, int causal);
int fa_fwd_ws(const void* Q, const void* K, const void* V, void* O, float* L,
              int B, int H, int Nq, int Nk, int d, float scale, int causal,
              fa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/* fa_fwd_noalloc -- fa_fwd_ws for callers that cannot allocate device memory.
 *
 * The method this library implements has no counterpart for this entry point; it exists
 * for programs that must not call cudaMalloc from inside a library: hosts that hand the
 * whole device to their own memory pool at start-up, runtimes with a fixed memory budget
 * that must not grow, and latency-sensitive paths where an allocation (which may
 * synchronise the device or fail under memory pressure) is not acceptable.
 *
 * Same arguments, results and errors as fa_fwd. Full (non-causal) attention whose work
 * items do not fill whole waves of SMs is split across CTAs exactly like fa_fwd_ws, with
 * the workspace taken from one file-scope device array of FA_NOALLOC_SCRATCH_BYTES that
 * every device which loads the library holds until the process exits. Nothing is
 * allocated: no cudaMalloc, cudaFree or allocating library routine is called.
 *   - The first call on a device looks up that array's device address (once per device,
 *     with the device current); make that first call before any stream capture.
 *   - Each call clears the part of the array that must start at zero (with
 *     cudaMemsetAsync on `stream`) before its launch.
 *   - All calls share the array: calls that overlap on the GPU (different streams, or
 *     different host threads) race and give wrong results; serialise them.
 *   - Returns FA_ERR_SCRATCH_LIMIT, without launching anything, when the sizes need more
 *     scratch than the array holds (fa_fwd_workspace_bytes() tells how much they need).
 * Causal attention and problems that need no split use no scratch at all. */
int fa_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* L,
                   int B, int H, int Nq, int Nk, int d, float scale, int causal,
                   fa_dtype dtype, void* stream);

/* fa_fwd_host -- fa_fwd on HOST buffers: Q, K, V are read from and O, L written to host
 * memory, with the copies overlapped with the computation.
 * The heads are processed in chunks that stream through a ring of up to 4 device slots in
 * `workspace`: chunks of enough heads for copies of at least 8 MB per tensor (where there
 * are that many heads), the last one a quarter of that size. Library streams carry the work: one takes every host-to-device
 * copy, one every device-to-host copy (so both directions run at once), and each slot
 * has one for its attention launches. Events chain them per slot: inputs in, launch,
 * outputs out, slot free for the next chunk.
 * Same results, arguments and errors as fa_fwd, except:
 *   Q, K, V, O, L  HOST pointers, same layout and alignment as fa_fwd. Make them
 *                  page-locked (cudaHostAlloc / cudaHostRegister), or the copies cannot
 *                  overlap the computation (the results are the same either way).
 *   workspace      DEVICE pointer, 256-byte aligned, at least fa_fwd_host_workspace_bytes()
 *                  bytes (no initialisation needed).
 *   stream         the library's streams start after the work queued on `stream` so far,
 *                  and `stream` waits for them: O and L are in host memory once `stream`
 *                  has been synchronised.
 * Calls from several host threads on one device are serialised while they queue their
 * work (the library's streams are shared); calls that overlap on the GPU need their own
 * workspaces and host buffers that do not alias. FA_ERR_WORKSPACE for a missing or small
 * workspace. */
size_t fa_fwd_host_workspace_bytes(int B, int H, int Nq, int Nk, int d);
int fa_fwd_host(const void* Q, const void* K, const void* V, void* O, float* L,
                int B, int H, int Nq, int Nk, int d, float scale, int causal,
                fa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/* fa_fwd_dropout -- the forward pass with dropout on the attention probabilities
 * ("Flash Attention" page, "Algorithm 2": P_dropped = dropout(P, p_drop), O = P_dropped V;
 * the forward returns the generator state, here the pair (seed, offset)):
 *     O[b,h,i,:] = sum_j P_ij Z_ij V[b,h,j,:],   L as in fa_fwd (undropped logsumexp)
 * with Z_ij = 256 / (256 - t) when element (i, j) is kept and 0 when it is dropped.
 * The mask (the pages name no generator; this is the library's definition):
 *   t = floor(p_drop * 256 + 0.5), an 8-bit threshold (p_drop is used to 1/256);
 *   with bh = b*H + h, the counter-based generator Philox-4x32-10 (Salmon, Moraes, Dror,
 *   Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11) is evaluated at
 *     counter (j >> 4, i, bh, offset), key (seed & 0xFFFFFFFF, seed >> 32)
 *   giving four 32-bit words w[0..3]; key j draws the byte x = byte number
 *   2 (j & 1) + ((j >> 1) & 1) of w[(j >> 2) & 3] (bytes counted from the least
 *   significant), and element (i, j) is kept iff x >= t.
 * Calls with the same (seed, offset) and sizes draw the same mask; use a new offset (or
 * seed) for every call that needs an independent mask.
 * Arguments, layout, ownership and errors as fa_fwd, plus FA_ERR_DROPOUT when p_drop is
 * negative, NaN, infinite, or at least 1 - 2^-9 (t would be 256: nothing kept).
 * p_drop small enough that t = 0 runs fa_fwd (nothing dropped, identical results). */
int fa_fwd_dropout(const void* Q, const void* K, const void* V, void* O, float* L,
                   int B, int H, int Nq, int Nk, int d, float scale, int causal,
                   fa_dtype dtype, float p_drop, unsigned long long seed, unsigned int offset,
                   void* stream);

/* fa_fwd_fp8 -- the forward pass on FP8 inputs (E4M3, the OCP 8-bit format with 4 exponent
 * and 3 mantissa bits, no infinities, |x| <= 448) with per-tensor descale factors, the
 * FP8 attention of FlashAttention-3 that the "手写 Flash Attention" page names in its
 * sections 6.1 and 7 (the pages give no further definition; this is the library's):
 *     O = v_descale * softmax(scale * q_descale * k_descale * Q K^T [+causal]) V
 *     L = ln sum_j exp(scale * q_descale * k_descale * <Q_i, K_j>)
 * with Q, K, V decoded exactly from E4M3. Products accumulate in fp32; the probabilities
 * fed to the second product are rounded to E4M3 (round to nearest even, as FlashAttention-3
 * does), relative to the running row maximum; O is written as `out_dtype` (FA_BF16 or FA_F16).
 * Arguments (DEVICE pointers, 16-byte aligned, dense row-major):
 *   Q [B, H, Nq, d], K and V [B, H, Nk, d]   E4M3 bytes; d must be 128
 *   O [B, H, Nq, d] out_dtype;  L [B, H, Nq] fp32 (natural log)
 *   q_descale, k_descale, v_descale  finite and > 0 (1 when the inputs are unscaled)
 *   workspace  at least fa_fwd_fp8_workspace_bytes(B, H, Nk, d) bytes, 16-byte aligned, no
 *              initialisation: it receives V^T ([B, H, d, Nk rounded up to 16], keys
 *              contiguous), which a first kernel writes and the attention kernel reads as
 *              its K-major operand
 * scale, causal and stream as in fa_fwd. Two kernels are queued on `stream`.
 * Errors as fa_fwd (FA_ERR_DTYPE for an out_dtype other than FA_F16/FA_BF16, FA_ERR_HEAD_DIM
 * for d != 128, FA_ERR_SCALE for a bad descale), plus FA_ERR_WORKSPACE for a missing or
 * small workspace. */
size_t fa_fwd_fp8_workspace_bytes(int B, int H, int Nk, int d);
int fa_fwd_fp8(const void* Q, const void* K, const void* V, void* O, float* L,
               int B, int H, int Nq, int Nk, int d, float scale, int causal,
               float q_descale, float k_descale, float v_descale, fa_dtype out_dtype,
               void* workspace, size_t workspace_bytes, void* stream);

/* fa_dropout_mask -- write the keep mask that fa_fwd_dropout uses for these arguments:
 * keep [B, H, Nq, Nk] bytes (DEVICE pointer, caller-owned), 1 = kept, 0 = dropped.
 * Causality does not enter the mask (masked-out keys have P = 0 either way). One kernel
 * on `stream`; same mask definition and errors as fa_fwd_dropout (FA_ERR_NULL for a NULL
 * `keep` when there is something to write; sizes of 0 are a no-op). */
int fa_dropout_mask(unsigned char* keep, int B, int H, int Nq, int Nk, float p_drop,
                    unsigned long long seed, unsigned int offset, void* stream);

/* fa_bwd -- gradients of the forward pass: dQ, dK, dV for the upstream gradient dO
 * (CS336 lecture 5 "05_flash_attention.py", part 3, flash_attention_backward; "Flash
 * Attention" page, "Algorithm 4: backward pass"): with S = scale Q K^T (masked as in the
 * forward) and P = exp(S - L) recomputed from the forward's logsumexp L,
 *     dV = P^T dO,  dP = dO V^T,  D_i = rowsum(dO_i o O_i),  dS = P o (dP - D),
 *     dQ = scale dS K,  dK = scale dS^T Q.
 * Arguments (DEVICE pointers, dense row-major, 16-byte aligned, element type `dtype`):
 *   Q, O, dO, dQ  [B, H, Nq, d];  K, V, dK, dV  [B, H, Nk, d]
 *   L             [B, H, Nq] fp32, the natural-log logsumexp fa_fwd wrote with O
 *   workspace     at least fa_bwd_workspace_bytes() bytes, 16-byte aligned, no
 *                 initialisation needed (it receives D, one fp32 per query row)
 * d, scale, causal, dtype and stream as in fa_fwd. Two kernels are queued on `stream`
 * (query tiles: D and dQ; then key tiles: dK and dV); nothing is accumulated with atomics.
 * dS is rounded to the input type before the products that use it, P before dV.
 * Errors as fa_fwd, plus FA_ERR_WORKSPACE for a missing or small workspace. */
size_t fa_bwd_workspace_bytes(int B, int H, int Nq, int Nk, int d);
int fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
           const float* L, void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nk, int d,
           float scale, int causal, fa_dtype dtype, void* workspace, size_t workspace_bytes,
           void* stream);

/* fa_bwd_dropout -- the backward pass of fa_fwd_dropout ("Flash Attention" page,
 * "Algorithm 4": the mask Z is regenerated from the forward's generator state, here
 * (p_drop, seed, offset), which must be the forward call's):
 *     dV = (P o Z)^T dO,  dP = (dO V^T) o Z,  D_i = rowsum(dO_i o O_i),  dS = P o (dP - D),
 *     dQ = scale dS K,  dK = scale dS^T Q
 * with Z_ij = 256 / (256 - t) where fa_fwd_dropout kept (i, j) and 0 where it dropped it
 * (the mask of fa_fwd_dropout). O is the dropout forward's output, L its logsumexp.
 * Arguments, layout, workspace and errors as fa_bwd, plus FA_ERR_DROPOUT for a bad p_drop;
 * p_drop with t = 0 runs fa_bwd. */
int fa_bwd_dropout(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                   const float* L, void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nk,
                   int d, float scale, int causal, fa_dtype dtype, float p_drop,
                   unsigned long long seed, unsigned int offset, void* workspace,
                   size_t workspace_bytes, void* stream);

/* fa_last_status -- synchronise the current device, then return the device-side status
 * word of libfa on that device: FA_OK, or the first error a kernel recorded since the
 * last fa_clear_status() (FA_ERR_TIMEOUT when a bounded pipeline wait gave up; the kernel
 * then returns without finishing and O/L are undefined). Returns FA_ERR_CUDA if the
 * synchronisation itself fails. */
int fa_last_status(void);

/* fa_stream_status -- the same status word, read once the work already queued on `stream`
 * (NULL: the legacy default stream) has finished; other streams are not waited for. The
 * word is shared by every launch of libfa on the device, so it may also hold an error that
 * a kernel on another stream recorded. Returns the status, or FA_ERR_CUDA if the read or the
 * stream synchronisation fails. */
int fa_stream_status(void* stream);

/* fa_clear_status -- reset the device-side status word of the current device to FA_OK.
 * Returns FA_OK or FA_ERR_CUDA. */
int fa_clear_status(void);

/* fa_strerror -- static, human-readable text for a status code (never NULL). */
const char* fa_strerror(int code);

/* fa_selftest_wait_timeout -- exercise the bounded-wait failure path without any fault:
 * launches one CTA on `stream` that waits on a pipeline barrier nothing ever signals,
 * with a wait limit of `limit_us` microseconds (1..1000000). The wait gives up, records
 * FA_ERR_TIMEOUT in the status word and the kernel returns normally; the context stays
 * usable. Returns FA_OK once queued, FA_ERR_SHAPE for a limit out of range, FA_ERR_DEVICE
 * or FA_ERR_CUDA on failure to launch. */
int fa_selftest_wait_timeout(int limit_us, void* stream);

/* fa_set_wait_limit_us -- time limit of every device-side pipeline wait (an mbarrier wait
 * of a kernel role on another role: a TMA copy landing, a tensor-core product completing,
 * a softmax warp handing P over) for the kernels launched after this call, process-wide and
 * on every device. A wait that exceeds it gives up: the kernel records FA_ERR_TIMEOUT (read
 * with fa_last_status), stops every role of its CTA, drains its in-flight copies and
 * products, frees its Tensor Memory and returns; O, L (or the gradients) are then undefined.
 * The default, FA_WAIT_LIMIT_DEFAULT_US (2 s), is hundreds of times the longest legitimate
 * wait of an unshared GPU; callers whose GPU is time-sliced or preempted by other work
 * (where a CTA can be descheduled for longer) raise it. No CUDA call is made.
 *   limit_us  FA_WAIT_LIMIT_MIN_US .. FA_WAIT_LIMIT_MAX_US; anything else returns
 *             FA_ERR_RANGE and leaves the limit unchanged.
 * fa_get_wait_limit_us -- the current limit in microseconds. */
int fa_set_wait_limit_us(unsigned long long limit_us);
unsigned long long fa_get_wait_limit_us(void);

/* fa_debug_cap_workspace -- test hook of the range-checked build (compiled with FA_DEBUG,
 * libfa_debug.so), which checks every stream-K workspace access and every TMA tile
 * coordinate on the device and records FA_ERR_BOUNDS for one outside its range (the access
 * is skipped, or for a load only recorded). In that build, later fa_fwd_ws launches tell the
 * kernel that the partial-state area holds at most `part_elems` floats, so that the checks
 * fire while every access still lies inside the real workspace; a negative value removes
 * the cut. Returns 1 in the range-checked build; the release build ignores the call and
 * returns 0. No CUDA call is made. */
int fa_debug_cap_workspace(long long part_elems);

/* fa_num_kernel_launches -- number of kernels libfa has launched in this process
 * (all devices), for accounting launches in a timed region. */
long long fa_num_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_FWD_H */
