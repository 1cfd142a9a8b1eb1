/*
 * fa.h -- C ABI of the exact tiled attention library (libfa.so) for NVIDIA
 * GB300 (sm_103a).
 *
 * The operation is exact scaled-dot-product attention, per (batch, head):
 *
 *     S = Q K^T * scale,   P = softmax_row(S),   O = P V,
 *     lse_i = ln sum_j exp(S_ij)
 *
 * as stated in "Flash attention and efficient attention -- Hinglish notes",
 * section "The Standard Attention Problem" (the page's "S / d_k" reads as
 * S / sqrt(d_k): its worked example's 0.707 for d = 2 needs the square root),
 * computed one tile at a time with running max / running sum statistics as in
 * that page's "Derivation: Incremental Softmax" (Steps 1-3) and in "Compute
 * attention one tile at a time" (TensorViz), step "tiles", so the N x N score
 * matrix never reaches device memory.  The optional local window follows the
 * notes' "Worked example Local Attention Window": query i attends to key j
 * iff |i - j| <= (window - 1) / 2.  The backward pass recomputes S and P on
 * chip from Q, K, V, O, dO and the saved lse ("Backward Pass: Recomputation").
 *
 * Common conventions for every entry point
 * ----------------------------------------
 * Layout     Q, K, V, O, dO, dQ, dK, dV are dense, contiguous, row-major
 *            [B, H, N, d] arrays in device memory; lse is [B, H, N] float32.
 *            Every base pointer must be 16-byte aligned.
 * dtype      FA_DTYPE_BF16: Q/K/V/O/dO/dQ/dK/dV are bfloat16, arithmetic is
 *            fp32-accumulated tensor-core math with P rounded to bf16 before
 *            the P V product; d must be 64, 96, 128 or 256 (256: forward
 *            only).
 *            FA_DTYPE_F32: all arrays are float32 and all arithmetic is exact
 *            fp32 on CUDA cores with the accurate expf/logf; 1 <= d <= 128.
 * scale      finite and > 0; usually 1/sqrt(d).
 * window     <= 0: unmasked.  Otherwise an odd full width w; r = (w - 1) / 2.
 *            Even widths are rejected (the pages give them no meaning).
 * stream     a cudaStream_t passed as void*; NULL is the legacy default
 *            stream.  All work is enqueued on it; no call synchronises except
 *            fa_last_device_status().
 * Ownership  the caller owns every buffer.  The library allocates no device
 *            memory and keeps no pointer after a call returns.
 * Errors     argument errors are detected on the host before anything is
 *            launched and return FA_ERR_INVALID or FA_ERR_UNSUPPORTED with no
 *            side effect.  A failed launch returns FA_ERR_CUDA.  Every wait
 *            inside the kernels is bounded in time; a wait that runs out
 *            records FA_ERR_TIMEOUT in the library's device status word and
 *            the kernel returns early (its outputs are then undefined), which
 *            fa_last_device_status() reports.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID = 1,      /* bad pointer, size, alignment, scale or window */
  FA_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement (dtype/d) */
  FA_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed */
  FA_ERR_TIMEOUT = 4       /* a bounded device-side wait ran out */
} fa_status;

typedef enum { FA_DTYPE_F32 = 0, FA_DTYPE_BF16 = 1 } fa_dtype;

/*
 * Forward pass: O = softmax(Q K^T * scale) V, and lse.
 *   q, k, v  [B,H,N,d] inputs (read only).
 *   o        [B,H,N,d] output, same dtype as the inputs.
 *   lse      [B,H,N] float32 output (natural log of the row sum of exp over
 *            the scaled, masked scores), or NULL if not wanted.
 * Sources: the notes' "The Standard Attention Problem" (what is computed),
 * "Derivation: Incremental Softmax" Steps 1-3 and TensorViz step "tiles" (how:
 * running max m, running sum l, rescale when m rises, divide by l at the end),
 * "Worked example Local Attention Window" (window; key tiles wholly outside
 * the band are never loaded).
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, float scale, int window, fa_dtype dt,
                 void* stream);

/*
 * Size in bytes of the workspace fa_bwd needs for a problem of this shape:
 * a float32 [B,H,N,d] dQ accumulator, then two [B,H,Npad] arrays derived
 * from lse_i and from D_i = sum_k dO_ik O_ik (Npad = N rounded up to a
 * multiple of 128; 4 bytes per row, or 16 bytes per row at d = 64, where
 * each value is kept as three bf16 terms), each section 256-byte aligned;
 * at d = 64, 96 and 128 then float32 dV and dK rows for up to 128 key tiles of
 * 128 keys (min(B*H*ceil(N/128), 128) * 2 * 128 * d * 4 bytes), which the
 * backward uses when it splits the key tiles of a last, partly filled wave
 * of CTAs in two.  Returns 0 for non-positive sizes.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * The same forward pass as fa_fwd, evaluated in the key-major loop order that
 * "Compute attention one tile at a time" (TensorViz), fidelity note,
 * attributes to the original Algorithm 1: the outer loop runs over 128-key
 * tiles (one launch each, in order on `stream`), and each launch merges that
 * tile into every query tile's running statistics (the notes' "Derivation:
 * Incremental Softmax", Steps 2-3), which live in `workspace` between
 * launches: fp32 unnormalised O~ [B,H,N,d], then m and l [B,H,N], each
 * section 256-byte aligned; a last launch writes O = O~ / l and lse.  It is
 * kept as a measured comparison point: every step reads and writes O~ in
 * device memory, which fa_fwd keeps on chip.
 *   workspace        at least fa_fwd_key_major_workspace_bytes() bytes,
 *                    256-byte aligned, owned by the caller; contents on entry
 *                    do not matter and are undefined on return.
 * bf16 with d = 64 or 128 only (others return FA_ERR_UNSUPPORTED); other
 * arguments, results and errors as fa_fwd.
 */
fa_status fa_fwd_key_major(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int N, int d, float scale, int window, fa_dtype dt,
                           void* workspace, size_t workspace_bytes, void* stream);
size_t fa_fwd_key_major_workspace_bytes(int B, int H, int N, int d);

/*
 * The float32 forward on the tensor cores.  Same operation, layouts, window
 * and results as fa_fwd with FA_DTYPE_F32 (q, k, v, o float32 [B,H,N,d], lse
 * float32 [B,H,N] or NULL), for 1 <= d <= 128.  The tensor cores multiply
 * tf32 values (11 significant bits), so every float32 operand x is split as
 * hi = tf32(x), lo = tf32(x - hi) and each product is taken as
 * hi*hi + hi*lo + lo*hi (the "3xTF32" scheme): S = Q K^T from split Q and K,
 * O += P V from split P and V, fp32 accumulation, fp32 output.  The dropped
 * lo*lo term and the rounding of lo are below 2^-21 relative.  fa_fwd with
 * FA_DTYPE_F32 stays the exact CUDA-core path; this entry point trades a
 * little of that accuracy for tensor-core speed.
 *   workspace        at least fa_fwd_f32_3xtf32_workspace_bytes() bytes,
 *                    256-byte aligned, owned by the caller (it receives the
 *                    split copies of Q, K and V: 6 x 4 x B*H*N*64 bytes for
 *                    d <= 64; for 64 < d <= 128 those of K and V only, 4 x 4
 *                    x B*H*N*128 bytes, the kernel splitting Q itself; N
 *                    rounded up to 64 for V); contents on entry do not
 *                    matter and are undefined on return.
 * d > 128 returns FA_ERR_UNSUPPORTED; other arguments and errors as fa_fwd.
 */
fa_status fa_fwd_f32_3xtf32(const float* q, const float* k, const float* v, float* o, float* lse,
                            int B, int H, int N, int d, float scale, int window,
                            void* workspace, size_t workspace_bytes, void* stream);
size_t fa_fwd_f32_3xtf32_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass by recomputation: given Q, K, V, the forward output O, its
 * lse and the output gradient dO, writes dQ, dK, dV (same dtype and layout
 * as Q).  S and P are rebuilt on chip from Q, K and lse; nothing of size
 * N x N is read or written.  Sources: the notes' "Backward Pass:
 * Recomputation" (recompute, do not store, S and P); the gradient formulas
 * are the derivative of the forward definition (the pages print none):
 * dV = P^T dO, dP = dO V^T, D_i = sum_j P_ij dP_ij = sum_k dO_ik O_ik,
 * dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q.
 *   workspace        device scratch of at least fa_bwd_workspace_bytes(),
 *                    owned by the caller, 256-byte aligned; its contents on
 *                    entry do not matter and are undefined on return.
 *   workspace_bytes  its size; smaller than required -> FA_ERR_INVALID.
 * bf16 with d = 64, 96 or 128 (other d, 256 included, return
 * FA_ERR_UNSUPPORTED), or float32
 * with 1 <= d <= 128 (CUDA cores; one warp per query row for dQ and one per
 * key row for dK and dV, so dK and dV need no atomics and the float32 path
 * is bitwise repeatable).
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dO, void* dq, void* dk, void* dv,
                 int B, int H, int N, int d, float scale, int window, fa_dtype dt,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_bwd for callers that cannot allocate device memory (code running where
 * device allocation is not permitted, or with no allocator to call): the same
 * arguments and results as fa_bwd, minus the workspace, which is replaced by
 * a fixed 64 MiB scratch array inside the library.  This function calls no
 * allocator.  The pages describe no such variant; it is a deployment aid.
 *   - Arguments are checked as fa_bwd checks them, with the same status
 *     codes; then problems with fa_bwd_workspace_bytes(B,H,N,d) > 64 MiB
 *     return FA_ERR_UNSUPPORTED.  Nothing is launched in either case.
 *   - Under CUDA's lazy module loading (the default), the array is brought
 *     onto a device, and its 64 MiB committed there, by the first call on
 *     that device; it then stays until the process exits.  That first call
 *     may therefore allocate and synchronise inside the CUDA driver: make it
 *     outside any region where allocation or stream capture is forbidden.
 *   - All calls share the one array: calls whose work overlaps on the GPU
 *     (e.g. on two concurrent streams) race on it; calls in order on one
 *     stream are fine.  Each call re-initialises what must start at zero.
 *   - The first call on each device looks up the array's device address;
 *     make that first call before any stream capture.
 */
fa_status fa_bwd_static_workspace(const void* q, const void* k, const void* v, const void* o,
                                  const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                  int B, int H, int N, int d, float scale, int window, fa_dtype dt,
                                  void* stream);

/*
 * Synchronises `stream` (as void* cudaStream_t), then reads and clears the
 * device status word that the kernels set when a bounded wait runs out.
 * Returns FA_OK, FA_ERR_TIMEOUT, or FA_ERR_CUDA if synchronising failed or a
 * kernel refused to run on the device (a layout check failed).
 */
fa_status fa_last_device_status(void* stream);

/*
 * Sets the time limit, in microseconds, of every device-side wait in kernels
 * launched afterwards by this process (default 1,000,000 = 1 s; values <= 0
 * restore the default).  Returns the previous limit.
 */
long long fa_set_wait_limit_us(long long limit_us);

/*
 * Self-test of the bounded wait: launches one block that waits on a shared
 * memory barrier nothing ever arrives on, for `limit_us` microseconds
 * (1..100000), then gives up, records FA_ERR_TIMEOUT in the status word and
 * returns.  A caller checks fa_last_device_status() == FA_ERR_TIMEOUT.
 */
fa_status fa_selftest_wait_timeout(int limit_us, void* stream);

/* Static, human-readable name of a status code. */
const char* fa_status_string(fa_status s);

/* Library version as major*10000 + minor*100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
