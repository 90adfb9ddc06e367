/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention forward library.
 *
 * The operation is the FlashAttention-2 forward pass: for every batch b,
 * head h and query row i,
 *
 *     O[b,h,i,:] = sum_j softmax_j(scale * Q[b,h,i,:] . K[b,h,j,:]) * V[b,h,j,:]
 *     LSE[b,h,i] = ln sum_j exp(scale * Q[b,h,i,:] . K[b,h,j,:])
 *
 * over the allowed keys j (j < Sk; with causal, also j <= i).  Sources:
 *   - "FlashAttention-2 相比 FlashAttention-1，到底改了什么" (source walk-through),
 *     section "第二处源码差异：kernel 主循环怎么组织": the online-softmax loop
 *     with O = acc / l and the epilogue that writes O and LSE;
 *     section "第一处源码差异：launch grid 怎么铺": the problem parameters
 *     (batch, heads, query length) and the stream passed at launch;
 *   - "FlashAttention-2 — L3 Cross-Paper Synthesis", §3 item 4: causal
 *     masking with whole-block skipping above the diagonal.
 *
 * Conventions shared by every entry point:
 *   - Tensors are row-major and contiguous, [B, H, S, D] for Q, K, V and O,
 *     [B, H, Sq] for LSE.  bf16 means IEEE bfloat16 bit patterns.
 *   - Every pointer is a DEVICE pointer on the current CUDA device, owned and
 *     allocated by the caller, 16-byte aligned.  The library allocates no
 *     device memory, performs no host<->device copy and no synchronisation:
 *     each call enqueues its kernel on `stream` (a cudaStream_t; NULL means
 *     the legacy default stream) and returns.  The outputs are complete when
 *     the stream reaches the end of that kernel.
 *   - Arguments are checked before anything is launched; a bad argument
 *     returns its negative code and launches nothing.  A launch failure
 *     returns FA_ERR_CUDA (fa_strerror gives the CUDA text of the last one).
 *   - Calls are thread-safe; per-device lazily initialised state (the
 *     driver's tensor-map encoder, kernel attributes) is guarded.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_NULLPTR = -1,            /* a required pointer is NULL                    */
    FA_ERR_BAD_SHAPE = -2,          /* B, H, Sq or Sk < 1, or a size out of range    */
    FA_ERR_UNSUPPORTED_D = -3,      /* head dim other than 64 or 128                 */
    FA_ERR_UNSUPPORTED_CAUSAL = -4, /* causal with Sq != Sk, or causal not 0/1       */
    FA_ERR_MISALIGNED = -5,         /* a pointer is not 16-byte aligned              */
    FA_ERR_BAD_SCALE = -6,          /* scale not finite or not > 0                   */
    FA_ERR_CUDA = -7,               /* CUDA runtime / driver error                   */
    FA_ERR_TIMEOUT = -8,            /* a bounded on-chip wait gave up (status word)  */
    FA_ERR_ALIAS = -9,              /* an output overlaps an input or the other one */
    FA_ERR_BAD_WINDOW = -10         /* window bound below -1                         */
} fa_status;

/*
 * fa_fwd -- attention forward, O = softmax(scale * Q K^T [+ causal mask]) V,
 * plus LSE (natural log).  Walk-through "FlashAttention-2 相比
 * FlashAttention-1，到底改了什么", section "第二处源码差异：kernel 主循环怎么组织".
 *
 *   q       bf16 [B, H, Sq, D]   device, read only
 *   k, v    bf16 [B, H, Sk, D]   device, read only
 *   o       bf16 [B, H, Sq, D]   device, written (rows < Sq only)
 *   lse     fp32 [B, H, Sq]      device, written: ln sum_j exp(scale q.k_j)
 *   B, H    batch and heads, >= 1
 *   Sq, Sk  query and key lengths, >= 1; causal requires Sq == Sk
 *   D       head dimension, 64 or 128
 *   scale   softmax temperature applied to Q.K before max/exp; finite, > 0
 *   causal  0: every key; 1: key j allowed for query i iff j <= i
 *   stream  cudaStream_t to launch on (NULL = default stream)
 *
 * Errors: FA_ERR_NULLPTR, FA_ERR_MISALIGNED, FA_ERR_BAD_SHAPE,
 * FA_ERR_UNSUPPORTED_D, FA_ERR_UNSUPPORTED_CAUSAL, FA_ERR_BAD_SCALE,
 * FA_ERR_ALIAS before launch; FA_ERR_CUDA if the launch fails.
 * Accumulation is fp32; P is rounded to bf16 before P*V; O is rounded to
 * bf16 (round-to-nearest-even).  No atomics: results are bitwise
 * deterministic for a given input.
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
           int Sq, int Sk, int D, float scale, int causal, void *stream);

/*
 * fa_fwd_window -- attention forward restricted to a band of keys around each
 * query: key j is allowed for query i iff  i - window_left <= j <= i + window_right.
 * A bound of -1 means unbounded on that side; window_right = 0 is causal, and
 * (window_left = W, window_right = 0) is causal sliding-window attention.
 * This is the sliding-window generalisation of causal block skipping named in
 * "FlashAttention-2 — L3 Cross-Paper Synthesis", §5 item 4: key tiles outside
 * every row's band are skipped whole, tiles crossing a band edge are masked.
 *
 * Arguments, layout, ownership and outputs are those of fa_fwd (O and LSE
 * over the allowed keys only).  A bounded window (either bound >= 0) needs
 * Sq == Sk, so every query row sees at least its own key.
 * Errors: those of fa_fwd, plus FA_ERR_BAD_WINDOW for a bound below -1 or a
 * bounded window with Sq != Sk.  fa_fwd(..., causal, ...) equals
 * fa_fwd_window(..., -1, causal ? 0 : -1, ...).
 */
int fa_fwd_window(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                  int Sq, int Sk, int D, float scale, int window_left, int window_right,
                  void *stream);

/*
 * fa_strerror -- static English text for a status code.  For FA_ERR_CUDA
 * the text of the most recent CUDA error seen by this thread is appended.
 * The returned pointer stays valid until the next call on the same thread.
 */
const char *fa_strerror(int status);

/*
 * fa_device_status -- the kernels' on-device status word, then clears it.
 * Every on-chip wait of every kernel in this library is bounded in time;
 * a wait that gives up records FA_ERR_TIMEOUT there (instead of hanging or
 * trapping) and the kernel winds down.  This call synchronises `stream`,
 * reads and resets the word on the current device, and returns FA_OK,
 * FA_ERR_TIMEOUT or FA_ERR_CUDA.  Meant for tests and debugging; it is the
 * only call here that synchronises.
 */
int fa_device_status(void *stream);

/*
 * fa_selftest_bounded_wait -- launches one CTA that waits on an on-chip
 * barrier that nothing ever arrives on, with a wait limit of `timeout_us`
 * microseconds (1 .. 1000000), using the same bounded-wait routine as the
 * attention kernels.  The wait must give up and record FA_ERR_TIMEOUT in the
 * status word, which fa_device_status then returns.  No fault, trap or hang
 * is involved: this exists so tests can show the give-up path works.
 */
int fa_selftest_bounded_wait(int timeout_us, void *stream);

/* fa_version -- library version, major*10000 + minor*100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
