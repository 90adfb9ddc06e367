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

#include <stddef.h>

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
    FA_ERR_BAD_WINDOW = -10,        /* window bound below -1, or band with Sq != Sk  */
    FA_ERR_WORKSPACE = -11,         /* workspace missing, misaligned or too small    */
    FA_ERR_SCRATCH_LIMIT = -12,     /* more scratch than the built-in buffer holds   */
    FA_ERR_BAD_MASK = -13           /* mask heads not 1 or B * H, or pair stride < 1 */
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
 * fa_fwd_blockmask -- attention forward over the key blocks a block mask keeps:
 * the "unified sparse-block-skip mechanism" into which "FlashAttention-2 — L3
 * Cross-Paper Synthesis", §5 item 4, generalises causal block skipping (the
 * sliding window and dilated patterns being instances).  Key j is allowed for
 * query i iff j < Sk, the band keeps it (i - window_left <= j <= i +
 * window_right, as in fa_fwd_window: -1 unbounded, (-1, 0) causal) and
 *     block_mask[m][i / FA_BLOCK_M][j / FA_BLOCK_N] != 0,
 * where m = 0 when mask_heads = 1 (one pattern for every head) and m = b*H + h
 * when mask_heads = B * H.  Key blocks a query block does not keep are never
 * loaded or multiplied.
 *
 *   block_mask  uint8 [mask_heads, ceil(Sq / FA_BLOCK_M), ceil(Sk / FA_BLOCK_N)]
 *               DEVICE pointer, read by the kernel (must stay valid until the
 *               stream passes it), any alignment, must not overlap O or LSE
 *   mask_heads  1 or B * H
 *   pair_stride >= 1, a scheduling hint that does not change the result: query
 *               blocks a and a + pair_stride are computed together (in groups
 *               of 2 * pair_stride blocks; the last blocks with their
 *               neighbours) and share the loads of the key blocks either keeps.
 *               1 suits masks whose neighbouring block rows keep like blocks
 *               (bands, local patterns); a dilated pattern with stride r wants r.
 * Other arguments, layout, ownership and outputs are those of fa_fwd_window.
 * A query row with no allowed key (its block row keeps nothing, or the band
 * leaves nothing of what it keeps) gets O = 0 and LSE = -inf.
 * Errors: those of fa_fwd_window, plus FA_ERR_NULLPTR for a null mask,
 * FA_ERR_BAD_MASK for mask_heads other than 1 or B * H or pair_stride < 1, and FA_ERR_ALIAS when
 * the mask overlaps O or LSE.  With every block kept it equals fa_fwd_window.
 */
#define FA_BLOCK_M 128
#define FA_BLOCK_N 128
int fa_fwd_blockmask(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                     int Sq, int Sk, int D, float scale, int window_left, int window_right,
                     const unsigned char *block_mask, int mask_heads, int pair_stride, void *stream);

/*
 * fa_fwd_fp8 -- attention forward with 8-bit (e4m3) Q, K, V and per-tensor
 * scaling: the FP8 tensor-core path that "Architectural Innovations in
 * FlashAttention-2 and FlashAttention-3" names as FA3's throughput lever
 * (section 三, FA3 item (3)), with the loss of precision held in check by
 * scaling and mixed precision (section 四, item ③).
 *
 * Each of q, k, v is an e4m3 tensor (1 byte per element: sign, 4 exponent
 * bits with bias 7, 3 mantissa bits; 0x7F and 0xFF are NaN) whose real value
 * is code * descale_x; layouts are fa_fwd's ([B, H, S, D] row-major, device
 * memory, 16-byte aligned).  The call computes, for the dequantised inputs,
 *   O   = softmax(scale * Q K^T [+ causal mask]) V   (bf16 [B, H, Sq, D])
 *   LSE = natural-log row log-sum-exp of scale * Q K^T  (fp32 [B, H, Sq])
 * S accumulates in fp32; P is rounded to e4m3 (times a power of two) for the
 * P V product, which accumulates in fp32; O is rounded to bf16 once.
 * D must be 128.  causal as in fa_fwd (needs Sq == Sk).  Ownership and
 * launch semantics are fa_fwd's.
 * Errors: those of fa_fwd; FA_ERR_UNSUPPORTED_D for D != 128;
 * FA_ERR_BAD_SCALE when scale or a descale is not finite and > 0 (or their
 * product underflows or overflows fp32).
 */
int fa_fwd_fp8(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
               int Sq, int Sk, int D, float scale, int causal, float descale_q, float descale_k,
               float descale_v, void *stream);

/*
 * fa_fwd_splitkv -- attention for decode: a few query rows per head against a
 * long key/value sequence, with the keys of each head split across CTAs.
 * "FlashAttention-2 — L3 Cross-Paper Synthesis", §5 item 5 (decode needs
 * parallelism over the key/value sequence); the split-and-merge of v1's
 * num_splits in "FlashAttention-2 相比 FlashAttention-1，到底改了什么", section
 * "第一处源码差异：launch grid 怎么铺".  Each split s of a head produces
 * lse_s = ln sum_{j in s} exp(scale q.k_j) and the normalised partial o_s;
 * the merge is lse = ln sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s.
 * Every query row sees every key (no mask).
 *
 *   q, k, v, o, lse, B, H, Sk, D, scale, stream: as fa_fwd
 *   Sq            1 .. 8 query rows per head
 *   num_splits    key ranges per head, 1 .. 256; <= 0 picks a count from the
 *                 problem size and the SM count (fa_splitkv_num_splits);
 *                 each range holds a multiple of 64 keys, so fewer ranges
 *                 may be used when Sk is short
 *   workspace     caller-owned DEVICE scratch of at least
 *                 fa_fwd_splitkv_workspace_bytes(...) bytes, 16-byte aligned,
 *                 not overlapping any other argument; it holds fp32 partial
 *                 results between the two kernels this call enqueues, and
 *                 must not be used by another call until the stream has run
 *                 past this one
 *   B * H         at most 65535
 *
 * Errors: those of fa_fwd (causal does not apply), FA_ERR_BAD_SHAPE for
 * Sq > 8, B*H > 65535 or num_splits > 256, FA_ERR_WORKSPACE for a missing,
 * misaligned or short workspace.  Deterministic; no atomics.  If an on-chip
 * wait gives up (fa_device_status then returns FA_ERR_TIMEOUT), the affected
 * partials are marked invalid and the merged O and LSE of their rows are NaN.
 */
int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                   int Sq, int Sk, int D, float scale, int num_splits, void *workspace,
                   size_t workspace_bytes, void *stream);

/*
 * fa_fwd_splitkv_workspace_bytes -- bytes of workspace fa_fwd_splitkv needs for
 * these sizes and num_splits (<= 0: the automatic count); 0 for unsupported sizes.
 */
size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int Sq, int Sk, int D, int num_splits);

/* fa_splitkv_num_splits -- the split count fa_fwd_splitkv picks automatically
 * for these sizes on the current device (or FA_ERR_BAD_SHAPE). */
int fa_splitkv_num_splits(int B, int H, int Sq, int Sk, int D);

/*
 * fa_fwd_splitkv_noalloc -- fa_fwd_splitkv for callers that cannot allocate
 * device memory.  The pages have no counterpart to this call: it exists for
 * callers such as a process whose device memory is all reserved up front by
 * another allocator (a cudaMalloc there fails or fragments that pool), or a
 * latency-critical path that must not take the implicit synchronisation and
 * driver locks that cudaMalloc/cudaFree can take.  It allocates nothing: the
 * scratch lives in a 16 MiB array inside this library's device image (every
 * GPU that loads the library holds it until the process exits).
 *
 * Arguments and results are those of fa_fwd_splitkv without the workspace;
 * the caller still provides q, k, v, o and lse.  Every call looks up the
 * array's device address in the current device's context
 * (cudaGetSymbolAddress); the first call on a device also loads the library's
 * module there, so make that first call before any stream capture.  All
 * calls on a device share the one array and it keeps the last call's bytes;
 * nothing in it needs to start at zero (each call's partial kernel writes
 * every partial result before its merge kernel reads it; after a wait that
 * gave up, the partials it could not finish are marked invalid, as for
 * fa_fwd_splitkv).  Calls whose kernels overlap on the GPU (two streams, or
 * two host threads) race on the array: serialise them.
 * Errors: those of fa_fwd_splitkv, plus FA_ERR_SCRATCH_LIMIT when the sizes
 * need more than 16 MiB of scratch (fa_fwd_splitkv_workspace_bytes tells the
 * need; pass a workspace to fa_fwd_splitkv for larger problems).
 */
int fa_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                           int H, int Sq, int Sk, int D, float scale, int num_splits, void *stream);

/*
 * fa_bwd -- gradients of fa_fwd: given dO = dL/dO for the forward's O,
 *   P = exp(scale Q K^T - LSE),  Delta_i = dO_i . O_i,  dS = P (dO V^T - Delta),
 *   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
 * "FlashAttention-2 — L3 Cross-Paper Synthesis", §3 items 1-2 (the backward
 * pass; FA2's atomic dQ accumulation is non-deterministic) and §5 item 2 (a
 * deterministic two-pass backward).  Two kernels run on `stream`: one CTA per
 * query tile writes dQ and Delta, then one CTA per key tile writes dK and dV.
 * No atomics: results are bitwise deterministic.
 *
 *   q, k, v, B, H, Sq, Sk, D, scale, causal   as passed to fa_fwd
 *   o, lse        the forward's outputs (bf16 [B,H,Sq,D], fp32 [B,H,Sq])
 *   dout          bf16 [B,H,Sq,D]
 *   dq            bf16 [B,H,Sq,D] written;  dk, dv  bf16 [B,H,Sk,D] written
 *   delta         fp32 [B,H,Sq] caller-owned scratch, written with Delta
 * All device pointers, 16-byte aligned; outputs may not overlap inputs or one
 * another.  Errors: those of fa_fwd (full and causal attention only).
 */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dout, void *dq, void *dk, void *dv, float *delta, int B, int H, int Sq,
           int Sk, int D, float scale, int causal, void *stream);

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

/*
 * fa_selftest_fwd_timeout -- fa_fwd with every on-chip wait of the forward
 * kernel bounded by `timeout_ns` (0 .. 2e9) instead of the 2 s that fa_fwd
 * uses.  With a limit shorter than a tile load (0 gives up at the first wait
 * that is not already satisfied), the kernel's own give-up path runs: the
 * wait raises the CTA's abort flag and records FA_ERR_TIMEOUT in the status
 * word, the other roles stop at their next wait, the producer waits (bounded,
 * 20 ms) for the copies it issued, the MMA issuer for its MMAs, TMEM is freed
 * and the CTA returns -- no trap, fault or hang.  O and LSE are then
 * undefined.  Arguments, checks and errors are fa_fwd's, plus
 * FA_ERR_BAD_SHAPE for timeout_ns above 2e9.  The surveyed pages have no
 * counterpart: it exists so tests can show the forward kernel winds down
 * cleanly and leaves the context usable.
 */
int fa_selftest_fwd_timeout(const void *q, const void *k, const void *v, void *o, float *lse,
                            int B, int H, int Sq, int Sk, int D, float scale, int causal,
                            unsigned long long timeout_ns, void *stream);

/*
 * fa_selftest_bwd_timeout -- fa_bwd with every on-chip wait of both backward
 * kernels bounded by `timeout_ns` (0 .. 2e9) instead of the 2 s that fa_bwd
 * uses.  With a limit shorter than a tile load the kernels' own give-up path
 * runs, as for fa_selftest_fwd_timeout: the CTA's abort flag is raised and
 * FA_ERR_TIMEOUT recorded in the status word, the other roles stop at their
 * next wait, copies and MMAs in flight are waited for (bounded), TMEM is freed
 * and the CTA returns.  dQ, dK, dV and delta are then undefined.  Arguments,
 * checks and errors are fa_bwd's, plus FA_ERR_BAD_SHAPE for timeout_ns above
 * 2e9.  The surveyed pages have no counterpart: it exists so tests can show
 * the backward kernels wind down cleanly and leave the context usable.
 */
int fa_selftest_bwd_timeout(const void *q, const void *k, const void *v, const void *o, const float *lse,
                            const void *dout, void *dq, void *dk, void *dv, float *delta, int B, int H,
                            int Sq, int Sk, int D, float scale, int causal, unsigned long long timeout_ns,
                            void *stream);

/*
 * fa_selftest_splitkv_timeout -- fa_fwd_splitkv with every on-chip wait of the
 * partial kernel bounded by `timeout_ns` (0 .. 2e9) instead of 2 s.  With a
 * limit shorter than a tile load the kernel gives up as the forward kernel
 * does (abort flag, FA_ERR_TIMEOUT in the status word, copies in flight
 * waited for, no trap); a CTA that gave up writes NaN as its partial
 * log-sum-exp, so the merged O and LSE of its rows come out NaN instead of
 * plausible stale values.  Arguments, checks and errors are fa_fwd_splitkv's,
 * plus FA_ERR_BAD_SHAPE for timeout_ns above 2e9.  The surveyed pages have no
 * counterpart: it exists so tests can show the decode kernels wind down
 * cleanly and leave the context usable.
 */
int fa_selftest_splitkv_timeout(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                                int H, int Sq, int Sk, int D, float scale, int num_splits, void *workspace,
                                size_t workspace_bytes, unsigned long long timeout_ns, void *stream);

/* fa_version -- library version, major*10000 + minor*100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
