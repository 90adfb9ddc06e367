// fa_internal.h -- declarations shared by the C-ABI layer and the kernels'
// translation unit.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

constexpr int kBlockM = 128;  // query rows per sub-tile (TMEM lanes)
constexpr int kCtaRows = 2 * kBlockM;  // query rows per CTA (two sub-tiles)
constexpr int kBlockN = 128;  // keys per K/V tile

// Runtime parameters of one forward launch.
struct FwdParams {
    void *o;           // [B*H, Sq, D] bf16
    float *lse;        // [B*H, Sq] fp32
    int Sq, Sk;
    int n_mblk;        // ceil(Sq / kCtaRows)
    int bh_count;      // B * H
    int n_items;       // n_mblk * B * H work items (256 query rows of one head each)
    int n_kv;          // ceil(Sk / kBlockN)
    int causal;        // longest-first query-block order (triangular work)
    int wl, wr;        // key j allowed for query i iff i-wl <= j <= i+wr; -1 = unbounded
    float scale_log2;  // scale * log2(e)  (8-bit path: times descale_q * descale_k)
    float o_scale;     // 8-bit path: descale_v (unused by the bf16 path)
    unsigned long long timeout_ns;  // bound of every on-chip wait
    // Block mask (banded kernel only; null: every block kept): bmask[h][a][c]
    // nonzero keeps key tile c for 128-row query block a of head h, where h is
    // the head for bmask_hstride = n_qb * n_kv and 0 for bmask_hstride = 0.
    const unsigned char *bmask;
    long long bmask_hstride;
    // Block mask: query blocks a and a + pair_stride share a work item (and its
    // K/V loads), in groups of 2 * pair_stride blocks; n_mblk then counts the
    // items of one head.  1 elsewhere.
    int pair_stride;
};

// Split-KV (decode) launch: partials per (head, split), then a merge.
constexpr int kSplitMaxSq = 8;     // query rows per head the split path takes
constexpr int kSplitTileKeys = 64;
struct SplitParams {
    const void *q;      // bf16 [B*H, Sq, D]
    void *o;            // bf16 [B*H, Sq, D]
    float *lse;         // fp32 [B*H, Sq]
    float *o_part;      // fp32 [B*H, splits, Sq, D]   (workspace)
    float *lse_part;    // fp32 [B*H, splits, Sq]      (workspace)
    int Sq, Sk;
    int chunk;          // keys per split, a multiple of kSplitTileKeys
    int splits;         // ceil(Sk / chunk)
    float scale_log2;
    unsigned long long timeout_ns;
};
int splitkv_smem_bytes(int D);
cudaError_t launch_splitkv(int D, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const SplitParams &p, int BH,
                           cudaStream_t stream);
cudaError_t splitkv_status_read_and_clear(int *out);
// Built-in scratch of fa_fwd_splitkv_noalloc: size, and its device address
// in the current device's context (looked up on every call).
constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB
cudaError_t splitkv_scratch(void **out);

// Backward launch (dQ kernel, then dK/dV kernel).
struct BwdParams {
    const float *lse;    // fp32 [B*H, Sq]     forward log-sum-exp (natural log)
    float *delta;        // fp32 [B*H, Sq]     workspace: rowsum(dO * O)
    int Sq, Sk;
    int n_qt, n_kt;      // 128-row query tiles, 128-key tiles
    int causal;
    float scale, scale_log2;
    unsigned long long timeout_ns;
};
int bwd_smem_bytes(int D);
cudaError_t launch_bwd(int D, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tdo, const CUtensorMap &to, const CUtensorMap &tdq, const CUtensorMap &tdk,
                       const CUtensorMap &tdv, const BwdParams &p, long long BH, cudaStream_t stream);
cudaError_t bwd_status_read_and_clear(int *out);

// Launch the forward kernel for head dim D (64 or 128) over the p.n_items
// work items on persistent CTAs (at most num_sms).
cudaError_t launch_fwd(int D, const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                       const FwdParams &p, int num_sms, cudaStream_t stream);

// Launch the 8-bit (e4m3 Q, K, V; D = 128; full or causal) forward kernel.
cudaError_t launch_fwd_fp8(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                           const FwdParams &p, int num_sms, cudaStream_t stream);

// Device status word: read it (after synchronising `stream`) and reset it.
cudaError_t status_read_and_clear(int *out, cudaStream_t stream);

// One CTA waiting on a barrier nothing arrives on, bounded by limit_ns.
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream);

}  // namespace fa
