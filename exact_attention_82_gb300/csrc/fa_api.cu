// fa_api.cu -- the C ABI declared in include/fa.h: argument checks, TMA
// tensor-map encoding and the launch on the caller's stream.  No device
// memory is allocated here and nothing is synchronised (except in
// fa_device_status, which exists to read the status word).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>

using std::max;
using std::min;

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

constexpr unsigned long long kWaitLimitNs = 2ull * 1000 * 1000 * 1000;  // 2 s per wait

thread_local char t_errbuf[256];
thread_local cudaError_t t_last_cuda = cudaSuccess;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int fail_cuda(cudaError_t e) {
    t_last_cuda = e;
    return FA_ERR_CUDA;
}

bool get_encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// 3-D map over a [BH, S, D] tensor of bf16 (eb = 2) or 8-bit (eb = 1)
// elements: dims (D, S, BH), box (128 bytes of a row, rows, 1), 128-byte
// swizzle, zero fill outside the tensor.  Being 3-D, a box never reaches into
// the next head's rows.
bool encode_bhsd(CUtensorMap *map, const void *ptr, int D, int S, long long BH, int box_rows, int eb = 2) {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D * eb, (cuuint64_t)S * (cuuint64_t)D * eb};
    const cuuint32_t box[3] = {128u / (cuuint32_t)eb, (cuuint32_t)box_rows, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = g_encode(map, eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                                const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" int fa_version(void) { return 100; }  // 0.1.0

extern "C" const char *fa_strerror(int status) {
    const char *s;
    switch (status) {
        case FA_OK: s = "ok"; break;
        case FA_ERR_NULLPTR: s = "a required pointer is NULL"; break;
        case FA_ERR_BAD_SHAPE: s = "bad shape: B, H, Sq, Sk must be >= 1 and sizes in range"; break;
        case FA_ERR_UNSUPPORTED_D: s = "unsupported head dim (64 or 128; 128 for the 8-bit path)"; break;
        case FA_ERR_UNSUPPORTED_CAUSAL: s = "causal must be 0 or 1, and causal needs Sq == Sk"; break;
        case FA_ERR_MISALIGNED: s = "a pointer is not 16-byte aligned"; break;
        case FA_ERR_BAD_SCALE: s = "scale (and each descale) must be finite and > 0"; break;
        case FA_ERR_CUDA: s = "CUDA error"; break;
        case FA_ERR_TIMEOUT: s = "an on-chip wait gave up (bounded-wait timeout)"; break;
        case FA_ERR_ALIAS: s = "an output buffer overlaps an input or the other output"; break;
        case FA_ERR_BAD_WINDOW: s = "window bounds must be >= -1, and a bounded window needs Sq == Sk"; break;
        case FA_ERR_WORKSPACE: s = "workspace missing, not 16-byte aligned, or smaller than required"; break;
        case FA_ERR_BAD_MASK: s = "mask_heads must be 1 or B * H, and pair_stride >= 1"; break;
        case FA_ERR_SCRATCH_LIMIT:
            s = "needs more scratch than the built-in 16 MiB buffer of fa_fwd_splitkv_noalloc holds; "
                "pass a workspace to fa_fwd_splitkv instead";
            break;
        default: s = "unknown status"; break;
    }
    if (status == FA_ERR_CUDA && t_last_cuda != cudaSuccess)
        snprintf(t_errbuf, sizeof t_errbuf, "%s: %s", s, cudaGetErrorString(t_last_cuda));
    else
        snprintf(t_errbuf, sizeof t_errbuf, "%s", s);
    return t_errbuf;
}

// SMs of the current device (cached per device): persistent forward kernels
// run at most one CTA per SM, and the split-KV heuristic sizes its grid by it.
static int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        cached[dev] = n;
    }
    return cached[dev];
}

// Checks shared by the forward entry points; FA_OK when the call may launch.
static int check_fwd(const void *q, const void *k, const void *v, const void *o, const float *lse, int B, int H,
                     int Sq, int Sk, int D, float scale) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_NULLPTR;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_MISALIGNED;
    if (B < 1 || H < 1 || Sq < 1 || Sk < 1) return FA_ERR_BAD_SHAPE;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED_D;
    if (!isfinite(scale) || !(scale > 0.f)) return FA_ERR_BAD_SCALE;
    const long long BH = (long long)B * H;
    const long long n_ctas = ((Sq + fa::kCtaRows - 1) / fa::kCtaRows) * BH;
    if (BH > (1ll << 31) || n_ctas > 0x7fffffffll) return FA_ERR_BAD_SHAPE;
    const size_t q_bytes = (size_t)BH * Sq * D * 2, kv_bytes = (size_t)BH * Sk * D * 2;
    const size_t lse_bytes = (size_t)BH * Sq * 4;
    if (overlaps(o, q_bytes, q, q_bytes) || overlaps(o, q_bytes, k, kv_bytes) ||
        overlaps(o, q_bytes, v, kv_bytes) || overlaps(lse, lse_bytes, q, q_bytes) ||
        overlaps(lse, lse_bytes, k, kv_bytes) || overlaps(lse, lse_bytes, v, kv_bytes) ||
        overlaps(lse, lse_bytes, o, q_bytes))
        return FA_ERR_ALIAS;
    return FA_OK;
}

// Encode the maps and launch; arguments already checked.  Key j is allowed
// for query i iff i - wl <= j <= i + wr (a negative bound: unbounded).
static int launch_checked(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Sq,
                          int Sk, int D, float scale, int wl, int wr, void *stream,
                          unsigned long long timeout_ns = kWaitLimitNs, const unsigned char *bmask = nullptr,
                          long long bmask_hstride = 0, int pair_stride = 1) {
    if (!get_encoder()) return fail_cuda(cudaErrorNotSupported);
    const long long BH = (long long)B * H;
    long long n_mblk = (Sq + fa::kCtaRows - 1) / fa::kCtaRows;
    if (bmask) {  // items of one head when query blocks a and a + pair_stride are paired
        const long long n_qb = (Sq + fa::kBlockM - 1) / fa::kBlockM, s = pair_stride;
        const long long whole = n_qb / (2 * s);
        n_mblk = whole * s + (n_qb - 2 * s * whole + 1) / 2;
    }
    CUtensorMap tm_q, tm_k, tm_v;
    if (!encode_bhsd(&tm_q, q, D, Sq, BH, fa::kBlockM) || !encode_bhsd(&tm_k, k, D, Sk, BH, fa::kBlockN) ||
        !encode_bhsd(&tm_v, v, D, Sk, BH, fa::kBlockN))
        return fail_cuda(cudaErrorInvalidValue);
    fa::FwdParams p;
    p.o = o;
    p.lse = lse;
    p.bh_count = (int)BH;
    p.n_items = (int)(n_mblk * BH);
    p.Sq = Sq;
    p.Sk = Sk;
    p.n_mblk = (int)n_mblk;
    p.n_kv = (Sk + fa::kBlockN - 1) / fa::kBlockN;
    p.causal = (wr >= 0 && wl < 0) ? 1 : 0;  // triangular work: longest blocks first
    p.wl = wl < 0 ? -1 : wl;
    p.wr = wr < 0 ? -1 : wr;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.o_scale = 1.f;
    p.timeout_ns = timeout_ns;
    p.bmask = bmask;
    p.bmask_hstride = bmask_hstride;
    p.pair_stride = pair_stride;
    const cudaError_t e = fa::launch_fwd(D, tm_q, tm_k, tm_v, p, sm_count(), (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return FA_OK;
}

extern "C" int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Sq,
                      int Sk, int D, float scale, int causal, void *stream) {
    const int st = check_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, scale);
    if (st != FA_OK) return st;
    if (causal != 0 && causal != 1) return FA_ERR_UNSUPPORTED_CAUSAL;
    if (causal && Sq != Sk) return FA_ERR_UNSUPPORTED_CAUSAL;
    return launch_checked(q, k, v, o, lse, B, H, Sq, Sk, D, scale, -1, causal ? 0 : -1, stream);
}

extern "C" int fa_fwd_window(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                             int Sq, int Sk, int D, float scale, int window_left, int window_right,
                             void *stream) {
    const int st = check_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, scale);
    if (st != FA_OK) return st;
    if (window_left < -1 || window_right < -1) return FA_ERR_BAD_WINDOW;
    if ((window_left >= 0 || window_right >= 0) && Sq != Sk) return FA_ERR_BAD_WINDOW;
    return launch_checked(q, k, v, o, lse, B, H, Sq, Sk, D, scale, window_left, window_right, stream);
}

extern "C" int fa_fwd_blockmask(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                                int Sq, int Sk, int D, float scale, int window_left, int window_right,
                                const unsigned char *block_mask, int mask_heads, int pair_stride, void *stream) {
    const int st = check_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, scale);
    if (st != FA_OK) return st;
    if (!block_mask) return FA_ERR_NULLPTR;
    if (window_left < -1 || window_right < -1) return FA_ERR_BAD_WINDOW;
    if ((window_left >= 0 || window_right >= 0) && Sq != Sk) return FA_ERR_BAD_WINDOW;
    const long long BH = (long long)B * H;
    if (mask_heads != 1 && (long long)mask_heads != BH) return FA_ERR_BAD_MASK;
    if (pair_stride < 1) return FA_ERR_BAD_MASK;
    const long long n_qb = (Sq + fa::kBlockM - 1) / fa::kBlockM, n_kb = (Sk + fa::kBlockN - 1) / fa::kBlockN;
    const size_t mask_bytes = (size_t)mask_heads * (size_t)(n_qb * n_kb);
    const size_t o_bytes = (size_t)BH * Sq * D * 2, lse_bytes = (size_t)BH * Sq * 4;
    if (overlaps(block_mask, mask_bytes, o, o_bytes) || overlaps(block_mask, mask_bytes, lse, lse_bytes))
        return FA_ERR_ALIAS;
    // a stride of n_qb or more pairs nothing apart: every block with its neighbour
    const int stride = (int)std::min<long long>(pair_stride, n_qb);
    return launch_checked(q, k, v, o, lse, B, H, Sq, Sk, D, scale, window_left, window_right, stream, kWaitLimitNs,
                          block_mask, mask_heads == 1 ? 0 : n_qb * n_kb, stride);
}

extern "C" int fa_fwd_fp8(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                          int Sq, int Sk, int D, float scale, int causal, float descale_q, float descale_k,
                          float descale_v, void *stream) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_NULLPTR;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_MISALIGNED;
    if (B < 1 || H < 1 || Sq < 1 || Sk < 1) return FA_ERR_BAD_SHAPE;
    if (D != 128) return FA_ERR_UNSUPPORTED_D;
    if (causal != 0 && causal != 1) return FA_ERR_UNSUPPORTED_CAUSAL;
    if (causal && Sq != Sk) return FA_ERR_UNSUPPORTED_CAUSAL;
    const float sc[4] = {scale, descale_q, descale_k, descale_v};
    for (float x : sc)
        if (!isfinite(x) || !(x > 0.f)) return FA_ERR_BAD_SCALE;
    const float scale_log2 = scale * descale_q * descale_k * 1.4426950408889634f;
    if (!isfinite(scale_log2) || !(scale_log2 > 0.f)) return FA_ERR_BAD_SCALE;
    const long long BH = (long long)B * H;
    const long long n_mblk = (Sq + fa::kCtaRows - 1) / fa::kCtaRows;
    if (BH > (1ll << 31) || n_mblk * BH > 0x7fffffffll) return FA_ERR_BAD_SHAPE;
    const size_t q_bytes = (size_t)BH * Sq * D, kv_bytes = (size_t)BH * Sk * D;
    const size_t o_bytes = 2 * q_bytes, lse_bytes = (size_t)BH * Sq * 4;
    if (overlaps(o, o_bytes, q, q_bytes) || overlaps(o, o_bytes, k, kv_bytes) || overlaps(o, o_bytes, v, kv_bytes) ||
        overlaps(lse, lse_bytes, q, q_bytes) || overlaps(lse, lse_bytes, k, kv_bytes) ||
        overlaps(lse, lse_bytes, v, kv_bytes) || overlaps(lse, lse_bytes, o, o_bytes))
        return FA_ERR_ALIAS;
    if (!get_encoder()) return fail_cuda(cudaErrorNotSupported);
    CUtensorMap tm_q, tm_k, tm_v;
    if (!encode_bhsd(&tm_q, q, D, Sq, BH, fa::kBlockM, 1) || !encode_bhsd(&tm_k, k, D, Sk, BH, fa::kBlockN, 1) ||
        !encode_bhsd(&tm_v, v, D, Sk, BH, fa::kBlockN, 1))
        return fail_cuda(cudaErrorInvalidValue);
    fa::FwdParams p;
    p.o = o;
    p.lse = lse;
    p.bh_count = (int)BH;
    p.n_items = (int)(n_mblk * BH);
    p.Sq = Sq;
    p.Sk = Sk;
    p.n_mblk = (int)n_mblk;
    p.n_kv = (Sk + fa::kBlockN - 1) / fa::kBlockN;
    p.causal = causal;
    p.wl = -1;
    p.wr = causal ? 0 : -1;
    p.scale_log2 = scale_log2;
    p.o_scale = descale_v;
    p.timeout_ns = kWaitLimitNs;
    p.bmask = nullptr;
    p.bmask_hstride = 0;
    p.pair_stride = 1;
    const cudaError_t e = fa::launch_fwd_fp8(tm_q, tm_k, tm_v, p, sm_count(), (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return FA_OK;
}

// ------------------------------------------------------------- split-KV path
// Keys per split for `splits` ranges: a multiple of the 64-key split tile.
static int split_chunk(int Sk, int splits) {
    const int per = (Sk + splits - 1) / splits;
    return ((per + fa::kSplitTileKeys - 1) / fa::kSplitTileKeys) * fa::kSplitTileKeys;
}

static int resolve_splits(int B, int H, int Sk, int num_splits) {
    const int max_splits = (Sk + fa::kSplitTileKeys - 1) / fa::kSplitTileKeys;
    int s = num_splits;
    if (s <= 0) {
        // Our heuristic: among split counts keeping >= 256 keys per split (up to
        // 256 splits), take the one whose CTAs fill the SMs' last wave best,
        // preferring at least four waves; ties go to fewer splits.
        const long long bh = (long long)B * H;
        const int nsm = sm_count();
        const int cap = max(1, min(256, (Sk + 255) / 256));
        double best = -1.0;
        s = 1;
        for (int c = 1; c <= cap; ++c) {
            const long long ctas = bh * c;
            const long long waves = (ctas + nsm - 1) / nsm;
            double score = (double)ctas / (double)(waves * nsm);
            if (ctas < 4ll * nsm) score *= (double)ctas / (4.0 * nsm);
            if (score > best + 1e-9) {
                best = score;
                s = c;
            }
        }
    }
    s = min(s, max_splits);
    const int chunk = split_chunk(Sk, s);
    return (Sk + chunk - 1) / chunk;  // no empty split
}

static size_t splitkv_bytes(long long BH, int Sq, int D, int splits) {
    const size_t o_bytes = (size_t)BH * splits * Sq * D * sizeof(float);
    const size_t o_pad = (o_bytes + 255) & ~(size_t)255;
    return o_pad + (size_t)BH * splits * Sq * sizeof(float);
}

static bool splitkv_shape_ok(int B, int H, int Sq, int Sk, int D) {
    return B >= 1 && H >= 1 && Sq >= 1 && Sq <= fa::kSplitMaxSq && Sk >= 1 && (D == 64 || D == 128) &&
           (long long)B * H <= 65535;
}

extern "C" int fa_splitkv_num_splits(int B, int H, int Sq, int Sk, int D) {
    if (!splitkv_shape_ok(B, H, Sq, Sk, D)) return FA_ERR_BAD_SHAPE;
    return resolve_splits(B, H, Sk, 0);
}

extern "C" size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int Sq, int Sk, int D, int num_splits) {
    if (!splitkv_shape_ok(B, H, Sq, Sk, D) || num_splits > 256) return 0;
    return splitkv_bytes((long long)B * H, Sq, D, resolve_splits(B, H, Sk, num_splits));
}

static int splitkv_checked(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                           int Sq, int Sk, int D, float scale, int num_splits, void *workspace,
                           size_t workspace_bytes, void *stream, unsigned long long timeout_ns) {
    const int st = check_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, scale);
    if (st != FA_OK) return st;
    if (Sq > fa::kSplitMaxSq || (long long)B * H > 65535 || num_splits > 256) return FA_ERR_BAD_SHAPE;
    const long long BH = (long long)B * H;
    const int splits = resolve_splits(B, H, Sk, num_splits);
    const size_t need = splitkv_bytes(BH, Sq, D, splits);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return FA_ERR_WORKSPACE;
    const size_t kv_bytes = (size_t)BH * Sk * D * 2, q_bytes = (size_t)BH * Sq * D * 2;
    if (overlaps(workspace, need, q, q_bytes) || overlaps(workspace, need, k, kv_bytes) ||
        overlaps(workspace, need, v, kv_bytes) || overlaps(workspace, need, o, q_bytes) ||
        overlaps(workspace, need, lse, (size_t)BH * Sq * 4))
        return FA_ERR_ALIAS;
    if (!get_encoder()) return fail_cuda(cudaErrorNotSupported);
    CUtensorMap tm_k, tm_v;
    if (!encode_bhsd(&tm_k, k, D, Sk, BH, fa::kSplitTileKeys) || !encode_bhsd(&tm_v, v, D, Sk, BH, fa::kSplitTileKeys))
        return fail_cuda(cudaErrorInvalidValue);
    fa::SplitParams p;
    p.q = q;
    p.o = o;
    p.lse = lse;
    p.o_part = static_cast<float *>(workspace);
    p.lse_part = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                           (((size_t)BH * splits * Sq * D * sizeof(float) + 255) & ~(size_t)255));
    p.Sq = Sq;
    p.Sk = Sk;
    p.chunk = split_chunk(Sk, splits);
    p.splits = splits;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.timeout_ns = timeout_ns;
    const cudaError_t e = fa::launch_splitkv(D, tm_k, tm_v, p, (int)BH, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return FA_OK;
}

extern "C" int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                              int Sq, int Sk, int D, float scale, int num_splits, void *workspace,
                              size_t workspace_bytes, void *stream) {
    return splitkv_checked(q, k, v, o, lse, B, H, Sq, Sk, D, scale, num_splits, workspace, workspace_bytes, stream,
                           kWaitLimitNs);
}

extern "C" int fa_selftest_splitkv_timeout(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                                           int H, int Sq, int Sk, int D, float scale, int num_splits,
                                           void *workspace, size_t workspace_bytes,
                                           unsigned long long timeout_ns, void *stream) {
    if (timeout_ns > kWaitLimitNs) return FA_ERR_BAD_SHAPE;
    return splitkv_checked(q, k, v, o, lse, B, H, Sq, Sk, D, scale, num_splits, workspace, workspace_bytes, stream,
                           timeout_ns);
}

extern "C" int fa_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                                      int H, int Sq, int Sk, int D, float scale, int num_splits, void *stream) {
    // Same checks as fa_fwd_splitkv, then the size limit, before any CUDA call.
    const int st = check_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, scale);
    if (st != FA_OK) return st;
    if (Sq > fa::kSplitMaxSq || (long long)B * H > 65535 || num_splits > 256) return FA_ERR_BAD_SHAPE;
    const size_t need = splitkv_bytes((long long)B * H, Sq, D, resolve_splits(B, H, Sk, num_splits));
    if (need > fa::kNoAllocScratchBytes) return FA_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    const cudaError_t e = fa::splitkv_scratch(&scratch);
    if (e != cudaSuccess) return fail_cuda(e);
    return fa_fwd_splitkv(q, k, v, o, lse, B, H, Sq, Sk, D, scale, num_splits, scratch, fa::kNoAllocScratchBytes,
                          stream);
}

// ------------------------------------------------------------------ backward
static int bwd_checked(const void *q, const void *k, const void *v, const void *o, const float *lse,
                       const void *dout, void *dq, void *dk, void *dv, float *delta, int B, int H, int Sq, int Sk,
                       int D, float scale, int causal, void *stream, unsigned long long timeout_ns) {
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !delta) return FA_ERR_NULLPTR;
    const void *ptrs[10] = {q, k, v, o, lse, dout, dq, dk, dv, delta};
    for (const void *ptr : ptrs)
        if (!aligned16(ptr)) return FA_ERR_MISALIGNED;
    if (B < 1 || H < 1 || Sq < 1 || Sk < 1) return FA_ERR_BAD_SHAPE;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED_D;
    if (causal != 0 && causal != 1) return FA_ERR_UNSUPPORTED_CAUSAL;
    if (causal && Sq != Sk) return FA_ERR_UNSUPPORTED_CAUSAL;
    if (!isfinite(scale) || !(scale > 0.f)) return FA_ERR_BAD_SCALE;
    const long long BH = (long long)B * H;
    const long long n_qt = (Sq + 127) / 128, n_kt = (Sk + 127) / 128;
    if (n_qt * BH > 0x7fffffffll || n_kt * BH > 0x7fffffffll) return FA_ERR_BAD_SHAPE;
    const size_t qb = (size_t)BH * Sq * D * 2, kb = (size_t)BH * Sk * D * 2, lb = (size_t)BH * Sq * 4;
    // outputs (dq, dk, dv, delta) must not overlap any input or each other
    const void *outs[4] = {dq, dk, dv, delta};
    const size_t out_b[4] = {qb, kb, kb, lb};
    const void *ins[6] = {q, k, v, o, lse, dout};
    const size_t in_b[6] = {qb, kb, kb, qb, lb, qb};
    for (int a = 0; a < 4; ++a) {
        for (int b = 0; b < 6; ++b)
            if (overlaps(outs[a], out_b[a], ins[b], in_b[b])) return FA_ERR_ALIAS;
        for (int b = a + 1; b < 4; ++b)
            if (overlaps(outs[a], out_b[a], outs[b], out_b[b])) return FA_ERR_ALIAS;
    }
    if (!get_encoder()) return fail_cuda(cudaErrorNotSupported);
    CUtensorMap tq, tk, tv, tdo, to, tdq, tdk, tdv;
    if (!encode_bhsd(&tq, q, D, Sq, BH, 128) || !encode_bhsd(&tk, k, D, Sk, BH, 128) ||
        !encode_bhsd(&tv, v, D, Sk, BH, 128) || !encode_bhsd(&tdo, dout, D, Sq, BH, 128) ||
        !encode_bhsd(&to, o, D, Sq, BH, 128) ||
        !encode_bhsd(&tdq, dq, D, Sq, BH, 128) || !encode_bhsd(&tdk, dk, D, Sk, BH, 128) ||
        !encode_bhsd(&tdv, dv, D, Sk, BH, 128))
        return fail_cuda(cudaErrorInvalidValue);
    fa::BwdParams p;
    p.lse = lse;
    p.delta = delta;
    p.Sq = Sq;
    p.Sk = Sk;
    p.n_qt = (int)n_qt;
    p.n_kt = (int)n_kt;
    p.causal = causal;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.timeout_ns = timeout_ns;
    const cudaError_t e = fa::launch_bwd(D, tq, tk, tv, tdo, to, tdq, tdk, tdv, p, BH, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return FA_OK;
}

extern "C" int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                      const void *dout, void *dq, void *dk, void *dv, float *delta, int B, int H, int Sq, int Sk,
                      int D, float scale, int causal, void *stream) {
    return bwd_checked(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, Sq, Sk, D, scale, causal, stream,
                       kWaitLimitNs);
}

extern "C" int fa_selftest_bwd_timeout(const void *q, const void *k, const void *v, const void *o, const float *lse,
                                       const void *dout, void *dq, void *dk, void *dv, float *delta, int B, int H,
                                       int Sq, int Sk, int D, float scale, int causal, unsigned long long timeout_ns,
                                       void *stream) {
    if (timeout_ns > kWaitLimitNs) return FA_ERR_BAD_SHAPE;
    return bwd_checked(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H, Sq, Sk, D, scale, causal, stream, timeout_ns);
}

extern "C" int fa_device_status(void *stream) {
    int v = 0, w = 0, x = 0;
    cudaError_t e = fa::status_read_and_clear(&v, (cudaStream_t)stream);
    if (e == cudaSuccess) e = fa::splitkv_status_read_and_clear(&w);
    if (e == cudaSuccess) e = fa::bwd_status_read_and_clear(&x);
    if (e != cudaSuccess) return fail_cuda(e);
    return v != FA_OK ? v : (w != FA_OK ? w : x);
}

extern "C" int fa_selftest_bounded_wait(int timeout_us, void *stream) {
    if (timeout_us < 1 || timeout_us > 1000000) return FA_ERR_BAD_SHAPE;
    const cudaError_t e = fa::launch_wait_selftest((unsigned long long)timeout_us * 1000ull, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return FA_OK;
}

extern "C" int fa_selftest_fwd_timeout(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                                       int H, int Sq, int Sk, int D, float scale, int causal,
                                       unsigned long long timeout_ns, void *stream) {
    const int st = check_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, scale);
    if (st != FA_OK) return st;
    if (causal != 0 && causal != 1) return FA_ERR_UNSUPPORTED_CAUSAL;
    if (causal && Sq != Sk) return FA_ERR_UNSUPPORTED_CAUSAL;
    if (timeout_ns > kWaitLimitNs) return FA_ERR_BAD_SHAPE;
    return launch_checked(q, k, v, o, lse, B, H, Sq, Sk, D, scale, -1, causal ? 0 : -1, stream, timeout_ns);
}
