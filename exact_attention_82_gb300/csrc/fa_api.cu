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

#include <mutex>

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

// 3-D map over a [BH, S, D] bf16 tensor: dims (D, S, BH), box (64, rows, 1),
// 128-byte swizzle, zero fill outside the tensor.  Being 3-D, a box never
// reaches into the next head's rows.
bool encode_bhsd(CUtensorMap *map, const void *ptr, int D, int S, long long BH, int box_rows) {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2u, (cuuint64_t)S * (cuuint64_t)D * 2u};
    const cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
                                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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
        case FA_ERR_UNSUPPORTED_D: s = "unsupported head dim (64 or 128)"; break;
        case FA_ERR_UNSUPPORTED_CAUSAL: s = "causal must be 0 or 1, and causal needs Sq == Sk"; break;
        case FA_ERR_MISALIGNED: s = "a pointer is not 16-byte aligned"; break;
        case FA_ERR_BAD_SCALE: s = "scale must be finite and > 0"; break;
        case FA_ERR_CUDA: s = "CUDA error"; break;
        case FA_ERR_TIMEOUT: s = "an on-chip wait gave up (bounded-wait timeout)"; break;
        case FA_ERR_ALIAS: s = "an output buffer overlaps an input or the other output"; break;
        case FA_ERR_BAD_WINDOW: s = "window bounds must be >= -1, and a bounded window needs Sq == Sk"; break;
        default: s = "unknown status"; break;
    }
    if (status == FA_ERR_CUDA && t_last_cuda != cudaSuccess)
        snprintf(t_errbuf, sizeof t_errbuf, "%s: %s", s, cudaGetErrorString(t_last_cuda));
    else
        snprintf(t_errbuf, sizeof t_errbuf, "%s", s);
    return t_errbuf;
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
                          int Sk, int D, float scale, int wl, int wr, void *stream) {
    if (!get_encoder()) return fail_cuda(cudaErrorNotSupported);
    const long long BH = (long long)B * H;
    const long long n_mblk = (Sq + fa::kCtaRows - 1) / fa::kCtaRows;
    CUtensorMap tm_q, tm_k, tm_v, tm_o;
    if (!encode_bhsd(&tm_q, q, D, Sq, BH, fa::kBlockM) || !encode_bhsd(&tm_k, k, D, Sk, BH, fa::kBlockN) ||
        !encode_bhsd(&tm_v, v, D, Sk, BH, fa::kBlockN) || !encode_bhsd(&tm_o, o, D, Sq, BH, fa::kBlockM))
        return fail_cuda(cudaErrorInvalidValue);
    fa::FwdParams p;
    p.lse = lse;
    p.Sq = Sq;
    p.Sk = Sk;
    p.n_mblk = (int)n_mblk;
    p.n_kv = (Sk + fa::kBlockN - 1) / fa::kBlockN;
    p.causal = (wr >= 0 && wl < 0) ? 1 : 0;  // triangular work: longest blocks first
    p.wl = wl < 0 ? -1 : wl;
    p.wr = wr < 0 ? -1 : wr;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.timeout_ns = kWaitLimitNs;
    const cudaError_t e = fa::launch_fwd(D, tm_q, tm_k, tm_v, tm_o, p, n_mblk * BH, (cudaStream_t)stream);
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

extern "C" int fa_device_status(void *stream) {
    int v = 0;
    const cudaError_t e = fa::status_read_and_clear(&v, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return v;
}

extern "C" int fa_selftest_bounded_wait(int timeout_us, void *stream) {
    if (timeout_us < 1 || timeout_us > 1000000) return FA_ERR_BAD_SHAPE;
    const cudaError_t e = fa::launch_wait_selftest((unsigned long long)timeout_us * 1000ull, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return FA_OK;
}
