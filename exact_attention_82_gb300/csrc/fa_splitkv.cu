// fa_splitkv.cu -- split-KV attention for decode on GB300 (sm_103a).
//
// When a head has only a few query rows (decode: one new token attends to the
// whole key/value cache), the query-block parallelism of the forward kernel
// has nothing to split ("FlashAttention-2 — L3 Cross-Paper Synthesis", §5
// item 5: decode needs parallelism over the key/value sequence instead).  So
// the keys of each (batch, head) are cut into `splits` ranges; one CTA per
// (range, head) computes a partial result over its range, and a second kernel
// merges the partials -- the "merging intermediate results" the source
// walk-through "FlashAttention-2 相比 FlashAttention-1，到底改了什么" (section
// "第一处源码差异：launch grid 怎么铺") describes for v1's num_splits.
//
// Partial of range s for query row i, over its keys J_s:
//   lse_s = ln sum_{j in J_s} exp(scale q_i.k_j)
//   o_s   = sum_{j in J_s} exp(scale q_i.k_j - lse_s) v_j
// Merge:  lse = ln sum_s exp(lse_s),  o = sum_s exp(lse_s - lse) o_s.
//
// The work is bound by reading K and V from HBM, so it stays on the CUDA
// cores: a producer warp streams 64-key K and V tiles into a three-stage
// shared-memory ring with TMA (128-byte swizzle); in each of two consumer
// warps, lane l owns key 32w+l of a tile for the scores (its swizzled row
// reads are bank-conflict free) and columns of V for P*V; each warp runs an
// online softmax over its keys, and the two warps are merged in shared
// memory before the partial is written to the caller's workspace (fp32).
// About 100 KB of shared memory lets two CTAs share an SM, so one CTA's
// pipeline fill overlaps the other's streaming.
#include <math.h>
#include <stdint.h>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

__device__ int g_status_splitkv = 0;

template <int D>
struct SkvCfg {
    static constexpr int KEYS = kSplitTileKeys;        // keys per tile (64)
    static constexpr int ST = 3;                       // ring stages
    static constexpr int NCH = D / 64;                 // 64-column chunks per row
    static constexpr int CPL = D / 32;                 // V columns per lane
    static constexpr uint32_t TILE = KEYS * D * 2;     // one K or V tile
    static constexpr uint32_t CHUNK = KEYS * 128;      // KEYS rows x 128 bytes
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = ST * TILE;
    static constexpr uint32_t OFF_Q = 2 * ST * TILE;                 // q rows, fp32 [8][D]
    static constexpr int NW = KEYS / 32;               // consumer warps (a key per lane)
    static constexpr uint32_t OFF_ML = OFF_Q + kSplitMaxSq * D * 4;  // per-warp (m, l) [NW][8][2]
    static constexpr uint32_t OFF_BAR = OFF_ML + NW * kSplitMaxSq * 2 * 4;
    static constexpr uint32_t SMEM = OFF_BAR + 128 + 1024;          // + alignment slack
    static_assert(NW * kSplitMaxSq * D * 4 <= ST * TILE, "warp partials fit in the K ring");
    static_assert(SMEM <= 113 * 1024, "two CTAs per SM");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

constexpr int kSkvThreads = 96;  // warps 0-1 consumers (a key per lane), warp 2 producer
constexpr unsigned long long kSkvDrainNs = 20ull * 1000 * 1000;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int D, int SQ>
__global__ void __launch_bounds__(kSkvThreads, 2)
    fa_splitkv_partial(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const SplitParams p) {
    using C = SkvCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (sbase - raw_u32);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, bh = blockIdx.y;
    const int key0 = split * p.chunk;
    const int key1 = min(p.Sk, key0 + p.chunk);
    const int n_tiles = (key1 - key0 + C::KEYS - 1) / C::KEYS;

    float *sq = reinterpret_cast<float *>(gbase + C::OFF_Q);
    float *sml = reinterpret_cast<float *>(gbase + C::OFF_ML);
    const uint32_t bars = sbase + C::OFF_BAR;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };  // full[0..2], empty[3..5]
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + C::OFF_BAR + 64);

    // q rows of this head, widened to fp32 and pre-multiplied by scale*log2(e)
    const uint16_t *qg = reinterpret_cast<const uint16_t *>(p.q) + (size_t)bh * SQ * D;
    for (int t = threadIdx.x; t < SQ * D; t += kSkvThreads)
        sq[t] = __uint_as_float((uint32_t)qg[t] << 16) * p.scale_log2;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::ST; ++s) {
            mbar_init(bar(s), 1);
            mbar_init(bar(C::ST + s), C::NW);
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    auto wait = [&](int b, uint32_t parity) {
        return mbar_wait(bar(b), parity, abort_flag, p.timeout_ns, &g_status_splitkv, FA_ERR_TIMEOUT);
    };

    if (warp == C::NW) {
        // ===================================================== TMA producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();  // each key is read once
            int issued = 0;
            for (int it = 0; it < n_tiles; ++it) {
                const int st = it % C::ST;
                if (!wait(C::ST + st, ((uint32_t)(it / C::ST) & 1u) ^ 1u)) break;
                mbar_arrive_expect_tx(bar(st), 2 * C::TILE);
                const int row = key0 + it * C::KEYS;
                for (int c = 0; c < C::NCH; ++c) {
                    tma_load_3d(sbase + C::OFF_K + st * C::TILE + c * C::CHUNK, &tm_k, c * 64, row, bh, bar(st), pol);
                    tma_load_3d(sbase + C::OFF_V + st * C::TILE + c * C::CHUNK, &tm_v, c * 64, row, bh, bar(st), pol);
                }
                issued = it + 1;
            }
            for (int it = (issued > C::ST ? issued - C::ST : 0); it < issued; ++it)
                mbar_wait_drain(bar(it % C::ST), (uint32_t)(it / C::ST) & 1u, kSkvDrainNs);
        }
        __syncthreads();
        return;
    }

    // ===================================================== consumers
    float m[SQ], l[SQ], acc[SQ][C::CPL];
#pragma unroll
    for (int r = 0; r < SQ; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int c = 0; c < C::CPL; ++c) acc[r][c] = 0.f;
    }
    const int kr = warp * 32 + lane;  // this lane's key row within a tile
    bool ok = true;
    for (int it = 0; it < n_tiles; ++it) {
        const int st = it % C::ST;
        ok = ok && wait(st, (uint32_t)(it / C::ST) & 1u);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint32_t kt = C::OFF_K + st * C::TILE, vt = C::OFF_V + st * C::TILE;
        // ---- scores: this lane's key against every query row (exp2 units)
        float s[SQ];
#pragma unroll
        for (int r = 0; r < SQ; ++r) s[r] = 0.f;
#pragma unroll
        for (int u = 0; u < D / 8; ++u) {  // 16-byte unit u of the key row (8 elements)
            const uint32_t off = kt + (u >> 3) * C::CHUNK + kr * 128 + (((u & 7) ^ (kr & 7)) << 4);
            const uint4 w = *reinterpret_cast<const uint4 *>(gbase + off);
            const float kf[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                                 bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
#pragma unroll
            for (int r = 0; r < SQ; ++r) {
                const float4 q0 = *reinterpret_cast<const float4 *>(sq + r * D + u * 8);
                const float4 q1 = *reinterpret_cast<const float4 *>(sq + r * D + u * 8 + 4);
                s[r] = fmaf(q0.x, kf[0], s[r]);
                s[r] = fmaf(q0.y, kf[1], s[r]);
                s[r] = fmaf(q0.z, kf[2], s[r]);
                s[r] = fmaf(q0.w, kf[3], s[r]);
                s[r] = fmaf(q1.x, kf[4], s[r]);
                s[r] = fmaf(q1.y, kf[5], s[r]);
                s[r] = fmaf(q1.z, kf[6], s[r]);
                s[r] = fmaf(q1.w, kf[7], s[r]);
            }
        }
        const bool valid = key0 + it * C::KEYS + kr < key1;
        // ---- online softmax over this warp's 32 keys
        float pr[SQ];
#pragma unroll
        for (int r = 0; r < SQ; ++r) {
            if (!valid) s[r] = -INFINITY;
            const float m_new = fmaxf(m[r], warp_max(s[r]));
            const float mu = (m_new == -INFINITY) ? 0.f : m_new;  // no key yet: p = 0
            pr[r] = ex2_approx(s[r] - mu);
            const float alpha = (m_new == -INFINITY) ? 1.f : ex2_approx(m[r] - m_new);
            l[r] = l[r] * alpha + warp_sum(pr[r]);
#pragma unroll
            for (int c = 0; c < C::CPL; ++c) acc[r][c] *= alpha;
            m[r] = m_new;
        }
        // ---- P V: lane l owns columns [CPL*l, CPL*l + CPL) of V
#pragma unroll 4
        for (int j = 0; j < 32; ++j) {
            const int jr = warp * 32 + j;
            const int col = lane * C::CPL;
            const uint32_t off = vt + (col >> 6) * C::CHUNK + jr * 128 + ((((col & 63) >> 3) ^ (jr & 7)) << 4) +
                                 ((col & 7) << 1);
            float vf[C::CPL];
            if constexpr (C::CPL == 4) {
                const uint2 w = *reinterpret_cast<const uint2 *>(gbase + off);
                vf[0] = bf16lo(w.x);
                vf[1] = bf16hi(w.x);
                vf[2] = bf16lo(w.y);
                vf[3] = bf16hi(w.y);
            } else {
                const uint32_t w = *reinterpret_cast<const uint32_t *>(gbase + off);
                vf[0] = bf16lo(w);
                vf[1] = bf16hi(w);
            }
#pragma unroll
            for (int r = 0; r < SQ; ++r) {
                const float pj = __shfl_sync(0xffffffffu, pr[r], j);
#pragma unroll
                for (int c = 0; c < C::CPL; ++c) acc[r][c] = fmaf(pj, vf[c], acc[r][c]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::ST + st));
    }

    // ---- merge the consumer warps (their partials go into the drained K ring)
    named_bar_sync(1, 32 * C::NW);  // every consumer is past its last read of the ring
    float *sacc = reinterpret_cast<float *>(gbase + C::OFF_K);  // [NW][SQ][D]
#pragma unroll
    for (int r = 0; r < SQ; ++r) {
        if (lane == 0) {
            sml[(warp * kSplitMaxSq + r) * 2] = m[r];
            sml[(warp * kSplitMaxSq + r) * 2 + 1] = l[r];
        }
#pragma unroll
        for (int c = 0; c < C::CPL; ++c) sacc[(warp * SQ + r) * D + lane * C::CPL + c] = acc[r][c];
    }
    named_bar_sync(1, 32 * C::NW);
    const bool all_ok = ok && *abort_flag == 0u;
    for (int t = threadIdx.x; t < SQ * D; t += 32 * C::NW) {
        const int r = t / D, d = t % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::NW; ++w) M = fmaxf(M, sml[(w * kSplitMaxSq + r) * 2]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < C::NW; ++w) {
            const float mw = sml[(w * kSplitMaxSq + r) * 2];
            const float f = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
            L += sml[(w * kSplitMaxSq + r) * 2 + 1] * f;
            O += sacc[(w * SQ + r) * D + d] * f;
        }
        const size_t base = ((size_t)bh * p.splits + split) * SQ + r;
        if (all_ok) {
            p.o_part[base * D + d] = O / L;
            if (d == 0) p.lse_part[base] = (M + lg2_approx(L)) * 0.69314718055994531f;
        } else if (d == 0) {
            // a wait gave up: mark this partial invalid, so the merge yields NaN
            // rather than a blend of whatever the workspace held before
            p.lse_part[base] = __int_as_float(0x7fc00000);
        }
    }
    __syncthreads();
}

// Merge the splits of one (head, query row): one thread per output column.
template <int D>
__global__ void __launch_bounds__(128) fa_splitkv_combine(const SplitParams p) {
    const int r = blockIdx.x, bh = blockIdx.y, d = threadIdx.x;
    const size_t base = (size_t)bh * p.splits * p.Sq + r;  // partial (bh, split 0, row r)
    const size_t step = (size_t)p.Sq;                      // to the next split
    float M = -INFINITY;
    for (int s = 0; s < p.splits; ++s) M = fmaxf(M, p.lse_part[base + s * step]);
    float W = 0.f, O = 0.f;
    for (int s = 0; s < p.splits; ++s) {
        const float w = ex2_approx((p.lse_part[base + s * step] - M) * 1.4426950408889634f);
        W += w;
        if (d < D) O = fmaf(w, p.o_part[(base + s * step) * D + d], O);
    }
    const size_t orow = (size_t)bh * p.Sq + r;
    if (d < D) {
        __nv_bfloat16 h = __float2bfloat16_rn(O / W);
        reinterpret_cast<__nv_bfloat16 *>(p.o)[orow * D + d] = h;
    }
    if (d == 0) p.lse[orow] = M + lg2_approx(W) * 0.69314718055994531f;
}

int splitkv_smem_bytes(int D) { return D == 64 ? (int)SkvCfg<64>::SMEM : (int)SkvCfg<128>::SMEM; }

template <int D, int SQ>
static cudaError_t launch_partial(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const SplitParams &p,
                                  int BH, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(fa_splitkv_partial<D, SQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SkvCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    fa_splitkv_partial<D, SQ><<<dim3(p.splits, BH), dim3(kSkvThreads), SkvCfg<D>::SMEM, stream>>>(tm_k, tm_v, p);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_partial_sq(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const SplitParams &p,
                                     int BH, cudaStream_t stream) {
    switch (p.Sq) {
        case 1: return launch_partial<D, 1>(tm_k, tm_v, p, BH, stream);
        case 2: return launch_partial<D, 2>(tm_k, tm_v, p, BH, stream);
        case 3: return launch_partial<D, 3>(tm_k, tm_v, p, BH, stream);
        case 4: return launch_partial<D, 4>(tm_k, tm_v, p, BH, stream);
        case 5: return launch_partial<D, 5>(tm_k, tm_v, p, BH, stream);
        case 6: return launch_partial<D, 6>(tm_k, tm_v, p, BH, stream);
        case 7: return launch_partial<D, 7>(tm_k, tm_v, p, BH, stream);
        default: return launch_partial<D, 8>(tm_k, tm_v, p, BH, stream);
    }
}

cudaError_t launch_splitkv(int D, const CUtensorMap &tm_k, const CUtensorMap &tm_v, const SplitParams &p, int BH,
                           cudaStream_t stream) {
    cudaError_t e = (D == 64) ? launch_partial_sq<64>(tm_k, tm_v, p, BH, stream)
                              : launch_partial_sq<128>(tm_k, tm_v, p, BH, stream);
    if (e != cudaSuccess) return e;
    if (D == 64)
        fa_splitkv_combine<64><<<dim3(p.Sq, BH), dim3(128), 0, stream>>>(p);
    else
        fa_splitkv_combine<128><<<dim3(p.Sq, BH), dim3(128), 0, stream>>>(p);
    return cudaGetLastError();
}

// ------------------------------------------------- built-in scratch buffer
// Scratch for callers that cannot allocate device memory themselves (see
// fa_fwd_splitkv_noalloc in fa.h).  It lives in the library's own device
// image: every GPU that loads the library holds these bytes until the
// process exits, and every call on a device shares them.
static __device__ __align__(256) unsigned char g_splitkv_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the current device's context.  In
// host code the array's name is only a host-side stand-in, never a device
// address, so it is looked up with cudaGetSymbolAddress, with the device
// current, on every call: after the module is loaded that is a host-side
// table read, and nothing is cached that a context reset (cudaDeviceReset, or
// a primary context released and created again) could leave pointing at a
// module image that no longer exists.  The first call on a device loads the
// library's module there (with lazy loading), so it should come before any
// stream capture.
cudaError_t splitkv_scratch(void **out) {
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_splitkv_scratch);
    if (e != cudaSuccess) return e;
    *out = ptr;
    return cudaSuccess;
}

cudaError_t splitkv_status_read_and_clear(int *out) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_status_splitkv, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_status_splitkv, &zero, sizeof(int));
    *out = v;
    return e;
}

}  // namespace fa
