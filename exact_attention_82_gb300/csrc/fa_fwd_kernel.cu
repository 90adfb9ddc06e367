// fa_fwd_kernel.cu -- FlashAttention-2 forward for GB300 (sm_103a).
//
// What it computes: O = softmax(scale * Q K^T [+ causal mask]) V and the row
// log-sum-exp, with the online softmax of the source walk-through
// "FlashAttention-2 相比 FlashAttention-1，到底改了什么", section
// "第二处源码差异：kernel 主循环怎么组织" (running row max m, running sum l,
// acc rescaled by exp(m - m_new), one division by l at the end).
//
// How it maps onto the chip (one CTA per 128-row query tile, the grid of the
// same page's section "第一处源码差异：launch grid 怎么铺": query blocks x
// batch x heads):
//   warp 4     TMA producer: the Q tile once, then K_j and V_j tiles into a
//              two-stage shared-memory ring (128-byte swizzle);
//   warp 5     allocates tensor memory and issues the tcgen05 MMAs from one
//              thread: S_j = Q K_j^T into one of two TMEM S buffers, and
//              O += P_j V_j into the TMEM O accumulator;
//   warps 0-3  softmax: thread t owns query row t (TMEM lane t), reads its S
//              row from TMEM, masks (first tile only), updates m and l,
//              writes P_j (bf16) to shared memory, rescales its O row in
//              TMEM when m grew, and in the epilogue multiplies O by 1/l,
//              stages it in shared memory for a TMA store and writes LSE.
// Key/value tiles run from the last one to the first, so the only tile that
// needs masking (the causal diagonal or the ragged last tile) comes first,
// as in the page's split into masking steps then unmasked steps; tiles
// wholly above the causal diagonal are never visited ("FlashAttention-2 —
// L3 Cross-Paper Synthesis", §3 item 4).
//
// Every barrier wait is bounded in time; a wait that gives up records a
// status code and the CTA winds down without trapping.
#include <math.h>
#include <stdint.h>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

__device__ int g_status_word = 0;

template <int D>
struct FwdCfg {
    static constexpr int BM = kBlockM, BN = kBlockN, STAGES = 2;
    static constexpr int NCH = D / 64;                       // 64-column (128-byte) chunks
    static constexpr uint32_t Q_BYTES = BM * D * 2;
    static constexpr uint32_t KV_BYTES = BN * D * 2;         // one K or one V tile
    static constexpr uint32_t P_BYTES = BM * BN * 2;
    static constexpr uint32_t Q_CHUNK = BM * 128;            // bytes per 64-col chunk
    static constexpr uint32_t KV_CHUNK = BN * 128;
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + STAGES * KV_BYTES;
    static constexpr uint32_t OFF_P = OFF_V + STAGES * KV_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_P + P_BYTES;
    static constexpr uint32_t BAR_BYTES = 256;
    static constexpr uint32_t USED = OFF_BAR + BAR_BYTES;
    // + alignment slack; at least 120 KB so that one CTA occupies an SM
    // (each CTA takes all 512 TMEM columns)
    static constexpr uint32_t SMEM = (USED + 1024 > 120 * 1024) ? USED + 1024 : 120 * 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O = 256;
    static constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, true);
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(OFF_P % 1024 == 0 && OFF_K % 1024 == 0 && OFF_V % 1024 == 0, "atoms");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

// barrier slots (8 bytes each) inside the OFF_BAR block
enum : uint32_t {
    B_Q_FULL = 0,
    B_K_FULL = 1,   // + stage (2)
    B_K_EMPTY = 3,  // + stage
    B_V_FULL = 5,   // + stage
    B_V_EMPTY = 7,  // + stage
    B_S_FULL = 9,   // + buffer (2)
    B_S_FREE = 11,  // + buffer
    B_P_FULL = 13,
    B_O_DONE = 14,
    B_DRAIN = 15,
    N_BARS = 16
};
constexpr uint32_t SLOT_TMEM = 160;   // byte offset of the TMEM base address
constexpr uint32_t SLOT_ABORT = 164;  // byte offset of the abort flag
constexpr unsigned long long kDrainNs = 20ull * 1000 * 1000;  // 20 ms

template <int D>
__global__ void __launch_bounds__(192, 1)
    fa_fwd_sm103a(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (sbase - raw_u32);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- which tile: blockIdx.x = bh * n_mblk + (query-block order)
    const int mi = (int)(blockIdx.x % (unsigned)p.n_mblk);
    const int bh = (int)(blockIdx.x / (unsigned)p.n_mblk);
    const int mblk = p.causal ? (p.n_mblk - 1 - mi) : mi;  // causal: longest first
    int j_hi = p.n_kv - 1;
    if (p.causal) j_hi = min(j_hi, (mblk * C::BM + C::BM - 1) / C::BN);
    const int n_iter = j_hi + 1;
    const bool mask_first = p.causal || (p.Sk % C::BN) != 0;

    const uint32_t sQ = sbase + C::OFF_Q;
    const uint32_t sK = sbase + C::OFF_K;
    const uint32_t sV = sbase + C::OFF_V;
    const uint32_t sP = sbase + C::OFF_P;
    const uint32_t bars = sbase + C::OFF_BAR;
    auto bar = [&](uint32_t i) { return bars + 8u * i; };
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + C::OFF_BAR + SLOT_ABORT);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbase + C::OFF_BAR + SLOT_TMEM);

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q_FULL), 1);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar(B_K_FULL + s), 1);
            mbar_init(bar(B_K_EMPTY + s), 1);
            mbar_init(bar(B_V_FULL + s), 1);
            mbar_init(bar(B_V_EMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_S_FULL + s), 1);
            mbar_init(bar(B_S_FREE + s), 128);
        }
        mbar_init(bar(B_P_FULL), 128);
        mbar_init(bar(B_O_DONE), 1);
        mbar_init(bar(B_DRAIN), 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(sbase + C::OFF_BAR + SLOT_TMEM, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const unsigned long long tlim = p.timeout_ns;

    if (warp == 4) {
        // ===================================================== TMA producer
        if (lane == 0) {
            tma_prefetch_map(&tm_q);
            tma_prefetch_map(&tm_k);
            tma_prefetch_map(&tm_v);
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            mbar_arrive_expect_tx(bar(B_Q_FULL), C::Q_BYTES);
            for (int c = 0; c < C::NCH; ++c)
                tma_load_3d(sQ + c * C::Q_CHUNK, &tm_q, c * 64, mblk * C::BM, bh, bar(B_Q_FULL), pol_q);
            int issued = 0;
            for (int it = 0; it < n_iter; ++it) {
                const int j = j_hi - it;
                const int st = it % C::STAGES;
                const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
                if (!mbar_wait(bar(B_K_EMPTY + st), ph ^ 1u, abort_flag, tlim, &g_status_word, FA_ERR_TIMEOUT))
                    break;
                mbar_arrive_expect_tx(bar(B_K_FULL + st), C::KV_BYTES);
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_3d(sK + st * C::KV_BYTES + c * C::KV_CHUNK, &tm_k, c * 64, j * C::BN, bh,
                                bar(B_K_FULL + st), pol_kv);
                if (!mbar_wait(bar(B_V_EMPTY + st), ph ^ 1u, abort_flag, tlim, &g_status_word, FA_ERR_TIMEOUT)) {
                    issued = it * 2 + 1;
                    break;
                }
                mbar_arrive_expect_tx(bar(B_V_FULL + st), C::KV_BYTES);
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_3d(sV + st * C::KV_BYTES + c * C::KV_CHUNK, &tm_v, c * 64, j * C::BN, bh,
                                bar(B_V_FULL + st), pol_kv);
                issued = it * 2 + 2;
            }
            // wind down: every copy this thread issued has landed before the
            // CTA may exit (already true on the normal path)
            mbar_wait_drain(bar(B_Q_FULL), 0, kDrainNs);
            for (int t = (issued > 4 ? issued - 4 : 0); t < issued; ++t) {
                const int it = t >> 1;
                const int st = it % C::STAGES;
                const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
                mbar_wait_drain(bar(((t & 1) ? B_V_FULL : B_K_FULL) + st), ph, kDrainNs);
            }
        }
    } else if (warp == 5) {
        // ======================================================= MMA issuer
        if (lane == 0) {
            bool ok = mbar_wait(bar(B_Q_FULL), 0, abort_flag, tlim, &g_status_word, FA_ERR_TIMEOUT);
            auto issue_pv = [&](int t) -> bool {
                const int st = t % C::STAGES;
                const uint32_t ph = (uint32_t)(t / C::STAGES) & 1u;
                if (!mbar_wait(bar(B_P_FULL), (uint32_t)t & 1u, abort_flag, tlim, &g_status_word, FA_ERR_TIMEOUT))
                    return false;
                if (!mbar_wait(bar(B_V_FULL + st), ph, abort_flag, tlim, &g_status_word, FA_ERR_TIMEOUT))
                    return false;
                tc_fence_after();
                const uint32_t vbase = sV + st * C::KV_BYTES;
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk) {
                    // A = P (K-major, 64-column chunks of 128 rows)
                    const uint64_t ad = sw128_desc(sP + (kk >> 2) * C::Q_CHUNK + (kk & 3) * 32, 16, 1024);
                    // B = V (MN-major: D contiguous; 16 key rows per step)
                    const uint64_t bd = sw128_desc(vbase + kk * 2048, C::KV_CHUNK, 1024);
                    tc_mma_ss(tmem + C::TM_O, ad, bd, C::IDESC_PV, (t > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar(B_O_DONE));
                tc_commit(bar(B_V_EMPTY + st));
                return true;
            };
            for (int it = 0; ok && it < n_iter; ++it) {
                const int st = it % C::STAGES;
                const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
                const int sb = it & 1;
                const uint32_t sph = (uint32_t)(it >> 1) & 1u;
                ok = mbar_wait(bar(B_K_FULL + st), ph, abort_flag, tlim, &g_status_word, FA_ERR_TIMEOUT) &&
                     mbar_wait(bar(B_S_FREE + sb), sph ^ 1u, abort_flag, tlim, &g_status_word, FA_ERR_TIMEOUT);
                if (!ok) break;
                tc_fence_after();
                const uint32_t kbase = sK + st * C::KV_BYTES;
                const uint32_t s_tmem = tmem + (sb ? C::TM_S1 : C::TM_S0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t ad = sw128_desc(sQ + (kk >> 2) * C::Q_CHUNK + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = sw128_desc(kbase + (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32, 16, 1024);
                    tc_mma_ss(s_tmem, ad, bd, C::IDESC_S, kk > 0 ? 1u : 0u);
                }
                tc_commit(bar(B_S_FULL + sb));
                tc_commit(bar(B_K_EMPTY + st));
                if (it > 0) ok = issue_pv(it - 1);
            }
            if (ok) issue_pv(n_iter - 1);
            // wind down: all MMAs issued here are complete before TMEM is freed
            tc_commit(bar(B_DRAIN));
            mbar_wait_drain(bar(B_DRAIN), 0, kDrainNs);
        }
    } else {
        // ============================================ softmax warpgroup
        const int row = threadIdx.x;  // 0..127 == TMEM lane
        const int row_g = mblk * C::BM + row;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const float sl2 = p.scale_log2;
        float m_run = -INFINITY;  // running max of the raw scores q.k
        float l_run = 0.f;        // running sum of exp2((s - m) * scale*log2e)
        bool ok = true;
        for (int it = 0; it < n_iter; ++it) {
            const int sb = it & 1;
            const uint32_t sph = (uint32_t)(it >> 1) & 1u;
            ok = mbar_wait(bar(B_S_FULL + sb), sph, abort_flag, tlim, &g_status_word, FA_ERR_TIMEOUT);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t s[4][32];
            const uint32_t s_tmem = tmem + lane_off + (sb ? C::TM_S1 : C::TM_S0);
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(s_tmem + c * 32, s[c]);
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_wait(s[c]);
            tc_fence_before();
            mbar_arrive(bar(B_S_FREE + sb));

            if (it == 0 && mask_first) {
                const int col0 = j_hi * C::BN;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int col = col0 + c * 32 + e;
                        if (col >= p.Sk || (p.causal && col > row_g)) s[c][e] = __float_as_uint(-INFINITY);
                    }
            }
            float mx = m_run;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(s[c][e]));
            const float neg_m = -mx * sl2;
            float sum = 0.f;
            uint32_t pk[4][16];
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float p0 = ex2_approx(fmaf(__uint_as_float(s[c][2 * e]), sl2, neg_m));
                    const float p1 = ex2_approx(fmaf(__uint_as_float(s[c][2 * e + 1]), sl2, neg_m));
                    sum += p0 + p1;
                    pk[c][e] = pack_bf16x2(p0, p1);
                }
            const float alpha = ex2_approx((m_run - mx) * sl2);  // 0 on the first tile
            l_run = l_run * alpha + sum;
            m_run = mx;

            if (it > 0) {
                // O holds P_{it-1} V_{it-1}; it must be complete before O is
                // rescaled and before the P buffer is overwritten
                ok = mbar_wait(bar(B_O_DONE), (uint32_t)(it - 1) & 1u, abort_flag, tlim, &g_status_word,
                               FA_ERR_TIMEOUT);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
                    const uint32_t o_tmem = tmem + lane_off + C::TM_O;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(o_tmem + c * 32, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(o_tmem + c * 32, o);
                        tmem_st_wait(o);
                    }
                }
            }
            // P row -> shared memory, K-major with the 128-byte swizzle:
            // 16-byte unit U of the row goes to chunk U/8, unit (U%8)^(row%8)
#pragma unroll
            for (int U = 0; U < 16; ++U) {
                const uint32_t addr = sP + (U >> 3) * C::Q_CHUNK + row * 128 + ((((uint32_t)U & 7u) ^ ((uint32_t)row & 7u)) << 4);
                st_shared_v4(addr, pk[U >> 2][(U & 3) * 4 + 0], pk[U >> 2][(U & 3) * 4 + 1],
                             pk[U >> 2][(U & 3) * 4 + 2], pk[U >> 2][(U & 3) * 4 + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B_P_FULL));
        }
        if (ok) {
            ok = mbar_wait(bar(B_O_DONE), (uint32_t)(n_iter - 1) & 1u, abort_flag, tlim, &g_status_word,
                           FA_ERR_TIMEOUT);
            ok = __all_sync(0xffffffffu, ok);
        }
        // all four warps agree before the shared epilogue barrier
        named_bar_sync(1, 128);
        const bool all_ok = (*abort_flag == 0u);
        if (ok && all_ok) {
            tc_fence_after();
            const float inv_l = 1.f / l_run;
            const uint32_t o_tmem = tmem + lane_off + C::TM_O;
            const uint32_t sO = sP;  // the P buffer is free once the last P V is done
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(o_tmem + c * 32, o);
                tmem_ld_wait(o);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int U = c * 4 + u;  // 16-byte unit (8 columns) of the output row
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack_bf16x2(__uint_as_float(o[u * 8 + 2 * e]) * inv_l,
                                           __uint_as_float(o[u * 8 + 2 * e + 1]) * inv_l);
                    const uint32_t addr = sO + (U >> 3) * C::Q_CHUNK + row * 128 + ((((uint32_t)U & 7u) ^ ((uint32_t)row & 7u)) << 4);
                    st_shared_v4(addr, w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (row == 0) {
#pragma unroll
                for (int c = 0; c < C::NCH; ++c) tma_store_3d(&tm_o, sO + c * C::Q_CHUNK, c * 64, mblk * C::BM, bh);
                bulk_commit_group();
                bulk_wait_group_read0();
            }
            if (row_g < p.Sq) {
                const float lse2 = m_run * sl2 + lg2_approx(l_run);  // log2 of sum exp
                p.lse[(size_t)bh * p.Sq + row_g] = lse2 * 0.69314718055994531f;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Wait-limit self test: one warp waits on a barrier that nothing arrives on.
__global__ void fa_wait_selftest(unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t barrier_word;
    __shared__ uint32_t abort_word;
    const uint32_t b = smem_u32(&barrier_word);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_word = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        (void)mbar_wait(b, 0, reinterpret_cast<volatile uint32_t *>(&abort_word), limit_ns, &g_status_word,
                        FA_ERR_TIMEOUT);
    __syncthreads();
}

int fwd_smem_bytes(int D) {
    return D == 64 ? (int)FwdCfg<64>::SMEM : (int)FwdCfg<128>::SMEM;
}

template <int D>
static cudaError_t launch_fwd_d(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                const CUtensorMap &tm_o, const FwdParams &p, long long n_ctas,
                                cudaStream_t stream) {
    static_assert(FwdCfg<D>::SMEM > 0, "");
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_sm103a<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)FwdCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    fa_fwd_sm103a<D><<<dim3((unsigned)n_ctas), dim3(192), FwdCfg<D>::SMEM, stream>>>(tm_q, tm_k, tm_v, tm_o, p);
    return cudaGetLastError();
}

cudaError_t launch_fwd(int D, const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                       const CUtensorMap &tm_o, const FwdParams &p, long long n_ctas, cudaStream_t stream) {
    if (D == 64) return launch_fwd_d<64>(tm_q, tm_k, tm_v, tm_o, p, n_ctas, stream);
    return launch_fwd_d<128>(tm_q, tm_k, tm_v, tm_o, p, n_ctas, stream);
}

cudaError_t status_read_and_clear(int *out, cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int));
    *out = v;
    return e;
}

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream) {
    fa_wait_selftest<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

}  // namespace fa
