// fa_fwd_kernel.cu -- FlashAttention-2 forward for GB300 (sm_103a).
//
// What it computes: O = softmax(scale * Q K^T [+ causal mask]) V and the row
// log-sum-exp, with the online softmax of the source walk-through
// "FlashAttention-2 相比 FlashAttention-1，到底改了什么", section
// "第二处源码差异：kernel 主循环怎么组织" (running row max m, running sum l,
// acc rescaled by exp(m - m_new), a single division by l at the end).
//
// Mapping onto the chip.  The work items are the (query block, batch x head)
// pairs of the same page's launch grid (section "第一处源码差异：launch grid
// 怎么铺"); the kernel is persistent: one CTA per SM takes one item per round
// of gridDim.x items, in snake order (causal: all heads' longest query blocks
// first).  TMEM is allocated and the barriers initialised once, and the next
// item's Q and first K/V tiles load while the current item finishes, which
// takes the fixed cost of a CTA (launch, setup, load latency, epilogue) off
// every item but the first.  Each item is 256 query rows as two 128-row
// sub-tiles t = 0, 1, which share every K/V tile:
//   warps 10-11 idle (they complete the third warpgroup, whose registers go
//              to the softmax warpgroups);
//   warp 9     TMA producer: Q0 and Q1 of each item (as soon as the item
//              that used the buffer before has read it with its last S MMA;
//              with the three-tile query ring of 16-bit D = 128, the next
//              item's Q0 a whole item ahead), then K_j and V_j into two
//              shared-memory rings (128-byte swizzle), K one tile ahead;
//   warp 8     allocates all 512 tensor-memory (TMEM) columns and issues the
//              tcgen05 MMAs (the whole warp runs the issue loop, one elected
//              lane issues each instruction), in the order
//                S0_j = Q0 K_j^T,  O1 += P1_{j+1} V_{j+1},  S1_j = Q1 K_j^T,
//                O0 += P0_j V_j
//              so that while the tensor core works on one sub-tile the other
//              sub-tile's softmax runs (each softmax has two MMAs of slack);
//              16-bit D = 128 takes P_t V in two halves of 64 keys, the first
//              as soon as the softmax has written it;
//   warps 0-3  softmax of sub-tile 0, warps 4-7 of sub-tile 1: thread r owns
//              query row r (TMEM lane r): it reads its S row from TMEM, masks
//              (only on its first key tile), updates the running max and sum,
//              writes P (bf16) back over its S row in TMEM, where the P V MMA
//              reads it as its A operand, and at the end scales O by 1/l and
//              writes its O row straight to global memory, and its LSE.
// TMEM: S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D,256+2D); P_t sits in
// the first 64 columns of S_t (128 bf16 packed in pairs) -- except at 16-bit
// D = 64, where the 128 columns O leaves free hold P0 and P1 on their own
// [384,448) [448,512), and in the 8-bit path, where P_t (128 one-byte keys a
// row) goes to a shared-memory tile that the P V MMA reads as its A operand.
// With P separate the next S_t is issued as soon as the softmax has read S_t,
// instead of after P_t V has consumed P_t, and an item's O epilogue is
// deferred to the next item's first tile (see SEPP below).
//
// The row max is taken on a sub-tile's first key tile only (16-bit path);
// later tiles compute P against that stale max, which is exact because O and
// l are relative to the same max and divided at the end, and it takes the
// max pass and the O rescale off almost every iteration ("reduce non-matmul
// work", same page, section "第四处差异：v2 减少非 matmul 开销").  A tile is
// redone against its true max (and O and l rescaled) only when its row sum
// exceeds 2^64 or is not finite, i.e. when a score has grown more than 64
// (exp2 units) past the max in use.  The 8-bit path takes the row max every
// tile and moves the running max when it is exceeded by more than 2 (P must
// fit e4m3).  O_t is stable while sub-tile t is between "S_t full" and
// "P_t full" (S_t is issued after the previous P_t V; with P separate, from
// the previous P_t V's PV_DONE on), so the softmax thread rescales its own O
// row there when needed.
//
// Key tiles run from the last one to the first, so the only tile of a
// sub-tile that needs masking (causal diagonal or ragged last tile) is its
// first, and tiles wholly above the causal diagonal are never visited
// ("FlashAttention-2 — L3 Cross-Paper Synthesis", §3 item 4).
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

// QB: query buffers per sub-tile, 1 or 2 (2: a persistent CTA loads the next
// item's Q while the current item runs, where shared memory has room for it);
// or QB = 3: a ring of three query tiles shared by the two sub-tiles, one K
// stage fewer, so that a persistent CTA loads the next item's Q_0 a whole item
// ahead (16-bit inputs, D = 128).
template <int D, bool F8, int QB = 1>
struct FwdCfg {
    static constexpr int BM = kBlockM;  // rows per sub-tile (TMEM lanes)
    static constexpr int BN = kBlockN;  // keys per K/V tile
    static constexpr int EB = F8 ? 1 : 2;                 // bytes per Q/K/V element
    static constexpr int NQ = QB == 3 ? 3 : 2 * QB;       // query tile slots
    static constexpr int KST = (F8 || D == 64) ? 4 : (QB == 3 ? 2 : 3);
    static constexpr int VST = (F8 || D == 64) ? 4 : 2;
    static constexpr int NCH = D * EB / 128;              // 128-byte column chunks per Q/K/V row
    static constexpr int CH_ELEMS = 128 / EB;             // elements per chunk
    static constexpr uint32_t QT_BYTES = BM * D * EB;     // one query sub-tile
    static constexpr uint32_t KV_BYTES = BN * D * EB;     // one K or V tile
    static constexpr uint32_t CHUNK = 128 * 128;          // 128 rows x 128 bytes
    static constexpr uint32_t OFF_Q = 0;                  // query tile slots
    static constexpr uint32_t OFF_K = OFF_Q + NQ * QT_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + KST * KV_BYTES;
    // separate P (below): the 8-bit path keeps P_t in shared memory, 128 rows of
    // 128 one-byte keys (K-major, 128-byte swizzle), the A operand of its P V MMA
    static constexpr bool P_SMEM = F8;
    static constexpr uint32_t P_BYTES = P_SMEM ? BM * BN * EB : 0;  // one sub-tile's P
    static constexpr uint32_t OFF_P = OFF_V + VST * KV_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_P + 2 * P_BYTES;
    static constexpr uint32_t BAR_BYTES = 384;
    static constexpr uint32_t SMEM = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TM_O = 256;
    // Separate P: P_t does not overwrite S_t, so the next S_t can be issued as
    // soon as the softmax has read S_t (not only after P_t V has consumed P_t).
    // 16-bit D = 64 puts P_t in the 128 TMEM columns O leaves free; the 8-bit
    // path in shared memory (P_SMEM).
    static constexpr bool SEPP = D == 64 || F8;
    static constexpr uint32_t TM_P = TM_O + 2 * D;  // 16-bit separate P: P_t at TM_P + 64 t
    // one MMA takes 32 bytes of the contraction: 16 bf16 or 32 e4m3 elements
    static constexpr int S_STEPS = D * EB / 32;
    static constexpr int PV_STEPS = BN * EB / 32;
    static constexpr uint32_t V_STEP = (32 / EB) * 128;   // V bytes per PV step (keys x 128 B)
    static constexpr uint32_t IDESC_S = F8 ? idesc_e4m3_f32(BM, BN, false) : idesc_bf16_f32(BM, BN, false);
    static constexpr uint32_t IDESC_PV = F8 ? idesc_e4m3_f32(BM, D, true) : idesc_bf16_f32(BM, D, true);
    static_assert(D == 64 || D == 128, "head dim");
    static_assert(!F8 || D == 128, "8-bit rows must fill one 128-byte swizzle atom");
    static_assert(BM == 128 && BN == 128, "tile");
    static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && OFF_P % 1024 == 0 && OFF_BAR % 1024 == 0, "atoms");
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(SMEM > 114 * 1024, "one CTA per SM (it takes all TMEM columns)");
};

// 8-bit path: P is stored as e4m3 scaled by 2^kF8PShift, and the running max
// only moves when a tile's max exceeds it by more than kF8Lazy (exp2 units),
// so every stored value is at most 2^(kF8Lazy + kF8PShift) = 256 <= 448, the
// largest finite e4m3, while values down to 2^-16 of the running max stay
// representable (e4m3's smallest subnormal is 2^-9).
constexpr float kF8PShift = 6.f;
constexpr float kF8Lazy = 2.f;

// barrier slots (8 bytes each) inside the OFF_BAR block
enum : uint32_t {
    B_Q_FULL = 0,    // + 2 * buffer + sub-tile: an item's Q_t loaded
    B_Q_FREE = 4,    // + 2 * buffer + sub-tile: that item's last S_t has read Q_t
    B_K_FULL = 8,    // + stage (up to 4)
    B_K_EMPTY = 12,  // + stage
    B_V_FULL = 16,   // + stage
    B_V_EMPTY = 20,  // + stage
    B_S_FULL = 24,   // + sub-tile
    B_P_FULL = 26,   // + sub-tile
    B_O_DONE = 28,   // + sub-tile: the item's last P_t V is complete
    B_O_FREE = 30,   // + sub-tile: the softmax warps have read O_t out (128 arrivals)
    B_DRAIN = 32,
    B_S_FREE = 33,   // + sub-tile (separate P): the softmax warps have read S_t (128 arrivals)
    B_PV_DONE = 35,  // + sub-tile (separate P): a P_t V product is complete
    B_P_HALF = 37,   // + sub-tile: the first half of P_t (keys 0-63) is written (128 arrivals)
    B_PH_DONE = 39,  // + sub-tile: the P V product of that first half is complete
};
constexpr uint32_t SLOT_TMEM = 368;   // byte offset of the TMEM base address
constexpr uint32_t SLOT_ABORT = 372;  // byte offset of the abort flag
constexpr unsigned long long kDrainNs = 20ull * 1000 * 1000;  // 20 ms
constexpr int kThreads = 384;  // 3 warpgroups: softmax 0, softmax 1, MMA/TMA (+2 idle)
// Register split.  At launch every thread has 168 (3 warps per SM sub-partition);
// the MMA/TMA warpgroup drops to 104 and the softmax warpgroups rise to 200:
// 256 x 200 + 128 x 104 = 64512 = 384 x 168, the block's launch total.  Both
// sides then compile without spills (the MMA-issue loop is the critical path).
constexpr uint32_t kRegsSoftmax = 200, kRegsOther = 104;
static_assert(256 * kRegsSoftmax + 128 * kRegsOther == 384 * 168, "register split");

// Query buffers: two per sub-tile where they fit in shared memory (D = 64 and
// the 8-bit path), so that a persistent CTA loads the next item's Q while the
// current item runs; a three-tile ring for 16-bit D = 128 (see FwdCfg).
__host__ __device__ constexpr int query_buffers(int D, bool F8) { return (D == 64 || F8) ? 2 : 3; }

// One work item: 256 query rows (two sub-tiles) of one (batch, head), and the
// key tiles [jlo_t, jhi_t] each sub-tile needs.  Key tiles are loaded from J
// down to J - N + 1; sub-tile t takes part in load-order tiles first_t..last_t.
struct Item {
    int bh, row0;
    int qrow[2];  // first query row of each sub-tile (row0 and row0 + 128 unless paired apart)
    bool act1;  // sub-tile 1 has rows (sub-tile 0 always has)
    int jhi[2], jlo[2];
    int J, N;
    int first[2], last[2];
    // Block mask: mrow[t] is sub-tile t's row of the mask (null: every tile of
    // its range [jlo, jhi] taken -- no mask, or a row that keeps a contiguous
    // run).  A sub-tile whose row keeps no tile of its range ("none") takes part,
    // unmasked, in one loaded tile, and its rows are written as O = 0, LSE = -inf.
    const unsigned char *mrow[2];
    bool none[2];
    int cnt[2];  // (block mask) tiles sub-tile t takes part in
};

// Kept tiles of one mask row within [lo_b, hi_b]: the highest, the lowest (-1
// when none) and their count.  32 tiles at a time with independent loads, so a
// long row costs a few memory latencies rather than one per tile.
__device__ __forceinline__ void scan_mask_row(const unsigned char *mr, int lo_b, int hi_b, int &hi, int &lo,
                                              int &cnt) {
    hi = lo = -1;
    cnt = 0;
    for (int c0 = lo_b; c0 <= hi_b; c0 += 32) {
        uint32_t bits = 0;
#pragma unroll
        for (int b = 0; b < 32; ++b)
            if (c0 + b <= hi_b && __ldg(mr + c0 + b) != 0) bits |= 1u << b;
        if (bits) {
            if (lo < 0) lo = c0 + __ffs((int)bits) - 1;
            hi = c0 + 31 - __clz((int)bits);
            cnt += __popc(bits);
        }
    }
}

// The r-th item of this CTA: items are dealt out in rounds of gridDim.x in
// snake order (CTA b takes r G + b in even rounds, r G + G - 1 - b in odd
// ones), which evens out the CTAs' totals when items come longest first.
// Past the last item: a value >= p.n_items, and every later round's too.
__device__ __forceinline__ int item_index(int r) {
    const int G = (int)gridDim.x, b = (int)blockIdx.x;
    return r * G + ((r & 1) ? G - 1 - b : b);
}

template <bool WIN, bool MASK>
__device__ __forceinline__ Item item_at(const FwdParams &p, int k) {
    Item g;
    int mi;
    if (p.causal) {  // all heads' longest query blocks first
        mi = k / p.bh_count;
        g.bh = k - mi * p.bh_count;
    } else {
        g.bh = k / p.n_mblk;
        mi = k - g.bh * p.n_mblk;
    }
    const int mblk = p.causal ? (p.n_mblk - 1 - mi) : mi;
    g.row0 = mblk * kCtaRows;
    g.qrow[0] = g.row0;
    g.qrow[1] = g.row0 + kBlockM;
    if constexpr (MASK) {
        // Block mask: query blocks a and a + s (s = pair_stride) share an item, in
        // groups of 2 s blocks; the blocks after the last whole group pair up
        // with their neighbours.  With s = 1 this is the usual pairing.
        const int s = p.pair_stride, whole = (p.Sq + kBlockM - 1) / kBlockM / (2 * s);
        int qb0, qb1;
        if (mblk < whole * s) {
            qb0 = 2 * s * (mblk / s) + mblk % s;
            qb1 = qb0 + s;
        } else {
            qb0 = 2 * s * whole + 2 * (mblk - whole * s);
            qb1 = qb0 + 1;
        }
        g.qrow[0] = qb0 * kBlockM;
        g.qrow[1] = qb1 * kBlockM;
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int r_first = g.qrow[t], r_last = r_first + kBlockM - 1;
        g.jhi[t] = p.n_kv - 1;
        if (p.wr >= 0) g.jhi[t] = min(g.jhi[t], (r_last + p.wr) / kBlockN);
        g.jlo[t] = (WIN && p.wl >= 0) ? max(0, (r_first - p.wl) / kBlockN) : 0;
    }
    g.act1 = g.qrow[1] < p.Sq;
    g.mrow[0] = g.mrow[1] = nullptr;
    g.none[0] = g.none[1] = false;
    g.cnt[0] = g.cnt[1] = 0;
    if constexpr (MASK) {
        {
            // each sub-tile's range shrinks to the tiles its mask row keeps
            const unsigned char *mh = p.bmask + (size_t)g.bh * (size_t)p.bmask_hstride;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (t == 1 && !g.act1) break;
                const unsigned char *mr = mh + (size_t)(g.qrow[t] / kBlockM) * (size_t)p.n_kv;
                int hi, lo, cnt;
                scan_mask_row(mr, g.jlo[t], g.jhi[t], hi, lo, cnt);
                // a row that keeps every tile from its lowest to its highest is a plain
                // range: no per-tile lookups for it
                g.mrow[t] = (hi >= 0 && cnt == hi - lo + 1) ? nullptr : mr;
                g.none[t] = hi < 0;
                g.jhi[t] = hi;
                g.jlo[t] = lo;
                g.cnt[t] = hi < 0 ? 1 : cnt;
            }
            // a sub-tile that keeps nothing rides along on the other's first tile
            // (tile 0 when neither keeps anything)
            const bool live1 = g.act1 && !g.none[1];
            if (g.none[0]) g.jhi[0] = g.jlo[0] = live1 ? g.jhi[1] : 0;
            if (g.act1 && g.none[1]) g.jhi[1] = g.jlo[1] = g.jhi[0];
        }
    }
    g.J = g.act1 ? max(g.jhi[0], g.jhi[1]) : g.jhi[0];
    if constexpr (MASK)
        g.N = g.J - (g.act1 ? min(g.jlo[0], g.jlo[1]) : g.jlo[0]) + 1;
    else
        g.N = g.J - g.jlo[0] + 1;  // sub-tile 0 reaches lowest
    g.first[0] = g.J - g.jhi[0];
    g.last[0] = g.J - g.jlo[0];
    g.first[1] = g.act1 ? g.J - g.jhi[1] : g.N;
    g.last[1] = g.act1 ? g.J - g.jlo[1] : -1;
    return g;
}

// Does sub-tile t of item g take part in load-order tile `it`?  Without a block
// mask: every tile of its range; with one: the tiles its mask row keeps.
template <bool MASK>
__device__ __forceinline__ bool takes_part(const Item &g, int t, int it) {
    if (it < g.first[t] || it > g.last[t]) return false;
    if constexpr (MASK) {
        if (g.mrow[t] && !g.none[t]) return __ldg(g.mrow[t] + (g.J - it)) != 0;
    }
    return true;
}
// Is load-order tile `it` loaded at all (some sub-tile takes part)?
template <bool MASK>
__device__ __forceinline__ bool tile_live(const Item &g, int it) {
    return takes_part<MASK>(g, 0, it) || takes_part<MASK>(g, 1, it);
}
// The next load-order tile after `it` that is loaded (g.N if none).
template <bool MASK>
__device__ __forceinline__ int next_live(const Item &g, int it) {
    if constexpr (MASK) {
        do {
            ++it;
        } while (it < g.N && !tile_live<MASK>(g, it));
        return it;
    } else {
        return it + 1;
    }
}

// Block mask, MMA warp: which sub-tiles take part in 128 load-order tiles at a
// time, gathered by the warp's 32 lanes with ballots, so that the issue loop
// tests register bits instead of waiting on the mask's bytes in memory.  Every
// lane runs the issue loop and takes the same branches, as the ballots need.
struct PartBits {
    int base;               // first load-order tile the words cover (a multiple of 128)
    uint32_t w0[4], w1[4];  // bit b of word q: tile base + 32 q + b taken by sub-tile 0 / 1
};
template <bool MASK>
__device__ __forceinline__ void part_fill(PartBits &pb, const Item &g, int base, int lane) {
    pb.base = base;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int it = base + 32 * q + lane;
        pb.w0[q] = __ballot_sync(0xffffffffu, it < g.N && takes_part<MASK>(g, 0, it));
        pb.w1[q] = __ballot_sync(0xffffffffu, it < g.N && takes_part<MASK>(g, 1, it));
    }
}
__device__ __forceinline__ uint32_t part_word(const uint32_t (&w)[4], int q) {
    return q == 0 ? w[0] : q == 1 ? w[1] : q == 2 ? w[2] : w[3];
}
// bit 0: sub-tile 0 takes tile `it`, bit 1: sub-tile 1 does (it >= pb.base)
template <bool MASK>
__device__ __forceinline__ uint32_t part_of(PartBits &pb, const Item &g, int it, int lane) {
    if (it - pb.base >= 128) part_fill<MASK>(pb, g, it & ~127, lane);
    const int q = (it - pb.base) >> 5, b = (it - pb.base) & 31;
    return ((part_word(pb.w0, q) >> b) & 1u) | (((part_word(pb.w1, q) >> b) & 1u) << 1);
}
// the next tile after `it` that some sub-tile takes (g.N if none)
template <bool MASK>
__device__ __forceinline__ int part_next(PartBits &pb, const Item &g, int it, int lane) {
    for (int j = it + 1; j < g.N;) {
        if (j - pb.base >= 128) part_fill<MASK>(pb, g, j & ~127, lane);
        const int q = (j - pb.base) >> 5, b = (j - pb.base) & 31;
        const uint32_t w = (part_word(pb.w0, q) | part_word(pb.w1, q)) >> b;
        if (w) return j + __ffs((int)w) - 1;
        j += 32 - b;
    }
    return g.N;
}

// WIN: a bounded key band (window_left >= 0 or window_right > 0).  Without it
// (full or causal attention) only a sub-tile's first key tile can need a mask
// and every row has an allowed key in it, which the code below exploits.
// F8: Q, K, V are e4m3 with per-tensor scales (D = 128, no bounded band).
// MASK: a block mask keeps, per 128-row query block, a set of 128-key
// tiles ("FlashAttention-2 — L3 Cross-Paper Synthesis", §5 item 4: causal block
// skipping generalised into one sparse-block-skip mechanism).  An item's two
// sub-tiles still share one K/V stream -- the tiles either of them keeps, in the
// same descending order; tiles neither keeps are never loaded -- and each
// sub-tile takes part only in its own tiles, so its S, P and P V run on those
// alone.  Causal and full attention keep the property that only a sub-tile's
// first processed tile needs a mask and that every row has a key in it (the
// tiles a row keeps lie at or below its diagonal tile).  A sub-tile that keeps
// nothing rides along, unmasked, on one loaded tile and its rows are written as
// O = 0 and LSE = -inf.  (Instantiations of their own: the scan of the mask,
// even untaken, slowed the plain banded kernel by 11%.)
template <int D, bool WIN, bool F8, bool MASK>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_sm103a(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    constexpr int QB = query_buffers(D, F8);
    using C = FwdCfg<D, F8, QB>;
    static_assert(!(F8 && WIN), "the 8-bit path has no bounded band");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (sbase - raw_u32);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const uint32_t sQ = sbase + C::OFF_Q;
    const uint32_t sK = sbase + C::OFF_K;
    const uint32_t sV = sbase + C::OFF_V;
    const uint32_t bars = sbase + C::OFF_BAR;
    auto bar = [&](uint32_t i) { return bars + 8u * i; };
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(gbase + C::OFF_BAR + SLOT_ABORT);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(gbase + C::OFF_BAR + SLOT_TMEM);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::KST; ++s) {
            mbar_init(bar(B_K_FULL + s), 1);
            mbar_init(bar(B_K_EMPTY + s), 1);
        }
        for (int s = 0; s < C::VST; ++s) {
            mbar_init(bar(B_V_FULL + s), 1);
            mbar_init(bar(B_V_EMPTY + s), 1);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(bar(B_Q_FULL + i), 1);
            mbar_init(bar(B_Q_FREE + i), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(B_S_FULL + t), 1);
            mbar_init(bar(B_P_FULL + t), 128);
            mbar_init(bar(B_O_DONE + t), 1);
            mbar_init(bar(B_O_FREE + t), 128);
        }
        mbar_init(bar(B_DRAIN), 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(B_S_FREE + t), 128);
            mbar_init(bar(B_PV_DONE + t), 1);
            mbar_init(bar(B_P_HALF + t), 128);
            mbar_init(bar(B_PH_DONE + t), 1);
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 8) {
        tmem_alloc(sbase + C::OFF_BAR + SLOT_TMEM, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const unsigned long long tlim = p.timeout_ns;

    auto wait = [&](uint32_t b, uint32_t parity) {
        return mbar_wait(bar(b), parity, abort_flag, tlim, &g_status_word, FA_ERR_TIMEOUT);
    };

    if (warp >= 10) {
        regs_decrease<kRegsOther>();  // idle warps: give their registers away
    } else if (warp == 9) {
        // ===================================================== TMA producer
        regs_decrease<kRegsOther>();
        if (lane == 0) {
            tma_prefetch_map(&tm_q);
            tma_prefetch_map(&tm_k);
            tma_prefetch_map(&tm_v);
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            int nk = 0, nv = 0;      // K and V tiles loaded so far (ring positions), over all items
            int qn0 = 0, qn1 = 0;    // Q_0 and Q_1 loads so far
            bool ok = true;
            auto load_k = [&](const Item &g, int it) -> bool {
                const int st = nk % C::KST;
                if (!wait(B_K_EMPTY + st, ((uint32_t)(nk / C::KST) & 1u) ^ 1u)) return false;
                mbar_arrive_expect_tx(bar(B_K_FULL + st), C::KV_BYTES);
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_3d(sK + st * C::KV_BYTES + c * C::CHUNK, &tm_k, c * C::CH_ELEMS, (g.J - it) * C::BN,
                                g.bh, bar(B_K_FULL + st), pol_kv);
                ++nk;
                return true;
            };
            auto load_v = [&](const Item &g, int it) -> bool {
                const int st = nv % C::VST;
                if (!wait(B_V_EMPTY + st, ((uint32_t)(nv / C::VST) & 1u) ^ 1u)) return false;
                mbar_arrive_expect_tx(bar(B_V_FULL + st), C::KV_BYTES);
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_3d(sV + st * C::KV_BYTES + c * C::CHUNK, &tm_v, c * C::CH_ELEMS, (g.J - it) * C::BN,
                                g.bh, bar(B_V_FULL + st), pol_kv);
                ++nv;
                return true;
            };
            // three-tile ring: the q-th query tile loaded goes to slot q % 3, in the
            // order Q_0, Q_1 of item 0, Q_0, Q_1 of item 1, ... (Q_1 only where
            // the item has a second sub-tile), once the tile three loads earlier
            // has been read by its item's last S
            int qr = 0;
            auto load_q_ring = [&](const Item &g, int t) -> bool {
                const int slot = qr % 3, use = qr / 3;
                if (use > 0 && !wait(B_Q_FREE + slot, (uint32_t)(use - 1) & 1u)) return false;
                mbar_arrive_expect_tx(bar(B_Q_FULL + slot), C::QT_BYTES);
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_3d(sQ + slot * C::QT_BYTES + c * C::CHUNK, &tm_q, c * C::CH_ELEMS,
                                t ? g.qrow[1] : g.qrow[0], g.bh, bar(B_Q_FULL + slot), pol_q);
                ++qr;
                return true;
            };
            for (int r = 0, k = item_index(0); ok && k < p.n_items; k = item_index(++r)) {
                const Item g = item_at<WIN, MASK>(p, k);
                if constexpr (QB == 3) {
                    // this item's Q_0 was loaded one item ahead (below), except the first
                    if (r == 0) ok = load_q_ring(g, 0);
                    if (ok && g.act1) ok = load_q_ring(g, 1);
                    if (ok) ok = load_k(g, 0);
                    const int kn = item_index(r + 1);
                    if (ok && kn < p.n_items) ok = load_q_ring(item_at<WIN, MASK>(p, kn), 0);
                    for (int it = 0, nx; ok && it < g.N; it = nx) {  // tiles no sub-tile takes are skipped
                        nx = next_live<MASK>(g, it);
                        if (nx < g.N) ok = load_k(g, nx);
                        if (ok) ok = load_v(g, it);
                    }
                    continue;
                }
                // Q_t of this item into buffer qn % QB, once the last S_t of the item
                // that used the buffer before has read it
                auto load_q = [&](int t, int &qn) -> bool {
                    const int b = qn % QB, use = qn / QB;  // use-th load into buffer b
                    const uint32_t qb = 2 * b + t;
                    if (use > 0 && !wait(B_Q_FREE + qb, (uint32_t)(use - 1) & 1u)) return false;
                    mbar_arrive_expect_tx(bar(B_Q_FULL + qb), C::QT_BYTES);
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_3d(sQ + qb * C::QT_BYTES + c * C::CHUNK, &tm_q, c * C::CH_ELEMS,
                                    t ? g.qrow[1] : g.qrow[0], g.bh, bar(B_Q_FULL + qb), pol_q);
                    ++qn;
                    return true;
                };
                ok = load_q(0, qn0) && (!g.act1 || load_q(1, qn1));
                if (ok) ok = load_k(g, 0);
                for (int it = 0, nx; ok && it < g.N; it = nx) {
                    nx = next_live<MASK>(g, it);
                    if (nx < g.N) ok = load_k(g, nx);
                    if (ok) ok = load_v(g, it);
                }
            }
            // wind down: every copy issued here has landed before the CTA may exit
            for (int i = (qr > 3 ? qr - 3 : 0); i < qr; ++i)
                mbar_wait_drain(bar(B_Q_FULL + i % 3), (uint32_t)(i / 3) & 1u, kDrainNs);
            for (int i = (qn0 > QB ? qn0 - QB : 0); i < qn0; ++i)
                mbar_wait_drain(bar(B_Q_FULL + 2 * (i % QB)), (uint32_t)(i / QB) & 1u, kDrainNs);
            for (int i = (qn1 > QB ? qn1 - QB : 0); i < qn1; ++i)
                mbar_wait_drain(bar(B_Q_FULL + 2 * (i % QB) + 1), (uint32_t)(i / QB) & 1u, kDrainNs);
            for (int i = (nk > C::KST ? nk - C::KST : 0); i < nk; ++i)
                mbar_wait_drain(bar(B_K_FULL + i % C::KST), (uint32_t)(i / C::KST) & 1u, kDrainNs);
            for (int i = (nv > C::VST ? nv - C::VST : 0); i < nv; ++i)
                mbar_wait_drain(bar(B_V_FULL + i % C::VST), (uint32_t)(i / C::VST) & 1u, kDrainNs);
        }
    } else if (warp == 8) {
        // ======================================================= MMA issuer
        regs_decrease<kRegsOther>();
        {
            // The whole warp runs this loop and every lane takes the same
            // branches (the waits' results are agreed across the warp); each
            // MMA and commit is issued by one elected lane as a predicated
            // instruction.  A single thread looping alone over the same code,
            // with a branch around every group, issued ~10% fewer MMAs per
            // second: issuing is on the critical path of every tile (one
            // tcgen05.mma costs nearly as long as a 128x128x16 MMA runs), so
            // the loop is also kept lean: descriptors are a 64-bit base plus
            // compile-time offsets (the start-address field cannot carry:
            // shared addresses < 256 KB), ring stages and phases advance
            // incrementally, and participation is a precomputed iteration
            // range per sub-tile.
            auto wait = [&](uint32_t b, uint32_t parity) {
                return __all_sync(0xffffffffu,
                                  mbar_wait(bar(b), parity, abort_flag, tlim, &g_status_word, FA_ERR_TIMEOUT));
            };
            const uint64_t dqb = sw128_desc(sQ, 16, 1024);  // query buffer 0 of sub-tile 0
            const uint64_t dk = sw128_desc(sK, 16, 1024);
            const uint64_t dv = sw128_desc(sV, C::CHUNK, 1024);
            const uint64_t dp = sw128_desc(sbase + C::OFF_P, 16, 1024);  // 8-bit P_0 (shared memory)
            int sk = 0, sv = 0;       // ring stage of the next K and V tile to be read, over all items
            uint32_t kph = 0, vph = 0;
            int qn0 = 0, qn1 = 0;     // items so far in which sub-tile 0 / 1 took part
            int qr = 0;               // three-tile ring: query tiles consumed so far
            int npv0 = 0, npv1 = 0;   // P V products so far per sub-tile (P_FULL phases)
            uint32_t qfb0 = 0, qfb1 = 0, qfp0 = 0, qfp1 = 0;  // this item's Q_FULL barrier and phase per sub-tile
            bool ok = true;
            auto issue_s = [&](uint64_t dq, uint32_t s_tm, int stage) {
                const uint64_t dks = dk + ((stage * C::KV_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < C::S_STEPS; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
                    if constexpr (F8)
                        tc_mma_ss_f8(s_tm, dq + off, dks + off, C::IDESC_S, kk > 0 ? 1u : 0u);
                    else
                        tc_mma_ss(s_tm, dq + off, dks + off, C::IDESC_S, kk > 0 ? 1u : 0u);
                }
            };
            // O_t += P_t V over K-steps [k0, k1) (the item's first product
            // overwrites O_t); its waits are the caller's
            auto issue_pv_mma = [&](int t, bool accumulate, int stage, int k0, int k1) {
                const uint64_t dvs = dv + ((stage * C::KV_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < C::PV_STEPS; ++kk) {
                    if (kk < k0 || kk >= k1) continue;
                    // A = P_t in TMEM (8 columns = 32 bytes of keys per step); B = V, MN-major
                    tc_mma_ts(tmem + C::TM_O + t * D, tmem + t * 128 + kk * 8, dvs + ((kk * C::V_STEP) >> 4),
                              C::IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
                }
            };
            // before an item's first S_t: its Q_t has landed
            auto q_ready = [&](int t) { return wait(t ? qfb1 : qfb0, t ? qfp1 : qfp0); };
            // before an item's first P_t V: the softmax warps have read the previous item's O_t
            auto o_free = [&](int t) {
                const int q = t ? qn1 : qn0;
                return q == 0 || wait(B_O_FREE + t, (uint32_t)(q - 1) & 1u);
            };
            if constexpr (C::SEPP) {
                // Separate P (own TMEM columns at 16-bit D = 64, shared memory at
                // 8 bits).  Per key tile: S0_j and S1_j, each as soon as the softmax
                // has read the previous S_t (S_FREE), then the P V products of the
                // previous key tile -- so that, across an item boundary too, the next
                // S runs while this item's last softmax is still computing.  (Issuing
                // each sub-tile's S and previous P V together, S0 PV0 S1 PV1,
                // measured slower.)  Each P_t V product
                // commits PV_DONE_t, after which the softmax may overwrite P_t,
                // rescale O_t or (after an item's last product) read O_t out.  The
                // softmax reads an item's O_t before it signals the next item's
                // first P_t, and that product (which overwrites O_t) waits for the
                // signal, so O needs no hand-over barrier of its own.
                int ns0 = 0, ns1 = 0;  // S_t issued so far, over all items (S_FREE phases)
                struct PendingPV {     // a sub-tile's P V product still to issue (previous key tile)
                    bool on, first;
                    int stage;
                    uint32_t phase;
                } pd0 = {false, false, 0, 0u}, pd1 = {false, false, 0, 0u};
                bool vpend = false;    // the previous key tile's V stage is still to be released
                int svp = 0;
                auto pv_sepp = [&](int t, bool first, int stage, uint32_t phase) -> bool {
                    int &npv = t ? npv1 : npv0;
                    if (!wait(B_P_FULL + t, (uint32_t)npv & 1u)) return false;
                    if (!wait(B_V_FULL + stage, phase)) return false;
                    tc_fence_after();
                    const uint64_t dvs = dv + ((stage * C::KV_BYTES) >> 4);
                    if constexpr (C::P_SMEM) {
                        const uint64_t dps = dp + ((t * C::P_BYTES) >> 4);
#pragma unroll
                        for (int kk = 0; kk < C::PV_STEPS; ++kk)
                            tc_mma_ss_f8(tmem + C::TM_O + t * D, dps + ((kk * 32) >> 4), dvs + ((kk * C::V_STEP) >> 4),
                                         C::IDESC_PV, (!first || kk > 0) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < C::PV_STEPS; ++kk)
                            tc_mma_ts(tmem + C::TM_O + t * D, tmem + C::TM_P + t * 64 + kk * 8,
                                      dvs + ((kk * C::V_STEP) >> 4), C::IDESC_PV, (!first || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(bar(B_PV_DONE + t));
                    ++npv;
                    return true;
                };
                auto flush_pv = [&](int t, PendingPV &pd) -> bool {
                    if (!pd.on) return true;
                    pd.on = false;
                    return pv_sepp(t, pd.first, pd.stage, pd.phase);
                };
                for (int r = 0, k = item_index(0); ok && k < p.n_items; k = item_index(++r)) {
                    const Item g = item_at<WIN, MASK>(p, k);
                    const int qb0 = 2 * (qn0 % QB), qb1 = 2 * (qn1 % QB) + 1;
                    qfb0 = B_Q_FULL + qb0;
                    qfb1 = B_Q_FULL + qb1;
                    qfp0 = (uint32_t)(qn0 / QB) & 1u;
                    qfp1 = (uint32_t)(qn1 / QB) & 1u;
                    const uint64_t dq0 = dqb + ((qb0 * C::QT_BYTES) >> 4), dq1 = dqb + ((qb1 * C::QT_BYTES) >> 4);
                    PartBits pb;
                    if constexpr (MASK) part_fill<MASK>(pb, g, 0, lane);
                    // (block mask: tiles no sub-tile keeps are not loaded and skipped here)
                    for (int it = 0, nxt; ok && it < g.N; it = nxt) {
                        uint32_t pbits = 0;
                        if constexpr (MASK) {
                            pbits = part_of<MASK>(pb, g, it, lane);
                            nxt = part_next<MASK>(pb, g, it, lane);
                        } else {
                            nxt = it + 1;
                        }
                        ok = wait(B_K_FULL + sk, kph);
                        if (!ok) break;
                        const bool p0 = MASK ? (pbits & 1u) != 0 : takes_part<MASK>(g, 0, it);
                        const bool p1 = MASK ? (pbits & 2u) != 0 : takes_part<MASK>(g, 1, it);
                        if (p0) {
                            if (it == g.first[0]) ok = q_ready(0);
                            if (ok && ns0 > 0) ok = wait(B_S_FREE + 0, (uint32_t)(ns0 - 1) & 1u);
                            if (!ok) break;
                            tc_fence_after();
                            issue_s(dq0, tmem, sk);
                            tc_commit(bar(B_S_FULL + 0));
                            ++ns0;
                            if (it == g.last[0]) tc_commit(bar(B_Q_FREE + qb0));
                        }
                        if (p1) {
                            if (it == g.first[1]) ok = q_ready(1);
                            if (ok && ns1 > 0) ok = wait(B_S_FREE + 1, (uint32_t)(ns1 - 1) & 1u);
                            if (!ok) break;
                            tc_fence_after();
                            issue_s(dq1, tmem + 128, sk);
                            tc_commit(bar(B_S_FULL + 1));
                            ++ns1;
                            if (it == g.last[1]) tc_commit(bar(B_Q_FREE + qb1));
                        }
                        tc_commit(bar(B_K_EMPTY + sk));
                        ok = flush_pv(0, pd0) && flush_pv(1, pd1);
                        if (!ok) break;
                        if (vpend) tc_commit(bar(B_V_EMPTY + svp));  // both products of that tile are issued
                        pd0 = {p0, it == g.first[0], sv, vph};
                        pd1 = {p1, it == g.first[1], sv, vph};
                        vpend = true;
                        svp = sv;
                        if (++sk == C::KST) { sk = 0; kph ^= 1u; }
                        if (++sv == C::VST) { sv = 0; vph ^= 1u; }
                    }
                    ++qn0;
                    if (g.act1) ++qn1;
                }
                if (ok) ok = flush_pv(0, pd0) && flush_pv(1, pd1);
                if (ok && vpend) tc_commit(bar(B_V_EMPTY + svp));
            } else {
                for (int r = 0, k = item_index(0); ok && k < p.n_items; k = item_index(++r)) {
                    const Item g = item_at<WIN, MASK>(p, k);
                    const int first0 = g.first[0], last0 = g.last[0], first1 = g.first[1], last1 = g.last[1];
                    const int N = g.N;
                    // this item's query buffers (slots), their descriptors and barriers:
                    // buffer q % QB of sub-tile t for its q-th item, or ring slots
                    int qb0, qb1;
                    if constexpr (QB == 3) {
                        qb0 = qr % 3;
                        qb1 = (qr + 1) % 3;
                        qfp0 = (uint32_t)(qr / 3) & 1u;
                        qfp1 = (uint32_t)((qr + 1) / 3) & 1u;
                    } else {
                        qb0 = 2 * (qn0 % QB);
                        qb1 = 2 * (qn1 % QB) + 1;
                        qfp0 = (uint32_t)(qn0 / QB) & 1u;
                        qfp1 = (uint32_t)(qn1 / QB) & 1u;
                    }
                    qfb0 = B_Q_FULL + qb0;
                    qfb1 = B_Q_FULL + qb1;
                    const uint64_t dq0 = dqb + ((qb0 * C::QT_BYTES) >> 4), dq1 = dqb + ((qb1 * C::QT_BYTES) >> 4);
                    const uint32_t qf0 = B_Q_FREE + qb0, qf1 = B_Q_FREE + qb1;
                    int ipv0 = 0, ipv1 = 0;  // P V products of this item per sub-tile
                    {
                        // Tile by tile: S0_j, PV1_{j-1}, S1_j, PV0_j.
                        int svp = 0;          // V stage of the previous tile
                        uint32_t vpph = 0;
                        // P_t V in two halves: keys 0-63 once the softmax has written them
                        // (P_HALF; their completion is committed to PH_DONE), then keys
                        // 64-127 (P_FULL)
                        auto issue_pv = [&](int t, int ipv, int stage, uint32_t phase) -> bool {
                            int &npv = t ? npv1 : npv0;
                            if (!wait(B_P_HALF + t, (uint32_t)npv & 1u)) return false;
                            if (!wait(B_V_FULL + stage, phase)) return false;
                            if (ipv == 0 && !o_free(t)) return false;
                            tc_fence_after();
                            issue_pv_mma(t, ipv > 0, stage, 0, C::PV_STEPS / 2);
                            tc_commit(bar(B_PH_DONE + t));
                            if (!wait(B_P_FULL + t, (uint32_t)npv & 1u)) return false;
                            tc_fence_after();
                            issue_pv_mma(t, true, stage, C::PV_STEPS / 2, C::PV_STEPS);
                            ++npv;
                            return true;
                        };
                        bool kready = false;  // K_FULL of key tile `it` already waited for
                        bool prev1 = false;   // (block mask) sub-tile 1 took part in the previous loaded tile
                        int prev_it = -1;     // (block mask) that tile
                        PartBits pb;
                        if constexpr (MASK) part_fill<MASK>(pb, g, 0, lane);
                        // (block mask: tiles no sub-tile keeps are not loaded and skipped here)
                        for (int it = 0, nxt; ok && it < N; it = nxt) {
                            uint32_t pbits = 0;
                            if constexpr (MASK) {
                                pbits = part_of<MASK>(pb, g, it, lane);
                                nxt = part_next<MASK>(pb, g, it, lane);
                            } else {
                                nxt = it + 1;
                            }
                            if (!kready) ok = wait(B_K_FULL + sk, kph);
                            kready = false;
                            if (!ok) break;
                            tc_fence_after();
                            const bool p0 = MASK ? (pbits & 1u) != 0 : takes_part<MASK>(g, 0, it);
                            const bool p1 = MASK ? (pbits & 2u) != 0 : takes_part<MASK>(g, 1, it);
                            // sub-tile 1 took part in the previous tile, and whether that was its last
                            const bool pv1 = MASK ? prev1 : (it > first1 && it - 1 <= last1);
                            const bool pv1_last = MASK ? prev_it == last1 : it - 1 == last1;
                            if (p0) {
                                if (it == first0) {
                                    ok = q_ready(0);
                                    if (!ok) break;
                                    tc_fence_after();
                                }
                                issue_s(dq0, tmem, sk);
                                tc_commit(bar(B_S_FULL + 0));
                                if (it == last0) tc_commit(bar(qf0));
                            }
                            if (pv1) {
                                ok = issue_pv(1, ipv1++, svp, vpph);
                                if (!ok) break;
                                if (pv1_last) tc_commit(bar(B_O_DONE + 1));
                                tc_commit(bar(B_V_EMPTY + svp));
                            }
                            if (p1) {
                                if (it == first1) {
                                    ok = q_ready(1);
                                    if (!ok) break;
                                    tc_fence_after();
                                }
                                issue_s(dq1, tmem + 128, sk);
                                tc_commit(bar(B_S_FULL + 1));
                                if (it == last1) tc_commit(bar(qf1));
                            }
                            tc_commit(bar(B_K_EMPTY + sk));
                            // the next key tile's K is waited for here, so that P0 V and
                            // the next S0 issue back to back (S0 then waits on nothing)
                            if (nxt < N) {
                                ok = wait(B_K_FULL + (sk + 1 == C::KST ? 0 : sk + 1), sk + 1 == C::KST ? kph ^ 1u : kph);
                                if (!ok) break;
                                kready = true;
                            }
                            if (p0) {
                                ok = issue_pv(0, ipv0++, sv, vph);
                                if (!ok) break;
                                if (it == last0) tc_commit(bar(B_O_DONE + 0));
                                if (!p1) tc_commit(bar(B_V_EMPTY + sv));
                            }
                            if (++sk == C::KST) { sk = 0; kph ^= 1u; }
                            svp = sv;
                            vpph = vph;
                            if (++sv == C::VST) { sv = 0; vph ^= 1u; }
                            prev1 = p1;
                            prev_it = it;
                        }
                        if (ok && (MASK ? prev1 : last1 == N - 1)) {
                            ok = issue_pv(1, ipv1, svp, vpph);
                            if (ok) {
                                tc_commit(bar(B_O_DONE + 1));
                                tc_commit(bar(B_V_EMPTY + svp));
                            }
                        }
                    }
                    ++qn0;
                    if (g.act1) ++qn1;
                    qr += g.act1 ? 2 : 1;
                }
            }
            // wind down: every MMA issued here is complete before TMEM is freed
            tc_commit(bar(B_DRAIN));
            mbar_wait_drain(bar(B_DRAIN), 0, kDrainNs);
        }
    } else {
        // ============================================ softmax warpgroups
        regs_increase<kRegsSoftmax>();
        const int t = warp >> 2;            // sub-tile
        const int row = threadIdx.x & 127;  // row in the sub-tile == TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_tm = tmem + lane_off + t * 128;
        const uint32_t o_tm = tmem + lane_off + C::TM_O + t * D;
        const uint32_t p_tm = tmem + lane_off + C::TM_P + t * 64;  // 16-bit separate P only
        const uint32_t p_sm = sbase + C::OFF_P + t * C::P_BYTES + row * 128;  // 8-bit: this thread's P row
        const uint32_t p_sw = (uint32_t)row & 7u;  // 128-byte swizzle of that row
        const float sl2 = p.scale_log2;
        int ns = 0;  // S_t tiles so far, over all items (S_FULL phases)
        int od = 0;  // items so far in which this sub-tile took part (O_DONE phases)
        int npv = 0; // separate P: P_t tiles handed over so far (PV_DONE phases)
        // Separate P: an item's O epilogue is deferred until the next item's
        // first P_t is computed, so the O read sits beside that tile's work and
        // the global stores come after its P is handed over.
        bool pend = false;
        float pm = 0.f, pl = 1.f;
        int prow = 0, pbh = 0;
        // O / l -> bf16 -> row `rg` of head `bh` in global memory (16-byte
        // stores), and LSE; rows >= Sq are not written
        auto store_row = [&](const uint32_t (&o)[D / 32][32], float m, float l, int rg, int bh) {
            if (rg >= p.Sq) return;
            // 8-bit: O = descale_v * sum p' v / sum p' (the 2^kF8PShift cancels).
            // Block mask: a row with no allowed key (l = 0) is written as O = 0
            // exactly and LSE = -inf.
            const bool empty = MASK && !(l > 0.f);
            const float inv_l = empty ? 0.f : (F8 ? p.o_scale : 1.f) / l;
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.o) + ((size_t)bh * p.Sq + rg) * D);
#pragma unroll
            for (int c = 0; c < D / 32; ++c)
#pragma unroll
                for (int u = 0; u < 4; ++u) {  // 16-byte unit (8 columns) c * 4 + u of the row
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = empty ? 0u
                                     : pack_bf16x2(__uint_as_float(o[c][u * 8 + 2 * e]) * inv_l,
                                                   __uint_as_float(o[c][u * 8 + 2 * e + 1]) * inv_l);
                    dst[c * 4 + u] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            p.lse[(size_t)bh * p.Sq + rg] = empty
                                                ? -INFINITY
                                                : (m - (F8 ? kF8PShift : 0.f) + lg2_approx(l)) * 0.69314718055994531f;
        };
        // Each thread stores its own O row straight from registers, so a sub-tile's
        // Q buffer can take the next item's Q as early as possible.
        bool ok = true;
        Item g;
        float m_used = -INFINITY;  // max in exp2 units (raw score * scale*log2e) used for P
        float l_run = 0.f;         // sum of P over the keys seen, relative to m_used
        for (int r = 0, k = item_index(0); ok && k < p.n_items; k = item_index(++r)) {
            g = item_at<WIN, MASK>(p, k);
            if (t == 1 && !g.act1) continue;
            const int my_jhi = t ? g.jhi[1] : g.jhi[0], my_jlo = t ? g.jlo[1] : g.jlo[0];
            const int r_first = t ? g.qrow[1] : g.qrow[0], r_last = r_first + C::BM - 1;
            const int row_g = r_first + row;
            int n_t = my_jhi - my_jlo + 1;
            // block mask: the tiles of [my_jlo, my_jhi] this sub-tile's row keeps,
            // visited from the highest (jt steps down to each in turn)
            const bool none = MASK && (t ? g.none[1] : g.none[0]);
            const unsigned char *mrow = (MASK && !none) ? (t ? g.mrow[1] : g.mrow[0]) : nullptr;
            if constexpr (MASK) n_t = t ? g.cnt[1] : g.cnt[0];
            int jt = my_jhi + 1;
            // allowed keys of this row: [k_lo, k_hi)
            const int k_lo = (p.wl >= 0) ? row_g - p.wl : 0;
            const int k_hi = (p.wr >= 0) ? min(p.Sk, row_g + p.wr + 1) : p.Sk;
            m_used = -INFINITY;
            l_run = 0.f;
            for (int i = 0; i < n_t; ++i) {
                ok = wait(B_S_FULL + t, (uint32_t)ns & 1u);
                ++ns;
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                // S_t in two halves: the second half's load is in flight while the
                // exp pass works on the first (a tile that needs the whole row
                // first -- max, mask, 8-bit -- waits for both halves here)
                uint32_t s[4][32];
                tmem_ld32(s_tm, s[0]);
                tmem_ld32(s_tm + 32, s[1]);
                tmem_ld_wait2(s[0], s[1]);
                tmem_ld32(s_tm + 64, s[2]);
                tmem_ld32(s_tm + 96, s[3]);
                // A tile needs the mask unless every row of the sub-tile may see all
                // of its keys (causal: only the diagonal tile; ragged: the last).
                if constexpr (MASK) {
                    do {
                        --jt;
                    } while (mrow && __ldg(mrow + jt) == 0);
                }
                const int col0 = (MASK ? jt : my_jhi - i) * C::BN;
                // (A sub-tile whose mask row keeps nothing runs its one tile unmasked,
                // on finite scores, and its rows are written as O = 0, LSE = -inf.)
                const bool masked = (MASK && none)
                                        ? false
                                        : WIN ? (col0 + C::BN > p.Sk ||
                                                 (p.wr >= 0 && col0 + C::BN - 1 > r_first + p.wr) ||
                                                 (p.wl >= 0 && col0 < r_last - p.wl))
                                              : (i == 0 && (p.wr >= 0 || (p.Sk % C::BN) != 0));
                const int lim_lo = k_lo - col0, lim_hi = k_hi - col0;
                if (F8 || masked || (WIN ? __any_sync(0xffffffffu, m_used == -INFINITY) : i == 0))
                    tmem_ld_wait2(s[2], s[3]);
                if constexpr (C::P_SMEM) {
                    // the 8-bit path redoes nothing (its max is taken every tile), so
                    // S_t may be overwritten as soon as it is in registers
                    tc_fence_before();
                    mbar_arrive(bar(B_S_FREE + t));
                }
                auto apply_mask = [&]() {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (c * 32 + e < lim_lo || c * 32 + e >= lim_hi) s[c][e] = __float_as_uint(-INFINITY);
                };
                // Separate P (16-bit D = 64), full or causal attention: only the
                // right bound lim_hi cuts a row (k_lo = 0 <= col0), so each
                // 32-column chunk is, for the whole warp, either kept, cut partway
                // (masked element by element) or wholly past every row's bound --
                // then it is skipped (P = 0 there, and it takes no part in the max
                // or the sum).  On a causal diagonal tile a warp's 32 rows cut only
                // its own chunk.  (At D = 128 the extra code measured slower.)
                bool skip[4] = {false, false, false, false};
                auto mask_tile = [&]() {
                    if constexpr (WIN || F8 || !C::SEPP) {
                        apply_mask();
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            skip[c] = __all_sync(0xffffffffu, lim_hi <= c * 32);
                            if (!skip[c] && !__all_sync(0xffffffffu, lim_hi >= c * 32 + 32)) {
#pragma unroll
                                for (int e = 0; e < 32; ++e)
                                    if (c * 32 + e >= lim_hi) s[c][e] = __float_as_uint(-INFINITY);
                            }
                        }
                    }
                };
                if (masked) mask_tile();
                // O_t (this thread's row) times f, 16 columns at a time (few registers:
                // it runs while part of S and P is held).  O_t is stable from "S_t
                // full" until this sub-tile hands P_t (or its first half) over: S_t is
                // issued after the previous P_t V.
                auto scale_o = [&](float f) {
#pragma unroll 1
                    for (int c = 0; c < D / 16; ++c) {
                        uint32_t o[16];
                        tmem_ld16(o_tm + c * 16, o);
                        tmem_ld_wait16(o);
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                        tmem_st16(o_tm + c * 16, o);
                        tmem_st_wait16(o);
                    }
                };
                // 16-bit inputs without separate P hand P_t to the MMA warp in two
                // halves (keys 0-63, then 64-127): the first half's P V runs while
                // the second half is computed.
                auto hand_over_first_half = [&]() {
                    tc_fence_before();
                    mbar_arrive(bar(B_P_HALF + t));
                };
                if constexpr (F8) {
                    // The tile's row max every tile; the running max moves only when
                    // it is exceeded by more than kF8Lazy, and O is then rescaled.
                    float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int e = 0; e < 32; e += 8)
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                mq[q] = max3f(mq[q], __uint_as_float(s[c][e + 2 * q]),
                                              __uint_as_float(s[c][e + 2 * q + 1]));
                    const float m_tile = max3f(mq[0], mq[1], fmaxf(mq[2], mq[3])) * sl2;
                    const bool move = m_tile > m_used + kF8Lazy;  // always on the first tile
                    float alpha = 1.f;
                    if (move) {
                        alpha = ex2_approx(m_used - m_tile);  // 0 on the first tile
                        m_used = m_tile;
                    }
                    // p' = 2^(s*scale*log2e - m + kF8PShift) <= 256, packed four
                    // keys to a TMEM column (lowest key in the lowest byte)
                    const uint64_t c2 = f2_pack(sl2, sl2);
                    const float nm = kF8PShift - m_used;
                    const uint64_t nm2 = f2_pack(nm, nm);
                    uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
                    uint32_t pk[32];
                    auto exp8 = [&](int c) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            float x0, x1, x2, x3;
                            f2_unpack(f2_fma(f2_pack(__uint_as_float(s[c][4 * e]), __uint_as_float(s[c][4 * e + 1])),
                                             c2, nm2),
                                      x0, x1);
                            f2_unpack(f2_fma(f2_pack(__uint_as_float(s[c][4 * e + 2]),
                                                     __uint_as_float(s[c][4 * e + 3])),
                                             c2, nm2),
                                      x2, x3);
                            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                            const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
                            acc[(2 * e) & 3] = f2_add(acc[(2 * e) & 3], f2_pack(p0, p1));
                            acc[(2 * e + 1) & 3] = f2_add(acc[(2 * e + 1) & 3], f2_pack(p2, p3));
                            pk[c * 8 + e] = pack_e4m3x4(p0, p1, p2, p3);
                        }
                    };
#pragma unroll
                    for (int c = 0; c < 4; ++c) exp8(c);
                    float a0, a1, b0, b1;
                    f2_unpack(f2_add(acc[0], acc[1]), a0, a1);
                    f2_unpack(f2_add(acc[2], acc[3]), b0, b1);
                    l_run = l_run * alpha + ((a0 + a1) + (b0 + b1));
                    // P_t's buffer and O_t are ours once the previous P_t V product is complete
                    if (npv > 0) ok = __all_sync(0xffffffffu, wait(B_PV_DONE + t, (uint32_t)(npv - 1) & 1u));
                    if (!ok) break;
                    tc_fence_after();
                    // this row of P_t: eight 16-byte units, swizzled as the MMA reads them
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        st_shared_v4(p_sm + (((uint32_t)u ^ p_sw) << 4), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2],
                                     pk[4 * u + 3]);
                    fence_proxy_async_smem();  // visible to the tensor core before P_FULL
                    if (i > 0 && __any_sync(0xffffffffu, move)) {
                        // O rescaled 32 columns at a time (S and P are no longer held here,
                        // and the 8-bit max moves often enough for the width to matter)
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(o_tm + c * 32, o);
                            tmem_ld_wait(o);
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(o_tm + c * 32, o);
                            tmem_st_wait(o);
                        }
                    }
                } else {
                    // P is computed against the max already in use.  The row max is
                    // only taken on the first tile, or again when a score shows up
                    // more than 2^64 above that max (the sum of a half tile shows it,
                    // and inf and NaN too).  In the first half (nothing handed over
                    // yet, S intact in TMEM) the tile is redone against its true max;
                    // in the second half the max is raised to that half's and, once the
                    // first half's product has reached O, O is rescaled.
                    const uint64_t c2 = f2_pack(sl2, sl2);
                    float alpha = 1.f;
                    uint32_t pk[64];
                    auto take_max = [&]() {
                        // row max: four independent chains of three-input max
                        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            if (skip[c]) continue;
#pragma unroll
                            for (int e = 0; e < 32; e += 8)
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    mq[q] = max3f(mq[q], __uint_as_float(s[c][e + 2 * q]),
                                                  __uint_as_float(s[c][e + 2 * q + 1]));
                        }
                        const float m_new = fmaxf(m_used, max3f(mq[0], mq[1], fmaxf(mq[2], mq[3])) * sl2);
                        // 0 on a row's first keys; 1 while a row has seen no allowed key
                        alpha = (WIN && m_new == -INFINITY) ? 1.f : ex2_approx(m_used - m_new);
                        m_used = m_new;
                    };
                    // p = 2^(s*scale*log2e - m) for chunks [cb, ce): packed FMA pairs,
                    // then MUFU ex2; the sum in four packed partial sums.  use_skip:
                    // honour skipped chunks (a masked tile of full or causal attention
                    // with separate P); every other tile takes the straight-line pass.
                    auto exp_range = [&](int cb, int ce, bool use_skip) -> float {
                        const float nm = (WIN && m_used == -INFINITY) ? 0.f : -m_used;  // all-masked row: p = 0
                        const uint64_t nm2 = f2_pack(nm, nm);
                        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            if (c < cb || c >= ce) continue;
                            if (c == 2) tmem_ld_wait2(s[2], s[3]);  // the second half of S_t
                            if (use_skip && skip[c]) {
#pragma unroll
                                for (int e = 0; e < 16; ++e) pk[c * 16 + e] = 0u;
                                continue;
                            }
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                float x0, x1;
                                f2_unpack(f2_fma(f2_pack(__uint_as_float(s[c][2 * e]), __uint_as_float(s[c][2 * e + 1])),
                                                 c2, nm2),
                                          x0, x1);
                                const float p0 = ex2_approx(x0);
                                const float p1 = ex2_approx(x1);
                                acc[e & 3] = f2_add(acc[e & 3], f2_pack(p0, p1));
                                pk[c * 16 + e] = pack_bf16x2(p0, p1);
                            }
                        }
                        float a0, a1, b0, b1;
                        f2_unpack(f2_add(acc[0], acc[1]), a0, a1);
                        f2_unpack(f2_add(acc[2], acc[3]), b0, b1);
                        return (a0 + a1) + (b0 + b1);
                    };
                    auto reload_s = [&]() {
#pragma unroll
                        for (int c = 0; c < 4; ++c) tmem_ld32(s_tm + c * 32, s[c]);
#pragma unroll
                        for (int c = 0; c < 4; ++c) tmem_ld_wait(s[c]);
                    };
                    // the max is taken while any row of the warp has no allowed key
                    // yet (always on the first tile)
                    const bool took_max = WIN ? __any_sync(0xffffffffu, m_used == -INFINITY) : (i == 0);
                    if (took_max) take_max();
                    if constexpr (C::SEPP) {
                        const bool skips = !WIN && masked;
                        float sum = skips ? exp_range(0, 4, true) : exp_range(0, 4, false);
                        const bool redo = !took_max && __any_sync(0xffffffffu, !(sum <= 0x1p64f));
                        if (redo) {
                            reload_s();
                            if (masked) mask_tile();
                            take_max();
                            sum = exp_range(0, 4, false);  // a redo is never on a masked tile of full or causal attention
                        }
                        // S_t is read: the next S_t may overwrite it.  P_t and O_t are
                        // ours once the previous P_t V product is complete.
                        tc_fence_before();
                        mbar_arrive(bar(B_S_FREE + t));
                        if (npv > 0) ok = __all_sync(0xffffffffu, wait(B_PV_DONE + t, (uint32_t)(npv - 1) & 1u));
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll
                        for (int c = 0; c < 4; ++c) tmem_st16(p_tm + c * 16, &pk[c * 16]);
                        tmem_st_wait64(pk);
                        l_run = l_run * alpha + sum;
                        if (redo || (WIN && took_max && i > 0)) scale_o(alpha);
                    } else {
                        float sa = exp_range(0, 2, false);
                        const bool redo = !took_max && __any_sync(0xffffffffu, !(sa <= 0x1p64f));
                        if (redo) {
                            reload_s();
                            if (masked) mask_tile();
                            take_max();
                            sa = exp_range(0, 2, false);
                        }
                        if (redo || (WIN && took_max && i > 0)) scale_o(alpha);  // O holds earlier tiles at the old max
                        tmem_st16(s_tm, pk);  // keys 0-63: columns 0-31
                        tmem_st16(s_tm + 16, pk + 16);
                        tmem_st_wait(*reinterpret_cast<const uint32_t(*)[32]>(pk));
                        hand_over_first_half();
                        float sb = exp_range(2, 4, false);
                        float beta = 1.f;
                        if (!took_max && !redo && __any_sync(0xffffffffu, !(sb <= 0x1p64f))) {
                            // the first half's product must be in O before O is rescaled
                            ok = __all_sync(0xffffffffu, wait(B_PH_DONE + t, (uint32_t)(ns - 1) & 1u));
                            if (!ok) break;
                            tc_fence_after();
                            // keys 64-127 of S_t are still in TMEM (only columns 0-31 hold P)
                            tmem_ld32(s_tm + 64, s[2]);
                            tmem_ld32(s_tm + 96, s[3]);
                            tmem_ld_wait2(s[2], s[3]);
                            if (masked) mask_tile();
                            float mq[2] = {-INFINITY, -INFINITY};
#pragma unroll
                            for (int c = 2; c < 4; ++c)
#pragma unroll
                                for (int e = 0; e < 32; e += 4)
#pragma unroll
                                    for (int q = 0; q < 2; ++q)
                                        mq[q] = max3f(mq[q], __uint_as_float(s[c][e + 2 * q]),
                                                      __uint_as_float(s[c][e + 2 * q + 1]));
                            const float m_new = fmaxf(m_used, fmaxf(mq[0], mq[1]) * sl2);
                            beta = ex2_approx(m_used - m_new);
                            m_used = m_new;
                            scale_o(beta);
                            sb = exp_range(2, 4, false);
                        }
                        tmem_st16(s_tm + 32, pk + 32);  // keys 64-127: columns 32-63
                        tmem_st16(s_tm + 48, pk + 48);
                        tmem_st_wait(*reinterpret_cast<const uint32_t(*)[32]>(pk + 32));
                        l_run = (l_run * alpha + sa) * beta + sb;
                    }
                }
                if constexpr (C::SEPP) {
                    if (i == 0 && pend) {
                        // the previous item's O_t is complete (its last P_t V is): read it
                        // out before this P_t is handed over, whose product overwrites O_t
                        uint32_t o[D / 32][32];
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) tmem_ld32(o_tm + c * 32, o[c]);
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) tmem_ld_wait(o[c]);
                        tc_fence_before();
                        mbar_arrive(bar(B_P_FULL + t));
                        store_row(o, pm, pl, prow, pbh);
                        pend = false;
                    } else {
                        tc_fence_before();
                        mbar_arrive(bar(B_P_FULL + t));
                    }
                    ++npv;
                } else {
                    tc_fence_before();
                    mbar_arrive(bar(B_P_FULL + t));
                }
            }
            if (!ok) break;
            if (MASK && none) l_run = 0.f;  // no allowed key: O = 0, LSE = -inf
            if constexpr (C::SEPP) {  // epilogue deferred to the next item's first tile
                pend = true;
                pm = m_used;
                pl = l_run;
                prow = row_g;
                pbh = g.bh;
                continue;
            }
            ok = __all_sync(0xffffffffu, wait(B_O_DONE + t, (uint32_t)od & 1u));
            ++od;
            if (!ok) break;
            // ---- epilogue: O_t out of TMEM (after which the next item may
            // overwrite it), O / l -> bf16 -> this row of O in global memory; LSE
            tc_fence_after();
            uint32_t o[D / 32][32];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tmem_ld32(o_tm + c * 32, o[c]);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tmem_ld_wait(o[c]);
            tc_fence_before();
            mbar_arrive(bar(B_O_FREE + t));
            store_row(o, m_used, l_run, row_g, g.bh);
        }
        if constexpr (C::SEPP) {
            if (ok && pend) {  // the last item's epilogue
                ok = __all_sync(0xffffffffu, wait(B_PV_DONE + t, (uint32_t)(npv - 1) & 1u));
                if (ok) {
                    tc_fence_after();
                    uint32_t o[D / 32][32];
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) tmem_ld32(o_tm + c * 32, o[c]);
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) tmem_ld_wait(o[c]);
                    store_row(o, pm, pl, prow, pbh);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        __syncwarp();
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

template <int D, bool WIN, bool F8, bool MASK = false>
static cudaError_t launch_fwd_d(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                const FwdParams &p, int num_sms, cudaStream_t stream) {
    constexpr uint32_t smem = FwdCfg<D, F8, query_buffers(D, F8)>::SMEM;
    cudaError_t e =
        cudaFuncSetAttribute(fa_fwd_sm103a<D, WIN, F8, MASK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // Persistent CTAs (at most one per SM, each walking many items) take the
    // fixed cost of a CTA off every item but the first and even out items of
    // different length (causal: longest first, dealt out in snake order).
    const int n_ctas = p.n_items > num_sms ? num_sms : p.n_items;
    fa_fwd_sm103a<D, WIN, F8, MASK><<<dim3((unsigned)n_ctas), dim3(kThreads), smem, stream>>>(tm_q, tm_k, tm_v, p);
    return cudaGetLastError();
}

cudaError_t launch_fwd(int D, const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                       const FwdParams &p, int num_sms, cudaStream_t stream) {
    const bool win = p.wl >= 0 || p.wr > 0;
    if (p.bmask) {  // block mask: on the banded kernel only where a band is given
        if (D == 64)
            return win ? launch_fwd_d<64, true, false, true>(tm_q, tm_k, tm_v, p, num_sms, stream)
                       : launch_fwd_d<64, false, false, true>(tm_q, tm_k, tm_v, p, num_sms, stream);
        return win ? launch_fwd_d<128, true, false, true>(tm_q, tm_k, tm_v, p, num_sms, stream)
                   : launch_fwd_d<128, false, false, true>(tm_q, tm_k, tm_v, p, num_sms, stream);
    }
    if (D == 64)
        return win ? launch_fwd_d<64, true, false>(tm_q, tm_k, tm_v, p, num_sms, stream)
                   : launch_fwd_d<64, false, false>(tm_q, tm_k, tm_v, p, num_sms, stream);
    return win ? launch_fwd_d<128, true, false>(tm_q, tm_k, tm_v, p, num_sms, stream)
               : launch_fwd_d<128, false, false>(tm_q, tm_k, tm_v, p, num_sms, stream);
}

cudaError_t launch_fwd_fp8(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                           const FwdParams &p, int num_sms, cudaStream_t stream) {
    return launch_fwd_d<128, false, true>(tm_q, tm_k, tm_v, p, num_sms, stream);
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
