// Causal grouped-head attention on tcgen05 for sm_103a: forward, and the
// backward split into a key-side kernel (dK, dV) and a query-side kernel (dQ).
//
// Layout (padded token order, see routing.cu): the fused projection buffer
// qkv [P x W] holds for each row the query heads (n_heads x 128), then the
// key heads, then the value heads (n_kv x 128 each), bf16, after the rotary
// embedding.  seq_start[p] is the padded row where row p's sequence starts;
// rows of one sequence are consecutive, so row p attends to the keys
// [seq_start[p], p].  Query head j reads key/value head j / (n_heads / n_kv).
//
// Softmax statistics travel "transposed", one contiguous run per head:
// lseT [n_heads x ld_t] (log-sum-exp of a row's scaled scores, in log2 units)
// and DT [n_heads x ld_t] (rowsum(dO * O)), so that 128 consecutive rows of
// one head are one 512-byte bulk copy.
//
// Every kernel: warp 0 issues TMA loads (one elected thread), warp 1 owns
// TMEM and issues tcgen05.mma (one elected thread), warps 2-5 (128 threads,
// one tile row each, TMEM lane quarter = warp % 4) run the softmax arithmetic
// from tcgen05.ld and write bf16 operands back to shared memory in the
// 128-byte-swizzled K-major layout the next MMA reads.  Every mbarrier wait
// is bounded; on expiry the CTA raises the timeout status bit, every role
// stops, outstanding copies and MMAs are drained (bounded) and TMEM is freed.
#include <cuda.h>

#include <type_traits>

#include "internal.h"
#include "tc_ptx.cuh"

namespace mlk {

namespace {

using namespace tcx;

constexpr int HD = 128;                 // head width
constexpr int TB = 128;                 // rows per query / key tile
constexpr int BLK = TB * 128;           // one 128-row x 64-element bf16 block (16 KB)
constexpr float LOG2E = 1.4426950408889634f;

struct AttnMaps {
    CUtensorMap rows128;   // qkv, boxes of 64 columns x 128 rows
    CUtensorMap do128;     // dO [P x n_heads*128], boxes of 64 x 128 (backward only)
    CUtensorMap ds128;     // stored dS blocks [blocks*128 x 128], boxes of 64 x 128 (stored mode only)
};

struct AttnParams {
    const bf16* qkv;
    int ld_qkv;            // elements per row of qkv
    int n_heads, n_kv;
    const int* seq_start;  // [P] padded row where the row's sequence starts
    const int* meta;       // meta[0] = valid 128-row tiles
    int max_tiles;
    float scale;           // 1 / sqrt(head width)
    // forward outputs
    bf16* o;               // [P x n_heads*128]
    float* lseT;           // [n_heads x ld_t]
    int ld_t;
    // backward inputs / outputs
    const float* DT;       // [n_heads x ld_t]
    bf16* dqkv;            // [P x ld_qkv]: dQ, dK, dV in the columns of q, k, v
    int* counter;          // item counter of the persistent kernels (zeroed before each launch)
    bf16* ds;              // stored dS blocks (null: the query side recomputes them), see AttnArgs
    int ktc;               // key tiles per query tile in the stored layout
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Wait of one warp.  Fast path: every lane tests the barrier (converged, no
// shuffle); otherwise lane 0 polls it with the bounded wait and the warp
// learns the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int lane) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(bar, parity, abort_flag) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// 2^x with subnormal results flushed to zero (ex2.approx.ftz): one MUFU
// operation; softmax probabilities below 2^-126 do not matter.
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Dynamic item scheduling of the persistent kernels.  The loading thread takes
// item indices from a global counter (reset before each launch) and publishes
// each through a RING-slot ring in shared memory (slot value, then an arrive
// on the slot's "full" barrier, whose release orders the value before it);
// every other role takes the items from the ring in the same order and frees
// each slot on its "empty" barrier.  -1 ends the work.  Items are taken in
// the order of the counter, so the CTAs that finish early take more work.
constexpr int RING = 4;

struct RingPos {
    int slot = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void advance() {
        if (++slot == RING) { slot = 0; ph ^= 1u; }
    }
};

// Publish t (one thread).
__device__ __forceinline__ bool ring_put(uint32_t full, uint32_t empty, volatile int* slots, RingPos& rp, int t,
                                         volatile int* abort_flag) {
    if (!mbar_wait(empty + 8 * rp.slot, rp.ph ^ 1u, abort_flag)) return false;
    slots[rp.slot] = t;
    mbar_arrive(full + 8 * rp.slot);
    rp.advance();
    return true;
}

// Take the next item (one thread).
__device__ __forceinline__ bool ring_get(uint32_t full, uint32_t empty, const volatile int* slots, RingPos& rp, int& t,
                                         volatile int* abort_flag) {
    if (!mbar_wait(full + 8 * rp.slot, rp.ph, abort_flag)) return false;
    t = slots[rp.slot];
    mbar_arrive(empty + 8 * rp.slot);
    rp.advance();
    return true;
}

// Take the next item for a whole warp: lane 0 waits and frees the slot, the
// warp learns the item.
__device__ __forceinline__ bool ring_get_warp(uint32_t full, uint32_t empty, const volatile int* slots, RingPos& rp,
                                              int& t, volatile int* abort_flag, int lane) {
    int ok = 1, v = -1;
    if (lane == 0) {
        ok = mbar_wait(full + 8 * rp.slot, rp.ph, abort_flag) ? 1 : 0;
        if (ok) {
            v = slots[rp.slot];
            mbar_arrive(empty + 8 * rp.slot);
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    t = __shfl_sync(0xffffffffu, v, 0);
    rp.advance();
    return ok != 0;
}

// Descriptors are built once per product and moved by additions to their
// start-address field (bits 0-13, address >> 4): shared-memory addresses stay
// below 2^18, so the field never carries.  The one issuing thread then spends
// a few integer adds per MMA instead of rebuilding two descriptors.
// K-major 128-row operand block of 64 elements per row, K step 0; +2 per K
// step of 16 elements, +BLK_STEP per 64-element block.
__device__ __forceinline__ uint64_t kdesc(uint32_t blk) { return sdesc(blk, 16, 1024); }
constexpr uint32_t BLK_STEP = BLK >> 4;
// The same bytes read as an MN-major operand whose K index is the row: K block
// kb (64 rows) at +512 kb, 16-row K step at +128 kk, MN halves 16 KB apart.
__device__ __forceinline__ uint64_t mndesc(uint32_t base) { return sdesc(base, 2 * 8192, 1024); }

// 128 x 128 x 128 product: D (+)= A B^T with A, B both K-major (two 64-wide
// K blocks each).
__device__ __forceinline__ void mma_kk(uint32_t d, uint32_t a, uint32_t b, bool acc) {
    const uint32_t id = idesc_bf16(128, 0, 0, 128);
    const uint64_t ad = kdesc(a), bd = kdesc(b);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            umma_bf16(d, ad + kb * BLK_STEP + 2 * kk, bd + kb * BLK_STEP + 2 * kk, id,
                      (acc || kb || kk) ? 1u : 0u);
}

// Load a 128-row x 128-column bf16 tile of a row-major matrix as two
// K-major blocks (columns 0-63, 64-127).
__device__ __forceinline__ void load_tile128(uint32_t dst, const CUtensorMap* map, uint32_t bar, int col, int row) {
    tma_load_2d(dst, map, bar, col, row);
    tma_load_2d(dst + BLK, map, bar, col + 64, row);
}

}  // namespace

// ----------------------------------------------------------------------------
// Forward.  Work item = (128-row query tile, two query heads of one key/value
// group); key tiles of 128 rows run from the first row of the tile's first
// sequence up to the tile's last row and are loaded once for both heads.
// The kernel is persistent: one CTA per SM takes items from a global counter
// in tile-major order (so the CTAs running together share K / V tiles in L2),
// keeps its TMEM and barriers across items, and lets the next item's Q / K
// loads and first scores overlap the current item's output store.  Barrier phases follow a running count of the key tiles this CTA
// has processed.
//
// Warps: 0 loads K, 1 loads Q and V (K and V double-buffered), 2 issues the
// MMAs, 3-6 and 7-10 are the softmax warpgroups of the two heads (one query
// row per thread; warp w reads TMEM lanes 32 (w % 4) ..).  Per key tile j and
// head h:  S_h = Q_h K_j^T into TMEM; the warpgroup reads the score row into
// registers (one tensor-memory read of its 128 columns), takes its max, and writes P_h = exp(S_h - m) in bf16 back into
// the first 64 columns of S_h; O_h += P_h V_j reads P_h from TMEM.  The MMA
// thread issues head h's P V and right after it head h's next S (over the
// same columns: the tensor core runs one thread's MMAs in issue order), so
// while one warpgroup computes exponentials the tensor core works for the
// other head, and the commit of the next S also tells the warpgroup that
// O_h is stable.  For head width 128 a tile's exponentials (16 per clock per
// SM) take as long as its MMAs, so the two alternate rather than wait on
// each other.  The running max m of a row is raised (and O_h, l rescaled in
// place) only when the tile's max exceeds it by more than 2^8 in exp2 units;
// otherwise P is formed against the stale m (entries up to 2^8), which the
// final O / l and log-sum-exp m + log2(l) account for exactly.
// ----------------------------------------------------------------------------
namespace {

constexpr int FWD_THREADS = 352;
constexpr float RESCALE_LOG2 = 8.f;

struct FwdSmem {
    static constexpr int Q0 = 0;                // Q of head 0, then head 1 (32 KB each)
    static constexpr int K0 = 4 * BLK;          // K of key tile g in stage g % 2 (32 KB each)
    static constexpr int V0 = 8 * BLK;          // V of key tile g in stage g % 2 (32 KB each)
    static constexpr int BAR = 12 * BLK;
    enum { Q_FULL = 0, Q_EMPTY = 1, K_FULL = 2, K_EMPTY = 4, V_FULL = 6, V_EMPTY = 8, S_FULL = 10,
           P_FULL = 12, O_DONE = 14, O_FREE = 16, DRAIN = 18, SCHED_FULL = 19, SCHED_EMPTY = 19 + RING,
           NBARS = 19 + 2 * RING };
    static constexpr int MISC = BAR + NBARS * 8;     // TMEM base, abort flag, then the item ring
    static constexpr int TOTAL = MISC + 32 + 1024;
};

// One forward work item: query tile, key/value group, the two heads, and the
// key range [kstart, m0 + 128) in nt tiles.
struct FwdItem {
    int tile, g, h0, h1, m0, kstart, nt;
};

__device__ __forceinline__ FwdItem fwd_item(const AttnParams& p, int item) {
    FwdItem it;
    const int grp = p.n_heads / p.n_kv;
    const int pairs = (grp + 1) / 2;                    // head pairs per key/value group
    it.tile = item / (p.n_kv * pairs);
    const int rest = item % (p.n_kv * pairs);
    it.g = rest / pairs;
    it.h0 = it.g * grp + 2 * (rest % pairs);
    it.h1 = it.h0 + 1 < (it.g + 1) * grp ? it.h0 + 1 : it.h0;  // an odd group's last pair repeats its head
    it.m0 = it.tile * TB;
    it.kstart = p.seq_start[it.m0];
    it.nt = (it.m0 + TB - it.kstart + TB - 1) / TB;
    return it;
}

// O (+)= P V: M = 128 query rows, N = 128 head columns, K = 128 keys; A = P
// (bf16 pairs) in TMEM columns a_tmem .. a_tmem + 63, B = the row-major V tile
// read MN-major.
__device__ __forceinline__ void mma_pv_tmem(uint32_t d, uint32_t a_tmem, uint32_t v, bool acc) {
    const uint32_t id = idesc_bf16(128, 0, 1, 128);
    const uint64_t bd = mndesc(v);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            umma_bf16_ts(d, a_tmem + 32 * kb + 8 * kk, bd + 512 * kb + 128 * kk, id, (acc || kb || kk) ? 1u : 0u);
}

__global__ void __launch_bounds__(FWD_THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ AttnMaps maps, const AttnParams p, int n_items, int* status) {
    using SL = FwdSmem;
    const int mt_valid = *p.meta < p.max_tiles ? *p.meta : p.max_tiles;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sb + SL::BAR + 8 * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SL::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SL::MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* ring = reinterpret_cast<volatile int*>(smem + SL::MISC + 16);
    // items in order; the valid tiles are a prefix of the tile-major order
    const int pairs = (p.n_heads / p.n_kv + 1) / 2;
    auto valid = [&](int item) -> bool { return item >= 0 && item < n_items && item / (p.n_kv * pairs) < mt_valid; };
    if (blockIdx.x >= mt_valid * p.n_kv * pairs) return;   // more CTAs than items

    if (threadIdx.x == 0) {
        const int cnt[19] = {1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 4, 4, 1, 1, 4, 4, 1};
        for (int i = 0; i < 19; ++i) mbar_init(bar(i), cnt[i]);
        for (int i = 0; i < RING; ++i) {
            mbar_init(bar(SL::SCHED_FULL + i), 1);
            mbar_init(bar(SL::SCHED_EMPTY + i), 10);   // Q/V loader, MMA thread, eight softmax warps
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
        tma_prefetch_desc(&maps.rows128);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;   // S_h (and P_h over its first 64 columns) at 128 h, O_h at 256 + 128 h
    int dummy = 0;

    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            uint32_t gk = 0;                          // K tiles loaded by this CTA
            int last[2] = {-1, -1};
            RingPos rp;
            while (ok) {
                int item = atomicAdd(p.counter, 1);
                if (!valid(item)) item = -1;
                if (!ring_put(bar(SL::SCHED_FULL), bar(SL::SCHED_EMPTY), ring, rp, item, abort_flag)) {
                    ok = false;
                    break;
                }
                if (item < 0) break;
                const FwdItem it = fwd_item(p, item);
                const int kcol = (p.n_heads + it.g) * HD;
                for (int j = 0; j < it.nt; ++j, ++gk) {
                    const int ks = gk & 1;
                    const uint32_t kp = (gk >> 1) & 1u;
                    if (!mbar_wait(bar(SL::K_EMPTY + ks), kp ^ 1u, abort_flag)) { ok = false; break; }
                    mbar_expect_tx(bar(SL::K_FULL + ks), 2 * BLK);
                    load_tile128(sb + SL::K0 + ks * 2 * BLK, &maps.rows128, bar(SL::K_FULL + ks), kcol,
                                 it.kstart + j * TB);
                    last[ks] = (int)kp;
                }
            }
            for (int ks = 0; ks < 2; ++ks)      // our copies have landed
                if (last[ks] >= 0 && !mbar_wait(bar(SL::K_FULL + ks), (uint32_t)last[ks], (volatile int*)&dummy))
                    ok = false;
            if (!ok) { atomicOr(status, ST_TIMEOUT); *abort_flag = 1; }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = true;
            uint32_t gv = 0, nq = 0;                  // V tiles and Q tiles loaded
            int last[2] = {-1, -1};
            RingPos rp;
            while (ok) {
                int item;
                if (!ring_get(bar(SL::SCHED_FULL), bar(SL::SCHED_EMPTY), ring, rp, item, abort_flag)) {
                    ok = false;
                    break;
                }
                if (item < 0) break;
                const FwdItem it = fwd_item(p, item);
                const int vcol = (p.n_heads + p.n_kv + it.g) * HD;
                // the previous item's last scores have read Q
                if (nq > 0 && !mbar_wait(bar(SL::Q_EMPTY), (nq - 1) & 1u, abort_flag)) { ok = false; break; }
                mbar_expect_tx(bar(SL::Q_FULL), 4 * BLK);
                load_tile128(sb + SL::Q0, &maps.rows128, bar(SL::Q_FULL), it.h0 * HD, it.m0);
                load_tile128(sb + SL::Q0 + 2 * BLK, &maps.rows128, bar(SL::Q_FULL), it.h1 * HD, it.m0);
                ++nq;
                for (int j = 0; j < it.nt; ++j, ++gv) {
                    const int vs = gv & 1;
                    const uint32_t vp = (gv >> 1) & 1u;
                    if (!mbar_wait(bar(SL::V_EMPTY + vs), vp ^ 1u, abort_flag)) { ok = false; break; }
                    mbar_expect_tx(bar(SL::V_FULL + vs), 2 * BLK);
                    load_tile128(sb + SL::V0 + vs * 2 * BLK, &maps.rows128, bar(SL::V_FULL + vs), vcol,
                                 it.kstart + j * TB);
                    last[vs] = (int)vp;
                }
            }
            for (int vs = 0; vs < 2; ++vs)      // our copies have landed
                if (last[vs] >= 0 && !mbar_wait(bar(SL::V_FULL + vs), (uint32_t)last[vs], (volatile int*)&dummy))
                    ok = false;
            if (nq > 0 && !mbar_wait(bar(SL::Q_FULL), (nq - 1) & 1u, (volatile int*)&dummy)) ok = false;
            if (!ok) { atomicOr(status, ST_TIMEOUT); *abort_flag = 1; }
        }
    } else if (warp == 2) {
        if (lane == 0) {
            bool ok = true;
            uint32_t g0 = 0, nit = 0;                 // key tiles and items processed before this item
            RingPos rp;
            while (ok) {
                int item;
                if (!ring_get(bar(SL::SCHED_FULL), bar(SL::SCHED_EMPTY), ring, rp, item, abort_flag)) {
                    ok = false;
                    break;
                }
                if (item < 0) break;
                const int nt = fwd_item(p, item).nt;
                // the item's first scores.  S_h last held the previous item's last P_h,
                // whose P V was issued before (in order on the tensor core).
                ok = mbar_wait(bar(SL::Q_FULL), nit & 1u, abort_flag) &&
                     mbar_wait(bar(SL::K_FULL + (g0 & 1)), (g0 >> 1) & 1u, abort_flag);
                if (!ok) break;
                tc_fence_after();
                for (int hh = 0; hh < 2; ++hh) {
                    mma_kk(tmem + 128 * hh, sb + SL::Q0 + hh * 2 * BLK, sb + SL::K0 + (g0 & 1) * 2 * BLK, false);
                    umma_commit(bar(SL::S_FULL + hh));
                }
                umma_commit(bar(SL::K_EMPTY + (g0 & 1)));
                if (nt == 1) umma_commit(bar(SL::Q_EMPTY));
                for (int j = 0; j < nt && ok; ++j) {
                    const uint32_t g = g0 + j;
                    const uint32_t ph = g & 1u;
                    const int vs = g & 1, ks = (g + 1) & 1;
                    if (!mbar_wait(bar(SL::V_FULL + vs), (g >> 1) & 1u, abort_flag)) { ok = false; break; }
                    if (j + 1 < nt && !mbar_wait(bar(SL::K_FULL + ks), ((g + 1) >> 1) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    for (int hh = 0; hh < 2 && ok; ++hh) {
                        if (!mbar_wait(bar(SL::P_FULL + hh), ph, abort_flag)) { ok = false; break; }
                        // O_h of the previous item has been read out
                        if (j == 0 && nit > 0 && !mbar_wait(bar(SL::O_FREE + hh), (nit - 1) & 1u, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        mma_pv_tmem(tmem + 256 + 128 * hh, tmem + 128 * hh, sb + SL::V0 + vs * 2 * BLK, j > 0);
                        if (j + 1 == nt) umma_commit(bar(SL::O_DONE + hh));
                        if (j + 1 < nt) {
                            // next scores over S_h / P_h: after this P V in issue order
                            mma_kk(tmem + 128 * hh, sb + SL::Q0 + hh * 2 * BLK, sb + SL::K0 + ks * 2 * BLK, false);
                            umma_commit(bar(SL::S_FULL + hh));
                        }
                    }
                    if (!ok) break;
                    umma_commit(bar(SL::V_EMPTY + vs));
                    if (j + 1 < nt) {
                        umma_commit(bar(SL::K_EMPTY + ks));
                        if (j + 2 == nt) umma_commit(bar(SL::Q_EMPTY));   // the item's last scores
                    }
                }
                g0 += nt;
                ++nit;
            }
            if (!ok) { atomicOr(status, ST_TIMEOUT); *abort_flag = 1; }
            umma_commit(bar(SL::DRAIN));
            if (!mbar_wait(bar(SL::DRAIN), 0, (volatile int*)&dummy)) atomicOr(status, ST_TIMEOUT);
        }
    } else {
        const int hh = (warp - 3) >> 2;                 // head slot of this warpgroup
        const int q4 = warp & 3;
        const int r = 32 * q4 + lane;
        const uint32_t tS = tmem + ((uint32_t)(32 * q4) << 16) + 128 * hh;
        const uint32_t tO = tS + 256;
        const float sc = p.scale * LOG2E;
        bool ok = true;
        uint32_t rr[32];
        uint32_t g0 = 0, nit = 0;                       // key tiles and items processed before this item
        RingPos rp;
        while (ok) {
            int item;
            if (!ring_get_warp(bar(SL::SCHED_FULL), bar(SL::SCHED_EMPTY), ring, rp, item, abort_flag, lane)) {
                ok = false;
                break;
            }
            if (item < 0) break;
            const FwdItem it = fwd_item(p, item);
            const int h = hh ? it.h1 : it.h0;
            const int i = it.m0 + r;
            const int ss = p.seq_start[i];
            const int nt = it.nt;
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < nt; ++j) {
                const uint32_t ph = (g0 + j) & 1u;
                // S_h of this tile; its commit also covers head h's previous P V, so
                // O_h is stable and the P_h columns are free
                if (!warp_wait(bar(SL::S_FULL + hh), ph, abort_flag, lane)) { ok = false; break; }
                tc_fence_after();
                const int key0 = it.kstart + j * TB;
                // valid key columns of this row: [lo, hi]; a warp whose rows all see
                // the whole tile takes the unmasked copy of the loops
                const int lo = ss - key0, hi = i - key0;
                const bool whole = __all_sync(0xffffffffu, lo <= 0 && hi >= TB - 1);
                // the score row, read from TMEM once into registers
                uint32_t s0[32], s1[32], s2[32], s3[32];
                tmem_ld32(tS, s0);
                tmem_ld32(tS + 32, s1);
                tmem_ld32(tS + 64, s2);
                tmem_ld32(tS + 96, s3);
                tmem_ld_wait_regs(s0);
                tmem_ld_wait_regs(s1);
                tmem_ld_wait_regs(s2);
                tmem_ld_wait_regs(s3);
                float mx = -INFINITY, alpha = 1.f, rs = 0.f;
                bool raise = false;
                // the row max of the raw scores (the scale is positive, so scaling the
                // max equals the max of the scaled scores)
                auto chunk_max = [&](const uint32_t (&cur)[32], int c, auto masked) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int idx = 32 * c + e;
                        const bool v = !decltype(masked)::value || ((idx >= lo) & (idx <= hi));
                        mx = fmaxf(mx, v ? __uint_as_float(cur[e]) : -INFINITY);
                    }
                };
                // P = exp2(scale s - m) in bf16, written over the first 64 columns of
                // S_h (bf16 pairs): the whole row is already in registers
                auto chunk_p = [&](const uint32_t (&cur)[32], int c, auto masked) {
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const int idx = 32 * c + e;
                        const bool v0 = !decltype(masked)::value || ((idx >= lo) & (idx <= hi));
                        const bool v1 = !decltype(masked)::value || ((idx + 1 >= lo) & (idx + 1 <= hi));
                        // masked entries give exp2(-inf) = 0: no branch around the exponential
                        const float p0 = ex2_ftz(v0 ? fmaf(__uint_as_float(cur[e]), sc, -m_run) : -INFINITY);
                        const float p1 = ex2_ftz(v1 ? fmaf(__uint_as_float(cur[e + 1]), sc, -m_run) : -INFINITY);
                        rs += p0 + p1;
                        w[e >> 1] = pack_bf16x2(p0, p1);
                    }
                    tmem_st16(tS + 16 * c, w);     // keys 32 c .. 32 c + 31
                };
                auto row = [&](auto masked) {
                    chunk_max(s0, 0, masked);
                    chunk_max(s1, 1, masked);
                    chunk_max(s2, 2, masked);
                    chunk_max(s3, 3, masked);
                    mx *= sc;
                    raise = mx > m_run + RESCALE_LOG2;
                    alpha = raise ? ex2_ftz(m_run - mx) : 1.f;
                    if (raise) m_run = mx;
                    chunk_p(s0, 0, masked);
                    chunk_p(s1, 1, masked);
                    chunk_p(s2, 2, masked);
                    chunk_p(s3, 3, masked);
                };
                if (whole) row(std::false_type{});
                else row(std::true_type{});
                // a raised max rescales O_h before this tile's P V accumulates into it
                if (j > 0 && __any_sync(0xffffffffu, raise)) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        tmem_ld32(tO + 32 * c, rr);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
                        tmem_st32(tO + 32 * c, rr);
                    }
                }
                tmem_st_wait();
                l_run = l_run * alpha + rs;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(SL::P_FULL + hh));
            }
            if (ok) ok = warp_wait(bar(SL::O_DONE + hh), nit & 1u, abort_flag, lane);
            if (!ok) break;
            tc_fence_after();
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            bf16* dst = p.o + (int64_t)i * p.n_heads * HD + h * HD;
            const bool store = hh == 0 || it.h1 != it.h0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                tmem_ld32(tO + 32 * c, rr);
                tmem_ld_wait();
                float t[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) t[e] = __uint_as_float(rr[e]) * inv;
                if (store) store32<bf16>(dst + 32 * c, t);
            }
            if (store) p.lseT[(int64_t)h * p.ld_t + i] = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
            // O_h has been read: the next item's first P V may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(SL::O_FREE + hh));
            g0 += nt;
            ++nit;
        }
        if (!ok && lane == 0) {
            atomicOr(status, ST_TIMEOUT);
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tmem, 512);
}

}  // namespace

// ----------------------------------------------------------------------------
// Backward, key side.  Work item = (128-row key tile, key/value head g).  For every
// query head of the group and every query tile that can see these keys, in
// two halves of 64 query rows:
//   S^T = K Q^T, dP^T = V dO^T                   (TMEM, two buffers)
//   P^T = exp(scale S^T - lse_q), dS^T = P^T (dP^T - D_q)   (softmax warps,
//        one key row per thread; bf16, written back into TMEM over the
//        S^T / dP^T columns just read)
//   dV += P^T dO,  dK += dS^T Q                   (A operand read from TMEM)
// and finally dK *= scale.  The MMA warp issues the next half's S^T and dP^T
// before it waits for this half's P^T, so the tensor core works while the
// softmax warps do.  Query-side tiles (Q, dO, their log-sum-exp, rowsum and
// sequence starts) are double-buffered.  Each dK / dV element has one writer.
// ----------------------------------------------------------------------------
namespace {

struct KvSmem {
    static constexpr int K = 0;
    static constexpr int V = 2 * BLK;
    static constexpr int Q0 = 4 * BLK;           // stage s: Q at Q0 + 4 BLK s, dO 2 BLK after
    static constexpr int VEC0 = 12 * BLK;        // stage s: lse[128] (log2 units), D[128], seq_start[128]
    static constexpr int BAR = VEC0 + 2 * 3 * 512;
    // (slots 9-10 are spare)
    enum { KV_FULL = 0, QD_FULL = 1, QD_EMPTY = 3, ST_FULL = 5, P_FULL = 7, SPARE = 9, ACC_FULL = 11,
           DRAIN = 12, KV_EMPTY = 13, ACC_FREE = 14, SCHED_FULL = 15, SCHED_EMPTY = 15 + RING,
           NBARS = 15 + 2 * RING };
    static constexpr int MISC = BAR + NBARS * 8;     // TMEM base, abort flag, then the item ring
    static constexpr int TOTAL = MISC + 32 + 1024;
};

// D = A B^T, M = 128, N = 64, K = 128: A a K-major 128-row tile, B 64 rows
// (half `s` of a K-major 128-row tile).
__device__ __forceinline__ void mma_kk64(uint32_t d, uint32_t a, uint32_t b, int s) {
    const uint32_t id = idesc_bf16(64, 0, 0, 128);
    const uint64_t ad = kdesc(a), bd = kdesc(b + 8192 * s);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            umma_bf16(d, ad + kb * BLK_STEP + 2 * kk, bd + kb * BLK_STEP + 2 * kk, id, (kb || kk) ? 1u : 0u);
}
// Key-side work item: key tile kt of key/value head g; the query tiles
// kt .. kt + nqt - 1 are those whose first row starts its sequence at or
// before this tile's last key, taken for every query head of the group.
struct KvItem {
    int kt, g, k0, nqt, niter;
};

__device__ __forceinline__ KvItem kv_item(const AttnParams& p, int item, int mt_valid) {
    KvItem it;
    it.kt = item / p.n_kv;
    it.g = item % p.n_kv;
    it.k0 = it.kt * TB;
    int nqt = 0;
    while (it.kt + nqt < mt_valid && p.seq_start[(it.kt + nqt) * TB] <= it.k0 + TB - 1) ++nqt;
    it.nqt = nqt;
    it.niter = (p.n_heads / p.n_kv) * nqt;
    return it;
}

// Persistent: one CTA per SM takes items (key tile * n_kv + head) from the
// global counter, keeping TMEM and barriers; barrier
// phases follow running counts of query tiles and halves.  The next item's
// K / V load starts once the current item's last scores are issued, and its
// first products overlap the read-out of the current dK / dV.
// D (+)= A B^T, M = 128, N = 128, K = 64: B rows 64 s .. 64 s + 63 of a
// row-major smem tile read MN-major; A (bf16 pairs) in TMEM in two 16-column
// pieces: K rows 0-31 (bf16 pairs) at
// a_tmem .. a_tmem + 15 and K rows 32-63 at a_tmem + 32 .. a_tmem + 47, as the
// two softmax warpgroups write them (each over the columns it has read).
__device__ __forceinline__ void mma_t64mn_split(uint32_t d, uint32_t a_tmem, uint32_t b, int s, bool acc) {
    const uint32_t id = idesc_bf16(128, 0, 1, 128);
    const uint64_t bd = mndesc(b) + 512 * s;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        umma_bf16_ts(d, a_tmem + 8 * kk + (kk >= 2 ? 16 : 0), bd + 128 * kk, id, (acc || kk) ? 1u : 0u);
}

// Backward kernels: warp 0 loads, warp 1 issues the MMAs, warps 2-9 are two
// softmax warpgroups over the same TMEM lanes (warp w reads lanes
// 32 (w % 4) ..); warpgroup c takes columns 32 c .. 32 c + 31 of each half.
constexpr int BWD_THREADS = 320;

__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_kv_kernel(const __grid_constant__ AttnMaps maps, const AttnParams p, int n_items, int* status) {
    using SL = KvSmem;
    const int mt_valid = *p.meta < p.max_tiles ? *p.meta : p.max_tiles;
    auto valid = [&](int item) -> bool { return item >= 0 && item < n_items && item / p.n_kv < mt_valid; };
    if (blockIdx.x >= mt_valid * p.n_kv) return;   // more CTAs than items
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sb + SL::BAR + 8 * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SL::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SL::MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = p.n_heads / p.n_kv;

    volatile int* ring = reinterpret_cast<volatile int*>(smem + SL::MISC + 16);
    if (threadIdx.x == 0) {
        const int cnt[15] = {1, 1, 1, 1, 1, 1, 1, 8, 8, 1, 1, 1, 1, 1, 8};
        for (int i = 0; i < 15; ++i) mbar_init(bar(i), cnt[i]);
        for (int i = 0; i < RING; ++i) {
            mbar_init(bar(SL::SCHED_FULL + i), 1);
            mbar_init(bar(SL::SCHED_EMPTY + i), 9);    // MMA thread, eight softmax warps
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
        tma_prefetch_desc(&maps.rows128);
        tma_prefetch_desc(&maps.do128);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // buffer b: S^T / P^T at columns 64 b, dP^T / dS^T at 128 + 64 b; dV 256, dK 384
    const uint32_t tmem = *tmem_slot;
    int dummy = 0;

    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            int last[2] = {-1, -1};
            uint32_t nkv = 0, gn = 0;                  // K / V tiles and query tiles loaded
            RingPos rp;
            while (ok) {
                int item = atomicAdd(p.counter, 1);
                if (!valid(item)) item = -1;
                if (!ring_put(bar(SL::SCHED_FULL), bar(SL::SCHED_EMPTY), ring, rp, item, abort_flag)) {
                    ok = false;
                    break;
                }
                if (item < 0) break;
                const KvItem it = kv_item(p, item, mt_valid);
                const int kcol = (p.n_heads + it.g) * HD, vcol = (p.n_heads + p.n_kv + it.g) * HD;
                // the previous item's last scores have read K and V
                if (nkv > 0 && !mbar_wait(bar(SL::KV_EMPTY), (nkv - 1) & 1u, abort_flag)) { ok = false; break; }
                mbar_expect_tx(bar(SL::KV_FULL), 4 * BLK);
                load_tile128(sb + SL::K, &maps.rows128, bar(SL::KV_FULL), kcol, it.k0);
                load_tile128(sb + SL::V, &maps.rows128, bar(SL::KV_FULL), vcol, it.k0);
                ++nkv;
                for (int n = 0; n < it.niter; ++n, ++gn) {
                    const int s = gn & 1;
                    const uint32_t sp = (gn >> 1) & 1u;
                    const int h = it.g * grp + n / it.nqt, q0 = (it.kt + n % it.nqt) * TB;
                    if (!mbar_wait(bar(SL::QD_EMPTY + s), sp ^ 1u, abort_flag)) { ok = false; break; }
                    const uint32_t fb = bar(SL::QD_FULL + s);
                    const uint32_t st = sb + SL::Q0 + s * 4 * BLK, vec = sb + SL::VEC0 + s * 1536;
                    mbar_expect_tx(fb, 4 * BLK + 3 * 512);
                    load_tile128(st, &maps.rows128, fb, h * HD, q0);
                    load_tile128(st + 2 * BLK, &maps.do128, fb, h * HD, q0);
                    bulk_load(vec, p.lseT + (int64_t)h * p.ld_t + q0, 512, fb);
                    bulk_load(vec + 512, p.DT + (int64_t)h * p.ld_t + q0, 512, fb);
                    bulk_load(vec + 1024, p.seq_start + q0, 512, fb);
                    last[s] = (int)sp;
                }
            }
            if (!ok) { atomicOr(status, ST_TIMEOUT); *abort_flag = 1; }
            bool dr = nkv == 0 || mbar_wait(bar(SL::KV_FULL), (nkv - 1) & 1u, (volatile int*)&dummy);
            for (int s = 0; s < 2; ++s)
                if (last[s] >= 0) dr &= mbar_wait(bar(SL::QD_FULL + s), (uint32_t)last[s], (volatile int*)&dummy);
            if (!dr) atomicOr(status, ST_TIMEOUT);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = true;
            uint32_t gm = 0, gn0 = 0, nit = 0;        // halves, query tiles and items before this item
            RingPos rp;
            while (ok) {
                int item;
                if (!ring_get(bar(SL::SCHED_FULL), bar(SL::SCHED_EMPTY), ring, rp, item, abort_flag)) {
                    ok = false;
                    break;
                }
                if (item < 0) break;
                const KvItem it = kv_item(p, item, mt_valid);
                const int nhalf = 2 * it.niter;        // >= 2: the key tile's own query tile
                // half m: query tile gn0 + m / 2 in stage (gn0 + m / 2) & 1, rows 64 (m & 1) ..,
                // TMEM buffer m & 1 (gm is even)
                auto issue_s = [&](int m) -> bool {
                    const uint32_t N = gn0 + (m >> 1);
                    const int b = m & 1;
                    const uint32_t st = sb + SL::Q0 + (N & 1) * 4 * BLK;
                    if (b == 0 && !mbar_wait(bar(SL::QD_FULL + (N & 1)), (N >> 1) & 1u, abort_flag)) return false;
                    // buffer b last held half m - 2's P^T / dS^T, read by its dV / dK
                    // products, which this thread issued before: the tensor core runs
                    // one thread's MMAs in issue order, so no wait is needed here
                    tc_fence_after();
                    mma_kk64(tmem + 64 * b, sb + SL::K, st, b);
                    mma_kk64(tmem + 128 + 64 * b, sb + SL::V, st + 2 * BLK, b);
                    umma_commit(bar(SL::ST_FULL + b));
                    return true;
                };
                ok = mbar_wait(bar(SL::KV_FULL), nit & 1u, abort_flag) && issue_s(0);
                for (int m = 0; m < nhalf && ok; ++m) {
                    const uint32_t M = gm + m, N = gn0 + (m >> 1);
                    const int b = m & 1;
                    const uint32_t st = sb + SL::Q0 + (N & 1) * 4 * BLK;
                    if (m + 1 < nhalf) {
                        if (!issue_s(m + 1)) { ok = false; break; }
                        if (m + 2 == nhalf) umma_commit(bar(SL::KV_EMPTY));   // the item's last scores
                    }
                    if (!mbar_wait(bar(SL::P_FULL + b), (M >> 1) & 1u, abort_flag)) { ok = false; break; }
                    // dV / dK of the previous item have been read out
                    if (m == 0 && nit > 0 && !mbar_wait(bar(SL::ACC_FREE), (nit - 1) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    mma_t64mn_split(tmem + 256, tmem + 64 * b, st + 2 * BLK, b, m > 0);
                    mma_t64mn_split(tmem + 384, tmem + 128 + 64 * b, st, b, m > 0);
                    if (b == 1) umma_commit(bar(SL::QD_EMPTY + (N & 1)));
                }
                if (!ok) break;
                umma_commit(bar(SL::ACC_FULL));
                gm += nhalf;
                gn0 += it.niter;
                ++nit;
            }
            if (!ok) { atomicOr(status, ST_TIMEOUT); *abort_flag = 1; }
            umma_commit(bar(SL::DRAIN));
            if (!mbar_wait(bar(SL::DRAIN), 0, (volatile int*)&dummy)) atomicOr(status, ST_TIMEOUT);
        }
    } else {
        const int q4 = warp & 3;
        const int wg = (warp - 2) >> 2;                // column half of each 64-column half
        const int r = 32 * q4 + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
        const float sc = p.scale * LOG2E;
        bool ok = true;
        uint32_t ra[32], rb[32];
        uint32_t gm = 0, gn0 = 0, nit = 0;
        RingPos rp;
        while (ok) {
            int item;
            if (!ring_get_warp(bar(SL::SCHED_FULL), bar(SL::SCHED_EMPTY), ring, rp, item, abort_flag, lane)) {
                ok = false;
                break;
            }
            if (item < 0) break;
            const KvItem it = kv_item(p, item, mt_valid);
            const int j = it.k0 + r;                       // this thread's key row
            const int kcol = (p.n_heads + it.g) * HD, vcol = (p.n_heads + p.n_kv + it.g) * HD;
            const int nhalf = 2 * it.niter;
            int qmin = 0, qmax = -1;
            for (int m = 0; m < nhalf; ++m) {
                const int n = m >> 1, b = m & 1;
                const uint32_t M = gm + m, N = gn0 + n;
                const int s = N & 1;
                const int q0 = (it.kt + n % it.nqt) * TB;
                // stored mode: this thread's 32 dS values of the half, row r of block
                // (query tile, key tile, head), columns 64 b + 32 wg ..
                bf16* dsp = nullptr;
                if (p.ds) {
                    const int qt = it.kt + n % it.nqt, hq = it.g * grp + n / it.nqt;
                    if (qt - it.kt < p.ktc)
                        dsp = p.ds + (((int64_t)qt * p.ktc + (qt - it.kt)) * p.n_heads + hq) * (TB * TB) +
                              (int64_t)r * TB + 64 * b + 32 * wg;
                    else if (lane == 0)
                        raise_status(status, ST_RANGE);
                }
                const float* lse_s = reinterpret_cast<const float*>(smem + SL::VEC0 + s * 1536);
                const float* D_s = lse_s + 128;
                const int* ss_s = reinterpret_cast<const int*>(lse_s + 256);
                if (b == 0) {
                    if (!warp_wait(bar(SL::QD_FULL + s), (N >> 1) & 1u, abort_flag, lane)) { ok = false; break; }
                    // valid query columns of this key row: [qmin, qmax] -- queries at or
                    // after it whose sequence starts at or before it (sequence starts do
                    // not decrease along the tile, so the second condition is a prefix)
                    qmin = j - q0;
                    qmax = -1;
                    if (ss_s[0] <= j) {
                        int a = 0, c = TB - 1;
                        while (a < c) {
                            const int mid = (a + c + 1) >> 1;
                            if (ss_s[mid] <= j) a = mid; else c = mid - 1;
                        }
                        qmax = a;
                    }
                }
                if (!warp_wait(bar(SL::ST_FULL + b), (M >> 1) & 1u, abort_flag, lane)) { ok = false; break; }
                tc_fence_after();
                // this warpgroup's 32 query columns of the half
                const int lo = qmin - 64 * b - 32 * wg, hi = qmax - 64 * b - 32 * wg;
                const bool whole = __all_sync(0xffffffffu, lo <= 0 && hi >= 31);
                auto write_pd = [&](auto masked) {
                    const uint32_t cs = tl + 64 * b + 32 * wg, cd = tl + 128 + 64 * b + 32 * wg;
                    tmem_ld32(cs, ra);
                    tmem_ld32(cd, rb);
                    tmem_ld_wait_regs(ra);
                    tmem_ld_wait_regs(rb);
                    uint32_t wp[16], wd[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        // the query columns' lse and D, four at a time (same address in every lane)
                        const float4 l4 = *reinterpret_cast<const float4*>(lse_s + 64 * b + 32 * wg + e);
                        const float4 d4 = *reinterpret_cast<const float4*>(D_s + 64 * b + 32 * wg + e);
                        const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv[4] = {d4.x, d4.y, d4.z, d4.w};
                        float pr[4], ds[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int qc = e + u;
                            const bool valid_q = !decltype(masked)::value || ((qc >= lo) & (qc <= hi));
                            pr[u] = ex2_ftz(valid_q ? fmaf(__uint_as_float(ra[e + u]), sc, -lv[u]) : -INFINITY);
                            ds[u] = pr[u] * (__uint_as_float(rb[e + u]) - dv[u]);
                        }
                        wp[e >> 1] = pack_bf16x2(pr[0], pr[1]);
                        wp[(e >> 1) + 1] = pack_bf16x2(pr[2], pr[3]);
                        wd[e >> 1] = pack_bf16x2(ds[0], ds[1]);
                        wd[(e >> 1) + 1] = pack_bf16x2(ds[2], ds[3]);
                    }
                    tmem_st16(cs, wp);           // over this warpgroup's columns, already read
                    tmem_st16(cd, wd);
                    if (dsp) {
                        uint4* d4 = reinterpret_cast<uint4*>(dsp);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            d4[u] = make_uint4(wd[4 * u], wd[4 * u + 1], wd[4 * u + 2], wd[4 * u + 3]);
                    }
                };
                if (whole) write_pd(std::false_type{});
                else write_pd(std::true_type{});
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(SL::P_FULL + b));
            }
            if (ok) ok = warp_wait(bar(SL::ACC_FULL), nit & 1u, abort_flag, lane);
            if (!ok) break;
            tc_fence_after();
            bf16* row = p.dqkv + (int64_t)j * p.ld_qkv;
            float v[32];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {           // this warpgroup's 64 of the 128 columns
                const int c = 2 * wg + cc;
                tmem_ld32(tl + 256 + 32 * c, ra);
                tmem_ld32(tl + 384 + 32 * c, rb);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(ra[e]);
                store32<bf16>(row + vcol + 32 * c, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(rb[e]) * p.scale;
                store32<bf16>(row + kcol + 32 * c, v);
            }
            // dV / dK have been read: the next item's first products may overwrite them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(SL::ACC_FREE));
            gm += nhalf;
            gn0 += it.niter;
            ++nit;
        }
        if (!ok && lane == 0) {
            atomicOr(status, ST_TIMEOUT);
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

// ----------------------------------------------------------------------------
// Backward, query side.  Work item = (128-row query tile, query head).  Over the
// forward's key tiles, in halves of 64 keys:  S = Q K^T, dP = dO V^T (TMEM,
// two buffers);  P = exp(scale S - lse), dS = P (dP - D) (softmax warps, one
// query row per thread, bf16 written back into TMEM over the S columns just
// read);  dQ += dS K (A operand from TMEM);  finally dQ *= scale.  The MMA
// warp issues the next half's S and dP before it waits for this half's dS.
// ----------------------------------------------------------------------------
namespace {

struct QSmem {
    static constexpr int Q = 0;
    static constexpr int DO = 2 * BLK;
    static constexpr int K0 = 4 * BLK;          // stage s: K at K0 + 4 BLK s, V 2 BLK after
    static constexpr int BAR = 12 * BLK;
    // (slots 9-10 are spare)
    enum { Q_FULL = 0, KV_FULL = 1, KV_EMPTY = 3, S_FULL = 5, DS_FULL = 7, SPARE = 9, ACC_FULL = 11,
           DRAIN = 12, Q_EMPTY = 13, ACC_FREE = 14, SCHED_FULL = 15, SCHED_EMPTY = 15 + RING,
           NBARS = 15 + 2 * RING };
    static constexpr int MISC = BAR + NBARS * 8;     // TMEM base, abort flag, then the item ring
    static constexpr int TOTAL = MISC + 32 + 1024;
};

// Query-side work item: query tile `tile` of query head h, over the
// forward's key tiles [kstart, m0 + 128).
struct QItem {
    int tile, h, m0, kstart, nt;
};

__device__ __forceinline__ QItem q_item(const AttnParams& p, int item) {
    QItem it;
    it.tile = item / p.n_heads;
    it.h = item % p.n_heads;
    it.m0 = it.tile * TB;
    it.kstart = p.seq_start[it.m0];
    it.nt = (it.m0 + TB - it.kstart + TB - 1) / TB;
    return it;
}

// Persistent like the key side: items query tile * n_heads + head; the next
// item's Q / dO load starts once the current item's last scores are issued.
__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_q_kernel(const __grid_constant__ AttnMaps maps, const AttnParams p, int n_items, int* status) {
    using SL = QSmem;
    const int mt_valid = *p.meta < p.max_tiles ? *p.meta : p.max_tiles;
    auto valid = [&](int item) -> bool { return item >= 0 && item < n_items && item / p.n_heads < mt_valid; };
    if (blockIdx.x >= mt_valid * p.n_heads) return;   // more CTAs than items
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sb + SL::BAR + 8 * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SL::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SL::MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = p.n_heads / p.n_kv;

    volatile int* ring = reinterpret_cast<volatile int*>(smem + SL::MISC + 16);
    if (threadIdx.x == 0) {
        const int cnt[15] = {1, 1, 1, 1, 1, 1, 1, 8, 8, 1, 1, 1, 1, 1, 8};
        for (int i = 0; i < 15; ++i) mbar_init(bar(i), cnt[i]);
        for (int i = 0; i < RING; ++i) {
            mbar_init(bar(SL::SCHED_FULL + i), 1);
            mbar_init(bar(SL::SCHED_EMPTY + i), 9);    // MMA thread, eight softmax warps
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
        tma_prefetch_desc(&maps.rows128);
        tma_prefetch_desc(&maps.do128);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;   // buffer b: S / dS at 64 b, dP at 128 + 64 b; dQ at 256
    int dummy = 0;

    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            int last[2] = {-1, -1};
            uint32_t nq = 0, gj = 0;                   // Q / dO tiles and key tiles loaded
            RingPos rp;
            while (ok) {
                int item = atomicAdd(p.counter, 1);
                if (!valid(item)) item = -1;
                if (!ring_put(bar(SL::SCHED_FULL), bar(SL::SCHED_EMPTY), ring, rp, item, abort_flag)) {
                    ok = false;
                    break;
                }
                if (item < 0) break;
                const QItem it = q_item(p, item);
                const int g = it.h / grp;
                const int qcol = it.h * HD, kcol = (p.n_heads + g) * HD, vcol = (p.n_heads + p.n_kv + g) * HD;
                // the previous item's last scores have read Q and dO
                if (nq > 0 && !mbar_wait(bar(SL::Q_EMPTY), (nq - 1) & 1u, abort_flag)) { ok = false; break; }
                mbar_expect_tx(bar(SL::Q_FULL), 4 * BLK);
                load_tile128(sb + SL::Q, &maps.rows128, bar(SL::Q_FULL), qcol, it.m0);
                load_tile128(sb + SL::DO, &maps.do128, bar(SL::Q_FULL), qcol, it.m0);
                ++nq;
                for (int j = 0; j < it.nt; ++j, ++gj) {
                    const int s = gj & 1;
                    const uint32_t sp = (gj >> 1) & 1u;
                    if (!mbar_wait(bar(SL::KV_EMPTY + s), sp ^ 1u, abort_flag)) { ok = false; break; }
                    const int key0 = it.kstart + j * TB;
                    const uint32_t fb = bar(SL::KV_FULL + s), st = sb + SL::K0 + s * 4 * BLK;
                    mbar_expect_tx(fb, 4 * BLK);
                    load_tile128(st, &maps.rows128, fb, kcol, key0);
                    load_tile128(st + 2 * BLK, &maps.rows128, fb, vcol, key0);
                    last[s] = (int)sp;
                }
            }
            if (!ok) { atomicOr(status, ST_TIMEOUT); *abort_flag = 1; }
            bool dr = nq == 0 || mbar_wait(bar(SL::Q_FULL), (nq - 1) & 1u, (volatile int*)&dummy);
            for (int s = 0; s < 2; ++s)
                if (last[s] >= 0) dr &= mbar_wait(bar(SL::KV_FULL + s), (uint32_t)last[s], (volatile int*)&dummy);
            if (!dr) atomicOr(status, ST_TIMEOUT);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = true;
            uint32_t gm = 0, gj0 = 0, nit = 0;         // halves, key tiles and items before this item
            RingPos rp;
            while (ok) {
                int item;
                if (!ring_get(bar(SL::SCHED_FULL), bar(SL::SCHED_EMPTY), ring, rp, item, abort_flag)) {
                    ok = false;
                    break;
                }
                if (item < 0) break;
                const int nhalf = 2 * q_item(p, item).nt;   // >= 2
                // half m: key tile gj0 + m / 2 in stage (gj0 + m / 2) & 1, keys 64 (m & 1) ..,
                // TMEM buffer m & 1 (gm is even)
                auto issue_s = [&](int m) -> bool {
                    const uint32_t J = gj0 + (m >> 1);
                    const int b = m & 1;
                    const uint32_t st = sb + SL::K0 + (J & 1) * 4 * BLK;
                    if (b == 0 && !mbar_wait(bar(SL::KV_FULL + (J & 1)), (J >> 1) & 1u, abort_flag)) return false;
                    // buffer b last held half m - 2's dS, read by its dQ product, issued
                    // before by this thread: in-order on the tensor core, no wait
                    tc_fence_after();
                    mma_kk64(tmem + 64 * b, sb + SL::Q, st, b);
                    mma_kk64(tmem + 128 + 64 * b, sb + SL::DO, st + 2 * BLK, b);
                    umma_commit(bar(SL::S_FULL + b));
                    return true;
                };
                ok = mbar_wait(bar(SL::Q_FULL), nit & 1u, abort_flag) && issue_s(0);
                for (int m = 0; m < nhalf && ok; ++m) {
                    const uint32_t M = gm + m, J = gj0 + (m >> 1);
                    const int b = m & 1;
                    const uint32_t st = sb + SL::K0 + (J & 1) * 4 * BLK;
                    if (m + 1 < nhalf) {
                        if (!issue_s(m + 1)) { ok = false; break; }
                        if (m + 2 == nhalf) umma_commit(bar(SL::Q_EMPTY));   // the item's last scores
                    }
                    if (!mbar_wait(bar(SL::DS_FULL + b), (M >> 1) & 1u, abort_flag)) { ok = false; break; }
                    // dQ of the previous item has been read out
                    if (m == 0 && nit > 0 && !mbar_wait(bar(SL::ACC_FREE), (nit - 1) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    mma_t64mn_split(tmem + 256, tmem + 64 * b, st, b, m > 0);
                    if (b == 1) umma_commit(bar(SL::KV_EMPTY + (J & 1)));
                }
                if (!ok) break;
                umma_commit(bar(SL::ACC_FULL));
                gm += nhalf;
                gj0 += nhalf >> 1;
                ++nit;
            }
            if (!ok) { atomicOr(status, ST_TIMEOUT); *abort_flag = 1; }
            umma_commit(bar(SL::DRAIN));
            if (!mbar_wait(bar(SL::DRAIN), 0, (volatile int*)&dummy)) atomicOr(status, ST_TIMEOUT);
        }
    } else {
        const int q4 = warp & 3;
        const int wg = (warp - 2) >> 2;                // column half of each 64-column half
        const int r = 32 * q4 + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
        const float sc = p.scale * LOG2E;
        bool ok = true;
        uint32_t ra[32], rb[32];
        uint32_t gm = 0, nit = 0;
        RingPos rp;
        while (ok) {
            int item;
            if (!ring_get_warp(bar(SL::SCHED_FULL), bar(SL::SCHED_EMPTY), ring, rp, item, abort_flag, lane)) {
                ok = false;
                break;
            }
            if (item < 0) break;
            const QItem it = q_item(p, item);
            const int i = it.m0 + r;
            const int ss = p.seq_start[i];
            const float lse2 = p.lseT[(int64_t)it.h * p.ld_t + i];
            const float Di = p.DT[(int64_t)it.h * p.ld_t + i];
            const int nhalf = 2 * it.nt;
            for (int m = 0; m < nhalf; ++m) {
                const int b = m & 1;
                const uint32_t M = gm + m;
                if (!warp_wait(bar(SL::S_FULL + b), (M >> 1) & 1u, abort_flag, lane)) { ok = false; break; }
                tc_fence_after();
                // this warpgroup's 32 key columns of the half: valid keys [lo, hi]
                const int key0 = it.kstart + (m >> 1) * TB + 64 * b + 32 * wg;
                const int lo = ss - key0, hi = i - key0;
                const bool whole = __all_sync(0xffffffffu, lo <= 0 && hi >= 31);
                auto write_ds = [&](auto masked) {
                    const uint32_t cs = tl + 64 * b + 32 * wg;
                    tmem_ld32(cs, ra);
                    tmem_ld32(tl + 128 + 64 * b + 32 * wg, rb);
                    tmem_ld_wait_regs(ra);
                    tmem_ld_wait_regs(rb);
                    uint32_t wd[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float ds[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int idx = e + u;
                            const bool v = !decltype(masked)::value || ((idx >= lo) & (idx <= hi));
                            const float pr = ex2_ftz(v ? fmaf(__uint_as_float(ra[e + u]), sc, -lse2) : -INFINITY);
                            ds[u] = pr * (__uint_as_float(rb[e + u]) - Di);
                        }
                        wd[e >> 1] = pack_bf16x2(ds[0], ds[1]);
                    }
                    tmem_st16(cs, wd);           // over this warpgroup's columns, already read
                };
                if (whole) write_ds(std::false_type{});
                else write_ds(std::true_type{});
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(SL::DS_FULL + b));
            }
            if (ok) ok = warp_wait(bar(SL::ACC_FULL), nit & 1u, abort_flag, lane);
            if (!ok) break;
            tc_fence_after();
            bf16* row = p.dqkv + (int64_t)i * p.ld_qkv + it.h * HD;
            float v[32];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {           // this warpgroup's 64 of the 128 columns
                const int c = 2 * wg + cc;
                tmem_ld32(tl + 256 + 32 * c, ra);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(ra[e]) * p.scale;
                store32<bf16>(row + 32 * c, v);
            }
            // dQ has been read: the next item's first products may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(SL::ACC_FREE));
            gm += nhalf;
            ++nit;
        }
        if (!ok && lane == 0) {
            atomicOr(status, ST_TIMEOUT);
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ----------------------------------------------------------------------------
// Backward, query side from stored dS.  When the key-side kernel has written
// every dS block (128 key rows x 128 query columns, bf16, the values its dK
// product reads), dQ = scale sum_kt dS_kt K_kt is a plain product chain: no
// scores, no softmax.  Work item = (128-row query tile qt, query head h); its
// key tiles are the 128-aligned tiles kt = floor(seq_start / 128) .. qt (the
// key-side kernel's tiles; keys before the sequence start carry dS = 0).  Per
// key tile one stage holds the dS block (A, read MN-major: queries are its
// contiguous columns) and the K tile (B, read MN-major: head columns), and
// the MMA thread adds the 128 x 128 x 128 product into one of two TMEM
// accumulators, so the read-out of one item overlaps the next item's
// products.  Warps: 0 loads, 1 issues the MMAs, 2-5 read dQ out (one query
// row per thread, TMEM lane quarter = warp % 4).
// ----------------------------------------------------------------------------
constexpr int QS_STAGES = 3;
constexpr int QS_THREADS = 192;

struct QsSmem {
    static constexpr int ST0 = 0;                 // stage s: dS block at ST0 + 4 BLK s, K tile 2 BLK after
    static constexpr int BAR = QS_STAGES * 4 * BLK;
    enum { FULL = 0, EMPTY = QS_STAGES, ACC_FULL = 2 * QS_STAGES, ACC_FREE = 2 * QS_STAGES + 2,
           DRAIN = 2 * QS_STAGES + 4, SCHED_FULL = 2 * QS_STAGES + 5, SCHED_EMPTY = SCHED_FULL + RING,
           NBARS = SCHED_EMPTY + RING };
    static constexpr int MISC = BAR + NBARS * 8;     // TMEM base, abort flag, then the item ring
    static constexpr int TOTAL = MISC + 32 + 1024;
};
static_assert(QsSmem::TOTAL <= 232448, "dynamic shared memory of one CTA");

// Query-side item over stored blocks: query tile qt of head h, key tiles
// kt0 .. qt (at most ktc of them; more would mean a sequence longer than the
// stored layout holds, which the row metadata rules out).
struct QsItem {
    int qt, h, kt0, nt;
};

__device__ __forceinline__ QsItem qs_item(const AttnParams& p, int item) {
    QsItem it;
    it.qt = item / p.n_heads;
    it.h = item % p.n_heads;
    it.kt0 = p.seq_start[it.qt * TB] / TB;
    if (it.qt - it.kt0 >= p.ktc) it.kt0 = it.qt - p.ktc + 1;
    it.nt = it.qt - it.kt0 + 1;
    return it;
}

// dQ (+)= dS K: M = 128 queries, N = 128 head columns, K = 128 keys; both
// operands MN-major tiles of 128 rows (keys) x 128 columns.
__device__ __forceinline__ void mma_dsk(uint32_t d, uint32_t ds, uint32_t k, bool acc) {
    const uint32_t id = idesc_bf16(128, 1, 1, 128);
    const uint64_t ad = mndesc(ds), bd = mndesc(k);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            umma_bf16(d, ad + 512 * kb + 128 * kk, bd + 512 * kb + 128 * kk, id, (acc || kb || kk) ? 1u : 0u);
}

__global__ void __launch_bounds__(QS_THREADS, 1)
    attn_bwd_q_stored_kernel(const __grid_constant__ AttnMaps maps, const AttnParams p, int n_items, int* status) {
    using SL = QsSmem;
    const int mt_valid = *p.meta < p.max_tiles ? *p.meta : p.max_tiles;
    auto valid = [&](int item) -> bool { return item >= 0 && item < n_items && item / p.n_heads < mt_valid; };
    if (blockIdx.x >= mt_valid * p.n_heads) return;   // more CTAs than items
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sb + SL::BAR + 8 * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SL::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SL::MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = p.n_heads / p.n_kv;

    volatile int* ring = reinterpret_cast<volatile int*>(smem + SL::MISC + 16);
    if (threadIdx.x == 0) {
        for (int i = 0; i < QS_STAGES; ++i) {
            mbar_init(bar(SL::FULL + i), 1);
            mbar_init(bar(SL::EMPTY + i), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(SL::ACC_FULL + a), 1);
            mbar_init(bar(SL::ACC_FREE + a), 4);      // the four read-out warps
        }
        mbar_init(bar(SL::DRAIN), 1);
        for (int i = 0; i < RING; ++i) {
            mbar_init(bar(SL::SCHED_FULL + i), 1);
            mbar_init(bar(SL::SCHED_EMPTY + i), 5);   // MMA thread, four read-out warps
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
        tma_prefetch_desc(&maps.rows128);
        tma_prefetch_desc(&maps.ds128);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;   // accumulator a at columns 128 a
    int dummy = 0;

    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            int last[QS_STAGES];
            for (int s = 0; s < QS_STAGES; ++s) last[s] = -1;
            uint32_t gj = 0;                           // blocks loaded by this CTA
            RingPos rp;
            while (ok) {
                int item = atomicAdd(p.counter, 1);
                if (!valid(item)) item = -1;
                if (!ring_put(bar(SL::SCHED_FULL), bar(SL::SCHED_EMPTY), ring, rp, item, abort_flag)) {
                    ok = false;
                    break;
                }
                if (item < 0) break;
                const QsItem it = qs_item(p, item);
                if (p.seq_start[it.qt * TB] / TB != it.kt0) raise_status(status, ST_RANGE);
                const int kcol = (p.n_heads + it.h / grp) * HD;
                for (int j = 0; j < it.nt; ++j, ++gj) {
                    const int s = (int)(gj % QS_STAGES);
                    const uint32_t sp = (gj / QS_STAGES) & 1u;
                    if (!mbar_wait(bar(SL::EMPTY + s), sp ^ 1u, abort_flag)) { ok = false; break; }
                    const int kt = it.kt0 + j;
                    const int64_t blk = ((int64_t)it.qt * p.ktc + (it.qt - kt)) * p.n_heads + it.h;
                    const uint32_t fb = bar(SL::FULL + s), st = sb + SL::ST0 + s * 4 * BLK;
                    mbar_expect_tx(fb, 4 * BLK);
                    load_tile128(st, &maps.ds128, fb, 0, (int)(blk * TB));
                    load_tile128(st + 2 * BLK, &maps.rows128, fb, kcol, kt * TB);
                    last[s] = (int)sp;
                }
            }
            if (!ok) { atomicOr(status, ST_TIMEOUT); *abort_flag = 1; }
            bool dr = true;                            // our copies have landed
            for (int s = 0; s < QS_STAGES; ++s)
                if (last[s] >= 0) dr &= mbar_wait(bar(SL::FULL + s), (uint32_t)last[s], (volatile int*)&dummy);
            if (!dr) atomicOr(status, ST_TIMEOUT);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = true;
            uint32_t gj = 0, nit = 0;                  // blocks and items consumed
            RingPos rp;
            while (ok) {
                int item;
                if (!ring_get(bar(SL::SCHED_FULL), bar(SL::SCHED_EMPTY), ring, rp, item, abort_flag)) {
                    ok = false;
                    break;
                }
                if (item < 0) break;
                const int nt = qs_item(p, item).nt;
                const int a = nit & 1;
                // the read-out of this accumulator's previous item is done
                if (nit >= 2 && !mbar_wait(bar(SL::ACC_FREE + a), ((nit >> 1) - 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                for (int j = 0; j < nt; ++j, ++gj) {
                    const int s = (int)(gj % QS_STAGES);
                    if (!mbar_wait(bar(SL::FULL + s), (gj / QS_STAGES) & 1u, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t st = sb + SL::ST0 + s * 4 * BLK;
                    mma_dsk(tmem + 128 * a, st, st + 2 * BLK, j > 0);
                    umma_commit(bar(SL::EMPTY + s));
                }
                if (!ok) break;
                umma_commit(bar(SL::ACC_FULL + a));
                ++nit;
            }
            if (!ok) { atomicOr(status, ST_TIMEOUT); *abort_flag = 1; }
            umma_commit(bar(SL::DRAIN));
            if (!mbar_wait(bar(SL::DRAIN), 0, (volatile int*)&dummy)) atomicOr(status, ST_TIMEOUT);
        }
    } else {
        const int q4 = warp & 3;
        const int r = 32 * q4 + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
        bool ok = true;
        uint32_t ra[32];
        uint32_t nit = 0;
        RingPos rp;
        while (ok) {
            int item;
            if (!ring_get_warp(bar(SL::SCHED_FULL), bar(SL::SCHED_EMPTY), ring, rp, item, abort_flag, lane)) {
                ok = false;
                break;
            }
            if (item < 0) break;
            const QsItem it = qs_item(p, item);
            const int a = nit & 1;
            if (!warp_wait(bar(SL::ACC_FULL + a), (nit >> 1) & 1u, abort_flag, lane)) { ok = false; break; }
            tc_fence_after();
            bf16* row = p.dqkv + (int64_t)(it.qt * TB + r) * p.ld_qkv + it.h * HD;
            float v[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                tmem_ld32(tl + 128 * a + 32 * c, ra);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(ra[e]) * p.scale;
                store32<bf16>(row + 32 * c, v);
            }
            // this accumulator has been read: a later item's products may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(SL::ACC_FREE + a));
            ++nit;
        }
        if (!ok && lane == 0) {
            atomicOr(status, ST_TIMEOUT);
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 256);
}

// D[h][p] = sum_c dO[p][h*128 + c] O[p][h*128 + c]: 16 threads per (row, head),
// 8 elements each.
__global__ void attn_rowdot_kernel(const bf16* __restrict__ dO, const bf16* __restrict__ O, int n_heads,
                                   const int* __restrict__ meta, int max_tiles, float* __restrict__ DT, int ld_t) {
    const int mt = *meta < max_tiles ? *meta : max_tiles;
    const int64_t rows = (int64_t)mt * TB;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t unit = gid >> 4;                 // (row, head)
    const int part = (int)(gid & 15);
    const int64_t row = unit / n_heads;
    const int h = (int)(unit % n_heads);
    float acc = 0.f;
    if (row < rows) {
        const int64_t off = row * (int64_t)n_heads * HD + h * HD + part * 8;
        const uint4 a = *reinterpret_cast<const uint4*>(dO + off);
        const uint4 b = *reinterpret_cast<const uint4*>(O + off);
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wa[e]));
            const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wb[e]));
            acc = fmaf(fa.x, fb.x, acc);
            acc = fmaf(fa.y, fb.y, acc);
        }
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (row < rows && part == 0) DT[(int64_t)h * ld_t + row] = acc;
}

// A persistent kernel: one CTA per SM (at most one per work item); the item
// counter starts at zero.
template <typename K>
cudaError_t launch_attn_persistent(K kernel, int smem_bytes, int threads, const AttnMaps& maps,
                                   const AttnParams& p, int n_items, int num_sms, int* status, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    if (n_items <= 0) return cudaSuccess;
    const int grid = n_items < num_sms ? n_items : num_sms;
    e = cudaMemsetAsync(p.counter, 0, sizeof(int), s);
    if (e != cudaSuccess) return e;
    kernel<<<grid, threads, smem_bytes, s>>>(maps, p, n_items, status);
    return cudaGetLastError();
}

bool make_maps(AttnMaps& m, const AttnArgs& a) {
    const int64_t W = (int64_t)(a.n_heads + 2 * a.n_kv) * HD;
    if (!tc_encode_bf16(&m.rows128, a.qkv, a.max_rows, W, W, 64, TB)) return false;
    if (a.dO) {
        if (!tc_encode_bf16(&m.do128, a.dO, a.max_rows, (int64_t)a.n_heads * HD, (int64_t)a.n_heads * HD, 64, TB))
            return false;
    } else {
        m.do128 = m.rows128;
    }
    if (a.ds) {
        const int64_t rows = (int64_t)(a.max_rows / TB) * a.ktc * a.n_heads * TB;
        if (a.ktc < 1 || rows > INT32_MAX || !tc_encode_bf16(&m.ds128, a.ds, rows, TB, TB, 64, TB)) return false;
    } else {
        m.ds128 = m.rows128;
    }
    return true;
}

AttnParams make_params(const AttnArgs& a) {
    AttnParams p;
    p.qkv = a.qkv;
    p.ld_qkv = (a.n_heads + 2 * a.n_kv) * HD;
    p.n_heads = a.n_heads;
    p.n_kv = a.n_kv;
    p.seq_start = a.seq_start;
    p.meta = a.meta;
    p.max_tiles = a.max_rows / TB;
    p.scale = 1.0f / sqrtf((float)HD);
    p.o = a.o;
    p.lseT = a.lseT;
    p.ld_t = a.ld_t;
    p.DT = a.DT;
    p.dqkv = a.dqkv;
    p.counter = a.counter;
    p.ds = a.ds;
    p.ktc = a.ktc;
    return p;
}

}  // namespace

cudaError_t launch_attention_fwd(const AttnArgs& a, int* status, cudaStream_t s) {
    AttnMaps maps;
    if (!make_maps(maps, a) || a.max_rows % TB || a.ld_t % 4) return cudaErrorInvalidValue;
    const AttnParams p = make_params(a);
    const int pairs = (a.n_heads / a.n_kv + 1) / 2;
    if (a.num_sms < 1 || !a.counter) return cudaErrorInvalidValue;
    return launch_attn_persistent(attn_fwd_kernel, FwdSmem::TOTAL, FWD_THREADS, maps, p, p.max_tiles * a.n_kv * pairs,
                                  a.num_sms, status, s);
}

cudaError_t launch_attention_bwd(const AttnArgs& a, int* status, cudaStream_t s) {
    AttnMaps maps;
    if (!a.dO || !make_maps(maps, a) || a.max_rows % TB || a.ld_t % 4) return cudaErrorInvalidValue;
    const AttnParams p = make_params(a);
    const int threads = 256;
    const int64_t units = (int64_t)a.max_rows * a.n_heads * 16;
    attn_rowdot_kernel<<<(unsigned)((units + threads - 1) / threads), threads, 0, s>>>(
        a.dO, a.o, a.n_heads, a.meta, p.max_tiles, a.DT, a.ld_t);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (a.num_sms < 1 || !a.counter) return cudaErrorInvalidValue;
    e = launch_attn_persistent(attn_bwd_kv_kernel, KvSmem::TOTAL, BWD_THREADS, maps, p, p.max_tiles * a.n_kv,
                               a.num_sms, status, s);
    if (e != cudaSuccess) return e;
    if (a.ds)   // dQ from the dS blocks the key side stored
        return launch_attn_persistent(attn_bwd_q_stored_kernel, QsSmem::TOTAL, QS_THREADS, maps, p,
                                      p.max_tiles * a.n_heads, a.num_sms, status, s);
    return launch_attn_persistent(attn_bwd_q_kernel, QSmem::TOTAL, BWD_THREADS, maps, p, p.max_tiles * a.n_heads,
                                  a.num_sms, status, s);
}

}  // namespace mlk
