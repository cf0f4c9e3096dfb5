// Tensor-core GEMM engine for sm_103a: C = A B^T (+ Ax Bx^T) on tcgen05 with
// TMEM accumulators, operands staged in shared memory by TMA, and the fused
// epilogues of gemm_common.cuh.
//
// One persistent CTA per SM, 6 warps:
//   warp 0      TMA producer (one elected thread) filling an S-stage ring of
//               128x64 A tiles and BNx64 B tiles (bf16, 128-byte swizzle)
//   warp 1      TMEM allocator and MMA issuer (one elected thread):
//               tcgen05.mma.cta_group::1.kind::f16, M=128, N=BN, K=16, into
//               one of two TMEM accumulators (2 x BN fp32 columns)
//   warps 2-5   epilogue: tcgen05.ld 32x32b.x32 of the finished accumulator,
//               one output row per thread, 32 columns at a time, while the
//               MMA warp already fills the other accumulator
// Tiles are scheduled statically (tile = blockIdx.x + i * gridDim.x) in
// bands of group_m row tiles, so CTAs running together share B tiles in L2.
// The adapter of a row tile (routing guarantees one per tile) selects the
// per-adapter rows of B / Bx: the SGMV shrink and expand of tinker-ticks
// ("How the SGMV kernel works") become one extra K block of the base GEMM.
//
// Every wait on an mbarrier is bounded (about 4 s of %globaltimer); on
// expiry the CTA raises the timeout status bit, stops issuing work, drains
// its own copies and MMAs (again bounded), frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "tc_ptx.cuh"

namespace mlk {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;                     // bf16 elements = 128 bytes per row
constexpr int NUM_THREADS = 192;

using namespace tcx;

// TMA loads of one stage's A tile (ROWS x 64, K-major box or two MN-major
// boxes) and B tile (ROWS x 64).  `pair` loads complete on the leader CTA's
// barrier (bar is then a shared::cluster address).
template <int ROWS>
__device__ __forceinline__ void load_tile_a(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            const GemmOperand& op, int m0, int k, int arow, bool pair) {
    if (!op.mn_major) {
        if (pair) tma_load_2d_pair(dst, map, bar, k, arow);
        else tma_load_2d(dst, map, bar, k, arow);
    } else {
#pragma unroll
        for (int i = 0; i < ROWS / 64; ++i) {
            if (pair) tma_load_2d_pair(dst + i * 8192, map, bar, m0 + 64 * i, (int)(k + op.row_shift));
            else tma_load_2d(dst + i * 8192, map, bar, m0 + 64 * i, (int)(k + op.row_shift));
        }
    }
}

template <int ROWS>
__device__ __forceinline__ void load_tile_b(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            const GemmOperand& op, int n0, int k, int adapter, bool pair) {
    const int brow = (int)((int64_t)adapter * op.ad_rows + op.row_shift);
    if (!op.mn_major) {
        if (pair) tma_load_2d_pair(dst, map, bar, k, brow + n0);
        else tma_load_2d(dst, map, bar, k, brow + n0);
    } else {
#pragma unroll
        for (int i = 0; i < ROWS / 64; ++i) {
            if (pair) tma_load_2d_pair(dst + i * 8192, map, bar, n0 + 64 * i, brow + k);
            else tma_load_2d(dst + i * 8192, map, bar, n0 + 64 * i, brow + k);
        }
    }
}

// EPI_LMFWD's first pass over a finished accumulator row: the maximum over the
// tile's columns < V, read from TMEM 32 columns at a time (the next chunk in
// flight while one is reduced).
template <int BN>
__device__ __forceinline__ float lm_tile_max(const GemmParams& p, uint32_t tbase, int col_base) {
    float m = -INFINITY;
    uint32_t ra[32], rb[32];
    auto red = [&](const uint32_t (&r)[32], int ch) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
        if (col_base + ch * 32 < p.N) m = fmaxf(m, lm_chunk_max(p.ep, col_base + ch * 32, v));
    };
    tmem_ld32(tbase, ra);
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ch += 2) {
        tmem_ld_wait();
        tmem_ld32(tbase + (ch + 1) * 32, rb);
        red(ra, ch);
        tmem_ld_wait();
        if (ch + 2 < BN / 32) tmem_ld32(tbase + (ch + 2) * 32, ra);
        red(rb, ch + 1);
    }
    return m;
}

// Epilogue of one finished accumulator for one thread's row: BN columns in
// chunks of 32.  The TMEM read of chunk c+1 is issued before chunk c is
// processed, so the load latency overlaps the epilogue arithmetic.
template <int BN>
__device__ __forceinline__ void epilogue_row(const GemmParams& p, uint32_t tbase, int64_t row, bool row_ok,
                                             int col_base, int adapter, int nt) {
    static_assert((BN / 32) % 2 == 0, "chunks are processed in pairs");
    EpiRowState st;
    epi_row_begin(st);
    if (p.ep.kind == EPI_LMFWD && row_ok) st.m = lm_tile_max<BN>(p, tbase, col_base);
    uint32_t ra[32], rb[32];
    tmem_ld32(tbase, ra);
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ch += 2) {
        tmem_ld_wait();
        tmem_ld32(tbase + (ch + 1) * 32, rb);
        {
            const int col0 = col_base + ch * 32;
            if (row_ok && col0 < p.N) {
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(ra[j]);
                epi_chunk<bf16>(p.ep, row, col0, adapter, v, st);
            }
        }
        tmem_ld_wait();
        if (ch + 2 < BN / 32) tmem_ld32(tbase + (ch + 2) * 32, ra);
        {
            const int col0 = col_base + (ch + 1) * 32;
            if (row_ok && col0 < p.N) {
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(rb[j]);
                epi_chunk<bf16>(p.ep, row, col0, adapter, v, st);
            }
        }
    }
    if (row_ok) epi_row_end(p.ep, row, nt, st);
}

// Epilogue of the export merge (EPI_MERGE: out = bf16(W + gamma acc)).  Its
// GEMM has K = 192, so unlike the other epilogues this one is not hidden
// behind a long mainloop: its time is the reads of W.  All of a row's W
// pieces of the tile (BN / 32 chunks of 32 columns) are requested before the
// first accumulator chunk is read, so each thread waits for memory once per
// tile instead of once per chunk.  The arithmetic (fmaf(gamma, acc, w), one
// rounding) is that of epi_chunk's EPI_MERGE.
template <int BN>
__device__ __forceinline__ void epilogue_row_merge(const GemmParams& p, uint32_t tbase, int64_t row, bool row_ok,
                                                   int col_base, int adapter) {
    constexpr int NCH = BN / 32;
    constexpr int D = NCH;
    const bf16* w = reinterpret_cast<const bf16*>(p.ep.aux) + row * p.ep.ld_aux + col_base;
    bf16* out = reinterpret_cast<bf16*>(p.ep.out0) + row * p.ep.ld0 + col_base;
    const float gm = p.ep.gamma[adapter];
    uint4 wb[D][4];
    auto load_w = [&](int ch, uint4 (&dst)[4]) {
        if (row_ok && col_base + 32 * ch < p.N) {
            const uint4* s4 = reinterpret_cast<const uint4*>(w + 32 * ch);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = __ldcs(s4 + q);     // read once: evict first
        }
    };
#pragma unroll
    for (int c = 0; c < D; ++c) load_w(c, wb[c]);
    uint32_t ra[32];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
        tmem_ld32(tbase + ch * 32, ra);
        tmem_ld_wait();
        if (row_ok && col_base + 32 * ch < p.N) {
            float v[32];
            load32<bf16>(reinterpret_cast<const bf16*>(wb[ch % D]), v);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = fmaf(gm, __uint_as_float(ra[j]), v[j]);
            store32<bf16>(out + 32 * ch, v);
        }
        if (ch + D < NCH) load_w(ch + D, wb[ch % D]);
    }
}

// Staged-store epilogues.  Each epilogue thread owns one row of the tile; a
// direct store writes the row's 32 columns of a chunk as 16-byte pieces, so
// one warp store instruction touches 32 rows, each piece a partial sector at
// the L2, and the load/store unit that also issues the producer's TMA copies
// and the MMA thread's tcgen05 instructions is busy for 32 wavefronts.  An
// ablation of the W1 forward GEMM (16,384 tokens, 8B widths) read the tensor
// pipe 88 % active without its epilogue's stores and math, 81 % with the
// math alone and 76 % with both.  Here the warp writes each 32 x 32 chunk of
// an output into a box in shared memory (st.shared.v4, conflict-free) and
// one lane writes the box out with a TMA store: whole 64- or 128-byte row
// segments.  The arithmetic is epi_chunk's, helper for helper.
//   SK_LMFWD  kept fp16 e = exp(z - tile max) (box 0 -> map C) + the row's
//             log-sum-exp state
//   SK_LMDZ   recomputed bf16 dz (box 0 -> map C)
//   SK_SILU   u = acc (box 0 -> map C) and act = silu(acc) (box 1 -> map D)
//   SK_DSILU  du = acc * silu'(u), u read directly (box 0 -> map C)
//   SK_RESID  h32 = (f32_in or h32) + acc (box F -> map D), its bf16 copy (box 0 -> map C)
// Boxes: fp32 32 x 32 with 128-byte rows and 128-byte swizzle (16-byte piece
// j of row r at piece j ^ (r & 7)); bf16 (or fp16) 32 x 32 with 64-byte rows
// and 64-byte swizzle (piece j at j ^ ((r >> 1) & 3)).  Both match the tensor
// maps' swizzle and put each quarter-warp's st.shared.v4 on distinct banks.
// A warp owns NBUF sets of boxes; the set of chunk c is refilled once the
// TMA stores of chunk c - NBUF have read it (one bulk group per chunk).
//   SK_MERGE  the export merge (see merge_tile): W boxes loaded by TMA one
//             tile ahead, out = bf16(W + gamma acc) in place, stored by TMA
enum { SK_NONE = 0, SK_LMFWD = 1, SK_LMDZ = 2, SK_SILU = 3, SK_DSILU = 4, SK_RESID = 5, SK_MERGE = 6 };

template <int SK>
struct StagedCfg {
    static constexpr bool F32 = SK == SK_RESID;                          // an fp32 box, first in the set
    static constexpr int N16 = SK == SK_MERGE ? 4 : (SK == SK_SILU ? 2 : 1);   // 16-bit boxes after it
    static constexpr int SET_BYTES = (F32 ? 4096 : 0) + 2048 * N16;
    static constexpr int NBUF = (SET_BYTES <= 4096 || SK == SK_MERGE) ? 2 : 1;
    static constexpr int WARP_BYTES = SK == SK_NONE ? 0 : NBUF * SET_BYTES;   // a multiple of 1024
    // epilogue warps per CTA: one per TMEM lane quadrant, two (each half of
    // the tile's columns) for the merge, whose epilogue is its whole time
    static constexpr int EPI_WARPS = SK == SK_MERGE ? 8 : 4;
    // every box staged_chunk / merge_tile addresses lies inside the warp's area
    static_assert(SK == SK_NONE || (SET_BYTES >= 2048 && WARP_BYTES >= SET_BYTES && WARP_BYTES % 1024 == 0),
                  "a staged kind needs room for its boxes");
};

template <int SK>
constexpr int pair_threads() { return 64 + 32 * StagedCfg<SK>::EPI_WARPS; }

__device__ __forceinline__ void box_row_f32(uint32_t box, int lane, const float* v) {
    const uint32_t rb = box + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        st_shared_v4(rb + ((j ^ (lane & 7)) << 4), __float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                     __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
}

__device__ __forceinline__ void box_row_half(uint32_t box, int lane, const float* v) {
    const uint32_t rb = box + lane * 64;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            __half2 h = __floats2half2_rn(v[8 * j + 2 * u], v[8 * j + 2 * u + 1]);
            w[u] = *reinterpret_cast<uint32_t*>(&h);
        }
        st_shared_v4(rb + ((j ^ ((lane >> 1) & 3)) << 4), w[0], w[1], w[2], w[3]);
    }
}

__device__ __forceinline__ void box_row_bf16(uint32_t box, int lane, const float* v) {
    const uint32_t rb = box + lane * 64;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        st_shared_v4(rb + ((j ^ ((lane >> 1) & 3)) << 4), pack_bf16x2(v[8 * j], v[8 * j + 1]),
                     pack_bf16x2(v[8 * j + 2], v[8 * j + 3]), pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                     pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
}

// One chunk C[row][col0 .. col0+31] of a staged epilogue.  `stg` is the
// warp's staging area, y0 its first output row, `nbox` counts its chunks.
template <int SK>
__device__ __forceinline__ void staged_chunk(const GemmParams& p, const CUtensorMap* mc, const CUtensorMap* md,
                                             int64_t row, int col0, const uint32_t (&r)[32], EpiRowState& st,
                                             uint32_t stg, uint32_t& nbox, int y0) {
    using CF = StagedCfg<SK>;
    const int lane = threadIdx.x & 31;
    const EpiParams& ep = p.ep;
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    // the directly read operand first, so its latency overlaps the wait below
    if (SK == SK_DSILU) {
        float u[32];
        load32<bf16>(reinterpret_cast<const bf16*>(ep.aux) + row * ep.ld_aux + col0, u);
        dsilu_values(v, u);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = u[j];
    } else if (SK == SK_RESID) {
        float h[32];
        load32<float>((ep.f32_in ? ep.f32_in : ep.f32) + row * ep.ldf + col0, h);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += h[j];
    }
    const uint32_t set = stg + (nbox % (uint32_t)CF::NBUF) * (uint32_t)CF::SET_BYTES;
    const uint32_t b16 = set + (CF::F32 ? 4096u : 0u);
    if (lane == 0) bulk_wait_read<CF::NBUF - 1>();
    __syncwarp();
    if (SK == SK_LMFWD) {
        float e[32];
        lmfwd_stats(ep, row, col0, v, st, e);
        box_row_half(b16, lane, e);
    } else if (SK == SK_LMDZ) {
        float o[32];
        lmdz_values<true>(ep, row, col0, v, o);
        box_row_bf16(b16, lane, o);
    } else if (SK == SK_SILU) {
        box_row_bf16(b16, lane, v);
        float a[32];
        silu_values(v, a);
        box_row_bf16(b16 + 2048, lane, a);
    } else if (SK == SK_DSILU) {
        box_row_bf16(b16, lane, v);
    } else {   // SK_RESID
        box_row_f32(set, lane, v);
        if (ep.out0) box_row_bf16(b16, lane, v);
    }
    fence_async_shared();
    __syncwarp();
    if (lane == 0) {
        // written once here and read by a later launch: evict-first in L2, so
        // that the outputs do not displace the operand tiles the GEMM re-reads
        const uint64_t pol = l2_policy_evict_first();
        if (SK == SK_LMFWD || SK == SK_LMDZ || SK == SK_DSILU) tma_store_2d_hint(mc, b16, col0, y0, pol);
        if (SK == SK_SILU) {
            tma_store_2d_hint(mc, b16, col0, y0, pol);
            tma_store_2d_hint(md, b16 + 2048, col0, y0, pol);
        }
        if (SK == SK_RESID) {
            tma_store_2d_hint(md, set, col0, y0, pol);
            if (ep.out0) tma_store_2d_hint(mc, b16, col0, y0, pol);
        }
        bulk_commit();
    }
    ++nbox;
}

// The staged epilogue of one thread's row; `row_ok` is uniform over the warp
// here (whole row tiles: M is a multiple of 128).
template <int BN, int SK>
__device__ __forceinline__ void epilogue_row_staged(const GemmParams& p, const CUtensorMap* mc,
                                                    const CUtensorMap* md, uint32_t tbase, int64_t row, bool row_ok,
                                                    int col_base, int nt, uint32_t stg, uint32_t& nbox, int y0) {
    static_assert((BN / 32) % 2 == 0, "chunks are processed in pairs");
    if (!row_ok) return;
    EpiRowState st;
    epi_row_begin(st);
    if (SK == SK_LMFWD) st.m = lm_tile_max<BN>(p, tbase, col_base);
    uint32_t ra[32], rb[32];
    tmem_ld32(tbase, ra);
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ch += 2) {
        tmem_ld_wait();
        tmem_ld32(tbase + (ch + 1) * 32, rb);
        if (col_base + ch * 32 < p.N)
            staged_chunk<SK>(p, mc, md, row, col_base + ch * 32, ra, st, stg, nbox, y0);
        tmem_ld_wait();
        if (ch + 2 < BN / 32) tmem_ld32(tbase + (ch + 2) * 32, ra);
        if (col_base + (ch + 1) * 32 < p.N)
            staged_chunk<SK>(p, mc, md, row, col_base + (ch + 1) * 32, rb, st, stg, nbox, y0);
    }
    epi_row_end(p.ep, row, nt, st);
}

// The export merge's chunks of one warp (SK_MERGE): W's 32 x 32 bf16 boxes
// of this warp's rows sit in shared memory (64-byte swizzle, as in
// box_row_bf16); each thread turns its row into bf16(W + gamma acc) in place,
// the arithmetic of epi_chunk's EPI_MERGE (one fmaf, one rounding).
__device__ __forceinline__ void merge_tile(uint32_t tbase, uint32_t set, int lane, int n, float gm) {
    uint32_t ra[32], rb[32];
    tmem_ld32(tbase, ra);
    auto chunk = [&](int ch, const uint32_t (&r)[32]) {
        const uint32_t rowb = set + (uint32_t)ch * 2048u + (uint32_t)lane * 64u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t a = rowb + ((j ^ ((lane >> 1) & 3)) << 4);
            uint32_t w0, w1, w2, w3;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3) : "r"(a));
            const uint32_t wv[4] = {w0, w1, w2, w3};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[e]));
                o[e] = pack_bf16x2(fmaf(gm, __uint_as_float(r[8 * j + 2 * e]), f.x),
                                   fmaf(gm, __uint_as_float(r[8 * j + 2 * e + 1]), f.y));
            }
            st_shared_v4(a, o[0], o[1], o[2], o[3]);
        }
    };
#pragma unroll 1
    for (int ch = 0; ch < n; ch += 2) {
        tmem_ld_wait();
        if (ch + 1 < n) tmem_ld32(tbase + (ch + 1) * 32, rb);
        chunk(ch, ra);
        if (ch + 1 >= n) break;
        tmem_ld_wait();
        if (ch + 2 < n) tmem_ld32(tbase + (ch + 2) * 32, ra);
        chunk(ch + 1, rb);
    }
    tmem_ld_wait();
}

struct TcMaps {
    CUtensorMap A, B, Ax, Bx;
    CUtensorMap C, D;  // outputs of the staged-store epilogues (32 x 32 boxes)
};

struct TileCoord {
    int valid;
    int mt;       // global m-tile (dense) / m-tile in the chunk (grouped)
    int nt;
    int adapter;
    int k0;       // first contraction index of the main operands
    int nkb;      // main K blocks
    int nkbx;     // extension K blocks
};

template <int BN>
__device__ __forceinline__ int total_tiles(const GemmParams& p) {
    const int n_nt = (p.N + BN - 1) / BN;
    if (!p.grouped) {
        int nmt = p.mtiles_dev ? *p.mtiles_dev : (p.M + BM - 1) / BM;
        int cnt = nmt - p.mt_base;
        if (cnt > p.mt_count) cnt = p.mt_count;
        if (cnt < 0) cnt = 0;
        return cnt * n_nt;
    }
    const int mtiles = (p.M + BM - 1) / BM;
    int nch = *p.nchunks_dev;
    if (nch > p.max_chunks) nch = p.max_chunks;
    return nch * mtiles * n_nt;
}

template <int BN>
__device__ __forceinline__ TileCoord tile_coord(const GemmParams& p, int t) {
    TileCoord c;
    const int n_nt = (p.N + BN - 1) / BN;
    c.valid = 1;
    if (!p.grouped) {
        int nmt = p.mtiles_dev ? *p.mtiles_dev : (p.M + BM - 1) / BM;
        int cnt = nmt - p.mt_base;
        if (cnt > p.mt_count) cnt = p.mt_count;
        const int G = p.group_m > 0 ? p.group_m : 1;
        const int band = t / (G * n_nt);
        const int r = t - band * G * n_nt;
        int bm = cnt - band * G;
        if (bm > G) bm = G;
        const int ml = band * G + r % bm;
        c.mt = p.mt_base + ml;
        c.nt = r / bm;
        c.adapter = p.tile_ad ? p.tile_ad[c.mt] : 0;
        if (c.adapter < 0) c.adapter = 0;
        c.k0 = 0;
        c.nkb = (p.K + BK - 1) / BK;
        c.nkbx = (p.Kx + BK - 1) / BK;
    } else {
        const int mtiles = (p.M + BM - 1) / BM;
        const int per_chunk = mtiles * n_nt;
        const int ci = t / per_chunk;
        const int r = t - ci * per_chunk;
        c.mt = r % mtiles;
        c.nt = r / mtiles;
        const int4 ch = p.chunks[ci];
        c.adapter = ch.x;
        c.k0 = ch.y;
        c.nkb = (ch.z + BK - 1) / BK;
        c.nkbx = 0;
    }
    return c;
}

template <int BN, int STAGES, int SUB = 1>
struct SmemLayout {
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int SUB_BYTES = A_BYTES + B_BYTES;         // one 64-wide K block: A rows, then B rows
    static constexpr int STAGE_BYTES = SUB * SUB_BYTES;         // a stage holds up to SUB consecutive K blocks
    static constexpr int TILES_BYTES = STAGES * STAGE_BYTES;
    static constexpr int BAR_OFF = TILES_BYTES;                 // full[S], empty[S], tfull[2], tempty[2], drain
    static constexpr int NBARS = 2 * STAGES + 5;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;        // tmem base, abort flag
    static constexpr int TOTAL = MISC_OFF + 16 + 1024;          // + alignment slack
};

// MERGE selects the export-merge epilogue (a separate instantiation, so the
// other GEMMs keep their register allocation).  SUB: K blocks per stage (the
// main blocks and the extension's are grouped separately; a group's last
// stage may hold fewer), so that each barrier hand-off moves SUB blocks.
template <int BN, int STAGES, bool MERGE = false, int SUB = 1>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ TcMaps maps, const GemmParams p, int* status) {
    using SL = SmemLayout<BN, STAGES, SUB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + SL::BAR_OFF;
    const uint32_t bar_empty = bar_full + STAGES * 8;
    const uint32_t bar_tfull = bar_empty + STAGES * 8;
    const uint32_t bar_tempty = bar_tfull + 2 * 8;
    const uint32_t bar_drain = bar_tempty + 2 * 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SL::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SL::MISC_OFF + 4);
    constexpr uint32_t TMEM_COLS = (2 * BN < 32) ? 32 : 2 * BN;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_tfull + 8 * b, 1);
            mbar_init(bar_tempty + 8 * b, 4);
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tma_prefetch_desc(&maps.A);
        tma_prefetch_desc(&maps.B);
        if (p.Kx > 0) {
            tma_prefetch_desc(&maps.Ax);
            tma_prefetch_desc(&maps.Bx);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int ntiles = total_tiles<BN>(p);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued[STAGES];
            for (int s = 0; s < STAGES; ++s) issued[s] = -1;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const TileCoord c = tile_coord<BN>(p, t);
                const int m0 = c.mt * BM;
                const int n0 = c.nt * BN;
                const int withhold = (blockIdx.x == 0 && t == 0) ? p.test_withhold_kb : -1;
                for (int kb = 0; kb < c.nkb && ok; kb += SUB) {
                    const int cnt = c.nkb - kb < SUB ? c.nkb - kb : SUB;
                    if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, abort_flag)) { ok = false; break; }
                    if (withhold >= kb && withhold < kb + cnt) {   // test hook: this stage is never filled
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                        continue;
                    }
                    const uint32_t fb = bar_full + 8 * stage;
                    const uint32_t sa = sbase + stage * SL::STAGE_BYTES;
                    mbar_expect_tx(fb, cnt * SL::SUB_BYTES);
                    for (int u = 0; u < cnt; ++u) {
                        const int k = c.k0 + (kb + u) * BK;
                        const uint32_t su = sa + u * SL::SUB_BYTES;
                        load_tile_a<BM>(su, &maps.A, fb, p.A, m0, k, (int)(m0 + p.A.row_shift), false);
                        load_tile_b<BN>(su + SL::A_BYTES, &maps.B, fb, p.B, n0, k, c.adapter, false);
                    }
                    issued[stage] = (int)phase;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                for (int kb = 0; kb < c.nkbx && ok; kb += SUB) {
                    const int cnt = c.nkbx - kb < SUB ? c.nkbx - kb : SUB;
                    if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, abort_flag)) { ok = false; break; }
                    const uint32_t fb = bar_full + 8 * stage;
                    const uint32_t sa = sbase + stage * SL::STAGE_BYTES;
                    mbar_expect_tx(fb, cnt * SL::SUB_BYTES);
                    for (int u = 0; u < cnt; ++u) {
                        const int k = (kb + u) * BK;
                        const uint32_t su = sa + u * SL::SUB_BYTES;
                        load_tile_a<BM>(su, &maps.Ax, fb, p.Ax, m0, k, (int)(m0 + p.Ax.row_shift), false);
                        load_tile_b<BN>(su + SL::A_BYTES, &maps.Bx, fb, p.Bx, n0, k, c.adapter, false);
                    }
                    issued[stage] = (int)phase;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                atomicOr(status, ST_TIMEOUT);
                *abort_flag = 1;
            }
            // our copies must have landed before the CTA may exit
            for (int s = 0; s < STAGES; ++s)
                if (issued[s] >= 0) {
                    int dummy = 0;
                    if (!mbar_wait(bar_full + 8 * s, (uint32_t)issued[s], (volatile int*)&dummy)) {
                        atomicOr(status, ST_TIMEOUT);
                    }
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            const uint32_t id_main = idesc_bf16(BN, p.A.mn_major, p.B.mn_major);
            const uint32_t id_ext = idesc_bf16(BN, p.Ax.mn_major, p.Bx.mn_major);
            const uint64_t full_limit = p.test_wait_ns ? p.test_wait_ns : TIMEOUT_NS;
            // stage-0 descriptors, advanced by additions to the start-address field
            // (see the CTA-pair kernel's MMA thread)
            const uint32_t sb0 = sbase + SL::A_BYTES;
            const uint64_t a0 = p.A.mn_major ? sdesc(sbase, 8192, 1024) : sdesc(sbase, 16, 1024);
            const uint64_t b0 = p.B.mn_major ? sdesc(sb0, 8192, 1024) : sdesc(sb0, 16, 1024);
            const uint64_t ax0 = p.Ax.mn_major ? sdesc(sbase, 8192, 1024) : sdesc(sbase, 16, 1024);
            const uint64_t bx0 = p.Bx.mn_major ? sdesc(sb0, 8192, 1024) : sdesc(sb0, 16, 1024);
            const uint32_t a_step = p.A.mn_major ? (2048 >> 4) : (32 >> 4);
            const uint32_t b_step = p.B.mn_major ? (2048 >> 4) : (32 >> 4);
            const uint32_t ax_step = p.Ax.mn_major ? (2048 >> 4) : (32 >> 4);
            const uint32_t bx_step = p.Bx.mn_major ? (2048 >> 4) : (32 >> 4);
            constexpr uint32_t STAGE_STEP = SL::STAGE_BYTES >> 4;
            constexpr uint32_t SUB_STEP = SL::SUB_BYTES >> 4;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const TileCoord c = tile_coord<BN>(p, t);
                if (!mbar_wait(bar_tempty + 8 * acc, acc_phase ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < c.nkb; kb += SUB) {
                    const int cnt = c.nkb - kb < SUB ? c.nkb - kb : SUB;
                    if (!mbar_try_wait(bar_full + 8 * stage, phase) &&
                        !mbar_wait(bar_full + 8 * stage, phase, abort_flag, full_limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int u = 0; u < cnt; ++u) {
                        const uint64_t ad = a0 + (uint64_t)(stage * STAGE_STEP + u * SUB_STEP);
                        const uint64_t bd = b0 + (uint64_t)(stage * STAGE_STEP + u * SUB_STEP);
                        umma_bf16(d_tmem, ad, bd, id_main, (kb + u) > 0 ? 1u : 0u);
#pragma unroll
                        for (int kk = 1; kk < BK / 16; ++kk)
                            umma_bf16(d_tmem, ad + kk * a_step, bd + kk * b_step, id_main, 1u);
                    }
                    umma_commit(bar_empty + 8 * stage);     // frees the stage when the MMAs finish
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                for (int kb = 0; kb < c.nkbx && ok; kb += SUB) {
                    const int cnt = c.nkbx - kb < SUB ? c.nkbx - kb : SUB;
                    if (!mbar_try_wait(bar_full + 8 * stage, phase) &&
                        !mbar_wait(bar_full + 8 * stage, phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int u = 0; u < cnt; ++u) {
                        const uint64_t ad = ax0 + (uint64_t)(stage * STAGE_STEP + u * SUB_STEP);
                        const uint64_t bd = bx0 + (uint64_t)(stage * STAGE_STEP + u * SUB_STEP);
                        umma_bf16(d_tmem, ad, bd, id_ext, (c.nkb > 0 || kb + u > 0) ? 1u : 0u);
#pragma unroll
                        for (int kk = 1; kk < BK / 16; ++kk)
                            umma_bf16(d_tmem, ad + kk * ax_step, bd + kk * bx_step, id_ext, 1u);
                    }
                    umma_commit(bar_empty + 8 * stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(bar_tfull + 8 * acc);           // accumulator ready
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            if (!ok) {
                atomicOr(status, ST_TIMEOUT);
                *abort_flag = 1;
            }
            // drain: every MMA issued by this thread completes before TMEM is freed
            umma_commit(bar_drain);
            int dummy = 0;
            if (!mbar_wait(bar_drain, 0, (volatile int*)&dummy)) atomicOr(status, ST_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
            const TileCoord c = tile_coord<BN>(p, t);
            bool ok = true;
            if (lane == 0) ok = mbar_wait(bar_tfull + 8 * acc, acc_phase, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                if (lane == 0) { atomicOr(status, ST_TIMEOUT); *abort_flag = 1; }
                break;
            }
            tc_fence_after();
            const int64_t row = (int64_t)c.mt * BM + 32 * q + lane;
            const bool row_ok = row < p.M;
            const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN);
            if (MERGE) epilogue_row_merge<BN>(p, tbase, row, row_ok, c.nt * BN, c.adapter);
            else epilogue_row<BN>(p, tbase, row, row_ok, c.nt * BN, c.adapter, c.nt);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ---- CTA-pair kernel: 256 x BN tiles with tcgen05.mma.cta_group::2 ---------
//
// A cluster of two CTAs on two SMs computes one 256-row x BN tile.  Each CTA
// stages its own 128 rows of A and half of the B tile (BN/2 rows); the MMA
// issued by the leader (cluster rank 0) reads both CTAs' shared memory and
// writes rows 0-127 of the accumulator into the leader's TMEM and rows
// 128-255 into the peer's.  Both CTAs' TMA loads complete on the leader's
// "full" barrier; the leader's MMA commits arrive on the "empty" and "tmem
// full" barriers of both CTAs (multicast); both CTAs' epilogue warps release
// the accumulator on the leader's "tmem empty" barrier.  Used for GEMMs whose
// B operand is shared by all rows (the LM head); the per-adapter GEMMs keep
// the single-CTA kernel.
// SK: the staged-store epilogue kind (SK_NONE: stores straight from
// registers); its four epilogue warps' staging boxes follow the stages.
template <int BN, int STAGES, int NUM_ACC, int SUB, int SK = SK_NONE>
struct SmemLayoutPair {
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = (BN / 2) * BK * 2;
    static constexpr int SUB_BYTES = A_BYTES + B_BYTES;   // one 64-wide K block: A rows, then B rows
    static constexpr int STAGE_BYTES = SUB * SUB_BYTES;   // a stage holds SUB consecutive K blocks
    static constexpr int TILES_BYTES = STAGES * STAGE_BYTES;
    static constexpr int STG_WARP = StagedCfg<SK>::WARP_BYTES;
    static constexpr int STG_OFF = TILES_BYTES;            // 1024-aligned (swizzled boxes)
    static constexpr int STG_BYTES = StagedCfg<SK>::EPI_WARPS * STG_WARP;
    static constexpr int SCHED = 4;                     // tile-index ring depth
    static constexpr int BAR_OFF = STG_OFF + STG_BYTES;
    static constexpr int NBARS = 2 * STAGES + 2 * NUM_ACC + 1 + 2 * SCHED + 2 * StagedCfg<SK>::EPI_WARPS;
    static constexpr int SLOT_OFF = BAR_OFF + NBARS * 8;
    static constexpr int MISC_OFF = SLOT_OFF + SCHED * 4;
    static constexpr int TOTAL = MISC_OFF + 16 + 1024;
    static_assert(TOTAL <= 232448, "dynamic shared memory of one CTA");
    static_assert(STG_BYTES == StagedCfg<SK>::EPI_WARPS * StagedCfg<SK>::WARP_BYTES, "staging area");
};

struct PairCoord {
    int mt;       // first global m-tile of the pair
    int nt;
    int k0, nkb;
    int a0, a1;   // adapters of the pair's two row tiles
    int nkbx;     // extension K blocks per adapter
    int next;     // extension stages: nkbx, or 2 * nkbx when a0 != a1
};

template <int BN>
__device__ __forceinline__ int pair_mcount(const GemmParams& p) {
    int nmt = p.mtiles_dev ? *p.mtiles_dev : (p.M + BM - 1) / BM;
    int cnt = nmt - p.mt_base;
    if (cnt > p.mt_count) cnt = p.mt_count;
    return cnt < 0 ? 0 : cnt;
}

template <int BN>
__device__ __forceinline__ PairCoord pair_coord(const GemmParams& p, int t, int cnt) {
    PairCoord c;
    const int n_nt = (p.N + BN - 1) / BN;
    const int pairs = (cnt + 1) / 2;
    int G = p.group_m / 2;
    if (G < 1) G = 1;
    const int band = t / (G * n_nt);
    const int r = t - band * G * n_nt;
    int bm = pairs - band * G;
    if (bm > G) bm = G;
    c.mt = p.mt_base + 2 * (band * G + r % bm);
    c.nt = r / bm;
    c.k0 = 0;
    c.nkb = (p.K + BK - 1) / BK;
    c.a0 = c.a1 = 0;
    if (p.tile_ad) {
        c.a0 = p.tile_ad[c.mt];
        c.a1 = (c.mt + 1 - p.mt_base) < cnt ? p.tile_ad[c.mt + 1] : c.a0;
        if (c.a0 < 0) c.a0 = 0;
        if (c.a1 < 0) c.a1 = c.a0;
    }
    c.nkbx = (p.Kx + BK - 1) / BK;
    c.next = (c.a0 == c.a1) ? c.nkbx : 2 * c.nkbx;
    return c;
}

// Tile scheduling: the leader's producer thread takes pair-tile indices from
// a global counter (atomicAdd), so the tiles in flight on the GPU stay
// consecutive and the band raster keeps its L2 reuse (a static per-cluster
// list lets clusters drift apart over thousands of tiles).  Each index is
// published through a small ring in both CTAs' shared memory; the peer's
// producer, the leader's MMA thread and all eight epilogue warps take it
// from there and release the slot on the leader's "sched empty" barrier.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __noinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > TIMEOUT_NS) return false;
        }
    }
}

__device__ __forceinline__ void st_shared_cluster(uint32_t cluster_addr, int v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Take the next tile index from ring slot `slot` (phase `ph`) and release the
// slot on the leader's barrier.  Returns false on timeout; t = -1 ends the work.
__device__ __forceinline__ bool sched_take(uint32_t bar_sfull, uint32_t sempty_leader, const volatile int* slots,
                                           int& slot, uint32_t& ph, bool leader, volatile int* abort_flag,
                                           int& t) {
    if (!mbar_wait_cluster(bar_sfull + 8 * slot, ph, abort_flag)) return false;
    t = slots[slot];
    if (leader) mbar_arrive(sempty_leader + 8 * slot);
    else mbar_arrive_cluster(sempty_leader + 8 * slot);
    if (++slot == 4) { slot = 0; ph ^= 1u; }
    return true;
}

template <int BN, int STAGES, int NUM_ACC, int SUB, bool MERGE = false, int SK = SK_NONE>
__global__ void __launch_bounds__(pair_threads<SK>(), 1)
    tc_gemm_pair_kernel(const __grid_constant__ TcMaps maps, const GemmParams p, int* status, int* dbg) {
    using SL = SmemLayoutPair<BN, STAGES, NUM_ACC, SUB, SK>;
    static_assert(SK == SK_NONE || (!MERGE && BN == 256), "staged stores: 256-wide tiles");
    static_assert(SK != SK_MERGE || (NUM_ACC == 2 && SUB == 1), "merge: two accumulators, one-block stages");
    static_assert(SL::SCHED == 4, "sched_take assumes a 4-slot ring");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + SL::BAR_OFF;
    const uint32_t bar_empty = bar_full + STAGES * 8;
    const uint32_t bar_tfull = bar_empty + STAGES * 8;
    const uint32_t bar_tempty = bar_tfull + NUM_ACC * 8;
    const uint32_t bar_drain = bar_tempty + NUM_ACC * 8;
    const uint32_t bar_sfull = bar_drain + 8;
    const uint32_t bar_sempty = bar_sfull + SL::SCHED * 8;
    const uint32_t bar_epi = bar_sempty + SL::SCHED * 8;     // 2 per epilogue warp (the merge's W loads)
    volatile int* slots = reinterpret_cast<volatile int*>(smem + SL::SLOT_OFF);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SL::MISC_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SL::MISC_OFF + 4);
    constexpr uint32_t TMEM_COLS = NUM_ACC * BN;
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation must be a power of two");
    // WIDE: 256 x 512 tiles, each K step two N = 256 MMAs into TMEM columns
    // 0-255 and 256-511; each CTA holds B columns [256 h + 128 rank, +128) of
    // tile half h (the operand split of a cta_group::2 MMA), 16 KB apart
    constexpr bool WIDE = BN > 256;
    constexpr int BN_MMA = WIDE ? 256 : BN;
    static_assert(!WIDE || (BN == 512 && NUM_ACC == 1), "wide tiles: 256 x 512, one accumulator");

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b = 0; b < NUM_ACC; ++b) {
            mbar_init(bar_tfull + 8 * b, 1);
            mbar_init(bar_tempty + 8 * b, 2 * StagedCfg<SK>::EPI_WARPS);
        }
        mbar_init(bar_drain, 1);
        for (int s = 0; s < SL::SCHED; ++s) {
            mbar_init(bar_sfull + 8 * s, 1);
            // peer producer, leader MMA, both CTAs' epilogue warps
            mbar_init(bar_sempty + 8 * s, 2 + 2 * StagedCfg<SK>::EPI_WARPS);
        }
        for (int b = 0; b < 2 * StagedCfg<SK>::EPI_WARPS; ++b) mbar_init(bar_epi + 8 * b, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tma_prefetch_desc(&maps.A);
        tma_prefetch_desc(&maps.B);
        if (p.Kx > 0) {
            tma_prefetch_desc(&maps.Ax);
            tma_prefetch_desc(&maps.Bx);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (dbg && threadIdx.x == 0) dbg[blockIdx.x] = (int)tmem_base;

    const int cnt = pair_mcount<BN>(p);
    const int n_nt = (p.N + BN - 1) / BN;
    const int ntiles = ((cnt + 1) / 2) * n_nt;
    const uint32_t full_leader = map_to_rank(bar_full, 0);
    const uint32_t tempty_leader = map_to_rank(bar_tempty, 0);
    const uint32_t sempty_leader = map_to_rank(bar_sempty, 0);

    if (warp == 0) {
        // ------------------------------------------------------------ producers (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued[STAGES];
            for (int s = 0; s < STAGES; ++s) issued[s] = -1;
            bool ok = true;
            int sslot = 0;
            uint32_t sph = 0;
            const uint32_t sfull_peer = map_to_rank(bar_sfull, 1);
            const uint32_t slot_peer = map_to_rank(smem_u32(const_cast<int*>(slots)), 1);
            // scheduler (leader): the next pair tile is fetched from the global
            // counter when the current one starts and published to both CTAs after
            // the current tile's first stage is queued, so neither the atomic nor
            // the peer's ring wait sits between two tiles' loads
            auto publish = [&](int tp) -> bool {
                if (!mbar_wait(bar_sempty + 8 * sslot, sph ^ 1u, abort_flag)) return false;
                slots[sslot] = tp;
                st_shared_cluster(slot_peer + 4 * sslot, tp);
                mbar_arrive(bar_sfull + 8 * sslot);
                mbar_arrive_cluster(sfull_peer + 8 * sslot);
                if (++sslot == SL::SCHED) { sslot = 0; sph ^= 1u; }
                return true;
            };
            auto fetch = [&]() -> int {
                const int tf = atomicAdd(p.tile_counter, 1);
                return tf >= ntiles ? -1 : tf;
            };
            int t_cur = -1;
            if (leader) {
                t_cur = fetch();
                ok = publish(t_cur);
            }
            for (; ok;) {
                int t;
                if (leader) {
                    t = t_cur;
                } else if (!sched_take(bar_sfull, sempty_leader, slots, sslot, sph, false, abort_flag, t)) {
                    ok = false;
                    break;
                }
                if (t < 0) break;
                const int t_next = leader ? fetch() : -1;
                bool published = !leader;
                const PairCoord c = pair_coord<BN>(p, t, cnt);
                const int m0 = (c.mt + (int)rank) * BM;
                const int n0 = c.nt * BN + (int)rank * (BN_MMA / 2);
                const int nst = (c.nkb + SUB - 1) / SUB;
                for (int ks = 0; ks < nst && ok; ++ks) {
                    if (ks == 1 && !published) {
                        if (!publish(t_next)) { ok = false; break; }
                        published = true;
                    }
                    if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, abort_flag)) { ok = false; break; }
                    const int nsub = c.nkb - ks * SUB < SUB ? c.nkb - ks * SUB : SUB;
                    if (leader) mbar_expect_tx(bar_full + 8 * stage, 2 * nsub * SL::SUB_BYTES);
                    const uint32_t fb = full_leader + 8 * stage;
                    for (int h = 0; h < nsub; ++h) {
                        const uint32_t sa = sbase + stage * SL::STAGE_BYTES + h * SL::SUB_BYTES;
                        const int k = c.k0 + (ks * SUB + h) * BK;
                        load_tile_a<BM>(sa, &maps.A, fb, p.A, m0, k, (int)(m0 + p.A.row_shift), true);
                        load_tile_b<BN_MMA / 2>(sa + SL::A_BYTES, &maps.B, fb, p.B, n0, k, 0, true);
                        if (WIDE)
                            load_tile_b<BN_MMA / 2>(sa + SL::A_BYTES + (BN_MMA / 2) * BK * 2, &maps.B, fb, p.B,
                                                    n0 + BN_MMA, k, 0, true);
                    }
                    issued[stage] = (int)phase;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                // K extension: with two adapters in the pair, stage `half` multiplies
                // adapter a_half's factor with only that half's rows (the other CTA
                // loads zeros, read out of bounds)
                for (int e = 0; e < c.next && ok; ++e) {
                    if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, abort_flag)) { ok = false; break; }
                    if (leader) mbar_expect_tx(bar_full + 8 * stage, 2 * SL::SUB_BYTES);   // one K block
                    const uint32_t fb = full_leader + 8 * stage;
                    const uint32_t sa = sbase + stage * SL::STAGE_BYTES;
                    const int half = e / c.nkbx;
                    const int k = (e - half * c.nkbx) * BK;
                    int adapter = c.a0;
                    int arow = (int)(m0 + p.Ax.row_shift);
                    if (c.a0 != c.a1) {
                        adapter = half ? c.a1 : c.a0;
                        if ((int)rank != half) arow = -BM;
                    }
                    load_tile_a<BM>(sa, &maps.Ax, fb, p.Ax, m0, k, arow, true);
                    load_tile_b<BN / 2>(sa + SL::A_BYTES, &maps.Bx, fb, p.Bx, n0, k, adapter, true);
                    issued[stage] = (int)phase;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (ok && !published) ok = publish(t_next);
                if (!ok) break;
                t_cur = t_next;
            }
            if (!ok) {
                atomicOr(status, ST_TIMEOUT);
                *abort_flag = 1;
            }
            if (leader) {
                // the pair's copies of every issued stage have landed (counted here)
                for (int s = 0; s < STAGES; ++s)
                    if (issued[s] >= 0) {
                        int dummy = 0;
                        if (!mbar_wait(bar_full + 8 * s, (uint32_t)issued[s], (volatile int*)&dummy))
                            atomicOr(status, ST_TIMEOUT);
                    }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA (leader)
        if (leader && lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            int sslot = 0;
            uint32_t sph = 0;
            const uint32_t id_main = idesc_bf16(BN_MMA, p.A.mn_major, p.B.mn_major, 2 * BM);
            const uint32_t id_ext = idesc_bf16(BN_MMA, p.Ax.mn_major, p.Bx.mn_major, 2 * BM);
            constexpr uint32_t B_HALF = ((BN_MMA / 2) * BK * 2) >> 4;   // second half's B, descriptor units
            // Descriptors of stage 0; a stage / K step only moves the start-address
            // field (bits 0-13, address >> 4), which stays below 2^14 for any
            // shared-memory address, so they are advanced by plain additions.  A
            // single thread issues every MMA: its work per K block is kept to a
            // try-wait, a few adds, four MMAs and the commit.
            const uint64_t a0 = sdesc(sbase, 16, 1024);   // A and Ax are K-major here
            const uint64_t b0 = p.B.mn_major ? sdesc(sbase + SL::A_BYTES, 8192, 1024)
                                             : sdesc(sbase + SL::A_BYTES, 16, 1024);
            const uint64_t bx0 = p.Bx.mn_major ? sdesc(sbase + SL::A_BYTES, 8192, 1024)
                                               : sdesc(sbase + SL::A_BYTES, 16, 1024);
            const uint32_t b_step = p.B.mn_major ? (2048 >> 4) : (32 >> 4);
            const uint32_t bx_step = p.Bx.mn_major ? (2048 >> 4) : (32 >> 4);
            constexpr uint32_t STAGE_STEP = SL::STAGE_BYTES >> 4;
            constexpr uint32_t SUB_STEP = SL::SUB_BYTES >> 4;
            for (;;) {
                int t;
                if (!sched_take(bar_sfull, sempty_leader, slots, sslot, sph, true, abort_flag, t)) {
                    ok = false;
                    break;
                }
                if (t < 0) break;
                const PairCoord c = pair_coord<BN>(p, t, cnt);
                if (!mbar_wait(bar_tempty + 8 * acc, acc_phase ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                const int nst = (c.nkb + SUB - 1) / SUB;
                for (int ks = 0; ks < nst; ++ks) {
                    if (!mbar_try_wait(bar_full + 8 * stage, phase) &&
                        !mbar_wait(bar_full + 8 * stage, phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = a0 + (uint64_t)(stage * STAGE_STEP);
                    const uint64_t bd = b0 + (uint64_t)(stage * STAGE_STEP);
                    umma_bf16_pair(d_tmem, ad, bd, id_main, ks > 0 ? 1u : 0u);
                    if (WIDE) umma_bf16_pair(d_tmem + BN_MMA, ad, bd + B_HALF, id_main, ks > 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 1; kk < BK / 16; ++kk) {
                        umma_bf16_pair(d_tmem, ad + kk * 2, bd + kk * b_step, id_main, 1u);
                        if (WIDE) umma_bf16_pair(d_tmem + BN_MMA, ad + kk * 2, bd + B_HALF + kk * b_step, id_main, 1u);
                    }
#pragma unroll
                    for (int h = 1; h < SUB; ++h) {
                        if (ks * SUB + h >= c.nkb) break;
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            umma_bf16_pair(d_tmem, ad + h * SUB_STEP + kk * 2, bd + h * SUB_STEP + kk * b_step,
                                           id_main, 1u);
                            if (WIDE)
                                umma_bf16_pair(d_tmem + BN_MMA, ad + h * SUB_STEP + kk * 2,
                                               bd + B_HALF + h * SUB_STEP + kk * b_step, id_main, 1u);
                        }
                    }
                    umma_commit_pair_mc(bar_empty + 8 * stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                for (int e = 0; e < c.next && ok; ++e) {
                    if (!mbar_try_wait(bar_full + 8 * stage, phase) &&
                        !mbar_wait(bar_full + 8 * stage, phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = a0 + (uint64_t)(stage * STAGE_STEP);
                    const uint64_t bd = bx0 + (uint64_t)(stage * STAGE_STEP);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16_pair(d_tmem, ad + kk * 2, bd + kk * bx_step, id_ext, 1u);
                    umma_commit_pair_mc(bar_empty + 8 * stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit_pair_mc(bar_tfull + 8 * acc);
                if (++acc == NUM_ACC) { acc = 0; acc_phase ^= 1u; }
            }
            if (!ok) {
                atomicOr(status, ST_TIMEOUT);
                *abort_flag = 1;
            }
            umma_commit_pair(bar_drain);
            int dummy = 0;
            if (!mbar_wait(bar_drain, 0, (volatile int*)&dummy)) atomicOr(status, ST_TIMEOUT);
        }
    } else if constexpr (SK == SK_MERGE) {
        // ------------------------------------------------------------ export-merge epilogue (both CTAs)
        const int q = warp & 3;
        const uint32_t stg = sbase + SL::STG_OFF + (uint32_t)(warp - 2) * (uint32_t)SL::STG_WARP;
        const uint32_t wbar = bar_epi + (uint32_t)(warp - 2) * 16u;
        const int cbase = ((warp - 2) >> 2) * (BN / 2);           // this warp's half of the columns
        constexpr uint32_t SET = 4u * 2048u;                      // one tile's W boxes
        const float gm = p.ep.gamma[0];
        int acc = 0;
        uint32_t acc_phase = 0;
        int sslot = 0;
        uint32_t sph = 0;
        uint32_t wph = 0;      // bit s: parity of set s's barrier
        uint32_t pend = 0;     // bit s: set s has W loads in flight not yet waited for
        auto take = [&](int& t) -> bool {
            bool ok = true;
            t = -1;
            if (lane == 0) ok = sched_take(bar_sfull, sempty_leader, slots, sslot, sph, leader, abort_flag, t);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            t = __shfl_sync(0xffffffffu, t, 0);
            sslot = __shfl_sync(0xffffffffu, sslot, 0);
            sph = __shfl_sync(0xffffffffu, sph, 0);
            return ok;
        };
        // this warp's 32 rows of tile t: first output row, or -1 when it has none
        auto warp_row0 = [&](const PairCoord& c) -> int {
            const int my_mt = c.mt + (int)rank;
            const int y0 = my_mt * BM + 32 * q;
            return ((my_mt - p.mt_base) < cnt && y0 < p.M) ? y0 : -1;
        };
        auto nchunks = [&](const PairCoord& c) -> int {
            const int left = p.N - c.nt * BN - cbase;
            return left <= 0 ? 0 : (left >= BN / 2 ? BN / 64 : (left + 31) / 32);
        };
        // request tile t's W boxes (32 x 32 bf16 each) into set `set`
        auto request = [&](int t, int set) -> int {
            const PairCoord c = pair_coord<BN>(p, t, cnt);
            const int y0 = warp_row0(c);
            const int n = y0 < 0 ? 0 : nchunks(c);
            if (n > 0) pend |= 1u << set;
            if (n > 0 && lane == 0) {
                const uint32_t bar = wbar + 8u * (uint32_t)set;
                mbar_expect_tx(bar, (uint32_t)n * 2048u);
                for (int ch = 0; ch < n; ++ch)
                    tma_load_2d(stg + (uint32_t)set * SET + (uint32_t)ch * 2048u, &maps.D, bar,
                                c.nt * BN + cbase + 32 * ch, y0);
            }
            return n;
        };
        int t = -1;
        bool ok = take(t);
        int n_cur = (ok && t >= 0) ? request(t, 0) : 0;
        for (int i = 0; ok && t >= 0; ++i) {
            const int set = i & 1;
            int t_next = -1;
            if (!(ok = take(t_next))) break;
            int n_next = 0;
            if (t_next >= 0) {
                // the other set held tile i-1, whose stores must have read it
                if (lane == 0) bulk_wait_read<0>();
                __syncwarp();
                n_next = request(t_next, set ^ 1);
            }
            if (lane == 0) ok = mbar_wait(bar_tfull + 8 * acc, acc_phase, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            tc_fence_after();
            if (n_cur > 0) {
                const PairCoord c = pair_coord<BN>(p, t, cnt);
                const int y0 = warp_row0(c);
                if (lane == 0) ok = mbar_wait(wbar + 8u * (uint32_t)set, (wph >> set) & 1u, abort_flag);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                wph ^= 1u << set;
                pend &= ~(1u << set);
                const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN + cbase);
                merge_tile(tbase, stg + (uint32_t)set * SET, lane, n_cur, gm);
                fence_async_shared();
                __syncwarp();
                if (lane == 0) {
                    const uint64_t pol = l2_policy_evict_first();
                    for (int ch = 0; ch < n_cur; ++ch)
                        tma_store_2d_hint(&maps.C, stg + (uint32_t)set * SET + (uint32_t)ch * 2048u,
                                          c.nt * BN + cbase + 32 * ch, y0, pol);
                    bulk_commit();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive(bar_tempty + 8 * acc);
                else mbar_arrive_cluster(tempty_leader + 8 * acc);
            }
            if (++acc == NUM_ACC) { acc = 0; acc_phase ^= 1u; }
            t = t_next;
            n_cur = n_next;
        }
        if (!ok && lane == 0) { atomicOr(status, ST_TIMEOUT); *abort_flag = 1; }
        if (lane == 0) {
            // W loads still in flight land before the CTA exits (bounded), stores are written
            for (int set = 0; set < 2; ++set)
                if (pend & (1u << set)) {
                    int dummy = 0;
                    if (!mbar_wait(wbar + 8u * (uint32_t)set, (wph >> set) & 1u, (volatile int*)&dummy))
                        atomicOr(status, ST_TIMEOUT);
                }
            bulk_wait_all();
        }
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const uint32_t stg = sbase + SL::STG_OFF + (uint32_t)(warp - 2) * (uint32_t)SL::STG_WARP;
        uint32_t nbox = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        int sslot = 0;
        uint32_t sph = 0;
        for (;;) {
            int t = -1;
            bool ok = true;
            if (lane == 0) ok = sched_take(bar_sfull, sempty_leader, slots, sslot, sph, leader, abort_flag, t);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            t = __shfl_sync(0xffffffffu, t, 0);
            sslot = __shfl_sync(0xffffffffu, sslot, 0);
            sph = __shfl_sync(0xffffffffu, sph, 0);
            if (!ok) {
                if (lane == 0) { atomicOr(status, ST_TIMEOUT); *abort_flag = 1; }
                break;
            }
            if (t < 0) break;
            const PairCoord c = pair_coord<BN>(p, t, cnt);
            if (lane == 0) ok = mbar_wait(bar_tfull + 8 * acc, acc_phase, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                if (lane == 0) { atomicOr(status, ST_TIMEOUT); *abort_flag = 1; }
                break;
            }
            tc_fence_after();
            const int my_mt = c.mt + (int)rank;
            const int64_t row = (int64_t)my_mt * BM + 32 * q + lane;
            const bool tile_ok = (my_mt - p.mt_base) < cnt && row < p.M;
            const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN);
            if constexpr (MERGE) {
                epilogue_row_merge<BN>(p, tbase, row, tile_ok, c.nt * BN, rank ? c.a1 : c.a0);
            } else if constexpr (SK != SK_NONE) {
                epilogue_row_staged<BN, SK>(p, &maps.C, &maps.D, tbase, row, tile_ok, c.nt * BN, c.nt, stg, nbox,
                                            (int)((int64_t)my_mt * BM + 32 * q + p.ep.out_row_shift));
            } else {
                epilogue_row<BN>(p, tbase, row, tile_ok, c.nt * BN, rank ? c.a1 : c.a0, c.nt);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive(bar_tempty + 8 * acc);
                else mbar_arrive_cluster(tempty_leader + 8 * acc);
            }
            if (++acc == NUM_ACC) { acc = 0; acc_phase ^= 1u; }
        }
        if (SK != SK_NONE && lane == 0) bulk_wait_all();   // staged stores written before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// ---- host ------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool get_encode() {
    if (g_encode) return true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        return false;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return true;
}

bool encode_2d(CUtensorMap* m, const GemmOperand& op, uint32_t box_cols, uint32_t box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)op.cols, (cuuint64_t)op.rows};
    cuuint64_t strides[1] = {(cuuint64_t)op.ld * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(op.ptr), dims, strides,
                          box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool operand_ok(const GemmOperand& op) {
    // TMA: 16-byte aligned base, row pitch a multiple of 16 bytes.
    return op.ptr && (reinterpret_cast<uintptr_t>(op.ptr) % 16 == 0) && (op.ld % 8 == 0) && op.rows > 0 &&
           op.cols > 0 && op.rows < (1LL << 31) && op.cols < (1LL << 31);
}

template <int BN, int STAGES, bool MERGE = false, int SUB = 1>
cudaError_t launch_bn(const GemmParams& p, cudaStream_t s, int num_sms, int* status) {
    using SL = SmemLayout<BN, STAGES, SUB>;
    TcMaps maps;
    auto enc = [&](CUtensorMap* m, const GemmOperand& op, int rows_mn) -> bool {
        if (!operand_ok(op)) return false;
        if (op.mn_major) return encode_2d(m, op, 64, 64);
        return encode_2d(m, op, 64, (uint32_t)rows_mn);
    };
    if (!enc(&maps.A, p.A, BM) || !enc(&maps.B, p.B, BN)) return cudaErrorInvalidValue;
    if (p.Kx > 0) {
        if (p.Kx % BK || !enc(&maps.Ax, p.Ax, BM) || !enc(&maps.Bx, p.Bx, BN)) return cudaErrorInvalidValue;
    } else {
        maps.Ax = maps.A;
        maps.Bx = maps.B;
    }
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<BN, STAGES, MERGE, SUB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SL::TOTAL);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int n_nt = (p.N + BN - 1) / BN;
    int64_t upper = p.grouped ? (int64_t)p.max_chunks * ((p.M + BM - 1) / BM) * n_nt
                              : (int64_t)p.mt_count * n_nt;
    if (upper <= 0) return cudaSuccess;
    int grid = (int)(upper < num_sms ? upper : num_sms);
    tc_gemm_kernel<BN, STAGES, MERGE, SUB><<<grid, NUM_THREADS, SL::TOTAL, s>>>(maps, p, status);
    return cudaGetLastError();
}

// Tensor map of a staged-store output: [rows x cols] of fp32 (esize 4, 128-byte
// swizzle) or bf16 (esize 2, 64-byte swizzle), row pitch ld elements, 32 x 32
// boxes.  TMA stores need a 16-byte aligned base and pitch.
bool encode_out(CUtensorMap* m, void* ptr, int64_t rows, int64_t cols, int64_t ld, int esize, bool half = false) {
    if (!ptr || reinterpret_cast<uintptr_t>(ptr) % 16 || (ld * esize) % 16 || rows <= 0 || cols <= 0 ||
        rows >= (1LL << 31) || cols >= (1LL << 31))
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * esize)};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t es[2] = {1, 1};
    const CUtensorMapDataType dt = esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : (half ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    CUresult r = g_encode(m, dt, 2,
                          ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          esize == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool out_aligned(const void* ptr, int64_t ld, int esize) {
    return ptr && reinterpret_cast<uintptr_t>(ptr) % 16 == 0 && (ld * esize) % 16 == 0;
}

// The staged-store kind of a CTA-pair launch, or SK_NONE: whole row tiles
// (M a multiple of 128) and outputs a TMA store can address.
int staged_kind(const GemmParams& p) {
    if (p.M % BM) return SK_NONE;
    const EpiParams& e = p.ep;
    switch (e.kind) {
    case EPI_LMFWD:
        return e.out0 && e.e16 && e.out_rows > 0 && out_aligned(e.out0, e.ld0, 2) ? SK_LMFWD : SK_NONE;
    case EPI_LMDZ:
        return e.out_rows > 0 && out_aligned(e.out0, e.ld0, 2) ? SK_LMDZ : SK_NONE;
    case EPI_SILU:
        return out_aligned(e.out0, e.ld0, 2) && out_aligned(e.out1, e.ld1, 2) ? SK_SILU : SK_NONE;
    case EPI_DSILU:
        return out_aligned(e.out0, e.ld0, 2) ? SK_DSILU : SK_NONE;
    case EPI_RESID:
        return out_aligned(e.f32, e.ldf, 4) && (!e.out0 || out_aligned(e.out0, e.ld0, 2)) ? SK_RESID : SK_NONE;
    default:
        return SK_NONE;
    }
}

// The export merge's staged form: whole 32-row warp slices (M a multiple of
// 32), W and the output addressable by TMA, one adapter for every tile.
bool merge_staged(const GemmParams& p) {
    const EpiParams& e = p.ep;
    return p.M % 32 == 0 && !p.tile_ad && out_aligned(e.aux, e.ld_aux, 2) && out_aligned(e.out0, e.ld0, 2);
}

// Output maps of a staged kind (the box layouts of staged_chunk).
template <int SK>
bool encode_staged(TcMaps& maps, const GemmParams& p) {
    const EpiParams& e = p.ep;
    switch (SK) {
    case SK_LMFWD:
        return encode_out(&maps.C, e.out0, e.out_rows, e.Vpad, e.ld0, 2, true);
    case SK_LMDZ:
        return encode_out(&maps.C, e.out0, e.out_rows, e.Vpad, e.ld0, 2);
    case SK_SILU:
        return encode_out(&maps.C, e.out0, p.M, p.N, e.ld0, 2) && encode_out(&maps.D, e.out1, p.M, p.N, e.ld1, 2);
    case SK_DSILU:
        return encode_out(&maps.C, e.out0, p.M, p.N, e.ld0, 2);
    case SK_RESID:
        if (!encode_out(&maps.D, e.f32, p.M, p.N, e.ldf, 4)) return false;
        if (e.out0) return encode_out(&maps.C, e.out0, p.M, p.N, e.ld0, 2);
        maps.C = maps.D;
        return true;
    case SK_MERGE:
        return encode_out(&maps.D, const_cast<void*>(e.aux), p.M, p.N, e.ld_aux, 2) &&
               encode_out(&maps.C, e.out0, p.M, p.N, e.ld0, 2);
    default:
        return true;
    }
}

template <int BN, int STAGES, int NUM_ACC, int SUB, bool MERGE = false, int SK = SK_NONE>
cudaError_t launch_pair(const GemmParams& p, cudaStream_t s, int num_sms, int* status, int* dbg) {
    using SL = SmemLayoutPair<BN, STAGES, NUM_ACC, SUB, SK>;
    TcMaps maps;
    auto enc = [&](CUtensorMap* m, const GemmOperand& op, int rows_mn) -> bool {
        if (!operand_ok(op)) return false;
        if (op.mn_major) return encode_2d(m, op, 64, 64);
        return encode_2d(m, op, 64, (uint32_t)rows_mn);
    };
    constexpr int BN_MMA = BN > 256 ? 256 : BN;
    if (p.grouped || p.B.ad_rows != 0 || p.A.mn_major || !p.tile_counter) return cudaErrorInvalidValue;
    if (BN > 256 && p.Kx > 0) return cudaErrorInvalidValue;    // wide tiles carry no K extension
    if (!enc(&maps.A, p.A, BM) || !enc(&maps.B, p.B, BN_MMA / 2)) return cudaErrorInvalidValue;
    if (p.Kx > 0) {
        if (p.Kx % BK || p.Ax.mn_major || !enc(&maps.Ax, p.Ax, BM) || !enc(&maps.Bx, p.Bx, BN / 2))
            return cudaErrorInvalidValue;
    } else {
        maps.Ax = maps.A;
        maps.Bx = maps.B;
    }
    if (SK != SK_NONE) {
        // the staged-store epilogue writes whole 32-row boxes: whole row tiles
        // (32-row warp slices for the merge), and the lowest output row
        // (mt_base's first row) may not be negative
        if (p.M % (SK == SK_MERGE ? 32 : BM) || (int64_t)p.mt_base * BM + p.ep.out_row_shift < 0 ||
            !encode_staged<SK>(maps, p))
            return cudaErrorInvalidValue;
    } else {
        maps.C = maps.A;
        maps.D = maps.A;
    }
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(tc_gemm_pair_kernel<BN, STAGES, NUM_ACC, SUB, MERGE, SK>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SL::TOTAL);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int n_nt = (p.N + BN - 1) / BN;
    const int64_t upper = (int64_t)((p.mt_count + 1) / 2) * n_nt;
    if (upper <= 0) return cudaSuccess;
    int nclusters = num_sms / 2;
    if (upper < nclusters) nclusters = (int)upper;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * nclusters, 1, 1);
    cfg.blockDim = dim3(pair_threads<SK>(), 1, 1);
    cfg.dynamicSmemBytes = SL::TOTAL;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaMemsetAsync(p.tile_counter, 0, sizeof(int), s);   // fresh tile counter
    if (e != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, tc_gemm_pair_kernel<BN, STAGES, NUM_ACC, SUB, MERGE, SK>, maps, p, status, dbg);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

// CTA-pair variants (exposed for the engine's own checks): acc_buffers = 1 or 2
// with one 64-wide K block per stage; 3 = the engine's configuration (two
// accumulators, two K blocks per stage).
cudaError_t launch_tc_gemm_pair(const GemmParams& p, cudaStream_t s, int num_sms, int* status,
                                int acc_buffers, int* dbg) {
    if (!get_encode()) return cudaErrorNotSupported;
    if (p.N < 256) return cudaErrorInvalidValue;
    if (acc_buffers == 1) return launch_pair<256, 6, 1, 1>(p, s, num_sms, status, dbg);
    if (acc_buffers == 2) return launch_pair<256, 6, 2, 1>(p, s, num_sms, status, dbg);
    return launch_pair<256, 3, 2, 2>(p, s, num_sms, status, dbg);
}

bool tc_engine_available() { return get_encode(); }

bool tc_encode_bf16(void* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, uint32_t box_cols,
                    uint32_t box_rows) {
    if (!get_encode()) return false;
    GemmOperand op;
    op.ptr = ptr; op.rows = rows; op.cols = cols; op.ld = ld;
    if (!operand_ok(op)) return false;
    return encode_2d(reinterpret_cast<CUtensorMap*>(map), op, box_cols, box_rows);
}

cudaError_t launch_tc_gemm(const GemmParams& p, cudaStream_t s, int num_sms, int* status) {
    if (!get_encode()) return cudaErrorNotSupported;
    if (p.ep.kind == EPI_MERGE) {
        if (p.N <= 64 || p.force_bn64) return launch_bn<64, 8, true>(p, s, num_sms, status);
        if (!p.grouped && p.B.ad_rows == 0 && !p.A.mn_major && p.N >= 256 && p.tile_counter) {
            // K is a few blocks: one-block stages, and W requested a tile ahead
            if (merge_staged(p)) return launch_pair<256, 3, 2, 1, false, SK_MERGE>(p, s, num_sms, status, nullptr);
            return launch_pair<256, 3, 2, 2, true>(p, s, num_sms, status, nullptr);
        }
        return launch_bn<256, 4, true>(p, s, num_sms, status);
    }
    // 128 x 64 tiles: three stages of three K blocks (216 KB in flight; decode
    // 1.11 ms against 1.18 with four stages of two and 1.36 with eight of one)
    if (p.N <= 64 || p.force_bn64) return launch_bn<64, 3, false, 3>(p, s, num_sms, status);
    // a very long contraction (the LM head's dh, K = the vocabulary): 256 x 512
    // tiles, so the 76 clusters' tiles in flight read the A band about half as
    // often; one accumulator, whose unhidden epilogue is ~1 % of a tile here.
    // Bands of 12 row pairs: 76 tiles in flight cover ~6 of a band's 8 column
    // tiles, which balances the re-reads of A (per column tile not in flight)
    // against those of B (per band).
    if (!p.grouped && p.B.ad_rows == 0 && !p.A.mn_major && p.K >= 65536 && p.Kx == 0 && p.N % 512 == 0 &&
        p.tile_counter) {
        GemmParams q = p;
        q.group_m = 24;
        return launch_pair<512, 4, 1, 1>(q, s, num_sms, status, nullptr);
    }
    // main B shared by every row: 256 x 256 tiles on CTA pairs (the per-adapter
    // K extension, if any, is split per row half inside the kernel)
    if (!p.grouped && p.B.ad_rows == 0 && !p.A.mn_major && p.N >= 256 && p.tile_counter) {
        // outputs leave through shared memory and TMA stores where they can
        switch (staged_kind(p)) {
        case SK_LMFWD: return launch_pair<256, 3, 2, 2, false, SK_LMFWD>(p, s, num_sms, status, nullptr);
        case SK_LMDZ: return launch_pair<256, 3, 2, 2, false, SK_LMDZ>(p, s, num_sms, status, nullptr);
        case SK_SILU: return launch_pair<256, 3, 2, 2, false, SK_SILU>(p, s, num_sms, status, nullptr);
        case SK_DSILU: return launch_pair<256, 3, 2, 2, false, SK_DSILU>(p, s, num_sms, status, nullptr);
        case SK_RESID: return launch_pair<256, 3, 2, 2, false, SK_RESID>(p, s, num_sms, status, nullptr);
        default: return launch_pair<256, 3, 2, 2>(p, s, num_sms, status, nullptr);
        }
    }
    return launch_bn<256, 4>(p, s, num_sms, status);
}

}  // namespace mlk
