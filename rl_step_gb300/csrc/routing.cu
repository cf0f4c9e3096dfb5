// Token routing: a stable counting sort of token positions by adapter id
// (tinker-ticks, "How the SGMV kernel works": the flattened token matrix
// carries segment indices recording which adapter owns each row).
//
// Output layout: every adapter's segment is padded to a multiple of TILE_M
// rows ("padded order"), so each 128-row GEMM tile belongs to exactly one
// adapter.  perm_pad[p] is the batch position of padded row p, or -1 for a
// padding row.  The same pass emits the per-tile adapter map and the list of
// gradient work chunks (at most chunk_rows padded rows of one adapter each;
// chunk_rows == 0 makes each adapter's whole padded segment one chunk, so
// its gradient reduction runs in one fixed order with one writer per
// element: the deterministic mode).
//
// Three launches, all on the caller's stream, no host synchronisation:
//   route_count    per 1024-token block, per-adapter counts
//   route_scan     one CTA: exclusive prefixes over blocks and adapters,
//                  tile map, chunk list, touched flags
//   route_scatter  per block: stable in-block ranks (warps in order), final
//                  positions
#include "internal.h"

namespace mlk {

__global__ void route_count(const int* __restrict__ ids, int64_t n, int n_ad, int* blk_cnt,
                            int* status) {
    extern __shared__ int sh[];
    for (int a = threadIdx.x; a < n_ad; a += blockDim.x) sh[a] = 0;
    __syncthreads();
    int64_t t = (int64_t)blockIdx.x * ROUTE_BLOCK + threadIdx.x;
    if (t < n) {
        int a = ids[t];
        if (a >= 0 && a < n_ad) atomicAdd(&sh[a], 1);
        else raise_status(status, ST_RANGE);
    }
    __syncthreads();
    for (int a = threadIdx.x; a < n_ad; a += blockDim.x)
        blk_cnt[(int64_t)blockIdx.x * n_ad + a] = sh[a];
}

__global__ void route_scan(int nblk, int n_ad, int* blk_cnt, int* seg_off, int* pad_off,
                           int* tile_ad, int max_tiles, int* meta, int4* chunks, int max_chunks,
                           int chunk_rows, int* touched) {
    extern __shared__ int sh[];
    int* s_cnt = sh;             // [n_ad]
    int* s_pad = sh + n_ad;      // [n_ad + 1] padded offsets
    int* s_ch = sh + 2 * n_ad + 1;  // [n_ad + 1] chunk offsets
    for (int a = threadIdx.x; a < n_ad; a += blockDim.x) {
        int run = 0;
        for (int b = 0; b < nblk; ++b) {
            int64_t i = (int64_t)b * n_ad + a;
            int c = blk_cnt[i];
            blk_cnt[i] = run;
            run += c;
        }
        s_cnt[a] = run;
        if (touched && run > 0) touched[a] = 1;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int seg = 0, pad = 0, nch = 0;
        for (int a = 0; a < n_ad; ++a) {
            seg_off[a] = seg;
            pad_off[a] = pad;
            s_pad[a] = pad;
            s_ch[a] = nch;
            int c = s_cnt[a];
            int padded = (c + TILE_M - 1) / TILE_M * TILE_M;
            seg += c;
            pad += padded;
            nch += chunk_rows > 0 ? (padded + chunk_rows - 1) / chunk_rows : (padded > 0);
        }
        seg_off[n_ad] = seg;
        pad_off[n_ad] = pad;
        s_pad[n_ad] = pad;
        s_ch[n_ad] = nch;
        meta[0] = pad / TILE_M;
        meta[1] = nch;
    }
    __syncthreads();
    for (int a = threadIdx.x; a < n_ad; a += blockDim.x) {
        int t0 = s_pad[a] / TILE_M, t1 = s_pad[a + 1] / TILE_M;
        for (int j = t0; j < t1 && j < max_tiles; ++j) tile_ad[j] = a;
        int padded = s_pad[a + 1] - s_pad[a];
        const int step = chunk_rows > 0 ? chunk_rows : padded;
        const int nc = padded > 0 ? (padded + step - 1) / step : 0;
        for (int c = 0; c < nc; ++c) {
            int ci = s_ch[a] + c;
            if (ci < max_chunks)
                chunks[ci] = make_int4(a, s_pad[a] + c * step, min(step, padded - c * step), 0);
        }
    }
    for (int j = s_pad[n_ad] / TILE_M + threadIdx.x; j < max_tiles; j += blockDim.x) tile_ad[j] = -1;
}

__global__ void route_scatter(const int* __restrict__ ids, int64_t n, int n_ad,
                              const int* __restrict__ blk_base, const int* __restrict__ pad_off,
                              int* perm_pad, int* inv) {
    extern __shared__ int s_next[];
    for (int a = threadIdx.x; a < n_ad; a += blockDim.x)
        s_next[a] = pad_off[a] + blk_base[(int64_t)blockIdx.x * n_ad + a];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * ROUTE_BLOCK + threadIdx.x;
    const int a = (t < n) ? ids[t] : -1;
    const bool ok = (a >= 0 && a < n_ad);
    const int key = ok ? a : -1;
    for (int w = 0; w < ROUTE_BLOCK / 32; ++w) {
        if (warp == w) {
            unsigned peers = __match_any_sync(0xffffffffu, key);
            int base = ok ? s_next[a] : 0;
            __syncwarp();
            if (ok) {
                int rank = __popc(peers & ((1u << lane) - 1u));
                int pos = base + rank;
                perm_pad[pos] = (int)t;
                inv[t] = pos;
                if (lane == __ffs(peers) - 1) s_next[a] = base + __popc(peers);
            } else if (t < n) {
                inv[t] = -1;
            }
        }
        __syncthreads();
    }
}

void launch_routing(const int* adapter_ids, int64_t n, int n_ad, const RouteBufs& rb, int* touched,
                    int* status, cudaStream_t s, int64_t* launches, int chunk_rows) {
    int nblk = (int)((n + ROUTE_BLOCK - 1) / ROUTE_BLOCK);
    cudaMemsetAsync(rb.perm_pad, 0xff, sizeof(int) * (size_t)rb.max_pad, s);
    if (nblk > 0) {
        route_count<<<nblk, ROUTE_BLOCK, sizeof(int) * n_ad, s>>>(adapter_ids, n, n_ad, rb.blk_cnt,
                                                                 status);
        ++*launches;
    }
    route_scan<<<1, 1024, sizeof(int) * (3 * n_ad + 2), s>>>(
        nblk, n_ad, rb.blk_cnt, rb.seg_off, rb.pad_off, rb.tile_ad, rb.max_tiles, rb.meta, rb.chunks,
        rb.max_chunks, chunk_rows, touched);
    ++*launches;
    if (nblk > 0) {
        route_scatter<<<nblk, ROUTE_BLOCK, sizeof(int) * n_ad, s>>>(adapter_ids, n, n_ad, rb.blk_cnt,
                                                                   rb.pad_off, rb.perm_pad, rb.inv);
        ++*launches;
    }
}

__global__ void compact_perm_kernel(const int* perm_pad, const int* tile_ad, const int* seg_off,
                                    const int* pad_off, const int* meta, int* perm) {
    int rows = meta[0] * TILE_M;
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < rows; p += gridDim.x * blockDim.x) {
        int t = perm_pad[p];
        if (t < 0) continue;
        int a = tile_ad[p / TILE_M];
        perm[seg_off[a] + (p - pad_off[a])] = t;
    }
}

void launch_compact_perm(const RouteBufs& rb, int n_ad, int* perm_out, cudaStream_t s,
                         int64_t* launches) {
    (void)n_ad;
    int blocks = (rb.max_pad + 255) / 256;
    if (blocks < 1) blocks = 1;
    compact_perm_kernel<<<blocks, 256, 0, s>>>(rb.perm_pad, rb.tile_ad, rb.seg_off, rb.pad_off,
                                               rb.meta, perm_out);
    ++*launches;
}

}  // namespace mlk
