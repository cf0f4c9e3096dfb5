// Bandwidth-bound kernels of the step: embedding gather, the LM-head partial
// combine fused with the loss epilogue, the per-adapter loss reduction, and
// the fused Adam update.
#include <math.h>

#include "internal.h"

namespace mlk {

// ----------------------------------------------------------------------------
// embedding: h0[p] = E[x_{perm[p]}] in padded order; padding rows are zero.
// One warp per row, 16-byte accesses.
// ----------------------------------------------------------------------------
template <typename T>
__global__ void embed_kernel(const int* __restrict__ perm_pad, const int* __restrict__ meta,
                             const int* __restrict__ tokens, const int* __restrict__ targets,
                             const T* __restrict__ E, int V, int d, T* __restrict__ hb,
                             float* __restrict__ h32, int* __restrict__ tgt_pad, int* status) {
    const int rows = meta[0] * TILE_M;
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    for (int p = blockIdx.x * wpb + (threadIdx.x >> 5); p < rows; p += gridDim.x * wpb) {
        int t = perm_pad[p];
        int x = -1;
        if (t >= 0) {
            x = tokens[t];
            int y = targets[t];
            if (x < 0 || x >= V) { if (lane == 0) raise_status(status, ST_RANGE); x = -1; y = -1; }
            if (y < 0 || y >= V) { if (lane == 0) raise_status(status, ST_RANGE); y = -1; }
            if (lane == 0) tgt_pad[p] = y;
        } else if (lane == 0) {
            tgt_pad[p] = -1;
        }
        constexpr int VEC = 16 / sizeof(T);   // elements per 16 bytes
        for (int c = lane * VEC; c < d; c += 32 * VEC) {
            float v[VEC];
            if (x >= 0) {
                uint4 raw = *reinterpret_cast<const uint4*>(E + (int64_t)x * d + c);
                if constexpr (sizeof(T) == 2) {
                    const bf16* b = reinterpret_cast<const bf16*>(&raw);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) v[e] = __bfloat162float(b[e]);
                } else {
                    const float* f = reinterpret_cast<const float*>(&raw);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) v[e] = f[e];
                }
                *reinterpret_cast<uint4*>(hb + (int64_t)p * d + c) = raw;
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[e] = 0.f;
                *reinterpret_cast<uint4*>(hb + (int64_t)p * d + c) = make_uint4(0, 0, 0, 0);
            }
            float* hp = h32 + (int64_t)p * d + c;
#pragma unroll
            for (int e = 0; e < VEC; e += 4)
                *reinterpret_cast<float4*>(hp + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
    }
}

template <typename T>
void launch_embed(const int* perm_pad, const int* meta, int max_rows, const int* tokens,
                  const int* targets, const T* E, int V, int d, T* hb, float* h32, int* tgt_pad,
                  int* status, cudaStream_t s) {
    int blocks = (max_rows + 7) / 8;
    if (blocks > 65535) blocks = 65535;
    if (blocks < 1) blocks = 1;
    embed_kernel<T><<<blocks, 256, 0, s>>>(perm_pad, meta, tokens, targets, E, V, d, hb, h32,
                                           tgt_pad, status);
}
template void launch_embed<float>(const int*, const int*, int, const int*, const int*, const float*,
                                  int, int, float*, float*, int*, int*, cudaStream_t);
template void launch_embed<bf16>(const int*, const int*, int, const int*, const int*, const bf16*,
                                 int, int, bf16*, float*, int*, int*, cudaStream_t);

// ----------------------------------------------------------------------------
// LM-head combine + loss epilogue.
// For padded row p: lse = logsumexp_j(lse_j) over the log-sum-exp lse_j of
// each 256-column vocabulary tile; l = z[y] - lse (Tinker API Implementation
// on TPUs, section 10.3: the target logprob is a gather minus a logsumexp).
// Then the per-token loss value and g = dL/dl (Deep Dive - Tinker, "The RL
// datum shape"; custom: g is the caller's dC/dl), with non-finite inputs
// contained (Tinker API Implementation on TPUs, section 12).  Per-row loss
// values (fp64) are summed per adapter in row order: deterministic.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void token_loss_dev(int kind, float ell, int t, const LossArgs& la,
                                               double& val, float& g) {
    val = 0.0;
    g = 0.f;
    if (kind < 0) return;
    bool ok = isfinite(ell);
    if (kind == 0) {
        float w = la.w[t];
        ok = ok && isfinite(w);
        if (ok) { val = -(double)w * ell; g = -w; }
    } else if (kind == 1 || kind == 2) {
        float A = la.adv[t], sl = la.slp[t];
        ok = ok && isfinite(A) && isfinite(sl);
        if (ok) {
            float r = expf(ell - sl);
            ok = isfinite(r);
            if (ok) {
                float un = r * A;
                if (kind == 1) {
                    val = -(double)un;
                    g = -un;
                } else {
                    float rc = fminf(fmaxf(r, 1.f - la.clip), 1.f + la.clip);
                    float cl = rc * A;
                    val = -(double)fminf(un, cl);
                    g = (un <= cl) ? -un : 0.f;
                }
                ok = isfinite(val) && isfinite(g);
            }
        }
    } else {
        float c = la.dl[t];
        ok = ok && isfinite(c);
        if (ok) { val = (double)c * ell; g = c; }
    }
    if (!ok) { val = 0.0; g = 0.f; }
}

// Combine: each warp takes groups of G consecutive padded rows (G <= 32,
// chosen at launch so that the groups cover the GPU's warps).  For every row
// of the group the warp reads the row's partials (one log-sum-exp per
// 256-column vocabulary tile) with lane-strided 16-byte loads -- the next
// row's loads are issued before the current row is reduced -- and reduces
// them in a fixed order: the maximum over each lane's values and a butterfly
// maximum, then the sum of exp(x - m) over each lane's values and a butterfly
// sum.  Lane i keeps row i's (m, s); then every lane finishes its own row
// (target logprob, loss value, dL/dl) and the per-row stores are coalesced.
// part_ld (a multiple of 4) is the pitch of a row of partials, n_nt the
// number in use.  Per-row loss values go to val_row for a deterministic
// per-adapter reduction in row order.  The result of a row depends on that
// row alone (batch-invariant) and repeats bit for bit.
constexpr int COMBINE_VEC = 5;      // float4 per lane per row prefetched: 640 partials
constexpr int COMBINE_CTAS_PER_SM = 3;   // resident at 256 threads and <= 85 registers

struct CombineRow {
    float4 v[COMBINE_VEC];
    float tail;                     // partial 4 * 32 * COMBINE_VEC + lane, if any
};

__device__ __forceinline__ void combine_load(CombineRow& r, const float* __restrict__ part, int64_t p,
                                             int n_nt, int part_ld, int lane) {
    const float* rowp = part + p * part_ld;
    const float4* row4 = reinterpret_cast<const float4*>(rowp);
    const int nvec = n_nt >> 2;
#pragma unroll
    for (int u = 0; u < COMBINE_VEC; ++u) {
        const int j = lane + 32 * u;
        r.v[u] = j < nvec ? row4[j] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
    const int done = 4 * min(nvec, 32 * COMBINE_VEC);
    r.tail = done + lane < n_nt ? rowp[done + lane] : -INFINITY;
}

__global__ void __launch_bounds__(256, COMBINE_CTAS_PER_SM) combine_loss_kernel(
    LossArgs la, const float* __restrict__ part, int n_nt, int part_ld, const float* __restrict__ zt,
    const int* __restrict__ perm_pad, const int* __restrict__ tgt_pad, const int* __restrict__ meta,
    int row0, int row1, int G, float* logprobs_out, float* lse_out, float* g_out, double* val_row) {
    const int rows = min(meta[0] * TILE_M, row1);
    const int lane = threadIdx.x & 31;
    const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    // partials past the prefetched float4 groups and the one tail value per lane
    const int beyond = 4 * min(n_nt >> 2, 32 * COMBINE_VEC) + 32;
    for (int g0 = row0 + G * wid; g0 < rows; g0 += G * nwarps) {
        const int gn = min(G, rows - g0);
        float my_m = -INFINITY, my_s = 0.f;
        CombineRow cur, nxt;
        combine_load(cur, part, g0, n_nt, part_ld, lane);
        for (int i = 0; i < gn; ++i) {
            const int64_t p = g0 + i;
            if (i + 1 < gn) combine_load(nxt, part, p + 1, n_nt, part_ld, lane);
            float m = cur.tail;
#pragma unroll
            for (int u = 0; u < COMBINE_VEC; ++u)
                m = fmaxf(fmaxf(m, fmaxf(cur.v[u].x, cur.v[u].y)), fmaxf(cur.v[u].z, cur.v[u].w));
            for (int j = beyond + lane; j < n_nt; j += 32) m = fmaxf(m, part[p * part_ld + j]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            float sm = 0.f;
            if (m > -INFINITY) {
                sm = __expf(cur.tail - m);
#pragma unroll
                for (int u = 0; u < COMBINE_VEC; ++u)
                    sm += (__expf(cur.v[u].x - m) + __expf(cur.v[u].y - m)) +
                          (__expf(cur.v[u].z - m) + __expf(cur.v[u].w - m));
                for (int j = beyond + lane; j < n_nt; j += 32) sm += __expf(part[p * part_ld + j] - m);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
            if (lane == i) { my_m = m; my_s = sm; }
            cur = nxt;
        }
        if (lane < gn) {
            const int p = g0 + lane;
            const int t = perm_pad[p];
            const int y = tgt_pad[p];
            double val = 0.0;
            float g = 0.f, lse = 0.f;
            if (t >= 0) {
                float ell;
                if (y >= 0) {
                    lse = my_m + __logf(my_s);
                    ell = zt[p] - lse;
                } else {
                    ell = __int_as_float(0x7fc00000);   // NaN: invalid token or target
                }
                token_loss_dev(la.kind, ell, t, la, val, g);
                if (y < 0) g = 0.f, val = 0.0;
                if (logprobs_out) logprobs_out[t] = ell;
            }
            lse_out[p] = lse;
            g_out[p] = g;
            val_row[p] = val;
        }
    }
}

void launch_combine_loss(const LossArgs& la, const float* part, int n_nt, int part_ld, const float* zt,
                         const int* perm_pad, const int* tgt_pad, const int* meta, int tile0, int ntiles,
                         float* logprobs_out, float* lse, float* g, double* val_row, int num_sms,
                         cudaStream_t s) {
    if (ntiles <= 0) return;
    const int rows = ntiles * TILE_M;
    const int warps = num_sms * COMBINE_CTAS_PER_SM * 8;
    int G = rows / warps;                 // rows per group: 1 .. 32
    if (G < 1) G = 1;
    if (G > 32) G = 32;
    int blocks = num_sms * COMBINE_CTAS_PER_SM;
    const int need = ((rows + G - 1) / G + 7) / 8;   // one group per warp at most
    if (blocks > need) blocks = need;
    combine_loss_kernel<<<blocks, 256, 0, s>>>(la, part, n_nt, part_ld, zt, perm_pad, tgt_pad, meta,
                                               tile0 * TILE_M, (tile0 + ntiles) * TILE_M, G,
                                               logprobs_out, lse, g, val_row);
}

// ----------------------------------------------------------------------------
// LM-head backward from stored logits, for the padded rows [row0, row0 + nrows)
// of one chunk (z and dz hold the chunk's rows, pitch ld):
//   dz[r][v] = g (onehot(v == y) - exp(z[r][v] - lse))   for v < V
//   dz[r][v] = 0                                          for V <= v < Vpad
// with g = dL/dl, lse and y of padded row row0 + r.  Rows with g = 0 (padding,
// masked or invalid tokens) are written as zeros without reading z.  Each
// thread covers 16 consecutive columns: four 16-byte loads in flight, one
// (bf16) or four (fp32) 16-byte stores.  Rows at or past the batch's valid
// m-tiles are skipped (the dh GEMM does not read them).
// ----------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ void store16(T* dst, const float* v);
template <> __device__ __forceinline__ void store16<bf16>(bf16* dst, const float* v) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 2; ++q)
        d4[q] = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                           pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
}
template <> __device__ __forceinline__ void store16<float>(float* dst, const float* v) {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

template <typename T>
__global__ void __launch_bounds__(256) lm_dz_kernel(const float* __restrict__ z, T* __restrict__ dz,
                                                    int64_t ld, int V, int Vpad, const float* __restrict__ g,
                                                    const float* __restrict__ lse,
                                                    const int* __restrict__ tgt, const int* __restrict__ meta,
                                                    int row0, int nrows) {
    const float LOG2E = 1.4426950408889634f;
    const int r = blockIdx.y;
    const int p = row0 + r;
    if (r >= nrows || p >= meta[0] * TILE_M) return;
    const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 16;
    if (c >= Vpad) return;
    const float gr = g[p];
    float d[16];
    if (gr == 0.f) {
#pragma unroll
        for (int j = 0; j < 16; ++j) d[j] = 0.f;
    } else {
        const float4* zp = reinterpret_cast<const float4*>(z + (int64_t)r * ld + c);
        float4 q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) q[u] = __ldcs(zp + u);
        const float lb = lse[p] * LOG2E;
        const int y = tgt[p];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float zz[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int v = c + 4 * u + e;
                const float pr = exp2f(fmaf(zz[e], LOG2E, -lb));
                d[4 * u + e] = v < V ? gr * ((v == y ? 1.f : 0.f) - pr) : 0.f;
            }
        }
    }
    store16<T>(dz + (int64_t)r * ld + c, d);
}

template <typename T>
void launch_lm_dz(const float* z, T* dz, int64_t ld, int V, int Vpad, const float* g, const float* lse,
                  const int* tgt, const int* meta, int row0, int nrows, cudaStream_t s) {
    if (nrows <= 0) return;
    dim3 grid((unsigned)((Vpad / 16 + 255) / 256), (unsigned)nrows);
    lm_dz_kernel<T><<<grid, 256, 0, s>>>(z, dz, ld, V, Vpad, g, lse, tgt, meta, row0, nrows);
}
template void launch_lm_dz<float>(const float*, float*, int64_t, int, int, const float*, const float*,
                                  const int*, const int*, int, int, cudaStream_t);
template void launch_lm_dz<bf16>(const float*, bf16*, int64_t, int, int, const float*, const float*,
                                 const int*, const int*, int, int, cudaStream_t);

// dz of the bf16 engine's kept-logits LM-head backward from the kept fp16
// e = exp(z - m) and the rows' tile maxima m: dz = g (onehot - e exp(m - lse)),
// 16 columns per thread (a partial tile holds whole groups of 16).  The
// recompute epilogue (lmdz_values<true>) forms the same values.
__global__ void __launch_bounds__(256) lm_dz_e16_kernel(const __half* __restrict__ e, bf16* __restrict__ dz,
                                                        int64_t ld, int V, int Vpad, const float* __restrict__ mt,
                                                        int part_ld, int lm_bn, const float* __restrict__ g,
                                                        const float* __restrict__ lse, const int* __restrict__ tgt,
                                                        const int* __restrict__ meta, int row0, int nrows) {
    const int r = blockIdx.y;
    const int p = row0 + r;
    if (r >= nrows || p >= meta[0] * TILE_M) return;
    const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 16;
    if (c >= Vpad) return;
    const float gr = g[p];
    float d[16];
    if (gr == 0.f) {
#pragma unroll
        for (int j = 0; j < 16; ++j) d[j] = 0.f;
    } else {
        const uint4* ep = reinterpret_cast<const uint4*>(e + (int64_t)r * ld + c);
        const uint4 q0 = __ldcs(ep), q1 = __ldcs(ep + 1);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const int nt_last = (V - 1) / lm_bn;
        const int nt = c / lm_bn < nt_last ? c / lm_bn : nt_last;   // columns >= V give 0 below
        const float cc = lm_tile_scale(mt[(int64_t)p * part_ld + nt], lse[p]);
        const int y = tgt[p];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[u]));
            const int v = c + 2 * u;
            d[2 * u] = v < V ? lm_dz_from_e(gr, v == y, f.x, cc) : 0.f;
            d[2 * u + 1] = v + 1 < V ? lm_dz_from_e(gr, v + 1 == y, f.y, cc) : 0.f;
        }
    }
    store16<bf16>(dz + (int64_t)r * ld + c, d);
}

void launch_lm_dz_e16(const __half* e, bf16* dz, int64_t ld, int V, int Vpad, const float* mt, int part_ld,
                      int lm_bn, const float* g, const float* lse, const int* tgt, const int* meta, int row0,
                      int nrows, cudaStream_t s) {
    if (nrows <= 0) return;
    dim3 grid((unsigned)((Vpad / 16 + 255) / 256), (unsigned)nrows);
    lm_dz_e16_kernel<<<grid, 256, 0, s>>>(e, dz, ld, V, Vpad, mt, part_ld, lm_bn, g, lse, tgt, meta, row0, nrows);
}

// Per-adapter loss: sum of its rows' loss values, in row order.
__global__ void loss_reduce_kernel(const double* val_row, const int* pad_off, int n_ad, double* loss_out) {
    const int a = blockIdx.x;
    if (a >= n_ad) return;
    __shared__ double sh[256];
    double s = 0.0;
    for (int j = pad_off[a] + threadIdx.x; j < pad_off[a + 1]; j += blockDim.x) s += val_row[j];
    sh[threadIdx.x] = s;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if (threadIdx.x < o) sh[threadIdx.x] += sh[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) loss_out[a] = sh[0];
}

void launch_loss_reduce(const double* val_row, const int* pad_off, int n_ad, double* loss_out,
                        cudaStream_t s) {
    loss_reduce_kernel<<<n_ad, 256, 0, s>>>(val_row, pad_off, n_ad, loss_out);
}

// ----------------------------------------------------------------------------
// Adam.  Parameters of adapter a occupy [ad_off[a], ad_off[a+1]) of the fp32
// buffers P, G, M, V; inside, layer l holds A1 [r x d], B1 [f x r], A2 [r x f],
// B2 [d x r].  The same element is mirrored into the padded-rank copies used
// by the GEMMs:  A1 -> A1s[l][(a*RP + j)*d + i],  B1 -> B1s[l][(a*f + i)*RP + j],
//                A2 -> A2s[l][(a*RP + j)*f + i],  B2 -> B2s[l][(a*d + i)*RP + j].
// ----------------------------------------------------------------------------
__global__ void adam_prep_kernel(int n_ad, const int* sel_mask, int* touched, int* nonfinite,
                                 int64_t* step, float beta1, float beta2, AdamTab* tab,
                                 int* skipped_out) {
    for (int a = threadIdx.x; a < n_ad; a += blockDim.x) {
        bool sel = sel_mask ? (sel_mask[a] != 0) : (touched[a] != 0);
        AdamTab e;
        e.mode = 0;
        e.c1 = e.c2 = 0.f;
        int skipped = 0;
        if (sel) {
            if (nonfinite[a]) {
                e.mode = 2;
                skipped = 1;
            } else {
                int64_t t = step[a] + 1;
                step[a] = t;
                e.mode = 1;
                e.c1 = (float)(1.0 / (1.0 - pow((double)beta1, (double)t)));
                e.c2 = (float)(1.0 / (1.0 - pow((double)beta2, (double)t)));
            }
            touched[a] = 0;
            nonfinite[a] = 0;
        }
        tab[a] = e;
        if (skipped_out) skipped_out[a] = skipped;
    }
}

void launch_adam_prep(int n_ad, const int* sel_mask, int* touched, int* nonfinite, int64_t* step,
                      float beta1, float beta2, AdamTab* tab, int* skipped_out, cudaStream_t s) {
    adam_prep_kernel<<<1, 1024, 0, s>>>(n_ad, sel_mask, touched, nonfinite, step, beta1, beta2, tab,
                                        skipped_out);
}

__device__ __forceinline__ int find_adapter(const int64_t* off, int n_ad, int64_t i) {
    int lo = 0, hi = n_ad - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= i) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// element index (inside adapter a) -> padded copy pointer offset
template <typename T>
__device__ __forceinline__ T* shadow_ptr(const ShadowMap& sh, int a, int r, int d, int f, int64_t rel) {
    const int64_t per_layer = 2LL * r * (d + f);
    const int l = (int)(rel / per_layer);
    int64_t q = rel - (int64_t)l * per_layer;
    const int64_t nA1 = (int64_t)r * d, nB1 = (int64_t)f * r, nA2 = (int64_t)r * f;
    if (q < nA1) {
        int64_t j = q / d, i = q % d;
        return reinterpret_cast<T*>(sh.A1[l]) + ((int64_t)a * RP + j) * d + i;
    }
    q -= nA1;
    if (q < nB1) {
        int64_t i = q / r, j = q % r;
        return reinterpret_cast<T*>(sh.B1[l]) + ((int64_t)a * f + i) * RP + j;
    }
    q -= nB1;
    if (q < nA2) {
        int64_t j = q / f, i = q % f;
        return reinterpret_cast<T*>(sh.A2[l]) + ((int64_t)a * RP + j) * f + i;
    }
    q -= nA2;
    int64_t i = q / r, j = q % r;
    return reinterpret_cast<T*>(sh.B2[l]) + ((int64_t)a * d + i) * RP + j;
}

template <typename T>
__device__ __forceinline__ void store4(T* dst, float4 v);
template <> __device__ __forceinline__ void store4<float>(float* dst, float4 v) {
    *reinterpret_cast<float4*>(dst) = v;
}
template <> __device__ __forceinline__ void store4<bf16>(bf16* dst, float4 v) {
    uint2 w;
    w.x = pack_bf16x2(v.x, v.y);
    w.y = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2*>(dst) = w;
}

template <typename T>
__global__ void __launch_bounds__(256) adam_kernel(int n_ad, const int64_t* __restrict__ ad_off,
                                                   const int* __restrict__ ranks, int d, int f,
                                                   int64_t total4, const AdamTab* __restrict__ tab,
                                                   float4* P, float4* G, float4* M, float4* Vm,
                                                   float lr, float b1, float b2, float eps, float wd,
                                                   ShadowMap sh) {
    __shared__ int64_t s_off[1025];
    for (int a = threadIdx.x; a <= n_ad; a += blockDim.x) s_off[a] = ad_off[a];
    __syncthreads();
    for (int64_t i4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i4 < total4;
         i4 += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = i4 * 4;
        const int a = find_adapter(s_off, n_ad, i);
        const AdamTab e = tab[a];
        if (e.mode == 0) continue;
        if (e.mode == 2) {
            G[i4] = make_float4(0.f, 0.f, 0.f, 0.f);
            continue;
        }
        float4 g = G[i4], p = P[i4], m = M[i4], v = Vm[i4];
        float gv[4] = {g.x, g.y, g.z, g.w};
        float pv[4] = {p.x, p.y, p.z, p.w};
        float mv[4] = {m.x, m.y, m.z, m.w};
        float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            mv[q] = b1 * mv[q] + (1.f - b1) * gv[q];
            vv[q] = b2 * vv[q] + (1.f - b2) * gv[q] * gv[q];
            float mh = mv[q] * e.c1;
            float vh = vv[q] * e.c2;
            pv[q] = pv[q] - lr * (mh / (sqrtf(vh) + eps) + wd * pv[q]);
        }
        float4 pn = make_float4(pv[0], pv[1], pv[2], pv[3]);
        P[i4] = pn;
        M[i4] = make_float4(mv[0], mv[1], mv[2], mv[3]);
        Vm[i4] = make_float4(vv[0], vv[1], vv[2], vv[3]);
        G[i4] = make_float4(0.f, 0.f, 0.f, 0.f);
        store4<T>(shadow_ptr<T>(sh, a, ranks[a], d, f, i - s_off[a]), pn);
    }
}

template <typename T>
void launch_adam(int n_ad, const int64_t* ad_off, const int* ranks, int L, int d, int f, int64_t total,
                 const AdamTab* tab, float* P, float* G, float* M, float* Vm, float lr, float beta1,
                 float beta2, float eps, float wd, const ShadowMap& sh, cudaStream_t s) {
    (void)L;
    int64_t total4 = total / 4;
    int blocks = (int)((total4 + 255) / 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    adam_kernel<T><<<blocks, 256, 0, s>>>(n_ad, ad_off, ranks, d, f, total4, tab,
                                          reinterpret_cast<float4*>(P), reinterpret_cast<float4*>(G),
                                          reinterpret_cast<float4*>(M), reinterpret_cast<float4*>(Vm),
                                          lr, beta1, beta2, eps, wd, sh);
}
template void launch_adam<float>(int, const int64_t*, const int*, int, int, int, int64_t,
                                 const AdamTab*, float*, float*, float*, float*, float, float, float,
                                 float, float, const ShadowMap&, cudaStream_t);
template void launch_adam<bf16>(int, const int64_t*, const int*, int, int, int, int64_t,
                                const AdamTab*, float*, float*, float*, float*, float, float, float,
                                float, float, const ShadowMap&, cudaStream_t);

template <typename T>
__global__ void shadow_sync_kernel(int n_ad, const int64_t* __restrict__ ad_off,
                                   const int* __restrict__ ranks, int d, int f, int64_t total4,
                                   const float4* __restrict__ P, ShadowMap sh) {
    __shared__ int64_t s_off[1025];
    for (int a = threadIdx.x; a <= n_ad; a += blockDim.x) s_off[a] = ad_off[a];
    __syncthreads();
    for (int64_t i4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i4 < total4;
         i4 += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = i4 * 4;
        const int a = find_adapter(s_off, n_ad, i);
        store4<T>(shadow_ptr<T>(sh, a, ranks[a], d, f, i - s_off[a]), P[i4]);
    }
}

template <typename T>
void launch_shadow_sync(int n_ad, const int64_t* ad_off, const int* ranks, int L, int d, int f,
                        int64_t total, const float* P, const ShadowMap& sh, cudaStream_t s) {
    (void)L;
    int64_t total4 = total / 4;
    int blocks = (int)((total4 + 255) / 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    shadow_sync_kernel<T><<<blocks, 256, 0, s>>>(n_ad, ad_off, ranks, d, f, total4,
                                                 reinterpret_cast<const float4*>(P), sh);
}
template void launch_shadow_sync<float>(int, const int64_t*, const int*, int, int, int, int64_t,
                                        const float*, const ShadowMap&, cudaStream_t);
template void launch_shadow_sync<bf16>(int, const int64_t*, const int*, int, int, int, int64_t,
                                       const float*, const ShadowMap&, cudaStream_t);

// ----------------------------------------------------------------------------
// out[c][r] = in[r][c] for a rows x cols matrix (32 x 32 tiles through smem).
// Used once at create to give the backward GEMMs K-major copies of W1, W2.
// ----------------------------------------------------------------------------
template <typename T>
__global__ void transpose_kernel(const T* __restrict__ in, T* __restrict__ out, int rows, int cols) {
    __shared__ T tile[32][33];
    const int bx = blockIdx.x * 32, by = blockIdx.y * 32;
    for (int i = threadIdx.y; i < 32; i += 8) {
        int r = by + i, c = bx + threadIdx.x;
        if (r < rows && c < cols) tile[i][threadIdx.x] = in[(int64_t)r * cols + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += 8) {
        int c = bx + i, r = by + threadIdx.x;
        if (c < cols && r < rows) out[(int64_t)c * rows + r] = tile[threadIdx.x][i];
    }
}

template <typename T>
void launch_transpose(const T* in, T* out, int rows, int cols, cudaStream_t s) {
    dim3 grid((cols + 31) / 32, (rows + 31) / 32);
    transpose_kernel<T><<<grid, dim3(32, 8), 0, s>>>(in, out, rows, cols);
}
template void launch_transpose<float>(const float*, float*, int, int, cudaStream_t);
template void launch_transpose<bf16>(const bf16*, bf16*, int, int, cudaStream_t);

// ----------------------------------------------------------------------------
// Operands of the merge W' = W + gamma B A (B: [M x r], A: [r x N], fp32
// masters) for one tensor-core GEMM with K = 3 * RP.  Each factor is split
// into bf16 parts, x = hi + lo with hi = bf16(x) and lo = bf16(x - hi), and
//   Aop [M x 3RP]  = [ B_hi | B_hi | B_lo ]      (K-major)
//   Bop [3RP x N]  = [ A_hi ; A_lo ; A_hi ]      (rows = K, MN-major)
// so that Aop Bop = B_hi A_hi + B_hi A_lo + B_lo A_hi, which differs from
// B A only by B_lo A_lo (relative size 2^-16).  Columns / rows j >= r are 0.
// For an fp32 base the factors are copied as they are into the first RP
// columns / rows (K = RP).
// ----------------------------------------------------------------------------
template <typename T>
__global__ void merge_operands_kernel(const float* __restrict__ Bf, const float* __restrict__ Af,
                                      int M, int N, int r, T* __restrict__ Aop, T* __restrict__ Bop) {
    constexpr bool SPLIT = sizeof(T) == 2;
    constexpr int KP = SPLIT ? 3 * RP : RP;
    const int64_t na = (int64_t)M * KP, nb = (int64_t)KP * N;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < na + nb;
         i += (int64_t)gridDim.x * blockDim.x) {
        if (i < na) {
            const int64_t m = i / KP;
            const int c = (int)(i - m * KP), part = c / RP, j = c % RP;
            float x = j < r ? Bf[m * r + j] : 0.f;
            if (SPLIT) {
                float hi = __bfloat162float(__float2bfloat16_rn(x));
                x = part < 2 ? hi : x - hi;
            }
            Aop[i] = from_f<T>(x);
        } else {
            const int64_t q = i - na;
            const int c = (int)(q / N);
            const int64_t n = q - (int64_t)c * N;
            const int part = c / RP, j = c % RP;
            float x = j < r ? Af[(int64_t)j * N + n] : 0.f;
            if (SPLIT) {
                float hi = __bfloat162float(__float2bfloat16_rn(x));
                x = part == 1 ? x - hi : hi;
            }
            Bop[q] = from_f<T>(x);
        }
    }
}

// The bf16 operands eight elements per thread (one 16-byte store, 32-bit
// index arithmetic), the same values as merge_operands_kernel: each group of
// eight lies in one part of K (RP is a multiple of 8), and N % 8 == 0.
__global__ void merge_operands_bf16x8_kernel(const float* __restrict__ Bf, const float* __restrict__ Af, int M,
                                             int N, int r, bf16* __restrict__ Aop, bf16* __restrict__ Bop) {
    constexpr int KP = 3 * RP, GK = KP / 8;
    const int gn = N / 8;
    const int ga = M * GK, gall = ga + KP * gn;
    for (int g = blockIdx.x * blockDim.x + threadIdx.x; g < gall; g += gridDim.x * blockDim.x) {
        float x[8];
        uint4 w;
        if (g < ga) {
            const int m = g / GK;
            const int c0 = (g - m * GK) * 8, part = c0 / RP, j0 = c0 % RP;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float v = j0 + e < r ? Bf[(int64_t)m * r + j0 + e] : 0.f;
                const float hi = __bfloat162float(__float2bfloat16_rn(v));
                x[e] = part < 2 ? hi : v - hi;
            }
            w = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                           pack_bf16x2(x[6], x[7]));
            *reinterpret_cast<uint4*>(Aop + (int64_t)m * KP + c0) = w;
        } else {
            const int q = g - ga;
            const int c = q / gn, n0 = (q - c * gn) * 8, part = c / RP, j = c % RP;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float v = j < r ? Af[(int64_t)j * N + n0 + e] : 0.f;
                const float hi = __bfloat162float(__float2bfloat16_rn(v));
                x[e] = part == 1 ? v - hi : hi;
            }
            w = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                           pack_bf16x2(x[6], x[7]));
            *reinterpret_cast<uint4*>(Bop + (int64_t)c * N + n0) = w;
        }
    }
}

template <typename T>
void launch_merge_operands(const float* Bf, const float* Af, int M, int N, int r, T* Aop, T* Bop,
                           cudaStream_t s) {
    if (sizeof(T) == 2 && N % 8 == 0 && (int64_t)(M + N) * 3 * RP / 8 < (1LL << 31)) {
        const int groups = (M + N) * (3 * RP / 8);
        int blocks = (groups + 255) / 256;
        if (blocks > 152 * 8) blocks = 152 * 8;
        merge_operands_bf16x8_kernel<<<blocks, 256, 0, s>>>(Bf, Af, M, N, r, reinterpret_cast<bf16*>(Aop),
                                                            reinterpret_cast<bf16*>(Bop));
        return;
    }
    merge_operands_kernel<T><<<152 * 8, 256, 0, s>>>(Bf, Af, M, N, r, Aop, Bop);
}
template void launch_merge_operands<float>(const float*, const float*, int, int, int, float*, float*,
                                           cudaStream_t);
template void launch_merge_operands<bf16>(const float*, const float*, int, int, int, bf16*, bf16*,
                                          cudaStream_t);

}  // namespace mlk
