// Bandwidth-bound kernels of the transformer block: per-row sequence
// metadata, RMSNorm forward and backward, the rotary embedding, and the
// table-driven Adam update of the seven-projection adapters.
#include <math.h>

#include "internal.h"

namespace mlk {

// ----------------------------------------------------------------------------
// Per padded row p (valid tiles only): position and first row of its
// sequence.  A token with position 0 starts a sequence; any other token must
// continue the token before it in the batch (same adapter, position one
// lower), so that routing's stable grouping keeps every sequence contiguous
// and row p attends to rows [p - pos, p].  A token that breaks this, or whose
// position is outside [0, max_pos), raises ST_RANGE and is treated as a
// sequence of its own at position 0.  Padding rows are one-row sequences.
// ----------------------------------------------------------------------------
__global__ void tf_rows_kernel(const int* __restrict__ perm_pad, const int* __restrict__ meta,
                               const int* __restrict__ tile_ad, const int* __restrict__ pad_off,
                               const int* __restrict__ positions, const int* __restrict__ adapter_ids,
                               int max_pos, int* __restrict__ pos_pad, int* __restrict__ seq_start,
                               int* status) {
    const int rows = meta[0] * TILE_M;
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < rows; p += gridDim.x * blockDim.x) {
        const int t = perm_pad[p];
        int pos = 0, start = p;
        if (t >= 0) {
            const int q = positions[t];
            bool ok = q >= 0 && q < max_pos;
            if (ok && q > 0)
                ok = t > 0 && positions[t - 1] == q - 1 && adapter_ids[t - 1] == adapter_ids[t];
            if (ok) {
                pos = q;
                const int lo = pad_off[tile_ad[p / TILE_M]];
                start = p - q < lo ? lo : p - q;
            } else {
                raise_status(status, ST_RANGE);
            }
        }
        pos_pad[p] = pos;
        seq_start[p] = start;
    }
}

void launch_tf_rows(const int* perm_pad, const int* meta, const int* tile_ad, const int* pad_off,
                    const int* positions, const int* adapter_ids, int max_pos, int max_rows, int* pos_pad,
                    int* seq_start, int* status, cudaStream_t s) {
    int blocks = (max_rows + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    tf_rows_kernel<<<blocks, 256, 0, s>>>(perm_pad, meta, tile_ad, pad_off, positions, adapter_ids, max_pos,
                                          pos_pad, seq_start, status);
}

// ----------------------------------------------------------------------------
// RMSNorm: y = x / sqrt(mean(x^2) + eps) * g, one warp per row (d % 128 == 0).
// Writes y (bf16) and 1/rms per row.  Rows past the valid tiles are skipped.
// ----------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void load4_bf16(const bf16* p, float (&v)[4]) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}

__device__ __forceinline__ void load8_bf16(const bf16* p, float (&v)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[e]));
        v[2 * e] = f.x;
        v[2 * e + 1] = f.y;
    }
}

__global__ void __launch_bounds__(256) rmsnorm_fwd_kernel(const float* __restrict__ x, const bf16* __restrict__ g,
                                                          int d, float eps, const int* __restrict__ meta,
                                                          bf16* __restrict__ y, float* __restrict__ rstd) {
    const int rows = meta[0] * TILE_M;
    const int lane = threadIdx.x & 31;
    const int64_t p = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (p >= rows) return;
    const float* xr = x + p * d;
    float ss = 0.f;
    for (int c = lane * 4; c < d; c += 128) {
        const float4 v = *reinterpret_cast<const float4*>(xr + c);
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    ss = warp_sum(ss);
    const float r = rsqrtf(ss / (float)d + eps);
    if (lane == 0) rstd[p] = r;
    for (int c = lane * 4; c < d; c += 128) {
        const float4 v = *reinterpret_cast<const float4*>(xr + c);
        float gv[4];
        load4_bf16(g + c, gv);
        uint2 w;
        w.x = pack_bf16x2(v.x * r * gv[0], v.y * r * gv[1]);
        w.y = pack_bf16x2(v.z * r * gv[2], v.w * r * gv[3]);
        *reinterpret_cast<uint2*>(y + p * d + c) = w;
    }
}

// One-pass forms for d <= 512 NV: one block of 128 threads per row, thread t
// holding the row's float4 chunks t + 128 i (i < NV) in registers, so each
// input row is read from memory once.  (With one warp per row the second
// loop's re-read of x misses L2 whenever the rows in flight, ~16 KB each,
// outgrow it.)  The row's sum of squares: per-thread partials in chunk
// order, a warp tree, then the four warps' sums in warp order.
constexpr int NORM_THREADS = 128;

__device__ __forceinline__ float block128_sum(float v, float* part) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
    __syncthreads();
    return (part[0] + part[1]) + (part[2] + part[3]);
}

template <int NV>
__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_fwd_row_kernel(const float* __restrict__ x,
                                                                       const bf16* __restrict__ g, int d, float eps,
                                                                       const int* __restrict__ meta,
                                                                       bf16* __restrict__ y, float* __restrict__ rstd) {
    __shared__ float part[NORM_THREADS / 32];
    const int64_t p = blockIdx.x;
    if (p >= (int64_t)meta[0] * TILE_M) return;
    const int n4 = d >> 2;
    const float4* xr = reinterpret_cast<const float4*>(x + p * d);
    float4 v[NV];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int c = threadIdx.x + NORM_THREADS * i;
        if (c < n4) {
            v[i] = xr[c];
            ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
        }
    }
    const float r = rsqrtf(block128_sum(ss, part) / (float)d + eps);
    if (threadIdx.x == 0) rstd[p] = r;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int c = threadIdx.x + NORM_THREADS * i;
        if (c < n4) {
            float gv[4];
            load4_bf16(g + 4 * c, gv);
            uint2 w;
            w.x = pack_bf16x2(v[i].x * r * gv[0], v[i].y * r * gv[1]);
            w.y = pack_bf16x2(v[i].z * r * gv[2], v[i].w * r * gv[3]);
            reinterpret_cast<uint2*>(y + p * d)[c] = w;
        }
    }
}

void launch_rmsnorm_fwd(const float* x, const bf16* g, int d, float eps, const int* meta, int max_rows, bf16* y,
                        float* rstd, cudaStream_t s) {
    if (d <= 512 * 8)
        rmsnorm_fwd_row_kernel<8><<<max_rows, NORM_THREADS, 0, s>>>(x, g, d, eps, meta, y, rstd);
    else if (d <= 512 * 16)
        rmsnorm_fwd_row_kernel<16><<<max_rows, NORM_THREADS, 0, s>>>(x, g, d, eps, meta, y, rstd);
    else
        rmsnorm_fwd_kernel<<<(max_rows + 7) / 8, 256, 0, s>>>(x, g, d, eps, meta, y, rstd);
}

// dx = rstd (g dy) - x rstd^3 mean(x g dy);  dh (+)= dx;  dhb = bf16(dh).
__global__ void __launch_bounds__(256) rmsnorm_bwd_kernel(const float* __restrict__ dy, const float* __restrict__ x,
                                                          const bf16* __restrict__ g, const float* __restrict__ rstd,
                                                          int d, const int* __restrict__ meta, int accumulate,
                                                          float* __restrict__ dh, bf16* __restrict__ dhb) {
    const int rows = meta[0] * TILE_M;
    const int lane = threadIdx.x & 31;
    const int64_t p = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (p >= rows) return;
    float c = 0.f;
    for (int k = lane * 4; k < d; k += 128) {
        const float4 a = *reinterpret_cast<const float4*>(dy + p * d + k);
        const float4 b = *reinterpret_cast<const float4*>(x + p * d + k);
        float gv[4];
        load4_bf16(g + k, gv);
        c += a.x * gv[0] * b.x + a.y * gv[1] * b.y + a.z * gv[2] * b.z + a.w * gv[3] * b.w;
    }
    c = warp_sum(c) / (float)d;
    const float r = rstd[p];
    const float r3c = r * r * r * c;
    for (int k = lane * 4; k < d; k += 128) {
        const float4 a = *reinterpret_cast<const float4*>(dy + p * d + k);
        const float4 b = *reinterpret_cast<const float4*>(x + p * d + k);
        float gv[4];
        load4_bf16(g + k, gv);
        float4 o = make_float4(r * gv[0] * a.x - b.x * r3c, r * gv[1] * a.y - b.y * r3c,
                               r * gv[2] * a.z - b.z * r3c, r * gv[3] * a.w - b.w * r3c);
        float* hp = dh + p * d + k;
        if (accumulate) {
            const float4 h = *reinterpret_cast<const float4*>(hp);
            o.x += h.x; o.y += h.y; o.z += h.z; o.w += h.w;
        }
        *reinterpret_cast<float4*>(hp) = o;
        uint2 w;
        w.x = pack_bf16x2(o.x, o.y);
        w.y = pack_bf16x2(o.z, o.w);
        *reinterpret_cast<uint2*>(dhb + p * d + k) = w;
    }
}

// One-pass backward (d <= 512 NV): dy and x of the row held in registers.
template <int NV>
__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_bwd_row_kernel(const float* __restrict__ dy,
                                                                       const float* __restrict__ x,
                                                                       const bf16* __restrict__ g,
                                                                       const float* __restrict__ rstd, int d,
                                                                       const int* __restrict__ meta, int accumulate,
                                                                       float* __restrict__ dh, bf16* __restrict__ dhb) {
    __shared__ float part[NORM_THREADS / 32];
    const int64_t p = blockIdx.x;
    if (p >= (int64_t)meta[0] * TILE_M) return;
    const int n4 = d >> 2;
    const float4* dyr = reinterpret_cast<const float4*>(dy + p * d);
    const float4* xr = reinterpret_cast<const float4*>(x + p * d);
    float4 a[NV], b[NV];
    float c = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int k = threadIdx.x + NORM_THREADS * i;
        if (k < n4) {
            a[i] = dyr[k];
            b[i] = xr[k];
            float gv[4];
            load4_bf16(g + 4 * k, gv);
            c += a[i].x * gv[0] * b[i].x + a[i].y * gv[1] * b[i].y + a[i].z * gv[2] * b[i].z +
                 a[i].w * gv[3] * b[i].w;
        }
    }
    c = block128_sum(c, part) / (float)d;
    const float r = rstd[p];
    const float r3c = r * r * r * c;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int k = threadIdx.x + NORM_THREADS * i;
        if (k < n4) {
            float gv[4];
            load4_bf16(g + 4 * k, gv);
            float4 o = make_float4(r * gv[0] * a[i].x - b[i].x * r3c, r * gv[1] * a[i].y - b[i].y * r3c,
                                   r * gv[2] * a[i].z - b[i].z * r3c, r * gv[3] * a[i].w - b[i].w * r3c);
            float4* hp = reinterpret_cast<float4*>(dh + p * d) + k;
            if (accumulate) {
                const float4 h = *hp;
                o.x += h.x; o.y += h.y; o.z += h.z; o.w += h.w;
            }
            *hp = o;
            uint2 w;
            w.x = pack_bf16x2(o.x, o.y);
            w.y = pack_bf16x2(o.z, o.w);
            reinterpret_cast<uint2*>(dhb + p * d)[k] = w;
        }
    }
}

void launch_rmsnorm_bwd(const float* dy, const float* x, const bf16* g, const float* rstd, int d, const int* meta,
                        int max_rows, int accumulate, float* dh, bf16* dhb, cudaStream_t s) {
    if (d <= 512 * 8)
        rmsnorm_bwd_row_kernel<8><<<max_rows, NORM_THREADS, 0, s>>>(dy, x, g, rstd, d, meta, accumulate, dh, dhb);
    else if (d <= 512 * 16)
        rmsnorm_bwd_row_kernel<16><<<max_rows, NORM_THREADS, 0, s>>>(dy, x, g, rstd, d, meta, accumulate, dh, dhb);
    else
        rmsnorm_bwd_kernel<<<(max_rows + 7) / 8, 256, 0, s>>>(dy, x, g, rstd, d, meta, accumulate, dh, dhb);
}

// ----------------------------------------------------------------------------
// Rotary embedding in place on n_heads heads of width 128 starting at column
// col0 of a bf16 [rows x ld] buffer: for i < 64 the pair (x_i, x_{i+64}) of
// each head is rotated by angle pos * theta^(-i/64), read from the host-built
// table cs[pos][i] = (cos, sin); inverse = 1 rotates by minus the angle (the
// backward).  8 threads per (row, head), 8 pairs each.
// ----------------------------------------------------------------------------
__global__ void rope_kernel(bf16* __restrict__ buf, int64_t ld, int col0, int n_heads,
                            const int* __restrict__ pos_pad, const float2* __restrict__ cs,
                            const int* __restrict__ meta, int inverse) {
    const int64_t rows = (int64_t)meta[0] * TILE_M;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int part = (int)(gid & 7);
    const int64_t unit = gid >> 3;
    const int64_t p = unit / n_heads;
    const int hh = (int)(unit % n_heads);
    if (p >= rows) return;
    bf16* a = buf + p * ld + col0 + hh * 128 + part * 8;
    bf16* b = a + 64;
    const float2* t = cs + (int64_t)pos_pad[p] * 64 + part * 8;
    float va[8], vb[8];
    load8_bf16(a, va);
    load8_bf16(b, vb);
    const float sg = inverse ? -1.f : 1.f;
    uint32_t wa[4], wb[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const float2 c0 = t[e], c1 = t[e + 1];
        const float s0 = sg * c0.y, s1 = sg * c1.y;
        wa[e >> 1] = pack_bf16x2(va[e] * c0.x - vb[e] * s0, va[e + 1] * c1.x - vb[e + 1] * s1);
        wb[e >> 1] = pack_bf16x2(vb[e] * c0.x + va[e] * s0, vb[e + 1] * c1.x + va[e + 1] * s1);
    }
    *reinterpret_cast<uint4*>(a) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
    *reinterpret_cast<uint4*>(b) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
}

void launch_rope(bf16* buf, int64_t ld, int col0, int n_heads, const int* pos_pad, const float2* cs,
                 const int* meta, int max_rows, int inverse, cudaStream_t s) {
    const int64_t threads = (int64_t)max_rows * n_heads * 8;
    rope_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(buf, ld, col0, n_heads, pos_pad, cs, meta,
                                                                    inverse);
}

// ----------------------------------------------------------------------------
// Adam over the seven-projection adapters.  Adapter a's fp32 parameters
// occupy [ad_off[a], ad_off[a+1]) of P, G, M, V; inside, layer by layer, for
// each projection q, k, v, o, gate, up, down: A [r x in] then B [out x r].
// Each updated element is mirrored into the bf16 padded-rank copies the GEMMs
// read (TfMirror); sync_only copies P into them without an update.
// ----------------------------------------------------------------------------
__device__ __forceinline__ int tf_find_adapter(const int64_t* off, int n_ad, int64_t i) {
    int lo = 0, hi = n_ad - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= i) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ bf16* tf_mirror_ptr(const TfMirror& mr, int a, int r, int64_t rel) {
    const int64_t per_layer = (int64_t)r * mr.sum_in_out;
    const int l = (int)(rel / per_layer);
    int64_t q = rel - (int64_t)l * per_layer;
#pragma unroll 1
    for (int k = 0; k < TF_NPROJ; ++k) {
        const TfMirrorProj& m = mr.p[k];
        const int64_t na = (int64_t)r * m.in;
        if (q < na) {
            const int64_t i = q / m.in, j = q - i * m.in;
            return m.A + l * m.a_layer + ((int64_t)a * m.kx + 64 * m.sub + i) * m.in + j;
        }
        q -= na;
        const int64_t nb = (int64_t)m.out * r;
        if (q < nb || k == TF_NPROJ - 1) {
            const int64_t i = q / r, j = q - i * r;
            const int64_t row = m.ilv ? (i / m.ilv) * 2 * m.ilv + m.sub * m.ilv + i % m.ilv : m.row_off + i;
            return m.B + l * m.b_layer + ((int64_t)a * m.n_rows + row) * m.kx + 64 * m.sub + j;
        }
        q -= nb;
    }
    return nullptr;
}

__global__ void __launch_bounds__(256) tf_adam_kernel(int n_ad, const int64_t* __restrict__ ad_off,
                                                      const int* __restrict__ ranks, int64_t total4,
                                                      const AdamTab* __restrict__ tab, float4* P, float4* G,
                                                      float4* M, float4* Vm, float lr, float b1, float b2,
                                                      float eps, float wd, const __grid_constant__ TfMirror mr,
                                                      int sync_only) {
    __shared__ int64_t s_off[1025];
    for (int a = threadIdx.x; a <= n_ad; a += blockDim.x) s_off[a] = ad_off[a];
    __syncthreads();
    for (int64_t i4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i4 < total4;
         i4 += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = i4 * 4;
        const int a = tf_find_adapter(s_off, n_ad, i);
        float4 pn;
        if (sync_only) {
            pn = P[i4];
        } else {
            const AdamTab e = tab[a];
            if (e.mode == 0) continue;
            if (e.mode == 2) {
                G[i4] = make_float4(0.f, 0.f, 0.f, 0.f);
                continue;
            }
            const float4 g = G[i4], p = P[i4], m = M[i4], v = Vm[i4];
            const float gv[4] = {g.x, g.y, g.z, g.w};
            float pv[4] = {p.x, p.y, p.z, p.w};
            float mv[4] = {m.x, m.y, m.z, m.w};
            float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                mv[q] = b1 * mv[q] + (1.f - b1) * gv[q];
                vv[q] = b2 * vv[q] + (1.f - b2) * gv[q] * gv[q];
                const float mh = mv[q] * e.c1, vh = vv[q] * e.c2;
                pv[q] = pv[q] - lr * (mh / (sqrtf(vh) + eps) + wd * pv[q]);
            }
            pn = make_float4(pv[0], pv[1], pv[2], pv[3]);
            P[i4] = pn;
            M[i4] = make_float4(mv[0], mv[1], mv[2], mv[3]);
            Vm[i4] = make_float4(vv[0], vv[1], vv[2], vv[3]);
            G[i4] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        uint2 w;
        w.x = pack_bf16x2(pn.x, pn.y);
        w.y = pack_bf16x2(pn.z, pn.w);
        *reinterpret_cast<uint2*>(tf_mirror_ptr(mr, a, ranks[a], i - s_off[a])) = w;
    }
}

void launch_tf_adam(int n_ad, const int64_t* ad_off, const int* ranks, int64_t total, const AdamTab* tab, float* P,
                    float* G, float* M, float* Vm, float lr, float beta1, float beta2, float eps, float wd,
                    const TfMirror& mr, int sync_only, int num_sms, cudaStream_t s) {
    const int64_t total4 = total / 4;
    int64_t blocks = (total4 + 255) / 256;
    if (blocks > (int64_t)num_sms * 16) blocks = (int64_t)num_sms * 16;
    if (blocks < 1) blocks = 1;
    tf_adam_kernel<<<(unsigned)blocks, 256, 0, s>>>(n_ad, ad_off, ranks, total4, tab, reinterpret_cast<float4*>(P),
                                                    reinterpret_cast<float4*>(G), reinterpret_cast<float4*>(M),
                                                    reinterpret_cast<float4*>(Vm), lr, beta1, beta2, eps, wd, mr,
                                                    sync_only);
}

}  // namespace mlk
