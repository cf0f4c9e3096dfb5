// GEMM problem description and fused epilogues shared by the two GEMM
// engines of libmlora: the tcgen05/TMEM/TMA engine (bf16) and the FFMA engine
// (fp32 base).  Both call the same epilogue on the same unit of work: one
// output row and 32 consecutive output columns held by one thread.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace mlk {

// One operand of C[m][n] = sum_k A[m][k] B[n][k].
// Element (mn, k) of adapter a sits in the stored row-major matrix at
//   K-major  (mn_major == 0): row = a*ad_rows + mn + row_shift, col = k
//   MN-major (mn_major == 1): row = a*ad_rows + k  + row_shift, col = mn
// and reads as zero outside [0, rows) x [0, cols).
struct GemmOperand {
    const void* ptr = nullptr;
    int64_t ld = 0;          // elements between consecutive stored rows
    int64_t rows = 0, cols = 0;
    int mn_major = 0;
    int64_t ad_rows = 0;     // per-adapter row stride (0: shared by all adapters)
    int64_t row_shift = 0;
};

enum EpiKind : int {
    EPI_SILU = 0,     // out0 = u = acc ; out1 = silu(acc)                     (T)
    EPI_RESID = 1,    // f32 = (f32_in or f32) + acc ; out0 = T(f32)            (residual h / dh)
    EPI_STORE2 = 2,   // f32 = acc ; out0 = T(acc)                              (dh of the LM head)
    EPI_DSILU = 3,    // out0 = T(acc * silu'(aux))                             (du)
    EPI_SHRINK = 4,   // out0 = T(gamma[a] * acc)                               (LoRA shrink)
    EPI_LMFWD = 5,    // per row: log-sum-exp over the tile's cols < V, target z; z kept if out0 (LM head)
    EPI_GRAD = 6,     // grad[a] += acc (fp32 atomics), non-finite flag         (dA / dB)
    EPI_MERGE = 7,    // out0 = T(aux + gamma[a] * acc)                         (W' = W + gamma B A)
    EPI_SHRINK_SEL = 8, // column block s = col / RP: out0 = T(gamma[s] * acc) on rows whose
                        // slot is s, 0 elsewhere                                   (sampler shrink)
    EPI_STORE = 9,      // out0 = T(acc)                                            (q, k, v / dO)
    EPI_F32 = 10,       // f32 = acc                                                (norm input grads)
    EPI_SWIGLU = 11,    // columns interleave 16 gate / 16 up: out0 = T(acc) (kept for the
                        // backward), out1[col/2 ..] = T(silu(gate) * up)             (gated MLP)
    EPI_DSWIGLU = 12,   // acc = d act; aux = the kept gate/up rows (interleaved as above):
                        // out0 = T(d gate | d up) in the same interleaved columns
    EPI_LMDZ = 13       // acc = recomputed logits z: out0 = T(g (onehot(tgt) - exp(z - lse)))
                        // for cols < V, 0 for V <= col < Vpad          (LM-head backward)
};

// Gate/up interleave of the fused gated-MLP projection: output column n of
// the fused weight is gate row (n / 32) * 16 + n % 16 when (n / 16) is even,
// up row of the same index otherwise.
constexpr int GU_ILV = 16;

struct EpiParams {
    int kind = 0;
    void* out0 = nullptr;
    void* out1 = nullptr;
    int64_t ld0 = 0, ld1 = 0;
    float* f32 = nullptr;
    int64_t ldf = 0;
    const float* f32_in = nullptr;  // EPI_RESID: the residual read, pitch ldf (null: f32 itself)
    const void* aux = nullptr;
    int64_t ld_aux = 0;
    const float* gamma = nullptr;   // per adapter
    // LM head
    float* part = nullptr;          // [rows][part_ld] log-sum-exp of each n-tile's columns
    float* zt = nullptr;            // target logit per row
    const int* tgt = nullptr;       // target id per padded row (-1: none)
    int part_ld = 0;                // pitch of a row of partials (multiple of 4)
    int V = 0, Vpad = 0;
    int64_t out_row_shift = 0;      // output row = row + out_row_shift (chunk buffers)
    int64_t out_rows = 0;           // EPI_LMFWD (kept logits) / EPI_LMDZ: rows of out0's buffer;
                                    // > 0 lets the CTA-pair engine write out0 by TMA stores
                                    // (the other staged kinds write M rows)
    const float* gv = nullptr;      // EPI_LMDZ: dL/dl per padded row
    const float* lse = nullptr;     // EPI_LMDZ: log-sum-exp per padded row
    float* mt = nullptr;            // EPI_LMFWD (written, if set) / EPI_LMDZ (read, bf16 engine):
                                    // the row's max over each partial tile, [rows][part_ld]
    int lm_bn = 0;                  // columns per log-sum-exp partial tile
    int e16 = 0;                    // EPI_LMFWD: out0 keeps fp16 e = exp(z - tile max), not fp32 z
    // adapter gradients
    float* grad = nullptr;
    const int64_t* grad_off = nullptr;  // per adapter element offset of this tensor
    const int* ranks = nullptr;
    int grad_trans = 0;             // 0: grad[m*r + n]; 1: grad[n*M + m]
    int grad_M = 0;
    int grad_ilv = 0;               // > 0: rows interleave two tensors in blocks of grad_ilv;
    int grad_sub = 0;               //      only rows of block parity grad_sub are accumulated,
                                    //      at row (row / (2 ilv)) ilv + row % ilv
    int grad_sub_stride = 0;        // > 0: several tensors side by side in N, RP columns each;
                                    //      column block s is tensor s, whose per-adapter offsets
                                    //      are grad_off + s grad_sub_stride; with grad_ilv, the
                                    //      rows of block parity s go to tensor s (the rest skipped)
    int* nonfinite = nullptr;       // per adapter flag
    const int* row_slot = nullptr;  // sampler: adapter slot per row (-1: none)
};

struct GemmParams {
    int M = 0, N = 0, K = 0, Kx = 0;
    GemmOperand A, B, Ax, Bx;
    // dense mode: rows are padded token rows in 128-row tiles
    const int* mtiles_dev = nullptr;  // valid global m-tiles (nullptr: ceil(M/128))
    int mt_base = 0, mt_count = 0;    // this launch: global m-tiles [mt_base, mt_base+mt_count)
    const int* tile_ad = nullptr;     // adapter per global m-tile
    // grouped mode: M = output rows, K runs over one chunk of one adapter's tokens
    int grouped = 0;
    const int4* chunks = nullptr;     // (adapter, k0, klen, 0)
    const int* nchunks_dev = nullptr;
    int max_chunks = 0;
    int group_m = 8;                  // raster band height (m-tiles) for L2 reuse
    int* tile_counter = nullptr;      // device int, tile scheduler of the CTA-pair kernel
    int force_bn64 = 0;               // run on the 128 x 64 single-CTA kernel whatever N is
    // Test hook of the single-CTA kernel's bounded waits (mlk_test_gemm_withhold):
    // CTA 0 skips the loads of K block test_withhold_kb of its first tile, so the
    // MMA thread's wait for that stage gives up after test_wait_ns (0: the
    // default bound).  -1: off.
    int test_withhold_kb = -1;
    unsigned long long test_wait_ns = 0;
    EpiParams ep;
};

// ----------------------------------------------------------------------------
// vector stores of 32 consecutive values
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <typename T> __device__ __forceinline__ void store32(T* dst, const float* v);

template <> __device__ __forceinline__ void store32<bf16>(bf16* dst, const float* v) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
        w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
        w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
        w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
        d4[q] = w;
    }
}

template <> __device__ __forceinline__ void store32<float>(float* dst, const float* v) {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int q = 0; q < 8; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// 32 consecutive fp32 values with evict-first stores (st.global.cs): data
// written once and read once much later (the kept LM-head logits), which should
// not displace the GEMM operands in L2
__device__ __forceinline__ void store32_stream(float* dst, const float* v) {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int q = 0; q < 8; ++q) __stcs(d4 + q, make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
}

// 32 consecutive values as fp16 (round to nearest), evict-first stores
__device__ __forceinline__ void store32_half(__half* dst, const float* v) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            __half2 h = __floats2half2_rn(v[8 * q + 2 * u], v[8 * q + 2 * u + 1]);
            w[u] = *reinterpret_cast<uint32_t*>(&h);
        }
        __stcs(d4 + q, make_uint4(w[0], w[1], w[2], w[3]));
    }
}

// first 16 of the values, 16 consecutive elements (32 bytes bf16, 64 bytes fp32)
template <typename T> __device__ __forceinline__ void store16v(T* dst, const float* v);
template <> __device__ __forceinline__ void store16v<bf16>(bf16* dst, const float* v) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 2; ++q)
        d4[q] = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                           pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
}
template <> __device__ __forceinline__ void store16v<float>(float* dst, const float* v) {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

template <typename T> __device__ __forceinline__ void load32(const T* src, float* v);

template <> __device__ __forceinline__ void load32<bf16>(const bf16* src, float* v) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 w = s4[q];
        uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 p = *reinterpret_cast<__nv_bfloat162*>(&ws[e]);
            float2 f = __bfloat1622float2(p);
            v[8 * q + 2 * e] = f.x;
            v[8 * q + 2 * e + 1] = f.y;
        }
    }
}

template <> __device__ __forceinline__ void load32<float>(const float* src, float* v) {
    const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float4 f = s4[q];
        v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
    }
}

// ----------------------------------------------------------------------------
// epilogue: per thread, one row and 32 consecutive columns at a time
// ----------------------------------------------------------------------------
struct EpiRowState {
    float m, s, zt;
    int found;
};

__device__ __forceinline__ void epi_row_begin(EpiRowState& st) {
    st.m = -INFINITY;
    st.s = 0.f;
    st.zt = 0.f;
    st.found = 0;
}

// EPI_LMFWD, per partial tile of a row: the tile's maximum m over the columns
// < V is taken first (lm_chunk_max over the tile's chunks, before the first
// lmfwd_stats); then each column's e = exp(z - m), their sum s (the tile's
// log-sum-exp partial is m + log s) and the target's logit.  The kept-logits
// LM-head backward of the bf16 engine keeps e in fp16 beside m.
__device__ __forceinline__ float lm_chunk_max(const EpiParams& ep, int col0, const float* acc) {
    float cm = -INFINITY;
#pragma unroll
    for (int j = 0; j < 32; ++j) cm = fmaxf(cm, (col0 + j) < ep.V ? acc[j] : -INFINITY);
    return cm;
}

__device__ __forceinline__ void lmfwd_stats(const EpiParams& ep, int64_t row, int col0, const float* acc,
                                            EpiRowState& st, float* e) {
    const float LOG2E = 1.4426950408889634f;
    const int t = ep.tgt[row];
    const bool fin = st.m > -INFINITY;
    const float mb = st.m * LOG2E;
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        e[j] = (fin && (col0 + j) < ep.V) ? exp2f(fmaf(acc[j], LOG2E, -mb)) : 0.f;
        sum += e[j];
        if (col0 + j == t) { st.zt = acc[j]; st.found = 1; }
    }
    st.s += sum;
}

// exp(m - lse) in the kept form's dz = g (onehot - e exp(m - lse)): one
// expression for the dz pass and the recompute epilogue
__device__ __forceinline__ float lm_tile_scale(float m, float lse) {
    return exp2f((m - lse) * 1.4426950408889634f);
}

// dz of one column from its kept fp16 e: g (onehot - e c), the product and
// the difference in one explicit fma so that every caller rounds alike
__device__ __forceinline__ float lm_dz_from_e(float g, bool is_target, float e, float c) {
    return g * fmaf(-e, c, is_target ? 1.f : 0.f);
}

// EPI_LMDZ's values of one chunk, for the columns < V (0 beyond).  bf16
// engine (E16): e = fp16(exp(z - m)) against the forward's tile maximum m,
// then dz = g (onehot - e exp(m - lse)) -- the kept form's arithmetic, so the
// recomputed accumulator (bitwise the forward's) gives the kept-logits dz
// pass's values.  Otherwise dz = g (onehot - exp(z - lse)), the fp32 dz pass's.
template <bool E16>
__device__ __forceinline__ void lmdz_values(const EpiParams& ep, int64_t row, int col0, const float* acc,
                                            float* o) {
    const float LOG2E = 1.4426950408889634f;
    const float gr = ep.gv[row];
    if (gr == 0.f) {
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = 0.f;
        return;
    }
    const int y = ep.tgt[row];
    if (E16) {
        const float m = ep.mt[row * ep.part_ld + col0 / ep.lm_bn];
        const float c = lm_tile_scale(m, ep.lse[row]);
        const float mb = m * LOG2E;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int v = col0 + j;
            const float e = __half2float(__float2half_rn(exp2f(fmaf(acc[j], LOG2E, -mb))));
            o[j] = v < ep.V ? lm_dz_from_e(gr, v == y, e, c) : 0.f;
        }
    } else {
        const float lb = ep.lse[row] * LOG2E;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int v = col0 + j;
            const float pr = exp2f(fmaf(acc[j], LOG2E, -lb));
            o[j] = v < ep.V ? gr * ((v == y ? 1.f : 0.f) - pr) : 0.f;
        }
    }
}

// EPI_SILU's second output: a = silu(acc)
__device__ __forceinline__ void silu_values(const float* acc, float* a) {
#pragma unroll
    for (int j = 0; j < 32; ++j) a[j] = acc[j] * sigmoidf_(acc[j]);
}

// EPI_DSILU: u (the saved pre-activation) becomes dL/du = acc * silu'(u).
// Hardware reciprocal, as in EPI_DSWIGLU: with the IEEE division this
// epilogue, not the tensor core, set the W2-backward GEMM's pace (16 % slower
// in a same-box comparison); the forward SiLU keeps it.
__device__ __forceinline__ void dsilu_values(const float* acc, float* u) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float s = __fdividef(1.0f, 1.0f + __expf(-u[j]));
        u[j] = acc[j] * (s * (1.f + u[j] * (1.f - s)));
    }
}

// acc holds C[row][col0 .. col0+31].  `row` is the global output row (padded
// token row in dense mode, output-feature row in grouped mode).
template <typename T>
__device__ __forceinline__ void epi_chunk(const EpiParams& ep, int64_t row, int col0, int adapter,
                                          float* acc, EpiRowState& st) {
    switch (ep.kind) {
    case EPI_SILU: {
        store32<T>(reinterpret_cast<T*>(ep.out0) + row * ep.ld0 + col0, acc);
        float a[32];
        silu_values(acc, a);
        store32<T>(reinterpret_cast<T*>(ep.out1) + row * ep.ld1 + col0, a);
    } break;
    case EPI_RESID: {
        float* hp = ep.f32 + row * ep.ldf + col0;
        float h[32];
        load32<float>(ep.f32_in ? ep.f32_in + row * ep.ldf + col0 : hp, h);
#pragma unroll
        for (int j = 0; j < 32; ++j) h[j] += acc[j];
        store32<float>(hp, h);
        if (ep.out0) store32<T>(reinterpret_cast<T*>(ep.out0) + row * ep.ld0 + col0, h);
    } break;
    case EPI_STORE2: {
        store32<float>(ep.f32 + row * ep.ldf + col0, acc);
        if (ep.out0) store32<T>(reinterpret_cast<T*>(ep.out0) + row * ep.ld0 + col0, acc);
    } break;
    case EPI_STORE: {
        store32<T>(reinterpret_cast<T*>(ep.out0) + row * ep.ld0 + col0, acc);
    } break;
    case EPI_F32: {
        store32<float>(ep.f32 + row * ep.ldf + col0, acc);
    } break;
    case EPI_SWIGLU: {
        store32<T>(reinterpret_cast<T*>(ep.out0) + row * ep.ld0 + col0, acc);
        float a[32];
#pragma unroll
        for (int j = 0; j < 16; ++j) a[j] = acc[j] * sigmoidf_(acc[j]) * acc[16 + j];
#pragma unroll
        for (int j = 16; j < 32; ++j) a[j] = 0.f;
        store16v<T>(reinterpret_cast<T*>(ep.out1) + row * ep.ld1 + col0 / 2, a);
    } break;
    case EPI_DSWIGLU: {
        const T* gu = reinterpret_cast<const T*>(ep.aux) + row * ep.ld_aux + 2 * col0;
        T* dgu = reinterpret_cast<T*>(ep.out0) + row * ep.ld0 + 2 * col0;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            float g[32], o[32];
            load32<T>(gu + 32 * hb, g);     // g[0..15] gate, g[16..31] up
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float da = acc[16 * hb + j];
                // hardware reciprocal: this epilogue also waits on its gate/up
                // loads, and the IEEE division measured 14 % slower here
                const float sg = __fdividef(1.0f, 1.0f + __expf(-g[j]));
                o[j] = da * g[16 + j] * (sg * (1.f + g[j] * (1.f - sg)));
                o[16 + j] = da * g[j] * sg;
            }
            store32<T>(dgu + 32 * hb, o);
        }
    } break;
    case EPI_DSILU: {
        float u[32];
        load32<T>(reinterpret_cast<const T*>(ep.aux) + row * ep.ld_aux + col0, u);
        dsilu_values(acc, u);
        store32<T>(reinterpret_cast<T*>(ep.out0) + row * ep.ld0 + col0, u);
    } break;
    case EPI_SHRINK: {
        float gm = ep.gamma[adapter];
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] *= gm;
        store32<T>(reinterpret_cast<T*>(ep.out0) + row * ep.ld0 + col0, acc);
    } break;
    case EPI_LMFWD: {
        float e[32];
        lmfwd_stats(ep, row, col0, acc, st, e);
        if (ep.out0 && col0 < ep.Vpad) {   // keep the logits for the backward (or the sampler)
            if (ep.e16) store32_half(reinterpret_cast<__half*>(ep.out0) + (row + ep.out_row_shift) * ep.ld0 + col0, e);
            else store32_stream(reinterpret_cast<float*>(ep.out0) + (row + ep.out_row_shift) * ep.ld0 + col0, acc);
        }
    } break;
    case EPI_LMDZ: {
        float o[32];
        lmdz_values<std::is_same<T, bf16>::value>(ep, row, col0, acc, o);
        store32<T>(reinterpret_cast<T*>(ep.out0) + (row + ep.out_row_shift) * ep.ld0 + col0, o);
    } break;
    case EPI_SHRINK_SEL: {
        const int sl = col0 / RP;
        const bool mine = ep.row_slot[row] == sl;
        const float gm = ep.gamma[sl];
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = mine ? acc[j] * gm : 0.f;
        store32<T>(reinterpret_cast<T*>(ep.out0) + row * ep.ld0 + col0, acc);
    } break;
    case EPI_MERGE: {
        float w[32];
        load32<T>(reinterpret_cast<const T*>(ep.aux) + row * ep.ld_aux + col0, w);
        const float gm = ep.gamma[adapter];
#pragma unroll
        for (int j = 0; j < 32; ++j) w[j] = fmaf(gm, acc[j], w[j]);
        store32<T>(reinterpret_cast<T*>(ep.out0) + row * ep.ld0 + col0, w);
    } break;
    case EPI_GRAD: {
        int r = ep.ranks[adapter];
        int sub = ep.grad_sub;
        if (ep.grad_sub_stride) {       // column block -> tensor
            sub = col0 / RP;
            col0 -= sub * RP;
        }
        float* base = ep.grad + ep.grad_off[(int64_t)sub * ep.grad_sub_stride + adapter];
        if (ep.grad_ilv) {
            if ((int)((row / ep.grad_ilv) & 1) != sub) break;
            row = (row / (2 * ep.grad_ilv)) * ep.grad_ilv + row % ep.grad_ilv;
        }
        bool bad = false;
#pragma unroll
        for (int j = 0; j < 32; ++j) bad |= (col0 + j < r) && !isfinite(acc[j]);
        if (ep.grad_trans) {
            // [r x M] target: the warp's 32 rows are 32 consecutive floats per column
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (col0 + j < r) atomicAdd(base + (int64_t)(col0 + j) * ep.grad_M + row, acc[j]);
        } else {
            // [M x r] target: this row's columns are consecutive (r and col0 are
            // multiples of 4, so every group of four is 16-byte aligned): one
            // vector reduction per four values
            float* dst = base + row * (int64_t)r + col0;
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                if (col0 + j < r)
                    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + j), "f"(acc[j]),
                                 "f"(acc[j + 1]), "f"(acc[j + 2]), "f"(acc[j + 3])
                                 : "memory");
        }
        if (bad) ep.nonfinite[adapter] = 1;
    } break;
    default: break;
    }
}

__device__ __forceinline__ void epi_row_end(const EpiParams& ep, int64_t row, int ntile,
                                            const EpiRowState& st) {
    if (ep.kind == EPI_LMFWD) {
        ep.part[row * ep.part_ld + ntile] = st.s > 0.f ? st.m + __logf(st.s) : -INFINITY;
        if (ep.mt) ep.mt[row * ep.part_ld + ntile] = st.m;
        if (st.found) ep.zt[row] = st.zt;
    }
}

// ----------------------------------------------------------------------------
// tile bookkeeping shared by both engines
// ----------------------------------------------------------------------------
struct TileInfo {
    int mt;        // global m-tile (dense) or m-tile inside the chunk (grouped)
    int nt;        // n-tile
    int adapter;
    int k0, klen;  // contraction range of the main operands
    int valid;
};

}  // namespace mlk
