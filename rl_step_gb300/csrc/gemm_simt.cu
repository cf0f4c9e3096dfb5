// FFMA GEMM engine: C = A B^T (+ Ax Bx^T) with the fused epilogues of
// gemm_common.cuh, for the fp32 base (whose 1e-4 logprob tolerance rules out
// bf16 tensor cores).  One CTA computes a 128 x 32 tile; thread i owns output
// row i of the tile and its 32 columns, the same unit the tensor-core engine
// hands to the epilogue.
#include "gemm_common.cuh"
#include "internal.h"

namespace mlk {

template <typename T>
__device__ __forceinline__ float ld_op(const GemmOperand& op, int adapter, int64_t mn, int64_t k) {
    int64_t r = (int64_t)adapter * op.ad_rows + op.row_shift + (op.mn_major ? k : mn);
    int64_t c = op.mn_major ? mn : k;
    if (r < 0 || r >= op.rows || c < 0 || c >= op.cols) return 0.f;
    return to_f(reinterpret_cast<const T*>(op.ptr)[r * op.ld + c]);
}

template <typename T>
__device__ __forceinline__ void simt_k_loop(const GemmOperand& A, const GemmOperand& B, int adapter,
                                            int64_t m0, int64_t n0, int64_t kbeg, int64_t kend,
                                            float* acc, float (*As)[129], float (*Bs)[33]) {
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    for (int64_t kk = kbeg; kk < kend; kk += 32) {
        if (!A.mn_major) {
#pragma unroll 4
            for (int i = 0; i < 32; ++i) {
                int m = warp + 4 * i;
                int64_t k = kk + lane;
                As[lane][m] = (k < kend) ? ld_op<T>(A, adapter, m0 + m, k) : 0.f;
            }
        } else {
#pragma unroll 4
            for (int i = 0; i < 32; ++i) {
                int64_t k = kk + i;
                As[i][tid] = (k < kend) ? ld_op<T>(A, adapter, m0 + tid, k) : 0.f;
            }
        }
        if (!B.mn_major) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                int n = warp + 4 * i;
                int64_t k = kk + lane;
                Bs[lane][n] = (k < kend) ? ld_op<T>(B, adapter, n0 + n, k) : 0.f;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                int kl = warp + 4 * i;
                int64_t k = kk + kl;
                Bs[kl][lane] = (k < kend) ? ld_op<T>(B, adapter, n0 + lane, k) : 0.f;
            }
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < 32; ++k) {
            float a = As[k][tid];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = fmaf(a, Bs[k][j], acc[j]);
        }
        __syncthreads();
    }
}

template <typename T>
__global__ void __launch_bounds__(128) simt_gemm_kernel(GemmParams p) {
    __shared__ float As[32][129];
    __shared__ float Bs[32][33];
    const int nt = blockIdx.x;
    int mt, adapter;
    int64_t kbeg = 0, kend = p.K;
    if (!p.grouped) {
        int local = blockIdx.y;
        if (local >= p.mt_count) return;
        mt = p.mt_base + local;
        int nmt = p.mtiles_dev ? *p.mtiles_dev : (p.M + TILE_M - 1) / TILE_M;
        if (mt >= nmt) return;
        adapter = p.tile_ad ? p.tile_ad[mt] : 0;
        if (adapter < 0) return;
    } else {
        int mtiles = (p.M + TILE_M - 1) / TILE_M;
        int ci = blockIdx.y / mtiles;
        mt = blockIdx.y % mtiles;
        if (ci >= *p.nchunks_dev) return;
        int4 c = p.chunks[ci];
        adapter = c.x;
        kbeg = c.y;
        kend = (int64_t)c.y + c.z;
    }
    const int64_t m0 = (int64_t)mt * TILE_M;
    const int64_t n0 = (int64_t)nt * 32;
    float acc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.f;
    simt_k_loop<T>(p.A, p.B, adapter, m0, n0, kbeg, kend, acc, As, Bs);
    if (p.Kx > 0) simt_k_loop<T>(p.Ax, p.Bx, adapter, m0, n0, 0, p.Kx, acc, As, Bs);

    const int64_t row = m0 + threadIdx.x;
    if (row >= p.M) return;
    EpiRowState st;
    epi_row_begin(st);
    // the log-sum-exp partial tile is this block's 32 columns: its maximum first
    if (p.ep.kind == EPI_LMFWD) st.m = lm_chunk_max(p.ep, (int)n0, acc);
    epi_chunk<T>(p.ep, row, (int)n0, adapter, acc, st);
    epi_row_end(p.ep, row, nt, st);
}

template <typename T>
void launch_simt_gemm(const GemmParams& p, cudaStream_t s) {
    dim3 grid((p.N + 31) / 32, 1, 1);
    if (!p.grouped) {
        grid.y = p.mt_count;
    } else {
        grid.y = p.max_chunks * ((p.M + TILE_M - 1) / TILE_M);
    }
    if (grid.y == 0 || grid.x == 0) return;
    simt_gemm_kernel<T><<<grid, 128, 0, s>>>(p);
}

template void launch_simt_gemm<float>(const GemmParams&, cudaStream_t);
template void launch_simt_gemm<bf16>(const GemmParams&, cudaStream_t);

}  // namespace mlk
