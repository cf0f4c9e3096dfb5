// Internal host-side declarations shared by the translation units of libmlora.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm_common.cuh"

namespace mlk {

// Row tiles per chunk of the LM-head backward.  By default the tiles split
// into equal chunks (an even number each, for the CTA-pair GEMMs) of at most
// nc_tiles.  When the batch needs several chunks and dh runs on the tensor-core
// engine, each of whose dh tiles contracts the whole vocabulary (about 1.5 ms
// at 151,936 x 4,096), every chunk but the last takes the largest size whose
// dh tiles fill whole waves of the `clusters` CTA pairs: no chunk but the last
// ends on a partly idle wave.  dh_ntiles is dh's column tiles per row pair
// (0: no such rule).
inline int lm_chunk_tiles(int mt_upper, int nc_tiles, int dh_ntiles, int clusters) {
    const int n_chunks = (mt_upper + nc_tiles - 1) / nc_tiles;
    int chunk = (mt_upper + n_chunks - 1) / n_chunks;
    chunk = (chunk + 1) & ~1;
    if (chunk > nc_tiles) chunk = nc_tiles;
    if (n_chunks > 1 && dh_ntiles > 0 && clusters > 0) {
        int a = dh_ntiles, b = clusters;
        while (b) { const int t = a % b; a = b; b = t; }
        const int step = 2 * (clusters / a);          // row tiles per whole number of waves
        if (step <= nc_tiles) chunk = nc_tiles / step * step;
    }
    return chunk;
}

// Device allocation of every create call (cudaMalloc, with a test hook that
// can make one chosen allocation fail).
cudaError_t mlk_malloc(void** p, size_t bytes);

// ---- GEMM engines ----------------------------------------------------------
template <typename T> void launch_simt_gemm(const GemmParams& p, cudaStream_t s);
// tcgen05 engine (bf16 only).  Returns cudaSuccess or the first error.
cudaError_t launch_tc_gemm(const GemmParams& p, cudaStream_t s, int num_sms, int* status);
bool tc_engine_available();
// TMA descriptor (CUtensorMap, 128-byte swizzle) of a row-major bf16 matrix
// [rows x cols] with row pitch ld elements, boxes of box_cols x box_rows.
bool tc_encode_bf16(void* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, uint32_t box_cols,
                    uint32_t box_rows);
// CTA-pair (cta_group::2) variant for GEMMs whose B is shared by all rows.
cudaError_t launch_tc_gemm_pair(const GemmParams& p, cudaStream_t s, int num_sms, int* status,
                                int acc_buffers, int* dbg);

// ---- attention (attention_tc.cu) ---------------------------------------------
// Causal grouped-head attention over padded token rows; head width 128.
struct AttnArgs {
    const bf16* qkv = nullptr;     // [max_rows x (n_heads + 2 n_kv) * 128]: q heads, k heads, v heads
    int n_heads = 0, n_kv = 0;
    int max_rows = 0;              // rows of every buffer below (multiple of 128)
    const int* seq_start = nullptr;  // [max_rows] first padded row of the row's sequence
    const int* meta = nullptr;     // meta[0] = valid 128-row tiles
    bf16* o = nullptr;             // [max_rows x n_heads*128]
    float* lseT = nullptr;         // [n_heads x ld_t] log2-sum-exp2 of the scaled scores (log2 units)
    float* DT = nullptr;           // [n_heads x ld_t] rowsum(dO * O) (backward)
    int ld_t = 0;                  // multiple of 4
    const bf16* dO = nullptr;      // backward: dL/dO [max_rows x n_heads*128]
    bf16* dqkv = nullptr;          // backward: dL/d(q, k, v), same layout as qkv
    int num_sms = 0;               // persistent kernels: one CTA per SM
    int* counter = nullptr;        // device int: their work-item counter
    // backward with stored dS blocks (null: the query side recomputes S and dP):
    // [max_rows/128 x ktc x n_heads] blocks of 128 key rows x 128 query columns,
    // block (query tile qt, key tile kt, head h) at (qt ktc + qt - kt) n_heads + h;
    // every query tile sees at most ktc key tiles (sequences of at most
    // 128 (ktc - 1) + 1 rows)
    bf16* ds = nullptr;
    int ktc = 0;
};
cudaError_t launch_attention_fwd(const AttnArgs& a, int* status, cudaStream_t s);
// rowsum kernel, key-side (dK, dV) kernel, query-side (dQ) kernel
cudaError_t launch_attention_bwd(const AttnArgs& a, int* status, cudaStream_t s);

// ---- transformer block (tf_kernels.cu) ----------------------------------------
constexpr int TF_NPROJ = 7;        // q, k, v, o, gate, up, down
// Where the bf16 padded-rank copy of each projection's factors lives.  A
// projection belongs to a fused group (q/k/v, o, gate/up, down) whose
// shadows are A_g [n_ad * kx x in] (sub-projection s in rows 64 s ..) and
// B_g [n_ad * n_rows x kx] (sub-projection s in columns 64 s ..; its output
// rows at row_off + i, or interleaved in blocks of ilv for gate/up).
struct TfMirrorProj {
    bf16* A = nullptr;
    bf16* B = nullptr;
    int64_t a_layer = 0, b_layer = 0;  // elements between consecutive layers' shadows
    int in = 0, out = 0;
    int kx = 0, sub = 0, n_rows = 0, row_off = 0, ilv = 0;
};
struct TfMirror {
    TfMirrorProj p[TF_NPROJ];
    int64_t sum_in_out = 0;            // sum over projections of in + out
};
void launch_tf_rows(const int* perm_pad, const int* meta, const int* tile_ad, const int* pad_off,
                    const int* positions, const int* adapter_ids, int max_pos, int max_rows, int* pos_pad,
                    int* seq_start, int* status, cudaStream_t s);
void launch_rmsnorm_fwd(const float* x, const bf16* g, int d, float eps, const int* meta, int max_rows, bf16* y,
                        float* rstd, cudaStream_t s);
void launch_rmsnorm_bwd(const float* dy, const float* x, const bf16* g, const float* rstd, int d, const int* meta,
                        int max_rows, int accumulate, float* dh, bf16* dhb, cudaStream_t s);
void launch_rope(bf16* buf, int64_t ld, int col0, int n_heads, const int* pos_pad, const float2* cs,
                 const int* meta, int max_rows, int inverse, cudaStream_t s);

// ---- routing ----------------------------------------------------------------
struct RouteBufs {
    int* blk_cnt;     // [max_blocks][n_ad]
    int* perm_pad;    // [max_pad]
    int* inv;         // [max_tokens]
    int* seg_off;     // [n_ad+1]
    int* pad_off;     // [n_ad+1]
    int* tile_ad;     // [max_tiles]
    int* meta;        // [0] m-tiles, [1] grad chunks
    int4* chunks;     // [max_chunks]
    int max_pad, max_tiles, max_chunks;
};
constexpr int ROUTE_BLOCK = 1024;   // tokens per routing block
constexpr int GRAD_CHUNK = 1024;    // padded token rows per gradient work chunk

// chunk_rows: padded rows per gradient chunk; 0 = one chunk per adapter segment
void launch_routing(const int* adapter_ids, int64_t n, int n_ad, const RouteBufs& rb,
                    int* touched, int* status, cudaStream_t s, int64_t* launches,
                    int chunk_rows = GRAD_CHUNK);
void launch_compact_perm(const RouteBufs& rb, int n_ad, int* perm_out, cudaStream_t s,
                         int64_t* launches);

// ---- elementwise / reduction kernels ----------------------------------------
template <typename T>
void launch_embed(const int* perm_pad, const int* meta, int max_rows, const int* tokens,
                  const int* targets, const T* E, int V, int d, T* hb, float* h32, int* tgt_pad,
                  int* status, cudaStream_t s);

struct LossArgs {
    int kind;                 // -1 forward only, 0 CE, 1 IS, 2 PPO, 3 custom
    const float* w;
    const float* adv;
    const float* slp;
    float clip;
    const float* dl;
};
// LM-head partial combine + loss epilogue; per-row loss values to val_row.
// rows of the m-tiles [tile0, tile0 + ntiles) (and below the batch's valid m-tiles)
void launch_combine_loss(const LossArgs& la, const float* part, int n_nt, int part_ld, const float* zt,
                         const int* perm_pad, const int* tgt_pad, const int* meta, int tile0, int ntiles,
                         float* logprobs_out, float* lse, float* g, double* val_row, int num_sms,
                         cudaStream_t s);
// dz of the LM head from stored fp32 logits, one chunk of padded rows
template <typename T>
void launch_lm_dz(const float* z, T* dz, int64_t ld, int V, int Vpad, const float* g, const float* lse,
                  const int* tgt, const int* meta, int row0, int nrows, cudaStream_t s);
// dz of the bf16 engine's LM head from the kept fp16 e = exp(z - tile max)
// and the tile maxima mt [rows][part_ld], one chunk of padded rows
void launch_lm_dz_e16(const __half* e, bf16* dz, int64_t ld, int V, int Vpad, const float* mt, int part_ld,
                      int lm_bn, const float* g, const float* lse, const int* tgt, const int* meta, int row0,
                      int nrows, cudaStream_t s);
void launch_loss_reduce(const double* val_row, const int* pad_off, int n_ad, double* loss_out,
                        cudaStream_t s);

struct AdamTab {
    int mode;      // 0 leave, 1 step, 2 skip (consume gradient only)
    float c1, c2;  // 1/(1-b1^t), 1/(1-b2^t)
};
void launch_adam_prep(int n_ad, const int* sel_mask, int* touched, int* nonfinite, int64_t* step,
                      float beta1, float beta2, AdamTab* tab, int* skipped_out, cudaStream_t s);

void launch_tf_adam(int n_ad, const int64_t* ad_off, const int* ranks, int64_t total, const AdamTab* tab, float* P,
                    float* G, float* M, float* Vm, float lr, float beta1, float beta2, float eps, float wd,
                    const TfMirror& mr, int sync_only, int num_sms, cudaStream_t s);

struct ShadowMap {
    void* A1[64];
    void* B1[64];
    void* A2[64];
    void* B2[64];
};

// What the sampler (sampler.cu) reads from a training handle: the frozen base
// it shares and the adapters' current padded-rank copies it snapshots.
struct TrainerView {
    int V, d, f, L, dtype, n_ad, Vpad, n_nt, part_ld, lm_bn, num_sms, use_tc;
    size_t esize;
    const void* E;
    const void* Wout;
    const void* const* W1;
    const void* const* W2;
    const ShadowMap* shadow;
    const float* gamma_d;          // device, per adapter
    const int64_t* step_d;         // device, optimizer steps per adapter
    const int* ranks;              // host
    const float* alphas;           // host
};
template <typename T>
void launch_adam(int n_ad, const int64_t* ad_off, const int* ranks, int L, int d, int f,
                 int64_t total, const AdamTab* tab, float* P, float* G, float* M, float* Vm,
                 float lr, float beta1, float beta2, float eps, float wd, const ShadowMap& sh,
                 cudaStream_t s);
template <typename T>
void launch_shadow_sync(int n_ad, const int64_t* ad_off, const int* ranks, int L, int d, int f,
                        int64_t total, const float* P, const ShadowMap& sh, cudaStream_t s);

// GEMM operands of W' = W + gamma B A (bf16: hi/lo split, K = 3*RP; fp32: K = RP)
template <typename T>
void launch_merge_operands(const float* Bf, const float* Af, int M, int N, int r, T* Aop, T* Bop,
                           cudaStream_t s);

template <typename T>
void launch_transpose(const T* in, T* out, int rows, int cols, cudaStream_t s);

}  // namespace mlk
