// Internal host-side declarations shared by the translation units of libmlora.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm_common.cuh"

namespace mlk {

// ---- GEMM engines ----------------------------------------------------------
template <typename T> void launch_simt_gemm(const GemmParams& p, cudaStream_t s);
// tcgen05 engine (bf16 only).  Returns cudaSuccess or the first error.
cudaError_t launch_tc_gemm(const GemmParams& p, cudaStream_t s, int num_sms, int* status);
bool tc_engine_available();
// CTA-pair (cta_group::2) variant for GEMMs whose B is shared by all rows.
cudaError_t launch_tc_gemm_pair(const GemmParams& p, cudaStream_t s, int num_sms, int* status,
                                int acc_buffers, int* dbg);

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
void launch_loss_reduce(const double* val_row, const int* pad_off, int n_ad, double* loss_out,
                        cudaStream_t s);

struct AdamTab {
    int mode;      // 0 leave, 1 step, 2 skip (consume gradient only)
    float c1, c2;  // 1/(1-b1^t), 1/(1-b2^t)
};
void launch_adam_prep(int n_ad, const int* sel_mask, int* touched, int* nonfinite, int64_t* step,
                      float beta1, float beta2, AdamTab* tab, int* skipped_out, cudaStream_t s);

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
