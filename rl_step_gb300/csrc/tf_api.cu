// C ABI of the transformer-block model (include/mlora_tf.h) and the host-side
// launch sequence of its step.  Every step of the computation runs in this
// library's kernels on the caller's stream: routing and embedding
// (routing.cu, kernels_misc.cu), RMSNorm / rotary / sequence metadata / Adam
// (tf_kernels.cu), attention (attention_tc.cu), every projection on the
// tcgen05 GEMM engine (gemm_tc.cu), and the LM head with its loss epilogue
// (gemm_tc.cu, kernels_misc.cu).  The host validates, builds descriptors and
// queues work.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <cmath>
#include <string>
#include <vector>

#include "../../include/mlora_tf.h"
#include "internal.h"

using namespace mlk;

int mlk_report_error(int code, const char* msg);

namespace {

int tfail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int tfail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    return mlk_report_error(code, buf);
}

#define TF_CUDA(expr)                                                                     \
    do {                                                                                  \
        cudaError_t _e = (expr);                                                          \
        if (_e != cudaSuccess)                                                            \
            return tfail(MLORA_E_CUDA, "%s failed: %s", #expr, cudaGetErrorString(_e));   \
    } while (0)

// fused projection groups and their LoRA extension width (64 per member)
enum { G_QKV = 0, G_O = 1, G_GU = 2, G_D = 3, NGROUPS = 4 };
constexpr int GROUP_OF[TF_NPROJ] = {G_QKV, G_QKV, G_QKV, G_O, G_GU, G_GU, G_D};
constexpr int SUB_OF[TF_NPROJ] = {0, 1, 2, 0, 0, 1, 0};
constexpr int GROUP_KX[NGROUPS] = {3 * RP, RP, 2 * RP, RP};

}  // namespace

struct mlora_tf {
    int V = 0, d = 0, nh = 0, nkv = 0, f = 0, L = 0, n_ad = 0;
    int Q = 0, KV = 0, Nqkv = 0;     // n_heads*128, n_kv*128, Q + 2 KV
    float theta = 0.f, eps = 0.f;
    int64_t max_tokens = 0;
    int max_pad = 0, max_tiles = 0, max_chunks = 0, max_blocks = 0;
    int Vpad = 0, n_nt = 0, part_ld = 0, nc_tiles = 0;
    int num_sms = 0;
    std::vector<int> ranks;
    std::vector<float> alphas;
    std::vector<void*> allocs;
    std::vector<size_t> alloc_bytes;
    int64_t bytes = 0;
    int64_t launches = 0;

    // frozen base (bf16)
    bf16 *E = nullptr, *Wout = nullptr, *gfinal = nullptr;
    std::vector<bf16*> gattn, gmlp;
    std::vector<bf16*> W[NGROUPS], WT[NGROUPS];   // fused [N_g x in_g] and K-major copies [in_g x N_g]
    int gN[NGROUPS] = {0}, gIn[NGROUPS] = {0};
    // adapters: masters, gradients, moments; bf16 shadows per group and layer
    int64_t n_params = 0, per_layer_unit = 0;     // params per layer = rank * per_layer_unit
    std::vector<int64_t> ad_off_h;
    float *P = nullptr, *G = nullptr, *M = nullptr, *Vm = nullptr;
    int64_t* ad_off = nullptr;
    int* ranks_d = nullptr;
    float* gamma_d = nullptr;
    int64_t* grad_off = nullptr;                  // [((l * 7 + p) * 2 + factor) * n_ad + a]
    int64_t* step = nullptr;
    int *touched = nullptr, *nonfinite = nullptr, *sel_mask = nullptr;
    AdamTab* adam_tab = nullptr;
    bf16* As[NGROUPS] = {nullptr};                 // [L][n_ad * kx (+pad) x in_g]
    bf16* Bs[NGROUPS] = {nullptr};                 // [L][n_ad * N_g x kx]
    int64_t As_rows[NGROUPS] = {0}, As_layer[NGROUPS] = {0}, Bs_layer[NGROUPS] = {0};
    TfMirror mirror;
    // routing and sequence metadata
    RouteBufs rb;
    int *pos_pad = nullptr, *seq_start = nullptr;
    float2* rope_cs = nullptr;                     // [max_tokens x 64] (cos, sin)
    // activations, per layer
    std::vector<bf16*> x1, vqkv, qkv, o, vo, x2, vgu, gu, act, vd;
    std::vector<float*> lseT, snap1, snap2, rstd1, rstd2;
    bf16* xf = nullptr;
    float *snapf = nullptr, *rstdf = nullptr;
    float *h32 = nullptr, *dh32 = nullptr, *dxn32 = nullptr;
    bf16 *dhb = nullptr, *wbuf = nullptr, *dgu = nullptr, *dO = nullptr, *dqkv = nullptr, *embed_bf = nullptr;
    float* DT = nullptr;
    // LM head (as in the MLP model)
    float* part = nullptr;
    float *zt = nullptr, *lse = nullptr, *gvec = nullptr;
    int* tgt_pad = nullptr;
    // LM-head backward mode (mlora_tf_set_lm_backward): recompute (dz[0] only) or
    // kept logits (dz[0..1], zbuf[0..1], allocated when selected)
    int lm_keep = 0;
    bf16* dz[2] = {nullptr, nullptr};
    __half* zbuf[2] = {nullptr, nullptr};   // kept fp16 e = exp(z - tile max) of a chunk of rows
    float* mt = nullptr;                    // per row and partial tile: the tile's logit maximum
    // attention backward (mlora_tf_set_attention_backward): the query side
    // recomputes S and dP (attn_ds null), or reads the dS blocks the key side
    // stores for sequences of at most attn_max_seq tokens (attn_ktc key tiles
    // per query tile)
    bf16* attn_ds = nullptr;
    int attn_ktc = 0, attn_max_seq = 0;
    cudaStream_t side = nullptr;
    cudaEvent_t ev_comb[2] = {}, ev_dz[2] = {}, ev_dh[2] = {};
    double* val_row = nullptr;
    int* status = nullptr;
    int* tile_counter = nullptr;
    // measurement
    bool prof = false;
    std::vector<cudaEvent_t> ev;
    std::vector<int> ev_cls;
    size_t ev_used = 0;
    double prof_ms[MLORA_TF_PROF_CLASSES] = {0};
    int64_t prof_n[MLORA_TF_PROF_CLASSES] = {0};
};

namespace {

struct TfProf {
    mlora_tf_t* h;
    cudaStream_t s;
    int cls;
    size_t slot = (size_t)-1;
    TfProf(mlora_tf_t* h_, cudaStream_t s_, int cls_) : h(h_), s(s_), cls(cls_) {
        if (!h->prof) return;
        if (h->ev_used * 2 + 2 > h->ev.size()) {
            for (int i = 0; i < 64; ++i) {
                cudaEvent_t e;
                if (cudaEventCreate(&e) != cudaSuccess) return;
                h->ev.push_back(e);
            }
            h->ev_cls.resize(h->ev.size() / 2);
        }
        slot = h->ev_used++;
        cudaEventRecord(h->ev[2 * slot], s);
    }
    ~TfProf() {
        if (slot == (size_t)-1) return;
        cudaEventRecord(h->ev[2 * slot + 1], s);
        h->ev_cls[slot] = cls;
    }
};

int tf_alloc(mlora_tf_t* h, void** p, size_t bytes) {
    if (bytes == 0) bytes = 16;
    cudaError_t e = mlk_malloc(p, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return tfail(MLORA_E_NOMEM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
    }
    h->allocs.push_back(*p);
    h->alloc_bytes.push_back(bytes);
    h->bytes += (int64_t)bytes;
    return MLORA_OK;
}

// Frees one allocation made by tf_alloc (the caller has synchronised the device).
void tf_free(mlora_tf_t* h, void** p) {
    if (!*p) return;
    for (size_t i = 0; i < h->allocs.size(); ++i)
        if (h->allocs[i] == *p) {
            cudaFree(*p);
            h->bytes -= (int64_t)h->alloc_bytes[i];
            h->allocs.erase(h->allocs.begin() + (ptrdiff_t)i);
            h->alloc_bytes.erase(h->alloc_bytes.begin() + (ptrdiff_t)i);
            break;
        }
    *p = nullptr;
}

template <typename P>
int tf_alloc_t(mlora_tf_t* h, P** p, size_t count) {
    void* q = nullptr;
    int rc = tf_alloc(h, &q, count * sizeof(P));
    *p = reinterpret_cast<P*>(q);
    return rc;
}

void tf_free_all(mlora_tf_t* h) {
    for (void* p : h->allocs) cudaFree(p);
    h->allocs.clear();
    h->alloc_bytes.clear();
    for (cudaEvent_t e : h->ev) cudaEventDestroy(e);
    h->ev.clear();
    for (int b = 0; b < 2; ++b) {
        if (h->ev_comb[b]) cudaEventDestroy(h->ev_comb[b]);
        if (h->ev_dz[b]) cudaEventDestroy(h->ev_dz[b]);
        if (h->ev_dh[b]) cudaEventDestroy(h->ev_dh[b]);
        h->ev_comb[b] = h->ev_dz[b] = h->ev_dh[b] = nullptr;
    }
    if (h->side) cudaStreamDestroy(h->side);
    h->side = nullptr;
}

// (out, in) of projection p
inline void proj_shape(const mlora_tf_t* h, int p, int* out, int* in) {
    switch (p) {
    case MLORA_TF_Q: *out = h->Q; *in = h->d; break;
    case MLORA_TF_K: case MLORA_TF_V: *out = h->KV; *in = h->d; break;
    case MLORA_TF_O: *out = h->d; *in = h->Q; break;
    case MLORA_TF_GATE: case MLORA_TF_UP: *out = h->f; *in = h->d; break;
    default: *out = h->d; *in = h->f; break;
    }
}

// element offset of (adapter a, layer l, projection p, factor 0 = A / 1 = B)
inline int64_t tf_tensor_off(const mlora_tf_t* h, int a, int l, int p, int factor) {
    const int r = h->ranks[a];
    int64_t off = h->ad_off_h[a] + (int64_t)l * r * h->per_layer_unit;
    for (int q = 0; q < p; ++q) {
        int out, in;
        proj_shape(h, q, &out, &in);
        off += (int64_t)r * (in + out);
    }
    if (factor) {
        int out, in;
        proj_shape(h, p, &out, &in);
        off += (int64_t)r * in;
    }
    return off;
}

// padded-row upper bound for a batch of n tokens
inline int tf_pad_rows(const mlora_tf_t* h, int64_t n) {
    int64_t busy = n < h->n_ad ? n : h->n_ad;
    int64_t rows = n + (int64_t)(TILE_M - 1) * busy;
    return (int)((rows + TILE_M - 1) / TILE_M * TILE_M);
}

GemmOperand opnd(const void* p, int64_t rows, int64_t cols, int64_t ld, int mn_major, int64_t ad_rows = 0,
                 int64_t shift = 0) {
    GemmOperand o;
    o.ptr = p; o.rows = rows; o.cols = cols; o.ld = ld; o.mn_major = mn_major; o.ad_rows = ad_rows;
    o.row_shift = shift;
    return o;
}

// Raster band height (row tiles) for an A operand with K columns: tiles in
// flight share B through L2 while a band of A (about 48 MB) stays resident.
int tf_band_for_k(int K) {
    if (K >= 65536) return 16;
    int tiles = (int)((48ll << 20) / (2ll * K)) / TILE_M;
    tiles &= ~1;
    return tiles < 8 ? 8 : (tiles > 64 ? 64 : tiles);
}

}  // namespace

// ----------------------------------------------------------------------------
// create / destroy
// ----------------------------------------------------------------------------
extern "C" int mlora_tf_create(const mlora_tf_config* cfg, const mlora_tf_init* init, mlora_tf_t** out) {
    if (!cfg || !init || !out) return tfail(MLORA_E_ARG, "NULL argument");
    *out = nullptr;
    if (cfg->vocab < 1 || cfg->d_model < 128 || cfg->d_model % 128 || cfg->d_ffn < 128 || cfg->d_ffn % 128 ||
        cfg->n_layers < 1 || cfg->n_layers > 64 || cfg->n_heads < 1 || cfg->n_kv_heads < 1 ||
        cfg->n_heads % cfg->n_kv_heads || cfg->n_heads > 256)
        return tfail(MLORA_E_ARG, "bad model shape (V=%d d=%d f=%d L=%d heads=%d/%d): d and f must be multiples "
                     "of 128, 1 <= L <= 64, n_kv_heads must divide n_heads", cfg->vocab, cfg->d_model, cfg->d_ffn,
                     cfg->n_layers, cfg->n_heads, cfg->n_kv_heads);
    if (cfg->head_dim != MLORA_TF_HEAD_DIM)
        return tfail(MLORA_E_ARG, "head_dim %d: only %d is supported", cfg->head_dim, MLORA_TF_HEAD_DIM);
    if (!(cfg->rope_theta > 1.f) || !(cfg->rms_eps > 0.f) || !std::isfinite(cfg->rope_theta))
        return tfail(MLORA_E_ARG, "rope_theta must be > 1 and rms_eps > 0");
    if (cfg->n_adapters < 1 || cfg->n_adapters > 1024 || !cfg->ranks || !cfg->alphas)
        return tfail(MLORA_E_ARG, "n_adapters must be 1..1024 with ranks and alphas");
    if (cfg->max_tokens < 1 || cfg->max_tokens > (1LL << 24))
        return tfail(MLORA_E_ARG, "max_tokens out of range (1 .. 2^24)");
    for (int a = 0; a < cfg->n_adapters; ++a) {
        const int r = cfg->ranks[a];
        if (r < 4 || r > MLORA_MAX_RANK || r % 4)
            return tfail(MLORA_E_ARG, "adapter %d: rank %d must be in 4..%d and a multiple of 4", a, r, MLORA_MAX_RANK);
        if (!std::isfinite(cfg->alphas[a])) return tfail(MLORA_E_ARG, "adapter %d: alpha not finite", a);
    }
    if (!init->E || !init->Wout || !init->final_norm || !init->attn_norm || !init->mlp_norm)
        return tfail(MLORA_E_ARG, "NULL base tensor");
    for (int p = 0; p < MLORA_TF_NPROJ; ++p) {
        if (!init->W[p]) return tfail(MLORA_E_ARG, "NULL weight array of projection %d", p);
        for (int l = 0; l < cfg->n_layers; ++l)
            if (!init->W[p][l]) return tfail(MLORA_E_ARG, "NULL weight of projection %d, layer %d", p, l);
    }
    for (int l = 0; l < cfg->n_layers; ++l)
        if (!init->attn_norm[l] || !init->mlp_norm[l]) return tfail(MLORA_E_ARG, "NULL norm gain of layer %d", l);

    int dev = 0;
    TF_CUDA(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    TF_CUDA(cudaGetDeviceProperties(&prop, dev));
    if (prop.major != 10 || !tc_engine_available())
        return tfail(MLORA_E_UNSUPPORTED, "the transformer model needs an sm_100-family GPU with TMA (found %d.%d)",
                     prop.major, prop.minor);

    mlora_tf_t* h = new mlora_tf();
    h->V = cfg->vocab; h->d = cfg->d_model; h->nh = cfg->n_heads; h->nkv = cfg->n_kv_heads; h->f = cfg->d_ffn;
    h->L = cfg->n_layers; h->n_ad = cfg->n_adapters; h->max_tokens = cfg->max_tokens;
    h->theta = cfg->rope_theta; h->eps = cfg->rms_eps;
    h->Q = h->nh * MLORA_TF_HEAD_DIM; h->KV = h->nkv * MLORA_TF_HEAD_DIM; h->Nqkv = h->Q + 2 * h->KV;
    h->num_sms = prop.multiProcessorCount;
    h->ranks.assign(cfg->ranks, cfg->ranks + cfg->n_adapters);
    h->alphas.assign(cfg->alphas, cfg->alphas + cfg->n_adapters);
    h->Vpad = (h->V + 63) / 64 * 64;
    h->n_nt = (h->V + 255) / 256;
    h->part_ld = (h->n_nt + 3) & ~3;
    h->gN[G_QKV] = h->Nqkv; h->gIn[G_QKV] = h->d;
    h->gN[G_O] = h->d;      h->gIn[G_O] = h->Q;
    h->gN[G_GU] = 2 * h->f; h->gIn[G_GU] = h->d;
    h->gN[G_D] = h->d;      h->gIn[G_D] = h->f;
    h->per_layer_unit = 0;
    for (int p = 0; p < MLORA_TF_NPROJ; ++p) {
        int o_, i_;
        proj_shape(h, p, &o_, &i_);
        h->per_layer_unit += o_ + i_;
    }

    const int n_ad = h->n_ad, L = h->L, d = h->d, f = h->f, V = h->V;
    h->max_pad = tf_pad_rows(h, h->max_tokens);
    h->max_tiles = h->max_pad / TILE_M;
    h->max_chunks = h->max_pad / GRAD_CHUNK + n_ad + 1;
    h->max_blocks = (int)((h->max_tokens + ROUTE_BLOCK - 1) / ROUTE_BLOCK);
    const int64_t MP = h->max_pad;
    const size_t B2 = sizeof(bf16);

    int rc = MLORA_OK;
#define TA(ptr, count) do { if ((rc = tf_alloc_t(h, &(ptr), (size_t)(count))) != MLORA_OK) goto fail_out; } while (0)
    {
        TA(h->E, (size_t)V * d);
        TA(h->Wout, (size_t)V * d);
        TA(h->gfinal, d);
        h->gattn.resize(L); h->gmlp.resize(L);
        for (int l = 0; l < L; ++l) { TA(h->gattn[l], d); TA(h->gmlp[l], d); }
        for (int g = 0; g < NGROUPS; ++g) {
            h->W[g].resize(L); h->WT[g].resize(L);
            for (int l = 0; l < L; ++l) {
                TA(h->W[g][l], (size_t)h->gN[g] * h->gIn[g]);
                TA(h->WT[g][l], (size_t)h->gN[g] * h->gIn[g]);
            }
        }
        h->ad_off_h.resize(n_ad + 1);
        h->ad_off_h[0] = 0;
        for (int a = 0; a < n_ad; ++a)
            h->ad_off_h[a + 1] = h->ad_off_h[a] + (int64_t)L * h->ranks[a] * h->per_layer_unit;
        h->n_params = h->ad_off_h[n_ad];
        TA(h->P, h->n_params); TA(h->G, h->n_params); TA(h->M, h->n_params); TA(h->Vm, h->n_params);
        TA(h->ad_off, n_ad + 1);
        TA(h->ranks_d, n_ad);
        TA(h->gamma_d, n_ad);
        TA(h->grad_off, (size_t)L * MLORA_TF_NPROJ * 2 * n_ad);
        TA(h->step, n_ad);
        TA(h->touched, n_ad);
        TA(h->nonfinite, n_ad);
        TA(h->sel_mask, n_ad);
        TA(h->adam_tab, n_ad);
        for (int g = 0; g < NGROUPS; ++g) {
            const int64_t kx = GROUP_KX[g];
            // at least 256 rows: the 256-wide single-CTA tile reads whole boxes
            h->As_rows[g] = (int64_t)n_ad * kx < 256 ? 256 : (int64_t)n_ad * kx;
            h->As_layer[g] = h->As_rows[g] * h->gIn[g];
            h->Bs_layer[g] = (int64_t)n_ad * h->gN[g] * kx;
            TA(h->As[g], (size_t)L * h->As_layer[g]);
            TA(h->Bs[g], (size_t)L * h->Bs_layer[g]);
        }
        TA(h->rb.blk_cnt, (size_t)(h->max_blocks > 0 ? h->max_blocks : 1) * n_ad);
        TA(h->rb.perm_pad, MP);
        TA(h->rb.inv, h->max_tokens);
        TA(h->rb.seg_off, n_ad + 1);
        TA(h->rb.pad_off, n_ad + 1);
        TA(h->rb.tile_ad, h->max_tiles);
        TA(h->rb.meta, 4);
        TA(h->rb.chunks, h->max_chunks);
        h->rb.max_pad = h->max_pad; h->rb.max_tiles = h->max_tiles; h->rb.max_chunks = h->max_chunks;
        TA(h->pos_pad, MP);
        TA(h->seq_start, MP);
        TA(h->rope_cs, (size_t)h->max_tokens * 64);
        h->x1.resize(L); h->vqkv.resize(L); h->qkv.resize(L); h->o.resize(L); h->vo.resize(L);
        h->x2.resize(L); h->vgu.resize(L); h->gu.resize(L); h->act.resize(L); h->vd.resize(L);
        h->lseT.resize(L); h->snap1.resize(L); h->snap2.resize(L); h->rstd1.resize(L); h->rstd2.resize(L);
        for (int l = 0; l < L; ++l) {
            TA(h->x1[l], MP * d); TA(h->vqkv[l], MP * 3 * RP); TA(h->qkv[l], MP * h->Nqkv);
            TA(h->o[l], MP * h->Q); TA(h->vo[l], MP * RP); TA(h->x2[l], MP * d); TA(h->vgu[l], MP * 2 * RP);
            TA(h->gu[l], MP * 2 * f); TA(h->act[l], MP * f); TA(h->vd[l], MP * RP);
            TA(h->lseT[l], (size_t)h->nh * MP); TA(h->snap1[l], MP * d); TA(h->snap2[l], MP * d);
            TA(h->rstd1[l], MP); TA(h->rstd2[l], MP);
        }
        TA(h->xf, MP * d); TA(h->snapf, MP * d); TA(h->rstdf, MP);
        TA(h->h32, MP * d); TA(h->dh32, MP * d); TA(h->dxn32, MP * d);
        TA(h->dhb, MP * d); TA(h->wbuf, MP * 3 * RP); TA(h->dgu, MP * 2 * f); TA(h->dO, MP * h->Q);
        TA(h->dqkv, MP * h->Nqkv); TA(h->embed_bf, MP * d);
        TA(h->DT, (size_t)h->nh * MP);
        TA(h->part, (size_t)MP * h->part_ld);
        TA(h->mt, (size_t)MP * h->part_ld);
        TA(h->zt, MP); TA(h->lse, MP); TA(h->gvec, MP); TA(h->tgt_pad, MP);
        h->nc_tiles = h->max_tiles < 128 ? h->max_tiles : 128;
        TA(h->dz[0], (size_t)h->nc_tiles * TILE_M * h->Vpad);   // the kept-logits mode adds its buffers
        TA(h->val_row, MP);
        TA(h->status, 1);
        TA(h->tile_counter, 1);
        if (cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess) {
            h->side = nullptr;
            rc = tfail(MLORA_E_CUDA, "cudaStreamCreate failed");
            goto fail_out;
        }
        for (int b = 0; b < 2; ++b)
            if (cudaEventCreateWithFlags(&h->ev_comb[b], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&h->ev_dz[b], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&h->ev_dh[b], cudaEventDisableTiming) != cudaSuccess) {
                rc = tfail(MLORA_E_CUDA, "cudaEventCreate failed");
                goto fail_out;
            }
    }
#undef TA
    if ((rc = [&]() -> int {
             cudaStream_t s = 0;
             TF_CUDA(cudaMemcpyAsync(h->E, init->E, (size_t)V * d * B2, cudaMemcpyDeviceToDevice, s));
             TF_CUDA(cudaMemcpyAsync(h->Wout, init->Wout, (size_t)V * d * B2, cudaMemcpyDeviceToDevice, s));
             TF_CUDA(cudaMemcpyAsync(h->gfinal, init->final_norm, d * B2, cudaMemcpyDeviceToDevice, s));
             for (int l = 0; l < L; ++l) {
                 TF_CUDA(cudaMemcpyAsync(h->gattn[l], init->attn_norm[l], d * B2, cudaMemcpyDeviceToDevice, s));
                 TF_CUDA(cudaMemcpyAsync(h->gmlp[l], init->mlp_norm[l], d * B2, cudaMemcpyDeviceToDevice, s));
                 // q, k, v stacked
                 bf16* wq = h->W[G_QKV][l];
                 TF_CUDA(cudaMemcpyAsync(wq, init->W[MLORA_TF_Q][l], (size_t)h->Q * d * B2, cudaMemcpyDeviceToDevice, s));
                 TF_CUDA(cudaMemcpyAsync(wq + (size_t)h->Q * d, init->W[MLORA_TF_K][l], (size_t)h->KV * d * B2,
                                         cudaMemcpyDeviceToDevice, s));
                 TF_CUDA(cudaMemcpyAsync(wq + (size_t)(h->Q + h->KV) * d, init->W[MLORA_TF_V][l],
                                         (size_t)h->KV * d * B2, cudaMemcpyDeviceToDevice, s));
                 TF_CUDA(cudaMemcpyAsync(h->W[G_O][l], init->W[MLORA_TF_O][l], (size_t)d * h->Q * B2,
                                         cudaMemcpyDeviceToDevice, s));
                 // gate / up interleaved in blocks of GU_ILV rows
                 for (int sub = 0; sub < 2; ++sub)
                     TF_CUDA(cudaMemcpy2DAsync(h->W[G_GU][l] + (size_t)sub * GU_ILV * d, 2 * GU_ILV * d * B2,
                                               init->W[sub ? MLORA_TF_UP : MLORA_TF_GATE][l], GU_ILV * d * B2,
                                               GU_ILV * d * B2, f / GU_ILV, cudaMemcpyDeviceToDevice, s));
                 TF_CUDA(cudaMemcpyAsync(h->W[G_D][l], init->W[MLORA_TF_DOWN][l], (size_t)d * f * B2,
                                         cudaMemcpyDeviceToDevice, s));
                 for (int g = 0; g < NGROUPS; ++g) {
                     launch_transpose<bf16>(h->W[g][l], h->WT[g][l], h->gN[g], h->gIn[g], s);
                     ++h->launches;
                 }
             }
             TF_CUDA(cudaMemsetAsync(h->P, 0, sizeof(float) * h->n_params, s));
             TF_CUDA(cudaMemsetAsync(h->G, 0, sizeof(float) * h->n_params, s));
             TF_CUDA(cudaMemsetAsync(h->M, 0, sizeof(float) * h->n_params, s));
             TF_CUDA(cudaMemsetAsync(h->Vm, 0, sizeof(float) * h->n_params, s));
             for (int a = 0; a < n_ad; ++a)
                 for (int l = 0; l < L; ++l)
                     for (int p = 0; p < MLORA_TF_NPROJ; ++p) {
                         int o_, i_;
                         proj_shape(h, p, &o_, &i_);
                         const int r = h->ranks[a];
                         const float* srcA = init->A[p] ? init->A[p][a * L + l] : nullptr;
                         const float* srcB = init->B[p] ? init->B[p][a * L + l] : nullptr;
                         if (srcA)
                             TF_CUDA(cudaMemcpyAsync(h->P + tf_tensor_off(h, a, l, p, 0), srcA, sizeof(float) * r * i_,
                                                     cudaMemcpyDeviceToDevice, s));
                         if (srcB)
                             TF_CUDA(cudaMemcpyAsync(h->P + tf_tensor_off(h, a, l, p, 1), srcB, sizeof(float) * o_ * r,
                                                     cudaMemcpyDeviceToDevice, s));
                     }
             for (int g = 0; g < NGROUPS; ++g) {
                 TF_CUDA(cudaMemsetAsync(h->As[g], 0, (size_t)L * h->As_layer[g] * B2, s));
                 TF_CUDA(cudaMemsetAsync(h->Bs[g], 0, (size_t)L * h->Bs_layer[g] * B2, s));
             }
             // where each projection's factors are mirrored
             for (int p = 0; p < MLORA_TF_NPROJ; ++p) {
                 const int g = GROUP_OF[p];
                 TfMirrorProj& m = h->mirror.p[p];
                 int o_, i_;
                 proj_shape(h, p, &o_, &i_);
                 m.A = h->As[g]; m.B = h->Bs[g];
                 m.a_layer = h->As_layer[g]; m.b_layer = h->Bs_layer[g];
                 m.in = i_; m.out = o_; m.kx = GROUP_KX[g]; m.sub = SUB_OF[p]; m.n_rows = h->gN[g];
                 m.row_off = (p == MLORA_TF_K) ? h->Q : (p == MLORA_TF_V ? h->Q + h->KV : 0);
                 m.ilv = (g == G_GU) ? GU_ILV : 0;
             }
             h->mirror.sum_in_out = h->per_layer_unit;
             std::vector<float> gam(n_ad);
             for (int a = 0; a < n_ad; ++a) gam[a] = h->alphas[a] / (float)h->ranks[a];
             std::vector<int64_t> goff((size_t)L * MLORA_TF_NPROJ * 2 * n_ad);
             for (int l = 0; l < L; ++l)
                 for (int p = 0; p < MLORA_TF_NPROJ; ++p)
                     for (int fct = 0; fct < 2; ++fct)
                         for (int a = 0; a < n_ad; ++a)
                             goff[(((size_t)l * MLORA_TF_NPROJ + p) * 2 + fct) * n_ad + a] = tf_tensor_off(h, a, l, p, fct);
             // rotary table: cs[pos][i] = (cos, sin)(pos * theta^(-i/64)), angles in double
             std::vector<float2> cs((size_t)h->max_tokens * 64);
             for (int64_t pos = 0; pos < h->max_tokens; ++pos)
                 for (int i = 0; i < 64; ++i) {
                     const double ang = (double)pos * std::pow((double)h->theta, -(double)i / 64.0);
                     cs[(size_t)pos * 64 + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
                 }
             TF_CUDA(cudaMemcpy(h->rope_cs, cs.data(), sizeof(float2) * cs.size(), cudaMemcpyHostToDevice));
             TF_CUDA(cudaMemcpy(h->ad_off, h->ad_off_h.data(), sizeof(int64_t) * (n_ad + 1), cudaMemcpyHostToDevice));
             TF_CUDA(cudaMemcpy(h->ranks_d, h->ranks.data(), sizeof(int) * n_ad, cudaMemcpyHostToDevice));
             TF_CUDA(cudaMemcpy(h->gamma_d, gam.data(), sizeof(float) * n_ad, cudaMemcpyHostToDevice));
             TF_CUDA(cudaMemcpy(h->grad_off, goff.data(), sizeof(int64_t) * goff.size(), cudaMemcpyHostToDevice));
             TF_CUDA(cudaMemset(h->step, 0, sizeof(int64_t) * n_ad));
             TF_CUDA(cudaMemset(h->touched, 0, sizeof(int) * n_ad));
             TF_CUDA(cudaMemset(h->nonfinite, 0, sizeof(int) * n_ad));
             TF_CUDA(cudaMemset(h->status, 0, sizeof(int)));
             TF_CUDA(cudaMemset(h->part, 0, sizeof(float) * (size_t)MP * h->part_ld));
             TF_CUDA(cudaMemset(h->mt, 0, sizeof(float) * (size_t)MP * h->part_ld));
             TF_CUDA(cudaMemset(h->dz[0], 0, (size_t)h->nc_tiles * TILE_M * h->Vpad * B2));
             launch_tf_adam(n_ad, h->ad_off, h->ranks_d, h->n_params, h->adam_tab, h->P, h->G, h->M, h->Vm, 0.f, 0.f,
                            0.f, 0.f, 0.f, h->mirror, 1, h->num_sms, s);
             ++h->launches;
             TF_CUDA(cudaGetLastError());
             TF_CUDA(cudaDeviceSynchronize());
             return MLORA_OK;
         }()) != MLORA_OK)
        goto fail_out;
    *out = h;
    return MLORA_OK;
fail_out:
    tf_free_all(h);
    delete h;
    return rc;
}

extern "C" int mlora_tf_destroy(mlora_tf_t* h) {
    if (!h) return MLORA_OK;
    cudaDeviceSynchronize();
    tf_free_all(h);
    delete h;
    return MLORA_OK;
}

extern "C" int64_t mlora_tf_kernel_launches(const mlora_tf_t* h) { return h ? h->launches : 0; }
extern "C" int64_t mlora_tf_device_bytes(const mlora_tf_t* h) { return h ? h->bytes : 0; }

// ----------------------------------------------------------------------------
// one step
// ----------------------------------------------------------------------------
namespace {

int tf_gemm(mlora_tf_t* h, GemmParams& p, cudaStream_t s, int cls) {
    TfProf ps(h, s, cls);
    p.tile_counter = h->tile_counter;
    const cudaError_t e = launch_tc_gemm(p, s, h->num_sms, h->status);
    if (e != cudaSuccess) return tfail(MLORA_E_CUDA, "tensor-core GEMM launch: %s", cudaGetErrorString(e));
    ++h->launches;
    return MLORA_OK;
}

// dense GEMM over the padded token rows of the current batch
GemmParams tf_dense(mlora_tf_t* h, int mt_upper, int N, int K) {
    GemmParams p;
    p.M = mt_upper * TILE_M;
    p.N = N; p.K = K; p.Kx = 0;
    p.group_m = tf_band_for_k(K);
    p.mtiles_dev = h->rb.meta;
    p.mt_base = 0; p.mt_count = mt_upper;
    p.tile_ad = h->rb.tile_ad;
    return p;
}

// Per projection group g of layer l: the shadows of its LoRA factors.
const bf16* shadowA(const mlora_tf_t* h, int g, int l) { return h->As[g] + (size_t)l * h->As_layer[g]; }
const bf16* shadowB(const mlora_tf_t* h, int g, int l) { return h->Bs[g] + (size_t)l * h->Bs_layer[g]; }

// v = gamma_a [A_s x]_s for every member s of group g (tinker-ticks, "How the
// SGMV kernel works": the shrink), x [rows x in_g]
int shrink_fwd(mlora_tf_t* h, int g, int l, const bf16* x, bf16* v, int mt_upper, cudaStream_t s) {
    const int kx = GROUP_KX[g], in = h->gIn[g];
    GemmParams p = tf_dense(h, mt_upper, kx, in);
    p.A = opnd(x, h->max_pad, in, in, 0);
    p.B = opnd(shadowA(h, g, l), h->As_rows[g], in, in, 0, kx);
    p.ep.kind = EPI_SHRINK; p.ep.out0 = v; p.ep.ld0 = kx; p.ep.gamma = h->gamma_d;
    return tf_gemm(h, p, s, MLORA_TF_PROF_SHRINK);
}

// y = x W_g^T + v B_g^T: the shared base GEMM with the per-adapter expand as
// extra K blocks (tinker-ticks, "Forward pass: what actually happens")
GemmParams proj_fwd(mlora_tf_t* h, int g, int l, const bf16* x, const bf16* v, int mt_upper) {
    const int kx = GROUP_KX[g], in = h->gIn[g], N = h->gN[g];
    GemmParams p = tf_dense(h, mt_upper, N, in);
    p.A = opnd(x, h->max_pad, in, in, 0);
    p.B = opnd(h->W[g][l], N, in, in, 0);
    p.Kx = kx;
    p.Ax = opnd(v, h->max_pad, kx, kx, 0);
    p.Bx = opnd(shadowB(h, g, l), (int64_t)h->n_ad * N, kx, kx, 0, N);
    return p;
}

// w = gamma_a [B_s^T dy_s]_s  (dy [rows x N_g])
int shrink_bwd(mlora_tf_t* h, int g, int l, const bf16* dy, int mt_upper, cudaStream_t s) {
    const int kx = GROUP_KX[g], N = h->gN[g];
    GemmParams p = tf_dense(h, mt_upper, kx, N);
    p.A = opnd(dy, h->max_pad, N, N, 0);
    p.B = opnd(shadowB(h, g, l), (int64_t)h->n_ad * N, kx, kx, 1, N);
    p.ep.kind = EPI_SHRINK; p.ep.out0 = h->wbuf; p.ep.ld0 = kx; p.ep.gamma = h->gamma_d;
    return tf_gemm(h, p, s, MLORA_TF_PROF_SHRINK);
}

// dx = dy W_g + w A_g  (K-major copy of W_g; A_g read MN-major)
GemmParams proj_bwd(mlora_tf_t* h, int g, int l, const bf16* dy, int mt_upper) {
    const int kx = GROUP_KX[g], in = h->gIn[g], N = h->gN[g];
    GemmParams p = tf_dense(h, mt_upper, in, N);
    p.A = opnd(dy, h->max_pad, N, N, 0);
    p.B = opnd(h->WT[g][l], in, N, N, 0);
    p.Kx = kx;
    p.Ax = opnd(h->wbuf, h->max_pad, kx, kx, 0);
    p.Bx = opnd(shadowA(h, g, l), h->As_rows[g], in, in, 1, kx);
    return p;
}

// grad[a] (+)= X_seg^T Y_seg over each adapter's token chunks (fp32 atomics).
// ncols > RP: Y holds the factors of consecutive projections proj, proj + 1, ..
// side by side (RP columns each), and one pass over X feeds all of them.
int tf_grad(mlora_tf_t* h, int mp, int Dout, GemmOperand X, GemmOperand Y, int l, int proj, int factor, int trans,
            int ilv, int sub, cudaStream_t s, int ncols = RP) {
    GemmParams p;
    p.M = Dout; p.N = ncols; p.K = 0;
    p.force_bn64 = ncols <= RP;   // several members: one 256-column tile reads each X block once
    p.grouped = 1;
    p.chunks = h->rb.chunks;
    p.nchunks_dev = h->rb.meta + 1;
    p.max_chunks = mp / GRAD_CHUNK + (mp / TILE_M < h->n_ad ? mp / TILE_M : h->n_ad) + 1;
    if (p.max_chunks > h->max_chunks) p.max_chunks = h->max_chunks;
    p.A = X;
    p.B = Y;
    p.ep.kind = EPI_GRAD;
    p.ep.grad = h->G;
    p.ep.grad_off = h->grad_off + (((size_t)l * MLORA_TF_NPROJ + proj) * 2 + factor) * h->n_ad;
    p.ep.ranks = h->ranks_d;
    p.ep.grad_trans = trans;
    p.ep.grad_M = Dout;
    p.ep.grad_ilv = ilv;
    p.ep.grad_sub = sub;
    // the next projection's offsets: the same factor, one projection on
    p.ep.grad_sub_stride = ncols > RP ? 2 * h->n_ad : 0;
    p.ep.nonfinite = h->nonfinite;
    return tf_gemm(h, p, s, MLORA_TF_PROF_GRAD);
}

// Gradients of group g's projections: dB_p += dy_p^T v_p (v includes gamma),
// dA_p += w_p^T x.  dy [rows x N_g], v / w [rows x kx], the members' factors
// side by side.  Every dA of a group reads the group's input x once (one
// reduction over all members' w); gate and up also share one pass over the
// interleaved d gate|up (rows of block parity s to member s); q, k and v
// read their own column slices of dq|dk|dv.
int group_grads(mlora_tf_t* h, int g, int l, int mp, const bf16* dy, const bf16* v, const bf16* x, cudaStream_t s) {
    static constexpr int FIRST[NGROUPS] = {MLORA_TF_Q, MLORA_TF_O, MLORA_TF_GATE, MLORA_TF_DOWN};
    const int kx = GROUP_KX[g], N = h->gN[g], in = h->gIn[g], first = FIRST[g];
    const int64_t MP = h->max_pad;
    int rc;
    if (g == G_GU) {
        rc = tf_grad(h, mp, N, opnd(dy, MP, N, N, 1), opnd(v, MP, kx, kx, 1), l, first, 1, 0, GU_ILV, 0, s, kx);
    } else {
        rc = MLORA_OK;
        for (int sub = 0; sub * RP < kx && rc == MLORA_OK; ++sub) {
            const int proj = first + sub;
            int out, in_p;
            proj_shape(h, proj, &out, &in_p);
            const int off = (proj == MLORA_TF_K) ? h->Q : (proj == MLORA_TF_V ? h->Q + h->KV : 0);
            rc = tf_grad(h, mp, out, opnd(dy + off, MP, out, N, 1), opnd(v + RP * sub, MP, RP, kx, 1), l, proj, 1,
                         0, 0, 0, s);
        }
    }
    if (rc) return rc;
    return tf_grad(h, mp, in, opnd(x, MP, in, in, 1), opnd(h->wbuf, MP, kx, kx, 1), l, first, 0, 1, 0, 0, s, kx);
}

int tf_norm_fwd(mlora_tf_t* h, const float* x, const bf16* gain, bf16* y, float* rstd, int mp, cudaStream_t s) {
    TfProf ps(h, s, MLORA_TF_PROF_NORM);
    launch_rmsnorm_fwd(x, gain, h->d, h->eps, h->rb.meta, mp, y, rstd, s);
    ++h->launches;
    return MLORA_OK;
}

int tf_norm_bwd(mlora_tf_t* h, const float* snap, const bf16* gain, const float* rstd, int accumulate, int mp,
                cudaStream_t s) {
    TfProf ps(h, s, MLORA_TF_PROF_NORM);
    launch_rmsnorm_bwd(h->dxn32, snap, gain, rstd, h->d, h->rb.meta, mp, accumulate, h->dh32, h->dhb, s);
    ++h->launches;
    return MLORA_OK;
}

AttnArgs attn_args(mlora_tf_t* h, int l, int mp) {
    AttnArgs a;
    a.qkv = h->qkv[l];
    a.n_heads = h->nh;
    a.n_kv = h->nkv;
    a.max_rows = mp;
    a.seq_start = h->seq_start;
    a.meta = h->rb.meta;
    a.o = h->o[l];
    a.lseT = h->lseT[l];
    a.DT = h->DT;
    a.ld_t = h->max_pad;
    a.dO = h->dO;
    a.dqkv = h->dqkv;
    a.num_sms = h->num_sms;
    a.counter = h->tile_counter;
    return a;
}

int tf_step(mlora_tf_t* h, const mlora_tf_batch* b, const LossArgs& la, float* logprobs_out, double* loss_out,
            bool backward, cudaStream_t s) {
    const int64_t N = b->n_tokens;
    const int n_ad = h->n_ad, L = h->L, d = h->d, f = h->f, V = h->V;
    const int64_t MP = h->max_pad;
    const int mp = tf_pad_rows(h, N);
    const int mt_upper = mp / TILE_M;
    int rc;

    if (logprobs_out && N > 0) TF_CUDA(cudaMemsetAsync(logprobs_out, 0xff, sizeof(float) * N, s));
    if (N == 0) {
        if (loss_out) TF_CUDA(cudaMemsetAsync(loss_out, 0, sizeof(double) * n_ad, s));
        return MLORA_OK;
    }
    {
        TfProf ps(h, s, MLORA_TF_PROF_ROUTING);
        launch_routing(b->adapter_ids, N, n_ad, h->rb, backward ? h->touched : nullptr, h->status, s, &h->launches,
                       GRAD_CHUNK);
        // positions bound the sequence lengths the stored dS layout holds
        launch_tf_rows(h->rb.perm_pad, h->rb.meta, h->rb.tile_ad, h->rb.pad_off, b->positions, b->adapter_ids,
                       h->attn_ds ? h->attn_max_seq : (int)h->max_tokens, mp, h->pos_pad, h->seq_start, h->status,
                       s);
        ++h->launches;
    }
    // The fp32 residual stream.  With a backward to follow, every value that
    // feeds an RMSNorm is kept: the residual GEMMs read one version and write
    // the next (embedding -> snap1[0] -> snap2[0] -> snap1[1] ... -> snapf),
    // so the norms' backward finds its inputs without a copy; a forward alone
    // updates h32 in place.
    float* cur = backward ? h->snap1[0] : h->h32;
    auto resid_to = [&](float* next, GemmParams& p) {
        p.ep.kind = EPI_RESID; p.ep.f32 = next; p.ep.f32_in = cur; p.ep.ldf = d;
        cur = next;
    };
    {
        TfProf ps(h, s, MLORA_TF_PROF_EMBED);
        launch_embed<bf16>(h->rb.perm_pad, h->rb.meta, mp, b->tokens, b->targets, h->E, V, d, h->embed_bf, cur,
                           h->tgt_pad, h->status, s);
        ++h->launches;
    }
    for (int l = 0; l < L; ++l) {
        // attention sub-block
        if ((rc = tf_norm_fwd(h, cur, h->gattn[l], h->x1[l], h->rstd1[l], mp, s))) return rc;
        if ((rc = shrink_fwd(h, G_QKV, l, h->x1[l], h->vqkv[l], mt_upper, s))) return rc;
        {
            GemmParams p = proj_fwd(h, G_QKV, l, h->x1[l], h->vqkv[l], mt_upper);
            p.ep.kind = EPI_STORE; p.ep.out0 = h->qkv[l]; p.ep.ld0 = h->Nqkv;
            if ((rc = tf_gemm(h, p, s, MLORA_TF_PROF_QKV))) return rc;
        }
        {
            TfProf ps(h, s, MLORA_TF_PROF_ROPE);   // q and k heads are adjacent columns
            launch_rope(h->qkv[l], h->Nqkv, 0, h->nh + h->nkv, h->pos_pad, h->rope_cs, h->rb.meta, mp, 0, s);
            ++h->launches;
        }
        {
            TfProf ps(h, s, MLORA_TF_PROF_ATTN_FWD);
            const cudaError_t e = launch_attention_fwd(attn_args(h, l, mp), h->status, s);
            if (e != cudaSuccess) return tfail(MLORA_E_CUDA, "attention forward launch: %s", cudaGetErrorString(e));
            ++h->launches;
        }
        if ((rc = shrink_fwd(h, G_O, l, h->o[l], h->vo[l], mt_upper, s))) return rc;
        {
            GemmParams p = proj_fwd(h, G_O, l, h->o[l], h->vo[l], mt_upper);
            resid_to(backward ? h->snap2[l] : cur, p);
            if ((rc = tf_gemm(h, p, s, MLORA_TF_PROF_O))) return rc;
        }
        // MLP sub-block
        if ((rc = tf_norm_fwd(h, cur, h->gmlp[l], h->x2[l], h->rstd2[l], mp, s))) return rc;
        if ((rc = shrink_fwd(h, G_GU, l, h->x2[l], h->vgu[l], mt_upper, s))) return rc;
        {
            GemmParams p = proj_fwd(h, G_GU, l, h->x2[l], h->vgu[l], mt_upper);
            p.ep.kind = EPI_SWIGLU; p.ep.out0 = h->gu[l]; p.ep.ld0 = 2 * f; p.ep.out1 = h->act[l]; p.ep.ld1 = f;
            if ((rc = tf_gemm(h, p, s, MLORA_TF_PROF_GATEUP))) return rc;
        }
        if ((rc = shrink_fwd(h, G_D, l, h->act[l], h->vd[l], mt_upper, s))) return rc;
        {
            GemmParams p = proj_fwd(h, G_D, l, h->act[l], h->vd[l], mt_upper);
            resid_to(!backward ? cur : (l + 1 < L ? h->snap1[l + 1] : h->snapf), p);
            if ((rc = tf_gemm(h, p, s, MLORA_TF_PROF_DOWN))) return rc;
        }
    }
    if ((rc = tf_norm_fwd(h, cur, h->gfinal, h->xf, h->rstdf, mp, s))) return rc;

    // LM head (Tinker API Implementation on TPUs, section 10.3-10.4): per-tile
    // log-sum-exp partials and the target logit over all rows; the backward
    // walks the rows in chunks and by default recomputes each chunk's logits
    // with a second GEMM whose epilogue writes dz = g (onehot - softmax), then
    // dxf = dz Wout.  In the kept-logits mode the forward GEMM of each chunk
    // also stores fp16 e = exp(z - tile max) and the dz pass of chunk i runs on the side
    // stream beside chunk i+1's GEMMs (as in the MLP model's step).
    auto lm_fwd_params = [&](int c0, int cnt) {
        GemmParams p = tf_dense(h, mt_upper, V, d);
        p.mt_base = c0; p.mt_count = cnt;
        p.A = opnd(h->xf, MP, d, d, 0);
        p.B = opnd(h->Wout, V, d, d, 0);
        p.ep.kind = EPI_LMFWD; p.ep.part = h->part; p.ep.zt = h->zt; p.ep.tgt = h->tgt_pad;
        p.ep.part_ld = h->part_ld; p.ep.V = V; p.ep.Vpad = h->Vpad;
        p.ep.mt = h->mt; p.ep.lm_bn = 256;     // the partials' tile width (n_nt above)
        return p;
    };
    if (!backward || !h->lm_keep) {
        GemmParams p = lm_fwd_params(0, mt_upper);
        if ((rc = tf_gemm(h, p, s, MLORA_TF_PROF_LM_FWD))) return rc;
        {
            TfProf ps(h, s, MLORA_TF_PROF_LOSS);
            launch_combine_loss(la, h->part, h->n_nt, h->part_ld, h->zt, h->rb.perm_pad, h->tgt_pad, h->rb.meta, 0,
                                mt_upper, logprobs_out, h->lse, h->gvec, h->val_row, h->num_sms, s);
            ++h->launches;
        }
        if (loss_out) {
            TfProf ps(h, s, MLORA_TF_PROF_OTHER);
            launch_loss_reduce(h->val_row, h->rb.pad_off, n_ad, loss_out, s);
            ++h->launches;
        }
        if (!backward) return MLORA_OK;
    }
    // chunks of at most nc_tiles row tiles, sized so that dh fills whole waves
    // (dh: 256 x 512 tiles at the vocabulary's K)
    const int dh_nt = h->Vpad >= 65536 && d % 512 == 0 ? d / 512 : (d + 255) / 256;
    const int chunk = lm_chunk_tiles(mt_upper, h->nc_tiles, dh_nt, h->num_sms / 2);
    const int nch = (mt_upper + chunk - 1) / chunk;
    auto chunk_rows = [&](int i, int& c0, int& cnt) {
        c0 = i * chunk;
        cnt = mt_upper - c0 < chunk ? mt_upper - c0 : chunk;
    };
    auto dh_params = [&](int c0, int cnt, const bf16* dzb) {
        GemmParams p = tf_dense(h, mt_upper, d, h->Vpad);
        p.mt_base = c0; p.mt_count = cnt;
        p.A = opnd(dzb, (int64_t)h->nc_tiles * TILE_M, h->Vpad, h->Vpad, 0, 0, -(int64_t)c0 * TILE_M);
        p.B = opnd(h->Wout, V, d, d, 1);
        p.ep.kind = EPI_STORE2; p.ep.f32 = h->dxn32; p.ep.ldf = d; p.ep.out0 = nullptr;
        return p;
    };
    if (!h->lm_keep) {
        // recompute: chunk i's logits again, dz from them in the epilogue, then dxf
        for (int i = 0; i < nch; ++i) {
            int c0, cnt;
            chunk_rows(i, c0, cnt);
            {
                GemmParams p = lm_fwd_params(c0, cnt);
                p.ep.kind = EPI_LMDZ; p.ep.gv = h->gvec; p.ep.lse = h->lse;
                p.ep.out0 = h->dz[0]; p.ep.ld0 = h->Vpad; p.ep.out_row_shift = -(int64_t)c0 * TILE_M;
                p.ep.out_rows = (int64_t)h->nc_tiles * TILE_M;
                if ((rc = tf_gemm(h, p, s, MLORA_TF_PROF_LM_DZ))) return rc;
            }
            GemmParams p = dh_params(c0, cnt, h->dz[0]);
            if ((rc = tf_gemm(h, p, s, MLORA_TF_PROF_LM_DH))) return rc;
        }
    }
    auto queue_dh = [&](int i) -> int {
        int c0, cnt;
        chunk_rows(i, c0, cnt);
        const int buf = i & 1;
        TF_CUDA(cudaStreamWaitEvent(s, h->ev_dz[buf], 0));
        GemmParams p = dh_params(c0, cnt, h->dz[buf]);
        const int r = tf_gemm(h, p, s, MLORA_TF_PROF_LM_DH);
        if (r) return r;
        TF_CUDA(cudaEventRecord(h->ev_dh[buf], s));
        return MLORA_OK;
    };
    for (int i = 0; i < nch && h->lm_keep; ++i) {
        int c0, cnt;
        chunk_rows(i, c0, cnt);
        const int buf = i & 1;
        {
            GemmParams p = lm_fwd_params(c0, cnt);
            p.ep.out0 = h->zbuf[buf]; p.ep.ld0 = h->Vpad; p.ep.out_row_shift = -(int64_t)c0 * TILE_M;
            p.ep.out_rows = (int64_t)h->nc_tiles * TILE_M;
            p.ep.e16 = 1;
            if ((rc = tf_gemm(h, p, s, MLORA_TF_PROF_LM_FWD))) return rc;
        }
        {
            TfProf ps(h, s, MLORA_TF_PROF_LOSS);
            launch_combine_loss(la, h->part, h->n_nt, h->part_ld, h->zt, h->rb.perm_pad, h->tgt_pad, h->rb.meta, c0,
                                cnt, logprobs_out, h->lse, h->gvec, h->val_row, h->num_sms, s);
            ++h->launches;
        }
        TF_CUDA(cudaEventRecord(h->ev_comb[buf], s));
        TF_CUDA(cudaStreamWaitEvent(h->side, h->ev_comb[buf], 0));
        if (i >= 2) TF_CUDA(cudaStreamWaitEvent(h->side, h->ev_dh[buf], 0));
        {
            TfProf ps(h, h->side, MLORA_TF_PROF_LM_DZ);
            launch_lm_dz_e16(h->zbuf[buf], h->dz[buf], h->Vpad, V, h->Vpad, h->mt, h->part_ld, 256, h->gvec,
                             h->lse, h->tgt_pad, h->rb.meta, c0 * TILE_M, cnt * TILE_M, h->side);
            ++h->launches;
        }
        TF_CUDA(cudaEventRecord(h->ev_dz[buf], h->side));
        if (i >= 1 && (rc = queue_dh(i - 1))) return rc;
    }
    if (h->lm_keep) {
        if ((rc = queue_dh(nch - 1))) return rc;
        if (loss_out) {
            TfProf ps(h, s, MLORA_TF_PROF_OTHER);
            launch_loss_reduce(h->val_row, h->rb.pad_off, n_ad, loss_out, s);
            ++h->launches;
        }
    }
    // through the final norm: dh = RMSNorm_final'(dxf)
    if ((rc = tf_norm_bwd(h, h->snapf, h->gfinal, h->rstdf, 0, mp, s))) return rc;

    for (int l = L - 1; l >= 0; --l) {
        // h = h_mid + P_down(silu(gate) * up)
        if ((rc = shrink_bwd(h, G_D, l, h->dhb, mt_upper, s))) return rc;
        {
            GemmParams p = proj_bwd(h, G_D, l, h->dhb, mt_upper);
            p.ep.kind = EPI_DSWIGLU; p.ep.aux = h->gu[l]; p.ep.ld_aux = 2 * f; p.ep.out0 = h->dgu; p.ep.ld0 = 2 * f;
            if ((rc = tf_gemm(h, p, s, MLORA_TF_PROF_DOWN_BWD))) return rc;
        }
        if ((rc = group_grads(h, G_D, l, mp, h->dhb, h->vd[l], h->act[l], s))) return rc;
        if ((rc = shrink_bwd(h, G_GU, l, h->dgu, mt_upper, s))) return rc;
        {
            GemmParams p = proj_bwd(h, G_GU, l, h->dgu, mt_upper);
            p.ep.kind = EPI_F32; p.ep.f32 = h->dxn32; p.ep.ldf = d;
            if ((rc = tf_gemm(h, p, s, MLORA_TF_PROF_GATEUP_BWD))) return rc;
        }
        if ((rc = group_grads(h, G_GU, l, mp, h->dgu, h->vgu[l], h->x2[l], s))) return rc;
        if ((rc = tf_norm_bwd(h, h->snap2[l], h->gmlp[l], h->rstd2[l], 1, mp, s))) return rc;
        // h_mid = h_in + P_o(attention(rope(P_q x), rope(P_k x), P_v x))
        if ((rc = shrink_bwd(h, G_O, l, h->dhb, mt_upper, s))) return rc;
        {
            GemmParams p = proj_bwd(h, G_O, l, h->dhb, mt_upper);
            p.ep.kind = EPI_STORE; p.ep.out0 = h->dO; p.ep.ld0 = h->Q;
            if ((rc = tf_gemm(h, p, s, MLORA_TF_PROF_O_BWD))) return rc;
        }
        if ((rc = group_grads(h, G_O, l, mp, h->dhb, h->vo[l], h->o[l], s))) return rc;
        {
            TfProf ps(h, s, MLORA_TF_PROF_ATTN_BWD);
            AttnArgs aa = attn_args(h, l, mp);
            aa.ds = h->attn_ds;
            aa.ktc = h->attn_ktc;
            const cudaError_t e = launch_attention_bwd(aa, h->status, s);
            if (e != cudaSuccess) return tfail(MLORA_E_CUDA, "attention backward launch: %s", cudaGetErrorString(e));
            h->launches += 3;
        }
        {
            TfProf ps(h, s, MLORA_TF_PROF_ROPE);
            launch_rope(h->dqkv, h->Nqkv, 0, h->nh + h->nkv, h->pos_pad, h->rope_cs, h->rb.meta, mp, 1, s);
            ++h->launches;
        }
        if ((rc = shrink_bwd(h, G_QKV, l, h->dqkv, mt_upper, s))) return rc;
        {
            GemmParams p = proj_bwd(h, G_QKV, l, h->dqkv, mt_upper);
            p.ep.kind = EPI_F32; p.ep.f32 = h->dxn32; p.ep.ldf = d;
            if ((rc = tf_gemm(h, p, s, MLORA_TF_PROF_QKV_BWD))) return rc;
        }
        if ((rc = group_grads(h, G_QKV, l, mp, h->dqkv, h->vqkv[l], h->x1[l], s))) return rc;
        if ((rc = tf_norm_bwd(h, h->snap1[l], h->gattn[l], h->rstd1[l], 1, mp, s))) return rc;
    }
    return MLORA_OK;
}

int tf_check_batch(mlora_tf_t* h, const mlora_tf_batch* b) {
    if (!h || !b) return tfail(MLORA_E_ARG, "NULL handle or batch");
    if (b->n_tokens < 0 || b->n_tokens > h->max_tokens)
        return tfail(MLORA_E_ARG, "n_tokens %lld outside 0..max_tokens (%lld)", (long long)b->n_tokens,
                     (long long)h->max_tokens);
    if (b->n_tokens > 0 && (!b->tokens || !b->targets || !b->positions || !b->adapter_ids))
        return tfail(MLORA_E_ARG, "NULL token array");
    return MLORA_OK;
}

int tf_dispatch(mlora_tf_t* h, const mlora_tf_batch* b, const LossArgs& la, float* lp, double* loss, bool bwd,
                void* stream) {
    const int rc = tf_step(h, b, la, lp, loss, bwd, reinterpret_cast<cudaStream_t>(stream));
    if (rc) return rc;
    TF_CUDA(cudaGetLastError());
    return MLORA_OK;
}

}  // namespace

extern "C" int mlora_tf_forward(mlora_tf_t* h, const mlora_tf_batch* b, float* logprobs_out, void* stream) {
    int rc = tf_check_batch(h, b);
    if (rc) return rc;
    if (!logprobs_out && b->n_tokens > 0) return tfail(MLORA_E_ARG, "NULL logprobs_out");
    LossArgs la{-1, nullptr, nullptr, nullptr, 0.f, nullptr};
    return tf_dispatch(h, b, la, logprobs_out, nullptr, false, stream);
}

extern "C" int mlora_tf_forward_backward(mlora_tf_t* h, const mlora_tf_batch* b, int32_t loss_kind,
                                         const mlora_loss_inputs* li, float* logprobs_out, double* loss_out,
                                         void* stream) {
    int rc = tf_check_batch(h, b);
    if (rc) return rc;
    if (!li) return tfail(MLORA_E_ARG, "NULL loss inputs");
    LossArgs la{loss_kind, li->weights, li->advantages, li->sampler_logprobs, li->clip_eps, nullptr};
    if (b->n_tokens > 0) {
        if (loss_kind == MLORA_CROSS_ENTROPY) {
            if (!li->weights) return tfail(MLORA_E_ARG, "cross_entropy needs weights");
        } else if (loss_kind == MLORA_IMPORTANCE_SAMPLING || loss_kind == MLORA_PPO) {
            if (!li->advantages || !li->sampler_logprobs)
                return tfail(MLORA_E_ARG, "importance_sampling / ppo need advantages and sampler_logprobs");
            if (loss_kind == MLORA_PPO && !(li->clip_eps >= 0.f && li->clip_eps < 1.f))
                return tfail(MLORA_E_ARG, "ppo clip_eps must be in [0, 1)");
        } else {
            return tfail(MLORA_E_ARG, "unknown loss kind %d", loss_kind);
        }
    }
    return tf_dispatch(h, b, la, logprobs_out, loss_out, true, stream);
}

extern "C" int mlora_tf_forward_backward_custom(mlora_tf_t* h, const mlora_tf_batch* b, const float* dloss_dlogprobs,
                                                float* logprobs_out, double* loss_out, void* stream) {
    int rc = tf_check_batch(h, b);
    if (rc) return rc;
    if (!dloss_dlogprobs && b->n_tokens > 0) return tfail(MLORA_E_ARG, "NULL dloss_dlogprobs");
    LossArgs la{3, nullptr, nullptr, nullptr, 0.f, dloss_dlogprobs};
    return tf_dispatch(h, b, la, logprobs_out, loss_out, true, stream);
}

extern "C" int mlora_tf_optim_step(mlora_tf_t* h, const mlora_adam* p, const int32_t* adapters, int32_t n,
                                   int32_t* skipped_out, void* stream) {
    if (!h || !p) return tfail(MLORA_E_ARG, "NULL handle or adam params");
    if (!(p->lr >= 0.f) || !(p->beta1 >= 0.f && p->beta1 < 1.f) || !(p->beta2 >= 0.f && p->beta2 < 1.f) ||
        !(p->eps > 0.f) || !std::isfinite(p->weight_decay))
        return tfail(MLORA_E_ARG, "bad Adam hyper-parameters");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int* sel = nullptr;
    if (adapters) {
        if (n < 0) return tfail(MLORA_E_ARG, "negative adapter count");
        std::vector<int> mask(h->n_ad, 0);
        for (int i = 0; i < n; ++i) {
            if (adapters[i] < 0 || adapters[i] >= h->n_ad)
                return tfail(MLORA_E_ARG, "adapter id %d out of range", adapters[i]);
            mask[adapters[i]] = 1;
        }
        TF_CUDA(cudaMemcpyAsync(h->sel_mask, mask.data(), sizeof(int) * h->n_ad, cudaMemcpyHostToDevice, s));
        TF_CUDA(cudaStreamSynchronize(s));   // the host vector goes out of scope
        sel = h->sel_mask;
    }
    {
        TfProf ps(h, s, MLORA_TF_PROF_OTHER);
        launch_adam_prep(h->n_ad, sel, h->touched, h->nonfinite, h->step, p->beta1, p->beta2, h->adam_tab,
                         skipped_out, s);
        ++h->launches;
    }
    {
        TfProf ps(h, s, MLORA_TF_PROF_ADAM);
        launch_tf_adam(h->n_ad, h->ad_off, h->ranks_d, h->n_params, h->adam_tab, h->P, h->G, h->M, h->Vm, p->lr,
                       p->beta1, p->beta2, p->eps, p->weight_decay, h->mirror, 0, h->num_sms, s);
        ++h->launches;
    }
    TF_CUDA(cudaGetLastError());
    return MLORA_OK;
}

extern "C" int mlora_tf_read_adapter(mlora_tf_t* h, int32_t adapter, int32_t layer, int32_t proj, int32_t factor,
                                     int32_t kind, float* dst, void* stream) {
    if (!h || !dst) return tfail(MLORA_E_ARG, "NULL argument");
    if (adapter < 0 || adapter >= h->n_ad || layer < 0 || layer >= h->L || proj < 0 || proj >= MLORA_TF_NPROJ ||
        factor < 0 || factor > 1 || kind < 0 || kind > 3)
        return tfail(MLORA_E_ARG, "adapter/layer/projection/factor/kind out of range");
    int out, in;
    proj_shape(h, proj, &out, &in);
    const int64_t cnt = (int64_t)h->ranks[adapter] * (factor ? out : in);
    float* bufs[4] = {h->P, h->G, h->M, h->Vm};
    TF_CUDA(cudaMemcpyAsync(dst, bufs[kind] + tf_tensor_off(h, adapter, layer, proj, factor), sizeof(float) * cnt,
                            cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(stream)));
    return MLORA_OK;
}

extern "C" int mlora_tf_get_steps(mlora_tf_t* h, int64_t* steps_out, void* stream) {
    if (!h || !steps_out) return tfail(MLORA_E_ARG, "NULL argument");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    TF_CUDA(cudaMemcpyAsync(steps_out, h->step, sizeof(int64_t) * h->n_ad, cudaMemcpyDeviceToHost, s));
    TF_CUDA(cudaStreamSynchronize(s));
    return MLORA_OK;
}

extern "C" int mlora_tf_check_status(mlora_tf_t* h, void* stream) {
    if (!h) return tfail(MLORA_E_ARG, "NULL handle");
    TF_CUDA(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
    int st = 0;
    TF_CUDA(cudaMemcpy(&st, h->status, sizeof(int), cudaMemcpyDeviceToHost));
    TF_CUDA(cudaMemset(h->status, 0, sizeof(int)));
    if (st & ST_TIMEOUT) return tfail(MLORA_E_TIMEOUT, "a bounded device wait gave up");
    if (st & ST_RANGE) return tfail(MLORA_E_RANGE, "a token, target, adapter id or position was out of range");
    return MLORA_OK;
}

extern "C" int mlora_tf_set_lm_backward(mlora_tf_t* h, int32_t mode) {
    if (!h) return tfail(MLORA_E_ARG, "NULL handle");
    if (mode != MLORA_LM_RECOMPUTE && mode != MLORA_LM_KEEP_LOGITS)
        return tfail(MLORA_E_ARG, "unknown LM-head backward mode %d", mode);
    if (mode == h->lm_keep) return MLORA_OK;
    TF_CUDA(cudaDeviceSynchronize());   // no queued step may still use the buffers
    const size_t n = (size_t)h->nc_tiles * TILE_M * h->Vpad;
    auto drop = [&]() {
        tf_free(h, reinterpret_cast<void**>(&h->dz[1]));
        for (int b = 0; b < 2; ++b) tf_free(h, reinterpret_cast<void**>(&h->zbuf[b]));
    };
    if (mode == MLORA_LM_RECOMPUTE) {
        drop();
        h->lm_keep = 0;
        return MLORA_OK;
    }
    int rc = tf_alloc_t(h, &h->dz[1], n);
    for (int b = 0; b < 2 && rc == MLORA_OK; ++b) rc = tf_alloc_t(h, &h->zbuf[b], n);
    if (rc == MLORA_OK && cudaMemset(h->dz[1], 0, n * sizeof(bf16)) != cudaSuccess)
        rc = tfail(MLORA_E_CUDA, "cudaMemset of a dz chunk buffer failed");
    if (rc != MLORA_OK) {
        drop();
        return rc;
    }
    h->lm_keep = 1;
    return MLORA_OK;
}

extern "C" int mlora_tf_set_attention_backward(mlora_tf_t* h, int32_t max_seq_len) {
    if (!h) return tfail(MLORA_E_ARG, "NULL handle");
    if (max_seq_len < 0) return tfail(MLORA_E_ARG, "max_seq_len %d < 0", max_seq_len);
    const int S = (int64_t)max_seq_len > h->max_tokens ? (int)h->max_tokens : max_seq_len;
    const int ktc = S > 0 ? (S - 1 + 127) / 128 + 1 : 0;   // key tiles one query tile can see
    if (S > 0 && h->attn_ds && ktc == h->attn_ktc) {
        h->attn_max_seq = S;
        return MLORA_OK;
    }
    TF_CUDA(cudaDeviceSynchronize());   // no queued step may still use the buffer
    tf_free(h, reinterpret_cast<void**>(&h->attn_ds));
    h->attn_ktc = 0;
    h->attn_max_seq = 0;
    if (S == 0) return MLORA_OK;
    const int64_t blocks = (h->max_pad / 128) * (int64_t)ktc * h->nh;
    if (blocks * 128 > INT32_MAX)
        return tfail(MLORA_E_ARG, "stored attention blocks for %d-token sequences exceed the layout's range", S);
    const int rc = tf_alloc_t(h, &h->attn_ds, (size_t)blocks * 128 * 128);
    if (rc != MLORA_OK) return rc;
    h->attn_ktc = ktc;
    h->attn_max_seq = S;
    return MLORA_OK;
}

extern "C" int mlora_tf_profile_enable(mlora_tf_t* h, int32_t on) {
    if (!h) return tfail(MLORA_E_ARG, "NULL handle");
    h->prof = on != 0;
    return MLORA_OK;
}

extern "C" int mlora_tf_profile_read(mlora_tf_t* h, double* ms_out, int64_t* launches_out, int32_t reset) {
    if (!h) return tfail(MLORA_E_ARG, "NULL handle");
    for (size_t i = 0; i < h->ev_used; ++i) {
        TF_CUDA(cudaEventSynchronize(h->ev[2 * i + 1]));
        float ms = 0.f;
        TF_CUDA(cudaEventElapsedTime(&ms, h->ev[2 * i], h->ev[2 * i + 1]));
        int c = h->ev_cls[i];
        if (c < 0 || c >= MLORA_TF_PROF_CLASSES) c = MLORA_TF_PROF_OTHER;
        h->prof_ms[c] += ms;
        h->prof_n[c] += 1;
    }
    h->ev_used = 0;
    for (int c = 0; c < MLORA_TF_PROF_CLASSES; ++c) {
        if (ms_out) ms_out[c] = h->prof_ms[c];
        if (launches_out) launches_out[c] = h->prof_n[c];
        if (reset) { h->prof_ms[c] = 0.0; h->prof_n[c] = 0; }
    }
    return MLORA_OK;
}
