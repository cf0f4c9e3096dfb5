// C ABI of libmlora (include/mlora.h) and the host-side launch sequence of
// one training step.  Every step of the computation runs in this library's
// kernels on the caller's stream; the host only validates arguments, builds
// launch descriptors and queues work.
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <cmath>
#include <string>
#include <vector>

#include "internal.h"

using namespace mlk;

// ----------------------------------------------------------------------------
// errors
// ----------------------------------------------------------------------------
static thread_local std::string g_last_error;

static int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

#define CUDA_TRY(expr)                                                                   \
    do {                                                                                 \
        cudaError_t _e = (expr);                                                         \
        if (_e != cudaSuccess)                                                           \
            return fail(MLORA_E_CUDA, "%s failed: %s", #expr, cudaGetErrorString(_e));  \
    } while (0)

// ----------------------------------------------------------------------------
// handle
// ----------------------------------------------------------------------------
struct mlora {
    int V = 0, d = 0, f = 0, L = 0, dtype = 0, n_ad = 0;
    int64_t max_tokens = 0;
    int max_pad = 0, max_tiles = 0, max_chunks = 0, max_blocks = 0;
    int Vpad = 0;
    int num_sms = 0;
    int use_tc = 0;
    size_t esize = 2;
    std::vector<int> ranks;
    std::vector<float> alphas;
    std::vector<void*> allocs;
    std::vector<size_t> alloc_bytes;
    int64_t bytes = 0;
    int64_t launches = 0;
    int deterministic = 0;   // 1: one gradient chunk per adapter (fixed-order reductions)
    int test_withhold_kb = -1;          // test hook, applied to the next single-CTA GEMM
    unsigned long long test_wait_ns = 0;

    // frozen base
    void* E = nullptr;
    void* Wout = nullptr;
    std::vector<void*> W1, W2;
    std::vector<void*> W1T, W2T;        // K-major copies for the backward GEMMs
    // adapters
    int64_t n_params = 0;
    std::vector<int64_t> ad_off_h;      // [n_ad + 1]
    float *P = nullptr, *G = nullptr, *M = nullptr, *Vm = nullptr;
    int64_t* ad_off = nullptr;
    int* ranks_d = nullptr;
    float* gamma_d = nullptr;
    int64_t* grad_off = nullptr;        // [(l*4 + k) * n_ad + a]
    int64_t* step = nullptr;
    int *touched = nullptr, *nonfinite = nullptr, *sel_mask = nullptr;
    AdamTab* adam_tab = nullptr;
    ShadowMap shadow;                   // padded-rank copies per layer (dtype)
    // routing
    RouteBufs rb;
    // activations (dtype unless noted)
    std::vector<void*> hb, ub, actb, v1s, v2s;
    float* h32 = nullptr;
    float* dh32 = nullptr;
    void *dhb = nullptr, *dub = nullptr, *w1s = nullptr, *w2s = nullptr;
    // LM head
    int lm_bn = 32, n_nt = 0, part_ld = 0, nc_tiles = 0;
    float* part = nullptr;
    float* mt = nullptr;                // per row and partial tile: the tile's logit maximum
    float *zt = nullptr, *lse = nullptr, *gvec = nullptr;
    int* tgt_pad = nullptr;
    // LM-head backward (mlora_set_lm_backward).  Recompute: dz[0] only.  Kept
    // logits: dz[0..1] and zbuf[0..1] double-buffered, the dz pass of chunk i
    // on `side` beside the next chunk's GEMMs.
    int lm_keep = 0;
    void* dz[2] = {nullptr, nullptr};   // dz of a chunk of rows (base dtype)
    void* zbuf[2] = {nullptr, nullptr};   // kept logits of a chunk of rows: fp16 e = exp(z - tile
                                          // max) on the bf16 engine, fp32 z on the fp32 one
    cudaStream_t side = nullptr;
    cudaEvent_t ev_comb[2] = {}, ev_dz[2] = {}, ev_dh[2] = {};
    double* val_row = nullptr;          // per padded row loss value
    int* status = nullptr;
    int* tile_counter = nullptr;        // GEMM tile scheduler (reset before each launch)
    void *mg_a = nullptr, *mg_b = nullptr;  // merge operands, max(d, f) x 3*RP each
    // measurement: events around launches
    bool prof = false;
    std::vector<cudaEvent_t> ev;      // pairs (start, stop)
    std::vector<int> ev_cls;
    size_t ev_used = 0;
    double prof_ms[MLORA_PROF_CLASSES] = {0};
    int64_t prof_n[MLORA_PROF_CLASSES] = {0};
};

// Brackets one launch with events when profiling is on.
struct ProfScope {
    mlora_t* h;
    cudaStream_t s;
    int cls;
    size_t slot = (size_t)-1;
    ProfScope(mlora_t* h_, cudaStream_t s_, int cls_) : h(h_), s(s_), cls(cls_) {
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
    ~ProfScope() {
        if (slot == (size_t)-1) return;
        cudaEventRecord(h->ev[2 * slot + 1], s);
        h->ev_cls[slot] = cls;
    }
};

// Every device allocation of the library goes through here.  Test hook (not in
// the public headers): mlk_test_fail_alloc_at(n) makes the allocation with
// ordinal n (counted over the process, see mlk_test_alloc_calls) fail with
// cudaErrorMemoryAllocation without calling the driver, so the create calls'
// clean-up after a failed allocation can be exercised on any GPU.
static std::atomic<int64_t> g_alloc_calls{0};
static std::atomic<int64_t> g_fail_alloc_at{0};

cudaError_t mlk::mlk_malloc(void** p, size_t bytes) {
    const int64_t n = ++g_alloc_calls;
    if (n == g_fail_alloc_at.load()) {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMalloc(p, bytes);
}

extern "C" int64_t mlk_test_alloc_calls(void) { return g_alloc_calls.load(); }
extern "C" void mlk_test_fail_alloc_at(int64_t ordinal) { g_fail_alloc_at.store(ordinal); }

static int dalloc(mlora_t* h, void** p, size_t bytes) {
    if (bytes == 0) bytes = 16;
    cudaError_t e = mlk_malloc(p, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return fail(MLORA_E_NOMEM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
    }
    h->allocs.push_back(*p);
    h->alloc_bytes.push_back(bytes);
    h->bytes += (int64_t)bytes;
    return MLORA_OK;
}

// Frees one allocation made by dalloc (the caller has synchronised the device).
static void dfree(mlora_t* h, void** p) {
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
static int dalloc_t(mlora_t* h, P** p, size_t count) {
    void* q = nullptr;
    int rc = dalloc(h, &q, count * sizeof(P));
    *p = reinterpret_cast<P*>(q);
    return rc;
}

static void free_all(mlora_t* h) {
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

static inline int64_t tensor_size(int k, int r, int d, int f) {
    switch (k) {
    case 0: return (int64_t)r * d;   // A1
    case 1: return (int64_t)f * r;   // B1
    case 2: return (int64_t)r * f;   // A2
    default: return (int64_t)d * r;  // B2
    }
}

static inline int64_t tensor_off(const mlora_t* h, int a, int l, int k) {
    int r = h->ranks[a];
    int64_t off = h->ad_off_h[a] + (int64_t)l * 2 * r * (h->d + h->f);
    for (int q = 0; q < k; ++q) off += tensor_size(q, r, h->d, h->f);
    return off;
}

// padded-row upper bound for a batch of n tokens
static inline int pad_rows_for(const mlora_t* h, int64_t n) {
    int64_t busy = n < h->n_ad ? n : h->n_ad;
    int64_t rows = n + (int64_t)(TILE_M - 1) * busy;
    return (int)((rows + TILE_M - 1) / TILE_M * TILE_M);
}

extern "C" const char* mlora_last_error(void) { return g_last_error.c_str(); }

// Lets other translation units of the library report a failure through
// mlora_last_error().
int mlk_report_error(int code, const char* msg) {
    g_last_error = msg;
    return code;
}

// Read-only view of a handle for the sampler (sampler.cu).
void mlk_trainer_view(const mlora_t* h, TrainerView* v) {
    v->V = h->V; v->d = h->d; v->f = h->f; v->L = h->L; v->dtype = h->dtype; v->n_ad = h->n_ad;
    v->Vpad = h->Vpad; v->n_nt = h->n_nt; v->part_ld = h->part_ld; v->lm_bn = h->lm_bn;
    v->num_sms = h->num_sms; v->use_tc = h->use_tc; v->esize = h->esize;
    v->E = h->E; v->Wout = h->Wout;
    v->W1 = h->W1.data(); v->W2 = h->W2.data();
    v->shadow = &h->shadow;
    v->gamma_d = h->gamma_d; v->step_d = h->step;
    v->ranks = h->ranks.data(); v->alphas = h->alphas.data();
}

extern "C" int64_t mlora_kernel_launches(const mlora_t* h) { return h ? h->launches : 0; }

extern "C" int64_t mlora_device_bytes(const mlora_t* h) { return h ? h->bytes : 0; }

// ----------------------------------------------------------------------------
// create / destroy
// ----------------------------------------------------------------------------
extern "C" int mlora_create(const mlora_config* cfg, const mlora_init* init, mlora_t** out) {
    if (!cfg || !init || !out) return fail(MLORA_E_ARG, "NULL argument");
    *out = nullptr;
    if (cfg->vocab < 1 || cfg->d_model < 64 || cfg->d_model % 64 || cfg->d_ffn < 64 ||
        cfg->d_ffn % 64 || cfg->n_layers < 1 || cfg->n_layers > 64)
        return fail(MLORA_E_ARG, "bad model shape (V=%d d=%d f=%d L=%d): d and f must be "
                    "multiples of 64, 1 <= L <= 64", cfg->vocab, cfg->d_model, cfg->d_ffn,
                    cfg->n_layers);
    if (cfg->dtype != MLORA_BF16 && cfg->dtype != MLORA_FP32)
        return fail(MLORA_E_ARG, "bad dtype %d", cfg->dtype);
    if (cfg->n_adapters < 1 || cfg->n_adapters > 1024 || !cfg->ranks || !cfg->alphas)
        return fail(MLORA_E_ARG, "n_adapters must be 1..1024 with ranks and alphas");
    if (cfg->max_tokens < 1 || cfg->max_tokens > (1LL << 26))
        return fail(MLORA_E_ARG, "max_tokens out of range");
    for (int a = 0; a < cfg->n_adapters; ++a) {
        int r = cfg->ranks[a];
        if (r < 1 || r > MLORA_MAX_RANK || r % 4)
            return fail(MLORA_E_ARG, "adapter %d: rank %d must be in 4..%d and a multiple of 4", a, r,
                        MLORA_MAX_RANK);
        if (!std::isfinite(cfg->alphas[a])) return fail(MLORA_E_ARG, "adapter %d: alpha not finite", a);
    }
    if (!init->E || !init->Wout || !init->W1 || !init->W2) return fail(MLORA_E_ARG, "NULL base weight");
    for (int l = 0; l < cfg->n_layers; ++l)
        if (!init->W1[l] || !init->W2[l]) return fail(MLORA_E_ARG, "NULL W1/W2 for layer %d", l);

    int dev = 0;
    CUDA_TRY(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    CUDA_TRY(cudaGetDeviceProperties(&prop, dev));

    mlora_t* h = new mlora();
    h->V = cfg->vocab; h->d = cfg->d_model; h->f = cfg->d_ffn; h->L = cfg->n_layers;
    h->dtype = cfg->dtype; h->n_ad = cfg->n_adapters; h->max_tokens = cfg->max_tokens;
    h->num_sms = prop.multiProcessorCount;
    h->esize = cfg->dtype == MLORA_BF16 ? 2 : 4;
    h->ranks.assign(cfg->ranks, cfg->ranks + cfg->n_adapters);
    h->alphas.assign(cfg->alphas, cfg->alphas + cfg->n_adapters);
    // bf16 runs on the tcgen05 engine only (sm_100 family); fp32 on the FFMA engine.
    h->use_tc = cfg->dtype == MLORA_BF16;
    if (h->use_tc && (prop.major != 10 || !tc_engine_available())) {
        delete h;
        return fail(MLORA_E_UNSUPPORTED, "a bf16 handle needs an sm_100-family GPU with TMA "
                    "(found compute capability %d.%d)", prop.major, prop.minor);
    }
    h->Vpad = (h->V + 63) / 64 * 64;
    h->lm_bn = h->use_tc ? 256 : 32;
    h->n_nt = (h->V + h->lm_bn - 1) / h->lm_bn;
    h->part_ld = (h->n_nt + 3) & ~3;   // 16-byte aligned rows of partials

    const int n_ad = h->n_ad, L = h->L, d = h->d, f = h->f, V = h->V;
    const size_t es = h->esize;
    h->max_pad = pad_rows_for(h, h->max_tokens);
    h->max_tiles = h->max_pad / TILE_M;
    h->max_chunks = h->max_pad / GRAD_CHUNK + n_ad + 1;
    h->max_blocks = (int)((h->max_tokens + ROUTE_BLOCK - 1) / ROUTE_BLOCK);
    const int64_t MP = h->max_pad;

    int rc = MLORA_OK;
#define ALLOC(ptr, count) do { if ((rc = dalloc_t(h, &(ptr), (size_t)(count))) != MLORA_OK) goto fail_out; } while (0)
#define ALLOCB(ptr, bytes) do { if ((rc = dalloc(h, &(ptr), (size_t)(bytes))) != MLORA_OK) goto fail_out; } while (0)
    {
        // base
        ALLOCB(h->E, (size_t)V * d * es);
        ALLOCB(h->Wout, (size_t)V * d * es);
        h->W1.resize(L); h->W2.resize(L); h->W1T.resize(L); h->W2T.resize(L);
        for (int l = 0; l < L; ++l) {
            ALLOCB(h->W1[l], (size_t)f * d * es);
            ALLOCB(h->W2[l], (size_t)d * f * es);
            ALLOCB(h->W1T[l], (size_t)d * f * es);
            ALLOCB(h->W2T[l], (size_t)f * d * es);
        }
        // adapters
        h->ad_off_h.resize(n_ad + 1);
        h->ad_off_h[0] = 0;
        for (int a = 0; a < n_ad; ++a)
            h->ad_off_h[a + 1] = h->ad_off_h[a] + (int64_t)L * 2 * h->ranks[a] * (d + f);
        h->n_params = h->ad_off_h[n_ad];
        ALLOC(h->P, h->n_params); ALLOC(h->G, h->n_params);
        ALLOC(h->M, h->n_params); ALLOC(h->Vm, h->n_params);
        ALLOC(h->ad_off, n_ad + 1);
        ALLOC(h->ranks_d, n_ad);
        ALLOC(h->gamma_d, n_ad);
        ALLOC(h->grad_off, (size_t)L * 4 * n_ad);
        ALLOC(h->step, n_ad);
        ALLOC(h->touched, n_ad);
        ALLOC(h->nonfinite, n_ad);
        ALLOC(h->sel_mask, n_ad);
        ALLOC(h->adam_tab, n_ad);
        memset(&h->shadow, 0, sizeof(h->shadow));
        for (int l = 0; l < L; ++l) {
            ALLOCB(h->shadow.A1[l], (size_t)n_ad * RP * d * es);
            ALLOCB(h->shadow.B1[l], (size_t)n_ad * f * RP * es);
            ALLOCB(h->shadow.A2[l], (size_t)n_ad * RP * f * es);
            ALLOCB(h->shadow.B2[l], (size_t)n_ad * d * RP * es);
        }
        // routing
        ALLOC(h->rb.blk_cnt, (size_t)(h->max_blocks > 0 ? h->max_blocks : 1) * n_ad);
        ALLOC(h->rb.perm_pad, MP);
        ALLOC(h->rb.inv, h->max_tokens);
        ALLOC(h->rb.seg_off, n_ad + 1);
        ALLOC(h->rb.pad_off, n_ad + 1);
        ALLOC(h->rb.tile_ad, h->max_tiles);
        ALLOC(h->rb.meta, 4);
        ALLOC(h->rb.chunks, h->max_chunks);
        h->rb.max_pad = h->max_pad; h->rb.max_tiles = h->max_tiles; h->rb.max_chunks = h->max_chunks;
        // activations
        h->hb.resize(L + 1); h->ub.resize(L); h->actb.resize(L); h->v1s.resize(L); h->v2s.resize(L);
        for (int l = 0; l <= L; ++l) ALLOCB(h->hb[l], (size_t)MP * d * es);
        for (int l = 0; l < L; ++l) {
            ALLOCB(h->ub[l], (size_t)MP * f * es);
            ALLOCB(h->actb[l], (size_t)MP * f * es);
            ALLOCB(h->v1s[l], (size_t)MP * RP * es);
            ALLOCB(h->v2s[l], (size_t)MP * RP * es);
        }
        ALLOC(h->h32, (size_t)MP * d);
        ALLOC(h->dh32, (size_t)MP * d);
        ALLOCB(h->dhb, (size_t)MP * d * es);
        ALLOCB(h->dub, (size_t)MP * f * es);
        ALLOCB(h->w1s, (size_t)MP * RP * es);
        ALLOCB(h->w2s, (size_t)MP * RP * es);
        // LM head: partials, per-row scalars, and the bounded dz chunk buffer of
        // the recompute mode (the kept-logits mode adds its buffers on request)
        ALLOC(h->part, (size_t)MP * h->part_ld);
        ALLOC(h->mt, (size_t)MP * h->part_ld);
        ALLOC(h->zt, MP); ALLOC(h->lse, MP); ALLOC(h->gvec, MP);
        ALLOC(h->tgt_pad, MP);
        h->nc_tiles = h->max_tiles < 128 ? h->max_tiles : 128;   // chunks of up to 16,384 rows
        ALLOCB(h->dz[0], (size_t)h->nc_tiles * TILE_M * h->Vpad * es);
        // columns V..Vpad of dz are never written by the GEMM epilogue: zero once
        if (cudaMemset(h->dz[0], 0, (size_t)h->nc_tiles * TILE_M * h->Vpad * es) != cudaSuccess) {
            rc = fail(MLORA_E_CUDA, "cudaMemset of a dz chunk buffer failed");
            goto fail_out;
        }
        if (cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess) {
            h->side = nullptr;
            rc = fail(MLORA_E_CUDA, "cudaStreamCreate failed");
            goto fail_out;
        }
        for (int b = 0; b < 2; ++b) {
            if (cudaEventCreateWithFlags(&h->ev_comb[b], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&h->ev_dz[b], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&h->ev_dh[b], cudaEventDisableTiming) != cudaSuccess) {
                rc = fail(MLORA_E_CUDA, "cudaEventCreate failed");
                goto fail_out;
            }
        }
        ALLOC(h->val_row, (size_t)MP);
        ALLOC(h->status, 1);
        ALLOC(h->tile_counter, 1);
        ALLOCB(h->mg_a, (size_t)(d > f ? d : f) * 3 * RP * es);
        ALLOCB(h->mg_b, (size_t)(d > f ? d : f) * 3 * RP * es);
    }
#undef ALLOC
#undef ALLOCB
    // a failure while the handle is filled frees what it holds
#define CUDA_TRY_OUT(expr)                                                                   \
    do {                                                                                     \
        cudaError_t _e = (expr);                                                             \
        if (_e != cudaSuccess) {                                                             \
            rc = fail(MLORA_E_CUDA, "%s failed: %s", #expr, cudaGetErrorString(_e));         \
            goto fail_out;                                                                   \
        }                                                                                    \
    } while (0)
    {
        cudaStream_t s = 0;
        // copy the base
        CUDA_TRY_OUT(cudaMemcpyAsync(h->E, init->E, (size_t)V * d * es, cudaMemcpyDeviceToDevice, s));
        CUDA_TRY_OUT(cudaMemcpyAsync(h->Wout, init->Wout, (size_t)V * d * es, cudaMemcpyDeviceToDevice, s));
        for (int l = 0; l < L; ++l) {
            CUDA_TRY_OUT(cudaMemcpyAsync(h->W1[l], init->W1[l], (size_t)f * d * es, cudaMemcpyDeviceToDevice, s));
            CUDA_TRY_OUT(cudaMemcpyAsync(h->W2[l], init->W2[l], (size_t)d * f * es, cudaMemcpyDeviceToDevice, s));
            if (h->dtype == MLORA_BF16) {
                launch_transpose<bf16>(reinterpret_cast<const bf16*>(h->W1[l]), reinterpret_cast<bf16*>(h->W1T[l]), f, d, s);
                launch_transpose<bf16>(reinterpret_cast<const bf16*>(h->W2[l]), reinterpret_cast<bf16*>(h->W2T[l]), d, f, s);
            } else {
                launch_transpose<float>(reinterpret_cast<const float*>(h->W1[l]), reinterpret_cast<float*>(h->W1T[l]), f, d, s);
                launch_transpose<float>(reinterpret_cast<const float*>(h->W2[l]), reinterpret_cast<float*>(h->W2T[l]), d, f, s);
            }
            h->launches += 2;
        }
        // adapters
        CUDA_TRY_OUT(cudaMemsetAsync(h->P, 0, sizeof(float) * h->n_params, s));
        CUDA_TRY_OUT(cudaMemsetAsync(h->G, 0, sizeof(float) * h->n_params, s));
        CUDA_TRY_OUT(cudaMemsetAsync(h->M, 0, sizeof(float) * h->n_params, s));
        CUDA_TRY_OUT(cudaMemsetAsync(h->Vm, 0, sizeof(float) * h->n_params, s));
        const float* const* src[4] = {init->A1, init->B1, init->A2, init->B2};
        for (int a = 0; a < n_ad; ++a)
            for (int l = 0; l < L; ++l)
                for (int k = 0; k < 4; ++k) {
                    const float* p = src[k] ? src[k][a * L + l] : nullptr;
                    if (p)
                        CUDA_TRY_OUT(cudaMemcpyAsync(h->P + tensor_off(h, a, l, k), p,
                                                 sizeof(float) * tensor_size(k, h->ranks[a], d, f),
                                                 cudaMemcpyDeviceToDevice, s));
                }
        for (int l = 0; l < L; ++l) {
            CUDA_TRY_OUT(cudaMemsetAsync(h->shadow.A1[l], 0, (size_t)n_ad * RP * d * es, s));
            CUDA_TRY_OUT(cudaMemsetAsync(h->shadow.B1[l], 0, (size_t)n_ad * f * RP * es, s));
            CUDA_TRY_OUT(cudaMemsetAsync(h->shadow.A2[l], 0, (size_t)n_ad * RP * f * es, s));
            CUDA_TRY_OUT(cudaMemsetAsync(h->shadow.B2[l], 0, (size_t)n_ad * d * RP * es, s));
        }
        std::vector<float> gam(n_ad);
        for (int a = 0; a < n_ad; ++a) gam[a] = h->alphas[a] / (float)h->ranks[a];
        std::vector<int64_t> goff((size_t)L * 4 * n_ad);
        for (int l = 0; l < L; ++l)
            for (int k = 0; k < 4; ++k)
                for (int a = 0; a < n_ad; ++a) goff[((size_t)l * 4 + k) * n_ad + a] = tensor_off(h, a, l, k);
        CUDA_TRY_OUT(cudaMemcpy(h->ad_off, h->ad_off_h.data(), sizeof(int64_t) * (n_ad + 1), cudaMemcpyHostToDevice));
        CUDA_TRY_OUT(cudaMemcpy(h->ranks_d, h->ranks.data(), sizeof(int) * n_ad, cudaMemcpyHostToDevice));
        CUDA_TRY_OUT(cudaMemcpy(h->gamma_d, gam.data(), sizeof(float) * n_ad, cudaMemcpyHostToDevice));
        CUDA_TRY_OUT(cudaMemcpy(h->grad_off, goff.data(), sizeof(int64_t) * goff.size(), cudaMemcpyHostToDevice));
        CUDA_TRY_OUT(cudaMemset(h->step, 0, sizeof(int64_t) * n_ad));
        CUDA_TRY_OUT(cudaMemset(h->touched, 0, sizeof(int) * n_ad));
        CUDA_TRY_OUT(cudaMemset(h->nonfinite, 0, sizeof(int) * n_ad));
        CUDA_TRY_OUT(cudaMemset(h->status, 0, sizeof(int)));
        CUDA_TRY_OUT(cudaMemset(h->part, 0, sizeof(float) * (size_t)MP * h->part_ld));
        CUDA_TRY_OUT(cudaMemset(h->mt, 0, sizeof(float) * (size_t)MP * h->part_ld));
        if (h->dtype == MLORA_BF16)
            launch_shadow_sync<bf16>(n_ad, h->ad_off, h->ranks_d, L, d, f, h->n_params, h->P, h->shadow, s);
        else
            launch_shadow_sync<float>(n_ad, h->ad_off, h->ranks_d, L, d, f, h->n_params, h->P, h->shadow, s);
        ++h->launches;
        CUDA_TRY_OUT(cudaGetLastError());
        CUDA_TRY_OUT(cudaDeviceSynchronize());
    }
#undef CUDA_TRY_OUT
    *out = h;
    return MLORA_OK;
fail_out:
    free_all(h);
    delete h;
    return rc;
}

extern "C" int mlora_destroy(mlora_t* h) {
    if (!h) return MLORA_OK;
    cudaDeviceSynchronize();
    free_all(h);
    delete h;
    return MLORA_OK;
}

// ----------------------------------------------------------------------------
// GEMM descriptor helpers
// ----------------------------------------------------------------------------
static GemmOperand op_kmajor(const void* p, int64_t rows, int64_t cols, int64_t ad_rows = 0,
                             int64_t shift = 0) {
    GemmOperand o;
    o.ptr = p; o.ld = cols; o.rows = rows; o.cols = cols; o.mn_major = 0; o.ad_rows = ad_rows;
    o.row_shift = shift;
    return o;
}
static GemmOperand op_mnmajor(const void* p, int64_t rows, int64_t cols, int64_t ad_rows = 0) {
    GemmOperand o;
    o.ptr = p; o.ld = cols; o.rows = rows; o.cols = cols; o.mn_major = 1; o.ad_rows = ad_rows;
    return o;
}

template <typename T>
static int run_gemm(mlora_t* h, GemmParams& p, cudaStream_t s, int cls) {
    ProfScope ps(h, s, cls);
    p.tile_counter = h->tile_counter;
    if (h->use_tc && h->test_withhold_kb >= 0 && (p.N <= 64 || p.force_bn64)) {
        p.test_withhold_kb = h->test_withhold_kb;
        p.test_wait_ns = h->test_wait_ns;
        h->test_withhold_kb = -1;
    }
    if (h->use_tc) {
        cudaError_t e = launch_tc_gemm(p, s, h->num_sms, h->status);
        if (e != cudaSuccess) return fail(MLORA_E_CUDA, "tensor-core GEMM launch: %s", cudaGetErrorString(e));
    } else {
        launch_simt_gemm<T>(p, s);
    }
    ++h->launches;
    return MLORA_OK;
}

// Raster band height (row tiles) for an A operand with K columns: tiles in
// flight share B through L2 while a band of A (about 48 MB) stays resident.
// For very long K every tile streams its whole operands, and a band of 16
// row tiles keeps the set of tiles in flight close to square.
static int band_for_k(int K) {
    if (K >= 65536) return 16;
    int rows = (int)((48ll << 20) / (2ll * K));
    int tiles = rows / TILE_M;
    tiles &= ~1;
    if (tiles < 8) tiles = 8;
    if (tiles > 64) tiles = 64;
    return tiles;
}

// dense GEMM over the padded token rows of the current batch
static GemmParams dense_params(mlora_t* h, int mt_upper, int N, int K) {
    GemmParams p;
    p.M = mt_upper * TILE_M;
    p.N = N; p.K = K; p.Kx = 0;
    p.group_m = band_for_k(K);
    p.mtiles_dev = h->rb.meta;
    p.mt_base = 0; p.mt_count = mt_upper;
    p.tile_ad = h->rb.tile_ad;
    return p;
}

// per-adapter reduction over token rows: grad[a] (+)= X_seg^T Y_seg
static GemmParams grad_params(mlora_t* h, int mp, int Dout, const void* X, const void* Y, int l, int k,
                              int trans) {
    GemmParams p;
    p.M = Dout; p.N = RP; p.K = 0;
    p.grouped = 1;
    p.chunks = h->rb.chunks;
    p.nchunks_dev = h->rb.meta + 1;
    p.max_chunks = mp / GRAD_CHUNK + (mp / TILE_M < h->n_ad ? mp / TILE_M : h->n_ad) + 1;
    if (p.max_chunks > h->max_chunks) p.max_chunks = h->max_chunks;
    p.A = op_mnmajor(X, h->max_pad, Dout);
    p.B = op_mnmajor(Y, h->max_pad, RP);
    p.ep.kind = EPI_GRAD;
    p.ep.grad = h->G;
    p.ep.grad_off = h->grad_off + ((size_t)l * 4 + k) * h->n_ad;
    p.ep.ranks = h->ranks_d;
    p.ep.grad_trans = trans;
    p.ep.grad_M = Dout;
    p.ep.nonfinite = h->nonfinite;
    return p;
}

// ----------------------------------------------------------------------------
// one step
// ----------------------------------------------------------------------------
template <typename T>
static int step_impl(mlora_t* h, const mlora_batch* b, const LossArgs& la, float* logprobs_out,
                     double* loss_out, bool backward, cudaStream_t s) {
    const int64_t N = b->n_tokens;
    const int n_ad = h->n_ad, L = h->L, d = h->d, f = h->f, V = h->V;
    const int64_t MP = h->max_pad;
    const int mp = pad_rows_for(h, N);
    const int mt_upper = mp / TILE_M;
    int rc;

    if (logprobs_out && N > 0) CUDA_TRY(cudaMemsetAsync(logprobs_out, 0xff, sizeof(float) * N, s));
    if (N == 0) {
        if (loss_out) CUDA_TRY(cudaMemsetAsync(loss_out, 0, sizeof(double) * n_ad, s));
        return MLORA_OK;
    }
    // a1 routing
    {
        ProfScope ps(h, s, MLORA_PROF_ROUTING);
        launch_routing(b->adapter_ids, N, n_ad, h->rb, backward ? h->touched : nullptr, h->status, s,
                       &h->launches, h->deterministic ? 0 : GRAD_CHUNK);
    }
    // a2 embedding
    {
        ProfScope ps(h, s, MLORA_PROF_EMBED);
        launch_embed<T>(h->rb.perm_pad, h->rb.meta, mp, b->tokens, b->targets,
                        reinterpret_cast<const T*>(h->E), V, d, reinterpret_cast<T*>(h->hb[0]), h->h32,
                        h->tgt_pad, h->status, s);
        ++h->launches;
    }

    // a3-a5 layers
    for (int l = 0; l < L; ++l) {
        {   // v1s = gamma * A1_a h
            GemmParams p = dense_params(h, mt_upper, RP, d);
            p.A = op_kmajor(h->hb[l], MP, d);
            p.B = op_kmajor(h->shadow.A1[l], (int64_t)n_ad * RP, d, RP);
            p.ep.kind = EPI_SHRINK; p.ep.out0 = h->v1s[l]; p.ep.ld0 = RP; p.ep.gamma = h->gamma_d;
            if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_SHRINK))) return rc;
        }
        {   // u = W1 h + B1_a v1s ; act = silu(u)
            GemmParams p = dense_params(h, mt_upper, f, d);
            p.A = op_kmajor(h->hb[l], MP, d);
            p.B = op_kmajor(h->W1[l], f, d);
            p.Kx = RP;
            p.Ax = op_kmajor(h->v1s[l], MP, RP);
            p.Bx = op_kmajor(h->shadow.B1[l], (int64_t)n_ad * f, RP, f);
            p.ep.kind = EPI_SILU; p.ep.out0 = h->ub[l]; p.ep.ld0 = f; p.ep.out1 = h->actb[l]; p.ep.ld1 = f;
            if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_W1_FWD))) return rc;
        }
        {   // v2s = gamma * A2_a act
            GemmParams p = dense_params(h, mt_upper, RP, f);
            p.A = op_kmajor(h->actb[l], MP, f);
            p.B = op_kmajor(h->shadow.A2[l], (int64_t)n_ad * RP, f, RP);
            p.ep.kind = EPI_SHRINK; p.ep.out0 = h->v2s[l]; p.ep.ld0 = RP; p.ep.gamma = h->gamma_d;
            if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_SHRINK))) return rc;
        }
        {   // h += W2 act + B2_a v2s
            GemmParams p = dense_params(h, mt_upper, d, f);
            p.A = op_kmajor(h->actb[l], MP, f);
            p.B = op_kmajor(h->W2[l], d, f);
            p.Kx = RP;
            p.Ax = op_kmajor(h->v2s[l], MP, RP);
            p.Bx = op_kmajor(h->shadow.B2[l], (int64_t)n_ad * d, RP, d);
            p.ep.kind = EPI_RESID; p.ep.f32 = h->h32; p.ep.ldf = d; p.ep.out0 = h->hb[l + 1]; p.ep.ld0 = d;
            if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_W2_FWD))) return rc;
        }
    }
    // a6-a8 LM head.  Forward: per-tile log-sum-exp partials and the target
    // logit over all rows, then the combine + loss epilogue.  The backward
    // walks the rows in chunks: by default each chunk's logits are recomputed
    // by a second GEMM whose epilogue writes dz = g (onehot - softmax) into the
    // chunk buffer, then dh = dz Wout; in the kept-logits mode the forward GEMM
    // of each chunk also stores its logits (the bf16 engine: fp16 e = exp(z -
    // tile max), beside the tile maxima) and an elementwise pass forms dz.
    if (!backward || !h->lm_keep) {
        {
            GemmParams p = dense_params(h, mt_upper, V, d);
            p.A = op_kmajor(h->hb[L], MP, d);
            p.B = op_kmajor(h->Wout, V, d);
            p.ep.kind = EPI_LMFWD; p.ep.part = h->part; p.ep.zt = h->zt; p.ep.tgt = h->tgt_pad;
            p.ep.part_ld = h->part_ld; p.ep.V = V; p.ep.Vpad = h->Vpad;
            p.ep.mt = h->mt; p.ep.lm_bn = h->lm_bn;
            if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_LM_FWD))) return rc;
        }
        {
            ProfScope ps(h, s, MLORA_PROF_LOSS);
            launch_combine_loss(la, h->part, h->n_nt, h->part_ld, h->zt, h->rb.perm_pad, h->tgt_pad, h->rb.meta,
                                0, mt_upper, logprobs_out, h->lse, h->gvec, h->val_row, h->num_sms, s);
            ++h->launches;
        }
        if (loss_out) {
            ProfScope ps(h, s, MLORA_PROF_OTHER);
            launch_loss_reduce(h->val_row, h->rb.pad_off, n_ad, loss_out, s);
            ++h->launches;
        }
        if (!backward) return MLORA_OK;
    }
    // chunks of at most nc_tiles row tiles, sized so that dh fills whole waves
    // (dh on the tensor-core engine: 256 x 512 tiles at the vocabulary's K)
    const int dh_nt = sizeof(T) != 2 ? 0 : (h->Vpad >= 65536 && d % 512 == 0 ? d / 512 : (d + 255) / 256);
    const int chunk = lm_chunk_tiles(mt_upper, h->nc_tiles, dh_nt, h->num_sms / 2);
    const int nch = (mt_upper + chunk - 1) / chunk;
    auto dh_params = [&](int c0, int cnt, const void* dzb) {
        GemmParams p = dense_params(h, mt_upper, d, h->Vpad);
        p.mt_base = c0; p.mt_count = cnt;
        p.A = op_kmajor(dzb, (int64_t)h->nc_tiles * TILE_M, h->Vpad, 0, -(int64_t)c0 * TILE_M);
        p.B = op_mnmajor(h->Wout, V, d);
        p.ep.kind = EPI_STORE2; p.ep.f32 = h->dh32; p.ep.ldf = d; p.ep.out0 = h->dhb; p.ep.ld0 = d;
        return p;
    };
    if (!h->lm_keep) {
        // recompute: chunk i's logits again, dz from them in the epilogue, dh
        for (int c0 = 0; c0 < mt_upper; c0 += chunk) {
            const int cnt = mt_upper - c0 < chunk ? mt_upper - c0 : chunk;
            {
                GemmParams p = dense_params(h, mt_upper, V, d);
                p.mt_base = c0; p.mt_count = cnt;
                p.A = op_kmajor(h->hb[L], MP, d);
                p.B = op_kmajor(h->Wout, V, d);
                p.ep.kind = EPI_LMDZ; p.ep.tgt = h->tgt_pad; p.ep.gv = h->gvec; p.ep.lse = h->lse;
                p.ep.V = V; p.ep.Vpad = h->Vpad;
                p.ep.mt = h->mt; p.ep.part_ld = h->part_ld; p.ep.lm_bn = h->lm_bn;
                p.ep.out0 = h->dz[0]; p.ep.ld0 = h->Vpad; p.ep.out_row_shift = -(int64_t)c0 * TILE_M;
                p.ep.out_rows = (int64_t)h->nc_tiles * TILE_M;
                if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_LM_DZ))) return rc;
            }
            GemmParams p = dh_params(c0, cnt, h->dz[0]);
            if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_LM_DH))) return rc;
        }
    }
    // Chunk i uses logit / dz buffers i % 2.  The caller's stream runs
    //   LMfwd(0) comb(0) | LMfwd(1) comb(1) dh(0) | LMfwd(2) comb(2) dh(1) | ... dh(n-1)
    // and the side stream runs dz(i) after comb(i) (and after dh(i-2) has read
    // buffer i % 2), so each HBM-bound dz pass overlaps the next chunk's
    // compute-bound GEMMs on the SMs' spare warps.  dh(i) waits for dz(i); the
    // caller's stream has waited for every dz pass when the last dh is queued.
    auto chunk_rows = [&](int i, int& c0, int& cnt) {
        c0 = i * chunk;
        cnt = mt_upper - c0 < chunk ? mt_upper - c0 : chunk;
    };
    auto queue_dh = [&](int i) -> int {
        int c0, cnt;
        chunk_rows(i, c0, cnt);
        const int buf = i & 1;
        CUDA_TRY(cudaStreamWaitEvent(s, h->ev_dz[buf], 0));
        GemmParams p = dh_params(c0, cnt, h->dz[buf]);
        int r = run_gemm<T>(h, p, s, MLORA_PROF_LM_DH);
        if (r) return r;
        CUDA_TRY(cudaEventRecord(h->ev_dh[buf], s));
        return MLORA_OK;
    };
    for (int i = 0; i < nch && h->lm_keep; ++i) {
        int c0, cnt;
        chunk_rows(i, c0, cnt);
        const int buf = i & 1;
        {
            GemmParams p = dense_params(h, mt_upper, V, d);
            p.mt_base = c0; p.mt_count = cnt;
            p.A = op_kmajor(h->hb[L], MP, d);
            p.B = op_kmajor(h->Wout, V, d);
            p.ep.kind = EPI_LMFWD; p.ep.part = h->part; p.ep.zt = h->zt; p.ep.tgt = h->tgt_pad;
            p.ep.part_ld = h->part_ld; p.ep.V = V; p.ep.Vpad = h->Vpad;
            p.ep.mt = h->mt; p.ep.lm_bn = h->lm_bn;
            p.ep.out0 = h->zbuf[buf]; p.ep.ld0 = h->Vpad; p.ep.out_row_shift = -(int64_t)c0 * TILE_M;
            p.ep.out_rows = (int64_t)h->nc_tiles * TILE_M;
            p.ep.e16 = sizeof(T) == 2;      // the bf16 engine keeps fp16 e; the fp32 one fp32 z
            if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_LM_FWD))) return rc;
        }
        {
            ProfScope ps(h, s, MLORA_PROF_LOSS);
            launch_combine_loss(la, h->part, h->n_nt, h->part_ld, h->zt, h->rb.perm_pad, h->tgt_pad, h->rb.meta,
                                c0, cnt, logprobs_out, h->lse, h->gvec, h->val_row, h->num_sms, s);
            ++h->launches;
        }
        CUDA_TRY(cudaEventRecord(h->ev_comb[buf], s));
        CUDA_TRY(cudaStreamWaitEvent(h->side, h->ev_comb[buf], 0));
        if (i >= 2) CUDA_TRY(cudaStreamWaitEvent(h->side, h->ev_dh[buf], 0));
        {
            ProfScope ps(h, h->side, MLORA_PROF_LM_DZ);
            if constexpr (sizeof(T) == 2)
                launch_lm_dz_e16(reinterpret_cast<const __half*>(h->zbuf[buf]), reinterpret_cast<bf16*>(h->dz[buf]),
                                 h->Vpad, V, h->Vpad, h->mt, h->part_ld, h->lm_bn, h->gvec, h->lse, h->tgt_pad,
                                 h->rb.meta, c0 * TILE_M, cnt * TILE_M, h->side);
            else
                launch_lm_dz<T>(reinterpret_cast<const float*>(h->zbuf[buf]), reinterpret_cast<T*>(h->dz[buf]),
                                h->Vpad, V, h->Vpad, h->gvec, h->lse, h->tgt_pad, h->rb.meta, c0 * TILE_M,
                                cnt * TILE_M, h->side);
            ++h->launches;
        }
        CUDA_TRY(cudaEventRecord(h->ev_dz[buf], h->side));
        if (i >= 1 && (rc = queue_dh(i - 1))) return rc;
    }
    if (h->lm_keep) {
        if ((rc = queue_dh(nch - 1))) return rc;
        if (loss_out) {
            ProfScope ps(h, s, MLORA_PROF_OTHER);
            launch_loss_reduce(h->val_row, h->rb.pad_off, n_ad, loss_out, s);
            ++h->launches;
        }
    }

    // a9-a11 layers in reverse
    for (int l = L - 1; l >= 0; --l) {
        {   // w2s = gamma * B2_a^T dh
            GemmParams p = dense_params(h, mt_upper, RP, d);
            p.A = op_kmajor(h->dhb, MP, d);
            p.B = op_mnmajor(h->shadow.B2[l], (int64_t)n_ad * d, RP, d);
            p.ep.kind = EPI_SHRINK; p.ep.out0 = h->w2s; p.ep.ld0 = RP; p.ep.gamma = h->gamma_d;
            if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_SHRINK))) return rc;
        }
        {   // du = (W2^T dh + A2_a^T w2s) * silu'(u)
            GemmParams p = dense_params(h, mt_upper, f, d);
            p.A = op_kmajor(h->dhb, MP, d);
            p.B = op_kmajor(h->W2T[l], f, d);
            p.Kx = RP;
            p.Ax = op_kmajor(h->w2s, MP, RP);
            p.Bx = op_mnmajor(h->shadow.A2[l], (int64_t)n_ad * RP, f, RP);
            p.ep.kind = EPI_DSILU; p.ep.aux = h->ub[l]; p.ep.ld_aux = f; p.ep.out0 = h->dub; p.ep.ld0 = f;
            if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_W2_BWD))) return rc;
        }
        {   // dB2_a += dh^T v2s   [d x r]
            GemmParams p = grad_params(h, mp, d, h->dhb, h->v2s[l], l, 3, 0);
            if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_GRAD))) return rc;
        }
        {   // dA2_a += w2s^T act  [r x f], computed as act^T w2s
            GemmParams p = grad_params(h, mp, f, h->actb[l], h->w2s, l, 2, 1);
            if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_GRAD))) return rc;
        }
        {   // w1s = gamma * B1_a^T du
            GemmParams p = dense_params(h, mt_upper, RP, f);
            p.A = op_kmajor(h->dub, MP, f);
            p.B = op_mnmajor(h->shadow.B1[l], (int64_t)n_ad * f, RP, f);
            p.ep.kind = EPI_SHRINK; p.ep.out0 = h->w1s; p.ep.ld0 = RP; p.ep.gamma = h->gamma_d;
            if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_SHRINK))) return rc;
        }
        {   // dh += W1^T du + A1_a^T w1s
            GemmParams p = dense_params(h, mt_upper, d, f);
            p.A = op_kmajor(h->dub, MP, f);
            p.B = op_kmajor(h->W1T[l], d, f);
            p.Kx = RP;
            p.Ax = op_kmajor(h->w1s, MP, RP);
            p.Bx = op_mnmajor(h->shadow.A1[l], (int64_t)n_ad * RP, d, RP);
            p.ep.kind = EPI_RESID; p.ep.f32 = h->dh32; p.ep.ldf = d; p.ep.out0 = h->dhb; p.ep.ld0 = d;
            if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_W1_BWD))) return rc;
        }
        {   // dB1_a += du^T v1s   [f x r]
            GemmParams p = grad_params(h, mp, f, h->dub, h->v1s[l], l, 1, 0);
            if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_GRAD))) return rc;
        }
        {   // dA1_a += w1s^T h    [r x d], computed as h^T w1s
            GemmParams p = grad_params(h, mp, d, h->hb[l], h->w1s, l, 0, 1);
            if ((rc = run_gemm<T>(h, p, s, MLORA_PROF_GRAD))) return rc;
        }
    }
    return MLORA_OK;
}

static int check_batch(mlora_t* h, const mlora_batch* b) {
    if (!h || !b) return fail(MLORA_E_ARG, "NULL handle or batch");
    if (b->n_tokens < 0 || b->n_tokens > h->max_tokens)
        return fail(MLORA_E_ARG, "n_tokens %lld outside 0..max_tokens (%lld)", (long long)b->n_tokens,
                    (long long)h->max_tokens);
    if (b->n_tokens > 0 && (!b->tokens || !b->targets || !b->adapter_ids))
        return fail(MLORA_E_ARG, "NULL token array");
    return MLORA_OK;
}

static int dispatch_step(mlora_t* h, const mlora_batch* b, const LossArgs& la, float* lp,
                         double* loss, bool bwd, void* stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int rc = h->dtype == MLORA_BF16 ? step_impl<bf16>(h, b, la, lp, loss, bwd, s)
                                    : step_impl<float>(h, b, la, lp, loss, bwd, s);
    if (rc) return rc;
    CUDA_TRY(cudaGetLastError());
    return MLORA_OK;
}

extern "C" int mlora_forward(mlora_t* h, const mlora_batch* b, float* logprobs_out, void* stream) {
    int rc = check_batch(h, b);
    if (rc) return rc;
    if (!logprobs_out && b->n_tokens > 0) return fail(MLORA_E_ARG, "NULL logprobs_out");
    LossArgs la{-1, nullptr, nullptr, nullptr, 0.f, nullptr};
    return dispatch_step(h, b, la, logprobs_out, nullptr, false, stream);
}

extern "C" int mlora_forward_backward(mlora_t* h, const mlora_batch* b, int32_t loss_kind,
                                      const mlora_loss_inputs* li, float* logprobs_out,
                                      double* loss_out, void* stream) {
    int rc = check_batch(h, b);
    if (rc) return rc;
    if (!li) return fail(MLORA_E_ARG, "NULL loss inputs");
    LossArgs la{loss_kind, li->weights, li->advantages, li->sampler_logprobs, li->clip_eps, nullptr};
    if (b->n_tokens > 0) {
        if (loss_kind == MLORA_CROSS_ENTROPY) {
            if (!li->weights) return fail(MLORA_E_ARG, "cross_entropy needs weights");
        } else if (loss_kind == MLORA_IMPORTANCE_SAMPLING || loss_kind == MLORA_PPO) {
            if (!li->advantages || !li->sampler_logprobs)
                return fail(MLORA_E_ARG, "importance_sampling / ppo need advantages and sampler_logprobs");
            if (loss_kind == MLORA_PPO && !(li->clip_eps >= 0.f && li->clip_eps < 1.f))
                return fail(MLORA_E_ARG, "ppo clip_eps must be in [0, 1)");
        } else {
            return fail(MLORA_E_ARG, "unknown loss kind %d", loss_kind);
        }
    }
    return dispatch_step(h, b, la, logprobs_out, loss_out, true, stream);
}

extern "C" int mlora_forward_backward_custom(mlora_t* h, const mlora_batch* b,
                                             const float* dloss_dlogprobs, float* logprobs_out,
                                             double* loss_out, void* stream) {
    int rc = check_batch(h, b);
    if (rc) return rc;
    if (!dloss_dlogprobs && b->n_tokens > 0) return fail(MLORA_E_ARG, "NULL dloss_dlogprobs");
    LossArgs la{3, nullptr, nullptr, nullptr, 0.f, dloss_dlogprobs};
    return dispatch_step(h, b, la, logprobs_out, loss_out, true, stream);
}

extern "C" int mlora_optim_step(mlora_t* h, const mlora_adam* p, const int32_t* adapters, int32_t n,
                                int32_t* skipped_out, void* stream) {
    if (!h || !p) return fail(MLORA_E_ARG, "NULL handle or adam params");
    if (!(p->lr >= 0.f) || !(p->beta1 >= 0.f && p->beta1 < 1.f) || !(p->beta2 >= 0.f && p->beta2 < 1.f) ||
        !(p->eps > 0.f) || !std::isfinite(p->weight_decay))
        return fail(MLORA_E_ARG, "bad Adam hyper-parameters");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int* sel = nullptr;
    if (adapters) {
        if (n < 0) return fail(MLORA_E_ARG, "negative adapter count");
        std::vector<int> mask(h->n_ad, 0);
        for (int i = 0; i < n; ++i) {
            if (adapters[i] < 0 || adapters[i] >= h->n_ad) return fail(MLORA_E_ARG, "adapter id %d out of range", adapters[i]);
            mask[adapters[i]] = 1;
        }
        CUDA_TRY(cudaMemcpyAsync(h->sel_mask, mask.data(), sizeof(int) * h->n_ad, cudaMemcpyHostToDevice, s));
        CUDA_TRY(cudaStreamSynchronize(s));   // the host vector goes out of scope
        sel = h->sel_mask;
    }
    {
        ProfScope ps(h, s, MLORA_PROF_OTHER);
        launch_adam_prep(h->n_ad, sel, h->touched, h->nonfinite, h->step, p->beta1, p->beta2, h->adam_tab,
                         skipped_out, s);
        ++h->launches;
    }
    ProfScope ps_adam(h, s, MLORA_PROF_ADAM);
    if (h->dtype == MLORA_BF16)
        launch_adam<bf16>(h->n_ad, h->ad_off, h->ranks_d, h->L, h->d, h->f, h->n_params, h->adam_tab, h->P,
                          h->G, h->M, h->Vm, p->lr, p->beta1, p->beta2, p->eps, p->weight_decay, h->shadow, s);
    else
        launch_adam<float>(h->n_ad, h->ad_off, h->ranks_d, h->L, h->d, h->f, h->n_params, h->adam_tab, h->P,
                           h->G, h->M, h->Vm, p->lr, p->beta1, p->beta2, p->eps, p->weight_decay, h->shadow, s);
    ++h->launches;
    CUDA_TRY(cudaGetLastError());
    return MLORA_OK;
}

// ----------------------------------------------------------------------------
// inspection hooks, checkpoint, status
// ----------------------------------------------------------------------------
static int tensor_ptr(mlora_t* h, int a, int l, int which, float** ptr, int64_t* count) {
    if (!h) return fail(MLORA_E_ARG, "NULL handle");
    if (a < 0 || a >= h->n_ad || l < 0 || l >= h->L || which < 0 || which > 15)
        return fail(MLORA_E_ARG, "adapter/layer/tensor selector out of range");
    int k = which & 3;
    float* bufs[4] = {h->P, h->G, h->M, h->Vm};
    *ptr = bufs[which >> 2] + tensor_off(h, a, l, k);
    *count = tensor_size(k, h->ranks[a], h->d, h->f);
    return MLORA_OK;
}

extern "C" int mlora_read_adapter(mlora_t* h, int32_t adapter, int32_t layer, int32_t which, float* dst,
                                  void* stream) {
    float* src;
    int64_t cnt;
    int rc = tensor_ptr(h, adapter, layer, which, &src, &cnt);
    if (rc) return rc;
    if (!dst) return fail(MLORA_E_ARG, "NULL dst");
    CUDA_TRY(cudaMemcpyAsync(dst, src, sizeof(float) * cnt, cudaMemcpyDeviceToDevice,
                             reinterpret_cast<cudaStream_t>(stream)));
    return MLORA_OK;
}

extern "C" int mlora_write_adapter(mlora_t* h, int32_t adapter, int32_t layer, int32_t which,
                                   const float* src, void* stream) {
    if (which < 0 || which > 3) return fail(MLORA_E_ARG, "only weight tensors can be written");
    float* dst;
    int64_t cnt;
    int rc = tensor_ptr(h, adapter, layer, which, &dst, &cnt);
    if (rc) return rc;
    if (!src) return fail(MLORA_E_ARG, "NULL src");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CUDA_TRY(cudaMemcpyAsync(dst, src, sizeof(float) * cnt, cudaMemcpyDeviceToDevice, s));
    if (h->dtype == MLORA_BF16)
        launch_shadow_sync<bf16>(h->n_ad, h->ad_off, h->ranks_d, h->L, h->d, h->f, h->n_params, h->P, h->shadow, s);
    else
        launch_shadow_sync<float>(h->n_ad, h->ad_off, h->ranks_d, h->L, h->d, h->f, h->n_params, h->P, h->shadow, s);
    ++h->launches;
    CUDA_TRY(cudaGetLastError());
    return MLORA_OK;
}

extern "C" int mlora_get_steps(mlora_t* h, int64_t* steps_out, void* stream) {
    if (!h || !steps_out) return fail(MLORA_E_ARG, "NULL argument");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CUDA_TRY(cudaMemcpyAsync(steps_out, h->step, sizeof(int64_t) * h->n_ad, cudaMemcpyDeviceToHost, s));
    CUDA_TRY(cudaStreamSynchronize(s));
    return MLORA_OK;
}

extern "C" int mlora_get_routing(mlora_t* h, const int32_t* adapter_ids, int64_t n, int32_t* perm,
                                 int32_t* seg_off, int32_t* pad_off, int32_t* tile_ad, void* stream) {
    if (!h) return fail(MLORA_E_ARG, "NULL handle");
    if (n < 0 || n > h->max_tokens) return fail(MLORA_E_ARG, "n outside 0..max_tokens");
    if ((n > 0 && (!adapter_ids || !perm)) || !seg_off || !pad_off || !tile_ad)
        return fail(MLORA_E_ARG, "NULL output");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    launch_routing(adapter_ids, n, h->n_ad, h->rb, nullptr, h->status, s, &h->launches);
    if (n > 0) launch_compact_perm(h->rb, h->n_ad, perm, s, &h->launches);
    CUDA_TRY(cudaMemcpyAsync(seg_off, h->rb.seg_off, sizeof(int) * (h->n_ad + 1), cudaMemcpyDeviceToDevice, s));
    CUDA_TRY(cudaMemcpyAsync(pad_off, h->rb.pad_off, sizeof(int) * (h->n_ad + 1), cudaMemcpyDeviceToDevice, s));
    int ntile_out = (int)(n / TILE_M) + h->n_ad + 1;
    int ncopy = ntile_out < h->max_tiles ? ntile_out : h->max_tiles;
    CUDA_TRY(cudaMemcpyAsync(tile_ad, h->rb.tile_ad, sizeof(int) * ncopy, cudaMemcpyDeviceToDevice, s));
    if (ntile_out > ncopy) CUDA_TRY(cudaMemsetAsync(tile_ad + ncopy, 0xff, sizeof(int) * (ntile_out - ncopy), s));
    CUDA_TRY(cudaGetLastError());
    return MLORA_OK;
}

extern "C" int mlora_check_status(mlora_t* h, void* stream) {
    if (!h) return fail(MLORA_E_ARG, "NULL handle");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CUDA_TRY(cudaStreamSynchronize(s));
    int st = 0;
    CUDA_TRY(cudaMemcpy(&st, h->status, sizeof(int), cudaMemcpyDeviceToHost));
    CUDA_TRY(cudaMemset(h->status, 0, sizeof(int)));
    if (st & ST_TIMEOUT) return fail(MLORA_E_TIMEOUT, "a bounded device wait gave up");
    if (st & ST_RANGE) return fail(MLORA_E_RANGE, "a token, target or adapter id was out of range");
    return MLORA_OK;
}

extern "C" int mlora_save_state(mlora_t* h, const char* path, void* stream) {
    if (!h || !path) return fail(MLORA_E_ARG, "NULL argument");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CUDA_TRY(cudaStreamSynchronize(s));
    std::vector<float> P(h->n_params), M(h->n_params), Vv(h->n_params);
    std::vector<int64_t> steps(h->n_ad);
    CUDA_TRY(cudaMemcpy(P.data(), h->P, sizeof(float) * h->n_params, cudaMemcpyDeviceToHost));
    CUDA_TRY(cudaMemcpy(M.data(), h->M, sizeof(float) * h->n_params, cudaMemcpyDeviceToHost));
    CUDA_TRY(cudaMemcpy(Vv.data(), h->Vm, sizeof(float) * h->n_params, cudaMemcpyDeviceToHost));
    CUDA_TRY(cudaMemcpy(steps.data(), h->step, sizeof(int64_t) * h->n_ad, cudaMemcpyDeviceToHost));
    FILE* fh = fopen(path, "wb");
    if (!fh) return fail(MLORA_E_IO, "cannot open %s for writing", path);
    bool ok = true;
    auto put = [&](const void* p, size_t n) { ok = ok && fwrite(p, 1, n, fh) == n; };
    // The format is little-endian; both supported hosts (x86-64, aarch64) are.
    put("MLORASTA", 8);
    uint32_t hdr[6] = {1u, (uint32_t)h->n_ad, (uint32_t)h->L, (uint32_t)h->d, (uint32_t)h->f, 0u};
    put(hdr, sizeof(hdr));
    for (int a = 0; a < h->n_ad; ++a) {
        uint32_t r = (uint32_t)h->ranks[a];
        float al = h->alphas[a];
        uint64_t st = (uint64_t)steps[a];
        put(&r, 4); put(&al, 4); put(&st, 8);
        const std::vector<float>* grp[3] = {&P, &M, &Vv};
        for (int g = 0; g < 3; ++g)
            for (int l = 0; l < h->L; ++l)
                for (int k = 0; k < 4; ++k)
                    put(grp[g]->data() + tensor_off(h, a, l, k),
                        sizeof(float) * tensor_size(k, h->ranks[a], h->d, h->f));
    }
    ok = (fclose(fh) == 0) && ok;
    if (!ok) return fail(MLORA_E_IO, "write to %s failed", path);
    return MLORA_OK;
}

template <typename T>
static int export_impl(mlora_t* h, int a, int l, int which, void* out, cudaStream_t s) {
    const int r = h->ranks[a];
    // W1 [f x d] = W1 + g B1 [f x r] A1 [r x d];  W2 [d x f] = W2 + g B2 [d x r] A2 [r x f]
    const int M = which == 0 ? h->f : h->d;
    const int N = which == 0 ? h->d : h->f;
    const float* Bf = h->P + tensor_off(h, a, l, which == 0 ? 1 : 3);
    const float* Af = h->P + tensor_off(h, a, l, which == 0 ? 0 : 2);
    const int KP = sizeof(T) == 2 ? 3 * RP : RP;
    launch_merge_operands<T>(Bf, Af, M, N, r, reinterpret_cast<T*>(h->mg_a), reinterpret_cast<T*>(h->mg_b), s);
    ++h->launches;
    GemmParams p;
    p.M = M; p.N = N; p.K = KP; p.Kx = 0;
    p.group_m = band_for_k(KP);
    p.mtiles_dev = nullptr;
    p.mt_base = 0; p.mt_count = (M + TILE_M - 1) / TILE_M;
    p.tile_ad = nullptr;
    p.A = op_kmajor(h->mg_a, M, KP);
    p.B = op_mnmajor(h->mg_b, KP, N);
    p.ep.kind = EPI_MERGE;
    p.ep.aux = which == 0 ? h->W1[l] : h->W2[l];
    p.ep.ld_aux = N;
    p.ep.out0 = out;
    p.ep.ld0 = N;
    p.ep.gamma = h->gamma_d + a;
    return run_gemm<T>(h, p, s, MLORA_PROF_OTHER);
}

extern "C" int mlora_export_merged(mlora_t* h, int32_t adapter, int32_t layer, int32_t which, void* out,
                                   void* stream) {
    if (!h || !out) return fail(MLORA_E_ARG, "NULL argument");
    if (adapter < 0 || adapter >= h->n_ad) return fail(MLORA_E_ARG, "adapter %d out of range", adapter);
    if (layer < 0 || layer >= h->L) return fail(MLORA_E_ARG, "layer %d out of range", layer);
    if (which != 0 && which != 1) return fail(MLORA_E_ARG, "which must be 0 (W1) or 1 (W2)");
    if ((reinterpret_cast<uintptr_t>(out) & 15) != 0) return fail(MLORA_E_ARG, "out must be 16-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int rc = h->dtype == MLORA_BF16 ? export_impl<bf16>(h, adapter, layer, which, out, s)
                                    : export_impl<float>(h, adapter, layer, which, out, s);
    if (rc) return rc;
    CUDA_TRY(cudaGetLastError());
    return MLORA_OK;
}

// Reads the whole file into host memory and checks it before touching the
// handle, so a rejected file leaves the adapter state as it was.
extern "C" int mlora_load_state(mlora_t* h, const char* path, int32_t with_optimizer, void* stream) {
    if (!h || !path) return fail(MLORA_E_ARG, "NULL argument");
    if (with_optimizer != 0 && with_optimizer != 1) return fail(MLORA_E_ARG, "with_optimizer must be 0 or 1");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    FILE* fh = fopen(path, "rb");
    if (!fh) return fail(MLORA_E_IO, "cannot open %s for reading", path);
    std::vector<float> P(h->n_params), M(h->n_params), Vv(h->n_params);
    std::vector<int64_t> steps(h->n_ad);
    bool ok = true;
    auto get = [&](void* p, size_t n) { ok = ok && fread(p, 1, n, fh) == n; return ok; };
    char magic[8];
    uint32_t hdr[6];
    int rc = MLORA_OK;
    if (!get(magic, 8) || memcmp(magic, "MLORASTA", 8) != 0) {
        rc = fail(MLORA_E_IO, "%s is not an adapter checkpoint", path);
    } else if (!get(hdr, sizeof(hdr))) {
        rc = fail(MLORA_E_IO, "%s: truncated header", path);
    } else if (hdr[0] != 1u) {
        rc = fail(MLORA_E_IO, "%s: unsupported checkpoint version %u", path, hdr[0]);
    } else if (hdr[1] != (uint32_t)h->n_ad || hdr[2] != (uint32_t)h->L || hdr[3] != (uint32_t)h->d ||
               hdr[4] != (uint32_t)h->f) {
        rc = fail(MLORA_E_ARG, "%s holds %u adapters, L=%u d=%u f=%u; the handle has %d, L=%d d=%d f=%d",
                  path, hdr[1], hdr[2], hdr[3], hdr[4], h->n_ad, h->L, h->d, h->f);
    }
    for (int a = 0; a < h->n_ad && rc == MLORA_OK; ++a) {
        uint32_t r;
        float al;
        uint64_t st;
        if (!get(&r, 4) || !get(&al, 4) || !get(&st, 8)) {
            rc = fail(MLORA_E_IO, "%s: truncated at adapter %d", path, a);
            break;
        }
        if ((int)r != h->ranks[a] || al != h->alphas[a]) {
            rc = fail(MLORA_E_ARG, "%s: adapter %d has rank %u alpha %g; the handle has rank %d alpha %g",
                      path, a, r, (double)al, h->ranks[a], (double)h->alphas[a]);
            break;
        }
        steps[a] = (int64_t)st;
        std::vector<float>* grp[3] = {&P, &M, &Vv};
        for (int g = 0; g < 3; ++g)
            for (int l = 0; l < h->L; ++l)
                for (int k = 0; k < 4; ++k)
                    get(grp[g]->data() + tensor_off(h, a, l, k),
                        sizeof(float) * tensor_size(k, h->ranks[a], h->d, h->f));
        if (!ok) rc = fail(MLORA_E_IO, "%s: truncated in adapter %d", path, a);
    }
    if (rc == MLORA_OK && fgetc(fh) != EOF) rc = fail(MLORA_E_IO, "%s: trailing bytes", path);
    fclose(fh);
    if (rc != MLORA_OK) return rc;

    const size_t nb = sizeof(float) * h->n_params;
    CUDA_TRY(cudaStreamSynchronize(s));
    CUDA_TRY(cudaMemcpyAsync(h->P, P.data(), nb, cudaMemcpyHostToDevice, s));
    if (with_optimizer) {
        CUDA_TRY(cudaMemcpyAsync(h->M, M.data(), nb, cudaMemcpyHostToDevice, s));
        CUDA_TRY(cudaMemcpyAsync(h->Vm, Vv.data(), nb, cudaMemcpyHostToDevice, s));
        CUDA_TRY(cudaMemcpyAsync(h->step, steps.data(), sizeof(int64_t) * h->n_ad, cudaMemcpyHostToDevice, s));
    } else {
        CUDA_TRY(cudaMemsetAsync(h->M, 0, nb, s));
        CUDA_TRY(cudaMemsetAsync(h->Vm, 0, nb, s));
        CUDA_TRY(cudaMemsetAsync(h->step, 0, sizeof(int64_t) * h->n_ad, s));
    }
    CUDA_TRY(cudaMemsetAsync(h->G, 0, nb, s));
    CUDA_TRY(cudaMemsetAsync(h->touched, 0, sizeof(int) * h->n_ad, s));
    CUDA_TRY(cudaMemsetAsync(h->nonfinite, 0, sizeof(int) * h->n_ad, s));
    if (h->dtype == MLORA_BF16)
        launch_shadow_sync<bf16>(h->n_ad, h->ad_off, h->ranks_d, h->L, h->d, h->f, h->n_params, h->P, h->shadow, s);
    else
        launch_shadow_sync<float>(h->n_ad, h->ad_off, h->ranks_d, h->L, h->d, h->f, h->n_params, h->P, h->shadow, s);
    ++h->launches;
    CUDA_TRY(cudaGetLastError());
    CUDA_TRY(cudaStreamSynchronize(s));
    return MLORA_OK;
}

extern "C" int mlora_set_deterministic(mlora_t* h, int32_t on) {
    if (!h) return fail(MLORA_E_ARG, "NULL handle");
    if (on != 0 && on != 1) return fail(MLORA_E_ARG, "on must be 0 or 1");
    h->deterministic = on;
    return MLORA_OK;
}

// Test hook (not in the public headers) of the bounded device waits: the next
// single-CTA tensor-core GEMM this handle launches (the first LoRA shrink of a
// step) leaves K block `kb` of CTA 0's first tile unloaded, and its MMA thread
// gives up waiting for it after wait_ns nanoseconds.  No copy is in flight for
// that stage, so the kernel raises the timeout status bit, drains what it did
// issue, frees its tensor memory and returns; mlora_check_status then reports
// MLORA_E_TIMEOUT.  kb must be below the GEMM's K blocks (d / 64) to fire.
extern "C" int mlk_test_gemm_withhold(mlora_t* h, int32_t kb, int64_t wait_ns) {
    if (!h || kb < 0 || wait_ns < 0) return fail(MLORA_E_ARG, "bad test-hook argument");
    h->test_withhold_kb = kb;
    h->test_wait_ns = (unsigned long long)wait_ns;
    return MLORA_OK;
}

extern "C" int mlora_set_lm_backward(mlora_t* h, int32_t mode) {
    if (!h) return fail(MLORA_E_ARG, "NULL handle");
    if (mode != MLORA_LM_RECOMPUTE && mode != MLORA_LM_KEEP_LOGITS)
        return fail(MLORA_E_ARG, "unknown LM-head backward mode %d", mode);
    if (mode == h->lm_keep) return MLORA_OK;
    CUDA_TRY(cudaDeviceSynchronize());   // no queued step may still use the buffers
    const size_t rows = (size_t)h->nc_tiles * TILE_M;
    if (mode == MLORA_LM_RECOMPUTE) {
        dfree(h, &h->dz[1]);
        for (int b = 0; b < 2; ++b) dfree(h, &h->zbuf[b]);
        h->lm_keep = 0;
        return MLORA_OK;
    }
    int rc = dalloc(h, &h->dz[1], rows * h->Vpad * h->esize);
    const size_t zes = h->esize == 2 ? 2 : 4;   // fp16 e on the bf16 engine, fp32 logits otherwise
    for (int b = 0; b < 2 && rc == MLORA_OK; ++b) rc = dalloc(h, &h->zbuf[b], rows * h->Vpad * zes);
    if (rc == MLORA_OK && cudaMemset(h->dz[1], 0, rows * h->Vpad * h->esize) != cudaSuccess)
        rc = fail(MLORA_E_CUDA, "cudaMemset of a dz chunk buffer failed");
    if (rc != MLORA_OK) {
        dfree(h, &h->dz[1]);
        for (int b = 0; b < 2; ++b) dfree(h, &h->zbuf[b]);
        return rc;
    }
    h->lm_keep = 1;
    return MLORA_OK;
}

extern "C" int mlora_profile_enable(mlora_t* h, int32_t on) {
    if (!h) return fail(MLORA_E_ARG, "NULL handle");
    h->prof = on != 0;
    return MLORA_OK;
}

extern "C" int mlora_profile_read(mlora_t* h, double* ms_out, int64_t* launches_out, int32_t reset) {
    if (!h) return fail(MLORA_E_ARG, "NULL handle");
    for (size_t i = 0; i < h->ev_used; ++i) {
        CUDA_TRY(cudaEventSynchronize(h->ev[2 * i + 1]));
        float ms = 0.f;
        CUDA_TRY(cudaEventElapsedTime(&ms, h->ev[2 * i], h->ev[2 * i + 1]));
        int c = h->ev_cls[i];
        if (c < 0 || c >= MLORA_PROF_CLASSES) c = MLORA_PROF_OTHER;
        h->prof_ms[c] += ms;
        h->prof_n[c] += 1;
    }
    h->ev_used = 0;
    for (int c = 0; c < MLORA_PROF_CLASSES; ++c) {
        if (ms_out) ms_out[c] = h->prof_ms[c];
        if (launches_out) launches_out[c] = h->prof_n[c];
        if (reset) { h->prof_ms[c] = 0.0; h->prof_n[c] = 0; }
    }
    return MLORA_OK;
}
