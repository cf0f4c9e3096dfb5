// Sampler side of the multi-tenant LoRA path: scoring and one-token decode
// for rows that each name a pinned adapter snapshot ("slot").
//
// OpenTinker (paperlayer.ai summary, "Multi-LoRA rollout"): rollout batches
// active rows by pinned adapter version, reuses the shared base projection
// and adds each row's adapter residual.  tinker-ticks ("Why RL needs
// batch-invariant kernels"): rollout and training logprobs of the same
// tokens must agree bit for bit.
//
// Design.  Rows stay in batch order (no per-adapter padding, which would
// multiply the base GEMM's rows by up to 128 x slots at decode sizes).  Each
// layer runs the same kernels and operand values as the training forward:
//  * shrink: one GEMM of the rows against the rank-64 padded A factors of
//    all slots (N = slots x 64) on the same 128 x 64 single-CTA kernel; its
//    epilogue keeps gamma_s A_s x in column block s for rows of slot s and
//    writes zeros elsewhere (a row-masked, slot-blocked operand);
//  * base GEMM + expand: the base GEMM with a K extension of slots x 64
//    whose B holds every slot's B factor side by side.  A row's extension
//    K blocks are zero except its own slot's, and a zero A row adds exactly
//    zero to the fp32 accumulator, so each row's accumulator is the training
//    path's (main K blocks, then its own adapter's block) bit for bit;
//  * the same SiLU / residual epilogues, LM head and combine.
// Publishing copies a training adapter's current bf16 (or fp32) padded
// factors into a slot: the slot is immutable until published again.
// Sampling inverts the CDF of softmax(z) in vocabulary order at a caller
// supplied uniform u: the vocabulary tile is found from the LM head's
// per-tile log-sum-exp partials, the token inside the tile from the logits
// the LM-head GEMM kept for these rows.
#include <stdarg.h>
#include <stdio.h>

#include <string>
#include <vector>

#include "internal.h"

using namespace mlk;

void mlk_trainer_view(const mlora_t* h, TrainerView* v);
int mlk_report_error(int code, const char* msg);

namespace {

int sfail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int sfail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    return mlk_report_error(code, buf);
}

#define S_TRY(expr)                                                                      \
    do {                                                                                 \
        cudaError_t _e = (expr);                                                         \
        if (_e != cudaSuccess)                                                           \
            return sfail(MLORA_E_CUDA, "%s failed: %s", #expr, cudaGetErrorString(_e));  \
    } while (0)

// ----------------------------------------------------------------------------
// kernels
// ----------------------------------------------------------------------------

// Batch-order row maps for n rows padded to whole 128-row tiles: perm[p] = p
// for a row with a published slot, -1 for padding rows and rows whose slot
// is out of range or unpublished (flagged); row_slot[p] its slot or -1.
// targets: the caller's targets, or the tokens themselves when sampling (so
// the combine forms every row's log-sum-exp).
__global__ void sampler_prep_kernel(const int* __restrict__ slots, int n, int n_pad, int n_slots,
                                    const int* __restrict__ published, int* perm, int* row_slot,
                                    int* meta, int* status) {
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < n_pad; p += gridDim.x * blockDim.x) {
        int sl = -1;
        if (p < n) {
            sl = slots[p];
            if (sl < 0 || sl >= n_slots || !published[sl]) {
                raise_status(status, ST_RANGE);
                sl = -1;
            }
        }
        perm[p] = sl >= 0 ? p : -1;
        row_slot[p] = sl;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        meta[0] = n_pad / TILE_M;
        meta[1] = 0;
    }
}

// One warp per row: inverse CDF of softmax(z) at u in vocabulary order.
//   tile level: cumulative sum of exp(lse_j - lse) over the vocabulary
//   tiles j (lse_j the tile's log-sum-exp partial) until it passes u;
//   inside the chosen tile: cumulative sum of exp(z_v - lse) from the tile's
//   first column.
// When rounding leaves the cumulative sum at or below u, the last column
// with a non-zero probability is taken.  Output: the token and its logprob
// z_v - lse (the value the combine would return for that target).
__global__ void __launch_bounds__(256) sample_kernel(const float* __restrict__ part, int n_nt, int part_ld,
                                                     int bn, const float* __restrict__ z, int64_t ldz, int V,
                                                     const float* __restrict__ lse_row,
                                                     const int* __restrict__ perm,
                                                     const int* __restrict__ tgt_pad,
                                                     const float* __restrict__ uniforms, int n,
                                                     int* next_out, float* lp_out, int* status) {
    const int lane = threadIdx.x & 31;
    const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int p = wid; p < n; p += nwarps) {
        const float u = uniforms[p];
        const bool ok_row = perm[p] >= 0 && tgt_pad[p] >= 0;
        const bool ok_u = u >= 0.f && u < 1.f;
        if (!ok_row || !ok_u) {
            if (lane == 0) {
                if (!ok_u) raise_status(status, ST_RANGE);
                next_out[p] = -1;
                lp_out[p] = __int_as_float(0x7fc00000);
            }
            continue;
        }
        const float lse = lse_row[p];
        const float* prow = part + (int64_t)p * part_ld;
        // --- vocabulary tile
        float run = 0.f;          // mass of the tiles before `base`
        int T = -1, last_nz = -1;
        float before_T = 0.f;
        for (int base = 0; base < n_nt && T < 0; base += 32) {
            const int j = base + lane;
            const float m = j < n_nt ? __expf(prow[j] - lse) : 0.f;
            float c = m;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float x = __shfl_up_sync(0xffffffffu, c, o);
                if (lane >= o) c += x;
            }
            const unsigned nz = __ballot_sync(0xffffffffu, m > 0.f);
            if (nz) last_nz = base + 31 - __clz(nz);
            const unsigned pass = __ballot_sync(0xffffffffu, run + c > u);
            if (pass) {
                const int L = __ffs(pass) - 1;
                T = base + L;
                const float cprev = __shfl_sync(0xffffffffu, c - m, L);
                before_T = run + cprev;
            } else {
                run += __shfl_sync(0xffffffffu, c, 31);
            }
        }
        if (T < 0) {                 // rounding: u at or above the total mass
            T = last_nz >= 0 ? last_nz : 0;
            before_T = -INFINITY;    // take the tile's last non-zero column
        }
        // --- column inside tile T (bn = 256: 8 columns per lane; bn = 32: 1)
        const int c0 = T * bn;
        const int per = bn / 32;
        float pv[8];
        float ls = 0.f;
        for (int e = 0; e < per; ++e) {
            const int v = c0 + lane * per + e;
            pv[e] = v < V ? __expf(z[(int64_t)p * ldz + v] - lse) : 0.f;
            ls += pv[e];
        }
        float c = ls;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float x = __shfl_up_sync(0xffffffffu, c, o);
            if (lane >= o) c += x;
        }
        int pick = -1;
        const unsigned pass = __ballot_sync(0xffffffffu, before_T + c > u);
        if (pass) {
            const int L = __ffs(pass) - 1;
            if (lane == L) {
                float r = before_T + (c - ls);
                for (int e = 0; e < per; ++e) {
                    r += pv[e];
                    if (r > u) { pick = c0 + lane * per + e; break; }
                }
                if (pick < 0) {          // rounding inside the lane's columns
                    for (int e = per - 1; e >= 0; --e)
                        if (pv[e] > 0.f) { pick = c0 + lane * per + e; break; }
                }
            }
            pick = __shfl_sync(0xffffffffu, pick, L);
        }
        if (pick < 0) {                  // last non-zero column of the tile
            int mine = -1;
            for (int e = per - 1; e >= 0; --e)
                if (pv[e] > 0.f) { mine = c0 + lane * per + e; break; }
            const unsigned has = __ballot_sync(0xffffffffu, mine >= 0);
            pick = has ? __shfl_sync(0xffffffffu, mine, 31 - __clz(has)) : c0;
        }
        if (lane == 0) {
            next_out[p] = pick;
            lp_out[p] = z[(int64_t)p * ldz + pick] - lse;
        }
    }
}

__global__ void fill_nan_kernel(float* x, int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        x[i] = __int_as_float(0x7fc00000);
}

}  // namespace

// ----------------------------------------------------------------------------
// handle
// ----------------------------------------------------------------------------
struct mlora_sampler {
    const mlora_t* trainer = nullptr;
    TrainerView tv;
    int n_slots = 0, max_rows = 0, rows_alloc = 0;
    std::vector<void*> allocs;
    std::vector<int> published;         // host copy of the published flags
    std::vector<int> slot_rank;
    std::vector<float> slot_alpha;
    std::vector<int64_t> slot_version;
    // per layer, slot snapshots (trainer dtype):
    //   A1 [n_slots*64 x d]  B1 [f x n_slots*64]  A2 [n_slots*64 x f]  B2 [d x n_slots*64]
    std::vector<void*> A1, B1, A2, B2;
    float* gamma = nullptr;             // [n_slots]
    int* published_d = nullptr;         // [n_slots]
    // rows (rows_alloc = max_rows rounded up to 256)
    void *hb = nullptr, *ub = nullptr, *actb = nullptr, *v1 = nullptr, *v2 = nullptr;
    float* h32 = nullptr;
    float *part = nullptr, *zt = nullptr, *lse = nullptr, *gvec = nullptr, *zbuf = nullptr;
    double* val_row = nullptr;
    int *perm = nullptr, *row_slot = nullptr, *tgt = nullptr, *meta = nullptr;
    int *status = nullptr, *tile_counter = nullptr;
    int64_t launches = 0;
};

static int s_alloc(mlora_sampler_t* s, void** p, size_t bytes) {
    if (bytes == 0) bytes = 16;
    cudaError_t e = mlk_malloc(p, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return sfail(MLORA_E_NOMEM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
    }
    s->allocs.push_back(*p);
    return MLORA_OK;
}

template <typename P>
static void assign_ptr(P*& dst, void* src) { dst = static_cast<P*>(src); }

static void s_free(mlora_sampler_t* s) {
    for (void* p : s->allocs) cudaFree(p);
    s->allocs.clear();
}

extern "C" int mlora_sampler_create(mlora_t* trainer, int32_t n_slots, int64_t max_rows,
                                    mlora_sampler_t** out) {
    if (!trainer || !out) return sfail(MLORA_E_ARG, "NULL argument");
    *out = nullptr;
    if (n_slots < 1 || n_slots > MLORA_SAMPLER_MAX_SLOTS)
        return sfail(MLORA_E_ARG, "n_slots %d outside 1..%d", n_slots, MLORA_SAMPLER_MAX_SLOTS);
    if (max_rows < 1 || max_rows > MLORA_SAMPLER_MAX_ROWS)
        return sfail(MLORA_E_ARG, "max_rows %lld outside 1..%d", (long long)max_rows, MLORA_SAMPLER_MAX_ROWS);
    mlora_sampler_t* s = new mlora_sampler_t();
    s->trainer = trainer;
    mlk_trainer_view(trainer, &s->tv);
    const TrainerView& t = s->tv;
    s->n_slots = n_slots;
    s->max_rows = (int)max_rows;
    s->rows_alloc = (int)((max_rows + 255) / 256 * 256);
    s->published.assign(n_slots, 0);
    s->slot_rank.assign(n_slots, 0);
    s->slot_alpha.assign(n_slots, 0.f);
    s->slot_version.assign(n_slots, -1);
    const size_t es = t.esize, R = (size_t)s->rows_alloc, SK = (size_t)n_slots * RP;
    int rc = MLORA_OK;
#define SALLOC(ptr, bytes) do { void* q_ = nullptr; if ((rc = s_alloc(s, &q_, (bytes))) != MLORA_OK) goto fail_out; \
                                assign_ptr(ptr, q_); } while (0)
    s->A1.assign(t.L, nullptr); s->B1.assign(t.L, nullptr); s->A2.assign(t.L, nullptr); s->B2.assign(t.L, nullptr);
    for (int l = 0; l < t.L; ++l) {
        SALLOC(s->A1[l], SK * t.d * es);
        SALLOC(s->B1[l], (size_t)t.f * SK * es);
        SALLOC(s->A2[l], SK * t.f * es);
        SALLOC(s->B2[l], (size_t)t.d * SK * es);
    }
    SALLOC(s->gamma, sizeof(float) * n_slots);
    SALLOC(s->published_d, sizeof(int) * n_slots);
    SALLOC(s->hb, R * t.d * es);
    SALLOC(s->ub, R * t.f * es);
    SALLOC(s->actb, R * t.f * es);
    SALLOC(s->v1, R * SK * es);
    SALLOC(s->v2, R * SK * es);
    SALLOC(s->h32, R * t.d * sizeof(float));
    SALLOC(s->part, R * t.part_ld * sizeof(float));
    SALLOC(s->zt, R * sizeof(float));
    SALLOC(s->lse, R * sizeof(float));
    SALLOC(s->gvec, R * sizeof(float));
    SALLOC(s->zbuf, R * t.Vpad * sizeof(float));
    SALLOC(s->val_row, R * sizeof(double));
    SALLOC(s->perm, R * sizeof(int));
    SALLOC(s->row_slot, R * sizeof(int));
    SALLOC(s->tgt, R * sizeof(int));
    SALLOC(s->meta, 4 * sizeof(int));
    SALLOC(s->status, sizeof(int));
    SALLOC(s->tile_counter, sizeof(int));
#undef SALLOC
    // a failure while the sampler is filled frees what it holds
#define S_TRY_OUT(expr)                                                                  \
    do {                                                                                 \
        cudaError_t _e = (expr);                                                         \
        if (_e != cudaSuccess) {                                                         \
            rc = sfail(MLORA_E_CUDA, "%s failed: %s", #expr, cudaGetErrorString(_e));    \
            goto fail_out;                                                               \
        }                                                                                \
    } while (0)
    {
        cudaStream_t st = 0;
        for (int l = 0; l < t.L; ++l) {
            S_TRY_OUT(cudaMemsetAsync(s->A1[l], 0, SK * t.d * es, st));
            S_TRY_OUT(cudaMemsetAsync(s->B1[l], 0, (size_t)t.f * SK * es, st));
            S_TRY_OUT(cudaMemsetAsync(s->A2[l], 0, SK * t.f * es, st));
            S_TRY_OUT(cudaMemsetAsync(s->B2[l], 0, (size_t)t.d * SK * es, st));
        }
        S_TRY_OUT(cudaMemsetAsync(s->gamma, 0, sizeof(float) * n_slots, st));
        S_TRY_OUT(cudaMemsetAsync(s->published_d, 0, sizeof(int) * n_slots, st));
        S_TRY_OUT(cudaMemsetAsync(s->status, 0, sizeof(int), st));
        S_TRY_OUT(cudaMemsetAsync(s->v1, 0, R * SK * es, st));
        S_TRY_OUT(cudaMemsetAsync(s->v2, 0, R * SK * es, st));
        S_TRY_OUT(cudaStreamSynchronize(st));
    }
#undef S_TRY_OUT
    *out = s;
    return MLORA_OK;
fail_out:
    s_free(s);
    delete s;
    return rc;
}

extern "C" int mlora_sampler_destroy(mlora_sampler_t* s) {
    if (!s) return MLORA_OK;
    cudaDeviceSynchronize();
    s_free(s);
    delete s;
    return MLORA_OK;
}

// Copy adapter `adapter`'s current padded factors of every layer into `slot`.
extern "C" int mlora_sampler_publish(mlora_sampler_t* s, int32_t slot, int32_t adapter,
                                     int64_t* version_out, void* stream) {
    if (!s) return sfail(MLORA_E_ARG, "NULL sampler");
    const TrainerView& t = s->tv;
    if (slot < 0 || slot >= s->n_slots) return sfail(MLORA_E_ARG, "slot %d out of range", slot);
    if (adapter < 0 || adapter >= t.n_ad) return sfail(MLORA_E_ARG, "adapter %d out of range", adapter);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t es = t.esize, SK = (size_t)s->n_slots * RP, row = RP * es;
    for (int l = 0; l < t.L; ++l) {
        const char* a1 = static_cast<const char*>(t.shadow->A1[l]);
        const char* b1 = static_cast<const char*>(t.shadow->B1[l]);
        const char* a2 = static_cast<const char*>(t.shadow->A2[l]);
        const char* b2 = static_cast<const char*>(t.shadow->B2[l]);
        // A factors: RP contiguous rows; B factors: one RP-wide column block of every row
        S_TRY(cudaMemcpyAsync(static_cast<char*>(s->A1[l]) + (size_t)slot * RP * t.d * es,
                              a1 + (size_t)adapter * RP * t.d * es, (size_t)RP * t.d * es,
                              cudaMemcpyDeviceToDevice, st));
        S_TRY(cudaMemcpyAsync(static_cast<char*>(s->A2[l]) + (size_t)slot * RP * t.f * es,
                              a2 + (size_t)adapter * RP * t.f * es, (size_t)RP * t.f * es,
                              cudaMemcpyDeviceToDevice, st));
        S_TRY(cudaMemcpy2DAsync(static_cast<char*>(s->B1[l]) + (size_t)slot * row, SK * es,
                                b1 + (size_t)adapter * t.f * row, row, row, t.f, cudaMemcpyDeviceToDevice, st));
        S_TRY(cudaMemcpy2DAsync(static_cast<char*>(s->B2[l]) + (size_t)slot * row, SK * es,
                                b2 + (size_t)adapter * t.d * row, row, row, t.d, cudaMemcpyDeviceToDevice, st));
    }
    S_TRY(cudaMemcpyAsync(s->gamma + slot, t.gamma_d + adapter, sizeof(float), cudaMemcpyDeviceToDevice, st));
    int64_t ver = 0;
    S_TRY(cudaMemcpyAsync(&ver, t.step_d + adapter, sizeof(int64_t), cudaMemcpyDeviceToHost, st));
    const int one = 1;
    S_TRY(cudaMemcpyAsync(s->published_d + slot, &one, sizeof(int), cudaMemcpyHostToDevice, st));
    S_TRY(cudaStreamSynchronize(st));
    s->published[slot] = 1;
    s->slot_rank[slot] = t.ranks[adapter];
    s->slot_alpha[slot] = t.alphas[adapter];
    s->slot_version[slot] = ver;
    if (version_out) *version_out = ver;
    return MLORA_OK;
}

// ----------------------------------------------------------------------------
// forward over n rows in batch order
// ----------------------------------------------------------------------------
static int s_gemm(mlora_sampler_t* s, GemmParams& p, cudaStream_t st) {
    p.tile_counter = s->tile_counter;
    if (s->tv.use_tc) {
        cudaError_t e = launch_tc_gemm(p, st, s->tv.num_sms, s->status);
        if (e != cudaSuccess) return sfail(MLORA_E_CUDA, "tensor-core GEMM launch: %s", cudaGetErrorString(e));
    } else if (s->tv.dtype == MLORA_BF16) {
        launch_simt_gemm<bf16>(p, st);
    } else {
        launch_simt_gemm<float>(p, st);
    }
    ++s->launches;
    return MLORA_OK;
}

static GemmOperand s_op(const void* p, int64_t rows, int64_t cols, int mn_major = 0) {
    GemmOperand o;
    o.ptr = p; o.ld = cols; o.rows = rows; o.cols = cols; o.mn_major = mn_major;
    return o;
}

template <typename T>
static int s_forward(mlora_sampler_t* s, const int32_t* tokens, const int32_t* targets,
                     const int32_t* slots, int n, bool keep_logits, float* logprobs_out, cudaStream_t st) {
    const TrainerView& t = s->tv;
    const int mt = (n + TILE_M - 1) / TILE_M;
    const int n_pad = mt * TILE_M;
    const int64_t R = s->rows_alloc;
    const int SK = s->n_slots * RP;
    int rc;
    sampler_prep_kernel<<<(n_pad + 255) / 256, 256, 0, st>>>(slots, n, n_pad, s->n_slots, s->published_d,
                                                             s->perm, s->row_slot, s->meta, s->status);
    ++s->launches;
    launch_embed<T>(s->perm, s->meta, n_pad, tokens, targets, reinterpret_cast<const T*>(t.E), t.V, t.d,
                    reinterpret_cast<T*>(s->hb), s->h32, s->tgt, s->status, st);
    ++s->launches;
    auto dense = [&](int N, int K) {
        GemmParams p;
        p.M = n_pad; p.N = N; p.K = K; p.Kx = 0;
        p.group_m = 8;
        p.mtiles_dev = s->meta;
        p.mt_base = 0; p.mt_count = mt;
        p.tile_ad = nullptr;
        return p;
    };
    // Few rows (decode): when the 256 x 256 pair tiles of a block GEMM would
    // not fill the SMs once while the weights stream, it runs on the 128 x 64
    // single-CTA kernel instead (four times the tiles; the same per-element K
    // order and MMA K step, so the same bits).
    auto small = [&](int N) { return ((mt + 1) / 2) * ((N + 255) / 256) * 2 < t.num_sms; };
    for (int l = 0; l < t.L; ++l) {
        {   // v1[:, s-block] = gamma_s A1_s h on rows of slot s
            GemmParams p = dense(SK, t.d);
            p.force_bn64 = 1;
            p.A = s_op(s->hb, R, t.d);
            p.B = s_op(s->A1[l], SK, t.d);
            p.ep.kind = EPI_SHRINK_SEL; p.ep.out0 = s->v1; p.ep.ld0 = SK; p.ep.gamma = s->gamma;
            p.ep.row_slot = s->row_slot;
            if ((rc = s_gemm(s, p, st))) return rc;
        }
        {   // u = W1 h + sum_s B1_s v1[:, s-block] ; act = silu(u)
            GemmParams p = dense(t.f, t.d);
            p.force_bn64 = small(t.f);
            p.A = s_op(s->hb, R, t.d);
            p.B = s_op(t.W1[l], t.f, t.d);
            p.Kx = SK;
            p.Ax = s_op(s->v1, R, SK);
            p.Bx = s_op(s->B1[l], t.f, SK);
            p.ep.kind = EPI_SILU; p.ep.out0 = s->ub; p.ep.ld0 = t.f; p.ep.out1 = s->actb; p.ep.ld1 = t.f;
            if ((rc = s_gemm(s, p, st))) return rc;
        }
        {   // v2[:, s-block] = gamma_s A2_s act on rows of slot s
            GemmParams p = dense(SK, t.f);
            p.force_bn64 = 1;
            p.A = s_op(s->actb, R, t.f);
            p.B = s_op(s->A2[l], SK, t.f);
            p.ep.kind = EPI_SHRINK_SEL; p.ep.out0 = s->v2; p.ep.ld0 = SK; p.ep.gamma = s->gamma;
            p.ep.row_slot = s->row_slot;
            if ((rc = s_gemm(s, p, st))) return rc;
        }
        {   // h += W2 act + sum_s B2_s v2[:, s-block]
            GemmParams p = dense(t.d, t.f);
            p.force_bn64 = small(t.d);
            p.A = s_op(s->actb, R, t.f);
            p.B = s_op(t.W2[l], t.d, t.f);
            p.Kx = SK;
            p.Ax = s_op(s->v2, R, SK);
            p.Bx = s_op(s->B2[l], t.d, SK);
            p.ep.kind = EPI_RESID; p.ep.f32 = s->h32; p.ep.ldf = t.d; p.ep.out0 = s->hb; p.ep.ld0 = t.d;
            if ((rc = s_gemm(s, p, st))) return rc;
        }
    }
    {   // LM head: per-tile log-sum-exp partials, target logit, and (sampling) the logits
        GemmParams p = dense(t.V, t.d);
        p.A = s_op(s->hb, R, t.d);
        p.B = s_op(t.Wout, t.V, t.d);
        p.ep.kind = EPI_LMFWD; p.ep.part = s->part; p.ep.zt = s->zt; p.ep.tgt = s->tgt;
        p.ep.part_ld = t.part_ld; p.ep.V = t.V; p.ep.Vpad = t.Vpad;
        if (keep_logits) { p.ep.out0 = s->zbuf; p.ep.ld0 = t.Vpad; }
        if ((rc = s_gemm(s, p, st))) return rc;
    }
    LossArgs la;
    la.kind = -1; la.w = la.adv = la.slp = la.dl = nullptr; la.clip = 0.f;
    launch_combine_loss(la, s->part, t.n_nt, t.part_ld, s->zt, s->perm, s->tgt, s->meta, 0, mt, logprobs_out,
                        s->lse, s->gvec, s->val_row, t.num_sms, st);
    ++s->launches;
    S_TRY(cudaGetLastError());
    return MLORA_OK;
}

static int s_check_rows(mlora_sampler_t* s, int64_t n) {
    if (n < 0 || n > s->max_rows) return sfail(MLORA_E_ARG, "n = %lld outside 0..max_rows", (long long)n);
    return MLORA_OK;
}

extern "C" int mlora_sampler_logprobs(mlora_sampler_t* s, const int32_t* tokens, const int32_t* targets,
                                      const int32_t* slots, int64_t n, float* logprobs_out, void* stream) {
    if (!s) return sfail(MLORA_E_ARG, "NULL sampler");
    int rc = s_check_rows(s, n);
    if (rc) return rc;
    if (n > 0 && (!tokens || !targets || !slots || !logprobs_out)) return sfail(MLORA_E_ARG, "NULL argument");
    if (n == 0) return MLORA_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    fill_nan_kernel<<<(int)((n + 255) / 256), 256, 0, st>>>(logprobs_out, (int)n);
    ++s->launches;
    return s->tv.dtype == MLORA_BF16
               ? s_forward<bf16>(s, tokens, targets, slots, (int)n, false, logprobs_out, st)
               : s_forward<float>(s, tokens, targets, slots, (int)n, false, logprobs_out, st);
}

extern "C" int mlora_sampler_sample(mlora_sampler_t* s, const int32_t* tokens, const int32_t* slots,
                                    const float* uniforms, int64_t n, int32_t* next_out, float* logprob_out,
                                    void* stream) {
    if (!s) return sfail(MLORA_E_ARG, "NULL sampler");
    int rc = s_check_rows(s, n);
    if (rc) return rc;
    if (n > 0 && (!tokens || !slots || !uniforms || !next_out || !logprob_out))
        return sfail(MLORA_E_ARG, "NULL argument");
    if (n == 0) return MLORA_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the tokens double as targets: every valid row gets its log-sum-exp
    rc = s->tv.dtype == MLORA_BF16 ? s_forward<bf16>(s, tokens, tokens, slots, (int)n, true, nullptr, st)
                                   : s_forward<float>(s, tokens, tokens, slots, (int)n, true, nullptr, st);
    if (rc) return rc;
    int blocks = (int)((n + 7) / 8);
    if (blocks > s->tv.num_sms * 8) blocks = s->tv.num_sms * 8;
    sample_kernel<<<blocks, 256, 0, st>>>(s->part, s->tv.n_nt, s->tv.part_ld, s->tv.lm_bn, s->zbuf, s->tv.Vpad,
                                          s->tv.V, s->lse, s->perm, s->tgt, uniforms, (int)n, next_out,
                                          logprob_out, s->status);
    ++s->launches;
    S_TRY(cudaGetLastError());
    return MLORA_OK;
}

extern "C" int mlora_sampler_check_status(mlora_sampler_t* s, void* stream) {
    if (!s) return sfail(MLORA_E_ARG, "NULL sampler");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    S_TRY(cudaStreamSynchronize(st));
    int v = 0;
    S_TRY(cudaMemcpy(&v, s->status, sizeof(int), cudaMemcpyDeviceToHost));
    S_TRY(cudaMemset(s->status, 0, sizeof(int)));
    if (v & ST_TIMEOUT) return sfail(MLORA_E_TIMEOUT, "a bounded device wait gave up");
    if (v & ST_RANGE) return sfail(MLORA_E_RANGE, "a token, slot or uniform was out of range");
    return MLORA_OK;
}

extern "C" int64_t mlora_sampler_kernel_launches(const mlora_sampler_t* s) { return s ? s->launches : 0; }
