// gpt2.cu -- the C ABI of libgpt2.so: model state, memory layout, and the
// forward / backward / AdamW step sequence of llm.c "train_gpt2.cu"
// (gpt2_forward, gpt2_zero_grad, gpt2_backward, gpt2_update), rebuilt around
// one stream, one up-front allocation per buffer class, status codes
// instead of exit(), and the sm_103a kernels of this library.
#include "gpt2.h"
#include "internal.h"

#include <cuda_runtime.h>

#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

using namespace gk;

namespace {

char g_err[512] = "no error";
int g_status = GPT2_OK;
unsigned long long g_err_serial = 0;  // counts the errors recorded so far

int fail(int code, const char* fmt, ...) {
    g_status = code;
    g_err_serial++;
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

#define CUDA_TRY(x)                                                                         \
    do {                                                                                    \
        cudaError_t e_ = (x);                                                               \
        if (e_ != cudaSuccess)                                                              \
            return fail(e_ == cudaErrorMemoryAllocation ? GPT2_ERR_NOMEM : GPT2_ERR_CUDA,    \
                        "%s: %s", #x, cudaGetErrorString(e_));                              \
    } while (0)

#define TRY(x)                   \
    do {                         \
        int r_ = (x);            \
        if (r_ != GPT2_OK) return r_; \
    } while (0)

enum Family { FAM_GEMM = 0, FAM_ATTN_FWD, FAM_ATTN_BWD, FAM_LN_FWD, FAM_LN_BWD, FAM_CLASSIFIER,
              FAM_ADAMW, FAM_ENCODER, FAM_OTHER, FAM_COUNT };

struct Timing {
    bool on = false;
    int cap = 0, n = 0;
    std::vector<cudaEvent_t> ev;
    std::vector<int> fam;
    std::vector<double> work;
    double ms[FAM_COUNT] = {0};
    long long launches[FAM_COUNT] = {0};
    double works[FAM_COUNT] = {0};
};

constexpr int kEvents = 16;  // fork / join events of the two-stream backward

struct Model {
    int L, C, NH, V, Vp, maxT, HS;
    int prec;  // GPT2_FP32 / GPT2_BF16 / GPT2_FP16
    int tc;
    DType dt;
    size_t esz;
    size_t sizes[16], offs[16], nparams;
    void* params = nullptr;
    void* grads = nullptr;
    float* master = nullptr;
    LossScaler* scaler = nullptr;  // fp16 training: dynamic loss scaling (device state)
    bool sr = false;  // bf16 without a master copy: AdamW rounds stochastically
    // the seed stream of the stochastic rounding (xorshift*, one draw per update)
    unsigned long long rng_state = 13371337ULL;
    float* mom_m = nullptr;
    float* mom_v = nullptr;
    unsigned int* d_err = nullptr;
    cudaStream_t stream = nullptr;
    cudaStream_t own_stream = nullptr;
    cudaStream_t side = nullptr;  // the backward's weight-gradient stream
    cudaEvent_t ev[kEvents] = {};
    int grad_accum = 1;
    int fwd_done = 0, fwd_targets = 0;
    // activations
    int B = 0, T = 0;
    bool acts = false;
    void* act_mem = nullptr;
    int *tokens = nullptr, *targets = nullptr;
    int* h_pinned = nullptr;  // 2*B*T ints + 1 float
    void *encoded, *ln1, *qkv, *atty, *residual2, *ln2, *fch, *fch_gelu, *residual3, *lnf, *logits;
    float *ln1_mean, *ln1_rstd, *ln2_mean, *ln2_rstd, *lnf_mean, *lnf_rstd, *lse, *losses, *mean_loss;
    void *dresidual, *dbtc, *dbt4c;
    float *attn_D, *ws;
    float* coins = nullptr;    // (T, B) sampling coins of gpt2_sample / gpt2_generate
    int* sampled = nullptr;    // (B) indices drawn by gpt2_sample
    float* gemm_ws = nullptr;  // split-K partials of the weight-gradient GEMMs (side stream)
    float* gemm_ws_main = nullptr;  // split-K partials of the main stream's products
    bool in_side = false;           // launches are being issued for the side stream
    // LayerNorm and bias gradients as partial rows, reduced by one launch at
    // the end of the backward (areas: 2L+1 LayerNorms [ln1 of l = 2l, ln2 of
    // l = 2l+1, lnf = 2L], their column sums when not fused, fc and qkv biases)
    float* gpart = nullptr;
    PartialDesc* d_desc = nullptr;
    int ndesc = 0, P_ln = 0, R_cs = 0;
    // partial rows of the fc bias grad: 32-row groups written by the
    // GELU-backward GEMM's epilogue where it can (R_fcb = ceil(B T / 32)),
    // else R_cs slabs of launch_colsum_part (as for the qkv bias grad)
    int R_fcb = 0;
    bool cs_gemm = false;
    bool ln_fused = false;
    size_t ln_area = 0, cs_off = 0, fcb_off = 0, qkvb_off = 0;
    // gpt2_train_step: the captured step and what it was captured for
    float* d_hyper = nullptr;  // AdamW hyperparameters read by the replayed update
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t graph_exec = nullptr;
    const int* g_tokens = nullptr;
    const int* g_targets = nullptr;
    float* g_loss = nullptr;
    int g_B = 0, g_T = 0, g_accum = 0;
    long long g_launches = 0;  // kernel launches one replay makes
    int *enc_counts, *enc_offsets, *enc_cursor, *enc_order, *enc_sorted;
    // gpt2_train_step_host: device ids and losses of the host-buffer step, and
    // their pinned staging (2*n ids, then k losses); n = k*B*T ids per side
    int* hs_dev = nullptr;
    int* hs_pinned = nullptr;
    size_t hs_n = 0;
    int hs_k = 0;
    Timing timing;
};

Model* g = nullptr;
std::mutex g_mu;

const char* kParamNames[16] = {"wte", "wpe", "ln1w", "ln1b", "qkvw", "qkvb", "attprojw", "attprojb",
                               "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb", "lnfw", "lnfb"};

inline char* P(const Model* m, int t) { return (char*)m->params + m->offs[t] * m->esz; }
inline char* G(const Model* m, int t) { return (char*)m->grads + m->offs[t] * m->esz; }

// ------------------------------------------------------------------ timing
int tbegin(Model* m, int fam, double work) {
    Timing& t = m->timing;
    if (!t.on || t.n >= t.cap) return -1;
    int i = t.n++;
    t.fam[i] = fam;
    t.work[i] = work;
    cudaEventRecord(t.ev[2 * i], m->stream);
    return i;
}
void tend(Model* m, int i) {
    if (i >= 0) cudaEventRecord(m->timing.ev[2 * i + 1], m->stream);
}
#define TIMED(fam, work, stmt)             \
    do {                                   \
        int ti_ = tbegin(m, (fam), (work)); \
        stmt;                              \
        tend(m, ti_);                      \
    } while (0)

// ------------------------------------------------------------------ GEMM dispatch
int gemm(Model* m, int epi, const void* A, long long lda, int a_km, const void* B, long long ldb,
         int b_km, void* D, long long ldd, const void* bias, const void* aux, long long ldaux,
         void* D2, int M, int N, int K, float* cs = nullptr, long long ldcs = 0) {
    GemmParams p;
    memset(&p, 0, sizeof(p));
    p.A = A; p.lda = lda; p.a_kmajor = a_km;
    p.B = B; p.ldb = ldb; p.b_kmajor = b_km;
    p.D = D; p.ldd = ldd; p.bias = bias; p.aux = aux; p.ldaux = ldaux; p.D2 = D2;
    p.M = M; p.N = N; p.K = K; p.epi = epi;
    p.cs = cs; p.ldcs = ldcs;
    // each stream has its own split-K scratch, so concurrent products never share one
    if (m->in_side) {
        if (m->gemm_ws) {
            p.ws = m->gemm_ws;
            p.ws_floats = gemm_ws_floats(m->C);
        }
    } else if (m->gemm_ws_main) {
        p.ws = m->gemm_ws_main;
        p.ws_floats = gemm_ws_main_floats((size_t)m->B * m->T, m->C);
    }
    int rc;
    int ti = tbegin(m, FAM_GEMM, 2.0 * M * N * K);
    if (m->tc) rc = gemm_tc(p, m->dt, m->stream, m->d_err);
    else rc = gemm_simt(p, m->dt, m->stream);
    tend(m, ti);
    if (rc != GPT2_OK) return fail(rc, "gemm (M=%d N=%d K=%d epi=%d) rejected", M, N, K, epi);
    return GPT2_OK;
}

// ------------------------------------------------------------------ lifecycle
void free_acts(Model* m) {
    if (m->act_mem) cudaFree(m->act_mem);
    if (m->gpart) cudaFree(m->gpart);
    if (m->d_desc) cudaFree(m->d_desc);
    m->gpart = nullptr;
    m->d_desc = nullptr;
    if (m->h_pinned) cudaFreeHost(m->h_pinned);
    m->act_mem = nullptr;
    m->h_pinned = nullptr;
    m->acts = false;
}

void free_model(Model* m) {
    if (!m) return;
    if (m->stream) cudaStreamSynchronize(m->stream);
    free_acts(m);
    cudaFree(m->params);
    cudaFree(m->grads);
    cudaFree(m->master);
    cudaFree(m->mom_m);
    cudaFree(m->mom_v);
    cudaFree(m->d_err);
    cudaFree(m->d_hyper);
    cudaFree(m->scaler);
    cudaFree(m->hs_dev);
    if (m->hs_pinned) cudaFreeHost(m->hs_pinned);
    if (m->graph_exec) cudaGraphExecDestroy(m->graph_exec);
    if (m->graph) cudaGraphDestroy(m->graph);
    for (cudaEvent_t e : m->timing.ev) cudaEventDestroy(e);
    if (m->own_stream) cudaStreamDestroy(m->own_stream);
    if (m->side) cudaStreamDestroy(m->side);
    for (cudaEvent_t e : m->ev)
        if (e) cudaEventDestroy(e);
    delete m;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

float* ln_part(const Model* m, int i) { return m->gpart + (size_t)i * m->ln_area; }
float* cs_part(const Model* m, int i) { return m->gpart + m->cs_off + (size_t)i * m->R_cs * m->C; }
float* fcb_part(const Model* m, int l) { return m->gpart + m->fcb_off + (size_t)l * m->R_fcb * 4 * m->C; }
float* qkvb_part(const Model* m, int l) { return m->gpart + m->qkvb_off + (size_t)l * m->R_cs * 3 * m->C; }

// partial-row areas and the device table of their reductions (fixed for a B x T)
int alloc_partials(Model* m) {
    const int L = m->L, C = m->C;
    const int BT = m->B * m->T;
    const size_t es = m->esz;
    m->ln_fused = layernorm_backward_fuses_colsum(m->dt, C);
    m->P_ln = layernorm_backward_part_rows(m->dt, BT, C);
    m->R_cs = colsum_part_rows(BT);
    // GPT2_FUSE_COLSUM=0 computes fc's bias grad partials with a separate
    // column-sum pass instead of in the GELU-backward epilogue (tuning)
    static const bool fuse = [] {
        const char* e = getenv("GPT2_FUSE_COLSUM");
        return e ? atoi(e) != 0 : true;
    }();
    m->cs_gemm = fuse && m->tc != 0 && m->dt != DT_F32;
    m->R_fcb = m->cs_gemm ? (BT + 31) / 32 : m->R_cs;
    m->ln_area = (size_t)m->P_ln * 3 * C;
    m->cs_off = (size_t)(2 * L + 1) * m->ln_area;
    m->fcb_off = m->cs_off + (m->ln_fused ? 0 : (size_t)(2 * L + 1) * m->R_cs * C);
    m->qkvb_off = m->fcb_off + (size_t)L * m->R_fcb * 4 * C;
    const size_t total = m->qkvb_off + (size_t)L * m->R_cs * 3 * C;
    CUDA_TRY(cudaMalloc((void**)&m->gpart, total * 4 + 256));
    std::vector<PartialDesc> d;
    const long long lstride = m->ln_fused ? 3LL * C : 2LL * C;
    auto add = [&](const float* part, long long pstride, int P, int width, char* dst) {
        d.push_back(PartialDesc{part, pstride, P, width, dst});
    };
    // the column sums of LayerNorm i's output: the bias grad of the matmul below it
    auto add_cs = [&](int i, char* dst) {
        if (m->ln_fused) add(ln_part(m, i) + 2 * C, lstride, m->P_ln, C, dst);
        else add(cs_part(m, i), C, m->R_cs, C, dst);
    };
    add(ln_part(m, 2 * L), lstride, m->P_ln, C, G(m, 14));
    add(ln_part(m, 2 * L) + C, lstride, m->P_ln, C, G(m, 15));
    if (L > 0) add_cs(2 * L, G(m, 13) + (size_t)(L - 1) * C * es);
    for (int l = 0; l < L; l++) {
        add(ln_part(m, 2 * l + 1), lstride, m->P_ln, C, G(m, 8) + (size_t)l * C * es);
        add(ln_part(m, 2 * l + 1) + C, lstride, m->P_ln, C, G(m, 9) + (size_t)l * C * es);
        add_cs(2 * l + 1, G(m, 7) + (size_t)l * C * es);
        add(ln_part(m, 2 * l), lstride, m->P_ln, C, G(m, 2) + (size_t)l * C * es);
        add(ln_part(m, 2 * l) + C, lstride, m->P_ln, C, G(m, 3) + (size_t)l * C * es);
        if (l > 0) add_cs(2 * l, G(m, 13) + (size_t)(l - 1) * C * es);
        add(fcb_part(m, l), 4LL * C, m->R_fcb, 4 * C, G(m, 11) + (size_t)l * 4 * C * es);
        add(qkvb_part(m, l), 3LL * C, m->R_cs, 3 * C, G(m, 5) + (size_t)l * 3 * C * es);
    }
    m->ndesc = (int)d.size();
    CUDA_TRY(cudaMalloc((void**)&m->d_desc, d.size() * sizeof(PartialDesc) + 256));
    CUDA_TRY(cudaMemcpy(m->d_desc, d.data(), d.size() * sizeof(PartialDesc), cudaMemcpyHostToDevice));
    return GPT2_OK;
}

int alloc_acts(Model* m, int B, int T) {
    const size_t L = m->L, C = m->C, BT = (size_t)B * T, es = m->esz;
    const size_t NH = m->NH;
    struct Item { void** p; size_t bytes; };
    std::vector<Item> items = {
        {(void**)&m->tokens, BT * 4}, {(void**)&m->targets, BT * 4},
        {&m->encoded, BT * C * es}, {&m->ln1, L * BT * C * es},
        {(void**)&m->ln1_mean, L * BT * 4}, {(void**)&m->ln1_rstd, L * BT * 4},
        {&m->qkv, L * BT * 3 * C * es}, {&m->atty, L * BT * C * es},
        {(void**)&m->lse, L * B * NH * T * 4}, {&m->residual2, L * BT * C * es},
        {&m->ln2, L * BT * C * es}, {(void**)&m->ln2_mean, L * BT * 4},
        {(void**)&m->ln2_rstd, L * BT * 4}, {&m->fch, L * BT * 4 * C * es},
        {&m->fch_gelu, L * BT * 4 * C * es}, {&m->residual3, L * BT * C * es},
        {&m->lnf, BT * C * es}, {(void**)&m->lnf_mean, BT * 4}, {(void**)&m->lnf_rstd, BT * 4},
        {&m->logits, BT * (size_t)m->Vp * es}, {(void**)&m->losses, BT * 4},
        {(void**)&m->mean_loss, 256}, {&m->dresidual, BT * C * es}, {&m->dbtc, BT * C * es},
        {&m->dbt4c, BT * 4 * C * es}, {(void**)&m->attn_D, (size_t)B * NH * T * 4},
        {(void**)&m->ws, 4 * std::max(layernorm_backward_ws_floats(m->C), colsum_ws_floats(4 * m->C))},
        {(void**)&m->gemm_ws, 4 * gemm_ws_floats(m->C)},
        {(void**)&m->gemm_ws_main, 4 * std::max(gemm_ws_floats(m->C), gemm_ws_main_floats(BT, m->C))},
        {(void**)&m->enc_counts, (size_t)m->Vp * 4}, {(void**)&m->enc_offsets, ((size_t)m->Vp + 1) * 4},
        {(void**)&m->enc_cursor, (size_t)m->Vp * 4}, {(void**)&m->enc_order, BT * 4},
        {(void**)&m->enc_sorted, BT * 4},
        {(void**)&m->coins, BT * 4}, {(void**)&m->sampled, (size_t)B * 4},
    };
    size_t total = 0;
    for (auto& it : items) total += align256(it.bytes);
    void* mem = nullptr;
    cudaError_t e = cudaMalloc(&mem, total);
    if (e != cudaSuccess)
        return fail(GPT2_ERR_NOMEM, "activations: cudaMalloc(%zu MiB) failed: %s", total >> 20,
                    cudaGetErrorString(e));
    char* p = (char*)mem;
    for (auto& it : items) {
        *it.p = p;
        p += align256(it.bytes);
    }
    m->act_mem = mem;
    e = cudaMallocHost((void**)&m->h_pinned, 2 * BT * 4 + 16);
    if (e != cudaSuccess) {
        cudaFree(mem);
        m->act_mem = nullptr;
        return fail(GPT2_ERR_NOMEM, "pinned host buffer: %s", cudaGetErrorString(e));
    }
    m->B = B;
    m->T = T;
    m->acts = true;
    return alloc_partials(m);
}

int check_model() {
    if (!g) return fail(GPT2_ERR_STATE, "no model: call gpt2_init first");
    return GPT2_OK;
}

int check_shape(Model* m, int B, int T) {
    if (B <= 0 || T <= 0) return fail(GPT2_ERR_ARG, "B=%d T=%d must be positive", B, T);
    if (T > m->maxT) return fail(GPT2_ERR_SHAPE, "T=%d exceeds maxT=%d", T, m->maxT);
    if (m->acts && (B != m->B || T != m->T))
        return fail(GPT2_ERR_SHAPE, "B,T=%d,%d differ from the first forward's %d,%d", B, T, m->B,
                    m->T);
    if (!m->acts) TRY(alloc_acts(m, B, T));
    return GPT2_OK;
}

int init_params(Model* m, unsigned long long seed) {
    const DType dt = m->dt;
    const float std0 = 0.02f;
    const float std_resid = m->L > 0 ? 0.02f / sqrtf(2.0f * m->L) : 0.02f;
    for (int t = 0; t < 16; t++) {
        void* p = P(m, t);
        size_t n = m->sizes[t];
        const char* nm = kParamNames[t];
        if (!strcmp(nm, "wte")) {
            launch_init_normal(dt, p, (size_t)m->V * m->C, std0, seed, t, m->stream);
            launch_fill(dt, (char*)p + (size_t)m->V * m->C * m->esz, (size_t)(m->Vp - m->V) * m->C, 0.f,
                        m->stream);
        } else if (!strcmp(nm, "wpe") || !strcmp(nm, "qkvw") || !strcmp(nm, "fcw")) {
            launch_init_normal(dt, p, n, std0, seed, t, m->stream);
        } else if (!strcmp(nm, "attprojw") || !strcmp(nm, "fcprojw")) {
            launch_init_normal(dt, p, n, std_resid, seed, t, m->stream);
        } else if (!strcmp(nm, "ln1w") || !strcmp(nm, "ln2w") || !strcmp(nm, "lnfw")) {
            launch_fill(dt, p, n, 1.f, m->stream);
        } else {
            launch_fill(dt, p, n, 0.f, m->stream);
        }
    }
    return GPT2_OK;
}

int reset_optimizer(Model* m) {
    launch_zero(m->mom_m, m->nparams * 4, m->stream);
    launch_zero(m->mom_v, m->nparams * 4, m->stream);
    if (m->master) launch_to_f32(m->dt, m->master, m->params, m->nparams, m->stream);
    return GPT2_OK;
}

// ------------------------------------------------------------------ forward
int run_forward(Model* m, bool has_targets) {
    const int B = m->B, T = m->T, C = m->C, L = m->L, NH = m->NH;
    const size_t BT = (size_t)B * T, es = m->esz;
    const DType dt = m->dt;
    cudaStream_t s = m->stream;
    auto act = [&](void* base, int l, size_t width) { return (char*)base + (size_t)l * BT * width * es; };
    TIMED(FAM_ENCODER, 3.0 * BT * C * es,
          launch_encoder_forward(dt, m->encoded, m->tokens, P(m, 0), P(m, 1), B, T, C, s));
    const double ln_bytes = 2.0 * BT * C * es + 8.0 * BT;
    for (int l = 0; l < L; l++) {
        void* resid_in = l == 0 ? m->encoded : act(m->residual3, l - 1, C);
        void* ln1 = act(m->ln1, l, C);
        void* qkv = act(m->qkv, l, 3 * C);
        void* atty = act(m->atty, l, C);
        void* res2 = act(m->residual2, l, C);
        void* ln2 = act(m->ln2, l, C);
        void* fch = act(m->fch, l, 4 * C);
        void* fchg = act(m->fch_gelu, l, 4 * C);
        void* res3 = act(m->residual3, l, C);
        float* lse = m->lse + (size_t)l * B * NH * T;
        TIMED(FAM_LN_FWD, ln_bytes,
              launch_layernorm_forward(dt, ln1, m->ln1_mean + l * BT, m->ln1_rstd + l * BT, resid_in,
                                       P(m, 2) + (size_t)l * C * es, P(m, 3) + (size_t)l * C * es,
                                       (int)BT, C, s));
        TRY(gemm(m, EPI_STORE, ln1, C, 1, P(m, 4) + (size_t)l * 3 * C * C * es, C, 1, qkv, 3 * C,
                 P(m, 5) + (size_t)l * 3 * C * es, nullptr, 0, nullptr, (int)BT, 3 * C, C));
        {
            int rc_ = GPT2_OK;
            TIMED(FAM_ATTN_FWD, 2.0 * B * NH * (double)T * (T + 1) * (C / NH),
                  rc_ = launch_attention_forward(dt, m->tc, atty, lse, qkv, B, T, C, NH, s, m->d_err));
            if (rc_ != GPT2_OK) return rc_;  // the launcher recorded the reason
        }
        TRY(gemm(m, EPI_RESID, atty, C, 1, P(m, 6) + (size_t)l * C * C * es, C, 1, res2, C,
                 P(m, 7) + (size_t)l * C * es, resid_in, C, nullptr, (int)BT, C, C));
        TIMED(FAM_LN_FWD, ln_bytes,
              launch_layernorm_forward(dt, ln2, m->ln2_mean + l * BT, m->ln2_rstd + l * BT, res2,
                                       P(m, 8) + (size_t)l * C * es, P(m, 9) + (size_t)l * C * es,
                                       (int)BT, C, s));
        TRY(gemm(m, EPI_GELU, ln2, C, 1, P(m, 10) + (size_t)l * 4 * C * C * es, C, 1, fch, 4 * C,
                 P(m, 11) + (size_t)l * 4 * C * es, nullptr, 0, fchg, (int)BT, 4 * C, C));
        TRY(gemm(m, EPI_RESID, fchg, 4 * C, 1, P(m, 12) + (size_t)l * 4 * C * C * es, 4 * C, 1, res3,
                 C, P(m, 13) + (size_t)l * C * es, res2, C, nullptr, (int)BT, C, 4 * C));
    }
    void* last = L == 0 ? m->encoded : act(m->residual3, L - 1, C);
    TIMED(FAM_LN_FWD, ln_bytes,
          launch_layernorm_forward(dt, m->lnf, m->lnf_mean, m->lnf_rstd, last, P(m, 14), P(m, 15),
                                   (int)BT, C, s));
    TRY(gemm(m, EPI_STORE, m->lnf, C, 1, P(m, 0), C, 1, m->logits, m->Vp, nullptr, nullptr, 0,
             nullptr, (int)BT, m->Vp, C));
    if (has_targets) {
        const float dloss = 1.0f / ((float)m->grad_accum * (float)BT);
        TIMED(FAM_CLASSIFIER, 2.0 * BT * m->Vp * es,
              launch_classifier(dt, m->logits, m->losses, m->targets, (int)BT, m->V, m->Vp, dloss, s,
                                m->scaler ? &m->scaler->scale : nullptr));
    }
    CUDA_TRY(cudaGetLastError());
    m->fwd_done = 1;
    m->fwd_targets = has_targets ? 1 : 0;
    return GPT2_OK;
}

// ------------------------------------------------------------------ backward
// The backward as two streams. The main stream carries the chain that feeds
// each next step (dX products, LayerNorm backward, attention backward); the
// weight-gradient products and the fc / qkv bias column sums go to a side
// stream as soon as their inputs exist and are joined right before the first
// kernel that overwrites one of those inputs. The side kernels fill the SMs the
// main kernels leave idle in their last waves. Nothing is reordered within a
// stream, and every tensor still receives the same += in the same order.
int run_backward(Model* m) {
    const int B = m->B, T = m->T, C = m->C, L = m->L, NH = m->NH, Vp = m->Vp;
    const size_t BT = (size_t)B * T, es = m->esz;
    const DType dt = m->dt;
    cudaStream_t s = m->stream;
    const bool par = m->side != nullptr && !m->timing.on;
    cudaStream_t side = par ? m->side : s;
    int evi = 0;
    // the main-stream chain launches at the device's greatest priority, the
    // side stream's at the default one (restored on every return)
    struct PriorityScope {
        explicit PriorityScope(int p) { set_launch_priority(p); }
        ~PriorityScope() { set_launch_priority(0); }
    };
    int prio_least = 0, prio_greatest = 0;
    if (par && cudaDeviceGetStreamPriorityRange(&prio_least, &prio_greatest) != cudaSuccess) prio_greatest = 0;
    PriorityScope prio_scope(par ? prio_greatest : 0);
    // a point on one stream that the other must pass before going on
    auto edge = [&](cudaStream_t from, cudaStream_t to) -> int {
        if (!par) return GPT2_OK;
        cudaEvent_t e = m->ev[evi++ % kEvents];
        CUDA_TRY(cudaEventRecord(e, from));
        CUDA_TRY(cudaStreamWaitEvent(to, e, 0));
        return GPT2_OK;
    };
    // run f with the model's launches going to the side stream
    auto on_side = [&](auto&& f) -> int {
        cudaStream_t keep = m->stream;
        m->stream = side;
        m->in_side = true;
        const int keep_prio = launch_priority();
        set_launch_priority(0);
        const int rc = f();
        set_launch_priority(keep_prio);
        m->in_side = false;
        m->stream = keep;
        return rc;
    };
    // a join: the event is recorded on the side stream now, waited on main later
    auto mark_side = [&](cudaEvent_t& e) -> int {
        if (!par) return GPT2_OK;
        e = m->ev[evi++ % kEvents];
        CUDA_TRY(cudaEventRecord(e, side));
        return GPT2_OK;
    };
    auto wait_side = [&](cudaEvent_t e) -> int {
        if (!par || !e) return GPT2_OK;
        CUDA_TRY(cudaStreamWaitEvent(s, e, 0));
        return GPT2_OK;
    };
    auto act = [&](void* base, int l, size_t width) { return (char*)base + (size_t)l * BT * width * es; };
    const double lnb_bytes = 4.0 * BT * C * es + 8.0 * BT;
    // classifier matmul: dlnf = dlogits . wte (main); dwte += dlogits^T . lnf
    // (side, joined before the encoder backward adds to dwte)
    TRY(edge(s, side));
    TRY(on_side([&] {
        return gemm(m, EPI_ACCUM, m->logits, Vp, 0, m->lnf, C, 0, G(m, 0), C, nullptr, nullptr, 0,
                    nullptr, Vp, C, (int)BT);
    }));
    TRY(gemm(m, EPI_STORE, m->logits, Vp, 1, P(m, 0), C, 0, m->dbtc, C, nullptr, nullptr, 0, nullptr,
             (int)BT, C, Vp));
    void* last = L == 0 ? m->encoded : act(m->residual3, L - 1, C);
    // LayerNorm i backward into its partial area; the column sums of its output
    // (the next-lower matmul's bias grad) come fused or from a colsum pass
    auto ln_bwd = [&](int i, void* inp, const void* w, const float* mean, const float* rstd,
                      int accumulate, bool need_cs) -> int {
        int P_ = 0;
        TIMED(FAM_LN_BWD, lnb_bytes - (accumulate ? 0.0 : 1.0 * BT * C * es),
              P_ = launch_layernorm_backward_part(dt, m->dresidual, ln_part(m, i), m->dbtc, inp, w, mean,
                                                  rstd, (int)BT, C, accumulate, m->ln_fused ? 1 : 0,
                                                  m->d_err, s));
        if (P_ != m->P_ln) return fail(GPT2_ERR_CUDA, "LayerNorm backward partial rows changed");
        if (need_cs && !m->ln_fused)
            TIMED(FAM_OTHER, 1.0 * BT * C * es,
                  launch_colsum_part(dt, cs_part(m, i), m->dresidual, (int)BT, C, s));
        return GPT2_OK;
    };
    TRY(ln_bwd(2 * L, last, P(m, 14), m->lnf_mean, m->lnf_rstd, 0, L > 0));
    cudaEvent_t qkv_done = nullptr;  // the previous layer's qkv weight grad has read dbt4c
    for (int l = L - 1; l >= 0; l--) {
        void* resid_in = l == 0 ? m->encoded : act(m->residual3, l - 1, C);
        void* ln1 = act(m->ln1, l, C);
        void* qkv = act(m->qkv, l, 3 * C);
        void* atty = act(m->atty, l, C);
        void* res2 = act(m->residual2, l, C);
        void* ln2 = act(m->ln2, l, C);
        void* fch = act(m->fch, l, 4 * C);
        void* fchg = act(m->fch_gelu, l, 4 * C);
        float* lse = m->lse + (size_t)l * B * NH * T;
        cudaEvent_t fcproj_w = nullptr, fc_w = nullptr, attproj_w = nullptr;
        // fcproj (W: C x 4C): dW += dresidual^T fch_gelu on the side
        TRY(edge(s, side));
        TRY(on_side([&] {
            return gemm(m, EPI_ACCUM, m->dresidual, C, 0, fchg, 4 * C, 0,
                        G(m, 12) + (size_t)l * 4 * C * C * es, 4 * C, nullptr, nullptr, 0, nullptr, C,
                        4 * C, (int)BT);
        }));
        TRY(mark_side(fcproj_w));
        // dX with the GELU backward fused into its epilogue (overwrites dbt4c)
        TRY(wait_side(qkv_done));
        // (with the column sums of its output, fc's bias grad, where the epilogue can)
        TRY(gemm(m, EPI_GELU_BWD, m->dresidual, C, 1, P(m, 12) + (size_t)l * 4 * C * C * es, 4 * C, 0,
                 m->dbt4c, 4 * C, nullptr, fch, 4 * C, nullptr, (int)BT, 4 * C, C,
                 m->cs_gemm ? fcb_part(m, l) : nullptr, 4LL * C));
        // (fcproj's bias grad: the column sums of the LayerNorm backward above)
        // fc (W: 4C x C): dW and the bias column sums read dbt4c, on the side
        TRY(edge(s, side));
        TRY(on_side([&] {
            TRY(gemm(m, EPI_ACCUM, m->dbt4c, 4 * C, 0, ln2, C, 0, G(m, 10) + (size_t)l * 4 * C * C * es,
                     C, nullptr, nullptr, 0, nullptr, 4 * C, C, (int)BT));
            if (!m->cs_gemm)
                TIMED(FAM_OTHER, 4.0 * BT * C * es,
                      launch_colsum_part(dt, fcb_part(m, l), m->dbt4c, (int)BT, 4 * C, m->stream));
            return GPT2_OK;
        }));
        TRY(mark_side(fc_w));
        TRY(gemm(m, EPI_STORE, m->dbt4c, 4 * C, 1, P(m, 10) + (size_t)l * 4 * C * C * es, C, 0, m->dbtc,
                 C, nullptr, nullptr, 0, nullptr, (int)BT, C, 4 * C));
        // LayerNorm 2 backward adds into dresidual, which fcproj's dW reads
        TRY(wait_side(fcproj_w));
        TRY(ln_bwd(2 * l + 1, res2, P(m, 8) + (size_t)l * C * es, m->ln2_mean + l * BT,
                   m->ln2_rstd + l * BT, 1, true));
        // attention projection (W: C x C): dW on the side
        TRY(edge(s, side));
        TRY(on_side([&] {
            return gemm(m, EPI_ACCUM, m->dresidual, C, 0, atty, C, 0, G(m, 6) + (size_t)l * C * C * es, C,
                        nullptr, nullptr, 0, nullptr, C, C, (int)BT);
        }));
        TRY(mark_side(attproj_w));
        TRY(gemm(m, EPI_STORE, m->dresidual, C, 1, P(m, 6) + (size_t)l * C * C * es, C, 0, m->dbtc, C,
                 nullptr, nullptr, 0, nullptr, (int)BT, C, C));
        // (attproj's bias grad: the column sums of LayerNorm 2's backward)
        // attention: dqkv (B,T,3C) into dbt4c, which fc's dW and bias sums read
        TRY(wait_side(fc_w));
        {
            int rc_ = GPT2_OK;
            TIMED(FAM_ATTN_BWD, 4.0 * B * NH * (double)T * (T + 1) * (C / NH),
                  rc_ = launch_attention_backward(dt, m->tc, m->dbt4c, m->dbtc, qkv, atty, lse, m->attn_D,
                                                  B, T, C, NH, s, m->d_err));
            if (rc_ != GPT2_OK) return rc_;
        }
        // qkv (W: 3C x C): dW and the bias column sums on the side
        TRY(edge(s, side));
        TRY(on_side([&] {
            TRY(gemm(m, EPI_ACCUM, m->dbt4c, 3 * C, 0, ln1, C, 0, G(m, 4) + (size_t)l * 3 * C * C * es, C,
                     nullptr, nullptr, 0, nullptr, 3 * C, C, (int)BT));
            TIMED(FAM_OTHER, 3.0 * BT * C * es,
                  launch_colsum_part(dt, qkvb_part(m, l), m->dbt4c, (int)BT, 3 * C, m->stream));
            return GPT2_OK;
        }));
        TRY(mark_side(qkv_done));
        TRY(gemm(m, EPI_STORE, m->dbt4c, 3 * C, 1, P(m, 4) + (size_t)l * 3 * C * C * es, C, 0, m->dbtc,
                 C, nullptr, nullptr, 0, nullptr, (int)BT, C, 3 * C));
        // LayerNorm 1 backward adds into dresidual, which attproj's dW reads
        TRY(wait_side(attproj_w));
        TRY(ln_bwd(2 * l, resid_in, P(m, 2) + (size_t)l * C * es, m->ln1_mean + l * BT,
                   m->ln1_rstd + l * BT, 1, l > 0));
    }
    // everything on the side stream is done before the sums are read
    TRY(edge(side, s));
    // every LayerNorm and bias grad: += its partial rows, summed in order
    TIMED(FAM_OTHER, 0.0, launch_reduce_partials_multi(dt, m->d_desc, m->ndesc, 4 * C, s));
    TIMED(FAM_ENCODER, 2.0 * BT * C * es,
          launch_encoder_backward(dt, G(m, 0), G(m, 1), m->dresidual, m->tokens, B, T, C, Vp,
                                  m->enc_counts, m->enc_offsets, m->enc_cursor, m->enc_order,
                                  m->enc_sorted, s));
    CUDA_TRY(cudaGetLastError());
    return GPT2_OK;
}

int read_err(Model* m) {
    unsigned int h = 0;
    CUDA_TRY(cudaMemcpyAsync(&h, m->d_err, 4, cudaMemcpyDeviceToHost, m->stream));
    CUDA_TRY(cudaStreamSynchronize(m->stream));
    if (h) {
        unsigned int z = 0;
        cudaMemcpyAsync(m->d_err, &z, 4, cudaMemcpyHostToDevice, m->stream);
        cudaStreamSynchronize(m->stream);
        if (h & DEVERR_TIMEOUT)
            return fail(GPT2_ERR_DEVICE_TIMEOUT, "a bounded in-kernel wait expired");
        if (h & DEVERR_TOKEN) return fail(GPT2_ERR_TOKEN, "a token id outside [0, V) was seen");
    }
    return GPT2_OK;
}

int to_host_f32(Model* m, float* host, const void* src, size_t n, DType dt) {
    float* tmp = nullptr;
    CUDA_TRY(cudaMalloc(&tmp, n * 4 + 16));
    launch_to_f32(dt, tmp, src, n, m->stream);
    cudaError_t e = cudaMemcpyAsync(host, tmp, n * 4, cudaMemcpyDeviceToHost, m->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(m->stream);
    cudaFree(tmp);
    if (e != cudaSuccess) return fail(GPT2_ERR_CUDA, "copy to host: %s", cudaGetErrorString(e));
    return GPT2_OK;
}

}  // namespace

namespace {
// llm.c "train_gpt2.cu", random_u32: xorshift* on the 64-bit state
uint32_t random_u32(unsigned long long* state) {
    unsigned long long x = *state;
    x ^= x >> 12;
    x ^= x << 25;
    x ^= x >> 27;
    *state = x;
    return (uint32_t)((x * 0x2545F4914F6CDD1DULL) >> 32);
}

// hyper != NULL: the launch is being recorded and reads its hyperparameters
// (and the rounding seed) from device memory at replay time
int run_adamw(Model* m, float lr, float beta1, float beta2, float eps, float weight_decay, int step,
              const float* hyper) {
    const float c1 = 1.0f - powf(beta1, (float)step);
    const float c2 = 1.0f - powf(beta2, (float)step);
    const double bytes = (double)m->nparams *
                         (m->master ? (2 * m->esz + 24) : m->sr ? (3.0 * m->esz + 16) : (4.0 * 7));
    const uint32_t seed = m->sr && !hyper ? random_u32(&m->rng_state) : 0u;
    // fp16: an update whose gradients overflowed is skipped and the scale adapts
    if (m->scaler)
        TIMED(FAM_OTHER, (double)m->nparams * m->esz,
              launch_nonfinite(m->dt, m->grads, m->nparams, m->scaler, m->stream));
    TIMED(FAM_ADAMW, bytes,
          launch_adamw(m->dt, m->params, m->master, m->grads, m->mom_m, m->mom_v, m->nparams, lr,
                       beta1, beta2, c1, c2, eps, weight_decay, hyper, m->stream, m->sr, seed, m->scaler));
    if (m->scaler) TIMED(FAM_OTHER, 0.0, launch_scaler_update(m->scaler, m->stream));
    CUDA_TRY(cudaGetLastError());
    return GPT2_OK;
}
}  // namespace

int gk::set_error(int code, const char* fmt, ...) {
    g_status = code;
    g_err_serial++;
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

unsigned long long gk::error_serial() { return g_err_serial; }

// =================================================================== C ABI
extern "C" {

const char* gpt2_last_error(void) { return g_err; }

int gpt2_last_status(void) { return g_status; }

long long gpt2_launch_count(void) { return launch_count(); }

int gpt2_init_ex(int L, int C, int NH, int V, int Vp, int maxT, unsigned long long seed,
                 int precision, int tensor_cores) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (L < 0 || C <= 0 || NH <= 0 || V <= 0 || Vp < V || maxT <= 0 || C % NH)
        return fail(GPT2_ERR_CONFIG, "invalid dims L=%d C=%d NH=%d V=%d Vp=%d maxT=%d", L, C, NH, V,
                    Vp, maxT);
    const int HS = C / NH;
    if (HS != 16 && HS != 32 && HS != 64 && HS != 128)
        return fail(GPT2_ERR_CONFIG, "head size %d not in {16,32,64,128}", HS);
    if (C % 8 || Vp % 8) return fail(GPT2_ERR_CONFIG, "C and Vp must be multiples of 8");
    if (precision != GPT2_FP32 && precision != GPT2_BF16 && precision != GPT2_FP16)
        return fail(GPT2_ERR_CONFIG, "precision %d unknown", precision);
    if (precision == GPT2_FP32 && tensor_cores)
        return fail(GPT2_ERR_CONFIG, "fp32 training runs on the SIMT path (tensor_cores=0)");
    if (C > (precision == GPT2_FP32 ? 1024 : 2048))
        return fail(GPT2_ERR_CONFIG, "C=%d too large for the row-in-registers LayerNorm", C);
    if (g) {
        free_model(g);
        g = nullptr;
    }
    Model* m = new Model();
    m->L = L; m->C = C; m->NH = NH; m->V = V; m->Vp = Vp; m->maxT = maxT; m->HS = HS;
    m->prec = precision;
    m->tc = tensor_cores ? 1 : 0;
    m->dt = precision == GPT2_BF16 ? DT_BF16 : precision == GPT2_FP16 ? DT_F16 : DT_F32;
    m->esz = dtype_size(m->dt);
    const size_t Cs = C, Ls = L;
    size_t sz[16] = {(size_t)Vp * Cs, (size_t)maxT * Cs, Ls * Cs, Ls * Cs, Ls * 3 * Cs * Cs,
                     Ls * 3 * Cs, Ls * Cs * Cs, Ls * Cs, Ls * Cs, Ls * Cs, Ls * 4 * Cs * Cs,
                     Ls * 4 * Cs, Ls * Cs * 4 * Cs, Ls * Cs, Cs, Cs};
    size_t off = 0;
    for (int i = 0; i < 16; i++) {
        m->sizes[i] = sz[i];
        m->offs[i] = off;
        off += sz[i];
    }
    m->nparams = off;
    cudaError_t e = cudaStreamCreateWithFlags(&m->own_stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
        delete m;
        return fail(GPT2_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
    }
    m->stream = m->own_stream;
    if (cudaStreamCreateWithFlags(&m->side, cudaStreamNonBlocking) != cudaSuccess) m->side = nullptr;
    for (int i = 0; m->side && i < kEvents; i++)
        if (cudaEventCreateWithFlags(&m->ev[i], cudaEventDisableTiming) != cudaSuccess) {
            cudaStreamDestroy(m->side);  // stay on one stream
            m->side = nullptr;
        }
    bool ok = cudaMalloc(&m->params, off * m->esz + 256) == cudaSuccess &&
              cudaMalloc(&m->grads, off * m->esz + 256) == cudaSuccess &&
              cudaMalloc((void**)&m->mom_m, off * 4 + 256) == cudaSuccess &&
              cudaMalloc((void**)&m->mom_v, off * 4 + 256) == cudaSuccess &&
              cudaMalloc((void**)&m->d_err, 256) == cudaSuccess &&
              cudaMalloc((void**)&m->d_hyper, 256) == cudaSuccess &&
              (precision == GPT2_FP32 || cudaMalloc((void**)&m->master, off * 4 + 256) == cudaSuccess) &&
              (precision != GPT2_FP16 || cudaMalloc((void**)&m->scaler, 256) == cudaSuccess);
    if (!ok) {
        free_model(m);
        return fail(GPT2_ERR_NOMEM, "parameter/optimizer allocation (%zu params) failed", off);
    }
    launch_zero(m->d_err, 4, m->stream);
    if (m->scaler) {
        // loss scale 2^16, doubled after 2000 good steps in a row
        const LossScaler sc = {65536.f, 0, 0, 2000, 0};
        e = cudaMemcpyAsync(m->scaler, &sc, sizeof(sc), cudaMemcpyHostToDevice, m->stream);
        if (e != cudaSuccess) {
            free_model(m);
            return fail(GPT2_ERR_CUDA, "loss scaler: %s", cudaGetErrorString(e));
        }
    }
    init_params(m, seed);
    launch_zero(m->grads, off * m->esz, m->stream);
    reset_optimizer(m);
    e = cudaStreamSynchronize(m->stream);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        free_model(m);
        return fail(GPT2_ERR_CUDA, "init: %s", cudaGetErrorString(e));
    }
    g = m;
    return GPT2_OK;
}

int gpt2_init(int L, int C, int NH, int V, int Vp, int maxT, unsigned long long seed) {
    return gpt2_init_ex(L, C, NH, V, Vp, maxT, seed, GPT2_BF16, 1);
}

int gpt2_set_stream(void* stream) {
    TRY(check_model());
    cudaStream_t s = stream ? (cudaStream_t)stream : g->own_stream;
    if (s != g->stream) {
        CUDA_TRY(cudaStreamSynchronize(g->stream));
        g->stream = s;
    }
    return GPT2_OK;
}

int gpt2_forward_device(const int* d_tokens, const int* d_targets, int B, int T, float* d_mean_loss) {
    TRY(check_model());
    Model* m = g;
    if (!d_tokens) return fail(GPT2_ERR_ARG, "tokens is NULL");
    TRY(check_shape(m, B, T));
    const int n = B * T;
    launch_copy_tokens(d_tokens, m->tokens, n, m->V, m->d_err, m->stream);
    if (d_targets) launch_copy_tokens(d_targets, m->targets, n, m->V, m->d_err, m->stream);
    TRY(run_forward(m, d_targets != nullptr));
    if (d_targets) launch_mean(m->losses, n, d_mean_loss ? d_mean_loss : m->mean_loss, m->stream);
    CUDA_TRY(cudaGetLastError());
    return GPT2_OK;
}

float gpt2_forward(const int* tokens, const int* targets, int B, int T) {
    if (check_model() != GPT2_OK) return NAN;
    Model* m = g;
    if (!tokens) {
        fail(GPT2_ERR_ARG, "tokens is NULL");
        return NAN;
    }
    if (check_shape(m, B, T) != GPT2_OK) return NAN;
    const int n = B * T;
    for (int i = 0; i < n; i++) {
        if (tokens[i] < 0 || tokens[i] >= m->V || (targets && (targets[i] < 0 || targets[i] >= m->V))) {
            fail(GPT2_ERR_TOKEN, "id at position %d outside [0, %d)", i, m->V);
            return NAN;
        }
    }
    // pinned staging: the previous step's copies have completed (its loss read synchronised)
    memcpy(m->h_pinned, tokens, (size_t)n * 4);
    if (targets) memcpy(m->h_pinned + n, targets, (size_t)n * 4);
    if (cudaMemcpyAsync(m->tokens, m->h_pinned, (size_t)n * 4, cudaMemcpyHostToDevice, m->stream) !=
            cudaSuccess ||
        (targets && cudaMemcpyAsync(m->targets, m->h_pinned + n, (size_t)n * 4,
                                    cudaMemcpyHostToDevice, m->stream) != cudaSuccess)) {
        fail(GPT2_ERR_CUDA, "token upload failed");
        return NAN;
    }
    if (run_forward(m, targets != nullptr) != GPT2_OK) return NAN;
    if (!targets) {
        if (cudaStreamSynchronize(m->stream) != cudaSuccess) {
            fail(GPT2_ERR_CUDA, "forward failed: %s", cudaGetErrorString(cudaGetLastError()));
            return NAN;
        }
        return -1.0f;
    }
    launch_mean(m->losses, n, m->mean_loss, m->stream);
    float* h_loss = (float*)(m->h_pinned + 2 * n);
    if (cudaMemcpyAsync(h_loss, m->mean_loss, 4, cudaMemcpyDeviceToHost, m->stream) != cudaSuccess ||
        cudaStreamSynchronize(m->stream) != cudaSuccess) {
        fail(GPT2_ERR_CUDA, "forward failed: %s", cudaGetErrorString(cudaGetLastError()));
        return NAN;
    }
    return *h_loss;
}

int gpt2_zero_grad(void) {
    TRY(check_model());
    Model* m = g;
    TIMED(FAM_OTHER, (double)m->nparams * m->esz, launch_zero(m->grads, m->nparams * m->esz, m->stream));
    CUDA_TRY(cudaGetLastError());
    return GPT2_OK;
}

int gpt2_set_grad_accum(int k) {
    TRY(check_model());
    if (k < 1) return fail(GPT2_ERR_ARG, "grad accumulation k=%d must be >= 1", k);
    g->grad_accum = k;
    return GPT2_OK;
}

int gpt2_get_grad_accum(void) {
    TRY(check_model());
    return g->grad_accum;
}

int gpt2_backward(void) {
    TRY(check_model());
    if (!g->fwd_done || !g->fwd_targets)
        return fail(GPT2_ERR_STATE, "backward needs a preceding forward with targets");
    TRY(run_backward(g));
    g->fwd_targets = 0;  // dlogits have been consumed
    return GPT2_OK;
}

int gpt2_adamw(float lr, float beta1, float beta2, float eps, float weight_decay, int step) {
    TRY(check_model());
    if (step < 1) return fail(GPT2_ERR_ARG, "step=%d must be >= 1", step);
    return run_adamw(g, lr, beta1, beta2, eps, weight_decay, step, nullptr);
}

// The whole step as CUDA graph replays. The first call with a given set of
// buffers, shape and accumulation count runs the step eagerly (which also
// performs every allocation and one-time set-up) and then records the same
// launches into a graph; later calls write the AdamW hyperparameters to
// device memory with one tiny kernel and replay the graph.
int gpt2_train_step(const int* d_tokens, const int* d_targets, int B, int T, float lr, float beta1,
                    float beta2, float eps, float weight_decay, int step, float* d_mean_loss) {
    TRY(check_model());
    Model* m = g;
    if (!d_tokens || !d_targets) return fail(GPT2_ERR_ARG, "tokens and targets are required");
    if (step < 1) return fail(GPT2_ERR_ARG, "step=%d must be >= 1", step);
    TRY(check_shape(m, B, T));
    const bool same = m->graph_exec && m->g_tokens == d_tokens && m->g_targets == d_targets &&
                      m->g_loss == d_mean_loss && m->g_B == B && m->g_T == T &&
                      m->g_accum == m->grad_accum;
    if (same && !m->timing.on) {
        const float c1 = 1.0f - powf(beta1, (float)step), c2 = 1.0f - powf(beta2, (float)step);
        const uint32_t seed = m->sr ? random_u32(&m->rng_state) : 0u;
        launch_set_hyper(m->d_hyper, lr, beta1, beta2, c1, c2, eps, weight_decay, seed, m->stream);
        CUDA_TRY(cudaGraphLaunch(m->graph_exec, m->stream));
        note_launch((int)m->g_launches);
        m->fwd_done = 1;
        m->fwd_targets = 0;
        return GPT2_OK;
    }
    // zero_grad, then k micro-steps (forward, backward) on consecutive B*T slices
    const int k = m->grad_accum;
    const size_t n = (size_t)B * T;
    auto micro_steps = [&]() -> int {
        TRY(gpt2_zero_grad());
        for (int i = 0; i < k; i++) {
            TRY(gpt2_forward_device(d_tokens + i * n, d_targets + i * n, B, T,
                                    d_mean_loss ? d_mean_loss + i : nullptr));
            TRY(gpt2_backward());
        }
        return GPT2_OK;
    };
    // eager step
    TRY(micro_steps());
    TRY(run_adamw(m, lr, beta1, beta2, eps, weight_decay, step, nullptr));
    if (m->timing.on) return GPT2_OK;  // timing events are not recorded into graphs
    // record the step for the next calls
    if (m->graph_exec) cudaGraphExecDestroy(m->graph_exec);
    if (m->graph) cudaGraphDestroy(m->graph);
    m->graph_exec = nullptr;
    m->graph = nullptr;
    const long long l0 = launch_count();
    CUDA_TRY(cudaStreamBeginCapture(m->stream, cudaStreamCaptureModeThreadLocal));
    int rc = micro_steps();
    if (rc == GPT2_OK) rc = run_adamw(m, lr, beta1, beta2, eps, weight_decay, step, m->d_hyper);
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(m->stream, &graph);
    if (rc != GPT2_OK || e != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        cudaGetLastError();
        return rc != GPT2_OK ? rc : fail(GPT2_ERR_CUDA, "step capture failed: %s", cudaGetErrorString(e));
    }
    e = cudaGraphInstantiate(&m->graph_exec, graph, 0);
    if (e != cudaSuccess) {
        cudaGraphDestroy(graph);
        m->graph_exec = nullptr;
        return fail(GPT2_ERR_CUDA, "step graph instantiation failed: %s", cudaGetErrorString(e));
    }
    m->graph = graph;
    m->g_launches = launch_count() - l0;
    m->g_tokens = d_tokens;
    m->g_targets = d_targets;
    m->g_loss = d_mean_loss;
    m->g_B = B;
    m->g_T = T;
    m->g_accum = m->grad_accum;
    // the capture recorded launches but ran nothing; undo its count
    note_launch(-(int)m->g_launches);
    m->fwd_done = 1;
    m->fwd_targets = 0;
    return GPT2_OK;
}

int gpt2_train_step_host(const int* tokens, const int* targets, int B, int T, float lr, float beta1,
                         float beta2, float eps, float weight_decay, int step, float* mean_loss) {
    TRY(check_model());
    Model* m = g;
    if (!tokens || !targets) return fail(GPT2_ERR_ARG, "tokens and targets are required");
    if (B <= 0 || T <= 0) return fail(GPT2_ERR_ARG, "B=%d T=%d must be positive", B, T);
    const int k = m->grad_accum;
    const size_t n = (size_t)k * B * T;
    for (size_t i = 0; i < n; i++)
        if (tokens[i] < 0 || tokens[i] >= m->V || targets[i] < 0 || targets[i] >= m->V)
            return fail(GPT2_ERR_TOKEN, "id at position %zu outside [0, %d)", i, m->V);
    // device ids and pinned staging, kept for the next calls of the same size
    if (m->hs_n != n || m->hs_k != k) {
        CUDA_TRY(cudaStreamSynchronize(m->stream));
        cudaFree(m->hs_dev);
        if (m->hs_pinned) cudaFreeHost(m->hs_pinned);
        m->hs_dev = nullptr;
        m->hs_pinned = nullptr;
        m->hs_n = 0;
        const size_t bytes = (2 * n + (size_t)k) * 4;
        CUDA_TRY(cudaMalloc((void**)&m->hs_dev, bytes + 256));
        CUDA_TRY(cudaMallocHost((void**)&m->hs_pinned, bytes + 256));
        m->hs_n = n;
        m->hs_k = k;
    }
    // the previous call synchronised, so its copies out of the staging are done
    memcpy(m->hs_pinned, tokens, n * 4);
    memcpy(m->hs_pinned + n, targets, n * 4);
    CUDA_TRY(cudaMemcpyAsync(m->hs_dev, m->hs_pinned, 2 * n * 4, cudaMemcpyHostToDevice, m->stream));
    float* d_loss = (float*)(m->hs_dev + 2 * n);
    TRY(gpt2_train_step(m->hs_dev, m->hs_dev + n, B, T, lr, beta1, beta2, eps, weight_decay, step,
                        d_loss));
    float* h_loss = (float*)(m->hs_pinned + 2 * n);
    CUDA_TRY(cudaMemcpyAsync(h_loss, d_loss, (size_t)k * 4, cudaMemcpyDeviceToHost, m->stream));
    CUDA_TRY(cudaStreamSynchronize(m->stream));
    TRY(read_err(m));
    if (mean_loss) memcpy(mean_loss, h_loss, (size_t)k * 4);
    return GPT2_OK;
}

int gpt2_set_wait_limit(unsigned long long ns) {
    const int rc[5] = {set_wait_limit_gemm(ns), set_wait_limit_attn_fwd(ns), set_wait_limit_attn_bwd(ns),
                       set_wait_limit_kernels(ns), set_wait_limit_fused(ns)};
    for (int r : rc)
        if (r != GPT2_OK) return fail(GPT2_ERR_CUDA, "setting the wait limit failed on the current device");
    return GPT2_OK;
}

int gpt2_sync(void) {
    TRY(check_model());
    CUDA_TRY(cudaStreamSynchronize(g->stream));
    return read_err(g);
}

size_t gpt2_num_params(void) { return g ? g->nparams : 0; }

int gpt2_param_sizes(size_t out[16]) {
    TRY(check_model());
    if (!out) return fail(GPT2_ERR_ARG, "out is NULL");
    for (int i = 0; i < 16; i++) out[i] = g->sizes[i];
    return GPT2_OK;
}

int gpt2_get_params(float* host) {
    TRY(check_model());
    if (!host) return fail(GPT2_ERR_ARG, "host is NULL");
    return to_host_f32(g, host, g->params, g->nparams, g->dt);
}

// fp16: the current loss scale (1 otherwise); synchronises
static int current_scale(Model* m, float* scale) {
    *scale = 1.f;
    if (!m->scaler) return GPT2_OK;
    CUDA_TRY(cudaMemcpyAsync(scale, &m->scaler->scale, 4, cudaMemcpyDeviceToHost, m->stream));
    CUDA_TRY(cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

int gpt2_get_grads(float* host) {
    TRY(check_model());
    if (!host) return fail(GPT2_ERR_ARG, "host is NULL");
    TRY(to_host_f32(g, host, g->grads, g->nparams, g->dt));
    float sc;
    TRY(current_scale(g, &sc));
    if (sc != 1.f) {  // the stored gradients are loss-scaled
        const float inv = 1.f / sc;
        for (size_t i = 0; i < g->nparams; i++) host[i] *= inv;
    }
    return GPT2_OK;
}

int gpt2_set_loss_scaling(float init_scale, int growth_interval) {
    TRY(check_model());
    Model* m = g;
    if (!m->scaler) return fail(GPT2_ERR_CONFIG, "loss scaling exists in GPT2_FP16 mode only");
    int ex = 0;
    if (!(init_scale > 0.f) || frexpf(init_scale, &ex) != 0.5f || growth_interval < 1)
        return fail(GPT2_ERR_ARG, "loss scale must be a power of two and growth_interval >= 1");
    const LossScaler sc = {init_scale, 0, 0, growth_interval, 0};
    CUDA_TRY(cudaMemcpyAsync(m->scaler, &sc, sizeof(sc), cudaMemcpyHostToDevice, m->stream));
    CUDA_TRY(cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

int gpt2_get_loss_scale(float* scale, long long* skipped) {
    TRY(check_model());
    Model* m = g;
    LossScaler sc = {1.f, 0, 0, 0, 0};
    if (m->scaler) {
        CUDA_TRY(cudaMemcpyAsync(&sc, m->scaler, sizeof(sc), cudaMemcpyDeviceToHost, m->stream));
        CUDA_TRY(cudaStreamSynchronize(m->stream));
    }
    if (scale) *scale = sc.scale;
    if (skipped) *skipped = sc.skipped;
    return GPT2_OK;
}

int gpt2_set_master_weights(int enabled) {
    TRY(check_model());
    Model* m = g;
    if (m->prec != GPT2_BF16)
        return enabled ? GPT2_OK : fail(GPT2_ERR_CONFIG, "only bf16 training runs without master weights");
    if (enabled && !m->master) {
        CUDA_TRY(cudaStreamSynchronize(m->stream));
        CUDA_TRY(cudaMalloc((void**)&m->master, m->nparams * 4 + 256));
        launch_to_f32(m->dt, m->master, m->params, m->nparams, m->stream);
        m->sr = false;
    } else if (!enabled && m->master) {
        CUDA_TRY(cudaStreamSynchronize(m->stream));
        cudaFree(m->master);
        m->master = nullptr;
        m->sr = true;
    }
    // a recorded step holds the old update kernel
    if (m->graph_exec) cudaGraphExecDestroy(m->graph_exec);
    if (m->graph) cudaGraphDestroy(m->graph);
    m->graph_exec = nullptr;
    m->graph = nullptr;
    CUDA_TRY(cudaGetLastError());
    return GPT2_OK;
}

int gpt2_get_master(float* host) {
    TRY(check_model());
    if (!host) return fail(GPT2_ERR_ARG, "host is NULL");
    if (!g->master) return fail(GPT2_ERR_STATE, "no master weights (fp32 mode, or turned off)");
    return to_host_f32(g, host, g->master, g->nparams, DT_F32);
}

int gpt2_set_params(const float* host) {
    TRY(check_model());
    if (!host) return fail(GPT2_ERR_ARG, "host is NULL");
    Model* m = g;
    float* tmp = nullptr;
    CUDA_TRY(cudaMalloc(&tmp, m->nparams * 4 + 16));
    cudaError_t e = cudaMemcpyAsync(tmp, host, m->nparams * 4, cudaMemcpyHostToDevice, m->stream);
    if (e == cudaSuccess) {
        launch_from_f32(m->dt, m->params, tmp, m->nparams, m->stream);
        reset_optimizer(m);
        e = cudaStreamSynchronize(m->stream);
    }
    cudaFree(tmp);
    if (e != cudaSuccess) return fail(GPT2_ERR_CUDA, "set_params: %s", cudaGetErrorString(e));
    return GPT2_OK;
}

int gpt2_set_grads(const float* host) {
    TRY(check_model());
    if (!host) return fail(GPT2_ERR_ARG, "host is NULL");
    Model* m = g;
    float sc;
    TRY(current_scale(m, &sc));
    std::vector<float> scaled;
    if (sc != 1.f) {  // stored loss-scaled, as the backward leaves them
        scaled.assign(host, host + m->nparams);
        for (float& x : scaled) x *= sc;
        host = scaled.data();
    }
    float* tmp = nullptr;
    CUDA_TRY(cudaMalloc(&tmp, m->nparams * 4 + 16));
    cudaError_t e = cudaMemcpyAsync(tmp, host, m->nparams * 4, cudaMemcpyHostToDevice, m->stream);
    if (e == cudaSuccess) {
        launch_from_f32(m->dt, m->grads, tmp, m->nparams, m->stream);
        e = cudaStreamSynchronize(m->stream);
    }
    cudaFree(tmp);
    if (e != cudaSuccess) return fail(GPT2_ERR_CUDA, "set_grads: %s", cudaGetErrorString(e));
    return GPT2_OK;
}

int gpt2_get_losses(float* host) {
    TRY(check_model());
    if (!host) return fail(GPT2_ERR_ARG, "host is NULL");
    if (!g->acts) return fail(GPT2_ERR_STATE, "no forward yet");
    CUDA_TRY(cudaMemcpyAsync(host, g->losses, (size_t)g->B * g->T * 4, cudaMemcpyDeviceToHost, g->stream));
    CUDA_TRY(cudaStreamSynchronize(g->stream));
    return GPT2_OK;
}

int gpt2_get_activation(int which, int layer, float* host, size_t* n_out) {
    TRY(check_model());
    Model* m = g;
    if (!m->acts) return fail(GPT2_ERR_STATE, "no forward yet");
    const size_t BT = (size_t)m->B * m->T, C = m->C, es = m->esz;
    if (layer < 0 || (m->L > 0 && layer >= m->L)) layer = 0;
    const void* src = nullptr;
    size_t n = 0;
    DType dt = m->dt;
    switch (which) {
        case GPT2_ACT_ENCODED: src = m->encoded; n = BT * C; break;
        case GPT2_ACT_LN1: n = BT * C; src = (char*)m->ln1 + layer * n * es; break;
        case GPT2_ACT_QKV: n = BT * 3 * C; src = (char*)m->qkv + layer * n * es; break;
        case GPT2_ACT_ATTY: n = BT * C; src = (char*)m->atty + layer * n * es; break;
        case GPT2_ACT_RESIDUAL2: n = BT * C; src = (char*)m->residual2 + layer * n * es; break;
        case GPT2_ACT_LN2: n = BT * C; src = (char*)m->ln2 + layer * n * es; break;
        case GPT2_ACT_FCH: n = BT * 4 * C; src = (char*)m->fch + layer * n * es; break;
        case GPT2_ACT_FCH_GELU: n = BT * 4 * C; src = (char*)m->fch_gelu + layer * n * es; break;
        case GPT2_ACT_RESIDUAL3: n = BT * C; src = (char*)m->residual3 + layer * n * es; break;
        case GPT2_ACT_LNF: src = m->lnf; n = BT * C; break;
        case GPT2_ACT_LOGITS: src = m->logits; n = BT * m->Vp; break;
        case GPT2_ACT_LSE: n = (size_t)m->B * m->NH * m->T; src = m->lse + layer * n; dt = DT_F32; break;
        case GPT2_ACT_PROBS: n = BT * m->Vp; break;
        default: return fail(GPT2_ERR_ARG, "unknown activation %d", which);
    }
    if (n_out) *n_out = n;
    if (!host) return GPT2_OK;
    if (which == GPT2_ACT_PROBS) {
        if (m->fwd_targets || !m->fwd_done)
            return fail(GPT2_ERR_STATE, "probabilities need a preceding forward without targets");
        float* tmp = nullptr;
        CUDA_TRY(cudaMalloc(&tmp, n * 4 + 16));
        launch_probs(m->dt, tmp, m->logits, (int)BT, m->V, m->Vp, m->stream);
        cudaError_t e = cudaMemcpyAsync(host, tmp, n * 4, cudaMemcpyDeviceToHost, m->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(m->stream);
        cudaFree(tmp);
        if (e != cudaSuccess) return fail(GPT2_ERR_CUDA, "probs: %s", cudaGetErrorString(e));
        return GPT2_OK;
    }
    if (m->L == 0 && (which >= GPT2_ACT_LN1 && which <= GPT2_ACT_RESIDUAL3))
        return fail(GPT2_ERR_ARG, "no layers");
    return to_host_f32(m, host, src, n, dt);
}

int gpt2_sample(int t, const float* coins, int* out) {
    TRY(check_model());
    Model* m = g;
    if (!coins || !out) return fail(GPT2_ERR_ARG, "coins and out are required");
    if (!m->acts || !m->fwd_done || m->fwd_targets)
        return fail(GPT2_ERR_STATE, "sampling needs a preceding forward without targets");
    if (t < 0 || t >= m->T) return fail(GPT2_ERR_ARG, "position t=%d outside [0, %d)", t, m->T);
    const int B = m->B;
    for (int b = 0; b < B; b++)
        if (!(coins[b] >= 0.f && coins[b] < 1.f)) return fail(GPT2_ERR_ARG, "coin %d outside [0, 1)", b);
    CUDA_TRY(cudaMemcpyAsync(m->coins, coins, (size_t)B * 4, cudaMemcpyHostToDevice, m->stream));
    launch_sample(m->dt, (const char*)m->logits + (size_t)t * m->Vp * m->esz, (long long)m->T * m->Vp, B,
                  m->V, m->coins, m->sampled, 1, m->stream);
    CUDA_TRY(cudaMemcpyAsync(out, m->sampled, (size_t)B * 4, cudaMemcpyDeviceToHost, m->stream));
    CUDA_TRY(cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

int gpt2_generate(int* tokens, int B, int T, int t_begin, int t_end, unsigned long long* rng_state) {
    TRY(check_model());
    Model* m = g;
    if (!tokens || !rng_state) return fail(GPT2_ERR_ARG, "tokens and rng_state are required");
    TRY(check_shape(m, B, T));
    if (t_begin < 1 || t_end > T || t_begin > t_end)
        return fail(GPT2_ERR_ARG, "positions [%d, %d) must lie in [1, T=%d]", t_begin, t_end, T);
    const size_t n = (size_t)B * T;
    for (size_t i = 0; i < n; i++)
        if (tokens[i] < 0 || tokens[i] >= m->V)
            return fail(GPT2_ERR_TOKEN, "id at position %zu outside [0, %d)", i, m->V);
    // every coin up front, in the order the loop draws them (t, then b)
    std::vector<float> coins((size_t)(t_end - t_begin) * B);
    unsigned long long st = *rng_state;
    for (float& c : coins) c = (float)(random_u32(&st) >> 8) / 16777216.0f;
    CUDA_TRY(cudaMemcpyAsync(m->tokens, tokens, n * 4, cudaMemcpyHostToDevice, m->stream));
    if (!coins.empty())
        CUDA_TRY(cudaMemcpyAsync(m->coins, coins.data(), coins.size() * 4, cudaMemcpyHostToDevice, m->stream));
    for (int t = t_begin; t < t_end; t++) {
        TRY(run_forward(m, false));
        // the distribution at position t-1 gives the token at position t
        launch_sample(m->dt, (const char*)m->logits + (size_t)(t - 1) * m->Vp * m->esz,
                      (long long)T * m->Vp, B, m->V, m->coins + (size_t)(t - t_begin) * B, m->tokens + t,
                      T, m->stream);
    }
    CUDA_TRY(cudaMemcpyAsync(tokens, m->tokens, n * 4, cudaMemcpyDeviceToHost, m->stream));
    CUDA_TRY(cudaStreamSynchronize(m->stream));
    TRY(read_err(m));
    *rng_state = st;
    m->fwd_done = 1;
    m->fwd_targets = 0;
    return GPT2_OK;
}

int gpt2_free(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g) {
        free_model(g);
        g = nullptr;
    }
    return GPT2_OK;
}

int gpt2_timing_begin(int max_launches) {
    TRY(check_model());
    Timing& t = g->timing;
    if (max_launches < 1) return fail(GPT2_ERR_ARG, "max_launches must be >= 1");
    while ((int)t.ev.size() < 2 * max_launches) {
        cudaEvent_t e;
        CUDA_TRY(cudaEventCreate(&e));
        t.ev.push_back(e);
    }
    t.cap = max_launches;
    t.fam.assign(max_launches, 0);
    t.work.assign(max_launches, 0.0);
    t.n = 0;
    for (int f = 0; f < FAM_COUNT; f++) {
        t.ms[f] = 0;
        t.launches[f] = 0;
        t.works[f] = 0;
    }
    t.on = true;
    return GPT2_OK;
}

int gpt2_timing_end(void) {
    TRY(check_model());
    Timing& t = g->timing;
    t.on = false;
    CUDA_TRY(cudaStreamSynchronize(g->stream));
    for (int i = 0; i < t.n; i++) {
        float ms = 0.f;
        CUDA_TRY(cudaEventElapsedTime(&ms, t.ev[2 * i], t.ev[2 * i + 1]));
        t.ms[t.fam[i]] += ms;
        t.launches[t.fam[i]] += 1;
        t.works[t.fam[i]] += t.work[i];
    }
    return GPT2_OK;
}

int gpt2_timing_get(int family, double* total_ms, long long* launches, double* work) {
    TRY(check_model());
    if (family < 0 || family >= FAM_COUNT) return fail(GPT2_ERR_ARG, "family %d", family);
    const Timing& t = g->timing;
    if (total_ms) *total_ms = t.ms[family];
    if (launches) *launches = t.launches[family];
    if (work) *work = t.works[family];
    return GPT2_OK;
}

}  // extern "C"
