// ppo.cu -- the on-device PPO update (include/ppo.h): per mini-batch, the
// actor's log-probabilities are recomputed, the clipped surrogate and the
// critic's squared error are formed and backpropagated, the gradient is
// clipped to a global L2 norm and one Adam step updates actor and critic.
//
// Page "PPO CUDA Pipeline Design -- Zero-Roundtrip Experience Collection",
// the training flow after the collector; page "Fused CUDA Training Kernel --
// Implementation Plan", "Chunk 3: Adam Optimizer Kernel" (norm, clip scale,
// Adam with bias correction and decoupled weight decay).
//
// Parameters, gradients and moments are float32, in the packed weight layout
// (actor, then critic; the curiosity part is carried along untrained).  Each
// dense layer's forward, weight-gradient and input-gradient products run on
// the tensor cores (ppo_gemm.cu: tcgen05 MMAs on a bf16 high/low split of the
// float32 operands, float32-grade products), with the bias and ReLU fused into
// the forward product, the bias gradient into the weight-gradient product (a
// row of ones appended to the layer input) and the ReLU derivative into the
// input-gradient product.  Each product also writes the transposed copy that
// the next product reads as its K-contiguous operand; the weights' transposes
// are refreshed after every Adam step.  The gather, the loss heads, the norm
// and Adam are the kernels below.  Every reduction runs in a fixed order (the
// tensor core's per tile, per block, then over the blocks), so a step's result
// does not depend on timing.  One optimizer step is captured as a CUDA graph
// (34 launches) and replayed for every step of a call: the step's mini-batch
// slice, statistics slot and Adam step count are read from device counters
// that a last 1-thread kernel advances, so that the same graph serves every
// step.
#include <math.h>
#include <string.h>

#include <new>

#include "../../include/ppo.h"
#include "internal.cuh"
#include "pdl.cuh"
#include "ppo_gemm.cuh"

using namespace rl;

namespace {

constexpr int kMaxLayers = 6;
constexpr int kMaxBatch = 4096;
constexpr int kMaxWidth = 1024;
constexpr int kNormBlocks = 304;   // fixed, so that the norm's summation order is fixed
constexpr int kNormThreads = 256;

constexpr int kGraphMinSteps = 4;              // calls with fewer steps launch directly

struct Net {
    int n = 0;
    size_t w[kMaxLayers] = {}, b[kMaxLayers] = {};
    int in[kMaxLayers] = {}, out[kMaxLayers] = {};
};

// what a captured step depends on besides the trainer's own buffers
struct GraphKey {
    const void *ptr[7] = {};           // states, actions, logp_old, adv, ret, indices, stats
    long long T = 0;
    int batch = 0;
    ppo_hparams hp{};
    bool operator==(const GraphKey &o) const
    {
        for (int i = 0; i < 7; ++i)
            if (ptr[i] != o.ptr[i]) return false;
        return T == o.T && batch == o.batch && memcmp(&hp, &o.hp, sizeof hp) == 0;
    }
};

}  // namespace

struct ppo_trainer {
    int device = 0;
    Net net[2];                        // 0 actor, 1 critic
    size_t n_weights = 0, n_trained = 0;
    float *d_w = nullptr, *d_g = nullptr, *d_m = nullptr, *d_v = nullptr;
    long long step = 0;
    // mini-batch buffers, `cap` rows
    int cap = 0;
    float *d_x = nullptr;              // [cap, 54]
    int32_t *d_a = nullptr;
    float *d_lpo = nullptr, *d_adv = nullptr, *d_ret = nullptr;
    float *d_xt = nullptr;             // [kState + 1, cap]: x^T and a row of ones
    float *d_act[2][kMaxLayers] = {};  // layer outputs [cap, out]
    float *d_actt[2][kMaxLayers] = {}; // their transposes [out + 1, cap], the last row ones
    float *d_dy[2][2] = {};            // per net, backpropagated gradients (ping-pong) [cap, kMaxWidth]
    float *d_dyt[2][2] = {};           // their transposes [kMaxWidth, cap]
    float *d_ws = nullptr;             // split-K partial tiles of the products of one stage
    unsigned int *d_cnt = nullptr;     // their per-tile arrival counters (zero between launches)
    long long ws_floats = 0;
    int n_cnt = 0;
    float *d_wt = nullptr;             // transposed weights: layer l's [in, out] at its offset
    float *d_rows = nullptr;           // per-row statistics [4][cap]
    double *d_part = nullptr;          // [kNormBlocks] partial sums of g^2
    int *d_status = nullptr;
    int *d_k = nullptr;                // step index within the current call
    long long *d_t = nullptr;          // Adam step count
    cudaStream_t last_stream = nullptr;
    int last_batch = 0;                // rows of the last forward pass (ppo_test_activations)
    cudaStream_t cap_stream = nullptr; // where one step is captured
    cudaGraphExec_t exec = nullptr;
    GraphKey key;
};

namespace {

int cuda_err(cudaError_t e, const char *what)
{
    return set_error(e == cudaErrorMemoryAllocation ? ROLLOUT_ERR_NOMEM : ROLLOUT_ERR_CUDA, "%s: %s", what,
                     cudaGetErrorString(e));
}


// ------------------------------------------------------------------ kernels

// one block per mini-batch row: copy the tuple the index names
__global__ void gather_kernel(const float *states, const int32_t *actions, const float *logp_old,
                              const float *adv, const float *ret, long long T, const int32_t *idx_base,
                              const int *step_k, float *x, float *xt, int ldt, int32_t *a, float *lpo, float *A,
                              float *R, int *status)
{
    const int r = blockIdx.x;
    long long i = idx_base[(size_t)*step_k * gridDim.x + r];
    if (i < 0 || i >= T) {
        if (threadIdx.x == 0) atomicCAS(status, 0, ROLLOUT_ERR_RANGE);
        i = 0;
    }
    for (int c = threadIdx.x; c < kState; c += blockDim.x) {
        const float v = states[i * kState + c];
        x[(size_t)r * kState + c] = v;
        xt[(size_t)c * ldt + r] = v;
    }
    if (threadIdx.x == 0) {
        int act = actions[i];
        if (act < 0 || act >= kActions) {
            atomicCAS(status, 0, ROLLOUT_ERR_RANGE);
            act = 0;
        }
        a[r] = act;
        lpo[r] = logp_old[i];
        A[r] = adv[i];
        R[r] = ret[i];
    }
}

// one warp per row: log-softmax of the taken action, ratio, clipped surrogate,
// and the gradient of the loss with respect to the logits
__global__ void actor_head_kernel(const float *logits, const int32_t *a, const float *lpo, const float *A, int B,
                                  float clip_eps, float *dl, float *dlt, int ldt, float *rows)
{
    pdl_wait();
    const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (w >= B) return;
    const float *l = logits + (size_t)w * kActions;
    const float l0 = l[lane], l1 = lane + 32 < kActions ? l[lane + 32] : -INFINITY;
    float m = fmaxf(l0, l1);
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float e0 = expf(l0 - m), e1 = lane + 32 < kActions ? expf(l1 - m) : 0.f;
    float z = e0 + e1;
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const int act = a[w];
    const float la = l[act];
    const float logp = (la - m) - logf(z);
    const float rho = expf(logp - lpo[w]);
    const float adv = A[w];
    const float rc = fminf(fmaxf(rho, 1.f - clip_eps), 1.f + clip_eps);
    const float s1 = rho * adv, s2 = rc * adv;
    const bool unclipped = s1 <= s2;
    const float glp = unclipped ? -adv * rho / (float)B : 0.f;
    float *d = dl + (size_t)w * kActions;
    const float g0 = glp * ((lane == act ? 1.f : 0.f) - e0 / z);
    d[lane] = g0;
    dlt[(size_t)lane * ldt + w] = g0;
    if (lane + 32 < kActions) {
        const float g1 = glp * ((lane + 32 == act ? 1.f : 0.f) - e1 / z);
        d[lane + 32] = g1;
        dlt[(size_t)(lane + 32) * ldt + w] = g1;
    }
    if (lane == 0) {
        rows[0 * B + w] = -(unclipped ? s1 : s2);
        rows[2 * B + w] = unclipped ? 0.f : 1.f;
        rows[3 * B + w] = rho;
    }
}

// critic head: squared error and its gradient with respect to v
__global__ void critic_head_kernel(const float *v, const float *R, int B, float value_coef, float *dv, float *dvt,
                                   float *rows)
{
    pdl_wait();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= B) return;
    const float d = v[r] - R[r];
    rows[1 * B + r] = d * d;
    const float g = 2.f * value_coef * d / (float)B;
    dv[r] = g;
    dvt[r] = g;                                  // [1, B]: the same values
}

__device__ __forceinline__ double block_sum(double v, double *sh)
{
    sh[threadIdx.x] = v;
    __syncthreads();
    for (int s = blockDim.x / 2; s > 0; s >>= 1) {
        if ((int)threadIdx.x < s) sh[threadIdx.x] += sh[threadIdx.x + s];
        __syncthreads();
    }
    const double r = sh[0];
    __syncthreads();
    return r;
}

// partial sums of g^2 over a fixed partition (kNormBlocks blocks)
__global__ void __launch_bounds__(kNormThreads) norm_partial_kernel(const float *g, size_t n, double *part)
{
    pdl_wait();
    __shared__ double sh[kNormThreads];
    double s = 0.0;
    for (size_t i = blockIdx.x * (size_t)kNormThreads + threadIdx.x; i < n; i += (size_t)kNormBlocks * kNormThreads)
        s += (double)g[i] * (double)g[i];
    s = block_sum(s, sh);
    if (threadIdx.x == 0) part[blockIdx.x] = s;
}

// every block first sums the partials in the same order (so all see the same
// norm), then updates its share of the parameters
__global__ void __launch_bounds__(kNormThreads) adam_kernel(float *p, const float *g, float *m, float *v, size_t n,
                                                             const double *part, ppo_hparams hp, const long long *step_t,
                                                             const int *step_k, float *stats)
{
    pdl_wait();
    __shared__ float sh_scale, sh_bc1, sh_bc2;
    __shared__ double sh[kNormThreads];
    // every block adds the partials in the same fixed order (a strided
    // per-thread sum, then the tree of block_sum), so all see the same norm
    double ps = 0.0;
    for (int b = threadIdx.x; b < kNormBlocks; b += kNormThreads) ps += part[b];
    const double ss = block_sum(ps, sh);
    if (threadIdx.x == 0) {
        const double t = (double)(*step_t + 1);
        sh_bc1 = (float)(1.0 - pow((double)hp.beta1, t));
        sh_bc2 = (float)(1.0 - pow((double)hp.beta2, t));
        float *norm_out = stats ? stats + (size_t)*step_k * 5 + 4 : nullptr;
        const double norm = sqrt(ss);
        double scale = 1.0;
        if (hp.max_grad_norm > 0.f) scale = fmin(1.0, (double)hp.max_grad_norm / (norm + 1e-6));
        sh_scale = (float)scale;
        if (blockIdx.x == 0 && norm_out) *norm_out = (float)norm;
    }
    __syncthreads();
    const float scale = sh_scale, bc1 = sh_bc1, bc2 = sh_bc2;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const float gi = g[i] * scale;
        const float mi = hp.beta1 * m[i] + (1.f - hp.beta1) * gi;
        const float vi = hp.beta2 * v[i] + (1.f - hp.beta2) * gi * gi;
        m[i] = mi;
        v[i] = vi;
        const float pi = p[i];
        p[i] = pi - (hp.lr * (mi / bc1) / (sqrtf(vi / bc2) + hp.adam_eps) + hp.weight_decay * pi);
    }
}

// means of the four per-row statistics, in row order, into slot step_k of stats
__global__ void stats_kernel(const float *rows, int B, float *stats, const int *step_k)
{
    pdl_wait();
    __shared__ double sh[256];
    float *out = stats + (size_t)*step_k * 5;
    for (int k = 0; k < 4; ++k) {
        double s = 0.0;
        for (int r = threadIdx.x; r < B; r += blockDim.x) s += (double)rows[k * B + r];
        s = block_sum(s, sh);
        if (threadIdx.x == 0) out[k] = (float)(s / B);
    }
}

// WT[l] = W[l]^T for every dense layer (layer l's [in, out] transpose at the
// offset of its [out, in] weights)
struct LayerTable {
    int n;
    long long off[2 * kMaxLayers];
    int in[2 * kMaxLayers], out[2 * kMaxLayers];
};

__global__ void transpose_weights_kernel(const float *w, float *wt, LayerTable lt)
{
    pdl_wait();
    for (int l = 0; l < lt.n; ++l) {
        const long long n = (long long)lt.in[l] * lt.out[l];
        const float *src = w + lt.off[l];
        float *dst = wt + lt.off[l];
        for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n;
             e += (long long)gridDim.x * blockDim.x) {
            const long long o = e / lt.in[l], j = e - o * lt.in[l];
            dst[j * lt.out[l] + o] = src[e];
        }
    }
}

// row `row` of a [rows, ld] buffer set to 1 (the ones row of a transposed input)
__global__ void ones_row_kernel(float *buf, int row, int ld)
{
    for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < ld; c += gridDim.x * blockDim.x)
        buf[(size_t)row * ld + c] = 1.f;
}

// the end of a step: the next step's slice and Adam count
__global__ void advance_kernel(int *step_k, long long *step_t)
{
    pdl_wait();
    *step_k += 1;
    *step_t += 1;
}

// ------------------------------------------------------------------ host side

void free_batch(ppo_trainer *t)
{
    cudaFree(t->d_x);
    cudaFree(t->d_xt);
    t->d_xt = nullptr;
    for (auto &net : t->d_actt)
        for (float *&p : net) {
            cudaFree(p);
            p = nullptr;
        }
    for (int k = 0; k < 2; ++k)
        for (int i = 0; i < 2; ++i) {
            cudaFree(t->d_dy[k][i]);
            cudaFree(t->d_dyt[k][i]);
            t->d_dy[k][i] = t->d_dyt[k][i] = nullptr;
        }
    cudaFree(t->d_ws);
    cudaFree(t->d_cnt);
    t->d_ws = nullptr;
    t->d_cnt = nullptr;
    cudaFree(t->d_a);
    cudaFree(t->d_lpo);
    cudaFree(t->d_adv);
    cudaFree(t->d_ret);
    for (auto &net : t->d_act)
        for (float *&p : net) {
            cudaFree(p);
            p = nullptr;
        }
    cudaFree(t->d_rows);
    t->d_x = nullptr;
    t->d_a = nullptr;
    t->d_lpo = t->d_adv = t->d_ret = t->d_rows = nullptr;
    t->cap = 0;
}

void plan_workspace(ppo_trainer *t, int B);

int ensure_batch(ppo_trainer *t, int B)
{
    if (B <= t->cap) return ROLLOUT_OK;
    if (t->exec) {   // the captured step names the old buffers
        cudaGraphExecDestroy(t->exec);
        t->exec = nullptr;
    }
    free_batch(t);   // cudaFree waits for work that may still use the old buffers
    cudaError_t e;
#define ALLOC(p, bytes) if ((e = cudaMalloc(&(p), (bytes))) != cudaSuccess) { free_batch(t); return cuda_err(e, "cudaMalloc(mini-batch)"); }
    ALLOC(t->d_x, (size_t)B * kState * 4);
    ALLOC(t->d_a, (size_t)B * 4);
    ALLOC(t->d_lpo, (size_t)B * 4);
    ALLOC(t->d_adv, (size_t)B * 4);
    ALLOC(t->d_ret, (size_t)B * 4);
    ALLOC(t->d_xt, (size_t)(kState + 1) * B * 4);
    for (int k = 0; k < 2; ++k)
        for (int l = 0; l < t->net[k].n; ++l) {
            ALLOC(t->d_act[k][l], (size_t)B * t->net[k].out[l] * 4);
            ALLOC(t->d_actt[k][l], (size_t)(t->net[k].out[l] + 1) * B * 4);
        }
    for (int k = 0; k < 2; ++k)
        for (int i = 0; i < 2; ++i) {
            ALLOC(t->d_dy[k][i], (size_t)B * kMaxWidth * 4);
            ALLOC(t->d_dyt[k][i], (size_t)B * kMaxWidth * 4);
        }
    ALLOC(t->d_rows, (size_t)4 * B * 4);
    t->cap = B;
    plan_workspace(t, B);
    ALLOC(t->d_ws, (size_t)(t->ws_floats > 0 ? t->ws_floats : 4) * 4);
    ALLOC(t->d_cnt, (size_t)(t->n_cnt > 0 ? t->n_cnt : 1) * 4);
#undef ALLOC
    if ((e = cudaMemset(t->d_cnt, 0, (size_t)(t->n_cnt > 0 ? t->n_cnt : 1) * 4)) != cudaSuccess) {
        free_batch(t);
        return cuda_err(e, "cudaMemset(counters)");
    }
    // the ones rows of the transposed layer inputs (their bias-gradient column)
    ones_row_kernel<<<1, 256>>>(t->d_xt, kState, B);
    for (int k = 0; k < 2; ++k)
        for (int l = 0; l < t->net[k].n; ++l) ones_row_kernel<<<1, 256>>>(t->d_actt[k][l], t->net[k].out[l], B);
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) {
        free_batch(t);
        return cuda_err(e, "mini-batch set-up");
    }
    return ROLLOUT_OK;
}

void free_trainer(ppo_trainer *t)
{
    if (!t) return;
    free_batch(t);
    cudaFree(t->d_w);
    cudaFree(t->d_g);
    cudaFree(t->d_m);
    cudaFree(t->d_v);
    cudaFree(t->d_part);
    cudaFree(t->d_status);
    cudaFree(t->d_k);
    cudaFree(t->d_t);
    cudaFree(t->d_wt);
    if (t->exec) cudaGraphExecDestroy(t->exec);
    if (t->cap_stream) cudaStreamDestroy(t->cap_stream);
    delete t;
}

constexpr int kMaxSplit = 4;        // CTAs a product's K may be split over
constexpr int kStages = 2 * kMaxLayers;

// the forward product of net k's layer l over B rows
GemmArgs fwd_args(ppo_trainer *t, int k, int l, int B)
{
    const Net &n = t->net[k];
    GemmArgs g;
    g.A = l == 0 ? t->d_x : t->d_act[k][l - 1];
    g.lda = n.in[l];
    g.B = t->d_w + n.w[l];                           // [out, in]
    g.ldb = n.in[l];
    g.M = B;
    g.N = n.out[l];
    g.K = n.in[l];
    g.epi = kGemmFwd;
    g.bias = t->d_w + n.b[l];
    g.relu = l < n.n - 1;
    g.Y = t->d_act[k][l];
    g.ldy = n.out[l];
    g.YT = l < n.n - 1 ? t->d_actt[k][l] : nullptr;
    g.ldt = t->cap;
    g.status = t->d_status;
    return g;
}

// the weight- and bias-gradient product dY^T [X | 1] of net k's layer l; dY^T
// is d_dyt[k][p]
GemmArgs dw_args(ppo_trainer *t, int k, int l, int p, int B)
{
    const Net &n = t->net[k];
    GemmArgs g;
    g.A = t->d_dyt[k][p];                            // [out, B]
    g.lda = t->cap;
    g.B = l == 0 ? t->d_xt : t->d_actt[k][l - 1];    // [in + 1, B], the last row ones
    g.ldb = t->cap;
    g.M = n.out[l];
    g.N = n.in[l] + 1;
    g.K = B;
    g.epi = kGemmDw;
    g.Y = t->d_g + n.w[l];
    g.ldy = n.in[l];
    g.nw = n.in[l];
    g.db = t->d_g + n.b[l];
    g.status = t->d_status;
    return g;
}

// the input-gradient product dY W masked by ReLU' of net k's layer l (l > 0):
// dY = d_dy[k][p], the result into d_dy[k][1 - p] and its transpose
GemmArgs dx_args(ppo_trainer *t, int k, int l, int p, int B)
{
    const Net &n = t->net[k];
    GemmArgs x;
    x.A = t->d_dy[k][p];                             // [B, out]
    x.lda = n.out[l];
    x.B = t->d_wt + n.w[l];                          // W^T [in, out]
    x.ldb = n.out[l];
    x.M = B;
    x.N = n.in[l];
    x.K = n.out[l];
    x.epi = kGemmDx;
    x.H = t->d_act[k][l - 1];
    x.ldh = n.in[l];
    x.Y = t->d_dy[k][1 - p];
    x.ldy = n.in[l];
    x.YT = t->d_dyt[k][1 - p];
    x.ldt = t->cap;
    x.status = t->d_status;
    return x;
}

// the products of stage j of a step, all independent of one another:
// j < kMaxLayers: the forward products of depth j of both nets; after that the
// backward products of depth j - kMaxLayers from the top of each net (its
// weight gradient and, below the first layer, its input gradient)
int stage_products(ppo_trainer *t, int j, int B, GemmArgs *g)
{
    int n = 0;
    for (int k = 0; k < 2; ++k) {
        const int L = t->net[k].n;
        if (j < kMaxLayers) {
            if (j < L) g[n++] = fwd_args(t, k, j, B);
        } else {
            const int d = j - kMaxLayers, l = L - 1 - d;
            if (l < 0) continue;
            g[n++] = dw_args(t, k, l, d & 1, B);
            if (l > 0) g[n++] = dx_args(t, k, l, d & 1, B);
        }
    }
    return n;
}

// split-K plans of a stage's products and their workspace regions (ws / cnt
// may be null when only the sizes are wanted)
void plan_stage(GemmArgs *g, int n, float *ws, unsigned int *cnt, long long *ws_floats, int *n_cnt)
{
    long long wo = 0;
    int co = 0;
    for (int i = 0; i < n; ++i) {
        long long wf;
        int c;
        gemm_plan(g[i], kMaxSplit, &wf, &c);
        g[i].ws = ws ? ws + wo : nullptr;
        g[i].cnt = cnt ? cnt + co : nullptr;
        wo += wf;
        co += c;
    }
    *ws_floats = wo;
    *n_cnt = co;
}

void plan_workspace(ppo_trainer *t, int B)
{
    t->ws_floats = 0;
    t->n_cnt = 0;
    for (int j = 0; j < kStages; ++j) {
        GemmArgs g[kGemmGroup];
        const int n = stage_products(t, j, B, g);
        if (n == 0) continue;
        long long wf;
        int c;
        plan_stage(g, n, nullptr, nullptr, &wf, &c);
        if (wf > t->ws_floats) t->ws_floats = wf;
        if (c > t->n_cnt) t->n_cnt = c;
    }
}

int run_stage(ppo_trainer *t, int j, int B, cudaStream_t s)
{
    GemmArgs g[kGemmGroup];
    const int n = stage_products(t, j, B, g);
    if (n == 0) return ROLLOUT_OK;
    long long wf;
    int c;
    plan_stage(g, n, t->d_ws, t->d_cnt, &wf, &c);
    cudaError_t e = launch_gemm_group(g, n, s);
    return e == cudaSuccess ? ROLLOUT_OK : cuda_err(e, "tensor-core product");
}

LayerTable layer_table(const ppo_trainer *t)
{
    LayerTable lt{};
    for (int k = 0; k < 2; ++k)
        for (int l = 0; l < t->net[k].n; ++l) {
            lt.off[lt.n] = (long long)t->net[k].w[l];
            lt.in[lt.n] = t->net[k].in[l];
            lt.out[lt.n] = t->net[k].out[l];
            ++lt.n;
        }
    return lt;
}

int check_update_args(ppo_trainer *t, const float *states, const int32_t *actions, const float *logp_old,
                      const float *adv, const float *ret, long long T, const int32_t *indices, int batch,
                      const ppo_hparams *hp)
{
    if (!t || !hp) return set_error(ROLLOUT_ERR_INVALID, "null argument");
    if (!states || !actions || !logp_old || !adv || !ret || !indices)
        return set_error(ROLLOUT_ERR_INVALID, "null array argument");
    if (T < 1 || T > (1LL << 31) - 1) return set_error(ROLLOUT_ERR_INVALID, "T must be in [1, 2^31)");
    if (batch < 1 || batch > kMaxBatch) return set_error(ROLLOUT_ERR_INVALID, "batch must be in [1, %d]", kMaxBatch);
    const float hv[] = {hp->clip_eps, hp->value_coef, hp->lr, hp->beta1, hp->beta2, hp->adam_eps, hp->max_grad_norm,
                        hp->weight_decay};
    for (float f : hv)
        if (!isfinite(f)) return set_error(ROLLOUT_ERR_INVALID, "hyperparameters must be finite");
    if (hp->clip_eps < 0.f || hp->lr < 0.f || hp->adam_eps <= 0.f || !(hp->beta1 >= 0.f && hp->beta1 < 1.f) ||
        !(hp->beta2 >= 0.f && hp->beta2 < 1.f))
        return set_error(ROLLOUT_ERR_INVALID, "need clip_eps >= 0, lr >= 0, adam_eps > 0, beta1 and beta2 in [0, 1)");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_err(e, "cudaGetDevice");
    if (dev != t->device) return set_error(ROLLOUT_ERR_INVALID, "current device is not the trainer's");
    return ensure_batch(t, batch);
}

// the loss statistics (per row, in d_rows) and the gradient (d_g) of the
// mini-batch rows[d_k * B .. d_k * B + B) at the current weights
int loss_gradient(ppo_trainer *t, const float *states, const int32_t *actions, const float *logp_old,
                  const float *adv, const float *ret, long long T, const int32_t *rows, int B, const ppo_hparams *hp,
                  cudaStream_t s)
{
    int rc;
    t->last_batch = B;
    gather_kernel<<<B, 64, 0, s>>>(states, actions, logp_old, adv, ret, T, rows, t->d_k, t->d_x, t->d_xt, t->cap,
                                   t->d_a, t->d_lpo, t->d_adv, t->d_ret, t->d_status);
    // forward products of both nets, depth by depth
    for (int j = 0; j < kMaxLayers; ++j)
        if ((rc = run_stage(t, j, B, s))) return rc;
    // the two loss heads: the actor's surrogate and the critic's squared error,
    // each with its gradient at the net's output (and that gradient's transpose)
    cudaError_t e = launch_dependent(actor_head_kernel, dim3((B * 32 + 255) / 256), dim3(256), 0, s,
                                     (const float *)t->d_act[0][2], (const int32_t *)t->d_a, (const float *)t->d_lpo,
                                     (const float *)t->d_adv, B, hp->clip_eps, t->d_dy[0][0], t->d_dyt[0][0], t->cap,
                                     t->d_rows);
    if (e == cudaSuccess)
        e = launch_dependent(critic_head_kernel, dim3((B + 255) / 256), dim3(256), 0, s,
                             (const float *)t->d_act[1][kCriticLayers - 1], (const float *)t->d_ret, B,
                             hp->value_coef, t->d_dy[1][0], t->d_dyt[1][0], t->d_rows);
    if (e != cudaSuccess) return cuda_err(e, "PPO loss-head launch");
    // backward products of both nets, depth by depth from the top
    for (int j = kMaxLayers; j < kStages; ++j)
        if ((rc = run_stage(t, j, B, s))) return rc;
    return ROLLOUT_OK;
}

// one optimizer step (the counters pick the mini-batch, the statistics slot and t)
int step(ppo_trainer *t, const float *states, const int32_t *actions, const float *logp_old, const float *adv,
         const float *ret, long long T, const int32_t *indices, int B, const ppo_hparams *hp, float *stats,
         cudaStream_t s)
{
    int rc = loss_gradient(t, states, actions, logp_old, adv, ret, T, indices, B, hp, s);
    if (rc) return rc;
    const dim3 nb(kNormBlocks), nt(kNormThreads);
    cudaError_t e = launch_dependent(norm_partial_kernel, nb, nt, 0, s, (const float *)t->d_g, t->n_trained, t->d_part);
    if (e == cudaSuccess)
        e = launch_dependent(adam_kernel, nb, nt, 0, s, t->d_w, (const float *)t->d_g, t->d_m, t->d_v, t->n_trained,
                             (const double *)t->d_part, *hp, (const long long *)t->d_t, (const int *)t->d_k, stats);
    if (e == cudaSuccess)
        e = launch_dependent(transpose_weights_kernel, nb, nt, 0, s, (const float *)t->d_w, t->d_wt, layer_table(t));
    if (e == cudaSuccess && stats)
        e = launch_dependent(stats_kernel, dim3(1), dim3(256), 0, s, (const float *)t->d_rows, B, stats,
                             (const int *)t->d_k);
    if (e == cudaSuccess) e = launch_dependent(advance_kernel, dim3(1), dim3(1), 0, s, t->d_k, t->d_t);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? ROLLOUT_OK : cuda_err(e, "PPO step launch");
}

// the graph of one step for these arguments (captured on the trainer's own
// stream; reused while the arguments stay the same)
int step_graph(ppo_trainer *t, const GraphKey &key, const float *states, const int32_t *actions,
               const float *logp_old, const float *adv, const float *ret, long long T, const int32_t *indices, int B,
               const ppo_hparams *hp, float *stats)
{
    if (t->exec && t->key == key) return ROLLOUT_OK;
    if (t->exec) {
        cudaGraphExecDestroy(t->exec);
        t->exec = nullptr;
    }
    cudaError_t e = cudaStreamBeginCapture(t->cap_stream, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_err(e, "cudaStreamBeginCapture");
    int rc = step(t, states, actions, logp_old, adv, ret, T, indices, B, hp, stats, t->cap_stream);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(t->cap_stream, &g);
    if (rc) {
        if (g) cudaGraphDestroy(g);
        return rc;
    }
    if (e != cudaSuccess) return cuda_err(e, "cudaStreamEndCapture");
    e = cudaGraphInstantiate(&t->exec, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) {
        t->exec = nullptr;
        return cuda_err(e, "cudaGraphInstantiate");
    }
    t->key = key;
    return ROLLOUT_OK;
}

}  // namespace

extern "C" {

int ppo_create(const float *weights, const rollout_dims *dims, ppo_trainer **out)
{
    clear_error();
    if (!weights || !dims || !out) return set_error(ROLLOUT_ERR_INVALID, "null argument");
    int rc = validate_dims(dims);
    if (rc) return rc;
    ppo_trainer *t = new (std::nothrow) ppo_trainer();
    if (!t) return set_error(ROLLOUT_ERR_NOMEM, "host allocation failed");
    // packed layout: actor (3 layers), critic (5 hidden + head), curiosity (2 layers)
    size_t off = 0;
    const int ain[3] = {kState, kActorH1, kActorH2}, aout[3] = {kActorH1, kActorH2, kActions};
    Net &A = t->net[0], &Cn = t->net[1];
    A.n = 3;
    for (int l = 0; l < 3; ++l) {
        A.in[l] = ain[l];
        A.out[l] = aout[l];
        A.w[l] = off; off += (size_t)ain[l] * aout[l];
        A.b[l] = off; off += aout[l];
    }
    Cn.n = kCriticLayers;
    int prev = kState;
    for (int l = 0; l < kCriticLayers; ++l) {
        const int o = l < 5 ? dims->critic_h[l] : 1;
        Cn.in[l] = prev;
        Cn.out[l] = o;
        Cn.w[l] = off; off += (size_t)prev * o;
        Cn.b[l] = off; off += o;
        prev = o;
    }
    t->n_trained = off;
    off += (size_t)(kState + kActions) * kCurH + kCurH + (size_t)kCurH * kState + kState;
    t->n_weights = off;
    cudaError_t e = cudaGetDevice(&t->device);
    if (e != cudaSuccess) { free_trainer(t); return cuda_err(e, "cudaGetDevice"); }
    if ((e = cudaMalloc(&t->d_w, t->n_weights * 4)) != cudaSuccess ||
        (e = cudaMalloc(&t->d_g, t->n_trained * 4)) != cudaSuccess ||
        (e = cudaMalloc(&t->d_m, t->n_trained * 4)) != cudaSuccess ||
        (e = cudaMalloc(&t->d_v, t->n_trained * 4)) != cudaSuccess ||
        (e = cudaMalloc(&t->d_part, kNormBlocks * sizeof(double))) != cudaSuccess ||
        (e = cudaMalloc(&t->d_status, sizeof(int))) != cudaSuccess ||
        (e = cudaMalloc(&t->d_k, sizeof(int))) != cudaSuccess ||
        (e = cudaMalloc(&t->d_t, sizeof(long long))) != cudaSuccess ||
        (e = cudaMalloc(&t->d_wt, t->n_trained * 4)) != cudaSuccess) {
        free_trainer(t);
        return cuda_err(e, "cudaMalloc(trainer)");
    }
    if ((e = cudaStreamCreateWithFlags(&t->cap_stream, cudaStreamNonBlocking)) != cudaSuccess) {
        free_trainer(t);
        return cuda_err(e, "cudaStreamCreateWithFlags");
    }
    if ((e = cudaMemcpy(t->d_w, weights, t->n_weights * 4, cudaMemcpyHostToDevice)) != cudaSuccess ||
        (e = cudaMemset(t->d_m, 0, t->n_trained * 4)) != cudaSuccess ||
        (e = cudaMemset(t->d_v, 0, t->n_trained * 4)) != cudaSuccess ||
        (e = cudaMemset(t->d_status, 0, sizeof(int))) != cudaSuccess ||
        (e = cudaMemset(t->d_k, 0, sizeof(int))) != cudaSuccess ||
        (e = cudaMemset(t->d_t, 0, sizeof(long long))) != cudaSuccess) {
        free_trainer(t);
        return cuda_err(e, "trainer upload");
    }
    transpose_weights_kernel<<<kNormBlocks, kNormThreads>>>(t->d_w, t->d_wt, layer_table(t));
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) {
        free_trainer(t);
        return cuda_err(e, "transposed weights");
    }
    *out = t;
    return ROLLOUT_OK;
}

int ppo_update(ppo_trainer *t, const float *states, const int32_t *actions, const float *logp_old,
               const float *adv, const float *ret, long long T, const int32_t *indices, int n_steps, int batch,
               const ppo_hparams *hp, float *stats, void *stream)
{
    clear_error();
    if (n_steps < 0) return set_error(ROLLOUT_ERR_INVALID, "n_steps must be >= 0");
    int rc = check_update_args(t, states, actions, logp_old, adv, ret, T, indices, batch, hp);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    t->last_stream = s;
    if (n_steps == 0) return ROLLOUT_OK;
    cudaError_t e = cudaMemsetAsync(t->d_k, 0, sizeof(int), s);
    if (e != cudaSuccess) return cuda_err(e, "cudaMemsetAsync(step index)");
    if (n_steps >= kGraphMinSteps) {
        GraphKey key;
        const void *ptrs[7] = {states, actions, logp_old, adv, ret, indices, stats};
        memcpy(key.ptr, ptrs, sizeof ptrs);
        key.T = T;
        key.batch = batch;
        key.hp = *hp;
        if ((rc = step_graph(t, key, states, actions, logp_old, adv, ret, T, indices, batch, hp, stats))) return rc;
        for (int k = 0; k < n_steps; ++k)
            if ((e = cudaGraphLaunch(t->exec, s)) != cudaSuccess) return cuda_err(e, "cudaGraphLaunch");
    } else {
        for (int k = 0; k < n_steps; ++k)
            if ((rc = step(t, states, actions, logp_old, adv, ret, T, indices, batch, hp, stats, s))) return rc;
    }
    t->step += n_steps;
    return ROLLOUT_OK;
}

int ppo_gradient(ppo_trainer *t, const float *states, const int32_t *actions, const float *logp_old,
                 const float *adv, const float *ret, long long T, const int32_t *indices, int batch,
                 const ppo_hparams *hp, float *grad, float *stats, void *stream)
{
    clear_error();
    if (!grad) return set_error(ROLLOUT_ERR_INVALID, "null gradient buffer");
    int rc = check_update_args(t, states, actions, logp_old, adv, ret, T, indices, batch, hp);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    t->last_stream = s;
    cudaError_t e = cudaMemsetAsync(t->d_k, 0, sizeof(int), s);
    if (e != cudaSuccess) return cuda_err(e, "cudaMemsetAsync(step index)");
    if ((rc = loss_gradient(t, states, actions, logp_old, adv, ret, T, indices, batch, hp, s))) return rc;
    if (stats) stats_kernel<<<1, 256, 0, s>>>(t->d_rows, batch, stats, t->d_k);
    e = cudaMemcpyAsync(grad, t->d_g, t->n_trained * 4, cudaMemcpyDefault, s);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? ROLLOUT_OK : cuda_err(e, "PPO gradient");
}

int ppo_test_activations(ppo_trainer *t, float *act, void *stream)
{
    clear_error();
    if (!t || !act) return set_error(ROLLOUT_ERR_INVALID, "null argument");
    const int B = t->last_batch;
    if (B <= 0) return set_error(ROLLOUT_ERR_INVALID, "no forward pass yet");
    int width = 0;
    for (int k = 0; k < 2; ++k)
        for (int l = 0; l < t->net[k].n - 1; ++l) width += t->net[k].out[l];
    int col = 0;
    for (int k = 0; k < 2; ++k)
        for (int l = 0; l < t->net[k].n - 1; ++l) {
            const int o = t->net[k].out[l];
            cudaError_t e = cudaMemcpy2DAsync(act + col, (size_t)width * 4, t->d_act[k][l], (size_t)o * 4,
                                              (size_t)o * 4, (size_t)B, cudaMemcpyDefault, (cudaStream_t)stream);
            if (e != cudaSuccess) return cuda_err(e, "cudaMemcpy2DAsync(activations)");
            col += o;
        }
    return ROLLOUT_OK;
}

int ppo_get_weights(ppo_trainer *t, float *weights, void *stream)
{
    clear_error();
    if (!t || !weights) return set_error(ROLLOUT_ERR_INVALID, "null argument");
    cudaError_t e = cudaMemcpyAsync(weights, t->d_w, t->n_weights * 4, cudaMemcpyDefault, (cudaStream_t)stream);
    return e == cudaSuccess ? ROLLOUT_OK : cuda_err(e, "cudaMemcpyAsync(weights)");
}

int ppo_device_weights(ppo_trainer *t, const float **weights)
{
    clear_error();
    if (!t || !weights) return set_error(ROLLOUT_ERR_INVALID, "null argument");
    *weights = t->d_w;
    return ROLLOUT_OK;
}

int ppo_reset_optimizer(ppo_trainer *t, void *stream)
{
    clear_error();
    if (!t) return set_error(ROLLOUT_ERR_INVALID, "null trainer");
    cudaError_t e;
    if ((e = cudaMemsetAsync(t->d_m, 0, t->n_trained * 4, (cudaStream_t)stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(t->d_v, 0, t->n_trained * 4, (cudaStream_t)stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(t->d_t, 0, sizeof(long long), (cudaStream_t)stream)) != cudaSuccess)
        return cuda_err(e, "cudaMemsetAsync(moments)");
    t->step = 0;
    return ROLLOUT_OK;
}

int ppo_status(ppo_trainer *t)
{
    clear_error();
    if (!t) return set_error(ROLLOUT_ERR_INVALID, "null trainer");
    cudaError_t e = cudaStreamSynchronize(t->last_stream);
    if (e != cudaSuccess) return cuda_err(e, "cudaStreamSynchronize");
    int st = 0;
    if ((e = cudaMemcpy(&st, t->d_status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess ||
        (e = cudaMemset(t->d_status, 0, sizeof(int))) != cudaSuccess)
        return cuda_err(e, "status read");
    return st;
}

void ppo_destroy(ppo_trainer *t)
{
    if (!t) return;
    cudaDeviceSynchronize();
    free_trainer(t);
}

}  // extern "C"
