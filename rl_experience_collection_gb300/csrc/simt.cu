// simt.cu -- float32 CUDA-core kernels (dtype ROLLOUT_FP32).
//
// Phase 1 (rollout): one thread per episode runs the serial chain of page
// "PPO CUDA Pipeline Design -- Zero-Roundtrip Experience Collection",
// section "Kernel Phases", Phase A steps 1-4 and 6-12: state, actor MLP
// 54->128->64->45, softmax/CDF/LCG sample, environment step, reset.
// The actor weights sit in shared memory, transposed so that every thread
// reads the same weight (a broadcast) while it accumulates its own episode.
//
// Phase 2 (value): tiles of rows (tuples) run the critic MLP
// 54->512->384->256->128->64->1 (Phase A step 5), the curiosity model
// (step 9, bonus = cur_coef * MSE against the pre-reset next state); the
// stored state rows come from states.cu.  Every dense layer is out[j] = b[j] + sum_k in[k] *
// W[j][k] with f32 accumulation in k order (page "GPU Pipeline Phase 2b",
// "Kernel Components" 1).
#include "env.cuh"
#include "internal.cuh"

namespace rl {

namespace {

// actor weights packed for phase 1: W^T [in][out_pad] then b[out_pad]
constexpr int kA1 = 0;                                   // W1^T [54][128]
constexpr int kB1 = kA1 + kState * kActorH1;
constexpr int kA2 = kB1 + kActorH1;                      // W2^T [128][64]
constexpr int kB2 = kA2 + kActorH1 * kActorH2;
constexpr int kA3 = kB2 + kActorH2;                      // W3^T [64][48]
constexpr int kB3 = kA3 + kActorH2 * 48;
constexpr int kActorPacked = kB3 + 48;

constexpr int kP1Threads = 32;

__device__ __forceinline__ void acc_row32(float (&acc)[32], const float *w, float x)
{
    const float4 *w4 = reinterpret_cast<const float4 *>(w);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 v = w4[q];
        acc[4 * q + 0] = fmaf(v.x, x, acc[4 * q + 0]);
        acc[4 * q + 1] = fmaf(v.y, x, acc[4 * q + 1]);
        acc[4 * q + 2] = fmaf(v.z, x, acc[4 * q + 2]);
        acc[4 * q + 3] = fmaf(v.w, x, acc[4 * q + 3]);
    }
}

__global__ void __launch_bounds__(kP1Threads) phase1_simt_kernel(Phase1Args a, const float *__restrict__ wp)
{
    extern __shared__ __align__(16) float sm[];
    float *W = sm;                                        // kActorPacked floats
    float *xs = W + kActorPacked;                         // [54][T]
    float *h1 = xs + kState * kP1Threads;                 // [128][T]
    float *h2 = h1 + kActorH1 * kP1Threads;               // [64][T]
    const int tid = threadIdx.x;
    for (int i = tid; i < kActorPacked; i += kP1Threads) W[i] = wp[i];
    __syncthreads();

    const int n = blockIdx.x * kP1Threads + tid;
    if (n >= a.N) return;
    const int L = a.L;
    const long long row0 = (long long)n * L;
    const int start = a.starts[n];
    if (!start_ok(start, L, a.n_bars)) {
        set_status(a.status, ROLLOUT_ERR_RANGE);
        for (int t = 0; t < L; ++t) {
            a.actions[row0 + t] = 0; a.logp[row0 + t] = 0.f; a.dones[row0 + t] = 0;
            a.rewards[row0 + t] = 0.f; a.v_in[row0 + t] = 0.f; a.v_post[row0 + t] = 0.f;
        }
        return;
    }
    EpState st;
    ep_reset(st);
    st.rng = a.seeds[n];
    const float *F = a.F;

    for (int t = 0; t < L; ++t) {
        const long long b = (long long)start + t;
        const float *fr = F + b * kMarket;
#pragma unroll 3
        for (int i = 0; i < kMarket; ++i) xs[i * kP1Threads + tid] = __ldg(fr + i);
        xs[kMarket * kP1Threads + tid] = st.V;
        xs[(kMarket + 1) * kP1Threads + tid] = st.e;
        xs[(kMarket + 2) * kP1Threads + tid] = a.env.spread;
        const float f0n = __ldg(fr + kMarket);            // F[b+1, 0]

        // actor layer 1: 54 -> 128, ReLU
        for (int jc = 0; jc < kActorH1 / 32; ++jc) {
            float acc[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = 0.f;
            for (int i = 0; i < kState; ++i)
                acc_row32(acc, W + kA1 + i * kActorH1 + jc * 32, xs[i * kP1Threads + tid]);
#pragma unroll
            for (int j = 0; j < 32; ++j)
                h1[(jc * 32 + j) * kP1Threads + tid] = relu(acc[j] + W[kB1 + jc * 32 + j]);
        }
        // actor layer 2: 128 -> 64, ReLU
        for (int jc = 0; jc < kActorH2 / 32; ++jc) {
            float acc[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = 0.f;
            for (int i = 0; i < kActorH1; ++i)
                acc_row32(acc, W + kA2 + i * kActorH2 + jc * 32, h1[i * kP1Threads + tid]);
#pragma unroll
            for (int j = 0; j < 32; ++j)
                h2[(jc * 32 + j) * kP1Threads + tid] = relu(acc[j] + W[kB2 + jc * 32 + j]);
        }
        // actor layer 3: 64 -> 45 logits
        float lg[48];
#pragma unroll
        for (int j = 0; j < 48; ++j) lg[j] = 0.f;
        for (int i = 0; i < kActorH2; ++i) {
            const float hv = h2[i * kP1Threads + tid];
            const float4 *w4 = reinterpret_cast<const float4 *>(W + kA3 + i * 48);
#pragma unroll
            for (int q = 0; q < 12; ++q) {
                const float4 v = w4[q];
                lg[4 * q + 0] = fmaf(v.x, hv, lg[4 * q + 0]);
                lg[4 * q + 1] = fmaf(v.y, hv, lg[4 * q + 1]);
                lg[4 * q + 2] = fmaf(v.z, hv, lg[4 * q + 2]);
                lg[4 * q + 3] = fmaf(v.w, hv, lg[4 * q + 3]);
            }
        }
        float logits[kActions];
#pragma unroll
        for (int j = 0; j < kActions; ++j) logits[j] = lg[j] + W[kB3 + j];

        const float u = lcg_uniform(st.rng);
        float logp;
        const int act = sample_action<kActions>(logits, u, logp);
        const float v_in = st.V;
        float v_post;
        int done;
        const float rew = env_step(st, act, f0n, a.env, v_post, done);
        a.actions[row0 + t] = act;
        a.logp[row0 + t] = logp;
        a.dones[row0 + t] = done;
        a.rewards[row0 + t] = rew;
        a.v_in[row0 + t] = v_in;
        a.v_post[row0 + t] = v_post;
    }
}

// ---------------------------------------------------------------- phase 2

constexpr int kVThreads = 256;

// out[r][j] = (relu_ ? relu : identity)(b[j] + sum_k in[r][k] * W^T[k][j]) for the block's ROWS rows.
template <int ROWS>
__device__ void dense_rows(const float *__restrict__ WT, const float *__restrict__ bias, int K, int N,
                           const float *in, int ldi, float *out, int ldo, bool relu_,
                           const int *onehot = nullptr)
{
    constexpr int RPT = ROWS / 4;
    const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;
    for (int c0 = 0; c0 < N; c0 += 64) {
        const int j = c0 + tx;
        const bool ok = j < N;
        float acc[RPT];
#pragma unroll
        for (int r = 0; r < RPT; ++r) acc[r] = 0.f;
        for (int k = 0; k < K; ++k) {
            const float w = ok ? __ldg(WT + (long long)k * N + j) : 0.f;
#pragma unroll
            for (int r = 0; r < RPT; ++r) acc[r] = fmaf(in[(ty * RPT + r) * ldi + k], w, acc[r]);
        }
        if (onehot) {   // one-hot input block after the first K inputs: a column gather
#pragma unroll
            for (int r = 0; r < RPT; ++r)
                acc[r] += ok ? __ldg(WT + (long long)(K + onehot[ty * RPT + r]) * N + j) : 0.f;
        }
        if (ok) {
            const float bj = __ldg(bias + j);
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                float v = acc[r] + bj;
                out[(ty * RPT + r) * ldo + j] = relu_ ? rl::relu(v) : v;
            }
        }
    }
}

template <int ROWS, int LD>
__global__ void __launch_bounds__(kVThreads) value_simt_kernel(ValueArgs a, SimtWeights w)
{
    extern __shared__ __align__(16) float sm[];
    float *A = sm;                       // [ROWS][LD]
    float *B = A + ROWS * LD;            // [ROWS][LD]
    float *T = B + ROWS * LD;            // [ROWS][56] curiosity target
    float *Z = T + ROWS * 56;            // [ROWS][64]
    float *P = Z + ROWS * 64;            // [ROWS][56]
    __shared__ long long s_bar[ROWS];    // bar of the state row
    __shared__ long long s_row[ROWS];    // flat tuple index, or -1
    __shared__ int s_kind[ROWS];         // 0 tuple, 1 bootstrap, -1 none / invalid episode
    __shared__ int s_act[ROWS];
    __shared__ float s_vin[ROWS], s_vpost[ROWS], s_ein[ROWS], s_epost[ROWS];
    __shared__ long long s_boot_dst[ROWS];

    const int tid = threadIdx.x;
    const long long NL = (long long)a.N * a.L;
    const long long total = NL + a.N;
    const int L = a.L;

    for (long long tile = blockIdx.x; tile * ROWS < total; tile += gridDim.x) {
        if (tid < ROWS) {
            const long long r = tile * ROWS + tid;
            int kind = -1;
            long long bar = 0, row = -1, boot_dst = -1;
            int act = 0;
            float vin = 0.f, vpost = 0.f, ein = 0.f, epost = 0.f;
            if (r < NL) {
                const int n = (int)(r / L), t = (int)(r % L);
                const int start = a.starts[n];
                row = r;
                if (start_ok(start, L, a.n_bars)) {
                    kind = 0;
                    bar = (long long)start + t;
                    act = a.actions[r];
                    vin = a.values[r];
                    vpost = a.v_post[r];
                    epost = exposure_of(act);
                    ein = (t == 0 || a.dones[r - 1]) ? 0.f : exposure_of(a.actions[r - 1]);
                } else {
                    kind = -2;            // invalid episode: zero outputs
                }
            } else if (r < total) {
                const int n = (int)(r - NL);
                const int start = a.starts[n];
                const long long last = (long long)n * L + L - 1;
                boot_dst = last;
                if (start_ok(start, L, a.n_bars)) {
                    kind = 1;
                    bar = (long long)start + L;   // pre-reset next state of step L-1
                    act = a.actions[last];
                    vin = a.v_post[last];
                    ein = exposure_of(act);
                } else {
                    kind = -3;
                }
            }
            s_kind[tid] = kind; s_bar[tid] = bar; s_row[tid] = row; s_act[tid] = act;
            s_vin[tid] = vin; s_vpost[tid] = vpost; s_ein[tid] = ein; s_epost[tid] = epost;
            s_boot_dst[tid] = boot_dst;
        }
        __syncthreads();
        // state rows (A) and curiosity targets (T)
        for (int idx = tid; idx < ROWS * kState; idx += kVThreads) {
            const int rr = idx / kState, j = idx % kState;
            const int kind = s_kind[rr];
            float x = 0.f, tg = 0.f;
            if (kind >= 0) {
                const long long bar = s_bar[rr];
                if (j < kMarket) {
                    x = __ldg(a.F + bar * kMarket + j);
                    if (kind == 0) tg = __ldg(a.F + (bar + 1) * kMarket + j);
                } else if (j == kMarket) { x = s_vin[rr]; tg = s_vpost[rr]; }
                else if (j == kMarket + 1) { x = s_ein[rr]; tg = s_epost[rr]; }
                else { x = a.env.spread; tg = a.env.spread; }
            }
            A[rr * LD + j] = x;
            T[rr * 56 + j] = tg;
        }
        __syncthreads();
        // curiosity: [x ; onehot(a)] -> 64 ReLU -> 54
        dense_rows<ROWS>(w.cur0_T, w.cur0_b, kState, kCurH, A, LD, Z, 64, true, s_act);
        __syncthreads();
        dense_rows<ROWS>(w.cur1_T, w.cur1_b, kCurH, kState, Z, 64, P, 56, false);
        __syncthreads();
        // critic chain A -> B -> A -> ... ; the last hidden layer lands in `h`
        float *src = A, *dst = B;
        for (int l = 0; l < kCriticLayers - 1; ++l) {
            dense_rows<ROWS>(w.critic_T[l], w.critic_b[l], w.critic_w[l], w.critic_w[l + 1], src, LD,
                             dst, LD, true);
            __syncthreads();
            float *tmp = src; src = dst; dst = tmp;
        }
        // head (width 1) and curiosity MSE, one warp per row group
        const int warp = tid >> 5, lane = tid & 31;
        const int K5 = w.critic_w[kCriticLayers - 1];
        for (int rr = warp; rr < ROWS; rr += kVThreads / 32) {
            float hv = 0.f;
            for (int k = lane; k < K5; k += 32) hv = fmaf(src[rr * LD + k], __ldg(w.critic_T[kCriticLayers - 1] + k), hv);
            float se = 0.f;
            for (int j = lane; j < kState; j += 32) {
                const float d = P[rr * 56 + j] - T[rr * 56 + j];
                se = fmaf(d, d, se);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                hv += __shfl_xor_sync(0xffffffffu, hv, o);
                se += __shfl_xor_sync(0xffffffffu, se, o);
            }
            if (lane == 0) {
                const int kind = s_kind[rr];
                const float v = hv + __ldg(w.critic_b[kCriticLayers - 1]);
                if (kind == 0) {
                    const long long r = s_row[rr];
                    a.values[r] = v;
                    a.rewards[r] += a.env.cur_coef * (se / (float)kState);
                } else if (kind == -2) {
                    a.values[s_row[rr]] = 0.f;
                } else if (kind == 1) {
                    a.boot[s_boot_dst[rr]] = v;
                } else if (kind == -3) {
                    a.boot[s_boot_dst[rr]] = 0.f;
                }
            }
        }
        __syncthreads();
    }
}

}  // namespace



cudaError_t launch_phase1_simt(const Phase1Args &a, const float *actor_packed, cudaStream_t s)
{
    const size_t smem = sizeof(float) * (kActorPacked + (kState + kActorH1 + kActorH2) * kP1Threads);
    static std::atomic<unsigned long long> attr{0};   // devices whose attributes are set
    {
        const cudaError_t e_attr = once_per_device(attr, [&]() -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(phase1_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return e;
            return cudaSuccess;
        });
        if (e_attr != cudaSuccess) return e_attr;
    }
    const int blocks = (a.N + kP1Threads - 1) / kP1Threads;
    phase1_simt_kernel<<<blocks, kP1Threads, smem, s>>>(a, actor_packed);
    return cudaGetLastError();
}

template <int ROWS, int LD>
static cudaError_t launch_value_t(const ValueArgs &a, const SimtWeights &w, cudaStream_t s)
{
    const size_t smem = sizeof(float) * (2 * ROWS * LD + ROWS * (56 + 64 + 56));
    static std::atomic<unsigned long long> attr{0};   // devices whose attributes are set
    {
        const cudaError_t e_attr = once_per_device(attr, [&]() -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(value_simt_kernel<ROWS, LD>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            return cudaSuccess;
        });
        if (e_attr != cudaSuccess) return e_attr;
    }
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long total = (long long)a.N * a.L + a.N;
    const long long tiles = (total + ROWS - 1) / ROWS;
    const int grid = (int)(tiles < (long long)sms * 8 ? tiles : (long long)sms * 8);
    value_simt_kernel<ROWS, LD><<<grid, kVThreads, smem, s>>>(a, w);
    return cudaGetLastError();
}

cudaError_t launch_value_simt(const ValueArgs &a, const SimtWeights &w, cudaStream_t s)
{
    int widest = 0;
    for (int l = 1; l < kCriticLayers; ++l) widest = w.critic_w[l] > widest ? w.critic_w[l] : widest;
    if (widest <= 512) return launch_value_t<32, 516>(a, w, s);
    return launch_value_t<16, 1028>(a, w, s);
}

}  // namespace rl
