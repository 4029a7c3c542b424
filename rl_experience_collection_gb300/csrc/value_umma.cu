// value_umma.cu -- tensor-core value phase (phase 2) for ROLLOUT_BF16.
//
// Page "PPO CUDA Pipeline Design -- Zero-Roundtrip Experience Collection",
// section "Kernel Phases", Phase A step 5 (critic 54->512->384->256->128->64->1),
// step 9 (curiosity forward model, bonus = cur_coef * MSE against the
// pre-reset next state) and step 11 (state rows); section "Weight Layout".
//
// The critic and the curiosity model do not feed the state trajectory, so
// they run here over every tuple at once instead of inside the serial step
// loop: a persistent CTA takes tiles of 128 consecutive tuples (plus one
// bootstrap row per episode: the pre-reset next state after the last step)
// and runs each layer as M=128 tcgen05 MMAs with f32 accumulators in tensor
// memory.  Warp roles:
//   warps 0-3  rows: build the state rows (A operand + out_states), drain
//              TMEM after every layer (bias, ReLU, bf16 rounding) into the
//              next layer's swizzled A operand, head dot product, curiosity
//              MSE, final stores
//   warp 4     producer: streams the weight units (K-chunk x N-block tiles,
//              pre-swizzled on the host) from L2 with 1-D bulk TMA into a
//              two-stage ring
//   warp 5     allocates TMEM; one lane issues the MMAs and the commits
// Activations stay resident in shared memory (slots of 128 rows x 128 B);
// each layer's output overwrites its input after the layer's MMAs complete.
#include "env.cuh"
#include "umma.cuh"
#include "umma_path.cuh"

namespace rl {

namespace {

using namespace umma;

constexpr int kVThreads = 192;
constexpr int kSlot = 128 * 128;          // one activation K-chunk (128 rows x 128 B)
constexpr int kStage = 256 * 128;         // one weight unit (<= 256 rows x 128 B)
constexpr int kStages = 2;
constexpr int kXSlot = 8;                 // state operand
constexpr int kZSlot = 2;                 // curiosity hidden operand
constexpr int kNumSlots = 9;
constexpr int kValueSmem = kNumSlots * kSlot + kStages * kStage + 1024;

// the producer and the MMA issuer both walk the jobs in enum order:
// critic 1..5, then curiosity 1..2
__host__ __device__ constexpr int a_slot_of(int j) { return (j == kJobCrit1 || j == kJobCur1) ? kXSlot : (j == kJobCur2 ? kZSlot : 0); }
__host__ __device__ constexpr int d_col_of(int j) { return j == kJobCur1 ? 64 : (j == kJobCur2 ? 128 : 0); }
__host__ __device__ constexpr bool waits_act(int j) { return j != kJobCur1; }
__host__ __device__ constexpr int acc_bar_of(int j) { return (j == kJobCur1 || j == kJobCur2) ? 1 : 0; }

// 32 f32 values -> 4 bf16 units (64 bytes) of row r at column c0 of the activation slots
__device__ __forceinline__ void put32_bf16(uint8_t *slots, int r, int c0, const float (&v)[32])
{
    uint8_t *tile = slots + (c0 >> 6) * kSlot;
    const int u0 = (c0 & 63) >> 3;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 p;
        p.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
        p.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
        p.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
        p.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
        *reinterpret_cast<uint4 *>(tile + sw128_offset(r, u0 + q)) = p;
    }
}

__device__ __forceinline__ float bf16_round(float x) { return __uint_as_float(pack_bf16x2(0.f, x) & 0xFFFF0000u); }

struct RowInfo {
    int kind;            // 0 tuple, 1 bootstrap row, 2 tuple of an invalid episode, 3 bootstrap of one, -1 none
    long long row;       // flat tuple index (kind 0/2) or the slot receiving the bootstrap value (kind 1/3)
    long long bar;       // bar of the state row
    int act;
    float vin, ein, vpost, epost;
};

__device__ __forceinline__ RowInfo decode_row(const ValueArgs &a, long long r)
{
    RowInfo ri{};
    ri.kind = -1;
    const long long NL = (long long)a.N * a.L;
    const int L = a.L;
    if (r < NL) {
        const int n = (int)(r / L), t = (int)(r % L);
        const int start = a.starts[n];
        ri.row = r;
        if (start_ok(start, L, a.n_bars)) {
            ri.kind = 0;
            ri.bar = (long long)start + t;
            ri.act = a.actions[r];
            ri.vin = a.values[r];
            ri.vpost = a.v_post[r];
            ri.epost = exposure_of(ri.act);
            ri.ein = (t == 0 || a.dones[r - 1]) ? 0.f : exposure_of(a.actions[r - 1]);
        } else {
            ri.kind = 2;
        }
    } else if (r < NL + a.N) {
        const int n = (int)(r - NL);
        const int start = a.starts[n];
        const long long last = (long long)n * L + L - 1;
        ri.row = last;
        if (start_ok(start, L, a.n_bars)) {
            ri.kind = 1;
            ri.bar = (long long)start + L;
            ri.act = a.actions[last];
            ri.vin = a.v_post[last];
            ri.ein = exposure_of(ri.act);
        } else {
            ri.kind = 3;
        }
    }
    return ri;
}

__global__ void __launch_bounds__(kVThreads, 1) value_umma_bf16_kernel(ValueArgs a, UmmaWeights w)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *slots = sm;
    uint8_t *ring = sm + kNumSlots * kSlot;
    __shared__ __align__(8) uint64_t bar_full[kStages], bar_empty[kStages], bar_acc[2], bar_act, bar_final;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        abort_sh = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], 1);
        }
        mbar_init(&bar_acc[0], 1);
        mbar_init(&bar_acc[1], 1);
        mbar_init(&bar_act, 128);
        mbar_init(&bar_final, 1);
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    volatile int *abort = &abort_sh;

    const long long total = (long long)a.N * a.L + a.N;
    const long long n_tiles = (total + 127) / 128;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (long long tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                for (int jj = 0; jj < kNumJobs && ok; ++jj) {
                    const UmmaLayer &Ly = w.job[jj];
                    const uint8_t *src = w.stream + Ly.w_off;
                    for (int c = 0; c < Ly.k_chunks && ok; ++c) {
                        for (int nb = 0; nb < Ly.n_blocks && ok; ++nb) {
                            const uint32_t bytes = (uint32_t)Ly.nb_rows[nb] * 128u;
                            ok = mbar_wait(&bar_empty[stage], phase ^ 1u, abort);
                            if (!ok) break;
                            mbar_arrive_expect_tx(&bar_full[stage], bytes);
                            bulk_g2s(ring + stage * kStage, src, bytes, &bar_full[stage]);
                            src += bytes;
                            if (++stage == kStages) { stage = 0; phase ^= 1u; }
                        }
                    }
                }
            }
            // wait until every issued copy has landed before the CTA may exit
            for (int s = 0; s < kStages && ok; ++s) {
                ok = mbar_wait(&bar_empty[stage], phase ^ 1u, abort);
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
            if (!ok) {   // aborted: give copies already issued time to land (bounded)
                const uint64_t t0 = global_ns();
                while (global_ns() - t0 < 2000000ull) { }
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, act_phase = 0;
            bool ok = true;
            const uint32_t s_slots = smem_u32(slots), s_ring = smem_u32(ring);
            for (long long tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                for (int jj = 0; jj < kNumJobs && ok; ++jj) {
                    const int j = jj;
                    const UmmaLayer &Ly = w.job[j];
                    if (waits_act(j)) {
                        ok = mbar_wait(&bar_act, act_phase, abort);
                        act_phase ^= 1u;
                        tc_fence_after();
                    }
                    const uint32_t a_base = s_slots + a_slot_of(j) * kSlot;
                    for (int c = 0; c < Ly.k_chunks && ok; ++c) {
                        int col = d_col_of(j);
                        for (int nb = 0; nb < Ly.n_blocks && ok; ++nb) {
                            const int rows = Ly.nb_rows[nb];
                            ok = mbar_wait(&bar_full[stage], phase, abort);
                            if (!ok) break;
                            tc_fence_after();
                            const uint32_t b_base = s_ring + stage * kStage;
                            const uint32_t id = idesc(true, 128, rows);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma<true>(tmem + col, desc_sw128(a_base + c * kSlot + 32 * k),
                                          desc_sw128(b_base + 32 * k), id, (c | k) != 0);
                            mma_commit(&bar_empty[stage]);
                            col += rows;
                            if (++stage == kStages) { stage = 0; phase ^= 1u; }
                        }
                    }
                    mma_commit(&bar_acc[acc_bar_of(j)]);
                }
            }
            // every MMA issued must complete before TMEM is released (bounded wait)
            mma_commit(&bar_final);
            int never = 0;
            mbar_wait(&bar_final, 0, &never, 100000000ull);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ row warps
        const int r = tid;                                  // TMEM lane / operand row
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
        uint32_t acc_phase[2] = {0, 0};
        bool ok = true;
        const float *vec = w.vec;
        for (long long tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
            const RowInfo ri = decode_row(a, tile * 128 + r);
            // ---- state row: A operand (bf16) and out_states (f32)
            {
                float x[64];
                const bool has = ri.kind == 0 || ri.kind == 1;
                const float *fr = a.F + (has ? ri.bar : 0) * kMarket;
#pragma unroll
                for (int j = 0; j < kMarket; ++j) x[j] = has ? __ldg(fr + j) : 0.f;
                x[kMarket] = has ? ri.vin : 0.f;
                x[kMarket + 1] = has ? ri.ein : 0.f;
                x[kMarket + 2] = has ? a.env.spread : 0.f;
#pragma unroll
                for (int j = kState; j < 64; ++j) x[j] = 0.f;
                float lo[32], hi[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) { lo[j] = x[j]; hi[j] = x[32 + j]; }
                put32_bf16(slots + kXSlot * kSlot, r, 0, lo);
                put32_bf16(slots + kXSlot * kSlot, r, 32, hi);
                if (ri.kind == 0 || ri.kind == 2) {
                    float2 *dst = reinterpret_cast<float2 *>(a.states + ri.row * kState);
#pragma unroll
                    for (int j = 0; j < kState / 2; ++j) dst[j] = make_float2(x[2 * j], x[2 * j + 1]);
                }
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(&bar_act);
            // ---- critic hidden layers 1-4
            for (int l = 0; l < 4 && ok; ++l) {
                const UmmaLayer &Ly = w.job[kJobCrit1 + l];
                ok = __all_sync(0xffffffffu, mbar_wait(&bar_acc[0], acc_phase[0], abort));
                acc_phase[0] ^= 1u;
                tc_fence_after();
                const float *bias = vec + Ly.bias_off;
                for (int g = 0; g < Ly.n_out / 32; ++g) {
                    float v[32];
                    tmem_ld32(lane_addr + 32 * g, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = fmaxf(v[i] + __ldg(bias + 32 * g + i), 0.f);
                    put32_bf16(slots, r, 32 * g, v);
                }
                fence_async_smem();
                tc_fence_before();
                mbar_arrive(&bar_act);
            }
            // ---- critic layer 5 + scalar head
            float value = 0.f;
            if (ok) {
                const UmmaLayer &Ly = w.job[kJobCrit5];
                ok = __all_sync(0xffffffffu, mbar_wait(&bar_acc[0], acc_phase[0], abort));
                acc_phase[0] ^= 1u;
                tc_fence_after();
                const float *bias = vec + Ly.bias_off, *hw = vec + w.head_w_off;
                for (int g = 0; g < Ly.n_out / 32; ++g) {
                    float v[32];
                    tmem_ld32(lane_addr + 32 * g, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        value = fmaf(bf16_round(fmaxf(v[i] + __ldg(bias + 32 * g + i), 0.f)), __ldg(hw + 32 * g + i), value);
                }
                value += __ldg(vec + w.head_b_off);
            }
            // ---- curiosity layer 1: state part from TMEM + one-hot column gather
            if (ok) {
                const UmmaLayer &Ly = w.job[kJobCur1];
                ok = __all_sync(0xffffffffu, mbar_wait(&bar_acc[1], acc_phase[1], abort));
                acc_phase[1] ^= 1u;
                tc_fence_after();
                const float *bias = vec + Ly.bias_off;
                const float *oh = vec + w.onehot_off + (ri.act >= 0 && ri.act < kActions ? ri.act : 0) * kCurH;
#pragma unroll
                for (int g = 0; g < kCurH / 32; ++g) {
                    float v[32];
                    tmem_ld32(lane_addr + d_col_of(kJobCur1) + 32 * g, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] = fmaxf((v[i] + __ldg(oh + 32 * g + i)) + __ldg(bias + 32 * g + i), 0.f);
                    put32_bf16(slots + kZSlot * kSlot, r, 32 * g, v);
                }
                fence_async_smem();
                tc_fence_before();
                mbar_arrive(&bar_act);
            }
            // ---- curiosity layer 2 + MSE against the pre-reset next state
            float se = 0.f;
            if (ok) {
                const UmmaLayer &Ly = w.job[kJobCur2];
                ok = __all_sync(0xffffffffu, mbar_wait(&bar_acc[1], acc_phase[1], abort));
                acc_phase[1] ^= 1u;
                tc_fence_after();
                const float *bias = vec + Ly.bias_off;
                const float *fn = a.F + (ri.kind == 0 ? ri.bar + 1 : 0) * kMarket;
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    float v[32];
                    tmem_ld32(lane_addr + d_col_of(kJobCur2) + 32 * g, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int j = 32 * g + i;
                        if (j < kState) {
                            const float tgt = j < kMarket ? __ldg(fn + j)
                                              : (j == kMarket ? ri.vpost : (j == kMarket + 1 ? ri.epost : a.env.spread));
                            const float d = (v[i] + __ldg(bias + j)) - tgt;
                            se = fmaf(d, d, se);
                        }
                    }
                }
                tc_fence_before();
            }
            // ---- outputs
            if (ri.kind == 0) {
                a.values[ri.row] = value;
                a.rewards[ri.row] += a.env.cur_coef * (se / (float)kState);
            } else if (ri.kind == 2) {
                a.values[ri.row] = 0.f;
            } else if (ri.kind == 1) {
                a.boot[ri.row] = value;
            } else if (ri.kind == 3) {
                a.boot[ri.row] = 0.f;
            }
        }
    }
    if (abort_sh && tid == 0) set_status(a.status, ROLLOUT_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_value_umma(const ValueArgs &a, const UmmaWeights &w, cudaStream_t s)
{
    if (!w.bf16 || w.wide) return cudaErrorNotSupported;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(value_umma_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kValueSmem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long total = (long long)a.N * a.L + a.N;
    const long long tiles = (total + 127) / 128;
    const int grid = (int)(tiles < sms ? tiles : sms);
    value_umma_bf16_kernel<<<grid, kVThreads, kValueSmem, s>>>(a, w);
    return cudaGetLastError();
}

}  // namespace rl
