// per.cu -- the GPU-resident prioritised experience replay buffer
// (include/per.h).
//
// Page "GPU-Resident Prioritized Experience Replay": the ring of transitions
// and priorities ("New struct: GpuReplayBuffer"), proportional sampling with
// importance-sampling weights ("Sampling Kernels / Proportional"), the
// priority scatter ("Priority update"), device-to-device insertion at the
// maximum priority ("Experience Insertion") and the clamp of non-finite
// priorities ("Error Handling").
//
// The page rebuilds (or incrementally maintains) the cumulative priorities
// for each sampling call.  Here the sums are kept current in three levels, all
// in double and in a fixed order: a sum per sub-block of 128 slots, a sum per
// block of 64 sub-blocks (8192 slots), and the prefix over the blocks.  An
// insert re-sums the sub-blocks and blocks it wrote, an update those of the
// slots it named, and each then rebuilds the prefix (one CTA; a two-level
// chain, so that it never decreases and a block of zero sum is an empty
// interval).  A sampling call reads no whole array: one warp per sample
// searches the block prefix 128 ways at a time (two rounds up to 16384
// blocks), then the block's 64 sub-sums, then the sub-block's 128 priorities,
// with warp-wide running sums, and the last CTA to finish normalises the
// weights (in float: the weight scales a loss; the slot is what must be exact).
// GB300's double-precision rate is low (about 2 operations per clock per SM),
// so the levels keep the double additions per sample to about 600, block sums
// are warp trees, and the update's double pow runs 32 threads per CTA, spread
// over SMs.  Only positive slots can be picked; where rounding puts
// the target past a level's running total, the level's last positive entry is
// taken (the exact answer's neighbour).  Nothing depends on timing: every sum
// has one order, and where an update names a slot twice the later entry wins
// through an owner array (atomicMax of the entry number), so repeated calls
// give identical results.
#include <math.h>
#include <string.h>

#include <new>

#include "../../include/per.h"
#include "internal.cuh"

using namespace rl;

namespace {

constexpr int kSub = 128;               // priorities per sub-block (a warp's float4 each)
constexpr int kSubs = 64;               // sub-blocks per block (two per lane)
constexpr int kBlock = kSub * kSubs;    // priorities per block
constexpr int kScanThreads = 1024;      // 32 groups of 32 chunks
constexpr int kStagedBlocks = 16384;    // the prefix rebuild stages up to this many block sums in smem
constexpr int kWarpsPerCta = 8;
constexpr int kSampleWarps = 4;         // samples per CTA (128 CTAs for a batch of 512)
constexpr int kFp64Threads = 32;        // CTA size of the double-heavy update kernel (spread over SMs)
constexpr int kMaxBatch = 65536;
constexpr int kMaxDim = 4096;

int cuda_err(cudaError_t e, const char *what)
{
    return set_error(e == cudaErrorMemoryAllocation ? ROLLOUT_ERR_NOMEM : ROLLOUT_ERR_CUDA, "%s: %s", what,
                     cudaGetErrorString(e));
}

long long blocks_for(long long n) { return (n + kBlock - 1) / kBlock; }

// SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): output n of the generator
// seeded with `seed`, that is the state after n + 1 golden-ratio increments
// put through the generator's mixing function
__device__ __forceinline__ uint64_t splitmix64_output(uint64_t seed, uint64_t n)
{
    uint64_t z = seed + (n + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// every lane ends with the same sum, formed in the same order on every call
__device__ __forceinline__ double warp_sum(double v)
{
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Re-sums sub-blocks, one warp each: sub-block first + w, or, when `slots` is
// given, the sub-block of slots[w] (entries outside [0, size) skipped).
// Slots at or past `size` count as zero.
__global__ void __launch_bounds__(kWarpsPerCta * 32) sub_sum_kernel(const float *__restrict__ prio, long long size,
                                                                   long long first, long long n,
                                                                   const int32_t *__restrict__ slots,
                                                                   double *__restrict__ sub)
{
    const long long w = blockIdx.x * (long long)kWarpsPerCta + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= n) return;
    long long sb;
    if (slots) {
        const int32_t i = slots[w];
        if (i < 0 || i >= size) return;
        sb = i / kSub;
    } else {
        sb = first + w;
    }
    const long long e = sb * kSub + lane * 4;
    const float4 x = reinterpret_cast<const float4 *>(prio + e)[0];
    const float v[4] = {x.x, x.y, x.z, x.w};
    double s = 0.0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (e + j < size) s += (double)v[j];
    s = warp_sum(s);
    if (lane == 0) sub[sb] = s;
}

// Block sums from their 64 sub-sums, one warp each (lane l adds sub-blocks 2l
// and 2l+1, then the fixed xor tree): block first + w, or the block of
// slots[w].  A dependent chain of 6 double additions, not 64.
__global__ void __launch_bounds__(kWarpsPerCta * 32) block_sum_kernel(const double *__restrict__ sub, long long size,
                                                                     long long first, long long n,
                                                                     const int32_t *__restrict__ slots,
                                                                     double *__restrict__ bsum)
{
    const long long w = blockIdx.x * (long long)kWarpsPerCta + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= n) return;
    long long b;
    if (slots) {
        const int32_t i = slots[w];
        if (i < 0 || i >= size) return;
        b = i / kBlock;
    } else {
        b = first + w;
    }
    const double2 v = reinterpret_cast<const double2 *>(sub + b * kSubs)[lane];
    const double s = warp_sum(v.x + v.y);
    if (lane == 0) bsum[b] = s;
}

// prefix[b] = the block sums before b, prefix[nb] = total.  Thread t owns a
// contiguous chunk of blocks (sum S_t, accumulated from zero in order); the 32
// chunks of group g are chained by one lane (H[t+1] = H[t] + S_t, group total
// T_g = H[last] + S_last) and the groups by thread 0 (K[g+1] = K[g] + T_g);
// then prefix[b] = K[g] + (H[t] + the chunk's blocks before b).  Each step of a
// chain adds exactly the sum the level below formed, so rounding (monotone)
// never makes the prefix decrease, and prefix[b+1] == prefix[b] whenever block
// b sums to zero, across chunk and group boundaries too.  The group chains run
// in one warp, lane g on group g: the double pipe is narrow on GB300, and 32
// chains a lane apart cost 32 warp instructions, not 1024.
template <bool STAGED>
__global__ void __launch_bounds__(kScanThreads) top_scan_kernel(const double *__restrict__ bsum_g, long long nb,
                                                                double *__restrict__ prefix, float *__restrict__ maxp)
{
    __shared__ double S[kScanThreads], H[kScanThreads], T[32], K[33];
    extern __shared__ double staged[];
    const int t = threadIdx.x, g = t >> 5;
    const double *bsum = bsum_g;
    if (STAGED) {                                   // coalesced, independent loads, once
        for (long long b = t; b < nb; b += kScanThreads) staged[b] = bsum_g[b];
        __syncthreads();
        bsum = staged;
    }
    const long long chunk = (nb + kScanThreads - 1) / kScanThreads;
    const long long lo = min(nb, (long long)t * chunk), hi = min(nb, lo + chunk);
    // chunk t = 32 g + i is kept at [i][g], so that lane g reads its group's
    // chunks without bank conflicts
    const int tr = (t & 31) * 32 + g;
    double s = 0.0;
    for (long long b = lo; b < hi; ++b) s += bsum[b];
    S[tr] = s;
    __syncthreads();
    if (t < 32) {                                   // lane t chains group t (32 lanes, one warp)
        double h = 0.0;
#pragma unroll
        for (int half = 0; half < 2; ++half) {       // operands loaded ahead of each 16-add chain
            double x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = S[(half * 16 + i) * 32 + t];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const double before = h;
                h += x[i];
                x[i] = before;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) H[(half * 16 + i) * 32 + t] = x[i];
        }
        T[t] = h;
        __syncwarp();
        if (t == 0) {
            double k = 0.0;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                double y[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) y[i] = T[half * 16 + i];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    K[half * 16 + i] = k;
                    k += y[i];
                }
            }
            K[32] = k;
        }
    }
    __syncthreads();
    const double kg = K[g], ht = H[tr];
    double part = 0.0;
    for (long long b = lo; b < hi; ++b) {
        prefix[b] = kg + (ht + part);
        part += bsum[b];
    }
    if (t == 0) {
        prefix[nb] = K[32];
        maxp[1] = maxp[0];          // the maximum priority before the next update (its +inf clamp)
    }
}

__global__ void fill_kernel(float *__restrict__ prio, long long lo, long long n, const float *__restrict__ maxp)
{
    const float v = maxp[0];
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        prio[lo + i] = v;
}

struct SampleArgs {
    const float *prio, *states, *next_states, *rewards;
    const int32_t *actions;
    const uint8_t *dones;
    const double *prefix, *sub;
    long long size, nb;
    int dim, batch;
    float beta;
    uint64_t seed, offset;
    int32_t *o_idx;
    float *o_wraw;
    float *o_w;
    unsigned *done;
    float *o_states, *o_next, *o_rewards;
    int32_t *o_actions;
    uint8_t *o_dones;
    int *status;
};

// One level of the in-block search over 32 M entries, M consecutive entries a
// lane (x >= 0); `before0` is the running total ahead of entry 0.  Returns the
// first positive entry whose running total passes t, else the last positive
// entry (-1 if none), and sets *ahead to the running total before it.
template <int M>
__device__ __forceinline__ int level_pick(const double (&x)[M], double before0, double t, int lane, double *ahead)
{
    double l[M];
    double run = 0.0;
#pragma unroll
    for (int j = 0; j < M; ++j) {
        run += x[j];
        l[j] = run;
    }
    double inc = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    double excl = __shfl_up_sync(0xffffffffu, inc, 1);
    if (lane == 0) excl = 0.0;
    const double before = before0 + excl;
    int first = -1, lastj = -1;
#pragma unroll
    for (int j = M - 1; j >= 0; --j)
        if (x[j] > 0.0) {
            if (before + l[j] > t) first = j;
            if (lastj < 0) lastj = j;
        }
    const int mine = first >= 0 ? first : lastj;
    double prev = 0.0;
#pragma unroll
    for (int j = 1; j < M; ++j)
        if (j == mine) prev = l[j - 1];
    const unsigned hit = __ballot_sync(0xffffffffu, first >= 0);
    const unsigned pos = __ballot_sync(0xffffffffu, lastj >= 0);
    const int L = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
    if (L < 0) return -1;
    *ahead = __shfl_sync(0xffffffffu, before + prev, L);
    return L * M + __shfl_sync(0xffffffffu, mine, L);
}

// One warp per sample; the last CTA to finish divides the weights by their
// maximum (a completion counter, no waiting).
__global__ void __launch_bounds__(kSampleWarps * 32) sample_kernel(SampleArgs a)
{
    const int k = blockIdx.x * kSampleWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (k < a.batch) {                                         // warp-uniform
        long long pick = -1;
        float p_pick = 0.f;
        double total = 0.0;
        const double u = (double)(splitmix64_output(a.seed, a.offset + (uint64_t)k) >> 11) * 0x1p-53;
        // the block b with prefix[b] <= t < prefix[b+1], 128 ways a round (4 probes a
        // lane); the first round's last probe is prefix[nb] = total, which fixes t
        long long lo = 0, hi = a.nb;
        double t = 0.0;
        bool first_round = true;
        for (;;) {
            const long long span = hi - lo;
            double v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = a.prefix[lo + ((long long)(lane * 4 + j + 1) * span) / 128];
            if (first_round) {
                total = __shfl_sync(0xffffffffu, v[3], 31);
                t = u * total;
                if (t >= total) t = nextafter(total, 0.0);     // u * total can round up to total
                first_round = false;
                if (!(total > 0.0)) break;
            }
            if (span <= 1) break;
            int c = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) c += v[j] <= t;
            c = __reduce_add_sync(0xffffffffu, c);             // probes 0..c-1 are at or below t
            c = min(c, 127);
            const long long nlo = c > 0 ? lo + ((long long)c * span) / 128 : lo;
            hi = lo + ((long long)(c + 1) * span) / 128;
            lo = nlo;
        }
        if (total > 0.0) {
            lo = min(lo, a.nb - 1);                             // holds already: prefix[nb] = total > t
            // the block's 64 sub-sums (two a lane), then the chosen sub-block's 128 slots
            double ahead = 0.0, ahead2 = 0.0;
            const double2 sv = reinterpret_cast<const double2 *>(a.sub + lo * kSubs)[lane];
            const double xs[2] = {sv.x, sv.y};
            const int sl = level_pick<2>(xs, a.prefix[lo], t, lane, &ahead);
            if (sl >= 0) {
                const long long e0 = (lo * kSubs + sl) * kSub + lane * 4;
                const float4 pv = reinterpret_cast<const float4 *>(a.prio + e0)[0];
                float p[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (e0 + q >= a.size) p[q] = 0.f;
                const double xe[4] = {p[0], p[1], p[2], p[3]};
                const int el = level_pick<4>(xe, ahead, t, lane, &ahead2);
                if (el >= 0) {
                    pick = (lo * kSubs + sl) * kSub + el;
                    float mine = p[0];
#pragma unroll
                    for (int q = 1; q < 4; ++q)
                        if ((el & 3) == q) mine = p[q];
                    p_pick = __shfl_sync(0xffffffffu, mine, el >> 2);
                }
            }
        }
        float w = 0.f;
        if (pick < 0) {                                         // no positive priority
            if (lane == 0) *a.status = ROLLOUT_ERR_RANGE;
            pick = 0;
        } else if (lane == 0) {
            // (size p / total)^-beta in float: the weight scales a loss, the slot
            // (above, in double) is what must be exact
            const float x = (float)a.size * p_pick / (float)total;
            w = exp2f(-a.beta * log2f(x));
        }
        if (lane == 0) {
            a.o_idx[k] = (int32_t)pick;
            a.o_wraw[k] = w;
            if (a.o_actions) a.o_actions[k] = a.actions[pick];
            if (a.o_rewards) a.o_rewards[k] = a.rewards[pick];
            if (a.o_dones) a.o_dones[k] = a.dones[pick];
        }
        const long long src = pick * a.dim, dst = (long long)k * a.dim;
        for (int c = lane; c < a.dim; c += 32) {
            if (a.o_states) a.o_states[dst + c] = a.states[src + c];
            if (a.o_next) a.o_next[dst + c] = a.next_states[src + c];
        }
    }
    // the last CTA normalises every weight by the batch maximum
    __shared__ int last;
    __shared__ float wmax[kSampleWarps];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(a.done, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    float m = 0.f;
    for (int i = threadIdx.x; i < a.batch; i += blockDim.x) m = fmaxf(m, __ldcg(a.o_wraw + i));
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    m = 0.f;
#pragma unroll
    for (int i = 0; i < kSampleWarps; ++i) m = fmaxf(m, wmax[i]);
    for (int i = threadIdx.x; i < a.batch; i += blockDim.x) a.o_w[i] = m > 0.f ? __ldcg(a.o_wraw + i) / m : 0.f;
    if (threadIdx.x == 0) *a.done = 0u;                         // ready for the next call
}

// |td|^alpha + eps in double, rounded once; NaN td -> eps, +inf -> the maximum
// priority before the call (maxp[1], refreshed by every prefix rebuild)
__device__ __forceinline__ float priority_of(float d, double alpha, float eps, const float *maxp)
{
    if (isnan(d)) return eps;
    const float v = (float)(pow(fabs((double)d), alpha) + (double)eps);
    return isinf(v) ? maxp[1] : v;
}

// the update, first launch: the last entry naming a slot owns it
__global__ void claim_kernel(const int32_t *__restrict__ idx, int batch, long long size, int32_t *__restrict__ owner,
                             int *__restrict__ status)
{
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= batch) return;
    const int32_t i = idx[k];
    if (i < 0 || i >= size) {
        *status = ROLLOUT_ERR_RANGE;
        return;
    }
    atomicMax(&owner[i], k);
}

// second launch: every named entry computes its priority (all of them count
// towards the running maximum); the owner writes it and releases the slot
__global__ void write_kernel(const int32_t *__restrict__ idx, const float *__restrict__ td, int batch, long long size,
                             double alpha, float eps, int32_t *__restrict__ owner, float *__restrict__ prio,
                             float *__restrict__ maxp)
{
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= batch) return;
    const int32_t i = idx[k];
    if (i < 0 || i >= size) return;
    const float v = priority_of(td[k], alpha, eps, maxp);
    atomicMax(reinterpret_cast<int *>(&maxp[0]), __float_as_int(v));     // v >= 0: integer order is float order
    if (owner[i] == k) {
        prio[i] = v;
        owner[i] = -1;
    }
}

}  // namespace

struct per_buffer {
    long long capacity = 0, size = 0, cursor = 0, n_alloc_blocks = 0;
    int dim = 0;
    float *d_states = nullptr, *d_next = nullptr, *d_rewards = nullptr, *d_prio = nullptr;
    int32_t *d_actions = nullptr, *d_owner = nullptr;
    uint8_t *d_dones = nullptr;
    double *d_sub = nullptr, *d_bsum = nullptr, *d_prefix = nullptr;
    float *d_wraw = nullptr;
    float *d_maxp = nullptr;     // [0] the running maximum priority, [1] its value when the last call ended
    int *d_status = nullptr;
    unsigned *d_done = nullptr;  // CTAs of the running sample call that have finished
    cudaStream_t last_stream = nullptr;
};

namespace {

void free_buffer(per_buffer *b)
{
    if (!b) return;
    cudaFree(b->d_states);
    cudaFree(b->d_next);
    cudaFree(b->d_rewards);
    cudaFree(b->d_prio);
    cudaFree(b->d_actions);
    cudaFree(b->d_owner);
    cudaFree(b->d_dones);
    cudaFree(b->d_sub);
    cudaFree(b->d_bsum);
    cudaFree(b->d_prefix);
    cudaFree(b->d_wraw);
    cudaFree(b->d_maxp);
    cudaFree(b->d_status);
    cudaFree(b->d_done);
    delete b;
}

// re-sums blocks [first, first + n) (their sub-blocks, then the blocks)
void resum_blocks(per_buffer *b, long long first, long long n, cudaStream_t s)
{
    const long long nb = blocks_for(b->size);
    if (first + n > nb) n = nb - first;
    if (n <= 0) return;
    const long long subs = n * kSubs;
    sub_sum_kernel<<<(unsigned)((subs + kWarpsPerCta - 1) / kWarpsPerCta), kWarpsPerCta * 32, 0, s>>>(
        b->d_prio, b->size, first * kSubs, subs, nullptr, b->d_sub);
    block_sum_kernel<<<(unsigned)((n + kWarpsPerCta - 1) / kWarpsPerCta), kWarpsPerCta * 32, 0, s>>>(
        b->d_sub, b->size, first, n, nullptr, b->d_bsum);
}

int rebuild_prefix(per_buffer *b, cudaStream_t s)
{
    const long long nb = blocks_for(b->size);
    if (nb <= kStagedBlocks)
        top_scan_kernel<true><<<1, kScanThreads, nb * sizeof(double), s>>>(b->d_bsum, nb, b->d_prefix, b->d_maxp);
    else
        top_scan_kernel<false><<<1, kScanThreads, 0, s>>>(b->d_bsum, nb, b->d_prefix, b->d_maxp);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ROLLOUT_OK : cuda_err(e, "replay prefix");
}

int copy(void *dst, const void *src, size_t bytes, cudaStream_t s)
{
    if (!bytes) return ROLLOUT_OK;
    const cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, s);
    return e == cudaSuccess ? ROLLOUT_OK : cuda_err(e, "replay insert copy");
}

}  // namespace

extern "C" {

int per_create(long long capacity, int state_dim, per_buffer **out)
{
    clear_error();
    if (!out) return set_error(ROLLOUT_ERR_INVALID, "null argument");
    if (capacity < 1 || capacity >= (1ll << 31)) return set_error(ROLLOUT_ERR_INVALID, "capacity must be in [1, 2^31)");
    if (state_dim < 1 || state_dim > kMaxDim) return set_error(ROLLOUT_ERR_INVALID, "state_dim must be in [1, 4096]");
    per_buffer *b = new (std::nothrow) per_buffer();
    if (!b) return set_error(ROLLOUT_ERR_NOMEM, "host allocation failed");
    b->capacity = capacity;
    b->dim = state_dim;
    b->n_alloc_blocks = blocks_for(capacity);
    const size_t slots = (size_t)b->n_alloc_blocks * kBlock;   // the priority array covers whole blocks
    const size_t rows = (size_t)capacity * state_dim;
    cudaError_t e;
    if ((e = cudaMalloc(&b->d_states, rows * 4)) != cudaSuccess || (e = cudaMalloc(&b->d_next, rows * 4)) != cudaSuccess ||
        (e = cudaMalloc(&b->d_rewards, capacity * 4)) != cudaSuccess ||
        (e = cudaMalloc(&b->d_actions, capacity * 4)) != cudaSuccess ||
        (e = cudaMalloc(&b->d_dones, capacity)) != cudaSuccess || (e = cudaMalloc(&b->d_prio, slots * 4)) != cudaSuccess ||
        (e = cudaMalloc(&b->d_owner, capacity * 4)) != cudaSuccess ||
        (e = cudaMalloc(&b->d_sub, b->n_alloc_blocks * kSubs * 8)) != cudaSuccess ||
        (e = cudaMalloc(&b->d_bsum, b->n_alloc_blocks * 8)) != cudaSuccess ||
        (e = cudaMalloc(&b->d_prefix, (b->n_alloc_blocks + 1) * 8)) != cudaSuccess ||
        (e = cudaMalloc(&b->d_wraw, kMaxBatch * 4)) != cudaSuccess || (e = cudaMalloc(&b->d_maxp, 8)) != cudaSuccess ||
        (e = cudaMalloc(&b->d_status, 4)) != cudaSuccess || (e = cudaMalloc(&b->d_done, 4)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(top_scan_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kStagedBlocks * (int)sizeof(double))) != cudaSuccess) {
        free_buffer(b);
        return cuda_err(e, "cudaMalloc(replay buffer)");
    }
    const float one[2] = {1.f, 1.f};
    if ((e = cudaMemset(b->d_prio, 0, slots * 4)) != cudaSuccess ||
        (e = cudaMemset(b->d_owner, 0xFF, capacity * 4)) != cudaSuccess ||
        (e = cudaMemset(b->d_sub, 0, b->n_alloc_blocks * kSubs * 8)) != cudaSuccess ||
        (e = cudaMemset(b->d_bsum, 0, b->n_alloc_blocks * 8)) != cudaSuccess ||
        (e = cudaMemset(b->d_prefix, 0, (b->n_alloc_blocks + 1) * 8)) != cudaSuccess ||
        (e = cudaMemset(b->d_status, 0, 4)) != cudaSuccess || (e = cudaMemset(b->d_done, 0, 4)) != cudaSuccess ||
        (e = cudaMemcpy(b->d_maxp, one, 8, cudaMemcpyHostToDevice)) != cudaSuccess ||
        (e = cudaDeviceSynchronize()) != cudaSuccess) {
        free_buffer(b);
        return cuda_err(e, "replay buffer initialisation");
    }
    *out = b;
    return ROLLOUT_OK;
}

int per_insert(per_buffer *b, const float *states, const float *next_states, const int32_t *actions,
               const float *rewards, const uint8_t *dones, long long count, void *stream)
{
    clear_error();
    if (!b || !states || !next_states || !actions || !rewards || !dones)
        return set_error(ROLLOUT_ERR_INVALID, "null argument");
    if (count < 0) return set_error(ROLLOUT_ERR_INVALID, "count must be >= 0");
    if (count == 0) return ROLLOUT_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const long long C = b->capacity, D = b->dim;
    const long long skip = count > C ? count - C : 0, n = count - skip;   // the survivors
    const long long start = (b->cursor + skip) % C;
    const long long n1 = n < C - start ? n : C - start, n2 = n - n1;
    const long long seg_dst[2] = {start, 0}, seg_src[2] = {skip, skip + n1}, seg_n[2] = {n1, n2};
    int rc;
    for (int g = 0; g < 2; ++g) {
        const long long d = seg_dst[g], o = seg_src[g], m = seg_n[g];
        if (!m) continue;
        if ((rc = copy(b->d_states + d * D, states + o * D, (size_t)m * D * 4, s)) ||
            (rc = copy(b->d_next + d * D, next_states + o * D, (size_t)m * D * 4, s)) ||
            (rc = copy(b->d_actions + d, actions + o, (size_t)m * 4, s)) ||
            (rc = copy(b->d_rewards + d, rewards + o, (size_t)m * 4, s)) ||
            (rc = copy(b->d_dones + d, dones + o, (size_t)m, s)))
            return rc;
        const long long grid = (m + 255) / 256;
        fill_kernel<<<(unsigned)(grid < 1216 ? grid : 1216), 256, 0, s>>>(b->d_prio, d, m, b->d_maxp);
    }
    b->size = b->size + count < C ? b->size + count : C;
    b->cursor = (b->cursor + count) % C;
    b->last_stream = s;
    // re-sum the blocks written (while the ring is not full these are also all
    // the blocks whose share of [0, size) changed), then the prefix
    for (int g = 0; g < 2; ++g) {
        if (!seg_n[g]) continue;
        const long long f = seg_dst[g] / kBlock, l = (seg_dst[g] + seg_n[g] - 1) / kBlock;
        resum_blocks(b, f, l - f + 1, s);
    }
    return rebuild_prefix(b, s);
}

int per_sample(per_buffer *b, int batch, float beta, uint64_t seed, uint64_t offset, int32_t *indices,
               float *is_weights, float *states, float *next_states, int32_t *actions, float *rewards, uint8_t *dones,
               void *stream)
{
    clear_error();
    if (!b || !indices || !is_weights) return set_error(ROLLOUT_ERR_INVALID, "null argument");
    if (batch < 1 || batch > kMaxBatch) return set_error(ROLLOUT_ERR_INVALID, "batch must be in [1, 65536]");
    if (!(beta >= 0.f) || !isfinite(beta)) return set_error(ROLLOUT_ERR_INVALID, "beta must be finite and >= 0");
    if (b->size == 0) return set_error(ROLLOUT_ERR_INVALID, "the buffer is empty");
    cudaStream_t s = (cudaStream_t)stream;
    SampleArgs a{};
    a.prio = b->d_prio;
    a.states = b->d_states;
    a.next_states = b->d_next;
    a.rewards = b->d_rewards;
    a.actions = b->d_actions;
    a.dones = b->d_dones;
    a.prefix = b->d_prefix;
    a.sub = b->d_sub;
    a.size = b->size;
    a.nb = blocks_for(b->size);
    a.dim = b->dim;
    a.batch = batch;
    a.beta = beta;
    a.seed = seed;
    a.offset = offset;
    a.o_idx = indices;
    a.o_wraw = b->d_wraw;
    a.o_w = is_weights;
    a.done = b->d_done;
    a.o_states = states;
    a.o_next = next_states;
    a.o_rewards = rewards;
    a.o_actions = actions;
    a.o_dones = dones;
    a.status = b->d_status;
    sample_kernel<<<(batch + kSampleWarps - 1) / kSampleWarps, kSampleWarps * 32, 0, s>>>(a);
    b->last_stream = s;
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ROLLOUT_OK : cuda_err(e, "replay sample launch");
}

int per_update_priorities(per_buffer *b, const int32_t *indices, const float *td_errors, int batch, float alpha,
                          float eps, void *stream)
{
    clear_error();
    if (!b || !indices || !td_errors) return set_error(ROLLOUT_ERR_INVALID, "null argument");
    if (batch < 1 || batch > kMaxBatch) return set_error(ROLLOUT_ERR_INVALID, "batch must be in [1, 65536]");
    if (!(alpha >= 0.f) || !isfinite(alpha) || !(eps >= 0.f) || !isfinite(eps))
        return set_error(ROLLOUT_ERR_INVALID, "alpha and eps must be finite and >= 0");
    cudaStream_t s = (cudaStream_t)stream;
    const int grid = (batch + 255) / 256, grid64 = (batch + kFp64Threads - 1) / kFp64Threads;
    claim_kernel<<<grid, 256, 0, s>>>(indices, batch, b->size, b->d_owner, b->d_status);
    write_kernel<<<grid64, kFp64Threads, 0, s>>>(indices, td_errors, batch, b->size, (double)alpha, eps, b->d_owner,
                                                 b->d_prio, b->d_maxp);
    sub_sum_kernel<<<(batch + kWarpsPerCta - 1) / kWarpsPerCta, kWarpsPerCta * 32, 0, s>>>(b->d_prio, b->size, 0,
                                                                                          batch, indices, b->d_sub);
    block_sum_kernel<<<(batch + kWarpsPerCta - 1) / kWarpsPerCta, kWarpsPerCta * 32, 0, s>>>(b->d_sub, b->size, 0,
                                                                                            batch, indices, b->d_bsum);
    b->last_stream = s;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_err(e, "replay update launch");
    return rebuild_prefix(b, s);
}

int per_size(per_buffer *b, long long *size, long long *cursor)
{
    clear_error();
    if (!b) return set_error(ROLLOUT_ERR_INVALID, "null buffer");
    if (size) *size = b->size;
    if (cursor) *cursor = b->cursor;
    return ROLLOUT_OK;
}

int per_read(per_buffer *b, float *priorities, float *max_priority, void *stream)
{
    clear_error();
    if (!b) return set_error(ROLLOUT_ERR_INVALID, "null buffer");
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaSuccess;
    if (priorities) e = cudaMemcpyAsync(priorities, b->d_prio, b->capacity * 4, cudaMemcpyDefault, s);
    if (e == cudaSuccess && max_priority) e = cudaMemcpyAsync(max_priority, b->d_maxp, 4, cudaMemcpyDefault, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e == cudaSuccess ? ROLLOUT_OK : cuda_err(e, "replay read");
}

int per_status(per_buffer *b)
{
    clear_error();
    if (!b) return set_error(ROLLOUT_ERR_INVALID, "null buffer");
    cudaError_t e = cudaStreamSynchronize(b->last_stream);
    if (e != cudaSuccess) return cuda_err(e, "cudaStreamSynchronize");
    int st = 0;
    if ((e = cudaMemcpy(&st, b->d_status, 4, cudaMemcpyDeviceToHost)) != cudaSuccess ||
        (e = cudaMemset(b->d_status, 0, 4)) != cudaSuccess)
        return cuda_err(e, "status read");
    return st;
}

void per_destroy(per_buffer *b)
{
    if (!b) return;
    cudaDeviceSynchronize();
    free_buffer(b);
}

}  // extern "C"
