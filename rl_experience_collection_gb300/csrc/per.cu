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
// block of 16 sub-blocks (2048 slots), and the prefix over the blocks.  An
// insert re-sums the sub-blocks and blocks it wrote, an update those of the
// slots it named, and each then rebuilds the prefix (one CTA; a two-level
// chain, so that it never decreases and a block of zero sum is an empty
// interval).  A sampling call reads no whole array: one warp per sample
// searches the block prefix 32 ways at a time, then the block's 16 sub-sums,
// then the sub-block's 128 priorities, with warp-wide running sums.  GB300's
// double-precision rate is low, so the levels keep the double additions per
// sample to about 600.  Only positive slots can be picked; where rounding puts
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
constexpr int kSubs = 16;               // sub-blocks per block
constexpr int kBlock = kSub * kSubs;    // priorities per block
constexpr int kScanThreads = 1024;      // 32 groups of 32 chunks
constexpr int kWarpsPerCta = 8;
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

// Block sums from their sub-sums, in sub-block order, one thread each: block
// first + t, or the block of slots[t].
__global__ void block_sum_kernel(const double *__restrict__ sub, long long size, long long first, long long n,
                                 const int32_t *__restrict__ slots, double *__restrict__ bsum)
{
    const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (t >= n) return;
    long long b;
    if (slots) {
        const int32_t i = slots[t];
        if (i < 0 || i >= size) return;
        b = i / kBlock;
    } else {
        b = first + t;
    }
    double s = 0.0;
#pragma unroll
    for (int j = 0; j < kSubs; ++j) s += sub[b * kSubs + j];
    bsum[b] = s;
}

// prefix[b] = the block sums before b, prefix[nb] = total.  Thread t owns a
// contiguous chunk of blocks (sum S_t, accumulated from zero in order); the 32
// chunks of group g are chained by one lane (H[t+1] = H[t] + S_t, group total
// T_g = H[last] + S_last) and the groups by thread 0 (K[g+1] = K[g] + T_g);
// then prefix[b] = K[g] + (H[t] + the chunk's blocks before b).  Each step of a
// chain adds exactly the sum the level below formed, so rounding (monotone)
// never makes the prefix decrease, and prefix[b+1] == prefix[b] whenever block
// b sums to zero, across chunk and group boundaries too.
__global__ void __launch_bounds__(kScanThreads) top_scan_kernel(const double *__restrict__ bsum, long long nb,
                                                                double *__restrict__ prefix)
{
    __shared__ double S[kScanThreads], H[kScanThreads], T[32], K[33];
    const int t = threadIdx.x, g = t >> 5;
    const long long chunk = (nb + kScanThreads - 1) / kScanThreads;
    const long long lo = min(nb, (long long)t * chunk), hi = min(nb, lo + chunk);
    double s = 0.0;
    for (long long b = lo; b < hi; ++b) s += bsum[b];
    S[t] = s;
    __syncthreads();
    if ((t & 31) == 0) {
        double h = 0.0;
        for (int i = 0; i < 32; ++i) {
            H[t + i] = h;
            h += S[t + i];
        }
        T[g] = h;
    }
    __syncthreads();
    if (t == 0) {
        double k = 0.0;
        for (int i = 0; i < 32; ++i) {
            K[i] = k;
            k += T[i];
        }
        K[32] = k;
    }
    __syncthreads();
    double part = 0.0;
    for (long long b = lo; b < hi; ++b) {
        prefix[b] = K[g] + (H[t] + part);
        part += bsum[b];
    }
    if (t == 0) prefix[nb] = K[32];
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
    double beta;
    uint64_t seed, offset;
    int32_t *o_idx;
    double *o_wraw;
    float *o_states, *o_next, *o_rewards;
    int32_t *o_actions;
    uint8_t *o_dones;
    int *status;
};

// one level of the in-block search: x (>= 0) is this lane's share, `before0`
// the running total ahead of lane 0.  Returns the first lane whose positive
// share takes the running total past t, else the last lane with a positive
// share (-1 if none), and sets *ahead to the running total before that lane.
__device__ __forceinline__ int level_pick(double x, double before0, double t, int lane, double *ahead)
{
    double inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    double excl = __shfl_up_sync(0xffffffffu, inc, 1);
    if (lane == 0) excl = 0.0;
    const double before = before0 + excl;
    const unsigned hit = __ballot_sync(0xffffffffu, x > 0.0 && before + x > t);
    const unsigned pos = __ballot_sync(0xffffffffu, x > 0.0);
    const int l = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
    *ahead = __shfl_sync(0xffffffffu, before, l < 0 ? 0 : l);
    return l;
}

// one warp per sample
__global__ void __launch_bounds__(kWarpsPerCta * 32) sample_kernel(SampleArgs a)
{
    const int k = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (k >= a.batch) return;                                  // warp-uniform
    const double total = a.prefix[a.nb];
    long long pick = -1;
    if (total > 0.0) {
        const double u = (double)(splitmix64_output(a.seed, a.offset + (uint64_t)k) >> 11) * 0x1p-53;
        double t = u * total;
        if (t >= total) t = nextafter(total, 0.0);             // u * total can round up to total
        // the block b with prefix[b] <= t < prefix[b+1], 32 ways at a time (the
        // invariant holds at the start: prefix[0] = 0 and prefix[nb] = total)
        long long lo = 0, hi = a.nb;
        while (hi - lo > 1) {
            const long long span = hi - lo;
            const long long q = lo + ((long long)(lane + 1) * span) / 32;    // q of lane 31 is hi
            const unsigned below = __ballot_sync(0xffffffffu, a.prefix[q] <= t);
            const int c = __popc(below);                        // lanes 0..c-1 are at or below t
            const long long qc = __shfl_sync(0xffffffffu, q, min(c, 31));
            const long long qp = __shfl_sync(0xffffffffu, q, max(c - 1, 0));
            if (c > 0) lo = qp;
            hi = qc;
        }
        lo = min(lo, a.nb - 1);                                 // holds already: prefix[nb] = total > t
        // its sub-blocks (lanes 0-15), then the chosen sub-block's 128 slots (4 a lane)
        double ahead = 0.0;
        const double xs = lane < kSubs ? a.sub[lo * kSubs + lane] : 0.0;
        const int sl = level_pick(xs, a.prefix[lo], t, lane, &ahead);
        if (sl >= 0) {
            const long long e0 = (lo * kSubs + sl) * kSub + lane * 4;
            const float4 v = reinterpret_cast<const float4 *>(a.prio + e0)[0];
            float p[4] = {v.x, v.y, v.z, v.w};
            double l[4];
            double run = 0.0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (e0 + q >= a.size) p[q] = 0.f;
                run += (double)p[q];
                l[q] = run;
            }
            double before = 0.0;
            const int el = level_pick(l[3], ahead, t, lane, &before);
            if (el >= 0) {
                // within the lane: the first positive slot past t, else its last positive slot
                int first = -1, lastq = -1;
#pragma unroll
                for (int q = 3; q >= 0; --q)
                    if (p[q] > 0.f) {
                        if (before + l[q] > t) first = q;
                        if (lastq < 0) lastq = q;
                    }
                const int qq = __shfl_sync(0xffffffffu, first >= 0 ? first : lastq, el);
                pick = (lo * kSubs + sl) * kSub + el * 4 + qq;
            }
        }
    }
    double w = 0.0;
    if (pick < 0) {                                             // no positive priority
        if (lane == 0) *a.status = ROLLOUT_ERR_RANGE;
        pick = 0;
    } else {
        w = pow((double)a.size * (double)a.prio[pick] / total, -a.beta);
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

// w_k / max_j w_j (max over the batch); all zero when every sample failed
__global__ void __launch_bounds__(1024) normalize_kernel(const double *__restrict__ wraw, int batch,
                                                         float *__restrict__ w)
{
    __shared__ double ws[32];
    double m = 0.0;
    for (int k = threadIdx.x; k < batch; k += blockDim.x) m = fmax(m, wraw[k]);
    for (int o = 16; o; o >>= 1) m = fmax(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = ws[threadIdx.x];
        for (int o = 16; o; o >>= 1) m = fmax(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (threadIdx.x == 0) ws[0] = m;
    }
    __syncthreads();
    m = ws[0];
    for (int k = threadIdx.x; k < batch; k += blockDim.x) w[k] = m > 0.0 ? (float)(wraw[k] / m) : 0.f;
}

// the update, first launch: the last entry naming a slot owns it; the maximum
// priority before the call is kept for the +inf clamp
__global__ void claim_kernel(const int32_t *__restrict__ idx, int batch, long long size, int32_t *__restrict__ owner,
                             float *__restrict__ maxp, int *__restrict__ status)
{
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k == 0) maxp[1] = maxp[0];
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
    const float d = td[k];
    float v;
    if (isnan(d)) {
        v = eps;
    } else {
        v = (float)(pow(fabs((double)d), alpha) + (double)eps);
        if (isinf(v)) v = maxp[1];
    }
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
    double *d_sub = nullptr, *d_bsum = nullptr, *d_prefix = nullptr, *d_wraw = nullptr;
    float *d_maxp = nullptr;     // [0] the running maximum priority, [1] its value before the last update
    int *d_status = nullptr;
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
    block_sum_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(b->d_sub, b->size, first, n, nullptr, b->d_bsum);
}

int rebuild_prefix(per_buffer *b, cudaStream_t s)
{
    top_scan_kernel<<<1, kScanThreads, 0, s>>>(b->d_bsum, blocks_for(b->size), b->d_prefix);
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
        (e = cudaMalloc(&b->d_wraw, kMaxBatch * 8)) != cudaSuccess || (e = cudaMalloc(&b->d_maxp, 8)) != cudaSuccess ||
        (e = cudaMalloc(&b->d_status, 4)) != cudaSuccess) {
        free_buffer(b);
        return cuda_err(e, "cudaMalloc(replay buffer)");
    }
    const float one[2] = {1.f, 1.f};
    if ((e = cudaMemset(b->d_prio, 0, slots * 4)) != cudaSuccess ||
        (e = cudaMemset(b->d_owner, 0xFF, capacity * 4)) != cudaSuccess ||
        (e = cudaMemset(b->d_sub, 0, b->n_alloc_blocks * kSubs * 8)) != cudaSuccess ||
        (e = cudaMemset(b->d_bsum, 0, b->n_alloc_blocks * 8)) != cudaSuccess ||
        (e = cudaMemset(b->d_prefix, 0, (b->n_alloc_blocks + 1) * 8)) != cudaSuccess ||
        (e = cudaMemset(b->d_status, 0, 4)) != cudaSuccess ||
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
    a.o_states = states;
    a.o_next = next_states;
    a.o_rewards = rewards;
    a.o_actions = actions;
    a.o_dones = dones;
    a.status = b->d_status;
    sample_kernel<<<(batch + kWarpsPerCta - 1) / kWarpsPerCta, kWarpsPerCta * 32, 0, s>>>(a);
    normalize_kernel<<<1, 1024, 0, s>>>(b->d_wraw, batch, is_weights);
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
    const int grid = (batch + 255) / 256;
    claim_kernel<<<grid, 256, 0, s>>>(indices, batch, b->size, b->d_owner, b->d_maxp, b->d_status);
    write_kernel<<<grid, 256, 0, s>>>(indices, td_errors, batch, b->size, (double)alpha, eps, b->d_owner, b->d_prio,
                                      b->d_maxp);
    sub_sum_kernel<<<(batch + kWarpsPerCta - 1) / kWarpsPerCta, kWarpsPerCta * 32, 0, s>>>(b->d_prio, b->size, 0,
                                                                                          batch, indices, b->d_sub);
    block_sum_kernel<<<grid, 256, 0, s>>>(b->d_sub, b->size, 0, batch, indices, b->d_bsum);
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
