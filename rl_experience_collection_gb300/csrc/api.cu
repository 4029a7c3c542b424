// api.cu -- the C ABI (include/rollout.h): argument checks, weight
// conversion, and the stream-ordered launch of the phases.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <new>
#include <vector>

#include "internal.cuh"
#include "ppo_gemm.cuh"
#include "umma_path.cuh"

using namespace rl;

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(e == cudaErrorMemoryAllocation ? ROLLOUT_ERR_NOMEM : ROLLOUT_ERR_CUDA, "%s: %s", what,
                cudaGetErrorString(e));
}

// kernels of one run, timed when rollout_set_timing is on: rollout, state rows, value, GAE
constexpr int kTimedKernels = 4;

// points of a run after which outputs are final: the rollout (actions, log-probs,
// dones), the state rows, the value kernel (values, rewards), GAE (advantages, returns)
enum RunPoint { kAfterRollout = 0, kAfterStates, kAfterValue, kAfterGae, kRunPoints };

// streams rollout_run_host spreads its device-to-host copies over (the copy engines
// work on several at once)
constexpr int kCopyStreams = 4;

}  // namespace

struct rollout_handle {
    rollout_dims dims;
    int device = 0;
    int critic_w[kCriticLayers + 1] = {};
    size_t n_weights = 0;
    // float32 path
    float *d_actor_packed = nullptr;   // phase-1 actor (SIMT layout)
    float *d_simt = nullptr;           // transposed critic/curiosity + biases
    SimtWeights simt{};
    // tensor-core path
    UmmaWeights umma{};
    void *d_umma = nullptr;
    // per-CTA activation scratch of the generic value kernel (tf32 / widened critic)
    uint8_t *d_scratch = nullptr;
    long long scratch_per_cta = 0;
    int scratch_ctas = 0;
    // bf16 rollout: feature rows padded to kFPad floats and a tensor map over them
    float *d_fpad = nullptr;
    CUtensorMap fmap{};   // the type carries its own alignment
    // environment
    uint32_t *d_div_low = nullptr;
    int *d_status = nullptr;
    cudaStream_t last_stream = nullptr;
    // optional per-kernel timing
    bool timing = false, timed_run = false;
    // rollout_test_stall: runs launch the value kernel's stalling test build
    bool test_stall = false;
    // rollout_test_activations: runs launch the kernels' dump builds
    float *dump = nullptr;
    int dump_episodes = 0;
    // rollout_forward: the packed float32 weights and the forward pass's
    // buffers (grown on demand)
    float *d_wf32 = nullptr;
    uint8_t *d_fwd = nullptr;
    size_t fwd_bytes = 0;
    cudaEvent_t ev[kTimedKernels + 1] = {};
    // rollout_run_host: device copies of the inputs and outputs (one allocation,
    // grown on demand), the copy streams and their events
    uint8_t *d_stage = nullptr;
    size_t stage_bytes = 0;
    cudaStream_t copy_stream[kCopyStreams] = {};
    cudaEvent_t point_ev[kRunPoints] = {};
    cudaEvent_t copy_done[kCopyStreams] = {};
    // rollout_set_weights_device: per region of the converted device weights,
    // the source of each element in the packed float32 vector
    struct Region {
        uint8_t *dev;
        const int32_t *map;
        long long n;
        int elem;
    } repack[4] = {};
    int n_repack = 0;
    int32_t *d_maps = nullptr;
};

namespace {

constexpr int kA1 = 0, kB1 = kA1 + kState * kActorH1, kA2 = kB1 + kActorH1, kB2 = kA2 + kActorH1 * kActorH2,
              kA3 = kB2 + kActorH2, kB3 = kA3 + kActorH2 * 48, kActorPacked = kB3 + 48;

int check_dims(const rollout_dims *d)
{
    if (d->n_market != kMarket || d->n_actions != kActions || d->actor_h1 != kActorH1 ||
        d->actor_h2 != kActorH2 || d->cur_h != kCurH)
        return fail(ROLLOUT_ERR_UNSUPPORTED, "unsupported network shape (need 51 market features, 45 actions, "
                    "actor 128/64, curiosity 64)");
    if (d->critic_nh != 5) return fail(ROLLOUT_ERR_UNSUPPORTED, "critic_nh must be 5");
    static const int std_h[5] = {512, 384, 256, 128, 64}, wide_h[5] = {1024, 768, 512, 256, 128};
    bool is_std = true, is_wide = true;
    for (int i = 0; i < 5; ++i) {
        is_std &= d->critic_h[i] == std_h[i];
        is_wide &= d->critic_h[i] == wide_h[i];
    }
    if (!is_std && !is_wide)
        return fail(ROLLOUT_ERR_UNSUPPORTED, "critic widths must be 512,384,256,128,64 or 1024,768,512,256,128");
    if (d->dtype != ROLLOUT_FP32 && d->dtype != ROLLOUT_TF32 && d->dtype != ROLLOUT_BF16)
        return fail(ROLLOUT_ERR_UNSUPPORTED, "unknown dtype %d", d->dtype);
    if (d->n_bars < 2) return fail(ROLLOUT_ERR_INVALID, "n_bars must be >= 2");
    if (d->div_window < 1 || d->div_window > 31)
        return fail(ROLLOUT_ERR_UNSUPPORTED, "div_window must be in [1, 31]");
    if (d->max_hold < 1) return fail(ROLLOUT_ERR_INVALID, "max_hold must be >= 1");
    const float fs[] = {d->barrier, d->pt_scale, d->sl_scale, d->div_thresh, d->div_penalty, d->cur_coef,
                        d->risk_coef, d->tx_base, d->spread};
    for (float f : fs)
        if (!isfinite(f)) return fail(ROLLOUT_ERR_INVALID, "environment constants must be finite");
    return ROLLOUT_OK;
}

// offsets of the packed host buffer (rollout.h: actor, critic, curiosity)
struct HostLayout {
    size_t a_w[3], a_b[3], c_w[kCriticLayers], c_b[kCriticLayers], q_w[2], q_b[2], total;
    int a_in[3], a_out[3], c_in[kCriticLayers], c_out[kCriticLayers], q_in[2], q_out[2];
};

HostLayout host_layout(const rollout_dims &d)
{
    HostLayout lo{};
    size_t off = 0;
    const int ain[3] = {kState, kActorH1, kActorH2}, aout[3] = {kActorH1, kActorH2, kActions};
    for (int l = 0; l < 3; ++l) {
        lo.a_in[l] = ain[l]; lo.a_out[l] = aout[l];
        lo.a_w[l] = off; off += (size_t)ain[l] * aout[l];
        lo.a_b[l] = off; off += aout[l];
    }
    int prev = kState;
    for (int l = 0; l < kCriticLayers; ++l) {
        const int o = l < 5 ? d.critic_h[l] : 1;
        lo.c_in[l] = prev; lo.c_out[l] = o;
        lo.c_w[l] = off; off += (size_t)prev * o;
        lo.c_b[l] = off; off += o;
        prev = o;
    }
    const int qin[2] = {kState + kActions, kCurH}, qout[2] = {kCurH, kState};
    for (int l = 0; l < 2; ++l) {
        lo.q_in[l] = qin[l]; lo.q_out[l] = qout[l];
        lo.q_w[l] = off; off += (size_t)qin[l] * qout[l];
        lo.q_b[l] = off; off += qout[l];
    }
    lo.total = off;
    return lo;
}

void transpose_into(std::vector<float> &dst, size_t at, const float *W, int out, int in, int out_pad)
{
    for (int i = 0; i < in; ++i)
        for (int j = 0; j < out_pad; ++j) dst[at + (size_t)i * out_pad + j] = j < out ? W[(size_t)j * in + i] : 0.f;
}

// float32 path: actor packed for phase 1, critic/curiosity transposed for phase 2
struct SimtHost {
    std::vector<float> ap, sp;
    size_t offs_T[kCriticLayers], offs_b[kCriticLayers], q_T[2], q_b[2];
};

void simt_pack_host(const rollout_dims &d, const float *w, SimtHost *out)
{
    const HostLayout lo = host_layout(d);
    std::vector<float> &ap = out->ap, &sp = out->sp;
    size_t *offs_T = out->offs_T, *offs_b = out->offs_b, *q_T = out->q_T, *q_b = out->q_b;
    ap.assign(kActorPacked, 0.f);
    sp.clear();
    transpose_into(ap, kA1, w + lo.a_w[0], kActorH1, kState, kActorH1);
    memcpy(&ap[kB1], w + lo.a_b[0], sizeof(float) * kActorH1);
    transpose_into(ap, kA2, w + lo.a_w[1], kActorH2, kActorH1, kActorH2);
    memcpy(&ap[kB2], w + lo.a_b[1], sizeof(float) * kActorH2);
    transpose_into(ap, kA3, w + lo.a_w[2], kActions, kActorH2, 48);
    memcpy(&ap[kB3], w + lo.a_b[2], sizeof(float) * kActions);

    for (int l = 0; l < kCriticLayers; ++l) {
        offs_T[l] = sp.size();
        sp.resize(sp.size() + (size_t)lo.c_in[l] * lo.c_out[l]);
        transpose_into(sp, offs_T[l], w + lo.c_w[l], lo.c_out[l], lo.c_in[l], lo.c_out[l]);
        offs_b[l] = sp.size();
        sp.insert(sp.end(), w + lo.c_b[l], w + lo.c_b[l] + lo.c_out[l]);
    }
    for (int l = 0; l < 2; ++l) {
        q_T[l] = sp.size();
        sp.resize(sp.size() + (size_t)lo.q_in[l] * lo.q_out[l]);
        transpose_into(sp, q_T[l], w + lo.q_w[l], lo.q_out[l], lo.q_in[l], lo.q_out[l]);
        q_b[l] = sp.size();
        sp.insert(sp.end(), w + lo.q_b[l], w + lo.q_b[l] + lo.q_out[l]);
    }
}

int upload_simt(rollout_handle *h, const float *w)
{
    const HostLayout lo = host_layout(h->dims);
    SimtHost sh;
    simt_pack_host(h->dims, w, &sh);
    const std::vector<float> &ap = sh.ap, &sp = sh.sp;
    const size_t *offs_T = sh.offs_T, *offs_b = sh.offs_b, *q_T = sh.q_T, *q_b = sh.q_b;
    cudaError_t e;
    if (!h->d_actor_packed) {
        if ((e = dev_alloc((void **)&h->d_actor_packed, sizeof(float) * ap.size())) != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(actor)");
        if ((e = dev_alloc((void **)&h->d_simt, sizeof(float) * sp.size())) != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(critic)");
    }
    if ((e = cudaMemcpy(h->d_actor_packed, ap.data(), sizeof(float) * ap.size(), cudaMemcpyHostToDevice)) !=
        cudaSuccess)
        return cuda_fail(e, "cudaMemcpy(actor)");
    if ((e = cudaMemcpy(h->d_simt, sp.data(), sizeof(float) * sp.size(), cudaMemcpyHostToDevice)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy(critic)");
    for (int l = 0; l < kCriticLayers; ++l) {
        h->simt.critic_T[l] = h->d_simt + offs_T[l];
        h->simt.critic_b[l] = h->d_simt + offs_b[l];
        h->simt.critic_w[l] = lo.c_in[l];
    }
    h->simt.critic_w[kCriticLayers] = 1;
    h->simt.cur0_T = h->d_simt + q_T[0];
    h->simt.cur0_b = h->d_simt + q_b[0];
    h->simt.cur1_T = h->d_simt + q_T[1];
    h->simt.cur1_b = h->d_simt + q_b[1];
    h->simt.actor = h->d_actor_packed;
    return ROLLOUT_OK;
}

// exact diversity decision per histogram (c0, c1, c2), c_k < 32
int upload_div_table(rollout_handle *h)
{
    std::vector<uint32_t> bits(1024, 0u);
    for (int c0 = 0; c0 < 32; ++c0)
        for (int c1 = 0; c1 < 32; ++c1)
            for (int c2 = 0; c2 < 32; ++c2) {
                const int n = c0 + c1 + c2;
                if (n == 0 || n > h->dims.div_window) continue;
                double H = 0.0;
                const int c[3] = {c0, c1, c2};
                for (int k = 0; k < 3; ++k)
                    if (c[k] > 0) {
                        const double p = (double)c[k] / (double)n;
                        H -= p * log2(p);
                    }
                if (H < (double)h->dims.div_thresh) {
                    const int bit = c0 * 1024 + c1 * 32 + c2;
                    bits[bit >> 5] |= 1u << (bit & 31);
                }
            }
    cudaError_t e;
    if (!h->d_div_low && (e = dev_alloc((void **)&h->d_div_low, bits.size() * 4)) != cudaSuccess)
        return cuda_fail(e, "cudaMalloc(div table)");
    if ((e = cudaMemcpy(h->d_div_low, bits.data(), bits.size() * 4, cudaMemcpyHostToDevice)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy(div table)");
    return ROLLOUT_OK;
}

UmmaHostLayout umma_layout(const HostLayout &lo)
{
    UmmaHostLayout ul{};
    ul.n_critic = kCriticLayers;
    for (int l = 0; l < 3; ++l) { ul.a_w[l] = lo.a_w[l]; ul.a_b[l] = lo.a_b[l]; }
    for (int l = 0; l < kCriticLayers; ++l) {
        ul.c_w[l] = lo.c_w[l]; ul.c_b[l] = lo.c_b[l]; ul.c_in[l] = lo.c_in[l]; ul.c_out[l] = lo.c_out[l];
    }
    for (int l = 0; l < 2; ++l) { ul.q_w[l] = lo.q_w[l]; ul.q_b[l] = lo.q_b[l]; }
    return ul;
}

int upload_weights(rollout_handle *h, const float *w)
{
    const HostLayout lo = host_layout(h->dims);
    for (size_t i = 0; i < lo.total; ++i)
        if (!isfinite(w[i])) return fail(ROLLOUT_ERR_INVALID, "weight %zu is not finite", i);
    cudaError_t ew;
    if (!h->d_wf32 && (ew = dev_alloc((void **)&h->d_wf32, lo.total * 4)) != cudaSuccess)
        return cuda_fail(ew, "cudaMalloc(float32 weights)");
    if ((ew = cudaMemcpy(h->d_wf32, w, lo.total * 4, cudaMemcpyHostToDevice)) != cudaSuccess)
        return cuda_fail(ew, "cudaMemcpy(float32 weights)");
    if (h->dims.dtype == ROLLOUT_FP32) return upload_simt(h, w);
    int rc = umma_upload(&h->umma, &h->d_umma, h->dims.dtype == ROLLOUT_BF16, w, umma_layout(lo), g_err, sizeof(g_err));
    if (rc) return rc;
    if (value_needs_scratch(h->umma) && !h->d_scratch) {
        int sms = 0;
        cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, h->device);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        h->scratch_per_cta = value_generic_scratch_per_cta(h->umma);
        h->scratch_ctas = sms;
        if ((e = dev_alloc((void **)&h->d_scratch, (size_t)h->scratch_per_cta * sms)) != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(value scratch)");
    }
    return ROLLOUT_OK;
}

// ---------------------------------------------------------------------------
// Device-side weight refresh.  The host packers only copy weights into place
// or round them once (bf16 or tf32), so each converted element is a function
// of one weight.  Once per handle, three probe vectors go through the same
// packer as the real weights: two whose values are exact in bf16, tf32 and
// float32 give each element the index of its source (13 bits each, as
// mantissa and exponent), and a third (1 + 2^-20, exact in neither reduced
// format) tells the rounded elements from the copied ones.  The resulting map
// is a gather that rounds as the host packer does.

// 13 bits as (1 + m/128) 2^(e-32), m < 128, e < 64
float probe_value(uint32_t bits)
{
    return ldexpf(1.f + (float)(bits & 0x7Fu) / 128.f, (int)((bits >> 7) & 0x3Fu) - 32);
}

long long probe_bits(float v)
{
    int e = 0;
    const float f = frexpf(v, &e);                 // v = f 2^e, f in [0.5, 1)
    return ((long long)(e + 31) << 7) | (long long)lrintf((2.f * f - 1.f) * 128.f);
}

float element(const uint8_t *base, long long s, int elem)
{
    uint32_t u = 0;
    if (elem == 2) {
        uint16_t b;
        memcpy(&b, base + (size_t)s * 2, 2);
        u = (uint32_t)b << 16;
    } else {
        memcpy(&u, base + (size_t)s * 4, 4);
    }
    float f;
    memcpy(&f, &u, 4);
    return f;
}

// one region of converted weights in a host image, and where it lives on the device
struct ProbeRegion {
    const uint8_t *host;
    long long n;
    int elem;
    uint8_t *dev;
};

int build_repack(rollout_handle *h)
{
    const HostLayout lo = host_layout(h->dims);
    const size_t nw = lo.total;
    if (nw + 1 >= ((size_t)1 << 26)) return fail(ROLLOUT_ERR_UNSUPPORTED, "too many weights for the refresh map");
    constexpr float kRoundProbe = 1.f + 0x1p-20f;
    std::vector<float> probe(nw);
    std::vector<ProbeRegion> reg[3];
    SimtHost sh[3];
    UmmaHostImage im[3];
    for (int k = 0; k < 3; ++k) {
        for (size_t i = 0; i < nw; ++i) {
            const uint32_t j = (uint32_t)i + 1;    // 0 marks padding
            probe[i] = k == 0 ? probe_value(j & 0x1FFFu) : k == 1 ? probe_value(j >> 13) : kRoundProbe;
        }
        if (h->dims.dtype == ROLLOUT_FP32) {
            simt_pack_host(h->dims, probe.data(), &sh[k]);
            reg[k].push_back({(const uint8_t *)sh[k].ap.data(), (long long)sh[k].ap.size(), 4, (uint8_t *)h->d_actor_packed});
            reg[k].push_back({(const uint8_t *)sh[k].sp.data(), (long long)sh[k].sp.size(), 4, (uint8_t *)h->d_simt});
        } else {
            UmmaWeights tables = h->umma;
            umma_pack_host(&tables, h->dims.dtype == ROLLOUT_BF16, probe.data(), umma_layout(lo), &im[k]);
            for (const UmmaRegion &r : im[k].region)
                reg[k].push_back({im[k].bytes.data() + r.off, (long long)(r.bytes / r.elem), r.elem,
                                  (uint8_t *)h->d_umma + r.off});
        }
    }
    std::vector<int32_t> maps;
    std::vector<size_t> starts;
    for (size_t r = 0; r < reg[0].size(); ++r) {
        const ProbeRegion &a = reg[0][r], &b = reg[1][r], &c = reg[2][r];
        starts.push_back(maps.size());
        for (long long s = 0; s < a.n; ++s) {
            const float va = element(a.host, s, a.elem);
            if (va == 0.f) {
                maps.push_back(0);
                continue;
            }
            const long long j = probe_bits(va) | (probe_bits(element(b.host, s, b.elem)) << 13);
            if (j < 1 || j > (long long)nw)
                return fail(ROLLOUT_ERR_CUDA, "weight refresh map: element %lld of region %zu decodes to %lld", s, r, j);
            const bool rounded = element(c.host, s, c.elem) != kRoundProbe;
            maps.push_back((int32_t)j | (rounded ? (int32_t)1 << 30 : 0));
        }
    }
    cudaError_t e;
    if ((e = dev_alloc((void **)&h->d_maps, maps.size() * 4)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(weight map)");
    if ((e = cudaMemcpy(h->d_maps, maps.data(), maps.size() * 4, cudaMemcpyHostToDevice)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy(weight map)");
    h->n_repack = (int)reg[0].size();
    for (int r = 0; r < h->n_repack; ++r)
        h->repack[r] = {reg[0][r].dev, h->d_maps + starts[r], reg[0][r].n, reg[0][r].elem};
    return ROLLOUT_OK;
}

// one region of the refresh: element s takes weight map[s]-1 (0: padding, a
// zero), rounded where bit 30 says so, as the host packer rounds
__global__ void repack_kernel(const float *__restrict__ w, const int32_t *__restrict__ map, long long n, int elem,
                              int tf32, uint8_t *__restrict__ dst)
{
    for (long long s = blockIdx.x * (long long)blockDim.x + threadIdx.x; s < n; s += (long long)gridDim.x * blockDim.x) {
        const int32_t code = map[s];
        const uint32_t u = code ? __float_as_uint(w[(code & 0x3FFFFFFF) - 1]) : 0u;
        const uint32_t bf = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;     // bf16, nearest even
        if (elem == 2) {
            reinterpret_cast<uint16_t *>(dst)[s] = (uint16_t)bf;
        } else {
            const uint32_t rnd = tf32 ? ((u + 0x1000u) & 0xFFFFE000u) : (bf << 16);   // tf32: nearest, ties away
            reinterpret_cast<uint32_t *>(dst)[s] = (code & (1 << 30)) ? rnd : u;
        }
    }
}

// the padded copy of the feature matrix and the 2-D tensor map the bf16
// rollout kernel gathers its rows with ([n_bars][kFPad] f32, box kFPad x 1)
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int make_feature_map(rollout_handle *h)
{
    const size_t bytes = (size_t)h->dims.n_bars * kFPad * sizeof(float);
    cudaError_t e;
    if ((e = dev_alloc((void **)&h->d_fpad, bytes)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(padded features)");
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(ROLLOUT_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const cuuint64_t dims[2] = {(cuuint64_t)kFPad, (cuuint64_t)h->dims.n_bars};
    const cuuint64_t strides[1] = {(cuuint64_t)kFPad * sizeof(float)};
    const cuuint32_t box[2] = {(cuuint32_t)kFPad, 1};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = reinterpret_cast<EncodeTiledFn>(fn)(
        &h->fmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, h->d_fpad, dims, strides, box, elem,
        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ROLLOUT_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return ROLLOUT_OK;
}

void free_handle(rollout_handle *h)
{
    if (!h) return;
    dev_free(h->d_fpad);
    dev_free(h->d_actor_packed);
    dev_free(h->d_simt);
    dev_free(h->d_umma);
    dev_free(h->d_scratch);
    dev_free(h->d_div_low);
    dev_free(h->d_status);
    for (cudaEvent_t e : h->ev)
        if (e) cudaEventDestroy(e);
    dev_free(h->d_stage);
    for (cudaStream_t st : h->copy_stream)
        if (st) cudaStreamDestroy(st);
    for (cudaEvent_t e : h->point_ev)
        if (e) cudaEventDestroy(e);
    for (cudaEvent_t e : h->copy_done)
        if (e) cudaEventDestroy(e);
    dev_free(h->d_maps);
    dev_free(h->d_wf32);
    dev_free(h->d_fwd);
    delete h;
}

}  // namespace

// shared with the PPO trainer (ppo.cu): one error message per host thread, one shape check
namespace rl {

int set_error(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

void clear_error() { g_err[0] = 0; }

int validate_dims(const rollout_dims *d) { return check_dims(d); }

static std::atomic<long long> g_alloc_fail_at{0};   // 0: no injected failure
static std::atomic<long long> g_alloc_seen{0};      // allocations requested since the hook was set
static std::atomic<long long> g_alloc_live{0};      // allocations not yet freed

cudaError_t dev_alloc(void **p, size_t bytes)
{
    const long long k = g_alloc_fail_at.load();
    if (k > 0 && ++g_alloc_seen == k) {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    cudaError_t e = cudaMalloc(p, bytes);
    if (e == cudaSuccess) ++g_alloc_live;
    return e;
}

void dev_free(void *p)
{
    if (!p) return;
    cudaFree(p);
    --g_alloc_live;
}

}  // namespace rl

extern "C" {

const char *rollout_last_error(void) { return g_err; }

int rollout_create(const float *weights, const rollout_dims *dims, rollout_handle **out)
{
    g_err[0] = 0;
    if (!weights || !dims || !out) return fail(ROLLOUT_ERR_INVALID, "null argument");
    int rc = check_dims(dims);
    if (rc) return rc;
    rollout_handle *h = new (std::nothrow) rollout_handle();
    if (!h) return fail(ROLLOUT_ERR_NOMEM, "host allocation failed");
    h->dims = *dims;
    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) { free_handle(h); return cuda_fail(e, "cudaGetDevice"); }
    if ((e = dev_alloc((void **)&h->d_status, sizeof(int))) != cudaSuccess) { free_handle(h); return cuda_fail(e, "cudaMalloc(status)"); }
    if ((e = cudaMemset(h->d_status, 0, sizeof(int))) != cudaSuccess) { free_handle(h); return cuda_fail(e, "cudaMemset"); }
    if ((rc = upload_div_table(h)) || (rc = upload_weights(h, weights)) || (rc = build_repack(h)) ||
        (dims->dtype == ROLLOUT_BF16 && (rc = make_feature_map(h)))) {
        free_handle(h);
        return rc;
    }
    *out = h;
    return ROLLOUT_OK;
}

int rollout_set_weights(rollout_handle *h, const float *weights)
{
    g_err[0] = 0;
    if (!h || !weights) return fail(ROLLOUT_ERR_INVALID, "null argument");
    return upload_weights(h, weights);
}

int rollout_set_weights_device(rollout_handle *h, const float *weights, void *stream)
{
    g_err[0] = 0;
    if (!h || !weights) return fail(ROLLOUT_ERR_INVALID, "null argument");
    if (((uintptr_t)weights & 3u) != 0) return fail(ROLLOUT_ERR_INVALID, "weights must be 4-byte aligned");
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t ec = cudaMemcpyAsync(h->d_wf32, weights, host_layout(h->dims).total * 4, cudaMemcpyDeviceToDevice, st);
    if (ec != cudaSuccess) return cuda_fail(ec, "cudaMemcpyAsync(float32 weights)");
    for (int r = 0; r < h->n_repack; ++r) {
        const auto &g = h->repack[r];
        const long long blocks = (g.n + 255) / 256;
        repack_kernel<<<(int)(blocks < 1216 ? blocks : 1216), 256, 0, st>>>(weights, g.map, g.n, g.elem,
                                                                           h->dims.dtype == ROLLOUT_TF32, g.dev);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "weight refresh launch");
    h->last_stream = st;
    return ROLLOUT_OK;
}

}  // extern "C"

namespace {

// the device arrays of one run
struct RunBuffers {
    const float *features;
    const int32_t *starts;
    const uint32_t *seeds;
    float *states;
    int32_t *actions;
    float *logp;
    float *values;
    float *rewards;
    int32_t *dones;
    float *adv;
    float *ret;
};

// where the generic value kernel takes its per-CTA activation scratch
struct ValueScratch {
    uint8_t *ptr = nullptr;
    long long per_cta = 0;
    int grid = 0;
};

int check_run_args(rollout_handle *h, int N, int L, float gamma, float lambda)
{
    if (N <= 0 || L <= 0) return fail(ROLLOUT_ERR_INVALID, "N and L must be positive (N=%d, L=%d)", N, L);
    if ((long long)L > (long long)h->dims.n_bars - 1)
        return fail(ROLLOUT_ERR_INVALID, "L=%d needs at least L+1 bars (n_bars=%d)", L, h->dims.n_bars);
    if ((long long)N * L * kState >= (1LL << 40)) return fail(ROLLOUT_ERR_INVALID, "N*L too large");
    if (!(gamma >= 0.f && gamma <= 1.f) || !(lambda >= 0.f && lambda <= 1.f))
        return fail(ROLLOUT_ERR_INVALID, "gamma and lambda must lie in [0, 1]");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != h->device) return fail(ROLLOUT_ERR_INVALID, "current device %d is not the handle's device %d", dev, h->device);
    return ROLLOUT_OK;
}

int check_device_buffers(const RunBuffers &b)
{
    const void *ptrs[] = {b.features, b.starts, b.seeds, b.states, b.actions, b.logp,
                          b.values, b.rewards, b.dones, b.adv, b.ret};
    for (const void *p : ptrs) {
        if (!p) return fail(ROLLOUT_ERR_INVALID, "null array argument");
        if (((uintptr_t)p & 15u) != 0) return fail(ROLLOUT_ERR_INVALID, "array arguments must be 16-byte aligned");
    }
    return ROLLOUT_OK;
}

// Enqueues the kernels of one run on s.  points (kRunPoints events, or null) are
// recorded after the kernels that finish each group of outputs.
int enqueue_run(rollout_handle *h, const RunBuffers &b, int N, int L, float gamma, float lambda,
                const ValueScratch &vs, cudaStream_t s, cudaEvent_t *points)
{
    const rollout_dims &d = h->dims;
    cudaError_t e;
    h->last_stream = s;
    if ((e = cudaMemsetAsync(h->d_status, 0, sizeof(int), s)) != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    EnvConst env{d.barrier, d.max_hold, d.pt_scale, d.sl_scale, d.div_window, d.div_thresh, d.div_penalty,
                 d.cur_coef, d.risk_coef, d.tx_base, d.spread, h->d_div_low};
    Phase1Args p1{b.features, b.starts, b.seeds, N, L, d.n_bars, b.actions, b.logp, b.dones,
                  b.rewards, b.values, b.adv, h->d_status, env};
    StatesArgs sa{b.features, b.starts, N, L, d.n_bars, b.actions, b.dones, b.values, d.spread, b.states};
    if (d.dtype == ROLLOUT_BF16) sa.Fpad = h->d_fpad;   // refilled by launch_pad_features before the state rows
    ValueArgs va{b.features, b.starts, N, L, d.n_bars, b.actions, b.dones, b.values,
                 b.adv, b.rewards, b.ret, h->d_status, env};
    GaeArgs ga{b.rewards, b.values, b.dones, b.adv, b.ret, N, L, gamma, lambda};
    if (h->dump && d.dtype != ROLLOUT_FP32) {
        ActDump ad;
        ad.p = h->dump;
        ad.n_ep = h->dump_episodes;
        int col = kDumpIn + kActorH1 + kActorH2;
        for (int l = 0; l < kCriticLayers - 1; ++l) {
            ad.crit_off[l] = col;
            col += d.critic_h[l];
        }
        ad.cur_off = col;
        ad.width = col + d.cur_h;
        p1.dump = ad;
        va.dump = ad;
    }

    auto mark = [&](int i) { return h->timing ? cudaEventRecord(h->ev[i], s) : cudaSuccess; };
    auto point = [&](int p) { return points ? cudaEventRecord(points[p], s) : cudaSuccess; };
    if ((e = mark(0)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    if (d.dtype == ROLLOUT_FP32) {
        if ((e = launch_phase1_simt(p1, h->d_actor_packed, s)) != cudaSuccess) return cuda_fail(e, "phase 1 launch");
    } else {
        if (d.dtype == ROLLOUT_BF16 && (e = launch_pad_features(b.features, h->d_fpad, d.n_bars, s)) != cudaSuccess)
            return cuda_fail(e, "feature padding launch");
        if ((e = launch_phase1_umma(p1, h->umma, h->fmap, s)) != cudaSuccess) return cuda_fail(e, "phase 1 launch");
    }
    if ((e = mark(1)) != cudaSuccess || (e = point(kAfterRollout)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    if ((e = launch_states(sa, s)) != cudaSuccess) return cuda_fail(e, "state-row launch");
    if ((e = mark(2)) != cudaSuccess || (e = point(kAfterStates)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    if (d.dtype == ROLLOUT_FP32) e = launch_value_simt(va, h->simt, s);
    else if (value_needs_scratch(h->umma))
        e = launch_value_generic(va, h->umma, vs.ptr, vs.per_cta, vs.grid, s, h->test_stall);
    else e = launch_value_umma(va, h->umma, s, h->test_stall);
    if (e != cudaSuccess) return cuda_fail(e, "value launch");
    if ((e = mark(3)) != cudaSuccess || (e = point(kAfterValue)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    if ((e = launch_gae(ga, s)) != cudaSuccess) return cuda_fail(e, "gae launch");
    if ((e = mark(4)) != cudaSuccess || (e = point(kAfterGae)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    h->timed_run = h->timing;
    return ROLLOUT_OK;
}

// the handle's own scratch (allocated by rollout_create) for rollout_run
ValueScratch handle_scratch(rollout_handle *h, int N, int L)
{
    ValueScratch vs;
    if (h->dims.dtype == ROLLOUT_FP32 || !value_needs_scratch(h->umma)) return vs;
    const long long tiles = ((long long)N * L + N + 127) / 128;
    vs.ptr = h->d_scratch;
    vs.per_cta = h->scratch_per_cta;
    vs.grid = (int)(tiles < h->scratch_ctas ? tiles : h->scratch_ctas);
    return vs;
}

}  // namespace

extern "C" {

int rollout_run(rollout_handle *h, const float *features, const int32_t *episode_starts, const uint32_t *seeds,
                int N, int L, float gamma, float lambda, float *out_states, int32_t *out_actions,
                float *out_logp, float *out_values, float *out_rewards, int32_t *out_dones, float *out_adv,
                float *out_ret, void *stream)
{
    g_err[0] = 0;
    if (!h) return fail(ROLLOUT_ERR_INVALID, "null handle");
    const RunBuffers b{features, episode_starts, seeds, out_states, out_actions, out_logp,
                       out_values, out_rewards, out_dones, out_adv, out_ret};
    int rc = check_device_buffers(b);
    if (rc || (rc = check_run_args(h, N, L, gamma, lambda))) return rc;
    return enqueue_run(h, b, N, L, gamma, lambda, handle_scratch(h, N, L), (cudaStream_t)stream, nullptr);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant (rollout_run_static): the generic value kernel's
// per-CTA activation scratch comes from this fixed device array instead of
// memory allocated by rollout_create.  Its device address is looked up once
// per device, with that device current, and cached.
static __device__ __align__(256) uint8_t g_static_scratch[ROLLOUT_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
uint8_t *g_static_ptr[kMaxDevices] = {};

int static_scratch(int dev, uint8_t **out)
{
    if (dev < 0 || dev >= kMaxDevices) return fail(ROLLOUT_ERR_UNSUPPORTED, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        g_static_ptr[dev] = (uint8_t *)p;
    }
    *out = g_static_ptr[dev];
    return ROLLOUT_OK;
}

// ---------------------------------------------------------------------------
// rollout_run_host: device staging and the download schedule

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Lays out the staging allocation for (N, L); grows it when it is too small.
int stage_buffers(rollout_handle *h, int N, int L, RunBuffers *b)
{
    const size_t nl = (size_t)N * L;
    const size_t sizes[11] = {(size_t)h->dims.n_bars * kMarket * 4, (size_t)N * 4, (size_t)N * 4,
                              nl * kState * 4, nl * 4, nl * 4, nl * 4, nl * 4, nl * 4, nl * 4, nl * 4};
    size_t total = 0;
    for (size_t z : sizes) total += align256(z);
    cudaError_t e;
    if (total > h->stage_bytes) {
        // the previous run's copies may still read the old allocation: cudaFree waits for the device
        dev_free(h->d_stage);
        h->d_stage = nullptr;
        h->stage_bytes = 0;
        if ((e = dev_alloc((void **)&h->d_stage, total)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(staging)");
        h->stage_bytes = total;
    }
    uint8_t *p[11];
    size_t at = 0;
    for (int i = 0; i < 11; ++i) {
        p[i] = h->d_stage + at;
        at += align256(sizes[i]);
    }
    *b = RunBuffers{(const float *)p[0], (const int32_t *)p[1], (const uint32_t *)p[2], (float *)p[3],
                    (int32_t *)p[4], (float *)p[5], (float *)p[6], (float *)p[7], (int32_t *)p[8],
                    (float *)p[9], (float *)p[10]};
    return ROLLOUT_OK;
}

int make_copy_streams(rollout_handle *h)
{
    if (h->copy_stream[0]) return ROLLOUT_OK;
    cudaError_t e;
    for (int k = 0; k < kCopyStreams; ++k) {
        if ((e = cudaStreamCreateWithFlags(&h->copy_stream[k], cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail(e, "cudaStreamCreateWithFlags");
        if ((e = cudaEventCreateWithFlags(&h->copy_done[k], cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e, "cudaEventCreateWithFlags");
    }
    for (cudaEvent_t &ev : h->point_ev)
        if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e, "cudaEventCreateWithFlags");
    return ROLLOUT_OK;
}

// one output's download: host destination, device source, bytes, the run point after which it is final
struct Download {
    void *host;
    const void *dev;
    size_t bytes;
    int point;
};

}  // namespace

extern "C" {

int rollout_run_static(rollout_handle *h, const float *features, const int32_t *episode_starts, const uint32_t *seeds,
                       int N, int L, float gamma, float lambda, float *out_states, int32_t *out_actions,
                       float *out_logp, float *out_values, float *out_rewards, int32_t *out_dones, float *out_adv,
                       float *out_ret, void *stream)
{
    g_err[0] = 0;
    if (!h) return fail(ROLLOUT_ERR_INVALID, "null handle");
    const RunBuffers b{features, episode_starts, seeds, out_states, out_actions, out_logp,
                       out_values, out_rewards, out_dones, out_adv, out_ret};
    int rc = check_device_buffers(b);
    if (rc || (rc = check_run_args(h, N, L, gamma, lambda))) return rc;
    ValueScratch vs;
    if (h->dims.dtype != ROLLOUT_FP32 && value_needs_scratch(h->umma)) {
        vs.per_cta = value_generic_scratch_per_cta(h->umma);
        if (vs.per_cta > (long long)ROLLOUT_STATIC_SCRATCH_BYTES)
            return fail(ROLLOUT_ERR_UNSUPPORTED, "these layer shapes need %lld bytes of scratch per CTA, more than "
                        "the %u-byte static array", vs.per_cta, (unsigned)ROLLOUT_STATIC_SCRATCH_BYTES);
        if ((rc = static_scratch(h->device, &vs.ptr))) return rc;
        int sms = 0;
        cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, h->device);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        const long long fit = (long long)ROLLOUT_STATIC_SCRATCH_BYTES / vs.per_cta;
        const long long tiles = ((long long)N * L + N + 127) / 128;
        const long long g = tiles < sms ? tiles : sms;
        vs.grid = (int)(g < fit ? g : fit);
    }
    return enqueue_run(h, b, N, L, gamma, lambda, vs, (cudaStream_t)stream, nullptr);
}

int rollout_run_host(rollout_handle *h, const float *features, const int32_t *episode_starts, const uint32_t *seeds,
                     int N, int L, float gamma, float lambda, float *out_states, int32_t *out_actions,
                     float *out_logp, float *out_values, float *out_rewards, int32_t *out_dones, float *out_adv,
                     float *out_ret, void *stream)
{
    g_err[0] = 0;
    if (!h) return fail(ROLLOUT_ERR_INVALID, "null handle");
    if (!features || !episode_starts || !seeds) return fail(ROLLOUT_ERR_INVALID, "null input array");
    int rc = check_run_args(h, N, L, gamma, lambda);
    RunBuffers b{};
    if (rc || (rc = make_copy_streams(h)) || (rc = stage_buffers(h, N, L, &b))) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    const size_t nl = (size_t)N * L;
    if ((e = cudaMemcpyAsync((void *)b.features, features, (size_t)h->dims.n_bars * kMarket * 4,
                             cudaMemcpyHostToDevice, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync((void *)b.starts, episode_starts, (size_t)N * 4, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync((void *)b.seeds, seeds, (size_t)N * 4, cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpyAsync(inputs)");
    if ((rc = enqueue_run(h, b, N, L, gamma, lambda, handle_scratch(h, N, L), s, h->point_ev))) return rc;

    // Each output is copied back as soon as the kernel that finishes it is done;
    // the large ones are split over the copy streams.  The caller's stream then
    // waits for every copy stream, so the call stays stream-ordered.
    const Download downloads[] = {
        {out_actions, b.actions, nl * 4, kAfterRollout}, {out_logp, b.logp, nl * 4, kAfterRollout},
        {out_dones, b.dones, nl * 4, kAfterRollout},     {out_states, b.states, nl * kState * 4, kAfterStates},
        {out_values, b.values, nl * 4, kAfterValue},     {out_rewards, b.rewards, nl * 4, kAfterValue},
        {out_adv, b.adv, nl * 4, kAfterGae},             {out_ret, b.ret, nl * 4, kAfterGae}};
    constexpr size_t kSplitBytes = 64u << 20;   // outputs larger than this go out in kCopyStreams pieces
    int next = 0;
    for (int p = 0; p < kRunPoints; ++p) {
        for (int k = 0; k < kCopyStreams; ++k)
            if ((e = cudaStreamWaitEvent(h->copy_stream[k], h->point_ev[p], 0)) != cudaSuccess)
                return cuda_fail(e, "cudaStreamWaitEvent");
        for (const Download &dl : downloads) {
            if (dl.point != p || !dl.host) continue;
            const int pieces = dl.bytes > kSplitBytes ? kCopyStreams : 1;
            const size_t piece = ((dl.bytes / pieces) + 255) & ~(size_t)255;
            for (size_t at = 0; at < dl.bytes; at += piece) {
                const size_t n = dl.bytes - at < piece ? dl.bytes - at : piece;
                if ((e = cudaMemcpyAsync((uint8_t *)dl.host + at, (const uint8_t *)dl.dev + at, n,
                                         cudaMemcpyDeviceToHost, h->copy_stream[next])) != cudaSuccess)
                    return cuda_fail(e, "cudaMemcpyAsync(outputs)");
                next = (next + 1) % kCopyStreams;
            }
        }
    }
    for (int k = 0; k < kCopyStreams; ++k)
        if ((e = cudaEventRecord(h->copy_done[k], h->copy_stream[k])) != cudaSuccess ||
            (e = cudaStreamWaitEvent(s, h->copy_done[k], 0)) != cudaSuccess)
            return cuda_fail(e, "cudaEventRecord / cudaStreamWaitEvent");
    return ROLLOUT_OK;
}

}  // extern "C"

namespace {

// the curiosity model's input [state ; one-hot(action)], row stride ldc
__global__ void forward_prep_kernel(const float *states, const int32_t *actions, int M, float *ci, int ldc,
                                    int *status)
{
    const long long total = (long long)M * ldc;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long m = e / ldc;
        const int c = (int)(e - m * ldc);
        float v = 0.f;
        if (c < kState) {
            v = states[m * kState + c];
        } else if (c < kState + kActions) {
            const int a = actions[m];
            if (a < 0 || a >= kActions) {
                if (c == kState) atomicCAS(status, 0, ROLLOUT_ERR_RANGE);
            } else {
                v = (c - kState == a) ? 1.f : 0.f;
            }
        }
        ci[e] = v;
    }
}

constexpr int kFwdCi = 100;   // row stride of the curiosity input (99 used)

}  // namespace

extern "C" {

int rollout_forward(rollout_handle *h, const float *states, const int32_t *actions, int M, float *logits,
                    float *values, float *cur_pred, void *stream)
{
    g_err[0] = 0;
    if (!h || !states || !actions || !logits || !values || !cur_pred) return fail(ROLLOUT_ERR_INVALID, "null argument");
    if (M <= 0 || M > (1 << 24)) return fail(ROLLOUT_ERR_INVALID, "M must be in [1, 2^24]");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != h->device) return fail(ROLLOUT_ERR_INVALID, "current device %d is not the handle's device %d", dev, h->device);
    const rollout_dims &d = h->dims;
    const HostLayout lo = host_layout(d);
    const int ops = d.dtype == ROLLOUT_BF16 ? kGemmBf16 : d.dtype == ROLLOUT_TF32 ? kGemmTf32 : kGemmSplit3;
    cudaStream_t st = (cudaStream_t)stream;
    h->last_stream = st;
    // buffers: curiosity input, every hidden layer, split-K workspace and counters
    int csum = 0;
    for (int l = 0; l < kCriticLayers - 1; ++l) csum += lo.c_out[l];
    const size_t act_floats = (size_t)M * (kFwdCi + kActorH1 + kActorH2 + csum + kCurH);
    float *buf_probe = nullptr;
    float *ci = buf_probe, *ah[2], *ch[kCriticLayers - 1], *qz;
    auto layout_bufs = [&](float *base) {
        float *p = base;
        ci = p; p += (size_t)M * kFwdCi;
        ah[0] = p; p += (size_t)M * kActorH1;
        ah[1] = p; p += (size_t)M * kActorH2;
        for (int l = 0; l < kCriticLayers - 1; ++l) { ch[l] = p; p += (size_t)M * lo.c_out[l]; }
        qz = p;
    };
    // the products of depth j of the three networks
    auto stage = [&](int j, GemmArgs *g) -> int {
        int n = 0;
        auto prod = [&](const float *A, int lda, size_t w, size_t b, int in, int out, bool relu, float *Y) {
            GemmArgs x;
            x.A = A; x.lda = lda;
            x.B = h->d_wf32 + w; x.ldb = in;
            x.M = M; x.N = out; x.K = in;
            x.epi = kGemmFwd; x.operands = ops;
            x.bias = h->d_wf32 + b; x.relu = relu ? 1 : 0;
            x.Y = Y; x.ldy = out;
            x.status = h->d_status;
            g[n++] = x;
        };
        if (j < 3) prod(j == 0 ? states : ah[j - 1], j == 0 ? kState : lo.a_in[j], lo.a_w[j], lo.a_b[j], lo.a_in[j],
                        lo.a_out[j], j < 2, j < 2 ? ah[j] : logits);
        prod(j == 0 ? states : ch[j - 1], j == 0 ? kState : lo.c_in[j], lo.c_w[j], lo.c_b[j], lo.c_in[j], lo.c_out[j],
             j < kCriticLayers - 1, j < kCriticLayers - 1 ? ch[j] : values);
        if (j < 2) prod(j == 0 ? ci : qz, j == 0 ? kFwdCi : kCurH, lo.q_w[j], lo.q_b[j], lo.q_in[j], lo.q_out[j],
                        j == 0, j == 0 ? qz : cur_pred);
        return n;
    };
    // workspace: the largest over the stages
    layout_bufs(nullptr);
    long long ws_max = 0;
    int cnt_max = 0;
    for (int j = 0; j < kCriticLayers; ++j) {
        GemmArgs g[kGemmGroup];
        const int n = stage(j, g);
        long long wsum = 0;
        int csm = 0;
        for (int i = 0; i < n; ++i) {
            long long wf;
            int c;
            gemm_plan(g[i], 4, &wf, &c);
            wsum += wf;
            csm += c;
        }
        ws_max = wsum > ws_max ? wsum : ws_max;
        cnt_max = csm > cnt_max ? csm : cnt_max;
    }
    const size_t need = act_floats * 4 + (size_t)ws_max * 4 + (size_t)(cnt_max + 1) * 4 + 256;
    if (need > h->fwd_bytes) {
        dev_free(h->d_fwd);                      // cudaFree waits for work that may still use it
        h->d_fwd = nullptr;
        h->fwd_bytes = 0;
        if ((e = dev_alloc((void **)&h->d_fwd, need)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(forward buffers)");
        h->fwd_bytes = need;
    }
    float *base = reinterpret_cast<float *>(h->d_fwd);
    layout_bufs(base);
    float *ws = base + act_floats;
    unsigned int *cnt = reinterpret_cast<unsigned int *>(ws + ws_max);
    if ((e = cudaMemsetAsync(cnt, 0, (size_t)(cnt_max + 1) * 4, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(h->d_status, 0, sizeof(int), st)) != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync");
    const long long tot = (long long)M * kFwdCi;
    forward_prep_kernel<<<(int)((tot + 255) / 256 < 4096 ? (tot + 255) / 256 : 4096), 256, 0, st>>>(
        states, actions, M, ci, kFwdCi, h->d_status);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "forward input launch");
    for (int j = 0; j < kCriticLayers; ++j) {
        GemmArgs g[kGemmGroup];
        const int n = stage(j, g);
        long long wo = 0;
        int co = 0;
        for (int i = 0; i < n; ++i) {
            long long wf;
            int c;
            gemm_plan(g[i], 4, &wf, &c);
            g[i].ws = ws + wo;
            g[i].cnt = cnt + co;
            wo += wf;
            co += c;
        }
        if ((e = launch_gemm_group(g, n, st)) != cudaSuccess) return cuda_fail(e, "forward product launch");
    }
    return ROLLOUT_OK;
}

int rollout_status(rollout_handle *h)
{
    if (!h) return fail(ROLLOUT_ERR_INVALID, "null handle");
    cudaError_t e = cudaStreamSynchronize(h->last_stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int st = 0;
    if ((e = cudaMemcpy(&st, h->d_status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy(status)");
    return st;
}

int rollout_set_timing(rollout_handle *h, int on)
{
    g_err[0] = 0;
    if (!h) return fail(ROLLOUT_ERR_INVALID, "null handle");
    if (on && !h->ev[0]) {
        for (cudaEvent_t &ev : h->ev) {
            cudaError_t e = cudaEventCreate(&ev);
            if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
        }
    }
    h->timing = on != 0;
    h->timed_run = false;
    return ROLLOUT_OK;
}

int rollout_test_stall(rollout_handle *h, int on)
{
    g_err[0] = 0;
    if (!h) return fail(ROLLOUT_ERR_INVALID, "null handle");
    if (h->dims.dtype == ROLLOUT_FP32) return fail(ROLLOUT_ERR_INVALID, "the fp32 path has no bounded waits to stall");
    h->test_stall = on != 0;
    return ROLLOUT_OK;
}

int rollout_test_activations(rollout_handle *h, float *dump, int n_episodes)
{
    g_err[0] = 0;
    if (!h) return fail(ROLLOUT_ERR_INVALID, "null handle");
    if (h->dims.dtype == ROLLOUT_FP32) return fail(ROLLOUT_ERR_INVALID, "the fp32 path rounds no activations");
    if (dump && (n_episodes <= 0 || ((uintptr_t)dump & 15u)))
        return fail(ROLLOUT_ERR_INVALID, "the dump needs n_episodes > 0 and a 16-byte aligned array");
    h->dump = dump;
    h->dump_episodes = dump ? n_episodes : 0;
    return ROLLOUT_OK;
}

int rollout_test_alloc(long long fail_at, long long *live)
{
    g_err[0] = 0;
    rl::g_alloc_seen = 0;
    rl::g_alloc_fail_at = fail_at > 0 ? fail_at : 0;
    if (live) *live = rl::g_alloc_live.load();
    return ROLLOUT_OK;
}

int rollout_phase_ms(rollout_handle *h, float *ms)
{
    g_err[0] = 0;
    if (!h || !ms) return fail(ROLLOUT_ERR_INVALID, "null argument");
    if (!h->timed_run) return fail(ROLLOUT_ERR_INVALID, "no timed run (call rollout_set_timing first)");
    cudaError_t e = cudaEventSynchronize(h->ev[kTimedKernels]);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    for (int i = 0; i < kTimedKernels; ++i)
        if ((e = cudaEventElapsedTime(&ms[i], h->ev[i], h->ev[i + 1])) != cudaSuccess)
            return cuda_fail(e, "cudaEventElapsedTime");
    return ROLLOUT_OK;
}

void rollout_destroy(rollout_handle *h)
{
    if (!h) return;
    cudaDeviceSynchronize();
    free_handle(h);
}

}  // extern "C"
