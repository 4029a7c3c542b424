// umma_path.cuh -- tensor-core (tcgen05) path for dtypes ROLLOUT_BF16 and
// ROLLOUT_TF32: weight images and the phase-1 / phase-2 launchers.
#pragma once

#include <stddef.h>

#include <vector>

#include "internal.cuh"

namespace rl {

// One dense layer as the value kernel streams it.  Its weights are a sequence
// of "units": for every 128-byte K-chunk k (in order) and every N-block nb (in
// order), a swizzled K-major tile of nb_rows[nb] rows x 128 bytes.
struct UmmaLayer {
    int n_out;          // valid outputs
    int k_chunks;       // 128-byte K-chunks of the (zero-padded) input
    int n_blocks;       // MMA N-blocks
    int nb_rows[4];     // rows of each N-block (multiple of 16, <= 256)
    long long w_off;    // byte offset of the layer's first unit in the stream
    int bias_off;       // float offset of the bias in `vec`
};

enum { kJobCrit1 = 0, kJobCrit2, kJobCrit3, kJobCrit4, kJobCrit5, kJobCur1, kJobCur2, kNumJobs };

struct UmmaWeights {
    bool bf16 = true;
    bool wide = false;          // critic 1024/768/512/256/128
    // phase 1: actor image [W1 chunks | W2 chunks | W3 chunks], copied whole into shared memory
    const uint8_t *actor_img = nullptr;
    uint32_t actor_img_bytes = 0;
    uint32_t actor_off[3] = {};  // byte offsets of W1, W2, W3 in the image
    const float *actor_bias = nullptr;   // b1[128] | b2[64] | b3[48] (b3 zero-padded)
    // phase 2: weight-unit stream and per-layer table
    const uint8_t *stream = nullptr;
    long long stream_bytes = 0;
    UmmaLayer job[kNumJobs];
    // bulk-copy units of the stream, in consumption order (one tile's worth)
    int n_units = 0;
    long long unit_off[32] = {};
    uint32_t unit_bytes[32] = {};
    const float *vec = nullptr;  // biases, head weights, curiosity one-hot columns (f32)
    size_t buf_bytes = 0;        // size of the device allocation (reused by later uploads)
    int head_w_off = 0;          // critic head weights [h5] (rounded to the operand format)
    int head_b_off = 0;          // critic head bias [1]
    int onehot_off = 0;          // curiosity layer-1 one-hot columns [45][64] (rounded)
};

// what the host packer needs from the packed f32 weight buffer (float offsets)
struct UmmaHostLayout {
    size_t a_w[3], a_b[3];
    size_t c_w[kCriticLayers], c_b[kCriticLayers];
    int c_in[kCriticLayers], c_out[kCriticLayers];
    size_t q_w[2], q_b[2];
    int n_critic;
};

// the packed bytes of one upload and where its regions lie (element size 2 for
// bf16 tiles, 4 for tf32 tiles and float32 vectors)
struct UmmaRegion {
    size_t off, bytes;
    int elem;
};
struct UmmaHostImage {
    std::vector<uint8_t> bytes;
    UmmaRegion region[4];   // actor image, actor bias, unit stream, vec
};
// packs on the host (fills w's tables, not its device pointers)
void umma_pack_host(UmmaWeights *w, bool bf16, const float *host_w, const UmmaHostLayout &lo, UmmaHostImage *out);

// converts/uploads; *d_buf receives (or reuses) the device allocation
int umma_upload(UmmaWeights *w, void **d_buf, bool bf16, const float *host_w, const UmmaHostLayout &lo,
                char *err, size_t err_len);

// fmap: 2-D tensor map over the padded feature copy [n_bars][kFPad] (f32,
// box 52 x 1), used by the bf16 kernel; fpad is filled by launch_pad_features
cudaError_t launch_phase1_umma(const Phase1Args &a, const UmmaWeights &w, const CUtensorMap &fmap, cudaStream_t s);
// bf16 operands with the 512/384/256/128/64 critic: activations resident in shared memory
// stall: launch the test build whose first weight producer in CTA 0 issues
// nothing (that CTA's bounded wait expires and the run reports a timeout)
cudaError_t launch_value_umma(const ValueArgs &a, const UmmaWeights &w, cudaStream_t s, bool stall);
// every other shape: activations in per-CTA global scratch (see value_generic.cu)
long long value_generic_scratch_per_cta(const UmmaWeights &w);
cudaError_t launch_value_generic(const ValueArgs &a, const UmmaWeights &w, uint8_t *scratch, long long per_cta,
                                 int grid, cudaStream_t s, bool stall);
inline bool value_needs_scratch(const UmmaWeights &w) { return !w.bf16 || w.wide; }

}  // namespace rl
