// umma_pack.cu -- host-side conversion of the packed float32 weights into the
// tensor-core images: operands rounded once to the MMA format (bf16
// round-to-nearest-even, or tf32 round-to-nearest ties away from zero, the
// rounding of cvt.rna.tf32.f32), laid out as K-major 128-byte-swizzled tiles
// (see umma.cuh), zero-padded in K and N.
#include <stdio.h>
#include <string.h>

#include <vector>

#include "umma_path.cuh"

namespace rl {

namespace {

uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

// bf16 bit pattern, round to nearest even (finite inputs)
uint16_t bf16_bits(float x)
{
    const uint32_t u = f2u(x);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

// tf32 value in a 32-bit container, round to nearest, ties away from zero
uint32_t tf32_bits(float x) { return (f2u(x) + 0x1000u) & 0xFFFFE000u; }

float rounded(float x, bool bf16) { return bf16 ? u2f((uint32_t)bf16_bits(x) << 16) : u2f(tf32_bits(x)); }

struct Packer {
    bool bf16;
    int kc;   // elements per 128-byte K-chunk
    explicit Packer(bool b) : bf16(b), kc(b ? 64 : 32) {}

    // one swizzled tile: rows [row0, row0+nrows) of W[n_out][ld] (columns
    // [0, k_valid) used, K-chunk `chunk`), appended to `out`
    void tile(std::vector<uint8_t> &out, const float *W, int n_out, int ld, int k_valid, int row0, int nrows,
              int chunk) const
    {
        const size_t base = out.size();
        out.resize(base + (size_t)nrows * 128, 0);
        for (int r = 0; r < nrows; ++r) {
            const int n = row0 + r;
            for (int c = 0; c < kc; ++c) {
                const int k = chunk * kc + c;
                const float v = (n < n_out && k < k_valid) ? W[(size_t)n * ld + k] : 0.f;
                const int byte = c * (bf16 ? 2 : 4);
                const int unit = byte >> 4, within = byte & 15;
                const size_t off = base + (size_t)(r >> 3) * 1024 + (r & 7) * 128 + ((unit ^ (r & 7)) << 4) + within;
                if (bf16) {
                    const uint16_t b = bf16_bits(v);
                    memcpy(&out[off], &b, 2);
                } else {
                    const uint32_t b = tf32_bits(v);
                    memcpy(&out[off], &b, 4);
                }
            }
        }
    }
};

void set_layer(UmmaLayer &L, int n_out, int k_in, int kc, std::initializer_list<int> blocks)
{
    L.n_out = n_out;
    L.k_chunks = (k_in + kc - 1) / kc;
    L.n_blocks = 0;
    for (int b : blocks) L.nb_rows[L.n_blocks++] = b;
}

}  // namespace

void umma_pack_host(UmmaWeights *w, bool bf16, const float *hw, const UmmaHostLayout &lo, UmmaHostImage *out)
{
    const Packer P(bf16);
    const int kc = P.kc;
    const bool wide = lo.c_out[0] == 1024;
    // ---------------- phase-1 actor image
    std::vector<uint8_t> img;
    const int k1 = (kState + kc - 1) / kc, k2 = kActorH1 / kc, k3 = kActorH2 / kc;
    w->actor_off[0] = 0;
    for (int c = 0; c < k1; ++c) P.tile(img, hw + lo.a_w[0], kActorH1, kState, kState, 0, kActorH1, c);
    w->actor_off[1] = (uint32_t)img.size();
    for (int c = 0; c < k2; ++c) P.tile(img, hw + lo.a_w[1], kActorH2, kActorH1, kActorH1, 0, kActorH2, c);
    w->actor_off[2] = (uint32_t)img.size();
    for (int c = 0; c < k3; ++c) P.tile(img, hw + lo.a_w[2], kActions, kActorH2, kActorH2, 0, 48, c);
    w->actor_img_bytes = (uint32_t)img.size();

    std::vector<float> abias(kActorH1 + kActorH2 + 48, 0.f);
    memcpy(&abias[0], hw + lo.a_b[0], sizeof(float) * kActorH1);
    memcpy(&abias[kActorH1], hw + lo.a_b[1], sizeof(float) * kActorH2);
    memcpy(&abias[kActorH1 + kActorH2], hw + lo.a_b[2], sizeof(float) * kActions);

    // ---------------- phase-2 unit stream
    UmmaLayer *J = w->job;
    if (!wide) {
        set_layer(J[kJobCrit1], 512, kState, kc, {256, 256});
        set_layer(J[kJobCrit2], 384, 512, kc, {256, 128});
        set_layer(J[kJobCrit3], 256, 384, kc, {256});
        set_layer(J[kJobCrit4], 128, 256, kc, {128});
        set_layer(J[kJobCrit5], 64, 128, kc, {64});
    } else {
        set_layer(J[kJobCrit1], 1024, kState, kc, {256, 256, 256, 256});
        set_layer(J[kJobCrit2], 768, 1024, kc, {256, 256, 256});
        set_layer(J[kJobCrit3], 512, 768, kc, {256, 256});
        set_layer(J[kJobCrit4], 256, 512, kc, {256});
        set_layer(J[kJobCrit5], 128, 256, kc, {128});
    }
    set_layer(J[kJobCur1], kCurH, kState, kc, {64});
    set_layer(J[kJobCur2], kState, kCurH, kc, {64});

    std::vector<uint8_t> stream;
    std::vector<float> vec;
    auto add_bias = [&](int j, const float *bias) {
        UmmaLayer &L = J[j];
        L.bias_off = (int)vec.size();
        int npad = 0;
        for (int nb = 0; nb < L.n_blocks; ++nb) npad += L.nb_rows[nb];
        for (int n = 0; n < npad; ++n) vec.push_back(n < L.n_out ? bias[n] : 0.f);
    };
    for (int l = 0; l < 5; ++l) add_bias(kJobCrit1 + l, hw + lo.c_b[l]);
    add_bias(kJobCur1, hw + lo.q_b[0]);
    add_bias(kJobCur2, hw + lo.q_b[1]);
    w->n_units = 0;
    auto begin_unit = [&]() { w->unit_off[w->n_units] = (long long)stream.size(); };
    auto end_unit = [&]() {
        w->unit_bytes[w->n_units] = (uint32_t)((long long)stream.size() - w->unit_off[w->n_units]);
        w->n_units++;
    };
    const float *V[5];
    int vin[5];
    for (int l = 0; l < 5; ++l) { V[l] = hw + lo.c_w[l]; vin[l] = lo.c_in[l]; }
    const float *C1 = hw + lo.q_w[0], *C2 = hw + lo.q_w[1];
    if (bf16 && !wide) {
        // value-kernel consumption order (see value_umma.cu): 26 units of <= 32 KB
        begin_unit();
        P.tile(stream, C1, kCurH, kState + kActions, kState, 0, 64, 0);          // curiosity 1 (state part)
        P.tile(stream, V[0], 512, vin[0], vin[0], 0, 128, 0);                     // layer-1 chunk 0 (128 rows)
        P.tile(stream, C2, kState, kCurH, kCurH, 0, 64, 0);                      // curiosity 2
        end_unit();
        for (int i = 0; i < 8; ++i) {
            // K-chunk 0: rows 0-255 of W2, then rows 256-383; later K-chunks the other
            // way round, for odd i < 7 with the next 128 layer-1 rows in front
            if (i == 0) {
                begin_unit();
                P.tile(stream, V[1], 384, vin[1], vin[1], 0, 256, i);
                end_unit();
            }
            begin_unit();
            if ((i & 1) && i < 7) P.tile(stream, V[0], 512, vin[0], vin[0], 128 * ((i + 1) / 2), 128, 0);
            P.tile(stream, V[1], 384, vin[1], vin[1], 256, 128, i);
            end_unit();
            if (i > 0) {
                begin_unit();
                P.tile(stream, V[1], 384, vin[1], vin[1], 0, 256, i);
                end_unit();
            }
        }
        const int order3[6] = {4, 5, 0, 1, 2, 3};
        for (int kk = 0; kk < 6; ++kk) {
            begin_unit();
            P.tile(stream, V[2], 256, vin[2], vin[2], 0, 256, order3[kk]);       // layer 3
            end_unit();
        }
        for (int h = 0; h < 2; ++h) {
            begin_unit();
            for (int k = 2 * h; k < 2 * h + 2; ++k) P.tile(stream, V[3], 128, vin[3], vin[3], 0, 128, k);  // layer 4
            end_unit();
        }
        begin_unit();
        for (int k = 0; k < 2; ++k) P.tile(stream, V[4], 64, vin[4], vin[4], 0, 64, k);     // layer 5
        end_unit();
    } else {
        // generic kernel order: per layer, N-block-major; the K-chunk tiles of
        // one N-block are contiguous
        auto emit = [&](int j, const float *W, int ld, int k_valid) {
            UmmaLayer &L = J[j];
            L.w_off = (long long)stream.size();
            int row0 = 0;
            for (int nb = 0; nb < L.n_blocks; ++nb) {
                for (int c = 0; c < L.k_chunks; ++c) P.tile(stream, W, L.n_out, ld, k_valid, row0, L.nb_rows[nb], c);
                row0 += L.nb_rows[nb];
            }
        };
        for (int l = 0; l < 5; ++l) emit(kJobCrit1 + l, V[l], vin[l], vin[l]);
        emit(kJobCur1, C1, kState + kActions, kState);
        emit(kJobCur2, C2, kCurH, kCurH);
    }
    w->head_w_off = (int)vec.size();
    const int h5 = lo.c_in[5];
    for (int k = 0; k < h5; ++k) vec.push_back(rounded(hw[lo.c_w[5] + k], bf16));
    w->head_b_off = (int)vec.size();
    vec.push_back(hw[lo.c_b[5]]);
    while (vec.size() % 4) vec.push_back(0.f);
    w->onehot_off = (int)vec.size();
    for (int a = 0; a < kActions; ++a)
        for (int j = 0; j < kCurH; ++j)
            vec.push_back(rounded(hw[lo.q_w[0] + (size_t)j * (kState + kActions) + kState + a], bf16));

    // ---------------- one allocation: image | actor bias | stream | vec
    auto align = [](size_t x) { return (x + 1023) & ~(size_t)1023; };
    UmmaHostImage &im = *out;
    im.region[0] = {0, img.size(), bf16 ? 2 : 4};                                   // actor image
    im.region[1] = {align(img.size()), abias.size() * 4, 4};                         // actor bias (f32)
    im.region[2] = {align(im.region[1].off + im.region[1].bytes), stream.size(), bf16 ? 2 : 4};   // unit stream
    im.region[3] = {align(im.region[2].off + im.region[2].bytes), vec.size() * 4, 4};            // vec (f32)
    im.bytes.assign(align(im.region[3].off + im.region[3].bytes), 0);
    memcpy(&im.bytes[im.region[0].off], img.data(), img.size());
    memcpy(&im.bytes[im.region[1].off], abias.data(), abias.size() * 4);
    memcpy(&im.bytes[im.region[2].off], stream.data(), stream.size());
    memcpy(&im.bytes[im.region[3].off], vec.data(), vec.size() * 4);
    w->bf16 = bf16;
    w->wide = wide;
    w->stream_bytes = (long long)stream.size();
}

int umma_upload(UmmaWeights *w, void **d_buf, bool bf16, const float *hw, const UmmaHostLayout &lo, char *err,
                size_t err_len)
{
    UmmaHostImage im;
    umma_pack_host(w, bf16, hw, lo, &im);
    const size_t total = im.bytes.size();
    cudaError_t e;
    // later uploads of the same shapes reuse the allocation, so device pointers
    // into it (the weight-refresh maps) stay valid
    if (*d_buf && w->buf_bytes != total) {
        dev_free(*d_buf);
        *d_buf = nullptr;
    }
    if (!*d_buf) {
        if ((e = dev_alloc(d_buf, total)) != cudaSuccess) {
            snprintf(err, err_len, "cudaMalloc(tensor-core weights): %s", cudaGetErrorString(e));
            return e == cudaErrorMemoryAllocation ? ROLLOUT_ERR_NOMEM : ROLLOUT_ERR_CUDA;
        }
        w->buf_bytes = total;
    }
    if ((e = cudaMemcpy(*d_buf, im.bytes.data(), total, cudaMemcpyHostToDevice)) != cudaSuccess) {
        snprintf(err, err_len, "cudaMemcpy(tensor-core weights): %s", cudaGetErrorString(e));
        return ROLLOUT_ERR_CUDA;
    }
    uint8_t *base = (uint8_t *)*d_buf;
    w->actor_img = base + im.region[0].off;
    w->actor_bias = (const float *)(base + im.region[1].off);
    w->stream = base + im.region[2].off;
    w->vec = (const float *)(base + im.region[3].off);
    return ROLLOUT_OK;
}

}  // namespace rl
