// sdpa_f32.cu -- fp32 scaled dot-product attention on the SIMT cores.
//
// The full-precision path: o = softmax(scale * q k^T + mask) v with fp32
// FFMA dot products and expf (no tensor cores: TF32 would round q and k to
// 10 mantissa bits).  One warp per query row; lane l owns feature columns
// l, l+32, l+64, l+96.  Keys are visited in order with a running maximum
// and sum (online softmax: the partial output is rescaled by
// exp(m_old - m_new) whenever the maximum grows), which equals the textbook
// softmax up to rounding ("Attention Is All You Need" (azimuth.plus), "The
// same idea in code": subtract the row maximum, exponentiate, normalise).
// Masked keys are never visited, i.e. they get exactly zero weight
// (notebook chapter, "Masked Attention in the Decoder").
#include "kernels.h"

namespace mha {
namespace {

constexpr int kRowsPerCta = 4;  // one warp per row
constexpr int kMaxPerLane = 4;  // d_k, d_v <= 128

__global__ void __launch_bounds__(kRowsPerCta * 32)
    sdpa_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                    const float *__restrict__ v, float *__restrict__ o, int H, int Tq, int Tk,
                    int dk, int dv, float scale, int mask, const int32_t *__restrict__ key_lens) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long bh = blockIdx.x;
    const int b = static_cast<int>(bh / H);
    const int row = blockIdx.y * kRowsPerCta + warp;
    if (row >= Tq) return;

    int end = Tk;
    if ((mask & kMaskPaddingBit) && key_lens) end = min(max(key_lens[b], 0), Tk);
    if (mask & kMaskCausalBit) end = min(end, row + 1);

    const float *qr = q + (bh * Tq + row) * dk;
    float qv[kMaxPerLane], acc[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
        const int c = lane + 32 * i;
        qv[i] = c < dk ? qr[c] : 0.f;
        acc[i] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const float *kb = k + bh * Tk * dk;
    const float *vb = v + bh * Tk * dv;
    for (int j = 0; j < end; ++j) {
        const float *kr = kb + static_cast<long long>(j) * dk;
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            const int c = lane + 32 * i;
            if (c < dk) part = fmaf(qv[i], kr[c], part);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        const float s = part * scale;
        const float m_new = fmaxf(m, s);
        const float alpha = expf(m - m_new);  // 0 on the first key
        const float pj = expf(s - m_new);
        l = l * alpha + pj;
        const float *vr = vb + static_cast<long long>(j) * dv;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            const int c = lane + 32 * i;
            if (c < dv) acc[i] = fmaf(pj, vr[c], acc[i] * alpha);
        }
        m = m_new;
    }
    const float inv = l > 0.f ? 1.0f / l : 0.f;
    float *orow = o + (bh * Tq + row) * dv;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
        const int c = lane + 32 * i;
        if (c < dv) orow[c] = acc[i] * inv;
    }
}

}  // namespace

cudaError_t launch_sdpa_f32(const float *q, const float *k, const float *v, float *o, int B,
                            int H, int Tq, int Tk, int dk, int dv, float scale, int mask,
                            const int32_t *key_lens, cudaStream_t stream) {
    dim3 grid(static_cast<unsigned>(B * H),
              static_cast<unsigned>((Tq + kRowsPerCta - 1) / kRowsPerCta));
    sdpa_f32_kernel<<<grid, kRowsPerCta * 32, 0, stream>>>(q, k, v, o, H, Tq, Tk, dk, dv, scale,
                                                          mask, key_lens);
    return cudaGetLastError();
}

}  // namespace mha
