// sdpa_f32.cu -- fp32 scaled dot-product attention on the SIMT cores.
//
// The full-precision path: o = softmax(scale * q k^T + mask) v with fp32
// FFMA dot products and expf (no tensor cores: TF32 would round q and k to
// 10 mantissa bits).  The softmax is taken online over chunks of 32 keys:
// per chunk the row's maximum, the partial output and sum rescaled by
// exp(m_old - m_new) when the maximum grows, which equals the textbook
// softmax up to rounding ("Attention Is All You Need" (azimuth.plus), "The
// same idea in code": subtract the row maximum, exponentiate, normalise).
// Masked keys get weight exactly zero (notebook chapter, "Masked Attention in
// the Decoder"): causal keys past the row and padded keys are never scored.
//
// One CTA per (b, h) and block of kF32RowsPerCta query rows, one warp per
// row.  Each chunk of 32 key and value rows is first copied into shared
// memory by the whole CTA -- every load of the chunk in flight at once, so a
// chunk costs one memory round trip instead of one per key -- and then
// serves all the CTA's rows: lane j scores key j of the chunk (K rows padded
// by one float so the 32 lanes read 32 different banks), the warp reduces
// the chunk's maximum and sum with shuffles, and lane l accumulates output
// columns l, l+32, l+64, l+96 from the value rows.
#include "kernels.h"

namespace mha {
namespace {

constexpr int kRows = kF32RowsPerCta;  // one warp per query row
constexpr int kChunk = 32;             // keys per shared-memory chunk (one per lane)
constexpr int kMaxD = 128;             // d_k, d_v <= 128
constexpr int kMaxPerLane = kMaxD / 32;

// DK = 64: head dimensions fixed at compile time (the common case: constant
// loop bounds, no per-feature range checks); DK = 0: d_k, d_v <= 128 at run
// time.
template <int DK>
__global__ void __launch_bounds__(kRows * 32)
    sdpa_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                    const float *__restrict__ v, float *__restrict__ o, int H, int Tq, int Tk,
                    int dk_rt, int dv_rt, float scale, int mask, const int32_t *__restrict__ key_lens) {
    const int dk = DK ? DK : dk_rt, dv = DK ? DK : dv_rt;
    __shared__ float ks[kChunk][kMaxD + 1];
    __shared__ float vs[kChunk][kMaxD];
    __shared__ __align__(16) float qs[kRows][kMaxD];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long bh = blockIdx.x;
    const int b = static_cast<int>(bh / H);
    const int row0 = blockIdx.y * kRows;
    const int row = row0 + warp;
    const bool live = row < Tq;

    int kv_len = Tk;
    if ((mask & kMaskPaddingBit) && key_lens) kv_len = min(max(key_lens[b], 0), Tk);
    const bool causal = (mask & kMaskCausalBit) != 0;
    // Keys this row sees, and keys any row of the CTA sees.
    const int end = live ? (causal ? min(kv_len, row + 1) : kv_len) : 0;
    const int last_row = min(row0 + kRows, Tq) - 1;
    const int cta_end = causal ? min(kv_len, last_row + 1) : kv_len;

    if (live) {
        const float *qr = q + (bh * Tq + row) * dk;
        for (int c = lane; c < dk; c += 32) qs[warp][c] = qr[c];
    }
    float acc[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) acc[i] = 0.f;
    float m = -INFINITY, l = 0.f;

    const float *kb = k + bh * Tk * dk;
    const float *vb = v + bh * Tk * dv;
    for (int c0 = 0; c0 < cta_end; c0 += kChunk) {
        const int n = min(kChunk, cta_end - c0);
        __syncthreads();  // the previous chunk (and, first time, q) is consumed / written
        {
            const float *ksrc = kb + static_cast<long long>(c0) * dk;
            const float *vsrc = vb + static_cast<long long>(c0) * dv;
            const int nk = n * dk, nv = n * dv;
#pragma unroll 4
            for (int x = threadIdx.x; x < nk; x += kRows * 32) {
                const int j = x / dk;
                ks[j][x - j * dk] = ksrc[x];
            }
#pragma unroll 4
            for (int x = threadIdx.x; x < nv; x += kRows * 32) {
                const int j = x / dv;
                vs[j][x - j * dv] = vsrc[x];
            }
        }
        __syncthreads();
        if (c0 >= end) continue;  // this row sees none of the chunk's keys
        // Lane j: score of key c0 + j (-inf past the row's visible keys).
        float s = -INFINITY;
        if (c0 + lane < end) {
            float part[4] = {0.f, 0.f, 0.f, 0.f};  // four chains for ILP
            if constexpr (DK > 0) {
#pragma unroll
                for (int c = 0; c < DK; c += 4) {
                    const float4 q4 = *reinterpret_cast<const float4 *>(&qs[warp][c]);
                    part[0] = fmaf(q4.x, ks[lane][c], part[0]);
                    part[1] = fmaf(q4.y, ks[lane][c + 1], part[1]);
                    part[2] = fmaf(q4.z, ks[lane][c + 2], part[2]);
                    part[3] = fmaf(q4.w, ks[lane][c + 3], part[3]);
                }
            } else {
                int c = 0;
                for (; c + 4 <= dk; c += 4) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) part[u] = fmaf(qs[warp][c + u], ks[lane][c + u], part[u]);
                }
                for (; c < dk; ++c) part[0] = fmaf(qs[warp][c], ks[lane][c], part[0]);
            }
            s = ((part[0] + part[1]) + (part[2] + part[3])) * scale;
        }
        float mc = s;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, off));
        const float m_new = fmaxf(m, mc);  // finite: key c0 is visible
        const float alpha = expf(m - m_new);  // 0 for the row's first chunk
        const float pj = expf(s - m_new);     // 0 for masked keys
        float ps = pj;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        l = l * alpha + ps;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) acc[i] *= alpha;
        const int nj = min(n, end - c0);
        for (int j = 0; j < nj; ++j) {
            const float pb = __shfl_sync(0xffffffffu, pj, j);
#pragma unroll
            for (int i = 0; i < kMaxPerLane; ++i) {
                const int c = lane + 32 * i;
                if (c < dv) acc[i] = fmaf(pb, vs[j][c], acc[i]);
            }
        }
        m = m_new;
    }
    if (!live) return;
    const float inv = l > 0.f ? 1.0f / l : 0.f;  // no visible key: zeros
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
    dim3 grid(static_cast<unsigned>(B * H), static_cast<unsigned>((Tq + kRows - 1) / kRows));
    if (dk == 64 && dv == 64)
        sdpa_f32_kernel<64><<<grid, kRows * 32, 0, stream>>>(q, k, v, o, H, Tq, Tk, dk, dv, scale, mask,
                                                            key_lens);
    else
        sdpa_f32_kernel<0><<<grid, kRows * 32, 0, stream>>>(q, k, v, o, H, Tq, Tk, dk, dv, scale, mask,
                                                           key_lens);
    return cudaGetLastError();
}

}  // namespace mha
