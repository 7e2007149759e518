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
//
// Short key sets (T_k <= 32 with d_k = d_v = 64, the base model's head size)
// take a second kernel without the staging: each warp loads its row's whole
// key set straight into registers -- lane j key row j as 16 float4, every
// lane the query row and value columns lane and lane + 32 of each key -- so
// all of a warp's loads are in flight together and no shared-memory copy or
// CTA barrier sits between them and the arithmetic.  Its dot products,
// softmax and weighted sum are the chunked kernel's for a single chunk, in
// the same order, so both kernels give bitwise the same result there.
#include <cstdint>

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

constexpr int kShortRows = 4;   // query rows (warps) per CTA of the short-key kernel
constexpr int kShortMaxKeys = 32;

__global__ void __launch_bounds__(kShortRows * 32)
    sdpa_f32_short_kernel(const float *__restrict__ q, const float *__restrict__ k,
                          const float *__restrict__ v, float *__restrict__ o, int H, int Tq, int Tk,
                          float scale, int mask, const int32_t *__restrict__ key_lens) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long bh = blockIdx.x;
    const int b = static_cast<int>(bh / H);
    const int row = blockIdx.y * kShortRows + warp;
    if (row >= Tq) return;  // the whole warp

    // Every load first, all in bounds whatever the mask (1 <= Tk <= 32);
    // keys the row does not see are left out below, never read as weights.
    const float4 *qr = reinterpret_cast<const float4 *>(q + (bh * Tq + row) * 64);
    const float4 *kr = reinterpret_cast<const float4 *>(k + (bh * Tk + min(lane, Tk - 1)) * 64);
    const float *vb = v + bh * Tk * 64;
    float4 qa[16], ka[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        qa[c] = __ldg(qr + c);
        ka[c] = __ldg(kr + c);
    }
    float v_lo[kShortMaxKeys], v_hi[kShortMaxKeys];  // columns lane, lane + 32 of key j
#pragma unroll
    for (int j = 0; j < kShortMaxKeys; ++j) {
        v_lo[j] = 0.f;
        v_hi[j] = 0.f;
        if (j < Tk) {
            v_lo[j] = __ldg(vb + j * 64 + lane);
            v_hi[j] = __ldg(vb + j * 64 + 32 + lane);
        }
    }
    int kv_len = Tk;
    if ((mask & kMaskPaddingBit) && key_lens) kv_len = min(max(key_lens[b], 0), Tk);
    const int end = (mask & kMaskCausalBit) ? min(kv_len, row + 1) : kv_len;
    float *orow = o + (bh * Tq + row) * 64;
    if (end <= 0) {  // no visible key: zeros
        orow[lane] = 0.f;
        orow[lane + 32] = 0.f;
        return;
    }
    float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        part[0] = fmaf(qa[c].x, ka[c].x, part[0]);
        part[1] = fmaf(qa[c].y, ka[c].y, part[1]);
        part[2] = fmaf(qa[c].z, ka[c].z, part[2]);
        part[3] = fmaf(qa[c].w, ka[c].w, part[3]);
    }
    const float s = lane < end ? ((part[0] + part[1]) + (part[2] + part[3])) * scale : -INFINITY;
    float m = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float pj = expf(s - m);  // 0 for keys the row does not see
    float l = pj;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    float a_lo = 0.f, a_hi = 0.f;
#pragma unroll
    for (int j = 0; j < kShortMaxKeys; ++j) {
        if (j < end) {  // end is the same for the whole warp
            const float pb = __shfl_sync(0xffffffffu, pj, j);
            a_lo = fmaf(pb, v_lo[j], a_lo);
            a_hi = fmaf(pb, v_hi[j], a_hi);
        }
    }
    const float inv = 1.0f / l;  // l >= 1: the row maximum's weight is exactly 1
    orow[lane] = a_lo * inv;
    orow[lane + 32] = a_hi * inv;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t launch_sdpa_f32(const float *q, const float *k, const float *v, float *o, int B,
                            int H, int Tq, int Tk, int dk, int dv, float scale, int mask,
                            const int32_t *key_lens, cudaStream_t stream) {
    // Short key sets: the register kernel (float4 loads of q and k need
    // 16-byte aligned rows; otherwise, or past its grid limit, the chunked one).
    if (dk == 64 && dv == 64 && Tk >= 1 && Tk <= kShortMaxKeys && aligned16(q) && aligned16(k) &&
        (Tq + kShortRows - 1) / kShortRows <= 65535) {
        dim3 grid(static_cast<unsigned>(B * H), static_cast<unsigned>((Tq + kShortRows - 1) / kShortRows));
        sdpa_f32_short_kernel<<<grid, kShortRows * 32, 0, stream>>>(q, k, v, o, H, Tq, Tk, scale, mask,
                                                                   key_lens);
        return cudaGetLastError();
    }
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
