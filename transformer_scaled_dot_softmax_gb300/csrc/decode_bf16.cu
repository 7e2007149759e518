// decode_bf16.cu -- attention for decoding steps: a few new query rows per
// (batch b, head h) against a key/value cache, on sm_103a.
//
// Generation is a loop that emits one token at a time and feeds it back in
// (aiany.app Step 10, "The decoder"); at each step the new query row of a
// sequence attends to every cached key of that sequence -- its own earlier
// positions for self-attention (the causal mask of the notebook chapter
// "Masked Attention in the Decoder", restricted to the newest row, is exactly
// "keys j < len_b") or the encoder output for cross-attention ("The
// Decoder's Cross-Attention").  So each of the T_q query rows computes
//   o = softmax(scale * q K[0:len_b]^T) V[0:len_b],
// the same scaled dot-product attention as the full kernel, with a
// key-padding length per sequence.
//
// With one or a few query rows there is no matrix product worth the tensor
// cores: every cached key costs 256 bytes of K and V read for 4*d*T_q flops,
// so the kernel is bound by HBM bandwidth.  Layout of the work:
//
//   * the keys of one (b, h) are split over the 8 CTAs of a thread-block
//     cluster; each CTA streams its contiguous key range with 16-byte
//     loads (8 lanes read one 128-byte key row, a warp 4 consecutive rows =
//     512 contiguous bytes per load instruction), 6 rows per lane group in
//     flight per step (4 measured 5 % slower, 8 no faster);
//   * every warp keeps, per query row, an online-softmax state (running
//     maximum m, sum l, partial output o) over its keys; the 4 warps of a CTA
//     and then the 8 CTAs of the cluster are merged exactly:
//       M = max_i m_i,  l = sum_i l_i 2^(m_i - M),  o = sum_i o_i 2^(m_i - M),
//     the CTA partials through distributed shared memory, so one launch
//     needs no workspace;
//   * the output row is o / l in bf16 (0 when len_b = 0).
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace mha {
namespace {

constexpr int kSplits = 8;    // CTAs per cluster = key-range splits per (b, h)
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kUnroll = 6;    // key rows in flight per lane group
constexpr int kKeysPerStep = kWarps * 4 * kUnroll;  // 96 keys per CTA step
constexpr int HD = kAttnHeadDim;

template <int NQ>
struct SmemDecode {
    float w_m[kWarps][NQ];
    float w_l[kWarps][NQ];
    float w_o[kWarps][NQ][HD];
    // This CTA's merged partial, read by the cluster's rank 0.
    float c_m[NQ];
    float c_l[NQ];
    float c_o[NQ][HD];
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ float dsmem_ld(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Weight of a partial with maximum m against the merged maximum M: 0 for a
// partial that saw no key (m = -inf).
__device__ __forceinline__ float merge_weight(float m, float M) {
    return m == -INFINITY ? 0.f : ex2_approx(m - M);
}

template <int NQ>
__global__ void __cluster_dims__(kSplits, 1, 1) __launch_bounds__(kThreads)
    decode_bf16_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                       const __nv_bfloat16 *__restrict__ v, __nv_bfloat16 *__restrict__ o,
                       DecodeParams p) {
    __shared__ SmemDecode<NQ> sm;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int slot = lane >> 3;  // which of the warp's 4 consecutive key rows
    const int part = lane & 7;   // which 8 of the 64 features
    const long long bh = blockIdx.x / kSplits;
    const int split = static_cast<int>(cluster_rank());
    const int b = static_cast<int>(bh / p.H);

    int len = p.Tk;
    if (p.key_lens) len = min(max(p.key_lens[b], 0), p.Tk);
    // Contiguous key range of this split, a multiple of one CTA step.
    const int per = ((len + kSplits - 1) / kSplits + kKeysPerStep - 1) / kKeysPerStep * kKeysPerStep;
    const int k_begin = min(len, split * per);
    const int k_end = min(len, k_begin + per);

    // Query features of this lane, pre-scaled so scores are in log2 units.
    float qf[NQ][8];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        if (i < p.Tq) {
            const uint4 u = *reinterpret_cast<const uint4 *>(q + (bh * p.Tq + i) * HD + part * 8);
            bf16x8_to_f32(u, qf[i]);
#pragma unroll
            for (int c = 0; c < 8; ++c) qf[i][c] *= p.scale_log2;
        } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) qf[i][c] = 0.f;
        }
    }

    float m_run[NQ], l_run[NQ], acc[NQ][8];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        m_run[i] = -INFINITY;
        l_run[i] = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[i][c] = 0.f;
    }

    const __nv_bfloat16 *kb = k + bh * static_cast<long long>(p.Tk) * HD + part * 8;
    const __nv_bfloat16 *vb = v + bh * static_cast<long long>(p.Tk) * HD + part * 8;
    for (int base = k_begin; base < k_end; base += kKeysPerStep) {
        uint4 ku[kUnroll], vu[kUnroll];
        bool live[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int key = base + (u * kWarps + warp) * 4 + slot;
            live[u] = key < k_end;
            if (live[u]) {
                ku[u] = __ldcs(reinterpret_cast<const uint4 *>(kb + static_cast<long long>(key) * HD));
                vu[u] = __ldcs(reinterpret_cast<const uint4 *>(vb + static_cast<long long>(key) * HD));
            } else {
                ku[u] = make_uint4(0u, 0u, 0u, 0u);
                vu[u] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            float s[kUnroll];
            float smax = -INFINITY;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                float kf[8];
                bf16x8_to_f32(ku[u], kf);
                float d = 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) d = fmaf(qf[i][c], kf[c], d);
                // Sum over the 8 lanes that hold this key row.
                d += __shfl_xor_sync(0xffffffffu, d, 1);
                d += __shfl_xor_sync(0xffffffffu, d, 2);
                d += __shfl_xor_sync(0xffffffffu, d, 4);
                s[u] = live[u] ? d : -INFINITY;
                smax = fmaxf(smax, s[u]);
            }
            // Maximum over the warp's 4 key rows of each step.
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 8));
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 16));
            const float m_new = fmaxf(m_run[i], smax);
            if (m_new == -INFINITY) continue;  // nothing visible yet (warp-uniform)
            const float alpha = m_run[i] == -INFINITY ? 0.f : ex2_approx(m_run[i] - m_new);
            m_run[i] = m_new;
            l_run[i] *= alpha;
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[i][c] *= alpha;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const float pu = ex2_approx(s[u] - m_new);  // 0 for a masked row
                l_run[i] += pu;
                float vf[8];
                bf16x8_to_f32(vu[u], vf);
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[i][c] = fmaf(pu, vf[c], acc[i][c]);
            }
        }
    }

    // Warp partial: the 4 key slots of a lane group hold disjoint keys of the
    // same features; l counts each slot once (8 lanes hold the same value).
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        float l = l_run[i];
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float a = acc[i][c];
            a += __shfl_xor_sync(0xffffffffu, a, 8);
            a += __shfl_xor_sync(0xffffffffu, a, 16);
            acc[i][c] = a;
        }
        if (lane < 8) {
#pragma unroll
            for (int c = 0; c < 8; ++c) sm.w_o[warp][i][part * 8 + c] = acc[i][c];
        }
        if (lane == 0) {
            sm.w_m[warp][i] = m_run[i];
            sm.w_l[warp][i] = l;
        }
    }
    __syncthreads();

    // CTA partial: thread t merges feature (t % 64) of query rows t / 64, +2, ...
    for (int idx = threadIdx.x; idx < NQ * HD; idx += kThreads) {
        const int i = idx / HD, c = idx - i * HD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.w_m[w][i]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float f = merge_weight(sm.w_m[w][i], M);
            L += f * sm.w_l[w][i];
            O += f * sm.w_o[w][i][c];
        }
        sm.c_o[i][c] = O;
        if (c == 0) {
            sm.c_m[i] = M;
            sm.c_l[i] = L;
        }
    }
    // Every CTA's partial is complete and visible to the cluster.
    cluster_sync();

    if (split == 0) {
        for (int idx = threadIdx.x; idx < p.Tq * HD; idx += kThreads) {
            const int i = idx / HD, c = idx - i * HD;
            float ms[kSplits];
            float M = -INFINITY;
#pragma unroll
            for (int r = 0; r < kSplits; ++r) {
                ms[r] = dsmem_ld(dsmem_addr(&sm.c_m[i], r));
                M = fmaxf(M, ms[r]);
            }
            float L = 0.f, O = 0.f;
#pragma unroll
            for (int r = 0; r < kSplits; ++r) {
                const float f = merge_weight(ms[r], M);
                L += f * dsmem_ld(dsmem_addr(&sm.c_l[i], r));
                O += f * dsmem_ld(dsmem_addr(&sm.c_o[i][c], r));
            }
            o[(bh * p.Tq + i) * HD + c] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
        }
    }
    // Keep every CTA's shared memory alive until rank 0 has read it.
    cluster_sync();
}

template <int NQ>
cudaError_t launch_nq(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                      __nv_bfloat16 *o, const DecodeParams &p, cudaStream_t stream) {
    const long long bh = static_cast<long long>(p.B) * p.H;
    decode_bf16_kernel<NQ><<<static_cast<unsigned>(bh * kSplits), kThreads, 0, stream>>>(q, k, v, o, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_bf16(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                               const __nv_bfloat16 *v, __nv_bfloat16 *o, const DecodeParams &p,
                               cudaStream_t stream) {
    if (p.Tq <= 1) return launch_nq<1>(q, k, v, o, p, stream);
    if (p.Tq <= 2) return launch_nq<2>(q, k, v, o, p, stream);
    if (p.Tq <= 4) return launch_nq<4>(q, k, v, o, p, stream);
    if (p.Tq <= kDecodeMaxRows) return launch_nq<kDecodeMaxRows>(q, k, v, o, p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace mha
