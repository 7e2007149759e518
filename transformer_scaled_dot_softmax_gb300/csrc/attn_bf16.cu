// attn_bf16.cu -- fused scaled dot-product attention forward for sm_103a.
//
// Computes, per (batch b, head h), O = softmax(scale * Q K^T + mask) V
// ("Attention Is All You Need" (azimuth.plus), "The idea: every word queries
// every word"; aiany.app Step 6, matrix form S = QK^T/sqrt(d_k),
// A = softmax(S), Z = AV) without ever writing S or A to global memory: the
// softmax is taken online over 128-key tiles (running row maximum m and row
// sum l, rescaling the partial output when m grows), which reaches the same
// result up to rounding order.
//
// One CTA owns 256 query rows of one (b, h) as two 128-row tiles Q0, Q1 and
// streams the visible K/V tiles through shared memory:
//
//   warp 8      TMA producer: Q0, Q1 once; K_j, V_j into a 3-stage ring.
//   warp 9      MMA issuer (one thread): S_t = Q_t K_j^T and O_t += P_t V_j
//               on the tensor cores (tcgen05.mma kind::f16, fp32 accumulators
//               in tensor memory).  P_t is read straight from tensor memory.
//   warps 0-3   softmax for Q0, warps 4-7 softmax for Q1: one thread per
//               query row (= tensor-memory lane).  Each thread loads its
//               128 scores, applies the causal / key-padding mask in-tile
//               (masked score = -inf, i.e. exactly zero weight: aiany.app
//               Step 10; notebook chapter "Masked Attention in the Decoder"),
//               updates m and l, writes P = bf16(2^(s*c - m*c)) back over its
//               scores, and finally normalises O by 1/l and stores it.
//
// The MMA warp issues PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), ... so that while
// one softmax warpgroup works on its tile the tensor cores run the other
// group's two products (ping-pong).  A tcgen05.commit arrives once every
// earlier MMA of the issuing thread has completed, so "S_t(j+1) is full"
// also means "PV_t(j) is done": the softmax group may then rescale O_t in
// tensor memory without another barrier.  O_t is only rescaled when the row
// maximum has grown by more than 2^8 (otherwise the stale maximum is kept;
// the probabilities then stay below 256, exact in fp32 and fine in bf16).
//
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,320),
// O1 [320,384).  P_t (bf16 pairs) overwrites the first 64 columns of S_t.
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace mha {
namespace {

constexpr int BM = 128;        // query rows per tile
constexpr int BN = 128;        // keys per tile
constexpr int HD = kAttnHeadDim;
constexpr int NQ = 2;          // query tiles per CTA
constexpr int STAGES = 3;      // K/V ring depth
constexpr int kThreads = 320;  // 8 softmax warps + load warp + MMA warp
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTileBytes = BM * HD * 2;  // 16 KiB, one 128 x 64 bf16 tile
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;    // log2 units

__device__ __forceinline__ uint32_t s_col(int t) { return t == 0 ? 0u : 128u; }
__device__ __forceinline__ uint32_t o_col(int t) { return t == 0 ? 256u : 320u; }

struct __align__(1024) SmemAttn {
    uint8_t q[NQ][kTileBytes];
    uint8_t k[STAGES][kTileBytes];
    uint8_t v[STAGES][kTileBytes];
    uint64_t q_full;
    uint64_t k_full[STAGES];
    uint64_t v_full[STAGES];
    uint64_t kv_empty[STAGES];
    uint64_t s_full[NQ];
    uint64_t p_full[NQ];
    uint64_t o_final[NQ];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    SmemAttn &sm = *reinterpret_cast<SmemAttn *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int qb = p.num_qblocks - 1 - static_cast<int>(blockIdx.y);  // longest first
    const int b = bh / p.H;
    const int hh = bh - b * p.H;
    const int q0 = qb * (NQ * BM);
    const bool causal = (p.mask & kMaskCausalBit) != 0;

    // Visible key range of each query tile.
    int kv_len = p.Tk;
    if ((p.mask & kMaskPaddingBit) && p.key_lens) kv_len = min(max(p.key_lens[b], 0), p.Tk);
    int n_tiles[NQ];
#pragma unroll
    for (int t = 0; t < NQ; ++t) {
        const int row_lo = q0 + t * BM;
        int end = kv_len;
        if (row_lo >= p.Tq) end = 0;
        else if (causal) end = min(end, min(row_lo + BM, p.Tq));
        n_tiles[t] = (end + BN - 1) / BN;
    }
    const int n_kv = max(n_tiles[0], n_tiles[1]);

    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, 1);
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&sm.k_full[i], 1);
            mbar_init(&sm.v_full[i], 1);
            mbar_init(&sm.kv_empty[i], 1);
        }
        for (int t = 0; t < NQ; ++t) {
            mbar_init(&sm.s_full[t], 1);
            mbar_init(&sm.p_full[t], BM);
            mbar_init(&sm.o_final[t], 1);
        }
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kLoadWarp && lane == 0) {
        prefetch_tensormap(&tmap_q);
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    const AbortState ab{&sm.abort_flag, p.status};

    if (warp == kLoadWarp) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0 && n_kv > 0) {
            mbar_arrive_expect_tx(&sm.q_full, NQ * kTileBytes);
            for (int t = 0; t < NQ; ++t) tma_load_3d(&tmap_q, &sm.q_full, sm.q[t], 0, q0 + t * BM, bh);
            int issued = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int st = j % STAGES;
                if (j >= STAGES && !mbar_wait(&sm.kv_empty[st], ((j / STAGES) - 1) & 1, ab)) break;
                mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
                tma_load_3d(&tmap_k, &sm.k_full[st], sm.k[st], 0, j * BN, bh);
                mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
                tma_load_3d(&tmap_v, &sm.v_full[st], sm.v[st], 0, j * BN, bh);
                issued = j + 1;
            }
            if (sm.abort_flag) {
                // Let every copy still in flight land before the CTA exits.
                mbar_wait_drain(&sm.q_full, 0);
                for (int j = max(0, issued - STAGES); j < issued; ++j) {
                    mbar_wait_drain(&sm.k_full[j % STAGES], (j / STAGES) & 1);
                    mbar_wait_drain(&sm.v_full[j % STAGES], (j / STAGES) & 1);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && n_kv > 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(BM, HD, false, true);
            const int n0 = n_tiles[0], n1 = n_tiles[1];
            // S_t = Q_t K^T: A = Q_t (K-major), B = K tile (K-major), K dim 64 = 4 x 16.
            auto issue_s = [&](int t, int st) {
                const uint32_t qa = smem_u32(sm.q[t]);
                const uint32_t ka = smem_u32(sm.k[st]);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    mma_bf16_ss(tmem + s_col(t), smem_desc_sw128(qa + kk * 32, 16, 1024),
                                smem_desc_sw128(ka + kk * 32, 16, 1024), idesc_s, kk > 0);
                mma_commit(&sm.s_full[t]);
            };
            // O_t (+)= P_t V: A = P_t in tensor memory (8 columns per 16 keys),
            // B = V tile (keys x 64, MN-major: 16 keys = 2 swizzle atoms = 2 KiB).
            auto issue_o = [&](int t, int st, int j) {
                const uint32_t va = smem_u32(sm.v[st]);
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_bf16_ts(tmem + o_col(t), tmem + s_col(t) + kk * 8,
                                smem_desc_sw128(va + kk * 2048, kTileBytes, 1024), idesc_o,
                                (j > 0 || kk > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(&sm.q_full, 0, ab) && mbar_wait(&sm.k_full[0], 0, ab);
            if (ok) {
                tc_fence_after_sync();
                if (n0 > 0) issue_s(0, 0);
                if (n1 > 0) issue_s(1, 0);
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                const int st = j % STAGES;
                const bool has_next = j + 1 < n_kv;
                const int st1 = (j + 1) % STAGES;
                if (!(ok = mbar_wait(&sm.v_full[st], (j / STAGES) & 1, ab))) break;
                if (j < n0) {
                    if (!(ok = mbar_wait(&sm.p_full[0], j & 1, ab))) break;
                    tc_fence_after_sync();
                    issue_o(0, st, j);
                    if (j == n0 - 1) mma_commit(&sm.o_final[0]);
                }
                if (has_next) {
                    if (!(ok = mbar_wait(&sm.k_full[st1], ((j + 1) / STAGES) & 1, ab))) break;
                    tc_fence_after_sync();
                    if (j + 1 < n0) issue_s(0, st1);
                }
                if (j < n1) {
                    if (!(ok = mbar_wait(&sm.p_full[1], j & 1, ab))) break;
                    tc_fence_after_sync();
                    issue_o(1, st, j);
                    if (j == n1 - 1) mma_commit(&sm.o_final[1]);
                }
                mma_commit(&sm.kv_empty[st]);
                if (has_next && j + 1 < n1) issue_s(1, st1);
            }
            if (!ok) {
                // Wait (bounded) for the MMAs already issued before tensor
                // memory is released.
                mma_commit(&sm.drain);
                mbar_wait_drain(&sm.drain, 0);
            }
        }
    } else {
        // --------------------------------------------------------- softmax
        const int t = warp >> 2;
        const uint32_t lane_base = static_cast<uint32_t>(warp & 3) * 32;
        const int r = static_cast<int>(lane_base) + lane;  // row in tile = TMEM lane
        const int row = q0 + t * BM + r;                   // query index
        const uint32_t ts = tmem_addr(tmem, lane_base, s_col(t));
        const uint32_t to = tmem_addr(tmem, lane_base, o_col(t));
        const int nt = t == 0 ? n_tiles[0] : n_tiles[1];
        const float C = p.scale_log2;
        const int row_lim = causal ? min(kv_len, row + 1) : kv_len;  // keys < row_lim visible
        const int tile_row_lo = q0 + t * BM;
        float m_run = -INFINITY;
        float l_run = 0.f;
        bool ok = true;

        for (int j = 0; j < nt; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(&sm.s_full[t], j & 1, ab));
            if (!ok) break;
            tc_fence_after_sync();

            // In-tile mask: only tiles that reach past the padding length or
            // the diagonal need it (tile-uniform branch).  Keys with index
            // >= row_lim get -inf, i.e. weight exactly zero.
            const int k0 = j * BN;
            const bool need_mask =
                (k0 + BN > kv_len) || (causal && k0 + BN - 1 > tile_row_lo);
            const int lim = row_lim - k0;

            // Pass 1: row maximum over the 128 scores, read as two halves.
            float mx = -INFINITY;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                uint32_t a[32], b2[32];
                tmem_ld32(ts + half * 64, a);
                tmem_ld32(ts + half * 64 + 32, b2);
                tmem_ld_wait(a);
                reg_fence32(b2);
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        if (half * 64 + c >= lim) a[c] = f2u(-INFINITY);
                        if (half * 64 + 32 + c >= lim) b2[c] = f2u(-INFINITY);
                    }
                }
#pragma unroll
                for (int c = 0; c < 32; ++c) mx = fmaxf(mx, fmaxf(u2f(a[c]), u2f(b2[c])));
            }

            // Running maximum: keep the stale one unless it grew by > 2^8.
            // The decision is per row, so a row's result never depends on
            // another row's scores; the warp only shares the tensor-memory
            // access (rows that keep their maximum scale O by exactly 1).
            const float m_new = fmaxf(m_run, mx);
            const bool grow = j > 0 && (m_new - m_run) * C > kRescaleThreshold;
            const bool rescale = __any_sync(0xffffffffu, grow);
            float alpha = 1.f;
            if (j == 0) {
                m_run = m_new;
            } else if (grow) {
                alpha = ex2_approx((m_run - m_new) * C);
                l_run *= alpha;
                m_run = m_new;
            }
            const float mc = m_run * C;

            // Pass 2: P = 2^(s*c - m*c) in bf16, written over the scores: half
            // h reads score columns [64h, 64h+64) and writes P columns
            // [32h, 32h+32) (column c holds keys 2c and 2c+1), which only
            // overwrites scores already consumed.
            float sum0 = 0.f, sum1 = 0.f;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                uint32_t a[32], b2[32];
                tmem_ld32(ts + half * 64, a);
                tmem_ld32(ts + half * 64 + 32, b2);
                tmem_ld_wait(a);
                reg_fence32(b2);
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        if (half * 64 + c >= lim) a[c] = f2u(-INFINITY);
                        if (half * 64 + 32 + c >= lim) b2[c] = f2u(-INFINITY);
                    }
                }
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float e0 = ex2_approx(fmaf(u2f(a[2 * c]), C, -mc));
                    const float e1 = ex2_approx(fmaf(u2f(a[2 * c + 1]), C, -mc));
                    const float e2 = ex2_approx(fmaf(u2f(b2[2 * c]), C, -mc));
                    const float e3 = ex2_approx(fmaf(u2f(b2[2 * c + 1]), C, -mc));
                    sum0 += e0 + e1;
                    sum1 += e2 + e3;
                    pk[c] = pack_bf16x2(e0, e1);
                    pk[c + 16] = pack_bf16x2(e2, e3);
                }
                tmem_st32(ts + half * 32, pk);
            }
            l_run += sum0 + sum1;
            if (rescale) {
                // O_t holds sum_{j' < j} P V; all those MMAs are complete
                // (the commit that signalled S_t(j) covers them).
                uint32_t o0[32], o1[32];
                tmem_ld32(to, o0);
                tmem_ld32(to + 32, o1);
                tmem_ld_wait(o0);
                reg_fence32(o1);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    o0[c] = f2u(u2f(o0[c]) * alpha);
                    o1[c] = f2u(u2f(o1[c]) * alpha);
                }
                tmem_st32(to, o0);
                tmem_st32(to + 32, o1);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&sm.p_full[t]);
        }

        // ----------------------------------------------------------- epilogue
        if (ok && nt > 0) ok = __all_sync(0xffffffffu, mbar_wait(&sm.o_final[t], 0, ab));
        if (ok) {
            uint32_t o0[32], o1[32];
            if (nt > 0) {
                tc_fence_after_sync();
                tmem_ld32(to, o0);
                tmem_ld32(to + 32, o1);
                tmem_ld_wait(o0);
                reg_fence32(o1);
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) o0[c] = o1[c] = 0u;
            }
            if (row < p.Tq) {
                const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
                uint32_t packed[32];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    packed[c] = pack_bf16x2(u2f(o0[2 * c]) * inv, u2f(o0[2 * c + 1]) * inv);
                    packed[c + 16] = pack_bf16x2(u2f(o1[2 * c]) * inv, u2f(o1[2 * c + 1]) * inv);
                }
                __nv_bfloat16 *dst = p.o + b * p.o_stride_b + hh * p.o_stride_h +
                                     static_cast<long long>(row) * p.o_stride_t;
                uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    d4[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2],
                                       packed[4 * c + 3]);
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_attn_bf16(const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, const AttnParams &p, cudaStream_t stream) {
    const size_t smem = sizeof(SmemAttn) + 1024;
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_bf16_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(p.B * p.H), static_cast<unsigned>(p.num_qblocks));
    attn_fwd_bf16_kernel<<<grid, kThreads, smem, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace mha
