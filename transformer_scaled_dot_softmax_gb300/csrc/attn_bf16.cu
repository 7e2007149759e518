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
//   warp 8      TMA producer: Q0, Q1 once; K_j and V_j together into a
//               4-stage ring (one barrier per stage for both tiles).
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
// Score tiles rotate through three tensor-memory buffers (S_t(j) uses buffer
// (2j + t) mod 3), so the MMA warp can compute the next score tile of a
// query tile before the current P.V product of that tile has been issued:
// it issues S_0(j+1), PV_0(j), S_1(j+1), PV_1(j), ...  While one softmax
// group works on S_t(j+1) the tensor cores still hold PV_t(j), S_u(j+1),
// PV_u(j) and S_t(j+2) of queued work.  Every M=128 MMA costs at least ~64
// cycles whatever its N, so PV (N = 64) runs at half rate; the queue depth is
// what keeps the pipe busy.
//
// Handshakes are per score buffer: "S in buffer b is ready" and "P in buffer
// b is ready".  A buffer's next use needs the MMA warp to have consumed the
// current one, so neither barrier can run two phases ahead of its waiter.
//
// The running maximum is rescaled in O_t only when it grows by more than 2^8
// (otherwise the stale maximum is kept; the probabilities then stay below
// 256, exact in fp32 and fine in bf16), decided per row.  A rescale at tile j
// needs PV_t(j-1) complete: it waits for the release of tile j-1's K/V stage,
// which is committed after both products of that tile.
//
// Tensor memory (512 columns): S buffers [0,128), [128,256), [256,384);
// O0 [384,448), O1 [448,512).  P overwrites the first 64 columns of its S
// buffer.
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace mha {
namespace {

constexpr int BM = 128;        // query rows per tile
constexpr int BN = 128;        // keys per tile
constexpr int HD = kAttnHeadDim;
constexpr int NQ = 2;          // query tiles per CTA
constexpr int STAGES = 4;      // K/V ring depth
constexpr int kThreads = 320;  // 8 softmax warps + load warp + MMA warp
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTileBytes = BM * HD * 2;  // 16 KiB, one 128 x 64 bf16 tile
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 3;                    // score buffers in tensor memory
constexpr float kRescaleThreshold = 8.0f;    // log2 units

// Score slots are numbered in issue order over the (tile j, query tile t)
// pairs that exist (query tile t has n_t key tiles): slot u uses buffer
// u mod 3 (128 columns each) for the (u / 3)-th time.
__device__ __forceinline__ int score_slot(int j, int t, int n0, int n1) {
    return min(j, n0) + min(j, n1) + ((t == 1 && j < n0) ? 1 : 0);
}
__device__ __forceinline__ uint32_t s_col(int u) { return 128u * static_cast<uint32_t>(u % kSBufs); }
__device__ __forceinline__ uint32_t o_col(int t) { return 384u + 64u * static_cast<uint32_t>(t); }

struct __align__(1024) SmemAttn {
    uint8_t q[NQ][kTileBytes];
    uint8_t k[STAGES][kTileBytes];
    uint8_t v[STAGES][kTileBytes];
    uint64_t q_full;
    uint64_t kv_full[STAGES];
    uint64_t kv_empty[STAGES];
    uint64_t s_full[kSBufs];
    uint64_t p_full[kSBufs];
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
            mbar_init(&sm.kv_full[i], 1);
            mbar_init(&sm.kv_empty[i], 1);
        }
        for (int b = 0; b < kSBufs; ++b) {
            mbar_init(&sm.s_full[b], 1);
            mbar_init(&sm.p_full[b], BM / 32);  // one arrival per softmax warp
        }
        for (int t = 0; t < NQ; ++t) mbar_init(&sm.o_final[t], 1);
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
                mbar_arrive_expect_tx(&sm.kv_full[st], 2 * kTileBytes);
                tma_load_3d(&tmap_k, &sm.kv_full[st], sm.k[st], 0, j * BN, bh);
                tma_load_3d(&tmap_v, &sm.kv_full[st], sm.v[st], 0, j * BN, bh);
                issued = j + 1;
            }
            // Let every copy still in flight land before the CTA exits (on the
            // normal path these phases completed long ago).
            mbar_wait_drain(&sm.q_full, 0);
            for (int j = max(0, issued - STAGES); j < issued; ++j)
                mbar_wait_drain(&sm.kv_full[j % STAGES], (j / STAGES) & 1);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && n_kv > 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(BM, HD, false, true);
            const int n0 = n_tiles[0], n1 = n_tiles[1];
            // Shared-memory descriptors, built once.  Tiles of one kind are
            // contiguous, so stage st adds st * 16 KiB (>> 4 = 1024) to the
            // start-address field; a K step of 16 adds 32 bytes (2) within a
            // K-major row and 16 V rows (2 KiB, 128) for the MN-major V tile.
            const uint64_t q_desc0 = smem_desc_sw128(smem_u32(sm.q[0]), 16, 1024);
            const uint64_t k_desc0 = smem_desc_sw128(smem_u32(sm.k[0]), 16, 1024);
            const uint64_t v_desc0 = smem_desc_sw128(smem_u32(sm.v[0]), 1024, 1024);
            constexpr uint64_t kTileDesc = kTileBytes >> 4;

            // One group per query tile t: S_t(j_s) (if has_s) and PV_t(j_pv)
            // (if has_pv), interleaved so the PV chain (one accumulator) and
            // the S chain overlap in the tensor pipe.  The group opens with
            // two PV MMAs: the S it carries overwrites a buffer the previous
            // group's PV read, and the gap keeps that reuse off the critical
            // path.  The S-ready commit follows the last S MMA (it also
            // covers the PV MMAs issued before it).
            auto issue_group = [&](int t, bool has_s, int st_s, int j_s, bool has_pv, int st_pv,
                                   int j_pv) {
                const int us = has_s ? score_slot(j_s, t, n0, n1) : 0;
                const int up = has_pv ? score_slot(j_pv, t, n0, n1) : 0;
                const uint32_t d_s = tmem + s_col(us);
                const uint32_t a_p = tmem + s_col(up);
                const uint32_t d_o = tmem + o_col(t);
                const uint64_t qd = q_desc0 + static_cast<uint64_t>(t) * kTileDesc;
                const uint64_t kd = k_desc0 + static_cast<uint64_t>(st_s) * kTileDesc;
                const uint64_t vd = v_desc0 + static_cast<uint64_t>(st_pv) * kTileDesc;
                const uint32_t acc0 = j_pv > 0 ? 1u : 0u;
                // schedule: PV0 PV1 S0 PV2 S1 PV3 S2 PV4 S3 [commit] PV5 PV6 PV7
#pragma unroll
                for (int step = 0; step < 13; ++step) {
                    constexpr int kind_tab[13] = {0, 0, 1, 0, 1, 0, 1, 0, 1, 2, 0, 0, 0};
                    constexpr int idx_tab[13] = {0, 1, 0, 2, 1, 3, 2, 4, 3, 0, 5, 6, 7};
                    const int kind = kind_tab[step], i = idx_tab[step];
                    if (kind == 0 && has_pv)
                        mma_bf16_ts(d_o, a_p + 8 * i, vd + 128 * i, idesc_o, (i > 0) ? 1u : acc0);
                    else if (kind == 1 && has_s)
                        mma_bf16_ss(d_s, qd + 2 * i, kd + 2 * i, idesc_s, i > 0 ? 1u : 0u);
                    else if (kind == 2 && has_s)
                        mma_commit(&sm.s_full[us % kSBufs]);
                }
            };
            // P of query tile t, key tile j is ready.
            auto wait_p = [&](int t, int j) {
                const int u = score_slot(j, t, n0, n1);
                return mbar_wait(&sm.p_full[u % kSBufs], (u / kSBufs) & 1, ab);
            };
            // Each wait sits right after an MMA group has been issued, so the
            // tensor pipe has queued work while this thread polls.
            auto wait_kv = [&](int j) {
                return mbar_wait(&sm.kv_full[j % STAGES], (j / STAGES) & 1, ab);
            };
            bool ok = mbar_wait(&sm.q_full, 0, ab) && wait_kv(0);
            if (ok) {
                tc_fence_after_sync();
                if (n0 > 0) issue_group(0, true, 0, 0, false, 0, 0);
                if (n1 > 0) issue_group(1, true, 0, 0, false, 0, 0);
                if (n_kv > 1) ok = wait_kv(1);
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                const int st = j % STAGES;
                const int st1 = (j + 1) % STAGES;
                const bool next0 = j + 1 < n0, next1 = j + 1 < n1;
                const bool pv0 = j < n0, pv1 = j < n1;
                // K/V of tiles j and j+1 are resident (waited one group ago).
                // Tile 0: S_0(j+1) looks ahead into the buffer PV_1(j-1) has
                // already consumed; PV_0(j) needs P_0(j).
                if (pv0 && !(ok = wait_p(0, j))) break;
                tc_fence_after_sync();
                issue_group(0, next0, st1, j + 1, pv0, st, j);
                if (pv0 && j == n0 - 1) mma_commit(&sm.o_final[0]);
                // Tile 1: S_1(j+1) reuses the buffer of P_0(j), read by the
                // group just issued (tensor-core operations of one thread run
                // in order).
                if (pv1 && !(ok = wait_p(1, j))) break;
                tc_fence_after_sync();
                issue_group(1, next1, st1, j + 1, pv1, st, j);
                if (pv1 && j == n1 - 1) mma_commit(&sm.o_final[1]);
                mma_commit(&sm.kv_empty[st]);
                if (j + 2 < n_kv && !(ok = wait_kv(j + 2))) break;
            }
            // Always wait (time-bounded, whatever the abort state) until every
            // MMA this thread issued has completed: tensor memory is released
            // and the CTA exits only after that.
            mma_commit(&sm.drain);
            mbar_wait_drain(&sm.drain, 0);
        }
    } else {
        // --------------------------------------------------------- softmax
        const int t = warp >> 2;
        const uint32_t lane_base = static_cast<uint32_t>(warp & 3) * 32;
        const int r = static_cast<int>(lane_base) + lane;  // row in tile = TMEM lane
        const int row = q0 + t * BM + r;                   // query index
        const uint32_t tl = tmem_addr(tmem, lane_base, 0);
        const uint32_t to = tl + o_col(t);
        const int nt = t == 0 ? n_tiles[0] : n_tiles[1];
        const float C = p.scale_log2;
        const int row_lim = causal ? min(kv_len, row + 1) : kv_len;  // keys < row_lim visible
        const int tile_row_lo = q0 + t * BM;
        float m_run = -INFINITY;
        float l_run = 0.f;
        bool ok = true;

        for (int j = 0; j < nt; ++j) {
            const int u = score_slot(j, t, n_tiles[0], n_tiles[1]);
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&sm.s_full[u % kSBufs], (u / kSBufs) & 1, ab));
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t ts = tl + s_col(u);
            uint32_t s0[32], s1[32], s2[32], s3[32];
            tmem_ld32(ts + 0, s0);
            tmem_ld32(ts + 32, s1);
            tmem_ld32(ts + 64, s2);
            tmem_ld32(ts + 96, s3);
            tmem_ld_wait(s0);
            reg_fence32(s1);
            reg_fence32(s2);
            reg_fence32(s3);

            // In-tile mask: only tiles that reach past the padding length or
            // the diagonal need it (tile-uniform branch).  Keys with index
            // >= row_lim get -inf, i.e. weight exactly zero.
            const int k0 = j * BN;
            if ((k0 + BN > kv_len) || (causal && k0 + BN - 1 > tile_row_lo)) {
                const int lim = row_lim - k0;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    if (c >= lim) s0[c] = f2u(-INFINITY);
                    if (c + 32 >= lim) s1[c] = f2u(-INFINITY);
                    if (c + 64 >= lim) s2[c] = f2u(-INFINITY);
                    if (c + 96 >= lim) s3[c] = f2u(-INFINITY);
                }
            }

            // Row maximum of the tile: eight independent chains of three-input
            // maxima, then a small tree.
            float tm[8];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                tm[i] = fmaxf(u2f(s0[i]), u2f(s0[i + 2]));
                tm[2 + i] = fmaxf(u2f(s1[i]), u2f(s1[i + 2]));
                tm[4 + i] = fmaxf(u2f(s2[i]), u2f(s2[i + 2]));
                tm[6 + i] = fmaxf(u2f(s3[i]), u2f(s3[i + 2]));
            }
#pragma unroll
            for (int c = 4; c < 32; c += 4) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    tm[i] = fmax3(tm[i], u2f(s0[c + i]), u2f(s0[c + i + 2]));
                    tm[2 + i] = fmax3(tm[2 + i], u2f(s1[c + i]), u2f(s1[c + i + 2]));
                    tm[4 + i] = fmax3(tm[4 + i], u2f(s2[c + i]), u2f(s2[c + i + 2]));
                    tm[6 + i] = fmax3(tm[6 + i], u2f(s3[c + i]), u2f(s3[c + i + 2]));
                }
            }
            tm[0] = fmax3(tm[0], tm[1], tm[2]);
            tm[3] = fmax3(tm[3], tm[4], tm[5]);
            tm[0] = fmax3(tm[0], tm[3], fmaxf(tm[6], tm[7]));

            // Running maximum: keep the stale one unless it grew by > 2^8.
            // The decision is per row, so a row's result never depends on
            // another row's scores; the warp only shares the tensor-memory
            // access (rows that keep their maximum scale O by exactly 1).
            const float m_new = fmaxf(m_run, tm[0]);
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

            // P = 2^(s*c - m*c) in bf16 over the first 64 columns of the
            // buffer (column c holds keys 2c, 2c+1; chunk q of 32 scores
            // becomes P columns [16q, 16q+16), all already read).
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#define MHA_EXP_CHUNK(SRC, COL)                                               \
            {                                                                 \
                uint32_t pk[16];                                              \
                _Pragma("unroll") for (int c = 0; c < 16; ++c) {              \
                    const float e0 = ex2_approx(fmaf(u2f(SRC[2 * c]), C, -mc));     \
                    const float e1 = ex2_approx(fmaf(u2f(SRC[2 * c + 1]), C, -mc)); \
                    acc[(2 * c) & 7] += e0;                                   \
                    acc[(2 * c + 1) & 7] += e1;                               \
                    pk[c] = pack_bf16x2(e0, e1);                              \
                }                                                             \
                tmem_st16(ts + (COL), pk);                                    \
            }
            MHA_EXP_CHUNK(s0, 0)
            MHA_EXP_CHUNK(s1, 16)
            MHA_EXP_CHUNK(s2, 32)
            MHA_EXP_CHUNK(s3, 48)
#undef MHA_EXP_CHUNK
            l_run += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));

            if (rescale) {
                // O_t must hold exactly sum_{j' < j} P V: wait for the
                // release of tile j-1's stage (committed after PV_0(j-1) and
                // PV_1(j-1)).  Its next release needs P_t(j), which this
                // thread has not yet published, so the parity cannot alias.
                ok = __all_sync(0xffffffffu, mbar_wait(&sm.kv_empty[(j - 1) % STAGES],
                                                       ((j - 1) / STAGES) & 1, ab));
                if (!ok) {
                    tmem_st_wait();  // no tensor-memory store may outlive the CTA
                    break;
                }
                tc_fence_after_sync();
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
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.p_full[u % kSBufs]);
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
