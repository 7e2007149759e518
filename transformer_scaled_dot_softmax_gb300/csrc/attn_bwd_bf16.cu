// attn_bwd_bf16.cu -- gradients of scaled dot-product attention for sm_103a.
//
// With S = scale Q K^T (masked entries -inf), P = softmax(S) row-wise,
// O = P V and the output gradient dO, the chain rule gives
//   dV = P^T dO,  dP = dO V^T,  dS = P (.) (dP - D),  D_i = sum_c dO_ic O_ic,
//   dQ = scale dS K,  dK = scale dS^T Q
// (D_i = sum_j P_ij dP_ij, the softmax Jacobian's row term).  The weights are
// not stored by the forward pass; they are recomputed from the forward's
// per-row log-sum-exp: P_ij = exp(S_ij - lse_i).
//
// Three launches:
//   attn_bwd_pre   D_i, -lse_i in log2 units (-inf for a padded or fully masked
//                  row, so its weights are 0), and a zeroed fp32 dQ accumulator;
//   attn_bwd_main  one CTA per (b, h, block of 128 keys): keeps dK and dV of
//                  its keys in tensor memory and walks the query blocks that
//                  see them (see the kernel comment);
//   attn_bwd_post  dQ = bf16(scale * accumulator).
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace mha {
namespace {

constexpr int HD = kAttnHeadDim;  // 64
constexpr int BQ = 128;           // query rows per block
constexpr int BKB = 128;          // keys per CTA
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------ pre and post
// One thread per 8 features of a row; rows past Tq (padding up to a whole
// query block) get lse = +inf, D = 0.
__global__ void attn_bwd_pre(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
                             const float *__restrict__ lse, float *__restrict__ nlse2,
                             float *__restrict__ dvec, float *__restrict__ dq_acc, long long BH,
                             int Tq, int Tq_pad) {
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long row = t >> 3;  // over BH * Tq_pad
    const int part = static_cast<int>(t & 7);
    // no early return: the row sum below is a full-warp shuffle
    const bool valid = row < BH * Tq_pad;
    const long long bh = valid ? row / Tq_pad : 0;
    const int i = valid ? static_cast<int>(row - bh * Tq_pad) : Tq;
    float acc = 0.f;
    if (i < Tq) {
        const long long src = (bh * Tq + i) * HD + part * 8;
        const uint4 a = *reinterpret_cast<const uint4 *>(o + src);
        const uint4 g = *reinterpret_cast<const uint4 *>(dout + src);
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc = fmaf(__uint_as_float(aw[e] << 16), __uint_as_float(gw[e] << 16), acc);
            acc = fmaf(__uint_as_float(aw[e] & 0xffff0000u), __uint_as_float(gw[e] & 0xffff0000u), acc);
        }
    }
    // reduce over the 8 threads of the row (consecutive lanes)
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if (!valid) return;
    float4 *z = reinterpret_cast<float4 *>(dq_acc + row * HD + part * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (part == 0) {
        dvec[row] = acc;
        float l = -INFINITY;
        if (i < Tq) {
            const float x = lse[bh * Tq + i];
            l = x == -INFINITY ? -INFINITY : -x * kLog2e;
        }
        nlse2[row] = l;
    }
}

// The dQ accumulator of a query block j of head bh is 128 rows x 64 fp32 at
// (bh Tq_pad + 128 j) 64, stored as four 8 KiB quarters (rows 32w .. 32w+31),
// each ordered [16-byte chunk x of the row][row within the quarter][4 floats]:
// the order in which a dQ warp stages its rows without shared-memory bank
// conflicts, so that one untiled bulk reduction adds the whole quarter.
__device__ __forceinline__ long long dq_acc_index(long long bh, int Tq_pad, int i, int chunk) {
    return (bh * Tq_pad + (i & ~31)) * HD + chunk * 128 + (i & 31) * 4;
}

// One thread per 8 features of a row; a warp takes 32 consecutive rows of one
// feature group (coalesced accumulator reads).
__global__ void attn_bwd_post(const float *__restrict__ dq_acc, __nv_bfloat16 *__restrict__ dq,
                              long long BH, int Tq, int Tq_pad, float scale) {
    pdl_wait();  // the accumulator is complete once the main kernel is
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long grp = t >> 8;  // 32-row group over BH * Tq_pad / 32
    const int part = static_cast<int>((t >> 5) & 7);
    const int groups = Tq_pad >> 5;
    if (grp >= BH * groups) return;
    const long long bh = grp / groups;
    const int i = static_cast<int>(grp - bh * groups) * 32 + static_cast<int>(t & 31);
    if (i >= Tq) return;
    const float4 a = *reinterpret_cast<const float4 *>(dq_acc + dq_acc_index(bh, Tq_pad, i, 2 * part));
    const float4 b = *reinterpret_cast<const float4 *>(dq_acc + dq_acc_index(bh, Tq_pad, i, 2 * part + 1));
    const uint4 w = make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                               pack_bf16x2(b.x * scale, b.y * scale), pack_bf16x2(b.z * scale, b.w * scale));
    *reinterpret_cast<uint4 *>(dq + (bh * Tq + i) * HD + part * 8) = w;
}

// P^T and dS^T of N of one thread's query columns for its key:
// p = 2^(s c - lse2) (nlse2 = -lse2), ds = p (dp - D), as bf16 pairs, in
// packed fp32 pair arithmetic.  kMasked: column e counts iff e >= lim.
template <int N, bool kMasked>
__device__ __forceinline__ void softmax_terms(const uint32_t (&sv)[N], const uint32_t (&dp)[N],
                                              const float *nlse2, const float *dvec, float C, int lim,
                                              uint32_t (&pk)[N / 2], uint32_t (&dsk)[N / 2]) {
    const uint64_t C2 = f32x2_pack(C, C);
#pragma unroll
    for (int g = 0; g < N / 4; ++g) {
        const float4 l4 = reinterpret_cast<const float4 *>(nlse2)[g];
        const float4 d4 = reinterpret_cast<const float4 *>(dvec)[g];
        const uint64_t nl[2] = {f32x2_pack(l4.x, l4.y), f32x2_pack(l4.z, l4.w)};
        const uint64_t d[2] = {f32x2_pack(d4.x, d4.y), f32x2_pack(d4.z, d4.w)};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int e = 4 * g + 2 * h;
            float x0, x1;
            f32x2_unpack(fma_f32x2(f32x2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), C2, nl[h]), x0, x1);
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            if (kMasked) {
                if (e < lim) p0 = 0.f;
                if (e + 1 < lim) p1 = 0.f;
            }
            const uint64_t dd =
                mul_f32x2(f32x2_pack(p0, p1), sub_f32x2(f32x2_pack(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), d[h]));
            float ds0, ds1;
            f32x2_unpack(dd, ds0, ds1);
            pk[2 * g + h] = pack_bf16x2(p0, p1);
            dsk[2 * g + h] = pack_bf16x2(ds0, ds1);
        }
    }
}

// ------------------------------------------------------------------- main
// One CTA = one (b, h) and a block of 128 keys; it walks the query blocks j
// that see any of its keys (all of them, or j >= kb under the causal mask).
// Warp roles (18 warps):
//
//   warp 0      TMA: the K and V blocks once; per query block Q_j, dO_j (3-D
//               tensor maps) and its 128 lse and D values (bulk copies) into
//               a 3-stage ring.
//   warp 1      MMA issuer (whole warp, elected lane), per query block:
//                 (1) S^T  = K Q_j^T     M=128 keys, N=128 queries, K=64
//                 (2) dP^T = V dO_j^T    same shape
//                 (3) dV  += P^T dO_j    M=128 keys, N=64, K=128 queries, A = P^T in
//                                        tensor memory
//                 (4) dK  += dS^T Q_j    same, A = dS^T from shared memory (key
//                                        rows, queries contiguous: K-major)
//                 (5) dQ_j = dS K        M=128 queries, N=64, K=128 keys, A = dS from
//                                        the same shared memory (MN-major)
//               Computing S and dP transposed puts the keys on the
//               tensor-memory lanes, so P^T feeds (3) straight from tensor
//               memory.  Issue order: (1) and (2) of block j+1 as soon as
//               the softmax warps have loaded block j's S^T and dP^T into
//               registers (they overwrite those columns while the terms of
//               block j are still being computed), then (4), (3) and (5) of
//               block j once its terms are written -- no product of block j
//               stands between its softmax terms and block j+1's scores.
//               (4) reads dS^T from shared memory rather than tensor memory
//               for that reason: in tensor memory it would have to sit over
//               dP^T's columns, and (2) of block j+1 would wait for it.
//   warps 2-17  one thread per (key, chunk of 32 queries) -- warp w takes the
//               keys of lane quadrant w%4 and chunk (w-2)/4:
//               P^T = 2^(S^T c - lse_j) (masked: 0), dS^T = P^T (dP^T - D_j),
//               elementwise (lse and D are per-query inputs, no row
//               reduction); P^T written as bf16 into tensor memory, dS into
//               shared memory for (4) and (5) (two buffers: block j+2 reuses
//               block j's, whose (4) and (5) the commit of block j+2's
//               scores, which the warps wait for, already covers).  After
//               block j's terms, the same warps add the
//               dQ_{j-1} partial (warp w: the rows of quadrant w%4, features
//               [16c, 16c+16)) to the fp32 accumulator in global memory with
//               vector reductions, each warp instruction covering 512
//               contiguous bytes of the accumulator's layout (other key blocks
//               add theirs).  At the end chunks 0, 1 write dK (times scale) and
//               chunks 2, 3 dV, 32 features each.
//
// Tensor memory: S^T [0,128), dP^T [128,256), P^T [256,320), dV [320,384),
// dK [384,448), dQ_j [448,512).  P^T has columns of its own and dS^T stays
// in shared memory, so the next block's scores wait for neither (3) nor (4).
constexpr uint32_t kTile = BQ * HD * 2;  // 16 KiB
constexpr uint32_t kColS = 0, kColDP = 128, kColP = 256, kColDV = 320, kColDK = 384, kColDQ = 448;
constexpr int kBwdThreads = 576;
constexpr int kSoftmaxWarps = 16;
constexpr int kStages = 3;  // Q_j / dO_j / lse_j / D_j ring

struct __align__(1024) SmemBwd {
    uint8_t k[kTile];
    uint8_t v[kTile];
    uint8_t q[kStages][kTile];
    uint8_t g[kStages][kTile];  // dO
    uint8_t ds[2][2 * kTile]; // dS, the A operand of (4) and (5): 2 blocks of 64 queries x 128 key rows
    float nlse2[kStages][BQ];
    float dvec[kStages][BQ];
    uint64_t kv_full;
    uint64_t stage_full[kStages];
    uint64_t q_empty[kStages];  // (1), (4) have read Q_j (and the softmax lse_j, D_j)
    uint64_t g_empty[kStages];  // (2), (3) have read dO_j
    uint64_t sdp_full;   // (1), (2) complete
    uint64_t sdp_read;   // S^T, dP^T loaded into registers (16 warps)
    uint64_t pds_full;   // P^T (tensor memory), dS (shared memory) written (16 warps)
    uint64_t tmem_free;  // (4) of the block complete
    uint64_t p_free;     // (3) complete: the P^T columns reusable
    uint64_t dq_full;    // (5) complete
    uint64_t dq_free;    // dQ_j read (16 warps)
    uint64_t acc_done;   // every product complete
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_main(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_g,
                  const BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    SmemBwd &sm = *reinterpret_cast<SmemBwd *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bh = static_cast<int>(blockIdx.x);
    const int kb = static_cast<int>(blockIdx.y);  // key block 0 (most query blocks when causal) first
    const int b = bh / p.H;
    const int k0 = kb * BKB;
    const bool causal = (p.mask & kMaskCausalBit) != 0;
    int key_hi = p.Tk;  // keys [0, key_hi) exist and are not padding
    if ((p.mask & kMaskPaddingBit) && p.key_lens) key_hi = min(max(p.key_lens[b], 0), p.Tk);
    const int n_qb = (p.Tq + BQ - 1) / BQ;
    // Query i sees key k iff k <= i (causal, top-left aligned): query blocks
    // from k0 / BQ on.
    const int j_begin = causal ? k0 / BQ : 0;
    const int n_j = k0 < key_hi ? max(0, n_qb - j_begin) : 0;

    if (threadIdx.x == 0) {
        mbar_init(&sm.kv_full, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.stage_full[i], 1);
            mbar_init(&sm.q_empty[i], 1);
            mbar_init(&sm.g_empty[i], 1);
        }
        mbar_init(&sm.p_free, 1);
        mbar_init(&sm.sdp_full, 1);
        mbar_init(&sm.sdp_read, kSoftmaxWarps);
        mbar_init(&sm.pds_full, kSoftmaxWarps);
        mbar_init(&sm.tmem_free, 1);
        mbar_init(&sm.dq_full, 1);
        mbar_init(&sm.dq_free, kSoftmaxWarps);
        mbar_init(&sm.acc_done, 1);
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmap_q);
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
        prefetch_tensormap(&tmap_g);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    const AbortState ab{&sm.abort_flag, p.status};
    // Programmatic dependent launch: the next kernel may begin its prologue;
    // nothing below touches global memory written by the kernel before this
    // one until that kernel has completed.
    pdl_launch_dependents();
    pdl_wait();

    if (warp == 0) {
        // -------------------------------------------------------------- TMA
        if (lane == 0 && n_j > 0) {
            mbar_arrive_expect_tx(&sm.kv_full, 2 * kTile);
            if (in_bounds(k0 < p.Tk && bh < p.B * p.H, p.status)) {
                tma_load_3d(&tmap_k, &sm.kv_full, sm.k, 0, k0, bh);
                tma_load_3d(&tmap_v, &sm.kv_full, sm.v, 0, k0, bh);
            }
            int issued = 0;
            for (int t = 0; t < n_j; ++t) {
                const int st = t % kStages, use = t / kStages;
                if (t >= kStages && !mbar_wait(&sm.q_empty[st], (use - 1) & 1, ab)) break;
                const int j = j_begin + t;
                const long long vrow = static_cast<long long>(bh) * p.Tq_pad + j * BQ;
                mbar_arrive_expect_tx(&sm.stage_full[st], 2 * kTile + 2 * BQ * 4);
                // query block j of (B*H, T_q_pad) rows: the row terms are padded
                // to whole blocks, the Q / dO maps clip at T_q
                const bool j_ok = in_bounds(j * BQ < p.Tq && j * BQ + BQ <= p.Tq_pad, p.status);
                if (j_ok) {
                    tma_load_3d(&tmap_q, &sm.stage_full[st], sm.q[st], 0, j * BQ, bh);
                    bulk_load_1d(sm.nlse2[st], p.nlse2 + vrow, BQ * 4, &sm.stage_full[st]);
                    bulk_load_1d(sm.dvec[st], p.dvec + vrow, BQ * 4, &sm.stage_full[st]);
                }
                issued = t + 1;
                // dO_j last: its slot frees later (after (3))
                if (t >= kStages && !mbar_wait(&sm.g_empty[st], (use - 1) & 1, ab)) break;
                if (j_ok) tma_load_3d(&tmap_g, &sm.stage_full[st], sm.g[st], 0, j * BQ, bh);
            }
            mbar_wait_drain(&sm.kv_full, 0);
            for (int x = max(0, issued - kStages); x < issued; ++x)
                mbar_wait_drain(&sm.stage_full[x % kStages], (x / kStages) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA
        if (n_j > 0) {
            constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);  // (1), (2)
            constexpr uint32_t id_kv = idesc_bf16_f32(128, HD, false, true);   // (3), (4)
            constexpr uint32_t id_q = idesc_bf16_f32(128, HD, true, true);     // (5)
            constexpr uint64_t kT = kTile >> 4;
            // K-major operands (a K step of 16 = 32 bytes = 2), MN-major
            // operands (16 rows of 128 bytes = 2 KiB = 128 per K step).
            // One base descriptor (K-major, at sm.k): every operand lies a
            // whole number of 16 KiB tiles further (the address field counts
            // 16-byte units and stays below 2^14), and the MN-major form
            // differs only in the leading byte offset field (1024 bytes
            // instead of 16; 16 KiB between dS's two 64-query blocks).
            const uint64_t k_km = smem_desc_sw128(smem_u32(sm.k), 16, 1024);
            constexpr uint64_t kMn = static_cast<uint64_t>((1024 >> 4) - 1) << 16;
            constexpr uint64_t kDsMn = static_cast<uint64_t>((kTile >> 4) - 1) << 16;
            const uint64_t v_km = k_km + kT;
            const uint64_t q_km = k_km + 2 * kT;
            const uint64_t g_km = k_km + (2 + kStages) * kT;
            const uint64_t ds_km0 = k_km + (2 + 2 * kStages) * kT;
            const uint64_t q_mn = q_km + kMn;
            const uint64_t g_mn = g_km + kMn;
            const uint64_t k_mn = k_km + kMn;
            const uint64_t ds_mn = ds_km0 + kDsMn;
            // (1) and (2) of the block in stage s
            auto score_s = [&](int s) {
                const uint64_t so = static_cast<uint64_t>(s) * kT;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    warp_mma_bf16_ss(tmem + kColS, k_km + 2 * kk, q_km + so + 2 * kk, id_s, kk > 0 ? 1u : 0u);
            };
            auto score_dp = [&](int s) {
                const uint64_t so = static_cast<uint64_t>(s) * kT;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    warp_mma_bf16_ss(tmem + kColDP, v_km + 2 * kk, g_km + so + 2 * kk, id_s, kk > 0 ? 1u : 0u);
            };
            bool ok = warp_wait(&sm.kv_full, 0, ab) && warp_wait(&sm.stage_full[0], 0, ab);
            if (ok) {
                tc_fence_after_sync();
                score_s(0);
                score_dp(0);
                warp_commit(&sm.sdp_full);
            }
            for (int t = 0; ok && t < n_j; ++t) {
                const int st = t % kStages, nst = (t + 1) % kStages;
                const uint64_t so = static_cast<uint64_t>(st) * kT;  // q[st], g[st] stage offset
                if (t + 1 < n_j) {
                    // The next block's scores as soon as the softmax warps
                    // have loaded block t's S^T and dP^T into registers: they
                    // run on the tensor pipe while the softmax terms of block t
                    // are still being computed (the terms go to P^T's own
                    // columns and to shared memory, not over S^T or dP^T).
                    if (!(ok = warp_wait(&sm.sdp_read, t & 1, ab))) break;
                    if (!(ok = warp_wait(&sm.stage_full[nst], ((t + 1) / kStages) & 1, ab))) break;
                    tc_fence_after_sync();
                    score_s(nst);
                    score_dp(nst);
                    warp_commit(&sm.sdp_full);
                }
                if (!(ok = warp_wait(&sm.pds_full, t & 1, ab))) break;
                tc_fence_after_sync();
                // (4) from dS^T in shared memory
                const uint64_t dso = static_cast<uint64_t>(t & 1) * (2 * kT);
#pragma unroll
                for (int kk = 0; kk < BQ / 16; ++kk)
                    warp_mma_bf16_ss(tmem + kColDK, ds_km0 + dso + (kk >> 2) * kT + 2 * (kk & 3),
                                     q_mn + so + 128 * kk, id_kv, (t > 0 || kk > 0) ? 1u : 0u);
                warp_commit(&sm.q_empty[st]);
                warp_commit(&sm.tmem_free);
                // (3) after the next block's scores: P^T has columns of its
                // own, which the softmax warps rewrite only after p_free
#pragma unroll
                for (int kk = 0; kk < BQ / 16; ++kk)
                    warp_mma_bf16_ts(tmem + kColDV, tmem + kColP + 8 * kk, g_mn + so + 128 * kk, id_kv,
                                     (t > 0 || kk > 0) ? 1u : 0u);
                warp_commit(&sm.p_free);
                warp_commit(&sm.g_empty[st]);
                if (t >= 1 && !(ok = warp_wait(&sm.dq_free, (t - 1) & 1, ab))) break;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < BKB / 16; ++kk)
                    warp_mma_bf16_ss(tmem + kColDQ, ds_mn + dso + 128 * kk, k_mn + 128 * kk, id_q,
                                     kk > 0 ? 1u : 0u);
                warp_commit(&sm.dq_full);
                // (4) of this block complete before the next block's
                // scores are issued: it has long finished by then, and the
                // kernel measured slightly faster with the wait than without.
                if (!(ok = warp_wait(&sm.tmem_free, t & 1, ab))) break;
            }
            if (ok) warp_commit(&sm.acc_done);
        }
        warp_commit(&sm.drain);
        mbar_wait_drain(&sm.drain, 0);
    } else if (warp < 2 + kSoftmaxWarps) {
        // ------------------------------------------- per-key softmax terms
        const int c = (warp - 2) >> 2;  // query chunk [32c, 32c + 32)
        const uint32_t lane_base = static_cast<uint32_t>(warp & 3) * 32;
        const int r = static_cast<int>(lane_base) + lane;  // key row in the block
        const int key = k0 + r;
        const bool key_ok = key < key_hi;
        const uint32_t tl = tmem_addr(tmem, lane_base, 0);
        const float C = p.scale_log2;
        // dQ_u of this warp's rows and features [16c, 16c+16): chunks
        // [4c, 4c+4) of the quadrant's accumulator quarter.
        auto add_dq = [&](int u) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait(&sm.dq_full, u & 1, ab))) return false;
            tc_fence_after_sync();
            uint32_t a[16];
            tmem_ld16(tl + kColDQ + 16u * c, a);
            tmem_ld_wait(a);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.dq_free);
            // chunks [4c, 4c+4) of the quadrant's quarter: per chunk the 32
            // lanes' vectors are 512 contiguous bytes
            float *dst = p.dq_acc + (static_cast<long long>(bh) * p.Tq_pad + (j_begin + u) * BQ + lane_base) * HD +
                         512 * c + 4 * lane;
            if (!in_bounds((j_begin + u) * BQ + BQ <= p.Tq_pad && bh < p.B * p.H, p.status)) return true;
#pragma unroll
            for (int x = 0; x < 4; ++x)
                red_add_v4(dst + 128 * x, __uint_as_float(a[4 * x]), __uint_as_float(a[4 * x + 1]),
                           __uint_as_float(a[4 * x + 2]), __uint_as_float(a[4 * x + 3]));
            return true;
        };
        bool ok = true;
        for (int t = 0; t < n_j; ++t) {
            const int st = t % kStages;
            const int q0 = (j_begin + t) * BQ + 32 * c;
            ok = __all_sync(0xffffffffu, mbar_wait(&sm.sdp_full, t & 1, ab)) &&
                 __all_sync(0xffffffffu, mbar_wait(&sm.stage_full[st], (t / kStages) & 1, ab));
            if (!ok) break;
            tc_fence_after_sync();
            // two halves of 16 query columns, 32 registers in flight each
            uint8_t *blk = sm.ds[t & 1] + (c >> 1) * kTile + r * 128;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                const uint32_t col = 32u * c + 16u * h;
                uint32_t sv[16], dp[16];
                tmem_ld16(tl + kColS + col, sv);
                tmem_ld16(tl + kColDP + col, dp);
                // query column e of the half sees the key iff e >= lim
                const int lim = key_ok ? (causal ? key - (q0 + 16 * h) : 0) : 16;
                tmem_ld_wait(sv);
                tmem_ld_wait(dp);
                if (h == 1) {
                    // this warp's S^T and dP^T columns are all in registers
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.sdp_read);
                }
                uint32_t pk[8], dsk[8];
                const float *l2 = sm.nlse2[st] + 32 * c + 16 * h, *dv = sm.dvec[st] + 32 * c + 16 * h;
                if (__all_sync(0xffffffffu, lim <= 0))
                    softmax_terms<16, false>(sv, dp, l2, dv, C, 0, pk, dsk);
                else
                    softmax_terms<16, true>(sv, dp, l2, dv, C, lim, pk, dsk);
                // P^T into its own columns once (3) of the previous block has
                // read them
                if (h == 0 && t >= 1 && !(ok = __all_sync(0xffffffffu, mbar_wait(&sm.p_free, (t - 1) & 1, ab))))
                    break;
                tmem_st8(tl + kColP + 16u * c + 8u * h, pk);
                // dS into shared memory as the A operand of (4) and (5): queries
                // contiguous, 128-byte swizzled rows (16-byte chunk x of key
                // row r at x ^ (r % 8)), 64 queries per 16 KiB block.
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const int chunk = 4 * (c & 1) + 2 * h + x;
                    *reinterpret_cast<uint4 *>(blk + ((chunk ^ (r & 7)) << 4)) =
                        make_uint4(dsk[4 * x], dsk[4 * x + 1], dsk[4 * x + 2], dsk[4 * x + 3]);
                }
            }
            if (!ok) break;
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.pds_full);
            if (t >= 1 && !(ok = add_dq(t - 1))) break;
        }
        if (ok && n_j > 0) ok = add_dq(n_j - 1);
        // dK = scale dS^T Q (chunks 0, 1) and dV = P^T dO (chunks 2, 3) of
        // this block's keys, 32 features per warp.
        if (ok && n_j > 0) ok = __all_sync(0xffffffffu, mbar_wait(&sm.acc_done, 0, ab));
        // `ok` and n_j are warp-uniform: every lane issues the tensor-memory
        // load; only the stores depend on the key row.
        if (ok) {
            const bool is_dv = c >= 2;
            const int f0 = 32 * (c & 1);  // first feature
            uint32_t a[32];
            if (n_j > 0) {
                tc_fence_after_sync();
                __syncwarp();
                tmem_ld32(tl + (is_dv ? kColDV : kColDK) + f0, a);
                tmem_ld_wait(a);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) a[e] = 0u;
            }
            if (key < p.Tk && in_bounds(key >= 0 && bh < p.B * p.H, p.status)) {
                const float f = is_dv ? 1.f : p.scale;
                __nv_bfloat16 *dst = (is_dv ? p.dv : p.dk) + (static_cast<long long>(bh) * p.Tk + key) * HD + f0;
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(a[2 * e]) * f, __uint_as_float(a[2 * e + 1]) * f);
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    reinterpret_cast<uint4 *>(dst)[x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
            }
        }
        if (!ok) tmem_st_wait();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

size_t bwd_workspace_bytes(long long BH, int Tq) {
    const long long Tq_pad = (Tq + BQ - 1) / BQ * BQ;
    const size_t rows = static_cast<size_t>(BH) * Tq_pad;
    auto r256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    return r256(rows * HD * 4) + 2 * r256(rows * 4);
}

cudaError_t launch_attn_bwd_bf16(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                 const CUtensorMap &tg, const __nv_bfloat16 *o,
                                 const __nv_bfloat16 *dout, const float *lse, __nv_bfloat16 *dq,
                                 BwdParams p, void *workspace, cudaStream_t stream) {
    const long long BH = static_cast<long long>(p.B) * p.H;
    const size_t rows = static_cast<size_t>(BH) * p.Tq_pad;
    auto r256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *nlse2 = reinterpret_cast<float *>(ws + r256(rows * HD * 4));
    float *dvec = reinterpret_cast<float *>(ws + r256(rows * HD * 4) + r256(rows * 4));
    p.dq_acc = reinterpret_cast<float *>(ws);
    p.nlse2 = nlse2;
    p.dvec = dvec;
    cudaError_t e = cudaSuccess;
    const long long pre_threads = static_cast<long long>(rows) * 8;
    if (pre_threads > 0) {
        attn_bwd_pre<<<static_cast<unsigned>((pre_threads + 255) / 256), 256, 0, stream>>>(
            o, dout, lse, nlse2, dvec, p.dq_acc, BH, p.Tq, p.Tq_pad);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (p.Tk > 0) {
        const size_t smem = sizeof(SmemBwd) + 1024;
        e = cudaFuncSetAttribute(attn_bwd_main, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        dim3 grid(static_cast<unsigned>(BH), static_cast<unsigned>((p.Tk + BKB - 1) / BKB));
        if ((e = launch_kernel(attn_bwd_main, grid, dim3(kBwdThreads), smem, stream, true, 1, tq, tk, tv, tg, p)) !=
            cudaSuccess)
            return e;
    }
    const long long post_threads = p.Tq > 0 ? BH * p.Tq_pad * 8 : 0;
    if (post_threads == 0) return cudaSuccess;
    return launch_kernel(attn_bwd_post, dim3(static_cast<unsigned>((post_threads + 255) / 256)), dim3(256), 0,
                         stream, true, 1, static_cast<const float *>(p.dq_acc), dq, BH, p.Tq, p.Tq_pad, p.scale);
}

}  // namespace mha
