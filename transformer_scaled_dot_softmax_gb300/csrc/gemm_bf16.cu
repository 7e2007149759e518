// gemm_bf16.cu -- bf16 projection GEMMs of multi-head attention for sm_103a.
//
// y = x W in the row-vector convention of the pages (Q = X W^Q, K = X W^K,
// V = X W^V: muhitai.com Step 1; notebook chapter "Multi-Head
// Self-Attention", W^Q in R^{d_model x d_k}; the output projection
// Concat(head_1..head_h) W^O: muhitai.com "Multi-Head Attention Formula").
//
// One launch runs up to three independent problems (the Q, K and V
// projections share a launch), cut into 128 x BN output tiles (BN = 128 or
// 256, chosen per launch by the host for the better balance).  The kernel
// is persistent: one CTA per SM takes tiles c, c + G, c + 2G, ... (all tiles
// of a launch have the same K, so round robin balances them), and the
// accumulator is double-buffered in tensor memory, so the epilogue of one
// tile overlaps the main loop of the next:
//
//   warp 0      TMA producer: A tile (128 rows x 64 k, K-major) and B tile
//               (64 k x BN n of W, N contiguous = MN-major) per k-block,
//               6-stage (BN = 128) or 4-stage (BN = 256) ring.
//   warp 1      MMA issuer: tcgen05.mma kind::f16, M=128 N=BN K=16, fp32
//               accumulators in two BN-column tensor-memory buffers; the
//               whole warp runs the loop and one elected lane issues.  With
//               BN = 256 the A tile is read from shared memory once per 256
//               output columns (96 instead of 128 bytes per cycle at the
//               tensor rate).
//   warps 2-5   epilogue: tensor memory -> registers (the buffer is handed
//               back as soon as it is read) -> [+ bias, ReLU] -> bf16 -> a
//               128-byte swizzled 128 x 128 staging block in shared memory,
//               which one thread stores with TMA (two 64-column boxes; rows
//               and columns past the output are clipped), 128 columns at a
//               time.  In head-split mode column n = head*64 + c of row
//               m = b*T + t goes to ((b*H + head)*T + t)*64 + c, i.e. straight
//               into the (B, H, T, 64) layout attention reads -- the
//               view/transpose of the head split costs no extra pass over
//               memory; the box is then (head, rows t0 .. t0+127 of batch b),
//               so T must be a multiple of 128, else each thread stores its
//               row directly.
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace mha {
namespace {

constexpr int BM = kGemmBM, BK = kGemmBK;
constexpr int kThreads = 192;
constexpr uint32_t kABytes = BM * BK * 2;  // 16 KiB
constexpr uint32_t kBBlock = BK * 64 * 2;  // 8 KiB: one 64-column block of a B tile
constexpr uint32_t kYBox = BM * 128;       // 16 KiB: 128 rows x 64 output columns

template <int BN>
struct GemmCfg {
    static constexpr int kStages = BN == 128 ? 6 : 4;
    static constexpr uint32_t kBBytes = BK * BN * 2;  // BN/64 column blocks
    static constexpr uint32_t kTmemCols = 2 * BN;     // two accumulators
};

template <int BN>
struct __align__(1024) SmemGemm {
    static constexpr int STAGES = GemmCfg<BN>::kStages;
    uint8_t a[STAGES][kABytes];
    uint8_t b[STAGES][GemmCfg<BN>::kBBytes];
    uint8_t ys[2][kYBox];  // output staging: 128 columns, 128-byte swizzled
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full[2];   // MMA -> epilogue (commit)
    uint64_t acc_empty[2];  // epilogue -> MMA (4 warps)
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

// Problem and tile coordinates of launch-wide tile `tile`.
struct Tile {
    int pi, tm, tn;
};
__device__ __forceinline__ Tile locate(const GemmParams &p, int tile) {
    Tile t;
    int pi = 0;
    while (pi + 1 < p.num_problems && tile >= p.prob[pi + 1].tile_start) ++pi;
    const int local = tile - p.prob[pi].tile_start;
    t.pi = pi;
    t.tm = local / p.prob[pi].tiles_n;
    t.tn = local - t.tm * p.prob[pi].tiles_n;
    return t;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap a0, const __grid_constant__ CUtensorMap a1,
                     const __grid_constant__ CUtensorMap a2, const __grid_constant__ CUtensorMap b0,
                     const __grid_constant__ CUtensorMap b1, const __grid_constant__ CUtensorMap b2,
                     const __grid_constant__ CUtensorMap y0, const __grid_constant__ CUtensorMap y1,
                     const __grid_constant__ CUtensorMap y2, const GemmParams p) {
    constexpr int STAGES = GemmCfg<BN>::kStages;
    constexpr uint32_t kBBytes = GemmCfg<BN>::kBBytes;
    constexpr uint32_t kTmemCols = GemmCfg<BN>::kTmemCols;
    extern __shared__ uint8_t smem_raw[];
    SmemGemm<BN> &sm = *reinterpret_cast<SmemGemm<BN> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = static_cast<int>(gridDim.x);
    const int num_k = (p.prob[0].K + BK - 1) / BK;  // the same K for every problem of a launch

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.acc_full[i], 1);
            mbar_init(&sm.acc_empty[i], 4);
        }
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&a0);
        prefetch_tensormap(&b0);
        if (p.prob[0].tma_store) prefetch_tensormap(&y0);
        if (p.num_problems > 1) {
            prefetch_tensormap(&a1);
            prefetch_tensormap(&b1);
            if (p.prob[1].tma_store) prefetch_tensormap(&y1);
        }
        if (p.num_problems > 2) {
            prefetch_tensormap(&a2);
            prefetch_tensormap(&b2);
            if (p.prob[2].tma_store) prefetch_tensormap(&y2);
        }
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
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int kg = 0;  // k-blocks issued over all tiles of this CTA
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += G) {
                const Tile t = locate(p, tile);
                const CUtensorMap *ta = t.pi == 0 ? &a0 : (t.pi == 1 ? &a1 : &a2);
                const CUtensorMap *tb = t.pi == 0 ? &b0 : (t.pi == 1 ? &b1 : &b2);
                for (int kb = 0; kb < num_k; ++kb, ++kg) {
                    const int st = kg % STAGES;
                    if (kg >= STAGES && !(ok = mbar_wait(&sm.empty[st], ((kg / STAGES) - 1) & 1, ab)))
                        break;
                    mbar_arrive_expect_tx(&sm.full[st], kABytes + kBBytes);
                    const GemmProblem &pr = p.prob[t.pi];
                    if (in_bounds(kb * BK < pr.K && t.tm * BM < pr.M && t.tn * BN < pr.N, p.status)) {
                        tma_load_2d(ta, &sm.full[st], sm.a[st], kb * BK, t.tm * BM);
                        tma_load_3d(tb, &sm.full[st], sm.b[st], 0, kb * BK, t.tn * (BN / 64));
                    }
                }
            }
            // Let every copy still in flight land before the CTA exits.
            for (int x = max(0, kg - STAGES); x < kg; ++x)
                mbar_wait_drain(&sm.full[x % STAGES], (x / STAGES) & 1);
        }
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer
        // Accumulator i % 2 for the CTA's i-th tile; it is reused once the
        // epilogue has read tile i-2 out of it.  Descriptors as base +
        // constant: a K step of 16 adds 32 bytes (2) to the K-major A row and
        // 16 rows of 128 bytes (2 KiB = 128) to each 64-column block of the
        // MN-major B tile; the blocks are 8 KiB apart (leading byte offset).
        constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, false, true);
        const uint64_t a_desc0 = smem_desc_sw128(smem_u32(sm.a[0]), 16, 1024);
        const uint64_t b_desc0 = smem_desc_sw128(smem_u32(sm.b[0]), kBBlock, 1024);
        constexpr uint64_t kADesc = kABytes >> 4, kBDesc = kBBytes >> 4;
        int kg = 0, i = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += G, ++i) {
            const int acc = i & 1;
            if (i >= 2 && !(ok = warp_wait(&sm.acc_empty[acc], ((i - 2) >> 1) & 1, ab))) break;
            tc_fence_after_sync();
            const uint32_t d = tmem + static_cast<uint32_t>(acc) * BN;
            for (int kb = 0; kb < num_k; ++kb, ++kg) {
                const int st = kg % STAGES;
                if (!(ok = warp_wait(&sm.full[st], (kg / STAGES) & 1, ab))) break;
                tc_fence_after_sync();
                const uint64_t ad = a_desc0 + static_cast<uint64_t>(st) * kADesc;
                const uint64_t bd = b_desc0 + static_cast<uint64_t>(st) * kBDesc;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    warp_mma_bf16_ss(d, ad + 2 * kk, bd + 128 * kk, idesc,
                                     (kb > 0 || kk > 0) ? 1u : 0u);
                warp_commit(&sm.empty[st]);
            }
            if (!ok) break;
            warp_commit(&sm.acc_full[acc]);
        }
        // Always wait (time-bounded, whatever the abort state) until every
        // MMA this warp issued has completed before tensor memory is
        // released.
        warp_commit(&sm.drain);
        mbar_wait_drain(&sm.drain, 0);
    } else {
        // --------------------------------------------------------- epilogue
        // Warp w reads tensor-memory lanes 32*(w%4) .. +31 (warps 2-5 cover
        // the four quadrants).
        const uint32_t lane_base = static_cast<uint32_t>(warp & 3) * 32;
        int i = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += G, ++i) {
            const Tile t = locate(p, tile);
            const GemmProblem &pr = p.prob[t.pi];
            const int acc = i & 1;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(&sm.acc_full[acc], (i >> 1) & 1, ab))))
                break;
            tc_fence_after_sync();
            const int m = t.tm * BM + static_cast<int>(lane_base) + lane;
            long long row_off = 0;
            if (pr.out_mode == kOutHeadSplit) {
                const int bb = m / pr.T, tt = m - bb * pr.T;
                row_off = static_cast<long long>(bb) * pr.H * pr.T + tt;  // + head*T below
            } else {
                row_off = static_cast<long long>(m) * pr.N;
            }
            const CUtensorMap *ty = t.pi == 0 ? &y0 : (t.pi == 1 ? &y1 : &y2);
            // 128 columns at a time; after the last group the accumulator is
            // handed back (the MMA warp may start the tile after next in it).
#pragma unroll 1
            for (int grp = 0; grp < BN / 128; ++grp) {
                uint32_t r[4][32];
                const uint32_t src =
                    tmem_addr(tmem, lane_base, static_cast<uint32_t>(acc) * BN + 128u * grp);
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(src + 32u * c, r[c]);
                tmem_ld_wait(r[0]);
                reg_fence32(r[1]);
                reg_fence32(r[2]);
                reg_fence32(r[3]);
                if (grp == BN / 128 - 1) {
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.acc_empty[acc]);
                }
                if (pr.tma_store) {
                    // the previous group's store has read the staging block
                    if (warp == 2 && lane == 0) bulk_wait_read();
                    asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
                }
                const int rr = static_cast<int>(lane_base) + lane;  // row in the tile
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int n0 = t.tn * BN + grp * 128 + c * 32;
                    uint32_t packed[16];
                    if (pr.bias && n0 < pr.N) {
                        // bias (+ ReLU): the feed-forward network's first layer
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint4 bw = *reinterpret_cast<const uint4 *>(pr.bias + n0 + 8 * q);
                            const uint32_t bb[4] = {bw.x, bw.y, bw.z, bw.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                float v0 = __uint_as_float(r[c][8 * q + 2 * e]) + __uint_as_float(bb[e] << 16);
                                float v1 = __uint_as_float(r[c][8 * q + 2 * e + 1]) +
                                           __uint_as_float(bb[e] & 0xffff0000u);
                                if (pr.relu) {
                                    v0 = fmaxf(v0, 0.f);
                                    v1 = fmaxf(v1, 0.f);
                                }
                                packed[4 * q + e] = pack_bf16x2(v0, v1);
                            }
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 16; ++q)
                            packed[q] = pack_bf16x2(__uint_as_float(r[c][2 * q]), __uint_as_float(r[c][2 * q + 1]));
                    }
                    if (pr.tma_store) {
                        // 16-byte chunk j = 4c + q of the row: box j / 8, position
                        // (j % 8) ^ (row % 8)
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int j = 4 * c + q;
                            *reinterpret_cast<uint4 *>(sm.ys[j >> 3] + rr * 128 + (((j & 7) ^ (rr & 7)) << 4)) =
                                make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                        }
                    } else if (m < pr.M && n0 < pr.N &&
                               in_bounds(pr.out_mode != kOutHeadSplit || (n0 >> 6) < pr.H, p.status)) {
                        __nv_bfloat16 *dst;
                        if (pr.out_mode == kOutHeadSplit) {
                            const int head = n0 >> 6, c0 = n0 & 63;
                            dst = pr.out + (row_off + static_cast<long long>(head) * pr.T) * 64 + c0;
                        } else {
                            dst = pr.out + row_off + n0;
                        }
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            d4[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                               packed[4 * q + 3]);
                    }
                }
                if (pr.tma_store) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    if (warp == 2 && lane == 0) {
#pragma unroll
                        for (int bx = 0; bx < 2; ++bx) {
                            const int nb = t.tn * BN + grp * 128 + 64 * bx;
                            if (nb >= pr.N) break;
                            if (!in_bounds(t.tm * BM < pr.M && (pr.out_mode != kOutHeadSplit ||
                                                                (nb >> 6) < pr.H), p.status))
                                break;
                            if (pr.out_mode == kOutHeadSplit) {
                                const int m0 = t.tm * BM, bb = m0 / pr.T;
                                tma_store_3d(ty, sm.ys[bx], 0, m0 - bb * pr.T, bb * pr.H + (nb >> 6));
                            } else {
                                tma_store_2d(ty, sm.ys[bx], nb, t.tm * BM);
                            }
                        }
                        bulk_commit_group();
                    }
                }
            }
        }
        if (warp == 2 && lane == 0) bulk_wait_all();  // the last stores have landed
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap (&a)[kGemmMaxProblems],
                      const CUtensorMap (&b)[kGemmMaxProblems],
                      const CUtensorMap (&y)[kGemmMaxProblems], const GemmParams &p, int sms,
                      cudaStream_t stream, bool pdl) {
    const size_t smem = sizeof(SmemGemm<BN>) + 1024;
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel<BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // One persistent CTA per SM (fewer if there are fewer tiles).
    const int grid = p.total_tiles < sms ? p.total_tiles : sms;
    if (grid <= 0) return cudaSuccess;
    return launch_kernel(gemm_bf16_kernel<BN>, dim3(grid), dim3(kThreads), smem, stream, pdl, 1, a[0], a[1],
                         a[2], b[0], b[1], b[2], y[0], y[1], y[2], p);
}

}  // namespace

cudaError_t sm_count(int *sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
}

cudaError_t launch_gemm_bf16(const CUtensorMap (&a)[kGemmMaxProblems],
                             const CUtensorMap (&b)[kGemmMaxProblems],
                             const CUtensorMap (&y)[kGemmMaxProblems], const GemmParams &p,
                             cudaStream_t stream, bool pdl) {
    int sms = 0;
    cudaError_t e = sm_count(&sms);
    if (e != cudaSuccess) return e;
    if (p.bn == 256) return launch_bn<256>(a, b, y, p, sms, stream, pdl);
    if (p.bn == 128) return launch_bn<128>(a, b, y, p, sms, stream, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace mha
