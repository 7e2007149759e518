// gemm_bf16.cu -- bf16 projection GEMMs of multi-head attention for sm_103a.
//
// y = x W in the row-vector convention of the pages (Q = X W^Q, K = X W^K,
// V = X W^V: muhitai.com Step 1; notebook chapter "Multi-Head
// Self-Attention", W^Q in R^{d_model x d_k}; the output projection
// Concat(head_1..head_h) W^O: muhitai.com "Multi-Head Attention Formula").
//
// One launch runs up to three independent problems (the Q, K and V
// projections share a launch); a CTA owns one 128 x 128 output tile:
//
//   warp 0      TMA producer: A tile (128 rows x 64 k, K-major) and B tile
//               (64 k x 128 n of W, N contiguous = MN-major) per k-block,
//               4-stage ring.
//   warp 1      MMA issuer: tcgen05.mma kind::f16, M=128 N=128 K=16,
//               fp32 accumulator in 128 tensor-memory columns.
//   warps 2-5   epilogue: tensor memory -> registers -> bf16 -> global.  In
//               head-split mode column n = head*64 + c of row m = b*T + t is
//               stored at ((b*H + head)*T + t)*64 + c, i.e. straight into the
//               (B, H, T, 64) layout attention reads -- the view/transpose of
//               the head split costs no extra pass over memory.
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace mha {
namespace {

constexpr int BM = kGemmBM, BN = kGemmBN, BK = kGemmBK;
constexpr int STAGES = 4;
constexpr int kThreads = 192;
constexpr uint32_t kABytes = BM * BK * 2;  // 16 KiB
constexpr uint32_t kBBytes = BK * BN * 2;  // 16 KiB: two 64-column blocks of 8 KiB
constexpr uint32_t kTmemCols = 128;

struct __align__(1024) SmemGemm {
    uint8_t a[STAGES][kABytes];
    uint8_t b[STAGES][kBBytes];
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full;
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap a0, const __grid_constant__ CUtensorMap a1,
                     const __grid_constant__ CUtensorMap a2, const __grid_constant__ CUtensorMap b0,
                     const __grid_constant__ CUtensorMap b1, const __grid_constant__ CUtensorMap b2,
                     const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    SmemGemm &sm = *reinterpret_cast<SmemGemm *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Which problem and tile.
    const int tile = blockIdx.x;
    int pi = 0;
    while (pi + 1 < p.num_problems && tile >= p.prob[pi + 1].tile_start) ++pi;
    const GemmProblem &pr = p.prob[pi];
    const int local = tile - pr.tile_start;
    const int tm = local / pr.tiles_n;
    const int tn = local - tm * pr.tiles_n;
    const int num_k = (pr.K + BK - 1) / BK;
    const CUtensorMap *ta = pi == 0 ? &a0 : (pi == 1 ? &a1 : &a2);
    const CUtensorMap *tb = pi == 0 ? &b0 : (pi == 1 ? &b1 : &b2);

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
        }
        mbar_init(&sm.acc_full, 1);
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(ta);
        prefetch_tensormap(tb);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    const AbortState ab{&sm.abort_flag, p.status};

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int kb = 0; kb < num_k; ++kb) {
                const int st = kb % STAGES;
                if (kb >= STAGES && !mbar_wait(&sm.empty[st], ((kb / STAGES) - 1) & 1, ab)) break;
                mbar_arrive_expect_tx(&sm.full[st], kABytes + kBBytes);
                tma_load_2d(ta, &sm.full[st], sm.a[st], kb * BK, tm * BM);
                tma_load_3d(tb, &sm.full[st], sm.b[st], 0, kb * BK, tn * (BN / 64));
                issued = kb + 1;
            }
            // Let every copy still in flight land before the CTA exits.
            for (int kb = max(0, issued - STAGES); kb < issued; ++kb)
                mbar_wait_drain(&sm.full[kb % STAGES], (kb / STAGES) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, false, true);
            bool ok = true;
            for (int kb = 0; kb < num_k; ++kb) {
                const int st = kb % STAGES;
                if (!(ok = mbar_wait(&sm.full[st], (kb / STAGES) & 1, ab))) break;
                tc_fence_after_sync();
                const uint32_t aa = smem_u32(sm.a[st]);
                const uint32_t ba = smem_u32(sm.b[st]);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_bf16_ss(tmem, smem_desc_sw128(aa + kk * 32, 16, 1024),
                                smem_desc_sw128(ba + kk * 2048, kBBytes / 2, 1024), idesc,
                                (kb > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&sm.empty[st]);
            }
            if (ok) mma_commit(&sm.acc_full);
            // Always wait (time-bounded, whatever the abort state) until every
            // MMA this thread issued has completed before tensor memory is
            // released.
            mma_commit(&sm.drain);
            mbar_wait_drain(&sm.drain, 0);
        }
    } else {
        // Epilogue: warp w reads tensor-memory lanes 32*(w%4) .. +31.
        const uint32_t lane_base = static_cast<uint32_t>(warp & 3) * 32;
        const int m = tm * BM + static_cast<int>(lane_base) + lane;
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&sm.acc_full, 0, ab));
        if (ok) {
            tc_fence_after_sync();
            long long row_off = 0;
            if (m < pr.M) {
                if (pr.out_mode == kOutHeadSplit) {
                    const int bb = m / pr.T, t = m - bb * pr.T;
                    row_off = static_cast<long long>(bb) * pr.H * pr.T + t;  // + head*T later
                } else {
                    row_off = static_cast<long long>(m) * pr.N;
                }
            }
#pragma unroll 1
            for (int chunk = 0; chunk < BN / 32; ++chunk) {
                uint32_t r[32];
                tmem_ld32(tmem_addr(tmem, lane_base, chunk * 32), r);
                tmem_ld_wait(r);
                const int n0 = tn * BN + chunk * 32;
                if (m < pr.M && n0 < pr.N) {
                    uint32_t packed[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        packed[c] = pack_bf16x2(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1]));
                    __nv_bfloat16 *dst;
                    if (pr.out_mode == kOutHeadSplit) {
                        const int head = n0 >> 6, c0 = n0 & 63;
                        dst = pr.out + (row_off + static_cast<long long>(head) * pr.T) * 64 + c0;
                    } else {
                        dst = pr.out + row_off + n0;
                    }
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        d4[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2],
                                           packed[4 * c + 3]);
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_gemm_bf16(const CUtensorMap (&a)[kGemmMaxProblems],
                             const CUtensorMap (&b)[kGemmMaxProblems], const GemmParams &p,
                             cudaStream_t stream) {
    const size_t smem = sizeof(SmemGemm) + 1024;
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    gemm_bf16_kernel<<<p.total_tiles, kThreads, smem, stream>>>(a[0], a[1], a[2], b[0], b[1], b[2],
                                                                  p);
    return cudaGetLastError();
}

}  // namespace mha
