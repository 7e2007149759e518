// gemm_ln_bf16.cu -- output projection fused with the residual connection and
// layer normalisation that wrap the attention sublayer, for sm_103a:
//
//   out = LayerNorm(x + Concat(heads) W^O),  or, for the feed-forward
//   sublayer, LayerNorm(x + H W_2 + b_2) (the same kernel with a bias),
//   LayerNorm(v) = (v - mu) / sqrt(var + eps) * gamma + beta per row,
//
// ("Attention Is All You Need" (aiany.app) Step 9, LayerNorm(x + Sublayer(x));
// notebook chapter "Layer Normalization and Residual Connections": mu and the
// standard deviation over the feature dimension, learned gamma and beta; eps
// is the caller's, the variance the population one).
//
// A row's statistics need all D output features, more than one tensor-memory
// accumulator holds, so a 128-row block is computed by a cluster of D / BN
// CTAs (BN = 256, or 128 when D is not a multiple of 256), CTA r owning output
// columns [r*BN, (r+1)*BN).  Per CTA:
//
//   warp 0      TMA producer: first this CTA's 128 x BN block of the residual
//               x (128-byte swizzled, for the epilogue, landing while the
//               products run), then A = 128 rows x 64 k of the merged heads,
//               B = 64 k x BN columns of W^O, 3-stage (BN = 256) / 5-stage ring.
//   warp 1      MMA issuer (tcgen05.mma kind::f16, M=128 N=BN, fp32
//               accumulator in BN tensor-memory columns, elected lane).
//   warps 2-5   epilogue, one thread per row, three passes over the
//               accumulator (x read from shared memory: 16-byte chunk j of row
//               r at j ^ (r % 8), no bank conflicts): (1) v = acc + x, row sum;
//               (2) sum of (v - mu)^2;
//               (3) normalise, scale, shift, bf16 over the residual block in
//               shared memory, which one thread then stores with TMA (a
//               thread's own row is 32 scattered 16-byte stores otherwise).
//               After (1) and (2) the CTAs of the cluster exchange their
//               per-row partial sums through distributed shared memory, so
//               mean and variance are exact two-pass statistics over the whole
//               row.
//
// Every thread of every CTA passes the same three cluster barriers, whatever
// its role and whether a bounded wait ran out, so no CTA can be left waiting.
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace mha {
namespace {

constexpr int BM = kGemmBM, BK = kGemmBK;
constexpr int kThreads = 192;
constexpr uint32_t kABytes = BM * BK * 2;  // 16 KiB
constexpr uint32_t kBBlock = BK * 64 * 2;  // 8 KiB: one 64-column block of a B tile

template <int BN>
struct LnCfg {
    static constexpr int kStages = BN == 128 ? 5 : 3;
    static constexpr uint32_t kBBytes = BK * BN * 2;
};
constexpr uint32_t kXBox = BM * 128;  // 16 KiB: 128 rows x 64 features of the residual

template <int BN>
struct __align__(1024) SmemLn {
    static constexpr int STAGES = LnCfg<BN>::kStages;
    uint8_t a[STAGES][kABytes];
    uint8_t b[STAGES][LnCfg<BN>::kBBytes];
    uint8_t xs[BN / 64][kXBox];  // residual block, 64 features per box
    __nv_bfloat16 gamma[BN];     // this CTA's columns of gamma, beta and the bias
    __nv_bfloat16 beta[BN];
    __nv_bfloat16 bias[BN];
    float part[2][BM];  // this CTA's per-row partial: [0] sum of v, [1] sum of (v - mu)^2
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full;
    uint64_t x_full;
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

// Reconverges the warp first: the cluster barrier is an aligned instruction.
__device__ __forceinline__ void cluster_sync_all() {
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ float dsmem_ld_f32(const void *p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ void bf16x8(const uint4 &u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Eight residual features [8j', 8j'+8) of row r, j' = column / 8 within the
// block: box j'/8, chunk j' % 8 swizzled with the row.
template <int BN>
__device__ __forceinline__ uint4 *x_chunk(SmemLn<BN> &sm, int r, int j) {
    return reinterpret_cast<uint4 *>(sm.xs[j >> 3] + r * 128 + (((j & 7) ^ (r & 7)) << 4));
}

// x[0..7] += bias[n .. n+7] (bf16, this CTA's columns in shared memory), if
// there is a bias: the residual and the sublayer's output bias enter the row
// together.
__device__ __forceinline__ void add_bias(float (&x)[8], bool has_bias, const __nv_bfloat16 *bias, int n) {
    if (!has_bias) return;
    float b[8];
    bf16x8(*reinterpret_cast<const uint4 *>(bias + n), b);
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] += b[e];
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_ln_bf16_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                        const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap ty,
                        const LnParams p) {
    constexpr int STAGES = LnCfg<BN>::kStages;
    constexpr uint32_t kBBytes = LnCfg<BN>::kBBytes;
    extern __shared__ uint8_t smem_raw[];
    SmemLn<BN> &sm = *reinterpret_cast<SmemLn<BN> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int csize = p.D / BN;  // CTAs per cluster
    const uint32_t rank = cluster_rank();
    const int tm = static_cast<int>(blockIdx.x) / csize;
    const int n_base = static_cast<int>(rank) * BN;
    const int num_k = (p.K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
        }
        mbar_init(&sm.acc_full, 1);
        mbar_init(&sm.x_full, 1);
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, BN);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&ta);
        prefetch_tensormap(&tb);
        prefetch_tensormap(&tx);
        prefetch_tensormap(&ty);
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

    // Epilogue state (warps 2-5): row of this thread and its statistics.
    const uint32_t lane_base = static_cast<uint32_t>(warp & 3) * 32;
    const int r = static_cast<int>(lane_base) + lane;
    const int m = tm * BM + r;
    const bool row_ok = m < p.M;
    const bool epi = warp >= 2;
    const bool has_bias = p.bias != nullptr;
    bool ok = true;
    float mu = 0.f;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            mbar_arrive_expect_tx(&sm.x_full, (BN / 64) * kXBox);
            const bool tile_ok = in_bounds(tm * BM < p.M && n_base + BN <= p.D, p.status);
#pragma unroll
            for (int bx = 0; bx < BN / 64; ++bx)
                if (tile_ok) tma_load_2d(&tx, &sm.x_full, sm.xs[bx], n_base + 64 * bx, tm * BM);
            int issued = 0;
            for (int kb = 0; kb < num_k; ++kb) {
                const int st = kb % STAGES;
                if (kb >= STAGES && !mbar_wait(&sm.empty[st], ((kb / STAGES) - 1) & 1, ab)) break;
                mbar_arrive_expect_tx(&sm.full[st], kABytes + kBBytes);
                if (tile_ok && in_bounds(kb * BK < p.K, p.status)) {
                    tma_load_2d(&ta, &sm.full[st], sm.a[st], kb * BK, tm * BM);
                    tma_load_3d(&tb, &sm.full[st], sm.b[st], 0, kb * BK, n_base / 64);
                }
                issued = kb + 1;
            }
            for (int x = max(0, issued - STAGES); x < issued; ++x)
                mbar_wait_drain(&sm.full[x % STAGES], (x / STAGES) & 1);
            mbar_wait_drain(&sm.x_full, 0);
        }
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer
        constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, false, true);
        const uint64_t a_desc0 = smem_desc_sw128(smem_u32(sm.a[0]), 16, 1024);
        const uint64_t b_desc0 = smem_desc_sw128(smem_u32(sm.b[0]), kBBlock, 1024);
        constexpr uint64_t kADesc = kABytes >> 4, kBDesc = kBBytes >> 4;
        bool mok = true;
        for (int kb = 0; kb < num_k; ++kb) {
            const int st = kb % STAGES;
            if (!(mok = warp_wait(&sm.full[st], (kb / STAGES) & 1, ab))) break;
            tc_fence_after_sync();
            const uint64_t ad = a_desc0 + static_cast<uint64_t>(st) * kADesc;
            const uint64_t bd = b_desc0 + static_cast<uint64_t>(st) * kBDesc;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
                warp_mma_bf16_ss(tmem, ad + 2 * kk, bd + 128 * kk, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
            warp_commit(&sm.empty[st]);
        }
        if (mok) warp_commit(&sm.acc_full);
        warp_commit(&sm.drain);
        mbar_wait_drain(&sm.drain, 0);
    } else {
        // The CTA's columns of gamma, beta (and the bias) into shared memory
        // while the products run (every (c, q) step of the passes below reads
        // a new 16-byte piece of each).
        for (int i = threadIdx.x - 64; i < BN / 8; i += 128) {
            reinterpret_cast<uint4 *>(sm.gamma)[i] = reinterpret_cast<const uint4 *>(p.gamma + n_base)[i];
            reinterpret_cast<uint4 *>(sm.beta)[i] = reinterpret_cast<const uint4 *>(p.beta + n_base)[i];
            if (has_bias) reinterpret_cast<uint4 *>(sm.bias)[i] = reinterpret_cast<const uint4 *>(p.bias + n_base)[i];
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
        // ----------------------------------------- epilogue pass 1: row sums
        ok = __all_sync(0xffffffffu, mbar_wait(&sm.acc_full, 0, ab)) &&
             __all_sync(0xffffffffu, mbar_wait(&sm.x_full, 0, ab));
        float s1 = 0.f;
        if (ok) {
            tc_fence_after_sync();
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t acc[32];
                __syncwarp();
                tmem_ld32(tmem_addr(tmem, lane_base, 32u * c), acc);
                tmem_ld_wait(acc);
                if (row_ok) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float xf[8];
                        bf16x8(*x_chunk(sm, r, 4 * c + q), xf);
                        add_bias(xf, has_bias, sm.bias, 32 * c + 8 * q);
#pragma unroll
                        for (int e = 0; e < 8; ++e) s1 += __uint_as_float(acc[8 * q + e]) + xf[e];
                    }
                }
            }
        }
        sm.part[0][r] = s1;
    }

    cluster_sync_all();  // every CTA's row sums are in place

    float s2 = 0.f;
    if (epi) {
        // -------------------------------- epilogue pass 2: squared deviations
        float tot = 0.f;
        for (int q = 0; q < csize; ++q) tot += dsmem_ld_f32(&sm.part[0][r], static_cast<uint32_t>(q));
        mu = tot / static_cast<float>(p.D);
        // `ok` is warp-uniform; every lane issues the tensor-memory loads
        // (rows past M included) and only the arithmetic depends on the row.
        if (ok) {
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t acc[32];
                __syncwarp();
                tmem_ld32(tmem_addr(tmem, lane_base, 32u * c), acc);
                tmem_ld_wait(acc);
                if (row_ok) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float xf[8];
                        bf16x8(*x_chunk(sm, r, 4 * c + q), xf);
                        add_bias(xf, has_bias, sm.bias, 32 * c + 8 * q);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float d = __uint_as_float(acc[8 * q + e]) + xf[e] - mu;
                            s2 = fmaf(d, d, s2);
                        }
                    }
                }
            }
        }
        sm.part[1][r] = s2;
    }

    cluster_sync_all();  // every CTA's squared deviations are in place

    if (epi) {
        // ---------------------------- epilogue pass 3: normalise and store
        float tot = 0.f;
        for (int q = 0; q < csize; ++q) tot += dsmem_ld_f32(&sm.part[1][r], static_cast<uint32_t>(q));
        const float rstd = rsqrtf(tot / static_cast<float>(p.D) + p.eps);
        if (ok) {
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t acc[32];
                __syncwarp();
                tmem_ld32(tmem_addr(tmem, lane_base, 32u * c), acc);
                tmem_ld_wait(acc);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 *xy = x_chunk(sm, r, 4 * c + q);  // x in, y out (same row, same chunk)
                    float xf[8], gf[8], bf[8];
                    bf16x8(*xy, xf);
                    add_bias(xf, has_bias, sm.bias, 32 * c + 8 * q);
                    bf16x8(*reinterpret_cast<const uint4 *>(sm.gamma + 32 * c + 8 * q), gf);
                    bf16x8(*reinterpret_cast<const uint4 *>(sm.beta + 32 * c + 8 * q), bf);
                    uint32_t packed[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float y0 = (__uint_as_float(acc[8 * q + 2 * e]) + xf[2 * e] - mu) *
                                             rstd * gf[2 * e] + bf[2 * e];
                        const float y1 = (__uint_as_float(acc[8 * q + 2 * e + 1]) + xf[2 * e + 1] -
                                          mu) * rstd * gf[2 * e + 1] + bf[2 * e + 1];
                        packed[e] = pack_bf16x2(y0, y1);
                    }
                    *xy = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                }
            }
        }
        // The block in shared memory is complete: one thread stores it (rows
        // past M are clipped by the tensor map), unless a wait ran out.
        fence_proxy_async_smem();
        __syncwarp();
        asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
        if (warp == 2 && lane == 0) {
            if (!*ab.cta_flag) {
#pragma unroll
                for (int bx = 0; bx < BN / 64; ++bx)
                    if (in_bounds(tm * BM < p.M && n_base + 64 * bx < p.D, p.status))
                        tma_store_2d(&ty, sm.xs[bx], n_base + 64 * bx, tm * BM);
                bulk_commit_group();
            }
            bulk_wait_all();
        }
    }

    // No CTA leaves while another may still read its row statistics, and
    // tensor memory is freed only after every read of the accumulator.
    tc_fence_before_sync();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, BN);
    }
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &x,
                      const CUtensorMap &y, const LnParams &p, cudaStream_t stream, bool pdl) {
    const size_t smem = sizeof(SmemLn<BN>) + 1024;
    cudaError_t e = cudaFuncSetAttribute(gemm_ln_bf16_kernel<BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int csize = p.D / BN;
    const int row_tiles = (p.M + BM - 1) / BM;
    return launch_kernel(gemm_ln_bf16_kernel<BN>, dim3(static_cast<unsigned>(row_tiles * csize)), dim3(kThreads),
                         smem, stream, pdl, static_cast<unsigned>(csize), a, b, x, y, p);
}

}  // namespace

int ln_tile_width(int D, long long M, int sms) {
    const bool w256 = D % 256 == 0 && D / 256 <= kLnMaxCluster;
    const bool w128 = D % 128 == 0 && D / 128 <= kLnMaxCluster;
    // 256 columns per CTA read each A tile once per 256 outputs; 128 columns
    // double the CTAs.  Measured on GB300 (self / causal / cross MHA
    // workloads), the narrower tiles pay only while 256-wide blocks would fill
    // less than half of the SMs and the cluster stays at 4 CTAs or fewer.
    const long long blocks256 = (M + BM - 1) / BM * (D / 256);
    if (w128 && (!w256 || (2 * blocks256 < sms && D / 128 <= 4))) return 128;
    if (w256) return 256;
    return 0;
}

cudaError_t launch_gemm_ln_bf16(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &x,
                                const CUtensorMap &y, const LnParams &p, cudaStream_t stream, bool pdl) {
    if (p.M <= 0) return cudaSuccess;
    if (p.bn == 256) return launch_bn<256>(a, b, x, y, p, stream, pdl);
    if (p.bn == 128) return launch_bn<128>(a, b, x, y, p, stream, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace mha
