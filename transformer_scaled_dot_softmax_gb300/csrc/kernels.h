// kernels.h -- launch interfaces between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mha.h"

namespace mha {

constexpr int kMaskCausalBit = 1;
constexpr int kMaskPaddingBit = 2;

// ------------------------------------------------ launch helper
// Launches `kernel` on `stream`.  With pdl the launch may begin while the
// kernel before it on the stream finishes (programmatic dependent launch);
// every kernel launched that way waits for its predecessor (pdl_wait) after
// its prologue and before it touches global memory.  Optional cluster size.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, bool pdl, unsigned cluster, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ------------------------------------------------ fused bf16 attention
struct AttnParams {
    int B, H, Tq, Tk;
    float scale_log2;  // scale * log2(e): scores are exponentiated with ex2
    float scale;
    float *lse;        // optional (B, H, Tq) fp32: log sum_j exp(scale q.k_j); null: not written
    int mask;          // kMaskCausalBit | kMaskPaddingBit
    const int32_t *key_lens;
    __nv_bfloat16 *o;  // output; element (b, h, t, c) at o + b*sb + h*sh + t*st + c
    long long o_stride_b, o_stride_h, o_stride_t;
    int num_qblocks;   // ceil(Tq / rows per item)
    int total_items;   // B * H * num_qblocks work items (query tiles)
    int *status;
    // Failure-detection drill only (both 0 on every product path): the wait
    // limit in ns (0: the default 1 s), and n > 0 makes every CTA's loader
    // issue no copy for its (n-1)-th key tile, so the waits on it run out.
    unsigned long long wait_limit_ns;
    int drill_skip_tile;
};
constexpr int kAttnRowsPerCta = 128;  // one work item = one 128-row query tile
constexpr int kAttnHeadDim = 64;

// The kernel's two softmax groups split a row's keys either into the two
// 64-key halves of every tile or into alternate tiles; alternate tiles keep
// the groups out of lockstep and pay once a query tile has, on average,
// kAttnTilesSplitMin key tiles or more (measured on GB300: +3 % at causal
// T = 8192), while short items finish sooner by halves.
constexpr int kAttnTilesSplitMin = 8;
bool attn_bf16_splits_by_tiles(int Tq, int Tk, int mask);

// q, k, v: head-split (B, H, T, 64) bf16 tensors described by 3-D TMA maps
// over (64, T, B*H) with 128-byte swizzling and 128-row boxes.
cudaError_t launch_attn_bf16(const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, const AttnParams &p, cudaStream_t stream,
                             bool pdl = false);

// ------------------------------------------------ bf16 decode attention
constexpr int kDecodeMaxRows = 8;  // query rows per (b, h) in one decode call
struct DecodeParams {
    int B, H, Tq, Tk;
    float scale_log2;          // scale * log2(e)
    const int32_t *key_lens;   // cached keys per batch entry; null: all Tk
};
// q (B, H, Tq, 64), k and v (B, H, Tk, 64), o (B, H, Tq, 64), all bf16 and
// contiguous; Tq <= kDecodeMaxRows.
cudaError_t launch_decode_bf16(const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                               const __nv_bfloat16 *v, __nv_bfloat16 *o, const DecodeParams &p,
                               cudaStream_t stream);

// ------------------------------------------------ bf16 attention backward
struct BwdParams {
    int B, H, Tq, Tk, Tq_pad;   // Tq_pad: Tq rounded up to whole 128-row blocks
    float scale, scale_log2;
    int mask;
    const int32_t *key_lens;
    const float *nlse2;         // (B, H, Tq_pad) -lse * log2(e), -inf for padded / empty rows
    const float *dvec;          // (B, H, Tq_pad) rowsum(dO * O)
    float *dq_acc;              // (B, H, Tq_pad, 64) fp32
    __nv_bfloat16 *dk, *dv;     // (B, H, Tk, 64)
    int *status;
};
// Bytes of workspace the backward needs (fp32 dQ accumulator, lse, D).
size_t bwd_workspace_bytes(long long BH, int Tq);
// q, k, v, dout: 3-D TMA maps like the forward's; o, dout, lse as device
// arrays; fills dq (bf16), p.dk, p.dv.  `workspace`: bwd_workspace_bytes(),
// 256-byte aligned.
cudaError_t launch_attn_bwd_bf16(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                 const CUtensorMap &tg, const __nv_bfloat16 *o,
                                 const __nv_bfloat16 *dout, const float *lse, __nv_bfloat16 *dq,
                                 BwdParams p, void *workspace, cudaStream_t stream);

// ------------------------------------------------ positional encoding
// out (rows, D) = x + PE(pos0 + row % T); D % 8 == 0; x and out may alias.
cudaError_t launch_posenc_add_bf16(const __nv_bfloat16 *x, __nv_bfloat16 *out, long long rows, int T,
                                   int D, int pos0, cudaStream_t stream);

// ------------------------------------------------ fp32 SIMT attention
constexpr int kF32RowsPerCta = 8;  // query rows per CTA (one warp each)
cudaError_t launch_sdpa_f32(const float *q, const float *k, const float *v, float *o, int B,
                            int H, int Tq, int Tk, int dk, int dv, float scale, int mask,
                            const int32_t *key_lens, cudaStream_t stream);

// ------------------------------------------------ bf16 projection GEMM
constexpr int kGemmMaxProblems = 3;
enum GemmOutMode { kOutRowMajor = 0, kOutHeadSplit = 1 };
struct GemmProblem {
    int M, N, K;
    int tiles_n, tile_start, tile_count;
    __nv_bfloat16 *out;
    int out_mode;  // kOutRowMajor: out (M, N); kOutHeadSplit: row m = b*T + t,
                   // column n = head*64 + c -> out ((b*H + head)*T + t)*64 + c
    int T, H;
    const __nv_bfloat16 *bias;  // optional (N): added to every row
    int relu;                   // nonzero: max(0, .) after the bias
    int tma_store;              // nonzero: the output goes out through its TMA map (y below)
};
struct GemmParams {
    int num_problems;
    int total_tiles;
    int bn;  // output tile width: 128 or 256
    GemmProblem prob[kGemmMaxProblems];
    int *status;
};
constexpr int kGemmBM = 128, kGemmBK = 64;

// a[i]: 2-D TMA map over the activation (K inner, M rows), box (64, 128).
// b[i]: 3-D TMA map over the weight viewed as (64, K, N/64), box (64, 64, bn/64).
// y[i] (problems with tma_store): the output, 2-D (N inner, M rows) box (64, 128)
// for row-major, 3-D (64, T, B*H) box (64, 128, 1) for head-split with T a
// multiple of 128.
cudaError_t launch_gemm_bf16(const CUtensorMap (&a)[kGemmMaxProblems],
                             const CUtensorMap (&b)[kGemmMaxProblems],
                             const CUtensorMap (&y)[kGemmMaxProblems], const GemmParams &p,
                             cudaStream_t stream, bool pdl = false);

// Number of SMs of the current device.
cudaError_t sm_count(int *sms);

// Records "what: detail" as the calling thread's mha_last_error() text and
// returns MHA_ERR_CUDA.
mha_status record_cuda_failure(const char *what, const char *detail);

// ------------------------------------ output projection + residual + LayerNorm
constexpr int kLnMaxCluster = 8;  // CTAs per 128-row block (portable cluster size)
struct LnParams {
    int M, D, K;                  // out (M, D) = LN(resid + A (M, K) W (K, D) [+ bias])
    int bn;                       // columns per CTA: ln_tile_width(D)
    const __nv_bfloat16 *resid;   // (M, D)
    const __nv_bfloat16 *bias;    // optional (D): added to the product before the residual
    const __nv_bfloat16 *gamma;   // (D)
    const __nv_bfloat16 *beta;    // (D)
    float eps;
    __nv_bfloat16 *out;           // (M, D)
    int *status;
};
// 256 or 128 columns per CTA for rows of D features (D / width CTAs <= 8) over
// M rows on `sms` SMs, or 0 if D is not supported.
int ln_tile_width(int D, long long M, int sms);
// a: 2-D TMA map over A (K inner, M rows), box (64, 128); b: 3-D map over W
// viewed as (64, K, D/64), box (64, 64, bn/64); x, y: 2-D maps over the
// residual and the output (D inner, M rows), box (64, 128).
cudaError_t launch_gemm_ln_bf16(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &x,
                                const CUtensorMap &y, const LnParams &p, cudaStream_t stream,
                                bool pdl = false);

}  // namespace mha
