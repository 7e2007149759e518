// api.cu -- the C ABI declared in include/mha.h: argument checks, TMA
// tensor-map encoding and kernel launches on the caller's stream.  Nothing
// here allocates device memory, frees or synchronises; sdpa_forward_host
// keeps two copy streams and a few events per device for its pipeline.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <stdio.h>

#include <algorithm>
#include <mutex>

#include "../../include/mha.h"
#include "kernels.h"

#define MHA_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime so the
// library does not link libcuda directly.
EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

thread_local char g_last_error[256] = "";

mha_status cuda_fail(const char *what, const char *detail) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", what, detail);
    return MHA_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// bf16 tensor map with 128-byte swizzling.  dims/strides are innermost first;
// strides are in bytes for dims 1..rank-1.
mha_status encode_bf16(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
                       const uint64_t *strides_bytes, const uint32_t *box) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cuda_fail("cuTensorMapEncodeTiled", "driver entry point not found");
    cuuint64_t d[5], s[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) s[i] = strides_bytes[i];
    }
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                    const_cast<void *>(base), d, s, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[96];
        snprintf(buf, sizeof(buf), "CUresult %d (rank %d, dims %llu x %llu x %llu)", (int)r, rank,
                 (unsigned long long)d[0], (unsigned long long)(rank > 1 ? d[1] : 0),
                 (unsigned long long)(rank > 2 ? d[2] : 0));
        return cuda_fail("cuTensorMapEncodeTiled", buf);
    }
    return MHA_OK;
}

// (B*H, T, 64) head-split bf16 tensor, 128-row boxes.
mha_status encode_heads(CUtensorMap *m, const void *base, long long BH, int T) {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(T), static_cast<uint64_t>(BH)};
    const uint64_t strides[2] = {128, static_cast<uint64_t>(T) * 128};
    const uint32_t box[3] = {64, 128, 1};
    return encode_bf16(m, base, 3, dims, strides, box);
}

// Activation (M rows x K) row-major: box 64 (K) x 128 (rows).
mha_status encode_act(CUtensorMap *m, const void *base, long long M, int K) {
    const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(K) * 2};
    const uint32_t box[2] = {64, 128};
    return encode_bf16(m, base, 2, dims, strides, box);
}

// Weight (K rows x N) row-major viewed as (64, K, N/64): box (64, 64, bn/64).
mha_status encode_weight(CUtensorMap *m, const void *base, int K, int N, int bn) {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(K), static_cast<uint64_t>(N / 64)};
    const uint64_t strides[2] = {static_cast<uint64_t>(N) * 2, 128};
    const uint32_t box[3] = {64, 64, static_cast<uint32_t>(bn / 64)};
    return encode_bf16(m, base, 3, dims, strides, box);
}

// Output tile width for a launch: a 128 x 256 tile reads A from shared memory
// once per 256 columns and costs about 1.8 times a 128 x 128 tile, but halves
// the tile count; take the width with the smaller cost in whole waves over
// the SMs (small launches keep 128 so that every SM gets work).
int choose_bn(const long long *M, int np, int N, int sms) {
    long long t128 = 0, t256 = 0;
    for (int i = 0; i < np; ++i) {
        const long long mt = (M[i] + mha::kGemmBM - 1) / mha::kGemmBM;
        t128 += mt * ((N + 127) / 128);
        t256 += mt * ((N + 255) / 256);
    }
    const long long w128 = (t128 + sms - 1) / sms, w256 = (t256 + sms - 1) / sms;
    return 10 * w256 * 18 < 100 * w128 ? 256 : 128;
}

bool valid_mask(int mask) { return mask >= MHA_MASK_NONE && mask <= MHA_MASK_CAUSAL_KEY_PADDING; }

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Output map of a projection problem for the GEMM's TMA-store epilogue: 2-D
// over a row-major output, 3-D (64, T, B*H) over a head-split one whose T is a
// multiple of 128 (a 128-row tile then lies in one batch entry).  Sets
// pr.tma_store; a head-split output with another T is stored row by row.
mha_status encode_out(CUtensorMap *m, mha::GemmProblem &pr) {
    pr.tma_store = 0;
    mha_status s = MHA_OK;
    if (pr.out_mode == mha::kOutHeadSplit) {
        if (pr.T <= 0 || pr.T % mha::kGemmBM != 0) return MHA_OK;
        s = encode_heads(m, pr.out, static_cast<long long>(pr.M / pr.T) * pr.H, pr.T);
    } else {
        s = encode_act(m, pr.out, pr.M, pr.N);
    }
    if (s == MHA_OK) pr.tma_store = 1;
    return s;
}

mha_status launch_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return MHA_OK;
    return cuda_fail(what, cudaGetErrorName(e));
}

mha_status run_attention_bf16(const void *q, const void *k, const void *v, void *o,
                              long long o_sb, long long o_sh, long long o_st, int B, int h,
                              int T_q, int T_k, float scale, int mask, const int32_t *key_lens,
                              int *status_dev, cudaStream_t stream, float *lse = nullptr,
                              bool pdl = false, unsigned long long drill_wait_limit_ns = 0,
                              int drill_skip_tile = 0) {
    CUtensorMap tq, tk, tv;
    const long long BH = static_cast<long long>(B) * h;
    mha_status s;
    // T_k == 0: keys do not exist; the kernel then writes zeros.  A TMA map
    // needs every extent >= 1, so describe a one-row tensor it never loads.
    const int Tk_map = T_k > 0 ? T_k : 1;
    if ((s = encode_heads(&tq, q, BH, T_q)) != MHA_OK) return s;
    if ((s = encode_heads(&tk, k, BH, Tk_map)) != MHA_OK) return s;
    if ((s = encode_heads(&tv, v, BH, Tk_map)) != MHA_OK) return s;
    mha::AttnParams p;
    p.B = B;
    p.H = h;
    p.Tq = T_q;
    p.Tk = T_k;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.scale = scale;
    p.lse = lse;
    p.mask = mask;
    p.key_lens = key_lens;
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.o_stride_b = o_sb;
    p.o_stride_h = o_sh;
    p.o_stride_t = o_st;
    p.num_qblocks = (T_q + mha::kAttnRowsPerCta - 1) / mha::kAttnRowsPerCta;
    const long long items = BH * p.num_qblocks;
    if (items >= (1ll << 30)) return MHA_ERR_UNSUPPORTED;
    p.total_items = static_cast<int>(items);
    p.status = status_dev;
    p.wait_limit_ns = drill_wait_limit_ns;
    p.drill_skip_tile = drill_skip_tile;
    return launch_status(mha::launch_attn_bf16(tq, tk, tv, p, stream, pdl), "attention launch");
}

}  // namespace

MHA_EXPORT const char *mha_status_string(mha_status status) {
    switch (status) {
        case MHA_OK: return "ok";
        case MHA_ERR_INVALID_ARG: return "invalid argument";
        case MHA_ERR_UNSUPPORTED: return "unsupported configuration";
        case MHA_ERR_WORKSPACE: return "workspace missing or too small";
        case MHA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case MHA_ERR_CUDA: return "CUDA error";
        case MHA_ERR_TIMEOUT: return "kernel wait timed out";
        case MHA_ERR_BOUNDS: return "device-side bounds check failed";
    }
    return "unknown status";
}

MHA_EXPORT const char *mha_last_error(void) { return g_last_error; }

namespace mha {
mha_status record_cuda_failure(const char *what, const char *detail) { return cuda_fail(what, detail); }
}  // namespace mha

namespace {

mha_status sdpa_impl(mha_dtype dt, const void *q, const void *k, const void *v, void *o,
                     float *lse, int B, int h, int T_q, int T_k, int d_k, int d_v, float scale,
                     mha_mask mask, const int32_t *key_lens, int *status_dev,
                     cudaStream_t stream) {
    if (B < 0 || h < 0 || T_q < 0 || T_k < 0 || d_k <= 0 || d_v <= 0) return MHA_ERR_INVALID_ARG;
    if (!valid_mask(mask) || !isfinite(scale)) return MHA_ERR_INVALID_ARG;
    if ((mask & MHA_MASK_KEY_PADDING) && !key_lens) return MHA_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * h >= (1ll << 31)) return MHA_ERR_UNSUPPORTED;
    if (B == 0 || h == 0 || T_q == 0) return MHA_OK;
    if (!q || !o || (T_k > 0 && (!k || !v))) return MHA_ERR_INVALID_ARG;
    if (lse && dt != MHA_BF16) return dt == MHA_F32 ? MHA_ERR_UNSUPPORTED : MHA_ERR_INVALID_ARG;
    if (dt == MHA_F32) {
        if (d_k > 128 || d_v > 128) return MHA_ERR_UNSUPPORTED;
        if ((T_q + mha::kF32RowsPerCta - 1) / mha::kF32RowsPerCta > 65535) return MHA_ERR_UNSUPPORTED;
        return launch_status(mha::launch_sdpa_f32(
            static_cast<const float *>(q), static_cast<const float *>(k),
            static_cast<const float *>(v), static_cast<float *>(o), B, h, T_q, T_k, d_k, d_v,
            scale, mask, key_lens, stream), "fp32 attention launch");
    }
    if (dt != MHA_BF16) return MHA_ERR_INVALID_ARG;
    if (d_k != 64 || d_v != 64) return MHA_ERR_UNSUPPORTED;
    if ((T_q + mha::kAttnRowsPerCta - 1) / mha::kAttnRowsPerCta > 65535) return MHA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(o) || (T_k > 0 && (!aligned16(k) || !aligned16(v))))
        return MHA_ERR_MISALIGNED;
    const long long so_t = 64, so_h = static_cast<long long>(T_q) * 64, so_b = so_h * h;
    return run_attention_bf16(q, T_k > 0 ? k : q, T_k > 0 ? v : q, o, so_b, so_h, so_t, B, h,
                              T_q, T_k, scale, mask, key_lens, status_dev, stream, lse);
}

}  // namespace

MHA_EXPORT mha_status sdpa_forward(mha_dtype dt, const void *q, const void *k, const void *v,
                                   void *o, int B, int h, int T_q, int T_k, int d_k, int d_v,
                                   float scale, mha_mask mask, const int32_t *key_lens,
                                   int *status_dev, cudaStream_t stream) {
    return sdpa_impl(dt, q, k, v, o, nullptr, B, h, T_q, T_k, d_k, d_v, scale, mask, key_lens,
                     status_dev, stream);
}

MHA_EXPORT mha_status sdpa_forward_timeout_drill(const void *q, const void *k, const void *v,
                                                void *o, int B, int h, int T_q, int T_k,
                                                float scale, mha_mask mask,
                                                const int32_t *key_lens,
                                                unsigned long long wait_limit_ns, int skip_tile,
                                                int *status_dev, cudaStream_t stream) {
    if (B <= 0 || h <= 0 || T_q <= 0 || T_k <= 0 || skip_tile < 0) return MHA_ERR_INVALID_ARG;
    if (!valid_mask(mask) || !isfinite(scale)) return MHA_ERR_INVALID_ARG;
    if ((mask & MHA_MASK_KEY_PADDING) && !key_lens) return MHA_ERR_INVALID_ARG;
    if (wait_limit_ns < 100000ull || wait_limit_ns > 1000000000ull) return MHA_ERR_INVALID_ARG;
    if (!q || !k || !v || !o || !status_dev) return MHA_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * h >= (1ll << 31)) return MHA_ERR_UNSUPPORTED;
    if ((T_q + mha::kAttnRowsPerCta - 1) / mha::kAttnRowsPerCta > 65535) return MHA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(o) || !aligned16(k) || !aligned16(v)) return MHA_ERR_MISALIGNED;
    const long long so_t = 64, so_h = static_cast<long long>(T_q) * 64, so_b = so_h * h;
    return run_attention_bf16(q, k, v, o, so_b, so_h, so_t, B, h, T_q, T_k, scale, mask, key_lens,
                              status_dev, stream, nullptr, false, wait_limit_ns, skip_tile + 1);
}

MHA_EXPORT mha_status sdpa_forward_lse(mha_dtype dt, const void *q, const void *k, const void *v,
                                       void *o, float *lse, int B, int h, int T_q, int T_k,
                                       int d_k, int d_v, float scale, mha_mask mask,
                                       const int32_t *key_lens, int *status_dev,
                                       cudaStream_t stream) {
    if (!lse && B > 0 && h > 0 && T_q > 0) return MHA_ERR_INVALID_ARG;
    return sdpa_impl(dt, q, k, v, o, lse, B, h, T_q, T_k, d_k, d_v, scale, mask, key_lens,
                     status_dev, stream);
}

namespace {

// Internal streams and events of sdpa_forward_host, one set per device,
// created on first use and kept for the life of the process.  The enqueue
// sequence of one call holds the device's mutex: an event is re-recorded only
// after every wait on its previous record has been enqueued.
constexpr int kHostChunks = 6;  // measured best of 4-8 on the 32-head causal T=8192 workload
struct HostPipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr, in[kHostChunks] = {}, comp[kHostChunks] = {};
};
constexpr int kMaxDevices = 64;
HostPipe g_host_pipe[kMaxDevices];

mha_status host_pipe_init(HostPipe &hp) {
    if (hp.ready) return MHA_OK;
    cudaError_t e = cudaStreamCreateWithFlags(&hp.s_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.s_out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming);
    for (int i = 0; e == cudaSuccess && i < kHostChunks; ++i) {
        e = cudaEventCreateWithFlags(&hp.in[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.comp[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return cuda_fail("sdpa_forward_host setup", cudaGetErrorString(e));
    hp.ready = true;
    return MHA_OK;
}

// Device bytes of one copy of q, k, v, o and key_lens (each 256-byte aligned).
size_t host_ws_parts(mha_dtype dt, int B, int h, int T_q, int T_k, int d_k, int d_v, size_t *off) {
    const size_t es = dt == MHA_F32 ? 4 : 2;
    const size_t BH = static_cast<size_t>(B) * static_cast<size_t>(h);
    const size_t sz[5] = {BH * T_q * d_k * es, BH * T_k * d_k * es, BH * T_k * d_v * es,
                          BH * T_q * d_v * es, static_cast<size_t>(B) * 4};
    size_t at = 0;
    for (int i = 0; i < 5; ++i) {
        off[i] = at;
        at += round256(sz[i]);
    }
    return at;
}

}  // namespace

MHA_EXPORT int sdpa_bf16_key_split(int T_q, int T_k, mha_mask mask) {
    if (T_q < 0 || T_k < 0 || !valid_mask(mask)) return -1;
    return mha::attn_bf16_splits_by_tiles(T_q, T_k, static_cast<int>(mask)) ? 1 : 0;
}

MHA_EXPORT size_t sdpa_forward_host_workspace_bytes(mha_dtype dt, int B, int h, int T_q, int T_k,
                                                    int d_k, int d_v) {
    if (B < 0 || h < 0 || T_q < 0 || T_k < 0 || d_k <= 0 || d_v <= 0) return 0;
    size_t off[5];
    return host_ws_parts(dt, B, h, T_q, T_k, d_k, d_v, off);
}

MHA_EXPORT mha_status sdpa_forward_host(mha_dtype dt, const void *q_host, const void *k_host,
                                        const void *v_host, void *o_host, void *workspace,
                                        size_t workspace_bytes, int B, int h, int T_q, int T_k,
                                        int d_k, int d_v, float scale, mha_mask mask,
                                        const int32_t *key_lens_host, int *status_dev,
                                        cudaStream_t stream) {
    if (B < 0 || h < 0 || T_q < 0 || T_k < 0 || d_k <= 0 || d_v <= 0) return MHA_ERR_INVALID_ARG;
    if (dt != MHA_F32 && dt != MHA_BF16) return MHA_ERR_INVALID_ARG;
    if (!valid_mask(mask) || !isfinite(scale)) return MHA_ERR_INVALID_ARG;
    if ((mask & MHA_MASK_KEY_PADDING) && !key_lens_host) return MHA_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * h >= (1ll << 31)) return MHA_ERR_UNSUPPORTED;
    if (B == 0 || h == 0 || T_q == 0) return MHA_OK;
    if (!q_host || !o_host || (T_k > 0 && (!k_host || !v_host))) return MHA_ERR_INVALID_ARG;
    size_t off[5];
    const size_t need = host_ws_parts(dt, B, h, T_q, T_k, d_k, d_v, off);
    if (!workspace || workspace_bytes < need) return MHA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MHA_ERR_MISALIGNED;
    if (dt == MHA_BF16 && (d_k != 64 || d_v != 64)) return MHA_ERR_UNSUPPORTED;
    if (dt == MHA_F32 && (d_k > 128 || d_v > 128)) return MHA_ERR_UNSUPPORTED;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail("cudaGetDevice", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return MHA_ERR_UNSUPPORTED;
    HostPipe &hp = g_host_pipe[dev];
    std::lock_guard<std::mutex> lock(hp.mu);
    mha_status st = host_pipe_init(hp);
    if (st != MHA_OK) return st;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *qd = ws + off[0], *kd = ws + off[1], *vd = ws + off[2], *od = ws + off[3];
    int32_t *lens_d = reinterpret_cast<int32_t *>(ws + off[4]);
    const size_t es = dt == MHA_F32 ? 4 : 2;
    const size_t q_head = static_cast<size_t>(T_q) * d_k * es, k_head = static_cast<size_t>(T_k) * d_k * es;
    const size_t v_head = static_cast<size_t>(T_k) * d_v * es, o_head = static_cast<size_t>(T_q) * d_v * es;
    const bool padded = (mask & MHA_MASK_KEY_PADDING) != 0;

    // Chunks: whole batch items when h is small, else groups of heads of one
    // batch item (the kernels take key_lens per batch item).
    const long long BH = static_cast<long long>(B) * h;
    const long long per = (BH + kHostChunks - 1) / kHostChunks;
    const int nb = per >= h ? static_cast<int>(per / h) : 0;  // batch items per chunk
    const int nh = per >= h ? h : static_cast<int>(per);      // heads per chunk (of one item)

    auto fail = [](cudaError_t err, const char *what) { return cuda_fail(what, cudaGetErrorString(err)); };
    if ((e = cudaEventRecord(hp.start, stream)) != cudaSuccess) return fail(e, "cudaEventRecord");
    if ((e = cudaStreamWaitEvent(hp.s_in, hp.start, 0)) != cudaSuccess) return fail(e, "cudaStreamWaitEvent");
    if ((e = cudaStreamWaitEvent(hp.s_out, hp.start, 0)) != cudaSuccess) return fail(e, "cudaStreamWaitEvent");
    if (padded && (e = cudaMemcpyAsync(lens_d, key_lens_host, static_cast<size_t>(B) * 4,
                                       cudaMemcpyHostToDevice, hp.s_in)) != cudaSuccess)
        return fail(e, "key_lens copy");

    int chunk = 0;
    for (int b = 0; b < B;) {
        const int cb = nb > 0 ? std::min(nb, B - b) : 1;  // batch items [b, b + cb)
        for (int h0 = 0; h0 < h; h0 += (nb > 0 ? h : nh), ++chunk) {
            const int ch = nb > 0 ? h : std::min(nh, h - h0);  // heads [h0, h0 + ch) of each
            const size_t f = static_cast<size_t>(b) * h + h0;  // first flattened head
            const size_t nheads = static_cast<size_t>(cb) * ch;
            const int slot = chunk % kHostChunks;
            const char *qh = static_cast<const char *>(q_host), *kh = static_cast<const char *>(k_host);
            const char *vh = static_cast<const char *>(v_host);
            if ((e = cudaMemcpyAsync(qd + f * q_head, qh + f * q_head, nheads * q_head,
                                     cudaMemcpyHostToDevice, hp.s_in)) != cudaSuccess)
                return fail(e, "q copy");
            if (T_k > 0) {
                if ((e = cudaMemcpyAsync(kd + f * k_head, kh + f * k_head, nheads * k_head,
                                         cudaMemcpyHostToDevice, hp.s_in)) != cudaSuccess)
                    return fail(e, "k copy");
                if ((e = cudaMemcpyAsync(vd + f * v_head, vh + f * v_head, nheads * v_head,
                                         cudaMemcpyHostToDevice, hp.s_in)) != cudaSuccess)
                    return fail(e, "v copy");
            }
            if ((e = cudaEventRecord(hp.in[slot], hp.s_in)) != cudaSuccess) return fail(e, "cudaEventRecord");
            if ((e = cudaStreamWaitEvent(stream, hp.in[slot], 0)) != cudaSuccess)
                return fail(e, "cudaStreamWaitEvent");
            st = sdpa_impl(dt, qd + f * q_head, kd + f * k_head, vd + f * v_head, od + f * o_head, nullptr, cb,
                           ch, T_q, T_k, d_k, d_v, scale, mask, padded ? lens_d + b : nullptr, status_dev,
                           stream);
            if (st != MHA_OK) return st;
            if ((e = cudaEventRecord(hp.comp[slot], stream)) != cudaSuccess) return fail(e, "cudaEventRecord");
            if ((e = cudaStreamWaitEvent(hp.s_out, hp.comp[slot], 0)) != cudaSuccess)
                return fail(e, "cudaStreamWaitEvent");
            if ((e = cudaMemcpyAsync(static_cast<char *>(o_host) + f * o_head, od + f * o_head,
                                     nheads * o_head, cudaMemcpyDeviceToHost, hp.s_out)) != cudaSuccess)
                return fail(e, "o copy");
        }
        b += cb;
    }
    // later work on `stream` (and its synchronisation) covers the copies
    if ((e = cudaEventRecord(hp.done, hp.s_out)) != cudaSuccess) return fail(e, "cudaEventRecord");
    if ((e = cudaStreamWaitEvent(stream, hp.done, 0)) != cudaSuccess) return fail(e, "cudaStreamWaitEvent");
    return MHA_OK;
}

MHA_EXPORT size_t sdpa_backward_workspace_bytes(int B, int h, int T_q, int T_k, int d_k, int d_v) {
    if (B < 0 || h < 0 || T_q < 0 || T_k < 0 || d_k < 0 || d_v < 0) return 0;
    (void)T_k;
    return mha::bwd_workspace_bytes(static_cast<long long>(B) * h, T_q);
}

MHA_EXPORT mha_status sdpa_backward(mha_dtype dt, const void *q, const void *k, const void *v,
                                    const void *o, const void *dout, const float *lse, void *dq,
                                    void *dk, void *dv, void *workspace, size_t workspace_bytes,
                                    int B, int h, int T_q, int T_k, int d_k, int d_v, float scale,
                                    mha_mask mask, const int32_t *key_lens, int *status_dev,
                                    cudaStream_t stream) {
    if (B < 0 || h < 0 || T_q < 0 || T_k < 0 || d_k <= 0 || d_v <= 0) return MHA_ERR_INVALID_ARG;
    if (!valid_mask(mask) || !isfinite(scale)) return MHA_ERR_INVALID_ARG;
    if ((mask & MHA_MASK_KEY_PADDING) && !key_lens) return MHA_ERR_INVALID_ARG;
    if (dt != MHA_BF16) return dt == MHA_F32 ? MHA_ERR_UNSUPPORTED : MHA_ERR_INVALID_ARG;
    if (d_k != 64 || d_v != 64) return MHA_ERR_UNSUPPORTED;
    const long long BH = static_cast<long long>(B) * h;
    if (BH >= (1ll << 31) || (T_k + 127) / 128 > 65535) return MHA_ERR_UNSUPPORTED;
    if (BH == 0 || (T_q == 0 && T_k == 0)) return MHA_OK;
    if ((T_q > 0 && (!q || !o || !dout || !lse || !dq)) || (T_k > 0 && (!k || !v || !dk || !dv)))
        return MHA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < mha::bwd_workspace_bytes(BH, T_q)) return MHA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MHA_ERR_MISALIGNED;
    if ((T_q > 0 && (!aligned16(q) || !aligned16(o) || !aligned16(dout) || !aligned16(dq))) ||
        (T_k > 0 && (!aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv))))
        return MHA_ERR_MISALIGNED;
    // A tensor map needs every extent >= 1: describe a one-row tensor for an
    // empty side (the kernels never load it).
    const void *q_src = T_q > 0 ? q : k, *g_src = T_q > 0 ? dout : k;
    const void *k_src = T_k > 0 ? k : q, *v_src = T_k > 0 ? v : q;
    CUtensorMap tq, tk, tv, tg;
    mha_status s;
    if ((s = encode_heads(&tq, q_src, BH, T_q > 0 ? T_q : 1)) != MHA_OK) return s;
    if ((s = encode_heads(&tg, g_src, BH, T_q > 0 ? T_q : 1)) != MHA_OK) return s;
    if ((s = encode_heads(&tk, k_src, BH, T_k > 0 ? T_k : 1)) != MHA_OK) return s;
    if ((s = encode_heads(&tv, v_src, BH, T_k > 0 ? T_k : 1)) != MHA_OK) return s;
    mha::BwdParams p{};
    p.B = B;
    p.H = h;
    p.Tq = T_q;
    p.Tk = T_k;
    p.Tq_pad = (T_q + 127) / 128 * 128;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.mask = mask;
    p.key_lens = key_lens;
    p.dk = static_cast<__nv_bfloat16 *>(dk);
    p.dv = static_cast<__nv_bfloat16 *>(dv);
    p.status = status_dev;
    return launch_status(
        mha::launch_attn_bwd_bf16(tq, tk, tv, tg, static_cast<const __nv_bfloat16 *>(o),
                                  static_cast<const __nv_bfloat16 *>(dout), lse,
                                  static_cast<__nv_bfloat16 *>(dq), p, workspace, stream),
        "attention backward launch");
}

MHA_EXPORT mha_status sdpa_decode_forward(const void *q, const void *k_cache,
                                          const void *v_cache, void *o, int B, int h, int T_q,
                                          int T_k, int d_k, int d_v, float scale,
                                          const int32_t *cache_lens, cudaStream_t stream) {
    if (B < 0 || h < 0 || T_q < 0 || T_k < 0 || d_k <= 0 || d_v <= 0 || !isfinite(scale))
        return MHA_ERR_INVALID_ARG;
    if (T_q > mha::kDecodeMaxRows) return MHA_ERR_UNSUPPORTED;
    if (d_k != 64 || d_v != 64) return MHA_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * h * 8 >= (1ll << 31)) return MHA_ERR_UNSUPPORTED;
    if (B == 0 || h == 0 || T_q == 0) return MHA_OK;
    if (!q || !o || (T_k > 0 && (!k_cache || !v_cache))) return MHA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(o) || (T_k > 0 && (!aligned16(k_cache) || !aligned16(v_cache))))
        return MHA_ERR_MISALIGNED;
    mha::DecodeParams p;
    p.B = B;
    p.H = h;
    p.Tq = T_q;
    p.Tk = T_k;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.key_lens = cache_lens;
    return launch_status(
        mha::launch_decode_bf16(static_cast<const __nv_bfloat16 *>(q),
                                static_cast<const __nv_bfloat16 *>(k_cache),
                                static_cast<const __nv_bfloat16 *>(v_cache),
                                static_cast<__nv_bfloat16 *>(o), p, stream),
        "decode attention launch");
}

MHA_EXPORT size_t mha_workspace_bytes(int B, int h, int T_q, int T_k, int d_k, int d_v) {
    if (B < 0 || h < 0 || T_q < 0 || T_k < 0 || d_k < 0 || d_v < 0) return 0;
    const size_t bh = static_cast<size_t>(B) * h;
    return round256(bh * T_q * d_k * 2) + round256(bh * T_k * d_k * 2) +
           round256(bh * T_k * d_v * 2) + round256(bh * T_q * d_v * 2);
}

namespace {

// Residual + layer normalisation applied after the output projection.
struct LnArgs {
    const void *gamma, *beta;
    float eps;
};

mha_status mha_impl(mha_dtype dt, const void *x_q, const void *x_kv, const void *w_q,
                    const void *w_k, const void *w_v, const void *w_o, void *out,
                    void *workspace, size_t workspace_bytes, int B, int h, int T_q, int T_k,
                    int d_model, int d_k, int d_v, float scale, mha_mask mask,
                    const int32_t *key_lens, int *status_dev, cudaStream_t stream,
                    const LnArgs *ln) {
    if (B < 0 || h <= 0 || T_q < 0 || T_k < 0 || d_model <= 0 || d_k <= 0 || d_v <= 0)
        return MHA_ERR_INVALID_ARG;
    if (!valid_mask(mask) || !isfinite(scale)) return MHA_ERR_INVALID_ARG;
    if ((mask & MHA_MASK_KEY_PADDING) && !key_lens) return MHA_ERR_INVALID_ARG;
    if (dt != MHA_BF16) return dt == MHA_F32 ? MHA_ERR_UNSUPPORTED : MHA_ERR_INVALID_ARG;
    if (d_k != 64 || d_v != 64) return MHA_ERR_UNSUPPORTED;
    if (d_model % 64 != 0) return MHA_ERR_UNSUPPORTED;
    if (ln && mha::ln_tile_width(d_model, 1, 1) == 0) return MHA_ERR_UNSUPPORTED;
    if (ln && !(ln->eps >= 0.f && isfinite(ln->eps))) return MHA_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * h >= (1ll << 31) ||
        static_cast<long long>(B) * (T_q > T_k ? T_q : T_k) >= (1ll << 31))
        return MHA_ERR_UNSUPPORTED;
    if ((T_q + mha::kAttnRowsPerCta - 1) / mha::kAttnRowsPerCta > 65535) return MHA_ERR_UNSUPPORTED;
    if (B == 0 || T_q == 0) return MHA_OK;
    if (!x_q || !out || !w_q || !w_o || (T_k > 0 && (!x_kv || !w_k || !w_v)))
        return MHA_ERR_INVALID_ARG;
    if (ln && (!ln->gamma || !ln->beta)) return MHA_ERR_INVALID_ARG;
    if (ln && (!aligned16(ln->gamma) || !aligned16(ln->beta))) return MHA_ERR_MISALIGNED;
    if (!workspace || workspace_bytes < mha_workspace_bytes(B, h, T_q, T_k, d_k, d_v))
        return MHA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MHA_ERR_MISALIGNED;
    if (!aligned16(x_q) || !aligned16(out) || !aligned16(w_q) || !aligned16(w_o) ||
        (T_k > 0 && (!aligned16(x_kv) || !aligned16(w_k) || !aligned16(w_v))))
        return MHA_ERR_MISALIGNED;

    const int hd = h * 64;
    const size_t bh = static_cast<size_t>(B) * h;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *qh = ws;
    void *kh = ws + round256(bh * T_q * 128);
    void *vh = static_cast<uint8_t *>(kh) + round256(bh * T_k * 128);
    void *om = static_cast<uint8_t *>(vh) + round256(bh * T_k * 128);
    const long long Mq = static_cast<long long>(B) * T_q, Mk = static_cast<long long>(B) * T_k;
    int sms = 0;
    if (mha::sm_count(&sms) != cudaSuccess || sms <= 0)
        return cuda_fail("cudaDeviceGetAttribute", "SM count");

    // 1. Q, K, V projections with the head split folded into the epilogue.
    CUtensorMap ta[mha::kGemmMaxProblems], tb[mha::kGemmMaxProblems], ty[mha::kGemmMaxProblems] = {};
    mha::GemmParams gp{};
    gp.status = status_dev;
    mha_status s;
    struct In {
        const void *x, *w;
        void *out;
        long long M;
        int T;
    } ins[3] = {{x_q, w_q, qh, Mq, T_q}, {x_kv, w_k, kh, Mk, T_k}, {x_kv, w_v, vh, Mk, T_k}};
    long long Ms[3];
    int nm = 0;
    for (int i = 0; i < 3; ++i)
        if (ins[i].M > 0) Ms[nm++] = ins[i].M;
    gp.bn = choose_bn(Ms, nm, hd, sms);
    int np = 0, tiles = 0;
    for (int i = 0; i < 3; ++i) {
        if (ins[i].M == 0) continue;
        if ((s = encode_act(&ta[np], ins[i].x, ins[i].M, d_model)) != MHA_OK) return s;
        if ((s = encode_weight(&tb[np], ins[i].w, d_model, hd, gp.bn)) != MHA_OK) return s;
        mha::GemmProblem &pr = gp.prob[np];
        pr.M = static_cast<int>(ins[i].M);
        pr.N = hd;
        pr.K = d_model;
        pr.tiles_n = (hd + gp.bn - 1) / gp.bn;
        pr.tile_start = tiles;
        pr.tile_count = pr.tiles_n * static_cast<int>((ins[i].M + mha::kGemmBM - 1) / mha::kGemmBM);
        pr.out = static_cast<__nv_bfloat16 *>(ins[i].out);
        pr.out_mode = mha::kOutHeadSplit;
        pr.T = ins[i].T;
        pr.H = h;
        if ((s = encode_out(&ty[np], pr)) != MHA_OK) return s;
        tiles += pr.tile_count;
        ++np;
    }
    for (int i = np; i < mha::kGemmMaxProblems; ++i) {
        ta[i] = ta[0];
        tb[i] = tb[0];
        ty[i] = ty[0];
    }
    gp.num_problems = np;
    gp.total_tiles = tiles;
    if ((s = launch_status(mha::launch_gemm_bf16(ta, tb, ty, gp, stream), "projection GEMM launch")) !=
        MHA_OK)
        return s;

    // 2. Fused attention, writing the merged (B, T_q, h*64) layout directly.
    if ((s = run_attention_bf16(qh, T_k > 0 ? kh : qh, T_k > 0 ? vh : qh, om,
                                static_cast<long long>(T_q) * hd, 64, hd, B, h, T_q, T_k, scale,
                                mask, key_lens, status_dev, stream, nullptr, true)) != MHA_OK)
        return s;

    // 3. Output projection Concat(heads) W^O, alone or fused with the
    //    residual connection and layer normalisation.
    if (ln) {
        mha::LnParams lp{};
        lp.M = static_cast<int>(Mq);
        lp.D = d_model;
        lp.K = hd;
        lp.bn = mha::ln_tile_width(d_model, Mq, sms);
        lp.resid = static_cast<const __nv_bfloat16 *>(x_q);
        lp.gamma = static_cast<const __nv_bfloat16 *>(ln->gamma);
        lp.beta = static_cast<const __nv_bfloat16 *>(ln->beta);
        lp.eps = ln->eps;
        lp.out = static_cast<__nv_bfloat16 *>(out);
        lp.status = status_dev;
        CUtensorMap la, lb, lx, ly;
        if ((s = encode_act(&la, om, Mq, hd)) != MHA_OK) return s;
        if ((s = encode_weight(&lb, w_o, hd, d_model, lp.bn)) != MHA_OK) return s;
        if ((s = encode_act(&lx, x_q, Mq, d_model)) != MHA_OK) return s;
        if ((s = encode_act(&ly, lp.out, Mq, d_model)) != MHA_OK) return s;
        return launch_status(mha::launch_gemm_ln_bf16(la, lb, lx, ly, lp, stream, true),
                             "output projection + layer norm launch");
    }
    mha::GemmParams go{};
    go.status = status_dev;
    go.bn = choose_bn(&Mq, 1, d_model, sms);
    if ((s = encode_act(&ta[0], om, Mq, hd)) != MHA_OK) return s;
    if ((s = encode_weight(&tb[0], w_o, hd, d_model, go.bn)) != MHA_OK) return s;
    mha::GemmProblem &pr = go.prob[0];
    pr.M = static_cast<int>(Mq);
    pr.N = d_model;
    pr.K = hd;
    pr.tiles_n = (d_model + go.bn - 1) / go.bn;
    pr.tile_start = 0;
    pr.tile_count = pr.tiles_n * static_cast<int>((Mq + mha::kGemmBM - 1) / mha::kGemmBM);
    pr.out = static_cast<__nv_bfloat16 *>(out);
    pr.out_mode = mha::kOutRowMajor;
    pr.T = T_q;
    pr.H = h;
    if ((s = encode_out(&ty[0], pr)) != MHA_OK) return s;
    for (int i = 1; i < mha::kGemmMaxProblems; ++i) {
        ta[i] = ta[0];
        tb[i] = tb[0];
        ty[i] = ty[0];
    }
    go.num_problems = 1;
    go.total_tiles = pr.tile_count;
    return launch_status(mha::launch_gemm_bf16(ta, tb, ty, go, stream, true), "output GEMM launch");
}

}  // namespace

MHA_EXPORT mha_status mha_forward(mha_dtype dt, const void *x_q, const void *x_kv,
                                  const void *w_q, const void *w_k, const void *w_v,
                                  const void *w_o, void *out, void *workspace,
                                  size_t workspace_bytes, int B, int h, int T_q, int T_k,
                                  int d_model, int d_k, int d_v, float scale, mha_mask mask,
                                  const int32_t *key_lens, int *status_dev, cudaStream_t stream) {
    return mha_impl(dt, x_q, x_kv, w_q, w_k, w_v, w_o, out, workspace, workspace_bytes, B, h,
                    T_q, T_k, d_model, d_k, d_v, scale, mask, key_lens, status_dev, stream,
                    nullptr);
}

MHA_EXPORT mha_status positional_encoding_add(const void *x, void *out, int B, int T, int d_model,
                                              int pos0, cudaStream_t stream) {
    if (B < 0 || T < 0 || d_model <= 0 || pos0 < 0) return MHA_ERR_INVALID_ARG;
    if (d_model % 8 != 0) return MHA_ERR_UNSUPPORTED;
    if (static_cast<long long>(pos0) + T >= (1ll << 24)) return MHA_ERR_UNSUPPORTED;  // exact fp32 positions
    if (B == 0 || T == 0) return MHA_OK;
    if (!x || !out) return MHA_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out)) return MHA_ERR_MISALIGNED;
    return launch_status(mha::launch_posenc_add_bf16(static_cast<const __nv_bfloat16 *>(x),
                                                     static_cast<__nv_bfloat16 *>(out),
                                                     static_cast<long long>(B) * T, T, d_model,
                                                     pos0, stream),
                         "positional encoding launch");
}

MHA_EXPORT size_t encoder_layer_workspace_bytes(int B, int T, int d_model, int h, int d_ff) {
    if (B < 0 || T < 0 || d_model < 0 || h < 0 || d_ff < 0) return 0;
    const size_t rows = static_cast<size_t>(B) * T;
    return round256(mha_workspace_bytes(B, h, T, T, 64, 64)) + round256(rows * d_model * 2) +
           round256(rows * d_ff * 2);
}

MHA_EXPORT mha_status encoder_layer_forward(
    const void *x, const void *w_q, const void *w_k, const void *w_v, const void *w_o,
    const void *gamma1, const void *beta1, const void *w1, const void *b1, const void *w2,
    const void *b2, const void *gamma2, const void *beta2, float eps, void *out, void *workspace,
    size_t workspace_bytes, int B, int T, int d_model, int h, int d_ff, float scale, mha_mask mask,
    const int32_t *key_lens, int *status_dev, cudaStream_t stream) {
    if (B < 0 || T < 0 || d_model <= 0 || h <= 0 || d_ff <= 0) return MHA_ERR_INVALID_ARG;
    if (d_ff % 64 != 0 || d_model != h * 64) return MHA_ERR_UNSUPPORTED;
    if (B == 0 || T == 0) return MHA_OK;
    if (!x || !out || !w1 || !b1 || !w2 || !b2 || !gamma2 || !beta2) return MHA_ERR_INVALID_ARG;
    if (!(eps >= 0.f && isfinite(eps))) return MHA_ERR_INVALID_ARG;
    if (!aligned16(w1) || !aligned16(b1) || !aligned16(w2) || !aligned16(b2) || !aligned16(gamma2) ||
        !aligned16(beta2))
        return MHA_ERR_MISALIGNED;
    if (!workspace || workspace_bytes < encoder_layer_workspace_bytes(B, T, d_model, h, d_ff))
        return MHA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MHA_ERR_MISALIGNED;
    const size_t rows = static_cast<size_t>(B) * T;
    const size_t mha_ws = round256(mha_workspace_bytes(B, h, T, T, 64, 64));
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *y1 = ws + mha_ws;
    void *hid = ws + mha_ws + round256(rows * d_model * 2);
    // 1. y1 = LayerNorm1(x + MultiHead(x, x)): the attention sublayer (checks
    //    the remaining arguments, including d_model's support by the fused
    //    normalisation).
    const LnArgs ln1{gamma1, beta1, eps};
    mha_status s = mha_impl(MHA_BF16, x, x, w_q, w_k, w_v, w_o, y1, ws, mha_ws, B, h, T, T,
                            d_model, 64, 64, scale, mask, key_lens, status_dev, stream, &ln1);
    if (s != MHA_OK) return s;
    int sms = 0;
    if (mha::sm_count(&sms) != cudaSuccess || sms <= 0)
        return cuda_fail("cudaDeviceGetAttribute", "SM count");
    const long long M = static_cast<long long>(rows);
    // 2. hid = max(0, y1 W1 + b1): projection GEMM with a bias + ReLU epilogue.
    CUtensorMap ta[mha::kGemmMaxProblems], tb[mha::kGemmMaxProblems], ty[mha::kGemmMaxProblems] = {};
    mha::GemmParams gp{};
    gp.status = status_dev;
    gp.bn = choose_bn(&M, 1, d_ff, sms);
    if ((s = encode_act(&ta[0], y1, M, d_model)) != MHA_OK) return s;
    if ((s = encode_weight(&tb[0], w1, d_model, d_ff, gp.bn)) != MHA_OK) return s;
    mha::GemmProblem &pr = gp.prob[0];
    pr.M = static_cast<int>(M);
    pr.N = d_ff;
    pr.K = d_model;
    pr.tiles_n = (d_ff + gp.bn - 1) / gp.bn;
    pr.tile_start = 0;
    pr.tile_count = pr.tiles_n * static_cast<int>((M + mha::kGemmBM - 1) / mha::kGemmBM);
    pr.out = static_cast<__nv_bfloat16 *>(hid);
    pr.out_mode = mha::kOutRowMajor;
    pr.bias = static_cast<const __nv_bfloat16 *>(b1);
    pr.relu = 1;
    if ((s = encode_out(&ty[0], pr)) != MHA_OK) return s;
    for (int i = 1; i < mha::kGemmMaxProblems; ++i) {
        ta[i] = ta[0];
        tb[i] = tb[0];
        ty[i] = ty[0];
    }
    gp.num_problems = 1;
    gp.total_tiles = pr.tile_count;
    if ((s = launch_status(mha::launch_gemm_bf16(ta, tb, ty, gp, stream, true), "feed-forward GEMM launch")) !=
        MHA_OK)
        return s;
    // 3. out = LayerNorm2(y1 + hid W2 + b2): the normalising GEMM with a bias.
    mha::LnParams lp{};
    lp.M = static_cast<int>(M);
    lp.D = d_model;
    lp.K = d_ff;
    lp.bn = mha::ln_tile_width(d_model, M, sms);
    lp.resid = static_cast<const __nv_bfloat16 *>(y1);
    lp.bias = static_cast<const __nv_bfloat16 *>(b2);
    lp.gamma = static_cast<const __nv_bfloat16 *>(gamma2);
    lp.beta = static_cast<const __nv_bfloat16 *>(beta2);
    lp.eps = eps;
    lp.out = static_cast<__nv_bfloat16 *>(out);
    lp.status = status_dev;
    CUtensorMap la, lb, lx, ly;
    if ((s = encode_act(&la, hid, M, d_ff)) != MHA_OK) return s;
    if ((s = encode_weight(&lb, w2, d_ff, d_model, lp.bn)) != MHA_OK) return s;
    if ((s = encode_act(&lx, y1, M, d_model)) != MHA_OK) return s;
    if ((s = encode_act(&ly, lp.out, M, d_model)) != MHA_OK) return s;
    return launch_status(mha::launch_gemm_ln_bf16(la, lb, lx, ly, lp, stream, true),
                         "feed-forward output + layer norm launch");
}

MHA_EXPORT mha_status mha_forward_add_layernorm(
    mha_dtype dt, const void *x_q, const void *x_kv, const void *w_q, const void *w_k,
    const void *w_v, const void *w_o, const void *gamma, const void *beta, float eps, void *out,
    void *workspace, size_t workspace_bytes, int B, int h, int T_q, int T_k, int d_model,
    int d_k, int d_v, float scale, mha_mask mask, const int32_t *key_lens, int *status_dev,
    cudaStream_t stream) {
    const LnArgs ln{gamma, beta, eps};
    return mha_impl(dt, x_q, x_kv, w_q, w_k, w_v, w_o, out, workspace, workspace_bytes, B, h,
                    T_q, T_k, d_model, d_k, d_v, scale, mask, key_lens, status_dev, stream, &ln);
}
