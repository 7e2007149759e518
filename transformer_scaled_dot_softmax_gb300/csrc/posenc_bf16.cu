// posenc_bf16.cu -- adds the sinusoidal positional encoding to a batch of
// embedding rows, on sm_103a:
//   out[b, t, 2i]   = x[b, t, 2i]   + sin(pos / 10000^(2i/D)),
//   out[b, t, 2i+1] = x[b, t, 2i+1] + cos(pos / 10000^(2i/D)),   pos = pos0 + t
// ("Attention is All You Need" notebook chapter, Positional Encoding;
// aiany.app Step 8).  Elementwise and bound by memory: one thread per 8
// features (one 16-byte load and store), the angle in fp32 (pos is exact, the
// frequency 10000^(-2i/D) has a relative error ~1e-7, so the angle is good to
// ~1e-7 * pos radians -- far below the bf16 rounding of the output).
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace mha {
namespace {

__global__ void posenc_add_kernel(const __nv_bfloat16 *__restrict__ x, __nv_bfloat16 *out,
                                  long long rows, int T, int D, int pos0) {
    const int per_row = D / 8;
    const long long t_id = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t_id >= rows * per_row) return;
    const long long row = t_id / per_row;
    const int c0 = static_cast<int>(t_id - row * per_row) * 8;
    const float pos = static_cast<float>(pos0 + static_cast<int>(row % T));
    const uint4 u = *reinterpret_cast<const uint4 *>(x + row * D + c0);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    const float kLog2Base = 13.287712379549449f;  // log2(10000)
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int i2 = c0 + 2 * e;  // the pair (2i, 2i+1) shares one frequency
        const float angle = pos * exp2f(-kLog2Base * static_cast<float>(i2) / static_cast<float>(D));
        float sn, cs;
        sincosf(angle, &sn, &cs);
        o[e] = pack_bf16x2(__uint_as_float(w[e] << 16) + sn, __uint_as_float(w[e] & 0xffff0000u) + cs);
    }
    *reinterpret_cast<uint4 *>(out + row * D + c0) = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

cudaError_t launch_posenc_add_bf16(const __nv_bfloat16 *x, __nv_bfloat16 *out, long long rows, int T,
                                   int D, int pos0, cudaStream_t stream) {
    const long long threads = rows * (D / 8);
    if (threads == 0) return cudaSuccess;
    posenc_add_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(x, out, rows, T, D,
                                                                                      pos0);
    return cudaGetLastError();
}

}  // namespace mha
