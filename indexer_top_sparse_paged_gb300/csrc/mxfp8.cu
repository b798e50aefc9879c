// MXFP8 quantisation of the indexer query ("Day0 Inference Support ... on Huawei Ascend CANN
// Architecture" §3: MXFP8 dynamic quantisation in the indexing stage; OCP Microscaling Formats:
// E4M3 elements sharing one E8M0 scale per 32 consecutive elements).
//
// One thread per group of 32 consecutive elements of q_I (within one head's row): amax, the shared
// exponent X = floor(log2(amax)) - 8 (at least -127), codes RNE_e4m3(x * 2^-X) saturating at
// +-448, and the decoded values code * 2^X written back as bf16 (exact), so the indexer kernels
// read an ordinary bf16 query whose values are the MXFP8 ones and keep exact bf16 products.
#include "internal.h"

namespace dsa {

constexpr int kMxThreads = 256;

__global__ void __launch_bounds__(kMxThreads)
    mx_quantize_q_kernel(const uint16_t* __restrict__ q, uint16_t* __restrict__ out, int64_t groups) {
    griddep_launch_dependents();  // the indexer may start its prologue (it waits for this grid)
    const int64_t g = static_cast<int64_t>(blockIdx.x) * kMxThreads + threadIdx.x;
    if (g >= groups) return;
    const uint4* src = reinterpret_cast<const uint4*>(q + g * 32);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = src[i];
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    uint32_t codes[8];
    const int X = mx_encode32(w, codes);
    const float up = e8m0_value(static_cast<uint32_t>(X + 127));  // 2^X
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {  // element pair 2i, 2i + 1: bytes 2(i % 2), 2(i % 2) + 1 of code word i / 2
        const __nv_fp8x2_storage_t c = static_cast<__nv_fp8x2_storage_t>((codes[i >> 1] >> (16 * (i & 1))) & 0xFFFFu);
        const __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(c, __NV_E4M3);
        const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&h2));  // .x = the lower code
        const __nv_bfloat162 b = __floats2bfloat162_rn(v.x * up, v.y * up);
        o[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + g * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
}

bool launch_mx_quantize_q(const void* q_I, void* out, int64_t elements, cudaStream_t s, int* launches) {
    const int64_t groups = elements / 32;
    if (groups == 0) return true;
    const int64_t grid = (groups + kMxThreads - 1) / kMxThreads;
    // the first kernel of its call: it waits for all earlier work on the stream
    if (!launch_kernel(false, mx_quantize_q_kernel, dim3(static_cast<unsigned>(grid)), dim3(kMxThreads), 0, s,
                       static_cast<const uint16_t*>(q_I), static_cast<uint16_t*>(out), groups))
        return false;
    ++*launches;
    return true;
}

}  // namespace dsa
