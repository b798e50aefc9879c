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
    mx_quantize_group32(q + g * 32, out + g * 32);
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
