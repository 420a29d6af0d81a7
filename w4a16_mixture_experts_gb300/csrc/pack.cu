// INT4 packing into the storage format of the expert weights.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// INT4 packing (model card, "What is quantized": pack-quantized storage):
// word w of a row holds q[8w+i] + 8 in bits [4i, 4i+4).
__global__ void pack_int4_kernel(const int8_t *__restrict__ q, int64_t nwords, int32_t *__restrict__ packed,
                                 int32_t *__restrict__ bad) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nwords) return;
    const uint2 v = *reinterpret_cast<const uint2 *>(q + 8 * i);
    uint32_t word = 0;
    int nbad = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        int x = (int)(int8_t)((b < 4 ? v.x >> (8 * b) : v.y >> (8 * (b - 4))) & 0xffu);
        if (x < -8) { x = -8; ++nbad; }
        if (x > 7) { x = 7; ++nbad; }
        word |= (uint32_t)(x + 8) << (4 * b);
    }
    packed[i] = (int32_t)word;
    if (nbad && bad) atomicAdd(bad, nbad);
}

cudaError_t launch_pack_int4(const int8_t *q, int64_t N, int64_t K, int32_t *packed, int32_t *bad,
                             cudaStream_t s) {
    const int64_t nwords = N * (K / 8);
    if (nwords == 0) return cudaSuccess;
    const int64_t blocks = (nwords + 255) / 256;
    pack_int4_kernel<<<(unsigned)blocks, 256, 0, s>>>(q, nwords, packed, bad);
    return cudaGetLastError();
}

}  // namespace moe
