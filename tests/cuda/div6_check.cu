// Exhaustive check of div6_rn (the quantizer's block-scale division) against
// IEEE division: every non-negative finite float a, RN(a / 6).  Prints the
// number of mismatches; exit status 0 iff the kernel ran.
#include <cstdio>
#include <cstdint>

#include "device_common.cuh"

__global__ void check_div6(unsigned long long* bad) {
    for (uint32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < 0x7F800000u; u += gridDim.x * blockDim.x) {
        const float a = __uint_as_float(u);
        if (__float_as_uint(nvfp4::div6_rn(a)) != __float_as_uint(__fdiv_rn(a, 6.0f))) atomicAdd(bad, 1ull);
    }
}

int main() {
    unsigned long long* bad = nullptr;
    if (cudaMalloc(&bad, sizeof(*bad)) != cudaSuccess) return 1;
    cudaMemset(bad, 0, sizeof(*bad));
    check_div6<<<1024, 256>>>(bad);
    const cudaError_t e = cudaDeviceSynchronize();
    unsigned long long h = ~0ull;
    cudaMemcpy(&h, bad, sizeof(h), cudaMemcpyDeviceToHost);
    printf("mismatches %llu (%s)\n", h, cudaGetErrorString(e));
    return e == cudaSuccess ? 0 : 1;
}
