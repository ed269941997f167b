// Test helper (not part of the library): converts every fp32 bit pattern of a
// range with the same device conversion the writer uses (pairwise, saturating,
// round-to-nearest-even E4M3), so the test can compare it with the oracle codec.
#include <cstdint>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

__global__ void cvt_pairs(uint64_t lo, uint64_t n_pairs, uint8_t* out) {
    const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
    for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_pairs; i += stride) {
        const float2 v = make_float2(__uint_as_float(static_cast<uint32_t>(lo + 2 * i)),
                                     __uint_as_float(static_cast<uint32_t>(lo + 2 * i + 1)));
        const __nv_fp8x2_storage_t p = __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);
        out[2 * i] = static_cast<uint8_t>(p & 0xFF);
        out[2 * i + 1] = static_cast<uint8_t>(p >> 8);
    }
}

extern "C" int e4m3_cvt_range(uint64_t lo, uint64_t n, uint8_t* out_dev) {
    if (n % 2) return -1;
    cvt_pairs<<<4096, 256>>>(lo, n / 2, out_dev);
    if (cudaGetLastError() != cudaSuccess) return -2;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : -3;
}
