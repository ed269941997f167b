// Test helper (not part of the library): compares the E4M3 code the writer stores
// for x / s (its fast division) with the code of the IEEE quotient, on every pair
// (bf16 amax > 0, bf16 x with |x| <= amax, or NaN), s = RN(amax / 448) as the
// writer forms it.
#include <cstdint>
#include <cuda_runtime.h>

#include "../../fp8_mla_kv_gb300/csrc/mla_device.cuh"

__global__ void check(unsigned long long* n_checked, unsigned long long* n_bad, unsigned long long* n_ex,
                      uint32_t* examples) {
    const uint32_t amax_bits = blockIdx.x + 1;                  // 0x0001 .. 0x7F7F (finite, > 0)
    const float amax = __uint_as_float(amax_bits << 16);
    const float s = __fdiv_rn(amax, MLA_FP8_MAX);
    if (!(s >= mla::kDivFastMin && s <= mla::kDivFastMax)) return;   // writer takes the IEEE path
    const float y = __frcp_rn(s);
    unsigned long long checked = 0, bad = 0;
    for (uint32_t xb = threadIdx.x; xb < 65536; xb += blockDim.x) {
        const float x = __uint_as_float(xb << 16);
        if (!(fabsf(x) <= amax) && !isnan(x)) continue;
        const float a = mla::div_by_scale(x, s, y);
        const float b = __fdiv_rn(x, s);
        ++checked;
        const bool same = __nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3) ==
                          __nv_cvt_float_to_fp8(b, __NV_SATFINITE, __NV_E4M3);
        if (!same) {
            ++bad;
            const unsigned long long k = atomicAdd(n_ex, 1ull);     // one example slot per mismatch
            if (k < 8) { examples[2 * k] = amax_bits; examples[2 * k + 1] = xb; }
        }
    }
    atomicAdd(n_checked, checked);
    if (bad) atomicAdd(n_bad, bad);
}

extern "C" int div_check(unsigned long long* host_counts, uint32_t* host_examples) {
    unsigned long long* d;
    uint32_t* e;
    if (cudaMalloc(&d, 3 * sizeof(unsigned long long)) != cudaSuccess) return -1;
    if (cudaMalloc(&e, 16 * sizeof(uint32_t)) != cudaSuccess) return -1;
    cudaMemset(d, 0, 3 * sizeof(unsigned long long));
    cudaMemset(e, 0, 16 * sizeof(uint32_t));
    check<<<0x7F7F, 256>>>(d, d + 1, d + 2, e);
    if (cudaDeviceSynchronize() != cudaSuccess) return -2;
    cudaMemcpy(host_counts, d, 2 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    cudaMemcpy(host_examples, e, 16 * sizeof(uint32_t), cudaMemcpyDeviceToHost);
    cudaFree(d);
    cudaFree(e);
    return 0;
}
