// mla_gather_upconvert: gather rows of the packed FP8 cache and widen them to
// BF16 [n, 576] (vLLM PR #55277, Changes table: cp_gather_and_upconvert_fp8_
// kv_cache for the chunked-context path; the NoPE tail is written as zeros).
//
// Each latent value is the BF16 nearest to the exact product e4m3(byte) * scale
// (ties to even). Rounding the fp32 product p = RN(v * s) to BF16 gives that
// value except when p falls exactly on a BF16 midpoint while v * s does not; the
// FMA residual e = v * s - p (exact for |p| >= 2^-100) then says which way to
// go. Products below 2^-100 are formed in double and rounded once. A NaN code
// gives 0x7FC0.
//
// One warp per row: lane l converts latent values 16l .. 16l+15 (one 16-byte
// load, two 16-byte stores); lanes 0..7 copy the 128-byte tail (pe_dim 64) or
// write zeros (pe_dim 0: the tail is not read). An absent slot (<= 0) gives a
// row of zeros; a slot >= num_slots also sets MLA_ERR_GATHER_INDEX_RANGE.
#include "mla_device.cuh"

namespace {

using namespace mla;

constexpr int kThreads = 256;   // 8 rows in flight per CTA
constexpr int kOutWidth = kLatent + kRope;   // 576

__device__ __forceinline__ uint32_t product_to_bf16(float v, float s) {
    const float p = __fmul_rn(v, s);
    if (isnan(p)) return 0x7FC0u;
    const uint32_t u = __float_as_uint(p);
    if (fabsf(p) < 0x1p-100f) {
        // Small products (rare): the exact product in double (4 + 24 bits),
        // rounded to 8 significant bits with the exponent held at >= -126 (the
        // BF16 subnormal quantum is 2^-133), then the exact fp32 of the result.
        const double x = static_cast<double>(v) * static_cast<double>(s);
        if (x == 0.0) return u >> 16;           // +-0 keeps its sign
        const int q = max(ilogb(x), -126) - 7;
        const double r = ldexp(rint(ldexp(x, -q)), q);
        return __float_as_uint(static_cast<float>(r)) >> 16;
    }
    const uint32_t lo = u & 0xFFFFu;
    uint32_t hi = u >> 16;
    if (lo > 0x8000u) {
        ++hi;                                   // away from zero (sign-magnitude bits)
    } else if (lo == 0x8000u) {
        const float e = __fmaf_rn(v, s, -p);    // exact residual (|p| >= 2^-100)
        if (e == 0.0f) hi += (hi & 1u);         // a true tie: to even
        else if ((e > 0.0f) == (p > 0.0f)) ++hi;   // the product lies past the midpoint
    }
    return hi;
}

__global__ void __launch_bounds__(kThreads)
mla_gather_upconvert_kernel(const uint8_t* __restrict__ cache, int64_t num_slots, int64_t row_bytes,
                            const int32_t* __restrict__ slots, int64_t n, int pe_dim,
                            uint16_t* __restrict__ out, int* __restrict__ err) {
    const int lane = threadIdx.x & 31;
    const int64_t stride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < n; r += stride) {
        const int64_t slot = __ldg(slots + r);
        uint16_t* orow = out + r * kOutWidth;
        if (slot <= 0 || slot >= num_slots) {
            if (slot >= num_slots && lane == 0) atomicOr(err, MLA_ERR_GATHER_INDEX_RANGE);
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            st_v4(orow + 16 * lane, z);
            st_v4(orow + 16 * lane + 8, z);
            if (lane < 8) st_v4(orow + kLatent + 8 * lane, z);
            continue;
        }
        const uint8_t* row = cache + slot * row_bytes;
        const uint4 codes = ld_nc_v4(row + 16 * lane);
        const float s = __uint_as_float(__ldg(reinterpret_cast<const uint32_t*>(row + kScaleOff) + (lane >> 3)));
        uint4 tail = make_uint4(0u, 0u, 0u, 0u);
        if (pe_dim == kRope && lane < 8) tail = ld_nc_v4(row + kTailOff + 16 * lane);
        const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t h01, h23;
            e4m3x4_to_f16x2x2(w[i], h01, h23);  // exact
            const float v0 = __half2float(__ushort_as_half(static_cast<unsigned short>(h01 & 0xFFFFu)));
            const float v1 = __half2float(__ushort_as_half(static_cast<unsigned short>(h01 >> 16)));
            const float v2 = __half2float(__ushort_as_half(static_cast<unsigned short>(h23 & 0xFFFFu)));
            const float v3 = __half2float(__ushort_as_half(static_cast<unsigned short>(h23 >> 16)));
            o[2 * i] = product_to_bf16(v0, s) | (product_to_bf16(v1, s) << 16);
            o[2 * i + 1] = product_to_bf16(v2, s) | (product_to_bf16(v3, s) << 16);
        }
        st_v4(orow + 16 * lane, make_uint4(o[0], o[1], o[2], o[3]));
        st_v4(orow + 16 * lane + 8, make_uint4(o[4], o[5], o[6], o[7]));
        if (lane < 8) st_v4(orow + kLatent + 8 * lane, tail);
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int mla_gather_upconvert(mla_kv_cache_t kv, const int32_t* slots, int64_t n, int pe_dim,
                                    void* out_bf16, void* stream) {
    if (n < 0 || kv.num_slots < 0 || (pe_dim != 0 && pe_dim != MLA_ROPE_DIM)) return MLA_EINVAL;
    if (kv.row_bytes != MLA_ROW_BYTES && !(kv.row_bytes == MLA_ROW_BYTES_NOPE && pe_dim == 0)) return MLA_EINVAL;
    if (n == 0) return MLA_OK;
    if (kv.data == nullptr || slots == nullptr || out_bf16 == nullptr) return MLA_EINVAL;
    if (!aligned16(kv.data) || !aligned16(out_bf16) || (reinterpret_cast<uintptr_t>(slots) & 3u)) return MLA_EINVAL;
    int* err = mla_host::device_error_word();
    const int sms = mla_host::sm_count();
    if (err == nullptr || sms <= 0) return MLA_ECUDA;
    const int64_t rows_per_cta = kThreads / 32;
    int64_t blocks = (n + rows_per_cta - 1) / rows_per_cta;
    const int64_t max_blocks = static_cast<int64_t>(sms) * 8;
    if (blocks > max_blocks) blocks = max_blocks;
    mla_gather_upconvert_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(kv.data), kv.num_slots, kv.row_bytes, slots, n, pe_dim,
        static_cast<uint16_t*>(out_bf16), err);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ECUDA;
}
