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
// Rows move global -> shared by one cp.async.bulk each (two producer warps
// taking alternate blocks, a 5-stage ring of 32-row blocks on mbarriers), then
// twelve converter warps widen them: per row, lane l converts latent values 16l .. 16l+15 (two 16-byte
// stores) and lanes 0..7 store the 128-byte tail (pe_dim 64) or zeros (pe_dim 0:
// the tail is not read). An absent slot (<= 0) gives a row of zeros; a slot >=
// num_slots also sets MLA_ERR_GATHER_INDEX_RANGE.
#include <cfloat>

#include "mla_device.cuh"

namespace {

using namespace mla;

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

constexpr int kUStages = 5;
constexpr int kUNB = 32;                              // rows per block
constexpr int kUWarps = 12;                           // converter warps (rows w, w + 12, w + 24 of a block)
constexpr int kUProducers = 2;                        // copy-issuing warps (alternate blocks)
constexpr int kUThreads = (kUWarps + kUProducers) * 32;
constexpr int kUStageBytes = kUNB * kRowBytes;
constexpr int kUSmem = kUStages * kUStageBytes + kUStages * kUNB * 4 + 2 * kUStages * 8;
constexpr int kUCtasPerSm = 2;

// Persistent: CTA c takes blocks c, c + grid, ... of 32 consecutive output rows.
// The last two warps (producers, alternate blocks) copy each present row global
// -> shared with one cp.async.bulk into a 5-stage ring and record the block's
// slots; converter
// warp w widens rows w, w + 12, w + 24 of the block from shared memory.
// Two products rounded to BF16 by the hardware conversion (round to nearest even
// of the fp32 product). That is the nearest BF16 of the exact product unless the
// fp32 product sits on a BF16 midpoint, is NaN, or is nonzero below 2^-100. The
// last two are ruled out per row (row_needs_exact); midpoints are tracked below,
// and a row slice with any of them is redone by product_to_bf16.
// The two products come from one packed fp32 multiply (the same IEEE product per
// value); their low 16 bits, each XORed with 0x8000, go into a running unsigned
// 16x2 minimum, which ends with a zero half exactly when some product sat on a
// BF16 midpoint (midpoint_seen).
__device__ __forceinline__ uint32_t pair_to_bf16x2(float v0, float v1, uint64_t s2, uint32_t& lows_min) {
    uint64_t v2, p2;
    asm("mov.b64 %0, {%1, %2};" : "=l"(v2) : "f"(v0), "f"(v1));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(p2) : "l"(v2), "l"(s2));
    float p0, p1;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(p0), "=f"(p1) : "l"(p2));
    const uint32_t lows = __byte_perm(__float_as_uint(p0), __float_as_uint(p1), 0x5410) ^ 0x80008000u;
    asm("min.u16x2 %0, %1, %2;" : "=r"(lows_min) : "r"(lows_min), "r"(lows));
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(p1), "f"(p0));   // high half <- p1
    return r;
}

__device__ __forceinline__ bool midpoint_seen(uint32_t lows_min) {
    return (lows_min & 0xFFFFu) == 0u || (lows_min >> 16) == 0u;
}

// Whether a lane's 16 codes with tile scale s can give a product that the
// hardware conversion does not round as required: s outside [2^-80, FLT_MAX]
// (NaN, infinite, negative, zero or tiny: with s >= 2^-80 a nonzero E4M3 value,
// at least 2^-9 in magnitude, gives a product of at least 2^-89), or a NaN code
// (S.1111.111: the low seven bits of a byte all set).
__device__ __forceinline__ bool row_needs_exact(const uint4& codes, float s) {
    const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
    uint32_t nan = 0u;
#pragma unroll
    for (int q = 0; q < 4; ++q) nan |= ((w[q] & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
    return nan != 0u || !(s >= 0x1p-80f && s <= FLT_MAX);
}

__global__ void __launch_bounds__(kUThreads, kUCtasPerSm)
mla_gather_upconvert_kernel(const uint8_t* __restrict__ cache, int64_t num_slots, int64_t row_bytes,
                            const int32_t* __restrict__ slots, int64_t n, int pe_dim,
                            uint16_t* __restrict__ out, int* __restrict__ err) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* stages = smem;
    int* slot_s = reinterpret_cast<int*>(smem + kUStages * kUStageBytes);      // [stage][row]
    uint64_t* full = reinterpret_cast<uint64_t*>(slot_s + kUStages * kUNB);
    uint64_t* empty = full + kUStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nblk = (n + kUNB - 1) / kUNB;
    const uint32_t row_read = (pe_dim == kRope) ? kRowBytes : kNopeReadBytes;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kUStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kUWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp >= kUWarps) {
        // ---- producers: warp kUWarps + p issues the CTA's blocks p, p + 2, ... ----
        const int pw = warp - kUWarps;
        const int64_t step = static_cast<int64_t>(kUProducers) * gridDim.x;
        int64_t blk = blockIdx.x + static_cast<int64_t>(pw) * gridDim.x;
        int64_t r = blk * kUNB + lane;
        int next_slot = (blk < nblk && r < n) ? __ldg(slots + r) : 0;
        for (int k = pw; blk < nblk; k += kUProducers, blk += step) {
            const int slot = next_slot;
            const int64_t rn = (blk + step) * kUNB + lane;            // this warp's next block, early
            next_slot = (blk + step < nblk && rn < n) ? __ldg(slots + rn) : 0;
            const int s = k % kUStages;
            if (k >= kUStages && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>(((k / kUStages) - 1) & 1))) {
                // Record it, let the copies already issued land (bounded), and
                // leave; the converters' own waits run out on the next block.
                if (lane == 0) {
                    atomicOr(err, MLA_ERR_PIPELINE_TIMEOUT);
                    for (int kk = k - kUProducers; kk >= 0 && kk >= k - kUStages; kk -= kUProducers)
                        (void)mbar_wait_bounded(&full[kk % kUStages], static_cast<uint32_t>((kk / kUStages) & 1));
                }
                return;
            }
            const bool in_range = blk * kUNB + lane < n;
            const bool present = in_range && slot > 0 && slot < num_slots;
            if (in_range && slot >= num_slots) atomicOr(err, MLA_ERR_GATHER_INDEX_RANGE);
            slot_s[s * kUNB + lane] = present ? slot : (in_range ? 0 : -1);   // -1: past the end
            const unsigned m = __ballot_sync(0xffffffffu, present);
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(__popc(m)) * row_read);
            __syncwarp();
            if (present)
                bulk_g2s(stages + s * kUStageBytes + lane * kRowBytes, cache + static_cast<int64_t>(slot) * row_bytes,
                         row_read, &full[s]);
        }
        return;
    }

    // ---- converters ----
    int64_t blk = blockIdx.x;
    for (int k = 0; blk < nblk; ++k, blk += gridDim.x) {
        const int s = k % kUStages;
        if (!mbar_wait_bounded(&full[s], static_cast<uint32_t>((k / kUStages) & 1))) {
            if (lane == 0) atomicOr(err, MLA_ERR_PIPELINE_TIMEOUT);
            return;
        }
        const uint8_t* st = stages + s * kUStageBytes;
        for (int rr = warp; rr < kUNB; rr += kUWarps) {
            const int slot = slot_s[s * kUNB + rr];
            if (slot < 0) break;                                      // past the end of the output
            uint16_t* orow = out + (blk * kUNB + rr) * kOutWidth;
            if (slot == 0) {                                          // absent: a row of zeros
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                st_v4(orow + 16 * lane, z);
                st_v4(orow + 16 * lane + 8, z);
                if (lane < 8) st_v4(orow + kLatent + 8 * lane, z);
                continue;
            }
            const uint8_t* row = st + rr * kRowBytes;
            const uint4 codes = *reinterpret_cast<const uint4*>(row + 16 * lane);
            const float sc = *reinterpret_cast<const float*>(row + kScaleOff + 4 * (lane >> 3));
            uint4 tail = make_uint4(0u, 0u, 0u, 0u);
            if (pe_dim == kRope && lane < 8) tail = *reinterpret_cast<const uint4*>(row + kTailOff + 16 * lane);
            const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
            float v[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t h01, h23;
                e4m3x4_to_f16x2x2(w[q], h01, h23);  // exact
                v[4 * q + 0] = __half2float(__ushort_as_half(static_cast<unsigned short>(h01 & 0xFFFFu)));
                v[4 * q + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(h01 >> 16)));
                v[4 * q + 2] = __half2float(__ushort_as_half(static_cast<unsigned short>(h23 & 0xFFFFu)));
                v[4 * q + 3] = __half2float(__ushort_as_half(static_cast<unsigned short>(h23 >> 16)));
            }
            uint32_t o[8];
            uint64_t s2;
            asm("mov.b64 %0, {%1, %1};" : "=l"(s2) : "f"(sc));
            uint32_t lows_min = 0xFFFFFFFFu;
#pragma unroll
            for (int q = 0; q < 8; ++q) o[q] = pair_to_bf16x2(v[2 * q], v[2 * q + 1], s2, lows_min);
            if (row_needs_exact(codes, sc) || midpoint_seen(lows_min)) {   // rare
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    o[q] = product_to_bf16(v[2 * q], sc) | (product_to_bf16(v[2 * q + 1], sc) << 16);
            }
            st_v4(orow + 16 * lane, make_uint4(o[0], o[1], o[2], o[3]));
            st_v4(orow + 16 * lane + 8, make_uint4(o[4], o[5], o[6], o[7]));
            if (lane < 8) st_v4(orow + kLatent + 8 * lane, tail);
        }
        // The stage is next written by the async proxy (cp.async.bulk): order this
        // warp's generic reads of it before that write.
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
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
    if (!mla_host::max_dynamic_smem(reinterpret_cast<const void*>(mla_gather_upconvert_kernel), kUSmem))
        return MLA_ECUDA;
    const int64_t nblk = (n + kUNB - 1) / kUNB;
    int64_t grid = static_cast<int64_t>(sms) * kUCtasPerSm;
    if (grid > nblk) grid = nblk;
    mla_gather_upconvert_kernel<<<static_cast<unsigned>(grid), kUThreads, kUSmem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(kv.data), kv.num_slots, kv.row_bytes, slots, n, pe_dim,
        static_cast<uint16_t*>(out_bf16), err);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ECUDA;
}
