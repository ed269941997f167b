// mla_sparse_decode: sparse top-k MLA decode over the packed FP8 cache, on the
// sm_100-family tensor cores (tcgen05 + tensor memory + TMA gathers).
//
// What it computes follows the decode statement in the C header, with the
// masking rule of sglang PR #39288 (Root cause: a -1 candidate must add nothing
// and must not gather slot 0) and sglang PR #47013 (Motivation: masking only the
// score does not stop a NaN row). Here an absent entry is removed before
// anything is fetched: each CTA compacts its slice of the top-k list in shared
// memory, so -1, slot 0 and out-of-range indices are never dereferenced.
//
// One CTA per (token, split of the top-k list, group of 16 heads); 6 warps:
//   warp 0     producer: TMA tile::gather4 of 128 present rows per block into a
//              2-stage ring. The four 128-byte latent tiles and the RoPE tail land
//              in 128-byte-swizzled UMMA layouts (8-row atoms), the 16-byte scale
//              groups in a plain array. Rows past the end of the list get an
//              out-of-range row coordinate, which TMA fills with zeros without
//              reading memory.
//   warp 1     MMA issuer (one thread) and tensor-memory owner.
//   warps 2-5  compute, thread j <-> row j of the block <-> tensor-memory lane j.
// Per 128-row block:
//   dequant  each compute thread converts its row's 512 E4M3 codes to f16
//            (exact) and stores them into tensor memory: the A operand of QK.
//   QK       S^T[j, h] = sum_t scale[j, t] * (E_t[j] . q_t[h]) + rope[j] . qr[h]:
//            f16 MMAs (M = 128 rows, N = 16 heads, A from tensor memory) into four
//            per-tile fp32 accumulators plus a bf16 MMA for the RoPE part, so every
//            product is exact before fp32 accumulation and the fp32 tile scales are
//            applied per row afterwards.
//   softmax  online, per head, in log2 units; the exp2 offset moves only when a
//            score exceeds it by more than 2^8.
//   PV       O^T[d, h] += sum_j E[j, d] * P~_t[j, h], P~_t = p * scale[j, t] /
//            sigma_t * 1.75 in [0, 448] split into two E4M3 terms (hi + lo, about
//            2^-8 relative); kind::f8f6f4 MMAs read V^T straight from the gathered
//            E4M3 tiles (MN-major) and accumulate O^T in tensor memory.
// Splits write a normalised partial (o, lse) to the caller's workspace; a second
// kernel merges them in split order (deterministic: no float atomics).
#include <cfloat>
#include <cmath>
#include <cstring>
#include <mutex>

#include "mla_device.cuh"
#include "mla_tcgen05.cuh"

namespace {

using namespace mla;
namespace tc = mla::tc;

constexpr int kBM = 128;               // rows per block: M of QK, K of PV
constexpr int kHG = 16;                // heads per CTA: N of both MMAs
constexpr int kListMax = 1024;         // top-k positions one CTA compacts
constexpr int kThreads = 192;
constexpr int kWarpsAll = kThreads / 32;
constexpr int kComputeThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleSlack = 8.0f;  // log2 units: p <= 2^8
constexpr float kPScale = 1.75f;       // maps [0, 256] onto [0, 448]

// Shared memory, offsets from a 1024-byte aligned base.
constexpr uint32_t kLatBytes = 4 * 16 * 1024;        // 4 tiles x 16 atoms of 8 rows x 128 B
constexpr uint32_t kRopeBytes = 16 * 1024;           // 16 atoms of 8 rows x 64 bf16
constexpr uint32_t kScaleBytes = 32 * 128;           // 32 groups of 4 rows x 16 B
constexpr uint32_t kStageBytes = kLatBytes + kRopeBytes + kScaleBytes;   // 86,016
constexpr uint32_t kOffQ = 2 * kStageBytes;          // f16 q latent, K-major 128-B swizzle
constexpr uint32_t kOffQR = kOffQ + 16384;           // bf16 q RoPE
constexpr uint32_t kOffP = kOffQR + 2048;            // 2 x P~ [tile][term][16 core matrices of 128 B]
constexpr uint32_t kPBytes = 4 * 2 * 16 * 128;
constexpr uint32_t kOffList = kOffP + 2 * kPBytes;
constexpr uint32_t kOffRed = kOffList + kListMax * 4;   // [4 warps][32] floats
constexpr uint32_t kOffBar = kOffRed + 512;
constexpr uint32_t kSmemUsed = kOffBar + 192;
constexpr uint32_t kSmemAlloc = kSmemUsed + 1024;    // slack to align the base to 1024 B

// Tensor-memory columns (one CTA per SM allocates all 512).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColA = 0;     // 256: f16 latent rows of the block
constexpr uint32_t kColS = 256;   // 80: S^T per tile (4 x 16) + RoPE (16)
constexpr uint32_t kColO = 336;   // 64: O^T per tile (4 x 16)

struct DecodeArgs {
    const __nv_bfloat16* q;
    const int32_t* topk;
    __nv_bfloat16* out;
    float* lse;
    float* ws_o;      // [T, nsplit, H, 512] (nsplit > 1)
    float* ws_lse;    // [T, nsplit, H]
    int* err;
    int64_t num_slots;
    int oob_row;      // a row coordinate past the tensor map (zero fill)
    int T, H, d_qk, W, nsplit, split_len;
    float sm_scale_log2;   // sm_scale * log2(e)
};

// Bounded wait that also gives up when another role has already given up.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitCycles) {
            *abort_flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Two E4M3 codes of (x0, x1): low byte = x0. Round to nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x2(float x0, float x1) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3));
}
// hi + lo E4M3 split of a pair: hi = e4m3(x), lo = e4m3(x - hi).
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    hi = e4m3x2(x0, x1);
    uint32_t hf, unused;
    e4m3x4_to_f16x2x2(hi, hf, unused);
    const float2 hv = __half22float2(*reinterpret_cast<const __half2*>(&hf));
    lo = e4m3x2(x0 - hv.x, x1 - hv.y);
}

template <bool kRopeOn>
__global__ void __launch_bounds__(kThreads, 1)
mla_sparse_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_row, const __grid_constant__ CUtensorMap tm_scale,
                            const DecodeArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* full = bars;          // [2] stage landed (TMA bytes)
    uint64_t* empty = bars + 2;     // [2] PV of the stage's block complete
    uint64_t* a_ready = bars + 4;   // dequant written to tensor memory (4 warps)
    uint64_t* s_full = bars + 5;    // QK complete
    uint64_t* p_ready = bars + 6;   // [2] P~ written (4 warps)
    uint64_t* drain = bars + 8;     // all MMAs complete (end of kernel)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 9);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* issued_s = reinterpret_cast<int*>(tmem_slot + 2);
    int* wcount = reinterpret_cast<int*>(tmem_slot + 3);          // [6]
    int* list = reinterpret_cast<int*>(smem + kOffList);
    float* red = reinterpret_cast<float*>(smem + kOffRed);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x;
    const int split = blockIdx.y;
    const int hg = blockIdx.z;
    const int H = args.H;

    if (threadIdx.x == 0) {
        mbar_init(&full[0], 1); mbar_init(&full[1], 1);
        mbar_init(&empty[0], 1); mbar_init(&empty[1], 1);
        mbar_init(a_ready, 4); mbar_init(s_full, 1);
        mbar_init(&p_ready[0], 4); mbar_init(&p_ready[1], 4);
        mbar_init(drain, 1);
        *abort_flag = 0;
        *issued_s = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
        tc::fence_before_sync();
    }

    // ---- compact the present entries of this split's positions (all warps) ----
    const int p0 = split * args.split_len;
    const int p1 = min(args.W, p0 + args.split_len);
    const int32_t* trow = args.topk + static_cast<int64_t>(t) * args.W;
    int n_valid = 0;
    for (int base = p0; base < p1; base += kThreads) {
        const int pos = base + threadIdx.x;
        const int idx = (pos < p1) ? __ldg(trow + pos) : -1;
        const bool valid = idx > 0 && static_cast<int64_t>(idx) < args.num_slots;
        if (idx > 0 && !valid) atomicOr(args.err, MLA_ERR_DECODE_INDEX_RANGE);
        const unsigned m = __ballot_sync(0xffffffffu, valid);
        if (lane == 0) wcount[warp] = __popc(m);
        __syncthreads();
        int off = n_valid, total = 0;
#pragma unroll
        for (int w = 0; w < kWarpsAll; ++w) {
            const int cw = wcount[w];
            off += (w < warp) ? cw : 0;
            total += cw;
        }
        if (valid) list[off + __popc(m & ((1u << lane) - 1u))] = idx;
        n_valid += total;
        __syncthreads();
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int nblk = (n_valid + kBM - 1) / kBM;

    if (warp == 0) {
        // ================= producer =================
        int b = 0;
        for (; b < nblk; ++b) {
            const int s = b & 1;
            if (b >= 2 && !wait_or_abort(&empty[s], static_cast<uint32_t>(((b >> 1) - 1) & 1), abort_flag)) break;
            uint8_t* st = smem + s * kStageBytes;
            if (lane == 0) mbar_arrive_expect_tx(&full[s], kBM * ((kRopeOn ? 640u : 512u) + 16u));
            __syncwarp();
            // lane g gathers rows 4g .. 4g+3 of the block: half an 8-row atom
            const int r0 = b * kBM + 4 * lane;
            int y[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) y[i] = (r0 + i < n_valid) ? list[r0 + i] : args.oob_row;
            uint8_t* dst = st + (lane >> 1) * 1024 + (lane & 1) * 512;
#pragma unroll
            for (int tt = 0; tt < 4; ++tt)
                tc::tma_gather4(dst + tt * 16384, &tm_row, 128 * tt, y[0], y[1], y[2], y[3], &full[s]);
            if (kRopeOn)
                tc::tma_gather4(dst + kLatBytes, &tm_row, kTailOff, y[0], y[1], y[2], y[3], &full[s]);
            tc::tma_gather4(st + kLatBytes + kRopeBytes + lane * 128, &tm_scale, kScaleOff, y[0], y[1], y[2], y[3],
                            &full[s]);
        }
        if (lane == 0) *issued_s = b;
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t id_qk = tc::instr_desc(tc::kF16, tc::kF16, false, false, 128, kHG);
            constexpr uint32_t id_qr = tc::instr_desc(tc::kBF16, tc::kBF16, false, false, 128, kHG);
            constexpr uint32_t id_pv = tc::instr_desc(tc::kE4M3, tc::kE4M3, true, true, 128, kHG);
            for (int b = 0; b < nblk; ++b) {
                const int s = b & 1;
                if (!wait_or_abort(a_ready, static_cast<uint32_t>(b & 1), abort_flag)) break;
                tc::fence_after_sync();
                // QK^T latent: A = f16 rows in tensor memory, B = q (K-major, 128-B swizzle)
#pragma unroll 4
                for (int ks = 0; ks < 32; ++ks) {
                    const uint64_t bd = tc::smem_desc(sbase + kOffQ + (ks >> 2) * 2048 + (ks & 3) * 32, 16, 1024, tc::kSw128);
                    tc::mma_f16_ts(tmem + kColS + 16 * (ks >> 3), tmem + kColA + 8 * ks, bd, id_qk,
                                   (ks & 7) != 0 ? 1u : 0u);
                }
                if (kRopeOn) {
                    const uint32_t rb = sbase + s * kStageBytes + kLatBytes;
#pragma unroll
                    for (int kr = 0; kr < 4; ++kr) {
                        const uint64_t ad = tc::smem_desc(rb + kr * 32, 16, 1024, tc::kSw128);
                        const uint64_t bd = tc::smem_desc(sbase + kOffQR + kr * 32, 16, 1024, tc::kSw128);
                        tc::mma_f16_ss(tmem + kColS + 64, ad, bd, id_qr, kr != 0 ? 1u : 0u);
                    }
                }
                tc::commit(s_full);
                if (!wait_or_abort(&p_ready[b & 1], static_cast<uint32_t>((b >> 1) & 1), abort_flag)) break;
                tc::fence_after_sync();
                // PV: A = V^T (E4M3, MN-major, the gathered tiles), B = P~ (E4M3, MN-major)
                const uint32_t lat = sbase + s * kStageBytes;
                const uint32_t pb = sbase + kOffP + (b & 1) * kPBytes;
#pragma unroll
                for (int tt = 0; tt < 4; ++tt) {
#pragma unroll
                    for (int term = 0; term < 2; ++term) {
#pragma unroll
                        for (int ke = 0; ke < 4; ++ke) {
                            const uint64_t ad = tc::smem_desc(lat + tt * 16384 + ke * 4096, 16384, 1024, tc::kSw128);
                            const uint64_t bd = tc::smem_desc(pb + (tt * 2 + term) * 2048 + ke * 512, 128, 2048, tc::kSwNone);
                            tc::mma_f8_ss(tmem + kColO + 16 * tt, ad, bd, id_pv, (b | term | ke) != 0 ? 1u : 0u);
                        }
                    }
                }
                tc::commit(&empty[s]);
            }
            // Let every MMA this thread issued finish before the CTA tears down.
            tc::commit(drain);
            (void)mbar_wait_bounded(drain, 0);
        }
        __syncwarp();
    } else {
        // ================= compute warps =================
        const int qd = warp & 3;                     // tensor-memory lane quarter of this warp
        const int j = 32 * qd + lane;                // row of the block / tensor-memory lane
        const int ct = threadIdx.x - 64;             // 0 .. 127
        const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
        const int64_t qrow0 = static_cast<int64_t>(t) * H + hg * kHG;

        // ---- q: per-head exponent shift into f16 range, then the UMMA layouts ----
        {
            const int h = ct >> 3, part = ct & 7;
            float mx = 0.0f;
            if (hg * kHG + h < H) {
                const __nv_bfloat16* qh = args.q + (qrow0 + h) * args.d_qk;
                const uint8_t* pl = reinterpret_cast<const uint8_t*>(qh + 64 * part);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint4 v = ld_nc_v4(pl + 16 * k);
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) mx = fmaxf(mx, fmaxf(fabsf(bf16lo(wv[i])), fabsf(bf16hi(wv[i]))));
                }
                if (kRopeOn) {
                    const uint4 v = ld_nc_v4(qh + kLatent + 8 * part);
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) mx = fmaxf(mx, fmaxf(fabsf(bf16lo(wv[i])), fabsf(bf16hi(wv[i]))));
                }
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            if (part == 0) red[h] = mx;
        }
        bar_sync_or(1, kComputeThreads, false);
        float rowf[kHG];
#pragma unroll
        for (int h = 0; h < kHG; ++h) {
            int e = 0;
            frexpf(red[h], &e);                              // max|q_h| < 2^e
            rowf[h] = args.sm_scale_log2 * ldexpf(1.0f, (e > 15) ? (e - 15) : 0);
        }
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int k = ct + kComputeThreads * it;         // 16 heads x 64 chunks of 8 dims
            const int h = k >> 6, cc = k & 63;
            int e = 0;
            frexpf(red[h], &e);
            const float down = ldexpf(1.0f, (e > 15) ? (15 - e) : 0);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (hg * kHG + h < H) v = ld_nc_v4(args.q + (qrow0 + h) * args.d_qk + 8 * cc);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
            uint4 o;
            o.x = pack_f16x2(bf16lo(wv[0]) * down, bf16hi(wv[0]) * down);
            o.y = pack_f16x2(bf16lo(wv[1]) * down, bf16hi(wv[1]) * down);
            o.z = pack_f16x2(bf16lo(wv[2]) * down, bf16hi(wv[2]) * down);
            o.w = pack_f16x2(bf16lo(wv[3]) * down, bf16hi(wv[3]) * down);
            const int c64 = cc >> 3, u = cc & 7, r = h & 7;
            *reinterpret_cast<uint4*>(smem + kOffQ + (c64 * 2 + (h >> 3)) * 1024 + r * 128 + ((u ^ r) << 4)) = o;
        }
        if (kRopeOn) {
            const int h = ct >> 3, u = ct & 7, r = h & 7;
            int e = 0;
            frexpf(red[h], &e);
            const float down = ldexpf(1.0f, (e > 15) ? (15 - e) : 0);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (hg * kHG + h < H) v = ld_nc_v4(args.q + (qrow0 + h) * args.d_qk + kLatent + 8 * u);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
            uint4 o;
            o.x = pack_bf16x2(bf16lo(wv[0]) * down, bf16hi(wv[0]) * down);
            o.y = pack_bf16x2(bf16lo(wv[1]) * down, bf16hi(wv[1]) * down);
            o.z = pack_bf16x2(bf16lo(wv[2]) * down, bf16hi(wv[2]) * down);
            o.w = pack_bf16x2(bf16lo(wv[3]) * down, bf16hi(wv[3]) * down);
            *reinterpret_cast<uint4*>(smem + kOffQR + (h >> 3) * 1024 + r * 128 + ((u ^ r) << 4)) = o;
        }
        fence_proxy_async_smem();
        bar_sync_or(1, kComputeThreads, false);      // red[] reads done before its reuse

        float m_ref[kHG], l_part[kHG];
#pragma unroll
        for (int h = 0; h < kHG; ++h) { m_ref[h] = -INFINITY; l_part[h] = 0.0f; }
        float sigma[4] = {FLT_MIN, FLT_MIN, FLT_MIN, FLT_MIN};
        float inv_sigma[4] = {1.0f / FLT_MIN, 1.0f / FLT_MIN, 1.0f / FLT_MIN, 1.0f / FLT_MIN};
        bool ok = true;

        for (int b = 0; b < nblk; ++b) {
            const int s = b & 1;
            const uint8_t* st = smem + s * kStageBytes;
            // ---- dequant: this row's E4M3 codes -> f16 -> tensor memory ----
            // Every failure decision is voted across the four warps, so they always
            // take the same path through the named barrier.
            bool okl = wait_or_abort(&full[s], static_cast<uint32_t>((b >> 1) & 1), abort_flag);
            if (bar_sync_or(1, kComputeThreads, !okl)) { ok = false; break; }
            {
                const uint8_t* rowp = st + (j >> 3) * 1024 + (j & 7) * 128;
                const int r = j & 7;
#pragma unroll
                for (int tt = 0; tt < 4; ++tt) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {          // 16 columns = 32 dims = 2 chunks
                        uint32_t w[16];
#pragma unroll
                        for (int uu = 0; uu < 2; ++uu) {
                            const int u = 2 * q4 + uu;
                            const uint4 v = *reinterpret_cast<const uint4*>(rowp + tt * 16384 + ((u ^ r) << 4));
                            e4m3x4_to_f16x2x2(v.x, w[8 * uu + 0], w[8 * uu + 1]);
                            e4m3x4_to_f16x2x2(v.y, w[8 * uu + 2], w[8 * uu + 3]);
                            e4m3x4_to_f16x2x2(v.z, w[8 * uu + 4], w[8 * uu + 5]);
                            e4m3x4_to_f16x2x2(v.w, w[8 * uu + 6], w[8 * uu + 7]);
                        }
                        tc::tmem_st16(tmem + lane_base + kColA + 64 * tt + 16 * q4, w);
                    }
                }
            }
            tc::wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_ready);

            // ---- softmax ----
            okl = wait_or_abort(s_full, static_cast<uint32_t>(b & 1), abort_flag);
            if (bar_sync_or(1, kComputeThreads, !okl)) { ok = false; break; }
            tc::fence_after_sync();
            const float4 scv = *reinterpret_cast<const float4*>(st + kLatBytes + kRopeBytes + (j >> 2) * 128 + (j & 3) * 16);
            const float sc[4] = {scv.x, scv.y, scv.z, scv.w};
            float sv[kHG];
            {
                uint32_t acc[16];
#pragma unroll
                for (int h = 0; h < kHG; ++h) sv[h] = 0.0f;
                if (kRopeOn) {
                    tc::tmem_ld16(tmem + lane_base + kColS + 64, acc);
                    tc::wait_ld();
#pragma unroll
                    for (int h = 0; h < kHG; ++h) sv[h] = __uint_as_float(acc[h]);
                }
#pragma unroll
                for (int tt = 0; tt < 4; ++tt) {
                    tc::tmem_ld16(tmem + lane_base + kColS + 16 * tt, acc);
                    tc::wait_ld();
#pragma unroll
                    for (int h = 0; h < kHG; ++h) sv[h] = fmaf(sc[tt], __uint_as_float(acc[h]), sv[h]);
                }
            }
            const bool present = b * kBM + j < n_valid;
            bool need = false;
#pragma unroll
            for (int h = 0; h < kHG; ++h) {
                sv[h] = present ? sv[h] * rowf[h] : -INFINITY;
                need |= sv[h] > m_ref[h] + kRescaleSlack;
            }
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) need |= sc[tt] > sigma[tt];
            tc::fence_before_sync();
            if (bar_sync_or(1, kComputeThreads, need)) {
                // Rare after the first blocks: new per-head offsets and per-tile sigma.
                float* rw = red + qd * 32;
#pragma unroll
                for (int h = 0; h < kHG; ++h) {
                    const float mh = warp_max(sv[h]);
                    if (lane == 0) rw[h] = mh;
                }
#pragma unroll
                for (int tt = 0; tt < 4; ++tt) {
                    const float sm = warp_max(sc[tt]);
                    if (lane == 0) rw[16 + tt] = sm;
                }
                bar_sync_or(1, kComputeThreads, false);
                float alpha[kHG], rs[4];
#pragma unroll
                for (int h = 0; h < kHG; ++h) {
                    const float bm = fmaxf(fmaxf(red[h], red[32 + h]), fmaxf(red[64 + h], red[96 + h]));
                    const float mn = (bm > m_ref[h] + kRescaleSlack) ? bm : m_ref[h];
                    alpha[h] = ex2_approx(m_ref[h] - mn);     // -inf -> 0
                    m_ref[h] = mn;
                    l_part[h] *= alpha[h];
                }
#pragma unroll
                for (int tt = 0; tt < 4; ++tt) {
                    const float bs = fmaxf(fmaxf(red[16 + tt], red[48 + tt]), fmaxf(red[80 + tt], red[112 + tt]));
                    const float sn = fmaxf(sigma[tt], bs);
                    rs[tt] = sigma[tt] / sn;
                    sigma[tt] = sn;
                    inv_sigma[tt] = 1.0f / sn;
                }
                if (b > 0) {
                    // O^T is rescaled in tensor memory once PV of the previous block is done.
                    okl = wait_or_abort(&empty[(b - 1) & 1], static_cast<uint32_t>(((b - 1) >> 1) & 1), abort_flag);
                    if (bar_sync_or(1, kComputeThreads, !okl)) {
                        ok = false;
                    } else {
                        tc::fence_after_sync();
#pragma unroll
                        for (int tt = 0; tt < 4; ++tt) {
                            uint32_t ov[16];
                            tc::tmem_ld16(tmem + lane_base + kColO + 16 * tt, ov);
                            tc::wait_ld();
#pragma unroll
                            for (int h = 0; h < kHG; ++h)
                                ov[h] = __float_as_uint(__uint_as_float(ov[h]) * (alpha[h] * rs[tt]));
                            tc::tmem_st16(tmem + lane_base + kColO + 16 * tt, ov);
                        }
                        tc::wait_st();
                    }
                }
                bar_sync_or(1, kComputeThreads, false);   // red[] free again
                if (!ok) break;
            }
            // ---- P~ = p * scale / sigma * 1.75 as E4M3 hi + lo, MN-major core matrices ----
            {
                float p[kHG];
#pragma unroll
                for (int h = 0; h < kHG; ++h) {
                    p[h] = ex2_approx(sv[h] - m_ref[h]);
                    l_part[h] += p[h];
                }
                uint8_t* pbuf = smem + kOffP + (b & 1) * kPBytes + (j >> 3) * 128 + (j & 7) * 16;
#pragma unroll
                for (int tt = 0; tt < 4; ++tt) {
                    const float rt = sc[tt] * inv_sigma[tt] * kPScale;
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) split2(p[2 * k] * rt, p[2 * k + 1] * rt, hi[k], lo[k]);
                    *reinterpret_cast<uint4*>(pbuf + (tt * 2 + 0) * 2048) =
                        make_uint4(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16), hi[4] | (hi[5] << 16), hi[6] | (hi[7] << 16));
                    *reinterpret_cast<uint4*>(pbuf + (tt * 2 + 1) * 2048) =
                        make_uint4(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16), lo[4] | (lo[5] << 16), lo[6] | (lo[7] << 16));
                }
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_ready[b & 1]);
        }

        // ---- epilogue ----
        if (ok && nblk > 0)
            ok = wait_or_abort(&empty[(nblk - 1) & 1], static_cast<uint32_t>(((nblk - 1) >> 1) & 1), abort_flag);
        tc::fence_after_sync();
        if (!bar_sync_or(1, kComputeThreads, !ok)) {
            float* rw = red + qd * 32;
#pragma unroll
            for (int h = 0; h < kHG; ++h) {
                const float lh = warp_sum(l_part[h]);
                if (lane == 0) rw[h] = lh;
            }
            bar_sync_or(1, kComputeThreads, false);
            float mult[kHG];
#pragma unroll
            for (int h = 0; h < kHG; ++h) {
                const float lh = (red[h] + red[32 + h]) + (red[64 + h] + red[96 + h]);
                mult[h] = lh > 0.0f ? 1.0f / (kPScale * lh) : 0.0f;
                l_part[h] = lh;
            }
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) {
                uint32_t ov[16];
                if (nblk > 0) {
                    tc::tmem_ld16(tmem + lane_base + kColO + 16 * tt, ov);
                    tc::wait_ld();
                } else {
#pragma unroll
                    for (int h = 0; h < kHG; ++h) ov[h] = 0u;
                }
                const int d = 128 * tt + j;
#pragma unroll
                for (int h = 0; h < kHG; ++h) {
                    if (hg * kHG + h >= H) continue;
                    const float v = __uint_as_float(ov[h]) * sigma[tt] * mult[h];
                    if (args.nsplit == 1) {
                        args.out[(qrow0 + h) * kLatent + d] = __float2bfloat16_rn(v);
                    } else {
                        const int64_t prow = (static_cast<int64_t>(t) * args.nsplit + split) * H + hg * kHG + h;
                        args.ws_o[prow * kLatent + d] = v;
                    }
                }
            }
            if (ct < kHG && hg * kHG + ct < H) {
                const float lh = l_part[ct];
                const float lse2 = lh > 0.0f ? (m_ref[ct] + log2f(lh)) * kLn2 : -INFINITY;
                if (args.nsplit == 1) {
                    args.lse[qrow0 + ct] = lse2;
                } else {
                    args.ws_lse[(static_cast<int64_t>(t) * args.nsplit + split) * H + hg * kHG + ct] = lse2;
                }
            }
        } else if (ct == 0) {
            atomicOr(args.err, MLA_ERR_PIPELINE_TIMEOUT);
        }
    }

    // ---- teardown: copies landed, MMAs done, tensor memory released ----
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        atomicOr(args.err, MLA_ERR_PIPELINE_TIMEOUT);
        const int issued = *issued_s;
        for (int bb = max(0, issued - 2); bb < issued; ++bb)
            (void)mbar_wait_bounded(&full[bb & 1], static_cast<uint32_t>((bb >> 1) & 1));
    }
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// Merge of the split partials of one (token, head): lse = ln sum_s exp(lse_s),
// out = sum_s exp(lse_s - lse) o_s, in split order.
__global__ void __launch_bounds__(128)
mla_split_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                         int H, int nsplit, __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
    const int64_t th = blockIdx.x;              // t * H + h
    const int64_t t = th / H;
    const int h = static_cast<int>(th % H);
    float mx = -INFINITY;
    for (int s = 0; s < nsplit; ++s) mx = fmaxf(mx, ws_lse[(t * nsplit + s) * H + h]);
    const int d = 4 * threadIdx.x;
    __nv_bfloat16* orow = out + th * kLatent + d;
    if (mx == -INFINITY) {
        *reinterpret_cast<uint2*>(orow) = make_uint2(0u, 0u);
        if (threadIdx.x == 0) lse[th] = -INFINITY;
        return;
    }
    float wsum = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < nsplit; ++s) {
        const int64_t prow = (t * nsplit + s) * H + h;
        const float ls = ws_lse[prow];
        if (ls == -INFINITY) continue;
        const float w = expf(ls - mx);
        wsum += w;
        const float4 v = *reinterpret_cast<const float4*>(ws_o + prow * kLatent + d);
        acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
    }
    const float inv = 1.0f / wsum;
    *reinterpret_cast<uint2*>(orow) = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv),
                                                 pack_bf16x2(acc.z * inv, acc.w * inv));
    if (threadIdx.x == 0) lse[th] = mx + logf(wsum);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Splits of each token's top-k list: about two CTAs per SM overall (one CTA
// per SM is resident), at least 128 positions per split, at most kListMax.
int choose_nsplit(int T, int H, int W, int sms) {
    if (T <= 0 || W <= 0) return 1;
    const int64_t base = static_cast<int64_t>(T) * ((H + kHG - 1) / kHG);
    const int64_t target = 2ll * sms;
    int64_t ns = (target + base - 1) / base;
    const int64_t max_ns = (W >= 128) ? W / 128 : 1;
    if (ns > max_ns) ns = max_ns;
    const int64_t min_ns = (W + kListMax - 1) / kListMax;
    if (ns < min_ns) ns = min_ns;
    if (ns < 1) ns = 1;
    return static_cast<int>(ns);
}

size_t workspace_for(int T, int H, int nsplit) {
    if (nsplit <= 1) return 0;
    const size_t rows = static_cast<size_t>(T) * nsplit * H;
    const size_t o_bytes = rows * kLatent * sizeof(float);
    return o_bytes + ((rows * sizeof(float) + 255) & ~static_cast<size_t>(255));
}

// ---- TMA tensor maps over the cache (driver entry point, looked up once) ----
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Cache viewed as a 2-D byte tensor [rows, 656]; boxes one row high (gather4).
bool make_row_map(CUtensorMap* m, void* data, int64_t rows, uint32_t box_bytes, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kRowBytes), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRowBytes)};
    const cuuint32_t box[2] = {box_bytes, 1};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, data, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              sw, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" size_t mla_sparse_decode_workspace_bytes(int T, int H, int W) {
    if (T <= 0 || H <= 0 || H > 128 || W < 0) return 0;
    const int sms = mla_host::sm_count();
    if (sms <= 0) return 0;
    return workspace_for(T, H, choose_nsplit(T, H, W, sms));
}

extern "C" int mla_sparse_decode(const void* q_bf16, int T, int H, int d_qk, mla_kv_cache_t kv,
                                 const int32_t* topk_idx, int W, float sm_scale, void* out_bf16,
                                 float* lse, void* workspace, size_t workspace_bytes, void* stream) {
    if (T < 0 || W < 0 || kv.row_bytes != MLA_ROW_BYTES || kv.num_slots < 0 || !std::isfinite(sm_scale))
        return MLA_EINVAL;
    if (d_qk != kLatent && d_qk != kLatent + kRope) return MLA_EUNSUPPORTED;
    if (H < 1 || H > 128) return MLA_EUNSUPPORTED;
    if (kv.num_slots >= INT32_MAX) return MLA_EUNSUPPORTED;     // row coordinates are 32-bit
    if (T == 0) return MLA_OK;
    if (q_bf16 == nullptr || out_bf16 == nullptr || lse == nullptr || (W > 0 && topk_idx == nullptr) ||
        (W > 0 && kv.data == nullptr))
        return MLA_EINVAL;
    if (!aligned16(q_bf16) || !aligned16(out_bf16) || (kv.data && !aligned16(kv.data)) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(topk_idx) & 3u))
        return MLA_EINVAL;
    int* err = mla_host::device_error_word();
    const int sms = mla_host::sm_count();
    if (err == nullptr || sms <= 0) return MLA_ECUDA;
    const int nsplit = choose_nsplit(T, H, W, sms);
    const size_t need = workspace_for(T, H, nsplit);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
        return MLA_ENOWORKSPACE;

    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ECUDA;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(mla_sparse_decode_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemAlloc) != cudaSuccess ||
            cudaFuncSetAttribute(mla_sparse_decode_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemAlloc) != cudaSuccess)
            return MLA_ECUDA;
        attr_set[dev] = true;
    }
    // Tensor maps: rows are 1 .. num_slots-1 at most; a coordinate >= the row
    // count reads as zeros (used for the ragged end of a block).
    alignas(64) CUtensorMap tm_row;
    alignas(64) CUtensorMap tm_scale;
    std::memset(&tm_row, 0, sizeof tm_row);
    std::memset(&tm_scale, 0, sizeof tm_scale);
    const int64_t rows = kv.num_slots > 0 ? kv.num_slots : 1;
    if (W > 0) {
        if (!make_row_map(&tm_row, kv.data, rows, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_row_map(&tm_scale, kv.data, rows, 16, CU_TENSOR_MAP_SWIZZLE_NONE))
            return MLA_ECUDA;
    }
    DecodeArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q_bf16);
    a.topk = topk_idx;
    a.out = static_cast<__nv_bfloat16*>(out_bf16);
    a.lse = lse;
    a.ws_o = static_cast<float*>(workspace);
    a.ws_lse = nsplit > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                     static_cast<size_t>(T) * nsplit * H * kLatent * sizeof(float))
                          : nullptr;
    a.err = err;
    a.num_slots = kv.num_slots;
    a.oob_row = static_cast<int>(rows);
    a.T = T; a.H = H; a.d_qk = d_qk; a.W = W; a.nsplit = nsplit;
    a.split_len = (W + nsplit - 1) / nsplit;
    a.sm_scale_log2 = sm_scale * kLog2e;
    const dim3 grid(static_cast<unsigned>(T), static_cast<unsigned>(nsplit), static_cast<unsigned>((H + kHG - 1) / kHG));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (d_qk == kLatent + kRope)
        mla_sparse_decode_tc_kernel<true><<<grid, kThreads, kSmemAlloc, st>>>(tm_row, tm_scale, a);
    else
        mla_sparse_decode_tc_kernel<false><<<grid, kThreads, kSmemAlloc, st>>>(tm_row, tm_scale, a);
    if (cudaGetLastError() != cudaSuccess) return MLA_ECUDA;
    if (nsplit > 1) {
        mla_split_combine_kernel<<<static_cast<unsigned>(static_cast<int64_t>(T) * H), 128, 0, st>>>(
            a.ws_o, a.ws_lse, H, nsplit, a.out, a.lse);
        if (cudaGetLastError() != cudaSuccess) return MLA_ECUDA;
    }
    return MLA_OK;
}
