// mla_sparse_decode: sparse top-k MLA decode over the packed FP8 cache, on the
// sm_100-family tensor cores (tcgen05 MMAs with tensor-memory accumulators).
//
// What it computes follows the decode statement quoted in the C header, with
// the masking rule of sglang PR #39288 (Root cause: a -1 candidate must add
// nothing and must not gather slot 0) and sglang PR #47013 (Motivation: masking
// only the score does not stop a NaN row). Absent entries are removed before
// anything is fetched, so -1, slot 0 and out-of-range indices are never
// dereferenced and the result does not depend on what slot 0 holds.
//
// Three launches:
//   1. compaction: one CTA per token writes the token's present slots, in list
//      order, to the workspace (positions go through the block table first for
//      the paged entry point, vLLM PR #55277 Purpose item 2) and counts them,
//      and writes the token's q in the layout the MMAs read (below);
//   2. decode: one persistent CTA per SM (per head group). When there are few
//      tokens, the tokens' present entries, laid end to end, are cut into equal
//      row ranges, one per CTA, so every SM gathers the same number of rows
//      whatever the list lengths (vLLM PR #55277 Purpose item 2: the buffer
//      width is a capacity; the active length is what costs). A range covers
//      whole tokens and at most two pieces of tokens shared with its neighbours;
//      a piece writes a normalised partial (o, lse) to the workspace. With many
//      tokens, CTAs take whole tokens;
//   3. merge (few-tokens mode only): tokens split across ranges are merged in
//      range order (lse = ln sum exp lse_i, o = sum exp(lse_i - lse) o_i; no
//      float atomics, so the result is deterministic); empty tokens get 0 / -inf.
//
// Decode CTA: 8 warps. Warps 4..6 copy rows global -> shared, one cp.async.bulk
// per row (656 B, or the 528 B without the tail for NoPE), into a ring of
// 32-row stages; warp 7 issues the MMAs; warps 0..3 own tensor-memory lanes
// 0..127 (thread j <-> row j of a 128-row block, and <-> output dim j of each
// 128-value tile). The work of a block is pipelined per 128-value tile t: QK of
// tile t starts as soon as tile t of every row is in place, PV of tile t as soon
// as the P of tile t is written, and the next block's tile t reuses the buffer
// once PV of tile t is done. Per 128-row block:
//   copy     thread j moves its row's 512 E4M3 codes into the 128-byte-swizzled
//            K-major tile layout (which is also the MN-major layout of V^T for
//            PV), its 64 RoPE values into tensor memory (A of the RoPE MMA) and
//            keeps its four fp32 tile scales in registers;
//   QK       per latent tile t: S_t[j, :] = K_t[j] . [q_hi | q_lo]_t, E4M3 MMAs
//            (M = 128 rows, N = 2 x heads). q is split into two E4M3 terms after
//            a per-head power-of-two shift (hi = e4m3(q'), lo = e4m3(q' - hi)),
//            which holds every bf16 q value but the smallest ones exactly; each
//            tile partial lands in a ring of tensor-memory slots, the RoPE part
//            (bf16 MMA, A in tensor memory) in the next slot. The fp32 tile
//            scales are applied per row afterwards:
//            s_j = (2^k sum_t scale_jt (S_hi + S_lo)_t + R_j) * sm_scale;
//   softmax  online, per head, in log2 units; the exp2 offset moves only when a
//            score exceeds it by more than 2^16;
//   PV       O^T_t[d, h] += V^T_t[d, j] * [P_hi | P_lo]_t[j, h], E4M3 MMAs (M =
//            128 dims of tile t, N = 2 x heads, K = rows), with
//            P_t[j, h] = p_jh * scale_jt * 2 / tau_th split into two E4M3 terms.
//            tau_th is a running maximum of p * scale over the rows seen so far,
//            per (tile, head), raised (and O^T rescaled) only when some P would
//            pass 448: the largest contributions keep E4M3's full precision
//            whatever the spread of the rows' scales. O^T stays in tensor memory
//            until the piece ends.
#include <cfloat>
#include <climits>
#include <cmath>

#include "mla_device.cuh"
#include "mla_tcgen05.cuh"

namespace {

using namespace mla;
namespace tc = mla::tc;

constexpr int kBlockRows = 128;          // rows per block: M of QK, K of PV
constexpr int kStageRows = 32;           // rows per copy stage (one per compute warp)
constexpr int kComputeWarps = 4;
constexpr int kProducerWarp0 = 4;
constexpr int kProducers = 3;
constexpr int kMmaWarp = 7;
constexpr int kThreads = 8 * 32;         // two warps per SM sub-partition: up to 255 registers
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kRawStage = kStageRows * kRowBytes;     // 20,992
constexpr int kMaxBalancedT = 1216;      // tokens up to which rows are balanced across CTAs
constexpr int kMinRowsPerCta = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kSlack = 16.0f;          // log2 units: p <= 2^16
constexpr float kPTarget = 2.0f;         // P of the largest product right after tau is raised (224x headroom)
constexpr float kPMax = 448.0f;          // largest finite E4M3
constexpr int kCompactThreads = 256;
constexpr int kMergeThreads = 128;

template <int NH, bool kRope>
struct Cfg {
    static constexpr int NQ = 2 * NH;                      // N of the latent QK: [hi | lo] q terms
    static constexpr int NP = 2 * NH;                      // N of PV: [hi | lo] P terms
    static constexpr int kSlots = NH == 16 ? 4 : 3;        // tensor-memory slots for QK partials
    static constexpr int kParts = kRope ? 5 : 4;           // partials per block (4 tiles + RoPE)
    static constexpr int kRS = NH == 16 ? 5 : 4;           // copy stages
    static constexpr uint32_t kColO = 0;
    static constexpr uint32_t kColS = 4 * NP;
    static constexpr uint32_t kColRope = kColS + kSlots * NQ;
    static_assert(kColRope + 32 <= 512, "tensor memory");
    // q block of one (token, head group), as the compaction kernel writes it:
    // [4 tiles][NQ rows][128 B] E4M3 terms | [NH rows][128 B] bf16 RoPE | [NH] fp32 2^k
    static constexpr uint32_t kQLat = 4 * NQ * 128;
    static constexpr uint32_t kQBytes = kQLat + NH * 128 + NH * 4;
    static constexpr uint32_t kOffLat = 0;                              // 4 tiles x 16 KB
    static constexpr uint32_t kOffQ = 65536;                            // the q block
    static constexpr uint32_t kOffQR = kOffQ + kQLat;
    static constexpr uint32_t kOffQexp = kOffQR + NH * 128;
    static constexpr uint32_t kOffP = kOffQ + ((kQBytes + 127) & ~127u); // 4 tiles x NP/16 x 2 KB
    static constexpr uint32_t kOffRaw = kOffP + 4 * NP * 128;
    static constexpr uint32_t kOffRed = kOffRaw + kRS * kRawStage;      // [4 warps][4 tiles][NH]
    static constexpr uint32_t kOffTau = kOffRed + 16 * NH * 4;          // [2][tau 4 x NH | 32 / tau 4 x NH]
    static constexpr uint32_t kOffFac = kOffTau + 16 * NH * 4;          // [4 tiles][NP] O^T rescale factors
    static constexpr uint32_t kOffPrefix = kOffFac + 4 * NP * 4;
    static constexpr uint32_t kOffBar = (kOffPrefix + (kMaxBalancedT + 1) * 4 + 7) & ~7u;
    static constexpr int kNumBars = 2 * kRS + 2 * kSlots + 12 + 3;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kSmemUsed = kOffMisc + 64;
    static constexpr uint32_t kSmemAlloc = kSmemUsed + 1024;            // base aligned up to 1024 B
    static_assert(kSmemAlloc <= 232448, "shared memory");
    static_assert(kOffQ % 1024 == 0 && kOffQR % 1024 == 0, "swizzled operands need 1024-B alignment");
};

struct DecodeArgs {
    const __nv_bfloat16* q;
    const uint8_t* cache;
    int64_t row_bytes;
    const int32_t* comp;       // [T, W] present slots of each token, in list order
    const int32_t* cnt;        // [T]
    const uint8_t* qc;         // [T, HG] q blocks (Cfg::kQBytes each)
    __nv_bfloat16* out;
    float* lse;
    float* ws_o;               // [2G, H, 512] partials (few-tokens mode)
    float* ws_lse;             // [2G, H]
    int32_t* ws_prefix;        // [T + 1]
    int32_t* ws_ctl;           // [0] = number of row ranges in use
    int* err;
    int T, H, d_qk, W, HG, G, balanced;
    float sm_scale_log2;       // sm_scale * log2(e)
};

// q block layout for NH heads per group (mirrors Cfg).
__host__ __device__ constexpr uint32_t q_block_bytes(int NH) { return 4 * (2 * NH) * 128 + NH * 128 + NH * 4; }

// Bounded wait that also gives up once another role has given up.
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

// Monotonic per-slot release counters for the copy ring. Three producers share
// the slots and the four consumer warps release their stages in any order
// within a block, so a producer may reach a slot two uses ahead of its last
// release; a phase-parity wait cannot tell those uses apart, a count can.
__device__ __forceinline__ void release_slot(uint32_t* ctr) {
    asm volatile("red.release.cta.shared::cta.add.u32 [%0], 1;" :: "r"(smem_u32(ctr)) : "memory");
}
__device__ __forceinline__ uint32_t released(const uint32_t* ctr) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(ctr)) : "memory");
    return v;
}
// Bounded wait until the slot has been released `uses` times.
__device__ __forceinline__ bool wait_released(const uint32_t* ctr, uint32_t uses, volatile int* abort_flag) {
    if (released(ctr) >= uses) return true;
    const long long t0 = clock64();
    for (;;) {
        __nanosleep(32);
        if (released(ctr) >= uses) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitCycles) {
            *abort_flag = 1;
            return false;
        }
    }
}

// Warp maximum in one redux.sync: floats mapped to unsigned keys in the same order.
__device__ __forceinline__ float warp_max_redux(float v) {
    const uint32_t u = __float_as_uint(v);
    const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    const uint32_t r = __reduce_max_sync(0xffffffffu, key);
    return __uint_as_float((r & 0x80000000u) ? (r & 0x7FFFFFFFu) : ~r);
}
// Same for values known to be >= 0 (their bit patterns already sort as unsigned).
__device__ __forceinline__ float warp_max_nonneg(float v) {
    return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
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

// E4M3 pair (low byte = x0), round to nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x2(float x0, float x1) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3));
}
// hi + lo split of a pair: hi = e4m3(x), lo = e4m3(x - hi); returns hi | lo << 16.
__device__ __forceinline__ uint32_t split_pair(float x0, float x1) {
    const uint32_t hi = e4m3x2(x0, x1);
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(hi), __NV_E4M3);
    const float2 hv = __half22float2(*reinterpret_cast<const __half2*>(&hr));
    return hi | (e4m3x2(x0 - hv.x, x1 - hv.y) << 16);
}

// Token whose present rows contain global row x: the largest t with prefix[t] <= x.
__device__ __forceinline__ int token_of(const int32_t* prefix, int T, int64_t x) {
    int lo = 0, hi = T;          // prefix[lo] <= x < prefix[hi] when x < prefix[T]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= x) lo = mid; else hi = mid;
    }
    return lo;
}
__device__ __forceinline__ int64_t range_start(int64_t P, int G, int r) { return P * r / G; }

// The piece of token t handled by the CTA whose rows are [start, end): local
// rows [pa, pb) of the token's present list. False when the token has none here.
__device__ __forceinline__ bool piece_of(const DecodeArgs& a, const int32_t* prefix, int t, int64_t start, int64_t end,
                                         int& pa, int& pb) {
    if (a.balanced) {
        const int64_t p0 = prefix[t], p1 = prefix[t + 1];
        const int64_t lo = max(start, p0), hi = min(end, p1);
        if (lo >= hi) return false;
        pa = static_cast<int>(lo - p0);
        pb = static_cast<int>(hi - p0);
        return true;
    }
    pa = 0;
    pb = __ldg(a.cnt + t);
    return true;
}

// ======================= 1. compaction =======================
__global__ void __launch_bounds__(kCompactThreads)
mla_topk_compact_kernel(const int32_t* __restrict__ topk, int W, int64_t num_slots, const int32_t* __restrict__ block_table,
                        const int32_t* __restrict__ token_seq, int bt_pages, int n_seq, int page_size,
                        int32_t* __restrict__ comp, int32_t* __restrict__ cnt, int* __restrict__ err,
                        const __nv_bfloat16* __restrict__ q, int H, int d_qk, int NH, int HG, uint8_t* __restrict__ qc) {
    pdl_launch_dependents();
    __shared__ int wsum[kCompactThreads / 32];
    const int t = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- q of token t, per head group, in the layout of the MMA operands: the
    // latent part as two E4M3 terms after a per-head power-of-two shift
    // (q' = q 2^(8-e) with max|q'| < 256; hi = e4m3(q'), lo = e4m3(q' - hi), which
    // holds every bf16 value of the head but the smallest ones exactly), rows
    // 0..NH-1 = hi and NH..2NH-1 = lo of each 128-value tile, 128-byte swizzled
    // K-major; the RoPE part as bf16 in the same swizzled form; then 2^(e-8). ----
    const int NQ = 2 * NH;
    const uint32_t qbytes = q_block_bytes(NH);
    // All of this warp's q loads are issued before any is used (one latency, not one per head).
    constexpr int kMaxHeadsPerWarp = 128 / (kCompactThreads / 32);
    uint4 qv[kMaxHeadsPerWarp][2];
    uint4 rv[kMaxHeadsPerWarp];
#pragma unroll
    for (int i = 0; i < kMaxHeadsPerWarp; ++i) {
        const int hh = warp + i * (kCompactThreads / 32);
        qv[i][0] = qv[i][1] = rv[i] = make_uint4(0u, 0u, 0u, 0u);
        if (hh < H) {
            const __nv_bfloat16* qh = q + (static_cast<int64_t>(t) * H + hh) * d_qk;
            qv[i][0] = ld_nc_v4(qh + 16 * lane);
            qv[i][1] = ld_nc_v4(qh + 16 * lane + 8);
            if (lane < 8 && d_qk > kLatent) rv[i] = ld_nc_v4(qh + kLatent + 8 * lane);
        }
    }
#pragma unroll
    for (int i = 0; i < kMaxHeadsPerWarp; ++i) {
        const int hh = warp + i * (kCompactThreads / 32);
        if (hh >= HG * NH) break;
        const int g = hh / NH, h = hh % NH;
        uint8_t* qb = qc + (static_cast<int64_t>(t) * HG + g) * qbytes;
        const uint32_t v[8] = {qv[i][0].x, qv[i][0].y, qv[i][0].z, qv[i][0].w,
                               qv[i][1].x, qv[i][1].y, qv[i][1].z, qv[i][1].w};
        float mx = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) mx = fmaxf(mx, fmaxf(fabsf(bf16lo(v[k])), fabsf(bf16hi(v[k]))));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        int e = 0;
        frexpf(mx, &e);                                   // mx < 2^e
        const float down = ldexpf(1.0f, 8 - e);
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float a0 = bf16lo(v[2 * k]) * down, a1 = bf16hi(v[2 * k]) * down;
            const float b0 = bf16lo(v[2 * k + 1]) * down, b1 = bf16hi(v[2 * k + 1]) * down;
            const uint32_t ha = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a0, a1), __NV_SATFINITE, __NV_E4M3));
            const uint32_t hb = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(b0, b1), __NV_SATFINITE, __NV_E4M3));
            const __half2_raw ra = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(ha), __NV_E4M3);
            const __half2_raw rb = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(hb), __NV_E4M3);
            const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&ra));
            const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&rb));
            const uint32_t la = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a0 - fa.x, a1 - fa.y), __NV_SATFINITE, __NV_E4M3));
            const uint32_t lb = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(b0 - fb.x, b1 - fb.y), __NV_SATFINITE, __NV_E4M3));
            hi[k] = ha | (hb << 16);
            lo[k] = la | (lb << 16);
        }
        const int tile = lane >> 3, u = lane & 7;
        uint8_t* tb = qb + tile * (NQ * 128);
        const int rh = h, rl = NH + h;
        *reinterpret_cast<uint4*>(tb + (rh >> 3) * 1024 + (rh & 7) * 128 + ((u ^ (rh & 7)) << 4)) =
            make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(tb + (rl >> 3) * 1024 + (rl & 7) * 128 + ((u ^ (rl & 7)) << 4)) =
            make_uint4(lo[0], lo[1], lo[2], lo[3]);
        if (lane < 8)
            *reinterpret_cast<uint4*>(qb + 4 * NQ * 128 + (h >> 3) * 1024 + (h & 7) * 128 + ((lane ^ (h & 7)) << 4)) = rv[i];
        if (lane == 0) *reinterpret_cast<float*>(qb + 4 * NQ * 128 + NH * 128 + 4 * h) = ldexpf(1.0f, e - 8);
    }

    // ---- the token's present slots, in list order: every position loaded at once ----
    const int32_t* row = topk + static_cast<int64_t>(t) * W;
    int32_t* dst = comp + static_cast<int64_t>(t) * W;
    const int32_t* bt = nullptr;
    bool seq_ok = true;
    if (page_size > 0) {
        const int sq = token_seq ? __ldg(token_seq + t) : 0;
        seq_ok = sq >= 0 && sq < n_seq;
        bt = block_table + static_cast<int64_t>(seq_ok ? sq : 0) * bt_pages;
    }
    constexpr int kPerThreadMax = 16;                     // positions per thread held in registers
    int base = 0;
    for (int c0 = 0; c0 < W; c0 += kCompactThreads * kPerThreadMax) {
        int64_t idx[kPerThreadMax];
#pragma unroll
        for (int k = 0; k < kPerThreadMax; ++k) {
            const int pp = c0 + k * kCompactThreads + static_cast<int>(threadIdx.x);
            idx[k] = (pp < W) ? __ldg(row + pp) : -1;
        }
        if (page_size > 0) {
            // Positions -> slots (vLLM PR #55277, Purpose item 2): a negative
            // position or an unassigned (negative) page is absent; a page past the
            // table or a sequence outside it is absent and flagged.
            int phys[kPerThreadMax];
#pragma unroll
            for (int k = 0; k < kPerThreadMax; ++k) {
                const int64_t page = idx[k] >= 0 ? idx[k] / page_size : -1;
                phys[k] = (idx[k] >= 0 && seq_ok && page < bt_pages) ? __ldg(bt + page) : -1;
            }
#pragma unroll
            for (int k = 0; k < kPerThreadMax; ++k) {
                if (idx[k] < 0) continue;
                const int64_t page = idx[k] / page_size;
                if (!seq_ok || page >= bt_pages) {
                    atomicOr(err, MLA_ERR_DECODE_INDEX_RANGE);
                    idx[k] = -1;
                } else {
                    idx[k] = (phys[k] < 0) ? -1 : static_cast<int64_t>(phys[k]) * page_size + (idx[k] - page * page_size);
                }
            }
        }
#pragma unroll 1
        for (int k = 0; k < kPerThreadMax && c0 + k * kCompactThreads < W; ++k) {
            const bool valid = idx[k] > 0 && idx[k] < num_slots;
            if (idx[k] > 0 && !valid) atomicOr(err, MLA_ERR_DECODE_INDEX_RANGE);
            const unsigned m = __ballot_sync(0xffffffffu, valid);
            if (lane == 0) wsum[warp] = __popc(m);
            __syncthreads();
            int off = base, tot = 0;
#pragma unroll
            for (int w = 0; w < kCompactThreads / 32; ++w) {
                const int c = wsum[w];
                off += (w < warp) ? c : 0;
                tot += c;
            }
            if (valid) dst[off + __popc(m & ((1u << lane) - 1u))] = static_cast<int32_t>(idx[k]);
            base += tot;
            __syncthreads();
        }
    }
    if (threadIdx.x == 0) cnt[t] = base;
    // Complete only after the previous kernel on the stream (the writer, when the
    // decode follows it) has completed: the decode kernel reads the cache once
    // this grid is done.
    pdl_wait();
}

// ======================= 2. decode =======================
template <int NH, bool kRope>
__global__ void __launch_bounds__(kThreads, 1)
mla_sparse_decode_kernel(const DecodeArgs a) {
    using C = Cfg<NH, kRope>;
    constexpr int NQ = C::NQ, NP = C::NP;
    constexpr uint32_t kRowRead = kRope ? kRowBytes : kNopeReadBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);   // [kRS] stage landed
    uint32_t* rel = reinterpret_cast<uint32_t*>(full + C::kRS);        // [kRS] stage releases (counts)
    uint64_t* s_full = full + 2 * C::kRS;                              // [kSlots] QK partial ready
    uint64_t* s_free = s_full + C::kSlots;                             // [kSlots] partial read
    uint64_t* canon = s_free + C::kSlots;                              // [4] tile t of the block in place
    uint64_t* ptile = canon + 4;                                       // [4] P of tile t written
    uint64_t* pvdone = ptile + 4;                                      // [4] PV of tile t done
    uint64_t* q_full = pvdone + 4;                                     // q block of the piece landed
    uint64_t* q_drain = q_full + 1;                                    // last QK of the piece done
    uint64_t* drain = q_drain + 1;                                     // all MMAs done (teardown)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* issued = reinterpret_cast<int*>(tmem_slot + 2);               // [kRS] stage uses issued
    int* q_issued = issued + C::kRS;                                   // q copies issued
    int* wsum = q_issued + 1;                                          // [8] scan scratch
    int32_t* prefix = reinterpret_cast<int32_t*>(smem + C::kOffPrefix);
    float* red = reinterpret_cast<float*>(smem + C::kOffRed);
    float* tau_s = reinterpret_cast<float*>(smem + C::kOffTau);
    float* fac_s = reinterpret_cast<float*>(smem + C::kOffFac);
    const float* qexp_s = reinterpret_cast<const float*>(smem + C::kOffQexp);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kRS; ++s) {
            mbar_init(&full[s], 1);
            rel[s] = 0u;
            issued[s] = 0;
        }
        for (int s = 0; s < C::kSlots; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&s_free[s], kComputeWarps);
        }
        for (int t = 0; t < 4; ++t) {
            mbar_init(&canon[t], kComputeWarps);
            mbar_init(&ptile[t], kComputeWarps);
            mbar_init(&pvdone[t], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_drain, 1);
        mbar_init(drain, 1);
        *q_issued = 0;
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
        tc::fence_before_sync();
    }
    // Launched with programmatic stream serialization: the compaction grid (and,
    // through it, the kernel before it) is complete from here on.
    pdl_wait();

    // ---- schedule: this CTA's rows (few tokens) or tokens (many) ----
    const int hg = static_cast<int>(blockIdx.x) % a.HG;
    const int r = static_cast<int>(blockIdx.x) / a.HG;
    int64_t start = 0, end = 0;
    int t_lo = 0, t_hi = 0;
    if (a.balanced) {
        // prefix[t] = present rows of tokens < t (block-wide scan of the counts)
        const int per = (a.T + kThreads - 1) / kThreads;
        const int t0 = static_cast<int>(threadIdx.x) * per;
        int local = 0;
        for (int i = 0; i < per; ++i)
            if (t0 + i < a.T) local += __ldg(a.cnt + t0 + i);
        int incl = local;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        int off = incl - local;
        for (int w = 0; w < warp; ++w) off += wsum[w];
        for (int i = 0; i < per; ++i) {
            if (t0 + i < a.T) {
                prefix[t0 + i] = off;
                off += __ldg(a.cnt + t0 + i);
            }
        }
        if (threadIdx.x == kThreads - 1) prefix[a.T] = off;
        __syncthreads();
        const int64_t P = prefix[a.T];
        const int G = P == 0 ? 0 : static_cast<int>(min(static_cast<int64_t>(a.G), (P + kMinRowsPerCta - 1) / kMinRowsPerCta));
        if (blockIdx.x == 0) {
            for (int i = threadIdx.x; i <= a.T; i += kThreads) a.ws_prefix[i] = prefix[i];
            if (threadIdx.x == 0) a.ws_ctl[0] = G;
        }
        if (r < G) {
            start = range_start(P, G, r);
            end = range_start(P, G, r + 1);
            if (end > start) {
                t_lo = token_of(prefix, a.T, start);
                t_hi = token_of(prefix, a.T, end - 1) + 1;
            }
        }
    } else {
        t_lo = static_cast<int>(static_cast<int64_t>(a.T) * r / a.G);
        t_hi = static_cast<int>(static_cast<int64_t>(a.T) * (r + 1) / a.G);
    }
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // The merge launch behind this one may start its set-up; it waits for this
    // grid's completion before it reads anything.
    pdl_launch_dependents();

    if (warp >= kProducerWarp0 && warp < kProducerWarp0 + kProducers) {
        // ================= producers: warp p copies stages k = p, p + 3, ... =================
        // Stage k holds rows 32 (k % 4) .. +31 of block k / 4 (the rows of compute
        // warp k % 4); lane i copies row i of the stage.
        const int p = warp - kProducerWarp0;
        uint32_t gbk = 0;
        for (int t = t_lo; t < t_hi; ++t) {
            int pa, pb;
            if (!piece_of(a, prefix, t, start, end, pa, pb)) continue;
            const int32_t* list = a.comp + static_cast<int64_t>(t) * a.W + pa;
            const int nrows = pb - pa;
            const int nblk = (nrows + kBlockRows - 1) / kBlockRows;
            for (int kb = 0; kb < nblk; ++kb, ++gbk) {
                for (int sw = 0; sw < kComputeWarps; ++sw) {
                    const uint32_t k = gbk * kComputeWarps + sw;
                    if (k % kProducers != static_cast<uint32_t>(p)) continue;
                    const uint32_t slot = k % C::kRS, use = k / C::kRS;
                    const int row0 = kb * kBlockRows + sw * kStageRows;
                    const int n = max(0, min(kStageRows, nrows - row0));
                    const int sidx = (lane < n) ? __ldg(list + row0 + lane) : 0;
                    if (use > 0 && !wait_released(&rel[slot], use, abort_flag)) goto producer_done;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(n) * kRowRead);
                        issued[slot] = static_cast<int>(use) + 1;
                    }
                    __syncwarp();
                    if (lane < n)
                        bulk_g2s(smem + C::kOffRaw + slot * kRawStage + lane * kRowBytes,
                                 a.cache + static_cast<int64_t>(sidx) * a.row_bytes, kRowRead, &full[slot]);
                }
            }
        }
    producer_done:;
    } else if (warp == kMmaWarp) {
        // ================= MMA issuer (one thread), also the q copies =================
        if (lane == 0) {
            constexpr uint32_t id_qk = tc::instr_desc(tc::kE4M3, tc::kE4M3, false, false, 128, NQ);
            constexpr uint32_t id_rope = tc::instr_desc(tc::kBF16, tc::kBF16, false, false, 128, NH);
            constexpr uint32_t id_pv = tc::instr_desc(tc::kE4M3, tc::kE4M3, true, true, 128, NP);
            const uint32_t lat = sbase + C::kOffLat;
            const uint64_t q_desc0 = tc::smem_desc(sbase + C::kOffQ, 16, 1024, tc::kSw128);
            const uint64_t qr_desc0 = tc::smem_desc(sbase + C::kOffQR, 16, 1024, tc::kSw128);
            const uint64_t lat_desc0 = tc::smem_desc(lat, 16, 1024, tc::kSw128);
            const uint64_t v_desc0 = tc::smem_desc(lat, 16384, 1024, tc::kSw128);
            const uint64_t p_desc0 = tc::smem_desc(sbase + C::kOffP, 128, 2048, tc::kSwNone);
            uint32_t gbk = 0, sk = 0, qn = 0;        // blocks, QK partials, pieces with work
            // q of the first piece with work
            int tq = t_lo;
            for (; tq < t_hi; ++tq) {
                int pa, pb;
                if (piece_of(a, prefix, tq, start, end, pa, pb) && pb > pa) break;
            }
            if (tq < t_hi) {
                mbar_arrive_expect_tx(q_full, C::kQBytes);
                *q_issued = 1;
                bulk_g2s(smem + C::kOffQ, a.qc + (static_cast<int64_t>(tq) * a.HG + hg) * C::kQBytes, C::kQBytes, q_full);
            }
            for (int t = t_lo; t < t_hi; ++t) {
                int pa, pb;
                if (!piece_of(a, prefix, t, start, end, pa, pb)) continue;
                const int nblk = (pb - pa + kBlockRows - 1) / kBlockRows;
                if (nblk == 0) continue;
                if (!wait_or_abort(q_full, qn & 1, abort_flag)) goto mma_done;
                for (int kb = 0; kb < nblk; ++kb, ++gbk) {
                    // ---- QK: one partial per latent tile as soon as the tile is in place, then RoPE ----
                    for (int part = 0; part < C::kParts; ++part, ++sk) {
                        if (part < 4 && !wait_or_abort(&canon[part], gbk & 1, abort_flag)) goto mma_done;
                        const uint32_t slot = sk % C::kSlots, use = sk / C::kSlots;
                        if (use > 0 && !wait_or_abort(&s_free[slot], (use - 1) & 1, abort_flag)) goto mma_done;
                        tc::fence_after_sync();
                        const uint32_t d = tmem + C::kColS + slot * NQ;
                        if (part < 4) {
                            // S_t = K_t . [q_hi | q_lo]_t: four K-steps of 32 codes
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
                                tc::mma_f8_ss(d, lat_desc0 + static_cast<uint64_t>((part * 16384 + ks * 32) >> 4),
                                              q_desc0 + static_cast<uint64_t>((part * NQ * 128 + ks * 32) >> 4), id_qk,
                                              ks > 0 ? 1u : 0u);
                        } else {
                            // R = rope . q_rope: A (bf16 rows) in tensor memory, four K-steps of 16
#pragma unroll
                            for (int kr = 0; kr < 4; ++kr)
                                tc::mma_f16_ts(d, tmem + C::kColRope + 8 * kr,
                                               qr_desc0 + static_cast<uint64_t>((kr * 32) >> 4), id_rope, kr > 0 ? 1u : 0u);
                        }
                        tc::commit(&s_full[slot]);
                    }
                    if (kb == nblk - 1) {
                        // Last QK of the piece issued: once it is done, fetch the next
                        // piece's q into the same buffer.
                        tc::commit(q_drain);
                        int tn = t + 1;
                        for (; tn < t_hi; ++tn) {
                            int qa, qb2;
                            if (piece_of(a, prefix, tn, start, end, qa, qb2) && qb2 > qa) break;
                        }
                        if (!wait_or_abort(q_drain, qn & 1, abort_flag)) goto mma_done;
                        if (tn < t_hi) {
                            mbar_arrive_expect_tx(q_full, C::kQBytes);
                            *q_issued = static_cast<int>(qn) + 2;
                            bulk_g2s(smem + C::kOffQ, a.qc + (static_cast<int64_t>(tn) * a.HG + hg) * C::kQBytes,
                                     C::kQBytes, q_full);
                        }
                    }
                    // ---- PV: tile t as soon as its P is written ----
#pragma unroll 1
                    for (int tt = 0; tt < 4; ++tt) {
                        if (!wait_or_abort(&ptile[tt], gbk & 1, abort_flag)) goto mma_done;
                        tc::fence_after_sync();
#pragma unroll
                        for (int ke = 0; ke < 4; ++ke)
                            tc::mma_f8_ss(tmem + C::kColO + tt * NP,
                                          v_desc0 + static_cast<uint64_t>((tt * 16384 + ke * 4096) >> 4),
                                          p_desc0 + static_cast<uint64_t>((tt * NP * 128 + ke * 512) >> 4), id_pv,
                                          (kb > 0 || ke > 0) ? 1u : 0u);
                        tc::commit(&pvdone[tt]);
                    }
                }
                ++qn;
            }
        mma_done:
            // Every MMA this thread issued completes before the CTA tears down.
            tc::commit(drain);
            (void)mbar_wait_bounded(drain, 0);
        }
        __syncwarp();
    } else if (warp < kComputeWarps) {
        // ================= compute warps: thread j = row j / output dim j =================
        const int w = warp;
        const int j = w * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * w) << 16;
        const int jr = j & 7;
        uint8_t* lat_row = smem + C::kOffLat + (j >> 3) * 1024 + jr * 128;
        uint8_t* p_row = smem + C::kOffP + (j >> 3) * 128 + jr * 16;
        const int H = a.H;
        uint32_t gbk = 0, sk = 0, qn = 0;
        bool ok = true;
        for (int t = t_lo; t < t_hi && ok; ++t) {
            int pa, pb;
            if (!piece_of(a, prefix, t, start, end, pa, pb)) continue;
            const int nrows = pb - pa;
            const int nblk = (nrows + kBlockRows - 1) / kBlockRows;
            const bool whole = !a.balanced || (pa == 0 && pb == prefix[t + 1] - prefix[t]);
            const int64_t out_slot = (t == t_lo) ? 2 * r : 2 * r + 1;

            int tb = 0;                                   // which tau buffer is current (CTA-uniform)
            if (j < 4 * NH) {
                tau_s[j] = 0.0f;
                tau_s[4 * NH + j] = 0.0f;
            }
            float qexp[NH];
            {
                bool okq = nblk == 0 || wait_or_abort(q_full, qn & 1, abort_flag);
                okq = __all_sync(0xffffffffu, okq);
                if (bar_sync_or(1, kComputeThreads, !okq)) { ok = false; break; }
#pragma unroll
                for (int h = 0; h < NH; ++h) qexp[h] = nblk > 0 ? qexp_s[h] : 1.0f;
            }

            float m_ref[NH], l_part[NH];
#pragma unroll
            for (int h = 0; h < NH; ++h) { m_ref[h] = -INFINITY; l_part[h] = 0.0f; }

            for (int kb = 0; kb < nblk; ++kb, ++gbk) {
                // ---- copy this warp's 32 rows into the MMA layouts, tile by tile ----
                const uint32_t k = gbk * kComputeWarps + w;
                const uint32_t slot = k % C::kRS, use = k / C::kRS;
                bool okw = wait_or_abort(&full[slot], use & 1, abort_flag);
                okw = __all_sync(0xffffffffu, okw);
                const int n_b = min(kBlockRows, nrows - kb * kBlockRows);
                const bool present = j < n_b;
                const uint8_t* src = smem + C::kOffRaw + slot * kRawStage + lane * kRowBytes;
                float sc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if (okw && present) {
                    const float4 s4 = *reinterpret_cast<const float4*>(src + kScaleOff);
                    sc[0] = s4.x; sc[1] = s4.y; sc[2] = s4.z; sc[3] = s4.w;
                }
#pragma unroll 1
                for (int tt = 0; tt < 4; ++tt) {
                    // the previous block's PV of this tile has read the buffer
                    if (gbk > 0) okw = okw && wait_or_abort(&pvdone[tt], (gbk - 1) & 1, abort_flag);
                    okw = __all_sync(0xffffffffu, okw);
                    if (okw) {
                        uint4 v[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            v[u] = present ? *reinterpret_cast<const uint4*>(src + tt * 128 + 16 * u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            *reinterpret_cast<uint4*>(lat_row + tt * 16384 + ((u ^ jr) << 4)) = v[u];
                    }
                    if (tt == 3 && kRope && okw) {
                        // RoPE values into tensor memory (A of the RoPE MMA, read after tile 3)
                        tc::fence_after_sync();
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint32_t rv[16];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const uint4 x = present ? *reinterpret_cast<const uint4*>(src + kTailOff + 64 * half + 16 * u)
                                                        : make_uint4(0u, 0u, 0u, 0u);
                                rv[4 * u] = x.x; rv[4 * u + 1] = x.y; rv[4 * u + 2] = x.z; rv[4 * u + 3] = x.w;
                            }
                            tc::tmem_st16(tmem + lane_base + C::kColRope + 16 * half, rv);
                        }
                        tc::wait_st();
                    }
                    fence_proxy_async_smem();
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&canon[tt]);
                }
                if (lane == 0) release_slot(&rel[slot]);

                // ---- scores: tile partials times the row's scales, plus RoPE ----
                float s[NH];
#pragma unroll
                for (int h = 0; h < NH; ++h) s[h] = 0.0f;
#pragma unroll 1
                for (int part = 0; part < C::kParts; ++part, ++sk) {
                    const uint32_t ss = sk % C::kSlots, su = sk / C::kSlots;
                    okw = okw && wait_or_abort(&s_full[ss], su & 1, abort_flag);
                    okw = __all_sync(0xffffffffu, okw);
                    tc::fence_after_sync();
                    if (okw) {
                        const uint32_t base = tmem + lane_base + C::kColS + ss * NQ;
                        if (part < 4) {
                            const float scp = part == 0 ? sc[0] : part == 1 ? sc[1] : part == 2 ? sc[2] : sc[3];
#pragma unroll
                            for (int i = 0; i < NH / 16; ++i) {
                                uint32_t vh[16], vl[16];
                                tc::tmem_ld16(base + 16 * i, vh);
                                tc::tmem_ld16(base + NH + 16 * i, vl);
                                tc::wait_ld();
#pragma unroll
                                for (int h = 0; h < 16; ++h)
                                    s[16 * i + h] = fmaf(scp, __uint_as_float(vh[h]) + __uint_as_float(vl[h]), s[16 * i + h]);
                            }
                        } else {
                            // latent part back in q units (2^k), then the RoPE partial
#pragma unroll
                            for (int i = 0; i < NH / 16; ++i) {
                                uint32_t vr[16];
                                tc::tmem_ld16(base + 16 * i, vr);
                                tc::wait_ld();
#pragma unroll
                                for (int h = 0; h < 16; ++h)
                                    s[16 * i + h] = fmaf(s[16 * i + h], qexp[16 * i + h], __uint_as_float(vr[h]));
                            }
                        }
                    }
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s_free[ss]);
                }
                if (bar_sync_or(1, kComputeThreads, !okw)) { ok = false; break; }
                bool need = false;
                float pv[NH];
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    const float sv = kRope ? s[h] : s[h] * qexp[h];
                    s[h] = present ? sv * a.sm_scale_log2 : -INFINITY;
                    need |= s[h] > m_ref[h] + kSlack;
                    pv[h] = ex2_approx(s[h] - m_ref[h]);
                }
                {
                    // Would any P of this block pass the largest E4M3?
                    const float4* pf4 = reinterpret_cast<const float4*>(tau_s + tb * 8 * NH + 4 * NH);
#pragma unroll
                    for (int tt = 0; tt < 4; ++tt) {
#pragma unroll
                        for (int h4 = 0; h4 < NH / 4; ++h4) {
                            const float4 f = pf4[tt * (NH / 4) + h4];
                            const float st = sc[tt];
                            need |= (pv[4 * h4] * st * f.x > kPMax) | (pv[4 * h4 + 1] * st * f.y > kPMax) |
                                    (pv[4 * h4 + 2] * st * f.z > kPMax) | (pv[4 * h4 + 3] * st * f.w > kPMax);
                        }
                    }
                }
                if (bar_sync_or(1, kComputeThreads, need)) {
                    // (1) per-head offsets from this block's score maxima
                    float* rw = red + w * NH;
#pragma unroll
                    for (int h = 0; h < NH; ++h) {
                        const float mh = warp_max_redux(s[h]);
                        if (lane == 0) rw[h] = mh;
                    }
                    bar_sync_or(1, kComputeThreads, false);
                    float alpha[NH];
#pragma unroll
                    for (int h = 0; h < NH; ++h) {
                        const float bm = fmaxf(fmaxf(red[h], red[NH + h]), fmaxf(red[2 * NH + h], red[3 * NH + h]));
                        const float mn = (bm > m_ref[h] + kSlack) ? bm : m_ref[h];
                        alpha[h] = (mn == m_ref[h]) ? 1.0f : ex2_approx(m_ref[h] - mn);
                        m_ref[h] = mn;
                        l_part[h] *= alpha[h];
                        pv[h] = ex2_approx(s[h] - mn);
                    }
                    bar_sync_or(1, kComputeThreads, false);     // red[] read
                    // (2) per-(tile, head) maxima of p * scale -> normalisers tau
#pragma unroll 1
                    for (int tt = 0; tt < 4; ++tt) {
#pragma unroll
                        for (int h = 0; h < NH; ++h) {
                            const float bx = warp_max_nonneg(pv[h] * sc[tt]);
                            if (lane == 0) red[(w * 4 + tt) * NH + h] = bx;
                        }
                    }
                    bar_sync_or(1, kComputeThreads, false);
                    const float* tau_old = tau_s + tb * 8 * NH;
                    float* tau_new = tau_s + (tb ^ 1) * 8 * NH;
                    if (j < 4 * NH) {
                        const int tt = j / NH, hj = j % NH;
                        float a_h = 1.0f;
#pragma unroll
                        for (int h = 0; h < NH; ++h)
                            if (h == hj) a_h = alpha[h];
                        const float bx = fmaxf(fmaxf(red[(0 * 4 + tt) * NH + hj], red[(1 * 4 + tt) * NH + hj]),
                                               fmaxf(red[(2 * 4 + tt) * NH + hj], red[(3 * 4 + tt) * NH + hj]));
                        const float tn = fmaxf(fmaxf(tau_old[j] * a_h, bx), 0.0f);
                        tau_new[j] = tn;
                        tau_new[4 * NH + j] = tn > 0.0f ? kPTarget / tn : 0.0f;
                        // O^T columns h (P_hi part) and NH + h (P_lo part) of tile tt
                        const float f = tn > 0.0f ? a_h * (tau_old[j] / tn) : 0.0f;
                        fac_s[tt * NP + hj] = f;
                        fac_s[tt * NP + NH + hj] = f;
                    }
                    bar_sync_or(1, kComputeThreads, false);
                    if (kb > 0) {
                        // O^T (complete up to the previous block: every tile's PV of it
                        // was waited for above) in the new units: column h of tile t
                        // times alpha_h * tau_old / tau_new.
                        tc::fence_after_sync();
#pragma unroll 1
                        for (int ci = 0; ci < 4 * NP / 16; ++ci) {
                            uint32_t ov[16];
                            const uint32_t addr = tmem + lane_base + C::kColO + 16 * ci;
                            tc::tmem_ld16(addr, ov);
                            const float4* f4 = reinterpret_cast<const float4*>(fac_s + 16 * ci);
                            tc::wait_ld();
#pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4) {
                                const float4 f = f4[c4];
                                ov[4 * c4 + 0] = __float_as_uint(__uint_as_float(ov[4 * c4 + 0]) * f.x);
                                ov[4 * c4 + 1] = __float_as_uint(__uint_as_float(ov[4 * c4 + 1]) * f.y);
                                ov[4 * c4 + 2] = __float_as_uint(__uint_as_float(ov[4 * c4 + 2]) * f.z);
                                ov[4 * c4 + 3] = __float_as_uint(__uint_as_float(ov[4 * c4 + 3]) * f.w);
                            }
                            tc::tmem_st16(addr, ov);
                        }
                        tc::wait_st();
                    }
                    tb ^= 1;
                    bar_sync_or(1, kComputeThreads, false);     // red[] and tau_old read
                }
                // ---- P = p * scale * 2 / tau as E4M3 hi + lo, tile by tile (the B operand of PV) ----
#pragma unroll
                for (int h = 0; h < NH; ++h) l_part[h] += pv[h];
                const float* pf_cur = tau_s + tb * 8 * NH + 4 * NH;
#pragma unroll 1
                for (int tt = 0; tt < 4; ++tt) {
                    const float st = tt == 0 ? sc[0] : tt == 1 ? sc[1] : tt == 2 ? sc[2] : sc[3];
#pragma unroll
                    for (int hc = 0; hc < NH / 16; ++hc) {
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int h = 16 * hc + 4 * i;
                            const float4 f = reinterpret_cast<const float4*>(pf_cur + tt * NH + h)[0];
                            const uint32_t s0 = split_pair(pv[h] * st * f.x, pv[h + 1] * st * f.y);
                            const uint32_t s1 = split_pair(pv[h + 2] * st * f.z, pv[h + 3] * st * f.w);
                            hi[i] = (s0 & 0xFFFFu) | (s1 << 16);
                            lo[i] = (s0 >> 16) | (s1 & 0xFFFF0000u);
                        }
                        uint8_t* pt = p_row + tt * (NP * 128);
                        *reinterpret_cast<uint4*>(pt + hc * 2048) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4*>(pt + (NH / 16 + hc) * 2048) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                    fence_proxy_async_smem();
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ptile[tt]);
                }
            }
            if (!ok) break;
            if (nblk > 0) ++qn;

            // ---- piece epilogue: l over the 128 rows, then O^T * tau / (2 l) ----
            bool okw = true;
#pragma unroll 1
            for (int tt = 0; tt < 4 && nblk > 0; ++tt)
                okw = okw && wait_or_abort(&pvdone[tt], (gbk - 1) & 1, abort_flag);
            okw = __all_sync(0xffffffffu, okw);
            if (bar_sync_or(1, kComputeThreads, !okw)) { ok = false; break; }
            tc::fence_after_sync();
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                const float lh = warp_sum(l_part[h]);
                if (lane == 0) red[w * NH + h] = lh;
            }
            bar_sync_or(1, kComputeThreads, false);
            float lsum = 0.0f, mref_j = 0.0f;                // thread j < NH: head j's l and offset
            if (j < NH) {
                lsum = (red[j] + red[NH + j]) + (red[2 * NH + j] + red[3 * NH + j]);
#pragma unroll
                for (int h = 0; h < NH; ++h)
                    if (h == j) mref_j = m_ref[h];
            }
            // per (tile, head): tau / (2 l), in fac_s
            if (j < 4 * NH) {
                const int hj = j % NH;
                const float lh = (red[hj] + red[NH + hj]) + (red[2 * NH + hj] + red[3 * NH + hj]);
                fac_s[j] = lh > 0.0f ? tau_s[tb * 8 * NH + j] / (kPTarget * lh) : 0.0f;
            }
            bar_sync_or(1, kComputeThreads, false);
#pragma unroll 1
            for (int tt = 0; tt < 4; ++tt) {
                float o[NH];
#pragma unroll
                for (int h = 0; h < NH; ++h) o[h] = 0.0f;
                if (nblk > 0) {
#pragma unroll
                    for (int i = 0; i < NH / 16; ++i) {
                        uint32_t vh[16], vl[16];
                        tc::tmem_ld16(tmem + lane_base + C::kColO + tt * NP + 16 * i, vh);
                        tc::tmem_ld16(tmem + lane_base + C::kColO + tt * NP + NH + 16 * i, vl);
                        tc::wait_ld();
#pragma unroll
                        for (int h = 0; h < 16; ++h)
                            o[16 * i + h] = (__uint_as_float(vh[h]) + __uint_as_float(vl[h])) * fac_s[tt * NH + 16 * i + h];
                    }
                }
                const int d = 128 * tt + j;
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    const int hh = hg * NH + h;
                    if (hh >= H) continue;
                    if (whole)
                        a.out[(static_cast<int64_t>(t) * H + hh) * kLatent + d] = __float2bfloat16_rn(o[h]);
                    else
                        a.ws_o[(out_slot * H + hh) * kLatent + d] = o[h];
                }
            }
            if (j < NH && hg * NH + j < H) {
                const float lse2 = lsum > 0.0f ? (mref_j + log2f(lsum)) * kLn2 : -INFINITY;
                const int hh = hg * NH + j;
                if (whole) a.lse[static_cast<int64_t>(t) * H + hh] = lse2;
                else a.ws_lse[out_slot * H + hh] = lse2;
            }
            tc::fence_before_sync();
            bar_sync_or(1, kComputeThreads, false);          // fac_s and red[] read before the next piece
        }
        if (!ok && j == 0) atomicOr(a.err, MLA_ERR_PIPELINE_TIMEOUT);
    }

    // ---- teardown: copies landed, MMAs done, tensor memory released ----
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        atomicOr(a.err, MLA_ERR_PIPELINE_TIMEOUT);
        for (int s = 0; s < C::kRS; ++s)
            if (issued[s] > 0) (void)mbar_wait_bounded(&full[s], static_cast<uint32_t>(issued[s] - 1) & 1);
        if (*q_issued > 0) (void)mbar_wait_bounded(q_full, static_cast<uint32_t>(*q_issued - 1) & 1);
    }
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ======================= 3. merge of split tokens =======================
// One CTA per (token, head); 128 threads x 4 output dims.
__global__ void __launch_bounds__(kMergeThreads)
mla_split_merge_kernel(const int32_t* __restrict__ prefix, const int32_t* __restrict__ ctl, const float* __restrict__ ws_o,
                       const float* __restrict__ ws_lse, int T, int H, __nv_bfloat16* __restrict__ out,
                       float* __restrict__ lse) {
    pdl_wait();
    const int64_t th = blockIdx.x;               // t * H + h
    const int t = static_cast<int>(th / H);
    const int h = static_cast<int>(th % H);
    const int G = ctl[0];
    const int64_t P = prefix[T];
    const int64_t p0 = prefix[t], p1 = prefix[t + 1];
    const int d = 4 * threadIdx.x;
    __nv_bfloat16* orow = out + th * kLatent + d;
    if (p1 == p0) {                              // no present entry: 0 and -inf
        *reinterpret_cast<uint2*>(orow) = make_uint2(0u, 0u);
        if (threadIdx.x == 0) lse[th] = -INFINITY;
        return;
    }
    auto range_of = [&](int64_t x) {
        int rr = static_cast<int>(x * G / P);
        while (rr + 1 < G && range_start(P, G, rr + 1) <= x) ++rr;
        while (rr > 0 && range_start(P, G, rr) > x) --rr;
        return rr;
    };
    const int r_lo = range_of(p0), r_hi = range_of(p1 - 1);
    if (r_lo == r_hi) return;                    // one CTA held the whole token and wrote it
    const bool first_is_t = token_of(prefix, T, range_start(P, G, r_lo)) == t;
    // lse of every piece first (independent loads), then the weighted sum in range order.
    constexpr int kMaxPieces = 8;
    float ls[kMaxPieces];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMaxPieces; ++i) {
        const int rr = r_lo + i;
        const int64_t slot = (rr == r_lo && !first_is_t) ? 2 * rr + 1 : 2 * rr;
        ls[i] = rr <= r_hi ? ws_lse[slot * H + h] : -INFINITY;
        mx = fmaxf(mx, ls[i]);
    }
    for (int rr = r_lo + kMaxPieces; rr <= r_hi; ++rr) mx = fmaxf(mx, ws_lse[(2 * static_cast<int64_t>(rr)) * H + h]);
    if (mx == -INFINITY) {
        *reinterpret_cast<uint2*>(orow) = make_uint2(0u, 0u);
        if (threadIdx.x == 0) lse[th] = -INFINITY;
        return;
    }
    float wsum = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int rr = r_lo; rr <= r_hi; ++rr) {
        const int i = rr - r_lo;
        const int64_t slot = (rr == r_lo && !first_is_t) ? 2 * rr + 1 : 2 * rr;
        float l = -INFINITY;
#pragma unroll
        for (int k = 0; k < kMaxPieces; ++k)
            if (k == i) l = ls[k];
        if (i >= kMaxPieces) l = ws_lse[slot * H + h];
        if (l == -INFINITY) continue;
        const float wgt = expf(l - mx);
        wsum += wgt;
        const float4 v = *reinterpret_cast<const float4*>(ws_o + (slot * H + h) * kLatent + d);
        acc.x += wgt * v.x; acc.y += wgt * v.y; acc.z += wgt * v.z; acc.w += wgt * v.w;
    }
    const float inv = 1.0f / wsum;
    *reinterpret_cast<uint2*>(orow) = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv),
                                                 pack_bf16x2(acc.z * inv, acc.w * inv));
    if (threadIdx.x == 0) lse[th] = mx + logf(wsum);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Plan {
    int NH, HG, G, balanced;
    size_t off_comp, off_cnt, off_prefix, off_ctl, off_qc, off_ws_o, off_ws_lse, total;
};

Plan make_plan(int T, int H, int W, int sms) {
    Plan p{};
    p.NH = H <= 16 ? 16 : 32;
    p.HG = (H + p.NH - 1) / p.NH;
    p.G = max(1, sms / p.HG);
    p.balanced = T <= kMaxBalancedT ? 1 : 0;
    size_t off = 0;
    p.off_comp = off; off = align256(off + static_cast<size_t>(T) * static_cast<size_t>(W) * 4);
    p.off_cnt = off; off = align256(off + static_cast<size_t>(T) * 4);
    p.off_prefix = off; off = align256(off + (static_cast<size_t>(T) + 1) * 4);
    p.off_ctl = off; off = align256(off + 16);
    p.off_qc = off; off = align256(off + static_cast<size_t>(T) * p.HG * q_block_bytes(p.NH));
    p.off_ws_o = off;
    if (p.balanced) off = align256(off + static_cast<size_t>(2) * p.G * H * kLatent * 4);
    p.off_ws_lse = off;
    if (p.balanced) off = align256(off + static_cast<size_t>(2) * p.G * H * 4);
    p.total = off;
    return p;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <int NH, bool kRope>
int launch_main(const DecodeArgs& a, int ctas, cudaStream_t st) {
    using C = Cfg<NH, kRope>;
    if (!mla_host::max_dynamic_smem(reinterpret_cast<const void*>(mla_sparse_decode_kernel<NH, kRope>), C::kSmemAlloc))
        return MLA_ECUDA;
    return launch_pdl(mla_sparse_decode_kernel<NH, kRope>, dim3(ctas), dim3(kThreads), C::kSmemAlloc, st, a) ==
                   cudaSuccess
               ? MLA_OK
               : MLA_ECUDA;
}

struct PageArgs {
    const int32_t* block_table;
    const int32_t* token_seq;
    int bt_pages, n_seq, page_size;
};

int launch_decode(const void* q_bf16, int T, int H, int d_qk, mla_kv_cache_t kv, const int32_t* topk_idx, int W,
                  float sm_scale, void* out_bf16, float* lse, void* workspace, size_t workspace_bytes, void* stream,
                  const PageArgs& pg) {
    if (T < 0 || W < 0 || kv.num_slots < 0 || !std::isfinite(sm_scale)) return MLA_EINVAL;
    if (kv.row_bytes != MLA_ROW_BYTES && kv.row_bytes != MLA_ROW_BYTES_NOPE) return MLA_EINVAL;
    if (d_qk != kLatent && d_qk != kLatent + kRope) return MLA_EUNSUPPORTED;
    if (kv.row_bytes == MLA_ROW_BYTES_NOPE && d_qk != kLatent) return MLA_EUNSUPPORTED;   // no tail to read
    if (H < 1 || H > 128) return MLA_EUNSUPPORTED;
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
    const Plan p = make_plan(T, H, W, sms);
    if (workspace == nullptr || workspace_bytes < p.total || !aligned16(workspace)) return MLA_ENOWORKSPACE;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t* comp = reinterpret_cast<int32_t*>(ws + p.off_comp);
    int32_t* cnt = reinterpret_cast<int32_t*>(ws + p.off_cnt);
    if (launch_pdl(mla_topk_compact_kernel, dim3(T), dim3(kCompactThreads), 0, st, topk_idx, W,
                   static_cast<int64_t>(kv.num_slots), pg.block_table, pg.token_seq, pg.bt_pages, pg.n_seq,
                   pg.page_size, comp, cnt, err, static_cast<const __nv_bfloat16*>(q_bf16), H, d_qk, p.NH, p.HG,
                   ws + p.off_qc) != cudaSuccess)
        return MLA_ECUDA;

    DecodeArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q_bf16);
    a.cache = static_cast<const uint8_t*>(kv.data);
    a.row_bytes = kv.row_bytes;
    a.comp = comp;
    a.cnt = cnt;
    a.qc = ws + p.off_qc;
    a.out = static_cast<__nv_bfloat16*>(out_bf16);
    a.lse = lse;
    a.ws_o = reinterpret_cast<float*>(ws + p.off_ws_o);
    a.ws_lse = reinterpret_cast<float*>(ws + p.off_ws_lse);
    a.ws_prefix = reinterpret_cast<int32_t*>(ws + p.off_prefix);
    a.ws_ctl = reinterpret_cast<int32_t*>(ws + p.off_ctl);
    a.err = err;
    a.T = T; a.H = H; a.d_qk = d_qk; a.W = W; a.HG = p.HG; a.G = p.G; a.balanced = p.balanced;
    a.sm_scale_log2 = sm_scale * kLog2e;
    const int ctas = p.G * p.HG;
    const bool rope = d_qk == kLatent + kRope;
    int rc;
    if (p.NH == 16) rc = rope ? launch_main<16, true>(a, ctas, st) : launch_main<16, false>(a, ctas, st);
    else rc = rope ? launch_main<32, true>(a, ctas, st) : launch_main<32, false>(a, ctas, st);
    if (rc != MLA_OK || cudaGetLastError() != cudaSuccess) return MLA_ECUDA;
    if (p.balanced) {
        if (launch_pdl(mla_split_merge_kernel, dim3(static_cast<unsigned>(static_cast<int64_t>(T) * H)), dim3(kMergeThreads), 0, st,
                       static_cast<const int32_t*>(a.ws_prefix), static_cast<const int32_t*>(a.ws_ctl),
                       static_cast<const float*>(a.ws_o), static_cast<const float*>(a.ws_lse), T, H, a.out, a.lse) !=
            cudaSuccess)
            return MLA_ECUDA;
    }
    return MLA_OK;
}

}  // namespace

extern "C" size_t mla_sparse_decode_workspace_bytes(int T, int H, int W) {
    if (T <= 0 || H <= 0 || H > 128 || W < 0) return 0;
    const int sms = mla_host::sm_count();
    if (sms <= 0) return 0;
    return make_plan(T, H, W, sms).total;
}

extern "C" int mla_sparse_decode(const void* q_bf16, int T, int H, int d_qk, mla_kv_cache_t kv,
                                 const int32_t* topk_idx, int W, float sm_scale, void* out_bf16,
                                 float* lse, void* workspace, size_t workspace_bytes, void* stream) {
    const PageArgs none{nullptr, nullptr, 0, 0, 0};
    return launch_decode(q_bf16, T, H, d_qk, kv, topk_idx, W, sm_scale, out_bf16, lse, workspace, workspace_bytes,
                         stream, none);
}

extern "C" int mla_sparse_decode_paged(const void* q_bf16, int T, int H, int d_qk, mla_kv_cache_t kv,
                                       const int32_t* topk_pos, int W, const int32_t* block_table, int n_seq,
                                       int max_pages, const int32_t* token_seq, int page_size, float sm_scale,
                                       void* out_bf16, float* lse, void* workspace, size_t workspace_bytes,
                                       void* stream) {
    if (page_size <= 0 || max_pages <= 0 || n_seq <= 0 || block_table == nullptr ||
        (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(token_seq) & 3u))
        return MLA_EINVAL;
    const PageArgs pg{block_table, token_seq, max_pages, n_seq, page_size};
    return launch_decode(q_bf16, T, H, d_qk, kv, topk_pos, W, sm_scale, out_bf16, lse, workspace, workspace_bytes,
                         stream, pg);
}
