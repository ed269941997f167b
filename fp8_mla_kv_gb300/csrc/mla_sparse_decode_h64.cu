// mla_sparse_decode for 64 heads per CTA on the fifth-generation tensor cores.
//
// Computes what mla_sparse_decode computes (the decode statement in the C header,
// with absent entries removed before anything is fetched: sglang PR #39288, Root
// cause; sglang PR #47013, Motivation), for head counts that are a multiple of 64:
// one CTA per (token, group of 64 heads, split of the list). All 64 heads of a
// token share one gather and one E4M3 -> f16 conversion of every row, where the
// 16-head kernel repeats both for each group of 16 heads.
//
// Roles (12 warps): warps 0-7 are two warpgroups of math threads, warp 8 owns the
// tensor memory and issues every tcgen05.mma from one thread, warps 9-11 copy
// rows (one cp.async.bulk per listed row) into a ring of four 32-row stages.
// A block is 64 listed rows (two stages): warpgroup g converts the rows of
// stage g and folds the scores of keys 32g .. 32g+31.
//
// Per 64-row block, with q (64 heads x 576) resident in shared memory as f16
// (latent; exact after an exponent-only per-head shift) and bf16 (RoPE):
//   QK   latent tile t = 0..3: S_t[64 heads x 64 keys] = q_t . K_t^T on
//        tcgen05.mma M=64 N=64 (f16, fp32 in tensor memory), K_t = the exact f16
//        values of the E4M3 codes; RoPE: S_r = q_r . R^T (bf16 operands). The
//        math threads read each S_t back as soon as it is done and fold it:
//        s = S_r + sum_t scale_t(key) * S_t, so every product is exact before
//        fp32 accumulation, as in the 16-head kernel. Two S buffers in rotation.
//   softmax  online, per head, in the threads that hold the head's scores
//        (exp2, sm_scale * log2 e folded in; the offset moves only when a block
//        maximum runs more than kRescaleSlack above it, so p <= 2^8 fits f16).
//   PV   O^T[512 dims x 64 heads] in tensor memory (dims as M = 128 per latent
//        tile, heads as N = 64): O^T_t += V'_t^T . P^T, where V'_t = code *
//        scale_t(key) / sigma_t in f16 (sigma_t = running maximum of tile t's row
//        scales; O^T_t rescaled in tensor memory when it moves) and P^T the f16
//        probabilities, both from shared memory.
// The epilogue reads O^T back, multiplies by sigma_t / l and writes bf16 out and
// lse (or the normalised fp32 partial of a split, merged afterwards in split
// order by the 16-head kernel's merge).
//
// Every wait is bounded; a wait that runs out raises MLA_ERR_PIPELINE_TIMEOUT,
// sets a CTA-wide abort flag that ends every other wait, and the CTA leaves
// without writing its outputs once its copies and MMAs in flight have landed.
#include <cfloat>
#include <climits>
#include <cmath>

#include "mla_device.cuh"
#include "mla_decode_internal.h"

namespace {

using namespace mla;

constexpr int kHG = 64;                          // heads per CTA (M of the QK MMA)
constexpr int kMathWarps = 8;
constexpr int kMathThreads = kMathWarps * 32;    // two warpgroups
constexpr int kMmaWarp = 8;
constexpr int kProd0 = 9;                        // first copy-issuing warp
constexpr int kProds = 3;                        // 12 warps: 3 per scheduler, so 168 registers a thread
constexpr int kThreads = (kProd0 + kProds) * 32; // 384
constexpr int kStageRows = 32;
constexpr int kBlockRows = 64;                   // keys per block (N of the QK MMA)
constexpr int kStages = 4;
constexpr int kListMax = 2304;
constexpr int kPerThread = (kListMax + kThreads - 1) / kThreads;
constexpr float kRescaleSlack = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

// Shared memory (offsets from a 1024-byte aligned base). Operand tiles use the
// 128-byte swizzled K-major layout: rows of 64 16-bit values (128 B) in 8-row
// groups of 1 KB, the 16-byte unit u of row r stored at unit u ^ (r & 7); a
// tile wider than 64 values is a sequence of such 64-column chunks.
constexpr int kOffQ = 0;                                   // q latent: 4 tiles x 64 heads x 128 f16
constexpr int kOffQr = kOffQ + 4 * 16384;                  // q RoPE: 64 heads x 64 bf16
constexpr int kNumBuf = 3;                                 // operand buffers: 64 keys x 128 f16 each
constexpr int kOffBuf = kOffQr + 8192;
constexpr int kOffP = kOffBuf + kNumBuf * 16384;           // P^T: 64 heads x 64 keys f16
constexpr int kOffRing = kOffP + 8192;                     // 4 stages x 32 rows x 656 B
constexpr int kStageBytes = kStageRows * kRowBytes;        // 20,992
constexpr int kOffList = kOffRing + kStages * kStageBytes;
constexpr int kOffBars = kOffList + kListMax * 4;
// barriers: full[4], empty[4], kready[3], bdone[3], sready[3], sfree[3], scready[2], pready, pvdone, fin
constexpr int kNumBars = 25;
constexpr int kOffSmall = kOffBars + 32 * 8;
// small arrays (floats / ints). Per-block data is double-buffered by block parity.
constexpr int kOffRowf = kOffSmall;                        // [64] sm_scale * log2 e * 2^k per head
constexpr int kOffAlpha = kOffRowf + 64 * 4;               // [64] per-head O rescale; epilogue: 1 / l
constexpr int kOffLsum = kOffAlpha + 64 * 4;               // [64] epilogue: lse per head
constexpr int kOffSc = kOffLsum + 64 * 4;                  // [2 parity][4 tiles][64 keys] row scales
constexpr int kOffSmax = kOffSc + 2 * 4 * 64 * 4;          // [2 parity][2 row halves][4 tiles] scale maxima
constexpr int kOffWcount = kOffSmax + 2 * 2 * 4 * 4;       // [16] per-warp counts of the compaction
constexpr int kOffMisc = kOffWcount + 16 * 4;              // tmem base, abort flag, issued[3], converter failed, failed[2 parity]
constexpr int kSmemUsed = kOffMisc + 8 * 4;
constexpr int kSmemTotal = kSmemUsed + 1024;               // room to align the base
static_assert(kSmemTotal <= 232448, "shared memory");
static_assert(kNumBars <= 32, "barrier space");

// Tensor memory columns: O^T tile t at 64t (t = 0..3), three S slots at 256, 320, 384.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 256;

// ---- tcgen05 wrappers ----
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// kind::f16 instruction descriptor: fp32 D, A/B format (0 f16, 1 bf16), majors, M, N.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t fmt, bool a_mn, bool b_mn, uint32_t m, uint32_t n) {
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(a_mn) << 15) |
           (static_cast<uint32_t>(b_mn) << 16) | ((n >> 3) << 17) | ((m >> 4) << 24);
}
constexpr uint32_t kIdQK = idesc_f16(0, false, false, 64, 64);     // S = q_t . K_t^T
constexpr uint32_t kIdQR = idesc_f16(1, false, false, 64, 64);     // S_r = q_r . R^T (bf16)
constexpr uint32_t kIdPV = idesc_f16(0, true, false, 128, 64);     // O^T_t += V'_t^T . P^T

__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d), "l"(a), "l"(b), "r"(id), "r"(static_cast<uint32_t>(acc)) : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

#define MLA_R16 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}"
#define MLA_O16(r) "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), \
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
// 16 lanes x 256 bits: thread t gets lanes t/4 and t/4 + 8, columns 8j + 2(t%4) + {0,1}
// in r[4j], r[4j+1] (lane t/4) and r[4j+2], r[4j+3] (lane t/4 + 8).
#define MLA_R32 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}"
// The same, eight times (64 columns): r[4j .. 4j+3] for columns 8j .. 8j+7.
__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x8.b32 " MLA_R32 ", [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
                   "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}
// 32 lanes x 32 bits, 16 columns: thread t gets lane t, columns c .. c+15.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 " MLA_R16 ", [%16];" : MLA_O16(r) : "r"(taddr));
}
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
           "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Byte offset of 16-byte unit u (0 .. 8*chunks-1) of row r in a swizzled tile of `rows` rows.
__device__ __forceinline__ uint32_t swz(int rows, int r, int u) {
    return static_cast<uint32_t>((u >> 3) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + (((u & 7) ^ (r & 7)) << 4));
}

// A bounded wait that also ends as soon as another role has given up (abort flag).
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (int i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15) == 15) {
            if (*abort_flag) return false;
            if (clock64() - t0 > kWaitCycles) {
                *abort_flag = 1;
                return false;
            }
        }
    }
}
// The same wait taken by every lane of a warp, with one answer for the warp
// (tcgen05.ld / st that follow must be issued by the whole warp together).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    const bool ok = wait_or_abort(bar, parity, abort_flag);
    return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

template <bool kRopeOn>
__global__ void __launch_bounds__(kThreads, 1)
mla_sparse_decode_h64_kernel(const mla_host::DecodeCall args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    int* list = reinterpret_cast<int*>(smem + kOffList);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    uint64_t* full = bars;            // [4] stage landed (producer expect_tx + bulk copies)
    uint64_t* empty = bars + 4;       // [4] stage read by the converting warpgroup (4 warps)
    uint64_t* kready = bars + 8;      // [3] operand buffer written (4 converting warps)
    uint64_t* bdone = bars + 11;      // [3] the MMAs that read an operand buffer are done (commit)
    uint64_t* sready = bars + 14;     // [3] QK into an S slot done (commit)
    uint64_t* sfree = bars + 17;      // [3] S slot read back (4 softmax warps)
    uint64_t* scready = bars + 20;    // [2] a block's row scales and scale maxima written (4 converting warps)
    uint64_t* pready = bars + 22;     // P^T written, O^T rescaled (4 softmax warps)
    uint64_t* pvdone = bars + 23;     // a block's PV done (commit)
    uint64_t* fin = bars + 24;        // every MMA done (commit, used on the way out)
    float* rowf_s = reinterpret_cast<float*>(smem + kOffRowf);
    float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);
    float* lsum_s = reinterpret_cast<float*>(smem + kOffLsum);
    float* sc_s = reinterpret_cast<float*>(smem + kOffSc);
    float* smax_s = reinterpret_cast<float*>(smem + kOffSmax);
    int* wcount = reinterpret_cast<int*>(smem + kOffWcount);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
    int* issued_s = reinterpret_cast<int*>(smem + kOffMisc + 8);

    // blockIdx.x = (T - 1 - t) * head_groups + hg: tokens from the last to the
    // first (in a causal batch the later lists are the longest); no result
    // depends on the order.
    const int head_groups = args.H / kHG;
    const int t = args.T - 1 - static_cast<int>(blockIdx.x / head_groups);
    const int hg = static_cast<int>(blockIdx.x % head_groups);
    const int split = blockIdx.y;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr uint32_t kRowRead = kRopeOn ? kRowBytes : kNopeReadBytes;

    const bool by_rank = args.rank_chunk > 0;
    const int p0 = by_rank ? 0 : split * args.split_len;
    const int p1 = by_rank ? args.W : min(args.W, p0 + args.split_len);
    const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(args.q) +
                              (static_cast<int64_t>(t) * args.H + hg * kHG) * args.d_qk;
    {
        // Before waiting for the previous kernel: bring this CTA's positions and
        // q rows into L2 (prefetches read nothing into the kernel).
        const char* lb = reinterpret_cast<const char*>(args.topk + static_cast<int64_t>(t) * args.W + p0);
        const int lines = (max(0, p1 - p0) * 4 + 127) / 128;
        for (int i = threadIdx.x; i < lines; i += kThreads) prefetch_l2(lb + 128 * i);
        const int qlines = (kHG * args.d_qk * 2 + 127) / 128;
        for (int i = threadIdx.x; i < qlines; i += kThreads) prefetch_l2(reinterpret_cast<const char*>(qg) + 128 * i);
    }
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 4);
        }
        for (int i = 0; i < kNumBuf; ++i) {
            mbar_init(&kready[i], 4);
            mbar_init(&bdone[i], 1);
            mbar_init(&sready[i], 1);
            mbar_init(&sfree[i], 4);
        }
        for (int i = 0; i < 2; ++i) mbar_init(&scready[i], 4);
        mbar_init(pready, 4);
        mbar_init(pvdone, 1);
        mbar_init(fin, 1);
        *abort_flag = 0;
        reinterpret_cast<int*>(smem + kOffMisc)[5] = 0;
        reinterpret_cast<int*>(smem + kOffMisc)[6] = 0;
        reinterpret_cast<int*>(smem + kOffMisc)[7] = 0;
        for (int p = 0; p < kProds; ++p) issued_s[p] = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }

    // ---- 0. q loads (math threads: 4 per head, 18 units of 8 values each), issued first ----
    // Units 0..63 are the latent (tile u / 16, unit u % 16 of the tile), 64..71 RoPE.
    const int qh = threadIdx.x >> 2;          // head (math threads)
    const int qpart = threadIdx.x & 3;
    constexpr int kQUnits = 18;
    uint4 qv[kQUnits];
    if (warp < kMathWarps) {
        const int nunits = args.d_qk / 8;     // 72 or 64
        const __nv_bfloat16* qrow = qg + static_cast<int64_t>(qh) * args.d_qk;
#pragma unroll
        for (int k = 0; k < kQUnits; ++k) {
            const int u = qpart * kQUnits + k;
            qv[k] = (u < nunits) ? ld_nc_v4(qrow + 8 * u) : make_uint4(0u, 0u, 0u, 0u);
        }
    }

    // ---- 1. compact the present entries of this CTA's positions (all threads) ----
    const int per = (max(0, p1 - p0) + kThreads - 1) / kThreads;     // <= kPerThread
    const int32_t* trow = args.topk + static_cast<int64_t>(t) * args.W + p0 + threadIdx.x * per;
    const int mine = max(0, min(per, p1 - (p0 + static_cast<int>(threadIdx.x) * per)));
    int idxv[kPerThread];
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) idxv[k] = (k < mine) ? __ldg(trow + k) : -1;
    if (args.page_size > 0) {
        // Positions -> slots through the block table (vLLM PR #55277, Purpose
        // item 2): a negative position or an unassigned page is absent; a
        // position past the table is absent and flagged.
        const int sq = args.token_seq ? __ldg(args.token_seq + t) : 0;
        const bool seq_ok = sq >= 0 && sq < args.n_seq;
        const int32_t* bt = args.block_table + static_cast<int64_t>(seq_ok ? sq : 0) * args.bt_pages;
#pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            const int pos = idxv[k];
            if (pos < 0) continue;
            const int page = pos / args.page_size;
            if (!seq_ok || page >= args.bt_pages) {
                atomicOr(args.err, MLA_ERR_DECODE_INDEX_RANGE);
                idxv[k] = -1;
                continue;
            }
            const int phys = __ldg(bt + page);
            const int64_t slot = static_cast<int64_t>(phys) * args.page_size + (pos - page * args.page_size);
            idxv[k] = (phys < 0) ? -1 : static_cast<int>(min(slot, static_cast<int64_t>(INT32_MAX)));
        }
    }
    int cnt = 0;
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        const int idx = idxv[k];
        const bool valid = idx > 0 && static_cast<int64_t>(idx) < args.num_slots;
        if (idx > 0 && !valid) atomicOr(args.err, MLA_ERR_DECODE_INDEX_RANGE);
        idxv[k] = valid ? idx : 0;
        cnt += valid ? 1 : 0;
    }
    int incl = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
    }
    if (lane == 31) wcount[warp] = incl;
    __syncthreads();
    int off = incl - cnt, n_valid = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        const int cw = wcount[w];
        off += (w < warp) ? cw : 0;
        n_valid += cw;
    }
#pragma unroll
    for (int k = 0; k < kPerThread; ++k)
        if (idxv[k] != 0) list[off++] = idxv[k];
    int lbase = 0;
    if (by_rank) {
        const int shares = min(args.nsplit, max(1, (n_valid + args.rank_chunk - 1) / args.rank_chunk));
        const int len = (n_valid + shares - 1) / shares;
        lbase = min(n_valid, split * len);
        n_valid = min(n_valid, lbase + len) - lbase;
    }
    const int nblk = (n_valid + kBlockRows - 1) / kBlockRows;

    // ---- 2. q into shared memory (math threads): exponent-only shift per head so
    // that |q| < 2^15 in f16, the same power of two on the RoPE part; undone on
    // the scores through rowf. ----
    if (warp < kMathWarps) {
        float qm = 0.0f;
#pragma unroll
        for (int k = 0; k < kQUnits; ++k) {
            const uint32_t w4[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) qm = fmaxf(qm, fmaxf(fabsf(bf16lo(w4[i])), fabsf(bf16hi(w4[i]))));
        }
        qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, 1));
        qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, 2));
        int e = 0;
        frexpf(qm, &e);                        // qm < 2^e
        const int ks = (e > 15) ? (e - 15) : 0;
        const float qdown = ldexpf(1.0f, -ks);
        if (qpart == 0) rowf_s[qh] = args.sm_scale_log2 * ldexpf(1.0f, ks);
#pragma unroll
        for (int k = 0; k < kQUnits; ++k) {
            const int u = qpart * kQUnits + k;
            const uint32_t w4[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
            uint4 o;
            uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
            if (u < 64) {
#pragma unroll
                for (int i = 0; i < 4; ++i) ow[i] = pack_f16x2(bf16lo(w4[i]) * qdown, bf16hi(w4[i]) * qdown);
                *reinterpret_cast<uint4*>(smem + kOffQ + (u >> 4) * 16384 + swz(64, qh, u & 15)) = o;
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) ow[i] = pack_bf16x2(bf16lo(w4[i]) * qdown, bf16hi(w4[i]) * qdown);
                *reinterpret_cast<uint4*>(smem + kOffQr + swz(64, qh, u - 64)) = o;
            }
        }
    }
    fence_proxy_async_smem();      // q is read by the tensor cores (async proxy)
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = smem_u32(smem);

    if (warp >= kProd0) {
        // ---- producers: warp kProd0 + p issues stages p, p + 3, ... (stage i = rows
        // 32i .. 32i+31 of the list, into ring slot i % 4; lane j copies row j) ----
        const int p = warp - kProd0;
        const int nst = 2 * nblk;
        int cntp = 0;
        for (int si = p; si < nst; si += kProds, ++cntp) {
            const int slot = si % kStages;
            if (si >= kStages && !warp_wait(&empty[slot], static_cast<uint32_t>(((si / kStages) - 1) & 1), abort_flag))
                break;
            uint8_t* dst = smem + kOffRing + slot * kStageBytes;
            const int n_r = max(0, min(kStageRows, n_valid - si * kStageRows));
            if (n_r < kStageRows) {
                // Rows past the end of the list load nothing: zeros (E4M3 0, scale 0).
                if (lane >= n_r) {
                    uint4* z = reinterpret_cast<uint4*>(dst + lane * kRowBytes);
                    for (int k = 0; k < kRowBytes / 16; ++k) z[k] = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(n_r) * kRowRead);
            __syncwarp();
            if (lane < n_r)
                bulk_g2s(dst + lane * kRowBytes,
                         args.cache + static_cast<int64_t>(list[lbase + si * kStageRows + lane]) * args.row_bytes,
                         kRowRead, &full[slot]);
        }
        if (lane == 0) issued_s[p] = cntp;
    } else if (warp == kMmaWarp) {
        // ---- one thread issues every MMA. MMA groups run in the order the
        // converting warps fill the operand buffers (group i reads buffer i % 3):
        // QK0, QK1 of block 0; then per block b: QK2, QK3, RoPE, QK0 and QK1 of
        // block b+1 (they run during block b's softmax), and after P^T(b) the four
        // PV of block b. QK group j writes S slot j % 3. ----
        if (lane == 0) {
            uint32_t nk[kNumBuf] = {0u, 0u, 0u}, nf[kNumBuf] = {0u, 0u, 0u}, np = 0u;
            int gi = 0, qi = 0;
            bool ok = true;
            const uint64_t dQ = sw128_desc(sbase + kOffQ, 16, 1024);
            const uint64_t dQr = sw128_desc(sbase + kOffQr, 16, 1024);
            const uint64_t dP = sw128_desc(sbase + kOffP, 16, 1024);
            // descriptor start addresses are in 16-byte units: adding off >> 4 moves the operand
            auto take_buf = [&]() {
                const int buf = gi % kNumBuf;
                ok = ok && wait_or_abort(&kready[buf], nk[buf]++ & 1u, abort_flag);
                return buf;
            };
            auto qk = [&](int tt) {                       // tt = 0..3 latent tile, 4 RoPE
                const int buf = take_buf();
                const int slot = qi % kNumBuf;
                if (qi >= kNumBuf) ok = ok && wait_or_abort(&sfree[slot], nf[slot]++ & 1u, abort_flag);
                if (!ok) return;
                tc_after();
                const uint64_t dB = sw128_desc(sbase + kOffBuf + buf * 16384, 16, 1024);
                const uint32_t d = tmem + kColS + 64 * slot;
                if (tt < 4) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t off = static_cast<uint64_t>(((ks >> 2) * 8192 + (ks & 3) * 32) >> 4);
                        umma(d, dQ + static_cast<uint64_t>((tt * 16384) >> 4) + off, dB + off, kIdQK, ks > 0);
                    }
                } else {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        umma(d, dQr + static_cast<uint64_t>(ks * 2), dB + static_cast<uint64_t>(ks * 2), kIdQR, ks > 0);
                }
                umma_commit(&sready[slot]);
                umma_commit(&bdone[buf]);
                ++gi;
                ++qi;
            };
            auto pv = [&](int tt, bool first) {
                const int buf = take_buf();
                if (!ok) return;
                tc_after();
                const uint64_t dV = sw128_desc(sbase + kOffBuf + buf * 16384, 8192, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    umma(tmem + 64 * tt, dV + static_cast<uint64_t>(ks * 128), dP + static_cast<uint64_t>(ks * 2), kIdPV,
                         !first || ks > 0);
                umma_commit(&bdone[buf]);
                ++gi;
            };
            if (nblk > 0) {
                qk(0);
                qk(1);
            }
            for (int b = 0; b < nblk && ok; ++b) {
                qk(2);
                qk(3);
                if (kRopeOn) qk(4);
                if (b + 1 < nblk) {
                    qk(0);
                    qk(1);
                }
                ok = ok && wait_or_abort(pready, np++ & 1u, abort_flag);
                if (!ok) break;
                tc_after();
                for (int tt = 0; tt < 4; ++tt) pv(tt, b == 0);
                umma_commit(pvdone);
            }
            // Every MMA issued has completed before tensor memory is read back or freed.
            umma_commit(fin);
            (void)mbar_wait_bounded(fin, 0);
        }
        __syncwarp();
    } else {
        // ---- math: warpgroup 0 folds the scores, runs the softmax and owns l, m;
        // warpgroup 1 converts every operand tile. Both keep the same sigma. ----
        const int g = warp >> 2;
        const int wq = warp & 3;                 // tensor-memory lane quarter
        const uint32_t lane_q = static_cast<uint32_t>(32 * wq) << 16;
        uint8_t* buf = smem + kOffBuf;
        uint8_t* pT = smem + kOffP;
        // failed waits of warpgroup 0, by the parity of the block whose barrier 1 reads them
        volatile int* fail_s = reinterpret_cast<volatile int*>(smem + kOffMisc + 24);
        float sigma[4], inv_sigma[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            sigma[i] = FLT_MIN;
            inv_sigma[i] = 1.0f / FLT_MIN;
        }
        // sigma_t after block b: the running maximum of tile t's row scales
        auto sigma_step = [&](int b, float (&sig_new)[4]) {
            bool moved = false;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float m = fmaxf(smax_s[8 * (b & 1) + i], smax_s[8 * (b & 1) + 4 + i]);
                moved = moved || m > sigma[i];
                sig_new[i] = (m > sigma[i]) ? m : sigma[i];
            }
            return moved;
        };
        auto sigma_commit = [&](const float (&sig_new)[4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (sig_new[i] > sigma[i]) {
                    sigma[i] = sig_new[i];
                    inv_sigma[i] = 1.0f / sig_new[i];
                }
            }
        };
        bool failed = false;
        float mA = -INFINITY, mB = -INFINITY, lA = 0.0f, lB = 0.0f;
        // warpgroup 0: heads hA = 16wq + lane/4 and hB = hA + 8 (M = 64 layout: head
        // 16wq + i in lane 32wq + i), keys 8j + 2(lane % 4) + e, j = 0..7
        const int hA = 16 * wq + (lane >> 2), hB = hA + 8;
        const int kq = 2 * (lane & 3);

        if (g == 1) {
            // ---- converting warpgroup: row 32 (wq & 1) + lane of each block,
            // 16-byte units 2up, 2up+1 with up = (wq >> 1) + 2k ----
            const int rw = 32 * (wq & 1) + lane;
            int ci = 0;
            uint32_t nb[kNumBuf] = {0u, 0u, 0u};
            bool ok = true;
            auto row_of = [&](int b) {
                const int si = 2 * b + (wq & 1);
                return smem + kOffRing + (si % kStages) * kStageBytes + lane * kRowBytes;
            };
            auto claim = [&]() {
                const int bi = ci % kNumBuf;
                if (ci >= kNumBuf) ok = warp_wait(&bdone[bi], nb[bi]++ & 1u, abort_flag) && ok;
                return bi;
            };
            auto publish = [&](int bi) {
                fence_proxy_async_smem();        // generic writes, read by the tensor cores
                tc_before();
                warp_arrive(&kready[bi]);
                ++ci;
            };
            // E4M3 codes of latent tile tt -> f16 (exact), or times scale / sigma_tt (V')
            auto convert = [&](int b, int tt, bool scaled) {
                const int bi = claim();
                const uint8_t* row = row_of(b);
                uint8_t* dst = buf + bi * 16384;
                uint32_t s2 = 0u;
                if (scaled) {
                    const float sr = *reinterpret_cast<const float*>(row + kScaleOff + 4 * tt) * inv_sigma[tt];
                    s2 = pack_f16x2(sr, sr);
                }
                uint4 w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) w[k] = *reinterpret_cast<const uint4*>(row + 128 * tt + 16 * ((wq >> 1) + 2 * k));
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int up = (wq >> 1) + 2 * k;     // codes 16up .. 16up+15 of the tile
                    uint4 o0, o1;
                    e4m3x4_to_f16x2x2(w[k].x, o0.x, o0.y);
                    e4m3x4_to_f16x2x2(w[k].y, o0.z, o0.w);
                    e4m3x4_to_f16x2x2(w[k].z, o1.x, o1.y);
                    e4m3x4_to_f16x2x2(w[k].w, o1.z, o1.w);
                    if (scaled) {
                        o0.x = hmul2(o0.x, s2); o0.y = hmul2(o0.y, s2); o0.z = hmul2(o0.z, s2); o0.w = hmul2(o0.w, s2);
                        o1.x = hmul2(o1.x, s2); o1.y = hmul2(o1.y, s2); o1.z = hmul2(o1.z, s2); o1.w = hmul2(o1.w, s2);
                    }
                    *reinterpret_cast<uint4*>(dst + swz(64, rw, 2 * up)) = o0;
                    *reinterpret_cast<uint4*>(dst + swz(64, rw, 2 * up + 1)) = o1;
                }
                publish(bi);
            };
            auto rope_tile = [&](int b) {
                const int bi = claim();
                const uint8_t* row = row_of(b);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int u = (wq >> 1) + 2 * k;
                    *reinterpret_cast<uint4*>(buf + bi * 16384 + swz(64, rw, u)) =
                        *reinterpret_cast<const uint4*>(row + kTailOff + 16 * u);
                }
                publish(bi);
            };
            // A block's rows have landed: its row scales and their maxima for the others.
            auto prep = [&](int b) {
                const int si = 2 * b + (wq & 1);
                ok = warp_wait(&full[si % kStages], static_cast<uint32_t>((si / kStages) & 1), abort_flag) && ok;
                if (wq < 2) {
                    const float4 s4 = *reinterpret_cast<const float4*>(row_of(b) + kScaleOff);
                    float* sc = sc_s + 256 * (b & 1);
                    sc[rw] = s4.x;
                    sc[64 + rw] = s4.y;
                    sc[128 + rw] = s4.z;
                    sc[192 + rw] = s4.w;
                    float m4[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
#pragma unroll
                        for (int d = 16; d > 0; d >>= 1) m4[i] = fmaxf(m4[i], __shfl_xor_sync(0xffffffffu, m4[i], d));
                    }
                    if (lane == 0) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) smax_s[8 * (b & 1) + 4 * wq + i] = m4[i];
                    }
                }
                warp_arrive(&scready[b & 1]);
            };
            if (nblk > 0) {
                prep(0);
                convert(0, 0, false);
                convert(0, 1, false);
            }
            for (int b = 0; b < nblk && ok; ++b) {
                convert(b, 2, false);
                convert(b, 3, false);
                if (kRopeOn) rope_tile(b);
                if (b + 1 < nblk) {
                    prep(b + 1);
                    convert(b + 1, 0, false);
                    convert(b + 1, 1, false);
                }
                float sig_new[4];
                (void)sigma_step(b, sig_new);
                sigma_commit(sig_new);
#pragma unroll
                for (int tt = 0; tt < 4; ++tt) convert(b, tt, true);
                // the block's stages are next written by bulk copies (async proxy)
                fence_proxy_async_smem();
                warp_arrive(&empty[(2 * b) % kStages]);
                warp_arrive(&empty[(2 * b + 1) % kStages]);
            }
            if (!ok) {
                failed = true;
                if (warp == 4 && lane == 0) reinterpret_cast<volatile int*>(smem + kOffMisc)[5] = 1;
            }
        } else {
            // ---- softmax warpgroup ----
            const float rowfA = rowf_s[hA], rowfB = rowf_s[hB];
            int fq = 0;
            uint32_t nsr[kNumBuf] = {0u, 0u, 0u}, npv = 0u;
            bool ok = true;
            float acc[32];
            // S of the next QK group (slot fq % 3) read back and folded into acc:
            // a latent tile times its row scales, or the RoPE part as it is.
            auto fold = [&](const float* sc) {
                const int slot = fq % kNumBuf;
                ok = warp_wait(&sready[slot], nsr[slot]++ & 1u, abort_flag) && ok;
                tc_after();
                uint32_t r[32];
                tmem_ld_16x256b_x8(tmem + lane_q + kColS + 64 * slot, r);
                tc_wait_ld();
                tc_before();
                warp_arrive(&sfree[slot]);
                ++fq;
                if (sc == nullptr) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[i] += __uint_as_float(r[i]);
                    return;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float2 s2 = *reinterpret_cast<const float2*>(sc + 8 * j + kq);
                    acc[4 * j + 0] = fmaf(__uint_as_float(r[4 * j + 0]), s2.x, acc[4 * j + 0]);
                    acc[4 * j + 1] = fmaf(__uint_as_float(r[4 * j + 1]), s2.y, acc[4 * j + 1]);
                    acc[4 * j + 2] = fmaf(__uint_as_float(r[4 * j + 2]), s2.x, acc[4 * j + 2]);
                    acc[4 * j + 3] = fmaf(__uint_as_float(r[4 * j + 3]), s2.y, acc[4 * j + 3]);
                }
            };
            for (int b = 0; b < nblk; ++b) {
                const int n_b = min(kBlockRows, n_valid - b * kBlockRows);
                ok = warp_wait(&scready[b & 1], static_cast<uint32_t>((b >> 1) & 1), abort_flag) && ok;
                const float* sc = sc_s + 256 * (b & 1);
                float sig_new[4];
                const bool sig_move = sigma_step(b, sig_new);     // read now: the slot is reused two blocks on
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
#pragma unroll 1
                for (int tt = 0; tt < 4; ++tt) fold(sc + 64 * tt);
                if (kRopeOn) fold(nullptr);
                if (b > 0) ok = warp_wait(pvdone, npv++ & 1u, abort_flag) && ok;   // P^T and O^T free of block b-1
                tc_after();

                // softmax of this thread's 2 heads x 16 keys (the 4 threads of a
                // head quad hold its 64 keys); barrier 1 carries any failed wait.
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int key = 8 * (i >> 2) + kq + (i & 1);
                    v[i] = (key < n_b) ? acc[i] * ((i & 2) ? rowfB : rowfA) : -INFINITY;
                }
                float bmA = -INFINITY, bmB = -INFINITY;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    bmA = fmaxf(bmA, fmaxf(v[4 * j], v[4 * j + 1]));
                    bmB = fmaxf(bmB, fmaxf(v[4 * j + 2], v[4 * j + 3]));
                }
                bmA = fmaxf(bmA, __shfl_xor_sync(0xffffffffu, bmA, 1));
                bmA = fmaxf(bmA, __shfl_xor_sync(0xffffffffu, bmA, 2));
                bmB = fmaxf(bmB, __shfl_xor_sync(0xffffffffu, bmB, 1));
                bmB = fmaxf(bmB, __shfl_xor_sync(0xffffffffu, bmB, 2));
                if (!ok) fail_s[b & 1] = 1;
                const bool need = bmA > mA + kRescaleSlack || bmB > mB + kRescaleSlack;
                const bool any_need = bar_sync_or(1, 128, need || !ok);
                if (fail_s[b & 1]) {
                    failed = true;
                    break;
                }
                float aA = 1.0f, aB = 1.0f;
                if (any_need) {
                    const float nA = (bmA > mA + kRescaleSlack) ? bmA : mA;
                    const float nB = (bmB > mB + kRescaleSlack) ? bmB : mB;
                    aA = ex2_approx(mA - nA);        // -inf -> 0
                    aB = ex2_approx(mB - nB);
                    lA *= aA;
                    lB *= aB;
                    mA = nA;
                    mB = nB;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float p0 = ex2_approx(v[4 * j] - mA), p1 = ex2_approx(v[4 * j + 1] - mA);
                    const float p2 = ex2_approx(v[4 * j + 2] - mB), p3 = ex2_approx(v[4 * j + 3] - mB);
                    lA += p0 + p1;
                    lB += p2 + p3;
                    // keys 8j .. 8j+7 are 16-byte unit j of the P^T row
                    *reinterpret_cast<uint32_t*>(pT + swz(64, hA, j) + 2 * kq) = pack_f16x2(p0, p1);
                    *reinterpret_cast<uint32_t*>(pT + swz(64, hB, j) + 2 * kq) = pack_f16x2(p2, p3);
                }
                if (b > 0 && (any_need || sig_move)) {
                    // Rare after the first block: O^T (dims in this warp's lanes,
                    // heads as columns) times the heads' offset factors and
                    // sigma_old / sigma_new. Block b-1's PV is complete, block b's
                    // has not begun.
                    if ((lane & 3) == 0) {
                        alpha_s[hA] = aA;
                        alpha_s[hB] = aB;
                    }
                    asm volatile("bar.sync 2, 128;" ::: "memory");
#pragma unroll
                    for (int tt = 0; tt < 4; ++tt) {
                        const float fs = sigma[tt] / sig_new[tt];
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint32_t r[16];
                            tmem_ld_32x32b_x16(tmem + lane_q + 64 * tt + 16 * c, r);
                            tc_wait_ld();
#pragma unroll
                            for (int k = 0; k < 16; ++k)
                                r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha_s[16 * c + k] * fs);
                            tmem_st_32x32b_x16(tmem + lane_q + 64 * tt + 16 * c, r);
                        }
                    }
                    tc_wait_st();
                    asm volatile("bar.sync 2, 128;" ::: "memory");     // alpha_s is rewritten at the next rescale
                }
                sigma_commit(sig_new);
                fence_proxy_async_smem();
                tc_before();
                warp_arrive(pready);
                ok = true;
            }
            if (!failed && nblk > 0) {
                ok = warp_wait(pvdone, npv++ & 1u, abort_flag) && ok;     // the last block's PV
                if (!ok) fail_s[nblk & 1] = 1;
            }
            tc_after();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            failed = failed || fail_s[nblk & 1] != 0;
            if (!failed) {
                // l of each head over its quad; lse and 1 / l per head for both warpgroups.
                lA += __shfl_xor_sync(0xffffffffu, lA, 1);
                lA += __shfl_xor_sync(0xffffffffu, lA, 2);
                lB += __shfl_xor_sync(0xffffffffu, lB, 1);
                lB += __shfl_xor_sync(0xffffffffu, lB, 2);
            }
        }

        // ---- epilogue (both warpgroups): O^T tiles 2g, 2g+1 -> out ----
        const int64_t out_row0 = static_cast<int64_t>(t) * args.H + hg * kHG;              // (t, first head)
        const int64_t part_row0 = (static_cast<int64_t>(t) * args.nsplit + split) * args.H + hg * kHG;
        const float kNaN = __int_as_float(0x7FC00000);
        if (g == 0 && !failed && (lane & 3) == 0) {
            // l = 0: nothing present (out 0, lse -inf); l NaN: a listed row holds
            // a NaN (out and lse NaN, as the decode statement gives).
            const int hs[2] = {hA, hB};
            const float ls[2] = {lA, lB};
            const float ms[2] = {mA, mB};
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float lt = ls[i];
                alpha_s[hs[i]] = lt > 0.0f ? 1.0f / lt : (lt == 0.0f ? 0.0f : kNaN);
                const float lse_v = lt > 0.0f ? (ms[i] + log2f(lt)) * kLn2 : (lt == 0.0f ? -INFINITY : kNaN);
                lsum_s[hs[i]] = lse_v;
                if (args.nsplit == 1) args.lse[out_row0 + hs[i]] = lse_v;
                else args.ws_lse[part_row0 + hs[i]] = lse_v;
            }
        }
        // both warpgroups: the failure state and the per-head factors
        if (g == 0 && lane == 0 && wq == 0) fail_s[(nblk + 1) & 1] = failed ? 1 : 0;
        asm volatile("bar.sync 3, %0;" :: "n"(kMathThreads) : "memory");
        tc_after();
        failed = fail_s[(nblk + 1) & 1] != 0 || reinterpret_cast<volatile int*>(smem + kOffMisc)[5] != 0;
        if (!failed) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int tt = 2 * g + q;
                const int d = 128 * tt + 32 * wq + lane;
                // (register arrays indexed by constants only: g selects the pair)
                const float sg = g ? sigma[2 + q] : sigma[q];
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[16];
                    if (nblk > 0) {
                        tmem_ld_32x32b_x16(tmem + lane_q + 64 * tt + 16 * c, r);
                        tc_wait_ld();
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k) r[k] = 0u;
                    }
                    if (args.nsplit == 1) {
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            const int h = 16 * c + k;
                            const float x = __uint_as_float(r[k]) * sg * alpha_s[h];
                            const float y = __shfl_xor_sync(0xffffffffu, x, 1);
                            // lanes 2i and 2i+1 hold dims d, d+1: the even lane stores
                            // the pair for even heads, the odd lane for odd heads
                            if ((lane & 1) == (k & 1)) {
                                const uint32_t w = (lane & 1) ? pack_bf16x2(y, x) : pack_bf16x2(x, y);
                                __nv_bfloat16* o = static_cast<__nv_bfloat16*>(args.out) + (out_row0 + h) * kLatent + (d & ~1);
                                *reinterpret_cast<uint32_t*>(o) = w;
                            }
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            const int h = 16 * c + k;
                            if (lsum_s[h] == -INFINITY) continue;     // no present entry: the merge skips o
                            args.ws_o[(part_row0 + h) * kLatent + d] = __uint_as_float(r[k]) * sg * alpha_s[h];
                        }
                    }
                }
            }
        }
    }

    // ---- teardown: every role is done; tensor memory is freed by its owner warp ----
    tc_before();
    __syncthreads();
    tc_after();
    if (threadIdx.x == 0 && *abort_flag) {
        // A wait ran out: record it and let the copies in flight land before the
        // CTA exits. A slot's stages are issued in order, and issuing one waited
        // for the previous one to be read, so only the latest stage of each slot
        // can still be in flight.
        atomicOr(args.err, MLA_ERR_PIPELINE_TIMEOUT);
        int last[kStages] = {-1, -1, -1, -1};
        for (int q = 0; q < kProds; ++q)
            for (int k = 0; k < issued_s[q]; ++k) {
                const int si = q + kProds * k;
                last[si % kStages] = max(last[si % kStages], si);
            }
        for (int s = 0; s < kStages; ++s)
            if (last[s] >= 0) (void)mbar_wait_bounded(&full[s], static_cast<uint32_t>((last[s] / kStages) & 1));
    }
    if (warp == kMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(kTmemCols) : "memory");
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace mla_host {

// One CTA per (token, 64-head group) when that fills the GPU; otherwise each
// token's list is split into as many pieces as there are free SMs for, each of
// at least kSplitMinRows positions and at most kListMax (one CTA per SM: the
// kernel's shared memory admits no second one).
int choose_nsplit_h64(int T, int H, int W, int sms) {
    constexpr int kSplitMinRows = 256;
    if (T <= 0 || W <= 0 || H % kHG != 0) return 1;
    const int64_t base = static_cast<int64_t>(T) * (H / kHG);
    int64_t ns = (base < sms) ? sms / base : 1;
    const int64_t max_ns = (W >= kSplitMinRows) ? W / kSplitMinRows : 1;
    if (ns > max_ns) ns = max_ns;
    const int64_t min_ns = (W + kListMax - 1) / kListMax;
    if (ns < min_ns) ns = min_ns;
    if (ns < 1) ns = 1;
    return static_cast<int>(ns);
}

int rank_chunk_h64(int W, int nsplit) {
    if (nsplit <= 1 || W > kListMax) return 0;
    return (W + nsplit - 1) / nsplit;
}

int launch_decode_h64(const DecodeCall& c, cudaStream_t stream) {
    if (c.H % kHG != 0 || !aligned16(c.cache) || !aligned16(c.q)) return MLA_EINVAL;
    if (!max_dynamic_smem(reinterpret_cast<const void*>(mla_sparse_decode_h64_kernel<true>), kSmemTotal) ||
        !max_dynamic_smem(reinterpret_cast<const void*>(mla_sparse_decode_h64_kernel<false>), kSmemTotal))
        return MLA_ECUDA;
    const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(c.T) * (c.H / kHG)), static_cast<unsigned>(c.nsplit));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemTotal;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t lr = (c.d_qk == kLatent + kRope) ? cudaLaunchKernelEx(&cfg, mla_sparse_decode_h64_kernel<true>, c)
                                                       : cudaLaunchKernelEx(&cfg, mla_sparse_decode_h64_kernel<false>, c);
    if (lr != cudaSuccess || cudaGetLastError() != cudaSuccess) return MLA_ECUDA;
    return MLA_OK;
}

}  // namespace mla_host
