// mla_sparse_decode: sparse top-k MLA decode over the packed FP8 cache.
//
// What it computes follows the decode statement quoted in the C header, with
// the masking rule of sglang PR #39288 (Root cause: a -1 candidate must add
// nothing and must not gather slot 0) and sglang PR #47013 (Motivation: masking
// only the score does not stop a NaN row). Here an absent entry is removed
// before anything is fetched: each CTA compacts its slice of the top-k list in
// shared memory, so -1, slot 0 and out-of-range indices are never dereferenced.
//
// Work decomposition: one CTA per (token, split of the top-k list, group of 16
// heads), the head groups of a token adjacent in launch order and tokens taken
// from the last to the first; 4 consumer warps and 2 producer warps. A token's
// list is split only when there are fewer (token, head group) pairs than SMs.
// Lists that one CTA can compact are then split by a plan: a first kernel
// compacts every token's list once (mla_list_compact_kernel), and each decode
// CTA reads all tokens' counts and cuts every list into pieces of at most C
// present entries, C the smallest multiple of 32 (at least kPlanMinRows) for
// which all pieces fit in one wave of CTAs, so a long list gets more pieces
// than a short one. Longer lists are split by positions. Every thread loads a
// contiguous run of the positions at once (the q loads are issued before them),
// maps them through the block table when the list holds sequence positions (the
// paged entry point, vLLM PR #55277, Purpose item 2), and one block-wide scan
// places the present slots in a shared-memory list. When the CTA's first 32
// positions (or a planned piece's first 32 entries) are all present, the first
// copy-issuing warp copies them (block 0) before the list is in shared memory,
// so the first block lands meanwhile. Rows are 656 bytes, or 528 for a cache
// of NoPE rows without a tail (sglang PR #39288, "Relation to other changes"). The
// producers copy each listed row global -> shared with one cp.async.bulk (656 B,
// or 528 B for NoPE: the tail is not read) into a 4-stage ring of 32-row blocks,
// each stage completing on an mbarrier; producer p issues blocks p, p+2, ...
// (one warp's copy issue is what limits a CTA's row rate, so two issue in
// parallel).
//
// Arithmetic per 32-row block, on tensor cores (m16n8k16, heads as M):
//   QK  : warp w takes latent tile w (dims 128w .. 128w+127) and RoPE dims
//         16w .. 16w+15 for all 32 rows. The E4M3 latent goes to f16 exactly
//         (cvt.f16x2.e4m3x2); q goes to f16 exactly after an exponent-only
//         per-head rescale that keeps it in f16 range; the per-row, per-tile
//         fp32 scale multiplies each tile partial afterwards, so q.K is exact
//         before fp32 accumulation. RoPE dims run as a bf16 MMA.
//   softmax: the four tile partials meet in shared memory and warp w finishes
//         the scores of rows 8w .. 8w+7 only; online max / sum in fp32 with exp2
//         (log2 e folded into sm_scale). The exp2 offset of a head is shared by
//         all warps and moves only when a block maximum runs more than
//         kRescaleSlack above it, so P <= 2^8 fits the f16 operand.
//   PV  : warp w owns output dims 128w .. 128w+127; P (f16, from shared memory)
//         times scale_row / sigma (sigma = running max of tile w's scales) times
//         the exact f16 E4M3 codes, with 16-byte V loads; O stays in registers.
//         What does not need P (sigma, O's rescale when it moves, the f16 pairs
//         scale_row / sigma, the first V rows) is done before the barriers, off
//         the path from P to the first PV MMA.
// A consumer warp releases a stage only after fencing the async proxy, since the
// next write to the stage is a bulk copy and its own reads were generic loads.
// Splits write a normalised partial (o, lse) to the caller's workspace and a
// second kernel, launched with programmatic stream serialization, merges them in
// split order (deterministic: no float atomics).
#include <cfloat>
#include <climits>
#include <cmath>

#include "mla_device.cuh"

namespace {

using namespace mla;

constexpr int kHeads = 16;                   // heads per CTA (M of m16n8k16)
constexpr int kWarps = 4;                    // consumer warps (one per latent tile)
constexpr int kProducer = kWarps;            // warp index of the first copy-issuing warp
constexpr int kProducers = 2;                // copy-issuing warps (alternate blocks)
constexpr int kThreads = (kWarps + kProducers) * 32;
constexpr int kConsumerThreads = kWarps * 32;
constexpr int kNB = 32;                      // rows per block
constexpr int kStages = 4;
constexpr int kListMax = 2304;               // positions one CTA compacts
constexpr int kPlanMinRows = 128;            // shortest planned piece (fewer partials to merge)
constexpr int kPerThread = (kListMax + kThreads - 1) / kThreads;   // positions per thread in the compaction
constexpr int kStageBytes = kNB * kRowBytes; // 20,992
constexpr int kSmemStages = kStages * kStageBytes;
constexpr int kSmemList = kListMax * 4;
constexpr int kSmemRed = kWarps * 4 * 32 * 16;       // QK tile partials: float4 [warp][n-tile][lane]
constexpr int kSmemP = 4 * 32 * 8;                   // P (f16): uint2 [n-tile][lane], A-fragment order
constexpr int kSmemQmax = 3 * kWarps * kHeads * 4;   // |q| maxima, block score maxima, l partials
constexpr int kSmemMisc = 32 + 2 * kStages * 8 + 16; // warp counts, full + empty barriers, issued count
constexpr int kSmemTotal = kSmemStages + kSmemList + kSmemRed + kSmemP + kSmemQmax + kSmemMisc;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// The running max used as the exp2 offset is only moved when a score exceeds it
// by more than this (log2 units): p <= 2^8 keeps the f16 P operand in range.
constexpr float kRescaleSlack = 8.0f;

__device__ __forceinline__ float quad_max(float v) {
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
    return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}

struct DecodeArgs {
    const __nv_bfloat16* q;
    const uint8_t* cache;
    const int32_t* topk;
    __nv_bfloat16* out;
    float* lse;
    float* ws_o;      // [T * nsplit, H, 512], or [plan_pieces, H, 512] when planned
    float* ws_lse;    // [T * nsplit, H], or [plan_pieces, H]
    int* err;
    int64_t num_slots;
    int64_t row_bytes;          // 656, or 528 (NoPE rows without a tail)
    // Paged top-k (page_size > 0): entries are sequence positions, mapped to
    // slots through block_table[seq][position / page_size].
    const int32_t* block_table; // [n_seq, bt_pages]
    const int32_t* token_seq;   // [T] block-table row of each token, or null (row 0)
    int bt_pages, n_seq, page_size;
    int T, H, d_qk, W, nsplit;
    // Split of a token's list by positions (nsplit > 1, no plan): split_len each.
    int split_len;
    // Planned split (plan_list != nullptr, W <= kListMax): the compacted lists,
    // their lengths, and per token its first piece and piece count (written by
    // the decode for the merge); plan_pieces piece slots per head group.
    int32_t* plan_list;    // [T, W]
    int32_t* plan_count;   // [T]
    int2* plan_tok;        // [T]
    int plan_pieces;
    float sm_scale_log2;   // sm_scale * log2(e)
};

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    return v;
}

// Position -> slot through the block table (vLLM PR #55277, Purpose item 2): a
// negative position or an unassigned (negative) page is absent (-1); a position
// past the table, or any position of a token whose sequence row is out of range,
// is absent and flagged.
__device__ __forceinline__ int paged_slot(const DecodeArgs& a, const int32_t* bt, bool seq_ok, int pos) {
    if (pos < 0) return -1;
    const int page = pos / a.page_size;
    if (!seq_ok || page >= a.bt_pages) {
        atomicOr(a.err, MLA_ERR_DECODE_INDEX_RANGE);
        return -1;
    }
    const int phys = __ldg(bt + page);
    const int64_t slot = static_cast<int64_t>(phys) * a.page_size + (pos - page * a.page_size);
    return (phys < 0) ? -1 : static_cast<int>(min(slot, static_cast<int64_t>(INT32_MAX)));
}

// Chunk length of the planned split, from the T list lengths in cnt (one warp,
// every lane gets the result): the smallest multiple of kNB, at least
// kPlanMinRows and at least total / G, for which the pieces
// sum_t max(1, ceil(n_t / C)) number at most G. T <= G, so C = kListMax (one
// piece per token) always fits and ends the search.
__device__ __forceinline__ int plan_chunk(const int* cnt, int T, int G, int lane) {
    int total = 0;
    for (int i = lane; i < T; i += 32) total += cnt[i];
    total = warp_sum(total);
    int C = max(kPlanMinRows, ((total + G - 1) / G + kNB - 1) / kNB * kNB);
    for (; C < kListMax; C += kNB) {
        int pieces = 0;
        for (int i = lane; i < T; i += 32) pieces += max(1, (cnt[i] + C - 1) / C);
        if (warp_sum(pieces) <= G) break;
    }
    return min(C, kListMax);
}

template <bool kRopeOn, bool kPlanned>
__global__ void __launch_bounds__(kThreads, 2)
mla_sparse_decode_kernel(const DecodeArgs args) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* stages = smem;
    int* list = reinterpret_cast<int*>(smem + kSmemStages);
    float4* red = reinterpret_cast<float4*>(smem + kSmemStages + kSmemList);
    uint32_t* pbuf = reinterpret_cast<uint32_t*>(smem + kSmemStages + kSmemList + kSmemRed);
    float* qmax_s = reinterpret_cast<float*>(smem + kSmemStages + kSmemList + kSmemRed + kSmemP);
    float* rmax_s = qmax_s + kWarps * kHeads;
    float* lsum_s = rmax_s + kWarps * kHeads;
    int* wcount = reinterpret_cast<int*>(smem + kSmemStages + kSmemList + kSmemRed + kSmemP + kSmemQmax);
    uint64_t* full = reinterpret_cast<uint64_t*>(wcount + 8);
    uint64_t* empty = full + kStages;
    int* issued_s = reinterpret_cast<int*>(empty + kStages);

    // blockIdx.x = (T - 1 - t) * head_groups + hg: the head groups of a token run
    // side by side and gather the same rows, so all but the first read them from
    // L2; tokens are taken from the last to the first, because in a causal
    // (prefill-shaped) batch the later tokens have the longest lists and starting
    // them first shortens the tail (the prefill shape: 103.6 us against 111.7 in
    // token order). No result depends on the order. A planned split has
    // blockIdx.x = piece * head_groups + hg; the piece's token comes from the plan.
    constexpr bool planned = kPlanned;   // args.plan_list != nullptr
    const int head_groups = (args.H + kHeads - 1) / kHeads;
    int t = planned ? 0 : args.T - 1 - static_cast<int>(blockIdx.x / head_groups);
    const int hg = static_cast<int>(blockIdx.x % head_groups);
    const int split = planned ? static_cast<int>(blockIdx.x / head_groups) : static_cast<int>(blockIdx.y);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int H = args.H;
    constexpr uint32_t kRowRead = kRopeOn ? kRowBytes : kNopeReadBytes;

    // The positions this CTA compacts (none when planned).
    const int p0 = planned ? 0 : split * args.split_len;
    const int p1 = planned ? 0 : min(args.W, p0 + args.split_len);
    // While the previous kernel on the stream may still be running, bring those
    // positions and this head group's q rows into L2. A prefetch returns nothing
    // to the kernel; every load after the wait below sees the previous kernel's
    // writes.
    if (!planned) {
        const char* lb = reinterpret_cast<const char*>(args.topk + static_cast<int64_t>(t) * args.W + p0);
        const int lines = (max(0, p1 - p0) * 4 + 127) / 128;
        for (int i = threadIdx.x; i < lines; i += kThreads) prefetch_l2(lb + 128 * i);
        const int nh = min(kHeads, args.H - hg * kHeads);
        const char* qb = reinterpret_cast<const char*>(args.q + (static_cast<int64_t>(t) * args.H + hg * kHeads) * args.d_qk);
        const int qlines = (nh * args.d_qk * 2 + 127) / 128;
        for (int i = threadIdx.x; i < qlines; i += kThreads) prefetch_l2(qb + 128 * i);
    }
    // Launched with programmatic stream serialization: wait for the previous
    // kernel on the stream (and its memory) before reading any input. The
    // merge of split partials may then start launching; it waits for this grid.
    pdl_wait();
    pdl_launch_dependents();

    // Planned split: all tokens' list lengths to shared memory (the list area,
    // free until the piece is copied there); warp 0 finds the chunk length and
    // this piece's token and entry range, and the first piece of each token
    // records the token's pieces for the merge. A piece slot past the last piece
    // has no work and returns.
    int lbase = 0, n_valid = 0;
    if (planned) {
        for (int i = threadIdx.x; i < args.T; i += kThreads) list[i] = __ldg(args.plan_count + i);
        __syncthreads();
        if (warp == 0) {
            const int C = plan_chunk(list, args.T, args.plan_pieces, lane);
            int acc = 0, tok = -1, first = 0, k_t = 0;
            for (int base = 0; base < args.T && tok < 0; base += 32) {
                const int i = base + lane;
                const int k = (i < args.T) ? max(1, (list[i] + C - 1) / C) : 0;
                int incl = k;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, d);
                    if (lane >= d) incl += v;
                }
                const unsigned hit = __ballot_sync(0xffffffffu, k > 0 && split >= acc + incl - k && split < acc + incl);
                if (hit != 0u) {
                    const int src = __ffs(hit) - 1;
                    tok = base + src;
                    first = __shfl_sync(0xffffffffu, acc + incl - k, src);
                    k_t = __shfl_sync(0xffffffffu, k, src);
                }
                acc += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) {
                wcount[0] = tok;
                if (tok >= 0) {
                    const int n = list[tok];
                    const int len = (n + k_t - 1) / k_t;
                    const int lb = min(n, (split - first) * len);
                    wcount[1] = lb;
                    wcount[2] = min(n, lb + len) - lb;
                    if (split == first && hg == 0) args.plan_tok[tok] = make_int2(first, k_t);
                }
            }
        }
        __syncthreads();
        t = wcount[0];
        if (t < 0) return;
        lbase = wcount[1];
        n_valid = wcount[2];
    }

    // The first copy-issuing warp sets up the ring. When this CTA's first 32
    // positions are all present (unsplit or split by positions; through the block
    // table for the paged entry point), they are exactly the first 32 entries of the
    // compacted list, so the warp copies block 0 right away and the copies land
    // while the whole list is compacted. A planned piece holds present slots only:
    // its first 32 entries are block 0 whenever it has that many.
    bool block0_issued = false;
    if (warp == kProducer) {
        if (lane == 0) {
            for (int s = 0; s < kStages; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], kWarps);
            }
            issued_s[0] = issued_s[1] = 0;
            fence_mbar_init();
        }
        __syncwarp();
        if (planned && n_valid >= kNB) {
            const int idx = __ldg(args.plan_list + static_cast<int64_t>(t) * args.W + lbase + lane);
            if (lane == 0) mbar_arrive_expect_tx(&full[0], kNB * kRowRead);
            __syncwarp();
            bulk_g2s(stages + lane * kRowBytes, args.cache + static_cast<int64_t>(idx) * args.row_bytes, kRowRead,
                     &full[0]);
            block0_issued = true;
        } else if (!planned && p1 - p0 >= kNB) {
            int idx = __ldg(args.topk + static_cast<int64_t>(t) * args.W + p0 + lane);
            bool present = true;
            if (args.page_size > 0) {
                // the same translation as the compaction's; anything it would drop
                // or flag only turns this shortcut off
                const int sq = args.token_seq ? __ldg(args.token_seq + t) : 0;
                const int page = idx >= 0 ? idx / args.page_size : 0;
                present = idx >= 0 && sq >= 0 && sq < args.n_seq && page < args.bt_pages;
                const int phys = present ? __ldg(args.block_table + static_cast<int64_t>(sq) * args.bt_pages + page) : -1;
                const int64_t slot = static_cast<int64_t>(phys) * args.page_size + (idx - page * args.page_size);
                present = present && phys >= 0 && slot <= INT32_MAX;
                idx = present ? static_cast<int>(slot) : 0;
            }
            present = present && idx > 0 && static_cast<int64_t>(idx) < args.num_slots;
            if (__all_sync(0xffffffffu, present)) {
                if (lane == 0) mbar_arrive_expect_tx(&full[0], kNB * kRowRead);
                __syncwarp();
                bulk_g2s(stages + lane * kRowBytes, args.cache + static_cast<int64_t>(idx) * args.row_bytes, kRowRead,
                         &full[0]);
                block0_issued = true;
            }
        }
    }

    // ---- 0. q of this token and head group (consumer warps), loads issued first ----
    const int g = lane >> 2;
    const int c = lane & 3;
    const int h_lo = hg * kHeads + g;
    const int h_hi = h_lo + 8;
    uint32_t qraw[2][16];
    uint32_t qr[2][2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int h = r ? h_hi : h_lo;
        qr[r][0] = qr[r][1] = 0u;
#pragma unroll
        for (int k = 0; k < 16; ++k) qraw[r][k] = 0u;
        if (warp < kWarps && h < H) {
            const __nv_bfloat16* qh = args.q + (static_cast<int64_t>(t) * H + h) * args.d_qk;
            const uint8_t* p = reinterpret_cast<const uint8_t*>(qh + 128 * warp + 32 * c);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 v = ld_nc_v4(p + 16 * k);
                qraw[r][4 * k + 0] = v.x; qraw[r][4 * k + 1] = v.y;
                qraw[r][4 * k + 2] = v.z; qraw[r][4 * k + 3] = v.w;
            }
            if (kRopeOn) {
                const uint2 v = *reinterpret_cast<const uint2*>(qh + kLatent + 16 * warp + 4 * c);
                qr[r][0] = v.x; qr[r][1] = v.y;
            }
        }
    }

    // ---- 1. compact the present entries of this split's positions (all warps) ----
    // Thread i takes a contiguous run of `per` positions, loaded all at once; one
    // block-wide scan of the per-thread counts places them in position order. A
    // planned piece is already compacted: it is copied to the list.
    if (planned) {
        const int32_t* src = args.plan_list + static_cast<int64_t>(t) * args.W + lbase;
        for (int i = threadIdx.x; i < n_valid; i += kThreads) list[i] = __ldg(src + i);
        lbase = 0;
        __syncthreads();
    } else {
        const int per = (max(0, p1 - p0) + kThreads - 1) / kThreads;     // <= kPerThread
        const int32_t* trow = args.topk + static_cast<int64_t>(t) * args.W + p0 + threadIdx.x * per;
        const int mine = max(0, min(per, p1 - (p0 + static_cast<int>(threadIdx.x) * per)));
        int idxv[kPerThread];
#pragma unroll
        for (int k = 0; k < kPerThread; ++k) idxv[k] = (k < mine) ? __ldg(trow + k) : -1;
        if (args.page_size > 0) {
            const int sq = args.token_seq ? __ldg(args.token_seq + t) : 0;
            const bool seq_ok = sq >= 0 && sq < args.n_seq;
            const int32_t* bt = args.block_table + static_cast<int64_t>(seq_ok ? sq : 0) * args.bt_pages;
#pragma unroll
            for (int k = 0; k < kPerThread; ++k) idxv[k] = paged_slot(args, bt, seq_ok, idxv[k]);
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
        int off = incl - cnt;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            const int cw = wcount[w];
            off += (w < warp) ? cw : 0;
            n_valid += cw;
        }
#pragma unroll
        for (int k = 0; k < kPerThread; ++k)
            if (idxv[k] != 0) list[off++] = idxv[k];
        __syncthreads();
    }
    const int nblk = (n_valid + kNB - 1) / kNB;

    if (warp >= kProducer) {
        // ---- producers: warp kProducer + p issues blocks p, p + kProducers, ...;
        // lane j copies row j of the block into the stage ring ----
        const int pw = warp - kProducer;
        int b = pw, cnt = 0;
        if (block0_issued) {                   // producer 0, block 0 already on its way
            b += kProducers;
            cnt = 1;
        }
        for (; b < nblk; b += kProducers, ++cnt) {
            const int s = b % kStages;
            if (b >= kStages && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>(((b / kStages) - 1) & 1))) {
                if (lane == 0) atomicOr(args.err, MLA_ERR_PIPELINE_TIMEOUT);
                break;
            }
            uint8_t* dst = stages + s * kStageBytes;
            const int n_b = min(kNB, n_valid - b * kNB);
            if (n_b < kNB) {
                // Rows past the end of the list load nothing: zero them so the
                // block's arithmetic sees finite zeros (E4M3 0, scale 0.0).
                if (lane >= n_b) {
                    uint4* z = reinterpret_cast<uint4*>(dst + lane * kRowBytes);
                    for (int k = 0; k < kRowBytes / 16; ++k) z[k] = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(n_b) * kRowRead);
            __syncwarp();
            if (lane < n_b)
                bulk_g2s(dst + lane * kRowBytes,
                         args.cache + static_cast<int64_t>(list[lbase + b * kNB + lane]) * args.row_bytes, kRowRead, &full[s]);
        }
        if (lane == 0) issued_s[pw] = cnt;
        __syncthreads();     // matches the consumers' final barrier
        return;
    }

    // ---- consumers: q fragments ----
    float qm[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        qm[r] = 0.0f;
#pragma unroll
        for (int k = 0; k < 16; ++k) qm[r] = fmaxf(qm[r], fmaxf(fabsf(bf16lo(qraw[r][k])), fabsf(bf16hi(qraw[r][k]))));
#pragma unroll
        for (int k = 0; k < 2; ++k) qm[r] = fmaxf(qm[r], fmaxf(fabsf(bf16lo(qr[r][k])), fabsf(bf16hi(qr[r][k]))));
        qm[r] = quad_max(qm[r]);
    }
    if (c == 0) {
        qmax_s[warp * kHeads + g] = qm[0];
        qmax_s[warp * kHeads + g + 8] = qm[1];
    }
    bar_sync_or(1, kConsumerThreads, false);
    // Exponent-only rescale so that |q| < 2^15 in f16 (exact in f16's normal
    // range); the same power of two scales the RoPE part, and is undone on the
    // scores through the per-row softmax factor.
    float qdown[2], rowf[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        float mx = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, qmax_s[w * kHeads + g + 8 * r]);
        int e = 0;
        frexpf(mx, &e);                              // mx < 2^e
        const int k = (e > 15) ? (e - 15) : 0;
        qdown[r] = ldexpf(1.0f, -k);
        rowf[r] = args.sm_scale_log2 * ldexpf(1.0f, k);
    }
    uint32_t qa[8][4];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int wi = 8 * hf + 2 * kk;
            qa[4 * hf + kk][0] = pack_f16x2(bf16lo(qraw[0][wi]) * qdown[0], bf16hi(qraw[0][wi]) * qdown[0]);
            qa[4 * hf + kk][1] = pack_f16x2(bf16lo(qraw[1][wi]) * qdown[1], bf16hi(qraw[1][wi]) * qdown[1]);
            qa[4 * hf + kk][2] = pack_f16x2(bf16lo(qraw[0][wi + 1]) * qdown[0], bf16hi(qraw[0][wi + 1]) * qdown[0]);
            qa[4 * hf + kk][3] = pack_f16x2(bf16lo(qraw[1][wi + 1]) * qdown[1], bf16hi(qraw[1][wi + 1]) * qdown[1]);
        }
    }
    uint32_t qra[4];
    qra[0] = pack_bf16x2(bf16lo(qr[0][0]) * qdown[0], bf16hi(qr[0][0]) * qdown[0]);
    qra[1] = pack_bf16x2(bf16lo(qr[1][0]) * qdown[1], bf16hi(qr[1][0]) * qdown[1]);
    qra[2] = pack_bf16x2(bf16lo(qr[0][1]) * qdown[0], bf16hi(qr[0][1]) * qdown[0]);
    qra[3] = pack_bf16x2(bf16lo(qr[1][1]) * qdown[1], bf16hi(qr[1][1]) * qdown[1]);

    // ---- consumers: main loop ----
    // Per 32-row block: (1) QK partial of tile `warp` for all 32 rows, (2) the
    // four tile partials meet in shared memory and warp w finishes the scores of
    // rows 8w .. 8w+7 (its n-tile) and writes their P, (3) every warp multiplies
    // all 32 rows of P into V of its own tile. Two barriers per block; the exp2
    // offset of each head is common to all warps and moves only when a block
    // maximum runs more than kRescaleSlack above it (a third barrier then).
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m_ref[2] = {-INFINITY, -INFINITY};   // exp2 offset per head row (log2 units)
    float l_run[2] = {0.0f, 0.0f};             // sum of p over this warp's rows
    float sigma = FLT_MIN;                     // running max of tile `warp`'s row scales
    float inv_sigma = 1.0f / FLT_MIN;
    bool failed = false;

    for (int b = 0; b < nblk; ++b) {
        const int s = b % kStages;
        const bool ok = mbar_wait_bounded(&full[s], static_cast<uint32_t>((b / kStages) & 1));
        const uint8_t* st = stages + s * kStageBytes;
        const int n_b = min(kNB, n_valid - b * kNB);

        // (1) QK^T of tile `warp`: latent on f16 MMA, RoPE slice on bf16 MMA.
        float acc[4][4], accr[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[nt][i] = accr[nt][i] = 0.0f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            uint4 kv[4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
                kv[nt] = *reinterpret_cast<const uint4*>(st + (nt * 8 + g) * kRowBytes + 128 * warp + 32 * c + 16 * hf);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const uint32_t wrd = kk == 0 ? kv[nt].x : kk == 1 ? kv[nt].y : kk == 2 ? kv[nt].z : kv[nt].w;
                    uint32_t b0, b1;
                    e4m3x4_to_f16x2x2(wrd, b0, b1);
                    mma_f16(acc[nt], qa[4 * hf + kk], b0, b1);
                }
            }
        }
        if (kRopeOn) {
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const uint2 rb = *reinterpret_cast<const uint2*>(st + (nt * 8 + g) * kRowBytes + kTailOff + 32 * warp + 8 * c);
                mma_bf16(accr[nt], qra, rb.x, rb.y);
            }
        }
        // Scale of tile `warp` for rows nt*8 + 2c + e (rows past n_b were
        // zero-filled: scale 0). The same registers serve the PV step.
        float sc[4][2];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                sc[nt][e] = *reinterpret_cast<const float*>(st + (nt * 8 + 2 * c + e) * kRowBytes + kScaleOff + 4 * warp);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
            red[(warp * 4 + nt) * 32 + lane] =
                make_float4(fmaf(acc[nt][0], sc[nt][0], accr[nt][0]), fmaf(acc[nt][1], sc[nt][1], accr[nt][1]),
                            fmaf(acc[nt][2], sc[nt][0], accr[nt][2]), fmaf(acc[nt][3], sc[nt][1], accr[nt][3]));
        // The part of PV that does not need P, ahead of the barriers: sigma (the
        // running max of tile `warp`'s scales, so p * scale / sigma <= 2^8 in f16),
        // O rescaled when it moves, and the rows' scale / sigma as f16 pairs.
        float smax = 0.0f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) smax = fmaxf(smax, fmaxf(sc[nt][0], sc[nt][1]));
        smax = quad_max(smax);                 // all 32 rows: the same in every lane
        if (smax > sigma) {
            const float f = sigma / smax;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                o[i][0] *= f; o[i][1] *= f; o[i][2] *= f; o[i][3] *= f;
            }
            sigma = smax;
            inv_sigma = 1.0f / smax;
        }
        uint32_t rs[2][2];
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            rs[kb][0] = pack_f16x2(sc[2 * kb][0] * inv_sigma, sc[2 * kb][1] * inv_sigma);
            rs[kb][1] = pack_f16x2(sc[2 * kb + 1][0] * inv_sigma, sc[2 * kb + 1][1] * inv_sigma);
        }
        // Barrier 1 also carries a timeout of any warp to all of them.
        if (bar_sync_or(1, kConsumerThreads, !ok)) { failed = true; break; }

        // (2) scores of n-tile `warp`: rows 8*warp + 2c + {0,1}, heads g and g+8.
        float4 a = red[warp * 32 + lane];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) {
            const float4 bq = red[(w * 4 + warp) * 32 + lane];
            a.x += bq.x; a.y += bq.y; a.z += bq.z; a.w += bq.w;
        }
        float sv[4] = {a.x * rowf[0], a.y * rowf[0], a.z * rowf[1], a.w * rowf[1]};
        if (n_b < kNB) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (8 * warp + 2 * c + (i & 1) >= n_b) sv[i] = -INFINITY;
        }
        const float bm0 = quad_max(fmaxf(sv[0], sv[1]));
        const float bm1 = quad_max(fmaxf(sv[2], sv[3]));
        if (c == 0) {
            rmax_s[warp * kHeads + g] = bm0;
            rmax_s[warp * kHeads + g + 8] = bm1;
        }
        const bool need = bm0 > m_ref[0] + kRescaleSlack || bm1 > m_ref[1] + kRescaleSlack;
        float p[4];
        p[0] = ex2_approx(sv[0] - m_ref[0]);
        p[1] = ex2_approx(sv[1] - m_ref[0]);
        p[2] = ex2_approx(sv[2] - m_ref[1]);
        p[3] = ex2_approx(sv[3] - m_ref[1]);
        uint2* pw = reinterpret_cast<uint2*>(pbuf) + warp * 32 + lane;
        *pw = make_uint2(pack_f16x2(p[0], p[1]), pack_f16x2(p[2], p[3]));
        // V rows of the first PV step: loaded before barrier 2 (they do not depend on P).
        const uint8_t* vb = st + 128 * warp + 16 * g;
        uint4 Vn[4];
        Vn[0] = *reinterpret_cast<const uint4*>(vb + (2 * c + 0) * kRowBytes);
        Vn[1] = *reinterpret_cast<const uint4*>(vb + (2 * c + 1) * kRowBytes);
        Vn[2] = *reinterpret_cast<const uint4*>(vb + (2 * c + 8) * kRowBytes);
        Vn[3] = *reinterpret_cast<const uint4*>(vb + (2 * c + 9) * kRowBytes);
        if (bar_sync_or(1, kConsumerThreads, need)) {
            // Rare after the first block: move the offsets of the heads whose
            // block maximum ran ahead, rescale O and l, and rewrite this warp's P.
            float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                M0 = fmaxf(M0, rmax_s[w * kHeads + g]);
                M1 = fmaxf(M1, rmax_s[w * kHeads + g + 8]);
            }
            const float mn0 = (M0 > m_ref[0] + kRescaleSlack) ? M0 : m_ref[0];
            const float mn1 = (M1 > m_ref[1] + kRescaleSlack) ? M1 : m_ref[1];
            const float a0 = ex2_approx(m_ref[0] - mn0);     // -inf -> 0
            const float a1 = ex2_approx(m_ref[1] - mn1);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                o[i][0] *= a0; o[i][1] *= a0; o[i][2] *= a1; o[i][3] *= a1;
            }
            l_run[0] *= a0;
            l_run[1] *= a1;
            m_ref[0] = mn0;
            m_ref[1] = mn1;
            p[0] = ex2_approx(sv[0] - mn0);
            p[1] = ex2_approx(sv[1] - mn0);
            p[2] = ex2_approx(sv[2] - mn1);
            p[3] = ex2_approx(sv[3] - mn1);
            *pw = make_uint2(pack_f16x2(p[0], p[1]), pack_f16x2(p[2], p[3]));
            bar_sync_or(1, kConsumerThreads, false);
        }
        l_run[0] += p[0] + p[1];
        l_run[1] += p[2] + p[3];

        // (3) PV of tile `warp`.
        const uint2* pr = reinterpret_cast<const uint2*>(pbuf) + lane;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            // A: P of heads (g, g+8) x rows 16kb + 2c + {0,1} and + 8, times the
            // row's tile scale / sigma.
            const uint2 plo = pr[(2 * kb) * 32];
            const uint2 phi = pr[(2 * kb + 1) * 32];
            const uint32_t r01 = rs[kb][0];
            const uint32_t r89 = rs[kb][1];
            uint32_t pa[4];
            pa[0] = hmul2(plo.x, r01);
            pa[1] = hmul2(plo.y, r01);
            pa[2] = hmul2(phi.x, r89);
            pa[3] = hmul2(phi.y, r89);
            // B: V rows j0, j0+1, j0+8, j0+9; lane g takes dims 128w + 16g .. +15,
            // so n-tile (q, i) column n is dim 128w + 16n + 4q + i.
            const int j0 = 16 * kb + 2 * c;
            const uint4 V0 = kb == 0 ? Vn[0] : *reinterpret_cast<const uint4*>(vb + (j0 + 0) * kRowBytes);
            const uint4 V1 = kb == 0 ? Vn[1] : *reinterpret_cast<const uint4*>(vb + (j0 + 1) * kRowBytes);
            const uint4 V2 = kb == 0 ? Vn[2] : *reinterpret_cast<const uint4*>(vb + (j0 + 8) * kRowBytes);
            const uint4 V3 = kb == 0 ? Vn[3] : *reinterpret_cast<const uint4*>(vb + (j0 + 9) * kRowBytes);
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                const uint32_t W0 = qd == 0 ? V0.x : qd == 1 ? V0.y : qd == 2 ? V0.z : V0.w;
                const uint32_t W1 = qd == 0 ? V1.x : qd == 1 ? V1.y : qd == 2 ? V1.z : V1.w;
                const uint32_t W2 = qd == 0 ? V2.x : qd == 1 ? V2.y : qd == 2 ? V2.z : V2.w;
                const uint32_t W3 = qd == 0 ? V3.x : qd == 1 ? V3.y : qd == 2 ? V3.z : V3.w;
                uint32_t b0a, b0b, b0c, b0d, b1a, b1b, b1c, b1d;
                e4m3x4_to_f16x2x2(prmt(W0, W1, 0x5140), b0a, b0b);   // d offsets 0, 1
                e4m3x4_to_f16x2x2(prmt(W0, W1, 0x7362), b0c, b0d);   // d offsets 2, 3
                e4m3x4_to_f16x2x2(prmt(W2, W3, 0x5140), b1a, b1b);
                e4m3x4_to_f16x2x2(prmt(W2, W3, 0x7362), b1c, b1d);
                mma_f16(o[4 * qd + 0], pa, b0a, b1a);
                mma_f16(o[4 * qd + 1], pa, b0b, b1b);
                mma_f16(o[4 * qd + 2], pa, b0c, b1c);
                mma_f16(o[4 * qd + 3], pa, b0d, b1d);
            }
        }
        // The stage is next written by the async proxy (cp.async.bulk): order this
        // warp's generic reads of it before that write.
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }

    __syncthreads();     // all warps: producers done issuing, consumers done reading
    if (failed || issued_s[0] + issued_s[1] < nblk) {
        // A wait ran out: record it, let the copies already issued land (bounded)
        // and leave without touching the outputs.
        if (threadIdx.x == 0) {
            atomicOr(args.err, MLA_ERR_PIPELINE_TIMEOUT);
            for (int p = 0; p < kProducers; ++p) {
                const int cnt = issued_s[p];
                for (int k = max(0, cnt - kStages / kProducers); k < cnt; ++k) {
                    const int bb = p + kProducers * k;
                    (void)mbar_wait_bounded(&full[bb % kStages], static_cast<uint32_t>((bb / kStages) & 1));
                }
            }
        }
        return;
    }

    // ---- epilogue: l over the four warps' rows, then O * sigma / l ----
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        float l = l_run[r];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        if (c == 0) lsum_s[warp * kHeads + g + 8 * r] = l;
    }
    bar_sync_or(1, kConsumerThreads, false);
    float lt[2] = {0.0f, 0.0f};
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        lt[0] += lsum_s[w * kHeads + g];
        lt[1] += lsum_s[w * kHeads + g + 8];
    }
    // l = 0: nothing present (out 0, lse -inf). l NaN: a listed row holds a NaN
    // (out and lse NaN, as the decode statement gives).
    const float kNaN = __int_as_float(0x7FC00000);
    float mult[2], lse_r[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        mult[r] = lt[r] > 0.0f ? sigma / lt[r] : (lt[r] == 0.0f ? 0.0f : kNaN);
        lse_r[r] = lt[r] > 0.0f ? (m_ref[r] + log2f(lt[r])) * kLn2 : (lt[r] == 0.0f ? -INFINITY : kNaN);
    }
    const int hs[2] = {h_lo, h_hi};
    // Thread (g, c) holds, for head row r, dims 128w + 32c + 16e + 4q + i in
    // o[4q + i][2r + e]: 32 contiguous output values per head row.
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int h = hs[r];
        if (h >= H) continue;
        const float mm = mult[r];
        if (args.nsplit == 1) {
            __nv_bfloat16* orow = args.out + (static_cast<int64_t>(t) * H + h) * kLatent + 128 * warp + 32 * c;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {
                    uint4 v;
                    v.x = pack_bf16x2(o[8 * hq + 0][2 * r + e] * mm, o[8 * hq + 1][2 * r + e] * mm);
                    v.y = pack_bf16x2(o[8 * hq + 2][2 * r + e] * mm, o[8 * hq + 3][2 * r + e] * mm);
                    v.z = pack_bf16x2(o[8 * hq + 4][2 * r + e] * mm, o[8 * hq + 5][2 * r + e] * mm);
                    v.w = pack_bf16x2(o[8 * hq + 6][2 * r + e] * mm, o[8 * hq + 7][2 * r + e] * mm);
                    st_v4(orow + 16 * e + 8 * hq, v);
                }
            }
            if (warp == 0 && c == 0) args.lse[static_cast<int64_t>(t) * H + h] = lse_r[r];
        } else {
            const int64_t part = planned ? split : static_cast<int64_t>(t) * args.nsplit + split;
            const int64_t prow = part * H + h;
            if (warp == 0 && c == 0) args.ws_lse[prow] = lse_r[r];
            if (lt[r] == 0.0f) continue;       // lse = -inf: the merge skips this partial's o
            float* orow = args.ws_o + prow * kLatent + 128 * warp + 32 * c;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
#pragma unroll
                for (int qd = 0; qd < 4; ++qd)
                    reinterpret_cast<float4*>(orow + 16 * e + 4 * qd)[0] =
                        make_float4(o[4 * qd + 0][2 * r + e] * mm, o[4 * qd + 1][2 * r + e] * mm,
                                    o[4 * qd + 2][2 * r + e] * mm, o[4 * qd + 3][2 * r + e] * mm);
            }
        }
    }
}

// First kernel of a planned split: one CTA per token compacts the present
// entries of the token's list into plan_list[t][0 .. n_t), in position order,
// and writes n_t to plan_count[t], with the decode's rules (absent: -1 and other
// negatives, slot 0, out-of-range slots, which also set the error word; sequence
// positions mapped through the block table first). Launched with programmatic
// stream serialization; the decode after it waits for this grid before reading.
constexpr int kCompactThreads = 256;
constexpr int kCompactPer = (kListMax + kCompactThreads - 1) / kCompactThreads;

__global__ void __launch_bounds__(kCompactThreads)
mla_list_compact_kernel(const DecodeArgs args) {
    __shared__ int wtotal[kCompactThreads / 32];
    pdl_wait();
    pdl_launch_dependents();
    const int t = blockIdx.x;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int per = (args.W + kCompactThreads - 1) / kCompactThreads;    // <= kCompactPer
    const int p0 = static_cast<int>(threadIdx.x) * per;
    const int mine = max(0, min(per, args.W - p0));
    const int32_t* trow = args.topk + static_cast<int64_t>(t) * args.W + p0;
    int idxv[kCompactPer];
#pragma unroll
    for (int k = 0; k < kCompactPer; ++k) idxv[k] = (k < mine) ? __ldg(trow + k) : -1;
    if (args.page_size > 0) {
        const int sq = args.token_seq ? __ldg(args.token_seq + t) : 0;
        const bool seq_ok = sq >= 0 && sq < args.n_seq;
        const int32_t* bt = args.block_table + static_cast<int64_t>(seq_ok ? sq : 0) * args.bt_pages;
#pragma unroll
        for (int k = 0; k < kCompactPer; ++k) idxv[k] = paged_slot(args, bt, seq_ok, idxv[k]);
    }
    int cnt = 0;
#pragma unroll
    for (int k = 0; k < kCompactPer; ++k) {
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
    if (lane == 31) wtotal[warp] = incl;
    __syncthreads();
    int off = incl - cnt, n = 0;
#pragma unroll
    for (int w = 0; w < kCompactThreads / 32; ++w) {
        off += (w < warp) ? wtotal[w] : 0;
        n += wtotal[w];
    }
    int32_t* dst = args.plan_list + static_cast<int64_t>(t) * args.W;
#pragma unroll
    for (int k = 0; k < kCompactPer; ++k)
        if (idxv[k] != 0) dst[off++] = idxv[k];
    if (threadIdx.x == 0) args.plan_count[t] = n;
}

// Merge of the split partials of one (token, head): lse = ln sum_s exp(lse_s),
// out = sum_s exp(lse_s - lse) o_s, in split order; a NaN partial makes both NaN. Thread x takes dims 4x ..
// 4x + 3; the loads of kMergeBatch splits are issued together. Launched with
// programmatic stream serialization behind the decode, whose grid it waits for.
// The partials of token t are rows t * nsplit .. t * nsplit + nsplit - 1, or,
// after a planned split, the token's pieces as the decode recorded them.
constexpr int kMergeBatch = 8;

__global__ void __launch_bounds__(128)
mla_split_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                         const int2* __restrict__ plan_tok, int plan_pieces, int H, int nsplit,
                         __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
    pdl_wait();
    const int64_t th = blockIdx.x;              // t * H + h
    const int64_t t = th / H;
    const int h = static_cast<int>(th % H);
    const int d = 4 * threadIdx.x;
    int64_t row0 = t * nsplit;                  // first partial of the token
    int np = nsplit;                            // its number of partials
    if (plan_tok != nullptr) {
        const int2 pt = plan_tok[t];
        row0 = min(max(pt.x, 0), plan_pieces - 1);
        np = min(max(pt.y, 1), plan_pieces - static_cast<int>(row0));
    }
    float mx = -INFINITY;
    bool nan = false;
    for (int s0 = 0; s0 < np; s0 += kMergeBatch) {
        float ls[kMergeBatch];
#pragma unroll
        for (int q = 0; q < kMergeBatch; ++q)
            ls[q] = (s0 + q < np) ? ws_lse[(row0 + s0 + q) * H + h] : -INFINITY;
#pragma unroll
        for (int q = 0; q < kMergeBatch; ++q) {
            mx = fmaxf(mx, ls[q]);
            nan = nan || ls[q] != ls[q];
        }
    }
    __nv_bfloat16* orow = out + th * kLatent + d;
    if (nan) {
        // A split met a NaN row: the whole result is NaN, as unsplit.
        const uint32_t qn = pack_bf16x2(__int_as_float(0x7FC00000), __int_as_float(0x7FC00000));
        *reinterpret_cast<uint2*>(orow) = make_uint2(qn, qn);
        if (threadIdx.x == 0) lse[th] = __int_as_float(0x7FC00000);
        return;
    }
    if (mx == -INFINITY) {
        *reinterpret_cast<uint2*>(orow) = make_uint2(0u, 0u);
        if (threadIdx.x == 0) lse[th] = -INFINITY;
        return;
    }
    float wsum = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < np; s0 += kMergeBatch) {
        float ls[kMergeBatch];
        float4 v[kMergeBatch];
#pragma unroll
        for (int q = 0; q < kMergeBatch; ++q) {
            const int64_t prow = (row0 + min(s0 + q, np - 1)) * H + h;
            ls[q] = (s0 + q < np) ? ws_lse[prow] : -INFINITY;
            // A split with no present entry (lse -inf) left its o unwritten.
            v[q] = (ls[q] == -INFINITY) ? make_float4(0.f, 0.f, 0.f, 0.f)
                                        : *reinterpret_cast<const float4*>(ws_o + prow * kLatent + d);
        }
#pragma unroll
        for (int q = 0; q < kMergeBatch; ++q) {
            const float w = (ls[q] == -INFINITY) ? 0.0f : expf(ls[q] - mx);
            wsum += w;
            acc.x = fmaf(w, v[q].x, acc.x);
            acc.y = fmaf(w, v[q].y, acc.y);
            acc.z = fmaf(w, v[q].z, acc.z);
            acc.w = fmaf(w, v[q].w, acc.w);
        }
    }
    const float inv = 1.0f / wsum;
    *reinterpret_cast<uint2*>(orow) = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv),
                                                 pack_bf16x2(acc.z * inv, acc.w * inv));
    if (threadIdx.x == 0) lse[th] = mx + logf(wsum);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Number of splits of each token's top-k list. A split costs a partial write, a
// merge and one more prologue, so a token's list is split only when there are
// fewer (token, head group) pairs than SMs; then into enough pieces for about
// kSplitCtasPerSm CTAs per SM, each of at least kSplitMinRows positions (a
// shorter piece saves less loop time than the merge launch costs: the 4-token,
// 128-position case runs 13.4 us unsplit against 15.5 us in two pieces), and at
// most kListMax positions per split.
constexpr int kSplitCtasPerSm = 2;
constexpr int kSplitMinRows = 256;

int choose_nsplit(int T, int H, int W, int sms) {
    if (T <= 0 || W <= 0) return 1;
    const int64_t base = static_cast<int64_t>(T) * ((H + kHeads - 1) / kHeads);
    int64_t ns = 1;
    if (base < sms) ns = (static_cast<int64_t>(kSplitCtasPerSm) * sms + base - 1) / base;
    const int64_t max_ns = (W >= kSplitMinRows) ? W / kSplitMinRows : 1;
    if (ns > max_ns) ns = max_ns;
    const int64_t min_ns = (W + kListMax - 1) / kListMax;
    if (ns < min_ns) ns = min_ns;
    if (ns < 1) ns = 1;
    return static_cast<int>(ns);
}

// Lists that one CTA can compact are split by a plan (see the kernel's header):
// `pieces` piece slots per head group, one wave of CTAs at kSplitCtasPerSm per SM
// and never fewer than the tokens (T * head_groups < SMs whenever a list is
// split, so this bound is slack). Longer lists are split by positions (pieces 0).
struct Split {
    int nsplit;
    int pieces;
};

Split choose_split(int T, int H, int W, int sms) {
    Split sp{choose_nsplit(T, H, W, sms), 0};
    if (sp.nsplit > 1 && W <= kListMax && T <= kListMax) {
        const int head_groups = (H + kHeads - 1) / kHeads;
        sp.pieces = max(T, kSplitCtasPerSm * sms / head_groups);
    }
    return sp;
}

size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

// Rows of split partials: T * nsplit * H, or pieces * H when planned.
size_t partial_rows(int T, int H, const Split& sp) {
    return sp.pieces > 0 ? static_cast<size_t>(sp.pieces) * H : static_cast<size_t>(T) * sp.nsplit * H;
}

// Workspace: the partial o rows, their lse, and for a planned split the
// compacted lists [T, W], their lengths [T] and each token's pieces [T].
size_t workspace_for(int T, int H, int W, const Split& sp) {
    if (sp.nsplit <= 1) return 0;
    const size_t rows = partial_rows(T, H, sp);
    size_t bytes = rows * kLatent * sizeof(float) + align256(rows * sizeof(float));
    if (sp.pieces > 0)
        bytes += align256(static_cast<size_t>(T) * W * sizeof(int32_t)) + align256(static_cast<size_t>(T) * sizeof(int32_t)) +
                 align256(static_cast<size_t>(T) * sizeof(int2));
    return bytes;
}

}  // namespace

extern "C" size_t mla_sparse_decode_workspace_bytes(int T, int H, int W) {
    if (T <= 0 || H <= 0 || H > 128 || W < 0) return 0;
    const int sms = mla_host::sm_count();
    if (sms <= 0) return 0;
    return workspace_for(T, H, W, choose_split(T, H, W, sms));
}

namespace {

struct PageArgs {
    const int32_t* block_table;
    const int32_t* token_seq;
    int bt_pages, n_seq, page_size;
};

int launch_decode(const void* q_bf16, int T, int H, int d_qk, mla_kv_cache_t kv, const int32_t* topk_idx,
                  int W, float sm_scale, void* out_bf16, float* lse, void* workspace, size_t workspace_bytes,
                  void* stream, const PageArgs& pg) {
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
    const Split sp = choose_split(T, H, W, sms);
    const int nsplit = sp.nsplit;
    const bool planned = sp.pieces > 0;
    const size_t need = workspace_for(T, H, W, sp);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
        return MLA_ENOWORKSPACE;

    if (!mla_host::max_dynamic_smem(reinterpret_cast<const void*>(mla_sparse_decode_kernel<true, false>), kSmemTotal) ||
        !mla_host::max_dynamic_smem(reinterpret_cast<const void*>(mla_sparse_decode_kernel<false, false>), kSmemTotal) ||
        !mla_host::max_dynamic_smem(reinterpret_cast<const void*>(mla_sparse_decode_kernel<true, true>), kSmemTotal) ||
        !mla_host::max_dynamic_smem(reinterpret_cast<const void*>(mla_sparse_decode_kernel<false, true>), kSmemTotal))
        return MLA_ECUDA;
    DecodeArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q_bf16);
    a.cache = static_cast<const uint8_t*>(kv.data);
    a.topk = topk_idx;
    a.out = static_cast<__nv_bfloat16*>(out_bf16);
    a.lse = lse;
    const size_t rows = partial_rows(T, H, sp);
    a.ws_o = static_cast<float*>(workspace);
    a.ws_lse = nsplit > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + rows * kLatent * sizeof(float))
                          : nullptr;
    a.plan_list = nullptr;
    a.plan_count = nullptr;
    a.plan_tok = nullptr;
    a.plan_pieces = 0;
    if (planned) {
        uint8_t* p = reinterpret_cast<uint8_t*>(a.ws_lse) + align256(rows * sizeof(float));
        a.plan_list = reinterpret_cast<int32_t*>(p);
        p += align256(static_cast<size_t>(T) * W * sizeof(int32_t));
        a.plan_count = reinterpret_cast<int32_t*>(p);
        p += align256(static_cast<size_t>(T) * sizeof(int32_t));
        a.plan_tok = reinterpret_cast<int2*>(p);
        a.plan_pieces = sp.pieces;
    }
    a.err = err;
    a.num_slots = kv.num_slots;
    a.row_bytes = kv.row_bytes;
    a.block_table = pg.block_table;
    a.token_seq = pg.token_seq;
    a.bt_pages = pg.bt_pages;
    a.n_seq = pg.n_seq;
    a.page_size = pg.page_size;
    a.T = T; a.H = H; a.d_qk = d_qk; a.W = W; a.nsplit = nsplit;
    a.split_len = (W + nsplit - 1) / nsplit;
    a.sm_scale_log2 = sm_scale * kLog2e;
    const int head_groups = (H + kHeads - 1) / kHeads;
    const dim3 grid = planned ? dim3(static_cast<unsigned>(sp.pieces * head_groups), 1u)
                              : dim3(static_cast<unsigned>(static_cast<int64_t>(T) * head_groups), static_cast<unsigned>(nsplit));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (planned) {
        cudaLaunchConfig_t ccfg = {};
        ccfg.gridDim = dim3(static_cast<unsigned>(T));
        ccfg.blockDim = dim3(kCompactThreads);
        ccfg.stream = st;
        ccfg.attrs = attr;
        ccfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&ccfg, mla_list_compact_kernel, a) != cudaSuccess || cudaGetLastError() != cudaSuccess)
            return MLA_ECUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemTotal;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool rope = d_qk == kLatent + kRope;
    const cudaError_t lr =
        planned ? (rope ? cudaLaunchKernelEx(&cfg, mla_sparse_decode_kernel<true, true>, a)
                        : cudaLaunchKernelEx(&cfg, mla_sparse_decode_kernel<false, true>, a))
                : (rope ? cudaLaunchKernelEx(&cfg, mla_sparse_decode_kernel<true, false>, a)
                        : cudaLaunchKernelEx(&cfg, mla_sparse_decode_kernel<false, false>, a));
    if (lr != cudaSuccess || cudaGetLastError() != cudaSuccess) return MLA_ECUDA;
    if (nsplit > 1) {
        cudaLaunchConfig_t mcfg = {};
        mcfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(T) * H));
        mcfg.blockDim = dim3(128);
        mcfg.stream = st;
        mcfg.attrs = attr;
        mcfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&mcfg, mla_split_combine_kernel, static_cast<const float*>(a.ws_o),
                               static_cast<const float*>(a.ws_lse), static_cast<const int2*>(a.plan_tok), a.plan_pieces,
                               H, nsplit, a.out, a.lse) != cudaSuccess ||
            cudaGetLastError() != cudaSuccess)
            return MLA_ECUDA;
    }
    return MLA_OK;
}

}  // namespace

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
