// mla_sparse_prefill: sparse top-k MLA attention in which one CTA serves two
// adjacent tokens (16 heads each) over one stream of gathered rows.
//
// Prefill batches are where the pages send more query rows than the decode
// kernel is built for (sglang PR #39288, Motivation: above 64 query rows a
// dedicated prefill kernel runs) and where today's decode kernel also serves
// prefill (sglang PR #47013, Speed Tests: prefill uses the same kernel). In a
// causal prefill, adjacent tokens select almost the same rows: token i's list is
// a subset of token i+1's. A per-token kernel gathers and converts each such row
// once per token; here a CTA takes a pair of tokens, so each row shared by the
// pair is copied and converted once for 32 query rows.
//
// What is computed is exactly the per-token decode statement of the C header
// (out, lse of every token and head over its own present entries). The pair's
// two compacted lists are merged in shared memory into three segments, each
// starting on a 32-row block:
//   shared : rows present in both lists (the first token's order)
//   first  : rows present only in the first token's list
//   second : rows present only in the second token's list (its order)
// A block belongs to one segment, and a group computes only the blocks of the
// segments it owns. A row that only one token lists never reaches the other
// token's arithmetic: the pages' masking rule (sglang PR #47013, Motivation:
// masking the score does not stop a NaN row; sglang PR #39288, Root cause: an
// absent candidate contributes nothing) holds per token, as in the decode. When
// either list holds a slot twice, the merge is skipped (shared segment empty,
// each token's list whole in its own segment), so duplicates count as often as
// they are listed.
//
// CTA layout: 8 consumer warps and 2 copy-issuing warps (one CTA per SM: O of
// 32 query rows x 512 dims lives in the consumers' registers). Rows are copied
// global -> shared with one cp.async.bulk each (656 B, or 528 B for NoPE) into a
// 4-stage ring of 32-row blocks, as in the decode. Arithmetic per block, on
// m16n8k16 tensor-core MMAs with the query groups as two M tiles:
//   QK  : consumer warp w takes latent dims 64w .. 64w+63 (tile w/2) and RoPE
//         dims 8w .. 8w+7. Each E4M3 fragment is converted to f16 once (exact)
//         and multiplied into both groups' q; the row's tile scale multiplies
//         the partial afterwards; the RoPE slice runs as a bf16 m16n8k8 MMA.
//   softmax: the eight slice partials meet in shared memory; warp w finishes
//         group w/4, rows 8(w%4) .. +7 of the block (online max / sum in fp32
//         with exp2; the offset of a head moves only when a block maximum runs
//         more than kRescaleSlack above it, so P <= 2^8 fits the f16 operand).
//   PV  : warp w owns output dims 64w .. 64w+63 of both groups: P (f16) times
//         scale_row / sigma_group times the exact f16 codes, each converted V
//         fragment serving both groups.
// Before its first wait the CTA brings its lists and q rows into L2; the merge
// (an open-addressing table of the first list in shared memory, one lookup per
// entry of the second, one block-wide scan) takes all ten warps.
#include <cfloat>
#include <climits>
#include <cmath>

#include "mla_device.cuh"

namespace {

using namespace mla;

constexpr int kHeads = 16;                   // heads of one query group (one M tile)
constexpr int kGroups = 2;                   // query groups per CTA
constexpr int kWarps = 8;                    // consumer warps (one per 64-dim latent slice)
constexpr int kProducer = kWarps;            // warp index of the first copy-issuing warp
constexpr int kProducers = 2;
constexpr int kThreads = (kWarps + kProducers) * 32;
constexpr int kConsumerThreads = kWarps * 32;
constexpr int kNB = 32;                      // rows per block
constexpr int kStages = 4;
constexpr int kListMax = 2304;               // positions of one token's list
constexpr int kPerThread = (kListMax + kThreads - 1) / kThreads;              // compaction run
constexpr int kUnionMax = 2 * kListMax + 3 * kNB;   // three segments, each padded to a block
constexpr int kHashBits = 12;
constexpr int kHashSize = 1 << kHashBits;    // open addressing, load <= 0.57
constexpr int kStageBytes = kNB * kRowBytes;

// Shared-memory map (bytes).
constexpr int kOffList = kStages * kStageBytes;                   // int [kUnionMax]: merged list
constexpr int kOffA = kOffList + kUnionMax * 4;                   // int [kListMax]: first token's list
constexpr int kOffB = kOffA + kListMax * 4;                       // int [kListMax]: second token's list
constexpr int kOffHashKey = kOffB + kListMax * 4;                 // int [kHashSize]: slot, 0 = empty
constexpr int kOffHashPos = kOffHashKey + kHashSize * 4;          // uint16 [kHashSize]: index in the first list
constexpr int kOffClaim = kOffHashPos + kHashSize * 2;            // uint32 [kListMax / 32]: shared-row bits
constexpr int kOffRed = kOffClaim + kListMax / 8;                 // float4 [warp][group][n-tile][lane]
constexpr int kOffP = kOffRed + kWarps * kGroups * 4 * 32 * 16;   // uint2 [group][n-tile][lane]
constexpr int kOffQmax = kOffP + kGroups * 4 * 32 * 8;            // float [group][warp][16]
constexpr int kOffRmax = kOffQmax + kGroups * kWarps * kHeads * 4;   // float [group][n-tile][16]
constexpr int kOffLsum = kOffRmax + kGroups * 4 * kHeads * 4;     // float [group][n-tile][16]
constexpr int kOffMisc = kOffLsum + kGroups * 4 * kHeads * 4;     // ints: warp counts, segment sizes, issued
constexpr int kOffBar = kOffMisc + 256;                           // full + empty mbarriers
constexpr int kSmemTotal = kOffBar + 2 * kStages * 8;
static_assert(kOffBar % 8 == 0 && kOffRed % 16 == 0 && kOffList % 16 == 0, "alignment");
static_assert(kSmemTotal <= 227 * 1024, "shared memory");

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleSlack = 8.0f;

__device__ __forceinline__ float quad_max(float v) {
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
    return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}

__device__ __forceinline__ void mma_bf16_k8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(b0));
}

__device__ __forceinline__ uint32_t slot_hash(int s) {
    return (static_cast<uint32_t>(s) * 0x9E3779B1u) >> (32 - kHashBits);
}

struct PairArgs {
    const __nv_bfloat16* q;
    const uint8_t* cache;
    const int32_t* topk;
    __nv_bfloat16* out;
    float* lse;
    int* err;
    int64_t num_slots;
    int64_t row_bytes;          // 656, or 528 (NoPE rows without a tail)
    // Paged top-k (page_size > 0): entries are sequence positions, mapped to
    // slots through block_table[seq][position / page_size].
    const int32_t* block_table;
    const int32_t* token_seq;
    int bt_pages, n_seq, page_size;
    int T, H, d_qk, W;
    int head_groups;            // ceil(H / 16)
    float sm_scale_log2;        // sm_scale * log2(e)
};

// Loads `per` positions of token t's list from position p0 (all at once), maps
// them through the block table when the list holds positions, and leaves in v
// the present slots (0 for an absent entry). Returns how many are present.
__device__ __forceinline__ int load_present(const PairArgs& a, int t, int p0, int per, int (&v)[kPerThread]) {
    const int32_t* row = a.topk + static_cast<int64_t>(t) * a.W;
    const int mine = max(0, min(per, a.W - p0));
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) v[k] = (k < mine) ? __ldg(row + p0 + k) : -1;
    if (a.page_size > 0) {
        // Positions -> slots (vLLM PR #55277, Purpose item 2): a negative
        // position or an unassigned (negative) page is absent; a position past
        // the table or a sequence outside the table is absent and flagged.
        const int sq = a.token_seq ? __ldg(a.token_seq + t) : 0;
        const bool seq_ok = sq >= 0 && sq < a.n_seq;
        const int32_t* bt = a.block_table + static_cast<int64_t>(seq_ok ? sq : 0) * a.bt_pages;
#pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            const int pos = v[k];
            if (pos < 0) continue;
            const int page = pos / a.page_size;
            if (!seq_ok || page >= a.bt_pages) {
                atomicOr(a.err, MLA_ERR_DECODE_INDEX_RANGE);
                v[k] = -1;
                continue;
            }
            const int phys = __ldg(bt + page);
            const int64_t slot = static_cast<int64_t>(phys) * a.page_size + (pos - page * a.page_size);
            v[k] = (phys < 0) ? -1 : static_cast<int>(min(slot, static_cast<int64_t>(INT32_MAX)));
        }
    }
    int cnt = 0;
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        const int idx = v[k];
        const bool valid = idx > 0 && static_cast<int64_t>(idx) < a.num_slots;
        if (idx > 0 && !valid) atomicOr(a.err, MLA_ERR_DECODE_INDEX_RANGE);
        v[k] = valid ? idx : 0;
        cnt += valid ? 1 : 0;
    }
    return cnt;
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += u;
    }
    return v;
}

// Segment of block b: which groups own it (bit j = group j) and how many of its
// 32 rows are listed.
struct Segs {
    int nS, nA, nB;     // rows of the shared, first-only and second-only segments
    int bS, bA;         // blocks of the first two
};
__device__ __forceinline__ void block_info(const Segs& sg, int b, int& own, int& n_b) {
    if (b < sg.bS) {
        own = 3;
        n_b = min(kNB, sg.nS - kNB * b);
    } else if (b < sg.bS + sg.bA) {
        own = 1;
        n_b = min(kNB, sg.nA - kNB * (b - sg.bS));
    } else {
        own = 2;
        n_b = min(kNB, sg.nB - kNB * (b - sg.bS - sg.bA));
    }
}

// Group j of CTA (u, hg) is token 2u + j with heads 16 hg .. 16 hg + 15.
template <bool kRopeOn>
__global__ void __launch_bounds__(kThreads, 1)
mla_sparse_pair_kernel(const PairArgs args) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* stages = smem;
    int* list = reinterpret_cast<int*>(smem + kOffList);
    int* lst_a = reinterpret_cast<int*>(smem + kOffA);
    int* lst_b = reinterpret_cast<int*>(smem + kOffB);
    int* hkey = reinterpret_cast<int*>(smem + kOffHashKey);
    uint16_t* hpos = reinterpret_cast<uint16_t*>(smem + kOffHashPos);
    uint32_t* claim = reinterpret_cast<uint32_t*>(smem + kOffClaim);
    float4* red = reinterpret_cast<float4*>(smem + kOffRed);
    uint32_t* pbuf = reinterpret_cast<uint32_t*>(smem + kOffP);
    float* qmax_s = reinterpret_cast<float*>(smem + kOffQmax);
    float* rmax_s = reinterpret_cast<float*>(smem + kOffRmax);
    float* lsum_s = reinterpret_cast<float*>(smem + kOffLsum);
    int* wc = reinterpret_cast<int*>(smem + kOffMisc);          // [3][16] warp counts
    int* issued_s = wc + 48;                                     // [2]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* empty = full + kStages;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int H = args.H;
    constexpr uint32_t kRowRead = kRopeOn ? kRowBytes : kNopeReadBytes;

    // Pairs are taken from the last to the first: in a causal batch the later
    // tokens have the longest lists, and starting them first shortens the tail.
    // No result depends on the order.
    const int n_pairs = (args.T + 1) / 2;
    const int pair = n_pairs - 1 - static_cast<int>(blockIdx.x / args.head_groups);
    const int hgi = static_cast<int>(blockIdx.x % args.head_groups);
    const int tok[kGroups] = {2 * pair, 2 * pair + 1};
    const int hg[kGroups] = {hgi, hgi};
    const bool gvalid[kGroups] = {true, 2 * pair + 1 < args.T};
    const bool second_list = gvalid[1];

    // While the previous kernel on the stream may still be running, bring the
    // lists and q rows into L2 (a prefetch returns nothing to the kernel; every
    // load after the wait below sees the previous kernel's writes).
    {
        const int lines = (args.W * 4 + 127) / 128;
#pragma unroll
        for (int j = 0; j < kGroups; ++j) {
            if (j == 1 && !second_list) break;
            const char* lb = reinterpret_cast<const char*>(args.topk + static_cast<int64_t>(tok[j]) * args.W);
            for (int i = threadIdx.x; i < lines; i += kThreads) prefetch_l2(lb + 128 * i);
        }
#pragma unroll
        for (int j = 0; j < kGroups; ++j) {
            if (!gvalid[j]) break;
            const int nh = min(kHeads, H - hg[j] * kHeads);
            const char* qb = reinterpret_cast<const char*>(args.q + (static_cast<int64_t>(tok[j]) * H + hg[j] * kHeads) * args.d_qk);
            const int qlines = (nh * args.d_qk * 2 + 127) / 128;
            for (int i = threadIdx.x; i < qlines; i += kThreads) prefetch_l2(qb + 128 * i);
        }
    }
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        issued_s[0] = issued_s[1] = 0;
        fence_mbar_init();
    }

    // ---- 0. q of both groups (consumer warps), loads issued first ----
    // Warp w takes latent dims 64w .. 64w+63 and RoPE dims 8w .. 8w+7 of heads
    // g and g + 8 of each group.
    const int g = lane >> 2;
    const int c = lane & 3;
    uint32_t qraw[kGroups][2][8];
    uint32_t qr[kGroups][2];
#pragma unroll
    for (int j = 0; j < kGroups; ++j) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int h = hg[j] * kHeads + g + 8 * r;
            qr[j][r] = 0u;
#pragma unroll
            for (int k = 0; k < 8; ++k) qraw[j][r][k] = 0u;
            if (warp < kWarps && gvalid[j] && h < H) {
                const __nv_bfloat16* qh = args.q + (static_cast<int64_t>(tok[j]) * H + h) * args.d_qk;
                const uint8_t* p = reinterpret_cast<const uint8_t*>(qh + 64 * warp + 16 * c);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const uint4 v = ld_nc_v4(p + 16 * k);
                    qraw[j][r][4 * k + 0] = v.x; qraw[j][r][4 * k + 1] = v.y;
                    qraw[j][r][4 * k + 2] = v.z; qraw[j][r][4 * k + 3] = v.w;
                }
                if (kRopeOn) qr[j][r] = *reinterpret_cast<const uint32_t*>(qh + kLatent + 8 * warp + 2 * c);
            }
        }
    }

    // ---- 1. compact the present entries of each list (all warps) ----
    // Thread i takes a contiguous run of `per` positions; one block-wide scan of
    // the per-thread counts places the present slots in position order.
    const int per = (args.W + kThreads - 1) / kThreads;          // <= kPerThread
    const int p0 = static_cast<int>(threadIdx.x) * per;
    int va[kPerThread], vb[kPerThread];
    const int ca = load_present(args, tok[0], p0, per, va);
    int cb = 0;
    if (second_list) cb = load_present(args, tok[1], p0, per, vb);
    else {
#pragma unroll
        for (int k = 0; k < kPerThread; ++k) vb[k] = 0;
    }
    {
        const int ia = warp_incl_scan(ca, lane);
        const int ib = warp_incl_scan(cb, lane);
        if (lane == 31) { wc[warp] = ia; wc[16 + warp] = ib; }
        for (int i = threadIdx.x; i < kHashSize; i += kThreads) hkey[i] = 0;
        for (int i = threadIdx.x; i < kListMax / 32; i += kThreads) claim[i] = 0u;
        __syncthreads();
        int oa = ia - ca, ob = ib - cb, na = 0, nb = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            const int xa = wc[w], xb = wc[16 + w];
            oa += (w < warp) ? xa : 0;
            ob += (w < warp) ? xb : 0;
            na += xa;
            nb += xb;
        }
#pragma unroll
        for (int k = 0; k < kPerThread; ++k) {
            if (va[k] != 0) lst_a[oa++] = va[k];
            if (vb[k] != 0) lst_b[ob++] = vb[k];
        }
        __syncthreads();
        va[0] = na;       // carried below in registers
        vb[0] = nb;
    }
    const int na = va[0], nb = vb[0];

    Segs sg;
    {
        // ---- 2. merge the two lists into block-aligned segments (all warps) ----
        // (a) The first list into the table: slot -> index. A slot met twice
        // marks a duplicate.
        bool dup = false;
        for (int i = threadIdx.x; i < na; i += kThreads) {
            const int s = lst_a[i];
            uint32_t h = slot_hash(s);
            for (int probe = 0; probe < kHashSize; ++probe) {      // a free bucket exists: na < kHashSize
                const int prev = atomicCAS(&hkey[h], 0, s);
                if (prev == 0) { hpos[h] = static_cast<uint16_t>(i); break; }
                if (prev == s) { dup = true; break; }
                h = (h + 1) & (kHashSize - 1);
            }
        }
        __syncthreads();
        // (b) Every entry of the second list claims the matching entry of the
        // first; a claim found taken means the second list holds that slot twice.
        // Thread i takes a contiguous run of the second list, so that the entries
        // left over keep their order through the scan below.
        const int per_b = (nb + kThreads - 1) / kThreads;        // <= kPerThread
        const int b0 = static_cast<int>(threadIdx.x) * per_b;
        const int run_b = max(0, min(per_b, nb - b0));
        uint32_t only_b = 0u;                                     // bit k: entry b0 + k is not in the first list
#pragma unroll 1
        for (int k = 0; k < run_b; ++k) {
            const int s = lst_b[b0 + k];
            uint32_t h = slot_hash(s);
            bool found = false;
            for (int probe = 0; probe < kHashSize; ++probe) {
                const int key = hkey[h];
                if (key == 0) break;
                if (key == s) {
                    const int i = hpos[h];
                    const uint32_t bit = 1u << (i & 31);
                    if (atomicOr(&claim[i >> 5], bit) & bit) dup = true;
                    found = true;
                    break;
                }
                h = (h + 1) & (kHashSize - 1);
            }
            if (!found) only_b |= 1u << k;
        }
        // With a duplicate anywhere the lists are not merged: each goes whole
        // into its own segment (the result is the same; only the sharing is lost).
        const bool any_dup = __syncthreads_or(dup) != 0;
        if (any_dup) only_b = (run_b >= 32) ? 0xffffffffu : ((1u << run_b) - 1u);
        // (c) Shared rows in the first list's order, then the first list's own
        // rows, then the second list's own rows, each segment from a block start.
        const int per_a = (na + kThreads - 1) / kThreads;        // <= kPerThread
        const int a0 = static_cast<int>(threadIdx.x) * per_a;
        const int run_a = max(0, min(per_a, na - a0));
        int cs = 0;
#pragma unroll 1
        for (int k = 0; k < run_a; ++k) {
            const int i = a0 + k;
            cs += (!any_dup && ((claim[i >> 5] >> (i & 31)) & 1u)) ? 1 : 0;
        }
        const int cA = run_a - cs;
        const int cB = __popc(only_b);
        const int is = warp_incl_scan(cs, lane);
        const int iA = warp_incl_scan(cA, lane);
        const int iB = warp_incl_scan(cB, lane);
        if (lane == 31) { wc[warp] = is; wc[16 + warp] = iA; wc[32 + warp] = iB; }
        __syncthreads();
        int os = is - cs, oA = iA - cA, oB = iB - cB, nS = 0, nA = 0, nB = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            const int xs = wc[w], xA = wc[16 + w], xB = wc[32 + w];
            os += (w < warp) ? xs : 0;
            oA += (w < warp) ? xA : 0;
            oB += (w < warp) ? xB : 0;
            nS += xs; nA += xA; nB += xB;
        }
        const int baseA = (nS + kNB - 1) / kNB * kNB;
        const int baseB = baseA + (nA + kNB - 1) / kNB * kNB;
#pragma unroll 1
        for (int k = 0; k < run_a; ++k) {
            const int i = a0 + k;
            const bool shared = !any_dup && ((claim[i >> 5] >> (i & 31)) & 1u);
            if (shared) list[os++] = lst_a[i];
            else list[baseA + oA++] = lst_a[i];
        }
#pragma unroll 1
        for (int k = 0; k < run_b; ++k)
            if ((only_b >> k) & 1u) list[baseB + oB++] = lst_b[b0 + k];
        __syncthreads();
        sg.nS = nS; sg.nA = nA; sg.nB = nB;
        sg.bS = (nS + kNB - 1) / kNB;
        sg.bA = (nA + kNB - 1) / kNB;
    }
    const int nblk = sg.bS + sg.bA + (sg.nB + kNB - 1) / kNB;

    if (warp >= kProducer) {
        // ---- producers: warp kProducer + p issues blocks p, p + kProducers, ...;
        // lane j copies row j of the block into the stage ring ----
        const int pw = warp - kProducer;
        int b = pw, cnt = 0;
        for (; b < nblk; b += kProducers, ++cnt) {
            const int s = b % kStages;
            if (b >= kStages && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>(((b / kStages) - 1) & 1))) {
                if (lane == 0) atomicOr(args.err, MLA_ERR_PIPELINE_TIMEOUT);
                break;
            }
            uint8_t* dst = stages + s * kStageBytes;
            int own, n_b;
            block_info(sg, b, own, n_b);
            if (n_b < kNB) {
                // Rows past the end of a segment load nothing: zero them so the
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
                         args.cache + static_cast<int64_t>(list[kNB * b + lane]) * args.row_bytes, kRowRead, &full[s]);
        }
        if (lane == 0) issued_s[pw] = cnt;
        __syncthreads();     // matches the consumers' final barrier
        return;
    }

    // ---- consumers: q fragments of both groups ----
#pragma unroll
    for (int j = 0; j < kGroups; ++j) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float m = 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k) m = fmaxf(m, fmaxf(fabsf(bf16lo(qraw[j][r][k])), fabsf(bf16hi(qraw[j][r][k]))));
            m = fmaxf(m, fmaxf(fabsf(bf16lo(qr[j][r])), fabsf(bf16hi(qr[j][r]))));
            m = quad_max(m);
            if (c == 0) qmax_s[(j * kWarps + warp) * kHeads + g + 8 * r] = m;
        }
    }
    bar_sync_or(1, kConsumerThreads, false);
    const int snt = warp & 3;                  // n-tile whose scores this warp finishes
    const int gq = warp >> 2;                  // group whose scores this warp finishes
    const int tile = warp >> 1;                // scale tile of the warp's latent slice
    // Exponent-only rescale so that |q| < 2^15 in f16 (exact in f16's normal
    // range); the same power of two scales the RoPE part, and is undone on the
    // scores through the per-row softmax factor.
    float qdown[kGroups][2], rowf[2];
#pragma unroll
    for (int j = 0; j < kGroups; ++j) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float mx = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, qmax_s[(j * kWarps + w) * kHeads + g + 8 * r]);
            int e = 0;
            frexpf(mx, &e);                          // mx < 2^e
            const int k = (e > 15) ? (e - 15) : 0;
            qdown[j][r] = ldexpf(1.0f, -k);
            if (j == gq) rowf[r] = args.sm_scale_log2 * ldexpf(1.0f, k);
        }
    }
    // A fragments of k-step kk: dims 16c + 4kk + {0,1} (a0, a1) and + {2,3} (a2,
    // a3) of the warp's slice, the same dims the B fragments take from word kk of
    // a row's 16 bytes at 64w + 16c.
    uint32_t qa[kGroups][4][4];
    uint32_t qra[kGroups][2];
#pragma unroll
    for (int j = 0; j < kGroups; ++j) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            qa[j][kk][0] = pack_f16x2(bf16lo(qraw[j][0][2 * kk]) * qdown[j][0], bf16hi(qraw[j][0][2 * kk]) * qdown[j][0]);
            qa[j][kk][1] = pack_f16x2(bf16lo(qraw[j][1][2 * kk]) * qdown[j][1], bf16hi(qraw[j][1][2 * kk]) * qdown[j][1]);
            qa[j][kk][2] = pack_f16x2(bf16lo(qraw[j][0][2 * kk + 1]) * qdown[j][0], bf16hi(qraw[j][0][2 * kk + 1]) * qdown[j][0]);
            qa[j][kk][3] = pack_f16x2(bf16lo(qraw[j][1][2 * kk + 1]) * qdown[j][1], bf16hi(qraw[j][1][2 * kk + 1]) * qdown[j][1]);
        }
        qra[j][0] = pack_bf16x2(bf16lo(qr[j][0]) * qdown[j][0], bf16hi(qr[j][0]) * qdown[j][0]);
        qra[j][1] = pack_bf16x2(bf16lo(qr[j][1]) * qdown[j][1], bf16hi(qr[j][1]) * qdown[j][1]);
    }

    // ---- consumers: main loop ----
    // Per 32-row block: (1) QK partials of slice `warp` for the owning groups,
    // (2) the eight slice partials meet in shared memory and warp w finishes the
    // scores of group w/4, n-tile w%4 and writes their P, (3) every warp
    // multiplies P of the owning groups into V of its own slice.
    float o[kGroups][8][4];
#pragma unroll
    for (int j = 0; j < kGroups; ++j)
#pragma unroll
        for (int i = 0; i < 8; ++i) o[j][i][0] = o[j][i][1] = o[j][i][2] = o[j][i][3] = 0.0f;
    float m_ref[kGroups][2];                   // exp2 offset per group and head row (log2 units)
    float sigma[kGroups], inv_sigma[kGroups];  // running max of tile `tile`'s scales over the group's rows
#pragma unroll
    for (int j = 0; j < kGroups; ++j) {
        m_ref[j][0] = m_ref[j][1] = -INFINITY;
        sigma[j] = FLT_MIN;
        inv_sigma[j] = 1.0f / FLT_MIN;
    }
    float l_run[2] = {0.0f, 0.0f};             // sum of p over this warp's rows, group gq, heads g and g + 8
    bool failed = false;

    for (int b = 0; b < nblk; ++b) {
        const int s = b % kStages;
        const bool ok = mbar_wait_bounded(&full[s], static_cast<uint32_t>((b / kStages) & 1));
        const uint8_t* st = stages + s * kStageBytes;
        int own, n_b;
        block_info(sg, b, own, n_b);
        const bool act[kGroups] = {(own & 1) != 0, (own & 2) != 0};

        // (1) QK^T of slice `warp`: latent on f16 MMA; the tile scale, then the
        // RoPE slice (bf16 MMA, k = 8) into the same accumulator. Two n-tiles at a
        // time, which keeps the accumulators of both groups and the raw rows
        // within the register budget of ten warps per SM.
        // Scales of tile `tile` for rows nt*8 + 2c + e (rows past n_b were
        // zero-filled: scale 0); the same registers serve the PV step.
        float sc[4][2];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float acc[kGroups][2][4];
#pragma unroll
            for (int j = 0; j < kGroups; ++j)
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[j][u][i] = 0.0f;
            uint4 kv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u)
                kv[u] = *reinterpret_cast<const uint4*>(st + ((2 * half + u) * 8 + g) * kRowBytes + 64 * warp + 16 * c);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint32_t wrd = kk == 0 ? kv[u].x : kk == 1 ? kv[u].y : kk == 2 ? kv[u].z : kv[u].w;
                    uint32_t b0, b1;
                    e4m3x4_to_f16x2x2(wrd, b0, b1);
#pragma unroll
                    for (int j = 0; j < kGroups; ++j)
                        if (act[j]) mma_f16(acc[j][u], qa[j][kk], b0, b1);
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    sc[2 * half + u][e] =
                        *reinterpret_cast<const float*>(st + ((2 * half + u) * 8 + 2 * c + e) * kRowBytes + kScaleOff + 4 * tile);
            uint32_t rb[2] = {0u, 0u};
            if (kRopeOn) {
#pragma unroll
                for (int u = 0; u < 2; ++u)
                    rb[u] = *reinterpret_cast<const uint32_t*>(st + ((2 * half + u) * 8 + g) * kRowBytes + kTailOff + 16 * warp + 4 * c);
            }
#pragma unroll
            for (int j = 0; j < kGroups; ++j) {
                if (!act[j]) continue;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int nt = 2 * half + u;
                    acc[j][u][0] *= sc[nt][0];
                    acc[j][u][1] *= sc[nt][1];
                    acc[j][u][2] *= sc[nt][0];
                    acc[j][u][3] *= sc[nt][1];
                    if (kRopeOn) mma_bf16_k8(acc[j][u], qra[j][0], qra[j][1], rb[u]);
                    red[((warp * kGroups + j) * 4 + nt) * 32 + lane] =
                        make_float4(acc[j][u][0], acc[j][u][1], acc[j][u][2], acc[j][u][3]);
                }
            }
        }
        // The part of PV that does not need P, ahead of the barriers: sigma of
        // each owning group (the running max of the tile's scales over the rows
        // that group has seen, so p * scale / sigma <= 2^8 in f16), O rescaled
        // when it moves, and the rows' scale / sigma as f16 pairs.
        float smax = 0.0f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) smax = fmaxf(smax, fmaxf(sc[nt][0], sc[nt][1]));
        smax = quad_max(smax);                 // all 32 rows: the same in every lane
        uint32_t rs[kGroups][2][2];
#pragma unroll
        for (int j = 0; j < kGroups; ++j) {
            if (act[j] && smax > sigma[j]) {
                const float f = sigma[j] / smax;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    o[j][i][0] *= f; o[j][i][1] *= f; o[j][i][2] *= f; o[j][i][3] *= f;
                }
                sigma[j] = smax;
                inv_sigma[j] = 1.0f / smax;
            }
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                rs[j][kb][0] = pack_f16x2(sc[2 * kb][0] * inv_sigma[j], sc[2 * kb][1] * inv_sigma[j]);
                rs[j][kb][1] = pack_f16x2(sc[2 * kb + 1][0] * inv_sigma[j], sc[2 * kb + 1][1] * inv_sigma[j]);
            }
        }
        // Barrier 1 also carries a timeout of any warp to all of them.
        if (bar_sync_or(1, kConsumerThreads, !ok)) { failed = true; break; }

        // (2) scores of group gq, n-tile snt: rows 8 snt + 2c + {0, 1}, heads g
        // and g + 8 of the group.
        const bool mine = gq ? act[1] : act[0];
        float sv[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float p[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        float mr0 = gq ? m_ref[1][0] : m_ref[0][0];
        float mr1 = gq ? m_ref[1][1] : m_ref[0][1];
        bool need = false;
        uint2* pw = reinterpret_cast<uint2*>(pbuf) + (gq * 4 + snt) * 32 + lane;
        if (mine) {
            float4 a = red[((0 * kGroups + gq) * 4 + snt) * 32 + lane];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) {
                const float4 bq = red[((w * kGroups + gq) * 4 + snt) * 32 + lane];
                a.x += bq.x; a.y += bq.y; a.z += bq.z; a.w += bq.w;
            }
            sv[0] = a.x * rowf[0]; sv[1] = a.y * rowf[0];
            sv[2] = a.z * rowf[1]; sv[3] = a.w * rowf[1];
            if (n_b < kNB) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (8 * snt + 2 * c + (i & 1) >= n_b) sv[i] = -INFINITY;
            }
            const float bm0 = quad_max(fmaxf(sv[0], sv[1]));
            const float bm1 = quad_max(fmaxf(sv[2], sv[3]));
            if (c == 0) {
                rmax_s[(gq * 4 + snt) * kHeads + g] = bm0;
                rmax_s[(gq * 4 + snt) * kHeads + g + 8] = bm1;
            }
            need = bm0 > mr0 + kRescaleSlack || bm1 > mr1 + kRescaleSlack;
            // A row past the segment's end is -inf: p = 0 whatever the offset.
            p[0] = sv[0] == -INFINITY ? 0.0f : ex2_approx(sv[0] - mr0);
            p[1] = sv[1] == -INFINITY ? 0.0f : ex2_approx(sv[1] - mr0);
            p[2] = sv[2] == -INFINITY ? 0.0f : ex2_approx(sv[2] - mr1);
            p[3] = sv[3] == -INFINITY ? 0.0f : ex2_approx(sv[3] - mr1);
            *pw = make_uint2(pack_f16x2(p[0], p[1]), pack_f16x2(p[2], p[3]));
        }
        // V rows of the first PV step: loaded before barrier 2 (they do not depend on P).
        const uint8_t* vb = st + 64 * warp + 8 * g;
        uint2 Vn[4];
        Vn[0] = *reinterpret_cast<const uint2*>(vb + (2 * c + 0) * kRowBytes);
        Vn[1] = *reinterpret_cast<const uint2*>(vb + (2 * c + 1) * kRowBytes);
        Vn[2] = *reinterpret_cast<const uint2*>(vb + (2 * c + 8) * kRowBytes);
        Vn[3] = *reinterpret_cast<const uint2*>(vb + (2 * c + 9) * kRowBytes);
        if (bar_sync_or(1, kConsumerThreads, need)) {
            // Rare after a group's first block: move the offsets of the heads
            // whose block maximum ran ahead, rescale O and l, and rewrite P.
#pragma unroll
            for (int j = 0; j < kGroups; ++j) {
                if (!act[j]) continue;
                float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    M0 = fmaxf(M0, rmax_s[(j * 4 + nt) * kHeads + g]);
                    M1 = fmaxf(M1, rmax_s[(j * 4 + nt) * kHeads + g + 8]);
                }
                const float mn0 = (M0 > m_ref[j][0] + kRescaleSlack) ? M0 : m_ref[j][0];
                const float mn1 = (M1 > m_ref[j][1] + kRescaleSlack) ? M1 : m_ref[j][1];
                const float a0 = (mn0 == m_ref[j][0]) ? 1.0f : ex2_approx(m_ref[j][0] - mn0);   // -inf -> 0
                const float a1 = (mn1 == m_ref[j][1]) ? 1.0f : ex2_approx(m_ref[j][1] - mn1);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    o[j][i][0] *= a0; o[j][i][1] *= a0; o[j][i][2] *= a1; o[j][i][3] *= a1;
                }
                if (j == gq) {
                    l_run[0] *= a0;
                    l_run[1] *= a1;
                }
                m_ref[j][0] = mn0;
                m_ref[j][1] = mn1;
            }
            if (mine) {
                mr0 = gq ? m_ref[1][0] : m_ref[0][0];
                mr1 = gq ? m_ref[1][1] : m_ref[0][1];
                p[0] = sv[0] == -INFINITY ? 0.0f : ex2_approx(sv[0] - mr0);
                p[1] = sv[1] == -INFINITY ? 0.0f : ex2_approx(sv[1] - mr0);
                p[2] = sv[2] == -INFINITY ? 0.0f : ex2_approx(sv[2] - mr1);
                p[3] = sv[3] == -INFINITY ? 0.0f : ex2_approx(sv[3] - mr1);
                *pw = make_uint2(pack_f16x2(p[0], p[1]), pack_f16x2(p[2], p[3]));
            }
            bar_sync_or(1, kConsumerThreads, false);
        }
        l_run[0] += p[0] + p[1];
        l_run[1] += p[2] + p[3];

        // (3) PV of slice `warp` for the owning groups; each converted V
        // fragment serves both.
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            // A: P of heads (g, g+8) x rows 16kb + 2c + {0,1} and + 8, times the
            // row's tile scale / sigma of the group.
            uint32_t pa[kGroups][4];
#pragma unroll
            for (int j = 0; j < kGroups; ++j) {
                const uint2* pr = reinterpret_cast<const uint2*>(pbuf) + (j * 4) * 32 + lane;
                const uint2 plo = act[j] ? pr[(2 * kb) * 32] : make_uint2(0u, 0u);
                const uint2 phi = act[j] ? pr[(2 * kb + 1) * 32] : make_uint2(0u, 0u);
                pa[j][0] = hmul2(plo.x, rs[j][kb][0]);
                pa[j][1] = hmul2(plo.y, rs[j][kb][0]);
                pa[j][2] = hmul2(phi.x, rs[j][kb][1]);
                pa[j][3] = hmul2(phi.y, rs[j][kb][1]);
            }
            // B: V rows j0, j0+1, j0+8, j0+9; lane g takes dims 64w + 8g .. +7, so
            // n-tile (q, i) column n is dim 64w + 8n + 4q + i.
            const int j0 = 16 * kb + 2 * c;
            const uint2 V0 = kb == 0 ? Vn[0] : *reinterpret_cast<const uint2*>(vb + (j0 + 0) * kRowBytes);
            const uint2 V1 = kb == 0 ? Vn[1] : *reinterpret_cast<const uint2*>(vb + (j0 + 1) * kRowBytes);
            const uint2 V2 = kb == 0 ? Vn[2] : *reinterpret_cast<const uint2*>(vb + (j0 + 8) * kRowBytes);
            const uint2 V3 = kb == 0 ? Vn[3] : *reinterpret_cast<const uint2*>(vb + (j0 + 9) * kRowBytes);
#pragma unroll
            for (int qd = 0; qd < 2; ++qd) {
                const uint32_t W0 = qd == 0 ? V0.x : V0.y;
                const uint32_t W1 = qd == 0 ? V1.x : V1.y;
                const uint32_t W2 = qd == 0 ? V2.x : V2.y;
                const uint32_t W3 = qd == 0 ? V3.x : V3.y;
                uint32_t b0a, b0b, b0c, b0d, b1a, b1b, b1c, b1d;
                e4m3x4_to_f16x2x2(prmt(W0, W1, 0x5140), b0a, b0b);   // d offsets 0, 1
                e4m3x4_to_f16x2x2(prmt(W0, W1, 0x7362), b0c, b0d);   // d offsets 2, 3
                e4m3x4_to_f16x2x2(prmt(W2, W3, 0x5140), b1a, b1b);
                e4m3x4_to_f16x2x2(prmt(W2, W3, 0x7362), b1c, b1d);
#pragma unroll
                for (int j = 0; j < kGroups; ++j) {
                    if (!act[j]) continue;
                    mma_f16(o[j][4 * qd + 0], pa[j], b0a, b1a);
                    mma_f16(o[j][4 * qd + 1], pa[j], b0b, b1b);
                    mma_f16(o[j][4 * qd + 2], pa[j], b0c, b1c);
                    mma_f16(o[j][4 * qd + 3], pa[j], b0d, b1d);
                }
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
            for (int pp = 0; pp < kProducers; ++pp) {
                const int cnt = issued_s[pp];
                for (int k = max(0, cnt - kStages / kProducers); k < cnt; ++k) {
                    const int bb = pp + kProducers * k;
                    (void)mbar_wait_bounded(&full[bb % kStages], static_cast<uint32_t>((bb / kStages) & 1));
                }
            }
        }
        return;
    }

    // ---- epilogue: l over the four n-tiles' rows of each group, then O * sigma / l ----
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        float l = l_run[r];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        if (c == 0) lsum_s[(gq * 4 + snt) * kHeads + g + 8 * r] = l;
    }
    bar_sync_or(1, kConsumerThreads, false);
#pragma unroll
    for (int j = 0; j < kGroups; ++j) {
        if (!gvalid[j]) continue;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int h = hg[j] * kHeads + g + 8 * r;
            if (h >= H) continue;
            float lt = 0.0f;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) lt += lsum_s[(j * 4 + nt) * kHeads + g + 8 * r];
            // l = 0: nothing present (out 0, lse -inf); l NaN: a listed row holds a NaN.
            const float mm = lt > 0.0f ? sigma[j] / lt : (lt == 0.0f ? 0.0f : __int_as_float(0x7FC00000));
            // Thread (g, c) holds, for head row r, dims 64w + 16c + 8e + 4q + i in
            // o[j][4q + i][2r + e]: 16 contiguous output values per head row.
            __nv_bfloat16* orow = args.out + (static_cast<int64_t>(tok[j]) * H + h) * kLatent + 64 * warp + 16 * c;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                uint4 v;
                v.x = pack_bf16x2(o[j][0][2 * r + e] * mm, o[j][1][2 * r + e] * mm);
                v.y = pack_bf16x2(o[j][2][2 * r + e] * mm, o[j][3][2 * r + e] * mm);
                v.z = pack_bf16x2(o[j][4][2 * r + e] * mm, o[j][5][2 * r + e] * mm);
                v.w = pack_bf16x2(o[j][6][2 * r + e] * mm, o[j][7][2 * r + e] * mm);
                st_v4(orow + 8 * e, v);
            }
            if (warp == 0 && c == 0)
                args.lse[static_cast<int64_t>(tok[j]) * H + h] =
                    lt > 0.0f ? (m_ref[j][r] + log2f(lt)) * kLn2 : (lt == 0.0f ? -INFINITY : __int_as_float(0x7FC00000));
        }
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace {

int launch_prefill(const void* q_bf16, int T, int H, int d_qk, mla_kv_cache_t kv, const int32_t* topk, int W,
                   float sm_scale, void* out_bf16, float* lse, void* stream, const int32_t* block_table,
                   const int32_t* token_seq, int bt_pages, int n_seq, int page_size) {
    if (T < 0 || W < 0 || kv.num_slots < 0 || !std::isfinite(sm_scale)) return MLA_EINVAL;
    if (kv.row_bytes != MLA_ROW_BYTES && kv.row_bytes != MLA_ROW_BYTES_NOPE) return MLA_EINVAL;
    if (d_qk != kLatent && d_qk != kLatent + kRope) return MLA_EUNSUPPORTED;
    if (kv.row_bytes == MLA_ROW_BYTES_NOPE && d_qk != kLatent) return MLA_EUNSUPPORTED;   // no tail to read
    if (H < 1 || H > 128 || W > kListMax) return MLA_EUNSUPPORTED;
    if (T == 0) return MLA_OK;
    if (q_bf16 == nullptr || out_bf16 == nullptr || lse == nullptr || (W > 0 && topk == nullptr) ||
        (W > 0 && kv.data == nullptr))
        return MLA_EINVAL;
    if (!aligned16(q_bf16) || !aligned16(out_bf16) || (kv.data && !aligned16(kv.data)) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(topk) & 3u))
        return MLA_EINVAL;
    int* err = mla_host::device_error_word();
    if (err == nullptr) return MLA_ECUDA;
    const bool rope = d_qk == kLatent + kRope;
    const void* kern = rope ? reinterpret_cast<const void*>(mla_sparse_pair_kernel<true>)
                            : reinterpret_cast<const void*>(mla_sparse_pair_kernel<false>);
    if (!mla_host::max_dynamic_smem(kern, kSmemTotal)) return MLA_ECUDA;

    PairArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q_bf16);
    a.cache = static_cast<const uint8_t*>(kv.data);
    a.topk = topk;
    a.out = static_cast<__nv_bfloat16*>(out_bf16);
    a.lse = lse;
    a.err = err;
    a.num_slots = kv.num_slots;
    a.row_bytes = kv.row_bytes;
    a.block_table = block_table;
    a.token_seq = token_seq;
    a.bt_pages = bt_pages;
    a.n_seq = n_seq;
    a.page_size = page_size;
    a.T = T; a.H = H; a.d_qk = d_qk; a.W = W;
    a.head_groups = (H + kHeads - 1) / kHeads;
    a.sm_scale_log2 = sm_scale * kLog2e;
    const int64_t units = (static_cast<int64_t>(T) + 1) / 2 * a.head_groups;
    if (units > INT32_MAX) return MLA_EUNSUPPORTED;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemTotal;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t lr = rope ? cudaLaunchKernelEx(&cfg, mla_sparse_pair_kernel<true>, a)
                                : cudaLaunchKernelEx(&cfg, mla_sparse_pair_kernel<false>, a);
    if (lr != cudaSuccess || cudaGetLastError() != cudaSuccess) return MLA_ECUDA;
    return MLA_OK;
}

}  // namespace

extern "C" int mla_sparse_prefill(const void* q_bf16, int T, int H, int d_qk, mla_kv_cache_t kv,
                                  const int32_t* topk_idx, int W, float sm_scale, void* out_bf16, float* lse,
                                  void* stream) {
    return launch_prefill(q_bf16, T, H, d_qk, kv, topk_idx, W, sm_scale, out_bf16, lse, stream, nullptr, nullptr, 0,
                          0, 0);
}

extern "C" int mla_sparse_prefill_paged(const void* q_bf16, int T, int H, int d_qk, mla_kv_cache_t kv,
                                        const int32_t* topk_pos, int W, const int32_t* block_table, int n_seq,
                                        int max_pages, const int32_t* token_seq, int page_size, float sm_scale,
                                        void* out_bf16, float* lse, void* stream) {
    if (page_size <= 0 || max_pages <= 0 || n_seq <= 0 || block_table == nullptr ||
        (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(token_seq) & 3u))
        return MLA_EINVAL;
    return launch_prefill(q_bf16, T, H, d_qk, kv, topk_pos, W, sm_scale, out_bf16, lse, stream, block_table,
                          token_seq, max_pages, n_seq, page_size);
}
