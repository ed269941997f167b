/*
 * libmlasparse - FP8 MLA KV cache writer and sparse top-k MLA decode on one
 * GB300 GPU (sm_103a). Plain C ABI: device pointers, sizes, a CUDA stream.
 *
 * Row layout (vLLM PR #55277 "Support NoPE sparse MLA (GLM-5.3-Flash) on the
 * FlashInfer SM120 backend", Purpose item 1): every cache slot is one 656-byte
 * row
 *     bytes [  0, 512)  512 E4M3 latent values, value i at byte i, in four
 *                       tiles of 128 values (tile t = bytes 128t .. 128t+127)
 *     bytes [512, 528)  four little-endian fp32 tile scales, tile t at 512 + 4t
 *     bytes [528, 656)  64 bf16 RoPE values, or 128 zero bytes for NoPE rows
 * and a stored value decodes as e4m3(byte) * scale[tile].
 *
 * Slot 0 is reserved (sglang PR #47013 "zero-RoPE writer skips reserved slot 0",
 * Summary and Motivation): the allocators never hand it out, padding rows aim
 * at it, and no write may land there.
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers on the current CUDA device, owned
 *     by the caller; the library never allocates, frees or retains them.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Calls are asynchronous on that stream.
 *   - The return value is MLA_OK (0) or a negative MLA_E* code; arguments are
 *     validated on the host before any launch and nothing is launched on error.
 *     No C++ exception crosses this boundary.
 *   - Range violations found on the device (a slot or a top-k index past the
 *     cache) never trap: the row or entry is dropped and a bit is set in the
 *     library's device error word, read with mla_get_error().
 */
#ifndef MLASPARSE_H
#define MLASPARSE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- row layout (vLLM PR #55277, Purpose item 1) ---- */
#define MLA_ROW_BYTES      656
#define MLA_LATENT_DIM     512
#define MLA_TILE_VALUES    128
#define MLA_NUM_TILES      4
#define MLA_SCALE_OFFSET   512
#define MLA_TAIL_OFFSET    528
#define MLA_ROPE_DIM       64
#define MLA_FP8_MAX        448.0f   /* largest finite E4M3 value */
/* The canonical NoPE row of flashinfer#5075 (sglang PR #39288, "Relation to
 * other changes"): the 656-byte row without its 128-byte tail. */
#define MLA_ROW_BYTES_NOPE 528

/* ---- return codes ---- */
#define MLA_OK             0
#define MLA_EINVAL        (-1)   /* null pointer, negative size, misaligned pointer, bad layout */
#define MLA_EUNSUPPORTED  (-2)   /* d_qk not in {512, 576}, H outside [1, 128] */
#define MLA_ENOWORKSPACE  (-3)   /* workspace NULL or smaller than mla_sparse_decode_workspace_bytes() */
#define MLA_ECUDA         (-4)   /* a CUDA runtime call or a kernel launch failed */

/* ---- device error word bits (mla_get_error) ---- */
#define MLA_ERR_WRITE_SLOT_RANGE   0x1  /* mla_kv_write: slot >= num_slots, row dropped */
#define MLA_ERR_DECODE_INDEX_RANGE 0x2  /* mla_sparse_decode: index >= num_slots, entry absent */
#define MLA_ERR_PIPELINE_TIMEOUT   0x4  /* a kernel's bounded wait on its own copies ran out */
#define MLA_ERR_GATHER_INDEX_RANGE 0x8  /* mla_gather_upconvert: slot >= num_slots, zero row */

/* A cache: `data` is a device array of num_slots rows of row_bytes bytes,
 * 16-byte aligned. row_bytes is MLA_ROW_BYTES (656), or MLA_ROW_BYTES_NOPE
 * (528) for a cache of NoPE rows only: latent and scales at the same offsets,
 * no tail. A 528-byte cache takes only NoPE calls (rope_bf16 NULL, d_qk 512,
 * pe_dim 0); others return MLA_EINVAL or MLA_EUNSUPPORTED. */
typedef struct {
    void*   data;
    int64_t num_slots;
    int64_t row_bytes;
} mla_kv_cache_t;

/*
 * mla_kv_write - per-token FP8 quantise-and-scatter into packed rows.
 *
 * Defined by vLLM PR #55277 (Purpose item 1: the 656-byte row; NoPE rows zero
 * the 128-byte tail; pe_dim must be 64 or 0) and sglang PR #47013 (Summary,
 * Motivation, Modifications: rows aimed at the reserved slot are dropped; BF16
 * NaNs are kept by the quantiser, not clamped).
 *
 * For each row r in [0, n_rows) with s = slot_idx[r]:
 *   - s == reserved_slot or s < 0: the row is dropped and none of its inputs is
 *     read (its latent may hold NaN);
 *   - s >= kv.num_slots: the row is dropped and MLA_ERR_WRITE_SLOT_RANGE is set;
 *   - otherwise row s of the cache is overwritten: for each tile t,
 *       scale_t = amax_t / 448 (IEEE fp32 division; 1.0 when amax_t == 0;
 *                 amax ignores NaN),
 *       byte    = e4m3 round-to-nearest-even, saturating to +-448, of x / scale_t
 *                 (IEEE fp32 division; a NaN x gives the NaN code 0x7F),
 *     the four scales go to bytes 512..527, and bytes 528..655 receive rope row r
 *     verbatim, or zeros when rope_bf16 is NULL (a 528-byte row has no tail).
 * No other byte of the cache is touched.
 *
 * Arguments:
 *   kv            cache (device, 16-byte aligned, row_bytes 656, or 528 with
 *                 rope_bf16 NULL)
 *   slot_idx      int64 [n_rows], device
 *   latent_bf16   bf16 [n_rows, 512] row-major, device, 16-byte aligned
 *   rope_bf16     bf16 [n_rows, 64] row-major, device, 16-byte aligned; or NULL
 *                 for pe_dim = 0 (NoPE)
 *   n_rows        >= 0 (0 launches nothing)
 *   reserved_slot the slot writes must never land in (0 in every caller)
 * Precondition: no two rows of one call name the same non-reserved slot (which
 * of them would land is unspecified).
 * Ordering: the writer is launched with programmatic stream serialization: its
 * CTAs may become resident while the previous kernel on the stream finishes, and
 * they read nothing (slot indices, inputs, cache) until that kernel and its
 * memory are complete (griddepcontrol.wait). It also lets the next kernel on the
 * stream begin launching while it runs; only a kernel launched with programmatic
 * stream serialization can start early, and such a kernel must wait for its
 * predecessor before reading the cache, as mla_sparse_decode and the writer
 * itself do. Ordinary launches and copies are ordered as usual.
 * Returns MLA_OK, MLA_EINVAL or MLA_ECUDA.
 */
int mla_kv_write(mla_kv_cache_t kv, const int64_t* slot_idx, const void* latent_bf16,
                 const void* rope_bf16, int64_t n_rows, int64_t reserved_slot, void* stream);

/*
 * mla_sparse_decode_workspace_bytes - bytes of device workspace that
 * mla_sparse_decode needs for these sizes on the CURRENT device (the split of
 * the top-k list across CTAs depends on the device's SM count). 0 means no
 * workspace is needed. Returns 0 for invalid sizes as well.
 */
size_t mla_sparse_decode_workspace_bytes(int T, int H, int W);

/*
 * mla_sparse_decode - sparse top-k MLA decode over the packed FP8 cache.
 *
 * Sparse top-k MLA attention over the listed rows, written out below, with the
 * masking rules of sglang PR #47013 (Motivation: unused top-k entries must not
 * reach the result, even when slot 0 holds NaN), sglang PR #39288 ("SM120
 * sparse MLA: zero-initialise the page-split scratch", Root cause: a -1
 * candidate contributes nothing and must not gather slot 0), and vLLM PR #55277 (Purpose item 2: the index buffer
 * width W is a capacity; the active entries are bounded by the -1 padding;
 * Purpose item 1 and "Relation to #53969": NoPE decode reads no tail).
 *
 * For each token t < T and head h < H, with J = { j : 0 < topk_idx[t,j] <
 * kv.num_slots } (-1 or any negative, the reserved slot 0, and out-of-range
 * indices are absent: never dereferenced, contributing nothing; an index >=
 * num_slots also sets MLA_ERR_DECODE_INDEX_RANGE):
 *   s_j       = sm_scale * ( q[t,h,0:512] . K_j  +  [d_qk == 576] q[t,h,512:576] . rope_j )
 *   K_j[d]    = e4m3(byte_d of row) * scale[d / 128]      (V_j = K_j)
 *   out[t,h]  = sum_j softmax(s)_j V_j                     (bf16)
 *   lse[t,h]  = ln sum_j exp(s_j)                          (fp32, natural log)
 * An empty J gives out = 0 and lse = -inf; a row of J holding a NaN code gives
 * NaN out and lse for that token, whether or not its list is split. The result
 * does not depend on the order of the entries nor on what slot 0 holds
 * (bit-identical output).
 *
 * Arguments:
 *   q_bf16     bf16 [T, H, d_qk] row-major, device, 16-byte aligned
 *   T, H       tokens (>= 0; 0 launches nothing) and heads (1..128)
 *   d_qk       576 (512 latent + 64 RoPE) or 512 (NoPE: the row tail is not read)
 *   kv         the cache (16-byte aligned; row_bytes 656, or 528 with d_qk 512)
 *   topk_idx   int32 [T, W] row-major, device; W >= 0
 *   sm_scale   softmax scale applied to q . k (finite)
 *   out_bf16   bf16 [T, H, 512] row-major, device, 16-byte aligned
 *   lse        fp32 [T, H], device
 *   workspace  device scratch of at least mla_sparse_decode_workspace_bytes(T,H,W)
 *              bytes, 16-byte aligned (may be NULL when that is 0). Its contents
 *              on entry do not matter; it is clobbered.
 * The decode kernel is launched with programmatic stream serialization and waits
 * for the previous kernel on the stream, and its memory, before it reads any
 * input; behind mla_kv_write its launch overlaps the writer's last CTAs.
 * Returns MLA_OK, MLA_EINVAL, MLA_EUNSUPPORTED, MLA_ENOWORKSPACE or MLA_ECUDA.
 */
int mla_sparse_decode(const void* q_bf16, int T, int H, int d_qk, mla_kv_cache_t kv,
                      const int32_t* topk_idx, int W, float sm_scale, void* out_bf16,
                      float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_sparse_decode_paged - mla_sparse_decode with the top-k list given as
 * sequence positions and a block table (vLLM PR #55277, Purpose item 2: the
 * sparse attention reads its top-k entries through block tables, a page table
 * whose width is a capacity; here the kernel maps each position to a slot).
 *
 * Entry j of token t is position p = topk_pos[t,j] of the token's sequence
 * s = token_seq[t] (every token uses row 0 when token_seq is NULL). It stands for
 * the slot  block_table[s, p / page_size] * page_size + p % page_size,  and
 * the decode is then exactly mla_sparse_decode over those slots. A negative
 * position or a negative (unassigned) block-table entry is absent; a page past
 * max_pages, a sequence outside [0, n_seq) or a slot >= num_slots is absent and
 * sets MLA_ERR_DECODE_INDEX_RANGE. Slot 0 stays absent.
 *
 * Arguments as mla_sparse_decode, plus:
 *   topk_pos     int32 [T, W] positions, device
 *   block_table  int32 [n_seq, max_pages] physical page of each logical page,
 *                device, 4-byte aligned
 *   token_seq    int32 [T] block-table row of each token, device, or NULL
 *   page_size    slots per page (> 0)
 * The workspace is mla_sparse_decode_workspace_bytes(T, H, W).
 */
int mla_sparse_decode_paged(const void* q_bf16, int T, int H, int d_qk, mla_kv_cache_t kv,
                            const int32_t* topk_pos, int W, const int32_t* block_table, int n_seq,
                            int max_pages, const int32_t* token_seq, int page_size, float sm_scale,
                            void* out_bf16, float* lse, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * mla_sparse_prefill - what mla_sparse_decode computes, for batches whose
 * adjacent tokens share most of their top-k rows (a causal prefill: token i's
 * list is nearly a subset of token i+1's).
 *
 * The pages route prefill-sized batches to a dedicated kernel (sglang PR
 * #39288, Motivation: above 64 query rows the prefill kernel runs) and note
 * that the decode kernel also serves prefill today (sglang PR #47013, Speed
 * Tests). Here one CTA takes tokens 2u and 2u+1 with one group of 16 heads; the
 * rows present in both lists are copied and converted once for both tokens.
 * A row present in one list only is computed for that token only, so the result
 * of every token is exactly the decode statement of mla_sparse_decode over its
 * own list (same masking rules, bit-identical whatever slot 0 holds); only the
 * order of accumulation differs from mla_sparse_decode, so the two agree to
 * rounding, not bit for bit. A slot listed twice counts twice, as in the decode.
 *
 * Arguments as mla_sparse_decode, without the workspace; W is at most 2304
 * (MLA_EUNSUPPORTED otherwise). Batches whose adjacent tokens share few rows
 * compute correctly but gain nothing; batches of fewer than about two tokens
 * per SM leave SMs idle (no list is split): use mla_sparse_decode for those.
 * Launched with programmatic stream serialization like the decode.
 * Returns MLA_OK, MLA_EINVAL, MLA_EUNSUPPORTED or MLA_ECUDA.
 */
int mla_sparse_prefill(const void* q_bf16, int T, int H, int d_qk, mla_kv_cache_t kv,
                       const int32_t* topk_idx, int W, float sm_scale, void* out_bf16, float* lse,
                       void* stream);

/*
 * mla_sparse_prefill_paged - mla_sparse_prefill with the top-k list given as
 * sequence positions and a block table, mapped exactly as in
 * mla_sparse_decode_paged (vLLM PR #55277, Purpose item 2). Arguments as
 * mla_sparse_decode_paged, without the workspace.
 */
int mla_sparse_prefill_paged(const void* q_bf16, int T, int H, int d_qk, mla_kv_cache_t kv,
                             const int32_t* topk_pos, int W, const int32_t* block_table, int n_seq,
                             int max_pages, const int32_t* token_seq, int page_size, float sm_scale,
                             void* out_bf16, float* lse, void* stream);

/*
 * mla_gather_upconvert - gather rows of the cache and widen them to BF16
 * (vLLM PR #55277, Changes table: cp_gather_and_upconvert_fp8_kv_cache, the
 * chunked-context path; the NoPE tail is written as exact zeros).
 *
 * For i < n with s = slots[i]:
 *   out[i, d]       = the BF16 value nearest to e4m3(byte_d) * scale[d / 128]
 *                     (the exact product, rounded once, ties to even; a NaN
 *                     code gives 0x7FC0),                         d < 512
 *   out[i, 512 + k] = the RoPE value k of the row's tail (pe_dim 64), or 0
 *                     (pe_dim 0: the tail is not read),           k < 64
 * An absent slot (s <= 0) gives a row of zeros; s >= num_slots as well, and
 * sets MLA_ERR_GATHER_INDEX_RANGE.
 *
 * Arguments:
 *   kv        the cache (16-byte aligned; row_bytes 656, or 528 with pe_dim 0)
 *   slots     int32 [n], device, 4-byte aligned
 *   n         >= 0 (0 launches nothing)
 *   pe_dim    64 or 0
 *   out_bf16  bf16 [n, 576] row-major, device, 16-byte aligned
 * Returns MLA_OK, MLA_EINVAL or MLA_ECUDA.
 */
int mla_gather_upconvert(mla_kv_cache_t kv, const int32_t* slots, int64_t n, int pe_dim,
                         void* out_bf16, void* stream);

/*
 * mla_sparse_decode_noalloc - mla_sparse_decode for callers that cannot
 * allocate device memory where they call it.
 *
 * The pages have no counterpart to this entry point; it exists for users of
 * this library. mla_sparse_decode needs a caller-owned workspace whenever it
 * splits a token's top-k list across CTAs (mla_sparse_decode_workspace_bytes()
 * > 0). A caller that runs inside another framework's memory pool without an
 * allocator handle, or a process that has already committed all the device
 * memory it may use, has no way to provide one. This variant computes exactly
 * what mla_sparse_decode computes, with the same arguments minus the
 * workspace, and uses instead a fixed array of MLA_NOALLOC_SCRATCH_BYTES in the
 * library's own device memory. That array exists on every GPU that loads the
 * library's device code and stays allocated until the process exits. The call
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 *
 *   - Sizes whose workspace would exceed MLA_NOALLOC_SCRATCH_BYTES are rejected
 *     with MLA_ENOWORKSPACE before anything is launched.
 *   - All calls on a device share the one array and it keeps what the last call
 *     left there: calls whose work overlaps on the GPU (other streams, or
 *     concurrently replayed graphs) race and produce wrong results. Issue them
 *     on one stream. Nothing in the array needs to start at zero.
 *   - The first call on a device looks up the array's address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 * Returns what mla_sparse_decode returns.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (64u << 20)   /* 64 MiB per device */
int mla_sparse_decode_noalloc(const void* q_bf16, int T, int H, int d_qk, mla_kv_cache_t kv,
                              const int32_t* topk_idx, int W, float sm_scale, void* out_bf16,
                              float* lse, void* stream);

/*
 * mla_get_error - read and clear the device error word of the current device
 * (MLA_ERR_* bits accumulated by every launch since the last read). Blocks
 * until the device is idle. Returns MLA_OK or MLA_ECUDA; *host_code receives
 * the bits (host pointer, not NULL).
 */
int mla_get_error(int32_t* host_code);

/* Human-readable name of a return code (static string). */
const char* mla_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* MLASPARSE_H */
