// Scalar CPU oracle for the FP8 MLA KV cache: the packed-row writer and the
// sparse top-k MLA decode that reads it.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the library's product path links,
// loads or calls this file; only the tests, the smoke check and the bench's
// CPU-baseline / reference leg do. It shares no code, header, table or
// constant with the CUDA library: every constant below is restated from the
// pages it cites.
//
// Sources (cited by page title and section):
//   [vLLM-55277] vLLM PR #55277 "Support NoPE sparse MLA (GLM-5.3-Flash) on the
//                FlashInfer SM120 backend", Purpose item 1 and the Changes table:
//                the 656-byte fp8_ds_mla row = 512 B of FP8 latent, 16 B of tile
//                scales, 128 B of RoPE values or padding; NoPE rows zero the
//                128-byte tail; pe_dim must be 64 or 0.
//   [sglang-47013] sglang PR #47013 "zero-RoPE writer skips reserved slot 0",
//                Summary and Motivation: writes aimed at the reserved slot 0 are
//                dropped; per-token FP8 quantisation keeps BF16 NaNs.
//   [sglang-39288] sglang PR #39288 "SM120 sparse MLA: zero-initialise the
//                page-split scratch", Root cause: a masked (-1) top-k candidate
//                must contribute nothing, whatever slot 0 holds.
//   [sglang-39288] "Relation to other changes": the canonical NoPE row of
//                flashinfer#5075 is 528 bytes (the 512-byte latent and the 16
//                bytes of scales, no tail).
//   [vLLM-55277] Changes table, cp_gather_and_upconvert_fp8_kv_cache: gathers
//                rows of the cache and widens them to BF16 for the chunked-
//                context path, the NoPE tail written as exact zeros.
//   OCP 8-bit Floating Point Specification (OFP8), E4M3 format: bias 7,
//                3 mantissa bits, no infinities, S.1111.111 is NaN, max finite
//                448, subnormals m * 2^-9.
//
// Readings where the pages leave a step open (each also listed in the design
// notes):
//   * tile scale = amax / 448 in IEEE fp32 (round to nearest), 1.0 if amax == 0;
//   * value = e4m3_rne_satfinite(x / scale), the division in IEEE fp32;
//   * amax ignores every NaN (quiet or signaling); a NaN element encodes as 0x7F;
//   * +-inf saturates to +-448 (0x7E / 0xFE), like any out-of-range value;
//   * latent value i is stored at byte i; tile t holds bytes 128t .. 128t+127;
//   * scales are four little-endian fp32 at bytes 512 + 4t;
//   * a decode entry is present iff 0 < idx < num_slots; -1 (any negative), the
//     reserved slot 0 and out-of-range slots are absent and never read;
//   * lse is the natural log of the sum of exp of the *scaled* scores;
//     an empty entry set gives out = 0 and lse = -inf;
//   * a 528-byte row is the 656-byte row without its tail (NoPE only);
//   * the upconverted latent value is the BF16 nearest to the exact product
//     e4m3(byte) * scale (ties to even), NaN codes give 0x7FC0; an absent slot
//     gives a row of zeros.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>
#include <atomic>

namespace {

// Row layout, restated from [vLLM-55277] Purpose item 1 (656 bytes) and
// [sglang-39288] "Relation to other changes" (528 bytes, no tail).
constexpr int64_t kRowBytes = 656;
constexpr int64_t kRowBytesNope = 528;
constexpr int kLatent = 512;
constexpr int kTileValues = 128;
constexpr int kTiles = 4;
constexpr int kScaleOffset = 512;
constexpr int kTailOffset = 528;
constexpr int kRope = 64;

// bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 bits.
float bf16_to_float(uint16_t bits) {
    uint32_t u = static_cast<uint32_t>(bits) << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return f;
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// E4M3 codec, written from the OCP OFP8 specification.
// ---------------------------------------------------------------------------

// Decode one E4M3 byte to its exact value (NaN for S.1111.111).
double oracle_e4m3_decode(uint8_t b) {
    const int sign = (b >> 7) & 1;
    const int e = (b >> 3) & 0xF;
    const int m = b & 0x7;
    double v;
    if (e == 0xF && m == 0x7) {
        return std::numeric_limits<double>::quiet_NaN();
    } else if (e == 0) {
        v = std::ldexp(static_cast<double>(m), -9);          // subnormal: m * 2^-9
    } else {
        v = std::ldexp(1.0 + m / 8.0, e - 7);                 // normal: 2^(e-7) * 1.m
    }
    return sign ? -v : v;
}

// Encode an fp32 value as E4M3: round to nearest, ties to even, saturating
// finite overflow (and +-inf) to +-448; NaN -> 0x7F; the sign of zero is kept.
uint8_t oracle_e4m3_encode(float x) {
    if (std::isnan(x)) return 0x7F;
    const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
    const double a = std::fabs(static_cast<double>(x));      // exact widening
    if (a == 0.0) return sign;
    // Spacing of the E4M3 grid around a: 2^-9 below the smallest normal 2^-6,
    // else 2^(floor(log2 a) - 3) (three mantissa bits).
    int ex;
    std::frexp(a, &ex);            // a = f * 2^ex, f in [0.5, 1)  => floor(log2 a) = ex - 1
    const int e_floor = ex - 1;
    const int q_exp = (e_floor < -6) ? -9 : (e_floor - 3);
    const double n = std::ldexp(a, -q_exp);                  // exact: power-of-two scaling
    double r = std::nearbyint(n);                            // default rounding mode: ties to even
    double v = std::ldexp(r, q_exp);
    if (v > 448.0) v = 448.0;                                // satfinite (also catches +inf)
    if (v == 0.0) return sign;
    if (v < std::ldexp(1.0, -6)) {
        const int m = static_cast<int>(std::ldexp(v, 9));    // 1..7
        return static_cast<uint8_t>(sign | m);
    }
    int vex;
    const double f = std::frexp(v, &vex);                    // v = f * 2^vex, f in [0.5,1)
    const int e = vex - 1;                                   // -6..8
    const int m = static_cast<int>(f * 16.0) - 8;            // (2f - 1) * 8
    return static_cast<uint8_t>(sign | ((e + 7) << 3) | m);
}

// Bulk helpers for the tests.
void oracle_e4m3_encode_array(const float* x, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}

// Encode every fp32 bit pattern in [lo, hi) (as uint32) into out[0 .. hi-lo).
void oracle_e4m3_encode_bit_range(uint64_t lo, uint64_t hi, uint8_t* out, int n_threads) {
    if (n_threads < 1) n_threads = 1;
    std::vector<std::thread> pool;
    const uint64_t count = hi - lo;
    for (int t = 0; t < n_threads; ++t) {
        pool.emplace_back([=]() {
            const uint64_t a = lo + count * t / n_threads;
            const uint64_t b = lo + count * (t + 1) / n_threads;
            for (uint64_t u = a; u < b; ++u) {
                uint32_t bits = static_cast<uint32_t>(u);
                float f;
                std::memcpy(&f, &bits, sizeof f);
                out[u - lo] = oracle_e4m3_encode(f);
            }
        });
    }
    for (auto& th : pool) th.join();
}

// ---------------------------------------------------------------------------
// Writer: per-token FP8 quantise-and-scatter into the 656-byte row.
// [vLLM-55277] Purpose item 1 (layout, NoPE zero tail, pe_dim in {64, 0});
// [sglang-47013] Summary / Motivation (drop rows aimed at the reserved slot).
// Returns the number of rows whose slot was >= num_slots (dropped as well).
// ---------------------------------------------------------------------------
// row_bytes is 656 or 528; a 528-byte row has no tail, so rope must be null
// (returns -1 otherwise).
int64_t oracle_kv_write_rows(uint8_t* cache, int64_t num_slots, int64_t row_bytes, const int64_t* slot_idx,
                             const uint16_t* latent_bf16, const uint16_t* rope_bf16,
                             int64_t n_rows, int64_t reserved_slot) {
    if (row_bytes != kRowBytes && !(row_bytes == kRowBytesNope && rope_bf16 == nullptr)) return -1;
    int64_t out_of_range = 0;
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t slot = slot_idx[r];
        // Step 1: rows aimed at the reserved slot (or a negative slot) are
        // dropped before any of their inputs is read.
        if (slot == reserved_slot || slot < 0) continue;
        if (slot >= num_slots) { ++out_of_range; continue; }
        uint8_t* row = cache + slot * row_bytes;
        const uint16_t* x = latent_bf16 + r * kLatent;
        for (int t = 0; t < kTiles; ++t) {
            // Step 2: tile amax, ignoring every NaN (quiet or signaling: a bf16 NaN
            // whose top mantissa bit is clear widens to a signaling fp32 NaN).
            float amax = 0.0f;
            for (int i = 0; i < kTileValues; ++i) {
                const float a = std::fabs(bf16_to_float(x[t * kTileValues + i]));
                if (!std::isnan(a) && a > amax) amax = a;
            }
            // Step 3: fp32 scale.
            const float scale = (amax > 0.0f) ? (amax / 448.0f) : 1.0f;
            // Step 4: quantise value i of tile t to byte 128t + i.
            for (int i = 0; i < kTileValues; ++i) {
                const float v = bf16_to_float(x[t * kTileValues + i]) / scale;
                row[t * kTileValues + i] = oracle_e4m3_encode(v);
            }
            // Step 5: the scale as little-endian fp32 at byte 512 + 4t.
            uint32_t sbits;
            std::memcpy(&sbits, &scale, sizeof sbits);
            for (int k = 0; k < 4; ++k)
                row[kScaleOffset + 4 * t + k] = static_cast<uint8_t>((sbits >> (8 * k)) & 0xFF);
        }
        // Step 6: the tail: 64 bf16 RoPE values bit for bit, or 128 zero bytes
        // (a 528-byte row has none).
        if (row_bytes == kRowBytesNope) continue;
        for (int k = 0; k < kRope; ++k) {
            const uint16_t v = rope_bf16 ? rope_bf16[r * kRope + k] : 0;
            row[kTailOffset + 2 * k] = static_cast<uint8_t>(v & 0xFF);
            row[kTailOffset + 2 * k + 1] = static_cast<uint8_t>(v >> 8);
        }
    }
    return out_of_range;
}

int64_t oracle_kv_write(uint8_t* cache, int64_t num_slots, const int64_t* slot_idx,
                        const uint16_t* latent_bf16, const uint16_t* rope_bf16,
                        int64_t n_rows, int64_t reserved_slot) {
    return oracle_kv_write_rows(cache, num_slots, kRowBytes, slot_idx, latent_bf16, rope_bf16, n_rows,
                                reserved_slot);
}

// ---------------------------------------------------------------------------
// Sparse top-k MLA decode, in float64.
// For each query token t and head h, over the present entries j of topk[t, :]:
//   s_j   = sm_scale * ( sum_{d<512} q[t,h,d] * K_j[d]  +  [d_qk == 576] sum_{d<64} q[t,h,512+d] * rope_j[d] )
//   K_j[d] = e4m3(byte_d) * scale_{d / 128}        (V_j = K_j, the latent)
//   m = max_j s_j,  l = sum_j exp(s_j - m)
//   out[t,h,:] = sum_j exp(s_j - m) V_j / l,   lse[t,h] = m + ln l
// Present = 0 < idx < num_slots; everything else contributes nothing and is
// never read ([sglang-39288] Root cause; [sglang-47013] Motivation).
// tokens: optional list of token ids to compute (n_tokens of them); when null
// all T tokens are computed. Outputs are written at the token's own row.
// Returns the number of out-of-range (>= num_slots) entries seen.
// ---------------------------------------------------------------------------
int64_t oracle_sparse_decode_rows(const uint16_t* q_bf16, int T, int H, int d_qk,
                                  const uint8_t* cache, int64_t num_slots, int64_t row_bytes,
                                  const int32_t* topk, int W, float sm_scale_f,
                                  double* out, double* lse,
                                  const int32_t* tokens, int n_tokens, int n_threads) {
    if (row_bytes != kRowBytes && !(row_bytes == kRowBytesNope && d_qk == kLatent)) return -1;
    const double sm_scale = static_cast<double>(sm_scale_f);
    const bool with_rope = (d_qk == kLatent + kRope);
    const int n_work = tokens ? n_tokens : T;
    std::atomic<int> next{0};
    std::atomic<int64_t> bad{0};
    auto worker = [&]() {
        std::vector<double> kv(static_cast<size_t>(W) * kLatent);
        std::vector<double> rope(static_cast<size_t>(W) * kRope);
        std::vector<double> s(W);
        for (;;) {
            const int w = next.fetch_add(1);
            if (w >= n_work) break;
            const int t = tokens ? tokens[w] : w;
            // Gather and dequantise the present rows once per token.
            int n = 0;
            int64_t local_bad = 0;
            for (int j = 0; j < W; ++j) {
                const int64_t idx = topk[static_cast<int64_t>(t) * W + j];
                if (idx <= 0) continue;
                if (idx >= num_slots) { ++local_bad; continue; }
                const uint8_t* row = cache + idx * row_bytes;
                for (int tt = 0; tt < kTiles; ++tt) {
                    uint32_t sbits = 0;
                    for (int k = 0; k < 4; ++k)
                        sbits |= static_cast<uint32_t>(row[kScaleOffset + 4 * tt + k]) << (8 * k);
                    float sc;
                    std::memcpy(&sc, &sbits, sizeof sc);
                    for (int i = 0; i < kTileValues; ++i)
                        kv[static_cast<size_t>(n) * kLatent + tt * kTileValues + i] =
                            oracle_e4m3_decode(row[tt * kTileValues + i]) * static_cast<double>(sc);
                }
                if (with_rope) {
                    for (int k = 0; k < kRope; ++k) {
                        const uint16_t bits = static_cast<uint16_t>(row[kTailOffset + 2 * k]) |
                                              static_cast<uint16_t>(row[kTailOffset + 2 * k + 1] << 8);
                        rope[static_cast<size_t>(n) * kRope + k] = bf16_to_float(bits);
                    }
                }
                ++n;
            }
            bad += local_bad;
            for (int h = 0; h < H; ++h) {
                const uint16_t* qh = q_bf16 + (static_cast<int64_t>(t) * H + h) * d_qk;
                double* oh = out + (static_cast<int64_t>(t) * H + h) * kLatent;
                if (n == 0) {
                    for (int d = 0; d < kLatent; ++d) oh[d] = 0.0;
                    lse[static_cast<int64_t>(t) * H + h] = -std::numeric_limits<double>::infinity();
                    continue;
                }
                double m = -std::numeric_limits<double>::infinity();
                for (int j = 0; j < n; ++j) {
                    double acc = 0.0;
                    for (int d = 0; d < kLatent; ++d)
                        acc += static_cast<double>(bf16_to_float(qh[d])) * kv[static_cast<size_t>(j) * kLatent + d];
                    if (with_rope)
                        for (int k = 0; k < kRope; ++k)
                            acc += static_cast<double>(bf16_to_float(qh[kLatent + k])) * rope[static_cast<size_t>(j) * kRope + k];
                    s[j] = sm_scale * acc;
                    if (s[j] > m) m = s[j];
                }
                double l = 0.0;
                for (int d = 0; d < kLatent; ++d) oh[d] = 0.0;
                for (int j = 0; j < n; ++j) {
                    const double p = std::exp(s[j] - m);
                    l += p;
                    for (int d = 0; d < kLatent; ++d) oh[d] += p * kv[static_cast<size_t>(j) * kLatent + d];
                }
                for (int d = 0; d < kLatent; ++d) oh[d] /= l;
                lse[static_cast<int64_t>(t) * H + h] = m + std::log(l);
            }
        }
    };
    if (n_threads < 1) n_threads = 1;
    std::vector<std::thread> pool;
    for (int i = 1; i < n_threads; ++i) pool.emplace_back(worker);
    worker();
    for (auto& th : pool) th.join();
    return bad.load();
}

int64_t oracle_sparse_decode(const uint16_t* q_bf16, int T, int H, int d_qk,
                             const uint8_t* cache, int64_t num_slots,
                             const int32_t* topk, int W, float sm_scale_f,
                             double* out, double* lse,
                             const int32_t* tokens, int n_tokens, int n_threads) {
    return oracle_sparse_decode_rows(q_bf16, T, H, d_qk, cache, num_slots, kRowBytes, topk, W, sm_scale_f,
                                     out, lse, tokens, n_tokens, n_threads);
}

// ---------------------------------------------------------------------------
// Gather and upconvert ([vLLM-55277] Changes table, cp_gather_and_upconvert_
// fp8_kv_cache): out[i, 0:512] = BF16 nearest to e4m3(byte_d) * scale_{d/128}
// for the row at slots[i]; out[i, 512:576] = the 64 BF16 RoPE values of the
// tail when pe_dim == 64, zeros when pe_dim == 0 (the tail is not read). An
// absent slot (<= 0, or >= num_slots, counted) gives a row of zeros.
// Returns the number of slots >= num_slots.
// ---------------------------------------------------------------------------

// BF16 bits of the value nearest to x, ties to even (x is the exact product, a
// double); NaN -> 0x7FC0. BF16 has 8 significant bits and fp32's exponent range:
// normal quantum 2^(e-7) for 2^e <= |x| < 2^(e+1), e >= -126; below 2^-126 the
// quantum is 2^-133.
uint16_t oracle_double_to_bf16(double x) {
    if (std::isnan(x)) return 0x7FC0;
    const double a = std::fabs(x);
    double r;
    if (a == 0.0) {
        r = 0.0;
    } else {
        int ex;
        std::frexp(a, &ex);                          // a = f * 2^ex, f in [0.5, 1)
        const int e = ex - 1;                        // floor(log2 a)
        const int q_exp = (e < -126) ? -133 : (e - 7);
        r = std::ldexp(std::nearbyint(std::ldexp(a, -q_exp)), q_exp);   // ties to even
    }
    if (r > 3.3895313892515355e38) r = std::numeric_limits<double>::infinity();   // past the largest BF16
    float f = static_cast<float>(std::signbit(x) ? -r : r);     // exact: r is a BF16 value
    uint32_t u;
    std::memcpy(&u, &f, sizeof u);
    return static_cast<uint16_t>(u >> 16);
}

int64_t oracle_gather_upconvert(const uint8_t* cache, int64_t num_slots, int64_t row_bytes,
                                const int32_t* slots, int64_t n, int pe_dim, uint16_t* out) {
    if (row_bytes != kRowBytes && !(row_bytes == kRowBytesNope && pe_dim == 0)) return -1;
    if (pe_dim != 0 && pe_dim != kRope) return -1;
    int64_t bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        uint16_t* o = out + i * (kLatent + kRope);
        const int64_t idx = slots[i];
        if (idx <= 0 || idx >= num_slots) {
            if (idx >= num_slots) ++bad;
            for (int d = 0; d < kLatent + kRope; ++d) o[d] = 0;
            continue;
        }
        const uint8_t* row = cache + idx * row_bytes;
        for (int t = 0; t < kTiles; ++t) {
            uint32_t sbits = 0;
            for (int k = 0; k < 4; ++k) sbits |= static_cast<uint32_t>(row[kScaleOffset + 4 * t + k]) << (8 * k);
            float sc;
            std::memcpy(&sc, &sbits, sizeof sc);
            for (int v = 0; v < kTileValues; ++v) {
                // 4 significant bits times 24: the product is exact in a double.
                const double prod = oracle_e4m3_decode(row[t * kTileValues + v]) * static_cast<double>(sc);
                o[t * kTileValues + v] = oracle_double_to_bf16(prod);
            }
        }
        for (int k = 0; k < kRope; ++k)
            o[kLatent + k] = (pe_dim == kRope)
                ? static_cast<uint16_t>(row[kTailOffset + 2 * k] | (row[kTailOffset + 2 * k + 1] << 8))
                : static_cast<uint16_t>(0);
    }
    return bad;
}

}  // extern "C"
