// Oracle for paged Multi-head Latent Attention (MLA) decode.
//
// TEST INFRASTRUCTURE ONLY. Plain, slow, single-threaded C++17 in double
// precision. Only the tests, the smoke check and the CPU-baseline leg of the
// bench may load or call it; the product path never does. It shares no code,
// header, table or helper with the CUDA library.
//
// What it computes, and where the pages state it:
//  * The latent cache row of a DeepSeek-V2/V3 MLA layer: kv_lora_rank 512
//    (c_kv) plus qk_rope_head_dim 64 per token, no per-head K or V
//    (SGLang PR #32972 "Let Kimi-Linear use the paged MLA attention
//    backends", Validation). The absorbed query (q_nope * W_UK || q_rope) is
//    576-d and every head shares the latent key (576-d) and value (first 512).
//  * Paged pool with a per-layer leading dimension; without it the layers
//    alias the same slots (MoE-Infinity PR #195 "DeepSeek-V2/V3
//    paged-attention shim (MLA)", Root causes 5 and Changes).
//  * The new token's row is written through slot_mapping on every decode step
//    (same page, Root causes 2); pad rows carry a negative slot and write
//    nothing (SGLang PR #32972, Cuda-graph safety: stale pad locations
//    scatter garbage).
//  * context_length excludes the just-generated token (MoE-Infinity PR #195,
//    Root causes 4), so the new token sits at position L and is attended.
//  * Only the prefix of the page list that the request needs is read
//    (SGLang PR #32972, Correction).
//  * The MLA geometry qk_head_dim 192 = 128 nope + 64 rope and v_head_dim 128
//    (MoE-Infinity PR #195, Root causes 3) defines the unabsorbed form used as
//    an independent check, and the softmax scale 192^-1/2.
//  * Sliding window over the most recent tokens (FastDeploy PR #8049
//    "Support MLA_SWA functionality", Motivation): window W covers positions
//    [max(0, L+1-W), L]; W = 0 means full attention.
//  * fp8_e4m3 latent cache (SGLang PR #32972, Validation table,
//    tokenspeed_mla row): one fp32 scale per pool; stored = e4m3(x / scale),
//    read = e4m3 * scale. The codec is written here from the OCP 8-bit
//    floating point definition of E4M3: 1 sign, 4 exponent (bias 7),
//    3 mantissa bits, subnormals, no infinities, S.1111.111 = NaN, max 448.
//
// Build without -ffast-math and with -ffp-contract=off: the fp8 quantiser's
// fp32 division must be the correctly rounded IEEE one.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

constexpr int kDimCkv = 512;   // kv_lora_rank
constexpr int kDimRope = 64;   // qk_rope_head_dim
constexpr int kDimRow = kDimCkv + kDimRope;  // 576
constexpr int kDimNope = 128;  // qk_nope_head_dim of the unabsorbed form
constexpr int kDimV = 128;     // v_head_dim of the unabsorbed form

constexpr int kBf16 = 0;
constexpr int kFp8E4M3 = 1;

// Error codes shared in meaning (not in code) with the library's C ABI.
constexpr int kOk = 0;
constexpr int kErrArg = -1;

// bfloat16 is the upper half of an IEEE binary32: widening is exact.
double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// Round a non-negative double to the nearest integer, ties to even.
double round_half_even(double v) {
  double fl = std::floor(v);
  double diff = v - fl;
  if (diff > 0.5) return fl + 1.0;
  if (diff < 0.5) return fl;
  return (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

}  // namespace

extern "C" {

// E4M3 code -> value (OCP FP8 E4M3 definition).
double oracle_e4m3_decode(uint8_t code) {
  const int sign = (code >> 7) & 1;
  const int e = (code >> 3) & 0xF;
  const int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) {
    mag = NAN;
  } else if (e == 0) {
    mag = std::ldexp(static_cast<double>(m), -9);  // m/8 * 2^(1-7)
  } else {
    mag = std::ldexp(1.0 + m / 8.0, e - 7);
  }
  return sign ? -mag : mag;
}

// fp32 value -> E4M3 code, round to nearest even, saturating to +-448.
uint8_t oracle_e4m3_encode(float x) {
  if (std::isnan(x)) return 0x7F;
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs(static_cast<double>(x));
  if (a >= 448.0) return sign | 0x7E;
  if (a < std::ldexp(1.0, -6)) {
    // Subnormal range: multiples of 2^-9. A result of 8 is the smallest
    // normal (exponent field 1, mantissa 0), which is code 8.
    const double q = round_half_even(a * 512.0);
    return sign | static_cast<uint8_t>(q);
  }
  int e = static_cast<int>(std::floor(std::log2(a)));
  // Guard log2 rounding at exact powers of two.
  if (std::ldexp(1.0, e) > a) e -= 1;
  if (std::ldexp(1.0, e + 1) <= a) e += 1;
  double q = round_half_even((a / std::ldexp(1.0, e) - 1.0) * 8.0);
  if (q == 8.0) {
    q = 0.0;
    e += 1;
  }
  // a < 448 keeps the result at or below 1.75 * 2^8 (code 0x7E).
  return sign | static_cast<uint8_t>(((e + 7) << 3) | static_cast<int>(q));
}

// Value of element d of latent row (layer, page, offset) as the kernel reads it.
static double pool_value(const uint8_t* pool, int dtype, int num_pages,
                         int page_size, float kv_scale, int layer, int page,
                         int offset, int d) {
  const int64_t row =
      (static_cast<int64_t>(layer) * num_pages + page) * page_size + offset;
  if (dtype == kBf16) {
    uint16_t bits;
    std::memcpy(&bits, pool + (row * kDimRow + d) * 2, 2);
    return bf16_bits_to_double(bits);
  }
  return oracle_e4m3_decode(pool[row * kDimRow + d]) *
         static_cast<double>(kv_scale);
}

// Latent write through slot_mapping: pool[layer][slot / ps][slot % ps] = row.
// Negative slots are pad rows and write nothing. Slots at or beyond
// num_pages * page_size are rejected.
int oracle_kv_write(uint8_t* pool, int dtype, int num_layers, int num_pages,
                    int page_size, float kv_scale, int layer,
                    const uint16_t* new_rows, const int64_t* slot_mapping,
                    int n) {
  if (layer < 0 || layer >= num_layers || page_size <= 0 || n < 0)
    return kErrArg;
  if (dtype != kBf16 && dtype != kFp8E4M3) return kErrArg;
  const int64_t slots = static_cast<int64_t>(num_pages) * page_size;
  for (int i = 0; i < n; ++i) {
    const int64_t s = slot_mapping[i];
    if (s < 0) continue;
    if (s >= slots) return kErrArg;
    const int64_t row = static_cast<int64_t>(layer) * slots + s;
    for (int d = 0; d < kDimRow; ++d) {
      const uint16_t bits = new_rows[static_cast<int64_t>(i) * kDimRow + d];
      if (dtype == kBf16) {
        std::memcpy(pool + (row * kDimRow + d) * 2, &bits, 2);
      } else {
        const float x = static_cast<float>(bf16_bits_to_double(bits));
        const float t = x / kv_scale;  // IEEE fp32 division
        pool[row * kDimRow + d] = oracle_e4m3_encode(t);
      }
    }
  }
  return kOk;
}

// Physical page holding logical block j of request b. page_indptr != NULL:
// CSR (kv_indices) form; else block_table [batch, max_blocks].
static int page_of(const int32_t* page_indptr, const int32_t* page_ids,
                   int max_blocks, int b, int j) {
  if (page_indptr) return page_ids[page_indptr[b] + j];
  return page_ids[static_cast<int64_t>(b) * max_blocks + j];
}

// Absorbed decode. For each request b in `requests` (all when NULL) and each
// head h:  s_t = scale * q[b,h,:] . K[t,:] over t in [start, L_b], with
// start = 0 (window 0) or max(0, L_b + 1 - window); out = softmax(s) @ K[:, :512];
// lse = log(sum exp(s)) (natural log). Output row r holds requests[r].
int oracle_decode(const uint8_t* pool, int dtype, int num_layers,
                  int num_pages, int page_size, float kv_scale, int layer,
                  const double* q, const int32_t* page_indptr,
                  const int32_t* page_ids, int max_blocks,
                  const int32_t* context_lens, int batch, int num_heads,
                  double softmax_scale, int window, const int32_t* requests,
                  int num_requests, double* out, double* lse) {
  if (layer < 0 || layer >= num_layers || page_size <= 0 || num_heads <= 0 ||
      window < 0)
    return kErrArg;
  const int nr = requests ? num_requests : batch;
  for (int r = 0; r < nr; ++r) {
    const int b = requests ? requests[r] : r;
    if (b < 0 || b >= batch) return kErrArg;
    const int L = context_lens[b];
    if (L < 0) return kErrArg;
    const int start = window > 0 ? (L + 1 - window > 0 ? L + 1 - window : 0) : 0;
    const int n = L + 1 - start;
    // Blocks 0..L/ps hold positions 0..L; only those from start/ps on are read.
    const int n_blocks = L / page_size + 1;
    if (!page_indptr && n_blocks > max_blocks) return kErrArg;
    if (page_indptr && page_indptr[b + 1] - page_indptr[b] < n_blocks)
      return kErrArg;
    for (int j = start / page_size; j < n_blocks; ++j) {
      const int p = page_of(page_indptr, page_ids, max_blocks, b, j);
      if (p < 0 || p >= num_pages) return kErrArg;
    }
    // Decode the attended rows once per request.
    std::vector<double> K(static_cast<size_t>(n) * kDimRow);
    for (int i = 0; i < n; ++i) {
      const int t = start + i;
      const int p = page_of(page_indptr, page_ids, max_blocks, b, t / page_size);
      for (int d = 0; d < kDimRow; ++d)
        K[static_cast<size_t>(i) * kDimRow + d] = pool_value(
            pool, dtype, num_pages, page_size, kv_scale, layer, p,
            t % page_size, d);
    }
    std::vector<double> s(n);
    for (int h = 0; h < num_heads; ++h) {
      const double* qh = q + (static_cast<int64_t>(b) * num_heads + h) * kDimRow;
      double m = -INFINITY;
      for (int i = 0; i < n; ++i) {
        double acc = 0.0;
        for (int d = 0; d < kDimRow; ++d)
          acc += qh[d] * K[static_cast<size_t>(i) * kDimRow + d];
        s[i] = softmax_scale * acc;
        if (s[i] > m) m = s[i];
      }
      double denom = 0.0;
      for (int i = 0; i < n; ++i) {
        s[i] = std::exp(s[i] - m);
        denom += s[i];
      }
      double* o = out + (static_cast<int64_t>(r) * num_heads + h) * kDimCkv;
      std::vector<double> acc(kDimCkv, 0.0);
      for (int i = 0; i < n; ++i)
        for (int d = 0; d < kDimCkv; ++d)
          acc[d] += s[i] * K[static_cast<size_t>(i) * kDimRow + d];
      for (int d = 0; d < kDimCkv; ++d) o[d] = acc[d] / denom;
      if (lse) lse[static_cast<int64_t>(r) * num_heads + h] = m + std::log(denom);
    }
  }
  return kOk;
}

// Query absorption: q_abs[b,h,0:512] = W_UK[h]^T q_nope[b,h],
// q_abs[b,h,512:576] = q_rope[b,h]. W_UK is [H, 128, 512].
int oracle_absorb_query(const double* q_nope, const double* q_rope,
                        const double* w_uk, int batch, int num_heads,
                        double* q_abs) {
  for (int b = 0; b < batch; ++b)
    for (int h = 0; h < num_heads; ++h) {
      const int64_t bh = static_cast<int64_t>(b) * num_heads + h;
      double* qa = q_abs + bh * kDimRow;
      for (int d = 0; d < kDimCkv; ++d) {
        double acc = 0.0;
        for (int e = 0; e < kDimNope; ++e)
          acc += q_nope[bh * kDimNope + e] *
                 w_uk[(static_cast<int64_t>(h) * kDimNope + e) * kDimCkv + d];
        qa[d] = acc;
      }
      for (int d = 0; d < kDimRope; ++d) qa[kDimCkv + d] = q_rope[bh * kDimRope + d];
    }
  return kOk;
}

// W_UV projection of the latent attention output: y[b,h,:] = out[b,h,:] W_UV[h],
// W_UV is [H, 512, 128] (v_head_dim 128).
int oracle_uv_project(const double* attn, const double* w_uv, int batch,
                      int num_heads, double* y) {
  for (int b = 0; b < batch; ++b)
    for (int h = 0; h < num_heads; ++h) {
      const int64_t bh = static_cast<int64_t>(b) * num_heads + h;
      for (int e = 0; e < kDimV; ++e) {
        double acc = 0.0;
        for (int d = 0; d < kDimCkv; ++d)
          acc += attn[bh * kDimCkv + d] *
                 w_uv[(static_cast<int64_t>(h) * kDimCkv + d) * kDimV + e];
        y[bh * kDimV + e] = acc;
      }
    }
  return kOk;
}

// Unabsorbed multi-head form, an independent formulation of the same layer:
// per head, k_nope[t] = W_UK[h] c_kv[t] (128), k = [k_nope ; k_rope[t]] (192),
// v[t] = W_UV[h]^T c_kv[t] (128), score = scale * (q_nope.k_nope + q_rope.k_rope),
// y = softmax(score) @ v. Same pool addressing and window as oracle_decode.
int oracle_decode_unabsorbed(const uint8_t* pool, int dtype, int num_layers,
                             int num_pages, int page_size, float kv_scale,
                             int layer, const double* q_nope,
                             const double* q_rope, const double* w_uk,
                             const double* w_uv, const int32_t* page_indptr,
                             const int32_t* page_ids, int max_blocks,
                             const int32_t* context_lens, int batch,
                             int num_heads, double softmax_scale, int window,
                             double* y) {
  if (layer < 0 || layer >= num_layers || page_size <= 0 || window < 0)
    return kErrArg;
  for (int b = 0; b < batch; ++b) {
    const int L = context_lens[b];
    if (L < 0) return kErrArg;
    const int start = window > 0 ? (L + 1 - window > 0 ? L + 1 - window : 0) : 0;
    const int n = L + 1 - start;
    for (int h = 0; h < num_heads; ++h) {
      const int64_t bh = static_cast<int64_t>(b) * num_heads + h;
      std::vector<double> score(n);
      std::vector<double> v(static_cast<size_t>(n) * kDimV);
      double m = -INFINITY;
      for (int i = 0; i < n; ++i) {
        const int t = start + i;
        const int p = page_of(page_indptr, page_ids, max_blocks, b, t / page_size);
        if (p < 0 || p >= num_pages) return kErrArg;
        std::vector<double> c(kDimRow);
        for (int d = 0; d < kDimRow; ++d)
          c[d] = pool_value(pool, dtype, num_pages, page_size, kv_scale, layer,
                            p, t % page_size, d);
        double dot = 0.0;
        for (int e = 0; e < kDimNope; ++e) {
          double k_nope = 0.0;
          for (int d = 0; d < kDimCkv; ++d)
            k_nope += w_uk[(static_cast<int64_t>(h) * kDimNope + e) * kDimCkv + d] * c[d];
          dot += q_nope[bh * kDimNope + e] * k_nope;
        }
        for (int d = 0; d < kDimRope; ++d)
          dot += q_rope[bh * kDimRope + d] * c[kDimCkv + d];
        score[i] = softmax_scale * dot;
        if (score[i] > m) m = score[i];
        for (int e = 0; e < kDimV; ++e) {
          double acc = 0.0;
          for (int d = 0; d < kDimCkv; ++d)
            acc += w_uv[(static_cast<int64_t>(h) * kDimCkv + d) * kDimV + e] * c[d];
          v[static_cast<size_t>(i) * kDimV + e] = acc;
        }
      }
      double denom = 0.0;
      for (int i = 0; i < n; ++i) {
        score[i] = std::exp(score[i] - m);
        denom += score[i];
      }
      for (int e = 0; e < kDimV; ++e) {
        double acc = 0.0;
        for (int i = 0; i < n; ++i) acc += score[i] * v[static_cast<size_t>(i) * kDimV + e];
        y[bh * kDimV + e] = acc / denom;
      }
    }
  }
  return kOk;
}

}  // extern "C"
