// Plain CPU oracle for the fused per-token decoder path (RMSNorm, residual-add +
// RMSNorm, RoPE with paged KV-cache store, SwiGLU/ReGLU, UClip/DyHT) and the
// decode-attention read of the paged cache.
//
// TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the bench's
// CPU-baseline leg load this file's library. The CUDA library never links,
// includes or calls it, and it shares no source with the CUDA path.
//
// Every value is decoded to double, the operator's formula is applied in double
// in the order the pages state it, and the result is rounded once to the
// output format with round-to-nearest, ties-to-even. No blocking, no fusion,
// no reordering beyond what the formula says.
//
// Sources ("pages"):
//   [koas]  koas-w.github.io, "preformanceimprovement" (Qwen2.5-1.5B engine):
//           section 1 (fused RoPE + paged KV store), section 2 (fused SwiGLU),
//           section 3 (RMSNorm chain x.pow(2).mean(-1).add(eps).rsqrt().mul(x).mul(weight),
//           fp32 compute, cast back on write), section 4 (fused add + norm, x updated
//           in place, normed result returned).
//   [lsln]  m.lsln.cn/news/61269, section 2.3 (RMSNorm in fp32, y.to(dtype) once;
//           precomputed cos/sin caches).
//   [mer]   mer.dev "AsyncT vllm ..." section 0 (DyHT replacing RMSNorm), section 1.1
//           (KV cache layout [2, num_blocks, block_size, num_kv_heads, head_size]) and
//           section 3.3 (relu_and_mul for ReGLU; the uclip kernel; 3-D Q/K views).
//   [csdn]  agent.csdn.net "使用Triton实现RMSNorm算子" (rsqrt(sum/D + eps) per row).
//
// Parity pins: every function here is pinned by the CPU tests (closed forms,
// exhaustive format round trips, exact-rational brute force); none is "parity
// unpinned". The one unpinned quantity is the drift accumulated over a
// 28-layer chain, which the chain test reports rather than bounds.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <set>
#include <vector>

namespace {

// Element formats. The numbering mirrors the public enum by value only; the
// two are declared separately on purpose.
enum Fmt { F32 = 0, F16 = 1, BF16 = 2 };

struct FormatSpec {
    int p;     // significand bits, hidden bit included
    int emin;  // exponent of the smallest normal
    int emax;  // exponent of the largest finite
};

bool format_spec(int fmt, FormatSpec* s) {
    switch (fmt) {
        case F32:  *s = {24, -126, 127}; return true;
        case F16:  *s = {11, -14, 15};   return true;
        case BF16: *s = {8, -126, 127};  return true;
        default:   return false;
    }
}

// Round a double to the nearest value of a binary format with spec `s`,
// ties to even, overflow to infinity (IEEE 754 roundTiesToEven).
double round_to_format(double v, const FormatSpec& s) {
    if (std::isnan(v) || std::isinf(v) || v == 0.0) return v;
    double a = std::fabs(v);
    int e2;
    std::frexp(a, &e2);               // a = m * 2^e2 with m in [0.5, 1)
    int lead = e2 - 1;                // exponent of a's leading bit
    int q = (lead > s.emin ? lead : s.emin) - (s.p - 1);  // exponent of one ulp
    double scaled = std::ldexp(a, -q);   // exact: a power-of-two rescale
    double fl = std::floor(scaled);
    double frac = scaled - fl;           // exact
    if (frac > 0.5 || (frac == 0.5 && std::fmod(fl, 2.0) != 0.0)) fl += 1.0;
    double r = std::ldexp(fl, q);
    double maxfin = std::ldexp(std::ldexp(1.0, s.p) - 1.0, s.emax - (s.p - 1));
    if (r > maxfin) r = INFINITY;
    return std::copysign(r, v);
}

uint32_t encode_f16(double r) {
    // r is already a representable half value (or inf / nan / zero).
    uint32_t sign = std::signbit(r) ? 0x8000u : 0u;
    if (std::isnan(r)) return 0x7E00u;
    double a = std::fabs(r);
    if (std::isinf(a)) return sign | 0x7C00u;
    if (a == 0.0) return sign;
    int e2;
    std::frexp(a, &e2);
    int lead = e2 - 1;
    if (lead < -14) {  // subnormal: a = m * 2^-24 with integer m < 1024
        uint32_t m = static_cast<uint32_t>(std::ldexp(a, 24));
        return sign | m;
    }
    uint32_t exp_field = static_cast<uint32_t>(lead + 15);
    uint32_t m = static_cast<uint32_t>(std::ldexp(a, 10 - lead)) - 1024u;
    return sign | (exp_field << 10) | m;
}

double decode_f16(uint32_t b) {
    double sign = (b & 0x8000u) ? -1.0 : 1.0;
    uint32_t e = (b >> 10) & 0x1Fu;
    uint32_t m = b & 0x3FFu;
    if (e == 0x1Fu) return m ? NAN : sign * INFINITY;
    if (e == 0) return sign * std::ldexp(static_cast<double>(m), -24);
    return sign * std::ldexp(1024.0 + m, static_cast<int>(e) - 25);
}

uint32_t encode(double v, int fmt) {
    FormatSpec s;
    format_spec(fmt, &s);
    if (std::isnan(v)) return fmt == F32 ? 0x7FC00000u : (fmt == BF16 ? 0x7FC0u : 0x7E00u);
    double r = round_to_format(v, s);
    if (fmt == F16) return encode_f16(r);
    float f = static_cast<float>(r);  // exact: r is representable in binary32
    uint32_t bits;
    std::memcpy(&bits, &f, 4);
    return fmt == F32 ? bits : (bits >> 16);
}

double decode(uint32_t bits, int fmt) {
    if (fmt == F16) return decode_f16(bits & 0xFFFFu);
    uint32_t b32 = fmt == F32 ? bits : ((bits & 0xFFFFu) << 16);
    float f;
    std::memcpy(&f, &b32, 4);
    return static_cast<double>(f);
}

int elem_size(int fmt) { return fmt == F32 ? 4 : 2; }

double load(const void* base, int64_t idx, int fmt) {
    if (fmt == F32) {
        uint32_t b;
        std::memcpy(&b, static_cast<const char*>(base) + idx * 4, 4);
        return decode(b, fmt);
    }
    uint16_t h;
    std::memcpy(&h, static_cast<const char*>(base) + idx * 2, 2);
    return decode(h, fmt);
}

void store(void* base, int64_t idx, double v, int fmt) {
    uint32_t b = encode(v, fmt);
    if (fmt == F32) {
        std::memcpy(static_cast<char*>(base) + idx * 4, &b, 4);
    } else {
        uint16_t h = static_cast<uint16_t>(b);
        std::memcpy(static_cast<char*>(base) + idx * 2, &h, 2);
    }
}

// RMSNorm of one row already decoded to double ([koas] section 3; [lsln] 2.3;
// [csdn]): mean of squares over D, eps inside the root, one rounding on write.
void rmsnorm_row(const double* x, const void* w, void* out, int64_t out_off, int64_t D,
                 double eps, int fmt) {
    double sum_sq = 0.0;
    for (int64_t j = 0; j < D; ++j) sum_sq += x[j] * x[j];
    double mean_sq = sum_sq / static_cast<double>(D);
    double inv_rms = 1.0 / std::sqrt(mean_sq + eps);
    for (int64_t j = 0; j < D; ++j) {
        double wj = load(w, j, fmt);
        store(out, out_off + j, x[j] * inv_rms * wj, fmt);
    }
}

}  // namespace

extern "C" {

int orc_version(void) { return 1; }

// Round `v` to format `fmt` (0 = fp32, 1 = fp16, 2 = bf16), returning its bits.
uint32_t orc_encode(double v, int fmt) { return encode(v, fmt); }

// Value of the bit pattern `bits` in format `fmt`.
double orc_decode(uint32_t bits, int fmt) { return decode(bits, fmt); }

// out[r, :] = x[r, :] / sqrt(mean_j x[r, j]^2 + eps) * w[:]
// x, out: rows x D, row strides in elements. Returns 0, or -1 on bad arguments.
int orc_rmsnorm(const void* x, const void* w, void* out, int64_t rows, int64_t D,
                int64_t x_row_stride, int64_t out_row_stride, double eps, int fmt) {
    FormatSpec s;
    if (!format_spec(fmt, &s) || rows < 0 || D <= 0) return -1;
    double* row = new double[D];
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < D; ++j) row[j] = load(x, r * x_row_stride + j, fmt);
        rmsnorm_row(row, w, out, r * out_row_stride, D, eps, fmt);
    }
    delete[] row;
    return 0;
}

// Residual add then RMSNorm ([koas] section 4): x[r, :] <- round(x[r, :] + res[r, :])
// in place; out[r, :] = rmsnorm(the rounded, stored x[r, :]).
int orc_add_rmsnorm(void* x, const void* res, const void* w, void* out, int64_t rows,
                    int64_t D, int64_t x_row_stride, int64_t res_row_stride,
                    int64_t out_row_stride, double eps, int fmt) {
    FormatSpec s;
    if (!format_spec(fmt, &s) || rows < 0 || D <= 0) return -1;
    double* row = new double[D];
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < D; ++j) {
            double sum = load(x, r * x_row_stride + j, fmt) + load(res, r * res_row_stride + j, fmt);
            store(x, r * x_row_stride + j, sum, fmt);
            row[j] = load(x, r * x_row_stride + j, fmt);  // the rounded value
        }
        rmsnorm_row(row, w, out, r * out_row_stride, D, eps, fmt);
    }
    delete[] row;
    return 0;
}

// Rotation partner layout of a head of width head_dim, h = head_dim / 2, pair i < h:
//   neox (style 0, [koas] section 1: slice halves, negate, concatenate): (i, i + h)
//   interleaved (style 1, GPT-J; m.lsln.cn "21 个算子" section 2.3: even/odd
//   partner d, d +- 1):                                                  (2i, 2i + 1)
// Both use c = cos[p, i], s = sin[p, i] for pair i.
static void pair_index(int style, int i, int h, int* lo, int* hi) {
    if (style == 0) {
        *lo = i;
        *hi = i + h;
    } else {
        *lo = 2 * i;
        *hi = 2 * i + 1;
    }
}

// Neox half-rotation of every Q and K head at position pos[t], Q rotated in place,
// K_rot and V written through slot_mapping into a paged cache ([koas] section 1;
// cache layout [2, num_blocks, block_size, n_kv_head, head_dim] from [mer] 1.1).
// With h = head_dim / 2, c = cos[p, i], s = sin[p, i] (tables [max_pos, h], fp32):
//   y[i]     = x[i] * c - x[i + h] * s
//   y[i + h] = x[i + h] * c + x[i] * s
// Token t: a position outside [0, max_pos) counts one error and leaves q[t] and the
// cache untouched; slot < 0 is a padding token (no cache write, no error); a slot
// >= num_blocks * block_size counts one error and skips the cache write.
// Returns the error count, or -1 on bad arguments or duplicate valid slots.
int64_t orc_rope_kv_store_style(void* q, const void* k, const void* v, const float* cos_t,
                                const float* sin_t, const int64_t* pos, const int64_t* slot_mapping,
                                void* kv_cache, int64_t T, int n_head, int n_kv_head, int head_dim,
                                int64_t q_tok_stride, int64_t k_tok_stride, int64_t v_tok_stride,
                                int64_t max_pos, int64_t num_blocks, int block_size, int fmt, int style) {
    FormatSpec s;
    if (!format_spec(fmt, &s) || T < 0 || n_head <= 0 || n_kv_head <= 0 || head_dim <= 0 ||
        head_dim % 2 != 0 || n_head % n_kv_head != 0 || block_size <= 0 || num_blocks < 0 ||
        (style != 0 && style != 1))
        return -1;
    const int h = head_dim / 2;
    const int64_t capacity = num_blocks * block_size;
    std::set<int64_t> seen;
    for (int64_t t = 0; t < T; ++t) {
        int64_t sl = slot_mapping[t];
        if (sl >= 0 && sl < capacity && pos[t] >= 0 && pos[t] < max_pos) {
            if (!seen.insert(sl).second) return -1;
        }
    }
    int64_t errors = 0;
    double* xin = new double[head_dim];
    for (int64_t t = 0; t < T; ++t) {
        const int64_t p = pos[t];
        const int64_t sl = slot_mapping[t];
        const bool pos_ok = p >= 0 && p < max_pos;
        const bool slot_in_range = sl < capacity;
        if (!pos_ok) errors += 1;
        if (sl >= 0 && !slot_in_range) errors += 1;
        if (!pos_ok) continue;
        const float* c_row = cos_t + p * h;
        const float* s_row = sin_t + p * h;
        // Q heads: rotate in place.
        for (int hd = 0; hd < n_head; ++hd) {
            const int64_t base = t * q_tok_stride + static_cast<int64_t>(hd) * head_dim;
            for (int d = 0; d < head_dim; ++d) xin[d] = load(q, base + d, fmt);
            for (int i = 0; i < h; ++i) {
                const double c = c_row[i], sn = s_row[i];
                int lo, hi;
                pair_index(style, i, h, &lo, &hi);
                store(q, base + lo, xin[lo] * c - xin[hi] * sn, fmt);
                store(q, base + hi, xin[hi] * c + xin[lo] * sn, fmt);
            }
        }
        if (sl < 0 || !slot_in_range) continue;
        const int64_t blk = sl / block_size;
        const int64_t off = sl % block_size;
        for (int kvh = 0; kvh < n_kv_head; ++kvh) {
            // cache[0 or 1, blk, off, kvh, :]
            const int64_t k_dst = (((0 * num_blocks + blk) * block_size + off) * n_kv_head + kvh) *
                                  static_cast<int64_t>(head_dim);
            const int64_t v_dst = (((1 * num_blocks + blk) * block_size + off) * n_kv_head + kvh) *
                                  static_cast<int64_t>(head_dim);
            const int64_t k_src = t * k_tok_stride + static_cast<int64_t>(kvh) * head_dim;
            const int64_t v_src = t * v_tok_stride + static_cast<int64_t>(kvh) * head_dim;
            for (int d = 0; d < head_dim; ++d) xin[d] = load(k, k_src + d, fmt);
            for (int i = 0; i < h; ++i) {
                const double c = c_row[i], sn = s_row[i];
                int lo, hi;
                pair_index(style, i, h, &lo, &hi);
                store(kv_cache, k_dst + lo, xin[lo] * c - xin[hi] * sn, fmt);
                store(kv_cache, k_dst + hi, xin[hi] * c + xin[lo] * sn, fmt);
            }
            // V is stored unchanged: copy the element bits.
            const int es = elem_size(fmt);
            std::memcpy(static_cast<char*>(kv_cache) + v_dst * es,
                        static_cast<const char*>(v) + v_src * es, static_cast<size_t>(head_dim) * es);
        }
    }
    delete[] xin;
    return errors;
}

// The neox layout (style 0) of orc_rope_kv_store_style.
int64_t orc_rope_kv_store(void* q, const void* k, const void* v, const float* cos_t, const float* sin_t,
                          const int64_t* pos, const int64_t* slot_mapping, void* kv_cache, int64_t T,
                          int n_head, int n_kv_head, int head_dim, int64_t q_tok_stride,
                          int64_t k_tok_stride, int64_t v_tok_stride, int64_t max_pos, int64_t num_blocks,
                          int block_size, int fmt) {
    return orc_rope_kv_store_style(q, k, v, cos_t, sin_t, pos, slot_mapping, kv_cache, T, n_head,
                                   n_kv_head, head_dim, q_tok_stride, k_tok_stride, v_tok_stride, max_pos,
                                   num_blocks, block_size, fmt, 0);
}

// Gated linear unit over a fused gate_up tensor [T, 2I] (gate = columns [0, I),
// up = columns [I, 2I)): out[t, j] = act(g) * u with act = silu (g / (1 + e^-g),
// [koas] section 2) for act == 0 or relu (max(g, 0), [mer] section 3.3) for act == 1.
int orc_glu(const void* gate_up, void* out, int64_t T, int64_t I, int64_t in_row_stride,
            int64_t out_row_stride, int act, int fmt) {
    FormatSpec s;
    if (!format_spec(fmt, &s) || T < 0 || I <= 0 || (act != 0 && act != 1)) return -1;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t j = 0; j < I; ++j) {
            const double g = load(gate_up, t * in_row_stride + j, fmt);
            const double u = load(gate_up, t * in_row_stride + I + j, fmt);
            double a;
            if (act == 0) {
                a = g / (1.0 + std::exp(-g));
            } else {
                a = g > 0.0 ? g : 0.0;
            }
            store(out, t * out_row_stride + j, a * u, fmt);
        }
    }
    return 0;
}

// UClip / DyHT "norm" over rows of D channels: out = clamp(a * x, lo, hi) * g
// ([mer] section 0: DyHT(x) = y * clamp(a x, -1, 1), replacing every RMSNorm;
// section 3.3: the uclip kernel's per-channel or scalar alpha and gamma and its
// clip bounds). x and out are [N, H, D] with element strides (n_stride, h_stride, 1)
// each, so narrow Q/K views of a fused QKV buffer are read in place. alpha and
// gamma are fp32, D entries each when per-channel, else one entry. The page's
// kernel clamps with fmaxf then fminf, which return the non-NaN operand, so a NaN
// a * x becomes the lower bound; lo > hi or a NaN bound is an error.
//
// Precision: the page's kernel fixes it. It converts x to float and evaluates
// a * x and the product with g in float, so this function does the same: two
// fp32 roundings (a * x, then * g) around the clamp, with the bounds taken as
// fp32 values, then one RNE to the output format.
int orc_uclip(const void* x, const float* alpha, const float* gamma, void* out, int64_t N, int64_t H,
              int64_t D, int64_t x_n_stride, int64_t x_h_stride, int64_t out_n_stride, int64_t out_h_stride,
              int alpha_per_channel, int gamma_per_channel, double lo, double hi, int fmt) {
    FormatSpec s;
    if (!format_spec(fmt, &s) || N < 0 || H < 0 || D <= 0) return -1;
    if (std::isnan(lo) || std::isnan(hi) || lo > hi) return -1;
    const float lo32 = static_cast<float>(lo), hi32 = static_cast<float>(hi);
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t hh = 0; hh < H; ++hh) {
            for (int64_t d = 0; d < D; ++d) {
                const float a = alpha[alpha_per_channel ? d : 0];
                const float g = gamma[gamma_per_channel ? d : 0];
                // a value of any of the three formats is exact in float
                const float xf = static_cast<float>(load(x, n * x_n_stride + hh * x_h_stride + d, fmt));
                float v = a * xf;
                if (std::isnan(v)) v = lo32;  // the page's fmaxf keeps the bound when a * x is NaN
                if (v < lo32) v = lo32;
                if (v > hi32) v = hi32;
                const float y = v * g;
                store(out, n * out_n_stride + hh * out_h_stride + d, static_cast<double>(y), fmt);
            }
        }
    }
    return 0;
}

// Decode attention over a paged KV cache: for request b and query head h,
//   s_t = scale * sum_d q[b, h, d] * K_t[d],   o = sum_t softmax(s)_t * V_t,
// over the request's first seq_lens[b] tokens, token t living in cache block
// block_table[b, t / block_size] at offset t % block_size, kv head h / (n_head /
// n_kv_head) ([mer] section 1.1: cache [2, num_blocks, block_size, n_kv, head]
// with a block table and seq lens per request; section 3.1: the decode kernel
// reads that layout through the block table; [lsln] section 2.1: qk_score,
// scale + softmax and pv_agg as one attention read of the cache). Softmax is
// taken with its maximum subtracted (the same function, written stably).
// Bad inputs are skipped and counted: a seq_len outside [0, max_blocks *
// block_size] is clamped into it (one error per request); a block id outside
// [0, num_blocks) drops that block's tokens (one error per block entry used). A
// request with no token left gets o = 0. Returns the error count, or -1 for bad
// arguments.
int64_t orc_paged_decode_attention(const void* q, const void* kv_cache, const int32_t* block_table,
                                   const int32_t* seq_lens, void* out, int64_t B, int n_head, int n_kv_head,
                                   int head_dim, int64_t q_tok_stride, int64_t out_tok_stride, int64_t num_blocks,
                                   int block_size, int64_t max_blocks, double scale, int fmt) {
    FormatSpec spec;
    if (!format_spec(fmt, &spec) || B < 0 || n_head <= 0 || n_kv_head <= 0 || n_head % n_kv_head != 0 ||
        head_dim <= 0 || block_size <= 0 || max_blocks < 0 || num_blocks < 0)
        return -1;
    const int group = n_head / n_kv_head;
    int64_t errors = 0;
    std::vector<double> s, qd(head_dim), acc(head_dim);
    std::vector<int64_t> rows;  // element offset of each valid token's K row (kv head 0)
    for (int64_t b = 0; b < B; ++b) {
        int64_t L = seq_lens[b];
        if (L < 0 || L > max_blocks * block_size) {
            ++errors;
            L = L < 0 ? 0 : max_blocks * block_size;
        }
        rows.clear();
        for (int64_t j = 0; j * block_size < L; ++j) {
            const int64_t blk = block_table[b * max_blocks + j];
            if (blk < 0 || blk >= num_blocks) {
                ++errors;
                continue;
            }
            for (int64_t off = 0; off < block_size && j * block_size + off < L; ++off)
                rows.push_back((blk * block_size + off) * n_kv_head * static_cast<int64_t>(head_dim));
        }
        const int64_t v_plane = num_blocks * block_size * n_kv_head * static_cast<int64_t>(head_dim);
        for (int h = 0; h < n_head; ++h) {
            const int64_t kvh_off = static_cast<int64_t>(h / group) * head_dim;
            for (int d = 0; d < head_dim; ++d) qd[d] = load(q, b * q_tok_stride + static_cast<int64_t>(h) * head_dim + d, fmt);
            s.assign(rows.size(), 0.0);
            double m = -INFINITY;
            for (size_t t = 0; t < rows.size(); ++t) {
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d) dot += qd[d] * load(kv_cache, rows[t] + kvh_off + d, fmt);
                s[t] = scale * dot;
                if (s[t] > m) m = s[t];
            }
            double denom = 0.0;
            std::fill(acc.begin(), acc.end(), 0.0);
            for (size_t t = 0; t < rows.size(); ++t) {
                const double p = std::exp(s[t] - m);
                denom += p;
                for (int d = 0; d < head_dim; ++d) acc[d] += p * load(kv_cache, v_plane + rows[t] + kvh_off + d, fmt);
            }
            for (int d = 0; d < head_dim; ++d)
                store(out, b * out_tok_stride + static_cast<int64_t>(h) * head_dim + d,
                      rows.empty() ? 0.0 : acc[d] / denom, fmt);
        }
    }
    return errors;
}

// The linear layer of a decoder (nn.Linear's layout): y[b, n] = sum_k h[b, k] * W[n, k]
// with W [N, K] row-major, accumulated in double and rounded once ([lsln] section
// 2.2: ln1 feeds qkv_proj; the norm's output h is what the separate norm kernel
// stores, in the same format). Used after rmsnorm (norm as the GEMV's prologue) and
// after the GLU (the activation fused into the down projection).
int orc_linear(const void* h, const void* W, void* y, int64_t B, int64_t K, int64_t N, int64_t h_row_stride,
               int64_t y_row_stride, int fmt) {
    FormatSpec s;
    if (!format_spec(fmt, &s) || B < 0 || K <= 0 || N <= 0) return -1;
    std::vector<double> hb(K);
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t k = 0; k < K; ++k) hb[k] = load(h, b * h_row_stride + k, fmt);
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += hb[k] * load(W, n * K + k, fmt);
            store(y, b * y_row_stride + n, acc, fmt);
        }
    }
    return 0;
}

}  // extern "C"
