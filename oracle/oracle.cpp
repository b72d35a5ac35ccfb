// Oracle for decode_step_batch: a plain, slow, obviously correct CPU model.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or call
// this file; only the test suite, the package's smoke check and the bench's
// CPU-baseline leg use it. It shares no code, header, table or constant
// generator with the CUDA library.
//
// Arithmetic: IEEE f32, compiled with -ffp-contract=off (no fused multiply-add)
// and without -ffast-math, so every sum is a single accumulator taken in
// ascending index order. That is the structural rule the pages give for the
// batched step being bit-identical to the serial step:
//   MODEL-BATCHING-RESULTS, "Correctness — proven, not asserted": row b of the
//   batched matmul is the same dot product in the same index order as the
//   serial matvec, and per-user attention replays the serial scalar arithmetic
//   (a dot for each score, an in-order V accumulation); no FMA ("The honest
//   ceiling": FMA is forgone to keep scalar bit-identity).
//
// Model: dense Llama-style decoder (RMSNorm, rotate-half RoPE, GQA attention,
// SwiGLU FFN), as named for the path in "The lever": seven weight matmuls per
// layer (Q, K, V, O, gate, up, down) plus the LM head over a [B, d] panel, with
// attention per user over that user's own KV cache.
//
// Readings taken where the pages are silent:
//   * RMSNorm: y = x * (1/sqrtf(sum(x^2)/d + eps)) * g, sum ascending.
//   * RoPE: rotate-half pairing (i, i + hd/2), theta_i = theta^(-2i/hd), the
//     angle and its cos/sin taken in double and rounded to f32; the position
//     is the number of tokens already in the lane, captured once for Q and K
//     (mlx-bun parallel-slots design, "S1b decode: design traps", trap 2).
//   * attention keys are 0..pos inclusive (the new token is appended first);
//     scale 1/sqrtf(hd); softmax subtracts the max, expf, ascending sum, then
//     p_t = e_t / sum; o = sum_t p_t * v_t in ascending t.
//   * silu(z) = z / (1 + expf(-z)).
//   * Q8_0 weights are dequantised to f32 as q * float(d16) before the dot.
//   * greedy ties go to the lowest index; temperature sampling draws
//     u = (Philox4x32-10(key=seed, ctr=counter) >> 11) * 2^-53 and picks the
//     first index whose ascending cumulative sum of exp(z_i - max z) (in
//     double, z = logit / T) reaches u * total.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <cstdlib>
#include <vector>
#include <thread>
#include <algorithm>

static int g_threads = 1;

// Output rows are split across threads; each row is computed by exactly one
// thread in the serial order, so the bits do not depend on the thread count.
template <class Fn>
static void par_rows(int rows, Fn fn) {
  int nt = std::min(g_threads, std::max(1, rows / 8));
  if (nt <= 1) {
    fn(0, rows);
    return;
  }
  std::vector<std::thread> ts;
  int chunk = (rows + nt - 1) / nt;
  for (int t = 0; t < nt; ++t) {
    int a = t * chunk, b = std::min(rows, a + chunk);
    if (a >= b) break;
    ts.emplace_back([=, &fn] { fn(a, b); });
  }
  for (auto& t : ts) t.join();
}


extern "C" {

void or_set_threads(int n) { g_threads = n < 1 ? 1 : n; }
int or_get_threads(void) { return g_threads; }

// ---------------------------------------------------------------------------
// Scalar encodings (input formats)
// ---------------------------------------------------------------------------

float or_bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// IEEE binary16 -> binary32, exact (normals, subnormals, inf, nan).
float or_f16_to_f32(uint16_t h) {
  uint32_t sign = (uint32_t)(h >> 15) << 31;
  uint32_t exp = (h >> 10) & 0x1f;
  uint32_t man = h & 0x3ff;
  uint32_t u;
  if (exp == 0) {
    if (man == 0) {
      u = sign;
    } else {  // subnormal: value = man * 2^-24
      float f = (float)man * (1.0f / 16777216.0f);
      std::memcpy(&u, &f, 4);
      u |= sign;
    }
  } else if (exp == 31) {
    u = sign | 0x7f800000u | (man << 13);
  } else {
    u = sign | ((exp - 15 + 127) << 23) | (man << 13);
  }
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// IEEE binary32 -> binary16 with round-to-nearest-even (overflow -> inf).
uint16_t or_f32_to_f16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000);
  uint32_t a = u & 0x7fffffffu;
  if (a >= 0x7f800000u) {  // inf or nan
    return sign | (a > 0x7f800000u ? 0x7e00 : 0x7c00);
  }
  int e = (int)(a >> 23) - 127;  // unbiased exponent
  uint32_t m = (a & 0x7fffff) | 0x800000;  // 24-bit significand (normal)
  if (a < 0x00800000u) return sign;  // f32 subnormals are far below f16 range
  if (e > 15) return sign | 0x7c00;
  int shift;       // bits to drop from the 24-bit significand
  uint16_t hexp;
  if (e >= -14) {  // normal in f16: keep 11 bits
    shift = 13;
    hexp = (uint16_t)(e + 15);
  } else {         // subnormal in f16: value = m * 2^(e-23); unit is 2^-24
    shift = 13 + (-14 - e);
    hexp = 0;
    if (shift > 24) return sign;  // rounds to zero (below half of 2^-24)
  }
  uint32_t keep = m >> shift;
  uint32_t rem = m & ((1u << shift) - 1);
  uint32_t half = 1u << (shift - 1);
  if (rem > half || (rem == half && (keep & 1))) keep += 1;
  uint32_t out;
  if (hexp == 0) {
    out = keep;  // may carry into the smallest normal, which encodes correctly
  } else {
    out = ((uint32_t)hexp << 10) + (keep - 0x400);  // drop the hidden bit
    if (keep == 0x800) out = ((uint32_t)(hexp + 1) << 10);  // carry
  }
  if (out >= 0x7c00) return sign | 0x7c00;
  return sign | (uint16_t)out;
}

// f32 -> bf16 with round-to-nearest-even (nan kept quiet).
uint16_t or_f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1;
  u += 0x7fff + lsb;
  return (uint16_t)(u >> 16);
}

// ---------------------------------------------------------------------------
// Q8_0: blocks of 32 inputs, each stored as fp16 scale d then 32 int8 codes
// (34 bytes). d = max|x| / 127, q = round-half-away(x / d) via x * (1/d),
// clamped to [-127, 127]; d stored as fp16 (RNE); d == 0 gives q = 0.
// ---------------------------------------------------------------------------

void or_quantize_q8_0(const float* x, int64_t n, uint8_t* blocks) {
  for (int64_t b = 0; b < n / 32; ++b) {
    const float* xb = x + b * 32;
    float amax = 0.0f;
    for (int j = 0; j < 32; ++j) amax = std::max(amax, std::fabs(xb[j]));
    float d = amax / 127.0f;
    float id = d != 0.0f ? 1.0f / d : 0.0f;
    uint16_t d16 = or_f32_to_f16(d);
    uint8_t* out = blocks + b * 34;
    out[0] = (uint8_t)(d16 & 0xff);
    out[1] = (uint8_t)(d16 >> 8);
    for (int j = 0; j < 32; ++j) {
      float v = std::round(xb[j] * id);
      if (v > 127.0f) v = 127.0f;
      if (v < -127.0f) v = -127.0f;
      out[2 + j] = (uint8_t)(int8_t)v;
    }
  }
}

void or_dequantize_q8_0(const uint8_t* blocks, int64_t n, float* x) {
  for (int64_t b = 0; b < n / 32; ++b) {
    const uint8_t* in = blocks + b * 34;
    float d = or_f16_to_f32((uint16_t)(in[0] | (in[1] << 8)));
    for (int j = 0; j < 32; ++j) x[b * 32 + j] = (float)(int8_t)in[2 + j] * d;
  }
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC 2011): 10 rounds of the 4x32 Philox S-box with multipliers
// 0xD2511F53 / 0xCD9E8D57 and Weyl key increments 0x9E3779B9 / 0xBB67AE85.
// ---------------------------------------------------------------------------

void or_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                      uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int r = 0; r < 10; ++r) {
    uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

// u in [0, 1) with 53 random bits, from (seed, counter).
double or_uniform(uint64_t seed, uint64_t counter) {
  uint32_t ctr[4] = {(uint32_t)counter, (uint32_t)(counter >> 32), 0u, 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t o[4];
  or_philox4x32_10(ctr, key, o);
  uint64_t bits = ((uint64_t)o[0] << 32) | o[1];
  return (double)(bits >> 11) * (1.0 / 9007199254740992.0);
}

// Per-lane sampler. temp == 0: argmax, lowest index on ties.
int or_sample(const float* logits, int V, float temp, uint64_t seed,
              uint64_t counter) {
  if (temp == 0.0f) {
    int best = 0;
    for (int i = 1; i < V; ++i)
      if (logits[i] > logits[best]) best = i;
    return best;
  }
  std::vector<double> z(V);
  double m = -INFINITY;
  for (int i = 0; i < V; ++i) {
    z[i] = (double)logits[i] / (double)temp;
    if (z[i] > m) m = z[i];
  }
  double total = 0.0;
  for (int i = 0; i < V; ++i) {
    z[i] = std::exp(z[i] - m);
    total += z[i];
  }
  double target = or_uniform(seed, counter) * total;
  double cum = 0.0;
  int last_pos = 0;
  for (int i = 0; i < V; ++i) {
    if (z[i] > 0.0) last_pos = i;
    cum += z[i];
    if (cum >= target && z[i] > 0.0) return i;
  }
  return last_pos;
}

// ---------------------------------------------------------------------------
// Building blocks, each callable on its own for the brute-force pins.
// ---------------------------------------------------------------------------

static float dot_f32(const float* a, const float* b, int n) {
  float acc = 0.0f;
  for (int k = 0; k < n; ++k) acc += a[k] * b[k];
  return acc;
}

// y[o] = sum_k W[o,k] * x[k], W row-major [rows, cols].
void or_matvec(const float* W, int rows, int cols, const float* x, float* y) {
  par_rows(rows, [&](int a, int b) {
    for (int o = a; o < b; ++o) y[o] = dot_f32(W + (int64_t)o * cols, x, cols);
  });
}

// Panel matmul Y[b, o] = sum_k W[o,k] * X[b,k]: each weight row is taken once
// and reused across the n panel rows; per element the same dot as or_matvec.
void or_matmul_panel(const float* W, int rows, int cols, const float* X, int n,
                     float* Y) {
  par_rows(rows, [&](int a, int b) {
    for (int o = a; o < b; ++o) {
      const float* w = W + (int64_t)o * cols;
      for (int r = 0; r < n; ++r)
        Y[(int64_t)r * rows + o] = dot_f32(w, X + (int64_t)r * cols, cols);
    }
  });
}

void or_rmsnorm(const float* x, const float* g, int d, float eps, float* y) {
  float ss = 0.0f;
  for (int i = 0; i < d; ++i) ss += x[i] * x[i];
  float r = 1.0f / std::sqrt(ss / (float)d + eps);
  for (int i = 0; i < d; ++i) y[i] = x[i] * r * g[i];
}

// cos/sin of pos * theta^(-2i/hd) for i < hd/2, taken in double, rounded to f32.
void or_rope_table(int pos, int hd, double theta, float* cos_out,
                   float* sin_out) {
  for (int i = 0; i < hd / 2; ++i) {
    double inv = std::pow(theta, -2.0 * (double)i / (double)hd);
    double ang = (double)pos * inv;
    cos_out[i] = (float)std::cos(ang);
    sin_out[i] = (float)std::sin(ang);
  }
}

// Rotate-half RoPE applied in place to nheads vectors of length hd.
void or_rope(float* v, int nheads, int hd, int pos, double theta) {
  std::vector<float> c(hd / 2), s(hd / 2);
  or_rope_table(pos, hd, theta, c.data(), s.data());
  int half = hd / 2;
  for (int h = 0; h < nheads; ++h) {
    float* x = v + (int64_t)h * hd;
    for (int i = 0; i < half; ++i) {
      float a = x[i], b = x[i + half];
      x[i] = a * c[i] - b * s[i];
      x[i + half] = b * c[i] + a * s[i];
    }
  }
}

// softmax over n scores in place: subtract max, expf, ascending sum, divide.
void or_softmax(float* s, int n) {
  float m = s[0];
  for (int t = 1; t < n; ++t) m = std::max(m, s[t]);
  float sum = 0.0f;
  for (int t = 0; t < n; ++t) {
    s[t] = std::exp(s[t] - m);
    sum += s[t];
  }
  for (int t = 0; t < n; ++t) s[t] = s[t] / sum;
}

// One query head against n_keys cached keys/values; kv rows have stride
// kv_stride floats between consecutive positions.
void or_attend_head(const float* q, const float* K, const float* V, int n_keys,
                    int hd, int64_t kv_stride, float* o) {
  std::vector<float> s(n_keys);
  float scale = 1.0f / std::sqrt((float)hd);
  for (int t = 0; t < n_keys; ++t)
    s[t] = dot_f32(q, K + (int64_t)t * kv_stride, hd) * scale;
  or_softmax(s.data(), n_keys);
  for (int i = 0; i < hd; ++i) o[i] = 0.0f;
  for (int t = 0; t < n_keys; ++t) {
    const float* v = V + (int64_t)t * kv_stride;
    for (int i = 0; i < hd; ++i) o[i] += s[t] * v[i];
  }
}

float or_silu(float z) { return z / (1.0f + std::exp(-z)); }

// ---------------------------------------------------------------------------
// Model and lanes
// ---------------------------------------------------------------------------

typedef struct {
  int L, d, H, Hkv, hd, F, V;
  float rms_eps;
  double rope_theta;
  int tied;  // LM head shares the embedding matrix
} or_desc;

enum { OR_F32 = 0, OR_BF16 = 1, OR_Q8_0 = 2 };

struct OrLayer {
  std::vector<float> wq, wk, wv, wo, wg, wu, wd, g_attn, g_ffn;
};

struct OrModel {
  or_desc c;
  // KV storage: 0 = f32; 1 = bf16 values (a roped key and a value are
  // rounded to bf16, nearest-even, when they enter the cache; the un-roped
  // keys stay f32), the storage of a bf16 KV arena
  int kv_bf16 = 0;
  std::vector<float> embed, head, g_final;
  std::vector<OrLayer> layers;
  const float* head_ptr() const { return c.tied ? embed.data() : head.data(); }
};

struct OrLane {
  int pos = 0;
  int max_pos = 0;
  // per layer: [max_pos][Hkv][hd]
  std::vector<std::vector<float>> K, Kraw, V;
};

static std::vector<float> load_matrix(const void* src, int dtype, int64_t rows,
                                      int64_t cols) {
  std::vector<float> w((size_t)(rows * cols));
  int64_t n = rows * cols;
  if (dtype == OR_F32) {
    std::memcpy(w.data(), src, (size_t)n * 4);
  } else if (dtype == OR_BF16) {
    const uint16_t* s = (const uint16_t*)src;
    for (int64_t i = 0; i < n; ++i) w[i] = or_bf16_to_f32(s[i]);
  } else {
    or_dequantize_q8_0((const uint8_t*)src, n, w.data());
  }
  return w;
}

// layer_ptrs: L * 9 pointers, per layer in the order
//   wq [H*hd, d], wk [Hkv*hd, d], wv [Hkv*hd, d], wo [d, H*hd],
//   w_gate [F, d], w_up [F, d], w_down [d, F]  (all in `dtype`),
//   attn_norm [d], ffn_norm [d]  (f32).
// embed [V, d] and head [V, d] are in `dtype`; head may be NULL when tied.
void* or_model_create(const or_desc* c, int dtype, const void* embed,
                      const void* head, const float* final_norm,
                      const void* const* layer_ptrs) {
  OrModel* m = new OrModel();
  m->c = *c;
  int d = c->d, qd = c->H * c->hd, kvd = c->Hkv * c->hd, F = c->F;
  m->embed = load_matrix(embed, dtype, c->V, d);
  if (!c->tied) m->head = load_matrix(head, dtype, c->V, d);
  m->g_final.assign(final_norm, final_norm + d);
  m->layers.resize(c->L);
  for (int l = 0; l < c->L; ++l) {
    const void* const* p = layer_ptrs + l * 9;
    OrLayer& ly = m->layers[l];
    ly.wq = load_matrix(p[0], dtype, qd, d);
    ly.wk = load_matrix(p[1], dtype, kvd, d);
    ly.wv = load_matrix(p[2], dtype, kvd, d);
    ly.wo = load_matrix(p[3], dtype, d, qd);
    ly.wg = load_matrix(p[4], dtype, F, d);
    ly.wu = load_matrix(p[5], dtype, F, d);
    ly.wd = load_matrix(p[6], dtype, d, F);
    ly.g_attn.assign((const float*)p[7], (const float*)p[7] + d);
    ly.g_ffn.assign((const float*)p[8], (const float*)p[8] + d);
  }
  return m;
}

void or_model_free(void* m) { delete (OrModel*)m; }

void* or_lane_create(void* mp, int max_pos) {
  OrModel* m = (OrModel*)mp;
  OrLane* ln = new OrLane();
  ln->max_pos = max_pos;
  size_t per = (size_t)max_pos * m->c.Hkv * m->c.hd;
  ln->K.assign(m->c.L, std::vector<float>(per, 0.0f));
  ln->Kraw.assign(m->c.L, std::vector<float>(per, 0.0f));
  ln->V.assign(m->c.L, std::vector<float>(per, 0.0f));
  return ln;
}

void or_lane_free(void* l) { delete (OrLane*)l; }
void or_lane_reset(void* l) { ((OrLane*)l)->pos = 0; }
int or_lane_pos(void* l) { return ((OrLane*)l)->pos; }

// which: 0 = K (roped), 1 = Kraw (un-roped), 2 = V. Copies pos*Hkv*hd floats.
void or_lane_export(void* mp, void* lp, int layer, int which, float* out) {
  OrModel* m = (OrModel*)mp;
  OrLane* ln = (OrLane*)lp;
  const std::vector<float>& src =
      which == 0 ? ln->K[layer] : (which == 1 ? ln->Kraw[layer] : ln->V[layer]);
  size_t n = (size_t)ln->pos * m->c.Hkv * m->c.hd;
  std::memcpy(out, src.data(), n * 4);
}

// Writes KV for positions [0, n) of one layer and sets the lane length to n
// on the last layer's import (used to seed long synthetic contexts).
void or_lane_import(void* mp, void* lp, int layer, const float* K,
                    const float* V, int n) {
  OrModel* m = (OrModel*)mp;
  OrLane* ln = (OrLane*)lp;
  size_t cnt = (size_t)n * m->c.Hkv * m->c.hd;
  std::memcpy(ln->K[layer].data(), K, cnt * 4);
  std::memcpy(ln->V[layer].data(), V, cnt * 4);
  if (m->kv_bf16)  // stored as the cache stores it
    for (size_t i = 0; i < cnt; ++i) {
      ln->K[layer][i] = or_bf16_to_f32(or_f32_to_bf16(ln->K[layer][i]));
      ln->V[layer][i] = or_bf16_to_f32(or_f32_to_bf16(ln->V[layer][i]));
    }
  std::fill(ln->Kraw[layer].begin(), ln->Kraw[layer].begin() + cnt, 0.0f);
  ln->pos = n;
}

// Clone ("MODEL-BATCHING-RESULTS", "Why in-kernel batching, not vLLM":
// per-user prefix reuse): lane dst becomes a copy of lane src's history
// (K, un-roped K, V of every layer and the length). Both lanes must have
// the same max_pos.
int or_lane_clone(void* srcp, void* dstp) {
  OrLane* src = (OrLane*)srcp;
  OrLane* dst = (OrLane*)dstp;
  if (src->max_pos != dst->max_pos) return -1;
  dst->K = src->K;
  dst->Kraw = src->Kraw;
  dst->V = src->V;
  dst->pos = src->pos;
  return 0;
}

// Evict (same passage: quarantine of a span of one user's history): the
// entries at positions [start, end) leave the cache; the entry at p >= end
// becomes the entry at p - (end - start), its V and un-roped K as they
// were and its K the un-roped K rotated at the new position. K/V are not
// recomputed. Returns -1 unless 0 <= start <= end <= length.
int or_lane_evict(void* mp, void* lp, int start, int end) {
  OrModel* m = (OrModel*)mp;
  OrLane* ln = (OrLane*)lp;
  if (start < 0 || start > end || end > ln->pos) return -1;
  const or_desc& c = m->c;
  const int delta = end - start;
  const size_t row = (size_t)c.Hkv * c.hd;
  for (int l = 0; l < c.L; ++l) {
    for (int p = end; p < ln->pos; ++p) {
      const int q = p - delta;
      std::memcpy(ln->Kraw[l].data() + q * row, ln->Kraw[l].data() + p * row, row * 4);
      std::memcpy(ln->V[l].data() + q * row, ln->V[l].data() + p * row, row * 4);
      float* k = ln->K[l].data() + q * row;
      std::memcpy(k, ln->Kraw[l].data() + q * row, row * 4);
      or_rope(k, c.Hkv, c.hd, q, c.rope_theta);
      if (m->kv_bf16)  // stored as the cache stores it
        for (size_t i = 0; i < row; ++i) k[i] = or_bf16_to_f32(or_f32_to_bf16(k[i]));
    }
  }
  ln->pos -= delta;
  return 0;
}

// Attention sub-step for one lane after its K/V at `pos` are appended:
// every query head h reads KV head h / (H / Hkv) over keys 0..pos.
static void lane_attention(const OrModel* m, const OrLane* ln, int layer,
                           const float* q, int pos, float* o) {
  const or_desc& c = m->c;
  int group = c.H / c.Hkv;
  int64_t stride = (int64_t)c.Hkv * c.hd;
  for (int h = 0; h < c.H; ++h) {
    int g = h / group;
    or_attend_head(q + (int64_t)h * c.hd, ln->K[layer].data() + g * c.hd,
                   ln->V[layer].data() + g * c.hd, pos + 1, c.hd, stride,
                   o + (int64_t)h * c.hd);
  }
}

// A value as the cache stores it.
static float kv_store(const OrModel* m, float x) {
  return m->kv_bf16 ? or_bf16_to_f32(or_f32_to_bf16(x)) : x;
}

static void append_kv(const OrModel* m, OrLane* ln, int layer, int pos,
                      const float* k_raw, const float* k_roped,
                      const float* v) {
  const or_desc& c = m->c;
  size_t n = (size_t)c.Hkv * c.hd;
  size_t off = (size_t)pos * n;
  std::memcpy(ln->Kraw[layer].data() + off, k_raw, n * 4);
  for (size_t i = 0; i < n; ++i) {
    ln->K[layer][off + i] = kv_store(m, k_roped[i]);
    ln->V[layer][off + i] = kv_store(m, v[i]);
  }
}

void or_model_set_kv_bf16(void* mp, int on) { ((OrModel*)mp)->kv_bf16 = on ? 1 : 0; }

// The batched step over n lanes; with n == 1 it is the serial Step. Every
// per-lane quantity is computed with the same scalar arithmetic either way.
// Returns 0, or -1 if a lane is full.
static int step_panel(OrModel* m, OrLane** lanes, const int* tokens, int n,
                      float* logits) {
  const or_desc& c = m->c;
  int d = c.d, qd = c.H * c.hd, kvd = c.Hkv * c.hd, F = c.F;
  for (int b = 0; b < n; ++b)
    if (lanes[b]->pos >= lanes[b]->max_pos) return -1;
  std::vector<float> x((size_t)n * d), h((size_t)n * d);
  std::vector<float> q((size_t)n * qd), k((size_t)n * kvd), v((size_t)n * kvd);
  std::vector<float> kr(kvd), att((size_t)n * qd), y((size_t)n * d);
  std::vector<float> gt((size_t)n * F), up((size_t)n * F), a((size_t)n * F);
  for (int b = 0; b < n; ++b)
    std::memcpy(&x[(size_t)b * d], &m->embed[(size_t)tokens[b] * d], d * 4);
  for (int l = 0; l < c.L; ++l) {
    OrLayer& ly = m->layers[l];
    for (int b = 0; b < n; ++b)
      or_rmsnorm(&x[(size_t)b * d], ly.g_attn.data(), d, c.rms_eps,
                 &h[(size_t)b * d]);
    or_matmul_panel(ly.wq.data(), qd, d, h.data(), n, q.data());
    or_matmul_panel(ly.wk.data(), kvd, d, h.data(), n, k.data());
    or_matmul_panel(ly.wv.data(), kvd, d, h.data(), n, v.data());
    for (int b = 0; b < n; ++b) {
      int pos = lanes[b]->pos;  // captured once for Q and K
      float* qb = &q[(size_t)b * qd];
      float* kb = &k[(size_t)b * kvd];
      std::memcpy(kr.data(), kb, kvd * 4);
      or_rope(qb, c.H, c.hd, pos, c.rope_theta);
      or_rope(kb, c.Hkv, c.hd, pos, c.rope_theta);
      append_kv(m, lanes[b], l, pos, kr.data(), kb, &v[(size_t)b * kvd]);
      lane_attention(m, lanes[b], l, qb, pos, &att[(size_t)b * qd]);
    }
    or_matmul_panel(ly.wo.data(), d, qd, att.data(), n, y.data());
    for (size_t i = 0; i < (size_t)n * d; ++i) x[i] = x[i] + y[i];
    for (int b = 0; b < n; ++b)
      or_rmsnorm(&x[(size_t)b * d], ly.g_ffn.data(), d, c.rms_eps,
                 &h[(size_t)b * d]);
    or_matmul_panel(ly.wg.data(), F, d, h.data(), n, gt.data());
    or_matmul_panel(ly.wu.data(), F, d, h.data(), n, up.data());
    for (size_t i = 0; i < (size_t)n * F; ++i) a[i] = or_silu(gt[i]) * up[i];
    or_matmul_panel(ly.wd.data(), d, F, a.data(), n, y.data());
    for (size_t i = 0; i < (size_t)n * d; ++i) x[i] = x[i] + y[i];
  }
  for (int b = 0; b < n; ++b) {
    or_rmsnorm(&x[(size_t)b * d], m->g_final.data(), d, c.rms_eps,
               &h[(size_t)b * d]);
    lanes[b]->pos += 1;
  }
  if (logits) or_matmul_panel(m->head_ptr(), c.V, d, h.data(), n, logits);
  return 0;
}

// Serial Step: one lane, one token; logits [V].
int or_step(void* m, void* lane, int token, float* logits) {
  OrLane* l = (OrLane*)lane;
  return step_panel((OrModel*)m, &l, &token, 1, logits);
}

// StepBatch: n lanes (distinct), one token each; logits [n, V] in input order.
int or_step_batch(void* m, void* const* lanes, const int* tokens, int n,
                  float* logits) {
  return step_panel((OrModel*)m, (OrLane**)lanes, tokens, n, logits);
}

// Serial prompt ingestion: one Step per token, logits of the last step kept.
int or_prefill(void* m, void* lane, const int* tokens, int n, float* logits) {
  for (int i = 0; i < n; ++i)
    if (or_step(m, lane, tokens[i], i == n - 1 ? logits : nullptr)) return -1;
  return 0;
}

// Serial greedy generation after a prompt: n_new tokens.
int or_generate(void* mp, void* lane, const int* prompt, int n_prompt,
                int n_new, int* out) {
  OrModel* m = (OrModel*)mp;
  std::vector<float> lg(m->c.V);
  if (or_prefill(m, lane, prompt, n_prompt, lg.data())) return -1;
  for (int t = 0; t < n_new; ++t) {
    out[t] = or_sample(lg.data(), m->c.V, 0.0f, 0, 0);
    if (t + 1 < n_new && or_step(m, lane, out[t], lg.data())) return -1;
  }
  return 0;
}

// Lockstep greedy over n lanes with ragged prompts: each lane is prefilled on
// its own (serial steps), then all lanes decode together through the panel.
int or_generate_batch(void* mp, void* const* lanes, const int* prompts,
                      const int* prompt_lens, int n, int n_new, int* out) {
  OrModel* m = (OrModel*)mp;
  int V = m->c.V;
  std::vector<float> lg((size_t)n * V);
  int off = 0;
  for (int b = 0; b < n; ++b) {
    if (or_prefill(m, lanes[b], prompts + off, prompt_lens[b],
                   &lg[(size_t)b * V]))
      return -1;
    off += prompt_lens[b];
  }
  std::vector<int> toks(n);
  for (int t = 0; t < n_new; ++t) {
    for (int b = 0; b < n; ++b) {
      toks[b] = or_sample(&lg[(size_t)b * V], V, 0.0f, 0, 0);
      out[(size_t)b * n_new + t] = toks[b];
    }
    if (t + 1 < n_new && or_step_batch(m, lanes, toks.data(), n, lg.data()))
      return -1;
  }
  return 0;
}

}  // extern "C"
